// qlora_gemv.cuh -- fused QLoRA forward for a few tokens (M <= 8, M * k <=
// 16384) of a group of projections that share one input:
//
//   Y_g = X deq(Q_g)^T + s_g (X A_g^T) B_g^T      X: M x k bf16, Q_g: d_g x k NF4
//
// ("PEFT course notes" §2.2, h = Wx + BAx; "QLoRA paper summary": the frozen
// weight is 4-bit NF4 with blockwise constants.)  The call is bound by the
// bytes of the packed weights (8-50 MB at decode sizes).  On this part an SM
// needs ~100 KB of reads in flight to cover HBM latency under load, and
// shared-memory copies with cp.async carry that with no registers, so:
//
// * the group's rows form one list, cut into equal contiguous ranges, one
//   per CTA (one CTA per SM, 16 warps); a range is cut into 16-row tiles and
//   each tile into stages of 16 rows x 2048 columns (16 KiB of codes);
// * all threads copy stages with 16-byte cp.async (whole 128-byte lines,
//   xor-swizzled in shared memory) into a kGvRing-deep ring: kGvRing - 1
//   stages (80 KiB) in flight while one is consumed; one barrier per stage
//   both publishes the stage and frees the slot of the previous one;
// * warp w takes 64-blocks w and w + 16 of each stage: a lane (group g,
//   thread t) reads 8 code bytes of rows g and g + 8, turns each byte into a
//   bf16x2 pair through a per-lane replicated byte-pair table (one byte
//   permute and one shared load with an immediate base per byte),
//   multiplies on mma.sync m16n8k16 (tokens are the N columns) against x,
//   which is staged as bf16 in the unused half of every table row, and
//   scales each block's dot products by its block constant in fp32.  The
//   MMA's k order is a permutation of the block's elements, the same for
//   both operands.  Each lane decodes one block constant per stage (row
//   lane mod 16, block w + 16 (lane / 16)) from the DQ codes and scales
//   copied to shared memory at the start;
// * at the end of a tile the warps' partial sums go to a double-buffered
//   area; during the next stage one warp adds them in warp order;
// * the adapter rows u = s X A^T are spread over the CTAs (row j by CTA
//   j mod G, split over the 16 warps) before the weight loop and published
//   through a ready counter; after the loop one thread per CTA waits
//   (bounded) for all of them, then thread i adds u . B[row i] and writes
//   bf16 Y = row sum + adapter term.
//
// Programmatic dependent launch: the kernel lets the next call launch at
// entry; before griddepcontrol.wait a CTA only builds its tables and
// prefetches its first stages into L2 (a prefetch cannot return stale data).
// Everything a kernel may have written -- codes, constants, X, A, B, u, Y,
// the counters -- is read after the wait, through L2 (ld.global.cg,
// cp.async.cg).  Every CTA of the grid is resident at once (one per SM), so
// the wait for u always ends; it is bounded all the same (QN_DEV_TIMEOUT).
// The last CTA to leave returns both counters to zero.
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace qn {

constexpr int kGvWarps = 16;
constexpr int kGvThreads = kGvWarps * 32;
constexpr int kGvRing = 6;                          // stage slots (kGvRing - 1 in flight)
constexpr int kGvStageBlocks = 32;                  // 64-blocks per stage (2048 columns)
constexpr uint32_t kGvStageBytes = 16 * kGvStageBlocks * 32;  // 16 KiB of codes
constexpr int kGvMaxM = 8;
constexpr int kGvMaxGroup = 8;
constexpr int kGvMaxXElems = 16384;                 // M * k staged in the table rows
constexpr uint32_t kGvLutBytes = 256 * 256;         // entry b of lane l at 256 b + 4 l; bytes 128..255 of each row hold x
constexpr int kGvMaxURows = 4;                      // adapter rows per CTA
constexpr int kGvUVec = 2;                          // 16-byte A loads per lane in flight
constexpr int kGvMaxU = 2048;                       // M * (adapter rows of the group)
constexpr uint32_t kGvSmemCap = 227 * 1024;
constexpr int64_t kGvPrefetchBytes = (kGvRing - 1) * static_cast<int64_t>(kGvStageBytes);  // before the wait
constexpr unsigned kGvSpinLimit = 1u << 20;         // polls of the ready counter (128 ns apart)
constexpr int kGvFlagReady = 0, kGvFlagExit = 1;    // zero-area words

struct GvProj {
  const uint8_t *codes;
  const void *consts;          // int8 DQ codes (dq) or fp32 block constants
  const float *absmax_scale;   // DQ group scales (dq)
  const float *absmax_mean;    // DQ mean (dq)
  const uint16_t *A;           // r x k bf16
  const uint16_t *B;           // d x r bf16
  uint16_t *Y;                 // M x d bf16
  int64_t d;
  int64_t row_off;             // first row of this projection in the group's row list
  int64_t u_off;               // first adapter row of this projection
  int r, dq;
  float s;
};

struct GvGroup {
  GvProj p[kGvMaxGroup];
  int n, M;
  int64_t k, rows, rtot;       // shared k, total rows, total adapter rows
  const uint16_t *X;           // M x k bf16
  float *u;                    // M x rtot fp32 (workspace)
  unsigned int *zero_area;     // ready and exit counters, zero between calls
  // shared-memory layout: byte offsets from the start of dynamic shared memory (gv_plan)
  uint32_t off_ring, off_raw, off_sig, off_rows, off_mw, off_part, off_rsum, off_us, off_ured, off_meta, smem;
  int rows_cta;                // largest row range of a CTA
  int bvec;                    // every r is a multiple of 8: B rows read in 16-byte pieces
};

// A CTA's rows of one projection, with where its block constants and DQ
// scales sit in shared memory.  Each copy covers the 16-byte-aligned superset
// of the bytes it needs: [g0, g0 + len) of the source array.
struct GvSeg {
  int p, lr0, lr1;             // projection; CTA-local rows [lr0, lr1)
  int64_t ra;                  // projection row of lr0
  int64_t raw_g0, sig_g0;
  uint32_t raw_off, sig_off, raw_len, sig_len;  // shared addresses and byte counts
};
// One row of a CTA's range, or a padding row of its last tile (dq == -1; it
// points at the range's first row).
struct GvRow {
  const uint8_t *code;         // the row's packed codes
  uint32_t raw;                // shared address of the row's first block constant
  uint32_t sig;                // shared address of the DQ scale of the row's first block
  int prow;                    // row within its projection
  short e0;                    // (first block of the row) mod 256: its place in its DQ group
  signed char p;               // projection
  signed char dq;              // 1: DQ constants, 0: fp32 constants, -1: padding row
};
struct GvMeta {
  GvSeg seg[kGvMaxGroup];
  GvProj p[kGvMaxGroup];
  float mu[kGvMaxGroup];
  int nseg;
};

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ uint4 ld_cg_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_cg_v2(const void *p) {
  uint2 v;
  asm volatile("ld.global.cg.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_cg_f32(const float *p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_cg_u16(const uint16_t *p) {
  unsigned short v;
  asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ unsigned int gv_ld_acquire(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// 16-byte cp.async that reads `src_bytes` (1..16) and zero-fills the rest.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void gv_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds_v2(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds_v2_off8k(uint32_t a) {  // 8 rows of a stage further
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2+8192];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
// Shared address where dynamic shared memory starts for a kernel without
// static shared memory (the level table sits there; checked on the host once
// per device and by the kernel itself).
constexpr uint32_t kGvSmemBase = 1024;
__device__ __forceinline__ uint32_t lds_lut(uint32_t off) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1+1024];" : "=r"(v) : "r"(off));
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_f32_off32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1+32];" : "=f"(v) : "r"(a));
  return v;
}
// Table offset of byte `sel` of `w` for this lane: (byte << 8) | (lane << 2).
__device__ __forceinline__ uint32_t gv_lut_off(uint32_t w, uint32_t lane4, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(w), "r"(lane4), "r"(sel));
  return r;
}
// Offset (within the table region) of 16-byte chunk c of the staged X, token
// t: chunks live in the odd halves of the table rows, xor-swizzled by token
// so that eight tokens' chunks at the same column hit different banks.
__device__ __forceinline__ uint32_t gv_x_chunk(uint32_t c, uint32_t t) {
  const uint32_t cs = c ^ (t & 7u);
  return ((cs >> 3) << 8) + 128u + ((cs & 7u) << 4);
}


// Layout of one launch (host side).  False if the group does not fit.
inline bool gv_plan(GvGroup &g, int grid, int esz_max, bool any_dq) {
  const int64_t k = g.k, nb = k >> 6;
  const int64_t rows_cta = qn_ceil_div(g.rows, grid);
  const int64_t ntl = qn_ceil_div(rows_cta, 16);
  const int M = g.M, n = g.n;
  if (M < 1 || M > kGvMaxM || static_cast<int64_t>(M) * k > kGvMaxXElems) return false;
  if (g.rtot > static_cast<int64_t>(kGvMaxURows) * grid || g.rtot * M > kGvMaxU) return false;
  g.bvec = 1;
  for (int i = 0; i < n; ++i)
    if (g.p[i].r % 8) g.bvec = 0;
  auto a16 = [](int64_t v) { return (v + 15) & ~int64_t{15}; };
  int64_t off = kGvLutBytes;
  g.off_ring = static_cast<uint32_t>(off);
  off += static_cast<int64_t>(kGvRing) * kGvStageBytes;
  g.off_raw = static_cast<uint32_t>(off);
  off += a16(rows_cta * nb * esz_max + 32 * n);
  g.off_sig = static_cast<uint32_t>(off);
  off += any_dq ? a16((rows_cta * nb / 256 + 2 + 8) * 4 * n) : 0;
  g.off_rows = static_cast<uint32_t>(off);
  off += a16(ntl * 16 * static_cast<int64_t>(sizeof(GvRow)));
  g.off_mw = static_cast<uint32_t>(off);
  off += static_cast<int64_t>(kGvWarps) * 32 * 4;
  g.off_part = static_cast<uint32_t>(off);
  off += a16(2LL * kGvWarps * 16 * M * 4);
  g.off_rsum = static_cast<uint32_t>(off);
  off += a16(ntl * 16 * M * 4);
  g.off_us = static_cast<uint32_t>(off);
  off += a16(g.rtot * M * 4);
  g.off_ured = static_cast<uint32_t>(off);
  off += a16(static_cast<int64_t>(kGvMaxURows) * kGvWarps * M * 4);
  g.off_meta = static_cast<uint32_t>(off);
  off += a16(sizeof(GvMeta));
  if (off > kGvSmemCap) return false;
  g.smem = static_cast<uint32_t>(off);
  g.rows_cta = static_cast<int>(rows_cta);
  return true;
}

// Shared-memory offset of byte x (0..1023) of row r (0..15) of a stage: the
// 16-byte pieces of each 128-byte span are xor-swizzled by r mod 8, so the
// 8-byte reads of rows g (and g + 8) of one column by eight lane groups hit
// different banks.
__device__ __forceinline__ uint32_t gv_stage_off(uint32_t r, uint32_t x) {
  return r * 1024u + (x & ~127u) + ((((x >> 4) & 7u) ^ (r & 7u)) << 4) + (x & 15u);
}

// Copies [g0, g0 + len) of an array of `size` bytes to shared memory (16-byte
// pieces, the piece that crosses the end of the array zero-filled).
__device__ __forceinline__ void gv_copy(uint32_t dst, const void *base, int64_t g0, uint32_t len, int64_t size) {
  const char *src = static_cast<const char *>(base) + g0;
  const int64_t avail = size - g0;
  for (uint32_t c = threadIdx.x * 16u; c < len; c += kGvThreads * 16u) {
    const int64_t left = avail - c;
    cp_async16_zfill(dst + c, src + c, static_cast<uint32_t>(left < 16 ? left : 16));
  }
}
__device__ __forceinline__ void gv_prefetch(const void *base, int64_t g0, int64_t len, int64_t size) {
  int64_t end = g0 + len;
  if (end > (size & ~int64_t{15})) end = size & ~int64_t{15};
  const char *src = static_cast<const char *>(base);
  for (int64_t o = g0; o < end; o += 32768) {
    const int64_t l = (end - o < 32768) ? end - o : 32768;
    prefetch_l2_bulk(src + o, static_cast<uint32_t>(l));
  }
}


template <int MT>
__global__ void __launch_bounds__(kGvThreads, 1)
qlora_gemv_kernel(const __grid_constant__ GvGroup g) {
  extern __shared__ __align__(1024) unsigned char gv_raw[];
  pdl_trigger();  // the next call may launch as soon as SMs free up
  // The level table is addressed with an immediate offset: the window must
  // start where the host's probe found it.
  if (smem_u32(gv_raw) != kGvSmemBase) {
    if (threadIdx.x == 0) atomicOr(&g_qn_status, QN_DEV_LAYOUT);
    return;
  }
  unsigned char *base = gv_raw;
  const uint32_t sb = kGvSmemBase;
  GvMeta &mt = *reinterpret_cast<GvMeta *>(base + g.off_meta);
  GvRow *rows = reinterpret_cast<GvRow *>(base + g.off_rows);
  float *part = reinterpret_cast<float *>(base + g.off_part);
  float *rsum = reinterpret_cast<float *>(base + g.off_rsum);
  float *us = reinterpret_cast<float *>(base + g.off_us);
  float *ured = reinterpret_cast<float *>(base + g.off_ured);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int64_t k = g.k, kh = k >> 1;
  const int nb = static_cast<int>(k >> 6);
  const int M = g.M;
  const int G = gridDim.x;
  const int64_t R0 = g.rows * blockIdx.x / G, R1 = g.rows * (blockIdx.x + 1) / G;
  const int nrows = static_cast<int>(R1 - R0);
  const int ntl = (nrows + 15) >> 4;
  const int nch = (nb + kGvStageBlocks - 1) / kGvStageBlocks;  // stages per tile
  const int nst = ntl * nch;
  const int64_t rtot = g.rtot;
  const int nu = static_cast<int>((rtot - blockIdx.x + G - 1) / G);  // adapter rows of this CTA (j = blockIdx + G i)

  // ---- before the wait: segments, L2 prefetch, level table, row table ------------
  if (tid == 0) {
    int ns = 0;
    uint32_t raw = sb + g.off_raw, sig = sb + g.off_sig;
    for (int i = 0; i < g.n; ++i) mt.p[i] = g.p[i];
    for (int iu = 0; iu < nu; ++iu) {  // A rows of this CTA's adapter rows
      const int64_t j = blockIdx.x + static_cast<int64_t>(G) * iu;
      int pi = 0;
      for (int i = 1; i < g.n; ++i)
        if (j >= g.p[i].u_off) pi = i;
      gv_prefetch(g.p[pi].A, (j - g.p[pi].u_off) * k * 2, k * 2, static_cast<int64_t>(g.p[pi].r) * k * 2);
    }
    // the first stages' rows
    const int pre_rows = 16 * ((kGvRing - 1 + nch - 1) / nch);
    for (int i = 0; i < g.n; ++i) {
      const GvProj &p = g.p[i];
      const int64_t a = R0 > p.row_off ? R0 : p.row_off;
      const int64_t e = R1 < p.row_off + p.d ? R1 : p.row_off + p.d;
      if (a >= e) continue;
      GvSeg &s = mt.seg[ns++];
      s.p = i;
      s.lr0 = static_cast<int>(a - R0);
      s.lr1 = static_cast<int>(e - R0);
      s.ra = a - p.row_off;
      const int64_t nr = e - a;
      const int esz = p.dq ? 1 : 4;
      const int64_t b0 = s.ra * nb * esz, b1 = (s.ra + nr) * nb * esz;
      s.raw_g0 = b0 & ~int64_t{15};
      s.raw_len = static_cast<uint32_t>(((b1 + 15) & ~int64_t{15}) - s.raw_g0);
      s.raw_off = raw;
      raw += s.raw_len;
      if (p.dq) {  // DQ group scales: floats [f0, f1]
        const int64_t f0 = (s.ra * nb) >> 8, f1 = ((s.ra + nr) * nb - 1) >> 8;
        s.sig_g0 = (f0 * 4) & ~int64_t{15};
        s.sig_len = static_cast<uint32_t>((((f1 + 1) * 4 + 15) & ~int64_t{15}) - s.sig_g0);
      } else {
        s.sig_g0 = 0;
        s.sig_len = 0;
      }
      s.sig_off = sig;
      sig += s.sig_len;
      gv_prefetch(p.consts, s.raw_g0, s.raw_len, p.d * nb * esz);
      if (p.dq) gv_prefetch(p.absmax_scale, s.sig_g0, s.sig_len, ((p.d * nb + 255) >> 8) * 4);
      gv_prefetch(p.B, (s.ra * p.r * 2) & ~int64_t{15}, nr * p.r * 2 + 16, p.d * p.r * 2);
      const int64_t pr = pre_rows - s.lr0;
      if (pr > 0) gv_prefetch(p.codes, s.ra * kh, (pr < nr ? pr : nr) * kh, p.d * kh);
    }
    mt.nseg = ns;
  }
  // table entry b of lane l: bf16(level[b & 15]) | bf16(level[b >> 4]) << 16
  for (int e = tid; e < 256 * 32; e += kGvThreads) {
    const int b = e >> 5;
    *reinterpret_cast<uint32_t *>(base + b * 256 + (e & 31) * 4) =
        pack_bf16x2(c_nf4_levels[b & 15], c_nf4_levels[b >> 4]);
  }
  __syncthreads();
  for (int lr = tid; lr < ntl * 16; lr += kGvThreads) {
    // padding rows of the last tile read the first row's codes (their block
    // constants are 0)
    const bool pad = lr >= nrows;
    const int lq = pad ? 0 : lr;
    int si = 0;
    for (int i = 1; i < mt.nseg; ++i)
      if (lq >= mt.seg[i].lr0) si = i;
    const GvSeg &s = mt.seg[si];
    const GvProj &p = mt.p[s.p];
    const int64_t prow = s.ra + (lq - s.lr0);
    const int64_t e0 = prow * nb;  // first block of the row
    GvRow rw;
    rw.code = p.codes + prow * kh;
    rw.prow = static_cast<int>(prow);
    rw.p = static_cast<signed char>(s.p);
    rw.dq = pad ? static_cast<signed char>(-1) : static_cast<signed char>(p.dq);
    rw.e0 = static_cast<short>(e0 & 255);
    rw.raw = s.raw_off + static_cast<uint32_t>(e0 * (p.dq ? 1 : 4) - s.raw_g0);
    rw.sig = p.dq ? s.sig_off + static_cast<uint32_t>((e0 >> 8) * 4 - s.sig_g0) : 0u;
    rows[lr] = rw;
  }
  __syncthreads();
  pdl_wait_grid();

  // ---- after the wait: small copies (one group), then the first stages ----------
  const uint32_t kc = static_cast<uint32_t>(k >> 3);  // 16-byte chunks per token
  for (int t = 0; t < M; ++t)
    for (uint32_t v = tid; v < kc; v += kGvThreads)
      cp_async16(sb + gv_x_chunk(t * kc + v, t), g.X + static_cast<int64_t>(t) * k + v * 8);
  for (int i = 0; i < mt.nseg; ++i) {
    const GvSeg &s = mt.seg[i];
    const GvProj &p = mt.p[s.p];
    gv_copy(s.raw_off, p.consts, s.raw_g0, s.raw_len, p.d * nb * (p.dq ? 1 : 4));
    if (p.dq) gv_copy(s.sig_off, p.absmax_scale, s.sig_g0, s.sig_len, ((p.d * nb + 255) >> 8) * 4);
  }
  cp_async_commit();
  // Stage s (tile s / nch, chunk s % nch) into slot s % kGvRing: thread i
  // copies 16-byte pieces i and i + 512 of the stage (row = piece / 64).
  const uint32_t ring = sb + g.off_ring;
  auto issue_stage = [&](int s) {
    if (s < nst) {
      const int tl = s / nch, ch = s - tl * nch;
      const int cbl = (nb - ch * kGvStageBlocks) < kGvStageBlocks ? nb - ch * kGvStageBlocks : kGvStageBlocks;
      const uint32_t slot = ring + static_cast<uint32_t>(s % kGvRing) * kGvStageBytes;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int pc = tid + h * kGvThreads;  // piece 0..1023
        const int r = pc >> 6, x = (pc & 63) << 4;
        if (x < cbl * 32)
          cp_async16(slot + gv_stage_off(r, x), rows[tl * 16 + r].code + ch * (kGvStageBlocks * 32) + x);
      }
    }
    cp_async_commit();
  };
#pragma unroll 1
  for (int s = 0; s < kGvRing - 1; ++s) issue_stage(s);
  // adapter rows of this CTA: warp slice [v0, v1) of the k / 8 vectors
  const int v0 = static_cast<int>(kc * warp / kGvWarps), v1 = static_cast<int>(kc * (warp + 1) / kGvWarps);
  uint4 av[kGvUVec];
  auto load_a = [&](int iu, int bt) {
    const int64_t j = blockIdx.x + static_cast<int64_t>(G) * iu;
    int pi = 0;
    for (int i = 1; i < g.n; ++i)
      if (j >= mt.p[i].u_off) pi = i;
    const uint16_t *arow = mt.p[pi].A + (j - mt.p[pi].u_off) * k;
#pragma unroll
    for (int i = 0; i < kGvUVec; ++i) {
      const int v = v0 + lane + 32 * (bt * kGvUVec + i);
      av[i] = (v < v1) ? ld_cg_v4(arow + static_cast<int64_t>(v) * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  if (nu > 0) load_a(0, 0);
  if (tid < g.n) mt.mu[tid] = mt.p[tid].dq ? ld_cg_f32(mt.p[tid].absmax_mean) : 0.f;
  cp_async_wait_group<kGvRing - 1>();  // the small copies
  __syncthreads();

  {
    const int span = v1 - v0;
    const int nbt = span > 0 ? (span + 32 * kGvUVec - 1) / (32 * kGvUVec) : 1;
    for (int iu = 0; iu < nu; ++iu) {
      float ua[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) ua[t] = 0.f;
      for (int bt = 0; bt < nbt; ++bt) {
        if (iu > 0 || bt > 0) load_a(iu, bt);
#pragma unroll
        for (int i = 0; i < kGvUVec; ++i) {
          const int v = v0 + lane + 32 * (bt * kGvUVec + i);
          if (v >= v1) continue;
          const uint32_t aw[4] = {av[i].x, av[i].y, av[i].z, av[i].w};
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            if (t >= M) break;
            const uint4 xq = lds_v4(sb + gv_x_chunk(t * kc + static_cast<uint32_t>(v), t));
            const uint32_t xw[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              ua[t] = fmaf(__uint_as_float(aw[c] << 16), __uint_as_float(xw[c] << 16), ua[t]);
              ua[t] = fmaf(__uint_as_float(aw[c] & 0xFFFF0000u), __uint_as_float(xw[c] & 0xFFFF0000u), ua[t]);
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < MT; ++t) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ua[t] += __shfl_xor_sync(0xffffffffu, ua[t], off);
      }
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < MT; ++t)
          if (t < M) ured[(iu * kGvWarps + warp) * M + t] = ua[t];
      }
    }
  }
  __syncthreads();
  if (warp == 0 && nu > 0) {
    // warp 0 finishes this CTA's adapter rows; the other warps go on
    if (lane < nu * M) {
      const int iu = lane / M, t = lane - iu * M;
      const int64_t j = blockIdx.x + static_cast<int64_t>(G) * iu;
      int pi = 0;
      for (int i = 1; i < g.n; ++i)
        if (j >= mt.p[i].u_off) pi = i;
      float v = 0.f;
      for (int w = 0; w < kGvWarps; ++w) v += ured[(iu * kGvWarps + w) * M + t];
      g.u[t * rtot + j] = mt.p[pi].s * v;
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      atomicAdd(&g.zero_area[kGvFlagReady], static_cast<unsigned>(nu));
    }
  }

  // ---- weight loop: one barrier per stage ---------------------------------------
  float *mw = reinterpret_cast<float *>(base + g.off_mw) + warp * 32;  // [block 0/1][16 rows]
  const uint32_t mw_s = smem_u32(mw) + static_cast<uint32_t>(gq) * 4u;
  const uint32_t lane4 = static_cast<uint32_t>(lane) << 2;
  const uint32_t xb0 = sb + gv_x_chunk(gq * kc + 2u * tq, gq);
  const uint32_t xb1 = sb + gv_x_chunk(gq * kc + 2u * tq + 1u, gq);
  // tile sums: warp tl mod 16 adds the 16 warps' partials of tile tl in warp order
  auto reduce_tile = [&](int tl) {
    const float *pb = part + (tl & 1) * (kGvWarps * 16 * M);
    for (int e = lane; e < 16 * M; e += 32) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kGvWarps; ++w) v += pb[w * 16 * M + e];
      rsum[tl * 16 * M + e] = v;
    }
  };
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int s = 0; s < nst; ++s) {
    cp_async_wait_group<kGvRing - 2>();  // this thread's pieces of stage s
    __syncthreads();                     // every piece of stage s; the slot of stage s - 1 is free
    issue_stage(s + kGvRing - 1);
    const int tl = s / nch, ch = s - tl * nch;
    const int cbl = (nb - ch * kGvStageBlocks) < kGvStageBlocks ? nb - ch * kGvStageBlocks : kGvStageBlocks;
    if (ch == 0 && tl > 0 && warp == ((tl - 1) & (kGvWarps - 1))) reduce_tile(tl - 1);
    {
      // block constant of row lane mod 16, block warp + 16 (lane / 16) of this stage
      const int rr = lane & 15, blk = warp + 16 * (lane >> 4);
      const GvRow &rw = rows[tl * 16 + rr];
      float m = 0.f;
      if (blk < cbl && rw.dq >= 0) {
        const int b = ch * kGvStageBlocks + blk;
        if (rw.dq) {
          const int8_t q = *reinterpret_cast<const int8_t *>(base + (rw.raw - kGvSmemBase) + b);
          const float sg = *reinterpret_cast<const float *>(base + (rw.sig - kGvSmemBase) + ((rw.e0 + b) >> 8) * 4);
          m = dq_absmax(q, sg, mt.mu[rw.p]);
        } else {
          m = *reinterpret_cast<const float *>(base + (rw.raw - kGvSmemBase) + b * 4);
        }
      }
      __syncwarp();
      mw[(lane >> 4) * 16 + rr] = m;
      __syncwarp();
    }
    const uint32_t slot = ring + static_cast<uint32_t>(s % kGvRing) * kGvStageBytes;
#pragma unroll
    for (int bi = 0; bi < 2; ++bi) {
      const int blk = warp + 16 * bi;
      if (blk >= cbl) break;
      const uint32_t ca = slot + gv_stage_off(static_cast<uint32_t>(gq), static_cast<uint32_t>(blk * 32 + tq * 8));
      const uint2 c0 = lds_v2(ca), c1 = lds_v2_off8k(ca);
      uint32_t a0[8], a1[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t sel = 0x5504u | (static_cast<uint32_t>(i) << 4);
        a0[i] = lds_lut(gv_lut_off(c0.x, lane4, sel));
        a0[4 + i] = lds_lut(gv_lut_off(c0.y, lane4, sel));
        a1[i] = lds_lut(gv_lut_off(c1.x, lane4, sel));
        a1[4 + i] = lds_lut(gv_lut_off(c1.y, lane4, sel));
      }
      uint4 x0 = make_uint4(0u, 0u, 0u, 0u), x1 = x0;
      if (gq < M) {
        const uint32_t xo = static_cast<uint32_t>(ch * kGvStageBlocks + blk) << 8;
        x0 = lds_v4(xb0 + xo);
        x1 = lds_v4(xb1 + xo);
      }
      float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
      gv_mma(d0, a0[0], a1[0], a0[1], a1[1], x0.x, x0.y);
      gv_mma(d1, a0[2], a1[2], a0[3], a1[3], x0.z, x0.w);
      gv_mma(d0, a0[4], a1[4], a0[5], a1[5], x1.x, x1.y);
      gv_mma(d1, a0[6], a1[6], a0[7], a1[7], x1.z, x1.w);
      const uint32_t mo = mw_s + static_cast<uint32_t>(bi) * 64u;
      const float m0 = lds_f32(mo), m1 = lds_f32_off32(mo);
      acc[0] = fmaf(d0[0] + d1[0], m0, acc[0]);
      acc[1] = fmaf(d0[1] + d1[1], m0, acc[1]);
      acc[2] = fmaf(d0[2] + d1[2], m1, acc[2]);
      acc[3] = fmaf(d0[3] + d1[3], m1, acc[3]);
    }
    if (ch == nch - 1) {
      // end of tile tl: this warp's partial sums
      float *pw = part + (tl & 1) * (kGvWarps * 16 * M) + warp * 16 * M;
      if (2 * tq < M) {
        pw[gq * M + 2 * tq] = acc[0];
        pw[(gq + 8) * M + 2 * tq] = acc[2];
      }
      if (2 * tq + 1 < M) {
        pw[gq * M + 2 * tq + 1] = acc[1];
        pw[(gq + 8) * M + 2 * tq + 1] = acc[3];
      }
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    }
  }
  cp_async_wait_all();

  // ---- adapter terms and output -------------------------------------------------
  // Thread lr takes row lr of the range: the first 64 values of its B row are
  // loaded (16-byte pieces) before the wait for u, so both round trips overlap.
  const bool bvec = g.bvec != 0;  // every r a multiple of 8 (rows of B 16-byte aligned)
  uint4 bq[8];
  if (bvec && tid < nrows) {
    const GvRow &rw = rows[tid];
    const GvProj &p = mt.p[rw.p];
    const uint16_t *br = p.B + static_cast<int64_t>(rw.prow) * p.r;
#pragma unroll
    for (int c = 0; c < 8; ++c) bq[c] = (8 * c < p.r) ? ld_cg_v4(br + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();  // every partial sum written
  if (ntl > 0 && warp == ((ntl - 1) & (kGvWarps - 1))) reduce_tile(ntl - 1);
  if (tid == 0) {
    unsigned int spins = 0;
    while (gv_ld_acquire(&g.zero_area[kGvFlagReady]) < static_cast<unsigned>(rtot)) {
      if (++spins > kGvSpinLimit) {
        qn_flag_timeout();
        break;
      }
      __nanosleep(128);
    }
    __threadfence();
  }
  __syncthreads();
  for (int e = tid; e < rtot * M; e += kGvThreads) us[e] = ld_cg_f32(g.u + e);
  __syncthreads();
  // Y = row sum + u . B[row]
  for (int lr = tid; lr < nrows; lr += kGvThreads) {
    const GvRow &rw = rows[lr];
    const GvProj &p = mt.p[rw.p];
    const uint16_t *br = p.B + static_cast<int64_t>(rw.prow) * p.r;
    const float *ur = us + p.u_off;
    float a[MT][2];
#pragma unroll
    for (int t = 0; t < MT; ++t) a[t][0] = a[t][1] = 0.f;
    for (int q0 = 0; q0 < p.r; q0 += 64) {
      if (bvec) {
        if (q0 > 0 || lr != tid) {
#pragma unroll
          for (int c = 0; c < 8; ++c)
            bq[c] = (q0 + 8 * c < p.r) ? ld_cg_v4(br + q0 + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          if (q0 + 8 * c >= p.r) break;
          const uint32_t bw[4] = {bq[c].x, bq[c].y, bq[c].z, bq[c].w};
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            const float b = (h & 1) ? __uint_as_float(bw[h >> 1] & 0xFFFF0000u) : __uint_as_float(bw[h >> 1] << 16);
            const int q = q0 + 8 * c + h;
#pragma unroll
            for (int t = 0; t < MT; ++t)
              if (t < M) a[t][h & 1] = fmaf(ur[t * rtot + q], b, a[t][h & 1]);
          }
        }
      } else {
        const int qe = p.r < q0 + 64 ? p.r : q0 + 64;
        for (int q = q0; q < qe; ++q) {
          const float b = bf16_bits_to_f32(ld_cg_u16(br + q));
#pragma unroll
          for (int t = 0; t < MT; ++t)
            if (t < M) a[t][0] = fmaf(ur[t * rtot + q], b, a[t][0]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      if (t >= M) break;
      p.Y[t * p.d + rw.prow] = f32_to_bf16_bits(rsum[lr * M + t] + (a[t][0] + a[t][1]));
    }
  }
  // the last CTA to get here returns the counters to zero
  if (tid == 0) {
    const unsigned int prev = atomicAdd(&g.zero_area[kGvFlagExit], 1u);
    if (prev == static_cast<unsigned>(G) - 1u) {
      atomicExch(&g.zero_area[kGvFlagReady], 0u);
      atomicExch(&g.zero_area[kGvFlagExit], 0u);
    }
  }
}

}  // namespace qn
