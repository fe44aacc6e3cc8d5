// qlora_gemv.cuh -- fused QLoRA forward for a few tokens (M <= 8, M * k <=
// 16384) of a group of projections that share one input:
//
//   Y_g = X deq(Q_g)^T + s_g (X A_g^T) B_g^T      X: M x k bf16, Q_g: d_g x k NF4
//
// ("PEFT course notes" §2.2, h = Wx + BAx; "QLoRA paper summary": the frozen
// weight is 4-bit NF4 with blockwise constants.)  The call is bound by the
// bytes of the packed weights (8-50 MB at decode sizes).  On this part an SM
// needs ~100 KB of reads in flight to cover HBM latency under load, and
// asynchronous copies into shared memory carry that with no registers, so:
//
// * the group's rows form one list, cut into equal contiguous ranges, one
//   per CTA (one CTA per SM); a range is cut into 16-row tiles and each tile
//   into stages of 16 rows x 4096 columns (32 KiB of codes);
// * a producer warp brings each stage into a ring of 2..8 slots (what the
//   shared memory leaves) with one bulk copy (TMA) per row, counted on
//   the slot's full barrier; rows sit 2080 bytes apart, so the consumers'
//   8-byte reads are conflict-free.  Bulk copies keep the stage traffic out
//   of the load/store pipe that the table lookups need;
// * 16 consumer warps: warp w takes 64-blocks w, w + 16, w + 32, w + 48 of
//   each stage: a lane (group g, thread t) reads 8 code bytes of rows g and
//   g + 8, turns each byte into a bf16x2 pair through a per-lane replicated
//   byte-pair table (one byte permute and one shared load with an immediate
//   base per byte), multiplies on mma.sync m16n8k16 (tokens are the N
//   columns) against x, which is staged as bf16 in the unused half of every
//   table row, and scales each block's dot products by its fp32 block
//   constant (decoded once per CTA into shared memory).  The MMA's k order
//   is a permutation of the block's elements, the same for both operands.
//   A warp arrives on the slot's empty barrier when it is done with it;
// * at the end of a tile each warp writes its partial sums; the output
//   phase adds them in warp order;
// * the adapter rows u = s X A^T are spread over the CTAs (row j by CTA
//   j mod G, split over the 16 warps) before the weight loop and published
//   through a ready counter by the second producer warp; after its copies
//   the first producer warp waits (bounded) for all of them and stages u;
//   then thread i adds u . B[row i] and writes bf16 Y = row sum + adapter
//   term.
//
// Programmatic dependent launch: the kernel lets the next call launch at
// entry; before griddepcontrol.wait a CTA only builds its tables and
// prefetches its A rows into L2 (a prefetch cannot return stale data).
// Everything a kernel may have written -- codes, constants, X, A, B, u, Y,
// the counters -- is read after the wait, through L2 (ld.global.cg,
// cp.async.cg, bulk copies).  Every CTA of the grid is resident at once (one
// per SM), so the wait for u always ends; it is bounded all the same
// (QN_DEV_TIMEOUT).  The last CTA to leave returns both counters to zero.
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace qn {

constexpr int kGvWarps = 16;                        // consumer warps (MMA)
constexpr int kGvProducers = 64;                    // producer threads (two warps: stage copies, u)
constexpr int kGvThreads = kGvWarps * 32 + kGvProducers;
constexpr int kGvMaxRing = 8;                       // stage slots at most (the plan picks what fits)
constexpr int kGvStageBlocks = 64;                  // 64-blocks per stage (4096 columns)
constexpr uint32_t kGvStageRow = kGvStageBlocks * 32;  // code bytes of one row in a stage
constexpr uint32_t kGvRowPitch = kGvStageRow + 32;    // shared-memory bytes per row: 32 bytes of padding
constexpr uint32_t kGvStageBytes = 16 * kGvRowPitch;  // 32 KiB of codes + padding
static_assert(kGvStageBlocks % 32 == 0, "a warp takes blocks w + 16 j in pairs");
constexpr int kGvMaxM = 8;
constexpr int kGvMaxGroup = 8;
constexpr int kGvMaxXElems = 16384;                 // M * k staged in the table rows
constexpr uint32_t kGvLutBytes = 256 * 256;         // entry b of lane l at 256 b + 4 l; bytes 128..255 of each row hold x
constexpr int kGvMaxURows = 4;                      // adapter rows per CTA
constexpr int kGvUVec = 2;                          // 16-byte A loads per lane in flight
constexpr int kGvMaxU = 2048;                       // M * (adapter rows of the group)
constexpr uint32_t kGvSmemCap = 227 * 1024;
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

struct GvGroup {  // the kernel's parameter block (copied to shared memory at entry)
  GvProj p[kGvMaxGroup];
  int n, M;
  int64_t k, rows, rtot;       // shared k, total rows, total adapter rows
  const uint16_t *X;           // M x k bf16
  float *u;                    // M x rtot fp32 (workspace)
  unsigned int *zero_area;     // ready and exit counters, zero between calls
  // shared-memory layout: byte offsets from the start of dynamic shared memory (gv_plan)
  uint32_t off_ring, off_rows, off_m, off_part, off_us, off_ured, off_bar, smem;
  int rows_cta;                // largest row range of a CTA
  int ring;                    // stage slots
  int ms;                      // row stride (floats, odd) of the decoded block constants
  uint16_t lev16[16];          // bf16 bits of the 16 levels (round to nearest even)
  int bvec;                    // every r is a multiple of 8: B rows read in 16-byte pieces
};

static_assert(sizeof(GvGroup) % 8 == 0, "parameter block copied in 8-byte pieces");

// One row of a CTA's range, or a padding row of its last tile (dq == -1; it
// points at the range's first row).
struct GvRow {
  const uint8_t *code;         // the row's packed codes
  int prow;                    // row within its projection
  signed char p;               // projection
  signed char dq;              // 1: DQ constants, 0: fp32 constants, -1: padding row
};
constexpr int kGvDecRows = 6;  // rows whose block constants a thread loads at once

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
__device__ __forceinline__ float ld_cg_f32(const float *p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_cg_u32(const void *p) {
  uint32_t v;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_cg_s8(const void *p) {  // sign-extended
  int v;
  asm volatile("ld.global.cg.s8 %0, [%1];" : "=r"(v) : "l"(p));
  return static_cast<uint32_t>(v);
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
__device__ __forceinline__ void gv_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint2 lds_v2(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds_v2_off8r(uint32_t a) {  // 8 rows of a stage further
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2+16640];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
static_assert(8 * kGvRowPitch == 16640, "immediate offset of lds_v2_off8r");
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


// Layout of one launch (host side): the stage ring gets what the rest
// leaves of the shared memory, 2..kGvMaxRing slots.  False if the group does
// not fit.
inline bool gv_plan(GvGroup &g, int grid) {
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
  g.ms = static_cast<int>(nb | 1);
  int64_t off = kGvLutBytes + a16(sizeof(GvGroup));  // the table, then a copy of this block
  g.off_rows = static_cast<uint32_t>(off);
  off += a16(ntl * 16 * static_cast<int64_t>(sizeof(GvRow)));
  g.off_m = static_cast<uint32_t>(off);
  off += a16(ntl * 16 * g.ms * 4);
  g.off_part = static_cast<uint32_t>(off);
  off += a16(ntl * kGvWarps * 16 * M * 4);
  g.off_us = static_cast<uint32_t>(off);
  off += a16(g.rtot * M * 4);
  g.off_ured = static_cast<uint32_t>(off);
  off += a16(static_cast<int64_t>(kGvMaxURows) * kGvWarps * M * 4);
  g.off_bar = static_cast<uint32_t>(off);
  off += a16(2 * kGvMaxRing * 8 + 16);
  off = (off + 1023) & ~int64_t{1023};
  const int64_t room = (static_cast<int64_t>(kGvSmemCap) - off) / kGvStageBytes;
  if (room < 2) return false;
  g.ring = static_cast<int>(room < kGvMaxRing ? room : kGvMaxRing);
  g.off_ring = static_cast<uint32_t>(off);
  g.smem = static_cast<uint32_t>(off + static_cast<int64_t>(g.ring) * kGvStageBytes);
  g.rows_cta = static_cast<int>(rows_cta);
  return true;
}

// A stage holds row r (0..15) at r * kGvRowPitch.  The 32 bytes of padding
// per row shift consecutive rows by eight banks, so the 8-byte reads of rows
// g = 0..3 (and 4..7) by the four lanes of each group cover all 32 banks once
// per half-warp: conflict-free.

// Bulk L2 prefetch of [g0, g0 + len) of an array of `size` bytes (g0 and len
// multiples of 16; the range is cut at the last whole 16 bytes of the array).
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
qlora_gemv_kernel(const __grid_constant__ GvGroup gp) {
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
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t *full = reinterpret_cast<uint64_t *>(base + gp.off_bar);  // [kGvMaxRing]: a stage has landed
  uint64_t *empty = full + kGvMaxRing;                                // [kGvMaxRing]: every warp is done with it
  uint64_t *upart = empty + kGvMaxRing;                               // the consumers' parts of u are written
  volatile int *abort = reinterpret_cast<volatile int *>(upart + 1);
  {
    // The parameter block into shared memory: one parallel read instead of a
    // chain of constant-cache misses over its ~900 bytes.  The level table and
    // the barriers need none of it and are set up meanwhile.
    const uint2 *src = reinterpret_cast<const uint2 *>(&gp);
    uint2 *dst = reinterpret_cast<uint2 *>(base + kGvLutBytes);
    for (int i = tid; i < static_cast<int>(sizeof(GvGroup) / 8); i += kGvThreads) dst[i] = src[i];
  }
  if (tid < 256) {
    // table entry b: bf16(level[b & 15]) | bf16(level[b >> 4]) << 16, written by
    // thread b into all 32 lane slots of row b (16-byte stores in a rotated
    // order, so that eight neighbouring threads hit different banks)
    const uint32_t lv = gp.lev16[lane & 15];
    const uint32_t v = __shfl_sync(0xffffffffu, lv, tid & 15) | (__shfl_sync(0xffffffffu, lv, tid >> 4) << 16);
    const uint4 v4 = make_uint4(v, v, v, v);
#pragma unroll
    for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4 *>(base + tid * 256 + 16 * ((q + tid) & 7)) = v4;
  }
  if (warp == 9 && lane == 0) {
    for (int i = 0; i < kGvMaxRing; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kGvWarps);
    }
    mbar_init(smem_u32(upart), 1);
    *abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const GvGroup &g = *reinterpret_cast<const GvGroup *>(base + kGvLutBytes);
  GvRow *rows = reinterpret_cast<GvRow *>(base + g.off_rows);
  float *part = reinterpret_cast<float *>(base + g.off_part);
  float *mconst = reinterpret_cast<float *>(base + g.off_m);
  float *us = reinterpret_cast<float *>(base + g.off_us);
  float *ured = reinterpret_cast<float *>(base + g.off_ured);

  const int gq = lane >> 2, tq = lane & 3;
  const int64_t k = g.k, kh = k >> 1;
  const int nb = static_cast<int>(k >> 6);
  const int M = g.M;
  const int G = gridDim.x;
  int64_t R0, R1;  // this CTA's rows [R0, R1) of the group's list
  if (g.rows < (int64_t{1} << 24)) {
    const uint32_t rr = static_cast<uint32_t>(g.rows);
    R0 = rr * blockIdx.x / static_cast<uint32_t>(G);
    R1 = rr * (blockIdx.x + 1) / static_cast<uint32_t>(G);
  } else {
    R0 = g.rows * blockIdx.x / G;
    R1 = g.rows * (blockIdx.x + 1) / G;
  }
  const int nrows = static_cast<int>(R1 - R0);
  const int ntl = (nrows + 15) >> 4;
  const int nch = (nb + kGvStageBlocks - 1) / kGvStageBlocks;  // stages per tile
  const int nst = ntl * nch;
  const int64_t rtot = g.rtot;
  const int nu = static_cast<int>((rtot - blockIdx.x + G - 1) / G);  // adapter rows of this CTA (j = blockIdx + G i)

  // ---- before the wait: row table, L2 prefetch of A ------------------------------------
  if (tid >= 32 && tid < 32 + nu) {  // A rows of this CTA's adapter rows into L2
    const int64_t j = blockIdx.x + static_cast<int64_t>(G) * (tid - 32);
    int pi = 0;
    for (int i = 1; i < g.n; ++i)
      if (j >= g.p[i].u_off) pi = i;
    gv_prefetch(g.p[pi].A, (j - g.p[pi].u_off) * k * 2, k * 2, static_cast<int64_t>(g.p[pi].r) * k * 2);
  }
  for (int lr = tid; lr < ntl * 16; lr += kGvThreads) {
    // a padding row of the last tile points at the range's first row (its
    // codes are not copied and its block constants are 0)
    const bool pad = lr >= nrows;
    const int64_t R = R0 + (pad ? 0 : lr);
    int pi = 0;
#pragma unroll
    for (int i = 1; i < kGvMaxGroup; ++i)
      if (i < g.n && R >= g.p[i].row_off) pi = i;
    const GvProj &p = g.p[pi];
    const int prow = static_cast<int>(R - p.row_off);
    GvRow rw;
    rw.code = p.codes + prow * kh;
    rw.prow = prow;
    rw.p = static_cast<signed char>(pi);
    rw.dq = pad ? static_cast<signed char>(-1) : static_cast<signed char>(p.dq);
    rows[lr] = rw;
  }
  __syncthreads();
  pdl_wait_grid();

  // ---- after the wait -----------------------------------------------------------
  const uint32_t kc = static_cast<uint32_t>(k >> 3);  // 16-byte chunks per token
  const uint32_t ring = sb + g.off_ring;
  const int R = g.ring;
  if (warp >= kGvWarps) {
    // ================================ producers =================================
    if (warp == kGvWarps + 1) {
      // The second producer warp adds the consumers' parts of this CTA's
      // adapter rows (in warp order) and publishes them.
      bool got = false;
      if (nu > 0 && lane == 0) got = mbar_wait(smem_u32(upart), 0, abort);
      __syncwarp();
      if (__shfl_sync(0xffffffffu, got, 0)) {
        if (lane < nu * M) {
          const int iu = lane / M, t = lane - iu * M;
          const int64_t j = blockIdx.x + static_cast<int64_t>(G) * iu;
          int pi = 0;
          for (int i = 1; i < g.n; ++i)
            if (j >= g.p[i].u_off) pi = i;
          float v = 0.f;
          for (int w = 0; w < kGvWarps; ++w) v += ured[(iu * kGvWarps + w) * M + t];
          g.u[t * rtot + j] = g.p[pi].s * v;
        }
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          atomicAdd(&g.zero_area[kGvFlagReady], static_cast<unsigned>(nu));
        }
      }
    } else {
      // Stages in order (tile, chunk) into slots 0, 1, ... R - 1, 0, ...: lane r
      // issues the bulk copy of row r of the tile (padding rows are not copied:
      // their block constants are 0), counted on the slot's full barrier after
      // lane 0 has announced the stage's bytes.
      int tl = 0, ch = 0, s = 0;
      const uint8_t *rowp = lane < 16 && lane < nrows ? rows[lane].code : nullptr;
      // The consumers' small copies (x, block constants, A) go out first.
      asm volatile("bar.sync 2, %0;" ::"n"((kGvWarps + 1) * 32) : "memory");
      for (; s < nst; ++s) {
        const int slot = s % R;
        if (s >= R) {
          bool free_ = false;
          if (lane == 0) free_ = mbar_wait(smem_u32(&empty[slot]), ((s / R) - 1) & 1, abort);
          __syncwarp();
          if (!__shfl_sync(0xffffffffu, free_, 0)) break;
        }
        const int cbl = (nb - ch * kGvStageBlocks) < kGvStageBlocks ? nb - ch * kGvStageBlocks : kGvStageBlocks;
        const uint32_t bytes = static_cast<uint32_t>(cbl) * 32u;
        const int nv = (nrows - 16 * tl) < 16 ? nrows - 16 * tl : 16;
        const uint32_t fb = smem_u32(&full[slot]);
        if (lane == 0) mbar_arrive_expect_tx(fb, bytes * static_cast<uint32_t>(nv));
        __syncwarp();
        if (lane < nv)
          bulk_load(ring + static_cast<uint32_t>(slot) * kGvStageBytes + static_cast<uint32_t>(lane) * kGvRowPitch,
                    rowp + static_cast<int64_t>(ch) * kGvStageRow, bytes, fb);
        if (++ch == nch) {
          ch = 0;
          ++tl;
          if (lane < 16 && 16 * tl + lane < nrows) rowp = rows[16 * tl + lane].code;
        }
      }
      // The CTA's rows of B into L2 for the output phase, a few stages before
      // the end (an earlier prefetch would be evicted by the stream of codes).
      if (lane < g.n) {
        const GvProj &p = g.p[lane];
        const int64_t a = R0 > p.row_off ? R0 : p.row_off, e = R1 < p.row_off + p.d ? R1 : p.row_off + p.d;
        if (a < e) {
          const int64_t b0 = (a - p.row_off) * p.r * 2, b1 = (e - p.row_off) * p.r * 2;
          const int64_t a0 = b0 & ~int64_t{15};  // 16-byte aligned start and length
          gv_prefetch(p.B, a0, ((b1 + 15) & ~int64_t{15}) - a0, p.d * p.r * 2);
        }
      }
      if (lane == 0) {
        // After an abort the copies still in flight target this CTA's shared
        // memory: wait (bounded) for the last one of every slot.
        if (s < nst)
          for (int q = s > R ? s - R : 0; q < s; ++q) mbar_wait_drain(smem_u32(&full[q % R]), (q / R) & 1);
        // While the consumers finish: wait (bounded) until every CTA has
        // published its rows of u, then stage u; the final barrier hands it over.
        unsigned int spins = 0;
        while (gv_ld_acquire(&g.zero_area[kGvFlagReady]) < static_cast<unsigned>(rtot)) {
          if (++spins > kGvSpinLimit) {
            qn_flag_timeout();
            break;
          }
          __nanosleep(128);
        }
      }
      __syncwarp();
#pragma unroll 4
      for (int e = lane; e < rtot * M; e += 32) us[e] = ld_cg_f32(g.u + e);
    }
  } else {
  // ================================ consumers ===================================
  // X into the odd halves of the table rows (swizzled by token)
  for (int t = 0; t < M; ++t)
    for (uint32_t v = tid; v < kc; v += kGvWarps * 32)
      cp_async16(sb + gv_x_chunk(t * kc + v, t), g.X + static_cast<int64_t>(t) * k + v * 8);
  cp_async_commit();
  // Block constants of the range, decoded once into mconst[lr * ms + b]
  // straight from global memory (through L2): thread (r0, c) takes item c of
  // rows r0, r0 + rpp, ..., loading kGvDecRows rows' inputs before it decodes
  // any; the first batch goes out before the stage copies.  When nb is a
  // multiple of 4, item c is blocks 4c .. 4c + 3 (one 32-bit read of DQ
  // codes: a row starts at a multiple of 4 blocks, so the four share one
  // 256-block DQ group; or one 16-byte read of fp32 constants), else item c
  // is block c.  k <= 16384, so a row has at most 256 items and rpp >= 2.
  const bool by4 = (nb & 3) == 0;
  const int dper = by4 ? nb >> 2 : nb;          // items per row
  const int rpp = (kGvWarps * 32) / dper;       // rows per pass
  const int dc = tid % dper, dr0 = tid / dper;
  const int nrt = ntl * 16;
  const int64_t eb = by4 ? 4 * dc : dc;         // first block of the item within its row
  // per row: DQ {codes, scale, mean} or fp32 constants, in .x .. .w; dq flag
  uint4 dv[kGvDecRows];
  int dqv[kGvDecRows];
  auto dec_load = [&](int lb) {
#pragma unroll
    for (int i = 0; i < kGvDecRows; ++i) {
      const int lr = lb + i * rpp;
      dqv[i] = -1;
      dv[i] = make_uint4(0u, 0u, 0u, 0u);
      if (dr0 < rpp && lr < nrt) {
        const GvRow rw = rows[lr];
        dqv[i] = rw.dq;
        if (rw.dq >= 0) {
          const GvProj &p = g.p[rw.p];
          const int64_t e = static_cast<int64_t>(rw.prow) * nb + eb;  // the item's first block
          if (rw.dq > 0) {
            const int8_t *q = static_cast<const int8_t *>(p.consts) + e;
            dv[i].x = by4 ? ld_cg_u32(q) : ld_cg_s8(q);
            dv[i].y = __float_as_uint(ld_cg_f32(p.absmax_scale + (e >> 8)));
            dv[i].z = __float_as_uint(ld_cg_f32(p.absmax_mean));
          } else {
            const float *f = static_cast<const float *>(p.consts) + e;
            if (by4)
              dv[i] = ld_cg_v4(f);
            else
              dv[i].x = __float_as_uint(ld_cg_f32(f));
          }
        }
      }
    }
  };
  auto dec_store = [&](int lb) {
#pragma unroll
    for (int i = 0; i < kGvDecRows; ++i) {
      const int lr = lb + i * rpp;
      if (dr0 >= rpp || lr >= nrt) break;
      float *mr = mconst + lr * g.ms;
      const float sg = __uint_as_float(dv[i].y), mu = __uint_as_float(dv[i].z);
      if (by4) {
        float m[4] = {0.f, 0.f, 0.f, 0.f};
        if (dqv[i] > 0) {
#pragma unroll
          for (int j = 0; j < 4; ++j) m[j] = dq_absmax(static_cast<int8_t>((dv[i].x >> (8 * j)) & 0xFFu), sg, mu);
        } else if (dqv[i] == 0) {
          m[0] = __uint_as_float(dv[i].x);
          m[1] = __uint_as_float(dv[i].y);
          m[2] = __uint_as_float(dv[i].z);
          m[3] = __uint_as_float(dv[i].w);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) mr[4 * dc + j] = m[j];
      } else {
        float m = 0.f;
        if (dqv[i] > 0)
          m = dq_absmax(static_cast<int8_t>(dv[i].x & 0xFFu), sg, mu);
        else if (dqv[i] == 0)
          m = __uint_as_float(dv[i].x);
        mr[dc] = m;
      }
    }
  };
  dec_load(dr0);
  asm volatile("bar.arrive 2, %0;" ::"n"((kGvWarps + 1) * 32) : "memory");  // the stage copies may start
  // adapter rows of this CTA: warp slice [v0, v1) of the k / 8 vectors
  const int v0 = static_cast<int>(kc * warp / kGvWarps), v1 = static_cast<int>(kc * (warp + 1) / kGvWarps);
  uint4 av0[kGvUVec], av1[kGvUVec];  // A pieces of two adapter rows
  auto load_a = [&](uint4 (&av)[kGvUVec], int iu, int bt) {
    const int64_t j = blockIdx.x + static_cast<int64_t>(G) * iu;
    int pi = 0;
    for (int i = 1; i < g.n; ++i)
      if (j >= g.p[i].u_off) pi = i;
    const uint16_t *arow = g.p[pi].A + (j - g.p[pi].u_off) * k;
#pragma unroll
    for (int i = 0; i < kGvUVec; ++i) {
      const int v = v0 + lane + 32 * (bt * kGvUVec + i);
      av[i] = (v < v1) ? ld_cg_v4(arow + static_cast<int64_t>(v) * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  if (nu > 0) load_a(av0, 0, 0);
  if (nu > 1) load_a(av1, 1, 0);
  dec_store(dr0);
  for (int lb = dr0 + kGvDecRows * rpp; lb < nrt; lb += kGvDecRows * rpp) {
    dec_load(lb);
    dec_store(lb);
  }
  cp_async_wait_all();  // X
  asm volatile("bar.sync 1, %0;" ::"n"(kGvWarps * 32) : "memory");

  {
    const int span = v1 - v0;
    const int nbt = span > 0 ? (span + 32 * kGvUVec - 1) / (32 * kGvUVec) : 1;
    // this warp's part of u[t, j] for adapter row j = blockIdx + G iu, into ured
    auto u_row = [&](uint4 (&av)[kGvUVec], int iu) {
      float ua[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) ua[t] = 0.f;
      for (int bt = 0; bt < nbt; ++bt) {
        if (bt > 0) load_a(av, iu, bt);
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
    };
    for (int iu = 0; iu < nu; iu += 2) {
      if (iu >= 2) {
        load_a(av0, iu, 0);
        if (iu + 1 < nu) load_a(av1, iu + 1, 0);
      }
      u_row(av0, iu);
      if (iu + 1 < nu) u_row(av1, iu + 1);
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kGvWarps * 32) : "memory");
  if (tid == 0) mbar_arrive(smem_u32(upart));  // the second producer warp finishes and publishes them

  // ---- weight loop: wait for a stage, consume blocks warp + 16 j, j = 0..3 ---------
  const uint32_t lane4 = static_cast<uint32_t>(lane) << 2;
  // this lane's code bytes of block `warp`, row gq (block warp + 16 j: +512 j; row gq + 8: +16384)
  const uint32_t cofs = static_cast<uint32_t>(gq) * kGvRowPitch + static_cast<uint32_t>(warp * 32 + tq * 8);
  // x of token gq, elements 64 warp + 16 tq .. + 15 (block warp + 16 j: +4096 j bytes)
  const uint32_t xw0 = sb + gv_x_chunk(gq * kc + 2u * tq, gq) + (static_cast<uint32_t>(warp) << 8);
  const uint32_t xw1 = sb + gv_x_chunk(gq * kc + 2u * tq + 1u, gq) + (static_cast<uint32_t>(warp) << 8);
  const bool xtok = gq < M;
  auto lut8 = [&](uint2 c, uint32_t (&a)[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t sel = 0x5504u | (static_cast<uint32_t>(i) << 4);
      a[i] = lds_lut(gv_lut_off(c.x, lane4, sel));
      a[4 + i] = lds_lut(gv_lut_off(c.y, lane4, sel));
    }
  };
  const uint32_t mrow = static_cast<uint32_t>(16 * g.ms * 4);  // bytes per tile of decoded constants
  uint32_t mb0 = smem_u32(mconst) + static_cast<uint32_t>(gq * g.ms * 4) + static_cast<uint32_t>(warp * 4);
  uint32_t mb1 = mb0 + static_cast<uint32_t>(8 * g.ms * 4);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  bool ok = true;
  int tl = 0, ch = 0;
#pragma unroll 1
  for (int s = 0; s < nst; ++s) {
    const int slot = s % R;
    if (ok) ok = mbar_wait(smem_u32(&full[slot]), (s / R) & 1, abort);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      const int cbl = (nb - ch * kGvStageBlocks) < kGvStageBlocks ? nb - ch * kGvStageBlocks : kGvStageBlocks;
      const uint32_t ca = ring + static_cast<uint32_t>(slot) * kGvStageBytes + cofs;
      const uint32_t xo = static_cast<uint32_t>(ch * kGvStageBlocks) << 8;  // 256 bytes of table row per block
      const uint32_t mo = static_cast<uint32_t>(ch * kGvStageBlocks) * 4u;
#pragma unroll
      for (int jp = 0; jp < kGvStageBlocks / 16; jp += 2) {
        // blocks warp + 16 jp and warp + 16 (jp + 1) side by side; a block past
        // the chunk's end reads in-bounds leftovers of the slot with x = 0, m = 0
        const bool v0 = warp + 16 * jp < cbl, v1 = warp + 16 * (jp + 1) < cbl;
        if (!v0) break;  // the same in the whole warp
        const uint32_t cj = ca + 512u * jp;
        const uint2 c00 = lds_v2(cj), c01 = lds_v2_off8r(cj), c10 = lds_v2(cj + 512u), c11 = lds_v2_off8r(cj + 512u);
        uint4 x00 = make_uint4(0u, 0u, 0u, 0u), x01 = x00, x10 = x00, x11 = x00;
        const uint32_t xj = xo + 4096u * jp;
        if (xtok) {
          x00 = lds_v4(xw0 + xj);
          x01 = lds_v4(xw1 + xj);
          if (v1) {
            x10 = lds_v4(xw0 + xj + 4096u);
            x11 = lds_v4(xw1 + xj + 4096u);
          }
        }
        const uint32_t mj = mo + 64u * jp;
        const float m00 = lds_f32(mb0 + mj), m01 = lds_f32(mb1 + mj);
        const float m10 = v1 ? lds_f32(mb0 + mj + 64u) : 0.f, m11 = v1 ? lds_f32(mb1 + mj + 64u) : 0.f;
        uint32_t a0[8], a1[8], b0[8], b1[8];  // bf16 pairs: block 0 rows g, g + 8; block 1 rows g, g + 8
        lut8(c00, a0);
        lut8(c01, a1);
        lut8(c10, b0);
        lut8(c11, b1);
        float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
        gv_mma(d, a0[0], a1[0], a0[1], a1[1], x00.x, x00.y);
        gv_mma(e, b0[0], b1[0], b0[1], b1[1], x10.x, x10.y);
        gv_mma(d, a0[2], a1[2], a0[3], a1[3], x00.z, x00.w);
        gv_mma(e, b0[2], b1[2], b0[3], b1[3], x10.z, x10.w);
        gv_mma(d, a0[4], a1[4], a0[5], a1[5], x01.x, x01.y);
        gv_mma(e, b0[4], b1[4], b0[5], b1[5], x11.x, x11.y);
        gv_mma(d, a0[6], a1[6], a0[7], a1[7], x01.z, x01.w);
        gv_mma(e, b0[6], b1[6], b0[7], b1[7], x11.z, x11.w);
        acc[0] = fmaf(e[0], m10, fmaf(d[0], m00, acc[0]));
        acc[1] = fmaf(e[1], m10, fmaf(d[1], m00, acc[1]));
        acc[2] = fmaf(e[2], m11, fmaf(d[2], m01, acc[2]));
        acc[3] = fmaf(e[3], m11, fmaf(d[3], m01, acc[3]));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));  // this warp is done with the slot
    if (++ch == nch) {
      // end of tile tl: this warp's partial sums
      float *pw = part + (tl * kGvWarps + warp) * 16 * M;
      if (2 * tq < M) {
        pw[gq * M + 2 * tq] = acc[0];
        pw[(gq + 8) * M + 2 * tq] = acc[2];
      }
      if (2 * tq + 1 < M) {
        pw[gq * M + 2 * tq + 1] = acc[1];
        pw[(gq + 8) * M + 2 * tq + 1] = acc[3];
      }
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
      ch = 0;
      ++tl;
      mb0 += mrow;
      mb1 += mrow;
    }
  }
  }  // consumers

  // ---- adapter terms and output -------------------------------------------------
  // Thread lr takes row lr of the range: the first 64 values of its B row are
  // loaded (16-byte pieces) before the wait for u, so both round trips overlap.
  const bool bvec = g.bvec != 0;  // every r a multiple of 8 (rows of B 16-byte aligned)
  uint4 bq[8];
  if (bvec && tid < nrows) {
    const GvRow &rw = rows[tid];
    const GvProj &p = g.p[rw.p];
    const uint16_t *br = p.B + static_cast<int64_t>(rw.prow) * p.r;
#pragma unroll
    for (int c = 0; c < 8; ++c) bq[c] = (8 * c < p.r) ? ld_cg_v4(br + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();  // every partial sum written; u staged
  // Y = (partial sums of the warps, in warp order) + u . B[row]
  for (int lr = tid; lr < nrows; lr += kGvThreads) {
    const GvRow &rw = rows[lr];
    const GvProj &p = g.p[rw.p];
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
          for (int t = 0; t < MT; ++t) {
            if (t >= M) break;
            // u[t, q0 + 8c ..] in two 16-byte reads (every r and u_off is a multiple of 8)
            const float4 ua = *reinterpret_cast<const float4 *>(ur + t * rtot + q0 + 8 * c);
            const float4 ub = *reinterpret_cast<const float4 *>(ur + t * rtot + q0 + 8 * c + 4);
            const float uv[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              const float b = (h & 1) ? __uint_as_float(bw[h >> 1] & 0xFFFF0000u) : __uint_as_float(bw[h >> 1] << 16);
              a[t][h & 1] = fmaf(uv[h], b, a[t][h & 1]);
            }
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
    const int tl = lr >> 4, r16 = lr & 15;
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      if (t >= M) break;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kGvWarps; ++w) v += part[((tl * kGvWarps + w) * 16 + r16) * M + t];
      p.Y[t * p.d + rw.prow] = f32_to_bf16_bits(v + (a[t][0] + a[t][1]));
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
