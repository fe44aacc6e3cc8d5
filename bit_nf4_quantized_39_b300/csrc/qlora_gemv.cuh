// qlora_gemv.cuh -- fused QLoRA forward for one token (and up to eight when
// M * k <= 16384) of a group of projections of one input, in one persistent
// kernel per call:
//
//   Y_g = X deq(Q_g)^T + s_g (X A_g^T) B_g^T      X: M x k bf16, Q_g: d_g x k NF4
//
// ("PEFT course notes" §2.2, h = Wx + BAx; "QLoRA paper summary": the frozen
// weight is 4-bit NF4 with blockwise constants.)  The call is bound by the
// bytes of the packed weights (8-50 MB per call at decode sizes), so the
// design keeps HBM streaming across call boundaries:
//
// * one CTA per SM; the group's rows are cut into 16-row tiles and every CTA
//   takes one contiguous range of tiles (equal up to one tile);
// * programmatic dependent launch: the kernel lets the next call launch as
//   soon as it starts (launch_dependents at entry), so on every SM the next
//   call's CTA starts as soon as this one retires.  Before griddepcontrol.wait
//   a CTA only prefetches its first code bytes into L2 (a prefetch cannot
//   return stale data), builds its level table and initialises its
//   barriers; everything that another kernel may write -- codes, block
//   constants, X, A, B, u, Y, the workspace counters -- is read or written
//   after the wait, through L2 (TMA, bulk copies, ld.global.cg);
// * warp 16 streams each tile's codes with TMA (16 rows x 16 blocks = 8 KiB
//   per stage, four 128-byte-swizzled boxes) through an 8-stage ring, plus
//   the tile's block constants (int8 DQ codes or fp32 absmax) as one bulk
//   copy with its first stage;
// * warps 0-15 take one 64-block of every stage each: a lane (group g,
//   thread t) turns 8 code bytes of rows g and g+8 into bf16x2 A-fragment
//   registers through a per-lane replicated byte-pair table (one byte
//   permute and one shared load per byte), multiplies them on mma.sync
//   (m16n8k16; tokens are the N columns) against x, which is staged as bf16
//   in the unused half of every table row, and scales each block's dot
//   products by its block constant in fp32.  The MMA's k order is a
//   permutation of the block's elements, the same for both operands.  At the
//   end of a tile the sixteen warps' partial sums are added in a fixed order
//   into the tile's row sums (shared memory).  The consumer warps also
//   compute the adapter rows u = s X A^T (row j by warp j / gridDim of CTA
//   j mod gridDim) right after staging X, and publish them through a
//   workspace counter;
// * warp 17 copies the B rows of its CTA's range into shared memory, waits
//   (bounded) until every CTA has published its rows of u, and forms
//   u . B[row] for every row of the range while the weights stream;
// * the epilogue writes bf16 Y = row sum + adapter term.
//
// Every CTA is resident at once (one per SM, at most one per SM), so the
// grid-wide wait for u always ends; it is bounded all the same (QN_DEV_TIMEOUT).
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace qn {

constexpr int kGvConsumers = 16;                     // one 64-block of every stage each
constexpr int kGvProducerWarp = kGvConsumers;
constexpr int kGvAdapterWarp = kGvConsumers + 1;
constexpr int kGvThreads = (kGvConsumers + 2) * 32;
constexpr int kGvRows = 16;                          // rows per tile (MMA M)
constexpr int kGvStageBlocks = 16;                   // 64-blocks per stage
constexpr int kGvStageBytes = kGvRows * kGvStageBlocks * 32;  // 8 KiB of codes
constexpr int kGvBoxBytes = 128;                     // TMA box width: one swizzle span, 4 blocks
constexpr int kGvStages = 8;                         // ring depth (64 KiB in flight per SM)
constexpr int kGvMaxNb = 256;                        // 64-blocks per row (k <= 16384)
constexpr int kGvCSlots = 2;                         // block-constant tiles in flight
constexpr int kGvCSlotBytes = kGvRows * kGvMaxNb * 4;  // one tile's fp32 constants (or int8 codes)
constexpr int kGvLutBytes = 256 * 256;               // 256 rows: table entry b at 256 b + 4 lane, x in bytes 128..255
constexpr int kGvMaxXElems = 16384;                  // M * k staged in the table rows
constexpr int kGvMaxM = 8;
constexpr int kGvPartBytes = 2 * kGvConsumers * kGvRows * kGvMaxM * 4;  // two tile-end slots
constexpr int kGvMaxRowVals = 1024;                  // (rows of a CTA) * M
constexpr int kGvMaxSig = 1040;                      // DQ group scales of a CTA's rows
constexpr int kGvMaxU = 2048;                        // M * (adapter rows of the group)
constexpr int kGvBRowBytes = 24 * 1024;              // B rows of a CTA prefetched to shared memory (when they fit)
constexpr int kGvXPer = kGvMaxXElems / 8 / (kGvConsumers * 32);  // 16-byte X loads per consumer thread
constexpr int kGvMaxGroup = 8;
constexpr int kGvPrefetch = 96 * 1024;               // code bytes per CTA prefetched into L2 before the wait
constexpr unsigned kGvSpinLimit = 1u << 22;
constexpr int kGvFlagReady = 0, kGvFlagExit = 1;     // zero-area words

struct GvProj {
  CUtensorMap tmap;    // codes as uint32 [d][k / 8], box {32, 16}, 128-byte swizzle
  QnNF4View q;
  const uint16_t *A;   // r x k bf16
  const uint16_t *B;   // d x r bf16
  uint16_t *Y;         // M x d bf16
  int r;
  float s;
  int64_t tile_off;    // first tile of this projection in the group's tile list
  int64_t u_off;       // first adapter row of this projection
};
struct GvGroup {
  GvProj p[kGvMaxGroup];
  int n;
  int M;
  int64_t k;
  int64_t ntiles;      // total tiles
  int64_t rtot;        // total adapter rows
  const uint16_t *X;   // M x k bf16
  float *u;            // M x rtot fp32 (workspace)
  unsigned int *zero_area;
};

// Shared-memory layout (offsets from a 1024-aligned base).
constexpr size_t kGvOffRing = 0;
constexpr size_t kGvOffLut = kGvOffRing + static_cast<size_t>(kGvStages) * kGvStageBytes;
constexpr size_t kGvOffCtile = kGvOffLut + kGvLutBytes;
constexpr size_t kGvOffPart = kGvOffCtile + static_cast<size_t>(kGvCSlots) * kGvCSlotBytes;
constexpr size_t kGvOffRowsum = kGvOffPart + kGvPartBytes;
constexpr size_t kGvOffAdp = kGvOffRowsum + kGvMaxRowVals * 4;
constexpr size_t kGvOffSig = kGvOffAdp + kGvMaxRowVals * 4;
constexpr size_t kGvOffU = kGvOffSig + kGvMaxSig * 4;
constexpr size_t kGvOffBRows = kGvOffU + kGvMaxU * 4;
constexpr size_t kGvOffBars = kGvOffBRows + kGvBRowBytes;
constexpr size_t kGvSmemBytes = 1024 + kGvOffBars + 512;

struct GvBars {
  uint64_t full[kGvStages], empty[kGvStages], cfree[kGvCSlots];
  float mu[kGvMaxGroup];     // DQ mean of each projection
  int sig_base[kGvMaxGroup]; // index of DQ scale 0 of each projection in the staged scales
  int abort;
};
static_assert(sizeof(GvBars) <= 512, "barrier area");

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ uint4 ld_cg_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
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
__device__ __forceinline__ int ld_cg_s8(const int8_t *p) {
  short v;
  asm volatile("ld.global.cg.s8 %0, [%1];" : "=h"(v) : "l"(p));
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
// Byte offset of the table entry of byte `i` of `w` for this lane: (byte << 8) | (lane << 2).
__device__ __forceinline__ uint32_t gv_lut_off(uint32_t w, uint32_t lane4, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(w), "r"(lane4), "r"(sel));
  return r;
}
// Shared-memory byte offset (within the table region) of byte o of the staged X.
__device__ __forceinline__ uint32_t gv_x_off(uint32_t o) { return ((o >> 7) << 8) + 128u + (o & 127u); }

__device__ __forceinline__ const CUtensorMap *gv_map(const GvGroup &g, int pi) {
  switch (pi) {
    case 0: return &g.p[0].tmap;
    case 1: return &g.p[1].tmap;
    case 2: return &g.p[2].tmap;
    case 3: return &g.p[3].tmap;
    case 4: return &g.p[4].tmap;
    case 5: return &g.p[5].tmap;
    case 6: return &g.p[6].tmap;
    default: return &g.p[7].tmap;
  }
}

__device__ __forceinline__ int gv_proj_of_tile(const GvGroup &g, int64_t t) {
  int i = 0;
#pragma unroll
  for (int j = 1; j < kGvMaxGroup; ++j)
    if (j < g.n && t >= g.p[j].tile_off) i = j;
  return i;
}
__device__ __forceinline__ int gv_proj_of_urow(const GvGroup &g, int64_t j) {
  int i = 0;
#pragma unroll
  for (int q = 1; q < kGvMaxGroup; ++q)
    if (q < g.n && j >= g.p[q].u_off) i = q;
  return i;
}

// Bytes of a tile's block constants that one bulk copy brings in (a multiple
// of 16; the rest, in a projection's last tile only, is read from L2).
__device__ __forceinline__ uint32_t gv_cbytes(const QnNF4View &q, int64_t row0, int nb) {
  const uintptr_t base = q.dq ? reinterpret_cast<uintptr_t>(q.absmax_q) : reinterpret_cast<uintptr_t>(q.absmax);
  if (base & 15u) return 0u;
  const int64_t nrows = (q.d - row0 < kGvRows) ? q.d - row0 : static_cast<int64_t>(kGvRows);
  return static_cast<uint32_t>(nrows * nb * (q.dq ? 1 : 4)) & ~15u;
}

// 320 threads are allocated as 12 warps' worth of registers: at most 168 per thread.
__global__ void __launch_bounds__(kGvThreads, 1)
qlora_gemv_kernel(const __grid_constant__ GvGroup g) {
  extern __shared__ unsigned char gv_raw[];
  unsigned char *base = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(gv_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char *ring = base + kGvOffRing;
  unsigned char *lut = base + kGvOffLut;
  unsigned char *ctile = base + kGvOffCtile;
  float *part = reinterpret_cast<float *>(base + kGvOffPart);
  float *rowsum = reinterpret_cast<float *>(base + kGvOffRowsum);
  float *adp = reinterpret_cast<float *>(base + kGvOffAdp);
  float *sig = reinterpret_cast<float *>(base + kGvOffSig);
  float *us = reinterpret_cast<float *>(base + kGvOffU);
  uint16_t *brows = reinterpret_cast<uint16_t *>(base + kGvOffBRows);
  GvBars *bars = reinterpret_cast<GvBars *>(base + kGvOffBars);
  volatile int *abort = &bars->abort;

  pdl_trigger();  // the next call may launch on every SM this grid retires from

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t k = g.k;
  const int nb = static_cast<int>(k >> 6);
  const int nst = (nb + kGvStageBlocks - 1) / kGvStageBlocks;  // stages per tile
  const int M = g.M;
  const int G = gridDim.x;
  const int64_t t0 = g.ntiles * blockIdx.x / G, t1 = g.ntiles * (blockIdx.x + 1) / G;
  const int ntl = static_cast<int>(t1 - t0);

  if (tid == 0) {
    for (int i = 0; i < kGvStages; ++i) {
      mbar_init(smem_u32(&bars->full[i]), 1);
      mbar_init(smem_u32(&bars->empty[i]), kGvConsumers);
    }
    for (int i = 0; i < kGvCSlots; ++i) mbar_init(smem_u32(&bars->cfree[i]), 1);
    bars->abort = 0;
    mbar_fence_init();
  }
  if (warp == kGvProducerWarp && lane == 0) {
    // Pre-wait: the first code bytes of this CTA's range into L2 only.
    for (int i = 0; i < g.n; ++i) tma_prefetch_desc(gv_map(g, i));
    int64_t left = kGvPrefetch;
    for (int64_t t = t0; t < t1 && left > 0;) {
      const int pi = gv_proj_of_tile(g, t);
      const GvProj &p = g.p[pi];
      const int64_t tend = (pi + 1 < g.n) ? g.p[pi + 1].tile_off : g.ntiles;
      const int64_t te = tend < t1 ? tend : t1;
      const int64_t row0 = (t - p.tile_off) * kGvRows;
      int64_t rows = (te - t) * kGvRows;
      if (row0 + rows > p.q.d) rows = p.q.d - row0;
      int64_t bytes = rows * (k >> 1);
      if (bytes > left) bytes = left;
      const unsigned char *src = p.q.codes + row0 * (k >> 1);
      for (int64_t o = 0; o + 16 <= bytes; o += 32768) {
        const int64_t len = (bytes - o < 32768) ? ((bytes - o) & ~int64_t{15}) : 32768;
        prefetch_l2_bulk(src + o, static_cast<uint32_t>(len));
      }
      left -= bytes;
      t = te;
    }
  }
  __syncthreads();

  if (warp == kGvProducerWarp) {
    // ================================ producer =================================
    pdl_wait_grid();
    if (lane == 0) {
      uint32_t qi = 0;
      bool ok = true;
      for (int tl = 0; tl < ntl && ok; ++tl) {
        const int64_t t = t0 + tl;
        const int pi = gv_proj_of_tile(g, t);
        const QnNF4View &q = g.p[pi].q;
        const int64_t row0 = (t - g.p[pi].tile_off) * kGvRows;
        const CUtensorMap *map = gv_map(g, pi);
        for (int s = 0; s < nst; ++s, ++qi) {
          const uint32_t slot = qi % kGvStages;
          if (qi >= kGvStages && !mbar_wait(smem_u32(&bars->empty[slot]), ((qi / kGvStages) - 1) & 1, abort)) {
            ok = false;
            break;
          }
          uint32_t cb = 0;
          if (s == 0) {
            if (tl >= kGvCSlots &&
                !mbar_wait(smem_u32(&bars->cfree[tl % kGvCSlots]), ((tl / kGvCSlots) - 1) & 1, abort)) {
              ok = false;
              break;
            }
            cb = gv_cbytes(q, row0, nb);
          }
          const uint32_t full = smem_u32(&bars->full[slot]);
          mbar_arrive_expect_tx(full, kGvStageBytes + cb);
          if (cb) {
            const void *src = q.dq ? static_cast<const void *>(q.absmax_q + row0 * nb)
                                   : static_cast<const void *>(q.absmax + row0 * nb);
            bulk_load(smem_u32(ctile + (tl % kGvCSlots) * kGvCSlotBytes), src, cb, full);
          }
#pragma unroll
          for (int j = 0; j < kGvStageBytes / (kGvRows * kGvBoxBytes); ++j)
            tma_load_2d(smem_u32(ring + slot * kGvStageBytes + j * kGvRows * kGvBoxBytes), map,
                        (s * kGvStageBlocks + 4 * j) * 8, static_cast<int32_t>(row0), full);
        }
      }
      // Every copy this CTA started lands before it may retire.
      for (uint32_t r = (qi > kGvStages ? qi - kGvStages : 0); r < qi; ++r)
        mbar_wait_drain(smem_u32(&bars->full[r % kGvStages]), (r / kGvStages) & 1);
    }
    return;
  }

  if (warp == kGvAdapterWarp) {
    // ============================== adapter warp ===============================
    // B rows of this CTA's range (contiguous per projection) into shared
    // memory with cp.async, then -- once every CTA has published its rows of
    // u -- adp[row, t] = u[t, proj] . B[row] for every row of the range.
    pdl_wait_grid();
    const int64_t rtot = g.rtot;
    const int64_t nrows_cta = static_cast<int64_t>(ntl) * kGvRows;
    // brows + bro[i] + row * r is row `row` of projection i's B when staged;
    // the offset itself may be negative (rows before the range are not staged).
    int64_t bro[kGvMaxGroup];
    bool staged[kGvMaxGroup];
    {
      int64_t off = 0;
      bool fits = true;
#pragma unroll
      for (int i = 0; i < kGvMaxGroup; ++i) {
        bro[i] = 0;
        staged[i] = false;
      }
      for (int i = 0; i < g.n; ++i) {
        const GvProj &p = g.p[i];
        const int64_t tend = (i + 1 < g.n) ? g.p[i + 1].tile_off : g.ntiles;
        const int64_t ta = t0 > p.tile_off ? t0 : p.tile_off, tb = t1 < tend ? t1 : tend;
        if (ta >= tb) continue;
        const int64_t ra = (ta - p.tile_off) * kGvRows;
        int64_t rb = (tb - p.tile_off) * kGvRows;
        if (rb > p.q.d) rb = p.q.d;
        const int64_t elems = (rb - ra) * p.r;
        const int64_t padded = (elems + 7) & ~int64_t{7};
        if (!fits || (off + padded) * 2 > kGvBRowBytes || (p.r & 7) || (reinterpret_cast<uintptr_t>(p.B) & 15u)) {
          fits = false;
          continue;
        }
        const uint16_t *src = p.B + ra * p.r;
        for (int64_t e = static_cast<int64_t>(lane) * 8; e < elems; e += 32 * 8) cp_async16(smem_u32(brows + off + e), src + e);
        bro[i] = off - ra * p.r;
        staged[i] = true;
        off += padded;
      }
      cp_async_commit();
    }
    // wait until every adapter row of the group is published
    if (lane == 0) {
      unsigned int spins = 0;
      while (gv_ld_acquire(&g.zero_area[kGvFlagReady]) < static_cast<unsigned>(rtot)) {
        if (++spins > kGvSpinLimit) { qn_flag_timeout(); break; }
        __nanosleep(32);
      }
    }
    __syncwarp();
    {
      const int64_t nu = static_cast<int64_t>(M) * rtot;
      for (int64_t i0 = 0; i0 < nu; i0 += 32 * 8) {
        float v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int64_t i = i0 + c * 32 + lane;
          v[c] = (i < nu) ? ld_cg_f32(g.u + i) : 0.f;
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int64_t i = i0 + c * 32 + lane;
          if (i < nu) us[i] = v[c];
        }
      }
    }
    cp_async_wait_all();
    __syncwarp();
    for (int64_t lr = lane; lr < nrows_cta; lr += 32) {
      const int64_t t = t0 + lr / kGvRows;
      const int pi = gv_proj_of_tile(g, t);
      const GvProj &p = g.p[pi];
      const int64_t row = (t - p.tile_off) * kGvRows + lr % kGvRows;
      float a[kGvMaxM];
#pragma unroll
      for (int tt = 0; tt < kGvMaxM; ++tt) a[tt] = 0.f;
      if (row < p.q.d) {
        const float *ur = us + p.u_off;
        if (staged[pi]) {
          const uint16_t *br = brows + bro[pi] + row * p.r;
          for (int q = 0; q < p.r; q += 2) {
            const uint32_t bw = *reinterpret_cast<const uint32_t *>(br + q);
            const float b0 = __uint_as_float(bw << 16), b1 = __uint_as_float(bw & 0xFFFF0000u);
#pragma unroll
            for (int tt = 0; tt < kGvMaxM; ++tt)
              if (tt < M) a[tt] = fmaf(ur[tt * rtot + q + 1], b1, fmaf(ur[tt * rtot + q], b0, a[tt]));
          }
        } else if ((p.r & 7) == 0 && (reinterpret_cast<uintptr_t>(p.B) & 15u) == 0) {
          // not staged: 8 values per 16-byte load, four loads in flight
          const uint16_t *brow = p.B + row * p.r;
          for (int q0 = 0; q0 < p.r; q0 += 32) {
            uint4 bv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
              bv[c] = (q0 + 8 * c < p.r) ? ld_cg_v4(brow + q0 + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              if (q0 + 8 * c >= p.r) break;
              const uint32_t bw[4] = {bv[c].x, bv[c].y, bv[c].z, bv[c].w};
#pragma unroll
              for (int h = 0; h < 8; ++h) {
                const float b = (h & 1) ? __uint_as_float(bw[h >> 1] & 0xFFFF0000u) : __uint_as_float(bw[h >> 1] << 16);
#pragma unroll
                for (int tt = 0; tt < kGvMaxM; ++tt)
                  if (tt < M) a[tt] = fmaf(ur[tt * rtot + q0 + 8 * c + h], b, a[tt]);
              }
            }
          }
        } else {
          const uint16_t *brow = p.B + row * p.r;
          for (int q = 0; q < p.r; ++q) {
            const float b = bf16_bits_to_f32(ld_cg_u16(brow + q));
#pragma unroll
            for (int tt = 0; tt < kGvMaxM; ++tt)
              if (tt < M) a[tt] = fmaf(ur[tt * rtot + q], b, a[tt]);
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < kGvMaxM; ++tt)
        if (tt < M) adp[lr * M + tt] = a[tt];
    }
    __syncwarp();
    asm volatile("bar.arrive 3, %0;" ::"n"((kGvConsumers + 1) * 32) : "memory");  // adapter terms ready
    // the last CTA to get here returns the counters to zero
    if (lane == 0) {
      const unsigned int prev = atomicAdd(&g.zero_area[kGvFlagExit], 1u);
      if (prev == static_cast<unsigned>(G) - 1u) {
        atomicExch(&g.zero_area[kGvFlagReady], 0u);
        atomicExch(&g.zero_area[kGvFlagExit], 0u);
      }
    }
    return;
  }

  // ================================= consumers ==================================
  const int gq = lane >> 2, tq = lane & 3;
  const int cw = warp;  // takes block cw of every stage
  const uint32_t lane4 = static_cast<uint32_t>(lane) << 2;
  {
    // table entry b of lane l: bf16(level[b & 15]) | bf16(level[b >> 4]) << 16
    const int b0 = tid >> 5, l = tid & 31;
    uint32_t lv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) lv[i] = f32_to_bf16_bits(c_nf4_levels[i]);
    uint32_t *lw = reinterpret_cast<uint32_t *>(lut);
#pragma unroll
    for (int n = 0; n < 256 / kGvConsumers; ++n) {
      const int b = b0 + kGvConsumers * n;  // b & 15 = b0, b >> 4 = n
      lw[b * 64 + l] = lv[b0] | (lv[n] << 16);
    }
  }
  pdl_wait_grid();
  // Adapter rows of u done by this warp: j = blockIdx + G (warp + 8 i).  The
  // X loads and the first 2048 columns of the first row of A are issued
  // together, then X goes to shared memory.
  const int64_t rtot = g.rtot;
  const int64_t j_first = blockIdx.x + static_cast<int64_t>(G) * warp;
  constexpr int kAV = 4;  // 16-byte A loads per lane in flight (1024 columns)
  uint4 apre[kAV];
  {
    const int64_t nvec = static_cast<int64_t>(M) * k / 8;
    uint4 xv[kGvXPer];
#pragma unroll
    for (int v = 0; v < kGvXPer; ++v) {
      const int64_t i = v * (kGvConsumers * 32) + tid;
      xv[v] = (i < nvec) ? ld_cg_v4(g.X + i * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
    if (j_first < rtot) {
      const GvProj &p = g.p[gv_proj_of_urow(g, j_first)];
      const uint16_t *arow = p.A + (j_first - p.u_off) * k;
#pragma unroll
      for (int v = 0; v < kAV; ++v) {
        const int64_t e = (v * 32 + lane) * 8;
        apre[v] = (e < k) ? ld_cg_v4(arow + e) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int v = 0; v < kGvXPer; ++v) {
      const int64_t i = v * (kGvConsumers * 32) + tid;
      if (i < nvec) *reinterpret_cast<uint4 *>(lut + gv_x_off(static_cast<uint32_t>(i * 16))) = xv[v];
    }
  }
  // DQ group scales of this CTA's rows: for each projection in the range,
  // scales (row_a * nb) >> 8 .. ((row_b * nb) - 1) >> 8, stored consecutively.
  {
    int off = 0;
    if (tid < kGvMaxGroup) {
      bars->sig_base[tid] = 0;
      bars->mu[tid] = (tid < g.n && g.p[tid].q.dq) ? ld_cg_f32(g.p[tid].q.absmax_mean) : 0.f;
    }
    for (int i = 0; i < g.n; ++i) {
      const GvProj &p = g.p[i];
      const int64_t tend = (i + 1 < g.n) ? g.p[i + 1].tile_off : g.ntiles;
      const int64_t ta = t0 > p.tile_off ? t0 : p.tile_off, tb = t1 < tend ? t1 : tend;
      if (ta >= tb || !p.q.dq) continue;
      const int64_t ra = (ta - p.tile_off) * kGvRows;
      int64_t rb = (tb - p.tile_off) * kGvRows;
      if (rb > p.q.d) rb = p.q.d;
      const int64_t ga = (ra * nb) >> 8, gb = ((rb * nb) - 1) >> 8;
      for (int64_t x = tid; x <= gb - ga; x += kGvConsumers * 32) sig[off + x] = ld_cg_f32(p.q.absmax_scale + ga + x);
      if (tid == 0) bars->sig_base[i] = off - static_cast<int>(ga);
      off += static_cast<int>(gb - ga + 1);
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kGvConsumers * 32) : "memory");
  // This warp's adapter rows: u[t, j] = s A[j] . X[t], published through the
  // ready counter.
  for (int64_t j = j_first; j < rtot; j += static_cast<int64_t>(G) * kGvConsumers) {
    const GvProj &p = g.p[gv_proj_of_urow(g, j)];
    const uint16_t *arow = p.A + (j - p.u_off) * k;
    float acc[kGvMaxM];
#pragma unroll
    for (int t = 0; t < kGvMaxM; ++t) acc[t] = 0.f;
    for (int64_t e0 = 0; e0 < k; e0 += 32 * 8 * kAV) {
      uint4 av[kAV];
#pragma unroll
      for (int v = 0; v < kAV; ++v) {
        const int64_t e = e0 + (v * 32 + lane) * 8;
        if (j == j_first && e0 == 0) av[v] = apre[v];
        else av[v] = (e < k) ? ld_cg_v4(arow + e) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int v = 0; v < kAV; ++v) {
        const int64_t e = e0 + (v * 32 + lane) * 8;
        if (e >= k) continue;
        const uint32_t aw[4] = {av[v].x, av[v].y, av[v].z, av[v].w};
#pragma unroll
        for (int t = 0; t < kGvMaxM; ++t) {
          if (t >= M) break;
          const uint4 xq = *reinterpret_cast<const uint4 *>(lut + gv_x_off(static_cast<uint32_t>((t * k + e) * 2)));
          const uint32_t xw[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            acc[t] = fmaf(__uint_as_float(aw[c] << 16), __uint_as_float(xw[c] << 16), acc[t]);
            acc[t] = fmaf(__uint_as_float(aw[c] & 0xFFFF0000u), __uint_as_float(xw[c] & 0xFFFF0000u), acc[t]);
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kGvMaxM; ++t) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
    }
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < kGvMaxM; ++t)
        if (t < M) g.u[t * rtot + j] = p.s * acc[t];
      __threadfence();
      atomicAdd(&g.zero_area[kGvFlagReady], 1u);
    }
  }

  // After a timeout (ok == false) the warp skips the work of the remaining
  // stages but still meets every named barrier, like the other warps.
  bool ok = true;
  uint32_t qc = 0;  // stages consumed
  for (int tl = 0; tl < ntl; ++tl) {
    const int64_t t = t0 + tl;
    const int pi = gv_proj_of_tile(g, t);
    const GvProj &p = g.p[pi];
    const QnNF4View &qv = p.q;
    const int64_t row0 = (t - p.tile_off) * kGvRows;
    const bool dq = qv.dq != 0;
    const float mu = bars->mu[pi];
    const int sbase = bars->sig_base[pi];
    const unsigned char *ct = ctile + (tl % kGvCSlots) * kGvCSlotBytes;
    const uint32_t cbytes = gv_cbytes(qv, row0, nb);
    const bool row_ok[2] = {row0 + gq < qv.d, row0 + gq + 8 < qv.d};
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < nst && ok; ++s, ++qc) {
      const uint32_t slot = qc % kGvStages;
      ok = mbar_wait(smem_u32(&bars->full[slot]), (qc / kGvStages) & 1, abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const unsigned char *stage = ring + slot * kGvStageBytes;
      uint32_t av[2][8];  // [row half][byte]: bf16 pairs of the block's codes
      float m[2];
      const int cb = cw;
      const int b = s * kGvStageBlocks + cb;
      {
        const int chunk = 2 * (cb & 3) + (tq >> 1);
        const uint32_t off =
            (cb >> 2) * (kGvRows * kGvBoxBytes) + gq * kGvBoxBytes + ((chunk ^ gq) << 4) + ((tq & 1) << 3);
        const uint2 c0 = *reinterpret_cast<const uint2 *>(stage + off);
        const uint2 c1 = *reinterpret_cast<const uint2 *>(stage + off + 8 * kGvBoxBytes);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          av[0][i] = *reinterpret_cast<const uint32_t *>(lut + gv_lut_off(c0.x, lane4, 0x5504u | (i << 4)));
          av[0][4 + i] = *reinterpret_cast<const uint32_t *>(lut + gv_lut_off(c0.y, lane4, 0x5504u | (i << 4)));
          av[1][i] = *reinterpret_cast<const uint32_t *>(lut + gv_lut_off(c1.x, lane4, 0x5504u | (i << 4)));
          av[1][4 + i] = *reinterpret_cast<const uint32_t *>(lut + gv_lut_off(c1.y, lane4, 0x5504u | (i << 4)));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float mm = 0.f;
          if (row_ok[h] && b < nb) {
            const int lr = gq + 8 * h;
            const uint32_t o = static_cast<uint32_t>(lr * nb + b);
            const int64_t blk = (row0 + lr) * nb + b;
            if (dq) {
              const int qc8 = (o < cbytes) ? static_cast<int>(reinterpret_cast<const int8_t *>(ct)[o])
                                           : ld_cg_s8(qv.absmax_q + blk);
              mm = dq_absmax(static_cast<int8_t>(qc8), sig[sbase + static_cast<int>(blk >> 8)], mu);
            } else {
              mm = (o * 4 < cbytes) ? reinterpret_cast<const float *>(ct)[o] : ld_cg_f32(qv.absmax + blk);
            }
          }
          m[h] = mm;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->empty[slot]));  // codes are in registers now
      if (b < nb) {
        uint4 x0 = make_uint4(0u, 0u, 0u, 0u), x1 = x0;
        if (gq < M) {
          const uint32_t o = static_cast<uint32_t>((gq * k + static_cast<int64_t>(b) * 64 + tq * 16) * 2);
          x0 = *reinterpret_cast<const uint4 *>(lut + gv_x_off(o));
          x1 = *reinterpret_cast<const uint4 *>(lut + gv_x_off(o + 16));
        }
        const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        // two independent accumulation chains (steps 0, 2 and 1, 3)
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
        gv_mma(d0, av[0][0], av[1][0], av[0][1], av[1][1], xw[0], xw[1]);
        gv_mma(d1, av[0][2], av[1][2], av[0][3], av[1][3], xw[2], xw[3]);
        gv_mma(d0, av[0][4], av[1][4], av[0][5], av[1][5], xw[4], xw[5]);
        gv_mma(d1, av[0][6], av[1][6], av[0][7], av[1][7], xw[6], xw[7]);
        acc[0] = fmaf(d0[0] + d1[0], m[0], acc[0]);
        acc[1] = fmaf(d0[1] + d1[1], m[0], acc[1]);
        acc[2] = fmaf(d0[2] + d1[2], m[1], acc[2]);
        acc[3] = fmaf(d0[3] + d1[3], m[1], acc[3]);
      }
    }
    // ---- end of the tile: the warps' partial sums, added in warp order
    float *ps = part + (tl & 1) * (kGvConsumers * kGvRows * kGvMaxM);
    {
      float *pw = ps + cw * (kGvRows * kGvMaxM);
      pw[gq * kGvMaxM + 2 * tq] = acc[0];
      pw[gq * kGvMaxM + 2 * tq + 1] = acc[1];
      pw[(gq + 8) * kGvMaxM + 2 * tq] = acc[2];
      pw[(gq + 8) * kGvMaxM + 2 * tq + 1] = acc[3];
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kGvConsumers * 32) : "memory");
    if (tid == 0) mbar_arrive(smem_u32(&bars->cfree[tl % kGvCSlots]));  // every warp is done with the constants
    if (cw == (tl % kGvConsumers)) {
      for (int e = lane; e < kGvRows * M; e += 32) {
        const int row = e / M, tok = e % M;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kGvConsumers; ++w) v += ps[(w * kGvRows + row) * kGvMaxM + tok];
        rowsum[(tl * kGvRows + row) * M + tok] = v;
      }
    }
  }
  // ---- epilogue: wait for the adapter terms, then Y = row sum + adapter term
  asm volatile("bar.sync 3, %0;" ::"n"((kGvConsumers + 1) * 32) : "memory");
  asm volatile("bar.sync 1, %0;" ::"n"(kGvConsumers * 32) : "memory");  // every tile's row sums are written
  ok = !*abort && ok;
  const int64_t nvals = static_cast<int64_t>(ntl) * kGvRows * M;
  for (int64_t e = tid; e < nvals; e += kGvConsumers * 32) {
    const int64_t lr = e / M;
    const int tok = static_cast<int>(e % M);
    const int64_t t = t0 + lr / kGvRows;
    const int pi = gv_proj_of_tile(g, t);
    const GvProj &p = g.p[pi];
    const int64_t row = (t - p.tile_off) * kGvRows + lr % kGvRows;
    if (ok && row < p.q.d) p.Y[tok * p.q.d + row] = f32_to_bf16_bits(rowsum[e] + adp[e]);
  }
}

// Host-side limits of this kernel for a group: M * k staged, rows and DQ
// scales per CTA, total adapter rows.
inline bool gv_fits(int M, int64_t k, int64_t ntiles, int64_t rtot, int grid) {
  if (M < 1 || M > kGvMaxM || static_cast<int64_t>(M) * k > kGvMaxXElems || k > 64 * kGvMaxNb) return false;
  const int64_t tiles_cta = (ntiles + grid - 1) / grid;
  if (tiles_cta * kGvRows * M > kGvMaxRowVals) return false;
  // DQ scales: rows * nb / 256 + 2 per projection in the range (at most 8)
  if (tiles_cta * kGvRows * (k >> 6) / 256 + 2 * kGvMaxGroup > kGvMaxSig) return false;
  return rtot * M <= kGvMaxU;
}

}  // namespace qn
