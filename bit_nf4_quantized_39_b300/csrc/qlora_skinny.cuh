// qlora_skinny.cuh -- fused QLoRA forward for a few tokens (M <= 16) of a
// group of projections of one input:
//
//   Y_g = X deq(Q_g)^T + s_g (X A_g^T) B_g^T      X: M x k bf16, Q_g: d_g x k NF4
//
// ("PEFT course notes" §2.2, h = Wx + BAx; "QLoRA paper summary": the frozen
// weight is 4-bit NF4 with blockwise constants.)  The call is bound by the
// bytes of the packed weights, so the design goal is to keep HBM busy with
// as few instructions per weight byte as possible and no grid-wide waits.
//
// Two kernels, chained with programmatic dependent launch (PDL):
//
// 1. skinny_u_kernel: u[t, j] = s_g A_g[j] . X[t] for every adapter row j of
//    the group and token t; one CTA per (j, t).  It reads nothing before
//    waiting on the previous kernel: X and A (an adapter that an optimiser
//    step may just have written) both come after griddepcontrol.wait.  The
//    weight kernel's own early reads (codes and block constants) are safe
//    because this kernel always runs between it and any earlier writer and
//    waits for that writer to complete before it exits.
// 2. skinny_kernel: the weights, one CTA per SM.  Work items are row groups
//    of 16 rows of one projection (the M side of an m16n8k16 MMA).  A
//    producer warp streams each row group's codes with TMA in stages of 16
//    rows x 16 blocks (8 KiB, four 128-byte boxes with the 128-byte swizzle)
//    through a 10-stage shared-memory ring (80 KiB in flight per SM).
//    Sixteen consumer warps take one 64-block of every stage each.  A lane (group g, thread t) reads 8 code
//    bytes of rows g and g+8 (elements 16t .. 16t+15 of its block; the
//    swizzle makes the reads conflict-free); every byte becomes one bf16x2
//    A-fragment register with one byte permute (address) and one shared-
//    memory load from a per-lane replicated byte-pair table of the 16 levels.
//    Four MMAs against the matching X fragment (tokens are the N columns, so
//    every M <= 8 costs the same; M <= 16 takes a second column tile) give
//    the block's dot products, scaled by the block constants in fp32.  The
//    row group's block constants (int8 codes, or fp32 absmax) arrive with its
//    first stage as one bulk copy into a shared-memory tile; the group scale
//    sigma comes through L1.  Without X staged in shared memory, the X
//    fragments of the next stage are loaded (through L2) while the current
//    stage is decoded.  The MMA's k order is a permutation of the block's elements, the same one for
//    A and X, so the sum is unchanged.  At the end of a row group each warp
//    writes its partial sums to a shared-memory ring slot and arrives on the
//    slot's mbarrier; the group's finisher warp (group index mod 8) sums the
//    8 partials in a fixed order, adds u[t] . B[row] on the MMA (B rows
//    prefetched with cp.async when the group starts) and writes bf16 Y.
//    The producer streams and the consumers build the table before
//    griddepcontrol.wait; X, u and Y are touched only after it.  Neither
//    kernel issues launch_dependents: a dependent's wait is only guaranteed
//    to see writes made before the trigger (inside a CUDA graph a chained
//    call was observed to read its input early when the trigger came first),
//    and a CTA that never issues it counts as triggering when it exits.
//
// Every mbarrier wait is bounded (QN_DEV_TIMEOUT, then the warp winds down);
// there is no wait on another CTA.
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace qn {

constexpr int kSkConsumers = 16;                     // consumer warps (one 64-block of each stage each)
constexpr int kSkItems = 16 / kSkConsumers;          // 64-blocks per consumer warp and stage
constexpr int kSkProducer = kSkConsumers;            // the TMA producer warp
constexpr int kSkThreads = (kSkConsumers + 1) * 32;
constexpr int kSkRows = 16;                          // rows per row group (MMA M)
constexpr int kSkStageBlocks = 16;                   // 64-blocks per stage
constexpr int kSkStageBytes = kSkRows * kSkStageBlocks * 32;  // 8 KiB of codes
constexpr int kSkBoxBytes = 128;                     // TMA box width: one swizzle span, 4 blocks
constexpr int kSkStages = 10;                        // stage ring depth (80 KiB in flight)
constexpr int kSkMaxNb = 256;                        // 64-blocks per row (k <= 16384)
constexpr int kSkCTiles = 3;                         // int8 block-constant tiles (row groups in flight)
constexpr int kSkCTileBytes = kSkRows * kSkMaxNb;    // one group's int8 constants
constexpr int kSkSlots = 2;                          // partial-sum ring slots
constexpr int kSkScratchR = 64;                      // ranks whose B rows are prefetched to shared memory
constexpr int kSkScratchSlots = 4;                   // B-row scratch slots (finishers of groups it mod 4)
constexpr int kSkUBytes = 4 * 1024;                  // u staged in shared memory up to this size
constexpr int kSkMaxM = 16;
constexpr int kSkMaxGroup = 8;
constexpr int kSkLutBytes = 256 * 256;               // entry b of lane l at byte 256 b + 4 l
constexpr int kSkUThreads = 256;

struct SkProj {
  CUtensorMap tmap;    // codes as uint32 [d][k / 8], box {32, 16}, 128-byte swizzle
  QnNF4View q;
  const uint16_t *A;   // r x k bf16
  const uint16_t *B;   // d x r bf16
  uint16_t *Y;         // M x d bf16
  int r;
  float s;
  int64_t group_off;   // first row group of this projection in the group's list
  int64_t u_off;       // first adapter row (column of u)
};
struct SkGroup {
  SkProj p[kSkMaxGroup];
  int n;
  int M;
  int64_t k;
  int64_t ngroups;     // total row groups
  int64_t rtot;        // total adapter rows (row length of u)
  const uint16_t *X;   // M x k bf16
  float *u;            // M x rtot fp32
};

__host__ __device__ constexpr size_t sk_part_bytes(int MT) {
  return static_cast<size_t>(kSkSlots) * kSkConsumers * kSkRows * 8 * MT * sizeof(float);
}
constexpr size_t kSkScratchBytes = static_cast<size_t>(kSkScratchSlots) * kSkRows * kSkScratchR * 2;
constexpr size_t kSkTileBytes = static_cast<size_t>(kSkCTiles) * kSkCTileBytes;
constexpr size_t kSkBarBytes = 256;
// Shared memory: stage ring, table, block-constant tiles, partial ring, B-row
// scratch, barriers, u, then X when staged (plus slack to align the ring).
__host__ __device__ constexpr size_t sk_smem_bytes(int MT, int M, int64_t k, bool xs) {
  return 1024 + static_cast<size_t>(kSkStages) * kSkStageBytes + kSkLutBytes + kSkTileBytes + sk_part_bytes(MT) +
         kSkScratchBytes + kSkBarBytes + kSkUBytes + (xs ? static_cast<size_t>(M) * k * 2 : 0);
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulator.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// Kernel 1: u[t, j] = s_g * A_g[j - u_off_g] . X[t]      grid (rtot, M)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSkUThreads)
skinny_u_kernel(const __grid_constant__ SkGroup g) {
  const int64_t j = blockIdx.x;
  const int t = blockIdx.y;
  const int64_t k = g.k;
  int pi = 0;
#pragma unroll
  for (int i = 1; i < kSkMaxGroup; ++i)
    if (i < g.n && j >= g.p[i].u_off) pi = i;
  const SkProj &p = g.p[pi];
  const uint4 *arow = reinterpret_cast<const uint4 *>(p.A + (j - p.u_off) * k);
  const uint4 *xrow = reinterpret_cast<const uint4 *>(g.X + static_cast<int64_t>(t) * k);
  const int64_t nvec = k >> 3;
  constexpr int kPer = 8;
  float acc = 0.f;
  pdl_wait();  // X and A may be written by the kernel before this one
  for (int64_t base = 0; base < nvec; base += static_cast<int64_t>(kSkUThreads) * kPer) {
    uint4 a[kPer], x[kPer];
#pragma unroll
    for (int v = 0; v < kPer; ++v) {
      const int64_t c = base + v * kSkUThreads + threadIdx.x;
      a[v] = (c < nvec) ? arow[c] : make_uint4(0u, 0u, 0u, 0u);
      x[v] = (c < nvec) ? xrow[c] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int v = 0; v < kPer; ++v) {
      const uint32_t aw[4] = {a[v].x, a[v].y, a[v].z, a[v].w};
      const uint32_t xw[4] = {x[v].x, x[v].y, x[v].z, x[v].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__uint_as_float(aw[e] << 16), __uint_as_float(xw[e] << 16), acc);
        acc = fmaf(__uint_as_float(aw[e] & 0xFFFF0000u), __uint_as_float(xw[e] & 0xFFFF0000u), acc);
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  __shared__ float red[kSkUThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kSkUThreads / 32; ++w) s += red[w];
    g.u[static_cast<int64_t>(t) * g.rtot + j] = p.s * s;
  }
}

// ---------------------------------------------------------------------------
// Kernel 2: the weights.
// ---------------------------------------------------------------------------
// Shared-memory byte offset of the table entry for byte `i` of `w` in this
// lane's column: (byte << 8) | (lane << 2), one byte permute.
__device__ __forceinline__ uint32_t sk_lut_off(uint32_t w, uint32_t lane4, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(w), "r"(lane4), "r"(sel));
  return r;
}

// Tensor map of projection pi, addressed at a compile-time offset into the
// kernel parameters (a run-time index into the parameter array is slower).
__device__ __forceinline__ const CUtensorMap *sk_map(const SkGroup &g, int pi) {
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

template <int MT, bool XS>
__global__ void __launch_bounds__(kSkThreads, 1)
skinny_kernel(const __grid_constant__ SkGroup g) {
  extern __shared__ unsigned char sk_raw[];
  unsigned char *base = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(sk_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char *ring = base;
  unsigned char *lut = ring + kSkStages * kSkStageBytes;
  unsigned char *ctile = lut + kSkLutBytes;
  float *part = reinterpret_cast<float *>(ctile + kSkTileBytes);
  uint16_t *bscr = reinterpret_cast<uint16_t *>(reinterpret_cast<unsigned char *>(part) + sk_part_bytes(MT));
  uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<unsigned char *>(bscr) + kSkScratchBytes);
  uint64_t *st_full = bars, *st_empty = bars + kSkStages;
  uint64_t *pt_full = bars + 2 * kSkStages, *pt_empty = pt_full + kSkSlots, *tile_free = pt_empty + kSkSlots;
  volatile int *abort = reinterpret_cast<volatile int *>(tile_free + kSkCTiles);
  float *us = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(bars) + kSkBarBytes);
  uint16_t *xs = reinterpret_cast<uint16_t *>(reinterpret_cast<unsigned char *>(us) + kSkUBytes);

  constexpr int NC = 8 * MT;  // partial columns (tokens) per row
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t k = g.k;
  const int nb = static_cast<int>(k >> 6);
  const int nst = (nb + kSkStageBlocks - 1) / kSkStageBlocks;  // stages per row group
  const int M = g.M;
  const int G = gridDim.x;
  const int ngroups = static_cast<int>(g.ngroups);

  if (tid == 0) {
    for (int i = 0; i < kSkStages; ++i) {
      mbar_init(smem_u32(&st_full[i]), 1);
      mbar_init(smem_u32(&st_empty[i]), kSkConsumers);
    }
    for (int i = 0; i < kSkSlots; ++i) {
      mbar_init(smem_u32(&pt_full[i]), kSkConsumers);
      mbar_init(smem_u32(&pt_empty[i]), 1);
    }
    for (int i = 0; i < kSkCTiles; ++i) mbar_init(smem_u32(&tile_free[i]), kSkConsumers);
    *abort = 0;
    mbar_fence_init();
  }
  __syncthreads();

  auto proj_of = [&](int rg) {
    int i = 0;
#pragma unroll
    for (int t = 1; t < kSkMaxGroup; ++t)
      if (t < g.n && rg >= g.p[t].group_off) i = t;
    return i;
  };
  // Bytes of a row group's int8 block constants that one bulk copy brings
  // into its tile (a multiple of 16; the rest, in the last row group only,
  // is read from global memory).  0 for fp32 absmax constants (read through L1).
  auto ctile_bytes = [&](const QnNF4View &q, int row0) -> uint32_t {
    if (!q.dq || (reinterpret_cast<uintptr_t>(q.absmax_q) & 15u)) return 0u;  // bulk copies need 16-byte alignment
    const int64_t nrows = (q.d - row0 < kSkRows) ? q.d - row0 : static_cast<int64_t>(kSkRows);
    return static_cast<uint32_t>(nrows * nb) & ~15u;
  };

  if (warp == kSkProducer) {
    // ================================ producer =================================
    // Streams every stage of this CTA's row groups; the weights do not depend
    // on the kernel before, so this starts before griddepcontrol.wait.
    if (lane == 0) {
      for (int i = 0; i < g.n; ++i) tma_prefetch_desc(sk_map(g, i));
      uint32_t qi = 0;
      bool ok = true;
      for (int it = 0, rg = blockIdx.x; rg < ngroups && ok; ++it, rg += G) {
        const int pi = proj_of(rg);
        const QnNF4View &q = g.p[pi].q;
        const int row0 = static_cast<int>(rg - g.p[pi].group_off) * kSkRows;
        const CUtensorMap *map = sk_map(g, pi);
        for (int s = 0; s < nst; ++s, ++qi) {
          const uint32_t slot = qi % kSkStages;
          if (qi >= kSkStages && !mbar_wait(smem_u32(&st_empty[slot]), ((qi / kSkStages) - 1) & 1, abort)) {
            ok = false;
            break;
          }
          uint32_t cbytes = 0;
          if (s == 0) {
            if (it >= kSkCTiles &&
                !mbar_wait(smem_u32(&tile_free[it % kSkCTiles]), ((it / kSkCTiles) - 1) & 1, abort)) {
              ok = false;
              break;
            }
            cbytes = ctile_bytes(q, row0);
          }
          const uint32_t full = smem_u32(&st_full[slot]);
          mbar_arrive_expect_tx(full, kSkStageBytes + cbytes);
          if (cbytes)
            bulk_load(smem_u32(ctile + (it % kSkCTiles) * kSkCTileBytes), q.absmax_q + static_cast<int64_t>(row0) * nb,
                      cbytes, full);
#pragma unroll
          for (int j = 0; j < kSkStageBytes / (kSkRows * kSkBoxBytes); ++j)
            tma_load_2d(smem_u32(ring + slot * kSkStageBytes + j * kSkRows * kSkBoxBytes), map,
                        (s * kSkStageBlocks + 4 * j) * 8, row0, full);
        }
      }
      // Every copy this CTA started lands before it may retire (a drain wait:
      // not cut short when another warp has given up).
      for (uint32_t r = (qi > kSkStages ? qi - kSkStages : 0); r < qi; ++r)
        mbar_wait_drain(smem_u32(&st_full[r % kSkStages]), (r / kSkStages) & 1);
    }
    return;
  }

  // ================================= consumers ==================================
  const int gq = lane >> 2, tq = lane & 3;  // MMA group id, thread in group
  const int cw = warp;                      // takes block cw of every stage
  const uint32_t lane4 = static_cast<uint32_t>(lane) << 2;
  {
    // entry b of lane l: bf16(level[b & 15]) | bf16(level[b >> 4]) << 16.
    // Thread tid writes the words of entries b = (tid >> 5) + 16 n of lane
    // tid & 31 (16 consumer warps: b & 15 = tid >> 5, b >> 4 = n).
    static_assert(kSkConsumers == 16, "table build assumes 16 consumer warps");
    const int b0 = tid >> 5, l = tid & 31;
    const uint32_t lo = f32_to_bf16_bits(c_nf4_levels[b0]);
    uint32_t *lw = reinterpret_cast<uint32_t *>(lut);
#pragma unroll
    for (int n = 0; n < 16; ++n) lw[(b0 + 16 * n) * 64 + l] = lo | (f32_to_bf16_bits(c_nf4_levels[n]) << 16);
  }
  pdl_wait();  // X and u are written by the kernels before this one
  const int64_t nu = static_cast<int64_t>(M) * g.rtot;
  const bool u_smem = nu * 4 <= kSkUBytes;
  if (u_smem)
    for (int64_t i = tid; i < nu; i += kSkConsumers * 32) us[i] = g.u[i];
  if (XS) {
    const int64_t nvec = static_cast<int64_t>(M) * k / 8;
    for (int64_t i = tid; i < nvec; i += kSkConsumers * 32)
      reinterpret_cast<uint4 *>(xs)[i] = reinterpret_cast<const uint4 *>(g.X)[i];
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kSkConsumers * 32) : "memory");  // table, X and u ready
  const float *ubase = u_smem ? us : g.u;

  float acc[MT][4];
  bool ok = true;
  uint32_t q = 0;  // stages consumed

  for (int it = 0, rg = blockIdx.x; rg < ngroups && ok; ++it, rg += G) {
    const int pi = proj_of(rg);
    const SkProj &p = g.p[pi];
    const QnNF4View &qv = p.q;
    const int row0 = static_cast<int>(rg - p.group_off) * kSkRows;
    const bool finisher = (it % kSkConsumers) == cw;
    uint16_t *my_scr = bscr + (it % kSkScratchSlots) * (kSkRows * kSkScratchR);
    if (finisher && p.r <= kSkScratchR) {
      // B rows of the group (contiguous, 16-byte aligned since row0 is a
      // multiple of 16) into a scratch slot, used at the group's end.
      const int64_t nrows = (qv.d - row0 < kSkRows) ? qv.d - row0 : static_cast<int64_t>(kSkRows);
      const int64_t bytes = nrows * p.r * 2;
      const unsigned char *src = reinterpret_cast<const unsigned char *>(p.B + static_cast<int64_t>(row0) * p.r);
      const uint32_t dst = smem_u32(my_scr);
      for (int64_t o = static_cast<int64_t>(lane) * 16; o + 16 <= bytes; o += 32 * 16) cp_async16(dst + o, src + o);
      cp_async_commit();
      const int64_t tail = bytes & ~static_cast<int64_t>(15);
      for (int64_t o = tail + lane * 2; o < bytes; o += 64) my_scr[o >> 1] = *reinterpret_cast<const uint16_t *>(src + o);
    }
    const bool dq = qv.dq != 0;
    const float mu = dq ? __ldg(qv.absmax_mean) : 0.f;
    const int8_t *ct = reinterpret_cast<const int8_t *>(ctile + (it % kSkCTiles) * kSkCTileBytes);
    const uint32_t cbytes = ctile_bytes(qv, row0);
    const bool row_ok[2] = {row0 + gq < qv.d, row0 + gq + 8 < qv.d};
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;

    // ---- the group's stages: this warp takes block s*16 + cw.
    // What comes from global memory through L2 is loaded one stage ahead,
    // while the stage before is decoded: the X fragments (without staged X)
    // and the per-block value behind the block constant (the DQ group scale,
    // or the fp32 absmax).
    uint4 xc[kSkItems][MT][2], xn[kSkItems][MT][2];
    float sc[kSkItems][2], sn[kSkItems][2];
    auto prefetch = [&](int s2, uint4 (&xo)[kSkItems][MT][2], float (&so)[kSkItems][2]) {
#pragma unroll
      for (int t = 0; t < kSkItems; ++t) {
        const int b = s2 * kSkStageBlocks + cw + kSkConsumers * t;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int tok = gq + 8 * mt;
          xo[t][mt][0] = make_uint4(0u, 0u, 0u, 0u);
          xo[t][mt][1] = xo[t][mt][0];
          if (!XS && s2 < nst && b < nb && tok < M) {
            const int64_t e = static_cast<int64_t>(tok) * k + static_cast<int64_t>(b) * 64 + tq * 16;
            xo[t][mt][0] = __ldcg(reinterpret_cast<const uint4 *>(g.X + e));
            xo[t][mt][1] = __ldcg(reinterpret_cast<const uint4 *>(g.X + e + 8));
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float v = 0.f;
          if (s2 < nst && row_ok[h] && b < nb) {
            const int64_t blk = static_cast<int64_t>(row0 + gq + 8 * h) * nb + b;
            v = dq ? __ldcg(qv.absmax_scale + (blk >> 8)) : __ldcg(qv.absmax + blk);
          }
          so[t][h] = v;
        }
      }
    };
    prefetch(0, xc, sc);
    for (int s = 0; s < nst; ++s, ++q) {
      prefetch(s + 1, xn, sn);
      const uint32_t slot = q % kSkStages;
      ok = mbar_wait(smem_u32(&st_full[slot]), (q / kSkStages) & 1, abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const unsigned char *stage = ring + slot * kSkStageBytes;
      uint32_t a[kSkItems][2][8];  // [item][row half][byte]: bf16 pair of elements 16 tq + 2 byte, +1
      float m[kSkItems][2];        // [item][row half]: block constants
      int bi[kSkItems];
#pragma unroll
      for (int t = 0; t < kSkItems; ++t) {
        const int cb = cw + kSkConsumers * t;  // block of the stage
        const int b = s * kSkStageBlocks + cb;
        bi[t] = b;
        // Code bytes 8 tq .. 8 tq + 7 of block b for rows gq and gq + 8: box
        // cb / 4, 32-byte block cb % 4 inside the 128-byte row, 16-byte chunk
        // index XOR (row mod 8) from the 128-byte swizzle.
        const int chunk = 2 * (cb & 3) + (tq >> 1);
        const uint32_t off =
            (cb >> 2) * (kSkRows * kSkBoxBytes) + gq * kSkBoxBytes + ((chunk ^ gq) << 4) + ((tq & 1) << 3);
        const uint2 c0 = *reinterpret_cast<const uint2 *>(stage + off);
        const uint2 c1 = *reinterpret_cast<const uint2 *>(stage + off + 8 * kSkBoxBytes);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          a[t][0][i] = *reinterpret_cast<const uint32_t *>(lut + sk_lut_off(c0.x, lane4, 0x5504u | (i << 4)));
          a[t][0][4 + i] = *reinterpret_cast<const uint32_t *>(lut + sk_lut_off(c0.y, lane4, 0x5504u | (i << 4)));
          a[t][1][i] = *reinterpret_cast<const uint32_t *>(lut + sk_lut_off(c1.x, lane4, 0x5504u | (i << 4)));
          a[t][1][4 + i] = *reinterpret_cast<const uint32_t *>(lut + sk_lut_off(c1.y, lane4, 0x5504u | (i << 4)));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float mm = 0.f;
          if (row_ok[h] && b < nb) {
            const int lr = gq + 8 * h;
            const uint32_t o = static_cast<uint32_t>(lr * nb + b);
            const int64_t blk = static_cast<int64_t>(row0 + lr) * nb + b;
            if (dq) {
              const int qc = (o < cbytes) ? static_cast<int>(ct[o]) : static_cast<int>(__ldg(qv.absmax_q + blk));
              mm = dq_absmax(static_cast<int8_t>(qc), sc[t][h], mu);
            } else {
              mm = sc[t][h];
            }
          }
          m[t][h] = mm;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&st_empty[slot]));  // codes are in registers now
#pragma unroll
      for (int t = 0; t < kSkItems; ++t) {
        const int b = bi[t];
        if (b >= nb) continue;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          // X fragment: token gq + 8 mt, elements 16 tq .. 16 tq + 15 of block b
          uint4 x0 = xc[t][mt][0], x1 = xc[t][mt][1];
          const int tok = gq + 8 * mt;
          if (XS && tok < M) {
            const int64_t e = static_cast<int64_t>(tok) * k + static_cast<int64_t>(b) * 64 + tq * 16;
            x0 = *reinterpret_cast<const uint4 *>(xs + e);
            x1 = *reinterpret_cast<const uint4 *>(xs + e + 8);
          }
          const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          float dsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int st = 0; st < 4; ++st)
            mma_bf16_16816(dsum, a[t][0][2 * st], a[t][1][2 * st], a[t][0][2 * st + 1], a[t][1][2 * st + 1],
                           xw[2 * st], xw[2 * st + 1]);
          acc[mt][0] = fmaf(dsum[0], m[t][0], acc[mt][0]);
          acc[mt][1] = fmaf(dsum[1], m[t][0], acc[mt][1]);
          acc[mt][2] = fmaf(dsum[2], m[t][1], acc[mt][2]);
          acc[mt][3] = fmaf(dsum[3], m[t][1], acc[mt][3]);
        }
      }
#pragma unroll
      for (int t = 0; t < kSkItems; ++t) {
        sc[t][0] = sn[t][0];
        sc[t][1] = sn[t][1];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          xc[t][mt][0] = xn[t][mt][0];
          xc[t][mt][1] = xn[t][mt][1];
        }
      }
    }
    if (!ok) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&tile_free[it % kSkCTiles]));  // done with the constants tile

    // ---- end of the group: partial sums into ring slot it % 2 -----------------
    const int slot = it % kSkSlots;
    const uint32_t full = smem_u32(&pt_full[slot]), empty = smem_u32(&pt_empty[slot]);
    if (it >= kSkSlots) ok = mbar_wait(empty, ((it / kSkSlots) - 1) & 1, abort);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    {
      float *pw = part + ((slot * kSkConsumers + cw) * kSkRows) * NC;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        pw[gq * NC + 8 * mt + 2 * tq] = acc[mt][0];
        pw[gq * NC + 8 * mt + 2 * tq + 1] = acc[mt][1];
        pw[(gq + 8) * NC + 8 * mt + 2 * tq] = acc[mt][2];
        pw[(gq + 8) * NC + 8 * mt + 2 * tq + 1] = acc[mt][3];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(full);
    if (!finisher) continue;
    // ---- finisher: sum the partials, add the adapter term, write Y -----------
    ok = mbar_wait(full, (it / kSkSlots) & 1, abort);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    const int64_t d = qv.d;
    // y in the MMA accumulator layout: rows gq, gq+8; tokens 2 tq, 2 tq + 1 (+8 mt)
    float y[MT][4];
    {
      const float *ps = part + (slot * kSkConsumers * kSkRows) * NC;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = gq + 8 * (e >> 1), col = 8 * mt + 2 * tq + (e & 1);
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < kSkConsumers; ++w) v += ps[(w * kSkRows + row) * NC + col];
          y[mt][e] = v;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty);
    // Adapter term s (X A^T) B^T = u B^T on the MMA: A = B rows (bf16), the
    // column operand = u split into bf16 hi + lo (about 16 significant bits).
    const bool scr = p.r <= kSkScratchR;
    if (scr) {
      cp_async_wait_all();
      __syncwarp();
    }
    const uint16_t *brow0 = p.B + static_cast<int64_t>(row0 + gq) * p.r;
    const uint16_t *brow1 = p.B + static_cast<int64_t>(row0 + gq + 8) * p.r;
    for (int j0 = 0; j0 < p.r; j0 += 16) {
      uint32_t af[4];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {  // af[qq]: row gq + 8 (qq & 1), columns j0 + 2 tq + 8 (qq >> 1) + {0, 1}
        const int j = j0 + 2 * tq + 8 * (qq >> 1);
        const int rr = gq + 8 * (qq & 1);
        uint32_t lo = 0u, hi = 0u;
        if (scr) {
          if (j < p.r) lo = my_scr[rr * p.r + j];
          if (j + 1 < p.r) hi = my_scr[rr * p.r + j + 1];
        } else if (row_ok[qq & 1]) {
          const uint16_t *br = (qq & 1) ? brow1 : brow0;
          if (j < p.r) lo = br[j];
          if (j + 1 < p.r) hi = br[j + 1];
        }
        af[qq] = lo | (hi << 16);
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int tok = gq + 8 * mt;
        uint32_t bh[2], bl[2];
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {  // column rows j0 + 2 tq + 8 qq + {0, 1}
          const int j = j0 + 2 * tq + 8 * qq;
          float u0 = 0.f, u1 = 0.f;
          if (tok < M) {
            const float *ut = ubase + static_cast<int64_t>(tok) * g.rtot + p.u_off;
            if (j < p.r) u0 = ut[j];
            if (j + 1 < p.r) u1 = ut[j + 1];
          }
          const uint32_t h0 = f32_to_bf16_bits(u0), h1 = f32_to_bf16_bits(u1);
          bh[qq] = h0 | (h1 << 16);
          bl[qq] = static_cast<uint32_t>(f32_to_bf16_bits(u0 - bf16_bits_to_f32(h0))) |
                   (static_cast<uint32_t>(f32_to_bf16_bits(u1 - bf16_bits_to_f32(h1))) << 16);
        }
        mma_bf16_16816(y[mt], af[0], af[1], af[2], af[3], bh[0], bh[1]);
        mma_bf16_16816(y[mt], af[0], af[1], af[2], af[3], bl[0], bl[1]);
      }
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t row = row0 + gq + 8 * (e >> 1);
        const int tok = 8 * mt + 2 * tq + (e & 1);
        if (tok < M && row < d) p.Y[static_cast<int64_t>(tok) * d + row] = f32_to_bf16_bits(y[mt][e]);
      }
    }
  }
  cp_async_wait_all();  // a warp that left early may still have a B-row prefetch in flight
}

}  // namespace qn
