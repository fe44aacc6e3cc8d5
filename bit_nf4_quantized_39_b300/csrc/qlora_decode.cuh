// qlora_decode.cuh -- single-token (M = 1) fused QLoRA forward of a group of
// projections of one input, in one kernel:
//
//   Y_g = x deq(Q_g)^T + s_g (x A_g^T) B_g^T      x: 1 x k bf16, Q_g: d_g x k NF4
//
// ("PEFT course notes" §2.2, h = Wx + BAx; "QLoRA paper summary": the frozen
// weight is 4-bit NF4.)  A single projection is the group of one; several
// projections of the same activation (query/key/value, gate/up) share one
// launch so that their memory round trips overlap.  The call is bound by the
// bytes of the packed weights; at decode sizes (8-45 MB per launch) what
// limits it is how many bytes each SM keeps in flight and how many dependent
// round trips lie on the longest path, so:
//
// * persistent grid (every CTA resident, at least one per SM);
// * every weight is cut into units of 2 whole rows; the units of all
//   projections form one list; unit u goes to warp slot u mod W with slots
//   interleaved across CTAs, so every SM gets an equal share;
// * a warp walks the 1024-column lane steps of its units as one flat
//   sequence and keeps the loads of the next kDecDepth steps in flight, across
//   unit boundaries, so a finishing unit never drains the pipeline;
// * decode: x is staged once per CTA in shared memory as fp32, lane-
//   interleaved so that each lane's 32-element chunk is read with
//   conflict-free 128-bit loads; two codes at a time are looked up in a
//   byte-pair table of fp32 level pairs replicated per lane (entry b of lane
//   l at byte 256 b + 8 l: one byte permute forms the address, and a warp
//   never conflicts on a bank) and multiplied into packed fp32x2
//   accumulators (fma.rn.f32x2); each 32-element partial is scaled by its
//   64-block constant;
// * a unit is a whole row, so its sum is complete in one warp (no cross-warp
//   combine, a fixed summation order): the warp adds u . B[row] and writes
//   bf16 Y;
// * the adapter rows u_g[j] = s_g A_g[j] . x are spread one per warp slot,
//   done right after x is staged with all their loads in flight; each bumps a
//   ready counter (release) that finishing warps wait on (acquire, bounded
//   spin, no trap) before their first adapter term.
//
// Workspace: the two counters live in the caller's zero area (zero before
// the first call; the last CTA to leave returns them to zero); u lives after
// it.
#pragma once

#include "common.cuh"

namespace qn {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecRows = 2;            // weight rows per unit (whole rows)
constexpr int kDecDepth = 4;           // lane steps whose loads are in flight per warp
constexpr int kDecLutBytes = 256 * 256;  // entry b of lane l: fp32 pair at byte 256 b + 8 l
constexpr int kDecMaxK = 16384;
constexpr unsigned kDecSpinLimit = 1u << 22;
// Zero-area words: adapter rows done, CTAs done.
constexpr int kDecFlagReady = 0, kDecFlagExit = 1;
constexpr int kDecMaxGroup = 8;

// One projection of a group (device pointers; k is shared by the group).
struct DecProj {
  QnNF4View q;
  const uint16_t *A;   // r x k bf16
  const uint16_t *B;   // d x r bf16
  uint16_t *Y;         // d bf16
  int r;
  float s;
  int64_t unit_off;    // first unit of this projection in the group's list
  int64_t u_off;       // first adapter row (element of u)
};
struct DecGroup {
  DecProj p[kDecMaxGroup];
  int n;
  int64_t k;
  int64_t nunits, nadapter;  // totals: weight units, adapter rows
  const uint16_t *X;
};

// Staging covers whole 1024-element steps so that ragged tails read zeros.
__host__ __device__ constexpr int64_t dec_xs_floats(int64_t k) { return qn_ceil_div(k, 1024) * 1024; }
__host__ __device__ constexpr size_t dec_smem_bytes(int64_t k) {
  return kDecLutBytes + sizeof(float) * dec_xs_floats(k);
}

__device__ __forceinline__ unsigned long long pack_f2(float lo, float hi) {
  unsigned long long v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
  return v;
}
__device__ __forceinline__ float sum_f2(unsigned long long v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}
// acc += a * b on both halves (packed fp32x2 FMA, sm_100+).
__device__ __forceinline__ void ffma2(unsigned long long &acc, unsigned long long a, unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// Position of element e of x in the lane-interleaved staging buffer: the
// 32-element chunk c = e/32 belongs to lane c % 32 at step c / 32; within a
// step, float4 e4 of lane l sits at float4 index (step * 8 + e4) * 32 + l.
__device__ __forceinline__ int64_t dec_xs_index(int64_t e) {
  const int64_t c = e >> 5;
  const int o = static_cast<int>(e & 31);
  return ((((c >> 5) * 8 + (o >> 2)) * 32 + (c & 31)) << 2) + (o & 3);
}

// One lane step of a unit's rows as loaded: code chunks plus the raw constants of
// their 64-block (int8 code and group scale, or the exact absmax).  The
// block constant is formed only when the step is decoded, so that no load
// of a step waits on another.
struct DecStep {
  uint4 w[kDecRows];
  float sc[kDecRows];   // group scale sigma (dq) or exact absmax
  int qv[kDecRows];     // int8 code of the constant (dq)
};

// Loads lane step `st` of the rows starting at row0 (codes and constants).
__device__ __forceinline__ void dec_load_step(const QnNF4View &q, int64_t row0, int64_t st, int lane,
                                              DecStep &out) {
  const int64_t d = q.d, k = q.k;
  const int64_t nchunk = k >> 5, kb = k >> 6;
  const int64_t c = st * 32 + lane;
#pragma unroll
  for (int rr = 0; rr < kDecRows; ++rr) {
    const int64_t row = row0 + rr;
    if (row < d && c < nchunk) {
      out.w[rr] = __ldcs(reinterpret_cast<const uint4 *>(q.codes + row * (k >> 1)) + c);
      const int64_t blk = row * kb + (c >> 1);
      if (q.dq) {
        out.qv[rr] = __ldg(q.absmax_q + blk);
        out.sc[rr] = __ldg(q.absmax_scale + (blk >> 8));
      } else {
        out.qv[rr] = 0;
        out.sc[rr] = __ldg(q.absmax + blk);
      }
    } else {
      out.w[rr] = make_uint4(0x77777777u, 0x77777777u, 0x77777777u, 0x77777777u);  // level 7 = 0.0
      out.qv[rr] = 0;
      out.sc[rr] = 0.f;
    }
  }
}

// Block constant of a loaded step: fp32(fp32(q * sigma) + mu) or the absmax.
__device__ __forceinline__ float dec_step_scale(const DecStep &sp, int rr, bool dq, float mu) {
  return dq ? dq_absmax(static_cast<int8_t>(sp.qv[rr]), sp.sc[rr], mu) : sp.sc[rr];
}

// Adds the dot products of one lane step of a unit's rows with the staged x.
// Each code byte (two elements) costs one byte permute (its table address,
// (byte << 8) | (lane << 3)), one 64-bit shared load (the two fp32 levels)
// and one packed fp32x2 FMA.
__device__ __forceinline__ void dec_compute_step(const DecStep &sp, int64_t st, const float *__restrict__ xs,
                                                 const unsigned char *__restrict__ lut, uint32_t lane8, int lane,
                                                 bool dq, float mu, float (&rsum)[kDecRows]) {
  const float4 *xp = reinterpret_cast<const float4 *>(xs) + st * 8 * 32 + lane;
  unsigned long long acc[kDecRows];
#pragma unroll
  for (int rr = 0; rr < kDecRows; ++rr) acc[rr] = pack_f2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 x0 = xp[(2 * i) * 32], x1 = xp[(2 * i + 1) * 32];
    const unsigned long long xpair[4] = {pack_f2(x0.x, x0.y), pack_f2(x0.z, x0.w), pack_f2(x1.x, x1.y),
                                         pack_f2(x1.z, x1.w)};
#pragma unroll
    for (int rr = 0; rr < kDecRows; ++rr) {
      const uint32_t word = (i == 0) ? sp.w[rr].x : (i == 1) ? sp.w[rr].y : (i == 2) ? sp.w[rr].z : sp.w[rr].w;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        uint32_t off;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(off) : "r"(word), "r"(lane8), "r"(0x5504u | (b << 4)));
        ffma2(acc[rr], *reinterpret_cast<const unsigned long long *>(lut + off), xpair[b]);
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < kDecRows; ++rr) rsum[rr] = fmaf(sum_f2(acc[rr]), dec_step_scale(sp, rr, dq, mu), rsum[rr]);
}

// A[j, e0 .. e0 + 8) . x[e0 .. e0 + 8) (the lane's 8 A values in av).
__device__ __forceinline__ float dec_adapter_unit(const uint4 &av, int64_t e0, const float *__restrict__ xs) {
  const float4 x0 = *reinterpret_cast<const float4 *>(xs + dec_xs_index(e0));
  const float4 x1 = *reinterpret_cast<const float4 *>(xs + dec_xs_index(e0 + 4));
  float acc = 0.f;
  acc = fmaf(__uint_as_float(av.x << 16), x0.x, acc);
  acc = fmaf(__uint_as_float(av.x & 0xFFFF0000u), x0.y, acc);
  acc = fmaf(__uint_as_float(av.y << 16), x0.z, acc);
  acc = fmaf(__uint_as_float(av.y & 0xFFFF0000u), x0.w, acc);
  acc = fmaf(__uint_as_float(av.z << 16), x1.x, acc);
  acc = fmaf(__uint_as_float(av.z & 0xFFFF0000u), x1.y, acc);
  acc = fmaf(__uint_as_float(av.w << 16), x1.z, acc);
  acc = fmaf(__uint_as_float(av.w & 0xFFFF0000u), x1.w, acc);
  return acc;
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Index of the projection that owns list position `pos` given the
// per-projection offsets `off` (ascending, off[0] = 0).
template <typename F>
__device__ __forceinline__ int dec_find(const DecGroup &g, int64_t pos, F off) {
  int i = 0;
#pragma unroll
  for (int t = 1; t < kDecMaxGroup; ++t)
    if (t < g.n && pos >= off(g.p[t])) i = t;
  return i;
}

__global__ void __launch_bounds__(kDecThreads, 2)
qlora_decode_kernel(const __grid_constant__ DecGroup g, unsigned int *__restrict__ zero_area, float *__restrict__ u) {
  extern __shared__ __align__(16) unsigned char dec_smem[];
  unsigned char *lut = dec_smem;
  float *xs = reinterpret_cast<float *>(dec_smem + kDecLutBytes);
  const int64_t k = g.k;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lane8 = static_cast<uint32_t>(lane) << 3;
  const int G = gridDim.x;
  const int64_t nsteps = qn_ceil_div(k >> 5, 32);  // 1024-column lane steps per row
  // warp slots interleaved across CTAs: slot = warp * G + cta
  const int64_t wslot = static_cast<int64_t>(warp) * G + blockIdx.x;
  const int64_t W = static_cast<int64_t>(G) * kDecWarps;
  const int64_t nunits = g.nunits;
  auto unit_of = [](const DecProj &p) { return p.unit_off; };
  auto uoff_of = [](const DecProj &p) { return p.u_off; };

  // ---- load cursor: (unit, step) of the next step to load --------------------
  int64_t l_unit = wslot, l_st = 0, l_row0 = 0;
  int l_p = 0;
  if (l_unit < nunits) {
    l_p = dec_find(g, l_unit, unit_of);
    l_row0 = (l_unit - g.p[l_p].unit_off) * kDecRows;
  }
  auto load_next = [&](DecStep &dst) {
    if (l_unit < nunits) {
      dec_load_step(g.p[l_p].q, l_row0, l_st, lane, dst);
      if (++l_st == nsteps) {
        l_st = 0;
        l_unit += W;
        if (l_unit < nunits) {
          l_p = dec_find(g, l_unit, unit_of);
          l_row0 = (l_unit - g.p[l_p].unit_off) * kDecRows;
        }
      }
    }
  };

  // ---- prologue: x loads first (one round covers k <= 16384), the weight
  // loads behind them, the level-pair table while they are in flight, then x
  // into shared memory and one barrier -------------------------------------------
  constexpr int kPer = 8;  // 16-byte x loads per thread
  static_assert(kPer * kDecThreads * 8 >= kDecMaxK, "one round of x loads must cover k");
  const int64_t nvec = dec_xs_floats(k) / 8;
  uint4 xt[kPer];
#pragma unroll
  for (int v = 0; v < kPer; ++v) {
    const int64_t vi = v * kDecThreads + tid;
    xt[v] = (vi * 8 < k) ? __ldg(reinterpret_cast<const uint4 *>(g.X) + vi) : make_uint4(0u, 0u, 0u, 0u);
  }
  DecStep buf[kDecDepth];
#pragma unroll
  for (int i = 0; i < kDecDepth; ++i) load_next(buf[i]);
#pragma unroll 4
  for (int n = 0; n < 32; ++n) {
    const int b = warp + 8 * n;  // entry b of this lane: (level[b & 15], level[b >> 4]); warp-uniform index
    *reinterpret_cast<float2 *>(lut + 256 * b + 8 * lane) = make_float2(c_nf4_levels[b & 15], c_nf4_levels[b >> 4]);
  }
#pragma unroll
  for (int v = 0; v < kPer; ++v) {
    const int64_t vi = v * kDecThreads + tid;
    if (vi < nvec) {
      const int64_t e = vi * 8;  // 8 consecutive elements: two float4 groups of one lane
      *reinterpret_cast<float4 *>(xs + dec_xs_index(e)) =
          make_float4(__uint_as_float(xt[v].x << 16), __uint_as_float(xt[v].x & 0xFFFF0000u),
                      __uint_as_float(xt[v].y << 16), __uint_as_float(xt[v].y & 0xFFFF0000u));
      *reinterpret_cast<float4 *>(xs + dec_xs_index(e + 4)) =
          make_float4(__uint_as_float(xt[v].z << 16), __uint_as_float(xt[v].z & 0xFFFF0000u),
                      __uint_as_float(xt[v].w << 16), __uint_as_float(xt[v].w & 0xFFFF0000u));
    }
  }
  __syncthreads();  // table and x ready

  // ---- adapter rows: u[j] = s * A[j] . x, one warp slot per row ---------------
  for (int64_t j = wslot; j < g.nadapter; j += W) {
    const DecProj &p = g.p[dec_find(g, j, uoff_of)];
    const uint16_t *arow = p.A + (j - p.u_off) * k;
    float acc = 0.f;
    for (int64_t base = 0; base < k; base += 8 * 256) {
      uint4 t[8];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const int64_t e = base + v * 256 + lane * 8;
        t[v] = (e < k) ? __ldg(reinterpret_cast<const uint4 *>(arow + e)) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const int64_t e = base + v * 256 + lane * 8;
        if (e < k) acc += dec_adapter_unit(t[v], e, xs);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      u[j] = p.s * acc;
      __threadfence();
      atomicAdd(&zero_area[kDecFlagReady], 1u);
    }
  }

  // ---- main loop: the warp's units as one flat sequence of lane steps --------
  int64_t c_unit = wslot, c_st = 0, c_row0 = 0;
  int c_p = 0;
  float mu = 0.f;
  bool c_dq = false;
  // Adapter operands of the current unit, fetched when the unit starts so
  // that finishing it needs no memory round trip: B[row, lane + 32 h] for the
  // unit's rows (ranks up to 64 in registers, larger ones read at the end),
  // and u[lane + 32 h] once the ready counter has been seen.
  constexpr int kPreR = 64;
  float bpre[kDecRows][2];
  float upre[2] = {0.f, 0.f};
  int upre_p = -1;  // projection whose u is in upre
  bool have_u = false;
  auto load_u = [&]() {
    const DecProj &p = g.p[c_p];
#pragma unroll
    for (int h = 0; h < 2; ++h) upre[h] = (lane + 32 * h < p.r) ? __ldcg(u + p.u_off + lane + 32 * h) : 0.f;
    upre_p = c_p;
  };
  auto enter_unit = [&]() {
    if (c_unit < nunits) {
      c_p = dec_find(g, c_unit, unit_of);
      c_row0 = (c_unit - g.p[c_p].unit_off) * kDecRows;
      const DecProj &p = g.p[c_p];
      c_dq = p.q.dq != 0;
      mu = c_dq ? __ldg(p.q.absmax_mean) : 0.f;
#pragma unroll
      for (int rr = 0; rr < kDecRows; ++rr) {
        const int64_t row = c_row0 + rr;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          bpre[rr][h] = (row < p.q.d && lane + 32 * h < p.r) ? bf16_bits_to_f32(__ldg(p.B + row * p.r + lane + 32 * h)) : 0.f;
      }
      if (have_u && upre_p != c_p) load_u();
    }
  };
  enter_unit();
  float rsum[kDecRows];
#pragma unroll
  for (int rr = 0; rr < kDecRows; ++rr) rsum[rr] = 0.f;

  // y = row sum + u . B[row] for the rows of the current unit.
  auto finish_unit = [&]() {
    const DecProj &p = g.p[c_p];
    const int64_t d = p.q.d;
#pragma unroll
    for (int rr = 0; rr < kDecRows; ++rr) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) rsum[rr] += __shfl_xor_sync(0xffffffffu, rsum[rr], off);
    }
    if (!have_u) {
      if (lane == 0) {
        unsigned int spins = 0;
        while (ld_acquire_u32(&zero_area[kDecFlagReady]) < static_cast<unsigned>(g.nadapter)) {
          if (++spins > kDecSpinLimit) { qn_flag_timeout(); break; }
          __nanosleep(32);
        }
      }
      __syncwarp();
      have_u = true;
      load_u();
    } else if (upre_p != c_p) {
      load_u();
    }
    float acc[kDecRows];
#pragma unroll
    for (int rr = 0; rr < kDecRows; ++rr) {
      const int64_t row = c_row0 + rr;
      float a = fmaf(upre[0], bpre[rr][0], upre[1] * bpre[rr][1]);
      if (row < d && p.r > kPreR)
        for (int j = lane + kPreR; j < p.r; j += 32)
          a = fmaf(__ldcg(u + p.u_off + j), bf16_bits_to_f32(p.B[row * p.r + j]), a);
      acc[rr] = a;
    }
#pragma unroll
    for (int rr = 0; rr < kDecRows; ++rr) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[rr] += __shfl_xor_sync(0xffffffffu, acc[rr], off);
    }
    if (lane < kDecRows && c_row0 + lane < d) {
      float y = rsum[0] + acc[0];
#pragma unroll
      for (int rr = 1; rr < kDecRows; ++rr)
        if (lane == rr) y = rsum[rr] + acc[rr];
      p.Y[c_row0 + lane] = f32_to_bf16_bits(y);
    }
#pragma unroll
    for (int rr = 0; rr < kDecRows; ++rr) rsum[rr] = 0.f;
  };

  while (c_unit < nunits) {
#pragma unroll
    for (int i = 0; i < kDecDepth; ++i) {
      if (c_unit < nunits) {
        const DecStep cur = buf[i];
        load_next(buf[i]);
        dec_compute_step(cur, c_st, xs, lut, lane8, lane, c_dq, mu, rsum);
        if (++c_st == nsteps) {
          finish_unit();
          c_st = 0;
          c_unit += W;
          enter_unit();
        }
      }
    }
  }

  // ---- exit: the last CTA returns the counters to zero ------------------------
  __syncthreads();
  if (tid == 0) {
    const unsigned int prev = atomicAdd(&zero_area[kDecFlagExit], 1u);
    if (prev == static_cast<unsigned>(G) - 1u) {
      atomicExch(&zero_area[kDecFlagReady], 0u);
      atomicExch(&zero_area[kDecFlagExit], 0u);
    }
  }
}

}  // namespace qn
