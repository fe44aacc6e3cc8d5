// nf4_codec.cuh -- blockwise NF4 quantise / double-quantise / dequantise kernels.
//
// Method ("QLoRA technical analysis" §2.1; "QLoRA paper summary", NF4 and
// double-quantisation bullets): per 64-element block divide by the block
// absmax and replace each value by its nearest NF4 level; pack two 4-bit codes
// per byte; quantise the fp32 absmax constants again to int8 in groups of 256
// after subtracting their mean.
//
// Kernels
//   nf4_quant_kernel      full 64-blocks: per-warp cp.async ring, shuffle absmax,
//                         IEEE division, threshold count, packed stores,
//                         exact exponent-binned sum of the absmax constants.
//   nf4_quant_tail_kernel the final partial block (n % 64 != 0).
//   nf4_dq_kernel         per 256-group: exact mean from the bins, int8 codes.
//   nf4_dequant_kernel    codes + constants -> fp32 / bf16, warp-contiguous
//                         loads and 128-bit stores.
#pragma once

#include "common.cuh"

namespace qn {

constexpr int kQuantThreads = 512;
constexpr int kNumBins = 256;  // one bin per fp32 exponent field value

// Adds a block absmax to the exponent-binned exact sum: bin e' = max(e, 1)
// accumulates the integer significand (implicit bit included), so that
// sum = sum_e bins[e] * 2^(e - 150).
__device__ __forceinline__ void bin_add_shared(unsigned long long *s_bins, float m) {
  const uint32_t b = __float_as_uint(m);
  const uint32_t e = (b >> 23) & 0xFFu;
  const uint32_t sig = (b & 0x7FFFFFu) | (e ? 0x800000u : 0u);
  if (sig) atomicAdd(&s_bins[e ? e : 1u], static_cast<unsigned long long>(sig));
}

// Register-held part of the same exact sum: a lane folds the constants whose
// bin lies within 4 of a reference bin (the first one it meets) into one
// 64-bit integer in units of bin eref - 4 (significand << (bin - eref + 4));
// others go to the shared bins.  flush adds the integer to bin eref - 4.  The
// fold is used only while every bin stays below 2^63 (nblk <= 2^31).
struct BinFold {
  unsigned long long acc;
  int eref;
};

__device__ __forceinline__ void bin_fold(BinFold &f, unsigned long long *s_bins, float m, bool fold) {
  const uint32_t b = __float_as_uint(m);
  const uint32_t e = (b >> 23) & 0xFFu;
  const uint32_t sig = (b & 0x7FFFFFu) | (e ? 0x800000u : 0u);
  if (!sig) return;
  const int be = e ? static_cast<int>(e) : 1;
  if (fold && f.eref < 0 && be >= 5) f.eref = be;
  const int sh = be - f.eref + 4;
  if (fold && f.eref >= 0 && sh >= 0 && sh <= 8) f.acc += static_cast<unsigned long long>(sig) << sh;
  else atomicAdd(&s_bins[be], static_cast<unsigned long long>(sig));
}

__device__ __forceinline__ void bin_flush(const BinFold &f, unsigned long long *s_bins) {
  if (f.acc) atomicAdd(&s_bins[f.eref - 4], f.acc);
}

// ---------------------------------------------------------------------------
// Exact mean of the absmax constants, rounded once to fp32 (ties to even).
// bins[e] holds sum of significands with exponent field e (bin 1 also holds
// subnormals); the exact sum in units of 2^-149 is sum_e bins[e] << (e - 1),
// a number below 2^320 kept in ten 32-bit limbs.
// ---------------------------------------------------------------------------
constexpr int kLimbs = 10;

__device__ __forceinline__ void limbs_add(uint32_t (&acc)[kLimbs], const uint32_t (&add)[kLimbs]) {
  uint64_t carry = 0;
#pragma unroll
  for (int i = 0; i < kLimbs; ++i) {
    const uint64_t s = static_cast<uint64_t>(acc[i]) + add[i] + carry;
    acc[i] = static_cast<uint32_t>(s);
    carry = s >> 32;
  }
}

// Adds value << shift (value < 2^64, shift <= 253) into the accumulator.
__device__ __forceinline__ void limbs_add_shifted(uint32_t (&acc)[kLimbs], uint64_t value, int shift) {
  const int ls = shift >> 5, bs = shift & 31;
  const uint64_t lo64 = value << bs;                                          // bits 0..63
  const uint32_t hi32 = bs ? static_cast<uint32_t>(value >> (64 - bs)) : 0u;  // bits 64..95
  uint32_t add[kLimbs];
#pragma unroll
  for (int i = 0; i < kLimbs; ++i) {
    uint32_t w = 0;
    if (i == ls) w = static_cast<uint32_t>(lo64);
    else if (i == ls + 1) w = static_cast<uint32_t>(lo64 >> 32);
    else if (i == ls + 2) w = hi32;
    add[i] = w;
  }
  limbs_add(acc, add);
}

// Warp-cooperative exact mean; every lane returns the same fp32.
__device__ float exact_mean_from_bins(const unsigned long long *__restrict__ bins, uint64_t count) {
  const int lane = threadIdx.x & 31;
  uint32_t acc[kLimbs];
#pragma unroll
  for (int i = 0; i < kLimbs; ++i) acc[i] = 0u;
  for (int j = 0; j < kNumBins / 32; ++j) {
    const int e = lane * (kNumBins / 32) + j;
    const unsigned long long s = __ldcg(bins + e);
    if (e >= 1 && s) limbs_add_shifted(acc, s, e - 1);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    uint32_t other[kLimbs];
#pragma unroll
    for (int i = 0; i < kLimbs; ++i) other[i] = __shfl_xor_sync(0xffffffffu, acc[i], off);
    limbs_add(acc, other);
  }
  if (count == 0) return 0.f;
  // Long division by count, most significant limb first.  count < 2^32 uses
  // 64-bit steps; larger counts fall back to bit-serial division.
  uint32_t quo[kLimbs];
  uint64_t rem = 0;
  if (count < (1ull << 32)) {
    for (int i = kLimbs - 1; i >= 0; --i) {
      const uint64_t cur = (rem << 32) | acc[i];
      quo[i] = static_cast<uint32_t>(cur / count);
      rem = cur % count;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kLimbs; ++i) quo[i] = 0u;
    for (int bit = 32 * kLimbs - 1; bit >= 0; --bit) {
      const uint32_t in = (acc[bit >> 5] >> (bit & 31)) & 1u;
      const bool top = (rem >> 63) != 0;  // rem < count < 2^64; 2*rem may need 65 bits
      rem = (rem << 1) | in;
      if (top || rem >= count) {
        rem -= count;
        quo[bit >> 5] |= 1u << (bit & 31);
      }
    }
  }
  // Position of the quotient's top set bit.
  int p = -1;
  for (int i = kLimbs - 1; i >= 0 && p < 0; --i)
    if (quo[i]) p = 32 * i + 31 - __clz(quo[i]);
  // Significand = quotient >> shift, shift = max(p - 23, 0) (2^-149 units).
  const int shift = p > 23 ? p - 23 : 0;
  // 24 quotient bits starting at bit `pos` (they span at most two limbs).
  auto bits_at = [&](int pos) -> uint64_t {
    const int li = pos >> 5, bi = pos & 31;
    const uint64_t lo = quo[li];
    const uint64_t hi = (li + 1 < kLimbs) ? quo[li + 1] : 0u;
    return ((hi << 32) | lo) >> bi;
  };
  uint32_t mant = static_cast<uint32_t>(bits_at(shift) & 0xFFFFFFu);
  bool round_up;
  const bool odd = mant & 1u;
  if (shift == 0) {
    // The remainder alone decides: compare 2 * rem with count.
    const bool gt = (rem > count - rem);
    const bool eq = (rem == count - rem);
    round_up = gt || (eq && odd);
  } else {
    const int gpos = shift - 1;
    const bool guard = (quo[gpos >> 5] >> (gpos & 31)) & 1u;
    bool sticky = rem != 0;
    // bits strictly below gpos: whole limbs below, then a partial limb
    for (int i = 0; i < (gpos >> 5) && !sticky; ++i) sticky = quo[i] != 0u;
    if (!sticky && (gpos & 31)) sticky = (quo[gpos >> 5] & ((1u << (gpos & 31)) - 1u)) != 0u;
    round_up = guard && (sticky || odd);
  }
  int sh = shift;
  mant += round_up ? 1u : 0u;
  if (mant == (1u << 24)) { mant = 1u << 23; sh += 1; }
  uint32_t bits;
  if (mant >= (1u << 23)) bits = (static_cast<uint32_t>(sh + 1) << 23) | (mant - (1u << 23));
  else bits = mant;  // subnormal (only reachable with sh == 0)
  return __uint_as_float(bits);
}

// Each lane owns 8 elements of one block per iteration (32 bytes of fp32 or
// 16 bytes of bf16); eight lanes share a block.
template <typename T> struct QuantVec;
template <> struct QuantVec<float> { static constexpr int kVec = 8; };
template <> struct QuantVec<__nv_bfloat16> { static constexpr int kVec = 8; };

// ---------------------------------------------------------------------------
// Nearest-level decision by bucket lookup.  A normalised value v in [-1, 1]
// is bucketed by its sign, its exponent clamped below at 2^-6 and the top 3
// bits of its significand (112 buckets).  Every bucket contains at most one
// decision threshold, so code(v) = base[b] + (v > thr[b]) with thr[b] = +inf
// when the bucket holds none.  Values below 2^-5 in magnitude are all code 7
// (the smallest threshold magnitude is 0.0398), which is why the clamp at
// 2^-6 is exact.  The table is rebuilt from the threshold constants by every
// CTA (one entry per thread).
// ---------------------------------------------------------------------------
constexpr int kBuckets = 112;
constexpr uint32_t kBucketKeyMin = 121u << 3;   // exponent 121 (2^-6), 3 significand bits

struct BucketEntry { float thr; uint32_t base; };

__device__ __forceinline__ void build_bucket_entry(int idx, BucketEntry *tab) {
  const int neg = idx >= 56;
  const int key = idx % 56;
  const int e = 121 + (key >> 3), m3 = key & 7;
  // |v| range of the bucket: [L, H) = [(8 + m3), (9 + m3)) * 2^(e - 130)
  const float L = ldexpf(static_cast<float>(8 + m3), e - 130);
  const float H = ldexpf(static_cast<float>(9 + m3), e - 130);
  uint32_t base = 0;
  float thr = __int_as_float(0x7f800000);  // +inf: no threshold inside
  if (!neg) {       // v in [L, H): count thresholds below L, pick the one in [L, H)
    for (int i = 0; i < 15; ++i) {
      const float t = c_nf4_thresholds[i];
      if (t < L) ++base;
      else if (t < H) thr = t;
    }
  } else {          // v in (-H, -L]: count thresholds <= -H, pick the one in (-H, -L]
    for (int i = 0; i < 15; ++i) {
      const float t = c_nf4_thresholds[i];
      if (t <= -H) ++base;
      else if (t <= -L) thr = t;
    }
  }
  tab[idx].thr = thr;
  tab[idx].base = base;
}

// `tab` is the lane's column of the per-lane replicated table: entry b of
// lane l sits at tab[b * 32 + l], so the 32 lanes of a warp never conflict on
// a bank whatever buckets they hit.  The key comes from max(|v|, 2^-6) (every
// value below 2^-5 in magnitude has code 7, so the clamp is exact; a NaN maps
// to the smallest bucket), the sign picks the half of the table, and the
// decision v > thr is read off the sign of the fp32 difference thr - v (which
// is +0 only for v = thr and negative exactly when v > thr), so that most of
// the work runs on the multiply-add pipe rather than the integer/logic one.
__device__ __forceinline__ uint32_t bucket_code(float v, const BucketEntry *tab) {
  const float qc = fmaxf(fabsf(v), 0x1.0p-6f);
  const uint32_t key = (__float_as_uint(qc) >> 20) - kBucketKeyMin;  // 0 .. 48 for |v| <= 1
  const uint32_t half = (__float_as_uint(v) >> 31) * 56u;
  const BucketEntry en = tab[(key + half) * 32u];
  const float d = en.thr - v;
  return en.base + (__float_as_uint(d) >> 31);
}

// IEEE-correct x / m for |x| <= m with m in [2^-125, 2^125], from the
// correctly rounded reciprocal rcp = RN(1/m): q0 = RN(x * rcp) is within one
// ulp of x/m, the residual x - q0 * m is exact under one fused multiply-add,
// and q0 + residual * rcp rounded once is RN(x/m) (Markstein's correction
// theorem, P. Markstein, IBM J. Res. Dev. 34(1), 1990).  Two quotients at a
// time with the packed fp32x2 operations of sm_100+.  Checked bit-exact
// against the oracle's IEEE division on near-threshold inputs.
__device__ __forceinline__ void div_pair_by_scale(float &x0, float &x1, unsigned long long m2,
                                                  unsigned long long rcp2, unsigned long long nm2) {
  unsigned long long x, q, res;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q) : "l"(x), "l"(rcp2));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(res) : "l"(q), "l"(nm2), "l"(x));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(res), "l"(rcp2), "l"(q));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x0), "=f"(x1) : "l"(q));
  (void)m2;
}

// Quantises the 8 elements a lane holds of a 64-block that 8 consecutive
// lanes own together (every lane of the warp must call it): m = the block
// absmax (max |x| over the 64 elements, same on the 8 lanes), and the 8
// nearest-level codes of fp32(x / m), packed element 0 in the low nibble.
__device__ __forceinline__ uint32_t nf4_quant_lane8(float (&v)[8], const BucketEntry *tab, float &m_out) {
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (m >= 0x1.0p-125f && m <= 0x1.0p+125f) {
    const float rcp = __frcp_rn(m);
    unsigned long long rcp2, nm2;
    asm("mov.b64 %0, {%1, %1};" : "=l"(rcp2) : "f"(rcp));
    asm("mov.b64 %0, {%1, %1};" : "=l"(nm2) : "f"(-m));
#pragma unroll
    for (int i = 0; i < 8; i += 2) div_pair_by_scale(v[i], v[i + 1], 0ull, rcp2, nm2);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = (m > 0.f) ? __fdiv_rn(v[i], m) : 0.f;
  }
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // packed += code << 4 i, as a multiply-add
    const uint32_t c = bucket_code(v[i], tab);
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(packed) : "r"(c), "r"(1u << (4 * i)), "r"(packed));
  }
  m_out = m;
  return packed;
}

// The bucket table, per-lane replicated in shared memory (s_one: kBuckets
// entries of scratch, s_tab: kBuckets * 32); every thread of the CTA calls it.
__device__ __forceinline__ void build_bucket_tables(BucketEntry *s_one, BucketEntry *s_tab) {
  if (threadIdx.x < kBuckets) build_bucket_entry(threadIdx.x, s_one);
  __syncthreads();
  for (int i = threadIdx.x; i < kBuckets * 32; i += blockDim.x) s_tab[i] = s_one[i >> 5];
  __syncthreads();
}

// End of a quantising kernel with double quantisation (every thread of the
// CTA calls it): the CTA's exponent bins go to the global bins; the last CTA
// of the whole grid (1-D or not) to finish forms the exact mean of all nblk
// block constants, stores it and returns the ticket and the bins to zero
// (both are zero on entry: they live in a zero area).
__device__ __forceinline__ void quant_mean_epilogue(unsigned long long *s_bins, unsigned long long *bins,
                                                    unsigned int *ticket, int64_t nblk, float *absmax_mean) {
  __shared__ bool s_last;
  __syncthreads();
  for (int i = threadIdx.x; i < kNumBins; i += blockDim.x)
    if (s_bins[i]) atomicAdd(&bins[i], s_bins[i]);
  __threadfence();
  __syncthreads();
  const unsigned int nctas = gridDim.x * gridDim.y * gridDim.z;  // every CTA of the grid, whatever its shape
  if (threadIdx.x == 0) s_last = (atomicAdd(ticket, 1u) == nctas - 1u);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x < 32) {
    const float mu = exact_mean_from_bins(bins, static_cast<uint64_t>(nblk));
    if (threadIdx.x == 0) {
      *absmax_mean = mu;
      *ticket = 0u;
    }
  }
  __syncthreads();  // the bins are read; return them to zero for the next call
  for (int i = threadIdx.x; i < kNumBins; i += blockDim.x) bins[i] = 0ull;
}

// Quantiser main loop.  Each warp streams its own ring of kQuantRing stages
// of 1 KiB of input (32 bytes per lane) with 16-byte cp.async, so that about
// 128 KiB of loads are in flight per SM (two CTAs of 16 warps); a lane waits
// only for its own copies, and a __syncwarp hands the stage to the lanes that
// read it.  A stage holds 8 blocks of bf16 input (every lane quantises two
// blocks with 7 other lanes, one 8-element part of each) or 4 blocks of fp32
// input (one block per lane).  Inside a stage, the 16-byte unit u is stored
// at unit u ^ ((u >> 3) & 1), which keeps both the cp.async writes and the
// fp32 layout's 32-byte reads free of bank conflicts.  The last CTA to finish
// derives the double-quantisation mean from the exact exponent-binned sum and
// resets the ticket counter.
constexpr int kQuantWarps = kQuantThreads / 32;
constexpr int kQuantRing = 5;
constexpr int kQuantStage = 1024;
constexpr int kQuantSmem = kQuantWarps * kQuantRing * kQuantStage;  // dynamic shared memory per CTA

__device__ __forceinline__ uint32_t quant_unit(uint32_t u) { return (u ^ ((u >> 3) & 1u)) * 16u; }

__device__ __forceinline__ void quant_cp16(uint32_t dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kQuantThreads, 2)
nf4_quant_kernel(const T *__restrict__ x, int64_t nfull, int64_t nblk, uint8_t *__restrict__ codes,
                 float *__restrict__ absmax, unsigned long long *__restrict__ bins,
                 unsigned int *__restrict__ ticket, float *__restrict__ absmax_mean) {
  constexpr bool kF32 = sizeof(T) == 4;
  constexpr int kBps = kQuantStage / (64 * static_cast<int>(sizeof(T)));  // blocks per stage: 8 or 4
  extern __shared__ __align__(16) uint8_t q_ring[];
  __shared__ unsigned long long s_bins[kNumBins];
  __shared__ BucketEntry s_one[kBuckets];
  __shared__ BucketEntry s_tab[kBuckets * 32];
  for (int i = threadIdx.x; i < kNumBins; i += blockDim.x) s_bins[i] = 0ull;
  build_bucket_tables(s_one, s_tab);
  const int lane = threadIdx.x & 31;
  const BucketEntry *my_tab = s_tab + lane;
  const int li = lane & 7;
  const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(q_ring)) +
                        static_cast<uint32_t>((threadIdx.x >> 5) * (kQuantRing * kQuantStage));
  const int64_t nst = (nfull + kBps - 1) / kBps;  // stages of the whole input
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kQuantWarps + (threadIdx.x >> 5);
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kQuantWarps;
  const char *xb = reinterpret_cast<const char *>(x);
  BinFold fold_st = {0ull, -1};
  const bool fold = nblk <= (int64_t(1) << 31);

  // Issues this lane's two 16-byte copies of stage s into ring slot `slot`
  // (units c * 32 + lane; a unit past the last full block reads nothing and
  // is zero-filled) and closes the copy group, which is empty past the end.
  auto issue = [&](int64_t s, int slot) {
    if (s < nst) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint32_t u = static_cast<uint32_t>(c * 32 + lane);
        const int64_t blk = s * kBps + (u * 16u) / (64u * sizeof(T));
        const bool ok = blk < nfull;
        quant_cp16(ring + slot * kQuantStage + quant_unit(u), ok ? xb + s * kQuantStage + u * 16u : xb,
                   ok ? 16u : 0u);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

#pragma unroll
  for (int j = 0; j < kQuantRing - 1; ++j) issue(gw + j * nw, j);
  int slot = 0;
  for (int64_t s = gw; s < nst; s += nw) {
    issue(s + (kQuantRing - 1) * nw, slot == 0 ? kQuantRing - 1 : slot - 1);
    asm volatile("cp.async.wait_group %0;" ::"n"(kQuantRing - 1) : "memory");
    __syncwarp();
    const uint32_t base = ring + slot * kQuantStage;
    if constexpr (kF32) {
      // Lane l: block l / 8 of the stage, elements 8 (l % 8) .. + 7 (units 2l, 2l + 1).
      uint4 a, b;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w) : "r"(base + quant_unit(2u * lane)));
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w) : "r"(base + quant_unit(2u * lane + 1u)));
      __syncwarp();  // the slot may be refilled once every lane holds its part
      float v[8] = {__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z), __uint_as_float(a.w),
                    __uint_as_float(b.x), __uint_as_float(b.y), __uint_as_float(b.z), __uint_as_float(b.w)};
      float m;
      const uint32_t packed = nf4_quant_lane8(v, my_tab, m);
      const int64_t blk = s * kBps + (lane >> 3);
      if (blk < nfull) {
        reinterpret_cast<uint32_t *>(codes + blk * 32)[li] = packed;
        if (li == 0) {
          absmax[blk] = m;
          if (bins) bin_fold(fold_st, s_bins, m, fold);
        }
      }
    } else {
      // Lane l: blocks l / 8 and 4 + l / 8 of the stage, elements 8 (l % 8) .. + 7 of each.
      uint4 w[2];
#pragma unroll
      for (int c = 0; c < 2; ++c)
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[c].x), "=r"(w[c].y), "=r"(w[c].z), "=r"(w[c].w)
                     : "r"(base + quant_unit(static_cast<uint32_t>(c * 32 + lane))));
      __syncwarp();
      float v0[8], v1[8];
      const uint32_t a[4] = {w[0].x, w[0].y, w[0].z, w[0].w};
      const uint32_t b[4] = {w[1].x, w[1].y, w[1].z, w[1].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v0[2 * i] = __uint_as_float(a[i] << 16);
        v0[2 * i + 1] = __uint_as_float(a[i] & 0xFFFF0000u);
        v1[2 * i] = __uint_as_float(b[i] << 16);
        v1[2 * i + 1] = __uint_as_float(b[i] & 0xFFFF0000u);
      }
      float m0, m1;
      const uint32_t p0 = nf4_quant_lane8(v0, my_tab, m0);
      const uint32_t p1 = nf4_quant_lane8(v1, my_tab, m1);
      const int64_t blk0 = s * kBps + (lane >> 3), blk1 = blk0 + 4;
      if (blk0 < nfull) {
        reinterpret_cast<uint32_t *>(codes + blk0 * 32)[li] = p0;
        if (li == 0) {
          absmax[blk0] = m0;
          if (bins) bin_fold(fold_st, s_bins, m0, fold);
        }
      }
      if (blk1 < nfull) {
        reinterpret_cast<uint32_t *>(codes + blk1 * 32)[li] = p1;
        if (li == 0) {
          absmax[blk1] = m1;
          if (bins) bin_fold(fold_st, s_bins, m1, fold);
        }
      }
    }
    slot = (slot + 1 == kQuantRing) ? 0 : slot + 1;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (!bins) return;
  bin_flush(fold_st, s_bins);
  quant_mean_epilogue(s_bins, bins, ticket, nblk, absmax_mean);
}

// The final partial block: one warp, scalar loads.
template <typename T>
__global__ void nf4_quant_tail_kernel(const T *__restrict__ x, int64_t n, int64_t blk,
                                      uint8_t *__restrict__ codes, float *__restrict__ absmax,
                                      unsigned long long *__restrict__ bins) {
  const int lane = threadIdx.x;
  const int64_t base = blk * 64;
  const int cnt = static_cast<int>(n - base);  // 1..63
  float v0 = 0.f, v1 = 0.f;
  const int e0 = 2 * lane, e1 = 2 * lane + 1;
  if (e0 < cnt) v0 = static_cast<float>(x[base + e0]);
  if (e1 < cnt) v1 = static_cast<float>(x[base + e1]);
  float m = fmaxf(fabsf(v0), fabsf(v1));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  const uint32_t c0 = nf4_code_of(m > 0.f ? __fdiv_rn(v0, m) : 0.f);
  const uint32_t c1 = nf4_code_of(m > 0.f ? __fdiv_rn(v1, m) : 0.f);
  if (e0 < cnt) codes[blk * 32 + lane] = static_cast<uint8_t>(c0 | ((e1 < cnt) ? (c1 << 4) : 0u));
  if (lane == 0) {
    absmax[blk] = m;
    if (bins) {
      const uint32_t b = __float_as_uint(m);
      const uint32_t e = (b >> 23) & 0xFFu;
      const uint32_t sig = (b & 0x7FFFFFu) | (e ? 0x800000u : 0u);
      if (sig) atomicAdd(&bins[e ? e : 1u], static_cast<unsigned long long>(sig));
    }
  }
}

constexpr int kDqWarps = 8;

// One warp per group of 256 constants; the mean was stored by the last CTA
// of nf4_quant_kernel.
__global__ void __launch_bounds__(kDqWarps * 32)
nf4_dq_kernel(const float *__restrict__ absmax, int64_t nblk, const float *__restrict__ absmax_mean,
              int8_t *__restrict__ absmax_q, float *__restrict__ absmax_scale) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the constants and the mean come from the quantiser
  const float mu = __ldcg(absmax_mean);
  const int64_t ngrp = qn_ceil_div(nblk, 256);
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * kDqWarps + warp; g < ngrp;
       g += static_cast<int64_t>(gridDim.x) * kDqWarps) {
    const int64_t base = g * 256 + lane * 8;
    float c[8];
    float S = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t j = base + i;
      c[i] = (j < nblk) ? __fsub_rn(__ldcg(absmax + j), mu) : 0.f;
      S = fmaxf(S, fabsf(c[i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) S = fmaxf(S, __shfl_xor_sync(0xffffffffu, S, off));
    const float sigma = __fdiv_rn(S, 127.f);
    if (lane == 0) absmax_scale[g] = sigma;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t j = base + i;
      if (j < nblk) {
        int q = 0;
        if (sigma > 0.f) {
          q = __float2int_rn(__fdiv_rn(c[i], sigma));
          q = q > 127 ? 127 : (q < -127 ? -127 : q);
        }
        absmax_q[j] = static_cast<int8_t>(q);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Dequantisation: a lane decodes 4-byte words of codes (8 elements each).  A
// warp-iteration covers 128 consecutive words (1024 elements): lane l takes
// words l, l + 32, l + 64 and l + 96, so that every load of codes (128 bytes
// per warp) and every store of results (512 bytes of bf16, or two stores of
// 512 bytes of fp32, per warp) is contiguous.  The four code words and their
// block constants are loaded before any is decoded.
// ---------------------------------------------------------------------------
constexpr int kDeqThreads = 256;
constexpr int kDeqWords = 4;  // words per lane per warp-iteration

template <bool kBf16Out>
__global__ void __launch_bounds__(kDeqThreads)
nf4_dequant_kernel(QnNF4View q, int64_t n, void *__restrict__ out) {
  __shared__ float s_lut[16];
  if (threadIdx.x < 16) s_lut[threadIdx.x] = c_nf4_levels[threadIdx.x];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t nword = n / 8;
  const int64_t ntile = qn_ceil_div(nword, 32 * kDeqWords);
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const uint32_t *__restrict__ cw = reinterpret_cast<const uint32_t *>(q.codes);
  const float mu = q.dq ? __ldg(q.absmax_mean) : 0.f;
  for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < ntile; t += nw) {
    const int64_t w0 = t * (32 * kDeqWords) + lane;
    uint32_t w[kDeqWords];
    float m[kDeqWords];
#pragma unroll
    for (int i = 0; i < kDeqWords; ++i) {
      const int64_t wi = w0 + 32 * i;
      w[i] = (wi < nword) ? __ldcs(cw + wi) : 0u;
    }
#pragma unroll
    for (int i = 0; i < kDeqWords; ++i) {
      const int64_t wi = w0 + 32 * i;
      const int64_t j = ((wi < nword) ? wi : 0) >> 3;  // block of the word
      m[i] = q.dq ? dq_absmax(q.absmax_q[j], q.absmax_scale[j >> 8], mu) : q.absmax[j];
    }
#pragma unroll
    for (int i = 0; i < kDeqWords; ++i) {
      const int64_t wi = w0 + 32 * i;
      if (wi >= nword) break;
      if constexpr (kBf16Out) {
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o[e] = pack_bf16x2(__fmul_rn(s_lut[(w[i] >> (8 * e)) & 15u], m[i]),
                             __fmul_rn(s_lut[(w[i] >> (8 * e + 4)) & 15u], m[i]));
        __stcs(reinterpret_cast<uint4 *>(out) + wi, make_uint4(o[0], o[1], o[2], o[3]));
      } else {
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = __fmul_rn(s_lut[(w[i] >> (4 * e)) & 15u], m[i]);
        float4 *dst = reinterpret_cast<float4 *>(out) + 2 * wi;
        __stcs(dst, make_float4(f[0], f[1], f[2], f[3]));
        __stcs(dst + 1, make_float4(f[4], f[5], f[6], f[7]));
      }
    }
  }
  // Tail: elements [nword * 8, n), one thread each.
  const int64_t t0 = nword * 8;
  if (blockIdx.x == 0) {
    for (int64_t e = t0 + threadIdx.x; e < n; e += blockDim.x) {
      const uint32_t byte = q.codes[e >> 1];
      const uint32_t code = (e & 1) ? (byte >> 4) : (byte & 15u);
      const float wv = __fmul_rn(s_lut[code], block_scale(q, e >> 6));
      if constexpr (kBf16Out) static_cast<uint16_t *>(out)[e] = f32_to_bf16_bits(wv);
      else static_cast<float *>(out)[e] = wv;
    }
  }
}

}  // namespace qn
