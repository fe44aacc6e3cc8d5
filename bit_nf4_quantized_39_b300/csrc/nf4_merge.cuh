// nf4_merge.cuh -- merge / unmerge of a LoRA adapter into an NF4 weight:
//
//   Q_out = NF4( deq(Q) + sign * s * B A ),   sign = +1 (merge) or -1 (unmerge)
//
// ("PEFT quantization guide", merging adapters into quantised weights:
// dequantise the base weight, add the adapter weight, quantise again;
// unmerging subtracts it, so a merge/unmerge cycle does not give back the
// original codes.)  One pass: every element is dequantised, gets its adapter
// term and is requantised in registers, so the call reads the codes, the
// constants and the adapter once and writes the new codes once.
//
// Arithmetic (identical, operation for operation, to the oracle's reading):
// (B A)[i, j] = sum over q ascending of B[i, q] A[q, j] in fp32 -- A and B
// are bf16, so every product is exact and a fused multiply-add rounds only
// the sum; t = fp32(s * (B A)); x = fp32(deq + t) or fp32(deq - t); then the
// NF4 quantiser of nf4_codec.cuh (block absmax, IEEE division, nearest
// level, exact DQ mean).
//
// CTA tile 64 rows x 256 columns, 256 threads: warp w owns rows 8w .. 8w+7,
// lane l owns columns 8l .. 8l+7 of each (eight lanes per 64-block, the
// quantiser's layout); ranks are staged 32 at a time in shared memory (A as
// fp32, B rows as fp32).  In-place use (Q_out == Q) is safe: each thread
// reads its codes and constants before it writes them, and the DQ mean is
// replaced only after every CTA has finished.
#pragma once

#include "nf4_codec.cuh"

namespace qn {

constexpr int kMgThreads = 256;
constexpr int kMgRows = 64;
constexpr int kMgCols = 256;
constexpr int kMgRChunk = 32;
constexpr size_t kMgSmemBytes = static_cast<size_t>(kMgRChunk) * kMgCols * 4 +     // A chunk
                                static_cast<size_t>(kMgRows) * (kMgRChunk + 1) * 4 +  // B chunk
                                kNumBins * 8 + static_cast<size_t>(kBuckets) * 8 * 33;  // bins, tables

__global__ void __launch_bounds__(kMgThreads)
nf4_merge_kernel(QnNF4View qin, const uint16_t *__restrict__ A, const uint16_t *__restrict__ B, int r, float s,
                 int sign, uint8_t *codes_out, float *absmax_out, unsigned long long *bins, unsigned int *ticket,
                 float *absmax_mean_out) {
  extern __shared__ __align__(16) unsigned char mg_smem[];
  float *sA = reinterpret_cast<float *>(mg_smem);                     // [kMgRChunk][kMgCols]
  float *sB = sA + kMgRChunk * kMgCols;                               // [kMgRows][kMgRChunk + 1]
  unsigned long long *s_bins = reinterpret_cast<unsigned long long *>(sB + kMgRows * (kMgRChunk + 1));
  BucketEntry *s_one = reinterpret_cast<BucketEntry *>(s_bins + kNumBins);
  BucketEntry *s_tab = s_one + kBuckets;
  __shared__ float s_lv[16];  // the levels, indexed per lane (a constant-bank read would serialise)
  for (int i = threadIdx.x; i < kNumBins; i += blockDim.x) s_bins[i] = 0ull;
  if (threadIdx.x < 16) s_lv[threadIdx.x] = c_nf4_levels[threadIdx.x];
  build_bucket_tables(s_one, s_tab);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const BucketEntry *my_tab = s_tab + lane;
  const int64_t d = qin.d, k = qin.k, nb = k >> 6;
  const int64_t row0 = static_cast<int64_t>(blockIdx.y) * kMgRows + warp * 8;
  const int64_t col = static_cast<int64_t>(blockIdx.x) * kMgCols + lane * 8;
  const bool col_ok = col < k;  // k is a multiple of 64: a block is valid or not as a whole
  BinFold fold_st = {0ull, -1};
  const bool fold = d * nb <= (int64_t(1) << 31);

  // The input codes and block constants of this thread's 8 rows x 8 columns.
  uint32_t win[8];
  float min_[8];
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    const int64_t row = row0 + rr;
    win[rr] = 0x77777777u;
    min_[rr] = 0.f;
    if (row < d && col_ok) {
      const int64_t e = row * k + col;
      win[rr] = *reinterpret_cast<const uint32_t *>(qin.codes + (e >> 1));
      min_[rr] = block_scale(qin, e >> 6);
    }
  }

  float acc[8][8];
#pragma unroll
  for (int rr = 0; rr < 8; ++rr)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[rr][j] = 0.f;
  const int64_t cta_col0 = static_cast<int64_t>(blockIdx.x) * kMgCols;
  const int64_t cta_row0 = static_cast<int64_t>(blockIdx.y) * kMgRows;
  for (int q0 = 0; q0 < r; q0 += kMgRChunk) {
    const int qn_ = (r - q0 < kMgRChunk) ? r - q0 : kMgRChunk;
    // A[q0 .. q0 + qn_, cta_col0 .. + 256) as fp32: 8 bf16 (16 bytes) per load
    for (int i = tid; i < kMgRChunk * kMgCols / 8; i += kMgThreads) {
      const int q = i / (kMgCols / 8), c8 = (i % (kMgCols / 8)) * 8;
      const int64_t c = cta_col0 + c8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (q < qn_ && c < k) v = *reinterpret_cast<const uint4 *>(A + static_cast<int64_t>(q0 + q) * k + c);
      float *dst = sA + q * kMgCols + c8;
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        dst[2 * h] = __uint_as_float(w4[h] << 16);
        dst[2 * h + 1] = __uint_as_float(w4[h] & 0xFFFF0000u);
      }
    }
    // B[cta_row0 .. + 64, q0 .. q0 + qn_) as fp32
    for (int i = tid; i < kMgRows * kMgRChunk; i += kMgThreads) {
      const int rrow = i / kMgRChunk, q = i % kMgRChunk;
      const int64_t row = cta_row0 + rrow;
      sB[rrow * (kMgRChunk + 1) + q] =
          (q < qn_ && row < d) ? bf16_bits_to_f32(B[row * r + q0 + q]) : 0.f;
    }
    __syncthreads();
    for (int q = 0; q < qn_; ++q) {
      const float4 a0 = *reinterpret_cast<const float4 *>(sA + q * kMgCols + lane * 8);
      const float4 a1 = *reinterpret_cast<const float4 *>(sA + q * kMgCols + lane * 8 + 4);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const float b = sB[(warp * 8 + rr) * (kMgRChunk + 1) + q];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[rr][j] = fmaf(b, a[j], acc[rr][j]);  // b * a is exact: one rounding
      }
    }
    __syncthreads();
  }

  // Dequantise, add or subtract the adapter term, requantise.
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    const int64_t row = row0 + rr;
    const bool valid = row < d && col_ok;
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float base = __fmul_rn(s_lv[(win[rr] >> (4 * j)) & 15u], min_[rr]);
      const float t = __fmul_rn(s, acc[rr][j]);
      x[j] = (sign > 0) ? __fadd_rn(base, t) : __fsub_rn(base, t);
    }
    float m;
    const uint32_t packed = nf4_quant_lane8(x, my_tab, m);  // every lane takes part (shuffles)
    if (valid) {
      const int64_t e = row * k + col;
      *reinterpret_cast<uint32_t *>(codes_out + (e >> 1)) = packed;
      if ((lane & 7) == 0) {
        absmax_out[e >> 6] = m;
        if (bins) bin_fold(fold_st, s_bins, m, fold);
      }
    }
  }
  if (!bins) return;
  bin_flush(fold_st, s_bins);
  quant_mean_epilogue(s_bins, bins, ticket, d * nb, absmax_mean_out);
}

}  // namespace qn
