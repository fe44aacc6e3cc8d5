// qlora_simt.cuh -- CUDA-core kernels of the QLoRA layer:
//   * the LoRA projections u = s X A^T (forward) and v = s dY B (backward);
//   * the small-M fused forward (decode): split-K over the 4-bit weight,
//     decoded in registers, bound by the bytes of the packed weight;
//   * a tiled fused GEMM used for shapes the tensor-core kernel does not take.
//
// Layer ("PEFT course notes" §2.2, h = Wx + BAx with W in R^{d x k},
// B in R^{d x r}, A in R^{r x k}; scale s = alpha / r):
//   Y  = X deq(Q)^T + s (X A^T) B^T
//   dX = dY deq(Q)  + s (dY B) A
#pragma once

#include "common.cuh"

namespace qn {

// ---------------------------------------------------------------------------
// Skinny projection  C[m, n] = s * sum_kk P[m, kk] * Qop(n, kk)   (fp32 out)
// with Qop(n, kk) = Qm[n * qs_n + kk * qs_k].  P is bf16 [M x K] row-major.
// 64 x 32 output tile, K chunks of 32, 256 threads, 8 outputs per thread.
// ---------------------------------------------------------------------------
constexpr int kProjTM = 64, kProjTN = 32, kProjTK = 32;

__global__ void __launch_bounds__(256)
lora_proj_kernel(const uint16_t *__restrict__ P, int64_t M, int64_t K,
                 const uint16_t *__restrict__ Qm, int64_t N, int64_t qs_n, int64_t qs_k,
                 float s, float *__restrict__ C) {
  __shared__ float sP[kProjTK][kProjTM + 1];
  __shared__ float sQ[kProjTK][kProjTN + 1];
  const int tid = threadIdx.x;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kProjTM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kProjTN;
  const int tm = tid / 8;        // 0..31 -> rows tm and tm + 32
  const int tn = (tid % 8) * 4;  // 4 consecutive columns
  float acc[2][4] = {};
  for (int64_t k0 = 0; k0 < K; k0 += kProjTK) {
    for (int i = tid; i < kProjTM * kProjTK; i += 256) {
      const int r = i / kProjTK, c = i % kProjTK;
      const int64_t gm = m0 + r, gk = k0 + c;
      sP[c][r] = (gm < M && gk < K) ? bf16_bits_to_f32(P[gm * K + gk]) : 0.f;
    }
    for (int i = tid; i < kProjTN * kProjTK; i += 256) {
      const int r = i / kProjTK, c = i % kProjTK;
      const int64_t gn = n0 + r, gk = k0 + c;
      sQ[c][r] = (gn < N && gk < K) ? bf16_bits_to_f32(Qm[gn * qs_n + gk * qs_k]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kProjTK; ++kk) {
      const float a0 = sP[kk][tm], a1 = sP[kk][tm + 32];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float b = sQ[kk][tn + j];
        acc[0][j] = fmaf(a0, b, acc[0][j]);
        acc[1][j] = fmaf(a1, b, acc[1][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t gm = m0 + tm + 32 * i, gn = n0 + tn + j;
      if (gm < M && gn < N) C[gm * N + gn] = s * acc[i][j];
    }
}

// ---------------------------------------------------------------------------
// Small-M fused forward (M <= kGemvMaxM).  Grid: (row groups, k splits).
// One warp owns one weight row per iteration; each lane streams 16-byte code
// chunks (32 elements, half a 64-block), decodes through a shared LUT and
// accumulates sum_e c[code_e] x[t, e] per token, scaled once per chunk by the
// block constant.  Partial sums of the k splits go to `part` (fp32
// [splits x M x d]); the last split to finish a row group reduces them in
// order, adds the adapter term u B^T and writes bf16 Y.  Counters live in the
// workspace and are returned to zero by the reducing CTA.
// ---------------------------------------------------------------------------
constexpr int kGemvMaxM = 16;
constexpr int kGemvWarps = 8;           // rows per CTA
constexpr int kGemvThreads = kGemvWarps * 32;

template <int MT>
__global__ void __launch_bounds__(kGemvThreads)
qlora_fwd_gemv_kernel(QnNF4View q, const uint16_t *__restrict__ X, int M,
                      const float *__restrict__ u, const uint16_t *__restrict__ Bm, int r,
                      uint16_t *__restrict__ Y, float *__restrict__ part,
                      unsigned int *__restrict__ counters, int splits, int64_t chunks_per_split) {
  __shared__ float s_lut[16];
  __shared__ bool s_last;
  if (threadIdx.x < 16) s_lut[threadIdx.x] = c_nf4_levels[threadIdx.x];
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t d = q.d, k = q.k;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kGemvWarps + warp;
  const int split = blockIdx.y;
  const int64_t nchunk_row = k / 32;  // 16-byte chunks per row
  const int64_t c_begin = split * chunks_per_split;
  const int64_t c_end = (c_begin + chunks_per_split < nchunk_row) ? c_begin + chunks_per_split : nchunk_row;

  float acc[MT];
#pragma unroll
  for (int t = 0; t < MT; ++t) acc[t] = 0.f;
  if (row < d) {
    const uint4 *wrow = reinterpret_cast<const uint4 *>(q.codes + row * (k / 2));
    for (int64_t c = c_begin + lane; c < c_end; c += 32) {
      const uint4 w4 = __ldcs(wrow + c);
      const float m = block_scale(q, row * (k / 64) + (c >> 1));
      const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
      float dec[32];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) dec[8 * i + j] = s_lut[(w[i] >> (4 * j)) & 15u];
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        if (t < M) {
          const uint4 *xp = reinterpret_cast<const uint4 *>(X + t * k + c * 32);
          float sum = 0.f;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 xv = __ldg(xp + v);
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              sum = fmaf(dec[8 * v + 2 * h], __uint_as_float(xw[h] << 16), sum);
              sum = fmaf(dec[8 * v + 2 * h + 1], __uint_as_float(xw[h] & 0xFFFF0000u), sum);
            }
          }
          acc[t] = fmaf(sum, m, acc[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < MT; ++t) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
  }
  if (splits == 1) {
    if (row < d && lane < M) {
      float y = 0.f;
#pragma unroll
      for (int t = 0; t < MT; ++t) if (t == lane) y = acc[t];
      for (int j = 0; j < r; ++j) y = fmaf(u[lane * r + j], bf16_bits_to_f32(Bm[row * r + j]), y);
      Y[lane * d + row] = f32_to_bf16_bits(y);
    }
    return;
  }
  // Split-K: publish partials, the last CTA of this row group reduces.
  if (row < d && lane < M) {
    float y = 0.f;
#pragma unroll
    for (int t = 0; t < MT; ++t) if (t == lane) y = acc[t];
    part[(static_cast<int64_t>(split) * M + lane) * d + row] = y;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int prev = atomicAdd(&counters[blockIdx.x], 1u);
    s_last = (prev == static_cast<unsigned int>(splits - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (row < d && lane < M) {
    float y = 0.f;
    for (int sp = 0; sp < splits; ++sp) y += __ldcg(&part[(static_cast<int64_t>(sp) * M + lane) * d + row]);
    for (int j = 0; j < r; ++j) y = fmaf(u[lane * r + j], bf16_bits_to_f32(Bm[row * r + j]), y);
    Y[lane * d + row] = f32_to_bf16_bits(y);
  }
  if (threadIdx.x == 0) counters[blockIdx.x] = 0u;
}

// ---------------------------------------------------------------------------
// Tiled fused GEMM on CUDA cores (any M; fallback path).
//   kTrans == false (forward):  C[m, c] = sum_j P[m, j] W'[c, j] + sum_q L[m, q] Bm[c, q]
//   kTrans == true  (backward): C[m, c] = sum_i P[m, i] W'[i, c] + sum_q L[m, q] Am[q, c]
// P is bf16 [M x K]; W' is decoded on the fly; L is fp32 [M x r] (already
// scaled by s); the adapter factor is bf16.  64 x 64 tile, K chunks of 16.
// ---------------------------------------------------------------------------
constexpr int kTileM = 64, kTileN = 64, kTileK = 16;

template <bool kTrans>
__global__ void __launch_bounds__(256)
qlora_gemm_simt_kernel(QnNF4View q, const uint16_t *__restrict__ P, int64_t M,
                       const float *__restrict__ L, const uint16_t *__restrict__ F, int r,
                       uint16_t *__restrict__ C) {
  __shared__ float sA[kTileK][kTileM + 4];
  __shared__ float sB[kTileK][kTileN + 4];
  __shared__ float s_lut[16];
  if (threadIdx.x < 16) s_lut[threadIdx.x] = c_nf4_levels[threadIdx.x];
  const int64_t d = q.d, kdim = q.k;
  const int64_t K = kTrans ? d : kdim;      // reduction length
  const int64_t N = kTrans ? kdim : d;      // output columns
  const int tid = threadIdx.x;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kTileM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kTileN;
  const int ty = tid / 16, tx = tid % 16;   // 4 x 4 outputs per thread
  float acc[4][4] = {};
  __syncthreads();
  for (int64_t k0 = 0; k0 < K; k0 += kTileK) {
    for (int i = tid; i < kTileM * kTileK; i += 256) {
      const int rr = i / kTileK, cc = i % kTileK;
      const int64_t gm = m0 + rr, gk = k0 + cc;
      sA[cc][rr] = (gm < M && gk < K) ? bf16_bits_to_f32(P[gm * K + gk]) : 0.f;
    }
    for (int i = tid; i < kTileN * kTileK; i += 256) {
      int rr, cc;
      if (kTrans) { cc = i / kTileN; rr = i % kTileN; }   // coalesce along columns
      else { rr = i / kTileK; cc = i % kTileK; }
      const int64_t gn = n0 + rr, gk = k0 + cc;
      float wv = 0.f;
      if (gn < N && gk < K) {
        const int64_t wi = kTrans ? gk : gn;    // weight row
        const int64_t wj = kTrans ? gn : gk;    // weight column
        const int64_t e = wi * kdim + wj;
        const uint32_t byte = q.codes[e >> 1];
        const uint32_t code = (e & 1) ? (byte >> 4) : (byte & 15u);
        wv = bf16_bits_to_f32(f32_to_bf16_bits(__fmul_rn(s_lut[code], block_scale(q, e >> 6))));
      }
      sB[cc][rr] = wv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kTileK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = sA[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = sB[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t gn = n0 + tx * 4 + j;
      if (gn >= N) continue;
      float y = acc[i][j];
      for (int qq = 0; qq < r; ++qq) {
        const float f = kTrans ? bf16_bits_to_f32(F[qq * N + gn]) : bf16_bits_to_f32(F[gn * r + qq]);
        y = fmaf(L[gm * r + qq], f, y);
      }
      C[gm * N + gn] = f32_to_bf16_bits(y);
    }
  }
}

}  // namespace qn
