// qlora_simt.cuh -- CUDA-core kernels of the QLoRA layer:
//   * the LoRA projections u = s X A^T (forward) and v = s dY B (backward);
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
// K is split over gridDim.z CTAs of kchunk columns each (a multiple of 32);
// split z writes its partial sums to part + z * M * N, and
// lora_reduce_kernel adds the splits in order.
// ---------------------------------------------------------------------------
constexpr int kProjTM = 64, kProjTN = 32, kProjTK = 32;
constexpr int kProjMaxSplit = 16;

__global__ void __launch_bounds__(256)
lora_proj_kernel(const uint16_t *__restrict__ P, int64_t M, int64_t K,
                 const uint16_t *__restrict__ Qm, int64_t N, int64_t qs_n, int64_t qs_k,
                 float s, int64_t kchunk, float *__restrict__ part) {
  __shared__ float sP[kProjTK][kProjTM + 1];
  __shared__ float sQ[kProjTK][kProjTN + 1];
  const int tid = threadIdx.x;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kProjTM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kProjTN;
  const int64_t kb = static_cast<int64_t>(blockIdx.z) * kchunk;
  const int64_t ke = (kb + kchunk < K) ? kb + kchunk : K;
  const int tm = tid / 8;        // 0..31 -> rows tm and tm + 32
  const int tn = (tid % 8) * 4;  // 4 consecutive columns
  float acc[2][4] = {};
  for (int64_t k0 = kb; k0 < ke; k0 += kProjTK) {
    for (int i = tid; i < kProjTM * kProjTK; i += 256) {
      const int r = i / kProjTK, c = i % kProjTK;
      const int64_t gm = m0 + r, gk = k0 + c;
      sP[c][r] = (gm < M && gk < ke) ? bf16_bits_to_f32(P[gm * K + gk]) : 0.f;
    }
    for (int i = tid; i < kProjTN * kProjTK; i += 256) {
      const int r = i / kProjTK, c = i % kProjTK;
      const int64_t gn = n0 + r, gk = k0 + c;
      sQ[c][r] = (gn < N && gk < ke) ? bf16_bits_to_f32(Qm[gn * qs_n + gk * qs_k]) : 0.f;
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
  float *C = part + static_cast<int64_t>(blockIdx.z) * M * N;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t gm = m0 + tm + 32 * i, gn = n0 + tn + j;
      if (gm < M && gn < N) C[gm * N + gn] = s * acc[i][j];
    }
}

// C = sum over the S splits of part (in split order).  Writes the fp32 result
// to C32 (if not null) and, if C2 is not null, its bf16 hi/lo split
// C2[m, :] = [bf16(c) | bf16(c - bf16(c))], each half zero-padded to R columns.
__global__ void lora_reduce_kernel(const float *__restrict__ part, int S, int64_t M, int64_t N,
                                   float *__restrict__ C32, int R, uint16_t *__restrict__ C2) {
  const int64_t cols = C2 ? R : N;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= M * cols) return;
  const int64_t m = i / cols, j = i % cols;
  float v = 0.f;
  if (j < N)
    for (int z = 0; z < S; ++z) v += part[(static_cast<int64_t>(z) * M + m) * N + j];
  if (C32 && j < N) C32[m * N + j] = v;
  if (C2) {
    const uint16_t hi = f32_to_bf16_bits(v);
    C2[m * 2 * R + j] = hi;
    C2[m * 2 * R + R + j] = f32_to_bf16_bits(v - bf16_bits_to_f32(hi));
  }
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
