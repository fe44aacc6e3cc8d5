// loftq.cuh -- device kernels of the LoftQ initialisation.
//
// "LoftQ explainer" (mhpn.cn) §2.2: minimise ||W - (Q + Delta)||_F^2 over a
// quantised Q and a rank-r Delta; §2.3: alternate the Q-step Q = quantise(W -
// Delta) with the Delta-step Delta = best rank-r approximation of W - Q.
//
// The rank-r step is a randomised subspace iteration (Halko, Martinsson and
// Tropp, "Finding structure with randomness", SIAM Review 2011, Alg. 4.4):
// Y = R Omega, re-orthonormalised after every product (CholeskyQR2), then the
// small p x p eigenproblem of (Y^T R)(Y^T R)^T gives singular values and
// vectors.  Omega is Gaussian from Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC 2011) with Box-Muller.
#pragma once

#include "common.cuh"

namespace qn {

constexpr int kLqMaxP = 32;  // r + oversample

// ---------------------------------------------------------------- Philox4x32-10
struct U4 { uint32_t x, y, z, w; };

__device__ __forceinline__ U4 philox4x32_10(U4 ctr, uint32_t k0, uint32_t k1) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t hi0 = __umulhi(M0, ctr.x), lo0 = M0 * ctr.x;
    const uint32_t hi1 = __umulhi(M1, ctr.z), lo1 = M1 * ctr.z;
    ctr = U4{hi1 ^ ctr.y ^ k0, lo1, hi0 ^ ctr.w ^ k1, lo0};
    k0 += W0;
    k1 += W1;
  }
  return ctr;
}

// Omega (rows x P, row-major): element (j, c) ~ N(0, 1) for c < p, 0 otherwise.
// Gaussian pair i comes from the Philox block with counter (i, 0, 0, 0) and
// key = seed via Box-Muller; element number j * p + c takes half (j*p+c) % 2
// of pair (j*p+c) / 2, so the draw does not depend on the padding P.
__global__ void omega_kernel(float *__restrict__ out, int64_t rows, int p, int P, uint64_t seed) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= rows * P) return;
  const int64_t j = idx / P;
  const int c = static_cast<int>(idx % P);
  if (c >= p) { out[idx] = 0.f; return; }
  const int64_t e = j * p + c;
  const int64_t pair = e >> 1;
  const U4 r = philox4x32_10(U4{static_cast<uint32_t>(pair), static_cast<uint32_t>(pair >> 32), 0u, 0u},
                             static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  // Uniforms: u1 in (0, 1] (never 0), u2 in [0, 1).
  const float u1 = (static_cast<float>(r.x) + 1.0f) * 2.3283064e-10f;
  const float u2 = static_cast<float>(r.y) * 2.3283064e-10f;
  const float rad = sqrtf(-2.0f * logf(fminf(u1, 1.0f)));
  float sv, cv;
  sincospif(2.0f * u2, &sv, &cv);
  out[idx] = (e & 1) ? rad * sv : rad * cv;
}

// ----------------------------------------------------------- element-wise passes
// T = W - s * B A   (B: d x r fp32, A: r x k fp32), 4 columns per thread.
__global__ void __launch_bounds__(256)
lowrank_sub_kernel(const float *__restrict__ W, const float *__restrict__ B, const float *__restrict__ A,
                   int64_t d, int64_t k, int r, float s, float *__restrict__ T) {
  const int64_t n4 = d * k / 4;
  for (int64_t i4 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i4 < n4;
       i4 += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i4 * 4;
    const int64_t row = e / k, col = e % k;
    float4 w = __ldg(reinterpret_cast<const float4 *>(W) + i4);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int q = 0; q < r; ++q) {
      const float b = __ldg(B + row * r + q);
      const float4 a = __ldg(reinterpret_cast<const float4 *>(A + q * k + col));
      acc[0] = fmaf(b, a.x, acc[0]); acc[1] = fmaf(b, a.y, acc[1]);
      acc[2] = fmaf(b, a.z, acc[2]); acc[3] = fmaf(b, a.w, acc[3]);
    }
    w.x -= s * acc[0]; w.y -= s * acc[1]; w.z -= s * acc[2]; w.w -= s * acc[3];
    reinterpret_cast<float4 *>(T)[i4] = w;
  }
}

// R = W - deq(Q) in fp32 (the exact fp32 dequantised weight), 32 per thread.
__global__ void __launch_bounds__(256)
residual_kernel(QnNF4View q, const float *__restrict__ W, float *__restrict__ R, int64_t n) {
  __shared__ float s_lut[16];
  if (threadIdx.x < 16) s_lut[threadIdx.x] = c_nf4_levels[threadIdx.x];
  __syncthreads();
  const int64_t nchunk = n / 32;
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < nchunk;
       c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 w4 = __ldg(reinterpret_cast<const uint4 *>(q.codes) + c);
    const float m = block_scale(q, c >> 1);
    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
    const float4 *src = reinterpret_cast<const float4 *>(W + c * 32);
    float4 *dst = reinterpret_cast<float4 *>(R + c * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t nib = w[i / 2] >> (16 * (i & 1));
      float4 x = __ldg(src + i);
      x.x -= __fmul_rn(s_lut[nib & 15u], m);
      x.y -= __fmul_rn(s_lut[(nib >> 4) & 15u], m);
      x.z -= __fmul_rn(s_lut[(nib >> 8) & 15u], m);
      x.w -= __fmul_rn(s_lut[(nib >> 12) & 15u], m);
      dst[i] = x;
    }
  }
}

// ------------------------------------------------------------- skinny products
// Y[i, c] = sum_j R[i, j] Z[j, c]   (R: n_rows x n_cols, Z: n_cols x p).
// One warp per row; lanes stride the row; per-lane partial sums reduced by
// shuffles.  Z rows are read through the read-only cache.
template <int P>
__global__ void __launch_bounds__(256)
rz_kernel(const float *__restrict__ R, int64_t n_rows, int64_t n_cols,
          const float *__restrict__ Z, int p, float *__restrict__ Y) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 8 + warp; i < n_rows;
       i += static_cast<int64_t>(gridDim.x) * 8) {
    float acc[P];
#pragma unroll
    for (int c = 0; c < P; ++c) acc[c] = 0.f;
    const float *row = R + i * n_cols;
    for (int64_t j = lane; j < n_cols; j += 32) {
      const float rv = __ldcs(row + j);
      const float4 *zr = reinterpret_cast<const float4 *>(Z + j * P);
#pragma unroll
      for (int c4 = 0; c4 < P / 4; ++c4) {
        const float4 z = __ldg(zr + c4);
        acc[4 * c4] = fmaf(rv, z.x, acc[4 * c4]);
        acc[4 * c4 + 1] = fmaf(rv, z.y, acc[4 * c4 + 1]);
        acc[4 * c4 + 2] = fmaf(rv, z.z, acc[4 * c4 + 2]);
        acc[4 * c4 + 3] = fmaf(rv, z.w, acc[4 * c4 + 3]);
      }
    }
#pragma unroll
    for (int c = 0; c < P; ++c) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], off);
    }
    {
      float v = 0.f;
#pragma unroll
      for (int c = 0; c < P; ++c) if (c == lane) v = acc[c];
      if (lane < P) Y[i * P + lane] = (lane < p) ? v : 0.f;
    }
  }
}

// Zt[j, c] += sum_{i in slice} R[i, j] Y[i, c]  (Zt zeroed by the caller).
// Threads own columns j; the row slice is split across blockIdx.y.
template <int P>
__global__ void __launch_bounds__(128)
rty_kernel(const float *__restrict__ R, int64_t n_rows, int64_t n_cols,
           const float *__restrict__ Y, int64_t rows_per_slice, float *__restrict__ Zt) {
  __shared__ float sY[64][P];
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t i_begin = static_cast<int64_t>(blockIdx.y) * rows_per_slice;
  const int64_t i_end = (i_begin + rows_per_slice < n_rows) ? i_begin + rows_per_slice : n_rows;
  float acc[P];
#pragma unroll
  for (int c = 0; c < P; ++c) acc[c] = 0.f;
  for (int64_t i0 = i_begin; i0 < i_end; i0 += 64) {
    __syncthreads();
    for (int t = threadIdx.x; t < 64 * P; t += blockDim.x) {
      const int64_t ii = i0 + t / P;
      sY[t / P][t % P] = (ii < i_end) ? Y[ii * P + t % P] : 0.f;
    }
    __syncthreads();
    const int lim = static_cast<int>((i_end - i0) < 64 ? (i_end - i0) : 64);
    if (j < n_cols) {
      for (int ii = 0; ii < lim; ++ii) {
        const float rv = __ldcs(R + (i0 + ii) * n_cols + j);
#pragma unroll
        for (int c = 0; c < P; ++c) acc[c] = fmaf(rv, sY[ii][c], acc[c]);
      }
    }
  }
  if (j < n_cols) {
#pragma unroll
    for (int c = 0; c < P; ++c) atomicAdd(&Zt[j * P + c], acc[c]);
  }
}

// G[a, b] += sum_i Y[i, a] Y[i, b]   (fp64, G zeroed by the caller, p x p).
template <int P>
__global__ void __launch_bounds__(P * P)
gram_kernel(const float *__restrict__ Y, int64_t n, int64_t rows_per_block, double *__restrict__ G) {
  __shared__ float sY[32][P];
  const int a = threadIdx.x / P, b = threadIdx.x % P;
  const int64_t i_begin = static_cast<int64_t>(blockIdx.x) * rows_per_block;
  const int64_t i_end = (i_begin + rows_per_block < n) ? i_begin + rows_per_block : n;
  double acc = 0.0;
  for (int64_t i0 = i_begin; i0 < i_end; i0 += 32) {
    __syncthreads();
    for (int t = threadIdx.x; t < 32 * P; t += blockDim.x) {
      const int64_t ii = i0 + t / P;
      sY[t / P][t % P] = (ii < i_end) ? Y[ii * P + t % P] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int ii = 0; ii < 32; ++ii) acc += static_cast<double>(sY[ii][a]) * static_cast<double>(sY[ii][b]);
  }
  atomicAdd(&G[a * P + b], acc);
}

// One CTA of P threads: Cholesky G = L L^T of the leading p x p block of the
// Gram matrix (accumulated in fp64, factored in fp32) and Linv = L^{-1}
// (lower triangular, fp32 [P x P], zero outside the p x p block).  A pivot
// that is not positive (rank deficiency) is clamped to a tiny positive value.
template <int P>
__global__ void __launch_bounds__(P)
chol_inv_kernel(const double *__restrict__ G, int p, float *__restrict__ Linv) {
  __shared__ float L[P][P + 1];
  __shared__ float Li[P][P + 1];
  __shared__ float s_diag_floor;
  const int t = threadIdx.x;
  for (int j = 0; j < P; ++j) {
    L[t][j] = (t < p && j < p) ? static_cast<float>(G[t * P + j]) : 0.f;
    Li[t][j] = 0.f;
  }
  __syncthreads();
  if (t == 0) {
    float mx = 0.f;
    for (int i = 0; i < p; ++i) mx = fmaxf(mx, L[i][i]);
    s_diag_floor = fmaxf(mx, 1e-30f) * 1e-12f;
  }
  __syncthreads();
  // Right-looking Cholesky on the lower triangle held in L.
  for (int j = 0; j < p; ++j) {
    if (t == 0) L[j][j] = sqrtf(fmaxf(L[j][j], s_diag_floor));
    __syncthreads();
    const float inv = 1.0f / L[j][j];
    if (t > j && t < p) L[t][j] *= inv;
    __syncthreads();
    if (t > j && t < p) {
      const float ltj = L[t][j];
      for (int c = j + 1; c <= t; ++c) L[t][c] -= ltj * L[c][j];
    }
    __syncthreads();
  }
  // Column t of L^{-1} by forward substitution.
  if (t < p) {
    for (int i = t; i < p; ++i) {
      float acc = (i == t) ? 1.f : 0.f;
      for (int q = t; q < i; ++q) acc -= L[i][q] * Li[q][t];
      Li[i][t] = acc / L[i][i];
    }
  }
  __syncthreads();
  for (int j = 0; j < P; ++j) Linv[t * P + j] = Li[t][j];
}

// Y[i, :] <- Y[i, :] Linv^T   (in place).  One warp per row: lane c holds
// Y[i, c] and computes sum_b Y[i, b] Linv[c, b] with the row broadcast by
// shuffles (P == 32).
template <int P>
__global__ void __launch_bounds__(256)
apply_linv_kernel(float *__restrict__ Y, int64_t n, const float *__restrict__ Linv, int p) {
  static_assert(P == 32, "one lane per column");
  __shared__ float sL[P][P + 1];
  for (int t = threadIdx.x; t < P * P; t += blockDim.x) sL[t / P][t % P] = Linv[t];
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 8 + warp; i < n; i += static_cast<int64_t>(gridDim.x) * 8) {
    const float y = Y[i * P + lane];
    float acc = 0.f;
#pragma unroll
    for (int b = 0; b < P; ++b) acc = fmaf(__shfl_sync(0xffffffffu, y, b), sL[lane][b], acc);
    Y[i * P + lane] = (lane < p) ? acc : 0.f;
  }
}

// One CTA of P threads: cyclic Jacobi eigen-decomposition (fp32) of the
// symmetric leading p x p block of G (accumulated in fp64).  Outputs the
// eigenvalues sorted descending (lam[P], zero past p) and the matching
// eigenvectors as the columns of V (fp32 [P x P], V[row * P + col]).
template <int P>
__global__ void __launch_bounds__(P)
jacobi_eig_kernel(const double *__restrict__ G, int p, float *__restrict__ lam, float *__restrict__ V) {
  __shared__ float A[P][P + 1];
  __shared__ float E[P][P + 1];
  __shared__ float s_c, s_s;
  __shared__ int s_done;
  const int t = threadIdx.x;
  for (int j = 0; j < P; ++j) {
    A[t][j] = (t < p && j < p) ? static_cast<float>(G[t * P + j]) : 0.f;
    E[t][j] = (t == j) ? 1.f : 0.f;
  }
  __syncthreads();
  for (int sweep = 0; sweep < 20; ++sweep) {
    if (t == 0) {
      float off = 0.f, dg = 0.f;
      for (int i = 0; i < p; ++i) {
        dg += A[i][i] * A[i][i];
        for (int j = 0; j < p; ++j) if (i != j) off += A[i][j] * A[i][j];
      }
      s_done = (off <= 1e-13f * dg) ? 1 : 0;
    }
    __syncthreads();
    if (s_done) break;
    for (int i = 0; i < p - 1; ++i) {
      for (int j = i + 1; j < p; ++j) {
        if (t == 0) {
          const float aij = A[i][j];
          float c = 1.f, sn = 0.f;
          if (fabsf(aij) > 1e-30f * (fabsf(A[i][i]) + fabsf(A[j][j]))) {
            const float theta = (A[j][j] - A[i][i]) / (2.f * aij);
            const float tt = copysignf(1.f, theta) / (fabsf(theta) + sqrtf(theta * theta + 1.f));
            c = 1.f / sqrtf(tt * tt + 1.f);
            sn = tt * c;
          }
          s_c = c;
          s_s = sn;
        }
        __syncthreads();
        const float c = s_c, sn = s_s;
        if (sn != 0.f) {
          // A <- J^T A J and E <- E J for the rotation in the (i, j) plane.
          const float ati = A[t][i], atj = A[t][j];
          __syncthreads();
          A[t][i] = c * ati - sn * atj;
          A[t][j] = sn * ati + c * atj;
          __syncthreads();
          const float ait = A[i][t], ajt = A[j][t];
          __syncthreads();
          A[i][t] = c * ait - sn * ajt;
          A[j][t] = sn * ait + c * ajt;
          const float eti = E[t][i], etj = E[t][j];
          E[t][i] = c * eti - sn * etj;
          E[t][j] = sn * eti + c * etj;
        }
        __syncthreads();
      }
    }
  }
  __syncthreads();
  if (t == 0) {
    int order[P];
    for (int i = 0; i < P; ++i) order[i] = i;
    for (int i = 0; i < p; ++i) {
      int best = i;
      for (int j = i + 1; j < p; ++j) if (A[order[j]][order[j]] > A[order[best]][order[best]]) best = j;
      const int tmp = order[i]; order[i] = order[best]; order[best] = tmp;
    }
    for (int i = 0; i < P; ++i) lam[i] = (i < p) ? A[order[i]][order[i]] : 0.f;
    for (int row = 0; row < P; ++row)
      for (int col = 0; col < P; ++col) V[row * P + col] = (col < p) ? E[row][order[col]] : 0.f;
  }
}

// out[i, q] = sum_b in[i, b] * V[b, q] * scale[q]  for q < r;  in: n x P fp32.
// transpose_out: write out[q * n + i] (r x n) instead of out[i * r + q].
template <int P>
__global__ void __launch_bounds__(256)
project_kernel(const float *__restrict__ in, int64_t n, const float *__restrict__ V,
               const float *__restrict__ lam, int r, float s, int for_A,
               float *__restrict__ out, int transpose_out) {
  __shared__ float sC[P][P];
  // for_A == 0 (B):  coefficient V[b, q] * sqrt(sigma_q) / sqrt(s)
  // for_A == 1 (A):  coefficient V[b, q] / (sqrt(sigma_q) * sqrt(s)),
  // sigma_q = sqrt(lam_q) (lam are eigenvalues of the Gram matrix).
  for (int t = threadIdx.x; t < P * P; t += blockDim.x) {
    const int b = t / P, q = t % P;
    float cval = 0.f;
    if (q < r) {
      const float sigma = sqrtf(fmaxf(lam[q], 0.f));
      const float rs = sqrtf(sigma);
      float sc;
      if (for_A) sc = (rs > 0.f) ? 1.f / (rs * sqrtf(s)) : 0.f;
      else sc = rs / sqrtf(s);
      cval = V[b * P + q] * sc;
    }
    sC[b][q] = cval;
  }
  __syncthreads();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float x[P];
#pragma unroll
    for (int b = 0; b < P; ++b) x[b] = in[i * P + b];
    for (int q = 0; q < r; ++q) {
      float acc = 0.f;
#pragma unroll
      for (int b = 0; b < P; ++b) acc = fmaf(x[b], sC[b][q], acc);
      if (transpose_out) out[static_cast<int64_t>(q) * n + i] = acc;
      else out[i * r + q] = acc;
    }
  }
}

// partial[block] = sum over its elements of (R - s * B A)^2 in fp64.
__global__ void __launch_bounds__(256)
resid_norm_kernel(const float *__restrict__ R, const float *__restrict__ B, const float *__restrict__ A,
                  int64_t d, int64_t k, int r, float s, double *__restrict__ partial) {
  __shared__ double red[256];
  double acc = 0.0;
  const int64_t n = d * k;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = e / k, col = e % k;
    float lr = 0.f;
    for (int q = 0; q < r; ++q) lr = fmaf(__ldg(B + row * r + q), __ldg(A + q * k + col), lr);
    const double diff = static_cast<double>(R[e]) - static_cast<double>(s) * static_cast<double>(lr);
    acc += diff * diff;
  }
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) partial[blockIdx.x] = red[0];
}

__global__ void sum_partials_kernel(const double *__restrict__ partial, int count, double *__restrict__ out) {
  __shared__ double red[256];
  double acc = 0.0;
  for (int i = threadIdx.x; i < count; i += blockDim.x) acc += partial[i];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *out = red[0];
}

}  // namespace qn
