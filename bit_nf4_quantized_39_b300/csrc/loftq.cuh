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

constexpr int kLqMaxP = 96;  // largest r + oversample (panels of 32, 64 or 96 columns)

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

// R = W - deq(Q) in fp32 (the exact fp32 dequantised weight).  A lane takes
// 4-byte words of codes (8 elements), a warp 32 consecutive words per step,
// so code loads and the 32-byte W reads and R writes of a lane are
// contiguous across the warp.  n % 8 == 0.
__global__ void __launch_bounds__(256)
residual_kernel(QnNF4View q, const float *__restrict__ W, float *__restrict__ R, int64_t n) {
  __shared__ float s_lut[16];
  if (threadIdx.x < 16) s_lut[threadIdx.x] = c_nf4_levels[threadIdx.x];
  __syncthreads();
  const int64_t nword = n / 8;
  const uint32_t *__restrict__ cw = reinterpret_cast<const uint32_t *>(q.codes);
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; w < nword;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t c = __ldg(cw + w);
    const float m = block_scale(q, w >> 3);
    const float4 *src = reinterpret_cast<const float4 *>(W) + 2 * w;
    float4 x0 = __ldcs(src), x1 = __ldcs(src + 1);
    x0.x -= __fmul_rn(s_lut[c & 15u], m);
    x0.y -= __fmul_rn(s_lut[(c >> 4) & 15u], m);
    x0.z -= __fmul_rn(s_lut[(c >> 8) & 15u], m);
    x0.w -= __fmul_rn(s_lut[(c >> 12) & 15u], m);
    x1.x -= __fmul_rn(s_lut[(c >> 16) & 15u], m);
    x1.y -= __fmul_rn(s_lut[(c >> 20) & 15u], m);
    x1.z -= __fmul_rn(s_lut[(c >> 24) & 15u], m);
    x1.w -= __fmul_rn(s_lut[c >> 28], m);
    float4 *dst = reinterpret_cast<float4 *>(R) + 2 * w;
    dst[0] = x0;
    dst[1] = x1;
  }
}

// ------------------------------------------------------------- skinny products
// The rank-r step works on panels of P columns (P = 32, 64 or 96, the padded
// r + oversample; columns past p are kept zero).  Both products read R once;
// K is split over gridDim.y so that enough CTAs stream it, each split's
// partial panel goes to `part`, and lq_split_reduce_kernel adds the splits
// in order (no atomics: the result does not depend on the launch).  Tiles
// are double-buffered through shared memory with cp.async.

constexpr int kLqTile = 32;  // rows of the output panel per CTA, and the K chunk

// part[split][i][c] = sum over the split's j of R[i, j] Z[j, c]  (R: n_rows x n_cols, Z: n_cols x P).
// Thread (row tid / 8, panel columns (tid % 8) P/8 ..).  n_cols % 32 == 0.
template <int P>
__global__ void __launch_bounds__(256)
lq_rz_kernel(const float *__restrict__ R, int64_t n_rows, int64_t n_cols, const float *__restrict__ Z,
             int64_t cols_per_split, float *__restrict__ part) {
  constexpr int CW = P / 8;
  __shared__ __align__(16) float sR[2][kLqTile][kLqTile + 4];
  __shared__ __align__(16) float sZ[2][kLqTile][P];
  const int tid = threadIdx.x, tr = tid / 8, tc = tid % 8;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kLqTile;
  const int64_t jb = static_cast<int64_t>(blockIdx.y) * cols_per_split;
  int64_t je = jb + cols_per_split;
  if (je > n_cols) je = n_cols;
  auto stage = [&](int b, int64_t j0) {
    for (int t = tid; t < kLqTile * kLqTile / 4; t += 256) {  // R tile: 32 rows x 32 columns
      const int rr = t / (kLqTile / 4), c4 = (t % (kLqTile / 4)) * 4;
      const int64_t i = i0 + rr;
      if (i < n_rows) cp_async16(smem_u32(&sR[b][rr][c4]), R + i * n_cols + j0 + c4);
      else *reinterpret_cast<float4 *>(&sR[b][rr][c4]) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int t = tid; t < kLqTile * P / 4; t += 256) {  // Z tile: 32 rows x P
      const int rr = t / (P / 4), c4 = (t % (P / 4)) * 4;
      cp_async16(smem_u32(&sZ[b][rr][c4]), Z + (j0 + rr) * P + c4);
    }
    cp_async_commit();
  };
  float acc[CW];
#pragma unroll
  for (int c = 0; c < CW; ++c) acc[c] = 0.f;
  const int nch = static_cast<int>((je - jb) / kLqTile);
  if (nch > 0) stage(0, jb);
  for (int ch = 0; ch < nch; ++ch) {
    const int b = ch & 1;
    if (ch + 1 < nch) {
      stage(b ^ 1, jb + static_cast<int64_t>(ch + 1) * kLqTile);
      cp_async_wait_group<1>();
    } else {
      cp_async_wait_group<0>();
    }
    __syncthreads();
#pragma unroll 8
    for (int jj = 0; jj < kLqTile; ++jj) {
      const float rv = sR[b][tr][jj];
#pragma unroll
      for (int c = 0; c < CW; ++c) acc[c] = fmaf(rv, sZ[b][jj][tc * CW + c], acc[c]);
    }
    __syncthreads();
  }
  const int64_t i = i0 + tr;
  if (i < n_rows) {
    float *dst = part + (static_cast<int64_t>(blockIdx.y) * n_rows + i) * P + tc * CW;
#pragma unroll
    for (int c = 0; c < CW; ++c) dst[c] = acc[c];
  }
}

// part[split][j][c] = sum over the split's i of R[i, j] Y[i, c]  (R: n_rows x n_cols, Y: n_rows x P).
// Thread (column tid / 8, panel columns (tid % 8) P/8 ..).  n_cols % 32 == 0.
template <int P>
__global__ void __launch_bounds__(256)
lq_rty_kernel(const float *__restrict__ R, int64_t n_rows, int64_t n_cols, const float *__restrict__ Y,
              int64_t rows_per_split, float *__restrict__ part) {
  constexpr int CW = P / 8;
  __shared__ __align__(16) float sR[2][kLqTile][kLqTile + 4];
  __shared__ __align__(16) float sY[2][kLqTile][P];
  const int tid = threadIdx.x, tj = tid / 8, tc = tid % 8;
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kLqTile;
  const int64_t ib = static_cast<int64_t>(blockIdx.y) * rows_per_split;
  int64_t ie = ib + rows_per_split;
  if (ie > n_rows) ie = n_rows;
  auto stage = [&](int b, int64_t i0) {
    for (int t = tid; t < kLqTile * kLqTile / 4; t += 256) {  // R tile: 32 rows x 32 columns
      const int rr = t / (kLqTile / 4), c4 = (t % (kLqTile / 4)) * 4;
      const int64_t i = i0 + rr;
      if (i < ie) cp_async16(smem_u32(&sR[b][rr][c4]), R + i * n_cols + j0 + c4);
      else *reinterpret_cast<float4 *>(&sR[b][rr][c4]) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int t = tid; t < kLqTile * P / 4; t += 256) {  // Y tile: 32 rows x P
      const int rr = t / (P / 4), c4 = (t % (P / 4)) * 4;
      const int64_t i = i0 + rr;
      if (i < ie) cp_async16(smem_u32(&sY[b][rr][c4]), Y + i * P + c4);
      else *reinterpret_cast<float4 *>(&sY[b][rr][c4]) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    cp_async_commit();
  };
  float acc[CW];
#pragma unroll
  for (int c = 0; c < CW; ++c) acc[c] = 0.f;
  const int nch = static_cast<int>((ie - ib + kLqTile - 1) / kLqTile);
  if (nch > 0) stage(0, ib);
  for (int ch = 0; ch < nch; ++ch) {
    const int b = ch & 1;
    if (ch + 1 < nch) {
      stage(b ^ 1, ib + static_cast<int64_t>(ch + 1) * kLqTile);
      cp_async_wait_group<1>();
    } else {
      cp_async_wait_group<0>();
    }
    __syncthreads();
#pragma unroll 8
    for (int ii = 0; ii < kLqTile; ++ii) {
      const float rv = sR[b][ii][tj];
#pragma unroll
      for (int c = 0; c < CW; ++c) acc[c] = fmaf(rv, sY[b][ii][tc * CW + c], acc[c]);
    }
    __syncthreads();
  }
  const int64_t j = j0 + tj;
  if (j < n_cols) {
    float *dst = part + (static_cast<int64_t>(blockIdx.y) * n_cols + j) * P + tc * CW;
#pragma unroll
    for (int c = 0; c < CW; ++c) dst[c] = acc[c];
  }
}

// Register-tiled products for 32-column panels (the common r + oversample
// <= 32).  A thread accumulates a 4 x 4 block of the output from 16-byte
// shared-memory reads (8 multiply-adds per read); tiles arrive through a
// kLqPipe-deep cp.async ring (one CTA barrier per 32-deep K step).  K is
// split over gridDim.y as in lq_rz_kernel / lq_rty_kernel.
constexpr int kLqPipe = 3;
constexpr int kLqBig = 128;  // output rows per CTA
constexpr int kLqRzStage = (kLqBig * (kLqTile + 4) + kLqTile * 32) * 4;   // R tile [128][36] + Z tile [32][32]
constexpr int kLqRtyStage = (kLqTile * (kLqBig + 4) + kLqTile * 32) * 4;  // R tile [32][132] + Y tile [32][32]

__device__ __forceinline__ void lq_cp16(uint32_t dst, const void *src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(ok ? 16u : 0u) : "memory");
}

// part[split][i][c] = sum over the split's j of R[i, j] Z[j, c]; thread
// (rows 4 (tid / 8) .., columns 4 (tid % 8) ..) of a 128-row tile.
__global__ void __launch_bounds__(256)
lq_rz32_kernel(const float *__restrict__ R, int64_t n_rows, int64_t n_cols, const float *__restrict__ Z,
               int64_t cols_per_split, float *__restrict__ part) {
  extern __shared__ __align__(16) float lq_pipe_smem[];
  const int tid = threadIdx.x, rg = tid >> 3, cg = tid & 7;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kLqBig;
  const int64_t jb = static_cast<int64_t>(blockIdx.y) * cols_per_split;
  const int64_t je = (jb + cols_per_split < n_cols) ? jb + cols_per_split : n_cols;
  const int nch = static_cast<int>((je - jb) / kLqTile);
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(lq_pipe_smem));
  auto load = [&](int slot, int64_t j0) {
    const uint32_t sr = sbase + slot * kLqRzStage, sz = sr + kLqBig * (kLqTile + 4) * 4;
#pragma unroll
    for (int u = 0; u < 4; ++u) {  // R: 128 rows x 8 chunks
      const int ch = tid + 256 * u, rr = ch >> 3, c4 = (ch & 7) * 4;
      const int64_t i = i0 + rr;
      lq_cp16(sr + (rr * (kLqTile + 4) + c4) * 4, (i < n_rows) ? R + i * n_cols + j0 + c4 : R, i < n_rows);
    }
    {  // Z: 32 rows x 8 chunks
      const int rr = tid >> 3, c4 = (tid & 7) * 4;
      lq_cp16(sz + (rr * 32 + c4) * 4, Z + (j0 + rr) * 32 + c4, true);
    }
  };
  float acc[4][4] = {};
#pragma unroll
  for (int st = 0; st < kLqPipe - 1; ++st) {
    if (st < nch) load(st, jb + static_cast<int64_t>(st) * kLqTile);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int ch = 0; ch < nch; ++ch) {
    asm volatile("cp.async.wait_group %0;" ::"n"(kLqPipe - 2) : "memory");
    __syncthreads();
    const int nx = ch + kLqPipe - 1;
    if (nx < nch) load(nx % kLqPipe, jb + static_cast<int64_t>(nx) * kLqTile);
    asm volatile("cp.async.commit_group;" ::: "memory");
    const float *sR = lq_pipe_smem + (ch % kLqPipe) * (kLqRzStage / 4);
    const float *sZ = sR + kLqBig * (kLqTile + 4);
#pragma unroll
    for (int kq = 0; kq < kLqTile / 4; ++kq) {
      float4 rv[4], zv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) rv[a] = *reinterpret_cast<const float4 *>(sR + (4 * rg + a) * (kLqTile + 4) + 4 * kq);
#pragma unroll
      for (int q = 0; q < 4; ++q) zv[q] = *reinterpret_cast<const float4 *>(sZ + (4 * kq + q) * 32 + 4 * cg);
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float r4[4] = {rv[a].x, rv[a].y, rv[a].z, rv[a].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[a][0] = fmaf(r4[q], zv[q].x, acc[a][0]);
          acc[a][1] = fmaf(r4[q], zv[q].y, acc[a][1]);
          acc[a][2] = fmaf(r4[q], zv[q].z, acc[a][2]);
          acc[a][3] = fmaf(r4[q], zv[q].w, acc[a][3]);
        }
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int64_t i = i0 + 4 * rg + a;
    if (i < n_rows)
      *reinterpret_cast<float4 *>(part + (static_cast<int64_t>(blockIdx.y) * n_rows + i) * 32 + 4 * cg) =
          make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
  }
}

// part[split][j][c] = sum over the split's i of R[i, j] Y[i, c]; thread
// (columns 4 (tid / 8) .. of a 128-column tile, panel columns 4 (tid % 8) ..).
__global__ void __launch_bounds__(256)
lq_rty32_kernel(const float *__restrict__ R, int64_t n_rows, int64_t n_cols, const float *__restrict__ Y,
                int64_t rows_per_split, float *__restrict__ part) {
  extern __shared__ __align__(16) float lq_pipe_smem[];
  const int tid = threadIdx.x, jg = tid >> 3, cg = tid & 7;
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kLqBig;
  const int64_t ib = static_cast<int64_t>(blockIdx.y) * rows_per_split;
  const int64_t ie = (ib + rows_per_split < n_rows) ? ib + rows_per_split : n_rows;
  const int nch = static_cast<int>((ie - ib + kLqTile - 1) / kLqTile);
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(lq_pipe_smem));
  auto load = [&](int slot, int64_t ia) {
    const uint32_t sr = sbase + slot * kLqRtyStage, sy = sr + kLqTile * (kLqBig + 4) * 4;
#pragma unroll
    for (int u = 0; u < 4; ++u) {  // R: 32 rows x 32 chunks
      const int ch = tid + 256 * u, rr = ch >> 5, c4 = (ch & 31) * 4;
      const int64_t i = ia + rr, j = j0 + c4;
      const bool ok = i < ie && j < n_cols;
      lq_cp16(sr + (rr * (kLqBig + 4) + c4) * 4, ok ? R + i * n_cols + j : R, ok);
    }
    {  // Y: 32 rows x 8 chunks
      const int rr = tid >> 3, c4 = (tid & 7) * 4;
      const int64_t i = ia + rr;
      lq_cp16(sy + (rr * 32 + c4) * 4, (i < ie) ? Y + i * 32 + c4 : Y, i < ie);
    }
  };
  float acc[4][4] = {};
#pragma unroll
  for (int st = 0; st < kLqPipe - 1; ++st) {
    if (st < nch) load(st, ib + static_cast<int64_t>(st) * kLqTile);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int ch = 0; ch < nch; ++ch) {
    asm volatile("cp.async.wait_group %0;" ::"n"(kLqPipe - 2) : "memory");
    __syncthreads();
    const int nx = ch + kLqPipe - 1;
    if (nx < nch) load(nx % kLqPipe, ib + static_cast<int64_t>(nx) * kLqTile);
    asm volatile("cp.async.commit_group;" ::: "memory");
    const float *sR = lq_pipe_smem + (ch % kLqPipe) * (kLqRtyStage / 4);
    const float *sY = sR + kLqTile * (kLqBig + 4);
#pragma unroll 8
    for (int ii = 0; ii < kLqTile; ++ii) {
      const float4 rv = *reinterpret_cast<const float4 *>(sR + ii * (kLqBig + 4) + 4 * jg);
      const float4 yv = *reinterpret_cast<const float4 *>(sY + ii * 32 + 4 * cg);
      const float r4[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        acc[a][0] = fmaf(r4[a], yv.x, acc[a][0]);
        acc[a][1] = fmaf(r4[a], yv.y, acc[a][1]);
        acc[a][2] = fmaf(r4[a], yv.z, acc[a][2]);
        acc[a][3] = fmaf(r4[a], yv.w, acc[a][3]);
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int64_t j = j0 + 4 * jg + a;
    if (j < n_cols)
      *reinterpret_cast<float4 *>(part + (static_cast<int64_t>(blockIdx.y) * n_cols + j) * 32 + 4 * cg) =
          make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
  }
}

// out[e] = sum over the S splits, in order, of part[split][e]   (e < n).
__global__ void lq_split_reduce_kernel(const float *__restrict__ part, int S, int64_t n, float *__restrict__ out) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= n) return;
  float v = 0.f;
  for (int z = 0; z < S; ++z) v += part[static_cast<int64_t>(z) * n + e];
  out[e] = v;
}

// Gram matrix G = Y^T Y (P x P) of a panel Y (n x P): kLqGramRows rows per
// CTA summed in fp32 into part[block][P][P], then lq_gram_reduce_kernel adds
// the blocks in order in fp64.  Thread (a-tile, b-tile) holds an
// (P/16) x (P/16) tile of the P x P result.
constexpr int kLqGramRows = 32;

template <int P>
__global__ void __launch_bounds__(256)
lq_gram_part_kernel(const float *__restrict__ Y, int64_t n, float *__restrict__ part) {
  constexpr int TW = P / 16;
  __shared__ __align__(16) float sY[32][P];
  const int tid = threadIdx.x, ta = tid / 16, tb = tid % 16;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kLqGramRows;
  float acc[TW][TW];
#pragma unroll
  for (int a = 0; a < TW; ++a)
#pragma unroll
    for (int b = 0; b < TW; ++b) acc[a][b] = 0.f;
  for (int64_t i0 = r0; i0 < r0 + kLqGramRows && i0 < n; i0 += 32) {
    for (int t = tid; t < 32 * P; t += 256) {
      const int rr = t / P, cc = t % P;
      const int64_t i = i0 + rr;
      sY[rr][cc] = (i < n && i < r0 + kLqGramRows) ? Y[i * P + cc] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int ii = 0; ii < 32; ++ii) {
      float ya[TW], yb[TW];
#pragma unroll
      for (int a = 0; a < TW; ++a) ya[a] = sY[ii][ta * TW + a];
#pragma unroll
      for (int b = 0; b < TW; ++b) yb[b] = sY[ii][tb * TW + b];
#pragma unroll
      for (int a = 0; a < TW; ++a)
#pragma unroll
        for (int b = 0; b < TW; ++b) acc[a][b] = fmaf(ya[a], yb[b], acc[a][b]);
    }
    __syncthreads();
  }
  float *pp = part + static_cast<int64_t>(blockIdx.x) * P * P;
#pragma unroll
  for (int a = 0; a < TW; ++a)
#pragma unroll
    for (int b = 0; b < TW; ++b) pp[(ta * TW + a) * P + tb * TW + b] = acc[a][b];
}

// G[e] = sum over the blocks of part[block][e] in fp64: one warp per entry
// (lane-strided partial sums, then a fixed shuffle tree).
template <int P>
__global__ void lq_gram_reduce_kernel(const float *__restrict__ part, int nblocks, double *__restrict__ G) {
  const int e = static_cast<int>((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (e >= P * P) return;  // uniform over the warp
  double v = 0.0;
  for (int b = lane; b < nblocks; b += 32) v += static_cast<double>(part[static_cast<int64_t>(b) * P * P + e]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) G[e] = v;
}

// One CTA of 256 threads: Cholesky G = L L^T of the leading p x p block (G
// accumulated in fp64, factored in fp32).  L (lower triangular, fp32 [P x P])
// is the identity outside the p x p block.  A pivot that is not positive
// (rank deficiency) is clamped to a tiny positive value.
template <int P>
__global__ void __launch_bounds__(256)
lq_chol_kernel(const double *__restrict__ G, int p, float *__restrict__ Lout) {
  __shared__ float Mx[P][P + 1];
  __shared__ float s_floor;
  const int tid = threadIdx.x;
  for (int t = tid; t < P * P; t += 256) {
    const int i = t / P, j = t % P;
    Mx[i][j] = (i < p && j < p) ? static_cast<float>(G[i * P + j]) : 0.f;
  }
  __syncthreads();
  if (tid < 32) {
    float mx = 0.f;
    for (int i = tid; i < p; i += 32) mx = fmaxf(mx, Mx[i][i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (tid == 0) s_floor = fmaxf(mx, 1e-30f) * 1e-12f;
  }
  __syncthreads();
  for (int j = 0; j < p; ++j) {
    if (tid == 0) Mx[j][j] = sqrtf(fmaxf(Mx[j][j], s_floor));
    __syncthreads();
    const float inv = 1.0f / Mx[j][j];
    for (int i = j + 1 + tid; i < p; i += 256) Mx[i][j] *= inv;
    __syncthreads();
    // trailing update of the lower triangle: M[i][c] -= L[i][j] L[c][j], j < c <= i < p
    const int m = p - j - 1;
    for (int t = tid; t < m * m; t += 256) {
      const int i = j + 1 + t / m, c = j + 1 + t % m;
      if (c <= i) Mx[i][c] -= Mx[i][j] * Mx[c][j];
    }
    __syncthreads();
  }
  for (int e = tid; e < P * P; e += 256) {
    const int i = e / P, c = e % P;
    Lout[e] = (i < p && c < p) ? ((c <= i) ? Mx[i][c] : 0.f) : ((i == c) ? 1.f : 0.f);
  }
}

// Y[i, :] <- Y[i, :] L^{-T} in place (the Q factor of CholeskyQR): each row
// solves L q = y by forward substitution, one thread per row; columns past
// p come out zero.
template <int P>
__global__ void __launch_bounds__(128)
lq_trsm_rows_kernel(float *__restrict__ Y, int64_t n, const float *__restrict__ L, int p) {
  __shared__ float sL[P][P + 1];
  for (int t = threadIdx.x; t < P * P; t += blockDim.x) sL[t / P][t % P] = L[t];
  __syncthreads();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float y[P];
#pragma unroll
  for (int c = 0; c < P; c += 4) {
    const float4 v = *reinterpret_cast<const float4 *>(Y + i * P + c);
    y[c] = v.x; y[c + 1] = v.y; y[c + 2] = v.z; y[c + 3] = v.w;
  }
#pragma unroll
  for (int c = 0; c < P; ++c) {
    float acc = y[c];
#pragma unroll
    for (int b = 0; b < c; ++b) acc = fmaf(-sL[c][b], y[b], acc);
    y[c] = (c < p) ? acc / sL[c][c] : 0.f;
  }
#pragma unroll
  for (int c = 0; c < P; c += 4)
    *reinterpret_cast<float4 *>(Y + i * P + c) = make_float4(y[c], y[c + 1], y[c + 2], y[c + 3]);
}

// ---------------------------------------------------------------------------
// CholeskyQR2 of a 32-column panel in one launch (Fukaya, Nakatsukasa,
// Yanagisawa, Yamamoto, "CholeskyQR2: a simple and communication-avoiding
// algorithm for computing a tall-skinny QR factorization", ScalA 2014): two
// rounds of  G = Y^T Y,  G = L L^T,  Y <- Y L^{-T}.  Every CTA is resident
// at once (cooperative launch) and owns a contiguous range of rows.  With
// S > 0 the panel is first formed as the sum, in split order, of the S
// split-K partials of the product that made it (part[z][n][32], the sums
// lq_split_reduce_kernel forms) and written to Y.  A round:
//   1. each CTA sums y y^T over its rows (fp32 within 32-row chunks, fp64
//      across chunks) into its fp64 partial;
//   2. grid barrier; the P*P entries of G are split over the grid's warps,
//      each summing the CTAs' partials in a fixed order (fp64);
//   3. grid barrier; every CTA factors G itself (one warp, lane i holding row
//      i of the matrix in registers, fp32: pivots clamped to a floor of
//      1e-12 times the largest diagonal entry, as lq_chol_kernel, but with
//      the hardware reciprocal square root) and solves its rows against L
//      by forward substitution (multiplying by the reciprocal pivots).
// Grid barriers are counters in the zero area with bounded waits: a wait
// that expires records QN_DEV_TIMEOUT and the kernel carries on (the panel is
// then wrong and the host reports the status).  The last CTA to leave resets
// both counters.
// ---------------------------------------------------------------------------
constexpr unsigned kLqSpinLimit = 1u << 20;  // polls, 64 ns apart

__device__ __forceinline__ void lq_grid_barrier(unsigned int *cnt, unsigned int target) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(cnt, 1u);
    unsigned int v = 0, spins = 0;
    for (;;) {
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
      if (v >= target) break;
      if (++spins > kLqSpinLimit) {
        qn_flag_timeout();
        break;
      }
      __nanosleep(64);
    }
  }
  __syncthreads();
}

// Step K of the one-warp Cholesky of a 32 x 32 matrix, lane i holding row i
// in a[] (compile-time indices only): pivot from lane K (hardware reciprocal
// square root), column K scaled below it, the scaled column published in
// shared memory (col, 16-byte aligned) and read back four entries at a time
// for the trailing update.  Updates of entries right of a lane's diagonal are
// harmless (never read) and are not masked; rows past p stay identity rows.
template <int K>
__device__ __forceinline__ void lq_chol_warp_step(float (&a)[32], int lane, int p, float floor_v, float *col) {
  if constexpr (K < 32) {
    const float dk = __shfl_sync(0xffffffffu, a[K], K);
    const float x = fmaxf(dk, floor_v);
    const float rs = rsqrtf(x);  // hardware reciprocal square root
    if (lane == K) a[K] = (K < p) ? x * rs : 1.f;
    if (lane > K && lane < p) a[K] *= rs;
    const float lik = a[K];
    col[lane] = lik;
    __syncwarp();
#pragma unroll
    for (int g = (K + 1) / 4; g < 8; ++g) {
      const float4 v = reinterpret_cast<const float4 *>(col)[g];
      const float cv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (4 * g + e > K) a[4 * g + e] = fmaf(-lik, cv[e], a[4 * g + e]);
    }
    __syncwarp();
    lq_chol_warp_step<K + 1>(a, lane, p, floor_v, col);
  }
}

__global__ void __launch_bounds__(256, 1)
lq_cholqr2_p32_kernel(const float *__restrict__ part, int S, float *__restrict__ Y, int64_t n, int p,
                      double *__restrict__ gpart, double *__restrict__ G, unsigned int *__restrict__ bar) {
  constexpr int P = 32;
  __shared__ __align__(16) float sY[32][P];
  __shared__ float sL[P][P + 1];
  __shared__ float sRinv[P];
  __shared__ __align__(16) float sCol[P];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ta = tid / 16, tb = tid % 16;  // 2 x 2 tile of G: rows 2 ta.., columns 2 tb..
  const unsigned int nct = gridDim.x;
  const int64_t rpc = (n + nct - 1) / nct;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * rpc;
  const int64_t r1 = (r0 + rpc < n) ? r0 + rpc : n;
  unsigned int nbar = 0;

  for (int round = 0; round < 2; ++round) {
    // 1. partial Gram matrix of this CTA's rows
    double acc[2][2] = {{0.0, 0.0}, {0.0, 0.0}};
    for (int64_t i0 = r0; i0 < r1; i0 += 32) {
      for (int t = tid; t < 32 * P / 4; t += 256) {
        const int rr = t / (P / 4), c4 = (t % (P / 4)) * 4;
        const int64_t i = i0 + rr;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < r1) {
          if (round == 0 && S > 0) {  // the panel is the sum of the S partials, in split order
            const float *src = part + i * P + c4;
            v = __ldcg(reinterpret_cast<const float4 *>(src));
            for (int z = 1; z < S; ++z) {
              const float4 w = __ldcg(reinterpret_cast<const float4 *>(src + static_cast<int64_t>(z) * n * P));
              v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
            }
            __stcg(reinterpret_cast<float4 *>(Y + i * P + c4), v);
          } else {
            v = __ldcg(reinterpret_cast<const float4 *>(Y + i * P + c4));
          }
        }
        *reinterpret_cast<float4 *>(&sY[rr][c4]) = v;
      }
      __syncthreads();
      float f[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll 8
      for (int ii = 0; ii < 32; ++ii) {
        const float ya0 = sY[ii][2 * ta], ya1 = sY[ii][2 * ta + 1];
        const float yb0 = sY[ii][2 * tb], yb1 = sY[ii][2 * tb + 1];
        f[0][0] = fmaf(ya0, yb0, f[0][0]);
        f[0][1] = fmaf(ya0, yb1, f[0][1]);
        f[1][0] = fmaf(ya1, yb0, f[1][0]);
        f[1][1] = fmaf(ya1, yb1, f[1][1]);
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) acc[a][b] += static_cast<double>(f[a][b]);
      __syncthreads();
    }
    double *pp = gpart + static_cast<int64_t>(blockIdx.x) * P * P;
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 2; ++b) __stcg(pp + (2 * ta + a) * P + 2 * tb + b, acc[a][b]);
    lq_grid_barrier(bar, ++nbar * nct);

    // 2. G = sum of the partials, entries split over the grid's warps
    for (int e = static_cast<int>(blockIdx.x) * 8 + warp; e < P * P; e += static_cast<int>(nct) * 8) {
      double v = 0.0;
      for (unsigned int b = lane; b < nct; b += 32) v += __ldcg(gpart + static_cast<int64_t>(b) * P * P + e);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) __stcg(G + e, v);
    }
    lq_grid_barrier(bar, ++nbar * nct);

    // 3. Cholesky in one warp: lane i holds row i (identity past p)
    if (warp == 0) {
      float a[P];
#pragma unroll
      for (int j = 0; j < P; ++j)
        a[j] = (lane < p && j < p) ? static_cast<float>(__ldcg(G + lane * P + j)) : ((lane == j) ? 1.f : 0.f);
      float mx = 0.f;
#pragma unroll
      for (int j = 0; j < P; ++j)
        if (j == lane && lane < p) mx = a[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float floor_v = fmaxf(mx, 1e-30f) * 1e-12f;
      lq_chol_warp_step<0>(a, lane, p, floor_v, sCol);
#pragma unroll
      for (int j = 0; j < P; ++j)
        sL[lane][j] = (lane < p && j < p) ? ((j <= lane) ? a[j] : 0.f) : ((lane == j) ? 1.f : 0.f);
      float dgl = 1.f;  // L[lane][lane]
#pragma unroll
      for (int j = 0; j < P; ++j)
        if (j == lane && lane < p) dgl = a[j];
      sRinv[lane] = 1.0f / dgl;
    }
    __syncthreads();
    // rows of this CTA: y <- y L^{-T} (forward substitution per row)
    for (int64_t i = r0 + tid; i < r1; i += 256) {
      float y[P];
#pragma unroll
      for (int c = 0; c < P; c += 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(Y + i * P + c));
        y[c] = v.x; y[c + 1] = v.y; y[c + 2] = v.z; y[c + 3] = v.w;
      }
#pragma unroll
      for (int c = 0; c < P; ++c) {
        float acc2 = y[c];
#pragma unroll
        for (int b = 0; b < c; ++b) acc2 = fmaf(-sL[c][b], y[b], acc2);
        y[c] = (c < p) ? acc2 * sRinv[c] : 0.f;
      }
#pragma unroll
      for (int c = 0; c < P; c += 4)
        __stcg(reinterpret_cast<float4 *>(Y + i * P + c), make_float4(y[c], y[c + 1], y[c + 2], y[c + 3]));
    }
    // the next round reads only this CTA's own rows (after this barrier); G
    // and the partials are rewritten only after the next grid barrier
    __syncthreads();
  }
  // leave: the last CTA out resets the counters
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(bar + 1, 1u) == nct - 1u) {
      bar[0] = 0u;
      bar[1] = 0u;
      __threadfence();
    }
  }
}

// One CTA of kLqJacThreads threads: parallel cyclic Jacobi eigen-
// decomposition (fp32) of the symmetric leading p x p block of G (accumulated
// in fp64), with the round-robin ("circle") pair ordering, so that n / 2
// disjoint rotations run at once (n = p rounded up to even; a padding row and
// column stay zero).  In round t the pairs are (n-1, t) and ((t+k) mod (n-1),
// (t-k) mod (n-1)), k = 1 .. n/2-1; the whole schedule is tabulated once.  A
// round takes two barriers: the rotations of all pairs are formed (the
// reciprocal square root for the cosine), then A <- J^T A J is applied one
// 2 x 2 block (a pair of rows by a pair of columns, rows first) per item,
// together with E <- E J; each thread's items are the same in every round.
// Sweeps stop once the off-diagonal mass is at the fp32 noise level.  Outputs
// the eigenvalues sorted descending (lam[P], zero past p) and the matching
// eigenvectors as the columns of V (fp32 [P x P], V[row * P + col]).
constexpr int kLqJacThreads = 512;

template <int P>
constexpr size_t lq_jacobi_smem() {
  return 2 * static_cast<size_t>(P) * (P + 1) * sizeof(float) + static_cast<size_t>(P - 1) * (P / 2) * 2;
}

template <int P>
__global__ void __launch_bounds__(kLqJacThreads)
lq_jacobi_kernel(const double *__restrict__ G, int p, float *__restrict__ lam, float *__restrict__ V) {
  extern __shared__ float lq_jac_smem[];  // A, E (P x (P + 1) each), then the pair schedule
  float (*A)[P + 1] = reinterpret_cast<float (*)[P + 1]>(lq_jac_smem);
  float (*E)[P + 1] = reinterpret_cast<float (*)[P + 1]>(lq_jac_smem + P * (P + 1));
  unsigned char (*sched)[P / 2][2] = reinterpret_cast<unsigned char (*)[P / 2][2]>(lq_jac_smem + 2 * P * (P + 1));
  __shared__ float cs[P / 2][2];
  __shared__ float s_off, s_dg;
  __shared__ int order[P];
  const int tid = threadIdx.x;
  const int n = p + (p & 1);
  const int np = n / 2;
  for (int t = tid; t < P * P; t += kLqJacThreads) {
    const int i = t / P, j = t % P;
    A[i][j] = (i < p && j < p) ? static_cast<float>(G[i * P + j]) : 0.f;
    E[i][j] = (i == j) ? 1.f : 0.f;
  }
  for (int t = tid; t < (n - 1) * np; t += kLqJacThreads) {
    const int step = t / np, k = t % np, m = n - 1;
    const int x = (k == 0) ? m : (step + k) % m;
    const int y = (k == 0) ? step : (step - k + m) % m;
    sched[step][k][0] = static_cast<unsigned char>(x < y ? x : y);
    sched[step][k][1] = static_cast<unsigned char>(x < y ? y : x);
  }
  // this thread's items (the same every round): blocks (k1, k2), then E rows
  constexpr int kIpt = ((P / 2) * (P / 2) + (P / 2) * P + kLqJacThreads - 1) / kLqJacThreads;  // items per thread
  const int items = np * np + np * n;
  int it_k1[kIpt], it_k2[kIpt], it_row[kIpt];
#pragma unroll
  for (int u = 0; u < kIpt; ++u) {
    const int t = tid + u * kLqJacThreads;
    if (t < np * np) {
      it_k1[u] = t / np;
      it_k2[u] = t % np;
      it_row[u] = -1;
    } else {
      const int v = t - np * np;
      it_k1[u] = it_k2[u] = v / n;
      it_row[u] = v % n;
    }
  }
  __syncthreads();
  for (int sweep = 0; sweep < 15; ++sweep) {
    if (tid < 32) {  // convergence: off-diagonal mass against the diagonal
      float off = 0.f, dg = 0.f;
      for (int t = tid; t < n * n; t += 32) {
        const int i = t / n, j = t % n;
        const float v = A[i][j] * A[i][j];
        if (i == j) dg += v; else off += v;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        off += __shfl_xor_sync(0xffffffffu, off, o);
        dg += __shfl_xor_sync(0xffffffffu, dg, o);
      }
      if (tid == 0) { s_off = off; s_dg = dg; }
    }
    __syncthreads();
    if (s_off <= 1e-10f * s_dg) break;  // off-diagonal mass at the fp32 noise level
    for (int step = 0; step < n - 1; ++step) {
      if (tid < np) {  // rotation of pair tid
        const int a = sched[step][tid][0], b = sched[step][tid][1];
        const float aij = A[a][b];
        float c = 1.f, sn = 0.f;
        if (fabsf(aij) > 1e-30f * (fabsf(A[a][a]) + fabsf(A[b][b]))) {
          const float theta = (A[b][b] - A[a][a]) / (2.f * aij);
          const float tt = copysignf(1.f, theta) / (fabsf(theta) + sqrtf(theta * theta + 1.f));
          c = rsqrtf(tt * tt + 1.f);
          sn = tt * c;
        }
        cs[tid][0] = c;
        cs[tid][1] = sn;
      }
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kIpt; ++u) {
        if (tid + u * kLqJacThreads >= items) break;
        const int k1 = it_k1[u], k2 = it_k2[u];
        const int a = sched[step][k1][0], b = sched[step][k1][1];
        const float c1 = cs[k1][0], s1 = cs[k1][1];
        if (it_row[u] < 0) {
          const int c0 = sched[step][k2][0], d0 = sched[step][k2][1];
          const float c2 = cs[k2][0], s2 = cs[k2][1];
          const float ra_c = c1 * A[a][c0] - s1 * A[b][c0], ra_d = c1 * A[a][d0] - s1 * A[b][d0];
          const float rb_c = s1 * A[a][c0] + c1 * A[b][c0], rb_d = s1 * A[a][d0] + c1 * A[b][d0];
          A[a][c0] = c2 * ra_c - s2 * ra_d;
          A[a][d0] = s2 * ra_c + c2 * ra_d;
          A[b][c0] = c2 * rb_c - s2 * rb_d;
          A[b][d0] = s2 * rb_c + c2 * rb_d;
        } else {
          const int row = it_row[u];
          const float ea = E[row][a], eb = E[row][b];
          E[row][a] = c1 * ea - s1 * eb;
          E[row][b] = s1 * ea + c1 * eb;
        }
      }
      __syncthreads();
    }
  }
  // descending order of the eigenvalues: rank of each (ties by index)
  for (int i = tid; i < P; i += kLqJacThreads) {
    if (i < p) {
      const float di = A[i][i];
      int rank = 0;
      for (int j = 0; j < p; ++j) {
        const float dj = A[j][j];
        rank += (dj > di || (dj == di && j < i)) ? 1 : 0;
      }
      order[rank] = i;
    } else {
      order[i] = i;
    }
  }
  __syncthreads();
  for (int i = tid; i < P; i += kLqJacThreads) lam[i] = (i < p) ? A[order[i]][order[i]] : 0.f;
  for (int t = tid; t < P * P; t += kLqJacThreads) {
    const int row = t / P, col = t % P;
    V[t] = (col < p) ? E[row][order[col]] : 0.f;
  }
}

// out[i, q] = sum_b in[i, b] * V[b, q] * scale[q]  for q < r;  in: n x P fp32.
// for_A == 0 (B): coefficient V[b, q] sqrt(sigma_q) / sqrt(s); for_A == 1 (A):
// V[b, q] / (sqrt(sigma_q) sqrt(s)), sigma_q = sqrt(lam_q) (lam: eigenvalues of
// the Gram matrix).  transpose_out: out[q * n + i] (r x n) instead of out[i * r + q].
template <int P>
__global__ void __launch_bounds__(256)
lq_project_kernel(const float *__restrict__ in, int64_t n, const float *__restrict__ V,
                  const float *__restrict__ lam, int r, float s, int for_A,
                  float *__restrict__ out, int transpose_out) {
  __shared__ float sC[P][P + 1];
  for (int t = threadIdx.x; t < P * P; t += blockDim.x) {
    const int b = t / P, q = t % P;
    float cval = 0.f;
    if (q < r) {
      const float sigma = sqrtf(fmaxf(lam[q], 0.f));
      const float rs = sqrtf(sigma);
      const float sc = for_A ? ((rs > 0.f) ? 1.f / (rs * sqrtf(s)) : 0.f) : rs / sqrtf(s);
      cval = V[b * P + q] * sc;
    }
    sC[b][q] = cval;
  }
  __syncthreads();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    for (int q0 = 0; q0 < r; q0 += 16) {
      float acc[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) acc[q] = 0.f;
      for (int b = 0; b < P; ++b) {
        const float x = in[i * P + b];
#pragma unroll
        for (int q = 0; q < 16; ++q) acc[q] = fmaf(x, sC[b][(q0 + q) < P ? q0 + q : P - 1], acc[q]);
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        if (q0 + q >= r) break;
        if (transpose_out) out[static_cast<int64_t>(q0 + q) * n + i] = acc[q];
        else out[i * r + q0 + q] = acc[q];
      }
    }
  }
}

// partial[block] = sum over its elements of (R - s * B A)^2.  Tiles of 64
// rows x 128 columns (grid-strided); thread (8 rows 8 (tid / 32) .., 4 columns
// 4 (tid % 32) ..): B A in fp32 from shared-memory tiles of 16 adapter
// columns at a time, the 32 squared differences summed in fp32, tiles and the
// CTA's threads summed in fp64.
constexpr int kRnRows = 64, kRnCols = 128;

__global__ void __launch_bounds__(256)
resid_norm_kernel(const float *__restrict__ R, const float *__restrict__ B, const float *__restrict__ A,
                  int64_t d, int64_t k, int r, float s, double *__restrict__ partial) {
  __shared__ __align__(16) float sA[16][kRnCols];
  __shared__ __align__(16) float sB[kRnRows][16 + 4];
  __shared__ double red[256];
  const int tid = threadIdx.x, rg = tid >> 5, cg = tid & 31;
  const int64_t tiles_c = (k + kRnCols - 1) / kRnCols, tiles = tiles_c * ((d + kRnRows - 1) / kRnRows);
  double total = 0.0;
  for (int64_t tl = blockIdx.x; tl < tiles; tl += gridDim.x) {
    const int64_t r0 = (tl / tiles_c) * kRnRows, c0 = (tl % tiles_c) * kRnCols;
    float acc[8][4] = {};
    for (int q0 = 0; q0 < r; q0 += 16) {
      for (int t = tid; t < 16 * kRnCols; t += 256) {
        const int q = t / kRnCols, c = t % kRnCols;
        sA[q][c] = (q0 + q < r && c0 + c < k) ? __ldg(A + static_cast<int64_t>(q0 + q) * k + c0 + c) : 0.f;
      }
      for (int t = tid; t < kRnRows * 16; t += 256) {
        const int i = t / 16, q = t % 16;
        sB[i][q] = (q0 + q < r && r0 + i < d) ? __ldg(B + (r0 + i) * r + q0 + q) : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 av = *reinterpret_cast<const float4 *>(&sA[q][4 * cg]);
#pragma unroll
        for (int a = 0; a < 8; ++a) {
          const float bv = sB[8 * rg + a][q];
          acc[a][0] = fmaf(bv, av.x, acc[a][0]);
          acc[a][1] = fmaf(bv, av.y, acc[a][1]);
          acc[a][2] = fmaf(bv, av.z, acc[a][2]);
          acc[a][3] = fmaf(bv, av.w, acc[a][3]);
        }
      }
      __syncthreads();
    }
    float sq = 0.f;
    const int64_t col = c0 + 4 * cg;
    if (col < k) {
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        const int64_t row = r0 + 8 * rg + a;
        if (row < d) {
          const float4 rv = __ldcs(reinterpret_cast<const float4 *>(R + row * k + col));
          const float e0 = fmaf(-s, acc[a][0], rv.x), e1 = fmaf(-s, acc[a][1], rv.y);
          const float e2 = fmaf(-s, acc[a][2], rv.z), e3 = fmaf(-s, acc[a][3], rv.w);
          sq = fmaf(e0, e0, sq);
          sq = fmaf(e1, e1, sq);
          sq = fmaf(e2, e2, sq);
          sq = fmaf(e3, e3, sq);
        }
      }
    }
    total += static_cast<double>(sq);
  }
  red[tid] = total;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (tid < w) red[tid] += red[tid + w];
    __syncthreads();
  }
  if (tid == 0) partial[blockIdx.x] = red[0];
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
