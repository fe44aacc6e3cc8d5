// lora_grad.cuh -- gradients of the adapter factors of the QLoRA layer:
//
//   dB = s dY^T (X A^T)        (d x r)
//   dA = s (dY B)^T X          (r x k)
//
// ("QLoRA paper summary", abstract: gradients are back-propagated through the
// frozen 4-bit weight into the low-rank adapters; "PEFT course notes" §2.2:
// B in R^{d x r}, A in R^{r x k}.)  Both are contractions over the tokens:
// with V = u = s X A^T (or v = s dY B), M x r fp32, and P = dY (or X), M x N
// bf16,
//
//   C[q, n] = sum_m V[m, q] P[m, n]         q < r, n < N,
//
// which is dB^T (P = dY, V = u) or dA (P = X, V = v).  The call reads P once
// from HBM, so it is bandwidth bound; the arithmetic runs on mma.sync
// (m16n8k16, bf16 in, fp32 accumulate) with V split into bf16 hi + lo (about
// 16 significant bits).
//
// Kernels
//   lora_vt_pack_kernel  V (M x r fp32) -> Vt2 [2][Rp][Mp] bf16: rows q of
//                        bf16(V) and of bf16(V - bf16(V)), zero padded.
//   lora_grad_kernel     one CTA per 128 columns n x RCH ranks x one token
//                        split; token chunks of 32 double-buffered through
//                        shared memory by cp.async; A fragments (Vt2) by
//                        ldmatrix, B fragments (P, stored token-major) by
//                        ldmatrix.trans; fp32 partial sums per split.
//   lora_grad_reduce_kernel  sums the splits in order and writes C or C^T.
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace qn {

constexpr int kLgThreads = 128;                 // 4 warps, 32 columns each
constexpr int kLgTN = 128;                      // columns n per CTA
constexpr int kLgTK = 32;                       // tokens per stage
constexpr int kLgPPitch = kLgTN + 8;            // bf16 elements per staged P row (272 B: ldmatrix conflict-free)
constexpr int kLgVPitch = kLgTK + 8;            // bf16 elements per staged Vt2 row (80 B)
constexpr int kLgMaxRT = 4;                     // 16-rank tiles per CTA (64 ranks)
constexpr int kLgMaxSplit = 16;

__host__ __device__ constexpr int64_t lg_round(int64_t a, int64_t b) { return ((a + b - 1) / b) * b; }

// Rank chunk handled by one CTA (a multiple of 16, at most 64) and the padded rank count.
__host__ __device__ constexpr int lg_rch(int r) { return lg_round(r, 16) < 64 ? static_cast<int>(lg_round(r, 16)) : 64; }
__host__ __device__ constexpr int64_t lg_rp(int r) { return lg_round(r, lg_rch(r)); }

// Token splits: enough CTAs for about four per SM, each split a multiple of 32 tokens.
inline int lg_splits(int64_t M, int64_t N, int r) {
  const int64_t tiles = lg_round(N, kLgTN) / kLgTN * (lg_rp(r) / lg_rch(r));
  int64_t S = (600 + tiles - 1) / tiles;
  const int64_t smax = lg_round(M, kLgTK) / kLgTK;
  if (S > smax) S = smax;
  if (S > kLgMaxSplit) S = kLgMaxSplit;
  return S < 1 ? 1 : static_cast<int>(S);
}

__global__ void lora_vt_pack_kernel(const float *__restrict__ V, int64_t M, int r, int64_t Rp, int64_t Mp,
                                    uint16_t *__restrict__ vt2) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= Rp * Mp) return;
  const int64_t q = i / Mp, m = i % Mp;
  const float v = (q < r && m < M) ? V[m * r + q] : 0.f;
  const uint16_t hi = f32_to_bf16_bits(v);
  vt2[i] = hi;
  vt2[Rp * Mp + i] = f32_to_bf16_bits(v - bf16_bits_to_f32(hi));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// grid (ceil(N / 128), S, Rp / RCH); RT = RCH / 16.
// part[((split * Rp) + q) * N + n] = sum over the split's tokens of V[m, q] P[m, n].
template <int RT>
__global__ void __launch_bounds__(kLgThreads)
lora_grad_kernel(const uint16_t *__restrict__ P, int64_t M, int64_t N, const uint16_t *__restrict__ vt2,
                 int64_t Rp, int64_t Mp, int64_t tokens_per_split, float *__restrict__ part) {
  constexpr int RCH = RT * 16;
  __shared__ __align__(16) uint16_t sP[2][kLgTK][kLgPPitch];
  __shared__ __align__(16) uint16_t sV[2][2][RCH][kLgVPitch];   // [stage][hi/lo][rank][token]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kLgTN;
  const int split = blockIdx.y;
  const int64_t q0 = static_cast<int64_t>(blockIdx.z) * RCH;
  const int64_t mb = static_cast<int64_t>(split) * tokens_per_split;
  int64_t me = mb + tokens_per_split;
  if (me > M) me = M;
  const bool pvec = (N % 8) == 0 && (reinterpret_cast<uintptr_t>(P) & 15u) == 0;

  auto load_stage = [&](int st, int64_t m0) {
    // P: 32 tokens x 128 columns = 512 chunks of 8 bf16
#pragma unroll
    for (int c = 0; c < (kLgTK * kLgTN / 8) / kLgThreads; ++c) {
      const int idx = c * kLgThreads + tid;
      const int row = idx >> 4, col = (idx & 15) * 8;
      const int64_t m = m0 + row, n = n0 + col;
      uint16_t *dst = &sP[st][row][col];
      if (m < me && pvec && n + 8 <= N) {
        cp_async16(smem_u32(dst), P + m * N + n);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[e] = (m < me && n + e < N) ? P[m * N + n + e] : static_cast<uint16_t>(0);
      }
    }
    // Vt2: 2 halves x RCH ranks x 32 tokens (zero padded, always in range)
#pragma unroll
    for (int c = 0; c < (2 * RCH * kLgTK / 8 + kLgThreads - 1) / kLgThreads; ++c) {
      const int idx = c * kLgThreads + tid;
      if (idx < 2 * RCH * kLgTK / 8) {
        const int h = idx / (RCH * 4), rem = idx % (RCH * 4);
        const int q = rem >> 2, t8 = (rem & 3) * 8;
        cp_async16(smem_u32(&sV[st][h][q][t8]), vt2 + (static_cast<int64_t>(h) * Rp + q0 + q) * Mp + m0 + t8);
      }
    }
    cp_async_commit();
  };

  float acc[RT][4][4];
#pragma unroll
  for (int a = 0; a < RT; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[a][b][e] = 0.f;

  const int nchunks = static_cast<int>((me - mb + kLgTK - 1) / kLgTK);
  if (nchunks > 0) load_stage(0, mb);
  for (int ch = 0; ch < nchunks; ++ch) {
    const int st = ch & 1;
    if (ch + 1 < nchunks) {
      load_stage(st ^ 1, mb + static_cast<int64_t>(ch + 1) * kLgTK);
      cp_async_wait_group<1>();
    } else {
      cp_async_wait_group<0>();
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kLgTK; kk += 16) {
      // B fragments of the warp's four 8-column tiles (P stored [token][column]).
      uint32_t bf[4][2];
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int j = lane >> 3;  // matrix: (k half j & 1, n tile j >> 1)
        const uint32_t addr =
            smem_u32(&sP[st][kk + (j & 1) * 8 + (lane & 7)][warp * 32 + np * 16 + (j >> 1) * 8]);
        ldsm_x4_t(addr, bf[2 * np][0], bf[2 * np][1], bf[2 * np + 1][0], bf[2 * np + 1][1]);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int mt = 0; mt < RT; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(smem_u32(&sV[st][h][mt * 16 + (lane & 15)][kk + (lane >> 4) * 8]), a0, a1, a2, a3);
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) mma_16816(acc[mt][nt], a0, a1, a2, a3, bf[nt][0], bf[nt][1]);
        }
      }
    }
    __syncthreads();
  }

  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int mt = 0; mt < RT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t q = q0 + mt * 16 + g + 8 * (e >> 1);
        const int64_t n = n0 + warp * 32 + nt * 8 + 2 * t + (e & 1);
        if (n < N) part[(static_cast<int64_t>(split) * Rp + q) * N + n] = acc[mt][nt][e];
      }
}

// out = sum over the S splits (in order) of part, for q < r, n < N:
// transpose_out == 0: out[q * N + n]  (dA, r x k);  1: out[n * r + q]  (dB, d x r).
__global__ void lora_grad_reduce_kernel(const float *__restrict__ part, int S, int64_t Rp, int64_t N, int r,
                                        int transpose_out, float *__restrict__ out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(r) * N) return;
  int64_t q, n;
  if (transpose_out) { n = i / r; q = i % r; }   // consecutive threads write consecutive dB entries
  else { q = i / N; n = i % N; }
  float v = 0.f;
  for (int z = 0; z < S; ++z) v += part[(static_cast<int64_t>(z) * Rp + q) * N + n];
  out[i] = v;
}

}  // namespace qn
