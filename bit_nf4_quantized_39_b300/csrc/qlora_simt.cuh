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
// Adapter projection  C[m, n] = s * sum_kk P[m, kk] * Qop(n, kk)   (fp32 out)
// with Qop(n, kk) = Qm[n * qs_n + kk * qs_k] and P bf16 [M x K] row-major,
// on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate).
// CTA tile 64 x TN (4 warps of 16 rows x TN / 8 n8-tiles; TN = 16 for ranks up
// to 16, else 64), K staged 64 at a time
// through padded shared-memory tiles (row stride 72 elements, so fragment
// loads do not conflict).  K is split over gridDim.z CTAs of kchunk columns
// each (a multiple of 64); split z writes its partial sums to
// part + z * M * N, and lora_reduce_kernel adds the splits in order.
// ---------------------------------------------------------------------------
constexpr int kProjTM = 64, kProjTK = 64, kProjStride = kProjTK + 8;
constexpr int kProjMaxSplit = 16;

__device__ __forceinline__ void mma_bf16_16816_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                   uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int TN>
__global__ void __launch_bounds__(128)
lora_proj_kernel(const uint16_t *__restrict__ P, int64_t M, int64_t K,
                 const uint16_t *__restrict__ Qm, int64_t N, int64_t qs_n, int64_t qs_k,
                 float s, int64_t kchunk, float *__restrict__ part) {
  __shared__ __align__(16) uint16_t sP[kProjTM][kProjStride];
  __shared__ __align__(16) uint16_t sQ[TN][kProjStride];
  constexpr int NT = TN / 8;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kProjTM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * TN;
  const int64_t kb = static_cast<int64_t>(blockIdx.z) * kchunk;
  const int64_t ke = (kb + kchunk < K) ? kb + kchunk : K;
  const bool pvec = (K % 8) == 0;
  const bool qvec = qs_k == 1 && (qs_n % 8) == 0;
  float acc[NT][4] = {};
  for (int64_t k0 = kb; k0 < ke; k0 += kProjTK) {
    // P tile: 64 rows x 64 columns
    if (pvec) {
      for (int i = tid; i < kProjTM * kProjTK / 8; i += 128) {
        const int r = i >> 3, c = (i & 7) * 8;
        const int64_t gm = m0 + r, gk = k0 + c;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (gm < M && gk + 8 <= ke) v = __ldg(reinterpret_cast<const uint4 *>(P + gm * K + gk));
        else if (gm < M)
          for (int e = 0; e < 8; ++e)
            if (gk + e < ke) reinterpret_cast<uint16_t *>(&v)[e] = P[gm * K + gk + e];
        *reinterpret_cast<uint4 *>(&sP[r][c]) = v;
      }
    } else {
      for (int i = tid; i < kProjTM * kProjTK; i += 128) {
        const int r = i / kProjTK, c = i % kProjTK;
        const int64_t gm = m0 + r, gk = k0 + c;
        sP[r][c] = (gm < M && gk < ke) ? P[gm * K + gk] : static_cast<uint16_t>(0);
      }
    }
    // Q tile: sQ[n][kk] = Qop(n0 + n, k0 + kk)
    if (qvec) {
      for (int i = tid; i < TN * kProjTK / 8; i += 128) {
        const int n = i >> 3, c = (i & 7) * 8;
        const int64_t gn = n0 + n, gk = k0 + c;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (gn < N && gk + 8 <= ke) v = __ldg(reinterpret_cast<const uint4 *>(Qm + gn * qs_n + gk));
        else if (gn < N)
          for (int e = 0; e < 8; ++e)
            if (gk + e < ke) reinterpret_cast<uint16_t *>(&v)[e] = Qm[gn * qs_n + gk + e];
        *reinterpret_cast<uint4 *>(&sQ[n][c]) = v;
      }
    } else {
      // consecutive threads take consecutive n (contiguous when qs_n == 1)
      for (int i = tid; i < TN * kProjTK; i += 128) {
        const int n = i % TN, c = i / TN;
        const int64_t gn = n0 + n, gk = k0 + c;
        sQ[n][c] = (gn < N && gk < ke) ? Qm[gn * qs_n + gk * qs_k] : static_cast<uint16_t>(0);
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kProjTK; kk += 16) {
      const int r = warp * 16 + g;
      const uint32_t a0 = *reinterpret_cast<const uint32_t *>(&sP[r][kk + 2 * t]);
      const uint32_t a1 = *reinterpret_cast<const uint32_t *>(&sP[r + 8][kk + 2 * t]);
      const uint32_t a2 = *reinterpret_cast<const uint32_t *>(&sP[r][kk + 2 * t + 8]);
      const uint32_t a3 = *reinterpret_cast<const uint32_t *>(&sP[r + 8][kk + 2 * t + 8]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint32_t b0 = *reinterpret_cast<const uint32_t *>(&sQ[nt * 8 + g][kk + 2 * t]);
        const uint32_t b1 = *reinterpret_cast<const uint32_t *>(&sQ[nt * 8 + g][kk + 2 * t + 8]);
        mma_bf16_16816_acc(acc[nt], a0, a1, a2, a3, b0, b1);
      }
    }
    __syncthreads();
  }
  float *C = part + static_cast<int64_t>(blockIdx.z) * M * N;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t gm = m0 + warp * 16 + g + 8 * (e >> 1), gn = n0 + nt * 8 + 2 * t + (e & 1);
      if (gm < M && gn < N) C[gm * N + gn] = s * acc[nt][e];
    }
  }
}

// Pipelined variant for 16-byte aligned operands (K % 8 == 0; Qop either
// contiguous along kk, kQT == false: Qm[n * qs_n + kk] with qs_n % 8 == 0, or
// contiguous along n, kQT == true: Qm[kk * qs_k + n] with qs_k % 8 == 0 and
// N % 8 == 0).  The same 64 x TN tile and split-K as lora_proj_kernel, but
// the P and Q tiles of kProjStages K-steps are in flight at once through
// 16-byte cp.async (zero-filled past the matrix), one CTA barrier per step.
constexpr int kProjStages = 4;

template <int TN, bool kQT>
__host__ __device__ constexpr int proj_q_tile_bytes() {
  return kQT ? kProjTK * (TN + 8) * 2 : TN * kProjStride * 2;
}
template <int TN, bool kQT>
__host__ __device__ constexpr int proj_stage_bytes() {
  return kProjTM * kProjStride * 2 + proj_q_tile_bytes<TN, kQT>();
}
template <int TN, bool kQT>
__host__ __device__ constexpr int proj_pipe_smem() {
  return kProjStages * proj_stage_bytes<TN, kQT>();
}

__device__ __forceinline__ void proj_cp16(uint32_t dst, const void *src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(ok ? 16u : 0u)
               : "memory");
}

template <int TN, bool kQT>
__global__ void __launch_bounds__(128)
lora_proj_pipe_kernel(const uint16_t *__restrict__ P, int64_t M, int64_t K,
                      const uint16_t *__restrict__ Qm, int64_t N, int64_t qs_n, int64_t qs_k,
                      float s, int64_t kchunk, float *__restrict__ part) {
  extern __shared__ __align__(16) uint8_t proj_smem[];
  constexpr int NT = TN / 8;
  constexpr int kQS = kQT ? TN + 8 : kProjStride;  // row stride of the Q tile (elements)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kProjTM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * TN;
  const int64_t kb = static_cast<int64_t>(blockIdx.z) * kchunk;
  const int64_t ke = (kb + kchunk < K) ? kb + kchunk : K;
  const int nsteps = static_cast<int>((ke - kb + kProjTK - 1) / kProjTK);
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(proj_smem));

  auto load = [&](int slot, int64_t k0) {
    const uint32_t sp = sbase + slot * proj_stage_bytes<TN, kQT>();
    const uint32_t sq = sp + kProjTM * kProjStride * 2;
#pragma unroll
    for (int j = 0; j < kProjTM * kProjTK / 8 / 128; ++j) {  // P: 64 rows x 8 chunks
      const int i = tid + 128 * j, r = i >> 3, c = (i & 7) * 8;
      const int64_t gm = m0 + r, gk = k0 + c;
      const bool ok = gm < M && gk + 8 <= ke;
      proj_cp16(sp + (r * kProjStride + c) * 2, ok ? P + gm * K + gk : P, ok);
    }
    if constexpr (!kQT) {  // Q tile [n][kk]
      for (int i = tid; i < TN * 8; i += 128) {
        const int n = i >> 3, c = (i & 7) * 8;
        const int64_t gn = n0 + n, gk = k0 + c;
        const bool ok = gn < N && gk + 8 <= ke;
        proj_cp16(sq + (n * kQS + c) * 2, ok ? Qm + gn * qs_n + gk : Qm, ok);
      }
    } else {  // Q tile [kk][n]
      for (int i = tid; i < kProjTK * (TN / 8); i += 128) {
        const int kk = i / (TN / 8), c = (i % (TN / 8)) * 8;
        const int64_t gk = k0 + kk, gn = n0 + c;
        const bool ok = gk < ke && gn + 8 <= N;
        proj_cp16(sq + (kk * kQS + c) * 2, ok ? Qm + gk * qs_k + gn : Qm, ok);
      }
    }
  };

  float acc[NT][4] = {};
#pragma unroll
  for (int st = 0; st < kProjStages - 1; ++st) {
    if (st < nsteps) load(st, kb + static_cast<int64_t>(st) * kProjTK);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int step = 0; step < nsteps; ++step) {
    asm volatile("cp.async.wait_group %0;" ::"n"(kProjStages - 2) : "memory");
    __syncthreads();  // stage `step` visible to all; stage step - 1 no longer read
    const int nxt = step + kProjStages - 1;
    if (nxt < nsteps) load(nxt % kProjStages, kb + static_cast<int64_t>(nxt) * kProjTK);
    asm volatile("cp.async.commit_group;" ::: "memory");
    const uint8_t *stg = proj_smem + (step % kProjStages) * proj_stage_bytes<TN, kQT>();
    const uint16_t *sP = reinterpret_cast<const uint16_t *>(stg);
    const uint16_t *sQ = reinterpret_cast<const uint16_t *>(stg + kProjTM * kProjStride * 2);
#pragma unroll
    for (int kk = 0; kk < kProjTK; kk += 16) {
      const int r = warp * 16 + g;
      const uint32_t a0 = *reinterpret_cast<const uint32_t *>(sP + r * kProjStride + kk + 2 * t);
      const uint32_t a1 = *reinterpret_cast<const uint32_t *>(sP + (r + 8) * kProjStride + kk + 2 * t);
      const uint32_t a2 = *reinterpret_cast<const uint32_t *>(sP + r * kProjStride + kk + 2 * t + 8);
      const uint32_t a3 = *reinterpret_cast<const uint32_t *>(sP + (r + 8) * kProjStride + kk + 2 * t + 8);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        uint32_t b0, b1;
        if constexpr (!kQT) {
          b0 = *reinterpret_cast<const uint32_t *>(sQ + (nt * 8 + g) * kQS + kk + 2 * t);
          b1 = *reinterpret_cast<const uint32_t *>(sQ + (nt * 8 + g) * kQS + kk + 2 * t + 8);
        } else {
          const uint16_t *q = sQ + (kk + 2 * t) * kQS + nt * 8 + g;
          b0 = static_cast<uint32_t>(q[0]) | (static_cast<uint32_t>(q[kQS]) << 16);
          b1 = static_cast<uint32_t>(q[8 * kQS]) | (static_cast<uint32_t>(q[9 * kQS]) << 16);
        }
        mma_bf16_16816_acc(acc[nt], a0, a1, a2, a3, b0, b1);
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  float *C = part + static_cast<int64_t>(blockIdx.z) * M * N;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t gm = m0 + warp * 16 + g + 8 * (e >> 1), gn = n0 + nt * 8 + 2 * t + (e & 1);
      if (gm < M && gn < N) C[gm * N + gn] = s * acc[nt][e];
    }
  }
}

// C = sum over the S splits of part (in split order).  Writes the fp32 result
// to C32 (if not null) and, if C2 is not null, its bf16 hi/lo split
// C2[m, :] = [bf16(c) | bf16(c - bf16(c)) | 0], each half zero-padded to R
// columns and the row zero-padded to its pitch ld2 >= 2R.
__global__ void lora_reduce_kernel(const float *__restrict__ part, int S, int64_t M, int64_t N,
                                   float *__restrict__ C32, int R, uint16_t *__restrict__ C2, int64_t ld2) {
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
    C2[m * ld2 + j] = hi;
    C2[m * ld2 + R + j] = f32_to_bf16_bits(v - bf16_bits_to_f32(hi));
    for (int64_t p = 2 * R + j; p < ld2; p += R) C2[m * ld2 + p] = 0;
  }
}

// lora_reduce_kernel four columns at a time (N, R and ld2 multiples of 4, C32
// and C2 16- and 8-byte aligned): thread (m, c4) sums columns 4 c4 .. + 3 of
// row m over the splits in split order (the same sums) and writes them, or
// the zero padding of C2 when 4 c4 >= N.
__global__ void lora_reduce4_kernel(const float *__restrict__ part, int S, int64_t M, int64_t N,
                                    float *__restrict__ C32, int R, uint16_t *__restrict__ C2, int64_t ld2) {
  const int64_t cols4 = (C2 ? R : N) / 4;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= M * cols4) return;
  const int64_t m = i / cols4, j = (i % cols4) * 4;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (j < N)
    for (int z = 0; z < S; ++z) {
      const float4 w = *reinterpret_cast<const float4 *>(part + (static_cast<int64_t>(z) * M + m) * N + j);
      v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
    }
  if (C32 && j < N) *reinterpret_cast<float4 *>(C32 + m * N + j) = v;
  if (C2) {
    const float f[4] = {v.x, v.y, v.z, v.w};
    uint32_t hi[2], lo[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint16_t h0 = f32_to_bf16_bits(f[2 * e]), h1 = f32_to_bf16_bits(f[2 * e + 1]);
      hi[e] = h0 | (static_cast<uint32_t>(h1) << 16);
      lo[e] = f32_to_bf16_bits(f[2 * e] - bf16_bits_to_f32(h0)) |
              (static_cast<uint32_t>(f32_to_bf16_bits(f[2 * e + 1] - bf16_bits_to_f32(h1))) << 16);
    }
    *reinterpret_cast<uint2 *>(C2 + m * ld2 + j) = make_uint2(hi[0], hi[1]);
    *reinterpret_cast<uint2 *>(C2 + m * ld2 + R + j) = make_uint2(lo[0], lo[1]);
    for (int64_t q = 2 * R + j; q < ld2; q += R) *reinterpret_cast<uint2 *>(C2 + m * ld2 + q) = make_uint2(0u, 0u);
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
