// qlora_f32.cuh -- the QLoRA layer with fp32 compute dtype (X, A, B, Y, dY,
// dX all fp32; the weight enters as its exact fp32 dequantisation):
//
//   Y  = X deq(Q)^T + s (X A^T) B^T,      dX = dY deq(Q) + s (dY B) A
//
// The layer is that of "PEFT course notes" §2.2; the compute dtype is the
// bnb_4bit_compute_dtype of "LoftQ explainer" §3.2 / "PEFT quantization
// guide", which may be fp32 (slower than bf16, as "LoftQ explainer" notes in
// its troubleshooting table).  There is no fp32 tensor-core path on B300
// other than tf32, which would round the operands, so the arithmetic runs on
// the CUDA cores in fp32 FMA.
//
// One tiled GEMM kernel serves all four products:
//   C[m, n] = scale * sum_{kk < K1} P1[m, kk] Op1(kk, n) + sum_{kk < K2} P2[m, kk] Op2(kk, n)
// P1, P2: fp32 row-major (M x K1, M x K2).  Op1: the NF4 weight, W'[n, kk]
// (forward) or W'[kk, n] (backward), or a plain fp32 matrix
// Op(kk, n) = F[n * sn + kk * sk].  Op2 (the adapter term, folded in as
// extra K) is a plain fp32 matrix.  Tile BM x 128, K chunks of 16 through
// shared memory; each thread holds (BM / 16) x 8 outputs.
#pragma once

#include "common.cuh"

namespace qn {

constexpr int kF32BN = 128, kF32BK = 16, kF32Threads = 256;

enum F32OpKind { F32_OP_MAT = 0, F32_OP_NF4_ROWS = 1, F32_OP_NF4_COLS = 2 };

struct F32Operand {
  int kind;            // F32OpKind
  QnNF4View q;         // NF4_ROWS: Op(kk, n) = W'[n, kk];  NF4_COLS: Op(kk, n) = W'[kk, n]
  const float *F;      // MAT: Op(kk, n) = F[n * sn + kk * sk]
  int64_t sn, sk;
};

struct F32Gemm {
  const float *P1;  int64_t K1;  F32Operand op1;
  const float *P2;  int64_t K2;  F32Operand op2;   // K2 = 0: no second term
  int64_t M, N;
  float scale;
  float *C;         // M x N fp32, row stride N
};

__device__ __forceinline__ float f32_nf4_at(const QnNF4View &q, int64_t e) {
  const uint32_t byte = q.codes[e >> 1];
  const uint32_t code = (e & 1) ? (byte >> 4) : (byte & 15u);
  return __fmul_rn(c_nf4_levels[code], block_scale(q, e >> 6));
}

// Op(kk, n) for one element (bounds already checked).
__device__ __forceinline__ float f32_op_at(const F32Operand &op, int64_t kk, int64_t n) {
  if (op.kind == F32_OP_MAT) return op.F[n * op.sn + kk * op.sk];
  if (op.kind == F32_OP_NF4_ROWS) return f32_nf4_at(op.q, n * op.q.k + kk);
  return f32_nf4_at(op.q, kk * op.q.k + n);
}

template <int BM>
__global__ void __launch_bounds__(kF32Threads)
f32_gemm_kernel(const F32Gemm gp) {
  constexpr int TM = BM / 16;  // rows per thread
  __shared__ float sP[kF32BK][BM + 4];
  __shared__ float sO[kF32BK][kF32BN + 4];
  __shared__ float s_lv[16];  // the levels, indexed per lane (a constant-bank read would serialise)
  const int tid = threadIdx.x;
  if (tid < 16) s_lv[tid] = c_nf4_levels[tid];
  __syncthreads();
  const int ty = tid / 16, tx = tid % 16;  // thread tile: rows ty*TM.., columns tx*8..
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kF32BN;
  float acc[TM][8];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  const int64_t Ktot = gp.K1 + gp.K2;
  for (int64_t k0 = 0; k0 < Ktot; k0 += kF32BK) {
    // P tile (BM x 16) -> sP[kk][m]
    for (int i = tid; i < BM * kF32BK; i += kF32Threads) {
      const int mm = i / kF32BK, kk = i % kF32BK;
      const int64_t m = m0 + mm, kg = k0 + kk;
      float v = 0.f;
      if (m < gp.M) {
        if (kg < gp.K1) v = gp.P1[m * gp.K1 + kg];
        else if (kg < Ktot) v = gp.P2[m * gp.K2 + (kg - gp.K1)];
      }
      sP[kk][mm] = v;
    }
    // Op tile (16 x 128) -> sO[kk][n]; the NF4 column layout reads 8
    // consecutive n of one weight row (4 code bytes) per thread.
    const bool in1 = k0 + kF32BK <= gp.K1;  // the whole chunk lies in the first term
    if (in1 && gp.op1.kind == F32_OP_NF4_COLS && (gp.N % 8) == 0) {
      const int kk = tid / 16, nn = (tid % 16) * 8;
      const int64_t kg = k0 + kk, n = n0 + nn;
      if (n < gp.N) {
        const QnNF4View &q = gp.op1.q;
        const int64_t e = kg * q.k + n;  // 8 consecutive elements inside one 64-block
        const uint32_t w = *reinterpret_cast<const uint32_t *>(q.codes + (e >> 1));
        const float m = block_scale(q, e >> 6);
#pragma unroll
        for (int j = 0; j < 8; ++j) sO[kk][nn + j] = __fmul_rn(s_lv[(w >> (4 * j)) & 15u], m);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) sO[kk][nn + j] = 0.f;
      }
    } else if (in1 && gp.op1.kind == F32_OP_NF4_ROWS) {
      // 8 consecutive kk of one weight row n per thread: (n, kk-half)
      const int nn = tid / 2, kh = (tid % 2) * 8;
      const int64_t n = n0 + nn, kg = k0 + kh;
      if (n < gp.N) {
        const QnNF4View &q = gp.op1.q;
        const int64_t e = n * q.k + kg;
        const uint32_t w = *reinterpret_cast<const uint32_t *>(q.codes + (e >> 1));
        const float m = block_scale(q, e >> 6);
#pragma unroll
        for (int j = 0; j < 8; ++j) sO[kh + j][nn] = __fmul_rn(s_lv[(w >> (4 * j)) & 15u], m);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) sO[kh + j][nn] = 0.f;
      }
    } else {
      for (int i = tid; i < kF32BK * kF32BN; i += kF32Threads) {
        const int kk = i / kF32BN, nn = i % kF32BN;
        const int64_t kg = k0 + kk, n = n0 + nn;
        float v = 0.f;
        if (n < gp.N) {
          if (kg < gp.K1) v = f32_op_at(gp.op1, kg, n);
          else if (kg < Ktot) v = f32_op_at(gp.op2, kg - gp.K1, n);
        }
        sO[kk][nn] = v;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kF32BK; ++kk) {
      float a[TM], b[8];
#pragma unroll
      for (int i = 0; i < TM; ++i) a[i] = sP[kk][ty * TM + i];
      const float4 b0 = *reinterpret_cast<const float4 *>(&sO[kk][tx * 8]);
      const float4 b1 = *reinterpret_cast<const float4 *>(&sO[kk][tx * 8 + 4]);
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w; b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int64_t m = m0 + ty * TM + i;
    if (m >= gp.M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t n = n0 + tx * 8 + j;
      if (n < gp.N) gp.C[m * gp.N + n] = gp.scale * acc[i][j];
    }
  }
}

}  // namespace qn
