// common.cuh -- shared device helpers of the QLoRA NF4 library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "qlora_nf4.h"

// ---------------------------------------------------------------------------
// NF4 levels.  The 16 normal-quantile levels of the QLoRA NF4 data type
// ("QLoRA paper summary", NF4 bullet: quantiles of the standard normal,
// normalised to [-1, 1], with an exact zero).  Written as fp32 hex literals.
// ---------------------------------------------------------------------------
#define QN_NF4_LEVELS                                                          \
  {-0x1.0p+0f,      -0x1.647362p-1f, -0x1.0cd65cp-1f, -0x1.94653cp-2f,       \
   -0x1.234496p-2f, -0x1.7a6a7ap-3f, -0x1.74f0d2p-4f, 0x0p+0f,               \
   0x1.45f602p-4f,  0x1.4995bep-3f,  0x1.f809b4p-3f,  0x1.5a066cp-2f,        \
   0x1.c3496ap-2f,  0x1.200f52p-1f,  0x1.722760p-1f,  0x1.0p+0f}

// Decision thresholds: t_i is the largest fp32 not above the exact midpoint
// of levels i and i+1, so the nearest level (ties to the lower index) of an
// fp32 value v is the number of thresholds strictly below v.  The host checks
// this table against the levels at load time (qn_tables_consistent()).
#define QN_NF4_THRESHOLDS                                                      \
  {-0x1.b239b2p-1f, -0x1.38a4e0p-1f, -0x1.d708fap-2f, -0x1.5bd4eap-2f,       \
   -0x1.e079d4p-3f, -0x1.1a7172p-3f, -0x1.74f0d2p-5f, 0x1.45f602p-5f,        \
   0x1.ec90bep-4f,  0x1.a0cfb8p-3f,  0x1.2b05a2p-2f,  0x1.8ea7eap-2f,        \
   0x1.00da02p-1f,  0x1.491b58p-1f,  0x1.b913b0p-1f}

// Host copies (argument checks, qn_nf4_tables) and device copies (constant
// bank, read directly as instruction operands) of the same literal tables.
static constexpr float kNF4Levels[16] = QN_NF4_LEVELS;
static constexpr float kNF4Thresholds[15] = QN_NF4_THRESHOLDS;
__constant__ float c_nf4_levels[16] = QN_NF4_LEVELS;
__constant__ float c_nf4_thresholds[15] = QN_NF4_THRESHOLDS;

// Device status word written by bounded waits that expire (never a trap).
__device__ unsigned int g_qn_status;

enum : unsigned int { QN_DEV_OK = 0u, QN_DEV_TIMEOUT = 1u, QN_DEV_LAYOUT = 2u };

__device__ __forceinline__ void qn_flag_timeout() { atomicOr(&g_qn_status, QN_DEV_TIMEOUT); }

// Nearest NF4 level of a finite fp32 value in [-1, 1]: count of thresholds
// strictly below v.
__device__ __forceinline__ uint32_t nf4_code_of(float v) {
  uint32_t c = 0;
#pragma unroll
  for (int i = 0; i < 15; ++i) c += (v > c_nf4_thresholds[i]) ? 1u : 0u;
  return c;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half)
  return *reinterpret_cast<uint32_t *>(&h);
}

// Decoded double-quantised block constant: fp32(fp32(q * sigma) + mu), two
// separate roundings (no fused multiply-add).
__device__ __forceinline__ float dq_absmax(int8_t q, float sigma, float mu) {
  return __fadd_rn(__fmul_rn(static_cast<float>(q), sigma), mu);
}

struct QnNF4View {  // by-value kernel argument mirroring qn_nf4
  const uint8_t *codes;
  const float *absmax;
  const int8_t *absmax_q;
  const float *absmax_scale;
  const float *absmax_mean;
  int64_t d, k;
  int dq;
};

// Effective constant of block j (exact absmax, or its DQ decode).
__device__ __forceinline__ float block_scale(const QnNF4View &q, int64_t j) {
  if (q.dq) return dq_absmax(q.absmax_q[j], q.absmax_scale[j >> 8], *q.absmax_mean);
  return q.absmax[j];
}

__host__ __device__ constexpr int64_t qn_ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// Register decode of 4-bit codes into exactly bf16(fp32(level * m)): the 16
// levels scaled by a block constant m are built once as bf16 and split into
// low- and high-byte tables (four registers each); eight codes then become
// four bf16x2 words with byte permutes and two bit selects, no memory access.
// ---------------------------------------------------------------------------
namespace qn {
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Byte tables of the 16 scaled levels: L[i] / H[i] hold the low / high bytes
// of the bf16 values of levels 4i .. 4i+3.
struct ScaledLevels {
  uint32_t L[4], H[4];
};

__device__ __forceinline__ ScaledLevels scaled_levels(float m) {
  uint32_t P[8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    P[j] = pack_bf16x2(__fmul_rn(c_nf4_levels[2 * j], m), __fmul_rn(c_nf4_levels[2 * j + 1], m));
  ScaledLevels t;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    t.L[i] = prmt(P[2 * i], P[2 * i + 1], 0x6420u);
    t.H[i] = prmt(P[2 * i], P[2 * i + 1], 0x7531u);
  }
  return t;
}

// Eight 4-bit codes (element 0 in the low nibble) -> four bf16x2 words.
__device__ __forceinline__ void decode_word(uint32_t w, const ScaledLevels &t, uint32_t *out) {
  const uint32_t sel = w & 0x77777777u;   // level index within its half of the table
  const uint32_t w4 = w << 4;
  // byte masks: 0xFF where the code's bit 3 is set (upper half of the table)
  const uint32_t m_lo = prmt(w4, w, 0xD9C8u);
  const uint32_t m_hi = prmt(w4, w, 0xFBEAu);
  const uint32_t s_hi = sel >> 16;
  {
    const uint32_t la = prmt(t.L[0], t.L[1], sel), lb = prmt(t.L[2], t.L[3], sel);
    const uint32_t ha = prmt(t.H[0], t.H[1], sel), hb = prmt(t.H[2], t.H[3], sel);
    const uint32_t lo = (la & ~m_lo) | (lb & m_lo), hi = (ha & ~m_lo) | (hb & m_lo);
    out[0] = prmt(lo, hi, 0x5140u);
    out[1] = prmt(lo, hi, 0x7362u);
  }
  {
    const uint32_t la = prmt(t.L[0], t.L[1], s_hi), lb = prmt(t.L[2], t.L[3], s_hi);
    const uint32_t ha = prmt(t.H[0], t.H[1], s_hi), hb = prmt(t.H[2], t.H[3], s_hi);
    const uint32_t lo = (la & ~m_hi) | (lb & m_hi), hi = (ha & ~m_hi) | (hb & m_hi);
    out[2] = prmt(lo, hi, 0x5140u);
    out[3] = prmt(lo, hi, 0x7362u);
  }
}

}  // namespace qn
