// api.cu -- the C ABI of libqlora_nf4 (see include/qlora_nf4.h): argument
// checks, workspace carving, launch configuration and the LoftQ host loop.
// The whole library is one translation unit: the kernel headers are included
// here.

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <string>

#include "common.cuh"
#include "nf4_codec.cuh"
#include "qlora_simt.cuh"
#include "qlora_decode.cuh"
#include "qlora_skinny.cuh"
#include "qlora_m16.cuh"
#include "qlora_gemv.cuh"
#include "qlora_tc.cuh"
#include "lora_grad.cuh"
#include "qlora_f32.cuh"
#include "nf4_merge.cuh"
#include "loftq.cuh"

namespace {

thread_local std::string g_last_error;

qn_status fail(qn_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
qn_status fail(qn_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

qn_status cuda_check(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return QN_OK;
  return fail(QN_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define QN_TRY(expr)                 \
  do {                               \
    const qn_status st_ = (expr);    \
    if (st_ != QN_OK) return st_;    \
  } while (0)

// With QN_DEBUG_SYNC=1 in the environment every launch is followed by a
// device synchronisation, so that an asynchronous fault is reported with the
// name of the kernel that raised it.
bool debug_sync() {
  static const bool on = [] {
    const char *e = std::getenv("QN_DEBUG_SYNC");
    return e && e[0] == '1';
  }();
  return on;
}

qn_status launch_check(const char *what) {
  QN_TRY(cuda_check(cudaGetLastError(), what));
  if (debug_sync()) QN_TRY(cuda_check(cudaDeviceSynchronize(), what));
  return QN_OK;
}

#define QN_LAUNCH_CHECK(what) QN_TRY(launch_check(what))

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  static int cached[64] = {0};
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  int n = 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

// Checks the threshold table against the level table: t_i must be the largest
// fp32 not above the exact midpoint of levels i and i+1.
bool tables_consistent() {
  for (int i = 0; i < 15; ++i) {
    const double mid = (static_cast<double>(kNF4Levels[i]) + static_cast<double>(kNF4Levels[i + 1])) * 0.5;
    const float t = kNF4Thresholds[i];
    if (static_cast<double>(t) > mid) return false;
    const float up = std::nextafter(t, INFINITY);
    if (static_cast<double>(up) <= mid) return false;
  }
  return true;
}

struct Span {  // bump allocator over the caller's workspace
  char *base;
  size_t size, used;
  template <typename T> T *take(size_t count) {
    const size_t off = (used + 255) & ~static_cast<size_t>(255);
    used = off + count * sizeof(T);
    return reinterpret_cast<T *>(base + off);
  }
};

size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// The first kSemBytes of every workspace are a zero area: semaphores
// (grid-wide counters) and accumulators that must be zero before the first
// call on that workspace; every kernel that uses them returns them to zero
// before it exits.  Every other scratch buffer lives after it.
constexpr size_t kSemBytes = 256 * 1024;
// Word of the zero area where the LoftQ CholeskyQR2 kernel keeps its two
// grid-barrier counters (word 0 is the quantiser's ticket).
constexpr int kLqBarWord = 32;

qn_status check_nf4(const qn_nf4 *Q, bool need_dq_ptrs) {
  if (!Q) return fail(QN_EINVAL, "Q is NULL");
  if (Q->block != 64) return fail(QN_EUNSUPPORTED, "block must be 64 (got %d)", Q->block);
  if (Q->dq && Q->dq_block != 256) return fail(QN_EUNSUPPORTED, "dq_block must be 256 (got %d)", Q->dq_block);
  if (Q->d <= 0 || Q->k <= 0) return fail(QN_ESHAPE, "d and k must be positive");
  if (Q->d > (int64_t(1) << 40) / Q->k) return fail(QN_ESHAPE, "d*k too large");
  if (!Q->codes || !Q->absmax) return fail(QN_EINVAL, "codes/absmax NULL");
  if (!aligned(Q->codes, 16) || !aligned(Q->absmax, 16)) return fail(QN_EALIGN, "codes/absmax not 16-byte aligned");
  if (Q->dq && need_dq_ptrs) {
    if (!Q->absmax_q || !Q->absmax_scale || !Q->absmax_mean) return fail(QN_EINVAL, "dq pointers NULL");
    if (!aligned(Q->absmax_scale, 4) || !aligned(Q->absmax_mean, 4)) return fail(QN_EALIGN, "dq scale/mean misaligned");
  }
  return QN_OK;
}

QnNF4View view_of(const qn_nf4 *Q) {
  QnNF4View v;
  v.codes = Q->codes;
  v.absmax = Q->absmax;
  v.absmax_q = Q->absmax_q;
  v.absmax_scale = Q->absmax_scale;
  v.absmax_mean = Q->absmax_mean;
  v.d = Q->d;
  v.k = Q->k;
  v.dq = Q->dq ? 1 : 0;
  return v;
}

// Launch with programmatic stream serialisation (PDL): the kernel may start
// before the previous kernel on the stream has finished; the kernels
// themselves call griddepcontrol.wait before touching anything that the
// previous kernel may write.
template <typename... KArgs, typename... Args>
qn_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     const char *what, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  QN_TRY(cuda_check(cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...), what));
  QN_LAUNCH_CHECK(what);
  return QN_OK;
}

constexpr size_t kQuantWs = kSemBytes + qn::kNumBins * sizeof(unsigned long long);
// Byte offset in the zero area of the quantiser's exponent bins (2 KiB); the
// kernels return them to zero.
constexpr size_t kBinsOffset = 64 * 1024;

// Quantise n elements (internal; arguments already checked).  `bins` (2 KiB,
// zero on entry, zero again on exit)
// and `ticket` (one word, zero on entry, zero again on exit) are scratch.
qn_status launch_quantize(const void *W, qn_dtype wdt, const qn_nf4 *Q, unsigned long long *bins,
                          unsigned int *ticket, cudaStream_t st) {
  const int64_t n = Q->d * Q->k;
  const int64_t nfull = n / 64;
  const int64_t nblk = qn_ceil_div(n, 64);
  unsigned long long *b = Q->dq ? bins : nullptr;
  const int sms = sm_count();
  // The partial last block goes first: its constant must be in the bins
  // before the main kernel's last CTA forms the mean.
  if (nblk > nfull) {
    if (wdt == QN_F32)
      qn::nf4_quant_tail_kernel<float><<<1, 32, 0, st>>>(static_cast<const float *>(W), n, nfull, Q->codes,
                                                         Q->absmax, b);
    else
      qn::nf4_quant_tail_kernel<__nv_bfloat16><<<1, 32, 0, st>>>(static_cast<const __nv_bfloat16 *>(W), n, nfull,
                                                                 Q->codes, Q->absmax, b);
    QN_LAUNCH_CHECK("nf4_quant_tail_kernel");
  }
  {
    // Stages of 1 KiB of input, one per warp-iteration; two CTAs per SM
    // (80 KiB of copy ring and 31 KiB of tables each).
    const int64_t bps = (wdt == QN_F32) ? 4 : 8;
    const int64_t nst = qn_ceil_div(nfull, bps);
    int64_t grid = qn_ceil_div(nst, qn::kQuantWarps);
    const int64_t cap = static_cast<int64_t>(sms) * 2;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    QN_TRY(cuda_check((wdt == QN_F32)
                          ? cudaFuncSetAttribute(qn::nf4_quant_kernel<float>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, qn::kQuantSmem)
                          : cudaFuncSetAttribute(qn::nf4_quant_kernel<__nv_bfloat16>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, qn::kQuantSmem),
                      "cudaFuncSetAttribute(quantiser smem)"));
    // Two CTAs of 112 KiB per SM only fit with the largest shared-memory carveout.
    QN_TRY(cuda_check((wdt == QN_F32)
                          ? cudaFuncSetAttribute(qn::nf4_quant_kernel<float>,
                                                 cudaFuncAttributePreferredSharedMemoryCarveout, 100)
                          : cudaFuncSetAttribute(qn::nf4_quant_kernel<__nv_bfloat16>,
                                                 cudaFuncAttributePreferredSharedMemoryCarveout, 100),
                      "cudaFuncSetAttribute(quantiser carveout)"));
    // Size the grid to what is resident at once (the loop is grid-strided).
    int occ = 0;
    QN_TRY(cuda_check((wdt == QN_F32)
                          ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, qn::nf4_quant_kernel<float>,
                                                                          qn::kQuantThreads, qn::kQuantSmem)
                          : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, qn::nf4_quant_kernel<__nv_bfloat16>,
                                                                          qn::kQuantThreads, qn::kQuantSmem),
                      "quantiser occupancy"));
    if (occ < 1) occ = 1;
    if (grid > static_cast<int64_t>(sms) * occ) grid = static_cast<int64_t>(sms) * occ;
    if (wdt == QN_F32)
      qn::nf4_quant_kernel<float><<<static_cast<unsigned>(grid), qn::kQuantThreads, qn::kQuantSmem, st>>>(
          static_cast<const float *>(W), nfull, nblk, Q->codes, Q->absmax, b, ticket, Q->absmax_mean);
    else
      qn::nf4_quant_kernel<__nv_bfloat16><<<static_cast<unsigned>(grid), qn::kQuantThreads, qn::kQuantSmem, st>>>(
          static_cast<const __nv_bfloat16 *>(W), nfull, nblk, Q->codes, Q->absmax, b, ticket, Q->absmax_mean);
    QN_LAUNCH_CHECK("nf4_quant_kernel");
  }
  if (Q->dq) {
    const int64_t ngrp = qn_ceil_div(nblk, 256);
    int64_t grid = qn_ceil_div(ngrp, qn::kDqWarps);
    const int64_t cap = static_cast<int64_t>(sms) * 4;
    if (grid > cap) grid = cap;
    QN_TRY(launch_pdl(qn::nf4_dq_kernel, dim3(static_cast<unsigned>(grid)), dim3(qn::kDqWarps * 32), 0, st,
                      "nf4_dq_kernel", static_cast<const float *>(Q->absmax), nblk,
                      static_cast<const float *>(Q->absmax_mean), Q->absmax_q, Q->absmax_scale));
  }
  return QN_OK;
}

qn_status launch_dequantize(const qn_nf4 *Q, void *out, qn_dtype odt, cudaStream_t st) {
  const int64_t n = Q->d * Q->k;
  // One warp-iteration per 1024 elements; eight warps per CTA, eight CTAs per SM.
  const int64_t ntile = qn_ceil_div(n / 8, 32 * qn::kDeqWords);
  int64_t grid = qn_ceil_div(ntile > 0 ? ntile : 1, qn::kDeqThreads / 32);
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (grid > cap) grid = cap;
  if (odt == QN_BF16)
    qn::nf4_dequant_kernel<true><<<static_cast<unsigned>(grid), qn::kDeqThreads, 0, st>>>(view_of(Q), n, out);
  else
    qn::nf4_dequant_kernel<false><<<static_cast<unsigned>(grid), qn::kDeqThreads, 0, st>>>(view_of(Q), n, out);
  QN_LAUNCH_CHECK("nf4_dequant_kernel");
  return QN_OK;
}

// ----------------------------------------------------------------- the layer
bool use_decode(int64_t M, int64_t k) { return M == 1 && k <= qn::kDecMaxK; }
bool use_skinny(int64_t M, int64_t k) { return M <= qn::kSkMaxM && k <= 64 * qn::kSkMaxNb; }

// Split-K partial sums of the adapter projection (large-M paths).
size_t proj_ws_bytes(int64_t M, int32_t r) {
  return round256(static_cast<size_t>(qn::kProjMaxSplit) * M * r * sizeof(float));
}

size_t fwd_ws_bytes(int64_t M, int64_t d, int64_t k, int32_t r) {
  size_t b = kSemBytes + round256(static_cast<size_t>(M) * r * sizeof(float));  // u
  if (!use_skinny(M, k)) b += proj_ws_bytes(M, r) + qn::tc_fwd_ws_bytes(M, d, k, r);
  return b;
}

// Adapter gradients: u, v (M x r fp32), the projection's split-K partials,
// the bf16 hi/lo transposes of u and v, and the token-split partials of the
// larger of the two contractions.
size_t lg_ws_bytes(int64_t M, int64_t d, int64_t k, int32_t r) {
  const int64_t Rp = qn::lg_rp(r), Mp = qn::lg_round(M, qn::kLgTK);
  const int64_t Nmax = d > k ? d : k;
  const int Smax = qn::lg_splits(M, d, r) > qn::lg_splits(M, k, r) ? qn::lg_splits(M, d, r) : qn::lg_splits(M, k, r);
  // two independent chains (dB from u, dA from v), each with its own split partials
  return kSemBytes + 2 * round256(static_cast<size_t>(M) * r * sizeof(float)) + 2 * proj_ws_bytes(M, r) +
         2 * round256(static_cast<size_t>(2) * Rp * Mp * sizeof(uint16_t)) +
         2 * round256(static_cast<size_t>(Smax) * Rp * Nmax * sizeof(float));
}

size_t loftq_ws_bytes(int64_t d, int64_t k);  // LoftQ workspace (defined with the LoftQ loop)

// fp32-compute layer: the adapter projection (M x r fp32).
size_t f32_ws_bytes(int64_t M, int32_t r) { return kSemBytes + round256(static_cast<size_t>(M) * r * sizeof(float)); }

size_t bwd_ws_bytes(int64_t M, int64_t d, int64_t k, int32_t r) {
  return kSemBytes + round256(static_cast<size_t>(M) * r * sizeof(float)) + proj_ws_bytes(M, r) +
         qn::tc_bwd_ws_bytes(M, d, k, r);
}


// Single-token forward of a group of projections of one input: one
// persistent kernel (every CTA resident, at least one per SM); its two
// counters live in the zero area.
qn_status launch_decode_group(int n, const qn_nf4 *const *Q, const uint16_t *X, const uint16_t *const *A,
                              const uint16_t *const *B, const int32_t *r, const float *alpha, uint16_t *const *Y,
                              unsigned int *zero_area, Span &sp, cudaStream_t st) {
  const int64_t k = Q[0]->k;
  const size_t smem = qn::dec_smem_bytes(k);
  static int attr_set[64] = {0};
  int dev = 0;
  QN_TRY(cuda_check(cudaGetDevice(&dev), "cudaGetDevice"));
  if (dev < 0 || dev >= 64) return fail(QN_EUNSUPPORTED, "device ordinal out of range");
  if (!attr_set[dev]) {
    QN_TRY(cuda_check(cudaFuncSetAttribute(qn::qlora_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(qn::dec_smem_bytes(qn::kDecMaxK))),
                      "cudaFuncSetAttribute(decode smem)"));
    attr_set[dev] = 1;
  }
  int per_sm = 0;
  QN_TRY(cuda_check(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qn::qlora_decode_kernel, qn::kDecThreads,
                                                                  smem), "occupancy query"));
  if (per_sm < 1) return fail(QN_EUNSUPPORTED, "decode kernel does not fit on an SM");
  qn::DecGroup g = {};
  g.n = n;
  g.k = k;
  g.X = X;
  int64_t units = 0, us = 0;
  for (int i = 0; i < n; ++i) {
    qn::DecProj &p = g.p[i];
    p.q = view_of(Q[i]);
    p.A = A[i];
    p.B = B[i];
    p.Y = Y[i];
    p.r = r[i];
    p.s = alpha[i] / static_cast<float>(r[i]);
    p.unit_off = units;
    p.u_off = us;
    units += qn_ceil_div(Q[i]->d, qn::kDecRows);
    us += r[i];
  }
  g.nunits = units;
  g.nadapter = us;
  const int64_t sms = sm_count();
  int64_t grid = qn_ceil_div(units, qn::kDecWarps);
  if (grid < sms) grid = sms;
  if (grid > sms * per_sm) grid = sms * per_sm;
  float *u = sp.take<float>(static_cast<size_t>(us));
  qn::qlora_decode_kernel<<<static_cast<unsigned>(grid), qn::kDecThreads, smem, st>>>(g, zero_area, u);
  QN_LAUNCH_CHECK("qlora_decode_kernel");
  return QN_OK;
}

// bf16 bits of a finite float, rounded to nearest even (host side).
uint16_t bf16_bits_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof(u));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// Where dynamic shared memory starts for a kernel without static shared
// memory (the few-token kernel addresses its level table with an immediate
// offset from there).  One launch per device, cached.
__global__ void qn_smem_base_probe(unsigned int *out) {
  extern __shared__ __align__(1024) unsigned char probe_smem[];
  if (threadIdx.x == 0) out[0] = static_cast<unsigned int>(__cvta_generic_to_shared(probe_smem));
}

qn_status smem_base_matches(unsigned int *scratch, cudaStream_t st, bool *ok) {
  static int known[64] = {0};  // 1: matches, -1: does not
  int dev = 0;
  QN_TRY(cuda_check(cudaGetDevice(&dev), "cudaGetDevice"));
  if (dev < 0 || dev >= 64) return fail(QN_EUNSUPPORTED, "device ordinal out of range");
  if (!known[dev]) {
    // Inside a stream capture nothing may synchronize: take the path and let
    // the kernel's own check (QN_DEV_LAYOUT) report a mismatch.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    QN_TRY(cuda_check(cudaStreamIsCapturing(st, &cs), "cudaStreamIsCapturing"));
    if (cs != cudaStreamCaptureStatusNone) {
      *ok = true;
      return QN_OK;
    }
    const int bytes = 64 * 1024;
    QN_TRY(cuda_check(cudaFuncSetAttribute(qn_smem_base_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                      "cudaFuncSetAttribute(probe)"));
    unsigned int h = 0;
    qn_smem_base_probe<<<1, 32, bytes, st>>>(scratch);
    QN_LAUNCH_CHECK("qn_smem_base_probe");
    QN_TRY(cuda_check(cudaMemcpyAsync(&h, scratch, sizeof(h), cudaMemcpyDeviceToHost, st), "probe readback"));
    QN_TRY(cuda_check(cudaStreamSynchronize(st), "probe synchronize"));
    known[dev] = (h == qn::kGvSmemBase) ? 1 : -1;
  }
  *ok = known[dev] > 0;
  return QN_OK;
}

// Forward of a group of projections of one input with M <= 8 tokens and
// M * k <= 16384 (qlora_gemv_kernel), launched as a programmatic dependent of
// the kernel before it.  Sets *taken to false, launching nothing, when the
// group exceeds that kernel's limits or its pointers are not 16-byte aligned.
qn_status launch_gemv_group(int n, const qn_nf4 *const *Q, const uint16_t *X, int64_t M, const uint16_t *const *A,
                            const uint16_t *const *B, const int32_t *r, const float *alpha, uint16_t *const *Y,
                            unsigned int *zero_area, Span &sp, cudaStream_t st, bool *taken) {
  *taken = false;
  const int64_t k = Q[0]->k;
  if (M < 1 || M > qn::kGvMaxM || n > qn::kGvMaxGroup || !aligned(X, 16)) return QN_OK;
  qn::GvGroup g = {};
  g.n = n;
  g.M = static_cast<int>(M);
  g.k = k;
  g.X = X;
  g.zero_area = zero_area;
  int64_t rows = 0, us = 0;
  for (int i = 0; i < n; ++i) {
    qn::GvProj &p = g.p[i];
    p.codes = Q[i]->codes;
    p.dq = Q[i]->dq ? 1 : 0;
    p.consts = p.dq ? static_cast<const void *>(Q[i]->absmax_q) : static_cast<const void *>(Q[i]->absmax);
    p.absmax_scale = Q[i]->absmax_scale;
    p.absmax_mean = Q[i]->absmax_mean;
    p.A = A[i];
    p.B = B[i];
    p.Y = Y[i];
    p.d = Q[i]->d;
    p.r = r[i];
    p.s = alpha[i] / static_cast<float>(r[i]);
    p.row_off = rows;
    p.u_off = us;
    if (!aligned(p.codes, 16) || !aligned(p.consts, 16) || !aligned(p.A, 16) || !aligned(p.B, 16) ||
        (p.dq && !aligned(p.absmax_scale, 16)))
      return QN_OK;
    rows += Q[i]->d;
    us += r[i];
  }
  g.rows = rows;
  g.rtot = us;
  for (int i = 0; i < 16; ++i) g.lev16[i] = bf16_bits_rne(kNF4Levels[i]);
  const int grid = static_cast<int>(sm_count());
  if (!qn::gv_plan(g, grid)) return QN_OK;
  g.u = sp.take<float>(static_cast<size_t>(M) * us);
  bool base_ok = false;  // the u buffer is scratch for the one-time probe
  QN_TRY(smem_base_matches(reinterpret_cast<unsigned int *>(g.u), st, &base_ok));
  if (!base_ok) return QN_OK;
  const int mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;
  void (*kern)(qn::GvGroup) = mt == 1 ? qn::qlora_gemv_kernel<1>
                              : mt == 2 ? qn::qlora_gemv_kernel<2>
                              : mt == 4 ? qn::qlora_gemv_kernel<4>
                                        : qn::qlora_gemv_kernel<8>;
  static int attr_set[64][4] = {};
  int dev = 0;
  QN_TRY(cuda_check(cudaGetDevice(&dev), "cudaGetDevice"));
  if (dev < 0 || dev >= 64) return fail(QN_EUNSUPPORTED, "device ordinal out of range");
  const int vi = mt == 1 ? 0 : mt == 2 ? 1 : mt == 4 ? 2 : 3;
  if (!attr_set[dev][vi]) {
    QN_TRY(cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(qn::kGvSmemCap)),
                      "cudaFuncSetAttribute(few-token forward smem)"));
    QN_TRY(cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100),
                      "cudaFuncSetAttribute(few-token forward carveout)"));
    cudaFuncAttributes fa;
    QN_TRY(cuda_check(cudaFuncGetAttributes(&fa, kern), "cudaFuncGetAttributes"));
    attr_set[dev][vi] = fa.maxThreadsPerBlock >= qn::kGvThreads ? 1 : -1;
  }
  if (attr_set[dev][vi] < 0) return QN_OK;
  *taken = true;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(qn::kGvThreads), g.smem, st,
                    "qlora_gemv_kernel", g);
}

template <int MT, bool XS>
qn_status launch_skinny_variant(const qn::SkGroup &g, size_t smem, cudaStream_t st) {
  auto kern = qn::skinny_kernel<MT, XS>;
  static int attr_set[64] = {0};
  int dev = 0;
  QN_TRY(cuda_check(cudaGetDevice(&dev), "cudaGetDevice"));
  if (dev < 0 || dev >= 64) return fail(QN_EUNSUPPORTED, "device ordinal out of range");
  if (!attr_set[dev]) {
    QN_TRY(cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024),
                      "cudaFuncSetAttribute(skinny smem)"));
    attr_set[dev] = 1;
  }
  int64_t grid = sm_count();
  if (grid > g.ngroups) grid = g.ngroups;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(qn::kSkThreads), smem, st, "skinny_kernel", g);
}

// Forward of a group of projections of one input with M <= 16 tokens: the
// adapter down-projection u, then the weights (both kernels PDL-launched).
qn_status launch_skinny_group(int n, const qn_nf4 *const *Q, const uint16_t *X, int64_t M,
                              const uint16_t *const *A, const uint16_t *const *B, const int32_t *r,
                              const float *alpha, uint16_t *const *Y, Span &sp, cudaStream_t st) {
  const int64_t k = Q[0]->k;
  qn::SkGroup g = {};
  g.n = n;
  g.M = static_cast<int>(M);
  g.k = k;
  g.X = X;
  int64_t groups = 0, us = 0;
  for (int i = 0; i < n; ++i) {
    qn::SkProj &p = g.p[i];
    p.q = view_of(Q[i]);
    p.A = A[i];
    p.B = B[i];
    p.Y = Y[i];
    p.r = r[i];
    p.s = alpha[i] / static_cast<float>(r[i]);
    p.group_off = groups;
    p.u_off = us;
    // codes as uint32 [d][k / 8]: one box = 16 rows x 128 bytes (4 blocks)
    if (const char *e = qn::make_tile_map(&p.tmap, Q[i]->codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4,
                                          static_cast<uint64_t>(k / 8), static_cast<uint64_t>(Q[i]->d),
                                          qn::kSkBoxBytes / 4, qn::kSkRows, CU_TENSOR_MAP_SWIZZLE_128B))
      return fail(QN_ECUDA, "few-token forward: %s", e);
    groups += qn_ceil_div(Q[i]->d, qn::kSkRows);
    us += r[i];
  }
  if (groups > (int64_t{1} << 30)) return fail(QN_ESHAPE, "too many rows for the few-token kernel");
  g.ngroups = groups;
  g.rtot = us;
  g.u = sp.take<float>(static_cast<size_t>(M) * us);
  QN_TRY(launch_pdl(qn::skinny_u_kernel, dim3(static_cast<unsigned>(us), static_cast<unsigned>(M)),
                    dim3(qn::kSkUThreads), 0, st, "skinny_u_kernel", g));
  const int MT = M <= 8 ? 1 : 2;
  const bool xs = qn::sk_smem_bytes(MT, g.M, k, true) <= 227 * 1024;
  const size_t smem = qn::sk_smem_bytes(MT, g.M, k, xs);
  if (MT == 1) return xs ? launch_skinny_variant<1, true>(g, smem, st) : launch_skinny_variant<1, false>(g, smem, st);
  return xs ? launch_skinny_variant<2, true>(g, smem, st) : launch_skinny_variant<2, false>(g, smem, st);
}

// Forward of a group of projections of one input with 8 < M <= 16 tokens on
// the K-slice kernel: the adapter down-projection u (skinny_u_kernel), then
// the weights (qlora_m16_kernel), both PDL-launched.  `taken` is false (and
// nothing is launched) when the shapes or alignments do not suit it: k a
// multiple of 256, the int8 block constants 4-byte aligned.
qn_status launch_m16_group(int n, const qn_nf4 *const *Q, const uint16_t *X, int64_t M, const uint16_t *const *A,
                           const uint16_t *const *B, const int32_t *r, const float *alpha, uint16_t *const *Y,
                           Span &sp, cudaStream_t st, bool *taken) {
  *taken = false;
  const int64_t k = Q[0]->k;
  if (M <= 8 || M > 16 || (k % 256) != 0) return QN_OK;
  for (int i = 0; i < n; ++i)
    if (Q[i]->dq && !aligned(Q[i]->absmax_q, 4)) return QN_OK;
  qn::SkGroup g = {};
  g.n = n;
  g.M = static_cast<int>(M);
  g.k = k;
  g.X = X;
  int64_t tiles = 0, us = 0;
  for (int i = 0; i < n; ++i) {
    qn::SkProj &p = g.p[i];
    p.q = view_of(Q[i]);
    p.A = A[i];
    p.B = B[i];
    p.Y = Y[i];
    p.r = r[i];
    p.s = alpha[i] / static_cast<float>(r[i]);
    p.group_off = tiles;
    p.u_off = us;
    tiles += qn_ceil_div(Q[i]->d, 16);
    us += r[i];
  }
  if (tiles > (int64_t{1} << 30)) return QN_OK;
  g.ngroups = tiles;
  g.rtot = us;
  g.u = sp.take<float>(static_cast<size_t>(M) * us);
  QN_TRY(launch_pdl(qn::skinny_u_kernel, dim3(static_cast<unsigned>(us), static_cast<unsigned>(M)),
                    dim3(qn::kSkUThreads), 0, st, "skinny_u_kernel", g));
  QN_TRY(cuda_check(cudaFuncSetAttribute(qn::qlora_m16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(qn::kM16SmemBytes)),
                    "cudaFuncSetAttribute(m16 smem)"));
  int64_t grid = sm_count();
  if (grid > tiles) grid = tiles;
  QN_TRY(launch_pdl(qn::qlora_m16_kernel, dim3(static_cast<unsigned>(grid)), dim3(qn::kM16Threads),
                    qn::kM16SmemBytes, st, "qlora_m16_kernel", g));
  *taken = true;
  return QN_OK;
}

qn_status check_layer(const qn_nf4 *Q, const void *in, int64_t M, const void *A, const void *B, int32_t r,
                      float alpha, const void *out) {
  QN_TRY(check_nf4(Q, true));
  if (Q->k % 64) return fail(QN_ESHAPE, "k must be a multiple of 64 (got %lld)", (long long)Q->k);
  if (M < 1) return fail(QN_ESHAPE, "M must be >= 1");
  if (r < 1 || r > 256) return fail(QN_ESHAPE, "r must be in [1, 256] (got %d)", r);
  if (!std::isfinite(alpha)) return fail(QN_EINVAL, "alpha must be finite");
  if (!in || !A || !B || !out) return fail(QN_EINVAL, "NULL tensor pointer");
  if (!aligned(in, 16) || !aligned(A, 16) || !aligned(B, 16) || !aligned(out, 16))
    return fail(QN_EALIGN, "tensor pointers must be 16-byte aligned");
  return QN_OK;
}

// A second stream per device and calling thread, for side kernels that are
// independent of the caller's stream work until a join: fork records an
// event on `st` that the side stream waits for; join makes `st` wait for
// everything issued on the side stream since.  Both are plain event
// dependencies, so the pattern is also valid inside a stream capture.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

qn_status side_stream(SideStream **out) {
  thread_local SideStream tab[64];
  int dev = 0;
  QN_TRY(cuda_check(cudaGetDevice(&dev), "cudaGetDevice"));
  if (dev < 0 || dev >= 64) return fail(QN_EUNSUPPORTED, "device ordinal out of range");
  SideStream &ss = tab[dev];
  if (!ss.s) {
    QN_TRY(cuda_check(cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking), "side stream"));
    QN_TRY(cuda_check(cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming), "side stream event"));
    QN_TRY(cuda_check(cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming), "side stream event"));
  }
  *out = &ss;
  return QN_OK;
}

qn_status side_fork(SideStream *ss, cudaStream_t st) {
  QN_TRY(cuda_check(cudaEventRecord(ss->fork, st), "fork record"));
  return cuda_check(cudaStreamWaitEvent(ss->s, ss->fork, 0), "fork wait");
}

qn_status side_join(SideStream *ss, cudaStream_t st) {
  QN_TRY(cuda_check(cudaEventRecord(ss->join, ss->s), "join record"));
  return cuda_check(cudaStreamWaitEvent(st, ss->join, 0), "join wait");
}

// Adapter projection C = s P Qop^T (M x N, K deep) split over K so that
// enough CTAs to fill the SMs run, then the splits summed in order into C32 (fp32)
// or, with C2 set, its bf16 hi/lo split (each half padded to R columns, rows
// of pitch ld2 >= 2R, zero past 2R).
qn_status launch_lora_proj(const uint16_t *P, int64_t M, int64_t K, const uint16_t *Qm, int64_t N, int64_t qs_n,
                           int64_t qs_k, float s, float *part, float *C32, int R, uint16_t *C2, int64_t ld2,
                           cudaStream_t st) {
  const int TN = N <= 16 ? 16 : 64;
  const int64_t tiles = qn_ceil_div(M, qn::kProjTM) * qn_ceil_div(N, TN);
  // 16-byte aligned operands take the pipelined kernel (about four CTAs per
  // SM, one wave); others the plain one.
  const bool pal = (K % 8) == 0 && aligned(P, 16) && aligned(Qm, 16);
  const bool q_rows = pal && qs_k == 1 && (qs_n % 8) == 0;                 // Qop contiguous along kk
  const bool q_cols = pal && qs_n == 1 && (qs_k % 8) == 0 && (N % 8) == 0;  // Qop contiguous along n
  const bool pipe = q_rows || q_cols;
  // one wave: the pipelined kernel holds four CTAs per SM
  int64_t S = pipe ? (4 * static_cast<int64_t>(sm_count())) / tiles
                   : qn_ceil_div(6 * static_cast<int64_t>(sm_count()), tiles);
  const int64_t smax = qn_ceil_div(K, 256);
  if (S > smax) S = smax;
  if (S > qn::kProjMaxSplit) S = qn::kProjMaxSplit;
  if (S < 1) S = 1;
  const int64_t kchunk = qn_ceil_div(qn_ceil_div(K, S), qn::kProjTK) * qn::kProjTK;
  S = qn_ceil_div(K, kchunk);
  dim3 grid(static_cast<unsigned>(qn_ceil_div(M, qn::kProjTM)), static_cast<unsigned>(qn_ceil_div(N, TN)),
            static_cast<unsigned>(S));
  if (pipe) {
    auto run = [&](auto kern, int smem) -> qn_status {
      QN_TRY(cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                        "cudaFuncSetAttribute(lora_proj_pipe smem)"));
      kern<<<grid, 128, smem, st>>>(P, M, K, Qm, N, qs_n, qs_k, s, kchunk, part);
      return QN_OK;
    };
    if (TN == 16 && q_rows) QN_TRY(run(qn::lora_proj_pipe_kernel<16, false>, qn::proj_pipe_smem<16, false>()));
    else if (TN == 16) QN_TRY(run(qn::lora_proj_pipe_kernel<16, true>, qn::proj_pipe_smem<16, true>()));
    else if (q_rows) QN_TRY(run(qn::lora_proj_pipe_kernel<64, false>, qn::proj_pipe_smem<64, false>()));
    else QN_TRY(run(qn::lora_proj_pipe_kernel<64, true>, qn::proj_pipe_smem<64, true>()));
  } else if (TN == 16) {
    qn::lora_proj_kernel<16><<<grid, 128, 0, st>>>(P, M, K, Qm, N, qs_n, qs_k, s, kchunk, part);
  } else {
    qn::lora_proj_kernel<64><<<grid, 128, 0, st>>>(P, M, K, Qm, N, qs_n, qs_k, s, kchunk, part);
  }
  QN_LAUNCH_CHECK("lora_proj_kernel");
  const int64_t n = M * (C2 ? R : N);
  if ((N % 4) == 0 && (R % 4) == 0 && (ld2 % 4) == 0 && aligned(C32, 16) && aligned(C2, 8)) {
    qn::lora_reduce4_kernel<<<static_cast<unsigned>(qn_ceil_div(n / 4, 256)), 256, 0, st>>>(
        part, static_cast<int>(S), M, N, C32, R, C2, ld2);
    QN_LAUNCH_CHECK("lora_reduce4_kernel");
    return QN_OK;
  }
  qn::lora_reduce_kernel<<<static_cast<unsigned>(qn_ceil_div(n, 256)), 256, 0, st>>>(part, static_cast<int>(S), M, N,
                                                                                      C32, R, C2, ld2);
  QN_LAUNCH_CHECK("lora_reduce_kernel");
  return QN_OK;
}

// Large-M backward dX on the tensor cores: W^T dequantised into the
// workspace and the adapter row operand AT2 packed, then one CTA per 128
// columns of W x 256 tokens (qlora_bwd_tc_kernel); v2 is the bf16 hi/lo split
// of v = s dY B in the U2 layout of the forward.
qn_status launch_tc_bwd(const qn_nf4 *Q, const uint16_t *dY, int64_t M, const uint16_t *v2, const uint16_t *A,
                        int32_t r, uint16_t *dX, Span &sp, cudaStream_t st, SideStream *side) {
  const int64_t d = Q->d, k = Q->k;
  const int64_t ldw = qn::tb_ldw(d);
  uint16_t *wt = sp.take<uint16_t>(static_cast<size_t>(ldw) * k);
  uint16_t *at2 = sp.take<uint16_t>(static_cast<size_t>(k) * qn::kTfUCols);
  {
    int64_t grid = (k / 64) * qn_ceil_div(d, 64);
    if (grid > static_cast<int64_t>(sm_count()) * 8) grid = static_cast<int64_t>(sm_count()) * 8;
    qn::nf4_dequant_t_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(view_of(Q), ldw, wt);
    QN_LAUNCH_CHECK("nf4_dequant_t_kernel");
    // AT2 on the side stream (when there is one), next to the adapter projection
    qn::lora_pack_at2_kernel<<<static_cast<unsigned>(qn_ceil_div(k * qn::kTfUCols, 256)), 256, 0,
                               side ? side->s : st>>>(A, r, k, at2);
    QN_LAUNCH_CHECK("lora_pack_at2_kernel");
  }
  CUtensorMap amap, bmap, atmap, vmap;
  if (const char *e = qn::make_tile_map(&amap, wt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(d),
                                        static_cast<uint64_t>(k), 64, qn::kTcBN, CU_TENSOR_MAP_SWIZZLE_128B,
                                        static_cast<uint64_t>(ldw) * 2))
    return fail(QN_ECUDA, "tcgen05 backward: %s", e);
  if (const char *e = qn::make_bf16_tile_map(&bmap, dY, static_cast<uint64_t>(d), static_cast<uint64_t>(M), qn::kTcBM))
    return fail(QN_ECUDA, "tcgen05 backward: %s", e);
  if (const char *e = qn::make_bf16_tile_map(&atmap, at2, static_cast<uint64_t>(qn::kTfUCols), static_cast<uint64_t>(k),
                                             qn::kTcBN))
    return fail(QN_ECUDA, "tcgen05 backward: %s", e);
  if (const char *e = qn::make_bf16_tile_map(&vmap, v2, static_cast<uint64_t>(qn::kTfUCols), static_cast<uint64_t>(M),
                                             qn::kTcBM))
    return fail(QN_ECUDA, "tcgen05 backward: %s", e);
  QN_TRY(cuda_check(cudaFuncSetAttribute(qn::qlora_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(qn::kTbSmemBytes)),
                    "tcgen05 backward shared-memory limit"));
  if (side) QN_TRY(side_join(side, st));  // v2 and AT2 come from the side stream
  dim3 grid(static_cast<unsigned>(qn_ceil_div(k, qn::kTcBN)), static_cast<unsigned>(qn_ceil_div(M, qn::kTcBM)));
  qn::qlora_bwd_tc_kernel<<<grid, qn::kTbThreads, qn::kTbSmemBytes, st>>>(amap, bmap, atmap, vmap, M, d, k, dX);
  QN_LAUNCH_CHECK("qlora_bwd_tc_kernel");
  return QN_OK;
}

// Large-M forward on the tensor cores: the block constants of W into the
// workspace (nf4_block_scale_kernel), then one CTA per 128 weight rows x 256
// tokens (qlora_fwd_tc_kernel); u2 is the bf16 hi/lo split of u = s X A^T,
// rows [hi | lo] of kTfUCols columns, each half zero-padded to 64.
qn_status launch_tc_fwd(const qn_nf4 *Q, const uint16_t *X, int64_t M, const uint16_t *u2, const uint16_t *B,
                        int32_t r, uint16_t *Y, Span &sp, cudaStream_t st, SideStream *side) {
  const int64_t d = Q->d, k = Q->k, kp = qn::tf_scale_pitch(k);
  float *scales = sp.take<float>(static_cast<size_t>(d) * kp);
  qn::nf4_block_scale_kernel<<<static_cast<unsigned>(qn_ceil_div(d * kp, 256)), 256, 0, st>>>(view_of(Q), kp, scales);
  QN_LAUNCH_CHECK("nf4_block_scale_kernel");
  CUtensorMap xmap, umap;
  if (const char *e = qn::make_bf16_tile_map(&xmap, X, static_cast<uint64_t>(k), static_cast<uint64_t>(M), qn::kTcBM))
    return fail(QN_ECUDA, "tcgen05 forward: %s", e);
  if (const char *e = qn::make_bf16_tile_map(&umap, u2, static_cast<uint64_t>(qn::kTfUCols), static_cast<uint64_t>(M),
                                             qn::kTcBM))
    return fail(QN_ECUDA, "tcgen05 forward: %s", e);
  QN_TRY(cuda_check(cudaFuncSetAttribute(qn::qlora_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(qn::kTfSmemBytes)),
                    "tcgen05 forward shared-memory limit"));
  if (side) QN_TRY(side_join(side, st));  // u2 comes from the side stream
  dim3 grid(static_cast<unsigned>(qn_ceil_div(d, qn::kTcBN)), static_cast<unsigned>(qn_ceil_div(M, qn::kTcBM)));
  qn::qlora_fwd_tc_kernel<<<grid, qn::kTfThreads, qn::kTfSmemBytes, st>>>(
      xmap, umap, static_cast<const uint8_t *>(Q->codes), scales, d, k, M, B, r, Y);
  QN_LAUNCH_CHECK("qlora_fwd_tc_kernel");
  return QN_OK;
}

// C = scale * P1 Op1 (+ P2 Op2) on the fp32 CUDA-core GEMM (qlora_f32.cuh).
qn_status launch_f32_gemm(const qn::F32Gemm &gp, cudaStream_t st) {
  const unsigned gx = static_cast<unsigned>(qn_ceil_div(gp.N, qn::kF32BN));
  if (gp.M <= 16) {
    qn::f32_gemm_kernel<16><<<dim3(gx, static_cast<unsigned>(qn_ceil_div(gp.M, 16))), qn::kF32Threads, 0, st>>>(gp);
  } else {
    qn::f32_gemm_kernel<64><<<dim3(gx, static_cast<unsigned>(qn_ceil_div(gp.M, 64))), qn::kF32Threads, 0, st>>>(gp);
  }
  QN_LAUNCH_CHECK("f32_gemm_kernel");
  return QN_OK;
}

qn::F32Operand f32_mat(const float *F, int64_t sn, int64_t sk) {
  qn::F32Operand o = {};
  o.kind = qn::F32_OP_MAT;
  o.F = F;
  o.sn = sn;
  o.sk = sk;
  return o;
}
qn::F32Operand f32_nf4(const qn_nf4 *Q, bool cols) {
  qn::F32Operand o = {};
  o.kind = cols ? qn::F32_OP_NF4_COLS : qn::F32_OP_NF4_ROWS;
  o.q = view_of(Q);
  return o;
}

// Token contraction C[q, n] = sum_m V[m, q] P[m, n] of the adapter gradients
// (lora_grad.cuh), written as C (transpose_out = 0) or C^T.
qn_status launch_lora_grad(const uint16_t *P, int64_t M, int64_t N, const uint16_t *vt2, int32_t r, float *part,
                           int transpose_out, float *out, cudaStream_t st) {
  const int64_t Rp = qn::lg_rp(r), Mp = qn::lg_round(M, qn::kLgTK);
  const int rch = qn::lg_rch(r);
  const int S = qn::lg_splits(M, N, r);
  const int64_t tps = qn::lg_round(qn_ceil_div(M, S), qn::kLgTK);
  const int Sused = static_cast<int>(qn_ceil_div(M, tps));
  dim3 grid(static_cast<unsigned>(qn_ceil_div(N, qn::kLgTN)), static_cast<unsigned>(Sused),
            static_cast<unsigned>(Rp / rch));
  switch (rch / 16) {
    case 1: qn::lora_grad_kernel<1><<<grid, qn::kLgThreads, 0, st>>>(P, M, N, vt2, Rp, Mp, tps, part); break;
    case 2: qn::lora_grad_kernel<2><<<grid, qn::kLgThreads, 0, st>>>(P, M, N, vt2, Rp, Mp, tps, part); break;
    case 3: qn::lora_grad_kernel<3><<<grid, qn::kLgThreads, 0, st>>>(P, M, N, vt2, Rp, Mp, tps, part); break;
    default: qn::lora_grad_kernel<4><<<grid, qn::kLgThreads, 0, st>>>(P, M, N, vt2, Rp, Mp, tps, part); break;
  }
  QN_LAUNCH_CHECK("lora_grad_kernel");
  qn::lora_grad_reduce_kernel<<<static_cast<unsigned>(qn_ceil_div(static_cast<int64_t>(r) * N, 256)), 256, 0, st>>>(
      part, Sused, Rp, N, r, transpose_out, out);
  QN_LAUNCH_CHECK("lora_grad_reduce_kernel");
  return QN_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// Scratch for nf4_quantize_noalloc.  Some callers cannot call cudaMalloc:
// code that runs while another allocator owns all free device memory (a
// framework's pre-reserved pool), or a latency-bound loop that must not pay
// the implicit device-wide synchronisation of an allocation.  For them the
// exponent bins and the ticket word the quantiser needs (2 KiB + 256 B) live
// in this file-scope device array.  Every GPU that loads the library holds it until the process exits.
// In host code the name is only a host-side stand-in: the device address is
// obtained once per device with cudaGetSymbolAddress and passed to the kernels.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned long long g_noalloc_bins[qn::kNumBins + 32];  // bins, then a ticket word

namespace {

constexpr int kNoallocMaxDevices = 64;
// Largest tensor nf4_quantize_noalloc accepts: 2^40 elements keeps every
// 64-bit bin of the fixed scratch exact (at most 2^34 block constants,
// each adding a significand below 2^24).
constexpr int64_t kNoallocMaxElements = int64_t(1) << 40;
std::mutex g_noalloc_mutex;
unsigned long long *g_noalloc_dev_ptr[kNoallocMaxDevices] = {};

// Device address of g_noalloc_bins on the current device; looked up on the
// first call per device.
qn_status noalloc_bins(unsigned long long **out) {
  int dev = 0;
  QN_TRY(cuda_check(cudaGetDevice(&dev), "cudaGetDevice"));
  if (dev < 0 || dev >= kNoallocMaxDevices) return fail(QN_EUNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_dev_ptr[dev]) {
    void *p = nullptr;
    QN_TRY(cuda_check(cudaGetSymbolAddress(&p, g_noalloc_bins), "cudaGetSymbolAddress(scratch)"));
    g_noalloc_dev_ptr[dev] = static_cast<unsigned long long *>(p);
  }
  *out = g_noalloc_dev_ptr[dev];
  return QN_OK;
}

}  // namespace

extern "C" {

int qn_abi_version(void) { return QN_ABI_VERSION; }

const char *qn_last_error(void) { return g_last_error.c_str(); }

void qn_nf4_tables(float codebook[16], float thresholds[15]) {
  if (codebook) std::memcpy(codebook, kNF4Levels, sizeof(kNF4Levels));
  if (thresholds) std::memcpy(thresholds, kNF4Thresholds, sizeof(kNF4Thresholds));
}

size_t qn_workspace_bytes(qn_op op, int64_t M, int64_t d, int64_t k, int32_t r) {
  switch (op) {
    case QN_OP_QUANTIZE: return kQuantWs;
    case QN_OP_DEQUANTIZE: return 0;
    case QN_OP_LINEAR_FWD: return (M < 1 || d < 1 || k < 1 || r < 1) ? 0 : fwd_ws_bytes(M, d, k, r);
    case QN_OP_LINEAR_BWD_DX: return (M < 1 || d < 1 || k < 1 || r < 1) ? 0 : bwd_ws_bytes(M, d, k, r);
    case QN_OP_LINEAR_BWD_LORA: return (M < 1 || d < 1 || k < 1 || r < 1) ? 0 : lg_ws_bytes(M, d, k, r);
    case QN_OP_LINEAR_F32: return (M < 1 || r < 1) ? 0 : f32_ws_bytes(M, r);
    case QN_OP_MERGE: return kQuantWs;
    case QN_OP_LOFTQ: return (d < 1 || k < 1) ? 0 : loftq_ws_bytes(d, k);
  }
  return 0;
}

qn_status nf4_quantize(const void *W, qn_dtype wdt, const qn_nf4 *Q, void *ws, size_t ws_bytes, void *stream) {
  g_last_error.clear();
  if (!tables_consistent()) return fail(QN_EUNSUPPORTED, "internal NF4 tables inconsistent");
  QN_TRY(check_nf4(Q, true));
  if (!W) return fail(QN_EINVAL, "W is NULL");
  if (wdt != QN_F32 && wdt != QN_BF16) return fail(QN_EINVAL, "bad input dtype %d", (int)wdt);
  if (!aligned(W, 16)) return fail(QN_EALIGN, "W not 16-byte aligned");
  if (Q->dq) {
    if (!ws) return fail(QN_EINVAL, "workspace NULL");
    if (ws_bytes < kQuantWs) return fail(QN_ENOMEM, "workspace %zu < %zu bytes", ws_bytes, kQuantWs);
    if (!aligned(ws, 16)) return fail(QN_EALIGN, "workspace not 16-byte aligned");
  }
  return launch_quantize(W, wdt, Q, reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kBinsOffset),
                         static_cast<unsigned int *>(ws), static_cast<cudaStream_t>(stream));
}

qn_status nf4_dequantize(const qn_nf4 *Q, void *Wout, qn_dtype odt, void *stream) {
  g_last_error.clear();
  QN_TRY(check_nf4(Q, true));
  if (!Wout) return fail(QN_EINVAL, "Wout is NULL");
  if (odt != QN_F32 && odt != QN_BF16) return fail(QN_EINVAL, "bad output dtype %d", (int)odt);
  if (!aligned(Wout, 16)) return fail(QN_EALIGN, "Wout not 16-byte aligned");
  return launch_dequantize(Q, Wout, odt, static_cast<cudaStream_t>(stream));
}

qn_status qlora_linear_fwd(const qn_nf4 *Q, const uint16_t *X, int64_t M, const uint16_t *A, const uint16_t *B,
                           int32_t r, float alpha, uint16_t *Y, void *ws, size_t ws_bytes, void *stream) {
  g_last_error.clear();
  QN_TRY(check_layer(Q, X, M, A, B, r, alpha, Y));
  const int64_t d = Q->d, k = Q->k;
  const size_t need = fwd_ws_bytes(M, d, k, r);
  if (!ws) return fail(QN_EINVAL, "workspace NULL");
  if (ws_bytes < need) return fail(QN_ENOMEM, "workspace %zu < %zu bytes", ws_bytes, need);
  if (!aligned(ws, 256)) return fail(QN_EALIGN, "workspace not 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Span sp{static_cast<char *>(ws), ws_bytes, 0};
  unsigned int *sem = sp.take<unsigned int>(kSemBytes / sizeof(unsigned int));
  const float s = alpha / static_cast<float>(r);
  if (use_skinny(M, k)) {
    bool taken = false;
    QN_TRY(launch_gemv_group(1, &Q, X, M, &A, &B, &r, &alpha, &Y, sem, sp, st, &taken));
    if (taken) return QN_OK;
  }
  if (use_decode(M, k)) return launch_decode_group(1, &Q, X, &A, &B, &r, &alpha, &Y, sem, sp, st);
  if (use_skinny(M, k)) {
    bool taken = false;
    QN_TRY(launch_m16_group(1, &Q, X, M, &A, &B, &r, &alpha, &Y, sp, st, &taken));
    if (taken) return QN_OK;
    return launch_skinny_group(1, &Q, X, M, &A, &B, &r, &alpha, &Y, sp, st);
  }
  float *u = sp.take<float>(static_cast<size_t>(M) * r);
  float *part = sp.take<float>(static_cast<size_t>(qn::kProjMaxSplit) * M * r);
  if (qn::tc_supported(M, d, k, r)) {
    uint16_t *u2 = sp.take<uint16_t>(static_cast<size_t>(M) * qn::kTfUCols);
    // u2 on the side stream while the block constants are formed on st
    SideStream *side = nullptr;
    QN_TRY(side_stream(&side));
    QN_TRY(side_fork(side, st));
    QN_TRY(launch_lora_proj(X, M, k, A, r, k, 1, s, part, nullptr, qn::kTfUCols / 2, u2, qn::kTfUCols, side->s));
    return launch_tc_fwd(Q, X, M, u2, B, r, Y, sp, st, side);
  }
  QN_TRY(launch_lora_proj(X, M, k, A, r, k, 1, s, part, u, 0, nullptr, 0, st));
  dim3 grid(static_cast<unsigned>(qn_ceil_div(d, qn::kTileN)), static_cast<unsigned>(qn_ceil_div(M, qn::kTileM)));
  qn::qlora_gemm_simt_kernel<false><<<grid, 256, 0, st>>>(view_of(Q), X, M, u, B, r, Y);
  QN_LAUNCH_CHECK("qlora_gemm_simt_kernel<fwd>");
  return QN_OK;
}

qn_status qlora_linear_fwd_group(int32_t n, const qn_nf4 *const *Q, const uint16_t *X, int64_t M,
                                 const uint16_t *const *A, const uint16_t *const *B, const int32_t *r,
                                 const float *alpha, uint16_t *const *Y, void *ws, size_t ws_bytes, void *stream) {
  g_last_error.clear();
  if (n < 1 || n > qn::kSkMaxGroup || n > qn::kDecMaxGroup) return fail(QN_ESHAPE, "group size must be in [1, %d]", qn::kSkMaxGroup);
  if (!Q || !A || !B || !r || !alpha || !Y) return fail(QN_EINVAL, "NULL array");
  int64_t dsum = 0, rsum = 0;
  for (int i = 0; i < n; ++i) {
    QN_TRY(check_layer(Q[i], X, M, A[i], B[i], r[i], alpha[i], Y[i]));
    if (Q[i]->k != Q[0]->k) return fail(QN_ESHAPE, "all projections of a group share k");
    dsum += Q[i]->d;
    rsum += r[i];
  }
  const int64_t k = Q[0]->k;
  const size_t need = qn_workspace_bytes(QN_OP_LINEAR_FWD, M, dsum, k, static_cast<int32_t>(rsum));
  if (!ws) return fail(QN_EINVAL, "workspace NULL");
  if (ws_bytes < need) return fail(QN_ENOMEM, "workspace %zu < %zu bytes", ws_bytes, need);
  if (!aligned(ws, 256)) return fail(QN_EALIGN, "workspace not 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (use_decode(M, k) || use_skinny(M, k)) {
    Span sp{static_cast<char *>(ws), ws_bytes, 0};
    unsigned int *sem = sp.take<unsigned int>(kSemBytes / sizeof(unsigned int));
    bool taken = false;
    QN_TRY(launch_gemv_group(n, Q, X, M, A, B, r, alpha, Y, sem, sp, st, &taken));
    if (taken) return QN_OK;
    if (use_decode(M, k)) return launch_decode_group(n, Q, X, A, B, r, alpha, Y, sem, sp, st);
    QN_TRY(launch_m16_group(n, Q, X, M, A, B, r, alpha, Y, sp, st, &taken));
    if (taken) return QN_OK;
    return launch_skinny_group(n, Q, X, M, A, B, r, alpha, Y, sp, st);
  }
  for (int i = 0; i < n; ++i)
    QN_TRY(qlora_linear_fwd(Q[i], X, M, A[i], B[i], r[i], alpha[i], Y[i], ws, ws_bytes, stream));
  return QN_OK;
}

qn_status qlora_linear_bwd_dx(const qn_nf4 *Q, const uint16_t *dY, int64_t M, const uint16_t *A, const uint16_t *B,
                              int32_t r, float alpha, uint16_t *dX, void *ws, size_t ws_bytes, void *stream) {
  g_last_error.clear();
  QN_TRY(check_layer(Q, dY, M, A, B, r, alpha, dX));
  const int64_t d = Q->d, k = Q->k;
  const size_t need = bwd_ws_bytes(M, d, k, r);
  if (!ws) return fail(QN_EINVAL, "workspace NULL");
  if (ws_bytes < need) return fail(QN_ENOMEM, "workspace %zu < %zu bytes", ws_bytes, need);
  if (!aligned(ws, 256)) return fail(QN_EALIGN, "workspace not 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Span sp{static_cast<char *>(ws), ws_bytes, 0};
  (void)sp.take<unsigned int>(kSemBytes / sizeof(unsigned int));
  const float s = alpha / static_cast<float>(r);
  float *v = sp.take<float>(static_cast<size_t>(M) * r);
  float *part = sp.take<float>(static_cast<size_t>(qn::kProjMaxSplit) * M * r);
  // v[m, q] = s * sum_i dY[m, i] B[i, q]: Qop(n = q, kk = i) = B[i * r + q].
  if (qn::tc_bwd_supported(M, d, k, r)) {
    uint16_t *v2 = sp.take<uint16_t>(static_cast<size_t>(M) * qn::kTfUCols);
    // v2 on the side stream while W^T and AT2 are formed on st
    SideStream *side = nullptr;
    QN_TRY(side_stream(&side));
    QN_TRY(side_fork(side, st));
    QN_TRY(launch_lora_proj(dY, M, d, B, r, 1, r, s, part, nullptr, qn::kTfUCols / 2, v2, qn::kTfUCols, side->s));
    return launch_tc_bwd(Q, dY, M, v2, A, r, dX, sp, st, side);
  }
  QN_TRY(launch_lora_proj(dY, M, d, B, r, 1, r, s, part, v, 0, nullptr, 0, st));
  dim3 grid(static_cast<unsigned>(qn_ceil_div(k, qn::kTileN)), static_cast<unsigned>(qn_ceil_div(M, qn::kTileM)));
  qn::qlora_gemm_simt_kernel<true><<<grid, 256, 0, st>>>(view_of(Q), dY, M, v, A, r, dX);
  QN_LAUNCH_CHECK("qlora_gemm_simt_kernel<bwd>");
  return QN_OK;
}

qn_status qlora_linear_bwd_lora(const uint16_t *X, const uint16_t *dY, int64_t M, int64_t d, int64_t k,
                                const uint16_t *A, const uint16_t *B, int32_t r, float alpha, float *dA, float *dB,
                                void *ws, size_t ws_bytes, void *stream) {
  g_last_error.clear();
  if (!X || !dY || !A || !B || !dA || !dB) return fail(QN_EINVAL, "NULL tensor pointer");
  if (M < 1 || d < 1 || k < 1) return fail(QN_ESHAPE, "M, d and k must be positive");
  if (d > (int64_t(1) << 40) / k || M > (int64_t(1) << 40) / (d > k ? d : k)) return fail(QN_ESHAPE, "sizes too large");
  if (r < 1 || r > 256) return fail(QN_ESHAPE, "r must be in [1, 256] (got %d)", r);
  if (!std::isfinite(alpha)) return fail(QN_EINVAL, "alpha must be finite");
  if (!aligned(X, 16) || !aligned(dY, 16) || !aligned(A, 16) || !aligned(B, 16) || !aligned(dA, 16) ||
      !aligned(dB, 16))
    return fail(QN_EALIGN, "tensor pointers must be 16-byte aligned");
  const size_t need = lg_ws_bytes(M, d, k, r);
  if (!ws) return fail(QN_EINVAL, "workspace NULL");
  if (ws_bytes < need) return fail(QN_ENOMEM, "workspace %zu < %zu bytes", ws_bytes, need);
  if (!aligned(ws, 256)) return fail(QN_EALIGN, "workspace not 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Span sp{static_cast<char *>(ws), ws_bytes, 0};
  (void)sp.take<unsigned int>(kSemBytes / sizeof(unsigned int));
  const float s = alpha / static_cast<float>(r);
  float *u = sp.take<float>(static_cast<size_t>(M) * r);
  float *v = sp.take<float>(static_cast<size_t>(M) * r);
  float *part_u = sp.take<float>(static_cast<size_t>(qn::kProjMaxSplit) * M * r);
  float *part_v = sp.take<float>(static_cast<size_t>(qn::kProjMaxSplit) * M * r);
  const int64_t Rp = qn::lg_rp(r), Mp = qn::lg_round(M, qn::kLgTK);
  uint16_t *ut2 = sp.take<uint16_t>(static_cast<size_t>(2) * Rp * Mp);
  uint16_t *vt2 = sp.take<uint16_t>(static_cast<size_t>(2) * Rp * Mp);
  const int Sd = qn::lg_splits(M, d, r), Sk = qn::lg_splits(M, k, r);
  const size_t gpart_n = std::max(static_cast<size_t>(Sd) * Rp * d, static_cast<size_t>(Sk) * Rp * k);
  float *gpart_u = sp.take<float>(gpart_n);
  float *gpart_v = sp.take<float>(gpart_n);
  const unsigned pg = static_cast<unsigned>(qn_ceil_div(Rp * Mp, 256));
  // Two independent chains, the first on a side stream:
  //   u = s X A^T (Qop(n = q, kk = j) = A[q * k + j]);  dB^T[q, i] = sum_m u[m, q] dY[m, i]  (written as dB, d x r)
  //   v = s dY B (Qop(n = q, kk = i) = B[i * r + q]);   dA[q, j] = sum_m v[m, q] X[m, j]
  SideStream *side = nullptr;
  QN_TRY(side_stream(&side));
  QN_TRY(side_fork(side, st));
  QN_TRY(launch_lora_proj(X, M, k, A, r, k, 1, s, part_u, u, 0, nullptr, 0, side->s));
  qn::lora_vt_pack_kernel<<<pg, 256, 0, side->s>>>(u, M, r, Rp, Mp, ut2);
  QN_LAUNCH_CHECK("lora_vt_pack_kernel(u)");
  QN_TRY(launch_lora_grad(dY, M, d, ut2, r, gpart_u, 1, dB, side->s));
  QN_TRY(launch_lora_proj(dY, M, d, B, r, 1, r, s, part_v, v, 0, nullptr, 0, st));
  qn::lora_vt_pack_kernel<<<pg, 256, 0, st>>>(v, M, r, Rp, Mp, vt2);
  QN_LAUNCH_CHECK("lora_vt_pack_kernel(v)");
  QN_TRY(launch_lora_grad(X, M, k, vt2, r, gpart_v, 0, dA, st));
  return side_join(side, st);
}

qn_status qlora_linear_fwd_f32(const qn_nf4 *Q, const float *X, int64_t M, const float *A, const float *B, int32_t r,
                               float alpha, float *Y, void *ws, size_t ws_bytes, void *stream) {
  g_last_error.clear();
  QN_TRY(check_layer(Q, X, M, A, B, r, alpha, Y));
  const int64_t d = Q->d, k = Q->k;
  const size_t need = f32_ws_bytes(M, r);
  if (!ws) return fail(QN_EINVAL, "workspace NULL");
  if (ws_bytes < need) return fail(QN_ENOMEM, "workspace %zu < %zu bytes", ws_bytes, need);
  if (!aligned(ws, 256)) return fail(QN_EALIGN, "workspace not 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Span sp{static_cast<char *>(ws), ws_bytes, 0};
  (void)sp.take<unsigned int>(kSemBytes / sizeof(unsigned int));
  float *u = sp.take<float>(static_cast<size_t>(M) * r);
  const float s = alpha / static_cast<float>(r);
  qn::F32Gemm g1 = {};  // u = s X A^T: Op(kk = j, n = q) = A[q * k + j]
  g1.P1 = X; g1.K1 = k; g1.op1 = f32_mat(A, k, 1); g1.M = M; g1.N = r; g1.scale = s; g1.C = u;
  QN_TRY(launch_f32_gemm(g1, st));
  qn::F32Gemm g2 = {};  // Y = X W'^T + u B^T: Op1(kk = j, n) = W'[n, j], Op2(kk = q, n) = B[n * r + q]
  g2.P1 = X; g2.K1 = k; g2.op1 = f32_nf4(Q, false);
  g2.P2 = u; g2.K2 = r; g2.op2 = f32_mat(B, r, 1);
  g2.M = M; g2.N = d; g2.scale = 1.f; g2.C = Y;
  return launch_f32_gemm(g2, st);
}

qn_status qlora_linear_bwd_dx_f32(const qn_nf4 *Q, const float *dY, int64_t M, const float *A, const float *B,
                                  int32_t r, float alpha, float *dX, void *ws, size_t ws_bytes, void *stream) {
  g_last_error.clear();
  QN_TRY(check_layer(Q, dY, M, A, B, r, alpha, dX));
  const int64_t d = Q->d, k = Q->k;
  const size_t need = f32_ws_bytes(M, r);
  if (!ws) return fail(QN_EINVAL, "workspace NULL");
  if (ws_bytes < need) return fail(QN_ENOMEM, "workspace %zu < %zu bytes", ws_bytes, need);
  if (!aligned(ws, 256)) return fail(QN_EALIGN, "workspace not 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Span sp{static_cast<char *>(ws), ws_bytes, 0};
  (void)sp.take<unsigned int>(kSemBytes / sizeof(unsigned int));
  float *v = sp.take<float>(static_cast<size_t>(M) * r);
  const float s = alpha / static_cast<float>(r);
  qn::F32Gemm g1 = {};  // v = s dY B: Op(kk = i, n = q) = B[i * r + q]
  g1.P1 = dY; g1.K1 = d; g1.op1 = f32_mat(B, 1, r); g1.M = M; g1.N = r; g1.scale = s; g1.C = v;
  QN_TRY(launch_f32_gemm(g1, st));
  qn::F32Gemm g2 = {};  // dX = dY W' + v A: Op1(kk = i, n = c) = W'[i, c], Op2(kk = q, n = c) = A[q * k + c]
  g2.P1 = dY; g2.K1 = d; g2.op1 = f32_nf4(Q, true);
  g2.P2 = v; g2.K2 = r; g2.op2 = f32_mat(A, 1, k);
  g2.M = M; g2.N = k; g2.scale = 1.f; g2.C = dX;
  return launch_f32_gemm(g2, st);
}

qn_status nf4_quantize_noalloc(const void *W, qn_dtype wdt, const qn_nf4 *Q, void *stream) {
  g_last_error.clear();
  if (!tables_consistent()) return fail(QN_EUNSUPPORTED, "internal NF4 tables inconsistent");
  QN_TRY(check_nf4(Q, true));
  if (!W) return fail(QN_EINVAL, "W is NULL");
  if (wdt != QN_F32 && wdt != QN_BF16) return fail(QN_EINVAL, "bad input dtype %d", (int)wdt);
  if (!aligned(W, 16)) return fail(QN_EALIGN, "W not 16-byte aligned");
  if (Q->d * Q->k > kNoallocMaxElements)
    return fail(QN_ESHAPE, "nf4_quantize_noalloc: %lld elements exceed the maximum of 2^40 its static scratch covers",
                (long long)(Q->d * Q->k));
  unsigned long long *bins = nullptr;
  QN_TRY(noalloc_bins(&bins));
  unsigned int *ticket = reinterpret_cast<unsigned int *>(bins + qn::kNumBins);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // bins and ticket start from zero on every call (the kernels also leave them zero)
  QN_TRY(cuda_check(cudaMemsetAsync(bins, 0, (qn::kNumBins + 32) * sizeof(unsigned long long), st),
                    "clear scratch"));
  return launch_quantize(W, wdt, Q, bins, ticket, st);
}

qn_status qn_device_status(void *stream) {
  g_last_error.clear();
  QN_TRY(cuda_check(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream synchronize"));
  unsigned int h = 0, zero = 0;
  QN_TRY(cuda_check(cudaMemcpyFromSymbol(&h, g_qn_status, sizeof(h)), "read status word"));
  QN_TRY(cuda_check(cudaMemcpyToSymbol(g_qn_status, &zero, sizeof(zero)), "clear status word"));
  if (h & QN_DEV_TIMEOUT) return fail(QN_ETIMEOUT, "a bounded device wait expired");
  if (h & QN_DEV_LAYOUT) return fail(QN_EUNSUPPORTED, "a kernel found its shared memory at an unexpected address");
  return QN_OK;
}

}  // extern "C"

namespace {

// K splits of the two panel products: about four CTAs per SM, at least four
// 32-wide chunks of K per split.
int lq_splits(int64_t out_rows, int64_t kdim) {
  const int64_t tiles = qn_ceil_div(out_rows, qn::kLqTile);
  int64_t S = qn_ceil_div(4 * static_cast<int64_t>(sm_count()), tiles);
  const int64_t smax = kdim / (4 * qn::kLqTile);
  if (S > smax) S = smax;
  if (S > 16) S = 16;
  return S < 1 ? 1 : static_cast<int>(S);
}

// LoftQ workspace: the d x k residual, the panels Y (d x P), Zt and Omega
// (k x P), the split partials of the products, the Gram partials and the
// small P x P factors.
size_t loftq_ws_bytes(int64_t d, int64_t k) {
  const size_t P = qn::kLqMaxP;
  const size_t nb = static_cast<size_t>(qn_ceil_div(d > k ? d : k, qn::kLqGramRows));
  const size_t prt = std::max(static_cast<size_t>(lq_splits(d, k)) * d, static_cast<size_t>(lq_splits(k, d)) * k);
  size_t b = kSemBytes + round256(static_cast<size_t>(d) * k * sizeof(float));  // target / residual
  b += round256(static_cast<size_t>(d) * P * sizeof(float));                  // Y
  b += 2 * round256(static_cast<size_t>(k) * P * sizeof(float));              // Zt, Omega
  b += round256(prt * P * sizeof(float));                                     // product split partials
  b += round256(nb * P * P * sizeof(float));                                  // Gram partials
  b += round256(P * P * sizeof(double)) + 2 * round256(P * P * sizeof(float)) + round256(P * sizeof(float));
  b += round256(1024 * sizeof(double)) + round256(65 * sizeof(double));       // norm partials, T + 1 norms
  b += round256(kQuantWs);
  return b;
}

// The LoftQ loop on panels of P columns (r + oversample <= P).  requantise:
// Q_0 = NF4(W) and T alternations (loftq_init); otherwise Q is the caller's
// quantised weight, kept as it is, and one Delta-step is taken against it
// (loftq_replace_lora, T == 1).
template <int P>
qn_status loftq_run_p(const float *W, int64_t d, int64_t k, int32_t r, float alpha, int32_t T, uint64_t seed, int p,
                      int32_t power_iters, const qn_nf4 *Q, float *A, float *B, double *resid, void *ws,
                      size_t ws_bytes, cudaStream_t st, bool requantise) {
  Span sp{static_cast<char *>(ws), ws_bytes, 0};
  unsigned int *sem = sp.take<unsigned int>(kSemBytes / sizeof(unsigned int));  // zero on entry and exit
  float *Tbuf = sp.take<float>(static_cast<size_t>(d) * k);
  float *Y = sp.take<float>(static_cast<size_t>(d) * qn::kLqMaxP);
  float *Zt = sp.take<float>(static_cast<size_t>(k) * qn::kLqMaxP);
  float *Om = sp.take<float>(static_cast<size_t>(k) * qn::kLqMaxP);
  const int Srz = lq_splits(d, k), Srty = lq_splits(k, d);
  float *ppart = sp.take<float>(std::max(static_cast<size_t>(Srz) * d, static_cast<size_t>(Srty) * k) * qn::kLqMaxP);
  const int64_t nbmax = qn_ceil_div(d > k ? d : k, qn::kLqGramRows);
  float *gpart = sp.take<float>(static_cast<size_t>(nbmax) * qn::kLqMaxP * qn::kLqMaxP);
  double *G = sp.take<double>(qn::kLqMaxP * qn::kLqMaxP);
  float *V = sp.take<float>(qn::kLqMaxP * qn::kLqMaxP);
  float *Lf = sp.take<float>(qn::kLqMaxP * qn::kLqMaxP);
  float *lam = sp.take<float>(qn::kLqMaxP);
  double *partial = sp.take<double>(1024);
  double *norm2 = sp.take<double>(65);  // squared residual norms, copied to the host once at the end
  unsigned long long *bins = reinterpret_cast<unsigned long long *>(reinterpret_cast<char *>(sem) + kBinsOffset);

  const float s = alpha / static_cast<float>(r);
  const int sms = sm_count();
  const int64_t n = d * k;
  const QnNF4View qv = view_of(Q);
  const int red_blocks = sms * 4 < 1024 ? sms * 4 : 1024;
  static int attr_set[64] = {0};
  int dev = 0;
  QN_TRY(cuda_check(cudaGetDevice(&dev), "cudaGetDevice"));
  if (dev < 0 || dev >= 64) return fail(QN_EUNSUPPORTED, "device ordinal out of range");
  if (!attr_set[dev]) {
    QN_TRY(cuda_check(cudaFuncSetAttribute(qn::lq_jacobi_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(qn::lq_jacobi_smem<P>())),
                      "cudaFuncSetAttribute(jacobi smem)"));
    attr_set[dev] = 1;
  }

  QN_TRY(cuda_check(cudaMemsetAsync(A, 0, sizeof(float) * r * k, st), "memset A"));
  QN_TRY(cuda_check(cudaMemsetAsync(B, 0, sizeof(float) * d * r, st), "memset B"));

  auto residual_norm = [&](int rr, int t) -> qn_status {  // norm2[t] = ||R - s B A||^2
    qn::resid_norm_kernel<<<red_blocks, 256, 0, st>>>(Tbuf, B, A, d, k, rr, s, partial);
    QN_LAUNCH_CHECK("resid_norm_kernel");
    qn::sum_partials_kernel<<<1, 256, 0, st>>>(partial, red_blocks, norm2 + t);
    QN_LAUNCH_CHECK("sum_partials_kernel");
    return QN_OK;
  };
  auto gram = [&](const float *Ym, int64_t rows) -> qn_status {  // G = Ym^T Ym (fp64)
    const int nb = static_cast<int>(qn_ceil_div(rows, qn::kLqGramRows));
    qn::lq_gram_part_kernel<P><<<nb, 256, 0, st>>>(Ym, rows, gpart);
    QN_LAUNCH_CHECK("lq_gram_part_kernel");
    qn::lq_gram_reduce_kernel<P><<<static_cast<unsigned>(qn_ceil_div(P * P * 32, 256)), 256, 0, st>>>(gpart, nb, G);
    QN_LAUNCH_CHECK("lq_gram_reduce_kernel");
    return QN_OK;
  };
  // P == 32: CholeskyQR2 in one cooperative launch; the panel is Ym itself
  // (S == 0) or the sum of the S split partials in ppart, written to Ym.
  auto cholqr2_32 = [&](const float *parts, int S, float *Ym, int64_t rows) -> qn_status {
    int64_t grid = qn_ceil_div(rows, 32);
    if (grid > sms) grid = sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    QN_TRY(cuda_check(cudaLaunchKernelEx(&cfg, qn::lq_cholqr2_p32_kernel, parts, S, Ym, rows, p,
                                         reinterpret_cast<double *>(gpart), G, sem + kLqBarWord),
                      "lq_cholqr2_p32_kernel"));
    QN_LAUNCH_CHECK("lq_cholqr2_p32_kernel");
    return QN_OK;
  };
  auto orth = [&](float *Ym, int64_t rows) -> qn_status {  // CholeskyQR2: Ym <- Ym L^{-T}, twice
    if constexpr (P == 32) {
      return cholqr2_32(nullptr, 0, Ym, rows);
    } else {
      for (int rep = 0; rep < 2; ++rep) {
        QN_TRY(gram(Ym, rows));
        qn::lq_chol_kernel<P><<<1, 256, 0, st>>>(G, p, Lf);
        QN_LAUNCH_CHECK("lq_chol_kernel");
        qn::lq_trsm_rows_kernel<P><<<static_cast<unsigned>(qn_ceil_div(rows, 128)), 128, 0, st>>>(Ym, rows, Lf, p);
        QN_LAUNCH_CHECK("lq_trsm_rows_kernel");
      }
      return QN_OK;
    }
  };
  auto reduce = [&](int S, int64_t n_out, float *out) -> qn_status {
    qn::lq_split_reduce_kernel<<<static_cast<unsigned>(qn_ceil_div(n_out, 256)), 256, 0, st>>>(ppart, S, n_out, out);
    QN_LAUNCH_CHECK("lq_split_reduce_kernel");
    return QN_OK;
  };
  // Splits of the register-tiled 32-column products: about three CTAs per
  // SM, within what the partial buffer holds.
  const size_t ppart_floats = std::max(static_cast<size_t>(Srz) * d, static_cast<size_t>(Srty) * k) * qn::kLqMaxP;
  auto big_splits = [&](int64_t out_rows, int64_t kdim, int occ) -> int64_t {  // one wave of occ CTAs per SM
    int64_t S = (static_cast<int64_t>(occ) * sms) / qn_ceil_div(out_rows, qn::kLqBig);
    if (S > 16) S = 16;
    if (S > kdim / 64) S = kdim / 64;
    const int64_t cap = static_cast<int64_t>(ppart_floats / (static_cast<size_t>(out_rows) * 32));
    if (S > cap) S = cap;
    return S < 1 ? 1 : S;
  };
  // P == 32: the register-tiled product into the split partials; returns the
  // number of splits.  right: R Z (d rows, K = k); otherwise R^T Y (k rows).
  auto prod32 = [&](bool right, const float *in, int *S_out) -> qn_status {
    const int64_t rows = right ? d : k, kdim = right ? k : d;
    constexpr int smem_rz = qn::kLqPipe * qn::kLqRzStage, smem_rty = qn::kLqPipe * qn::kLqRtyStage;
    int occ = 1;
    if (right) {
      QN_TRY(cuda_check(cudaFuncSetAttribute(qn::lq_rz32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_rz),
                        "cudaFuncSetAttribute(rz smem)"));
      QN_TRY(cuda_check(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, qn::lq_rz32_kernel, 256, smem_rz),
                        "rz occupancy"));
    } else {
      QN_TRY(cuda_check(
          cudaFuncSetAttribute(qn::lq_rty32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_rty),
          "cudaFuncSetAttribute(rty smem)"));
      QN_TRY(cuda_check(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, qn::lq_rty32_kernel, 256, smem_rty),
                        "rty occupancy"));
    }
    const int64_t per = qn_ceil_div(qn_ceil_div(kdim, big_splits(rows, kdim, occ < 1 ? 1 : occ)), qn::kLqTile) *
                        qn::kLqTile;
    const int S = static_cast<int>(qn_ceil_div(kdim, per));
    const dim3 grid(static_cast<unsigned>(qn_ceil_div(rows, qn::kLqBig)), static_cast<unsigned>(S));
    if (right) {
      qn::lq_rz32_kernel<<<grid, 256, smem_rz, st>>>(Tbuf, d, k, in, per, ppart);
      QN_LAUNCH_CHECK("lq_rz32_kernel");
    } else {
      qn::lq_rty32_kernel<<<grid, 256, smem_rty, st>>>(Tbuf, d, k, in, per, ppart);
      QN_LAUNCH_CHECK("lq_rty32_kernel");
    }
    *S_out = S;
    return QN_OK;
  };
  auto r_times = [&](const float *Z, float *Yo) -> qn_status {  // Yo = R Z   (d x P)
    if constexpr (P == 32) {
      int S = 1;
      QN_TRY(prod32(true, Z, &S));
      return reduce(S, d * P, Yo);
    }
    const int64_t cps = qn_ceil_div(qn_ceil_div(k, Srz), qn::kLqTile) * qn::kLqTile;
    const int S = static_cast<int>(qn_ceil_div(k, cps));
    qn::lq_rz_kernel<P><<<dim3(static_cast<unsigned>(qn_ceil_div(d, qn::kLqTile)), static_cast<unsigned>(S)), 256, 0,
                         st>>>(Tbuf, d, k, Z, cps, ppart);
    QN_LAUNCH_CHECK("lq_rz_kernel");
    return reduce(S, d * P, Yo);
  };
  auto rt_times = [&](const float *Ym, float *Zo) -> qn_status {  // Zo = R^T Y  (k x P)
    if constexpr (P == 32) {
      int S = 1;
      QN_TRY(prod32(false, Ym, &S));
      return reduce(S, k * P, Zo);
    }
    const int64_t rps = qn_ceil_div(qn_ceil_div(d, Srty), qn::kLqTile) * qn::kLqTile;
    const int S = static_cast<int>(qn_ceil_div(d, rps));
    qn::lq_rty_kernel<P><<<dim3(static_cast<unsigned>(k / qn::kLqTile), static_cast<unsigned>(S)), 256, 0, st>>>(
        Tbuf, d, k, Ym, rps, ppart);
    QN_LAUNCH_CHECK("lq_rty_kernel");
    return reduce(S, k * P, Zo);
  };
  // P == 32: out = orthonormalised (R Z or R^T Y); the split partials are
  // summed inside the CholeskyQR2 launch.
  auto prod_orth32 = [&](bool right, const float *in, float *out) -> qn_status {
    int S = 1;
    QN_TRY(prod32(right, in, &S));
    return cholqr2_32(ppart, S, out, right ? d : k);
  };

  // t = 0: Q_0 = NF4(W) (or the caller's Q), residual without adapter.
  if (requantise) QN_TRY(launch_quantize(W, QN_F32, Q, bins, sem, st));
  qn::residual_kernel<<<sms * 8, 256, 0, st>>>(qv, W, Tbuf, n);
  QN_LAUNCH_CHECK("residual_kernel");
  QN_TRY(residual_norm(0, 0));

  for (int t = 1; t <= T; ++t) {
    if (t > 1) {  // Q-step: Q_t = NF4(W - s B A)
      qn::lowrank_sub_kernel<<<sms * 8, 256, 0, st>>>(W, B, A, d, k, r, s, Tbuf);
      QN_LAUNCH_CHECK("lowrank_sub_kernel");
      QN_TRY(launch_quantize(Tbuf, QN_F32, Q, bins, sem, st));
      qn::residual_kernel<<<sms * 8, 256, 0, st>>>(qv, W, Tbuf, n);
      QN_LAUNCH_CHECK("residual_kernel");
    }
    // Delta-step on R = W - deq(Q_t) (in Tbuf).
    qn::omega_kernel<<<static_cast<unsigned>(qn_ceil_div(k * P, 256)), 256, 0, st>>>(
        Om, k, p, P, seed ^ (0x9E3779B97F4A7C15ull * static_cast<uint64_t>(t)));
    QN_LAUNCH_CHECK("omega_kernel");
    if constexpr (P == 32) {
      QN_TRY(prod_orth32(true, Om, Y));
      for (int it = 0; it < power_iters; ++it) {
        QN_TRY(prod_orth32(false, Y, Zt));
        QN_TRY(prod_orth32(true, Zt, Y));
      }
    } else {
      QN_TRY(r_times(Om, Y));
      QN_TRY(orth(Y, d));
      for (int it = 0; it < power_iters; ++it) {
        QN_TRY(rt_times(Y, Zt));
        QN_TRY(orth(Zt, k));
        QN_TRY(r_times(Zt, Y));
        QN_TRY(orth(Y, d));
      }
    }
    QN_TRY(rt_times(Y, Zt));  // Zt = R^T Y, i.e. (Y^T R)^T
    QN_TRY(gram(Zt, k));
    qn::lq_jacobi_kernel<P><<<1, qn::kLqJacThreads, qn::lq_jacobi_smem<P>(), st>>>(G, p, lam, V);
    QN_LAUNCH_CHECK("lq_jacobi_kernel");
    qn::lq_project_kernel<P><<<static_cast<unsigned>(qn_ceil_div(d, 256)), 256, 0, st>>>(Y, d, V, lam, r, s, 0, B, 0);
    QN_LAUNCH_CHECK("lq_project_kernel(B)");
    qn::lq_project_kernel<P><<<static_cast<unsigned>(qn_ceil_div(k, 256)), 256, 0, st>>>(Zt, k, V, lam, r, s, 1, A,
                                                                                         1);
    QN_LAUNCH_CHECK("lq_project_kernel(A)");
    QN_TRY(residual_norm(r, t));
  }
  QN_TRY(cuda_check(cudaMemcpyAsync(resid, norm2, sizeof(double) * (T + 1), cudaMemcpyDeviceToHost, st),
                    "copy norms"));
  QN_TRY(cuda_check(cudaStreamSynchronize(st), "synchronize"));
  for (int t = 0; t <= T; ++t) resid[t] = std::sqrt(resid[t]);
  return QN_OK;
}

qn_status loftq_run(const float *W, int64_t d, int64_t k, int32_t r, float alpha, int32_t T, uint64_t seed,
                    int32_t oversample, int32_t power_iters, const qn_nf4 *Q, float *A, float *B, double *resid,
                    void *ws, size_t ws_bytes, void *stream, bool requantise) {
  if (!W || !A || !B || !resid || !Q) return fail(QN_EINVAL, "NULL pointer");
  QN_TRY(check_nf4(Q, true));
  if (Q->d != d || Q->k != k) return fail(QN_ESHAPE, "Q shape %lldx%lld != W shape", (long long)Q->d, (long long)Q->k);
  if (d % 64 || k % 64) return fail(QN_ESHAPE, "d and k must be multiples of 64");
  const int p = r + oversample;
  if (r < 1 || oversample < 0 || p > qn::kLqMaxP)
    return fail(QN_ESHAPE, "need 1 <= r and r + oversample <= %d", qn::kLqMaxP);
  if (p > d || p > k) return fail(QN_ESHAPE, "r + oversample exceeds a matrix dimension");
  if (T < 0 || T > 64) return fail(QN_ESHAPE, "T must be in [0, 64]");
  if (power_iters < 0 || power_iters > 32) return fail(QN_ESHAPE, "power_iters must be in [0, 32]");
  if (!std::isfinite(alpha) || alpha == 0.f) return fail(QN_EINVAL, "alpha must be finite and non-zero");
  if (!aligned(W, 16) || !aligned(A, 16) || !aligned(B, 16)) return fail(QN_EALIGN, "W/A/B not 16-byte aligned");
  const size_t need = loftq_ws_bytes(d, k);
  if (!ws) return fail(QN_EINVAL, "workspace NULL");
  if (ws_bytes < need) return fail(QN_ENOMEM, "workspace %zu < %zu bytes", ws_bytes, need);
  if (!aligned(ws, 256)) return fail(QN_EALIGN, "workspace not 256-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p <= 32) return loftq_run_p<32>(W, d, k, r, alpha, T, seed, p, power_iters, Q, A, B, resid, ws, ws_bytes, st, requantise);
  if (p <= 64) return loftq_run_p<64>(W, d, k, r, alpha, T, seed, p, power_iters, Q, A, B, resid, ws, ws_bytes, st, requantise);
  return loftq_run_p<96>(W, d, k, r, alpha, T, seed, p, power_iters, Q, A, B, resid, ws, ws_bytes, st, requantise);
}

}  // namespace

extern "C" {

qn_status loftq_init(const float *W, int64_t d, int64_t k, int32_t r, float alpha, int32_t T, uint64_t seed,
                     int32_t oversample, int32_t power_iters, const qn_nf4 *Q, float *A, float *B, double *resid,
                     void *ws, size_t ws_bytes, void *stream) {
  g_last_error.clear();
  return loftq_run(W, d, k, r, alpha, T, seed, oversample, power_iters, Q, A, B, resid, ws, ws_bytes, stream, true);
}

qn_status loftq_replace_lora(const float *W, const qn_nf4 *Q, int32_t r, float alpha, uint64_t seed,
                             int32_t oversample, int32_t power_iters, float *A, float *B, double *resid,
                             void *ws, size_t ws_bytes, void *stream) {
  g_last_error.clear();
  if (!Q) return fail(QN_EINVAL, "Q is NULL");
  return loftq_run(W, Q->d, Q->k, r, alpha, 1, seed, oversample, power_iters, Q, A, B, resid, ws, ws_bytes, stream,
                   false);
}

qn_status nf4_merge_lora(const qn_nf4 *Q, const uint16_t *A, const uint16_t *B, int32_t r, float alpha, int32_t sign,
                         const qn_nf4 *Qout, void *ws, size_t ws_bytes, void *stream) {
  g_last_error.clear();
  if (!tables_consistent()) return fail(QN_EUNSUPPORTED, "internal NF4 tables inconsistent");
  QN_TRY(check_nf4(Q, true));
  QN_TRY(check_nf4(Qout, true));
  if (Qout->d != Q->d || Qout->k != Q->k) return fail(QN_ESHAPE, "Qout shape differs from Q");
  if (Q->k % 64) return fail(QN_ESHAPE, "k must be a multiple of 64 (got %lld)", (long long)Q->k);
  if (r < 1 || r > 256) return fail(QN_ESHAPE, "r must be in [1, 256] (got %d)", r);
  if (sign != 1 && sign != -1) return fail(QN_EINVAL, "sign must be +1 (merge) or -1 (unmerge)");
  if (!std::isfinite(alpha)) return fail(QN_EINVAL, "alpha must be finite");
  if (!A || !B) return fail(QN_EINVAL, "NULL adapter pointer");
  if (!aligned(A, 16) || !aligned(B, 16)) return fail(QN_EALIGN, "A/B not 16-byte aligned");
  if (Qout->dq) {
    if (!ws) return fail(QN_EINVAL, "workspace NULL");
    if (ws_bytes < kQuantWs) return fail(QN_ENOMEM, "workspace %zu < %zu bytes", ws_bytes, kQuantWs);
    if (!aligned(ws, 16)) return fail(QN_EALIGN, "workspace not 16-byte aligned");
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t d = Q->d, k = Q->k, nblk = d * (k >> 6);
  unsigned long long *bins = Qout->dq ? reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kBinsOffset)
                                      : nullptr;
  unsigned int *ticket = static_cast<unsigned int *>(ws);
  static int attr_set[64] = {0};
  int dev = 0;
  QN_TRY(cuda_check(cudaGetDevice(&dev), "cudaGetDevice"));
  if (dev < 0 || dev >= 64) return fail(QN_EUNSUPPORTED, "device ordinal out of range");
  if (!attr_set[dev]) {
    QN_TRY(cuda_check(cudaFuncSetAttribute(qn::nf4_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(qn::kMgSmemBytes)),
                      "cudaFuncSetAttribute(merge smem)"));
    attr_set[dev] = 1;
  }
  const float s = alpha / static_cast<float>(r);
  dim3 grid(static_cast<unsigned>(qn_ceil_div(k, qn::kMgCols)), static_cast<unsigned>(qn_ceil_div(d, qn::kMgRows)));
  qn::nf4_merge_kernel<<<grid, qn::kMgThreads, qn::kMgSmemBytes, st>>>(
      view_of(Q), A, B, r, s, sign, Qout->codes, Qout->absmax, bins, ticket, Qout->absmax_mean);
  QN_LAUNCH_CHECK("nf4_merge_kernel");
  if (Qout->dq) {
    const int64_t ngrp = qn_ceil_div(nblk, 256);
    int64_t g2 = qn_ceil_div(ngrp, qn::kDqWarps);
    const int64_t cap = static_cast<int64_t>(sm_count()) * 4;
    if (g2 > cap) g2 = cap;
    qn::nf4_dq_kernel<<<static_cast<unsigned>(g2), qn::kDqWarps * 32, 0, st>>>(Qout->absmax, nblk, Qout->absmax_mean,
                                                                              Qout->absmax_q, Qout->absmax_scale);
    QN_LAUNCH_CHECK("nf4_dq_kernel");
  }
  return QN_OK;
}

}  // extern "C"
