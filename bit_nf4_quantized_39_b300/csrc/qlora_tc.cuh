// qlora_tc.cuh -- fused QLoRA forward and backward on the 5th-generation
// tensor cores (tcgen05, sm_100 family).
//
// Forward, per output tile of 128 weight rows x 256 tokens (one CTA):
//
//   Y^T tile = sum over K stages of deq(Q) stage . X stage^T  +  [B | B] . U2^T
//
// A stage is 128 columns of K; 320 threads in three roles.
//   warps 0-7  dequantisers, then epilogue.  Warp w owns the 32 weight rows of
//              tensor-memory lane quadrant w % 4 and half w / 4 (64 columns)
//              of every stage: its code bytes and block constant arrive by
//              cp.async two stages ahead (the constants precomputed in fp32 by
//              nf4_block_scale_kernel), it builds the 16 levels scaled by the
//              constant as bf16 (exactly bf16(fp32(c * m')), the value
//              nf4_dequantize writes), selects them with byte permutes and
//              writes the 64 bf16 weights straight into tensor memory with
//              tcgen05.st -- the weight operand never touches shared memory.
//   warp 8     TMA producer: X stages (256 tokens x 128, two 128-byte-swizzled
//              64-column halves) into a 3-stage shared-memory ring.
//   warp 9     allocates tensor memory and issues the MMAs (one thread): A =
//              weights from tensor memory, B = X from shared memory, fp32
//              accumulator in tensor memory.  It waits on one barrier per
//              stage (eight MMAs), which the producer's bytes and all eight
//              dequantiser warps complete together.
// The adapter term is one more stage at the end: the producer loads U2 =
// [hi | lo] (hi = bf16(u), lo = bf16(u - hi), u = s X A^T from
// lora_reduce_kernel, each half zero-padded to 64 columns) in place of X and
// the dequantisers write the row [B | B] (each copy zero-padded to 64) in
// place of weights, so the product keeps about 16 significant bits of u.
//
// Tensor memory: accumulator columns [0, 256), three 64-column weight stages
// at [256, 448).
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace qn {

constexpr int kTcBN = 128;   // weight rows per tile  (MMA M)
constexpr int kTcBM = 256;   // tokens per tile       (MMA N)
constexpr int kTcBK = 64;    // K per stage
constexpr int kTcMaxR = 64;  // largest adapter rank r
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;

// ---- forward ----------------------------------------------------------------
// A stage covers 128 columns of K: two 64-column halves (one 128-byte swizzle
// span each for X), so the MMA issuer waits on one barrier per eight MMAs.
constexpr int kTfBK = 128;
constexpr int kTfStages = 3;                                  // operand ring depth
constexpr int kTfCodeStages = 3;                              // code + constant ring depth (cp.async)
constexpr int kTfDeqWarps = 8;                                // two per weight-row quadrant: one per half stage
constexpr int kTfThreads = (kTfDeqWarps + 2) * 32;            // + TMA producer + MMA issuer
constexpr int kTfProducerWarp = kTfDeqWarps, kTfMmaWarp = kTfDeqWarps + 1;
constexpr uint32_t kTfXHalfBytes = kTcBM * 64 * 2;            // 32 KiB
constexpr uint32_t kTfXStageBytes = 2 * kTfXHalfBytes;        // 64 KiB
// Code ring slot: four 2 KiB chunks (chunk j of row i at j * 2 KiB + i * 16:
// code bytes 16 j .. 16 j + 15 of the row's 64 in this stage), then the two
// block constants of every row (half h of row i at 8 KiB + h * 512 + i * 4).
constexpr uint32_t kTfCodeStageBytes = 4 * 2048 + 2 * kTcBN * 4;  // 9 KiB
constexpr uint32_t kTfACols = kTfBK / 2;                      // tensor-memory columns of a weight stage
constexpr uint32_t kTfACol = 256;                             // weight stages at [256, 256 + 3 * 64)
constexpr int kTfUCols = 128;                                 // U2 row: [hi | 0 .. | lo | 0 ..], 64 + 64
constexpr size_t kTfSmemBytes = 1024 + static_cast<size_t>(kTfStages) * kTfXStageBytes +
                                static_cast<size_t>(kTfCodeStages) * kTfCodeStageBytes + 256;

// Block constants per weight stage: 2 per 128 columns, rows of tf_scale_pitch(k) floats.
__host__ __device__ constexpr int64_t tf_scale_pitch(int64_t k) { return 2 * ((k + kTfBK - 1) / kTfBK); }

// m[n, j] = the effective constant of block j of row n (exact absmax or its
// DQ decode, the value nf4_dequantize uses), zero for the pad slot past k / 64.
__global__ void nf4_block_scale_kernel(QnNF4View q, int64_t kp, float *__restrict__ out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= q.d * kp) return;
  const int64_t n = i / kp, j = i % kp, kb = q.k >> 6;
  out[i] = (j < kb) ? block_scale(q, n * kb + j) : 0.f;
}

struct TfBars {
  uint64_t full[kTfStages], empty[kTfStages];
  uint64_t acc_full, done;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(kTfThreads, 1)
qlora_fwd_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap umap,
                    const uint8_t *__restrict__ codes, const float *__restrict__ scales, int64_t d, int64_t k,
                    int64_t M, const uint16_t *__restrict__ Bm, int r, uint16_t *__restrict__ Y) {
  extern __shared__ __align__(1024) unsigned char tc_smem_raw[];
  unsigned char *base = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char *xring = base;
  unsigned char *cring = xring + kTfStages * kTfXStageBytes;
  TfBars *bars = reinterpret_cast<TfBars *>(cring + kTfCodeStages * kTfCodeStageBytes);
  volatile int *abort = &bars->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kTcBN;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kTcBM;
  const int nk = static_cast<int>((k + kTfBK - 1) / kTfBK);  // weight stages; stage nk is the adapter's

  if (tid == 0) {
    for (int i = 0; i < kTfStages; ++i) {
      mbar_init(smem_u32(&bars->full[i]), 1 + kTfDeqWarps);  // the producer's arrival (+ bytes), one per dequantiser warp
      mbar_init(smem_u32(&bars->empty[i]), 1);
    }
    mbar_init(smem_u32(&bars->acc_full), 1);
    mbar_init(smem_u32(&bars->done), 1);
    bars->abort = 0;
    mbar_fence_init();
  }
  if (warp == kTfMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTfProducerWarp && lane == 0) {
    tma_prefetch_desc(&xmap);
    tma_prefetch_desc(&umap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < kTfDeqWarps) {
    // ======================= dequantisers, then epilogue =======================
    // Warp w owns weight rows 32 (w % 4) .. (tensor-memory lanes of its
    // quadrant) and half h = w / 4 of every stage (columns 64 h .. 64 h + 63).
    const int quad = warp & 3, h = warp >> 2;
    const int row = quad * 32 + lane;
    const int64_t n = n0 + row;
    const bool row_ok = n < d;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int64_t kp = tf_scale_pitch(k);
    const unsigned char *crow = codes + (row_ok ? n : 0) * (k >> 1);
    const float *srow = scales + (row_ok ? n : 0) * kp;
    const uint32_t cbase = smem_u32(cring);
    auto prefetch = [&](int s) {
      if (row_ok && s < nk && static_cast<int64_t>(s) * kTfBK + h * 64 < k) {
        const uint32_t slot = cbase + static_cast<uint32_t>(s % kTfCodeStages) * kTfCodeStageBytes;
        const unsigned char *src = crow + static_cast<int64_t>(s) * (kTfBK / 2) + h * 32;
        cp_async16(slot + (2 * h) * 2048u + row * 16u, src);
        cp_async16(slot + (2 * h + 1) * 2048u + row * 16u, src + 16);
        cp_async4(slot + 8192u + h * 512u + row * 4u, srow + 2 * s + h);
      }
      cp_async_commit();  // one group per stage, empty or not
    };
    for (int s = 0; s < kTfCodeStages - 1; ++s) prefetch(s);
    // This row of B as bf16 pairs (word c = columns 2c, 2c + 1), zero past r.
    uint32_t bw[kTcMaxR / 2];
#pragma unroll
    for (int c = 0; c < kTcMaxR / 2; ++c) {
      uint32_t w = 0;
      if (row_ok && 2 * c < r) {
        w = Bm[n * r + 2 * c];
        if (2 * c + 1 < r) w |= static_cast<uint32_t>(Bm[n * r + 2 * c + 1]) << 16;
      }
      bw[c] = w;
    }

    bool ok = true;
    for (int s = 0; s <= nk; ++s) {
      const uint32_t slot = s % kTfStages;
      if (s >= kTfStages) ok = mbar_wait(smem_u32(&bars->empty[slot]), ((s / kTfStages) - 1) & 1, abort);
      ok = __all_sync(0xffffffffu, ok);  // tcgen05.st is warp-collective: leave together
      if (!ok) break;
      tc_fence_after();
      const uint32_t aaddr = lane_addr + kTfACol + slot * kTfACols + h * 32;
      if (s < nk) {
        cp_async_wait_group<kTfCodeStages - 2>();  // this stage's copies have landed
        const uint32_t cs = cbase + static_cast<uint32_t>(s % kTfCodeStages) * kTfCodeStageBytes;
        uint4 c0, c1;
        float m;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(c0.x), "=r"(c0.y), "=r"(c0.z), "=r"(c0.w) : "r"(cs + (2 * h) * 2048u + row * 16u));
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(c1.x), "=r"(c1.y), "=r"(c1.z), "=r"(c1.w) : "r"(cs + (2 * h + 1) * 2048u + row * 16u));
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(m) : "r"(cs + 8192u + h * 512u + row * 4u));
        prefetch(s + kTfCodeStages - 1);  // refills the slot read one stage ago
        uint32_t v[32];
        if (row_ok && static_cast<int64_t>(s) * kTfBK + h * 64 < k) {
          const ScaledLevels tl = scaled_levels(m);
          decode_word(c0.x, tl, v + 0);
          decode_word(c0.y, tl, v + 4);
          decode_word(c0.z, tl, v + 8);
          decode_word(c0.w, tl, v + 12);
          decode_word(c1.x, tl, v + 16);
          decode_word(c1.y, tl, v + 20);
          decode_word(c1.z, tl, v + 24);
          decode_word(c1.w, tl, v + 28);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = 0u;
        }
        tmem_st_x32(aaddr, v);
      } else {
        // Adapter stage: the row [B | B], each copy zero-padded to 64 columns,
        // against U2 = [hi | lo] padded the same way.
        tmem_st_x32(aaddr, bw);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->full[slot]));
    }
    cp_async_wait_all();  // no copy may still target shared memory at exit

    // Epilogue: accumulator lane = this row, columns = tokens 128 h .. 128 h + 127.
    if (ok) ok = mbar_wait(smem_u32(&bars->acc_full), 0, abort);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < kTcBM / 64; ++c) {
        const int tc0 = h * (kTcBM / 2) + c * 32;
        uint32_t acc[32];
        tmem_ld_x32(lane_addr + kAccCol + tc0, acc);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t t = m0 + tc0 + j;
            if (t < M) Y[t * d + n] = f32_to_bf16_bits(__uint_as_float(acc[j]));
          }
        }
      }
    }
  } else if (warp == kTfProducerWarp) {
    // ================================ TMA producer ================================
    if (lane == 0) {
      int issued = 0;
      for (int s = 0; s <= nk; ++s) {
        const uint32_t slot = s % kTfStages;
        if (s >= kTfStages && !mbar_wait(smem_u32(&bars->empty[slot]), ((s / kTfStages) - 1) & 1, abort)) break;
        const uint32_t full = smem_u32(&bars->full[slot]);
        mbar_arrive_expect_tx(full, kTfXStageBytes);
        const uint32_t dst = smem_u32(xring + slot * kTfXStageBytes);
        const CUtensorMap *map = (s < nk) ? &xmap : &umap;
        const int32_t x0 = (s < nk) ? s * kTfBK : 0;
        tma_load_2d(dst, map, x0, static_cast<int32_t>(m0), full);
        tma_load_2d(dst + kTfXHalfBytes, map, x0 + 64, static_cast<int32_t>(m0), full);
        ++issued;
      }
      // Before the CTA can retire, every copy it started must have landed.
      // (After an abort a stage's barrier may also lack the dequantisers'
      // arrivals; the drain then gives up after its bound, by which time the
      // bytes have long landed.)
      for (int s = (issued > kTfStages ? issued - kTfStages : 0); s < issued; ++s)
        mbar_wait_drain(smem_u32(&bars->full[s % kTfStages]), (s / kTfStages) & 1);
    }
  } else {
    // ================================= MMA issuer =================================
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTcBN, kTcBM);
      const uint32_t d_tmem = tmem + kAccCol;
      bool ok = true;
      for (int s = 0; s <= nk && ok; ++s) {
        const uint32_t slot = s % kTfStages;
        if (!(ok = mbar_wait(smem_u32(&bars->full[slot]), (s / kTfStages) & 1, abort))) break;
        tc_fence_after();
        const uint32_t xbase = smem_u32(xring + slot * kTfXStageBytes);
        const uint32_t abase = tmem + kTfACol + slot * kTfACols;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_tmem_a(d_tmem, abase + hh * 32 + kk * 8,
                          smem_desc(xbase + hh * kTfXHalfBytes + kk * 32, 16, 1024, 2), idesc,
                          (s > 0 || hh > 0 || kk > 0) ? 1u : 0u);
        tc_commit(smem_u32(&bars->empty[slot]));
      }
      if (ok) tc_commit(smem_u32(&bars->acc_full));
      // Every MMA issued must be complete before tensor memory is released.
      tc_commit(smem_u32(&bars->done));
      mbar_wait_drain(smem_u32(&bars->done), 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kTfMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Backward dX = dY deq(Q) + s (dY B) A on the tensor cores, as
//   dX^T tile [128 columns of W x 256 tokens] = W^T tile . dY tile^T + AT2 . V2^T
// with W^T the dequantised weight transposed (bf16, written once per call by
// nf4_dequant_t_kernel) so that both operands stream K-major (K = d) through
// TMA in stages of 128 columns (one barrier per eight MMAs).  The adapter
// term is one more stage at the end: AT2 = [A^T | A^T] and V2 = [bf16(v) |
// bf16(v - bf16(v))], v = s dY B, each half zero-padded to 64 columns.
// Warps: 0-3 epilogue, 4 TMA producer, 5 MMA issuer.
// ---------------------------------------------------------------------------
constexpr int kTbBK = 128;
constexpr int kTbStages = 2;
constexpr int kTbThreads = 192;
constexpr uint32_t kTbAHalfBytes = kTcBN * 64 * 2;                 // 16 KiB
constexpr uint32_t kTbBHalfBytes = kTcBM * 64 * 2;                 // 32 KiB
constexpr uint32_t kTbStageBytes = 2 * (kTbAHalfBytes + kTbBHalfBytes);  // 96 KiB
constexpr size_t kTbSmemBytes = 1024 + static_cast<size_t>(kTbStages) * kTbStageBytes + 256;

struct TbBars {
  uint64_t full[kTbStages], empty[kTbStages];
  uint64_t acc_full, done;
  uint32_t tmem_base;
  int abort;
};

// W^T[c, r] = bf16(level[code(r, c)] * m(r, c / 64)), 64 x 64 tiles of W
// (grid-strided); W^T has row stride ldw (d rounded up to a multiple of 8).
// A thread decodes rows r, r + 1 of W at 8 columns (two 4-byte code words;
// a warp reads 8 rows x 32 contiguous bytes) into 8 words, each the pair
// (W[r][c], W[r+1][c]), of a shared tile T[c][r / 2] (row stride 36 words;
// word column xor 4 * (c / 8 mod 8), so neither these stores nor the 16-byte
// reads below conflict).  Then 8 threads write one 128-byte row of W^T.
constexpr int kDtStride = 36;

__global__ void __launch_bounds__(256) nf4_dequant_t_kernel(QnNF4View q, int64_t ldw, uint16_t *__restrict__ wt) {
  __shared__ float lv[16];
  __shared__ __align__(16) uint32_t tile[64][kDtStride];
  const int tid = threadIdx.x;
  if (tid < 16) lv[tid] = c_nf4_levels[tid];
  __syncthreads();
  const int cg = tid & 7, rp = tid >> 3;  // 8 columns 8 cg .. ; rows 2 rp, 2 rp + 1
  const int64_t tiles_c = (q.k + 63) / 64, tiles = tiles_c * ((q.d + 63) / 64);
  for (int64_t tl = blockIdx.x; tl < tiles; tl += gridDim.x) {
    const int64_t r0 = (tl / tiles_c) * 64, c0 = (tl % tiles_c) * 64;
    uint32_t w[2] = {0u, 0u};
    float m[2] = {0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t row = r0 + 2 * rp + h;
      if (row < q.d && c0 + 8 * cg < q.k) {
        w[h] = __ldg(reinterpret_cast<const uint32_t *>(q.codes + row * (q.k >> 1) + (c0 >> 1)) + cg);
        m[h] = block_scale(q, row * (q.k >> 6) + (c0 >> 6));
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t lo = f32_to_bf16_bits(__fmul_rn(lv[(w[0] >> (4 * j)) & 15u], m[0]));
      const uint32_t hi = f32_to_bf16_bits(__fmul_rn(lv[(w[1] >> (4 * j)) & 15u], m[1]));
      tile[8 * cg + j][rp ^ (4 * cg)] = lo | (hi << 16);
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int ch = tid + 256 * h, oc = ch >> 3, qd = ch & 7;  // row oc of the tile, rows 8 qd .. of W
      const int64_t col = c0 + oc;
      const int64_t rr = r0 + 8 * qd;
      if (col < q.k && rr < q.d) {
        const uint4 v = *reinterpret_cast<const uint4 *>(&tile[oc][(4 * qd) ^ (4 * ((oc >> 3) & 7))]);
        if (rr + 8 <= q.d) {
          *reinterpret_cast<uint4 *>(wt + col * ldw + rr) = v;
        } else {
          const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
          for (int e = 0; e < 8 && rr + e < q.d; ++e)
            wt[col * ldw + rr + e] = static_cast<uint16_t>(vv[e >> 1] >> (16 * (e & 1)));
        }
      }
    }
    __syncthreads();
  }
}

// AT2[c, :] = [A[0 .. 63, c] | A[0 .. 63, c]] (rows of A past r read as zero):
// the adapter stage's row operand, k rows of kTfUCols bf16.
__global__ void lora_pack_at2_kernel(const uint16_t *__restrict__ Am, int r, int64_t k, uint16_t *__restrict__ at2) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= k * kTfUCols) return;
  const int64_t c = i / kTfUCols;
  const int j = static_cast<int>(i % kTfUCols) & 63;
  at2[i] = (j < r) ? Am[static_cast<int64_t>(j) * k + c] : 0;
}

__global__ void __launch_bounds__(kTbThreads, 1)
qlora_bwd_tc_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                    const __grid_constant__ CUtensorMap atmap, const __grid_constant__ CUtensorMap vmap, int64_t M,
                    int64_t d, int64_t k, uint16_t *__restrict__ dX) {
  extern __shared__ __align__(1024) unsigned char tb_smem_raw[];
  unsigned char *base = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(tb_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char *ring = base;  // stage s: A halves (2 x 16 KiB) then B halves (2 x 32 KiB)
  TbBars *bars = reinterpret_cast<TbBars *>(ring + kTbStages * kTbStageBytes);
  volatile int *abort = &bars->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kTcBN;  // columns of W (rows of the MMA)
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kTcBM;  // tokens
  const int nk = static_cast<int>((d + kTbBK - 1) / kTbBK);     // stages over d; stage nk is the adapter's

  if (tid == 0) {
    for (int i = 0; i < kTbStages; ++i) {
      mbar_init(smem_u32(&bars->full[i]), 1);
      mbar_init(smem_u32(&bars->empty[i]), 1);
    }
    mbar_init(smem_u32(&bars->acc_full), 1);
    mbar_init(smem_u32(&bars->done), 1);
    bars->abort = 0;
    mbar_fence_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&amap);
    tma_prefetch_desc(&bmap);
    tma_prefetch_desc(&atmap);
    tma_prefetch_desc(&vmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < 4) {
    // ================================== epilogue ==================================
    const int64_t c = c0 + tid;  // this thread's column of W = tensor-memory lane tid
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    bool ok = mbar_wait(smem_u32(&bars->acc_full), 0, abort);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
#pragma unroll 1
      for (int cb = 0; cb < kTcBM / 32; ++cb) {
        uint32_t acc[32];
        tmem_ld_x32(lane_addr + kAccCol + cb * 32, acc);
        tmem_ld_wait();
        if (c < k) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t t = m0 + cb * 32 + j;
            if (t < M) dX[t * k + c] = f32_to_bf16_bits(__uint_as_float(acc[j]));
          }
        }
      }
    }
  } else if (warp == 4) {
    // =============================== TMA producer ===============================
    if (lane == 0) {
      int issued = 0;
      for (int s = 0; s <= nk; ++s) {
        const uint32_t slot = s % kTbStages;
        if (s >= kTbStages && !mbar_wait(smem_u32(&bars->empty[slot]), ((s / kTbStages) - 1) & 1, abort)) break;
        const uint32_t full = smem_u32(&bars->full[slot]);
        mbar_arrive_expect_tx(full, kTbStageBytes);
        const uint32_t stage = smem_u32(ring + slot * kTbStageBytes);
        const CUtensorMap *am = (s < nk) ? &amap : &atmap;
        const CUtensorMap *bm = (s < nk) ? &bmap : &vmap;
        const int32_t x0 = (s < nk) ? s * kTbBK : 0;
        tma_load_2d(stage, am, x0, static_cast<int32_t>(c0), full);
        tma_load_2d(stage + kTbAHalfBytes, am, x0 + 64, static_cast<int32_t>(c0), full);
        tma_load_2d(stage + 2 * kTbAHalfBytes, bm, x0, static_cast<int32_t>(m0), full);
        tma_load_2d(stage + 2 * kTbAHalfBytes + kTbBHalfBytes, bm, x0 + 64, static_cast<int32_t>(m0), full);
        ++issued;
      }
      for (int s = (issued > kTbStages ? issued - kTbStages : 0); s < issued; ++s)
        mbar_wait_drain(smem_u32(&bars->full[s % kTbStages]), (s / kTbStages) & 1);
    }
  } else {
    // ================================ MMA issuer ================================
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTcBN, kTcBM);
      const uint32_t d_tmem = tmem + kAccCol;
      bool ok = true;
      for (int s = 0; s <= nk && ok; ++s) {
        const uint32_t slot = s % kTbStages;
        if (!(ok = mbar_wait(smem_u32(&bars->full[slot]), (s / kTbStages) & 1, abort))) break;
        tc_fence_after();
        const uint32_t abase = smem_u32(ring + slot * kTbStageBytes);
        const uint32_t bbase = abase + 2 * kTbAHalfBytes;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_ss(d_tmem, smem_desc(abase + hh * kTbAHalfBytes + kk * 32, 16, 1024, 2),
                      smem_desc(bbase + hh * kTbBHalfBytes + kk * 32, 16, 1024, 2), idesc,
                      (s > 0 || hh > 0 || kk > 0) ? 1u : 0u);
        tc_commit(smem_u32(&bars->empty[slot]));
      }
      if (ok) tc_commit(smem_u32(&bars->acc_full));
      tc_commit(smem_u32(&bars->done));
      mbar_wait_drain(smem_u32(&bars->done), 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
inline bool tc_supported(int64_t M, int64_t d, int64_t k, int32_t r) {
  (void)d;
  return M > 16 && r <= kTcMaxR && (k % kTcBK) == 0 && k >= kTcBK;
}
inline bool tc_bwd_supported(int64_t M, int64_t d, int64_t k, int32_t r) {
  return M > 16 && r <= kTcMaxR && (d % 8) == 0 && k >= kTcBK;
}
// u2 (forward, row pitch kTfUCols) or v2 (backward, row pitch 2R <= kTfUCols).
inline size_t tc_ws_bytes(int64_t M, int64_t, int64_t, int32_t) {
  return ((static_cast<size_t>(M) * kTfUCols * sizeof(uint16_t)) + 255) & ~static_cast<size_t>(255);
}
// Forward: u2 plus the block constants of every row (tf_scale_pitch(k) floats per row).
inline size_t tc_fwd_ws_bytes(int64_t M, int64_t d, int64_t k, int32_t r) {
  return tc_ws_bytes(M, d, k, r) +
         ((static_cast<size_t>(d) * tf_scale_pitch(k) * sizeof(float) + 255) & ~static_cast<size_t>(255));
}
inline int64_t tb_ldw(int64_t d) { return (d + 7) & ~int64_t{7}; }
// Backward: v2, W^T (k rows of tb_ldw(d) bf16) and AT2 (k rows of kTfUCols bf16).
inline size_t tc_bwd_ws_bytes(int64_t M, int64_t d, int64_t k, int32_t r) {
  return tc_ws_bytes(M, d, k, r) + ((static_cast<size_t>(tb_ldw(d)) * k * 2 + 255) & ~static_cast<size_t>(255)) +
         ((static_cast<size_t>(k) * kTfUCols * 2 + 255) & ~static_cast<size_t>(255));
}

// Tensor map of a row-major bf16 matrix [rows x cols] read in boxes of
// box_rows rows x 64 columns (128 bytes, the swizzle span) with the 128-byte
// swizzle; rows beyond the matrix read as zero.
inline const char *make_bf16_tile_map(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
                                      uint32_t box_rows) {
  return make_tile_map(map, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, rows, 64, box_rows,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace qn
