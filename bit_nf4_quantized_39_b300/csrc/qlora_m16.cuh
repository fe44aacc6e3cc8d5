// qlora_m16.cuh -- fused QLoRA forward of a group of projections of one
// input for 8 < M <= 16 tokens when X is too large to keep in shared memory:
//
//   Y_g = X deq(Q_g)^T + s_g (X A_g^T) B_g^T      X: M x k bf16, Q_g: d_g x k NF4
//
// ("PEFT course notes" §2.2, h = Wx + BAx; "QLoRA paper summary": the frozen
// weight is 4-bit NF4 with blockwise constants.)  With 16 tokens, X holds 4
// bytes per byte of 4-bit codes, so a kernel that streams 16-row groups of
// weights past X re-reads X four times as often as it reads the weights.
// Here a CTA owns up to kM16MaxTiles 16-row tiles at once and walks K in
// slices of 256 columns: each slice brings the codes of all its tiles (plus
// their block constants) and the 16 x 256 slice of X, which every tile of
// the CTA then uses — X moves once per CTA instead of once per tile.
//
// u = s_g X A_g^T comes from skinny_u_kernel (launched before, PDL).
//
// Per CTA batch of tiles: a ring of kM16Ring slices in shared memory, filled
// with 16-byte cp.async by all threads (rows past d and tokens past M are
// zero-filled; 16-byte chunks xor-swizzled by row / token so that the
// fragment reads are conflict-free); one CTA barrier per slice.  Warp w
// takes the (tile, block) items w, w + 16, w + 32 of every slice (item i =
// tile i / 4, block i % 4 of the slice), decodes each lane's 8 code bytes of
// rows g and g + 8 through the per-lane byte-pair table of the levels (as
// skinny_kernel), and runs two m16n8k16 MMAs chains (tokens 0-7 and 8-15)
// against the X fragments, scaling each block's sums by its fp32 constant.
// At the end of the batch the four items of a tile are summed in order, the
// adapter term u . B[row] is added on the MMA (u split into bf16 hi + lo),
// and Y is written in bf16.  No spin waits: only cp.async groups and CTA
// barriers.
#pragma once

#include "qlora_skinny.cuh"

namespace qn {

constexpr int kM16Warps = 16;
constexpr int kM16Threads = kM16Warps * 32;
constexpr int kM16SliceBlocks = 4;                          // 64-blocks per K-slice
constexpr int kM16MaxTiles = 12;                            // 16-row tiles per CTA batch
constexpr int kM16Ring = 4;                                 // slices in the ring
constexpr int kM16Items = kM16MaxTiles * kM16SliceBlocks / kM16Warps;  // items per warp per slice (3)
constexpr int kM16CodeBytes = kM16MaxTiles * 16 * 128;      // [tile][row][128 B]
constexpr int kM16XBytes = 16 * kM16SliceBlocks * 128;      // [token][block][128 B]
constexpr int kM16ConstBytes = kM16MaxTiles * 16 * 16;      // [tile][row][16 B]: 4 int8 or 4 fp32 constants
constexpr int kM16ScaleBytes = kM16MaxTiles * 16 * 4;       // [tile][row]: the DQ group scale
constexpr int kM16StageBytes = kM16CodeBytes + kM16XBytes + kM16ConstBytes + kM16ScaleBytes;
constexpr size_t kM16SmemBytes = 1024 + static_cast<size_t>(kM16Ring) * kM16StageBytes + kSkLutBytes;
static_assert(kM16MaxTiles * 4 * 256 * 4 <= kM16Ring * kM16StageBytes, "partial sums fit in the ring");

struct M16Tile {  // one 16-row tile of a batch
  const uint8_t *codes;   // first code byte of the tile's first row
  const void *cst;        // int8 DQ codes or fp32 absmax of that row (block 0)
  const float *scale;     // DQ group scales (dq only)
  int64_t blk0;           // flattened block index of the tile's first row, block 0
  int rows;               // valid rows (<= 16)
  int pi;                 // projection
  int row0;               // first row within the projection
  int dq;
  float mu;               // DQ mean (dq only)
};

__device__ __forceinline__ void m16_cp(uint32_t dst, const void *src, uint32_t bytes, bool ok) {
  if (bytes == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(ok ? 16u : 0u) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(ok ? 4u : 0u) : "memory");
}

__global__ void __launch_bounds__(kM16Threads, 1)
qlora_m16_kernel(const __grid_constant__ SkGroup g) {
  extern __shared__ unsigned char m16_raw[];
  unsigned char *base = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(m16_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char *ring = base;
  unsigned char *lut = ring + kM16Ring * kM16StageBytes;
  __shared__ M16Tile tiles[kM16MaxTiles];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const uint32_t lane4 = static_cast<uint32_t>(lane) << 2;
  const int M = g.M;
  const int64_t k = g.k;
  const int64_t nb = k >> 6;
  const int nsl = static_cast<int>(nb / kM16SliceBlocks);
  const int64_t ntiles = g.ngroups;
  const int64_t per = (ntiles + gridDim.x - 1) / gridDim.x;
  const int tc = per < kM16MaxTiles ? static_cast<int>(per) : kM16MaxTiles;  // tiles per batch

  {  // table: entry b of lane l = bf16(level[b & 15]) | bf16(level[b >> 4]) << 16, entries b = warp + 16 n
    const uint32_t lo = f32_to_bf16_bits(c_nf4_levels[warp]);
    uint32_t *lw = reinterpret_cast<uint32_t *>(lut);
#pragma unroll
    for (int n = 0; n < 16; ++n) lw[(warp + 16 * n) * 64 + lane] = lo | (f32_to_bf16_bits(c_nf4_levels[n]) << 16);
  }
  pdl_wait();  // X and u are written by the kernels before this one

  for (int64_t tb = static_cast<int64_t>(blockIdx.x) * tc; tb < ntiles; tb += static_cast<int64_t>(gridDim.x) * tc) {
    const int nt = (ntiles - tb < tc) ? static_cast<int>(ntiles - tb) : tc;
    if (tid < nt) {
      const int64_t T = tb + tid;
      int pi = 0;
#pragma unroll
      for (int i = 1; i < kSkMaxGroup; ++i)
        if (i < g.n && T >= g.p[i].group_off) pi = i;
      const SkProj &p = g.p[pi];
      const int row0 = static_cast<int>(T - p.group_off) * 16;
      M16Tile &tl = tiles[tid];
      tl.pi = pi;
      tl.row0 = row0;
      tl.rows = (p.q.d - row0 < 16) ? static_cast<int>(p.q.d - row0) : 16;
      tl.codes = p.q.codes + static_cast<int64_t>(row0) * (k >> 1);
      tl.blk0 = static_cast<int64_t>(row0) * nb;
      tl.dq = p.q.dq;
      tl.cst = p.q.dq ? static_cast<const void *>(p.q.absmax_q) : static_cast<const void *>(p.q.absmax);
      tl.scale = p.q.absmax_scale;
      tl.mu = p.q.dq ? __ldcg(p.q.absmax_mean) : 0.f;
    }
    __syncthreads();

    // Issues slice sl into ring slot `slot` (every thread; an empty group past the end).
    auto issue = [&](int sl, int slot) {
      if (sl < nsl) {
        const uint32_t sb = static_cast<uint32_t>(__cvta_generic_to_shared(ring + slot * kM16StageBytes));
        for (int i = tid; i < nt * 16 * 8; i += kM16Threads) {  // codes: tile, row, 16-byte chunk
          const int t = i >> 7, r = (i >> 3) & 15, c = i & 7;
          const M16Tile &tl = tiles[t];
          const bool ok = r < tl.rows;
          const uint8_t *src = tl.codes + static_cast<int64_t>(r) * (k >> 1) + static_cast<int64_t>(sl) * 128 + c * 16;
          m16_cp(sb + (t * 16 + r) * 128 + ((c ^ (r & 7)) << 4), ok ? src : tl.codes, 16, ok);
        }
        {  // X: token, block, 16-byte chunk (one per thread)
          const int tk = tid >> 5, j = (tid >> 3) & 3, c = tid & 7;
          const bool ok = tk < M;
          const uint16_t *src = g.X + static_cast<int64_t>(tk) * k + (static_cast<int64_t>(sl) * 4 + j) * 64 + c * 8;
          m16_cp(sb + kM16CodeBytes + (tk * 4 + j) * 128 + ((c ^ (tk & 7)) << 4), ok ? src : g.X, 16, ok);
        }
        for (int i = tid; i < nt * 16; i += kM16Threads) {  // block constants (and DQ scales) of tile row i
          const int t = i >> 4, r = i & 15;
          const M16Tile &tl = tiles[t];
          const bool ok = r < tl.rows;
          const int64_t blk = tl.blk0 + static_cast<int64_t>(r) * nb + static_cast<int64_t>(sl) * 4;
          const uint32_t cdst = sb + kM16CodeBytes + kM16XBytes + i * 16;
          if (tl.dq) {
            m16_cp(cdst, ok ? static_cast<const int8_t *>(tl.cst) + blk : tl.cst, 4, ok);
            m16_cp(sb + kM16CodeBytes + kM16XBytes + kM16ConstBytes + i * 4, ok ? tl.scale + (blk >> 8) : tl.scale, 4,
                   ok);
          } else {
            m16_cp(cdst, ok ? static_cast<const float *>(tl.cst) + blk : tl.cst, 16, ok);
          }
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };

    float acc[kM16Items][2][4];
#pragma unroll
    for (int u = 0; u < kM16Items; ++u)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[u][mt][e] = 0.f;

#pragma unroll
    for (int j = 0; j < kM16Ring - 1; ++j) issue(j, j);
    for (int sl = 0; sl < nsl; ++sl) {
      asm volatile("cp.async.wait_group %0;" ::"n"(kM16Ring - 2) : "memory");
      __syncthreads();  // slice sl visible to all; slot (sl - 1) % ring no longer read
      issue(sl + kM16Ring - 1, (sl + kM16Ring - 1) % kM16Ring);
      const unsigned char *stage = ring + (sl % kM16Ring) * kM16StageBytes;
      const unsigned char *xs = stage + kM16CodeBytes;
      const unsigned char *cs = xs + kM16XBytes;
      const float *scs = reinterpret_cast<const float *>(cs + kM16ConstBytes);
#pragma unroll
      for (int u = 0; u < kM16Items; ++u) {
        const int it = warp + kM16Warps * u, t = it >> 2, j = it & 3;
        if (t >= nt) break;  // the same in the whole warp
        const M16Tile &tl = tiles[t];
        // code bytes 8 tq .. 8 tq + 7 of block j for rows gq and gq + 8
        const int chunk = 2 * j + (tq >> 1);
        const uint32_t off = ((chunk ^ (gq & 7)) << 4) + ((tq & 1) << 3);
        const uint2 c0 = *reinterpret_cast<const uint2 *>(stage + (t * 16 + gq) * 128 + off);
        const uint2 c1 = *reinterpret_cast<const uint2 *>(stage + (t * 16 + gq + 8) * 128 + off);
        uint32_t a0[8], a1[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          a0[i] = *reinterpret_cast<const uint32_t *>(lut + sk_lut_off(c0.x, lane4, 0x5504u | (i << 4)));
          a0[4 + i] = *reinterpret_cast<const uint32_t *>(lut + sk_lut_off(c0.y, lane4, 0x5504u | (i << 4)));
          a1[i] = *reinterpret_cast<const uint32_t *>(lut + sk_lut_off(c1.x, lane4, 0x5504u | (i << 4)));
          a1[4 + i] = *reinterpret_cast<const uint32_t *>(lut + sk_lut_off(c1.y, lane4, 0x5504u | (i << 4)));
        }
        float m[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = t * 16 + gq + 8 * h;
          if (tl.dq)
            m[h] = dq_absmax(static_cast<int8_t>(cs[row * 16 + j]), scs[row], tl.mu);
          else
            m[h] = reinterpret_cast<const float *>(cs + row * 16)[j];
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const int tk = gq + 8 * mt;
          const unsigned char *xr = xs + (tk * 4 + j) * 128;
          const uint4 x0 = *reinterpret_cast<const uint4 *>(xr + (((2 * tq) ^ (tk & 7)) << 4));
          const uint4 x1 = *reinterpret_cast<const uint4 *>(xr + (((2 * tq + 1) ^ (tk & 7)) << 4));
          const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          float dsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int st = 0; st < 4; ++st)
            mma_bf16_16816(dsum, a0[2 * st], a1[2 * st], a0[2 * st + 1], a1[2 * st + 1], xw[2 * st], xw[2 * st + 1]);
          acc[u][mt][0] = fmaf(dsum[0], m[0], acc[u][mt][0]);
          acc[u][mt][1] = fmaf(dsum[1], m[0], acc[u][mt][1]);
          acc[u][mt][2] = fmaf(dsum[2], m[1], acc[u][mt][2]);
          acc[u][mt][3] = fmaf(dsum[3], m[1], acc[u][mt][3]);
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();  // every slice consumed: the ring holds the partial sums now

    // partials [tile][block j][row][token]
    float *part = reinterpret_cast<float *>(ring);
#pragma unroll
    for (int u = 0; u < kM16Items; ++u) {
      const int it = warp + kM16Warps * u, t = it >> 2, j = it & 3;
      if (t >= nt) break;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          part[((t * 4 + j) * 16 + gq + 8 * (e >> 1)) * 16 + 8 * mt + 2 * tq + (e & 1)] = acc[u][mt][e];
    }
    __syncthreads();

    // finisher: warp t sums tile t's four blocks in order, adds u . B[row], writes Y
    if (warp < nt) {
      const M16Tile &tl = tiles[warp];
      const SkProj &p = g.p[tl.pi];
      const int64_t d = p.q.d;
      const int t = warp;
      float y[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = gq + 8 * (e >> 1), col = 8 * mt + 2 * tq + (e & 1);
          float v = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) v += part[((t * 4 + j) * 16 + row) * 16 + col];
          y[mt][e] = v;
        }
      // Adapter term s (X A^T) B^T = u B^T on the MMA: A = B rows (bf16), the
      // column operand = u split into bf16 hi + lo.
      const bool rok[2] = {gq < tl.rows, gq + 8 < tl.rows};
      const uint16_t *brow0 = p.B + static_cast<int64_t>(tl.row0 + gq) * p.r;
      const uint16_t *brow1 = p.B + static_cast<int64_t>(tl.row0 + gq + 8) * p.r;
      for (int j0 = 0; j0 < p.r; j0 += 16) {
        uint32_t af[4];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {  // af[qq]: row gq + 8 (qq & 1), columns j0 + 2 tq + 8 (qq >> 1) + {0, 1}
          const int jj = j0 + 2 * tq + 8 * (qq >> 1);
          uint32_t lo = 0u, hi = 0u;
          if (rok[qq & 1]) {
            const uint16_t *br = (qq & 1) ? brow1 : brow0;
            if (jj < p.r) lo = br[jj];
            if (jj + 1 < p.r) hi = br[jj + 1];
          }
          af[qq] = lo | (hi << 16);
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const int tok = gq + 8 * mt;
          uint32_t bh[2], bl[2];
#pragma unroll
          for (int qq = 0; qq < 2; ++qq) {  // column rows j0 + 2 tq + 8 qq + {0, 1}
            const int jj = j0 + 2 * tq + 8 * qq;
            float u0 = 0.f, u1 = 0.f;
            if (tok < M) {
              const float *ut = g.u + static_cast<int64_t>(tok) * g.rtot + p.u_off;
              if (jj < p.r) u0 = __ldcg(ut + jj);
              if (jj + 1 < p.r) u1 = __ldcg(ut + jj + 1);
            }
            const uint32_t h0 = f32_to_bf16_bits(u0), h1 = f32_to_bf16_bits(u1);
            bh[qq] = h0 | (h1 << 16);
            bl[qq] = static_cast<uint32_t>(f32_to_bf16_bits(u0 - bf16_bits_to_f32(h0))) |
                     (static_cast<uint32_t>(f32_to_bf16_bits(u1 - bf16_bits_to_f32(h1))) << 16);
          }
          mma_bf16_16816(y[mt], af[0], af[1], af[2], af[3], bh[0], bh[1]);
          mma_bf16_16816(y[mt], af[0], af[1], af[2], af[3], bl[0], bl[1]);
        }
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t row = tl.row0 + gq + 8 * (e >> 1);
          const int tok = 8 * mt + 2 * tq + (e & 1);
          if (tok < M && row < d) p.Y[static_cast<int64_t>(tok) * d + row] = f32_to_bf16_bits(y[mt][e]);
        }
    }
    __syncthreads();  // the next batch refills the ring and the tile table
  }
}

}  // namespace qn
