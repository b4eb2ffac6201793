// mass.cu -- attention-mass characterisation: where the dense causal decode
// softmax of each (request, query head) puts its weight.
//
// Follows "Understanding and Exploiting Diagonal Attention Sparsity in
// Autoregressive Image Generation": the arXiv abstract reports attention
// concentrated on prompt and local tokens and a diagonal pattern from spatial
// locality; the paper-daily summary (section 技术方法详解) explains that raster
// order puts a token's spatial neighbours at offsets k*w +- r.  Bins:
//   0 prompt  (j < P), 1 local (o <= r_local), 2 diagonal (o <= W, |o - k w| <=
//   r_diag for some k >= 1), 3 other; plus the weight of every window offset.
//
// One pass over K only.  grid (chunk, kv head, request); each warp keeps, per
// query head, the running max m, the running sum l and the four running bin
// sums, all rescaled together like the online-softmax sum.  Window rows store
// their raw log2-domain score into offset_mass; mass_merge_kernel combines the
// chunks by log-sum-exp and turns raw scores into weights exp2(s - lse2).
//
// Two score engines: mass_mma_kernel (bf16 q and K, grouped-query heads) puts
// the G dot products of 16-row blocks on the tensor cores; mass_kernel (every
// other case) sums per-lane partial dot products with a reduce-scatter.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "mma.cuh"

namespace dsa {

#ifndef DSA_MASS_CC_STAGES
#define DSA_MASS_CC_STAGES 2
#endif
#ifndef DSA_MASS_CC_STAGE_BYTES
#define DSA_MASS_CC_STAGE_BYTES 4096
#endif
#ifndef DSA_MASS_CC_WARPS
#define DSA_MASS_CC_WARPS 4
#endif
template <int D, typename KV, int G>
struct MassTiling {
  static constexpr int kRowBytes = D * static_cast<int>(sizeof(KV));
  static constexpr int kTByBytes = DSA_MASS_CC_STAGE_BYTES / kRowBytes;
  static constexpr int kTByRegs = 64 / G;
  static constexpr int kT0 = kTByBytes < kTByRegs ? kTByBytes : kTByRegs;
  static constexpr int T = kT0 > 32 ? 32 : (kT0 < 8 ? 8 : kT0);
  static constexpr int S = DSA_MASS_CC_STAGES;
  static constexpr int NW = DSA_MASS_CC_WARPS;
  static constexpr int kDPL = D / 32;
  static constexpr int kStageBytes = T * kRowBytes;
  static constexpr int kWarpBytes = S * kStageBytes;
  static constexpr int kBarOff = NW * kWarpBytes;
  static constexpr int kMOff = kBarOff + NW * S * 8;
  static constexpr int kSmem = kMOff + NW * G * 6 * 4;
};

constexpr int kMassPart = 6;  // m, l, bin0..bin3

// Same validity rule in both mass kernels.
__device__ __forceinline__ int mass_request_check(const MassLaunch& a, int b, int* L, int* P,
                                                  int* W, int* w) {
  *L = a.seq_len[b];
  *P = a.prompt_len[b];
  *W = a.window[b];
  *w = a.grid_w[b];
  if (*L < 1 || *L > a.max_pages * kPage) return DSA_DEV_BAD_SEQ_LEN;
  if (*P < 0) return DSA_DEV_BAD_PROMPT;
  if (*W < 0 || *W > a.max_window) return DSA_DEV_BAD_WINDOW;
  if (*w < 1) return DSA_DEV_BAD_GRID_W;
  return 0;
}

// Bin of row j (offset o = i - j) under the rule in the file comment.
__device__ __forceinline__ int mass_bin(const MassLaunch& a, int j, int o, int P, int W, int w) {
  if (j < P) return 0;
  if (o <= a.r_local) return 1;
  if (o <= W) {
    const int k0 = o / w;
    if ((k0 >= 1 && o - k0 * w <= a.r_diag) || ((k0 + 1) * w - o <= a.r_diag)) return 2;
  }
  return 3;
}

template <int D, typename KV, int G>
__global__ void __launch_bounds__(MassTiling<D, KV, G>::NW * 32) mass_kernel(const MassLaunch a) {
  griddep_wait();
  griddep_launch_dependents();
  using Tl = MassTiling<D, KV, G>;
  constexpr int T = Tl::T, S = Tl::S, NW = Tl::NW, DPL = Tl::kDPL;
  constexpr int kRowBytes = Tl::kRowBytes;
  extern __shared__ __align__(128) unsigned char smem[];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  int L, P, W, w;
  const int code = mass_request_check(a, b, &L, &P, &W, &w);
  if (code != 0) {
    if (c == 0 && threadIdx.x == 0) set_error(a.err, code);
    return;
  }
  const int i = L - 1;
  const int row0 = c * a.chunk;
  if (row0 >= L) return;
  const int row1 = min(L, row0 + a.chunk);
  const int ntiles = (row1 - row0 + T - 1) / T;

  KV* kst = reinterpret_cast<KV*>(smem + warp * Tl::kWarpBytes);  // [S][T][D]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tl::kBarOff) + warp * S;
  float* mbuf = reinterpret_cast<float*>(smem + Tl::kMOff);  // [NW][G][6]
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const KV* kg = reinterpret_cast<const KV*>(a.k);
  const int32_t* pt = a.page_table + static_cast<size_t>(b) * a.max_pages;
  const int my_tiles = warp < ntiles ? (ntiles - warp + NW - 1) / NW : 0;
  // page id of this lane's row of tile t, loaded a tile before its copy
  auto load_pg = [&](int t) -> int {
    const int j = row0 + (warp + t * NW) * T + lane;
    return (t < my_tiles && lane < T && j < row1) ? __ldg(pt + (j >> 4)) : 0;
  };
  auto issue = [&](int t, int stage, int pg) {
    const int tr0 = row0 + (warp + t * NW) * T;
    const int nrows = min(T, row1 - tr0);
    if (lane == 0) mbar_arrive_expect_tx(&bars[stage], static_cast<uint32_t>(nrows * kRowBytes));
    __syncwarp();
    if (lane < nrows) {
      const int j = tr0 + lane;
      if (static_cast<unsigned>(pg) >= static_cast<unsigned>(a.num_pages)) {
        set_error(a.err, DSA_DEV_BAD_PAGE);
        pg = 0;
      }
      const size_t off = ((static_cast<size_t>(pg) * kPage + (j & (kPage - 1))) * a.hkv + hk) * D;
      bulk_copy_g2s(kst + (static_cast<size_t>(stage) * T + lane) * D, kg + off, kRowBytes,
                    &bars[stage]);
    }
  };

  float qv[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h)
    load_q<DPL>(a.q, a.q_bf16 != 0, (static_cast<size_t>(b) * a.hq + hk * G + h) * D + lane * DPL,
                a.scale_log2, qv[h]);

  float m_run[G], l_run[G], bins[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) bins[h][k] = 0.f;
  }

  {
    int pg0[S];
#pragma unroll
    for (int t = 0; t < S; ++t) pg0[t] = load_pg(t);
#pragma unroll
    for (int t = 0; t < S; ++t)
      if (t < my_tiles) issue(t, t, pg0[t]);
  }
  int pg_next = load_pg(S);  // next tile to issue: S
  const int myrow = RowMap<T>::row(lane);
  const bool own = RowMap<T>::owner(lane);
  const size_t om_stride = static_cast<size_t>(a.max_window) + 1;
  int failed_at = -1;
  for (int t = 0; t < my_tiles; ++t) {
    const int stage = t % S;
    if (!__all_sync(0xffffffffu, mbar_wait(&bars[stage], static_cast<uint32_t>(t / S) & 1u))) {
      failed_at = t;  // the whole warp leaves together
      break;
    }
    const int tr0 = row0 + (warp + t * NW) * T;
    const int nrows = min(T, row1 - tr0);
    const KV* kt = kst + static_cast<size_t>(stage) * T * D + lane * DPL;
    float part[G][T];
#pragma unroll
    for (int r = 0; r < T; ++r) {
      float kf[DPL];
      Vec<KV, DPL>::load(kt + r * D, kf);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) s = fmaf(qv[h][e], kf[e], s);
        part[h][r] = s;
      }
    }
    // bin of this lane's row
    const int j = tr0 + myrow;
    const int o = i - j;
    const int bin = mass_bin(a, j, o, P, W, w);
    const bool valid = myrow < nrows;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float s = reduce_scatter<T>(part[h], lane);
      s = valid ? s : -INFINITY;
      if (own && valid && o <= W && a.offset_mass != nullptr)
        a.offset_mass[(static_cast<size_t>(b) * a.hq + hk * G + h) * om_stride + o] = s;
      const float mnew = fmaxf(m_run[h], warp_max(s));
      const float alpha = exp2f(m_run[h] - mnew);
      const float p = own ? exp2f(s - mnew) : 0.f;
      l_run[h] = l_run[h] * alpha + p;
#pragma unroll
      for (int k = 0; k < 4; ++k) bins[h][k] = bins[h][k] * alpha + (bin == k ? p : 0.f);
      m_run[h] = mnew;
    }
    __syncwarp();
    fence_proxy_async_smem();
    if (t + S < my_tiles) issue(t + S, stage, pg_next);
    pg_next = load_pg(t + S + 1);
  }
  if (failed_at >= 0) {
    if (lane == 0) set_error(a.err, DSA_DEV_TIMEOUT);
    for (int t = failed_at; t < my_tiles && t < failed_at + S; ++t)
      mbar_wait(&bars[t % S], static_cast<uint32_t>(t / S) & 1u);
  }

#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float l = warp_sum(l_run[h]);
    float bs[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) bs[k] = warp_sum(bins[h][k]);
    if (lane == 0) {
      float* mw = mbuf + (warp * G + h) * kMassPart;
      mw[0] = m_run[h];
      mw[1] = l;
#pragma unroll
      for (int k = 0; k < 4; ++k) mw[2 + k] = bs[k];
    }
  }
  __syncthreads();
  for (int x = threadIdx.x; x < G * kMassPart; x += NW * 32) {
    const int h = x / kMassPart, f = x % kMassPart;
    float mstar = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < NW; ++ww) mstar = fmaxf(mstar, mbuf[(ww * G + h) * kMassPart]);
    float v = mstar;
    if (f > 0) {
      v = 0.f;
#pragma unroll
      for (int ww = 0; ww < NW; ++ww) {
        const float* src = mbuf + (ww * G + h) * kMassPart;
        const float sc = src[0] == -INFINITY ? 0.f : exp2f(src[0] - mstar);
        v = fmaf(sc, src[f], v);
      }
    }
    const size_t qh = static_cast<size_t>(b) * a.hq + hk * G + h;
    a.part[(qh * a.num_chunks + c) * kMassPart + f] = v;
  }
}

// Tensor-core tiling: K rows only, T rows per tile, rows padded by 16 bytes so
// that the ldmatrix row addresses of one 8x8 tile fall in distinct banks.
#ifndef DSA_MASS_STAGES
#define DSA_MASS_STAGES 2
#endif
#ifndef DSA_MASS_WARPS
#define DSA_MASS_WARPS 4
#endif
#ifndef DSA_MASS_STAGE_BYTES
#define DSA_MASS_STAGE_BYTES 4096
#endif
template <int D>
struct MassMmaTiling {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kT0 = DSA_MASS_STAGE_BYTES / kRowBytes;
  static constexpr int T = kT0 > 64 ? 64 : (kT0 < 16 ? 16 : kT0);
  static_assert(T == 16 || T == 32 || T == 64, "tile rows: whole mma blocks, <= 2 per lane");
  static constexpr int S = DSA_MASS_STAGES;
  static constexpr int NW = DSA_MASS_WARPS;
  static constexpr int kRowStride = kRowBytes + 16;
  static constexpr int kStageBytes = T * kRowStride;
  static constexpr int kWarpBytes = S * kStageBytes;
  static constexpr int kBarOff = NW * kWarpBytes;
  static constexpr int kMOff = kBarOff + NW * S * 8;
  static constexpr int kSmem = kMOff + NW * 8 * kMassPart * 4;
};

// Scores S = K q^T of a 16-row block with mma.sync m16n8k16 (A: 16 K rows x
// 16 dims via ldmatrix, B: q of the G <= 8 heads as columns).  Thread (g4 =
// lane/4, tig = lane%4) ends with rows g4 and g4+8 of the block for heads
// 2 tig and 2 tig + 1, the layout of the mma accumulator.
template <int D, int G>
__global__ void __launch_bounds__(MassMmaTiling<D>::NW * 32)
    mass_mma_kernel(const MassLaunch a) {
  griddep_wait();
  griddep_launch_dependents();
  using Tl = MassMmaTiling<D>;
  constexpr int T = Tl::T, S = Tl::S, NW = Tl::NW, RB = T / 16, NK = D / 16;
  constexpr int RPL = (T + 31) / 32;  // rows of a tile per lane (lane + 32 u < T)
  constexpr int kRowBytes = Tl::kRowBytes, kRowStride = Tl::kRowStride;
  extern __shared__ __align__(128) unsigned char smem[];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  int L, P, W, w;
  const int code = mass_request_check(a, b, &L, &P, &W, &w);
  if (code != 0) {
    if (c == 0 && threadIdx.x == 0) set_error(a.err, code);
    return;
  }
  const int i = L - 1;
  const int row0 = c * a.chunk;
  if (row0 >= L) return;
  const int row1 = min(L, row0 + a.chunk);
  const int ntiles = (row1 - row0 + T - 1) / T;
  const int my_tiles = warp < ntiles ? (ntiles - warp + NW - 1) / NW : 0;

  unsigned char* kst = smem + warp * Tl::kWarpBytes;  // [S][T] K rows, kRowStride apart
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tl::kBarOff) + warp * S;
  float* mbuf = reinterpret_cast<float*>(smem + Tl::kMOff);  // [NW][G][6]
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const bf16_t* kg = reinterpret_cast<const bf16_t*>(a.k);
  const int32_t* pt = a.page_table + static_cast<size_t>(b) * a.max_pages;
  auto tile_r0 = [&](int t) { return row0 + (warp + t * NW) * T; };
  // page ids of this lane's rows (lane + 32 u) of tile t, loaded a tile ahead
  auto load_pg = [&](int t, int (&pg)[RPL]) {
#pragma unroll
    for (int u = 0; u < RPL; ++u) {
      const int j = tile_r0(t) + lane + 32 * u;
      pg[u] = (t < my_tiles && lane + 32 * u < T && j < row1) ? __ldg(pt + (j >> 4)) : 0;
    }
  };
  auto issue = [&](int t, int stage, const int (&pg)[RPL]) {
    const int tr0 = tile_r0(t);
    const int nrows = min(T, row1 - tr0);
    if (lane == 0) mbar_arrive_expect_tx(&bars[stage], static_cast<uint32_t>(nrows * kRowBytes));
    __syncwarp();
#pragma unroll
    for (int u = 0; u < RPL; ++u) {
      const int r = lane + 32 * u;
      if (r < nrows) {
        int p = pg[u];
        if (static_cast<unsigned>(p) >= static_cast<unsigned>(a.num_pages)) {
          set_error(a.err, DSA_DEV_BAD_PAGE);
          p = 0;
        }
        const int j = tr0 + r;
        const size_t off = ((static_cast<size_t>(p) * kPage + (j & (kPage - 1))) * a.hkv + hk) * D;
        bulk_copy_g2s(kst + (static_cast<size_t>(stage) * T + r) * kRowStride, kg + off, kRowBytes,
                      &bars[stage]);
      }
    }
  };

  const int g4 = lane >> 2, tig = lane & 3;
  uint32_t qf[NK][2];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(a.q) +
                          (static_cast<size_t>(b) * a.hq + hk * G + (g4 < G ? g4 : 0)) * (D / 2);
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
      qf[kk][0] = g4 < G ? __ldg(q32 + kk * 8 + tig) : 0u;
      qf[kk][1] = g4 < G ? __ldg(q32 + kk * 8 + 4 + tig) : 0u;
    }
  }
  float m2[2], l2[2], bins[2][4];
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    m2[jj] = -INFINITY;
    l2[jj] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) bins[jj][k] = 0.f;
  }

  int pgn[RPL];
#pragma unroll
  for (int t = 0; t < S; ++t) {
    if (t < my_tiles) {
      load_pg(t, pgn);
      issue(t, t, pgn);
    }
  }
  load_pg(S, pgn);

  const size_t om_stride = static_cast<size_t>(a.max_window) + 1;
  int failed_at = -1;
  for (int t = 0; t < my_tiles; ++t) {
    const int stage = t % S;
    if (!__all_sync(0xffffffffu, mbar_wait(&bars[stage], static_cast<uint32_t>(t / S) & 1u))) {
      failed_at = t;  // the whole warp leaves together
      break;
    }
    const int tr0 = tile_r0(t);
    const int nrows = min(T, row1 - tr0);
    const unsigned char* kt = kst + static_cast<size_t>(stage) * T * kRowStride;
    float sm[RB][4];
#pragma unroll
    for (int rb = 0; rb < RB; ++rb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) sm[rb][e] = 0.f;
      const unsigned char* arow =
          kt + (rb * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * kRowStride + 16 * (lane >> 4);
#pragma unroll
      for (int kk = 0; kk < NK; ++kk) {
        uint32_t af[4];
        ldsm_x4(af, arow + 32 * kk);
        mma_bf16(sm[rb], af, qf[kk][0], qf[kk][1]);
      }
    }
    // bins and window offsets of the thread's rows (shared by its two heads)
    int rbin[RB][2], roff[RB][2];
#pragma unroll
    for (int rb = 0; rb < RB; ++rb)
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        const int r = rb * 16 + g4 + 8 * hi;
        const int j = tr0 + r;
        roff[rb][hi] = r < nrows ? i - j : -1;
        rbin[rb][hi] = r < nrows ? mass_bin(a, j, i - j, P, W, w) : 3;
      }
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int h = 2 * tig + jj;
      float tmax = -INFINITY;
#pragma unroll
      for (int rb = 0; rb < RB; ++rb)
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          float& x = sm[rb][2 * hi + jj];
          x = roff[rb][hi] >= 0 ? x * a.scale_log2 : -INFINITY;
          tmax = fmaxf(tmax, x);
          if (h < G && roff[rb][hi] >= 0 && roff[rb][hi] <= W && a.offset_mass != nullptr)
            a.offset_mass[(static_cast<size_t>(b) * a.hq + hk * G + h) * om_stride +
                          roff[rb][hi]] = x;
        }
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
      const float mnew = fmaxf(m2[jj], tmax);
      const float alpha = exp2f(m2[jj] - mnew);
      m2[jj] = mnew;
      float psum = 0.f, pb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int rb = 0; rb < RB; ++rb)
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          const float p = exp2f(sm[rb][2 * hi + jj] - mnew);
          psum += p;
#pragma unroll
          for (int k = 0; k < 4; ++k) pb[k] += rbin[rb][hi] == k ? p : 0.f;
        }
      l2[jj] = l2[jj] * alpha + psum;
#pragma unroll
      for (int k = 0; k < 4; ++k) bins[jj][k] = bins[jj][k] * alpha + pb[k];
    }
    __syncwarp();
    fence_proxy_async_smem();
    if (t + S < my_tiles) issue(t + S, stage, pgn);
    load_pg(t + S + 1, pgn);
  }
  if (failed_at >= 0) {
    // Give the copies still in flight a bounded chance to land before exiting.
    if (lane == 0) set_error(a.err, DSA_DEV_TIMEOUT);
    for (int t = failed_at; t < my_tiles && t < failed_at + S; ++t)
      mbar_wait(&bars[t % S], static_cast<uint32_t>(t / S) & 1u);
  }

  // the 8 lanes of a column pair share m; sum their l and bins
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    float v[5] = {l2[jj], bins[jj][0], bins[jj][1], bins[jj][2], bins[jj][3]};
#pragma unroll
    for (int f = 0; f < 5; ++f) {
      v[f] += __shfl_xor_sync(0xffffffffu, v[f], 4);
      v[f] += __shfl_xor_sync(0xffffffffu, v[f], 8);
      v[f] += __shfl_xor_sync(0xffffffffu, v[f], 16);
    }
    const int h = 2 * tig + jj;
    if (g4 == 0 && h < G) {
      float* mw = mbuf + (warp * G + h) * kMassPart;
      mw[0] = m2[jj];
#pragma unroll
      for (int f = 0; f < 5; ++f) mw[1 + f] = v[f];
    }
  }
  __syncthreads();
  for (int x = threadIdx.x; x < G * kMassPart; x += NW * 32) {
    const int h = x / kMassPart, f = x % kMassPart;
    float mstar = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < NW; ++ww) mstar = fmaxf(mstar, mbuf[(ww * G + h) * kMassPart]);
    float v = mstar;
    if (f > 0) {
      v = 0.f;
#pragma unroll
      for (int ww = 0; ww < NW; ++ww) {
        const float* src = mbuf + (ww * G + h) * kMassPart;
        const float sc = src[0] == -INFINITY ? 0.f : exp2f(src[0] - mstar);
        v = fmaf(sc, src[f], v);
      }
    }
    const size_t qh = static_cast<size_t>(b) * a.hq + hk * G + h;
    a.part[(qh * a.num_chunks + c) * kMassPart + f] = v;
  }
}

// One warp per (request, query head): combine chunks, normalise bins, and turn
// raw window scores into weights.
__global__ void __launch_bounds__(128) mass_merge_kernel(const MassLaunch a) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (gw >= a.batch * a.hq) return;
  const int b = gw / a.hq;
  int L, P, W, w;
  const size_t om_stride = static_cast<size_t>(a.max_window) + 1;
  const float qnan = __int_as_float(0x7fc00000);
  if (mass_request_check(a, b, &L, &P, &W, &w) != 0) {
    if (lane < 4) a.mass[static_cast<size_t>(gw) * 4 + lane] = qnan;
    if (a.offset_mass != nullptr)
      for (int o = lane; o <= a.max_window; o += 32) a.offset_mass[gw * om_stride + o] = qnan;
    return;
  }
  const int i = L - 1;
  const int nch = (L + a.chunk - 1) / a.chunk;
  const float* pp = a.part + static_cast<size_t>(gw) * a.num_chunks * kMassPart;
  float mstar = -INFINITY;
  for (int c = lane; c < nch; c += 32) mstar = fmaxf(mstar, pp[c * kMassPart]);
  mstar = warp_max(mstar);
  float acc[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
  for (int c = lane; c < nch; c += 32) {
    const float sc = exp2f(pp[c * kMassPart] - mstar);
#pragma unroll
    for (int f = 0; f < 5; ++f) acc[f] = fmaf(sc, pp[c * kMassPart + 1 + f], acc[f]);
  }
#pragma unroll
  for (int f = 0; f < 5; ++f) acc[f] = warp_sum(acc[f]);
  if (lane < 4) a.mass[static_cast<size_t>(gw) * 4 + lane] = acc[1 + lane] / acc[0];
  if (a.offset_mass != nullptr) {
    const float lse2 = mstar + log2f(acc[0]);
    for (int o = lane; o <= a.max_window; o += 32) {
      float* dst = a.offset_mass + gw * om_stride + o;
      *dst = (o <= W && o <= i) ? exp2f(*dst - lse2) : 0.f;
    }
  }
}

// Tensor cores for bf16 q and K with grouped-query heads.
bool mass_uses_tensor_cores(bool kv_bf16, bool q_bf16, int group) {
  return kv_bf16 && q_bf16 && group >= 2;
}

template <typename Kern>
cudaError_t launch_mass_kernel(Kern kern, int smem, int threads, const MassLaunch& a,
                               cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(a.num_chunks, a.hkv, a.batch), dim3(threads), smem, s, a);
  if (e != cudaSuccess) return e;
  const int pairs = a.batch * a.hq;
  return launch_pdl(mass_merge_kernel, dim3((pairs + 3) / 4), dim3(128), 0, s, a);
}

// Calls f(kernel, dynamic smem, threads per CTA, rows per CTA pass) for the
// instantiation that serves (head_dim, group, dtypes); returns `fallback` when
// none does.
template <typename F, typename R>
R with_mass_kernel(int head_dim, int group, bool kv_bf16, bool q_bf16, F f, R fallback) {
#define DSA_MMA_CASE(DD, GG)                                                            \
  if (head_dim == DD && group == GG) {                                                  \
    using Tl = MassMmaTiling<DD>;                                                       \
    return f(mass_mma_kernel<DD, GG>, Tl::kSmem, Tl::NW * 32, Tl::NW * Tl::T);          \
  }
#define DSA_CASE(KV, DD, GG)                                                            \
  if (head_dim == DD && group == GG) {                                                  \
    using Tl = MassTiling<DD, KV, GG>;                                                  \
    return f(mass_kernel<DD, KV, GG>, Tl::kSmem, Tl::NW * 32, Tl::NW * Tl::T);          \
  }
  if (mass_uses_tensor_cores(kv_bf16, q_bf16, group)) {
    DSA_MMA_CASE(64, 2)
    DSA_MMA_CASE(64, 4)
    DSA_MMA_CASE(64, 8)
    DSA_MMA_CASE(128, 2)
    DSA_MMA_CASE(128, 4)
    DSA_MMA_CASE(128, 8)
  } else if (kv_bf16) {
    DSA_CASE(bf16_t, 64, 1)
    DSA_CASE(bf16_t, 64, 2)
    DSA_CASE(bf16_t, 64, 4)
    DSA_CASE(bf16_t, 64, 8)
    DSA_CASE(bf16_t, 128, 1)
    DSA_CASE(bf16_t, 128, 2)
    DSA_CASE(bf16_t, 128, 4)
    DSA_CASE(bf16_t, 128, 8)
  } else {
    DSA_CASE(float, 64, 1)
    DSA_CASE(float, 64, 2)
    DSA_CASE(float, 64, 4)
    DSA_CASE(float, 64, 8)
    DSA_CASE(float, 128, 1)
    DSA_CASE(float, 128, 2)
    DSA_CASE(float, 128, 4)
    DSA_CASE(float, 128, 8)
  }
#undef DSA_MMA_CASE
#undef DSA_CASE
  return fallback;
}

cudaError_t launch_mass(const MassLaunch& a, bool kv_bf16, cudaStream_t s) {
  return with_mass_kernel(
      a.head_dim, a.hq / a.hkv, kv_bf16, a.q_bf16 != 0,
      [&](auto kern, int smem, int threads, int) {
        return launch_mass_kernel(kern, smem, threads, a, s);
      },
      cudaErrorInvalidValue);
}

int mass_rows_per_pass(int head_dim, int group, bool kv_bf16, bool q_bf16) {
  return with_mass_kernel(
      head_dim, group, kv_bf16, q_bf16, [](auto, int, int, int rows) { return rows; }, 0);
}

int mass_ctas_per_sm(int head_dim, int group, bool kv_bf16, bool q_bf16) {
  return with_mass_kernel(
      head_dim, group, kv_bf16, q_bf16,
      [](auto kern, int smem, int threads, int) {
        int n = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess)
          return 1;
        return n < 1 ? 1 : n;
      },
      1);
}

}  // namespace dsa
