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
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dsa {

template <int D, typename KV, int G>
struct MassTiling {
  static constexpr int kRowBytes = D * static_cast<int>(sizeof(KV));
  static constexpr int kTByBytes = 8192 / kRowBytes;
  static constexpr int kTByRegs = 64 / G;
  static constexpr int kT0 = kTByBytes < kTByRegs ? kTByBytes : kTByRegs;
  static constexpr int T = kT0 > 32 ? 32 : (kT0 < 8 ? 8 : kT0);
  static constexpr int S = 3;
  static constexpr int NW = 4;
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

template <int D, typename KV, int G>
__global__ void __launch_bounds__(MassTiling<D, KV, G>::NW * 32) mass_kernel(const MassLaunch a) {
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
  auto issue = [&](int t, int stage) {
    const int tr0 = row0 + (warp + t * NW) * T;
    const int nrows = min(T, row1 - tr0);
    if (lane == 0) mbar_arrive_expect_tx(&bars[stage], static_cast<uint32_t>(nrows * kRowBytes));
    __syncwarp();
    if (lane < nrows) {
      const int j = tr0 + lane;
      int pg = pt[j >> 4];
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

  const int my_tiles = warp < ntiles ? (ntiles - warp + NW - 1) / NW : 0;
  for (int t = 0; t < S && t < my_tiles; ++t) issue(t, t);
  const int myrow = RowMap<T>::row(lane);
  const bool own = RowMap<T>::owner(lane);
  const size_t om_stride = static_cast<size_t>(a.max_window) + 1;
  int failed_at = -1;
  for (int t = 0; t < my_tiles; ++t) {
    const int stage = t % S;
    if (!mbar_wait(&bars[stage], static_cast<uint32_t>(t / S) & 1u)) {
      failed_at = t;
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
    int bin = 3;
    if (j < P) {
      bin = 0;
    } else if (o <= a.r_local) {
      bin = 1;
    } else if (o <= W) {
      const int k0 = o / w;
      if ((k0 >= 1 && o - k0 * w <= a.r_diag) || ((k0 + 1) * w - o <= a.r_diag)) bin = 2;
    }
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
    if (t + S < my_tiles) issue(t + S, stage);
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

// One warp per (request, query head): combine chunks, normalise bins, and turn
// raw window scores into weights.
__global__ void __launch_bounds__(128) mass_merge_kernel(const MassLaunch a) {
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

template <int D, typename KV, int G>
cudaError_t launch_mass_one(const MassLaunch& a, cudaStream_t s) {
  using Tl = MassTiling<D, KV, G>;
  auto kern = mass_kernel<D, KV, G>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Tl::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(a.num_chunks, a.hkv, a.batch), Tl::NW * 32, Tl::kSmem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int pairs = a.batch * a.hq;
  mass_merge_kernel<<<(pairs + 3) / 4, 128, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename KV>
cudaError_t launch_mass_t(const MassLaunch& a, cudaStream_t s) {
  const int g = a.hq / a.hkv;
#define DSA_CASE(DD, GG) \
  if (a.head_dim == DD && g == GG) return launch_mass_one<DD, KV, GG>(a, s);
  DSA_CASE(64, 1)
  DSA_CASE(64, 2)
  DSA_CASE(64, 4)
  DSA_CASE(64, 8)
  DSA_CASE(128, 1)
  DSA_CASE(128, 2)
  DSA_CASE(128, 4)
  DSA_CASE(128, 8)
#undef DSA_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_mass(const MassLaunch& a, bool kv_bf16, cudaStream_t s) {
  return kv_bf16 ? launch_mass_t<bf16_t>(a, s) : launch_mass_t<float>(a, s);
}

}  // namespace dsa
