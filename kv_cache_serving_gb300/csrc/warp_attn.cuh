// warp_attn.cuh -- one warp's share of decode attention for the G query heads
// of one kv head: q in registers, the online-softmax state over the rows the
// warp has seen, the step on one tile of K/V rows staged in shared memory, and
// the flush of that state as G x [acc(D), m, l] floats for a log-sum-exp merge.
//
// The method's masked softmax (paper-daily summary of "Understanding and
// Exploiting Diagonal Attention Sparsity in Autoregressive Image Generation",
// section 核心公式) over the kept rows only: scores s = scale q.k, running max
// m and sum l = sum 2^(s log2 e - m) in the log2 domain, acc = sum p v; a row
// outside the tile (past nrows) is masked to -inf.
//
// Two engines:
//  * CUDA cores (group 1, or fp32 operands): a row is served by 8 lanes holding
//    16-byte vectors at byte offsets 16 j + 128 u; the G dot products are summed
//    over the 8 lanes by a 3-step butterfly; with bf16 q and K the products use
//    fma.rn.f32.bf16 (bf16 x bf16 is exact in fp32).
//  * tensor cores (bf16 q and K, group >= 2): S = K q^T per 16-row block with
//    mma.sync m16n8k16 (K via ldmatrix, q as the B operand, heads as columns),
//    then O^T += V^T P with V via ldmatrix.trans and P split into bf16 hi + lo,
//    moved from the S accumulators into B fragments by movmatrix (no shared memory).
#pragma once

#include <math.h>

#include "common.cuh"
#include "mma.cuh"

namespace dsa {

// acc += lo(k2)*lo(q2) + hi(k2)*hi(q2), bf16 operands, fp32 accumulation (the
// product of two bf16 values is exact in fp32).
__device__ __forceinline__ float fma2_bf16(uint32_t k2, uint32_t q2, float acc) {
  asm("{\n\t.reg .b16 kl, kh, ql, qh;\n\t"
      "mov.b32 {kl, kh}, %1;\n\t"
      "mov.b32 {ql, qh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, kl, ql, %0;\n\t"
      "fma.rn.f32.bf16 %0, kh, qh, %0;\n\t}"
      : "+f"(acc)
      : "r"(k2), "r"(q2));
  return acc;
}

// The 16 / sizeof(KV) elements of a 16-byte vector as fp32.
template <typename KV>
__device__ __forceinline__ void vec_to_f32(const uint4& v, float* o);
template <>
__device__ __forceinline__ void vec_to_f32<bf16_t>(const uint4& v, float* o) {
  o[0] = bf16_lo(v.x);
  o[1] = bf16_hi(v.x);
  o[2] = bf16_lo(v.y);
  o[3] = bf16_hi(v.y);
  o[4] = bf16_lo(v.z);
  o[5] = bf16_hi(v.z);
  o[6] = bf16_lo(v.w);
  o[7] = bf16_hi(v.w);
}
template <>
__device__ __forceinline__ void vec_to_f32<float>(const uint4& v, float* o) {
  o[0] = __uint_as_float(v.x);
  o[1] = __uint_as_float(v.y);
  o[2] = __uint_as_float(v.z);
  o[3] = __uint_as_float(v.w);
}

// The G query vectors of one kv head in the registers of a warp.  CUDA cores:
// this lane's elements (packed bf16 pairs with QMIX, else fp32).  Tensor cores:
// mma B fragments (thread t holds head t/4, dims 16k + 2(t%4) + {0,1,8,9}).
template <int D, typename KV, int G, bool QMIX>
struct WarpQ {
  static constexpr bool kMMA = QMIX && G >= 2;
  static constexpr int kElt = static_cast<int>(sizeof(KV));
  static constexpr int kVE = 16 / kElt;
  static constexpr int kEPL = D / 8;
  static constexpr int kNV = kEPL / kVE;
  static constexpr int kQW = QMIX ? kEPL / 2 : kEPL;
  static constexpr int GC = kMMA ? 1 : G;
  static constexpr int NK = D / 16;
  uint32_t qv[GC][kMMA ? 1 : kQW];
  uint32_t qf[kMMA ? NK : 1][2];

  __device__ __forceinline__ static int elem(int u, int j, int w) {
    return u * (128 / kElt) + j * kVE + w;
  }

  // q rows qhead0 .. qhead0+G-1 of [*][D] (bf16 when q_bf16, else fp32).
  __device__ __forceinline__ void load(const void* q, bool q_bf16, size_t qhead0, int lane) {
    if constexpr (kMMA) {
      const int g4 = lane >> 2, tig = lane & 3;
      const uint32_t* q32 =
          reinterpret_cast<const uint32_t*>(q) + (qhead0 + (g4 < G ? g4 : 0)) * (D / 2);
#pragma unroll
      for (int kk = 0; kk < NK; ++kk) {
        qf[kk][0] = g4 < G ? __ldg(q32 + kk * 8 + tig) : 0u;
        qf[kk][1] = g4 < G ? __ldg(q32 + kk * 8 + 4 + tig) : 0u;
      }
    } else {
      const int jl = lane & 7;
#pragma unroll
      for (int h = 0; h < GC; ++h) {
        const size_t qrow = (qhead0 + h) * D;
        if (QMIX) {
          const uint4* q4 =
              reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(q) + qrow);
#pragma unroll
          for (int u = 0; u < kNV; ++u) {
            const uint4 v = __ldg(q4 + u * 8 + jl);
            qv[h][4 * u] = v.x;
            qv[h][4 * u + 1] = v.y;
            qv[h][4 * u + 2] = v.z;
            qv[h][4 * u + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int u = 0; u < kNV; ++u)
#pragma unroll
            for (int w = 0; w < kVE; ++w) {
              const size_t e = qrow + elem(u, jl, w);
              const float x = q_bf16 ? bf16_lo(reinterpret_cast<const uint16_t*>(q)[e])
                                     : reinterpret_cast<const float*>(q)[e];
              qv[h][u * kVE + w] = __float_as_uint(x);
            }
        }
      }
    }
  }
};

// QMIX: q and K are bf16 (mixed-precision FMA, or tensor cores when G >= 2).
// T: rows per tile.  Shared-memory rows are kRowStride bytes apart.
template <int D, typename KV, int G, bool QMIX, int T>
struct WarpAttn {
  static constexpr bool kMMA = QMIX && G >= 2;
  static constexpr int kElt = static_cast<int>(sizeof(KV));
  static constexpr int kRowBytes = D * kElt;
  static constexpr int kVE = 16 / kElt;     // elements per 16-byte vector
  static constexpr int kEPL = D / 8;        // elements of a row per lane
  static constexpr int kNV = kEPL / kVE;    // 16-byte vectors of a row per lane
  static constexpr int kRPL = T / 4;        // rows of a tile per lane
  static constexpr int kRowStride = kRowBytes + (kMMA ? 16 : 0);
  static constexpr int GC = kMMA ? 1 : G;
  static constexpr int NK = D / 16;
  static_assert((T & (T - 1)) == 0 && T <= 32, "tile rows: a power of two <= 32");
  static_assert(!kMMA || T % 16 == 0, "tile rows: whole 16-row mma blocks");

  // Element of a row held in slot w of vector u by lane j of a row group.
  __device__ __forceinline__ static int elem(int u, int j, int w) {
    return u * (128 / kElt) + j * kVE + w;
  }

  using Q = WarpQ<D, KV, G, QMIX>;
  // CUDA cores: per-head state over the lane's rows.  Tensor cores: the state
  // of heads 2(t%4), 2(t%4)+1 for thread t.
  float m_run[GC], l_run[GC], acc[GC][kMMA ? 1 : kEPL];
  float m2[2], l2[2], oacc[kMMA ? NK : 1][4];
  // Tensor cores: P of the tile as mma B fragments per 16-row block (hi rows
  // 0-7, hi rows 8-15, lo rows 0-7, lo rows 8-15), from qk_softmax to pv.
  uint32_t pb[kMMA ? T / 16 : 1][4];

  __device__ __forceinline__ void reset() {
    if constexpr (kMMA) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        m2[j] = -INFINITY;
        l2[j] = 0.f;
      }
#pragma unroll
      for (int mt = 0; mt < NK; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[mt][e] = 0.f;
    } else {
#pragma unroll
      for (int h = 0; h < GC; ++h) {
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
#pragma unroll
        for (int e = 0; e < kEPL; ++e) acc[h][e] = 0.f;
      }
    }
  }

  // Tensor cores, first half of a tile: S = K q^T, the online-softmax update,
  // and P (bf16 hi + lo) as the B fragments of pv.  Reads kt only.
  __device__ __forceinline__ void qk_softmax(const Q& q, const unsigned char* kt, int nrows,
                                             float scale_log2, int lane) {
    static_assert(kMMA, "tensor-core engine");
    const int g4 = lane >> 2;
    constexpr int RB = T / 16;
    float sm[RB][4];
#pragma unroll
    for (int rb = 0; rb < RB; ++rb) {
      // two accumulator chains (even / odd 16-dim slices) halve the
      // dependent mma latency; summed once at the end
      float s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 4; ++e) sm[rb][e] = 0.f;
      const unsigned char* arow =
          kt + (rb * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * kRowStride + 16 * (lane >> 4);
#pragma unroll
      for (int kk = 0; kk < NK; ++kk) {
        uint32_t af[4];
        ldsm_x4(af, arow + 32 * kk);
        if (kk & 1)
          mma_bf16(s2, af, q.qf[kk][0], q.qf[kk][1]);
        else
          mma_bf16(sm[rb], af, q.qf[kk][0], q.qf[kk][1]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sm[rb][e] += s2[e];
    }
    // scale, mask rows past nrows (stale data), online softmax for the
    // thread's two heads (rows spread over the 8 lanes of a column pair)
    float alpha[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float tmax = -INFINITY;
#pragma unroll
      for (int rb = 0; rb < RB; ++rb)
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          const int r = rb * 16 + g4 + 8 * hi;
          float& x = sm[rb][2 * hi + j];
          x = (r < nrows) ? x * scale_log2 : -INFINITY;
          tmax = fmaxf(tmax, x);
        }
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
      const float mnew = fmaxf(m2[j], tmax);
      alpha[j] = exp2f(m2[j] - mnew);
      m2[j] = mnew;
      float psum = 0.f;
#pragma unroll
      for (int rb = 0; rb < RB; ++rb)
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          float& x = sm[rb][2 * hi + j];
          x = exp2f(x - mnew);
          psum += x;
        }
      l2[j] = l2[j] * alpha[j] + psum;
    }
#pragma unroll
    for (int mt = 0; mt < NK; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[mt][e] *= alpha[e & 1];
    // P as bf16 hi + lo, straight into B fragments: an 8x8 block of S (rows =
    // K rows, columns = heads) in accumulator layout, transposed across the
    // warp, is the B fragment (rows 2(t%4), +1 of head t/4)
#pragma unroll
    for (int rb = 0; rb < RB; ++rb) {
      const uint32_t h0 = bf16x2_rn(sm[rb][0], sm[rb][1]);  // rows g4
      const uint32_t h1 = bf16x2_rn(sm[rb][2], sm[rb][3]);  // rows g4 + 8
      const uint32_t l0 = bf16x2_rn(sm[rb][0] - __uint_as_float(h0 << 16),
                                    sm[rb][1] - __uint_as_float(h0 & 0xffff0000u));
      const uint32_t l1 = bf16x2_rn(sm[rb][2] - __uint_as_float(h1 << 16),
                                    sm[rb][3] - __uint_as_float(h1 & 0xffff0000u));
      pb[rb][0] = movmatrix_trans(h0);
      pb[rb][1] = movmatrix_trans(h1);
      pb[rb][2] = movmatrix_trans(l0);
      pb[rb][3] = movmatrix_trans(l1);
    }
  }

  // Tensor cores, second half: O^T += V^T P (P from qk_softmax).  Zeroes V rows
  // past nrows in place (stale shared memory times p = 0 must stay 0).
  __device__ __forceinline__ void pv(unsigned char* vt, int nrows, int lane) {
    static_assert(kMMA, "tensor-core engine");
    constexpr int RB = T / 16;
    // rows past nrows may hold stale shared memory: zero them so 0 * V stays 0
    if (nrows < T) {
      for (int r = nrows; r < T; ++r)
        for (int x = lane * 16; x < kRowBytes; x += 32 * 16)
          *reinterpret_cast<uint4*>(vt + r * kRowStride + x) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncwarp();
#pragma unroll
    for (int kb = 0; kb < RB; ++kb) {
      const uint32_t bh0 = pb[kb][0], bh1 = pb[kb][1], bl0 = pb[kb][2], bl1 = pb[kb][3];
      const unsigned char* vrow =
          vt + (kb * 16 + (lane & 7) + 8 * (lane >> 4)) * kRowStride + 16 * ((lane >> 3) & 1);
#pragma unroll
      for (int mt = 0; mt < NK; ++mt) {
        uint32_t af[4];
        ldsm_x4_trans(af, vrow + 32 * mt);
        mma_bf16(oacc[mt], af, bh0, bh1);
        mma_bf16(oacc[mt], af, bl0, bl1);
      }
    }
  }

  // One tile: rows 0..nrows-1 of kt / vt (kRowStride apart; rows past nrows may
  // hold stale data).  The tensor-core engine zeroes V rows past nrows in place.
  __device__ __forceinline__ void tile(const Q& q, const unsigned char* kt, unsigned char* vt,
                                       int nrows, float scale_log2, int lane) {
    if constexpr (kMMA) {
      qk_softmax(q, kt, nrows, scale_log2, lane);
      pv(vt, nrows, lane);
    } else {
      const int grp = lane >> 3, jl = lane & 7;  // row group, lane in group
      // scores of this lane's rows (rows past nrows hold stale data: masked)
      float sc[G][kRPL];
#pragma unroll
      for (int i = 0; i < kRPL; ++i) {
        const int r = grp + 4 * i;
        uint4 kv[kNV];
#pragma unroll
        for (int u = 0; u < kNV; ++u)
          kv[u] = *reinterpret_cast<const uint4*>(kt + r * kRowStride + 128 * u + 16 * jl);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float d0 = 0.f, d1 = 0.f;
          if (QMIX) {
#pragma unroll
            for (int u = 0; u < kNV; ++u) {
              d0 = fma2_bf16(kv[u].x, q.qv[h][4 * u], d0);
              d1 = fma2_bf16(kv[u].y, q.qv[h][4 * u + 1], d1);
              d0 = fma2_bf16(kv[u].z, q.qv[h][4 * u + 2], d0);
              d1 = fma2_bf16(kv[u].w, q.qv[h][4 * u + 3], d1);
            }
          } else {
#pragma unroll
            for (int u = 0; u < kNV; ++u) {
              float kf[kVE];
              vec_to_f32<KV>(kv[u], kf);
#pragma unroll
              for (int w = 0; w < kVE; w += 2) {
                d0 = fmaf(__uint_as_float(q.qv[h][u * kVE + w]), kf[w], d0);
                d1 = fmaf(__uint_as_float(q.qv[h][u * kVE + w + 1]), kf[w + 1], d1);
              }
            }
          }
          float d = d0 + d1;
          d += __shfl_xor_sync(0xffffffffu, d, 4);
          d += __shfl_xor_sync(0xffffffffu, d, 2);
          d += __shfl_xor_sync(0xffffffffu, d, 1);
          sc[h][i] = (r < nrows) ? d * scale_log2 : -INFINITY;
        }
      }
      // online softmax (log2 domain); the max is over the whole warp's rows
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float tmax = sc[h][0];
#pragma unroll
        for (int i = 1; i < kRPL; ++i) tmax = fmaxf(tmax, sc[h][i]);
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
        const float mnew = fmaxf(m_run[h], tmax);
        const float alpha = exp2f(m_run[h] - mnew);
        float psum = 0.f;
#pragma unroll
        for (int i = 0; i < kRPL; ++i) {
          sc[h][i] = exp2f(sc[h][i] - mnew);
          psum += sc[h][i];
        }
        l_run[h] = l_run[h] * alpha + psum;
#pragma unroll
        for (int e = 0; e < kEPL; ++e) acc[h][e] *= alpha;
        m_run[h] = mnew;
      }
      // acc += p_r v_r over this lane's rows
      auto pv_row = [&](int i) {
        const int r = grp + 4 * i;
#pragma unroll
        for (int u = 0; u < kNV; ++u) {
          const uint4 vv = *reinterpret_cast<const uint4*>(vt + r * kRowStride + 128 * u + 16 * jl);
          float vf[kVE];
          vec_to_f32<KV>(vv, vf);
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int w = 0; w < kVE; ++w)
              acc[h][u * kVE + w] = fmaf(sc[h][i], vf[w], acc[h][u * kVE + w]);
        }
      };
      if (nrows == T) {
#pragma unroll
        for (int i = 0; i < kRPL; ++i) pv_row(i);
      } else {
#pragma unroll
        for (int i = 0; i < kRPL; ++i)
          if (grp + 4 * i < nrows) pv_row(i);
      }
    }
  }

  // The warp's state as G x [acc(D), m, l] floats at mw (shared or global
  // memory): the lanes' partial sums are combined first.
  __device__ __forceinline__ void flush(float* mw, int lane) {
    if constexpr (kMMA) {
      const int g4 = lane >> 2, tig = lane & 3;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float l = l2[j];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        const int h = 2 * tig + j;
        if (h < G) {
#pragma unroll
          for (int mt = 0; mt < NK; ++mt) {
            mw[h * (D + 2) + mt * 16 + g4] = oacc[mt][j];
            mw[h * (D + 2) + mt * 16 + g4 + 8] = oacc[mt][j + 2];
          }
          if (g4 == 0) {
            mw[h * (D + 2) + D] = m2[j];
            mw[h * (D + 2) + D + 1] = l;
          }
        }
      }
    } else {
      const int grp = lane >> 3, jl = lane & 7;
#pragma unroll
      for (int h = 0; h < GC; ++h) {
        float l = l_run[h];
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
#pragma unroll
        for (int e = 0; e < kEPL; ++e) {
          acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], 8);
          acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], 16);
        }
        if (grp == 0) {
#pragma unroll
          for (int u = 0; u < kNV; ++u)
#pragma unroll
            for (int w = 0; w < kVE; ++w) mw[h * (D + 2) + elem(u, jl, w)] = acc[h][u * kVE + w];
        }
        if (lane == 0) {
          mw[h * (D + 2) + D] = m_run[h];
          mw[h * (D + 2) + D + 1] = l;
        }
      }
    }
  }
};

}  // namespace dsa
