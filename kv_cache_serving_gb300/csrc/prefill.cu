// prefill.cu -- several query tokens per request under the diagonal-aware mask
// (a chunk of prompt or image tokens prefilled, or several image tokens decoded,
// in one step).
//
// Method: the masked softmax of "Understanding and Exploiting Diagonal Attention
// Sparsity in Autoregressive Image Generation" (paper-daily summary, section
// 核心公式 / core formula), applied at every query position of the chunk: the
// last n rows of a request's cache are its query tokens i = L-n .. L-1, and
// query i attends over its own causal kept set -- every prompt row j < P, the
// row i itself, and the window rows i-o (1 <= o <= W) whose mask bit o-1 is
// set (arXiv abstract: entries along the diagonal inside the recent window are
// skipped).  The abstract also reports prefill attention to be diffuse; the
// call serves chunks whose queries share one mask, as decode steps do.
//
// Work decomposition: a unit is (query tile, kv head, request).  A unit holds
// 16 NW (query, head) rows (NW = 2 or 4 warps, the fewest that hold max_q x G)
// -- 16 NW/G consecutive query tokens times the G query heads of one kv head --
// and scans the union of their kept rows: the prompt rows
// [0, min(P, i_last+1)) and the window range [max(., i_first-W), i_last].  A
// 1-D grid runs the first units whole, one CTA each, and the rest split along
// the scanned blocks into parts merged by the unit's last part (plan_split).
// This is a dense contraction (every staged K/V row meets up to 64 query rows),
// so it runs on the tensor cores: each warp owns 16 (query, head) rows, its q
// fragments stay in registers, S = q K^T and O += P V are mma.sync m16n8k16
// (bf16 in, fp32 accumulate), the online softmax runs in the log2 domain, and a
// (query, row) pair the query does not keep is masked to -inf before it.
//
// Staging: blocks of 32 consecutive row positions, K then V, in a ring of
// DSA_MQ_STAGES stages shared by the CTA's warps.  The producer of a block (the
// role rotates: block b is staged by warp b mod NW) fills a stage with one
// bulk async copy per K row and per V row (completing on the stage's "full"
// mbarrier with the expected byte count), the rows' page ids held in its
// registers; every warp arrives on the stage's "empty" mbarrier once its reads
// are done, and the next block's producer refills that stage before it computes
// its own next block.
// A row in the scanned range that no query of the tile keeps is never read:
// its slot is zero-filled instead, so skipped rows have no effect even when
// they hold NaN (0 x NaN would be NaN inside the mma).  Every wait is bounded
// (DSA_DEV_TIMEOUT).
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "mma.cuh"

// Stages of the 2-warp and the 4-warp builds (the 4-warp CTAs are fewer per
// SM, limited by registers, and have shared memory for more stages).
#ifndef DSA_MQ_STAGES
#define DSA_MQ_STAGES 2
#endif
#ifndef DSA_MQ_STAGES4
#define DSA_MQ_STAGES4 4
#endif

namespace dsa {
namespace {

#ifndef DSA_MQ_BLOCK
#define DSA_MQ_BLOCK 32
#endif
constexpr int kMqBlock = DSA_MQ_BLOCK;    // K/V rows per staged block (16 or 32)
static_assert(kMqBlock == 16 || kMqBlock == 32, "block rows");
constexpr int kMqNT = kMqBlock / 8;       // 8-row tiles of S per block
constexpr int kMqHeld = 3;                // page ids every warp holds per lane

template <int D, int NW>
struct MqTiling {
  static constexpr int kRowBytes = D * 2;              // bf16
  static constexpr int kStride = kRowBytes + 16;       // padded: conflict-free ldmatrix
  static constexpr int kStage = 2 * kMqBlock * kStride;  // K rows, then V rows
  static constexpr int kS = NW == 4 ? DSA_MQ_STAGES4 : DSA_MQ_STAGES;
  static constexpr int kBarOff = kS * kStage;          // full[kS], empty[kS]
  static constexpr int kMaskOff = kBarOff + 2 * kS * 8;
  static int smem(int mask_words) { return kMaskOff + mask_words * 4; }
  static_assert(kStage % 128 == 0, "stage alignment");
};

// Two floats as packed bf16 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Any set bit among bits lo..hi (inclusive, 0 <= lo <= hi) of the words at m.
__device__ __forceinline__ bool any_bit(const uint32_t* m, int lo, int hi) {
  for (int w = lo >> 5; w <= (hi >> 5); ++w) {
    uint32_t x = m[w];
    if (w == (lo >> 5)) x &= 0xffffffffu << (lo & 31);
    if (w == (hi >> 5) && (hi & 31) != 31) x &= (2u << (hi & 31)) - 1u;
    if (x != 0u) return true;
  }
  return false;
}

// End of one part of a split unit: its partial state goes to the workspace --
// [16 NW rows][head_dim] unnormalised O, then [16 NW rows][2] (running max in
// the log2 domain, sum) -- and the unit's last part to arrive merges the parts
// as a split softmax does: M = max m_p, l = sum l_p 2^(m_p - M), O = sum O_p
// 2^(m_p - M) / l.  Parts are summed in part order, so the result does not
// depend on which part arrives last.  The arrival counter is back at 0 after
// the merge.
template <int D, int G, int NW>
__device__ __forceinline__ void multi_merge_parts(const MultiLaunch& a, unsigned char* smem,
                                                  int item, int unit,
                                                  int nparts, int b, int hk, int t0, int t1,
                                                  bool warp_active, bool v0, bool v1, int pr0,
                                                  int pr1, const float (&o)[D / 8][4], float m0,
                                                  float m1, float l0, float l1) {
  constexpr int kRows = 16 * NW;
  constexpr int kPartFloats = kRows * (D + 2);
  const int tig = threadIdx.x & 3;
  float* mine = a.part + static_cast<size_t>(item - a.n_whole) * kPartFloats;
  if (warp_active) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int d = 8 * nt + 2 * tig;
      if (v0) *reinterpret_cast<float2*>(mine + pr0 * D + d) = make_float2(o[nt][0], o[nt][1]);
      if (v1) *reinterpret_cast<float2*>(mine + pr1 * D + d) = make_float2(o[nt][2], o[nt][3]);
    }
    if (tig == 0) {
      if (v0) *reinterpret_cast<float2*>(mine + kRows * D + 2 * pr0) = make_float2(m0, l0);
      if (v1) *reinterpret_cast<float2*>(mine + kRows * D + 2 * pr1) = make_float2(m1, l1);
    }
  }
  __threadfence();
  __syncthreads();
  __shared__ int last;
  const int su = unit - a.n_whole;
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(a.part_count + su, 1);
    last = prev == nparts - 1;
    if (last) a.part_count[su] = 0;  // every part has arrived
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  // the stages are free (every block was consumed before the barriers above):
  // weights 2^(m_p - M) [16 NW rows][kMultiMaxParts], then 1/l per row
  float* wsm = reinterpret_cast<float*>(smem);
  const float* ub = a.part + static_cast<size_t>(su) * nparts * kPartFloats;
  const int rows = (t1 - t0) * G;  // row r: query t0 + r / G, head hk G + r % G
  auto qh_of = [&](int r) {
    return (static_cast<size_t>(b) * a.max_q + t0 + r / G) * a.hq + hk * G + r % G;
  };
  if (static_cast<int>(threadIdx.x) < rows) {
    const int r = threadIdx.x;
    float mp[kMultiMaxParts], lp[kMultiMaxParts];
    float mx = -INFINITY;
#pragma unroll
    for (int p = 0; p < kMultiMaxParts; ++p) {
      if (p < nparts) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(ub + p * kPartFloats + kRows * D) + r);
        mp[p] = ml.x;
        lp[p] = ml.y;
        mx = fmaxf(mx, ml.x);
      }
    }
    float lsum = 0.f;
#pragma unroll
    for (int p = 0; p < kMultiMaxParts; ++p) {
      if (p < nparts) {
        const float w = mp[p] == -INFINITY ? 0.f : exp2f(mp[p] - mx);
        wsm[r * kMultiMaxParts + p] = w;
        lsum += lp[p] * w;
      }
    }
    wsm[kRows * kMultiMaxParts + r] = 1.f / lsum;
    if (a.lse != nullptr) a.lse[qh_of(r)] = (mx + log2f(lsum)) * kLn2;
  }
  __syncthreads();
  // O: each thread owns D/8 float4 chunks of the [16 NW][D] tile; one part's
  // chunks are loaded together, so each part costs about one L2 round trip
  constexpr int kPer = D / 8;
  float4 acc[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int p = 0; p < nparts; ++p) {
    const float4* pp = reinterpret_cast<const float4*>(ub + p * kPartFloats);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int c = threadIdx.x + j * NW * 32, r = c / (D / 4);
      if (r < rows) {
        const float4 v = __ldcg(pp + c);
        const float w = wsm[r * kMultiMaxParts + p];
        acc[j].x += v.x * w;
        acc[j].y += v.y * w;
        acc[j].z += v.z * w;
        acc[j].w += v.w * w;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int c = threadIdx.x + j * NW * 32, r = c / (D / 4);
    if (r < rows) {
      const float inv = wsm[kRows * kMultiMaxParts + r];
      float* dst = a.out + qh_of(r) * D + 4 * (c % (D / 4));
      *reinterpret_cast<float2*>(dst) = make_float2(acc[j].x * inv, acc[j].y * inv);
      *reinterpret_cast<float2*>(dst + 2) = make_float2(acc[j].z * inv, acc[j].w * inv);
    }
  }
}

// Resident CTAs per SM the 2-warp and 4-warp builds must allow for (register
// budget: 168 per thread either way, no spills).  With two 17 KB stages, six
// 2-warp CTAs fit an SM: Janus-like 32-token chunk 176 -> 143 us against the
// compiler's own choice (176 registers, smem for 4 CTAs of 3 stages).
#ifndef DSA_MQ_MINB2
#define DSA_MQ_MINB2 6
#endif
#ifndef DSA_MQ_MINB4
#define DSA_MQ_MINB4 3
#endif

template <int D, int G, int NW>
__global__ void __launch_bounds__(NW * 32, NW == 2 ? DSA_MQ_MINB2 : DSA_MQ_MINB4)
    multi_kernel(const MultiLaunch a) {
  using Tl = MqTiling<D, NW>;
  constexpr int kMqWarps = NW;      // warps per CTA, 16 (query, head) rows each
  constexpr int QT = 16 * NW / G;   // query tokens per CTA
  constexpr int NKD = D / 16;       // k-steps of S = q K^T
  constexpr int NTD = D / 8;        // 8-column tiles of O
  constexpr int S = Tl::kS;
  extern __shared__ __align__(128) unsigned char smem[];

  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g4 = lane >> 2, tig = lane & 3;
  // work item -> unit (query tile, kv head, request) and part of the unit
  const int item = blockIdx.x;
  int unit = item, part = 0, nparts = 1;
  if (item >= a.n_whole) {
    const int x = item - a.n_whole;
    unit = a.n_whole + x / a.split;
    part = x % a.split;
    nparts = a.split;
  }
  const int qtile = unit % a.q_tiles, hk = (unit / a.q_tiles) % a.hkv;
  const int bpos = unit / (a.q_tiles * a.hkv);  // position in the request order
  const int b = a.order != nullptr ? __ldg(a.order + bpos) : bpos;
  if (static_cast<unsigned>(b) >= static_cast<unsigned>(a.batch)) {
    if (qtile == 0 && hk == 0 && part == 0 && threadIdx.x == 0) set_error(a.err, DSA_DEV_BAD_ORDER);
    return;
  }
  const int L = a.seq_len[b], n = a.q_len[b], P = a.prompt_len[b], W = a.window[b];
  int code = 0;
  if (L < 1 || L > a.max_pages * kPage) code = DSA_DEV_BAD_SEQ_LEN;
  else if (n < 0 || n > L || n > a.max_q) code = DSA_DEV_BAD_QLEN;
  else if (P < 0) code = DSA_DEV_BAD_PROMPT;
  else if (W < 0 || W > a.max_window) code = DSA_DEV_BAD_WINDOW;
  const int t0 = qtile * QT;
  if (code != 0) {
    // q_len is not trusted: NaN into every slot this unit covers (by part 0)
    if (part != 0) return;
    if (qtile == 0 && hk == 0 && threadIdx.x == 0) set_error(a.err, code);
    for (int x = threadIdx.x; x < QT * G * D; x += kMqWarps * 32) {
      const int t = t0 + x / (G * D);
      if (t >= a.max_q) break;
      const size_t qh = (static_cast<size_t>(b) * a.max_q + t) * a.hq + hk * G + (x / D) % G;
      a.out[qh * D + x % D] = __int_as_float(0x7fc00000);
      if (a.lse != nullptr && x % D == 0) a.lse[qh] = __int_as_float(0x7fc00000);
    }
    return;
  }
  if (t0 >= n) return;
  const int t1 = min(t0 + QT, n);
  const int i_first = L - n + t0, i_last = L - n + t1 - 1;
  // scanned positions: prompt rows [0, nA), then window rows [bstart, i_last]
  const int nA = min(P, i_last + 1);
  const int bstart = max(nA, i_first - W);
  const int R = nA + (i_last >= bstart ? i_last - bstart + 1 : 0);
  // this part's blocks kb0 .. kb0 + nblocks - 1 of the unit's
  const int nb_unit = (R + kMqBlock - 1) / kMqBlock;
  const int kb0 = static_cast<int>(static_cast<int64_t>(nb_unit) * part / nparts);
  const int nblocks = static_cast<int>(static_cast<int64_t>(nb_unit) * (part + 1) / nparts) - kb0;
  auto row_of = [&](int p) { return p < nA ? p : bstart + (p - nA); };

  uint32_t* msk = reinterpret_cast<uint32_t*>(smem + Tl::kMaskOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Tl::kBarOff);
  uint64_t* empty = full + S;
  {
    const uint32_t* mrow = a.keep_mask + (static_cast<size_t>(b) * a.hkv + hk) * a.mask_words;
    for (int x = threadIdx.x; x < a.mask_words; x += kMqWarps * 32) msk[x] = __ldg(mrow + x);
  }
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kMqWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const bf16_t* kg = reinterpret_cast<const bf16_t*>(a.k);
  const bf16_t* vg = reinterpret_cast<const bf16_t*>(a.v);
  const int32_t* pt = a.page_table + static_cast<size_t>(b) * a.max_pages;
  // Page slots of the scanned rows: those of the prompt range, then those of
  // the window range.  Every warp holds up to 32 * kMqHeld of them (lane
  // l: slots l, l + 32, ...), loaded once, so a block's copies wait on no
  // page-table load; longer ranges load their page ids per block.
  const int slotsA = nA > 0 ? ((nA - 1) >> 4) + 1 : 0;
  const int sB0 = bstart >> 4;
  const int nslots = slotsA + (R > nA ? (i_last >> 4) - sB0 + 1 : 0);
  const bool held = nslots <= 32 * kMqHeld;
  int hpg[kMqHeld] = {0, 0, 0};
  if (held) {
#pragma unroll
    for (int h = 0; h < kMqHeld; ++h) {
      const int x = lane + 32 * h;
      if (x < nslots) hpg[h] = __ldg(pt + (x < slotsA ? x : sB0 + (x - slotsA)));
    }
  }

  // The calling warp stages block `blk` into stage s.  32-row blocks: lane l copies the K
  // and V rows of position 32 blk + l; 16-row blocks: lanes 0-15 the K rows and
  // lanes 16-31 the V rows of positions 16 blk + (l % 16).
  auto produce = [&](int blk, int s) {
    const int r = lane & (kMqBlock - 1);
    const int p = blk * kMqBlock + r;
    const int j = p < R ? row_of(p) : 0;
    bool need = false;
    if (p < R) {
      if (j < nA || j >= i_first) {
        need = true;  // a prompt row (query i_last keeps it) or a query's own row
      } else {
        // kept by query i in [i_first, i_last] iff bit (i-j-1) is set, i-j <= W
        const int lo = i_first - j, hi = min(W, i_last - j);
        need = lo <= hi && any_bit(msk, lo - 1, hi - 1);
      }
    }
    unsigned char* kst = smem + s * Tl::kStage;
    unsigned char* vst = kst + kMqBlock * Tl::kStride;
    const unsigned need_mask = __ballot_sync(0xffffffffu, need);
    // page id of this lane's row: from the held ids (every lane takes part)
    int hp = 0;
    if (held) {
      const int x = p < nA ? (j >> 4) : slotsA + ((j >> 4) - sB0);
#pragma unroll
      for (int h = 0; h < kMqHeld; ++h) {
        const int v = __shfl_sync(0xffffffffu, hpg[h], x & 31);
        if ((x >> 5) == h) hp = v;
      }
    }
    constexpr int kCopies = kMqBlock == 32 ? 2 : 1;  // bulk copies per lane
    const bool do_k = kMqBlock == 32 || lane < 16, do_v = kMqBlock == 32 || lane >= 16;
    if (!need) {
      // not read: zeros (finite under p = 0) in the K and V slots of this row
#pragma unroll
      for (int x = 0; x < Tl::kRowBytes; x += 16) {
        if (do_k) *reinterpret_cast<uint4*>(kst + r * Tl::kStride + x) = make_uint4(0u, 0u, 0u, 0u);
        if (do_v) *reinterpret_cast<uint4*>(vst + r * Tl::kStride + x) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    // this warp's earlier generic accesses of the stage before the async writes
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0)
      mbar_arrive_expect_tx(&full[s],
                            static_cast<uint32_t>(__popc(need_mask) * kCopies * Tl::kRowBytes));
    __syncwarp();
    if (need) {
      int pg = held ? hp : __ldg(pt + (j >> 4));
      if (static_cast<unsigned>(pg) >= static_cast<unsigned>(a.num_pages)) {
        set_error(a.err, DSA_DEV_BAD_PAGE);
        pg = 0;
      }
      const size_t off = ((static_cast<size_t>(pg) * kPage + (j & (kPage - 1))) * a.hkv + hk) * D;
      if (do_k) bulk_copy_g2s(kst + r * Tl::kStride, kg + off, Tl::kRowBytes, &full[s]);
      if (do_v) bulk_copy_g2s(vst + r * Tl::kStride, vg + off, Tl::kRowBytes, &full[s]);
    }
  };

  // local block kb is staged by warp producer_of(kb); my_last: the last one this warp staged
  auto producer_of = [&](int kb) { return kb % kMqWarps; };
  int my_last = -1;
  for (int kb = 0; kb < S && kb < nblocks; ++kb)
    if (producer_of(kb) == warp) {
      produce(kb0 + kb, kb);
      my_last = kb;
    }

  // This thread's two (query, head) rows of the warp's 16: r0 = g4, r1 = g4 + 8.
  const int pr0 = warp * 16 + g4, pr1 = pr0 + 8;
  const bool v0 = t0 + pr0 / G < t1, v1 = t0 + pr1 / G < t1;
  const int iq0 = i_first + pr0 / G, iq1 = i_first + pr1 / G;
  const size_t qrow0 = (static_cast<size_t>(b) * a.max_q + t0 + pr0 / G) * a.hq + hk * G + pr0 % G;
  const size_t qrow1 = (static_cast<size_t>(b) * a.max_q + t0 + pr1 / G) * a.hq + hk * G + pr1 % G;
  const bool warp_active = t0 + (warp * 16) / G < t1;
  uint32_t qa[NKD][4];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(a.q);
#pragma unroll
    for (int kk = 0; kk < NKD; ++kk) {
      const int c = (16 * kk + 2 * tig) / 2;  // 32-bit word of the pair
      qa[kk][0] = v0 ? __ldg(q32 + qrow0 * (D / 2) + c) : 0u;
      qa[kk][1] = v1 ? __ldg(q32 + qrow1 * (D / 2) + c) : 0u;
      qa[kk][2] = v0 ? __ldg(q32 + qrow0 * (D / 2) + c + 4) : 0u;
      qa[kk][3] = v1 ? __ldg(q32 + qrow1 * (D / 2) + c + 4) : 0u;
    }
  }
  float o[NTD][4];
#pragma unroll
  for (int nt = 0; nt < NTD; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  // Lane offsets of the ldmatrix rows inside a stage.  K (x4, two 8-row tiles of
  // one 16-dim slice): row np*16 + 8*(lane>>4 & 1) + (lane & 7), bytes
  // 16*(lane>>3 & 1) into the slice.  V (x4 trans, 16 rows x two 8-dim tiles):
  // row 8*(lane>>3 & 1) + (lane & 7), bytes 16*(lane>>4) into the 16-dim slice.
  const uint32_t smem_u32 = smem_addr(smem);
  const uint32_t k_lane_off =
      (((lane >> 4) & 1) * 8 + (lane & 7)) * Tl::kStride + ((lane >> 3) & 1) * 16;
  const uint32_t v_lane_off = (((lane >> 3) & 1) * 8 + (lane & 7)) * Tl::kStride + (lane >> 4) * 16;

  // kept(i, j) for a valid query i and a scanned row j
  auto kept = [&](int i, int j) -> bool {
    if (j > i) return false;
    if (j < P) return true;
    const int off = i - j;
    if (off == 0) return true;
    if (off > W) return false;
    return (msk[(off - 1) >> 5] >> ((off - 1) & 31)) & 1u;
  };
  // Window rows j0 .. j0+31 (consecutive, all >= P) against query i: bit x set
  // iff i keeps row j0 + x, i.e. offset o = o0 - x (o0 = i - j0) is 0, or lies in
  // 1..W with mask bit o-1 set.  E holds offsets lo .. lo+31 (lo = o0 - 31)
  // ascending, so the answer is E bit-reversed.
  auto kept_word = [&](int o0) -> uint32_t {
    const int lo = o0 - 31, sbit = lo - 1;  // mask bit of offset lo
    const int w = sbit >= 0 ? (sbit >> 5) : -((31 - sbit) >> 5);
    const int sh = sbit - 32 * w;
    const uint32_t x0 = (w >= 0 && w < a.mask_words) ? msk[w] : 0u;
    const uint32_t x1 = (w + 1 >= 0 && w + 1 < a.mask_words) ? msk[w + 1] : 0u;
    uint32_t e = __funnelshift_r(x0, x1, sh);
    const int kmin = max(0, 1 - lo), kmax = min(31, W - lo);
    e = kmin > kmax ? 0u
                    : e & (kmax == 31 ? 0xffffffffu : (2u << kmax) - 1u) & (0xffffffffu << kmin);
    if (lo <= 0 && lo >= -31) e |= 1u << (-lo);  // offset 0: the query's own row
    return __brev(e);
  };

  bool failed = false;
  int k = 0;
  for (; k < nblocks; ++k) {
    const int s = k % S;
    // the producer of block k-1+S refills the stage of block k-1 (once every
    // warp is done with it) before computing block k, so that its copies fly
    // during that work
    if (k >= 1 && k - 1 + S < nblocks && producer_of(k - 1 + S) == warp) {
      const int sp = (k - 1) % S;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&empty[sp], static_cast<uint32_t>((k - 1) / S) & 1u))) {
        failed = true;
        break;
      }
      produce(kb0 + k - 1 + S, sp);
      my_last = k - 1 + S;
    }
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>(k / S) & 1u))) {
      failed = true;
      break;
    }
    if (warp_active) {
      // this lane's ldmatrix row addresses in the stage (shared-space, bytes)
      const uint32_t kbase = smem_u32 + s * Tl::kStage + k_lane_off;
      const uint32_t vbase = smem_u32 + s * Tl::kStage + kMqBlock * Tl::kStride + v_lane_off;
      // S = q K^T over the block's rows, 8-row tiles, each summed in two
      // chains (even and odd 16-dim slices) to halve the dependent mma latency
      float sc[kMqNT][4], s2[kMqNT][4];
#pragma unroll
      for (int nt = 0; nt < kMqNT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] = s2[nt][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < NKD; ++kk)
#pragma unroll
        for (int np = 0; np < kMqNT / 2; ++np) {
          uint32_t bf[4];
          ldsm_x4_at(bf, kbase + np * 16 * Tl::kStride + 32 * kk);
          if (kk & 1) {
            mma_bf16(s2[2 * np], qa[kk], bf[0], bf[1]);
            mma_bf16(s2[2 * np + 1], qa[kk], bf[2], bf[3]);
          } else {
            mma_bf16(sc[2 * np], qa[kk], bf[0], bf[1]);
            mma_bf16(sc[2 * np + 1], qa[kk], bf[2], bf[3]);
          }
        }
#pragma unroll
      for (int nt = 0; nt < kMqNT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] += s2[nt][e];
      // scale; mask pairs the query does not keep (and positions past R).  A
      // whole block of prompt rows at or before every query of the tile is kept
      // by all of them.
      const int p0 = (kb0 + k) * kMqBlock;
      if (p0 + kMqBlock <= nA && p0 + kMqBlock - 1 <= i_first) {
#pragma unroll
        for (int nt = 0; nt < kMqNT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            sc[nt][c] = v0 ? sc[nt][c] * a.scale_log2 : -INFINITY;
            sc[nt][2 + c] = v1 ? sc[nt][2 + c] * a.scale_log2 : -INFINITY;
          }
      } else if (p0 >= nA) {
        // a block of window rows: the kept bits of this thread's two queries as
        // words (columns past R are rows after i_last: offsets below 0, unset)
        const int j0 = bstart + (p0 - nA);
        const uint32_t kw0 = v0 ? kept_word(iq0 - j0) : 0u;
        const uint32_t kw1 = v1 ? kept_word(iq1 - j0) : 0u;
#pragma unroll
        for (int nt = 0; nt < kMqNT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int col = nt * 8 + 2 * tig + c;
            sc[nt][c] = (kw0 >> col) & 1u ? sc[nt][c] * a.scale_log2 : -INFINITY;
            sc[nt][2 + c] = (kw1 >> col) & 1u ? sc[nt][2 + c] * a.scale_log2 : -INFINITY;
          }
      } else {
#pragma unroll
        for (int nt = 0; nt < kMqNT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int p = p0 + nt * 8 + 2 * tig + c;
            const int j = row_of(p);
            const bool in = p < R;
            const bool k0 = v0 && in && kept(iq0, j);
            const bool k1 = v1 && in && kept(iq1, j);
            sc[nt][c] = k0 ? sc[nt][c] * a.scale_log2 : -INFINITY;
            sc[nt][2 + c] = k1 ? sc[nt][2 + c] * a.scale_log2 : -INFINITY;
          }
      }
      // online softmax of rows r0 (elements 0, 1) and r1 (elements 2, 3)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < kMqNT; ++nt) {
        mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      // a row with no kept entry yet keeps m = -inf, o = l = 0
      const float al0 = mn0 == -INFINITY ? 1.f : ex2_approx(m0 - mn0);
      const float al1 = mn1 == -INFINITY ? 1.f : ex2_approx(m1 - mn1);
      const float bs0 = mn0 == -INFINITY ? 0.f : mn0, bs1 = mn1 == -INFINITY ? 0.f : mn1;
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < kMqNT; ++nt) {
        sc[nt][0] = ex2_approx(sc[nt][0] - bs0);
        sc[nt][1] = ex2_approx(sc[nt][1] - bs0);
        sc[nt][2] = ex2_approx(sc[nt][2] - bs1);
        sc[nt][3] = ex2_approx(sc[nt][3] - bs1);
        ps0 += sc[nt][0] + sc[nt][1];
        ps1 += sc[nt][2] + sc[nt][3];
      }
      l0 = l0 * al0 + ps0;
      l1 = l1 * al1 + ps1;
      // O is rescaled only when some row's running max moved (else every
      // factor is exactly 1)
      if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int nt = 0; nt < NTD; ++nt) {
          o[nt][0] *= al0;
          o[nt][1] *= al0;
          o[nt][2] *= al1;
          o[nt][3] *= al1;
        }
      }
      // O += P V: P (bf16) straight from the score registers as A fragments
#pragma unroll
      for (int j2 = 0; j2 < kMqBlock / 16; ++j2) {
        uint32_t pa[4];
        pa[0] = pack_bf16(sc[2 * j2][0], sc[2 * j2][1]);
        pa[1] = pack_bf16(sc[2 * j2][2], sc[2 * j2][3]);
        pa[2] = pack_bf16(sc[2 * j2 + 1][0], sc[2 * j2 + 1][1]);
        pa[3] = pack_bf16(sc[2 * j2 + 1][2], sc[2 * j2 + 1][3]);
#pragma unroll
        for (int dp = 0; dp < NTD / 2; ++dp) {
          uint32_t bf[4];
          ldsm_x4_trans_at(bf, vbase + 16 * j2 * Tl::kStride + 32 * dp);
          mma_bf16(o[2 * dp], pa, bf[0], bf[1]);
          mma_bf16(o[2 * dp + 1], pa, bf[2], bf[3]);
        }
      }
    }
    // this warp's reads of the stage are done (the producer orders them before
    // its copies: it acquires the stage through this barrier, then fences)
#ifndef DSA_MQ_CFENCE
#define DSA_MQ_CFENCE 1
#endif
    if (DSA_MQ_CFENCE) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (failed) {
    if (lane == 0) set_error(a.err, DSA_DEV_TIMEOUT);
    // copies this warp issued and nobody waited for: give them a bounded chance to land
    for (int kb = k; kb <= my_last; ++kb)
      if (producer_of(kb) == warp) mbar_wait(&full[kb % S], static_cast<uint32_t>(kb / S) & 1u);
    if (nparts == 1) return;
    // a part still arrives (with an empty state), so the unit's count stays whole
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < NTD; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
  }
  if (nparts > 1) {
    multi_merge_parts<D, G, NW>(a, smem, item, unit, nparts, b, hk, t0, t1, warp_active, v0, v1, pr0,
                                pr1, o, m0, m1, l0, l1);
    return;
  }
  if (!warp_active) return;
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float r0 = 1.f / l0, r1 = 1.f / l1;
#pragma unroll
  for (int nt = 0; nt < NTD; ++nt) {
    const int d = 8 * nt + 2 * tig;
    if (v0) *reinterpret_cast<float2*>(a.out + qrow0 * D + d) = make_float2(o[nt][0] * r0, o[nt][1] * r0);
    if (v1) *reinterpret_cast<float2*>(a.out + qrow1 * D + d) = make_float2(o[nt][2] * r1, o[nt][3] * r1);
  }
  if (a.lse != nullptr && tig == 0) {
    if (v0) a.lse[qrow0] = (m0 + log2f(l0)) * kLn2;
    if (v1) a.lse[qrow1] = (m1 + log2f(l1)) * kLn2;
  }
}

// Most parts of the automatic split.
#ifndef DSA_MQ_MAX_SPLIT
#define DSA_MQ_MAX_SPLIT 4
#endif

// Which units run split, and into how many parts.  Units of equal work fill the
// resident CTA slots in waves, so a last wave of `rem` units leaves most slots
// idle for a whole unit's time: those units are split into up to
// slots / rem parts (and a batch of fewer units than slots into up to
// slots / units parts): at most one wave of parts, which the workspace's
// partials region is sized for; never past its partial rows and counters.
// With a fixed setting n >= 2 every unit the workspace holds is split in n.
void plan_split(MultiLaunch& a, int64_t units, int64_t slots, int rows) {
  a.n_whole = static_cast<int32_t>(units);
  a.split = 1;
  int64_t n_split = 0, parts = 1;
  if (a.split_setting >= 2) {
    parts = a.split_setting;
    n_split = units;
  } else if (a.split_setting == 0 && slots > 0 && units > 0) {
    n_split = units >= slots ? units % slots : units;
    parts = n_split > 0 ? slots / n_split : 1;
    if (parts > DSA_MQ_MAX_SPLIT) parts = DSA_MQ_MAX_SPLIT;
  }
  if (parts < 2 || n_split == 0) return;
  if (n_split > a.count_cap) n_split = a.count_cap;
  if (n_split * parts * rows > a.part_rows_cap) n_split = a.part_rows_cap / (parts * rows);
  if (n_split <= 0) return;
  a.n_whole = static_cast<int32_t>(units - n_split);
  a.split = static_cast<int32_t>(parts);
}

template <int D, int G, int NW>
cudaError_t launch_multi_nw(MultiLaunch a, cudaStream_t s, MultiPlan* plan, bool launch) {
  const int smem = MqTiling<D, NW>::smem(a.mask_words);
  auto kern = multi_kernel<D, G, NW>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, smem);
  if (e != cudaSuccess) return e;
  const int64_t units = static_cast<int64_t>(a.q_tiles) * a.hkv * a.batch;
  plan_split(a, units, static_cast<int64_t>(per_sm) * a.sms, 16 * NW);
  const int64_t items = a.n_whole + (units - a.n_whole) * a.split;
  if (plan != nullptr)
    *plan = MultiPlan{NW, static_cast<int32_t>(units), a.n_whole, a.split, per_sm,
                      static_cast<int32_t>(items)};
  if (!launch) return cudaSuccess;
  return launch_pdl(kern, dim3(static_cast<unsigned>(items)), dim3(NW * 32),
                    static_cast<size_t>(smem), s, a);
}

template <int D, int G>
cudaError_t launch_multi_one(const MultiLaunch& a, cudaStream_t s, MultiPlan* plan, bool launch) {
  return a.warps == 2 ? launch_multi_nw<D, G, 2>(a, s, plan, launch)
                      : launch_multi_nw<D, G, 4>(a, s, plan, launch);
}

}  // namespace

int multi_warps(int max_q, int group) { return static_cast<int64_t>(max_q) * group <= 32 ? 2 : 4; }

int multi_queries_per_cta(int warps, int group) { return 16 * warps / group; }

cudaError_t launch_multi(const MultiLaunch& a, cudaStream_t s, MultiPlan* plan, bool launch) {
  const int g = a.hq / a.hkv;
#define DSA_MQ_CASE(DD, GG) \
  if (a.head_dim == DD && g == GG) return launch_multi_one<DD, GG>(a, s, plan, launch);
  DSA_MQ_CASE(64, 1)
  DSA_MQ_CASE(64, 2)
  DSA_MQ_CASE(64, 4)
  DSA_MQ_CASE(64, 8)
  DSA_MQ_CASE(128, 1)
  DSA_MQ_CASE(128, 2)
  DSA_MQ_CASE(128, 4)
  DSA_MQ_CASE(128, 8)
#undef DSA_MQ_CASE
  return cudaErrorInvalidValue;
}

}  // namespace dsa
