// decode.cuh -- split-KV flash-decode over a paged KV cache, and the
// log-sum-exp merge of its per-chunk partials.
//
// Method: softmax(q K^T * scale) V of one decode query per (request, head) over
// the rows of the kept set -- the masked attention of "Understanding and
// Exploiting Diagonal Attention Sparsity in Autoregressive Image Generation",
// paper-daily summary, section 核心公式 (core formula), with masked entries
// skipped rather than zeroed (arXiv abstract: KV entries are skipped).
//
// Row sources (template MODE): dense rows 0..L-1; the kept list written by
// dsa_build_index; or the kept set read straight from the keep mask (each lane
// holds one 32-bit word of the window's mask bits and a prefix count, and finds
// the row of a list position by a binary search over the lanes plus a
// rank-select inside the word -- no kept list in memory).
//
// Work decomposition: grid (chunk, kv head, request).  A CTA owns `chunk`
// consecutive entries of the row list of one (request, kv head) and all G query
// heads of that kv head (grouped-query attention shares the rows).  Its NW
// warps take tiles of T rows round-robin.  Each warp runs its own
// shared-memory ring: lanes issue one bulk async copy per K row and per V row
// (the row's page comes from the page table, loaded a tile ahead; the kept
// row two tiles ahead), completing on the stage's mbarrier with the expected
// byte count; compute never waits for anything but its own copies.  Either S
// stages of K and V, or -- for 16-row tensor-core tiles too large for the
// stage size -- one K buffer and one V buffer refilled as soon as their half
// of the tile is computed.  The per-tile arithmetic (CUDA-core or tensor-core
// engine) is WarpAttn (warp_attn.cuh).
//
// End of a CTA: the warps' (m, l, acc) merge in shared memory; the CTA then
// writes the output (one chunk), a partial for merge_kernel (several chunks),
// or -- when the CTAs of a (request, kv head) form a thread-block cluster --
// its state into the first CTA's shared memory for an in-cluster merge.
//
// Builds (warps per CTA, stage bytes, stages) are template parameters: the
// default one, and for the sparse calls with bf16 KV a big-batch build (more
// warps per SM), a small-batch build (one wave of CTAs) and a wide build (one
// 8-warp CTA per unit for batches of at most one unit per SM); the host plan
// picks one per call.
#pragma once

#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "mma.cuh"
#include "warp_attn.cuh"

namespace dsa {

// Build-time tuning knobs: stages per warp, warps per CTA and bytes of K+V per
// stage; the _BIG pair is the build of the fused call for batches of more than
// two waves of units (more, smaller CTAs and tiles: more warps per SM overlap
// the latency of the gathers; tensor-core tiles keep at least 16 rows).
#ifndef DSA_DECODE_WARPS_BIG
#define DSA_DECODE_WARPS_BIG 3
#endif
#ifndef DSA_DECODE_WARPS_BIG_MMA
#define DSA_DECODE_WARPS_BIG_MMA 4
#endif
#ifndef DSA_DECODE_STAGE_BYTES_BIG
#define DSA_DECODE_STAGE_BYTES_BIG 4096
#endif
#ifndef DSA_DECODE_WARPS_SMALL
#define DSA_DECODE_WARPS_SMALL 5
#endif
#ifndef DSA_DECODE_WARPS_WIDE
#define DSA_DECODE_WARPS_WIDE 8
#endif
#ifndef DSA_DECODE_STAGE_BYTES_DENSE
#define DSA_DECODE_STAGE_BYTES_DENSE 4096  // dense rows: long, split into many chunks
#endif
#ifndef DSA_DECODE_STAGE_BYTES
#define DSA_DECODE_STAGE_BYTES 8192
#endif
#ifndef DSA_DECODE_STAGES
#define DSA_DECODE_STAGES 2
#endif
#ifndef DSA_DECODE_WARPS
#define DSA_DECODE_WARPS 4
#endif
// Rows on a stage ring are gathered with 16-byte cp.async copies: 1 for rows of
// 128 bytes, dense rows and the wide build, 2 for every stage ring, 0 never (one
// bulk copy per row).
#ifndef DSA_GATHER_CPASYNC
#define DSA_GATHER_CPASYNC 1
#endif
// Cluster launches (sparse decode split over a thread-block cluster) are also
// programmatic dependents when set.
#ifndef DSA_PDL_CLUSTER
#define DSA_PDL_CLUSTER 1
#endif

template <int D, typename KV, int G, bool MMA = false, int NWARPS = DSA_DECODE_WARPS,
          int STAGE_BYTES = DSA_DECODE_STAGE_BYTES, int STAGES = DSA_DECODE_STAGES>
struct DecodeTiling {
  static constexpr int kElt = static_cast<int>(sizeof(KV));
  static constexpr int kRowBytes = D * kElt;
  static constexpr int kT0 = STAGE_BYTES / (2 * kRowBytes);  // K+V of one stage
  static constexpr int kTmin = MMA ? 16 : 8;  // whole 16-row mma blocks
  static constexpr int T = kT0 > 32 ? 32 : (kT0 < kTmin ? kTmin : kT0);
  static constexpr int S = STAGES;             // stages per warp
  static constexpr int NW = NWARPS;            // warps per CTA
  static constexpr int kVE = 16 / kElt;        // elements per 16-byte vector
  static constexpr int kEPL = D / 8;           // elements of a row per lane
  static constexpr int kNV = kEPL / kVE;       // 16-byte vectors of a row per lane
  static constexpr int kRPL = T / 4;           // rows of a tile per lane
  // With tensor cores, shared-memory rows are padded by 16 bytes so that
  // ldmatrix (8 rows at one column) is free of bank conflicts; the CUDA-core
  // loads (8 lanes over 128 contiguous bytes) need no padding.
  static constexpr int kRowStride = kRowBytes + (MMA ? 16 : 0);
  static constexpr int kStageBytes = 2 * T * kRowStride;
  // A 16-row tensor-core tile whose K and V do not fit STAGE_BYTES is staged
  // as one K buffer and one V buffer per warp (each refilled as soon as its
  // half of the tile is computed) instead of S stages of K and V.
  static constexpr bool kSplit = MMA && (2 * 16 * kRowBytes > STAGE_BYTES);
  static constexpr int kBars = kSplit ? 2 : S;  // mbarriers per warp
  static constexpr int kWarpBytes = kSplit ? kStageBytes : S * kStageBytes;
  static constexpr int kBarOff = NW * kWarpBytes;
  static constexpr int kBarEnd = kBarOff + NW * kBars * 8;
  // End-of-CTA state of each warp, G x [acc(D), m, l] floats: at the start of
  // the warp's own ring (idle by then) when it fits, else in a region of its own.
  static constexpr int kSlotBytes = G * (D + 2) * 4;
  static constexpr bool kSlotInRing = kSlotBytes <= kWarpBytes;
  static constexpr int kSlotOff = kBarEnd;
  static constexpr int kSmem = kSlotOff + (kSlotInRing ? 0 : NW * kSlotBytes);
  // a warp's end-of-CTA state [G][D+2] floats reuses the start of its own ring
  // Largest cluster whose merge buffer [cluster][G][D+2] floats fits the rings.
  static constexpr int kClusterFit = NW * kWarpBytes / (G * (D + 2) * 4);
  static constexpr int kMaxClusterHere = kClusterFit >= 8 ? 8 : kClusterFit >= 4 ? 4
                                         : kClusterFit >= 2 ? 2 : 1;
  static_assert(kStageBytes % 128 == 0, "stage alignment");
  // lane l serves row l % T of a tile: T must be a power of two of at most 32,
  // and a multiple of the 16-row mma blocks on the tensor-core path
  static_assert((T & (T - 1)) == 0 && T <= 32, "tile rows: a power of two <= 32");
  static_assert(!MMA || T % 16 == 0, "tile rows: whole 16-row mma blocks");
  static_assert(kEPL % kVE == 0 && kRowBytes % 128 == 0, "row vector layout");
  // Element of a row held in slot w of vector u by lane j of a row group.
  __device__ __forceinline__ static int elem(int u, int j, int w) {
    return u * (128 / kElt) + j * kVE + w;
  }
};

// Rows of the work list of (b, hk), or a negative device error code.  Shared
// by the decode and merge kernels so that both take the same decision.
// Row sources of the decode kernel (the launch modes of internal.h).
constexpr int kRowsDense = kModeDense;  // rows 0..L-1
constexpr int kRowsList = kModeList;    // the kept list written by dsa_build_index
constexpr int kRowsMask = kModeMask;    // the kept set built in the kernel from the mask

// Position (0..31) of the set bit of rank r (0-based, ascending) in w; any
// value in 0..31 when w has no such bit.
__device__ __forceinline__ int select_bit(unsigned w, int r) {
  int pos = 0, c = __popc(w & 0xffffu);
  if (r >= c) { r -= c; w >>= 16; pos += 16; }
  c = __popc(w & 0xffu);
  if (r >= c) { r -= c; w >>= 8; pos += 8; }
  c = __popc(w & 0xfu);
  if (r >= c) { r -= c; w >>= 4; pos += 4; }
  c = __popc(w & 0x3u);
  if (r >= c) { r -= c; w >>= 2; pos += 2; }
  if (r >= static_cast<int>(w & 1u)) pos += 1;
  return pos;
}

template <int MODE>
__device__ __forceinline__ int request_rows(const DecodeLaunch& a, int b, int hk, int L) {
  if (L < 1 || L > a.max_pages * kPage) return -DSA_DEV_BAD_SEQ_LEN;
  if (MODE == kRowsDense) return L;
  // kRowsMask: the count the decode CTAs of this unit recorded in the workspace
  const int n = MODE == kRowsList ? a.kept_cnt[static_cast<size_t>(b) * a.hkv + hk]
                                  : a.unit_rows[static_cast<size_t>(b) * a.hkv + hk];
  if (MODE == kRowsMask && n < 0) return n;
  if (n < 1 || n > a.max_kept || n > L) return -DSA_DEV_BAD_COUNT;
  return n;
}

// QMIX: q and K are bf16 and the dot products use the mixed-precision FMA.
#ifndef DSA_DECODE_SPLIT_MIN_CTAS
#define DSA_DECODE_SPLIT_MIN_CTAS 5
#endif
// Resident CTAs per SM the compiler must allow for (register budget): the
// split-staged builds are small enough in shared memory for several; 0 leaves
// the other builds to the compiler's own register choice.
template <int D, typename KV, int G, bool QMIX, int NWARPS, int STAGE_BYTES, int STAGES>
constexpr int decode_min_ctas() {
  return DecodeTiling<D, KV, G, QMIX && G >= 2, NWARPS, STAGE_BYTES, STAGES>::kSplit
             ? DSA_DECODE_SPLIT_MIN_CTAS
             : 0;
}

template <int D, typename KV, int G, int MODE, bool QMIX, int NWARPS = DSA_DECODE_WARPS,
          int STAGE_BYTES = DSA_DECODE_STAGE_BYTES, int STAGES = DSA_DECODE_STAGES>
__global__ void __launch_bounds__(NWARPS * 32,
                                  (decode_min_ctas<D, KV, G, QMIX, NWARPS, STAGE_BYTES, STAGES>()))
    decode_kernel(const DecodeLaunch a) {
  using Tl = DecodeTiling<D, KV, G, QMIX && G >= 2, NWARPS, STAGE_BYTES, STAGES>;
  constexpr int T = Tl::T, S = Tl::S, NW = Tl::NW;
  constexpr int kRowBytes = Tl::kRowBytes;
  extern __shared__ __align__(128) unsigned char smem[];

  // Launched as a programmatic dependent: the CTAs may be scheduled while the
  // previous kernel on the stream drains, but touch no memory before it has
  // completed; the next launch may then be scheduled the same way.
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x, hk = blockIdx.y;
  int b = a.order != nullptr ? __ldg(a.order + blockIdx.z) : static_cast<int>(blockIdx.z);
  if (MODE == kRowsList && a.sched != nullptr) {
    // the schedule dsa_build_index left, when it was written for this batch size
    const int tag = a.sched_tag[0], sb = a.sched[blockIdx.z];
    if (tag == a.sched_expect) b = sb;
  }
  if (static_cast<unsigned>(b) >= static_cast<unsigned>(a.batch)) {
    if (c == 0 && hk == 0 && threadIdx.x == 0) set_error(a.err, DSA_DEV_BAD_ORDER);
    return;
  }
  const int L = a.seq_len[b];
  // Page ids of this lane's rows in the warp's first S+1 tiles, loaded
  // speculatively with the request's sizes (they need only b and the CTA's
  // first row): a row that is its own kept index -- every dense row, and the
  // prompt rows of a kept set, and of a kept list outside the split-staged
  // builds (the ids are used only where the loaded kept index equals the row;
  // on the split-staged build the kept-list step measured slower with them) --
  // then needs no dependent page-table load before its first copy.
  constexpr bool kSpec = MODE != kRowsList || !Tl::kSplit;
  const int spec_row0 = a.cluster > 1 ? (c == 0 ? 0 : -1) : c * a.chunk;
  int spec_pg[Tl::S + 1];
#pragma unroll
  for (int t = 0; t <= Tl::S; ++t) {
    const int r = spec_row0 + (warp + t * Tl::NW) * Tl::T + (lane & (Tl::T - 1));
    spec_pg[t] = (kSpec && spec_row0 >= 0 && (r >> 4) < a.max_pages)
                     ? __ldg(a.page_table + static_cast<size_t>(b) * a.max_pages + (r >> 4))
                     : 0;
  }
  // kRowsMask: the kept set is read straight from the keep mask.  Lane l holds
  // the bits of window offsets 32l+1 .. 32l+32 that lie in 1..omax (wbits) and
  // the inclusive prefix count of set bits over lanes 0..l (wincl).
  int n, np = 0, wq = 0, wcnt = 0;
  unsigned wbits = 0;
  int wincl = 0;
  if constexpr (MODE == kRowsMask) {
    const uint32_t* mrow = a.keep_mask + (static_cast<size_t>(b) * a.hkv + hk) * a.mask_words;
    const unsigned raw = lane < a.mask_words ? __ldg(mrow + lane) : 0u;  // issued with the sizes
    const int P = a.prompt_len[b], W = a.window[b];
    int code = 0;
    if (L < 1 || L > a.max_pages * kPage) code = DSA_DEV_BAD_SEQ_LEN;
    else if (P < 0) code = DSA_DEV_BAD_PROMPT;
    else if (W < 0 || W > a.max_window) code = DSA_DEV_BAD_WINDOW;
    if (code == 0) {
      np = min(P, L);
      wq = L - 1;
      // window rows j = i-o, o = omax..0 (ascending j); none when the query is a prompt row
      const int omax = wq >= np ? min(wq - np, W) : -1;
      const int vb = min(max(omax - 32 * lane, 0), 32);
      wbits = vb == 0 ? 0u : raw & (vb == 32 ? 0xffffffffu : (1u << vb) - 1u);
      wincl = __popc(wbits);
#pragma unroll
      for (int s = 1; s < 32; s <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, wincl, s);
        if (lane >= s) wincl += v;
      }
      wcnt = __shfl_sync(0xffffffffu, wincl, 31);
      n = np + (omax >= 0 ? wcnt + 1 : 0);
      if (n > a.max_kept) n = -DSA_DEV_BAD_COUNT;
    } else {
      n = -code;
    }
    if (c == 0 && threadIdx.x == 0) a.unit_rows[static_cast<size_t>(b) * a.hkv + hk] = n;
  } else {
    n = request_rows<MODE>(a, b, hk, L);
  }
  if (n < 0) {
    if (c == 0) {
      if (threadIdx.x == 0) set_error(a.err, -n);
      for (int x = threadIdx.x; x < G * D; x += NW * 32) {
        const size_t qh = static_cast<size_t>(b) * a.hq + hk * G + x / D;
        a.out[qh * D + x % D] = __int_as_float(0x7fc00000);
        if (a.lse != nullptr && x % D == 0) a.lse[qh] = __int_as_float(0x7fc00000);
      }
    }
    return;
  }
  // Append: row L-1 (the query token) comes from k_new / v_new; the first CTA
  // of the unit also stores it into its page slot for later steps.  No CTA of
  // this launch reads that slot, so the store needs no ordering with the copies.
  const KV* knew = a.k_new != nullptr
                       ? reinterpret_cast<const KV*>(a.k_new) + (static_cast<size_t>(b) * a.hkv + hk) * D
                       : nullptr;
  const KV* vnew = a.v_new != nullptr
                       ? reinterpret_cast<const KV*>(a.v_new) + (static_cast<size_t>(b) * a.hkv + hk) * D
                       : nullptr;
  if (knew != nullptr && c == 0 && warp == 0) {
    int pg = __ldg(a.page_table + static_cast<size_t>(b) * a.max_pages + ((L - 1) >> 4));
    if (static_cast<unsigned>(pg) >= static_cast<unsigned>(a.num_pages)) {
      if (lane == 0) set_error(a.err, DSA_DEV_BAD_PAGE);
    } else {
      const size_t off = ((static_cast<size_t>(pg) * kPage + ((L - 1) & (kPage - 1))) * a.hkv + hk) * D;
      constexpr int kVec = Tl::kRowBytes / 16;  // 16-byte vectors per row
      uint4* kd = reinterpret_cast<uint4*>(const_cast<void*>(a.k)) + off * sizeof(KV) / 16;
      uint4* vd = reinterpret_cast<uint4*>(const_cast<void*>(a.v)) + off * sizeof(KV) / 16;
      for (int v = lane; v < 2 * kVec; v += 32) {
        if (v < kVec) kd[v] = __ldg(reinterpret_cast<const uint4*>(knew) + v);
        else vd[v - kVec] = __ldg(reinterpret_cast<const uint4*>(vnew) + v - kVec);
      }
    }
  }
  // Rows of this CTA.  Cluster mode: the a.cluster CTAs of a cluster split the
  // unit's rows evenly (tile-aligned) and every one of them reaches the cluster
  // merge, rows or not.  Otherwise: fixed chunks, partials merged by merge_kernel.
  const int ncl = a.cluster;
  int row0, row1, nchunks;
  if (ncl > 1) {
    const int per = ((n + ncl - 1) / ncl + T - 1) / T * T;
    row0 = min(n, c * per);
    row1 = min(n, row0 + per);
    nchunks = 1;
  } else {
    row0 = c * a.chunk;
    if (row0 >= n) return;
    row1 = min(n, row0 + a.chunk);
    nchunks = (n + a.chunk - 1) / a.chunk;
  }
  const int ntiles = (row1 - row0 + T - 1) / T;

  constexpr int kRowStride = Tl::kRowStride;
  constexpr bool kSplit = Tl::kSplit;
  unsigned char* kst = smem + warp * Tl::kWarpBytes;  // [S][T] K rows, kRowStride apart
  unsigned char* vst = kst + (kSplit ? 1 : S) * T * kRowStride;  // [S][T] V rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tl::kBarOff) + warp * Tl::kBars;
  // end-of-CTA state of warp w: [G][D+2] floats at the start of w's ring
  auto mslot = [&](int w) {
    return reinterpret_cast<float*>(
        smem + (Tl::kSlotInRing ? w * Tl::kWarpBytes : Tl::kSlotOff + w * Tl::kSlotBytes));
  };

  // Stage rings gathered with 16-byte cp.async copies (kRowBytes/16 lanes per
  // row) instead of one bulk copy per row: rows of 128 bytes (a bulk copy of that
  // size streams far below the HBM rate), dense rows and the wide build (both
  // measured faster); the stage barrier then counts one arrival per lane
  // instead of transaction bytes.
  constexpr bool kWideBuild = NWARPS == DSA_DECODE_WARPS_WIDE && STAGES == 1;
  constexpr bool kCpa =
      !kSplit && (DSA_GATHER_CPASYNC == 2 ||
                  (DSA_GATHER_CPASYNC == 1 &&
                   (kRowBytes == 128 || MODE == kRowsDense || kWideBuild)));
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < Tl::kBars; ++s) mbar_init(&bars[s], kCpa ? 32 : 1);
    fence_mbar_init();
  }
  __syncwarp();

  const KV* kg = reinterpret_cast<const KV*>(a.k);
  const KV* vg = reinterpret_cast<const KV*>(a.v);
  const int32_t* idx = MODE == kRowsList
                           ? a.kept_idx + (static_cast<size_t>(b) * a.hkv + hk) * a.max_kept
                           : nullptr;
  const int32_t* pt = a.page_table + static_cast<size_t>(b) * a.max_pages;

  const int my_tiles = warp < ntiles ? (ntiles - warp + NW - 1) / NW : 0;

  // Row addresses are produced by a software pipeline so that no copy waits on
  // the dependent loads kept index -> page id: the kept index of a tile is
  // loaded two tiles before its copy is issued, its page id one tile before.
  // Lane l serves row l % T of a tile: lanes [0,T) copy K rows, [T,2T) V rows
  // (with T = 32 every lane copies both).
  const int my_r = lane & (T - 1);
  auto tile_r0 = [&](int t) { return row0 + (warp + t * NW) * T; };
  auto tile_rows = [&](int t) { return min(T, row1 - tile_r0(t)); };
  // kRowsMask: row at position p of the ascending window rows (all lanes take
  // part; p outside 0..wcnt gives an unused value).  Position wcnt is the query
  // row; position p < wcnt is offset rank q = wcnt-1-p in ascending offset
  // order, found by a binary search over the lanes' prefix counts, then the
  // rank within that lane's word.
  auto window_row = [&](int p) -> int {
    const int q = wcnt - 1 - p;
    int w = 0;
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1)
      if (__shfl_sync(0xffffffffu, wincl, w + s - 1) <= q) w += s;
    const unsigned word = __shfl_sync(0xffffffffu, wbits, w);
    const int below = __shfl_sync(0xffffffffu, wincl, w) - __popc(word);
    return q < 0 ? wq : wq - (32 * w + select_bit(word, q - below) + 1);
  };
  auto load_j = [&](int t) -> int {
    if (t >= my_tiles) return 0;
    const int r = tile_r0(t) + my_r;
    if constexpr (MODE == kRowsMask) {
      if (tile_r0(t) + tile_rows(t) > np) {  // warp-uniform: the tile reaches window rows
        const int jw = window_row(r - np);
        return my_r >= tile_rows(t) ? 0 : (r < np ? r : jw);
      }
    }
    if (my_r >= tile_rows(t)) return 0;
    if constexpr (MODE == kRowsList) return __ldg(idx + r);
    return r;
  };
  auto load_pg = [&](int t, int& j) -> int {
    if (t >= my_tiles || my_r >= tile_rows(t)) return 0;
    if (static_cast<unsigned>(j) >= static_cast<unsigned>(L)) {
      set_error(a.err, DSA_DEV_BAD_INDEX);
      j = 0;
    }
    return __ldg(pt + (j >> 4));
  };
  // Enqueue the bulk copies of local tile t (rows of global tile warp + t*NW).
  auto issue = [&](int t, int stage, int j, int pg) {
    const int nrows = tile_rows(t);
    if constexpr (kCpa) {
      // global row of this lane's row (page * 16 + slot), -2 for the appended row
      int rg = 0;
      if (my_r < nrows) {
        if (static_cast<unsigned>(pg) >= static_cast<unsigned>(a.num_pages)) {
          set_error(a.err, DSA_DEV_BAD_PAGE);
          pg = 0;
        }
        rg = (knew != nullptr && j == L - 1) ? -2 : pg * kPage + (j & (kPage - 1));
      }
      // kLpr lanes per row (16 bytes each), kRpg rows per 32-lane group
      constexpr int kLpr = kRowBytes / 16, kRpg = 32 / kLpr;
      const int rq = lane / kLpr, c16 = (lane % kLpr) * 16;
#pragma unroll
      for (int g = 0; g < T / kRpg; ++g) {
        const int r = kRpg * g + rq;
        const int src_rg = __shfl_sync(0xffffffffu, rg, r);
        if (r < nrows) {
          const size_t dst = (static_cast<size_t>(stage) * T + r) * kRowStride + c16;
          const KV* ks = src_rg == -2 ? knew : kg + (static_cast<size_t>(src_rg) * a.hkv + hk) * D;
          const KV* vs = src_rg == -2 ? vnew : vg + (static_cast<size_t>(src_rg) * a.hkv + hk) * D;
          cp_async16(kst + dst, reinterpret_cast<const unsigned char*>(ks) + c16);
          cp_async16(vst + dst, reinterpret_cast<const unsigned char*>(vs) + c16);
        }
      }
      cp_async_arrive(&bars[stage]);
      return;
    }
    if (lane == 0) mbar_arrive_expect_tx(&bars[stage], static_cast<uint32_t>(nrows * 2 * kRowBytes));
    __syncwarp();
    if (my_r < nrows && (T == 32 || lane < 2 * T)) {
      if (static_cast<unsigned>(pg) >= static_cast<unsigned>(a.num_pages)) {
        set_error(a.err, DSA_DEV_BAD_PAGE);
        pg = 0;
      }
      const size_t off = ((static_cast<size_t>(pg) * kPage + (j & (kPage - 1))) * a.hkv + hk) * D;
      const size_t dst = (static_cast<size_t>(stage) * T + my_r) * kRowStride;
      const bool fresh = knew != nullptr && j == L - 1;  // the appended row
      if (T == 32 || lane < T)
        bulk_copy_g2s(kst + dst, fresh ? knew : kg + off, kRowBytes, &bars[stage]);
      if (T == 32 || lane >= T)
        bulk_copy_g2s(vst + dst, fresh ? vnew : vg + off, kRowBytes, &bars[stage]);
    }
  };

  // Split staging: the K (half 0) or V (half 1) rows of local tile t into
  // their buffer, completing on bars[half]; lanes [0,T) copy one row each.
  auto issue_half = [&](int t, int half, int j, int pg) {
    const int nrows = tile_rows(t);
    if (lane == 0) mbar_arrive_expect_tx(&bars[half], static_cast<uint32_t>(nrows * kRowBytes));
    __syncwarp();
    if (my_r < nrows && lane < T) {
      if (static_cast<unsigned>(pg) >= static_cast<unsigned>(a.num_pages)) {
        set_error(a.err, DSA_DEV_BAD_PAGE);
        pg = 0;
      }
      const size_t off = ((static_cast<size_t>(pg) * kPage + (j & (kPage - 1))) * a.hkv + hk) * D;
      const bool fresh = knew != nullptr && j == L - 1;  // the appended row
      const KV* src = half == 0 ? (fresh ? knew : kg + off) : (fresh ? vnew : vg + off);
      bulk_copy_g2s((half == 0 ? kst : vst) + static_cast<size_t>(my_r) * kRowStride, src,
                    kRowBytes, &bars[half]);
    }
  };

  WarpAttn<D, KV, G, QMIX, T> wa;
  static_assert(WarpAttn<D, KV, G, QMIX, T>::kRowStride == Tl::kRowStride, "row stride");
  typename WarpAttn<D, KV, G, QMIX, T>::Q wq_;
  wq_.load(a.q, a.q_bf16 != 0, static_cast<size_t>(b) * a.hq + hk * G, lane);
  wa.reset();

  // prologue: kept indices of tiles 0..S+1, page ids of tiles 0..S, copies of
  // tiles 0..S-1 (two dependent round trips in all)
  int jr[S + 2], pr[S + 1];
#pragma unroll
  for (int t = 0; t < S + 2; ++t) jr[t] = load_j(t);
#pragma unroll
  for (int t = 0; t < S + 1; ++t) {
    const int rr = tile_r0(t) + my_r;
    if (kSpec && row0 == spec_row0 && jr[t] == rr)
      pr[t] = (t < my_tiles && my_r < tile_rows(t)) ? spec_pg[t] : 0;
    else
      pr[t] = load_pg(t, jr[t]);
  }
  int failed_at = -1;
  if constexpr (kSplit) {
    // K and V of tile 0 in flight; then per tile: QK^T + softmax on K(t),
    // refill the K buffer with tile t+1, PV on V(t), refill the V buffer
    if (my_tiles > 0) {
      issue_half(0, 0, jr[0], pr[0]);
      issue_half(0, 1, jr[0], pr[0]);
    }
    int ja = jr[1], pa = pr[1], jb = jr[2];  // addresses of tiles 1 and 2
    bool failed_on_v = false;
    for (int t = 0; t < my_tiles; ++t) {
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[0], static_cast<uint32_t>(t) & 1u))) {
        failed_at = t;
        break;
      }
      const int nrows = min(T, row1 - (row0 + (warp + t * NW) * T));
      wa.qk_softmax(wq_, kst, nrows, a.scale_log2, lane);
      __syncwarp();
      fence_proxy_async_smem();
      if (t + 1 < my_tiles) issue_half(t + 1, 0, ja, pa);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[1], static_cast<uint32_t>(t) & 1u))) {
        failed_at = t;
        failed_on_v = true;
        break;
      }
      wa.pv(vst, nrows, lane);
      __syncwarp();
      fence_proxy_async_smem();
      if (t + 1 < my_tiles) issue_half(t + 1, 1, ja, pa);
      ja = jb;
      pa = load_pg(t + 2, ja);
      jb = load_j(t + 3);
    }
    if (failed_at >= 0) {
      // Give the copies still in flight a bounded chance to land before exiting.
      if (lane == 0) set_error(a.err, DSA_DEV_TIMEOUT);
      // in flight: V of the failed tile, and K of it (failed on K) or of the next
      mbar_wait(&bars[1], static_cast<uint32_t>(failed_at) & 1u);
      if (!failed_on_v) mbar_wait(&bars[0], static_cast<uint32_t>(failed_at) & 1u);
      else if (failed_at + 1 < my_tiles)
        mbar_wait(&bars[0], static_cast<uint32_t>(failed_at + 1) & 1u);
    }
  } else {
#pragma unroll
  for (int t = 0; t < S; ++t)
    if (t < my_tiles) issue(t, t, jr[t], pr[t]);
  int j0 = jr[S], pg0 = pr[S], j1 = jr[S + 1];  // next tile to issue: S

  for (int t = 0; t < my_tiles; ++t) {
    const int stage = t % S;
    if (!__all_sync(0xffffffffu, mbar_wait(&bars[stage], static_cast<uint32_t>(t / S) & 1u))) {
      failed_at = t;  // the whole warp leaves together
      break;
    }
    const int nrows = min(T, row1 - (row0 + (warp + t * NW) * T));
    const unsigned char* kt = kst + static_cast<size_t>(stage) * T * kRowStride;
    unsigned char* vt = vst + static_cast<size_t>(stage) * T * kRowStride;

    wa.tile(wq_, kt, vt, nrows, a.scale_log2, lane);
    __syncwarp();
    fence_proxy_async_smem();
    if (t + S < my_tiles) issue(t + S, stage, j0, pg0);
    // advance the address pipeline: page id of tile t+S+1, kept index of t+S+2
    j0 = j1;
    pg0 = load_pg(t + S + 1, j0);
    j1 = load_j(t + S + 2);
  }
  if (failed_at >= 0) {
    // Give the copies still in flight a bounded chance to land before exiting.
    if (lane == 0) set_error(a.err, DSA_DEV_TIMEOUT);
    for (int t = failed_at; t < my_tiles && t < failed_at + S; ++t)
      mbar_wait(&bars[t % S], static_cast<uint32_t>(t / S) & 1u);
  }
  }  // S-stage staging

  // sum the warp's partial states, then merge the warps of this CTA (each
  // warp's ring is idle now: its copies have all landed)
  wa.flush(mslot(warp), lane);
  __syncthreads();
  // CTA merge of the warps' states: item k of this thread is x = tid + k*NW*32
  constexpr int kItems = (G * D + NW * 32 - 1) / (NW * 32);
  float it_o[kItems], it_m[kItems], it_l[kItems];
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int x = threadIdx.x + k * NW * 32;
    it_o[k] = 0.f;
    it_m[k] = -INFINITY;
    it_l[k] = 0.f;
    if (x < G * D) {
      const int h = x / D, d = x % D;
      float mstar = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) mstar = fmaxf(mstar, mslot(w)[h * (D + 2) + D]);
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float* src = mslot(w) + h * (D + 2);
        const float sc = src[D] == -INFINITY ? 0.f : exp2f(src[D] - mstar);
        it_o[k] = fmaf(sc, src[d], it_o[k]);
        it_l[k] = fmaf(sc, src[D + 1], it_l[k]);
      }
      it_m[k] = mstar;
    }
  }
  if (ncl > 1) {
    // Cluster merge through distributed shared memory: once every CTA of the
    // cluster is past its own reads of shared memory, each writes its state
    // into slot `rank` of rank 0's buffer [ncl][G][D+2]; rank 0 combines them.
    const uint32_t rank = cluster_ctarank();
    float* recv = reinterpret_cast<float*>(smem);
    cluster_sync();
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int x = threadIdx.x + k * NW * 32;
      if (x < G * D) {
        const int h = x / D, d = x % D;
        float* slot = recv + (rank * G + h) * (D + 2);
        st_cluster_f32(map_cluster_rank(slot + d, 0), it_o[k]);
        if (d == 0) {
          st_cluster_f32(map_cluster_rank(slot + D, 0), it_m[k]);
          st_cluster_f32(map_cluster_rank(slot + D + 1, 0), it_l[k]);
        }
      }
    }
    cluster_sync();
    if (rank != 0) return;
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int x = threadIdx.x + k * NW * 32;
      if (x < G * D) {
        const int h = x / D, d = x % D;
        float mstar = -INFINITY;
        for (int r = 0; r < ncl; ++r) mstar = fmaxf(mstar, recv[(r * G + h) * (D + 2) + D]);
        float o = 0.f, ls = 0.f;
        for (int r = 0; r < ncl; ++r) {
          const float* src = recv + (r * G + h) * (D + 2);
          const float sc = src[D] == -INFINITY ? 0.f : exp2f(src[D] - mstar);
          o = fmaf(sc, src[d], o);
          ls = fmaf(sc, src[D + 1], ls);
        }
        const size_t qh = static_cast<size_t>(b) * a.hq + hk * G + h;
        a.out[qh * D + d] = o / ls;
        if (a.lse != nullptr && d == 0) a.lse[qh] = (mstar + log2f(ls)) * kLn2;
      }
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int x = threadIdx.x + k * NW * 32;
    if (x < G * D) {
      const int h = x / D, d = x % D;
      const size_t qh = static_cast<size_t>(b) * a.hq + hk * G + h;
      if (nchunks == 1) {
        a.out[qh * D + d] = it_o[k] / it_l[k];
        if (a.lse != nullptr && d == 0) a.lse[qh] = (it_m[k] + log2f(it_l[k])) * kLn2;
      } else {
        float* pp = a.part + (qh * a.num_chunks + c) * (D + 2);
        pp[d] = it_o[k];
        if (d == 0) {
          pp[D] = it_m[k];
          pp[D + 1] = it_l[k];
        }
      }
    }
  }
}

// One warp per (request, query head): combine the chunk partials by
// log-sum-exp.  Heads whose rows fit one chunk were finished by decode_kernel.
template <int D, int MODE>
__global__ void __launch_bounds__(128) merge_kernel(const DecodeLaunch a) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int DPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (gw >= a.batch * a.hq) return;
  const int b = gw / a.hq, qh = gw % a.hq;
  const int hk = qh / (a.hq / a.hkv);
  const int n = request_rows<MODE>(a, b, hk, a.seq_len[b]);
  if (n < 0) return;  // decode_kernel wrote NaN and the error code
  const int nch = (n + a.chunk - 1) / a.chunk;
  if (nch <= 1) return;
  const float* pp = a.part + static_cast<size_t>(gw) * a.num_chunks * (D + 2);
  float mstar = -INFINITY;
  for (int c = lane; c < nch; c += 32) mstar = fmaxf(mstar, pp[c * (D + 2) + D]);
  mstar = warp_max(mstar);
  float o[DPL], ls = 0.f;
#pragma unroll
  for (int e = 0; e < DPL; ++e) o[e] = 0.f;
  for (int c = 0; c < nch; ++c) {
    const float* src = pp + c * (D + 2);
    const float sc = exp2f(src[D] - mstar);
    ls = fmaf(sc, src[D + 1], ls);
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] = fmaf(sc, src[lane * DPL + e], o[e]);
  }
  float* out = a.out + static_cast<size_t>(gw) * D + lane * DPL;
#pragma unroll
  for (int e = 0; e < DPL; ++e) out[e] = o[e] / ls;
  if (a.lse != nullptr && lane == 0) a.lse[gw] = (mstar + log2f(ls)) * kLn2;
}

template <typename KV>
struct IsBf16 {
  static constexpr bool value = false;
};
template <>
struct IsBf16<bf16_t> {
  static constexpr bool value = true;
};

template <int D, typename KV, int G, int MODE, bool QMIX, int NWARPS, int SB, int ST>
cudaError_t launch_decode_one(const DecodeLaunch& a, cudaStream_t s) {
  using Tl = DecodeTiling<D, KV, G, QMIX && G >= 2, NWARPS, SB, ST>;
  auto kern = decode_kernel<D, KV, G, MODE, QMIX, NWARPS, SB, ST>;
  const int smem = Tl::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_chunks, a.hkv, a.batch);
  cfg.blockDim = dim3(Tl::NW * 32);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (a.cluster > 1) {
    // the CTAs of one (request, kv head) form one cluster along x
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(a.cluster);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (a.cluster <= 1 || DSA_PDL_CLUSTER) {
    // programmatic dependent launch: scheduled while the previous kernel drains
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = DSA_PDL;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// Calls f.template operator()<D, G>() for the built (head_dim, group), or
// returns `fallback`.
#define DSA_FOR_SHAPE(HEAD_DIM, GROUP, BODY)      \
  do {                                            \
    const int hd_ = (HEAD_DIM), g_ = (GROUP);     \
    if (hd_ == 64 && g_ == 1) { BODY(64, 1) }     \
    if (hd_ == 64 && g_ == 2) { BODY(64, 2) }     \
    if (hd_ == 64 && g_ == 4) { BODY(64, 4) }     \
    if (hd_ == 64 && g_ == 8) { BODY(64, 8) }     \
    if (hd_ == 128 && g_ == 1) { BODY(128, 1) }   \
    if (hd_ == 128 && g_ == 2) { BODY(128, 2) }   \
    if (hd_ == 128 && g_ == 4) { BODY(128, 4) }   \
    if (hd_ == 128 && g_ == 8) { BODY(128, 8) }   \
  } while (0)

// Stage bytes of the default build of a row mode.
constexpr int default_stage_bytes(int mode) {
  return mode == kRowsDense ? DSA_DECODE_STAGE_BYTES_DENSE : DSA_DECODE_STAGE_BYTES;
}

// The sparse calls with bf16 KV have two builds besides the default one.
// Big-batch build: 4 KB stages and its own warps per CTA (measured best: 3 on
// the CUDA-core engine, 4 with a 5-CTA register budget on the split-staged
// tensor-core engine).  Small-batch build: 5 warps of one 8 KB stage, so that
// a batch that needs two waves of the default build runs in one.
template <typename KV>
constexpr bool has_build(int mode, int build) {
  return build == kBuildDefault || (IsBf16<KV>::value && mode != kRowsDense);
}
template <int G, bool QMIX, int BUILD>
constexpr int build_warps() {
  return BUILD == kBuildBig
             ? ((QMIX && G >= 2) ? DSA_DECODE_WARPS_BIG_MMA : DSA_DECODE_WARPS_BIG)
             : (BUILD == kBuildSmall  ? DSA_DECODE_WARPS_SMALL
                : BUILD == kBuildWide ? DSA_DECODE_WARPS_WIDE
                                      : DSA_DECODE_WARPS);
}
template <int MODE, int BUILD>
constexpr int build_stage_bytes() {
  return BUILD == kBuildBig                             ? DSA_DECODE_STAGE_BYTES_BIG
         : (BUILD == kBuildSmall || BUILD == kBuildWide) ? DSA_DECODE_STAGE_BYTES
                                                         : default_stage_bytes(MODE);
}
template <int BUILD>
constexpr int build_stages() {
  return (BUILD == kBuildSmall || BUILD == kBuildWide) ? 1 : DSA_DECODE_STAGES;
}

template <typename KV, int MODE, int BUILD>
cudaError_t launch_decode_dispatch(const DecodeLaunch& a, cudaStream_t s) {
  const bool qmix = IsBf16<KV>::value && a.q_bf16 != 0;
  constexpr bool kQ = IsBf16<KV>::value;
  constexpr int kSB = build_stage_bytes<MODE, BUILD>(), kST = build_stages<BUILD>();
#define DSA_BODY(DD, GG)                                                                      \
  return qmix ? launch_decode_one<DD, KV, GG, MODE, kQ, build_warps<GG, kQ, BUILD>(), kSB,    \
                                  kST>(a, s)                                                  \
              : launch_decode_one<DD, KV, GG, MODE, false, build_warps<GG, false, BUILD>(),   \
                                  kSB, kST>(a, s);
  DSA_FOR_SHAPE(a.head_dim, a.hq / a.hkv, DSA_BODY);
#undef DSA_BODY
  return cudaErrorInvalidValue;
}

// One row mode in the build the plan asks for (a.build), if there is one.
template <typename KV, int MODE>
cudaError_t launch_decode_mode(const DecodeLaunch& a, cudaStream_t s) {
  if constexpr (has_build<KV>(MODE, kBuildBig))
    if (a.build == kBuildBig) return launch_decode_dispatch<KV, MODE, kBuildBig>(a, s);
  if constexpr (has_build<KV>(MODE, kBuildSmall))
    if (a.build == kBuildSmall) return launch_decode_dispatch<KV, MODE, kBuildSmall>(a, s);
  if constexpr (has_build<KV>(MODE, kBuildWide))
    if (a.build == kBuildWide) return launch_decode_dispatch<KV, MODE, kBuildWide>(a, s);
  return launch_decode_dispatch<KV, MODE, kBuildDefault>(a, s);
}

template <typename KV, int MODE, int BUILD>
DecodeShape decode_shape_m(int head_dim, int group) {
  DecodeShape r{0, 1, 1, DSA_DECODE_WARPS, 0, BUILD};
  constexpr bool kQ = IsBf16<KV>::value;
  constexpr int kSB = build_stage_bytes<MODE, BUILD>(), kST = build_stages<BUILD>();
#define DSA_BODY(DD, GG)                                                                   \
  constexpr int kNW = build_warps<GG, kQ, BUILD>();                                        \
  using Tl = DecodeTiling<DD, KV, GG, kQ && (GG >= 2), kNW, kSB, kST>;                     \
  auto kern = decode_kernel<DD, KV, GG, MODE, kQ, kNW, kSB, kST>;                          \
  r.warps = kNW;                                                                           \
  r.rows_per_pass = Tl::NW * Tl::T;                                                        \
  r.tile_rows = Tl::T;                                                                     \
  r.cluster_limit = Tl::kMaxClusterHere;                                                   \
  int n = 0;                                                                               \
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Tl::kSmem) == \
          cudaSuccess &&                                                                   \
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Tl::NW * 32, Tl::kSmem) ==   \
          cudaSuccess &&                                                                   \
      n > 1)                                                                               \
    r.ctas_per_sm = n;                                                                     \
  return r;
  DSA_FOR_SHAPE(head_dim, group, DSA_BODY);
#undef DSA_BODY
  return r;
}

template <typename KV, int MODE>
DecodeShape decode_shape_mode(int head_dim, int group, int build) {
  if constexpr (has_build<KV>(MODE, kBuildBig))
    if (build == kBuildBig) return decode_shape_m<KV, MODE, kBuildBig>(head_dim, group);
  if constexpr (has_build<KV>(MODE, kBuildSmall))
    if (build == kBuildSmall) return decode_shape_m<KV, MODE, kBuildSmall>(head_dim, group);
  if constexpr (has_build<KV>(MODE, kBuildWide))
    if (build == kBuildWide) return decode_shape_m<KV, MODE, kBuildWide>(head_dim, group);
  return decode_shape_m<KV, MODE, kBuildDefault>(head_dim, group);
}

}  // namespace dsa
