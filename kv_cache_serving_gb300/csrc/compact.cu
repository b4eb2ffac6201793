// compact.cu -- keep mask -> ascending kept-row list (index compaction).
//
// The kept set of the decode query i = L-1 of request b, kv head hk is every
// prompt row j < P, the query row i, and every window row i-o (1 <= o <= W)
// whose mask bit o-1 is set: the band/window mask of "Understanding and
// Exploiting Diagonal Attention Sparsity in Autoregressive Image Generation"
// (paper-daily summary, section 核心公式, and its worked example, section
// 具体技术细节示例), read causally, plus the prompt prefix the arXiv abstract
// reports attention concentrates on.
//
// One warp per (b, hk).  Prompt rows are written as a plain range, window rows
// by window_rows() (ballot + popcount prefix, sorted with no sort).  The last
// CTA also leaves a request schedule in the workspace for the decode.
#include "common.cuh"
#include "internal.h"

namespace dsa {

// Window part of the kept set of decode query i (one warp, all lanes): the
// ascending rows j in max(np, i - W) .. i whose offset o = i - j is 0 or has
// mask bit o - 1 set, np = min(P, L) being the prompt rows kept before them.
// Rows are scanned 32 at a time; a ballot finds the kept lanes and a popcount
// prefix places them, so the list comes out sorted.  Writes the first `cap`
// rows to out[0..] and returns the full count.
__device__ __forceinline__ int window_rows(const uint32_t* mask, int i, int np, int W, int lane,
                                           int32_t* out, int cap) {
  int n = 0;
  if (i < np) return 0;
  const int lo = max(np, i - W);
  for (int base = lo; base <= i; base += 32) {
    const int j = base + lane;
    bool keep = false;
    if (j <= i) {
      const int o = i - j;
      keep = (o == 0) || ((__ldg(mask + ((o - 1) >> 5)) >> ((o - 1) & 31)) & 1u);
    }
    const unsigned ballot = __ballot_sync(0xffffffffu, keep);
    const int pos = n + __popc(ballot & ((1u << lane) - 1u));
    if (keep && pos < cap) out[pos] = j;
    n += __popc(ballot);
  }
  return n;
}

// One warp per (request, kv head); the last CTA to finish also writes the
// request schedule: requests by decreasing total kept rows (ties by index),
// the order in which dsa_decode_sparse hands them to the GPU so that long
// requests do not end up in the tail of the launch.
__global__ void __launch_bounds__(256) compact_kernel(const CompactLaunch a) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (gw < a.batch * a.hkv) {
    const int b = gw / a.hkv;
    const int L = a.seq_len[b], P = a.prompt_len[b], W = a.window[b];
    int code = 0;
    if (L < 1 || L > a.max_pages * kPage) code = DSA_DEV_BAD_SEQ_LEN;
    else if (P < 0) code = DSA_DEV_BAD_PROMPT;
    else if (W < 0 || W > a.max_window) code = DSA_DEV_BAD_WINDOW;
    if (code != 0) {
      if (lane == 0) {
        set_error(a.err, code);
        a.kept_cnt[gw] = 0;
      }
    } else {
      const int i = L - 1;
      const int np = min(P, L);
      int32_t* out = a.kept_idx + static_cast<size_t>(gw) * a.max_kept;
      const uint32_t* mask = a.keep_mask + static_cast<size_t>(gw) * a.mask_words;
      const int cap = a.max_kept;
      for (int j = lane; j < np && j < cap; j += 32) out[j] = j;
      const int n_win = window_rows(mask, i, np, W, lane, out + min(np, cap), max(0, cap - np));
      int n = np + n_win;
      if (lane == 0) {
        if (n > cap) {
          set_error(a.err, DSA_DEV_BAD_COUNT);
          n = 0;
        }
        a.kept_cnt[gw] = n;
      }
    }
  }
  if (a.sched == nullptr || a.batch > kSchedMaxBatch) return;
  // last CTA done: every CTA's counts are visible to it (fence, then count)
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(a.done_count, 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  __shared__ int est[kSchedMaxBatch];
  for (int b = threadIdx.x; b < a.batch; b += blockDim.x) {
    int sum = 0;
    for (int hk = 0; hk < a.hkv; ++hk) sum += __ldcg(a.kept_cnt + static_cast<size_t>(b) * a.hkv + hk);
    est[b] = sum;
  }
  __syncthreads();
  // rank of request b: requests with more rows, or as many and a smaller index
  for (int b = threadIdx.x; b < a.batch; b += blockDim.x) {
    const int e = est[b];
    int rank = 0;
    for (int c = 0; c < a.batch; ++c) rank += (est[c] > e) || (est[c] == e && c < b);
    a.sched[rank] = b;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    *a.sched_tag = kSchedMagic ^ a.batch;
    *a.done_count = 0;
  }
}

cudaError_t launch_compact(const CompactLaunch& a, cudaStream_t s) {
  const int warps = a.batch * a.hkv;
  if (warps == 0) return cudaSuccess;
  return launch_pdl(compact_kernel, dim3((warps + 7) / 8), dim3(256), 0, s, a);
}

}  // namespace dsa
