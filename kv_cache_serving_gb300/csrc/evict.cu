// evict.cu -- return to the caller the pages of the paged KV cache that no
// later decode step can read.
//
// Under the method's kept set (paper-daily summary of "Understanding and
// Exploiting Diagonal Attention Sparsity in Autoregressive Image Generation",
// section 核心公式: the band/window mask; arXiv abstract: attention on prompt
// and local tokens, the rest of the KV entries skipped), the query at
// i = L-1 and every later one read only prompt rows j < P and rows of their
// window i'-W .. i'.  The window only moves forward, so a row with
// P <= j < i - W is never read again; a page whose 16 rows are all such rows
// can be unmapped and reused (P and W of a request are taken as fixed while it
// decodes).  For a long request this is most of its cache: the resident set
// shrinks from L rows to about P + W + 16.
//
// One thread per (request, page slot of the page table): the test is a range
// check on the page's first and last row.  Freed page ids are appended to the
// caller's list through one atomic per warp (order unspecified).
#include "common.cuh"
#include "internal.h"

namespace dsa {

__global__ void __launch_bounds__(256) evict_kernel(const EvictLaunch a) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  int pg = -1;  // page this thread unmaps, or -1
  if (idx < static_cast<int64_t>(a.batch) * a.max_pages) {
    const int b = static_cast<int>(idx / a.max_pages);
    const int p = static_cast<int>(idx % a.max_pages);
    const int L = a.seq_len[b], P = a.prompt_len[b], W = a.window[b];
    int code = 0;
    if (L < 1 || L > a.max_pages * kPage) code = DSA_DEV_BAD_SEQ_LEN;
    else if (P < 0) code = DSA_DEV_BAD_PROMPT;
    else if (W < 0 || W > a.max_window) code = DSA_DEV_BAD_WINDOW;
    if (code != 0) {
      if (p == 0) set_error(a.err, code);
    } else if (p < (L + kPage - 1) / kPage) {  // a page of the request's rows
      const int first = p * kPage, last = first + kPage - 1, i = L - 1;
      if (first >= P && last < i - W) pg = a.page_table[idx];  // -1: already unmapped
    }
  }
  // one atomic per warp: the lanes with a page take consecutive list slots
  const unsigned want = __ballot_sync(0xffffffffu, pg >= 0);
  if (want == 0) return;
  int base = 0;
  if (lane == __ffs(want) - 1) base = atomicAdd(a.freed_count, __popc(want));
  base = __shfl_sync(0xffffffffu, base, __ffs(want) - 1);
  if (pg < 0) return;
  const int slot = base + __popc(want & ((1u << lane) - 1u));
  if (slot >= a.capacity) {  // no room: the page stays mapped
    set_error(a.err, DSA_DEV_FREE_LIST_FULL);
    return;
  }
  a.freed[slot] = pg;
  a.page_table[idx] = -1;
}

cudaError_t launch_evict(const EvictLaunch& a, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(a.batch) * a.max_pages;
  if (n == 0) return cudaSuccess;
  return launch_pdl(evict_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0,
                    s, a);
}

}  // namespace dsa
