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
// caller's list with an atomic counter (order unspecified).
#include "common.cuh"
#include "internal.h"

namespace dsa {

__global__ void __launch_bounds__(256) evict_kernel(const EvictLaunch a) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(a.batch) * a.max_pages) return;
  const int b = static_cast<int>(idx / a.max_pages);
  const int p = static_cast<int>(idx % a.max_pages);
  const int L = a.seq_len[b], P = a.prompt_len[b], W = a.window[b];
  int code = 0;
  if (L < 1 || L > a.max_pages * kPage) code = DSA_DEV_BAD_SEQ_LEN;
  else if (P < 0) code = DSA_DEV_BAD_PROMPT;
  else if (W < 0 || W > a.max_window) code = DSA_DEV_BAD_WINDOW;
  if (code != 0) {
    if (p == 0) set_error(a.err, code);
    return;
  }
  if (p >= (L + kPage - 1) / kPage) return;  // beyond the request's rows
  const int first = p * kPage, last = first + kPage - 1, i = L - 1;
  if (!(first >= P && last < i - W)) return;  // some row may still be read
  int32_t* entry = a.page_table + idx;
  const int pg = *entry;
  if (pg < 0) return;  // already unmapped
  const int slot = atomicAdd(a.freed_count, 1);
  if (slot >= a.capacity) {  // no room: the page stays mapped
    set_error(a.err, DSA_DEV_FREE_LIST_FULL);
    return;
  }
  a.freed[slot] = pg;
  *entry = -1;
}

cudaError_t launch_evict(const EvictLaunch& a, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(a.batch) * a.max_pages;
  if (n == 0) return cudaSuccess;
  evict_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
