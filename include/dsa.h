/*
 * dsa.h -- C ABI of libdsa: diagonal-aware sparse decode attention over a paged
 * KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The operation is the decode step of the method on the page "Understanding and
 * Exploiting Diagonal Attention Sparsity in Autoregressive Image Generation":
 * for each request, one query token attends only to the prompt-prefix rows of
 * the KV cache and to the rows of a recent window W whose offset is kept by a
 * per-head keep mask (arXiv abstract: "selectively skips KV entries along the
 * diagonal attention direction within a recent window"; paper-daily summary,
 * section 核心公式 / core formula: Attention = softmax(QK^T/sqrt(d) (.) M) V,
 * with the band mask M_ij = 1 iff |i-j| <= B and j >= i-W as one instance).
 *
 * Conventions shared by every call
 * --------------------------------
 * Shapes (row-major, element counts):
 *   q            [batch][hq][head_dim]                 dtype dims->q_dtype
 *   k_pages      [num_pages][16][hkv][head_dim]        dtype dims->kv_dtype
 *   v_pages      [num_pages][16][hkv][head_dim]        dtype dims->kv_dtype
 *   page_table   [batch][max_pages_per_req] int32: row j of request b lives in
 *                page page_table[b][j / 16], slot j % 16.  Entries past
 *                ceil(seq_len[b] / 16) are never read.
 *   seq_len      [batch] int32, L_b >= 1 rows already in the cache; the query
 *                is token i = L_b - 1, whose own K/V row is row i.
 *   prompt_len   [batch] int32, P_b >= 0 prompt rows (always kept).
 *   window       [batch] int32, 0 <= W_b <= max_window.
 *   keep_mask    [batch][hkv][mask_words] uint32: bit (o-1) of the little-endian
 *                bit string keeps window offset o = i - j, 1 <= o <= W_b.
 * Query head h reads KV head h / (hq / hkv) (grouped-query attention).
 * The kept set of (b, kv head hk) is
 *   K(b,hk) = { j < min(P_b, L_b) } U { i } U { i-o : 1 <= o <= W_b, bit o-1 set, i-o >= P_b }
 * in ascending j.  Masked rows are not read and do not enter the softmax.
 *
 * Memory: every pointer is a DEVICE pointer owned by the caller; the library
 * allocates nothing and keeps no pointer after a call returns.  `ws` is a
 * caller-owned device workspace of dsa_workspace_size(dims) bytes, aligned to
 * 256 bytes, zero-filled once before its first use (cudaMemsetAsync), and not
 * shared by calls that may run concurrently.
 *
 * Ordering: every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 * legacy default stream) and returns once its kernels are enqueued.  The
 * kernels are launched as programmatic dependents: a kernel's CTAs may be
 * scheduled while the previous kernel on the stream is still running, but read
 * and write no memory before that kernel has completed, so stream order holds
 * exactly as for plain launches.
 *
 * Errors: calls return a dsa_status and never throw or abort.  Shapes, dtypes,
 * sizes and null pointers are checked on the host before anything is launched
 * (DSA_ERR_INVALID_ARG / DSA_ERR_UNSUPPORTED; nothing is written).  Launch
 * failures give DSA_ERR_CUDA.  Per-request values live on the device, so the
 * kernels check them there: an invalid seq_len / prompt_len / window / kept
 * count, a kept index outside 0..i, or a page id outside 0..num_pages-1 sets
 * the workspace's error word (first error wins), no memory outside the
 * caller's buffers is touched, and the outputs of the affected request are
 * unspecified (NaN where the request itself is invalid).
 * dsa_get_device_error() reads the word.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1, /* null pointer, bad size or inconsistent dims      */
  DSA_ERR_UNSUPPORTED = 2, /* dtype, head_dim, page size or group not built    */
  DSA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed             */
  DSA_ERR_DEVICE = 4,      /* the kernels flagged invalid per-request data     */
  DSA_ERR_TIMEOUT = 5,     /* a bounded on-device wait gave up                 */
  DSA_ERR_SCRATCH_LIMIT = 6 /* the problem needs more than the fixed scratch of
                               dsa_decode_sparse_noalloc                        */
} dsa_status;

typedef enum { DSA_F32 = 0, DSA_BF16 = 1 } dsa_dtype;

/* Device error codes stored in the workspace error word. */
enum {
  DSA_DEV_OK = 0,
  DSA_DEV_BAD_SEQ_LEN = 1,  /* seq_len < 1 or > max_pages_per_req * 16     */
  DSA_DEV_BAD_PROMPT = 2,   /* prompt_len < 0                              */
  DSA_DEV_BAD_WINDOW = 3,   /* window < 0 or > max_window                  */
  DSA_DEV_BAD_PAGE = 4,     /* page id outside 0..num_pages-1              */
  DSA_DEV_BAD_INDEX = 5,    /* kept index outside 0..seq_len-1             */
  DSA_DEV_BAD_COUNT = 6,    /* kept count < 1 or > max_kept                */
  DSA_DEV_TIMEOUT = 7,      /* a bounded wait for an async copy gave up    */
  DSA_DEV_BAD_GRID_W = 8,   /* grid width < 1 (attention mass)             */
  DSA_DEV_BAD_ORDER = 9,    /* request_order entry outside 0..batch-1      */
  DSA_DEV_FREE_LIST_FULL = 10, /* dsa_evict_pages: more pages than capacity  */
  DSA_DEV_BAD_QLEN = 11     /* dsa_prefill_sparse: q_len < 0 or above
                               min(seq_len, max_q)                          */
};

/* Problem sizes, shared by all calls on one KV cache. */
typedef struct {
  int32_t batch;             /* requests B >= 0                               */
  int32_t hq;                /* query heads                                   */
  int32_t hkv;               /* KV heads; hq % hkv == 0, hq/hkv in {1,2,4,8}   */
  int32_t head_dim;          /* d in {64, 128}                                */
  int32_t page_size;         /* rows per page; must be 16                     */
  int32_t num_pages;         /* pages in k_pages / v_pages                    */
  int32_t max_pages_per_req; /* columns of page_table                         */
  int32_t max_window;        /* largest W_b allowed                           */
  int32_t mask_words;        /* uint32 words per keep mask, >= ceil(max_window/32) */
  int32_t max_kept;          /* capacity of each kept_idx list, >= 1          */
  int32_t q_dtype;           /* dsa_dtype of q                                */
  int32_t kv_dtype;          /* dsa_dtype of k_pages and v_pages              */
} dsa_dims;

/* Library version, (major << 16) | minor. */
int32_t dsa_version(void);

/* Human-readable name of a status; never NULL. */
const char* dsa_status_string(dsa_status status);

/* Bytes of device workspace every call on `dims` needs (0 if dims is invalid).
 * Depends on dims only.  Zero-fill it before the first call: its error word
 * must start at zero (dsa_clear_device_error resets it after an error). */
size_t dsa_workspace_size(const dsa_dims* dims);

/*
 * dsa_build_index -- mask -> kept-row list (index compaction).
 * Writes, for every (b, hk), kept_cnt[b][hk] = |K(b,hk)| and the ascending
 * logical rows of K(b,hk) into kept_idx[b][hk][0 .. cnt-1]; entries past cnt are
 * unspecified.  Follows the band/window formula of the paper-daily summary
 * (section 核心公式) with its worked example (section 具体技术细节示例: for
 * N=8, W=4, B=2, query 6 the kept keys are 4..7, or 4..6 once decode is causal),
 * plus the prompt prefix the abstract reports attention concentrates on.
 *   seq_len, prompt_len, window  [batch] int32 (device)
 *   keep_mask                    [batch][hkv][mask_words] uint32 (device)
 *   kept_idx  (out)              [batch][hkv][max_kept] int32 (device)
 *   kept_cnt  (out)              [batch][hkv] int32 (device)
 * A count above max_kept sets DSA_DEV_BAD_COUNT and stores count 0.
 * For batches of at most 1024 requests the call also leaves in `ws` a request
 * schedule -- the requests by decreasing total kept rows, ties by index --
 * tagged with the batch size; dsa_decode_sparse on the same workspace hands
 * its requests to the GPU in that order (long requests first, so they do not
 * form the tail of the launch).  Results never depend on it.
 */
dsa_status dsa_build_index(const dsa_dims* dims, const int32_t* seq_len,
                           const int32_t* prompt_len, const int32_t* window,
                           const uint32_t* keep_mask, int32_t* kept_idx, int32_t* kept_cnt,
                           void* ws, void* stream);

/*
 * dsa_decode_sparse -- decode attention over the kept rows only.
 * out[b][h][:] = sum_{j in K(b,hk)} a_j v_j with a = softmax_j(scale * q_bh . k_j),
 * lse[b][h]    = ln sum_{j in K(b,hk)} exp(scale * q_bh . k_j)      (natural log),
 * for hk = h / (hq/hkv) -- the masked softmax of the summary's core formula,
 * masked entries removed.  Only the kept K/V rows are read.  fp32 accumulation.
 *   q                 [batch][hq][head_dim] (q_dtype)
 *   k_pages, v_pages  [num_pages][16][hkv][head_dim] (kv_dtype)
 *   page_table        [batch][max_pages_per_req] int32
 *   seq_len           [batch] int32
 *   kept_idx, kept_cnt  as written by dsa_build_index
 *   scale             softmax scale, normally 1/sqrt(head_dim)
 *   out   (out)       [batch][hq][head_dim] float32
 *   lse   (out)       [batch][hq] float32, or NULL
 * Requests are scheduled in the order dsa_build_index left in `ws` when it was
 * written for this batch size, else in batch order (same results either way).
 */
dsa_status dsa_decode_sparse(const dsa_dims* dims, const void* q, const void* k_pages,
                             const void* v_pages, const int32_t* page_table,
                             const int32_t* seq_len, const int32_t* kept_idx,
                             const int32_t* kept_cnt, float scale, float* out, float* lse,
                             void* ws, void* stream);

/*
 * dsa_decode_sparse_masked -- dsa_build_index followed by dsa_decode_sparse in
 * one call, without the kept lists in device memory: each decode CTA reads
 * the kept set K(b,hk) of its (request, kv head) straight from prompt_len,
 * window and keep_mask (the same set, in the same ascending order, that
 * dsa_build_index writes; same definition as there) and attends over it.  When
 * dsa_decode_plan gives modes 1 and 2 the same plan, out and lse equal those
 * of the two-call path bit for bit.
 *   q, k_pages, v_pages, page_table, seq_len, scale, out, lse  as in
 *                     dsa_decode_sparse
 *   prompt_len, window, keep_mask  as in dsa_build_index
 *   request_order     [batch] int32 (device), or NULL: a permutation of
 *                     0..batch-1 giving the order in which requests are handed
 *                     to the GPU (NULL: 0, 1, ...).  Results do not depend on
 *                     it; scheduling the requests with the most kept rows
 *                     first (e.g. by min(P,L) + min(W, L-1-min(P,L))) shortens
 *                     the tail of a batch with mixed lengths.  An entry
 *                     outside 0..batch-1 sets DSA_DEV_BAD_ORDER and is
 *                     skipped; a request missing from a non-permutation is
 *                     left unspecified.
 *   k_new, v_new      [batch][hkv][head_dim] (kv_dtype, device, 16-byte
 *                     aligned), or both NULL: the K and V rows of the query
 *                     token L_b - 1, appended by this call -- attention reads
 *                     row L_b - 1 from here, and the call stores it into
 *                     k_pages / v_pages at page_table[b][(L_b-1)/16], slot
 *                     (L_b-1)%16, for later steps (the page must be mapped;
 *                     else DSA_DEV_BAD_PAGE).  With NULL the cache must
 *                     already hold row L_b - 1 and is only read.
 * max_window must be <= 1024 (each warp holds the window's mask bits, one
 * 32-bit word per lane), else DSA_ERR_UNSUPPORTED: use the two calls then.  Invalid per-request data
 * (the DSA_DEV_BAD_SEQ_LEN / _PROMPT / _WINDOW / _COUNT cases of
 * dsa_build_index) sets the workspace error word and NaN in that request's out
 * and lse rows of the affected kv head.  The workspace also holds the kept
 * count of every (request, kv head) for the LSE merge of split work.
 */
dsa_status dsa_decode_sparse_masked(const dsa_dims* dims, const void* q, void* k_pages,
                                    void* v_pages, const int32_t* page_table,
                                    const int32_t* seq_len, const int32_t* prompt_len,
                                    const int32_t* window, const uint32_t* keep_mask,
                                    const int32_t* request_order, const void* k_new,
                                    const void* v_new, float scale, float* out, float* lse,
                                    void* ws, void* stream);

/*
 * dsa_host_io -- the host side of one decode step: a contiguous block of inputs
 * copied up before the attention and a contiguous block of results copied back
 * after it, both issued by the call itself on its stream.
 *   host_in   host memory, in_bytes, the source of the upload; pinned
 *             (page-locked) for the copy to be asynchronous
 *   dev_in    device memory, in_bytes, the destination of the upload (the
 *             call's device inputs normally point into it)
 *   dev_out   device memory, out_bytes, the source of the download (normally
 *             holding the call's out and lse)
 *   host_out  host memory, out_bytes, the destination of the download; pinned
 * A size of 0 skips that copy (its two pointers may then be NULL).  The caller
 * owns all four buffers; the library keeps no pointer after the call returns.
 */
typedef struct {
  const void* host_in;
  void* dev_in;
  size_t in_bytes;
  const void* dev_out;
  void* host_out;
  size_t out_bytes;
} dsa_host_io;

/*
 * dsa_decode_sparse_masked_io -- one decode step from host memory in one call:
 * on `stream`, the upload host_in -> dev_in, then exactly the work of
 * dsa_decode_sparse_masked on the remaining (device) arguments, then the
 * download dev_out -> host_out.  Everything is asynchronous; host_out holds the
 * results once the stream has passed the call (e.g. cudaStreamSynchronize).
 * A host buffer that is page-locked and mapped into the device's address space
 * (cudaHostAlloc, or any page-locked memory under unified addressing) is copied
 * by a small kernel that reads or writes it directly, without the copy
 * engines' fixed latency; other host memory goes through cudaMemcpyAsync
 * (synchronous for pageable memory).
 * All arguments are checked before the upload: a call that returns
 * DSA_ERR_INVALID_ARG or DSA_ERR_UNSUPPORTED has issued nothing.  A failed copy
 * returns DSA_ERR_CUDA.  io must not be NULL.
 */
dsa_status dsa_decode_sparse_masked_io(const dsa_host_io* io, const dsa_dims* dims,
                                       const void* q, void* k_pages, void* v_pages,
                                       const int32_t* page_table, const int32_t* seq_len,
                                       const int32_t* prompt_len, const int32_t* window,
                                       const uint32_t* keep_mask, const int32_t* request_order,
                                       const void* k_new, const void* v_new, float scale,
                                       float* out, float* lse, void* ws, void* stream);

/*
 * dsa_graph -- a recorded sequence of libdsa calls, replayed with one launch
 * (a CUDA graph).  A serving loop whose step issues the same calls on the same
 * buffers every time records the step once and replays it: the host then pays
 * one launch per step instead of one per copy and kernel.
 *   dsa_graph_begin(stream)   starts recording `stream` (not the legacy NULL
 *                             stream: DSA_ERR_INVALID_ARG).  The libdsa calls
 *                             issued on it afterwards, by this thread, are
 *                             recorded, not run; their own return values still
 *                             report argument errors.  No call that waits on
 *                             the stream (dsa_get_device_error) may be
 *                             recorded.  Host buffers in recorded copies must be
 *                             pinned.
 *   dsa_graph_end(stream, &g) ends the recording and creates *g, which owns the
 *                             instantiated graph; a failed recording returns
 *                             DSA_ERR_CUDA with *g = NULL.  The recording is
 *                             ended in every case.
 *   dsa_graph_launch(g, stream)  replays every recorded call, in order, on
 *                             `stream`, with the pointers and sizes they were
 *                             recorded with (the buffers must still exist; their
 *                             contents are read at replay time).
 *   dsa_graph_destroy(g)      frees g (NULL is a no-op); replays already
 *                             queued still run (the graph is released when the
 *                             last one finishes).
 * The handle is the only resource the library creates; it holds no device
 * memory of the caller.
 */
typedef struct dsa_graph dsa_graph;
dsa_status dsa_graph_begin(void* stream);
dsa_status dsa_graph_end(void* stream, dsa_graph** graph);
dsa_status dsa_graph_launch(const dsa_graph* graph, void* stream);
dsa_status dsa_graph_destroy(dsa_graph* graph);

/*
 * dsa_decode_dense -- the dense causal baseline: the same as dsa_decode_sparse
 * with K(b,hk) = {0 .. L_b - 1} (the T_dense of the summary's speedup
 * T_dense / T_sparse, section 核心公式).  Arguments as above.
 */
dsa_status dsa_decode_dense(const dsa_dims* dims, const void* q, const void* k_pages,
                            const void* v_pages, const int32_t* page_table,
                            const int32_t* seq_len, float scale, float* out, float* lse,
                            void* ws, void* stream);

/*
 * dsa_attention_mass -- where the dense decode softmax puts its mass, per
 * (request, query head): the characterisation behind the method (abstract:
 * attention concentrates on prompt and local tokens, with a diagonal pattern
 * from the spatial locality of visual tokens; summary, section 技术方法详解:
 * raster order makes spatial neighbours sit at offsets k*w +- r).
 * With a_j the dense causal softmax weights of query i = L_b - 1 and o = i - j:
 *   mass[b][h][0]  prompt    sum of a_j over j < P_b
 *   mass[b][h][1]  local     j >= P_b and o <= r_local
 *   mass[b][h][2]  diagonal  j >= P_b, r_local < o <= W_b, |o - k*w_b| <= r_diag for a k >= 1
 *   mass[b][h][3]  other     every remaining row
 *   offset_mass[b][h][o] = a_{i-o} for 0 <= o <= min(W_b, i), else 0;
 *                          [batch][hq][max_window+1] float32, or NULL.
 *   grid_w   [batch] int32, image grid width w_b >= 1 (row stride in tokens).
 *   prompt_len, window as above; r_local, r_diag >= 0.
 * Only K rows are read (one pass).
 */
dsa_status dsa_attention_mass(const dsa_dims* dims, const void* q, const void* k_pages,
                              const int32_t* page_table, const int32_t* seq_len,
                              const int32_t* prompt_len, const int32_t* window,
                              const int32_t* grid_w, int32_t r_local, int32_t r_diag,
                              float scale, float* mass, float* offset_mass, void* ws,
                              void* stream);

/*
 * dsa_prefill_sparse -- several query tokens per request under the same mask:
 * a chunk of prompt or image tokens prefilled at once, or several image tokens
 * decoded in one step.  The last q_len[b] rows of request b's cache are its
 * query tokens i = L_b - q_len[b] + t, t = 0 .. q_len[b]-1 (their K/V rows must
 * already be in the cache), and query i attends over its own causal kept set,
 * the set of dsa_build_index for a request of length i+1:
 *   K_i(b,hk) = { j < min(P_b, i+1) } U { i } U { i-o : 1 <= o <= W_b, bit o-1, i-o >= P_b }
 * -- the core formula of the paper-daily summary (section 核心公式) read at
 * every query position, with masked entries removed.  The arXiv abstract
 * reports prefill attention to be diffuse, so a chunk gains less from the mask
 * than a decode step; the call serves chunks that keep the decode mask.
 *   max_q             query slots per request (>= 0; 0 is a no-op)
 *   q                 [batch][max_q][hq][head_dim] bf16 (device); slot t of
 *                     request b is query token L_b - q_len[b] + t
 *   k_pages, v_pages, page_table, seq_len, prompt_len, window, keep_mask
 *                     as in dsa_decode_sparse_masked (K/V bf16)
 *   q_len             [batch] int32 (device), 0 <= q_len[b] <= min(L_b, max_q)
 *   request_order     [batch] int32 (device), or NULL: the order in which
 *                     requests are handed to the GPU, as in
 *                     dsa_decode_sparse_masked; the requests that scan the most
 *                     rows first (about min(P,L) + min(W + q_len, L - min(P,L)))
 *                     shortens the tail of a batch with mixed lengths.  An entry
 *                     outside 0..batch-1 sets DSA_DEV_BAD_ORDER and is skipped.
 *   scale             softmax scale, normally 1/sqrt(head_dim)
 *   out   (out)       [batch][max_q][hq][head_dim] float32; slots t >= q_len[b]
 *                     are not written
 *   lse   (out)       [batch][max_q][hq] float32 natural-log LSE, or NULL
 * Rows of the scanned range that no query of a CTA's tile keeps are not read.
 * Units may be split over several CTAs (dsa_set_prefill_split), which use the
 * workspace's partials region and its arrival counters: those counters are
 * back at zero after every call that completes without a device error (after
 * one, zero-fill the workspace again).
 * q and KV must be bf16 and max_window <= 32768, else DSA_ERR_UNSUPPORTED.  An
 * invalid per-request value (seq_len, prompt_len, window as above; q_len gives
 * DSA_DEV_BAD_QLEN) sets the error word and NaN in that request's slots.
 */
dsa_status dsa_prefill_sparse(const dsa_dims* dims, int32_t max_q, const void* q,
                              const void* k_pages, const void* v_pages,
                              const int32_t* page_table, const int32_t* seq_len,
                              const int32_t* q_len, const int32_t* prompt_len,
                              const int32_t* window, const uint32_t* keep_mask,
                              const int32_t* request_order, float scale, float* out, float* lse,
                              void* ws, void* stream);

/*
 * dsa_evict_pages -- unmap the pages no later decode step can read, and hand
 * them back for reuse: the memory side of the method (its kept set reads only
 * the prompt and a window that moves forward; arXiv abstract: the other KV
 * entries are skipped), so a long request keeps about P + W + 16 rows resident
 * instead of L.  A page of request b holding rows 16p .. 16p+15 is evicted when
 * every row j of it satisfies P_b <= j < (L_b - 1) - W_b (P_b and W_b taken as
 * fixed while the request decodes); such rows are outside the kept set of the
 * current query and of every later one, for any keep mask.
 *   seq_len, prompt_len, window  [batch] int32 (device), as in dsa_build_index
 *   page_table   [batch][max_pages_per_req] int32 (device, updated in place):
 *                evicted entries become -1; entries already -1 are skipped
 *   freed_pages  [capacity] int32 (device, out): the evicted page ids, in no
 *                particular order, from index *freed_count (as it was) on
 *   freed_count  one int32 (device, in/out): entries already in freed_pages;
 *                advanced by the number of pages evicted
 *   capacity     size of freed_pages (>= 0)
 * A page that finds the list full stays mapped and sets DSA_DEV_FREE_LIST_FULL
 * (freed_count may then exceed capacity: only the first `capacity` entries are
 * written).  Invalid sizes set DSA_DEV_BAD_SEQ_LEN / _PROMPT / _WINDOW and leave
 * that request's pages alone.  The decode calls never read evicted rows, so a
 * batch decodes the same after eviction.
 */
dsa_status dsa_evict_pages(const dsa_dims* dims, const int32_t* seq_len,
                           const int32_t* prompt_len, const int32_t* window, int32_t* page_table,
                           int32_t* freed_pages, int32_t* freed_count, int32_t capacity, void* ws,
                           void* stream);

/*
 * dsa_decode_plan -- how a decode call will split its work on the CURRENT
 * device: rows per CTA (*chunk), CTAs per (request, kv head) at most
 * (*num_chunks), kernel launches per call (*launches), warps per CTA (*warps)
 * and rows per tile (*tile_rows).  mode selects the call: 0 dsa_decode_dense, 1 dsa_decode_sparse,
 * 2 dsa_decode_sparse_masked (other values: DSA_ERR_INVALID_ARG).  Two calls
 * with the same plan sum in the same order.  Host-only; any output pointer may
 * be NULL.
 */
dsa_status dsa_decode_plan(const dsa_dims* dims, int32_t mode, int32_t* chunk,
                           int32_t* num_chunks, int32_t* launches, int32_t* warps,
                           int32_t* tile_rows);

/*
 * dsa_decode_sparse_noalloc -- dsa_decode_sparse for callers that cannot
 * allocate device memory.  The paper has no counterpart: this is a packaging
 * variant of the same computation, for hosts that only lend us pointers.
 *
 * Who needs it: code that runs where device allocation is unavailable or
 * forbidden -- a plugin inside an inference server whose memory pool owns all
 * of the device memory and hands out nothing but tensors, a real-time decode
 * loop where a cudaMalloc/cudaFree would synchronise the device and miss its
 * deadline, or a host application that receives input and output buffers from
 * another runtime and has no way to ask it for a scratch buffer of our size.
 *
 * Instead of a caller workspace, the call uses one scratch array that the
 * library itself places in device memory at load time
 * (DSA_NOALLOC_SCRATCH_BYTES on every GPU that loads the library, held until
 * the process exits).  Arguments, layouts and results are those of
 * dsa_decode_sparse, without `ws`; the caller still owns q, the KV pages, the
 * page table, the kept lists and out / lse.
 *   dev_error  device pointer to one int32, or NULL: receives this call's
 *              device error code (DSA_DEV_*, 0 when clean), asynchronously on
 *              `stream`.
 * Returns DSA_ERR_SCRATCH_LIMIT, before touching the GPU, when the batch needs
 * more scratch than DSA_NOALLOC_SCRATCH_BYTES (256 bytes plus
 * batch * hq * chunks * (head_dim + 2) * 4, chunks as in dsa_decode_plan);
 * use dsa_decode_sparse with a workspace then.
 * Set-up: the first call on each device looks up the scratch array's device
 * address (with that device current); make that first call before any stream
 * capture on the device.
 * Every call shares the one scratch array and clears the part that must start
 * at zero; calls whose work overlaps on the GPU (other streams, other host
 * threads) race on it and must be serialised by the caller.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
#define DSA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
dsa_status dsa_decode_sparse_noalloc(const dsa_dims* dims, const void* q, const void* k_pages,
                                     const void* v_pages, const int32_t* page_table,
                                     const int32_t* seq_len, const int32_t* kept_idx,
                                     const int32_t* kept_cnt, float scale, float* out,
                                     float* lse, int32_t* dev_error, void* stream);

/*
 * dsa_set_sparse_cluster -- process-wide tuning of dsa_decode_sparse and
 * dsa_decode_sparse_masked (not in the paper: a scheduling choice).  With
 * ctas >= 2, the rows of each (request, kv head) are split evenly over `ctas`
 * CTAs launched as one thread-block cluster, which combine their partial
 * softmax states through distributed shared memory (no merge launch, no
 * partials in device memory); with 1, a (request, kv head) whose kept rows fit
 * one chunk runs in one CTA and longer ones are split into chunks merged by a
 * second kernel; with 0 (the default) each call picks: clusters of 2, 4 or 8
 * only when the batch has too few (request, kv head) pairs to fill half of the
 * GPU's resident CTA slots, else 1.  Results equal the oracle's within the same
 * bounds either way, but the floating-point summation order depends on the
 * split.  ctas in 0..8, else DSA_ERR_INVALID_ARG.  Takes effect for calls
 * issued afterwards; not synchronised with calls in flight on other host
 * threads.  dsa_get_sparse_cluster returns the current value.
 */
dsa_status dsa_set_sparse_cluster(int32_t ctas);
int32_t dsa_get_sparse_cluster(void);

/*
 * dsa_prefill_plan -- the launch dsa_prefill_sparse makes for dims and max_q on
 * the current device under the current dsa_set_prefill_split setting: warps per
 * CTA (2 or 4), units (query tiles x kv heads x requests), the units run whole
 * (one CTA each; the later ones are split), the parts of each split unit, the
 * resident CTAs per SM of the kernel and the CTAs launched.  Host-only (no
 * kernel is enqueued); any output pointer may be NULL.  The same argument
 * checks as dsa_prefill_sparse; DSA_ERR_CUDA if the device cannot be queried.
 */
dsa_status dsa_prefill_plan(const dsa_dims* dims, int32_t max_q, int32_t* warps, int32_t* units,
                            int32_t* whole, int32_t* parts, int32_t* ctas_per_sm, int32_t* ctas);

/*
 * dsa_set_prefill_split -- process-wide tuning of dsa_prefill_sparse (not in
 * the paper: a scheduling choice).  A unit of that call (a tile of query tokens
 * of one request and kv head) normally runs in one CTA.  With parts >= 2 every
 * unit (as many as the workspace holds: the last ones) is split into `parts`
 * CTAs along its scanned rows; their partial softmax states go to the workspace
 * and the unit's last CTA to finish merges them (no second kernel).  With 1 no
 * unit is split; with 0 (the default) each call splits only what balances the
 * GPU: the units of a last, partial wave of resident CTAs (or every unit of a
 * batch smaller than one wave) into up to 4 parts.  Results equal the oracle's
 * within the same bounds either way; the floating-point summation order depends
 * on the split.  parts in 0..8, else DSA_ERR_INVALID_ARG.  Takes effect for
 * calls issued afterwards.  dsa_get_prefill_split returns the current value.
 */
dsa_status dsa_set_prefill_split(int32_t parts);
int32_t dsa_get_prefill_split(void);

/*
 * Waits for `stream`, then reads the workspace error word into *code_out (one of
 * DSA_DEV_*).  Returns DSA_OK when the word is 0, DSA_ERR_TIMEOUT when it is
 * DSA_DEV_TIMEOUT, DSA_ERR_DEVICE for any other code, DSA_ERR_CUDA if the copy
 * fails.  Synchronising.
 */
dsa_status dsa_get_device_error(const void* ws, void* stream, int32_t* code_out);

/* Clears the workspace error word (asynchronous on `stream`). */
dsa_status dsa_clear_device_error(void* ws, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
