// dsa_api.cu -- the extern "C" entry points of libdsa (declared in dsa.h):
// host-side validation, work-chunk sizing, and kernel dispatch.  Nothing here
// computes attention; every step of the path runs in the kernels.
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <new>

#include <cuda_runtime.h>

#include "common.cuh"
#include "dsa.h"
#include "internal.h"

// Build-time tuning knobs: waves of resident CTAs the chunking aims for.  Kept
// lists are short, so sparse decode wants one chunk per (request, kv head)
// where possible (no merge launch); dense rows vary with seq_len, so dense
// decode and attention mass want more, shorter chunks for balance (the mass
// kernel's two score engines measured best at different counts).
#ifndef DSA_SPARSE_WAVES
#define DSA_SPARSE_WAVES 1
#endif
#ifndef DSA_DENSE_WAVES
#define DSA_DENSE_WAVES 8
#endif
#ifndef DSA_MASS_WAVES
#define DSA_MASS_WAVES 4
#endif
#ifndef DSA_MASS_WAVES_MMA
#define DSA_MASS_WAVES_MMA 8
#endif
// CTAs that share one (request, kv head) of sparse decode as a thread-block
// cluster, merging through distributed shared memory (1: no cluster, 0: chosen
// per call by sparse_cluster_auto()).
#ifndef DSA_SPARSE_CLUSTER
#define DSA_SPARSE_CLUSTER 0
#endif

namespace dsa {
namespace {

constexpr int kMaxDevices = 64;

// Process-wide: CTAs per cluster of sparse decode (dsa_set_sparse_cluster).
std::atomic<int> g_sparse_cluster{DSA_SPARSE_CLUSTER};
// Process-wide: parts of dsa_prefill_sparse's units (dsa_set_prefill_split).
std::atomic<int> g_prefill_split{0};

bool dims_valid(const dsa_dims* d) {
  if (d == nullptr) return false;
  if (d->batch < 0 || d->hq < 1 || d->hkv < 1 || d->head_dim < 1) return false;
  if (d->hq % d->hkv != 0) return false;
  if (d->num_pages < 1 || d->max_pages_per_req < 1 || d->max_window < 0) return false;
  if (d->mask_words < 1 || static_cast<int64_t>(d->mask_words) * 32 < d->max_window) return false;
  if (d->max_kept < 1) return false;
  if (d->q_dtype != DSA_F32 && d->q_dtype != DSA_BF16) return false;
  if (d->kv_dtype != DSA_F32 && d->kv_dtype != DSA_BF16) return false;
  // page_table entries index rows as page * 16 * hkv * head_dim elements in 64-bit math;
  // logical positions are int32.
  if (static_cast<int64_t>(d->max_pages_per_req) * kPage > INT32_MAX / 2) return false;
  return true;
}

bool dims_supported(const dsa_dims* d) {
  const int g = d->hq / d->hkv;
  return d->page_size == kPage && (d->head_dim == 64 || d->head_dim == 128) &&
         (g == 1 || g == 2 || g == 4 || g == 8);
}

dsa_status check_dims(const dsa_dims* d) {
  if (!dims_valid(d)) return DSA_ERR_INVALID_ARG;
  if (!dims_supported(d)) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Upper bound of chunks per (request, kv head) for a row count n_max.
int chunk_bound(int64_t n_max) {
  const int64_t c = ceil_div(n_max, kChunkQuantum);
  return static_cast<int>(c < kMaxChunks ? (c < 1 ? 1 : c) : kMaxChunks);
}

int64_t dense_rows(const dsa_dims* d) { return static_cast<int64_t>(d->max_pages_per_req) * kPage; }

size_t partial_bytes(const dsa_dims* d, int per_head_floats) {
  const int64_t n_max = dense_rows(d) > d->max_kept ? dense_rows(d) : d->max_kept;
  return static_cast<size_t>(d->batch) * d->hq * chunk_bound(n_max) * per_head_floats *
         sizeof(float);
}

int sm_count() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < kMaxDevices && cache[dev] > 0) return cache[dev];
  int n = 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    n = 1;
  if (dev >= 0 && dev < kMaxDevices) cache[dev] = n;
  return n;
}

// Rows per CTA: enough CTAs for `waves` waves of resident CTAs, at most
// kMaxChunks chunks per (request, kv head), a multiple of the CTA's rows per pass.
// With `whole_split` a unit is cut into floor(target / units) equal chunks (at
// least one): n_max is only a bound on a unit's rows, so a cut sized from it
// would add CTAs (and a merge launch) past the wave without shortening any.
void choose_chunks(int64_t n_max, int64_t units, int resident, int quantum, int waves,
                   bool whole_split, int* chunk, int* num_chunks) {
  if (quantum < kChunkQuantum) quantum = kChunkQuantum;
  const int64_t target = static_cast<int64_t>(waves) * resident;
  int64_t c = ceil_div(n_max * units, target > 0 ? target : 1);
  if (whole_split) {
    const int64_t k = units > 0 ? target / units : 1;
    c = ceil_div(n_max, k > 1 ? k : 1);
  }
  const int64_t lo = ceil_div(n_max, kMaxChunks);
  if (c < lo) c = lo;
  c = ceil_div(c, quantum) * quantum;
  const int64_t hi = ceil_div(n_max, quantum) * quantum;
  if (c > hi) c = hi;
  if (c < quantum) c = quantum;
  // chunk_bound() sizes the workspace with chunks of kChunkQuantum rows, so any
  // chunk >= max(quantum, n_max / kMaxChunks) fits.
  *chunk = static_cast<int>(c);
  *num_chunks = static_cast<int>(ceil_div(n_max, c));
}

dsa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

int32_t* err_word(void* ws) { return reinterpret_cast<int32_t*>(ws); }

float* partials(void* ws) {
  return reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(ws) + kWsHeader);
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Partials region of the workspace, the same for every entry point.
size_t partials_region(const dsa_dims* d) {
  const size_t dec = partial_bytes(d, d->head_dim + 2);
  const size_t mass = partial_bytes(d, 6);
  // dsa_prefill_sparse's split parts: at most one wave of resident CTAs, at
  // most kMultiPartWarpsPerSm warps of 16 (query, head) rows each per SM
  const size_t multi = static_cast<size_t>(sm_count()) * kMultiPartWarpsPerSm * 16 *
                       (d->head_dim + 2) * sizeof(float);
  size_t r = dec > mass ? dec : mass;
  if (multi > r) r = multi;
  return round_up(r, 256);
}

// [batch][hkv] kept counts of dsa_decode_sparse_masked, after the partials.
int32_t* unit_rows(const dsa_dims* d, void* ws) {
  return reinterpret_cast<int32_t*>(reinterpret_cast<unsigned char*>(ws) + kWsHeader +
                                    partials_region(d));
}

size_t unit_ints_region(const dsa_dims* d) {
  return round_up(static_cast<size_t>(d->batch) * d->hkv * sizeof(int32_t), 256);
}

// [batch] request schedule dsa_build_index leaves for dsa_decode_sparse, after
// the kept counts of the fused call.
int32_t* sched_region(const dsa_dims* d, void* ws) {
  return reinterpret_cast<int32_t*>(reinterpret_cast<unsigned char*>(ws) + kWsHeader +
                                    partials_region(d) + unit_ints_region(d));
}

size_t sched_bytes(const dsa_dims* d) {
  return round_up(static_cast<size_t>(d->batch) * sizeof(int32_t), 256);
}

// Arrival counters of dsa_prefill_sparse's split units, after the schedule.
int32_t* multi_count_region(const dsa_dims* d, void* ws) {
  return reinterpret_cast<int32_t*>(reinterpret_cast<unsigned char*>(ws) + kWsHeader +
                                    partials_region(d) + unit_ints_region(d) + sched_bytes(d));
}

constexpr size_t kMultiCountBytes = kMultiCounters * sizeof(int32_t);


bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Plan {
  int chunk, num_chunks, quantum, per_sm, cluster, warps, tile_rows, build;
};

// Automatic cluster size: a CTA's fixed latency (first copies, end-of-CTA
// merge) makes short CTAs slow, so split units over clusters only when there
// are too few of them to occupy the GPU -- the largest size in {2, 4, 8} whose
// CTAs still fit in half of the resident slots, else 1.
int sparse_cluster_auto(int64_t units, int64_t slots) {
  int best = 1;
  for (int c = 2; c <= kMaxCluster; c *= 2)
    if (units * c <= slots / 2) best = c;
  return best;
}

DecodeShape decode_shape(const dsa_dims* d, int mode, int build) {
  const int g = d->hq / d->hkv;
  return d->kv_dtype == DSA_BF16 ? decode_shape_bf16(d->head_dim, g, mode, build)
                                 : decode_shape_f32(d->head_dim, g, mode, build);
}

// The wide build takes a unit in one CTA when its kept rows need at most this
// many passes of the CTA's warps.
constexpr int kWideMaxPasses = 4;

Plan decode_plan(const dsa_dims* d, int mode) {
  const int64_t n_max = mode == kModeDense ? dense_rows(d) : d->max_kept;
  const int64_t units = static_cast<int64_t>(d->batch) * d->hkv;
  const int setting = g_sparse_cluster.load(std::memory_order_relaxed);
  if (mode != kModeDense && setting == 0 && units <= sm_count()) {
    // at most one unit per SM: each unit in one 8-warp CTA (rows spread over its
    // warps, merged in shared memory), no cluster and no merge launch
    const DecodeShape wide = decode_shape(d, mode, kBuildWide);
    if (wide.build == kBuildWide &&
        n_max <= static_cast<int64_t>(kWideMaxPasses) * wide.rows_per_pass) {
      Plan p{};
      p.quantum = wide.rows_per_pass;
      p.per_sm = wide.ctas_per_sm;
      p.warps = wide.warps;
      p.tile_rows = wide.tile_rows;
      p.build = kBuildWide;
      p.cluster = 1;
      p.num_chunks = 1;
      p.chunk = static_cast<int>(ceil_div(n_max, p.quantum) * p.quantum);
      return p;
    }
  }
  DecodeShape sh = decode_shape(d, mode, kBuildDefault);
  const int64_t slots = static_cast<int64_t>(sm_count()) * sh.ctas_per_sm;
  if (mode != kModeDense && units > 2 * slots) {
    // more than two waves of units: the big-batch build (smaller stages, more
    // warps per SM to overlap the latency of the gathers), when there is one
    const DecodeShape big = decode_shape(d, mode, kBuildBig);
    if (big.build == kBuildBig) sh = big;
  } else if (mode != kModeDense && units > slots) {
    // two waves of the default build: the small-batch build if it takes the
    // whole batch in one wave
    const DecodeShape small = decode_shape(d, mode, kBuildSmall);
    if (small.build == kBuildSmall && units <= static_cast<int64_t>(sm_count()) * small.ctas_per_sm)
      sh = small;
  }
  Plan p{};
  p.quantum = sh.rows_per_pass;
  p.per_sm = sh.ctas_per_sm;
  p.warps = sh.warps;
  p.tile_rows = sh.tile_rows;
  p.build = sh.build;
  p.cluster = 1;
  int ncl = setting;
  if (ncl == 0) ncl = sparse_cluster_auto(units, sm_count() * p.per_sm);
  while (ncl > sh.cluster_limit) ncl /= 2;
  if (mode != kModeDense && ncl > 1 && n_max > p.quantum) {
    // the rows of a unit split evenly over a cluster of ncl CTAs
    p.cluster = ncl;
    p.num_chunks = ncl;
    p.chunk = static_cast<int>(ceil_div(n_max, ncl));
    return p;
  }
  choose_chunks(n_max, units, sm_count() * p.per_sm, p.quantum,
                mode == kModeDense ? DSA_DENSE_WAVES : DSA_SPARSE_WAVES, mode != kModeDense,
                &p.chunk, &p.num_chunks);
  return p;
}

// Row sources of decode_common: the kept list (kModeList) or the per-request
// prompt length, window and keep mask (kModeMask).
struct RowSource {
  const int32_t* kept_idx = nullptr;
  const int32_t* kept_cnt = nullptr;
  const int32_t* prompt_len = nullptr;
  const int32_t* window = nullptr;
  const uint32_t* keep_mask = nullptr;
  const int32_t* order = nullptr;
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  bool use_sched = false;  // kModeList: the schedule dsa_build_index left in ws
};

dsa_status decode_launch(const dsa_dims* d, int mode, const Plan& plan, const void* q,
                         const void* k, const void* v, const int32_t* page_table,
                         const int32_t* seq_len, const RowSource& rs, float scale, float* out,
                         float* lse, void* ws, cudaStream_t s);

// Checks a decode call's arguments, then (with io) the host-to-device copy, the
// launches and (with io) the device-to-host copy, in that order on the stream.
// `plan`, when given, is the split to launch with (computed once by a caller
// that sized its scratch from it); else decode_plan() is taken here.
dsa_status decode_common(const dsa_dims* d, int mode, const void* q, const void* k,
                         const void* v, const int32_t* page_table, const int32_t* seq_len,
                         const RowSource& rs, float scale, float* out, float* lse, void* ws,
                         void* stream, const dsa_host_io* io = nullptr,
                         const Plan* plan = nullptr) {
  const dsa_status st = check_dims(d);
  if (st != DSA_OK) return st;
  if (!q || !k || !v || !page_table || !seq_len || !out || !ws) return DSA_ERR_INVALID_ARG;
  if (mode == kModeList && (!rs.kept_idx || !rs.kept_cnt)) return DSA_ERR_INVALID_ARG;
  if (mode == kModeMask && (!rs.prompt_len || !rs.window || !rs.keep_mask))
    return DSA_ERR_INVALID_ARG;
  if (mode == kModeMask && d->max_window > kMaskModeMaxWindow) return DSA_ERR_UNSUPPORTED;
  if ((rs.k_new == nullptr) != (rs.v_new == nullptr)) return DSA_ERR_INVALID_ARG;
  if (rs.k_new != nullptr && (!aligned(rs.k_new, 16) || !aligned(rs.v_new, 16)))
    return DSA_ERR_INVALID_ARG;
  if (!(scale == scale) || !aligned(ws, 256) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(q, 16))
    return DSA_ERR_INVALID_ARG;
  if (io != nullptr && ((io->in_bytes > 0 && (!io->host_in || !io->dev_in)) ||
                        (io->out_bytes > 0 && (!io->dev_out || !io->host_out))))
    return DSA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (io != nullptr && copy_host_to_device(io->dev_in, io->host_in, io->in_bytes, s) != cudaSuccess)
    return DSA_ERR_CUDA;
  dsa_status rc = DSA_OK;
  if (d->batch > 0) {
    const Plan p = plan != nullptr ? *plan : decode_plan(d, mode);
    rc = decode_launch(d, mode, p, q, k, v, page_table, seq_len, rs, scale, out, lse, ws, s);
  }
  if (rc != DSA_OK) return rc;
  if (io != nullptr &&
      copy_device_to_host(io->host_out, io->dev_out, io->out_bytes, s) != cudaSuccess)
    return DSA_ERR_CUDA;
  return DSA_OK;
}

// The launches of one decode call (arguments already checked, batch >= 1).
dsa_status decode_launch(const dsa_dims* d, int mode, const Plan& plan, const void* q,
                         const void* k, const void* v, const int32_t* page_table,
                         const int32_t* seq_len, const RowSource& rs, float scale, float* out,
                         float* lse, void* ws, cudaStream_t s) {
  const bool kv_bf16 = d->kv_dtype == DSA_BF16;
  DecodeLaunch a{};
  a.q = q;
  a.q_bf16 = d->q_dtype == DSA_BF16;
  a.k = k;
  a.v = v;
  a.page_table = page_table;
  a.seq_len = seq_len;
  a.kept_idx = rs.kept_idx;
  a.kept_cnt = rs.kept_cnt;
  a.prompt_len = rs.prompt_len;
  a.window = rs.window;
  a.keep_mask = rs.keep_mask;
  a.unit_rows = mode == kModeMask ? unit_rows(d, ws) : nullptr;
  a.order = rs.order;
  if (rs.use_sched) {
    a.sched = sched_region(d, ws);
    a.sched_tag = err_word(ws) + kWsSchedTag;
    a.sched_expect = kSchedMagic ^ d->batch;
  }
  a.k_new = rs.k_new;
  a.v_new = rs.v_new;
  a.max_window = d->max_window;
  a.mask_words = d->mask_words;
  a.batch = d->batch;
  a.hq = d->hq;
  a.hkv = d->hkv;
  a.head_dim = d->head_dim;
  a.max_pages = d->max_pages_per_req;
  a.num_pages = d->num_pages;
  a.max_kept = d->max_kept;
  a.chunk = plan.chunk;
  a.num_chunks = plan.num_chunks;
  a.cluster = plan.cluster;
  a.warps = plan.warps;
  a.build = plan.build;
  a.scale_log2 = scale * kLog2e;
  a.out = out;
  a.lse = lse;
  a.part = partials(ws);
  a.err = err_word(ws);
  cudaError_t e = kv_bf16 ? launch_decode_bf16(a, mode, s) : launch_decode_f32(a, mode, s);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  if (a.cluster > 1) return DSA_OK;  // merged inside the clusters
  return from_cuda(launch_merge(a, mode, s));
}

// The shape of a multi-query launch on dims (every field but the pointers),
// or DSA_ERR_UNSUPPORTED when its work items do not fit a 1-D grid.
dsa_status multi_shape(const dsa_dims* dims, int32_t max_q, MultiLaunch* out) {
  MultiLaunch a{};
  a.batch = dims->batch;
  a.hq = dims->hq;
  a.hkv = dims->hkv;
  a.head_dim = dims->head_dim;
  a.max_pages = dims->max_pages_per_req;
  a.num_pages = dims->num_pages;
  a.max_window = dims->max_window;
  a.mask_words = dims->mask_words;
  a.max_q = max_q;
  a.warps = multi_warps(max_q, dims->hq / dims->hkv);
  const int per_cta = multi_queries_per_cta(a.warps, dims->hq / dims->hkv);
  a.q_tiles = static_cast<int32_t>(ceil_div(max_q, per_cta));
  // work items (units times parts) index a 1-D grid
  if (static_cast<int64_t>(a.q_tiles) * dims->hkv * dims->batch * kMultiMaxParts > INT32_MAX)
    return DSA_ERR_UNSUPPORTED;
  a.split_setting = g_prefill_split.load(std::memory_order_relaxed);
  a.part_rows_cap = static_cast<int64_t>(partials_region(dims) / ((dims->head_dim + 2) * sizeof(float)));
  a.count_cap = kMultiCounters;
  a.sms = sm_count();
  *out = a;
  return DSA_OK;
}

dsa_status multi_dims_ok(const dsa_dims* dims, int32_t max_q) {
  const dsa_status st = check_dims(dims);
  if (st != DSA_OK) return st;
  if (max_q < 0) return DSA_ERR_INVALID_ARG;
  if (dims->q_dtype != DSA_BF16 || dims->kv_dtype != DSA_BF16 ||
      dims->max_window > kMultiMaxWindow)
    return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

int32_t dsa_version(void) { return (0 << 16) | 1; }

const char* dsa_status_string(dsa_status status) {
  switch (status) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_DEVICE: return "DSA_ERR_DEVICE";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
    case DSA_ERR_SCRATCH_LIMIT: return "DSA_ERR_SCRATCH_LIMIT";
  }
  return "DSA_ERR_UNKNOWN";
}

size_t dsa_workspace_size(const dsa_dims* dims) {
  if (check_dims(dims) != DSA_OK) return 0;
  return kWsHeader + partials_region(dims) + unit_ints_region(dims) + sched_bytes(dims) +
         kMultiCountBytes;
}

dsa_status dsa_build_index(const dsa_dims* dims, const int32_t* seq_len,
                           const int32_t* prompt_len, const int32_t* window,
                           const uint32_t* keep_mask, int32_t* kept_idx, int32_t* kept_cnt,
                           void* ws, void* stream) {
  const dsa_status st = check_dims(dims);
  if (st != DSA_OK) return st;
  if (!seq_len || !prompt_len || !window || !keep_mask || !kept_idx || !kept_cnt || !ws)
    return DSA_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return DSA_ERR_INVALID_ARG;
  CompactLaunch a{};
  a.seq_len = seq_len;
  a.prompt_len = prompt_len;
  a.window = window;
  a.keep_mask = keep_mask;
  a.kept_idx = kept_idx;
  a.kept_cnt = kept_cnt;
  a.batch = dims->batch;
  a.hkv = dims->hkv;
  a.max_pages = dims->max_pages_per_req;
  a.max_window = dims->max_window;
  a.mask_words = dims->mask_words;
  a.max_kept = dims->max_kept;
  a.err = err_word(ws);
  a.sched = sched_region(dims, ws);
  a.sched_tag = err_word(ws) + kWsSchedTag;
  a.done_count = err_word(ws) + kWsDoneCount;
  return from_cuda(launch_compact(a, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_evict_pages(const dsa_dims* dims, const int32_t* seq_len,
                           const int32_t* prompt_len, const int32_t* window, int32_t* page_table,
                           int32_t* freed_pages, int32_t* freed_count, int32_t capacity, void* ws,
                           void* stream) {
  const dsa_status st = check_dims(dims);
  if (st != DSA_OK) return st;
  if (!seq_len || !prompt_len || !window || !page_table || !freed_count || !ws || capacity < 0 ||
      (capacity > 0 && !freed_pages))
    return DSA_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return DSA_ERR_INVALID_ARG;
  EvictLaunch a{};
  a.seq_len = seq_len;
  a.prompt_len = prompt_len;
  a.window = window;
  a.page_table = page_table;
  a.freed = freed_pages;
  a.freed_count = freed_count;
  a.batch = dims->batch;
  a.max_pages = dims->max_pages_per_req;
  a.max_window = dims->max_window;
  a.capacity = capacity;
  a.err = err_word(ws);
  return from_cuda(launch_evict(a, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_decode_sparse(const dsa_dims* dims, const void* q, const void* k_pages,
                             const void* v_pages, const int32_t* page_table,
                             const int32_t* seq_len, const int32_t* kept_idx,
                             const int32_t* kept_cnt, float scale, float* out, float* lse,
                             void* ws, void* stream) {
  RowSource rs;
  rs.kept_idx = kept_idx;
  rs.kept_cnt = kept_cnt;
  rs.use_sched = true;
  return decode_common(dims, kModeList, q, k_pages, v_pages, page_table, seq_len, rs, scale, out,
                       lse, ws, stream);
}

dsa_status dsa_decode_sparse_masked(const dsa_dims* dims, const void* q, void* k_pages,
                                    void* v_pages, const int32_t* page_table,
                                    const int32_t* seq_len, const int32_t* prompt_len,
                                    const int32_t* window, const uint32_t* keep_mask,
                                    const int32_t* request_order, const void* k_new,
                                    const void* v_new, float scale, float* out, float* lse,
                                    void* ws, void* stream) {
  RowSource rs;
  rs.prompt_len = prompt_len;
  rs.window = window;
  rs.keep_mask = keep_mask;
  rs.order = request_order;
  rs.k_new = k_new;
  rs.v_new = v_new;
  return decode_common(dims, kModeMask, q, k_pages, v_pages, page_table, seq_len, rs, scale, out,
                       lse, ws, stream);
}

dsa_status dsa_decode_sparse_masked_io(const dsa_host_io* io, const dsa_dims* dims,
                                       const void* q, void* k_pages, void* v_pages,
                                       const int32_t* page_table, const int32_t* seq_len,
                                       const int32_t* prompt_len, const int32_t* window,
                                       const uint32_t* keep_mask, const int32_t* request_order,
                                       const void* k_new, const void* v_new, float scale,
                                       float* out, float* lse, void* ws, void* stream) {
  if (io == nullptr) return DSA_ERR_INVALID_ARG;
  RowSource rs;
  rs.prompt_len = prompt_len;
  rs.window = window;
  rs.keep_mask = keep_mask;
  rs.order = request_order;
  rs.k_new = k_new;
  rs.v_new = v_new;
  return decode_common(dims, kModeMask, q, k_pages, v_pages, page_table, seq_len, rs, scale, out,
                       lse, ws, stream, io);
}

dsa_status dsa_decode_dense(const dsa_dims* dims, const void* q, const void* k_pages,
                            const void* v_pages, const int32_t* page_table,
                            const int32_t* seq_len, float scale, float* out, float* lse,
                            void* ws, void* stream) {
  return decode_common(dims, kModeDense, q, k_pages, v_pages, page_table, seq_len, RowSource{},
                       scale, out, lse, ws, stream);
}

dsa_status dsa_attention_mass(const dsa_dims* dims, const void* q, const void* k_pages,
                              const int32_t* page_table, const int32_t* seq_len,
                              const int32_t* prompt_len, const int32_t* window,
                              const int32_t* grid_w, int32_t r_local, int32_t r_diag,
                              float scale, float* mass, float* offset_mass, void* ws,
                              void* stream) {
  const dsa_status st = check_dims(dims);
  if (st != DSA_OK) return st;
  if (!q || !k_pages || !page_table || !seq_len || !prompt_len || !window || !grid_w || !mass ||
      !ws)
    return DSA_ERR_INVALID_ARG;
  if (r_local < 0 || r_diag < 0 || !(scale == scale) || !aligned(ws, 256) ||
      !aligned(k_pages, 16) || !aligned(q, 16))
    return DSA_ERR_INVALID_ARG;
  if (dims->batch == 0) return DSA_OK;
  const int64_t n_max = dense_rows(dims);
  MassLaunch a{};
  a.q = q;
  a.q_bf16 = dims->q_dtype == DSA_BF16;
  a.k = k_pages;
  a.page_table = page_table;
  a.seq_len = seq_len;
  a.prompt_len = prompt_len;
  a.window = window;
  a.grid_w = grid_w;
  a.batch = dims->batch;
  a.hq = dims->hq;
  a.hkv = dims->hkv;
  a.head_dim = dims->head_dim;
  a.max_pages = dims->max_pages_per_req;
  a.num_pages = dims->num_pages;
  a.max_window = dims->max_window;
  a.r_local = r_local;
  a.r_diag = r_diag;
  const bool kv_bf16 = dims->kv_dtype == DSA_BF16, q_bf16 = dims->q_dtype == DSA_BF16;
  const int g = dims->hq / dims->hkv;
  choose_chunks(n_max, static_cast<int64_t>(dims->batch) * dims->hkv,
                sm_count() * mass_ctas_per_sm(dims->head_dim, g, kv_bf16, q_bf16),
                mass_rows_per_pass(dims->head_dim, g, kv_bf16, q_bf16),
                mass_uses_tensor_cores(kv_bf16, q_bf16, g) ? DSA_MASS_WAVES_MMA : DSA_MASS_WAVES,
                false, &a.chunk, &a.num_chunks);
  a.scale_log2 = scale * kLog2e;
  a.mass = mass;
  a.offset_mass = offset_mass;
  a.part = partials(ws);
  a.err = err_word(ws);
  return from_cuda(launch_mass(a, dims->kv_dtype == DSA_BF16, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_prefill_sparse(const dsa_dims* dims, int32_t max_q, const void* q,
                              const void* k_pages, const void* v_pages,
                              const int32_t* page_table, const int32_t* seq_len,
                              const int32_t* q_len, const int32_t* prompt_len,
                              const int32_t* window, const uint32_t* keep_mask,
                              const int32_t* request_order, float scale, float* out, float* lse,
                              void* ws, void* stream) {
  const dsa_status st = check_dims(dims);
  if (st != DSA_OK) return st;
  if (max_q < 0 || !q || !k_pages || !v_pages || !page_table || !seq_len || !q_len ||
      !prompt_len || !window || !keep_mask || !out || !ws)
    return DSA_ERR_INVALID_ARG;
  if (!(scale == scale) || !aligned(ws, 256) || !aligned(q, 16) || !aligned(k_pages, 16) ||
      !aligned(v_pages, 16) || !aligned(out, 8) || !aligned(lse, 4))
    return DSA_ERR_INVALID_ARG;
  const dsa_status sm = multi_dims_ok(dims, max_q);
  if (sm != DSA_OK) return sm;
  if (dims->batch == 0 || max_q == 0) return DSA_OK;
  MultiLaunch a{};
  const dsa_status ss = multi_shape(dims, max_q, &a);
  if (ss != DSA_OK) return ss;
  a.q = q;
  a.k = k_pages;
  a.v = v_pages;
  a.page_table = page_table;
  a.seq_len = seq_len;
  a.q_len = q_len;
  a.prompt_len = prompt_len;
  a.window = window;
  a.keep_mask = keep_mask;
  a.order = request_order;
  a.scale_log2 = scale * kLog2e;
  a.out = out;
  a.lse = lse;
  a.err = err_word(ws);
  a.part = partials(ws);
  a.part_count = multi_count_region(dims, ws);
  return from_cuda(launch_multi(a, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_prefill_plan(const dsa_dims* dims, int32_t max_q, int32_t* warps, int32_t* units,
                            int32_t* whole, int32_t* parts, int32_t* ctas_per_sm, int32_t* ctas) {
  const dsa_status st = multi_dims_ok(dims, max_q);
  if (st != DSA_OK) return st;
  MultiPlan p{multi_warps(max_q, dims->hq / dims->hkv), 0, 0, 1, 0, 0};
  if (dims->batch > 0 && max_q > 0) {
    MultiLaunch a{};
    const dsa_status ss = multi_shape(dims, max_q, &a);
    if (ss != DSA_OK) return ss;
    const cudaError_t e = launch_multi(a, nullptr, &p, false);
    if (e != cudaSuccess) return from_cuda(e);
  }
  if (warps) *warps = p.warps;
  if (units) *units = p.units;
  if (whole) *whole = p.n_whole;
  if (parts) *parts = p.parts;
  if (ctas_per_sm) *ctas_per_sm = p.ctas_per_sm;
  if (ctas) *ctas = p.ctas;
  return DSA_OK;
}

dsa_status dsa_decode_plan(const dsa_dims* dims, int32_t mode, int32_t* chunk,
                           int32_t* num_chunks, int32_t* launches, int32_t* warps,
                           int32_t* tile_rows) {
  const dsa_status st = check_dims(dims);
  if (st != DSA_OK) return st;
  if (mode < kModeDense || mode > kModeMask) return DSA_ERR_INVALID_ARG;
  if (mode == kModeMask && dims->max_window > kMaskModeMaxWindow) return DSA_ERR_UNSUPPORTED;
  const Plan p = decode_plan(dims, mode);
  if (chunk) *chunk = p.chunk;
  if (num_chunks) *num_chunks = p.num_chunks;
  if (launches)
    *launches = dims->batch == 0 ? 0 : (p.num_chunks > 1 && p.cluster <= 1 ? 2 : 1);
  if (warps) *warps = p.warps;
  if (tile_rows) *tile_rows = p.tile_rows;
  return DSA_OK;
}

struct dsa_graph {
  cudaGraphExec_t exec;
};

dsa_status dsa_graph_begin(void* stream) {
  if (stream == nullptr) return DSA_ERR_INVALID_ARG;  // the legacy stream cannot record
  return from_cuda(
      cudaStreamBeginCapture(static_cast<cudaStream_t>(stream), cudaStreamCaptureModeThreadLocal));
}

dsa_status dsa_graph_end(void* stream, dsa_graph** graph) {
  if (stream == nullptr) return DSA_ERR_INVALID_ARG;
  if (graph != nullptr) *graph = nullptr;
  cudaGraph_t g = nullptr;
  // the recording ends whatever else fails, so the stream is usable again
  cudaError_t e = cudaStreamEndCapture(static_cast<cudaStream_t>(stream), &g);
  if (e != cudaSuccess || g == nullptr) {
    if (g != nullptr) cudaGraphDestroy(g);
    return DSA_ERR_CUDA;
  }
  if (graph == nullptr) {
    cudaGraphDestroy(g);
    return DSA_ERR_INVALID_ARG;
  }
  cudaGraphExec_t x = nullptr;
  e = cudaGraphInstantiate(&x, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  dsa_graph* h = new (std::nothrow) dsa_graph{x};
  if (h == nullptr) {
    cudaGraphExecDestroy(x);
    return DSA_ERR_CUDA;
  }
  *graph = h;
  return DSA_OK;
}

dsa_status dsa_graph_launch(const dsa_graph* graph, void* stream) {
  if (graph == nullptr) return DSA_ERR_INVALID_ARG;
  return from_cuda(cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_graph_destroy(dsa_graph* graph) {
  if (graph == nullptr) return DSA_OK;
  const cudaError_t e = cudaGraphExecDestroy(graph->exec);
  delete graph;
  return from_cuda(e);
}

dsa_status dsa_set_sparse_cluster(int32_t ctas) {
  if (ctas < 0 || ctas > kMaxCluster) return DSA_ERR_INVALID_ARG;
  g_sparse_cluster.store(ctas, std::memory_order_relaxed);
  return DSA_OK;
}

int32_t dsa_get_sparse_cluster(void) { return g_sparse_cluster.load(std::memory_order_relaxed); }

dsa_status dsa_set_prefill_split(int32_t parts) {
  if (parts < 0 || parts > kMultiMaxParts) return DSA_ERR_INVALID_ARG;
  g_prefill_split.store(parts, std::memory_order_relaxed);
  return DSA_OK;
}

int32_t dsa_get_prefill_split(void) { return g_prefill_split.load(std::memory_order_relaxed); }

dsa_status dsa_get_device_error(const void* ws, void* stream, int32_t* code_out) {
  if (!ws || !code_out) return DSA_ERR_INVALID_ARG;
  int32_t code = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&code, ws, sizeof(code), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSA_ERR_CUDA;
  *code_out = code;
  if (code == DSA_DEV_OK) return DSA_OK;
  return code == DSA_DEV_TIMEOUT ? DSA_ERR_TIMEOUT : DSA_ERR_DEVICE;
}

dsa_status dsa_clear_device_error(void* ws, void* stream) {
  if (!ws) return DSA_ERR_INVALID_ARG;
  return from_cuda(cudaMemsetAsync(ws, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// dsa_decode_sparse_noalloc: the sparse decode with its scratch (error word and
// split-KV partials) in a fixed array the library owns, for callers that cannot
// allocate device memory.
// ---------------------------------------------------------------------------
namespace dsa {
namespace {

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of g_noalloc_scratch on the current device (looked up once per
// device: the host-side name is only a stand-in, never a device address).
dsa_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return DSA_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_decode_sparse_noalloc(const dsa_dims* dims, const void* q,
                                                const void* k_pages, const void* v_pages,
                                                const int32_t* page_table, const int32_t* seq_len,
                                                const int32_t* kept_idx, const int32_t* kept_cnt,
                                                float scale, float* out, float* lse,
                                                int32_t* dev_error, void* stream) {
  const dsa_status st = check_dims(dims);
  if (st != DSA_OK) return st;
  if (!q || !k_pages || !v_pages || !page_table || !seq_len || !kept_idx || !kept_cnt || !out)
    return DSA_ERR_INVALID_ARG;
  // Scratch this call needs: the header plus one partial per (request, query
  // head, chunk), counted even when a single chunk leaves it unused.  The plan
  // is taken once and the launch uses it, so the split checked here is the one
  // launched even if dsa_set_sparse_cluster runs meanwhile on another thread.
  const Plan plan = decode_plan(dims, kModeList);
  const size_t need = kWsHeader + static_cast<size_t>(dims->batch) * dims->hq *
                                      static_cast<size_t>(plan.num_chunks > 0 ? plan.num_chunks
                                                                              : 1) *
                                      (dims->head_dim + 2) * sizeof(float);
  if (need > DSA_NOALLOC_SCRATCH_BYTES) return DSA_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  const dsa_status su = noalloc_scratch(&ws);
  if (su != DSA_OK) return su;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the error word (and the rest of the header) must start at zero
  if (cudaMemsetAsync(ws, 0, kWsHeader, s) != cudaSuccess) return DSA_ERR_CUDA;
  RowSource rs;
  rs.kept_idx = kept_idx;
  rs.kept_cnt = kept_cnt;
  const dsa_status rc = decode_common(dims, kModeList, q, k_pages, v_pages, page_table, seq_len,
                                      rs, scale, out, lse, ws, stream, nullptr, &plan);
  if (rc != DSA_OK) return rc;
  if (dev_error != nullptr &&
      cudaMemcpyAsync(dev_error, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return DSA_ERR_CUDA;
  return DSA_OK;
}
