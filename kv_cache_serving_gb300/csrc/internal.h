// internal.h -- host-side launch interface between the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace dsa {

// Rows of one decode / mass work unit are split into chunks of `chunk` rows;
// each chunk is one CTA.  At most kMaxChunks chunks per (request, kv head).
constexpr int kMaxChunks = 32;
// Largest cluster of decode CTAs sharing one (request, kv head).
constexpr int kMaxCluster = 8;
constexpr int kChunkQuantum = 64;  // chunk sizes are multiples of this

struct DecodeLaunch {
  const void* q;
  int q_bf16;
  const void* k;
  const void* v;
  const int32_t* page_table;
  const int32_t* seq_len;
  const int32_t* kept_idx;  // kRowsList only
  const int32_t* kept_cnt;  // kRowsList only
  const int32_t* prompt_len;  // kRowsMask only
  const int32_t* window;      // kRowsMask only
  const uint32_t* keep_mask;  // kRowsMask only: [batch][hkv][mask_words]
  int32_t* unit_rows;         // kRowsMask only: [batch][hkv] kept count or -error
  const int32_t* order;       // [batch] request scheduled at each grid z, or null (z itself)
  const int32_t* sched;       // kRowsList: [batch] schedule left by dsa_build_index, used
  const int32_t* sched_tag;   //   when *sched_tag == sched_expect (else z itself), or null
  int32_t sched_expect;
  const void* k_new;          // [batch][hkv][head_dim] K/V of row seq_len-1, or null (the
  const void* v_new;          //   cache already holds it); written into its page slot
  int32_t batch, hq, hkv, head_dim, max_pages, num_pages, max_kept;
  int32_t max_window, mask_words;  // kRowsMask only
  int32_t chunk, num_chunks;
  int32_t cluster;   // > 1: the num_chunks (== cluster) CTAs of a unit merge in a cluster
  int32_t warps;     // warps per CTA of the build to launch (see DecodeShape)
  int32_t build;     // kBuildDefault / kBuildBig / kBuildSmall (see DecodeShape)
  float scale_log2;  // softmax scale * log2(e)
  float* out;
  float* lse;
  float* part;  // [batch][hq][num_chunks][head_dim + 2]
  int32_t* err;
};

struct MassLaunch {
  const void* q;
  int q_bf16;
  const void* k;
  const int32_t* page_table;
  const int32_t* seq_len;
  const int32_t* prompt_len;
  const int32_t* window;
  const int32_t* grid_w;
  int32_t batch, hq, hkv, head_dim, max_pages, num_pages, max_window;
  int32_t r_local, r_diag;
  int32_t chunk, num_chunks;
  float scale_log2;
  float* mass;         // [batch][hq][4]
  float* offset_mass;  // [batch][hq][max_window+1] or null
  float* part;         // [batch][hq][num_chunks][6]
  int32_t* err;
};

struct CompactLaunch {
  const int32_t* seq_len;
  const int32_t* prompt_len;
  const int32_t* window;
  const uint32_t* keep_mask;
  int32_t* kept_idx;
  int32_t* kept_cnt;
  int32_t batch, hkv, max_pages, max_window, mask_words, max_kept;
  int32_t* err;
  int32_t* sched;       // [batch] requests by decreasing kept rows (written by the last CTA)
  int32_t* sched_tag;   // set to kSchedMagic ^ batch once sched is written
  int32_t* done_count;  // CTAs done; zero between calls
};

struct EvictLaunch {
  const int32_t* seq_len;
  const int32_t* prompt_len;
  const int32_t* window;
  int32_t* page_table;   // [batch][max_pages], evicted entries set to -1
  int32_t* freed;        // [capacity] freed page ids
  int32_t* freed_count;  // appended to atomically
  int32_t batch, max_pages, max_window, capacity;
  int32_t* err;
};

// Several query tokens per request (prefill.cu): q [batch][max_q][hq][head_dim].
struct MultiLaunch {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* page_table;
  const int32_t* seq_len;
  const int32_t* q_len;       // [batch] query tokens of each request (its last rows)
  const int32_t* prompt_len;
  const int32_t* window;
  const uint32_t* keep_mask;  // [batch][hkv][mask_words]
  const int32_t* order;       // [batch] request handed to the GPU at each position, or null
  int32_t batch, hq, hkv, head_dim, max_pages, num_pages, max_window, mask_words, max_q;
  int32_t q_tiles;            // CTAs along the query axis of one (request, kv head)
  int32_t warps;              // warps per CTA (multi_warps)
  float scale_log2;
  float* out;                 // [batch][max_q][hq][head_dim]
  float* lse;                 // [batch][max_q][hq] or null
  int32_t* err;
  // Units are (query tile, kv head, request) in that order, x fastest.  The first
  // n_whole run whole, one CTA each; every later one is split along its scanned
  // rows into `split` parts whose partial states the unit's last-arriving part
  // merges.  Filled by launch_multi from the fields below it.
  int32_t n_whole, split;
  float* part;                // [split unit][part][16 warps][head_dim + 2]
  int32_t* part_count;        // [split unit] arrivals, 0 between launches
  // host only: split setting (0 automatic, 1 never, n: every unit in n parts),
  // partial rows the workspace holds, arrival counters it holds, SMs
  int32_t split_setting;
  int64_t part_rows_cap;
  int32_t count_cap, sms;
};

// Row sources of a decode launch (`mode` below).
constexpr int kModeDense = 0;  // rows 0..L-1
constexpr int kModeList = 1;   // kept_idx / kept_cnt from dsa_build_index
constexpr int kModeMask = 2;   // kept set built in the kernel from keep_mask

// Largest max_window of kModeMask: the kernel holds the window's mask bits one
// 32-bit word per lane of a warp.
constexpr int kMaskModeMaxWindow = 1024;

// Each returns cudaSuccess or the launch error.
cudaError_t launch_decode_bf16(const DecodeLaunch& a, int mode, cudaStream_t s);
cudaError_t launch_decode_f32(const DecodeLaunch& a, int mode, cudaStream_t s);
cudaError_t launch_merge(const DecodeLaunch& a, int mode, cudaStream_t s);
cudaError_t launch_mass(const MassLaunch& a, bool kv_bf16, cudaStream_t s);
// Rows one pass of all warps of an attention-mass CTA covers, and its resident
// CTAs per SM (>= 1), for the host's chunk choice.
int mass_rows_per_pass(int head_dim, int group, bool kv_bf16, bool q_bf16);
// The attention-mass build for these dtypes scores on the tensor cores.
bool mass_uses_tensor_cores(bool kv_bf16, bool q_bf16, int group);
int mass_ctas_per_sm(int head_dim, int group, bool kv_bf16, bool q_bf16);
cudaError_t launch_compact(const CompactLaunch& a, cudaStream_t s);
// Several query tokens per request: bf16 q and KV only.  Warps per CTA for a
// call (2 when max_q x group fits 32 (query, head) rows, else 4) and the query
// tokens a CTA of that many warps holds.
// The launch of a multi-query call: warps per CTA, units, units run whole,
// parts of each later unit, resident CTAs per SM, CTAs launched.
struct MultiPlan {
  int32_t warps, units, n_whole, parts, ctas_per_sm, ctas;
};
// Plans the launch (into *plan when not null) and launches it unless `launch`
// is false (then nothing is enqueued).
cudaError_t launch_multi(const MultiLaunch& a, cudaStream_t s, MultiPlan* plan = nullptr,
                         bool launch = true);
int multi_warps(int max_q, int group);
int multi_queries_per_cta(int warps, int group);
// Largest max_window of the multi-query call (its mask words sit in shared memory).
constexpr int kMultiMaxWindow = 32768;
// Arrival counters of split multi-query units in the workspace, and the most
// parts a unit is split into.
constexpr int kMultiCounters = 4096;
constexpr int kMultiMaxParts = 8;
// Resident warps per SM of the multi-query kernel the workspace's partials
// region is sized for (6 CTAs of 2 warps, or 3 of 4).
constexpr int kMultiPartWarpsPerSm = 12;
cudaError_t launch_evict(const EvictLaunch& a, cudaStream_t s);

// Host copies of a step (hostio.cu): a copy kernel when the host side is
// page-locked memory the device can address, else cudaMemcpyAsync.
cudaError_t copy_host_to_device(void* dev, const void* host, size_t bytes, cudaStream_t s);
cudaError_t copy_device_to_host(void* host, const void* dev, size_t bytes, cudaStream_t s);

// Builds of the decode kernel.  The sparse calls with bf16 KV have three more
// besides the default: one for batches of more than two waves of units (more
// warps per SM), one for batches that fit one wave only with it (5 warps of a
// single stage, each warp about one tile of a unit), and one for batches of at
// most one unit per SM (8 warps of a single stage: a unit's rows spread over
// the warps of one CTA, merged in its shared memory, no cluster).
enum : int { kBuildDefault = 0, kBuildBig = 1, kBuildSmall = 2, kBuildWide = 3 };

// Host-side facts about one build of the decode kernel, for the chunk choice.
struct DecodeShape {
  int rows_per_pass;  // warps x tile rows
  int ctas_per_sm;    // resident CTAs per SM (>= 1)
  int cluster_limit;  // largest cluster whose merge buffer fits the rings
  int warps;          // warps per CTA of this build
  int tile_rows;      // rows per tile of this build
  int build;          // which build this is
};
// The requested build of (head_dim, group, mode) when there is one, else the
// default build.
DecodeShape decode_shape_bf16(int head_dim, int group, int mode, int build);
DecodeShape decode_shape_f32(int head_dim, int group, int mode, int build);

}  // namespace dsa
