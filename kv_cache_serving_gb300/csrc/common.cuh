// common.cuh -- device helpers shared by the libdsa kernels (sm_103a).
//
// Row gathers use the Blackwell bulk-copy engine: one lane issues a
// cp.async.bulk of a whole K or V row (head_dim elements, 128-512 bytes,
// 16-byte aligned) from global memory into shared memory, completing on an
// mbarrier that carries the expected byte count.  Waits on mbarriers are
// bounded: after kWaitLimitNs a kernel records DSA_DEV_TIMEOUT and stops.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "dsa.h"

namespace dsa {

constexpr int kPage = 16;
constexpr uint64_t kWaitLimitNs = 500ull * 1000 * 1000;  // give up on a copy after 0.5 s
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Workspace: [0, 256) header, then per-call regions.  Header words: 0 the
// device error word; 1 the tag of the request schedule dsa_build_index leaves
// for dsa_decode_sparse (kSchedMagic ^ batch when valid); 2 the count of
// index-compaction CTAs done (the last one writes the schedule, then resets it).
constexpr size_t kWsHeader = 256;
constexpr int kWsSchedTag = 1;
constexpr int kWsDoneCount = 2;
constexpr int32_t kSchedMagic = 0x5c4ed000;
// Largest batch whose schedule the index compaction sorts (one CTA, rank sort).
constexpr int kSchedMaxBatch = 1024;

__device__ __forceinline__ void set_error(int32_t* err, int32_t code) {
  atomicCAS(err, 0, code);
}

// Programmatic dependent launch (a no-op for grids launched without it):
// griddep_wait() returns once the grids this one depends on have completed and
// their writes are visible; griddep_launch_dependents() lets the next grid on
// the stream be scheduled once every CTA of this one has issued it.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#ifndef DSA_PDL
#define DSA_PDL 1  // kernels launch as programmatic dependents (0: plain launches)
#endif

// kern<<<grid, block, smem, s>>>(args...) as a programmatic dependent launch:
// the grid may be scheduled while the previous kernel on the stream drains.
// Every libdsa kernel starts with griddep_wait(), so none touches memory before
// its predecessor has completed.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = DSA_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Plain arrival (no transaction bytes), release semantics at CTA scope.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// 2^x by the hardware approximation (ex2.approx.ftz: relative error about
// 2^-22, subnormal results flushed to zero, 2^-inf = +0), for the online
// softmax weights and rescale factors.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait for phase `parity` of `bar` to complete: false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int it = 0; it < 64; ++it)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// 16 bytes global -> shared through the L2 (cp.async, completion tracked below).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
// One arrival on `bar` once every cp.async this thread issued so far has landed
// (the barrier's count must include it).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) writes to the same shared memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One bulk copy global -> shared; `bytes` and both addresses are multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// element loads: N consecutive elements -> fp32 registers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

struct bf16_t {
  uint16_t bits;
};

template <typename T, int N>
struct Vec;

template <>
struct Vec<float, 2> {
  __device__ __forceinline__ static void load(const float* p, float* o) {
    float2 v = *reinterpret_cast<const float2*>(p);
    o[0] = v.x;
    o[1] = v.y;
  }
};
template <>
struct Vec<float, 4> {
  __device__ __forceinline__ static void load(const float* p, float* o) {
    float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x;
    o[1] = v.y;
    o[2] = v.z;
    o[3] = v.w;
  }
};
template <>
struct Vec<bf16_t, 2> {
  __device__ __forceinline__ static void load(const bf16_t* p, float* o) {
    uint32_t v = *reinterpret_cast<const uint32_t*>(p);
    o[0] = bf16_lo(v);
    o[1] = bf16_hi(v);
  }
};
template <>
struct Vec<bf16_t, 4> {
  __device__ __forceinline__ static void load(const bf16_t* p, float* o) {
    uint2 v = *reinterpret_cast<const uint2*>(p);
    o[0] = bf16_lo(v.x);
    o[1] = bf16_hi(v.x);
    o[2] = bf16_lo(v.y);
    o[3] = bf16_hi(v.y);
  }
};

// q[DPL] of one head from global memory, either dtype, scaled.
template <int DPL>
__device__ __forceinline__ void load_q(const void* q, bool q_bf16, size_t elem, float mul,
                                       float* o) {
  if (q_bf16)
    Vec<bf16_t, DPL>::load(reinterpret_cast<const bf16_t*>(q) + elem, o);
  else
    Vec<float, DPL>::load(reinterpret_cast<const float*>(q) + elem, o);
#pragma unroll
  for (int e = 0; e < DPL; ++e) o[e] *= mul;
}

// ---------------------------------------------------------------------------
// warp reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Reduce-scatter of T per-lane partial sums across the 32 lanes of a warp:
// on return, lane l holds the full warp sum of v[row] for row = l >> (5 - log2 T)
// (each row's sum is replicated on 32/T lanes).  Each halving step sends half
// of the remaining values to the partner lane and keeps the other half.
template <int T>
__device__ __forceinline__ float reduce_scatter(float (&v)[T], int lane) {
  static_assert(T == 8 || T == 16 || T == 32, "tile rows");
#pragma unroll
  for (int n = T, off = 16; n > 1; n >>= 1, off >>= 1) {
    const bool hi = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float lo_v = v[i], hi_v = v[i + n / 2];
      const float send = hi ? lo_v : hi_v;
      const float keep = hi ? hi_v : lo_v;
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float s = v[0];
#pragma unroll
  for (int off = 32 / T / 2; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

template <int T>
struct RowMap {
  static constexpr int kShift = (T == 32) ? 0 : (T == 16 ? 1 : 2);
  __device__ __forceinline__ static int row(int lane) { return lane >> kShift; }
  __device__ __forceinline__ static bool owner(int lane) {
    return (lane & ((1 << kShift) - 1)) == 0;
  }
};

// ---- thread-block clusters ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of all CTAs of the cluster; orders shared-memory accesses
// (local and distributed) before the barrier with those after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address in CTA `rank`'s shared memory of the variable at local address p.
__device__ __forceinline__ uint32_t map_cluster_rank(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

}  // namespace dsa
