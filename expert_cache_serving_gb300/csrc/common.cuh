// Shared definitions of the moecache CUDA library (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moecache.h"

namespace moe {

constexpr int kMaxE = 1024;          // experts per layer
constexpr int kMaxK = 16;            // experts per token
constexpr int kMaxB = 16;            // tokens per decode call
constexpr int kMaxPairs = kMaxB * kMaxK;
constexpr int kMaxU = kMaxPairs;     // distinct experts per call
constexpr int kMaxItems = kMaxU + 1; // + shared expert
constexpr int kCtrlThreads = 1024;
constexpr int kFfnThreads = 512;
constexpr int kFfnWarps = kFfnThreads / 32;

// Per-call plan written by the control kernel into device memory and read by
// the expert-FFN kernels of the same call.
struct Plan {
  int32_t err;        // MOE_OK or MOE_ERR_CAPACITY
  int32_t B, k, n_u, n_miss;
  int32_t n_items[2];             // [0]: resident experts (+ shared), [1]: fills
  int32_t items[2][kMaxItems];    // rank r in U, or n_u for the shared expert
  int32_t u_expert[kMaxU];        // U ascending
  int32_t u_slot[kMaxU];          // slot after the call
  int32_t u_fill[kMaxU];          // 1 if the expert is filled by this call
  int32_t u_off[kMaxU + 1];       // group starts in perm
  int32_t perm[kMaxPairs];        // flat pair t*k+j grouped by expert (stable)
  int32_t pair_rank[kMaxPairs];   // rank in U of each flat pair
  float pair_w[kMaxPairs];        // routing weight of each flat pair
};

// Host-visible (pinned, mapped) summary of one call: the miss list the host
// needs to issue the fills, the undo log, and a sequence number written last.
struct HostWork {
  volatile uint32_t seq;
  int32_t err;
  int32_t n_u, n_miss;
  uint64_t g_before;
  int32_t key[kMaxU];
  int32_t slot[kMaxU];
  int32_t evicted[kMaxU];
  int32_t fill[kMaxU];
  int32_t pairs[kMaxU];        // routed pairs of this expert
  uint64_t old_stamp[kMaxU];   // stamp of the slot before the call
};

struct CacheDev {
  int32_t* map;      // [L*E] key -> slot or -1
  int32_t* owner;    // [C_max] slot -> key or -1
  uint64_t* stamp;   // [C_max]
  uint64_t* g;       // global recency counter
};

// ---------------------------------------------------------------- helpers --

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Exclusive block-wide prefix sum of one int per thread; *total gets the sum.
// scratch: >= 33 ints of shared memory.  All threads of the block must call.
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) scratch[lane] = s;  // inclusive per-warp sums
    if (lane == 31) scratch[32] = s;
  }
  __syncthreads();
  int before = (warp ? scratch[warp - 1] : 0) + x - v;
  *total = scratch[32];
  __syncthreads();
  return before;
}

// Grid-wide barrier for a cooperative launch.  The spin gives up after
// ~`limit_ns` nanoseconds, records MOE_ERR_TIMEOUT in *err and returns false.
__device__ __forceinline__ bool grid_barrier(unsigned* count, unsigned* gen, int* err,
                                             unsigned long long limit_ns = 2000000000ull) {
  __shared__ int s_ok;
  __threadfence();  // publish this thread's global writes before arriving
  __syncthreads();
  if (threadIdx.x == 0) {
    s_ok = 1;
    const unsigned nblocks = gridDim.x * gridDim.y * gridDim.z;
    volatile unsigned* vgen = gen;
    unsigned my_gen = *vgen;
    __threadfence();
    unsigned arrived = atomicAdd(count, 1u);
    if (arrived == nblocks - 1) {
      atomicExch(count, 0u);
      __threadfence();
      atomicAdd(gen, 1u);
    } else {
      unsigned long long t0;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
      while (*vgen == my_gen) {
        __nanosleep(64);
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > limit_ns) {
          atomicExch(err, MOE_ERR_TIMEOUT);
          s_ok = 0;
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
  return s_ok != 0;
}

}  // namespace moe
