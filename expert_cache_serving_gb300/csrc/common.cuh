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
constexpr int kThreads = 512;  // layer kernel CTA size
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFlagError = 0x80000000u;  // fill flag: the copy was not issued
// Bounds checks of the debug build (compiled with -DMOE_DEBUG_BOUNDS, the
// stand-in for a memory checker): in_bounds(dbg, ok, site) is true when the
// index it guards is valid; when it is not, the debug build counts the
// violation in dbg[0], keeps the first site in dbg[1] and returns false so
// the caller skips the access.  The release build checks nothing (always
// true; the condition is dead code).
__device__ __forceinline__ bool in_bounds(unsigned* dbg, bool ok, unsigned site) {
#ifdef MOE_DEBUG_BOUNDS
  if (!ok) {
    if (dbg) {
      atomicAdd(dbg, 1u);
      atomicCAS(dbg + 1, 0u, site);
    }
    return false;
  }
#else
  (void)dbg;
  (void)ok;
  (void)site;
#endif
  return true;
}

constexpr int kWaveCtrs = 16;  // per-call counters of the layer kernel (two sets, by call parity)

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
  int32_t u_key[kMaxU];           // undo log: key of each member of U
  uint64_t u_old_stamp[kMaxU];    // undo log: stamp of its slot before the call
  uint64_t g_before;              // undo log: counter before the call
};

// Host-visible (pinned, mapped) summary of one call: the miss list the host
// needs to issue the fills, the undo log, and a sequence number written last.
constexpr int kSummaryRing = 256;  // host summaries in flight (one per call, by call sequence number)
struct HostWork {
  volatile uint32_t seq;
  int32_t err;
  int32_t layer, B;             // the call's layer and token count
  int32_t n_u, n_miss;
  uint64_t g_before;
  int32_t key[kMaxU];
  int32_t slot[kMaxU];
  int32_t evicted[kMaxU];
  int32_t fill[kMaxU];
  int32_t pairs[kMaxU];        // routed pairs of this expert
  int32_t fill_order[kMaxU];   // f-th fill the kernel consumes -> rank in U
  int32_t qstar;               // fill count of the bandwidth split for this call's misses
};

// Completion state of one decode call in copy-fill mode, read by the
// completion kernel that runs after the call's copies: whether the layer
// kernel stopped waiting for a fill's gate/up half (then the completion
// kernel computes every fill), and per CTA how many fills its saved partial
// sums already hold (-1: the CTA wrote its outputs itself).
constexpr int kMaxGrid = 1024;
struct CallState {
  int gu_stop;             // a CTA gave up waiting for a first (gate/up) half
  int pad[31];
  int part[kMaxGrid];      // per CTA: -1 complete, >= 0 fills in its saved sums, -2 failed fill
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

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---- shared-memory addresses, mbarriers and 1-D bulk copies ------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Wait for the phase with the given parity; false on time-out (~limit_ns).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns = 2000000000ull) {
  const uint32_t a = smem_u32(bar);
  unsigned long long t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 255) == 0) {
      const unsigned long long t = globaltimer_ns();
      if (t0 == 0) t0 = t;
      else if (t - t0 > limit_ns) return false;
    }
  }
}

// 1-D bulk copy global -> shared (the async proxy), completing `bytes` on the
// mbarrier, L2 evict-first (streamed weights).  dst, src and bytes must be
// multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "{\n .reg .b64 pol;\n createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n"
      " cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], pol;\n}\n"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Grid-wide barrier of a launch whose CTAs are all resident, over a counter
// that only grows and that only full grids of gridDim.x CTAs arrive at:
// arrival number a belongs to the barrier that completes when the counter
// reaches (a / G + 1) * G, so no base has to be carried from launch to launch.
// The wait gives up after limit_ns, records MOE_ERR_TIMEOUT in *err and
// returns false (the counter is then out of step until the host resets it).
__device__ __forceinline__ bool grid_barrier(unsigned long long* count, int* err,
                                             unsigned long long limit_ns = 2000000000ull) {
  __shared__ int s_ok;
  __syncthreads();  // the CTA's global writes happen before thread 0's fence (cumulative)
  if (threadIdx.x == 0) {
    s_ok = 1;
    const unsigned long long G = gridDim.x;
    __threadfence();  // publish the CTA's writes before arriving
    const unsigned long long target = (atomicAdd(count, 1ull) / G + 1) * G;
    const unsigned long long t0 = globaltimer_ns();
    while (ld_acquire_u64(count) < target) {
      __nanosleep(32);
      if (globaltimer_ns() - t0 > limit_ns) {
        atomicExch(err, MOE_ERR_TIMEOUT);
        s_ok = 0;
        break;
      }
    }
    __threadfence();
  }
  __syncthreads();
  return s_ok != 0;
}

// Wait until *flag == want (returns 0) or want | kFlagError (returns 1).
// Gives up (returns 2) after limit_ns, or as soon as *stop becomes non-zero
// when stop is given.  Thread 0 polls, the CTA waits on it.  Giving up is
// not an error here: the caller decides what it means.
__device__ __forceinline__ int wait_flag(const unsigned* flag, unsigned want, const int* stop,
                                         unsigned long long limit_ns, unsigned sleep_ns = 256) {
  __shared__ int s_res;
  __syncthreads();
  if (threadIdx.x == 0) {
    int res = 2;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
      // relaxed polling at GPU scope, one acquire fence once the value is seen
      // (system-scope acquires from every CTA slowed the copy engine down)
      unsigned v;
      asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
      if (v == want || v == (want | kFlagError)) {
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        res = v == want ? 0 : 1;
        break;
      }
      if (stop) {
        int sv;
        asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(sv) : "l"(stop) : "memory");
        if (sv) break;
      }
      if (globaltimer_ns() - t0 >= limit_ns) break;
      __nanosleep(sleep_ns);
    }
    s_res = res;
  }
  __syncthreads();
  return s_res;
}

// Programmatic dependent launch: wait until the previous launch on the stream
// has completed and its memory is visible (a no-op when the kernel was not
// launched as a dependent), and let the next launch begin its start-up.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace moe
