// Per-layer cache control for decode: routing, deduplication, residency
// lookup, LRU restamp, one-pass victim selection, id -> slot rewrite and the
// stable grouping of (token, rank) pairs by expert.
//
// FreeToken write-up, "CUDA Graph-compatible LRU cache": one GPU kernel per
// MoE layer deduplicates the routed experts, classifies them against the
// residency table, selects eviction victims and rewrites logical routing ids
// to physical slot ids; victim selection finds K candidate slots in a single
// pass and the miss path consumes the first q <= K of them, whatever the
// number of misses.  "Router-following LRU cache": a hit refreshes recency, a
// fill admits the selected expert, eviction removes the expert not requested
// for the longest time.
//
// Deterministic rules (shared with the CPU reference simulator by
// specification, not by code):
//  * top-k by logit, descending, ties to the lower expert id (NaN counts as
//    -inf); weights = softmax over the k selected logits;
//  * U = sorted distinct routed experts; member of rank r gets stamp g + r;
//    then g += |U|;
//  * victims: among slots not holding a hit of this call, empty slots first
//    by index, then occupied slots by ascending stamp; the i-th miss (in
//    ascending expert order) takes the i-th victim.
#include <float.h>

#include "params.cuh"

namespace moe {



// logits[t][e] = sum_h x[t][h] * W_r[e][h] in float32; one warp per (t, e).
template <typename XT>
__global__ void router_logits_kernel(const XT* __restrict__ x, const float* __restrict__ wr, int B, int E, int H,
                                     float* __restrict__ logits) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= B * E) return;
  const int t = warp / E, e = warp % E;
  const XT* xr = x + (size_t)t * H;
  const float* w = wr + (size_t)e * H;
  float acc = 0.f;
  for (int h = lane; h < H; h += 32) {
    float xv;
    if constexpr (sizeof(XT) == 2)
      xv = __bfloat162float(xr[h]);
    else
      xv = xr[h];
    acc = fmaf(xv, w[h], acc);
  }
  acc = warp_sum(acc);
  if (lane == 0) logits[warp] = acc;
}

__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}

__global__ void __launch_bounds__(kCtrlThreads) ctrl_kernel(CtrlParams p) {
  __shared__ int s_ids[kMaxPairs];
  __shared__ float s_w[kMaxPairs];
  __shared__ int s_prank[kMaxPairs];
  __shared__ unsigned s_bits[kMaxE / 32];
  __shared__ int s_wpre[kMaxE / 32];
  __shared__ int s_U[kMaxU];
  __shared__ int s_slot[kMaxU];
  __shared__ int s_fill[kMaxU];
  __shared__ int s_mrank[kMaxU];
  __shared__ int s_cnt[kMaxU];
  __shared__ int s_off[kMaxU + 1];
  __shared__ int s_victim[kMaxU];
  __shared__ unsigned long long s_vkey[kMaxU];
  __shared__ int s_scan[33];
  __shared__ unsigned s_hist[2048];
  __shared__ int s_nu, s_nmiss, s_nvict, s_err;
  __shared__ unsigned long long s_g, s_kmin, s_kmax, s_prefix;
  __shared__ int s_remaining, s_bin;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E, k = p.k, B = p.B, npairs = B * k;
  const int64_t C = p.C;
  Plan* plan = p.plan;

  for (int i = tid; i < p.n_bar_reset; i += blockDim.x) p.bar_reset[i] = 0u;

  // ---- 1. router: one warp per token ----------------------------------------
  for (int t = warp; t < B; t += blockDim.x / 32) {
    const float* lg = p.logits + (size_t)t * E;
    if (p.aux_logits)
      for (int e = lane; e < E; e += 32) p.aux_logits[(size_t)t * E + e] = lg[e];
    int sel[kMaxK];
    float selv[kMaxK];
    for (int r = 0; r < k; ++r) {
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
      for (int e = lane; e < E; e += 32) {
        bool taken = false;
        for (int q = 0; q < r; ++q) taken |= (sel[q] == e);
        if (taken) continue;
        float v = lg[e];
        if (v != v) v = -INFINITY;
        if (better(v, e, bv, bi)) { bv = v; bi = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
        int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      sel[r] = bi;
      selv[r] = bv;
    }
    if (lane == 0) {
      float m = selv[0], sum = 0.f, ex[kMaxK];
      for (int r = 0; r < k; ++r) { ex[r] = expf(selv[r] - m); sum += ex[r]; }
      for (int r = 0; r < k; ++r) {
        s_ids[t * k + r] = sel[r];
        s_w[t * k + r] = ex[r] / sum;
      }
    }
  }
  for (int i = tid; i < kMaxE / 32; i += blockDim.x) s_bits[i] = 0u;
  if (tid == 0) { s_err = MOE_OK; s_g = *p.st.g; s_nvict = 0; }
  __syncthreads();

  // ---- 2. dedup: U = sorted distinct routed experts --------------------------
  if (tid < npairs) atomicOr(&s_bits[s_ids[tid] >> 5], 1u << (s_ids[tid] & 31));
  __syncthreads();
  const int nwords = (E + 31) / 32;
  if (warp == 0) {
    int c = lane < nwords ? __popc(s_bits[lane]) : 0, x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane < nwords) s_wpre[lane] = x - c;
    if (lane == 31) s_nu = x;
  }
  __syncthreads();
  const int n_u = s_nu;
  if (tid < n_u) s_cnt[tid] = 0;
  __syncthreads();
  if (tid < npairs) {
    int e = s_ids[tid];
    int r = s_wpre[e >> 5] + __popc(s_bits[e >> 5] & ((1u << (e & 31)) - 1u));
    s_prank[tid] = r;
    s_U[r] = e;
    atomicAdd(&s_cnt[r], 1);
  }
  if (tid == 0 && n_u > C) s_err = MOE_ERR_CAPACITY;
  __syncthreads();
  if (s_err != MOE_OK) {
    if (tid == 0) {
      plan->err = s_err;
      plan->B = B; plan->k = k; plan->n_u = n_u; plan->n_miss = 0;
      plan->n_items[0] = 0; plan->n_items[1] = 0;
      p.work->err = s_err; p.work->n_u = n_u; p.work->n_miss = 0; p.work->g_before = s_g;
      __threadfence_system();
      p.work->seq = p.seq;
    }
    return;
  }

  // ---- 3. classify against the residency table --------------------------------
  int is_miss = 0;
  if (tid < n_u) {
    int key = p.layer * E + s_U[tid];
    int s = p.st.map[key];
    s_slot[tid] = s;
    is_miss = s < 0;
    s_fill[tid] = is_miss;
  }
  int nmiss;
  int mr = block_excl_scan(is_miss, s_scan, &nmiss);
  if (tid < n_u) s_mrank[tid] = mr;
  if (tid == 0) s_nmiss = nmiss;
  __syncthreads();

  // ---- 4. one-pass selection of the n_miss oldest candidate slots -------------
  // candidate key: empty slot s -> s; occupied -> C + stamp; hit slots excluded
  if (nmiss > 0) {
    auto cand_key = [&](int64_t s, unsigned long long* out) -> bool {
      int own = p.st.owner[s];
      if (own < 0) { *out = (unsigned long long)s; return true; }
      if (own / E == p.layer) {
        int e = own % E;
        if (s_bits[e >> 5] & (1u << (e & 31))) return false;  // a hit of this call
      }
      *out = (unsigned long long)C + p.st.stamp[s];
      return true;
    };
    unsigned long long lmin = ~0ull, lmax = 0ull;
    for (int64_t s = tid; s < C; s += blockDim.x) {
      unsigned long long kk;
      if (cand_key(s, &kk)) { lmin = min(lmin, kk); lmax = max(lmax, kk); }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lmin = min(lmin, __shfl_xor_sync(0xFFFFFFFFu, lmin, o));
      lmax = max(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
    }
    if (tid == 0) { s_kmin = ~0ull; s_kmax = 0ull; s_prefix = 0ull; s_remaining = nmiss; }
    __syncthreads();
    if (lane == 0) { atomicMin(&s_kmin, lmin); atomicMax(&s_kmax, lmax); }
    __syncthreads();
    const unsigned long long kmin = s_kmin, span = s_kmax - s_kmin;
    const int nbits = span ? 64 - __clzll((long long)span) : 1;
    const int passes = (nbits + 10) / 11;
    for (int pass = passes - 1; pass >= 0; --pass) {
      const int shift = pass * 11;
      for (int i = tid; i < 2048; i += blockDim.x) s_hist[i] = 0u;
      __syncthreads();
      const unsigned long long prefix = s_prefix;
      const int hs = shift + 11;
      for (int64_t s = tid; s < C; s += blockDim.x) {
        unsigned long long kk;
        if (!cand_key(s, &kk)) continue;
        unsigned long long d = kk - kmin;
        if (hs < 64 && (d >> hs) != (prefix >> hs)) continue;
        atomicAdd(&s_hist[(d >> shift) & 2047ull], 1u);
      }
      __syncthreads();
      // find the bin where the running count reaches s_remaining
      int c0 = s_hist[2 * tid], c1 = s_hist[2 * tid + 1];
      int tot;
      int before = block_excl_scan(c0 + c1, s_scan, &tot);
      const int rem = s_remaining;
      __syncthreads();
      if (before < rem && rem <= before + c0) { s_bin = 2 * tid; s_remaining = rem - before; }
      else if (before + c0 < rem && rem <= before + c0 + c1) { s_bin = 2 * tid + 1; s_remaining = rem - before - c0; }
      __syncthreads();
      if (tid == 0) s_prefix = prefix | ((unsigned long long)s_bin << shift);
      __syncthreads();
    }
    const unsigned long long thr = s_prefix;  // offset of the nmiss-th smallest key
    for (int64_t s = tid; s < C; s += blockDim.x) {
      unsigned long long kk;
      if (!cand_key(s, &kk)) continue;
      if (kk - kmin <= thr) {
        int pos = atomicAdd(&s_nvict, 1);
        if (pos < kMaxU) { s_victim[pos] = (int)s; s_vkey[pos] = kk; }
      }
    }
    __syncthreads();
    if (s_nvict != nmiss) {  // cannot happen with consistent state; never write outside the table
      if (tid == 0) {
        plan->err = MOE_ERR_CUDA;
        plan->n_items[0] = 0; plan->n_items[1] = 0;
        p.work->err = MOE_ERR_CUDA; p.work->n_u = n_u; p.work->n_miss = 0; p.work->g_before = s_g;
        __threadfence_system();
        p.work->seq = p.seq;
      }
      return;
    }
    // order the (unique) selected keys ascending
    int vslot = -1;
    int vrank = -1;
    if (tid < nmiss) {
      unsigned long long mine = s_vkey[tid];
      vslot = s_victim[tid];
      vrank = 0;
      for (int j = 0; j < nmiss; ++j) vrank += s_vkey[j] < mine;
    }
    __syncthreads();
    if (tid < nmiss) s_victim[vrank] = vslot;
    __syncthreads();
  }

  // ---- 5. apply: restamp hits, assign victims to misses, log undo data -------
  const unsigned long long g0 = s_g;
  if (tid < n_u) {
    const int key = p.layer * E + s_U[tid];
    p.work->key[tid] = key;
    p.work->pairs[tid] = s_cnt[tid];
    if (!s_fill[tid]) {
      const int s = s_slot[tid];
      p.work->old_stamp[tid] = p.st.stamp[s];
      p.st.stamp[s] = g0 + tid;
      p.work->slot[tid] = s;
      p.work->evicted[tid] = -1;
      p.work->fill[tid] = 0;
    } else {
      const int v = s_victim[s_mrank[tid]];
      const int ev = p.st.owner[v];
      p.work->old_stamp[tid] = p.st.stamp[v];
      if (ev >= 0) p.st.map[ev] = -1;
      p.st.map[key] = v;
      p.st.owner[v] = key;
      p.st.stamp[v] = g0 + tid;
      s_slot[tid] = v;
      p.work->slot[tid] = v;
      p.work->evicted[tid] = ev;
      p.work->fill[tid] = 1;
    }
  }
  if (tid == 0) *p.st.g = g0 + n_u;

  // ---- 6. stable grouping of the pairs by expert (block-scan histogram) -------
  int tot;
  int off = block_excl_scan(tid < n_u ? s_cnt[tid] : 0, s_scan, &tot);
  if (tid < n_u) s_off[tid] = off;
  if (tid == 0) s_off[n_u] = npairs;
  __syncthreads();
  if (tid < npairs) {
    const int r = s_prank[tid];
    int before = 0;
    for (int q = 0; q < tid; ++q) before += (s_prank[q] == r);
    const int pos = s_off[r] + before;
    plan->perm[pos] = tid;
    plan->pair_rank[tid] = r;
    plan->pair_w[tid] = s_w[tid];
    if (p.aux_perm) p.aux_perm[pos] = tid;
    if (p.aux_ids) p.aux_ids[tid] = s_ids[tid];
    if (p.aux_w) p.aux_w[tid] = s_w[tid];
    if (p.aux_slots) p.aux_slots[tid] = s_slot[r];
  }
  if (p.aux_offsets) {
    for (int e = tid; e <= E; e += blockDim.x) {
      int r = (e < E) ? s_wpre[e >> 5] + __popc(s_bits[e >> 5] & ((1u << (e & 31)) - 1u)) : n_u;
      p.aux_offsets[e] = r < n_u ? s_off[r] : npairs;
    }
  }
  if (tid < n_u) {
    plan->u_expert[tid] = s_U[tid];
    plan->u_slot[tid] = s_slot[tid];
    plan->u_fill[tid] = s_fill[tid];
  }
  if (tid <= n_u) plan->u_off[tid] = s_off[tid];
  // item lists: resident experts then the shared expert (index n_u); fills
  int is_res = tid < n_u && !s_fill[tid];
  int nres;
  int rpos = block_excl_scan(is_res, s_scan, &nres);
  if (is_res) plan->items[0][rpos] = tid;
  if (tid < n_u && s_fill[tid]) plan->items[1][s_mrank[tid]] = tid;
  if (tid == 0) {
    if (p.has_shared) plan->items[0][nres] = n_u;  // the shared expert is item index n_u
    plan->err = MOE_OK;
    plan->B = B;
    plan->k = k;
    plan->n_u = n_u;
    plan->n_miss = s_nmiss;
    plan->n_items[0] = nres + (p.has_shared ? 1 : 0);
    plan->n_items[1] = s_nmiss;
    p.work->err = MOE_OK;
    p.work->n_u = n_u;
    p.work->n_miss = s_nmiss;
    p.work->g_before = g0;
  }
  __threadfence_system();  // every writer publishes its part of the host summary
  __syncthreads();
  if (tid == 0) {
    __threadfence_system();
    p.work->seq = p.seq;
  }
}

// Undo of a call whose fills could not be issued: recency and the counter go
// back to their values before the call; every victim slot of the call is left
// empty, because its previous contents may already have been overwritten.


__global__ void undo_kernel(UndoParams p) {
  const HostWork* w = p.work;
  const int n_u = w->n_u;
  for (int r = threadIdx.x; r < n_u; r += blockDim.x) {
    const int s = w->slot[r];
    if (!w->fill[r]) {
      p.st.stamp[s] = w->old_stamp[r];
    } else {
      p.st.map[w->key[r]] = -1;
      p.st.owner[s] = -1;
      p.st.stamp[s] = 0;
    }
  }
  if (threadIdx.x == 0) *p.st.g = w->g_before;
}

cudaError_t launch_router_logits(const void* x, bool x_bf16, const float* wr, int B, int E, int H, float* logits,
                                 cudaStream_t s) {
  const int warps = B * E, threads = 256, blocks = (warps * 32 + threads - 1) / threads;
  if (x_bf16)
    router_logits_kernel<__nv_bfloat16><<<blocks, threads, 0, s>>>((const __nv_bfloat16*)x, wr, B, E, H, logits);
  else
    router_logits_kernel<float><<<blocks, threads, 0, s>>>((const float*)x, wr, B, E, H, logits);
  return cudaGetLastError();
}

cudaError_t launch_ctrl(const CtrlParams& p, cudaStream_t s) {
  ctrl_kernel<<<1, kCtrlThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_undo(const UndoParams& p, cudaStream_t s) {
  undo_kernel<<<1, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
