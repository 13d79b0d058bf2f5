// Per-call cache control, executed by one CTA of the layer kernel.
//
// FreeToken write-up, "CUDA Graph-compatible LRU cache": per MoE layer one GPU
// step deduplicates the routed experts, classifies them against the residency
// table, derives the fill count, selects eviction victims and rewrites logical
// routing ids to physical slot ids; victim discovery costs one pass that finds
// K candidate slots at once, of which the miss path consumes the first q <= K,
// whatever the number of misses.  "Router-following LRU cache": a hit refreshes
// recency, a fill admits the selected expert, eviction removes the expert not
// requested for the longest time.
//
// Deterministic rules (specified identically for the CPU reference simulator):
//  * top-k by logit, descending, ties to the lower expert id (NaN counts as
//    -inf); weights = softmax over the k selected logits;
//  * U = sorted distinct routed experts; the member of rank r gets stamp g + r,
//    then g += |U|;
//  * victims: among slots not holding a hit of this call, empty slots first by
//    index, then occupied slots by ascending stamp; the i-th miss (ascending
//    expert) takes the i-th victim.
//
// The one pass is amortised: the cache keeps the K oldest slots (keys: empty
// slot s -> s, occupied -> C + stamp; K = min(256, C)) as a sorted list.  A
// call takes its victims as the first n_miss list entries that are not its own
// hits, then drops from the list every slot it touched (its hits and victims
// now carry the newest stamps, every other listed slot is still older than all
// unlisted ones), so the list stays exactly the oldest slots of the new state.
// Only when it holds fewer entries than the call has distinct experts (or after
// creation, resize or a rolled-back call) does the call rank all C slots.
#pragma once
#include "params.cuh"

namespace moe {

struct CtrlSmem {
  int ids[kMaxPairs];
  float w[kMaxPairs];
  int prank[kMaxPairs];
  unsigned bits[kMaxE / 32];
  int wpre[kMaxE / 32];
  int U[kMaxU];
  int slot[kMaxU];
  int fill[kMaxU];
  int mrank[kMaxU];
  int cnt[kMaxU];
  int off[kMaxU + 1];
  int sel_slot[kMaxU];
  unsigned long long sel_key[kMaxU];
  int victim[kMaxU];
  int scan[33];
  unsigned hist[2048];
  int nu, nmiss, nsel, err, remaining, bin;
  unsigned long long g, kmin, kmax, prefix;
};

__device__ __forceinline__ bool better_logit(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}

// Rank key of slot s for victim selection; false if s is excluded (a slot
// holding one of this call's hits, when `bits`/`layer` are given).
__device__ __forceinline__ bool slot_key(const CacheDev& st, int64_t C, int64_t s, int E, int layer,
                                         const unsigned* bits, unsigned long long* key) {
  const int own = st.owner[s];
  if (own < 0) {
    *key = (unsigned long long)s;
    return true;
  }
  if (bits && own / E == layer) {
    const int e = own % E;
    if (bits[e >> 5] & (1u << (e & 31))) return false;
  }
  *key = (unsigned long long)C + st.stamp[s];
  return true;
}

// The `want` smallest keys over slots [0, C) (all keys are distinct), sorted
// ascending into cs.sel_slot / cs.sel_key; returns how many were found.
// Radix select with 11-bit digits over the span of the keys, then a rank sort
// of the selected few.  Every thread of the CTA must call.
__device__ int select_oldest(CtrlSmem& cs, const CacheDev& st, int64_t C, int want, int E, int layer,
                             const unsigned* bits) {
  const int tid = threadIdx.x, lane = tid & 31, nt = blockDim.x;
  unsigned long long lmin = ~0ull, lmax = 0ull;
  int lcount = 0;
  for (int64_t s = tid; s < C; s += nt) {
    unsigned long long kk;
    if (slot_key(st, C, s, E, layer, bits, &kk)) {
      lmin = min(lmin, kk);
      lmax = max(lmax, kk);
      ++lcount;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lmin = min(lmin, __shfl_xor_sync(0xFFFFFFFFu, lmin, o));
    lmax = max(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
  }
  int ncand;
  block_excl_scan(lcount, cs.scan, &ncand);
  if (tid == 0) { cs.kmin = ~0ull; cs.kmax = 0ull; cs.prefix = 0ull; cs.nsel = 0; }
  __syncthreads();
  if (lane == 0) { atomicMin(&cs.kmin, lmin); atomicMax(&cs.kmax, lmax); }
  __syncthreads();
  if (want > ncand) want = ncand;
  if (want <= 0) return 0;
  if (tid == 0) cs.remaining = want;
  __syncthreads();
  const unsigned long long kmin = cs.kmin, span = cs.kmax - cs.kmin;
  const int nbits = span ? 64 - __clzll((long long)span) : 1;
  const int passes = (nbits + 10) / 11;
  const int bpt = 2048 / nt;  // histogram bins per thread
  for (int pass = passes - 1; pass >= 0; --pass) {
    const int shift = pass * 11, hs = shift + 11;
    for (int i = tid; i < 2048; i += nt) cs.hist[i] = 0u;
    __syncthreads();
    const unsigned long long prefix = cs.prefix;
    for (int64_t s = tid; s < C; s += nt) {
      unsigned long long kk;
      if (!slot_key(st, C, s, E, layer, bits, &kk)) continue;
      const unsigned long long d = kk - kmin;
      if (hs < 64 && (d >> hs) != (prefix >> hs)) continue;
      atomicAdd(&cs.hist[(d >> shift) & 2047ull], 1u);
    }
    __syncthreads();
    int mine = 0;
    for (int b = 0; b < bpt; ++b) mine += cs.hist[tid * bpt + b];
    int tot;
    int before = block_excl_scan(mine, cs.scan, &tot);
    const int rem = cs.remaining;
    __syncthreads();
    if (before < rem && rem <= before + mine) {
      int run = before;
      for (int b = 0; b < bpt; ++b) {
        const int c = cs.hist[tid * bpt + b];
        if (run < rem && rem <= run + c) {
          cs.bin = tid * bpt + b;
          cs.remaining = rem - run;
          break;
        }
        run += c;
      }
    }
    __syncthreads();
    if (tid == 0) cs.prefix = prefix | ((unsigned long long)cs.bin << shift);
    __syncthreads();
  }
  const unsigned long long thr = cs.prefix;  // offset of the want-th smallest key
  for (int64_t s = tid; s < C; s += nt) {
    unsigned long long kk;
    if (!slot_key(st, C, s, E, layer, bits, &kk)) continue;
    if (kk - kmin <= thr) {
      const int pos = atomicAdd(&cs.nsel, 1);
      if (pos < kMaxU) { cs.victim[pos] = (int)s; cs.sel_key[pos] = kk; }
    }
  }
  __syncthreads();
  const int nsel = min(cs.nsel, kMaxU);
  int vslot = -1, vrank = -1;
  unsigned long long vkey = 0;
  if (tid < nsel) {
    vkey = cs.sel_key[tid];
    vslot = cs.victim[tid];
    vrank = 0;
    for (int j = 0; j < nsel; ++j) vrank += cs.sel_key[j] < vkey;
  }
  __syncthreads();
  if (tid < nsel) {
    cs.sel_slot[vrank] = vslot;
    cs.sel_key[vrank] = vkey;
  }
  __syncthreads();
  return nsel == want ? want : -1;
}

// Routing, deduplication, lookup, victim choice, state update and grouping.
// Writes the plan (device), the host summary (pinned) and the inspection
// outputs.  Returns the status (MOE_OK or an error) to every thread.
__device__ int control_step(const LayerParams& p, CtrlSmem& cs) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarp = blockDim.x >> 5;
  const int E = p.E, k = p.k, B = p.B, npairs = B * k;
  const int64_t C = p.C;
  Plan* plan = p.plan;
  HostWork* work = p.work;

  // ---- router: one warp per token, logits held in registers ---------------
  for (int t = warp; t < B; t += nwarp) {
    const float* lg = p.logits + (size_t)t * E;
    float v[kMaxE / 32];
#pragma unroll
    for (int q = 0; q < kMaxE / 32; ++q) {
      const int e = lane + 32 * q;
      float x = -INFINITY;
      if (e < E) {
        x = lg[e];
        if (p.aux_logits) p.aux_logits[(size_t)t * E + e] = x;
        if (x != x) x = -INFINITY;
      }
      v[q] = x;
    }
    unsigned taken = 0u;  // bit q: element lane+32q already selected
    float m0 = 0.f, sum = 0.f;
    for (int r = 0; r < k; ++r) {
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
#pragma unroll
      for (int q = 0; q < kMaxE / 32; ++q) {
        const int e = lane + 32 * q;
        if (e < E && !(taken & (1u << q)) && better_logit(v[q], e, bv, bi)) { bv = v[q]; bi = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        if (better_logit(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (r == 0) m0 = bv;
      const float ex = expf(bv - m0);
      sum += ex;
      if (lane == 0) {
        cs.ids[t * k + r] = bi;
        cs.w[t * k + r] = ex;
      }
    }
    if (lane == 0)
      for (int r = 0; r < k; ++r) cs.w[t * k + r] = cs.w[t * k + r] / sum;
  }
  for (int i = tid; i < kMaxE / 32; i += blockDim.x) cs.bits[i] = 0u;
  if (tid == 0) { cs.err = MOE_OK; cs.g = *p.st.g; }
  __syncthreads();

  // ---- dedup: U = sorted distinct routed experts ----------------------------
  if (tid < npairs) atomicOr(&cs.bits[cs.ids[tid] >> 5], 1u << (cs.ids[tid] & 31));
  __syncthreads();
  const int nwords = (E + 31) / 32;
  if (warp == 0) {
    const int c = lane < nwords ? __popc(cs.bits[lane]) : 0;
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane < nwords) cs.wpre[lane] = x - c;
    if (lane == 31) cs.nu = x;
  }
  __syncthreads();
  const int n_u = cs.nu;
  if (tid < n_u) cs.cnt[tid] = 0;
  __syncthreads();
  if (tid < npairs) {
    const int e = cs.ids[tid];
    const int r = cs.wpre[e >> 5] + __popc(cs.bits[e >> 5] & ((1u << (e & 31)) - 1u));
    cs.prank[tid] = r;
    cs.U[r] = e;
    atomicAdd(&cs.cnt[r], 1);
  }
  if (tid == 0 && n_u > C) cs.err = MOE_ERR_CAPACITY;
  __syncthreads();

  // ---- classify against the residency table ---------------------------------
  int is_miss = 0;
  if (cs.err == MOE_OK && tid < n_u) {
    const int s = p.st.map[p.layer * E + cs.U[tid]];
    cs.slot[tid] = s;
    is_miss = s < 0;
    cs.fill[tid] = is_miss;
  }
  int nmiss;
  const int mr = block_excl_scan(is_miss, cs.scan, &nmiss);
  if (tid < n_u) cs.mrank[tid] = mr;

  // ---- victims: first nmiss entries of the oldest-slot list that are no hits --
  if (cs.err == MOE_OK && nmiss > 0) {
    int listed = *p.oldest_n;
    const int full = (int)(C < (int64_t)kMaxU ? C : (int64_t)kMaxU);
    if (listed < 0 || (listed < n_u && listed < full)) {  // rank all C slots again
      const int got = select_oldest(cs, p.st, C, full, E, -1, nullptr);
      listed = got == full ? full : 0;
      for (int i = tid; i < listed; i += blockDim.x) p.oldest[i] = cs.sel_slot[i];
      if (tid == 0) cs.err = got == full ? MOE_OK : MOE_ERR_CUDA;
      __syncthreads();
    }
    int ok = 0, slot = -1;
    if (tid < listed) {
      slot = p.oldest[tid];
      unsigned long long kk;
      ok = slot_key(p.st, C, slot, E, p.layer, cs.bits, &kk) ? 1 : 0;
    }
    int tot;
    const int pos = block_excl_scan(ok, cs.scan, &tot);
    if (ok && pos < nmiss) cs.victim[pos] = slot;
    if (tid == 0) {
      cs.nsel = listed;
      if (tot < nmiss) cs.err = MOE_ERR_CUDA;  // cannot happen with a consistent list
    }
    __syncthreads();
  } else if (tid == 0) {
    cs.nsel = *p.oldest_n;
  }
  if (cs.err != MOE_OK) {
    if (tid == 0) {
      plan->err = cs.err;
      plan->n_u = n_u;
      plan->n_miss = 0;
      plan->n_items[0] = plan->n_items[1] = 0;
      work->err = cs.err;
      work->n_u = n_u;
      work->n_miss = 0;
      work->g_before = cs.g;
      __threadfence_system();
      work->seq = p.seq;
    }
    return cs.err;
  }

  // ---- apply: restamp hits, assign victims, keep the undo log --------------------
  const unsigned long long g0 = cs.g;
  if (tid < n_u) {
    const int key = p.layer * E + cs.U[tid];
    plan->u_key[tid] = key;
    work->key[tid] = key;
    work->pairs[tid] = cs.cnt[tid];
    if (!cs.fill[tid]) {
      const int s = cs.slot[tid];
      plan->u_old_stamp[tid] = p.st.stamp[s];
      p.st.stamp[s] = g0 + tid;
      work->slot[tid] = s;
      work->evicted[tid] = -1;
      work->fill[tid] = 0;
    } else {
      const int v = cs.victim[cs.mrank[tid]];
      const int ev = p.st.owner[v];
      plan->u_old_stamp[tid] = p.st.stamp[v];
      if (ev >= 0) p.st.map[ev] = -1;
      p.st.map[key] = v;
      p.st.owner[v] = key;
      p.st.stamp[v] = g0 + tid;
      cs.slot[tid] = v;
      work->slot[tid] = v;
      work->evicted[tid] = ev;
      work->fill[tid] = 1;
    }
  }
  if (tid == 0) *p.st.g = g0 + n_u;

  // ---- stable grouping of (token, rank) pairs by expert (block-scan histogram)
  int tot;
  const int off = block_excl_scan(tid < n_u ? cs.cnt[tid] : 0, cs.scan, &tot);
  if (tid < n_u) cs.off[tid] = off;
  if (tid == 0) cs.off[n_u] = npairs;
  __syncthreads();
  if (tid < npairs) {
    const int r = cs.prank[tid];
    int before = 0;
    for (int q = 0; q < tid; ++q) before += (cs.prank[q] == r);
    const int pos = cs.off[r] + before;
    plan->perm[pos] = tid;
    plan->pair_rank[tid] = r;
    plan->pair_w[tid] = cs.w[tid];
    if (p.aux_perm) p.aux_perm[pos] = tid;
    if (p.aux_ids) p.aux_ids[tid] = cs.ids[tid];
    if (p.aux_w) p.aux_w[tid] = cs.w[tid];
    if (p.aux_slots) p.aux_slots[tid] = cs.slot[r];
  }
  if (p.aux_offsets) {
    for (int e = tid; e <= E; e += blockDim.x) {
      const int r = (e < E) ? cs.wpre[e >> 5] + __popc(cs.bits[e >> 5] & ((1u << (e & 31)) - 1u)) : n_u;
      p.aux_offsets[e] = r < n_u ? cs.off[r] : npairs;
    }
  }
  if (tid < n_u) {
    plan->u_expert[tid] = cs.U[tid];
    plan->u_slot[tid] = cs.slot[tid];
    plan->u_fill[tid] = cs.fill[tid];
  }
  if (tid <= n_u) plan->u_off[tid] = cs.off[tid];
  const int is_res = tid < n_u && !cs.fill[tid];
  int nres;
  const int rpos = block_excl_scan(is_res, cs.scan, &nres);
  if (is_res) plan->items[0][rpos] = tid;
  if (tid < n_u && cs.fill[tid]) {
    plan->items[1][cs.mrank[tid]] = tid;
    work->fill_order[cs.mrank[tid]] = tid;
  }
  if (tid == 0) {
    if (p.has_shared) plan->items[0][nres] = n_u;  // the shared expert is item index n_u
    plan->err = MOE_OK;
    plan->B = B;
    plan->k = k;
    plan->n_u = n_u;
    plan->n_miss = nmiss;
    plan->n_items[0] = nres + (p.has_shared ? 1 : 0);
    plan->n_items[1] = nmiss;
    plan->g_before = g0;
    work->err = MOE_OK;
    work->n_u = n_u;
    work->n_miss = nmiss;
    work->g_before = g0;
  }
  __threadfence_system();  // each writer publishes its part of the host summary
  __syncthreads();
  if (tid == 0) {
    __threadfence_system();
    work->seq = p.seq;
  }
  return MOE_OK;
}

// Drop from the oldest-slot list every slot this call touched (hits and
// victims now own keys of this call).  Run by the control CTA after the plan
// is published.
__device__ void compact_oldest(const LayerParams& p, CtrlSmem& cs) {
  __syncthreads();
  const int listed = cs.nsel;
  if (listed < 0) return;
  int keep = 0, slot = -1;
  if (threadIdx.x < listed) {
    slot = p.oldest[threadIdx.x];
    unsigned long long kk;
    keep = slot_key(p.st, p.C, slot, p.E, p.layer, cs.bits, &kk) ? 1 : 0;
  }
  int tot;
  const int pos = block_excl_scan(keep, cs.scan, &tot);
  if (keep) cs.victim[pos] = slot;
  __syncthreads();
  if (threadIdx.x < tot) p.oldest[threadIdx.x] = cs.victim[threadIdx.x];
  if (threadIdx.x == 0) *p.oldest_n = tot;
}

// Undo of a call whose fills did not arrive: recency and the counter go back
// to their values before the call; the call's victim slots are left empty
// (their previous contents may already be overwritten).
__device__ void undo_call(const LayerParams& p) {
  const Plan* pl = p.plan;
  for (int r = threadIdx.x; r < pl->n_u; r += blockDim.x) {
    const int s = pl->u_slot[r];
    if (!pl->u_fill[r]) {
      p.st.stamp[s] = pl->u_old_stamp[r];
    } else {
      p.st.map[pl->u_key[r]] = -1;
      p.st.owner[s] = -1;
      p.st.stamp[s] = 0;
    }
  }
  if (threadIdx.x == 0) {
    *p.st.g = pl->g_before;
    *p.oldest_n = -1;
  }
}

}  // namespace moe
