// Per-call cache control inside the layer kernel.  Routing, deduplication,
// residency lookup and grouping run in every CTA (route_lookup); victim
// choice, the plan, the host summary and the commit of recency and residency
// run in the control CTA (choose_victims, control_commit, compact_oldest).
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
//    -inf, -0 as +0); weights = softmax over the k selected logits;
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
  int perm[kMaxPairs];  // flat pair t*k+j grouped by expert (stable)
  int maprow[kMaxE];    // residency table row of this call's layer
  unsigned bits[kMaxE / 32];
  int wpre[kMaxE / 32];
  int U[kMaxU];
  int slot[kMaxU];  // slot of U[r] after the call (hit: its slot; miss: its victim)
  int fill[kMaxU];
  int mrank[kMaxU];
  int cnt[kMaxU];
  int off[kMaxU + 1];
  int sel_slot[kMaxU];
  unsigned long long sel_key[kMaxU];
  int victim[kMaxU];
  int victim_owner[kMaxU];  // key held by each victim before the call (-1: empty)
  int scan[33];
  unsigned hist[2048];
  int nu, nmiss, nsel, err, remaining, bin;
  unsigned long long g, kmin, kmax, prefix;
};

// Order-preserving 32-bit key of a logit for the router's max-reductions: NaN
// counts as -inf and -0 as +0, so equal logits give equal keys and the
// lower expert id wins the tie.  Real logits map to keys > 0; 0 marks "none".
__device__ __forceinline__ unsigned logit_key(float x) {
  unsigned u = __float_as_uint(x);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) u = 0xFF800000u;  // NaN -> -inf
  if ((u & 0x7FFFFFFFu) == 0u) u = 0u;                   // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(unsigned key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Top-k of one token's E logits by one warp: lane l holds experts l + 32q
// (q < NQ) as keys, keeps its own best, and each round the warp takes the
// largest key (redux max) and, among equal keys, the lowest expert id (redux
// min); only the winning lane rescans.  Weights = softmax over the k taken
// logits, exp(l_r - l_0) / sum, in the order taken.
template <int NQ>
__device__ __forceinline__ void route_token(const float* lg, int E, int k, int lane, float* aux, int* ids, float* w,
                                            unsigned long long* stamp = nullptr, const float* pre = nullptr) {
  unsigned key[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int e = lane + 32 * q;
    key[q] = 0u;
    if (e < E) {
      const float x = pre ? pre[q] : lg[e];
      if (aux) aux[e] = x;
      key[q] = logit_key(x);
    }
  }
  unsigned bk = 0u;
  int bq = 0;
#pragma unroll
  for (int q = 0; q < NQ; ++q)
    if (key[q] > bk) { bk = key[q]; bq = q; }
  if (stamp && lane == 0) *stamp = globaltimer_ns();  // profiling: the logits have landed
  float m0 = 0.f, sum = 0.f;
  for (int r = 0; r < k; ++r) {
    const unsigned m = __reduce_max_sync(0xFFFFFFFFu, bk);
    const int e = (int)__reduce_min_sync(0xFFFFFFFFu, bk == m ? (unsigned)(lane + 32 * bq) : 0xFFFFFFFFu);
    const float x = key_logit(m);
    if (r == 0) m0 = x;
    const float ex = x == m0 ? 1.f : expf(x - m0);  // equal to the largest (also +-inf): exp(0)
    sum += ex;
    if (lane == 0) {
      ids[r] = e;
      w[r] = ex;
    }
    if ((e & 31) == lane) {
      const int taken = e >> 5;
      bk = 0u;
      bq = 0;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (q == taken) key[q] = 0u;
        if (key[q] > bk) { bk = key[q]; bq = q; }
      }
    }
  }
  if (lane == 0)
    for (int r = 0; r < k; ++r) w[r] = w[r] / sum;
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
static __device__ int select_oldest(CtrlSmem& cs, const CacheDev& st, int64_t C, int want, int E, int layer,
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

// Sequence number of the current call and what derives from it, set once
// per CTA before the first CTA barrier (call_seq_init) and read from shared
// memory afterwards.  For a call launched from the host it is the launch's
// own; for a call replayed from a captured graph it comes from a counter
// every CTA adds 1 to per call, so consecutive replays get consecutive numbers.
struct CallSeq {
  uint32_t seq;
  HostWork* work;     // this call's host summary
  unsigned* wave_ctr;   // this call's counters
  unsigned* wave_next;  // the next call's counters (cleared by this call)
};
__device__ __forceinline__ CallSeq& cseq() {
  __shared__ CallSeq c;
  return c;
}
// One thread per CTA.
__device__ __forceinline__ void call_seq_init(const LayerParams& p) {
  CallSeq& c = cseq();
  if (p.seq_ctr) {
    const uint32_t s = (uint32_t)(atomicAdd(p.seq_ctr, 1ull) / gridDim.x + 1ull);
    c.seq = s;
    c.work = p.work + s % kSummaryRing;
    c.wave_ctr = p.wave_ctr + (s & 1u) * kWaveCtrs;
    c.wave_next = p.wave_ctr + ((s + 1u) & 1u) * kWaveCtrs;
  } else {
    c.seq = p.seq;
    c.work = p.work;
    c.wave_ctr = p.wave_ctr;
    c.wave_next = p.wave_next;
  }
}

// Publish the host summary of the call (its fields are already written):
// system-scope fences by every writer, then the sequence number last.
__device__ __forceinline__ void publish_summary(const LayerParams& p) {
  __threadfence_system();
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence_system();
    cseq().work->seq = cseq().seq;
  }
}

// Routing, deduplication, residency lookup and grouping of one call, run by
// every CTA of the layer kernel on its own (the inputs are a few KB and the
// result is deterministic, so every CTA arrives at the same tables without
// waiting for one another): top-k per token, U = sorted distinct experts,
// each member's slot (or a miss), the stable grouping of the (token, rank)
// pairs by expert (offsets and perm) and the miss ranks.  The residency table
// is only read here; the control CTA writes it after a grid barrier that every
// CTA reaches after this lookup.  Returns MOE_ERR_CAPACITY (|U| > C) or MOE_OK
// to every thread.
// The layer's residency row as route_lookup reads it: entry tid + j * kThreads
// in mrow[j] (issued at the kernel's start, next to the router's logits).
__device__ __forceinline__ void load_map_row(const LayerParams& p, int* mrow) {
#pragma unroll
  for (int j = 0; j < kMaxE / kThreads; ++j) {
    const int e = (int)threadIdx.x + j * kThreads;
    mrow[j] = e < p.E ? p.st.map[p.layer * p.E + e] : -1;
  }
}

// pre: the calling warp's first token's logits already in registers (E <= 256), or null.
// mrow: the layer's residency row from load_map_row.
static __device__ int route_lookup(const LayerParams& p, CtrlSmem& cs, bool write_aux, const int* mrow,
                                   const float* pre = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarp = blockDim.x >> 5;
  const bool rec = p.tl && blockIdx.x == 1 && tid == 0;
  const int E = p.E, k = p.k, B = p.B, npairs = B * k;
  for (int i = tid; i < kMaxE / 32; i += blockDim.x) cs.bits[i] = 0u;

  // ---- router: one warp per token ------------------------------------------------
  const int nq = (E + 31) >> 5;
  for (int t = warp; t < B; t += nwarp) {
    const float* lg = p.logits + (size_t)t * E;
    float* aux = (write_aux && p.aux_logits) ? p.aux_logits + (size_t)t * E : nullptr;
    int* ids = cs.ids + t * k;
    float* w = cs.w + t * k;
    unsigned long long* st = rec && t == 0 ? p.tl + 15 : nullptr;
    if (rec && t == 0) p.tl[13] = globaltimer_ns();  // profiling: the router starts loading
    const float* tp = t == warp ? pre : nullptr;  // this warp's first token may be preloaded
    if (nq <= 1) route_token<1>(lg, E, k, lane, aux, ids, w, st, tp);
    else if (nq <= 2) route_token<2>(lg, E, k, lane, aux, ids, w, st, tp);
    else if (nq <= 4) route_token<4>(lg, E, k, lane, aux, ids, w, st, tp);
    else if (nq <= 8) route_token<8>(lg, E, k, lane, aux, ids, w, st, tp);
    else if (nq <= 16) route_token<16>(lg, E, k, lane, aux, ids, w, st);
    else route_token<32>(lg, E, k, lane, aux, ids, w, st);
  }
  if (rec) p.tl[12] = globaltimer_ns();
#pragma unroll
  for (int j = 0; j < kMaxE / kThreads; ++j) {
    const int e = tid + j * kThreads;
    if (e < E) cs.maprow[e] = mrow[j];
  }
  __syncthreads();


  // ---- dedup: U = sorted distinct routed experts ----------------------------------
  if (tid < npairs && in_bounds(p.dbg, cs.ids[tid] >= 0 && cs.ids[tid] < E, 8))
    atomicOr(&cs.bits[cs.ids[tid] >> 5], 1u << (cs.ids[tid] & 31));
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
  __syncthreads();
  if (n_u > p.C) return MOE_ERR_CAPACITY;

  // ---- residency lookups, then one scan for the grouping offsets (pairs per
  // expert, high half) and the miss ranks (low half); both totals are <= 256
  int is_miss = 0;
  if (tid < n_u) {
    const int s = cs.maprow[cs.U[tid]];
    cs.slot[tid] = s;
    is_miss = s < 0;
    cs.fill[tid] = is_miss;
  }
  int packed_tot;
  const int packed = block_excl_scan(((tid < n_u ? cs.cnt[tid] : 0) << 16) | is_miss, cs.scan, &packed_tot);
  if (tid < n_u) {
    cs.off[tid] = packed >> 16;
    cs.mrank[tid] = packed & 0xFFFF;
  }
  if (tid == 0) {
    cs.off[n_u] = npairs;
    cs.nmiss = packed_tot & 0xFFFF;
  }
  __syncthreads();
  if (rec) p.tl[14] = globaltimer_ns();
  // stable grouping of the (token, rank) pairs by expert
  if (tid < npairs) {
    const int r = cs.prank[tid];
    int before = 0;
    for (int q = 0; q < tid; ++q) before += (cs.prank[q] == r);
    cs.perm[cs.off[r] + before] = tid;
  }
  __syncthreads();
  return MOE_OK;
}

// The plan's error and the host summary of a call that cannot run (capacity,
// or an inconsistent victim list); control CTA only.
static __device__ void publish_error(const LayerParams& p, const CtrlSmem& cs, int err) {
  if (threadIdx.x != 0) return;
  Plan* plan = p.plan;
  HostWork* work = cseq().work;
  plan->err = err;
  plan->n_u = cs.nu;
  plan->n_miss = 0;
  plan->n_items[0] = plan->n_items[1] = 0;
  work->err = err;
  work->layer = p.layer;
  work->B = p.B;
  work->n_u = cs.nu;
  work->n_miss = 0;
  work->g_before = *p.st.g;
  __threadfence_system();
  work->seq = cseq().seq;
  __threadfence();
  st_release_u32(p.plan_flag, cseq().seq);
}

// Fill count q* of the bandwidth split for m misses ("measured bandwidths
// decide the split" in the FreeToken write-up): q/(m-q) ~ B_P/(B_H - B_P), so
// q* ~ m B_P / B_H, rounded to the nearest integer (halves up), at least one
// fill, all m when B_H <= B_P or when no bandwidths are set; 0 without misses.
// Computed in float64 so that the rounding decision is the one the reference
// computation takes.
__device__ __forceinline__ int qstar_of(int m, double bp, double bh) {
  if (m <= 0) return 0;
  if (!(bp > 0.0) || !(bh > 0.0) || bh <= bp) return m;
  const int q = (int)floor((double)m * bp / bh + 0.5);
  return q < 1 ? 1 : (q > m ? m : q);
}

// Victims, the plan and the host summary (control CTA, after route_lookup):
// the first n_miss entries of the oldest-slot list that hold no hit of this
// call become the misses' slots (the whole pool is ranked again when the list
// runs short).  When the host issues this call's copies the summary is
// published before anything else.  Ends with thread 0's release store of the
// plan flag, which the other CTAs acquire before they read fill slots.
// Returns MOE_OK, or MOE_ERR_CUDA if the list was inconsistent (the plan and
// the summary then carry the error).
static __device__ int choose_victims(const LayerParams& p, CtrlSmem& cs) {
  const int tid = threadIdx.x;
  const int E = p.E, k = p.k, B = p.B, npairs = B * k, n_u = cs.nu, nmiss = cs.nmiss;
  const int64_t C = p.C;
  Plan* plan = p.plan;
  HostWork* work = cseq().work;
  const int my_listed = tid < kMaxU ? p.oldest[tid] : -1;
  if (tid == 0) {
    cs.err = MOE_OK;
    cs.g = *p.st.g;
    cs.nsel = *p.oldest_n;
  }
  __syncthreads();
  const int listed0 = cs.nsel;  // -1: the list must be rebuilt
  int my_owner = -1;
  if (tid < listed0 && my_listed >= 0 && my_listed < C) my_owner = p.st.owner[my_listed];

  if (nmiss > 0) {
    int listed = listed0;
    const int full = (int)(C < (int64_t)kMaxU ? C : (int64_t)kMaxU);
    bool rebuilt = false;
    if (listed < 0 || (listed < n_u && listed < full)) {  // rank all C slots again
      const int got = select_oldest(cs, p.st, C, full, E, -1, nullptr);
      listed = got == full ? full : 0;
      for (int i = tid; i < listed; i += blockDim.x) p.oldest[i] = cs.sel_slot[i];
      if (tid == 0) cs.err = got == full ? MOE_OK : MOE_ERR_CUDA;
      rebuilt = true;
      __syncthreads();
    }
    int ok = 0, slot = -1, own = -1;
    if (tid < listed) {
      slot = rebuilt ? cs.sel_slot[tid] : my_listed;
      own = rebuilt ? p.st.owner[slot] : my_owner;
      ok = 1;
      if (own >= 0 && own / E == p.layer) {
        const int e = own % E;
        if (cs.bits[e >> 5] & (1u << (e & 31))) ok = 0;  // holds one of this call's hits
      }
    }
    int navail;
    const int pos = block_excl_scan(ok, cs.scan, &navail);
    if (ok && pos < nmiss) {
      cs.victim[pos] = slot;
      cs.victim_owner[pos] = own;
    }
    if (tid == 0) {
      cs.nsel = listed;
      if (navail < nmiss) cs.err = MOE_ERR_CUDA;  // cannot happen with a consistent list
    }
    __syncthreads();
  }
  if (cs.err != MOE_OK) {
    publish_error(p, cs, cs.err);
    return cs.err;
  }

  // ---- the plan (and the fields of the host summary) ----------------------------------
  // copy mode: the host waits for this summary (it issues the fills and must
  // know there are none); device mode: published after the commit instead
  const bool host_first = !p.device_fill;
  if (tid < n_u) {
    const int key = p.layer * E + cs.U[tid];
    const int fill = cs.fill[tid];
    const int s = fill ? cs.victim[cs.mrank[tid]] : cs.slot[tid];
    in_bounds(p.dbg, s >= 0 && s < C && (!fill || cs.mrank[tid] < kMaxU), 9);  // recorded; the host sees the count
    cs.slot[tid] = s;
    plan->u_key[tid] = key;
    plan->u_expert[tid] = cs.U[tid];
    plan->u_slot[tid] = s;
    plan->u_fill[tid] = fill;
    work->key[tid] = key;
    work->slot[tid] = s;
    work->fill[tid] = fill;
    work->evicted[tid] = fill ? cs.victim_owner[cs.mrank[tid]] : -1;
    work->pairs[tid] = cs.cnt[tid];
    if (fill) work->fill_order[cs.mrank[tid]] = tid;
  }
  if (tid <= n_u) plan->u_off[tid] = cs.off[tid];
  __syncthreads();
  if (tid < npairs) {
    const int r = cs.prank[tid];
    plan->perm[tid] = cs.perm[tid];
    plan->pair_rank[tid] = r;
    plan->pair_w[tid] = cs.w[tid];
    if (p.aux_perm) p.aux_perm[tid] = cs.perm[tid];
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
  const int nres = n_u - nmiss;  // hits before rank r: r minus the misses before it
  if (tid < n_u && !cs.fill[tid]) plan->items[0][tid - cs.mrank[tid]] = tid;
  if (tid < n_u && cs.fill[tid]) plan->items[1][cs.mrank[tid]] = tid;
  if (tid == 0) {
    if (p.has_shared) plan->items[0][nres] = n_u;  // the shared expert is item index n_u
    plan->err = MOE_OK;
    plan->B = B;
    plan->k = k;
    plan->n_u = n_u;
    plan->n_miss = nmiss;
    plan->n_items[0] = nres + (p.has_shared ? 1 : 0);
    plan->n_items[1] = nmiss;
    plan->g_before = cs.g;
    work->err = MOE_OK;
    work->layer = p.layer;
    work->B = p.B;
    work->n_u = n_u;
    work->n_miss = nmiss;
    work->g_before = cs.g;
    work->qstar = qstar_of(nmiss, p.split_bp, p.split_bh);
    if (p.aux_qstar) *p.aux_qstar = work->qstar;
  }
  if (host_first) publish_summary(p);  // the host issues this call's copies from it
  // the CTA barrier orders every thread's plan writes before thread 0's
  // release store of the plan flag (GPU scope), which the other CTAs acquire
  __syncthreads();
  if (tid == 0) st_release_u32(p.plan_flag, cseq().seq);
  return MOE_OK;
}

// Recency, residency table and undo log of a planned call, written once every
// CTA has done its residency lookups (after the first grid barrier): hits and
// fills take stamps g + r in U order, each victim's previous key leaves the
// table, g advances by |U|.  Then the host summary in device-fill mode
// (choose_victims published it already in copy mode).
static __device__ void control_commit(const LayerParams& p, CtrlSmem& cs) {
  const int tid = threadIdx.x, n_u = cs.nu;
  const unsigned long long g0 = cs.g;
  if (tid < n_u) {
    const int s = cs.slot[tid];
    const int key = p.layer * p.E + cs.U[tid];
    p.plan->u_old_stamp[tid] = p.st.stamp[s];
    if (cs.fill[tid]) {
      const int ev = cs.victim_owner[cs.mrank[tid]];
      if (ev >= 0) p.st.map[ev] = -1;
      p.st.map[key] = s;
      p.st.owner[s] = key;
    }
    p.st.stamp[s] = g0 + tid;
  }
  if (tid == 0) *p.st.g = g0 + n_u;
  if (p.device_fill)
    publish_summary(p);
  else
    __syncthreads();
}

// Drop from the oldest-slot list every slot this call touched (hits and
// victims now own keys of this call).  Run by the control CTA after the plan
// is published.
static __device__ void compact_oldest(const LayerParams& p, CtrlSmem& cs) {
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

// Undo of a call whose fills could not be issued (run by the completion
// kernel once every copy of the call has ended): recency and the counter go
// back to their values before the call; the call's victim slots are left
// empty (their previous contents may already be overwritten).
static __device__ void undo_call(const LayerParams& p) {
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
