// One decode-size routed-MoE layer call as a single cooperative launch (plus,
// in copy-fill mode, a completion launch after the call's copies).
//
// FreeToken write-up: the router and the cache lookup run on the GPU ("decode
// co-design"); one GPU step per layer deduplicates, classifies, picks victims
// and rewrites ids ("CUDA Graph-compatible LRU cache"); the GPU evaluates the
// set G = H ∪ F as a grouped FFN once the batched copy of F has landed, and
// the partial sums merge exactly ("measured bandwidths decide the split",
// Fig. 2 caption); decode is memory-bound, each routed expert's weights being
// read once per token.
//
// Every CTA (512 threads, one per SM) routes the call and looks its experts up
// itself; CTA 0 also picks the victims and publishes the miss list to the
// host, which issues one cudaMemcpyAsync per half record (gate/up part, then
// W_down) on the copy streams, each followed by a stream write of a per-fill
// flag.  Then:
//  1. gate/up rows of the resident experts and the shared expert:
//     h = SiLU(x W_gate^T) * (x W_up^T); a warp streams one gate row and one up
//     row with 16-byte loads (FP4 dequantised in registers) and serves every
//     token routed to the expert; meanwhile each CTA's W_down rows of those
//     experts are staged in shared memory by bulk copies;
//  2. grid barrier (CTA 0 then commits recency and residency), then W_down
//     rows: each CTA owns a contiguous range of output rows n for every expert
//     and keeps o[t][j][n] in shared memory;
//  3. fills, in order, each as soon as its flag says the copy landed: gate/up
//     rows, one grid barrier, then W_down rows into the same shared buffer (a
//     CTA that waits too long hands its rows to the completion kernel);
//  4. y_t[n] = sum_j w_tj o_tj[n] (+ shared) in rank order, in float32.
// Every dot product has a fixed summation order independent of which phase
// or launch computes it, so outputs are bitwise identical whatever the
// residency.
#pragma once
#include "control.cuh"
#include "expert_math.cuh"

namespace moe {

constexpr int kEarlyItem = kMaxItems;
struct ItemTable {
  // entries 0 .. kMaxItems-1 in item order; entry kEarlyItem holds the shared
  // expert while its gate/up rows run alongside the routing
  const uint8_t* rec[kMaxItems + 1];  // where the record is read (slot, shared expert, or host pool)
  uint8_t* dst[kMaxItems + 1];        // slot a device-driven fill writes the record to (else null)
  int ntok[kMaxItems + 1];
  int pair0[kMaxItems + 1];  // -1 for the shared expert
  int hbase[kMaxItems + 2];  // running token count in item order
  int perm[kMaxPairs];       // the plan's grouped pair order, copied once per call
  float pair_w[kMaxPairs];   // the plan's routing weights, copied once per call
};

// A group of warps [w0, w0 + nw) of the CTA working together; bar 0 is the
// CTA-wide barrier, other ids are named barriers of the group's nw * 32 threads.
struct WarpGroup {
  int w0, nw, bar;
  __device__ __forceinline__ int tid() const { return (int)threadIdx.x - 32 * w0; }
  __device__ __forceinline__ int nthreads() const { return 32 * nw; }
  __device__ __forceinline__ void sync() const {
    if (bar == 0)
      __syncthreads();
    else
      asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(32 * nw) : "memory");
  }
};
__device__ __forceinline__ WarpGroup whole_cta() { return WarpGroup{0, kWarps, 0}; }

// Items of plan list `which` into tb at position `at` (list 1 from the host
// pool when `from_pool`); returns the new item count.  All threads call.
static __device__ int load_items(const LayerParams& p, const Plan* pl, int which, ItemTable& tb, int at = 0,
                          bool from_pool = false) {
  const int n = pl->n_items[which];
  if (at == 0 && which == 0)
    for (int i = threadIdx.x; i < p.B * p.k; i += blockDim.x) {
      tb.perm[i] = pl->perm[i];
      tb.pair_w[i] = pl->pair_w[i];
    }
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int r = pl->items[which][i];
    if (r == pl->n_u) {
      tb.rec[at + i] = p.shared_rec;
      tb.dst[at + i] = nullptr;
      tb.ntok[at + i] = p.B;
      tb.pair0[at + i] = -1;
    } else {
      if (!in_bounds(p.dbg, r >= 0 && r < kMaxU && pl->u_slot[r] >= 0 && pl->u_slot[r] < p.C &&
                                pl->u_key[r] >= 0 && pl->u_key[r] < p.L * p.E && at + i < kMaxItems, 2))
        continue;
      uint8_t* slot = const_cast<uint8_t*>(p.slots) + (int64_t)pl->u_slot[r] * p.S;
      tb.rec[at + i] = from_pool ? p.pool + (int64_t)pl->u_key[r] * p.S : slot;
      tb.dst[at + i] = from_pool ? slot : nullptr;
      tb.pair0[at + i] = pl->u_off[r];
      tb.ntok[at + i] = pl->u_off[r + 1] - pl->u_off[r];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = at ? tb.hbase[at] : 0;
    for (int i = at; i < at + n; ++i) { tb.hbase[i] = run; run += tb.ntok[i]; }
    tb.hbase[at + n] = run;
  }
  __syncthreads();
  return at + n;
}

// 16-byte unit v of the W_down rows [n0, n0 + nrows) of record `rec` (codes
// or values first, then the FP4 scales).  Row bytes and FP4 scale rows are
// multiples of 16 for every accepted shape (I % 64 == 0; FP4: I % 256 == 0).
template <int WD>
__device__ __forceinline__ const uint8_t* down_unit(const uint8_t* rec, int H, int I, int n0, int nv, int v) {
  const RecView r = rec_view<WD>(rec, H, I);
  if (v < nv) return r.down + (int64_t)n0 * Fmt<WD>::row_bytes(I) + (int64_t)v * 16;
  return r.down_sc + (int64_t)n0 * (I / 16) + (int64_t)(v - nv) * 16;
}

// The CTA's mbarrier for the h rows phase 2 copies into shared memory, and
// the parity of its current phase.
__device__ __forceinline__ uint64_t* h_bar() {
  __shared__ __align__(8) uint64_t b;
  return &b;
}
__device__ __forceinline__ uint32_t* h_bar_phase() {
  __shared__ uint32_t ph;
  return &ph;
}
// Thread 0, before the kernel's first CTA barrier.
__device__ __forceinline__ void h_bar_init() {
  mbar_init(h_bar(), 1);
  *h_bar_phase() = 0u;
  fence_mbar_init();
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// FP4 models: the staged bf16 activations become f16 in place (all threads),
// so the gate/up dot products run as mixed-precision f16 FMAs; exact for
// 2^-14 <= |x| <= 65504 and 0, smaller magnitudes round to the f16 subnormal
// grid (absolute error <= 2^-25).  Each token's row is also rearranged so
// that quarter q (values 8q .. 8q + 7) of every 32-value chunk c sits at
// q * H / 4 + 8c: a lane reads its chunk as four 16-byte loads from four
// contiguous runs, and eight lanes on eight consecutive chunks hit distinct
// banks (with whole chunks, 64 bytes apart, they shared two bank groups).
// H <= 16 * 2 * blockDim.x (16384 at 512 threads; the cache rejects larger).
template <int WD, typename XT>
__device__ __forceinline__ void x_to_f16(XT* xs, int B, int H) {
  if constexpr (WD == MOE_FP4) {
    constexpr int kPer = 16;  // words of one row per thread
    const int nw = H / 2;
    for (int t = 0; t < B; ++t) {
      uint32_t* w = reinterpret_cast<uint32_t*>(xs) + (size_t)t * nw;
      uint32_t v[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int i = (int)threadIdx.x + k * (int)blockDim.x;
        if (i < nw) {
          const __half2 h = __floats2half2_rn(bf16lo(w[i]), bf16hi(w[i]));
          v[k] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int i = (int)threadIdx.x + k * (int)blockDim.x;
        if (i < nw) {
          const int e = 2 * i, c = e >> 5, q = (e >> 3) & 3, r = e & 7;
          w[(q * (H >> 2) + 8 * c + r) >> 1] = v[k];
        }
      }
      __syncthreads();
    }
  }
}
// The activations as the gate/up dot products read them.
template <int WD, typename XT>
__device__ __forceinline__ auto x_dot(const XT* xs) {
  if constexpr (WD == MOE_FP4) return reinterpret_cast<const __half*>(xs);
  else return xs;
}

// Device-driven fill of this CTA's W_down rows [n0, n0 + nrows) of items
// [ib, ie): copy them from the host pool into the items' slots, with eight
// independent 16-byte loads in flight per thread (host-link latency bound).
template <int WD>
__device__ void copy_down_rows(const LayerParams& p, const ItemTable& tb, int ib, int ie, int n0, int nrows) {
  constexpr int U = 8;
  const int H = p.H, I = p.I;
  const int nv = (int)(nrows * Fmt<WD>::row_bytes(I) / 16);
  const int per = nv + (WD == MOE_FP4 ? nrows * (I / 16) / 16 : 0);
  const int total = (ie - ib) * per;
  for (int v0 = threadIdx.x; v0 < total; v0 += U * blockDim.x) {
    uint4 buf[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + u * (int)blockDim.x;
      if (v < total) buf[u] = ld_ro16(down_unit<WD>(tb.rec[ib + v / per], H, I, n0, nv, v % per));
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + u * (int)blockDim.x;
      if (v < total) {
        const uint8_t* d = tb.dst[ib + v / per];
        if (in_bounds(p.dbg, d >= p.slots && d < p.slots + p.C * p.S, 7))
          *reinterpret_cast<uint4*>(const_cast<uint8_t*>(down_unit<WD>(d, H, I, n0, nv, v % per))) = buf[u];
      }
    }
  }
}

// token, h row and rank slot of the q-th token of item `it`
__device__ __forceinline__ void item_token(const LayerParams& p, const ItemTable& tb, int it, int q, int* t,
                                           int* hrow, int* j) {
  const int p0 = tb.pair0[it];
  if (p0 < 0) {
    *t = q;
    *hrow = p.h_shared_row0 + q;
    *j = p.k;
  } else {
    const int pair = tb.perm[p0 + q];
    *t = pair / p.k;
    *hrow = pair;
    *j = pair % p.k;
    if (!in_bounds(p.dbg, p0 + q >= 0 && p0 + q < p.B * p.k && pair >= 0 && pair < p.B * p.k, 3)) {
      *t = 0;
      *hrow = 0;
      *j = 0;
    }
  }
}

// Gate/up rows of items [ib, ie), spread over CTAs [cta0, cta0 + ncta).
// WB: the rows are read from the host pool and also written to the slot.
template <int WD, int MAXT, bool FRESH, bool WB = false, typename XT>
__device__ void phase1(const LayerParams& p, const ItemTable& tb, int ib, int ie, int cta0, int ncta, const XT* xs,
                       WarpGroup grp = whole_cta()) {
  using F = Fmt<WD>;
  // fewer chunks in flight where the token registers grow (16 tokens; FP4 with converted chunks)
  constexpr int EPC = F::kElemsPerChunk, UNR = (MAXT >= 16 || (WD == MOE_FP4 && MAXT > 1)) ? F::kUnroll / 2 : F::kUnroll;
  const int rel = (int)blockIdx.x - cta0;
  if (rel < 0 || rel >= ncta || ie <= ib) return;
  const int H = p.H, I = p.I, lane = threadIdx.x & 31, warp = grp.tid() >> 5;
  const int64_t total = (int64_t)(ie - ib) * I;
  int64_t t0 = (int64_t)rel * total / ncta, t1 = (int64_t)(rel + 1) * total / ncta;
  if constexpr (MAXT > 1) {
    // rows of experts with more tokens cost more: split the rows so that each
    // CTA gets an equal share of rows x (tokens + 1) (the row's loads and
    // conversions, then one pass per token); every CTA computes the same split
    int64_t wtot = 0;
    for (int it = ib; it < ie; ++it) wtot += (int64_t)I * (tb.ntok[it] + 1);
    const int64_t w0 = rel * wtot / ncta, w1 = (rel + 1) * wtot / ncta;
    auto row_at = [&](int64_t wq) -> int64_t {  // first row whose weight span ends after wq
      int64_t acc = 0;
      for (int it = ib; it < ie; ++it) {
        const int64_t per = tb.ntok[it] + 1, span = (int64_t)I * per;
        if (wq < acc + span) return (int64_t)(it - ib) * I + (wq - acc + per - 1) / per;
        acc += span;
      }
      return total;
    };
    t0 = row_at(w0);
    t1 = rel + 1 == ncta ? total : row_at(w1);
  }
  const int nchunks = H / EPC;
  const int64_t rb = F::row_bytes(H);
  auto row_task = [&](int64_t task) {
    const int it = ib + (int)(task / I), i = (int)(task % I);
    const int ntok = tb.ntok[it];
    const RecView v = rec_view<WD>(tb.rec[it], H, I);
    const uint8_t* grow = v.gate + (int64_t)i * rb;
    const uint8_t* urow = v.up + (int64_t)i * rb;
    const uint8_t* gsc = (WD == MOE_FP4) ? v.gate_sc + (int64_t)i * (H / 16) : nullptr;
    const uint8_t* usc = (WD == MOE_FP4) ? v.up_sc + (int64_t)i * (H / 16) : nullptr;
    int tok[MAXT];
#pragma unroll
    for (int q = 0; q < MAXT; ++q) {
      int t = 0, hr, j;
      if (q < ntok) item_token(p, tb, it, q, &t, &hr, &j);
      tok[q] = t;
    }
    float ag[MAXT], au[MAXT];
#pragma unroll
    for (int q = 0; q < MAXT; ++q) { ag[q] = 0.f; au[q] = 0.f; }
    for (int c0 = 0; c0 < nchunks; c0 += 32 * UNR) {
      uint4 wg[UNR], wu[UNR];
      unsigned short sg[UNR], su[UNR];
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int c = c0 + lane + 32 * u;
        if (c < nchunks) {
          wg[u] = ld_w16<FRESH>(grow + (int64_t)c * 16);
          wu[u] = ld_w16<FRESH>(urow + (int64_t)c * 16);
          if (WD == MOE_FP4) {
            sg[u] = ld_w2<FRESH>(gsc + 2 * c);
            su[u] = ld_w2<FRESH>(usc + 2 * c);
          } else {
            sg[u] = su[u] = 0;
          }
        }
      }
      if constexpr (WB) {
        const RecView dv = rec_view<WD>(tb.dst[it], H, I);
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int c = c0 + lane + 32 * u;
          if (c < nchunks) {
            *reinterpret_cast<uint4*>(const_cast<uint8_t*>(dv.gate) + (int64_t)i * rb + (int64_t)c * 16) = wg[u];
            *reinterpret_cast<uint4*>(const_cast<uint8_t*>(dv.up) + (int64_t)i * rb + (int64_t)c * 16) = wu[u];
            if (WD == MOE_FP4) {
              *reinterpret_cast<unsigned short*>(const_cast<uint8_t*>(dv.gate_sc) + (int64_t)i * (H / 16) + 2 * c) = sg[u];
              *reinterpret_cast<unsigned short*>(const_cast<uint8_t*>(dv.up_sc) + (int64_t)i * (H / 16) + 2 * c) = su[u];
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int c = c0 + lane + 32 * u;
        if (c < nchunks) {
          if constexpr (WD == MOE_FP4 && MAXT > 1 && MAXT < 16) {
            // several tokens: each chunk's codes converted once (same sums as chunk_dot)
            // (activations in the quarter layout of x_to_f16)
            auto x_of = [&](int q) { return xs + (size_t)tok[q] * H + (size_t)c * 8; };
            fp4_chunk_tokens<MAXT, XT>(wg[u], sg[u], ntok, x_of, ag, H / 4);
            fp4_chunk_tokens<MAXT, XT>(wu[u], su[u], ntok, x_of, au, H / 4);
          } else {
#pragma unroll
            for (int q = 0; q < MAXT; ++q) {
              if (q < ntok) {
                if constexpr (WD == MOE_FP4) {  // activations in the quarter layout of x_to_f16
                  const XT* xr = xs + (size_t)tok[q] * H + (size_t)c * 8;
                  ag[q] += chunk_dot_fp4q(wg[u], sg[u], xr, H / 4);
                  au[q] += chunk_dot_fp4q(wu[u], su[u], xr, H / 4);
                } else {
                  const XT* xr = xs + (size_t)tok[q] * H + (size_t)c * EPC;
                  ag[q] += chunk_dot<WD, XT>(wg[u], sg[u], xr);
                  au[q] += chunk_dot<WD, XT>(wu[u], su[u], xr);
                }
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < MAXT; ++q) {
      if (q < ntok) {
        const float g = warp_sum(ag[q]);
        const float u = warp_sum(au[q]);
        if (lane == 0) {
          int t, hr, j;
          item_token(p, tb, it, q, &t, &hr, &j);
          p.h[(int64_t)hr * I + i] = g / (1.0f + expf(-g)) * u;
        }
      }
    }
  };
  for (int64_t task = t0 + warp; task < t1; task += grp.nw) row_task(task);
}

// Where W_down row `row` (and its FP4 scales) of item gi is read: its record,
// or, when STAGED, staged item j of this CTA in shared memory.
template <int WD, bool STAGED>
__device__ __forceinline__ void down_row(const ItemTable& tb, int j, int gi, int row, int n0, int nrows, int H, int I,
                                         const uint8_t* stage, int pitch, const uint8_t** drow, const uint8_t** dsc) {
  const int64_t rb = Fmt<WD>::row_bytes(I);
  if constexpr (STAGED) {
    const uint8_t* base = stage + (int64_t)j * pitch;
    *drow = base + (int64_t)(row - n0) * rb;
    *dsc = base + (int64_t)nrows * rb + (int64_t)(row - n0) * (I / 16);
  } else {
    const RecView v = rec_view<WD>(tb.rec[gi], H, I);
    *drow = v.down + (int64_t)row * rb;
    *dsc = (WD == MOE_FP4) ? v.down_sc + (int64_t)row * (I / 16) : nullptr;
  }
}
template <bool FRESH, bool STAGED>
__device__ __forceinline__ uint4 ld_down16(const uint8_t* q) {
  if constexpr (STAGED) return lds16(q); else return ld_w16<FRESH>(q);
}
template <bool FRESH, bool STAGED>
__device__ __forceinline__ unsigned short ld_down2(const uint8_t* q) {
  if constexpr (STAGED) return lds2(q); else return ld_w2<FRESH>(q);
}

// Staged h for the W_down phase.  float32 models: float32 rows, the chunks
// contiguous; bf16 models: float32 rows in two halves (see h_dot).  FP4
// models: f16 values (the SwiGLU intermediate
// rounded to f16, as in the FP4 prefill GEMMs), so the W_down dots run as
// mixed-precision f16 FMAs; each 32-value chunk (64 bytes) padded to 80
// bytes so that eight lanes reading eight consecutive chunks with 16-byte
// loads hit distinct banks.  h_chunk_stride: values of the staged type from
// one chunk to the next; h_row_floats: the staged row in float32 units.
template <int WD>
__host__ __device__ constexpr int h_chunk_stride() { return WD == MOE_FP4 ? 40 : Fmt<WD>::kElemsPerChunk; }
template <int WD>
__host__ __device__ constexpr int h_chunk_floats() { return WD == MOE_FP4 ? 20 : Fmt<WD>::kElemsPerChunk; }
template <int WD>
using HStage = typename std::conditional<WD == MOE_FP4, __half, float>::type;

// W_down chunk c of a row against the staged h row `hrow`.  bf16 models stage
// a row as two halves, floats 0-3 of every 8-value chunk and then floats 4-7,
// so the 16-byte loads of eight lanes reading eight consecutive chunks are
// contiguous (with whole 32-byte chunks they would be two-way bank
// conflicts); the products and their order are chunk_dot's.
template <int WD, typename HT>
__device__ __forceinline__ float h_dot(uint4 w, unsigned short sc, const HT* hrow, int c, int I) {
  if constexpr (WD == MOE_BF16) {
    const float* r = reinterpret_cast<const float*>(hrow);
    return dot8_bf16w(w, *reinterpret_cast<const float4*>(r + 4 * c), *reinterpret_cast<const float4*>(r + I / 2 + 4 * c));
  } else {
    return chunk_dot<WD, HT>(w, sc, hrow + (int64_t)c * h_chunk_stride<WD>());
  }
}

// W_down rows [n0, n0 + nrows) of items [ib, ie) -> os[row][t][j], by the
// warp group grp.  STAGED: the rows of item i sit in shared memory at
// stage + i * pitch (rows n0.., then their FP4 scales), copied there early.
template <int WD, int MAXT, bool FRESH, bool STAGED = false>
__device__ void phase2(const LayerParams& p, const ItemTable& tb, int ib, int ie, int n0, int nrows, float* hs,
                       float* os, const uint8_t* stage = nullptr, int pitch = 0, WarpGroup grp = whole_cta()) {
  if (STAGED && !in_bounds(p.dbg, ie <= p.stage_items && nrows <= p.rows_per_cta_max, 5)) return;
  using F = Fmt<WD>;
  constexpr int EPC = F::kElemsPerChunk;
  constexpr int kLanesPerRow = 8, kRowsPerWarp = 32 / kLanesPerRow;
  constexpr int kChunksPerLane = (MAXT >= 16 || (WD == MOE_FP4 && MAXT > 1)) ? 4 : 8;  // a lane still sums its chunks in order
  const int H = p.H, I = p.I, B = p.B, k = p.k, lane = threadIdx.x & 31, warp = grp.tid() >> 5;
  const int gt = grp.tid(), gn = grp.nthreads();
  const int ostride = B * (k + 1);
  const int nchunks = I / EPC;
  using HT = HStage<WD>;
  constexpr int CS = h_chunk_stride<WD>();     // in HT values
  const int hrow_f = nchunks * h_chunk_floats<WD>();  // staged row, float32 units
  const int hrow_h = nchunks * CS;                    // staged row, HT values
  const HT* hsv = reinterpret_cast<const HT*>(hs);
  int g0 = ib;
  while (g0 < ie) {
    int g1 = g0, used = 0;
    while (g1 < ie) {
      const int nt = tb.ntok[g1];
      if (used + nt * hrow_f > p.smem_h_floats && g1 > g0) break;
      used += nt * hrow_f;
      ++g1;
    }
    grp.sync();
    const uint32_t par = *h_bar_phase();
    if constexpr (WD == MOE_FP4 || WD == MOE_BF16) {
      // plain loads, four 16-byte loads in flight per thread, then stores:
      // FP4 models in the f16 padded layout (chunk c of a row at c * CS
      // values); bf16 models as two halves, floats 0-3 of every chunk, then
      // floats 4-7 (see h_dot)
      __shared__ int s_hrow[kMaxPairs + kMaxB];
      const int rows = tb.hbase[g1] - tb.hbase[g0];
      for (int rr = gt; rr < rows; rr += gn) {
        int g = g0;
        while (tb.hbase[g + 1] - tb.hbase[g0] <= rr) ++g;
        int t, hr, j;
        item_token(p, tb, g, rr - (tb.hbase[g] - tb.hbase[g0]), &t, &hr, &j);
        s_hrow[rr] = hr;
      }
      grp.sync();
      const int per = I / 4, n4 = rows * per;
      for (int e0 = gt; e0 < n4; e0 += 4 * gn) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = e0 + u * gn;
          if (e < n4) v[u] = __ldcg(reinterpret_cast<const float4*>(p.h + (int64_t)s_hrow[e / per] * I) + e % per);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = e0 + u * gn;
          if (e < n4) {
            const int r = e / per, f = (e % per) * 4;  // value index within the row
            if constexpr (WD == MOE_FP4) {
              const __half2 a = __floats2half2_rn(v[u].x, v[u].y), b = __floats2half2_rn(v[u].z, v[u].w);
              *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(hs) + (int64_t)r * hrow_h + (f / EPC) * CS + f % EPC) =
                  make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
            } else {
              *reinterpret_cast<float4*>(hs + (int64_t)r * hrow_h + ((f % EPC) ? I / 2 : 0) + (f / EPC) * 4) = v[u];
            }
          }
        }
      }
    } else {  // float32 models: h rows of the group, item-major, one bulk copy per row, all in flight together
      const int rows = tb.hbase[g1] - tb.hbase[g0];
      if (gt < 32) {
        fence_proxy_async_global();  // h was written through the generic proxy (ordered by a grid barrier)
        if (gt == 0) mbar_expect_tx(h_bar(), (uint32_t)(rows * I * 4));
        __syncwarp();
        for (int rr = gt; rr < rows; rr += 32) {
          int g = g0;
          while (tb.hbase[g + 1] - tb.hbase[g0] <= rr) ++g;
          int t, hr, j;
          item_token(p, tb, g, rr - (tb.hbase[g] - tb.hbase[g0]), &t, &hr, &j);
          bulk_g2s(hs + (int64_t)rr * I, p.h + (int64_t)hr * I, (uint32_t)(I * 4), h_bar());
        }
      }
      if (!mbar_wait(h_bar(), par)) {  // L2 copies: only a broken context gets here
        if (gt == 0) atomicExch(p.err, MOE_ERR_TIMEOUT);
        mbar_wait(h_bar(), par);
      }
    }
    grp.sync();
    if (gt == 0) *h_bar_phase() = par ^ 1u;
    // 8 lanes per row, 4 rows per warp: lane l of row group g reads chunks
    // l, l + 8, l + 16, ... of unit u0 + g in increasing order (8 in flight),
    // then the group's 8 partial sums reduce by a fixed butterfly
    const int rg = lane / kLanesPerRow, gl = lane % kLanesPerRow;
    if constexpr (MAXT == 1) {
      // one token per item: a row group takes two rows of the same item at
      // once, so each h chunk read from shared memory serves both (each row
      // keeps the order above: same chunks, same butterfly)
      const int npr = (nrows + 1) / 2;
      const int nunits2 = (g1 - g0) * npr;
      for (int u0 = warp * kRowsPerWarp; u0 < nunits2; u0 += grp.nw * kRowsPerWarp) {
        const int unit = u0 + rg;
        const bool live = unit < nunits2;
        const int gi = live ? g0 + unit / npr : g0;
        const int ra = live ? 2 * (unit % npr) : 0;
        const bool live_b = live && ra + 1 < nrows;
        const uint8_t *da = nullptr, *sa = nullptr, *db = nullptr, *sb = nullptr;
        if (live) down_row<WD, STAGED>(tb, gi, gi, n0 + ra, n0, nrows, H, I, stage, pitch, &da, &sa);
        if (live_b) down_row<WD, STAGED>(tb, gi, gi, n0 + ra + 1, n0, nrows, H, I, stage, pitch, &db, &sb);
        const HT* hrow = hsv + (int64_t)(tb.hbase[gi] - tb.hbase[g0]) * hrow_h;
        float acc_a = 0.f, acc_b = 0.f;
        constexpr int CPL = 4;
        for (int c0 = 0; c0 < nchunks; c0 += kLanesPerRow * CPL) {
          uint4 wa[CPL], wb[CPL];
          unsigned short ca[CPL], cb[CPL];
#pragma unroll
          for (int u = 0; u < CPL; ++u) {
            const int c = c0 + gl + kLanesPerRow * u;
            if (live && c < nchunks) {
              wa[u] = ld_down16<FRESH, STAGED>(da + (int64_t)c * 16);
              ca[u] = (WD == MOE_FP4) ? ld_down2<FRESH, STAGED>(sa + 2 * c) : (unsigned short)0;
            }
            if (live_b && c < nchunks) {
              wb[u] = ld_down16<FRESH, STAGED>(db + (int64_t)c * 16);
              cb[u] = (WD == MOE_FP4) ? ld_down2<FRESH, STAGED>(sb + 2 * c) : (unsigned short)0;
            }
          }
#pragma unroll
          for (int u = 0; u < CPL; ++u) {
            const int c = c0 + gl + kLanesPerRow * u;
            if (live && c < nchunks) acc_a += h_dot<WD, HT>(wa[u], ca[u], hrow, c, I);
            if (live_b && c < nchunks) acc_b += h_dot<WD, HT>(wb[u], cb[u], hrow, c, I);
          }
        }
        acc_a += __shfl_xor_sync(0xFFFFFFFFu, acc_a, 4);
        acc_a += __shfl_xor_sync(0xFFFFFFFFu, acc_a, 2);
        acc_a += __shfl_xor_sync(0xFFFFFFFFu, acc_a, 1);
        acc_b += __shfl_xor_sync(0xFFFFFFFFu, acc_b, 4);
        acc_b += __shfl_xor_sync(0xFFFFFFFFu, acc_b, 2);
        acc_b += __shfl_xor_sync(0xFFFFFFFFu, acc_b, 1);
        if (live && gl == 0) {
          int t, hr, j;
          item_token(p, tb, gi, 0, &t, &hr, &j);
          const bool okr = in_bounds(p.dbg, ra + (live_b ? 1 : 0) < p.rows_per_cta_max && t < B && j <= k, 4);
          if (okr) os[ra * ostride + t * (k + 1) + j] = acc_a;
          if (okr && live_b) os[(ra + 1) * ostride + t * (k + 1) + j] = acc_b;
        }
      }
      g0 = g1;
      continue;
    }
    const int nunits = (g1 - g0) * nrows;
    for (int u0 = warp * kRowsPerWarp; u0 < nunits; u0 += grp.nw * kRowsPerWarp) {
      const int unit = u0 + rg;
      const bool live = unit < nunits;
      const int gi = live ? g0 + unit / nrows : g0, row = live ? n0 + unit % nrows : n0;
      const uint8_t *drow = nullptr, *dsc = nullptr;
      if (live) down_row<WD, STAGED>(tb, gi, gi, row, n0, nrows, H, I, stage, pitch, &drow, &dsc);
      const int hbase = tb.hbase[gi] - tb.hbase[g0];
      const int ntok = live ? tb.ntok[gi] : 0;
      float acc[MAXT];
#pragma unroll
      for (int q = 0; q < MAXT; ++q) acc[q] = 0.f;
      for (int c0 = 0; c0 < nchunks; c0 += kLanesPerRow * kChunksPerLane) {
        uint4 w[kChunksPerLane];
        unsigned short sc[kChunksPerLane];
#pragma unroll
        for (int u = 0; u < kChunksPerLane; ++u) {
          const int c = c0 + gl + kLanesPerRow * u;
          if (live && c < nchunks) {
            w[u] = ld_down16<FRESH, STAGED>(drow + (int64_t)c * 16);
            sc[u] = (WD == MOE_FP4) ? ld_down2<FRESH, STAGED>(dsc + 2 * c) : (unsigned short)0;
          }
        }
#pragma unroll
        for (int u = 0; u < kChunksPerLane; ++u) {
          const int c = c0 + gl + kLanesPerRow * u;
          if (live && c < nchunks) {
            if constexpr (WD == MOE_FP4 && MAXT > 1 && MAXT < 16) {
              auto h_of = [&](int q) { return hsv + (int64_t)(hbase + q) * hrow_h + (int64_t)c * CS; };
              fp4_chunk_tokens<MAXT, HT>(w[u], sc[u], ntok, h_of, acc);
            } else {
#pragma unroll
              for (int q = 0; q < MAXT; ++q)
                if (q < ntok) acc[q] += h_dot<WD, HT>(w[u], sc[u], hsv + (int64_t)(hbase + q) * hrow_h, c, I);
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < MAXT; ++q) {
        float a = acc[q];
        a += __shfl_xor_sync(0xFFFFFFFFu, a, 4);
        a += __shfl_xor_sync(0xFFFFFFFFu, a, 2);
        a += __shfl_xor_sync(0xFFFFFFFFu, a, 1);
        if (live && gl == 0 && q < ntok) {
          int t, hr, j;
          item_token(p, tb, gi, q, &t, &hr, &j);
          if (in_bounds(p.dbg, row - n0 < p.rows_per_cta_max && t < B && j <= k, 4))
            os[(row - n0) * ostride + t * (k + 1) + j] = a;
        }
      }
    }
    g0 = g1;
  }
  grp.sync();
}

// Items of the call's resident experts (hits in U order, then the shared
// expert) and the call's pair order and weights, from this CTA's own control
// tables; returns the item count.  All threads call.
static __device__ int local_items(const LayerParams& p, const CtrlSmem& cs, ItemTable& tb) {
  const int n_u = cs.nu, npairs = p.B * p.k, nres = n_u - cs.nmiss;
  for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
    tb.perm[i] = cs.perm[i];
    tb.pair_w[i] = cs.w[i];
  }
  for (int r = threadIdx.x; r < n_u; r += blockDim.x) {
    if (cs.fill[r]) continue;
    const int i = r - cs.mrank[r];  // hits before rank r
    if (!in_bounds(p.dbg, cs.slot[r] >= 0 && cs.slot[r] < p.C && i >= 0 && i < kMaxItems, 1)) continue;
    tb.rec[i] = p.slots + (int64_t)cs.slot[r] * p.S;
    tb.dst[i] = nullptr;
    tb.pair0[i] = cs.off[r];
    tb.ntok[i] = cs.off[r + 1] - cs.off[r];
  }
  if (threadIdx.x == 0 && p.has_shared) {
    tb.rec[nres] = p.shared_rec;
    tb.dst[nres] = nullptr;
    tb.ntok[nres] = p.B;
    tb.pair0[nres] = -1;
  }
  __syncthreads();
  const int n = nres + (p.has_shared ? 1 : 0);
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < n; ++i) { tb.hbase[i] = run; run += tb.ntok[i]; }
    tb.hbase[n] = run;
  }
  __syncthreads();
  return n;
}

// y_t[n] = sum_j w_tj o_tj[n] (+ shared) in rank order for this CTA's rows.
template <int WD>
__device__ __forceinline__ void combine_rows(const LayerParams& p, const ItemTable& tb, const float* os, int n0,
                                             int nrows) {
  const int B = p.B, k = p.k, H = p.H, ostride = B * (k + 1);
  for (int e = threadIdx.x; e < nrows * B; e += blockDim.x) {
    const int nl = e / B, t = e % B, n = n0 + nl;
    if (!in_bounds(p.dbg, n < H && nl < p.rows_per_cta_max, 6)) continue;
    const float* o = os + nl * ostride + t * (k + 1);
    float acc = 0.f;
    for (int j = 0; j < k; ++j) acc = fmaf(tb.pair_w[t * k + j], o[j], acc);
    if (p.has_shared) acc += o[k];
    if constexpr (WD == MOE_FP32)
      reinterpret_cast<float*>(p.y)[(int64_t)t * H + n] = acc;
    else
      reinterpret_cast<__nv_bfloat16*>(p.y)[(int64_t)t * H + n] = __float2bfloat16_rn(acc);
  }
}

// A bounded wait of this CTA gave up: its output rows become NaN, so a caller
// that reads y without checking the status still cannot mistake it for a result.
template <int WD>
__device__ void poison_rows(const LayerParams& p, int n0, int nrows) {
  for (int e = threadIdx.x; e < nrows * p.B; e += blockDim.x) {
    const int t = e % p.B, n = n0 + e / p.B;
    if constexpr (WD == MOE_FP32)
      reinterpret_cast<float*>(p.y)[(int64_t)t * p.H + n] = __int_as_float(0x7FC00000);
    else
      reinterpret_cast<__nv_bfloat16*>(p.y)[(int64_t)t * p.H + n] = __ushort_as_bfloat16((unsigned short)0x7FC0);
  }
}

constexpr int kLookupCtr = 0;  // per-call counter of CTAs done with the residency lookups
constexpr int kTlSlots = 20;   // phase timestamps per call (profiling)

// Wait (thread 0 of the group polls, the group waits on it) until *c >=
// target; false after limit_ns (MOE_ERR_TIMEOUT is then recorded).
static __device__ bool wait_count(const unsigned* c, unsigned target, WarpGroup g, int* err,
                                  unsigned long long limit_ns = 2000000000ull) {
  __shared__ int s_ok[3];
  if (g.tid() == 0) {
    int ok = 1;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
      if (v >= target) break;
      if (globaltimer_ns() - t0 > limit_ns) {
        atomicExch(err, MOE_ERR_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    s_ok[g.bar] = ok;
  }
  g.sync();
  return s_ok[g.bar] != 0;
}

__device__ __forceinline__ int ld_relaxed_s32(const int* q) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(q) : "memory");
  return v;
}

// The layer kernel of one decode call.  Every CTA routes the call and looks
// its experts up itself, so the resident experts' rows start streaming at
// once; the control CTA also picks the victims, writes the plan and publishes
// the host summary (the miss list the host issues copies from), and after the
// first grid barrier (when every CTA has done its lookups) commits recency
// and residency.  In copy-fill mode each fill is consumed as its stream flag
// arrives; a CTA that has waited wait_gu_ns for a gate/up half, or wait_dn_ns
// for a W_down half, stops waiting: its partial sums go to o_part and the
// completion kernel, ordered after the call's copies on the stream, finishes
// its rows.  A call's result never depends on copy-engine work progressing
// while this kernel holds the SMs.
template <int WD, int MAXT>
__global__ void __launch_bounds__(kThreads, 1) layer_kernel(LayerParams p) {
  using XT = typename std::conditional<WD == MOE_FP32, float, __nv_bfloat16>::type;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ CtrlSmem cs;
  __shared__ ItemTable tb;
  __shared__ __align__(8) uint64_t s_stage;
  __shared__ __align__(8) uint64_t s_xin;
  __shared__ int s_flag;
  const int H = p.H, B = p.B, k = p.k;
  const int G = gridDim.x;
  const bool ctrl = blockIdx.x == 0;
  XT* xs = reinterpret_cast<XT*>(smem);
  float* hs = reinterpret_cast<float*>(smem + (((size_t)B * H * sizeof(XT) + 15) & ~(size_t)15));
  float* os = hs + p.smem_h_floats;
  const int n0 = (int)((int64_t)blockIdx.x * H / G), n1 = (int)((int64_t)(blockIdx.x + 1) * H / G);
  const int nrows = n1 - n0;
  const int ostride = B * (k + 1);
  const bool rec = p.tl && blockIdx.x == 1 && threadIdx.x == 0;

  grid_dep_wait();  // the previous call's commit and outputs are visible
  grid_dep_launch();
  // the router warps' first token's logits, requested before anything else
  // (E <= 256: up to eight per lane): issued later, behind the CTA's other
  // start-up traffic, they landed 3.5 us after the kernel started instead of 1.5
  float lg_pre[8];
  const bool use_pre = p.E <= 256 && (int)(threadIdx.x >> 5) < B;
  if (use_pre) {
    const float* lg = p.logits + (size_t)(threadIdx.x >> 5) * p.E;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = (threadIdx.x & 31) + 32 * q;
      lg_pre[q] = e < p.E ? lg[e] : 0.f;
    }
  }
  int mrow[kMaxE / kThreads];  // the layer's residency row, read in route_lookup
  load_map_row(p, mrow);
  if (rec) p.tl[0] = globaltimer_ns();
  if (p.tl_next && blockIdx.x == 0 && threadIdx.x >= 32 && threadIdx.x < 32 + kTlSlots) p.tl_next[threadIdx.x - 32] = 0ull;
  // warp 0 goes straight to the router (token 0): set-up with fences or
  // long-latency operations runs in other warps
  if (threadIdx.x == kThreads - 96) {
    s_flag = 0;  // read only after CTA barriers
    h_bar_init();
  }
  if (threadIdx.x == kThreads - 64) {  // the counter add may take a while
    call_seq_init(p);
    p.cst->part[blockIdx.x] = -1;
    if (ctrl) p.cst->gu_stop = 0;  // before the plan flag, which every later writer acquires
  }
  // activations into shared memory by one bulk copy (waited for before phase 1),
  // or by plain loads when the caller's pointer is not 16-byte aligned
  const uint32_t xbytes = (uint32_t)((size_t)B * H * sizeof(XT));
  const bool x_bulk = ((uintptr_t)p.x & 15) == 0;
  if (x_bulk && threadIdx.x == kThreads - 32) {  // the last warp: the router warps start at once
    mbar_init(&s_xin, 1);
    fence_mbar_init();
    mbar_expect_tx(&s_xin, xbytes);
    bulk_g2s(xs, p.x, xbytes, &s_xin);
  }
  if (!x_bulk) {
    const uint4* src = reinterpret_cast<const uint4*>(p.x);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    for (int i = threadIdx.x; i < (int)(xbytes / 16); i += blockDim.x) dst[i] = src[i];
  }

  // ---- the shared expert needs no routing: warps 1.. stream its gate/up rows
  // (split over every CTA) while warp 0 routes the call
  const bool early_shared = p.has_shared && x_bulk && WD != MOE_FP4;  // FP4 converts x first
  if (early_shared && threadIdx.x >= 32) {
    const WarpGroup rest{1, kWarps - 1, 1};
    if (threadIdx.x == 32) {
      tb.rec[kEarlyItem] = p.shared_rec;
      tb.dst[kEarlyItem] = nullptr;
      tb.ntok[kEarlyItem] = B;
      tb.pair0[kEarlyItem] = -1;
    }
    rest.sync();  // the entry and the activations' mbarrier are initialised
    if (mbar_wait(&s_xin, 0)) phase1<WD, MAXT, false>(p, tb, kEarlyItem, kEarlyItem + 1, 0, G, x_dot<WD>(xs), rest);
  }

  // ---- 0. routing and lookup (every CTA); victims, plan, summary (control CTA)
  int err = route_lookup(p, cs, ctrl, mrow, use_pre ? lg_pre : nullptr);
  // counters of the next call (this call's were cleared by the previous one);
  // on every path, errors included
  if (ctrl && threadIdx.x >= kThreads - kWaveCtrs) cseq().wave_next[threadIdx.x - (kThreads - kWaveCtrs)] = 0u;
  if (ctrl) err = err == MOE_OK ? choose_victims(p, cs) : (publish_error(p, cs, err), err);
  if (err != MOE_OK) {  // capacity: every CTA; inconsistent victim list: the control CTA
    if (x_bulk) mbar_wait(&s_xin, 0);  // no bulk copy outlives its CTA
    return;
  }
  if (ctrl && p.tl) p.tl[10] = globaltimer_ns();
  if (rec) p.tl[1] = globaltimer_ns();
  if (p.tl && threadIdx.x == 0) atomicMax(p.tl + 18, globaltimer_ns());

  // ---- 1. gate/up rows of the resident experts and the shared expert --------------
  const int n_res = local_items(p, cs, tb);
  // this CTA's W_down rows of the resident experts: the first n_stage items
  // into shared memory by bulk copies completing on s_stage, the rest into L2
  const int n_stage = nrows > 0 ? min(n_res, p.stage_items) : 0;
  const uint8_t* stage = smem + p.stage_off;
  {
    const int64_t rb = Fmt<WD>::row_bytes(p.I), sb = (WD == MOE_FP4) ? p.I / 16 : 0;
    if (threadIdx.x == 0 && n_stage > 0) {
      mbar_init(&s_stage, 1);
      fence_mbar_init();
      mbar_expect_tx(&s_stage, (uint32_t)(n_stage * nrows * (rb + sb)));
      for (int j = 0; j < n_stage; ++j) {
        const RecView v = rec_view<WD>(tb.rec[j], H, p.I);
        uint8_t* dst = smem + p.stage_off + (int64_t)j * p.stage_pitch;
        bulk_g2s(dst, v.down + (int64_t)n0 * rb, (uint32_t)(nrows * rb), &s_stage);
        if (WD == MOE_FP4) bulk_g2s(dst + nrows * rb, v.down_sc + (int64_t)n0 * sb, (uint32_t)(nrows * sb), &s_stage);
      }
    }
    if ((int)threadIdx.x >= n_stage && (int)threadIdx.x < n_res && nrows > 0) {
      const RecView v = rec_view<WD>(tb.rec[threadIdx.x], H, p.I);
      prefetch_l2(v.down + (int64_t)n0 * rb, (uint32_t)(nrows * rb));
      if (WD == MOE_FP4) prefetch_l2(v.down_sc + (int64_t)n0 * sb, (uint32_t)(nrows * sb));
    }
  }
  if (x_bulk && !mbar_wait(&s_xin, 0)) {
    if (threadIdx.x == 0) atomicExch(p.err, MOE_ERR_TIMEOUT);
    mbar_wait(&s_xin, 0);
    if (n_stage > 0) mbar_wait(&s_stage, 0);
    poison_rows<WD>(p, n0, nrows);
    return;
  }
  if constexpr (WD == MOE_FP4) {
    x_to_f16<WD>(xs, B, H);
    __syncthreads();
  }
  // this CTA has read the residency table: the control CTA may commit
  if (threadIdx.x == 0) atomicAdd(&cseq().wave_ctr[kLookupCtr], 1u);

  // ---- 1./2. gate/up rows of the resident experts and the shared expert (CTAs
  // 1..), one grid barrier, then every CTA's W_down rows; the control CTA
  // commits recency and residency meanwhile, once every CTA has done its lookups
  // (the shared expert, item n_res - 1, already done when early_shared)
  if (!ctrl) phase1<WD, MAXT, false>(p, tb, 0, early_shared ? n_res - 1 : n_res, 1, G - 1, x_dot<WD>(xs));
  if (rec) p.tl[2] = globaltimer_ns();
  if (p.tl && !ctrl && threadIdx.x == 0) {
    const unsigned long long now = globaltimer_ns();
    atomicMax(p.tl + 16, ~now);  // earliest, as a complement
    atomicMax(p.tl + 17, now);
  }
  bool bad = false;
  if (ctrl) {
    bad = !wait_count(&cseq().wave_ctr[kLookupCtr], (unsigned)G, whole_cta(), p.err);
    if (!bad) {
      control_commit(p, cs);
      compact_oldest(p, cs);
    }
    if (p.tl && threadIdx.x == 0) p.tl[11] = globaltimer_ns();
  }
  bad = !grid_barrier(p.bar, p.err) || bad;
  if (n_stage > 0 && !mbar_wait(&s_stage, 0)) {  // the staging copies never leave this CTA in flight
    if (threadIdx.x == 0) atomicExch(p.err, MOE_ERR_TIMEOUT);
    mbar_wait(&s_stage, 0);
    s_flag = 1;
  }
  if (bad) s_flag = 1;
  __syncthreads();
  if (s_flag) {  // a bounded wait gave up (recorded in p.err)
    poison_rows<WD>(p, n0, nrows);
    return;
  }
  if (rec) p.tl[3] = globaltimer_ns();
  for (int i = threadIdx.x; i < nrows * ostride; i += blockDim.x) os[i] = 0.f;
  phase2<WD, MAXT, false, true>(p, tb, 0, n_stage, n0, nrows, hs, os, stage, p.stage_pitch);
  phase2<WD, MAXT, false>(p, tb, n_stage, n_res, n0, nrows, hs, os);
  if (rec) p.tl[4] = globaltimer_ns();

  // the fills' slots come from the control CTA's plan (a call without misses,
  // which this CTA's own lookup shows, has no fills and needs no plan)
  const Plan* pl = p.plan;
  int nf = 0;
  if (cs.nmiss > 0) {
    bool ok = true;
    if (!ctrl && wait_flag(p.plan_flag, cseq().seq, nullptr, 5000000000ull, 32) != 0) {
      if (threadIdx.x == 0) atomicExch(p.err, MOE_ERR_TIMEOUT);
      ok = false;
    }
    if (ok && pl->err != MOE_OK) ok = false;
    if (!ok) return;
    nf = pl->n_items[1];
  }
  if (rec) p.tl[7] = globaltimer_ns();

  // ---- 3. fills ----------------------------------------------------------------------
  if (nf > 0 && p.device_fill) {
    // device-driven fills: pull each missed record from the host pool, use it
    // for this call and store it in its slot; each CTA copies its own W_down
    // rows of every fill into the slots and then reads them there, not over
    // the link
    const int n_all = load_items(p, pl, 1, tb, n_res, true);
    copy_down_rows<WD>(p, tb, n_res, n_all, n0, nrows);
    if (!ctrl) phase1<WD, MAXT, false, true>(p, tb, n_res, n_all, 1, G - 1, x_dot<WD>(xs));
    if (!grid_barrier(p.bar, p.err)) {
      poison_rows<WD>(p, n0, nrows);
      return;
    }
    for (int it = n_res + (int)threadIdx.x; it < n_all; it += blockDim.x) tb.rec[it] = tb.dst[it];
    __syncthreads();
    phase2<WD, MAXT, true>(p, tb, n_res, n_all, n0, nrows, hs, os);
  } else if (nf > 0) {
    // copy mode: each fill as soon as its copy has landed
    load_items(p, pl, 1, tb);
    for (int f = 0; f < nf; ++f) {
      if (wait_flag(&p.fill_flags[f], cseq().seq, &p.cst->gu_stop, p.wait_gu_ns) != 0) {
        if (threadIdx.x == 0) atomicExch(&p.cst->gu_stop, 1);  // every CTA stops waiting
        break;
      }
      if (rec && f == 0) p.tl[5] = globaltimer_ns();
      phase1<WD, MAXT, true>(p, tb, f, f + 1, 0, G, x_dot<WD>(xs));
    }
    if (rec) p.tl[6] = globaltimer_ns();
    if (!grid_barrier(p.bar, p.err)) {
      poison_rows<WD>(p, n0, nrows);
      return;
    }
    if (threadIdx.x == 0) s_flag = ld_relaxed_s32(&p.cst->gu_stop);
    __syncthreads();
    int handed = s_flag ? 0 : -1;  // fills whose W_down rows os holds when handing over
    for (int f = 0; f < nf && handed < 0; ++f) {
      if (wait_flag(&p.fill_flags[kMaxU + f], cseq().seq, nullptr, p.wait_dn_ns) != 0) {
        handed = f;
        break;
      }
      if (rec && f == nf - 1) p.tl[8] = globaltimer_ns();
      phase2<WD, MAXT, true>(p, tb, f, f + 1, n0, nrows, hs, os);
    }
    if (handed >= 0) {
      // the completion kernel finishes this CTA's rows after the copies
      float* dst = p.o_part + (int64_t)blockIdx.x * p.o_part_floats;
      for (int i = threadIdx.x; i < nrows * ostride; i += blockDim.x) dst[i] = os[i];
      if (threadIdx.x == 0) p.cst->part[blockIdx.x] = handed;
      return;
    }
  }

  // ---- 4. weighted combine in rank order --------------------------------------------
  combine_rows<WD>(p, tb, os, n0, nrows);
  if (rec) p.tl[9] = globaltimer_ns();
  if (p.tl && threadIdx.x == 0) atomicMax(p.tl + 19, globaltimer_ns());
}

// Completion kernel of a copy-fill call, launched on the compute stream after
// the call's copies have ended.  Every fill flag is final by then: if one
// carries the error bit (the host could not issue a copy), the call is undone.
// Otherwise the CTAs that handed over finish their rows: the fills' gate/up
// rows when the layer kernel stopped before them (then every CTA takes part
// and one grid barrier follows), the remaining W_down rows from the saved
// partial sums, and the combine, with the layer kernel's code and summation
// order, so the outputs are bitwise the same as when it finishes alone.
template <int WD, int MAXT>
__global__ void __launch_bounds__(kThreads, 1) layer_finish_kernel(LayerParams p) {
  using XT = typename std::conditional<WD == MOE_FP32, float, __nv_bfloat16>::type;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ ItemTable tb;
  __shared__ int s_state[3];
  const int H = p.H, B = p.B, k = p.k;
  const int G = gridDim.x;
  XT* xs = reinterpret_cast<XT*>(smem);
  float* hs = reinterpret_cast<float*>(smem + (((size_t)B * H * sizeof(XT) + 15) & ~(size_t)15));
  float* os = hs + p.smem_h_floats;
  const int n0 = (int)((int64_t)blockIdx.x * H / G), n1 = (int)((int64_t)(blockIdx.x + 1) * H / G);
  const int nrows = n1 - n0;
  const int ostride = B * (k + 1);
  const Plan* pl = p.plan;
  if (pl->err != MOE_OK) return;
  const int nf = pl->n_items[1];
  if (threadIdx.x == 0) {
    h_bar_init();
    call_seq_init(p);  // launched from the host only (copy-fill calls)
    int failed = 0;
    for (int f = 0; f < nf; ++f)
      if (p.fill_flags[f] != p.seq || p.fill_flags[kMaxU + f] != p.seq) failed = 1;
    s_state[0] = failed;
    s_state[1] = p.cst->gu_stop;
    s_state[2] = p.cst->part[blockIdx.x];
  }
  __syncthreads();
  if (s_state[0]) {
    if (blockIdx.x == 0) undo_call(p);
    return;
  }
  const int gu = s_state[1], part = s_state[2];
  if (!gu && part < 0) return;  // the layer kernel finished this CTA's rows
  for (int i = threadIdx.x; i < B * k; i += blockDim.x) {
    tb.perm[i] = pl->perm[i];
    tb.pair_w[i] = pl->pair_w[i];
  }
  load_items(p, pl, 1, tb);
  if (gu) {
    const int nvec = (int)((size_t)B * H * sizeof(XT) / 16);
    const uint4* src = reinterpret_cast<const uint4*>(p.x);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    for (int i = threadIdx.x; i < nvec; i += blockDim.x) dst[i] = src[i];
    __syncthreads();
    if constexpr (WD == MOE_FP4) {
      x_to_f16<WD>(xs, B, H);
      __syncthreads();
    }
    phase1<WD, MAXT, false>(p, tb, 0, nf, 0, G, x_dot<WD>(xs));
    if (!grid_barrier(p.bar, p.err)) {
      poison_rows<WD>(p, n0, nrows);
      return;
    }
  }
  const float* srcp = p.o_part + (int64_t)blockIdx.x * p.o_part_floats;
  for (int i = threadIdx.x; i < nrows * ostride; i += blockDim.x) os[i] = srcp[i];
  __syncthreads();
  phase2<WD, MAXT, false>(p, tb, gu ? 0 : part, nf, n0, nrows, hs, os);
  combine_rows<WD>(p, tb, os, n0, nrows);
  if (blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(p.deferred, 1ull);
}

// Launch of one instantiation as a cooperative grid (every CTA resident, for
// the grid barriers), optionally as a programmatic dependent of the previous
// launch on the stream; dynamic shared memory is raised once per kernel to the
// largest size asked for.
template <typename K>
static cudaError_t launch_coop(K fn, size_t* smem_set, const LayerParams& p, int grid, size_t smem, bool pdl,
                               cudaStream_t s) {
  if (smem > *smem_set) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    *smem_set = smem;
  }
  void* args[] = {const_cast<LayerParams*>(&p)};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelExC(&cfg, (const void*)fn, args);
}

template <int WD, int MAXT>
cudaError_t launch_t(const LayerParams& p, int grid, size_t smem, bool pdl, cudaStream_t s) {
  static size_t smem_set = 0;
  return launch_coop(layer_kernel<WD, MAXT>, &smem_set, p, grid, smem, pdl, s);
}

template <int WD, int MAXT>
cudaError_t launch_finish_t(const LayerParams& p, int grid, size_t smem, cudaStream_t s) {
  static size_t smem_set = 0;
  return launch_coop(layer_finish_kernel<WD, MAXT>, &smem_set, p, grid, smem, false, s);
}

}  // namespace moe
