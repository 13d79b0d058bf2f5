// Decode-size grouped SwiGLU expert FFN read straight out of cache slots.
//
// FreeToken write-up: decode is memory-bound, each routed expert's weights
// are read once per token ("decode: cache misses and the CPU bandwidth
// limit"); the GPU evaluates G = H ∪ F as one grouped FFN once the fills have
// landed, and the partial sums merge exactly ("measured bandwidths decide the
// split", Fig. 2 caption).
//
// One cooperative, persistent launch per item list (resident experts + the
// shared expert, or this call's fills), 512 threads per CTA, one CTA per SM:
//  phase 1  h[pair][i] = SiLU(W_gate[i]·x_t) * (W_up[i]·x_t); a warp streams
//           one gate row and one up row (16-byte non-allocating loads, FP4
//           dequantised in registers) and serves every token routed to the
//           expert from the same registers;
//  barrier  (grid-wide, bounded wait)
//  phase 2  o[pair][n] = W_down[n]·h[pair]; each CTA owns a contiguous range
//           of output rows n for all experts of the list, so it can finish
//           the weighted combine y_t[n] = sum_j w_tj o_tj[n] (+ shared) in rank
//           order without another grid-wide step; its W_down rows are
//           prefetched into L2 at kernel start.
// Every dot product has a fixed summation order that does not depend on which
// launch evaluates it, so outputs are bitwise identical whatever the hit/miss
// pattern or slot placement.
#include "params.cuh"

namespace moe {



__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ unsigned short ld_stream_u16(const void* p) {
  unsigned short r;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// two e2m1 codes (low nibble = first element) -> two floats
__device__ __forceinline__ float2 e2m1x2_to_float2(uint32_t byte) {
  uint32_t h2;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h2) : "r"(byte));
  __half2 hv = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hv);  // .x = low half, .y = high half
}

// two e4m3 bytes (low byte first) -> two floats
__device__ __forceinline__ float2 e4m3x2_to_float2(unsigned short two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
  __half2 hv = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hv);
}

// ---- per-format row access --------------------------------------------------
// A "chunk" is 16 bytes of a row's element stream:
//   fp32: 4 elements, bf16: 8 elements, fp4: 32 elements (+ 2 scale bytes).
template <int WD>
struct Fmt;

template <>
struct Fmt<0> {
  static constexpr int kElemsPerChunk = 4;
  static constexpr int kUnroll = 4;
  __device__ static int64_t row_bytes(int K) { return (int64_t)K * 4; }
};
template <>
struct Fmt<1> {
  static constexpr int kElemsPerChunk = 8;
  static constexpr int kUnroll = 4;
  __device__ static int64_t row_bytes(int K) { return (int64_t)K * 2; }
};
template <>
struct Fmt<2> {
  static constexpr int kElemsPerChunk = 32;
  static constexpr int kUnroll = 2;
  __device__ static int64_t row_bytes(int K) { return (int64_t)K / 2; }
};

// Record offsets of the three matrices' element streams and (FP4) scales.
struct RecView {
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* down;
  const uint8_t* gate_sc;
  const uint8_t* up_sc;
  const uint8_t* down_sc;
};

template <int WD>
__device__ __forceinline__ RecView rec_view(const uint8_t* rec, int H, int I) {
  RecView v;
  const int64_t HI = (int64_t)H * I;
  if (WD == 0) {
    v.gate = rec; v.up = rec + HI * 4; v.down = rec + 2 * HI * 4;
    v.gate_sc = v.up_sc = v.down_sc = nullptr;
  } else if (WD == 1) {
    v.gate = rec; v.up = rec + HI * 2; v.down = rec + 2 * HI * 2;
    v.gate_sc = v.up_sc = v.down_sc = nullptr;
  } else {
    v.gate = rec; v.up = rec + HI / 2; v.down = rec + HI;
    const uint8_t* sc = rec + 3 * HI / 2;
    v.gate_sc = sc; v.up_sc = sc + HI / 16; v.down_sc = sc + 2 * HI / 16;
  }
  return v;
}

// Dot of one 16-byte weight chunk with the matching activation elements.
// xs points at element 0 of the chunk in a float (fp32) / bf16 vector held in
// shared memory (phase 1) or at float h values (phase 2).
template <int WD, typename VT>
__device__ __forceinline__ float chunk_dot(uint4 w, unsigned short sc2, const VT* xs);

template <>
__device__ __forceinline__ float chunk_dot<0, float>(uint4 w, unsigned short, const float* xs) {
  float4 a = *reinterpret_cast<const float4*>(xs);
  float acc = __uint_as_float(w.x) * a.x;
  acc = fmaf(__uint_as_float(w.y), a.y, acc);
  acc = fmaf(__uint_as_float(w.z), a.z, acc);
  acc = fmaf(__uint_as_float(w.w), a.w, acc);
  return acc;
}

__device__ __forceinline__ float dot8_bf16w(uint4 w, float4 a, float4 b) {
  float acc = bf16lo(w.x) * a.x;
  acc = fmaf(bf16hi(w.x), a.y, acc);
  acc = fmaf(bf16lo(w.y), a.z, acc);
  acc = fmaf(bf16hi(w.y), a.w, acc);
  acc = fmaf(bf16lo(w.z), b.x, acc);
  acc = fmaf(bf16hi(w.z), b.y, acc);
  acc = fmaf(bf16lo(w.w), b.z, acc);
  acc = fmaf(bf16hi(w.w), b.w, acc);
  return acc;
}

template <>
__device__ __forceinline__ float chunk_dot<1, __nv_bfloat16>(uint4 w, unsigned short, const __nv_bfloat16* xs) {
  uint4 xv = *reinterpret_cast<const uint4*>(xs);
  float4 a = make_float4(bf16lo(xv.x), bf16hi(xv.x), bf16lo(xv.y), bf16hi(xv.y));
  float4 b = make_float4(bf16lo(xv.z), bf16hi(xv.z), bf16lo(xv.w), bf16hi(xv.w));
  return dot8_bf16w(w, a, b);
}

template <>
__device__ __forceinline__ float chunk_dot<1, float>(uint4 w, unsigned short, const float* xs) {
  float4 a = *reinterpret_cast<const float4*>(xs);
  float4 b = *reinterpret_cast<const float4*>(xs + 4);
  return dot8_bf16w(w, a, b);
}

// 16 e2m1 codes (8 bytes) against 16 activation values.
template <typename VT>
__device__ __forceinline__ float block16_dot(uint32_t c0, uint32_t c1, const VT* xs);

template <>
__device__ __forceinline__ float block16_dot<__nv_bfloat16>(uint32_t c0, uint32_t c1, const __nv_bfloat16* xs) {
  uint4 xa = *reinterpret_cast<const uint4*>(xs);
  uint4 xb = *reinterpret_cast<const uint4*>(xs + 8);
  const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
  float acc = 0.f;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const uint32_t byte = ((b < 4 ? c0 : c1) >> (8 * (b & 3))) & 0xFFu;
    float2 w2 = e2m1x2_to_float2(byte);
    acc = fmaf(w2.x, bf16lo(xw[b]), acc);
    acc = fmaf(w2.y, bf16hi(xw[b]), acc);
  }
  return acc;
}

template <>
__device__ __forceinline__ float block16_dot<float>(uint32_t c0, uint32_t c1, const float* xs) {
  float acc = 0.f;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const uint32_t byte = ((b < 4 ? c0 : c1) >> (8 * (b & 3))) & 0xFFu;
    float2 w2 = e2m1x2_to_float2(byte);
    acc = fmaf(w2.x, xs[2 * b], acc);
    acc = fmaf(w2.y, xs[2 * b + 1], acc);
  }
  return acc;
}

template <>
__device__ __forceinline__ float chunk_dot<2, __nv_bfloat16>(uint4 w, unsigned short sc2, const __nv_bfloat16* xs) {
  float2 s = e4m3x2_to_float2(sc2);
  float a0 = block16_dot<__nv_bfloat16>(w.x, w.y, xs);
  float a1 = block16_dot<__nv_bfloat16>(w.z, w.w, xs + 16);
  return fmaf(a1, s.y, a0 * s.x);
}

template <>
__device__ __forceinline__ float chunk_dot<2, float>(uint4 w, unsigned short sc2, const float* xs) {
  float2 s = e4m3x2_to_float2(sc2);
  float a0 = block16_dot<float>(w.x, w.y, xs);
  float a1 = block16_dot<float>(w.z, w.w, xs + 16);
  return fmaf(a1, s.y, a0 * s.x);
}

// ---- item bookkeeping -------------------------------------------------------
struct Item {
  const uint8_t* rec;
  int ntok;
  int pair0;   // index into perm of the first pair (routed experts)
  bool shared;
};

struct ItemTable {
  const uint8_t* rec[kMaxItems];
  int ntok[kMaxItems];
  int pair0[kMaxItems];   // -1 for the shared expert
  int hbase[kMaxItems + 1];  // running token count (h rows in item order)
};

__device__ __forceinline__ Item make_item(const FfnParams& p, const Plan* pl, int idx) {
  Item it;
  const int r = pl->items[p.which][idx];
  if (r == pl->n_u) {
    it.rec = p.shared_rec;
    it.ntok = p.B;
    it.pair0 = 0;
    it.shared = true;
  } else {
    it.rec = p.slots + (int64_t)pl->u_slot[r] * p.S;
    it.pair0 = pl->u_off[r];
    it.ntok = pl->u_off[r + 1] - it.pair0;
    it.shared = false;
  }
  return it;
}

__device__ __forceinline__ Item get_item(const ItemTable& tb, int idx) {
  Item it;
  it.rec = tb.rec[idx];
  it.ntok = tb.ntok[idx];
  it.shared = tb.pair0[idx] < 0;
  it.pair0 = it.shared ? 0 : tb.pair0[idx];
  return it;
}

// token index and h row of the q-th token of an item
__device__ __forceinline__ void item_token(const FfnParams& p, const Plan* pl, const Item& it, int q, int* t,
                                           int* hrow, int* j) {
  if (it.shared) {
    *t = q;
    *hrow = p.h_shared_row0 + q;
    *j = p.k;
  } else {
    const int pair = pl->perm[it.pair0 + q];
    *t = pair / p.k;
    *hrow = pair;
    *j = pair % p.k;
  }
}

template <int WD, int MAXT>
__global__ void __launch_bounds__(kFfnThreads, 1) ffn_decode_kernel(FfnParams p) {
  using XT = typename std::conditional<WD == 0, float, __nv_bfloat16>::type;
  using F = Fmt<WD>;
  constexpr int EPC = F::kElemsPerChunk;
  constexpr int UNR = F::kUnroll;
  extern __shared__ __align__(16) uint8_t smem[];
  const Plan* pl = p.plan;
  if (pl->err != MOE_OK) return;
  const int H = p.H, I = p.I, B = p.B, k = p.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_items = pl->n_items[p.which];
  const bool combine = (p.which == 1) || (pl->n_items[1] == 0);

  __shared__ ItemTable tb;
  for (int i = threadIdx.x; i < n_items; i += blockDim.x) {
    const Item it = make_item(p, pl, i);
    tb.rec[i] = it.rec;
    tb.ntok[i] = it.ntok;
    tb.pair0[i] = it.shared ? -1 : it.pair0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < n_items; ++i) { tb.hbase[i] = run; run += tb.ntok[i]; }
    tb.hbase[n_items] = run;
  }
  XT* xs = reinterpret_cast<XT*>(smem);
  float* hs = reinterpret_cast<float*>(smem + (((size_t)B * H * sizeof(XT) + 15) & ~(size_t)15));
  float* os = hs + p.smem_h_floats;

  // phase-2 row range of this CTA; prefetch its W_down rows into L2
  const int n0 = (int)((int64_t)blockIdx.x * H / gridDim.x);
  const int n1 = (int)((int64_t)(blockIdx.x + 1) * H / gridDim.x);
  const int nrows = n1 - n0;
  if (threadIdx.x < n_items && nrows > 0) {
    const Item it = get_item(tb, threadIdx.x);
    const RecView v = rec_view<WD>(it.rec, H, I);
    const int64_t rb = F::row_bytes(I);
    prefetch_l2(v.down + (int64_t)n0 * rb, (uint32_t)(nrows * rb));
    if (WD == 2) prefetch_l2(v.down_sc + (int64_t)n0 * (I / 16), (uint32_t)(nrows * (I / 16)));
  }

  // activations -> shared memory
  {
    const int nvec = (int)((size_t)B * H * sizeof(XT) / 16);
    const uint4* src = reinterpret_cast<const uint4*>(p.x);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    for (int i = threadIdx.x; i < nvec; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();

  // ---- phase 1: gate/up rows --------------------------------------------------
  {
    const int64_t total = (int64_t)n_items * I;
    const int64_t t0 = (int64_t)blockIdx.x * total / gridDim.x;
    const int64_t t1 = (int64_t)(blockIdx.x + 1) * total / gridDim.x;
    const int nchunks = H / EPC;
    const int64_t rb = F::row_bytes(H);
    for (int64_t task = t0 + warp; task < t1; task += kFfnWarps) {
      const int item = (int)(task / I), i = (int)(task % I);
      const Item it = get_item(tb, item);
      const RecView v = rec_view<WD>(it.rec, H, I);
      const uint8_t* grow = v.gate + (int64_t)i * rb;
      const uint8_t* urow = v.up + (int64_t)i * rb;
      const uint8_t* gsc = (WD == 2) ? v.gate_sc + (int64_t)i * (H / 16) : nullptr;
      const uint8_t* usc = (WD == 2) ? v.up_sc + (int64_t)i * (H / 16) : nullptr;
      int tok[MAXT];
#pragma unroll
      for (int q = 0; q < MAXT; ++q) {
        int t = 0, hr, j;
        if (q < it.ntok) item_token(p, pl, it, q, &t, &hr, &j);
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
            wg[u] = ld_stream(grow + (int64_t)c * 16);
            wu[u] = ld_stream(urow + (int64_t)c * 16);
            if (WD == 2) {
              sg[u] = ld_stream_u16(gsc + 2 * c);
              su[u] = ld_stream_u16(usc + 2 * c);
            } else {
              sg[u] = su[u] = 0;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int c = c0 + lane + 32 * u;
          if (c < nchunks) {
#pragma unroll
            for (int q = 0; q < MAXT; ++q) {
              if (q < it.ntok) {
                const XT* xr = xs + (size_t)tok[q] * H + (size_t)c * EPC;
                ag[q] += chunk_dot<WD, XT>(wg[u], sg[u], xr);
                au[q] += chunk_dot<WD, XT>(wu[u], su[u], xr);
              }
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < MAXT; ++q) {
        if (q < it.ntok) {
          const float g = warp_sum(ag[q]);
          const float u = warp_sum(au[q]);
          if (lane == 0) {
            int t, hr, j;
            item_token(p, pl, it, q, &t, &hr, &j);
            const float silu = g / (1.0f + expf(-g));
            p.h[(int64_t)hr * I + i] = silu * u;
          }
        }
      }
    }
  }

  if (!grid_barrier(p.bar, p.bar + 1, p.err)) return;

  // ---- phase 2: down rows [n0, n1) for every item, in h-groups ---------------
  const int ostride = B * (k + 1);
  for (int i = threadIdx.x; i < nrows * ostride; i += blockDim.x) os[i] = 0.f;
  {
    const int nchunks = I / EPC;
    const int64_t rb = F::row_bytes(I);
    int g0 = 0;
    while (g0 < n_items) {
      // gather the largest run of items whose h rows fit in shared memory
      int g1 = g0, used = 0;
      while (g1 < n_items) {
        const int nt = tb.ntok[g1];
        if (used + nt * I > p.smem_h_floats && g1 > g0) break;
        used += nt * I;
        ++g1;
      }
      __syncthreads();
      {  // load h rows of items g0..g1-1 (item-major, token-minor)
        int base = 0;
        for (int g = g0; g < g1; ++g) {
          const Item it = get_item(tb, g);
          for (int q = 0; q < it.ntok; ++q) {
            int t, hr, j;
            item_token(p, pl, it, q, &t, &hr, &j);
            const float4* src = reinterpret_cast<const float4*>(p.h + (int64_t)hr * I);
            float4* dst = reinterpret_cast<float4*>(hs + (int64_t)(base + q) * I);
            for (int e = threadIdx.x; e < I / 4; e += blockDim.x) dst[e] = __ldcg(src + e);
          }
          base += it.ntok;
        }
      }
      __syncthreads();
      // units: (item, row) pairs; the h base of an item is the running token count
      const int nunits = (g1 - g0) * nrows;
      constexpr int R2 = 4;     // rows in flight per warp
      constexpr int UNR2 = 2;   // 16-byte chunks per lane held in registers
      for (int u0 = warp * R2; u0 < nunits; u0 += kFfnWarps * R2) {
        uint4 w[R2][UNR2];
        unsigned short sc[R2][UNR2];
#pragma unroll
        for (int r = 0; r < R2; ++r) {
          const int unit = u0 + r;
          if (unit < nunits) {
            const int gi = g0 + unit / nrows;
            const int row = n0 + unit % nrows;
            const RecView v = rec_view<WD>(tb.rec[gi], H, I);
            const uint8_t* drow = v.down + (int64_t)row * rb;
            const uint8_t* dsc = (WD == 2) ? v.down_sc + (int64_t)row * (I / 16) : nullptr;
#pragma unroll
            for (int u = 0; u < UNR2; ++u) {
              const int c = lane + 32 * u;
              if (c < nchunks) {
                w[r][u] = ld_stream(drow + (int64_t)c * 16);
                sc[r][u] = (WD == 2) ? ld_stream_u16(dsc + 2 * c) : (unsigned short)0;
              }
            }
          }
        }
#pragma unroll
        for (int r = 0; r < R2; ++r) {
          const int unit = u0 + r;
          if (unit >= nunits) continue;
          const int gi = g0 + unit / nrows;
          const int row = n0 + unit % nrows;
          const Item it = get_item(tb, gi);
          const int hbase = tb.hbase[gi] - tb.hbase[g0];
#pragma unroll
          for (int q = 0; q < MAXT; ++q) {
            if (q < it.ntok) {
              const float* hrow = hs + (int64_t)(hbase + q) * I;
              float acc = 0.f;
#pragma unroll
              for (int u = 0; u < UNR2; ++u) {
                const int c = lane + 32 * u;
                if (c < nchunks) acc += chunk_dot<WD, float>(w[r][u], sc[r][u], hrow + (int64_t)c * EPC);
              }
              // chunks beyond 32*UNR2 (large I)
              for (int c = lane + 32 * UNR2; c < nchunks; c += 32) {
                const RecView v = rec_view<WD>(it.rec, H, I);
                const uint8_t* drow = v.down + (int64_t)row * rb;
                uint4 ww = ld_stream(drow + (int64_t)c * 16);
                unsigned short ss = (WD == 2) ? ld_stream_u16(v.down_sc + (int64_t)row * (I / 16) + 2 * c) : 0;
                acc += chunk_dot<WD, float>(ww, ss, hrow + (int64_t)c * EPC);
              }
              acc = warp_sum(acc);
              if (lane == 0) {
                int t, hr, j;
                item_token(p, pl, it, q, &t, &hr, &j);
                os[(row - n0) * ostride + t * (k + 1) + j] = acc;
              }
            }
          }
        }
      }
      g0 = g1;
    }
  }
  __syncthreads();

  // ---- combine or hand the partials to the fill launch -------------------------
  const int npairs = B * k;
  for (int e = threadIdx.x; e < nrows * B; e += blockDim.x) {
    const int nl = e / B, t = e % B, n = n0 + nl;
    const float* o = os + nl * ostride + t * (k + 1);
    if (combine) {
      float acc = 0.f;
      for (int j = 0; j < k; ++j) {
        const int pair = t * k + j;
        const int r = pl->pair_rank[pair];
        const bool mine = (p.which == 0) ? (pl->u_fill[r] == 0) : (pl->u_fill[r] != 0);
        const float ov = mine ? o[j] : __ldcg(p.partial + ((int64_t)t * (k + 1) + j) * H + n);
        acc = fmaf(pl->pair_w[pair], ov, acc);
      }
      if (p.has_shared) acc += (p.which == 0) ? o[k] : __ldcg(p.partial + ((int64_t)t * (k + 1) + k) * H + n);
      if constexpr (WD == 0)
        reinterpret_cast<float*>(p.y)[(int64_t)t * H + n] = acc;
      else
        reinterpret_cast<__nv_bfloat16*>(p.y)[(int64_t)t * H + n] = __float2bfloat16_rn(acc);
    } else {
      for (int j = 0; j < k; ++j) {
        const int r = pl->pair_rank[t * k + j];
        if (pl->u_fill[r] == 0) p.partial[((int64_t)t * (k + 1) + j) * H + n] = o[j];
      }
      if (p.has_shared) p.partial[((int64_t)t * (k + 1) + k) * H + n] = o[k];
    }
  }
  (void)npairs;
}

// ---- launch -------------------------------------------------------------------
size_t ffn_smem_bytes(int wdtype, int B, int H, int k, int smem_h_floats, int rows_per_cta_max) {
  const size_t xbytes = (((size_t)B * H * (wdtype == MOE_FP32 ? 4 : 2)) + 15) & ~(size_t)15;
  return xbytes + (size_t)smem_h_floats * 4 + (size_t)rows_per_cta_max * B * (k + 1) * 4;
}

template <int WD, int MAXT>
static cudaError_t launch_t(const FfnParams& p, int grid, size_t smem, cudaStream_t s) {
  auto fn = ffn_decode_kernel<WD, MAXT>;
  static size_t smem_set = 0;  // largest dynamic shared memory already allowed for this instantiation
  if (smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    smem_set = smem;
  }
  void* args[] = {const_cast<FfnParams*>(&p)};
  return cudaLaunchCooperativeKernel((const void*)fn, dim3(grid), dim3(kFfnThreads), args, smem, s);
}

template <int WD>
static cudaError_t launch_w(const FfnParams& p, int grid, size_t smem, cudaStream_t s) {
  if (p.B <= 1) return launch_t<WD, 1>(p, grid, smem, s);
  if (p.B <= 2) return launch_t<WD, 2>(p, grid, smem, s);
  if (p.B <= 4) return launch_t<WD, 4>(p, grid, smem, s);
  if (p.B <= 8) return launch_t<WD, 8>(p, grid, smem, s);
  return launch_t<WD, 16>(p, grid, smem, s);
}

cudaError_t launch_ffn(int wdtype, const FfnParams& p, int grid, size_t smem, cudaStream_t s) {
  switch (wdtype) {
    case MOE_FP32: return launch_w<0>(p, grid, smem, s);
    case MOE_BF16: return launch_w<1>(p, grid, smem, s);
    case MOE_FP4: return launch_w<2>(p, grid, smem, s);
  }
  return cudaErrorInvalidValue;
}

// Largest cooperative grid for this format (one CTA per SM at most).
int ffn_max_grid(int wdtype, size_t smem) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const void* fn = wdtype == MOE_FP32 ? (const void*)ffn_decode_kernel<0, 16>
                   : wdtype == MOE_BF16 ? (const void*)ffn_decode_kernel<1, 16>
                                        : (const void*)ffn_decode_kernel<2, 16>;
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kFfnThreads, smem) != cudaSuccess) return 0;
  return sms * (per_sm > 1 ? 1 : per_sm);
}

}  // namespace moe
