// Routed MoE layer over experts that all sit in a caller-owned device bank,
// for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: their device memory is wholly owned by
// another allocator (a framework's caching allocator, or a fixed budget
// reserved up front), or they run on a path where the device-wide
// synchronisation of cudaFree/cudaMalloc is not acceptable.  This entry point
// therefore allocates nothing.  Its only scratch (the routing of the call and
// the gate/up intermediate) lives in the file-scope device array below, which
// every GPU that loads this library holds until the process exits.
//
// The computation is the one moe_layer_forward performs with every expert
// resident: top-k softmax routing (the same tie, NaN and infinity rules),
// h = SiLU(x W_gate^T) * (x W_up^T) per (token, rank), o = h W_down^T,
// y_t = sum_j w_tj o_tj (+ shared expert) in rank order.  The dot products are
// summed in a different order (one warp per row here, 8 lanes per row and a
// fixed butterfly in the cached layer kernel), so the two entry points agree
// within the layer tolerance, not bit for bit.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "expert_math.cuh"
#include "params.cuh"

namespace moe {
namespace {

// 4 MiB for the gate/up intermediate plus 16 KiB for the routing of one call.
constexpr size_t kNoAllocHBytes = size_t(4) << 20;
constexpr size_t kNoAllocRouteBytes = size_t(16) << 10;
constexpr size_t kNoAllocScratchBytes = kNoAllocHBytes + kNoAllocRouteBytes;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct ResidentParams {
  int E, k, B, H, I, has_shared;
  const uint8_t* bank;        // E records of the layer, back to back
  const uint8_t* shared_rec;  // shared expert record or null
  int64_t S;
  const void* x;              // [B][H]
  const float* logits;        // [B][E]
  void* y;                    // [B][H]
  int32_t* ids;               // scratch: [B*k]
  float* w;                   // scratch: [B*k]
  float* h;                   // scratch: [(B*k + B)][I]
};

__device__ __forceinline__ bool better_l(float a, int ia, float b, int ib) { return a > b || (a == b && ia < ib); }

// Top-k softmax of token t by one warp: ties to the lower expert, NaN as -inf.
__device__ void route_token(const ResidentParams& p, int t, int32_t* ids, float* w) {
  const int lane = threadIdx.x & 31;
  const float* lg = p.logits + (size_t)t * p.E;
  int chosen[kMaxK];
  float m0 = 0.f, sum = 0.f;
  for (int r = 0; r < p.k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int e = lane; e < p.E; e += 32) {
      bool taken = false;
      for (int q = 0; q < r; ++q) taken |= chosen[q] == e;
      if (taken) continue;
      float v = lg[e];
      if (v != v) v = -INFINITY;
      if (better_l(v, e, bv, bi)) { bv = v; bi = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (better_l(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    chosen[r] = bi;
    if (r == 0) m0 = bv;
    const float ex = bv == m0 ? 1.f : expf(bv - m0);  // equal to the largest (also +-inf): exp(0)
    sum += ex;
    if (lane == 0) { ids[t * p.k + r] = bi; w[t * p.k + r] = ex; }
  }
  __syncwarp();
  if (lane == 0)
    for (int r = 0; r < p.k; ++r) w[t * p.k + r] = w[t * p.k + r] / sum;
}

// Launch 1: routing, then one warp per (item, row i) computes h for the
// item's token; items are the B*k routed pairs and then the B shared tokens.
template <int WD>
__global__ void __launch_bounds__(512) resident_gate_up_kernel(ResidentParams p) {
  using XT = typename std::conditional<WD == MOE_FP32, float, __nv_bfloat16>::type;
  using F = Fmt<WD>;
  constexpr int EPC = F::kElemsPerChunk;
  __shared__ int32_t s_ids[kMaxPairs];
  __shared__ float s_w[kMaxPairs];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  for (int t = warp; t < p.B; t += nwarp) route_token(p, t, s_ids, s_w);
  __syncthreads();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < p.B * p.k; i += blockDim.x) { p.ids[i] = s_ids[i]; p.w[i] = s_w[i]; }
  const int n_items = p.B * p.k + (p.has_shared ? p.B : 0);
  const int64_t tasks = (int64_t)n_items * p.I;
  const int nchunks = p.H / EPC;
  const int64_t rb = F::row_bytes(p.H);
  for (int64_t task = (int64_t)blockIdx.x * nwarp + warp; task < tasks; task += (int64_t)gridDim.x * nwarp) {
    const int item = (int)(task / p.I), i = (int)(task % p.I);
    const bool sh = item >= p.B * p.k;
    const int t = sh ? item - p.B * p.k : item / p.k;
    const uint8_t* rec = sh ? p.shared_rec : p.bank + (int64_t)s_ids[item] * p.S;
    const RecView v = rec_view<WD>(rec, p.H, p.I);
    const XT* xt = reinterpret_cast<const XT*>(p.x) + (size_t)t * p.H;
    float ag = 0.f, au = 0.f;
    for (int c = lane; c < nchunks; c += 32) {
      const uint4 wg = ld_ro16(v.gate + (int64_t)i * rb + (int64_t)c * 16);
      const uint4 wu = ld_ro16(v.up + (int64_t)i * rb + (int64_t)c * 16);
      unsigned short sg = 0, su = 0;
      if (WD == MOE_FP4) {
        sg = ld_ro2(v.gate_sc + (int64_t)i * (p.H / 16) + 2 * c);
        su = ld_ro2(v.up_sc + (int64_t)i * (p.H / 16) + 2 * c);
      }
      ag += chunk_dot<WD, XT>(wg, sg, xt + (size_t)c * EPC);
      au += chunk_dot<WD, XT>(wu, su, xt + (size_t)c * EPC);
    }
    const float g = warp_sum(ag), u = warp_sum(au);
    if (lane == 0) p.h[(int64_t)item * p.I + i] = g / (1.0f + expf(-g)) * u;
  }
}

// Launch 2: one warp per (token t, output row n): o_tj[n] for every rank j
// (and the shared expert), combined in rank order.
template <int WD>
__global__ void __launch_bounds__(512) resident_down_kernel(ResidentParams p) {
  using F = Fmt<WD>;
  constexpr int EPC = F::kElemsPerChunk;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  const int nchunks = p.I / EPC;
  const int64_t rb = F::row_bytes(p.I);
  const int64_t outs = (int64_t)p.B * p.H;
  for (int64_t o = (int64_t)blockIdx.x * nwarp + warp; o < outs; o += (int64_t)gridDim.x * nwarp) {
    const int t = (int)(o / p.H), n = (int)(o % p.H);
    float acc = 0.f;
    for (int j = 0; j <= p.k; ++j) {
      if (j == p.k && !p.has_shared) break;
      const int item = j < p.k ? t * p.k + j : p.B * p.k + t;
      const uint8_t* rec = j < p.k ? p.bank + (int64_t)p.ids[t * p.k + j] * p.S : p.shared_rec;
      const RecView v = rec_view<WD>(rec, p.H, p.I);
      const float* hrow = p.h + (int64_t)item * p.I;
      float d = 0.f;
      for (int c = lane; c < nchunks; c += 32) {
        const uint4 wd = ld_ro16(v.down + (int64_t)n * rb + (int64_t)c * 16);
        const unsigned short sc = WD == MOE_FP4 ? ld_ro2(v.down_sc + (int64_t)n * (p.I / 16) + 2 * c) : 0;
        d += chunk_dot<WD, float>(wd, sc, hrow + (int64_t)c * EPC);
      }
      d = warp_sum(d);
      acc = j < p.k ? fmaf(p.w[t * p.k + j], d, acc) : acc + d;
    }
    if (lane == 0) {
      if constexpr (WD == MOE_FP32)
        reinterpret_cast<float*>(p.y)[o] = acc;
      else
        reinterpret_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(acc);
    }
  }
}

template <int WD>
cudaError_t launch_resident(const ResidentParams& p, int sms, cudaStream_t s) {
  const int64_t tasks1 = (int64_t)(p.B * p.k + (p.has_shared ? p.B : 0)) * p.I;
  const int g1 = (int)std::min<int64_t>(4 * sms, (tasks1 + 15) / 16);
  resident_gate_up_kernel<WD><<<g1, 512, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int g2 = (int)std::min<int64_t>(4 * sms, ((int64_t)p.B * p.H + 15) / 16);
  resident_down_kernel<WD><<<g2, 512, 0, s>>>(p);
  return cudaGetLastError();
}

// device address of the scratch array, looked up once per device
constexpr int kMaxDevices = 64;
unsigned char* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

moe_status noalloc_fail(moe_status st, const char* msg) {
  set_last_error(msg);
  return st;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_layer_forward_resident_noalloc(const moe_model_desc* desc, const void* bank,
                                                         const void* shared_rec, const void* x, const float* logits,
                                                         int32_t B, void* y, void* stream) {
  set_last_error("");
  if (!desc || !bank || !x || !logits || !y) return noalloc_fail(MOE_ERR_INVALID_ARG, "NULL argument");
  const int E = desc->E, k = desc->k, H = desc->H, I = desc->I, wd = desc->wdtype;
  if (E < 1 || E > kMaxE || k < 1 || k > kMaxK || k > E) return noalloc_fail(MOE_ERR_INVALID_ARG, "need 1 <= k <= E <= 1024, k <= 16");
  if (B < 1 || B > kMaxB) return noalloc_fail(MOE_ERR_INVALID_ARG, "need 1 <= B <= 16");
  if (wd != MOE_FP32 && wd != MOE_BF16 && wd != MOE_FP4) return noalloc_fail(MOE_ERR_INVALID_ARG, "unknown wdtype");
  const int m = wd == MOE_FP4 ? 256 : 64;
  if (H < m || I < m || H % m || I % m) return noalloc_fail(MOE_ERR_INVALID_ARG, "H and I must be multiples of 64 (256 for FP4)");
  if (desc->has_shared && !shared_rec) return noalloc_fail(MOE_ERR_INVALID_ARG, "has_shared set but shared_rec is NULL");
  const size_t h_bytes = (size_t)(B * k + (desc->has_shared ? B : 0)) * I * sizeof(float);
  if (h_bytes > kNoAllocHBytes)
    return noalloc_fail(MOE_ERR_INVALID_ARG,
                        "(B*k + B) * I * 4 bytes exceeds the 4 MiB scratch of the no-allocation entry point");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return noalloc_fail(MOE_ERR_CUDA, "no usable CUDA device");
  unsigned char* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void* ptr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess || !ptr) {
        cudaGetLastError();
        return noalloc_fail(MOE_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed");
      }
      g_scratch_addr[dev] = static_cast<unsigned char*>(ptr);
    }
    base = g_scratch_addr[dev];
  }
  ResidentParams p{};
  p.E = E; p.k = k; p.B = B; p.H = H; p.I = I; p.has_shared = desc->has_shared;
  p.bank = static_cast<const uint8_t*>(bank);
  p.shared_rec = static_cast<const uint8_t*>(shared_rec);
  const size_t HI = (size_t)H * I;
  p.S = wd == MOE_FP32 ? 12 * HI : wd == MOE_BF16 ? 6 * HI : 3 * HI / 2 + 3 * HI / 16;
  p.x = x;
  p.logits = logits;
  p.y = y;
  p.ids = reinterpret_cast<int32_t*>(base + kNoAllocHBytes);
  p.w = reinterpret_cast<float*>(base + kNoAllocHBytes + kMaxPairs * sizeof(int32_t));
  p.h = reinterpret_cast<float*>(base);
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = wd == MOE_FP32 ? launch_resident<MOE_FP32>(p, sms, s)
                  : wd == MOE_BF16 ? launch_resident<MOE_BF16>(p, sms, s)
                                   : launch_resident<MOE_FP4>(p, sms, s);
  if (e != cudaSuccess) return noalloc_fail(MOE_ERR_CUDA, cudaGetErrorString(e));
  return MOE_OK;
}
