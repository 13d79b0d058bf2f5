// Prefill-size routed-MoE layer: routing of T tokens, stable grouping of the
// (token, rank) pairs by expert, gather of the activations per expert, the two
// grouped GEMMs on tcgen05/TMEM reading the layer buffer's bf16 weights or its
// FP4 codes and scales directly (gate/up with the SwiGLU epilogue, then down)
// and the weighted combine.
//
// FreeToken write-up, "전층 이중 버퍼링": prefill activates almost every expert
// of a layer, so the layer's full expert set is streamed into one of two
// full-layer buffers carved from the slot pool while the previous layer
// computes on the other; the host-side orchestration is in cache.cu.
#include "expert_math.cuh"
#include "params.cuh"
#include "tc_gemm.cuh"
#include "tc_nvf4.cuh"

namespace moe {
namespace pf {

// ---- 1. routing: one warp per token, same rule as the decode control step ----
__global__ void route_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
                             float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const float* lg = logits + (size_t)t * E;
  float v[kMaxE / 32];
#pragma unroll
  for (int q = 0; q < kMaxE / 32; ++q) {
    const int e = lane + 32 * q;
    float x = -INFINITY;
    if (e < E) {
      x = lg[e];
      if (x != x) x = -INFINITY;
    }
    v[q] = x;
  }
  unsigned taken = 0u;
  float m0 = 0.f, sum = 0.f, mine = 0.f;
  int my_id = 0;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int q = 0; q < kMaxE / 32; ++q) {
      const int e = lane + 32 * q;
      if (e < E && !(taken & (1u << q)) && (v[q] > bv || (v[q] == bv && e < bi))) { bv = v[q]; bi = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (r == 0) m0 = bv;
    const float ex = bv == m0 ? 1.f : expf(bv - m0);  // equal to the largest (also +-inf): exp(0)
    sum += ex;
    if (lane == r) { my_id = bi; mine = ex; }
  }
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = mine / sum;
  }
}

// Group of flat pair p: routed pairs t*k+j -> their expert; with a shared
// expert, pairs T*k + t form group E.
__device__ __forceinline__ int pair_group(const int32_t* ids, int Tk, int E, int p) { return p < Tk ? ids[p] : E; }

// ---- 2. stable counting sort of the pairs by group ---------------------------------
// chunk c = pairs [c*1024, (c+1)*1024): per-chunk histogram
__global__ void __launch_bounds__(1024) group_count_kernel(const int32_t* ids, int Tk, int n_pairs, int E, int G,
                                                           int32_t* cnt) {
  extern __shared__ int32_t h[];
  for (int g = threadIdx.x; g < G; g += blockDim.x) h[g] = 0;
  __syncthreads();
  const int p = blockIdx.x * 1024 + threadIdx.x;
  if (p < n_pairs) atomicAdd(&h[pair_group(ids, Tk, E, p)], 1);
  __syncthreads();
  for (int g = threadIdx.x; g < G; g += blockDim.x) cnt[(size_t)blockIdx.x * G + g] = h[g];
}

// one block: base[c][g] = start of chunk c's pairs of group g; offsets[g] = group starts
__global__ void __launch_bounds__(1024) group_scan_kernel(const int32_t* cnt, int n_chunks, int G, int32_t* base,
                                                          int32_t* offsets) {
  __shared__ int scratch[33];
  __shared__ int s_run;
  if (threadIdx.x == 0) s_run = 0;
  __syncthreads();
  const int total = G * n_chunks;  // group-major, chunk-minor
  for (int i0 = 0; i0 < total; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    const int g = i / n_chunks, c = i % n_chunks;
    const int v = i < total ? cnt[(size_t)c * G + g] : 0;
    int tot;
    const int ex = block_excl_scan(v, scratch, &tot);
    const int run = s_run;
    if (i < total) {
      base[(size_t)c * G + g] = run + ex;
      if (c == 0) offsets[g] = run + ex;
    }
    __syncthreads();
    if (threadIdx.x == 0) s_run = run + tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[G] = s_run;
}

// place the chunk's pairs in order: warps one after the other, ranks within a
// warp from the peer mask of equal groups
__global__ void __launch_bounds__(1024) group_place_kernel(const int32_t* ids, int Tk, int n_pairs, int E, int G,
                                                           const int32_t* base, int32_t* pos, int32_t* perm,
                                                           unsigned* dbg) {
  extern __shared__ int32_t run[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int g = threadIdx.x; g < G; g += blockDim.x) run[g] = base[(size_t)blockIdx.x * G + g];
  __syncthreads();
  const int p = blockIdx.x * 1024 + threadIdx.x;
  const bool valid = p < n_pairs;
  const int g = valid ? pair_group(ids, Tk, E, p) : -1 - lane;  // invalid lanes never match
  const unsigned peers = __match_any_sync(0xFFFFFFFFu, g);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  const bool leader = rank == 0;
  for (int w = 0; w < 32; ++w) {
    if (warp == w && valid) {
      const int at = run[g] + rank;
      pos[p] = at;
      if (in_bounds(dbg, at >= 0 && at < n_pairs, 101)) perm[at] = p;
      __syncwarp(peers);
      if (leader) run[g] += __popc(peers);
    }
    __syncthreads();
  }
}

// ---- 3. gather of the activations in group order -------------------------------------
// TO_F16: rows are written as f16 (the FP4 GEMMs run on f16 operands); bf16 ->
// f16 is exact for 2^-14 <= |x| <= 65504 and 0, smaller magnitudes round to
// the f16 subnormal grid (absolute error <= 2^-25).
template <bool TO_F16>
__global__ void gather_kernel(const __nv_bfloat16* __restrict__ x, int Tk, int k, int H, int n_pairs,
                              const int32_t* __restrict__ perm, __nv_bfloat16* __restrict__ xp, unsigned* dbg) {
  const int per = H / 8;  // 16-byte vectors per row
  const int64_t total = (int64_t)n_pairs * per;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int row = (int)(i / per), v = (int)(i % per);
    const int p = perm[row];
    const int t = p < Tk ? p / k : p - Tk;
    if (!in_bounds(dbg, p >= 0 && p < n_pairs && t < (Tk / k), 102)) continue;
    uint4 val = reinterpret_cast<const uint4*>(x + (int64_t)t * H)[v];
    if constexpr (TO_F16) {
      uint32_t* w = reinterpret_cast<uint32_t*>(&val);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 h2 = __floats2half2_rn(bf16lo(w[i]), bf16hi(w[i]));
        w[i] = *reinterpret_cast<const uint32_t*>(&h2);
      }
    }
    reinterpret_cast<uint4*>(xp + (int64_t)row * H)[v] = val;
  }
}

// FP4 x FP4 path: the gathered rows quantised to e2m1 codes [n_pairs][H/2]
// and e4m3 block scales [n_pairs][H/16]; one thread per 16-element block.
__global__ void gather_quant_kernel(const __nv_bfloat16* __restrict__ x, int Tk, int k, int H, int n_pairs,
                                    const int32_t* __restrict__ perm, uint8_t* __restrict__ codes,
                                    uint8_t* __restrict__ scales, unsigned* dbg) {
  const int per = H / 16;
  const int64_t total = (int64_t)n_pairs * per;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int row = (int)(i / per), b = (int)(i % per);
    const int p = perm[row];
    const int t = p < Tk ? p / k : p - Tk;
    if (!in_bounds(dbg, p >= 0 && p < n_pairs && t < (Tk / k), 103)) continue;
    const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)t * H + (int64_t)b * 16);
    const uint4 v0 = src[0], v1 = src[1];
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float f[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      f[2 * j] = bf16lo(w[j]);
      f[2 * j + 1] = bf16hi(w[j]);
    }
    uint32_t c01[2];
    scales[(int64_t)row * per + b] = (uint8_t)quant16(f, c01);
    *reinterpret_cast<uint2*>(codes + (int64_t)row * (H / 2) + (int64_t)b * 8) = make_uint2(c01[0], c01[1]);
  }
}

// Rows of bf16 or float32 values -> codes and scales (the library's quantiser).
template <typename T>
__global__ void quantize_kernel(const T* __restrict__ x, int64_t rows, int K, uint8_t* __restrict__ codes,
                                uint8_t* __restrict__ scales) {
  const int per = K / 16;
  const int64_t total = rows * per;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / per;
    const int b = (int)(i % per);
    float f[16];
    const T* src = x + row * K + (int64_t)b * 16;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if constexpr (std::is_same<T, float>::value) f[j] = src[j];
      else f[j] = __bfloat162float(src[j]);
    }
    uint32_t c01[2];
    scales[row * per + b] = (uint8_t)quant16(f, c01);
    *reinterpret_cast<uint2*>(codes + row * (K / 2) + (int64_t)b * 8) = make_uint2(c01[0], c01[1]);
  }
}

// ---- 4/5. grouped GEMMs ----------------------------------------------------------------------
struct BRowGateUp {
  int I;
  __device__ int operator()(int nb, int half) const { return half ? I + nb * 128 : nb * 128; }
};
struct BRowDown {
  __device__ int operator()(int nb, int half) const { return nb * 256 + half * 128; }
};

__global__ void __launch_bounds__(tc::kThreads, 1)
    gemm_gate_up_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                        const int32_t* offsets, const int32_t* slot_of, int n_groups, int H, int I, __nv_bfloat16* hp,
                        int* err) {
  tc::grouped_gemm_cta(&map_a, &map_b, offsets, slot_of, n_groups, I / 128, H, tc::EpiSwiGLU<>{hp, I}, BRowGateUp{I},
                       err);
}

__global__ void __launch_bounds__(tc::kThreads, 1)
    gemm_down_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                     const int32_t* offsets, const int32_t* slot_of, int n_groups, int H, int I, float* op, int* err) {
  tc::grouped_gemm_cta(&map_a, &map_b, offsets, slot_of, n_groups, H / 256, I, tc::EpiStoreF32{op, H}, BRowDown{},
                       err);
}

// FP4 weights read directly (codes + scales maps over the layer buffer)
__global__ void __launch_bounds__(tc::fp4::kThreads, 1)
    gemm_gate_up_fp4_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_c,
                            const __grid_constant__ CUtensorMap map_s, const int32_t* offsets,
                            const int32_t* slot_of, int n_groups, int H, int I, __half* hp, int* err) {
  tc::grouped_gemm_fp4_persistent(&map_a, &map_c, &map_s, offsets, slot_of, n_groups, I / 128, H,
                                  tc::EpiSwiGLU<__half>{hp, I}, BRowGateUp{I}, err);
}

__global__ void __launch_bounds__(tc::fp4::kThreads, 1)
    gemm_down_fp4_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_c,
                         const __grid_constant__ CUtensorMap map_s, const int32_t* offsets, const int32_t* slot_of,
                         int n_groups, int H, int I, float* op, int* err) {
  tc::grouped_gemm_fp4_persistent(&map_a, &map_c, &map_s, offsets, slot_of, n_groups, H / 256, I,
                                  tc::EpiStoreF32{op, H}, BRowDown{}, err);
}

// FP4 x FP4 with block scales (activations quantised): 128-column blocks,
// gate rows nb*64.. next to up rows I + nb*64..; down rows nb*128 + half*64..
struct BRowGateUp64 {
  int I;
  __device__ int operator()(int nb, int half) const { return half ? I + nb * 64 : nb * 64; }
};
struct BRowDown64 {
  __device__ int operator()(int nb, int half) const { return nb * 128 + half * 64; }
};

__global__ void __launch_bounds__(tc::nvf4::kThreads, 1)
    gemm_gate_up_nvf4_kernel(const __grid_constant__ CUtensorMap map_ac, const __grid_constant__ CUtensorMap map_as,
                             const __grid_constant__ CUtensorMap map_bc, const __grid_constant__ CUtensorMap map_bs,
                             const int32_t* offsets, const int32_t* slot_of, int n_groups, int H, int I,
                             uint8_t* hc, uint8_t* hs, int* err) {
  tc::grouped_gemm_nvf4(&map_ac, &map_as, &map_bc, &map_bs, offsets, slot_of, n_groups, I / 64, H,
                        tc::EpiSwiGLUQuant{hc, hs, I}, BRowGateUp64{I}, err);
}

__global__ void __launch_bounds__(tc::nvf4::kThreads, 1)
    gemm_down_nvf4_kernel(const __grid_constant__ CUtensorMap map_ac, const __grid_constant__ CUtensorMap map_as,
                          const __grid_constant__ CUtensorMap map_bc, const __grid_constant__ CUtensorMap map_bs,
                          const int32_t* offsets, const int32_t* slot_of, int n_groups, int H, int I, float* op,
                          int* err) {
  tc::grouped_gemm_nvf4(&map_ac, &map_as, &map_bc, &map_bs, offsets, slot_of, n_groups, H / 128, I,
                        tc::EpiStoreF32N128{op, H}, BRowDown64{}, err);
}

// ---- 6. combine ------------------------------------------------------------------------------
__global__ void combine_kernel(const float* __restrict__ op, const int32_t* __restrict__ pos, const float* __restrict__ w,
                               int T, int k, int H, int has_shared, __nv_bfloat16* __restrict__ y, unsigned* dbg) {
  const int per = H / 4;
  const int64_t total = (int64_t)T * per;
  const int Tk = T * k;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / per), v = (int)(i % per);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const int n_pairs = Tk + (has_shared ? T : 0);
    for (int j = 0; j < k; ++j) {
      const float wj = w[(int64_t)t * k + j];
      const int at = pos[(int64_t)t * k + j];
      if (!in_bounds(dbg, at >= 0 && at < n_pairs, 104)) continue;
      const float4 o = reinterpret_cast<const float4*>(op + (int64_t)at * H)[v];
      acc.x = fmaf(wj, o.x, acc.x);
      acc.y = fmaf(wj, o.y, acc.y);
      acc.z = fmaf(wj, o.z, acc.z);
      acc.w = fmaf(wj, o.w, acc.w);
    }
    if (has_shared) {
      const float4 o = reinterpret_cast<const float4*>(op + (int64_t)pos[Tk + t] * H)[v];
      acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
    }
    __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y), b = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 out = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    reinterpret_cast<uint2*>(y + (int64_t)t * H)[v] = out;
  }
}

}  // namespace pf

// ---- launchers ----------------------------------------------------------------------------
static int g_sms = 0;
static int sms() {
  if (!g_sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
  }
  return g_sms;
}

cudaError_t prefill_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s) {
  const int warps_per_block = 8;
  pf::route_kernel<<<(T + warps_per_block - 1) / warps_per_block, 32 * warps_per_block, 0, s>>>(logits, T, E, k, ids, w);
  return cudaGetLastError();
}

cudaError_t prefill_group(const int32_t* ids, int T, int k, int E, int has_shared, int32_t* cnt, int32_t* base,
                          int32_t* offsets, int32_t* pos, int32_t* perm, cudaStream_t s) {
  const int Tk = T * k, n_pairs = Tk + (has_shared ? T : 0), G = E + (has_shared ? 1 : 0);
  const int n_chunks = (n_pairs + 1023) / 1024;
  pf::group_count_kernel<<<n_chunks, 1024, G * sizeof(int32_t), s>>>(ids, Tk, n_pairs, E, G, cnt);
  pf::group_scan_kernel<<<1, 1024, 0, s>>>(cnt, n_chunks, G, base, offsets);
  pf::group_place_kernel<<<n_chunks, 1024, G * sizeof(int32_t), s>>>(ids, Tk, n_pairs, E, G, base, pos, perm,
                                                                       debug_counters());
  return cudaGetLastError();
}

cudaError_t prefill_gather(const void* x, int T, int k, int H, int n_pairs, const int32_t* perm, void* xp,
                           int to_f16, cudaStream_t s) {
  if (to_f16)
    pf::gather_kernel<true><<<sms() * 8, 256, 0, s>>>((const __nv_bfloat16*)x, T * k, k, H, n_pairs, perm,
                                                      (__nv_bfloat16*)xp, debug_counters());
  else
    pf::gather_kernel<false><<<sms() * 8, 256, 0, s>>>((const __nv_bfloat16*)x, T * k, k, H, n_pairs, perm,
                                                       (__nv_bfloat16*)xp, debug_counters());
  return cudaGetLastError();
}

static bool g_gemm_attr = false;
static cudaError_t gemm_attr() {
  if (g_gemm_attr) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(pf::gemm_gate_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tc::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pf::gemm_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc::kSmemBytes);
  g_gemm_attr = e == cudaSuccess;
  return e;
}

// grid: enough CTAs for every tile of n_rows rows over n_groups groups
static int gemm_grid(int n_rows, int n_groups, int nblocks_n) { return (n_rows / tc::kBM + n_groups) * nblocks_n; }
// persistent grid: one CTA per SM, at most one per possible tile
static int persistent_grid(int n_rows, int n_groups, int nblocks_n) {
  const int most = gemm_grid(n_rows, n_groups, nblocks_n);
  return most < sms() ? most : sms();
}

cudaError_t prefill_gemm_gate_up(const CUtensorMap& a, const CUtensorMap& b, const int32_t* offsets,
                                 const int32_t* slot_of, int n_groups, int n_rows, int H, int I, void* hp, int* err,
                                 cudaStream_t s) {
  if (cudaError_t e = gemm_attr()) return e;
  pf::gemm_gate_up_kernel<<<gemm_grid(n_rows, n_groups, I / 128), tc::kThreads, tc::kSmemBytes, s>>>(
      a, b, offsets, slot_of, n_groups, H, I, (__nv_bfloat16*)hp, err);
  return cudaGetLastError();
}

cudaError_t prefill_gemm_down(const CUtensorMap& a, const CUtensorMap& b, const int32_t* offsets,
                              const int32_t* slot_of, int n_groups, int n_rows, int H, int I, float* op, int* err,
                              cudaStream_t s) {
  if (cudaError_t e = gemm_attr()) return e;
  pf::gemm_down_kernel<<<gemm_grid(n_rows, n_groups, H / 256), tc::kThreads, tc::kSmemBytes, s>>>(
      a, b, offsets, slot_of, n_groups, H, I, op, err);
  return cudaGetLastError();
}

static bool g_gemm_fp4_attr = false;
static cudaError_t gemm_fp4_attr() {
  if (g_gemm_fp4_attr) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(pf::gemm_gate_up_fp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tc::fp4::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pf::gemm_down_fp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tc::fp4::kSmemBytes);
  g_gemm_fp4_attr = e == cudaSuccess;
  return e;
}

cudaError_t prefill_gemm_gate_up_fp4(const CUtensorMap& a, const CUtensorMap& codes, const CUtensorMap& scales,
                                     const int32_t* offsets, const int32_t* slot_of, int n_groups, int n_rows, int H,
                                     int I, void* hp, int* err, cudaStream_t s) {
  if (cudaError_t e = gemm_fp4_attr()) return e;
  pf::gemm_gate_up_fp4_kernel<<<persistent_grid(n_rows, n_groups, I / 128), tc::fp4::kThreads, tc::fp4::kSmemBytes,
                                s>>>(
      a, codes, scales, offsets, slot_of, n_groups, H, I, (__half*)hp, err);
  return cudaGetLastError();
}

cudaError_t prefill_gemm_down_fp4(const CUtensorMap& a, const CUtensorMap& codes, const CUtensorMap& scales,
                                  const int32_t* offsets, const int32_t* slot_of, int n_groups, int n_rows, int H,
                                  int I, float* op, int* err, cudaStream_t s) {
  if (cudaError_t e = gemm_fp4_attr()) return e;
  pf::gemm_down_fp4_kernel<<<persistent_grid(n_rows, n_groups, H / 256), tc::fp4::kThreads, tc::fp4::kSmemBytes,
                             s>>>(
      a, codes, scales, offsets, slot_of, n_groups, H, I, op, err);
  return cudaGetLastError();
}

cudaError_t prefill_gather_quant(const void* x, int T, int k, int H, int n_pairs, const int32_t* perm, uint8_t* codes,
                                 uint8_t* scales, cudaStream_t s) {
  pf::gather_quant_kernel<<<sms() * 8, 256, 0, s>>>((const __nv_bfloat16*)x, T * k, k, H, n_pairs, perm, codes, scales,
                                                    debug_counters());
  return cudaGetLastError();
}

cudaError_t quantize_rows(const void* x, int fp32, int64_t rows, int K, uint8_t* codes, uint8_t* scales,
                          cudaStream_t s) {
  if (fp32)
    pf::quantize_kernel<float><<<sms() * 8, 256, 0, s>>>((const float*)x, rows, K, codes, scales);
  else
    pf::quantize_kernel<__nv_bfloat16><<<sms() * 8, 256, 0, s>>>((const __nv_bfloat16*)x, rows, K, codes, scales);
  return cudaGetLastError();
}

static bool g_gemm_nvf4_attr = false;
static cudaError_t gemm_nvf4_attr() {
  if (g_gemm_nvf4_attr) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(pf::gemm_gate_up_nvf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tc::nvf4::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(pf::gemm_down_nvf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tc::nvf4::kSmemBytes);
  g_gemm_nvf4_attr = e == cudaSuccess;
  return e;
}

// persistent grid for 128-row x 128-column tiles
static int persistent_grid128(int n_rows, int n_groups, int nblocks_n) {
  const int most = (n_rows / 128 + n_groups) * nblocks_n;
  return most < sms() ? most : sms();
}

cudaError_t prefill_gemm_gate_up_nvf4(const CUtensorMap& ac, const CUtensorMap& as, const CUtensorMap& bc,
                                      const CUtensorMap& bs, const int32_t* offsets, const int32_t* slot_of,
                                      int n_groups, int n_rows, int H, int I, uint8_t* hc, uint8_t* hs, int* err,
                                      cudaStream_t s) {
  if (cudaError_t e = gemm_nvf4_attr()) return e;
  pf::gemm_gate_up_nvf4_kernel<<<persistent_grid128(n_rows, n_groups, I / 64), tc::nvf4::kThreads,
                                 tc::nvf4::kSmemBytes, s>>>(ac, as, bc, bs, offsets, slot_of, n_groups, H, I, hc, hs,
                                                            err);
  return cudaGetLastError();
}

cudaError_t prefill_gemm_down_nvf4(const CUtensorMap& ac, const CUtensorMap& as, const CUtensorMap& bc,
                                   const CUtensorMap& bs, const int32_t* offsets, const int32_t* slot_of, int n_groups,
                                   int n_rows, int H, int I, float* op, int* err, cudaStream_t s) {
  if (cudaError_t e = gemm_nvf4_attr()) return e;
  pf::gemm_down_nvf4_kernel<<<persistent_grid128(n_rows, n_groups, H / 128), tc::nvf4::kThreads,
                              tc::nvf4::kSmemBytes, s>>>(ac, as, bc, bs, offsets, slot_of, n_groups, H, I, op, err);
  return cudaGetLastError();
}

cudaError_t prefill_combine(const float* op, const int32_t* pos, const float* w, int T, int k, int H, int has_shared,
                            void* y, cudaStream_t s) {
  pf::combine_kernel<<<sms() * 8, 256, 0, s>>>(op, pos, w, T, k, H, has_shared, (__nv_bfloat16*)y, debug_counters());
  return cudaGetLastError();
}

}  // namespace moe
