// Decode layer kernel: host-side dispatch over its instantiations, shared-
// memory sizing and occupancy, and the router-logits kernel used when the
// caller passes W_r instead of logits.  The kernel itself is in
// layer_kernel.cuh (instantiated by layer_inst.cu).
#include "params.cuh"

namespace moe {

// ---- router logits (when the caller passes W_r instead of logits) ------------------
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

cudaError_t launch_router_logits(const void* x, bool x_bf16, const float* wr, int B, int E, int H, float* logits,
                                 cudaStream_t s) {
  const int warps = B * E, threads = 256, blocks = (warps * 32 + threads - 1) / threads;
  if (x_bf16)
    router_logits_kernel<__nv_bfloat16><<<blocks, threads, 0, s>>>((const __nv_bfloat16*)x, wr, B, E, H, logits);
  else
    router_logits_kernel<float><<<blocks, threads, 0, s>>>((const float*)x, wr, B, E, H, logits);
  return cudaGetLastError();
}

// ---- launch ------------------------------------------------------------------------------
size_t layer_smem_bytes(int wdtype, int B, int H, int k, int smem_h_floats, int rows_per_cta_max) {
  const size_t xbytes = (((size_t)B * H * (wdtype == MOE_FP32 ? 4 : 2)) + 15) & ~(size_t)15;
  return xbytes + (size_t)smem_h_floats * 4 + (size_t)rows_per_cta_max * B * (k + 1) * 4;
}

// The 15 instantiations (format x token bound 1, 2, 4, 8, 16) are compiled
// as separate objects from layer_inst.cu; each exports the launchers and the
// addresses of its layer kernel and completion kernel.
#define MOE_LAYER_DECL(F, M)                                                                                \
  cudaError_t layer_launch_##F##_##M(const LayerParams& p, int grid, size_t smem, bool pdl, cudaStream_t s); \
  cudaError_t layer_finish_##F##_##M(const LayerParams& p, int grid, size_t smem, cudaStream_t s);           \
  const void* layer_kernel_##F##_##M();                                                                     \
  const void* layer_finish_kernel_##F##_##M();
#define MOE_LAYER_DECL_F(F) \
  MOE_LAYER_DECL(F, 1) MOE_LAYER_DECL(F, 2) MOE_LAYER_DECL(F, 4) MOE_LAYER_DECL(F, 8) MOE_LAYER_DECL(F, 16)
MOE_LAYER_DECL_F(0)
MOE_LAYER_DECL_F(1)
MOE_LAYER_DECL_F(2)

using LayerLaunch = cudaError_t (*)(const LayerParams&, int, size_t, bool, cudaStream_t);
using FinishLaunch = cudaError_t (*)(const LayerParams&, int, size_t, cudaStream_t);
using LayerKernel = const void* (*)();
#define MOE_ROW(P, F) {P##F##_1, P##F##_2, P##F##_4, P##F##_8, P##F##_16}
static const LayerLaunch kLaunch[3][5] = {MOE_ROW(layer_launch_, 0), MOE_ROW(layer_launch_, 1),
                                          MOE_ROW(layer_launch_, 2)};
static const FinishLaunch kFinish[3][5] = {MOE_ROW(layer_finish_, 0), MOE_ROW(layer_finish_, 1),
                                           MOE_ROW(layer_finish_, 2)};
static const LayerKernel kKernel[3][5] = {MOE_ROW(layer_kernel_, 0), MOE_ROW(layer_kernel_, 1),
                                          MOE_ROW(layer_kernel_, 2)};
static const LayerKernel kFinishKernel[3][5] = {MOE_ROW(layer_finish_kernel_, 0), MOE_ROW(layer_finish_kernel_, 1),
                                                MOE_ROW(layer_finish_kernel_, 2)};
static_assert(MOE_FP32 == 0 && MOE_BF16 == 1 && MOE_FP4 == 2, "table rows follow the format codes");

static int maxt_index(int B) { return B <= 1 ? 0 : B <= 2 ? 1 : B <= 4 ? 2 : B <= 8 ? 3 : 4; }

cudaError_t launch_layer(int wdtype, const LayerParams& p, int grid, size_t smem, bool pdl, cudaStream_t s) {
  if (wdtype < 0 || wdtype > 2) return cudaErrorInvalidValue;
  return kLaunch[wdtype][maxt_index(p.B)](p, grid, smem, pdl, s);
}

cudaError_t launch_layer_finish(int wdtype, const LayerParams& p, int grid, size_t smem, cudaStream_t s) {
  if (wdtype < 0 || wdtype > 2) return cudaErrorInvalidValue;
  return kFinish[wdtype][maxt_index(p.B)](p, grid, smem, s);
}

// every kernel of a format: 5 layer kernels, then 5 completion kernels
static void kernels_of(int wdtype, const void** out) {
  for (int i = 0; i < 5; ++i) {
    out[i] = kKernel[wdtype][i]();
    out[5 + i] = kFinishKernel[wdtype][i]();
  }
}

size_t layer_static_smem(int wdtype) {
  const void* fns[10];
  kernels_of(wdtype, fns);
  size_t mx = 0;
  for (const void* f : fns) {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, f) == cudaSuccess) mx = a.sharedSizeBytes > mx ? a.sharedSizeBytes : mx;
  }
  return mx;
}

// Largest cooperative grid every instantiation supports with `smem` dynamic
// shared memory, capped at one CTA per SM.
int layer_max_grid(int wdtype, size_t smem) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const void* fns[10];
  kernels_of(wdtype, fns);
  int per_sm = 1;
  for (const void* f : fns) {
    int n = 0;
    if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, kThreads, smem) != cudaSuccess) return 0;
    per_sm = n < per_sm ? n : per_sm;
  }
  return sms * per_sm;
}

}  // namespace moe
