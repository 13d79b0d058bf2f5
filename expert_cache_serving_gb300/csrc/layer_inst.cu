// One instantiation of the decode layer kernel and its completion kernel,
// chosen at compile time: MOE_LAYER_FMT (0 fp32, 1 bf16, 2 FP4) and
// MOE_LAYER_MAXT (token bound 1, 2, 4, 8 or 16).  The build compiles this file
// once per pair, in parallel.
#include "layer_kernel.cuh"

#if !defined(MOE_LAYER_FMT) || !defined(MOE_LAYER_MAXT)
#error "compile with -DMOE_LAYER_FMT=<0|1|2> -DMOE_LAYER_MAXT=<1|2|4|8|16>"
#endif

namespace moe {

#define MOE_LAYER_DEF2(F, M)                                                                              \
  cudaError_t layer_launch_##F##_##M(const LayerParams& p, int grid, size_t smem, bool pdl, cudaStream_t s) { \
    return launch_t<F, M>(p, grid, smem, pdl, s);                                                          \
  }                                                                                                        \
  cudaError_t layer_finish_##F##_##M(const LayerParams& p, int grid, size_t smem, cudaStream_t s) {          \
    return launch_finish_t<F, M>(p, grid, smem, s);                                                        \
  }                                                                                                        \
  const void* layer_kernel_##F##_##M() { return (const void*)layer_kernel<F, M>; }                         \
  const void* layer_finish_kernel_##F##_##M() { return (const void*)layer_finish_kernel<F, M>; }
#define MOE_LAYER_DEF(F, M) MOE_LAYER_DEF2(F, M)

MOE_LAYER_DEF(MOE_LAYER_FMT, MOE_LAYER_MAXT)

}  // namespace moe
