// Safe-point compaction of the slot pool ("elastic memory management" in the
// FreeToken write-up: the GPU expert cache is rebuilt to a new budget without
// reloading the host pool).  The host computes which resident experts move
// from slots >= C' into vacant slots < C'; this kernel copies their records.
#include "params.cuh"

namespace moe {

// moves: [n_moves][2] = (src slot, dst slot); src and dst ranges never overlap.
__global__ void slot_move_kernel(uint8_t* __restrict__ base, int64_t S, const int32_t* __restrict__ moves,
                                 int n_moves) {
  const int64_t vec_per_rec = S / 16;
  const int64_t total = vec_per_rec * n_moves;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / vec_per_rec, v = i % vec_per_rec;
    const uint4* src = reinterpret_cast<const uint4*>(base + (int64_t)moves[2 * m] * S) + v;
    uint4* dst = reinterpret_cast<uint4*>(base + (int64_t)moves[2 * m + 1] * S) + v;
    *dst = __ldcs(src);
  }
}

cudaError_t launch_slot_moves(uint8_t* base, int64_t S, const int32_t* moves, int n_moves, cudaStream_t s) {
  if (n_moves <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  slot_move_kernel<<<sms * 4, 512, 0, s>>>(base, S, moves, n_moves);
  return cudaGetLastError();
}

}  // namespace moe
