// Kernel parameter blocks and launch entry points shared by the host code.
#pragma once
#include "common.cuh"

namespace moe {

struct CtrlParams {
  int L, E, k, B, layer;
  int64_t C;
  const float* logits;  // [B][E]
  CacheDev st;
  Plan* plan;
  HostWork* work;       // device alias of the pinned host summary
  uint32_t seq;
  unsigned* bar_reset;  // barrier counters of this call's FFN launches
  int n_bar_reset;
  int has_shared;
  // optional inspection outputs
  int32_t* aux_ids;
  float* aux_w;
  int32_t* aux_slots;
  int32_t* aux_perm;
  int32_t* aux_offsets;
  float* aux_logits;
};

// Undo of a call whose fills could not be issued.
struct UndoParams {
  CacheDev st;
  const HostWork* work;  // device alias
};

struct FfnParams {
  int H, I, k, B;
  int which;           // 0: resident list (+ shared), 1: fills of this call
  int has_shared;
  const uint8_t* slots;  // slot s at slots + s * S
  int64_t S;
  const uint8_t* shared_rec;  // shared expert record of this layer (or null)
  const void* x;              // [B][H]
  const Plan* plan;
  float* h;                   // [(max_tokens*k + max_tokens)][I]
  int h_shared_row0;          // h row of shared token 0
  float* partial;             // [max_tokens][k+1][H]
  void* y;                    // [B][H]
  unsigned* bar;              // count, gen
  int* err;
  int smem_h_floats;          // capacity of the shared-memory h buffer
  int rows_per_cta_max;
};

cudaError_t launch_router_logits(const void* x, bool x_bf16, const float* wr, int B, int E, int H, float* logits,
                                 cudaStream_t s);
cudaError_t launch_ctrl(const CtrlParams& p, cudaStream_t s);
cudaError_t launch_undo(const UndoParams& p, cudaStream_t s);
size_t ffn_smem_bytes(int wdtype, int B, int H, int k, int smem_h_floats, int rows_per_cta_max);
cudaError_t launch_ffn(int wdtype, const FfnParams& p, int grid, size_t smem, cudaStream_t s);
int ffn_max_grid(int wdtype, size_t smem);
cudaError_t launch_slot_moves(uint8_t* base, int64_t S, const int32_t* moves, int n_moves, cudaStream_t s);

}  // namespace moe
