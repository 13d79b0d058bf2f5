// Kernel parameter blocks and launch entry points shared by the host code.
#pragma once
#include "common.cuh"

namespace moe {

// One decode-size layer call, executed by one cooperative launch.
struct LayerParams {
  int L, E, k, B, layer, H, I;
  int64_t C;
  int M;                      // length of the precomputed victim order (max_tokens * k)
  const float* logits;        // [B][E]
  CacheDev st;
  Plan* plan;
  HostWork* work;             // device alias of the pinned host summary
  uint32_t seq;               // call sequence number
  unsigned* plan_flag;        // set to seq by the control CTA once the plan is written
  unsigned* fill_flags;       // [2][kMaxU]: first/second half of fill f landed (seq, or seq|kFlagError)
  unsigned long long* bar;    // grid barrier counter
  unsigned long long bar_base;
  int* err;
  int has_shared;
  int device_fill;            // 1: the kernel pulls each fill from the pool itself
  const uint8_t* pool;        // device-visible address of the pinned host pool (device_fill)
  const uint8_t* slots;       // slot s at slots + s * S
  int64_t S;
  const uint8_t* shared_rec;  // shared expert record of this layer (or null)
  const void* x;              // [B][H]
  float* h;                   // [(max_tokens*k + max_tokens)][I]
  int h_shared_row0;          // h row of shared token 0
  void* y;                    // [B][H]
  int smem_h_floats;          // capacity of the shared-memory h buffer
  int rows_per_cta_max;
  int32_t* oldest;            // [kMaxU] oldest slots, ascending key
  int* oldest_n;              // entries in it, -1 if invalid
  unsigned long long* tl;     // optional phase timestamps of this call [12] (profiling)
  // optional inspection outputs
  int32_t* aux_ids;
  float* aux_w;
  int32_t* aux_slots;
  int32_t* aux_perm;
  int32_t* aux_offsets;
  float* aux_logits;
};

cudaError_t launch_router_logits(const void* x, bool x_bf16, const float* wr, int B, int E, int H, float* logits,
                                 cudaStream_t s);
size_t layer_smem_bytes(int wdtype, int B, int H, int k, int smem_h_floats, int rows_per_cta_max);
size_t layer_static_smem(int wdtype);
cudaError_t launch_layer(int wdtype, const LayerParams& p, int grid, size_t smem, cudaStream_t s);
int layer_max_grid(int wdtype, size_t smem);
cudaError_t launch_slot_moves(uint8_t* base, int64_t S, const int32_t* moves, int n_moves, cudaStream_t s);
void set_last_error(const char* msg);  // message returned by moe_last_error() on this thread

}  // namespace moe
