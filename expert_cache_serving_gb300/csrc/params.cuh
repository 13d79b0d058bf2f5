// Kernel parameter blocks and launch entry points shared by the host code.
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace moe {

// One decode-size layer call, executed by one cooperative launch.
struct LayerParams {
  int L, E, k, B, layer, H, I;
  int64_t C;
  const float* logits;        // [B][E]
  CacheDev st;
  Plan* plan;
  HostWork* work;             // device alias of the pinned host summary
  uint32_t seq;               // call sequence number (when seq_ctr is null)
  unsigned long long* seq_ctr;  // captured calls: every CTA adds 1 per call, seq = value / gridDim.x + 1, and
                              // work / wave_ctr are then the bases of the summary ring and of the counter pairs
  unsigned* plan_flag;        // set to seq by the control CTA once the plan is written
  unsigned* fill_flags;       // [2][kMaxU]: first/second half of fill f landed (seq, or seq|kFlagError)
  unsigned long long* bar;    // grid barrier counter (only grows; see grid_barrier)
  int* err;                   // pinned, mapped: MOE_ERR_TIMEOUT when a bounded wait for the GPU gave up
  CallState* cst;             // copy-fill completion state of this call
  float* o_part;              // [gridDim.x][o_part_floats]: saved partial sums of CTAs that handed over
  int o_part_floats;          // rows_per_cta_max * max_tokens * (k + 1)
  unsigned long long wait_gu_ns;  // how long the layer kernel waits for a fill's gate/up half
  unsigned long long wait_dn_ns;  // ... and for its W_down half, before handing the rest over
  unsigned long long* deferred;   // calls the completion kernel finished (statistics)
  double split_bp, split_bh;  // measured B_P and B_H for the fill count q* (0: pure fill, q* = misses)
  int32_t* aux_qstar;         // optional: q* of this call
  unsigned* wave_ctr;         // [kWaveCtrs] this call's counters (CTAs done with their lookups)
  unsigned* wave_next;        // [kWaveCtrs] the next call's counters, cleared by this call
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
  int stage_items;            // resident items whose W_down rows a CTA stages in shared memory
  int stage_pitch;            // bytes per staged item (rows_per_cta_max rows, then their FP4 scales)
  int stage_off;              // byte offset of the staging area in dynamic shared memory
  int32_t* oldest;            // [kMaxU] oldest slots, ascending key
  int* oldest_n;              // entries in it, -1 if invalid
  unsigned long long* tl;     // optional phase timestamps of this call [20] (profiling)
  unsigned long long* tl_next;  // the next call's timestamp row, cleared by this call
  unsigned* dbg;              // bounds-check counters of the debug build ([0] count, [1] first site)
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
// Read rate of a kernel that only reads `bytes` per launch (calib.cu).
cudaError_t read_rate(const uint8_t* bufs, size_t bytes, int n_bufs, int reps, cudaStream_t s, double* gbps);
size_t layer_static_smem(int wdtype);
// The layer kernel of one call (pdl: launched as a programmatic dependent of
// the previous launch on the stream), and its completion kernel, which runs
// after the call's copies and finishes whatever the layer kernel handed over.
cudaError_t launch_layer(int wdtype, const LayerParams& p, int grid, size_t smem, bool pdl, cudaStream_t s);
cudaError_t launch_layer_finish(int wdtype, const LayerParams& p, int grid, size_t smem, cudaStream_t s);
int layer_max_grid(int wdtype, size_t smem);
cudaError_t launch_slot_moves(uint8_t* base, int64_t S, const int32_t* moves, int n_moves, cudaStream_t s);
void set_last_error(const char* msg);  // message returned by moe_last_error() on this thread
unsigned* debug_counters();  // the process's bounds-check counters (device, [2]); null if unavailable

// prefill (prefill.cu)
cudaError_t prefill_route(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s);
cudaError_t prefill_group(const int32_t* ids, int T, int k, int E, int has_shared, int32_t* cnt, int32_t* base,
                          int32_t* offsets, int32_t* pos, int32_t* perm, cudaStream_t s);
cudaError_t prefill_gather(const void* x, int T, int k, int H, int n_pairs, const int32_t* perm, void* xp,
                           int to_f16, cudaStream_t s);
// grouped GEMMs: group g's weights are record slot_of[g] of the weight maps
cudaError_t prefill_gemm_gate_up(const CUtensorMap& a, const CUtensorMap& b, const int32_t* offsets,
                                 const int32_t* slot_of, int n_groups, int n_rows, int H, int I, void* hp, int* err,
                                 cudaStream_t s);
cudaError_t prefill_gemm_down(const CUtensorMap& a, const CUtensorMap& b, const int32_t* offsets,
                              const int32_t* slot_of, int n_groups, int n_rows, int H, int I, float* op, int* err,
                              cudaStream_t s);
cudaError_t prefill_gemm_gate_up_fp4(const CUtensorMap& a, const CUtensorMap& codes, const CUtensorMap& scales,
                                     const int32_t* offsets, const int32_t* slot_of, int n_groups, int n_rows, int H,
                                     int I, void* hp, int* err, cudaStream_t s);
cudaError_t prefill_gemm_down_fp4(const CUtensorMap& a, const CUtensorMap& codes, const CUtensorMap& scales,
                                  const int32_t* offsets, const int32_t* slot_of, int n_groups, int n_rows, int H,
                                  int I, float* op, int* err, cudaStream_t s);
// FP4 x FP4 path: gathered rows quantised to codes [n_pairs][H/2] and block
// scales [n_pairs][H/16]; block-scaled GEMMs (A and B maps of codes and scales)
cudaError_t prefill_gather_quant(const void* x, int T, int k, int H, int n_pairs, const int32_t* perm, uint8_t* codes,
                                 uint8_t* scales, cudaStream_t s);
cudaError_t prefill_gemm_gate_up_nvf4(const CUtensorMap& ac, const CUtensorMap& as, const CUtensorMap& bc,
                                      const CUtensorMap& bs, const int32_t* offsets, const int32_t* slot_of,
                                      int n_groups, int n_rows, int H, int I, uint8_t* hc, uint8_t* hs, int* err,
                                      cudaStream_t s);
cudaError_t prefill_gemm_down_nvf4(const CUtensorMap& ac, const CUtensorMap& as, const CUtensorMap& bc,
                                   const CUtensorMap& bs, const int32_t* offsets, const int32_t* slot_of, int n_groups,
                                   int n_rows, int H, int I, float* op, int* err, cudaStream_t s);
// rows of bf16 (fp32 = 0) or float32 values -> FP4 codes and block scales
cudaError_t quantize_rows(const void* x, int fp32, int64_t rows, int K, uint8_t* codes, uint8_t* scales,
                          cudaStream_t s);
cudaError_t prefill_combine(const float* op, const int32_t* pos, const float* w, int T, int k, int H, int has_shared,
                            void* y, cudaStream_t s);

}  // namespace moe
