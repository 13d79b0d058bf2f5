// Host side of the moecache C ABI: the shared expert cache (slot memory,
// residency state), the per-call orchestration of control kernel, fills and
// expert-FFN launches, safe-point resize, statistics and tracing.
//
// FreeToken write-up, "FreeToken's design": the host expert pool is the source
// of truth and the remaining GPU memory becomes one elastic expert cache shared
// by every MoE layer; "elastic memory management": the cache is rebuilt to a
// new budget at a safe point without reloading the pool.  Slot memory is one
// reserved virtual range mapped in physical chunks, so a resize maps or
// unmaps the tail while the resident prefix stays where it is.
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <new>
#include <string>
#include <thread>
#include <mutex>
#include <vector>

#include "params.cuh"

using namespace moe;

// ------------------------------------------------------------------ errors --
static thread_local std::string g_err;

static moe_status fail(moe_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

void moe::set_last_error(const char* msg) { g_err = msg; }

#define CU_TRY(expr)                                                                      \
  do {                                                                                    \
    cudaError_t _e = (expr);                                                              \
    if (_e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(_e)); \
  } while (0)

// --------------------------------------------------------- driver entry points --
namespace {
struct Drv {
  CUresult (*memAddressReserve)(CUdeviceptr*, size_t, size_t, CUdeviceptr, unsigned long long) = nullptr;
  CUresult (*memAddressFree)(CUdeviceptr, size_t) = nullptr;
  CUresult (*memCreate)(CUmemGenericAllocationHandle*, size_t, const CUmemAllocationProp*, unsigned long long) = nullptr;
  CUresult (*memRelease)(CUmemGenericAllocationHandle) = nullptr;
  CUresult (*memMap)(CUdeviceptr, size_t, size_t, CUmemGenericAllocationHandle, unsigned long long) = nullptr;
  CUresult (*memUnmap)(CUdeviceptr, size_t) = nullptr;
  CUresult (*memSetAccess)(CUdeviceptr, size_t, const CUmemAccessDesc*, size_t) = nullptr;
  CUresult (*memGetAllocationGranularity)(size_t*, const CUmemAllocationProp*, CUmemAllocationGranularity_flags) = nullptr;
  CUresult (*streamWriteValue32)(CUstream, CUdeviceptr, cuuint32_t, unsigned int) = nullptr;
  CUresult (*tensorMapEncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill) = nullptr;
  bool ok = false;
};

template <typename F>
static bool get_entry(const char* name, F* fn) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !p)
    return false;
  *fn = reinterpret_cast<F>(p);
  return true;
}

static Drv& drv() {
  static Drv d;
  static bool init = false;
  if (!init) {
    init = true;
    d.ok = get_entry("cuMemAddressReserve", &d.memAddressReserve) && get_entry("cuMemAddressFree", &d.memAddressFree) &&
           get_entry("cuMemCreate", &d.memCreate) && get_entry("cuMemRelease", &d.memRelease) &&
           get_entry("cuMemMap", &d.memMap) && get_entry("cuMemUnmap", &d.memUnmap) &&
           get_entry("cuMemSetAccess", &d.memSetAccess) &&
           get_entry("cuMemGetAllocationGranularity", &d.memGetAllocationGranularity) &&
           get_entry("cuStreamWriteValue32", &d.streamWriteValue32) &&
           get_entry("cuTensorMapEncodeTiled", &d.tensorMapEncodeTiled);
  }
  return d;
}

// Slot memory: one virtual range for max_slots records, physically backed in
// fixed chunks from the start up to the current capacity.
struct SlotMemory {
  CUdeviceptr base = 0;
  size_t reserved = 0, chunk = 0;
  int device = 0;
  std::vector<CUmemGenericAllocationHandle> handles;

  moe_status init(int dev, size_t max_bytes) {
    Drv& d = drv();
    if (!d.ok) return fail(MOE_ERR_CUDA, "CUDA driver virtual-memory entry points unavailable");
    device = dev;
    CUmemAllocationProp prop = {};
    prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
    prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    prop.location.id = dev;
    size_t gran = 0;
    if (d.memGetAllocationGranularity(&gran, &prop, CU_MEM_ALLOC_GRANULARITY_RECOMMENDED) != CUDA_SUCCESS || !gran)
      return fail(MOE_ERR_CUDA, "cuMemGetAllocationGranularity failed");
    chunk = ((size_t(256) << 20) + gran - 1) / gran * gran;
    reserved = std::max<size_t>(chunk, (max_bytes + chunk - 1) / chunk * chunk);
    if (d.memAddressReserve(&base, reserved, 0, 0, 0) != CUDA_SUCCESS)
      return fail(MOE_ERR_OOM, "cuMemAddressReserve(%zu) failed", reserved);
    return MOE_OK;
  }

  // Make [0, bytes) backed by physical memory (mapping or unmapping chunks).
  moe_status resize(size_t bytes) {
    Drv& d = drv();
    const size_t want = (bytes + chunk - 1) / chunk;
    if (want * chunk > reserved) return fail(MOE_ERR_INVALID_ARG, "slot memory beyond the reserved range");
    while (handles.size() > want) {
      const size_t off = (handles.size() - 1) * chunk;
      d.memUnmap(base + off, chunk);
      d.memRelease(handles.back());
      handles.pop_back();
    }
    while (handles.size() < want) {
      CUmemAllocationProp prop = {};
      prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
      prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
      prop.location.id = device;
      CUmemGenericAllocationHandle h;
      if (d.memCreate(&h, chunk, &prop, 0) != CUDA_SUCCESS)
        return fail(MOE_ERR_OOM, "cuMemCreate: no device memory for %zu more slot bytes", (want - handles.size()) * chunk);
      const size_t off = handles.size() * chunk;
      if (d.memMap(base + off, chunk, 0, h, 0) != CUDA_SUCCESS) {
        d.memRelease(h);
        return fail(MOE_ERR_CUDA, "cuMemMap failed");
      }
      CUmemAccessDesc acc = {};
      acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
      acc.location.id = device;
      acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
      if (d.memSetAccess(base + off, chunk, &acc, 1) != CUDA_SUCCESS) {
        d.memUnmap(base + off, chunk);
        d.memRelease(h);
        return fail(MOE_ERR_CUDA, "cuMemSetAccess failed");
      }
      handles.push_back(h);
    }
    return MOE_OK;
  }

  void release() {
    if (!base) return;
    resize(0);
    drv().memAddressFree(base, reserved);
    base = 0;
  }
};
}  // namespace

// ------------------------------------------------------------------- cache --
struct moe_cache {
  moe_model_desc d{};
  int64_t S = 0, C = 0, C_max = 0;
  const uint8_t* host_pool = nullptr;
  const uint8_t* shared_dev = nullptr;
  int device = 0;
  SlotMemory slots;
  // device state
  int32_t* d_map = nullptr;
  int32_t* d_owner = nullptr;
  uint64_t* d_stamp = nullptr;
  uint64_t* d_g = nullptr;
  Plan* d_plan = nullptr;
  float* d_h = nullptr;
  float* d_logits = nullptr;
  unsigned long long* d_bar = nullptr;
  unsigned* d_flags = nullptr;  // [0]: plan flag, [1 ..]: fill flags [2][kMaxU]
  CallState* d_cst = nullptr;   // copy-fill completion state of the latest call
  float* d_o_part = nullptr;    // partial sums handed to the completion kernel
  int o_part_floats = 0;
  unsigned long long* d_deferred = nullptr;
  unsigned* d_wave = nullptr;   // [2][kWaveCtrs] per-call counters of the layer kernel, by call parity
  // graph mode: decode calls may be captured into CUDA graphs and replayed;
  // each layer-kernel CTA adds 1 to d_seqctr per call and takes its sequence
  // number from it, and the host reads the calls' summaries at moe_cache_sync
  bool graph = false;
  unsigned long long* d_seqctr = nullptr;
  unsigned long long deferred_base = 0;  // value of the device counter at the last statistics reset
  unsigned long long wait_gu_ns = 2000000, wait_dn_ns = 2000000;
  double split_bp = 0.0, split_bh = 0.0;  // bandwidths for q* (0: not set)
  bool pdl = true;              // launch layer kernels as programmatic dependents
  int32_t* d_oldest = nullptr;
  int* d_oldest_n = nullptr;
  int* h_err = nullptr;  // pinned, mapped: error word the kernels record timeouts in
  int* d_err = nullptr;
  int32_t* d_moves = nullptr;
  int64_t moves_cap = 0;
  HostWork* h_work = nullptr;  // ring of kRing call summaries (pinned, mapped), call seq at seq % kRing
  HostWork* d_work = nullptr;
  cudaStream_t copy = nullptr;
  cudaStream_t copy2 = nullptr;  // internal second copy stream: fills alternate between the two
  bool own_copy = false;
  cudaStream_t last_stream = nullptr;
  bool have_last = false;        // work of this cache has been enqueued on last_stream
  cudaEvent_t e_done = nullptr;  // recorded on last_stream when the stream changes or at a resize
  cudaEvent_t e_copy[2] = {nullptr, nullptr};  // end of a call's copies on each copy stream
  uint32_t seq = 0;
  // device-fill calls whose summaries the host has not read yet (oldest first)
  struct Inflight {
    uint32_t seq;
    int layer, B;
    cudaEvent_t ta, tb;
    int tl_row;
  };
  std::deque<Inflight> inflight;
  moe_status sticky = MOE_OK;  // first error found while reading summaries, for moe_cache_sync
  std::string sticky_msg;
  int64_t call_index = 0;  // successful forward calls (trace numbering; not reset with the stats)
  int grid = 0;
  size_t smem = 0;
  int smem_h_floats = 0, rows_per_cta_max = 0;
  int stage_items = 0, stage_pitch = 0, stage_off = 0;  // W_down rows staged in shared memory
  // accounting
  moe_stats st{};
  bool profiling = false, tracing = false;
  std::vector<moe_event> trace;
  int64_t trace_total = 0;
  std::vector<cudaEvent_t> ev_pool;
  struct Timed {
    cudaEvent_t a, b;
    bool hit_only;
    int64_t records;
  };
  std::vector<Timed> pending;
  int inject_after = -1;
  int fill_mode = MOE_FILL_COPY;
  int prefill_prec = MOE_PREFILL_W4A16;
  // phase timeline (profiling level 2): ring of [kTlRing][12] GPU timestamps
  int profile_level = 0;
  unsigned long long* d_tl = nullptr;
  std::vector<std::pair<int, int>> tl_calls;  // (ring row, had fills) not yet read
  int tl_next = 0;
  moe_phase_times pt{};
  // prefill scratch (allocated at the first moe_prefill_stream call, grown on demand)
  struct Prefill {
    int T_cap = 0;
    int32_t *ids = nullptr, *cnt = nullptr, *base = nullptr, *offsets = nullptr, *pos = nullptr, *perm = nullptr;
    float* w = nullptr;
    void *xp = nullptr, *hp = nullptr;
    float* op = nullptr;
    cudaEvent_t loaded[2] = {nullptr, nullptr}, consumed[2] = {nullptr, nullptr}, start = nullptr;
    int32_t* tab = nullptr;   // [steps][E] record slot of each expert per step
    int tab_steps = 0;
    int32_t* zero = nullptr;  // {0}: slot table of the shared expert's one-record maps
    // pinned host copies of the bookkeeping (the state after a prefill is uploaded from them)
    int32_t *h_owner = nullptr, *h_map = nullptr;
    uint64_t *h_stamp = nullptr, *h_g = nullptr;
    struct Timed {
      cudaEvent_t a, b;
      int kind;  // 0 whole call, 1 copy, 2 compute, 3 gemm
      double flop;
    };
    std::vector<Timed> timed;
  } pf;
};

static constexpr int kTlRing = 1024;
static constexpr int kTlStamps = 20;
static constexpr int kRing = kSummaryRing;  // call summaries in flight (device-fill calls the host has not read)

static const char* kNotFound = "";

static size_t record_bytes(const moe_model_desc* d) {
  const size_t HI = (size_t)d->H * d->I;
  switch (d->wdtype) {
    case MOE_FP32: return 12 * HI;
    case MOE_BF16: return 6 * HI;
    case MOE_FP4: return 3 * HI / 2 + 3 * HI / 16;
  }
  return 0;
}

static moe_status check_desc(const moe_model_desc* d) {
  if (!d) return fail(MOE_ERR_INVALID_ARG, "desc is NULL");
  if (d->L < 1 || d->E < 1 || d->E > kMaxE) return fail(MOE_ERR_INVALID_ARG, "need L >= 1 and 1 <= E <= %d", kMaxE);
  if (d->k < 1 || d->k > kMaxK || d->k > d->E) return fail(MOE_ERR_INVALID_ARG, "need 1 <= k <= min(E, %d)", kMaxK);
  if (d->max_tokens < 1 || d->max_tokens > kMaxB) return fail(MOE_ERR_INVALID_ARG, "need 1 <= max_tokens <= %d", kMaxB);
  if (d->wdtype != MOE_FP32 && d->wdtype != MOE_BF16 && d->wdtype != MOE_FP4)
    return fail(MOE_ERR_INVALID_ARG, "unknown wdtype %d", d->wdtype);
  const int m = d->wdtype == MOE_FP4 ? 256 : 64;
  if (d->H < m || d->I < m || d->H % m || d->I % m)
    return fail(MOE_ERR_INVALID_ARG, "H and I must be positive multiples of %d for this format", m);
  if (d->wdtype == MOE_FP4 && d->H > 16384)  // the decode kernel rearranges an activation row in registers
    return fail(MOE_ERR_INVALID_ARG, "FP4 models need H <= 16384");
  if (d->has_shared != 0 && d->has_shared != 1) return fail(MOE_ERR_INVALID_ARG, "has_shared must be 0 or 1");
  if ((int64_t)d->L * d->E > (int64_t)1 << 30) return fail(MOE_ERR_INVALID_ARG, "L*E too large");
  return MOE_OK;
}

static bool is_pinned(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

static void free_all(moe_cache* c) {
  if (!c) return;
  cudaDeviceSynchronize();
  for (void* p : {(void*)c->d_map, (void*)c->d_owner, (void*)c->d_stamp, (void*)c->d_g, (void*)c->d_plan,
                  (void*)c->d_h, (void*)c->d_logits, (void*)c->d_bar, (void*)c->d_flags, (void*)c->d_oldest,
                  (void*)c->d_oldest_n, (void*)c->d_moves, (void*)c->d_tl, (void*)c->d_cst, (void*)c->d_o_part,
                  (void*)c->d_deferred, (void*)c->d_wave, (void*)c->d_seqctr})
    if (p) cudaFree(p);
  if (c->h_work) cudaFreeHost(c->h_work);
  if (c->h_err) cudaFreeHost(c->h_err);
  for (cudaEvent_t e : {c->e_done, c->e_copy[0], c->e_copy[1]})
    if (e) cudaEventDestroy(e);
  for (auto& f : c->inflight) {
    if (f.ta) cudaEventDestroy(f.ta);
    if (f.tb) cudaEventDestroy(f.tb);
  }
  for (auto& t : c->pending) {
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  for (cudaEvent_t e : c->ev_pool) cudaEventDestroy(e);
  for (void* p : {(void*)c->pf.ids, (void*)c->pf.cnt, (void*)c->pf.base, (void*)c->pf.offsets, (void*)c->pf.pos,
                  (void*)c->pf.perm, (void*)c->pf.w, c->pf.xp, c->pf.hp, (void*)c->pf.op, (void*)c->pf.tab,
                  (void*)c->pf.zero})
    if (p) cudaFree(p);
  for (void* p : {(void*)c->pf.h_owner, (void*)c->pf.h_map, (void*)c->pf.h_stamp, (void*)c->pf.h_g})
    if (p) cudaFreeHost(p);
  for (cudaEvent_t e : {c->pf.loaded[0], c->pf.loaded[1], c->pf.consumed[0], c->pf.consumed[1], c->pf.start})
    if (e) cudaEventDestroy(e);
  for (auto& t : c->pf.timed) {
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  if (c->own_copy && c->copy) cudaStreamDestroy(c->copy);
  if (c->copy2) cudaStreamDestroy(c->copy2);
  c->slots.release();
  delete c;
}

extern "C" size_t moe_record_bytes(const moe_model_desc* desc) {
  if (check_desc(desc) != MOE_OK) return 0;
  return record_bytes(desc);
}

extern "C" int32_t moe_version(void) { return 1; }

extern "C" const char* moe_last_error(void) { return g_err.empty() ? kNotFound : g_err.c_str(); }

// bytes of the first part of a record (everything the gate/up rows read)
static int64_t first_part_bytes(const moe_model_desc& d) {
  const int64_t HI = (int64_t)d.H * d.I;
  switch (d.wdtype) {
    case MOE_FP32: return 8 * HI;
    case MOE_BF16: return 4 * HI;
    default: return HI + HI / 8;
  }
}

extern "C" moe_status moe_cache_create(const moe_model_desc* desc, const void* host_pool, const void* shared_dev,
                                       int64_t n_slots, int64_t max_slots, void* copy_stream, moe_cache_t* out) {
  g_err.clear();
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (moe_status s = check_desc(desc)) return s;
  const int64_t LE = (int64_t)desc->L * desc->E;
  if (!host_pool) return fail(MOE_ERR_INVALID_ARG, "host_pool is NULL");
  if (desc->has_shared && !shared_dev) return fail(MOE_ERR_INVALID_ARG, "has_shared set but shared_dev is NULL");
  if (max_slots == 0) max_slots = LE;
  if (n_slots < 0 || max_slots < 0 || n_slots > max_slots || max_slots > (int64_t)INT32_MAX)
    return fail(MOE_ERR_INVALID_ARG, "need 0 <= n_slots <= max_slots < 2^31");
  const size_t S = record_bytes(desc);
  const uint8_t* pool = (const uint8_t*)host_pool;
  if (!is_pinned(pool) || !is_pinned(pool + (size_t)LE * S - 1))
    return fail(MOE_ERR_INVALID_ARG, "host_pool must be page-locked (cudaHostAlloc / cudaHostRegister) over all L*E records");

  moe_cache* c = new (std::nothrow) moe_cache();
  if (!c) return fail(MOE_ERR_OOM, "host allocation failed");
  c->d = *desc;
  c->S = (int64_t)S;
  c->C = n_slots;
  c->C_max = max_slots;
  c->host_pool = pool;
  c->shared_dev = (const uint8_t*)shared_dev;
  auto bail = [&](moe_status s) {
    std::string keep = g_err;
    free_all(c);
    g_err = keep;
    return s;
  };
  auto cu = [&](cudaError_t e, const char* what) -> moe_status {
    if (e == cudaSuccess) return MOE_OK;
    cudaGetLastError();
    return fail(e == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  };
  if (cudaGetDevice(&c->device) != cudaSuccess) return bail(fail(MOE_ERR_CUDA, "no CUDA device"));
  if (moe_status s = c->slots.init(c->device, (size_t)max_slots * S)) return bail(s);
  if (moe_status s = c->slots.resize((size_t)n_slots * S)) return bail(s);

  const int Bm = desc->max_tokens, k = desc->k, H = desc->H, I = desc->I, E = desc->E;
  const size_t nslot_alloc = (size_t)std::max<int64_t>(1, max_slots);
  moe_status s = MOE_OK;
  if ((s = cu(cudaMalloc(&c->d_map, sizeof(int32_t) * LE), "map")) ||
      (s = cu(cudaMalloc(&c->d_owner, sizeof(int32_t) * nslot_alloc), "owner")) ||
      (s = cu(cudaMalloc(&c->d_stamp, sizeof(uint64_t) * nslot_alloc), "stamp")) ||
      (s = cu(cudaMalloc(&c->d_g, sizeof(uint64_t)), "counter")) ||
      (s = cu(cudaMalloc(&c->d_plan, sizeof(Plan)), "plan")) ||
      (s = cu(cudaMalloc(&c->d_h, sizeof(float) * (size_t)(Bm * k + Bm) * I), "h")) ||
      (s = cu(cudaMalloc(&c->d_logits, sizeof(float) * (size_t)Bm * E), "logits")) ||
      (s = cu(cudaMalloc(&c->d_bar, sizeof(unsigned long long)), "barrier")) ||
      (s = cu(cudaMalloc(&c->d_flags, sizeof(unsigned) * (1 + 2 * kMaxU)), "flags")) ||
      (s = cu(cudaMalloc(&c->d_oldest, sizeof(int32_t) * kMaxU), "victim order")) ||
      (s = cu(cudaMalloc(&c->d_oldest_n, sizeof(int)), "victim order")) ||
      (s = cu(cudaMalloc(&c->d_cst, sizeof(CallState)), "call state")) ||
      (s = cu(cudaMalloc(&c->d_deferred, sizeof(unsigned long long)), "counter")) ||
      (s = cu(cudaMalloc(&c->d_wave, sizeof(unsigned) * 2 * kWaveCtrs), "wave counters")) ||
      (s = cu(cudaMalloc(&c->d_seqctr, sizeof(unsigned long long)), "sequence counter")))
    return bail(s);
  if ((s = cu(cudaMemset(c->d_map, 0xFF, sizeof(int32_t) * LE), "memset")) ||
      (s = cu(cudaMemset(c->d_owner, 0xFF, sizeof(int32_t) * nslot_alloc), "memset")) ||
      (s = cu(cudaMemset(c->d_stamp, 0, sizeof(uint64_t) * nslot_alloc), "memset")) ||
      (s = cu(cudaMemset(c->d_g, 0, sizeof(uint64_t)), "memset")) ||
      (s = cu(cudaMemset(c->d_bar, 0, sizeof(unsigned long long)), "memset")) ||
      (s = cu(cudaMemset(c->d_flags, 0, sizeof(unsigned) * (1 + 2 * kMaxU)), "memset")) ||
      (s = cu(cudaMemset(c->d_oldest_n, 0xFF, sizeof(int)), "memset")) ||
      (s = cu(cudaMemset(c->d_cst, 0xFF, sizeof(CallState)), "memset")) ||
      (s = cu(cudaMemset(c->d_deferred, 0, sizeof(unsigned long long)), "memset")) ||
      (s = cu(cudaMemset(c->d_wave, 0, sizeof(unsigned) * 2 * kWaveCtrs), "memset")) ||
      (s = cu(cudaMemset(c->d_seqctr, 0, sizeof(unsigned long long)), "memset")))
    return bail(s);
  if ((s = cu(cudaHostAlloc((void**)&c->h_work, sizeof(HostWork) * kRing, cudaHostAllocMapped), "pinned summary")) ||
      (s = cu(cudaHostAlloc((void**)&c->h_err, sizeof(int), cudaHostAllocMapped), "pinned error word")))
    return bail(s);
  memset((void*)c->h_work, 0, sizeof(HostWork) * kRing);
  *c->h_err = 0;
  if ((s = cu(cudaHostGetDevicePointer((void**)&c->d_work, c->h_work, 0), "mapped summary")) ||
      (s = cu(cudaHostGetDevicePointer((void**)&c->d_err, c->h_err, 0), "mapped error word")))
    return bail(s);
  if ((s = cu(cudaEventCreateWithFlags(&c->e_done, cudaEventDisableTiming), "event")) ||
      (s = cu(cudaEventCreateWithFlags(&c->e_copy[0], cudaEventDisableTiming), "event")) ||
      (s = cu(cudaEventCreateWithFlags(&c->e_copy[1], cudaEventDisableTiming), "event")))
    return bail(s);
  if (copy_stream) {
    c->copy = (cudaStream_t)copy_stream;
  } else {
    if ((s = cu(cudaStreamCreateWithFlags(&c->copy, cudaStreamNonBlocking), "copy stream"))) return bail(s);
    c->own_copy = true;
  }
  if ((s = cu(cudaStreamCreateWithFlags(&c->copy2, cudaStreamNonBlocking), "copy stream"))) return bail(s);
  // the copy stream signals landed fills with stream memory writes: check they work here
  {
    Drv& dr = drv();
    if (!dr.streamWriteValue32) return bail(fail(MOE_ERR_CUDA, "cuStreamWriteValue32 unavailable"));
    if (dr.streamWriteValue32((CUstream)c->copy, (CUdeviceptr)(c->d_flags), 0x5A5Au, 0) != CUDA_SUCCESS)
      return bail(fail(MOE_ERR_CUDA, "stream memory operations are not supported on this device"));
    unsigned probe = 0;
    if ((s = cu(cudaStreamSynchronize(c->copy), "probe")) ||
        (s = cu(cudaMemcpy(&probe, c->d_flags, sizeof(unsigned), cudaMemcpyDeviceToHost), "probe")))
      return bail(s);
    if (probe != 0x5A5Au) return bail(fail(MOE_ERR_CUDA, "stream memory write did not land"));
    if ((s = cu(cudaMemset(c->d_flags, 0, sizeof(unsigned)), "memset"))) return bail(s);
  }

  // layer-kernel launch shape: one CTA per SM; dynamic shared memory for the
  // tokens, an h buffer and the CTA's output rows
  int sms = 0, smem_optin = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, c->device);
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device);
  c->rows_per_cta_max = (H + sms - 1) / sms;
  const size_t xbytes = (((size_t)Bm * H * (desc->wdtype == MOE_FP32 ? 4 : 2)) + 15) & ~(size_t)15;
  const size_t obytes = (size_t)c->rows_per_cta_max * Bm * (k + 1) * 4;
  const size_t static_smem = layer_static_smem(desc->wdtype);
  const size_t budget = (size_t)smem_optin > static_smem + 1024 ? (size_t)smem_optin - static_smem - 1024 : 0;
  // staged h rows, float32 units: I floats, or for FP4 f16 values padded to
  // 40 per 32 (against bank conflicts), 20 float32 units per 32 values
  const size_t hrow_f = desc->wdtype == MOE_FP4 ? (size_t)I / 32 * 20 : (size_t)I;
  const size_t need_h = (size_t)Bm * hrow_f * 4;  // one expert with every token
  if (xbytes + obytes + need_h > budget)
    return bail(fail(MOE_ERR_INVALID_ARG, "max_tokens * (H, I) too large for the layer kernel's shared memory"));
  c->smem_h_floats = (int)std::min<size_t>((budget - xbytes - obytes) / 4, (size_t)(Bm * k + Bm) * hrow_f);
  c->smem_h_floats &= ~3;
  // what is left holds this CTA's W_down rows of as many resident experts as fit
  const int64_t down_row_bytes = desc->wdtype == MOE_FP32   ? 4LL * I
                                 : desc->wdtype == MOE_BF16 ? 2LL * I
                                                            : I / 2 + I / 16;
  const size_t stage_off = (layer_smem_bytes(desc->wdtype, Bm, H, k, c->smem_h_floats, c->rows_per_cta_max) + 15) &
                           ~(size_t)15;
  c->stage_pitch = (int)(c->rows_per_cta_max * down_row_bytes);
  c->stage_off = (int)stage_off;
  c->stage_items =
      stage_off < budget ? (int)std::min<size_t>((budget - stage_off) / (size_t)c->stage_pitch, (size_t)kMaxItems) : 0;
  c->smem = stage_off + (size_t)c->stage_items * c->stage_pitch;
  c->grid = layer_max_grid(desc->wdtype, c->smem);
  if (c->grid != sms || c->grid > kMaxGrid)  // the per-CTA row split assumes one CTA on every SM
    return bail(fail(MOE_ERR_CUDA, "layer kernel cannot keep one CTA resident on every SM (%d of %d)", c->grid, sms));
  c->o_part_floats = c->rows_per_cta_max * Bm * (k + 1);
  if ((s = cu(cudaMalloc(&c->d_o_part, sizeof(float) * (size_t)c->o_part_floats * c->grid), "partial sums")))
    return bail(s);
  if (cudaDeviceSynchronize() != cudaSuccess) return bail(fail(MOE_ERR_CUDA, "initialisation failed"));
  *out = c;
  return MOE_OK;
}

extern "C" moe_status moe_cache_destroy(moe_cache_t c) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  free_all(c);
  return MOE_OK;
}

// ----------------------------------------------------------- profiling events --
static cudaEvent_t take_event(moe_cache* c) {
  if (!c->ev_pool.empty()) {
    cudaEvent_t e = c->ev_pool.back();
    c->ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

static void drain_pending(moe_cache* c, bool wait) {
  size_t keep = 0;
  for (size_t i = 0; i < c->pending.size(); ++i) {
    const auto t = c->pending[i];
    if (wait) cudaEventSynchronize(t.b);
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, t.a, t.b) == cudaSuccess) {
      c->st.layer_ms += ms;
      c->st.layer_timed += 1;
      if (t.hit_only) {
        c->st.hit_only_ms += ms;
        c->st.hit_only_timed += 1;
        c->st.hit_only_records += t.records;
      }
      c->ev_pool.push_back(t.a);
      c->ev_pool.push_back(t.b);
    } else {
      cudaGetLastError();
      c->pending[keep++] = t;
    }
  }
  c->pending.resize(keep);
}

// Fold the recorded phase stamps into the running means.
static void drain_timeline(moe_cache* c) {
  if (c->tl_calls.empty()) return;
  cudaDeviceSynchronize();
  std::vector<unsigned long long> tl((size_t)kTlRing * kTlStamps);
  if (cudaMemcpy(tl.data(), c->d_tl, tl.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    c->tl_calls.clear();
    return;
  }
  for (auto [row, fills] : c->tl_calls) {
    const unsigned long long* t = &tl[(size_t)row * kTlStamps];
    int64_t& n = fills ? c->pt.calls_with_fills : c->pt.calls_hit_only;
    double* acc = fills ? c->pt.with_fills_us : c->pt.hit_only_us;
    // running mean per stamp (stamps never reached stay 0 and are skipped)
    for (int i = 0; i < kTlStamps; ++i) {
      if (!t[i] || !t[0]) continue;
      const unsigned long long ti = i == 16 ? ~t[i] : t[i];  // stamp 16 is kept as a complement (earliest)
      const double us = ((double)ti - (double)t[0]) / 1e3;
      acc[i] += (us - acc[i]) / (double)(n + 1);
    }
    n += 1;
  }
  c->tl_calls.clear();
}

// Wait until the layer kernel of call `seq` has published its summary.
static moe_status wait_summary(moe_cache* c, uint32_t seq, cudaStream_t s) {
  const HostWork* w = c->h_work + seq % kRing;
  const auto t0 = std::chrono::steady_clock::now();
  for (uint64_t spin = 0;; ++spin) {
    if (__atomic_load_n(&w->seq, __ATOMIC_ACQUIRE) == seq) return MOE_OK;
    if ((spin & 1023) == 1023) {
      cudaError_t q = cudaStreamQuery(s);
      if (q != cudaSuccess && q != cudaErrorNotReady)
        return fail(MOE_ERR_CUDA, "layer kernel failed: %s", cudaGetErrorString(q));
      if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(30))
        return fail(MOE_ERR_TIMEOUT, "layer kernel summary not seen after 30 s");
      if (spin > (1u << 20)) std::this_thread::yield();
    }
  }
}

// A kernel recorded that a bounded wait for the GPU gave up: wait for the
// streams, put the barrier counter back in step and drop the victim order.
static moe_status recover_after_timeout(moe_cache* c, cudaStream_t s) {
  CU_TRY(cudaStreamSynchronize(s));
  CU_TRY(cudaStreamSynchronize(c->copy));
  CU_TRY(cudaStreamSynchronize(c->copy2));
  CU_TRY(cudaMemset(c->d_bar, 0, sizeof(unsigned long long)));
  CU_TRY(cudaMemset(c->d_oldest_n, 0xFF, sizeof(int)));
  CU_TRY(cudaDeviceSynchronize());
  *(volatile int*)c->h_err = 0;
  return fail(MOE_ERR_TIMEOUT,
              "a bounded wait inside a kernel of this cache gave up (the rows of that call are NaN); state recovered");
}

// Counters, profiling records and trace events of one completed call from its summary.
static void account_call(moe_cache* c, int layer, int B, const HostWork& w, cudaEvent_t ta, cudaEvent_t tb,
                         int tl_row) {
  const moe_model_desc& d = c->d;
  const int n_u = w.n_u, n_miss = w.n_miss;
  if (tl_row >= 0) c->tl_calls.emplace_back(tl_row, n_miss > 0 ? 1 : 0);
  if (ta) {
    c->pending.push_back({ta, tb, n_miss == 0, (int64_t)n_u + d.has_shared});
    if (c->pending.size() > 4096) drain_pending(c, false);
  }
  moe_stats& st = c->st;
  const int64_t call_id = c->call_index++;
  st.calls += 1;
  st.tokens += B;
  st.hits += n_u - n_miss;
  st.misses += n_miss;
  st.routed_pairs += (int64_t)B * d.k;
  st.bytes_filled += (int64_t)n_miss * c->S;
  st.qstar_fills += w.qstar;
  st.records_streamed += n_u + d.has_shared;
  for (int r = 0; r < n_u; ++r) {
    if (w.fill[r] && w.evicted[r] >= 0) st.evictions += 1;
    if (!w.fill[r]) st.routed_pair_hits += w.pairs[r];
  }
  if (c->tracing) {
    for (int r = 0; r < n_u; ++r) {
      moe_event ev{};
      ev.call = call_id;
      ev.layer = layer;
      ev.expert = w.key[r] - layer * d.E;
      ev.kind = w.fill[r] ? MOE_EV_MISS : MOE_EV_HIT;
      ev.slot = w.slot[r];
      ev.evicted_key = w.evicted[r];
      c->trace.push_back(ev);
    }
  }
}

// Read the summaries of device-fill calls in flight until at most `keep` remain.
static moe_status drain_inflight(moe_cache* c, size_t keep) {
  while (c->inflight.size() > keep) {
    const auto f = c->inflight.front();
    if (moe_status e = wait_summary(c, f.seq, c->last_stream)) return e;
    const HostWork& w = c->h_work[f.seq % kRing];
    if (w.err != MOE_OK) {
      if (c->sticky == MOE_OK) {
        c->sticky = MOE_ERR_CUDA;
        c->sticky_msg = "internal error: victim selection found an inconsistent cache state";
      }
      if (f.ta) {
        c->ev_pool.push_back(f.ta);
        c->ev_pool.push_back(f.tb);
      }
    } else {
      account_call(c, f.layer, f.B, w, f.ta, f.tb, f.tl_row);
    }
    c->inflight.pop_front();
  }
  return MOE_OK;
}

// Order this call after the cache's earlier work when it comes on another stream.
static moe_status follow_stream(moe_cache* c, cudaStream_t s) {
  if (c->have_last && s != c->last_stream) {
    CU_TRY(cudaEventRecord(c->e_done, c->last_stream));
    CU_TRY(cudaStreamWaitEvent(s, c->e_done, 0));
  }
  c->last_stream = s;
  c->have_last = true;
  return MOE_OK;
}

static cudaError_t launch_k1(moe_cache* c, const LayerParams& p, cudaStream_t s) {
  if (c->pdl) {
    cudaError_t e = launch_layer(c->d.wdtype, p, c->grid, c->smem, true, s);
    if (e == cudaSuccess) {
      c->st.pdl_launches += 1;
      return e;
    }
    cudaGetLastError();  // programmatic dependent launch refused for this launch: launch plainly from now on
    c->pdl = false;
  }
  return launch_layer(c->d.wdtype, p, c->grid, c->smem, false, s);
}

// Bounds-check counters of the debug build: one device pair per process
// (current device at first use), zero at start.
unsigned* moe::debug_counters() {
  static unsigned* d = nullptr;
  static std::mutex m;
  std::lock_guard<std::mutex> lk(m);
  if (!d) {
    if (cudaMalloc(&d, 2 * sizeof(unsigned)) != cudaSuccess || cudaMemset(d, 0, 2 * sizeof(unsigned)) != cudaSuccess) {
      cudaGetLastError();
      d = nullptr;
    }
  }
  return d;
}

extern "C" int32_t moe_debug_bounds_enabled(void) {
#ifdef MOE_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

extern "C" moe_status moe_debug_violations(int64_t* count, int32_t* first_site) {
  g_err.clear();
  if (!count || !first_site) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  unsigned h[2] = {0u, 0u};
  if (unsigned* d = debug_counters()) {
    CU_TRY(cudaDeviceSynchronize());
    CU_TRY(cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost));
  }
  *count = h[0];
  *first_site = (int32_t)h[1];
  return MOE_OK;
}

// The fields of one call's LayerParams that do not depend on its sequence number.
static LayerParams call_params(moe_cache* c, int32_t layer, const void* x, const float* lg, int32_t B, void* y,
                               const moe_layer_aux* aux) {
  const moe_model_desc& d = c->d;
  LayerParams p{};
  p.L = d.L; p.E = d.E; p.k = d.k; p.B = B; p.layer = layer; p.H = d.H; p.I = d.I;
  p.C = c->C;
  p.logits = lg;
  p.st = CacheDev{c->d_map, c->d_owner, c->d_stamp, c->d_g};
  p.plan = c->d_plan;
  p.plan_flag = c->d_flags;
  p.fill_flags = c->d_flags + 1;
  p.bar = c->d_bar;
  p.err = c->d_err;
  p.cst = c->d_cst;
  p.o_part = c->d_o_part;
  p.o_part_floats = c->o_part_floats;
  p.wait_gu_ns = c->wait_gu_ns;
  p.wait_dn_ns = c->wait_dn_ns;
  p.deferred = c->d_deferred;
  p.split_bp = c->split_bp;
  p.split_bh = c->split_bh;
  p.has_shared = d.has_shared;
  p.device_fill = c->fill_mode == MOE_FILL_DEVICE;
  p.pool = c->host_pool;  // pinned pages are mapped at the same address under unified addressing
  p.slots = (const uint8_t*)c->slots.base;
  p.S = c->S;
  p.shared_rec = d.has_shared ? c->shared_dev + (int64_t)layer * c->S : nullptr;
  p.x = x;
  p.h = c->d_h;
  p.h_shared_row0 = d.max_tokens * d.k;
  p.y = y;
  p.smem_h_floats = c->smem_h_floats;
  p.rows_per_cta_max = c->rows_per_cta_max;
  p.stage_items = c->stage_items;
  p.stage_pitch = c->stage_pitch;
  p.stage_off = c->stage_off;
  p.oldest = c->d_oldest;
  p.oldest_n = c->d_oldest_n;
  p.dbg = debug_counters();
  if (aux) {
    p.aux_ids = aux->ids; p.aux_w = aux->weights; p.aux_slots = aux->slots;
    p.aux_perm = aux->perm; p.aux_offsets = aux->offsets; p.aux_logits = aux->logits;
    p.aux_qstar = aux->qstar;
  }
  return p;
}

// A decode call in graph mode: nothing on the host depends on the call's
// progress (no wait, no event, no host counter of its own), so the launch can
// be captured into a CUDA graph and replayed; the kernel numbers the call from
// the device counter and moe_cache_sync reads the summaries.
static moe_status forward_graph(moe_cache* c, int32_t layer, const void* x, const float* logits,
                                const float* router_w, int32_t B, void* y, cudaStream_t s,
                                const moe_layer_aux* aux) {
  const moe_model_desc& d = c->d;
  if ((int64_t)B * d.k > c->C)
    return fail(MOE_ERR_INVALID_ARG, "graph mode needs B*k <= n_slots (a capacity error could not be reported)");
  // a stream being captured is ordered by whoever captures it (a wait on an
  // event recorded outside the capture would break it)
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  CU_TRY(cudaStreamIsCapturing(s, &cap));
  if (cap == cudaStreamCaptureStatusNone)
    if (moe_status e = follow_stream(c, s)) return e;
  const float* lg = logits;
  if (!lg) {
    CU_TRY(launch_router_logits(x, d.wdtype != MOE_FP32, router_w, B, d.E, d.H, c->d_logits, s));
    lg = c->d_logits;
  }
  LayerParams p = call_params(c, layer, x, lg, B, y, aux);
  p.seq_ctr = c->d_seqctr;
  p.work = c->d_work;     // the ring's base: the kernel picks entry seq % ring
  p.wave_ctr = c->d_wave;  // both counter sets: the kernel picks by seq parity
  CU_TRY(launch_k1(c, p, s));
  return MOE_OK;
}

// Graph mode: account every call whose summary the ring still holds, up to
// the device counter; calls whose entry a later call overwrote are counted as
// lost.  The stream must be idle.
static moe_status drain_graph(moe_cache* c) {
  unsigned long long ctr = 0;
  CU_TRY(cudaMemcpy(&ctr, c->d_seqctr, sizeof(ctr), cudaMemcpyDeviceToHost));
  const uint32_t last = (uint32_t)(ctr / (unsigned long long)c->grid);
  for (uint32_t q = c->seq + 1; q != last + 1; ++q) {
    const HostWork& w = c->h_work[q % kRing];
    c->st.layer_launches += 1;
    if (__atomic_load_n(&w.seq, __ATOMIC_ACQUIRE) != q) {
      c->st.summaries_lost += 1;
      continue;
    }
    if (w.err != MOE_OK) {
      if (c->sticky == MOE_OK) {
        c->sticky = MOE_ERR_CUDA;
        c->sticky_msg = "internal error: victim selection found an inconsistent cache state";
      }
      continue;
    }
    account_call(c, w.layer, w.B, w, nullptr, nullptr, -1);
  }
  c->seq = last;
  return MOE_OK;
}

extern "C" moe_status moe_cache_set_graph_mode(moe_cache_t c, int32_t on) {
  g_err.clear();
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  if (on && c->fill_mode != MOE_FILL_DEVICE)
    return fail(MOE_ERR_INVALID_ARG, "graph mode needs device-driven fills (moe_cache_set_fill_mode)");
  if ((bool)on == c->graph) return MOE_OK;
  CU_TRY(cudaDeviceSynchronize());
  if (on) {
    if (moe_status e = drain_inflight(c, 0)) return e;
    const unsigned long long ctr = (unsigned long long)c->seq * (unsigned long long)c->grid;
    CU_TRY(cudaMemcpy(c->d_seqctr, &ctr, sizeof(ctr), cudaMemcpyHostToDevice));
    c->graph = true;
  } else {
    if (moe_status e = drain_graph(c)) return e;
    c->graph = false;
  }
  return MOE_OK;
}

extern "C" moe_status moe_layer_forward_ex(moe_cache_t c, int32_t layer, const void* x, const float* logits,
                                           const float* router_w, int32_t B, void* y, void* stream,
                                           const moe_layer_aux* aux) {
  g_err.clear();
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  const moe_model_desc& d = c->d;
  if (layer < 0 || layer >= d.L) return fail(MOE_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (B < 1 || B > d.max_tokens) return fail(MOE_ERR_INVALID_ARG, "B=%d outside 1..%d", B, d.max_tokens);
  if (!x || !y) return fail(MOE_ERR_INVALID_ARG, "x and y must be device pointers");
  if (!logits && !router_w) return fail(MOE_ERR_INVALID_ARG, "need logits or router_w");
  cudaStream_t s = (cudaStream_t)stream;
  if (c->graph) return forward_graph(c, layer, x, logits, router_w, B, y, s, aux);
  if (*(volatile int*)c->h_err != 0) {
    drain_inflight(c, 0);
    return recover_after_timeout(c, s);
  }
  // device-fill calls run ahead of the host; a call that could exceed the
  // capacity (B*k > C) waits for its summary so the error is this call's
  const bool device = c->fill_mode == MOE_FILL_DEVICE;
  const bool async = device && (int64_t)B * d.k <= c->C;
  if (!async || c->inflight.size() >= (size_t)kRing - 1)
    if (moe_status e = drain_inflight(c, async ? (size_t)kRing / 2 : 0)) return e;
  if (moe_status e = follow_stream(c, s)) return e;

  const float* lg = logits;
  if (!lg) {
    CU_TRY(launch_router_logits(x, d.wdtype != MOE_FP32, router_w, B, d.E, d.H, c->d_logits, s));
    lg = c->d_logits;
  }
  const uint32_t seq = ++c->seq;
  LayerParams p = call_params(c, layer, x, lg, B, y, aux);
  p.work = c->d_work + seq % kRing;
  p.seq = seq;
  p.wave_ctr = c->d_wave + (seq & 1) * kWaveCtrs;
  p.wave_next = c->d_wave + ((seq + 1) & 1) * kWaveCtrs;
  int tl_row = -1;
  if (c->profile_level >= 2 && c->d_tl) {
    if ((int)c->tl_calls.size() >= kTlRing / 2) {
      if (moe_status e = drain_inflight(c, 0)) return e;
      drain_timeline(c);
    }
    tl_row = c->tl_next;
    c->tl_next = (c->tl_next + 1) % kTlRing;
    p.tl = c->d_tl + (size_t)tl_row * kTlStamps;
    p.tl_next = c->d_tl + (size_t)c->tl_next * kTlStamps;  // cleared by this call (no launch in between)
  }
  cudaEvent_t ta = nullptr, tb = nullptr;
  if (c->profiling) {
    ta = take_event(c);
    tb = take_event(c);
    cudaEventRecord(ta, s);
  }
  CU_TRY(launch_k1(c, p, s));
  if (c->profiling) cudaEventRecord(tb, s);
  c->st.layer_launches += 1;
  if (async) {
    c->inflight.push_back({seq, layer, B, ta, tb, tl_row});
    return MOE_OK;
  }

  const auto t_launch = std::chrono::steady_clock::now();
  if (moe_status w = wait_summary(c, seq, s)) return w;
  const auto t_seen = std::chrono::steady_clock::now();
  c->st.host_wait_us += std::chrono::duration<double, std::micro>(t_seen - t_launch).count();
  const HostWork& w = c->h_work[seq % kRing];
  if (w.err != MOE_OK) {
    if (ta) {
      c->ev_pool.push_back(ta);
      c->ev_pool.push_back(tb);
    }
    if (w.err == MOE_ERR_CAPACITY)
      return fail(MOE_ERR_CAPACITY, "layer %d routes %d distinct experts but the cache has %lld slots", layer, w.n_u,
                  (long long)c->C);
    return fail(MOE_ERR_CUDA, "internal error: victim selection found an inconsistent cache state");
  }
  const int n_miss = w.n_miss;
  if (n_miss > 0 && !device) {
    // one copy per half record, each followed by a flag the layer kernel waits
    // on; records alternate between two copy streams so that one stream's
    // flag write and next-copy start overlap the other's transfer.  No earlier
    // kernel can still read a victim slot: the summary is written after the
    // layer kernel's dependency wait, i.e. after everything before this call
    // on the compute stream has completed.
    Drv& dr = drv();
    const int64_t part1 = first_part_bytes(d), part2 = c->S - part1;
    unsigned* flags = c->d_flags + 1;
    int f = 0, half = 0;
    bool failed = false;
    std::string why;
    for (f = 0; f < n_miss && !failed; ++f) {
      const int r = w.fill_order[f];
      uint8_t* dst = (uint8_t*)c->slots.base + (int64_t)w.slot[r] * c->S;
      const uint8_t* src = c->host_pool + (int64_t)w.key[r] * c->S;
      for (half = 0; half < 2; ++half) {
        if (c->inject_after >= 0 && 2 * f + half >= 2 * c->inject_after) {
          failed = true;
          why = "injected fill failure";
          break;
        }
        const int64_t off = half ? part1 : 0, len = half ? part2 : part1;
        cudaStream_t cs = (f & 1) ? c->copy2 : c->copy;
        cudaError_t ce = cudaMemcpyAsync(dst + off, src + off, len, cudaMemcpyHostToDevice, cs);
        if (ce != cudaSuccess) {
          failed = true;
          why = cudaGetErrorString(ce);
          cudaGetLastError();
          break;
        }
        if (dr.streamWriteValue32((CUstream)cs, (CUdeviceptr)(flags + half * kMaxU + f), seq, 0) !=
            CUDA_SUCCESS) {
          failed = true;
          why = "cuStreamWriteValue32 failed";
          break;
        }
      }
      if (failed) break;
    }
    if (failed) {
      // release the kernel: this and every later half carries the error bit
      c->inject_after = -1;
      for (int g = f; g < n_miss; ++g)
        for (int hh = (g == f ? half : 0); hh < 2; ++hh)
          dr.streamWriteValue32((CUstream)c->copy, (CUdeviceptr)(flags + hh * kMaxU + g), seq | kFlagError, 0);
    }
    // the completion kernel runs after every copy of the call; it finishes
    // the rows the layer kernel handed over, or undoes the call after a failure
    CU_TRY(cudaEventRecord(c->e_copy[0], c->copy));
    CU_TRY(cudaStreamWaitEvent(s, c->e_copy[0], 0));
    if (n_miss > 1 || failed) {
      CU_TRY(cudaEventRecord(c->e_copy[1], c->copy2));
      CU_TRY(cudaStreamWaitEvent(s, c->e_copy[1], 0));
    }
    CU_TRY(launch_layer_finish(d.wdtype, p, c->grid, c->smem, s));
    c->st.finish_launches += 1;
    if (failed) {
      if (ta) {
        c->ev_pool.push_back(ta);
        c->ev_pool.push_back(tb);
      }
      return fail(MOE_ERR_CUDA, "fill %d of %d could not be issued (%s); cache rolled back", f + 1, n_miss,
                  why.c_str());
    }
    c->st.host_issue_us += std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t_seen).count();
  }
  account_call(c, layer, B, w, ta, tb, tl_row);
  return MOE_OK;
}

extern "C" moe_status moe_layer_forward(moe_cache_t c, int32_t layer, const void* x, const float* logits,
                                        const float* router_w, int32_t B, void* y, void* stream) {
  return moe_layer_forward_ex(c, layer, x, logits, router_w, B, y, stream, nullptr);
}

// --------------------------------------------------------------------- resize --
extern "C" moe_status moe_cache_resize(moe_cache_t c, int64_t n_slots, void* stream) {
  g_err.clear();
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  if (n_slots < 0 || n_slots > c->C_max)
    return fail(MOE_ERR_INVALID_ARG, "n_slots %lld outside 0..%lld", (long long)n_slots, (long long)c->C_max);
  if (c->have_last) {
    // everything enqueued on the cache's stream so far (its last calls among it)
    CU_TRY(cudaEventRecord(c->e_done, c->last_stream));
    if (cudaEventQuery(c->e_done) == cudaErrorNotReady)
      return fail(MOE_ERR_BUSY, "a forward of this cache is still running on the GPU");
  }
  if (cudaStreamQuery(c->copy) == cudaErrorNotReady || cudaStreamQuery(c->copy2) == cudaErrorNotReady)
    return fail(MOE_ERR_BUSY, "fills still in flight");
  cudaGetLastError();
  if (moe_status e = drain_inflight(c, 0)) return e;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t C = c->C, LE = (int64_t)c->d.L * c->d.E;
  std::vector<int32_t> owner(std::max<int64_t>(C, n_slots), -1);
  std::vector<uint64_t> stamp(std::max<int64_t>(C, n_slots), 0);
  if (C > 0) {
    CU_TRY(cudaMemcpy(owner.data(), c->d_owner, sizeof(int32_t) * C, cudaMemcpyDeviceToHost));
    CU_TRY(cudaMemcpy(stamp.data(), c->d_stamp, sizeof(uint64_t) * C, cudaMemcpyDeviceToHost));
  }
  if (n_slots < C) {
    // survivors: the n_slots most recent experts
    std::vector<int64_t> occ;
    for (int64_t i = 0; i < C; ++i)
      if (owner[i] >= 0) occ.push_back(i);
    std::vector<int64_t> by_recency = occ;
    std::sort(by_recency.begin(), by_recency.end(), [&](int64_t a, int64_t b) { return stamp[a] > stamp[b]; });
    std::vector<char> keep(C, 0);
    for (int64_t i = 0; i < (int64_t)by_recency.size() && i < n_slots; ++i) keep[by_recency[i]] = 1;
    for (int64_t i : occ) {  // ascending slot order
      if (keep[i]) continue;
      if (c->tracing) {
        moe_event ev{};
        ev.call = c->call_index;
        ev.layer = owner[i] / c->d.E;
        ev.expert = owner[i] % c->d.E;
        ev.kind = MOE_EV_RESIZE_EVICT;
        ev.slot = (int32_t)i;
        ev.evicted_key = owner[i];
        c->trace.push_back(ev);
      }
      owner[i] = -1;
      stamp[i] = 0;
      c->st.resize_evictions += 1;
    }
    std::vector<int32_t> moves;
    int64_t vac = 0;
    for (int64_t src = n_slots; src < C; ++src) {
      if (!keep[src]) continue;
      while (owner[vac] >= 0) ++vac;  // a vacancy below n_slots always exists here
      moves.push_back((int32_t)src);
      moves.push_back((int32_t)vac);
      owner[vac] = owner[src];
      stamp[vac] = stamp[src];
      owner[src] = -1;
      stamp[src] = 0;
      ++vac;
    }
    const int n_moves = (int)(moves.size() / 2);
    if (n_moves > 0) {
      if (c->moves_cap < (int64_t)moves.size()) {
        if (c->d_moves) cudaFree(c->d_moves);
        c->d_moves = nullptr;
        c->moves_cap = 0;
        CU_TRY(cudaMalloc(&c->d_moves, sizeof(int32_t) * moves.size()));
        c->moves_cap = (int64_t)moves.size();
      }
      CU_TRY(cudaMemcpyAsync(c->d_moves, moves.data(), sizeof(int32_t) * moves.size(), cudaMemcpyHostToDevice, s));
      CU_TRY(launch_slot_moves((uint8_t*)c->slots.base, c->S, c->d_moves, n_moves, s));
    }
    c->st.resize_moves += n_moves;
    CU_TRY(cudaStreamSynchronize(s));
    if (moe_status st = c->slots.resize((size_t)n_slots * c->S)) return st;
  } else if (n_slots > C) {
    if (moe_status st = c->slots.resize((size_t)n_slots * c->S)) return st;
  }
  // rebuild the residency table from the slot owners
  std::vector<int32_t> map(LE, -1);
  for (int64_t i = 0; i < n_slots; ++i)
    if (owner[i] >= 0) map[owner[i]] = (int32_t)i;
  if (n_slots > 0) {
    CU_TRY(cudaMemcpyAsync(c->d_owner, owner.data(), sizeof(int32_t) * n_slots, cudaMemcpyHostToDevice, s));
    CU_TRY(cudaMemcpyAsync(c->d_stamp, stamp.data(), sizeof(uint64_t) * n_slots, cudaMemcpyHostToDevice, s));
  }
  CU_TRY(cudaMemcpyAsync(c->d_map, map.data(), sizeof(int32_t) * LE, cudaMemcpyHostToDevice, s));
  CU_TRY(cudaMemsetAsync(c->d_oldest_n, 0xFF, sizeof(int), s));
  CU_TRY(cudaStreamSynchronize(s));
  c->C = n_slots;
  c->st.resize_calls += 1;
  return MOE_OK;
}

// -------------------------------------------------------------- introspection --
static void drain_prefill(moe_cache* c) {
  for (auto& t : c->pf.timed) {
    cudaEventSynchronize(t.b);
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, t.a, t.b) == cudaSuccess) {
      if (t.kind == 0) c->st.prefill_ms += ms;
      else if (t.kind == 1) c->st.prefill_copy_ms += ms;
      else if (t.kind == 2) c->st.prefill_compute_ms += ms;
      else {
        c->st.prefill_gemm_ms += ms;
        c->st.prefill_gemm_flop += t.flop;
      }
    }
    cudaGetLastError();
    c->ev_pool.push_back(t.a);
    c->ev_pool.push_back(t.b);
  }
  c->pf.timed.clear();
}

static unsigned long long read_deferred(moe_cache* c) {
  unsigned long long v = 0;
  if (cudaMemcpy(&v, c->d_deferred, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) cudaGetLastError();
  return v;
}

extern "C" moe_status moe_cache_stats(moe_cache_t c, moe_stats* out) {
  if (!c || !out) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  if (moe_status e = drain_inflight(c, 0)) return e;
  drain_pending(c, true);
  drain_prefill(c);
  *out = c->st;
  out->deferred_calls = (int64_t)(read_deferred(c) - c->deferred_base);
  return MOE_OK;
}

extern "C" moe_status moe_cache_reset_stats(moe_cache_t c) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  if (moe_status e = drain_inflight(c, 0)) return e;
  drain_pending(c, true);
  drain_timeline(c);
  drain_prefill(c);
  c->st = moe_stats{};
  c->pt = moe_phase_times{};
  c->deferred_base = read_deferred(c);
  return MOE_OK;
}

extern "C" moe_status moe_cache_sync(moe_cache_t c, void* stream) {
  g_err.clear();
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  cudaStream_t s = (cudaStream_t)stream;
  CU_TRY(cudaStreamSynchronize(s));
  if (c->have_last && c->last_stream != s) CU_TRY(cudaStreamSynchronize(c->last_stream));
  CU_TRY(cudaStreamSynchronize(c->copy));
  CU_TRY(cudaStreamSynchronize(c->copy2));
  if (c->graph) {
    CU_TRY(cudaDeviceSynchronize());  // replays may run on any stream
    if (moe_status e = drain_graph(c)) return e;
  }
  if (moe_status e = drain_inflight(c, 0)) return e;
  if (*(volatile int*)c->h_err != 0) return recover_after_timeout(c, s);
  if (c->sticky != MOE_OK) {
    const moe_status e = c->sticky;
    c->sticky = MOE_OK;
    return fail(e, "%s", c->sticky_msg.c_str());
  }
  return MOE_OK;
}

extern "C" moe_status moe_cache_set_split_bandwidths(moe_cache_t c, double b_p, double b_h) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  if (!(b_p >= 0.0) || !(b_h >= 0.0)) return fail(MOE_ERR_INVALID_ARG, "bandwidths must be >= 0");
  if (moe_status e = drain_inflight(c, 0)) return e;
  c->split_bp = b_p;
  c->split_bh = b_h;
  return MOE_OK;
}

extern "C" moe_status moe_cache_set_wait_limit_ns(moe_cache_t c, int64_t gate_up_ns, int64_t down_ns) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  if (gate_up_ns < 0 || down_ns < 0 || gate_up_ns > 60000000000LL || down_ns > 60000000000LL)
    return fail(MOE_ERR_INVALID_ARG, "wait limits must lie in 0 .. 60 s");
  c->wait_gu_ns = (unsigned long long)gate_up_ns;
  c->wait_dn_ns = (unsigned long long)down_ns;
  return MOE_OK;
}

extern "C" moe_status moe_cache_set_profiling(moe_cache_t c, int32_t on) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  c->profiling = on != 0;
  c->profile_level = on;
  if (on >= 2 && !c->d_tl)
    CU_TRY(cudaMalloc(&c->d_tl, sizeof(unsigned long long) * kTlRing * kTlStamps));
  if (on >= 2) {  // each call clears the row of the call after it; the first row starts clear
    CU_TRY(cudaDeviceSynchronize());
    CU_TRY(cudaMemset(c->d_tl + (size_t)c->tl_next * kTlStamps, 0, kTlStamps * sizeof(unsigned long long)));
  }
  return MOE_OK;
}

extern "C" moe_status moe_cache_phase_times(moe_cache_t c, moe_phase_times* out) {
  if (!c || !out) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  if (moe_status e = drain_inflight(c, 0)) return e;
  drain_timeline(c);
  *out = c->pt;
  return MOE_OK;
}

extern "C" moe_status moe_cache_set_trace(moe_cache_t c, int32_t on) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  c->tracing = on != 0;
  return MOE_OK;
}

extern "C" moe_status moe_cache_trace(moe_cache_t c, moe_event* buf, int64_t cap, int64_t* n) {
  if (!c || !n || (cap > 0 && !buf)) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  if (moe_status e = drain_inflight(c, 0)) return e;
  *n = (int64_t)c->trace.size();
  const int64_t m = std::min<int64_t>(cap, *n);
  if (m > 0) memcpy(buf, c->trace.data(), sizeof(moe_event) * m);
  return MOE_OK;
}

extern "C" moe_status moe_cache_state(moe_cache_t c, int32_t* owner, uint64_t* stamp, int64_t cap, int64_t* n_slots,
                                      uint64_t* counter) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  CU_TRY(cudaDeviceSynchronize());
  if (moe_status e = drain_inflight(c, 0)) return e;
  const int64_t m = std::min<int64_t>(cap, c->C);
  if (owner && m > 0) CU_TRY(cudaMemcpy(owner, c->d_owner, sizeof(int32_t) * m, cudaMemcpyDeviceToHost));
  if (stamp && m > 0) CU_TRY(cudaMemcpy(stamp, c->d_stamp, sizeof(uint64_t) * m, cudaMemcpyDeviceToHost));
  if (n_slots) *n_slots = c->C;
  if (counter) CU_TRY(cudaMemcpy(counter, c->d_g, sizeof(uint64_t), cudaMemcpyDeviceToHost));
  return MOE_OK;
}

extern "C" const void* moe_cache_slot_ptr(moe_cache_t c, int64_t s) {
  if (!c || s < 0 || s >= c->C) return nullptr;
  return (const uint8_t*)c->slots.base + s * c->S;
}

extern "C" moe_status moe_cache_set_fill_mode(moe_cache_t c, int32_t mode) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  if (mode != MOE_FILL_COPY && mode != MOE_FILL_DEVICE) return fail(MOE_ERR_INVALID_ARG, "unknown fill mode %d", mode);
  if (c->graph && mode != MOE_FILL_DEVICE) return fail(MOE_ERR_INVALID_ARG, "graph mode needs device-driven fills");
  if (moe_status e = drain_inflight(c, 0)) return e;
  if (mode == MOE_FILL_DEVICE) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, c->host_pool) != cudaSuccess || a.devicePointer != (void*)c->host_pool) {
      cudaGetLastError();
      return fail(MOE_ERR_INVALID_ARG, "the host pool is not mapped at the same device address");
    }
  }
  c->fill_mode = mode;
  return MOE_OK;
}

extern "C" moe_status moe_cache_set_prefill_precision(moe_cache_t c, int32_t mode) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  if (mode != MOE_PREFILL_W4A16 && mode != MOE_PREFILL_W4A4)
    return fail(MOE_ERR_INVALID_ARG, "unknown prefill precision %d", mode);
  if (mode == MOE_PREFILL_W4A4 && c->d.wdtype != MOE_FP4)
    return fail(MOE_ERR_INVALID_ARG, "FP4 x FP4 prefill needs a MOE_FP4 model");
  c->prefill_prec = mode;
  return MOE_OK;
}

extern "C" moe_status moe_quantize_fp4(const void* x, int32_t x_dtype, int64_t rows, int32_t K, uint8_t* codes,
                                       uint8_t* scales, void* stream) {
  g_err.clear();
  if (x_dtype != MOE_BF16 && x_dtype != MOE_FP32) return fail(MOE_ERR_INVALID_ARG, "x_dtype must be MOE_BF16 or MOE_FP32");
  if (rows < 0 || K <= 0 || K % 16) return fail(MOE_ERR_INVALID_ARG, "need rows >= 0 and K a positive multiple of 16");
  if (rows == 0) return MOE_OK;
  if (!x || !codes || !scales) return fail(MOE_ERR_INVALID_ARG, "x, codes and scales must be device pointers");
  if (((uintptr_t)codes & 7) || ((uintptr_t)x & (x_dtype == MOE_FP32 ? 3 : 1)))
    return fail(MOE_ERR_INVALID_ARG, "codes must be 8-byte aligned and x aligned to its element size");
  CU_TRY(quantize_rows(x, x_dtype == MOE_FP32, rows, K, codes, scales, (cudaStream_t)stream));
  return MOE_OK;
}

extern "C" moe_status moe_measure_read_rate(const void* bufs, int64_t bytes, int32_t n_bufs, int32_t reps,
                                            void* stream, double* gbps) {
  g_err.clear();
  if (!bufs || !gbps) return fail(MOE_ERR_INVALID_ARG, "bufs and gbps must not be NULL");
  if (bytes <= 0 || bytes % 16 || ((uintptr_t)bufs & 15))
    return fail(MOE_ERR_INVALID_ARG, "bytes must be a positive multiple of 16 and bufs 16-byte aligned");
  if (n_bufs < 1 || reps < 1) return fail(MOE_ERR_INVALID_ARG, "need n_bufs >= 1 and reps >= 1");
  CU_TRY(read_rate(static_cast<const uint8_t*>(bufs), (size_t)bytes, n_bufs, reps, (cudaStream_t)stream, gbps));
  return MOE_OK;
}

extern "C" moe_status moe_cache_inject_fill_failure(moe_cache_t c, int32_t after) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  c->inject_after = after;
  return MOE_OK;
}

// ---------------------------------------------------------------------- prefill --
static moe_status encode_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                             const uint32_t* box, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                             CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  Drv& d = drv();
  cuuint64_t gd[3], gs[2];
  cuuint32_t bx[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) { gd[i] = dims[i]; bx[i] = box[i]; }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides[i];
  const CUresult r = d.tensorMapEncodeTiled(m, dtype, rank, const_cast<void*>(base), gd, gs, bx, es,
                                            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
}

// [rows][K] bf16 activations, boxes of 128 rows x 64 elements
static moe_status map_rows(CUtensorMap* m, const void* base, int64_t rows, int K) {
  const uint64_t dims[2] = {(uint64_t)K, (uint64_t)rows}, strides[1] = {(uint64_t)K * 2};
  const uint32_t box[2] = {64, 128};
  return encode_map(m, base, 2, dims, strides, box);
}

// [n][rows][K] bf16 matrices n records apart, boxes of 128 rows x 64 elements
static moe_status map_weights(CUtensorMap* m, const void* base, int n, int rows, int K, int64_t rec_stride) {
  const uint64_t dims[3] = {(uint64_t)K, (uint64_t)rows, (uint64_t)n};
  const uint64_t strides[2] = {(uint64_t)K * 2, (uint64_t)rec_stride};
  const uint32_t box[3] = {64, 128, 1};
  return encode_map(m, base, 3, dims, strides, box);
}

// FP4 weights of n records: e2m1 codes [n][rows][K/2] bytes, boxes of 128
// rows x 32 bytes (one 64-element K-step); e4m3 scales [n][rows][K/16], boxes
// of 128 rows x 16 bytes (four K-steps).  Row strides K/2 and K/16 are
// multiples of 16 for every accepted FP4 shape (H, I multiples of 256).
static moe_status map_fp4_codes(CUtensorMap* m, const void* base, int n, int rows, int K, int64_t rec_stride) {
  const uint64_t dims[3] = {(uint64_t)K / 2, (uint64_t)rows, (uint64_t)n};
  const uint64_t strides[2] = {(uint64_t)K / 2, (uint64_t)rec_stride};
  const uint32_t box[3] = {32, 128, 1};
  return encode_map(m, base, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_NONE);
}
static moe_status map_fp4_scales(CUtensorMap* m, const void* base, int n, int rows, int K, int64_t rec_stride) {
  const uint64_t dims[3] = {(uint64_t)K / 16, (uint64_t)rows, (uint64_t)n};
  const uint64_t strides[2] = {(uint64_t)K / 16, (uint64_t)rec_stride};
  const uint32_t box[3] = {16, 128, 1};
  return encode_map(m, base, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// The four weight maps of one FP4 record range (gate/up codes and scales,
// down codes and scales), record layout gate codes | up codes | gate scales |
// up scales | down codes | down scales.
struct Fp4Maps {
  CUtensorMap gu_c, gu_s, dn_c, dn_s;
};
static moe_status map_fp4_layer(Fp4Maps* m, const uint8_t* base, int n, int H, int I, int64_t S) {
  const int64_t HI = (int64_t)H * I;
  if (moe_status e = map_fp4_codes(&m->gu_c, base, n, 2 * I, H, S)) return e;
  if (moe_status e = map_fp4_scales(&m->gu_s, base + HI, n, 2 * I, H, S)) return e;
  if (moe_status e = map_fp4_codes(&m->dn_c, base + HI + HI / 8, n, H, I, S)) return e;
  return map_fp4_scales(&m->dn_s, base + HI + HI / 8 + HI / 2, n, H, I, S);
}

// FP4 x FP4 maps: packed codes with 128-byte boxes (one 256-element K stage)
// in the 128-byte swizzle the MMA reads, block scales with 16-byte boxes.
// Activations [rows][K/2] and [rows][K/16], boxes of 128 rows; weights
// [n][rows][K/2] and [n][rows][K/16], boxes of 64 rows.
static moe_status map_act_codes(CUtensorMap* m, const void* base, int64_t rows, int K) {
  const uint64_t dims[2] = {(uint64_t)K / 2, (uint64_t)rows}, strides[1] = {(uint64_t)K / 2};
  const uint32_t box[2] = {128, 128};
  return encode_map(m, base, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_128B);
}
static moe_status map_act_scales(CUtensorMap* m, const void* base, int64_t rows, int K) {
  const uint64_t dims[2] = {(uint64_t)K / 16, (uint64_t)rows}, strides[1] = {(uint64_t)K / 16};
  const uint32_t box[2] = {16, 128};
  return encode_map(m, base, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_NONE);
}
static moe_status map_w_codes64(CUtensorMap* m, const void* base, int n, int rows, int K, int64_t rec_stride) {
  const uint64_t dims[3] = {(uint64_t)K / 2, (uint64_t)rows, (uint64_t)n};
  const uint64_t strides[2] = {(uint64_t)K / 2, (uint64_t)rec_stride};
  const uint32_t box[3] = {128, 64, 1};
  return encode_map(m, base, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_128B);
}
static moe_status map_w_scales64(CUtensorMap* m, const void* base, int n, int rows, int K, int64_t rec_stride) {
  const uint64_t dims[3] = {(uint64_t)K / 16, (uint64_t)rows, (uint64_t)n};
  const uint64_t strides[2] = {(uint64_t)K / 16, (uint64_t)rec_stride};
  const uint32_t box[3] = {16, 64, 1};
  return encode_map(m, base, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_NONE);
}
static moe_status map_nvf4_layer(Fp4Maps* m, const uint8_t* base, int n, int H, int I, int64_t S) {
  const int64_t HI = (int64_t)H * I;
  if (moe_status e = map_w_codes64(&m->gu_c, base, n, 2 * I, H, S)) return e;
  if (moe_status e = map_w_scales64(&m->gu_s, base + HI, n, 2 * I, H, S)) return e;
  if (moe_status e = map_w_codes64(&m->dn_c, base + HI + HI / 8, n, H, I, S)) return e;
  return map_w_scales64(&m->dn_s, base + HI + HI / 8 + HI / 2, n, H, I, S);
}

static constexpr int kPrefillChunk = 8192;  // tokens per pass over the layers (the pages' prefill chunk)

static moe_status prefill_staging(moe_cache* c) {
  auto& pf = c->pf;
  if (pf.h_owner) return MOE_OK;
  const int64_t cmax = std::max<int64_t>(1, c->C_max), LE = (int64_t)c->d.L * c->d.E;
  if (cudaHostAlloc((void**)&pf.h_owner, sizeof(int32_t) * cmax, 0) != cudaSuccess ||
      cudaHostAlloc((void**)&pf.h_stamp, sizeof(uint64_t) * cmax, 0) != cudaSuccess ||
      cudaHostAlloc((void**)&pf.h_map, sizeof(int32_t) * LE, 0) != cudaSuccess ||
      cudaHostAlloc((void**)&pf.h_g, sizeof(uint64_t), 0) != cudaSuccess) {
    cudaGetLastError();
    return fail(MOE_ERR_OOM, "pinned prefill staging could not be allocated");
  }
  return MOE_OK;
}

static moe_status prefill_tables(moe_cache* c, int n_steps) {
  auto& pf = c->pf;
  if (!pf.zero) {
    CU_TRY(cudaMalloc(&pf.zero, sizeof(int32_t)));
    CU_TRY(cudaMemset(pf.zero, 0, sizeof(int32_t)));
  }
  if (n_steps <= pf.tab_steps) return MOE_OK;
  if (pf.tab) cudaFree(pf.tab);
  pf.tab = nullptr;
  pf.tab_steps = 0;
  CU_TRY(cudaMalloc(&pf.tab, sizeof(int32_t) * (size_t)n_steps * c->d.E));
  pf.tab_steps = n_steps;
  return MOE_OK;
}

static moe_status prefill_scratch(moe_cache* c, int T) {
  auto& pf = c->pf;
  if (T <= pf.T_cap) return MOE_OK;
  const moe_model_desc& d = c->d;
  for (void* p : {(void*)pf.ids, (void*)pf.cnt, (void*)pf.base, (void*)pf.offsets, (void*)pf.pos, (void*)pf.perm,
                  (void*)pf.w, pf.xp, pf.hp, (void*)pf.op})
    if (p) cudaFree(p);
  pf.T_cap = 0;
  const int64_t n_pairs = (int64_t)T * d.k + (d.has_shared ? T : 0);
  const int G = d.E + (d.has_shared ? 1 : 0);
  const int64_t n_chunks = (n_pairs + 1023) / 1024;
  auto al = [&](void** p, size_t bytes) { return cudaMalloc(p, bytes); };
  if (al((void**)&pf.ids, sizeof(int32_t) * T * d.k) || al((void**)&pf.w, sizeof(float) * T * d.k) ||
      al((void**)&pf.cnt, sizeof(int32_t) * n_chunks * G) || al((void**)&pf.base, sizeof(int32_t) * n_chunks * G) ||
      al((void**)&pf.offsets, sizeof(int32_t) * (G + 1)) || al((void**)&pf.pos, sizeof(int32_t) * n_pairs) ||
      al((void**)&pf.perm, sizeof(int32_t) * n_pairs) || al(&pf.xp, (size_t)n_pairs * d.H * 2) ||
      al(&pf.hp, (size_t)n_pairs * d.I * 2) || al((void**)&pf.op, (size_t)n_pairs * d.H * 4)) {
    cudaGetLastError();
    return fail(MOE_ERR_OOM, "prefill scratch for T=%d does not fit", T);
  }
  for (int b = 0; b < 2; ++b) {
    if (!pf.loaded[b]) CU_TRY(cudaEventCreateWithFlags(&pf.loaded[b], cudaEventDisableTiming));
    if (!pf.consumed[b]) CU_TRY(cudaEventCreateWithFlags(&pf.consumed[b], cudaEventDisableTiming));
  }
  if (!pf.start) CU_TRY(cudaEventCreateWithFlags(&pf.start, cudaEventDisableTiming));
  pf.T_cap = T;
  return MOE_OK;
}

// Victims for one on-demand prefill chunk on the host copy of the state, with
// the decode rule: every expert of the chunk (ascending) gets stamp g + r; a
// miss takes, among slots not holding a hit of the chunk, the empty slots
// first (lowest index) then the oldest stamps.  Returns (slot, is_miss) per
// expert and logs the events.
static void host_access(moe_cache* c, int layer, const std::vector<int>& chunk, int32_t* owner, uint64_t* stamp,
                        int32_t* map, uint64_t* g, std::vector<std::pair<int32_t, bool>>* out) {
  const int64_t E = c->d.E, C = c->C;
  std::vector<char> hit_slot(C, 0);
  int n_miss = 0;
  for (int e : chunk) {
    const int32_t s = map[layer * E + e];
    if (s >= 0) hit_slot[s] = 1; else ++n_miss;
  }
  std::vector<int64_t> victims;
  if (n_miss > 0) {
    std::vector<std::pair<std::pair<int, uint64_t>, int64_t>> cand;
    cand.reserve(C);
    for (int64_t s = 0; s < C; ++s) {
      if (hit_slot[s]) continue;
      cand.push_back(owner[s] < 0 ? std::make_pair(std::make_pair(0, (uint64_t)s), s)
                                  : std::make_pair(std::make_pair(1, stamp[s]), s));
    }
    std::partial_sort(cand.begin(), cand.begin() + n_miss, cand.end());
    for (int i = 0; i < n_miss; ++i) victims.push_back(cand[i].second);
  }
  out->clear();
  int mi = 0;
  for (size_t r = 0; r < chunk.size(); ++r) {
    const int32_t key = (int32_t)(layer * E + chunk[r]);
    int32_t s = map[key], evicted = -1;
    const bool miss = s < 0;
    if (miss) {
      s = (int32_t)victims[mi++];
      evicted = owner[s];
      if (evicted >= 0) map[evicted] = -1;
      owner[s] = key;
      map[key] = s;
    }
    stamp[s] = *g + r;
    out->push_back({s, miss});
    if (c->tracing) {
      moe_event ev{};
      ev.call = c->call_index;
      ev.layer = layer;
      ev.expert = chunk[r];
      ev.kind = miss ? MOE_EV_MISS : MOE_EV_HIT;
      ev.slot = s;
      ev.evicted_key = evicted;
      c->trace.push_back(ev);
    }
  }
  *g += chunk.size();
  c->call_index += 1;
}

extern "C" moe_status moe_prefill_stream_ex(moe_cache_t c, int32_t layer_begin, int32_t layer_end, const void* x,
                                            const float* logits, int32_t T, void* y, void* stream,
                                            const moe_prefill_aux* aux) {
  g_err.clear();
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cache is NULL");
  const moe_model_desc& d = c->d;
  if (d.wdtype != MOE_BF16 && d.wdtype != MOE_FP4) return fail(MOE_ERR_INVALID_ARG, "prefill needs a bf16 or FP4 model");
  if (layer_begin < 0 || layer_end > d.L || layer_begin >= layer_end)
    return fail(MOE_ERR_INVALID_ARG, "layer range [%d, %d) invalid", layer_begin, layer_end);
  if (T < 1 || (int64_t)T * d.k > (int64_t)1 << 30) return fail(MOE_ERR_INVALID_ARG, "T=%d invalid", T);
  if (!x || !logits || !y) return fail(MOE_ERR_INVALID_ARG, "x, logits and y must be device pointers");
  if (d.I % 128 || d.H % 256) return fail(MOE_ERR_INVALID_ARG, "prefill needs I % 128 == 0 and H % 256 == 0");
  const int64_t E = d.E;
  if (c->C < 1) return fail(MOE_ERR_CAPACITY, "prefill needs at least one cache slot");
  // two full-layer buffers when the pool holds them, else on demand
  const bool on_demand = c->C < 2 * E;
  const int Tc = std::min<int>(T, kPrefillChunk), n_chunks = (T + kPrefillChunk - 1) / kPrefillChunk;
  if (aux && n_chunks > 1 && (aux->perm || aux->offsets || aux->slots))
    return fail(MOE_ERR_INVALID_ARG, "aux perm, offsets and slots need T <= %d", kPrefillChunk);
  cudaStream_t s = (cudaStream_t)stream;
  if (*(volatile int*)c->h_err != 0) return recover_after_timeout(c, s);
  if (moe_status st = prefill_scratch(c, Tc)) return st;
  auto& pf = c->pf;
  if (moe_status e = drain_inflight(c, 0)) return e;
  if (moe_status e = follow_stream(c, s)) return e;

  const int H = d.H, I = d.I, k = d.k, sh = d.has_shared;
  const int n_layers = layer_end - layer_begin, n_steps = n_chunks * n_layers;
  const int64_t S = c->S, C = c->C, LE = (int64_t)d.L * E;
  const int64_t buf0 = C - 2 * E;  // buffers: slots [C-2E, C-E) and [C-E, C)
  uint8_t* slots = (uint8_t*)c->slots.base;

  // ---- the cache's bookkeeping for the whole call, on a host copy of the
  // state after every earlier call of this cache
  CU_TRY(cudaStreamSynchronize(s));
  CU_TRY(cudaStreamSynchronize(c->copy));
  if (moe_status e = prefill_staging(c)) return e;
  int32_t* owner = pf.h_owner;
  uint64_t* stamp = pf.h_stamp;
  int32_t* map = pf.h_map;
  CU_TRY(cudaMemcpy(owner, c->d_owner, sizeof(int32_t) * C, cudaMemcpyDeviceToHost));
  CU_TRY(cudaMemcpy(stamp, c->d_stamp, sizeof(uint64_t) * C, cudaMemcpyDeviceToHost));
  CU_TRY(cudaMemcpy(map, c->d_map, sizeof(int32_t) * LE, cudaMemcpyDeviceToHost));
  CU_TRY(cudaMemcpy(pf.h_g, c->d_g, sizeof(uint64_t), cudaMemcpyDeviceToHost));
  if (moe_status e2 = prefill_tables(c, on_demand ? 1 : n_steps)) return e2;

  // the double-buffered plan (the rule of the FreeToken write-up's full-layer
  // double buffering): the buffers are carved out, then per step (chunk,
  // layer) each expert is read in place if resident, else streamed into its
  // buffer slot; the buffer contents stay cached afterwards to seed decode
  std::vector<int32_t> tab;
  std::vector<std::vector<std::pair<int, int>>> runs;  // streamed expert ranges [e0, e1) per step
  std::vector<char> wait_prev;
  int64_t streamed = 0, in_place = 0;
  if (!on_demand) {
    for (int64_t sl = buf0; sl < C; ++sl) {
      const int32_t key = owner[sl];
      if (key < 0) continue;
      if (c->tracing) {
        moe_event ev{};
        ev.call = c->call_index;
        ev.layer = key / (int32_t)E;
        ev.expert = key % (int32_t)E;
        ev.kind = MOE_EV_PREFILL_EVICT;
        ev.slot = (int32_t)sl;
        ev.evicted_key = key;
        c->trace.push_back(ev);
      }
      map[key] = -1;
      owner[sl] = -1;
      stamp[sl] = 0;
    }
    tab.resize((size_t)n_steps * E);
    runs.resize(n_steps);
    wait_prev.assign(n_steps, 0);
    uint64_t g = *pf.h_g;
    for (int i = 0; i < n_steps; ++i) {
      const int l = layer_begin + i % n_layers, b = i & 1;
      int run0 = -1;
      for (int e = 0; e < (int)E; ++e) {
        const int32_t key = (int32_t)(l * E + e);
        int64_t sl = map[key];
        if (sl < 0) {
          sl = buf0 + b * E + e;
          if (owner[sl] >= 0) map[owner[sl]] = -1;
          owner[sl] = key;
          map[key] = (int32_t)sl;
          ++streamed;
          if (run0 < 0) run0 = e;
        } else {
          ++in_place;
          if (run0 >= 0) {
            runs[i].push_back({run0, e});
            run0 = -1;
          }
        }
        stamp[sl] = g + (uint64_t)e;
        tab[(size_t)i * E + e] = (int32_t)sl;
      }
      if (run0 >= 0) runs[i].push_back({run0, (int)E});
      g += (uint64_t)E;
      // the copy of step i overwrites buffer slots that step i-1 may still read
      if (i > 0)
        for (auto [e0, e1] : runs[i])
          for (int e = 0; e < (int)E && !wait_prev[i]; ++e) {
            const int32_t r = tab[(size_t)(i - 1) * E + e];
            if (r >= buf0 + b * E + e0 && r < buf0 + b * E + e1) wait_prev[i] = 1;
          }
    }
    *pf.h_g = g;
    CU_TRY(cudaMemcpyAsync(pf.tab, tab.data(), sizeof(int32_t) * tab.size(), cudaMemcpyHostToDevice, s));
  }

  CU_TRY(cudaEventRecord(pf.start, s));
  CU_TRY(cudaStreamWaitEvent(c->copy, pf.start, 0));
  const int np_c = Tc * k + (sh ? Tc : 0);
  // FP4 x FP4: the gathered rows and the SwiGLU output as codes then block
  // scales in the same buffers
  const bool w4a4 = d.wdtype == MOE_FP4 && c->prefill_prec == MOE_PREFILL_W4A4;
  uint8_t* xq_c = (uint8_t*)pf.xp;
  uint8_t* xq_s = xq_c + (int64_t)np_c * H / 2;
  uint8_t* hq_c = (uint8_t*)pf.hp;
  uint8_t* hq_s = hq_c + (int64_t)np_c * I / 2;
  CUtensorMap map_xp, map_hp, map_xs, map_hs;
  if (w4a4) {
    if (moe_status e = map_act_codes(&map_xp, xq_c, np_c, H)) return e;
    if (moe_status e = map_act_scales(&map_xs, xq_s, np_c, H)) return e;
    if (moe_status e = map_act_codes(&map_hp, hq_c, np_c, I)) return e;
    if (moe_status e = map_act_scales(&map_hs, hq_s, np_c, I)) return e;
  } else {
    if (moe_status e = map_rows(&map_xp, pf.xp, np_c, H)) return e;
    if (moe_status e = map_rows(&map_hp, pf.hp, np_c, I)) return e;
  }
  // weight maps over the whole slot pool (group e reads record tab[e]) and
  // over the shared expert's record of each layer
  Fp4Maps pool_fp4{}, sh_fp4{};
  CUtensorMap bgu{}, bdn{}, bsgu{}, bsdn{};
  if (w4a4) {
    if (moe_status e = map_nvf4_layer(&pool_fp4, slots, (int)C, H, I, S)) return e;
  } else if (d.wdtype == MOE_FP4) {
    if (moe_status e = map_fp4_layer(&pool_fp4, slots, (int)C, H, I, S)) return e;
  } else {
    if (moe_status e = map_weights(&bgu, slots, (int)C, 2 * I, H, S)) return e;
    if (moe_status e = map_weights(&bdn, slots + (int64_t)4 * H * I, (int)C, H, I, S)) return e;
  }
  auto timed = [&](cudaStream_t on, int kind, double flop) -> std::pair<cudaEvent_t, cudaEvent_t> {
    if (!c->profiling) return {nullptr, nullptr};
    cudaEvent_t a = take_event(c), b = take_event(c);
    cudaEventRecord(a, on);
    pf.timed.push_back({a, b, kind, flop});
    return {a, b};
  };
  auto done = [&](std::pair<cudaEvent_t, cudaEvent_t> ev, cudaStream_t on) {
    if (ev.second) cudaEventRecord(ev.second, on);
  };
  // routing, grouping and gather of one step (they need no weights)
  auto front = [&](int li, int t0, int Tn, int n_pairs) -> moe_status {
    const float* lg = logits + ((int64_t)li * T + t0) * E;
    const uint8_t* xl = (const uint8_t*)x + ((int64_t)li * T + t0) * H * 2;
    CU_TRY(prefill_route(lg, Tn, (int)E, k, pf.ids, pf.w, s));
    CU_TRY(prefill_group(pf.ids, Tn, k, (int)E, sh, pf.cnt, pf.base, pf.offsets, pf.pos, pf.perm, s));
    if (w4a4)
      CU_TRY(prefill_gather_quant(xl, Tn, k, H, n_pairs, pf.perm, xq_c, xq_s, s));
    else
      CU_TRY(prefill_gather(xl, Tn, k, H, n_pairs, pf.perm, pf.xp, d.wdtype == MOE_FP4, s));  // FP4: f16 rows
    if (aux) {
      const int64_t at = ((int64_t)li * T + t0) * k, Tk = (int64_t)Tn * k;
      if (aux->ids) CU_TRY(cudaMemcpyAsync(aux->ids + at, pf.ids, sizeof(int32_t) * Tk, cudaMemcpyDeviceToDevice, s));
      if (aux->weights)
        CU_TRY(cudaMemcpyAsync(aux->weights + at, pf.w, sizeof(float) * Tk, cudaMemcpyDeviceToDevice, s));
      if (aux->perm)
        CU_TRY(cudaMemcpyAsync(aux->perm + (int64_t)li * Tk, pf.perm, sizeof(int32_t) * Tk, cudaMemcpyDeviceToDevice,
                               s));
      if (aux->offsets)
        CU_TRY(cudaMemcpyAsync(aux->offsets + (int64_t)li * (E + 1), pf.offsets, sizeof(int32_t) * (E + 1),
                               cudaMemcpyDeviceToDevice, s));
    }
    return MOE_OK;
  };
  // the expert GEMMs of the groups whose table entry is a slot (and, with
  // shared, the shared expert of layer l)
  auto gemms = [&](const int32_t* tab_i, int l, int n_pairs, bool shared) -> moe_status {
    const uint8_t* srec = shared ? c->shared_dev + (int64_t)l * S : nullptr;
    if (w4a4) {  // block-scaled FP4 x FP4 on the codes and scales where each expert sits
      if (shared)
        if (moe_status e = map_nvf4_layer(&sh_fp4, srec, 1, H, I, S)) return e;
      CU_TRY(prefill_gemm_gate_up_nvf4(map_xp, map_xs, pool_fp4.gu_c, pool_fp4.gu_s, pf.offsets, tab_i, (int)E,
                                       n_pairs, H, I, hq_c, hq_s, c->d_err, s));
      if (shared)
        CU_TRY(prefill_gemm_gate_up_nvf4(map_xp, map_xs, sh_fp4.gu_c, sh_fp4.gu_s, pf.offsets + E, pf.zero, 1,
                                         n_pairs, H, I, hq_c, hq_s, c->d_err, s));
      CU_TRY(prefill_gemm_down_nvf4(map_hp, map_hs, pool_fp4.dn_c, pool_fp4.dn_s, pf.offsets, tab_i, (int)E, n_pairs,
                                    H, I, pf.op, c->d_err, s));
      if (shared)
        CU_TRY(prefill_gemm_down_nvf4(map_hp, map_hs, sh_fp4.dn_c, sh_fp4.dn_s, pf.offsets + E, pf.zero, 1, n_pairs,
                                      H, I, pf.op, c->d_err, s));
    } else if (d.wdtype == MOE_FP4) {  // the GEMMs read the FP4 codes and scales where each expert sits
      if (shared)
        if (moe_status e = map_fp4_layer(&sh_fp4, srec, 1, H, I, S)) return e;
      CU_TRY(prefill_gemm_gate_up_fp4(map_xp, pool_fp4.gu_c, pool_fp4.gu_s, pf.offsets, tab_i, (int)E, n_pairs, H, I,
                                      pf.hp, c->d_err, s));
      if (shared)
        CU_TRY(prefill_gemm_gate_up_fp4(map_xp, sh_fp4.gu_c, sh_fp4.gu_s, pf.offsets + E, pf.zero, 1, n_pairs, H, I,
                                        pf.hp, c->d_err, s));
      CU_TRY(prefill_gemm_down_fp4(map_hp, pool_fp4.dn_c, pool_fp4.dn_s, pf.offsets, tab_i, (int)E, n_pairs, H, I,
                                   pf.op, c->d_err, s));
      if (shared)
        CU_TRY(prefill_gemm_down_fp4(map_hp, sh_fp4.dn_c, sh_fp4.dn_s, pf.offsets + E, pf.zero, 1, n_pairs, H, I,
                                     pf.op, c->d_err, s));
    } else {
      if (shared) {
        if (moe_status e = map_weights(&bsgu, srec, 1, 2 * I, H, S)) return e;
        if (moe_status e = map_weights(&bsdn, srec + (int64_t)4 * H * I, 1, H, I, S)) return e;
      }
      CU_TRY(prefill_gemm_gate_up(map_xp, bgu, pf.offsets, tab_i, (int)E, n_pairs, H, I, pf.hp, c->d_err, s));
      if (shared)
        CU_TRY(prefill_gemm_gate_up(map_xp, bsgu, pf.offsets + E, pf.zero, 1, n_pairs, H, I, pf.hp, c->d_err, s));
      CU_TRY(prefill_gemm_down(map_hp, bdn, pf.offsets, tab_i, (int)E, n_pairs, H, I, pf.op, c->d_err, s));
      if (shared)
        CU_TRY(prefill_gemm_down(map_hp, bsdn, pf.offsets + E, pf.zero, 1, n_pairs, H, I, pf.op, c->d_err, s));
    }
    return MOE_OK;
  };
  const auto whole = timed(s, 0, 0.0);

  if (!on_demand) {
    for (int i = 0; i < n_steps; ++i) {
      const int li = i % n_layers, ch = i / n_layers, l = layer_begin + li, b = i & 1;
      const int t0 = ch * kPrefillChunk, Tn = std::min(Tc, T - t0);
      const int n_pairs = Tn * k + (sh ? Tn : 0);
      // stream the layer's missing experts into buffer b once the computes that
      // read those slots have finished
      if (i >= 2) CU_TRY(cudaStreamWaitEvent(c->copy, pf.consumed[b], 0));
      if (wait_prev[i]) CU_TRY(cudaStreamWaitEvent(c->copy, pf.consumed[b ^ 1], 0));
      const auto cp = timed(c->copy, 1, 0.0);
      for (auto [e0, e1] : runs[i])
        CU_TRY(cudaMemcpyAsync(slots + (buf0 + b * E + e0) * S, c->host_pool + ((int64_t)l * E + e0) * S,
                               (int64_t)(e1 - e0) * S, cudaMemcpyHostToDevice, c->copy));
      done(cp, c->copy);
      CU_TRY(cudaEventRecord(pf.loaded[b], c->copy));
      if (moe_status e = front(li, t0, Tn, n_pairs)) return e;
      const int32_t* tab_i = pf.tab + (size_t)i * E;
      if (aux && aux->slots)
        CU_TRY(cudaMemcpyAsync(aux->slots + (int64_t)li * E, tab_i, sizeof(int32_t) * E, cudaMemcpyDeviceToDevice,
                               s));
      CU_TRY(cudaStreamWaitEvent(s, pf.loaded[b], 0));
      const auto comp = timed(s, 2, 0.0);
      const auto gm = timed(s, 3, 2.0 * n_pairs * (2.0 * I * H) + 2.0 * n_pairs * ((double)H * I));
      if (moe_status e = gemms(tab_i, l, n_pairs, sh)) return e;
      done(gm, s);
      CU_TRY(cudaEventRecord(pf.consumed[b], s));  // buffer b may be refilled
      CU_TRY(prefill_combine(pf.op, pf.pos, pf.w, Tn, k, H, sh, (uint8_t*)y + ((int64_t)li * T + t0) * H * 2, s));
      done(comp, s);
    }
  } else {
    // on demand: per step the layer's distinct routed experts, in chunks of
    // at most C, each accessed like one decode call; a chunk's copies wait
    // until the previous chunk's GEMMs no longer read the slots
    std::vector<int32_t> h_off(E + 1), tab1(E);
    std::vector<std::pair<int32_t, bool>> acc;
    uint64_t g = *pf.h_g;
    for (int i = 0; i < n_steps; ++i) {
      const int li = i % n_layers, ch = i / n_layers, l = layer_begin + li;
      const int t0 = ch * kPrefillChunk, Tn = std::min(Tc, T - t0);
      const int n_pairs = Tn * k + (sh ? Tn : 0);
      if (moe_status e = front(li, t0, Tn, n_pairs)) return e;
      CU_TRY(cudaMemcpyAsync(h_off.data(), pf.offsets, sizeof(int32_t) * (E + 1), cudaMemcpyDeviceToHost, s));
      CU_TRY(cudaStreamSynchronize(s));
      std::vector<int> U;
      for (int e = 0; e < (int)E; ++e)
        if (h_off[e + 1] > h_off[e]) U.push_back(e);
      std::vector<int32_t> layer_slots(E, -1);
      const auto comp = timed(s, 2, 0.0);
      for (size_t c0 = 0; c0 < U.size() || (c0 == 0 && sh); c0 += (size_t)C) {
        std::vector<int> chunk(U.begin() + std::min(c0, U.size()), U.begin() + std::min(c0 + (size_t)C, U.size()));
        host_access(c, l, chunk, owner, stamp, map, &g, &acc);
        std::fill(tab1.begin(), tab1.end(), -1);
        CU_TRY(cudaStreamWaitEvent(c->copy, pf.consumed[0], 0));  // the previous chunk's GEMMs are done
        const auto cp = timed(c->copy, 1, 0.0);
        for (size_t r = 0; r < chunk.size(); ++r) {
          const auto [sl, miss] = acc[r];
          tab1[chunk[r]] = sl;
          layer_slots[chunk[r]] = sl;
          if (miss) {
            CU_TRY(cudaMemcpyAsync(slots + (int64_t)sl * S, c->host_pool + ((int64_t)l * E + chunk[r]) * S, S,
                                   cudaMemcpyHostToDevice, c->copy));
            ++streamed;
          } else {
            ++in_place;
          }
        }
        done(cp, c->copy);
        CU_TRY(cudaEventRecord(pf.loaded[0], c->copy));
        CU_TRY(cudaMemcpyAsync(pf.tab, tab1.data(), sizeof(int32_t) * E, cudaMemcpyHostToDevice, s));
        CU_TRY(cudaStreamWaitEvent(s, pf.loaded[0], 0));
        int rows = 0;
        for (int e : chunk) rows += h_off[e + 1] - h_off[e];
        const int shared_rows = c0 == 0 && sh ? Tn : 0;
        const auto gm = timed(s, 3, 2.0 * (rows + shared_rows) * (3.0 * I * H));
        if (moe_status e = gemms(pf.tab, l, n_pairs, c0 == 0 && sh)) return e;
        done(gm, s);
        CU_TRY(cudaEventRecord(pf.consumed[0], s));
        if (U.empty()) break;
      }
      if (aux && aux->slots)
        CU_TRY(cudaMemcpyAsync(aux->slots + (int64_t)li * E, layer_slots.data(), sizeof(int32_t) * E,
                               cudaMemcpyHostToDevice, s));
      CU_TRY(prefill_combine(pf.op, pf.pos, pf.w, Tn, k, H, sh, (uint8_t*)y + ((int64_t)li * T + t0) * H * 2, s));
      done(comp, s);
    }
    *pf.h_g = g;
  }
  done(whole, s);
  // the cache after prefill: what the buffers (or the chunks) left stays cached
  CU_TRY(cudaMemcpyAsync(c->d_owner, owner, sizeof(int32_t) * C, cudaMemcpyHostToDevice, s));
  CU_TRY(cudaMemcpyAsync(c->d_stamp, stamp, sizeof(uint64_t) * C, cudaMemcpyHostToDevice, s));
  CU_TRY(cudaMemcpyAsync(c->d_map, map, sizeof(int32_t) * LE, cudaMemcpyHostToDevice, s));
  CU_TRY(cudaMemcpyAsync(c->d_g, pf.h_g, sizeof(uint64_t), cudaMemcpyHostToDevice, s));
  CU_TRY(cudaMemsetAsync(c->d_oldest_n, 0xFF, sizeof(int), s));
  c->st.prefill_layers += n_layers;
  c->st.prefill_tokens += (int64_t)T * n_layers;
  c->st.prefill_records_streamed += streamed;
  c->st.prefill_records_in_place += in_place;
  return MOE_OK;
}

extern "C" moe_status moe_prefill_stream(moe_cache_t c, int32_t layer_begin, int32_t layer_end, const void* x,
                                         const float* logits, int32_t T, void* y, void* stream) {
  return moe_prefill_stream_ex(c, layer_begin, layer_end, x, logits, T, y, stream, nullptr);
}
