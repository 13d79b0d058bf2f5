// Grouped bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), fed
// by TMA, for the prefill-size expert FFN.  The weight maps cover a range of
// records (the whole slot pool); group e's weights are record slot_of[e].
//
// FreeToken write-up, "전층 이중 버퍼링": in prefill a layer's routed tokens
// cover almost every expert, so each expert's FFN is a dense contraction over
// the ~T*k/E tokens routed to it.
//
// One CTA computes one 128 x 256 output tile of one expert:
//   rows    = 128 consecutive (token, rank) pairs of the expert in the grouped
//             activation matrix A [rows][K] (bf16, K-major), rows beyond the
//             expert's group are computed but never stored;
//   columns = 256 rows of the expert's weight matrix B [E][N][K] (bf16,
//             K-major), loaded as two 128-row boxes (b_row0, b_row1) so the
//             gate/up GEMM can place gate rows j.. and up rows I+j.. side by side.
// Warp roles (192 threads): warp 0 issues TMA loads into a 4-stage ring of
// 48 KB stages (128B swizzle), warp 1 owns TMEM (256 fp32 columns) and issues
// tcgen05.mma (M=128, N=256, K=16) from one elected thread, warps 2..5 read
// the accumulator back with tcgen05.ld (each warp its 32 TMEM lanes) and run
// the epilogue.  Every mbarrier wait is bounded: on time-out the kernel
// records MOE_ERR_TIMEOUT, stops issuing work and still frees its TMEM.
#pragma once
#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "expert_math.cuh"

namespace moe {
namespace tc {

constexpr int kBM = 128, kBN = 256, kBK = 64;  // tile; kBK bf16 = 128 bytes = one swizzle row
constexpr int kStages = 4;
constexpr int kAStage = kBM * kBK * 2;          // 16 KB
constexpr int kBStage = kBN * kBK * 2;          // 32 KB
constexpr int kStageBytes = kAStage + kBStage;  // 48 KB
constexpr int kThreads = 192;
constexpr int kTmemCols = 256;
constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;

// ---- PTX wrappers (smem_u32 and the mbarrier helpers are in common.cuh) ----------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// K-major operand tile in shared memory written by TMA with 128-byte swizzle:
// rows of 128 bytes, 8-row (1024-byte) swizzle atoms.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);       // start address
  d |= (uint64_t)0 << 16;                         // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;               // stride byte offset: one 8-row atom
  d |= (uint64_t)1 << 46;                         // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                         // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: bf16 x bf16 -> f32, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4)                  // D format f32
         | (1u << 7)                // A format bf16
         | (1u << 10)               // B format bf16
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// ---- tile scheduling -----------------------------------------------------------
// Work item of one CTA: expert e, rows [row0, row0 + 128) of A (clipped to
// row_end for stores), output column block nb.
struct Tile {
  int e, row0, row_end, nb;
};

// Tiles are enumerated expert-major, then row block, then column block; the
// grid is sized for the worst case and CTAs past the last tile exit.  Groups
// whose slot is negative are skipped (not part of this launch).
__device__ __forceinline__ bool find_tile(const int32_t* offsets, const int32_t* slot_of, int E, int nblocks_n,
                                          int cta, Tile* t) {
  int base = 0;
  for (int e = 0; e < E; ++e) {
    const int n = slot_of[e] < 0 ? 0 : offsets[e + 1] - offsets[e];
    const int mt = (n + kBM - 1) / kBM;
    const int cnt = mt * nblocks_n;
    if (cta < base + cnt) {
      const int r = cta - base;
      t->e = e;
      t->row0 = offsets[e] + (r / nblocks_n) * kBM;
      t->row_end = offsets[e + 1];
      t->nb = r % nblocks_n;
      return true;
    }
    base += cnt;
  }
  return false;
}

// Epilogues --------------------------------------------------------------------
// gate/up: columns [0,128) gate, [128,256) up of output block nb -> bf16 h.
template <typename OutT = __nv_bfloat16>
struct EpiSwiGLU {
  OutT* h;  // [rows][I], bf16 or f16
  int I;
  __device__ void operator()(uint32_t tmem, int row, bool valid, int nb) const {
    for (int c = 0; c < 128; c += 16) {
      float g[16], u[16];
      tmem_ld16(tmem + c, g);
      tmem_ld16(tmem + 128 + c, u);
      if (!valid) continue;
      uint32_t packed[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float h0 = g[2 * i] / (1.0f + expf(-g[2 * i])) * u[2 * i];
        const float h1 = g[2 * i + 1] / (1.0f + expf(-g[2 * i + 1])) * u[2 * i + 1];
        if constexpr (sizeof(OutT) == 2 && std::is_same<OutT, __half>::value) {
          __half2 p2 = __floats2half2_rn(h0, h1);
          packed[i] = *reinterpret_cast<uint32_t*>(&p2);
        } else {
          __nv_bfloat162 p2 = __floats2bfloat162_rn(h0, h1);
          packed[i] = *reinterpret_cast<uint32_t*>(&p2);
        }
      }
      uint4* dst = reinterpret_cast<uint4*>(h + (int64_t)row * I + (int64_t)nb * 128 + c);
      dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    }
  }
};

// down: 256 fp32 columns of output block nb -> o [rows][N].
struct EpiStoreF32 {
  float* o;
  int N;
  __device__ void operator()(uint32_t tmem, int row, bool valid, int nb) const {
    for (int c = 0; c < 256; c += 16) {
      float v[16];
      tmem_ld16(tmem + c, v);
      if (!valid) continue;
      float4* dst = reinterpret_cast<float4*>(o + (int64_t)row * N + (int64_t)nb * 256 + c);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
};

// A: 2D map over [rows][K]; B: 3D map over [E][Nrows][K].  b_row(nb, half)
// gives the first weight row of each 128-row half of the 256-column block.
template <typename Epi, typename BRow>
__device__ void grouped_gemm_cta(const CUtensorMap* map_a, const CUtensorMap* map_b, const int32_t* offsets,
                                 const int32_t* slot_of, int E, int nblocks_n, int K, Epi epi, BRow b_row, int* err) {
  extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  __shared__ Tile s_tile;
  __shared__ int s_has;
  __shared__ int s_fail;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    s_has = find_tile(offsets, slot_of, E, nblocks_n, blockIdx.x, &s_tile) ? 1 : 0;
    s_fail = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (!s_has) return;
  const Tile t = s_tile;
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ksteps = K / kBK;

  if (warp == 0 && lane == 0) {
    // TMA producer; the weights of group t.e sit in record slot_of[t.e]
    const int rec = slot_of[t.e];
    for (int ks = 0; ks < ksteps; ++ks) {
      const int s = ks % kStages;
      if (ks >= kStages && !mbar_wait(&empty[s], ((ks / kStages) - 1) & 1)) { s_fail = 1; break; }
      if (s_fail) break;
      uint8_t* a_dst = smem + s * kStageBytes;
      uint8_t* b_dst = a_dst + kAStage;
      mbar_expect_tx(&full[s], kStageBytes);
      tma_load_2d(a_dst, map_a, &full[s], ks * kBK, t.row0);
      tma_load_3d(b_dst, map_b, &full[s], ks * kBK, b_row(t.nb, 0), rec);
      tma_load_3d(b_dst + kBStage / 2, map_b, &full[s], ks * kBK, b_row(t.nb, 1), rec);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    constexpr uint32_t idesc = idesc_bf16(kBM, kBN);
    for (int ks = 0; ks < ksteps; ++ks) {
      const int s = ks % kStages;
      if (s_fail || !mbar_wait(&full[s], (ks / kStages) & 1)) { s_fail = 1; break; }
      tc_fence_after();
      const uint32_t a0 = smem_u32(smem + s * kStageBytes);
      const uint32_t b0 = a0 + kAStage;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        mma_bf16(tmem, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), idesc, (ks | kk) != 0);
      mma_commit(&empty[s]);
    }
    mma_commit(acc_full);
  } else if (warp >= 2) {
    // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31, i.e. tile rows
    const int q = warp & 3;
    const bool ok = mbar_wait(acc_full, 0, 4000000000ull);
    tc_fence_after();
    const int r = q * 32 + lane;
    const int row = t.row0 + r;
    if (ok && !s_fail) epi(tmem + ((uint32_t)(q * 32) << 16), row, row < t.row_end, t.nb);
    if (!ok) s_fail = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (s_fail && threadIdx.x == 0) atomicExch(err, MOE_ERR_TIMEOUT);
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---- FP4-reading variant, persistent ------------------------------------------------
// Same tiles and epilogues, but B is read as FP4 and the GEMM runs on f16
// operands: per K-step of 64 elements TMA brings the A tile (f16, 128-byte
// swizzle), the weight rows' e2m1 codes (256 rows x 32 bytes) and the 16-byte
// box of e4m3 scales that covers them (reloaded for 4 consecutive K-steps, an
// L2 hit after the first).  Converter warps expand the codes into the f16 B
// tile in the 128-byte-swizzled K-major layout the MMA reads (chunk j of row r
// at position j ^ (r & 7) of the row): cvt.rn.f16x2.e2m1x2 then one f16x2
// multiply by the block scale, exact (the product has at most 3 + 4
// significant bits and its exponent stays within the f16 normal range), so the
// GEMM equals the one on the dequantised weights.  The weight stream from DRAM
// is 0.5625 byte per element instead of 2.
//
// One CTA per SM walks the tile list (tile t, t + gridDim.x, ...; tiles are
// enumerated expert-major, then row block, then column block, from a table of
// per-expert tile counts built in shared memory at the start).  Every ring runs
// continuously across tiles, and the accumulator is double-buffered in TMEM
// (2 x 256 columns): the epilogue of tile i overlaps the mainloop of tile i+1.
// Rings: kRaw stages of (A 16 KB | codes 8 KB | scales 4 KB) filled by TMA and
// two converted B buffers (32 KB each); barriers full/empty per raw stage,
// conv/bfree per B buffer, acc_full/acc_empty per accumulator.  Warps: 0 TMA
// producer, 1 MMA issuer (and TMEM owner), 2..17 converters, 18..21 epilogue
// (warp w reads TMEM lanes 32 * (w % 4) .. + 31).  Every wait is bounded and
// also gives up once another role has failed; TMEM is freed on every path.
#ifndef MOE_FP4_RAW_STAGES
#define MOE_FP4_RAW_STAGES 5
#endif
#ifndef MOE_FP4_B_BUFFERS
#define MOE_FP4_B_BUFFERS 2
#endif
#ifndef MOE_FP4_CONV_WARPS
#define MOE_FP4_CONV_WARPS 16
#endif
namespace fp4 {
constexpr int kRaw = MOE_FP4_RAW_STAGES;
constexpr int kBBufs = MOE_FP4_B_BUFFERS;
constexpr int kConvWarps = MOE_FP4_CONV_WARPS;
constexpr int kEpiWarps = 4;
constexpr int kConv0 = 2, kEpi0 = kConv0 + kConvWarps;
constexpr int kThreads = 32 * (kEpi0 + kEpiWarps);
constexpr int kAStage = kBM * kBK * 2;      // 16 KB
constexpr int kBStage = kBN * kBK * 2;      // 32 KB
constexpr int kCodeStage = kBN * kBK / 2;   // 8 KB
constexpr int kScaleStage = kBN * 16;       // 4 KB
constexpr int kRawBytes = kAStage + kCodeStage + kScaleStage;  // 28 KB, 1024-aligned
constexpr uint32_t kTxBytes = kRawBytes;
constexpr int kAccCols = 256;               // one accumulator; two of them fill the TMEM
constexpr int kMaxE = 1024;
constexpr size_t kSmemBytes = (size_t)kBBufs * kBStage + (size_t)kRaw * kRawBytes + 1024 /*align*/ + 256 /*barriers*/;
static_assert(kRawBytes % 1024 == 0 && kBStage % 1024 == 0, "tiles must keep the 1024-byte swizzle alignment");
static_assert(kSmemBytes + 8 * 1024 <= 227 * 1024, "rings must fit the opt-in shared memory");
static_assert((kBN * 8) % (32 * kConvWarps) == 0, "converter warps must split a B tile evenly");
}  // namespace fp4

// kind::f16 instruction descriptor: f16 x f16 -> f32, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4)  // D format f32; A and B format f16 (0)
         | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Eight e2m1 codes (4 bytes, element 2i in the low nibble of byte i) times one
// e4m3 scale (given as f16x2 in both halves) -> eight f16 (exact).
__device__ __forceinline__ uint4 dequant8_f16(uint32_t c4, uint32_t s2) {
  uint32_t o[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    uint32_t h2;
    asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h2) : "r"(c4 >> (8 * b)));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[b]) : "r"(h2), "r"(s2));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}
__device__ __forceinline__ uint32_t e4m3_to_f16x2_both(uint32_t scale_byte) {
  uint32_t s2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2) : "h"((unsigned short)(scale_byte * 0x0101u)));
  return s2;
}

// Bounded wait that also gives up as soon as *fail is set by another role.
__device__ __forceinline__ bool mbar_wait_or(uint64_t* bar, uint32_t parity, const volatile int* fail,
                                             unsigned long long limit_ns = 2000000000ull) {
  const uint32_t a = smem_u32(bar);
  unsigned long long t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 63) == 63) {
      if (*fail) return false;
      const unsigned long long t = globaltimer_ns();
      if (t0 == 0) t0 = t;
      else if (t - t0 > limit_ns) return false;
    }
  }
}

// Tile t of the list: expert e = the last one whose first tile is <= t.
__device__ __forceinline__ Tile tile_of(const int* tile_base, const int32_t* offsets, int E, int nblocks_n, int t) {
  int lo = 0, hi = E;  // tile_base[lo] <= t < tile_base[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_base[mid] <= t) lo = mid; else hi = mid;
  }
  const int r = t - tile_base[lo];
  Tile tl;
  tl.e = lo;
  tl.row0 = offsets[lo] + (r / nblocks_n) * kBM;
  tl.row_end = offsets[lo + 1];
  tl.nb = r % nblocks_n;
  return tl;
}

// A: 2D f16 map over [rows][K]; codes: 3D u8 map over [records][Nrows][K/2]
// (box 32 bytes x 128 rows); scales: 3D u8 map over [records][Nrows][K/16]
// (box 16 x 128); group e's weights are record slot_of[e] (groups with a
// negative slot are not part of this launch).
template <typename Epi, typename BRow>
__device__ void grouped_gemm_fp4_persistent(const CUtensorMap* map_a, const CUtensorMap* map_codes,
                                            const CUtensorMap* map_scales, const int32_t* offsets,
                                            const int32_t* slot_of, int E, int nblocks_n, int K, Epi epi, BRow b_row,
                                            int* err) {
  constexpr int kRaw = fp4::kRaw, kBBufs = fp4::kBBufs, kConvWarps = fp4::kConvWarps, kEpiWarps = fp4::kEpiWarps;
  constexpr int kConv0 = fp4::kConv0, kEpi0 = fp4::kEpi0, kAccCols = fp4::kAccCols, kMaxE = fp4::kMaxE;
  constexpr int kAStage = fp4::kAStage, kBStage = fp4::kBStage, kCodeStage = fp4::kCodeStage;
  constexpr int kScaleStage = fp4::kScaleStage, kRawBytes = fp4::kRawBytes;
  constexpr uint32_t kTxBytes = fp4::kTxBytes;
  extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* btile = smem;                          // kBBufs converted B tiles
  uint8_t* raw = smem + kBBufs * kBStage;         // kRaw stages of A | codes | scales
  uint64_t* full = reinterpret_cast<uint64_t*>(raw + kRaw * kRawBytes);
  uint64_t* empty = full + kRaw;
  uint64_t* conv = empty + kRaw;
  uint64_t* bfree = conv + kBBufs;
  uint64_t* acc_full = bfree + kBBufs;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  __shared__ int tile_base[kMaxE + 1];
  __shared__ int s_scan[33];
  __shared__ volatile int s_fail;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // per-expert tile counts -> first tile of each expert (one block scan)
  int n_tiles;
  {
    int base = 0;
    for (int e0 = 0; e0 < E; e0 += blockDim.x) {
      const int e = e0 + (int)threadIdx.x;
      const int cnt = e < E && slot_of[e] >= 0 ? (offsets[e + 1] - offsets[e] + kBM - 1) / kBM * nblocks_n : 0;
      int tot;
      const int before = block_excl_scan(cnt, s_scan, &tot);
      if (e < E) tile_base[e] = base + before;
      base += tot;
    }
    n_tiles = base;
    if (threadIdx.x == 0) tile_base[E] = base;
  }
  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int i = 0; i < kRaw; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kBBufs; ++i) {
      mbar_init(&conv[i], kConvWarps);
      mbar_init(&bfree[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if ((int)blockIdx.x >= n_tiles) return;
  if (warp == 1) tmem_alloc(tmem_slot, 2 * kAccCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ksteps = K / kBK;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer: A tile, the 256 weight rows' codes, their scale boxes
      int g = 0;  // K-steps issued so far (all tiles)
      for (int t = blockIdx.x; t < n_tiles && !s_fail; t += gridDim.x) {
        const Tile tl = tile_of(tile_base, offsets, E, nblocks_n, t);
        const int rec = slot_of[tl.e];
        for (int ks = 0; ks < ksteps; ++ks, ++g) {
          const int s = g % kRaw;
          if (g >= kRaw && !mbar_wait_or(&empty[s], ((g / kRaw) - 1) & 1, &s_fail)) { s_fail = 1; break; }
          uint8_t* a = raw + s * kRawBytes;
          uint8_t* codes = a + kAStage;
          uint8_t* scales = codes + kCodeStage;
          mbar_expect_tx(&full[s], kTxBytes);
          tma_load_2d(a, map_a, &full[s], ks * kBK, tl.row0);
          tma_load_3d(codes, map_codes, &full[s], ks * (kBK / 2), b_row(tl.nb, 0), rec);
          tma_load_3d(codes + kCodeStage / 2, map_codes, &full[s], ks * (kBK / 2), b_row(tl.nb, 1), rec);
          tma_load_3d(scales, map_scales, &full[s], (ks >> 2) * 16, b_row(tl.nb, 0), rec);
          tma_load_3d(scales + kScaleStage / 2, map_scales, &full[s], (ks >> 2) * 16, b_row(tl.nb, 1), rec);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer: A from the raw stage, B from the converted buffer
      constexpr uint32_t idesc = idesc_f16(kBM, kBN);
      int g = 0, i = 0;  // K-steps and tiles so far
      for (int t = blockIdx.x; t < n_tiles && !s_fail; t += gridDim.x, ++i) {
        const int ab = i & 1;
        if (i >= 2 && !mbar_wait_or(&acc_empty[ab], ((i >> 1) - 1) & 1, &s_fail)) { s_fail = 1; break; }
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(ab * kAccCols);
        for (int ks = 0; ks < ksteps; ++ks, ++g) {
          const int s = g % kRaw, bb = g % kBBufs;
          if (!mbar_wait_or(&conv[bb], (g / kBBufs) & 1, &s_fail)) { s_fail = 1; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(raw + s * kRawBytes);
          const uint32_t b0 = smem_u32(btile + bb * kBStage);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16(acc, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), idesc, (ks | kk) != 0);
          mma_commit(&empty[s]);
          mma_commit(&bfree[bb]);
        }
        if (s_fail) break;
        mma_commit(&acc_full[ab]);
      }
    }
  } else if (warp < kEpi0) {
    // converters: 256 rows x 8 chunks of 8 elements per K-step, 8 per thread
    const int ct = threadIdx.x - 32 * kConv0;
    int g = 0;
    for (int t = blockIdx.x; t < n_tiles && !s_fail; t += gridDim.x) {
      for (int ks = 0; ks < ksteps; ++ks, ++g) {
        const int s = g % kRaw, bb = g % kBBufs;
        if (!mbar_wait_or(&full[s], (g / kRaw) & 1, &s_fail)) { s_fail = 1; break; }
        if (g >= kBBufs && !mbar_wait_or(&bfree[bb], ((g / kBBufs) - 1) & 1, &s_fail)) { s_fail = 1; break; }
        const uint8_t* codes = raw + s * kRawBytes + kAStage;
        const uint8_t* scales = codes + kCodeStage;
        uint8_t* bt = btile + bb * kBStage;
        const int sub = (ks & 3) * 4;  // this K-step's 4 scale bytes in each row's 16-byte box
#pragma unroll
        for (int q8 = 0; q8 < (kBN * 8) / (32 * kConvWarps); ++q8) {
          const int q = ct + 32 * kConvWarps * q8;
          const int r = q >> 3, j = q & 7;
          const uint32_t c4 = *reinterpret_cast<const uint32_t*>(codes + r * 32 + j * 4);
          const uint32_t s2 = e4m3_to_f16x2_both(scales[r * 16 + sub + (j >> 1)]);
          *reinterpret_cast<uint4*>(bt + r * 128 + ((j ^ (r & 7)) << 4)) = dequant8_f16(c4, s2);
        }
        fence_proxy_async_smem();  // generic-proxy writes -> the tensor core's async-proxy reads
        __syncwarp();
        if (lane == 0) mbar_arrive(&conv[bb]);
      }
    }
  } else {
    // epilogue: warp w reads TMEM lanes 32 * (w % 4) .. + 31, i.e. tile rows
    const int q = warp & 3;
    int i = 0;
    for (int t = blockIdx.x; t < n_tiles && !s_fail; t += gridDim.x, ++i) {
      const int ab = i & 1;
      if (!mbar_wait_or(&acc_full[ab], (i >> 1) & 1, &s_fail, 4000000000ull)) { s_fail = 1; break; }
      tc_fence_after();
      const Tile tl = tile_of(tile_base, offsets, E, nblocks_n, t);
      const int row = tl.row0 + q * 32 + lane;
      epi(tmem + (uint32_t)(ab * kAccCols) + ((uint32_t)(q * 32) << 16), row, row < tl.row_end, tl.nb);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (s_fail && threadIdx.x == 0) atomicExch(err, MOE_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kAccCols);
  }
}

}  // namespace tc
}  // namespace moe
