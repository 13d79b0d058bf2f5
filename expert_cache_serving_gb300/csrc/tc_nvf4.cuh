// Grouped FP4 x FP4 GEMM with block scaling on the 5th-generation tensor
// cores (tcgen05.mma kind::mxf4nvf4, scale_vec::4X: e2m1 operands, one e4m3
// scale per 16 elements of K), persistent, fed by TMA.  Used by the prefill
// path when the activations are quantised to the weights' FP4 format.
//
// FreeToken write-up, "전층 이중 버퍼링": a prefill layer activates almost
// every expert, so each expert's FFN is a dense contraction over the
// ~T*k/E (token, rank) pairs routed to it; experimental setup: the experts
// are deployed in MXFP4 / NVFP4.
//
// Tile: 128 pair rows (M) x 128 weight rows (N, loaded as two 64-row boxes so
// the gate/up GEMM places gate rows j.. and up rows I+j.. side by side) x 256
// K elements per pipeline stage (128 bytes of packed codes per row: one
// 128-byte swizzle row).  Per stage TMA brings the A codes (16 KB), the B
// codes (16 KB) and both operands' raw scale boxes (128 rows x 16 bytes
// each); a scale warp rearranges each K=64 step's scales into the 512-byte
// groups tcgen05.cp copies to tensor memory (row r of a 128-row operand at
// lane r % 32 and column r / 32, its four block scales in byte order, the 32
// lanes replicated to all four lane quarters), and the MMA thread issues per
// step two tcgen05.cp (A and B scales) and one MMA (M=128, N=128, K=64).
//
// Tensor memory: two 128-column fp32 accumulators (the epilogue of tile i
// overlaps the mainloop of tile i+1) and a ring of 32 scale columns per
// stage.  Warps: 0 TMA producer, 1 MMA issuer (and TMEM owner), 2 scale
// rearrangement, 3..6 epilogue (warp w reads TMEM lanes 32 * (w % 4) ..).
// Every wait is bounded and gives up once another role has failed; TMEM is
// freed on every path.
#pragma once
#include "nvfp4.cuh"
#include "tc_gemm.cuh"

namespace moe {
namespace tc {
namespace nvf4 {

constexpr int kBM = 128, kBN = 128, kBKBytes = 128;  // 256 FP4 elements of K per stage
constexpr int kStages = 5;
constexpr int kACodes = kBM * kBKBytes;   // 16 KB
constexpr int kBCodes = kBN * kBKBytes;   // 16 KB
constexpr int kARaw = kBM * 16, kBRaw = kBN * 16;  // 2 KB each: 16 scale bytes per row per stage
constexpr int kAtoms = 4 * 512;           // 4 K=64 steps x 128 rows x 4 bytes
constexpr int kStageBytes = kACodes + kBCodes + kARaw + kBRaw + 2 * kAtoms;  // 40 KB
constexpr uint32_t kTxBytes = kACodes + kBCodes + kARaw + kBRaw;
constexpr int kEpiWarps = 4, kEpi0 = 3;
constexpr int kThreads = 32 * (kEpi0 + kEpiWarps);
constexpr int kAccCols = 128, kSfCols = 32, kTmemCols = 512;
constexpr int kMaxE = 1024;
constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
static_assert(kStageBytes % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
static_assert(kSmemBytes + 9 * 1024 <= 227 * 1024, "the ring must fit the opt-in shared memory");
static_assert(2 * kAccCols + kStages * kSfCols <= kTmemCols, "tensor memory budget");

// kind::mxf4nvf4 instruction descriptor: e2m1 x e2m1 -> f32, both K-major,
// e4m3 (unsigned) block scales, scale data ids 0.
__host__ __device__ constexpr uint32_t idesc(int M, int N) {
  return (1u << 7)                      // A format e2m1
         | (1u << 10)                   // B format e2m1
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | (0u << 23)                   // scale format ue4m3
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}

// Shared-memory descriptor of one 512-byte scale group: 32 rows of 16 bytes,
// no swizzle, 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t sf_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)(128 >> 4) << 16;
  d |= (uint64_t)(128 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

__device__ __forceinline__ void sf_copy(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t sfa, uint32_t sfb,
                                    uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(
          d),
      "l"(a), "l"(b), "r"(id), "r"(sfa), "r"(sfb), "r"(accum)
      : "memory");
}

}  // namespace nvf4

// Tiles are enumerated expert-major, then row block, then column block (as in
// the bf16 and FP4-converting kernels).  map_ac / map_as: A codes [rows][K/2]
// (box 128 bytes x 128 rows, 128-byte swizzle) and A scales [rows][K/16] (box
// 16 x 128); map_bc / map_bs: B codes [records][Nrows][K/2] (box 128 x 64)
// and B scales [records][Nrows][K/16] (box 16 x 64); group e's weights are
// record slot_of[e], groups with a negative slot are not part of the launch.
// b_row(nb, half) gives the first weight row of each 64-row half of column
// block nb.
template <typename Epi, typename BRow>
__device__ void grouped_gemm_nvf4(const CUtensorMap* map_ac, const CUtensorMap* map_as, const CUtensorMap* map_bc,
                                  const CUtensorMap* map_bs, const int32_t* offsets, const int32_t* slot_of, int E,
                                  int nblocks_n, int K, Epi epi, BRow b_row, int* err) {
  constexpr int kStages = nvf4::kStages, kStageBytes = nvf4::kStageBytes, kBM = nvf4::kBM, kBN = nvf4::kBN;
  constexpr int kBKBytes = nvf4::kBKBytes, kACodes = nvf4::kACodes, kBCodes = nvf4::kBCodes;
  constexpr int kARaw = nvf4::kARaw, kBRaw = nvf4::kBRaw, kAtoms = nvf4::kAtoms, kEpiWarps = nvf4::kEpiWarps;
  constexpr int kAccCols = nvf4::kAccCols, kSfCols = nvf4::kSfCols, kTmemCols = nvf4::kTmemCols;
  constexpr int kMaxE = nvf4::kMaxE;
  constexpr uint32_t kTxBytes = nvf4::kTxBytes;
  extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* sfready = full + kStages;
  uint64_t* empty = sfready + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  __shared__ int tile_base[kMaxE + 1];
  __shared__ int s_scan[33];
  __shared__ volatile int s_fail;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

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
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&sfready[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if ((int)blockIdx.x >= n_tiles) return;
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ksteps = K / 256;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      int g = 0;
      for (int t = blockIdx.x; t < n_tiles && !s_fail; t += gridDim.x) {
        const Tile tl = tile_of(tile_base, offsets, E, nblocks_n, t);
        const int rec = slot_of[tl.e];
        for (int ks = 0; ks < ksteps; ++ks, ++g) {
          const int s = g % kStages;
          if (g >= kStages && !mbar_wait_or(&empty[s], ((g / kStages) - 1) & 1, &s_fail)) { s_fail = 1; break; }
          uint8_t* st = smem + s * kStageBytes;
          uint8_t* bc = st + kACodes;
          uint8_t* as = bc + kBCodes;
          uint8_t* bs = as + kARaw;
          mbar_expect_tx(&full[s], kTxBytes);
          tma_load_2d(st, map_ac, &full[s], ks * kBKBytes, tl.row0);
          tma_load_3d(bc, map_bc, &full[s], ks * kBKBytes, b_row(tl.nb, 0), rec);
          tma_load_3d(bc + kBCodes / 2, map_bc, &full[s], ks * kBKBytes, b_row(tl.nb, 1), rec);
          tma_load_2d(as, map_as, &full[s], ks * 16, tl.row0);
          tma_load_3d(bs, map_bs, &full[s], ks * 16, b_row(tl.nb, 0), rec);
          tma_load_3d(bs + kBRaw / 2, map_bs, &full[s], ks * 16, b_row(tl.nb, 1), rec);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      constexpr uint32_t id = nvf4::idesc(kBM, kBN);
      int g = 0, i = 0;
      for (int t = blockIdx.x; t < n_tiles && !s_fail; t += gridDim.x, ++i) {
        const int ab = i & 1;
        if (i >= 2 && !mbar_wait_or(&acc_empty[ab], ((i >> 1) - 1) & 1, &s_fail)) { s_fail = 1; break; }
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(ab * kAccCols);
        for (int ks = 0; ks < ksteps; ++ks, ++g) {
          const int s = g % kStages;
          if (!mbar_wait_or(&sfready[s], (g / kStages) & 1, &s_fail)) { s_fail = 1; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * kStageBytes);
          const uint32_t b0 = a0 + kACodes;
          const uint32_t atoms = b0 + kBCodes + kARaw + kBRaw;
          const uint32_t sf = tmem + (uint32_t)(2 * kAccCols + s * kSfCols);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            nvf4::sf_copy(sf + 4 * j, nvf4::sf_desc(atoms + j * 512));
            nvf4::sf_copy(sf + 16 + 4 * j, nvf4::sf_desc(atoms + kAtoms + j * 512));
            nvf4::mma(acc, smem_desc_sw128(a0 + j * 32), smem_desc_sw128(b0 + j * 32), id, sf + 4 * j, sf + 16 + 4 * j,
                (ks | j) != 0);
          }
          mma_commit(&empty[s]);
        }
        if (s_fail) break;
        mma_commit(&acc_full[ab]);
      }
    }
  } else if (warp == 2) {
    // scale rearrangement: group j of an operand holds, at bytes 16 m0 + 4 m1
    // + b, block scale b of K step j of row m0 + 32 m1
    int g = 0;
    for (int t = blockIdx.x; t < n_tiles && !s_fail; t += gridDim.x) {
      for (int ks = 0; ks < ksteps; ++ks, ++g) {
        const int s = g % kStages;
        if (!mbar_wait_or(&full[s], (g / kStages) & 1, &s_fail)) { s_fail = 1; break; }
        uint8_t* st = smem + s * kStageBytes;
        const uint32_t* raw_a = reinterpret_cast<const uint32_t*>(st + kACodes + kBCodes);
        const uint32_t* raw_b = raw_a + kARaw / 4;
        uint8_t* atoms = st + kACodes + kBCodes + kARaw + kBRaw;
#pragma unroll
        for (int op = 0; op < 2; ++op) {
          const uint32_t* raw = op ? raw_b : raw_a;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 v = make_uint4(raw[lane * 4 + j], raw[(lane + 32) * 4 + j], raw[(lane + 64) * 4 + j],
                                       raw[(lane + 96) * 4 + j]);
            *reinterpret_cast<uint4*>(atoms + op * kAtoms + j * 512 + lane * 16) = v;
          }
        }
        fence_proxy_async_smem();  // generic-proxy writes -> tcgen05.cp's async-proxy reads
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfready[s]);
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
    tmem_dealloc(tmem, kTmemCols);
  }
}

// gate/up epilogue: columns [0,64) gate, [64,128) up of output block nb ->
// h = SiLU(g) * u for 64 intermediate indices, quantised to FP4 (codes
// [rows][I/2], scales [rows][I/16]) for the down GEMM.
struct EpiSwiGLUQuant {
  uint8_t* hc;
  uint8_t* hs;
  int I;
  __device__ void operator()(uint32_t tmem, int row, bool valid, int nb) const {
    uint32_t sc = 0;
    uint32_t cw[8];
#pragma unroll
    for (int c = 0; c < 64; c += 16) {
      float g[16], u[16], h[16];
      tmem_ld16(tmem + c, g);
      tmem_ld16(tmem + 64 + c, u);
#pragma unroll
      for (int i = 0; i < 16; ++i) h[i] = g[i] / (1.0f + expf(-g[i])) * u[i];
      sc |= quant16(h, &cw[c / 8]) << (8 * (c / 16));
    }
    if (!valid) return;
    uint4* dst = reinterpret_cast<uint4*>(hc + (int64_t)row * (I / 2) + (int64_t)nb * 32);
    dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    *reinterpret_cast<uint32_t*>(hs + (int64_t)row * (I / 16) + (int64_t)nb * 4) = sc;
  }
};

// down epilogue: 128 fp32 columns of output block nb -> o [rows][N].
struct EpiStoreF32N128 {
  float* o;
  int N;
  __device__ void operator()(uint32_t tmem, int row, bool valid, int nb) const {
    for (int c = 0; c < 128; c += 16) {
      float v[16];
      tmem_ld16(tmem + c, v);
      if (!valid) continue;
      float4* dst = reinterpret_cast<float4*>(o + (int64_t)row * N + (int64_t)nb * 128 + c);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
};

}  // namespace tc
}  // namespace moe
