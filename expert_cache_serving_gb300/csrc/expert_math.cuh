// Row access and dot products of the SwiGLU expert, per weight format.
// A "chunk" is 16 bytes of a row's element stream: fp32 4 elements, bf16 8,
// FP4 32 (plus the 2 e4m3 scale bytes of its two 16-element blocks).
#pragma once
#include <cuda_fp16.h>

#include <type_traits>

#include "common.cuh"

namespace moe {

// 16-byte load of read-only streamed weights (resident slots, shared experts,
// host pool): no L1 allocation and L2 evict-first, so the weight stream does
// not push the kernel's code and the small cache state out of L2.
__device__ __forceinline__ uint4 ld_ro16(const void* p) {
  uint4 r;
  asm volatile(
      "{\n .reg .b64 pol;\n createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n"
      " ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], pol;\n}\n"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}
__device__ __forceinline__ unsigned short ld_ro2(const void* p) {
  unsigned short r;
  asm volatile(
      "{\n .reg .b64 pol;\n createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n"
      " ld.global.nc.L1::no_allocate.L2::cache_hint.u16 %0, [%1], pol;\n}\n"
      : "=h"(r)
      : "l"(p));
  return r;
}
// Loads of slots being filled while the kernel runs: bypass L1 and the
// read-only path, read at L2.
__device__ __forceinline__ uint4 ld_cg16(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ unsigned short ld_cg2(const void* p) {
  unsigned short r;
  asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}
template <bool FRESH>
__device__ __forceinline__ uint4 ld_w16(const void* p) {
  if constexpr (FRESH) return ld_cg16(p); else return ld_ro16(p);
}
template <bool FRESH>
__device__ __forceinline__ unsigned short ld_w2(const void* p) {
  if constexpr (FRESH) return ld_cg2(p); else return ld_ro2(p);
}

// Shared-memory loads of staged rows.
__device__ __forceinline__ uint4 lds16(const void* p) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(smem_u32(p)));
  return r;
}
__device__ __forceinline__ unsigned short lds2(const void* p) {
  unsigned short r;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(r) : "r"(smem_u32(p)));
  return r;
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// two e2m1 codes (low nibble = first element) -> two floats (exact)
__device__ __forceinline__ float2 e2m1x2_to_float2(uint32_t byte) {
  uint32_t h2;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h2) : "r"(byte));
  __half2 hv = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hv);
}

// two e4m3 bytes (low byte first) -> two floats (exact)
__device__ __forceinline__ float2 e4m3x2_to_float2(unsigned short two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
  __half2 hv = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hv);
}

// 16-byte chunks per lane and row in flight in the gate/up stream (a lane's
// chunks are lane, lane + 32, ... in that order whatever the unroll).
#ifndef MOE_P1_UNROLL_BF16
#define MOE_P1_UNROLL_BF16 8
#endif
#ifndef MOE_P1_UNROLL_FP4
#define MOE_P1_UNROLL_FP4 4
#endif
template <int WD>
struct Fmt;
template <>
struct Fmt<MOE_FP32> {
  static constexpr int kElemsPerChunk = 4;
  static constexpr int kUnroll = 4;
  __device__ static int64_t row_bytes(int K) { return (int64_t)K * 4; }
};
template <>
struct Fmt<MOE_BF16> {
  static constexpr int kElemsPerChunk = 8;
  static constexpr int kUnroll = MOE_P1_UNROLL_BF16;
  __device__ static int64_t row_bytes(int K) { return (int64_t)K * 2; }
};
template <>
struct Fmt<MOE_FP4> {
  static constexpr int kElemsPerChunk = 32;
  static constexpr int kUnroll = MOE_P1_UNROLL_FP4;
  __device__ static int64_t row_bytes(int K) { return (int64_t)K / 2; }
};

// Byte offsets of the matrices inside a record (see include/moecache.h).
struct RecView {
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* down;
  const uint8_t* gate_sc;
  const uint8_t* up_sc;
  const uint8_t* down_sc;
};

template <int WD>
__device__ __forceinline__ RecView rec_view(const uint8_t* rec, int H, int I) {
  RecView v;
  const int64_t HI = (int64_t)H * I;
  if (WD == MOE_FP32) {
    v.gate = rec; v.up = rec + HI * 4; v.down = rec + 2 * HI * 4;
    v.gate_sc = v.up_sc = v.down_sc = nullptr;
  } else if (WD == MOE_BF16) {
    v.gate = rec; v.up = rec + HI * 2; v.down = rec + 2 * HI * 2;
    v.gate_sc = v.up_sc = v.down_sc = nullptr;
  } else {
    v.gate = rec;
    v.up = rec + HI / 2;
    v.gate_sc = rec + HI;
    v.up_sc = rec + HI + HI / 16;
    v.down = rec + HI + HI / 8;
    v.down_sc = rec + HI + HI / 8 + HI / 2;
  }
  return v;
}

// ---- dot of one chunk with activations ---------------------------------------
template <int WD, typename VT>
__device__ __forceinline__ float chunk_dot(uint4 w, unsigned short sc2, const VT* xs);

template <>
__device__ __forceinline__ float chunk_dot<MOE_FP32, float>(uint4 w, unsigned short, const float* xs) {
  float4 a = *reinterpret_cast<const float4*>(xs);
  float acc = __uint_as_float(w.x) * a.x;
  acc = fmaf(__uint_as_float(w.y), a.y, acc);
  acc = fmaf(__uint_as_float(w.z), a.z, acc);
  acc = fmaf(__uint_as_float(w.w), a.w, acc);
  return acc;
}

__device__ __forceinline__ float dot8_bf16w(uint4 w, float4 a, float4 b) {
  float acc = bf16lo(w.x) * a.x;
  acc = fmaf(bf16hi(w.x), a.y, acc);
  acc = fmaf(bf16lo(w.y), a.z, acc);
  acc = fmaf(bf16hi(w.y), a.w, acc);
  acc = fmaf(bf16lo(w.z), b.x, acc);
  acc = fmaf(bf16hi(w.z), b.y, acc);
  acc = fmaf(bf16lo(w.w), b.z, acc);
  acc = fmaf(bf16hi(w.w), b.w, acc);
  return acc;
}

// acc + a * b with bf16 a, b (the halves of two words picked by HI) in one
// float32 rounding: the product of two bf16 values is exact in float32, so
// this is fmaf((float)a, (float)b, acc) bit for bit (acc = -0 gives a * b).
template <int HI>
__device__ __forceinline__ float fma_bf(uint32_t a2, uint32_t b2, float acc) {
  const unsigned short a = (unsigned short)(HI ? a2 >> 16 : a2), b = (unsigned short)(HI ? b2 >> 16 : b2);
  asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a), "h"(b));
  return acc;
}

// bf16 weights against bf16 activations: dot8_bf16w's operations in its order,
// as mixed-precision FMAs on the bf16 pairs (no conversions).
template <>
__device__ __forceinline__ float chunk_dot<MOE_BF16, __nv_bfloat16>(uint4 w, unsigned short, const __nv_bfloat16* xs) {
  const uint4 xv = *reinterpret_cast<const uint4*>(xs);
  float acc = fma_bf<0>(w.x, xv.x, -0.0f);
  acc = fma_bf<1>(w.x, xv.x, acc);
  acc = fma_bf<0>(w.y, xv.y, acc);
  acc = fma_bf<1>(w.y, xv.y, acc);
  acc = fma_bf<0>(w.z, xv.z, acc);
  acc = fma_bf<1>(w.z, xv.z, acc);
  acc = fma_bf<0>(w.w, xv.w, acc);
  acc = fma_bf<1>(w.w, xv.w, acc);
  return acc;
}

template <>
__device__ __forceinline__ float chunk_dot<MOE_BF16, float>(uint4 w, unsigned short, const float* xs) {
  float4 a = *reinterpret_cast<const float4*>(xs);
  float4 b = *reinterpret_cast<const float4*>(xs + 4);
  return dot8_bf16w(w, a, b);
}

// 16 e2m1 codes (8 bytes) against 16 activation values
template <typename VT>
__device__ __forceinline__ float block16_dot(uint32_t c0, uint32_t c1, const VT* xs);

template <>
__device__ __forceinline__ float block16_dot<__nv_bfloat16>(uint32_t c0, uint32_t c1, const __nv_bfloat16* xs) {
  uint4 xa = *reinterpret_cast<const uint4*>(xs);
  uint4 xb = *reinterpret_cast<const uint4*>(xs + 8);
  const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
  float acc = 0.f;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const uint32_t byte = ((b < 4 ? c0 : c1) >> (8 * (b & 3))) & 0xFFu;
    float2 w2 = e2m1x2_to_float2(byte);
    acc = fmaf(w2.x, bf16lo(xw[b]), acc);
    acc = fmaf(w2.y, bf16hi(xw[b]), acc);
  }
  return acc;
}

// xs 16-byte aligned: four 16-byte loads, the products in element order
template <>
__device__ __forceinline__ float block16_dot<float>(uint32_t c0, uint32_t c1, const float* xs) {
  float acc = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 v = reinterpret_cast<const float4*>(xs)[q];
    const uint32_t word = q < 2 ? c0 : c1;
    const float2 wa = e2m1x2_to_float2((word >> (16 * (q & 1))) & 0xFFu);
    const float2 wb = e2m1x2_to_float2((word >> (16 * (q & 1) + 8)) & 0xFFu);
    acc = fmaf(wa.x, v.x, acc);
    acc = fmaf(wa.y, v.y, acc);
    acc = fmaf(wb.x, v.z, acc);
    acc = fmaf(wb.y, v.w, acc);
  }
  return acc;
}

// Two e2m1 codes (low nibble = first element) -> two f16 in one word (exact).
__device__ __forceinline__ uint32_t e2m1x2_to_h2(uint32_t byte) {
  uint32_t h2;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h2) : "r"(byte));
  return h2;
}
// acc + a * b with f16 a, b (the halves of two words picked by HI) in one
// float32 rounding: the product of two f16 values is exact in float32, so this
// is fmaf((float)a, (float)b, acc) bit for bit, without the two conversions.
template <int HI>
__device__ __forceinline__ float fma_h(uint32_t a2, uint32_t b2, float acc) {
  const unsigned short a = (unsigned short)(HI ? a2 >> 16 : a2), b = (unsigned short)(HI ? b2 >> 16 : b2);
  asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a), "h"(b));
  return acc;
}

// 16 e2m1 codes against 16 f16 activations (16-byte aligned), in element
// order; the activations of FP4 decode are staged as f16 (see x_to_f16).
// The same with the block's two 8-value quarters at xa and xb (16-byte aligned).
__device__ __forceinline__ float block16_dot_q(uint32_t c0, uint32_t c1, const __half* xa_p, const __half* xb_p) {
  const uint4 xa = *reinterpret_cast<const uint4*>(xa_p), xb = *reinterpret_cast<const uint4*>(xb_p);
  const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
  float acc = 0.f;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const uint32_t w2 = e2m1x2_to_h2(((b < 4 ? c0 : c1) >> (8 * (b & 3))) & 0xFFu);
    acc = fma_h<0>(w2, xw[b], acc);
    acc = fma_h<1>(w2, xw[b], acc);
  }
  return acc;
}
template <>
__device__ __forceinline__ float block16_dot<__half>(uint32_t c0, uint32_t c1, const __half* xs) {
  return block16_dot_q(c0, c1, xs, xs + 8);
}

template <>
__device__ __forceinline__ float chunk_dot<MOE_FP4, __half>(uint4 w, unsigned short sc2, const __half* xs) {
  float2 s = e4m3x2_to_float2(sc2);
  float a0 = block16_dot<__half>(w.x, w.y, xs);
  float a1 = block16_dot<__half>(w.z, w.w, xs + 16);
  return fmaf(a1, s.y, a0 * s.x);
}

// chunk_dot<MOE_FP4, __half> with the chunk's four 8-value quarters qs values
// apart (x + k * qs for quarter k): the same operations in the same order.
__device__ __forceinline__ float chunk_dot_fp4q(uint4 w, unsigned short sc2, const __half* x, int qs) {
  float2 s = e4m3x2_to_float2(sc2);
  float a0 = block16_dot_q(w.x, w.y, x, x + qs);
  float a1 = block16_dot_q(w.z, w.w, x + 2 * qs, x + 3 * qs);
  return fmaf(a1, s.y, a0 * s.x);
}

template <>
__device__ __forceinline__ float chunk_dot<MOE_FP4, __nv_bfloat16>(uint4 w, unsigned short sc2, const __nv_bfloat16* xs) {
  float2 s = e4m3x2_to_float2(sc2);
  float a0 = block16_dot<__nv_bfloat16>(w.x, w.y, xs);
  float a1 = block16_dot<__nv_bfloat16>(w.z, w.w, xs + 16);
  return fmaf(a1, s.y, a0 * s.x);
}

template <>
__device__ __forceinline__ float chunk_dot<MOE_FP4, float>(uint4 w, unsigned short sc2, const float* xs) {
  float2 s = e4m3x2_to_float2(sc2);
  float a0 = block16_dot<float>(w.x, w.y, xs);
  float a1 = block16_dot<float>(w.z, w.w, xs + 16);
  return fmaf(a1, s.y, a0 * s.x);
}

// One half (16 codes) of an FP4 chunk converted once for several tokens
// (unscaled e2m1 values, exact), and its sum against one token's 16 values
// with block16_dot's operations in block16_dot's order.
__device__ __forceinline__ void fp4_half(uint32_t c0, uint32_t c1, float* v) {
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const float2 w2 = e2m1x2_to_float2(((b < 4 ? c0 : c1) >> (8 * (b & 3))) & 0xFFu);
    v[2 * b] = w2.x;
    v[2 * b + 1] = w2.y;
  }
}
__device__ __forceinline__ float block16_sum(const float* v, const __nv_bfloat16* xs) {
  const uint4 xa = reinterpret_cast<const uint4*>(xs)[0], xb = reinterpret_cast<const uint4*>(xs)[1];
  const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
  float acc = 0.f;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    acc = fmaf(v[2 * b], bf16lo(xw[b]), acc);
    acc = fmaf(v[2 * b + 1], bf16hi(xw[b]), acc);
  }
  return acc;
}
__device__ __forceinline__ float block16_sum(const float* v, const float* xs) {
  float acc = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 x4 = reinterpret_cast<const float4*>(xs)[q];
    acc = fmaf(v[4 * q], x4.x, acc);
    acc = fmaf(v[4 * q + 1], x4.y, acc);
    acc = fmaf(v[4 * q + 2], x4.z, acc);
    acc = fmaf(v[4 * q + 3], x4.w, acc);
  }
  return acc;
}

// acc[q] += chunk_dot<MOE_FP4>(w, sc2, xs(q)) for the first ntok tokens,
// each half of the chunk converted once: the same operations in the same
// order as chunk_dot, token by token.  f16 values: the chunk's quarter k at
// xs(q) + k * qs (qs = 8 for a contiguous chunk).
template <int MAXT, typename VT, typename XF>
__device__ __forceinline__ void fp4_chunk_tokens(uint4 w, unsigned short sc2, int ntok, XF xs_of, float* acc,
                                                 int qs = 8) {
  if constexpr (std::is_same<VT, __half>::value) {  // f16 activations: codes kept as f16 pairs
    float a0[MAXT];
    uint32_t h[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) h[b] = e2m1x2_to_h2(((b < 4 ? w.x : w.y) >> (8 * (b & 3))) & 0xFFu);
#pragma unroll
    for (int q = 0; q < MAXT; ++q) {
      if (q >= ntok) break;
      const __half* xq = xs_of(q);
      const uint4 xa = *reinterpret_cast<const uint4*>(xq), xb = *reinterpret_cast<const uint4*>(xq + qs);
      const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      float s0 = 0.f;
#pragma unroll
      for (int b = 0; b < 8; ++b) s0 = fma_h<1>(h[b], xw[b], fma_h<0>(h[b], xw[b], s0));
      a0[q] = s0;
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) h[b] = e2m1x2_to_h2(((b < 4 ? w.z : w.w) >> (8 * (b & 3))) & 0xFFu);
    const float2 s = e4m3x2_to_float2(sc2);
#pragma unroll
    for (int q = 0; q < MAXT; ++q) {
      if (q >= ntok) break;
      const __half* xq = xs_of(q) + 2 * qs;
      const uint4 xa = *reinterpret_cast<const uint4*>(xq), xb = *reinterpret_cast<const uint4*>(xq + qs);
      const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      float s1 = 0.f;
#pragma unroll
      for (int b = 0; b < 8; ++b) s1 = fma_h<1>(h[b], xw[b], fma_h<0>(h[b], xw[b], s1));
      acc[q] += fmaf(s1, s.y, a0[q] * s.x);
    }
  } else {
    float v[16], a0[MAXT];
    fp4_half(w.x, w.y, v);
#pragma unroll
    for (int q = 0; q < MAXT; ++q) {
      if (q >= ntok) break;
      a0[q] = block16_sum(v, (const VT*)xs_of(q));
    }
    fp4_half(w.z, w.w, v);
    const float2 s = e4m3x2_to_float2(sc2);
#pragma unroll
    for (int q = 0; q < MAXT; ++q) {
      if (q >= ntok) break;
      acc[q] += fmaf(block16_sum(v, (const VT*)xs_of(q) + 16), s.y, a0[q] * s.x);
    }
  }
}

}  // namespace moe
