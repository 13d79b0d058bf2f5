// GPU twin of the seeded expert-record generator (synth/__init__.py, synth.c):
// the same splitmix64 counter stream, Irwin-Hall sum of four 16-bit uniforms
// scaled in float32, bf16 round-to-nearest-even, and FP4 e2m1 codes with e4m3
// block scales by nearest value (ties to the even code).  It only produces
// inputs, for pools far too large to generate on the host in reasonable time;
// tests check it bit for bit against the numpy generator.  Every float
// operation uses an explicitly rounded intrinsic, so nothing is contracted.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

namespace {

enum { WD_FP32 = 0, WD_BF16 = 1, WD_FP4 = 2 };

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float element(uint64_t base, uint64_t n, float c) {
  const uint64_t r = mix64(base + (n + 1) * 0x9E3779B97F4A7C15ull);
  const int64_t s = (int64_t)((r & 0xFFFF) + ((r >> 16) & 0xFFFF) + ((r >> 32) & 0xFFFF) + (r >> 48)) - 131070;
  return __fmul_rn((float)s, c);
}

__device__ __forceinline__ uint16_t bf16_rne(float v) {
  const uint32_t b = __float_as_uint(v);
  return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

__constant__ float c_e4m3[127];  // non-negative finite e4m3 values, codes 0x00..0x7E

__device__ __forceinline__ int e4m3_rne(float t) {
  int lo = 0, hi = 127;  // first index with value > t
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (c_e4m3[mid] <= t) lo = mid + 1; else hi = mid;
  }
  int c = lo - 1;
  if (c < 0) c = 0;
  if (c >= 126) return 126;
  const float m = __fmul_rn(__fadd_rn(c_e4m3[c], c_e4m3[c + 1]), 0.5f);
  if (t > m || (t == m && (c & 1))) return c + 1;
  return c;
}

__device__ __forceinline__ int e2m1_rne(float a) {
  return (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
}

// one thread per 16 consecutive elements of one row of one record
__global__ void records_kernel(uint64_t seed, float c, int H, int I, int wdtype, int64_t key0, int64_t n_keys,
                               uint8_t* dst) {
  const int64_t HI = (int64_t)H * I;
  const int64_t units = 3 * HI / 16;
  const int64_t S = wdtype == WD_FP32 ? 12 * HI : wdtype == WD_BF16 ? 6 * HI : 3 * HI / 2 + 3 * HI / 16;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < units * n_keys;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t kidx = i / units, u = i % units;
    const uint64_t base = mix64((seed << 32) ^ (uint64_t)(key0 + kidx));
    const uint64_t n0 = (uint64_t)u * 16;  // element index within the record
    uint8_t* rec = dst + kidx * S;
    float v[16];
#pragma unroll
    for (int x = 0; x < 16; ++x) v[x] = element(base, n0 + x, c);
    if (wdtype == WD_FP32) {
      float4* o = reinterpret_cast<float4*>(rec + n0 * 4);
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else if (wdtype == WD_BF16) {
      uint32_t w[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) w[q] = (uint32_t)bf16_rne(v[2 * q]) | ((uint32_t)bf16_rne(v[2 * q + 1]) << 16);
      uint4* o = reinterpret_cast<uint4*>(rec + n0 * 2);
      o[0] = make_uint4(w[0], w[1], w[2], w[3]);
      o[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
      float amax = 0.f;
#pragma unroll
      for (int x = 0; x < 16; ++x) amax = fmaxf(amax, fabsf(v[x]));
      const int sc = e4m3_rne(__fdiv_rn(amax, 6.0f));
      const float sv = c_e4m3[sc];
      uint32_t w0 = 0, w1 = 0;
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        int mag = 0;
        if (sv > 0.f) mag = e2m1_rne(fabsf(__fdiv_rn(v[x], sv)));
        const uint32_t code = (uint32_t)(mag | ((v[x] < 0.f && mag > 0) ? 8 : 0));
        if (x < 8) w0 |= code << (4 * x); else w1 |= code << (4 * (x - 8));
      }
      // gate codes | up codes | gate scales | up scales | down codes | down scales
      const int t = (int)(n0 / HI);
      const int64_t in_t = (int64_t)(n0 % HI);
      uint8_t* codes = t < 2 ? rec + t * (HI / 2) + in_t / 2 : rec + HI + HI / 8 + in_t / 2;
      uint8_t* scales = t < 2 ? rec + HI + t * (HI / 16) + in_t / 16 : rec + HI + HI / 8 + HI / 2 + in_t / 16;
      *reinterpret_cast<uint2*>(codes) = make_uint2(w0, w1);
      *scales = (uint8_t)sc;
    }
  }
}

bool g_table = false;

int init_table() {
  if (g_table) return 0;
  float t[127];
  for (int c = 0; c < 127; ++c) {
    const int e = c >> 3, m = c & 7;
    double v;
    if (e == 0) {
      v = (m / 8.0) / 64.0;
    } else {
      v = 1.0 + m / 8.0;
      for (int i = 0; i < e - 7; ++i) v *= 2.0;
      for (int i = 0; i < 7 - e; ++i) v *= 0.5;
    }
    t[c] = (float)v;
  }
  if (cudaMemcpyToSymbol(c_e4m3, t, sizeof t) != cudaSuccess) return 1;
  g_table = true;
  return 0;
}

int64_t rec_bytes(int H, int I, int wd) {
  const int64_t HI = (int64_t)H * I;
  return wd == WD_FP32 ? 12 * HI : wd == WD_BF16 ? 6 * HI : 3 * HI / 2 + 3 * HI / 16;
}

}  // namespace

extern "C" {

// Records key0 .. key0+n_keys-1 into device memory dst (back to back).
int synth_gpu_records(uint64_t seed, float c, int H, int I, int wdtype, int64_t key0, int64_t n_keys, void* dst) {
  if (H % 16 || I % 16 || wdtype < 0 || wdtype > 2 || n_keys < 0) return 1;
  if (init_table()) return 2;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  records_kernel<<<sms * 8, 256>>>(seed, c, H, I, wdtype, key0, n_keys, (uint8_t*)dst);
  if (cudaGetLastError() != cudaSuccess) return 3;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 4;
}

// Fill a host buffer (ideally pinned) with records, generating chunks on the
// device and copying them back.
int synth_gpu_fill_host(uint64_t seed, float c, int H, int I, int wdtype, int64_t key0, int64_t n_keys, void* host,
                        int64_t chunk_bytes) {
  const int64_t S = rec_bytes(H, I, wdtype);
  int64_t per = chunk_bytes / S;
  if (per < 1) per = 1;
  if (per > n_keys) per = n_keys > 0 ? n_keys : 1;
  void* stage = nullptr;
  if (cudaMalloc(&stage, per * S) != cudaSuccess) return 5;
  int rc = 0;
  for (int64_t k = 0; k < n_keys && rc == 0; k += per) {
    const int64_t n = n_keys - k < per ? n_keys - k : per;
    rc = synth_gpu_records(seed, c, H, I, wdtype, key0 + k, n, stage);
    if (rc == 0 && cudaMemcpy((uint8_t*)host + k * S, stage, n * S, cudaMemcpyDeviceToHost) != cudaSuccess) rc = 6;
  }
  cudaFree(stage);
  return rc;
}

// Exact-size page-locked host memory (portable, mapped), and its release.
void* synth_host_alloc(size_t bytes) {
  void* p = nullptr;
  if (cudaHostAlloc(&p, bytes, cudaHostAllocPortable | cudaHostAllocMapped) != cudaSuccess) return nullptr;
  return p;
}

int synth_host_free(void* p) { return cudaFreeHost(p) == cudaSuccess ? 0 : 1; }
}
