"""Seeded synthetic inputs for the routed-MoE expert-cache layer.

This package only *generates inputs*: expert weight records, router logit
traces, router weights and activations.  It holds none of the layer's own
arithmetic (routing, cache bookkeeping, permutation, dequantisation, the
SwiGLU expert, the combine).  Both the CPU oracle side of the tests and the
GPU path draw their inputs from here, and from nowhere else.

Expert weights
--------------
Every weight of every expert record is a pure function of
``(seed, key, element index)``, so any record can be regenerated on its own
(the pools of the large configurations are far bigger than what the oracle
ever needs to see):

* ``splitmix64`` (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) is used as a counter-based generator:
  ``r_n = mix64(base + (n + 1) * 0x9E3779B97F4A7C15)`` with
  ``base = mix64((seed << 32) ^ key)``.
* The four 16-bit fields of ``r_n`` are summed (an Irwin-Hall sum of four
  uniforms), centred, and scaled in float32 so the value has mean 0 and
  standard deviation ``sigma``: an approximately normal weight whose bits do
  not depend on any libm.
* bf16 records round that float32 value to nearest-even.  FP4 records
  quantise each block of 16 consecutive values along a row: the block scale
  is the e4m3 value nearest to ``amax / 6`` (ties to the even code) and each
  element is the e2m1 value nearest to ``v / scale`` (ties to even,
  saturating at 6).

The C file next to this module implements the same generator for filling
whole host pools quickly; ``tests/test_synth.py`` checks the two agree bit
for bit.

Record layout (one record per (layer, expert) key ``l*E + e``; the shared
expert of layer ``l`` uses key ``L*E + l``):

* fp32 / bf16: ``W_gate[I][H] | W_up[I][H] | W_down[H][I]`` row-major.
* FP4: ``gate codes[I][H/2] | up codes[I][H/2] | gate scales[I][H/16] |
  up scales[I][H/16] | down codes[H][I/2] | down scales[H][I/16]`` (the
  gate/up half and the down half are each contiguous); code byte ``c`` of a
  row holds element ``2c`` in its low nibble and ``2c+1`` in its high
  nibble; scale byte ``b`` covers elements ``16b .. 16b+15``.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

WD_FP32, WD_BF16, WD_FP4 = 0, 1, 2
WD_NAMES = {WD_FP32: "fp32", WD_BF16: "bf16", WD_FP4: "fp4"}

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_U16 = np.uint64(0xFFFF)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def sigma_scale(sigma: float) -> np.float32:
    """float32 factor turning a centred sum of four 16-bit uniforms into N(0, sigma^2)-like values."""
    return np.float32(sigma * math.sqrt(3.0) / 65536.0)


def stream_base(seed: int, key: int) -> np.uint64:
    if not (0 <= seed < 2**31 and 0 <= key < 2**32):
        raise ValueError("seed must be < 2^31 and key < 2^32")
    with np.errstate(over="ignore"):
        return _mix64(np.array([(seed << 32) ^ key], dtype=np.uint64))[0]


def element_values(seed: int, key: int, n0: int, n: int, sigma: float) -> np.ndarray:
    """float32 weights for element indices n0 .. n0+n-1 of record ``key``."""
    base = stream_base(seed, key)
    idx = np.arange(n0 + 1, n0 + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        r = _mix64(base + idx * _GAMMA)
    s = (r & _U16) + ((r >> np.uint64(16)) & _U16) + ((r >> np.uint64(32)) & _U16) + (r >> np.uint64(48))
    s = s.astype(np.int64) - 131070
    return s.astype(np.float32) * sigma_scale(sigma)


def to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --- FP4 encoding (data generation only) ------------------------------------
# Non-negative finite e4m3 values (codes 0x00..0x7E) and e2m1 magnitudes
# (codes 0..7), built from the formats' definitions (OCP Microscaling Formats
# spec v1.0: e4m3 bias 7 with subnormals, e2m1 bias 1).

def _e4m3_encode_table() -> np.ndarray:
    vals = []
    for c in range(127):
        e, m = c >> 3, c & 7
        vals.append(m / 8.0 * 2.0 ** -6 if e == 0 else 2.0 ** (e - 7) * (1.0 + m / 8.0))
    return np.array(vals, dtype=np.float32)


E4M3_ENC = _e4m3_encode_table()
E2M1_ENC = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)


def _rne_encode(t: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Code of the table value nearest to t >= 0, ties to the even code, saturating."""
    t = np.asarray(t, dtype=np.float32)
    last = len(table) - 1
    c = np.searchsorted(table, t, side="right").astype(np.int64) - 1
    c = np.clip(c, 0, last)
    sat = c >= last
    cn = np.minimum(c + 1, last)
    lo, hi = table[c], table[cn]
    mid = (lo + hi) * np.float32(0.5)
    up = (t > mid) | ((t == mid) & ((c & 1) == 1))
    out = np.where(up, cn, c)
    return np.where(sat, last, out).astype(np.uint8)


def quantise_fp4_rows(v: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Quantise float32 rows [R, K] (K % 16 == 0) -> (codes u8 [R, K/2], scales u8 [R, K/16])."""
    R, K = v.shape
    blocks = v.reshape(R, K // 16, 16)
    amax = np.abs(blocks).max(axis=2)
    t = (amax / np.float32(6.0)).astype(np.float32)
    sc = _rne_encode(t, E4M3_ENC)
    sv = E4M3_ENC[sc]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = blocks / sv[:, :, None]
    mag = _rne_encode(np.where(sv[:, :, None] > 0, np.abs(q), 0.0), E2M1_ENC)
    code = mag | np.where((blocks < 0) & (mag > 0), np.uint8(8), np.uint8(0))
    code = code.reshape(R, K).astype(np.uint8)
    packed = (code[:, 0::2] | (code[:, 1::2] << np.uint8(4))).astype(np.uint8)
    return packed, sc.astype(np.uint8)


# --- records -----------------------------------------------------------------

def record_bytes(H: int, I: int, wdtype: int) -> int:
    if wdtype == WD_FP32:
        return 12 * H * I
    if wdtype == WD_BF16:
        return 6 * H * I
    if wdtype == WD_FP4:
        return 3 * H * I // 2 + 3 * H * I // 16
    raise ValueError(wdtype)


def expert_record(seed: int, key: int, H: int, I: int, wdtype: int, sigma: float = 0.02) -> np.ndarray:
    """One expert record (u8 [S]) in the layout described in the module docstring."""
    HI = H * I
    v = element_values(seed, key, 0, 3 * HI, sigma)
    if wdtype == WD_FP32:
        return v.view(np.uint8).copy()
    if wdtype == WD_BF16:
        return to_bf16_bits(v).view(np.uint8).copy()
    if wdtype != WD_FP4:
        raise ValueError(wdtype)
    out = np.empty(record_bytes(H, I, wdtype), dtype=np.uint8)
    parts = []
    for t, (R, K) in enumerate([(I, H), (I, H), (H, I)]):
        parts.append(quantise_fp4_rows(v[t * HI:(t + 1) * HI].reshape(R, K)))
    (gc, gs), (uc, us), (dc, ds) = parts
    off = 0
    for arr in (gc, uc, gs, us, dc, ds):
        out[off:off + arr.size] = arr.reshape(-1)
        off += arr.size
    return out


# --- fast pool fill (C, threaded) ---------------------------------------------

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = os.path.join(os.path.dirname(__file__), "_lib", "libsynth.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        lib.synth_records.argtypes = [ctypes.c_uint64, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                      ctypes.c_int]
        lib.synth_records.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def fill_records(dst_ptr: int, seed: int, key0: int, n_keys: int, H: int, I: int, wdtype: int,
                 sigma: float = 0.02, threads: int | None = None) -> None:
    """Write records key0 .. key0+n_keys-1 back to back at host address dst_ptr (C, threaded)."""
    if threads is None:
        threads = max(1, min(64, os.cpu_count() or 1))
    rc = _lib().synth_records(seed, float(sigma_scale(sigma)), H, I, wdtype, key0, n_keys,
                              ctypes.c_void_p(dst_ptr), threads)
    if rc != 0:
        raise RuntimeError(f"synth_records failed ({rc})")


# --- GPU twin (synth_gpu.cu) and exact-size pinned buffers -------------------------

_GLIB = None


def _gpu_lib():
    global _GLIB
    if _GLIB is None:
        path = os.path.join(os.path.dirname(__file__), "_lib", "libsynth_gpu.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        lib.synth_gpu_records.argtypes = [ctypes.c_uint64, ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
        lib.synth_gpu_fill_host.argtypes = [ctypes.c_uint64, ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64]
        lib.synth_host_alloc.argtypes = [ctypes.c_size_t]
        lib.synth_host_alloc.restype = ctypes.c_void_p
        lib.synth_host_free.argtypes = [ctypes.c_void_p]
        _GLIB = lib
    return _GLIB


def records_gpu(dst_dev_ptr: int, seed: int, key0: int, n_keys: int, H: int, I: int, wdtype: int,
                sigma: float = 0.02) -> None:
    """Records key0 .. key0+n_keys-1 written back to back at a device address."""
    rc = _gpu_lib().synth_gpu_records(seed, float(sigma_scale(sigma)), H, I, wdtype, key0, n_keys,
                                      ctypes.c_void_p(dst_dev_ptr))
    if rc:
        raise RuntimeError(f"synth_gpu_records failed ({rc})")


def mem_available_bytes() -> int:
    with open("/proc/meminfo") as f:
        for line in f:
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    return 0


class PinnedBuffer:
    """Exact-size page-locked host buffer; freed when the last view of it goes away."""

    def __init__(self, nbytes: int, reserve: int = 16 << 30):
        avail = mem_available_bytes()
        if avail and nbytes + reserve > avail:
            raise MemoryError(f"{nbytes / 1e9:.1f} GB pinned pool would leave less than "
                              f"{reserve / 1e9:.0f} GB of the {avail / 1e9:.1f} GB available host memory")
        self.nbytes = nbytes
        self.ptr = _gpu_lib().synth_host_alloc(nbytes)
        if not self.ptr:
            raise MemoryError(f"cudaHostAlloc of {nbytes} bytes failed")
        self.__array_interface__ = {"shape": (nbytes,), "typestr": "|u1", "data": (self.ptr, False), "version": 3}

    def __del__(self):
        if getattr(self, "ptr", None):
            _gpu_lib().synth_host_free(ctypes.c_void_p(self.ptr))
            self.ptr = None


def pinned_pool(seed: int, n_keys: int, H: int, I: int, wdtype: int, sigma: float = 0.02,
                chunk_bytes: int = 1 << 30) -> np.ndarray:
    """u8 [n_keys, S] numpy view of an exact-size pinned buffer filled on the GPU."""
    S = record_bytes(H, I, wdtype)
    buf = PinnedBuffer(n_keys * S)
    rc = _gpu_lib().synth_gpu_fill_host(seed, float(sigma_scale(sigma)), H, I, wdtype, 0, n_keys,
                                        ctypes.c_void_p(buf.ptr), chunk_bytes)
    if rc:
        raise RuntimeError(f"synth_gpu_fill_host failed ({rc})")
    return np.asarray(buf).reshape(n_keys, S)


def records_array(seed: int, key0: int, n_keys: int, H: int, I: int, wdtype: int,
                  sigma: float = 0.02) -> np.ndarray:
    """Records as a fresh numpy u8 [n_keys, S] array, filled by the C generator."""
    S = record_bytes(H, I, wdtype)
    out = np.empty((n_keys, S), dtype=np.uint8)
    fill_records(out.ctypes.data, seed, key0, n_keys, H, I, wdtype, sigma)
    return out


# --- routing traces and activations --------------------------------------------

def ar1_logits(seed: int, T: int, L: int, B: int, E: int, rho: float = 0.8, sd: float = 0.6) -> np.ndarray:
    """float32 [T, L, B, E]: logit_t = rho*logit_{t-1} + sd*N(0,1) per (layer, sequence, expert); logit_0 ~ N(0,1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.empty((T, L, B, E), dtype=np.float32)
    z = rng.standard_normal((L, B, E))
    out[0] = z
    for t in range(1, T):
        z = rho * z + sd * rng.standard_normal((L, B, E))
        out[t] = z
    return out


def iid_logits(seed: int, L: int, T: int, E: int) -> np.ndarray:
    """float32 [L, T, E] i.i.d. N(0,1) router logits (prefill)."""
    rng = np.random.Generator(np.random.PCG64([seed, 11]))
    return rng.standard_normal((L, T, E), dtype=np.float32)


def activations_f32(seed: int, step: int, layer: int, B: int, H: int) -> np.ndarray:
    """float32 [B, H] ~ N(0,1) for one (step, layer) call."""
    rng = np.random.Generator(np.random.PCG64([seed, 1, step, layer]))
    return rng.standard_normal((B, H), dtype=np.float32)


def activations_bf16(seed: int, step: int, layer: int, B: int, H: int) -> np.ndarray:
    """bf16 bit patterns (u16 [B, H]) of N(0,1) activations for one (step, layer) call."""
    return to_bf16_bits(activations_f32(seed, step, layer, B, H)).reshape(B, H)


def router_weights(seed: int, L: int, E: int, H: int, sigma: float = 0.02) -> np.ndarray:
    """float32 [L, E, H] router matrices W_r ~ N(0, sigma^2)."""
    rng = np.random.Generator(np.random.PCG64([seed, 7]))
    return (rng.standard_normal((L, E, H), dtype=np.float32) * np.float32(sigma)).astype(np.float32)
