"""Seeded synthetic inputs for the MoE FFN layer.

This module is shared by the fp64 oracle's tests and by the CUDA library's
tests and benchmark.  It holds no part of the layer's arithmetic: it only
draws the inputs (activations, router weights, the hash router's projection,
expert weights, int8 / int4 / e4m3 codes and scales, the skewed router bias) in the shapes and distributions of the five
workloads below, from a counter-based stream defined in ``synth.c``.

The workloads follow the layer shapes the Colibri pages discuss: a Mixtral-8x7B
shaped layer (8 experts of d_ff = 14336 over d_model = 4096, "Colibri：面向MoE架构的
C语言级高效推理引擎" §3.1), its prefill and decode sizes, a fine-grained 128-expert
top-4 layer with skewed popularity (the 128-expert top-4 model of the same page's
§1) and an int8 symmetric per-channel weight layer (int8 expert weights,
"lshu.cn/news/53496" §3 and §4.3).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")
_lib = None

# tensor ids of the counter streams
TID_X, TID_WR, TID_WG, TID_WU, TID_WD, TID_SG, TID_SU, TID_SD, TID_WH = 1, 2, 3, 4, 5, 6, 7, 8, 9
TID_ZG, TID_ZU, TID_ZD = 10, 11, 12

WEIGHT_STD = 0.02      # bf16 weights ~ N(0, 0.02^2)
INT8_SCALE = 40.0      # int8 codes round(40 N(0,1)) clipped to [-127, 127]
SCALE_LO, SCALE_HI = 0.5e-3, 1.0e-3   # per-output-channel fp32 scales ~ U
# int4 weights, asymmetric per output channel: W = s (q - z) with 4-bit codes
# q = z + clip(rint(2.5 N(0,1)), -6, 6), integer zero points z = 7 +
# clip(rint(1.2 N(0,1)), -1, 2) in 6..9 (so q stays in 0..15) and scales
# s ~ U(0.006, 0.010): weights of about the bf16 layers' N(0, 0.02^2) spread
INT4_CODE_SCALE, INT4_CODE_LO, INT4_CODE_HI = 2.5, -6, 6
INT4_ZERO_SCALE, INT4_ZERO_LO, INT4_ZERO_HI, INT4_ZERO_MID = 1.2, -1, 2, 7
INT4_SCALE_LO, INT4_SCALE_HI = 0.006, 0.010
# fp8 (e4m3) weights: codes of 32 N(0,1) rounded to the nearest e4m3 value
# (ties to the even code), scales ~ U(0.5e-3, 1e-3) per output channel as for
# int8
FP8_SCALE = 32.0


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so beside it (plain gcc, OpenMP)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.synth_normal_bf16.argtypes = [u64, u64, dbl, vp, i64, i64]
        lib.synth_normal_f64.argtypes = [u64, u64, dbl, vp, i64, i64]
        lib.synth_int8.argtypes = [u64, u64, dbl, ctypes.c_int, ctypes.c_int, vp, i64, i64]
        lib.synth_uniform_f32.argtypes = [u64, u64, dbl, dbl, vp, i64, i64]
        lib.synth_bits.argtypes = [u64, u64, vp, i64, i64]
        for f in (lib.synth_normal_bf16, lib.synth_normal_f64, lib.synth_int8,
                  lib.synth_uniform_f32, lib.synth_bits):
            f.restype = None
        _lib = lib
    return _lib


def normal_bf16(seed, tid, scale, shape, offset=0) -> np.ndarray:
    """bf16 bit patterns (uint16) of scale * N(0,1)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    _load().synth_normal_bf16(seed, tid, scale, out.ctypes.data, offset, n)
    return out.reshape(shape)


def normal_f64(seed, tid, scale, shape, offset=0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)
    _load().synth_normal_f64(seed, tid, scale, out.ctypes.data, offset, n)
    return out.reshape(shape)


def int8_codes(seed, tid, scale, shape, lo=-127, hi=127, offset=0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.int8)
    _load().synth_int8(seed, tid, scale, lo, hi, out.ctypes.data, offset, n)
    return out.reshape(shape)


def uniform_f32(seed, tid, lo, hi, shape, offset=0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    _load().synth_uniform_f32(seed, tid, lo, hi, out.ctypes.data, offset, n)
    return out.reshape(shape)


def pack_int4(q: np.ndarray) -> np.ndarray:
    """4-bit codes 0..15 [..., n] (n even) -> bytes [..., n/2]: element 2i in the
    low nibble of byte i, element 2i + 1 in its high nibble."""
    q = q.astype(np.uint8)
    return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)


def unpack_int4(b: np.ndarray) -> np.ndarray:
    """Inverse of pack_int4."""
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0x0F
    out[..., 1::2] = b >> 4
    return out


def int4_weights(seed, tid_w, tid_z, rows_shape, cols):
    """Packed int4 codes [..., cols/2] and their zero points [...] (uint8)."""
    z = (int8_codes(seed, tid_z, INT4_ZERO_SCALE, rows_shape, INT4_ZERO_LO, INT4_ZERO_HI).astype(np.int32)
         + INT4_ZERO_MID)
    c = int8_codes(seed, tid_w, INT4_CODE_SCALE, rows_shape + (cols,), INT4_CODE_LO, INT4_CODE_HI).astype(np.int32)
    q = c + z[..., None]
    return pack_int4(q), z.astype(np.uint8)


def _e4m3_grid() -> np.ndarray:
    """The non-negative finite e4m3 values, by code 0x00..0x7E (ascending)."""
    c = np.arange(0x7F)
    ex, man = c >> 3, c & 7
    return np.where(ex == 0, man / 8.0 * 2.0 ** -6, (1.0 + man / 8.0) * 2.0 ** (ex - 7))


def fp8_codes(seed, tid, scale, shape) -> np.ndarray:
    """e4m3 bytes of scale * N(0,1) draws."""
    return encode_e4m3(normal_f64(seed, tid, scale, shape))


def encode_e4m3(v) -> np.ndarray:
    """e4m3 bytes of float values: nearest value, ties to the even code,
    magnitudes past 448 saturated."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    grid = _e4m3_grid()
    i = np.clip(np.searchsorted(grid, a), 1, len(grid) - 1)
    lo, hi = grid[i - 1], grid[i]
    up = (a - lo > hi - a) | ((a - lo == hi - a) & (i % 2 == 0))
    code = np.where(up, i, i - 1)
    code = np.where(a >= grid[-1], len(grid) - 1, code)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def raw_bits(seed, tid, n, offset=0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_bits(seed, tid, out.ctypes.data, offset, n)
    return out


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Shape:
    """One MoE FFN layer workload: T tokens, d = d_model, f = d_ff, E experts, top-k."""
    name: str
    T: int
    d: int
    f: int
    E: int
    k: int
    wdtype: str = "bf16"       # "bf16", "int8", "int4" or "fp8"
    bias: bool = False         # skewed router bias b_e = 2 ln(1/(e+1))
    seed: int = 0
    router: str = "softmax"    # "softmax" (top-k, renormalised), "raw" (raw-logit weights), "hash"
    hash_dims: int = 0         # hash router: columns of the d x hash_dims projection


# The five workloads (sizes and distributions of the layer shapes above).
WORKLOADS = {
    "tiny": Shape("tiny", T=64, d=256, f=512, E=8, k=2, seed=1001),
    "mixtral_prefill": Shape("mixtral_prefill", T=4096, d=4096, f=14336, E=8, k=2, seed=1002),
    "mixtral_decode": Shape("mixtral_decode", T=64, d=4096, f=14336, E=8, k=2, seed=1003),
    "skewed": Shape("skewed", T=8192, d=2048, f=768, E=128, k=4, bias=True, seed=1004),
    "int8": Shape("int8", T=16384, d=4096, f=1536, E=64, k=6, wdtype="int8", seed=1005),
    # the int8 layer's shape with 4-bit weights (scale and zero point per channel)
    "int4": Shape("int4", T=16384, d=4096, f=1536, E=64, k=6, wdtype="int4", seed=1006),
    # the int8 layer's shape with fp8 (e4m3) weights and a scale per channel
    "fp8": Shape("fp8", T=16384, d=4096, f=1536, E=64, k=6, wdtype="fp8", seed=1007),
}


def skew_bias(E: int) -> np.ndarray:
    """b_e = 2 ln(1/(e+1)), evaluated in double and rounded once to float32."""
    return np.array([2.0 * math.log(1.0 / (e + 1)) for e in range(E)], dtype=np.float32)


@dataclass
class Layer:
    """Host copies of one layer's inputs (bf16 as uint16 bit patterns)."""
    shape: Shape
    x: np.ndarray                 # [T][d] bf16 bits
    wr: np.ndarray                # [E][d] bf16 bits
    bias: np.ndarray | None       # [E] float32
    wg: np.ndarray                # [E][f][d] bf16 bits, int8 or e4m3 bytes; int4: [E][f][d/2] packed
    wu: np.ndarray                # [E][f][d]
    wd: np.ndarray                # [E][d][f]
    sg: np.ndarray | None = None  # [E][f] float32 (int8, int4 and fp8)
    su: np.ndarray | None = None  # [E][f]
    sd: np.ndarray | None = None  # [E][d]
    wh: np.ndarray | None = None  # [hash_dims][d] bf16 bits (hash router only)
    zg: np.ndarray | None = None  # [E][f] uint8 zero points (int4 only)
    zu: np.ndarray | None = None  # [E][f]
    zd: np.ndarray | None = None  # [E][d]
    extra: dict = field(default_factory=dict)


def make_layer(shape: Shape, seed: int | None = None, T: int | None = None) -> Layer:
    """Draw a layer's inputs.  `T` overrides the token count (same weights)."""
    s = shape.seed if seed is None else seed
    T = shape.T if T is None else T
    d, f, E = shape.d, shape.f, shape.E
    x = normal_bf16(s, TID_X, 1.0, (T, d))
    wr = normal_bf16(s, TID_WR, WEIGHT_STD, (E, d))
    bias = skew_bias(E) if shape.bias else None
    wh = normal_bf16(s, TID_WH, WEIGHT_STD, (shape.hash_dims, d)) if shape.router == "hash" else None
    if shape.wdtype == "bf16":
        wg = normal_bf16(s, TID_WG, WEIGHT_STD, (E, f, d))
        wu = normal_bf16(s, TID_WU, WEIGHT_STD, (E, f, d))
        wd = normal_bf16(s, TID_WD, WEIGHT_STD, (E, d, f))
        return Layer(shape, x, wr, bias, wg, wu, wd, wh=wh)
    if shape.wdtype == "int4":
        wg, zg = int4_weights(s, TID_WG, TID_ZG, (E, f), d)
        wu, zu = int4_weights(s, TID_WU, TID_ZU, (E, f), d)
        wd, zd = int4_weights(s, TID_WD, TID_ZD, (E, d), f)
        sg = uniform_f32(s, TID_SG, INT4_SCALE_LO, INT4_SCALE_HI, (E, f))
        su = uniform_f32(s, TID_SU, INT4_SCALE_LO, INT4_SCALE_HI, (E, f))
        sd = uniform_f32(s, TID_SD, INT4_SCALE_LO, INT4_SCALE_HI, (E, d))
        return Layer(shape, x, wr, bias, wg, wu, wd, sg, su, sd, wh=wh, zg=zg, zu=zu, zd=zd)
    if shape.wdtype == "fp8":
        wg = fp8_codes(s, TID_WG, FP8_SCALE, (E, f, d))
        wu = fp8_codes(s, TID_WU, FP8_SCALE, (E, f, d))
        wd = fp8_codes(s, TID_WD, FP8_SCALE, (E, d, f))
    else:
        wg = int8_codes(s, TID_WG, INT8_SCALE, (E, f, d))
        wu = int8_codes(s, TID_WU, INT8_SCALE, (E, f, d))
        wd = int8_codes(s, TID_WD, INT8_SCALE, (E, d, f))
    sg = uniform_f32(s, TID_SG, SCALE_LO, SCALE_HI, (E, f))
    su = uniform_f32(s, TID_SU, SCALE_LO, SCALE_HI, (E, f))
    sd = uniform_f32(s, TID_SD, SCALE_LO, SCALE_HI, (E, d))
    return Layer(shape, x, wr, bias, wg, wu, wd, sg, su, sd, wh=wh)


def custom_shape(name, T, d, f, E, k, wdtype="bf16", bias=False, seed=7, router="softmax", hash_dims=0) -> Shape:
    return Shape(name, T=T, d=d, f=f, E=E, k=k, wdtype=wdtype, bias=bias, seed=seed, router=router,
                 hash_dims=hash_dims)


def with_router(shape: Shape, router: str, hash_dims: int = 8) -> Shape:
    """The same layer with another router: "raw" keeps k; "hash" routes each
    token to one expert (k = 1) through a d x hash_dims projection."""
    if router == "softmax":
        return shape
    if router == "raw":
        return Shape(shape.name + "_raw", shape.T, shape.d, shape.f, shape.E, shape.k, shape.wdtype, shape.bias,
                     shape.seed, router="raw")
    if router == "hash":
        return Shape(shape.name + "_hash", shape.T, shape.d, shape.f, shape.E, 1, shape.wdtype, shape.bias,
                     shape.seed, router="hash", hash_dims=hash_dims)
    raise ValueError(f"unknown router {router!r}")
