"""ctypes wrapper of the fp64 oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The CUDA library never
does, and this package imports nothing from the library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

EXACT, BF16H = 0, 1


class _Layer(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("f", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("wdtype", ctypes.c_int32),
                ("x", ctypes.c_void_p), ("wr", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("wg", ctypes.c_void_p), ("wu", ctypes.c_void_p), ("wd", ctypes.c_void_p),
                ("sg", ctypes.c_void_p), ("su", ctypes.c_void_p), ("sd", ctypes.c_void_p),
                ("router_mode", ctypes.c_int32), ("hash_dims", ctypes.c_int32), ("wh", ctypes.c_void_p),
                ("zg", ctypes.c_void_p), ("zu", ctypes.c_void_p), ("zd", ctypes.c_void_p)]

WDTYPES = {"bf16": 0, "int8": 1, "int4": 2, "fp8": 3}

ROUTER_MODES = {"softmax": 0, "raw": 1, "hash": 2}


def build(force: bool = False, extra_flags=()) -> str:
    """Compile moe_oracle.c with plain gcc (-O2, OpenMP, no fast-math, no FMA contraction)."""
    src = os.path.join(_HERE, "moe_oracle.c")
    if force or extra_flags or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", "-ffp-contract=off", *extra_flags,
                               src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _bind(lib):
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.moe_oracle_route.argtypes = [vp, vp, i64, vp, vp, vp, vp, vp]
    lib.moe_oracle_route.restype = i32
    lib.moe_oracle_gate.argtypes = [i32, i32, vp, vp, vp, vp, vp]
    lib.moe_oracle_gate.restype = i32
    lib.moe_oracle_gate_raw.argtypes = [i32, i32, vp, vp, vp, vp, vp]
    lib.moe_oracle_gate_raw.restype = i32
    lib.moe_oracle_hash_expert.argtypes = [vp, vp, i32, i32, i32]
    lib.moe_oracle_hash_expert.restype = ctypes.c_int32
    lib.moe_oracle_dispatch.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp]
    lib.moe_oracle_dispatch.restype = i32
    lib.moe_oracle_expert.argtypes = [vp, i32, vp, i32, vp]
    lib.moe_oracle_fp8_value.argtypes = [ctypes.c_uint8]
    lib.moe_oracle_fp8_value.restype = ctypes.c_double
    lib.moe_oracle_expert.restype = None
    lib.moe_oracle_forward.argtypes = [vp, vp, i64, i32, vp, vp, vp]
    lib.moe_oracle_forward.restype = i32
    lib.moe_oracle_round_bf16.argtypes = [ctypes.c_double]
    lib.moe_oracle_round_bf16.restype = ctypes.c_double
    lib.moe_oracle_bf16_bits.argtypes = [ctypes.c_double]
    lib.moe_oracle_bf16_bits.restype = ctypes.c_uint16
    lib.moe_oracle_set_threads.argtypes = [i32]
    lib.moe_oracle_set_threads.restype = None
    lib.moe_oracle_get_threads.argtypes = []
    lib.moe_oracle_get_threads.restype = i32
    return lib


def load(path: str | None = None):
    """Load the oracle library (building it first if needed)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_SO))
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


class Oracle:
    """The oracle bound to one layer's host inputs (a ``synth.Layer``)."""

    def __init__(self, layer, lib=None):
        self.layer = layer
        self.lib = lib or load()
        s = layer.shape
        T = layer.x.shape[0]
        self._keep = [np.ascontiguousarray(a) if a is not None else None
                      for a in (layer.x, layer.wr, layer.bias, layer.wg, layer.wu, layer.wd,
                                layer.sg, layer.su, layer.sd, getattr(layer, "wh", None),
                                getattr(layer, "zg", None), getattr(layer, "zu", None), getattr(layer, "zd", None))]
        x, wr, b, wg, wu, wd, sg, su, sd, wh, zg, zu, zd = self._keep
        self.T, self.d, self.f, self.E, self.k = T, s.d, s.f, s.E, s.k
        router = getattr(s, "router", "softmax")
        self.c = _Layer(T, s.d, s.f, s.E, s.k, WDTYPES[s.wdtype],
                        _p(x), _p(wr), _p(b), _p(wg), _p(wu), _p(wd), _p(sg), _p(su), _p(sd),
                        ROUTER_MODES[router], getattr(s, "hash_dims", 0), _p(wh), _p(zg), _p(zu), _p(zd))

    def route(self, tokens=None, want_logits=False):
        """Gate for the listed tokens (all when None): ids, w, gap_k, gap_slot[, logits]."""
        tk = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
        n = self.T if tk is None else len(tk)
        ids = np.empty((n, self.k), np.int32)
        w = np.empty((n, self.k), np.float64)
        gk = np.empty(n, np.float64)
        gs = np.empty(n, np.float64)
        lg = np.empty((n, self.E), np.float64) if want_logits else None
        rc = self.lib.moe_oracle_route(ctypes.byref(self.c), _p(tk), n, _p(lg), _p(ids), _p(w),
                                       _p(gk), _p(gs))
        if rc:
            raise RuntimeError("oracle route failed")
        return (ids, w, gk, gs, lg) if want_logits else (ids, w, gk, gs)

    def forward(self, tokens=None, mode=BF16H):
        """Layer output rows (double) for the listed tokens, with ids and w."""
        tk = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
        n = self.T if tk is None else len(tk)
        out = np.empty((n, self.d), np.float64)
        ids = np.empty((n, self.k), np.int32)
        w = np.empty((n, self.k), np.float64)
        rc = self.lib.moe_oracle_forward(ctypes.byref(self.c), _p(tk), n, mode, _p(out), _p(ids), _p(w))
        if rc:
            raise RuntimeError("oracle forward failed")
        return out, ids, w

    def expert(self, e, xrow_bits, mode=BF16H):
        y = np.empty(self.d, np.float64)
        xr = np.ascontiguousarray(xrow_bits, dtype=np.uint16)
        self.lib.moe_oracle_expert(ctypes.byref(self.c), int(e), xr.ctypes.data, mode, y.ctypes.data)
        return y


def gate(logits, k, lib=None, raw=False):
    """Gate of one token from its E logits (double): ids, w, gap_k, gap_slot
    (raw=True: the raw-logit gate, whose weights are the selected logits)."""
    lib = lib or load()
    l = np.ascontiguousarray(logits, dtype=np.float64)
    ids = np.empty(k, np.int32)
    w = np.empty(k, np.float64)
    gk = ctypes.c_double()
    gs = ctypes.c_double()
    fn = lib.moe_oracle_gate_raw if raw else lib.moe_oracle_gate
    if fn(len(l), k, l.ctypes.data, ids.ctypes.data, w.ctypes.data, ctypes.addressof(gk), ctypes.addressof(gs)):
        raise ValueError("bad gate sizes")
    return ids, w, gk.value, gs.value


def hash_expert(xrow_bits, wh_bits, E, lib=None):
    """The hash router's expert of one bf16 row under W_h [hash_dims][d] (bits)."""
    lib = lib or load()
    x = np.ascontiguousarray(xrow_bits, dtype=np.uint16)
    wh = np.ascontiguousarray(wh_bits, dtype=np.uint16)
    e = lib.moe_oracle_hash_expert(x.ctypes.data, wh.ctypes.data, x.shape[0], wh.shape[0], int(E))
    if e < 0:
        raise ValueError("bad hash sizes")
    return int(e)


def dispatch(ids, E, lib=None):
    """Counting-sort dispatch of ids[T][k]: cnt, off, tok, inv (flat [T*k])."""
    lib = lib or load()
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    cnt = np.empty(E, np.int32)
    off = np.empty(E + 1, np.int32)
    tok = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    if lib.moe_oracle_dispatch(T, E, k, ids.ctypes.data, cnt.ctypes.data, off.ctypes.data,
                               tok.ctypes.data, inv.ctypes.data):
        raise ValueError("bad routing ids")
    return cnt, off, tok, inv.reshape(T, k)


def round_bf16(v, lib=None):
    return (lib or load()).moe_oracle_round_bf16(float(v))


def bf16_bits(v, lib=None):
    return (lib or load()).moe_oracle_bf16_bits(float(v))


def set_threads(n, lib=None):
    (lib or load()).moe_oracle_set_threads(int(n))


def get_threads(lib=None):
    return (lib or load()).moe_oracle_get_threads()
