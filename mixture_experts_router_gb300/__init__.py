"""Python binding of libcbmoe.so, the GB300 MoE FFN layer (C ABI in include/cb_moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch is used by callers for device memory and streams; this module
takes raw pointers (ints) or torch tensors and forwards them.  There is no
fallback: if the shared library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcbmoe.so")

CB_OK, CB_ERR_INVALID_ARG, CB_ERR_UNSUPPORTED, CB_ERR_ALIGNMENT = 0, 1, 2, 3
CB_ERR_OOM, CB_ERR_CUDA, CB_ERR_TIMEOUT, CB_ERR_DEVICE = 4, 5, 6, 7
CB_W_BF16, CB_W_INT8, CB_W_INT4, CB_W_FP8 = 0, 1, 2, 3
WDTYPES = {"bf16": CB_W_BF16, "int8": CB_W_INT8, "int4": CB_W_INT4, "fp8": CB_W_FP8}
CB_FLAG_KEEP_LOGITS = 0x1
CB_FLAG_STAGE_TIMING = 0x2
CB_FLAG_TEST_STALL = 0x4
CB_FLAG_TEST_STALL_DISPATCH = 0x8
CB_FLAG_GUARDS = 0x10
CB_N_STAGES = 5
STAGE_NAMES = ("router", "dispatch", "gateup_gemm", "down_gemm", "combine")

# every symbol include/cb_moe.h declares
ABI_SYMBOLS = ("cb_moe_init", "cb_moe_forward", "cb_moe_forward_f32out", "cb_moe_forward_host",
               "cb_moe_routing", "cb_moe_stage_times", "cb_moe_last_error", "cb_moe_device_bytes",
               "cb_moe_free", "cb_status_string", "cb_moe_dispatch_noalloc", "cb_moe_kernels_per_forward",
               "cb_moe_set_stage_timing", "cb_moe_check_guards")


CB_ROUTER_SOFTMAX_TOPK, CB_ROUTER_RAW_LOGITS, CB_ROUTER_HASH = 0, 1, 2
CB_MAX_HASH_DIMS = 8
ROUTER_MODES = {"softmax": CB_ROUTER_SOFTMAX_TOPK, "raw": CB_ROUTER_RAW_LOGITS, "hash": CB_ROUTER_HASH}


class cb_moe_config_t(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int32), ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32), ("wdtype", ctypes.c_int32),
                ("device", ctypes.c_int32), ("flags", ctypes.c_uint32), ("router_mode", ctypes.c_int32),
                ("hash_dims", ctypes.c_int32)]


class cb_moe_weights_t(ctypes.Structure):
    _fields_ = [("w_router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("s_gate", ctypes.c_void_p), ("s_up", ctypes.c_void_p), ("s_down", ctypes.c_void_p),
                ("w_hash", ctypes.c_void_p),
                ("z_gate", ctypes.c_void_p), ("z_up", ctypes.c_void_p), ("z_down", ctypes.c_void_p)]


class cb_routing_view_t(ctypes.Structure):
    _fields_ = [("ids", ctypes.c_void_p), ("w", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("tok", ctypes.c_void_p), ("inv", ctypes.c_void_p),
                ("logits", ctypes.c_void_p), ("tile_offsets", ctypes.c_void_p)]


class CbMoeError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {cb_status_string(status)} (status {status})")


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libcbmoe.so (build it first with __graft_entry__.build() or build.py)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libcbmoe.so is not built ({path}); run mixture_experts_router_gb300/build.py")
    lib = ctypes.CDLL(path)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    lib.cb_moe_init.argtypes = [ctypes.POINTER(cb_moe_config_t), ctypes.POINTER(cb_moe_weights_t),
                                ctypes.POINTER(vp)]
    lib.cb_moe_forward.argtypes = [vp, vp, vp, vp]
    lib.cb_moe_forward_f32out.argtypes = [vp, vp, vp, vp]
    lib.cb_moe_forward_host.argtypes = [vp, vp, vp, vp]
    lib.cb_moe_routing.argtypes = [vp, ctypes.POINTER(cb_routing_view_t)]
    lib.cb_moe_stage_times.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.c_int32]
    lib.cb_moe_last_error.argtypes = [vp]
    lib.cb_moe_check_guards.argtypes = [vp]
    lib.cb_moe_device_bytes.argtypes = [ctypes.POINTER(cb_moe_config_t), ctypes.POINTER(ctypes.c_uint64)]
    lib.cb_moe_free.argtypes = [vp]
    lib.cb_moe_kernels_per_forward.argtypes = [vp, ctypes.POINTER(i32)]
    lib.cb_moe_set_stage_timing.argtypes = [vp, i32]
    lib.cb_moe_dispatch_noalloc.argtypes = [vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vp, vp, vp, vp,
                                            vp, vp]
    lib.cb_moe_dispatch_noalloc.restype = i32
    for name in ("cb_moe_init", "cb_moe_forward", "cb_moe_forward_f32out", "cb_moe_forward_host",
                 "cb_moe_routing", "cb_moe_stage_times", "cb_moe_last_error", "cb_moe_device_bytes",
                 "cb_moe_free", "cb_moe_kernels_per_forward", "cb_moe_set_stage_timing", "cb_moe_check_guards"):
        getattr(lib, name).restype = i32
    lib.cb_status_string.argtypes = [i32]
    lib.cb_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


# --------------------------------------------------------- same-name calls
def cb_status_string(status: int) -> str:
    return load_library().cb_status_string(int(status)).decode()


def cb_moe_init(cfg: cb_moe_config_t, weights: cb_moe_weights_t):
    """Returns (status, handle); handle is None unless status == CB_OK."""
    h = ctypes.c_void_p()
    st = load_library().cb_moe_init(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(h))
    return st, (h.value if st == CB_OK else None)


def cb_moe_forward(handle, x_ptr: int, out_ptr: int, stream: int = 0) -> int:
    return load_library().cb_moe_forward(handle, x_ptr, out_ptr, stream)


def cb_moe_forward_f32out(handle, x_ptr: int, out_ptr: int, stream: int = 0) -> int:
    return load_library().cb_moe_forward_f32out(handle, x_ptr, out_ptr, stream)


def cb_moe_forward_host(handle, x_host_ptr: int, out_host_ptr: int, stream: int = 0) -> int:
    return load_library().cb_moe_forward_host(handle, x_host_ptr, out_host_ptr, stream)


def cb_moe_routing(handle):
    v = cb_routing_view_t()
    st = load_library().cb_moe_routing(handle, ctypes.byref(v))
    return st, v


def cb_moe_stage_times(handle):
    """Returns (status, [router, dispatch, gate/up, down, combine] ms)."""
    ms = (ctypes.c_float * CB_N_STAGES)()
    st = load_library().cb_moe_stage_times(handle, ms, CB_N_STAGES)
    return st, list(ms)


def cb_moe_last_error(handle) -> int:
    return load_library().cb_moe_last_error(handle)


def cb_moe_check_guards(handle) -> int:
    return load_library().cb_moe_check_guards(handle)


def cb_moe_device_bytes(cfg: cb_moe_config_t):
    b = ctypes.c_uint64()
    st = load_library().cb_moe_device_bytes(ctypes.byref(cfg), ctypes.byref(b))
    return st, b.value


def cb_moe_kernels_per_forward(handle):
    n = ctypes.c_int32()
    st = load_library().cb_moe_kernels_per_forward(handle, ctypes.byref(n))
    return st, n.value


def cb_moe_free(handle) -> int:
    return load_library().cb_moe_free(handle)


def cb_moe_dispatch_noalloc(ids_ptr, n_tokens, top_k, n_experts, counts_ptr, offsets_ptr, tok_ptr, inv_ptr,
                            status_ptr=None, stream: int = 0) -> int:
    """Dispatch of routing ids with no device allocation (static scratch); see cb_moe.h."""
    return load_library().cb_moe_dispatch_noalloc(ids_ptr, n_tokens, top_k, n_experts, counts_ptr, offsets_ptr,
                                                  tok_ptr, inv_ptr, status_ptr, stream)


# ------------------------------------------------------- torch convenience
_cudart = None


def copy_from_device(dst_tensor, src_ptr: int, nbytes: int) -> None:
    """Copy nbytes of library-owned device memory (e.g. a cb_routing_view_t
    array) into a torch CUDA tensor, with the CUDA runtime torch has loaded."""
    global _cudart
    if _cudart is None:
        import glob
        import sys
        names = ["libcudart.so.13", "libcudart.so.12", "libcudart.so"]
        for p in sys.path:
            names += glob.glob(os.path.join(p, "nvidia", "cu*", "lib", "libcudart.so*"))
            names += glob.glob(os.path.join(p, "nvidia", "cuda_runtime", "lib", "libcudart.so*"))
        names += glob.glob("/usr/local/cuda/lib64/libcudart.so*")
        for n in names:
            try:
                lib = ctypes.CDLL(n)
                break
            except OSError:
                continue
        else:
            raise RuntimeError("no CUDA runtime library found")
        lib.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
        lib.cudaMemcpy.restype = ctypes.c_int
        _cudart = lib
    if nbytes:
        rc = _cudart.cudaMemcpy(dst_tensor.data_ptr(), src_ptr, nbytes, 3)  # device to device
        if rc != 0:
            raise RuntimeError(f"cudaMemcpy failed ({rc})")


def _ptr(t):
    return None if t is None else t.data_ptr()


class MoELayer:
    """One layer handle over torch device tensors (bf16 as torch.bfloat16 or int16 bits,
    int8 as torch.int8, e4m3 as uint8 bytes or torch.float8_e4m3fn).  Raises CbMoeError on
    any non-zero status."""

    def __init__(self, T, d, f, E, k, w_router, w_gate, w_up, w_down, router_bias=None,
                 s_gate=None, s_up=None, s_down=None, device=0, keep_logits=False, stage_timing=False,
                 flags=0, router="softmax", w_hash=None, z_gate=None, z_up=None, z_down=None, wdtype=None):
        """Expert weights: bf16; int8 codes with scales (s_*); packed int4 codes (two per
        byte along the input dimension) with scales and uint8 zero points (z_*); or e4m3
        bytes with scales (wdtype="fp8", or weights of dtype torch.float8_e4m3fn).  Without
        `wdtype` the format follows from which of s_* and z_* are given."""
        flags |= (CB_FLAG_KEEP_LOGITS if keep_logits else 0) | (CB_FLAG_STAGE_TIMING if stage_timing else 0)
        mode = ROUTER_MODES[router]
        hash_dims = 0 if w_hash is None else int(w_hash.shape[0])
        if wdtype is None:
            fp8 = str(getattr(w_gate, "dtype", "")).endswith("float8_e4m3fn")
            wdtype = (CB_W_INT4 if z_gate is not None else CB_W_FP8 if fp8 else
                      CB_W_INT8 if s_gate is not None else CB_W_BF16)
        elif isinstance(wdtype, str):
            wdtype = WDTYPES[wdtype]
        self.cfg = cb_moe_config_t(T, d, f, E, k, wdtype, device, flags, mode, hash_dims)
        w = cb_moe_weights_t(_ptr(w_router), _ptr(router_bias), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                             _ptr(s_gate), _ptr(s_up), _ptr(s_down), _ptr(w_hash),
                             _ptr(z_gate), _ptr(z_up), _ptr(z_down))
        st, h = cb_moe_init(self.cfg, w)
        if st != CB_OK:
            raise CbMoeError(st, "cb_moe_init")
        self.handle = h

    def forward(self, x, out, stream=None, f32out=False):
        s = 0 if stream is None else stream.cuda_stream
        fn = cb_moe_forward_f32out if f32out else cb_moe_forward
        st = fn(self.handle, x.data_ptr(), out.data_ptr(), s)
        if st != CB_OK:
            raise CbMoeError(st, "cb_moe_forward")
        return out

    def forward_host(self, x_host, out_host, stream=None):
        s = 0 if stream is None else stream.cuda_stream
        st = cb_moe_forward_host(self.handle, x_host.data_ptr(), out_host.data_ptr(), s)
        if st != CB_OK:
            raise CbMoeError(st, "cb_moe_forward_host")
        return out_host

    def routing(self):
        st, v = cb_moe_routing(self.handle)
        if st != CB_OK:
            raise CbMoeError(st, "cb_moe_routing")
        return v

    def stage_times(self):
        st, ms = cb_moe_stage_times(self.handle)
        if st != CB_OK:
            raise CbMoeError(st, "cb_moe_stage_times")
        return ms

    def set_stage_timing(self, on: bool):
        """Stage events on or off for later forwards (handle made with stage_timing=True)."""
        st = load_library().cb_moe_set_stage_timing(self.handle, 1 if on else 0)
        if st != CB_OK:
            raise CbMoeError(st, "cb_moe_set_stage_timing")

    def last_error(self) -> int:
        return cb_moe_last_error(self.handle)

    def check_guards(self) -> int:
        """CB_OK when every guard band of a CB_FLAG_GUARDS handle is intact."""
        return cb_moe_check_guards(self.handle)

    def kernels_per_forward(self) -> int:
        st, n = cb_moe_kernels_per_forward(self.handle)
        if st != CB_OK:
            raise CbMoeError(st, "cb_moe_kernels_per_forward")
        return n

    def close(self):
        if getattr(self, "handle", None) is not None:
            st = cb_moe_free(self.handle)
            self.handle = None
            if st != CB_OK:
                raise CbMoeError(st, "cb_moe_free")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
