"""The C ABI without a GPU: the library builds and loads, exports every symbol
include/cb_moe.h declares, and rejects bad configurations before any CUDA call."""
import ctypes
import os
import re

import pytest

import mixture_experts_router_gb300 as cb
from mixture_experts_router_gb300 import build as cbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cb_moe.h")


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return cb.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CB_API\s+[\w\s\*]*?\b(cb_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    assert declared_symbols() == sorted(cb.ABI_SYMBOLS)


def test_header_constants_match_the_binding():
    """Every CB_FLAG_* and the weight-format, router-mode and status enumerators of the
    header have the values the Python binding uses."""
    text = open(HEADER).read()
    flags = {n: int(v, 16) for n, v in re.findall(r"#define\s+(CB_FLAG_\w+)\s+(0x[0-9a-fA-F]+)u", text)}
    assert flags and all(getattr(cb, n) == v for n, v in flags.items()), flags
    enums = dict((n, int(v)) for n, v in re.findall(r"\b(CB_(?:W|ROUTER|OK|ERR)\w*)\s*=\s*(\d+)", text))
    for name in ("CB_W_BF16", "CB_W_INT8", "CB_W_INT4", "CB_W_FP8", "CB_OK", "CB_ERR_TIMEOUT", "CB_ERR_DEVICE"):
        assert name in enums and getattr(cb, name) == enums[name], name
    assert cb.WDTYPES == {"bf16": 0, "int8": 1, "int4": 2, "fp8": 3}


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(cb.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(raw, name), name


def test_status_strings(lib):
    for code in range(8):
        assert cb.cb_status_string(code) not in ("", "unknown status")
    assert cb.cb_status_string(99) == "unknown status"


def cfg(**kw):
    base = dict(n_tokens=64, d_model=256, d_ff=512, n_experts=8, top_k=2, wdtype=0, device=0, flags=0)
    base.update(kw)
    return cb.cb_moe_config_t(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(), cb.CB_OK),
    (dict(n_tokens=0), cb.CB_OK),
    (dict(n_tokens=-1), cb.CB_ERR_INVALID_ARG),
    (dict(top_k=9), cb.CB_ERR_INVALID_ARG),
    (dict(top_k=0), cb.CB_ERR_INVALID_ARG),
    (dict(d_model=384), cb.CB_ERR_UNSUPPORTED),
    (dict(d_ff=254), cb.CB_ERR_UNSUPPORTED),
    (dict(n_experts=257, top_k=2), cb.CB_ERR_UNSUPPORTED),
    (dict(n_experts=32, top_k=17), cb.CB_ERR_UNSUPPORTED),
    (dict(wdtype=5), cb.CB_ERR_INVALID_ARG),
    (dict(wdtype=4), cb.CB_ERR_INVALID_ARG),
    (dict(wdtype=3), cb.CB_OK),
    (dict(flags=0x8), cb.CB_OK),
    (dict(flags=0x10), cb.CB_OK),
    (dict(flags=0x20), cb.CB_ERR_INVALID_ARG),
    (dict(flags=0x80), cb.CB_ERR_INVALID_ARG),
    (dict(router_mode=1), cb.CB_OK),
    (dict(router_mode=2, top_k=1, hash_dims=8), cb.CB_OK),
    (dict(router_mode=3), cb.CB_ERR_INVALID_ARG),
    (dict(router_mode=-1), cb.CB_ERR_INVALID_ARG),
    (dict(router_mode=2, top_k=2, hash_dims=4), cb.CB_ERR_INVALID_ARG),
    (dict(router_mode=2, top_k=1, hash_dims=0), cb.CB_ERR_INVALID_ARG),
    (dict(router_mode=2, top_k=1, hash_dims=9), cb.CB_ERR_INVALID_ARG),
])
def test_config_validation(lib, kw, status):
    st, nbytes = cb.cb_moe_device_bytes(cfg(**kw))
    assert st == status
    if status == cb.CB_OK:
        assert nbytes > 0


def test_device_bytes_cover_the_workspace(lib):
    # mixtral prefill: 2 x 3 x 8 x 4096 x 14336 weight bytes plus activations
    st, nbytes = cb.cb_moe_device_bytes(cfg(n_tokens=4096, d_model=4096, d_ff=14336, n_experts=8, top_k=2))
    assert st == cb.CB_OK
    weights = 3 * 8 * 4096 * 14336 * 2
    assert weights < nbytes < weights + 2 * 10**9


def test_device_bytes_by_weight_format(lib):
    """fp8 and int8 experts take one byte per weight (plus the same fp32 scales), int4 half a
    byte plus uint8 zero points, bf16 two bytes."""
    big = dict(n_tokens=64, d_model=1024, d_ff=2048, n_experts=8, top_k=2)
    sizes = {w: cb.cb_moe_device_bytes(cfg(wdtype=w, **big)) for w in (0, 1, 2, 3)}
    assert all(st == cb.CB_OK for st, _ in sizes.values())
    n_w = 3 * 8 * 1024 * 2048
    assert sizes[3][1] == sizes[1][1]
    assert abs((sizes[0][1] - sizes[1][1]) - n_w) < 64 * 1024 + 8 * 3 * 2048 * 4
    assert sizes[2][1] < sizes[1][1]


def test_device_bytes_with_guard_bands(lib):
    """CB_FLAG_GUARDS adds a 4096-byte band after each non-empty workspace region."""
    st, plain = cb.cb_moe_device_bytes(cfg())
    st2, guarded = cb.cb_moe_device_bytes(cfg(flags=cb.CB_FLAG_GUARDS))
    assert st == st2 == cb.CB_OK
    extra = guarded - plain
    assert extra % 4096 == 0 and 20 <= extra // 4096 <= 48


def test_device_bytes_hold_the_hash_projection(lib):
    st, plain = cb.cb_moe_device_bytes(cfg(top_k=1))
    st2, hashed = cb.cb_moe_device_bytes(cfg(top_k=1, router_mode=2, hash_dims=3))
    assert st == st2 == cb.CB_OK
    assert 3 * 256 * 4 <= hashed - plain <= 3 * 256 * 4 + 256   # W_h kept in fp32


def test_init_rejects_bad_arguments_before_cuda(lib):
    w = cb.cb_moe_weights_t()
    st, h = cb.cb_moe_init(cfg(d_model=300), w)
    assert st == cb.CB_ERR_UNSUPPORTED and h is None
    st, h = cb.cb_moe_init(cfg(), w)                 # NULL weight pointers
    assert st == cb.CB_ERR_INVALID_ARG and h is None
    w = cb.cb_moe_weights_t(w_router=16, w_gate=32, w_up=48, w_down=66)   # misaligned
    st, h = cb.cb_moe_init(cfg(), w)
    assert st == cb.CB_ERR_ALIGNMENT
    w = cb.cb_moe_weights_t(w_router=16, w_gate=32, w_up=48, w_down=64)
    st, h = cb.cb_moe_init(cfg(wdtype=1), w)         # int8 without scales
    assert st == cb.CB_ERR_UNSUPPORTED
    st, h = cb.cb_moe_init(cfg(top_k=1, router_mode=2, hash_dims=4), w)   # hash router without W_h
    assert st == cb.CB_ERR_INVALID_ARG and h is None
    w = cb.cb_moe_weights_t(w_router=16, w_gate=32, w_up=48, w_down=64, w_hash=72)
    st, h = cb.cb_moe_init(cfg(top_k=1, router_mode=2, hash_dims=4), w)   # misaligned W_h
    assert st == cb.CB_ERR_ALIGNMENT
    assert cb.cb_moe_forward(None, 16, 32, 0) == cb.CB_ERR_INVALID_ARG
    assert cb.cb_moe_free(None) == cb.CB_OK
