"""The method's edge cases on the GPU, each with an answer fixed outside the oracle.

* Exact logit ties.  x and W_r take values on a coarse grid (x in {-2..2},
  W_r in {-1, 0, 1}/64, some router rows duplicated), so every logit is a small
  multiple of 1/64 that fp32 and fp64 both hold exactly: GPU and oracle logits
  are equal, a third or more of the tokens tie exactly at the k-th place, and
  every other gap is at least 1/64.  No token may be excused: at a tie the
  lower expert index wins, in the set and in the slot order (the gate of
  "Colibri：面向MoE模型的高性能C语言推理引擎" §2.1, ties read as going to the
  lower index).
* Zero router weights with equal biases: every expert ties, so each token takes
  experts 0..k-1 with weight 1/k.
* Identical experts: the gate weights sum to one, so the layer equals one dense
  SwiGLU FFN (numpy matmul + scipy expit on the decoded weights, h rounded to
  bf16 by torch), whatever the routing.
* A one-hot router (bias +100 on expert j): every token goes to j with weight
  exactly 1, and the layer equals expert j's dense FFN.
* Zero input: SiLU(0) * 0 = 0, so the output is exactly zero.
* Softmax with k = 1 over 8 experts: w = exp(0) / exp(0) = 1 exactly, the
  expert is the arg-max of the fp64 logits (numpy, first index on ties), and
  the output is that expert's dense FFN.

Each case runs on both routers (mma.sync for E <= 16, tcgen05 above, or forced
by CB_MOE_ROUTER) and, where it concerns the expert GEMMs, on the bf16 1-CTA
and CTA-pair kernels and the int8 / int4 / fp8 tensor-memory kernels.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

import synth

pytestmark = pytest.mark.gpu

gh = pytest.importorskip("gpu_harness")


# ----------------------------------------------------------------- helpers
def bf16_bits(v):
    """bf16 bit patterns of values that bf16 holds exactly (checked)."""
    f = np.asarray(v, np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(synth.bf16_bits_to_f32(bits), f), "value not on the bf16 grid"
    return bits


def grid_router(rng, T, d, E):
    """x in {-2..2} and W_r in {-1, 0, 1}/64, router rows 3j+1 copies of 3j."""
    x = rng.choice([-2, -1, 0, 1, 2], size=(T, d), p=[.1, .2, .4, .2, .1]).astype(np.float32)
    wr = (rng.choice([-1, 0, 1], size=(E, d), p=[.1, .8, .1]) / 64.0).astype(np.float32)
    for e in range(1, E, 3):
        wr[e] = wr[e - 1]
    return x, wr


def make_layer(shape, x=None, wr=None, bias=None, same_experts=False):
    """The synthetic layer of `shape` with x, W_r or the bias replaced, or with
    every expert a copy of expert 0."""
    layer = synth.make_layer(shape)
    if x is not None:
        layer.x = bf16_bits(x)
    if wr is not None:
        layer.wr = bf16_bits(wr)
    if bias is not None:
        layer.bias = np.asarray(bias, np.float32)
        layer.shape = synth.Shape(shape.name, shape.T, shape.d, shape.f, shape.E, shape.k, shape.wdtype, True,
                                  shape.seed)
    if same_experts:
        for n in ("wg", "wu", "wd", "sg", "su", "sd", "zg", "zu", "zd"):
            a = getattr(layer, n)
            if a is not None:
                setattr(layer, n, np.ascontiguousarray(np.broadcast_to(a[:1], a.shape)))
    return layer


def decoded_expert(layer, e):
    """Expert e's weights as float64 [f][d], [f][d], [d][f] from the stored
    format (int8 q s; int4 (q - z) s with the low nibble first; e4m3 through
    torch's float8_e4m3fn; bf16 widened)."""
    wd = layer.shape.wdtype

    def dec(w, s, z):
        if wd == "bf16":
            return synth.bf16_bits_to_f32(w[e]).astype(np.float64)
        if wd == "int8":
            q = w[e].astype(np.float64)
        elif wd == "int4":
            q = synth.unpack_int4(w[e]).astype(np.float64) - z[e].astype(np.float64)[:, None]
        else:
            q = torch.from_numpy(np.ascontiguousarray(w[e])).view(torch.float8_e4m3fn).double().numpy()
        return q * s[e].astype(np.float64)[:, None]

    return (dec(layer.wg, layer.sg, layer.zg), dec(layer.wu, layer.su, layer.zu),
            dec(layer.wd, layer.sd, layer.zd))


def dense_ffn(xv, wg, wu, wd):
    """Dense SwiGLU FFN in float64 with h rounded to bf16 (torch) before the
    down projection, as the layer's intermediate H is stored."""
    g = xv @ wg.T
    u = xv @ wu.T
    h = torch.from_numpy(g * expit(g) * u).to(torch.bfloat16).double().numpy()
    return h @ wd.T


def check_against(gl, ref, report):
    """The layer's fp32 and bf16 outputs against a reference, with the bounds
    the parity tests use."""
    o32 = gl.out32.cpu().numpy().astype(np.float64)
    o16 = gh.bf16_to_f64(gl.out)
    err32 = np.abs(o32 - ref)
    err16 = np.abs(o16 - ref)
    report.update(f32_max_abs=float(err32.max()), bf16_max_abs=float(err16.max()),
                  f32_mean_rel=float(err32.sum() / np.abs(ref).sum()),
                  bf16_mean_rel=float(err16.sum() / np.abs(ref).sum()))
    assert err32.max() <= gh.MAX_ABS, report
    assert np.all(err16 <= gh.MAX_ABS + gh.half_ulp_bf16(ref)), report
    assert report["f32_mean_rel"] <= gh.MEAN_REL and report["bf16_mean_rel"] <= gh.MEAN_REL, report


def run_layer(layer):
    gl = gh.GpuLayer(layer)
    gl.run()
    return gl


# mma: the mma.sync router (E <= 16: in one launch with the dispatch); tc: the
# tcgen05 router (17..256 experts: in one launch with the dispatch);
# tc-separate: the split-K tcgen05 router and top-k kernels, then the dispatch
ROUTERS = ["mma", "tc", "tc-separate"]


def set_router(monkeypatch, router):
    monkeypatch.setenv("CB_MOE_ROUTER", router.split("-")[0])
    if router.endswith("-separate"):
        monkeypatch.setenv("CB_MOE_ROUTE_DISPATCH", "0")


# ------------------------------------------------------------- exact ties
TIE_SHAPES = {
    "e8_k2": dict(T=2000, d=256, f=256, E=8, k=2),
    "e8_k3": dict(T=2000, d=256, f=256, E=8, k=3),
    "e16_k4": dict(T=1000, d=256, f=256, E=16, k=4),
    "e40_k3": dict(T=1000, d=512, f=256, E=40, k=3),
    "e128_k4": dict(T=1000, d=1024, f=256, E=128, k=4),
    "e256_k16": dict(T=300, d=256, f=256, E=256, k=16),
}


@pytest.mark.parametrize("router", ROUTERS)
@pytest.mark.parametrize("name", list(TIE_SHAPES))
def test_exact_logit_ties_go_to_the_lower_index(name, router, monkeypatch):
    set_router(monkeypatch, router)
    shape = synth.custom_shape("ties_" + name, seed=81, **TIE_SHAPES[name])
    x, wr = grid_router(np.random.default_rng(81), shape.T, shape.d, shape.E)
    rep = gh.full_check(make_layer(shape, x=x, wr=wr))
    print(name, router, rep)
    assert rep["logit_max_err"] == 0.0          # both sides hold the grid logits exactly
    assert rep["near_tie_tokens"] == 0           # nothing is excused
    assert rep["exact_tie_tokens"] >= shape.T // 5


@pytest.mark.parametrize("router", ROUTERS)
@pytest.mark.parametrize("E,k,bias", [(8, 2, 0.25), (8, 3, None), (40, 3, -1.5), (256, 16, 0.0)])
def test_zero_router_weights_equal_bias(E, k, bias, router, monkeypatch):
    """Every expert ties: experts 0..k-1 in slot order, w = 1/k."""
    set_router(monkeypatch, router)
    shape = synth.custom_shape(f"zero_router_e{E}", T=333, d=256, f=256, E=E, k=k, seed=82)
    layer = make_layer(shape, wr=np.zeros((E, 256), np.float32),
                       bias=None if bias is None else np.full(E, bias, np.float32))
    gl = run_layer(layer)
    try:
        r = gl.routing()
        assert np.array_equal(r["ids"], np.broadcast_to(np.arange(k, dtype=np.int32), (shape.T, k)))
        assert np.abs(r["w"] - 1.0 / k).max() <= 1e-7
    finally:
        gl.close()
    rep = gh.full_check(layer)
    assert rep["exact_tie_tokens"] == shape.T


# ------------------------------------------------------------ NaN logits
BF16_NAN = 0x7FC0


@pytest.mark.parametrize("router", ROUTERS)
@pytest.mark.parametrize("E,k", [(8, 2), (40, 3)])
def test_nan_logits_rank_after_every_number(E, k, router, monkeypatch):
    """A router row of NaN (expert 5's logit NaN for every token) and a token
    whose x is NaN (all its logits NaN).  NaN ranks after every number and,
    among NaNs, the lower index first: expert 5 is never chosen while numbers
    are left, and the NaN token takes experts 0..k-1 in slot order with NaN
    weights.  Every other token's ids (slot order) and weights match the
    oracle's; with this seed no other token has a gap below 2e-4."""
    import oracle
    set_router(monkeypatch, router)
    shape = synth.custom_shape(f"nan_e{E}_k{k}", T=200, d=256, f=256, E=E, k=k, seed=89)
    layer = synth.make_layer(shape)
    layer.wr = layer.wr.copy()
    layer.wr[5, :] = BF16_NAN
    layer.x = layer.x.copy()
    layer.x[7, :] = BF16_NAN
    oids, ow, _, _ = oracle.Oracle(layer).route()
    gl = run_layer(layer)
    try:
        r = gl.routing()
        ids, w = r["ids"], r["w"]
        assert np.array_equal(ids[7], np.arange(k, dtype=np.int32))
        assert np.all(np.isnan(w[7]))
        rest = np.arange(shape.T) != 7
        assert not np.any(ids[rest] == 5)
        assert np.array_equal(ids, oids)
        assert np.abs(w[rest] - ow[rest]).max() <= 1e-5
    finally:
        gl.close()


# --------------------------------------------------------- closed forms
IDENTICAL = [  # (name, shape kwargs, environment)
    ("bf16_e8", dict(T=300, d=512, f=768, E=8, k=2), {}),
    ("bf16_pairs", dict(T=600, d=512, f=768, E=4, k=2), {"CB_MOE_PAIR": "1"}),
    ("bf16_e40_tc", dict(T=500, d=512, f=256, E=40, k=3), {}),
    ("bf16_e8_tc", dict(T=300, d=512, f=768, E=8, k=2), {"CB_MOE_ROUTER": "tc"}),
    ("int8", dict(T=700, d=256, f=512, E=64, k=6, wdtype="int8"), {}),
    ("int8_pairs", dict(T=1100, d=512, f=768, E=4, k=2, wdtype="int8"), {}),
    ("int4", dict(T=700, d=256, f=512, E=64, k=6, wdtype="int4"), {}),
    ("fp8", dict(T=1100, d=512, f=768, E=4, k=2, wdtype="fp8"), {}),
]


@pytest.mark.parametrize("name,kw,env", IDENTICAL, ids=[c[0] for c in IDENTICAL])
def test_identical_experts_equal_one_dense_ffn(name, kw, env, monkeypatch):
    for key, v in env.items():
        monkeypatch.setenv(key, v)
    shape = synth.custom_shape("same_" + name, seed=83, **kw)
    layer = make_layer(shape, same_experts=True)
    xv = synth.bf16_bits_to_f32(layer.x).astype(np.float64)
    ref = dense_ffn(xv, *decoded_expert(layer, 0))
    gl = run_layer(layer)
    try:
        rep = {}
        check_against(gl, ref, rep)
        print(name, rep)
    finally:
        gl.close()


@pytest.mark.parametrize("name,kw,env", [
    ("e8_k2", dict(T=300, d=512, f=768, E=8, k=2), {}),
    ("e40_k3_tc", dict(T=400, d=512, f=256, E=40, k=3), {}),
    ("e8_k2_pairs", dict(T=600, d=512, f=768, E=8, k=2), {"CB_MOE_PAIR": "1"}),
    ("int4_e8", dict(T=300, d=512, f=768, E=8, k=2, wdtype="int4"), {}),
], ids=lambda v: v if isinstance(v, str) else "")
def test_one_hot_router_gives_that_expert_alone(name, kw, env, monkeypatch):
    for key, v in env.items():
        monkeypatch.setenv(key, v)
    shape = synth.custom_shape("onehot_" + name, seed=84, **kw)
    j = shape.E - 3
    bias = np.zeros(shape.E, np.float32)
    bias[j] = 100.0
    layer = make_layer(shape, bias=bias)
    xv = synth.bf16_bits_to_f32(layer.x).astype(np.float64)
    ref = dense_ffn(xv, *decoded_expert(layer, j))
    gl = run_layer(layer)
    try:
        r = gl.routing()
        assert np.all(r["ids"][:, 0] == j)
        assert np.all(r["w"][:, 0] == np.float32(1.0))
        rep = {}
        check_against(gl, ref, rep)
        print(name, rep)
    finally:
        gl.close()


@pytest.mark.parametrize("wdtype", ["bf16", "int8", "int4", "fp8"])
@pytest.mark.parametrize("E,k", [(8, 2), (40, 3)])
def test_zero_input_gives_zero_output(E, k, wdtype):
    shape = synth.custom_shape(f"zero_x_{wdtype}", T=300, d=512, f=512, E=E, k=k, wdtype=wdtype, seed=85)
    layer = make_layer(shape, x=np.zeros((shape.T, shape.d), np.float32))
    gl = run_layer(layer)
    try:
        assert torch.count_nonzero(gl.out32).item() == 0
        assert torch.count_nonzero(gl.out.float()).item() == 0
        r = gl.routing()
        assert np.array_equal(r["ids"], np.broadcast_to(np.arange(k, dtype=np.int32), (shape.T, k)))
    finally:
        gl.close()


@pytest.mark.parametrize("router", ROUTERS)
@pytest.mark.parametrize("wdtype", ["bf16", "int8"])
def test_softmax_top1_weight_is_exactly_one(wdtype, router, monkeypatch):
    set_router(monkeypatch, router)
    shape = synth.custom_shape(f"top1_{wdtype}", T=500, d=512, f=768, E=8, k=1, wdtype=wdtype, seed=86)
    layer = make_layer(shape)
    xv = synth.bf16_bits_to_f32(layer.x).astype(np.float64)
    logits = xv @ synth.bf16_bits_to_f32(layer.wr).astype(np.float64).T
    want = np.argmax(logits, axis=1)
    ref = np.zeros((shape.T, shape.d))
    for e in np.unique(want):
        rows = want == e
        ref[rows] = dense_ffn(xv[rows], *decoded_expert(layer, e))
    gl = run_layer(layer)
    try:
        r = gl.routing()
        assert np.array_equal(r["ids"][:, 0], want)
        assert np.all(r["w"] == np.float32(1.0))
        rep = {}
        check_against(gl, ref, rep)
        print(wdtype, router, rep)
    finally:
        gl.close()
