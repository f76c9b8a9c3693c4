"""Pins of the fp64 oracle to facts fixed outside the oracle itself.

Each ``pin_*`` takes a loaded oracle library (``oracle.load(path)``) and
raises AssertionError when the oracle disagrees with a closed form, a brute
force, a special case that reduces to a textbook dense SwiGLU FFN written
with numpy / scipy library routines, or the hand-derived worked example in
``tests/golden/tiny_layer.json``.  The same pins run against deliberately
broken copies of the oracle (``test_oracle_mutants.py``) to show that each
plausible mistake is caught by at least one of them.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
from scipy.special import expit, softmax

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_layer.json")
GOLDEN_ROUTERS = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "router_variants.json")


# ----------------------------------------------------------------- helpers
def f32_to_bf16_bits(a):
    """float32 values that are already bf16 numbers -> their bit patterns."""
    a = np.asarray(a, dtype=np.float32)
    bits = a.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "value not on the bf16 grid"
    return (bits >> 16).astype(np.uint16)


def bf16_bits_to_f64(b):
    return synth.bf16_bits_to_f32(np.asarray(b, dtype=np.uint16)).astype(np.float64)


def make_layer_from_values(x, wr, wg, wu, wd, k, bias=None, wdtype="bf16", sg=None, su=None, sd=None,
                           router="softmax", wh=None, zg=None, zu=None, zd=None):
    """A synth.Layer from explicit values (bf16-exact floats, int8 codes, or packed int4
    bytes with uint8 zero points)."""
    x = np.asarray(x, np.float64)
    wr = np.asarray(wr, np.float64)
    T, d = x.shape
    E = wr.shape[0]
    wg_a = np.asarray(wg)
    f = wg_a.shape[1]
    if wdtype == "int4":
        d = 2 * wg_a.shape[2]
    hd = 0 if wh is None else np.asarray(wh).shape[0]
    shape = synth.Shape("custom", T=T, d=d, f=f, E=E, k=k, wdtype=wdtype, bias=bias is not None, router=router,
                        hash_dims=hd)
    conv = f32_to_bf16_bits
    if wdtype == "bf16":
        wgb, wub, wdb = conv(wg), conv(wu), conv(wd)
    elif wdtype in ("int4", "fp8"):
        wgb, wub, wdb = (np.asarray(a, np.uint8) for a in (wg, wu, wd))
    else:
        wgb = np.asarray(wg, np.int8)
        wub = np.asarray(wu, np.int8)
        wdb = np.asarray(wd, np.int8)
    b = None if bias is None else np.asarray(bias, np.float32)
    return synth.Layer(shape, conv(x), conv(wr), b, wgb, wub, wdb,
                       None if sg is None else np.asarray(sg, np.float32),
                       None if su is None else np.asarray(su, np.float32),
                       None if sd is None else np.asarray(sd, np.float32),
                       wh=None if wh is None else conv(wh),
                       zg=None if zg is None else np.asarray(zg, np.uint8),
                       zu=None if zu is None else np.asarray(zu, np.uint8),
                       zd=None if zd is None else np.asarray(zd, np.uint8))


def dense_swiglu(xv, wg, wu, wd):
    """Textbook dense SwiGLU FFN in float64 with numpy matmul and scipy expit:
    (silu(x Wg^T) * (x Wu^T)) Wd^T, Wg/Wu [f][d], Wd [d][f]."""
    g = xv @ wg.T
    u = xv @ wu.T
    return (g * expit(g) * u) @ wd.T


def rng_bf16(rng, shape, scale):
    """Random values on the bf16 grid (float32 truncated to 8 significant bits)."""
    v = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (v.view(np.uint32) & 0xFFFF0000).view(np.float32).astype(np.float64)


def _key(l, e):
    """Total order used by the brute force: numbers before NaN, larger first, lower index on ties."""
    v = l[e]
    return (1, 0.0, e) if math.isnan(v) else (0, -v, e)


# -------------------------------------------------------------------- pins
def pin_round_bf16(lib):
    # hand-picked doubles: exact ties go to even, anything past a tie rounds
    # away from it (catches rounding through float32 first)
    cases = [
        (1.0, 1.0), (1 + 2**-8, 1.0), (1 + 3 * 2**-8, 1 + 2**-6), (1 + 2**-8 + 2**-40, 1 + 2**-7),
        (-(1 + 2**-8 + 2**-40), -(1 + 2**-7)), (1 + 2**-9, 1.0), (255.5, 256.0), (254.5, 254.0),
        (3.0 * 2**-130, 3.0 * 2**-130), (2**-134, 0.0), (1.5 * 2**-133, 2 * 2**-133),
        (0.0, 0.0), (2.0**127 * 1.9921875, 2.0**127 * 1.9921875), (2.0**128 * 1.5, math.inf),
    ]
    for v, want in cases:
        got = lib.moe_oracle_round_bf16(v)
        assert got == want, f"round_bf16({v!r}) = {got!r}, want {want!r}"
    # float32 inputs against torch's float32 -> bfloat16 conversion (round to nearest even)
    import torch
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        (np.arange(1, 4000) * 2.0 ** -7 + 2.0 ** -9)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([lib.moe_oracle_round_bf16(float(a)) for a in v])
    assert np.array_equal(got, ref), "round_bf16 disagrees with torch's bf16 conversion"


def pin_gate_bruteforce(lib):
    rng = np.random.default_rng(1)
    for trial in range(600):
        E = int(rng.integers(1, 11))
        k = int(rng.integers(1, min(4, E) + 1))
        kind = trial % 4
        if kind == 0:
            l = rng.standard_normal(E)
        elif kind == 1:      # many exact duplicates
            l = rng.integers(-2, 3, E).astype(np.float64)
        elif kind == 2:      # signed zeros and infinities
            l = rng.choice([0.0, -0.0, 1.0, -math.inf, math.inf], E)
        else:                # NaNs mixed in
            l = rng.standard_normal(E)
            l[rng.random(E) < 0.3] = math.nan
        ids, w, gk, gs = oracle.gate(l, k, lib)
        # brute force: the unique k-subset whose every member precedes every non-member
        keys = [_key(l, e) for e in range(E)]
        winners = [S for S in itertools.combinations(range(E), k)
                   if all(keys[a] < keys[b] for a in S for b in range(E) if b not in S)]
        assert len(winners) == 1
        assert sorted(ids.tolist()) == list(winners[0]), (l, k, ids)
        # slot order follows the total order
        assert all(keys[ids[s]] < keys[ids[s + 1]] for s in range(k - 1)), (l, ids)
        if all(math.isfinite(a) for a in l):
            srt = sorted(range(E), key=lambda e: keys[e])
            want_gk = l[srt[k - 1]] - l[srt[k]] if k < E else math.inf
            assert gk == want_gk
            want_gs = min([l[srt[s]] - l[srt[s + 1]] for s in range(k - 1)], default=math.inf)
            assert gs == want_gs


def pin_gate_weights(lib):
    rng = np.random.default_rng(2)
    for _ in range(300):
        E = int(rng.integers(1, 65))
        k = int(rng.integers(1, min(8, E) + 1))
        l = rng.standard_normal(E) * rng.choice([0.1, 1.0, 10.0, 50.0])
        ids, w, _, _ = oracle.gate(l, k, lib)
        # closed form: the full softmax over all E, restricted to the k and renormalised
        p = softmax(l)
        want = p[ids] / p[ids].sum()
        assert np.allclose(w, want, rtol=1e-12, atol=1e-300), (w, want)
        assert abs(w.sum() - 1.0) <= 1e-12
        assert np.all(np.diff(w) <= 0)
        if k == 1:
            assert w[0] == 1.0
        # the chosen logits are the k largest
        assert np.isclose(np.sort(l)[::-1][:k], l[ids]).all()


def pin_dispatch(lib):
    rng = np.random.default_rng(3)
    for trial in range(60):
        E = int(rng.integers(1, 40))
        k = int(rng.integers(1, min(6, E) + 1))
        T = int(rng.integers(0, 300))
        if trial % 3 == 0:   # skewed popularity, some experts empty
            p = rng.random(E) ** 6
            ids = np.stack([rng.choice(E, k, replace=False, p=p / p.sum()) for _ in range(T)]).reshape(T, k) \
                if T else np.zeros((0, k), np.int32)
        else:
            ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).reshape(T, k) if T else np.zeros((0, k), np.int32)
        ids = ids.astype(np.int32)
        cnt, off, tok, inv = oracle.dispatch(ids, E, lib)
        # brute force with a library stable sort over (expert, token) pairs
        pairs = sorted(((int(ids[t, s]), t, s) for t in range(T) for s in range(k)))
        want_tok = np.array([t for _, t, _ in pairs], np.int32)
        want_inv = np.empty((T, k), np.int32)
        for r, (_, t, s) in enumerate(pairs):
            want_inv[t, s] = r
        assert np.array_equal(cnt, np.bincount(ids.ravel(), minlength=E))
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(cnt)]))
        assert np.array_equal(tok, want_tok)
        assert np.array_equal(inv, want_inv)
        assert off[-1] == T * k and np.all(np.diff(off) >= 0)
    # rejects ids out of range and a token holding one expert twice
    for bad in (np.array([[0, 5]], np.int32), np.array([[1, 1]], np.int32), np.array([[-1, 0]], np.int32)):
        cnt = np.empty(3, np.int32); off = np.empty(4, np.int32)
        tok = np.empty(2, np.int32); inv = np.empty(2, np.int32)
        assert lib.moe_oracle_dispatch(1, 3, 2, bad.ctypes.data, cnt.ctypes.data, off.ctypes.data,
                                       tok.ctypes.data, inv.ctypes.data) != 0


def _random_layer(rng, T, d, f, E, k, identical=False, bias=None):
    x = rng_bf16(rng, (T, d), 1.0)
    wr = rng_bf16(rng, (E, d), 0.3)
    if identical:
        wg = np.broadcast_to(rng_bf16(rng, (f, d), 0.2), (E, f, d)).copy()
        wu = np.broadcast_to(rng_bf16(rng, (f, d), 0.2), (E, f, d)).copy()
        wd = np.broadcast_to(rng_bf16(rng, (d, f), 0.2), (E, d, f)).copy()
    else:
        wg, wu, wd = rng_bf16(rng, (E, f, d), 0.2), rng_bf16(rng, (E, f, d), 0.2), rng_bf16(rng, (E, d, f), 0.2)
    return make_layer_from_values(x, wr, wg, wu, wd, k, bias=bias), (x, wr, wg, wu, wd)


def pin_identical_experts(lib):
    """All experts equal and the weights summing to 1 => one dense SwiGLU FFN."""
    rng = np.random.default_rng(4)
    for (T, d, f, E, k) in [(7, 16, 24, 4, 2), (5, 8, 40, 6, 3), (3, 32, 8, 2, 2)]:
        L, (x, wr, wg, wu, wd) = _random_layer(rng, T, d, f, E, k, identical=True)
        out, ids, w = oracle.Oracle(L, lib).forward(mode=oracle.EXACT)
        want = dense_swiglu(x, wg[0], wu[0], wd[0])
        assert np.allclose(out, want, rtol=1e-11, atol=1e-12), np.abs(out - want).max()


def pin_one_hot_router(lib):
    """A router bias of +100 on expert j (zero router weights) sends every token to j with w = 1."""
    rng = np.random.default_rng(5)
    T, d, f, E = 6, 16, 24, 5
    for j in range(E):
        L, (x, wr, wg, wu, wd) = _random_layer(rng, T, d, f, E, 1, bias=None)
        bias = np.zeros(E, np.float32); bias[j] = 100.0
        L = make_layer_from_values(x, np.zeros_like(wr), wg, wu, wd, 1, bias=bias)
        out, ids, w = oracle.Oracle(L, lib).forward(mode=oracle.EXACT)
        assert np.all(ids == j) and np.all(w == 1.0)
        want = dense_swiglu(x, wg[j], wu[j], wd[j])
        assert np.allclose(out, want, rtol=1e-11, atol=1e-12)


def pin_two_expert_mix(lib):
    """Zero router weights, bias [0, ln 3, -1, -2]: every token takes experts (1, 0) with
    weights sig(b1 - b0) and sig(b0 - b1), so out = sig(b1) FFN_1 + sig(-b1) FFN_0."""
    rng = np.random.default_rng(6)
    T, d, f, E, k = 5, 8, 12, 4, 2
    L, (x, wr, wg, wu, wd) = _random_layer(rng, T, d, f, E, k)
    bias = np.array([0.0, math.log(3.0), -1.0, -2.0], np.float32)
    L = make_layer_from_values(x, np.zeros_like(wr), wg, wu, wd, k, bias=bias)
    out, ids, w = oracle.Oracle(L, lib).forward(mode=oracle.EXACT)
    b1 = float(bias[1])
    assert np.all(ids == np.array([1, 0]))
    assert np.allclose(w, [expit(b1), expit(-b1)], rtol=1e-14)
    want = expit(b1) * dense_swiglu(x, wg[1], wu[1], wd[1]) + expit(-b1) * dense_swiglu(x, wg[0], wu[0], wd[0])
    assert np.allclose(out, want, rtol=1e-11, atol=1e-12)


def pin_zero_input(lib):
    rng = np.random.default_rng(7)
    L, (x, wr, wg, wu, wd) = _random_layer(rng, 4, 16, 8, 3, 2)
    L = make_layer_from_values(np.zeros_like(x), wr, wg, wu, wd, 2)
    for mode in (oracle.EXACT, oracle.BF16H):
        out, _, _ = oracle.Oracle(L, lib).forward(mode=mode)
        assert np.all(out == 0.0)


def pin_bf16_h_mode(lib):
    """Mode BF16H = the dense FFN with h = silu(g) u rounded to bf16 before the down projection."""
    rng = np.random.default_rng(8)
    T, d, f, E = 6, 16, 24, 3
    L, (x, wr, wg, wu, wd) = _random_layer(rng, T, d, f, E, 1)
    bias = np.zeros(E, np.float32); bias[2] = 100.0
    L = make_layer_from_values(x, np.zeros_like(wr), wg, wu, wd, 1, bias=bias)
    out, _, _ = oracle.Oracle(L, lib).forward(mode=oracle.BF16H)
    g = x @ wg[2].T
    u = x @ wu[2].T
    h = g * expit(g) * u
    hr = np.vectorize(lambda v: lib.moe_oracle_round_bf16(float(v)))(h)
    assert not np.array_equal(hr, h)
    want = hr @ wd[2].T
    assert np.allclose(out, want, rtol=1e-11, atol=1e-12)


def pin_int8_equals_bf16(lib):
    """int8 codes Q with per-output-channel power-of-two scales s equal the bf16 layer whose
    weights are s[j] * Q[j][i] (exact in both), for gate/up (channel j) and down (channel c)."""
    rng = np.random.default_rng(9)
    T, d, f, E, k = 6, 16, 24, 4, 2
    x = rng_bf16(rng, (T, d), 1.0)
    wr = rng_bf16(rng, (E, d), 0.3)
    qg, qu = rng.integers(-127, 128, (E, f, d)), rng.integers(-127, 128, (E, f, d))
    qd = rng.integers(-127, 128, (E, d, f))
    sg = 2.0 ** -rng.integers(5, 10, (E, f)); su = 2.0 ** -rng.integers(5, 10, (E, f))
    sd = 2.0 ** -rng.integers(5, 10, (E, d))
    Li = make_layer_from_values(x, wr, qg, qu, qd, k, wdtype="int8", sg=sg, su=su, sd=sd)
    Lb = make_layer_from_values(x, wr, qg * sg[:, :, None], qu * su[:, :, None], qd * sd[:, :, None], k)
    for mode in (oracle.EXACT, oracle.BF16H):
        oi, ii, _ = oracle.Oracle(Li, lib).forward(mode=mode)
        ob, ib, _ = oracle.Oracle(Lb, lib).forward(mode=mode)
        assert np.array_equal(ii, ib)
        assert np.allclose(oi, ob, rtol=1e-13, atol=1e-15), np.abs(oi - ob).max()


def _torch_e4m3(codes):
    """Values of e4m3 bytes by PyTorch's float8_e4m3fn (a library decode)."""
    import torch
    c = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_fp8_decode(lib):
    """The oracle's e4m3 decode against PyTorch's float8_e4m3fn for all 256 bytes (NaN at
    0x7F and 0xFF), and the format's landmarks: 0x38 = 1, 0x7E = 448 (largest), 0x08 = 2^-6
    (smallest normal), 0x01 = 2^-9 (smallest subnormal), 0x80 = -0."""
    mine = np.array([lib.moe_oracle_fp8_value(c) for c in range(256)])
    ref = _torch_e4m3(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan) and set(np.flatnonzero(nan).tolist()) == {0x7F, 0xFF}
    assert np.array_equal(mine[~nan], ref[~nan])
    assert mine[0x38] == 1.0 and mine[0x7E] == 448.0 and mine[0x08] == 2.0 ** -6 and mine[0x01] == 2.0 ** -9
    assert mine[0x80] == 0.0 and np.signbit(mine[0x80]) and mine[0xB8] == -1.0


def pin_fp8_equals_bf16(lib):
    """e4m3 codes with per-output-channel power-of-two scales equal the bf16 layer whose weights
    are s[j] * v(c[j][i]), the values taken from PyTorch's decode (exact in bf16: at most four
    significant bits), for gate/up (channel j) and down (channel c)."""
    rng = np.random.default_rng(13)
    T, d, f, E, k = 6, 16, 24, 4, 2
    x = rng_bf16(rng, (T, d), 1.0)
    wr = rng_bf16(rng, (E, d), 0.3)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    cg, cu, cd = rng.choice(finite, (E, f, d)), rng.choice(finite, (E, f, d)), rng.choice(finite, (E, d, f))
    sg = 2.0 ** -rng.integers(5, 10, (E, f)); su = 2.0 ** -rng.integers(5, 10, (E, f))
    sd = 2.0 ** -rng.integers(5, 10, (E, d))
    Lq = make_layer_from_values(x, wr, cg, cu, cd, k, wdtype="fp8", sg=sg, su=su, sd=sd)
    Lb = make_layer_from_values(x, wr, _torch_e4m3(cg) * sg[:, :, None], _torch_e4m3(cu) * su[:, :, None],
                                _torch_e4m3(cd) * sd[:, :, None], k)
    for mode in (oracle.EXACT, oracle.BF16H):
        oq, iq, _ = oracle.Oracle(Lq, lib).forward(mode=mode)
        ob, ib, _ = oracle.Oracle(Lb, lib).forward(mode=mode)
        assert np.array_equal(iq, ib)
        assert np.allclose(oq, ob, rtol=1e-13, atol=1e-15), np.abs(oq - ob).max()


def _pack_nibbles(q):
    """The ABI's int4 layout written out: byte m of a row = q[2m] + 16 q[2m + 1]."""
    q = np.asarray(q, np.int64)
    return (q[..., 0::2] + 16 * q[..., 1::2]).astype(np.uint8)


def pin_int4_equals_bf16(lib):
    """4-bit codes q with per-output-channel zero points z and power-of-two scales s equal the
    bf16 layer whose weights are s[j] * (q[j][i] - z[j]) (exact in both), for gate/up (channel
    j) and down (channel c); a hand-packed byte 0x21 holds elements (1, 2)."""
    rng = np.random.default_rng(12)
    T, d, f, E, k = 6, 16, 24, 4, 2
    x = rng_bf16(rng, (T, d), 1.0)
    wr = rng_bf16(rng, (E, d), 0.3)
    qg, qu, qd = rng.integers(0, 16, (E, f, d)), rng.integers(0, 16, (E, f, d)), rng.integers(0, 16, (E, d, f))
    zg, zu, zd = rng.integers(0, 16, (E, f)), rng.integers(0, 16, (E, f)), rng.integers(0, 16, (E, d))
    sg = 2.0 ** -rng.integers(5, 10, (E, f)); su = 2.0 ** -rng.integers(5, 10, (E, f))
    sd = 2.0 ** -rng.integers(5, 10, (E, d))
    Li = make_layer_from_values(x, wr, _pack_nibbles(qg), _pack_nibbles(qu), _pack_nibbles(qd), k, wdtype="int4",
                                sg=sg, su=su, sd=sd, zg=zg, zu=zu, zd=zd)
    Lb = make_layer_from_values(x, wr, (qg - zg[:, :, None]) * sg[:, :, None], (qu - zu[:, :, None]) * su[:, :, None],
                                (qd - zd[:, :, None]) * sd[:, :, None], k)
    for mode in (oracle.EXACT, oracle.BF16H):
        oi, ii, _ = oracle.Oracle(Li, lib).forward(mode=mode)
        ob, ib, _ = oracle.Oracle(Lb, lib).forward(mode=mode)
        assert np.array_equal(ii, ib)
        assert np.allclose(oi, ob, rtol=1e-13, atol=1e-15), np.abs(oi - ob).max()
    assert _pack_nibbles([[1, 2]])[0, 0] == 0x21
    # the generator's packing is the same layout
    q = rng.integers(0, 16, (3, 8))
    assert np.array_equal(synth.pack_int4(q), _pack_nibbles(q))
    assert np.array_equal(synth.unpack_int4(_pack_nibbles(q)), q)


def pin_token_permutation(lib):
    rng = np.random.default_rng(10)
    L, (x, wr, wg, wu, wd) = _random_layer(rng, 9, 16, 8, 5, 2)
    out, ids, w = oracle.Oracle(L, lib).forward(mode=oracle.BF16H)
    p = rng.permutation(9)
    Lp = make_layer_from_values(x[p], wr, wg, wu, wd, 2)
    outp, idsp, wp = oracle.Oracle(Lp, lib).forward(mode=oracle.BF16H)
    assert np.array_equal(outp, out[p]) and np.array_equal(idsp, ids[p])
    # a token list routes the listed tokens only
    sub = np.array([3, 0, 8], np.int32)
    outs, idss, _ = oracle.Oracle(L, lib).forward(tokens=sub, mode=oracle.BF16H)
    assert np.array_equal(outs, out[sub]) and np.array_equal(idss, ids[sub])


def pin_expert_relabel(lib):
    rng = np.random.default_rng(11)
    E = 6
    L, (x, wr, wg, wu, wd) = _random_layer(rng, 8, 16, 8, E, 3)
    bias = rng.standard_normal(E).astype(np.float32)
    L = make_layer_from_values(x, wr, wg, wu, wd, 3, bias=bias)
    out, ids, w = oracle.Oracle(L, lib).forward(mode=oracle.EXACT)
    pi = rng.permutation(E)             # expert e becomes pi[e]
    inv = np.argsort(pi)
    Lp = make_layer_from_values(x, wr[inv], wg[inv], wu[inv], wd[inv], 3, bias=bias[inv])
    outp, idsp, wp = oracle.Oracle(Lp, lib).forward(mode=oracle.EXACT)
    assert np.array_equal(idsp, pi[ids])
    assert np.allclose(outp, out, rtol=1e-13, atol=1e-15) and np.allclose(wp, w, rtol=1e-15)


def pin_golden_tiny(lib):
    g = json.load(open(GOLDEN))
    L = make_layer_from_values(g["x"], g["wr"], g["wg"], g["wu"], g["wd"], g["shape"]["k"])
    out, ids, w = oracle.Oracle(L, lib).forward(mode=oracle.EXACT)
    env = {"sig": lambda z: float(expit(z)), "silu": lambda z: z * float(expit(z))}
    want_out = np.array([[eval(e, {"__builtins__": {}}, env) for e in row] for row in g["expected_out"]])
    want_w = np.array([eval(e, {"__builtins__": {}}, env) for e in g["expected_w"]]).reshape(2, 2)
    assert np.array_equal(ids, np.array(g["expected_ids"]))
    assert np.allclose(w, want_w, rtol=1e-14)
    assert np.allclose(out, want_out, rtol=1e-13, atol=1e-15), (out, want_out)
    cnt, off, tok, inv = oracle.dispatch(ids, g["shape"]["E"], lib)
    ex = g["expected_dispatch"]
    assert cnt.tolist() == ex["counts"] and off.tolist() == ex["offsets"]
    assert tok.tolist() == ex["tok"] and inv.tolist() == ex["inv"]


def pin_routing_invariants(lib):
    """On a synthetic skewed layer: k distinct ids in range per token, sum of counts = T k,
    bijective permutation, stable token order inside each expert segment."""
    sh = synth.custom_shape("inv", T=300, d=64, f=32, E=16, k=4, bias=True, seed=12)
    L = synth.make_layer(sh)
    ids, w, gk, gs = oracle.Oracle(L, lib).route()
    assert np.all((ids >= 0) & (ids < 16))
    assert all(len(set(r)) == 4 for r in ids.tolist())
    assert np.allclose(w.sum(1), 1.0, atol=1e-12)
    cnt, off, tok, inv = oracle.dispatch(ids, 16, lib)
    assert cnt.sum() == 300 * 4
    assert np.array_equal(np.sort(inv.ravel()), np.arange(1200))
    for t in range(300):
        for s in range(4):
            assert tok[inv[t, s]] == t
    for e in range(16):
        seg = tok[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)


# ---------------------------------------------------------- router variants
def pin_raw_gate(lib):
    """Raw-logit gate: the worked example of router_variants.json, and on random
    logits (with exact ties) the same ids as the softmax gate with w = the
    selected logits."""
    g = json.load(open(GOLDEN))
    gr = json.load(open(GOLDEN_ROUTERS))["raw"]
    L = make_layer_from_values(g["x"], g["wr"], g["wg"], g["wu"], g["wd"], 2, router="raw")
    out, ids, w = oracle.Oracle(L, lib).forward(mode=oracle.EXACT)
    env = {"silu": lambda z: z * float(expit(z))}
    want = np.array([[eval(e, {"__builtins__": {}}, env) for e in row] for row in gr["expected_out"]])
    assert np.array_equal(ids, np.array(gr["expected_ids"]))
    assert np.array_equal(w, np.array(gr["expected_w"]))
    assert np.allclose(out, want, rtol=1e-13, atol=1e-15), (out, want)
    rng = np.random.default_rng(21)
    for _ in range(200):
        E = int(rng.integers(2, 9))
        k = int(rng.integers(1, E + 1))
        l = np.round(rng.standard_normal(E) * 4) / 4      # quarter steps: exact ties happen
        ids_s, _, gk_s, gs_s = oracle.gate(l, k, lib)
        ids_r, w_r, gk_r, gs_r = oracle.gate(l, k, lib, raw=True)
        assert np.array_equal(ids_r, ids_s) and gk_r == gk_s and gs_r == gs_s
        assert np.array_equal(w_r, l[ids_r])


def pin_hash_golden(lib):
    """Hash router: the hand-derived ids of router_variants.json (truncation toward
    zero, negative values, saturation; a float sum that rounds, in both
    orders), one token at a time and through a layer."""
    gh = json.load(open(GOLDEN_ROUTERS))["hash"]
    E = gh["E"]
    xb = f32_to_bf16_bits(gh["x"])
    whb = f32_to_bf16_bits(gh["wh"])
    got = [oracle.hash_expert(xb[t], whb, E, lib) for t in range(xb.shape[0])]
    assert got == gh["expected_ids"], got
    T, d = xb.shape
    zeros = np.zeros((E, d))
    L = make_layer_from_values(gh["x"], zeros, np.zeros((E, 2, d)), np.zeros((E, 2, d)), np.zeros((E, d, 2)), 1,
                               router="hash", wh=gh["wh"])
    ids, w, gk, gs = oracle.Oracle(L, lib).route()
    assert ids.ravel().tolist() == gh["expected_ids"] and np.all(w == 1.0)
    go = json.load(open(GOLDEN_ROUTERS))["hash_order"]
    xo, who = f32_to_bf16_bits(go["x"]), f32_to_bf16_bits(go["wh"])
    got = [oracle.hash_expert(xo[t], who, go["E"], lib) for t in range(xo.shape[0])]
    assert got == go["expected_ids"], got


def pin_hash_invariants(lib):
    """Hash router on a random layer: the expert does not depend on the router
    weights, bias or experts; permuting the projection's rows leaves it
    unchanged (XOR is symmetric); zero input goes to expert 0; k = 1 with
    weight 1, and the layer's output is that expert's FFN."""
    rng = np.random.default_rng(22)
    T, d, f, E = 24, 32, 8, 5
    L, (x, wr, wg, wu, wd) = _random_layer(rng, T, d, f, E, 1)
    wh = rng_bf16(rng, (4, d), 0.5)
    La = make_layer_from_values(x, wr, wg, wu, wd, 1, router="hash", wh=wh)
    Lb = make_layer_from_values(x, rng_bf16(rng, wr.shape, 1.0), wg, wu, wd, 1,
                                bias=rng.standard_normal(E).astype(np.float32), router="hash", wh=wh[::-1])
    oa, ia, wa = oracle.Oracle(La, lib).forward(mode=oracle.EXACT)
    ob, ib, wb = oracle.Oracle(Lb, lib).forward(mode=oracle.EXACT)
    assert np.array_equal(ia, ib) and np.all(wa == 1.0) and np.all(wb == 1.0)
    assert len(set(ia.ravel().tolist())) > 1
    o = oracle.Oracle(La, lib)
    for t in range(T):
        assert np.array_equal(oa[t], o.expert(ia[t, 0], La.x[t], mode=oracle.EXACT))
    Lz = make_layer_from_values(np.zeros((3, d)), wr, wg, wu, wd, 1, router="hash", wh=wh)
    iz, _, _, _ = oracle.Oracle(Lz, lib).route()
    assert np.all(iz == 0)


ALL_PINS = [pin_round_bf16, pin_gate_bruteforce, pin_gate_weights, pin_dispatch, pin_identical_experts,
            pin_one_hot_router, pin_two_expert_mix, pin_zero_input, pin_bf16_h_mode, pin_int8_equals_bf16,
            pin_int4_equals_bf16, pin_fp8_decode, pin_fp8_equals_bf16,
            pin_token_permutation, pin_expert_relabel, pin_golden_tiny, pin_routing_invariants,
            pin_raw_gate, pin_hash_golden, pin_hash_invariants]
