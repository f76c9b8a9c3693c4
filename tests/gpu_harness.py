"""Run the CUDA layer on synthetic inputs and compare it with the fp64 oracle.

Tolerances (bf16 in/out, fp32 accumulate):
  * routing: a token is a near tie when its oracle gap l_(k-1) - l_(k) is
    nonzero and below 1e-5; every other token's id set must equal the oracle's,
    bit for bit.  An exact tie (gap 0) is not excused: there the lower expert
    index must win, as the gate of "Colibri：面向MoE模型的高性能C语言推理引擎"
    §2.1 is read.  Slot order must match except where an adjacent gap among
    the k is nonzero and below 1e-5.  Near-tie tokens are counted and must be
    at most 0.1 % of T (no floor: none at all below 1000 tokens);
  * dispatch: counts, offsets, tok, inv equal the oracle's dispatch of the
    GPU's own ids, bit for bit;
  * gate weights: |w_gpu - w_oracle| <= 1e-5 (the raw-logit router's weights
    are logits, the hash router's are 1);
  * hash router: the oracle has no near ties there (its gap is +inf), so every
    token's expert must match bit for bit;
  * outputs against the oracle with h rounded to bf16 (mode BF16H):
    fp32 output max |err| <= 2e-2; bf16 output |err| <= 2e-2 + half a bf16 ulp
    of the reference; mean relative error sum|err| / sum|ref| <= 5e-3 against
    both oracle modes.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import mixture_experts_router_gb300 as cb
import oracle
import synth

GAP = 1e-5
MAX_ABS = 2e-2
MEAN_REL = 5e-3

# (test id, layer name, report) of every full_check of the session, printed
# by tests/conftest.py at the end of the run
REPORTS = []


def to_dev(a, device="cuda"):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


class GpuLayer:
    def __init__(self, layer: synth.Layer, keep_logits=True, device=0, flags=0):
        s = layer.shape
        self.layer = layer
        self.T = layer.x.shape[0]
        self.dev = f"cuda:{device}"
        w = {n: to_dev(getattr(layer, n), self.dev)
             for n in ("wr", "bias", "wg", "wu", "wd", "sg", "su", "sd", "wh", "zg", "zu", "zd")}
        self.m = cb.MoELayer(self.T, s.d, s.f, s.E, s.k, w["wr"], w["wg"], w["wu"], w["wd"], router_bias=w["bias"],
                             s_gate=w["sg"], s_up=w["su"], s_down=w["sd"], device=device, keep_logits=keep_logits,
                             flags=flags, router=s.router, w_hash=w["wh"], z_gate=w["zg"], z_up=w["zu"],
                             z_down=w["zd"], wdtype=s.wdtype)
        del w
        self.x = to_dev(layer.x, self.dev)
        self.out = torch.empty((self.T, s.d), dtype=torch.bfloat16, device=self.dev)
        self.out32 = torch.empty((self.T, s.d), dtype=torch.float32, device=self.dev)

    def run(self, f32=True, bf16=True):
        if bf16:
            self.m.forward(self.x, self.out)
        if f32:
            self.m.forward(self.x, self.out32, f32out=True)
        torch.cuda.synchronize()
        st = self.m.last_error()
        assert st == cb.CB_OK, f"device status {st}"

    def routing(self):
        v = self.m.routing()
        s = self.layer.shape
        T, k, E = self.T, s.k, s.E

        def grab(ptr, n, dt):
            t = torch.empty(n, dtype=dt, device=self.dev)
            cb.copy_from_device(t, ptr, n * t.element_size())
            return t.cpu().numpy()

        r = dict(ids=grab(v.ids, T * k, torch.int32).reshape(T, k),
                 w=grab(v.w, T * k, torch.float32).reshape(T, k),
                 counts=grab(v.counts, E, torch.int32),
                 offsets=grab(v.offsets, E + 1, torch.int32),
                 tok=grab(v.tok, T * k, torch.int32),
                 inv=grab(v.inv, T * k, torch.int32).reshape(T, k),
                 tile_offsets=grab(v.tile_offsets, E + 1, torch.int32))
        if v.logits:
            r["logits"] = grab(v.logits, T * E, torch.float32).reshape(T, E)
        return r

    def close(self):
        self.m.close()


def half_ulp_bf16(ref):
    a = np.abs(ref).astype(np.float64)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 8)


def bf16_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def check_routing(gl: GpuLayer, orc: oracle.Oracle, report: dict):
    s = gl.layer.shape
    T, k, E = gl.T, s.k, s.E
    r = gl.routing()
    ids_o, w_o, gk, gs = orc.route()
    ids_g = r["ids"]
    set_eq = np.array([set(a) == set(b) for a, b in zip(ids_g.tolist(), ids_o.tolist())]) if T else np.zeros(0, bool)
    near = (gk > 0) & (gk < GAP)
    report["near_tie_tokens"] = int(near.sum())
    report["exact_tie_tokens"] = int((gk == 0).sum())
    report["flipped_tokens"] = int((~set_eq).sum())
    assert np.all(set_eq | near), f"id sets differ on {int((~set_eq & ~near).sum())} tokens (exact ties or gap >= {GAP})"
    assert near.sum() <= 0.001 * T, f"{int(near.sum())} near-tie tokens out of {T}"
    order_ok = np.all(ids_g == ids_o, axis=1) | near | ((gs > 0) & (gs < GAP))
    assert np.all(order_ok), "slot order differs"
    same = np.all(ids_g == ids_o, axis=1)
    if same.any():
        werr = np.abs(r["w"][same] - w_o[same]).max()
        report["w_max_err"] = float(werr)
        assert werr <= 1e-5, werr
    # dispatch of the GPU's own ids, bit for bit
    cnt, off, tok, inv = oracle.dispatch(ids_g, E)
    assert np.array_equal(r["counts"], cnt)
    assert np.array_equal(r["offsets"], off)
    assert np.array_equal(r["tok"], tok)
    assert np.array_equal(r["inv"], inv)
    want_tiles = np.concatenate([[0], np.cumsum((cnt + 127) // 128)])
    assert np.array_equal(r["tile_offsets"], want_tiles)
    if "logits" in r and s.router != "hash":   # the hash router computes no logits
        _, _, _, _, lg = orc.route(want_logits=True)
        report["logit_max_err"] = float(np.abs(r["logits"] - lg).max()) if T else 0.0
    return r, near, same


def check_outputs(gl: GpuLayer, orc: oracle.Oracle, tokens, skip_mask, report: dict):
    tokens = np.asarray(tokens, np.int32)
    tokens = tokens[~skip_mask[tokens]] if len(tokens) else tokens
    if len(tokens) == 0:
        return
    ref_f, _, _ = orc.forward(tokens=tokens, mode=oracle.BF16H)
    ref_e, _, _ = orc.forward(tokens=tokens, mode=oracle.EXACT)
    o32 = gl.out32.cpu().numpy().astype(np.float64)[tokens]
    o16 = bf16_to_f64(gl.out)[tokens]
    err32 = np.abs(o32 - ref_f)
    err16 = np.abs(o16 - ref_f)
    report["n_checked"] = int(len(tokens))
    report["f32_max_abs"] = float(err32.max())
    report["bf16_max_abs"] = float(err16.max())
    report["ref_max_abs"] = float(np.abs(ref_f).max())
    denom_f, denom_e = np.abs(ref_f).sum(), np.abs(ref_e).sum()
    report["f32_mean_rel_F"] = float(err32.sum() / denom_f)
    report["f32_mean_rel_exact"] = float(np.abs(o32 - ref_e).sum() / denom_e)
    report["bf16_mean_rel_F"] = float(err16.sum() / denom_f)
    report["bf16_mean_rel_exact"] = float(np.abs(o16 - ref_e).sum() / denom_e)
    assert err32.max() <= MAX_ABS, report
    assert np.all(err16 <= MAX_ABS + half_ulp_bf16(ref_f)), report
    for key in ("f32_mean_rel_F", "f32_mean_rel_exact", "bf16_mean_rel_F", "bf16_mean_rel_exact"):
        assert report[key] <= MEAN_REL, report


def sample_tokens(routing, T, n, seed=0, skip=None):
    """Tokens for the output check of a full-size layer: the first and the last
    comparable routed row of every 128-row m-tile of every expert (so every
    m-tile, every expert's last or half-pair tile, and every N-tile of the down
    GEMM has checked rows), then `n` random tokens more.  `skip` marks tokens
    whose outputs are not comparable (routed differently at a near tie)."""
    rng = np.random.default_rng(seed)
    off, tok = routing["offsets"], routing["tok"]
    skip = np.zeros(T, bool) if skip is None else skip
    chosen = set()
    for e in range(len(off) - 1):
        for r0 in range(int(off[e]), int(off[e + 1]), 128):
            rows = [int(t) for t in tok[r0:min(r0 + 128, int(off[e + 1]))] if not skip[t]]
            if rows:
                chosen.add(rows[0])
                chosen.add(rows[-1])
    rest = [int(t) for t in rng.permutation(T) if int(t) not in chosen and not skip[t]]
    chosen |= set(rest[:max(0, n)])
    return np.array(sorted(chosen), np.int32)


def mtiles_covered(routing, T, tokens):
    """(m-tiles with at least one checked row, all m-tiles)."""
    off, tok = routing["offsets"], routing["tok"]
    checked = np.zeros(T, bool)
    checked[np.asarray(tokens, np.int64)] = True
    hit = total = 0
    for e in range(len(off) - 1):
        for r0 in range(int(off[e]), int(off[e + 1]), 128):
            total += 1
            hit += bool(checked[tok[r0:min(r0 + 128, int(off[e + 1]))]].any())
    return hit, total


def full_check(layer: synth.Layer, sample=None, report=None):
    """Run the layer on the GPU and check routing, dispatch and outputs."""
    report = {} if report is None else report
    gl = GpuLayer(layer)
    try:
        gl.run()
        orc = oracle.Oracle(layer)
        r, near, same = check_routing(gl, orc, report)
        skip = ~same  # outputs of tokens routed differently (near ties) are not comparable
        tokens = np.arange(gl.T) if sample is None else sample_tokens(r, gl.T, sample, skip=skip)
        check_outputs(gl, orc, tokens, skip, report)
        if gl.T:
            # an m-tile made only of near-tie tokens routed differently has no comparable row
            report["mtiles_checked"], report["mtiles"] = mtiles_covered(r, gl.T, tokens[~skip[tokens]])
            hit_max, _ = mtiles_covered(r, gl.T, np.flatnonzero(~skip))
            assert report["mtiles_checked"] == hit_max, report
    finally:
        gl.close()
    REPORTS.append((os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], layer.shape, dict(report)))
    return report
