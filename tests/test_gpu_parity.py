"""CUDA layer vs the fp64 oracle through the C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

gh = pytest.importorskip("gpu_harness")

SMALL = {
    "tiny": synth.WORKLOADS["tiny"],
    # several M, N and K tiles with ragged per-expert tails
    "ragged_mid": synth.custom_shape("ragged_mid", T=300, d=512, f=768, E=8, k=2, seed=21),
    "one_expert": synth.custom_shape("one_expert", T=130, d=256, f=256, E=1, k=1, seed=22),
    "k_equals_E": synth.custom_shape("k_equals_E", T=200, d=256, f=512, E=4, k=4, seed=23),
    # skewed bias: most of the 128 experts get no rows
    "skewed_small": synth.custom_shape("skewed_small", T=1000, d=256, f=256, E=128, k=4, bias=True, seed=24),
    "e256_k16": synth.custom_shape("e256_k16", T=257, d=256, f=256, E=256, k=16, seed=25),
    # wide routers on a handful of tokens: the cooperative dispatch with 1 and 3 blocks
    # about 300 rows per expert: three m-tiles, a full CTA pair and a half pair
    "three_mtiles": synth.custom_shape("three_mtiles", T=600, d=512, f=768, E=4, k=2, seed=39),
    "one_token_e32": synth.custom_shape("one_token_e32", T=1, d=256, f=256, E=32, k=4, seed=37),
    "three_tokens_e64": synth.custom_shape("three_tokens_e64", T=3, d=512, f=256, E=64, k=6, seed=38),
    "odd_T": synth.custom_shape("odd_T", T=1, d=512, f=512, E=8, k=2, seed=26),
    # int8 experts with per-channel scales: several tiles, ragged tails
    "int8_mid": synth.custom_shape("int8_mid", T=300, d=512, f=768, E=8, k=2, wdtype="int8", seed=27),
    "int8_k6": synth.custom_shape("int8_k6", T=700, d=256, f=512, E=64, k=6, wdtype="int8", seed=28),
    # int8 experts of about five m-tiles each: full and half-empty m-tile pairs
    "int8_pairs": synth.custom_shape("int8_pairs", T=1100, d=512, f=768, E=4, k=2, wdtype="int8", seed=29),
    # int4 experts (scale and zero point per channel): one-m-tile experts, pairs, many experts
    "int4_mid": synth.custom_shape("int4_mid", T=300, d=512, f=768, E=8, k=2, wdtype="int4", seed=30),
    "int4_pairs": synth.custom_shape("int4_pairs", T=1100, d=512, f=768, E=4, k=2, wdtype="int4", seed=31),
    "int4_k6": synth.custom_shape("int4_k6", T=700, d=256, f=512, E=64, k=6, wdtype="int4", seed=32),
    # fp8 (e4m3) experts with a scale per channel: the same three layouts
    "fp8_mid": synth.custom_shape("fp8_mid", T=300, d=512, f=768, E=8, k=2, wdtype="fp8", seed=34),
    "fp8_pairs": synth.custom_shape("fp8_pairs", T=1100, d=512, f=768, E=4, k=2, wdtype="fp8", seed=35),
    "fp8_k6": synth.custom_shape("fp8_k6", T=700, d=256, f=512, E=64, k=6, wdtype="fp8", seed=36),
    # router and dispatch in one launch: several 16-token units per block, and 16 experts
    "many_units": synth.custom_shape("many_units", T=10000, d=512, f=256, E=8, k=2, seed=91),
    "e16_d512": synth.custom_shape("e16_d512", T=700, d=512, f=256, E=16, k=4, seed=95),
    "e3_k3_d1024": synth.custom_shape("e3_k3_d1024", T=77, d=1024, f=256, E=3, k=3, seed=93),
    "rd_one_expert": synth.custom_shape("rd_one_expert", T=130, d=512, f=256, E=1, k=1, seed=101),
    "rd_k_equals_E": synth.custom_shape("rd_k_equals_E", T=200, d=512, f=256, E=4, k=4, seed=102),
    # about 16 units per block, 272 owned tokens
    "rd_long": synth.custom_shape("rd_long", T=40000, d=512, f=256, E=8, k=2, seed=103),
    "rd_e16_k16": synth.custom_shape("rd_e16_k16", T=333, d=1024, f=256, E=16, k=16, seed=104),
    "rd_bias": synth.custom_shape("rd_bias", T=500, d=512, f=256, E=12, k=3, bias=True, seed=105),
    # quantised layers of at most 128 tokens: wide tiles (one m-tile, two weight blocks)
    "int8_wide": synth.custom_shape("int8_wide", T=100, d=512, f=768, E=8, k=2, wdtype="int8", seed=111),
    "int4_wide": synth.custom_shape("int4_wide", T=64, d=256, f=512, E=8, k=2, wdtype="int4", seed=112),
    "fp8_wide": synth.custom_shape("fp8_wide", T=128, d=512, f=512, E=4, k=2, wdtype="fp8", seed=113),
    "int8_wide_e64": synth.custom_shape("int8_wide_e64", T=100, d=256, f=512, E=64, k=6, wdtype="int8", seed=114),
    # the tcgen05 router and dispatch in one launch: blocks of 264 tokens (passes of 128, 128
    # and 8), 200 experts (padded to 256), 17 experts with one expert per token, 20 tokens on
    # two blocks
    "rdt_multi_pass": synth.custom_shape("rdt_multi_pass", T=40000, d=256, f=256, E=24, k=2, bias=True, seed=121),
    "rdt_e200": synth.custom_shape("rdt_e200", T=900, d=768, f=256, E=200, k=8, seed=122),
    "rdt_e17_k1": synth.custom_shape("rdt_e17_k1", T=500, d=256, f=256, E=17, k=1, seed=123),
    "rdt_small_T": synth.custom_shape("rdt_small_T", T=20, d=512, f=256, E=64, k=6, seed=124),
}

FULL = {  # workload: random tokens checked beyond the first and last row of every m-tile (None: every token)
    "mixtral_decode": None,
    "skewed": None,
    "mixtral_prefill": 24,
    "int8": 48,
    "int4": 48,
    "fp8": 48,
}


@pytest.mark.parametrize("name", list(SMALL))
def test_parity_small(name):
    rep = gh.full_check(synth.make_layer(SMALL[name]))
    print(name, rep)


@pytest.mark.parametrize("name", list(FULL))
def test_parity_full_size(name):
    layer = synth.make_layer(synth.WORKLOADS[name])
    rep = gh.full_check(layer, sample=FULL[name])
    print(name, rep)


def test_deterministic_and_host_entry_point():
    layer = synth.make_layer(SMALL["ragged_mid"])
    gl = gh.GpuLayer(layer)
    try:
        gl.run(f32=False)
        a = gl.out.clone()
        gl.run(f32=False)
        assert torch.equal(a.view(torch.int16), gl.out.view(torch.int16))
        xh = torch.from_numpy(layer.x.view(np.int16)).pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        gl.m.forward_host(xh, oh)
        torch.cuda.synchronize()
        assert torch.equal(oh, a.view(torch.int16).cpu())
    finally:
        gl.close()


def test_host_forwards_pipelined():
    """Back-to-back host-buffer forwards of different inputs (their copies overlap the
    neighbouring calls' layers through the two staging slots), with a device forward
    on another stream in between: every result equals the device forward of its input."""
    layer = synth.make_layer(SMALL["ragged_mid"])
    gl = gh.GpuLayer(layer)
    try:
        gen = torch.Generator().manual_seed(4)
        xs = [gl.x[torch.randperm(gl.T, generator=gen).to(gl.x.device)].contiguous() for _ in range(5)]
        refs = []
        for x in xs:
            gl.m.forward(x, gl.out)
            torch.cuda.synchronize()
            refs.append(gl.out.clone().view(torch.int16).cpu())
        xh = [x.view(torch.int16).cpu().pin_memory() for x in xs]
        oh = [torch.empty_like(a).pin_memory() for a in xh]
        side = torch.cuda.Stream()
        dev_out = torch.empty_like(gl.out)
        for i in range(5):
            gl.m.forward_host(xh[i], oh[i])
            if i == 2:
                with torch.cuda.stream(side):
                    gl.m.forward(xs[0], dev_out, stream=side)
        torch.cuda.synchronize()
        for i in range(5):
            assert torch.equal(oh[i], refs[i]), i
        assert torch.equal(dev_out.view(torch.int16).cpu(), refs[0])
    finally:
        gl.close()


def test_forwards_inside_a_caller_graph():
    """A device forward captured into the caller's own CUDA graph replays to the same
    bits (the handle's ordering event is left to the caller's graph); the host-buffer
    forward, whose copies run on the handle's streams, refuses a capturing stream."""
    import mixture_experts_router_gb300 as cb
    layer = synth.make_layer(SMALL["ragged_mid"])
    gl = gh.GpuLayer(layer)
    try:
        gl.run(f32=False)
        ref = gl.out.clone()
        out = torch.zeros_like(gl.out)
        s = torch.cuda.Stream()
        xh = torch.from_numpy(layer.x.view(np.int16)).pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            gl.m.forward(gl.x, out, stream=s)
            st = cb.cb_moe_forward_host(gl.m.handle, xh.data_ptr(), oh.data_ptr(), s.cuda_stream)
        assert st == cb.CB_ERR_UNSUPPORTED
        for _ in range(2):
            out.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert gl.m.last_error() == cb.CB_OK
        gl.run(f32=False)                  # the handle still runs outside the graph
        assert torch.equal(gl.out.view(torch.int16), ref.view(torch.int16))
    finally:
        gl.close()


GUARD_CASES = [
    ("tiny", {}), ("odd_T", {}), ("int8_wide", {}), ("int4_wide", {}), ("ragged_mid", {"CB_MOE_PAIR": "1"}), ("ragged_mid", {"CB_MOE_ROUTE_DISPATCH": "0"}),
    ("many_units", {}),
    ("ragged_mid", {"CB_MOE_PAIR": "1", "CB_MOE_FUSED_COMBINE": "1"}), ("ragged_mid", {"CB_MOE_GATHER": "1"}),
    ("three_mtiles", {"CB_MOE_PAIR": "1"}), ("skewed_small", {}), ("skewed_small", {"CB_MOE_ROUTE_DISPATCH": "0"}),
    ("skewed_small", {"CB_MOE_ROUTE_DISPATCH": "0", "CB_MOE_DISPATCH": "split"}), ("rdt_multi_pass", {}), ("rdt_e200", {}),
    ("e256_k16", {}), ("one_token_e32", {}), ("int8_k6", {}), ("int8_mid", {"CB_MOE_INT8": "smem"}),
    ("int4_k6", {}), ("fp8_mid", {}), ("hash", {}),
]


@pytest.mark.parametrize("name,env", GUARD_CASES, ids=[f"{n}-{'-'.join(e.values()) or 'default'}" for n, e in GUARD_CASES])
def test_kernels_stay_inside_the_workspace(name, env, monkeypatch):
    """With CB_FLAG_GUARDS a 4 KB band of 0xA5 follows every workspace region; after
    bf16, fp32 and host-buffer forwards on every kernel path none of them has changed
    (a check of out-of-range writes, with compute-sanitizer unavailable)."""
    import mixture_experts_router_gb300 as cb
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    shape = synth.with_router(SMALL["ragged_mid"], "hash") if name == "hash" else SMALL[name]
    layer = synth.make_layer(shape)
    gl = gh.GpuLayer(layer, flags=cb.CB_FLAG_GUARDS)
    try:
        gl.run()
        xh = torch.from_numpy(layer.x.view(np.int16)).pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        gl.m.forward_host(xh, oh)
        torch.cuda.synchronize()
        assert gl.m.last_error() == cb.CB_OK
        assert gl.m.check_guards() == cb.CB_OK
        assert torch.equal(oh, gl.out.view(torch.int16).cpu())
    finally:
        gl.close()


@pytest.mark.parametrize("name,expect", [
    ("skewed_small", "T=1000 d=256 f=256 E=128 k=4 weights=bf16 gate=softmax router=tcgen05 "
                     "dispatch=fused-with-router gemm=single-cta"),
    ("int8_k6", "E=64 k=6 weights=int8 gate=softmax router=tcgen05 dispatch=fused-with-router"),
    ("ragged_mid", "T=300 d=512 f=768 E=8 k=2 weights=bf16 gate=softmax router=mma dispatch=fused-with-router"),
    ("tiny", "T=64 d=256 f=512 E=8 k=2 weights=bf16 gate=softmax router=mma dispatch=router-ranked"),
    ("fp8_mid", "weights=fp8 gate=softmax router=mma dispatch=fused-with-router gemm=tensor-memory quantised"),
])
def test_init_log_line(name, expect, monkeypatch, capfd):
    """CB_MOE_LOG=1: cb_moe_init prints one stderr line naming the paths the handle runs."""
    monkeypatch.setenv("CB_MOE_LOG", "1")
    gl = gh.GpuLayer(synth.make_layer(SMALL[name]))
    try:
        err = capfd.readouterr().err
        assert "cbmoe: " in err and expect in err, err
    finally:
        gl.close()


def test_token_permutation_equivariance():
    layer = synth.make_layer(SMALL["ragged_mid"])
    gl = gh.GpuLayer(layer)
    try:
        gl.run(f32=False)
        base = gl.out.clone()
        p = torch.randperm(gl.T, generator=torch.Generator().manual_seed(3))
        gl.x.copy_(gl.x[p.to(gl.x.device)])
        gl.run(f32=False)
        assert torch.equal(gl.out.view(torch.int16), base[p.to(base.device)].view(torch.int16))
    finally:
        gl.close()


def test_empty_token_count():
    import mixture_experts_router_gb300 as cb
    layer = synth.make_layer(synth.custom_shape("empty", T=4, d=256, f=256, E=4, k=2, seed=5))
    w = {n: gh.to_dev(getattr(layer, n)) for n in ("wr", "wg", "wu", "wd")}
    m = cb.MoELayer(0, 256, 256, 4, 2, w["wr"], w["wg"], w["wu"], w["wd"])
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    x16 = torch.empty((16,), dtype=torch.bfloat16, device="cuda")
    o16 = torch.empty((16,), dtype=torch.bfloat16, device="cuda")
    m.forward(x16, o16)
    torch.cuda.synchronize()
    assert m.last_error() == cb.CB_OK
    m.close()
    del x


def test_argument_errors_on_device():
    import mixture_experts_router_gb300 as cb
    layer = synth.make_layer(synth.custom_shape("args", T=16, d=256, f=256, E=4, k=2, seed=6))
    gl = gh.GpuLayer(layer)
    try:
        h = gl.m.handle
        buf = torch.empty(16 * 256 + 64, dtype=torch.bfloat16, device="cuda")
        assert cb.cb_moe_forward(h, gl.x.data_ptr() + 2, gl.out.data_ptr(), 0) == cb.CB_ERR_ALIGNMENT
        assert cb.cb_moe_forward(h, buf.data_ptr(), buf.data_ptr() + 32, 0) == cb.CB_ERR_INVALID_ARG
        assert cb.cb_moe_forward(h, 0, gl.out.data_ptr(), 0) == cb.CB_ERR_INVALID_ARG
        assert cb.cb_moe_forward(None, gl.x.data_ptr(), gl.out.data_ptr(), 0) == cb.CB_ERR_INVALID_ARG
    finally:
        gl.close()


def test_injected_host_faults(monkeypatch):
    import mixture_experts_router_gb300 as cb
    layer = synth.make_layer(synth.custom_shape("faults", T=16, d=256, f=256, E=4, k=2, seed=7))
    monkeypatch.setenv("CB_MOE_INJECT_FAULT", "oom")
    with pytest.raises(cb.CbMoeError) as ei:
        gh.GpuLayer(layer)
    assert ei.value.status == cb.CB_ERR_OOM
    monkeypatch.setenv("CB_MOE_INJECT_FAULT", "launch")
    gl = gh.GpuLayer(layer)
    try:
        assert cb.cb_moe_forward(gl.m.handle, gl.x.data_ptr(), gl.out.data_ptr(), 0) == cb.CB_ERR_CUDA
        monkeypatch.delenv("CB_MOE_INJECT_FAULT")
        gl.run()
    finally:
        gl.close()


ROUTER_CASES = {
    "e8_small": synth.custom_shape("r_e8", T=333, d=512, f=256, E=8, k=2, seed=41),
    "e16_k4": synth.custom_shape("r_e16", T=200, d=256, f=256, E=16, k=4, seed=42),
    "e40_bias": synth.custom_shape("r_e40", T=257, d=768, f=256, E=40, k=3, bias=True, seed=43),
    "e128_k4": synth.custom_shape("r_e128", T=300, d=1024, f=256, E=128, k=4, bias=True, seed=44),
    "e256_k16": synth.custom_shape("r_e256", T=130, d=256, f=256, E=256, k=16, seed=45),
}


@pytest.mark.parametrize("router", ["mma", "tc"])
@pytest.mark.parametrize("name", list(ROUTER_CASES))
def test_both_routers(name, router, monkeypatch):
    """The mma.sync split-K router and the tcgen05 router both match the oracle
    (the library picks one by expert count; CB_MOE_ROUTER forces either)."""
    monkeypatch.setenv("CB_MOE_ROUTER", router)
    rep = gh.full_check(synth.make_layer(ROUTER_CASES[name]))
    print(name, router, rep)
    assert rep.get("logit_max_err", 0.0) <= 5e-6


def test_fp8_every_code():
    """fp8 weights drawn uniformly from all 254 finite e4m3 bytes (both zeros, every
    subnormal, the largest values), each about 2000 times: the kernel's byte -> bf16
    conversion is exact for every code, so the layer matches the oracle."""
    import dataclasses
    shape = synth.custom_shape("fp8_codes", T=300, d=256, f=512, E=4, k=2, wdtype="fp8", seed=33)
    layer = synth.make_layer(shape)
    rng = np.random.default_rng(33)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    wg, wu, wd = (rng.choice(finite, a.shape).astype(np.uint8) for a in (layer.wg, layer.wu, layer.wd))
    assert all(len(np.unique(w)) == len(finite) for w in (wg, wu, wd))
    small = lambda s: (s * np.float32(0.2)).astype(np.float32)  # weights of about 0.02 spread
    layer = dataclasses.replace(layer, wg=wg, wu=wu, wd=wd, sg=small(layer.sg), su=small(layer.su),
                                sd=small(layer.sd))
    rep = gh.full_check(layer)
    print("fp8 every code", rep)


@pytest.mark.parametrize("wdtype", ["bf16", "int8", "int4", "fp8"])
def test_device_wait_timeout_is_reported_and_context_survives(wdtype):
    """A bounded device wait that nothing satisfies (CB_FLAG_TEST_STALL) ends the
    kernel with CB_ERR_TIMEOUT in the status word instead of a hang or a fault;
    the context stays usable: a normal handle afterwards still matches the oracle."""
    import mixture_experts_router_gb300 as cb
    shape = synth.custom_shape("stall", T=300, d=512, f=512, E=8, k=2, wdtype=wdtype, seed=51)
    layer = synth.make_layer(shape)
    gl = gh.GpuLayer(layer, flags=cb.CB_FLAG_TEST_STALL)
    try:
        gl.m.forward(gl.x, gl.out)
        torch.cuda.synchronize()
        assert gl.m.last_error() == cb.CB_ERR_TIMEOUT
        assert gl.m.last_error() == cb.CB_OK     # reading the word clears it
    finally:
        gl.close()
    rep = gh.full_check(layer)
    assert rep["f32_max_abs"] <= gh.MAX_ABS


@pytest.mark.parametrize("name,dispatch", [("ragged_mid", None), ("skewed_small", None), ("tiny", None),
                                           ("skewed_small", "split"), ("ragged_mid", "split")])
def test_gathered_rows_path(name, dispatch, monkeypatch):
    """CB_MOE_GATHER=1: the gate/up GEMM loads its rows from x with TMA
    tile::gather4 instead of the dispatch's row copy; same results (also with
    the separate dispatch kernels, whose copy kernel then only writes the
    pairs' padded rows)."""
    monkeypatch.setenv("CB_MOE_GATHER", "1")
    if dispatch is not None:
        monkeypatch.setenv("CB_MOE_FUSED_RANKS", "0")
        monkeypatch.setenv("CB_MOE_DISPATCH", dispatch)
    rep = gh.full_check(synth.make_layer(SMALL[name]))
    print(name, "gather", rep)


def test_graph_replay_matches_direct_launches():
    """On a non-default stream each forward variant is captured once into a CUDA
    graph and replayed; replays, re-captures after a pointer change, and the
    stage-timing events all give the same bits as direct launches."""
    import mixture_experts_router_gb300 as cb
    layer = synth.make_layer(SMALL["ragged_mid"])
    gl = gh.GpuLayer(layer)
    timed = None
    try:
        gl.run()                                   # legacy stream: direct launches
        ref16 = gl.out.clone()
        ref32 = gl.out32.clone()
        s = torch.cuda.Stream()
        outs = [torch.empty_like(gl.out) for _ in range(2)]
        for it in range(3):                        # capture, replay, replay
            for o in outs:                         # alternate pointers: re-capture
                o.zero_()
                gl.m.forward(gl.x, o, stream=s)
                s.synchronize()
                assert torch.equal(o.view(torch.int16), ref16.view(torch.int16)), it
        o32 = torch.empty_like(gl.out32)
        for _ in range(2):
            gl.m.forward(gl.x, o32, stream=s, f32out=True)
            s.synchronize()
            assert torch.equal(o32, ref32)
        xh = torch.from_numpy(layer.x.view(np.int16)).pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        for _ in range(2):
            oh.zero_()
            gl.m.forward_host(xh, oh, stream=s)
            s.synchronize()
            assert torch.equal(oh, ref16.view(torch.int16).cpu())
        assert gl.m.last_error() == cb.CB_OK
        # stage timing through a replayed graph
        w = {n: gh.to_dev(getattr(layer, n)) for n in ("wr", "wg", "wu", "wd")}
        shp = layer.shape
        timed = cb.MoELayer(gl.T, shp.d, shp.f, shp.E, shp.k, w["wr"], w["wg"], w["wu"], w["wd"], stage_timing=True)
        ot = torch.empty_like(gl.out)
        for _ in range(3):
            timed.forward(gl.x, ot, stream=s)
            ms = timed.stage_times()
            assert all(v > 0 for v in ms) and sum(ms) < 1000
        s.synchronize()
        assert torch.equal(ot.view(torch.int16), ref16.view(torch.int16))
    finally:
        if timed is not None:
            timed.close()
        gl.close()


PAIR_SMALL = ["tiny", "ragged_mid", "one_expert", "k_equals_E", "skewed_small", "e256_k16", "odd_T", "three_mtiles"]


@pytest.mark.parametrize("name", PAIR_SMALL)
def test_pair_mma_path_small(name, monkeypatch):
    """CB_MOE_PAIR=1: bf16 expert GEMMs on CTA pairs with the 2-SM MMA
    (M = 256 over two m-tiles of one expert); an expert's last m-tile without
    a partner runs the M = 128 form, 64 of its rows on each CTA."""
    monkeypatch.setenv("CB_MOE_PAIR", "1")
    rep = gh.full_check(synth.make_layer(SMALL[name]))
    print(name, "pair", rep)


@pytest.mark.parametrize("name", ["mixtral_prefill", "skewed", "mixtral_decode"])
def test_pair_mma_path_full_size(name, monkeypatch):
    monkeypatch.setenv("CB_MOE_PAIR", "1")
    rep = gh.full_check(synth.make_layer(synth.WORKLOADS[name]), sample=FULL[name])
    print(name, "pair", rep)


def test_pair_mma_path_timeout(monkeypatch):
    import mixture_experts_router_gb300 as cb
    monkeypatch.setenv("CB_MOE_PAIR", "1")
    shape = synth.custom_shape("stall_pair", T=300, d=512, f=512, E=8, k=2, seed=52)
    layer = synth.make_layer(shape)
    gl = gh.GpuLayer(layer, flags=cb.CB_FLAG_TEST_STALL)
    try:
        gl.m.forward(gl.x, gl.out)
        torch.cuda.synchronize()
        assert gl.m.last_error() == cb.CB_ERR_TIMEOUT
    finally:
        gl.close()
    rep = gh.full_check(layer)
    assert rep["f32_max_abs"] <= gh.MAX_ABS


@pytest.mark.parametrize("name", PAIR_SMALL)
def test_fused_combine_small(name, monkeypatch):
    """CB_MOE_FUSED_COMBINE=1 (CTA-pair down GEMM forced on): the down
    epilogue adds each row's gate-weighted output into its token's fp32 sum
    and one pass rounds the sums; the same bounds against the oracle."""
    monkeypatch.setenv("CB_MOE_PAIR", "1")
    monkeypatch.setenv("CB_MOE_FUSED_COMBINE", "1")
    rep = gh.full_check(synth.make_layer(SMALL[name]))
    print(name, "fused combine", rep)


@pytest.mark.parametrize("name", ["mixtral_prefill", "skewed"])
def test_fused_combine_full_size(name, monkeypatch):
    monkeypatch.setenv("CB_MOE_FUSED_COMBINE", "1")
    rep = gh.full_check(synth.make_layer(synth.WORKLOADS[name]), sample=FULL[name])
    print(name, "fused combine", rep)


def test_fused_combine_repeatable_at_k2(monkeypatch):
    """With k = 2 each token sum is 0 + a + b in either order, so repeated
    forwards (device and host buffers) agree bit for bit."""
    monkeypatch.setenv("CB_MOE_PAIR", "1")
    monkeypatch.setenv("CB_MOE_FUSED_COMBINE", "1")
    layer = synth.make_layer(SMALL["ragged_mid"])
    gl = gh.GpuLayer(layer)
    try:
        gl.run(f32=False)
        a = gl.out.clone()
        for _ in range(3):
            gl.run(f32=False)
            assert torch.equal(a.view(torch.int16), gl.out.view(torch.int16))
        xh = torch.from_numpy(layer.x.view(np.int16)).pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        gl.m.forward_host(xh, oh)
        torch.cuda.synchronize()
        assert torch.equal(oh, a.view(torch.int16).cpu())
    finally:
        gl.close()


@pytest.mark.parametrize("name", ["tiny", "ragged_mid", "odd_T", "int8_mid", "skewed_small", "e256_k16", "int8_k6"])
def test_dispatch_own_ranking_small(name, monkeypatch):
    """CB_MOE_FUSED_RANKS=0: the dispatch ranks the routed pairs itself
    (one-block or count/scan/scatter kernels) instead of scanning the
    router's per-block counts; same routing views and outputs."""
    monkeypatch.setenv("CB_MOE_FUSED_RANKS", "0")
    rep = gh.full_check(synth.make_layer(SMALL[name]))
    print(name, "own ranking", rep)


@pytest.mark.parametrize("name", ["mixtral_prefill", "mixtral_decode", "skewed"])
def test_dispatch_own_ranking_full_size(name, monkeypatch):
    monkeypatch.setenv("CB_MOE_FUSED_RANKS", "0")
    rep = gh.full_check(synth.make_layer(synth.WORKLOADS[name]), sample=FULL[name])
    print(name, "own ranking", rep)


@pytest.mark.parametrize("name", ["tiny", "ragged_mid", "skewed_small", "e256_k16", "int8_k6", "one_expert"])
def test_dispatch_split_kernels_small(name, monkeypatch):
    """CB_MOE_DISPATCH=split (with the dispatch's own ranking): separate
    count, scan, scatter and row-copy kernels instead of the cooperative
    launch; same routing views and outputs."""
    monkeypatch.setenv("CB_MOE_FUSED_RANKS", "0")
    monkeypatch.setenv("CB_MOE_DISPATCH", "split")
    rep = gh.full_check(synth.make_layer(SMALL[name]))
    print(name, "split dispatch", rep)


@pytest.mark.parametrize("name,mode", [("skewed", "split"), ("int8", "coop"), ("int4", "coop"), ("fp8", "coop")])
def test_dispatch_forced_full_size(name, mode, monkeypatch):
    """With the separate router and dispatch launches, the dispatch form that
    is not the default at this size: separate kernels on the 128-expert layer,
    the cooperative launch past 65536 routed pairs."""
    monkeypatch.setenv("CB_MOE_ROUTE_DISPATCH", "0")
    monkeypatch.setenv("CB_MOE_DISPATCH", mode)
    rep = gh.full_check(synth.make_layer(synth.WORKLOADS[name]), sample=FULL[name])
    print(name, mode, "dispatch", rep)


def test_cooperative_dispatch_timeout(monkeypatch):
    """The cooperative dispatch's grid barrier, made to wait for a block that
    does not exist (CB_FLAG_TEST_STALL_DISPATCH, 1 ms bound), ends with
    CB_ERR_TIMEOUT and leaves the device usable; a new handle is correct."""
    import mixture_experts_router_gb300 as cb
    monkeypatch.setenv("CB_MOE_ROUTE_DISPATCH", "0")
    layer = synth.make_layer(SMALL["skewed_small"])
    gl = gh.GpuLayer(layer, flags=cb.CB_FLAG_TEST_STALL_DISPATCH)
    try:
        assert gl.m.kernels_per_forward() == 6  # tcgen05 router: 2, cooperative dispatch: 1
        gl.m.forward(gl.x, gl.out)
        torch.cuda.synchronize()
        assert gl.m.last_error() == cb.CB_ERR_TIMEOUT
    finally:
        gl.close()
    rep = gh.full_check(layer)
    assert rep["f32_max_abs"] <= gh.MAX_ABS


@pytest.mark.parametrize("fused,name,d,expect", [
    ("1", "mixtral_prefill", 256, 6), ("1", "skewed", 256, 4), ("0", "mixtral_prefill", 256, 5),
    ("0", "skewed", 256, 6), ("split", "mixtral_prefill", 256, 6), ("split", "skewed", 256, 9),
    ("1", "mixtral_prefill", 512, 4), ("1", "mixtral_decode", 512, 4), ("rd0", "mixtral_prefill", 512, 6),
    ("1", "skewed", 512, 4), ("rd0", "skewed", 512, 6), ("1", "int8", 512, 4)])
def test_kernels_per_forward(fused, name, d, expect, monkeypatch):
    """The launch count the library reports: router (the separate tcgen05
    router of wide layers: partial logits + top-k), dispatch kernels (none
    when the router's launch also dispatches: up to 16 experts and d a
    multiple of 512, or 17 to 256 experts; block scan + row copy after the
    mma router's per-block ranks; else one cooperative launch, or with
    CB_MOE_DISPATCH=split one-block / count-scan-scatter ranking + row copy),
    two grouped GEMMs, combine."""
    if fused in ("0", "split"):
        monkeypatch.setenv("CB_MOE_FUSED_RANKS", "0")
    if fused == "split":
        monkeypatch.setenv("CB_MOE_DISPATCH", "split")
    if fused == "rd0":
        monkeypatch.setenv("CB_MOE_ROUTE_DISPATCH", "0")
    shp = synth.WORKLOADS[name]
    gl = gh.GpuLayer(synth.make_layer(synth.custom_shape(name + "_n", T=shp.T, d=d, f=256, E=shp.E, k=shp.k,
                                                         seed=61)))
    try:
        assert gl.m.kernels_per_forward() == expect
    finally:
        gl.close()


@pytest.mark.parametrize("name", ["int8_mid", "int8_k6", "int8_pairs"])
def test_int8_smem_kernel_small(name, monkeypatch):
    """CB_MOE_INT8=smem: the int8 GEMMs that convert the weights into shared
    memory (the MMA's B operand) instead of tensor memory; same results."""
    monkeypatch.setenv("CB_MOE_INT8", "smem")
    rep = gh.full_check(synth.make_layer(SMALL[name]))
    print(name, "int8 smem", rep)


def test_int8_smem_kernel_full_size(monkeypatch):
    monkeypatch.setenv("CB_MOE_INT8", "smem")
    rep = gh.full_check(synth.make_layer(synth.WORKLOADS["int8"]), sample=FULL["int8"])
    print("int8 smem", rep)


@pytest.mark.parametrize("name", ["mixtral_prefill", "skewed"])
def test_single_cta_gemms_full_size(name, monkeypatch):
    """CB_MOE_PAIR=0: the 1-CTA grouped GEMMs (the default only for layers
    whose experts average under two m-tiles) at the full prefill sizes."""
    monkeypatch.setenv("CB_MOE_PAIR", "0")
    rep = gh.full_check(synth.make_layer(synth.WORKLOADS[name]), sample=FULL[name])
    print(name, "single CTA", rep)


RAW_SMALL = ["ragged_mid", "skewed_small", "e256_k16", "int8_k6"]


@pytest.mark.parametrize("name", RAW_SMALL)
def test_raw_logit_router_small(name):
    """CB_ROUTER_RAW_LOGITS: the same experts as the softmax gate, weighted by the
    raw logits (mma.sync router for E <= 16, tcgen05 router above)."""
    rep = gh.full_check(synth.make_layer(synth.with_router(SMALL[name], "raw")))
    print(name, "raw", rep)


HASH_SMALL = {
    "h_ragged": synth.custom_shape("h_ragged", T=300, d=512, f=768, E=8, k=1, seed=71, router="hash", hash_dims=8),
    "h_e128_d3": synth.custom_shape("h_e128", T=1000, d=256, f=256, E=128, k=1, seed=72, router="hash",
                                    hash_dims=3),
    "h_one_dim": synth.custom_shape("h_one", T=33, d=768, f=256, E=5, k=1, seed=73, router="hash", hash_dims=1),
    "h_int8": synth.custom_shape("h_int8", T=700, d=256, f=512, E=64, k=1, wdtype="int8", seed=74, router="hash",
                                 hash_dims=8),
}


@pytest.mark.parametrize("name", list(HASH_SMALL))
def test_hash_router_small(name):
    """CB_ROUTER_HASH: one expert per token from the hashed projection, bit for bit."""
    rep = gh.full_check(synth.make_layer(HASH_SMALL[name]))
    print(name, "hash", rep)


@pytest.mark.parametrize("router", ["raw", "hash"])
def test_router_variants_full_size(router):
    shape = synth.with_router(synth.WORKLOADS["mixtral_prefill"], router)
    rep = gh.full_check(synth.make_layer(shape), sample=24)
    print(router, rep)


@pytest.mark.parametrize("case", ["hash", "hash_order"])
def test_hash_router_golden_cases(case):
    """The hand-derived cases of tests/golden/router_variants.json (truncation,
    negative values, saturation, a float sum that rounds), in the first four
    columns of a d = 256 layer."""
    import json
    import os
    import oracle_pins
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "router_variants.json")))[case]
    T, d, E = len(g["x"]), 256, g["E"]
    x = np.zeros((T, d))
    x[:, :4] = g["x"]
    wh = np.zeros((len(g["wh"]), d))
    wh[:, :4] = g["wh"]
    zeros = np.zeros((E, d))
    layer = oracle_pins.make_layer_from_values(x, zeros, np.zeros((E, 256, d)), np.zeros((E, 256, d)),
                                               np.zeros((E, d, 256)), 1, router="hash", wh=wh)
    gl = gh.GpuLayer(layer, keep_logits=False)
    try:
        gl.run()
        assert gl.routing()["ids"].ravel().tolist() == g["expected_ids"]
    finally:
        gl.close()


def test_stage_timing_switch():
    """cb_moe_set_stage_timing: forwards with and without the stage events give
    the same bytes; stage times need the events; handles made without
    CB_FLAG_STAGE_TIMING refuse the switch."""
    import mixture_experts_router_gb300 as cb
    layer = synth.make_layer(SMALL["ragged_mid"])
    s = layer.shape
    w = {n: gh.to_dev(getattr(layer, n), "cuda:0") for n in ("wr", "bias", "wg", "wu", "wd")}
    m = cb.MoELayer(layer.x.shape[0], s.d, s.f, s.E, s.k, w["wr"], w["wg"], w["wu"], w["wd"],
                    router_bias=w["bias"], stage_timing=True)
    x = gh.to_dev(layer.x, "cuda:0")
    out_a = torch.empty((layer.x.shape[0], s.d), dtype=torch.bfloat16, device="cuda:0")
    out_b = torch.empty_like(out_a)
    m.forward(x, out_a)
    ms = m.stage_times()
    assert len(ms) == cb.CB_N_STAGES and all(v >= 0 for v in ms)
    m.set_stage_timing(False)
    m.forward(x, out_b)
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    with pytest.raises(cb.CbMoeError):
        m.stage_times()
    m.set_stage_timing(True)
    m.forward(x, out_b)
    assert len(m.stage_times()) == cb.CB_N_STAGES
    assert m.last_error() == cb.CB_OK
    m2 = cb.MoELayer(layer.x.shape[0], s.d, s.f, s.E, s.k, w["wr"], w["wg"], w["wu"], w["wd"],
                     router_bias=w["bias"])
    with pytest.raises(cb.CbMoeError):
        m2.set_stage_timing(True)
    del m, m2


@pytest.mark.parametrize("name", ["tiny", "skewed_small", "int8_pairs", "ragged_mid"])
def test_programmatic_dependent_launch(name, monkeypatch):
    """CB_MOE_PDL=1: the forward's kernels after the first are launched with
    programmatic stream serialization on a stream (each waits for its
    predecessor's grid before reading its output); same results."""
    monkeypatch.setenv("CB_MOE_PDL", "1")
    layer = synth.make_layer(SMALL[name])
    gl = gh.GpuLayer(layer)
    try:
        # on the legacy default stream the launches are plain: the reference
        gl.m.forward(gl.x, gl.out)
        torch.cuda.synchronize()
        plain = gl.out.clone()
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            for _ in range(4):
                gl.out.zero_()
                gl.m.forward(gl.x, gl.out, stream=stream)
        stream.synchronize()
        assert gl.m.last_error() == 0
        assert torch.equal(plain.view(torch.int16), gl.out.view(torch.int16))
    finally:
        gl.close()
    rep = gh.full_check(layer)
    print(name, "pdl", rep)


ROUTE_DISPATCH_SMALL = ["ragged_mid", "three_mtiles", "odd_T", "int8_mid", "many_units", "e16_d512", "e3_k3_d1024",
                        "rd_one_expert", "rd_k_equals_E", "rd_long", "rd_e16_k16", "rd_bias",
                        "skewed_small", "e256_k16", "int8_k6", "one_token_e32", "rdt_multi_pass", "rdt_e200"]


@pytest.mark.parametrize("name", ROUTE_DISPATCH_SMALL)
def test_separate_router_and_dispatch_small(name, monkeypatch):
    """CB_MOE_ROUTE_DISPATCH=0: the router kernel (with its per-block ranks),
    the block-count scan and the row copy as separate launches instead of the
    one cooperative launch; same routing views and outputs."""
    monkeypatch.setenv("CB_MOE_ROUTE_DISPATCH", "0")
    rep = gh.full_check(synth.make_layer(SMALL[name]))
    print(name, "separate router and dispatch", rep)


@pytest.mark.parametrize("name", ["mixtral_prefill", "mixtral_decode", "skewed"])
def test_separate_router_and_dispatch_full_size(name, monkeypatch):
    monkeypatch.setenv("CB_MOE_ROUTE_DISPATCH", "0")
    rep = gh.full_check(synth.make_layer(synth.WORKLOADS[name]), sample=FULL[name])
    print(name, "separate router and dispatch", rep)


def test_fused_route_dispatch_matches_separate_kernels_bit_for_bit(monkeypatch):
    """The one-launch router + dispatch gives the same ids, weights, logits,
    dispatch arrays and outputs, bit for bit, as the separate kernels."""
    layer = synth.make_layer(SMALL["many_units"])
    outs = []
    for rd in ("1", "0"):
        monkeypatch.setenv("CB_MOE_ROUTE_DISPATCH", rd)
        gl = gh.GpuLayer(layer)
        try:
            assert gl.m.kernels_per_forward() == (4 if rd == "1" else 6)
            gl.run()
            outs.append((gl.routing(), gl.out.clone(), gl.out32.clone()))
        finally:
            gl.close()
    (ra, oa, fa), (rb, ob, fb) = outs
    for key in ra:
        assert np.array_equal(ra[key], rb[key]), key
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(fa, fb)


def test_fused_route_dispatch_timeout():
    """The grid barrier of the router + dispatch launch, made to wait for a
    block that does not exist (CB_FLAG_TEST_STALL_DISPATCH, 1 ms bound), ends
    with CB_ERR_TIMEOUT and leaves the device usable."""
    import mixture_experts_router_gb300 as cb
    layer = synth.make_layer(SMALL["ragged_mid"])
    gl = gh.GpuLayer(layer, flags=cb.CB_FLAG_TEST_STALL_DISPATCH)
    try:
        assert gl.m.kernels_per_forward() == 4
        gl.m.forward(gl.x, gl.out)
        torch.cuda.synchronize()
        assert gl.m.last_error() == cb.CB_ERR_TIMEOUT
    finally:
        gl.close()
    rep = gh.full_check(layer)
    assert rep["f32_max_abs"] <= gh.MAX_ABS


def test_fused_tc_route_dispatch_timeout():
    """The grid barrier of the tcgen05 router + dispatch launch, made to wait
    for a block that does not exist (CB_FLAG_TEST_STALL_DISPATCH, 1 ms
    bound), ends with CB_ERR_TIMEOUT and leaves the device usable."""
    import mixture_experts_router_gb300 as cb
    layer = synth.make_layer(SMALL["skewed_small"])
    gl = gh.GpuLayer(layer, flags=cb.CB_FLAG_TEST_STALL_DISPATCH)
    try:
        assert gl.m.kernels_per_forward() == 4
        gl.m.forward(gl.x, gl.out)
        torch.cuda.synchronize()
        assert gl.m.last_error() == cb.CB_ERR_TIMEOUT
    finally:
        gl.close()
    rep = gh.full_check(layer)
    assert rep["f32_max_abs"] <= gh.MAX_ABS


@pytest.mark.parametrize("name", ["rdt_multi_pass", "rdt_e200", "rdt_e17_k1", "rdt_small_T", "one_token_e32",
                                  "three_tokens_e64", "e256_k16", "int8_wide_e64"])
def test_fused_tc_route_dispatch_edges(name):
    """The tcgen05 router + dispatch launch on its edges: blocks of several
    128-token passes (with a bias, and the raw-logit gate on the same layer),
    expert counts that pad to 256 and to 32, one expert per token, one to
    twenty tokens, 256 experts with k = 16."""
    layer = synth.make_layer(SMALL[name])
    gl = gh.GpuLayer(layer)
    try:
        assert gl.m.kernels_per_forward() == 4
    finally:
        gl.close()
    rep = gh.full_check(layer)
    print(name, "fused tcgen05", rep)
    if name == "rdt_multi_pass":
        rep = gh.full_check(synth.make_layer(synth.with_router(SMALL[name], "raw")))
        print(name, "fused tcgen05 raw", rep)


@pytest.mark.parametrize("name", ["rd_one_expert", "rd_k_equals_E", "rd_long", "rd_e16_k16", "rd_bias"])
def test_fused_route_dispatch_edges(name):
    """The one-launch router + dispatch on its edges: one expert, k = E, a long
    layer whose blocks own many units, 16 experts with k = 16, a router bias
    (and the raw-logit gate on the same layer)."""
    import mixture_experts_router_gb300 as cb
    layer = synth.make_layer(SMALL[name])
    gl = gh.GpuLayer(layer)
    try:
        assert gl.m.kernels_per_forward() == 4
    finally:
        gl.close()
    rep = gh.full_check(layer)
    print(name, "fused", rep)
    if name == "rd_bias":
        rep = gh.full_check(synth.make_layer(synth.with_router(SMALL[name], "raw")))
        print(name, "fused raw", rep)


@pytest.mark.parametrize("name", ["tiny", "skewed_small", "one_token_e32"])
def test_short_activation_boxes_match_whole_tiles(name, monkeypatch):
    """The 1-CTA GEMMs load 32-row activation boxes for m-tiles of at most 32
    routed rows (the other accumulator rows are padding); each output row
    depends on its own activation row only, so the outputs equal, bit for
    bit, those of whole 128-row boxes (CB_MOE_SHORT_A=0)."""
    layer = synth.make_layer(SMALL[name])
    outs = []
    for v in ("1", "0"):
        monkeypatch.setenv("CB_MOE_SHORT_A", v)
        gl = gh.GpuLayer(layer)
        try:
            gl.run()
            outs.append((gl.out.clone(), gl.out32.clone()))
        finally:
            gl.close()
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])


WIDE_SMALL = ["int8_wide", "int4_wide", "fp8_wide", "int8_wide_e64"]


@pytest.mark.parametrize("name", WIDE_SMALL)
def test_wide_quantised_tiles_small(name):
    """Quantised layers of at most 128 tokens: each tile pairs the single
    m-tile with two weight blocks (two accumulators, twice the weight bytes
    per k-block handshake); same routing and outputs as the oracle."""
    rep = gh.full_check(synth.make_layer(SMALL[name]))
    print(name, "wide", rep)


@pytest.mark.parametrize("wdtype", ["int8", "int4", "fp8"])
def test_wide_quantised_tiles_decode_shape(wdtype):
    """The Mixtral decode shape (T=64, d=4096, f=14336, E=8, top-2) with
    quantised weights, every token checked against the oracle."""
    shape = synth.custom_shape(f"{wdtype}_decode", T=64, d=4096, f=14336, E=8, k=2, wdtype=wdtype, seed=115)
    rep = gh.full_check(synth.make_layer(shape))
    print(wdtype, "decode shape wide", rep)


@pytest.mark.parametrize("name", WIDE_SMALL)
def test_wide_quantised_tiles_match_one_block_tiles(name, monkeypatch):
    """Wide tiles run the same M=128 N=128 MMAs in the same K order as tiles of
    one weight block (CB_MOE_WIDE_QUANT=0): the outputs agree bit for bit."""
    layer = synth.make_layer(SMALL[name])
    outs = []
    for v in ("1", "0"):
        monkeypatch.setenv("CB_MOE_WIDE_QUANT", v)
        gl = gh.GpuLayer(layer)
        try:
            gl.run()
            outs.append((gl.out.clone(), gl.out32.clone()))
        finally:
            gl.close()
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("wdtype", ["int8", "int4"])
def test_wide_quantised_tiles_timeout(wdtype):
    """A bounded device wait that nothing satisfies, on the wide tiles: the
    kernel ends with CB_ERR_TIMEOUT and the context stays usable."""
    import mixture_experts_router_gb300 as cb
    layer = synth.make_layer(SMALL[f"{wdtype}_wide"])
    gl = gh.GpuLayer(layer, flags=cb.CB_FLAG_TEST_STALL)
    try:
        gl.m.forward(gl.x, gl.out)
        torch.cuda.synchronize()
        assert gl.m.last_error() == cb.CB_ERR_TIMEOUT
    finally:
        gl.close()
    rep = gh.full_check(layer)
    assert rep["f32_max_abs"] <= gh.MAX_ABS
