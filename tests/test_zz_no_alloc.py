"""cb_moe_dispatch_noalloc against the oracle's dispatch and the forward's own.

The no-allocation entry point is for callers that cannot call cudaMalloc (for
example a host program whose own allocator has reserved the GPU's memory).
It keeps its scratch in one static device array that every call reuses, so
these tests make calls in a row on different routings and check each one,
bit for bit (integer work), against the oracle's dispatch of the same ids and
against the dispatch inside cb_moe_forward.  One test runs in a child process
that never creates a layer handle, at the sizes where the entry point's
kernels change form.  The file is collected last and builds everything it
needs, so it passes alone in a fresh process and after the other tests.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

gh = pytest.importorskip("gpu_harness")
HERE = os.path.dirname(os.path.abspath(__file__))


def _routing_of_forward(shape):
    layer = synth.make_layer(shape)
    gl = gh.GpuLayer(layer)
    try:
        gl.run(f32=False)
        return gl.routing()
    finally:
        gl.close()


def _noalloc(ids_np, E):
    import mixture_experts_router_gb300 as cb
    T, k = ids_np.shape
    dev = "cuda"
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).to(dev)
    counts = torch.full((E,), -7, dtype=torch.int32, device=dev)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    tok = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    inv = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    status = torch.full((1,), -7, dtype=torch.int32, device=dev)
    st = cb.cb_moe_dispatch_noalloc(ids.data_ptr(), T, k, E, counts.data_ptr(), offsets.data_ptr(),
                                    tok.data_ptr(), inv.data_ptr(), status.data_ptr(), 0)
    assert st == cb.CB_OK, cb.cb_status_string(st)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return counts.cpu().numpy(), offsets.cpu().numpy(), tok.cpu().numpy(), inv.cpu().numpy().reshape(T, k)


def test_noalloc_dispatch_matches_oracle_and_forward_twice_in_a_row():
    shapes = [synth.custom_shape("noalloc_a", T=3000, d=256, f=256, E=128, k=4, bias=True, seed=31),
              synth.custom_shape("noalloc_b", T=300, d=512, f=256, E=8, k=2, seed=32)]
    for shape in shapes:       # calls in a row; the second sees the first call's leftovers
        r = _routing_of_forward(shape)
        want = oracle.dispatch(r["ids"], shape.E)
        got = _noalloc(r["ids"], shape.E)
        for g, w, f, name in zip(got, want, (r["counts"], r["offsets"], r["tok"], r["inv"]),
                                 ("counts", "offsets", "tok", "inv")):
            assert np.array_equal(g, w), name
            assert np.array_equal(g, f), name


def test_noalloc_in_a_process_without_handles():
    """48 KB shared-memory band, the one-thread scan past the block scan, a
    size near the scratch limit and an out-of-range id, in a fresh process."""
    r = subprocess.run([sys.executable, os.path.join(HERE, "noalloc_fresh_process.py")], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "NOALLOC_OK" in r.stdout, r.stdout + r.stderr


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import mixture_experts_router_gb300 as cb
    big_T = 1 << 20          # 4M (token, slot) pairs at E = 256 exceed the 1 MiB scratch
    st = cb.cb_moe_dispatch_noalloc(16, big_T, 4, 256, 16, 16, 16, 16, None, 0)
    assert st == cb.CB_ERR_UNSUPPORTED
