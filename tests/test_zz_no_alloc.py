"""cb_moe_dispatch_noalloc against the dispatch of cb_moe_forward.

The no-allocation entry point is for callers that cannot call cudaMalloc (for
example a host program whose own allocator has reserved the GPU's memory).
It keeps its scratch in one static device array that every call reuses, so
this test makes two calls in a row on different routings and checks each
against the existing entry point's dispatch, bit for bit (integer work).  It
sits in a file of its own, collected last, and builds everything it needs, so
it passes alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

gh = pytest.importorskip("gpu_harness")


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


def test_noalloc_dispatch_matches_forward_twice_in_a_row():
    shapes = [synth.custom_shape("noalloc_a", T=3000, d=256, f=256, E=128, k=4, bias=True, seed=31),
              synth.custom_shape("noalloc_b", T=300, d=512, f=256, E=8, k=2, seed=32)]
    for shape in shapes:       # two calls in a row; the second sees the first call's leftovers
        r = _routing_of_forward(shape)
        cnt, off, tok, inv = _noalloc(r["ids"], shape.E)
        assert np.array_equal(cnt, r["counts"])
        assert np.array_equal(off, r["offsets"])
        assert np.array_equal(tok, r["tok"])
        assert np.array_equal(inv, r["inv"])


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import mixture_experts_router_gb300 as cb
    big_T = 1 << 20          # 4M (token, slot) pairs at E = 256 exceed the 1 MiB scratch
    st = cb.cb_moe_dispatch_noalloc(16, big_T, 4, 256, 16, 16, 16, 16, None, 0)
    assert st == cb.CB_ERR_UNSUPPORTED
