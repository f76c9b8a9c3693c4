"""Child process of tests/test_zz_no_alloc.py: cb_moe_dispatch_noalloc in a
process that never creates a layer handle (so nothing but the entry point's
own set-up has prepared the device), checked against the oracle's dispatch.

Cases (E = 256):
  * k = 4, T*k = 93 200: the per-chunk counts fill (47 x 257 words) just over
    the 48 KB a kernel gets without raising its shared-memory limit;
  * k = 4, T*k = 400 000: more chunks than the shared-memory block scan holds,
    so the one-thread-per-expert scan runs;
  * k = 16, T*k = 1 920 000: near the static scratch's limit;
  * an id out of range, reported through the status word.
Each case runs twice in a row.  Prints NOALLOC_OK and exits 0 when all pass.
"""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import mixture_experts_router_gb300 as cb  # noqa: E402
import oracle  # noqa: E402


def skewed_ids(T, E, k, seed):
    """k distinct experts per token, drawn Gumbel-top-k with a Zipf-like
    popularity 2 ln(1/(e+1)) (a few experts take most pairs)."""
    rng = np.random.default_rng(seed)
    pop = 2.0 * np.log(1.0 / (np.arange(E) + 1.0))
    ids = np.empty((T, k), np.int32)
    for t0 in range(0, T, 8192):
        g = pop - np.log(-np.log(rng.random((min(8192, T - t0), E))))
        ids[t0:t0 + len(g)] = np.argpartition(-g, k - 1, axis=1)[:, :k]
    return ids


def noalloc(ids_np, E):
    T, k = ids_np.shape
    ids = torch.from_numpy(np.ascontiguousarray(ids_np)).cuda()
    fill = lambda n: torch.full((n,), -7, dtype=torch.int32, device="cuda")
    counts, offsets, tok, inv, status = fill(E), fill(E + 1), fill(T * k), fill(T * k), fill(1)
    st = cb.cb_moe_dispatch_noalloc(ids.data_ptr(), T, k, E, counts.data_ptr(), offsets.data_ptr(),
                                    tok.data_ptr(), inv.data_ptr(), status.data_ptr(), 0)
    assert st == cb.CB_OK, cb.cb_status_string(st)
    torch.cuda.synchronize()
    return (counts.cpu().numpy(), offsets.cpu().numpy(), tok.cpu().numpy(), inv.cpu().numpy().reshape(T, k),
            int(status.item()))


def main():
    E = 256
    for T, k, seed in [(23300, 4, 1), (100000, 4, 2), (120000, 16, 3)]:
        ids = skewed_ids(T, E, k, seed)
        want = oracle.dispatch(ids, E)
        for _ in range(2):
            *got, status = noalloc(ids, E)
            assert status == 0, status
            for g, w, name in zip(got, want, ("counts", "offsets", "tok", "inv")):
                assert np.array_equal(g, w), (T, k, name)
        print(f"T={T} k={k}: counts, offsets, tok, inv equal the oracle's (two calls)")
    bad = skewed_ids(3000, E, 4, 4)
    bad[1234, 2] = E               # one id out of range
    for _ in range(2):
        *_, status = noalloc(bad, E)
        assert status == cb.CB_ERR_DEVICE, status
    print("out-of-range id reported as CB_ERR_DEVICE")
    print("NOALLOC_OK")


if __name__ == "__main__":
    main()
