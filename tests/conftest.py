import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


def pytest_terminal_summary(terminalreporter):
    """One line per default-path full-size GPU parity check (and a count of all
    checks): tokens whose outputs were compared, m-tiles covered, worst
    errors, near and exact ties."""
    harness = sys.modules.get("gpu_harness")
    reports = getattr(harness, "REPORTS", None)
    if not reports:
        return
    tr = terminalreporter
    big = [(t, s, r) for t, s, r in reports if "test_parity_full_size" in t]
    tr.write_sep("-", f"GPU parity against the oracle: {len(reports)} layers checked; the default path at full size:")
    tr.write_line(f"{'check':58s} {'T':>6s} {'E':>4s} {'k':>3s} {'tokens':>6s} {'m-tiles':>9s} {'f32 max':>8s} "
                  f"{'bf16 rel':>8s} {'near':>4s} {'exact':>5s}")
    for test, s, r in big:
        name = test.split("::")[-1].replace("test_parity_full_size", "full size")[:58]
        mt = f"{r.get('mtiles_checked', 0)}/{r.get('mtiles', 0)}"
        tr.write_line(f"{name:58s} {s.T:6d} {s.E:4d} {s.k:3d} {r.get('n_checked', 0):6d} {mt:>9s} "
                      f"{r.get('f32_max_abs', 0.0):8.2e} {r.get('bf16_mean_rel_F', 0.0):8.2e} "
                      f"{r.get('near_tie_tokens', 0):4d} {r.get('exact_tie_tokens', 0):5d}")
    worst = max(r.get("f32_max_abs", 0.0) for _, _, r in reports)
    tr.write_line(f"all {len(reports)} checks: worst fp32 max abs error {worst:.2e} (bound 2e-2); "
                  f"routing, counts, offsets, tok and inv bit-exact")
