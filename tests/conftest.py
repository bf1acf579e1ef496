import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session", autouse=True)
def _build_oracle():
    import oracle

    oracle.build()


def pytest_terminal_summary(terminalreporter):
    """Parity statistics of the GPU checks: near-tie pixels, and per gradient check the
    elements held to the derived fp32 bound with the worst ratios."""
    gu = sys.modules.get("gpu_util")
    stats = getattr(gu, "STATS", None) if gu else None
    if not stats:
        return
    tr = terminalreporter
    pix = [s for s in stats if s["kind"] == "pixels"]
    el = [s for s in stats if s["kind"] == "elements"]
    tr.write_line(f"parity: {len(pix)} forward checks, {sum(s['n'] for s in pix)} pixels, "
                  f"{sum(s['stop_ties'] for s in pix)} stop near-ties "
                  f"({sum(s['other_stop'] for s in pix)} took the other stop), "
                  f"{sum(s['clamp_ties'] for s in pix)} clamp near-ties")
    n, t2 = sum(s["n"] for s in el), sum(s["tier2"] for s in el)
    if el:
        tr.write_line(f"parity: {len(el)} gradient checks, {n} elements, {t2} held to the "
                      f"derived bound ({t2 / max(n, 1):.2%}); worst err/|ref| "
                      f"{max(s['worst_rel'] for s in el):.3g}, err/magnitude "
                      f"{max(s.get('worst_err_over_mag', 0.0) for s in el):.3g}, err/bound "
                      f"{max(s['worst_err_over_bound'] for s in el):.3g}")
