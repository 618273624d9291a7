import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on CPU")


@pytest.fixture(scope="session")
def oracle():
    from oracle import oracle as O
    O.build()
    return O


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter):
    """The verification band statistics of every GPU comparison in the
    session (ratio and match modes), against the bound of 1e-4 band cases per
    verify row under both readings of the draw's band."""
    parity = sys.modules.get("parity")
    if parity is None or not getattr(parity, "SESSION", None):
        return
    tr = terminalreporter
    tr.section("verification band cases (oracle flags; bound %.0e per verify row)"
               % parity.BAND_BOUND)
    for mode, c in sorted(parity.SESSION.items()):
        if mode == "greedy":
            tr.write_line("greedy: %d requests, %d rows, bit-exact" % (c.requests, c.rows))
            continue
        rows = max(1, c.rows)
        tr.write_line(
            "%s: %d requests, %d rows; ambiguous decisions %d; draws near a boundary: "
            "absolute %d, relative %d; band cases absolute %d (%.2e per row, %s), relative %d "
            "(%.2e per row, %s); GPU-only flags %d; requests differing outside the band %d, "
            "inside it %d, outside the relative band %d"
            % (mode, c.requests, c.rows, c.ambig, c.near_abs, c.near_rel, c.band_abs,
               c.band_abs / rows, "bound met" if c.band_abs <= parity.BAND_BOUND * rows
               else "bound NOT met", c.band_rel, c.band_rel / rows,
               "bound met" if c.band_rel <= parity.BAND_BOUND * rows else "bound NOT met",
               c.gpu_only, c.mismatch, c.band_mismatch, c.rel_mismatch))
