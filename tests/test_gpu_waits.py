"""The kernels' bounded waits give up (a 2 s limit) and report
DSPARK_ST_TIMEOUT instead of hanging, and the context stays usable: each
wait is run on a condition that nothing fulfils (an mbarrier that gets one
of its two arrivals; a counter that is never raised), next to the same wait
on a condition that holds.  No fault and no hang is involved."""
import ctypes
import time

import numpy as np
import pytest
import torch

import draft_sampling_verification_gb300 as ds
from draft_sampling_verification_gb300 import _lib
from parity import np_

pytestmark = pytest.mark.gpu


def wait(which, count=None, target=0):
    st = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    rc = _lib.load().dspark_debug_wait(
        which, ctypes.c_void_p(count.data_ptr()) if count is not None else None, target,
        ctypes.c_void_p(st.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    t0 = time.perf_counter()
    torch.cuda.synchronize()
    return int(st.item()), time.perf_counter() - t0


def test_mbarrier_wait_times_out_and_completes():
    st, secs = wait(0)
    assert st == ds.ST_TIMEOUT and 1.5 < secs < 30
    st, secs = wait(1)
    assert st == ds.ST_OK and secs < 1.0


def test_count_wait_times_out_and_completes():
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    st, secs = wait(2, cnt, 1)
    assert st == ds.ST_TIMEOUT and 1.5 < secs < 30
    cnt.fill_(5)
    st, secs = wait(2, cnt, 5)
    assert st == ds.ST_OK and secs < 1.0


def test_context_usable_after_timeouts():
    wait(0)
    x = torch.randn(4, 4099, device="cuda")
    q = ds.q_build(x)
    torch.cuda.synchronize()
    assert np.all(np_(q["status"]) == 0)
    assert np.all(np_(q["counts"]).view(np.uint32).astype(np.uint64).sum(axis=1) == 1 << 24)
