"""dspark_spec_step_noalloc -- the whole step with the library's own device
scratch array instead of a caller's workspace.  Two calls in a row (the
second must not depend on what the first left in the array) give exactly
the outputs of dspark_spec_step with a fresh caller workspace, in the
one-launch schedule (which uses the scratch) and the automatic one.  This
file is collected last and also passes alone."""
import pytest
import torch

import draft_sampling_verification_gb300 as ds
from draft_sampling_verification_gb300 import workloads as W
from parity import dev_inputs

pytestmark = pytest.mark.gpu


def outputs(wl, dev):
    B, depth, V = wl.B, wl.depth, wl.V
    mk = lambda *s: torch.full(s, -7, dtype=torch.int32, device=dev)
    return {"counts": mk(B * depth, V), "tok": mk(B, depth), "rst": mk(B * depth),
            "g": (mk(B), mk(B, depth + 1), mk(B)),
            "r": (mk(B), mk(B, depth + 1), mk(B), mk(B))}


def run(fn, wl, d, t, temps, req, schedule, **kw):
    o = outputs(wl, d.device)
    fn(d, t, wl.B, wl.depth, temps, wl.seed, req, o["counts"], o["tok"], o["rst"], o["g"], o["r"],
       schedule=schedule, **kw)
    torch.cuda.synchronize()
    return o


def same(a, b):
    for k in ("counts", "tok", "rst"):
        assert torch.equal(a[k], b[k]), k
    for k in ("g", "r"):
        for x, y in zip(a[k], b[k]):
            assert torch.equal(x, y), k


@pytest.mark.parametrize("name,B,schedule", [("c2", 4, ds.SCHEDULE_AUTO),
                                             ("c4", 8, ds.SCHEDULE_ONE_LAUNCH),
                                             ("c4", 24, ds.SCHEDULE_ONE_LAUNCH),
                                             ("c4", 24, ds.SCHEDULE_AUTO)])
def test_noalloc_equals_workspace_entry(name, B, schedule):
    wl = W.by_name(name, B=B)
    d, t, temps, req = dev_inputs(wl)
    work = torch.empty(B + 1, dtype=torch.int32, device=d.device)
    ref = run(ds.dspark_spec_step, wl, d, t, temps, req, schedule, workspace=work)
    first = run(ds.dspark_spec_step_noalloc, wl, d, t, temps, req, schedule)
    second = run(ds.dspark_spec_step_noalloc, wl, d, t, temps, req, schedule)
    same(first, ref)
    same(second, ref)
    assert int((ref["rst"] != 0).sum()) == 0


def test_noalloc_rejects_oversize_batch():
    wl = W.by_name("c2")
    d, t, temps, req = dev_inputs(wl)
    o = outputs(wl, d.device)
    lib = ds._lib.load()
    big = 65536  # one more than the scratch array holds
    rc = lib.dspark_spec_step_noalloc(
        d.data_ptr(), 0, wl.V, t.data_ptr(), 1, wl.V, big, wl.depth, wl.V, None, 0, None,
        o["counts"].data_ptr(), o["tok"].data_ptr(), o["rst"].data_ptr(), None, None, None,
        o["r"][0].data_ptr(), o["r"][1].data_ptr(), None, o["r"][3].data_ptr(), 0, None)
    assert rc == -2
