"""The C-ABI library builds for sm_103a, loads, exports every symbol the
public headers declare, and refuses bad arguments on the host (negative
return codes, nothing launched) -- no GPU needed."""
import ctypes

import pytest

from draft_sampling_verification_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    names = _lib.header_symbols()
    assert set(names) >= {"dspark_q_build", "dspark_draft_sample", "dspark_verify_greedy",
                          "dspark_verify_ratio", "dspark_target_probs", "dspark_version"}
    for n in names:
        assert hasattr(lib, n), n
    assert b"dyadic24-standard-v1" in lib.dspark_version()


def test_no_oracle_symbols_in_library(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True).stdout
    assert "oracle_" not in out


P = ctypes.c_void_p(16)  # a non-null, aligned placeholder; never dereferenced


def test_q_build_argument_errors(lib):
    f = lib.dspark_q_build
    assert f(P, 0, 8, 1, 0, None, 0, P, None, None, P, None) == -2      # V = 0
    assert f(P, 0, 8, 1, 131073, None, 0, P, None, None, P, None) == -2  # V too large
    assert f(P, 0, 4, 1, 8, None, 0, P, None, None, P, None) == -2      # ld < V
    assert f(P, 7, 8, 1, 8, None, 0, P, None, None, P, None) == -3      # dtype
    assert f(P, 0, 8, 1, 8, None, 9, P, None, None, P, None) == -4      # top_k > V
    assert f(P, 0, 8, 1, 8, None, -1, P, None, None, P, None) == -4
    assert f(None, 0, 8, 1, 8, None, 0, P, None, None, P, None) == -1   # null logits
    assert f(P, 0, 8, 1, 8, None, 4, P, None, None, P, None) == -1      # sparse w/o ids
    assert f(ctypes.c_void_p(18), 0, 8, 1, 8, None, 0, P, None, None, P, None) == -5
    assert f(P, 0, 8, 0, 8, None, 0, None, None, None, None, None) == 0  # empty batch


def test_sample_and_verify_argument_errors(lib):
    assert lib.dspark_draft_sample(P, None, None, 0, 1, 0, 8, 0, None, P, P, None) == -2
    assert lib.dspark_draft_sample(P, None, None, 0, 1, 9, 8, 0, None, P, P, None) == -2
    assert lib.dspark_draft_sample(None, None, None, 0, 1, 5, 8, 0, None, P, P, None) == -1
    assert lib.dspark_draft_sample(P, None, None, 0, 0, 5, 8, 0, None, P, P, None) == 0
    assert lib.dspark_verify_greedy(P, 0, 8, 1, 0, 8, P, P, P, P, None) == -2
    assert lib.dspark_verify_greedy(P, 1, 8, 1, 5, 8, None, P, P, P, None) == -1
    assert lib.dspark_verify_greedy(P, 1, 8, 0, 5, 8, P, P, P, P, None) == 0
    assert lib.dspark_verify_ratio(P, 0, 8, 1, 5, 8, P, None, None, None, 0, 0, None, P, P,
                                   None, P, None) == -1
    assert lib.dspark_verify_ratio(P, 0, 8, 1, 5, 8, P, P, None, None, 4, 0, None, P, P,
                                   None, P, None) == -1
    assert lib.dspark_target_probs(P, 0, 8, 1, 0, None, None, P, None) == -2
    assert lib.dspark_verify_stats(P, -1, P, None) == -2               # B < 0
    assert lib.dspark_verify_stats(P, 4, None, None) == -1             # no stats
    assert lib.dspark_verify_stats(None, 4, P, None) == -1             # no flags, B > 0
    assert lib.dspark_verify_stats(ctypes.c_void_p(18), 4, P, None) == -5
    assert lib.dspark_debug_philox(P, 0, -1, P, None) == -2
    assert lib.dspark_debug_exp_weights(None, 4, None, None, None) == -1


def test_spec_step_argument_errors(lib):
    f = lib.dspark_spec_step
    f.argtypes = _lib.SIGNATURES["dspark_spec_step"]
    # draft, dt, ld, target, dt, ld, B, depth, V, temps, seed, req, counts, tok, rst,
    # g_acc, g_com, g_st, r_acc, r_com, r_fl, r_st, workspace, schedule, stream
    ok = [P, 0, 8, P, 1, 8, 1, 5, 8, None, 0, None, P, P, P, P, P, P, P, P, None, P, P, 0, None]

    def call(**kw):
        a = list(ok)
        names = {"V": 8, "depth": 7, "B": 6, "workspace": 22, "schedule": 23, "g_com": 16,
                 "r_acc": 18, "ld_t": 5}
        for k, v in kw.items():
            a[names[k]] = v
        return f(*a)

    assert call(V=0) == -2
    assert call(depth=0) == -2
    assert call(depth=9) == -2
    assert call(ld_t=4) == -2
    assert call(schedule=3) == -7
    assert call(schedule=-1) == -7
    assert call(workspace=None) == -1
    assert call(g_com=None) == -1          # greedy outputs: all three or none
    assert call(B=0) == 0                  # empty batch: nothing enqueued


def test_spec_step_noalloc_host_checks(lib):
    """The no-allocation entry refuses a batch beyond its scratch array, and
    bad arguments, on the host (before any device lookup)."""
    f = lib.dspark_spec_step_noalloc
    # same arguments as dspark_spec_step minus the workspace
    a = [P, 0, 8, P, 1, 8, 1, 5, 8, None, 0, None, P, P, P, P, P, P, P, P, None, P, 0, None]
    big = list(a)
    big[6] = 65536                      # B > DSPARK_SPEC_STATIC_MAX_B
    assert f(*big) == -2
    bad = list(a)
    bad[22] = 5                         # schedule
    assert f(*bad) == -7
    empty = list(a)
    empty[6] = 0
    assert f(*empty) == 0


def test_sharded_argument_errors(lib):
    f = lib.dspark_q_build_sample_sharded
    # (logits, dtype, ld, B, depth, V, n_shards, T, top_k, seed, req, counts, ids, nnz,
    #  tokens, status, workspace, stream)
    ok = (P, 0, 8, 1, 1, 8, 2, None, 0, 0, None, P, None, None, P, P, P, None)

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)

    assert call(a6=0) == -7 and call(a6=9) == -7         # n_shards outside [1, 8]
    assert call(a5=0) == -2                              # V = 0
    assert call(a4=0) == -2                              # depth = 0
    assert call(a8=9) == -4                              # top_k > V
    assert call(a8=4) == -1                              # sparse without ids / nnz
    assert call(a16=None) == -1                          # no workspace
    assert call(a16=ctypes.c_void_p(24)) == -5           # workspace not 16-byte aligned
    assert call(a3=0) == 0                               # empty batch
    assert lib.dspark_q_sharded_workspace_bytes(-1) == 0
    assert lib.dspark_q_sharded_workspace_bytes(3) == 3 * lib.dspark_q_sharded_workspace_bytes(1)


def test_spec_step_host_argument_errors(lib):
    f = lib.dspark_spec_step_host
    # (draft, dd, target, td, B, depth, V, T, seed, req, tok, rst, g_acc, g_com, g_st, r_acc,
    #  r_com, r_flags, r_st, staging, schedule, stream)
    ok = [P, 0, P, 1, 2, 5, 8, None, 0, None, P, P, P, P, P, None, None, None, None,
          ctypes.c_void_p(256), 0, None]

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)

    assert call(a5=0) == -2                        # depth
    assert call(a6=0) == -2                        # V
    assert call(a1=9) == -3                        # dtype
    assert call(a20=7) == -7                       # schedule
    assert call(a19=None) == -1                    # no staging
    assert call(a19=ctypes.c_void_p(272)) == -5    # staging not 256-byte aligned
    assert call(a12=None, a13=None, a14=None) == -1  # no mode
    assert call(a13=None) == -1                    # a partial greedy triple
    assert call(a4=0) == 0                         # empty batch
    sb = lib.dspark_spec_step_host_staging_bytes
    assert sb(2, 5, 8, 0, 1) % 256 == 0 and sb(2, 5, 8, 0, 1) >= 2 * 5 * 8 * 8 + 2 * 6 * 8 * 2
    assert sb(2, 0, 8, 0, 1) == 0 and sb(-1, 5, 8, 0, 1) == 0


def test_debug_wait_argument_errors(lib):
    assert lib.dspark_debug_wait(3, None, 0, P, None) == -7      # which
    assert lib.dspark_debug_wait(0, None, 0, None, None) == -1   # no status
    assert lib.dspark_debug_wait(2, None, 1, P, None) == -1      # count wait without a counter
    assert lib.dspark_debug_wait(0, None, 0, ctypes.c_void_p(18), None) == -5
