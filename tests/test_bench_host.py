"""Host-side parts of bench.py, on CPU: the per-request bf16 widening the
oracle baseline uses, the oracle baseline over a process pool (same
outputs as one thread), and the algorithmic byte counts."""
import numpy as np

import bench
from draft_sampling_verification_gb300 import workloads as W


def test_target_rows_f32_widens_one_request_exactly():
    wl = W.config4(B=3, V=257)
    for b in range(wl.B):
        got = bench.target_rows_f32(wl, b)
        assert got.shape == (1, wl.depth + 1, wl.V) and got.dtype == np.float32
        assert np.array_equal(got[0], wl.target_f32()[b])


def test_pool_requests_match_one_thread(oracle):
    wl = W.config4(B=4, V=1031)
    # the pool worker's request function, run in this process, against the
    # single-thread loop's oracle calls
    meta = {"draft": wl.draft, "target": wl.target, "temperature": wl.temperature,
            "request_ids": wl.request_ids, "top_k": wl.top_k, "seed": wl.seed,
            "modes": tuple(wl.modes), "target_dtype": wl.target_dtype}
    bench._POOL_WL.clear()
    bench._POOL_WL.update(meta)
    for b in range(wl.B):
        assert bench.oracle_pool_request(b)["b"] == b
    n, secs = bench.oracle_sample_run(wl, wl.B, 60.0)
    assert n == wl.B and secs > 0


def test_cpu_baseline_reports_pool_and_single_thread(oracle):
    wl = W.config4(B=8, V=1031)
    out = bench.cpu_baseline(wl, 0.5)
    assert out["kind"] == "oracle" and out["unit"] == "verify rows/s" and out["value"] > 0
    assert out["single_thread"]["cores"] == 1 and out["single_thread"]["value"] > 0
    assert out["cores"] >= 1


def _gpu_like(wl, ref):
    """GPU-shaped outputs (whole batch) built from the oracle's per-request
    outputs, as the bench holds them after its step."""
    ref = sorted(ref, key=lambda r: r["b"])
    out = {"tok": np.stack([r["tok"].reshape(wl.depth) for r in ref]).astype(np.int32),
           "qst": np.stack([np.asarray(r["qst"]).reshape(wl.depth) for r in ref])}
    for m in wl.modes:
        out[m] = tuple(np.concatenate([np.asarray(x)[None] if np.ndim(x) == 0 else x
                                       for x in col]) for col in zip(*[r[m] for r in ref]))
    return out


def test_parity_band_counts(oracle):
    wl = W.config4(B=6, V=1031)
    ref = []
    bench.cpu_baseline(wl, 0.5, ref)
    assert sorted(r["b"] for r in ref) == list(range(len(ref)))
    gpu = _gpu_like(wl, ref)
    out = bench.parity_band(wl, gpu, ref)
    assert out["requests"] == len(ref) and out["verify_rows"] == len(ref) * (wl.depth + 1)
    assert out["draft_tokens_equal"] and out["row_status_equal"] and out["greedy_equal"]
    assert out["ratio_mismatch_outside_band"] == 0 and out["gpu_only_flags"] == 0
    assert out["band_cases_rel"] <= out["band_cases_abs"]
    # a changed committed token outside the band is a mismatch; a changed
    # draft token breaks the token equality
    ga, gc, gf, gs = gpu["ratio"]
    gc = gc.copy()
    gc[0, 0] = gc[0, 0] + 1
    gpu["ratio"] = (ga, gc, gf, gs)
    gpu["tok"] = gpu["tok"].copy()
    gpu["tok"][1, 0] += 1
    bad = bench.parity_band(wl, gpu, ref)
    assert not bad["draft_tokens_equal"]
    flags0 = int(np.asarray(ref[0]["ratio"][2]).ravel()[0])
    in_band = (flags0 & (bench.FLAG_AMBIG | bench.FLAG_NEAR)) != 0
    assert bad["ratio_mismatch_outside_band"] + bad["ratio_mismatch_in_band"] == 1
    assert bad["ratio_mismatch_in_band"] == int(in_band)


def test_algorithmic_bytes_dense_and_sparse():
    wl = W.config4(B=2, V=1031)
    acc = np.array([0, wl.depth], np.int32)
    ab = bench.algorithmic_bytes(wl, acc, acc)
    rows_d = wl.B * wl.depth
    assert ab["q_build_sample"] == rows_d * wl.V * 8 + rows_d * 4
    # request 0 reads 1 target row and its q row (a rejection); request 1 reads all 6
    esz = 2 if wl.target_dtype == "bf16" else 4
    assert ab["verify"] == (1 + wl.depth + 1) * wl.V * esz + wl.V * 4


def test_full_read_bytes_per_request():
    # per request: 5 draft rows read, q written, 6 target rows and one q row
    # read back, 5 tokens written
    V = 129280
    c4 = W.config4(B=1, V=V)
    assert c4.top_k == 0 and c4.target_dtype == "bf16"
    assert bench.full_read_bytes(c4) == 5 * V * 4 * 2 + 6 * V * 2 + V * 4 + 5 * 4
    c3 = W.config3(B=1, V=V)
    k = c3.top_k
    assert k > 0 and c3.target_dtype == "f32"
    assert bench.full_read_bytes(c3) == 5 * V * 4 + 5 * (8 * k + 4) + 6 * V * 4 + (8 * k + 4) \
        + 5 * 4
    # the outcome-dependent count never exceeds it
    acc = np.array([c4.depth], np.int32)
    assert sum(bench.algorithmic_bytes(c4, acc, acc).values()) <= bench.full_read_bytes(c4)


def _args(**kw):
    import types
    a = dict(workload="c1", steps=1, warmup=0, gpus=1)
    a.update(kw)
    return types.SimpleNamespace(**a)


def test_reference_arm_line(oracle, capsys):
    import json
    bench.run_reference(_args(), 0, 1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["unit"] == "verify rows/s" and line["higher_is_better"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_reference_arm_other_ranks_print_nothing(capsys):
    bench.run_reference(_args(), 1, 2)
    assert capsys.readouterr().out == ""
