"""Benchmark of the draft-sampling / verification hot path on GB300.

One step = the whole path over one batch: the q build with the draft draw
and the workload's verification modes.  With `--schedule auto` (default) a
dense-q step runs the one-launch dspark_spec_step where the library's
automatic choice is that schedule (small batches), and otherwise
dspark_q_build_sample (q and the draft draw, one launch) followed by
dspark_verify (every verification mode in one pass, one launch) -- the two
kernels dspark_spec_step's separate schedule enqueues, called one by one
here so that each is timed.  Default workload:
C4 -- B = 256 requests, depth 5, V = 129,280, fp32 draft / bf16 target logits,
Zipf rows with 10 % grammar masks and 1 % tied-remainder rows, dense q,
greedy and ratio verification (every step of the path but the top-k support,
which `--workload c3` covers).

Prints ONE JSON line (rank 0):
  value   verify rows/s (B x 6 rows per step) with inputs resident in HBM,
          device time from CUDA events on the launching stream;
  e2e     the same metric through the host-buffer C-ABI call
          (dspark_spec_step_host) on pinned host buffers: the H2D copies of
          the step's logits and the D2H copies of its results are inside the
          timed region; steps alternate over two streams;
  roofline  the dominant kernel's algorithmic bytes per launch / its mean
          CUDA-event duration, against the measured HBM copy bandwidth;
  cpu_baseline  the CPU oracle timed on a bounded sample of the workload.
`--impl reference` times the CPU oracle itself as the reference arm.
Multi-GPU (torchrun): every rank runs its own B requests (request ids offset
by rank), no collective on the data path; the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
METRIC = "verify rows/s at V=129280 (B x 6 rows)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c4")
    ap.add_argument("--batch", type=int, default=0, help="override B (requests per GPU)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-wire", action="store_true",
                    help="skip the received-q (pack + validate) measurement")
    ap.add_argument("--no-match", action="store_true",
                    help="skip the stochastic (match) verification measurement")
    ap.add_argument("--no-chain", action="store_true",
                    help="skip the Markov-conditioned draft chain measurement")
    ap.add_argument("--no-sharded", action="store_true",
                    help="skip the vocabulary-sharded (TP2 emulation) q build measurement")
    ap.add_argument("--no-c5", action="store_true",
                    help="skip the C5 B = 1024 (top-256 and dense q) measurement")
    ap.add_argument("--schedule", default="auto", choices=["auto", "one", "separate"],
                    help="dense q: one persistent launch, or q build then one verify pass")
    ap.add_argument("--sweep", action="store_true",
                    help="the batch sweep (B in 1..1024, top-256 q, all-accept and all-reject "
                         "targets, greedy and ratio timed apart): one JSON line per (B, "
                         "variant) instead of the single bench line")
    return ap.parse_args()


def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


# --------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", "dspark_clocks_%d_%d.csv" % (os.getpid(), device_index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------- multi-rank
def rank_request_ids(request_ids, rank, B):
    """Request ids of a rank's B requests: every rank runs its own requests,
    offset by rank * B, so the outputs equal those of one batch of all ranks'
    requests (the RNG is keyed by request id) and no data is exchanged."""
    return (np.asarray(request_ids, np.uint32) + np.uint32(rank * B)).astype(np.uint32)


def max_over_ranks(values):
    """In place: the element-wise max of a float tensor over all ranks."""
    import torch
    torch.distributed.all_reduce(values, op=torch.distributed.ReduceOp.MAX)
    return values


# ------------------------------------------------------------ our arm
# ncu summaries under profiles/: the kernel they cover, the sources it is
# built from, and the unit its traffic is given per
PROFILES = {
    ("q_build_sample", "dense"): ("q_dense_c4_b64.md", ("q_dense.cu", "q_dense.cuh", "common.cuh"),
                                  "traffic_bytes_per_row"),
    ("q_build_sample", "topk"): ("q_topk_c3_b64.md", ("q_topk.cu", "common.cuh",
                                                       "support_alloc.cuh"),
                                 "traffic_bytes_per_row"),
}


def profiled_traffic(wl, dom):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary (per draft row, scaled by the rows of one launch), or None when
    there is none for it or its sources changed since the counters were taken."""
    entry = PROFILES.get((dom, "topk" if wl.top_k else "dense"))
    if entry is None:
        return None
    fname, sources, unit = entry
    try:
        text = open(os.path.join(ROOT, "profiles", fname)).read()
        vals = {}
        for line in text.splitlines():
            if line.startswith((unit + ":", "sources_sha256_16:")):
                k, v = line.split(":", 1)
                vals[k] = v.strip()
        h = hashlib.sha256()
        for name in sources:
            with open(os.path.join(ROOT, "draft_sampling_verification_gb300", "csrc", name),
                      "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != vals.get("sources_sha256_16"):
            return None
        return int(vals[unit]) * wl.B * wl.depth
    except (OSError, KeyError, ValueError):
        return None


def algorithmic_bytes(wl, acc_greedy, acc_ratio):
    """Bytes each kernel must move per launch (what the method reads/writes)."""
    R_d = wl.B * wl.depth
    V = wl.V
    esz_t = 4 if wl.target_dtype == "f32" else 2
    # q build + draw: draft logits read, q written, tokens written
    if wl.top_k > 0:
        q_bytes = R_d * V * 4 + R_d * (wl.top_k * 8 + 4) + R_d * 4
        q_row = wl.top_k * 8 + 4
    else:
        q_bytes = R_d * V * 4 * 2 + R_d * 4
        q_row = V * 4
    # one verification pass: a request's target rows up to the later of the
    # modes' deciding rows, and the q row of a ratio rejection (residual)
    accs = [a for a in (acc_greedy, acc_ratio) if a is not None]
    acc = np.maximum.reduce(accs) if len(accs) > 1 else accs[0]
    rows = ((acc.astype(np.int64) + 1) * V * esz_t).sum()
    resid = (acc_ratio < wl.depth).sum() * q_row if acc_ratio is not None else 0
    return {"q_build_sample": q_bytes, "verify": int(rows + resid)}


def full_read_bytes(wl):
    """Bytes a step moves when every request reads all its target rows and
    one q row back for the residual, whatever the outcome: the upper bound
    that the outcome-dependent count above falls under."""
    ab = algorithmic_bytes(wl, None, np.zeros(wl.B, np.int32))
    esz_t = 4 if wl.target_dtype == "f32" else 2
    q_row = wl.top_k * 8 + 4 if wl.top_k > 0 else wl.V * 4
    return ab["q_build_sample"] + wl.B * ((wl.depth + 1) * wl.V * esz_t + q_row)


def run_ours(args, rank, world, local_rank):
    import torch

    import draft_sampling_verification_gb300 as ds
    from draft_sampling_verification_gb300 import build as dsbuild
    from draft_sampling_verification_gb300 import workloads as W

    dsbuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = W.by_name(args.workload, **({"B": args.batch} if args.batch else {}))
    B, depth, V = wl.B, wl.depth, wl.V
    req_np = rank_request_ids(wl.request_ids, rank, B)

    # inputs resident in HBM; a small step's inputs are rotated over enough
    # copies (> 3 x L2 in all) that each step reads them from HBM
    xd = torch.from_numpy(wl.draft).to(dev)
    if wl.target_dtype == "f32":
        xt = torch.from_numpy(wl.target).to(dev)
    else:
        xt = torch.from_numpy(wl.target.view(np.int16)).to(dev).view(torch.bfloat16)
    in_bytes = wl.draft.nbytes + wl.target.nbytes
    n_copies = max(1, -(-3 * L2_BYTES // in_bytes)) if in_bytes < 3 * L2_BYTES else 1
    copies = [(xd, xt)] + [(xd.clone(), xt.clone()) for _ in range(n_copies - 1)]
    temps = torch.from_numpy(wl.temperature).to(dev)
    req = torch.from_numpy(req_np.view(np.int32)).to(dev)
    rows_d = B * depth
    top_k = wl.top_k
    if top_k > 0:
        counts = torch.empty((rows_d, top_k), dtype=torch.int32, device=dev)
        ids = torch.empty((rows_d, top_k), dtype=torch.int32, device=dev)
        nnz = torch.empty((rows_d,), dtype=torch.int32, device=dev)
    else:
        counts = torch.empty((rows_d, V), dtype=torch.int32, device=dev)
        ids = nnz = None
    qst = torch.empty((rows_d,), dtype=torch.int32, device=dev)
    tok = torch.empty((B, depth), dtype=torch.int32, device=dev)
    sst = torch.empty((B, depth), dtype=torch.int32, device=dev)
    outs = {m: (torch.empty(B, dtype=torch.int32, device=dev),
                torch.empty((B, depth + 1), dtype=torch.int32, device=dev),
                torch.empty(B, dtype=torch.int32, device=dev),
                torch.empty(B, dtype=torch.int32, device=dev)) for m in wl.modes}
    stream = torch.cuda.current_stream(dev)
    if top_k > 0:
        one_launch = False
    elif args.schedule == "auto":
        one_launch = ds.dspark_spec_step_schedule(B, depth) == ds.SCHEDULE_ONE_LAUNCH
    else:
        one_launch = args.schedule == "one"
    work = torch.empty(B + 1, dtype=torch.int32, device=dev)
    kernels = ["spec_step"] if one_launch else ["q_build_sample", "verify"]
    sst.zero_()
    g = outs.get("greedy")
    g = (g[0], g[1], g[3]) if g else None
    r = outs.get("ratio")

    def step(x_d, x_t, marks=None):
        if marks:
            marks[0].record(stream)
        if one_launch:
            ds.dspark_spec_step(x_d, x_t, B, depth, temps, wl.seed, req, counts, tok, qst, g, r,
                                work, stream, ds.SCHEDULE_ONE_LAUNCH)
            if marks:
                marks[1].record(stream)
            return
        ds.dspark_q_build_sample(x_d, B, depth, temps, top_k, wl.seed, req, counts, ids, nnz,
                                 tok, qst, stream)
        if marks:
            marks[1].record(stream)
        ds.dspark_verify(x_t, B, depth, tok, g, r, counts, ids, nnz, top_k, wl.seed, req, stream)
        if marks:
            marks[2].record(stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step(xd, xt)
    torch.cuda.synchronize()
    assert int((qst != 0).sum()) == 0 and int((sst != 0).sum()) == 0, "refused rows in bench"
    for m in wl.modes:
        assert int((outs[m][3] != 0).sum()) == 0, "refused requests in bench"
    acc = {m: outs[m][0].cpu().numpy() for m in wl.modes}
    # the step's integer outputs, for the comparison with the oracle
    gpu_out = {"tok": tok.cpu().numpy(), "qst": qst.cpu().numpy().reshape(B, depth)}
    for m in wl.modes:
        o = [x.cpu().numpy() for x in outs[m]]
        gpu_out[m] = (o[0], o[1], o[3]) if m == "greedy" else (o[0], o[1], o[2], o[3])
    abytes = algorithmic_bytes(wl, acc.get("greedy"), acc.get("ratio"))
    if one_launch:
        abytes = {"spec_step": sum(abytes.values())}

    # ---- device-timed region (inputs resident)
    clocks = ClockSampler(local_rank)
    nmarks = len(kernels) + 1
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(nmarks)]
             for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        step(*copies[s % n_copies], marks[s])
    t_end.record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    per_kernel = {k: 0.0 for k in kernels}
    for s in range(args.steps):
        for i, k in enumerate(kernels):
            per_kernel[k] += marks[s][i].elapsed_time(marks[s][i + 1])
    per_kernel = {k: v / args.steps for k, v in per_kernel.items()}

    # ---- end to end: the host-buffer entry (dspark_spec_step_host) on pinned
    #      host buffers, its copies inside the timed region.  Steps alternate
    #      between two streams, each with its own staging buffer, so the copy
    #      engine loads one step's inputs while the SMs run the previous step.
    e2e = None
    if not args.no_e2e:
        h_d = torch.from_numpy(np.ascontiguousarray(wl.draft)).pin_memory()
        h_t = (torch.from_numpy(np.ascontiguousarray(wl.target)) if wl.target_dtype == "f32"
               else torch.from_numpy(np.ascontiguousarray(wl.target).view(np.int16)).view(
                   torch.bfloat16)).pin_memory()
        h_temp = torch.from_numpy(np.ascontiguousarray(wl.temperature)).pin_memory()
        h_req = torch.from_numpy(np.ascontiguousarray(req_np).view(np.int32)).pin_memory()
        n_st = 2
        streams = [torch.cuda.Stream(dev) for _ in range(n_st)]
        sbytes = ds.dspark_spec_step_host_staging_bytes(B, depth, V, ds._dtype_code(h_d),
                                                        ds._dtype_code(h_t))
        staging = [torch.empty((sbytes,), dtype=torch.uint8, device=dev) for _ in range(n_st)]

        def pinned(shape):
            return torch.empty(shape, dtype=torch.int32).pin_memory()

        h_out = []
        for _ in range(n_st):
            o = {"tok": pinned((B, depth)), "rst": pinned((rows_d,))}
            if "greedy" in wl.modes:
                o["greedy"] = (pinned((B,)), pinned((B, depth + 1)), pinned((B,)))
            if "ratio" in wl.modes:
                o["ratio"] = (pinned((B,)), pinned((B, depth + 1)), pinned((B,)), pinned((B,)))
            h_out.append(o)

        def e2e_step(i):
            o = h_out[i % n_st]
            ds.dspark_spec_step_host(h_d, h_t, B, depth, h_temp, wl.seed, h_req, o["tok"],
                                     o["rst"], staging[i % n_st], greedy_out=o.get("greedy"),
                                     ratio_out=o.get("ratio"), stream=streams[i % n_st])

        for i in range(max(2, args.warmup // 2)):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(streams[0])
        for st_ in streams[1:]:
            st_.wait_event(e0)
        for i in range(args.steps):
            e2e_step(i)
        for st_ in streams[1:]:
            streams[0].wait_stream(st_)
        e1.record(streams[0])
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.steps
        h2d = (h_d.numel() * h_d.element_size() + h_t.numel() * h_t.element_size()
               + h_temp.numel() * 4 + h_req.numel() * 4)
        o = h_out[0]
        d2h = (o["tok"].numel() + o["rst"].numel()
               + sum(t.numel() for m in ("greedy", "ratio") for t in o.get(m, ()))) * 4
        e2e = {"ms_per_step": e2e_ms, "h2d": h2d, "d2h": d2h, "streams": n_st}

    # ---- the received-q path on this step's q rows: the sender's pack
    #      (wire values + checksums), the receiver's validation (values,
    #      support, mass, the proposed tokens, the checksums); not part of the
    #      step above
    wire = None
    if not args.no_wire:
        width = counts.shape[1]
        qf = torch.empty((rows_d, width), dtype=torch.float32, device=dev)
        cs = torch.empty((rows_d,), dtype=torch.int64, device=dev)
        rec = torch.empty((rows_d, width), dtype=torch.int32, device=dev)
        wst = torch.empty((rows_d,), dtype=torch.int32, device=dev)
        toks = tok.reshape(-1)

        def wire_step(ev=None):
            if ev:
                ev[0].record(stream)
            ds.dspark_q_pack(counts, ids, nnz, top_k, V, qf, cs, stream)
            if ev:
                ev[1].record(stream)
            ds.dspark_q_validate(qf, ids, nnz, top_k, V, toks, cs, rec, wst, stream)
            if ev:
                ev[2].record(stream)

        for _ in range(max(3, args.warmup)):
            wire_step()
        torch.cuda.synchronize()
        assert int((wst != 0).sum()) == 0 and torch.equal(rec, counts), "wire round trip"
        wev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        for s_ in range(args.steps):
            wire_step(wev[s_])
        torch.cuda.synchronize()
        pack_ms = sum(e[0].elapsed_time(e[1]) for e in wev) / args.steps
        val_ms = sum(e[1].elapsed_time(e[2]) for e in wev) / args.steps
        entries = rows_d * width
        # pack: counts (and ids) read, q written, checksums written;
        # validate: q (and ids) read, counts written, tokens, checksums and
        # statuses
        per = 4 * entries + (4 * entries if top_k else 0)
        pack_b = per + 4 * entries + 8 * rows_d
        val_b = per + 4 * entries + 16 * rows_d
        wire = {"pack_ms": pack_ms, "validate_ms": val_ms, "pack_bytes": pack_b,
                "validate_bytes": val_b}

    # ---- stochastic (match) verification of this step's drafts, timed apart
    #      from the step: per request, the target rows up to the deciding row
    match = None
    if not args.no_match:
        mo = [torch.empty(B, dtype=torch.int32, device=dev),
              torch.empty((B, depth + 1), dtype=torch.int32, device=dev),
              torch.empty(B, dtype=torch.int32, device=dev),
              torch.empty(B, dtype=torch.int32, device=dev)]

        def match_step():
            ds.dspark_verify_match(xt, B, depth, tok, wl.seed, req, *mo, stream)

        for _ in range(max(3, args.warmup)):
            match_step()
        torch.cuda.synchronize()
        assert int((mo[3] != 0).sum()) == 0, "refused requests in the match verification"
        esz_t = xt.element_size()
        rows_read = (mo[0].to(torch.int64) + 1).sum().item()
        me0 = torch.cuda.Event(enable_timing=True)
        me1 = torch.cuda.Event(enable_timing=True)
        me0.record(stream)
        for _ in range(args.steps):
            match_step()
        me1.record(stream)
        torch.cuda.synchronize()
        match = {"ms": me0.elapsed_time(me1) / args.steps, "bytes": int(rows_read * V * esz_t),
                 "mean_accept": float(mo[0].float().mean().item())}

    # ---- the Markov-conditioned draft chain on this step's draft rows, with
    #      a synthetic bias table of 64 rows (dense q only), timed apart
    chain = None
    if not args.no_chain and top_k == 0:
        gbias = torch.Generator(device=dev)
        gbias.manual_seed(1234)
        bias = torch.randn((64, V), generator=gbias, device=dev, dtype=torch.float32)
        anchors = torch.from_numpy((req_np % V).astype(np.int32)).to(dev)
        ctok = torch.empty((B, depth), dtype=torch.int32, device=dev)
        cst = torch.empty((rows_d,), dtype=torch.int32, device=dev)
        cmg = torch.empty((B, depth), dtype=torch.float32, device=dev)

        def chain_step():
            ds.dspark_q_chain_sample(xd, B, depth, temps, bias, anchors, wl.seed, req, None,
                                     counts, ctok, cst, cmg, stream)

        for _ in range(max(3, args.warmup)):
            chain_step()
        torch.cuda.synchronize()
        assert int((cst != 0).sum()) == 0, "refused rows in the chain"
        ce0 = torch.cuda.Event(enable_timing=True)
        ce1 = torch.cuda.Event(enable_timing=True)
        ce0.record(stream)
        for _ in range(args.steps):
            chain_step()
        ce1.record(stream)
        torch.cuda.synchronize()
        # the method's bytes: base logits and the bias row read, counts written
        chain = {"ms": ce0.elapsed_time(ce1) / args.steps,
                 "bytes": rows_d * V * (wl.draft.itemsize + 4 + 4)}

    # ---- the vocabulary-sharded q build and draw (two emulated ranks) on
    #      this step's draft rows, timed apart from the step
    sharded = None
    if not args.no_sharded:
        sws = torch.empty((ds.dspark_q_sharded_workspace_bytes(rows_d),), dtype=torch.uint8,
                          device=dev)
        stok = torch.empty((B, depth), dtype=torch.int32, device=dev)
        sst2 = torch.empty((rows_d,), dtype=torch.int32, device=dev)

        def sharded_step():
            ds.dspark_q_build_sample_sharded(xd, B, depth, 2, temps, top_k, wl.seed, req, counts,
                                             ids, nnz, stok, sst2, sws, stream)

        for _ in range(max(3, args.warmup)):
            sharded_step()
        torch.cuda.synchronize()
        se0 = torch.cuda.Event(enable_timing=True)
        se1 = torch.cuda.Event(enable_timing=True)
        se0.record(stream)
        for _ in range(args.steps):
            sharded_step()
        se1.record(stream)
        torch.cuda.synchronize()
        sharded = {"ms": se0.elapsed_time(se1) / args.steps,
                   "bytes": abytes.get("q_build_sample", 0) if not one_launch
                   else rows_d * V * 8 + rows_d * 4,
                   "internal": int((sst2 == ds.ST_INTERNAL).sum())}

    # ---- C5 at its largest batch (B = 1,024, mixed targets), top-256 and
    #      dense q: the q build with its draw and one verification pass for
    #      greedy and ratio, timed apart from the step above
    c5 = None
    if not args.no_c5:
        c5 = time_c5_extremes(args, dev, stream, rank)
    ms = elapsed_ms / args.steps
    if world > 1:
        t = max_over_ranks(torch.tensor([ms, e2e["ms_per_step"] if e2e else 0.0], device=dev))
        ms, e2e_max = float(t[0]), float(t[1])
        if e2e:
            e2e["ms_per_step"] = e2e_max
    l2 = ("inputs larger than L2 (%.2f GB per step)" % (in_bytes / 1e9) if n_copies == 1 else
          "inputs rotated over %d copies (%.2f GB in all, > 3 x L2)" % (
              n_copies, n_copies * in_bytes / 1e9))
    return (wl, ms, per_kernel, abytes, clock_info, e2e, l2, wire, match, chain, sharded, gpu_out,
            c5)


def time_c5_extremes(args, dev, stream, rank):
    """C5 B = 1,024 mixed (the C3 generators), top-256 and dense q: per q
    kind the q build with its draw and one dspark_verify of both modes, each
    timed with CUDA events over args.steps launches (inputs larger than L2),
    with the algorithmic bytes of each kernel."""
    import dataclasses

    import torch

    import draft_sampling_verification_gb300 as ds
    from draft_sampling_verification_gb300 import workloads as W
    base = W.config5(1024, variant="mixed")
    base = dataclasses.replace(base, request_ids=rank_request_ids(base.request_ids, rank,
                                                                  base.B))
    xd = torch.from_numpy(base.draft).to(dev)
    xt = torch.from_numpy(base.target).to(dev)
    temps = torch.from_numpy(base.temperature).to(dev)
    req = torch.from_numpy(base.request_ids.view(np.int32)).to(dev)
    out = {"workload": "C5 B=1024 zipf fp32, mixed targets (greedy and ratio)"}
    for kind, k in (("top256", base.top_k), ("dense", 0)):
        wl = dataclasses.replace(base, top_k=k, modes=("greedy", "ratio"))
        B, depth, V = wl.B, wl.depth, wl.V
        q, tok = ds.q_build_sample(xd, B, depth, wl.seed, temps, k, req)
        i32 = lambda *sh: torch.empty(sh, dtype=torch.int32, device=dev)
        g = (i32(B), i32(B, depth + 1), i32(B))
        r = (i32(B), i32(B, depth + 1), i32(B), i32(B))

        def qb():
            ds.dspark_q_build_sample(xd, B, depth, temps, k, wl.seed, req, q["counts"], q["ids"],
                                     q["nnz"], tok, q["status"], stream)

        def vf():
            ds.dspark_verify(xt, B, depth, tok, g, r, q["counts"], q["ids"], q["nnz"], k, wl.seed,
                             req, stream)

        def timed(fn):
            for _ in range(max(3, args.warmup)):
                fn()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / args.steps

        q_ms = timed(qb)
        v_ms = timed(vf)
        qb()
        vf()
        torch.cuda.synchronize()
        assert int((q["status"] != 0).sum()) == 0 and int((g[2] != 0).sum()) == 0 and \
            int((r[3] != 0).sum()) == 0, "refused rows in C5"
        ab = algorithmic_bytes(wl, g[0].cpu().numpy(), r[0].cpu().numpy())
        out[kind] = {"q_build_ms": round(q_ms, 4), "verify_ms": round(v_ms, 4),
                     "step_ms": round(q_ms + v_ms, 4),
                     "verify_rows_per_s": B * (depth + 1) / ((q_ms + v_ms) * 1e-3),
                     "kernel_algorithmic_bytes": ab,
                     "q_build_gbs": ab["q_build_sample"] / (q_ms * 1e-3) / 1e9,
                     "verify_gbs": ab["verify"] / (v_ms * 1e-3) / 1e9,
                     "step_gbs": sum(ab.values()) / ((q_ms + v_ms) * 1e-3) / 1e9}
        del q, tok
    del xd, xt
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------ CPU oracle
def target_rows_f32(wl, b):
    """Request b's target rows as fp32 [1, depth+1, V] (bf16 widened exactly)."""
    t = wl.target[b:b + 1]
    return t if wl.target_dtype == "f32" else (t.astype(np.uint32) << 16).view(np.float32)


def oracle_sample_run(wl, n_req, budget_s):
    """Runs the oracle over up to n_req requests of the workload within about
    budget_s seconds; returns (requests done, seconds)."""
    from oracle import oracle as O
    O.build()
    V, depth = wl.V, wl.depth
    done = 0
    t0 = time.perf_counter()
    for b in range(min(n_req, wl.B)):
        x = wl.draft[b]
        counts, ids, nnz, st = O.q_build(x, wl.temperature[b * depth:(b + 1) * depth], wl.top_k)
        tok, sst = O.draft_sample(counts, ids, nnz, wl.top_k, 1, depth, wl.seed,
                                  wl.request_ids[b:b + 1], V=V)
        z = target_rows_f32(wl, b)
        drafts = tok.reshape(1, depth)
        for m in wl.modes:
            if m == "greedy":
                O.verify_greedy(z, drafts)
            else:
                O.verify_ratio(z, drafts, counts, ids, nnz, wl.top_k, wl.seed,
                               wl.request_ids[b:b + 1])
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return done, time.perf_counter() - t0


# ---- the oracle over a process pool: the workload's arrays sit in shared
#      memory (written once, outside the timed region); a task is one request
_POOL_WL = {}


def oracle_pool_init(meta):
    """Pool worker start: attach the workload's shared arrays, load the oracle."""
    from multiprocessing import shared_memory

    from oracle import oracle as O
    O.build()
    O.lib()
    for key in ("draft", "target"):
        name, shape, dtype = meta[key]
        shm = shared_memory.SharedMemory(name=name)
        _POOL_WL[key + "_shm"] = shm  # kept open for the worker's life
        _POOL_WL[key] = np.ndarray(shape, dtype=np.dtype(dtype), buffer=shm.buf)
    _POOL_WL.update({k: meta[k] for k in ("temperature", "request_ids", "top_k", "seed", "modes",
                                          "target_dtype")})


def oracle_pool_request(b):
    """One request through the oracle (q build, draft sample, verification);
    returns its integer outputs for the comparison with the GPU's."""
    from oracle import oracle as O
    w = _POOL_WL
    x = w["draft"][b]
    depth, V = x.shape
    t = w["target"][b:b + 1]
    z = t if w["target_dtype"] == "f32" else (t.astype(np.uint32) << 16).view(np.float32)
    top_k, seed, req = w["top_k"], w["seed"], w["request_ids"][b:b + 1]
    counts, ids, nnz, st = O.q_build(x, w["temperature"][b * depth:(b + 1) * depth], top_k)
    tok, sst = O.draft_sample(counts, ids, nnz, top_k, 1, depth, seed, req, V=V)
    drafts = tok.reshape(1, depth)
    out = {"b": b, "tok": tok, "qst": st}
    for m in w["modes"]:
        if m == "greedy":
            out[m] = O.verify_greedy(z, drafts)
        else:
            out[m] = O.verify_ratio(z, drafts, counts, ids, nnz, top_k, seed, req)
    return out


class OraclePool:
    """A spawn process pool of every core this process may run on, with the
    workload's arrays in shared memory (written once, outside any timing);
    run(indices) times the oracle over those requests, one task each."""

    def __init__(self, wl):
        self.wl = wl
        self.cores = (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                      else os.cpu_count()) or 1
        self.shms = []
        self.ex = None

    def __enter__(self):
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        from multiprocessing import shared_memory
        wl = self.wl
        meta = {"temperature": np.ascontiguousarray(wl.temperature),
                "request_ids": np.ascontiguousarray(wl.request_ids), "top_k": wl.top_k,
                "seed": wl.seed, "modes": tuple(wl.modes), "target_dtype": wl.target_dtype}
        try:
            for key, arr in (("draft", wl.draft), ("target", wl.target)):
                arr = np.ascontiguousarray(arr)
                shm = shared_memory.SharedMemory(create=True, size=max(1, arr.nbytes))
                self.shms.append(shm)
                np.ndarray(arr.shape, dtype=arr.dtype, buffer=shm.buf)[...] = arr
                meta[key] = (shm.name, arr.shape, arr.dtype.str)
            self.ex = ProcessPoolExecutor(max_workers=self.cores,
                                          mp_context=mp.get_context("spawn"),
                                          initializer=oracle_pool_init, initargs=(meta,))
            list(self.ex.map(int, range(self.cores)))  # every worker started and attached
        except BaseException:
            self.__exit__(None, None, None)
            raise
        return self

    def run(self, indices, keep=None):
        """Seconds for the oracle over these requests; their outputs are
        appended to `keep` (a list) when given."""
        t0 = time.perf_counter()
        res = list(self.ex.map(oracle_pool_request, list(indices)))
        secs = time.perf_counter() - t0
        if keep is not None:
            keep.extend(res)
        return secs

    def __exit__(self, *exc):
        if self.ex is not None:
            self.ex.shutdown()
            self.ex = None
        for shm in self.shms:
            shm.close()
            shm.unlink()
        self.shms = []
        return False


def cpu_baseline(wl, budget_s, keep=None):
    """The oracle on the host cores: one thread, then requests spread over a
    process pool (spawn) of every core this process may run on.  The pool's
    per-request outputs are appended to `keep` when given."""
    n, secs = oracle_sample_run(wl, wl.B, budget_s)
    rows = n * (wl.depth + 1)
    single = {"value": rows / secs, "unit": "verify rows/s", "cores": 1,
              "sample": "%d of %d requests, one thread, %.1f s" % (n, wl.B, secs)}
    out = {"value": single["value"], "unit": "verify rows/s", "cores": 1, "kind": "oracle",
           "sample": "%d of %d requests of the same workload (q build, draft sample, %s "
                     "verification), single thread, %.1f s" % (n, wl.B, "+".join(wl.modes), secs),
           "single_thread": single}
    if n < 1:
        return out
    with OraclePool(wl) as pool:
        if pool.cores < 2:
            return out
        per_req = secs / n
        n_par = int(min(wl.B, max(pool.cores, pool.cores * budget_s / per_req)))
        psecs = pool.run(range(n_par), keep)
    out.update({"value": n_par * (wl.depth + 1) / psecs, "cores": pool.cores,
                "sample": "%d of %d requests of the same workload (q build, draft sample, %s "
                          "verification) spread over a pool of %d processes, %.1f s; the "
                          "single-thread figure is beside it" % (n_par, wl.B, "+".join(wl.modes),
                                                                pool.cores, psecs)})
    return out


FLAG_AMBIG, FLAG_NEAR, FLAG_NEAR_REL = 1, 2, 8  # the oracle's verification flag bits
BAND_BOUND = 1e-4  # band cases per verify row


def parity_band(wl, gpu, ref):
    """The timed step's integer outputs against the oracle's on the requests
    the oracle ran (`ref`: its per-request outputs).  Draft tokens, row
    statuses and greedy outputs must be equal; ratio outputs must be equal
    outside the oracle's tolerance band (the benchmark definition's).  The band cases are counted from the
    oracle's flags under both readings of the draw's band: absolute (1e-6 in
    probability units) and relative (1e-6 of the picked token's own mass)."""
    depth = wl.depth
    ref = sorted(ref, key=lambda r: r["b"])
    idx = np.array([r["b"] for r in ref], np.int64)
    out = {"requests": int(idx.size), "verify_rows": int(idx.size * (depth + 1)),
           "bound_per_row": BAND_BOUND}
    if idx.size == 0:
        return out
    tok = np.stack([r["tok"].reshape(depth) for r in ref])
    qst = np.stack([np.asarray(r["qst"]).reshape(depth) for r in ref])
    out["draft_tokens_equal"] = bool(np.array_equal(gpu["tok"][idx], tok))
    out["row_status_equal"] = bool(np.array_equal(gpu["qst"][idx], qst))
    if "greedy" in wl.modes:
        acc = np.concatenate([r["greedy"][0] for r in ref])
        com = np.concatenate([r["greedy"][1] for r in ref])
        st = np.concatenate([r["greedy"][2] for r in ref])
        ga, gc, gs = gpu["greedy"]
        out["greedy_equal"] = bool(np.array_equal(ga[idx], acc) and
                                   np.array_equal(gc[idx], com) and np.array_equal(gs[idx], st))
    if "ratio" in wl.modes:
        acc = np.concatenate([r["ratio"][0] for r in ref])
        com = np.concatenate([r["ratio"][1] for r in ref])
        rf = np.concatenate([r["ratio"][2] for r in ref]).astype(np.uint32)
        st = np.concatenate([r["ratio"][3] for r in ref])
        ga, gc, gf, gs = gpu["ratio"]
        gf = gf[idx].astype(np.uint32)
        same = (ga[idx] == acc) & (gc[idx] == com).all(axis=1) & (gs[idx] == st)
        ambig = (rf & FLAG_AMBIG) != 0
        band_abs = ambig | ((rf & FLAG_NEAR) != 0)
        band_rel = ambig | ((rf & FLAG_NEAR_REL) != 0)
        rows = out["verify_rows"]
        out.update({
            "ratio_mismatch_outside_band": int((~same & ~band_abs).sum()),
            "ratio_mismatch_in_band": int((~same & band_abs).sum()),
            "ratio_mismatch_outside_rel_band": int((~same & ~band_rel).sum()),
            "ambiguous_decisions": int(ambig.sum()),
            "draws_near_boundary_abs": int(((rf & FLAG_NEAR) != 0).sum()),
            "draws_near_boundary_rel": int(((rf & FLAG_NEAR_REL) != 0).sum()),
            "band_cases_abs": int(band_abs.sum()), "band_rate_abs": band_abs.sum() / rows,
            "bound_met_abs": bool(band_abs.sum() <= BAND_BOUND * rows),
            "band_cases_rel": int(band_rel.sum()), "band_rate_rel": band_rel.sum() / rows,
            "bound_met_rel": bool(band_rel.sum() <= BAND_BOUND * rows),
            "gpu_only_flags": int((((gf & (FLAG_AMBIG | FLAG_NEAR)) != 0) & ~band_abs).sum()),
            "readings": "abs: a draw within 1e-6 (probability units) of a cumulative boundary; "
                        "rel: within 1e-6 of the picked token's own mass; both count the "
                        "decisions with |u*q - p| <= 1e-6*q"})
    return out


def run_sweep(args):
    """The batch sweep of the benchmark definition: B in {1, 8, 32, 128, 512,
    1024} x depth 5 x V = 129,280 with the Zipf generators, a top-256 and a
    dense q, the all-accept (target = draft) and all-reject (target mass off
    the draft support) extremes; the q build with its draw and each
    verification mode are timed apart with CUDA events, and each line gives
    rows/s and algorithmic GB/s per mode."""
    import dataclasses
    import torch

    import draft_sampling_verification_gb300 as ds
    from draft_sampling_verification_gb300 import build as dsbuild
    from draft_sampling_verification_gb300 import workloads as W

    dsbuild.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    peak = (load_peaks() or {}).get("hbm_gbs")
    def run_one(wl, B, variant, q_kind):
        depth, V, k = wl.depth, wl.V, wl.top_k
        xd = torch.from_numpy(wl.draft).to(dev)
        xt = torch.from_numpy(wl.target).to(dev)
        in_bytes = wl.draft.nbytes + wl.target.nbytes
        n_copies = max(1, -(-3 * L2_BYTES // in_bytes)) if in_bytes < 3 * L2_BYTES else 1
        copies = [(xd, xt)] + [(xd.clone(), xt.clone()) for _ in range(n_copies - 1)]
        temps = torch.from_numpy(wl.temperature).to(dev)
        req = torch.from_numpy(wl.request_ids.view(np.int32)).to(dev)
        rows_d = B * depth
        if k > 0:
            counts = torch.empty((rows_d, k), dtype=torch.int32, device=dev)
            ids = torch.empty((rows_d, k), dtype=torch.int32, device=dev)
            nnz = torch.empty((rows_d,), dtype=torch.int32, device=dev)
        else:
            counts = torch.empty((rows_d, V), dtype=torch.int32, device=dev)
            ids = nnz = None
        qst = torch.empty((rows_d,), dtype=torch.int32, device=dev)
        tok = torch.empty((B, depth), dtype=torch.int32, device=dev)
        i32 = lambda *shape: torch.empty(shape, dtype=torch.int32, device=dev)
        g = (i32(B), i32(B, depth + 1), i32(B))
        r = (i32(B), i32(B, depth + 1), i32(B), i32(B))

        def q_build(i):
            ds.dspark_q_build_sample(copies[i % n_copies][0], B, depth, temps, k, wl.seed,
                                     req, counts, ids, nnz, tok, qst, stream)

        def verify(i, mode):
            ds.dspark_verify(copies[i % n_copies][1], B, depth, tok,
                             g if mode == "greedy" else None,
                             r if mode == "ratio" else None, counts, ids, nnz, k, wl.seed,
                             req, stream)

        def timed(fn):
            for i in range(max(3, args.warmup)):
                fn(i)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(args.steps):
                fn(i)
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / args.steps

        q_ms = timed(q_build)
        q_build(0)
        per_mode = {}
        for mode in ("greedy", "ratio"):
            v_ms = timed(lambda i, m=mode: verify(i, m))
            verify(0, mode)
            torch.cuda.synchronize()
            out = g if mode == "greedy" else r
            assert int((out[-1] != 0).sum()) == 0, "refused requests in the sweep"
            acc = out[0].cpu().numpy()
            ab = algorithmic_bytes(wl, acc if mode == "greedy" else None,
                                   acc if mode == "ratio" else None)
            step_ms = q_ms + v_ms
            per_mode[mode] = {
                "verify_ms": round(v_ms, 4), "step_ms": round(step_ms, 4),
                "verify_rows_per_s": B * (depth + 1) / (step_ms * 1e-3),
                "step_gbs": (ab["q_build_sample"] + ab["verify"]) / (step_ms * 1e-3) / 1e9,
                "verify_gbs": ab["verify"] / (v_ms * 1e-3) / 1e9,
                "mean_accept_len": float(acc.mean())}
        qb = algorithmic_bytes(wl, np.zeros(B, np.int32), None)["q_build_sample"]
        print(json.dumps({
            "sweep": "batch sweep, %s q" % ("top-%d" % k if k else "dense"), "B": B,
            "variant": variant, "q": q_kind,
            "q_build_ms": round(q_ms, 4), "q_build_gbs": qb / (q_ms * 1e-3) / 1e9,
            "hbm_peak_gbs": peak, "modes": per_mode,
            "l2": "inputs larger than L2" if n_copies == 1 else
                  "inputs rotated over %d copies" % n_copies}), flush=True)
        del copies, xd, xt
        torch.cuda.empty_cache()

    for B in (1, 8, 32, 128, 512, 1024):
        for variant in ("accept", "reject"):
            wl_gen = W.config5(B, variant=variant)
            for q_kind in ("sparse", "dense"):
                run_one(wl_gen if q_kind == "sparse" else dataclasses.replace(wl_gen, top_k=0),
                        B, variant, q_kind)


def run_reference(args, rank, world):
    from draft_sampling_verification_gb300 import workloads as W
    if rank != 0:
        return
    wl = W.by_name(args.workload)
    from oracle import oracle as O
    O.build()
    # each step: two requests per core of the host (a bounded sample of the
    # workload's batch, taken in turn), spread over a process pool
    with OraclePool(wl) as pool:
        cores = pool.cores
        per_step = max(1, min(wl.B, 2 * cores))
        nxt = 0

        def step():
            nonlocal nxt
            idx = [(nxt + i) % wl.B for i in range(per_step)]
            nxt = (nxt + per_step) % wl.B
            return pool.run(idx)

        for _ in range(args.warmup):
            step()
        secs = sum(step() for _ in range(args.steps))
    done = per_step * args.steps
    value = done * (wl.depth + 1) / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "verify rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64+u64", "data": "synthetic (seeded generators)",
        "config": {"workload": wl.name, "B_per_gpu": wl.B, "depth": wl.depth, "V": wl.V,
                   "sample_per_step": "%d of %d requests" % (per_step, wl.B)},
        "cpu_baseline": {"value": value, "unit": "verify rows/s", "cores": cores, "kind": "oracle",
                         "sample": "%d requests per step of %s over a pool of %d processes" % (
                             per_step, wl.name, cores)},
        "e2e": {"value": value, "unit": "verify rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.sweep:
        run_sweep(args)
        return
    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    (wl, ms, per_kernel, abytes, clocks, e2e, l2, wire, match, chain, sharded, gpu_out,
     c5) = run_ours(args, rank, world, local_rank)
    if rank == 0:
        peaks = load_peaks()
        rows = wl.B * (wl.depth + 1) * world
        value = rows / (ms * 1e-3)
        dom = max(per_kernel, key=per_kernel.get)
        achieved = abytes[dom] / (per_kernel[dom] * 1e-3) / 1e9
        peak = peaks["hbm_gbs"] if peaks else 6800.0
        step_bytes = sum(abytes.values())
        line = {
            "metric": METRIC, "value": value, "unit": "verify rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32+u64", "data": "synthetic (seeded generators)",
            "config": {
                "workload": wl.name,
                "B_per_gpu": wl.B, "depth": wl.depth, "V": wl.V, "q": "top-%d" % wl.top_k
                if wl.top_k else "dense", "verify": list(wl.modes),
                "parallelism": "dp%d (independent requests)" % world,
                "l2": l2,
                "draft_positions_per_s": wl.B * wl.depth * world / (ms * 1e-3),
                "step_algorithmic_bytes": step_bytes,
                "step_full_read_bytes": full_read_bytes(wl),
                "step_achieved_gbs": step_bytes / (ms * 1e-3) / 1e9,
                "kernel_ms": {k: round(v, 4) for k, v in per_kernel.items()},
                "kernel_algorithmic_bytes": abytes,
                **{k: wl.notes[k] for k in ("tie_rows_straddling", "lowest_id_decisive_rows")
                   if k in wl.notes},
            },
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak,
                         "traffic": profiled_traffic(wl, dom),
                         "peak_source": "measured" if peaks else "fallback"},
            "clocks": clocks,
            "gpu_launches": len(per_kernel) * args.steps,
        }
        if e2e:
            line["e2e"] = {"value": rows / (e2e["ms_per_step"] * 1e-3), "unit": "verify rows/s",
                           "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                           "ms_per_step": e2e["ms_per_step"],
                           "how": "dspark_spec_step_host per step (host rows copied to a staging "
                                  "buffer, the step, the outputs copied back), steps alternating "
                                  "over %d streams and staging buffers" % e2e["streams"],
                           "h2d_link_gbs": round(e2e["h2d"] / (e2e["ms_per_step"] * 1e-3) / 1e9,
                                                 1)}
        if wire:
            gbs_p = wire["pack_bytes"] / (wire["pack_ms"] * 1e-3) / 1e9
            gbs_v = wire["validate_bytes"] / (wire["validate_ms"] * 1e-3) / 1e9
            line["received_q"] = {
                "what": "q_pack + q_validate on this step's q rows, timed apart from the step",
                "pack_ms": round(wire["pack_ms"], 4), "validate_ms": round(wire["validate_ms"], 4),
                "pack_algorithmic_bytes": wire["pack_bytes"],
                "validate_algorithmic_bytes": wire["validate_bytes"],
                "roofline": {"bound": "hbm", "unit": "GB/s", "peak": peak,
                             "pack_achieved": gbs_p, "pack_frac": gbs_p / peak,
                             "validate_achieved": gbs_v, "validate_frac": gbs_v / peak},
            }
        if match:
            gbs_m = match["bytes"] / (match["ms"] * 1e-3) / 1e9
            line["match_verify"] = {
                "what": "dspark_verify_match of this step's drafts, timed apart from the step",
                "ms": round(match["ms"], 4), "verify_rows_per_s": wl.B * (wl.depth + 1) * world /
                (match["ms"] * 1e-3), "mean_accept_len": round(match["mean_accept"], 3),
                "algorithmic_bytes": match["bytes"],
                "roofline": {"bound": "hbm", "unit": "GB/s", "peak": peak, "achieved": gbs_m,
                             "frac": gbs_m / peak},
            }
        if chain:
            gbs_c = chain["bytes"] / (chain["ms"] * 1e-3) / 1e9
            line["markov_chain"] = {
                "what": "dspark_q_chain_sample on this step's draft rows (64-row bias table), "
                        "timed apart from the step",
                "ms": round(chain["ms"], 4),
                "draft_positions_per_s": wl.B * wl.depth * world / (chain["ms"] * 1e-3),
                "algorithmic_bytes": chain["bytes"],
                "roofline": {"bound": "hbm", "unit": "GB/s", "peak": peak, "achieved": gbs_c,
                             "frac": gbs_c / peak},
            }
        if sharded:
            gbs_s = sharded["bytes"] / (sharded["ms"] * 1e-3) / 1e9
            line["sharded_q"] = {
                "what": "dspark_q_build_sample_sharded with 2 emulated ranks on this step's draft "
                        "rows, timed apart from the step",
                "ms": round(sharded["ms"], 4), "rows_refused_internal": sharded["internal"],
                "algorithmic_bytes": sharded["bytes"],
                "roofline": {"bound": "hbm", "unit": "GB/s", "peak": peak, "achieved": gbs_s,
                             "frac": gbs_s / peak},
            }
        if c5:
            for kind in ("top256", "dense"):
                e = c5[kind]
                e["roofline"] = {"bound": "hbm", "unit": "GB/s", "peak": peak,
                                 "q_build_frac": e["q_build_gbs"] / peak,
                                 "verify_frac": e["verify_gbs"] / peak,
                                 "step_frac": e["step_gbs"] / peak}
            line["c5_b1024"] = c5
        if not args.no_cpu:
            ref = []
            line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds, ref)
            line["parity_band"] = parity_band(wl, gpu_out, ref)
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
