"""GB300 draft sampling and verification (dyadic24-standard-v1).

Thin Python binding of the C ABI in ``include/dspark.h``: the functions named
like the C calls (``dspark_q_build``, ``dspark_draft_sample``,
``dspark_verify_greedy``, ``dspark_verify_ratio``, ``dspark_target_probs``)
take torch CUDA tensors, pass their device pointers, sizes and the current
stream to libdspark.so, and raise on a nonzero return.  Every step of the
path runs in the library's CUDA kernels; torch only provides device memory
and streams.  The lower-case helpers (``q_build`` ...) allocate the outputs
with torch and call the same entry points.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

M = 1 << 24
F32, BF16 = 0, 1
ST_OK, ST_NONFINITE, ST_ZERO_MASS, ST_ALLOC_INCONSISTENT = 0, 1, 2, 3
ST_BAD_TEMPERATURE, ST_BAD_Q, ST_BAD_DRAFT, ST_TIMEOUT, ST_INTERNAL = 4, 5, 6, 7, 8
ST_BAD_CHECKSUM = 9
FLAG_AMBIG_ACCEPT, FLAG_NEAR_BOUNDARY, FLAG_DEGENERATE = 1, 2, 4
SCHEDULE_AUTO, SCHEDULE_ONE_LAUNCH, SCHEDULE_SEPARATE = 0, 1, 2
PURPOSE_PROPOSAL, PURPOSE_ACCEPT, PURPOSE_RESIDUAL, PURPOSE_BONUS, PURPOSE_MATCH = 0, 1, 2, 3, 4

__all__ = ["dspark_q_build", "dspark_q_build_sample", "dspark_draft_sample", "dspark_verify_greedy",
           "dspark_verify_ratio", "dspark_verify", "dspark_verify_stats", "verify_stats",
           "dspark_target_probs", "dspark_spec_step",
           "dspark_spec_step_schedule", "dspark_spec_step_noalloc", "dspark_q_pack",
           "dspark_q_validate", "dspark_verify_match", "verify_match", "dspark_q_chain_sample",
           "q_chain_sample", "dspark_q_build_sample_sharded", "dspark_q_sharded_workspace_bytes",
           "q_build_sample_sharded", "dspark_spec_step_host",
           "dspark_spec_step_host_staging_bytes", "q_build",
           "draft_sample", "verify_greedy", "verify_ratio", "target_probs", "q_build_sample",
           "spec_step", "version"]


def version() -> str:
    return _lib.load().dspark_version().decode()


def _call(name, *args):
    rc = getattr(_lib.load(), name)(*args)
    if rc != 0:
        raise RuntimeError("%s failed with code %d" % (name, rc))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _dtype_code(t):
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("logits must be float32 or bfloat16, got %s" % t.dtype)


def _rows(t):
    """(rows, V, ld) of a logit tensor whose rows are uniformly strided."""
    if t.dim() < 2 or t.stride(-1) != 1:
        raise ValueError("logit rows must be contiguous in their last dimension")
    V = t.shape[-1]
    ld = t.stride(-2)
    rows = 1
    for i in range(t.dim() - 1):
        rows *= t.shape[i]
    # leading dimensions must be a plain multiple of the row stride
    expect = ld
    for i in range(t.dim() - 2, -1, -1):
        if t.shape[i] > 1 and t.stride(i) != expect:
            raise ValueError("logit rows must be uniformly strided")
        expect *= t.shape[i]
    return rows, V, ld


def _i32(t):
    if t is not None and t.dtype not in (torch.int32, torch.uint32):
        raise TypeError("expected an int32/uint32 tensor")
    return _ptr(t)


# ------------------------------------------------------------ C-named calls
def dspark_q_build(draft_logits, temperature, top_k, counts, sparse_ids, nnz, row_status,
                   stream=None):
    rows, V, ld = _rows(draft_logits)
    _call("dspark_q_build", _ptr(draft_logits), _dtype_code(draft_logits), ld, rows, V,
          _ptr(temperature), int(top_k), _i32(counts), _i32(sparse_ids), _i32(nnz),
          _i32(row_status), _stream(stream))


def dspark_q_build_sample(draft_logits, B, depth, temperature, top_k, seed, request_ids, counts,
                          sparse_ids, nnz, draft_tokens, row_status, stream=None):
    rows, V, ld = _rows(draft_logits)
    if rows != B * depth:
        raise ValueError("draft_logits must hold B*depth rows")
    _call("dspark_q_build_sample", _ptr(draft_logits), _dtype_code(draft_logits), ld, int(B),
          int(depth), V, _ptr(temperature), int(top_k), int(seed) & (2 ** 64 - 1),
          _i32(request_ids), _i32(counts), _i32(sparse_ids), _i32(nnz), _i32(draft_tokens),
          _i32(row_status), _stream(stream))


def dspark_draft_sample(counts, sparse_ids, nnz, top_k, B, depth, V, seed, request_ids,
                        draft_tokens, row_status, stream=None):
    _call("dspark_draft_sample", _i32(counts), _i32(sparse_ids), _i32(nnz), int(top_k), int(B),
          int(depth), int(V), int(seed) & (2 ** 64 - 1), _i32(request_ids), _i32(draft_tokens),
          _i32(row_status), _stream(stream))


def dspark_verify_greedy(target_logits, B, depth, draft_tokens, accept_len, committed,
                         req_status, stream=None):
    rows, V, ld = _rows(target_logits)
    if rows != B * (depth + 1):
        raise ValueError("target_logits must hold B*(depth+1) rows")
    _call("dspark_verify_greedy", _ptr(target_logits), _dtype_code(target_logits), ld, int(B),
          int(depth), V, _i32(draft_tokens), _i32(accept_len), _i32(committed),
          _i32(req_status), _stream(stream))


def dspark_verify_ratio(target_logits, B, depth, draft_tokens, counts, sparse_ids, nnz, top_k,
                        seed, request_ids, accept_len, committed, flags, req_status,
                        stream=None):
    rows, V, ld = _rows(target_logits)
    if rows != B * (depth + 1):
        raise ValueError("target_logits must hold B*(depth+1) rows")
    _call("dspark_verify_ratio", _ptr(target_logits), _dtype_code(target_logits), ld, int(B),
          int(depth), V, _i32(draft_tokens), _i32(counts), _i32(sparse_ids), _i32(nnz),
          int(top_k), int(seed) & (2 ** 64 - 1), _i32(request_ids), _i32(accept_len),
          _i32(committed), _i32(flags), _i32(req_status), _stream(stream))


def dspark_verify(target_logits, B, depth, draft_tokens, greedy_out=None, ratio_out=None,
                  counts=None, sparse_ids=None, nnz=None, top_k=0, seed=0, request_ids=None,
                  stream=None):
    """Both verification modes in one pass.  greedy_out = (accept_len,
    committed, status) or None; ratio_out = (accept_len, committed, flags,
    status) or None, with counts / sparse_ids / nnz / top_k / seed /
    request_ids as in dspark_verify_ratio."""
    rows, V, ld = _rows(target_logits)
    if rows != B * (depth + 1):
        raise ValueError("target_logits must hold B*(depth+1) rows")
    g = greedy_out or (None, None, None)
    r = ratio_out or (None, None, None, None)
    _call("dspark_verify", _ptr(target_logits), _dtype_code(target_logits), ld, int(B),
          int(depth), V, _i32(draft_tokens), _i32(counts), _i32(sparse_ids), _i32(nnz),
          int(top_k), int(seed) & (2 ** 64 - 1), _i32(request_ids), _i32(g[0]), _i32(g[1]),
          _i32(g[2]), _i32(r[0]), _i32(r[1]), _i32(r[2]), _i32(r[3]), _stream(stream))


def dspark_spec_step_noalloc(draft_logits, target_logits, B, depth, temperature, seed,
                             request_ids, counts, draft_tokens, row_status, greedy_out=None,
                             ratio_out=None, stream=None, schedule=0):
    """dspark_spec_step with the library's own device scratch array instead
    of a workspace (calls on one device must not overlap)."""
    rd, V, ld_d = _rows(draft_logits)
    rt, Vt, ld_t = _rows(target_logits)
    if rd != B * depth or rt != B * (depth + 1) or Vt != V:
        raise ValueError("draft_logits must hold B*depth rows and target_logits B*(depth+1) rows "
                         "of the same V")
    g = greedy_out or (None, None, None)
    r = ratio_out or (None, None, None, None)
    _call("dspark_spec_step_noalloc", _ptr(draft_logits), _dtype_code(draft_logits), ld_d,
          _ptr(target_logits), _dtype_code(target_logits), ld_t, int(B), int(depth), V,
          _ptr(temperature), int(seed) & (2 ** 64 - 1), _i32(request_ids), _i32(counts),
          _i32(draft_tokens), _i32(row_status), _i32(g[0]), _i32(g[1]), _i32(g[2]), _i32(r[0]),
          _i32(r[1]), _i32(r[2]), _i32(r[3]), int(schedule), _stream(stream))


def _host(t):
    if t is None:
        return None
    if t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous host tensor")
    return ctypes.c_void_p(t.data_ptr())


def dspark_spec_step_host_staging_bytes(B, depth, V, draft_dtype, target_dtype):
    return int(_lib.load().dspark_spec_step_host_staging_bytes(int(B), int(depth), int(V),
                                                               int(draft_dtype), int(target_dtype)))


def dspark_spec_step_host(draft_logits, target_logits, B, depth, temperature, seed, request_ids,
                          draft_tokens, row_status, staging, greedy_out=None, ratio_out=None,
                          stream=None, schedule=0):
    """dspark_spec_step on host tensors (page-locked for asynchronous copies):
    draft_logits [B*depth, V] and target_logits [B*(depth+1), V] (float32 or
    bfloat16), temperature / request_ids (or None), host outputs; staging is
    a device uint8 tensor of dspark_spec_step_host_staging_bytes bytes."""
    V = draft_logits.shape[-1]
    if (draft_logits.numel() != B * depth * V or target_logits.numel() != B * (depth + 1) * V
            or target_logits.shape[-1] != V):
        raise ValueError("draft_logits must hold B*depth rows and target_logits B*(depth+1) rows "
                         "of the same V")
    g = greedy_out or (None, None, None)
    r = ratio_out or (None, None, None, None)
    _call("dspark_spec_step_host", _host(draft_logits), _dtype_code(draft_logits),
          _host(target_logits), _dtype_code(target_logits), int(B), int(depth), int(V),
          _host(temperature), int(seed) & (2 ** 64 - 1), _host(request_ids), _host(draft_tokens),
          _host(row_status), _host(g[0]), _host(g[1]), _host(g[2]), _host(r[0]), _host(r[1]),
          _host(r[2]), _host(r[3]), _ptr(staging), int(schedule), _stream(stream))


def dspark_spec_step_schedule(B, depth):
    """The schedule dspark_spec_step takes with SCHEDULE_AUTO (host only)."""
    rc = _lib.load().dspark_spec_step_schedule(int(B), int(depth))
    if rc < 0:
        raise ValueError("dspark_spec_step_schedule: error %d" % rc)
    return rc


def dspark_verify_match(target_logits, B, depth, draft_tokens, seed, request_ids, accept_len,
                        committed, flags, req_status, stream=None):
    rows, V, ld = _rows(target_logits)
    if rows != B * (depth + 1):
        raise ValueError("target_logits must hold B*(depth+1) rows")
    _call("dspark_verify_match", _ptr(target_logits), _dtype_code(target_logits), ld, int(B),
          int(depth), V, _i32(draft_tokens), int(seed) & (2 ** 64 - 1), _i32(request_ids),
          _i32(accept_len), _i32(committed), _i32(flags), _i32(req_status), _stream(stream))


def dspark_q_chain_sample(draft_logits, B, depth, temperature, bias, anchors, seed,
                          request_ids, workspace, counts, draft_tokens, row_status, margins=None,
                          stream=None):
    """draft_logits [B*depth, V] (or [B, depth, V]); bias [n_bias, V] fp32 or None;
    anchors int32 [B]; workspace unused (may be None)."""
    rows, V, ld = _rows(draft_logits)
    if rows != B * depth:
        raise ValueError("draft_logits must hold B*depth rows")
    nb, bld = (0, V) if bias is None else (bias.shape[0], bias.stride(0))
    _call("dspark_q_chain_sample", _ptr(draft_logits), _dtype_code(draft_logits), ld, int(B),
          int(depth), V, _ptr(temperature), _ptr(bias), bld, nb, _i32(anchors),
          int(seed) & (2 ** 64 - 1), _i32(request_ids), _ptr(workspace), _i32(counts),
          _i32(draft_tokens), _i32(row_status), _ptr(margins), _stream(stream))


def dspark_q_sharded_workspace_bytes(n_rows):
    return int(_lib.load().dspark_q_sharded_workspace_bytes(int(n_rows)))


def dspark_q_build_sample_sharded(draft_logits, B, depth, n_shards, temperature, top_k, seed,
                                  request_ids, counts, sparse_ids, nnz, draft_tokens, row_status,
                                  workspace, stream=None):
    rows, V, ld = _rows(draft_logits)
    if rows != B * depth:
        raise ValueError("draft_logits must hold B*depth rows")
    _call("dspark_q_build_sample_sharded", _ptr(draft_logits), _dtype_code(draft_logits), ld,
          int(B), int(depth), V, int(n_shards), _ptr(temperature), int(top_k),
          int(seed) & (2 ** 64 - 1), _i32(request_ids), _i32(counts), _i32(sparse_ids), _i32(nnz),
          _i32(draft_tokens), _i32(row_status), _ptr(workspace), _stream(stream))


def dspark_q_pack(counts, sparse_ids, nnz, top_k, V, q_out, checksum_out, stream=None):
    """counts [n_rows, V] (dense) or [n_rows, top_k] with sparse_ids / nnz;
    q_out float32 of the same shape; checksum_out int64 [n_rows] (holding the
    uint64 checksums)."""
    _call("dspark_q_pack", _i32(counts), _i32(sparse_ids), _i32(nnz), int(top_k),
          counts.shape[0], int(V), _ptr(q_out), _ptr(checksum_out), _stream(stream))


def dspark_q_validate(q, sparse_ids, nnz, top_k, V, tokens, expect, counts_out, row_status,
                      stream=None):
    """q float32 [n_rows, width]; tokens int32 [n_rows] or None; expect int64
    [n_rows] or None; counts_out int32 [n_rows, width] or None."""
    n_rows = q.shape[0]
    _call("dspark_q_validate", _ptr(q), _i32(sparse_ids), _i32(nnz), int(top_k), n_rows, int(V),
          _i32(tokens), _ptr(expect), _i32(counts_out), _i32(row_status), _stream(stream))


def dspark_verify_stats(flags, stats, stream=None):
    """flags: int32 / uint32 [B] (device); stats: int32 [3] (device)."""
    _call("dspark_verify_stats", _ptr(flags), int(flags.numel()), _ptr(stats), _stream(stream))


def dspark_target_probs(target_logits, p_out, argmax, row_status, stream=None):
    rows, V, ld = _rows(target_logits)
    _call("dspark_target_probs", _ptr(target_logits), _dtype_code(target_logits), ld, rows, V,
          _ptr(p_out), _i32(argmax), _i32(row_status), _stream(stream))


def dspark_spec_step(draft_logits, target_logits, B, depth, temperature, seed, request_ids, counts,
                     draft_tokens, row_status, greedy_out=None, ratio_out=None, workspace=None,
                     stream=None, schedule=0):
    """greedy_out = (accept_len, committed, status) or None; ratio_out =
    (accept_len, committed, flags, status) or None; workspace: >= B + 1 int32
    (allocated here when None); schedule: SCHEDULE_AUTO, SCHEDULE_ONE_LAUNCH
    or SCHEDULE_SEPARATE."""
    rd, V, ld_d = _rows(draft_logits)
    rt, Vt, ld_t = _rows(target_logits)
    if rd != B * depth or rt != B * (depth + 1) or Vt != V:
        raise ValueError("draft_logits must hold B*depth rows and target_logits B*(depth+1) rows "
                         "of the same V")
    g = greedy_out or (None, None, None)
    r = ratio_out or (None, None, None, None)
    if workspace is None:
        workspace = _empty((B + 1,), torch.int32, draft_logits.device)
    _call("dspark_spec_step", _ptr(draft_logits), _dtype_code(draft_logits), ld_d,
          _ptr(target_logits), _dtype_code(target_logits), ld_t, int(B), int(depth), V,
          _ptr(temperature), int(seed) & (2 ** 64 - 1), _i32(request_ids), _i32(counts),
          _i32(draft_tokens), _i32(row_status), _i32(g[0]), _i32(g[1]), _i32(g[2]), _i32(r[0]),
          _i32(r[1]), _i32(r[2]), _i32(r[3]), _i32(workspace), int(schedule), _stream(stream))


# --------------------------------------------------- allocating helpers
def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


def q_build(draft_logits, temperature=None, top_k=0, stream=None):
    """draft_logits [..., V]; returns dict(counts, ids, nnz, status) (rows flattened)."""
    rows, V, _ = _rows(draft_logits)
    dev = draft_logits.device
    if top_k > 0:
        counts = _empty((rows, top_k), torch.int32, dev)
        ids = _empty((rows, top_k), torch.int32, dev)
        nnz = _empty((rows,), torch.int32, dev)
    else:
        counts = _empty((rows, V), torch.int32, dev)
        ids = nnz = None
    status = _empty((rows,), torch.int32, dev)
    dspark_q_build(draft_logits, temperature, top_k, counts, ids, nnz, status, stream)
    return {"counts": counts, "ids": ids, "nnz": nnz, "status": status, "top_k": top_k}


def q_build_sample(draft_logits, B, depth, seed, temperature=None, top_k=0, request_ids=None,
                   stream=None):
    """Fused q build + draft draw; returns (q dict, tokens [B, depth])."""
    rows, V, _ = _rows(draft_logits)
    dev = draft_logits.device
    if top_k > 0:
        counts = _empty((rows, top_k), torch.int32, dev)
        ids = _empty((rows, top_k), torch.int32, dev)
        nnz = _empty((rows,), torch.int32, dev)
    else:
        counts = _empty((rows, V), torch.int32, dev)
        ids = nnz = None
    status = _empty((rows,), torch.int32, dev)
    tokens = _empty((B, depth), torch.int32, dev)
    dspark_q_build_sample(draft_logits, B, depth, temperature, top_k, seed, request_ids, counts,
                          ids, nnz, tokens, status, stream)
    return {"counts": counts, "ids": ids, "nnz": nnz, "status": status, "top_k": top_k}, tokens


def spec_step(draft_logits, target_logits, B, depth, seed, temperature=None, request_ids=None,
              modes=("greedy", "ratio"), stream=None, schedule=0):
    """Fused q build + draft draw + verification (dense q).  Returns (q dict,
    tokens [B, depth], {mode: outputs as verify_greedy / verify_ratio})."""
    rows, V, _ = _rows(draft_logits)
    dev = draft_logits.device
    counts = _empty((rows, V), torch.int32, dev)
    status = _empty((rows,), torch.int32, dev)
    tokens = _empty((B, depth), torch.int32, dev)
    outs = {}
    if "greedy" in modes:
        outs["greedy"] = (_empty((B,), torch.int32, dev), _empty((B, depth + 1), torch.int32, dev),
                          _empty((B,), torch.int32, dev))
    if "ratio" in modes:
        outs["ratio"] = (_empty((B,), torch.int32, dev), _empty((B, depth + 1), torch.int32, dev),
                         _empty((B,), torch.int32, dev), _empty((B,), torch.int32, dev))
    dspark_spec_step(draft_logits, target_logits, B, depth, temperature, seed, request_ids, counts,
                     tokens, status, outs.get("greedy"), outs.get("ratio"), stream=stream,
                     schedule=schedule)
    q = {"counts": counts, "ids": None, "nnz": None, "status": status, "top_k": 0}
    return q, tokens, outs


def verify_match(target_logits, draft_tokens, seed, request_ids=None, stream=None):
    """Stochastic verification; returns (accept_len, committed, flags, status)."""
    B, depth = draft_tokens.shape
    dev = target_logits.device
    acc = _empty((B,), torch.int32, dev)
    com = _empty((B, depth + 1), torch.int32, dev)
    fl = _empty((B,), torch.int32, dev)
    st = _empty((B,), torch.int32, dev)
    dspark_verify_match(target_logits, B, depth, draft_tokens, seed, request_ids, acc, com, fl, st,
                        stream)
    return acc, com, fl, st


def q_chain_sample(draft_logits, B, depth, seed, anchors, bias=None, temperature=None,
                   request_ids=None, stream=None):
    """The Markov-conditioned draft chain; returns (q dict, tokens [B, depth],
    margins [B, depth])."""
    rows, V, _ = _rows(draft_logits)
    dev = draft_logits.device
    counts = _empty((rows, V), torch.int32, dev)
    status = _empty((rows,), torch.int32, dev)
    tokens = _empty((B, depth), torch.int32, dev)
    margins = _empty((B, depth), torch.float32, dev)
    dspark_q_chain_sample(draft_logits, B, depth, temperature, bias, anchors, seed, request_ids,
                          None, counts, tokens, status, margins, stream)
    q = {"counts": counts, "ids": None, "nnz": None, "status": status, "top_k": 0}
    return q, tokens, margins


def q_build_sample_sharded(draft_logits, B, depth, n_shards, seed, temperature=None, top_k=0,
                           request_ids=None, stream=None):
    """The vocabulary-sharded emulation of q_build_sample."""
    rows, V, _ = _rows(draft_logits)
    dev = draft_logits.device
    ws = _empty((dspark_q_sharded_workspace_bytes(rows),), torch.uint8, dev)
    if top_k > 0:
        counts = _empty((rows, top_k), torch.int32, dev)
        ids = _empty((rows, top_k), torch.int32, dev)
        nnz = _empty((rows,), torch.int32, dev)
    else:
        counts = _empty((rows, V), torch.int32, dev)
        ids = nnz = None
    status = _empty((rows,), torch.int32, dev)
    tokens = _empty((B, depth), torch.int32, dev)
    dspark_q_build_sample_sharded(draft_logits, B, depth, n_shards, temperature, top_k, seed,
                                  request_ids, counts, ids, nnz, tokens, status, ws, stream)
    return {"counts": counts, "ids": ids, "nnz": nnz, "status": status, "top_k": top_k}, tokens


def q_pack(q, V, stream=None):
    """Wire form of a q dict from q_build: (q float32 of the counts' shape,
    checksums int64 [n_rows] holding the uint64 bit patterns)."""
    counts = q["counts"]
    qf = _empty(counts.shape, torch.float32, counts.device)
    cs = _empty((counts.shape[0],), torch.int64, counts.device)
    dspark_q_pack(counts, q["ids"], q["nnz"], q["top_k"], V, qf, cs, stream)
    return qf, cs


def q_validate(qf, V, ids=None, nnz=None, top_k=0, tokens=None, expect=None, stream=None):
    """Validation of received q rows: (status int32 [n_rows], recovered counts
    int32 of qf's shape)."""
    counts = _empty(qf.shape, torch.int32, qf.device)
    st = _empty((qf.shape[0],), torch.int32, qf.device)
    dspark_q_validate(qf, ids, nnz, top_k, V, tokens, expect, counts, st, stream)
    return st, counts


def draft_sample(q, B, depth, V, seed, request_ids=None, stream=None):
    dev = q["counts"].device
    tokens = _empty((B * depth,), torch.int32, dev)
    status = _empty((B * depth,), torch.int32, dev)
    dspark_draft_sample(q["counts"], q["ids"], q["nnz"], q["top_k"], B, depth, V, seed,
                        request_ids, tokens, status, stream)
    return tokens.view(B, depth), status.view(B, depth)


def verify_greedy(target_logits, drafts, stream=None):
    B, depth = drafts.shape
    dev = target_logits.device
    acc = _empty((B,), torch.int32, dev)
    com = _empty((B, depth + 1), torch.int32, dev)
    st = _empty((B,), torch.int32, dev)
    dspark_verify_greedy(target_logits, B, depth, drafts, acc, com, st, stream)
    return acc, com, st


def verify_ratio(target_logits, drafts, q, seed, request_ids=None, stream=None):
    B, depth = drafts.shape
    dev = target_logits.device
    acc = _empty((B,), torch.int32, dev)
    com = _empty((B, depth + 1), torch.int32, dev)
    fl = _empty((B,), torch.int32, dev)
    st = _empty((B,), torch.int32, dev)
    dspark_verify_ratio(target_logits, B, depth, drafts, q["counts"], q["ids"], q["nnz"],
                        q["top_k"], seed, request_ids, acc, com, fl, st, stream)
    return acc, com, fl, st


def verify_stats(flags, stream=None):
    """Counts of the requests with each DSPARK_FLAG_* bit in flags [B]: a
    tensor [3] (ambiguous decisions, draws near a boundary, degenerate
    residuals)."""
    stats = _empty((3,), torch.int32, flags.device)
    dspark_verify_stats(flags, stats, stream)
    return stats


def target_probs(target_logits, want_p=True, stream=None):
    rows, V, _ = _rows(target_logits)
    dev = target_logits.device
    p = _empty((rows, V), torch.float32, dev) if want_p else None
    am = _empty((rows,), torch.int32, dev)
    st = _empty((rows,), torch.int32, dev)
    dspark_target_probs(target_logits, p, am, st, stream)
    return p, am, st
