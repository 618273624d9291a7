"""ctypes front end of the CPU oracle (``dspark_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg, never by the library.  ``build()`` compiles the
C file with gcc into ``oracle/_build/liboracle.so``; every function here only
marshals numpy arrays into the C calls (no arithmetic of the method lives in
this file).  bf16 inputs are widened to fp32 by the caller before they get
here (a bit shift, exact).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

M = 1 << 24
OK, NONFINITE, ZERO_MASS, ALLOC_INCONSISTENT, BAD_TEMPERATURE, BAD_Q, BAD_DRAFT = range(7)
BAD_CHECKSUM = 9
FLAG_AMBIG_ACCEPT, FLAG_NEAR_BOUNDARY, FLAG_DEGENERATE, FLAG_NEAR_BOUNDARY_REL = 1, 2, 4, 8
PURPOSE_PROPOSAL, PURPOSE_ACCEPT, PURPOSE_RESIDUAL, PURPOSE_BONUS, PURPOSE_MATCH = 0, 1, 2, 3, 4

_P = ctypes.c_void_p
_I32, _I64, _U32, _U64, _F32, _F64 = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                      ctypes.c_uint64, ctypes.c_float, ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE: no fast-math, no fp contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".%d.tmp" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            so = build()
            L = ctypes.CDLL(so)
            sig = {
                "oracle_philox4x32_10": (None, [_P, _P, _P]),
                "oracle_draw_u32": (_U32, [_U64, _U32, _U32, _U32]),
                "oracle_exp_ds": (_F32, [_F32]),
                "oracle_exp_ds_array": (None, [_P, _P, _I64]),
                "oracle_q_weights_row": (ctypes.c_int, [_P, _I32, _F32, _I32, _P, _P, _P]),
                "oracle_q_allocate_row": (ctypes.c_int, [_P, _P, _I32, _P]),
                "oracle_q_build_row": (ctypes.c_int, [_P, _I32, _F32, _I32, _P, _P, _P]),
                "oracle_q_build": (None, [_P, _I64, _I32, _I32, _P, _I32, _P, _P, _P, _P]),
                "oracle_categorical_pick": (_I32, [_P, _P, _I32, _U32]),
                "oracle_categorical_pick_many": (None, [_P, _P, _I32, _P, _I64, _P]),
                "oracle_draft_sample_row": (_I32, [_P, _P, _I32, _I32, _U64, _U32, _U32, _P]),
                "oracle_target_row": (ctypes.c_int, [_P, _I32, _P, _P]),
                "oracle_target_probs": (None, [_P, _I64, _I32, _I32, _P, _P, _P]),
                "oracle_ratio_accept": (ctypes.c_int, [_U32, _U32, _F64]),
                "oracle_ratio_accept_many": (None, [_P, _I64, _U32, _F64, _P]),
                "oracle_residual_pick": (_I32, [_P, _P, _I32, _U32, _P]),
                "oracle_verify_greedy_req": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _P, _P]),
                "oracle_verify_ratio_req": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _P, _P, _P,
                                                           _I32, _U64, _U32, _P, _P, _P]),
                "oracle_verify_match_req": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _U64, _U32,
                                                           _P, _P, _P]),
                "oracle_q_chain_request": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _P, _I64, _I32,
                                                          _I32, _U64, _U32, _P, _P, _P, _P]),
                "oracle_q_build_row_sharded": (ctypes.c_int, [_P, _I32, _F32, _I32, _I32, _P]),
                "oracle_draw_sharded": (_I32, [_P, _I32, _I32, _U32]),
                "oracle_verify_ratio_req_sharded": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _P,
                                                                   _I32, _U64, _U32, _P, _P, _P]),
                "oracle_fletcher64": (_U64, [_P, _I64]),
                "oracle_q_pack_row": (_U64, [_P, _P, _I32, _I32, _I32, _P]),
                "oracle_q_validate_row": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, ctypes.c_int,
                                                         _I32, ctypes.c_int, _U64, _P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- Philox / exp
def philox4x32_10(ctr, key):
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def draw_u32(seed: int, request: int, row: int, purpose: int) -> int:
    return int(lib().oracle_draw_u32(seed, request, row, purpose))


def exp_ds(d: np.ndarray) -> np.ndarray:
    d = _c(d, np.float32)
    out = np.empty_like(d)
    lib().oracle_exp_ds_array(_ptr(d), _ptr(out), d.size)
    return out


# ----------------------------------------------------------------- q building
def q_weights_row(x, T=1.0, top_k=0):
    x = _c(x, np.float32)
    V = x.size
    E = np.zeros(V, np.uint64)
    sup = np.zeros(V, np.uint8)
    S = np.zeros(1, np.uint64)
    st = lib().oracle_q_weights_row(_ptr(x), V, T, top_k, _ptr(E), _ptr(sup), _ptr(S))
    return st, E, sup.astype(bool), int(S[0])


def q_allocate_row(E, support):
    E = _c(E, np.uint64)
    sup = _c(support, np.uint8)
    counts = np.zeros(E.size, np.uint32)
    st = lib().oracle_q_allocate_row(_ptr(E), _ptr(sup), E.size, _ptr(counts))
    return st, counts


def q_build(x, temperature=None, top_k=0):
    """x: [n_rows, V] fp32.  Returns (counts, ids, nnz, status); dense: ids/nnz None."""
    x = _c(x, np.float32)
    n_rows, V = x.shape
    t = None if temperature is None else _c(np.broadcast_to(temperature, (n_rows,)), np.float32)
    status = np.zeros(n_rows, np.int32)
    if top_k > 0:
        counts = np.zeros((n_rows, top_k), np.uint32)
        ids = np.zeros((n_rows, top_k), np.int32)
        nnz = np.zeros(n_rows, np.int32)
    else:
        counts = np.zeros((n_rows, V), np.uint32)
        ids = nnz = None
    lib().oracle_q_build(_ptr(x), V, n_rows, V, _ptr(t), top_k, _ptr(counts), _ptr(ids),
                         _ptr(nnz), _ptr(status))
    return counts, ids, nnz, status


# ------------------------------------------------------------------- sampling
def categorical_pick_many(counts, D, ids=None):
    counts = _c(counts, np.uint32)
    ids = None if ids is None else _c(ids, np.int32)
    D = _c(D, np.uint32)
    out = np.empty(D.size, np.int32)
    lib().oracle_categorical_pick_many(_ptr(counts), _ptr(ids), counts.size, _ptr(D), D.size,
                                       _ptr(out))
    return out


def draft_sample(counts, ids, nnz, top_k, B, depth, seed, request_ids=None, V=None):
    """counts: dense [B*depth, V] or sparse [B*depth, top_k] (then V is needed)."""
    counts = _c(counts, np.uint32)
    if top_k == 0:
        V = counts.shape[1]
    n_rows = B * depth
    req = np.arange(B, dtype=np.uint32) if request_ids is None else _c(request_ids, np.uint32)
    tokens = np.full(n_rows, -1, np.int32)
    status = np.zeros(n_rows, np.int32)
    st = ctypes.c_int32(0)
    L = lib()
    for r in range(n_rows):
        b, j = divmod(r, depth)
        if top_k > 0:
            n = int(nnz[r])
            if n < 1 or n > top_k:
                tokens[r], status[r] = -1, BAD_Q
                continue
            c = _c(counts[r, :n], np.uint32)
            i = _c(ids[r, :n], np.int32)
            tok = L.oracle_draft_sample_row(_ptr(c), _ptr(i), n, V, seed, int(req[b]), j,
                                            ctypes.byref(st))
        else:
            c = _c(counts[r], np.uint32)
            tok = L.oracle_draft_sample_row(_ptr(c), None, c.size, V, seed, int(req[b]), j,
                                            ctypes.byref(st))
        tokens[r] = tok
        status[r] = st.value
    return tokens, status


# ------------------------------------------------------------------- target p
def target_probs(z, want_p=True):
    """z: [n_rows, V] fp32.  Returns (p float64 or None, argmax, status)."""
    z = _c(z, np.float32)
    n_rows, V = z.shape
    p = np.zeros((n_rows, V), np.float64) if want_p else None
    am = np.zeros(n_rows, np.int32)
    status = np.zeros(n_rows, np.int32)
    lib().oracle_target_probs(_ptr(z), V, n_rows, V, _ptr(p), _ptr(am), _ptr(status))
    return p, am, status


def ratio_accept_many(U, c, p):
    U = _c(U, np.uint32)
    out = np.zeros(U.size, np.uint8)
    lib().oracle_ratio_accept_many(_ptr(U), U.size, int(c), float(p), _ptr(out))
    return out.astype(bool)


def residual_pick(p, c, w):
    p = _c(p, np.float64)
    c = None if c is None else _c(c, np.uint32)
    fl = ctypes.c_uint32(0)
    tok = lib().oracle_residual_pick(_ptr(p), _ptr(c), p.size, int(w), ctypes.byref(fl))
    return int(tok), int(fl.value)


# ------------------------------------------------------------------ verifiers
def verify_greedy(z, drafts):
    """z: [B, depth+1, V] fp32; drafts: [B, depth] int32."""
    z = _c(z, np.float32)
    drafts = _c(drafts, np.int32)
    B, rows, V = z.shape
    depth = rows - 1
    acc = np.zeros(B, np.int32)
    com = np.full((B, depth + 1), -1, np.int32)
    status = np.zeros(B, np.int32)
    a = ctypes.c_int32(0)
    L = lib()
    for b in range(B):
        cm = np.zeros(depth + 1, np.int32)
        status[b] = L.oracle_verify_greedy_req(_ptr(z[b]), V, V, depth, _ptr(drafts[b]),
                                               ctypes.byref(a), _ptr(cm))
        acc[b] = a.value
        com[b] = cm
    return acc, com, status


def verify_ratio(z, drafts, counts, ids, nnz, top_k, seed, request_ids=None):
    """z: [B, depth+1, V] fp32; drafts [B, depth]; counts dense [B*depth, V] or
    sparse [B*depth, top_k] with ids [B*depth, top_k] and nnz [B*depth]."""
    z = _c(z, np.float32)
    drafts = _c(drafts, np.int32)
    counts = _c(counts, np.uint32)
    B, rows, V = z.shape
    depth = rows - 1
    if top_k > 0:
        ids = _c(ids, np.int32)
        nnz = _c(nnz, np.int32)
    req = np.arange(B, dtype=np.uint32) if request_ids is None else _c(request_ids, np.uint32)
    acc = np.zeros(B, np.int32)
    com = np.full((B, depth + 1), -1, np.int32)
    flags = np.zeros(B, np.uint32)
    status = np.zeros(B, np.int32)
    a = ctypes.c_int32(0)
    fl = ctypes.c_uint32(0)
    L = lib()
    per = V if top_k == 0 else top_k
    for b in range(B):
        cm = np.zeros(depth + 1, np.int32)
        cb = counts.reshape(B, depth, per)[b]
        ib = None if top_k == 0 else ids.reshape(B, depth, top_k)[b]
        nb = None if top_k == 0 else nnz.reshape(B, depth)[b]
        status[b] = L.oracle_verify_ratio_req(_ptr(z[b]), V, V, depth, _ptr(drafts[b]), _ptr(cb),
                                              _ptr(ib), _ptr(nb), top_k, seed, int(req[b]),
                                              ctypes.byref(a), _ptr(cm), ctypes.byref(fl))
        acc[b] = a.value
        com[b] = cm
        flags[b] = fl.value
    return acc, com, flags, status


# ------------------------------------------------------------ received q (wire)
def fletcher64(words) -> int:
    """Fletcher-64 of 32-bit words (A, B modulo 2^32 - 1; B << 32 | A)."""
    w = _c(words, np.uint32)
    return int(lib().oracle_fletcher64(_ptr(w), w.size))


def q_pack(counts, ids=None, nnz=None, top_k=0):
    """counts [n_rows, V] (dense) or [n_rows, top_k] with ids / nnz (sparse).
    Returns (q fp32 of the same shape, checksum uint64 [n_rows])."""
    counts = _c(counts, np.uint32)
    n_rows = counts.shape[0]
    q = np.zeros(counts.shape, np.float32)
    cs = np.zeros(n_rows, np.uint64)
    V = counts.shape[1]
    for r in range(n_rows):
        ir = None if ids is None else _c(ids[r], np.int32)
        nz = 0 if nnz is None else int(nnz[r])
        qr = np.zeros(V, np.float32)
        cs[r] = lib().oracle_q_pack_row(_ptr(counts[r]), _ptr(ir), nz, top_k, V, _ptr(qr))
        q[r] = qr
    return q, cs


def q_validate(q, ids=None, nnz=None, top_k=0, V=None, tokens=None, expect=None):
    """Validation of received q rows.  Returns (status int32 [n_rows],
    recovered counts uint32 of q's shape)."""
    q = _c(q, np.float32)
    n_rows, width = q.shape
    V = width if V is None else V
    st = np.zeros(n_rows, np.int32)
    counts = np.zeros(q.shape, np.uint32)
    for r in range(n_rows):
        ir = None if ids is None else _c(ids[r], np.int32)
        nz = 0 if nnz is None else int(nnz[r])
        has_tok = tokens is not None
        tok = int(tokens[r]) if has_tok else 0
        has = expect is not None
        ex = int(expect[r]) if has else 0
        cr = np.zeros(width, np.uint32)
        st[r] = lib().oracle_q_validate_row(_ptr(q[r]), _ptr(ir), nz, top_k, V, int(has_tok), tok,
                                            int(has), ex, _ptr(cr))
        counts[r] = cr
    return st, counts


# ------------------------------------------------------- stochastic (match)
def verify_match(z, drafts, seed, request_ids=None):
    """z: [B, depth+1, V] fp32; drafts [B, depth].  Returns (accept_len,
    committed, flags, status)."""
    z = _c(z, np.float32)
    drafts = _c(drafts, np.int32)
    B, rows, V = z.shape
    depth = rows - 1
    req = np.arange(B, dtype=np.uint32) if request_ids is None else _c(request_ids, np.uint32)
    acc = np.zeros(B, np.int32)
    com = np.full((B, depth + 1), -1, np.int32)
    flags = np.zeros(B, np.uint32)
    status = np.zeros(B, np.int32)
    a = ctypes.c_int32(0)
    fl = ctypes.c_uint32(0)
    for b in range(B):
        cm = np.zeros(depth + 1, np.int32)
        status[b] = lib().oracle_verify_match_req(_ptr(z[b]), V, V, depth, _ptr(drafts[b]), seed,
                                                  int(req[b]), ctypes.byref(a), _ptr(cm),
                                                  ctypes.byref(fl))
        acc[b] = a.value
        com[b] = cm
        flags[b] = fl.value
    return acc, com, flags, status


# ------------------------------------------------------ Markov draft chain
def q_chain(x, temperature, bias, anchors, seed, request_ids=None):
    """x: [B, depth, V] fp32 base logits; temperature [B*depth] or None; bias
    [n_bias, V] fp32 or None; anchors [B].  Returns (counts [B*depth, V],
    tokens [B, depth], status [B*depth], margins [B, depth])."""
    x = _c(x, np.float32)
    B, depth, V = x.shape
    t = None if temperature is None else _c(temperature, np.float32).reshape(B, depth)
    b = None if bias is None else _c(bias, np.float32)
    nb = 1 if b is None else b.shape[0]
    req = np.arange(B, dtype=np.uint32) if request_ids is None else _c(request_ids, np.uint32)
    counts = np.zeros((B, depth, V), np.uint32)
    tokens = np.zeros((B, depth), np.int32)
    status = np.zeros((B, depth), np.int32)
    margins = np.zeros((B, depth), np.float32)
    for r in range(B):
        tr = None if t is None else _c(t[r], np.float32)
        lib().oracle_q_chain_request(_ptr(x[r]), V, V, depth, _ptr(tr), _ptr(b), V, nb,
                                     int(anchors[r]), seed, int(req[r]), _ptr(counts[r]),
                                     _ptr(tokens[r]), _ptr(status[r]), _ptr(margins[r]))
    return counts.reshape(B * depth, V), tokens, status.reshape(-1), margins


# ------------------------------------------------- vocabulary-sharded emulator
def q_build_sharded(x, n_shards, temperature=None, top_k=0):
    """Dense counts [n_rows, V] and status from the sharded emulator."""
    x = _c(x, np.float32)
    n_rows, V = x.shape
    t = np.ones(n_rows, np.float32) if temperature is None else _c(
        np.broadcast_to(temperature, (n_rows,)), np.float32)
    counts = np.zeros((n_rows, V), np.uint32)
    st = np.zeros(n_rows, np.int32)
    for r in range(n_rows):
        cr = np.zeros(V, np.uint32)
        st[r] = lib().oracle_q_build_row_sharded(_ptr(x[r]), V, float(t[r]), top_k, n_shards,
                                                 _ptr(cr))
        counts[r] = cr
    return counts, st


def draw_sharded(counts_row, n_shards, D):
    c = _c(counts_row, np.uint32)
    return int(lib().oracle_draw_sharded(_ptr(c), c.size, n_shards, int(D)))


def verify_ratio_sharded(z, drafts, counts, n_shards, seed, request_ids=None):
    z = _c(z, np.float32)
    drafts = _c(drafts, np.int32)
    counts = _c(counts, np.uint32)
    B, rows, V = z.shape
    depth = rows - 1
    req = np.arange(B, dtype=np.uint32) if request_ids is None else _c(request_ids, np.uint32)
    acc = np.zeros(B, np.int32)
    com = np.full((B, depth + 1), -1, np.int32)
    flags = np.zeros(B, np.uint32)
    status = np.zeros(B, np.int32)
    a = ctypes.c_int32(0)
    fl = ctypes.c_uint32(0)
    for b in range(B):
        cm = np.zeros(depth + 1, np.int32)
        cb = counts.reshape(B, depth, V)[b]
        status[b] = lib().oracle_verify_ratio_req_sharded(_ptr(z[b]), V, V, depth, _ptr(drafts[b]),
                                                          _ptr(cb), n_shards, seed, int(req[b]),
                                                          ctypes.byref(a), _ptr(cm),
                                                          ctypes.byref(fl))
        acc[b] = a.value
        com[b] = cm
        flags[b] = fl.value
    return acc, com, flags, status
