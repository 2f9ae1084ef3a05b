"""ctypes front end of the CPU oracle (oracle/ss_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code
with the CUDA package: the two meet only through the seeded workload
dictionaries built by ``speculative_verification_gb300.workloads``.

A workload dictionary holds numpy arrays named like the C structs' fields.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None

OR_DTYPE = {"f32": 0, "bf16": 1}


class _Params(C.Structure):
    _fields_ = [
        ("temperature", C.c_void_p),
        ("top_k", C.c_void_p),
        ("top_p", C.c_void_p),
        ("min_p", C.c_void_p),
        ("repetition", C.c_void_p),
        ("frequency", C.c_void_p),
        ("presence", C.c_void_p),
        ("hist_offsets", C.c_void_p),
        ("hist_ids", C.c_void_p),
        ("bias_offsets", C.c_void_p),
        ("bias_ids", C.c_void_p),
        ("bias_vals", C.c_void_p),
        ("bitmask", C.c_void_p),
        ("bitmask_stride", C.c_int64),
        ("use_bitmask", C.c_void_p),
        ("seed", C.c_void_p),
        ("position", C.c_void_p),
        ("row_id", C.c_void_p),
    ]


class _SampleIn(C.Structure):
    _fields_ = [
        ("num_rows", C.c_int32),
        ("vocab", C.c_int32),
        ("row_stride", C.c_int64),
        ("dtype", C.c_int32),
        ("logits", C.c_void_p),
        ("p", _Params),
        ("force_kept", C.c_void_p),
    ]


class _SampleOut(C.Structure):
    _fields_ = [
        ("token", C.c_void_p),
        ("status", C.c_void_p),
        ("kept", C.c_void_p),
        ("processed", C.c_void_p),
        ("sub_margin", C.c_void_p),
        ("kept_lo", C.c_void_p),
        ("kept_hi", C.c_void_p),
        ("kept_own", C.c_void_p),
    ]


class _VerifyIn(C.Structure):
    _fields_ = [
        ("num_requests", C.c_int32),
        ("vocab", C.c_int32),
        ("max_draft", C.c_int32),
        ("row_stride", C.c_int64),
        ("dtype", C.c_int32),
        ("target_logits", C.c_void_p),
        ("draft_offsets", C.c_void_p),
        ("draft_tokens", C.c_void_p),
        ("draft_probs", C.c_void_p),
        ("draft_stride", C.c_int64),
        ("p", _Params),
        ("force_kept", C.c_void_p),
    ]


class _VerifyOut(C.Structure):
    _fields_ = [
        ("out_tokens", C.c_void_p),
        ("num_accepted", C.c_void_p),
        ("status", C.c_void_p),
        ("kept", C.c_void_p),
        ("processed", C.c_void_p),
        ("sub_margin", C.c_void_p),
        ("kept_lo", C.c_void_p),
        ("kept_hi", C.c_void_p),
        ("kept_own", C.c_void_p),
    ]


class _TreeIn(C.Structure):
    _fields_ = [
        ("num_requests", C.c_int32),
        ("vocab", C.c_int32),
        ("max_nodes", C.c_int32),
        ("row_stride", C.c_int64),
        ("dtype", C.c_int32),
        ("target_logits", C.c_void_p),
        ("node_offsets", C.c_void_p),
        ("parents", C.c_void_p),
        ("node_tokens", C.c_void_p),
        ("draft_probs", C.c_void_p),
        ("draft_stride", C.c_int64),
        ("p", _Params),
    ]


class _TreeOut(C.Structure):
    _fields_ = [
        ("out_tokens", C.c_void_p),
        ("out_path", C.c_void_p),
        ("num_accepted", C.c_void_p),
        ("status", C.c_void_p),
        ("sub_margin", C.c_void_p),
    ]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        L.or_philox4x32_10.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p]
        L.or_philox4x32_10.restype = None
        L.or_uniform.argtypes = [C.c_uint64, C.c_int32, C.c_uint32, C.c_int32, C.c_uint32]
        L.or_uniform.restype = C.c_float
        L.or_gumbel.argtypes = [C.c_uint64, C.c_int32, C.c_uint32, C.c_int32, C.c_uint32]
        L.or_gumbel.restype = C.c_double
        L.or_gumbel_row.argtypes = [C.c_uint64, C.c_int32, C.c_uint32, C.c_uint32, C.c_int32, C.c_void_p]
        L.or_gumbel_row.restype = None
        L.or_process_sample.argtypes = [C.POINTER(_SampleIn), C.POINTER(_SampleOut)]
        L.or_process_sample.restype = C.c_int
        L.or_spec_verify.argtypes = [C.POINTER(_VerifyIn), C.POINTER(_VerifyOut)]
        L.or_spec_verify.restype = C.c_int
        L.or_row_probs.argtypes = [C.POINTER(_SampleIn), C.c_int32, C.c_void_p, C.c_int32, C.c_void_p]
        L.or_row_probs.restype = C.c_int32
        L.or_residual_probs.argtypes = [C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]
        L.or_residual_probs.restype = C.c_int32
        L.or_commit_accepted.argtypes = [C.c_int32, C.c_int32] + [C.c_void_p] * 4 + [C.c_int32] + [C.c_void_p] * 4
        L.or_commit_accepted.restype = None
        L.or_tree_verify.argtypes = [C.POINTER(_TreeIn), C.POINTER(_TreeOut)]
        L.or_tree_verify.restype = C.c_int
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


def _params(w, keep):
    """Build the parameter struct; `keep` collects the arrays it points to."""
    fields = {
        "temperature": np.float32,
        "top_k": np.int32,
        "top_p": np.float32,
        "min_p": np.float32,
        "repetition": np.float32,
        "frequency": np.float32,
        "presence": np.float32,
        "hist_offsets": np.int32,
        "hist_ids": np.int32,
        "bias_offsets": np.int32,
        "bias_ids": np.int32,
        "bias_vals": np.float32,
        "bitmask": np.int32,
        "use_bitmask": np.uint8,
        "seed": np.uint64,
        "position": np.int64,
        "row_id": np.uint32,
    }
    p = _Params()
    for name, dt in fields.items():
        a = _c(w.get(name), dt)
        keep.append(a)
        setattr(p, name, _ptr(a))
    p.bitmask_stride = int(w.get("bitmask_stride", 0) or 0)
    return p


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    o = np.zeros(4, dtype=np.uint32)
    lib().or_philox4x32_10(c.ctypes.data, k.ctypes.data, o.ctypes.data)
    return o


def uniform(seed, row, position, token, stream):
    return float(lib().or_uniform(seed, row, position, token, stream))


def gumbel(seed, row, position, token, stream):
    return float(lib().or_gumbel(seed, row, position, token, stream))


def gumbel_row(seed, row, position, vocab, stream=0):
    """The Gumbel noise of every token of one row (fp64), stream 0 = the draw."""
    out = np.zeros(int(vocab), np.float64)
    lib().or_gumbel_row(seed, row, position, stream, int(vocab), out.ctypes.data)
    return out


def _sample_in(w, keep, force_kept=None):
    logits = np.ascontiguousarray(w["logits"])
    fk = _c(force_kept, np.int32)
    keep += [logits, fk]
    s = _SampleIn()
    s.force_kept = _ptr(fk)
    s.num_rows = int(w["num_rows"])
    s.vocab = int(w["vocab"])
    s.row_stride = int(w["row_stride"])
    s.dtype = OR_DTYPE[w["dtype"]]
    s.logits = logits.ctypes.data
    s.p = _params(w, keep)
    return s


def process_sample(w, want_processed=False, force_kept=None):
    """Run the oracle on a sampling workload; returns a dict of numpy arrays.

    `force_kept` (optional, per row): a kept-set size to draw from when it lies
    inside the oracle's margin range [kept_lo, kept_hi] (see ss_oracle.h)."""
    keep = []
    s = _sample_in(w, keep, force_kept)
    n, V = s.num_rows, s.vocab
    res = {
        "token": np.zeros(n, np.int32),
        "status": np.zeros(n, np.int32),
        "kept": np.zeros(n, np.int32),
        "sub_margin": np.zeros(n, np.uint8),
        "kept_lo": np.zeros(n, np.int32),
        "kept_hi": np.zeros(n, np.int32),
        "kept_own": np.zeros(n, np.int32),
    }
    if want_processed:
        res["processed"] = np.zeros((n, V), np.float32)
    o = _SampleOut()
    o.token = _ptr(res["token"])
    o.status = _ptr(res["status"])
    o.kept = _ptr(res["kept"])
    o.processed = _ptr(res.get("processed"))
    o.sub_margin = _ptr(res["sub_margin"])
    o.kept_lo = _ptr(res["kept_lo"])
    o.kept_hi = _ptr(res["kept_hi"])
    o.kept_own = _ptr(res["kept_own"])
    lib().or_process_sample(C.byref(s), C.byref(o))
    return res


def spec_verify(w, want_processed=False, force_kept=None):
    """Run the oracle on a verification workload; returns a dict of numpy arrays.

    `force_kept` (optional, per target row) as in `process_sample`."""
    keep = []
    fk = _c(force_kept, np.int32)
    keep.append(fk)
    tl = np.ascontiguousarray(w["target_logits"])
    dof = _c(w["draft_offsets"], np.int32)
    dtk = _c(w["draft_tokens"], np.int32)
    dpr = _c(w["draft_probs"], np.float32)
    keep += [tl, dof, dtk, dpr]
    v = _VerifyIn()
    v.num_requests = int(w["num_requests"])
    v.vocab = int(w["vocab"])
    v.max_draft = int(w["max_draft"])
    v.row_stride = int(w["row_stride"])
    v.dtype = OR_DTYPE[w["dtype"]]
    v.target_logits = tl.ctypes.data
    v.draft_offsets = dof.ctypes.data
    v.draft_tokens = dtk.ctypes.data if dtk.size else None
    v.draft_probs = dpr.ctypes.data if dpr.size else None
    v.draft_stride = int(w["draft_stride"])
    v.p = _params(w, keep)
    v.force_kept = _ptr(fk)
    R, V, width = v.num_requests, v.vocab, v.max_draft + 1
    rows = int(dof[-1]) + R
    res = {
        "out_tokens": np.full((R, width), -1, np.int32),
        "num_accepted": np.zeros(R, np.int32),
        "status": np.zeros(R, np.int32),
        "kept": np.zeros(rows, np.int32),
        "sub_margin": np.zeros(R, np.uint8),
        "kept_lo": np.zeros(rows, np.int32),
        "kept_hi": np.zeros(rows, np.int32),
        "kept_own": np.zeros(rows, np.int32),
    }
    if want_processed:
        res["processed"] = np.zeros((rows, V), np.float32)
    o = _VerifyOut()
    o.out_tokens = _ptr(res["out_tokens"])
    o.num_accepted = _ptr(res["num_accepted"])
    o.status = _ptr(res["status"])
    o.kept = _ptr(res["kept"])
    o.processed = _ptr(res.get("processed"))
    o.sub_margin = _ptr(res["sub_margin"])
    o.kept_lo = _ptr(res["kept_lo"])
    o.kept_hi = _ptr(res["kept_hi"])
    o.kept_own = _ptr(res["kept_own"])
    lib().or_spec_verify(C.byref(v), C.byref(o))
    return res


def tree_verify(w):
    """Run the oracle on a tree-verification workload (kind 'tree'); returns a
    dict of numpy arrays: out_tokens and out_path [R, max_nodes],
    num_accepted, status, sub_margin [R]."""
    keep = []
    tl = np.ascontiguousarray(w["target_logits"])
    nof = _c(w["node_offsets"], np.int32)
    par = _c(w["parents"], np.int32)
    ntk = _c(w["node_tokens"], np.int32)
    dpr = _c(w["draft_probs"], np.float32)
    keep += [tl, nof, par, ntk, dpr]
    v = _TreeIn()
    v.num_requests = int(w["num_requests"])
    v.vocab = int(w["vocab"])
    v.max_nodes = int(w["max_nodes"])
    v.row_stride = int(w["row_stride"])
    v.dtype = OR_DTYPE[w["dtype"]]
    v.target_logits = tl.ctypes.data
    v.node_offsets = nof.ctypes.data
    v.parents = par.ctypes.data if par.size else None
    v.node_tokens = ntk.ctypes.data if ntk.size else None
    v.draft_probs = dpr.ctypes.data if dpr.size else None
    v.draft_stride = int(w["draft_stride"])
    v.p = _params(w, keep)
    R, width = v.num_requests, v.max_nodes
    res = {
        "out_tokens": np.full((R, width), -1, np.int32),
        "out_path": np.full((R, width), -1, np.int32),
        "num_accepted": np.zeros(R, np.int32),
        "status": np.zeros(R, np.int32),
        "sub_margin": np.zeros(R, np.uint8),
    }
    o = _TreeOut()
    o.out_tokens = _ptr(res["out_tokens"])
    o.out_path = _ptr(res["out_path"])
    o.num_accepted = _ptr(res["num_accepted"])
    o.status = _ptr(res["status"])
    o.sub_margin = _ptr(res["sub_margin"])
    lib().or_tree_verify(C.byref(v), C.byref(o))
    return res


def row_probs(w, row, extra_hist=None):
    """Filtered distribution P of one row of a sampling workload (fp64)."""
    keep = []
    s = _sample_in(w, keep)
    eh = _c(extra_hist if extra_hist is not None else np.zeros(0, np.int32), np.int32)
    out = np.zeros(s.vocab, np.float64)
    st = lib().or_row_probs(C.byref(s), int(row), eh.ctypes.data if eh.size else None, int(eh.size), out.ctypes.data)
    return int(st), out


def residual_probs(P, q):
    P = np.ascontiguousarray(P, np.float64)
    q = np.ascontiguousarray(q, np.float32)
    out = np.zeros(P.size, np.float64)
    empty = lib().or_residual_probs(P.size, P.ctypes.data, q.ctypes.data, out.ctypes.data)
    return int(empty), out


def commit_accepted(out_tokens, num_accepted, status, tokens, seq_len, position):
    """The step after verification on copies of the state arrays; returns
    (tokens, seq_len, position, next_token, commit_status)."""
    out_tokens = np.ascontiguousarray(out_tokens, np.int32)
    R, width = out_tokens.shape
    tokens = np.array(tokens, np.int32, copy=True)
    seq_len = np.array(seq_len, np.int32, copy=True)
    position = np.array(position, np.int64, copy=True)
    next_token = np.full(R, -1, np.int32)
    cst = np.zeros(R, np.int32)
    na = np.ascontiguousarray(num_accepted, np.int32)
    st = np.ascontiguousarray(status, np.int32)
    lib().or_commit_accepted(R, width - 1, out_tokens.ctypes.data, na.ctypes.data, st.ctypes.data, tokens.ctypes.data,
                             tokens.shape[1], seq_len.ctypes.data, position.ctypes.data, next_token.ctypes.data,
                             cst.ctypes.data)
    return tokens, seq_len, position, next_token, cst


def lmhead_logits(hidden_bits, weight_bits):
    """logits = hidden @ weight.T of bf16 inputs, summed in fp64 and rounded
    to fp32 (a library matrix multiply as one step of the definition)."""
    h = (np.asarray(hidden_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w = (np.asarray(weight_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return (h @ w.T).astype(np.float32)


REL_MARGIN = 1e-5  # the decision margin of the C oracle (ss_oracle.c)


def interval_flags(logits, bound, temperature, seed, position, row_id=None):
    """Rows whose draw (temperature only: K is every token) can change when
    each logit z_t may lie anywhere in [z_t - bound_t, z_t + bound_t]: logits
    known only up to an error bound, such as an fp32 sum of many products.

    The draw is Gumbel-max, argmax_t y_t + g_t with y_t = z_t * fp32(1/T)
    (greedy, T = 0: argmax_t z_t), the lowest index among equals.  Each score
    is an interval: the logit's bound scaled by 1/T, plus the oracle's own
    margin of 1e-5 * max(1, |v|) on y_t and on g_t.  A row is flagged when
    some other token's highest score reaches the winner's lowest (the same
    test as the oracle's draw margin, with wider intervals)."""
    z = np.asarray(logits, np.float32)
    B, V = z.shape
    bound = np.broadcast_to(np.asarray(bound, np.float64), (B, V))
    flags = np.zeros(B, np.uint8)
    margin = lambda v: REL_MARGIN * np.maximum(1.0, np.abs(v))
    for r in range(B):
        T = np.float32(temperature[r])
        if T == 0:
            sc = z[r].astype(np.float64)
            unc = bound[r] + margin(sc)
        else:
            inv_t = np.float32(1.0) / T
            y = (z[r] * inv_t).astype(np.float64)
            rid = int(row_id[r]) if row_id is not None else r
            g = gumbel_row(int(seed[r]), rid, int(position[r]), V)
            sc = y + g
            unc = bound[r] * float(inv_t) + margin(y) + margin(g)
        b = int(np.argmax(sc))  # the first maximum: the lowest index
        hi = sc + unc
        hi[b] = -np.inf
        flags[r] = 1 if np.any(hi >= sc[b] - unc[b]) else 0
    return flags


def lmhead_sample(w):
    """The draw of the fused LM head: the sampling definition (temperature
    only) on the fp32 logits; returns process_sample's dict plus the logits."""
    z = lmhead_logits(w["hidden_states"], w["weight"])
    B, V = z.shape
    s = dict(kind="sample", num_rows=B, vocab=V, dtype="f32", logits=z, row_stride=V,
             temperature=w["temperature"], seed=w["seed"], position=w["position"])
    if w.get("row_id") is not None:
        s["row_id"] = w["row_id"]
    out = process_sample(s)
    out["logits"] = z
    return out
