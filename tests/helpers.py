"""Small builders for hand-made workload dictionaries used by the tests."""
import numpy as np

from speculative_verification_gb300 import workloads as W


def sample_workload(logits, dtype="f32", temperature=1.0, top_k=None, top_p=None, min_p=None,
                    repetition=None, frequency=None, presence=None, history=None, bias=None,
                    mask_words=None, use_mask=None, seed=0, position=None, row_stride=None, num_rows=None):
    """logits: [rows, V] float array.  Scalars broadcast over rows; history is a
    list of id lists; bias a list of (ids, vals); mask_words [rows, W] int32.
    With row_stride=0 every one of `num_rows` rows reads logits row 0."""
    z = np.atleast_2d(np.asarray(logits, np.float32))
    n, V = z.shape
    if num_rows is not None:
        n = int(num_rows)
    def col(v, dt):
        if v is None:
            return None
        a = np.asarray(v, dt)
        return np.full(n, a, dt) if a.ndim == 0 else a
    w = dict(kind="sample", num_rows=n, vocab=V, dtype=dtype,
             logits=(W.to_bf16_bits(z) if dtype == "bf16" else z),
             row_stride=V if row_stride is None else row_stride,
             temperature=col(temperature, np.float32), top_k=col(top_k, np.int32),
             top_p=col(top_p, np.float32), min_p=col(min_p, np.float32),
             repetition=col(repetition, np.float32), frequency=col(frequency, np.float32),
             presence=col(presence, np.float32),
             seed=col(seed, np.uint64),
             position=(np.arange(n, dtype=np.int64) if position is None else col(position, np.int64)))
    if history is not None:
        off = np.zeros(n + 1, np.int32)
        off[1:] = np.cumsum([len(h) for h in history])
        w["hist_offsets"] = off
        w["hist_ids"] = (np.concatenate([np.asarray(h, np.int32) for h in history])
                         if off[-1] else np.zeros(0, np.int32))
    if bias is not None:
        off = np.zeros(n + 1, np.int32)
        off[1:] = np.cumsum([len(b[0]) for b in bias])
        w["bias_offsets"] = off
        w["bias_ids"] = (np.concatenate([np.asarray(b[0], np.int32) for b in bias])
                         if off[-1] else np.zeros(0, np.int32))
        w["bias_vals"] = (np.concatenate([np.asarray(b[1], np.float32) for b in bias])
                          if off[-1] else np.zeros(0, np.float32))
    if mask_words is not None:
        m = np.atleast_2d(np.asarray(mask_words).astype(np.uint32).view(np.int32))
        w["bitmask"] = m
        w["bitmask_stride"] = m.shape[1]
        if use_mask is not None:
            w["use_bitmask"] = col(use_mask, np.uint8)
    return w


def verify_workload(target_logits, ks, drafts, draft_probs, dtype="f32", temperature=1.0, top_k=None,
                    top_p=None, min_p=None, seed=0, position=0, max_draft=None, history=None,
                    repetition=None, frequency=None, presence=None):
    """target_logits: [sum(k+1), V]; ks: per-request draft counts; drafts: [sum k];
    draft_probs: [sum k, V]."""
    z = np.atleast_2d(np.asarray(target_logits, np.float32))
    V = z.shape[1]
    ks = np.asarray(ks, np.int32)
    R = ks.size
    def col(v, dt):
        if v is None:
            return None
        a = np.asarray(v, dt)
        return np.full(R, a, dt) if a.ndim == 0 else a
    off = np.zeros(R + 1, np.int32)
    off[1:] = np.cumsum(ks)
    q = np.asarray(draft_probs, np.float32).reshape(-1, V) if int(ks.sum()) else np.zeros((0, V), np.float32)
    w = dict(kind="verify", num_requests=R, vocab=V, max_draft=int(ks.max() if max_draft is None else max_draft),
             dtype=dtype, target_logits=(W.to_bf16_bits(z) if dtype == "bf16" else z), row_stride=V,
             draft_offsets=off, draft_tokens=np.asarray(drafts, np.int32).reshape(-1),
             draft_probs=q, draft_stride=V,
             temperature=col(temperature, np.float32), top_k=col(top_k, np.int32),
             top_p=col(top_p, np.float32), min_p=col(min_p, np.float32),
             repetition=col(repetition, np.float32), frequency=col(frequency, np.float32),
             presence=col(presence, np.float32),
             seed=col(seed, np.uint64), position=col(position, np.int64))
    if history is not None:
        hoff = np.zeros(R + 1, np.int32)
        hoff[1:] = np.cumsum([len(h) for h in history])
        w["hist_offsets"] = hoff
        w["hist_ids"] = (np.concatenate([np.asarray(h, np.int32) for h in history])
                         if hoff[-1] else np.zeros(0, np.int32))
    return w


def tree_workload(target_logits, node_offsets, parents, node_tokens, draft_probs, max_nodes=None, dtype="f32",
                  temperature=1.0, top_k=None, top_p=None, min_p=None, seed=0, position=0, history=None,
                  repetition=None, frequency=None, presence=None):
    """target_logits / draft_probs: [sum n, V] (one row per node); node_offsets [R+1];
    parents / node_tokens: [sum n], local indices (root -1)."""
    z = np.atleast_2d(np.asarray(target_logits, np.float32))
    V = z.shape[1]
    off = np.asarray(node_offsets, np.int32)
    R = off.size - 1
    ns = np.diff(off)

    def col(v, dt):
        if v is None:
            return None
        a = np.asarray(v, dt)
        return np.full(R, a, dt) if a.ndim == 0 else a
    w = dict(kind="tree", num_requests=R, vocab=V, max_nodes=int(ns.max() if max_nodes is None else max_nodes),
             dtype=dtype, target_logits=(W.to_bf16_bits(z) if dtype == "bf16" else z), row_stride=V,
             node_offsets=off, parents=np.asarray(parents, np.int32).reshape(-1),
             node_tokens=np.asarray(node_tokens, np.int32).reshape(-1),
             draft_probs=np.asarray(draft_probs, np.float32).reshape(-1, V), draft_stride=V,
             temperature=col(temperature, np.float32), top_k=col(top_k, np.int32),
             top_p=col(top_p, np.float32), min_p=col(min_p, np.float32),
             repetition=col(repetition, np.float32), frequency=col(frequency, np.float32),
             presence=col(presence, np.float32),
             seed=col(seed, np.uint64), position=col(position, np.int64))
    if history is not None:
        hoff = np.zeros(R + 1, np.int32)
        hoff[1:] = np.cumsum([len(h) for h in history])
        w["hist_offsets"] = hoff
        w["hist_ids"] = (np.concatenate([np.asarray(h, np.int32) for h in history])
                         if hoff[-1] else np.zeros(0, np.int32))
    return w


def chain_from_linear(w):
    """The tree form of a linear verification workload: request i's nodes are
    its k_i + 1 target rows in order, node j + 1 the child of node j."""
    R, V = int(w["num_requests"]), int(w["vocab"])
    dof = np.asarray(w["draft_offsets"])
    ks = np.diff(dof)
    ns = ks + 1
    off = np.zeros(R + 1, np.int32)
    off[1:] = np.cumsum(ns)
    par, tok, q = [], [], []
    for i in range(R):
        k = int(ks[i])
        par.append(np.arange(-1, k, dtype=np.int32))
        tok.append(np.concatenate([[0], w["draft_tokens"][dof[i]:dof[i + 1]]]).astype(np.int32))
        q.append(np.concatenate([w["draft_probs"][dof[i]:dof[i + 1]], np.zeros((1, V), np.float32)]))
    t = dict(w)
    t.update(kind="tree", max_nodes=int(w["max_draft"]) + 1, node_offsets=off, parents=np.concatenate(par),
             node_tokens=np.concatenate(tok), draft_probs=np.concatenate(q))
    for key in ("draft_offsets", "draft_tokens", "max_draft"):
        t.pop(key)
    return t
