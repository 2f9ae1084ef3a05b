"""Element-by-element comparison of the CUDA path with the CPU oracle."""
import numpy as np

from oracle import oracle as O


def _bits_equal(a, b):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    both_nan = np.isnan(a) & np.isnan(b)
    return np.all((a.view(np.uint32) == b.view(np.uint32)) | both_nan)


class Counts:
    """What a parity check compared: `total` rows (requests) with status OK;
    `exact` of them compared exactly (tokens, kept sizes, accepted counts);
    `forced` of those where the GPU's kept-set size differs from the oracle's
    own and lies inside the oracle's margin range (the oracle then drew from
    the GPU's kept set); `sub` rows whose draw / accept / residual decision is
    within the 1e-5 margin (counted, not compared)."""

    def __init__(self, total, exact, forced, sub):
        self.total, self.exact, self.forced, self.sub = int(total), int(exact), int(forced), int(sub)

    def as_dict(self):
        return dict(rows=self.total, exact=self.exact, forced_kept=self.forced, sub_margin=self.sub)

    def __iter__(self):  # (checked, sub), as the older callers unpack it
        return iter((self.exact, self.sub))

    def __repr__(self):
        return "Counts(%r)" % self.as_dict()


def check_sample(w, gpu, rows=None):
    """gpu: dict of numpy arrays token/status/kept[/processed].  Returns a
    Counts.  `rows` restricts the check (and the oracle run) to a subset, for
    full-size workloads."""
    if rows is not None:
        w = subset_sample(w, rows)
        gpu = {k: (v[rows] if isinstance(v, np.ndarray) else v) for k, v in gpu.items()}
    ref = O.process_sample(w, want_processed="processed" in gpu, force_kept=gpu["kept"])
    assert np.array_equal(gpu["status"], ref["status"]), (gpu["status"], ref["status"])
    ok = ref["status"] == 0
    if "processed" in gpu:
        cmp = ref["status"] <= 2
        for r in np.flatnonzero(cmp):
            assert _bits_equal(gpu["processed"][r], ref["processed"][r]), ("processed", r)
    lo, hi = ref["kept_lo"], ref["kept_hi"]
    bad = ok & ((gpu["kept"] < lo) | (gpu["kept"] > hi))
    assert not bad.any(), ("kept outside margin range", np.flatnonzero(bad), gpu["kept"][bad], lo[bad], hi[bad])
    assert np.all(gpu["token"][~ok] == -1)
    sub = ok & (ref["sub_margin"] != 0)
    chk = ok & ~sub
    mism = np.flatnonzero(chk & (gpu["token"] != ref["token"]))
    assert mism.size == 0, ("token mismatch", mism, gpu["token"][mism], ref["token"][mism])
    forced = ok & (gpu["kept"] != ref["kept_own"])
    return Counts(ok.sum(), chk.sum(), forced.sum(), sub.sum())


def subset_sample(w, rows):
    rows = np.asarray(rows)
    n = int(w["num_rows"])
    out = dict(w)
    out["num_rows"] = len(rows)
    stride = int(w["row_stride"])
    out["logits"] = w["logits"][rows] if stride else w["logits"]
    for key in ("temperature", "top_k", "top_p", "min_p", "repetition", "frequency", "presence",
                "use_bitmask", "seed", "position", "row_id"):
        if w.get(key) is not None:
            out[key] = w[key][rows]
    if w.get("bitmask") is not None:
        out["bitmask"] = w["bitmask"][rows]
    for off, vals in (("hist_offsets", ("hist_ids",)), ("bias_offsets", ("bias_ids", "bias_vals"))):
        if w.get(off) is None:
            continue
        o = w[off]
        new_off = np.zeros(len(rows) + 1, np.int32)
        parts = {v: [] for v in vals}
        for i, r in enumerate(rows):
            a, b = int(o[r]), int(o[r + 1])
            new_off[i + 1] = new_off[i] + (b - a)
            for v in vals:
                parts[v].append(w[v][a:b])
        out[off] = new_off
        for v in vals:
            out[v] = np.concatenate(parts[v]) if parts[v] else w[v][:0]
    assert n >= len(rows)
    return out


def subset_tree(w, reqs):
    """The requests `reqs` of a tree-verification workload, with their nodes,
    rows and per-request parameters."""
    reqs = np.asarray(reqs)
    off = w["node_offsets"]
    out = dict(w)
    out["num_requests"] = len(reqs)
    nodes = np.concatenate([np.arange(off[r], off[r + 1]) for r in reqs]) if len(reqs) else np.zeros(0, int)
    new_off = np.zeros(len(reqs) + 1, np.int32)
    new_off[1:] = np.cumsum([off[r + 1] - off[r] for r in reqs])
    out["node_offsets"] = new_off
    out["parents"] = w["parents"][nodes]
    out["node_tokens"] = w["node_tokens"][nodes]
    out["target_logits"] = w["target_logits"][nodes]
    out["draft_probs"] = w["draft_probs"][nodes]
    per_req = subset_sample(dict(w, num_rows=int(w["num_requests"]), logits=w["target_logits"], row_stride=0), reqs)
    for key in ("temperature", "top_k", "top_p", "min_p", "repetition", "frequency", "presence", "use_bitmask",
                "seed", "position", "row_id", "bitmask", "hist_offsets", "hist_ids", "bias_offsets", "bias_ids",
                "bias_vals"):
        if w.get(key) is not None:
            out[key] = per_req[key]
    return out


def check_verify(w, gpu):
    """gpu: out_tokens/num_accepted/status/kept[/processed].  Returns a
    Counts over requests (a request is `forced` when any of its target rows
    is)."""
    ref = O.spec_verify(w, want_processed="processed" in gpu, force_kept=gpu["kept"])
    assert np.array_equal(gpu["status"], ref["status"]), (gpu["status"], ref["status"])
    ok = ref["status"] == 0
    R = int(w["num_requests"])
    d_off = w["draft_offsets"]
    for i in np.flatnonzero(ok):
        rows = np.arange(int(d_off[i]) + i, int(d_off[i + 1]) + i + 1)
        k = gpu["kept"][rows]
        assert np.all((k >= ref["kept_lo"][rows]) & (k <= ref["kept_hi"][rows])), ("kept", i, k, ref["kept_lo"][rows], ref["kept_hi"][rows])
        if "processed" in gpu:
            for r in rows:
                assert _bits_equal(gpu["processed"][r], ref["processed"][r]), ("processed", i, r)
    assert np.all(gpu["out_tokens"][~ok] == -1)
    sub = ok & (ref["sub_margin"] != 0)
    chk = ok & ~sub
    for i in np.flatnonzero(chk):
        assert gpu["num_accepted"][i] == ref["num_accepted"][i], ("accepted", i, gpu["num_accepted"][i], ref["num_accepted"][i])
        assert np.array_equal(gpu["out_tokens"][i], ref["out_tokens"][i]), ("tokens", i, gpu["out_tokens"][i], ref["out_tokens"][i])
    forced = np.zeros(R, bool)
    for i in np.flatnonzero(ok):
        rows = np.arange(int(d_off[i]) + i, int(d_off[i + 1]) + i + 1)
        forced[i] = np.any(gpu["kept"][rows] != ref["kept_own"][rows])
    return Counts(ok.sum(), chk.sum(), forced.sum(), sub.sum())


def check_tree(w, gpu):
    """gpu: out_tokens/out_path/num_accepted/status.  Returns (checked
    requests, sub-margin requests); a sub-margin request must still be a
    valid walk: accepted nodes form a downward path from the root, the
    emitted drafts are their tokens and the final token is a token id."""
    ref = O.tree_verify(w)
    assert np.array_equal(gpu["status"], ref["status"]), (gpu["status"], ref["status"])
    ok = ref["status"] == 0
    assert np.all(gpu["out_tokens"][~ok] == -1)
    assert np.all(gpu["num_accepted"][~ok] == 0)
    sub = ok & (ref["sub_margin"] != 0)
    chk = ok & ~sub
    for i in np.flatnonzero(chk):
        assert gpu["num_accepted"][i] == ref["num_accepted"][i], ("accepted", i, gpu["num_accepted"][i], ref["num_accepted"][i])
        assert np.array_equal(gpu["out_tokens"][i], ref["out_tokens"][i]), ("tokens", i, gpu["out_tokens"][i], ref["out_tokens"][i])
        assert np.array_equal(gpu["out_path"][i], ref["out_path"][i]), ("path", i, gpu["out_path"][i], ref["out_path"][i])
    off, par, tok = w["node_offsets"], w["parents"], w["node_tokens"]
    for i in np.flatnonzero(sub):
        n = int(gpu["num_accepted"][i])
        u = 0
        for s in range(n):
            v = int(gpu["out_path"][i, s])
            assert 0 < v < off[i + 1] - off[i] and par[off[i] + v] == u, ("sub-margin walk", i)
            assert gpu["out_tokens"][i, s] == tok[off[i] + v]
            u = v
        assert 0 <= gpu["out_tokens"][i, n] < int(w["vocab"])
        assert np.all(gpu["out_tokens"][i, n + 1:] == -1)
    return int(chk.sum()), int(sub.sum())
