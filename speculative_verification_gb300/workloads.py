"""Seeded synthetic inputs for the sampling / verification path.

This module holds no sampling arithmetic: it only draws logits, per-row
parameters, histories, bias lists, grammar masks and drafts with numpy's PCG64
and packs them into a dictionary of numpy arrays.  Both the CUDA binding and
the CPU oracle consume these dictionaries; that is the only thing the two
share.

The five workloads follow the shapes the SonicSampler abstract describes
(per-request heterogeneous sampling over large vocabularies, grammar masks,
penalties, bias, speculative verification) at the sizes of the five benchmark
configurations.  No public dataset is involved: logits are Gaussian noise with
a few "spike" tokens, which gives the low-entropy structure the abstract talks
about.

Dictionary keys (all numpy):
  sampling:  kind='sample', num_rows, vocab, dtype ('f32'|'bf16'), logits
             ([rows, row_stride] float32 or uint16 bf16 bits), row_stride,
             per-row parameter arrays (see PARAM_KEYS)
  verify:    kind='verify', num_requests, vocab, max_draft, dtype,
             target_logits ([rows, row_stride]), row_stride, draft_offsets
             ([R+1]), draft_tokens, draft_probs ([sum k, draft_stride] f32),
             draft_stride, per-request parameter arrays
"""
import numpy as np

PARAM_KEYS = (
    "temperature", "top_k", "top_p", "min_p", "repetition", "frequency", "presence",
    "hist_offsets", "hist_ids", "bias_offsets", "bias_ids", "bias_vals",
    "bitmask", "bitmask_stride", "use_bitmask", "seed", "position",
)

CONFIG_NAMES = {
    1: "tiny sampling B=4 V=32000 fp32",
    2: "heterogeneous decode B=64 V=128256 bf16",
    3: "grammar-constrained B=128 V=151936 bf16",
    4: "speculative verify B=32 k=4 V=128256 bf16",
    5: "large mixed stress B=256 V=262144 bf16",
}


def to_bf16_bits(x):
    """Round float32 to bfloat16 (round to nearest even) and return the bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(h):
    return (np.asarray(h, dtype=np.uint32) << 16).view(np.float32)


def _spiky_rows(rng, rows, vocab, sigma, n_spikes_lo, n_spikes_hi, add_lo, add_hi):
    z = rng.normal(0.0, sigma, size=(rows, vocab)).astype(np.float32)
    for r in range(rows):
        ns = int(rng.integers(n_spikes_lo, n_spikes_hi + 1))
        pos = rng.choice(vocab, size=ns, replace=False)
        z[r, pos] += rng.uniform(add_lo, add_hi, size=ns).astype(np.float32)
    return z


def _csr(lists, dtype):
    off = np.zeros(len(lists) + 1, np.int32)
    for i, l in enumerate(lists):
        off[i + 1] = off[i] + len(l)
    flat = np.concatenate([np.asarray(l, dtype) for l in lists]) if off[-1] else np.zeros(0, dtype)
    return off, flat


def _grammar_mask(rng, vocab, must_allow, f_lo=0.01, f_hi=0.20):
    words = (vocab + 31) // 32
    f = rng.uniform(f_lo, f_hi)
    n = max(1, int(f * vocab))
    ids = rng.choice(vocab, size=n, replace=False)
    allowed = np.zeros(words * 32, bool)
    allowed[ids] = True
    for t in must_allow:
        allowed[int(t)] = True
    bits = allowed.reshape(words, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)
    return bits.sum(axis=1).astype(np.uint32).view(np.int32)


def _cfg2_params(rng, n, greedy_frac=0.25, with_min_p=True):
    temp = rng.uniform(0.5, 1.5, size=n).astype(np.float32)
    temp[rng.random(n) < greedy_frac] = 0.0
    top_k = rng.choice(np.array([0, 20, 50, 1000], np.int32), size=n)
    top_p = rng.choice(np.array([1.0, 0.9, 0.95], np.float32), size=n)
    min_p = (rng.choice(np.array([0.0, 0.05], np.float32), size=n) if with_min_p
             else np.zeros(n, np.float32))
    return temp, top_k.astype(np.int32), top_p.astype(np.float32), min_p.astype(np.float32)


def _penalty_lists(rng, n, vocab, enabled, hist_len=512, n_bias=16):
    hist, bias_ids, bias_vals = [], [], []
    for r in range(n):
        if enabled["pen"][r]:
            hist.append(rng.integers(0, vocab, size=hist_len).astype(np.int32))
        else:
            hist.append(np.zeros(0, np.int32))
        if enabled["bias"][r]:
            bias_ids.append(rng.choice(vocab, size=min(n_bias, vocab), replace=False).astype(np.int32))
            bias_vals.append(rng.uniform(-5.0, 5.0, size=min(n_bias, vocab)).astype(np.float32))
        else:
            bias_ids.append(np.zeros(0, np.int32))
            bias_vals.append(np.zeros(0, np.float32))
    ho, hi = _csr(hist, np.int32)
    bo, bi = _csr(bias_ids, np.int32)
    _, bv = _csr(bias_vals, np.float32)
    rep = np.where(enabled["pen"], 1.1, 1.0).astype(np.float32)
    freq = np.where(enabled["pen"], 0.2, 0.0).astype(np.float32)
    pres = np.where(enabled["pen"], 0.3, 0.0).astype(np.float32)
    return dict(repetition=rep, frequency=freq, presence=pres, hist_offsets=ho, hist_ids=hi,
                bias_offsets=bo, bias_ids=bi, bias_vals=bv)


def config1(seed=1, rows=4, vocab=32000):
    """Tiny sampling: fp32 N(0,2) logits plus three +8 spikes per row."""
    rng = np.random.Generator(np.random.PCG64(seed))
    z = _spiky_rows(rng, rows, vocab, 2.0, 3, 3, 8.0, 8.0)
    base_t = np.array([0.0, 0.8, 1.0, 0.7], np.float32)
    base_k = np.array([0, 50, 0, 0], np.int32)
    base_p = np.array([1.0, 1.0, 0.9, 1.0], np.float32)
    base_m = np.array([0.0, 0.0, 0.0, 0.05], np.float32)
    idx = np.arange(rows) % 4
    return dict(kind="sample", name=CONFIG_NAMES[1], num_rows=rows, vocab=vocab, dtype="f32",
                logits=z, row_stride=vocab,
                temperature=base_t[idx], top_k=base_k[idx], top_p=base_p[idx], min_p=base_m[idx],
                seed=np.zeros(rows, np.uint64), position=np.arange(rows, dtype=np.int64))


def config2(seed=2, rows=64, vocab=128256):
    """Heterogeneous decode: bf16 N(0,3) + 1..5 spikes at +6..+12, mixed params,
    penalties over a 512-id history and 16 bias entries on every row."""
    rng = np.random.Generator(np.random.PCG64(seed))
    z = _spiky_rows(rng, rows, vocab, 3.0, 1, 5, 6.0, 12.0)
    temp, top_k, top_p, min_p = _cfg2_params(rng, rows)
    on = np.ones(rows, bool)
    pen = _penalty_lists(rng, rows, vocab, {"pen": on, "bias": on})
    w = dict(kind="sample", name=CONFIG_NAMES[2], num_rows=rows, vocab=vocab, dtype="bf16",
             logits=to_bf16_bits(z), row_stride=vocab,
             temperature=temp, top_k=top_k, top_p=top_p, min_p=min_p,
             seed=(1000 + np.arange(rows)).astype(np.uint64),
             position=rng.integers(0, 4096, size=rows).astype(np.int64))
    w.update(pen)
    return w


def config3(seed=3, rows=128, vocab=151936):
    """Grammar-constrained: logits as workload 2, 1%..20% of tokens allowed."""
    rng = np.random.Generator(np.random.PCG64(seed))
    z = _spiky_rows(rng, rows, vocab, 3.0, 1, 5, 6.0, 12.0)
    words = (vocab + 31) // 32
    mask = np.stack([_grammar_mask(rng, vocab, [int(np.argmax(z[r]))]) for r in range(rows)])
    return dict(kind="sample", name=CONFIG_NAMES[3], num_rows=rows, vocab=vocab, dtype="bf16",
                logits=to_bf16_bits(z), row_stride=vocab,
                temperature=np.ones(rows, np.float32), top_p=np.full(rows, 0.95, np.float32),
                bitmask=mask, bitmask_stride=words,
                seed=(1000 + np.arange(rows)).astype(np.uint64),
                position=rng.integers(0, 4096, size=rows).astype(np.int64))


def _draft_probs(rng, target_f32_rows, noise=0.5):
    x = target_f32_rows.astype(np.float64) + rng.normal(0.0, noise, size=target_f32_rows.shape)
    x -= x.max(axis=1, keepdims=True)
    e = np.exp(x)
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def _sample_drafts(rng, q):
    out = np.empty(q.shape[0], np.int32)
    for i in range(q.shape[0]):
        p = q[i].astype(np.float64)
        out[i] = rng.choice(q.shape[1], p=p / p.sum())
    return out


def _verify_dict(name, vocab, max_draft, ks, target_f32, q, drafts, params):
    R = len(ks)
    d_off = np.zeros(R + 1, np.int32)
    d_off[1:] = np.cumsum(ks)
    w = dict(kind="verify", name=name, num_requests=R, vocab=vocab, max_draft=max_draft, dtype="bf16",
             target_logits=to_bf16_bits(target_f32), row_stride=vocab,
             draft_offsets=d_off, draft_tokens=drafts.astype(np.int32),
             draft_probs=q, draft_stride=vocab)
    w.update(params)
    return w


def config4(seed=4, requests=32, k=4, vocab=128256):
    """Speculative verify, linear drafts of length k, drafts from a noisy copy
    of the target distribution."""
    rng = np.random.Generator(np.random.PCG64(seed))
    z = _spiky_rows(rng, requests * (k + 1), vocab, 3.0, 1, 5, 6.0, 12.0)
    zb = bf16_bits_to_f32(to_bf16_bits(z)).reshape(requests, k + 1, vocab)
    q = _draft_probs(rng, zb[:, :k, :].reshape(-1, vocab))
    drafts = _sample_drafts(rng, q)
    temp, top_k, top_p, _ = _cfg2_params(rng, requests, with_min_p=False)
    params = dict(temperature=temp, top_k=top_k, top_p=top_p,
                  seed=(1000 + np.arange(requests)).astype(np.uint64),
                  position=rng.integers(0, 4096, size=requests).astype(np.int64))
    return _verify_dict(CONFIG_NAMES[4], vocab, k, np.full(requests, k, np.int32), z, q, drafts, params)


def config5(seed=5, requests=256, vocab=262144, max_draft=7, plain_top_k_max=4096):
    """Mixed stress: first half plain sampling on flat logits (k = 0 drafts),
    second half verification with 1..max_draft drafts; penalties, bias and a
    grammar mask each switched on per request with probability 1/2."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n_plain = requests // 2
    ks = np.zeros(requests, np.int32)
    ks[n_plain:] = rng.integers(1, max_draft + 1, size=requests - n_plain)
    rows_per = ks + 1
    z_rows, q_rows, d_rows = [], [], []
    spike_allow = []
    for i in range(requests):
        if i < n_plain:
            zr = rng.normal(0.0, 0.5, size=(1, vocab)).astype(np.float32)
        else:
            zr = _spiky_rows(rng, int(rows_per[i]), vocab, 3.0, 1, 5, 6.0, 12.0)
        z_rows.append(zr)
        spike_allow.append([int(np.argmax(zr[j])) for j in range(zr.shape[0])])
        if ks[i] > 0:
            zb = bf16_bits_to_f32(to_bf16_bits(zr[: ks[i]]))
            qi = _draft_probs(rng, zb)
            q_rows.append(qi)
            d_rows.append(_sample_drafts(rng, qi))
    z = np.concatenate(z_rows, axis=0)
    q = np.concatenate(q_rows, axis=0) if q_rows else np.zeros((0, vocab), np.float32)
    drafts = np.concatenate(d_rows) if d_rows else np.zeros(0, np.int32)

    temp, top_k, top_p, _ = _cfg2_params(rng, requests, with_min_p=False)
    temp[:n_plain] = rng.uniform(0.5, 1.5, size=n_plain).astype(np.float32)
    top_k[:n_plain] = rng.integers(1, plain_top_k_max + 1, size=n_plain).astype(np.int32)
    top_p[:n_plain] = rng.choice(np.array([1.0, 0.9, 0.95], np.float32), size=n_plain)
    enabled = {"pen": rng.random(requests) < 0.5, "bias": rng.random(requests) < 0.5}
    use_mask = (rng.random(requests) < 0.5).astype(np.uint8)
    words = (vocab + 31) // 32
    mask = np.stack([_grammar_mask(rng, vocab, spike_allow[i]) if use_mask[i]
                     else np.full(words, -1, np.int32) for i in range(requests)])
    params = dict(temperature=temp, top_k=top_k, top_p=top_p,
                  seed=(1000 + np.arange(requests)).astype(np.uint64),
                  position=rng.integers(0, 4096, size=requests).astype(np.int64),
                  bitmask=mask, bitmask_stride=words, use_bitmask=use_mask)
    params.update(_penalty_lists(rng, requests, vocab, enabled))
    return _verify_dict(CONFIG_NAMES[5], vocab, max_draft, ks, z, q, drafts, params)


def random_tree(rng, n, window=4):
    """Parent of every node of an n-node draft tree (the root's entry is -1):
    node v hangs under one of the `window` nodes before it, so the shapes range
    from chains to bushy levels."""
    par = np.full(n, -1, np.int32)
    for v in range(1, n):
        par[v] = rng.integers(max(0, v - window), v)
    return par


def chain_tree(n):
    par = np.arange(-1, n - 1, dtype=np.int32)
    return par


def tree(seed=6, requests=16, vocab=32000, max_nodes=16, dtype="bf16", shapes=None, greedy_frac=0.25,
         draft_noise=0.5):
    """Tree-draft verification: request i has 1..max_nodes nodes (node 0 the
    root); every node has a target row and a draft distribution q (a noisy copy
    of its target row); the children of a node are independent draws from its
    q.  `shapes` (optional) gives each request's parent array instead of a
    random tree.  Mixed sampling parameters as in the decode workload;
    penalties and bias on half of the requests."""
    rng = np.random.Generator(np.random.PCG64(seed))
    pars, toks, zs, qs = [], [], [], []
    for i in range(requests):
        if shapes is not None:
            par = np.asarray(shapes[i], np.int32)
        else:
            par = random_tree(rng, int(rng.integers(1, max_nodes + 1)))
        n = par.size
        z = _spiky_rows(rng, n, vocab, 3.0, 1, 5, 6.0, 12.0)
        zb = bf16_bits_to_f32(to_bf16_bits(z)) if dtype == "bf16" else z
        q = _draft_probs(rng, zb, noise=draft_noise)
        tok = np.zeros(n, np.int32)
        for v in range(1, n):
            pv = q[par[v]].astype(np.float64)
            tok[v] = rng.choice(vocab, p=pv / pv.sum())
        pars.append(par)
        toks.append(tok)
        zs.append(z)
        qs.append(q)
    ns = np.array([p_.size for p_ in pars], np.int32)
    off = np.zeros(requests + 1, np.int32)
    off[1:] = np.cumsum(ns)
    z = np.concatenate(zs, axis=0)
    temp, top_k, top_p, min_p = _cfg2_params(rng, requests, greedy_frac=greedy_frac)
    enabled = {"pen": rng.random(requests) < 0.5, "bias": rng.random(requests) < 0.5}
    params = dict(temperature=temp, top_k=top_k, top_p=top_p, min_p=min_p,
                  seed=(2000 + np.arange(requests)).astype(np.uint64),
                  position=rng.integers(0, 4096, size=requests).astype(np.int64))
    params.update(_penalty_lists(rng, requests, vocab, enabled))
    w = dict(kind="tree", name="tree verify R=%d max_nodes=%d V=%d %s" % (requests, max_nodes, vocab, dtype),
             num_requests=requests, vocab=vocab, max_nodes=max_nodes, dtype=dtype,
             target_logits=to_bf16_bits(z) if dtype == "bf16" else z.astype(np.float32), row_stride=vocab,
             node_offsets=off, parents=np.concatenate(pars), node_tokens=np.concatenate(toks),
             draft_probs=np.concatenate(qs, axis=0), draft_stride=vocab)
    w.update(params)
    return w


def make(cfg, **overrides):
    """Workload `cfg` (1..5) with optional size overrides (rows/requests/vocab)."""
    return {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}[cfg](**overrides)


def algorithmic_bytes(w):
    """Bytes the method must move for one call (logits read dominates).

    Sampling row: V*s logits + 4W mask words if masked + 4*len(history) +
    8*len(bias) + 40 B of parameters + 4 B output.  Verification request:
    (k+1)*V*s target logits + 8k for the draft tokens and q_j(x_j) + the same
    per-request terms; the q gathers of a rejected position depend on the
    outcome and are not counted.  Tree request: n*V*s target logits (one row
    per node) + 8n for node tokens and parents + the per-request terms.
    """
    s = 2 if w["dtype"] == "bf16" else 4
    V = int(w["vocab"])
    W = (V + 31) // 32
    if w["kind"] == "sample":
        n = int(w["num_rows"])
        rows = n
    elif w["kind"] == "tree":
        n = int(w["num_requests"])
        rows = int(w["node_offsets"][-1])
    else:
        n = int(w["num_requests"])
        rows = int(w["draft_offsets"][-1]) + n
    total = rows * V * s + 44 * n
    if w.get("bitmask") is not None:
        use = w.get("use_bitmask")
        total += 4 * W * (n if use is None else int(np.count_nonzero(use)))
    if w.get("hist_ids") is not None:
        total += 4 * int(w["hist_ids"].size)
    if w.get("bias_ids") is not None:
        total += 8 * int(w["bias_ids"].size)
    if w["kind"] == "verify":
        total += 8 * int(w["draft_tokens"].size)
    if w["kind"] == "tree":
        total += 8 * int(w["node_tokens"].size)  # token and parent of every node
    return int(total)


def shardable(w, k=200):
    """The same workload with a top-k of `k` on every sampling row that uses
    top-p or min-p without one (what the vocabulary-sharded path needs)."""
    w = dict(w)
    n = int(w["num_rows"])
    tk = np.array(w["top_k"], np.int32) if w.get("top_k") is not None else np.zeros(n, np.int32)
    tp = w["top_p"] if w.get("top_p") is not None else np.ones(n, np.float32)
    mp = w["min_p"] if w.get("min_p") is not None else np.zeros(n, np.float32)
    need = (tk <= 0) & ((tp < 1) | (mp > 0)) & (w["temperature"] > 0)
    tk[need] = k
    w["top_k"] = tk
    return w


def even_shards(vocab, parts):
    """[(offset, length)] of `parts` shards covering [0, vocab), offsets
    multiples of 32 (the last shard takes the remainder)."""
    size = -(-int(vocab) // int(parts))
    size = -(-size // 32) * 32
    return [(o, min(size, int(vocab) - o)) for o in range(0, int(vocab), size)]


def lmhead(batch=64, hidden=4096, vocab=128256, seed=6):
    """Synthetic LM-head inputs: hidden states N(0, 1) and weights
    N(0, 3 / sqrt(hidden)) as bf16 bits (logits about N(0, 3), as in the
    decode workload), 25% greedy rows, else T ~ U[0.5, 1.5], seeds and
    positions as in the decode workload."""
    rng = np.random.default_rng(seed)
    h = to_bf16_bits(rng.standard_normal((batch, hidden), dtype=np.float32))
    w = to_bf16_bits((rng.standard_normal((vocab, hidden), dtype=np.float32) * np.float32(3.0 / np.sqrt(hidden))))
    temp = rng.uniform(0.5, 1.5, batch).astype(np.float32)
    temp[rng.random(batch) < 0.25] = 0.0
    return dict(kind="lmhead", name="lmhead B=%d d=%d V=%d bf16" % (batch, hidden, vocab), batch=batch, hidden=hidden,
                vocab=vocab, hidden_states=h, weight=w, temperature=temp,
                seed=(1000 + np.arange(batch)).astype(np.uint64),
                position=rng.integers(0, 4096, batch).astype(np.int64))


_PER_REQUEST = ("temperature", "top_k", "top_p", "min_p", "repetition", "frequency", "presence", "use_bitmask",
                "seed", "position", "row_id")


def _subset_csr(w, out, reqs, off_key, val_keys):
    if w.get(off_key) is None:
        return
    o = w[off_key]
    new_off = np.zeros(len(reqs) + 1, np.int32)
    parts = {v: [] for v in val_keys}
    for i, r in enumerate(reqs):
        a, b = int(o[r]), int(o[r + 1])
        new_off[i + 1] = new_off[i] + (b - a)
        for v in val_keys:
            parts[v].append(w[v][a:b])
    out[off_key] = new_off
    for v in val_keys:
        out[v] = np.concatenate(parts[v]) if parts[v] else w[v][:0]


def subset_requests(w, reqs):
    """The requests `reqs` (in that order) of a sampling or linear
    verification workload, with their rows, drafts and per-request
    parameters, and row ids equal to their original indices (so every draw
    is the one it is in the whole batch): a smaller workload of the same
    kind."""
    reqs = [int(r) for r in reqs]
    out = dict(w)
    for key in _PER_REQUEST:
        if w.get(key) is not None:
            out[key] = np.asarray(w[key])[reqs]
    if w.get("row_id") is None:  # the noise stays keyed by the original index
        out["row_id"] = np.asarray(reqs, np.uint32)
    if w.get("bitmask") is not None:
        out["bitmask"] = w["bitmask"][reqs]
    _subset_csr(w, out, reqs, "hist_offsets", ("hist_ids",))
    _subset_csr(w, out, reqs, "bias_offsets", ("bias_ids", "bias_vals"))
    if w["kind"] == "sample":
        out["num_rows"] = len(reqs)
        out["logits"] = w["logits"][reqs]
        return out
    d = w["draft_offsets"]
    rows, drafts = [], []
    new_d = np.zeros(len(reqs) + 1, np.int32)
    for i, r in enumerate(reqs):
        k = int(d[r + 1] - d[r])
        rows.extend(range(int(d[r]) + r, int(d[r]) + r + k + 1))
        drafts.extend(range(int(d[r]), int(d[r + 1])))
        new_d[i + 1] = new_d[i] + k
    out["num_requests"] = len(reqs)
    out["draft_offsets"] = new_d
    out["target_logits"] = w["target_logits"][rows]
    out["draft_tokens"] = np.asarray(w["draft_tokens"])[drafts]
    out["draft_probs"] = w["draft_probs"][drafts] if len(drafts) else w["draft_probs"][:0]
    return out
