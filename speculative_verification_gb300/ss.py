"""Thin ctypes binding of libss (include/ss.h).

Argument marshalling only: every step of sampling and verification runs in
the CUDA kernels of libss.so.  PyTorch supplies device memory and the current
stream.  There is no CPU fallback: if the library is missing or no GPU is
present, the calls raise.
"""
import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libss.so")

SS_OK = 0
SS_ERR_SCRATCH_LIMIT = 5
SS_ROW_TIMEOUT = 5
SS_DTYPE = {"f32": 0, "bf16": 1}
ROW_STATUS = {0: "ok", 1: "empty_set", 2: "nonfinite", 3: "bad_index", 4: "bad_param", 5: "timeout", 6: "limit"}


class SSError(RuntimeError):
    pass


class ss_params(C.Structure):
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


class ss_fused_args(C.Structure):
    _fields_ = [
        ("batch", C.c_int32),
        ("hidden", C.c_int32),
        ("vocab", C.c_int32),
        ("hidden_states", C.c_void_p),
        ("weight", C.c_void_p),
        ("temperature", C.c_void_p),
        ("seed", C.c_void_p),
        ("position", C.c_void_p),
        ("row_id", C.c_void_p),
        ("scratch", C.c_void_p),
        ("scratch_bytes", C.c_size_t),
        ("out_token", C.c_void_p),
        ("out_status", C.c_void_p),
        ("debug_logits", C.c_void_p),
    ]


class ss_sample_args(C.Structure):
    _fields_ = [
        ("num_rows", C.c_int32),
        ("vocab", C.c_int32),
        ("row_stride", C.c_int64),
        ("dtype", C.c_int32),
        ("logits", C.c_void_p),
        ("params", ss_params),
        ("out_token", C.c_void_p),
        ("out_status", C.c_void_p),
        ("out_kept", C.c_void_p),
        ("debug_processed", C.c_void_p),
        ("flags", C.c_int32),
    ]


SS_SAMPLE_OVERLAP_PREVIOUS = 1
SS_VERIFY_OVERLAP_PREVIOUS = 1
SS_TREE_OVERLAP_PREVIOUS = 1


class ss_verify_args(C.Structure):
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
        ("params", ss_params),
        ("out_tokens", C.c_void_p),
        ("out_num_accepted", C.c_void_p),
        ("out_status", C.c_void_p),
        ("out_kept", C.c_void_p),
        ("debug_processed", C.c_void_p),
        ("flags", C.c_int32),
        ("num_target_rows", C.c_int32),
    ]


class ss_tree_args(C.Structure):
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
        ("params", ss_params),
        ("out_tokens", C.c_void_p),
        ("out_path", C.c_void_p),
        ("out_num_accepted", C.c_void_p),
        ("out_status", C.c_void_p),
        ("out_kept", C.c_void_p),
        ("debug_processed", C.c_void_p),
        ("flags", C.c_int32),
        ("num_nodes_total", C.c_int32),
    ]


# Every symbol include/ss.h declares, with its ctypes signature.
SIGNATURES = {
    "ss_workspace_size": ([C.c_int32, C.c_int32], C.c_size_t),
    "ss_workspace_init": ([C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "ss_process_sample": ([C.POINTER(ss_sample_args), C.c_void_p], C.c_int),
    "ss_shard_round_record_bytes": ([], C.c_size_t),
    "ss_shard_round_state_bytes": ([C.c_int32], C.c_size_t),
    "ss_shard_round": ([C.POINTER(ss_sample_args), C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                        C.c_void_p], C.c_int),
    "ss_merge_round": ([C.POINTER(ss_sample_args), C.c_int32, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p],
                       C.c_int),
    "ss_selftest_wait_timeout": ([C.POINTER(ss_sample_args), C.c_uint32, C.c_void_p], C.c_int),
    "ss_spec_verify": ([C.POINTER(ss_verify_args), C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "ss_spec_verify_noalloc": ([C.POINTER(ss_verify_args), C.c_void_p], C.c_int),
    "ss_tree_verify": ([C.POINTER(ss_tree_args), C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "ss_cluster_size": ([C.c_int32, C.c_int32], C.c_int32),
    "ss_last_cuda_error": ([], C.c_int32),
    "ss_status_string": ([C.c_int], C.c_char_p),
    "ss_version": ([], C.c_char_p),
    "ss_shard_record_bytes": ([C.c_int32], C.c_size_t),
    "ss_fused_scratch_bytes": ([C.c_int32], C.c_size_t),
    "ss_fused_lmhead_sample": ([C.POINTER(ss_fused_args), C.c_void_p], C.c_int),
    "ss_commit_accepted": ([C.c_int32, C.c_int32] + [C.c_void_p] * 4 + [C.c_int32] + [C.c_void_p] * 5, C.c_int),
    "ss_sample_shard": ([C.POINTER(ss_sample_args), C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p], C.c_int),
    "ss_merge_shards": ([C.POINTER(ss_sample_args), C.c_int32, C.POINTER(C.c_void_p), C.c_int32, C.c_void_p], C.c_int),
}

_lib = None


def load(path=None):
    """Load libss.so (raises if it was not built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise SSError("libss.so not built (%s); run __graft_entry__.build()" % p)
    L = C.CDLL(p)
    for name, (argt, rest) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.argtypes = argt
        fn.restype = rest
    if path is None:
        _lib = L
    return L


def _check(rc):
    if rc != SS_OK:
        L = load()
        msg = L.ss_status_string(rc).decode()
        if rc == 3:
            msg += " (cudaError %d)" % L.ss_last_cuda_error()
        raise SSError("libss: " + msg)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


PARAM_FIELDS = ("temperature", "top_k", "top_p", "min_p", "repetition", "frequency", "presence",
                "hist_offsets", "hist_ids", "bias_offsets", "bias_ids", "bias_vals", "bitmask",
                "use_bitmask", "seed", "position", "row_id")


def make_params(p):
    """ss_params from a dict of device tensors (missing / None = off).  A
    history or bias list with no entries at all is passed as off (an empty
    tensor has no data pointer, and the library wants offsets and ids
    together)."""
    sp = ss_params()
    empty = set()
    for off, ids in (("hist_offsets", ("hist_ids",)), ("bias_offsets", ("bias_ids", "bias_vals"))):
        t = p.get(ids[0])
        if t is not None and t.numel() == 0:
            empty.update((off,) + ids)
    for name in PARAM_FIELDS:
        setattr(sp, name, None if name in empty else _ptr(p.get(name)))
    sp.bitmask_stride = int(p.get("bitmask_stride", 0) or 0)
    return sp


def ss_version():
    return load().ss_version().decode()


def ss_cluster_size(vocab, dtype):
    return int(load().ss_cluster_size(int(vocab), SS_DTYPE[dtype]))


def ss_workspace_size(max_requests, max_draft):
    return int(load().ss_workspace_size(int(max_requests), int(max_draft)))


def ss_workspace_init(workspace, stream=None):
    _check(load().ss_workspace_init(C.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(),
                                    _stream_handle(stream)))


def _sample_args(logits, params, out_token, out_status, vocab, dtype, row_stride, out_kept, debug_processed, flags=0):
    a = ss_sample_args()
    a.flags = int(flags)
    a.num_rows = int(out_token.numel())
    a.vocab = int(vocab)
    a.row_stride = int(vocab if row_stride is None else row_stride)
    a.dtype = SS_DTYPE[dtype]
    a.logits = _ptr(logits)
    a.params = make_params(params)
    a.out_token = _ptr(out_token)
    a.out_status = _ptr(out_status)
    a.out_kept = _ptr(out_kept)
    a.debug_processed = _ptr(debug_processed)
    return a


def ss_process_sample(logits, params, out_token, out_status, *, vocab, dtype, row_stride=None, out_kept=None,
                      debug_processed=None, stream=None, overlap_previous=False):
    """Sample one token per row of `logits` (device tensor, [rows, row_stride]).
    overlap_previous sets SS_SAMPLE_OVERLAP_PREVIOUS (see include/ss.h): only
    when no input is an output of the sampling call before it."""
    a = _sample_args(logits, params, out_token, out_status, vocab, dtype, row_stride, out_kept, debug_processed,
                     SS_SAMPLE_OVERLAP_PREVIOUS if overlap_previous else 0)
    _check(load().ss_process_sample(C.byref(a), _stream_handle(stream)))


def ss_selftest_wait_timeout(logits, params, out_token, out_status, *, vocab, dtype, polls, row_stride=None,
                             out_kept=None, stream=None):
    """ss_process_sample with one bounded wait per CTA that nothing completes
    (the timeout self-test): every valid row reports SS_ROW_TIMEOUT."""
    a = _sample_args(logits, params, out_token, out_status, vocab, dtype, row_stride, out_kept, None)
    _check(load().ss_selftest_wait_timeout(C.byref(a), int(polls), _stream_handle(stream)))


def ss_commit_accepted(out_tokens, num_accepted, status, tokens, seq_len, position, next_token, commit_status,
                       stream=None):
    """Append each accepted request's emitted tokens to its row of `tokens`
    ([R, capacity] int32) and advance seq_len / position, on the device."""
    R, width = out_tokens.shape
    _check(load().ss_commit_accepted(int(R), int(width) - 1, _ptr(out_tokens), _ptr(num_accepted), _ptr(status),
                                     _ptr(tokens), int(tokens.shape[1]), _ptr(seq_len), _ptr(position),
                                     _ptr(next_token), _ptr(commit_status), _stream_handle(stream)))


def ss_fused_scratch_bytes(batch):
    return int(load().ss_fused_scratch_bytes(int(batch)))


def ss_fused_lmhead_sample(hidden_states, weight, temperature, seed, position, scratch, out_token, out_status, *,
                           row_id=None, debug_logits=None, stream=None):
    """Sample one token per row of hidden_states @ weight.T (bf16 device
    tensors [B, d] and [V, d]) without materialising the logits."""
    a = ss_fused_args()
    a.batch, a.hidden = int(hidden_states.shape[0]), int(hidden_states.shape[1])
    a.vocab = int(weight.shape[0])
    a.hidden_states, a.weight = _ptr(hidden_states), _ptr(weight)
    a.temperature, a.seed, a.position, a.row_id = _ptr(temperature), _ptr(seed), _ptr(position), _ptr(row_id)
    a.scratch = _ptr(scratch)
    a.scratch_bytes = int(scratch.numel() * scratch.element_size())
    a.out_token, a.out_status = _ptr(out_token), _ptr(out_status)
    a.debug_logits = _ptr(debug_logits)
    _check(load().ss_fused_lmhead_sample(C.byref(a), _stream_handle(stream)))


def ss_shard_record_bytes(list_cap):
    return int(load().ss_shard_record_bytes(int(list_cap)))


def ss_sample_shard(logits, params, records, *, vocab, vocab_offset, shard_len, list_cap, num_rows, dtype,
                    row_stride=None, stream=None):
    """Records of one vocabulary shard: `logits` holds tokens
    [vocab_offset, vocab_offset + shard_len) of every row."""
    a = ss_sample_args()
    a.num_rows = int(num_rows)
    a.vocab = int(vocab)
    a.row_stride = int(shard_len if row_stride is None else row_stride)
    a.dtype = SS_DTYPE[dtype]
    a.logits = _ptr(logits)
    a.params = make_params(params)
    _check(load().ss_sample_shard(C.byref(a), int(vocab_offset), int(shard_len), int(list_cap), _ptr(records),
                                  _stream_handle(stream)))


def ss_merge_shards(records, params, out_token, out_status, *, vocab, list_cap, out_kept=None, stream=None):
    """Merge of the records of the shards that cover the vocabulary."""
    a = ss_sample_args()
    a.num_rows = int(out_token.numel())
    a.vocab = int(vocab)
    a.params = make_params(params)
    a.out_token = _ptr(out_token)
    a.out_status = _ptr(out_status)
    a.out_kept = _ptr(out_kept)
    ptrs = (C.c_void_p * len(records))(*[r.data_ptr() for r in records])
    _check(load().ss_merge_shards(C.byref(a), len(records), ptrs, int(list_cap), _stream_handle(stream)))


def ss_shard_round_record_bytes():
    return int(load().ss_shard_round_record_bytes())


def ss_shard_round_state_bytes(num_rows):
    return int(load().ss_shard_round_state_bytes(int(num_rows)))


def ss_shard_round(logits, params, state, records, *, round, vocab, vocab_offset, shard_len, num_rows, dtype,
                   row_stride=None, stream=None):
    """One round of one vocabulary shard (rows without a top-k cut)."""
    a = ss_sample_args()
    a.num_rows = int(num_rows)
    a.vocab = int(vocab)
    a.row_stride = int(shard_len if row_stride is None else row_stride)
    a.dtype = SS_DTYPE[dtype]
    a.logits = _ptr(logits)
    a.params = make_params(params)
    _check(load().ss_shard_round(C.byref(a), int(vocab_offset), int(shard_len), int(round), _ptr(state),
                                 _ptr(records), _stream_handle(stream)))


def ss_merge_round(records, params, state, out_token, out_status, *, round, vocab, out_kept=None, stream=None):
    """The merge of one round over every shard's records."""
    a = ss_sample_args()
    a.num_rows = int(out_token.numel())
    a.vocab = int(vocab)
    a.params = make_params(params)
    a.out_token = _ptr(out_token)
    a.out_status = _ptr(out_status)
    a.out_kept = _ptr(out_kept)
    ptrs = (C.c_void_p * len(records))(*[r.data_ptr() for r in records])
    _check(load().ss_merge_round(C.byref(a), len(records), ptrs, int(round), _ptr(state), _stream_handle(stream)))


def _verify_args(target_logits, draft_offsets, draft_tokens, draft_probs, params, out_tokens, out_num_accepted,
                 out_status, vocab, max_draft, dtype, row_stride, draft_stride, out_kept, debug_processed, flags=0,
                 num_target_rows=0):
    a = ss_verify_args()
    a.flags = int(flags)
    a.num_target_rows = int(num_target_rows)
    a.num_requests = int(out_num_accepted.numel())
    a.vocab = int(vocab)
    a.max_draft = int(max_draft)
    a.row_stride = int(vocab if row_stride is None else row_stride)
    a.dtype = SS_DTYPE[dtype]
    a.target_logits = _ptr(target_logits)
    a.draft_offsets = _ptr(draft_offsets)
    a.draft_tokens = _ptr(draft_tokens) if draft_tokens is not None and draft_tokens.numel() else None
    a.draft_probs = _ptr(draft_probs) if draft_probs is not None and draft_probs.numel() else None
    a.draft_stride = int(vocab if draft_stride is None else draft_stride)
    a.params = make_params(params)
    a.out_tokens = _ptr(out_tokens)
    a.out_num_accepted = _ptr(out_num_accepted)
    a.out_status = _ptr(out_status)
    a.out_kept = _ptr(out_kept)
    a.debug_processed = _ptr(debug_processed)
    return a


def ss_spec_verify(target_logits, draft_offsets, draft_tokens, draft_probs, params, out_tokens, out_num_accepted,
                   out_status, workspace, *, vocab, max_draft, dtype, row_stride=None, draft_stride=None,
                   out_kept=None, debug_processed=None, stream=None, overlap_previous=False, num_target_rows=0):
    """Verify the drafts of `out_num_accepted.numel()` requests
    (overlap_previous sets SS_VERIFY_OVERLAP_PREVIOUS; num_target_rows is
    ss_verify_args.num_target_rows: see include/ss.h)."""
    a = _verify_args(target_logits, draft_offsets, draft_tokens, draft_probs, params, out_tokens, out_num_accepted,
                     out_status, vocab, max_draft, dtype, row_stride, draft_stride, out_kept, debug_processed,
                     SS_VERIFY_OVERLAP_PREVIOUS if overlap_previous else 0, num_target_rows)
    _check(load().ss_spec_verify(C.byref(a), C.c_void_p(workspace.data_ptr()),
                                 workspace.numel() * workspace.element_size(), _stream_handle(stream)))


def ss_spec_verify_noalloc(target_logits, draft_offsets, draft_tokens, draft_probs, params, out_tokens,
                           out_num_accepted, out_status, *, vocab, max_draft, dtype, row_stride=None,
                           draft_stride=None, out_kept=None, debug_processed=None, stream=None, num_target_rows=0):
    """ss_spec_verify with the library's static device scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    a = _verify_args(target_logits, draft_offsets, draft_tokens, draft_probs, params, out_tokens, out_num_accepted,
                     out_status, vocab, max_draft, dtype, row_stride, draft_stride, out_kept, debug_processed,
                     0, num_target_rows)
    _check(load().ss_spec_verify_noalloc(C.byref(a), _stream_handle(stream)))


def ss_tree_verify(target_logits, node_offsets, parents, node_tokens, draft_probs, params, out_tokens,
                   out_num_accepted, out_status, workspace, *, vocab, max_nodes, dtype, row_stride=None,
                   draft_stride=None, out_path=None, out_kept=None, debug_processed=None, stream=None,
                   overlap_previous=False, num_nodes_total=0):
    """Verify the draft trees of `out_num_accepted.numel()` requests
    (overlap_previous sets SS_TREE_OVERLAP_PREVIOUS; num_nodes_total is
    ss_tree_args.num_nodes_total: see include/ss.h)."""
    a = ss_tree_args()
    a.flags = SS_TREE_OVERLAP_PREVIOUS if overlap_previous else 0
    a.num_nodes_total = int(num_nodes_total)
    a.num_requests = int(out_num_accepted.numel())
    a.vocab = int(vocab)
    a.max_nodes = int(max_nodes)
    a.row_stride = int(vocab if row_stride is None else row_stride)
    a.dtype = SS_DTYPE[dtype]
    a.target_logits = _ptr(target_logits)
    a.node_offsets = _ptr(node_offsets)
    a.parents = _ptr(parents)
    a.node_tokens = _ptr(node_tokens)
    a.draft_probs = _ptr(draft_probs) if draft_probs is not None and draft_probs.numel() else None
    a.draft_stride = int(vocab if draft_stride is None else draft_stride)
    a.params = make_params(params)
    a.out_tokens = _ptr(out_tokens)
    a.out_path = _ptr(out_path)
    a.out_num_accepted = _ptr(out_num_accepted)
    a.out_status = _ptr(out_status)
    a.out_kept = _ptr(out_kept)
    a.debug_processed = _ptr(debug_processed)
    _check(load().ss_tree_verify(C.byref(a), C.c_void_p(workspace.data_ptr()),
                                 workspace.numel() * workspace.element_size(), _stream_handle(stream)))


# ------------------------------------------------------------ workloads --

_NP_TO_TORCH = None


def _torch_dtype(np_dtype):
    import torch
    global _NP_TO_TORCH
    if _NP_TO_TORCH is None:
        _NP_TO_TORCH = {np.dtype(np.float32): torch.float32, np.dtype(np.int32): torch.int32,
                        np.dtype(np.int64): torch.int64, np.dtype(np.uint8): torch.uint8,
                        np.dtype(np.uint64): torch.int64, np.dtype(np.uint16): torch.int16}
    return _NP_TO_TORCH[np.dtype(np_dtype)]


def to_device(w, device="cuda", pin=False):
    """Copy a workload dictionary's arrays to the device (seed bits and bf16
    bits are reinterpreted, not converted).  With pin=True, returns pinned host
    tensors instead (for end-to-end timing)."""
    import torch
    out = {}
    for key, val in w.items():
        if isinstance(val, np.ndarray):
            arr = np.ascontiguousarray(val)
            if arr.dtype == np.uint64:
                arr = arr.view(np.int64)
            elif arr.dtype == np.uint32:
                arr = arr.view(np.int32)
            elif arr.dtype == np.uint16:
                arr = arr.view(np.int16)
            t = torch.from_numpy(arr)
            if pin:
                t = t.pin_memory()
            else:
                t = t.to(device)
            if np.dtype(val.dtype) == np.uint16:
                t = t.view(torch.bfloat16)
            out[key] = t
        else:
            out[key] = val
    return out


def _host_array(val):
    """A workload array as the bytes the device sees (the same
    reinterpretations as to_device) and the torch dtype of its view."""
    import torch
    arr = np.ascontiguousarray(val)
    if arr.dtype == np.uint64:
        arr = arr.view(np.int64)
    elif arr.dtype == np.uint32:
        arr = arr.view(np.int32)
    bf16 = arr.dtype == np.uint16
    if bf16:
        arr = arr.view(np.int16)
    return arr, (torch.bfloat16 if bf16 else _torch_dtype(arr.dtype))


def pack_layout(w, align=256):
    """Byte layout of a workload's arrays in one contiguous buffer:
    {key: (offset, nbytes, shape, torch dtype)} and the total size."""
    lay, off = {}, 0
    for key, val in w.items():
        if isinstance(val, np.ndarray):
            arr, dt = _host_array(val)
            lay[key] = (off, arr.nbytes, arr.shape, dt)
            off += (arr.nbytes + align - 1) // align * align
    return lay, max(off, align)


def pack_pinned(w, lay, total):
    """The workload's arrays in one pinned host buffer laid out by `lay`, so
    that one copy moves a whole input set to the device."""
    import torch
    buf = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    view = buf.numpy()
    for key, (off, nbytes, _, _) in lay.items():
        arr, _ = _host_array(w[key])
        view[off:off + nbytes] = arr.reshape(-1).view(np.uint8)
    return buf


def views(buf, lay, w):
    """A workload dictionary whose arrays are views into `buf` (a device
    buffer filled by one copy of a pack_pinned buffer); scalars from `w`."""
    import torch
    out = {}
    for key, val in w.items():
        if key in lay:
            off, nbytes, shape, dt = lay[key]
            itemsize = torch.empty(0, dtype=dt).element_size()
            out[key] = buf[off:off + nbytes].view(dt).view(shape) if nbytes else torch.empty(
                shape, dtype=dt, device=buf.device)
            assert out[key].numel() * itemsize == nbytes
        else:
            out[key] = val
    return out


class Outputs(dict):
    pass


def alloc_outputs(dw, device="cuda", debug=False):
    """Output tensors for a workload (host or device arrays: only its sizes
    are read, and a device workload's offsets must already hold its data)."""
    import torch
    o = Outputs()
    V = int(dw["vocab"])
    if dw["kind"] == "sample":
        n = int(dw["num_rows"])
        o["token"] = torch.empty(n, dtype=torch.int32, device=device)
        o["status"] = torch.empty(n, dtype=torch.int32, device=device)
        o["kept"] = torch.empty(n, dtype=torch.int32, device=device)
        rows = n
    elif dw["kind"] == "tree":
        R = int(dw["num_requests"])
        rows = int(dw["node_offsets"][-1].item())
        width = int(dw["max_nodes"])
        o["out_tokens"] = torch.empty((R, width), dtype=torch.int32, device=device)
        o["out_path"] = torch.empty((R, width), dtype=torch.int32, device=device)
        o["num_accepted"] = torch.empty(R, dtype=torch.int32, device=device)
        o["status"] = torch.empty(R, dtype=torch.int32, device=device)
        o["kept"] = torch.empty(rows, dtype=torch.int32, device=device)
        nbytes = ss_workspace_size(R, width - 1)
        o["workspace"] = torch.zeros((nbytes + 15) // 16 * 4, dtype=torch.int32, device=device)
    else:
        R = int(dw["num_requests"])
        rows = int(dw["draft_offsets"][-1].item()) + R
        o["out_tokens"] = torch.empty((R, int(dw["max_draft"]) + 1), dtype=torch.int32, device=device)
        o["num_accepted"] = torch.empty(R, dtype=torch.int32, device=device)
        o["status"] = torch.empty(R, dtype=torch.int32, device=device)
        o["kept"] = torch.empty(rows, dtype=torch.int32, device=device)
        nbytes = ss_workspace_size(R, int(dw["max_draft"]))
        o["workspace"] = torch.zeros((nbytes + 15) // 16 * 4, dtype=torch.int32, device=device)
    if debug:
        o["processed"] = torch.empty((rows, V), dtype=torch.float32, device=device)
    return o


def run(dw, o, stream=None, debug=False, overlap_previous=False, target_rows=False):
    """One library call on a device workload `dw` into outputs `o`
    (overlap_previous: see ss_process_sample; every kind of call).  With
    target_rows, a verification call states its number of target rows (the
    rows of dw["target_logits"]: ss_verify_args.num_target_rows,
    ss_tree_args.num_nodes_total)."""
    params = {k: dw.get(k) for k in PARAM_FIELDS}
    params["bitmask_stride"] = dw.get("bitmask_stride", 0)
    dbg = o.get("processed") if debug else None
    if dw["kind"] == "sample":
        ss_process_sample(dw["logits"], params, o["token"], o["status"], vocab=dw["vocab"], dtype=dw["dtype"],
                          row_stride=dw["row_stride"], out_kept=o["kept"], debug_processed=dbg, stream=stream,
                          overlap_previous=overlap_previous)
    elif dw["kind"] == "tree":
        ss_tree_verify(dw["target_logits"], dw["node_offsets"], dw["parents"], dw["node_tokens"], dw["draft_probs"],
                       params, o["out_tokens"], o["num_accepted"], o["status"], o["workspace"], vocab=dw["vocab"],
                       max_nodes=dw["max_nodes"], dtype=dw["dtype"], row_stride=dw["row_stride"],
                       draft_stride=dw["draft_stride"], out_path=o["out_path"], out_kept=o["kept"],
                       debug_processed=dbg, stream=stream, overlap_previous=overlap_previous,
                       num_nodes_total=int(dw["target_logits"].shape[0]) if target_rows else 0)
    else:
        ss_spec_verify(dw["target_logits"], dw["draft_offsets"], dw["draft_tokens"], dw["draft_probs"], params,
                       o["out_tokens"], o["num_accepted"], o["status"], o["workspace"], vocab=dw["vocab"],
                       max_draft=dw["max_draft"], dtype=dw["dtype"], row_stride=dw["row_stride"],
                       draft_stride=dw["draft_stride"], out_kept=o["kept"], debug_processed=dbg, stream=stream,
                       overlap_previous=overlap_previous,
                       num_target_rows=int(dw["target_logits"].shape[0]) if target_rows else 0)
