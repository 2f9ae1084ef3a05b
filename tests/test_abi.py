"""The C ABI library builds, loads and exports every symbol include/ss.h
declares (no compute calls: this runs without a GPU)."""
import os
import re

import pytest

from speculative_verification_gb300 import build as ss_build
from speculative_verification_gb300 import ss

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "ss.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ss_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    ss_build.build()
    return ss.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "ss_process_sample" in names and "ss_spec_verify" in names
    for name in names:
        assert hasattr(lib, name), name
        assert name in ss.SIGNATURES, name


def test_every_call_that_enqueues_work_opens_an_nvtx_range():
    # each public entry point returning ss_status names itself in one NVTX
    # range (the calls that only answer a size or a string have none)
    csrc = os.path.join(ROOT, "speculative_verification_gb300", "csrc")
    found = {}
    for f in sorted(os.listdir(csrc)):
        if f.endswith(".cu"):
            text = open(os.path.join(csrc, f)).read()
            for m in re.finditer(r"\nss_status (ss_[a-z0-9_]+)\(.*?\) \{\n(.*?)\n", text, flags=re.S):
                found[m.group(1)] = m.group(2).strip()
    declared = [n for n in _declared_functions() if n in found]
    assert "ss_process_sample" in declared and "ss_spec_verify_noalloc" in declared and "ss_merge_round" in declared
    for name in declared:
        assert found[name] == 'SS_NVTX_RANGE("%s");' % name, (name, found[name])


def test_host_only_queries(lib):
    assert ss.ss_version().startswith("ss ")
    assert ss.ss_cluster_size(128256, "bf16") == 4
    assert ss.ss_cluster_size(262144, "bf16") == 8
    assert ss.ss_cluster_size(32000, "f32") == 2
    assert ss.ss_cluster_size(10, "f32") == 1
    assert ss.ss_cluster_size(0, "f32") == 0
    assert ss.ss_cluster_size(10_000_000, "bf16") == 0
    # largest supported rows: 8 slices of at most 61,440 tokens / 160 KiB whose
    # shared-memory layout fits 227 KiB per CTA
    assert ss.ss_cluster_size(491_520, "bf16") == 8
    assert ss.ss_cluster_size(491_521, "bf16") == 0
    assert ss.ss_cluster_size(321_536, "f32") == 8
    assert ss.ss_cluster_size(321_537, "f32") == 0
    assert ss.ss_cluster_size(327_680, "f32") == 0  # 160 KiB slices, but the tables would not fit
    assert ss.ss_workspace_size(32, 4) >= 32 * 5 * 16 + 32 * 4
    assert lib.ss_status_string(0) == b"ok"


def test_host_side_argument_errors_launch_nothing(lib):
    import ctypes as C
    a = ss.ss_sample_args()
    a.num_rows = 4
    a.vocab = 0  # invalid
    assert lib.ss_process_sample(C.byref(a), None) == 1
    a.vocab = 100
    a.dtype = 7  # invalid dtype
    assert lib.ss_process_sample(C.byref(a), None) == 1
    a.dtype = 1
    a.logits = 16  # no output pointers
    assert lib.ss_process_sample(C.byref(a), None) == 1
    a.num_rows = 0  # empty batch: nothing to do
    assert lib.ss_process_sample(C.byref(a), None) == 0
    a.flags = 2  # an unknown flag bit
    assert lib.ss_process_sample(C.byref(a), None) == 1
    a.flags = ss.SS_SAMPLE_OVERLAP_PREVIOUS
    assert lib.ss_process_sample(C.byref(a), None) == 0
    assert lib.ss_process_sample(None, None) == 1
    v = ss.ss_verify_args()
    v.num_requests = 2
    v.vocab = 64
    v.max_draft = 2
    v.row_stride = 64
    v.target_logits = 16
    v.draft_offsets = 32
    v.draft_tokens = 48
    v.draft_probs = 64
    v.draft_stride = 64
    v.out_tokens, v.out_num_accepted, v.out_status = 80, 96, 112
    v.params.temperature, v.params.seed, v.params.position = 128, 144, 160
    assert lib.ss_spec_verify(C.byref(v), None, 0, None) == 4  # workspace missing
    assert lib.ss_spec_verify(C.byref(v), C.c_void_p(256), 8, None) == 4  # too small
    v.row_stride = 63  # stride < vocab
    assert lib.ss_spec_verify(C.byref(v), C.c_void_p(256), 1 << 20, None) == 1
    v.row_stride = 64
    for rows in (-1, 1, 7):  # outside [R, R * (max_draft + 1)] = [2, 6]
        v.num_target_rows = rows
        assert lib.ss_spec_verify(C.byref(v), C.c_void_p(256), 1 << 20, None) == 1, rows
        assert lib.ss_spec_verify_noalloc(C.byref(v), None) == 1, rows
    v.num_target_rows = 0
    t = ss.ss_tree_args()
    t.num_requests, t.vocab, t.max_nodes, t.dtype = 0, 100, 4, 1
    assert lib.ss_tree_verify(C.byref(t), None, 0, None) == 0  # no requests: nothing to do
    t.flags = 2  # an unknown flag bit
    assert lib.ss_tree_verify(C.byref(t), None, 0, None) == 1
    t.flags = ss.SS_TREE_OVERLAP_PREVIOUS
    assert lib.ss_tree_verify(C.byref(t), None, 0, None) == 0
    t.num_requests = 2
    for nodes in (-1, 1, 9):  # outside [R, R * max_nodes] = [2, 8]
        t.num_nodes_total = nodes
        assert lib.ss_tree_verify(C.byref(t), None, 0, None) == 1, nodes


def test_shard_entry_points_reject_bad_arguments(lib):
    import ctypes as C
    assert ss.ss_shard_record_bytes(1) == 40
    assert ss.ss_shard_record_bytes(1024) == 32 + 8 * 1024
    assert ss.ss_shard_record_bytes(0) == 0 and ss.ss_shard_record_bytes(1025) == 0
    a = ss.ss_sample_args()
    a.num_rows, a.vocab, a.dtype, a.row_stride, a.logits = 2, 1000, 1, 1000, 16
    a.params.temperature, a.params.seed, a.params.position = 128, 144, 160
    rec = C.c_void_p(4096)
    f = lib.ss_sample_shard
    assert f(C.byref(a), 16, 100, 8, rec, None) == 1    # offset not a multiple of 32
    assert f(C.byref(a), 960, 100, 8, rec, None) == 1   # shard past the vocabulary
    assert f(C.byref(a), 0, 0, 8, rec, None) == 1       # empty shard
    assert f(C.byref(a), 0, 100, 0, rec, None) == 1     # list capacity out of range
    assert f(C.byref(a), 0, 100, 8, C.c_void_p(4100), None) == 1  # records not 8-byte aligned
    assert f(C.byref(a), 0, 100, 8, None, None) == 1
    a.debug_processed = 512
    assert f(C.byref(a), 0, 100, 8, rec, None) == 1     # no debug output on a shard
    a.debug_processed = None
    a.num_rows = 0
    assert f(C.byref(a), 0, 100, 8, rec, None) == 0     # nothing to do
    a.num_rows = 2
    ptrs = (C.c_void_p * 9)(*([4096] * 9))
    m = lib.ss_merge_shards
    assert m(C.byref(a), 0, ptrs, 8, None) == 1         # no shards
    assert m(C.byref(a), 9, ptrs, 8, None) == 1         # more than 8 shards
    assert m(C.byref(a), 2, ptrs, 8, None) == 1         # no outputs
    assert m(None, 2, ptrs, 8, None) == 1


def test_empty_history_and_bias_lists_are_passed_as_off():
    torch = pytest.importorskip("torch")
    p = {"temperature": torch.ones(3), "hist_offsets": torch.zeros(4, dtype=torch.int32),
         "hist_ids": torch.zeros(0, dtype=torch.int32), "bias_offsets": torch.tensor([0, 1, 1, 2], dtype=torch.int32),
         "bias_ids": torch.tensor([5, 7], dtype=torch.int32), "bias_vals": torch.tensor([1.0, -1.0])}
    sp = ss.make_params(p)
    assert sp.hist_offsets is None and sp.hist_ids is None
    assert sp.bias_offsets and sp.bias_ids and sp.bias_vals and sp.temperature


def test_tree_entry_point_rejects_bad_arguments(lib):
    a = ss.ss_tree_args()
    assert lib.ss_tree_verify(None, None, 0, None) == 1
    a.num_requests, a.vocab, a.max_nodes, a.dtype = 1, 100, 65, 1  # more nodes than the limit
    assert lib.ss_tree_verify(ss.C.byref(a), None, 0, None) == 1
    a.max_nodes = 0
    assert lib.ss_tree_verify(ss.C.byref(a), None, 0, None) == 1
    a.max_nodes, a.num_requests = 4, 0  # nothing to do
    assert lib.ss_tree_verify(ss.C.byref(a), None, 0, None) == 0


def test_argument_structs_match_the_header():
    """The binding's ctypes structs list the header's fields, in order."""
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "ss.h")).read(), flags=re.S)
    structs = re.findall(r"typedef struct \{(.*?)\}\s*(\w+);", text, flags=re.S)
    assert len(structs) >= 5
    for body, name in structs:
        fields = []
        for decl in (d.strip() for d in body.split(";")):
            if decl:
                first, *more = decl.split(",")  # "int32_t a, b, c"
                fields += [re.split(r"[\s*]+", first.strip())[-1]] + [m.strip(" *") for m in more]
        cls = getattr(ss, name)
        assert [f[0] for f in cls._fields_] == fields, name
