"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports
every symbol the header declares, and rejects bad arguments on the host
before any CUDA call. The planner's host logic runs without a GPU."""
import ctypes
import os
import re
import shutil

import numpy as np
import pytest

import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specattn.h")

needs_nvcc = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="no CUDA toolkit")


@pytest.fixture(scope="module")
def sa():
    from speculative_decode_gb300 import build
    build.build()
    import speculative_decode_gb300 as mod
    mod.load_library()
    return mod


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SA_API\s+[\w\s\*]*?\b(sa_\w+)\s*\(", text)))


@needs_nvcc
def test_every_declared_symbol_is_exported(sa):
    names = declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(sa.library_path())
    for n in names:
        assert hasattr(lib, n), n


@needs_nvcc
def test_status_strings(sa):
    assert sa.status_string(0) == "ok"
    assert "out of range" in sa.status_string(3)
    assert sa.status_string(99) == "unknown status"


@needs_nvcc
def test_host_side_argument_checks_need_no_gpu(sa):
    lib = sa.load_library()
    d = sa.dims_for(4, 8, 2, 16, 4, 4, 1)
    d.head_dim = 64
    assert lib.sa_paged_attn(ctypes.byref(d), *([None] * 6), 0.1, None, None, None, 0, None, None) == 2
    d = sa.dims_for(4, 8, 3, 16, 4, 4, 1)      # Hq not a multiple of Hkv
    assert lib.sa_kv_append(ctypes.byref(d), *([None] * 9)) == 1
    d = sa.dims_for(4, 8, 2, 16, 4, 4, 513)    # max_q_len above 512
    assert lib.sa_paged_attn(ctypes.byref(d), *([None] * 6), 0.1, None, None, None, 0, None, None) == 2
    d = sa.dims_for(1, 8, 2, 16, 4, 17, 17)     # plans take max_q_len <= 16
    bt, sl, ql = np.zeros((1, 4), np.int32), np.array([17], np.int32), np.array([17], np.int32)
    assert lib.sa_plan_analyze(ctypes.byref(d), bt.ctypes.data, sl.ctypes.data, ql.ctypes.data, 148,
                               None, None, None, None) == 2
    d = sa.dims_for(4, 8, 2, 16, 4, 4, 1)
    assert lib.sa_paged_attn(ctypes.byref(d), *([None] * 6), 0.1, None, None, None, 0, None, None) == 1
    assert lib.sa_spec_verify_greedy(None, None, None, 2, 16, 100, *([None] * 4), 0, None, None) == 2
    assert lib.sa_spec_verify_greedy(None, None, None, -1, 3, 100, *([None] * 4), 0, None, None) == 1
    # the advancing variant needs the window and the three length buffers
    assert lib.sa_spec_verify_greedy_advance(None, None, None, 2, 3, 100, *([None] * 7), 0, None, None) == 1
    # the bounded-wait self-test needs a flag to set
    assert lib.sa_selftest_bounded_wait(None, None) == 1
    # quantised pages: null pools are argument errors before any GPU work
    for name in ("sa_paged_attn_q8", "sa_paged_attn_q4"):
        assert getattr(lib, name)(ctypes.byref(d), *([None] * 8), 0.1, None, None, 0, None, None) == 1
    for name in ("sa_kv_append_q8", "sa_kv_append_q4"):
        assert getattr(lib, name)(ctypes.byref(d), *([None] * 11)) == 1


@needs_nvcc
def test_workspace_sizes(sa):
    w = wl.config(1)
    d = sa.dims_for(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.num_pages,
                    w.max_pages_per_seq, w.total_q, 1)
    n = sa.paged_attn_workspace_size(d)
    # decode (4 query rows per KV head) takes the persistent kernel: a 4 KiB
    # counter region, then two partial slots per CTA (up to 256 CTAs) of 4
    # rows x (128 accumulators + max and sum) fp32
    assert n >= 4096 + 2 * 256 * 4 * 130 * 4
    assert n % 256 == 0
    # 24 query rows per KV head (verification) take the split path: up to 8
    # tensor-core pieces and 8 split pieces of 130 floats per row
    dv = sa.dims_for(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.num_pages,
                     w.max_pages_per_seq, 6 * w.num_seqs, 6)
    assert sa.paged_attn_workspace_size(dv) >= 16 * 6 * w.num_seqs * w.num_q_heads * 130 * 4
    assert sa.spec_verify_workspace_size(16, 5, 128256) >= 16 * 6 * 8
    assert sa.spec_verify_workspace_size(16, 16, 100) == 0


@needs_nvcc
def test_planner_finds_the_shared_prefix(sa):
    w = wl.config(2)
    d = sa.dims_for(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.num_pages,
                    w.max_pages_per_seq, w.total_q, 1)
    skip, slots, runs, tiles = sa.plan_analyze(d, w.block_table, w.seq_lens, w.q_lens, 148)
    assert runs == 1
    assert (skip == 16).all()                 # the 16 shared prefix pages
    assert (slots == slots[0]).all() and slots[0] >= 1
    assert tiles >= 148 // 2


@needs_nvcc
def test_planner_nested_runs_and_no_sharing(sa):
    P = wl.PAGE_SIZE
    # 40 sequences share pages 0-1; the first 20 of them also share page 2
    B = 40
    bt = np.full((B, 5), -1, np.int32)
    for b in range(B):
        bt[b, 0], bt[b, 1] = 0, 1
        bt[b, 2] = 2 if b < 20 else 3 + b
        bt[b, 3] = 100 + b
    seq = np.full(B, 3 * P + 10, np.int32)
    ql = np.ones(B, np.int32)
    d = sa.dims_for(B, 8, 2, 200, 5, B, 1)
    skip, slots, runs, _ = sa.plan_analyze(d, bt, seq, ql, 148)
    assert runs == 2
    assert (skip[:20] == 3).all() and (skip[20:] == 2).all()
    assert (slots[:20] > slots[20:].max()).all()
    # distinct pages everywhere: nothing shared
    w = wl.config(1)
    d = sa.dims_for(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.num_pages,
                    w.max_pages_per_seq, w.total_q, 1)
    skip, slots, runs, tiles = sa.plan_analyze(d, w.block_table, w.seq_lens, w.q_lens, 148)
    assert runs == 0 and tiles == 0 and (skip == 0).all()


@needs_nvcc
def test_planner_keeps_small_groups_on_the_split_path(sa):
    P = wl.PAGE_SIZE
    bt = np.array([[0, 1], [0, 2]], np.int32)     # two sequences, G=4: 8 rows < threshold
    d = sa.dims_for(2, 8, 2, 4, 2, 2, 1)
    skip, _, runs, tiles = sa.plan_analyze(d, bt, np.array([P + 3, P + 9], np.int32),
                                           np.ones(2, np.int32), 148)
    assert runs == 0 and tiles == 0 and (skip == 0).all()


@needs_nvcc
@pytest.mark.parametrize("seed,shared", [(0, 0), (1, 3), (2, 1)])
def test_defrag_planner_matches_oracle_without_gpu(sa, seed, shared):
    """The library's host planner gives exactly the oracle's compaction."""
    import oracle
    w = wl.random_case(900 + seed, num_seqs=7, Hq=4, Hkv=2, max_ctx=2000, q_len_choices=(1, 6),
                       num_pages=80, shared_prefix_pages=shared)
    d = sa.dims_for(w.num_seqs, 4, 2, w.num_pages, w.max_pages_per_seq, w.total_q, 6)
    new, moves, L = sa.defrag_moves(d, w.block_table, w.seq_lens)
    new_o, moves_o, L_o = oracle.defrag_plan(w.block_table, w.seq_lens, w.num_pages)
    assert L == L_o and np.array_equal(new, new_o) and np.array_equal(moves, moves_o)


@needs_nvcc
def test_defrag_planner_rejects_bad_tables(sa):
    d = sa.dims_for(1, 4, 2, 4, 2, 1, 1)
    with pytest.raises(sa.SpecAttnError):
        sa.defrag_moves(d, np.array([[0, 5]], np.int32), np.array([300], np.int32))
    with pytest.raises(sa.SpecAttnError):
        sa.defrag_moves(d, np.array([[0, 1]], np.int32), np.array([513], np.int32))
    lib = sa.load_library()
    assert lib.sa_defrag_apply(ctypes.byref(d), None, None, None, -1, None, None) == 1
    assert lib.sa_defrag_apply(ctypes.byref(d), None, None, None, 0, None, None) == 0
    # byte pools: page size must be a positive multiple of 16
    assert lib.sa_defrag_apply_bytes(4, 24, None, None, None, 1, None, None) == 1
    assert lib.sa_defrag_apply_bytes(4, 0, None, None, None, 0, None, None) == 1
    assert lib.sa_defrag_apply_bytes(4, 2048, None, None, None, 0, None, None) == 0
    assert lib.sa_defrag_apply_bytes(4, 2048, None, None, None, 1, None, None) == 1
