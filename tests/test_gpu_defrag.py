"""Cache compaction on the GPU against the oracle: the host planner's moves,
the page-copy kernel (bit-exact pools) and attention read through the new
tables (bit-identical to attention before the compaction)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_gb300 as sa
import workloads as wl
from gpu_path import dev_tensor, dims_of, run_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def apply_on_gpu(w, moves):
    d = dims_of(w)
    kp, vp = dev_tensor(w.k_pages), dev_tensor(w.v_pages)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mv = torch.from_numpy(np.ascontiguousarray(moves, np.int32).reshape(-1, 2)).cuda()
    sa.defrag_apply(d, kp, vp, mv, len(moves), err_flag=err)
    torch.cuda.synchronize()
    return kp.cpu().numpy().view(np.uint16), vp.cpu().numpy().view(np.uint16), int(err.item())


def moved(w, new_table, kp, vp):
    """The workload read through the compacted cache."""
    import dataclasses
    return dataclasses.replace(w, block_table=new_table, k_pages=kp, v_pages=vp)


@pytest.mark.parametrize("seed,shared", [(0, 0), (1, 4)])
def test_defrag_pools_bit_exact_and_attention_unchanged(seed, shared):
    w = wl.random_case(1200 + seed, num_seqs=6, Hq=32, Hkv=8, max_ctx=1800, q_len_choices=(1, 6),
                       num_pages=96, shared_prefix_pages=shared)
    d = dims_of(w)
    new, moves, L = sa.defrag_moves(d, w.block_table, w.seq_lens)
    assert len(moves) > 0
    kp, vp, err = apply_on_gpu(w, moves)
    kref, vref = oracle.defrag_move(w.k_pages, w.v_pages, moves)
    assert err == 0
    assert np.array_equal(kp, kref) and np.array_equal(vp, vref)
    before, e0, _, _ = run_attention(w, append=False)
    after, e1, _, _ = run_attention(moved(w, new, kp, vp), append=False)
    assert e0 == 0 and e1 == 0
    assert np.array_equal(before, after)


def test_defrag_full_size_dedup_pool():
    """The dedup batch's pool (256 pages, 8 KV heads): 100 tables sharing a
    16-page prefix, suffix pages scattered over the pool."""
    w = wl.config(2)
    d = dims_of(w)
    new, moves, L = sa.defrag_moves(d, w.block_table, w.seq_lens)
    new_o, moves_o, L_o = oracle.defrag_plan(w.block_table, w.seq_lens, w.num_pages)
    assert L == L_o and np.array_equal(new, new_o) and np.array_equal(moves, moves_o)
    kp, vp, err = apply_on_gpu(w, moves)
    kref, vref = oracle.defrag_move(w.k_pages, w.v_pages, moves)
    assert err == 0 and np.array_equal(kp, kref) and np.array_equal(vp, vref)


def test_defrag_out_of_range_move_is_flagged_and_skipped():
    w = wl.random_case(1300, num_seqs=2, Hq=4, Hkv=2, max_ctx=600, q_len_choices=(1,), num_pages=12)
    moves = np.array([[w.num_pages, 0], [3, 1], [2, w.num_pages + 5]], np.int32)
    kp, vp, err = apply_on_gpu(w, moves)
    assert err & (1 << 3)  # SA_ERR_PAGE_OOB
    kref, vref = oracle.defrag_move(w.k_pages, w.v_pages, moves[1:2])
    assert np.array_equal(kp, kref) and np.array_equal(vp, vref)
