"""int4 K/V pages on the GPU against the oracle: the append's nibbles and
scales bit-exact, attention over int4 pages within the attention tolerance
(the oracle attends the same (nibble - 8) * scale values in fp64)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decode_gb300 as sa
import workloads as wl
from gpu_path import assert_attention_close, dev_tensor, dims_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def q4_pools(w):
    kc, ks = oracle.quantize_q4(w.k_pages)
    vc, vs = oracle.quantize_q4(w.v_pages)
    return kc, vc, ks, vs


def attend_q4(w, pools, block_table=None):
    """paged_attn_q4 on the GPU over device pools; returns (out bits, err)."""
    d = dims_of(w)
    bt = dev_tensor(w.block_table if block_table is None else block_table)
    sl, ql = dev_tensor(w.seq_lens), dev_tensor(w.q_lens)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(sa.paged_attn_workspace_size(d), dtype=torch.uint8, device="cuda")
    q = dev_tensor(w.q)
    out = torch.zeros_like(q)
    sa.paged_attn_q4(d, q, *pools, bt, sl, ql, w.scale, out, ws, err_flag=err)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16), int(err.item())


def run_q4(w, append=True):
    """kv_append_q4 (optional) then paged_attn_q4 on the GPU from pools the
    oracle quantised; returns (out bits, err, pools after the call)."""
    d = dims_of(w)
    pools = [dev_tensor(a) for a in q4_pools(w)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if append:
        sa.kv_append_q4(d, dev_tensor(w.k_new), dev_tensor(w.v_new), *pools, dev_tensor(w.block_table),
                        dev_tensor(w.seq_lens), dev_tensor(w.q_lens), err_flag=err)
    out, e = attend_q4(w, pools)
    torch.cuda.synchronize()
    return out, int(err.item()) | e, tuple(t.cpu().numpy() for t in pools)


def oracle_q4(w, append=True):
    pools = q4_pools(w)
    if append:
        pools = oracle.kv_append_q4(*pools, w.k_new, w.v_new, w.block_table, w.pos_start, w.q_lens)
    kc, vc, ks, vs = pools
    return oracle.attention_rows_q4(w.q, kc, vc, ks, vs, w.block_table, w.seq_lens, w.q_lens, w.scale), pools


@pytest.mark.parametrize("seed", range(6))
def test_q4_random_small_cases(seed):
    """Random GQA ratios (1, 2, 4 query heads per KV head), context lengths
    from a few tokens to several pages and q_len 0-3: every row block size of
    the CUDA-core kernel (4, 8 and 16 rows) over int4 pages."""
    rng = np.random.default_rng(100 + seed)
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4]))
    w = wl.random_case(320 + seed, num_seqs=int(rng.integers(1, 6)), Hq=G * Hkv, Hkv=Hkv,
                       max_ctx=int(rng.choice([40, 300, 1300])), q_len_choices=(0, 1, 2, 3))
    out, err, pools = run_q4(w)
    ref, ref_pools = oracle_q4(w)
    assert err == 0
    for got, exp in zip(pools, ref_pools):  # the append's nibbles and scales, bit for bit
        assert np.array_equal(got.view(exp.dtype) if got.dtype != exp.dtype else got, exp)
    assert_attention_close(out, ref, f"seed {seed}")


def test_q4_llama3_decode_batch_all_rows():
    """The Llama3-8B-shaped decode batch (64 sequences, 32q/8kv) over int4 pages."""
    w = wl.config(1)
    out, err, _ = run_q4(w)
    ref, _ = oracle_q4(w)
    assert err == 0
    assert_attention_close(out, ref, "decode q4")


def test_q4_verify_batch_all_rows():
    """The speculative-verification batch (16 sequences, contexts 2048-8192,
    q_len 6 causal, 32q/8kv: 24 query rows per KV head, two blocks of 16)
    over int4 pages, every row against the oracle."""
    w = wl.config(3)
    out, err, _ = run_q4(w)
    ref, _ = oracle_q4(w)
    assert err == 0
    assert_attention_close(out, ref, "verify q4")


@pytest.mark.parametrize("G,q_choices", [(8, (1,)), (4, (1, 2, 3)), (2, (1, 4, 7)), (1, (1, 2, 4))])
def test_q4_persistent_kernel_row_blocks(G, q_choices):
    """Fewer than 16 query rows per KV head take the persistent kernel with 4,
    8 or 16 rows per segment; long contexts over few segments, so every
    segment is cut between many CTAs and merged across them."""
    w = wl.random_case(380 + G, num_seqs=3, Hq=2 * G, Hkv=2, max_ctx=3000, q_len_choices=q_choices)
    assert G * int(w.q_lens.max()) < 16
    out, err, _ = run_q4(w)
    assert err == 0
    ref, _ = oracle_q4(w)
    assert_attention_close(out, ref, f"G={G} q_lens={w.q_lens.tolist()}")


@pytest.mark.parametrize("seed", range(4))
def test_q4_many_rows_per_kv_head(seed):
    """Blocks of 16 query rows: G x q_len from 10 to 128 rows per KV head,
    causal inside the new tokens, random lengths and tables."""
    rng = np.random.default_rng(70 + seed)
    G = int(rng.choice([2, 4, 8]))
    Hkv = int(rng.choice([1, 2]))
    q_choices = {2: (5, 16, 33), 4: (3, 6, 17), 8: (2, 6, 16)}[G]
    w = wl.random_case(360 + seed, num_seqs=int(rng.integers(1, 5)), Hq=G * Hkv, Hkv=Hkv,
                       max_ctx=int(rng.choice([300, 1300])), q_len_choices=(1,) + q_choices)
    out, err, _ = run_q4(w)
    ref, _ = oracle_q4(w)
    assert err == 0
    assert_attention_close(out, ref, f"seed {seed}")


def test_q4_rejects_more_than_128_rows_per_kv_head():
    w = wl.random_case(310, num_seqs=2, Hq=8, Hkv=2, max_ctx=300, q_len_choices=(33,))  # 132 rows per KV head
    with pytest.raises(sa.SpecAttnError):
        run_q4(w, append=False)


def test_q4_defrag_codes_and_scales():
    """Compaction of int4 pools (code pages of Hkv*256*64 bytes, scale pages
    of Hkv*256*4): pools bit-exact against the oracle's page moves, attention
    through the new tables bit-identical to attention before."""
    w = wl.random_case(1310, num_seqs=5, Hq=16, Hkv=4, max_ctx=1500, q_len_choices=(1, 2),
                       num_pages=80, shared_prefix_pages=2)
    d = dims_of(w)
    new, moves, _ = sa.defrag_moves(d, w.block_table, w.seq_lens)
    assert len(moves) > 0
    host = q4_pools(w)
    g = [dev_tensor(a) for a in host]
    before, e0 = attend_q4(w, g)
    mv = torch.from_numpy(np.ascontiguousarray(moves, np.int32).reshape(-1, 2)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    npg = host[0].shape[0]
    sa.defrag_apply_bytes(npg, host[0][0].nbytes, g[0], g[1], mv, len(moves), err_flag=err)
    sa.defrag_apply_bytes(npg, host[2][0].nbytes, g[2], g[3], mv, len(moves), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    u16 = lambda a: a.view(np.uint16).reshape(npg, -1)  # the oracle moves pages of 16-bit words
    exp = oracle.defrag_move(u16(host[0]), u16(host[1]), moves) + oracle.defrag_move(u16(host[2]), u16(host[3]), moves)
    for t, e in zip(g, exp):
        assert np.array_equal(u16(t.cpu().numpy()), e)
    after, e1 = attend_q4(w, g, block_table=new)
    assert e0 == 0 and e1 == 0
    assert np.array_equal(before, after)


def test_q4_out_of_range_page_sets_the_flag():
    w = wl.random_case(351, num_seqs=3, Hq=4, Hkv=2, max_ctx=600, q_len_choices=(1,))
    w.block_table = w.block_table.copy()
    w.block_table[1, 0] = w.num_pages + 5
    _, err, _ = run_q4(w, append=False)
    assert err & (1 << 3)


def test_q4_repeated_calls_identical():
    """The cut of the work and every summation order are fixed: the same call
    twice gives the same bits."""
    w = wl.random_case(352, num_seqs=5, Hq=8, Hkv=2, max_ctx=1500, q_len_choices=(1, 2))
    pools = [dev_tensor(a) for a in q4_pools(w)]
    a, e0 = attend_q4(w, pools)
    b, e1 = attend_q4(w, pools)
    assert e0 == 0 and e1 == 0
    assert np.array_equal(a, b)
