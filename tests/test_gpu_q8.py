"""int8 K/V pages on the GPU against the oracle: the append's codes and
scales bit-exact, attention over int8 pages within the attention tolerance
(the oracle attends the same code * scale values in fp64)."""
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


def q8_pools(w):
    kc, ks = oracle.quantize_q8(w.k_pages)
    vc, vs = oracle.quantize_q8(w.v_pages)
    return kc, vc, ks, vs


def run_q8(w, append=True):
    """kv_append_q8 (optional) then paged_attn_q8 on the GPU from pools the
    oracle quantised; returns (out bits, err, pools after the call)."""
    d = dims_of(w)
    kc, vc, ks, vs = (dev_tensor(a) for a in q8_pools(w))
    bt, sl, ql = dev_tensor(w.block_table), dev_tensor(w.seq_lens), dev_tensor(w.q_lens)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if append:
        sa.kv_append_q8(d, dev_tensor(w.k_new), dev_tensor(w.v_new), kc, vc, ks, vs, bt, sl, ql, err_flag=err)
    ws = torch.zeros(sa.paged_attn_workspace_size(d), dtype=torch.uint8, device="cuda")
    q = dev_tensor(w.q)
    out = torch.zeros_like(q)
    sa.paged_attn_q8(d, q, kc, vc, ks, vs, bt, sl, ql, w.scale, out, ws, err_flag=err)
    torch.cuda.synchronize()
    return (out.cpu().numpy().view(np.uint16), int(err.item()),
            tuple(t.cpu().numpy() for t in (kc, vc, ks, vs)))


def oracle_q8(w, append=True):
    pools = q8_pools(w)
    if append:
        pools = oracle.kv_append_q8(*pools, w.k_new, w.v_new, w.block_table, w.pos_start, w.q_lens)
    kc, vc, ks, vs = pools
    return oracle.attention_rows_q8(w.q, kc, vc, ks, vs, w.block_table, w.seq_lens, w.q_lens, w.scale), pools


@pytest.mark.parametrize("seed", range(6))
def test_q8_random_small_cases(seed):
    rng = np.random.default_rng(seed)
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4]))
    w = wl.random_case(300 + seed, num_seqs=int(rng.integers(1, 6)), Hq=G * Hkv, Hkv=Hkv,
                       max_ctx=int(rng.choice([40, 300, 1300])), q_len_choices=(0, 1, 2, 3))
    out, err, pools = run_q8(w)
    ref, ref_pools = oracle_q8(w)
    assert err == 0
    for got, exp in zip(pools, ref_pools):  # the append's codes and scales, bit for bit
        assert np.array_equal(got.view(exp.dtype) if got.dtype != exp.dtype else got, exp)
    assert_attention_close(out, ref, f"seed {seed}")


def test_q8_llama3_decode_batch_all_rows():
    """The Llama3-8B-shaped decode batch (64 sequences, 32q/8kv) over int8 pages."""
    w = wl.config(1)
    out, err, _ = run_q8(w)
    ref, _ = oracle_q8(w)
    assert err == 0
    assert_attention_close(out, ref, "decode q8")


def test_q8_verify_batch_all_rows():
    """The speculative-verification batch (16 sequences, contexts 2048-8192,
    q_len 6 causal, 32q/8kv: 24 query rows per KV head, two blocks of 16)
    over int8 pages, every row against the oracle."""
    w = wl.config(3)
    out, err, _ = run_q8(w)
    ref, _ = oracle_q8(w)
    assert err == 0
    assert_attention_close(out, ref, "verify q8")


@pytest.mark.parametrize("G,q_choices", [(8, (1,)), (4, (1, 2, 3)), (2, (1, 4, 7)), (1, (1, 2, 4))])
def test_q8_persistent_kernel_row_blocks(G, q_choices):
    """Fewer than 16 query rows per KV head take the persistent kernel with 4,
    8 or 16 rows per segment; long contexts over few segments, so every
    segment is cut between many CTAs and merged across them."""
    w = wl.random_case(380 + G, num_seqs=3, Hq=2 * G, Hkv=2, max_ctx=3000, q_len_choices=q_choices)
    assert G * int(w.q_lens.max()) < 16
    out, err, _ = run_q8(w)
    assert err == 0
    ref, _ = oracle_q8(w)
    assert_attention_close(out, ref, f"G={G} q_lens={w.q_lens.tolist()}")


@pytest.mark.parametrize("seed", range(4))
def test_q8_many_rows_per_kv_head(seed):
    """Blocks of 16 query rows: G x q_len from 10 to 128 rows per KV head,
    causal inside the new tokens, random lengths and tables."""
    rng = np.random.default_rng(70 + seed)
    G = int(rng.choice([2, 4, 8]))
    Hkv = int(rng.choice([1, 2]))
    q_choices = {2: (5, 16, 33), 4: (3, 6, 17), 8: (2, 6, 16)}[G]
    w = wl.random_case(360 + seed, num_seqs=int(rng.integers(1, 5)), Hq=G * Hkv, Hkv=Hkv,
                       max_ctx=int(rng.choice([300, 1300])), q_len_choices=(1,) + q_choices)
    out, err, _ = run_q8(w)
    ref, _ = oracle_q8(w)
    assert err == 0
    assert_attention_close(out, ref, f"seed {seed}")


def test_q8_rejects_more_than_128_rows_per_kv_head():
    w = wl.random_case(310, num_seqs=2, Hq=8, Hkv=2, max_ctx=300, q_len_choices=(33,))  # 132 rows per KV head
    with pytest.raises(sa.SpecAttnError):
        run_q8(w, append=False)


@pytest.mark.parametrize("seed,Hkv", [(0, 2), (1, 8)])
def test_q8_defrag_codes_and_scales(seed, Hkv):
    """Compaction of int8 pools: the code pools and the scale pools (pages of
    Hkv*256*128 and Hkv*256*4 bytes, the latter not a whole 32 KiB chunk) move
    by one plan; pools bit-exact against the oracle's page moves, attention
    through the new tables bit-identical to attention before."""
    w = wl.random_case(1300 + seed, num_seqs=5, Hq=4 * Hkv, Hkv=Hkv, max_ctx=1500, q_len_choices=(1, 2),
                       num_pages=80, shared_prefix_pages=2 * seed)
    d = dims_of(w)
    new, moves, _ = sa.defrag_moves(d, w.block_table, w.seq_lens)
    assert len(moves) > 0
    kc, vc, ks, vs = q8_pools(w)
    g = [dev_tensor(a) for a in (kc, vc, ks, vs)]
    mv = torch.from_numpy(np.ascontiguousarray(moves, np.int32).reshape(-1, 2)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    npg = kc.shape[0]
    sa.defrag_apply_bytes(npg, kc[0].nbytes, g[0], g[1], mv, len(moves), err_flag=err)
    sa.defrag_apply_bytes(npg, ks[0].nbytes, g[2], g[3], mv, len(moves), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = [t.cpu().numpy() for t in g]
    u16 = lambda a: a.view(np.uint16).reshape(npg, -1)  # the oracle moves pages of 16-bit words
    kc2, vc2 = oracle.defrag_move(u16(kc), u16(vc), moves)
    ks2, vs2 = oracle.defrag_move(u16(ks), u16(vs), moves)
    for a, b in zip(got, (kc2, vc2, ks2, vs2)):
        assert np.array_equal(u16(a), b)
    before, e0, _ = run_q8(w, append=False)

    # attention from the moved pools through the new tables
    bt, sl, ql = dev_tensor(new), dev_tensor(w.seq_lens), dev_tensor(w.q_lens)
    ws = torch.zeros(sa.paged_attn_workspace_size(d), dtype=torch.uint8, device="cuda")
    q = dev_tensor(w.q)
    out = torch.zeros_like(q)
    sa.paged_attn_q8(d, q, g[0], g[1], g[2], g[3], bt, sl, ql, w.scale, out, ws, err_flag=err)
    torch.cuda.synchronize()
    assert e0 == 0 and int(err.item()) == 0
    assert np.array_equal(before, out.cpu().numpy().view(np.uint16))


def test_q8_out_of_range_page_sets_the_flag():
    w = wl.random_case(341, num_seqs=3, Hq=4, Hkv=2, max_ctx=600, q_len_choices=(1,))
    w.block_table = w.block_table.copy()
    w.block_table[1, 0] = w.num_pages + 5
    _, err, _ = run_q8(w, append=False)
    assert err & (1 << 3)
