"""GPU parity of kv_append + paged_attn against the fp64 CPU oracle.

Tolerance (bf16 inputs, fp32 accumulation, bf16 output): max |err| <= 2e-2
and mean |err| <= 2e-3 against the oracle's fp64 result. kv_append is a byte
copy and must match bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_path import (assert_attention_close, dev_tensor, dims_of, oracle_attention,
                      run_attention)
import speculative_decode_gb300 as sa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_gb300 import build
    build.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_config_parity_all_rows(cfg):
    """The five workloads at full size, every output row against the oracle."""
    w = wl.config(cfg)
    out, err, _, _ = run_attention(w)
    assert err == 0
    assert_attention_close(out, oracle_attention(w), f"config {cfg}")


@pytest.mark.parametrize("seed", range(12))
def test_random_small_cases(seed):
    rng = np.random.default_rng(seed)
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8]))
    w = wl.random_case(100 + seed, num_seqs=int(rng.integers(1, 7)), Hq=G * Hkv, Hkv=Hkv,
                       max_ctx=int(rng.choice([40, 300, 1300])),
                       q_len_choices=(0, 1, 2, 3, 6, 16))
    out, err, _, _ = run_attention(w)
    assert err == 0
    assert_attention_close(out, oracle_attention(w), f"seed {seed}")


@pytest.mark.parametrize("seed,G,q_choices", [(0, 4, (64, 200)), (1, 1, (17, 300)), (2, 8, (33, 128)),
                                              (3, 4, (1, 6, 512))])
def test_prefill_chunks(seed, G, q_choices):
    """Long blocks of new tokens (prefill chunks through the pages, causal
    inside the chunk; the tensor cores take them), appended then attended,
    every row against the oracle; the last case mixes decode, verify and
    prefill rows in one call."""
    Hkv = 2
    w = wl.random_case(1500 + seed, num_seqs=3, Hq=G * Hkv, Hkv=Hkv, max_ctx=1400, q_len_choices=q_choices)
    out, err, _, _ = run_attention(w)
    assert err == 0
    assert_attention_close(out, oracle_attention(w), f"seed {seed}")


def test_prefill_chunk_workload_sampled_rows():
    """The chunked-prefill workload the benchmark times, at full size (8
    sequences, 3584 cached + 512 new tokens, 32q/8kv): every chunk's first and
    last rows and 512 random rows against the oracle."""
    w = wl.prefill_chunk()
    out, err, _, _ = run_attention(w)
    assert err == 0
    rng = np.random.default_rng(5)
    starts = np.concatenate([[0], np.cumsum(w.q_lens)[:-1]])
    tok = np.concatenate([rng.integers(0, w.total_q, 512), starts, starts + w.q_lens - 1]).astype(np.int64)
    hd = rng.integers(0, w.num_q_heads, len(tok)).astype(np.int32)
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.pos_start, w.q_lens)
    ref = oracle.attention_rows(w.q, kp, vp, w.block_table, w.seq_lens, w.q_lens, w.scale, tok, hd)
    assert_attention_close(out[tok, hd], ref, "prefill chunk")


@pytest.mark.parametrize("chunk,waves", [(256, True), (264, False)])
def test_uniform_prefill_batch_all_rows(chunk, waves):
    """A batch of equal sequences with enough row tiles for whole-segment
    waves on the tensor cores (20 sequences x 2 KV heads x 8 row tiles of 128
    = 320 segments for 152 CTAs: one wave attended whole, written by the
    tensor-core kernel, the rest cut evenly and merged by the combine pass);
    with 264 new tokens the last row tile of each segment holds 32 rows and
    the batch takes the plain cut instead. Every row against the oracle."""
    w = wl.prefill_chunk(seed=1150 + chunk, num_seqs=20, cached=300, chunk=chunk, Hq=8, Hkv=2)
    rows = 4 * chunk
    assert (rows - (rows - 1) // 128 * 128 > 32) == waves
    out, err, _, _ = run_attention(w)
    assert err == 0
    assert_attention_close(out, oracle_attention(w), f"chunk {chunk}")


def test_kv_append_bit_exact():
    w = wl.random_case(31, num_seqs=5, Hq=8, Hkv=4, max_ctx=900, q_len_choices=(0, 1, 5, 16))
    _, err, kp, vp = run_attention(w)
    kref, vref = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                                  w.pos_start, w.q_lens)
    assert err == 0
    assert np.array_equal(kp, kref) and np.array_equal(vp, vref)


def test_whole_sequence_is_new_and_single_token_context():
    """q_len == seq_len (every key is a new token) and seq_len == 1."""
    w = wl.random_case(41, num_seqs=3, Hq=4, Hkv=2, max_ctx=16, q_len_choices=(16,))
    w.seq_lens = w.q_lens.copy()
    w.seq_lens[1] = 1
    w.q_lens[1] = 1
    w.q = w.q[: int(w.q_lens.sum())]
    w.k_new = w.k_new[: int(w.q_lens.sum())]
    w.v_new = w.v_new[: int(w.q_lens.sum())]
    out, err, _, _ = run_attention(w)
    assert err == 0
    assert_attention_close(out, oracle_attention(w), "q_len == seq_len")


def test_long_sequence_many_splits_and_ragged_tail():
    w = wl.random_case(43, num_seqs=2, Hq=8, Hkv=1, max_ctx=9000, q_len_choices=(1, 6))
    out, err, _, _ = run_attention(w)
    assert err == 0
    assert_attention_close(out, oracle_attention(w), "long")


def test_repeated_calls_identical():
    w = wl.config(0)
    a, _, _, _ = run_attention(w, reps=1)
    b, _, _, _ = run_attention(w, reps=3)
    assert np.array_equal(a, b)


def test_declared_max_q_len_above_actual():
    w = wl.random_case(47, num_seqs=4, Hq=8, Hkv=2, max_ctx=700, q_len_choices=(1, 2))
    out, err, _, _ = run_attention(w, max_q_len=16)
    assert err == 0
    assert_attention_close(out, oracle_attention(w), "max_q_len 16")


def test_out_of_range_page_sets_the_flag():
    w = wl.random_case(51, num_seqs=3, Hq=4, Hkv=2, max_ctx=600, q_len_choices=(1,))
    w.block_table = w.block_table.copy()
    w.block_table[1, 0] = w.num_pages + 5
    _, err, _, _ = run_attention(w, append=False)
    assert err & (1 << 3)


def test_q_len_above_seq_len_sets_the_flag():
    w = wl.random_case(52, num_seqs=3, Hq=4, Hkv=2, max_ctx=600, q_len_choices=(2,))
    w.seq_lens = w.seq_lens.copy()
    w.seq_lens[2] = 1
    _, err, _, _ = run_attention(w, append=False)
    assert err & (1 << 7)


def test_output_canary_untouched():
    w = wl.config(0)
    d = dims_of(w)
    q = dev_tensor(w.q)
    out = torch.full((w.total_q + 4, w.num_q_heads, 128), 0x1234, dtype=torch.int16, device="cuda")
    ws = torch.zeros(sa.paged_attn_workspace_size(d), dtype=torch.uint8, device="cuda")
    sa.paged_attn(d, q, dev_tensor(w.k_pages), dev_tensor(w.v_pages), dev_tensor(w.block_table),
                  dev_tensor(w.seq_lens), dev_tensor(w.q_lens), w.scale, out, ws)
    torch.cuda.synchronize()
    assert bool((out[w.total_q:] == 0x1234).all())


def test_host_argument_errors():
    w = wl.config(0)
    d = dims_of(w)
    q = dev_tensor(w.q)
    out = torch.zeros_like(q)
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    args = (q, dev_tensor(w.k_pages), dev_tensor(w.v_pages), dev_tensor(w.block_table),
            dev_tensor(w.seq_lens), dev_tensor(w.q_lens), w.scale, out)
    with pytest.raises(sa.SpecAttnError) as e:
        sa.paged_attn(d, *args, small)
    assert e.value.code == 6
    bad = dims_of(w)
    bad.head_dim = 64
    with pytest.raises(sa.SpecAttnError) as e:
        sa.paged_attn(bad, *args, small)
    assert e.value.code == 2


# ------------------------------------------------- shared prefix on tensor cores
def _plan_stats(w):
    return sa.Plan(dims_of(w), w.block_table, w.seq_lens, w.q_lens).stats()


@pytest.mark.parametrize("seed,nseq,prefix,qlens", [
    (61, 24, 1, (1,)),          # one shared page, one 128-row tile per KV head
    (62, 40, 3, (1, 6)),        # causal verify rows inside the shared run
    (63, 70, 2, (1, 2)),        # two 128-row tiles per KV head
])
def test_shared_prefix_runs_match_the_oracle(seed, nseq, prefix, qlens):
    w = wl.random_case(seed, num_seqs=nseq, Hq=8, Hkv=2, max_ctx=400, q_len_choices=qlens,
                       shared_prefix_pages=prefix)
    assert _plan_stats(w)["runs"] >= 1
    # no kv_append here: new tokens of short sequences would land in shared pages
    out, err, _, _ = run_attention(w, use_plan=True, append=False)
    assert err == 0
    assert_attention_close(out, oracle_attention(w, append=False), f"shared prefix seed {seed}")


def test_dedup_config_with_plan_all_rows():
    w = wl.config(2)
    st = _plan_stats(w)
    assert st["runs"] == 1 and st["members"] == 100 and st["pages"] == 16
    out, err, _, _ = run_attention(w, use_plan=True)
    assert err == 0
    assert_attention_close(out, oracle_attention(w), "dedup with plan")
    plain, _, _, _ = run_attention(w, use_plan=False)
    assert_attention_close(plain, oracle_attention(w), "dedup without plan")


def test_sequences_made_only_of_shared_pages():
    """Members whose whole context is the shared run: the split kernel has no
    keys left for them and only merges the tensor-core partials."""
    w = wl.random_case(64, num_seqs=36, Hq=4, Hkv=1, max_ctx=300, q_len_choices=(1,),
                       shared_prefix_pages=2)
    w.seq_lens = w.seq_lens.copy()
    w.seq_lens[::3] = 2 * wl.PAGE_SIZE          # every third sequence ends with the prefix
    out, err, _, _ = run_attention(w, use_plan=True, append=False)
    assert err == 0
    assert_attention_close(out, oracle_attention(w, append=False), "prefix-only members")


def test_nested_shared_runs():
    """A prefix shared by all sequences, then a deeper page shared by half."""
    rng = np.random.default_rng(65)
    P = wl.PAGE_SIZE
    B, Hq, Hkv = 48, 8, 2
    num_pages = 3 + B + 4
    bt = np.full((B, 4), -1, np.int32)
    for b in range(B):
        bt[b, :2] = [0, 1]
        bt[b, 2] = 2 if b < B // 2 else 3 + b
        bt[b, 3] = 3 + B + (b % 4)             # partial last pages (shared by accident, not full)
    seq = (3 * P + rng.integers(1, 200, size=B)).astype(np.int32)
    ql = rng.choice([1, 3], size=B).astype(np.int32)
    tq = int(ql.sum())
    w = wl.Workload(name="nested", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128, page_size=P,
                    q=wl.normal_bf16(rng, (tq, Hq, 128)),
                    k_pages=wl.normal_bf16(rng, (num_pages, Hkv, P, 128)),
                    v_pages=wl.normal_bf16(rng, (num_pages, Hkv, P, 128)),
                    block_table=bt, seq_lens=seq, q_lens=ql, scale=0.0883883,
                    k_new=wl.normal_bf16(rng, (tq, Hkv, 128)), v_new=wl.normal_bf16(rng, (tq, Hkv, 128)))
    assert _plan_stats(w)["runs"] == 2
    out, err, _, _ = run_attention(w, use_plan=True, append=False)
    assert err == 0
    assert_attention_close(out, oracle_attention(w, append=False), "nested runs")


def test_shared_run_of_interleaved_sequences():
    """Every other sequence shares the prefix: the run's query rows are not
    consecutive tokens, so they are copied row by row instead of loaded as
    one box (the other plan tests have consecutive members)."""
    rng = np.random.default_rng(66)
    P = wl.PAGE_SIZE
    B, Hq, Hkv = 64, 8, 2
    num_pages = 2 + 3 * B
    bt = np.full((B, 3), -1, np.int32)
    for b in range(B):
        own = 2 + 3 * b
        bt[b, :2] = [0, 1] if b % 2 == 0 else [own, own + 1]
        bt[b, 2] = own + 2
    seq = (2 * P + rng.integers(1, 200, size=B)).astype(np.int32)
    ql = np.ones(B, np.int32)
    w = wl.Workload(name="interleaved", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128, page_size=P,
                    q=wl.normal_bf16(rng, (B, Hq, 128)),
                    k_pages=wl.normal_bf16(rng, (num_pages, Hkv, P, 128)),
                    v_pages=wl.normal_bf16(rng, (num_pages, Hkv, P, 128)),
                    block_table=bt, seq_lens=seq, q_lens=ql, scale=0.0883883,
                    k_new=wl.normal_bf16(rng, (B, Hkv, 128)), v_new=wl.normal_bf16(rng, (B, Hkv, 128)))
    st = _plan_stats(w)
    assert st["runs"] == 1 and st["members"] == B // 2
    out, err, _, _ = run_attention(w, use_plan=True, append=False)
    assert err == 0
    assert_attention_close(out, oracle_attention(w, append=False), "interleaved members")


# ----------------------------------- multi-query rows on tensor cores (no plan)
@pytest.mark.parametrize("seed,G,Hkv,qlens,max_ctx", [
    (71, 4, 2, (6,), 3000),          # 24 rows per KV head: the verify shape
    (72, 8, 1, (1, 6), 2500),        # mixed: q_len 1 rows on the split kernel, q_len 6 on tensor cores
    (73, 16, 2, (16,), 700),         # 256 rows per KV head: two 128-row tiles
    (74, 4, 4, (4, 5, 16), 129),     # short contexts: partial 128-key tiles past the end
])
def test_multi_query_rows_on_tensor_cores(seed, G, Hkv, qlens, max_ctx):
    w = wl.random_case(seed, num_seqs=5, Hq=G * Hkv, Hkv=Hkv, max_ctx=max_ctx, q_len_choices=qlens)
    d = dims_of(w)
    assert sa.paged_attn_kernel_count(d) == 3      # tensor-core sequence pass, split pass, combine pass
    out, err, _, _ = run_attention(w)
    assert err == 0
    assert_attention_close(out, oracle_attention(w), f"multi-query seed {seed}")


def test_tensor_core_pieces_with_mixed_row_counts():
    """Sequences of 24 rows (four row copies) and 64 rows (one copy) per KV
    head on the tensor cores: persistent CTAs walk pieces of both kinds."""
    w = wl.random_case(75, num_seqs=8, Hq=8, Hkv=2, max_ctx=1500, q_len_choices=(6, 16))
    assert sa.paged_attn_kernel_count(dims_of(w)) == 3
    out, err, _, _ = run_attention(w)
    assert err == 0
    assert_attention_close(out, oracle_attention(w), "mixed tensor-core row counts")


def test_tensor_core_many_short_segments():
    """Many short verify sequences between decode ones: a CTA's range holds
    many tensor-core segments and skips the sequences that are not its."""
    w = wl.random_case(76, num_seqs=40, Hq=16, Hkv=2, max_ctx=200, q_len_choices=(1, 6))
    out, err, _, _ = run_attention(w)
    assert err == 0
    assert_attention_close(out, oracle_attention(w), "short tensor-core segments")
