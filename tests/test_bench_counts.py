"""The numerators of the benchmark's rooflines, recounted by brute force on
the CPU: the algorithmic K/V bytes of a paged_attn call (each cached
(page, slot) that some sequence's table names within its length, once, for
every KV head, K and V) and the algorithmic FLOPs (4 x head_dim per visible
key per (new token, query head) row, causal inside the new tokens)."""
import functools

import numpy as np
import pytest

import bench
import workloads as wl


@functools.lru_cache(maxsize=None)
def workload(cfg):
    """Each benchmark workload built once for this module."""
    return wl.prefill_chunk() if cfg == "prefill" else wl.config(cfg)


def brute_kv_bytes(w: wl.Workload) -> int:
    seen = np.zeros((w.num_pages, w.page_size), dtype=bool)
    for b in range(w.num_seqs):
        t = np.arange(int(w.seq_lens[b]))  # every cached position of the sequence
        seen[w.block_table[b, t // w.page_size], t % w.page_size] = True
    return int(seen.sum()) * w.num_kv_heads * w.head_dim * 2 * 2


def brute_flops(w: wl.Workload) -> int:
    rows = 0
    for b in range(w.num_seqs):
        T, n = int(w.seq_lens[b]), int(w.q_lens[b])
        rows += int((T - n + np.arange(n) + 1).sum())  # keys visible to new token i
    return 4 * w.head_dim * w.num_q_heads * rows


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_counted_kv_bytes_match_brute_force(cfg):
    w = workload(cfg)
    assert w.unique_kv_bytes() == brute_kv_bytes(w)
    extra = 2 * w.q.nbytes + w.block_table.nbytes + w.seq_lens.nbytes + w.q_lens.nbytes
    assert bench.counted_bytes(w) == brute_kv_bytes(w) + extra


def test_shared_prefix_pages_are_counted_once():
    """The dedup batch: 100 tables share their first 16 pages, so those
    4096 tokens count once, not 100 times."""
    w = workload(2)
    per_token = w.num_kv_heads * w.head_dim * 2 * 2
    naive = int(w.seq_lens.astype(np.int64).sum()) * per_token
    shared = 16 * w.page_size * per_token
    assert brute_kv_bytes(w) == naive - (w.num_seqs - 1) * shared


@pytest.mark.parametrize("seed", range(4))
def test_counts_on_random_cases_with_shared_pages(seed):
    w = wl.random_case(500 + seed, num_seqs=5, Hq=8, Hkv=2, max_ctx=900, q_len_choices=(0, 1, 4, 9),
                       shared_prefix_pages=seed % 3)
    assert w.unique_kv_bytes() == brute_kv_bytes(w)
    assert bench.attention_flops(w) == brute_flops(w)


def test_attention_flops_of_the_prefill_and_verify_workloads():
    for w in (workload("prefill"), workload(3)):
        assert bench.attention_flops(w) == brute_flops(w)


def test_decode_batch_bytes_pinned():
    """The decode batch's counted bytes (198.97 MB) are what the committed
    profiles and rooflines divide by; a change to the workload generator
    shows up here first."""
    assert bench.counted_bytes(workload(1)) == 198_968_832
