"""Seeded synthetic inputs for the paged-attention + greedy-verification path.

This module is the one piece shared by the CPU oracle's tests and the CUDA
path's tests and benchmark. It holds no arithmetic of the method itself: it
only draws random numbers, lays them out in the interface's formats and
builds block tables with a seeded page allocator.

Shapes follow the ExLlamaV2 "Dynamic Generator" page (section "Continuous
batching": fixed 256-token pages indexed by per-sequence block tables, pages
freed and refilled as jobs come and go; section "Deduplication": several
sequences indexing the same prefix pages; section "Usage": Llama3-8B with a
64k-token cache, i.e. 8 sequences of 8k or 64 of 1k) and the Hugging Face
"Assisted Generation" page (section "Assisted Generation loop": an initial
window of 5 draft tokens verified in one forward pass over k+1 positions).

Layouts (all little-endian, C-contiguous):
  q          uint16 (bf16 bits) [total_q, Hq, d]   rows packed by q_lens
  k_pages    uint16 (bf16 bits) [num_pages, Hkv, page_size, d]
  v_pages    same as k_pages
  block_table int32 [B, max_pages_per_seq]  (entries past a sequence's last
             page hold -1; they are never read)
  seq_lens   int32 [B]   tokens in the cache for each sequence, including the
             q_lens[b] new ones
  q_lens     int32 [B]   new query tokens per sequence
  k_new/v_new uint16 [total_q, Hkv, d]  K/V rows of the new tokens (written
             by kv_append at positions seq_lens[b]-q_lens[b] ...)
  logits     float32 [B, k_max + 1, V]
  candidates int32 [B, k_max]
  n_cand     int32 [B]
  window     int32 [B]
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

PAGE_SIZE = 256
HEAD_DIM = 128
LLAMA3_VOCAB = 128256


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


@dataclasses.dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    q: np.ndarray
    k_pages: np.ndarray
    v_pages: np.ndarray
    block_table: np.ndarray
    seq_lens: np.ndarray
    q_lens: np.ndarray
    scale: float
    k_new: Optional[np.ndarray] = None
    v_new: Optional[np.ndarray] = None
    logits: Optional[np.ndarray] = None
    candidates: Optional[np.ndarray] = None
    n_cand: Optional[np.ndarray] = None
    window: Optional[np.ndarray] = None
    planted_argmax: Optional[np.ndarray] = None

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def pos_start(self) -> np.ndarray:
        return (self.seq_lens - self.q_lens).astype(np.int32)

    def unique_kv_bytes(self) -> int:
        """Bytes of K and V that a call must read: each distinct (page, slot)
        counted once over the union of all sequences' valid tokens."""
        used = {}
        P = self.page_size
        for b in range(self.num_seqs):
            T = int(self.seq_lens[b])
            for j in range((T + P - 1) // P):
                pid = int(self.block_table[b, j])
                valid = min(P, T - j * P)
                used[pid] = max(used.get(pid, 0), valid)
        tokens = sum(used.values())
        return tokens * self.num_kv_heads * self.head_dim * 2 * 2


class PageAllocator:
    """Seeded free-list allocator standing in for the generator's page pool:
    pages are handed out from a shuffled free list and returned to it when a
    job ends, so later jobs fill the holes non-contiguously."""

    def __init__(self, num_pages: int, rng: np.random.Generator):
        self.free = list(rng.permutation(num_pages).tolist())

    def alloc(self, n: int) -> list:
        if n > len(self.free):
            raise RuntimeError("page pool exhausted")
        out, self.free = self.free[:n], self.free[n:]
        return out

    def release(self, pages: list) -> None:
        self.free.extend(pages)


def _pack_tables(tables: list, max_pages: Optional[int] = None) -> np.ndarray:
    width = max_pages if max_pages is not None else max(1, max(len(t) for t in tables))
    bt = np.full((len(tables), width), -1, dtype=np.int32)
    for b, t in enumerate(tables):
        bt[b, : len(t)] = t
    return bt


def _finish(name, rng, Hq, Hkv, num_pages, tables, seq_lens, q_lens, max_pages=None,
            d=HEAD_DIM, P=PAGE_SIZE) -> Workload:
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    total_q = int(q_lens.sum())
    k_pages = normal_bf16(rng, (num_pages, Hkv, P, d))
    v_pages = normal_bf16(rng, (num_pages, Hkv, P, d))
    q = normal_bf16(rng, (total_q, Hq, d))
    k_new = normal_bf16(rng, (total_q, Hkv, d))
    v_new = normal_bf16(rng, (total_q, Hkv, d))
    return Workload(name=name, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, page_size=P,
                    q=q, k_pages=k_pages, v_pages=v_pages,
                    block_table=_pack_tables(tables, max_pages), seq_lens=seq_lens,
                    q_lens=q_lens, scale=1.0 / math.sqrt(d), k_new=k_new, v_new=v_new)


def add_verify_inputs(w: Workload, rng: np.random.Generator, k_max: int, vocab: int,
                      p_match: float = 0.7, n_cand: Optional[np.ndarray] = None,
                      window: int = 5) -> Workload:
    """Verifier logits [B, k_max+1, V] ~ N(0,1) with one planted winner per row
    (a uniformly drawn token set to the row's largest draw plus 1), and draft
    candidates that equal the planted winner with probability p_match per
    position, else a uniform token different from it."""
    B = w.num_seqs
    logits = rng.standard_normal(size=(B, k_max + 1, vocab), dtype=np.float32)
    planted = rng.integers(0, vocab, size=(B, k_max + 1)).astype(np.int32)
    for b in range(B):
        for j in range(k_max + 1):
            logits[b, j, planted[b, j]] = logits[b, j].max() + np.float32(1.0)
    match = rng.random(size=(B, k_max)) < p_match
    if vocab > 1:
        other = rng.integers(0, vocab - 1, size=(B, k_max)).astype(np.int32)
        other = other + (other >= planted[:, :k_max])  # uniform over tokens != planted
    else:
        other = planted[:, :k_max].copy()             # a one-token vocabulary always matches
    cand = np.where(match, planted[:, :k_max], other).astype(np.int32)
    w.logits = logits
    w.candidates = cand
    w.n_cand = (np.full(B, k_max, dtype=np.int32) if n_cand is None
                else np.asarray(n_cand, dtype=np.int32))
    w.window = np.full(B, window, dtype=np.int32)
    w.planted_argmax = planted
    return w


def config(idx: int, seed: Optional[int] = None) -> Workload:
    """The five workloads, 0-based: 0 tiny decode, 1 Llama3-8B decode,
    2 dedup batch, 3 spec verify, 4 fragmented long context."""
    rng = np.random.default_rng(1000 + idx + 1 if seed is None else seed)
    P = PAGE_SIZE
    if idx == 0:
        seq_lens = [300, 1, 511, 700]
        alloc = PageAllocator(16, rng)
        tables = [alloc.alloc(-(-T // P)) for T in seq_lens]
        return _finish("tiny-decode-4seq-8q2kv", rng, 8, 2, 16, tables, seq_lens, [1] * 4)
    if idx == 1:
        B = 64
        seq_lens = rng.integers(512, 1025, size=B)
        alloc = PageAllocator(256, rng)
        tables = [alloc.alloc(-(-int(T) // P)) for T in seq_lens]
        return _finish("llama3-8b-decode-64seq-32q8kv-64k-cache", rng, 32, 8, 256, tables,
                       seq_lens, [1] * B, max_pages=4)
    if idx == 2:
        B = 100
        alloc = PageAllocator(256, rng)
        prefix = alloc.alloc(16)
        suffix = rng.integers(50, 301, size=B)
        tables, seq_lens = [], []
        for b in range(B):
            T = 16 * P + int(suffix[b])
            tables.append(prefix + alloc.alloc(-(-T // P) - 16))
            seq_lens.append(T)
        return _finish("dedup-100seq-4096-shared-prefix-32q8kv", rng, 32, 8, 256, tables,
                       seq_lens, [1] * B, max_pages=18)
    if idx == 3:
        B, k = 16, 5
        seq_lens = rng.integers(2048, 8193, size=B)
        alloc = PageAllocator(512, rng)
        tables = [alloc.alloc(-(-int(T) // P)) for T in seq_lens]
        w = _finish("spec-verify-16seq-qlen6-32q8kv", rng, 32, 8, 512, tables, seq_lens,
                    [k + 1] * B, max_pages=32)
        return add_verify_inputs(w, rng, k_max=k, vocab=LLAMA3_VOCAB)
    if idx == 4:
        num_pages, B = 256, 8
        alloc = PageAllocator(num_pages, rng)
        live = []
        for _ in range(200):  # seeded job churn: random allocs and frees
            if live and (rng.random() < 0.5 or len(alloc.free) < 32):
                alloc.release(live.pop(int(rng.integers(0, len(live)))))
            else:
                live.append(alloc.alloc(int(rng.integers(1, 33))))
        for pages in live:
            alloc.release(pages)
        tables = [alloc.alloc(32) for _ in range(B)]
        q_lens = rng.choice([1, 6], size=B)
        q_lens[0], q_lens[1] = 1, 6
        return _finish("fragmented-long-ctx-8x8192-64q8kv", rng, 64, 8, num_pages, tables,
                       [32 * P] * B, q_lens, max_pages=32)
    raise ValueError(f"no config {idx}")


def prefill_chunk(seed: int = 1100, num_seqs: int = 8, cached: int = 3584, chunk: int = 512,
                  Hq: int = 32, Hkv: int = 8) -> Workload:
    """Chunked prefill through the pages: every sequence has `cached` tokens
    in the cache and appends a `chunk`-token block of new tokens (causal
    inside the block), Llama3-8B-shaped heads, tables on a shuffled pool with
    spare pages."""
    rng = np.random.default_rng(seed)
    P = PAGE_SIZE
    T = cached + chunk
    per_seq = -(-T // P)
    alloc = PageAllocator(num_seqs * per_seq + 32, rng)
    tables = [alloc.alloc(per_seq) for _ in range(num_seqs)]
    return _finish(f"prefill-chunk-{num_seqs}seq-{cached}+{chunk}-{Hq}q{Hkv}kv", rng, Hq, Hkv,
                   num_seqs * per_seq + 32, tables, [T] * num_seqs, [chunk] * num_seqs, max_pages=per_seq)


def random_case(seed: int, num_seqs: int = 3, Hq: int = 4, Hkv: int = 2, max_ctx: int = 700,
                q_len_choices=(0, 1, 2, 6), num_pages: Optional[int] = None,
                shared_prefix_pages: int = 0) -> Workload:
    """Small randomized case: random context lengths, q_lens, GQA ratio and
    non-contiguous tables; optionally the first `shared_prefix_pages` entries
    of every table point at the same physical pages."""
    rng = np.random.default_rng(seed)
    P = PAGE_SIZE
    q_lens = rng.choice(q_len_choices, size=num_seqs).astype(np.int32)
    lo = shared_prefix_pages * P
    seq_lens = np.maximum(rng.integers(lo + 1, lo + max_ctx + 1, size=num_seqs), q_lens)
    need = shared_prefix_pages + sum(-(-int(T) // P) - shared_prefix_pages for T in seq_lens)
    npages = num_pages if num_pages is not None else need + 3
    alloc = PageAllocator(npages, rng)
    prefix = alloc.alloc(shared_prefix_pages)
    tables = [prefix + alloc.alloc(-(-int(T) // P) - shared_prefix_pages) for T in seq_lens]
    return _finish(f"random-{seed}", rng, Hq, Hkv, npages, tables, seq_lens, q_lens)
