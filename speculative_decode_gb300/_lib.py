"""ctypes binding of libspecattn.so: argument marshalling only.

Function names follow the C ABI without the ``sa_`` prefix. Tensors are
torch tensors on the current CUDA device (bf16 data may be passed as
torch.bfloat16 or as int16/uint16 bit patterns); the stream defaults to
torch's current stream. Status codes other than SA_OK raise SpecAttnError.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from .build import LIB

STATUS = {
    0: "SA_OK", 1: "SA_ERR_ARG", 2: "SA_ERR_UNSUPPORTED", 3: "SA_ERR_PAGE_OOB",
    4: "SA_ERR_CUDA", 5: "SA_ERR_TIMEOUT", 6: "SA_ERR_WORKSPACE", 7: "SA_ERR_QLEN",
}


class SpecAttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)} ({status_string(code)})")
        self.code = code


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_seqs", "num_q_heads", "num_kv_heads", "head_dim", "page_size", "num_pages",
        "max_pages_per_seq", "total_q", "max_q_len")]


_lib = None


def library_path() -> str:
    """The library this process loads: the in-tree build."""
    return LIB


def load_library() -> ctypes.CDLL:
    """Load the built library; fails loudly when it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with speculative_decode_gb300.build.build() "
                           "(or __graft_entry__.build()); there is no fallback path")
    lib = ctypes.CDLL(path)
    P, I32, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    DP = ctypes.POINTER(Dims)
    sig = {
        "sa_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "sa_device_sm_count": ([], ctypes.c_int),
        "sa_selftest_bounded_wait": ([ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
        "sa_kv_append": ([DP] + [P] * 8 + [P], ctypes.c_int),
        "sa_plan_create": ([DP, P, P, P, ctypes.POINTER(P)], ctypes.c_int),
        "sa_plan_destroy": ([P], None),
        "sa_plan_analyze": ([DP, P, P, P, I32, P, P, P, P], ctypes.c_int),
        "sa_plan_stats": ([P, P, P, P], ctypes.c_int),
        "sa_paged_attn_workspace_size": ([DP, P], SZ),
        "sa_paged_attn": ([DP, P, P, P, P, P, P, F, P, P, P, SZ, P, P], ctypes.c_int),
        "sa_paged_attn_kernel_count": ([DP, P], ctypes.c_int),
        "sa_paged_attn_noalloc": ([DP, P, P, P, P, P, P, F, P, P, P], ctypes.c_int),
        "sa_spec_verify_workspace_size": ([I32, I32, I32], SZ),
        "sa_spec_verify_greedy": ([P, P, P, I32, I32, I32, P, P, P, P, SZ, P, P], ctypes.c_int),
        "sa_spec_verify_greedy_advance": ([P, P, P, I32, I32, I32, P, P, P, P, P, P, P, SZ, P, P], ctypes.c_int),
        "sa_kv_append_q8": ([DP] + [P] * 11, ctypes.c_int),
        "sa_paged_attn_q8": ([DP, P, P, P, P, P, P, P, P, F, P, P, SZ, P, P], ctypes.c_int),
        "sa_kv_append_q4": ([DP] + [P] * 11, ctypes.c_int),
        "sa_paged_attn_q4": ([DP, P, P, P, P, P, P, P, P, F, P, P, SZ, P, P], ctypes.c_int),
        "sa_defrag_moves": ([DP, P, P, P, P, P, P], ctypes.c_int),
        "sa_defrag_apply": ([DP, P, P, P, I32, P, P], ctypes.c_int),
        "sa_defrag_apply_bytes": ([I32, ctypes.c_int64, P, P, P, I32, P, P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().sa_status_string(int(code)).decode()


def sm_count() -> int:
    return int(load_library().sa_device_sm_count())


def selftest_bounded_wait(err_flag, stream=None) -> None:
    """sa_selftest_bounded_wait: one CTA's bounded wait on an mbarrier that
    nothing completes; sets bit 1 << SA_ERR_TIMEOUT of err_flag."""
    _check(load_library().sa_selftest_bounded_wait(_ptr(err_flag), _stream(stream)),
           "sa_selftest_bounded_wait")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise SpecAttnError(rc, what)


def dims_for(num_seqs, num_q_heads, num_kv_heads, num_pages, max_pages_per_seq, total_q,
             max_q_len, head_dim=128, page_size=256) -> Dims:
    return Dims(num_seqs, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                max_pages_per_seq, total_q, max_q_len)


def kv_append(dims: Dims, k_new, v_new, k_pages, v_pages, block_table, seq_lens, q_lens,
              err_flag=None, stream=None) -> None:
    rc = load_library().sa_kv_append(ctypes.byref(dims), _ptr(k_new), _ptr(v_new), _ptr(k_pages),
                                      _ptr(v_pages), _ptr(block_table), _ptr(seq_lens),
                                      _ptr(q_lens), _ptr(err_flag), _stream(stream))
    _check(rc, "sa_kv_append")


class Plan:
    """Shared-run plan (sa_plan_create) built from host copies of the tables."""

    def __init__(self, dims: Dims, block_table_host, seq_lens_host, q_lens_host):
        import numpy as np
        bt = np.ascontiguousarray(block_table_host, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
        ql = np.ascontiguousarray(q_lens_host, dtype=np.int32)
        self._h = ctypes.c_void_p()
        lib = load_library()
        rc = lib.sa_plan_create(ctypes.byref(dims), bt.ctypes.data, sl.ctypes.data, ql.ctypes.data,
                                ctypes.byref(self._h))
        _check(rc, "sa_plan_create")

    @property
    def handle(self) -> int:
        return self._h.value or 0

    def stats(self):
        r, m, p = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(load_library().sa_plan_stats(self._h, ctypes.byref(r), ctypes.byref(m),
                                            ctypes.byref(p)), "sa_plan_stats")
        return {"runs": r.value, "members": m.value, "pages": p.value}

    def close(self) -> None:
        if self._h.value:
            load_library().sa_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def plan_analyze(dims: Dims, block_table_host, seq_lens_host, q_lens_host, sm_count_: int):
    """Host-only dry run of the planner: (skip_pages, run_slots, num_runs, num_tiles)."""
    import numpy as np
    bt = np.ascontiguousarray(block_table_host, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
    ql = np.ascontiguousarray(q_lens_host, dtype=np.int32)
    skip = np.zeros(dims.num_seqs, np.int32)
    slots = np.zeros(dims.num_seqs, np.int32)
    runs, tiles = ctypes.c_int32(), ctypes.c_int32()
    rc = load_library().sa_plan_analyze(ctypes.byref(dims), bt.ctypes.data, sl.ctypes.data,
                                        ql.ctypes.data, int(sm_count_), skip.ctypes.data,
                                        slots.ctypes.data, ctypes.byref(runs), ctypes.byref(tiles))
    _check(rc, "sa_plan_analyze")
    return skip, slots, runs.value, tiles.value


def paged_attn_workspace_size(dims: Dims, plan: Optional[Plan] = None) -> int:
    return int(load_library().sa_paged_attn_workspace_size(ctypes.byref(dims),
                                                           plan.handle if plan else None))


def paged_attn(dims: Dims, q, k_pages, v_pages, block_table, seq_lens, q_lens, scale: float, out,
               workspace, plan: Optional[Plan] = None, err_flag=None, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size()
    rc = load_library().sa_paged_attn(ctypes.byref(dims), _ptr(q), _ptr(k_pages), _ptr(v_pages),
                                      _ptr(block_table), _ptr(seq_lens), _ptr(q_lens),
                                      float(scale), _ptr(out), plan.handle if plan else None,
                                      _ptr(workspace), nbytes, _ptr(err_flag), _stream(stream))
    _check(rc, "sa_paged_attn")


def paged_attn_noalloc(dims: Dims, q, k_pages, v_pages, block_table, seq_lens, q_lens,
                       scale: float, out, err_flag=None, stream=None) -> None:
    """sa_paged_attn_noalloc: paged attention using the library's fixed 16 MiB
    scratch, for callers that cannot allocate device memory."""
    rc = load_library().sa_paged_attn_noalloc(ctypes.byref(dims), _ptr(q), _ptr(k_pages),
                                              _ptr(v_pages), _ptr(block_table), _ptr(seq_lens),
                                              _ptr(q_lens), float(scale), _ptr(out),
                                              _ptr(err_flag), _stream(stream))
    _check(rc, "sa_paged_attn_noalloc")


def paged_attn_kernel_count(dims: Dims, plan: Optional[Plan] = None) -> int:
    return int(load_library().sa_paged_attn_kernel_count(ctypes.byref(dims),
                                                         plan.handle if plan else None))


def spec_verify_workspace_size(num_seqs: int, k_max: int, vocab: int) -> int:
    return int(load_library().sa_spec_verify_workspace_size(num_seqs, k_max, vocab))


def spec_verify_greedy(logits, candidates, n_cand, accepted, next_tok, workspace, window=None,
                       err_flag=None, stream=None) -> None:
    B, k1, V = logits.shape
    nbytes = workspace.numel() * workspace.element_size()
    rc = load_library().sa_spec_verify_greedy(_ptr(logits), _ptr(candidates), _ptr(n_cand), B,
                                              k1 - 1, V, _ptr(accepted), _ptr(next_tok),
                                              _ptr(window), _ptr(workspace), nbytes,
                                              _ptr(err_flag), _stream(stream))
    _check(rc, "sa_spec_verify_greedy")


def spec_verify_greedy_advance(logits, candidates, n_cand, accepted, next_tok, window, seq_lens, q_lens,
                               n_cand_next, workspace, err_flag=None, stream=None) -> None:
    """spec_verify_greedy plus the next verify call's lengths (window,
    seq_lens and q_lens updated in place, n_cand_next written)."""
    B, k1, V = logits.shape
    nbytes = workspace.numel() * workspace.element_size()
    rc = load_library().sa_spec_verify_greedy_advance(
        _ptr(logits), _ptr(candidates), _ptr(n_cand), B, k1 - 1, V, _ptr(accepted), _ptr(next_tok),
        _ptr(window), _ptr(seq_lens), _ptr(q_lens), _ptr(n_cand_next), _ptr(workspace), nbytes,
        _ptr(err_flag), _stream(stream))
    _check(rc, "sa_spec_verify_greedy_advance")


def defrag_moves(dims: Dims, block_table_host, seq_lens_host):
    """Host compaction plan: (new_table, moves [n, 2] as (from, to), n_live)."""
    import numpy as np
    bt = np.ascontiguousarray(block_table_host, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
    new = np.empty_like(bt)
    moves = np.empty((max(dims.num_pages, 1), 2), np.int32)
    n_moves, n_live = ctypes.c_int32(), ctypes.c_int32()
    rc = load_library().sa_defrag_moves(ctypes.byref(dims), bt.ctypes.data, sl.ctypes.data,
                                        new.ctypes.data, moves.ctypes.data, ctypes.byref(n_moves),
                                        ctypes.byref(n_live))
    _check(rc, "sa_defrag_moves")
    return new, moves[:n_moves.value].copy(), n_live.value


def defrag_apply(dims: Dims, k_pages, v_pages, moves, n_moves: int, err_flag=None, stream=None) -> None:
    """Make the moves (a device int32 [n, 2] tensor) on both page pools."""
    rc = load_library().sa_defrag_apply(ctypes.byref(dims), _ptr(k_pages), _ptr(v_pages), _ptr(moves),
                                        int(n_moves), _ptr(err_flag), _stream(stream))
    _check(rc, "sa_defrag_apply")


def kv_append_q8(dims: Dims, k_new, v_new, k_codes, v_codes, k_scales, v_scales, block_table,
                 seq_lens, q_lens, err_flag=None, stream=None) -> None:
    """kv_append into int8 pages (codes int8 [pages, Hkv, 256, 128], scales fp32 [pages, Hkv, 256])."""
    rc = load_library().sa_kv_append_q8(ctypes.byref(dims), _ptr(k_new), _ptr(v_new), _ptr(k_codes),
                                        _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(block_table),
                                        _ptr(seq_lens), _ptr(q_lens), _ptr(err_flag), _stream(stream))
    _check(rc, "sa_kv_append_q8")


def paged_attn_q8(dims: Dims, q, k_codes, v_codes, k_scales, v_scales, block_table, seq_lens, q_lens,
                  scale: float, out, workspace, err_flag=None, stream=None) -> None:
    """paged_attn over int8 pages; the workspace is paged_attn_workspace_size(dims)."""
    rc = load_library().sa_paged_attn_q8(ctypes.byref(dims), _ptr(q), _ptr(k_codes), _ptr(v_codes),
                                         _ptr(k_scales), _ptr(v_scales), _ptr(block_table),
                                         _ptr(seq_lens), _ptr(q_lens), float(scale), _ptr(out),
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _ptr(err_flag), _stream(stream))
    _check(rc, "sa_paged_attn_q8")


def kv_append_q4(dims: Dims, k_new, v_new, k_codes, v_codes, k_scales, v_scales, block_table,
                 seq_lens, q_lens, err_flag=None, stream=None) -> None:
    """kv_append into int4 pages (nibbles uint8 [pages, Hkv, 256, 64], scales fp32 [pages, Hkv, 256])."""
    rc = load_library().sa_kv_append_q4(ctypes.byref(dims), _ptr(k_new), _ptr(v_new), _ptr(k_codes),
                                        _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(block_table),
                                        _ptr(seq_lens), _ptr(q_lens), _ptr(err_flag), _stream(stream))
    _check(rc, "sa_kv_append_q4")


def paged_attn_q4(dims: Dims, q, k_codes, v_codes, k_scales, v_scales, block_table, seq_lens, q_lens,
                  scale: float, out, workspace, err_flag=None, stream=None) -> None:
    """paged_attn over int4 pages; the workspace is paged_attn_workspace_size(dims)."""
    rc = load_library().sa_paged_attn_q4(ctypes.byref(dims), _ptr(q), _ptr(k_codes), _ptr(v_codes),
                                         _ptr(k_scales), _ptr(v_scales), _ptr(block_table),
                                         _ptr(seq_lens), _ptr(q_lens), float(scale), _ptr(out),
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _ptr(err_flag), _stream(stream))
    _check(rc, "sa_paged_attn_q4")


def defrag_apply_bytes(num_pages: int, page_bytes: int, pool_a, pool_b, moves, n_moves: int,
                       err_flag=None, stream=None) -> None:
    """Make the moves on two pools paged alike (page p = bytes [p * page_bytes, (p + 1) * page_bytes))."""
    rc = load_library().sa_defrag_apply_bytes(int(num_pages), int(page_bytes), _ptr(pool_a), _ptr(pool_b),
                                              _ptr(moves), int(n_moves), _ptr(err_flag), _stream(stream))
    _check(rc, "sa_defrag_apply_bytes")
