"""CPU fp64 oracle -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package; the product library never does. It wraps
``oracle.c`` (plain C, double precision) with numpy marshalling and builds
it with gcc on first use. See ``oracle.c`` for the definitions and the
passages of the pages each one follows.

Every function here is pinned by ``tests/test_oracle.py`` against closed
forms, invariants, brute force on tiny inputs, library routines and the
hand-worked cases under ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None

ERR_ARG, ERR_PAGE_OOB, ERR_NOMEM = 1, 3, 7


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (gcc, OpenMP, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if force or not fresh:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                        "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = D
        lib.oracle_kv_append.argtypes = [I] * 6 + [P] * 7
        lib.oracle_kv_append.restype = I
        lib.oracle_attention_rows.argtypes = [I] * 7 + [P] * 6 + [D, P, P, I64, P, I]
        lib.oracle_attention_rows.restype = I
        lib.oracle_paged_attention.argtypes = [I] * 7 + [P] * 6 + [D, P, I]
        lib.oracle_paged_attention.restype = I
        lib.oracle_argmax.argtypes = [P, I64]
        lib.oracle_argmax.restype = I64
        lib.oracle_verify_greedy.argtypes = [P, P, P, I, I, I64, P, P, P]
        lib.oracle_verify_greedy.restype = I
        lib.oracle_spec_advance.argtypes = [I, I, P, P, P, P, P, P]
        lib.oracle_spec_advance.restype = I
        lib.oracle_quantize_q8.argtypes = [P, I64, I, P, P]
        lib.oracle_quantize_q8.restype = I
        lib.oracle_kv_append_q8.argtypes = [I] * 6 + [P] * 9
        lib.oracle_kv_append_q8.restype = I
        lib.oracle_attention_rows_q8.argtypes = [I] * 7 + [P] * 8 + [D, P, P, I64, P, I]
        lib.oracle_attention_rows_q8.restype = I
        lib.oracle_quantize_q4.argtypes = [P, I64, I, P, P]
        lib.oracle_quantize_q4.restype = I
        lib.oracle_kv_append_q4.argtypes = [I] * 6 + [P] * 9
        lib.oracle_kv_append_q4.restype = I
        lib.oracle_attention_rows_q4.argtypes = [I] * 7 + [P] * 8 + [D, P, P, I64, P, I]
        lib.oracle_attention_rows_q4.restype = I
        lib.oracle_defrag_plan.argtypes = [I] * 4 + [P] * 6
        lib.oracle_defrag_plan.restype = I
        lib.oracle_defrag_move.argtypes = [I, I64, P, P, P, I]
        lib.oracle_defrag_move.restype = I
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = I
        _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise OracleError(f"{what}: oracle error code {rc}")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def bf16_to_f64(bits: int) -> float:
    return float(_load().oracle_bf16_to_f64(ctypes.c_uint16(bits)))


def kv_append(k_pages, v_pages, k_new, v_new, block_table, pos_start, new_lens, page_size=256):
    """Return copies of k_pages/v_pages with the new tokens' rows written."""
    kp, vp = _c(k_pages, np.uint16).copy(), _c(v_pages, np.uint16).copy()
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    bt, ps, nl = _c(block_table, np.int32), _c(pos_start, np.int32), _c(new_lens, np.int32)
    num_pages, hkv, P, d = kp.shape
    rc = _load().oracle_kv_append(len(nl), hkv, d, P, num_pages, bt.shape[1], _ptr(kn), _ptr(vn),
                                  _ptr(kp), _ptr(vp), _ptr(bt), _ptr(ps), _ptr(nl))
    _check(rc, "kv_append")
    return kp, vp


def _attn_common(q, k_pages, v_pages, block_table, seq_lens, q_lens):
    q, kp, vp = _c(q, np.uint16), _c(k_pages, np.uint16), _c(v_pages, np.uint16)
    bt, sl, ql = _c(block_table, np.int32), _c(seq_lens, np.int32), _c(q_lens, np.int32)
    num_pages, hkv, P, d = kp.shape
    hq = q.shape[1]
    dims = (len(sl), hq, hkv, d, P, num_pages, bt.shape[1])
    return dims, (q, kp, vp, bt, sl, ql)


def paged_attention(q, k_pages, v_pages, block_table, seq_lens, q_lens, scale,
                    n_threads: int = 0) -> np.ndarray:
    """fp64 attention output [total_q, Hq, d] for every new query token."""
    dims, arrs = _attn_common(q, k_pages, v_pages, block_table, seq_lens, q_lens)
    out = np.empty((arrs[0].shape[0], dims[1], dims[3]), dtype=np.float64)
    rc = _load().oracle_paged_attention(*dims, *[_ptr(a) for a in arrs], float(scale),
                                        _ptr(out), int(n_threads))
    _check(rc, "paged_attention")
    return out


def attention_rows(q, k_pages, v_pages, block_table, seq_lens, q_lens, scale,
                   tokens: Sequence[int], heads: Sequence[int], n_threads: int = 0) -> np.ndarray:
    """fp64 attention output for selected (packed query token, q head) rows: [n, d]."""
    dims, arrs = _attn_common(q, k_pages, v_pages, block_table, seq_lens, q_lens)
    tok, hd = _c(tokens, np.int64), _c(heads, np.int32)
    out = np.empty((len(tok), dims[3]), dtype=np.float64)
    rc = _load().oracle_attention_rows(*dims, *[_ptr(a) for a in arrs], float(scale), _ptr(tok),
                                       _ptr(hd), len(tok), _ptr(out), int(n_threads))
    _check(rc, "attention_rows")
    return out


def argmax(row) -> int:
    r = _c(row, np.float32)
    return int(_load().oracle_argmax(_ptr(r), r.shape[-1]))


def verify_greedy(logits, candidates, n_cand, window=None):
    """Return (accepted, next_tok, window_out or None) for every sequence."""
    lg = _c(logits, np.float32)
    B, k1, V = lg.shape
    k_max = k1 - 1
    cand = _c(candidates, np.int32).reshape(B, k_max) if k_max > 0 else np.zeros((B, 0), np.int32)
    nc = _c(n_cand, np.int32)
    acc = np.zeros(B, np.int32)
    nxt = np.zeros(B, np.int32)
    win = None if window is None else _c(window, np.int32).copy()
    rc = _load().oracle_verify_greedy(_ptr(lg), _ptr(cand), _ptr(nc), B, k_max, V, _ptr(acc),
                                      _ptr(nxt), _ptr(win))
    _check(rc, "verify_greedy")
    return acc, nxt, win


def spec_advance(k_max, n_cand, accepted, window, seq_lens, q_lens):
    """Shapes of the next verify call after a greedy accept (the assisted
    generation loop returning to its drafting step): returns (seq_lens,
    q_lens, n_cand) of that call, from this call's n_cand, accepted counts,
    windows after the adjustment, seq_lens and q_lens."""
    nc, acc, win = _c(n_cand, np.int32), _c(accepted, np.int32), _c(window, np.int32)
    sl, ql = _c(seq_lens, np.int32).copy(), _c(q_lens, np.int32).copy()
    out = np.zeros_like(nc)
    rc = _load().oracle_spec_advance(len(nc), int(k_max), _ptr(nc), _ptr(acc), _ptr(win), _ptr(sl), _ptr(ql),
                                     _ptr(out))
    _check(rc, "spec_advance")
    return sl, ql, out


def defrag_plan(block_table, seq_lens, num_pages, page_size=256):
    """Compaction of the cache: (new_table, moves [n, 2] as (from, to), n_live)."""
    bt, sl = _c(block_table, np.int32), _c(seq_lens, np.int32)
    B, max_pages = bt.shape
    new = np.empty_like(bt)
    moves = np.empty((max(num_pages, 1), 2), np.int32)
    n_moves, n_live = ctypes.c_int32(0), ctypes.c_int32(0)
    rc = _load().oracle_defrag_plan(B, page_size, num_pages, max_pages, _ptr(bt), _ptr(sl),
                                    _ptr(new), _ptr(moves), ctypes.byref(n_moves),
                                    ctypes.byref(n_live))
    _check(rc, "defrag_plan")
    return new, moves[:n_moves.value].copy(), int(n_live.value)


def defrag_move(k_pages, v_pages, moves):
    """Return copies of k_pages/v_pages with every move (from, to) made."""
    kp, vp = _c(k_pages, np.uint16).copy(), _c(v_pages, np.uint16).copy()
    mv = _c(moves, np.int32).reshape(-1, 2)
    num_pages = kp.shape[0]
    rc = _load().oracle_defrag_move(num_pages, int(np.prod(kp.shape[1:])), _ptr(kp), _ptr(vp),
                                    _ptr(mv), len(mv))
    _check(rc, "defrag_move")
    return kp, vp


def quantize_q8(x):
    """bf16 rows [..., d] -> (int8 codes [..., d], float32 scales [...])."""
    xb = _c(x, np.uint16)
    d = xb.shape[-1]
    n = xb.size // d
    codes = np.empty(xb.shape, np.int8)
    scales = np.empty(xb.shape[:-1], np.float32)
    _check(_load().oracle_quantize_q8(_ptr(xb), n, d, _ptr(codes), _ptr(scales)), "quantize_q8")
    return codes, scales


def kv_append_q8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, block_table, pos_start,
                 new_lens, page_size=256):
    """Return copies of the int8 pools with the new tokens' rows quantized and written."""
    kc, vc = _c(k_codes, np.int8).copy(), _c(v_codes, np.int8).copy()
    ks, vs = _c(k_scales, np.float32).copy(), _c(v_scales, np.float32).copy()
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    bt, ps, nl = _c(block_table, np.int32), _c(pos_start, np.int32), _c(new_lens, np.int32)
    num_pages, hkv, P, d = kc.shape
    rc = _load().oracle_kv_append_q8(len(nl), hkv, d, P, num_pages, bt.shape[1], _ptr(kn), _ptr(vn),
                                     _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(ps),
                                     _ptr(nl))
    _check(rc, "kv_append_q8")
    return kc, vc, ks, vs


def attention_rows_q8(q, k_codes, v_codes, k_scales, v_scales, block_table, seq_lens, q_lens,
                      scale, tokens=None, heads=None, n_threads: int = 0) -> np.ndarray:
    """fp64 attention over int8 pages; every row ([total_q, Hq, d]) or the
    selected (packed query token, q head) rows ([n, d])."""
    qb = _c(q, np.uint16)
    kc, vc = _c(k_codes, np.int8), _c(v_codes, np.int8)
    ks, vs = _c(k_scales, np.float32), _c(v_scales, np.float32)
    bt, sl, ql = _c(block_table, np.int32), _c(seq_lens, np.int32), _c(q_lens, np.int32)
    num_pages, hkv, P, d = kc.shape
    hq = qb.shape[1]
    full = tokens is None
    if full:
        tok = np.repeat(np.arange(qb.shape[0], dtype=np.int64), hq)
        hd = np.tile(np.arange(hq, dtype=np.int32), qb.shape[0])
    else:
        tok, hd = _c(tokens, np.int64), _c(heads, np.int32)
    out = np.empty((len(tok), d), dtype=np.float64)
    rc = _load().oracle_attention_rows_q8(len(sl), hq, hkv, d, P, num_pages, bt.shape[1], _ptr(qb),
                                          _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl),
                                          _ptr(ql), float(scale), _ptr(tok), _ptr(hd), len(tok),
                                          _ptr(out), int(n_threads))
    _check(rc, "attention_rows_q8")
    return out.reshape(qb.shape[0], hq, d) if full else out


def quantize_q4(x):
    """bf16 rows [..., d] -> (packed nibbles uint8 [..., d / 2], float32 scales [...])."""
    xb = _c(x, np.uint16)
    d = xb.shape[-1]
    n = xb.size // d
    packed = np.empty(xb.shape[:-1] + (d // 2,), np.uint8)
    scales = np.empty(xb.shape[:-1], np.float32)
    _check(_load().oracle_quantize_q4(_ptr(xb), n, d, _ptr(packed), _ptr(scales)), "quantize_q4")
    return packed, scales


def kv_append_q4(k_nib, v_nib, k_scales, v_scales, k_new, v_new, block_table, pos_start,
                 new_lens, page_size=256):
    """Return copies of the int4 pools with the new tokens' rows quantized and written."""
    kc, vc = _c(k_nib, np.uint8).copy(), _c(v_nib, np.uint8).copy()
    ks, vs = _c(k_scales, np.float32).copy(), _c(v_scales, np.float32).copy()
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    bt, ps, nl = _c(block_table, np.int32), _c(pos_start, np.int32), _c(new_lens, np.int32)
    num_pages, hkv, P, dh = kc.shape
    rc = _load().oracle_kv_append_q4(len(nl), hkv, 2 * dh, P, num_pages, bt.shape[1], _ptr(kn), _ptr(vn),
                                     _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(ps),
                                     _ptr(nl))
    _check(rc, "kv_append_q4")
    return kc, vc, ks, vs


def attention_rows_q4(q, k_nib, v_nib, k_scales, v_scales, block_table, seq_lens, q_lens,
                      scale, tokens=None, heads=None, n_threads: int = 0) -> np.ndarray:
    """fp64 attention over int4 pages (nibbles [num_pages, Hkv, P, d / 2]);
    every row ([total_q, Hq, d]) or the selected (packed query token, q head)
    rows ([n, d])."""
    qb = _c(q, np.uint16)
    kc, vc = _c(k_nib, np.uint8), _c(v_nib, np.uint8)
    ks, vs = _c(k_scales, np.float32), _c(v_scales, np.float32)
    bt, sl, ql = _c(block_table, np.int32), _c(seq_lens, np.int32), _c(q_lens, np.int32)
    num_pages, hkv, P, dh = kc.shape
    d = 2 * dh
    hq = qb.shape[1]
    full = tokens is None
    if full:
        tok = np.repeat(np.arange(qb.shape[0], dtype=np.int64), hq)
        hd = np.tile(np.arange(hq, dtype=np.int32), qb.shape[0])
    else:
        tok, hd = _c(tokens, np.int64), _c(heads, np.int32)
    out = np.empty((len(tok), d), dtype=np.float64)
    rc = _load().oracle_attention_rows_q4(len(sl), hq, hkv, d, P, num_pages, bt.shape[1], _ptr(qb),
                                          _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl),
                                          _ptr(ql), float(scale), _ptr(tok), _ptr(hd), len(tok),
                                          _ptr(out), int(n_threads))
    _check(rc, "attention_rows_q4")
    return out.reshape(qb.shape[0], hq, d) if full else out
