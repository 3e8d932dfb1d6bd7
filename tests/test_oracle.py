"""Pins of the CPU fp64 oracle against things other than itself.

Each test checks the oracle against a closed form, an invariant the pages
fix, brute force through a library routine on a differently built input, or
the hand-worked cases under tests/golden/. None of these run on a GPU.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "greedy_accept_cases.json")
P = wl.PAGE_SIZE


# --------------------------------------------------------------------- helpers
def dense_case(seed, seq_lens, q_lens, Hq, Hkv, d=128, extra_pages=3, scale=None):
    """Contiguous per-sequence K/V first, then scattered into randomly placed
    pages: the oracle must recover attention over the contiguous tensors."""
    rng = np.random.default_rng(seed)
    B = len(seq_lens)
    npages_seq = [-(-T // P) for T in seq_lens]
    num_pages = sum(npages_seq) + extra_pages
    perm = rng.permutation(num_pages)
    tables, k = [], 0
    for n in npages_seq:
        tables.append(perm[k:k + n].tolist())
        k += n
    width = max(1, max(npages_seq))
    bt = np.full((B, width), -1, np.int32)
    for b, t in enumerate(tables):
        bt[b, :len(t)] = t
    k_pages = wl.normal_bf16(rng, (num_pages, Hkv, P, d))
    v_pages = wl.normal_bf16(rng, (num_pages, Hkv, P, d))
    dense_k, dense_v = [], []
    for b, T in enumerate(seq_lens):
        kd = wl.normal_bf16(rng, (T, Hkv, d))
        vd = wl.normal_bf16(rng, (T, Hkv, d))
        for t in range(T):  # scatter token t into (page, slot)
            pg, slot = tables[b][t // P], t % P
            k_pages[pg, :, slot, :] = kd[t]
            v_pages[pg, :, slot, :] = vd[t]
        dense_k.append(kd)
        dense_v.append(vd)
    q = wl.normal_bf16(rng, (int(sum(q_lens)), Hq, d))
    sc = 1.0 / math.sqrt(d) if scale is None else scale
    return dict(q=q, k_pages=k_pages, v_pages=v_pages, block_table=bt,
                seq_lens=np.array(seq_lens, np.int32), q_lens=np.array(q_lens, np.int32),
                scale=sc), dense_k, dense_v


def run_oracle(case):
    return oracle.paged_attention(case["q"], case["k_pages"], case["v_pages"],
                                  case["block_table"], case["seq_lens"], case["q_lens"],
                                  case["scale"])


def f64(bits):
    return torch.from_numpy(wl.bf16_to_f32(bits).astype(np.float64))


# ------------------------------------------------------------ bf16 conversion
def test_bf16_conversion_is_exact_for_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(b)) for b in bits[::1]])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # the sign of zero survives
    assert math.copysign(1.0, oracle.bf16_to_f64(0x8000)) == -1.0


# ---------------------------------------------- attention vs dense brute force
@pytest.mark.parametrize("seed,seq_lens,q_lens,Hq,Hkv", [
    (1, [300, 1, 511, 700], [1, 1, 1, 1], 8, 2),
    (2, [257, 6, 1024], [6, 6, 1], 4, 4),
    (3, [40, 513], [0, 3], 6, 2),
    (4, [256, 255, 2], [2, 1, 2], 8, 1),
    (5, [700, 300], [300, 120], 4, 2),   # prefill chunks: long causal blocks of new tokens
])
def test_attention_matches_dense_sdpa(seed, seq_lens, q_lens, Hq, Hkv):
    case, dk, dv = dense_case(seed, seq_lens, q_lens, Hq, Hkv)
    got = run_oracle(case)
    G = Hq // Hkv
    row = 0
    for b, (T, n) in enumerate(zip(seq_lens, q_lens)):
        if n == 0:
            continue
        qb = f64(case["q"][row:row + n]).permute(1, 0, 2)           # [Hq, n, d]
        kb = f64(dk[b]).permute(1, 0, 2).repeat_interleave(G, 0)    # [Hq, T, d]
        vb = f64(dv[b]).permute(1, 0, 2).repeat_interleave(G, 0)
        # query i sits at position T-n+i and sees keys 0..T-n+i
        pos = torch.arange(T - n, T).unsqueeze(1)
        mask = torch.arange(T).unsqueeze(0) <= pos                  # [n, T]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qb, kb, vb, attn_mask=mask, scale=case["scale"])        # [Hq, n, d]
        ref = ref.permute(1, 0, 2).numpy()
        np.testing.assert_allclose(got[row:row + n], ref, rtol=1e-11, atol=1e-12)
        row += n
    assert row == got.shape[0]


def test_attention_rows_equal_full_call():
    case, _, _ = dense_case(5, [700, 300], [3, 2], 8, 2)
    full = run_oracle(case)
    toks = [0, 2, 3, 4, 1]
    heads = [7, 0, 5, 3, 1]
    rows = oracle.attention_rows(case["q"], case["k_pages"], case["v_pages"], case["block_table"],
                                 case["seq_lens"], case["q_lens"], case["scale"], toks, heads)
    for r, (t, h) in enumerate(zip(toks, heads)):
        assert np.array_equal(rows[r], full[t, h])


# ------------------------------------------------------------------ invariants
def test_page_permutation_invariance_bitwise():
    case, _, _ = dense_case(6, [600, 129, 1000], [1, 4, 2], 8, 2, extra_pages=5)
    base = run_oracle(case)
    rng = np.random.default_rng(60)
    n = case["k_pages"].shape[0]
    perm = rng.permutation(n)            # new physical id of old page i is perm[i]
    kp = np.empty_like(case["k_pages"])
    vp = np.empty_like(case["v_pages"])
    kp[perm] = case["k_pages"]
    vp[perm] = case["v_pages"]
    bt = np.where(case["block_table"] >= 0, perm[np.maximum(case["block_table"], 0)], -1)
    moved = dict(case, k_pages=kp, v_pages=vp, block_table=bt.astype(np.int32))
    assert np.array_equal(run_oracle(moved), base)


def test_shared_pages_equal_duplicated_pages_bitwise():
    """Deduplication (ExLlamaV2 page, 'Deduplication'): sequences indexing the
    same prefix pages give exactly what private copies of them give."""
    rng = np.random.default_rng(7)
    Hq, Hkv, d = 8, 2, 128
    B, prefix_pages = 3, 2
    suffix = [17, 300, 1]
    seq_lens = [prefix_pages * P + s for s in suffix]
    own = [-(-T // P) - prefix_pages for T in seq_lens]
    n_shared = prefix_pages + sum(own)
    n_dup = B * prefix_pages + sum(own)
    kp_s = wl.normal_bf16(rng, (n_shared, Hkv, P, d))
    vp_s = wl.normal_bf16(rng, (n_shared, Hkv, P, d))
    bt_s = np.full((B, prefix_pages + max(own)), -1, np.int32)
    kp_d = np.zeros((n_dup, Hkv, P, d), np.uint16)
    vp_d = np.zeros_like(kp_d)
    bt_d = np.full_like(bt_s, -1)
    nxt_s, nxt_d = prefix_pages, 0
    for b in range(B):
        pages = list(range(prefix_pages)) + list(range(nxt_s, nxt_s + own[b]))
        nxt_s += own[b]
        bt_s[b, :len(pages)] = pages
        for j, pg in enumerate(pages):      # private copy of every page
            kp_d[nxt_d] = kp_s[pg]
            vp_d[nxt_d] = vp_s[pg]
            bt_d[b, j] = nxt_d
            nxt_d += 1
    q = wl.normal_bf16(rng, (B, Hq, d))
    ql = np.ones(B, np.int32)
    sl = np.array(seq_lens, np.int32)
    a = oracle.paged_attention(q, kp_s, vp_s, bt_s, sl, ql, 0.088)
    b_ = oracle.paged_attention(q, kp_d, vp_d, bt_d, sl, ql, 0.088)
    assert np.array_equal(a, b_)


def test_causal_rows_equal_single_query_calls_bitwise():
    """Row i of a q_len=n call is the q_len=1 call on the same pages with the
    context cut to T-n+1+i tokens."""
    case, _, _ = dense_case(8, [900, 300], [6, 4], 8, 2)
    full = run_oracle(case)
    row = 0
    for b in range(2):
        T, n = int(case["seq_lens"][b]), int(case["q_lens"][b])
        for i in range(n):
            sl = case["seq_lens"].copy()
            ql = np.zeros_like(case["q_lens"])
            sl[b], ql[b] = T - n + 1 + i, 1
            single = oracle.paged_attention(case["q"][row + i:row + i + 1], case["k_pages"],
                                            case["v_pages"], case["block_table"], sl, ql,
                                            case["scale"])
            assert np.array_equal(single[0], full[row + i])
        row += n


# ---------------------------------------------------------------- closed forms
def test_single_key_returns_its_value_exactly():
    case, _, dv = dense_case(9, [1, 1], [1, 1], 4, 2)
    got = run_oracle(case)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(got[b, h], wl.bf16_to_f32(dv[b][0, h // 2]).astype(np.float64))


def test_zero_scale_gives_mean_of_visible_values():
    case, _, dv = dense_case(10, [513, 40], [3, 2], 4, 2, scale=0.0)
    got = run_oracle(case)
    row = 0
    for b, (T, n) in enumerate([(513, 3), (40, 2)]):
        vals = wl.bf16_to_f32(dv[b]).astype(np.float64)             # [T, Hkv, d]
        for i in range(n):
            p = T - n + i
            mean = vals[:p + 1].mean(axis=0)
            for h in range(4):
                np.testing.assert_allclose(got[row + i, h], mean[h // 2], rtol=0, atol=1e-13)
        row += n


def test_identical_keys_give_mean_of_values():
    case, _, dv = dense_case(11, [700], [2], 4, 2)
    key = case["k_pages"][case["block_table"][0, 0], :, 5, :].copy()   # one key per KV head
    for j in range(3):
        case["k_pages"][case["block_table"][0, j]] = key[:, None, :]
    got = run_oracle(case)
    vals = wl.bf16_to_f32(dv[0]).astype(np.float64)
    for i in range(2):
        p = 700 - 2 + i
        mean = vals[:p + 1].mean(axis=0)
        for h in range(4):
            np.testing.assert_allclose(got[i, h], mean[h // 2], rtol=0, atol=1e-12)


def test_dominant_key_selects_its_value():
    case, _, dv = dense_case(12, [600], [1], 2, 1)
    q = np.zeros_like(case["q"])
    q[0, :, 0] = wl.bf16_bits(np.array([8.0], np.float32))[0]
    case["q"] = q
    pg = case["block_table"][0]
    for j in range(3):
        case["k_pages"][pg[j], 0, :, 0] = 0
    star = 431                             # the one key aligned with q
    case["k_pages"][pg[star // P], 0, star % P, 0] = wl.bf16_bits(np.array([64.0], np.float32))[0]
    case["scale"] = 1.0                    # score gap 512: every other weight < e^-512
    got = run_oracle(case)
    want = wl.bf16_to_f32(dv[0][star, 0]).astype(np.float64)
    for h in range(2):
        np.testing.assert_allclose(got[0, h], want, rtol=0, atol=1e-200)


# ----------------------------------------------------------- edges and errors
def test_zero_length_queries_and_ignored_table_tail():
    case, _, _ = dense_case(13, [300, 20], [0, 2], 4, 2)
    bt = np.concatenate([case["block_table"], np.full((2, 3), 10 ** 6, np.int32)], axis=1)
    a = run_oracle(case)
    b = run_oracle(dict(case, block_table=bt))   # entries past the last page are never read
    assert a.shape == (2, 4, 128) and np.array_equal(a, b)


def test_out_of_range_page_is_an_error():
    case, _, _ = dense_case(14, [300], [1], 4, 2)
    case["block_table"][0, 1] = case["k_pages"].shape[0]
    with pytest.raises(oracle.OracleError, match="code 3"):
        run_oracle(case)


def test_q_len_above_seq_len_is_an_error():
    case, _, _ = dense_case(15, [3], [3], 4, 2)
    case["q_lens"] = np.array([4], np.int32)
    case["q"] = np.zeros((4, 4, 128), np.uint16)
    with pytest.raises(oracle.OracleError, match="code 1"):
        run_oracle(case)


# ------------------------------------------------------------------ kv_append
def test_kv_append_writes_through_the_block_table():
    w = wl.random_case(21, num_seqs=4, Hq=4, Hkv=2, q_len_choices=(0, 1, 3, 6))
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table,
                              w.pos_start, w.q_lens)
    touched = np.zeros(w.k_pages.shape[:1] + w.k_pages.shape[2:3], bool)   # [page, slot]
    row = 0
    for b in range(w.num_seqs):
        for i in range(int(w.q_lens[b])):
            pos = int(w.pos_start[b]) + i
            pg, slot = int(w.block_table[b, pos // P]), pos % P
            assert np.array_equal(kp[pg, :, slot, :], w.k_new[row])
            assert np.array_equal(vp[pg, :, slot, :], w.v_new[row])
            touched[pg, slot] = True
            row += 1
    keep = ~touched
    assert np.array_equal(kp.transpose(0, 2, 1, 3)[keep], w.k_pages.transpose(0, 2, 1, 3)[keep])
    assert np.array_equal(vp.transpose(0, 2, 1, 3)[keep], w.v_pages.transpose(0, 2, 1, 3)[keep])


def test_kv_append_across_a_page_boundary():
    """New tokens at positions 250..261 land in slots 250..255 of the second
    table entry's page and slots 0..5 of the third's."""
    rng = np.random.default_rng(23)
    Hkv, d = 2, 128
    kp0 = wl.normal_bf16(rng, (5, Hkv, P, d))
    vp0 = wl.normal_bf16(rng, (5, Hkv, P, d))
    kn = wl.normal_bf16(rng, (12, Hkv, d))
    vn = wl.normal_bf16(rng, (12, Hkv, d))
    bt = np.array([[4, 2, 0]], np.int32)
    kp, vp = oracle.kv_append(kp0, vp0, kn, vn, bt, np.array([250 + P], np.int32),
                              np.array([12], np.int32))
    assert np.array_equal(kp[2, :, 250:, :], kn[:6].transpose(1, 0, 2))
    assert np.array_equal(kp[0, :, :6, :], kn[6:].transpose(1, 0, 2))
    assert np.array_equal(vp[0, :, :6, :], vn[6:].transpose(1, 0, 2))
    assert np.array_equal(kp[0, :, 6:, :], kp0[0, :, 6:, :])
    assert np.array_equal(kp[[1, 3, 4]], kp0[[1, 3, 4]])


def test_kv_append_out_of_range_page_is_an_error():
    w = wl.random_case(22, num_seqs=2, q_len_choices=(2,))
    bt = w.block_table.copy()
    last = int(w.seq_lens[0]) - 1
    bt[0, last // P] = -1
    with pytest.raises(oracle.OracleError, match="code 3"):
        oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, bt, w.pos_start, w.q_lens)


# ------------------------------------------------------------ argmax / verify
def _row(spec):
    conv = {"nan": np.nan, "inf": np.inf, "-inf": -np.inf}
    fill = conv.get(spec["fill"], spec["fill"]) if isinstance(spec["fill"], str) else spec["fill"]
    r = np.full(spec["V"], fill, np.float32)
    for k, v in spec["set"].items():
        r[int(k)] = conv[v] if isinstance(v, str) else v
    return r


def test_golden_accept_cases():
    data = json.load(open(GOLDEN))
    for case in data["cases"]:
        rows = np.stack([_row(s) for s in case["rows"]])[None]      # [1, k+1, V]
        exp = case["expect"]
        assert [oracle.argmax(r) for r in rows[0]] == exp["argmax"], case["note"]
        acc, nxt, win = oracle.verify_greedy(rows, np.array([case["candidates"]], np.int32),
                                             np.array([case["n_cand"]], np.int32),
                                             np.array([case["window_in"]], np.int32))
        assert (acc[0], nxt[0], win[0]) == (exp["accepted"], exp["next_tok"],
                                            exp["window_out"]), case["note"]


def test_golden_window_sequence():
    seq = json.load(open(GOLDEN))["window_sequence"]
    w = np.array([seq["start"]], np.int32)
    V = 8
    for outcome, want in zip(seq["outcomes"], seq["windows"]):
        rows = np.zeros((1, 2, V), np.float32)
        rows[0, :, 3] = 1.0
        cand = np.array([[3 if outcome == "all" else 4]], np.int32)
        _, _, w = oracle.verify_greedy(rows, cand, np.array([1], np.int32), w)
        assert int(w[0]) == want


def test_argmax_matches_numpy_first_occurrence_on_finite_rows():
    rng = np.random.default_rng(31)
    for V in (1, 2, 7, 1000, wl.LLAMA3_VOCAB):
        for _ in range(3):
            r = rng.integers(-4, 5, size=V).astype(np.float32)       # many ties
            assert oracle.argmax(r) == int(np.argmax(r))
    r = np.zeros(wl.LLAMA3_VOCAB, np.float32)
    r[-1] = 1e-30                                                    # max in the last element
    assert oracle.argmax(r) == wl.LLAMA3_VOCAB - 1


def test_verify_on_planted_rows_at_full_vocab():
    """Rows whose winner is planted by construction: the accepted count is the
    leading run of candidates equal to the planted tokens."""
    rng = np.random.default_rng(41)
    w = wl.random_case(41, num_seqs=8)
    wl.add_verify_inputs(w, rng, k_max=5, vocab=wl.LLAMA3_VOCAB,
                         n_cand=rng.integers(0, 6, size=8))
    acc, nxt, win = oracle.verify_greedy(w.logits, w.candidates, w.n_cand, w.window)
    for b in range(8):
        a = 0
        while a < w.n_cand[b] and w.candidates[b, a] == w.planted_argmax[b, a]:
            a += 1
        assert acc[b] == a and nxt[b] == w.planted_argmax[b, a]
        assert win[b] == (7 if a == w.n_cand[b] else 4)


def test_verify_rejects_n_cand_above_k_max():
    with pytest.raises(oracle.OracleError, match="code 1"):
        oracle.verify_greedy(np.zeros((1, 3, 4), np.float32), np.zeros((1, 2), np.int32),
                             np.array([3], np.int32))


# ------------------------------------------------------------ defragmentation
DEFRAG = os.path.join(os.path.dirname(__file__), "golden", "defrag_cases.json")


def test_defrag_hand_worked_cases():
    for c in json.load(open(DEFRAG))["cases"]:
        new, moves, n_live = oracle.defrag_plan(np.array(c["block_table"], np.int32),
                                                np.array(c["seq_lens"], np.int32), c["num_pages"])
        e = c["expect"]
        assert n_live == e["n_live"], c["note"]
        assert moves.tolist() == e["moves"], c["note"]
        assert new.tolist() == e["new_table"], c["note"]


@pytest.mark.parametrize("seed,shared", [(0, 0), (1, 2), (2, 0), (3, 3)])
def test_defrag_compacts_and_keeps_attention_bitwise(seed, shared):
    """Live pages end up exactly at ids 0..L-1 through one map (shared pages
    stay shared), the moves are independent, and attention read through the
    new tables over the moved pools equals attention before, bit for bit."""
    w = wl.random_case(700 + seed, num_seqs=5, Hq=4, Hkv=2, max_ctx=1300, q_len_choices=(1, 2, 6),
                       num_pages=64, shared_prefix_pages=shared)
    used = [(b, j) for b, T in enumerate(w.seq_lens) for j in range(-(-int(T) // P))]
    new, moves, L = oracle.defrag_plan(w.block_table, w.seq_lens, w.num_pages)
    pairs = {(int(w.block_table[b, j]), int(new[b, j])) for b, j in used}
    assert L == len({o for o, _ in pairs})
    assert {n for _, n in pairs} == set(range(L))
    assert len({n for _, n in pairs}) == len(pairs)          # one-to-one: shared stays shared
    assert all(o == n for o, n in pairs if o < L)             # pages below L stay
    f, t = moves[:, 0], moves[:, 1]
    assert np.all(f >= L) and np.all(t < L) and len(set(t.tolist())) == len(t)
    assert sorted(zip(f.tolist(), t.tolist())) == sorted((o, n) for o, n in pairs if o != n)
    kp, vp = oracle.defrag_move(w.k_pages, w.v_pages, moves)
    args = (w.seq_lens, w.q_lens, w.scale)
    before = oracle.paged_attention(w.q, w.k_pages, w.v_pages, w.block_table, *args)
    assert np.array_equal(before, oracle.paged_attention(w.q, kp, vp, new, *args))
    if len(moves):  # the new tables without the moves read other pages
        assert not np.array_equal(before, oracle.paged_attention(w.q, w.k_pages, w.v_pages, new, *args))


def test_defrag_rejects_bad_tables():
    bt = np.array([[0, 1]], np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.defrag_plan(np.array([[0, 5]], np.int32), np.array([300], np.int32), 4)  # page 5 of 4
    with pytest.raises(oracle.OracleError):
        oracle.defrag_plan(bt, np.array([513], np.int32), 4)  # needs 3 entries, table has 2
    new, moves, L = oracle.defrag_plan(bt, np.array([0], np.int32), 4)
    assert L == 0 and len(moves) == 0 and new.tolist() == [[-1, -1]]


# ------------------------------------------------------------------ int8 pages
Q8 = os.path.join(os.path.dirname(__file__), "golden", "q8_cases.json")


def test_q8_hand_worked_rows():
    for c in json.load(open(Q8))["cases"]:
        bits = np.array([c["bits"]], np.uint16)
        assert np.array_equal(wl.bf16_to_f32(bits)[0], np.array(c["values"], np.float32)), c["note"]
        codes, scales = oracle.quantize_q8(bits)
        assert codes[0].tolist() == c["expect"]["codes"], c["note"]
        assert abs(float(scales[0]) * 127 - c["expect"]["scale_times_127"]) <= 1e-6 * max(1.0, c["expect"]["scale_times_127"])


def test_q8_error_within_half_a_step():
    """Every value is recovered within half a quantisation step, and the
    largest magnitude of a non-zero row maps to +-127."""
    rng = np.random.default_rng(3)
    x = wl.normal_bf16(rng, (500, 128))
    x[7] = 0
    codes, scales = oracle.quantize_q8(x)
    xf = wl.bf16_to_f32(x).astype(np.float64)
    rec = codes.astype(np.float64) * scales.astype(np.float64)[:, None]
    # half a step, plus the binary32 rounding of x / scale (|x / scale| <= 127,
    # so that quotient is off by at most 127 * 2^-23 steps)
    assert np.all(np.abs(rec - xf) <= scales.astype(np.float64)[:, None] * (0.5 + 127 * 2.0 ** -23))
    nz = np.abs(xf).max(axis=1) > 0
    assert np.all(np.abs(codes[nz]).max(axis=1) == 127)
    assert scales[7] == 0 and not codes[7].any()


def test_q8_attention_is_exact_on_representable_rows():
    """Rows of integers in [-127, 127] that contain 127 quantise exactly
    (scale 1), so attention over the int8 pages equals attention over the
    bf16 pages, bit for bit."""
    rng = np.random.default_rng(11)
    w = wl.random_case(41, num_seqs=3, Hq=8, Hkv=2, max_ctx=600, q_len_choices=(1, 2))
    for pool in (w.k_pages, w.v_pages):
        ints = rng.integers(-127, 128, size=pool.shape).astype(np.float32)
        ints[..., 5] = 127
        pool[...] = (ints.view(np.uint32) >> 16).astype(np.uint16)  # integers <= 127 are exact in bf16
    kc, ks = oracle.quantize_q8(w.k_pages)
    vc, vs = oracle.quantize_q8(w.v_pages)
    assert np.all(ks == 1) and np.all(vs == 1)
    args = (w.block_table, w.seq_lens, w.q_lens, w.scale)
    ref = oracle.paged_attention(w.q, w.k_pages, w.v_pages, *args)
    assert np.array_equal(oracle.attention_rows_q8(w.q, kc, vc, ks, vs, *args), ref)


def test_kv_append_q8_quantises_the_rows_kv_append_writes():
    w = wl.random_case(42, num_seqs=4, Hq=4, Hkv=2, max_ctx=700, q_len_choices=(1, 3, 6))
    kc, ks = oracle.quantize_q8(w.k_pages)
    vc, vs = oracle.quantize_q8(w.v_pages)
    kc2, vc2, ks2, vs2 = oracle.kv_append_q8(kc, vc, ks, vs, w.k_new, w.v_new, w.block_table,
                                             w.pos_start, w.q_lens)
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.pos_start, w.q_lens)
    for got, pages in (((kc2, ks2), kp), ((vc2, vs2), vp)):
        c, s = oracle.quantize_q8(pages)
        assert np.array_equal(got[0], c) and np.array_equal(got[1], s)


# ------------------------------------------------------------------ int4 pages
Q4 = os.path.join(os.path.dirname(__file__), "golden", "q4_cases.json")


def q4_values(packed, scales):
    """Decode packed int4 rows by the stated layout: value 2c is the low nibble
    of byte c, value 2c + 1 the high one, each nibble minus 8 times the scale."""
    b = np.asarray(packed, np.uint8)
    nib = np.stack([b & 15, b >> 4], axis=-1).reshape(b.shape[:-1] + (2 * b.shape[-1],))
    return (nib.astype(np.float64) - 8.0) * np.asarray(scales, np.float64)[..., None]


def test_q4_hand_worked_rows():
    for c in json.load(open(Q4))["cases"]:
        bits = np.array([c["bits"]], np.uint16)
        assert np.array_equal(wl.bf16_to_f32(bits)[0], np.array(c["values"], np.float32)), c["note"]
        packed, scales = oracle.quantize_q4(bits)
        assert packed[0].tolist() == c["expect"]["bytes"], c["note"]
        assert abs(float(scales[0]) * 7 - c["expect"]["scale_times_7"]) <= 1e-6 * max(1.0, c["expect"]["scale_times_7"])


def test_q4_error_within_half_a_step():
    """Every value is recovered within half a quantisation step, the largest
    magnitude of a non-zero row maps to +-7, and nibble 0 (code -8) is never
    written."""
    rng = np.random.default_rng(4)
    x = wl.normal_bf16(rng, (500, 128))
    x[9] = 0
    packed, scales = oracle.quantize_q4(x)
    assert packed.shape == (500, 64)
    xf = wl.bf16_to_f32(x).astype(np.float64)
    rec = q4_values(packed, scales)
    # half a step, plus the binary32 rounding of x / scale (|x / scale| <= 7)
    assert np.all(np.abs(rec - xf) <= scales.astype(np.float64)[:, None] * (0.5 + 7 * 2.0 ** -23))
    codes = np.rint(rec / np.where(scales > 0, scales, 1)[:, None])
    nz = np.abs(xf).max(axis=1) > 0
    assert np.all(np.abs(codes[nz]).max(axis=1) == 7)
    assert np.all((packed & 15) != 0) and np.all((packed >> 4) != 0)
    assert scales[9] == 0 and np.all(packed[9] == 0x88)


def test_q4_attention_is_exact_on_representable_rows():
    """Rows of quarter-integers in [-1.75, 1.75] that contain 1.75 quantise
    exactly (scale 0.25), so attention over the int4 pages equals attention
    over the bf16 pages, bit for bit."""
    rng = np.random.default_rng(12)
    w = wl.random_case(43, num_seqs=3, Hq=8, Hkv=2, max_ctx=600, q_len_choices=(1, 2))
    for pool in (w.k_pages, w.v_pages):
        v = rng.integers(-7, 8, size=pool.shape).astype(np.float32) * np.float32(0.25)
        v[..., 9] = -1.75
        pool[...] = (v.view(np.uint32) >> 16).astype(np.uint16)  # quarter-integers are exact in bf16
    kc, ks = oracle.quantize_q4(w.k_pages)
    vc, vs = oracle.quantize_q4(w.v_pages)
    assert np.all(ks == 0.25) and np.all(vs == 0.25)
    args = (w.block_table, w.seq_lens, w.q_lens, w.scale)
    ref = oracle.paged_attention(w.q, w.k_pages, w.v_pages, *args)
    assert np.array_equal(oracle.attention_rows_q4(w.q, kc, vc, ks, vs, *args), ref)


def test_q4_attention_equals_attention_over_decoded_values():
    """On random rows the int4 attention is the bf16-page attention applied to
    the decoded values wherever those are bf16-exact: rescale every row so its
    scale is a power of two (values then have at most 4 significant bits)."""
    rng = np.random.default_rng(13)
    w = wl.random_case(44, num_seqs=2, Hq=4, Hkv=1, max_ctx=400, q_len_choices=(1, 3))
    kc, ks = oracle.quantize_q4(w.k_pages)
    vc, vs = oracle.quantize_q4(w.v_pages)
    ks[...] = 2.0 ** rng.integers(-3, 2, size=ks.shape)
    vs[...] = 2.0 ** rng.integers(-3, 2, size=vs.shape)
    to_bf16 = lambda f: (f.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    kp, vp = to_bf16(q4_values(kc, ks)), to_bf16(q4_values(vc, vs))
    assert np.array_equal(wl.bf16_to_f32(kp), q4_values(kc, ks).astype(np.float32))
    args = (w.block_table, w.seq_lens, w.q_lens, w.scale)
    assert np.array_equal(oracle.attention_rows_q4(w.q, kc, vc, ks, vs, *args),
                          oracle.paged_attention(w.q, kp, vp, *args))


def test_kv_append_q4_quantises_the_rows_kv_append_writes():
    w = wl.random_case(45, num_seqs=4, Hq=4, Hkv=2, max_ctx=700, q_len_choices=(1, 3, 6))
    kc, ks = oracle.quantize_q4(w.k_pages)
    vc, vs = oracle.quantize_q4(w.v_pages)
    kc2, vc2, ks2, vs2 = oracle.kv_append_q4(kc, vc, ks, vs, w.k_new, w.v_new, w.block_table,
                                             w.pos_start, w.q_lens)
    kp, vp = oracle.kv_append(w.k_pages, w.v_pages, w.k_new, w.v_new, w.block_table, w.pos_start, w.q_lens)
    for got, pages in (((kc2, ks2), kp), ((vc2, vs2), vp)):
        c, s = oracle.quantize_q4(pages)
        assert np.array_equal(got[0], c) and np.array_equal(got[1], s)


ADVANCE = os.path.join(os.path.dirname(__file__), "golden", "advance_cases.json")


def test_golden_advance_cases():
    """The next call's shapes after a greedy accept, hand-worked from the
    Assisted Generation loop (step 5, then step 1 again)."""
    for case in json.load(open(ADVANCE))["cases"]:
        sl, ql, nc = oracle.spec_advance(case["k_max"], [case["n_cand"]], [case["accepted"]],
                                         [case["window_after"]], [case["seq_len"]], [case["q_len"]])
        want = case["expect"]
        assert (int(sl[0]), int(ql[0]), int(nc[0])) == (want["seq_len"], want["q_len"], want["n_cand"]), case["note"]


def test_advance_rejects_inconsistent_lengths():
    for n_cand, acc, sl, ql in ((3, 1, 10, 3), (2, 3, 10, 3), (1, 0, 2, 3), (1, -1, 10, 2)):
        with pytest.raises(Exception):
            oracle.spec_advance(4, [n_cand], [acc], [2], [sl], [ql])


def test_advance_chain_keeps_every_accepted_token():
    """Invariant over a chain of steps: the kept length grows by accepted + 1
    each step, the next call carries min(window, k_max) candidates, and the
    window follows the golden window sequence when the outcomes do."""
    seq = json.load(open(GOLDEN))["window_sequence"]
    k_max, L = 6, 777
    w = np.array([seq["start"]], np.int32)
    n = np.array([min(seq["start"], k_max)], np.int32)
    sl, ql = np.array([L + n[0] + 1], np.int32), n + 1
    V = 16
    for outcome, want_w in zip(seq["outcomes"], seq["windows"]):
        rows = np.zeros((1, k_max + 1, V), np.float32)
        rows[0, :, 5] = 1.0                                   # the verifier says 5 everywhere
        cand = np.full((1, k_max), 5, np.int32)
        if outcome == "miss":
            cand[0, n[0] - 1] = 6                             # the last candidate misses
        acc, _, w = oracle.verify_greedy(rows, cand, n, w)
        assert int(w[0]) == want_w
        assert int(acc[0]) == (n[0] if outcome == "all" else n[0] - 1)
        kept = int(sl[0]) - int(ql[0]) + 1 + int(acc[0])
        sl, ql, n = oracle.spec_advance(k_max, n, acc, w, sl, ql)
        assert int(n[0]) == min(want_w, k_max) and int(ql[0]) == n[0] + 1 and int(sl[0]) == kept + ql[0]
