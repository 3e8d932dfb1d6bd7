"""GPU parity of spec_verify_greedy against the oracle: bit-exact accepted
counts, correction tokens and window updates."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_path import run_verify

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "greedy_accept_cases.json")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def check(logits, cand, n_cand, window):
    a, n, w, err = run_verify(logits, cand, n_cand, window)
    ra, rn, rw = oracle.verify_greedy(logits, cand, n_cand, window)
    assert err == 0
    assert np.array_equal(a, ra) and np.array_equal(n, rn) and np.array_equal(w, rw)
    return a, n, w


def test_spec_verify_config_full_vocab():
    w = wl.config(3)
    a, _, _ = check(w.logits, w.candidates, w.n_cand, w.window)
    assert a.shape == (16,)


@pytest.mark.parametrize("seed", range(6))
def test_random_n_cand_and_vocab(seed):
    rng = np.random.default_rng(200 + seed)
    B = int(rng.integers(1, 40))
    k = int(rng.integers(0, 16))
    V = int(rng.choice([1, 3, 1000, 4097, 32000, wl.LLAMA3_VOCAB]))
    w = wl.random_case(seed, num_seqs=B, max_ctx=10)
    wl.add_verify_inputs(w, rng, k_max=k, vocab=V, n_cand=rng.integers(0, k + 1, size=B))
    w.window = rng.integers(1, 9, size=B).astype(np.int32)
    check(w.logits, w.candidates, w.n_cand, w.window)


def test_ties_nan_signed_zero_and_infinities():
    rng = np.random.default_rng(9)
    B, k, V = 6, 3, 5000
    logits = rng.integers(-3, 3, size=(B, k + 1, V)).astype(np.float32)   # heavy ties
    logits[0, :, :] = np.nan                          # all-NaN rows
    logits[1, 0, 100] = np.nan
    logits[1, 0, 4000] = np.float32(1e30)
    logits[2, :, :] = -3.0
    logits[2, 0, 7] = -0.0
    logits[2, 0, 3] = 0.0                             # +0 at 3 ties -0 at 7: 3 wins
    logits[3, 1, V - 1] = np.inf
    logits[4, :, :] = -np.inf                         # all -inf: index 0
    logits[5, 2, 4999] = 100.0
    cand = rng.integers(0, V, size=(B, k)).astype(np.int32)
    n_cand = np.array([3, 1, 2, 3, 0, 3], np.int32)
    check(logits, cand, n_cand, np.full(B, 5, np.int32))


def test_golden_cases_on_gpu():
    data = json.load(open(GOLDEN))
    conv = {"nan": np.nan, "inf": np.inf, "-inf": -np.inf}
    for case in data["cases"]:
        rows = []
        for s in case["rows"]:
            fill = conv[s["fill"]] if isinstance(s["fill"], str) else s["fill"]
            r = np.full(s["V"], fill, np.float32)
            for kk, v in s["set"].items():
                r[int(kk)] = conv[v] if isinstance(v, str) else v
            rows.append(r)
        logits = np.stack(rows)[None]
        a, n, w, err = run_verify(logits, np.array([case["candidates"]], np.int32),
                                  np.array([case["n_cand"]], np.int32),
                                  np.array([case["window_in"]], np.int32))
        exp = case["expect"]
        assert err == 0
        assert (a[0], n[0], w[0]) == (exp["accepted"], exp["next_tok"], exp["window_out"]), case["note"]


def test_repeated_calls_reset_counters():
    w = wl.config(3)
    a1, n1, w1, _ = run_verify(w.logits, w.candidates, w.n_cand, None, reps=1)
    a3, n3, w3, _ = run_verify(w.logits, w.candidates, w.n_cand, None, reps=3)
    assert np.array_equal(a1, a3) and np.array_equal(n1, n3)


def test_n_cand_above_k_max_sets_the_flag():
    logits = np.zeros((2, 3, 64), np.float32)
    _, _, _, err = run_verify(logits, np.zeros((2, 2), np.int32), np.array([1, 3], np.int32))
    assert err & (1 << 7)


def _planted_step(rng, B, k_max, V, n, force=None):
    """Logits with one planted winner per row and candidates equal to the
    winner with p = 0.7; force[b] = 'all' / 'miss' makes sequence b match
    every candidate / miss its last one."""
    logits = rng.standard_normal(size=(B, k_max + 1, V), dtype=np.float32)
    planted = rng.integers(0, V, size=(B, k_max + 1)).astype(np.int32)
    for b in range(B):
        for j in range(k_max + 1):
            logits[b, j, planted[b, j]] = logits[b, j].max() + np.float32(1.0)
    cand = np.where(rng.random((B, k_max)) < 0.7, planted[:, :k_max],
                    (planted[:, :k_max] + 1 + rng.integers(0, V - 1, (B, k_max))) % V).astype(np.int32)
    for b, f in (force or {}).items():
        cand[b, :] = planted[b, :k_max]
        if f == "miss" and n[b] > 0:
            cand[b, n[b] - 1] = (planted[b, n[b] - 1] + 1) % V
    return logits, cand


def test_advance_chain_matches_the_oracle_step_by_step():
    """Thirteen verify steps chained on the device: every step's accepted
    counts, correction tokens, windows and the next call's seq_lens, q_lens
    and candidate counts come from the previous step's device buffers, and
    each is compared bit for bit with the oracle's verify + advance.
    Sequence 0 is driven through the golden window sequence's outcomes."""
    from gpu_path import dev_tensor
    import speculative_decode_gb300 as sa
    seq = json.load(open(GOLDEN))["window_sequence"]
    rng = np.random.default_rng(314)
    B, k_max, V = 6, 7, 3000
    window = np.full(B, seq["start"], np.int32)
    n = np.minimum(window, k_max).astype(np.int32)
    sl = (rng.integers(100, 3000, size=B).astype(np.int32) + n + 1).astype(np.int32)
    ql = (n + 1).astype(np.int32)
    d_win, d_sl, d_ql, d_n = dev_tensor(window), dev_tensor(sl), dev_tensor(ql), dev_tensor(n)
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    nxt = torch.zeros_like(acc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(sa.spec_verify_workspace_size(B, k_max, V), dtype=torch.uint8, device="cuda")
    for step, (outcome, want_w0) in enumerate(zip(seq["outcomes"], seq["windows"])):
        logits, cand = _planted_step(rng, B, k_max, V, n, force={0: outcome})
        # the next step's candidate counts overwrite this step's, in place
        sa.spec_verify_greedy_advance(dev_tensor(logits), dev_tensor(cand), d_n, acc, nxt, d_win, d_sl, d_ql,
                                      d_n, ws, err_flag=err)
        ra, rn, rw = oracle.verify_greedy(logits, cand, n, window)
        rsl, rql, rnc = oracle.spec_advance(k_max, n, ra, rw, sl, ql)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = [t.cpu().numpy() for t in (acc, nxt, d_win, d_sl, d_ql, d_n)]
        for g, r, name in zip(got, (ra, rn, rw, rsl, rql, rnc), ("accepted", "next", "window", "seq_lens", "q_lens", "n_cand")):
            assert np.array_equal(g, r), (step, name, g, r)
        assert int(rw[0]) == want_w0
        window, n, sl, ql = rw, rnc, rsl, rql


def test_advance_golden_cases_on_gpu():
    from gpu_path import dev_tensor
    import speculative_decode_gb300 as sa
    cases = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "advance_cases.json")))["cases"]
    for c in cases:
        k, V = c["k_max"], 64
        # a window before step 5 that gives the case's window after it
        n = c["n_cand"]
        all_match = c["accepted"] == n
        w_in = c["window_after"] - 2 if all_match else c["window_after"] + 1
        if not all_match and c["window_after"] == 1:
            w_in = 1
        logits = np.zeros((1, k + 1, V), np.float32)
        logits[0, :, 9] = 1.0
        cand = np.full((1, max(k, 1)), 9, np.int32)[:, :k]
        if not all_match:
            cand[0, c["accepted"]] = 10
        d_win, d_sl, d_ql = (dev_tensor(np.array([v], np.int32)) for v in (w_in, c["seq_len"], c["q_len"]))
        d_nc = dev_tensor(np.array([n], np.int32))
        out_n = torch.zeros(1, dtype=torch.int32, device="cuda")
        acc = torch.zeros(1, dtype=torch.int32, device="cuda")
        nxt = torch.zeros_like(acc)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = torch.zeros(sa.spec_verify_workspace_size(1, k, V), dtype=torch.uint8, device="cuda")
        sa.spec_verify_greedy_advance(dev_tensor(logits), dev_tensor(cand), d_nc, acc, nxt, d_win, d_sl, d_ql,
                                      out_n, ws, err_flag=err)
        torch.cuda.synchronize()
        e = c["expect"]
        assert int(err.item()) == 0 and int(acc.item()) == c["accepted"] and int(d_win.item()) == c["window_after"]
        assert (int(d_sl.item()), int(d_ql.item()), int(out_n.item())) == (e["seq_len"], e["q_len"], e["n_cand"]), c["note"]


def test_advance_rejects_inconsistent_lengths_and_keeps_them():
    from gpu_path import dev_tensor
    import speculative_decode_gb300 as sa
    logits = np.zeros((2, 4, 32), np.float32)
    cand = np.zeros((2, 3), np.int32)
    d_nc = dev_tensor(np.array([3, 2], np.int32))
    d_win, d_sl, d_ql = dev_tensor(np.array([5, 5], np.int32)), dev_tensor(np.array([50, 50], np.int32)), \
        dev_tensor(np.array([4, 2], np.int32))              # sequence 1: q_len 2 < n_cand + 1
    out_n = torch.zeros(2, dtype=torch.int32, device="cuda")
    acc = torch.zeros(2, dtype=torch.int32, device="cuda")
    nxt = torch.zeros_like(acc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(sa.spec_verify_workspace_size(2, 3, 32), dtype=torch.uint8, device="cuda")
    sa.spec_verify_greedy_advance(dev_tensor(logits), dev_tensor(cand), d_nc, acc, nxt, d_win, d_sl, d_ql,
                                  out_n, ws, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & (1 << 7)
    assert int(d_sl[1].item()) == 50 and int(d_ql[1].item()) == 2 and int(d_win[1].item()) == 5
    assert int(d_ql[0].item()) == min(7, 3) + 1                # sequence 0 advanced: all matched, window 7


def test_workspace_reused_after_an_error_call():
    """A call with an out-of-range candidate count flags the error and still
    leaves the workspace's counters at zero: the next valid call on the same
    workspace is bit-exact."""
    from gpu_path import dev_tensor
    import speculative_decode_gb300 as sa
    w = wl.config(3)
    B, k1, V = w.logits.shape
    ws = torch.zeros(sa.spec_verify_workspace_size(B, k1 - 1, V), dtype=torch.uint8, device="cuda")
    lg, cand = dev_tensor(w.logits), dev_tensor(w.candidates)
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    nxt = torch.zeros_like(acc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = w.n_cand.copy()
    bad[3] = k1 + 4
    sa.spec_verify_greedy(lg, cand, dev_tensor(bad), acc, nxt, ws, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & (1 << 7)
    err.zero_()
    sa.spec_verify_greedy(lg, cand, dev_tensor(w.n_cand), acc, nxt, ws, err_flag=err)
    ra, rn, _ = oracle.verify_greedy(w.logits, w.candidates, w.n_cand)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(acc.cpu().numpy(), ra) and np.array_equal(nxt.cpu().numpy(), rn)
