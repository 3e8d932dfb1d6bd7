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
