"""Helpers for the GPU parity tests: upload a workload, run the CUDA path
through the C ABI, and compute the oracle's expected values on the CPU."""
import numpy as np
import torch

import oracle
import speculative_decode_gb300 as sa
import workloads as wl

TOL_MAX = 2e-2   # max |gpu - oracle| for bf16-in / fp32-accumulate attention
TOL_MEAN = 2e-3  # mean |gpu - oracle|


def dev_tensor(a, device="cuda"):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


def dims_of(w: wl.Workload, max_q_len=None):
    mq = int(w.q_lens.max()) if max_q_len is None else max_q_len
    return sa.dims_for(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.num_pages,
                       w.max_pages_per_seq, w.total_q, max(mq, 1))


def run_attention(w: wl.Workload, use_plan=False, append=True, max_q_len=None, reps=1):
    """kv_append (optional) then paged_attn on the GPU. Returns (out bits as
    numpy uint16 [total_q, Hq, 128], error flag, k_pages, v_pages)."""
    d = dims_of(w, max_q_len)
    kp, vp = dev_tensor(w.k_pages), dev_tensor(w.v_pages)
    bt, sl, ql = dev_tensor(w.block_table), dev_tensor(w.seq_lens), dev_tensor(w.q_lens)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if append:
        sa.kv_append(d, dev_tensor(w.k_new), dev_tensor(w.v_new), kp, vp, bt, sl, ql, err_flag=err)
    plan = sa.Plan(d, w.block_table, w.seq_lens, w.q_lens) if use_plan else None
    ws = torch.zeros(sa.paged_attn_workspace_size(d, plan), dtype=torch.uint8, device="cuda")
    q = dev_tensor(w.q)
    out = torch.zeros_like(q)
    for _ in range(reps):
        sa.paged_attn(d, q, kp, vp, bt, sl, ql, w.scale, out, ws, plan=plan, err_flag=err)
    torch.cuda.synchronize()
    return (out.cpu().numpy().view(np.uint16), int(err.item()),
            kp.cpu().numpy().view(np.uint16), vp.cpu().numpy().view(np.uint16))


def oracle_attention(w: wl.Workload, append=True):
    kp, vp = w.k_pages, w.v_pages
    if append:
        kp, vp = oracle.kv_append(kp, vp, w.k_new, w.v_new, w.block_table, w.pos_start, w.q_lens)
    return oracle.paged_attention(w.q, kp, vp, w.block_table, w.seq_lens, w.q_lens, w.scale)


def attention_errors(out_bits, ref):
    got = wl.bf16_to_f32(out_bits).astype(np.float64)
    e = np.abs(got - ref)
    return float(e.max()) if e.size else 0.0, float(e.mean()) if e.size else 0.0


def assert_attention_close(out_bits, ref, what=""):
    assert out_bits.shape == ref.shape
    mx, mean = attention_errors(out_bits, ref)
    assert mx <= TOL_MAX and mean <= TOL_MEAN, f"{what}: max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def run_verify(logits, candidates, n_cand, window=None, reps=1):
    B, k1, V = logits.shape
    lg = dev_tensor(logits.astype(np.float32))
    cand = dev_tensor(candidates.astype(np.int32).reshape(B, max(k1 - 1, 0)))
    nc = dev_tensor(n_cand.astype(np.int32))
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    win = None if window is None else dev_tensor(window.astype(np.int32))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(sa.spec_verify_workspace_size(B, k1 - 1, V), dtype=torch.uint8, device="cuda")
    for _ in range(reps):
        sa.spec_verify_greedy(lg, cand, nc, acc, nxt, ws, window=win, err_flag=err)
    torch.cuda.synchronize()
    return (acc.cpu().numpy(), nxt.cpu().numpy(), None if win is None else win.cpu().numpy(),
            int(err.item()))
