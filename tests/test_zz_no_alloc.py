"""sa_paged_attn_noalloc: the entry point for callers that cannot allocate
device memory (for example a plugin inside a serving process whose memory
pool owns the whole GPU). Its scratch is a fixed array inside the library, so
these checks call it twice in a row through the C ABI and compare each result
with the regular sa_paged_attn, which uses a caller-allocated workspace.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_path import TOL_MAX, TOL_MEAN, dev_tensor, dims_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    from speculative_decode_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    import speculative_decode_gb300 as mod
    return mod


def _bf16_to_f64(t):
    return wl.bf16_to_f32(t.cpu().numpy().view(np.uint16)).astype(np.float64)


def test_noalloc_matches_the_workspace_entry_point_on_two_calls(sa):
    # the Llama3-8B-shaped decode batch: most (sequence, KV head) segments are
    # split across warps, so the scratch's partials and counters are exercised
    w = wl.config(1)
    d = dims_of(w)
    q, kp, vp = dev_tensor(w.q), dev_tensor(w.k_pages), dev_tensor(w.v_pages)
    bt, sl, ql = dev_tensor(w.block_table), dev_tensor(w.seq_lens), dev_tensor(w.q_lens)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(sa.paged_attn_workspace_size(d), dtype=torch.uint8, device="cuda")
    ref = torch.zeros_like(q)
    sa.paged_attn(d, q, kp, vp, bt, sl, ql, w.scale, ref, ws, err_flag=err)
    lib = sa.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    outs = []
    for _ in range(2):
        out = torch.full_like(q, 0x7FC0)     # NaN bit patterns: every row must be written
        rc = lib.sa_paged_attn_noalloc(ctypes.byref(d), q.data_ptr(), kp.data_ptr(), vp.data_ptr(),
                                       bt.data_ptr(), sl.data_ptr(), ql.data_ptr(),
                                       ctypes.c_float(w.scale), out.data_ptr(), err.data_ptr(),
                                       stream)
        assert rc == 0, sa.status_string(rc)
        outs.append(out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    r = _bf16_to_f64(ref)
    for out in outs:
        e = np.abs(_bf16_to_f64(out) - r)
        assert e.max() <= TOL_MAX and e.mean() <= TOL_MEAN, (e.max(), e.mean())


def test_noalloc_rejects_shapes_beyond_its_scratch(sa):
    w = wl.config(1)
    d = dims_of(w)
    d.total_q = 1 << 20                       # a workspace far above 16 MiB
    lib = sa.load_library()
    rc = lib.sa_paged_attn_noalloc(ctypes.byref(d), *([None] * 6), ctypes.c_float(0.1), None,
                                   None, None)
    assert rc == 6                            # SA_ERR_WORKSPACE, before any GPU work
