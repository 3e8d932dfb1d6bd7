"""sa_paged_attn_noalloc: the entry point for callers that cannot allocate
device memory (for example a plugin inside a serving process whose memory
pool owns the whole GPU). Its scratch (partial accumulators and counters) is
a fixed array inside the library, so these checks call it twice in a row
through the C ABI and require each result to equal, bit for bit, that of the
regular sa_paged_attn, which uses a caller-allocated workspace; they also
check that calls after the first allocate no device memory.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_path import dev_tensor, dims_of

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module")
def sa():
    from speculative_decode_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    import speculative_decode_gb300 as mod
    return mod


def _case(name):
    if name == "llama3-8b-decode":
        # most (sequence, KV head) segments are cut across CTAs, so the
        # scratch's partials and merge counters are exercised
        return wl.config(1)
    # verify-shaped: q_len 6 per sequence, 24 query rows per KV head, which
    # takes the split kernel and its combine pass
    return wl.random_case(1701, num_seqs=4, Hq=32, Hkv=8, max_ctx=3000, q_len_choices=(6,))


def _noalloc(lib, d, q, kp, vp, bt, sl, ql, scale, out, err, stream):
    return lib.sa_paged_attn_noalloc(ctypes.byref(d), q.data_ptr(), kp.data_ptr(), vp.data_ptr(),
                                     bt.data_ptr(), sl.data_ptr(), ql.data_ptr(),
                                     ctypes.c_float(scale), out.data_ptr(), err.data_ptr(), stream)


@pytest.mark.parametrize("name", ["llama3-8b-decode", "verify-4seq-qlen6"])
def test_noalloc_equals_the_workspace_entry_point_bit_for_bit(sa, name):
    w = _case(name)
    d = dims_of(w)
    assert sa.paged_attn_workspace_size(d) <= STATIC_SCRATCH_BYTES
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
        rc = _noalloc(lib, d, q, kp, vp, bt, sl, ql, w.scale, out, err, stream)
        assert rc == 0, sa.status_string(rc)
        outs.append(out)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    r = ref.cpu().numpy()
    for out in outs:
        assert np.array_equal(out.cpu().numpy(), r)


def test_noalloc_allocates_nothing_after_the_first_call(sa):
    w = _case("verify-4seq-qlen6")
    d = dims_of(w)
    q, kp, vp = dev_tensor(w.q), dev_tensor(w.k_pages), dev_tensor(w.v_pages)
    bt, sl, ql = dev_tensor(w.block_table), dev_tensor(w.seq_lens), dev_tensor(w.q_lens)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    lib = sa.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    assert _noalloc(lib, d, q, kp, vp, bt, sl, ql, w.scale, out, err, stream) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        assert _noalloc(lib, d, q, kp, vp, bt, sl, ql, w.scale, out, err, stream) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert int(err.item()) == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(sa):
    w = wl.config(1)
    d = dims_of(w)
    d.max_q_len = 6                           # 24 rows per KV head: partials per query row,
    d.total_q = 1 << 16                       # a workspace far above 16 MiB
    assert sa.paged_attn_workspace_size(d) > STATIC_SCRATCH_BYTES
    lib = sa.load_library()
    rc = lib.sa_paged_attn_noalloc(ctypes.byref(d), *([None] * 6), ctypes.c_float(0.1), None,
                                   None, None)
    assert rc == 6                            # SA_ERR_WORKSPACE, before any GPU work
