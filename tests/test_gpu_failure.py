"""The failure path of the kernels' bounded waits, on the GPU, without a
fault: one CTA waits on an mbarrier that nothing completes (no copies in
flight), gives up after the wait's limit, sets the timeout bit of the
caller's flag and returns; the context stays usable, which a parity check
right after shows."""
import time

import pytest
import torch

import workloads as wl
from gpu_path import assert_attention_close, oracle_attention, run_attention
import speculative_decode_gb300 as sa

pytestmark = pytest.mark.gpu

SA_ERR_TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decode_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def test_bounded_wait_gives_up_and_flags_the_timeout():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    sa.selftest_bounded_wait(err)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(err.item()) == 1 << SA_ERR_TIMEOUT
    assert waited < 10.0                      # the wait is bounded (about 0.25 s)
    # the context is still usable: an attention call right after is correct
    w = wl.random_case(31, num_seqs=3, Hq=8, Hkv=2, max_ctx=600, q_len_choices=(1, 2))
    out, flag, _, _ = run_attention(w)
    assert flag == 0
    assert_attention_close(out, oracle_attention(w), "after a timed-out wait")


def test_timeout_bit_is_added_to_a_flag_already_set():
    err = torch.full((1,), 1 << 3, dtype=torch.int32, device="cuda")  # an earlier page error
    sa.selftest_bounded_wait(err)
    torch.cuda.synchronize()
    assert int(err.item()) == (1 << 3) | (1 << SA_ERR_TIMEOUT)
