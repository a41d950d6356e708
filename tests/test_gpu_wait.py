"""The bounded in-kernel wait, run out on purpose through kvc_selftest_wait_timeout.

Every attention kernel waits on shared-memory barriers with a time limit; when a wait runs out
the kernel flags KVC_DEV_WAIT_TIMEOUT and finishes instead of hanging.  The self-test kernel
waits on a barrier phase that nothing completes (no fault, no trap): the wait must give up
after its limit, report through the error word, and leave the context usable, which a normal
decode step against the oracle then checks."""
import time

import pytest
import torch

from kv_cache_decode_kvc_gb300 import kvc

from gpu_util import Case, check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


@pytest.mark.parametrize("limit_ns,lo,hi", [(20_000_000, 20e6, 1e9),   # a short limit
                                            (0, 2e9, 4e9)])            # the kernels' own 2 s
def test_wait_gives_up_and_reports(limit_ns, lo, hi):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    info = torch.full((2,), -1, dtype=torch.int64, device="cuda")
    t0 = time.perf_counter()
    kvc.kvc_selftest_wait_timeout(err, info, limit_ns)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    assert int(err.item()) & kvc.KVC_DEV_WAIT_TIMEOUT
    completed, waited = (int(x) for x in info.cpu())
    assert completed == 0                 # no thread saw the phase complete
    assert lo <= waited < hi, waited      # it waited its limit, then gave up
    assert wall < hi / 1e9 + 5.0


def test_context_is_usable_after_a_wait_ran_out():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    info = torch.zeros(2, dtype=torch.int64, device="cuda")
    kvc.kvc_selftest_wait_timeout(err, info, 5_000_000)
    case = Case(901, 3, 8, 2, 128, [300, 1, 650], "bf16")
    T_max = 700
    c = kvc.KVCache(1, case.B, case.H_q, case.H_kv, case.D, T_max, "bf16")
    try:
        d = case.to_device()
        out = torch.empty(case.B, case.H_q, case.D, dtype=torch.bfloat16, device="cuda")
        c.prefill_write(0, d["K"], d["V"], d["lens_pre"])
        c.decode_step(0, d["q"], d["k_new"], d["v_new"], out, d["lens"])
        assert c.last_error() == (kvc.KVC_OK, 0)
        check_close(out, case.oracle_out(T_max), torch.bfloat16, "decode after a timed-out wait")
    finally:
        c.close()
    assert int(err.item()) & kvc.KVC_DEV_WAIT_TIMEOUT
