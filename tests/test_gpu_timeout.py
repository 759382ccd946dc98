"""Failure detection without a GPU fault: every wait of the streaming ring
kernels is bounded in time, and a wait that runs out sets KD_DEV_TIMEOUT in the
device status word, drains the kernel's own copies and returns, leaving the
context usable.

The test shortens the limit to 2 ms (KD_TEST_WAIT_LIMIT_NS) and makes one
consumer warp keep its first release of a ring stage (KD_TEST_WITHHOLD_RELEASE):
nothing else ever completes that barrier phase, so the producer's wait for the
stage runs out.  The launch has one CTA (one token row of 11 ring chunks), and
the stage the producer waits for has no copy in flight.  The call must return
promptly with the timeout bit set, and the next call on the same stream must be
correct against the oracle.
"""
import time

import pytest
import torch

from lm_head_cross_vocab_gb300 import inputs as I
from lm_head_cross_vocab_gb300 import kd
from tests.parity_util import assert_parity, run_and_compare

pytestmark = pytest.mark.gpu

W = I.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kd.load_library()
    assert kd.kd_device_supported(0), "tests need an sm_103 GPU"


def test_ring_wait_runs_out_and_the_next_call_is_correct(monkeypatch):
    w = W[5].scaled(n_tokens=1, vocab=65536, variant="forward")
    t = I.make_inputs(w, "cuda")
    prob = kd.problem_for(w)
    torch.cuda.synchronize()
    monkeypatch.setenv("KD_TEST_WAIT_LIMIT_NS", "2000000")
    monkeypatch.setenv("KD_TEST_WITHHOLD_RELEASE", "1")
    t0 = time.perf_counter()
    out = kd.forward(prob, t, check=False)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    status = int(out["dev_status"].item())
    assert status & kd.KD_DEV_TIMEOUT, f"status {status:#x}"
    with pytest.raises(kd.KDError):
        kd.check_status(out["dev_status"])
    assert elapsed < 5.0, elapsed
    monkeypatch.delenv("KD_TEST_WAIT_LIMIT_NS")
    monkeypatch.delenv("KD_TEST_WITHHOLD_RELEASE")
    # the same stream and library state, a normal call
    assert_parity(run_and_compare(W[5].scaled(n_tokens=37, vocab=65536)), "bf16")
    again = kd.forward(prob, t)
    torch.cuda.synchronize()
    assert int(again["dev_status"].item()) == 0
