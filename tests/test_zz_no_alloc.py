"""The forward that allocates nothing (kd_fwd_static_scratch) against kd_fwd.

Callers that cannot allocate device memory -- a plugin whose host program owns
every device buffer, or a runtime that must not call cudaMalloc in the middle of
a step -- use kd_fwd_static_scratch, which takes its scratch from a fixed array
inside the library instead of a caller workspace.  This file is collected last
on purpose.  It checks, through the C ABI, that two calls in a row (on different
inputs, so the second call starts from the first call's leftover scratch) give
the same outputs as kd_fwd within the bf16 per-token tolerance, and that a
problem needing more scratch than the array holds is refused before any launch.
"""
import numpy as np
import pytest
import torch

from lm_head_cross_vocab_gb300 import inputs as I
from lm_head_cross_vocab_gb300 import kd
from tests.parity_util import TOK_TOL, token_rel_err

pytestmark = pytest.mark.gpu


def _static_forward(prob, t):
    dev = torch.device("cuda:0")
    n = prob.n_tokens
    out = {
        "ce_s": torch.empty(n, device=dev), "ce_t": torch.empty(n, device=dev),
        "kl": torch.empty(n, device=dev),
        "stats": torch.empty(n, kd.KD_STATS_PER_TOKEN, device=dev),
        "loss": torch.empty((), device=dev),
        "dev_status": torch.zeros((), device=dev, dtype=torch.int32),
    }
    st = kd.kd_fwd_static_scratch(prob.to_c(), kd.make_inputs(t), out["ce_s"].data_ptr(),
                                  out["ce_t"].data_ptr(), out["kl"].data_ptr(),
                                  out["stats"].data_ptr(), out["loss"].data_ptr(),
                                  out["dev_status"].data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert st == kd.KD_OK, kd.kd_status_string(st)
    return out


def test_static_scratch_forward_matches_kd_fwd_on_two_calls_in_a_row():
    kd.load_library()
    w = I.WORKLOADS[2].scaled(n_tokens=600, d_student=128, d_teacher=256, vocab=3000)
    prob = kd.problem_for(w)
    fwd_bytes, _ = kd.kd_workspace_size(prob.to_c())
    assert fwd_bytes <= kd.KD_STATIC_SCRATCH_BYTES
    tol = TOK_TOL["bf16"]
    for seed in (101, 202):
        t = {k: v.cuda() for k, v in I.make_inputs(w, "cpu", seed=seed).items()}
        ref = kd.forward(prob, t)
        got = _static_forward(prob, t)
        torch.cuda.synchronize()
        assert int(got["dev_status"].item()) == 0
        valid = (t["labels"] != w.ignore_index).cpu().numpy()
        for key in ("ce_s", "ce_t", "kl"):
            err = token_rel_err(got[key].cpu().double().numpy(),
                                ref[key].cpu().double().numpy(), valid)
            assert err <= tol, (seed, key, err)
        s_ref = ref["stats"].cpu().double().numpy()
        s_got = got["stats"].cpu().double().numpy()
        assert np.max(np.abs(s_got - s_ref) / np.maximum(np.abs(s_ref), 1e-3)) <= tol
        lr, lg = ref["loss"].item(), got["loss"].item()
        assert abs(lg - lr) <= tol * abs(lr), (seed, lr, lg)


def test_static_scratch_refuses_problems_larger_than_the_array():
    kd.load_library()
    w = I.WORKLOADS[4]  # 32768 tokens: its split records need far more than the array
    prob = kd.problem_for(w).to_c()
    fwd_bytes, _ = kd.kd_workspace_size(prob)
    assert fwd_bytes > kd.KD_STATIC_SCRATCH_BYTES
    fake = 1 << 20  # never dereferenced: the call is refused before any launch
    ins = kd.kd_inputs(h_s=fake, w_s=fake, topk_idx=fake, topk_p=fake)
    st = kd.kd_fwd_static_scratch(prob, ins, None, None, None, None, None, None, None)
    assert st == kd.KD_ERR_WORKSPACE
