"""Forward-only scoring of a hidden-state student (flash_kd API doc, module
description: only the forward pass exists and scoring runs without gradients).

kd_fwd is called with stats = NULL: no per-token statistics are handed back for a
backward.  Per-token CE / teacher CE / KL and the loss are compared with the fp64
oracle element by element, on a ragged multi-tile case for every KL variant (the
skew variants keep their first-pass statistics in the workspace for the second
pass), and at the separate-teacher workload's full size on a seeded token sample.
Outputs with and without saved statistics must be bit-identical.
"""
import numpy as np
import pytest
import torch

from lm_head_cross_vocab_gb300 import inputs as I
from lm_head_cross_vocab_gb300 import kd
from oracle import kd_oracle as O
from tests.parity_util import TOK_TOL, oracle_kwargs, oracle_logits, token_rel_err

pytestmark = pytest.mark.gpu

W = I.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kd.load_library()
    assert kd.kd_device_supported(0), "tests need an sm_103 GPU"


def _score(prob, t):
    out = kd.forward(prob, t, save_stats=False)
    torch.cuda.synchronize()
    assert out["stats"] is None
    return out


@pytest.mark.parametrize("variant", ["forward", "reverse", "jeffreys", "skew_js", "skew_forward",
                                     "skew_reverse"])
def test_hidden_student_scoring_without_stats(variant):
    w = W[2].scaled(n_tokens=601, vocab=5003, d_student=256, d_teacher=392, variant=variant)
    cpu = I.make_inputs(w, "cpu")
    t = {k: v.cuda() for k, v in cpu.items()}
    prob = kd.problem_for(w)
    got = _score(prob, t)
    z_s, z_t = oracle_logits(cpu, w)
    ref = O.forward(z_s, z_t, cpu["labels"].numpy(), **oracle_kwargs(w, prob))
    valid = ref["valid"]
    for key in ("ce_s", "ce_t", "kl"):
        err = token_rel_err(got[key].cpu().double().numpy(), ref[key], valid)
        assert err <= TOK_TOL["bf16"], (key, err)
        assert not got[key].cpu()[~torch.from_numpy(valid)].any(), key
    assert abs(got["loss"].item() - ref["loss"]) <= TOK_TOL["bf16"] * abs(ref["loss"])


def test_hidden_student_scoring_fullsize_sampled_tokens():
    """The separate-teacher workload (4096 tokens, V 32000) scored without saved
    statistics: a seeded token sample against the oracle, and every output equal
    to the same call with statistics."""
    w = W[2]
    t = I.make_inputs(w, "cuda")
    prob = kd.problem_for(w, vocab_chunk=0, seq_chunk=0)
    got = _score(prob, t)
    with_stats = kd.forward(prob, t)
    torch.cuda.synchronize()
    for key in ("ce_s", "ce_t", "kl", "loss"):
        assert torch.equal(got[key], with_stats[key]), key
    rows = np.sort(np.random.default_rng(23).choice(w.n_tokens, 64, replace=False))
    cpu = {k: t[k][rows].cpu() for k in ("h_s", "h_t", "labels")}
    z_s = O.project(cpu["h_s"], t["w_s"].cpu())
    z_t = O.project(cpu["h_t"], t["w_t"].cpu())
    labels = cpu["labels"].numpy()
    ref = O.forward(z_s, z_t, labels, **{**oracle_kwargs(w, prob), "reduction": "sum"})
    valid = labels != w.ignore_index
    for key in ("ce_s", "ce_t", "kl"):
        err = token_rel_err(got[key][rows].cpu().double().numpy(), ref[key], valid)
        assert err <= TOK_TOL["bf16"], (key, err)


def test_hidden_student_scoring_num_batch_labels():
    """Scoring with a caller-given label count as the mean's denominator
    (nemo_automodel KDLoss, forward(num_batch_labels))."""
    w = W[2].scaled(n_tokens=300, vocab=2056, d_student=128, d_teacher=64, variant="forward")
    cpu = I.make_inputs(w, "cpu")
    t = {k: v.cuda() for k, v in cpu.items()}
    prob = kd.problem_for(w, num_batch_labels=1000)
    got = _score(prob, t)
    z_s, z_t = oracle_logits(cpu, w)
    ref = O.forward(z_s, z_t, cpu["labels"].numpy(), **oracle_kwargs(w, prob))
    assert abs(got["loss"].item() - ref["loss"]) <= TOK_TOL["bf16"] * abs(ref["loss"])
