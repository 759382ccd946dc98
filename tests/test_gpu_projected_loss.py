"""The projected teacher inside the loss (KD_TEACHER_PROJECTED) on the GPU against
the oracle (orda-kernel README, "Cross-vocabulary distillation": token-map
projection into a PrecomputedTeacher with logits_temperature = T).

The library moves teacher logits over the teacher vocabulary onto the student
vocabulary inside its loss kernels and never stores the projected tensor.  The
oracle composes its own projection (tempered before the per-id aggregation,
duplicates summed in probability space, unmatched ids at -inf) with its loss at
teacher temperature 1 and student temperature T, on the same input bytes.
Per-token CE / teacher CE / KL, the loss and d z_s are compared element by
element; ignored tokens must give exact zeros.
"""
import numpy as np
import pytest
import torch

from lm_head_cross_vocab_gb300 import kd
from oracle import kd_oracle as O
from tests.parity_util import GRAD_TOL, TOK_TOL, rel_l2, token_rel_err

pytestmark = pytest.mark.gpu

DT = {"fp32": torch.float32, "bf16": torch.bfloat16}
VARIANTS = ["forward", "reverse", "jeffreys", "skew_js", "skew_forward", "skew_reverse"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kd.load_library()
    assert kd.kd_device_supported(0), "tests need an sm_103 GPU"


def _map(v_t, v_s, seed, unmatched=True):
    """Seeded token map with repeated student ids and unmatched teacher tokens;
    with `unmatched`, also student ids that no teacher token reaches."""
    rng = np.random.default_rng(seed)
    tmap = rng.integers(0, v_s, size=v_t)
    tmap[rng.random(v_t) < 0.15] = -1
    if unmatched:
        tmap[np.isin(tmap, rng.choice(v_s, v_s // 10, replace=False))] = -1
    else:  # every student id gets at least one teacher token
        tmap[rng.choice(v_t, v_s, replace=False)] = rng.permutation(v_s)
    return tmap.astype(np.int32)


def _run(n, v_t, v_s, dtype, variant, T, *, w_sce=0.5, w_tce=0.0, seed=0, unmatched=True,
         tmap=None):
    g = torch.Generator().manual_seed(seed)
    z_s = (torch.randn(n, v_s, generator=g) * 4.0).to(DT[dtype])
    z_t = (torch.randn(n, v_t, generator=g) * 4.0).to(DT[dtype])
    labels = torch.randint(0, v_s, (n,), generator=g)
    labels[torch.rand(n, generator=g) < 0.08] = -100
    if tmap is None:
        tmap = _map(v_t, v_s, seed + 1, unmatched)
    dev = torch.device("cuda:0")
    t = {"logits_s": z_s.to(dev), "logits_t": z_t.to(dev), "labels": labels.to(dev),
         "token_map": torch.from_numpy(tmap).to(dev)}
    prob = kd.Problem(n_tokens=n, vocab=v_s, dtype=dtype, student="logits", teacher="projected",
                      variant=variant, t_student=T, t_teacher=T, w_student_ce=w_sce,
                      w_teacher_ce=w_tce, w_kl=1.0, beta=0.1, ignore_index=-100,
                      vocab_teacher=v_t)
    fwd = kd.forward(prob, t)
    bwd = kd.backward(prob, t, fwd["stats"], want=("logits_s",))
    torch.cuda.synchronize()
    zp = O.project_teacher_logits(z_t, tmap, v_s, temperature=T)
    kw = dict(variant=variant, t_student=T, t_teacher=1.0, beta=0.1, w_student_ce=w_sce,
              w_teacher_ce=w_tce, w_kl=1.0, ignore_index=-100)
    lab = labels.numpy()
    ref = O.forward(O.as_f64(z_s), zp, lab, **kw)
    g_s, _ = O.grad_logits(O.as_f64(z_s), zp, lab, **kw)
    return fwd, bwd, ref, g_s


def _check(fwd, bwd, ref, g_s, dtype, variant, w_tce=0.0):
    valid = ref["valid"]
    kl = fwd["kl"].cpu().double().numpy()
    ce = fwd["ce_s"].cpu().double().numpy()
    gz = bwd["d_logits_s"].cpu().double().numpy()
    assert np.all(kl[~valid] == 0) and np.all(ce[~valid] == 0) and np.all(gz[~valid] == 0)
    if variant in ("reverse", "jeffreys") and np.isinf(ref["kl"][valid]).any():
        # reverse KL is infinite where the projected teacher gives an id no
        # probability and the student some: both sides agree
        assert np.all(kl[valid][np.isinf(ref["kl"][valid])] > 1e30)
        return
    assert token_rel_err(kl, ref["kl"], valid) <= TOK_TOL[dtype]
    assert token_rel_err(ce, ref["ce_s"], valid) <= TOK_TOL[dtype]
    if w_tce > 0:
        ce_t = fwd["ce_t"].cpu().double().numpy()
        assert token_rel_err(ce_t, ref["ce_t"], valid) <= TOK_TOL[dtype]
    assert abs(fwd["loss"].item() - ref["loss"]) <= TOK_TOL[dtype] * abs(ref["loss"])
    assert rel_l2(gz, g_s) <= GRAD_TOL[dtype]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("n,v_t,v_s", [(37, 1000, 700), (19, 60000, 50001)])
def test_projected_teacher_matches_oracle(dtype, variant, n, v_t, v_s):
    """One CTA per teacher row (1000 ids) and clusters of 2 (bf16) or 4 (fp32)
    CTAs exchanging their gathered values (60000 ids onto a ragged 50001)."""
    T = 2.0
    _check(*_run(n, v_t, v_s, dtype, variant, T, seed=v_t + n), dtype, variant)


@pytest.mark.parametrize("variant", ["forward", "skew_js"])
def test_projected_teacher_ce_at_t1(variant):
    """T = 1 with both CE terms; every student id has a teacher token, so the
    teacher CE of the projected distribution is finite."""
    w_tce = 0.3
    res = _run(41, 3000, 2000, "bf16", variant, 1.0, w_sce=0.7, w_tce=w_tce, seed=9,
               unmatched=False)
    _check(*res, "bf16", variant, w_tce=w_tce)


def test_projected_teacher_large_vocabularies():
    """152k teacher ids onto 128k student ids (a cluster of 4 bf16 CTAs), more
    rows than clusters, forward KL at T = 2."""
    _check(*_run(96, 151936, 128256, "bf16", "forward", 2.0, seed=3), "bf16", "forward")


def test_projected_teacher_skewed_map_is_reported():
    """A map that sends every teacher token into a few student ids overflows a
    receive buffer of the fused kernel: nothing is computed, the status word
    says so (the caller then projects first and uses a logits teacher)."""
    v_t, v_s = 100000, 70001
    rng = np.random.default_rng(21)
    tmap = rng.integers(0, 4000, size=v_t).astype(np.int32)
    with pytest.raises(kd.KDError):
        _run(3, v_t, v_s, "bf16", "forward", 1.0, tmap=tmap)


def test_projected_teacher_bad_map_entry_is_flagged():
    tmap = _map(300, 200, 3)
    tmap[17] = 200  # outside [-1, V_s)
    with pytest.raises(kd.KDError):
        _run(4, 300, 200, "bf16", "forward", 1.0, tmap=tmap)
