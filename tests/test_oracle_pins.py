"""Pins of the CPU fp64 oracle to facts that do not come from the oracle itself.

Each test ties one part of the oracle to a closed form, a scipy / torch library
routine, an inequality, a special case or finite differences, so that a
plausible slip in the oracle (swapped p/q, dropped T^2, wrong sign or index,
transposed operand, wrong skew weights) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.spatial.distance as ssd
import scipy.special as sps
import scipy.stats as sst
import torch

from oracle import kd_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def _eval(expr):
    return eval(expr, {"__builtins__": {}}, {"log": math.log, "sqrt": math.sqrt})


def _rand_logits(n, v, std=1.0, rng=RNG):
    return rng.normal(0.0, std, size=(n, v))


# ---------------------------------------------------------------- closed forms

def test_golden_closed_forms():
    with open(os.path.join(GOLDEN, "closed_form_v3.json")) as f:
        gold = json.load(f)
    for case in gold["cases"]:
        z_s = np.array([_eval(case["z_s"])])
        exp = case["expect"]
        t = case["t"]
        if "topk_idx" in case:
            idx = np.array([case["topk_idx"]])
            pk = np.array([_eval(case["topk_p"])])
            out = O.forward(z_s, None, None, topk_idx=idx, topk_p=pk, t_student=t,
                            w_student_ce=0.0, w_kl=1.0, reduction="sum")
            assert out["kl"][0] == pytest.approx(_eval(exp["topk"]), abs=1e-14)
            g, _ = O.grad_logits(z_s, None, None, topk_idx=idx, topk_p=pk, t_student=t,
                                 w_student_ce=0.0, w_kl=1.0, reduction="sum")
            np.testing.assert_allclose(g[0], _eval(exp["grad_topk_z"]), atol=1e-14)
            continue
        z_t = np.array([_eval(case["z_t"])])
        labels = np.array([case["label"]])
        for variant in ("forward", "reverse", "jeffreys", "skew_forward", "skew_reverse",
                        "skew_js"):
            if variant not in exp:
                continue
            out = O.forward(z_s, z_t, labels, variant=variant, t_student=t,
                            beta=case["beta"], w_teacher_ce=1.0)
            assert out["kl"][0] == pytest.approx(_eval(exp[variant]), abs=1e-14), variant
            assert out["ce_s"][0] == pytest.approx(_eval(exp["ce_s"]), abs=1e-14)
            assert out["ce_t"][0] == pytest.approx(_eval(exp["ce_t"]), abs=1e-14)
        if "loss_kl_only" in exp:
            out = O.forward(z_s, z_t, labels, variant="forward", t_student=t,
                            w_student_ce=0.0, w_teacher_ce=0.0, w_kl=1.0)
            assert out["loss"] == pytest.approx(_eval(exp["loss_kl_only"]), abs=1e-14)
        if "grad_forward_a" in exp:
            g, _ = O.grad_logits(z_s, z_t, labels, variant="forward", t_student=t,
                                 w_student_ce=0.0, w_kl=1.0)
            np.testing.assert_allclose(g[0], _eval(exp["grad_forward_a"]), atol=1e-14)
        if "grad_forward_z" in exp:
            g, _ = O.grad_logits(z_s, z_t, labels, variant="forward", t_student=t,
                                 w_student_ce=0.0, w_kl=1.0)
            np.testing.assert_allclose(g[0], _eval(exp["grad_forward_z"]), atol=1e-14)


def test_ce_uniform_logits_is_log_v():
    for v in (2, 7, 512, 32000):
        z = np.full((3, v), 1.25)
        ce = O.cross_entropy_rows(z, np.array([0, v // 2, v - 1]), np.ones(3, bool))
        np.testing.assert_allclose(ce, math.log(v), rtol=0, atol=1e-12)


def test_ce_dominant_label_goes_to_zero():
    v = 1000
    z = np.zeros((1, v))
    z[0, 17] = 60.0
    ce = O.cross_entropy_rows(z, np.array([17]), np.ones(1, bool))[0]
    assert ce == pytest.approx((v - 1) * math.exp(-60.0), rel=1e-9)


# ------------------------------------------------------------ library routines

def test_ce_matches_torch_cross_entropy():
    """flash_kd: CE matches F.cross_entropy(..., reduction='none') incl. ignore_index."""
    z = _rand_logits(16, 50, 3.0)
    labels = RNG.integers(0, 50, size=16)
    labels[[2, 9]] = -1
    ref = torch.nn.functional.cross_entropy(torch.from_numpy(z), torch.from_numpy(labels),
                                            ignore_index=-1, reduction="none").numpy()
    out = O.forward(z, z, labels, ignore_index=-1)
    np.testing.assert_allclose(out["ce_s"], ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("t", [1.0, 2.0, 0.7])
def test_forward_reverse_kl_match_scipy_entropy(t):
    z_s, z_t = _rand_logits(8, 40, 2.0), _rand_logits(8, 40, 2.0)
    p = sps.softmax(z_s / t, axis=1)
    q = sps.softmax(z_t / t, axis=1)
    fwd = O.forward(z_s, z_t, None, variant="forward", t_student=t)["kl"]
    rev = O.forward(z_s, z_t, None, variant="reverse", t_student=t)["kl"]
    jef = O.forward(z_s, z_t, None, variant="jeffreys", t_student=t)["kl"]
    np.testing.assert_allclose(fwd, sst.entropy(q, p, axis=1), rtol=1e-12)
    np.testing.assert_allclose(rev, sst.entropy(p, q, axis=1), rtol=1e-12)
    np.testing.assert_allclose(jef, sst.entropy(q, p, axis=1) + sst.entropy(p, q, axis=1),
                               rtol=1e-12)


def test_independent_teacher_temperature():
    z_s, z_t = _rand_logits(5, 30, 2.0), _rand_logits(5, 30, 2.0)
    p = sps.softmax(z_s / 1.5, axis=1)
    q = sps.softmax(z_t / 3.0, axis=1)
    fwd = O.forward(z_s, z_t, None, variant="forward", t_student=1.5, t_teacher=3.0)["kl"]
    np.testing.assert_allclose(fwd, sst.entropy(q, p, axis=1), rtol=1e-12)


def test_js_half_matches_scipy_jensenshannon():
    z_s, z_t = _rand_logits(6, 25, 2.0), _rand_logits(6, 25, 2.0)
    p, q = sps.softmax(z_s, axis=1), sps.softmax(z_t, axis=1)
    js = O.forward(z_s, z_t, None, variant="skew_js", beta=0.5)["kl"]
    ref = np.array([ssd.jensenshannon(p[i], q[i]) ** 2 for i in range(6)])
    np.testing.assert_allclose(js, ref, rtol=1e-10)


@pytest.mark.parametrize("beta", [0.1, 0.3, 0.9])
def test_skew_variants_match_scipy(beta):
    z_s, z_t = _rand_logits(6, 25, 2.0), _rand_logits(6, 25, 2.0)
    p, q = sps.softmax(z_s / 2, axis=1), sps.softmax(z_t / 2, axis=1)
    m = (1 - beta) * q + beta * p
    sf = sst.entropy(q, m, axis=1)
    sr = sst.entropy(p, m, axis=1)
    kw = dict(beta=beta, t_student=2.0)
    np.testing.assert_allclose(O.forward(z_s, z_t, None, variant="skew_forward", **kw)["kl"],
                               sf, rtol=1e-11)
    np.testing.assert_allclose(O.forward(z_s, z_t, None, variant="skew_reverse", **kw)["kl"],
                               sr, rtol=1e-11)
    np.testing.assert_allclose(O.forward(z_s, z_t, None, variant="skew_js", **kw)["kl"],
                               (1 - beta) * sf + beta * sr, rtol=1e-11)


# ------------------------------------------------------------- invariants

@pytest.mark.parametrize("variant", O.VARIANTS)
@pytest.mark.parametrize("t", [1.0, 2.0])
def test_kl_of_identical_distributions_is_zero(variant, t):
    z = _rand_logits(5, 64, 3.0)
    out = O.forward(z, z.copy(), None, variant=variant, t_student=t, beta=0.1)
    np.testing.assert_allclose(out["kl"], 0.0, atol=1e-13)
    g, _ = O.grad_logits(z, z.copy(), None, variant=variant, t_student=t, beta=0.1,
                         w_student_ce=0.0)
    np.testing.assert_allclose(g, 0.0, atol=1e-13)


@pytest.mark.parametrize("variant", O.VARIANTS)
def test_kl_nonnegative(variant):
    z_s, z_t = _rand_logits(64, 100, 4.0), _rand_logits(64, 100, 4.0)
    kl = O.forward(z_s, z_t, None, variant=variant, beta=0.25)["kl"]
    assert np.all(kl >= -1e-13)


@pytest.mark.parametrize("beta", [0.1, 0.5])
def test_skew_js_upper_bound(beta):
    """0 <= JS_beta <= h(beta) = -b ln b - (1-b) ln(1-b) (disjoint supports attain it)."""
    h = -beta * math.log(beta) - (1 - beta) * math.log(1 - beta)
    z_s, z_t = _rand_logits(64, 50, 5.0), _rand_logits(64, 50, 5.0)
    js = O.forward(z_s, z_t, None, variant="skew_js", beta=beta)["kl"]
    assert np.all(js <= h + 1e-12) and np.all(js >= -1e-13)
    # nearly disjoint one-hot distributions approach the bound
    zs = np.full((1, 4), -200.0)
    zt = zs.copy()
    zs[0, 0] = 0.0
    zt[0, 1] = 0.0
    js = O.forward(zs, zt, None, variant="skew_js", beta=beta)["kl"][0]
    assert js == pytest.approx(h, abs=1e-12)


def test_t_squared_scaling_and_raw_per_token_kl():
    """Loss KL term is T^2 * mean(raw KL(T)); the per-token output is raw (flash_kd)."""
    z_s, z_t = _rand_logits(10, 40, 3.0), _rand_logits(10, 40, 3.0)
    for t in (1.0, 2.0, 4.0):
        out = O.forward(z_s, z_t, None, variant="forward", t_student=t,
                        w_student_ce=0.0, w_kl=1.0)
        raw = sst.entropy(sps.softmax(z_t / t, axis=1), sps.softmax(z_s / t, axis=1), axis=1)
        np.testing.assert_allclose(out["kl"], raw, rtol=1e-12)
        assert out["loss"] == pytest.approx(t * t * raw.mean(), rel=1e-12)


def test_topk_equals_dense_forward_kl_at_full_support():
    """With K = V and M = 1 the sparse objective is the dense forward KL."""
    n, v = 6, 20
    z = _rand_logits(n, v, 2.0)
    q = sps.softmax(_rand_logits(n, v, 2.0), axis=1)
    idx = np.stack([RNG.permutation(v) for _ in range(n)])
    pk = np.take_along_axis(q, idx, axis=1)
    out = O.forward(z, None, None, topk_idx=idx, topk_p=pk, w_student_ce=0.0)
    np.testing.assert_allclose(out["kl"], sst.entropy(q, sps.softmax(z, axis=1), axis=1),
                               rtol=1e-11)
    np.testing.assert_allclose(out["mass"], 1.0, rtol=1e-13)


def test_topk_lower_bound_and_gradient_rows_sum_to_zero():
    """Log-sum inequality: L >= M ln M; dL/dz = M softmax - p sums to M - M = 0."""
    n, v, k = 32, 200, 10
    z = _rand_logits(n, v, 2.0)
    idx = np.stack([RNG.choice(v, size=k, replace=False) for _ in range(n)])
    pk = sps.softmax(RNG.normal(0, 2, size=(n, k)), axis=1) * RNG.uniform(0.85, 0.99, (n, 1))
    out = O.forward(z, None, None, topk_idx=idx, topk_p=pk, w_student_ce=0.0)
    m = pk.sum(1)
    assert np.all(out["kl"] >= m * np.log(m) - 1e-12)
    g, _ = O.grad_logits(z, None, None, topk_idx=idx, topk_p=pk, w_student_ce=0.0)
    np.testing.assert_allclose(g.sum(1), 0.0, atol=1e-13)


@pytest.mark.parametrize("variant", O.VARIANTS)
def test_dense_gradient_rows_sum_to_zero(variant):
    z_s, z_t = _rand_logits(8, 30, 2.0), _rand_logits(8, 30, 2.0)
    labels = RNG.integers(0, 30, size=8)
    g, g_t = O.grad_logits(z_s, z_t, labels, variant=variant, t_student=2.0, beta=0.2,
                           w_teacher_ce=0.5)
    np.testing.assert_allclose(g.sum(1), 0.0, atol=1e-13)
    np.testing.assert_allclose(g_t.sum(1), 0.0, atol=1e-13)


def test_ignored_rows_are_exactly_zero():
    n, v, d = 6, 24, 8
    h_s, w_s, h_t = RNG.normal(size=(n, d)), RNG.normal(0, .3, (v, d)), RNG.normal(size=(n, d))
    labels = RNG.integers(0, v, size=n)
    labels[[1, 4]] = -100
    z_s, z_t = O.project(h_s, w_s), O.project(h_t, w_s)
    for variant in O.VARIANTS:
        out = O.forward(z_s, z_t, labels, variant=variant, t_student=2.0, w_teacher_ce=1.0)
        for key in ("ce_s", "ce_t", "kl"):
            assert out[key][1] == 0.0 and out[key][4] == 0.0
        g, g_t = O.grad_logits(z_s, z_t, labels, variant=variant, t_student=2.0,
                               w_teacher_ce=1.0)
        assert not g[[1, 4]].any() and not g_t[[1, 4]].any()
        d_h, _ = O.hidden_grads(h_s, w_s, g, h_t, g_t, tied=True)
        assert not d_h[[1, 4]].any()


def test_mean_denominators_and_empty_batch():
    z_s, z_t = _rand_logits(8, 16), _rand_logits(8, 16)
    labels = RNG.integers(0, 16, size=8)
    labels[:3] = -100
    s = O.forward(z_s, z_t, labels, reduction="sum")["loss"]
    assert O.forward(z_s, z_t, labels)["loss"] == pytest.approx(s / 5, rel=1e-14)
    assert O.forward(z_s, z_t, labels, num_batch_labels=40)["loss"] == pytest.approx(s / 40)
    g_sum, _ = O.grad_logits(z_s, z_t, labels, reduction="sum")
    g_mean, _ = O.grad_logits(z_s, z_t, labels)
    np.testing.assert_allclose(g_mean, g_sum / 5, rtol=1e-14)
    none = np.full(8, -100)
    assert O.forward(z_s, z_t, none)["loss"] == 0.0
    g, _ = O.grad_logits(z_s, z_t, none)
    assert not g.any()


# ---------------------------------------------------------- brute force

def _brute_row(zs, zt, label, t, variant, beta):
    """Pure-Python two-pass evaluation with math.fsum (independent arithmetic)."""
    def lsm(z):
        mx = max(z)
        s = math.fsum(math.exp(x - mx) for x in z)
        return [x - mx - math.log(s) for x in z]
    lp = lsm([x / t for x in zs])
    lq = lsm([x / t for x in zt])
    p = [math.exp(x) for x in lp]
    q = [math.exp(x) for x in lq]
    kf = math.fsum(qi * (a - b) for qi, a, b in zip(q, lq, lp))
    kr = math.fsum(pi * (a - b) for pi, a, b in zip(p, lp, lq))
    m = [(1 - beta) * qi + beta * pi for pi, qi in zip(p, q)]
    kqm = math.fsum(qi * (math.log(qi) - math.log(mi)) for qi, mi in zip(q, m))
    kpm = math.fsum(pi * (math.log(pi) - math.log(mi)) for pi, mi in zip(p, m))
    kl = {"forward": kf, "reverse": kr, "jeffreys": kf + kr, "skew_forward": kqm,
          "skew_reverse": kpm, "skew_js": (1 - beta) * kqm + beta * kpm}[variant]
    ce = -lsm(zs)[label]
    return ce, kl


@pytest.mark.parametrize("variant", O.VARIANTS)
def test_brute_force_tiny(variant):
    z_s, z_t = _rand_logits(4, 16, 2.0), _rand_logits(4, 16, 2.0)
    labels = RNG.integers(0, 16, size=4)
    out = O.forward(z_s, z_t, labels, variant=variant, t_student=1.7, beta=0.3)
    for i in range(4):
        ce, kl = _brute_row(list(z_s[i]), list(z_t[i]), int(labels[i]), 1.7, variant, 0.3)
        assert out["ce_s"][i] == pytest.approx(ce, abs=1e-12)
        assert out["kl"][i] == pytest.approx(kl, abs=1e-12)


# ------------------------------------------------------ gradient checks

def _fd(fun, x, eps=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + eps
        fp = fun()
        x[i] = old - eps
        fm = fun()
        x[i] = old
        g[i] = (fp - fm) / (2 * eps)
    return g


KINDS = ["tied", "separate", "topk", "logits"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("variant", O.VARIANTS)
def test_finite_difference_gradients(kind, variant):
    if kind == "topk" and variant != "forward":
        pytest.skip("top-K teachers carry only the forward sparse objective")
    rng = np.random.default_rng(7)
    n, v, d = 4, 16, 8
    h_s = rng.normal(size=(n, d))
    w_s = rng.normal(0, 0.4, size=(v, d))
    h_t = rng.normal(size=(n, d))
    w_t = rng.normal(0, 0.4, size=(v, d)) if kind == "separate" else w_s
    labels = rng.integers(0, v, size=n)
    labels[2] = -100
    kw = dict(variant=variant, t_student=1.6, t_teacher=1.6, beta=0.3, w_student_ce=0.7,
              w_kl=1.3, ignore_index=-100)
    idx = pk = None
    if kind == "topk":
        idx = np.stack([rng.choice(v, 5, replace=False) for _ in range(n)])
        pk = sps.softmax(rng.normal(size=(n, 5)), axis=1) * 0.9
        kw.update(topk_idx=idx, topk_p=pk, w_teacher_ce=0.0)
    else:
        kw.update(w_teacher_ce=0.4 if kind == "tied" else 0.0)
    z_t_fixed = None if kind == "topk" else O.project(h_t, w_t)  # teacher detached in KL

    def loss():
        z_s = O.project(h_s, w_s)
        out = O.forward(z_s, z_t_fixed, labels, **{**kw, "w_teacher_ce": 0.0})
        extra = 0.0
        if kind == "tied":  # the tied teacher's CE reaches the shared weight
            ce_t = O.cross_entropy_rows(O.project(h_t, w_s), labels, labels != -100)
            extra = kw["w_teacher_ce"] * ce_t.sum() / max((labels != -100).sum(), 1)
        return out["loss"] + extra

    g_s, g_t = O.grad_logits(O.project(h_s, w_s), z_t_fixed, labels, **kw)
    d_h, d_w = O.hidden_grads(h_s, w_s, g_s, h_t, g_t, tied=(kind == "tied"))
    np.testing.assert_allclose(d_h, _fd(loss, h_s), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(d_w, _fd(loss, w_s), rtol=1e-6, atol=1e-8)
    # gradient w.r.t. the student logits themselves
    z_s = O.project(h_s, w_s)
    fl = lambda: O.forward(z_s, z_t_fixed, labels, **{**kw, "w_teacher_ce": 0.0})["loss"]
    g_only_s, _ = O.grad_logits(z_s, z_t_fixed, labels, **{**kw, "w_teacher_ce": 0.0})
    np.testing.assert_allclose(g_only_s, _fd(fl, z_s), rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("variant", ["forward", "reverse", "jeffreys"])
def test_gradients_match_torch_autograd(variant):
    """Library pin: torch fp64 log_softmax / kl_div / cross_entropy + autograd."""
    rng = np.random.default_rng(11)
    n, v, t = 6, 20, 2.0
    z_s = rng.normal(0, 2, size=(n, v))
    z_t = rng.normal(0, 2, size=(n, v))
    labels = rng.integers(0, v, size=n)
    labels[0] = -100
    zs = torch.tensor(z_s, requires_grad=True)
    lab = torch.from_numpy(labels)
    valid = lab != -100
    lp = torch.log_softmax(zs / t, dim=1)
    lq = torch.log_softmax(torch.from_numpy(z_t) / t, dim=1)
    fwd = torch.nn.functional.kl_div(lp, lq, log_target=True, reduction="none").sum(1)
    rev = torch.nn.functional.kl_div(lq, lp, log_target=True, reduction="none").sum(1)
    kl = {"forward": fwd, "reverse": rev, "jeffreys": fwd + rev}[variant]
    ce = torch.nn.functional.cross_entropy(zs, lab, ignore_index=-100, reduction="none")
    loss = ((ce + t * t * kl) * valid).sum() / valid.sum()
    loss.backward()
    out = O.forward(z_s, z_t, labels, variant=variant, t_student=t)
    assert out["loss"] == pytest.approx(loss.item(), rel=1e-12)
    g, _ = O.grad_logits(z_s, z_t, labels, variant=variant, t_student=t)
    np.testing.assert_allclose(g, zs.grad.numpy(), rtol=1e-10, atol=1e-14)


def test_no_teacher_is_plain_cross_entropy():
    """Without a teacher the loss is the mean CE, matching torch's cross_entropy."""
    z = _rand_logits(12, 30, 2.0)
    labels = RNG.integers(0, 30, size=12)
    labels[[0, 5]] = -100
    out = O.forward(z, None, labels)
    ref = torch.nn.functional.cross_entropy(torch.from_numpy(z), torch.from_numpy(labels))
    assert out["loss"] == pytest.approx(ref.item(), rel=1e-12)
    assert not out["kl"].any()
    zt = torch.tensor(z, requires_grad=True)
    torch.nn.functional.cross_entropy(zt, torch.from_numpy(labels)).backward()
    g, _ = O.grad_logits(z, None, labels)
    np.testing.assert_allclose(g, zt.grad.numpy(), rtol=1e-10, atol=1e-14)


# ---------------------------------------------------------------- token-map projection

def test_projection_identity_map_is_tempered_logits():
    """With every teacher token mapped to the student id of the same index, the
    projection is the tempered logits themselves."""
    z = _rand_logits(3, 11, std=3.0)
    out = O.project_teacher_logits(z, np.arange(11), 11, temperature=1.7)
    np.testing.assert_allclose(out, z / 1.7, rtol=0, atol=1e-13)


def test_projection_brute_force_with_duplicates_and_unmatched():
    """Pure-Python sum of exponentials per student id (math.fsum) on a map with
    repeated ids, unmatched teacher tokens and student ids nothing maps to."""
    rng = np.random.default_rng(77)
    v_t, v_s, T = 13, 7, 2.0
    tmap = np.array([3, -1, 0, 3, 5, 0, 0, -1, 6, 3, 1, -1, 5])  # id 2 and 4 unmatched
    z = rng.normal(0.0, 2.0, size=(4, v_t))
    out = O.project_teacher_logits(z, tmap, v_s, temperature=T)
    for n in range(z.shape[0]):
        for i in range(v_s):
            src = [j for j in range(v_t) if tmap[j] == i]
            if not src:
                assert out[n, i] == -math.inf
            else:
                ref = math.log(math.fsum(math.exp(z[n, j] / T) for j in src))
                assert abs(out[n, i] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_projection_moves_teacher_probability_mass():
    """softmax of the projected row = the tempered teacher distribution summed
    over each id's teacher tokens, renormalised over the matched tokens
    (scipy softmax on the teacher vocabulary)."""
    rng = np.random.default_rng(5)
    v_t, v_s, T = 40, 25, 1.5
    tmap = rng.integers(-1, v_s, size=v_t)
    z = rng.normal(0.0, 3.0, size=(5, v_t))
    q_t = sps.softmax(z / T, axis=1)
    matched = tmap >= 0
    q_ref = np.zeros((5, v_s))
    for j in np.flatnonzero(matched):
        q_ref[:, tmap[j]] += q_t[:, j]
    q_ref /= q_t[:, matched].sum(axis=1, keepdims=True)
    q = sps.softmax(O.project_teacher_logits(z, tmap, v_s, temperature=T), axis=1)
    np.testing.assert_allclose(q, q_ref, rtol=1e-12, atol=1e-15)


def test_projected_teacher_kl_drops_zero_probability_ids():
    """Forward KL(q'||p) of a projected teacher with unmatched student ids is finite
    and equals the brute-force sum over the ids that carry teacher mass."""
    rng = np.random.default_rng(9)
    v_t, v_s = 9, 6
    tmap = np.array([0, 0, 1, 2, -1, 2, 4, 4, 1])  # student ids 3 and 5 unmatched
    z_t = rng.normal(0.0, 2.0, size=(2, v_t))
    a_s = rng.normal(0.0, 2.0, size=(2, v_s))
    a_t = O.project_teacher_logits(z_t, tmap, v_s)
    kl, _ = O.kl_rows(a_s, a_t, "forward")
    for n in range(2):
        q = sps.softmax(a_t[n])
        p = sps.softmax(a_s[n])
        ref = math.fsum(q[i] * (math.log(q[i]) - math.log(p[i])) for i in range(v_s) if q[i] > 0)
        assert np.isfinite(kl[n]) and abs(kl[n] - ref) <= 1e-12


# ---------------------------------------------------------------- multi-teacher mixing

@pytest.mark.parametrize("mode", O.MIX_MODES)
def test_mix_of_one_teacher_is_its_log_softmax(mode):
    """A single teacher (any positive weight) is returned as its own
    log-probabilities (scipy log_softmax)."""
    z = _rand_logits(4, 13, std=3.0)
    out = O.mix_teacher_logits([z], [2.5], mode)
    np.testing.assert_allclose(out, sps.log_softmax(z, axis=-1), rtol=0, atol=1e-13)


def test_mix_hand_worked_example():
    """Two teachers over three tokens with known probabilities, weights 1 : 3.
    Probability average: 0.25 [.5 .25 .25] + 0.75 [.1 .2 .7] = [.2 .2125 .5875].
    Product of experts: p1^(1/4) p2^(3/4) per token, divided by its sum
    (math.pow products, not the oracle's log-space sum)."""
    p1, p2 = [0.5, 0.25, 0.25], [0.1, 0.2, 0.7]
    z1 = np.log([p1]) + 5.0  # logits = log-probabilities up to a row constant
    z2 = np.log([p2]) - 2.0
    ari = np.exp(O.mix_teacher_logits([z1, z2], [1.0, 3.0], "arithmetic"))[0]
    np.testing.assert_allclose(ari, [0.2, 0.2125, 0.5875], rtol=1e-14, atol=0)
    r = [math.pow(a, 0.25) * math.pow(b, 0.75) for a, b in zip(p1, p2)]
    geo = np.exp(O.mix_teacher_logits([z1, z2], [1.0, 3.0], "geometric"))[0]
    np.testing.assert_allclose(geo, [x / math.fsum(r) for x in r], rtol=1e-13, atol=0)


def test_mix_brute_force_probabilities():
    """Three teachers with random logits and weights: the arithmetic mixture is
    sum_k w_k softmax(z_k) and the geometric one prod_k softmax(z_k)^w_k
    renormalised, both computed token by token in probability space."""
    rng = np.random.default_rng(31)
    zs = [rng.normal(0.0, 2.0, size=(3, 7)) for _ in range(3)]
    w = np.array([0.2, 1.3, 0.5])
    wn = w / w.sum()
    ari = O.mix_teacher_logits(zs, w, "arithmetic")
    geo = O.mix_teacher_logits(zs, w, "geometric")
    for n in range(3):
        qs = [sps.softmax(z[n]) for z in zs]
        mix = [math.fsum(wn[k] * qs[k][v] for k in range(3)) for v in range(7)]
        np.testing.assert_allclose(np.exp(ari[n]), mix, rtol=1e-13, atol=0)
        poe = [math.prod(math.pow(qs[k][v], wn[k]) for k in range(3)) for v in range(7)]
        np.testing.assert_allclose(np.exp(geo[n]), [x / math.fsum(poe) for x in poe], rtol=1e-12)


@pytest.mark.parametrize("mode", O.MIX_MODES)
def test_mix_invariances_and_zero_weight(mode):
    """Shifting a teacher's row by a constant or scaling all weights changes
    nothing; a teacher with weight 0 takes no part; the output is a normalised
    log-distribution."""
    rng = np.random.default_rng(5)
    zs = [rng.normal(0.0, 3.0, size=(5, 17)) for _ in range(3)]
    base = O.mix_teacher_logits(zs[:2], [0.3, 0.7], mode)
    shifted = O.mix_teacher_logits([zs[0] + 4.0, zs[1] - 11.0], [3.0, 7.0], mode)
    np.testing.assert_allclose(shifted, base, rtol=0, atol=1e-12)
    with_zero = O.mix_teacher_logits([zs[0], zs[2] * 50.0, zs[1]], [0.3, 0.0, 0.7], mode)
    np.testing.assert_allclose(with_zero, base, rtol=0, atol=1e-12)
    np.testing.assert_allclose(sps.logsumexp(base, axis=-1), 0.0, atol=1e-13)


def test_mix_of_projected_teachers_with_zero_probability_ids():
    """Ids with probability 0 (-inf logits, as projection gives unmatched ids):
    the probability average keeps an id that any teacher supports, the product
    of experts drops an id that any teacher with weight > 0 rules out."""
    z1 = np.array([[0.0, -np.inf, 1.0, -np.inf]])
    z2 = np.array([[0.5, 2.0, -np.inf, -np.inf]])
    ari = O.mix_teacher_logits([z1, z2], None, "arithmetic")[0]
    geo = O.mix_teacher_logits([z1, z2], None, "geometric")[0]
    q1, q2 = sps.softmax(z1[0]), sps.softmax(z2[0])
    np.testing.assert_allclose(np.exp(ari), 0.5 * q1 + 0.5 * q2, rtol=1e-14)
    assert np.isneginf(ari[3]) and np.all(np.isfinite(ari[:3]))
    assert np.all(np.isneginf(geo[1:])) and geo[0] == 0.0


# ---------------------------------------------------------------- teacher gradients

@pytest.mark.parametrize("kind", ["separate", "tied"])
@pytest.mark.parametrize("variant", ["forward", "jeffreys", "skew_reverse"])
def test_teacher_gradients_finite_differences(kind, variant):
    """d loss / d H_t and d loss / d W_t (separate) of a teacher trained by its
    CE term, against central differences of the loss with the teacher detached
    from the KL: only w_tce * mean CE_t moves with the teacher."""
    rng = np.random.default_rng(17)
    n, v, d = 5, 12, 6
    h_s, h_t = rng.normal(size=(n, d)), rng.normal(size=(n, d))
    w_s = rng.normal(0, 0.4, size=(v, d))
    w_t = rng.normal(0, 0.4, size=(v, d)) if kind == "separate" else w_s
    labels = rng.integers(0, v, size=n)
    labels[3] = -100
    kw = dict(variant=variant, t_student=1.5, t_teacher=1.5, beta=0.3, w_student_ce=0.7,
              w_teacher_ce=0.45, w_kl=1.2, ignore_index=-100)
    z_s = O.project(h_s, w_s)
    z_t_kl = O.project(h_t, w_t)  # what the KL sees: fixed while the teacher moves

    def loss():
        out = O.forward(z_s, z_t_kl, labels, **{**kw, "w_teacher_ce": 0.0})
        ce_t = O.cross_entropy_rows(O.project(h_t, w_t), labels, labels != -100)
        return out["loss"] + kw["w_teacher_ce"] * ce_t.sum() / (labels != -100).sum()

    _, g_t = O.grad_logits(z_s, z_t_kl, labels, **kw)
    d_ht, d_wt = O.teacher_hidden_grads(h_t, w_t, g_t)
    np.testing.assert_allclose(d_ht, _fd(loss, h_t), rtol=1e-6, atol=1e-8)
    if kind == "separate":
        np.testing.assert_allclose(d_wt, _fd(loss, w_t), rtol=1e-6, atol=1e-8)
