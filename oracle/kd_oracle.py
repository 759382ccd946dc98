"""Plain fp64 CPU oracle of the fused LM-head + cross-entropy + KL distillation loss.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library
never calls it, and it shares no code with the CUDA library.

Every function materialises full logit rows in float64 from the exact stored
input values (bf16 / fp32 upcast without rounding) and evaluates the loss by
its textbook definition, row by row.  Rows are independent, so callers may
pass any subset of rows; nothing here blocks, fuses or reorders the vocabulary
reduction.

Notation (orda-kernel README, "KL variants": p = student, q = teacher):
    z_s = H_s W_s^T, z_t = H_t W_t^T          student / teacher logits
    a_s = z_s / T_s, a_t = z_t / T_t           tempered logits
    p = softmax(a_s), q = softmax(a_t)

Sources (page title, section):
  * orda-kernel README (pypi.org/project/orda-kernel): "KL variants" table
    (forward KL(q||p), reverse KL(p||q), Jeffreys, skew-forward
    KL(q||(1-b)q+bp), skew-reverse KL(p||(1-b)q+bp), skew-JS);
    "Parameters" (term weights, kl_temperature with each KL row scaled by
    T_s^2, ignore_index, reduction "mean"/"sum"); "Teacher descriptors"
    (tied / separate / precomputed; the teacher is detached in KL, and a
    tied teacher's CE term trains the shared weight).
  * flash_kd API doc, flash_ce_kd_loss: per-token CE = standard cross
    entropy with ignored tokens giving 0; per-token KD = KL(P_T||P_S) NOT
    multiplied by T^2.
  * Full-Chunked-KL-Loss README, "Methods": sparse top-K objective
    L = sum_S p log p - sum_S p z + M logsumexp(z), M = sum_S p not
    renormalised; "Full Chunked KL": closed-form gradient M softmax(z) - p.
  * nemo_automodel kd_loss API doc, KDLoss: loss multiplied by T^2; mean
    over valid tokens, or sum / num_batch_labels.
  * orda-kernel README, "Cross-vocabulary distillation": token-map
    projection (duplicates sum in probability space, unmatched ids -inf,
    tempering before aggregation) and multi-teacher mixing (probability
    average or product of experts of cached teacher distributions).

Readings where the pages are silent (each is also listed in the design notes):
  * Skew-JS(beta) = (1-beta) KL(q||m) + beta KL(p||m), m = (1-beta) q + beta p.
  * CE always uses T = 1 (raw logits); only the KL uses temperatures.
  * Ignored tokens give 0 CE, 0 KL and a 0 gradient row; the mean divides by
    the number of valid tokens (num_batch_labels overrides it); with no valid
    token the loss and every gradient are 0.
  * The loss is sum_valid(w_sce CE_s + w_tce CE_t + w_kl T_s^2 KL) / denom.
  * Top-K teachers use a_s = z_s / T_s in the objective (T_s = 1 in the
    pages' workload) and no labels unless CE is requested.
  * Multi-teacher mixing normalises its weights to sum to 1 and returns the
    mixture's log-probabilities; a teacher with weight 0 takes no part.

Parity pins: every function here is checked against closed forms, scipy
library routines, finite differences and brute force in
tests/test_oracle_pins.py.  No function is left unpinned.
"""
from __future__ import annotations

import numpy as np

VARIANTS = ("forward", "reverse", "jeffreys", "skew_js", "skew_forward", "skew_reverse")


# ----------------------------------------------------------------------------
# basic definitions
# ----------------------------------------------------------------------------

def as_f64(x):
    """Exact fp64 copy of an array (torch tensors are upcast on the CPU)."""
    if hasattr(x, "detach"):  # torch tensor: upcast exactly, then hand to numpy
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def project(h, w):
    """Logits z = H W^T (the LM-head projection), in fp64."""
    return as_f64(h) @ as_f64(w).T


def logsumexp(x):
    """Row-wise log sum_v exp(x_v), shifted by the row max for range."""
    m = np.max(x, axis=-1, keepdims=True)
    return m[..., 0] + np.log(np.sum(np.exp(x - m), axis=-1))


def log_softmax(x):
    return x - logsumexp(x)[..., None]


def _xlogy_rows(a, log_a_minus_log_b):
    """sum_v a_v (log a_v - log b_v) with the 0 log 0 = 0 convention."""
    with np.errstate(invalid="ignore"):  # 0 * -inf in the discarded branch
        return np.sum(np.where(a > 0, a * log_a_minus_log_b, 0.0), axis=-1)


# ----------------------------------------------------------------------------
# per-row KL variants in tempered space (orda-kernel README, "KL variants")
# ----------------------------------------------------------------------------

def kl_rows(a_s, a_t, variant, beta=0.5):
    """Per-row divergence between p = softmax(a_s) (student) and q = softmax(a_t).

    Returns (kl, aux) where aux holds quantities the backward needs:
    log p, log q, p, q, reverse KL, KL(p||m) and log m (skew variants).
    """
    logp = log_softmax(a_s)
    logq = log_softmax(a_t)
    p, q = np.exp(logp), np.exp(logq)
    aux = {"logp": logp, "logq": logq, "p": p, "q": q}
    kl_f = _xlogy_rows(q, logq - logp)            # KL(q || p)
    kl_r = _xlogy_rows(p, logp - logq)            # KL(p || q)
    aux["kl_rev"] = kl_r
    if variant in ("skew_js", "skew_forward", "skew_reverse"):
        # m = (1-beta) q + beta p, evaluated in log space for range
        logm = np.logaddexp(np.log1p(-beta) + logq, np.log(beta) + logp)
        kl_qm = _xlogy_rows(q, logq - logm)       # KL(q || m)
        kl_pm = _xlogy_rows(p, logp - logm)       # KL(p || m)
        aux.update(logm=logm, kl_qm=kl_qm, kl_pm=kl_pm)
    if variant == "forward":
        return kl_f, aux
    if variant == "reverse":
        return kl_r, aux
    if variant == "jeffreys":
        return kl_f + kl_r, aux
    if variant == "skew_forward":
        return kl_qm, aux
    if variant == "skew_reverse":
        return kl_pm, aux
    if variant == "skew_js":
        return (1.0 - beta) * kl_qm + beta * kl_pm, aux
    raise ValueError(f"unknown variant {variant!r}")


def kl_grad_rows(variant, aux, beta=0.5):
    """d KL / d a_s for the teacher-detached variants (a-space, per row).

    Derivations (softmax Jacobian dp_v/da_j = p_v (delta_vj - p_j)):
      forward  KL(q||p) = -sum q log p + const          ->  p - q
      reverse  KL(p||q) = sum p (log p - log q)         ->  p (log p - log q - KL(p||q))
      skew_fwd KL(q||m), dm_v/da_j = beta p_v(delta_vj - p_j)
                                                         ->  -beta p (q/m - sum_v p_v q_v/m_v)
      skew_rev KL(p||m)                                  ->  p (log p - log m - KL(p||m))
                                                              - beta p (p/m - sum_v p_v^2/m_v)
      skew_js  (1-beta) skew_fwd + beta skew_rev         ->  beta p (log p - log m - KL(p||m))
    """
    p, q, logp, logq = aux["p"], aux["q"], aux["logp"], aux["logq"]
    if variant == "forward":
        return p - q
    if variant in ("reverse", "jeffreys"):
        g_r = p * (logp - logq - aux["kl_rev"][:, None])
        return g_r if variant == "reverse" else (p - q) + g_r
    logm = aux["logm"]
    m = np.exp(logm)
    if variant == "skew_forward":
        return -beta * p * (q / m - np.sum(p * q / m, axis=-1, keepdims=True))
    if variant == "skew_reverse":
        return (p * (logp - logm - aux["kl_pm"][:, None])
                - beta * p * (p / m - np.sum(p * p / m, axis=-1, keepdims=True)))
    if variant == "skew_js":
        return beta * p * (logp - logm - aux["kl_pm"][:, None])
    raise ValueError(f"unknown variant {variant!r}")


# ----------------------------------------------------------------------------
# cross-vocabulary token map (orda-kernel README, "Cross-vocabulary
# distillation", token-map projection)
# ----------------------------------------------------------------------------

def project_teacher_logits(z_t, token_map, v_student, temperature=1.0):
    """Teacher logits over the teacher vocabulary -> logits over the student
    vocabulary.  token_map[j] is the student id of teacher token j, or -1.
    The teacher logits are tempered first (z / T), then each student id i
    receives log sum_{j: map[j] = i} exp(z_j / T): duplicate teacher tokens of
    one id sum in probability space, and an id no teacher token maps to gets
    -inf (probability 0).  Written out per student id with numpy's grouped
    reductions over the teacher columns sorted by student id.
    """
    z = as_f64(z_t) / float(temperature)
    tm = np.asarray(token_map, dtype=np.int64)
    out = np.full((z.shape[0], int(v_student)), -np.inf)
    cols = np.flatnonzero(tm >= 0)
    if cols.size == 0:
        return out
    ids = tm[cols]
    order = np.argsort(ids, kind="stable")
    cols, ids = cols[order], ids[order]
    starts = np.flatnonzero(np.r_[True, ids[1:] != ids[:-1]])
    lengths = np.diff(np.r_[starts, ids.size])
    zz = z[:, cols]
    m = np.maximum.reduceat(zz, starts, axis=1)                 # per-id maximum
    s = np.add.reduceat(np.exp(zz - np.repeat(m, lengths, axis=1)), starts, axis=1)
    out[:, ids[starts]] = m + np.log(s)
    return out


# ----------------------------------------------------------------------------
# multi-teacher mixing (orda-kernel README, "Cross-vocabulary distillation",
# multi-teacher mixing)
# ----------------------------------------------------------------------------

MIX_MODES = ("arithmetic", "geometric")


def mix_teacher_logits(logits, weights=None, mode="arithmetic"):
    """Mix K cached teacher distributions over one vocabulary into one, returned
    as normalised log-probabilities (logits of the mixture).  Teacher k gives
    q_k = softmax(z_k); the weights are non-negative and are normalised to sum
    to 1 (uniform when omitted).
      arithmetic (probability average): q = sum_k w_k q_k
      geometric (product of experts):  q proportional to prod_k q_k ** w_k
    """
    zs = [as_f64(z) for z in logits]
    k = len(zs)
    if k == 0:
        raise ValueError("need at least one teacher")
    w = np.ones(k) if weights is None else np.asarray(weights, dtype=np.float64)
    if w.shape != (k,) or np.any(w < 0) or not np.any(w > 0):
        raise ValueError("weights: k non-negative values, not all zero")
    w = w / w.sum()
    if mode == "arithmetic":
        # log sum_k w_k exp(log q_k), over the teachers with w_k > 0
        terms = np.stack([np.log(w[i]) + log_softmax(zs[i]) for i in range(k) if w[i] > 0])
        top = terms.max(axis=0)
        with np.errstate(invalid="ignore", divide="ignore"):
            shifted = np.where(np.isneginf(top), -np.inf, terms - top)
            return top + np.log(np.exp(shifted).sum(axis=0))
    if mode == "geometric":
        # log prod_k q_k^{w_k} = sum_k w_k log q_k, then normalised
        g = sum(w[i] * log_softmax(zs[i]) for i in range(k) if w[i] > 0)
        return g - logsumexp(g)[:, None]
    raise ValueError(f"unknown mode {mode!r}")


# ----------------------------------------------------------------------------
# sparse top-K teacher (Full-Chunked-KL-Loss README, "Methods")
# ----------------------------------------------------------------------------

def topk_rows(a, idx, pk):
    """L = sum_S p log p - sum_S p a_S + M logsumexp(a), M = sum_S p (no renormalisation)."""
    idx = np.asarray(idx, dtype=np.int64)
    pk = as_f64(pk)
    mass = pk.sum(axis=-1)
    ent = np.sum(np.where(pk > 0, pk * np.log(np.where(pk > 0, pk, 1.0)), 0.0), axis=-1)
    cross = np.sum(pk * np.take_along_axis(a, idx, axis=-1), axis=-1)
    return ent - cross + mass * logsumexp(a), mass


def topk_grad_rows(a, idx, pk):
    """dL/da = M softmax(a) - p scattered onto the support (Full Chunked KL)."""
    idx = np.asarray(idx, dtype=np.int64)
    pk = as_f64(pk)
    mass = pk.sum(axis=-1, keepdims=True)
    g = mass * np.exp(log_softmax(a))
    rows = np.arange(a.shape[0])[:, None]
    np.add.at(g, (np.broadcast_to(rows, idx.shape), idx), -pk)
    return g


# ----------------------------------------------------------------------------
# full loss: forward
# ----------------------------------------------------------------------------

def _weighted(w, x):
    """w * x, with a zero weight giving 0 whatever x is."""
    return w * np.asarray(x) if w != 0 else np.zeros_like(np.asarray(x, dtype=np.float64))


def _valid_mask(labels, n, ignore_index):
    if labels is None:
        return np.ones(n, dtype=bool)
    return np.asarray(labels, dtype=np.int64) != ignore_index


def cross_entropy_rows(z, labels, valid):
    """CE = logsumexp(z) - z_label (T = 1); 0 on ignored rows (flash_ce_kd_loss)."""
    lse = logsumexp(z)
    safe = np.where(valid, np.asarray(labels, dtype=np.int64), 0)
    picked = np.take_along_axis(z, safe[:, None], axis=-1)[:, 0]
    return np.where(valid, lse - picked, 0.0)


def loss_denominator(valid, reduction="mean", num_batch_labels=None):
    if reduction == "sum":
        return 1.0
    if num_batch_labels is not None and num_batch_labels > 0:
        return float(num_batch_labels)
    return float(max(int(np.sum(valid)), 1))


def forward(z_s, z_t=None, labels=None, *, topk_idx=None, topk_p=None,
            variant="forward", t_student=1.0, t_teacher=None, beta=0.5,
            w_student_ce=1.0, w_teacher_ce=0.0, w_kl=1.0, ignore_index=-100,
            reduction="mean", num_batch_labels=None):
    """Per-token CE_s, CE_t, raw KL and the scalar loss from full fp64 logits.

    z_s: [N, V] student logits; z_t: [N, V] teacher logits (None for top-K, and
    None without top-K for a plain CE with no teacher).
    Returns a dict: ce_s, ce_t, kl (per token, raw: no T^2), loss (scalar),
    lse_s1, lse_sT, lse_t1, lse_tT, kl_rev, kl_pm, mass, valid.
    """
    z_s = as_f64(z_s)
    n = z_s.shape[0]
    t_teacher = t_student if t_teacher is None else t_teacher
    valid = _valid_mask(labels, n, ignore_index)
    a_s = z_s / t_student
    out = {"valid": valid, "lse_s1": logsumexp(z_s), "lse_sT": logsumexp(a_s)}
    out["ce_s"] = (cross_entropy_rows(z_s, labels, valid) if labels is not None
                   else np.zeros(n))
    if topk_idx is not None:
        kl, mass = topk_rows(a_s, topk_idx, topk_p)
        out.update(ce_t=np.zeros(n), mass=mass)
    elif z_t is None:  # no teacher: plain CE (orda-kernel "Parameters": kl_weight 0.0)
        kl = np.zeros(n)
        out.update(ce_t=np.zeros(n))
    else:
        z_t = as_f64(z_t)
        a_t = z_t / t_teacher
        kl, aux = kl_rows(a_s, a_t, variant, beta)
        out.update(lse_t1=logsumexp(z_t), lse_tT=logsumexp(a_t), kl_rev=aux["kl_rev"])
        if "kl_pm" in aux:
            out["kl_pm"] = aux["kl_pm"]
        out["ce_t"] = (cross_entropy_rows(z_t, labels, valid) if labels is not None
                       else np.zeros(n))
    kl = np.where(valid, kl, 0.0)
    out["kl"] = kl
    # a term with weight 0 is absent (its CE may be infinite, e.g. a projected
    # teacher with no mass on the label)
    per_token = (_weighted(w_student_ce, out["ce_s"]) + _weighted(w_teacher_ce, out["ce_t"])
                 + _weighted(w_kl * t_student ** 2, kl))
    out["loss"] = float(np.sum(np.where(valid, per_token, 0.0))
                        / loss_denominator(valid, reduction, num_batch_labels))
    return out


# ----------------------------------------------------------------------------
# full loss: backward (gradients w.r.t. student logits, then dH, dW)
# ----------------------------------------------------------------------------

def grad_logits(z_s, z_t=None, labels=None, *, topk_idx=None, topk_p=None,
                variant="forward", t_student=1.0, t_teacher=None, beta=0.5,
                w_student_ce=1.0, w_teacher_ce=0.0, w_kl=1.0, ignore_index=-100,
                reduction="mean", num_batch_labels=None, d_loss=1.0):
    """G_s = d loss / d z_s and G_t = d loss / d z_t through the teacher CE only.

    The teacher is detached in every KL variant (orda-kernel README, "KL
    variants"); only the teacher CE term reaches teacher logits.  The KL term
    enters the loss as w_kl T_s^2 KL(a), so its z-space gradient is
    w_kl T_s dKL/da_s.
    """
    z_s = as_f64(z_s)
    n = z_s.shape[0]
    t_teacher = t_student if t_teacher is None else t_teacher
    valid = _valid_mask(labels, n, ignore_index)
    scale = d_loss / loss_denominator(valid, reduction, num_batch_labels)
    row = np.where(valid, scale, 0.0)[:, None]
    a_s = z_s / t_student
    if topk_idx is not None:
        g_a = topk_grad_rows(a_s, topk_idx, topk_p)
    elif z_t is None:  # no teacher: no KL term
        g_a = np.zeros_like(z_s)
    else:
        z_t = as_f64(z_t)
        _, aux = kl_rows(a_s, z_t / t_teacher, variant, beta)
        g_a = kl_grad_rows(variant, aux, beta)
    g_s = w_kl * t_student * g_a
    if w_student_ce > 0 and labels is not None:
        g_s = g_s + w_student_ce * _ce_grad(z_s, labels, valid)
    g_t = None
    if z_t is not None and w_teacher_ce > 0 and labels is not None:
        g_t = row * w_teacher_ce * _ce_grad(as_f64(z_t), labels, valid)
    return row * g_s, g_t


def _ce_grad(z, labels, valid):
    """d CE / d z = softmax(z) - onehot(label)."""
    g = np.exp(log_softmax(z))
    rows = np.nonzero(valid)[0]
    g[rows, np.asarray(labels, dtype=np.int64)[rows]] -= 1.0
    return g


def hidden_grads(h_s, w_s, g_s, h_t=None, g_t=None, tied=False):
    """dH_s = G_s W_s and dW_s = G_s^T H_s (+ G_t^T H_t for a tied teacher's CE)."""
    h_s, w_s = as_f64(h_s), as_f64(w_s)
    d_h = g_s @ w_s
    d_w = g_s.T @ h_s
    if tied and g_t is not None:
        d_w = d_w + g_t.T @ as_f64(h_t)
    return d_h, d_w


def teacher_hidden_grads(h_t, w_t, g_t):
    """Gradients reaching a trained teacher (orda-kernel README, "Teacher
    descriptors": teacher_ce_weight > 0 trains the teacher through its CE; the
    KL variants detach it): with G_t = d loss / d z_t from grad_logits,
    dH_t = G_t W_t and dW_t = G_t^T H_t (W_t = W_s for a tied teacher)."""
    h_t, w_t = as_f64(h_t), as_f64(w_t)
    g_t = np.broadcast_to(as_f64(g_t), (h_t.shape[0], w_t.shape[0]))  # 0 without a teacher CE
    return g_t @ w_t, g_t.T @ h_t
