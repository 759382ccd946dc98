"""Cross-vocabulary token-map projection on the GPU against the oracle
(orda-kernel README, "Cross-vocabulary distillation", token-map projection):
the projection itself element by element, and the whole cross-tokenizer
distillation -- teacher logits over the teacher vocabulary projected onto the
student vocabulary, then the fused CE + KL loss and its gradient -- against the
oracle's own projection and loss on the same inputs."""
import numpy as np
import pytest
import torch

from lm_head_cross_vocab_gb300 import kd
from oracle import kd_oracle as O
from tests.parity_util import GRAD_TOL, TOK_TOL, rel_l2, token_rel_err

pytestmark = pytest.mark.gpu

DT = {"fp32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kd.load_library()
    assert kd.kd_device_supported(0), "tests need an sm_103 GPU"


def _map(v_t, v_s, seed):
    """Seeded token map with repeated student ids, unmatched teacher tokens and
    student ids that no teacher token reaches."""
    rng = np.random.default_rng(seed)
    tmap = rng.integers(0, v_s, size=v_t)
    tmap[rng.random(v_t) < 0.15] = -1
    tmap[np.isin(tmap, rng.choice(v_s, v_s // 10, replace=False))] = -1  # ~10 % ids unmatched
    return tmap.astype(np.int32)


@pytest.mark.parametrize("din,dout", [("fp32", "fp32"), ("bf16", "fp32"), ("bf16", "bf16")])
@pytest.mark.parametrize("v_t,v_s,n", [(1000, 700, 37), (513, 2049, 37), (60000, 70001, 5),
                                       (120000, 5000, 6), (220000, 3000, 3), (430000, 2000, 2),
                                       (30000, 20000, 400)])
def test_projection_matches_oracle(din, dout, v_t, v_s, n):
    """Teacher rows held by one CTA (1000 / 513 ids, the latter unaligned), by
    clusters of 2 to 7 CTAs exchanging their gathered values (60000 to 220000
    ids), rows too long for a cluster of 8 on the slice path (220000 fp32,
    430000 ids: 12 to 18 slices), ragged student vocabularies, and 400 rows
    per launch."""
    g = torch.Generator().manual_seed(v_t + v_s)
    z = (torch.randn(n, v_t, generator=g) * 3.0).to(DT[din])
    tmap = _map(v_t, v_s, 11)
    out = kd.project_teacher_logits(torch.from_numpy(tmap), z.cuda(), v_s, temperature=1.5,
                                    out_dtype=DT[dout])
    torch.cuda.synchronize()
    got = out.cpu().double().numpy()
    ref = O.project_teacher_logits(z, tmap, v_s, temperature=1.5)
    empty = np.isneginf(ref)
    assert empty.any() and (~empty).any()
    assert np.all(got[empty] <= -1e38), "unmatched ids must carry no probability"
    tol = 1e-6 if dout == "fp32" else 2.0 ** -8
    err = np.abs(got[~empty] - ref[~empty]) / np.maximum(1.0, np.abs(ref[~empty]))
    assert err.max() <= tol, err.max()


def test_projection_flags_bad_map_entry():
    tmap = _map(300, 200, 3)
    tmap[17] = 200  # outside [-1, V_s)
    z = torch.randn(4, 300, device="cuda")
    with pytest.raises(kd.KDError):
        kd.project_teacher_logits(torch.from_numpy(tmap), z, 200)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("variant", ["forward", "skew_js", "skew_reverse", "jeffreys"])
@pytest.mark.parametrize("v_s,T", [(700, 2.0), (704, 2.0), (704, 1.0)])
def test_cross_vocab_distillation_end_to_end(dtype, variant, v_s, T):
    """Project teacher logits (T, tempered before aggregation) and distil into
    student logits with T_s = T and the projected teacher at T_t = 1.  Rows of
    700 ids take the plain streaming kernels, rows of 704 the TMA-staged ring
    (16-byte rows); at T = 1 both sides share the packed bf16 forms, whose
    unmatched-id teacher value (the lowest finite one) must carry no mass."""
    n, v_t = 67, 900
    g = torch.Generator().manual_seed(2024)
    z_s = (torch.randn(n, v_s, generator=g) * 4.0).to(DT[dtype])
    z_tv = (torch.randn(n, v_t, generator=g) * 4.0).to(DT[dtype])
    labels = torch.randint(0, v_s, (n,), generator=g)
    labels[torch.rand(n, generator=g) < 0.08] = -100
    tmap = _map(v_t, v_s, 5)
    dev = torch.device("cuda:0")
    proj = kd.project_teacher_logits(torch.from_numpy(tmap), z_tv.to(dev), v_s, temperature=T)
    t = {"logits_s": z_s.to(dev), "logits_t": proj, "labels": labels.to(dev)}
    prob = kd.Problem(n_tokens=n, vocab=v_s, d_student=0, d_teacher=0, topk=0, dtype=dtype,
                      student="logits", teacher="logits", variant=variant, t_student=T,
                      t_teacher=1.0, w_student_ce=0.5, w_teacher_ce=0.0, w_kl=1.0, beta=0.1,
                      ignore_index=-100)
    fwd = kd.forward(prob, t)
    bwd = kd.backward(prob, t, fwd["stats"], want=("logits_s",))
    torch.cuda.synchronize()
    # oracle: its own projection of the same teacher bytes, stored in the
    # problem dtype as the projection's output is
    zt_ref = O.project_teacher_logits(z_tv, tmap, v_s, temperature=T)
    if dtype == "bf16":
        zt_ref = torch.from_numpy(zt_ref).to(torch.bfloat16).double().numpy()
    kw = dict(variant=variant, t_student=T, t_teacher=1.0, beta=0.1, w_student_ce=0.5,
              w_teacher_ce=0.0, w_kl=1.0, ignore_index=-100)
    lab = labels.numpy()
    ref = O.forward(O.as_f64(z_s), zt_ref, lab, **kw)
    valid = ref["valid"]
    kl = fwd["kl"].cpu().double().numpy()
    ce = fwd["ce_s"].cpu().double().numpy()
    if variant == "jeffreys":  # reverse KL is infinite where q = 0 < p: both sides agree
        assert np.all(np.isinf(ref["kl"][valid])) and np.all(kl[valid] > 1e30)
        return
    assert token_rel_err(kl, ref["kl"], valid) <= TOK_TOL[dtype]
    assert token_rel_err(ce, ref["ce_s"], valid) <= TOK_TOL[dtype]
    assert abs(fwd["loss"].item() - ref["loss"]) <= TOK_TOL[dtype] * abs(ref["loss"])
    g_s, _ = O.grad_logits(O.as_f64(z_s), zt_ref, lab, **kw)
    gz = bwd["d_logits_s"].cpu().double().numpy()
    assert rel_l2(gz, g_s) <= GRAD_TOL[dtype]
    assert np.all(gz[~valid] == 0) and np.all(kl[~valid] == 0)


@pytest.mark.parametrize("dout", ["fp32", "bf16"])
def test_projection_skewed_map(dout):
    """Every teacher token maps into the first few student ids: one CTA's
    receive buffer of the exchange path would overflow, so the device takes
    the slice path instead; the result must not change."""
    v_t, v_s, n = 100000, 70001, 3
    rng = np.random.default_rng(21)
    tmap = rng.integers(0, 4000, size=v_t).astype(np.int32)
    tmap[rng.random(v_t) < 0.1] = -1
    g = torch.Generator().manual_seed(5)
    z = (torch.randn(n, v_t, generator=g) * 3.0).to(torch.bfloat16)
    out = kd.project_teacher_logits(torch.from_numpy(tmap), z.cuda(), v_s, temperature=0.7,
                                    out_dtype=DT[dout])
    torch.cuda.synchronize()
    got = out.cpu().double().numpy()
    ref = O.project_teacher_logits(z, tmap, v_s, temperature=0.7)
    empty = np.isneginf(ref)
    assert np.all(got[empty] <= -1e38)
    tol = 1e-6 if dout == "fp32" else 2.0 ** -8
    err = np.abs(got[~empty] - ref[~empty]) / np.maximum(1.0, np.abs(ref[~empty]))
    assert err.max() <= tol, err.max()


def test_projection_edge_cases():
    """No tokens (the map is still checked), one student id, and a map with
    no matched teacher token at all (every output at the lowest value)."""
    tmap = _map(300, 200, 3)
    out = kd.project_teacher_logits(torch.from_numpy(tmap), torch.randn(0, 300, device="cuda"), 200)
    assert out.shape == (0, 200)
    z = torch.randn(4, 300, device="cuda")
    one = kd.project_teacher_logits(torch.zeros(300, dtype=torch.int32), z, 1, temperature=1.0)
    ref = O.project_teacher_logits(z.cpu(), np.zeros(300, dtype=np.int64), 1)
    torch.cuda.synchronize()
    assert np.allclose(one.cpu().double().numpy(), ref, rtol=0, atol=2e-4)  # 300 folds in fp32
    none = kd.project_teacher_logits(torch.full((300,), -1, dtype=torch.int32), z, 50)
    torch.cuda.synchronize()
    assert torch.all(none <= -1e38)
