"""Multi-teacher mixing on the GPU against the oracle (orda-kernel README,
"Cross-vocabulary distillation", multi-teacher mixing): the mixture's
log-probabilities element by element for both modes, and distillation from a
mixture of teachers end to end."""
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


def _teachers(k, v, n, dtype, seed, holes=True):
    """k seeded teacher logit tensors; with `holes`, some entries carry no
    probability (-inf, or the most negative finite value as projection writes
    unmatched ids), in some rows for one teacher only, in others for all."""
    g = torch.Generator().manual_seed(seed)
    zs = [(torch.randn(n, v, generator=g) * (2.0 + i)).to(DT[dtype]) for i in range(k)]
    if holes:
        lo = torch.finfo(DT[dtype]).min
        zs[0][0, : v // 7] = float("-inf")
        zs[-1][0, v // 9: v // 5] = lo
        for z in zs:
            z[n // 2, -3:] = lo
    return zs


def _check(got, ref, dout):
    # no probability: -inf, or a log-probability at or below -1e30 (an input at
    # the most negative finite value, which the kernels read as probability 0)
    empty = ref <= -1e30
    assert np.all(got[empty] <= -1e38), "no-probability tokens must stay at the lowest value"
    tol = 2e-5 if dout == "fp32" else 2.0 ** -8
    err = np.abs(got[~empty] - ref[~empty]) / np.maximum(1.0, np.abs(ref[~empty]))
    assert err.max() <= tol, err.max()


@pytest.mark.parametrize("mode", ["arithmetic", "geometric"])
@pytest.mark.parametrize("din,dout", [("fp32", "fp32"), ("bf16", "fp32"), ("bf16", "bf16")])
@pytest.mark.parametrize("k,v,n", [(1, 1000, 37), (2, 513, 37), (3, 30000, 9), (2, 151936, 4),
                                   (3, 151936, 5), (4, 151936, 3), (8, 70001, 3),
                                   (8, 151936, 2), (2, 20000, 300)])
def test_mix_matches_oracle(mode, din, dout, k, v, n):
    """One CTA per row (1000 / 513 ids, the latter unaligned; double-buffered),
    clusters of 2 to 8 CTAs at two CTAs per SM (30000 to 151936 ids, 2 to 8
    teachers), the wide one-CTA-per-SM shape for rows that need more than
    8 x 100 KiB (three or four teachers of 151936 ids in bf16; in fp32 these
    take the row kernel), rows too long for an 8-CTA wide cluster on the row
    kernel (8 teachers of 151936 ids), and 300 rows per launch, double- and
    single-buffered."""
    zs = _teachers(k, v, n, din, seed=k * 1000 + v)
    rng = np.random.default_rng(v)
    w = rng.uniform(0.2, 2.0, size=k)
    out = kd.mix_teacher_logits([z.cuda() for z in zs], w, mode, out_dtype=DT[dout])
    torch.cuda.synchronize()
    ref = O.mix_teacher_logits(zs, w, mode)
    _check(out.cpu().double().numpy(), ref, dout)


@pytest.mark.parametrize("mode", ["arithmetic", "geometric"])
def test_mix_zero_weight_teacher_and_uniform_default(mode):
    """A teacher with weight 0 takes no part (its logits may be anything); no
    weights means uniform ones."""
    zs = _teachers(3, 4099, 11, "fp32", seed=3, holes=False)
    zs[1] = zs[1] * 1e4
    dev = [z.cuda() for z in zs]
    got = kd.mix_teacher_logits(dev, [1.0, 0.0, 3.0], mode).cpu().double().numpy()
    _check(got, O.mix_teacher_logits([zs[0], zs[2]], [1.0, 3.0], mode), "fp32")
    got = kd.mix_teacher_logits(dev[:2], None, mode).cpu().double().numpy()
    _check(got, O.mix_teacher_logits(zs[:2], [1.0, 1.0], mode), "fp32")


def test_mix_single_teacher_is_log_softmax():
    z = _teachers(1, 50000, 5, "fp32", seed=8, holes=False)[0]
    got = kd.mix_teacher_logits([z.cuda()], [0.3], "arithmetic").cpu().double().numpy()
    _check(got, O.log_softmax(O.as_f64(z)), "fp32")


@pytest.mark.parametrize("mode", ["arithmetic", "geometric"])
@pytest.mark.parametrize("dout", ["fp32", "bf16"])
def test_mix_rows_whose_maximum_keeps_rising(mode, dout):
    """Rows built so that the running maximum of a stream moves many times: a
    rising ramp (every step of every thread passes the previous offset), a
    falling one, and a flat row with one spike at the last id of a CTA's slice
    and one at the very end.  The packed bf16 passes keep each sum around an
    offset that moves only when a step's maximum passes it by 2^8 in base 2; every
    move rescales the sum."""
    v, n = 151936, 4
    ramp = torch.linspace(-30.0, 60.0, v)
    a = torch.stack([ramp, ramp.flip(0), torch.zeros(v), torch.sin(ramp) * 3]).to(torch.bfloat16)
    a[2, v // 8 - 1] = 25.0
    a[2, -1] = 30.0
    b = torch.stack([ramp.flip(0), ramp, torch.full((v,), -2.0), ramp * 0.5]).to(torch.bfloat16)
    w = [0.7, 0.3]
    out = kd.mix_teacher_logits([a.cuda(), b.cuda()], w, mode, out_dtype=DT[dout])
    torch.cuda.synchronize()
    _check(out.cpu().double().numpy(), O.mix_teacher_logits([a, b], w, mode), dout)


@pytest.mark.parametrize("mode", ["arithmetic", "geometric"])
def test_distillation_from_a_mixture(mode):
    """Mix three teachers (bf16), then distil student logits from the mixture
    (forward KL, T_s = 2, mixture at T_t = 1) against the oracle's own mixture
    stored in bf16 as the kernel stores it."""
    n, v, T = 67, 3000, 2.0
    zs = _teachers(3, v, n, "bf16", seed=44, holes=False)
    w = [0.5, 0.3, 0.2]
    g = torch.Generator().manual_seed(45)
    z_s = (torch.randn(n, v, generator=g) * 4.0).to(torch.bfloat16)
    labels = torch.randint(0, v, (n,), generator=g)
    labels[torch.rand(n, generator=g) < 0.08] = -100
    dev = torch.device("cuda:0")
    mix = kd.mix_teacher_logits([z.to(dev) for z in zs], w, mode)
    t = {"logits_s": z_s.to(dev), "logits_t": mix, "labels": labels.to(dev)}
    prob = kd.Problem(n_tokens=n, vocab=v, d_student=0, d_teacher=0, topk=0, dtype="bf16",
                      student="logits", teacher="logits", variant="forward", t_student=T,
                      t_teacher=1.0, w_student_ce=0.5, w_teacher_ce=0.0, w_kl=1.0, beta=0.5,
                      ignore_index=-100)
    fwd = kd.forward(prob, t)
    bwd = kd.backward(prob, t, fwd["stats"], want=("logits_s",))
    torch.cuda.synchronize()
    zt_ref = O.mix_teacher_logits(zs, w, mode)
    zt_ref = torch.from_numpy(zt_ref).to(torch.bfloat16).double().numpy()
    kw = dict(variant="forward", t_student=T, t_teacher=1.0, beta=0.5, w_student_ce=0.5,
              w_teacher_ce=0.0, w_kl=1.0, ignore_index=-100)
    lab = labels.numpy()
    ref = O.forward(O.as_f64(z_s), zt_ref, lab, **kw)
    valid = ref["valid"]
    kl = fwd["kl"].cpu().double().numpy()
    assert token_rel_err(kl, ref["kl"], valid) <= TOK_TOL["bf16"]
    assert abs(fwd["loss"].item() - ref["loss"]) <= TOK_TOL["bf16"] * abs(ref["loss"])
    g_s, _ = O.grad_logits(O.as_f64(z_s), zt_ref, lab, **kw)
    assert rel_l2(bwd["d_logits_s"].cpu().double().numpy(), g_s) <= GRAD_TOL["bf16"]


@pytest.mark.parametrize("mode", ["arithmetic", "geometric"])
def test_mix_edge_cases(mode):
    """No tokens (nothing written, no error), a one-id vocabulary (the mixture
    is log 1 = 0), and eight teachers with uniform weights."""
    z = torch.randn(0, 1000, device="cuda")
    assert kd.mix_teacher_logits([z, z], None, mode).shape == (0, 1000)
    one = kd.mix_teacher_logits([torch.randn(3, 1, device="cuda") * 5 for _ in range(2)], None,
                                mode)
    torch.cuda.synchronize()
    assert torch.all(one.abs() <= 1e-6)
    zs = _teachers(8, 5003, 4, "bf16", seed=12, holes=False)
    got = kd.mix_teacher_logits([t.cuda() for t in zs], None, mode, out_dtype=torch.float32)
    torch.cuda.synchronize()
    _check(got.cpu().double().numpy(), O.mix_teacher_logits(zs, None, mode), "fp32")
