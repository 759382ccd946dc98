"""GPU parity: the CUDA path through the C ABI vs the fp64 CPU oracle, element
by element on the same seeded inputs, at sizes that span several tiles and a
ragged tail, plus edge cases (ignored tokens, empty batches, bad labels,
chunking invariance)."""
import numpy as np
import pytest
import torch

from lm_head_cross_vocab_gb300 import inputs as I
from lm_head_cross_vocab_gb300 import kd
from tests.parity_util import assert_parity, rel_l2, run_and_compare

pytestmark = pytest.mark.gpu

W = I.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kd.load_library()
    assert kd.kd_device_supported(0), "tests need an sm_103 GPU"


# ----------------------------------------------------------- streaming path

@pytest.mark.parametrize("variant", ["forward", "reverse", "jeffreys", "skew_js", "skew_forward", "skew_reverse"])
@pytest.mark.parametrize("vocab", [4104, 4099])  # vectorised rows, ragged scalar rows
def test_logit_pair_streaming(variant, vocab):
    w = W[5].scaled(n_tokens=67, vocab=vocab, variant=variant)
    assert_parity(run_and_compare(w), "bf16")


@pytest.mark.parametrize("variant", ["jeffreys", "skew_js", "skew_reverse"])
def test_logit_pair_streaming_more_rows_than_ctas(variant):
    """More rows than persistent CTAs: each CTA streams several rows (two sweeps
    each for skew-JS) through one ring, so stage phases carry across rows."""
    w = W[5].scaled(n_tokens=341, vocab=8200, variant=variant, w_student_ce=0.3)
    assert_parity(run_and_compare(w), "bf16")


@pytest.mark.parametrize("variant", ["forward", "reverse"])
def test_logit_pair_streaming_rows_longer_than_the_ring(variant):
    """Rows longer than the ring (53256 ids: 4.3 pieces of 12288 ids over the
    one-sweep kernels' 4 stages): stages are refilled within a row, so
    consumers often wait on a stage whose copy is still in flight."""
    w = W[5].scaled(n_tokens=180, vocab=53256, variant=variant)
    assert_parity(run_and_compare(w), "bf16")


@pytest.mark.parametrize("variant", ["forward", "jeffreys", "skew_js"])
@pytest.mark.parametrize("t", [1.0, 2.0])
def test_logit_pair_streaming_rows_whose_maximum_keeps_rising(variant, t):
    """Rows built so that the running maxima move many times: rising and
    falling ramps, a flat row with two late spikes, a wave; the teacher is the
    student plus a small wave.  The packed kernels keep their sums around
    offsets that move only when a step's maximum passes them by 2^8 in base 2
    (tested on the raw bf16 words); every move rescales the sums."""
    v = 40968

    def mutate(cpu):
        n = cpu["logits_s"].shape[0]
        ramp = torch.linspace(-20.0, 40.0, v)
        rows = [ramp, ramp.flip(0), torch.zeros(v), torch.sin(ramp) * 4.0]
        for i in range(n):
            base = rows[i % 4].clone()
            if i % 4 == 2:
                base[v // 3] = 15.0
                base[-1] = 22.0
            wave = 0.5 * torch.sin(torch.arange(v, dtype=torch.float32) * 0.37 + i)
            cpu["logits_s"][i] = base.to(cpu["logits_s"].dtype)
            cpu["logits_t"][i] = (base + wave).to(cpu["logits_t"].dtype)

    w = W[5].scaled(n_tokens=24, vocab=v, variant=variant, t_student=t, t_teacher=t)
    res = run_and_compare(w, mutate=mutate)
    # The flat rows with spikes at T = 1 put nearly all of both distributions on
    # one id: their divergences are 1e-7 to 1e-5, formed in fp32 as the
    # difference of two terms of the size of the logit gap there (~0.3), so the
    # approximate exponentials' ~2-ulp error on the dominant terms leaves a few
    # 1e-7 absolute: 1e-6 absolute on top of the per-token relative bound.
    ref, valid = res["ref"]["kl"], res["valid"]
    got = res.pop("gpu_fwd")["kl"].cpu().double().numpy()
    res.pop("err_kl")
    floor = 1e-3 * np.mean(np.abs(ref[valid]))
    err = np.abs(got - ref)[valid]
    assert np.all(err <= 1e-6 + 2e-3 * np.maximum(np.abs(ref[valid]), floor)), err.max()
    assert_parity(res, "bf16")


@pytest.mark.parametrize("variant", ["forward", "jeffreys", "skew_js", "skew_forward"])
@pytest.mark.parametrize("vocab", [8, 6144, 6152, 12288, 12296, 24576, 24584, 110600])
def test_logit_pair_streaming_piece_boundaries(variant, vocab):
    """Rows at and just past the ring's piece boundaries.  The one-sweep
    forwards and their backwards stream 12288 bf16 ids a stage (two 16-byte
    slots per consumer thread), the skew variants' two-sweep forward and
    backward 6144 (one slot, 8 stages): rows of one 8-id group, of exactly
    one, two and four pieces, one group past each, and of ~9 and ~18 pieces
    (every stage refilled within a row)."""
    w = W[5].scaled(n_tokens=37, vocab=vocab, variant=variant)
    assert_parity(run_and_compare(w), "bf16")


@pytest.mark.parametrize("variant", ["forward", "reverse", "jeffreys", "skew_js", "skew_forward", "skew_reverse"])
def test_logit_pair_streaming_t1_with_student_ce(variant):
    """T = 1 with a student CE term: the packed kernels' T = 1 shortcut and
    their label-column correction."""
    w = W[5].scaled(n_tokens=70, vocab=4104, variant=variant, t_student=1.0, t_teacher=1.0,
                    w_student_ce=0.6)
    assert_parity(run_and_compare(w), "bf16")


@pytest.mark.parametrize("variant", ["forward", "jeffreys"])
def test_logit_pair_streaming_without_labels(variant):
    """No labels at all: no CE sums are kept."""
    w = W[5].scaled(n_tokens=48, vocab=6000, variant=variant, ignore_frac=0.0)
    assert "labels" not in I.make_inputs(w.scaled(n_tokens=1, vocab=8), "cpu")
    assert_parity(run_and_compare(w), "bf16")


def test_logit_pair_streaming_general_temperature_bf16():
    """T = 1.5 (no exact shortcut): the generic ring kernels in bf16."""
    w = W[5].scaled(n_tokens=60, vocab=5000, variant="jeffreys", t_student=1.5, t_teacher=1.5,
                    w_student_ce=0.4)
    assert_parity(run_and_compare(w), "bf16")


def test_logit_student_plain_ce_streaming():
    """Student logits, no teacher: CE only."""
    w = W[5].scaled(n_tokens=50, vocab=3000, teacher="none", w_student_ce=1.0, w_kl=0.0)
    assert_parity(run_and_compare(w), "bf16")


def test_logit_pair_streaming_fp32_with_ce():
    w = W[5].scaled(n_tokens=40, vocab=3000, dtype="fp32", w_student_ce=0.7, variant="jeffreys",
                    t_teacher=1.5)
    assert_parity(run_and_compare(w), "fp32")


def test_topk_with_logit_student_streaming():
    w = W[4].scaled(n_tokens=50, vocab=2048, student="logits", d_student=0, topk=16,
                    student_logit_std=2.0)
    assert_parity(run_and_compare(w), "bf16")


def test_topk_with_logit_student_t2_and_ce_streaming():
    w = W[4].scaled(n_tokens=45, vocab=3072, student="logits", d_student=0, topk=24,
                    student_logit_std=2.0, t_student=2.0, t_teacher=2.0, w_student_ce=0.5,
                    ignore_frac=0.1)
    assert_parity(run_and_compare(w), "bf16")


# ----------------------------------------------------------- fp32 CUDA cores

@pytest.mark.parametrize("variant", ["forward", "reverse", "jeffreys", "skew_js", "skew_forward", "skew_reverse"])
def test_tiny_tied_fp32(variant):
    """The tiny tied fp32 workload (64 tokens, D=64, V=512, T=2), all variants."""
    assert_parity(run_and_compare(W[1].scaled(variant=variant)), "fp32")


def test_fp32_separate_ragged_multichunk():
    w = W[2].scaled(n_tokens=77, d_student=40, d_teacher=24, vocab=333, dtype="fp32")
    assert_parity(run_and_compare(w, vocab_chunk=64, seq_chunk=32), "fp32")


def test_fp32_topk():
    w = W[4].scaled(n_tokens=45, d_student=32, vocab=700, topk=12, dtype="fp32")
    assert_parity(run_and_compare(w), "fp32")


# ----------------------------------------------------------- tcgen05 GEMM core

@pytest.mark.parametrize("a_kmajor,b_kmajor", [(True, True), (True, False), (False, True),
                                                (False, False)])
@pytest.mark.parametrize("m,n,k", [(128, 256, 64), (304, 504, 136), (600, 520, 200),
                                   (1000, 776, 1024)])
def test_tensor_core_gemm_matches_torch(m, n, k, a_kmajor, b_kmajor):
    """GEMM core against fp64 torch for every operand layout (K-major [rows, K]
    or MN-major [K, rows]); ragged in M, N and K."""
    g = torch.Generator(device="cpu").manual_seed(m + n + k)
    a = torch.randn(m, k, generator=g).to(torch.bfloat16)
    b = torch.randn(n, k, generator=g).to(torch.bfloat16)
    a_dev = (a if a_kmajor else a.T.contiguous()).cuda()
    b_dev = (b if b_kmajor else b.T.contiguous()).cuda()
    c = kd.kd_diag_gemm_bf16(a_dev, b_dev, a_kmajor, b_kmajor)
    ref = a.double() @ b.double().T
    torch.cuda.synchronize()
    assert rel_l2(c.cpu().numpy(), ref.numpy()) < 1e-5


# ----------------------------------------------------------- tcgen05 fused paths

def test_separate_teacher_bf16_small():
    """Separate-teacher bf16 workload at reduced size, ragged in every dim."""
    w = W[2].scaled(n_tokens=300, d_student=128, d_teacher=256, vocab=1000)
    assert_parity(run_and_compare(w), "bf16")


def test_separate_teacher_bf16_odd_row_tiles():
    """Three 256-row tiles, the last one ragged."""
    w = W[2].scaled(n_tokens=700, d_student=192, d_teacher=128, vocab=2600)
    assert_parity(run_and_compare(w), "bf16")


@pytest.mark.parametrize("variant", ["forward", "reverse", "skew_js", "skew_forward", "skew_reverse"])
def test_separate_teacher_bf16_variants(variant):
    w = W[2].scaled(n_tokens=200, d_student=64, d_teacher=192, vocab=1500, variant=variant,
                    t_teacher=1.5)
    assert_parity(run_and_compare(w), "bf16")


@pytest.mark.parametrize("variant", ["reverse", "jeffreys"])
def test_separate_teacher_bf16_t1(variant):
    """T = 1 on both sides (the T = 1 sums are the tempered ones): the paired
    forward update and the producer's reverse / Jeffreys element loops at
    that temperature, with both CE terms."""
    w = W[2].scaled(n_tokens=280, d_student=96, d_teacher=160, vocab=2200, variant=variant,
                    t_student=1.0, t_teacher=1.0, w_student_ce=0.7)
    assert_parity(run_and_compare(w), "bf16")


def test_tied_bf16_teacher_ce_flows_into_weight():
    w = W[1].scaled(n_tokens=257, d_student=64, d_teacher=64, vocab=777, dtype="bf16")
    assert_parity(run_and_compare(w), "bf16")


def test_topk_bf16():
    w = W[4].scaled(n_tokens=260, d_student=128, vocab=3000, topk=20)
    assert_parity(run_and_compare(w), "bf16")


def test_plain_ce_no_teacher_bf16():
    w = W[2].scaled(n_tokens=150, d_student=96, d_teacher=0, vocab=1200, teacher="none",
                    w_teacher_ce=0.0, w_kl=0.0)
    assert_parity(run_and_compare(w), "bf16")


def test_logit_student_separate_teacher_bf16():
    """Large-vocab scoring shape at reduced size (student logits, teacher GEMM)."""
    w = W[3].scaled(n_tokens=130, d_teacher=128, vocab=5000)
    assert_parity(run_and_compare(w, backward=True), "bf16")


@pytest.mark.parametrize("vchunk,schunk", [(256, 128), (512, 0), (0, 128)])
def test_chunking_invariance_bf16(vchunk, schunk):
    """Results do not depend on the backward chunk (fp32 accumulation across chunks)."""
    w = W[2].scaled(n_tokens=300, d_student=64, d_teacher=128, vocab=1000)
    base = run_and_compare(w)
    res = run_and_compare(w, vocab_chunk=vchunk, seq_chunk=schunk)
    assert_parity(res, "bf16")
    assert abs(res["err_dh"] - base["err_dh"]) < 5e-3
    assert abs(res["err_dw"] - base["err_dw"]) < 5e-3


# ----------------------------------------------------------- edge cases

def test_all_tokens_ignored_gives_zero_loss_and_grads():
    w = W[2].scaled(n_tokens=130, d_student=64, d_teacher=64, vocab=600)

    def mutate(cpu):
        cpu["labels"][:] = w.ignore_index
    res = run_and_compare(w, mutate=mutate)
    assert res["gpu_fwd"]["loss"].item() == 0.0
    assert res["ignored_zero"] and res["ignored_grad_zero"]


def test_bad_label_is_flagged_not_dereferenced():
    w = W[2].scaled(n_tokens=130, d_student=64, d_teacher=64, vocab=600)
    cpu = I.make_inputs(w, "cpu")
    cpu["labels"][5] = 10 ** 9
    cpu["labels"][6] = -7
    t = {k: v.cuda() for k, v in cpu.items()}
    prob = kd.problem_for(w)
    out = kd.forward(prob, t, check=False)
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) & kd.KD_DEV_BAD_LABEL
    ce = out["ce_s"].cpu().numpy()
    assert np.isnan(ce[5]) and np.isnan(ce[6]) and np.isfinite(np.delete(ce, [5, 6])).all()
    with pytest.raises(kd.KDError):
        kd.forward(prob, t)


def test_bad_topk_is_flagged():
    w = W[4].scaled(n_tokens=40, d_student=64, vocab=500, topk=8)
    cpu = I.make_inputs(w, "cpu")
    cpu["topk_idx"][3, 1] = cpu["topk_idx"][3, 0]  # repeated id
    cpu["topk_idx"][4, 2] = 500                     # out of range
    t = {k: v.cuda() for k, v in cpu.items()}
    out = kd.forward(kd.problem_for(w), t, check=False)
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) & kd.KD_DEV_BAD_TOPK


def test_empty_batch():
    w = W[2].scaled(n_tokens=0, d_student=64, d_teacher=64, vocab=600)
    prob = kd.problem_for(w)
    t = {k: v.cuda() for k, v in I.make_inputs(w.scaled(n_tokens=1), "cpu").items()}
    out = kd.forward(prob, t)
    torch.cuda.synchronize()
    assert out["loss"].item() == 0.0


def test_sum_reduction_and_num_batch_labels():
    w = W[2].scaled(n_tokens=128, d_student=64, d_teacher=64, vocab=512)
    assert_parity(run_and_compare(w, reduction="sum"), "bf16")
    assert_parity(run_and_compare(w, num_batch_labels=1000), "bf16")


@pytest.mark.parametrize("variant", ["skew_js", "skew_forward", "skew_reverse"])
def test_skew_near_identical_distributions(variant):
    """Teacher = student with one bf16 ulp of noise on a third of the logits:
    the skew divergences are 5e-7 to 2e-4 per token.  Both the bf16 fast
    logarithms and the fp32 precise path resolve them to about 1e-7 absolute
    (the fp32 summation floor every variant shares; the relative tolerances hold
    above ~1e-4)."""
    from oracle import kd_oracle as O
    n, v = 40, 8200
    g = torch.Generator().manual_seed(77)
    zs = (torch.randn(n, v, generator=g) * 4.0).to(torch.bfloat16)
    bump = (torch.rand(n, v, generator=g) < 1 / 3).to(torch.int16)
    zt = (zs.view(torch.int16) + bump).view(torch.bfloat16)  # next bf16 value
    labels = torch.randint(0, v, (n,), generator=g)
    for dtype, tol_abs, tol_rel in (("bf16", 2e-7, 2e-3), ("fp32", 1e-7, 1e-5)):
        dt = torch.bfloat16 if dtype == "bf16" else torch.float32
        t = {"logits_s": zs.to(dt).cuda(), "logits_t": zt.to(dt).cuda(), "labels": labels.cuda()}
        prob = kd.Problem(n_tokens=n, vocab=v, dtype=dtype, student="logits", teacher="logits",
                          variant=variant, t_student=2.0, t_teacher=2.0, w_student_ce=0.0,
                          w_kl=1.0, beta=0.1)
        fwd = kd.forward(prob, t)
        torch.cuda.synchronize()
        ref = O.forward(O.as_f64(zs), O.as_f64(zt), labels.numpy(), variant=variant,
                        t_student=2.0, t_teacher=2.0, beta=0.1, w_student_ce=0.0, w_kl=1.0)
        got = fwd["kl"].cpu().double().numpy()
        assert np.all(ref["kl"] > 0) and ref["kl"].max() < 3e-4
        err = np.abs(got - ref["kl"])
        assert np.all(err <= tol_abs + tol_rel * np.abs(ref["kl"])), (dtype, err.max())
