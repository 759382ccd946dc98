"""Both tile widths of the gradient producer against the oracle.  Two GEMM
sides on CTA pairs take 256 columns per side in one TMEM stage by default;
KD_TC_GRAD_COLS=128 selects 128 columns per side in two stages (the epilogue
of one tile overlapping the MMAs of the next).  Ragged in rows, columns and
both hidden sizes, with several row and vocabulary chunks."""
import pytest

from lm_head_cross_vocab_gb300 import inputs as I
from tests.parity_util import assert_parity, run_and_compare

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["256", "128"], ids=["cols256", "cols128"])
def grad_cols(request, monkeypatch):
    monkeypatch.setenv("KD_TC_GRAD_COLS", request.param)
    return request.param


@pytest.mark.parametrize("variant", ["forward", "jeffreys", "skew_js"])
def test_separate_teacher_grad_tiles(grad_cols, variant):
    w = I.WORKLOADS[2].scaled(n_tokens=600, d_student=136, d_teacher=200, vocab=1500,
                              variant=variant)
    assert_parity(run_and_compare(w, vocab_chunk=640, seq_chunk=256), "bf16")


def test_separate_teacher_grad_tiles_t1_with_ce(grad_cols):
    w = I.WORKLOADS[2].scaled(n_tokens=333, d_student=64, d_teacher=96, vocab=2100,
                              variant="reverse", t_student=1.0, t_teacher=1.0,
                              w_student_ce=0.6)
    assert_parity(run_and_compare(w), "bf16")
