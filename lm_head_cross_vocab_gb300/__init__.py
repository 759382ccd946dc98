"""GB300 (sm_103a) fused LM-head + cross-entropy + KL distillation loss.

The compute lives in ``libkdgb.so`` (hand-written CUDA: tcgen05 / TMA / TMEM
fused projection kernels, HBM-streaming logits kernels, fp32 CUDA-core
kernels) behind the C ABI in ``include/kd.h``; ``kd`` is its thin binding and
``inputs`` draws the seeded synthetic workloads.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs", "kd", "build"]
