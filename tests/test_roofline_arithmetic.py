"""The benchmark's roofline denominators (no GPU): algorithmic bytes and
FLOPs per cached iteration and per refresh for each workload, against the
figures worked out by hand from the workload shapes.

Weights (parameters): dense layers 4 d^2 (Q, K, V, O) + 3 d f (gate, up,
down); MoE layers 4 d^2 + E d (router) + 3 fe d per expert; plus the LM
head V d.  K/V: 2 (K and V) x (L - B) non-block positions x d x layers x
batch.  FLOPs: 2 per multiply-add of every GEMM row (the MoE rows through k
experts) plus 4 L d per query row and layer for attention; the LM head on
the block rows.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from block_denoising_gb300 import inputs  # noqa: E402

# workload -> (bytes per iteration, FLOPs per iteration, FLOPs per refresh)
HAND = {
    # 32 x (67.1 M + 151.0 M) + 518.0 M = 7.499 G params = 15.00 GB; K/V 1472 x 8192 x 32 x 2 B = 0.77 GB
    "llada8b_b1": (15.77e9, 1.011e12, 22.74e12),
    # 16 x (16.8 M + 0.13 M + 64 x 6.29 M) + 321.9 M = 7.035 G params = 14.07 GB; K/V 0.16 GB
    "lladamoe_b1": (14.23e9, 0.190e12, 3.01e12),
    # 15.00 GB of weights + 16 x 1248 x 8192 x 32 x 2 B = 10.47 GB of K/V
    "llada8b_b16": (25.46e9, 8.021e12, 300.1e12),
    # 14.07 GB + 8640 x 4096 x 16 x 2 B = 1.13 GB
    "lladamoe_long": (15.20e9, 0.252e12, 28.70e12),
    # fp32: 2.63 M params x 4 B = 10.5 MB; K/V 80 x 512 x 2 x 4 B = 0.33 MB
    "tiny_fp32": (10.85e6, 87.3e6, 356.0e6),
}


@pytest.mark.parametrize("name", sorted(HAND))
def test_roofline_work_per_workload(name):
    cfg, run, _ = inputs.WORKLOADS[name]
    b, L, B = run.batch, run.seq_len, run.block_length
    by, fi, fr = HAND[name]
    assert bench.iteration_bytes(cfg, b, L, B) == pytest.approx(by, rel=3e-3)
    assert bench.iteration_flops(cfg, b, L, B) == pytest.approx(fi, rel=3e-3)
    assert bench.refresh_flops(cfg, b, L, B) == pytest.approx(fr, rel=3e-3)


def test_moe_bytes_count_only_the_selected_experts():
    cfg, run, _ = inputs.WORKLOADS["lladamoe_b1"]
    b, L, B = run.batch, run.seq_len, run.block_length
    full = bench.iteration_bytes(cfg, b, L, B)
    # 8 of 64 experts per layer: 56 experts x 3 x 1024 x 2048 x 16 layers x 2 B fewer
    eight = bench.iteration_bytes(cfg, b, L, B, experts=8)
    assert full - eight == 56 * 3 * 1024 * 2048 * 16 * 2
