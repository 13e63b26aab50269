"""Derivation of the bf16 logit tolerance used by the GPU parity tests (CPU only).

The bf16 precision contract rounds GEMM inputs, queries and cached K/V to
bf16.  Two correct implementations of that contract that accumulate in
different precisions (the oracle in float64, a GPU in float32) still differ:
a rounding boundary that falls between the two accumulated values flips one
bf16 input by one ulp, and such flips cascade through RMSNorm and attention.
This floor is measured here by running the oracle twice on the same
iteration -- once exact, once with every matmul accumulated in float32 -- and
the GPU tests' delta must be at least about twice the floor.
"""
import numpy as np

from block_denoising_gb300 import inputs
from oracle import dinfer_oracle as O

SMALL_BF16 = inputs.shrink(inputs.LLADA_8B, n_layers=2, d_model=512, n_heads=4, ffn=1024, vocab=2048,
                           mask_id=2047)
DELTA_SMALL, MEAN_SMALL = 0.6, 0.08   # must equal BF16_SMALL in test_gpu_model.py
# twice the d_model, 16 times the sequence: a refresh of 2048 rows
LONG_BF16 = inputs.shrink(inputs.LLADA_8B, n_layers=2, d_model=1024, n_heads=8, ffn=2048, vocab=2048,
                          mask_id=2047)
DELTA_LONG, MEAN_LONG = 0.8, 0.14     # must equal BF16_LONG in test_gpu_model.py


def _refresh_logits(m, x, mask, P, B, lin):
    orig = O.linear
    O.linear = lin
    try:
        r = O.refresh_step(m, x.copy(), mask.copy(), P, B, 0.9, O.Cache(m.desc, x.shape[0], x.shape[1]),
                           commit=False)
    finally:
        O.linear = orig
    return r.logits


def _floor(cfg, P, G, B):
    m = O.Model(O.Desc.from_config(cfg), [w.float().numpy() for w in inputs.make_weights(cfg, 0)])
    x = np.full((1, P + G), cfg.mask_id)
    x[0, :P] = inputs.make_prompt(cfg, 1, P).numpy()
    mask = np.zeros((1, P + G), bool)
    mask[0, P:] = True
    exact = _refresh_logits(m, x, mask, P, B, O.linear)
    f32 = lambda a, w: (np.asarray(a, np.float32) @ np.asarray(w, np.float32).T).astype(np.float64)
    approx = _refresh_logits(m, x, mask, P, B, f32)
    fin = np.isfinite(exact)
    return np.abs(exact[fin] - approx[fin])


def test_bf16_noise_floor_long_refresh():
    # measured 0.39 max / 0.069 mean: the floor grows with d_model and with
    # the number of keys each attention row sums
    d = _floor(LONG_BF16, 1984, 64, 32)
    print(f"bf16 floor (d_model {LONG_BF16.d_model}, L 2048): max {d.max():.4f} mean {d.mean():.4f}")
    assert d.max() > 1e-3
    assert 2 * d.max() <= DELTA_LONG * 1.25
    assert 2 * d.mean() <= MEAN_LONG * 1.25


def test_bf16_noise_floor_small_model():
    cfg = SMALL_BF16
    m = O.Model(O.Desc.from_config(cfg), [w.float().numpy() for w in inputs.make_weights(cfg, 0)])
    P, G, B = 64, 64, 32
    x = np.full((1, P + G), cfg.mask_id)
    x[0, :P] = inputs.make_prompt(cfg, 1, P).numpy()
    mask = np.zeros((1, P + G), bool)
    mask[0, P:] = True
    exact = _refresh_logits(m, x, mask, P, B, O.linear)
    f32 = lambda a, w: (np.asarray(a, np.float32) @ np.asarray(w, np.float32).T).astype(np.float64)
    approx = _refresh_logits(m, x, mask, P, B, f32)
    fin = np.isfinite(exact)
    d = np.abs(exact[fin] - approx[fin])
    print(f"bf16 floor (d_model {cfg.d_model}): max {d.max():.4f} mean {d.mean():.4f}")
    # the floor is real (not zero) and the tests' tolerance is about twice it
    assert d.max() > 1e-3
    assert 2 * d.max() <= DELTA_SMALL * 1.25
    assert 2 * d.mean() <= MEAN_SMALL * 1.25


def test_fp32_models_have_no_rounding_floor():
    cfg = inputs.TINY
    m = O.Model(O.Desc.from_config(cfg), [w.numpy() for w in inputs.make_weights(cfg, 0)])
    P, G, B = 32, 64, 16
    x = np.full((1, P + G), cfg.mask_id)
    x[0, :P] = inputs.make_prompt(cfg, 1, P).numpy()
    mask = np.zeros((1, P + G), bool)
    mask[0, P:] = True
    exact = _refresh_logits(m, x, mask, P, B, O.linear)
    f32 = lambda a, w: (np.asarray(a, np.float32) @ np.asarray(w, np.float32).T).astype(np.float64)
    approx = _refresh_logits(m, x, mask, P, B, f32)
    fin = np.isfinite(exact)
    assert np.max(np.abs(exact[fin] - approx[fin])) < 1e-4   # the stated fp32 tolerance holds
