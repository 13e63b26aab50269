"""Derivation of the bf16 logit tolerance of the GPU parity tests (CPU only).

The tolerance is derived from the oracle alone (tests/parity.py): the oracle
runs exactly and under a CPU model of the GPU's arithmetic (fp32
accumulation, bf16 attention probabilities); delta = 2 x the largest logit
difference (the floor), the mean bound 2 x the mean difference.  The GPU
tests compute the floor over the very iterations they compare.  Here the
model and the factor are pinned: the floor is real, the model's parts do
what they say, delta is bounded on both sides by the floor, and delta stays
far below what a real mistake moves.
"""
import numpy as np
import pytest

from block_denoising_gb300 import inputs
from oracle import dinfer_oracle as O
from tests import parity as PT

SMALL_BF16 = inputs.shrink(inputs.LLADA_8B, n_layers=2, d_model=512, n_heads=4, ffn=1024, vocab=2048,
                           mask_id=2047)


def _state(cfg, P, G):
    x = np.full((1, P + G), cfg.mask_id)
    x[0, :P] = inputs.make_prompt(cfg, 1, P).numpy()
    mask = np.zeros((1, P + G), bool)
    mask[0, P:] = True
    return x, mask


def _refresh(m, x, mask, P, B):
    return O.refresh_step(m, x.copy(), mask.copy(), P, B, 0.9, O.Cache(m.desc, x.shape[0], x.shape[1]),
                          commit=False).logits


@pytest.fixture(scope="module")
def small():
    cfg = SMALL_BF16
    m = O.Model(O.Desc.from_config(cfg), [w.float().numpy() for w in inputs.make_weights(cfg, 0)])
    x, mask = _state(cfg, 64, 64)
    exact = _refresh(m, x, mask, 64, 32)
    with PT.gpu_arithmetic():
        model = _refresh(m, x, mask, 64, 32)
    return m, x, mask, exact, model


def test_floor_is_real_and_small(small):
    m, x, mask, exact, model = small
    fmax, fmean = PT.floor_stats(exact, model)
    print(f"bf16 floor (d_model 512, GPU arithmetic model): max {fmax:.4f} mean {fmean:.4f}")
    spread = np.std(exact[np.isfinite(exact)])
    assert fmax > 1e-3                  # the two arithmetics do differ
    assert fmax < 0.05 * spread         # ... by rounding only, not by a different computation


def test_delta_is_bounded_by_the_floor_on_both_sides(small):
    _, _, _, exact, model = small
    tol = PT.tolerance_from_floor(*PT.floor_stats(exact, model))
    assert 1.5 * tol["floor_max"] <= tol["delta"] <= 3.0 * tol["floor_max"]
    assert 1.5 * tol["floor_mean"] <= tol["logit_mean"] <= 3.0 * tol["floor_mean"]


def test_gpu_arithmetic_model_parts():
    rng = np.random.default_rng(0)
    q, k, v = rng.normal(size=(5, 2, 8)), rng.normal(size=(40, 2, 8)), rng.normal(size=(40, 2, 8))
    exact = O.attention(q, k, v)
    got = PT._attention_gpu_model(q, k, v)
    # bf16 probabilities: relative error of each weight <= 2^-8, so the output
    # moves by at most 2^-7 of max |v| (numerator and normaliser)
    assert np.max(np.abs(got - exact)) <= 2.0 ** -7 * np.abs(v).max() + 1e-6
    assert np.max(np.abs(got - exact)) > 0       # it does round
    a, w = rng.normal(size=(4, 64)), rng.normal(size=(16, 64))
    np.testing.assert_allclose(PT._linear_fp32(a, w), a @ w.T, rtol=0, atol=64 * 2.0 ** -22 * np.abs(a).max() * np.abs(w).max())
    with PT.gpu_arithmetic():
        assert O.linear is PT._linear_fp32 and O.attention is PT._attention_gpu_model
    assert O.linear is not PT._linear_fp32      # restored


def test_delta_separates_real_mistakes(small):
    # a slip anywhere in a forward moves logits far beyond delta
    m, x, mask, exact, model = small
    tol = PT.tolerance_from_floor(*PT.floor_stats(exact, model))
    fin = np.isfinite(exact)
    orig = O.dense_ffn

    def swapped(a, lw, prec):
        return orig(a, {"w_gate": lw["w_up"], "w_up": lw["w_gate"], "w_down": lw["w_down"]}, prec)

    O.dense_ffn = swapped
    try:
        bad = _refresh(m, x, mask, 64, 32)
    finally:
        O.dense_ffn = orig
    assert np.max(np.abs(bad[fin] - exact[fin])) > 10 * tol["delta"]
    # the attention scale 1/sqrt(head_dim) dropped
    orig_attn = O.attention
    O.attention = lambda q, k, v: orig_attn(np.asarray(q) * np.sqrt(q.shape[-1]), k, v)
    try:
        bad = _refresh(m, x, mask, 64, 32)
    finally:
        O.attention = orig_attn
    assert np.max(np.abs(bad[fin] - exact[fin])) > 3 * tol["delta"]


def test_fp32_models_have_no_rounding_floor():
    cfg = inputs.TINY
    m = O.Model(O.Desc.from_config(cfg), [w.numpy() for w in inputs.make_weights(cfg, 0)])
    x, mask = _state(cfg, 32, 64)
    exact = _refresh(m, x, mask, 32, 16)
    f32 = lambda a, w: (np.asarray(a, np.float32) @ np.asarray(w, np.float32).T).astype(np.float64)
    orig = O.linear
    O.linear = f32
    try:
        approx = _refresh(m, x, mask, 32, 16)
    finally:
        O.linear = orig
    fin = np.isfinite(exact)
    assert np.max(np.abs(exact[fin] - approx[fin])) < 1e-4   # the stated fp32 tolerance holds


def test_flags_cover_a_fallback_that_may_happen():
    """The threshold rule's fallback (no masked confidence above tau: commit
    the single most confident position) can happen as soon as no masked
    confidence is certainly above tau; then every masked position that could
    be the most confident is a decision that rounding may flip."""
    tau, delta = 0.9, 0.57
    conf = np.array([[0.7415, 0.7451, 0.05]])
    lo, hi = PT.conf_interval(conf[0], delta)
    assert hi[1] > tau > hi[0] and lo[1] < tau       # position 1 may reach tau, position 0 may not
    logits = np.zeros((1, 3, 4))
    logits[0, :, 0] = 10.0                             # wide top-2 gaps: no token flag
    masked = np.array([[True, True, True]])
    fl = PT.flags_for(logits, conf, masked, tau, delta)
    assert fl[0, 0] and fl[0, 1]                       # the fallback choice between 0 and 1
    assert not fl[0, 2]                                # 0.05 can never be the most confident
    # a position certainly above tau: the commit is by threshold, no fallback
    conf2 = np.array([[0.7415, 0.7451, 0.999]])
    fl2 = PT.flags_for(logits, conf2, masked, tau, delta)
    assert not fl2[0, 0] and fl2[0, 1] and not fl2[0, 2]
