"""Pins of the CPU oracle to things other than itself (no GPU).

Each test checks the oracle against a closed form, a library routine, an
invariant the method fixes, a special case that reduces to a simpler
decoder, or a pure-Python brute force on tiny inputs.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

from block_denoising_gb300 import inputs
from oracle import dinfer_oracle as O
from tests import bruteforce as BF


def tiny_desc(**kw):
    base = dict(n_layers=2, d_model=8, n_heads=2, head_dim=4, ffn=12, vocab=16,
                mask_id=15, rms_eps=1e-5, rope_theta=10000.0, logit_scale=40.0, dtype="fp32")
    base.update(kw)
    return O.Desc(**base)


def tiny_model(desc, seed=0, std=0.3, gains_random=True):
    cfg = inputs.ModelConfig(n_layers=desc.n_layers, d_model=desc.d_model, n_heads=desc.n_heads,
                             head_dim=desc.head_dim, ffn=desc.ffn, vocab=desc.vocab,
                             mask_id=desc.mask_id, n_experts=desc.n_experts, top_k=desc.top_k,
                             expert_ffn=desc.expert_ffn, dtype="fp32", weight_std=std)
    ws = [w.numpy().astype(np.float64) for w in inputs.make_weights(cfg, seed)]
    if gains_random:  # non-unit gains so that a dropped gain is visible
        for i, (name, shape, init) in enumerate(inputs.weight_specs(cfg)):
            if init == "ones":
                ws[i] = 0.5 + inputs.uniform_tensor(1000 + i, shape, 0.0, 1.0, seed).numpy()
    if desc.dtype == "bf16":
        ws = [O.round_bf16(w) for w in ws]
    return O.Model(desc, ws), ws


# ---------------------------------------------------------------------------
# elementwise pieces
# ---------------------------------------------------------------------------
def test_round_bf16_matches_torch():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(200000, generator=g, dtype=torch.float64) * torch.exp(torch.randn(200000, generator=g, dtype=torch.float64) * 4)
    # exact halfway cases in float32
    base = torch.randn(1000, generator=g).to(torch.bfloat16).float()
    half = base + base.abs() * (2.0 ** -9)
    x = torch.cat([x, half.double()])
    ref = x.to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_bf16(x.numpy()), ref)


def test_rmsnorm_unit_rms_and_gain():
    h = np.random.default_rng(0).normal(size=(5, 64)) * 3.0
    y = O.rmsnorm(h, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, -1)), 1.0, rtol=1e-12)
    g = np.linspace(0.5, 2.0, 64)
    np.testing.assert_allclose(O.rmsnorm(h, g, 0.0), y * g, rtol=1e-12)
    # eps enters under the square root
    z = np.full((1, 4), 1e-3)
    np.testing.assert_allclose(O.rmsnorm(z, np.ones(4), 1e-5), 1e-3 / math.sqrt(1e-6 + 1e-5), rtol=1e-12)


def test_silu_closed_form():
    x = np.linspace(-20, 20, 1001)
    np.testing.assert_allclose(O.silu(x), x * scipy.special.expit(x), rtol=1e-13, atol=1e-300)


def test_rope_relative_position_and_identity():
    rng = np.random.default_rng(1)
    q = rng.normal(size=(1, 3, 8))
    k = rng.normal(size=(1, 3, 8))
    np.testing.assert_allclose(O.rope(q, [0], 10000.0), q, rtol=0, atol=0)
    for (p, r, c) in [(3, 7, 11), (100, 2, 513), (0, 1535, 17)]:
        a = np.sum(O.rope(q, [p], 1e4) * O.rope(k, [r], 1e4), -1)
        b = np.sum(O.rope(q, [p + c], 1e4) * O.rope(k, [r + c], 1e4), -1)
        np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-9)
    # a rotation keeps the norm of each pair
    y = O.rope(q, [37], 1e4)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(q, axis=-1), rtol=1e-12)
    # pair (i, i+hd/2) rotated by p * theta^(-2i/hd): check one pair by hand
    e = np.zeros((1, 1, 8)); e[0, 0, 1] = 1.0
    ang = 5 * 10000.0 ** (-2.0 * 1 / 8)
    y = O.rope(e, [5], 1e4)
    np.testing.assert_allclose([y[0, 0, 1], y[0, 0, 5]], [math.cos(ang), math.sin(ang)], rtol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(2)
    k = rng.normal(size=(9, 2, 4))
    v = rng.normal(size=(9, 2, 4))
    # q = 0 -> uniform weights -> mean of the values
    np.testing.assert_allclose(O.attention(np.zeros((3, 2, 4)), k, v), np.broadcast_to(v.mean(0), (3, 2, 4)), rtol=1e-12)
    # identical keys -> mean of the values whatever q is
    kk = np.broadcast_to(k[:1], k.shape)
    np.testing.assert_allclose(O.attention(rng.normal(size=(3, 2, 4)), kk, v), np.broadcast_to(v.mean(0), (3, 2, 4)), rtol=1e-12)
    # one dominant key -> its value
    q = np.zeros((1, 2, 4)); q[0, :, 0] = 1e3
    k2 = np.zeros((9, 2, 4)); k2[4, :, 0] = 1.0
    np.testing.assert_allclose(O.attention(q, k2, v)[0], v[4], rtol=1e-12)
    # weights equal scipy's softmax of q.k/sqrt(hd)
    q = rng.normal(size=(3, 2, 4))
    w = scipy.special.softmax(np.einsum("qhd,khd->hqk", q, k) / 2.0, axis=-1)
    np.testing.assert_allclose(O.attention(q, k, v), np.einsum("hqk,khd->qhd", w, v), rtol=1e-12)
    # no mask: permuting the keys and values together changes nothing
    perm = rng.permutation(9)
    np.testing.assert_allclose(O.attention(q, k[perm], v[perm]), O.attention(q, k, v), rtol=1e-12)
    # query rows are independent: grouping them (memory bound) changes nothing
    q7 = rng.normal(size=(7, 2, 4))
    np.testing.assert_allclose(O.attention(q7, k, v, rows_per_group=2), O.attention(q7, k, v), rtol=1e-13)
    for i in range(7):
        np.testing.assert_allclose(O.attention(q7[i:i + 1], k, v)[0], O.attention(q7, k, v)[i], rtol=1e-13)


# ---------------------------------------------------------------------------
# decoding
# ---------------------------------------------------------------------------
def test_top1_confidence_closed_form():
    rng = np.random.default_rng(4)
    lg = rng.normal(size=(7, 50)) * 20
    lg[:, 13] = -np.inf  # the mask token
    tok, conf = O.top1_confidence(lg)
    p = scipy.special.softmax(lg, axis=-1)
    np.testing.assert_array_equal(tok, np.argmax(p, -1))
    np.testing.assert_allclose(conf, p.max(-1), rtol=1e-13)
    assert np.all(conf > 1 / 49) and np.all(conf <= 1)
    # all equal (except the masked entry) -> 1/(V-1) and the lowest index
    eq = np.zeros((1, 50)); eq[0, 13] = -np.inf
    t, c = O.top1_confidence(eq)
    assert t[0] == 0 and abs(c[0] - 1 / 49) < 1e-15
    # tie between two maxima -> lowest index
    tie = np.zeros((1, 6)); tie[0, [2, 4]] = 5.0
    assert O.top1_confidence(tie)[0][0] == 2


def test_lm_head_excludes_mask_token():
    desc = tiny_desc(n_layers=1)
    m, ws = tiny_model(desc)
    h = np.zeros((1, 8)); h[0] = 1.0
    m.lm_head = m.lm_head.copy()
    m.lm_head[desc.mask_id] = 100.0  # the mask row would dominate
    lg = O.lm_head_logits(m, h)
    assert lg[0, desc.mask_id] == -np.inf
    assert O.top1_confidence(lg)[0][0] != desc.mask_id


@pytest.mark.parametrize("conf,masked,tau,expect", [
    ([0.95, 0.5, 0.91, 0.2], [1, 1, 1, 1], 0.9, [1, 0, 1, 0]),     # parallel commit
    ([0.95, 0.5, 0.91, 0.2], [0, 1, 1, 1], 0.9, [0, 0, 1, 0]),     # only masked positions
    ([0.3, 0.8, 0.7, 0.8], [1, 1, 1, 1], 0.9, [0, 1, 0, 0]),       # fallback, tie -> lowest position
    ([0.3, 0.8, 0.7, 0.8], [1, 0, 1, 1], 0.9, [0, 0, 0, 1]),       # fallback among masked only
    ([0.9, 0.9, 0.1, 0.1], [1, 1, 1, 1], 0.9, [1, 0, 0, 0]),       # strict '>': equal is not above
    ([0.95, 0.99, 0.1, 0.1], [0, 0, 0, 0], 0.9, [0, 0, 0, 0]),     # nothing masked -> nothing
    ([0.1, 0.2, 0.3, 0.05], [1, 1, 1, 1], 0.0, [1, 1, 1, 1]),      # tau 0 -> whole block
    ([1.0, 1.0, 0.99, 1.0], [1, 1, 1, 1], 1.0, [1, 0, 0, 0]),      # tau 1 -> one per step
])
def test_threshold_commit_cases(conf, masked, tau, expect):
    got = O.threshold_commit(np.array(conf), np.array(masked, bool), tau)
    np.testing.assert_array_equal(got.astype(int), expect)


# ---------------------------------------------------------------------------
# forward vs brute force
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_forward_matches_bruteforce(dtype):
    desc = tiny_desc(dtype=dtype)
    m, ws = tiny_model(desc, std=0.4)
    ids = np.array([3, 7, 15, 15, 1, 15])
    bf = np.array(BF.forward_logits(desc, [w.tolist() for w in ws], list(ids), bf16_mode=(dtype == "bf16")))
    cache = O.Cache(desc, 1, len(ids))
    hid = O.forward(m, ids[None], cache, np.arange(len(ids)))
    lg = O.lm_head_logits(m, hid[0])
    fin = np.isfinite(bf)
    assert np.array_equal(fin, np.isfinite(lg))
    tol = 1e-9 if dtype == "fp32" else 2e-2  # bf16: rare rounding flips from summation order
    np.testing.assert_allclose(lg[fin], bf[fin], rtol=0, atol=tol)
    if dtype == "bf16":
        assert np.mean(np.abs(lg[fin] - bf[fin]) < 1e-9) > 0.9


def test_bidirectional_no_causal_mask():
    desc = tiny_desc()
    m, _ = tiny_model(desc)
    a = np.array([[3, 7, 15, 15, 1, 2]])
    b = a.copy(); b[0, 5] = 9  # change the LAST token
    ha = O.forward(m, a, O.Cache(desc, 1, 6), np.arange(6))
    hb = O.forward(m, b, O.Cache(desc, 1, 6), np.arange(6))
    assert np.max(np.abs(ha[0, 0] - hb[0, 0])) > 1e-6   # the first position sees it


# ---------------------------------------------------------------------------
# MoE special cases
# ---------------------------------------------------------------------------
def test_moe_single_expert_equals_dense():
    rng = np.random.default_rng(5)
    d, fe = 8, 6
    a = rng.normal(size=(5, d))
    w13 = rng.normal(size=(1, 2 * fe, d)) * 0.3
    w2 = rng.normal(size=(1, d, fe)) * 0.3
    desc = tiny_desc(n_experts=1, top_k=1, expert_ffn=fe, ffn=0)
    lw = {"router": rng.normal(size=(1, d)), "w13": w13, "w2": w2}
    got = O.moe_ffn(a, lw, desc, O.Precision("fp32"))
    dense = O.dense_ffn(a, {"w_gate": w13[0, :fe], "w_up": w13[0, fe:], "w_down": w2[0]}, O.Precision("fp32"))
    np.testing.assert_allclose(got, dense, rtol=1e-12)


def test_moe_all_experts_is_softmax_mixture():
    rng = np.random.default_rng(6)
    d, fe, E = 8, 4, 5
    a = rng.normal(size=(3, d))
    lw = {"router": rng.normal(size=(E, d)), "w13": rng.normal(size=(E, 2 * fe, d)) * 0.3,
          "w2": rng.normal(size=(E, d, fe)) * 0.3}
    desc = tiny_desc(n_experts=E, top_k=E, expert_ffn=fe, ffn=0)
    got = O.moe_ffn(a, lw, desc, O.Precision("fp32"))
    p = scipy.special.softmax(a @ lw["router"].T, axis=-1)
    g = np.einsum("rd,efd->ref", a, lw["w13"][:, :fe])
    u = np.einsum("rd,efd->ref", a, lw["w13"][:, fe:])
    y = np.einsum("ref,edf->red", g * scipy.special.expit(g) * u, lw["w2"])
    np.testing.assert_allclose(got, np.einsum("re,red->rd", p, y), rtol=1e-12)


def _moe_hand_case():
    """Two rows, four experts, top-2, expert FFN width 1; router logits are
    logarithms so that the router softmax is an exact fraction:
    row 0: logits ln[4, 2, 2, 1] -> p = [4, 2, 2, 1] / 9, experts {0, 1}
           (experts 1 and 2 tie: the lower index is taken);
    row 1: logits ln[1, 2, 4, 1] -> p = [1, 2, 4, 1] / 8, experts {2, 1}.
    Expert e's gate and up rows read features 0 and 1 with weights g_e and
    u_e, and its down column writes feature e only, so expert e alone fills
    output feature e with silu(g_e) * u_e."""
    d, E, fe = 4, 4, 1
    g = np.array([1.0, -2.0, 0.5, 3.0])
    u = np.array([2.0, -1.0, 4.0, 1.0])
    router = np.zeros((E, d))
    router[:, 0] = np.log([4.0, 2.0, 2.0, 1.0])
    router[:, 1] = np.log([1.0, 2.0, 4.0, 1.0])
    w13 = np.zeros((E, 2 * fe, d))
    w13[:, 0, 0] = w13[:, 0, 1] = g
    w13[:, 1, 0] = w13[:, 1, 1] = u
    w2 = np.zeros((E, d, fe))
    for e in range(E):
        w2[e, e, 0] = 1.0
    a = np.array([[1.0, 0, 0, 0], [0, 1.0, 0, 0]])
    y = g * scipy.special.expit(g) * u          # silu(g_e) * u_e
    expect = np.array([[4 / 9 * y[0], 2 / 9 * y[1], 0.0, 0.0],
                       [0.0, 2 / 8 * y[1], 4 / 8 * y[2], 0.0]])
    desc = tiny_desc(d_model=d, n_heads=1, head_dim=4, n_experts=E, top_k=2, expert_ffn=fe, ffn=0)
    return a, {"router": router, "w13": w13, "w2": w2}, desc, expect


def test_moe_hand_example_weights_are_the_full_softmax():
    # 1 < k < E: the chosen experts keep their probabilities under the softmax
    # over ALL experts (4/9 and 2/9), not renormalised over the chosen two
    a, lw, desc, expect = _moe_hand_case()
    got = O.moe_ffn(a, lw, desc, O.Precision("fp32"))
    np.testing.assert_allclose(got, expect, rtol=1e-13, atol=1e-15)
    p, idx = O.route(a, lw["router"], 2)
    assert idx.tolist() == [[0, 1], [2, 1]]
    np.testing.assert_allclose(p, [[4 / 9, 2 / 9, 2 / 9, 1 / 9], [1 / 8, 2 / 8, 4 / 8, 1 / 8]], rtol=1e-13)


def _moe_model():
    desc = tiny_desc(n_experts=4, top_k=2, expert_ffn=4, ffn=0)
    return desc, tiny_model(desc, std=0.4)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_moe_forward_matches_bruteforce(dtype):
    desc = tiny_desc(n_experts=4, top_k=2, expert_ffn=4, ffn=0, dtype=dtype)
    m, ws = tiny_model(desc, std=0.4)
    ids = np.array([3, 7, 15, 15, 1, 15])
    bf = np.array(BF.forward_logits(desc, [w.tolist() for w in ws], list(ids), bf16_mode=(dtype == "bf16")))
    hid = O.forward(m, ids[None], O.Cache(desc, 1, len(ids)), np.arange(len(ids)))
    lg = O.lm_head_logits(m, hid[0])
    fin = np.isfinite(bf)
    assert np.array_equal(fin, np.isfinite(lg))
    tol = 1e-9 if dtype == "fp32" else 2e-2
    np.testing.assert_allclose(lg[fin], bf[fin], rtol=0, atol=tol)


def test_route_topk_matches_full_sort():
    rng = np.random.default_rng(7)
    a = rng.normal(size=(40, 16))
    r = rng.normal(size=(64, 16)) / 4
    p, idx = O.route(a, r, 8)
    for i in range(40):
        order = sorted(range(64), key=lambda e: (-p[i, e], e))
        assert list(idx[i]) == order[:8]
    # ties go to the lower expert index
    p2, idx2 = O.route(np.zeros((1, 16)), r, 3)
    assert list(idx2[0]) == [0, 1, 2]


# ---------------------------------------------------------------------------
# dual cache
# ---------------------------------------------------------------------------
def _state(desc, P, G, seed=0):
    rng = np.random.default_rng(seed)
    x = np.full((1, P + G), desc.mask_id)
    x[0, :P] = rng.integers(0, desc.mask_id, size=P)
    mask = np.zeros((1, P + G), bool); mask[0, P:] = True
    return x, mask


def test_cached_step_on_unchanged_state_reproduces_refresh():
    desc = tiny_desc(n_layers=3, vocab=32, mask_id=31)
    m, _ = tiny_model(desc)
    x, mask = _state(desc, 5, 8)
    cache = O.Cache(desc, 1, 13)
    r1 = O.refresh_step(m, x, mask, 9, 4, 0.9, cache, commit=False)
    r2 = O.cached_step(m, x, mask, 9, 4, 0.9, cache, commit=False)
    np.testing.assert_allclose(r2.logits[np.isfinite(r2.logits)], r1.logits[np.isfinite(r1.logits)], rtol=1e-10, atol=1e-10)


def test_in_place_cache_equals_explicit_concatenation():
    desc = tiny_desc(n_layers=1, vocab=32, mask_id=31)
    m, _ = tiny_model(desc)
    x, mask = _state(desc, 5, 8)
    cache = O.Cache(desc, 1, 13)
    O.refresh_step(m, x, mask, 9, 4, 0.9, cache, commit=False)
    x2 = x.copy(); x2[0, 9] = 4  # a commit changes the block
    # cached step: block rows written in place, attend over [prefix | block | suffix]
    K0, V0 = cache.K[0][0].copy(), cache.V[0][0].copy()
    r = O.cached_step(m, x2, mask.copy(), 9, 4, 0.9, cache, commit=False)
    # explicit: layer-0 block K/V recomputed, then concatenated with the stale-free prefix/suffix
    d = desc
    lw = m.layers[0]
    pos = np.arange(9, 13)
    a = O.rmsnorm(O.embed(m, x2[0, pos]), lw["attn_norm"], d.rms_eps)
    kb = O.rope(O.linear(a, lw["wk"]).reshape(4, 2, 4), pos, d.rope_theta)
    vb = O.linear(a, lw["wv"]).reshape(4, 2, 4)
    Kc = np.concatenate([K0[:9], kb, K0[13:]])
    Vc = np.concatenate([V0[:9], vb, V0[13:]])
    np.testing.assert_allclose(cache.K[0][0], Kc, rtol=1e-13)
    np.testing.assert_allclose(cache.V[0][0], Vc, rtol=1e-13)
    assert r.logits.shape == (1, 4, 32)


def _same_trajectory(ta, tb, xa, xb):
    """Equal ids, commits and (to rounding) logits at every iteration."""
    np.testing.assert_array_equal(xa, xb)
    assert len(ta) == len(tb)
    for a, b in zip(ta, tb):
        assert a.commit.tolist() == b.commit.tolist()
        fin = np.isfinite(a.logits)
        np.testing.assert_array_equal(fin, np.isfinite(b.logits))
        np.testing.assert_allclose(a.logits[fin], b.logits[fin], rtol=1e-10, atol=1e-9)


def test_one_layer_dual_cache_equals_no_cache():
    # with one layer the cached prefix/suffix K/V depend only on the embeddings
    # and positions, so the dual cache is exact: the same logits at every
    # iteration.  tau >= 1 commits one token per iteration, so every block runs
    # cached iterations (at lower tau this model fills a block at once).
    desc = tiny_desc(n_layers=1, vocab=32, mask_id=31)
    m, _ = tiny_model(desc, std=0.5)
    prompt = np.array([[1, 5, 9, 2, 7]])
    for tau in (1.0, 0.9, 0.5):
        xa, ta = O.generate(m, prompt, 12, 4, tau, cache_mode="dual", keep_logits=True)
        xb, tb = O.generate(m, prompt, 12, 4, tau, cache_mode="none", keep_logits=True)
        _same_trajectory(ta, tb, xa, xb)
        if tau >= 1.0:
            assert sum(t.iteration > 1 for t in ta) == 9          # 3 cached iterations per block


def test_two_layer_dual_cache_is_an_approximation_after_commits():
    # reported statistic: after a commit inside a block, a 2-layer model's cached
    # prefix/suffix K/V are stale, so cached logits differ from recomputation
    desc = tiny_desc(n_layers=2, vocab=32, mask_id=31)
    m, _ = tiny_model(desc, std=0.5)
    x, mask = _state(desc, 5, 8)
    cache = O.Cache(desc, 1, 13)
    O.refresh_step(m, x, mask, 5, 4, 0.9, cache, commit=False)
    x[0, 5] = 3; mask[0, 5] = False
    rc = O.cached_step(m, x, mask.copy(), 5, 4, 0.9, cache, commit=False)
    rn = O.nocache_step(m, x, mask.copy(), 5, 4, 0.9, commit=False)
    fin = np.isfinite(rc.logits)
    assert np.max(np.abs(rc.logits[fin] - rn.logits[fin])) > 1e-9


# ---------------------------------------------------------------------------
# generation: special thresholds and invariants
# ---------------------------------------------------------------------------
def test_threshold_one_is_one_token_per_step():
    desc = tiny_desc(vocab=32, mask_id=31)
    m, _ = tiny_model(desc)
    x, tr = O.generate(m, np.array([[1, 2, 3]]), 8, 4, 1.0)
    assert all(int(t.commit.sum()) == 1 for t in tr)
    assert O.iterations_per_block(tr) == {0: 4, 1: 4}


def test_threshold_zero_is_blockwise_argmax_of_full_forward():
    desc = tiny_desc(vocab=32, mask_id=31)
    m, ws = tiny_model(desc)
    prompt = [1, 2, 3]
    x, tr = O.generate(m, np.array([prompt]), 8, 4, 0.0, keep_logits=True)
    assert O.iterations_per_block(tr) == {0: 1, 1: 1}
    # brute force: each block is the argmax of one full forward over the current
    # ids, and its logits are that forward's (the argmax alone is a weak check:
    # this small model puts one token far ahead at every position)
    ids = prompt + [31] * 8
    for t, s in zip(tr, (3, 7)):
        lg = np.array(BF.forward_logits(desc, [w.tolist() for w in ws], ids))
        fin = np.isfinite(lg[s:s + 4])
        np.testing.assert_array_equal(fin, np.isfinite(t.logits[0]))
        np.testing.assert_allclose(t.logits[0][fin], lg[s:s + 4][fin], rtol=1e-9, atol=1e-9)
        for i in range(s, s + 4):
            ids[i] = int(np.argmax(lg[i]))
    assert x[0].tolist() == ids


def check_invariants(x, trace, prompt, P, G, B, mask_id, eos_id=None):
    for t in trace:
        for s in range(x.shape[0]):
            blk = t.mask_before[s, P + t.block * B:P + (t.block + 1) * B]
            if blk.any():
                assert t.commit[s].sum() >= 1                   # >= 1 commit per iteration
            assert not (t.commit[s] & ~blk).any()               # only masked positions commit
            later = slice(P + (t.block + 1) * B, None)
            ended = eos_id is not None and not t.mask_before[s, later].any() and (t.x_before[s, later] == eos_id).all()
            assert t.mask_before[s, later].all() or ended       # later blocks still masked (or the sequence ended)
            assert not t.mask_before[s, :P + t.block * B].any()    # earlier blocks done
    for blk, n in O.iterations_per_block(trace).items():
        assert 1 <= n <= B                                       # <= B iterations per block
    assert (x != mask_id).all()                                  # no mask token in the output
    np.testing.assert_array_equal(x[:, :P], prompt)              # prompt kept
    # never re-mask: once a position is committed its id stays fixed
    final = x
    for t in trace:
        done = ~t.mask_before
        assert (t.x_before[done] == final[done]).all()


def test_invariants_tiny_workload():
    cfg, run, _ = inputs.WORKLOADS["tiny_fp32"]
    m = O.Model(O.Desc.from_config(cfg), [w.numpy() for w in inputs.make_weights(cfg)])
    prompt = inputs.make_prompt(cfg, run.batch, run.prompt_len).numpy()
    x, tr = O.generate(m, prompt, run.gen_length, run.block_length, run.threshold)
    check_invariants(x, tr, prompt, run.prompt_len, run.gen_length, run.block_length, cfg.mask_id)


def test_batch_equals_independent_sequences():
    desc = tiny_desc(vocab=32, mask_id=31)
    m, _ = tiny_model(desc)
    prompts = np.array([[1, 2, 3], [4, 5, 6]])
    xb, tb = O.generate(m, prompts, 8, 4, 0.6)
    for s in range(2):
        xs, _ = O.generate(m, prompts[s:s + 1], 8, 4, 0.6)
        np.testing.assert_array_equal(xb[s], xs[0])
    check_invariants(xb, tb, prompts, 3, 8, 4, 31)


# ---------------------------------------------------------------------------
# the input generator (shared by both sides)
# ---------------------------------------------------------------------------
def test_generator_statistics_and_determinism():
    w = inputs.normal_tensor(5, (512, 512), 0.02, 0, dtype=torch.float32)
    assert abs(w.mean().item()) < 2e-4 and abs(w.std().item() - 0.02) < 3e-4
    np.testing.assert_array_equal(w.numpy(), inputs.normal_tensor(5, (512, 512), 0.02, 0, dtype=torch.float32).numpy())
    assert not torch.equal(w, inputs.normal_tensor(6, (512, 512), 0.02, 0, dtype=torch.float32))
    # tails of a normal: about 0.27% beyond 3 sigma
    frac = (w.abs() > 0.06).float().mean().item()
    assert 0.002 < frac < 0.0035
    cfg = inputs.LLADA_8B
    p = inputs.make_prompt(cfg, 4, 4096)
    assert p.min() >= 0 and p.max() < cfg.vocab and not (p == cfg.mask_id).any()
    assert p.unique().numel() > 3000


def test_lowbias32_reference_values():
    # the integer hash evaluated in int64 torch ops equals plain Python integers
    xs = [0, 1, 2, 0xDEADBEEF, 0xFFFFFFFF, 123456789]
    t = inputs._h32(torch.tensor(xs, dtype=torch.int64)).tolist()
    assert t == [inputs._h32_int(x) for x in xs]


# ---------------------------------------------------------------------------
# planted mistakes: each plausible slip in the oracle must trip a pin
# ---------------------------------------------------------------------------
def _bruteforce_gap(m, ws, desc):
    ids = np.array([3, 7, 15, 15, 1, 15])
    bf = np.array(BF.forward_logits(desc, [w.tolist() for w in ws], list(ids)))
    hid = O.forward(m, ids[None], O.Cache(desc, 1, len(ids)), np.arange(len(ids)))
    lg = O.lm_head_logits(m, hid[0])
    fin = np.isfinite(bf) & np.isfinite(lg)
    if not np.array_equal(np.isfinite(bf), np.isfinite(lg)):
        return np.inf
    return float(np.max(np.abs(lg[fin] - bf[fin])))


def _rope_wrong_sign(x, pos, theta):
    y = _ORIG["rope"](x, pos, theta)
    half = y.shape[-1] // 2
    return _ORIG["rope"](x, -np.asarray(pos), theta) if half else y


def _attn_no_scale(q, k, v):
    return _ORIG["attention"](q * np.sqrt(q.shape[-1]), k, v)


def _rms_no_gain(h, g, eps):
    return _ORIG["rmsnorm"](h, np.ones_like(np.asarray(g)), eps)


def _swiglu_swapped(a, lw, prec):
    return _ORIG["dense_ffn"](a, {"w_gate": lw["w_up"], "w_up": lw["w_gate"], "w_down": lw["w_down"]}, prec)


def _transposed_linear(x, w):
    w = np.asarray(w, dtype=np.float64)
    return np.asarray(x, dtype=np.float64) @ (w.T if w.shape[0] != w.shape[1] else w)


_ORIG = {k: getattr(O, k) for k in ("rope", "attention", "rmsnorm", "dense_ffn", "linear")}


@pytest.mark.parametrize("name,fake", [
    ("rope", _rope_wrong_sign),
    ("attention", _attn_no_scale),
    ("rmsnorm", _rms_no_gain),
    ("dense_ffn", _swiglu_swapped),
    ("linear", _transposed_linear),
])
def test_planted_mistake_is_caught(monkeypatch, name, fake):
    desc = tiny_desc()
    m, ws = tiny_model(desc, std=0.4)
    assert _bruteforce_gap(m, ws, desc) < 1e-9
    monkeypatch.setattr(O, name, fake)
    assert _bruteforce_gap(m, ws, desc) > 1e-6


COMMIT_CASES = test_threshold_commit_cases.pytestmark[0].args[1]


def _commit_cases_failing():
    """How many of the threshold-commit pin cases the oracle's commit fails."""
    bad = 0
    for conf, masked, tau, expect in COMMIT_CASES:
        got = O.threshold_commit(np.array(conf), np.array(masked, bool), tau)
        bad += int(got.astype(int).tolist() != expect)
    return bad


def _commit_ge(conf, masked, tau):
    """'>=' in place of the strict '>' of "exceeds the threshold"."""
    masked = np.asarray(masked, dtype=bool)
    if not masked.any():
        return np.zeros_like(masked)
    sel = masked & (np.asarray(conf) >= tau)
    if not sel.any():
        c = np.where(masked, conf, -np.inf)
        sel = np.zeros_like(masked)
        sel[int(np.argmax(c))] = True
    return sel


def _commit_fallback_last(conf, masked, tau):
    """Fallback to the highest position among equally confident ones."""
    masked = np.asarray(masked, dtype=bool)
    if not masked.any():
        return np.zeros_like(masked)
    sel = masked & (np.asarray(conf) > tau)
    if not sel.any():
        c = np.where(masked, conf, -np.inf)
        sel = np.zeros_like(masked)
        sel[len(c) - 1 - int(np.argmax(c[::-1]))] = True
    return sel


def _commit_always_argmax_only(conf, masked, tau):
    """Only ever the single most confident position (no parallel commit)."""
    masked = np.asarray(masked, dtype=bool)
    sel = np.zeros_like(masked)
    if masked.any():
        sel[int(np.argmax(np.where(masked, conf, -np.inf)))] = True
    return sel


@pytest.mark.parametrize("fake", [_commit_ge, _commit_fallback_last, _commit_always_argmax_only])
def test_planted_commit_mistakes_are_caught(monkeypatch, fake):
    assert _commit_cases_failing() == 0
    monkeypatch.setattr(O, "threshold_commit", fake)
    assert _commit_cases_failing() > 0


# MoE: each plausible slip in the routing weights must fail the hand example
# or the brute force (1 < k < E)
def _moe_gaps():
    a, lw, desc, expect = _moe_hand_case()
    hand = float(np.max(np.abs(O.moe_ffn(a, lw, desc, O.Precision("fp32")) - expect)))
    desc2 = tiny_desc(n_experts=4, top_k=2, expert_ffn=4, ffn=0)
    m, ws = tiny_model(desc2, std=0.4)
    return hand, _bruteforce_gap(m, ws, desc2)


def _route_renormalised(a, router, top_k):
    p, idx = _ORIG["route"](a, router, top_k)
    q = np.zeros_like(p)
    rows = np.arange(p.shape[0])[:, None]
    q[rows, idx] = p[rows, idx] / p[rows, idx].sum(-1, keepdims=True)
    return q, idx


def _route_softmax_of_chosen(a, router, top_k):
    p, idx = _ORIG["route"](a, router, top_k)
    lg = O.linear(a, router)
    rows = np.arange(p.shape[0])[:, None]
    q = np.zeros_like(p)
    q[rows, idx] = scipy.special.softmax(lg[rows, idx], axis=-1)
    return q, idx


def _route_ties_to_higher_index(a, router, top_k):
    p, _ = _ORIG["route"](a, router, top_k)
    E = p.shape[-1]
    rev = np.argsort(-p[:, ::-1], axis=-1, kind="stable")[:, :top_k]
    return p, E - 1 - rev


_ORIG["route"] = O.route


@pytest.mark.parametrize("fake", [_route_renormalised, _route_softmax_of_chosen, _route_ties_to_higher_index])
def test_planted_moe_routing_mistakes_are_caught(monkeypatch, fake):
    hand, brute = _moe_gaps()
    assert hand < 1e-12 and brute < 1e-9
    monkeypatch.setattr(O, "route", fake)
    hand, brute = _moe_gaps()
    assert max(hand, brute) > 1e-6


def test_parity_helper_generation_is_the_oracle_generation():
    # the GPU tests replay the oracle block by block through tests/parity.py;
    # that replay must be the oracle's own generate
    from tests import parity as PT
    cfg, run, _ = inputs.WORKLOADS["tiny_fp32"]
    m = O.Model(O.Desc.from_config(cfg), [w.numpy() for w in inputs.make_weights(cfg)])
    prompt = inputs.make_prompt(cfg, run.batch, run.prompt_len).numpy()
    x, tr = O.generate(m, prompt, run.gen_length, run.block_length, run.threshold)
    y, recs = PT.oracle_generation(m, prompt, run.gen_length, run.block_length, run.threshold)
    np.testing.assert_array_equal(x, y)
    assert len(recs) == len(tr)
    for a, b in zip(tr, recs):
        assert (a.block, a.iteration) == (b.block, b.iteration)
        np.testing.assert_array_equal(a.commit, b.commit)
        np.testing.assert_array_equal(a.tok, b.tok)


# ---------------------------------------------------------------------------
# the KV-cache family: dual, no cache, prefix-only, vicinity refresh
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mode,s0,B,L,w,expect", [
    ("dual", 8, 4, 20, 3, (8, 12)),
    ("none", 8, 4, 20, 3, (0, 20)),
    ("prefix", 8, 4, 20, 3, (8, 20)),
    ("vicinity", 8, 4, 20, 3, (5, 15)),
    ("vicinity", 1, 4, 20, 3, (0, 8)),      # clipped at the sequence start
    ("vicinity", 16, 4, 20, 3, (13, 20)),   # clipped at the sequence end
    ("vicinity", 8, 4, 20, 0, (8, 12)),     # w = 0 is the dual cache
])
def test_recompute_windows(mode, s0, B, L, w, expect):
    assert O.recompute_window(mode, s0, B, L, w) == expect


def test_window_steps_reduce_to_dual_and_no_cache():
    desc = tiny_desc(n_layers=2, vocab=32, mask_id=31)
    m, _ = tiny_model(desc)
    x, mask = _state(desc, 5, 8)
    x[0, 5] = 3; mask[0, 5] = False        # a commit after the refresh: the cache is stale
    s0, B, L = 5, 4, 13
    fresh = lambda: O.Cache(desc, 1, L)
    c1, c2 = fresh(), fresh()
    O.refresh_step(m, *_state(desc, 5, 8), s0, B, 0.9, c1, commit=False)
    O.refresh_step(m, *_state(desc, 5, 8), s0, B, 0.9, c2, commit=False)
    a = O.window_step(m, x.copy(), mask.copy(), s0, B, 0.9, c1, s0, s0 + B, commit=False)
    b = O.cached_step(m, x.copy(), mask.copy(), s0, B, 0.9, c2, commit=False)
    np.testing.assert_array_equal(a.logits, b.logits)          # window = block: the dual cache
    c3 = fresh()
    O.refresh_step(m, *_state(desc, 5, 8), s0, B, 0.9, c3, commit=False)
    full = O.window_step(m, x.copy(), mask.copy(), s0, B, 0.9, c3, 0, L, commit=False)
    ref = O.nocache_step(m, x.copy(), mask.copy(), s0, B, 0.9, commit=False)
    np.testing.assert_array_equal(full.logits, ref.logits)     # window = all: no cache


def test_window_step_leaves_the_cache_outside_the_window():
    desc = tiny_desc(n_layers=2, vocab=32, mask_id=31)
    m, _ = tiny_model(desc)
    x, mask = _state(desc, 5, 8)
    cache = O.Cache(desc, 1, 13)
    O.refresh_step(m, x, mask.copy(), 5, 4, 0.9, cache, commit=False)
    before = [k.copy() for k in cache.K]
    x2 = x.copy(); x2[0, 6] = 7; mask2 = mask.copy(); mask2[0, 6] = False
    O.window_step(m, x2, mask2, 5, 4, 0.9, cache, 3, 11, commit=False)
    for l in range(2):
        np.testing.assert_array_equal(cache.K[l][0, :3], before[l][0, :3])
        np.testing.assert_array_equal(cache.K[l][0, 11:], before[l][0, 11:])
    assert np.max(np.abs(cache.K[1][0, 3:11] - before[1][0, 3:11])) > 1e-9   # recomputed (stale no more)


@pytest.mark.parametrize("mode", ["prefix", "vicinity", "dual"])
def test_one_layer_every_cache_mode_equals_no_cache(mode):
    # with one layer the cached K/V depend only on embeddings and positions,
    # so every cache policy is exact
    desc = tiny_desc(n_layers=1, vocab=32, mask_id=31)
    m, _ = tiny_model(desc, std=0.5)
    prompt = np.array([[1, 5, 9, 2, 7]])
    for tau in (1.0, 0.9):
        xa, ta = O.generate(m, prompt, 12, 4, tau, cache_mode=mode, window=2, keep_logits=True)
        xb, tb = O.generate(m, prompt, 12, 4, tau, cache_mode="none", keep_logits=True)
        _same_trajectory(ta, tb, xa, xb)
        if tau >= 1.0:
            assert sum(t.iteration > 1 for t in ta) == 9


def test_vicinity_wider_than_the_sequence_is_no_cache():
    desc = tiny_desc(n_layers=2, vocab=32, mask_id=31)
    m, _ = tiny_model(desc, std=0.5)
    prompt = np.array([[1, 5, 9, 2, 7]])
    xa, ta = O.generate(m, prompt, 12, 4, 0.6, cache_mode="vicinity", window=17, keep_logits=True)
    xb, tb = O.generate(m, prompt, 12, 4, 0.6, cache_mode="none", keep_logits=True)
    np.testing.assert_array_equal(xa, xb)
    for a, b in zip(ta, tb):
        np.testing.assert_array_equal(a.logits, b.logits)


def test_prefix_cache_is_an_approximation_between_dual_and_no_cache():
    # two layers, after a commit: the prefix-only cache recomputes the suffix,
    # so it differs from the dual cache and (stale prefix) from no cache
    desc = tiny_desc(n_layers=2, vocab=32, mask_id=31)
    m, _ = tiny_model(desc, std=0.5)
    x, mask = _state(desc, 5, 8)
    caches = [O.Cache(desc, 1, 13) for _ in range(2)]
    for c in caches:
        O.refresh_step(m, x.copy(), mask.copy(), 5, 4, 0.9, c, commit=False)
    x[0, 5] = 3; mask[0, 5] = False
    pre = O.window_step(m, x.copy(), mask.copy(), 5, 4, 0.9, caches[0], 5, 13, commit=False).logits
    dual = O.cached_step(m, x.copy(), mask.copy(), 5, 4, 0.9, caches[1], commit=False).logits
    none = O.nocache_step(m, x.copy(), mask.copy(), 5, 4, 0.9, commit=False).logits
    fin = np.isfinite(pre)
    assert np.max(np.abs(pre[fin] - dual[fin])) > 1e-9
    assert np.max(np.abs(pre[fin] - none[fin])) > 1e-9


@pytest.mark.parametrize("mode", O.CACHE_MODES)
def test_invariants_every_cache_mode(mode):
    desc = tiny_desc(vocab=32, mask_id=31)
    m, _ = tiny_model(desc)
    prompts = np.array([[1, 2, 3], [4, 5, 6]])
    x, tr = O.generate(m, prompts, 12, 4, 0.6, cache_mode=mode, window=2)
    check_invariants(x, tr, prompts, 3, 12, 4, 31)


# ---------------------------------------------------------------------------
# end-of-sequence: a sequence ends at the first completed block holding eos_id
# ---------------------------------------------------------------------------
def _eos_model():
    # wider than the other tiny models so that generations vary from block to block
    desc = tiny_desc(d_model=32, n_heads=2, head_dim=16, ffn=64, vocab=64, mask_id=63)
    m, _ = tiny_model(desc)
    return desc, m


def _first_seen(x, P, B, k, avoid=()):
    """An id that the generation x first produces in block k (>= 1), in a
    block that also holds another id (so that rewriting the block would show)."""
    blk = x[P + k * B:P + (k + 1) * B]
    for v in blk:
        if v not in x[P:P + k * B] and v not in avoid and (blk != v).any():
            return int(v)
    return None


def test_eos_never_generated_changes_nothing():
    desc, m = _eos_model()
    prompt = np.array([[1, 2, 3]])
    x0, t0 = O.generate(m, prompt, 12, 4, 0.6)
    unused = next(v for v in range(63) if v not in x0[0, 3:])
    x1, t1 = O.generate(m, prompt, 12, 4, 0.6, eos_id=unused)
    np.testing.assert_array_equal(x0, x1)
    assert [t.commit.tolist() for t in t0] == [t.commit.tolist() for t in t1]


def test_eos_in_a_block_ends_the_sequence_after_it():
    desc, m = _eos_model()
    P, G, B = 3, 16, 4
    for start in range(1, 40):
        prompt = np.array([[start, start + 1, start + 2]]) % 63
        x0, t0 = O.generate(m, prompt, G, B, 0.6)
        for k in (1, 2):
            eos = _first_seen(x0[0], P, B, k)
            if eos is not None:
                break
        if eos is not None:
            break
    assert eos is not None
    x1, t1 = O.generate(m, prompt, G, B, 0.6, eos_id=eos)
    end = P + (k + 1) * B
    np.testing.assert_array_equal(x1[0, :end], x0[0, :end])      # identical through block k
    assert (x1[0, end:] == eos).all()                             # the rest is end-of-sequence
    assert max(t.block for t in t1) == k                          # no iteration after the stop
    assert len(t1) == sum(1 for t in t0 if t.block <= k)


def test_eos_in_a_batch_stops_one_sequence_only():
    desc, m = _eos_model()
    P, G, B = 3, 16, 4
    found = None
    rng = np.random.default_rng(3)
    for _ in range(60):
        prompts = rng.integers(0, 63, size=(2, P))
        x0, _ = O.generate(m, prompts, G, B, 0.6)
        for k in (1, 2):
            eos = _first_seen(x0[0], P, B, k, avoid=set(x0[1, P:].tolist()))
            if eos is not None:
                found = prompts, x0, eos, k
                break
        if found:
            break
    assert found is not None
    prompts, x0, eos, k = found
    end = P + (k + 1) * B
    x1, t1 = O.generate(m, prompts, G, B, 0.6, eos_id=eos)
    np.testing.assert_array_equal(x1[1], x0[1])                 # the other sequence runs to the end
    np.testing.assert_array_equal(x1[0, :end], x0[0, :end])
    assert (x1[0, end:] == eos).all()
    for t in t1:                                                # the ended sequence commits nothing more
        if t.block > k:
            assert not t.commit[0].any()
    check_invariants(x1, t1, prompts, P, G, B, 63, eos_id=eos)


def test_eos_in_the_prompt_does_not_stop():
    desc, m = _eos_model()
    for first in range(63):
        prompt = np.array([[first, 2, 3]])
        x0, _ = O.generate(m, prompt, 12, 4, 0.6)
        if first not in x0[0, 3:]:
            break
    x1, _ = O.generate(m, prompt, 12, 4, 0.6, eos_id=first)      # the prompt holds eos_id: no stop
    np.testing.assert_array_equal(x0, x1)


# ---------------------------------------------------------------------------
# more planted mistakes: the LM head, the activations, the cache and the
# block loop.  Each must make a pin above fail.
# ---------------------------------------------------------------------------
_ORIG.update({k: getattr(O, k) for k in ("silu", "softmax", "lm_head_logits", "embed", "refresh_step",
                                          "cached_step", "eos_stop", "recompute_window")})


def _relu_for_silu(x):
    return np.maximum(x, 0.0)


def _rope_interleaved(x, pos, theta):
    """Rotates the adjacent pairs (2i, 2i+1) instead of (i, i + hd/2)."""
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    inv = theta ** (-(2.0 * np.arange(hd // 2)) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None, None] * inv[None, None, :]
    x1, x2 = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x1 * np.cos(ang) - x2 * np.sin(ang)
    y[..., 1::2] = x2 * np.cos(ang) + x1 * np.sin(ang)
    return y


def _softmax_wrong_axis(x, axis=-1):
    return _ORIG["softmax"](x, axis=-2 if x.ndim > 1 else axis)


def _rms_eps_outside_sqrt(h, g, eps):
    h = np.asarray(h, dtype=np.float64)
    return h / (np.sqrt(np.mean(h * h, axis=-1, keepdims=True)) + 1e3 * eps) * np.asarray(g, dtype=np.float64)


def _lm_head_keeps_mask(model, h):
    d = model.desc
    a = model.prec.r(O.rmsnorm(h, model.final_norm, d.rms_eps))
    return d.logit_scale * O.linear(a, model.lm_head)


def _lm_head_unscaled(model, h):
    return _ORIG["lm_head_logits"](model, h) / model.desc.logit_scale


def _lm_head_no_final_norm(model, h):
    d = model.desc
    logits = d.logit_scale * O.linear(model.prec.r(h), model.lm_head)
    logits[:, d.mask_id] = -np.inf
    return logits


def _embed_off_by_one(model, ids):
    return np.asarray(model.embed[(np.asarray(ids) + 1) % model.desc.vocab], dtype=np.float64)


@pytest.mark.parametrize("name,fake", [
    ("silu", _relu_for_silu),
    ("rope", _rope_interleaved),
    ("softmax", _softmax_wrong_axis),
    ("rmsnorm", _rms_eps_outside_sqrt),
    ("lm_head_logits", _lm_head_keeps_mask),
    ("lm_head_logits", _lm_head_unscaled),
    ("lm_head_logits", _lm_head_no_final_norm),
    ("embed", _embed_off_by_one),
])
def test_planted_forward_mistake_is_caught(monkeypatch, name, fake):
    desc = tiny_desc()
    m, ws = tiny_model(desc, std=0.4)
    assert _bruteforce_gap(m, ws, desc) < 1e-9
    monkeypatch.setattr(O, name, fake)
    assert _bruteforce_gap(m, ws, desc) > 1e-6


def _refresh_block_rows_only(model, x, mask, s0, B, tau, cache, commit=True):
    """A 'refresh' that computes only the block's rows: prefix and suffix K/V never cached."""
    hid = O.forward(model, x, cache, np.arange(s0, s0 + B))
    return O.decode_block(model, hid, x, mask, s0, B, tau, commit)


def _cached_step_without_cache(model, x, mask, s0, B, tau, cache, commit=True):
    """A cached iteration that attends over the block only (an empty cache)."""
    fresh = O.Cache(model.desc, x.shape[0], x.shape[1])
    hid = O.forward(model, x, fresh, np.arange(s0, s0 + B))
    return O.decode_block(model, hid, x, mask, s0, B, tau, commit)


def _eos_overwrites_the_block(x, mask, s0, B, eos_id):
    """Fills from the block's first position, rewriting committed tokens."""
    for i in range(x.shape[0]):
        if (x[i, s0:s0 + B] == eos_id).any():
            x[i, s0:] = eos_id
            mask[i, s0:] = False


def _eos_stops_every_sequence(x, mask, s0, B, eos_id):
    """Ends the whole batch when any sequence's block holds eos_id."""
    if (x[:, s0:s0 + B] == eos_id).any():
        x[:, s0 + B:] = eos_id
        mask[:, s0 + B:] = False


def _vicinity_one_sided(cache_mode, s0, B, L, w=0):
    if cache_mode == "vicinity":
        return max(0, s0 - w), s0 + B
    return _ORIG["recompute_window"](cache_mode, s0, B, L, w)


def _pin_fails(pin, *args):
    try:
        pin(*args)
    except AssertionError:
        return True
    return False


def _window_pins():
    return [_pin_fails(test_recompute_windows, *case) for case in
            test_recompute_windows.pytestmark[0].args[1]]


@pytest.mark.parametrize("name,fake,pins", [
    ("refresh_step", _refresh_block_rows_only, (test_threshold_zero_is_blockwise_argmax_of_full_forward,)),
    ("cached_step", _cached_step_without_cache, (test_one_layer_dual_cache_equals_no_cache,)),
    ("eos_stop", _eos_overwrites_the_block, (test_eos_in_a_block_ends_the_sequence_after_it,)),
    ("eos_stop", _eos_stops_every_sequence, (test_eos_in_a_batch_stops_one_sequence_only,)),
])
def test_planted_loop_mistake_is_caught(monkeypatch, name, fake, pins):
    for pin in pins:
        assert not _pin_fails(pin)
    monkeypatch.setattr(O, name, fake)
    assert any(_pin_fails(pin) for pin in pins)


def test_planted_window_mistake_is_caught(monkeypatch):
    assert not any(_window_pins())
    monkeypatch.setattr(O, "recompute_window", _vicinity_one_sided)
    assert any(_window_pins())


def _attention_causal(q, k, v, rows_per_group=1024):
    """A causal LM's attention: query i sees keys up to its own position."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    nq, nk = q.shape[0], k.shape[0]
    s = np.einsum("qhd,khd->hqk", q, k) / np.sqrt(q.shape[-1])
    later = np.arange(nk)[None, :] > np.arange(nq)[:, None] + (nk - nq)
    return np.einsum("hqk,khd->qhd", _ORIG["softmax"](np.where(later[None], -np.inf, s), axis=-1), v)


def _conf_squared(logits):
    tok = np.argmax(logits, axis=-1)
    lmax = logits[np.arange(logits.shape[0]), tok]
    return tok.astype(np.int64), 1.0 / np.sum(np.exp(logits - lmax[:, None]), axis=-1) ** 2


def _commit_ignores_mask(conf, masked, tau):
    """Commits every confident position, masked or not."""
    masked = np.asarray(masked, dtype=bool)
    if not masked.any():
        return np.zeros_like(masked)
    sel = np.asarray(conf) > tau
    if not (sel & masked).any():
        c = np.where(masked, conf, -np.inf)
        sel = np.zeros_like(masked)
        sel[int(np.argmax(c))] = True
    return sel


def _window_decodes_first_rows(model, x, mask, s0, B, tau, cache, r0, r1, commit=True):
    """Decodes the window's first B rows instead of the block's."""
    hid = O.forward(model, x, cache, np.arange(r0, r1))
    return O.decode_block(model, hid[:, :B], x, mask, s0, B, tau, commit)


def _eos_seen_in_the_prompt(x, mask, s0, B, eos_id):
    """Stops on eos_id anywhere before the block's end, the prompt included."""
    for i in range(x.shape[0]):
        if (x[i, :s0 + B] == eos_id).any():
            x[i, s0 + B:] = eos_id
            mask[i, s0 + B:] = False


def _route_one_expert_short(a, router, top_k):
    return _ORIG["route"](a, router, max(1, top_k - 1))


def _decode_rewrites_committed(model, hidden, x, mask, s0, B, tau, commit=True):
    """Also rewrites positions committed in earlier iterations with the new top-1."""
    done = ~mask[:, s0:s0 + B].copy()
    r = _ORIG["decode_block"](model, hidden, x, mask, s0, B, tau, commit)
    if commit:
        x[:, s0:s0 + B][done] = r.tok[done]
    return r


def _no_rounding(self, x):
    return np.asarray(x, dtype=np.float64)


_ORIG["decode_block"] = O.decode_block


@pytest.mark.parametrize("owner,name,fake,pins", [
    (O, "attention", _attention_causal, (test_bidirectional_no_causal_mask, test_attention_closed_forms)),
    (O.Precision, "r", _no_rounding, (lambda: test_forward_matches_bruteforce("bf16"),)),
    (O, "top1_confidence", _conf_squared, (test_top1_confidence_closed_form,)),
    (O, "threshold_commit", _commit_ignores_mask,
     (lambda: test_threshold_commit_cases(*test_threshold_commit_cases.pytestmark[0].args[1][1]),
      test_eos_in_a_batch_stops_one_sequence_only)),
    (O, "window_step", _window_decodes_first_rows, (test_vicinity_wider_than_the_sequence_is_no_cache,)),
    (O, "eos_stop", _eos_seen_in_the_prompt, (test_eos_in_the_prompt_does_not_stop,)),
    (O, "route", _route_one_expert_short, (test_moe_hand_example_weights_are_the_full_softmax,
                                           test_route_topk_matches_full_sort)),
    (O, "decode_block", _decode_rewrites_committed, (test_invariants_tiny_workload,)),
], ids=["causal-attention", "no-bf16-rounding", "confidence-squared", "commit-ignores-mask",
        "window-decodes-first-rows", "eos-in-prompt-stops", "top-k-minus-one", "decode-rewrites-committed"])
def test_planted_mistake_fails_its_pin(monkeypatch, owner, name, fake, pins):
    for pin in pins:
        assert not _pin_fails(pin)
    monkeypatch.setattr(owner, name, fake)
    assert any(_pin_fails(pin) for pin in pins)
