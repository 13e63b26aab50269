"""The GPU parity harness checked on the CPU (no GPU): tests/parity.py's
teacher-forced comparison is run against a stand-in for the library's
decoder that answers with the oracle under its CPU model of the GPU's
arithmetic.  Faithful, it must pass at the tolerance derived from the same
model; with a planted mistake -- a wrong token or commit at a decision the
tolerance does not flag, a logit off by more than delta, a confidence
outside its interval -- the harness must report it.  This keeps the GPU
parity tests from passing vacuously."""
import numpy as np
import pytest
import torch

from block_denoising_gb300 import inputs
from oracle import dinfer_oracle as O
from tests import parity as PT

CFG = inputs.shrink(inputs.LLADA_8B, n_layers=1, d_model=256, n_heads=2, ffn=512, vocab=512, mask_id=511)
P, G, B, TAU = 32, 32, 16, 0.9


class StandIn:
    """Answers prefill_cache / block_step like the library's Decoder, through
    the debug outputs, from the oracle under parity.gpu_arithmetic();
    `plant(logits, tok, conf, masked)` may alter what it reports and commits."""

    def __init__(self, m, plant=None):
        self.m, self.plant = m, plant
        self.out = (None, None, None)
        self.fin = None
        self.cache = None
        self.s0 = self.B = None
        self.steps = 0

    def set_debug_outputs(self, lg, tk, cf):
        self.out = (lg, tk, cf)

    def set_debug_hidden(self, hid, fin):
        self.fin = fin

    def sync(self):
        pass

    def prefill_cache(self, ids, mask, s0, b_len, tau, commit=True):
        self.s0, self.B = s0, b_len
        self.cache = O.Cache(self.m.desc, ids.shape[0], ids.shape[1])
        self._step(ids, mask, tau, O.refresh_step)

    def block_step(self, ids, mask, tau):
        self._step(ids, mask, tau, O.cached_step)

    def _step(self, ids, mask, tau, fn):
        s0, Bl = self.s0, self.B
        x = ids.numpy().astype(np.int64)
        mk = mask.numpy().astype(bool)
        with PT.gpu_arithmetic():
            r = fn(self.m, x, mk, s0, Bl, tau, self.cache, commit=False)
        logits, tok, conf = r.logits.copy(), r.tok.copy(), r.conf.copy()
        if self.plant is not None:
            logits, tok, conf = self.plant(self.steps, logits, tok, conf, mk[:, s0:s0 + Bl])
        self.steps += 1
        for i in range(x.shape[0]):
            sel = O.threshold_commit(conf[i], mk[i, s0:s0 + Bl], tau)
            x[i, s0:s0 + Bl][sel] = tok[i][sel]
            mk[i, s0:s0 + Bl][sel] = False
        lg, tk, cf = self.out
        lg.copy_(torch.from_numpy(logits.reshape(lg.shape).astype(np.float32)))
        tk.copy_(torch.from_numpy(tok.reshape(-1).astype(np.int32)))
        cf.copy_(torch.from_numpy(conf.reshape(-1).astype(np.float32)))
        ids.copy_(torch.from_numpy(x.astype(np.int32)))
        mask.copy_(torch.from_numpy(mk.astype(np.uint8)))
        if self.fin is not None:
            a = self.m.prec.r(O.rmsnorm(r.hidden, self.m.final_norm, self.m.desc.rms_eps))
            self.fin.copy_(torch.from_numpy(a.reshape(self.fin.shape).astype(np.float32)).to(self.fin.dtype))


@pytest.fixture(scope="module")
def case():
    W = inputs.make_weights(CFG, 0)
    m = O.Model(O.Desc.from_config(CFG), [w.float().numpy() for w in W])
    prompt = inputs.make_prompt(CFG, 2, P).numpy()
    _, recs = PT.oracle_generation(m, prompt, G, B, TAU)
    tol = PT.tolerance_from_floor(*PT.model_floor(m, recs, B, TAU))
    assert tol["delta"] > 0
    return m, recs, tol


def _run(case, plant=None):
    m, recs, tol = case
    return PT.gpu_compare(None, StandIn(m, plant), recs, m, B, TAU, tol, "cpu", lm_head_check=True)


def _unflagged_position(recs, tol):
    """(record, sequence, block position) of an unflagged decision: the one
    with the widest top-2 logit margin over all records."""
    best = (-np.inf, None)
    for k, r in enumerate(recs):
        fl = PT.flags_for(r.logits, r.conf, r.mask_before[:, r.s0:r.s0 + B], TAU, tol["delta"])
        srt = np.sort(r.logits, axis=-1)
        gap = np.where(fl, -np.inf, srt[..., -1] - srt[..., -2])
        i, j = np.unravel_index(int(np.argmax(gap)), gap.shape)
        if gap[i, j] > best[0]:
            best = (gap[i, j], (k, int(i), int(j)))
    assert best[1] is not None and np.isfinite(best[0])
    return best[1]


def test_faithful_stand_in_passes_and_checks_real_decisions(case):
    m, recs, tol = case
    st = _run(case)
    PT.assert_parity(st, tol)
    decisions = sum(r.conf.size for r in recs)
    assert st["n"] > 0 and st["flagged"] < decisions         # some decisions are compared exactly
    assert st["max_err"] > 0                                   # the stand-in really differs by rounding


def test_wrong_unflagged_token_is_caught(case):
    m, recs, tol = case
    k, i, j = _unflagged_position(recs, tol)

    def plant(step, logits, tok, conf, masked):
        if step == k:
            tok = tok.copy()
            tok[i, j] = (tok[i, j] + 1) % (CFG.vocab - 1)
        return logits, tok, conf

    st = _run(case, plant)
    assert st["unflagged_mismatch"] > 0
    with pytest.raises(AssertionError):
        PT.assert_parity(st, tol)


def test_logit_beyond_delta_is_caught(case):
    m, recs, tol = case

    def plant(step, logits, tok, conf, masked):
        logits = logits.copy()
        logits[0, 0, 7] += 1.5 * tol["delta"]
        return logits, tok, conf

    st = _run(case, plant)
    assert st["max_err"] >= 1.5 * tol["delta"] * 0.99
    with pytest.raises(AssertionError):
        PT.assert_parity(st, tol)


def test_confidence_outside_its_interval_is_caught(case):
    m, recs, tol = case

    def plant(step, logits, tok, conf, masked):
        return logits, tok, conf * 0.5

    st = _run(case, plant)
    assert st["conf_outside"] > 0
    with pytest.raises(AssertionError):
        PT.assert_parity(st, tol)


def test_missing_commit_is_caught(case):
    m, recs, tol = case

    def plant(step, logits, tok, conf, masked):
        # every confidence below the threshold: only the fallback position commits
        return logits, tok, np.minimum(conf, TAU * 0.999)

    st = _run(case, plant)
    with pytest.raises(AssertionError):
        PT.assert_parity(st, tol)


def test_follow_gpu_checks_the_stand_ins_own_trajectory(case):
    """parity.follow_gpu (used for the production graph path) follows the
    decoder's own trajectory and compares every decision against the
    oracle's at that state: faithful, it passes; committing a wrong token
    wherever a decision is clear (top-2 margin far above 2 delta, confidence
    far above the threshold), it fails."""
    m, _, tol0 = case
    prompt = inputs.make_prompt(CFG, 2, P).numpy()
    tol_fn = lambda recs: PT.tolerance_from_floor(*PT.model_floor(m, recs, B, TAU))
    x, st, recs, tol = PT.follow_gpu(None, StandIn(m), m, prompt, G, B, TAU, tol_fn, "cpu")
    PT.assert_parity(st, tol, lm_head=False)
    assert not (x == CFG.mask_id).any() and (x[:, :P] == prompt).all()

    def plant(step, logits, tok, conf, masked):
        srt = np.sort(logits, axis=-1)
        clear = masked & (srt[..., -1] - srt[..., -2] > 6 * tol0["delta"]) & (conf > TAU + 0.05)
        tok = np.where(clear, (tok + 1) % (CFG.vocab - 1), tok)
        return logits, tok, conf

    _, st2, _, tol2 = PT.follow_gpu(None, StandIn(m, plant), m, prompt, G, B, TAU, tol_fn, "cpu")
    assert st2["unflagged_mismatch"] > 0
    with pytest.raises(AssertionError):
        PT.assert_parity(st2, tol2, lm_head=False)


def test_route_flags_map_router_calls_to_sequences_and_block_rows():
    """The oracle's forward routes layer by layer, sequence by sequence, over
    the rows it computes (all positions at a refresh, the window otherwise);
    route_flags_for must pick each sequence's block rows out of those calls."""
    Bl, b, L, s0 = 4, 2, 12, 4

    class R:
        pass

    def rec(iteration, window, margins):
        r = R()
        r.iteration, r.s0, r.window, r.margins = iteration, s0, window, margins
        r.x_before = np.zeros((b, L), np.int64)
        return r

    big = lambda n: np.full(n, 1.0)
    # refresh: rows 0..11; sequence 1's block row 2 (position 6) is a near-tie in layer 1
    m1 = [big(L), big(L), big(L), big(L)]          # calls: (l0, s0), (l0, s1), (l1, s0), (l1, s1)
    m1[3] = m1[3].copy(); m1[3][s0 + 2] = 0.001
    # cached iteration recomputing the window [2, 10): sequence 0's block row 0 (position 4) in layer 0
    m2 = [big(8), big(8), big(8), big(8)]
    m2[0] = m2[0].copy(); m2[0][s0 - 2] = 0.001
    f1, f2 = PT.route_flags_for([rec(1, (0, L), m1), rec(2, (2, 10), m2)], 0.02, Bl)
    want1 = np.zeros((b, Bl), bool); want1[1, 2] = True
    want2 = np.zeros((b, Bl), bool); want2[0, 0] = True
    np.testing.assert_array_equal(f1, want1)
    np.testing.assert_array_equal(f2, want2)


def test_confidence_interval_is_the_reach_of_a_delta_logit_error():
    """conf_interval's ends are the confidences of the logits moved by delta
    against and for the top token, and every logit error within delta that
    keeps the argmax lands inside."""
    rng = np.random.default_rng(5)
    logits = rng.normal(size=(6, 50)) * 3.0
    delta = 0.4
    tok = logits.argmax(-1)
    conf = 1.0 / np.exp(logits - logits.max(-1, keepdims=True)).sum(-1)
    lo, hi = PT.conf_interval(conf, delta)
    top = np.zeros_like(logits, bool); top[np.arange(6), tok] = True
    worst = np.where(top, logits - delta, logits + delta)
    best = np.where(top, logits + delta, logits - delta)
    c = lambda l: np.exp(l[np.arange(6), tok]) / np.exp(l).sum(-1)
    np.testing.assert_allclose(lo, c(worst), rtol=1e-12)
    np.testing.assert_allclose(hi, c(best), rtol=1e-12)
    for _ in range(200):
        pert = logits + rng.uniform(-delta, delta, size=logits.shape)
        keep = pert.argmax(-1) == tok
        cp = c(pert)
        assert np.all((cp[keep] >= lo[keep] - 1e-12) & (cp[keep] <= hi[keep] + 1e-12))


@pytest.mark.parametrize("seed", range(4))
def test_unflagged_decisions_survive_every_delta_logit_error(seed):
    """flags_for is sound: at a position it leaves unflagged, no logit error
    within delta changes the top-1 token or the commit decision."""
    rng = np.random.default_rng(seed)
    b, Bl, V, tau, delta = 2, 16, 40, 0.9, 0.15
    logits = rng.normal(size=(b, Bl, V)) * rng.uniform(1.0, 4.0, size=(b, Bl, 1))
    logits[..., V - 1] = -np.inf                                   # the mask token
    masked = rng.random((b, Bl)) < 0.7
    masked[:, 0] = True

    def decide(lg):
        tok, conf = np.zeros((b, Bl), np.int64), np.zeros((b, Bl))
        com = np.zeros((b, Bl), bool)
        for i in range(b):
            tok[i], conf[i] = O.top1_confidence(lg[i])
            com[i] = O.threshold_commit(conf[i], masked[i], tau)
        return tok, conf, com

    tok, conf, com = decide(logits)
    fl = PT.flags_for(logits, conf, masked, tau, delta)
    assert (~fl).any()
    for _ in range(300):
        pert = logits + rng.uniform(-delta, delta, size=logits.shape)
        t2, _, c2 = decide(pert)
        assert np.array_equal(t2[~fl], tok[~fl])
        assert np.array_equal(c2[~fl], com[~fl])
