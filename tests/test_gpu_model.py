"""Model-level parity of the CUDA decoder against the oracle (through the C-ABI).

Every GPU iteration starts from the oracle's (ids, mask) state -- the
trajectory teacher-forced from the oracle -- and is compared on logits,
tokens, confidences and the commit set.  A decision is flagged (counted and
reported, allowed to differ) only if a logit error within the tolerance
delta could flip it: a top-2 logit gap below 2 delta (at least 1e-2), a
threshold inside the confidence interval that delta allows (or within 1e-2
of the confidence), or a fallback choice among positions whose intervals
overlap.  Every unflagged decision must match exactly.
"""

import numpy as np
import pytest
import torch

from block_denoising_gb300 import inputs
from oracle import dinfer_oracle as O

pytestmark = pytest.mark.gpu
dev = torch.device("cuda:0")

# Tolerances.  fp32: the stated ones (logits 1e-4, confidence 1e-2).  bf16:
# the logit bound delta is derived from the bf16 contract itself -- two
# correct fp32-accumulating implementations of the same bf16 rounding points
# differ by rare rounding flips that cascade through norm and attention; the
# floor is measured on the CPU in tests/test_tolerances.py and delta is set to
# about twice it.  Flags then follow from delta exactly (see flags_for).
FP32 = dict(delta=1e-4, logit_mean=1e-5)
BF16_SMALL = dict(delta=0.6, logit_mean=0.08)
BF16_LONG = dict(delta=0.8, logit_mean=0.14)  # d_model 1024, refresh of 2048 rows
NS_GAP, NS_CONF = 1e-2, 1e-2  # flag widths stated for the method's parity check


def conf_interval(conf, delta):
    """Confidences reachable when the top logit moves by +-delta and all others by -+delta."""
    c = np.clip(conf, 1e-300, 1.0)
    r = np.maximum(1.0 / c - 1.0, 0.0)
    return 1.0 / (1.0 + r * np.exp(2 * delta)), 1.0 / (1.0 + r * np.exp(-2 * delta))


@pytest.fixture(scope="module")
def D():
    from block_denoising_gb300 import build, dinfer
    build.build()
    return dinfer


def flags_for(rec, tau, tol, B, s0):
    """Block positions whose decision a logit error of at most delta could flip.

    token: top-2 logit gap < max(2 delta, 1e-2); threshold: tau inside the
    confidence interval (or |conf - tau| < 1e-2); fallback (no confidence
    above tau): every masked position whose interval reaches the lower end of
    the best one's.
    """
    d = tol["delta"]
    lg = rec.logits
    b = lg.shape[0]
    fl = np.zeros((b, B), dtype=bool)
    for i in range(b):
        srt = np.sort(lg[i], axis=-1)
        fl[i] |= (srt[:, -1] - srt[:, -2]) < max(2 * d, NS_GAP)
        lo, hi = conf_interval(rec.conf[i], d)
        fl[i] |= ((lo <= tau) & (tau < hi)) | (np.abs(rec.conf[i] - tau) < NS_CONF)
        masked = rec.mask_before[i, s0:s0 + B]
        if masked.any() and not (hi[masked] > tau).any():
            best = int(np.argmax(np.where(masked, rec.conf[i], -np.inf)))
            fl[i] |= masked & (hi >= lo[best] - NS_CONF)
    return fl


def teacher_forced(D, cfg, W, prompt, G, B, tau, tol, max_blocks=None, route_margin=None):
    """Run every oracle iteration on the GPU from the oracle's state; return error statistics.

    route_margin (MoE models): block rows whose router top-k margin (k-th minus
    (k+1)-th router logit, any layer) is below it are flagged too -- a routing
    decision inside the bf16 noise can send the row to another expert.
    """
    m = O.Model(O.Desc.from_config(cfg), [w.float().numpy() for w in W])
    margins = []
    if route_margin is not None:
        orig_route = O.route

        def recording_route(a, router, top_k):
            lg = O.linear(a, router)
            srt = np.sort(lg, axis=-1)[:, ::-1]
            margins.append(srt[:, top_k - 1] - srt[:, top_k])
            return orig_route(a, router, top_k)

        O.route = recording_route
    try:
        x, trace = O.generate(m, prompt, G, B, tau, keep_logits=True, max_blocks=max_blocks)
    finally:
        if route_margin is not None:
            O.route = orig_route
    b, P = prompt.shape
    L = P + G
    dec = D.Decoder(cfg, [w.to(dev) for w in W], max_batch=b, max_seq=L)
    lg = torch.empty((b * B, cfg.vocab), dtype=torch.float32, device=dev)
    tk = torch.empty(b * B, dtype=torch.int32, device=dev)
    cf = torch.empty(b * B, dtype=torch.float32, device=dev)
    dec.set_debug_outputs(lg, tk, cf)
    out = dict(max_err=0.0, sum_err=0.0, n=0, conf_err=0.0, conf_outside=0, tok_mismatch=0, commit_mismatch=0, flagged=0,
               unflagged_mismatch=0, iterations=len(trace), route_flagged_rows=0)
    # routing margins per iteration: each forward calls route once per layer
    per_iter = []
    if route_margin is not None:
        nl = cfg.n_layers
        b_ = prompt.shape[0]
        k = 0
        for rec in trace:
            rows_fwd = b_ * (P + G) if rec.iteration == 1 else b_ * B
            ms = []
            for _ in range(nl):
                mm = []
                for _s in range(b_):
                    mm.append(margins[k]); k += 1
                ms.append(mm)
            per_iter.append(ms)
    for it_i, rec in enumerate(trace):
        s0 = P + rec.block * B
        ids = torch.tensor(rec.x_before, dtype=torch.int32, device=dev)
        mask = torch.tensor(rec.mask_before.astype(np.uint8), device=dev)
        if rec.iteration == 1:
            dec.prefill_cache(ids, mask, s0, B, tau, commit=True)
        else:
            dec.block_step(ids, mask, tau)
        dec.sync()
        g_lg = lg.cpu().numpy().reshape(b, B, -1)
        fin = np.isfinite(rec.logits)
        assert np.array_equal(fin, np.isfinite(g_lg))
        if route_margin is not None:  # rows routed differently may differ beyond delta
            rows_ok = np.ones((b, B), bool)
            for si in range(b):
                mins = np.full(B, np.inf)
                for lm in per_iter[it_i]:
                    mg = lm[si]
                    mg = mg[s0:s0 + B] if len(mg) > B else mg
                    mins = np.minimum(mins, mg)
                rows_ok[si] = mins >= route_margin
            fin = fin & rows_ok[:, :, None]
        e = np.abs(g_lg[fin] - rec.logits[fin])
        out["max_err"] = max(out["max_err"], float(e.max()))
        out["sum_err"] += float(e.sum())
        out["n"] += e.size
        g_conf = cf.cpu().numpy().reshape(b, B)
        out["conf_err"] = max(out["conf_err"], float(np.abs(g_conf - rec.conf).max()))
        lo, hi = conf_interval(rec.conf, tol["delta"])
        out["conf_outside"] += int(((g_conf < lo - 1e-6) | (g_conf > hi + 1e-6)).sum())
        g_tok = tk.cpu().numpy().reshape(b, B)
        g_mask = mask.cpu().numpy().astype(bool)
        g_commit = rec.mask_before[:, s0:s0 + B] & ~g_mask[:, s0:s0 + B]
        fl = flags_for(rec, tau, tol, B, s0)
        if route_margin is not None:
            for si in range(b):
                mins = np.full(B, np.inf)
                for lm in per_iter[it_i]:
                    mg = lm[si]
                    mg = mg[s0:s0 + B] if len(mg) > B else mg  # refresh: all rows; iteration: block rows
                    mins = np.minimum(mins, mg)
                rf = mins < route_margin
                out["route_flagged_rows"] += int(rf.sum())
                fl[si] |= rf
        out["flagged"] += int(fl.sum())
        tm = g_tok != rec.tok
        cm = g_commit != rec.commit
        out["tok_mismatch"] += int(tm.sum())
        out["commit_mismatch"] += int(cm.sum())
        out["unflagged_mismatch"] += int(((tm | cm) & ~fl).sum())
        # committed positions received the GPU's own token
        g_ids = ids.cpu().numpy()
        assert np.array_equal(g_ids[:, s0:s0 + B][g_commit], g_tok[g_commit])
    dec.close()
    out["mean_err"] = out["sum_err"] / max(1, out["n"])
    return out, x, trace


def check_generation_invariants(out_ids, prompt, G, B, mask_id, stats):
    b, P = prompt.shape
    assert out_ids.shape == (b, P + G)
    assert np.array_equal(out_ids[:, :P], prompt)
    assert (out_ids != mask_id).all()
    assert stats["n_blocks"] == G // B
    assert stats["refreshes"] == G // B
    assert all(1 <= n <= B for n in stats["iters_per_block"])
    assert stats["iterations"] == sum(stats["iters_per_block"])


# ---------------------------------------------------------------------------
# tiny fp32 model (the full workload: 2 layers, d 256, V 4096, P32 G64 B16)
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def tiny():
    cfg, run, _ = inputs.WORKLOADS["tiny_fp32"]
    return cfg, run, inputs.make_weights(cfg, 0), inputs.make_prompt(cfg, run.batch, run.prompt_len)


def test_tiny_fp32_teacher_forced(D, tiny):
    cfg, run, W, prompt = tiny
    st, _, _ = teacher_forced(D, cfg, W, prompt.numpy(), run.gen_length, run.block_length, run.threshold, FP32)
    print(st)
    assert st["max_err"] < FP32["delta"]
    assert st["mean_err"] < FP32["logit_mean"]
    assert st["conf_err"] < NS_CONF and st["conf_outside"] == 0
    assert st["unflagged_mismatch"] == 0


def test_tiny_fp32_generate_matches_oracle(D, tiny):
    cfg, run, W, prompt = tiny
    dec = D.Decoder(cfg, [w.to(dev) for w in W], max_batch=1, max_seq=run.seq_len)
    out, stats = dec.generate(prompt.to(dev), run.gen_length, run.block_length, run.threshold)
    got = out.cpu().numpy()
    m = O.Model(O.Desc.from_config(cfg), [w.numpy() for w in W])
    x, trace = O.generate(m, prompt.numpy(), run.gen_length, run.block_length, run.threshold)
    check_generation_invariants(got, prompt.numpy(), run.gen_length, run.block_length, cfg.mask_id, stats)
    assert np.array_equal(got, x)
    assert stats["iters_per_block"] == [O.iterations_per_block(trace)[k] for k in range(len(stats["iters_per_block"]))]
    # host prompt / host output buffers give the same result
    out_h, _ = dec.generate(prompt, run.gen_length, run.block_length, run.threshold,
                            out=torch.empty((1, run.seq_len), dtype=torch.int32))
    assert np.array_equal(out_h.numpy(), x)
    dec.close()


@pytest.mark.parametrize("tau", [0.0, 1.0])
def test_tiny_fp32_special_thresholds(D, tiny, tau):
    cfg, run, W, prompt = tiny
    dec = D.Decoder(cfg, [w.to(dev) for w in W], max_batch=1, max_seq=run.seq_len)
    out, stats = dec.generate(prompt.to(dev), run.gen_length, run.block_length, tau)
    nb = run.gen_length // run.block_length
    if tau == 0.0:   # whole block at the refresh
        assert stats["iters_per_block"] == [1] * nb
    else:            # one token per step
        assert stats["iters_per_block"] == [run.block_length] * nb
    m = O.Model(O.Desc.from_config(cfg), [w.numpy() for w in W])
    x, _ = O.generate(m, prompt.numpy(), run.gen_length, run.block_length, tau)
    assert np.array_equal(out.cpu().numpy(), x)
    dec.close()


# ---------------------------------------------------------------------------
# small bf16 models on the tensor-core path
# ---------------------------------------------------------------------------
SMALL_BF16 = inputs.shrink(inputs.LLADA_8B, n_layers=2, d_model=512, n_heads=4, ffn=1024, vocab=2048,
                           mask_id=2047)


@pytest.mark.parametrize("batch,P,G,B,tau", [(1, 64, 64, 32, 0.9), (2, 40, 48, 16, 0.7)])
def test_small_bf16_teacher_forced(D, batch, P, G, B, tau):
    W = inputs.make_weights(SMALL_BF16, 0)
    prompt = inputs.make_prompt(SMALL_BF16, batch, P).numpy()
    st, _, _ = teacher_forced(D, SMALL_BF16, W, prompt, G, B, tau, BF16_SMALL)
    print(st)
    assert st["max_err"] < BF16_SMALL["delta"]
    assert st["mean_err"] < BF16_SMALL["logit_mean"]
    assert st["conf_outside"] == 0
    assert st["unflagged_mismatch"] == 0


# A refresh of 2048 rows at d_model 1024: the O projection runs as whole
# 128-token tiles (128 CTAs, residual added in the GEMM's epilogue), the other
# GEMMs stream-K, and both residual norms take the many-rows variant (the FFN
# norm a plain row norm, the next-layer norm with the down projection's
# partials).  First block only: its refresh and cached iterations.
LONG_BF16 = inputs.shrink(inputs.LLADA_8B, n_layers=2, d_model=1024, n_heads=8, ffn=2048, vocab=2048,
                          mask_id=2047)


def test_long_refresh_bf16_teacher_forced(D):
    W = inputs.make_weights(LONG_BF16, 0)
    prompt = inputs.make_prompt(LONG_BF16, 1, 1984).numpy()
    st, _, _ = teacher_forced(D, LONG_BF16, W, prompt, 64, 32, 0.9, BF16_LONG, max_blocks=1)
    print(st)
    assert st["max_err"] < BF16_LONG["delta"]
    assert st["mean_err"] < BF16_LONG["logit_mean"]
    assert st["conf_outside"] == 0
    assert st["unflagged_mismatch"] == 0


def test_small_bf16_generate_invariants_and_graph_equals_eager(D):
    W = [w.to(dev) for w in inputs.make_weights(SMALL_BF16, 0)]
    P, G, B = 64, 96, 32
    prompt = inputs.make_prompt(SMALL_BF16, 2, P, device=dev)
    dec = D.Decoder(SMALL_BF16, W, max_batch=2, max_seq=P + G)
    a, sa = dec.generate(prompt, G, B, 0.9)
    b, sb = dec.generate(prompt, G, B, 0.9)
    check_generation_invariants(a.cpu().numpy(), prompt.cpu().numpy(), G, B, SMALL_BF16.mask_id, sa)
    assert torch.equal(a, b) and sa["iters_per_block"] == sb["iters_per_block"]
    # same trajectory when the loop is driven step by step through the ABI (graphs per step)
    ids = torch.full((2, P + G), SMALL_BF16.mask_id, dtype=torch.int32, device=dev)
    ids[:, :P] = prompt
    mask = torch.zeros((2, P + G), dtype=torch.uint8, device=dev)
    mask[:, P:] = 1
    for blk in range(G // B):
        s0 = P + blk * B
        dec.prefill_cache(ids, mask, s0, B, 0.9)
        n = 1
        while mask[:, s0:s0 + B].any():
            dec.block_step(ids, mask, 0.9)
            n += 1
        assert n == sa["iters_per_block"][blk]
    assert torch.equal(ids, a)
    dec.close()


def test_cached_step_on_unchanged_state_reproduces_refresh(D):
    W = [w.to(dev) for w in inputs.make_weights(SMALL_BF16, 0)]
    P, G, B = 64, 64, 32
    prompt = inputs.make_prompt(SMALL_BF16, 1, P, device=dev)
    ids = torch.full((1, P + G), SMALL_BF16.mask_id, dtype=torch.int32, device=dev)
    ids[:, :P] = prompt
    mask = torch.zeros((1, P + G), dtype=torch.uint8, device=dev)
    mask[:, P:] = 1
    dec = D.Decoder(SMALL_BF16, W, max_batch=1, max_seq=P + G)
    lg = torch.empty((B, SMALL_BF16.vocab), dtype=torch.float32, device=dev)
    dec.set_debug_outputs(logits=lg)
    dec.prefill_cache(ids, mask, P, B, 0.9, commit=False)
    dec.sync()
    a = lg.clone()
    dec.block_step(ids, mask, 0.9)
    dec.sync()
    fin = torch.isfinite(a)
    assert torch.equal(fin, torch.isfinite(lg))
    # same arithmetic except the token tile of the GEMMs (rows L vs B): rounding only
    assert torch.max(torch.abs(a[fin] - lg[fin])).item() < BF16_SMALL["delta"]
    dec.close()


def test_errors_are_reported_not_raised_on_device(D):
    W = [w.to(dev) for w in inputs.make_weights(SMALL_BF16, 0)]
    dec = D.Decoder(SMALL_BF16, W, max_batch=1, max_seq=128)
    ids = torch.zeros((1, 128), dtype=torch.int32, device=dev)
    mask = torch.zeros((1, 128), dtype=torch.uint8, device=dev)
    with pytest.raises(D.DinferError) as e:
        dec.block_step(ids, mask, 0.9)
    assert e.value.status == D.ESTATE
    with pytest.raises(D.DinferError) as e:
        dec.prefill_cache(ids, mask, 100, 64, 0.9)      # block outside the sequence
    assert e.value.status == D.EINVAL
    with pytest.raises(D.DinferError) as e:
        dec.generate(torch.zeros((2, 8), dtype=torch.int32, device=dev), 64, 32, 0.9)  # batch > max_batch
    assert e.value.status == D.EINVAL
    with pytest.raises(D.DinferError) as e:
        dec.generate(torch.zeros((1, 8), dtype=torch.int32, device=dev), 60, 32, 0.9)  # G % B != 0
    assert e.value.status == D.EINVAL
    # an out-of-range token id is caught on the device and reported after the call
    bad = torch.full((1, 8), SMALL_BF16.vocab + 5, dtype=torch.int32, device=dev)
    with pytest.raises(D.DinferError) as e:
        dec.generate(bad, 32, 32, 0.9)
    assert e.value.status == D.EDEVICE
    dec.close()


# ---------------------------------------------------------------------------
# small mixture-of-experts model (OLMoE-style routing) on the tensor-core path
# ---------------------------------------------------------------------------
SMALL_MOE = inputs.shrink(inputs.LLADA_MOE, n_layers=2, d_model=256, n_heads=2, vocab=2048, mask_id=2047,
                          n_experts=8, top_k=2, expert_ffn=128)


def test_small_moe_teacher_forced(D):
    W = inputs.make_weights(SMALL_MOE, 0)
    prompt = inputs.make_prompt(SMALL_MOE, 1, 64).numpy()
    st, _, _ = teacher_forced(D, SMALL_MOE, W, prompt, 64, 32, 0.9, BF16_SMALL, route_margin=0.02)
    print(st)
    assert st["max_err"] < BF16_SMALL["delta"]
    assert st["mean_err"] < BF16_SMALL["logit_mean"]
    assert st["unflagged_mismatch"] == 0


def test_small_moe_generate_invariants(D):
    W = [w.to(dev) for w in inputs.make_weights(SMALL_MOE, 0)]
    P, G, B = 40, 64, 32
    prompt = inputs.make_prompt(SMALL_MOE, 2, P, device=dev)
    dec = D.Decoder(SMALL_MOE, W, max_batch=2, max_seq=P + G)
    a, sa = dec.generate(prompt, G, B, 0.9)
    b, sb = dec.generate(prompt, G, B, 0.9)
    check_generation_invariants(a.cpu().numpy(), prompt.cpu().numpy(), G, B, SMALL_MOE.mask_id, sa)
    assert torch.equal(a, b)
    dec.close()


# 64 experts, top-2: a block's rows leave some experts unselected, so the
# count the bench turns into weight bytes is not simply layers x experts.
MANY_EXPERTS = inputs.shrink(inputs.LLADA_MOE, n_layers=2, d_model=256, n_heads=2, vocab=2048, mask_id=2047,
                             n_experts=64, top_k=2, expert_ffn=128)


def test_moe_experts_touched_matches_oracle_routing(D):
    """The device's count of (layer forward, expert) pairs with rows, against
    the oracle's routing of the same refresh; a row whose 2nd and 3rd router
    logits are within 0.02 may route differently under bf16 rounding, so each
    such row may move the count by one."""
    cfg = MANY_EXPERTS
    W = inputs.make_weights(cfg, 0)
    P, G, B = 64, 32, 32
    prompt = inputs.make_prompt(cfg, 1, P).numpy()
    x = np.full((1, P + G), cfg.mask_id)
    x[0, :P] = prompt
    mask = np.zeros((1, P + G), bool)
    mask[0, P:] = True
    m = O.Model(O.Desc.from_config(cfg), [w.float().numpy() for w in W])
    chosen, near = [], 0
    orig = O.route

    def recording(a, router, top_k):
        nonlocal near
        p, idx = orig(a, router, top_k)
        lg = np.sort(O.linear(a, router), axis=-1)[:, ::-1]
        near += int(((lg[:, top_k - 1] - lg[:, top_k]) < 0.02).sum())
        chosen.append(np.unique(idx).size)
        return p, idx

    O.route = recording
    try:
        O.refresh_step(m, x.copy(), mask.copy(), P, B, 0.9, O.Cache(m.desc, 1, P + G), commit=False)
    finally:
        O.route = orig
    expected = sum(chosen)
    assert len(chosen) == cfg.n_layers and expected < cfg.n_layers * cfg.n_experts
    dec = D.Decoder(cfg, [w.to(dev) for w in W], max_batch=1, max_seq=P + G)
    ids = torch.tensor(x, dtype=torch.int32, device=dev)
    mk = torch.tensor(mask.astype(np.uint8), device=dev)
    dec.moe_experts_touched()
    dec.prefill_cache(ids, mk, P, B, 0.9, commit=False)
    got = dec.moe_experts_touched()
    print("experts touched: gpu", got, "oracle", expected, "near-tie rows", near)
    assert abs(got - expected) <= near
    # cached iterations: between one and min(E, B * top_k) experts per layer
    for _ in range(3):
        dec.block_step(ids, mk, 2.0)
    it = dec.moe_experts_touched()
    assert 3 * cfg.n_layers <= it <= 3 * cfg.n_layers * min(cfg.n_experts, B * cfg.top_k)
    assert dec.moe_experts_touched() == 0  # the count restarted
    dec.close()
    dense = D.Decoder(SMALL_BF16, [w.to(dev) for w in inputs.make_weights(SMALL_BF16, 0)], max_batch=1, max_seq=96)
    assert dense.moe_experts_touched() == 0
    dense.close()


# ---------------------------------------------------------------------------
# full-size models (the workloads' shapes and launch configuration): properties
# that hold at any size -- the fp64 oracle cannot run 32 LLaDA-8B layers
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("workload,G", [("llada8b_b1", 128), ("lladamoe_b1", 128)])
def test_full_size_generation_invariants(D, workload, G):
    cfg, run, _ = inputs.WORKLOADS[workload]
    P, B = run.prompt_len, run.block_length
    W = inputs.make_weights(cfg, 0, device=dev)
    prompt = inputs.make_prompt(cfg, 1, P, device=dev)
    dec = D.Decoder(cfg, W, max_batch=1, max_seq=P + G)
    a, sa = dec.generate(prompt, G, B, run.threshold)
    b, sb = dec.generate(prompt, G, B, run.threshold)
    out = a.cpu().numpy()
    check_generation_invariants(out, prompt.cpu().numpy(), G, B, cfg.mask_id, sa)
    assert ((out >= 0) & (out < cfg.vocab)).all()
    # deterministic: the same generation twice (CTA-order split-K sums, fixed routing order)
    assert torch.equal(a, b) and sa["iters_per_block"] == sb["iters_per_block"]
    # every cached iteration of the block decodes finite logits with confidences in (0, 1]
    ids = torch.full((1, P + G), cfg.mask_id, dtype=torch.int32, device=dev)
    ids[:, :P] = prompt
    mask = torch.zeros((1, P + G), dtype=torch.uint8, device=dev)
    mask[:, P:] = 1
    lg = torch.empty((B, cfg.vocab), dtype=torch.float32, device=dev)
    tk = torch.empty(B, dtype=torch.int32, device=dev)
    cf = torch.empty(B, dtype=torch.float32, device=dev)
    dec.set_debug_outputs(lg, tk, cf)
    dec.prefill_cache(ids, mask, P, B, run.threshold)
    dec.block_step(ids, mask, run.threshold)
    dec.sync()
    fin = torch.isfinite(lg)
    assert fin.sum(dim=1).eq(cfg.vocab - 1).all()      # only the mask token is excluded
    assert not fin[:, cfg.mask_id].any()
    assert torch.equal(tk.long(), torch.where(fin, lg, torch.full_like(lg, -float("inf"))).argmax(dim=1))
    # confidence = 1 / sum exp(l - l_max), from the same logits
    ref = 1.0 / torch.exp(lg[fin].view(B, -1) - lg[fin].view(B, -1).max(dim=1, keepdim=True).values).sum(dim=1)
    assert torch.allclose(cf, ref, rtol=1e-4, atol=1e-6)
    assert ((cf > 0) & (cf <= 1)).all()
    dec.close()
