"""Shared helpers of the parity tests (test infrastructure, CPU side).

Tolerance of the bf16 models, derived on the CPU alone.  The bf16 precision
contract rounds GEMM inputs, queries and cached keys/values to bf16; the
oracle accumulates everything else exactly (float64).  A correct GPU
implementation of the same contract accumulates in fp32 and, to feed its
tensor cores, also rounds the attention probabilities to bf16 before the P.V
product.  Both differences move a value across a bf16 rounding boundary now
and then, and such flips cascade through the norms and attention.  The size
of that effect -- the "floor" -- is measured by running the oracle twice on
the same state: exactly, and under `gpu_arithmetic()`, a CPU model of those
two differences (fp32 matmuls; bf16 attention probabilities, summed as
rounded for the normaliser).  The logit tolerance delta is DELTA_PER_FLOOR
times the floor's maximum, the mean bound MEAN_PER_FLOOR times its mean.
No GPU output enters the derivation.
"""
from __future__ import annotations

import contextlib

import numpy as np

from oracle import dinfer_oracle as O

DELTA_PER_FLOOR = 2.0   # logit bound = 2 x the largest CPU-model difference
MEAN_PER_FLOOR = 2.0    # mean bound = 2 x the CPU model's mean difference
FLAG_GAP, FLAG_CONF = 1e-2, 1e-2  # flag widths of the method's parity check
CONF_TOL = 1e-2                    # confidences at unflagged positions


def _linear_fp32(x, w):
    return (np.asarray(x, np.float32) @ np.asarray(w, np.float32).T).astype(np.float64)


def _attention_gpu_model(q, k, v, rows_per_group=512):
    """Attention as the GPU computes it: fp32 scores and softmax, the
    probabilities rounded to bf16 before P.V, the normaliser summed over the
    rounded values, fp32 accumulation."""
    hd = q.shape[-1]
    q32 = np.asarray(q, np.float32)
    kt = np.asarray(k, np.float32).transpose(1, 2, 0)
    vh = np.asarray(v, np.float32).transpose(1, 0, 2)
    out = np.empty(q.shape, dtype=np.float64)
    scale = np.float32(1.0 / np.sqrt(hd))
    for r0 in range(0, q.shape[0], rows_per_group):
        r1 = min(q.shape[0], r0 + rows_per_group)
        s = np.matmul(q32[r0:r1].transpose(1, 0, 2), kt) * scale
        p = np.exp(s - s.max(axis=-1, keepdims=True))
        pb = O.round_bf16(p).astype(np.float32)
        o = np.matmul(pb, vh) / pb.sum(axis=-1, keepdims=True)
        out[r0:r1] = o.transpose(1, 0, 2)
    return out


@contextlib.contextmanager
def gpu_arithmetic():
    """Run the oracle with the GPU's accumulation precision and its extra
    rounding of the attention probabilities (see the module doc)."""
    saved = O.linear, O.attention
    O.linear, O.attention = _linear_fp32, _attention_gpu_model
    try:
        yield
    finally:
        O.linear, O.attention = saved


def floor_stats(exact, model):
    fin = np.isfinite(exact)
    d = np.abs(np.asarray(exact)[fin] - np.asarray(model)[fin])
    return float(d.max()), float(d.mean())


def tolerance_from_floor(fmax, fmean):
    return dict(delta=DELTA_PER_FLOOR * fmax, logit_mean=MEAN_PER_FLOOR * fmean, floor_max=fmax, floor_mean=fmean)


def conf_interval(conf, delta):
    """Confidences reachable when the top logit moves by +-delta and all others by -+delta."""
    c = np.clip(conf, 1e-300, 1.0)
    r = np.maximum(1.0 / c - 1.0, 0.0)
    e = np.exp(min(2.0 * delta, 700.0))
    return 1.0 / (1.0 + r * e), 1.0 / (1.0 + r / e)


def flags_for(logits, conf, mask_block, tau, delta):
    """Block positions whose decision a logit error of at most delta could
    flip: top-2 logit gap < max(2 delta, 1e-2); tau inside the confidence
    interval (or |conf - tau| < 1e-2); fallback (possible whenever no masked
    confidence is certainly above tau, i.e. no interval lies wholly above it):
    every masked position whose interval reaches the best one's."""
    b, B = conf.shape
    fl = np.zeros((b, B), dtype=bool)
    for i in range(b):
        srt = np.sort(logits[i], axis=-1)
        fl[i] |= (srt[:, -1] - srt[:, -2]) < max(2 * delta, FLAG_GAP)
        lo, hi = conf_interval(conf[i], delta)
        fl[i] |= ((lo <= tau) & (tau < hi)) | (np.abs(conf[i] - tau) < FLAG_CONF)
        masked = mask_block[i]
        if masked.any() and not (lo[masked] > tau).any():
            best = int(np.argmax(np.where(masked, conf[i], -np.inf)))
            fl[i] |= masked & (hi >= lo[best] - FLAG_CONF)
    return fl


# ---------------------------------------------------------------------------
# oracle trajectories and the GPU comparison (teacher forcing)
# ---------------------------------------------------------------------------
class Record:
    """One denoising iteration of the oracle: the state it started from and
    what it decided."""

    def __init__(self, block, iteration, s0, x_before, mask_before, step, hidden=None):
        self.block, self.iteration, self.s0 = block, iteration, s0
        self.x_before, self.mask_before = x_before, mask_before
        self.logits, self.tok, self.conf, self.commit = step.logits, step.tok, step.conf, step.commit
        self.hidden = hidden          # [n_layers, b, B, d] block rows after each layer (optional)
        self.final_in = None


def _forward_recording(m, x, cache, rows, s0, B, record):
    """The oracle's forward (embed, then every layer for every sequence, as
    dinfer_oracle.forward composes them), keeping the block rows after each
    layer when `record`."""
    b = x.shape[0]
    hs = [O.embed(m, x[s, rows]) for s in range(b)]
    per_layer = []
    off = s0 - int(rows[0])
    for l in range(m.desc.n_layers):
        for s in range(b):
            hs[s] = O.layer_forward(m, l, hs[s], rows, cache.K[l][s], cache.V[l][s])
        if record:
            per_layer.append(np.stack([h[off:off + B] for h in hs]))
    return np.stack(hs), (np.stack(per_layer) if record else None)


def oracle_iterations(m, starts, B, tau, n_iters, record_hidden=False, route_margins=None, cache_mode="dual",
                      window=0):
    """Run the oracle from each (block index, s0, x, mask) start: the block's
    refresh (iteration 1) and up to n_iters - 1 cached iterations, committing
    as the method does.  Returns the Records in order and the state after each
    start's iterations.  With a RouteMargins context active, each Record keeps
    its forward's router margins.  Cached iterations recompute the window
    that cache_mode gives (dinfer_oracle.recompute_window)."""
    recs, finals = [], []
    for start in starts:
        blk, s0, x0, mask0 = start[:4]
        tau_s = start[4] if len(start) > 4 else tau  # a start may carry its own threshold
        x, mask = x0.copy(), mask0.copy()
        cache = O.Cache(m.desc, x.shape[0], x.shape[1])
        for it in range(1, n_iters + 1):
            if not mask[:, s0:s0 + B].any():
                break
            xb, mb = x.copy(), mask.copy()
            L = x.shape[1]
            r0, r1 = (0, L) if it == 1 else O.recompute_window(cache_mode, s0, B, L, window)
            rows = np.arange(r0, r1)
            n0 = len(route_margins.calls) if route_margins is not None else 0
            hid, per_layer = _forward_recording(m, x, cache, rows, s0, B, record_hidden)
            st = O.decode_block(m, hid[:, s0 - r0:s0 - r0 + B], x, mask, s0, B, tau_s)
            rec = Record(blk, it, s0, xb, mb, st, per_layer)
            rec.tau = tau_s
            rec.window = (r0, r1)
            rec.margins = route_margins.calls[n0:] if route_margins is not None else None
            recs.append(rec)
        finals.append((x, mask))
    return recs, finals


def records_from_trace(trace, P, B):
    return [Record(t.block, t.iteration, P + t.block * B, t.x_before, t.mask_before,
                   type("S", (), {"logits": t.logits, "tok": t.tok, "conf": t.conf, "commit": t.commit}))
            for t in trace]


def model_floor(m, recs, B, tau, route_flags=None):
    """The CPU floor over the same iterations: the oracle under
    gpu_arithmetic() from each record's state (its own cache, filled at the
    block's refresh).  Rows flagged for a router near-tie (route_flags) are
    left out, as in the comparison: a routing flip is a flagged decision, not
    rounding."""
    fmax, fsum, n = 0.0, 0.0, 0
    cache = None
    with gpu_arithmetic():
        for ri, r in enumerate(recs):
            x, mask = r.x_before.copy(), r.mask_before.copy()
            t = getattr(r, "tau", tau)
            if r.iteration == 1:
                cache = O.Cache(m.desc, x.shape[0], x.shape[1])
                st = O.refresh_step(m, x, mask, r.s0, B, t, cache, commit=False)
            else:
                r0, r1 = getattr(r, "window", (r.s0, r.s0 + B))
                st = O.window_step(m, x, mask, r.s0, B, t, cache, r0, r1, commit=False)
            fin = np.isfinite(r.logits)
            if route_flags is not None:
                fin = fin & ~route_flags[ri][:, :, None]
            d = np.abs(st.logits[fin] - r.logits[fin])
            fmax = max(fmax, float(d.max()))
            fsum += float(d.sum())
            n += d.size
    return fmax, fsum / max(1, n)


class RouteMargins:
    """Records, while active, each router call's top-k margin (k-th minus
    (k+1)-th router logit): a block row whose margin in some layer is inside
    the bf16 noise may route to another expert on the GPU, so it is flagged
    and left out of the logit statistics."""

    def __init__(self, margin):
        self.margin = margin
        self.calls = []

    def __enter__(self):
        self.orig = O.route

        def recording(a, router, top_k):
            lg = np.sort(O.linear(a, router), axis=-1)[:, ::-1]
            self.calls.append(lg[:, top_k - 1] - lg[:, top_k])
            return self.orig(a, router, top_k)

        O.route = recording
        return self

    def __exit__(self, *a):
        O.route = self.orig


def gpu_compare(D, dec, recs, m, B, tau, tol, dev, route_flags=None, per_layer=False, lm_head_check=False):
    """Run every record's iteration on the GPU from the record's state and
    compare.  route_flags: per record a bool [b, B] of rows to flag for
    routing near-ties.  Returns the statistics."""
    import torch
    cfg = m.desc
    b = recs[0].x_before.shape[0]
    rows = b * B
    d, V = cfg.d_model, cfg.vocab
    lg = torch.empty((rows, V), dtype=torch.float32, device=dev)
    tk = torch.empty(rows, dtype=torch.int32, device=dev)
    cf = torch.empty(rows, dtype=torch.float32, device=dev)
    dec.set_debug_outputs(lg, tk, cf)
    hid = fin = None
    if per_layer or lm_head_check:
        hid = torch.empty((cfg.n_layers, rows, d), dtype=torch.float32, device=dev) if per_layer else None
        fdt = torch.float32 if cfg.dtype == "fp32" else torch.bfloat16
        fin = torch.empty((rows, d), dtype=fdt, device=dev) if lm_head_check else None
        dec.set_debug_hidden(hid, fin)
    w_lm64 = np.asarray(m.lm_head, np.float64) if lm_head_check else None
    st = dict(iterations=len(recs), max_err=0.0, sum_err=0.0, n=0, conf_err_unflagged=0.0, conf_outside=0,
              tok_mismatch=0, commit_mismatch=0, flagged=0, unflagged_mismatch=0, route_flagged_rows=0,
              conf_sensitive=0,
              lm_head_tf_err=0.0, layer_rel=[0.0] * cfg.n_layers)
    for ri, r in enumerate(recs):
        s0 = r.s0
        t = getattr(r, "tau", tau)
        ids = torch.tensor(r.x_before, dtype=torch.int32, device=dev)
        mask = torch.tensor(r.mask_before.astype(np.uint8), device=dev)
        if r.iteration == 1:
            dec.prefill_cache(ids, mask, s0, B, t, commit=True)
        else:
            dec.block_step(ids, mask, t)
        dec.sync()
        g_lg = lg.cpu().numpy().reshape(b, B, V)
        fin_ok = np.isfinite(r.logits)
        assert np.array_equal(fin_ok, np.isfinite(g_lg)), "the excluded (mask) logit differs"
        rf = np.zeros((b, B), bool) if route_flags is None else route_flags[ri]
        st["route_flagged_rows"] += int(rf.sum())
        sel = fin_ok & ~rf[:, :, None]
        e = np.abs(g_lg[sel] - r.logits[sel])
        if e.size:
            st["max_err"] = max(st["max_err"], float(e.max()))
            st["sum_err"] += float(e.sum())
            st["n"] += e.size
        g_conf = cf.cpu().numpy().reshape(b, B)
        lo, hi = conf_interval(r.conf, tol["delta"])
        st["conf_outside"] += int((((g_conf < lo - 1e-6) | (g_conf > hi + 1e-6)) & ~rf).sum())
        # confidence-sensitive: the logit bound delta alone allows a confidence
        # change beyond the 1e-2 tolerance (the interval is wider than 2e-2)
        csens = (hi - lo) > 2 * CONF_TOL
        st["conf_sensitive"] += int((csens & ~rf).sum())
        g_tok = tk.cpu().numpy().reshape(b, B)
        g_mask = mask.cpu().numpy().astype(bool)
        g_commit = r.mask_before[:, s0:s0 + B] & ~g_mask[:, s0:s0 + B]
        fl = flags_for(r.logits, r.conf, r.mask_before[:, s0:s0 + B], t, tol["delta"]) | rf
        st["flagged"] += int(fl.sum())
        cok = ~fl & ~csens
        if cok.any():
            st["conf_err_unflagged"] = max(st["conf_err_unflagged"], float(np.abs(g_conf - r.conf)[cok].max()))
        tm = g_tok != r.tok
        cm = g_commit != r.commit
        st["tok_mismatch"] += int(tm.sum())
        st["commit_mismatch"] += int(cm.sum())
        st["unflagged_mismatch"] += int(((tm | cm) & ~fl).sum())
        g_ids = ids.cpu().numpy()
        assert np.array_equal(g_ids[:, s0:s0 + B][g_commit], g_tok[g_commit]), "committed id is not the GPU token"
        st["last_ids"], st["last_mask"] = g_ids, g_mask
        if per_layer and r.hidden is not None:
            gh = hid.cpu().numpy().reshape(cfg.n_layers, b, B, d)
            for l in range(cfg.n_layers):
                ref = r.hidden[l][~rf]
                if ref.size == 0:
                    continue
                rel = float(np.abs(gh[l][~rf] - ref).max() / np.sqrt(np.mean(ref * ref)))
                st["layer_rel"][l] = max(st["layer_rel"][l], rel)
        if lm_head_check:
            xh = fin.float().cpu().numpy().astype(np.float64)
            tf = cfg.logit_scale * (xh @ w_lm64.T)
            tf[:, cfg.mask_id] = -np.inf
            # fp32 accumulation of K exact bf16 x bf16 products: |error| <= K u sum |x w|
            bound = cfg.logit_scale * d * 2.0 ** -24 * (np.abs(xh) @ np.abs(w_lm64).T) + 1e-30
            gl = g_lg.reshape(rows, V)
            ok = np.isfinite(tf)
            err = np.abs(gl[ok] - tf[ok])
            st["lm_head_tf_err"] = max(st["lm_head_tf_err"], float(err.max()))
            st["lm_head_tf_ratio"] = max(st.get("lm_head_tf_ratio", 0.0), float((err / bound[ok]).max()))
    dec.set_debug_outputs(None, None, None)
    if hid is not None or fin is not None:
        dec.set_debug_hidden(None, None)
    st["mean_err"] = st["sum_err"] / max(1, st["n"])
    st["misses_3e-2_by"] = st["max_err"] / 3e-2
    return st


def route_flags_for(recs, margin, B):
    """Per record: block rows whose router margin (min over layers) is below `margin`."""
    out = []
    for r in recs:
        calls = r.margins
        b = r.x_before.shape[0]
        mins = np.full((b, B), np.inf)
        r0 = getattr(r, "window", (0, 0))[0] if r.iteration > 1 else 0
        for li, mg in enumerate(calls):
            s = li % b
            off = r.s0 - r0  # the block rows inside the forward's rows
            mg = mg[off:off + B]
            mins[s] = np.minimum(mins[s], mg)
        out.append(mins < margin)
    return out


def assert_parity(st, tol, lm_head=True):
    assert st["max_err"] < tol["delta"], (st["max_err"], tol)
    assert st["mean_err"] < tol["logit_mean"], (st["mean_err"], tol)
    assert st["conf_outside"] == 0
    assert st["conf_err_unflagged"] < CONF_TOL
    assert st["unflagged_mismatch"] == 0
    if lm_head:  # the GPU's own final rows through the oracle's LM head: fp32 accumulation bound
        assert st["lm_head_tf_ratio"] <= 1.0, st["lm_head_tf_err"]


def oracle_generation(m, prompt, G, B, tau, max_blocks=None, **kw):
    """The oracle's block-wise generation from `prompt` (as
    dinfer_oracle.generate runs it), block by block through
    oracle_iterations, carrying the state.  Returns (ids, Records)."""
    prompt = np.asarray(prompt, dtype=np.int64)
    b, P = prompt.shape
    L = P + G
    x = np.full((b, L), m.desc.mask_id, dtype=np.int64)
    x[:, :P] = prompt
    mask = np.zeros((b, L), dtype=bool)
    mask[:, P:] = True
    recs = []
    nblk = G // B if max_blocks is None else min(G // B, max_blocks)
    for blk in range(nblk):
        r, fin = oracle_iterations(m, [(blk, P + blk * B, x, mask)], B, tau, B, **kw)
        recs += r
        x, mask = fin[0]
    return x, recs


def follow_gpu(D, dec, m, prompt, G, B, tau, tol_fn, dev, cache_mode="dual", window=0, eos_id=None):
    """Run the generation on the GPU step by step (dinfer_prefill_cache /
    dinfer_block_step) and check every decision against the oracle's at the
    GPU's own state (the oracle keeps a dual cache filled at the same states).
    tol_fn(records) gives the tolerance.  Returns (final GPU ids, statistics,
    records)."""
    prompt = np.asarray(prompt, dtype=np.int64)
    b, P = prompt.shape
    L = P + G
    x = np.full((b, L), m.desc.mask_id, dtype=np.int64)
    x[:, :P] = prompt
    mask = np.zeros((b, L), dtype=bool)
    mask[:, P:] = True
    recs, states = [], []
    # pass 1: the GPU trajectory, with the oracle's decision at each GPU state
    for blk in range(G // B):
        s0 = P + blk * B
        if not mask.any():
            break  # every sequence ended (end-of-sequence)
        cache = O.Cache(m.desc, b, L)
        it = 0
        while mask[:, s0:s0 + B].any():
            it += 1
            assert it <= B, "more than block_length iterations"
            if it == 1:
                st = O.refresh_step(m, x.copy(), mask.copy(), s0, B, tau, cache)
                win = (0, L)
            else:
                win = O.recompute_window(cache_mode, s0, B, L, window)
                st = O.window_step(m, x.copy(), mask.copy(), s0, B, tau, cache, *win)
            rec = Record(blk, it, s0, x.copy(), mask.copy(), st)
            rec.window = win
            recs.append(rec)
            one = gpu_compare(D, dec, [rec], m, B, tau, dict(delta=1e3), dev)
            x, mask = one["last_ids"].astype(np.int64), one["last_mask"].astype(bool)
        if eos_id is not None:
            O.eos_stop(x, mask, s0, B, eos_id)
    # pass 2: the comparison with the tolerance of these iterations
    tol = tol_fn(recs)
    stats = gpu_compare(D, dec, recs, m, B, tau, tol, dev)
    return x, stats, recs, tol
