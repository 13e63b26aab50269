"""CPU oracle for block-wise diffusion-LLM decoding with a dual KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
shares no code with the CUDA library.

Plain numpy in float64 (matmul is the only library primitive), written to be
read against the method, not to be fast.

What it follows
---------------
* dInfer README, "Step 3: Use the model in dInfer": the generate call keeps the
  prompt, appends ``gen_length`` mask tokens and decodes them ``block_length``
  at a time left to right (``BlockWiseDiffusionLLM(...).generate``); the
  decoder is ``ThresholdParallelDecoder(0, threshold, mask_id, eos_id)``; the
  cache is ``KVCacheFactory('dual')``.
* dInfer abstract: four components -- model, diffusion iteration manager,
  decoding strategy, KV-cache manager.
* The method as a whole (block-wise denoising over a dual cache with
  threshold parallel commit): every denoising iteration is a bidirectional
  transformer forward of the block's tokens against cached prefix and suffix
  K/V that are recomputed at each block boundary; the LM head gives per
  position the top-1 token and its softmax probability (confidence); every
  masked position whose confidence exceeds the threshold is committed, else
  only the single most confident one.

Readings where the pages are silent (each listed in the design notes):
* confidence "exceeds" the threshold: strict ``conf > tau``;
* ties: lowest vocabulary index, lowest block position;
* the mask token's logit is excluded from argmax and softmax;
* decoder argument ``0`` is temperature 0 (greedy top-1, no sampling);
* the refresh forward at a block boundary is also iteration 1 of the block;
* the KV-cache family (README "Step 3": KVCacheFactory('dual') names one
  member of a family; README introduction: a vicinity refresh against cache
  staleness): each cached iteration recomputes a window of positions around
  the block -- the block (dual), the block and the suffix (prefix-only
  cache), the block and w positions each side (vicinity refresh), or all
  positions (no cache) -- and attends over the whole cached sequence;
* RMSNorm gains, no biases, untied LM head, rotate-half RoPE at absolute
  positions, attention scale 1/sqrt(head_dim), no causal mask;
* MoE: softmax over all experts, top-k by probability, weights not
  renormalised;
* eos_id (the decoder's end-of-sequence id; unused unless given): when a
  block completes and a sequence's block holds eos_id, every later position
  of that sequence is set to eos_id and unmasked (committed tokens are never
  rewritten); generation ends once no sequence has masked positions left;
* batch > 1: blocks advance in lockstep, a sequence whose block is done
  commits nothing until all are done; the fallback is per sequence.

Precision contract ("bf16" models): weights are bf16 values; every GEMM input
(normed activations, attention output, SiLU(gate)*up), the query and the
cached keys/values are rounded to bf16 (round to nearest even).  Everything
else -- residual stream, norms, softmaxes, accumulation -- is exact here
(float64).  "fp32" models round nothing.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

NEG_INF = -np.inf


# ---------------------------------------------------------------------------
# rounding
# ---------------------------------------------------------------------------
def round_bf16(x) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even), returned as float64.

    float64 -> float32 (nearest even), then keep the upper 16 bits of the
    float32 pattern with round-to-nearest-even on the dropped 16 bits.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


class Precision:
    def __init__(self, dtype: str):
        assert dtype in ("fp32", "bf16")
        self.dtype = dtype

    def r(self, x):
        """Apply the storage rounding of a GEMM input / cached tensor."""
        return round_bf16(x) if self.dtype == "bf16" else np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# model
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class Desc:
    n_layers: int
    d_model: int
    n_heads: int
    head_dim: int
    ffn: int
    vocab: int
    mask_id: int
    n_experts: int = 0
    top_k: int = 0
    expert_ffn: int = 0
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    logit_scale: float = 40.0
    dtype: str = "bf16"

    @classmethod
    def from_config(cls, cfg) -> "Desc":
        return cls(**{f.name: getattr(cfg, f.name) for f in dataclasses.fields(cls)})


class Model:
    """Weights in the library's pointer order (see the input generator).

    Each weight is kept as a float32 array of bf16-exact values (or fp32
    values) and widened to float64 where it is used.
    """

    def __init__(self, desc: Desc, weights: List[np.ndarray]):
        self.desc = desc
        self.prec = Precision(desc.dtype)
        w = [np.asarray(t, dtype=np.float32) for t in weights]
        self.embed = w[0]
        self.layers = []
        for l in range(desc.n_layers):
            b = 1 + 9 * l
            if desc.n_experts:
                keys = ["attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "router", "w13", "w2"]
            else:
                keys = ["attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down"]
            self.layers.append({k: w[b + i] for i, k in enumerate(keys)})
        self.final_norm = w[1 + 9 * desc.n_layers]
        self.lm_head = w[2 + 9 * desc.n_layers]


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def linear(x, w):
    """x [n, in] times w[out, in] transposed -> [n, out] (PyTorch Linear)."""
    return _f64(x) @ _f64(w).T


def rmsnorm(h, g, eps):
    """h / sqrt(mean(h^2) + eps) * g over the last axis."""
    h = _f64(h)
    return h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps) * _f64(g)


def silu(x):
    return x / (1.0 + np.exp(-x))


def rope(x, pos, theta):
    """Rotate-half rotary embedding of x [n, H, hd] at absolute positions pos [n].

    Frequencies theta^(-2i/hd), i < hd/2; pairs (i, i + hd/2) are rotated by
    angle pos * theta^(-2i/hd).
    """
    x = _f64(x)
    hd = x.shape[-1]
    half = hd // 2
    inv = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softmax(x, axis=-1):
    m = np.max(x, axis=axis, keepdims=True)
    e = np.exp(x - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def attention(q, k, v, rows_per_group=1024):
    """Bidirectional attention, no mask: q [nq,H,hd], k/v [nk,H,hd] -> [nq,H,hd].

    o[i, h] = sum_j softmax_j(q[i, h] . k[j, h] / sqrt(hd)) v[j, h].  Every
    query row is independent of the others; rows are taken in groups only to
    bound the memory of the [H, rows, nk] score array at long contexts.
    """
    hd = q.shape[-1]
    q, kt, vh = _f64(q), _f64(k).transpose(1, 2, 0), _f64(v).transpose(1, 0, 2)
    out = np.empty(q.shape, dtype=np.float64)
    for r0 in range(0, q.shape[0], rows_per_group):
        r1 = min(q.shape[0], r0 + rows_per_group)
        s = np.matmul(q[r0:r1].transpose(1, 0, 2), kt) / np.sqrt(hd)   # [H, rows, nk]
        p = softmax(s, axis=-1)
        out[r0:r1] = np.matmul(p, vh).transpose(1, 0, 2)
    return out


def dense_ffn(a, lw, prec):
    g = linear(a, lw["w_gate"])
    u = linear(a, lw["w_up"])
    act = prec.r(silu(g) * u)
    return linear(act, lw["w_down"])


def route(a, router, top_k):
    """Router probabilities and the chosen experts of each row.

    p = softmax(a . router^T) over all experts; the top_k experts by p,
    ties to the lower expert index.  Returns (p [n,E], idx [n,k]).
    """
    p = softmax(linear(a, router), axis=-1)
    idx = np.argsort(-p, axis=-1, kind="stable")[:, :top_k]
    return p, idx


def moe_ffn(a, lw, desc, prec):
    """Sum over each row's top-k experts of p_e * SwiGLU_e(a)."""
    fe = desc.expert_ffn
    p, idx = route(a, lw["router"], desc.top_k)
    out = np.zeros((a.shape[0], desc.d_model))
    for e in range(desc.n_experts):
        rows = np.nonzero((idx == e).any(axis=-1))[0]
        if rows.size == 0:
            continue
        w13 = lw["w13"][e]
        g = linear(a[rows], w13[:fe])
        u = linear(a[rows], w13[fe:])
        act = prec.r(silu(g) * u)
        out[rows] += p[rows, e][:, None] * linear(act, lw["w2"][e])
    return out


def layer_forward(model: Model, l: int, h, pos, K, V):
    """One transformer layer for the rows h [n,d] of ONE sequence at positions pos.

    K, V [L,H,hd] are that sequence's cache for layer l: the rows' fresh
    keys/values are written at pos, then every query attends over all L
    cached keys (the prefix, the fresh rows and the suffix) with no mask.
    """
    d = model.desc
    pr = model.prec
    lw = model.layers[l]
    n = h.shape[0]
    a = pr.r(rmsnorm(h, lw["attn_norm"], d.rms_eps))
    q = linear(a, lw["wq"]).reshape(n, d.n_heads, d.head_dim)
    k = linear(a, lw["wk"]).reshape(n, d.n_heads, d.head_dim)
    v = linear(a, lw["wv"]).reshape(n, d.n_heads, d.head_dim)
    q = pr.r(rope(q, pos, d.rope_theta))
    K[pos] = pr.r(rope(k, pos, d.rope_theta))
    V[pos] = pr.r(v)
    o = pr.r(attention(q, K, V).reshape(n, d.d_model))
    h = h + linear(o, lw["wo"])
    a = pr.r(rmsnorm(h, lw["ffn_norm"], d.rms_eps))
    if d.n_experts:
        h = h + moe_ffn(a, lw, d, pr)
    else:
        h = h + dense_ffn(a, lw, pr)
    return h


def embed(model: Model, ids):
    return _f64(model.embed[np.asarray(ids)])


def lm_head_logits(model: Model, h):
    """Scaled logits of the final hidden rows; the mask token's logit is -inf."""
    d = model.desc
    a = model.prec.r(rmsnorm(h, model.final_norm, d.rms_eps))
    logits = d.logit_scale * linear(a, model.lm_head)
    logits[:, d.mask_id] = NEG_INF
    return logits


def top1_confidence(logits):
    """Greedy token (lowest index on ties) and its softmax probability.

    conf = 1 / sum_v exp(l_v - l_max), the softmax value at the argmax.
    """
    tok = np.argmax(logits, axis=-1)
    lmax = logits[np.arange(logits.shape[0]), tok]
    conf = 1.0 / np.sum(np.exp(logits - lmax[:, None]), axis=-1)
    return tok.astype(np.int64), conf


def threshold_commit(conf, masked, tau):
    """Positions (within one sequence's block) to unmask this iteration.

    S = {i masked : conf_i > tau}; if S is empty, the single masked position
    with the highest confidence (lowest position on ties).  No masked
    position -> nothing.
    """
    masked = np.asarray(masked, dtype=bool)
    if not masked.any():
        return np.zeros_like(masked)
    sel = masked & (np.asarray(conf) > tau)
    if not sel.any():
        c = np.where(masked, conf, -np.inf)
        sel = np.zeros_like(masked)
        sel[int(np.argmax(c))] = True
    return sel


# ---------------------------------------------------------------------------
# forward passes over a batch of sequences
# ---------------------------------------------------------------------------
class Cache:
    """Dual KV cache: per layer, per sequence, keys/values of all L positions."""

    def __init__(self, desc: Desc, batch: int, seq_len: int):
        shp = (batch, seq_len, desc.n_heads, desc.head_dim)
        self.K = [np.zeros(shp) for _ in range(desc.n_layers)]
        self.V = [np.zeros(shp) for _ in range(desc.n_layers)]


def forward(model: Model, x, cache: Cache, rows: np.ndarray):
    """Forward of positions ``rows`` of every sequence of x [b, L].

    Writes those rows' K/V into ``cache`` and attends over the whole cached
    sequence.  With rows = all positions this is the full recomputation that
    refreshes the dual cache; with rows = the current block it is a cached
    denoising iteration.  Returns the final hidden rows [b, len(rows), d].
    """
    b = x.shape[0]
    hs = [embed(model, x[s, rows]) for s in range(b)]
    for l in range(model.desc.n_layers):
        for s in range(b):
            hs[s] = layer_forward(model, l, hs[s], rows, cache.K[l][s], cache.V[l][s])
    return np.stack(hs)


@dataclasses.dataclass
class StepResult:
    logits: np.ndarray      # [b, B, V]
    tok: np.ndarray         # [b, B]
    conf: np.ndarray        # [b, B]
    commit: np.ndarray      # [b, B] bool
    hidden: np.ndarray      # [b, B, d] final hidden rows


def decode_block(model: Model, hidden, x, mask, s0, B, tau, commit=True) -> StepResult:
    """LM head + top-1/confidence + threshold commit on the block rows, in place."""
    b = x.shape[0]
    logits = np.stack([lm_head_logits(model, hidden[i]) for i in range(b)])
    tok = np.zeros((b, B), dtype=np.int64)
    conf = np.zeros((b, B))
    sel = np.zeros((b, B), dtype=bool)
    for i in range(b):
        tok[i], conf[i] = top1_confidence(logits[i])
        if commit:
            sel[i] = threshold_commit(conf[i], mask[i, s0:s0 + B], tau)
            cols = s0 + np.nonzero(sel[i])[0]
            x[i, cols] = tok[i, sel[i]]
            mask[i, cols] = False
    return StepResult(logits, tok, conf, sel, hidden)


def refresh_step(model: Model, x, mask, s0, B, tau, cache: Cache, commit=True) -> StepResult:
    """Block boundary: full forward over all L positions (fills the cache), then decode the block."""
    L = x.shape[1]
    hid = forward(model, x, cache, np.arange(L))
    return decode_block(model, hid[:, s0:s0 + B], x, mask, s0, B, tau, commit)


def cached_step(model: Model, x, mask, s0, B, tau, cache: Cache, commit=True) -> StepResult:
    """One denoising iteration of the block against the dual cache."""
    hid = forward(model, x, cache, np.arange(s0, s0 + B))
    return decode_block(model, hid, x, mask, s0, B, tau, commit)


def window_step(model: Model, x, mask, s0, B, tau, cache: Cache, r0: int, r1: int, commit=True) -> StepResult:
    """A denoising iteration that recomputes the positions [r0, r1) -- the
    block and the part of the cache around it that the cache policy
    refreshes -- writing their K/V into the cache, with attention over the
    whole cached sequence; then decodes the block."""
    assert r0 <= s0 and s0 + B <= r1
    hid = forward(model, x, cache, np.arange(r0, r1))
    return decode_block(model, hid[:, s0 - r0:s0 - r0 + B], x, mask, s0, B, tau, commit)


CACHE_MODES = ("dual", "none", "prefix", "vicinity")


def recompute_window(cache_mode: str, s0: int, B: int, L: int, w: int = 0):
    """The positions a cached iteration recomputes under each KV-cache policy.

    dual: the block only (prefix and suffix K/V are cached at the block
    boundary); none: every position (no cache: full recomputation);
    prefix: the block and the suffix after it (only the prefix is cached);
    vicinity: the block and up to w positions on each side of it (the cached
    K/V nearest the block are refreshed every iteration).
    """
    if cache_mode == "dual":
        return s0, s0 + B
    if cache_mode == "none":
        return 0, L
    if cache_mode == "prefix":
        return s0, L
    if cache_mode == "vicinity":
        return max(0, s0 - w), min(L, s0 + B + w)
    raise ValueError(cache_mode)


def nocache_step(model: Model, x, mask, s0, B, tau, commit=True) -> StepResult:
    """Brute force: full recomputation of the whole sequence, then decode the block."""
    cache = Cache(model.desc, x.shape[0], x.shape[1])
    return refresh_step(model, x, mask, s0, B, tau, cache, commit)


@dataclasses.dataclass
class Iteration:
    block: int
    iteration: int          # 1-based within the block; 1 = the refresh
    x_before: np.ndarray
    mask_before: np.ndarray
    tok: np.ndarray
    conf: np.ndarray
    commit: np.ndarray
    logits: Optional[np.ndarray]


def eos_stop(x, mask, s0, B, eos_id):
    """After the block [s0, s0 + B) completed: a sequence whose block holds
    eos_id ends there -- its later positions become eos_id, unmasked."""
    for i in range(x.shape[0]):
        if (x[i, s0:s0 + B] == eos_id).any():
            x[i, s0 + B:] = eos_id
            mask[i, s0 + B:] = False


def generate(model: Model, prompt, gen_length: int, block_length: int, tau: float,
             cache_mode: str = "dual", keep_logits: bool = False, max_blocks: Optional[int] = None,
             window: int = 0, eos_id: Optional[int] = None):
    """Block-wise generation; returns (ids [b, P+G], list of Iteration records).

    Every block starts with a refresh (a forward over all positions that
    fills the cache).  Its later iterations recompute the positions that
    recompute_window gives for cache_mode ("dual": the block; "none":
    everything -- full recomputation; "prefix": the block and the suffix;
    "vicinity": the block and `window` positions on each side).  With eos_id,
    sequences end at the first completed block that holds it (eos_stop) and
    the generation ends when no sequence has masked positions left.
    """
    d = model.desc
    prompt = np.asarray(prompt, dtype=np.int64)
    b, P = prompt.shape
    G, B = gen_length, block_length
    assert G % B == 0
    L = P + G
    x = np.full((b, L), d.mask_id, dtype=np.int64)
    x[:, :P] = prompt
    mask = np.zeros((b, L), dtype=bool)
    mask[:, P:] = True
    trace: List[Iteration] = []
    nblk = G // B if max_blocks is None else min(G // B, max_blocks)
    for blk in range(nblk):
        s0 = P + blk * B
        if not mask.any():
            break  # every sequence ended (end-of-sequence)
        it = 0
        cache = Cache(d, b, L)
        while mask[:, s0:s0 + B].any():
            it += 1
            xb, mb = x.copy(), mask.copy()
            if it == 1 or cache_mode == "none":
                r = refresh_step(model, x, mask, s0, B, tau, cache)
            elif cache_mode == "dual":
                r = cached_step(model, x, mask, s0, B, tau, cache)
            else:
                r0, r1 = recompute_window(cache_mode, s0, B, L, window)
                r = window_step(model, x, mask, s0, B, tau, cache, r0, r1)
            trace.append(Iteration(blk, it, xb, mb, r.tok, r.conf, r.commit,
                                   r.logits if keep_logits else None))
        if eos_id is not None:
            eos_stop(x, mask, s0, B, eos_id)
    return x, trace


def iterations_per_block(trace: List[Iteration]) -> Dict[int, int]:
    out: Dict[int, int] = {}
    for t in trace:
        out[t.block] = max(out.get(t.block, 0), t.iteration)
    return out
