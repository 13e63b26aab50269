"""Kernel-level parity: each CUDA kernel vs the oracle's definition of its step.

Inputs are seeded (block_denoising_gb300.inputs); expected values come from
oracle/ only.  Shapes include the LLaDA-8B-shaped ones (d 4096, ffn 12288,
vocab 126464, L 1536) and ragged ones that exercise partial tiles.
"""
import numpy as np
import pytest
import torch

from block_denoising_gb300 import inputs
from oracle import dinfer_oracle as O

pytestmark = pytest.mark.gpu

dev = torch.device("cuda:0")


@pytest.fixture(scope="module")
def D():
    from block_denoising_gb300 import build, dinfer
    build.build()
    return dinfer


@pytest.fixture(scope="module")
def ws(D):
    return D.OpWorkspace()


def bf16_normal(tid, shape, std, seed=11):
    return inputs.normal_tensor(tid, shape, std, seed, device=dev)


def test_generator_cpu_and_gpu_agree_bitwise():
    a = inputs.normal_tensor(7, (1 << 20,), 0.02, 0, device="cpu")
    b = inputs.normal_tensor(7, (1 << 20,), 0.02, 0, device=dev).cpu()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    p = inputs.make_prompt(inputs.LLADA_8B, 2, 1000, device="cpu")
    q = inputs.make_prompt(inputs.LLADA_8B, 2, 1000, device=dev).cpu()
    assert torch.equal(p, q)


# ---------------------------------------------------------------------------
# GEMM (tcgen05, TMA, stream-K)
# ---------------------------------------------------------------------------
GEMM_SHAPES = [
    (64, 256, 128),        # one tile, 2 k-steps
    (50, 384, 192),        # ragged token count
    (64, 4096, 4096),      # LLaDA-8B O projection
    (64, 12288, 4096),     # LLaDA-8B QKV width
    (64, 4096, 12288),     # LLaDA-8B down projection (stream-K over long K)
    (200, 640, 320),       # token tile 256, ragged
    (1536, 1024, 512),     # refresh-like rows: several token tiles
    (512, 4096, 4096),     # batch-16 block rows (whole 128-token pair-CTA tiles)
    (700, 8192, 1024),     # whole 128-token pair-CTA tiles, ragged last token tile
    (384, 2048, 1024),     # pair-CTA tiles in stream-K order + the pair split-K fixup
    (1536, 4096, 1024),    # whole 176-token pair-CTA tiles (9 token tiles, the last 128 of 176 rows)
    (1536, 12288, 512),    # whole-tile schedule, several tiles per CTA
    (200, 24576, 256),     # whole-tile schedule, ragged token tile
]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_bf16_matches_oracle(D, ws, M, N, K):
    X = bf16_normal(1, (M, K), 1.0)
    W = bf16_normal(2, (N, K), 0.02)
    Y = D.op_gemm_bf16(X, W, ws)
    torch.cuda.synchronize()
    rows = np.arange(M) if M * N <= 4_000_000 else np.unique(np.linspace(0, M - 1, 24).astype(int))
    Xc = X.float().cpu().numpy()[rows]
    Wc = W.float().cpu().numpy()
    ref = O.linear(Xc, Wc)
    got = Y.cpu().numpy()[rows].astype(np.float64)
    # fp32 accumulation of K bf16 products: bound by K * 2^-24 * sum |x||w|
    bound = np.abs(Xc) @ np.abs(Wc).T * (K * 2.0 ** -24) + 1e-30
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))
    assert np.max(np.abs(got - ref)) < 1e-3


def test_gemm_is_deterministic(D, ws):
    X = bf16_normal(3, (64, 4096), 1.0)
    W = bf16_normal(4, (4096, 12288), 0.02)
    a = D.op_gemm_bf16(X, W, ws).clone()
    b = D.op_gemm_bf16(X, W, ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# ---------------------------------------------------------------------------
# fused LM head + online softmax
# ---------------------------------------------------------------------------
def _lm_reference(Xc, Wc, mask_id, scale):
    lg = scale * O.linear(Xc, Wc)
    lg[:, mask_id] = -np.inf
    tok, conf = O.top1_confidence(lg)
    return lg, tok, conf


@pytest.mark.parametrize("M,V,K", [(16, 1000, 256), (50, 4096, 512), (64, 126464, 4096)])
def test_lmhead_matches_oracle(D, ws, M, V, K):
    mask_id = V - 1
    X = inputs.normal_tensor(5, (M, K), 1.0, 3, device=dev)
    W = inputs.normal_tensor(6, (V, K), 0.02, 3, device=dev)
    tok, conf, logits = D.op_lmhead_bf16(X, W, mask_id, 40.0, ws, want_logits=True)
    torch.cuda.synchronize()
    ref, rtok, rconf = _lm_reference(X.float().cpu().numpy(), W.float().cpu().numpy(), mask_id, 40.0)
    lg = logits.cpu().numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(lg))
    assert np.max(np.abs(lg[fin] - ref[fin])) < 3e-2
    srt = np.sort(np.where(fin, ref, -np.inf), axis=-1)
    gap = srt[:, -1] - srt[:, -2]
    near = gap < 1e-2
    t = tok.cpu().numpy()
    assert np.all((t == rtok) | near), (t[~near] != rtok[~near]).sum()
    assert np.max(np.abs(conf.cpu().numpy() - rconf)) < 1e-2
    assert not np.any(t == mask_id)


def test_lmhead_never_picks_the_mask_token(D, ws):
    M, V, K = 8, 2048, 256
    X = inputs.normal_tensor(5, (M, K), 1.0, 4, device=dev)
    W = inputs.normal_tensor(6, (V, K), 0.02, 4, device=dev)
    W[V - 1] = X[0] * 10  # the mask row would win for row 0
    tok, conf, _ = D.op_lmhead_bf16(X, W, V - 1, 40.0, ws)
    torch.cuda.synchronize()
    assert not (tok == V - 1).any()


# ---------------------------------------------------------------------------
# attention over the dual cache
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("batch,rows,L,heads", [
    (1, 64, 1536, 32),    # LLaDA-8B block of 64 over the full cache (split keys)
    (1, 16, 96, 2),       # tiny, ragged key chunk
    (2, 100, 100, 2),     # refresh-like: every position queries, ragged query tile
    (2, 32, 1280, 4),     # batch of sequences
    (1, 300, 700, 2),     # three query tiles and five key chunks, both ragged
    (1, 64, 4160, 16),    # LLaDA-MoE block over a long cache (7 key splits)
    (1, 1536, 1536, 32),  # LLaDA-8B refresh: every position queries (rows sampled)
])
def test_attention_matches_oracle(D, ws, batch, rows, L, heads):
    d = heads * 128
    q = inputs.normal_tensor(7, (batch * rows, d), 1.0, 5, device=dev)
    k = inputs.normal_tensor(8, (batch, L, d), 1.0, 5, device=dev)
    v = inputs.normal_tensor(9, (batch, L, d), 1.0, 5, device=dev)
    o = D.op_attention_bf16(q, k, v, rows, ws)
    torch.cuda.synchronize()
    ws.check()
    # every row of small cases; at the refresh size rows spanning all query tiles
    sel = np.arange(rows) if rows * heads <= 4096 else np.unique(np.linspace(0, rows - 1, 40).astype(int))
    got = o.float().cpu().numpy().reshape(batch, rows, heads, 128)[:, sel]
    qc = q.float().cpu().numpy().reshape(batch, rows, heads, 128)[:, sel]
    kc = k.float().cpu().numpy().reshape(batch, L, heads, 128)
    vc = v.float().cpu().numpy().reshape(batch, L, heads, 128)
    for b in range(batch):
        ref = O.attention(qc[b], kc[b], vc[b])
        # bf16 output rounding (2^-9 relative) plus bf16 probabilities in P.V
        err = np.abs(got[b] - ref)
        assert np.all(err <= 4e-3 * np.abs(ref) + 4e-3), float(err.max())


@pytest.mark.parametrize("batch,rows,L,heads", [(1, 64, 1536, 4), (1, 256, 900, 2)])
def test_attention_growing_scores(D, ws, batch, rows, L, heads):
    # Key norms ramp up along the cache, so the running max of a query row keeps
    # growing from chunk to chunk (the rescaling of the accumulated output);
    # every other query row is damped, so within one warp some rows rescale and
    # their neighbours do not.
    d = heads * 128
    ramp = torch.linspace(0.25, 6.0, L, device=dev).view(1, L, 1)
    damp = torch.where(torch.arange(rows, device=dev) % 2 == 1, 0.05, 1.0).repeat(batch).view(-1, 1)
    q = (inputs.normal_tensor(7, (batch * rows, d), 1.0, 8, device=dev).float() * damp).bfloat16()
    k = (inputs.normal_tensor(8, (batch, L, d), 1.0, 8, device=dev).float() * ramp).bfloat16()
    v = inputs.normal_tensor(9, (batch, L, d), 1.0, 8, device=dev)
    o = D.op_attention_bf16(q, k, v, rows, ws)
    torch.cuda.synchronize()
    ws.check()
    got = o.float().cpu().numpy().reshape(batch, rows, heads, 128)
    qc = q.float().cpu().numpy().reshape(batch, rows, heads, 128)
    kc = k.float().cpu().numpy().reshape(batch, L, heads, 128)
    vc = v.float().cpu().numpy().reshape(batch, L, heads, 128)
    for b in range(batch):
        ref = O.attention(qc[b], kc[b], vc[b])
        err = np.abs(got[b] - ref)
        assert np.all(err <= 4e-3 * np.abs(ref) + 4e-3), float(err.max())


def test_attention_key_order_invariance(D, ws):
    # no mask: permuting the cached positions changes nothing (beyond rounding)
    batch, rows, L, heads = 1, 64, 640, 2
    d = heads * 128
    q = inputs.normal_tensor(7, (rows, d), 1.0, 6, device=dev)
    k = inputs.normal_tensor(8, (1, L, d), 1.0, 6, device=dev)
    v = inputs.normal_tensor(9, (1, L, d), 1.0, 6, device=dev)
    perm = torch.randperm(L, generator=torch.Generator().manual_seed(0)).to(dev)
    a = D.op_attention_bf16(q, k, v, rows, ws).float()
    b = D.op_attention_bf16(q, k[:, perm].contiguous(), v[:, perm].contiguous(), rows, ws).float()
    torch.cuda.synchronize()
    assert torch.max(torch.abs(a - b)).item() < 2e-2


# ---------------------------------------------------------------------------
# routed expert FFN (router + top-k + permutation + grouped GEMMs + combine)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,d,E,K,fe", [
    (64, 2048, 64, 8, 1024),   # LLaDA-MoE layer shape, one block of 64 rows
    (50, 256, 8, 2, 128),      # ragged rows
    (300, 512, 16, 4, 256),    # several token tiles per expert
])
def test_moe_ffn_matches_oracle(D, ws, M, d, E, K, fe):
    X = inputs.normal_tensor(11, (M, d), 1.0, 7, device=dev)
    router = inputs.normal_tensor(12, (E, d), 1.0 / np.sqrt(d), 7, device=dev)
    w13 = inputs.normal_tensor(13, (E, 2 * fe, d), 0.02, 7, device=dev)
    w2 = inputs.normal_tensor(14, (E, d, fe), 0.02, 7, device=dev)
    out, ids, w = D.op_moe_ffn_bf16(X, router, w13, w2, K, ws)
    torch.cuda.synchronize()
    Xc = X.float().cpu().numpy().astype(np.float64)
    lw = {"router": router.float().cpu().numpy(), "w13": w13.float().cpu().numpy(), "w2": w2.float().cpu().numpy()}
    desc = O.Desc(n_layers=1, d_model=d, n_heads=d // 128, head_dim=128, ffn=0, vocab=8, mask_id=7,
                  n_experts=E, top_k=K, expert_ffn=fe, dtype="bf16")
    ref = O.moe_ffn(Xc, lw, desc, O.Precision("bf16"))
    p, idx = O.route(Xc, lw["router"], K)
    # routing decisions: exact except rows whose k-th and (k+1)-th router logits are within 1e-4
    logits = Xc @ lw["router"].astype(np.float64).T
    srt = np.sort(logits, axis=-1)[:, ::-1]
    near = (srt[:, K - 1] - srt[:, K]) < 1e-4 if K < E else np.zeros(M, bool)
    g_ids = ids.cpu().numpy()
    same = (np.sort(g_ids, -1) == np.sort(idx, -1)).all(-1)
    assert np.all(same | near), int((~same & ~near).sum())
    np.testing.assert_allclose(w.cpu().numpy()[same], np.take_along_axis(p, g_ids.astype(np.int64), -1)[same],
                               rtol=1e-5, atol=1e-7)
    got = out.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)[same]
    # expert outputs differ only by rare bf16 roundings of SiLU(g)*u and fp32 accumulation
    assert np.all(err <= 1e-3 + 1e-2 * np.abs(ref[same])), float(err.max())
