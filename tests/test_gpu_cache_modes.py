"""The KV-cache family on the GPU against the oracle (dInfer README: the dual
cache as one member of a cache family; a vicinity refresh against cache
staleness).  Every block starts with a refresh; its cached iterations
recompute the block (dual), the block and the suffix (prefix-only), the block
and w positions each side (vicinity) or everything (no cache), through
dinfer_set_cache_mode.
"""
import numpy as np
import pytest
import torch

from block_denoising_gb300 import inputs
from oracle import dinfer_oracle as O
from tests import parity as PT

pytestmark = pytest.mark.gpu
dev = torch.device("cuda:0")
MODES = [("none", 0), ("prefix", 0), ("vicinity", 16), ("dual", 0)]

SMALL_BF16 = inputs.shrink(inputs.LLADA_8B, n_layers=2, d_model=512, n_heads=4, ffn=1024, vocab=2048,
                           mask_id=2047)
SMALL_MOE = inputs.shrink(inputs.LLADA_MOE, n_layers=2, d_model=256, n_heads=2, vocab=2048, mask_id=2047,
                          n_experts=8, top_k=2, expert_ffn=128)


@pytest.fixture(scope="module")
def D():
    from block_denoising_gb300 import build, dinfer
    build.build()
    return dinfer


@pytest.mark.parametrize("mode,w", MODES)
def test_tiny_fp32_generation_matches_oracle_in_every_cache_mode(D, mode, w):
    cfg, run, _ = inputs.WORKLOADS["tiny_fp32"]
    W = inputs.make_weights(cfg, 0)
    prompt = inputs.make_prompt(cfg, run.batch, run.prompt_len)
    dec = D.Decoder(cfg, [t.to(dev) for t in W], max_batch=1, max_seq=run.seq_len)
    dec.set_cache_mode(mode, w)
    out, stats = dec.generate(prompt.to(dev), run.gen_length, run.block_length, run.threshold)
    m = O.Model(O.Desc.from_config(cfg), [t.numpy() for t in W])
    x, trace = O.generate(m, prompt.numpy(), run.gen_length, run.block_length, run.threshold, cache_mode=mode,
                          window=w)
    assert np.array_equal(out.cpu().numpy(), x)
    ipb = O.iterations_per_block(trace)
    assert stats["iters_per_block"] == [ipb[k] for k in range(len(ipb))]
    dec.close()


def test_one_layer_every_cache_mode_equals_no_cache_on_the_gpu(D):
    # one layer: the cached K/V depend only on embeddings and positions, so
    # every policy computes the same logits (fp32 kernels sum in a fixed order)
    cfg = inputs.shrink(inputs.TINY, n_layers=1)
    W = [t.to(dev) for t in inputs.make_weights(cfg, 0)]
    prompt = inputs.make_prompt(cfg, 2, 24, device=dev)
    outs = {}
    for mode, w in MODES:
        dec = D.Decoder(cfg, W, max_batch=2, max_seq=24 + 48)
        dec.set_cache_mode(mode, w)
        outs[mode] = dec.generate(prompt, 48, 16, 0.8)[0].cpu().numpy()
        dec.close()
    for mode, _ in MODES:
        assert np.array_equal(outs[mode], outs["none"]), mode


@pytest.mark.parametrize("mode,w", MODES[:3])
@pytest.mark.parametrize("model", ["dense", "moe"])
def test_bf16_cache_modes_teacher_forced(D, mode, w, model):
    cfg = SMALL_BF16 if model == "dense" else SMALL_MOE
    W = inputs.make_weights(cfg, 0)
    b, P, G, B, tau = (2, 40, 48, 16, 0.7) if model == "dense" else (1, 64, 64, 32, 0.9)
    prompt = inputs.make_prompt(cfg, b, P).numpy()
    m = O.Model(O.Desc.from_config(cfg), [t.float().numpy() for t in W])
    if cfg.n_experts:
        with PT.RouteMargins(0.02) as rm:
            _, recs = PT.oracle_generation(m, prompt, G, B, tau, record_hidden=True, route_margins=rm,
                                           cache_mode=mode, window=w)
        rflags = PT.route_flags_for(recs, 0.02, B)
    else:
        _, recs = PT.oracle_generation(m, prompt, G, B, tau, record_hidden=True, cache_mode=mode, window=w)
        rflags = None
    assert any(r.iteration > 1 for r in recs)
    tol = PT.tolerance_from_floor(*PT.model_floor(m, recs, B, tau, rflags))
    dec = D.Decoder(cfg, [t.to(dev) for t in W], max_batch=b, max_seq=P + G)
    dec.set_cache_mode(mode, w)
    st = PT.gpu_compare(D, dec, recs, m, B, tau, tol, dev, route_flags=rflags, per_layer=True, lm_head_check=True)
    dec.close()
    print(f"\n[{model} cache {mode} w{w}] iterations {st['iterations']} logit max {st['max_err']:.4f} "
          f"(delta {tol['delta']:.4f}) flagged {st['flagged']} unflagged mismatches {st['unflagged_mismatch']}")
    PT.assert_parity(st, tol)


@pytest.mark.parametrize("mode,w", MODES[:3])
def test_bf16_cache_mode_generation_checked_by_oracle(D, mode, w):
    """dinfer_generate in a window policy (blocks enqueued from the host, each
    block's iterations in a device-side loop) ends on the generation that,
    run step by step, agrees decision by decision with the oracle."""
    W = inputs.make_weights(SMALL_BF16, 0)
    P, G, B, tau = 64, 96, 32, 0.9
    prompt = inputs.make_prompt(SMALL_BF16, 1, P)
    dec = D.Decoder(SMALL_BF16, [t.to(dev) for t in W], max_batch=1, max_seq=P + G)
    dec.set_cache_mode(mode, w)
    out, stats = dec.generate(prompt.to(dev), G, B, tau)
    out2, _ = dec.generate(prompt.to(dev), G, B, tau)
    assert torch.equal(out, out2)
    m = O.Model(O.Desc.from_config(SMALL_BF16), [t.float().numpy() for t in W])
    tol_fn = lambda recs: PT.tolerance_from_floor(*PT.model_floor(m, recs, B, tau))
    x, st, recs, tol = PT.follow_gpu(D, dec, m, prompt.numpy(), G, B, tau, tol_fn, dev, cache_mode=mode, window=w)
    dec.close()
    assert np.array_equal(x, out.cpu().numpy())
    assert len(recs) == stats["iterations"] == sum(stats["iters_per_block"])
    PT.assert_parity(st, tol, lm_head=False)


def test_cache_mode_is_validated(D):
    dec = D.Decoder(SMALL_BF16, [t.to(dev) for t in inputs.make_weights(SMALL_BF16, 0)], max_batch=1, max_seq=96)
    with pytest.raises(D.DinferError) as e:
        D._check(D.lib().dinfer_set_cache_mode(dec.h, 7, 0), dec.h)
    assert e.value.status == D.EINVAL
    with pytest.raises(D.DinferError):
        dec.set_cache_mode("vicinity", -1)
    dec.close()
