"""End-of-sequence stop on the GPU against the oracle (dInfer README "Step 3":
the decoder's eos_id).  A sequence ends at the first completed block that
holds eos_id; its later positions become eos_id; the generation stops on the
device once no sequence has masked positions left (later blocks are skipped:
no refresh, no iteration)."""
import os

import numpy as np
import pytest
import torch

from block_denoising_gb300 import inputs
from oracle import dinfer_oracle as O
from tests import parity as PT

pytestmark = pytest.mark.gpu
dev = torch.device("cuda:0")


@pytest.fixture(scope="module")
def D():
    from block_denoising_gb300 import build, dinfer
    build.build()
    return dinfer


def first_seen(x, P, B, k, avoid=()):
    for v in x[P + k * B:P + (k + 1) * B]:
        if v not in x[P:P + k * B] and v not in avoid:
            return int(v)
    return None


@pytest.fixture(scope="module")
def tiny():
    cfg, run, _ = inputs.WORKLOADS["tiny_fp32"]
    W = inputs.make_weights(cfg, 0)
    m = O.Model(O.Desc.from_config(cfg), [t.numpy() for t in W])
    return cfg, run, W, m


def eos_case(m, cfg, b, P, G, B, tau):
    """A seeded prompt whose first sequence produces, in a middle block k, an
    id seen neither earlier nor, up to block k, in the batch's other
    sequences (which then end later, or not at all)."""
    for seed in range(1, 200):
        prompt = inputs.make_prompt(cfg, b, P, seed=seed).numpy()
        x0, _ = O.generate(m, prompt, G, B, tau)
        for k in range(1, G // B - 1):
            eos = first_seen(x0[0], P, B, k, avoid=set(x0[1:, P:P + (k + 1) * B].ravel().tolist()))
            if eos is not None and eos != cfg.mask_id:
                return prompt, eos, k
    return None, None, None


@pytest.mark.parametrize("path", ["dual graph", "vicinity graph", "host loop"])
def test_tiny_fp32_eos_stop_matches_oracle(D, tiny, path):
    cfg, run, W, m = tiny
    P, G, B, tau = run.prompt_len, run.gen_length, run.block_length, run.threshold
    prompt, eos, k = eos_case(m, cfg, 1, P, G, B, tau)
    assert eos is not None, "no id first seen in a middle block"
    mode, w = ("vicinity", 8) if path == "vicinity graph" else ("dual", 0)
    x, trace = O.generate(m, prompt, G, B, tau, cache_mode=mode, window=w, eos_id=eos)
    assert (x[0, -B:] == eos).all()   # the sequence ended before its last block
    dec = D.Decoder(cfg, [t.to(dev) for t in W], max_batch=1, max_seq=P + G)
    dec.set_cache_mode(mode, w)
    dec.set_eos(eos)
    if path == "host loop":
        os.environ["DINFER_NO_GRAPH"] = "1"
    try:
        out, stats = dec.generate(torch.tensor(prompt, dtype=torch.int32, device=dev), G, B, tau)
    finally:
        os.environ.pop("DINFER_NO_GRAPH", None)
    assert np.array_equal(out.cpu().numpy(), x)
    ipb = O.iterations_per_block(trace)
    assert stats["refreshes"] == len(ipb) < G // B           # later blocks skipped
    assert stats["iters_per_block"] == [ipb.get(j, 0) for j in range(G // B)]
    assert stats["iterations"] == len(trace)
    # without eos_id the same context decodes every block
    dec.set_eos(-1)
    _, full = dec.generate(torch.tensor(prompt, dtype=torch.int32, device=dev), G, B, tau)
    assert full["refreshes"] == G // B
    dec.close()


def test_tiny_fp32_eos_stops_one_sequence_of_a_batch(D, tiny):
    cfg, run, W, m = tiny
    P, G, B, tau = run.prompt_len, run.gen_length, run.block_length, run.threshold
    prompt, eos, k = eos_case(m, cfg, 2, P, G, B, tau)
    assert eos is not None, "no id separates the two sequences"
    x, trace = O.generate(m, prompt, G, B, tau, eos_id=eos)
    dec = D.Decoder(cfg, [t.to(dev) for t in W], max_batch=2, max_seq=P + G)
    dec.set_eos(eos)
    out, stats = dec.generate(torch.tensor(prompt, dtype=torch.int32, device=dev), G, B, tau)
    dec.close()
    assert np.array_equal(out.cpu().numpy(), x)
    assert (x[0, P + (k + 1) * B:] == eos).all() and (x[1, P:P + (k + 1) * B] != eos).all()


SMALL_BF16 = inputs.shrink(inputs.LLADA_8B, n_layers=2, d_model=512, n_heads=4, ffn=1024, vocab=2048,
                           mask_id=2047)


@pytest.mark.parametrize("mode,w", [("dual", 0), ("prefix", 0)])
def test_bf16_eos_generation_checked_by_oracle(D, mode, w):
    W = inputs.make_weights(SMALL_BF16, 0)
    P, G, B, tau = 64, 128, 32, 0.9
    prompt = inputs.make_prompt(SMALL_BF16, 1, P)
    dec = D.Decoder(SMALL_BF16, [t.to(dev) for t in W], max_batch=1, max_seq=P + G)
    dec.set_cache_mode(mode, w)
    base, _ = dec.generate(prompt.to(dev), G, B, tau)
    base = base.cpu().numpy()[0]
    eos = None
    for k in range(1, G // B - 1):
        eos = first_seen(base, P, B, k)
        if eos is not None:
            break
    assert eos is not None
    dec.set_eos(eos)
    out, stats = dec.generate(prompt.to(dev), G, B, tau)
    assert stats["refreshes"] == k + 1
    m = O.Model(O.Desc.from_config(SMALL_BF16), [t.float().numpy() for t in W])
    tol_fn = lambda recs: PT.tolerance_from_floor(*PT.model_floor(m, recs, B, tau))
    x, st, recs, tol = PT.follow_gpu(D, dec, m, prompt.numpy(), G, B, tau, tol_fn, dev, cache_mode=mode, window=w,
                                     eos_id=eos)
    dec.close()
    assert np.array_equal(x, out.cpu().numpy())
    assert (x[0, P + (k + 1) * B:] == eos).all()
    PT.assert_parity(st, tol, lm_head=False)


def test_eos_id_is_validated(D):
    dec = D.Decoder(SMALL_BF16, [t.to(dev) for t in inputs.make_weights(SMALL_BF16, 0)], max_batch=1, max_seq=96)
    for bad in (SMALL_BF16.mask_id, SMALL_BF16.vocab, -2):
        with pytest.raises(D.DinferError) as e:
            dec.set_eos(bad)
        assert e.value.status == D.EINVAL
    dec.set_eos(5)
    dec.set_eos(-1)
    dec.close()
