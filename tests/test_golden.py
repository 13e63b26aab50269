"""Stored fixtures under tests/golden (no GPU).

* usage_example.json: the values the dInfer README's usage example prints
  ("Step 3: Use the model in dInfer").  The MoE workload and the defaults of
  the oracle and the library follow them.
* oracle_trajectories.json: written by tests/golden/make_oracle_golden.py
  from the CPU oracle alone.  Each trajectory is checked twice: against the
  method's rules directly (threshold commit, never re-mask, end of sequence),
  from the stored numbers and without the oracle's code; and against a fresh
  run of the oracle, so that a change to the oracle's arithmetic fails here
  until the fixture is rewritten and committed with its reason.
"""
import inspect
import json
import os
import re

import numpy as np
import pytest

from block_denoising_gb300 import inputs
from block_denoising_gb300.dinfer import Decoder
from oracle import dinfer_oracle as O
from tests.golden import make_oracle_golden as G

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# the usage example's values
# ---------------------------------------------------------------------------
def test_moe_workload_uses_the_usage_example_values():
    u = _load("usage_example.json")
    cfg, run, _ = inputs.WORKLOADS["lladamoe_b1"]
    assert cfg.is_moe and cfg.dtype == "bf16"
    assert cfg.mask_id == u["decoder"]["mask_id"]
    assert run.threshold == u["decoder"]["threshold"]
    assert run.gen_length == u["generate"]["gen_length"]
    assert run.block_length == u["generate"]["block_length"]
    # both ids are tokens of the MoE vocabulary; eos_id is one the library's
    # end-of-sequence setting accepts (inside the vocabulary, not mask_id)
    eos = u["decoder"]["eos_id"]
    assert 0 <= cfg.mask_id < cfg.vocab and 0 <= eos < cfg.vocab and eos != cfg.mask_id
    # the long-context MoE workload shares the model (and so mask_id)
    assert inputs.WORKLOADS["lladamoe_long"][0] == cfg


def test_default_cache_is_the_usage_examples_dual_cache():
    u = _load("usage_example.json")
    assert u["cache"] == "dual"
    assert inspect.signature(O.generate).parameters["cache_mode"].default == "dual"
    assert Decoder.CACHE_MODES["dual"] == 0
    with open(os.path.join(ROOT, "include", "dinfer.h")) as f:
        h = f.read()
    assert re.search(r"DINFER_CACHE_DUAL\s*=\s*0\b", h)
    assert re.search(r"DINFER_CACHE_DUAL\s+the block only \(default\)", h)


def test_decoder_first_argument_reads_as_greedy():
    # The decoder's first argument 0 is read as temperature 0: greedy top-1
    # with no sampling.  The oracle's top-1 is the plain argmax.
    u = _load("usage_example.json")
    assert u["decoder"]["first_argument"] == 0
    logits = np.array([[0.0, 2.0, 2.0, -1.0], [5.0, 1.0, 4.0, 4.5]])
    tok, conf = O.top1_confidence(logits)
    np.testing.assert_array_equal(tok, [1, 0])


# ---------------------------------------------------------------------------
# the oracle's stored trajectories
# ---------------------------------------------------------------------------
GOLD = _load("oracle_trajectories.json")["cases"]


@pytest.mark.parametrize("name", sorted(G.CASES))
def test_stored_trajectory_obeys_the_method(name):
    """Replays the stored iterations from the prompt with the method's rules
    alone: per iteration, every masked block position whose confidence
    exceeds the threshold commits its top-1 token, else the single most
    confident one (lowest position on ties); committed positions never
    change; a block runs until no position is masked; with an eos_id a
    sequence ends after the first completed block that holds it."""
    c = GOLD[name]
    cfg = G.CASES[name][0]
    b, P, Gn, B, tau = c["batch"], c["prompt_len"], c["gen_length"], c["block_length"], c["threshold"]
    eos = c["eos_id"]
    L = P + Gn
    prompt = inputs.make_prompt(cfg, b, P, seed=1).numpy()
    x = np.full((b, L), cfg.mask_id, dtype=np.int64)
    x[:, :P] = prompt
    mask = np.zeros((b, L), dtype=bool)
    mask[:, P:] = True
    its = c["iterations"]
    k = 0
    for blk in range(Gn // B):
        if not mask.any():
            break
        s0 = P + blk * B
        n = 0
        while mask[:, s0:s0 + B].any():
            it = its[k]
            k += 1
            n += 1
            assert (it["block"], it["iteration"]) == (blk, n)
            tok, conf, com = np.array(it["tok"]), np.array(it["conf"]), np.array(it["commit"], dtype=bool)
            assert np.all((conf > 0) & (conf <= 1))
            for i in range(b):
                m = mask[i, s0:s0 + B]
                if not m.any():
                    assert not com[i].any()  # a finished sequence waits for the others
                    continue
                want = m & (conf[i] > tau)
                if not want.any():
                    want = np.zeros(B, dtype=bool)
                    want[np.argmax(np.where(m, conf[i], -np.inf))] = True
                np.testing.assert_array_equal(com[i], want)
                x[i, s0:s0 + B][com[i]] = tok[i][com[i]]
                mask[i, s0:s0 + B][com[i]] = False
        if eos is not None:
            for i in range(b):
                if (x[i, s0:s0 + B] == eos).any():
                    x[i, s0 + B:] = eos
                    mask[i, s0 + B:] = False
    assert k == len(its)
    assert not mask.any() and not (x == cfg.mask_id).any()
    np.testing.assert_array_equal(x, np.array(c["ids"]))
    np.testing.assert_array_equal(x[:, :P], prompt)


@pytest.mark.parametrize("name", sorted(G.CASES))
def test_oracle_reproduces_the_stored_trajectory(name):
    c = GOLD[name]
    x, trace = G.run_case(name)
    np.testing.assert_array_equal(x, np.array(c["ids"]))
    assert len(trace) == len(c["iterations"])
    for t, s in zip(trace, c["iterations"]):
        assert (t.block, t.iteration) == (s["block"], s["iteration"])
        np.testing.assert_array_equal(t.tok, np.array(s["tok"]))
        np.testing.assert_array_equal(t.commit.astype(int), np.array(s["commit"]))
        np.testing.assert_allclose(t.conf, np.array(s["conf"]), rtol=1e-9, atol=0)


def test_fixture_covers_fallback_multi_commit_and_end_of_sequence():
    """The stored cases exercise every branch of the decoder: single-position
    fallback commits, multi-position commits, a sequence that waits while the
    other finishes its block, and an end-of-sequence stop."""
    singles = multis = waits = 0
    for c in GOLD.values():
        for it in c["iterations"]:
            for row in it["commit"]:
                s = sum(row)
                singles += s == 1
                multis += s > 1
                waits += s == 0
    assert singles and multis and waits
    v = GOLD["dense_bf16_vicinity"]
    eos = v["eos_id"]
    ended = [row for row in v["ids"] if row[-1] == eos]
    assert ended and len(ended) < v["batch"]
