"""Writes oracle_trajectories.json: the CPU oracle's generation trajectories
on three small seeded cases.  Run from the repository root:

    python tests/golden/make_oracle_golden.py

TEST INFRASTRUCTURE.  Calls only the oracle and the seeded input generator.

The file is a regression fixture, not a pin: the oracle's pins (closed forms,
brute force, special cases) live in the oracle pin tests.  What the fixture
adds is that any change to the oracle's arithmetic changes these
trajectories, so the change shows up as a failing test until the file is
rewritten by this script and committed with the reason for the change.

Cases (dInfer README, "Step 3: Use the model in dInfer": generate(ids,
gen_length, block_length) with a ThresholdParallelDecoder(threshold, mask_id,
eos_id) over a dual KV cache; the README's introduction for the vicinity
refresh and the MoE model family):
  dense_fp32_dual      dense SwiGLU, fp32, dual cache, batch 2
  moe_bf16_dual        E 4 top-2 experts, bf16 precision contract, dual cache
  dense_bf16_vicinity  dense, bf16, vicinity refresh (w 2) and an eos_id
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from block_denoising_gb300 import inputs  # noqa: E402
from oracle import dinfer_oracle as O  # noqa: E402

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_trajectories.json")

_SMALL = dict(n_layers=2, d_model=32, n_heads=2, head_dim=16, vocab=64, mask_id=63, weight_std=0.08)

# name -> (model config, batch, prompt_len, gen_length, block_length, tau, cache_mode, window, eos_id)
CASES = {
    "dense_fp32_dual": (inputs.ModelConfig(ffn=48, dtype="fp32", **_SMALL), 2, 8, 16, 8, 0.9, "dual", 0, None),
    "moe_bf16_dual": (inputs.ModelConfig(ffn=0, n_experts=4, top_k=2, expert_ffn=16, dtype="bf16",
                                         **dict(_SMALL, weight_std=0.05)), 1, 8, 16, 8, 0.85, "dual", 0, None),
    # eos_id 6 first completes in sequence 1's second block: that sequence
    # ends there while sequence 0 decodes the third block
    "dense_bf16_vicinity": (inputs.ModelConfig(ffn=48, dtype="bf16", **_SMALL), 2, 6, 24, 8, 0.9, "vicinity", 2,
                            6),
}


def run_case(name):
    """The oracle's trajectory of one case: (final ids, iteration records, logits per iteration)."""
    cfg, b, P, G, B, tau, mode, w, eos = CASES[name]
    desc = O.Desc.from_config(cfg)
    ws = [t.float().numpy() for t in inputs.make_weights(cfg, 0)]
    model = O.Model(desc, ws)
    prompt = inputs.make_prompt(cfg, b, P, seed=1).numpy()
    x, trace = O.generate(model, prompt, G, B, tau, cache_mode=mode, window=w, eos_id=eos, keep_logits=True)
    return x, trace


def record(name):
    """JSON-ready record of one case."""
    cfg, b, P, G, B, tau, mode, w, eos = CASES[name]
    x, trace = run_case(name)
    its = []
    for t in trace:
        its.append({
            "block": int(t.block),
            "iteration": int(t.iteration),
            "tok": t.tok.astype(int).tolist(),
            "conf": [[float(v) for v in row] for row in t.conf],
            "commit": t.commit.astype(int).tolist(),
        })
    return {"batch": b, "prompt_len": P, "gen_length": G, "block_length": B, "threshold": tau,
            "cache_mode": mode, "window": w, "eos_id": eos, "ids": x.astype(int).tolist(), "iterations": its}


def margins(name):
    """Smallest |conf - tau| over masked block positions and smallest top-2
    logit gap over the trajectory: how far each decision is from flipping."""
    cfg, b, P, G, B, tau, mode, w, eos = CASES[name]
    _, trace = run_case(name)
    dtau, gap = np.inf, np.inf
    for t in trace:
        s0 = P + t.block * B
        m = t.mask_before[:, s0:s0 + B]
        if m.any():
            dtau = min(dtau, float(np.abs(t.conf[m] - tau).min()))
        top2 = np.sort(t.logits, axis=-1)[..., -2:]
        gap = min(gap, float((top2[..., 1] - top2[..., 0]).min()))
    return dtau, gap


def main():
    out = {"generated_by": "tests/golden/make_oracle_golden.py (the CPU oracle, float64)", "cases": {}}
    for name in CASES:
        dtau, gap = margins(name)
        # a decision this close to flipping could move with BLAS summation order
        assert dtau > 1e-6 and gap > 1e-6, (name, dtau, gap)
        out["cases"][name] = record(name)
        its = out["cases"][name]["iterations"]
        print(f"{name}: {len(its)} iterations, min |conf - tau| {dtau:.2e}, min top-2 gap {gap:.2e}")
    with open(PATH, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
