"""Oracle parity at the full widths and sequence lengths of every workload.

The fp64 oracle cannot run 32 LLaDA-8B layers, so each workload's model keeps
its exact widths (d_model, heads, FFN or experts, vocabulary, mask id), its
batch, prompt, block length and threshold, with one or two of its layers.
For block 0 and for a middle block (earlier generated positions filled with
seeded ids, as if committed), the oracle runs the block's refresh and two
cached iterations; every GPU iteration starts from the oracle's state
(teacher forcing, tests/parity.py) through dinfer_prefill_cache /
dinfer_block_step.  bf16 tolerances are derived on the CPU over the same
iterations; the report gives, per workload, the logit errors against that
delta and against the stated logit bound 3e-2, the flagged decisions, the
per-layer divergence of the residual stream and the teacher-forced LM head.
"""
import numpy as np
import pytest
import torch

from block_denoising_gb300 import inputs
from oracle import dinfer_oracle as O
from tests import parity as PT

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
dev = torch.device("cuda:0")

# workload -> (layers kept, middle-block start)
CASES = {
    "llada8b_b1": (2, "mid"),     # d 4096, ffn 12288, V 126464, P 512, G 1024, B 64
    "lladamoe_b1": (2, "mid"),    # d 2048, E 64 top 8, fe 1024, V 157184, mask 156895, P 256, G 1024, B 64
    "llada8b_b16": (1, "mid"),    # batch 16, P 1024, G 256, B 32
    "lladamoe_long": (1, "mid"),  # P 8192 (L 8704), G 512, B 64, tau 0.85
}
ROUTE_MARGIN = 0.02


@pytest.fixture(scope="module")
def D():
    from block_denoising_gb300 import build, dinfer
    build.build()
    return dinfer


def starts_for(cfg, run, which):
    b, P, G, B = run.batch, run.prompt_len, run.gen_length, run.block_length
    L = P + G
    prompt = inputs.make_prompt(cfg, b, P).numpy().astype(np.int64)
    filler = inputs.make_prompt(cfg, b, L, seed=2).numpy().astype(np.int64)  # stand-in for committed ids
    out = []
    for blk, tau in ((0, run.threshold), ((G // B) // 2, 1.0)):
        # block 0 at the workload's threshold; the middle block at threshold 1
        # (one commit per iteration), so that its cached iterations run even
        # where the synthetic model commits a whole block at its refresh
        s0 = P + blk * B
        x = np.full((b, L), cfg.mask_id, dtype=np.int64)
        x[:, :P] = prompt
        x[:, P:s0] = filler[:, P:s0]
        mask = np.zeros((b, L), bool)
        mask[:, s0:] = True
        out.append((blk, s0, x, mask, tau))
    return out


@pytest.mark.parametrize("workload", list(CASES))
def test_full_width_teacher_forced(D, workload):
    cfg_full, run, _ = inputs.WORKLOADS[workload]
    n_layers, which = CASES[workload]
    cfg = inputs.shrink(cfg_full, n_layers=n_layers)
    W = inputs.make_weights(cfg, 0, device=dev)
    m = O.Model(O.Desc.from_config(cfg), [w.float().cpu().numpy() for w in W])
    B, tau = run.block_length, run.threshold
    starts = starts_for(cfg, run, which)
    if cfg.n_experts:
        with PT.RouteMargins(ROUTE_MARGIN) as rm:
            recs, _ = PT.oracle_iterations(m, starts, B, tau, 3, record_hidden=True, route_margins=rm)
        rflags = PT.route_flags_for(recs, ROUTE_MARGIN, B)
    else:
        recs, _ = PT.oracle_iterations(m, starts, B, tau, 3, record_hidden=True)
        rflags = None
    tol = PT.tolerance_from_floor(*PT.model_floor(m, recs, B, tau, rflags))
    dec = D.Decoder(cfg, W, max_batch=run.batch, max_seq=run.seq_len)
    st = PT.gpu_compare(D, dec, recs, m, B, tau, tol, dev, route_flags=rflags, per_layer=True, lm_head_check=True)
    dec.close()
    rel = " ".join(f"{v:.2e}" for v in st["layer_rel"])
    print(f"\n[{workload} {n_layers}L full width] iterations {st['iterations']} logit max {st['max_err']:.4f} "
          f"mean {st['mean_err']:.5f} (delta {tol['delta']:.4f} = 2 x floor {tol['floor_max']:.4f}; 3e-2 missed "
          f"by x{st['misses_3e-2_by']:.1f}) conf(unflagged) {st['conf_err_unflagged']:.2e} (conf-sensitive {st['conf_sensitive']}) flagged {st['flagged']} "
          f"route-flagged rows {st['route_flagged_rows']} token/commit mismatches {st['tok_mismatch']}/"
          f"{st['commit_mismatch']} unflagged {st['unflagged_mismatch']} lm-head(teacher-forced) "
          f"{st['lm_head_tf_err']:.2e} ({st.get('lm_head_tf_ratio', 0):.2f} of the fp32 bound) "
          f"layer rel. divergence [{rel}]")
    PT.assert_parity(st, tol)
