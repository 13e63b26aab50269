"""Benchmark: generated tokens/s of block-wise dual-cache diffusion decoding.

One step = one whole generation (every block: cache refresh + cached
denoising iterations until the block is committed) of the workload, through
the library's C-ABI (dinfer_generate).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

N > 1 (torchrun): the batch-1 workload does not shard; every rank runs an
independent replica and `value` is the tokens of all ranks over the slowest
rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "generated tokens/s at batch 1 (LLaDA-8B shape)"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            j = json.load(open(p))
            hbm = j.get("hbm_gbs") or j.get("hbm_GBs")
            tf = j.get("bf16_tflops")
            tfs = j.get("bf16_tflops_sustained", tf)
            if hbm and tf:
                return float(hbm), float(tf), float(tfs), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# algorithmic work (per unit) of the hot path
# ---------------------------------------------------------------------------
def _ffn_params(cfg, experts=None):
    """FFN weights per layer: dense SwiGLU, or router + the experts the rows
    select (`experts` per layer on average, as counted on the device; all of
    them when not given)."""
    d = cfg.d_model
    if cfg.n_experts:
        e = cfg.n_experts if experts is None else experts
        return cfg.n_experts * d + e * 3 * cfg.expert_ffn * d
    return 3 * d * cfg.ffn


def _ffn_flops_per_row(cfg):
    d = cfg.d_model
    if cfg.n_experts:
        return 2 * (cfg.n_experts * d + cfg.top_k * 3 * cfg.expert_ffn * d)
    return 2 * 3 * d * cfg.ffn


def iteration_bytes(cfg, b, L, B, experts=None):
    """Bytes one cached denoising iteration must move: every weight read once
    (embedding rows aside; of the experts, those the block's rows select) plus
    the cached K/V of the L - B non-block positions, at the model's storage
    type (bf16; fp32 for the fp32 model)."""
    d, nl, V = cfg.d_model, cfg.n_layers, cfg.vocab
    w = nl * (4 * d * d + _ffn_params(cfg, experts)) + V * d
    kv = b * (L - B) * 2 * d * nl
    return (4 if cfg.dtype == "fp32" else 2) * (w + kv)


def iteration_flops(cfg, b, L, B):
    d, nl, V = cfg.d_model, cfg.n_layers, cfg.vocab
    M = b * B
    return M * (nl * (8 * d * d + _ffn_flops_per_row(cfg)) + 2 * V * d) + 4 * M * L * d * nl


def refresh_flops(cfg, b, L, B):
    d, nl, V = cfg.d_model, cfg.n_layers, cfg.vocab
    M = b * L
    return M * nl * (8 * d * d + _ffn_flops_per_row(cfg)) + 4 * b * L * L * d * nl + 2 * b * B * V * d


class ClockSampler:
    def __init__(self, path):
        self.path = path
        self.p = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        self.f = None
        try:
            self.f = open(self.path, "w")
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms",
                                       "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None
            if self.f:
                self.f.close()
        return self

    def __exit__(self, *a):
        if self.p:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()
            self.f.close()

    def summary(self, gpu_index=0):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": []}
        try:
            rows = [r.split(",") for r in open(self.path).read().strip().splitlines()]
            rows = [[c.strip() for c in r] for r in rows if len(r) >= 9 and r[0].strip() == str(gpu_index)]
            sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
            if sm:
                out["sm_mhz"] = statistics.median(sm)
            mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
            if mx:
                out["sm_max_mhz"] = max(mx)
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            seen = set()
            for r in rows:
                for i, n in enumerate(names):
                    if r[5 + i].lower().startswith("active"):
                        seen.add(n)
            out["reasons"] = sorted(seen)
            out["samples"] = len(rows)
        except Exception:
            pass
        return out


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample of the workload
# ---------------------------------------------------------------------------
def seeded_sample_weights(cfg, n_layers, W_dev=None):
    """The workload's own seeded weights for its first n_layers layers, the
    final norm and the LM head, as host arrays (copied from the device copy
    when one is given, else drawn with the same generator; on a GPU when one
    is visible, which gives the same bits as the host generator)."""
    import numpy as np
    import torch
    from block_denoising_gb300 import inputs
    nl = cfg.n_layers
    idx = list(range(1 + 9 * n_layers)) + [1 + 9 * nl, 2 + 9 * nl]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    out = []
    for i in idx:
        t = W_dev[i] if W_dev is not None else inputs.make_weight(cfg, i, 0, device=dev)
        out.append(t.float().cpu().numpy())
    return out


def tiny_sample(cfg, run, n_layers=2, max_seqs=2):
    """The oracle runs this workload's whole generation within the sample's bound."""
    return cfg.n_layers <= n_layers and run.batch <= max_seqs and run.seq_len <= 512


def oracle_sample(cfg, run, iters_per_block=None, W_host=None, n_layers=2, max_seqs=2):
    """Time the oracle on a bounded sample of the workload.

    The tiny model: the whole generation, timed.  The others: a model with the
    workload's first `n_layers` seeded layers, its final norm and LM head, at
    the workload's sequence length; for block 0 and for a middle block (earlier
    blocks filled with seeded ids, as if committed) one refresh and two cached
    iterations, forward and decode timed apart; at most `max_seqs` sequences
    of the batch (sequences are independent).  The generation time is
    extrapolated from these: forward times x (layers / n_layers), x (batch /
    sequences timed); per block one refresh and (iterations - 1) cached
    iterations, with this run's iteration counts (or, without them, one
    iteration per block: an upper bound on the oracle's tokens/s)."""
    import numpy as np
    from block_denoising_gb300 import inputs
    from oracle import dinfer_oracle as O

    b, P, G, B = run.batch, run.prompt_len, run.gen_length, run.block_length
    L = P + G
    nblk = G // B
    cores = os.cpu_count()
    try:
        import threadpoolctl
        cores = max([i.get("num_threads", 0) for i in threadpoolctl.threadpool_info()] + [1])
    except Exception:
        pass
    if tiny_sample(cfg, run, n_layers, max_seqs):
        m = O.Model(O.Desc.from_config(cfg), [w.float().numpy() for w in inputs.make_weights(cfg, 0)])
        prompt = inputs.make_prompt(cfg, b, P).numpy()
        t0 = time.perf_counter()
        O.generate(m, prompt, G, B, run.threshold)
        total = time.perf_counter() - t0
        return {"value": b * G / total, "unit": UNIT, "cores": cores, "kind": "oracle", "extrapolated": False,
                "sample": f"float64 numpy oracle: the whole generation ({total:.2f} s), batch {b}"}
    one = inputs.shrink(cfg, n_layers=n_layers)
    m = O.Model(O.Desc.from_config(one), W_host if W_host is not None else seeded_sample_weights(cfg, n_layers))
    bs = min(b, max_seqs)
    prompt = inputs.make_prompt(cfg, b, P).numpy()[:bs]
    rng_ids = inputs.make_prompt(cfg, bs, L, seed=2).numpy()  # stand-in for committed ids
    mid = nblk // 2
    t_fwd_r, t_fwd_i, t_dec = [], [], []
    for blk in sorted({0, mid}):
        s0 = P + blk * B
        x = np.full((bs, L), cfg.mask_id, dtype=np.int64)
        x[:, :P] = prompt
        x[:, P:s0] = rng_ids[:, P:s0]
        mask = np.zeros((bs, L), bool)
        mask[:, s0:] = True
        cache = O.Cache(m.desc, bs, L)
        t0 = time.perf_counter()
        hid = O.forward(m, x, cache, np.arange(L))
        t1 = time.perf_counter()
        O.decode_block(m, hid[:, s0:s0 + B], x, mask, s0, B, run.threshold)
        t2 = time.perf_counter()
        t_fwd_r.append(t1 - t0)
        t_dec.append(t2 - t1)
        for _ in range(2):
            t0 = time.perf_counter()
            hid = O.forward(m, x, cache, np.arange(s0, s0 + B))
            t1 = time.perf_counter()
            O.decode_block(m, hid, x, mask, s0, B, run.threshold)
            t2 = time.perf_counter()
            t_fwd_i.append(t1 - t0)
            t_dec.append(t2 - t1)
    scale_l = cfg.n_layers / n_layers
    scale_b = b / bs
    dec = statistics.mean(t_dec) * scale_b
    per_refresh = statistics.mean(t_fwd_r) * scale_l * scale_b + dec
    per_iter = statistics.mean(t_fwd_i) * scale_l * scale_b + dec
    if iters_per_block is None:
        total = nblk * per_refresh
        note = "every block assumed complete at its refresh (an upper bound on the oracle's tokens/s)"
    else:
        total = nblk * per_refresh + (sum(iters_per_block) - nblk) * per_iter
        note = "with the iteration counts of this run"
    timed = sum(t_fwd_r) + sum(t_fwd_i) + sum(t_dec)
    return {
        "value": b * G / total,
        "unit": UNIT,
        "cores": cores,
        "kind": "oracle",
        "extrapolated": True,
        "sample": (f"float64 numpy oracle on the seeded weights of {n_layers} of {cfg.n_layers} layers + LM head, "
                   f"{bs} of {b} sequences, L={L}: one refresh and two cached iterations of block 0 and of block "
                   f"{mid} ({timed:.1f} s timed; refresh forward {statistics.mean(t_fwd_r):.2f} s, iteration "
                   f"forward {statistics.mean(t_fwd_i):.3f} s, decode {statistics.mean(t_dec):.2f} s); extrapolated "
                   f"x{scale_l:g} layers, x{scale_b:g} sequences to {nblk} blocks, {note}"),
        "us_per_refresh": per_refresh * 1e6,
        "us_per_iteration": per_iter * 1e6,
    }


# ---------------------------------------------------------------------------
def run_reference(args):
    from block_denoising_gb300 import inputs
    cfg, run, desc = inputs.WORKLOADS[args.workload]
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    vals = []
    W = None
    for i in range(args.warmup + args.steps):
        if W is None and not tiny_sample(cfg, run):
            W = seeded_sample_weights(cfg, 2)  # drawn once, outside the timed samples
        s = oracle_sample(cfg, run, W_host=W)
        progress(f"reference sample {i + 1}: {s['value']:.4g} tokens/s")
        if i >= args.warmup:
            vals.append(s)
    v = statistics.median([s["value"] for s in vals])
    ms = 1000.0 * run.batch * run.gen_length / v
    ex = vals[-1]["extrapolated"]
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "extrapolated": ex,
        "config": {"workload": args.workload, "description": desc, "global_batch": run.batch,
                   "seq_len": run.seq_len},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": vals[-1]["cores"], "kind": "oracle",
                         "extrapolated": ex, "sample": vals[-1]["sample"]},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if ex:
        line["note"] = ("ms_per_step and value are the oracle's whole-generation time extrapolated from the timed "
                        "sample (see cpu_baseline.sample); one step times that sample")
    print(json.dumps(line), flush=True)


def max_over_ranks(values, device):
    """Each value's maximum over the ranks of the process group (with times:
    the slowest replica's); the values themselves without a group."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def replica_tokens(world, steps, batch, gen_length):
    """Generated tokens of all replicas over the timed steps: every rank runs
    the whole workload (the batch-1 path does not shard)."""
    return world * steps * batch * gen_length


def progress(msg):
    print(f"[bench {time.strftime('%H:%M:%S')}] {msg}", file=sys.stderr, flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist
    from block_denoising_gb300 import build, dinfer, inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    cfg, run, desc = inputs.WORKLOADS[args.workload]
    b, P, G, B = run.batch, run.prompt_len, run.gen_length, run.block_length
    L = P + G
    W = inputs.make_weights(cfg, 0, device="cuda")
    stream = torch.cuda.Stream()
    dec = dinfer.Decoder(cfg, W, max_batch=b, max_seq=L, stream=stream)
    prompt_d = inputs.make_prompt(cfg, b, P, device="cuda")
    out_d = torch.empty((b, L), dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    # ---- dominant kernel: the refresh GEMMs (tensor-bound), timed alone before
    # the long generation loops (the burst regime of the measured bf16 peak) ----
    hbm, tf_burst, tf_sus, peak_src = load_peaks()
    dom = gemm_roofline(cfg, run, dinfer, stream, tf_burst)
    # warm-up (also captures and instantiates the graphs)
    progress(f"{args.workload}: weights and context ready; warm-up")
    for i in range(args.warmup):
        dec.generate(prompt_d, G, B, run.threshold, out=out_d)
        progress(f"warm-up generation {i + 1} done")
    # ---- device-timed region: inputs resident in HBM -------------------------
    # the 15 GB of weights streamed every iteration exceed the 129 MB L2, so no
    # flush is needed between steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(args.clock_log.replace("{rank}", str(rank)) if args.clock_log else
                          os.path.join(tempfile.gettempdir(), f"dinfer_clocks_rank{rank}.csv"))
    iters = []
    with clocks:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            _, st = dec.generate(prompt_d, G, B, run.threshold, out=out_d)
            iters.append(st["iters_per_block"])
        ev1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    t_dev = ev0.elapsed_time(ev1) / 1000.0
    progress(f"timed generations done ({t_dev:.3f} s)")
    # ---- end to end: host prompt in, host ids out, through the public API ----
    prompt_h = inputs.make_prompt(cfg, b, P).pin_memory()
    out_h = torch.empty((b, L), dtype=torch.int32).pin_memory()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        dec.generate(prompt_h, G, B, run.threshold, out=out_h)
    t_e2e = time.perf_counter() - t0
    # ---- the cached iteration alone (its HBM roofline) and the refresh --------
    ids = out_d.clone()
    ids[:, P:] = cfg.mask_id
    mask = torch.zeros((b, L), dtype=torch.uint8, device="cuda")
    mask[:, P:] = 1
    with torch.cuda.stream(stream):
        dec.prefill_cache(ids, mask, P, B, run.threshold, commit=False)
        n_it = 20
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ids2, mask2 = ids.clone(), mask.clone()
        dec.block_step(ids2, mask2, 2.0)  # threshold above 1: one commit per step, block never empties
        dec.moe_experts_touched()  # restart the device's count of selected experts
        e0.record(stream)
        for _ in range(n_it):
            dec.block_step(ids2, mask2, 2.0)
        e1.record(stream)
        stream.synchronize()
        us_iter = 1000.0 * e0.elapsed_time(e1) / n_it
        # experts per MoE layer that the block's rows selected, on average
        experts = dec.moe_experts_touched() / (n_it * cfg.n_layers) if cfg.n_experts else None
        e0.record(stream)
        for _ in range(3):
            dec.prefill_cache(ids, mask, P, B, run.threshold, commit=False)
        e1.record(stream)
        stream.synchronize()
        us_refresh = 1000.0 * e0.elapsed_time(e1) / 3
    dec.sync()

    progress(f"iteration {us_iter:.1f} us, refresh {us_refresh:.1f} us")

    # max over ranks: the slowest replica's times
    t_dev, t_e2e = max_over_ranks([t_dev, t_e2e], "cuda")
    tokens = replica_tokens(world, args.steps, b, G)
    value = tokens / t_dev
    e2e = tokens / t_e2e
    if rank == 0:
        ipb = iters[-1]
        bytes_it = iteration_bytes(cfg, b, L, B, experts)
        ach_gbs = bytes_it / (us_iter * 1e-6) / 1e9
        it_roof_us = max(bytes_it / (hbm * 1e9), iteration_flops(cfg, b, L, B) / (tf_burst * 1e12)) * 1e6
        it_roof_us_8t = max(bytes_it / 8e12, iteration_flops(cfg, b, L, B) / (tf_burst * 1e12)) * 1e6
        rf_roof_us = refresh_flops(cfg, b, L, B) / (tf_burst * 1e12) * 1e6
        n_launch = launches_per_generation(cfg, ipb)
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            progress("CPU oracle sample")
            Wh = None if tiny_sample(cfg, run) else seeded_sample_weights(cfg, 2, W)
            cpu = oracle_sample(cfg, run, ipb, W_host=Wh)
            cpu = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "extrapolated", "sample")}
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * t_dev / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "description": desc, "global_batch": b * world,
                       "seq_len": L, "prompt_len": P, "gen_length": G, "block_length": B,
                       "threshold": run.threshold, "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2 (weights 15 GB streamed per iteration); no flush"},
            "iterations_per_block": ipb,
            "us_per_iteration": us_iter,
            "us_per_refresh": us_refresh,
            "iteration_roofline": {"bound": "hbm", "bytes": bytes_it, "achieved_gbs": ach_gbs,
                                   "experts_per_layer": experts,
                                   "roofline_us_measured_peak": it_roof_us, "roofline_us_8tbs": it_roof_us_8t,
                                   "frac_of_measured": it_roof_us / us_iter, "frac_of_8tbs": it_roof_us_8t / us_iter,
                                   "peak_source": peak_src},
            "refresh_roofline": {"bound": "tensor", "flops": refresh_flops(cfg, b, L, B), "roofline_us": rf_roof_us,
                                 "frac": rf_roof_us / us_refresh},
            "tokens_per_s_roofline": b * G / ((G // B) * rf_roof_us * 1e-6 + (sum(ipb) - G // B) * it_roof_us * 1e-6),
            "roofline": dom,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e, "unit": UNIT, "h2d_bytes_per_step": b * P * 4, "d2h_bytes_per_step": b * L * 4},
            "gpu_launches": n_launch * args.steps,
            "clocks": clocks.summary(local),
        }
        print(json.dumps(line), flush=True)
    dec.close()
    if world > 1:
        dist.destroy_process_group()


def launches_per_generation(cfg, ipb):
    """Kernels of ours launched by one generation: per forward embed + 7 per
    layer (2 norms, 4 GEMMs, attention) + final norm + LM head; per block
    begin/inner-condition/advance; one init.  MoE layers launch 11 kernels in
    a block-rows forward (QKV, attention, O, norm, router, top-k, routing
    tables, scatter, two grouped GEMMs, combine) and up to 14 in a refresh
    (split-K fixups of the QKV and router GEMMs, a two-kernel counting sort);
    they are counted as 12."""
    per_layer = 7 if not cfg.n_experts else 12
    per_fwd = 1 + per_layer * cfg.n_layers + 2
    return 1 + len(ipb) * 3 + sum(ipb) * per_fwd


def gemm_roofline(cfg, run, dinfer, stream, peak_tflops):
    """The refresh's largest GEMM (gate/up: M = b L tokens, N = 2 ffn, K = d)
    at the launch configuration the step uses, timed with CUDA events: the best
    of three windows of 10 launches, as the burst peak it is graded against was
    taken (best of 10 runs of a GEMM alone)."""
    import torch
    from block_denoising_gb300 import inputs
    if cfg.dtype == "fp32":  # the fp32 parity model runs SIMT kernels, not the tensor-core GEMM
        return {"bound": "alu", "kernel": "gemm_f32_kernel (fp32 parity model)", "achieved": None, "peak": None,
                "unit": "TFLOP/s", "frac": None, "traffic": None,
                "note": "fp32 model: a parity case, not a performance configuration"}
    M = run.batch * run.seq_len
    N, K = (2 * cfg.ffn if cfg.ffn else 3 * cfg.d_model), cfg.d_model
    X = inputs.normal_tensor(1, (M, K), 1.0, 9, device="cuda")
    Wt = inputs.normal_tensor(2, (N, K), 0.02, 9, device="cuda")
    Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = dinfer.OpWorkspace()
    with torch.cuda.stream(stream):
        for _ in range(3):
            dinfer.op_gemm_bf16(X, Wt, ws, Y)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = 10
        dt = float("inf")
        for _ in range(3):
            e0.record(stream)
            for _ in range(n):
                dinfer.op_gemm_bf16(X, Wt, ws, Y)
            e1.record(stream)
            stream.synchronize()
            dt = min(dt, e0.elapsed_time(e1) / 1000.0 / n)
    flops = 2.0 * M * N * K
    ach = flops / dt / 1e12
    rw = NCU_DRAM_BYTES.get((M, N, K))
    return {"bound": "tensor", "kernel": f"gemm_tc2_kernel<256> (pair-CTA tiles; refresh GEMM {M}x{N}x{K}, fp32 out)",
            "achieved": ach, "peak": peak_tflops, "peak_kind": "measured burst (kernel timed alone)",
            "unit": "TFLOP/s", "frac": ach / peak_tflops,
            "traffic": None if rw is None else rw[0] + rw[1], "traffic_unit": "DRAM bytes per launch (ncu)",
            "us_per_launch": dt * 1e6, "flops_per_launch": flops}


# DRAM bytes (read, write) of one launch of the dominant kernel, from
#   python bench.py --profile gemm --gemm 1536 24576 4096 &&
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none
#       --profile-from-start off -k regex:gemm_tc2 -c 1 python bench.py --profile gemm --gemm 1536 24576 4096
# on a GB300, taken with the current gemm_tc2_kernel (a change to that kernel
# removes the entry until it is captured again).
NCU_DRAM_BYTES = {
    (1536, 24576, 4096): (215467776, 119083776),
}


def run_profile(args):
    """One region for ncu (--profile-from-start off): a cached iteration, a
    refresh, or one GEMM launch, after a warm-up outside the region."""
    import torch
    from block_denoising_gb300 import build, dinfer, inputs
    build.build()
    cfg, run, _ = inputs.WORKLOADS[args.workload]
    b, P, G, B = run.batch, run.prompt_len, run.gen_length, run.block_length
    L = P + G
    if args.profile in ("lmhead", "attention", "attention_refresh"):
        # one kernel of the workload's cached iteration (or, attention_refresh,
        # of its refresh: every position a query row) through the op API
        ws = dinfer.OpWorkspace()
        rows = b * B if args.profile != "attention_refresh" else b * L
        if args.profile == "lmhead":
            X = inputs.normal_tensor(5, (rows, cfg.d_model), 1.0, 3, device="cuda")
            Wl = inputs.normal_tensor(6, (cfg.vocab, cfg.d_model), 0.02, 3, device="cuda")
            call = lambda: dinfer.op_lmhead_bf16(X, Wl, cfg.mask_id, cfg.logit_scale, ws)
        else:
            d = cfg.d_model
            q = inputs.normal_tensor(7, (rows, d), 1.0, 5, device="cuda")
            k = inputs.normal_tensor(8, (b, L, d), 1.0, 5, device="cuda")
            v = inputs.normal_tensor(9, (b, L, d), 1.0, 5, device="cuda")
            call = lambda: dinfer.op_attention_bf16(q, k, v, rows // b, ws)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        torch.cuda.profiler.start()
        call()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        ws.check()
        return
    if args.profile == "gemm":
        M, N, K = args.gemm
        X = inputs.normal_tensor(1, (M, K), 1.0, 9, device="cuda")
        Wt = inputs.normal_tensor(2, (N, K), 0.02, 9, device="cuda")
        ws = dinfer.OpWorkspace()
        Y = dinfer.op_gemm_bf16(X, Wt, ws)
        torch.cuda.synchronize()
        torch.cuda.profiler.start()
        dinfer.op_gemm_bf16(X, Wt, ws, Y)
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        return
    W = inputs.make_weights(cfg, 0, device="cuda")
    dec = dinfer.Decoder(cfg, W, max_batch=b, max_seq=L)
    ids = torch.full((b, L), cfg.mask_id, dtype=torch.int32, device="cuda")
    ids[:, :P] = inputs.make_prompt(cfg, b, P, device="cuda")
    mask = torch.zeros((b, L), dtype=torch.uint8, device="cuda")
    mask[:, P:] = 1
    dec.prefill_cache(ids, mask, P, B, run.threshold, commit=False)
    dec.block_step(ids, mask, 2.0)
    dec.sync()
    torch.cuda.profiler.start()
    if args.profile == "iteration":
        dec.block_step(ids, mask, 2.0)
    else:
        dec.prefill_cache(ids, mask, P, B, run.threshold, commit=False)
    dec.sync()
    torch.cuda.profiler.stop()
    dec.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llada8b_b1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-log", default=None,
                    help="CSV of the nvidia-smi clock samples taken during the timed region "
                         "('{rank}' is replaced by the rank; default: the temp directory)")
    ap.add_argument("--profile", choices=["iteration", "refresh", "gemm", "lmhead", "attention", "attention_refresh"],
                    default=None)
    ap.add_argument("--gemm", type=int, nargs=3, default=[64, 24576, 4096], metavar=("M", "N", "K"))
    args = ap.parse_args()
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
