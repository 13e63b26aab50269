"""Seeded synthetic inputs: model shapes, weights and prompts.

This module holds no arithmetic of the decoding method.  It only draws the
numbers that both the CUDA path and the CPU oracle consume, so that the two
sides see bit-identical weights and prompts.

Generator (one published counter-based definition, identical on CPU and GPU):

* ``lowbias32`` integer hash (C. Wellons, "Prospecting for hash functions",
  2018): ``x ^= x>>16; x *= 0x7feb352d; x ^= x>>15; x *= 0x846ca68b;
  x ^= x>>16`` on 32-bit words.  Evaluated with int64 torch ops whose
  intermediates never exceed 2**50, so CPU and CUDA agree bit for bit.
* element ``i`` of tensor ``t`` under seed ``s`` draws two words
  ``w_j = H(H((2i+j) ^ k_t))`` with ``k_t = H(H(s) ^ t)``, ``j in {0,1}``.
* normals by Box-Muller in float64:
  ``z = sqrt(-2 ln u1) * cos(2 pi u2)``, ``u1 = (w_0+1) 2^-32``,
  ``u2 = w_1 2^-32``; a weight is ``bf16(fp32(z * std))`` (round to nearest
  even at both casts).
* prompt ids uniform over ``[0, V) \\ {mask_id}``: ``(w_0 * (V-1)) >> 32``,
  shifted up by one at and above ``mask_id``.

Shapes follow the five workloads of the dInfer setting: a tiny fp32 model,
LLaDA-8B-shaped dense (batch 1 and batch 16), LLaDA-MoE-7B-A1B-shaped
(OLMoE-style routing) and the same MoE model at long context.  Norm gains
are 1, every other matrix is N(0, 0.02) except the router, whose std is
1/sqrt(d_model) so that router logits of a unit-RMS input are about N(0, 1).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Tuple

import torch

_M32 = 0xFFFFFFFF


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    n_layers: int
    d_model: int
    n_heads: int
    head_dim: int
    ffn: int
    vocab: int
    mask_id: int
    n_experts: int = 0      # 0 => dense SwiGLU FFN
    top_k: int = 0
    expert_ffn: int = 0
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    logit_scale: float = 40.0
    dtype: str = "bf16"     # "fp32" or "bf16": storage type of weights, K/V and GEMM inputs
    weight_std: float = 0.02

    @property
    def is_moe(self) -> bool:
        return self.n_experts > 0

    @property
    def router_std(self) -> float:
        return 1.0 / math.sqrt(self.d_model)


@dataclasses.dataclass(frozen=True)
class RunConfig:
    batch: int
    prompt_len: int
    gen_length: int
    block_length: int
    threshold: float

    @property
    def seq_len(self) -> int:
        return self.prompt_len + self.gen_length


TINY = ModelConfig(n_layers=2, d_model=256, n_heads=4, head_dim=64, ffn=688,
                   vocab=4096, mask_id=4095, dtype="fp32")
LLADA_8B = ModelConfig(n_layers=32, d_model=4096, n_heads=32, head_dim=128,
                       ffn=12288, vocab=126464, mask_id=126463)
LLADA_MOE = ModelConfig(n_layers=16, d_model=2048, n_heads=16, head_dim=128,
                        ffn=0, vocab=157184, mask_id=156895, n_experts=64,
                        top_k=8, expert_ffn=1024)

# name -> (model, run, description)
WORKLOADS = {
    "tiny_fp32": (TINY, RunConfig(1, 32, 64, 16, 0.9),
                  "tiny fp32 2L d256 4x64 f688 V4096, b1 P32 G64 B16 tau0.9"),
    "llada8b_b1": (LLADA_8B, RunConfig(1, 512, 1024, 64, 0.9),
                   "LLaDA-8B-shaped dense bf16, b1 P512 G1024 B64 tau0.9"),
    "lladamoe_b1": (LLADA_MOE, RunConfig(1, 256, 1024, 64, 0.9),
                    "LLaDA-MoE-7B-A1B-shaped bf16 E64 top8, b1 P256 G1024 B64 tau0.9"),
    "llada8b_b16": (LLADA_8B, RunConfig(16, 1024, 256, 32, 0.9),
                    "LLaDA-8B-shaped dense bf16, b16 P1024 G256 B32 tau0.9"),
    "lladamoe_long": (LLADA_MOE, RunConfig(1, 8192, 512, 64, 0.85),
                      "LLaDA-MoE-shaped bf16 long context, b1 P8192 G512 B64 tau0.85"),
    # profiling / parity case: the LLaDA-8B shapes with 2 of the 32 layers
    "llada8b_b1_2layer": (dataclasses.replace(LLADA_8B, n_layers=2), RunConfig(1, 512, 1024, 64, 0.9),
                          "LLaDA-8B widths, 2 layers, b1 P512 G1024 B64 tau0.9"),
}


# --------------------------------------------------------------------------
# weight table in the C-ABI pointer order
# --------------------------------------------------------------------------
def weight_specs(cfg: ModelConfig) -> List[Tuple[str, Tuple[int, ...], str]]:
    """(name, shape, init) for every weight, in the library's pointer order.

    Order: embed [V,d]; per layer: attn_norm [d], wq [d,d], wk [d,d],
    wv [d,d], wo [d,d], ffn_norm [d], then dense w_gate [f,d], w_up [f,d],
    w_down [d,f] or MoE router [E,d], w13 [E,2fe,d] (gate rows then up rows),
    w2 [E,d,fe]; final_norm [d]; lm_head [V,d].  Matrices are row-major
    [out, in].  init is "ones", "normal" or "router".
    """
    d, hd, H = cfg.d_model, cfg.head_dim, cfg.n_heads
    assert H * hd == d
    specs = [("embed", (cfg.vocab, d), "normal")]
    for l in range(cfg.n_layers):
        p = f"layers.{l}."
        specs += [(p + "attn_norm", (d,), "ones"), (p + "wq", (d, d), "normal"),
                  (p + "wk", (d, d), "normal"), (p + "wv", (d, d), "normal"),
                  (p + "wo", (d, d), "normal"), (p + "ffn_norm", (d,), "ones")]
        if cfg.is_moe:
            E, fe = cfg.n_experts, cfg.expert_ffn
            specs += [(p + "router", (E, d), "router"),
                      (p + "w13", (E, 2 * fe, d), "normal"),
                      (p + "w2", (E, d, fe), "normal")]
        else:
            f = cfg.ffn
            specs += [(p + "w_gate", (f, d), "normal"), (p + "w_up", (f, d), "normal"),
                      (p + "w_down", (d, f), "normal")]
    specs += [("final_norm", (d,), "ones"), ("lm_head", (cfg.vocab, d), "normal")]
    return specs


def weights_per_layer(cfg: ModelConfig) -> int:
    return 9


# --------------------------------------------------------------------------
# counter-based generator
# --------------------------------------------------------------------------
def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & _M32


def _h32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    return x ^ (x >> 16)


def _h32_int(x: int) -> int:
    x &= _M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & _M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & _M32
    return x ^ (x >> 16)


def _stream_key(seed: int, tid: int) -> int:
    return _h32_int(_h32_int(seed) ^ (tid & _M32))


def _words(idx: torch.Tensor, key: int, j: int) -> torch.Tensor:
    return _h32(_h32(((2 * idx + j) & _M32) ^ key))


_CHUNK = 1 << 25


def normal_tensor(tid: int, shape, std: float, seed: int, device="cpu",
                  dtype=torch.bfloat16) -> torch.Tensor:
    """N(0, std^2) tensor of the counter-based generator (see module doc)."""
    n = 1
    for s in shape:
        n *= s
    assert n < (1 << 31), "tensor too large for the 32-bit counter"
    key = _stream_key(seed, tid)
    out = torch.empty(n, dtype=dtype, device=device)
    for a in range(0, n, _CHUNK):
        b = min(n, a + _CHUNK)
        idx = torch.arange(a, b, dtype=torch.int64, device=device)
        w0 = _words(idx, key, 0)
        w1 = _words(idx, key, 1)
        u1 = (w0.to(torch.float64) + 1.0) * (2.0 ** -32)
        u2 = w1.to(torch.float64) * (2.0 ** -32)
        z = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)
        out[a:b] = (z * std).to(torch.float32).to(dtype)
        del idx, w0, w1, u1, u2, z
    return out.view(*shape)


def make_weights(cfg: ModelConfig, seed: int = 0, device="cpu") -> List[torch.Tensor]:
    """All weights in pointer order; bf16 for bf16 models, fp32 for fp32 ones."""
    dt = torch.float32 if cfg.dtype == "fp32" else torch.bfloat16
    out = []
    for tid, (name, shape, init) in enumerate(weight_specs(cfg)):
        if init == "ones":
            out.append(torch.ones(shape, dtype=dt, device=device))
        else:
            std = cfg.router_std if init == "router" else cfg.weight_std
            out.append(normal_tensor(tid, shape, std, seed, device, dt))
    return out


def make_weight(cfg: ModelConfig, index: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """One weight of make_weights(cfg, seed) by its pointer-order index."""
    dt = torch.float32 if cfg.dtype == "fp32" else torch.bfloat16
    name, shape, init = weight_specs(cfg)[index]
    if init == "ones":
        return torch.ones(shape, dtype=dt, device=device)
    std = cfg.router_std if init == "router" else cfg.weight_std
    return normal_tensor(index, shape, std, seed, device, dt)


def make_prompt(cfg: ModelConfig, batch: int, prompt_len: int, seed: int = 1,
                device="cpu") -> torch.Tensor:
    """int32 [batch, prompt_len] ids uniform over [0, V) without mask_id."""
    n = batch * prompt_len
    key = _stream_key(seed, 0x7FFFFFFF)
    idx = torch.arange(n, dtype=torch.int64, device=device)
    w = _words(idx, key, 0)
    ids = (w * (cfg.vocab - 1)) >> 32
    ids = ids + (ids >= cfg.mask_id).to(torch.int64)
    return ids.to(torch.int32).view(batch, prompt_len)


def uniform_tensor(tid: int, shape, lo: float, hi: float, seed: int, device="cpu") -> torch.Tensor:
    """float32 uniform [lo, hi) tensor from the same generator (for kernel-level tests)."""
    n = 1
    for s in shape:
        n *= s
    key = _stream_key(seed, tid)
    idx = torch.arange(n, dtype=torch.int64, device=device)
    u = _words(idx, key, 0).to(torch.float64) * (2.0 ** -32)
    return (lo + (hi - lo) * u).to(torch.float32).view(*shape)


def shrink(cfg: ModelConfig, **kw) -> ModelConfig:
    """A copy of cfg with some fields replaced (parity cases at reduced depth/width)."""
    return dataclasses.replace(cfg, **kw)
