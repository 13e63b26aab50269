"""Thin ctypes binding of libdinfer.so (include/dinfer.h, include/dinfer_ops.h).

Argument marshalling only: every step of the decoder runs in the CUDA
library.  torch tensors provide device memory and streams.  Loading fails
loudly when the library is missing or no GPU is visible -- there is no CPU
path.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

from . import inputs as _inputs

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdinfer.so")

OK, EINVAL, ENOMEM, ECUDA, EDEVICE, ESTATE = 0, -1, -2, -3, -4, -5
FP32, BF16 = 0, 1


class ModelDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_layers", "d_model", "n_heads", "head_dim", "ffn", "vocab",
                                              "mask_id", "n_experts", "top_k", "expert_ffn")] + \
               [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("logit_scale", ctypes.c_float),
                ("dtype", ctypes.c_int32), ("max_batch", ctypes.c_int32), ("max_seq", ctypes.c_int32)]


class Stats(ctypes.Structure):
    _fields_ = [("n_blocks", ctypes.c_int32), ("iterations", ctypes.c_int32), ("refreshes", ctypes.c_int32),
                ("ms_device", ctypes.c_float), ("iters_per_block", ctypes.POINTER(ctypes.c_int32))]


class DinferError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"dinfer status {status}: {msg}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load libdinfer.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m block_denoising_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    L.dinfer_num_weights.argtypes = [ctypes.POINTER(ModelDesc)]
    L.dinfer_num_weights.restype = i32
    L.dinfer_create.argtypes = [ctypes.POINTER(ModelDesc), ctypes.POINTER(vp), vp, ctypes.POINTER(vp)]
    L.dinfer_create.restype = i32
    L.dinfer_destroy.argtypes = [vp]
    L.dinfer_destroy.restype = None
    L.dinfer_last_error.argtypes = [vp]
    L.dinfer_last_error.restype = ctypes.c_char_p
    L.dinfer_prefill_cache.argtypes = [vp, vp, vp, i32, i32, i32, i32, f32, i32, vp]
    L.dinfer_prefill_cache.restype = i32
    L.dinfer_block_step.argtypes = [vp, vp, vp, f32, vp]
    L.dinfer_block_step.restype = i32
    L.dinfer_generate.argtypes = [vp, vp, i32, i32, i32, i32, f32, vp, ctypes.POINTER(Stats)]
    L.dinfer_generate.restype = i32
    L.dinfer_set_debug_outputs.argtypes = [vp, vp, vp, vp]
    L.dinfer_set_debug_outputs.restype = i32
    L.dinfer_set_eos.argtypes = [vp, i32]
    L.dinfer_set_eos.restype = i32
    L.dinfer_set_cache_mode.argtypes = [vp, i32, i32]
    L.dinfer_set_cache_mode.restype = i32
    L.dinfer_set_debug_hidden.argtypes = [vp, vp, vp]
    L.dinfer_set_debug_hidden.restype = i32
    L.dinfer_sync.argtypes = [vp]
    L.dinfer_sync.restype = i32
    L.dinfer_moe_experts_touched.argtypes = [vp, ctypes.POINTER(ctypes.c_int64)]
    L.dinfer_moe_experts_touched.restype = i32
    L.dinfer_op_workspace_bytes.argtypes = []
    L.dinfer_op_workspace_bytes.restype = sz
    L.dinfer_op_gemm_bf16.argtypes = [vp, vp, vp, i32, i32, i32, vp, sz, vp]
    L.dinfer_op_gemm_bf16.restype = i32
    L.dinfer_op_lmhead_bf16.argtypes = [vp, vp, i32, i32, i32, i32, f32, vp, vp, vp, vp, sz, vp]
    L.dinfer_op_lmhead_bf16.restype = i32
    L.dinfer_op_attention_bf16.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, sz, vp]
    L.dinfer_op_attention_bf16.restype = i32
    L.dinfer_op_moe_ffn_bf16.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    L.dinfer_op_moe_ffn_bf16.restype = i32
    _lib = L
    return L


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(st: int, ctx=None):
    if st != OK:
        msg = lib().dinfer_last_error(ctx).decode(errors="replace")
        raise DinferError(st, msg)


def desc_from_config(cfg: _inputs.ModelConfig, max_batch: int, max_seq: int) -> ModelDesc:
    return ModelDesc(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.ffn, cfg.vocab, cfg.mask_id,
                     cfg.n_experts, cfg.top_k, cfg.expert_ffn, cfg.rms_eps, cfg.rope_theta, cfg.logit_scale,
                     FP32 if cfg.dtype == "fp32" else BF16, max_batch, max_seq)


class Decoder:
    """A dinfer context over caller-owned device weights (kept alive here)."""

    def __init__(self, cfg: _inputs.ModelConfig, weights: Sequence[torch.Tensor], max_batch: int, max_seq: int,
                 stream: Optional[torch.cuda.Stream] = None):
        L = lib()
        self.cfg = cfg
        self.desc = desc_from_config(cfg, max_batch, max_seq)
        n = L.dinfer_num_weights(ctypes.byref(self.desc))
        if n != len(weights):
            raise ValueError(f"model takes {n} weights, got {len(weights)}")
        self.weights: List[torch.Tensor] = [w.contiguous() for w in weights]
        arr = (ctypes.c_void_p * n)(*[w.data_ptr() for w in self.weights])
        # calls are ordered on this stream (default: torch's current stream)
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        h = ctypes.c_void_p()
        st = L.dinfer_create(ctypes.byref(self.desc), arr, ctypes.c_void_p(self.stream.cuda_stream), ctypes.byref(h))
        _check(st, None)
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            lib().dinfer_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill_cache(self, ids: torch.Tensor, mask: torch.Tensor, block_start: int, block_len: int,
                      threshold: float, commit: bool = True, committed: Optional[torch.Tensor] = None):
        b, L = ids.shape
        _check(lib().dinfer_prefill_cache(self.h, _ptr(ids), _ptr(mask), b, L, block_start, block_len,
                                          float(threshold), int(commit), _ptr(committed)), self.h)

    def block_step(self, ids: torch.Tensor, mask: torch.Tensor, threshold: float,
                   committed: Optional[torch.Tensor] = None):
        _check(lib().dinfer_block_step(self.h, _ptr(ids), _ptr(mask), float(threshold), _ptr(committed)), self.h)

    def generate(self, prompt: torch.Tensor, gen_length: int, block_length: int, threshold: float,
                 out: Optional[torch.Tensor] = None):
        """prompt [b, P] int32 (host or device) -> (out [b, P+G] int32, stats dict)."""
        b, P = prompt.shape
        if out is None:
            out = torch.empty((b, P + gen_length), dtype=torch.int32, device=prompt.device)
        nblk = gen_length // block_length if block_length > 0 else 0
        ipb = (ctypes.c_int32 * max(1, nblk))()
        stats = Stats(0, 0, 0, 0.0, ctypes.cast(ipb, ctypes.POINTER(ctypes.c_int32)))
        _check(lib().dinfer_generate(self.h, _ptr(prompt), b, P, gen_length, block_length, float(threshold),
                                     _ptr(out), ctypes.byref(stats)), self.h)
        return out, {"n_blocks": stats.n_blocks, "iterations": stats.iterations, "refreshes": stats.refreshes,
                     "ms_device": stats.ms_device, "iters_per_block": list(ipb)[:nblk]}

    def set_debug_outputs(self, logits=None, tok=None, conf=None):
        _check(lib().dinfer_set_debug_outputs(self.h, _ptr(logits), _ptr(tok), _ptr(conf)), self.h)

    def set_eos(self, eos_id: int = -1):
        """End-of-sequence id of generate (-1: none)."""
        _check(lib().dinfer_set_eos(self.h, int(eos_id)), self.h)

    CACHE_MODES = {"dual": 0, "none": 1, "prefix": 2, "vicinity": 3}

    def set_cache_mode(self, mode: str, window: int = 0):
        """KV-cache policy of the cached iterations: "dual", "none", "prefix" or "vicinity" (window w)."""
        _check(lib().dinfer_set_cache_mode(self.h, self.CACHE_MODES[mode], int(window)), self.h)

    def set_debug_hidden(self, hidden=None, final_in=None):
        """Per-layer residual stream [n_layers, rows, d] fp32 and LM-head input [rows, d] of the block rows."""
        _check(lib().dinfer_set_debug_hidden(self.h, _ptr(hidden), _ptr(final_in)), self.h)

    def sync(self):
        _check(lib().dinfer_sync(self.h), self.h)

    def moe_experts_touched(self):
        """(MoE layer forward, expert) pairs that received rows since the
        previous call (the count restarts); 0 for dense models."""
        n = ctypes.c_int64(0)
        _check(lib().dinfer_moe_experts_touched(self.h, ctypes.byref(n)), self.h)
        return int(n.value)


# ---------------------------------------------------------------------------
# kernel-level entry points
# ---------------------------------------------------------------------------
class OpWorkspace:
    def __init__(self, device="cuda"):
        n = lib().dinfer_op_workspace_bytes()
        self.buf = torch.zeros(n, dtype=torch.uint8, device=device)
        self.nbytes = n

    def check(self):
        """Raise if a kernel run on this workspace reported a device-side error
        (the status word of the device state at the head of the workspace)."""
        st = int(self.buf[:32].view(torch.int32)[6].item())
        if st:
            raise DinferError(EDEVICE, f"device status 0x{st:x}")


def _stream_ptr():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def op_gemm_bf16(X: torch.Tensor, W: torch.Tensor, ws: OpWorkspace, Y: Optional[torch.Tensor] = None):
    M, K = X.shape
    N = W.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    _check(lib().dinfer_op_gemm_bf16(_ptr(X), _ptr(W), _ptr(Y), M, N, K, _ptr(ws.buf), ws.nbytes, _stream_ptr()))
    return Y


def op_lmhead_bf16(X: torch.Tensor, W: torch.Tensor, mask_id: int, scale: float, ws: OpWorkspace,
                   want_logits: bool = False):
    M, K = X.shape
    V = W.shape[0]
    tok = torch.empty(M, dtype=torch.int32, device=X.device)
    conf = torch.empty(M, dtype=torch.float32, device=X.device)
    logits = torch.empty((M, V), dtype=torch.float32, device=X.device) if want_logits else None
    _check(lib().dinfer_op_lmhead_bf16(_ptr(X), _ptr(W), M, V, K, mask_id, float(scale), _ptr(tok), _ptr(conf),
                                       _ptr(logits), _ptr(ws.buf), ws.nbytes, _stream_ptr()))
    return tok, conf, logits


def op_attention_bf16(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, rows_per_seq: int, ws: OpWorkspace,
                      out: Optional[torch.Tensor] = None):
    b, L, d = k.shape
    heads = d // 128
    if out is None:
        out = torch.empty_like(q)
    _check(lib().dinfer_op_attention_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(out), b, rows_per_seq, L, heads,
                                          _ptr(ws.buf), ws.nbytes, _stream_ptr()))
    return out


def op_moe_ffn_bf16(X: torch.Tensor, router: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor, top_k: int,
                    ws: OpWorkspace):
    """Routed expert FFN output [M, d] fp32 and the routing (ids [M, k], weights [M, k])."""
    M, d = X.shape
    E, two_fe, _ = w13.shape
    out = torch.empty((M, d), dtype=torch.float32, device=X.device)
    ids = torch.empty((M, top_k), dtype=torch.int32, device=X.device)
    w = torch.empty((M, top_k), dtype=torch.float32, device=X.device)
    _check(lib().dinfer_op_moe_ffn_bf16(_ptr(X), _ptr(router), _ptr(w13), _ptr(w2), M, d, E, top_k, two_fe // 2,
                                        _ptr(out), _ptr(ids), _ptr(w), _ptr(ws.buf), ws.nbytes, _stream_ptr()))
    return out, ids, w
