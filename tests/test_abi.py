"""The C-ABI library loads and exports every symbol the headers declare (no GPU)."""
import ctypes
import os
import re

import pytest

from block_denoising_gb300 import build as B
from block_denoising_gb300 import dinfer, inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(dinfer_\w+)\s*\(", txt))
    return sorted(names)


@pytest.fixture(scope="module")
def L():
    B.build()
    return dinfer.lib()


def test_headers_declare_the_boundary():
    syms = declared_symbols()
    for s in ("dinfer_create", "dinfer_prefill_cache", "dinfer_block_step", "dinfer_generate", "dinfer_destroy"):
        assert s in syms


def test_library_exports_every_declared_symbol(L):
    missing = [s for s in declared_symbols() if not hasattr(L, s)]
    assert not missing, missing


def test_num_weights(L):
    d = dinfer.desc_from_config(inputs.LLADA_8B, 1, 1536)
    assert L.dinfer_num_weights(ctypes.byref(d)) == 1 + 9 * 32 + 2
    assert L.dinfer_num_weights(None) == -1


@pytest.mark.parametrize("field,value,needle", [
    ("d_model", 4000, "n_heads * head_dim"),
    ("mask_id", 126464, "mask_id"),
    ("head_dim", 64, "n_heads * head_dim"),
    ("dtype", 7, "dtype"),
    ("max_batch", 65, "max_batch"),
    ("n_experts", 4, "MoE"),
])
def test_create_rejects_bad_descriptions_without_touching_the_gpu(L, field, value, needle):
    d = dinfer.desc_from_config(inputs.LLADA_8B, 1, 1536)
    setattr(d, field, value)
    n = 1 + 9 * 32 + 2
    arr = (ctypes.c_void_p * n)(*([16] * n))
    h = ctypes.c_void_p()
    st = L.dinfer_create(ctypes.byref(d), arr, None, ctypes.byref(h))
    assert st == dinfer.EINVAL
    assert not h.value
    assert needle.split()[0].lower() in L.dinfer_last_error(None).decode().lower() or needle == "MoE"


def test_create_rejects_null_weight(L):
    d = dinfer.desc_from_config(inputs.TINY, 1, 96)
    n = L.dinfer_num_weights(ctypes.byref(d))
    arr = (ctypes.c_void_p * n)(*([16] * n))
    arr[3] = None
    h = ctypes.c_void_p()
    assert L.dinfer_create(ctypes.byref(d), arr, None, ctypes.byref(h)) == dinfer.EINVAL
    assert b"weight 3" in L.dinfer_last_error(None)


def test_calls_on_null_context_are_rejected(L):
    assert L.dinfer_block_step(None, None, None, 0.9, None) == dinfer.EINVAL
    assert L.dinfer_generate(None, None, 1, 1, 1, 1, 0.9, None, None) == dinfer.EINVAL
    assert L.dinfer_op_gemm_bf16(None, None, None, 1, 128, 64, None, 0, None) == dinfer.EINVAL
    n = ctypes.c_int64(7)
    assert L.dinfer_moe_experts_touched(None, ctypes.byref(n)) == dinfer.EINVAL and n.value == 7
    assert L.dinfer_sync(None) == dinfer.EINVAL


def _start(U, G, c):
    return (U * c) // G


def _owner(U, G, u):
    return ((u + 1) * G - 1) // U


@pytest.mark.parametrize("U,G", [(4, 4), (7, 3), (6144, 152), (64 * 96, 152), (999, 152), (152, 152), (153, 152)])
def test_stream_k_schedule_arithmetic(U, G):
    # the GEMM launches min(SMs, units) CTAs; CTA c owns units [U c / G, U (c+1) / G)
    G = min(G, U)
    starts = [_start(U, G, c) for c in range(G + 1)]
    assert starts[0] == 0 and starts[-1] == U
    assert all(starts[c + 1] > starts[c] for c in range(G))  # no empty CTA
    for c in range(G):
        assert _owner(U, G, starts[c]) == c
        assert _owner(U, G, starts[c + 1] - 1) == c


@pytest.mark.parametrize("tiles,KT", [(96, 64), (32, 64), (32, 192), (2, 2), (1, 64), (3, 5), (576, 64)])
def test_stream_k_contributors_per_tile_bounded(tiles, KT):
    # launcher: G = min(SMs, U / ceil(KT / 14)); every tile then has at most 16 contributors
    U = tiles * KT
    G = max(1, min(152, U // ((KT + 13) // 14)))
    for t in range(tiles):
        c_first = _owner(U, G, t * KT)
        c_last = _owner(U, G, t * KT + KT - 1)
        assert c_last - c_first + 1 <= 16
