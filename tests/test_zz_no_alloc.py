"""The allocation-free GEMM entry point gives the same result as the regular one.

dinfer_op_gemm_bf16_noalloc serves callers that cannot allocate device
memory when they run a projection (code inside another framework's memory
pool, real-time paths, plug-ins that must not grow their footprint): its
split-K scratch is a fixed array in the library instead of a workspace.
This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_denoising_gb300 import inputs

pytestmark = pytest.mark.gpu
dev = torch.device("cuda:0")


@pytest.fixture(scope="module")
def L():
    from block_denoising_gb300 import build, dinfer
    build.build()
    lib = dinfer.lib()
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.dinfer_op_gemm_bf16_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, vp]
    lib.dinfer_op_gemm_bf16_noalloc.restype = i32
    lib.dinfer_op_gemm_bf16_noalloc_status.argtypes = [vp]
    lib.dinfer_op_gemm_bf16_noalloc_status.restype = i32
    return dinfer, lib


@pytest.mark.parametrize("M,N,K", [
    (64, 4096, 4096),    # few tiles: split over the SMs, partial tiles in the fixed scratch
    (64, 4096, 12288),   # long reduction, many CTAs per tile
    (50, 12288, 4096),   # whole tiles (no scratch use), ragged token count
])
def test_noalloc_gemm_matches_regular_entry_point_twice(L, M, N, K):
    D, lib = L
    X = inputs.normal_tensor(1, (M, K), 1.0, 21, device=dev)
    W = inputs.normal_tensor(2, (N, K), 0.02, 21, device=dev)
    ref = D.op_gemm_bf16(X, W, D.OpWorkspace())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    Xc = X.float().cpu().numpy()
    Wc = W.float().cpu().numpy()
    # the same fp32-accumulation bound the regular GEMM's parity test uses
    bound = np.abs(Xc) @ np.abs(Wc).T * (K * 2.0 ** -24) + 1e-30
    r = ref.cpu().numpy().astype(np.float64)
    for call in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        st = lib.dinfer_op_gemm_bf16_noalloc(ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                             ctypes.c_void_p(Y.data_ptr()), M, N, K, stream)
        assert st == D.OK, lib.dinfer_last_error(None)
        torch.cuda.synchronize()
        y = Y.cpu().numpy().astype(np.float64)
        assert np.isfinite(y).all(), f"call {call}: output not fully written"
        assert np.all(np.abs(y - r) <= 2 * bound), f"call {call}"
        # no pipeline wait timed out (the query also clears the word)
        assert lib.dinfer_op_gemm_bf16_noalloc_status(stream) == D.OK, lib.dinfer_last_error(None)
        if torch.cuda.get_device_properties(dev).multi_processor_count <= 152:
            # the same schedule as the workspace entry point: the same fp32 sums
            assert torch.equal(Y, ref), f"call {call}: not bitwise equal to dinfer_op_gemm_bf16"


def test_noalloc_gemm_rejects_rows_beyond_its_scratch(L):
    D, lib = L
    X = torch.zeros((65, 128), dtype=torch.bfloat16, device=dev)
    W = torch.zeros((128, 128), dtype=torch.bfloat16, device=dev)
    Y = torch.zeros((65, 128), dtype=torch.float32, device=dev)
    st = lib.dinfer_op_gemm_bf16_noalloc(ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                         ctypes.c_void_p(Y.data_ptr()), 65, 128, 128, None)
    assert st == D.EINVAL
    assert b"M <= 64" in lib.dinfer_last_error(None)
