"""The allocation-free entry point gemm_f16_nt_noalloc (needs a GB300).

Some callers cannot allocate device memory at the moment they need a GEMM: servers whose device
memory all belongs to their own pool, plug-ins inside a host program that owns every allocation,
and latency-bound loops that cannot take cudaMalloc's implicit synchronisation.  gemm_f16_nt_noalloc
serves them by running the stream-K schedule with its workspace in a fixed device array that the
library reserves when it is loaded.

This test calls the new entry point through the C ABI twice in a row on shapes that do use the
scratch (the second call finds the first call's leftovers in the shared array) and checks each
output against the existing entry point gemm_f16_nt_ws (same kernel, caller-provided workspace)
within the tolerance the parity tests use, |x - y| <= 1e-3 * sqrt(K) + 2^-10 * |y|.  The file is
named so that pytest collects it last.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import blackwell_tensor_core_fp16_gb300 as g
from blackwell_tensor_core_fp16_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    g.build()
    g.load()
    yield


def _within_tolerance(x: torch.Tensor, y: torch.Tensor, K: int) -> None:
    xd = x.double().cpu().numpy()
    yd = y.double().cpu().numpy()
    assert np.isfinite(xd).all(), "non-finite output"
    tol = 1e-3 * np.sqrt(K) + np.abs(yd) * 2.0 ** -10
    err = np.abs(xd - yd)
    assert (err <= tol).all(), f"max err/tol {float((err / tol).max()):.3f}"


@pytest.mark.parametrize("shape", [(1000, 1032, 1536), (700, 2000, 4000), (8192, 8192, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_noalloc_matches_workspace_entry_point(shape):
    M, N, K = shape
    A_cpu, B_cpu = make_inputs(M, N, K, seed=900 + M + N + K, a_dist="normal",
                               a_scale=K ** -0.5, b_dist="normal", b_scale=1.0)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    stream = torch.cuda.current_stream()
    need = g.gemm_f16_workspace_bytes(M, N, K, 0)
    assert need > 0, "this shape is meant to use the scratch"

    # the existing entry point, with a caller-provided workspace
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ref = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert g.gemm_f16_nt_ws(A.data_ptr(), B.data_ptr(), ref.data_ptr(), M, N, K,
                            ws.data_ptr(), need, stream.cuda_stream) == g.OK, g.gemm_f16_last_error()

    # the new entry point, two calls in a row into fresh NaN-filled outputs
    for call in range(2):
        D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        rc = g.gemm_f16_nt_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                                   stream.cuda_stream)
        assert rc == g.OK, f"call {call}: {g.gemm_f16_last_error()}"
        rc, bits = g.gemm_f16_check_status(stream.cuda_stream)
        assert rc == g.OK, f"call {call}: status bits 0x{bits:x}"
        _within_tolerance(D, ref, K)


def test_noalloc_shapes_without_scratch_and_bad_arguments():
    # a single tile needs no scratch: the entry point still computes it
    A_cpu, B_cpu = make_inputs(128, 128, 64, seed=5)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    D = torch.empty((128, 128), dtype=torch.float16, device="cuda")
    ref = torch.empty_like(D)
    s = torch.cuda.current_stream().cuda_stream
    assert g.gemm_f16_nt_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), 128, 128, 64, s) == g.OK
    assert g.gemm_f16_nt(A.data_ptr(), B.data_ptr(), ref.data_ptr(), 128, 128, 64, s) == g.OK
    torch.cuda.synchronize()
    _within_tolerance(D, ref, 64)
    # argument checks are the same as gemm_f16_nt's
    assert g.gemm_f16_nt_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), 128, 128, 60, s) == \
        g.ERR_UNSUPPORTED
    assert g.gemm_f16_nt_noalloc(0, B.data_ptr(), D.data_ptr(), 128, 128, 64, s) == \
        g.ERR_INVALID_ARG
