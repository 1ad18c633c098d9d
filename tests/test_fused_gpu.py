"""bf16 inputs and the fused linear-layer epilogue, act(A W^T + bias), against the oracle
(needs a GB300).  Each case goes through the C ABI entry gemm_f16_nt_fused; the oracle adds the
bias and applies the activation to its binary64 sums, and the bound is

    |D_gpu - D_ref| <= 1e-3 * sqrt(K) + rel * |D_ref|,  rel = 2^-10 (fp16), 2^-7 (bf16)

(rel is twice the output type's half-ulp in both cases).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import blackwell_tensor_core_fp16_gb300 as g
import oracle
from blackwell_tensor_core_fp16_gb300.workloads import make_bias, make_inputs

pytestmark = pytest.mark.gpu
TDT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    g.build()
    g.load()
    yield


def run_fused(A, B, bias, dtype, act, variant=0, workspace=False):
    M, K = A.shape
    N = B.shape[0]
    Ad, Bd = A.cuda(), B.cuda()
    bd = None if bias is None else bias.cuda()
    D = torch.full((M, N), float("nan"), dtype=TDT[dtype], device="cuda")
    ws, need = None, 0
    if workspace:
        need = g.gemm_f16_workspace_bytes(M, N, K, variant)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_f16_nt_fused(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K,
                             g.DTYPES[dtype], 0 if bd is None else bd.data_ptr(),
                             g.ACTIVATIONS[act], variant, 0 if ws is None else ws.data_ptr(),
                             need, s)
    assert rc == g.OK, g.gemm_f16_last_error()
    rc, bits = g.gemm_f16_check_status(s)
    assert rc == g.OK, f"status bits 0x{bits:x}"
    return D.cpu(), need


def check(D, A, B, bias, dtype, act):
    K = A.shape[1]
    ref = oracle.epilogue(oracle.gemm_f64_dt(A, B, dtype), bias, act, dtype)
    d = D.double().numpy()
    assert np.isfinite(d).all(), "unwritten or non-finite output"
    err = np.abs(d - ref)
    tol = oracle.tolerance_dt(ref, K, dtype)
    bad = err > tol
    assert not bad.any(), f"{int(bad.sum())} out of tolerance, worst {float((err / tol).max()):.3f}"


SHAPES = [(300, 264, 200), (520, 776, 1000), (1000, 1032, 1536)]


@pytest.mark.parametrize("variant", [0, 2, 3, 4])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bf16_plain(shape, variant):
    M, N, K = shape
    A, B = make_inputs(M, N, K, seed=400 + M, dtype=torch.bfloat16)
    D, _ = run_fused(A, B, None, "bf16", "none", variant)
    check(D, A, B, None, "bf16", "none")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
@pytest.mark.parametrize("variant", [0, 3, 4])
def test_bias_and_activation(dtype, act, variant):
    M, N, K = 520, 776, 1000
    A, B = make_inputs(M, N, K, seed=500, a_dist="normal", a_scale=K ** -0.5,
                       b_dist="normal", b_scale=1.0, dtype=TDT[dtype])
    bias = make_bias(N, seed=501, dtype=TDT[dtype])
    D, _ = run_fused(A, B, bias, dtype, act, variant)
    check(D, A, B, bias, dtype, act)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_activation_without_bias_and_stream_k(dtype, act, stream_k_on):
    """No bias, and the stream-K fix-up path (the epilogue runs after the pieces are summed)."""
    M, N, K = 1000, 1032, 1536
    A, B = make_inputs(M, N, K, seed=600, a_dist="normal", a_scale=K ** -0.5,
                       b_dist="normal", b_scale=1.0, dtype=TDT[dtype])
    D, need = run_fused(A, B, None, dtype, act, 0, workspace=True)
    assert need > 0
    check(D, A, B, None, dtype, act)
    bias = make_bias(N, seed=601, dtype=TDT[dtype])
    D, _ = run_fused(A, B, bias, dtype, act, 0, workspace=True)
    check(D, A, B, bias, dtype, act)


def test_mlp_shape_bias_gelu_sampled():
    """The MLP up-projection with bias + GELU at full size, on sampled elements."""
    M, N, K = 16384, 14336, 4096
    A, B = make_inputs(M, N, K, seed=4, a_dist="normal", a_scale=1.0, b_dist="normal",
                       b_scale=1.0 / 64)
    bias = make_bias(N, seed=4, scale=0.1)
    D, _ = run_fused(A, B, bias, "f16", "gelu", 0)
    rng = np.random.default_rng(3)
    rows = rng.integers(0, M, 3000)
    cols = rng.integers(0, N, 3000)
    ref = oracle.epilogue(oracle.gemm_f64_sampled(A, B, rows, cols), bias, "gelu", "f16",
                          cols=cols)
    got = D[torch.from_numpy(rows), torch.from_numpy(cols)].double().numpy()
    tol = oracle.tolerance_dt(ref, K, "f16")
    assert (np.abs(got - ref) <= tol).all()


def test_linear_binding_and_rejections():
    A, B = make_inputs(200, 96, 64, seed=9, dtype=torch.bfloat16)
    bias = make_bias(96, seed=9, dtype=torch.bfloat16)
    D = g.linear(A.cuda(), B.cuda(), bias.cuda(), "relu")
    torch.cuda.synchronize()
    check(D.cpu(), A, B, bias, "bf16", "relu")
    s = torch.cuda.current_stream().cuda_stream
    Ad = A.cuda()
    Dd = torch.empty((200, 96), dtype=torch.bfloat16, device="cuda")
    # the single-tile cross-check variant has no fused form; unknown dtype / activation rejected
    assert g.gemm_f16_nt_fused(Ad.data_ptr(), Ad.data_ptr(), Dd.data_ptr(), 200, 96, 64, 1, 0, 1,
                               1, 0, 0, s) == g.ERR_UNSUPPORTED
    assert g.gemm_f16_nt_fused(Ad.data_ptr(), Ad.data_ptr(), Dd.data_ptr(), 200, 96, 64, 7, 0, 0,
                               0, 0, 0, s) == g.ERR_INVALID_ARG
    assert g.gemm_f16_nt_fused(Ad.data_ptr(), Ad.data_ptr(), Dd.data_ptr(), 200, 96, 64, 1, 0, 9,
                               0, 0, 0, s) == g.ERR_INVALID_ARG
