"""Failure detection on the GPU without faulting it (needs a GB300).

Every wait inside the kernels is bounded.  With the testing hook gemm_f16_set_fault_injection(1)
the load producer issues nothing, so the first wait for operand data waits on a barrier that
nothing will complete; with a 200 ms limit the wait runs out, the kernel stops cleanly (no copy
or MMA is ever in flight), and the host reads GEMM_F16_ERR_TIMEOUT with the roles that gave up.
The context must stay usable: a normal GEMM right after still matches the oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import blackwell_tensor_core_fp16_gb300 as g
import oracle
from blackwell_tensor_core_fp16_gb300.workloads import make_inputs
from gdn_bounds import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def restore_settings():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    g.build()
    g.load()
    yield
    g.gemm_f16_set_fault_injection(0)
    g.gemm_f16_set_wait_timeout_ms(4000)
    torch.cuda.synchronize()
    g.gemm_f16_check_status(0)


@pytest.mark.parametrize("variant,expect_bits", [
    (g.VARIANTS["tile"], 1),         # the single-tile kernel's load wait
    (g.VARIANTS["ws_128x128"], 2),   # the MMA issuer's wait for operand data
    (g.VARIANTS["ws_pair"], 2),      # same, in a CTA pair (the other CTA's epilogue also gives up)
])
def test_wait_runs_out_and_context_survives(variant, expect_bits):
    M, N, K = 520, 776, 1000
    A, B = make_inputs(M, N, K, seed=700)
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert g.gemm_f16_set_wait_timeout_ms(200) == g.OK
    assert g.gemm_f16_set_fault_injection(1) == g.OK
    assert g.gemm_f16_nt_variant(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, s,
                                 variant) == g.OK
    rc, bits = g.gemm_f16_check_status(s)
    assert rc == g.ERR_TIMEOUT, (rc, bits)
    assert bits & expect_bits, f"bits 0x{bits:x}"
    assert "bounded wait" in g.gemm_f16_last_error()
    # the status word was cleared by the read
    assert g.gemm_f16_check_status(s) == (g.OK, 0)

    # back to normal: the same context computes correctly
    assert g.gemm_f16_set_fault_injection(0) == g.OK
    assert g.gemm_f16_set_wait_timeout_ms(4000) == g.OK
    assert g.gemm_f16_nt_variant(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, s,
                                 variant) == g.OK
    assert g.gemm_f16_check_status(s) == (g.OK, 0)
    d = D.cpu().double().numpy()
    ref = oracle.gemm_f64(A, B)
    assert (np.abs(d - ref) <= oracle.tolerance(ref, K)).all()


@pytest.mark.parametrize("variant", [g.MX_VARIANTS["mx_128x128"], g.MX_VARIANTS["mx_pair_256x128"],
                                     g.MX_VARIANTS["mx_pair_256x256"]])
def test_block_scaled_wait_runs_out_and_context_survives(variant):
    """The block-scaled kernels share the bounded waits: with no loads issued the MMA issuer's
    wait for operand data (and its scales) runs out, and the next launch is correct."""
    from blackwell_tensor_core_fp16_gb300.workloads import make_mx_inputs
    M, N, K = 520, 776, 1056
    A, B, SA, SB = make_mx_inputs(M, N, K, seed=701)
    Ad, Bd = A.cuda(), B.cuda()
    sfa, sfb = g.pack_scales(SA.cuda()), g.pack_scales(SB.cuda())
    D = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def launch():
        return g.gemm_mxf8_nt(Ad.data_ptr(), Bd.data_ptr(), sfa.data_ptr(), sfb.data_ptr(),
                              D.data_ptr(), M, N, K, 0, 0, 0, 0, 0, variant, 0, 0, s)

    assert g.gemm_f16_set_wait_timeout_ms(200) == g.OK
    assert g.gemm_f16_set_fault_injection(1) == g.OK
    assert launch() == g.OK
    rc, bits = g.gemm_f16_check_status(s)
    assert rc == g.ERR_TIMEOUT, (rc, bits)
    assert bits & 2, f"bits 0x{bits:x}"
    assert g.gemm_f16_check_status(s) == (g.OK, 0)

    assert g.gemm_f16_set_fault_injection(0) == g.OK
    assert g.gemm_f16_set_wait_timeout_ms(4000) == g.OK
    assert launch() == g.OK
    assert g.gemm_f16_check_status(s) == (g.OK, 0)
    d = D.cpu().double().numpy()
    ref, ref_abs = oracle.gemm_mx_f64(A, B, SA, SB)
    assert (np.abs(d - ref) <= oracle.tolerance_mx(ref, ref_abs, K, "f16")).all()


@pytest.mark.parametrize("scan", ["tensor_core_16", "tensor_core_32", "mma_sync"])
def test_gdn_scan_wait_runs_out_and_context_survives(scan):
    """The Gated Delta Net scan waits on an mbarrier for each chunk's TMA loads.  With
    gdn_set_fault_injection(1) the second chunk's loads are never issued, the 200 ms wait runs
    out, every scan CTA stops cleanly and gdn_check_status reads GDN_ERR_TIMEOUT; the next call
    (which clears the status word) matches the oracle."""
    from blackwell_tensor_core_fp16_gb300.workloads import make_gdn_inputs
    inp = make_gdn_inputs(200, 2, 1, 2, 128, 128, seed=702, state=True)
    q, k, v = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda()
    a, b, cu = inp["alpha"].cuda(), inp["beta"].cuda(), inp["cu_seqlens"].cuda()
    s0 = inp["initial_state"].cuda()
    T, n, h_qk, h_v = 200, 2, 1, 2
    o = torch.zeros((T, h_v, 128), dtype=torch.bfloat16, device="cuda")
    sf = torch.zeros((n, h_v, 128, 128), dtype=torch.float32, device="cuda")
    need = g.gdn_prefill_workspace_bytes(T, n, h_v)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def call():
        return g.gdn_prefill(q.data_ptr(), k.data_ptr(), v.data_ptr(), a.data_ptr(), b.data_ptr(),
                             cu.data_ptr(), n, T, h_qk, h_v, 128, 0.73, s0.data_ptr(),
                             o.data_ptr(), sf.data_ptr(), ws.data_ptr(), need, s)

    assert int(inp["cu_seqlens"].diff().max()) > 64, "a sequence needs a second chunk"
    assert g.gdn_set_scan_kernel(g.GDN_SCAN_KERNELS[scan]) == g.GDN_OK
    try:
        assert g.gdn_set_wait_timeout_ms(200) == g.GDN_OK
        assert g.gdn_set_fault_injection(1) == g.GDN_OK
        assert call() == g.GDN_OK
        assert g.gdn_check_status(ws.data_ptr(), s) == g.GDN_ERR_TIMEOUT
        assert "bounded wait" in g.gdn_last_error()
    finally:
        g.gdn_set_fault_injection(0)
        g.gdn_set_wait_timeout_ms(2000)
    o.fill_(float("nan"))
    sf.fill_(float("nan"))
    assert call() == g.GDN_OK
    assert g.gdn_check_status(ws.data_ptr(), s) == g.GDN_OK
    assert_parity(inp, o.float().cpu().double().numpy(), sf.cpu().double().numpy(), 0.73,
                  "the call after the timeout")
    g.gdn_set_scan_kernel(g.GDN_SCAN_KERNELS["auto"])
