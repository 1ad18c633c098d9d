"""The C ABI recorded into CUDA graphs and replayed (needs a GB300).

A caller that captures a step into a CUDA graph records the library's launches, memsets and
programmatic-dependent-launch edges once and replays them later.  These tests record
gemm_f16_nt, gemm_f16_nt_noalloc (stream-K with the library's fixed scratch) and the Gated Delta
Net prefill (chunk list, prepare and scan kernels, several passes for grouped queries), replay
each graph into NaN-filled outputs, and compare the replays with eager calls on the same inputs:
bit for bit where the kernel's summation order is the eager call's, within the GEMM tolerance
|x - y| <= 1e-3 sqrt(K) + 2^-10 |y| for the stream-K schedule (turned on for these tests), whose
tail tiles group their fp32 additions differently; its replays equal one another bit for bit
(the piece that finishes a tile adds the others in k order, whenever they finish).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import blackwell_tensor_core_fp16_gb300 as g
from blackwell_tensor_core_fp16_gb300.workloads import make_gdn_inputs, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    g.build()
    g.load()
    yield


def record(call):
    """Runs `call(stream)` once eagerly on a side stream, then records it into a CUDA graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(side.cuda_stream)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return graph


def _within_tolerance(x, y, K):
    xd, yd = x.double().cpu().numpy(), y.double().cpu().numpy()
    assert np.isfinite(xd).all(), "non-finite output"
    err = np.abs(xd - yd)
    tol = 1e-3 * np.sqrt(K) + 2.0 ** -10 * np.abs(yd)
    assert (err <= tol).all(), f"max err/tol {float((err / tol).max()):.3f}"


@pytest.mark.parametrize("shape", [(1000, 1032, 1536), (4096, 4096, 2048), (8192, 8192, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gemm_replays_match_eager_calls(shape, stream_k_on):
    M, N, K = shape
    A_cpu, B_cpu = make_inputs(M, N, K, seed=1200 + M + K, a_dist="normal", a_scale=K ** -0.5,
                               b_dist="normal", b_scale=1.0)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    ref = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert g.gemm_f16_nt(A.data_ptr(), B.data_ptr(), ref.data_ptr(), M, N, K,
                         torch.cuda.current_stream().cuda_stream) == g.OK, g.gemm_f16_last_error()
    for entry, exact in ((g.gemm_f16_nt, True), (g.gemm_f16_nt_noalloc, False)):
        D = torch.empty((M, N), dtype=torch.float16, device="cuda")

        def call(s, entry=entry, D=D):
            assert entry(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, s) == g.OK, \
                g.gemm_f16_last_error()

        graph = record(call)
        # three replays: the stream-K flags alternate between two regions of the fixed array
        first = None
        for _ in range(3):
            D.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            rc, bits = g.gemm_f16_check_status(torch.cuda.current_stream().cuda_stream)
            assert rc == g.OK, f"status bits 0x{bits:x}"
            if exact:
                assert torch.equal(D, ref), f"{entry.__name__}: replay differs from the eager call"
            else:
                _within_tolerance(D, ref, K)
                if first is None:
                    first = D.clone()
                else:
                    assert torch.equal(D, first), f"{entry.__name__}: replays differ"


GDN_CASES = [
    # (T, n_seqs, h_q, h_k, h_v)
    (700, 1, 4, 4, 4),      # one sequence: prepare and scan only
    (900, 7, 2, 2, 4),      # packed, grouped values: chunk list, prepare, scan
    (500, 3, 4, 1, 2),      # grouped queries: two passes of prepare and scan
]


@pytest.mark.parametrize("case", GDN_CASES, ids=lambda s: "-".join(map(str, s)))
def test_gdn_replays_match_eager_calls(case):
    T, n, h_q, h_k, h_v = case
    inp = make_gdn_inputs(T, n, h_k, h_v, 128, 128, seed=1300 + T + n, state=True)
    gq = torch.Generator().manual_seed(1400 + T)
    x = torch.randn((T, h_q, 128), generator=gq)
    inp["q"] = (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    h_o = g.gdn_out_heads(h_q, h_k, h_v)
    need = g.gdn_prefill_workspace_bytes(T, n, h_v)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def outputs():
        return (torch.empty((T, h_o, 128), dtype=torch.bfloat16, device="cuda"),
                torch.empty((n, h_v, 128, 128), dtype=torch.float32, device="cuda"))

    def caller(o, sf):
        def call(s):
            rc = g.gdn_prefill_heads(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                                     d["alpha"].data_ptr(), d["beta"].data_ptr(),
                                     d["cu_seqlens"].data_ptr(), n, T, h_q, h_k, h_v, 128, 0.73,
                                     d["initial_state"].data_ptr(), o.data_ptr(), sf.data_ptr(),
                                     ws.data_ptr(), need, s)
            assert rc == g.GDN_OK, g.gdn_last_error()
        return call

    o_ref, s_ref = outputs()
    caller(o_ref, s_ref)(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    o, sf = outputs()
    graph = record(caller(o, sf))
    for _ in range(2):
        o.fill_(float("nan"))
        sf.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert g.gdn_check_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == g.GDN_OK
        assert torch.equal(o, o_ref), "output of the replay differs from the eager call"
        assert torch.equal(sf, s_ref), "final states of the replay differ from the eager call"
