"""The allocation-free entry point gemm_f16_nt_noalloc (needs a GB300).

Some callers cannot allocate device memory at the moment they need a GEMM: servers whose device
memory all belongs to their own pool, plug-ins inside a host program that owns every allocation,
and latency-bound loops that cannot take cudaMalloc's implicit synchronisation.  gemm_f16_nt_noalloc
serves them with the data-parallel schedule, or, with the stream-K tail turned on, with the
stream-K workspace in a fixed device array that the library reserves when it is loaded.

Every stream-K call shares that array and finds the previous call's partial sums and flags in it.
The test calls the entry point through the C ABI, with stream-K on and off, on a sequence of
shapes whose stream-K layouts differ (CTA pairs with 36 tail tiles and with all 64 tiles split,
single 128 x 128 CTAs with 72 and 96), one shape twice in a row and the first shape again at the
end, and checks every output element against the CPU oracle's binary64 sum with the parity tests'
bound
|D - D_ref| <= 1e-3 * sqrt(K) + 2^-10 * |D_ref| (in full for the mid-size shapes, on sampled
elements for 8192^3), plus the status word after each call.  The file is named so that pytest
collects it last.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import blackwell_tensor_core_fp16_gb300 as g
import oracle
from blackwell_tensor_core_fp16_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    g.build()
    g.load()
    yield


def _edge_and_random(M, N, rng, count=3000):
    edges_m = sorted({r for r in (0, 1, 127, 128, 255, 256, M // 2, M - 129, M - 128, M - 2,
                                  M - 1) if 0 <= r < M})
    edges_n = sorted({c for c in (0, 1, 63, 64, 127, 128, 255, 256, N // 2, N - 257, N - 256,
                                  N - 2, N - 1) if 0 <= c < N})
    er, ec = np.meshgrid(edges_m, edges_n, indexing="ij")
    rows = np.concatenate([er.ravel(), rng.integers(0, M, count)]).astype(np.int64)
    cols = np.concatenate([ec.ravel(), rng.integers(0, N, count)]).astype(np.int64)
    return rows, cols


def _assert_oracle_parity(got: np.ndarray, ref: np.ndarray, K: int, where: str) -> None:
    assert np.isfinite(got).all(), f"{where}: non-finite output (an element was not written)"
    err = np.abs(got - ref)
    tol = oracle.tolerance(ref, K)
    bad = err > tol
    assert not bad.any(), (f"{where}: {int(bad.sum())} elements out of bound, worst err/tol "
                           f"{float((err / tol).max()):.3f}")


# (M, N, K) in call order: the automatic variant and stream-K tail of each on 152 SMs are in
# the comments; 1000 x 1032 x 1536 runs twice in a row, 8192^3 first and last.
SEQUENCE = [
    (8192, 8192, 8192),    # CTA pair 256 x 256, 36 tail tiles over 76 pairs
    (1000, 1032, 1536),    # 128 x 128, all 72 tiles stream-K over 152 CTAs
    (1000, 1032, 1536),    # the same again: finds its own leftovers
    (2048, 2048, 2048),    # CTA pair, all 64 tiles stream-K
    (700, 2000, 4000),     # 128 x 128, 96 tiles
    (8192, 8192, 8192),    # back to the pair layout
]


@pytest.mark.parametrize("stream_k", [1, 0], ids=["stream_k", "data_parallel"])
def test_noalloc_sequence_matches_oracle(stream_k):
    stream = torch.cuda.current_stream()
    cache = {}
    assert g.gemm_f16_set_stream_k(stream_k) == g.OK
    try:
        _run_sequence(stream, cache, stream_k)
    finally:
        g.gemm_f16_set_stream_k(0)


def _run_sequence(stream, cache, stream_k):
    for call, (M, N, K) in enumerate(SEQUENCE):
        where = f"call {call} ({M}x{N}x{K}, stream-K {'on' if stream_k else 'off'})"
        need = g.gemm_f16_workspace_bytes(M, N, K, 0)
        if stream_k:
            assert 0 < need <= g.gemm_f16_noalloc_scratch_bytes(), \
                f"{where} is meant to use the scratch"
        else:
            assert need == 0, f"{where}: stream-K is off"
        if (M, N, K) not in cache:
            A_cpu, B_cpu = make_inputs(M, N, K, seed=900 + M + N + K, a_dist="normal",
                                       a_scale=K ** -0.5, b_dist="normal", b_scale=1.0)
            if M * N * K <= 2048 ** 3:
                ref = oracle.gemm_f64(A_cpu, B_cpu)
                idx = None
            else:
                idx = _edge_and_random(M, N, np.random.default_rng(M + K))
                ref = oracle.gemm_f64_sampled(A_cpu, B_cpu, *idx)
            cache[(M, N, K)] = (A_cpu.cuda(), B_cpu.cuda(), ref, idx)
        A, B, ref, idx = cache[(M, N, K)]
        D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        rc = g.gemm_f16_nt_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                                   stream.cuda_stream)
        assert rc == g.OK, f"{where}: {g.gemm_f16_last_error()}"
        rc, bits = g.gemm_f16_check_status(stream.cuda_stream)
        assert rc == g.OK, f"{where}: status bits 0x{bits:x}"
        if idx is None:
            got = D.double().cpu().numpy()
        else:
            assert not torch.isnan(D).any(), f"{where}: unwritten output elements"
            got = D[torch.from_numpy(idx[0]).cuda(), torch.from_numpy(idx[1]).cuda()]
            got = got.double().cpu().numpy()
        _assert_oracle_parity(got, ref, K, where)


def test_noalloc_shapes_without_scratch_and_bad_arguments():
    # a single tile needs no scratch: the entry point still computes it
    A_cpu, B_cpu = make_inputs(128, 128, 64, seed=5)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    D = torch.full((128, 128), float("nan"), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert g.gemm_f16_workspace_bytes(128, 128, 64, 0) == 0
    assert g.gemm_f16_nt_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), 128, 128, 64, s) == g.OK
    rc, bits = g.gemm_f16_check_status(s)
    assert rc == g.OK, f"status bits 0x{bits:x}"
    _assert_oracle_parity(D.double().cpu().numpy(), oracle.gemm_f64(A_cpu, B_cpu), 64,
                          "128x128x64")
    # argument checks are the same as gemm_f16_nt's
    assert g.gemm_f16_nt_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), 128, 128, 60, s) == \
        g.ERR_UNSUPPORTED
    assert g.gemm_f16_nt_noalloc(0, B.data_ptr(), D.data_ptr(), 128, 128, 64, s) == \
        g.ERR_INVALID_ARG
