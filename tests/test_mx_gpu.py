"""Parity of the block-scaled FP8 path (gemm_mxf8_nt) with the CPU oracle (needs a GB300).

Each case draws FP8 codes and E8M0 scales (workloads.make_mx_inputs), packs the scales with the
library's gemm_mxf8_pack_scales, runs gemm_mxf8_nt into a NaN-prefilled buffer flanked by guard
bands, and compares every output element with the oracle's binary64 sum D and its sum of
|terms| Dabs:

    |D_gpu - D| <= rel * |D| + 4 * (K/32 + 1) * 2^-24 * Dabs      (oracle.tolerance_mx)

with rel = 2^-10 for fp16 output and 2^-7 for bf16.  The probes with one 32-element block
(bf16 output, whose 8-bit exponent holds 2^-100 .. 2^100 exactly) recover which scale the
hardware applied to each output, so a layout mistake names the row, column or block it hit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import blackwell_tensor_core_fp16_gb300 as g
import oracle
from blackwell_tensor_core_fp16_gb300.workloads import (MX_WORKLOADS, make_mx_inputs,
                                                         mx_workload_inputs)

pytestmark = pytest.mark.gpu

GUARD = 4096
FILL = 0x7E5A                     # a NaN in fp16 and in bf16
VARIANTS = [g.MX_VARIANTS["mx_128x128"], g.MX_VARIANTS["mx_pair_256x128"],
            g.MX_VARIANTS["mx_pair_256x192"], g.MX_VARIANTS["mx_pair_256x256"]]
TDT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    g.build()
    g.load()
    torch.cuda.init()
    yield
    rc, bits = g.gemm_f16_check_status(0)
    assert rc == g.OK, f"a kernel gave up a bounded wait: bits 0x{bits:x}"


def tiled_layout_reference(S: np.ndarray, K: int) -> np.ndarray:
    """The tiled scale layout written out from its definition in include/gemm_f16.h."""
    rows, kb = S.shape
    kg = (kb + 3) // 4
    out = np.full(((rows + 127) // 128) * kg * 512, 127, np.uint8)
    for r in range(rows):
        for b in range(kb):
            off = ((r // 128) * kg + b // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + b % 4
            out[off] = S[r, b]
    return out


def run(A, B, SA, SB, variant=0, fmt_a="e4m3", fmt_b="e4m3", out_dtype="f16", bias=None,
        activation="none", workspace=None, on_device=False):
    """gemm_mxf8_nt through the C ABI on CPU uint8 inputs; returns D as float64 numpy (or the
    device tensor with on_device=True)."""
    M, K = A.shape
    N = B.shape[0]
    Ad, Bd = A.cuda(), B.cuda()
    sfa = g.pack_scales(SA.cuda())
    sfb = g.pack_scales(SB.cuda())
    buf = torch.full((2 * GUARD + M * N,), FILL, dtype=torch.int16, device="cuda")
    D = buf[GUARD:GUARD + M * N].view(TDT[out_dtype]).view(M, N)
    bias_d = None if bias is None else bias.cuda()
    ws_ptr, ws_bytes = 0, 0
    if workspace:
        need = g.gemm_mxf8_workspace_bytes(M, N, K, variant)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        ws_ptr, ws_bytes = ws.data_ptr(), need
    s = torch.cuda.current_stream()
    rc = g.gemm_mxf8_nt(Ad.data_ptr(), Bd.data_ptr(), sfa.data_ptr(), sfb.data_ptr(),
                        D.data_ptr(), M, N, K, g.FP8_FORMATS[fmt_a], g.FP8_FORMATS[fmt_b],
                        g.DTYPES[out_dtype], 0 if bias_d is None else bias_d.data_ptr(),
                        g.ACTIVATIONS[activation], variant, ws_ptr, ws_bytes, s.cuda_stream)
    assert rc == g.OK, g.gemm_f16_last_error()
    rc, bits = g.gemm_f16_check_status(s.cuda_stream)
    assert rc == g.OK, f"status bits 0x{bits:x}"
    assert bool((buf[:GUARD] == FILL).all()) and bool((buf[GUARD + M * N:] == FILL).all()), \
        "write outside D"
    if on_device:
        return D
    return D.float().double().cpu().numpy()


def assert_parity(d, d_ref, d_abs, K, out_dtype, where):
    assert np.isfinite(d).all(), f"{where}: non-finite output (unwritten element?)"
    err = np.abs(d - d_ref)
    tol = oracle.tolerance_mx(d_ref, d_abs, K, out_dtype)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        pytest.fail(f"{where}: {int(bad.sum())} of {bad.size} out of tolerance, worst err/tol "
                    f"{float((err / tol).max()):.3f}, first at {idx.tolist()}")


def full_parity(A, B, SA, SB, variant, where, fmt_a="e4m3", fmt_b="e4m3", out_dtype="f16",
                workspace=None):
    d = run(A, B, SA, SB, variant, fmt_a, fmt_b, out_dtype, workspace=workspace)
    ref, ref_abs = oracle.gemm_mx_f64(A, B, SA, SB, fmt_a, fmt_b)
    assert_parity(d, ref, ref_abs, A.shape[1], out_dtype, where)
    return d


# ---- the scale layout --------------------------------------------------------------------------

@pytest.mark.parametrize("rows,K", [(1, 32), (128, 128), (130, 96), (300, 1056), (513, 4096)])
def test_pack_scales_matches_the_layout(rows, K):
    rng = np.random.default_rng(rows + K)
    S = rng.integers(0, 255, size=(rows, K // 32)).astype(np.uint8)
    got = g.pack_scales(torch.from_numpy(S).cuda()).cpu().numpy()
    assert got.size == g.gemm_mxf8_scale_bytes(rows, K)
    assert np.array_equal(got, tiled_layout_reference(S, K))


# ---- probes: which scale reached which output --------------------------------------------------

def _probe(variant, M, N, SA, SB, K=32, live_block=None):
    A = np.zeros((M, K), np.uint8)
    lo, hi = (0, K) if live_block is None else (32 * live_block, 32 * live_block + 32)
    A[:, lo:hi] = 0x38                                 # 1.0
    B = np.full((N, K), 0x38, np.uint8)
    At, Bt = torch.from_numpy(A), torch.from_numpy(B)
    SAt, SBt = torch.from_numpy(SA), torch.from_numpy(SB)
    d = run(At, Bt, SAt, SBt, variant, out_dtype="bf16")
    ref, _ = oracle.gemm_mx_f64(A, B, SA, SB)
    return d, ref


@pytest.mark.parametrize("variant", VARIANTS)
def test_probe_row_scales(variant):
    M, N = 256, 128
    SA = (63 + (np.arange(M) % 128)).astype(np.uint8).reshape(M, 1)   # a distinct scale per row
    SB = np.full((N, 1), 127, np.uint8)
    d, ref = _probe(variant, M, N, SA, SB)
    if not np.array_equal(d, ref):
        used = np.log2(np.abs(d[:, 0]) / 32.0) + 127 - 63       # the row whose scale was used
        wrong = np.nonzero(used != np.arange(M) % 128)[0][:8]
        pytest.fail(f"rows {wrong.tolist()} used the scales of rows {used[wrong].tolist()}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_probe_column_scales(variant):
    M, N = 256, 384
    SA = np.full((M, 1), 127, np.uint8)
    SB = (63 + (np.arange(N) % 128)).astype(np.uint8).reshape(N, 1)
    d, ref = _probe(variant, M, N, SA, SB)
    if not np.array_equal(d, ref):
        used = np.log2(np.abs(d[0]) / 32.0) + 127 - 63
        wrong = np.nonzero(used != np.arange(N) % 128)[0][:8]
        pytest.fail(f"columns {wrong.tolist()} used the scales of columns "
                    f"{used[wrong].tolist()}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_probe_block_scales(variant):
    """K = 256 (two stages of 4 blocks); only one block of A is live at a time."""
    M, N, K = 256, 128, 256
    SA = (120 + np.arange(K // 32)).astype(np.uint8)[None, :].repeat(M, 0)
    SB = (100 + 2 * np.arange(K // 32)).astype(np.uint8)[None, :].repeat(N, 0)
    for b in range(K // 32):
        d, ref = _probe(variant, M, N, SA, SB, K=K, live_block=b)
        if not np.array_equal(d, ref):
            pytest.fail(f"live block {b}: got {d[0, 0]!r}, expected {ref[0, 0]!r} "
                        f"(2^{np.log2(ref[0, 0] / 32):.0f} * 32)")


# ---- the workloads that the oracle finishes in seconds, in full ---------------------------------

@pytest.mark.parametrize("variant", [0] + VARIANTS)
def test_single_tile_workload(variant):
    A, B, SA, SB = mx_workload_inputs(MX_WORKLOADS["mx_single_tile_128x128x128"])
    full_parity(A, B, SA, SB, variant, f"128x128x128 variant {variant}")


@pytest.mark.parametrize("variant", [0] + VARIANTS)
def test_square_2048_workload(variant):
    A, B, SA, SB = mx_workload_inputs(MX_WORKLOADS["mx_square_2048"])
    full_parity(A, B, SA, SB, variant, f"2048^3 variant {variant}")


@pytest.mark.parametrize("variant", [0] + VARIANTS)
def test_ragged_3000x5000x1056_workload(variant):
    A, B, SA, SB = mx_workload_inputs(MX_WORKLOADS["mx_ragged_3000x5000x1056"])
    full_parity(A, B, SA, SB, variant, f"3000x5000x1056 variant {variant}")


SHAPES = [
    (1, 8, 32),          # smallest legal problem: one block, part of one stage
    (129, 136, 96),      # one past a tile in M, ragged N, K tail of 3 blocks
    (255, 264, 160),     # one short of a pair tile; K of one stage and a block
    (520, 776, 1056),    # several tiles each way, every tail at once
    (64, 64, 16384),     # one tile, a long K loop (many ring wraps)
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_ragged_shapes(shape, variant):
    M, N, K = shape
    A, B, SA, SB = make_mx_inputs(M, N, K, seed=200 + M + N + K)
    full_parity(A, B, SA, SB, variant, f"{shape} variant {variant}")


@pytest.mark.parametrize("fmts", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
@pytest.mark.parametrize("variant", VARIANTS)
def test_formats(fmts, variant):
    fa, fb = fmts
    A, B, SA, SB = make_mx_inputs(392, 520, 480, seed=7, fmt_a=fa, fmt_b=fb)
    full_parity(A, B, SA, SB, variant, f"{fa} x {fb} variant {variant}", fa, fb)


@pytest.mark.parametrize("variant", VARIANTS)
def test_bf16_output(variant):
    A, B, SA, SB = make_mx_inputs(300, 264, 640, seed=8)
    full_parity(A, B, SA, SB, variant, f"bf16 out variant {variant}", out_dtype="bf16")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("activation", ["relu", "gelu"])
def test_fused_epilogue(variant, activation):
    from blackwell_tensor_core_fp16_gb300.workloads import make_bias
    M, N, K = 300, 264, 640
    A, B, SA, SB = make_mx_inputs(M, N, K, seed=9)
    bias = make_bias(N, seed=9, scale=4.0, dtype=torch.bfloat16)
    d = run(A, B, SA, SB, variant, out_dtype="bf16", bias=bias, activation=activation)
    ref, ref_abs = oracle.gemm_mx_f64(A, B, SA, SB)
    want = oracle.epilogue(ref, bias, activation, "bf16")
    # the epilogue's bias add and activation are 1-Lipschitz in the sum, so the bound carries
    tol = oracle.tolerance_mx(want, ref_abs, K, "bf16") + 2.0 ** -7 * np.abs(ref)
    err = np.abs(d - want)
    assert np.isfinite(d).all()
    assert (err <= tol).all(), f"worst err/tol {float((err / tol).max()):.3f}"


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", ["mx_square_2048", "ragged_1000x1800x1568"])
def test_stream_k_tail_parity(name, variant, stream_k_on):
    """With a workspace, the tiles of a partial last wave are split by K blocks across units
    (the pieces are summed by the last contributor).  Both shapes leave a partial last wave for
    every variant on a 152-SM GB300; the ragged one also has partial M / N tiles and a partial
    last K block (1568 = 12 x 128 + 32)."""
    if name in MX_WORKLOADS:
        w = MX_WORKLOADS[name]
        M, N, K = w.M, w.N, w.K
        A, B, SA, SB = mx_workload_inputs(w)
    else:
        M, N, K = 1000, 1800, 1568
        A, B, SA, SB = make_mx_inputs(M, N, K, seed=1568)
    assert g.gemm_mxf8_workspace_bytes(M, N, K, variant) > 0, \
        "this shape is meant to take the stream-K tail"
    full_parity(A, B, SA, SB, variant, f"{name} stream-K variant {variant}", workspace=True)


def test_deterministic():
    A, B, SA, SB = make_mx_inputs(520, 776, 1056, seed=11)
    d1 = run(A, B, SA, SB, 0)
    d2 = run(A, B, SA, SB, 0)
    assert np.array_equal(d1, d2)


def test_unit_values_sum_exactly():
    """A = B = 1.0 with scales 2^0: every output is exactly K (at every large shape's K)."""
    for K in (4096, 8192):
        M, N = 384, 392
        A = torch.full((M, K), 0x38, dtype=torch.uint8)
        B = torch.full((N, K), 0x38, dtype=torch.uint8)
        S = torch.full((M, K // 32), 127, dtype=torch.uint8)
        T = torch.full((N, K // 32), 127, dtype=torch.uint8)
        d = run(A, B, S, T, 0)
        assert (d == K).all()


# ---- the large workloads: sampled outputs ------------------------------------------------------

def _samples(M, N, rng, count=3000):
    edges_r = np.array([0, 1, 127, 128, 255, 256, M // 2, M - 129, M - 128, M - 2, M - 1])
    edges_c = np.array([0, 1, 127, 128, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1])
    r = np.concatenate([np.repeat(edges_r, edges_c.size), rng.integers(0, M, count)])
    c = np.concatenate([np.tile(edges_c, edges_r.size), rng.integers(0, N, count)])
    return r, c


@pytest.mark.parametrize("name", ["mx_square_8192", "mx_mlp_up_16384x14336x4096"])
def test_large_workloads_sampled(name):
    w = MX_WORKLOADS[name]
    A, B, SA, SB = mx_workload_inputs(w)
    D = run(A, B, SA, SB, 0, on_device=True)
    assert bool(torch.isfinite(D).all()), "an element was not written"
    r, c = _samples(w.M, w.N, np.random.default_rng(5))
    d = D[torch.from_numpy(r).cuda(), torch.from_numpy(c).cuda()].double().cpu().numpy()
    ref, ref_abs = oracle.gemm_mx_f64_sampled(A, B, SA, SB, r, c)
    assert_parity(d, ref, ref_abs, w.K, "f16", name)


# ---- argument checks ------------------------------------------------------------------------------

def test_rejects_bad_arguments():
    A = torch.zeros((128, 64), dtype=torch.uint8, device="cuda")
    S = g.pack_scales(torch.full((128, 2), 127, dtype=torch.uint8, device="cuda"))
    D = torch.empty((128, 128), dtype=torch.float16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def call(K=64, fa=0, dt=0, sfa=S.data_ptr(), variant=0):
        return g.gemm_mxf8_nt(A.data_ptr(), A.data_ptr(), sfa, S.data_ptr(), D.data_ptr(), 128,
                              128, K, fa, 0, dt, 0, 0, variant, 0, 0, s)

    assert call(K=48) == g.ERR_UNSUPPORTED           # not a multiple of the 32-element block
    assert call(fa=2) == g.ERR_INVALID_ARG           # unknown format
    assert call(dt=5) == g.ERR_INVALID_ARG           # unknown output type
    assert call(sfa=0) == g.ERR_INVALID_ARG          # null scales
    assert call(sfa=S.data_ptr() + 4) == g.ERR_UNSUPPORTED   # misaligned scales
    assert call(variant=9) == g.ERR_INVALID_ARG
    assert call() == g.OK
    torch.cuda.synchronize()
