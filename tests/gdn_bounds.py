"""Element-wise and RMS bounds of the Gated Delta Net prefill against the CPU oracle, shared by
the GPU tests.  The kernels compute in fp32 (unit roundoff 2^-24) in 64-token chunks; each chunk
adds rounding from sums of at most dk + 64 terms, and the state recurrence is contractive for
unit keys, 0 <= beta <= 1, 0 < alpha <= 1, so chunk errors add up at most linearly over a
sequence's n chunks.  With M the sequence's largest |o_ref| (largest |S_ref| for the state):
    |o - o_ref| <= 2^-7 |o_ref| + n (dk + 64) 2^-22 M         (2^-7: twice bf16's half-ulp)
    |S - S_ref| <= 2^-20 |S_ref| + n (dk + 64) 2^-22 M
and over a whole call the RMS error is at most 2^-8 of the RMS output and 2^-14 of the RMS
state."""
from __future__ import annotations

import numpy as np
import pytest

import oracle

C = 64


def assert_parity(inp, o, sf, scale, where, extra_chunks=0):
    ref_o, ref_s = oracle.gdn_f64(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"],
                                  inp["cu_seqlens"], scale, inp["initial_state"])
    cu = inp["cu_seqlens"].numpy()
    assert np.isfinite(o).all(), f"{where}: an output was not written"
    dk = inp["q"].shape[2]
    for i in range(len(cu) - 1):
        sl = slice(cu[i], cu[i + 1])
        n = max(1, -(-(cu[i + 1] - cu[i]) // C)) + extra_chunks
        ro = ref_o[sl]
        if ro.size == 0:
            continue
        M = np.abs(ro).max(axis=(0, 2), keepdims=True)     # per value head
        tol = 2.0 ** -7 * np.abs(ro) + n * (dk + C) * 2.0 ** -22 * M
        err = np.abs(o[sl] - ro)
        if (err > tol).any():
            idx = np.argwhere(err > tol)[:4]
            pytest.fail(f"{where}: sequence {i}: {int((err > tol).sum())} outputs out of bound, "
                        f"worst err/tol {float((err / tol).max()):.3f}, first at {idx.tolist()}")
        if sf is not None:
            rs = ref_s[i]
            Ms = np.abs(rs).max(axis=(1, 2), keepdims=True)
            tols = 2.0 ** -20 * np.abs(rs) + n * (dk + C) * 2.0 ** -22 * Ms
            errs = np.abs(sf[i] - rs)
            assert (errs <= tols).all(), \
                f"{where}: sequence {i}: state worst err/tol {float((errs / tols).max()):.3f}"
    rms = lambda x: float(np.sqrt(np.mean(np.square(x)))) if x.size else 0.0
    if ref_o.size:
        assert rms(o - ref_o) <= 2.0 ** -8 * rms(ref_o), \
            f"{where}: output RMS error {rms(o - ref_o) / rms(ref_o):.2e} of the RMS output"
    if sf is not None and ref_s.size:
        assert rms(sf - ref_s) <= 2.0 ** -14 * rms(ref_s), \
            f"{where}: state RMS error {rms(sf - ref_s) / rms(ref_s):.2e} of the RMS state"
