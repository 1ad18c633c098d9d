"""Host-side logic of the Gated Delta Net entry points (no GPU: every call here returns before
any CUDA work).  Argument and head-layout checks, the workspace size, the settings hooks and the
Python binding's layout rule, which must agree with the oracle's."""
from __future__ import annotations

import pytest

import blackwell_tensor_core_fp16_gb300 as g
import oracle

FAKE = 1 << 20   # a non-null address that is never dereferenced: the checks fail first


@pytest.fixture(scope="module", autouse=True)
def library():
    g.build()
    g.load()


def call_heads(h_q, h_k, h_v, T=4, n=1, d=128, q=FAKE, ws_bytes=1 << 30):
    return g.gdn_prefill_heads(q, FAKE, FAKE, FAKE, FAKE, FAKE, n, T, h_q, h_k, h_v, d, 1.0, 0,
                               FAKE, 0, FAKE, ws_bytes, 0)


def test_head_layout_rule_matches_the_oracle():
    for h_q in range(1, 9):
        for h_k in range(1, 9):
            for h_v in range(1, 9):
                try:
                    ours = g.gdn_out_heads(h_q, h_k, h_v)
                except ValueError:
                    ours = None
                try:
                    ref = oracle.gdn_out_heads(h_q, h_k, h_v)
                except ValueError:
                    ref = None
                assert ours == ref, (h_q, h_k, h_v)


@pytest.mark.parametrize("heads", [(3, 2, 2), (2, 2, 3), (6, 2, 4), (2, 4, 2), (0, 1, 1)])
def test_bad_head_layouts_are_rejected_before_any_launch(heads):
    assert call_heads(*heads) == g.GDN_ERR_INVALID_ARG
    assert g.gdn_last_error()


def test_other_argument_checks():
    assert call_heads(2, 2, 2, d=64) == g.GDN_ERR_UNSUPPORTED         # head dim
    assert call_heads(2, 2, 2, q=FAKE + 2) == g.GDN_ERR_UNSUPPORTED   # misaligned q
    assert call_heads(2, 2, 2, n=-1) == g.GDN_ERR_INVALID_ARG
    assert call_heads(2, 2, 2, T=-5) == g.GDN_ERR_INVALID_ARG
    assert call_heads(2, 2, 2, ws_bytes=16) == g.GDN_ERR_INVALID_ARG   # workspace too small
    assert call_heads(2, 2, 2, n=0) == g.GDN_OK                       # nothing to do
    # the two-head-count entry point is the same check with h_q == h_k
    assert g.gdn_prefill(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 3, 128, 1.0, 0, FAKE, 0,
                         FAKE, 1 << 30, 0) == g.GDN_ERR_INVALID_ARG


def test_workspace_size():
    # per (chunk, value head): W in 3 bf16 pieces (48 KiB), A' in 2 (16 KiB), U'^T fp32
    # (32 KiB) and 2 x 64 decays; chunks are bounded by T / 64 + n_seqs
    per_cj = 3 * 64 * 128 * 2 + 2 * 64 * 64 * 2 + 128 * 64 * 4 + 2 * 64 * 4
    for T, n, h_v in [(0, 1, 1), (64, 1, 1), (4096, 1, 16), (8192, 20, 16), (1000, 7, 3)]:
        b = g.gdn_prefill_workspace_bytes(T, n, h_v)
        assert b >= (T // 64 + n) * h_v * per_cj
        assert b < (T // 64 + n) * h_v * per_cj + 64 * 1024 + 64 * n
    with pytest.raises(g.GemmError):
        g.gdn_prefill_workspace_bytes(-1, 1, 1)


def test_settings_hooks():
    assert g.gdn_set_wait_timeout_ms(0) == g.GDN_ERR_INVALID_ARG
    assert g.gdn_set_wait_timeout_ms(2000) == g.GDN_OK
    assert g.gdn_set_fault_injection(2) == g.GDN_ERR_INVALID_ARG
    assert g.gdn_set_fault_injection(0) == g.GDN_OK
    assert g.gdn_check_status(0, 0) == g.GDN_ERR_INVALID_ARG             # no workspace


def test_torch_entry_point_checks_shapes_before_anything_else():
    """Shape mistakes are caught on the host, before any device is touched (CPU tensors here:
    every case fails its shape check before the device check)."""
    import torch
    T, h, d = 10, 2, 128
    bf = torch.bfloat16
    good = dict(q=torch.zeros(T, h, d, dtype=bf), k=torch.zeros(T, h, d, dtype=bf),
                v=torch.zeros(T, h, d, dtype=bf), alpha=torch.ones(T, h),
                beta=torch.zeros(T, h), cu_seqlens=torch.tensor([0, T], dtype=torch.int32))
    bad = [
        dict(q=torch.zeros(T, h * d, dtype=bf)),          # q not 3-D
        dict(k=torch.zeros(T - 1, h, d, dtype=bf)),       # k missing a token
        dict(v=torch.zeros(T, h, 64, dtype=bf)),          # v with another head dim
        dict(alpha=torch.ones(T, h + 1)),                 # alpha over the wrong heads
        dict(beta=torch.zeros(T)),                        # beta not [T, h_v]
        dict(cu_seqlens=torch.zeros((), dtype=torch.int32)),
    ]
    for change in bad:
        args = dict(good, **change)
        with pytest.raises(ValueError, match="must"):
            g.gated_delta_rule(args["q"], args["k"], args["v"], args["alpha"], args["beta"],
                               args["cu_seqlens"], 1.0)
    with pytest.raises(ValueError, match="CUDA"):       # right shapes, CPU tensors
        g.gated_delta_rule(good["q"], good["k"], good["v"], good["alpha"], good["beta"],
                           good["cu_seqlens"], 1.0)
