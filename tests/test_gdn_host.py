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


def _offsets_rule(cu, total_tokens):
    """The packed-input contract written out plainly: starts at 0, ends at total_tokens, never
    decreases (so every sequence stays inside [0, total_tokens) and none crosses another)."""
    if len(cu) == 0 or cu[0] != 0 or cu[-1] != total_tokens:
        return False
    return all(a <= b for a, b in zip(cu[:-1], cu[1:]))


@pytest.mark.parametrize("cu,T,ok", [
    ([0, 100], 100, True),                 # one sequence
    ([0, 30, 30, 100], 100, True),         # an empty sequence inside
    ([0, 0, 0], 0, True),                  # no tokens at all
    ([0, 100], 99, False),                 # last offset past total_tokens
    ([0, 99], 100, False),                 # last offset short of total_tokens
    ([1, 100], 100, False),                # first offset not 0
    ([0, 60, 40, 100], 100, False),        # a decreasing pair
    ([0, -5, 100], 100, False),            # an offset below 0
    ([0, 2 ** 31 - 1, 100], 100, False),   # an offset far past the end
    ([0], 0, True),                        # no sequence (n_seqs = 0)
    ([0], 5, False),
])
def test_offsets_rule_host_replay(cu, T, ok):
    """The device kernels' check of cu_seqlens, replayed on the host through the library's own
    copy of the rule, against the contract written out in this test."""
    assert _offsets_rule(cu, T) == ok
    assert g.gdn_offsets_valid_host(cu, T) == ok


def test_offsets_rule_random_arrays():
    import random
    rng = random.Random(5)
    for _ in range(2000):
        n = rng.randint(0, 6)
        T = rng.randint(0, 300)
        cu = sorted(rng.randint(0, T) for _ in range(n + 1))
        if cu:
            cu[0], cu[-1] = 0, T
        if rng.random() < 0.5 and n > 0:   # break it somewhere
            i = rng.randint(0, n)
            cu[i] += rng.choice([-3, -1, 1, 7])
        assert g.gdn_offsets_valid_host(cu, T) == _offsets_rule(cu, T), (cu, T)


def test_check_offsets_argument_checks():
    assert g.gdn_check_offsets(0, 2, 100, 4, FAKE, 1 << 30, 0) == g.GDN_ERR_INVALID_ARG
    assert g.gdn_check_offsets(FAKE, -1, 100, 4, FAKE, 1 << 30, 0) == g.GDN_ERR_INVALID_ARG
    assert g.gdn_check_offsets(FAKE, 2, 100, 4, FAKE, 16, 0) == g.GDN_ERR_INVALID_ARG
    assert g.gdn_check_offsets(FAKE, 2, 100, 4, 0, 1 << 30, 0) == g.GDN_ERR_INVALID_ARG
