"""Parity of the Gated Delta Net prefill (gdn_prefill) with the CPU oracle (needs a GB300).

Each case runs the C ABI on seeded inputs (workloads.make_gdn_inputs) and compares the bfloat16
outputs and the fp32 final states with the oracle's token-by-token binary64 recurrence.

Bounds, from the arithmetic.  The kernels compute in fp32 (unit roundoff 2^-24) in 64-token
chunks; each chunk adds rounding from sums of at most dk + 64 terms, and the state recurrence
is contractive for unit keys, 0 <= beta <= 1, 0 < alpha <= 1, so chunk errors add up at most
linearly over a sequence's n chunks.  With M the sequence's largest |o_ref| (largest |S_ref| for
the state):
    |o - o_ref| <= 2^-7 |o_ref| + n (dk + 64) 2^-22 M         (2^-7: twice bf16's half-ulp)
    |S - S_ref| <= 2^-20 |S_ref| + n (dk + 64) 2^-22 M
and, over a whole call, the root-mean-square error is at most 2^-8 of the RMS output (bfloat16
rounding alone gives about 0.58 * 2^-8) and 2^-14 of the RMS state: a mistake that shifts a
decay or drops a term fails these long before the elementwise bounds.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import blackwell_tensor_core_fp16_gb300 as g
from blackwell_tensor_core_fp16_gb300.workloads import (GDN_WORKLOADS, gdn_workload_inputs,
                                                         make_gdn_inputs)
from gdn_bounds import assert_parity

pytestmark = pytest.mark.gpu
C = 64


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    g.build()
    g.load()
    torch.cuda.init()


@pytest.fixture(autouse=True, params=["tensor_core_16", "tensor_core_32", "mma_sync"])
def scan_kernel(request, cuda_library):
    """Every case runs under every scan kernel: tcgen05 with 16 and with 32 state rows per work
    item (the default picks one by the item count) and mma.sync."""
    assert g.gdn_set_scan_kernel(g.GDN_SCAN_KERNELS[request.param]) == g.GDN_OK
    yield request.param
    g.gdn_set_scan_kernel(g.GDN_SCAN_KERNELS["auto"])


def run(inp, h_qk, h_v, scale=0.73, want_state=True):
    """gdn_prefill through the C ABI; outputs written into NaN-prefilled buffers."""
    q, k, v = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda()
    a, b = inp["alpha"].cuda(), inp["beta"].cuda()
    cu = inp["cu_seqlens"].cuda()
    s0 = None if inp["initial_state"] is None else inp["initial_state"].cuda()
    T, _, d = q.shape
    n = cu.numel() - 1
    o = torch.full((T, h_v, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    sf = torch.full((n, h_v, d, d), float("nan"), dtype=torch.float32, device="cuda") \
        if want_state else None
    need = g.gdn_prefill_workspace_bytes(T, n, h_v)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    rc = g.gdn_prefill(q.data_ptr(), k.data_ptr(), v.data_ptr(), a.data_ptr(), b.data_ptr(),
                       cu.data_ptr(), n, T, h_qk, h_v, d, scale,
                       0 if s0 is None else s0.data_ptr(), o.data_ptr(),
                       0 if sf is None else sf.data_ptr(), ws.data_ptr(), need,
                       torch.cuda.current_stream().cuda_stream)
    assert rc == g.GDN_OK, g.gdn_last_error()
    torch.cuda.synchronize()
    return o.float().cpu().double().numpy(), (None if sf is None else sf.cpu().double().numpy())


@pytest.mark.parametrize("name", list(GDN_WORKLOADS))
def test_page_scenarios(name):
    w = GDN_WORKLOADS[name]
    inp = gdn_workload_inputs(w)
    o, sf = run(inp, w.h_qk, w.h_v, w.scale, want_state=w.state)
    assert_parity(inp, o, sf, w.scale, name)


SHAPES = [
    # (T, n_seqs, h_qk, h_v, initial state)
    (1, 1, 1, 1, False),       # one token
    (7, 1, 2, 2, True),        # one short chunk
    (64, 1, 1, 1, True),       # exactly one chunk
    (65, 1, 1, 2, True),       # one chunk and one token, grouped values
    (200, 1, 2, 2, False),     # three chunks and a tail
    (300, 5, 2, 4, True),      # packed, ragged, grouped values
    (130, 3, 1, 1, True),      # packed with chunk-boundary-crossing lengths
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_shapes(shape):
    T, n, h_qk, h_v, st = shape
    inp = make_gdn_inputs(T, n, h_qk, h_v, 128, 128, seed=300 + T + n, state=st)
    o, sf = run(inp, h_qk, h_v)
    assert_parity(inp, o, sf, 0.73, f"{shape}")


def test_empty_sequences_keep_their_state():
    inp = make_gdn_inputs(100, 1, 1, 1, 128, 128, seed=9, state=True)
    # sequences of lengths 0, 40, 0, 60, 0 over the same 100 tokens
    inp["cu_seqlens"] = torch.tensor([0, 0, 40, 40, 100, 100], dtype=torch.int32)
    inp["initial_state"] = 0.1 * torch.randn((5, 1, 128, 128), generator=torch.Generator().manual_seed(3))
    o, sf = run(inp, 1, 1)
    assert_parity(inp, o, sf, 0.73, "empty sequences")
    s0 = inp["initial_state"].double().numpy()
    for i in (0, 2, 4):
        assert np.array_equal(sf[i], s0[i]), f"empty sequence {i} changed its state"


def test_deterministic():
    inp = make_gdn_inputs(300, 3, 2, 4, 128, 128, seed=10, state=True)
    o1, s1 = run(inp, 2, 4)
    o2, s2 = run(inp, 2, 4)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_rejects_bad_arguments():
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    x = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = x.data_ptr()
    s = torch.cuda.current_stream().cuda_stream

    def call(h_qk=1, h_v=1, d=128, n=1, T=4, wsb=1 << 20, qptr=p):
        return g.gdn_prefill(qptr, p, p, p, p, p, n, T, h_qk, h_v, d, 1.0, 0, p, 0,
                             ws.data_ptr(), wsb, s)

    assert call(h_qk=2, h_v=3) == g.GDN_ERR_INVALID_ARG      # h_v not a multiple of h_qk
    assert call(d=64) == g.GDN_ERR_UNSUPPORTED               # head dim other than 128
    assert call(qptr=p + 2) == g.GDN_ERR_UNSUPPORTED         # misaligned q
    assert call(wsb=16) == g.GDN_ERR_INVALID_ARG             # workspace too small
    assert call(n=-1) == g.GDN_ERR_INVALID_ARG
    assert call(n=0) == g.GDN_OK                             # nothing to do
    torch.cuda.synchronize()


# ---- cu_seqlens checked on the device -----------------------------------------------------------

@pytest.mark.parametrize("cu,T,ok", [
    ([0, 70, 100], 100, True),
    ([0, 0, 100, 100], 100, True),
    ([0, 70, 101], 100, False),          # past the last token
    ([0, -3, 100], 100, False),          # below 0
    ([0, 2 ** 31 - 1, 100], 100, False),
    ([0, 80, 70, 100], 100, False),      # decreasing
    ([5, 70, 100], 100, False),          # first offset not 0
    ([0, 70, 90], 100, False),           # last offset short
] + [([0] + list(range(3, 3 * 2000, 3)) + [6000], 6000, True),      # 2001 offsets, several
     ([0] + list(range(3, 3 * 2000, 3))[::-1] + [6000], 6000, False)],   # passes of the block
    ids=lambda x: None)
def test_offsets_checked_on_the_device(cu, T, ok):
    """gdn_check_offsets runs the chunk-list kernel alone: it reads the n + 1 offsets and writes
    only the workspace's tables, so offsets outside [0, T] are safe to give it.  The result read
    through gdn_check_status must follow the contract, and a valid check after a refused one
    clears the word."""
    n = len(cu) - 1
    need = g.gdn_prefill_workspace_bytes(T, n, 4)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dcu = torch.tensor(cu, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert g.gdn_check_offsets(dcu.data_ptr(), n, T, 4, ws.data_ptr(), need, s) == g.GDN_OK
    rc = g.gdn_check_status(ws.data_ptr(), s)
    assert rc == (g.GDN_OK if ok else g.GDN_ERR_INVALID_ARG), g.gdn_last_error()
    if not ok:
        assert "cu_seqlens" in g.gdn_last_error()
        good = torch.tensor([0, T], dtype=torch.int32, device="cuda")
        assert g.gdn_check_offsets(good.data_ptr(), 1, T, 4, ws.data_ptr(), need, s) == g.GDN_OK
        assert g.gdn_check_status(ws.data_ptr(), s) == g.GDN_OK


@pytest.mark.parametrize("cu", [[0, 99], [1, 100], [0, 120, 80, 200], [0, 100, 150],
                                [7, 90, 200]], ids=lambda c: "_".join(map(str, c)))
def test_broken_offsets_refuse_the_call(cu):
    """A whole call with offsets that break the contract but stay inside [0, T] (so that even an
    unchecked kernel could not leave its buffers): the call is refused on the device, no output is
    written (o keeps its NaN fill), every final state equals its initial state, and
    gdn_check_status reports GDN_ERR_INVALID_ARG.  The same workspace then serves a valid call,
    which matches the oracle."""
    T = 100 if len(cu) == 2 else 200
    n = len(cu) - 1
    inp = make_gdn_inputs(T, n, 1, 2, 128, 128, seed=61, state=True)
    q, k, v = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda()
    a, b = inp["alpha"].cuda(), inp["beta"].cuda()
    s0 = inp["initial_state"].cuda()
    o = torch.full((T, 2, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    sf = torch.full((n, 2, 128, 128), float("nan"), dtype=torch.float32, device="cuda")
    need = g.gdn_prefill_workspace_bytes(T, n, 2)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def call(cu_dev):
        return g.gdn_prefill(q.data_ptr(), k.data_ptr(), v.data_ptr(), a.data_ptr(),
                             b.data_ptr(), cu_dev.data_ptr(), n, T, 1, 2, 128, 0.73,
                             s0.data_ptr(), o.data_ptr(), sf.data_ptr(), ws.data_ptr(), need, s)

    bad = torch.tensor(cu, dtype=torch.int32, device="cuda")
    assert call(bad) == g.GDN_OK                       # enqueued: the host never reads cu
    assert g.gdn_check_status(ws.data_ptr(), s) == g.GDN_ERR_INVALID_ARG
    assert bool(torch.isnan(o.float()).all()), "a refused call wrote outputs"
    assert torch.equal(sf, s0), "a refused call changed a state"
    # the same buffers, valid offsets
    o.fill_(float("nan"))
    sf.fill_(float("nan"))
    assert call(inp["cu_seqlens"].cuda()) == g.GDN_OK
    assert g.gdn_check_status(ws.data_ptr(), s) == g.GDN_OK
    assert_parity(inp, o.float().cpu().double().numpy(), sf.cpu().double().numpy(), 0.73,
                  f"valid call after refused offsets {cu}")


def test_many_items_with_empty_sequences():
    """More work items than SMs (30 sequences x 8 value heads x 8 row blocks = 1920), so CTAs draw
    items dynamically and prefetch across items; a third of the sequences are empty and lie
    between non-empty ones."""
    T, n, h_qk, h_v = 2000, 30, 2, 8
    inp = make_gdn_inputs(T, n, h_qk, h_v, 128, 128, seed=41, state=True)
    g_ = torch.Generator().manual_seed(5)
    lens = torch.randint(1, 60, (n,), generator=g_)
    lens[::3] = 0                                   # every third sequence empty
    lens[-1] += T - int(lens.sum())                 # the rest to the last one
    assert int(lens.min()) >= 0 and int(lens.sum()) == T
    inp["cu_seqlens"] = torch.cat([torch.zeros(1, dtype=torch.int64), lens.cumsum(0)]).to(torch.int32)
    o, sf = run(inp, h_qk, h_v)
    assert_parity(inp, o, sf, 0.73, "30 sequences with empty ones")
    s0 = inp["initial_state"].double().numpy()
    for i in range(0, n, 3):
        assert np.array_equal(sf[i], s0[i]), f"empty sequence {i} changed its state"


def test_more_sequences_than_the_ranking_block():
    """1100 short sequences: beyond 1024 the scan takes sequences in index order."""
    n = 1100
    T = 3 * n
    inp = make_gdn_inputs(T, n, 1, 1, 128, 128, seed=42, state=True)
    o, sf = run(inp, 1, 1)
    assert_parity(inp, o, sf, 0.73, "1100 sequences")


def _grouped_query_inputs(T, n, h_q, h_k, h_v, seed, state=True):
    """make_gdn_inputs with h_k key heads, plus a separate q of h_q unit-norm bf16 heads."""
    inp = make_gdn_inputs(T, n, h_k, h_v, 128, 128, seed=seed, state=state)
    gq = torch.Generator().manual_seed(seed + 1000)
    x = torch.randn((T, h_q, 128), generator=gq)
    inp["q"] = (x / x.norm(dim=-1, keepdim=True).clamp_min(1e-6)).to(torch.bfloat16)
    return inp


def run_heads(inp, h_q, h_k, h_v, scale=0.73):
    """gdn_prefill_heads through the C ABI; outputs written into NaN-prefilled buffers."""
    q, k, v = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda()
    a, b = inp["alpha"].cuda(), inp["beta"].cuda()
    cu = inp["cu_seqlens"].cuda()
    s0 = None if inp["initial_state"] is None else inp["initial_state"].cuda()
    T = q.shape[0]
    n = cu.numel() - 1
    h_o = g.gdn_out_heads(h_q, h_k, h_v)
    o = torch.full((T, h_o, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    sf = torch.full((n, h_v, 128, 128), float("nan"), dtype=torch.float32, device="cuda")
    need = g.gdn_prefill_workspace_bytes(T, n, h_v)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    rc = g.gdn_prefill_heads(q.data_ptr(), k.data_ptr(), v.data_ptr(), a.data_ptr(), b.data_ptr(),
                             cu.data_ptr(), n, T, h_q, h_k, h_v, 128, scale,
                             0 if s0 is None else s0.data_ptr(), o.data_ptr(), sf.data_ptr(),
                             ws.data_ptr(), need, torch.cuda.current_stream().cuda_stream)
    assert rc == g.GDN_OK, g.gdn_last_error()
    torch.cuda.synchronize()
    return o.float().cpu().double().numpy(), sf.cpu().double().numpy()


GQA_SHAPES = [
    # (T, n_seqs, h_q, h_k, h_v)
    (300, 3, 4, 2, 2),      # GQA, 2 query heads per state, packed
    (200, 1, 8, 2, 2),      # GQA, 4 query heads per state, one sequence
    (150, 2, 4, 1, 2),      # grouped queries over grouped values
    (700, 30, 4, 1, 2),     # more work items than SMs, 2 passes
]


@pytest.mark.parametrize("shape", GQA_SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_grouped_queries(shape):
    T, n, h_q, h_k, h_v = shape
    inp = _grouped_query_inputs(T, n, h_q, h_k, h_v, seed=500 + T + n)
    o, sf = run_heads(inp, h_q, h_k, h_v)
    assert o.shape[1] == h_q
    assert_parity(inp, o, sf, 0.73, f"heads {shape}")


def test_grouped_query_torch_entry_point():
    inp = _grouped_query_inputs(130, 2, 4, 2, 2, seed=77)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    o, sf = g.gated_delta_rule(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["cu_seqlens"],
                               0.73, d["initial_state"], output_final_state=True)
    torch.cuda.synchronize()
    assert tuple(o.shape) == (130, 4, 128)
    assert_parity(inp, o.float().cpu().double().numpy(), sf.cpu().double().numpy(), 0.73,
                  "gated_delta_rule, grouped queries")


def test_rejects_bad_head_layouts():
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    x = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    p = x.data_ptr()
    s = torch.cuda.current_stream().cuda_stream

    def call(h_q, h_k, h_v):
        return g.gdn_prefill_heads(p, p, p, p, p, p, 1, 4, h_q, h_k, h_v, 128, 1.0, 0, p, 0,
                                   ws.data_ptr(), 1 << 20, s)

    assert call(3, 2, 2) == g.GDN_ERR_INVALID_ARG     # h_q neither h_k nor a multiple of h_v
    assert call(2, 2, 3) == g.GDN_ERR_INVALID_ARG     # h_v not a multiple of h_k
    assert call(18, 1, 2) == g.GDN_ERR_UNSUPPORTED    # 9 query heads per state
    torch.cuda.synchronize()


CARRY_CASES = [
    # (T, n_seqs, h_q, h_k, h_v)
    (300, 1, 2, 2, 2),      # one sequence, multi-head
    (500, 3, 4, 1, 2),      # packed, grouped queries over grouped values: two passes a call
    (700, 30, 2, 2, 4),     # grouped values, more work items than SMs
]


@pytest.mark.parametrize("case", CARRY_CASES, ids=lambda s: "-".join(map(str, s)))
def test_state_carried_in_place_across_calls(case):
    """Every sequence cut in two and run as two calls on one stream, one workspace and one state
    buffer that is both calls' initial and final state (updated in place), with no host
    synchronisation between the calls: the second call must see the first call's states, and
    the first call's workspace must be free before the second call writes it.  Compared with
    the oracle over the uncut sequences."""
    T, n, h_q, h_k, h_v = case
    inp = _grouped_query_inputs(T, n, h_q, h_k, h_v, seed=900 + T + n)
    cu = inp["cu_seqlens"].tolist()
    parts = ([], [])
    lens = ([], [])
    for i in range(n):
        mid = cu[i] + (cu[i + 1] - cu[i]) // 2
        for p, (a, b) in enumerate(((cu[i], mid), (mid, cu[i + 1]))):
            parts[p].append(torch.arange(a, b))
            lens[p].append(b - a)
    h_o = g.gdn_out_heads(h_q, h_k, h_v)
    o = torch.full((T, h_o, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    state = inp["initial_state"].cuda().clone()
    need = g.gdn_prefill_workspace_bytes(T, n, h_v)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    keep = []
    for p in range(2):
        idx = torch.cat(parts[p])
        Tp = int(idx.numel())
        cup = torch.tensor([0] + list(np.cumsum(lens[p])), dtype=torch.int32).cuda()
        d = {key: inp[key][idx].contiguous().cuda() for key in ("q", "k", "v", "alpha", "beta")}
        op = torch.empty((Tp, h_o, 128), dtype=torch.bfloat16, device="cuda")
        rc = g.gdn_prefill_heads(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                                 d["alpha"].data_ptr(), d["beta"].data_ptr(), cup.data_ptr(), n,
                                 Tp, h_q, h_k, h_v, 128, 0.73, state.data_ptr(), op.data_ptr(),
                                 state.data_ptr(), ws.data_ptr(), need, stream)
        assert rc == g.GDN_OK, g.gdn_last_error()
        keep.append((d, cup, op, idx))
    torch.cuda.synchronize()
    for d, cup, op, idx in keep:
        o[idx.cuda()] = op
    assert_parity(inp, o.float().cpu().double().numpy(), state.cpu().double().numpy(), 0.73,
                  f"carried state {case}", extra_chunks=1)


def test_long_sequence():
    """One sequence of 65,573 tokens (1,025 chunk steps, a ragged last chunk) in the grouped-value
    layout with an initial state: 64-bit offsets into q / k / v / o and a workspace of several
    hundred megabytes, and the chunk chain's rounding over a thousand dependent steps, against
    the oracle on every head."""
    T = 1025 * 64 - 27
    inp = make_gdn_inputs(T, 1, 2, 4, 128, 128, seed=65536, state=True)
    o, sf = run(inp, 2, 4)
    assert_parity(inp, o, sf, 0.73, f"one sequence of {T} tokens")
