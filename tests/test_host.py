"""Host-side tests of the CUDA library (no GPU): the C ABI loads and exports every declared
symbol, the encoders reproduce the values the pages print, the ring and scheduler logic
holds its invariants, and argument checks reject bad calls before any CUDA call is made."""
from __future__ import annotations

import ctypes
import os

import pytest

import blackwell_tensor_core_fp16_gb300 as g

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden_rows(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


@pytest.fixture(scope="session", autouse=True)
def built_library():
    g.build()
    return g.load()


def test_library_exports_every_declared_symbol(built_library):
    names = g.exported_symbols()
    assert "gemm_f16_nt" in names and len(names) >= 10
    for n in names:
        assert hasattr(built_library, n), f"{n} declared in include/gemm_f16.h but not exported"


def test_version():
    assert g.gemm_f16_version() >= 10000


# ---- encoders against the pages ---------------------------------------------------------------

def test_idesc_matches_page_constant():
    for M, N, bf16, want in golden_rows("idesc_f16.txt"):
        assert g.gemm_f16_idesc(int(M), int(N), int(bf16)) == int(want, 16)


def test_idesc_fields():
    d = g.gemm_f16_idesc(256, 256, 0)
    assert (d >> 4) & 3 == 1            # f32 accumulator
    assert (d >> 7) & 7 == 0 and (d >> 10) & 7 == 0  # f16 A and B
    assert (d >> 15) & 1 == 0 and (d >> 16) & 1 == 0  # both K-major
    assert (d >> 17) & 0x3F == 256 >> 3
    assert (d >> 24) & 0x1F == 256 >> 4
    assert d & 0xF == 0 and (d >> 13) & 3 == 0 and (d >> 29) == 0
    b = g.gemm_f16_idesc(128, 256, 1)
    assert (b >> 7) & 7 == 1 and (b >> 10) & 7 == 1


def test_swizzle_bank_map_matches_page():
    for i, bank_sw, bank_plain in golden_rows("sw128_f16_8x64_column0_banks.txt"):
        i = int(i)
        byte = g.gemm_f16_sw128(128 * i + 0)      # element (i, 0) of a 128-byte-row tile
        assert (byte // 4) % 32 == int(bank_sw)
        assert ((128 * i) // 4) % 32 == int(bank_plain)


def test_swizzle_element_formula_whole_tile():
    """addr = 64*i + 8*(q xor i) + r elements for every (i, j) of an (8, 64) fp16 tile, and the
    pattern repeats every 8 rows (rows 8..127 of a 128-row operand tile)."""
    for i in range(128):
        for j in range(64):
            q, r = divmod(j, 8)
            want_elem = 64 * i + 8 * (q ^ (i % 8)) + r
            assert g.gemm_f16_sw128(2 * (64 * i + j)) == 2 * want_elem


def test_swizzle_is_a_permutation_of_each_atom():
    for base in (0, 1024, 8192):
        outs = {g.gemm_f16_sw128(base + o) for o in range(0, 1024, 16)}
        assert outs == set(range(base, base + 1024, 16))


def test_smem_descriptor_fields():
    addr = 0x12400  # 1024-byte aligned shared address
    d = g.gemm_f16_smem_desc_sw128(addr, 1024)
    assert d & 0x3FFF == addr >> 4
    assert (d >> 16) & 0x3FFF == 1
    assert (d >> 32) & 0x3FFF == 1024 >> 4
    assert (d >> 46) & 7 == 1
    assert (d >> 49) & 7 == 0 and (d >> 52) & 1 == 0
    assert (d >> 61) & 7 == 2
    # advancing K by 16 fp16 (32 bytes) inside the swizzle row adds 2 to the address field
    assert g.gemm_f16_smem_desc_sw128(addr + 32, 1024) == d + 2


def test_expect_tx_bytes_match_page():
    (bm, bn, bk, want), = golden_rows("expect_tx_bytes.txt")
    info = g.gemm_f16_get_variant_info(g.VARIANTS["tile"])
    assert (info["block_m"], info["block_n"], info["block_k"]) == (int(bm), int(bn), int(bk))
    assert info["stage_tx_bytes"] == int(want)
    # the same formula for the other variants (a pair counts both CTAs' loads)
    for name in ("ws_128x256", "ws_128x128", "ws_pair", "ws_pair_256x192"):
        v = g.gemm_f16_get_variant_info(g.VARIANTS[name])
        assert v["stage_tx_bytes"] == (v["block_m"] * v["block_k"] + v["block_n"] * v["block_k"]) * 2


def test_variant_info_resources():
    for name, v in g.VARIANTS.items():
        if v == 0:
            continue
        info = g.gemm_f16_get_variant_info(v)
        assert info["smem_bytes"] <= 232448          # 227 KB per CTA
        assert info["tmem_cols"] in (32, 64, 128, 256, 512)
        if info["persistent"]:
            # two accumulators, in the power of two that tcgen05.alloc takes
            assert info["tmem_cols"] >= 2 * info["block_n"]
            assert info["tmem_cols"] < 4 * info["block_n"]
    with pytest.raises(g.GemmError):
        g.gemm_f16_get_variant_info(99)


# ---- pipeline phase bookkeeping ----------------------------------------------------------------

def test_single_barrier_phase_table_matches_page():
    """With one stage the ring position's parity is the page's phase before the wait, and the
    next iteration's parity is the phase after it."""
    for k, before, after in golden_rows("mbarrier_phase_table.txt"):
        k = int(k)
        assert g.gemm_f16_ring_pos(k, 1) == (0, int(before))
        assert g.gemm_f16_ring_pos(k + 1, 1)[1] == int(after)


def test_step6_parity_returns_after_even_uses():
    (K, bk, depth, mma_uses, stage_uses), = golden_rows("ring_parity_step6.txt")
    iters = int(K) // int(bk)
    assert iters == int(mma_uses)
    uses = [0] * int(depth)
    for it in range(iters):
        s, _ = g.gemm_f16_ring_pos(it, int(depth))
        uses[s] += 1
    assert uses == [int(stage_uses)] * int(depth)
    assert g.gemm_f16_ring_pos(iters, int(depth)) == (0, 0)  # parity back to the start


class _BarrierModel:
    """A host model of an mbarrier's phase: completes a phase per `complete()`;
    try_wait(parity) is true iff the phase with that parity has completed and no newer one."""

    def __init__(self):
        self.phase = 0

    def complete(self):
        self.phase += 1

    def try_wait(self, parity):
        # the current (incomplete) phase has parity phase & 1; the previous one is complete
        return (self.phase & 1) != parity


@pytest.mark.parametrize("stages", [1, 2, 4, 6])
@pytest.mark.parametrize("k_iters", [1, 3, 16, 17, 64])
def test_ring_protocol_model_across_tiles(stages, k_iters):
    """Simulate producer and consumer on per-stage full/empty barriers over several tiles whose
    K-iteration count is not a multiple of 2*stages: with positions carried across tiles, every
    wait returns exactly when its data is ready and never early."""
    full = [_BarrierModel() for _ in range(stages)]
    empty = [_BarrierModel() for _ in range(stages)]
    total = 3 * k_iters
    produced = consumed = 0
    stage_content = [None] * stages
    steps = 0
    while consumed < total:
        steps += 1
        assert steps < 100 * total
        # producer tries to fill iteration `produced`
        if produced < total:
            s, par = g.gemm_f16_ring_pos(produced, stages)
            if empty[s].try_wait(par ^ 1):
                assert stage_content[s] is None, "producer overwrote an unconsumed stage"
                stage_content[s] = produced
                full[s].complete()
                produced += 1
        # consumer tries iteration `consumed`
        s, par = g.gemm_f16_ring_pos(consumed, stages)
        if full[s].try_wait(par):
            assert stage_content[s] == consumed, "consumer saw the wrong iteration"
            stage_content[s] = None
            empty[s].complete()
            consumed += 1


# ---- persistent scheduler ----------------------------------------------------------------------

@pytest.mark.parametrize("num_m,num_n,group", [(1, 1, 8), (64, 32, 8), (24, 20, 8), (7, 5, 3),
                                               (13, 1, 8), (1, 13, 8), (128, 56, 16)])
def test_tile_order_is_a_bijection(num_m, num_n, group):
    seen = set()
    for t in range(num_m * num_n):
        m, n = g.gemm_f16_tile_coord(t, num_m, num_n, group)
        assert 0 <= m < num_m and 0 <= n < num_n
        seen.add((m, n))
    assert len(seen) == num_m * num_n


def test_tile_order_groups_walk_m_within_a_column():
    num_m, num_n, group = 64, 32, 8
    coords = [g.gemm_f16_tile_coord(t, num_m, num_n, group) for t in range(num_m * num_n)]
    for t in range(0, len(coords), group):
        block = coords[t:t + group]
        assert len({n for _, n in block}) == 1                 # one N column ...
        assert [m for m, _ in block] == list(range(block[0][0], block[0][0] + group))  # ... 8 M rows


def test_persistent_schedule_covers_every_tile_once():
    """Static persistent schedule: unit c takes tiles c, c + units, ...; every tile exactly once."""
    num_m, num_n, units = 24, 20, 152
    tiles = num_m * num_n
    hits = [0] * tiles
    for c in range(units):
        for t in range(c, tiles, units):
            hits[t] += 1
    assert hits == [1] * tiles


def test_choose_variant_returns_a_variant():
    for (M, N, K) in [(128, 128, 64), (2048, 2048, 2048), (3000, 5000, 1000), (8192, 8192, 8192),
                      (16384, 14336, 4096), (1, 8, 8), (100000, 8, 8)]:
        v = g.gemm_f16_choose_variant(M, N, K, 152)
        assert v in (1, 2, 3, 4)


def test_choose_variant_on_the_workloads():
    """The automatic choice on a 152-SM GB300 for the five workloads: the one-tile kernel for the
    single tile (short K, a grid of at most one wave), the 256 x 256 CTA pair for every other
    (2048^3 has 64 pair tiles: at least half the SMs), and 128 x 256 / 128 x 128 for shapes too
    short for a pair."""
    pair, w256, w128 = g.VARIANTS["ws_pair"], g.VARIANTS["ws_128x256"], g.VARIANTS["ws_128x128"]
    tile = g.VARIANTS["tile"]
    assert g.gemm_f16_choose_variant(128, 128, 64, 152) == tile
    assert g.gemm_f16_choose_variant(1024, 1024, 256, 152) == tile      # 64 tiles, K = 256
    assert g.gemm_f16_choose_variant(1024, 1024, 512, 152) == w128      # K = 512: the pipeline
    assert g.gemm_f16_choose_variant(2048, 2048, 64, 152) != tile       # 256 tiles: over a wave
    for shape in [(2048, 2048, 2048), (3000, 5000, 1000), (8192, 8192, 8192),
                  (16384, 14336, 4096)]:
        assert g.gemm_f16_choose_variant(*shape, 152) == pair, shape
    assert g.gemm_f16_choose_variant(128, 65536, 4096, 152) == w256     # 256 tiles of 128 x 256
    assert g.gemm_f16_choose_variant(128, 16384, 4096, 152) == w128     # 64: under half the SMs
    assert g.gemm_f16_choose_variant(512, 1024, 4096, 152) == w128      # 8 pair tiles only


# ---- argument checks (return before any CUDA call) ---------------------------------------------

FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced: every case below fails validation


@pytest.mark.parametrize("args,code", [
    ((FAKE, FAKE, FAKE, -1, 8, 8), g.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, 8, -8, 8), g.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, 8, 8, -8), g.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, 1 << 31, 8, 8), g.ERR_INVALID_ARG),
    ((FAKE, FAKE, 0, 8, 8, 8), g.ERR_INVALID_ARG),
    ((0, FAKE, FAKE, 8, 8, 8), g.ERR_INVALID_ARG),
    ((FAKE, 0, FAKE, 8, 8, 8), g.ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, 8, 8, 12), g.ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, 8, 12, 8), g.ERR_UNSUPPORTED),
    ((FAKE + 2, FAKE, FAKE, 8, 8, 8), g.ERR_UNSUPPORTED),
    ((FAKE, FAKE + 8, FAKE, 8, 8, 8), g.ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE + 4, 8, 8, 8), g.ERR_UNSUPPORTED),
])
def test_argument_checks(args, code):
    assert g.gemm_f16_nt(*args, 0) == code
    assert g.gemm_f16_last_error() != ""


def test_empty_output_is_a_no_op():
    # M == 0 or N == 0: nothing to do, no pointer is touched, no CUDA call is made
    assert g.gemm_f16_nt(0, 0, 0, 0, 8, 8, 0) == g.OK
    assert g.gemm_f16_nt(0, 0, 0, 8, 0, 8, 0) == g.OK


def test_unknown_variant_rejected():
    assert g.gemm_f16_nt_variant(FAKE, FAKE, FAKE, 8, 8, 8, 0, 17) == g.ERR_INVALID_ARG
    assert g.gemm_f16_nt_variant(FAKE, FAKE, FAKE, 8, 8, 8, 0, -1) == g.ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """With the extension absent the binding raises; it never computes another way."""
    monkeypatch.setattr(g, "_lib", None)
    monkeypatch.setattr(g, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        g.load()


def test_product_package_does_not_reference_the_oracle():
    pkg = os.path.dirname(g.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "gemm_ref" not in text, f


# ---- stream-K tail: the work split covers every k-block of every tile exactly once ----------

SPLITS = [  # (tiles, units, k_blocks): 8192^3 pairs, MLP pairs, 2048^3 pairs, odd cases
    (1024, 76, 128), (3584, 76, 64), (64, 76, 32), (20, 76, 24), (24, 76, 63), (480, 152, 16),
    (7, 5, 9), (13, 4, 40), (100, 7, 3),
]


@pytest.mark.parametrize("T,U,KB", SPLITS)
def test_stream_k_split_covers_each_k_block_once(T, U, KB):
    R = g.gemm_f16_sk_tail_tiles(T, U, KB)
    for tail in sorted({R, 0}):
        S = min(3 * tail, U)  # units sharing the tail: at most 3 per tail tile
        if tail:
            assert 0 < tail <= U and tail <= T and (T - tail) % U == 0 and tail * KB >= 4 * S
        cover = {}
        per_unit = []
        for c in range(U):
            n = g.gemm_f16_sk_items(T, U, KB, tail, c)
            assert n <= (T - tail) // U + (T - tail) % U + 2 if tail else True
            work = 0
            pieces = 0
            for i in range(n):
                tile, kb0, kb1, piece, partial = g.gemm_f16_sk_item(T, U, KB, tail, c, i)
                assert 0 <= tile < T and 0 <= kb0 < kb1 <= KB
                if tile < T - tail:
                    assert (kb0, kb1, partial) == (0, KB, 0)
                else:
                    assert piece == pieces and piece <= 1
                    pieces += 1
                    assert partial == int(not (kb0 == 0 and kb1 == KB))
                    r = tile - (T - tail)
                    # every k-block of this piece is in unit c's range
                    for kb in (kb0, kb1 - 1):
                        assert g.gemm_f16_sk_unit_of(T, U, KB, tail, r * KB + kb) == c
                for kb in range(kb0, kb1):
                    cover[(tile, kb)] = cover.get((tile, kb), 0) + 1
                work += kb1 - kb0
            per_unit.append(work)
        assert len(cover) == T * KB and set(cover.values()) == {1}
        if tail:
            assert max(per_unit[:S]) - min(per_unit[:S]) <= 1   # balanced to one k-block
            assert max(per_unit[S:], default=0) <= min(per_unit[:S])
            for r in range(tail):  # at most 4 contributors per tail tile
                u0 = g.gemm_f16_sk_unit_of(T, U, KB, tail, r * KB)
                u1 = g.gemm_f16_sk_unit_of(T, U, KB, tail, r * KB + KB - 1)
                assert 0 <= u0 <= u1 < S and u1 - u0 + 1 <= 4
        else:
            assert max(per_unit) - min(per_unit) <= KB  # at most one tile apart


def test_raster_group_rule():
    if "GEMM_F16_GROUP" in os.environ:
        pytest.skip("GEMM_F16_GROUP overrides the rule in this process")
    l2 = 126 << 20                                                  # a GB300's L2
    assert g.gemm_f16_raster_group(256, 8192, 2, l2) == 8          # 8192^3 pair tiles
    assert g.gemm_f16_raster_group(256, 4096, 2, l2) == 16         # 16384x14336x4096
    assert g.gemm_f16_raster_group(128, 8192, 2, l2) == 16         # 128-row tiles
    assert g.gemm_f16_raster_group(256, 8192, 1, l2) == 16         # fp8: one byte per element
    assert g.gemm_f16_raster_group(256, 65536, 2, l2) == 1         # one band already over L2/3
    assert g.gemm_f16_raster_group(256, 64, 2, l2) == 16           # capped at 16
    for K in (64, 512, 4096, 8192, 16384, 32768):                  # the invariant itself
        G = g.gemm_f16_raster_group(256, K, 2, l2)
        assert G in (1, 2, 4, 8, 16)
        assert G == 1 or G * 256 * K * 2 * 3 <= l2
        assert G == 16 or 2 * G * 256 * K * 2 * 3 > l2


def test_stream_k_tail_choice():
    assert g.gemm_f16_sk_tail_tiles(1024, 76, 128) == 36      # 8192^3: 13.47 waves of pairs
    assert g.gemm_f16_sk_tail_tiles(3584, 76, 64) == 12       # MLP: 47.16 waves
    assert g.gemm_f16_sk_tail_tiles(64, 76, 32) == 64         # 2048^3: under one wave
    assert g.gemm_f16_sk_tail_tiles(76 * 5, 76, 64) == 0      # whole waves
    assert g.gemm_f16_sk_tail_tiles(76 * 5 + 75, 76, 64) == 0  # last wave 99% full
    assert g.gemm_f16_sk_tail_tiles(240, 76, 16) == 12        # 12 tiles over 36 units
    assert g.gemm_f16_sk_tail_tiles(240, 76, 3) == 0          # pieces under 4 k-blocks


SK_HEADER = 8192                         # stream-K workspace header (flags and bookkeeping)
SK_FLAG_BASE, SK_FLAG_WORDS = 64, (8192 // 4 - 64) // 2
MAX_CONTRIB = 4


def test_noalloc_scratch_holds_every_gb300_workspace():
    """The allocation-free entry point's fixed array (40 MiB) holds the largest stream-K
    workspace any variant requests on a 152-SM GB300: an 8 KiB header plus one 128 x 256 fp32
    slot per CTA (76 pairs or 152 single CTAs).  A device whose request would not fit (here a
    hypothetical 400-SM part) is served by the data-parallel schedule, which needs none."""
    cap = g.gemm_f16_noalloc_scratch_bytes()
    assert cap == 40 << 20
    per_cta = 128 * 256 * 4
    assert SK_HEADER + 152 * per_cta <= cap       # 19 MiB: 1-CTA 128x256 or 76 CTA pairs
    assert SK_HEADER + 400 * per_cta > cap        # would take the no-workspace path


def test_stream_k_switch():
    assert g.gemm_f16_set_stream_k(2) == g.ERR_INVALID_ARG
    assert g.gemm_f16_set_stream_k(-1) == g.ERR_INVALID_ARG
    assert g.gemm_f16_set_stream_k(1) == g.OK
    assert g.gemm_f16_set_stream_k(0) == g.OK


def test_failure_hooks_validate_arguments():
    assert g.gemm_f16_set_wait_timeout_ms(0) == g.ERR_INVALID_ARG
    assert g.gemm_f16_set_fault_injection(2) == g.ERR_INVALID_ARG
    assert g.gemm_f16_set_fault_injection(-1) == g.ERR_INVALID_ARG
    assert g.gemm_f16_set_fault_injection(0) == g.OK
    assert g.gemm_f16_set_wait_timeout_ms(4000) == g.OK


# ---- code-generation records: no stack frame, no spills -------------------------------------

def test_every_kernel_compiles_without_stack_or_spills():
    """The page "TIRx" (zixuwang.me), section "验证如何支撑结论", keeps code-generation records
    with zero spills and a zero stack among its validation checks.  The same record here: ptxas
    reports, for every function of the library (each kernel instance and each non-inlined
    helper), a zero-byte stack frame and no spill stores or loads, so no kernel touches local
    memory.  Compiles into a temporary directory; needs nvcc, not a GPU."""
    from blackwell_tensor_core_fp16_gb300 import _build
    report = _build.ptxas_report()
    names = " ".join(report)
    for kernel in ("gemm_ws_kernel", "gemm_tile_kernel", "mx_pack_scales_kernel",
                   "gdn_scan_kernel", "gdn_prepare_kernel", "gdn_chunk_list_kernel"):
        assert kernel in names, f"ptxas reported no {kernel}"
    for name, r in report.items():
        assert {"stack", "spill_stores", "spill_loads"} <= r.keys(), f"no record for {name}"
        assert (r["stack"], r["spill_stores"], r["spill_loads"]) == (0, 0, 0), (name, r)
        if r.get("entry"):
            assert 0 < r["registers"] <= 255, (name, r)


# ---- the persistent kernels' address arithmetic, replayed on the CPU ---------------------------
# A stand-in for a memory checker (none runs on this hardware here): the coordinates and
# workspace offsets gemm_ws_kernel computes, rebuilt from the library's own scheduling functions
# for every variant and workload shape, must stay inside what the launch provides, and the
# output boxes must cover D exactly once.

GB300_L2 = 126 << 20


def _replay(variant, M, N, K, units, stream_k):
    info = g.gemm_f16_get_variant_info(variant)
    cg, mma_m, bn = info["cta_group"], info["block_m"], info["block_n"]
    b_rows = bn // cg
    num_m, num_n, KB = -(-M // mma_m), -(-N // bn), -(-K // 64)
    T = num_m * num_n
    R = g.gemm_f16_sk_tail_tiles(T, units, KB) if stream_k else 0
    used = units if R else min(T, units)
    ws_bytes = SK_HEADER + units * cg * 128 * bn * 4         # the header's workspace size
    part_bytes = 128 * bn * 4
    if R:
        assert R * MAX_CONTRIB * cg <= SK_FLAG_WORDS             # the host's flag bound
    group = g.gemm_f16_raster_group(mma_m, K, 2, GB300_L2)
    stores = {}
    parked = {}       # tail tile -> units that parked partial sums for it (one slot per unit)
    finished = {}     # tail tile -> the unit whose piece starts it and stores it
    for c in range(used):
        n_items = g.gemm_f16_sk_items(T, used, KB, R, c)
        for i in range(n_items):
            tile, kb0, kb1, piece, partial = g.gemm_f16_sk_item(T, used, KB, R, c, i)
            m_blk, n_blk = g.gemm_f16_tile_coord(tile, num_m, num_n, group)
            assert m_blk < num_m and n_blk < num_n
            assert 0 <= kb0 < kb1 <= KB and (kb0 * 64 * 2) % 16 == 0   # TMA x: 16-byte aligned
            r = tile - (T - R)
            if partial:
                u0 = g.gemm_f16_sk_unit_of(T, used, KB, R, r * KB)
                u1 = g.gemm_f16_sk_unit_of(T, used, KB, R, r * KB + KB - 1)
                assert u0 <= c <= u1 and u1 - u0 < MAX_CONTRIB
                for rank in range(cg):        # this piece's flag stays inside its region
                    assert (r * MAX_CONTRIB + (c - u0)) * cg + rank < SK_FLAG_WORDS
                if kb0 != 0:
                    # parks: the unit's first stream-K piece (after any data-parallel tiles,
                    # which wait for nothing either), into the unit's one slot
                    assert piece == 0
                    assert c not in {u for us in parked.values() for u in us}
                    parked.setdefault(r, set()).add(c)
                    for rank in range(cg):
                        assert SK_HEADER + ((c * cg + rank) + 1) * part_bytes <= ws_bytes
                    continue
                # finishes: the unit's last piece (so it waits only for first pieces)
                assert i == n_items - 1 and c == u0
                finished[r] = c
            for rank in range(cg):
                m0 = m_blk * mma_m + rank * 128
                assert m0 >= 0 and n_blk * bn + rank * b_rows >= 0    # load boxes
                for ch in range(bn // 64):
                    col0 = n_blk * bn + 64 * ch
                    if col0 < N and m0 < M:                           # stores never start outside
                        assert (col0 * 2) % 16 == 0
                        stores[(m0, col0)] = stores.get((m0, col0), 0) + 1
    # the piece that finishes tail tile r reads the slots of units u0 + 1 .. u1: exactly the
    # units that parked partial sums for it
    for r, u0 in finished.items():
        u1 = g.gemm_f16_sk_unit_of(T, used, KB, R, r * KB + KB - 1)
        assert parked.get(r, set()) == set(range(u0 + 1, u1 + 1))
    expect = {(128 * i, 64 * j) for i in range(-(-M // 128)) for j in range(-(-N // 64))}
    assert set(stores) == expect and set(stores.values()) == {1}


@pytest.mark.parametrize("variant", [2, 3, 4, 5, 6])
@pytest.mark.parametrize("shape", [(128, 128, 64), (2048, 2048, 2048), (3000, 5000, 1000),
                                   (8192, 8192, 8192), (16384, 14336, 4096), (129, 136, 72)],
                         ids=lambda s: "x".join(map(str, s)))
def test_kernel_addresses_stay_in_bounds_and_cover_d_once(variant, shape):
    M, N, K = shape
    units = 152 // g.gemm_f16_get_variant_info(variant)["cta_group"]
    for u in (units, units - 3):          # fewer co-resident units than SMs allow
        for stream_k in (False, True):
            _replay(variant, M, N, K, u, stream_k)


# ---- the half-width tail, replayed on the CPU --------------------------------------------------

def _replay_half(variant, M, N, K, units):
    """The items and boxes of a launch whose last partial wave runs as half-width items (no
    stream-K): every output box is stored once, every B box starts at an aligned column, and the
    half items cover the tail tiles' two halves exactly."""
    info = g.gemm_f16_get_variant_info(variant)
    cg, mma_m, bn = info["cta_group"], info["block_m"], info["block_n"]
    b_rows = bn // cg
    num_m, num_n, KB = -(-M // mma_m), -(-N // bn), -(-K // 64)
    T = num_m * num_n
    H = g.gemm_f16_half_tail_tiles(T, units) if (bn // 2) % 64 == 0 else 0
    if H == 0:
        return 0
    assert 2 * H <= units and (T - H) % units == 0
    used = 2 * H if T == H else units                 # the launch's grid, in units
    group = g.gemm_f16_raster_group(mma_m, K, 2, GB300_L2)
    stores, halves = {}, {}
    for c in range(used):
        for i in range(g.gemm_f16_half_items(T, used, KB, H, c)):
            tile, kb0, kb1, half = g.gemm_f16_half_item(T, used, KB, H, c, i)
            assert (kb0, kb1) == (0, KB)
            assert (half == 0) == (tile < T - H), (tile, half)
            m_blk, n_blk = g.gemm_f16_tile_coord(tile, num_m, num_n, group)
            assert m_blk < num_m and n_blk < num_n
            width = bn if half == 0 else bn // 2
            col_base = n_blk * bn + (half - 1) * (bn // 2 if half else 0)
            if half:
                halves.setdefault(tile, []).append(half)
            for rank in range(cg):
                m0 = m_blk * mma_m + rank * 128
                b0 = col_base + rank * (b_rows if half == 0 else b_rows // 2)
                assert b0 >= 0                                   # B box row
                for ch in range(width // 64):
                    col0 = col_base + 64 * ch
                    if col0 < N and m0 < M:
                        assert (col0 * 2) % 16 == 0
                        stores[(m0, col0)] = stores.get((m0, col0), 0) + 1
    assert sorted(halves) == list(range(T - H, T))
    assert all(sorted(h) == [1, 2] for h in halves.values())
    expect = {(128 * i, 64 * j) for i in range(-(-M // 128)) for j in range(-(-N // 64))}
    assert set(stores) == expect and set(stores.values()) == {1}
    return H


@pytest.mark.parametrize("variant", [2, 3, 4, 5])
@pytest.mark.parametrize("shape", [(8192, 8192, 8192), (16384, 14336, 4096), (3000, 5000, 1000),
                                   (2048, 2048, 2048), (512, 1024, 4096), (129, 136, 72)],
                         ids=lambda s: "x".join(map(str, s)))
def test_half_width_tail_covers_d_once(variant, shape):
    M, N, K = shape
    units = 152 // g.gemm_f16_get_variant_info(variant)["cta_group"]
    for u in (units, units - 3):
        _replay_half(variant, M, N, K, u)


def test_half_width_tail_rule():
    assert g.gemm_f16_half_tail_tiles(1024, 76) == 36       # 8192^3 pairs: 13 waves + 36
    assert g.gemm_f16_half_tail_tiles(3584, 76) == 12       # the MLP shape
    assert g.gemm_f16_half_tail_tiles(64, 76) == 0          # 2048^3: 128 halves would not fit
    assert g.gemm_f16_half_tail_tiles(8, 76) == 8           # few tiles: all of them halved
    assert g.gemm_f16_half_tail_tiles(152, 76) == 0         # whole waves
    assert g.gemm_f16_half_tail_tiles(76 + 39, 76) == 0     # 2 x 39 > 76


def test_gelu_erfc_fit_accuracy_in_fp32():
    """The fused epilogue's GELU evaluates erfc with the Chebyshev fit of Numerical Recipes
    (section 6.2): erfc(z) = t exp(-z^2 + P(t)), t = 1 / (1 + z/2), for z >= 0, and
    Phi(x) = 1 - erfc(|x|/sqrt2)/2 (x >= 0) or erfc(|x|/sqrt2)/2 (x < 0).  The same steps in
    float32 stay within 2e-7 (plus one fp32 rounding of the result) of the exact GELU (binary64
    math.erfc) for |x| <= 10, and within 5e-6 relative for |x| <= 6; a wrong or missing
    coefficient breaks both."""
    import math
    import numpy as np
    f32 = np.float32
    coef = [-1.26551223, 1.00002368, 0.37409196, 0.09678418, -0.18628806, 0.27886807,
            -1.13520398, 1.48851587, -0.82215223, 0.17087277]
    x = np.concatenate([np.linspace(-10, 10, 40001), np.linspace(-1e-3, 1e-3, 201)]).astype(f32)
    z = np.abs(x) * f32(0.70710678118654752)
    t = f32(1) / (f32(0.5) * z + f32(1))
    p = np.full_like(t, f32(coef[9]))
    for c in coef[8::-1]:
        p = p * t + f32(c)
    e = t * np.exp(-z * z + p)
    got = x * np.where(x >= 0, f32(1) - f32(0.5) * e, f32(0.5) * e)
    xd = x.astype(np.float64)
    ref = np.array([v * 0.5 * math.erfc(-v / math.sqrt(2.0)) for v in xd])
    err = np.abs(got.astype(np.float64) - ref)
    bound = 2e-7 + 2.0 ** -23 * np.abs(ref)   # plus one fp32 rounding of the result
    assert (err <= bound).all(), float((err / bound).max())
    mid = (np.abs(xd) <= 6) & (ref != 0)
    assert (err[mid] / np.abs(ref[mid])).max() < 5e-6
