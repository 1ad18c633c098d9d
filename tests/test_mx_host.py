"""Host-side checks of the block-scaled FP8 path (no GPU): encoders, the scale layout, budgets."""
from __future__ import annotations

import numpy as np
import pytest

import blackwell_tensor_core_fp16_gb300 as g


@pytest.fixture(scope="module", autouse=True)
def library():
    g.build()
    g.load()


def _fields(idesc):
    return {"b_sf_id": (idesc >> 4) & 3, "a_fmt": (idesc >> 7) & 7, "b_fmt": (idesc >> 10) & 7,
            "a_major": (idesc >> 15) & 1, "b_major": (idesc >> 16) & 1,
            "n": ((idesc >> 17) & 0x3F) << 3, "scale_e8m0": (idesc >> 23) & 1,
            "m": ((idesc >> 24) & 0x1F) << 4, "a_sf_id": (idesc >> 29) & 3,
            "low": idesc & 0xF, "bit6": (idesc >> 6) & 1, "bit31": idesc >> 31}


@pytest.mark.parametrize("M,N,fa,fb", [(128, 128, 0, 0), (256, 128, 1, 0), (128, 256, 0, 1),
                                       (256, 192, 1, 1)])
def test_mx_idesc_fields(M, N, fa, fb):
    f = _fields(g.gemm_mxf8_idesc(M, N, fa, fb))
    assert (f["m"], f["n"], f["a_fmt"], f["b_fmt"]) == (M, N, fa, fb)
    assert f["scale_e8m0"] == 1
    assert f["a_major"] == f["b_major"] == 0          # both operands K-major
    assert f["a_sf_id"] == f["b_sf_id"] == 0          # the issuer ORs in the K block
    assert f["low"] == 0 and f["bit6"] == 0 and f["bit31"] == 0


def test_mx_idesc_value():
    # E4M3 x E4M3, M = N = 128: N>>3 = 16 at bit 17, E8M0 at bit 23, M>>4 = 8 at bit 24
    assert g.gemm_mxf8_idesc(128, 128, 0, 0) == (16 << 17) | (1 << 23) | (8 << 24) == 0x08A00000


def test_scale_layout_is_the_documented_formula_and_a_bijection():
    for rows, K in ((1, 32), (130, 96), (300, 1056), (257, 4096)):
        kb = K // 32
        kg = (kb + 3) // 4
        total = g.gemm_mxf8_scale_bytes(rows, K)
        assert total == ((rows + 127) // 128) * kg * 512
        seen = set()
        for r in range(rows):
            for b in range(kb):
                off = g.gemm_mxf8_sf_offset(r, b, K)
                want = ((r // 128) * kg + b // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 \
                    + b % 4
                assert off == want
                assert 0 <= off < total
                seen.add(off)
        assert len(seen) == rows * kb


def test_scale_layout_row_of_a_chunk_is_one_lane():
    """The 16 bytes of chunk row l hold rows l, l+32, l+64, l+96 (4 K blocks each): the lane-l
    row of a 32 x 128-bit tensor-memory copy, column q = rows 32q + l."""
    K = 128
    for l in (0, 5, 31):
        offs = sorted(g.gemm_mxf8_sf_offset(32 * q + l, b, K) for q in range(4) for b in range(4))
        assert offs == list(range(16 * l, 16 * l + 16))
        for q in range(4):
            for b in range(4):
                assert g.gemm_mxf8_sf_offset(32 * q + l, b, K) == 16 * l + 4 * q + b


def test_scale_bytes_rejects_bad_k():
    assert g.gemm_mxf8_scale_bytes(10, 48) == -1
    assert g.gemm_mxf8_scale_bytes(-1, 64) == -1
    assert g.gemm_mxf8_scale_bytes(0, 64) == 0
    assert g.gemm_mxf8_sf_offset(0, 2, 64) == -1      # block past K/32


def test_sf_desc_fields():
    for addr in (0, 0x400, 0x1F200):
        d = g.gemm_mxf8_sf_desc(addr)
        assert d & 0x3FFF == (addr & 0x3FFFF) >> 4
        assert (d >> 16) & 0x3FFF == 128 >> 4           # 8-row core matrices 128 bytes apart
        assert (d >> 32) & 0x3FFF == 128 >> 4
        assert (d >> 46) & 7 == 1                       # descriptor version
        assert d >> 61 == 0                             # no swizzle


@pytest.mark.parametrize("variant", [1, 2, 3, 4])
def test_variant_budgets(variant):
    info = g.gemm_mxf8_get_variant_info(variant)
    assert info["smem_bytes"] <= 232448
    assert info["tmem_cols"] == 512
    bn, stages, cg = info["block_n"], info["stages"], info["cta_group"]
    chunks = bn // 128 if bn % 128 == 0 else bn // 128 + 1
    accs = 1 if bn == 256 else 2
    assert accs * bn + stages * 4 * (1 + chunks) <= 512  # accumulators + scale ring
    # a stage: A 128 x 128 B, B (bn / cg) x 128 B, scale chunks of 512 B, per CTA
    assert info["stage_tx_bytes"] == cg * (128 * 128 + (bn // cg) * 128 + 512 * (1 + chunks))
    assert info["block_k"] == 128


def test_choose_variant():
    assert g.gemm_mxf8_choose_variant(128, 128, 128, 152) == 1
    assert g.gemm_mxf8_choose_variant(2048, 2048, 2048, 152) == 4
    assert g.gemm_mxf8_choose_variant(8192, 8192, 8192, 152) == 4
    assert g.gemm_mxf8_choose_variant(16384, 14336, 4096, 152) == 4


def test_rejects_before_touching_the_gpu():
    # K not a multiple of the scale block and unknown formats are refused by the argument checks
    assert g.gemm_mxf8_nt(16, 16, 16, 16, 16, 128, 128, 48, 0, 0, 0, 0, 0, 0, 0, 0, 0) \
        == g.ERR_UNSUPPORTED
    assert g.gemm_mxf8_nt(16, 16, 16, 16, 16, 128, 128, 64, 3, 0, 0, 0, 0, 0, 0, 0, 0) \
        == g.ERR_INVALID_ARG
    assert g.gemm_mxf8_nt(16, 16, 0, 16, 16, 128, 128, 64, 0, 0, 0, 0, 0, 0, 0, 0, 0) \
        == g.ERR_INVALID_ARG
    assert g.gemm_mxf8_nt(16, 16, 16, 16, 16, -1, 128, 64, 0, 0, 0, 0, 0, 0, 0, 0, 0) \
        == g.ERR_INVALID_ARG
    assert g.gemm_mxf8_nt(16, 16, 16, 16, 16, 0, 128, 64, 0, 0, 0, 0, 0, 0, 0, 0, 0) == g.OK
    assert g.gemm_mxf8_nt(16, 16, 16, 16, 16, 128, 128, 64, 0, 0, 0, 0, 0, 7, 0, 0, 0) \
        == g.ERR_INVALID_ARG


@pytest.mark.parametrize("variant", [1, 2, 3, 4])
def test_b_scales_of_every_n_tile_fit_the_stage_slot(variant):
    """A stage loads `chunks` 128-row groups of B's scales, starting with the group that holds
    the tile's first row, into 4 tensor-memory columns per group after A's 4 (32 rows per
    column).  An N tile that starts inside a group (192-wide tiles start 64 rows in on every
    other tile) reads its scales from a column (rows into the group) / 32 further on.  For every
    tile position: the tile's rows lie in the groups the stage loads, and the columns the MMA
    reads stay inside the stage's slot."""
    info = g.gemm_mxf8_get_variant_info(variant)
    bn = info["block_n"]
    chunks = bn // 128 if bn % 128 == 0 else bn // 128 + 1
    slot_cols = 4 * (1 + chunks)
    for n_blk in range(64):
        row0 = n_blk * bn
        first_group, last_group = row0 // 128, (row0 + bn - 1) // 128
        assert last_group - first_group + 1 <= chunks
        shift = (row0 % 128) // 32
        assert 4 + shift + bn // 32 <= slot_cols
