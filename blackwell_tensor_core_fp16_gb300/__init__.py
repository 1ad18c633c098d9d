"""GB300-native fp16 GEMM: D = A * B^T (A: M x K, B: N x K, fp16 row-major; fp32 accumulation;
D: M x N fp16), computed by the hand-written sm_103a kernels of ``libgemm_f16.so``.

This module is a thin ctypes binding over the C ABI in ``include/gemm_f16.h``: the functions
named ``gemm_f16_*`` take plain integers (device pointers, sizes, a stream handle) exactly as
the C functions do, and ``gemm()`` marshals torch tensors into them.  Every step of the
computation runs in the CUDA library; there is no other code path.  If the library has not
been built, every call raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import re
import threading

from . import _build

__all__ = [
    "GemmError", "build", "load", "gemm", "check_status",
    "gemm_f16_nt", "gemm_f16_nt_variant", "gemm_f16_choose_variant", "gemm_f16_check_status",
    "gemm_f16_last_error", "gemm_f16_version", "gemm_f16_get_variant_info", "gemm_f16_idesc",
    "gemm_f16_smem_desc_sw128", "gemm_f16_sw128", "gemm_f16_tile_coord", "gemm_f16_ring_pos",
    "gemm_f16_nt_ws", "gemm_f16_nt_ex", "gemm_f16_nt_noalloc", "gemm_f16_noalloc_scratch_bytes",
    "gemm_f16_workspace_bytes",
    "gemm_f16_nt_fused", "linear", "DTYPES", "ACTIVATIONS", "gemm_f16_set_wait_timeout_ms",
    "gemm_f16_set_fault_injection",
    "gemm_f16_sk_tail_tiles", "gemm_f16_raster_group", "gemm_f16_set_stream_k",
    "gemm_f16_sk_items", "gemm_f16_sk_item", "gemm_f16_sk_unit_of",
    "gemm_f16_half_tail_tiles", "gemm_f16_half_items", "gemm_f16_half_item",
    "exported_symbols", "VARIANTS", "STATUS",
]

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA_ERROR", 4: "TIMEOUT"}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4
VARIANTS = {"auto": 0, "tile": 1, "ws_128x256": 2, "ws_pair": 3, "ws_128x128": 4,
            "ws_pair_direct": 5, "ws_pair_256x192": 6}

build = _build.build
LIB_PATH = _build.LIB_PATH

_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"gemm_f16 status {code} ({STATUS.get(code, '?')}): {message}")
        self.code = code


class VariantInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "cta_group", "block_m", "block_n", "block_k", "stages", "threads", "smem_bytes",
        "tmem_cols", "stage_tx_bytes", "persistent")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


def load():
    """Load libgemm_f16.so (raises RuntimeError if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        import os
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(blackwell_tensor_core_fp16_gb300.build()); there is no fallback path")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, u32, u64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32,
                                  ctypes.c_uint64)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        lib.gemm_f16_nt.argtypes = [vp, vp, vp, i64, i64, i64, vp]
        lib.gemm_f16_nt.restype = i32
        lib.gemm_f16_nt_variant.argtypes = [vp, vp, vp, i64, i64, i64, vp, i32]
        lib.gemm_f16_nt_variant.restype = i32
        lib.gemm_f16_choose_variant.argtypes = [i64, i64, i64, i32]
        lib.gemm_f16_choose_variant.restype = i32
        lib.gemm_f16_check_status.argtypes = [vp, u32p]
        lib.gemm_f16_check_status.restype = i32
        lib.gemm_f16_last_error.argtypes = []
        lib.gemm_f16_last_error.restype = ctypes.c_char_p
        lib.gemm_f16_version.argtypes = []
        lib.gemm_f16_version.restype = i32
        lib.gemm_f16_get_variant_info.argtypes = [i32, ctypes.POINTER(VariantInfo)]
        lib.gemm_f16_get_variant_info.restype = i32
        lib.gemm_f16_idesc.argtypes = [u32, u32, u32]
        lib.gemm_f16_idesc.restype = u32
        lib.gemm_f16_smem_desc_sw128.argtypes = [u32, u32]
        lib.gemm_f16_smem_desc_sw128.restype = u64
        lib.gemm_f16_sw128.argtypes = [u32]
        lib.gemm_f16_sw128.restype = u32
        lib.gemm_f16_tile_coord.argtypes = [u32, u32, u32, u32, u32p, u32p]
        lib.gemm_f16_tile_coord.restype = None
        lib.gemm_f16_ring_pos.argtypes = [u32, u32, u32p, u32p]
        lib.gemm_f16_ring_pos.restype = None
        sz = ctypes.c_size_t
        lib.gemm_f16_nt_ws.argtypes = [vp, vp, vp, i64, i64, i64, vp, sz, vp]
        lib.gemm_f16_nt_ws.restype = i32
        lib.gemm_f16_nt_ex.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp, sz, vp]
        lib.gemm_f16_nt_ex.restype = i32
        lib.gemm_f16_nt_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, vp]
        lib.gemm_f16_nt_noalloc.restype = i32
        lib.gemm_f16_noalloc_scratch_bytes.argtypes = []
        lib.gemm_f16_noalloc_scratch_bytes.restype = sz
        lib.gemm_f16_nt_fused.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp, i32, i32, vp, sz,
                                          vp]
        lib.gemm_f16_nt_fused.restype = i32
        lib.gemm_f16_set_wait_timeout_ms.argtypes = [u32]
        lib.gemm_f16_set_wait_timeout_ms.restype = i32
        lib.gemm_f16_set_fault_injection.argtypes = [i32]
        lib.gemm_f16_set_fault_injection.restype = i32
        lib.gemm_f16_workspace_bytes.argtypes = [i64, i64, i64, i32, ctypes.POINTER(sz)]
        lib.gemm_f16_workspace_bytes.restype = i32
        lib.gemm_f16_sk_tail_tiles.argtypes = [i64, i64, i64]
        lib.gemm_f16_sk_tail_tiles.restype = i64
        lib.gemm_f16_set_stream_k.argtypes = [i32]
        lib.gemm_f16_set_stream_k.restype = i32
        lib.gemm_f16_raster_group.argtypes = [i64, i64, i64, i64]
        lib.gemm_f16_raster_group.restype = u32
        lib.gemm_f16_sk_items.argtypes = [u32, u32, u32, u32, u32]
        lib.gemm_f16_sk_items.restype = u32
        lib.gemm_f16_sk_item.argtypes = [u32, u32, u32, u32, u32, u32, u32p]
        lib.gemm_f16_sk_item.restype = None
        lib.gemm_f16_sk_unit_of.argtypes = [u32, u32, u32, u32, u32]
        lib.gemm_f16_sk_unit_of.restype = u32
        lib.gemm_f16_half_tail_tiles.argtypes = [i64, i64]
        lib.gemm_f16_half_tail_tiles.restype = i64
        lib.gemm_f16_half_items.argtypes = [u32, u32, u32, u32, u32]
        lib.gemm_f16_half_items.restype = u32
        lib.gemm_f16_half_item.argtypes = [u32, u32, u32, u32, u32, u32, u32p]
        lib.gemm_f16_half_item.restype = None
        lib.gemm_mxf8_nt.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, i32, vp, i32,
                                     i32, vp, sz, vp]
        lib.gemm_mxf8_nt.restype = i32
        lib.gemm_mxf8_workspace_bytes.argtypes = [i64, i64, i64, i32, ctypes.POINTER(sz)]
        lib.gemm_mxf8_workspace_bytes.restype = i32
        lib.gemm_mxf8_choose_variant.argtypes = [i64, i64, i64, i32]
        lib.gemm_mxf8_choose_variant.restype = i32
        lib.gemm_mxf8_scale_bytes.argtypes = [i64, i64]
        lib.gemm_mxf8_scale_bytes.restype = i64
        lib.gemm_mxf8_pack_scales.argtypes = [vp, vp, i64, i64, vp]
        lib.gemm_mxf8_pack_scales.restype = i32
        lib.gemm_mxf8_idesc.argtypes = [u32, u32, u32, u32]
        lib.gemm_mxf8_idesc.restype = u32
        lib.gemm_mxf8_sf_offset.argtypes = [i64, i64, i64]
        lib.gemm_mxf8_sf_offset.restype = i64
        lib.gemm_mxf8_sf_desc.argtypes = [u32]
        lib.gemm_mxf8_sf_desc.restype = ctypes.c_uint64
        lib.gemm_mxf8_get_variant_info.argtypes = [i32, ctypes.POINTER(VariantInfo)]
        lib.gemm_mxf8_get_variant_info.restype = i32
        lib.gdn_prefill_workspace_bytes.argtypes = [i64, i64, i64, ctypes.POINTER(sz)]
        lib.gdn_prefill_workspace_bytes.restype = i32
        lib.gdn_prefill.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                    ctypes.c_float, vp, vp, vp, vp, sz, vp]
        lib.gdn_prefill.restype = i32
        lib.gdn_prefill_heads.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                          ctypes.c_float, vp, vp, vp, vp, sz, vp]
        lib.gdn_prefill_heads.restype = i32
        lib.gdn_last_error.argtypes = []
        lib.gdn_last_error.restype = ctypes.c_char_p
        lib.gdn_check_status.argtypes = [vp, vp]
        lib.gdn_check_status.restype = i32
        lib.gdn_check_offsets.argtypes = [vp, i64, i64, i64, vp, sz, vp]
        lib.gdn_check_offsets.restype = i32
        lib.gdn_offsets_valid_host.argtypes = [ctypes.POINTER(ctypes.c_int32), i64, i64]
        lib.gdn_offsets_valid_host.restype = i32
        lib.gdn_set_wait_timeout_ms.argtypes = [u32]
        lib.gdn_set_wait_timeout_ms.restype = i32
        lib.gdn_set_scan_kernel.argtypes = [i32]
        lib.gdn_set_scan_kernel.restype = i32
        lib.gdn_set_fault_injection.argtypes = [i32]
        lib.gdn_set_fault_injection.restype = i32
        _lib = lib
        return lib


# ---- the C ABI, one Python function per C function -------------------------------------------

def gemm_f16_nt(A: int, B: int, D: int, M: int, N: int, K: int, stream: int = 0) -> int:
    return load().gemm_f16_nt(A, B, D, M, N, K, stream)


def gemm_f16_nt_variant(A: int, B: int, D: int, M: int, N: int, K: int, stream: int,
                        variant: int) -> int:
    return load().gemm_f16_nt_variant(A, B, D, M, N, K, stream, variant)


def gemm_f16_nt_ws(A: int, B: int, D: int, M: int, N: int, K: int, workspace: int,
                   workspace_bytes: int, stream: int = 0) -> int:
    return load().gemm_f16_nt_ws(A, B, D, M, N, K, workspace, workspace_bytes, stream)


def gemm_f16_nt_ex(A: int, B: int, D: int, M: int, N: int, K: int, variant: int,
                   workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    return load().gemm_f16_nt_ex(A, B, D, M, N, K, variant, workspace, workspace_bytes, stream)


DTYPES = {"f16": 0, "bf16": 1}
ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2}


def gemm_f16_nt_fused(A: int, B: int, D: int, M: int, N: int, K: int, dtype: int, bias: int,
                      activation: int, variant: int, workspace: int, workspace_bytes: int,
                      stream: int = 0) -> int:
    return load().gemm_f16_nt_fused(A, B, D, M, N, K, dtype, bias, activation, variant,
                                    workspace, workspace_bytes, stream)


def linear(A, W, bias=None, activation: str = "none", out=None, variant: int = 0, stream=None):
    """act(A @ W.T + bias) for CUDA fp16 or bfloat16 tensors A (M, K), W (N, K), bias (N,);
    returns (M, N) in the same type.  The bias add and the activation run in the GEMM's epilogue
    on the fp32 sums.  Asynchronous on ``stream``; raises GemmError on a non-zero status."""
    import torch
    dt = {torch.float16: "f16", torch.bfloat16: "bf16"}.get(A.dtype)
    if dt is None or W.dtype != A.dtype or (bias is not None and bias.dtype != A.dtype):
        raise ValueError("A, W and bias must all be float16 or all bfloat16")
    for name, t in (("A", A), ("W", W)):
        if not t.is_cuda or t.dim() != 2 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 2-D CUDA tensor")
    M, K = A.shape
    N, K2 = W.shape
    if K2 != K:
        raise ValueError("K differs")
    if bias is not None and (bias.numel() != N or not bias.is_cuda or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous CUDA vector of N elements")
    if out is None:
        out = torch.empty((M, N), dtype=A.dtype, device=A.device)
    elif (out.dtype != A.dtype or not out.is_cuda or tuple(out.shape) != (M, N)
          or not out.is_contiguous()):
        raise ValueError("out must be a contiguous (M, N) CUDA tensor of A's dtype")
    dev = _one_device(("A", A), ("W", W), ("bias", bias), ("out", out))
    with torch.cuda.device(dev):
        rc = gemm_f16_nt_fused(A.data_ptr(), W.data_ptr(), out.data_ptr(), M, N, K, DTYPES[dt],
                               0 if bias is None else bias.data_ptr(), ACTIVATIONS[activation],
                               int(variant), 0, 0, _stream_handle(stream))
    if rc != OK:
        raise GemmError(rc, gemm_f16_last_error())
    return out


def gemm_f16_nt_noalloc(A: int, B: int, D: int, M: int, N: int, K: int, stream: int = 0) -> int:
    """D = A * B^T using the library's fixed device scratch instead of any allocation (for
    callers that cannot allocate, e.g. a server whose device memory all belongs to its own pool);
    see include/gemm_f16.h."""
    return load().gemm_f16_nt_noalloc(A, B, D, M, N, K, stream)


def gemm_f16_noalloc_scratch_bytes() -> int:
    """Size of the fixed device array gemm_f16_nt_noalloc uses (host-only)."""
    return int(load().gemm_f16_noalloc_scratch_bytes())


def gemm_f16_workspace_bytes(M: int, N: int, K: int, variant: int = 0) -> int:
    out = ctypes.c_size_t(0)
    rc = load().gemm_f16_workspace_bytes(M, N, K, variant, ctypes.byref(out))
    if rc != OK:
        raise GemmError(rc, gemm_f16_last_error())
    return out.value


def gemm_f16_sk_tail_tiles(tiles: int, units: int, k_blocks: int) -> int:
    return load().gemm_f16_sk_tail_tiles(tiles, units, k_blocks)


def gemm_f16_set_stream_k(enable: int) -> int:
    """Turn the stream-K tail of launches with a workspace on (1) or off (0, the default)."""
    return load().gemm_f16_set_stream_k(int(enable))


def gemm_f16_raster_group(mma_m: int, K: int, elem_bytes: int, l2_bytes: int) -> int:
    return load().gemm_f16_raster_group(mma_m, K, elem_bytes, l2_bytes)


def gemm_f16_sk_items(tiles: int, units: int, k_blocks: int, tail: int, unit: int) -> int:
    return load().gemm_f16_sk_items(tiles, units, k_blocks, tail, unit)


def gemm_f16_sk_item(tiles: int, units: int, k_blocks: int, tail: int, unit: int, idx: int):
    out = (ctypes.c_uint32 * 5)()
    load().gemm_f16_sk_item(tiles, units, k_blocks, tail, unit, idx, out)
    return tuple(out)


def gemm_f16_sk_unit_of(tiles: int, units: int, k_blocks: int, tail: int, x: int) -> int:
    return load().gemm_f16_sk_unit_of(tiles, units, k_blocks, tail, x)


def gemm_f16_half_tail_tiles(tiles: int, units: int) -> int:
    return load().gemm_f16_half_tail_tiles(tiles, units)


def gemm_f16_half_items(tiles: int, units: int, k_blocks: int, half: int, unit: int) -> int:
    return load().gemm_f16_half_items(tiles, units, k_blocks, half, unit)


def gemm_f16_half_item(tiles: int, units: int, k_blocks: int, half: int, unit: int, idx: int):
    out = (ctypes.c_uint32 * 4)()
    load().gemm_f16_half_item(tiles, units, k_blocks, half, unit, idx, out)
    return tuple(out)


def gemm_f16_choose_variant(M: int, N: int, K: int, num_sms: int) -> int:
    return load().gemm_f16_choose_variant(M, N, K, num_sms)


def gemm_f16_check_status(stream: int = 0):
    """Returns (status, bits)."""
    bits = ctypes.c_uint32(0)
    rc = load().gemm_f16_check_status(stream, ctypes.byref(bits))
    return rc, bits.value


def gemm_f16_set_wait_timeout_ms(ms: int) -> int:
    return load().gemm_f16_set_wait_timeout_ms(ms)


def gemm_f16_set_fault_injection(mode: int) -> int:
    return load().gemm_f16_set_fault_injection(mode)


def gemm_f16_last_error() -> str:
    return load().gemm_f16_last_error().decode()


def gemm_f16_version() -> int:
    return load().gemm_f16_version()


def gemm_f16_get_variant_info(variant: int) -> dict:
    info = VariantInfo()
    rc = load().gemm_f16_get_variant_info(variant, ctypes.byref(info))
    if rc != OK:
        raise GemmError(rc, f"unknown variant {variant}")
    return info.as_dict()


def gemm_f16_idesc(M: int, N: int, ab_bf16: int = 0) -> int:
    return load().gemm_f16_idesc(M, N, ab_bf16)


def gemm_f16_smem_desc_sw128(smem_addr: int, sbo_bytes: int) -> int:
    return load().gemm_f16_smem_desc_sw128(smem_addr, sbo_bytes)


def gemm_f16_sw128(off: int) -> int:
    return load().gemm_f16_sw128(off)


def gemm_f16_tile_coord(t: int, num_m: int, num_n: int, group: int):
    m, n = ctypes.c_uint32(0), ctypes.c_uint32(0)
    load().gemm_f16_tile_coord(t, num_m, num_n, group, ctypes.byref(m), ctypes.byref(n))
    return m.value, n.value


def gemm_f16_ring_pos(it: int, stages: int):
    s, p = ctypes.c_uint32(0), ctypes.c_uint32(0)
    load().gemm_f16_ring_pos(it, stages, ctypes.byref(s), ctypes.byref(p))
    return s.value, p.value


def exported_symbols(header_path: str | None = None):
    """Names of the functions the public headers (include/gemm_f16.h, include/gdn.h) declare."""
    paths = [header_path] if header_path else _build.HEADERS
    names = set()
    for path in paths:
        text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
        names.update(re.findall(r"\b((?:gemm_(?:f16|mxf8)|gdn)_\w+)\s*\(", text))
    return sorted(names)


# ---- block-scaled FP8 (MX) ---------------------------------------------------------------------

FP8_FORMATS = {"e4m3": 0, "e5m2": 1}
MX_VARIANTS = {"auto": 0, "mx_128x128": 1, "mx_pair_256x128": 2, "mx_pair_256x192": 3,
               "mx_pair_256x256": 4}


def gemm_mxf8_nt(A: int, B: int, SFA: int, SFB: int, D: int, M: int, N: int, K: int,
                 fmt_a: int, fmt_b: int, out_dtype: int, bias: int, activation: int,
                 variant: int, workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    return load().gemm_mxf8_nt(A, B, SFA, SFB, D, M, N, K, fmt_a, fmt_b, out_dtype, bias,
                               activation, variant, workspace, workspace_bytes, stream)


def gemm_mxf8_workspace_bytes(M: int, N: int, K: int, variant: int = 0) -> int:
    out = ctypes.c_size_t(0)
    rc = load().gemm_mxf8_workspace_bytes(M, N, K, variant, ctypes.byref(out))
    if rc != OK:
        raise GemmError(rc, gemm_f16_last_error())
    return out.value


def gemm_mxf8_choose_variant(M: int, N: int, K: int, num_sms: int) -> int:
    return load().gemm_mxf8_choose_variant(M, N, K, num_sms)


def gemm_mxf8_scale_bytes(rows: int, K: int) -> int:
    return load().gemm_mxf8_scale_bytes(rows, K)


def gemm_mxf8_pack_scales(src: int, dst: int, rows: int, K: int, stream: int = 0) -> int:
    return load().gemm_mxf8_pack_scales(src, dst, rows, K, stream)


def gemm_mxf8_idesc(M: int, N: int, fmt_a: int = 0, fmt_b: int = 0) -> int:
    return load().gemm_mxf8_idesc(M, N, fmt_a, fmt_b)


def gemm_mxf8_sf_offset(row: int, k_block: int, K: int) -> int:
    return load().gemm_mxf8_sf_offset(row, k_block, K)


def gemm_mxf8_sf_desc(smem_addr: int) -> int:
    return load().gemm_mxf8_sf_desc(smem_addr)


def gemm_mxf8_get_variant_info(variant: int) -> dict:
    info = VariantInfo()
    rc = load().gemm_mxf8_get_variant_info(variant, ctypes.byref(info))
    if rc != OK:
        raise GemmError(rc, f"unknown block-scaled variant {variant}")
    return info.as_dict()


def pack_scales(S, K: int | None = None, stream=None):
    """Row-major block scales (a contiguous CUDA uint8 tensor of rows x K/32 E8M0 codes) -> a new
    CUDA uint8 tensor in the tiled layout the block-scaled GEMM reads."""
    import torch
    if S.dtype != torch.uint8 or not S.is_cuda or S.dim() != 2 or not S.is_contiguous():
        raise ValueError("S must be a contiguous 2-D CUDA uint8 tensor")
    rows, kb = S.shape
    K = 32 * kb if K is None else K
    if K != 32 * kb:
        raise ValueError("S must have K/32 columns")
    out = torch.empty(max(gemm_mxf8_scale_bytes(rows, K), 0), dtype=torch.uint8,
                      device=S.device)
    with torch.cuda.device(S.device):
        rc = gemm_mxf8_pack_scales(S.data_ptr(), out.data_ptr(), rows, K, _stream_handle(stream))
    if rc != OK:
        raise GemmError(rc, gemm_f16_last_error())
    return out


def _u8(t, name):
    import torch
    if t.dtype in (getattr(torch, "float8_e4m3fn", None), getattr(torch, "float8_e5m2", None)):
        t = t.view(torch.uint8)
    if t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA uint8 (or float8) tensor")
    return t


def gemm_mx(A, B, SFA, SFB, out=None, fmt_a: str = "e4m3", fmt_b: str = "e4m3",
            out_dtype: str = "f16", bias=None, activation: str = "none",
            variant: int | str = 0, stream=None, workspace=True):
    """Block-scaled FP8 GEMM: D = act((A * 2^(SA-127)) @ (B * 2^(SB-127)).T + bias).

    A (M, K) and B (N, K): FP8 codes (uint8 or float8 CUDA tensors); SFA, SFB: their E8M0 scales
    in the tiled layout (``pack_scales`` of the row-major (rows, K/32) codes).  Returns D (M, N)
    in float16 or bfloat16.  Asynchronous on ``stream``; raises GemmError on a non-zero status.
    """
    import torch
    if isinstance(variant, str):
        variant = MX_VARIANTS[variant]
    A, B = _u8(A, "A"), _u8(B, "B")
    SFA, SFB = _u8(SFA, "SFA"), _u8(SFB, "SFB")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[1]:
        raise ValueError(f"A is {tuple(A.shape)} and B is {tuple(B.shape)}: K differs")
    M, K = A.shape
    N = B.shape[0]
    for name, t, rows in (("SFA", SFA, M), ("SFB", SFB, N)):
        need = gemm_mxf8_scale_bytes(rows, K)
        if need < 0 or t.numel() < need:
            raise ValueError(f"{name} must hold {need} bytes of tiled scales")
    tdt = torch.float16 if out_dtype == "f16" else torch.bfloat16
    if out is None:
        out = torch.empty((M, N), dtype=tdt, device=A.device)
    elif out.dtype != tdt or not out.is_cuda or tuple(out.shape) != (M, N) or \
            not out.is_contiguous():
        raise ValueError("out must be a contiguous (M, N) CUDA tensor of the output dtype")
    if bias is not None and (bias.dtype != tdt or bias.numel() != N or not bias.is_cuda
                             or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous CUDA vector of N elements of the output dtype")
    ws_ptr, ws_bytes = 0, 0
    if workspace is True and M and N and K:
        need = gemm_mxf8_workspace_bytes(M, N, K, int(variant))
        if need:
            s = stream if stream is not None else torch.cuda.current_stream()
            with torch.cuda.stream(s) if hasattr(s, "cuda_stream") else _nullctx():
                workspace = torch.empty(need, dtype=torch.uint8, device=A.device)
    if workspace is not None and workspace is not True and workspace is not False:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    dev = _one_device(("A", A), ("B", B), ("SFA", SFA), ("SFB", SFB), ("out", out),
                      ("bias", bias), ("workspace", workspace if ws_ptr else None))
    with torch.cuda.device(dev):
        rc = gemm_mxf8_nt(A.data_ptr(), B.data_ptr(), SFA.data_ptr(), SFB.data_ptr(),
                          out.data_ptr(), M, N, K, FP8_FORMATS[fmt_a], FP8_FORMATS[fmt_b],
                          DTYPES[out_dtype], 0 if bias is None else bias.data_ptr(),
                          ACTIVATIONS[activation], int(variant), ws_ptr, ws_bytes,
                          _stream_handle(stream))
    if rc != OK:
        raise GemmError(rc, gemm_f16_last_error())
    return out


# ---- Gated Delta Net prefill ----------------------------------------------------------------------

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_TIMEOUT = 0, 1, 2, 3, 4


def gdn_prefill_workspace_bytes(total_tokens: int, n_seqs: int, h_v: int) -> int:
    out = ctypes.c_size_t(0)
    rc = load().gdn_prefill_workspace_bytes(total_tokens, n_seqs, h_v, ctypes.byref(out))
    if rc != GDN_OK:
        raise GemmError(rc, gdn_last_error())
    return out.value


def gdn_prefill(q: int, k: int, v: int, alpha: int, beta: int, cu_seqlens: int, n_seqs: int,
                total_tokens: int, h_qk: int, h_v: int, head_dim: int, scale: float,
                initial_state: int, o: int, final_state: int, workspace: int,
                workspace_bytes: int, stream: int = 0) -> int:
    return load().gdn_prefill(q, k, v, alpha, beta, cu_seqlens, n_seqs, total_tokens, h_qk, h_v,
                              head_dim, scale, initial_state, o, final_state, workspace,
                              workspace_bytes, stream)


def gdn_prefill_heads(q: int, k: int, v: int, alpha: int, beta: int, cu_seqlens: int,
                      n_seqs: int, total_tokens: int, h_q: int, h_k: int, h_v: int,
                      head_dim: int, scale: float, initial_state: int, o: int, final_state: int,
                      workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    return load().gdn_prefill_heads(q, k, v, alpha, beta, cu_seqlens, n_seqs, total_tokens, h_q,
                                    h_k, h_v, head_dim, scale, initial_state, o, final_state,
                                    workspace, workspace_bytes, stream)


def gdn_out_heads(h_q: int, h_k: int, h_v: int) -> int:
    """Output heads of a head layout: h_v with h_q == h_k (MHA, GVA), h_q with h_q a multiple
    of h_v (GQA); ValueError otherwise (h_v must be a multiple of h_k)."""
    if h_q > 0 and h_k > 0 and h_v > 0 and h_v % h_k == 0:
        if h_q == h_k:
            return h_v
        if h_q % h_v == 0:
            return h_q
    raise ValueError(f"heads q {h_q}, k {h_k}, v {h_v} form no supported layout")


def gdn_last_error() -> str:
    return load().gdn_last_error().decode()


def gdn_check_status(workspace: int, stream: int) -> int:
    return load().gdn_check_status(workspace, stream)


def gdn_check_offsets(cu_seqlens: int, n_seqs: int, total_tokens: int, h_v: int,
                      workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    """Check cu_seqlens on the device (include/gdn.h); read the result with gdn_check_status."""
    return load().gdn_check_offsets(cu_seqlens, n_seqs, total_tokens, h_v, workspace,
                                    workspace_bytes, stream)


def gdn_offsets_valid_host(cu_seqlens, total_tokens: int) -> bool:
    """The offsets' contract applied to a host sequence of n_seqs + 1 offsets."""
    arr = (ctypes.c_int32 * len(cu_seqlens))(*[int(x) for x in cu_seqlens])
    return bool(load().gdn_offsets_valid_host(arr, len(cu_seqlens) - 1, total_tokens))


def gdn_set_wait_timeout_ms(ms: int) -> int:
    return load().gdn_set_wait_timeout_ms(ms)


GDN_SCAN_KERNELS = {"auto": 0, "tensor_core": 1, "mma_sync": 2, "tensor_core_16": 3,
                    "tensor_core_32": 4}


def gdn_set_scan_kernel(kernel: int) -> int:
    """Scan kernel for later calls: GDN_SCAN_KERNELS (include/gdn.h)."""
    return load().gdn_set_scan_kernel(kernel)


def gdn_set_fault_injection(mode: int) -> int:
    return load().gdn_set_fault_injection(mode)


def gated_delta_rule(q, k, v, alpha, beta, cu_seqlens, scale: float, initial_state=None,
                     output_final_state: bool = False, stream=None, workspace=None):
    """Gated Delta Net prefill over packed sequences (CUDA tensors): q [T, h_q, 128], k
    [T, h_k, 128] and v [T, h_v, 128] bfloat16; alpha, beta [T, h_v] float32; cu_seqlens [n + 1]
    int32, non-decreasing from 0 to T (not checked: the kernels trust these offsets and would
    access memory outside the tensors for others); initial_state [n, h_v, 128, 128] float32 or
    None.  h_v is a multiple of h_k, and h_q
    equals h_k (MHA, GVA: o has h_v heads) or is a multiple of h_v (GQA: o has h_q heads).
    Returns (o [T, h_o, 128] bfloat16, final_state or None).  Asynchronous on ``stream``; raises
    GemmError on a non-zero status."""
    import torch
    # shapes first: the kernels read exactly these extents, and no device check can catch a
    # buffer that is too small
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k and v must be [T, heads, head_dim] tensors")
    T, h_q, d = q.shape
    h_k, h_v = k.shape[1], v.shape[1]
    if tuple(k.shape) != (T, h_k, d) or tuple(v.shape) != (T, h_v, d):
        raise ValueError(f"k {tuple(k.shape)} and v {tuple(v.shape)} must have q's tokens and "
                         f"head dim ({T}, ., {d})")
    if tuple(alpha.shape) != (T, h_v) or tuple(beta.shape) != (T, h_v):
        raise ValueError(f"alpha {tuple(alpha.shape)} and beta {tuple(beta.shape)} must be "
                         f"[T, h_v] = ({T}, {h_v})")
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must be a 1-D tensor of n_seqs + 1 offsets")
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("alpha", alpha, torch.float32),
                        ("beta", beta, torch.float32), ("cu_seqlens", cu_seqlens, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    h_o = gdn_out_heads(h_q, h_k, h_v)
    n = cu_seqlens.numel() - 1
    if initial_state is not None and (initial_state.dtype != torch.float32 or
                                      tuple(initial_state.shape) != (n, h_v, d, d) or
                                      not initial_state.is_contiguous()):
        raise ValueError("initial_state must be a contiguous float32 [n, h_v, d, d] tensor")
    dev = _one_device(("q", q), ("k", k), ("v", v), ("alpha", alpha), ("beta", beta),
                      ("cu_seqlens", cu_seqlens), ("initial_state", initial_state),
                      ("workspace", workspace))
    if workspace is not None and (not workspace.is_cuda or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    o = torch.empty((T, h_o, d), dtype=torch.bfloat16, device=q.device)
    sf = (torch.empty((n, h_v, d, d), dtype=torch.float32, device=q.device)
          if output_final_state else None)
    if workspace is None:
        need = gdn_prefill_workspace_bytes(T, n, h_v)
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s) if hasattr(s, "cuda_stream") else _nullctx():
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(dev):
        rc = gdn_prefill_heads(q.data_ptr(), k.data_ptr(), v.data_ptr(), alpha.data_ptr(),
                               beta.data_ptr(), cu_seqlens.data_ptr(), n, T, h_q, h_k, h_v, d,
                               float(scale),
                               0 if initial_state is None else initial_state.data_ptr(),
                               o.data_ptr(), 0 if sf is None else sf.data_ptr(),
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                               _stream_handle(stream))
    if rc != GDN_OK:
        raise GemmError(rc, gdn_last_error())
    return o, sf


# ---- torch convenience ----------------------------------------------------------------------

def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def gemm(A, B, out=None, variant: int | str = 0, stream=None, workspace=True):
    """D = A @ B.T for CUDA fp16 tensors A (M, K) and B (N, K); returns D (M, N) fp16.

    ``out`` may be a preallocated contiguous (M, N) fp16 CUDA tensor.  The call is asynchronous
    on ``stream`` (default: torch's current stream).  ``workspace``: True (default) takes a
    stream-K workspace from torch's caching allocator when the shape benefits from one; a CUDA
    uint8 tensor supplies one; False or None runs without.  Raises GemmError on a non-zero
    status.
    """
    import torch
    if isinstance(variant, str):
        variant = VARIANTS[variant]
    for name, t in (("A", A), ("B", B)):
        if t.dtype != torch.float16 or not t.is_cuda or t.dim() != 2 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 2-D CUDA float16 tensor")
    M, K = A.shape
    N, K2 = B.shape
    if K2 != K:
        raise ValueError(f"A is {tuple(A.shape)} and B is {tuple(B.shape)}: K differs")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    elif (out.dtype != torch.float16 or not out.is_cuda or tuple(out.shape) != (M, N)
          or not out.is_contiguous()):
        raise ValueError("out must be a contiguous (M, N) CUDA float16 tensor")
    ws_ptr, ws_bytes = 0, 0
    if workspace is True and M and N and K:
        need = gemm_f16_workspace_bytes(M, N, K, int(variant))
        if need:
            s = stream if stream is not None else torch.cuda.current_stream()
            with torch.cuda.stream(s) if hasattr(s, "cuda_stream") else _nullctx():
                workspace = torch.empty(need, dtype=torch.uint8, device=A.device)
    if workspace is not None and workspace is not True and workspace is not False:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    dev = _one_device(("A", A), ("B", B), ("out", out),
                      ("workspace", workspace if ws_ptr else None))
    with torch.cuda.device(dev):
        rc = gemm_f16_nt_ex(A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K, int(variant),
                            ws_ptr, ws_bytes, _stream_handle(stream))
    if rc != OK:
        raise GemmError(rc, gemm_f16_last_error())
    return out


class _nullctx:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def _one_device(*named):
    """The device that every given tensor (None entries skipped) lives on.  The C entry points
    launch on the current CUDA device, so the torch entry points run them under this one: a
    tensor on another device would otherwise be read by the wrong GPU."""
    dev = None
    for name, t in named:
        if t is None or isinstance(t, bool):
            continue
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the other operands on {dev}")
    return dev


def check_status(stream=None) -> None:
    """Synchronise ``stream`` and raise GemmError if a kernel gave up a bounded wait."""
    rc, bits = gemm_f16_check_status(_stream_handle(stream))
    if rc != OK:
        raise GemmError(rc, f"{gemm_f16_last_error()} (bits 0x{bits:x})")
