"""The CPU oracle for D = A * B^T (fp16 in, binary64 sum).

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, loads or
runs this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may.  The library path fails loudly when its CUDA
extension is missing; it never falls back to this code.

The arithmetic lives in ``gemm_ref.c`` (plain C, binary64, OpenMP over output
rows), written from the definition D[i][j] = sum_k A[i][k] * B[j][k] on the
page "TIRx 与高性能GEMM (上)" (section "从 GEMM 公式到数据路径") and from the
IEEE 754 binary16 format.  This file only builds that C file with gcc and
marshals numpy arrays through ctypes.

Pins: ``tests/test_oracle.py`` checks every function here against values fixed
by the pages and by mathematics (all-ones, identity, permutation, rank-one
probes, exact rational brute force, exhaustive binary16 round trips, library
conversions).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_ref.c")
_SRCS = [_SRC, os.path.join(_HERE, "mx_ref.c"), os.path.join(_HERE, "gdn_ref.c")]
_LIB = os.path.join(_HERE, "liboracle_gemm.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gemm_ref.c``, ``mx_ref.c`` and ``gdn_ref.c`` into ``liboracle_gemm.so`` next to
    them (gcc, OpenMP)."""
    stale = not os.path.exists(_LIB) or any(os.path.getmtime(_LIB) < os.path.getmtime(f)
                                            for f in _SRCS)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-Wall"] + _SRCS + ["-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, u16p, f64p, i64p = (ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p)
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
            lib.oracle_f64_to_f16.restype = ctypes.c_uint16
            lib.oracle_decode_f16.argtypes = [u16p, f64p, i64]
            lib.oracle_decode_f16.restype = None
            lib.oracle_round_f16.argtypes = [f64p, u16p, i64]
            lib.oracle_round_f16.restype = None
            lib.oracle_gemm_f64.argtypes = [u16p, u16p, f64p, i64, i64, i64]
            lib.oracle_gemm_f64.restype = ctypes.c_int
            lib.oracle_gemm_f64_sampled.argtypes = [u16p, u16p, i64, i64, i64, i64p, i64p,
                                                    i64, f64p]
            lib.oracle_gemm_f64_sampled.restype = None
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
            lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
            lib.oracle_decode_bf16.argtypes = [u16p, f64p, i64]
            lib.oracle_decode_bf16.restype = None
            lib.oracle_round_bf16.argtypes = [f64p, u16p, i64]
            lib.oracle_round_bf16.restype = None
            lib.oracle_gemm_f64_dt.argtypes = [u16p, u16p, f64p, i64, i64, i64, ctypes.c_int]
            lib.oracle_gemm_f64_dt.restype = ctypes.c_int
            lib.oracle_gemm_f64_sampled_dt.argtypes = [u16p, u16p, i64, i64, i64, i64p, i64p,
                                                       i64, f64p, ctypes.c_int]
            lib.oracle_gemm_f64_sampled_dt.restype = None
            lib.oracle_epilogue_f64.argtypes = [f64p, i64, i64, u16p, ctypes.c_int, ctypes.c_int]
            lib.oracle_epilogue_f64.restype = None
            u8p = ctypes.c_void_p
            lib.oracle_fp8_to_f64.argtypes = [ctypes.c_uint8, ctypes.c_int]
            lib.oracle_fp8_to_f64.restype = ctypes.c_double
            lib.oracle_e8m0_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_e8m0_to_f64.restype = ctypes.c_double
            lib.oracle_decode_fp8.argtypes = [u8p, f64p, i64, ctypes.c_int]
            lib.oracle_decode_fp8.restype = None
            lib.oracle_decode_e8m0.argtypes = [u8p, f64p, i64]
            lib.oracle_decode_e8m0.restype = None
            lib.oracle_gemm_mx_f64.argtypes = [u8p, u8p, u8p, u8p, f64p, f64p, i64, i64, i64,
                                               ctypes.c_int, ctypes.c_int]
            lib.oracle_gemm_mx_f64.restype = ctypes.c_int
            lib.oracle_gemm_mx_f64_sampled.argtypes = [u8p, u8p, u8p, u8p, i64, i64, i64,
                                                       ctypes.c_int, ctypes.c_int, i64p, i64p,
                                                       i64, f64p, f64p]
            lib.oracle_gemm_mx_f64_sampled.restype = ctypes.c_int
            lib.oracle_gdn_f64.argtypes = [f64p, f64p, f64p, f64p, f64p, ctypes.c_void_p, i64,
                                           i64, i64, i64, i64, ctypes.c_double, f64p, f64p,
                                           f64p]
            lib.oracle_gdn_f64.restype = ctypes.c_int
            lib.oracle_gdn_heads_f64.argtypes = [f64p, f64p, f64p, f64p, f64p, ctypes.c_void_p,
                                                 i64, i64, i64, i64, i64, i64, ctypes.c_double,
                                                 f64p, f64p, f64p]
            lib.oracle_gdn_heads_f64.restype = ctypes.c_int
            lib.oracle_gdn_out_heads.argtypes = [i64, i64, i64]
            lib.oracle_gdn_out_heads.restype = i64
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


DTYPES = {"f16": 0, "bf16": 1}
ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2}


def _as_u16(x) -> np.ndarray:
    """16-bit array (numpy float16/uint16, or a CPU torch fp16/bf16 tensor) -> contiguous uint16
    view of its bits."""
    if hasattr(x, "detach"):  # a torch tensor: reinterpret its bits without arithmetic
        x = x.detach().cpu().contiguous().view(dtype=__import__("torch").int16).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16 or x.dtype == np.int16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError(f"expected fp16 bits, got {x.dtype}")
    return x


def f16_bits_to_f64(bits) -> np.ndarray:
    """binary16 bit patterns -> binary64 values (exact widening)."""
    b = _as_u16(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode_f16(b.ctypes.data, out.ctypes.data, b.size)
    return out


def f64_to_f16_bits(x) -> np.ndarray:
    """binary64 values -> binary16 bit patterns, round to nearest, ties to even."""
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_round_f16(v.ctypes.data, out.ctypes.data, v.size)
    return out


def gemm_f64(A, B) -> np.ndarray:
    """D64 = A * B^T summed in binary64.  A: (M, K) fp16, B: (N, K) fp16."""
    a, b = _as_u16(A), _as_u16(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"shapes {a.shape} and {b.shape} do not contract")
    M, K = a.shape
    N = b.shape[0]
    out = np.empty((M, N), dtype=np.float64)
    if _load().oracle_gemm_f64(a.ctypes.data, b.ctypes.data, out.ctypes.data, M, N, K) != 0:
        raise MemoryError("oracle could not allocate its binary64 copies")
    return out


def gemm_f16(A, B) -> np.ndarray:
    """The fp16 output value: RNE(A * B^T), as binary16 bit patterns (uint16)."""
    return f64_to_f16_bits(gemm_f64(A, B))


def gemm_f64_sampled(A, B, rows, cols) -> np.ndarray:
    """D64[rows[t], cols[t]] for each t, each an independent binary64 dot product."""
    a, b = _as_u16(A), _as_u16(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"shapes {a.shape} and {b.shape} do not contract")
    M, K = a.shape
    N = b.shape[0]
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in length")
    if r.size and (r.min() < 0 or r.max() >= M or c.min() < 0 or c.max() >= N):
        raise IndexError("sample index out of range")
    out = np.empty(r.shape, dtype=np.float64)
    _load().oracle_gemm_f64_sampled(a.ctypes.data, b.ctypes.data, M, N, K, r.ctypes.data,
                                    c.ctypes.data, r.size, out.ctypes.data)
    return out


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns -> binary64 values (exact widening)."""
    b = _as_u16(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode_bf16(b.ctypes.data, out.ctypes.data, b.size)
    return out


def f64_to_bf16_bits(x) -> np.ndarray:
    """binary64 values -> bfloat16 bit patterns, round to nearest, ties to even."""
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_round_bf16(v.ctypes.data, out.ctypes.data, v.size)
    return out


def gemm_f64_dt(A, B, dtype: str = "f16") -> np.ndarray:
    """D64 = A * B^T in binary64 for fp16 ("f16") or bfloat16 ("bf16") inputs."""
    a, b = _as_u16(A), _as_u16(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"shapes {a.shape} and {b.shape} do not contract")
    M, K = a.shape
    N = b.shape[0]
    out = np.empty((M, N), dtype=np.float64)
    if _load().oracle_gemm_f64_dt(a.ctypes.data, b.ctypes.data, out.ctypes.data, M, N, K,
                                  DTYPES[dtype]) != 0:
        raise MemoryError("oracle could not allocate its binary64 copies")
    return out


def gemm_f64_sampled_dt(A, B, rows, cols, dtype: str = "f16") -> np.ndarray:
    a, b = _as_u16(A), _as_u16(B)
    M, K = a.shape
    N = b.shape[0]
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.size and (r.min() < 0 or r.max() >= M or c.min() < 0 or c.max() >= N):
        raise IndexError("sample index out of range")
    out = np.empty(r.shape, dtype=np.float64)
    _load().oracle_gemm_f64_sampled_dt(a.ctypes.data, b.ctypes.data, M, N, K, r.ctypes.data,
                                       c.ctypes.data, r.size, out.ctypes.data, DTYPES[dtype])
    return out


def epilogue(X, bias=None, activation: str = "none", dtype: str = "f16", cols=None) -> np.ndarray:
    """act(X + bias[j]) in binary64 (a new array).  X: (M, N) binary64 sums, or a 1-D array of
    sampled elements whose column indices are `cols`.  bias: N elements of the given 16-bit type
    (bits or a torch tensor) or None."""
    x = np.array(X, dtype=np.float64, copy=True)
    b = None if bias is None else _as_u16(bias)
    if x.ndim == 1:  # sampled elements: gather the bias columns into a 1 x count problem
        bb = None if b is None else np.ascontiguousarray(b[np.asarray(cols)])
        x2 = np.ascontiguousarray(x.reshape(1, -1))
        _load().oracle_epilogue_f64(x2.ctypes.data, 1, x2.shape[1],
                                    None if bb is None else bb.ctypes.data, DTYPES[dtype],
                                    ACTIVATIONS[activation])
        return x2.reshape(-1)
    x = np.ascontiguousarray(x)
    M, N = x.shape
    if b is not None and b.size != N:
        raise ValueError("bias must have N elements")
    _load().oracle_epilogue_f64(x.ctypes.data, M, N, None if b is None else b.ctypes.data,
                                DTYPES[dtype], ACTIVATIONS[activation])
    return x


def tolerance_dt(d_ref: np.ndarray, K: int, dtype: str = "f16") -> np.ndarray:
    """The parity bound for an output of the given type: 1e-3 * sqrt(K) + rel * |D_ref| with
    rel = 2^-10 for fp16 (the stated bound: twice fp16's half-ulp 2^-11) and 2^-7 for bfloat16
    (twice bfloat16's half-ulp 2^-8, by the same derivation)."""
    rel = 2.0 ** -10 if dtype == "f16" else 2.0 ** -7
    return 1e-3 * np.sqrt(float(K)) + np.abs(d_ref) * rel


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().oracle_num_threads())


def tolerance(d_ref: np.ndarray, K: int) -> np.ndarray:
    """Per-element bound |D_gpu - D_ref| <= 1e-3 * sqrt(K) + 2^-10 * |D_ref|.

    D_ref is the binary64 sum (unrounded).  The bound's absolute term covers the
    fp32 accumulation of K terms of size O(1/sqrt(K)) to O(1); its relative term
    covers the final fp16 rounding (at most 2^-11 relative) with a factor of two
    to spare.
    """
    return 1e-3 * np.sqrt(float(K)) + np.abs(d_ref) * 2.0 ** -10


# ---- block-scaled FP8 (MX) ----------------------------------------------------------------------

FP8_FORMATS = {"e4m3": 0, "e5m2": 1}


def _as_u8(x) -> np.ndarray:
    """8-bit codes (numpy uint8/int8, or a CPU torch uint8/int8/float8 tensor) -> contiguous
    uint8 view of their bits."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().cpu().contiguous().view(dtype=torch.uint8).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.int8:
        x = x.view(np.uint8)
    if x.dtype != np.uint8:
        raise TypeError(f"expected 8-bit codes, got {x.dtype}")
    return x


def fp8_bits_to_f64(codes, fmt: str = "e4m3") -> np.ndarray:
    """FP8 codes -> binary64 values (exact)."""
    c = _as_u8(codes)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_decode_fp8(c.ctypes.data, out.ctypes.data, c.size, FP8_FORMATS[fmt])
    return out


def e8m0_to_f64(codes) -> np.ndarray:
    """E8M0 scale codes -> 2^(e - 127) (255: NaN)."""
    c = _as_u8(codes)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_decode_e8m0(c.ctypes.data, out.ctypes.data, c.size)
    return out


def _mx_args(A, B, SA, SB):
    a, b, sa, sb = _as_u8(A), _as_u8(B), _as_u8(SA), _as_u8(SB)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"shapes {a.shape} and {b.shape} do not contract")
    M, K = a.shape
    N = b.shape[0]
    if K % 32 != 0:
        raise ValueError("K must be a multiple of the 32-element scale block")
    if sa.shape != (M, K // 32) or sb.shape != (N, K // 32):
        raise ValueError(f"scale shapes {sa.shape}, {sb.shape}; want {(M, K // 32)}, "
                         f"{(N, K // 32)}")
    return a, b, sa, sb, M, N, K


def gemm_mx_f64(A, B, SA, SB, fmt_a: str = "e4m3", fmt_b: str = "e4m3"):
    """(D, Dabs): D = sum_k (a*sa) * (b*sb) in binary64 and Dabs = sum_k |(a*sa) * (b*sb)|.
    A: (M, K) FP8 codes, B: (N, K), SA: (M, K/32) E8M0 codes, SB: (N, K/32)."""
    a, b, sa, sb, M, N, K = _mx_args(A, B, SA, SB)
    D = np.empty((M, N), dtype=np.float64)
    Dabs = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_mx_f64(a.ctypes.data, b.ctypes.data, sa.ctypes.data, sb.ctypes.data,
                                    D.ctypes.data, Dabs.ctypes.data, M, N, K,
                                    FP8_FORMATS[fmt_a], FP8_FORMATS[fmt_b])
    if rc != 0:
        raise MemoryError("oracle could not allocate its binary64 copies")
    return D, Dabs


def gemm_mx_f64_sampled(A, B, SA, SB, rows, cols, fmt_a: str = "e4m3", fmt_b: str = "e4m3"):
    """(D, Dabs) at the output elements (rows[t], cols[t])."""
    a, b, sa, sb, M, N, K = _mx_args(A, B, SA, SB)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape or r.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    if r.size and (r.min() < 0 or r.max() >= M or c.min() < 0 or c.max() >= N):
        raise IndexError("sampled index out of range")
    out = np.empty(r.size, dtype=np.float64)
    out_abs = np.empty(r.size, dtype=np.float64)
    _load().oracle_gemm_mx_f64_sampled(a.ctypes.data, b.ctypes.data, sa.ctypes.data,
                                       sb.ctypes.data, M, N, K, FP8_FORMATS[fmt_a],
                                       FP8_FORMATS[fmt_b], r.ctypes.data, c.ctypes.data, r.size,
                                       out.ctypes.data, out_abs.ctypes.data)
    return out, out_abs


def tolerance_mx(d_ref: np.ndarray, d_abs: np.ndarray, K: int, out_dtype: str = "f16"):
    """Parity bound for the block-scaled GEMM: rel * |D| + 4 * (K/32 + 1) * 2^-24 * Dabs.

    Every product of two scaled FP8 values is exact in fp32's 24-bit significand (8 significant
    bits), so the only accumulation error is the rounding of partial sums, one per 32-element
    block and one per accumulate into the fp32 accumulator: at most (K/32 + 1) roundings of
    2^-24 relative to the sum of |terms|, with a factor of 4 to spare for the order of the
    tensor core's internal adds.  rel covers the final rounding as for the 16-bit GEMM: 2^-10
    for fp16 output and 2^-7 for bfloat16."""
    rel = 2.0 ** -10 if out_dtype == "f16" else 2.0 ** -7
    return np.abs(d_ref) * rel + 4.0 * (K / 32.0 + 1.0) * 2.0 ** -24 * np.asarray(d_abs)


# ---- Gated Delta Net prefill ----------------------------------------------------------------------

def _f64(x, name) -> np.ndarray:
    """A float array (numpy, or a CPU torch tensor of float32 / bfloat16 / float16) -> contiguous
    binary64.  bfloat16 is widened with the oracle's own decoder."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            return bf16_bits_to_f64(x)
        if x.dtype == torch.float16:
            return f16_bits_to_f64(x)
        x = x.numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def gdn_out_heads(h_q: int, h_k: int, h_v: int) -> int:
    """Output heads of the head layout (h_q, h_k, h_v); ValueError if it is none of MHA, GVA,
    GQA (h_v a multiple of h_k; h_q == h_k, or h_q a multiple of h_v)."""
    h_o = _load().oracle_gdn_out_heads(h_q, h_k, h_v)
    if h_o < 0:
        raise ValueError(f"head counts q {h_q}, k {h_k}, v {h_v} form no supported layout")
    return int(h_o)


def gdn_f64(q, k, v, alpha, beta, cu_seqlens, scale: float, initial_state=None):
    """(o, final_state) of the gated delta rule, token by token in binary64.

    q: [T, h_q, dk]; k: [T, h_k, dk]; v: [T, h_v, dv]; alpha, beta: [T, h_v]; cu_seqlens: n_seqs + 1
    offsets; initial_state: [n_seqs, h_v, dv, dk] or None (zero).  h_v is a multiple of h_k, and
    either h_q == h_k (one output per value head: MHA, GVA) or h_q is a multiple of h_v (one
    output per query head: GQA).  Returns o [T, h_o, dv] and the final states
    [n_seqs, h_v, dv, dk], both binary64."""
    qd, kd, vd = _f64(q, "q"), _f64(k, "k"), _f64(v, "v")
    ad, bd = _f64(alpha, "alpha"), _f64(beta, "beta")
    cu = np.ascontiguousarray(np.asarray(cu_seqlens), dtype=np.int32)
    T, h_q, dk = qd.shape
    h_k = kd.shape[1]
    h_v, dv = vd.shape[1], vd.shape[2]
    n = cu.size - 1
    if kd.shape != (T, h_k, dk) or vd.shape[0] != T or ad.shape != (T, h_v) or \
            bd.shape != (T, h_v):
        raise ValueError("inconsistent shapes")
    if n < 0 or cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must rise from 0 to T")
    h_o = gdn_out_heads(h_q, h_k, h_v)
    s0 = None
    if initial_state is not None:
        s0 = _f64(initial_state, "initial_state")
        if s0.shape != (n, h_v, dv, dk):
            raise ValueError(f"initial_state shape {s0.shape}; want {(n, h_v, dv, dk)}")
    o = np.empty((T, h_o, dv), dtype=np.float64)
    sf = np.empty((n, h_v, dv, dk), dtype=np.float64)
    rc = _load().oracle_gdn_heads_f64(qd.ctypes.data, kd.ctypes.data, vd.ctypes.data,
                                      ad.ctypes.data, bd.ctypes.data, cu.ctypes.data, n, h_q,
                                      h_k, h_v, dk, dv, float(scale),
                                      None if s0 is None else s0.ctypes.data, o.ctypes.data,
                                      sf.ctypes.data)
    if rc == -1:
        raise ValueError("inconsistent sizes")
    if rc != 0:
        raise MemoryError("oracle could not allocate its state")
    return o, sf
