"""Seeded synthetic inputs for D = A * B^T (fp16 A: M x K, fp16 B: N x K).

This module draws inputs and nothing else: it holds none of the GEMM's
arithmetic, so both the CUDA path's tests and the CPU oracle can be fed from it.

Each workload fixes a shape, a value distribution and a seed.  Values are drawn
in float32 from one ``torch.Generator`` on the CPU, A first and then B, and are
rounded to fp16 by the ordinary float32 -> fp16 conversion:

* ``uniform``: i.i.d. uniform on [-1, 1]  (``rand * 2 - 1``)
* ``normal``:  i.i.d. normal(0, 1) times ``scale``  (``randn * scale``)

The shapes are the ones the GEMM pages use (a single 128 x 128 x 64 tile, as in
Step 1 of "TIRx 与高性能GEMM (上)") plus square, ragged and MLP-projection
shapes of the size a linear layer has.  torch's CPU generator may produce
different streams on different CPU architectures, so expected values are
always computed on the machine that runs the comparison, never stored.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    seed: int
    a_dist: str
    a_scale: float
    b_dist: str
    b_scale: float

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def min_bytes(self) -> int:
        """Bytes that must cross HBM at least once: read A and B, write D (fp16)."""
        return 2 * (self.M * self.K + self.N * self.K + self.M * self.N)


def _normal_over_sqrt_k(name, M, N, K, seed):
    s = 1.0 / math.sqrt(K)
    return Workload(name, M, N, K, seed, "normal", s, "normal", s)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("single_tile_128x128x64", 128, 128, 64, 0, "uniform", 1.0, "uniform", 1.0),
        _normal_over_sqrt_k("square_2048", 2048, 2048, 2048, 1),
        Workload("ragged_3000x5000x1000", 3000, 5000, 1000, 2, "uniform", 1.0, "uniform", 1.0),
        _normal_over_sqrt_k("square_8192", 8192, 8192, 8192, 3),
        # MLP up-projection: 16384 tokens, hidden 4096 -> 14336; weights normal(0, 1/sqrt(4096)).
        Workload("mlp_up_16384x14336x4096", 16384, 14336, 4096, 4, "normal", 1.0, "normal",
                 1.0 / 64.0),
    ]
}

ORDER = list(WORKLOADS)


def _draw(gen: torch.Generator, shape, dist: str, scale: float,
          dtype=torch.float16) -> torch.Tensor:
    if dist == "uniform":
        x = torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32) * scale
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.to(dtype)


def make_inputs(M: int, N: int, K: int, seed: int, a_dist: str = "uniform",
                a_scale: float = 1.0, b_dist: str = "uniform", b_scale: float = 1.0,
                dtype=torch.float16):
    """(A, B) as contiguous CPU tensors of shapes (M, K) and (N, K), fp16 unless `dtype` says
    bfloat16 (drawn in float32, then rounded to the 16-bit type)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    A = _draw(gen, (M, K), a_dist, a_scale, dtype)
    B = _draw(gen, (N, K), b_dist, b_scale, dtype)
    return A.contiguous(), B.contiguous()


def make_bias(N: int, seed: int, scale: float = 1.0, dtype=torch.float16) -> torch.Tensor:
    """A bias vector of N elements, uniform on [-scale, scale]."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed) + 7919)
    return ((torch.rand(N, generator=gen, dtype=torch.float32) * 2.0 - 1.0) * scale).to(dtype)


def workload_inputs(w: Workload):
    return make_inputs(w.M, w.N, w.K, w.seed, w.a_dist, w.a_scale, w.b_dist, w.b_scale)


# ---- block-scaled FP8 (MX) inputs ----------------------------------------------------------------
#
# Elements: i.i.d. normal(0, 1) in float32, clamped to the format's largest finite value and
# rounded to FP8 (E4M3 or E5M2) by torch's float32 -> float8 conversion.  Scales: one E8M0 code
# per row and per block of 32 K elements, 127 - s + r with s = round(log2(K) / 4) and r uniform
# on {-2, ..., 2}, so that sums of K terms stay of order one in fp16 and bf16 whatever K is.
# Drawn from one torch.Generator in the order A, B, SA, SB.

FP8_MAX = {"e4m3": 448.0, "e5m2": 57344.0}
FP8_TORCH = {"e4m3": "float8_e4m3fn", "e5m2": "float8_e5m2"}


@dataclass(frozen=True)
class MxWorkload:
    name: str
    M: int
    N: int
    K: int
    seed: int
    fmt_a: str = "e4m3"
    fmt_b: str = "e4m3"

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def min_bytes(self) -> int:
        """Bytes that must cross HBM at least once: FP8 A and B, their scales, fp16 D."""
        return self.M * self.K + self.N * self.K + (self.M + self.N) * (self.K // 32) \
            + 2 * self.M * self.N


MX_WORKLOADS = {
    w.name: w
    for w in [
        MxWorkload("mx_single_tile_128x128x128", 128, 128, 128, 10),
        MxWorkload("mx_square_2048", 2048, 2048, 2048, 11),
        # ragged in M and N; K = 8 * 128 + 32 ends in a partial group of four scale blocks
        MxWorkload("mx_ragged_3000x5000x1056", 3000, 5000, 1056, 12),
        MxWorkload("mx_square_8192", 8192, 8192, 8192, 13),
        MxWorkload("mx_mlp_up_16384x14336x4096", 16384, 14336, 4096, 14),
    ]
}

MX_ORDER = list(MX_WORKLOADS)


def _draw_fp8(gen: torch.Generator, shape, fmt: str) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    x = x.clamp_(-FP8_MAX[fmt], FP8_MAX[fmt])
    return x.to(getattr(torch, FP8_TORCH[fmt])).view(torch.uint8).contiguous()


def mx_scale_shift(K: int) -> int:
    return int(round(math.log2(max(K, 1)) / 4.0))


def _draw_scales(gen: torch.Generator, rows: int, K: int) -> torch.Tensor:
    r = torch.randint(-2, 3, (rows, K // 32), generator=gen, dtype=torch.int32)
    return (127 - mx_scale_shift(K) + r).to(torch.uint8).contiguous()


def make_mx_inputs(M: int, N: int, K: int, seed: int, fmt_a: str = "e4m3",
                   fmt_b: str = "e4m3"):
    """(A, B, SA, SB) as contiguous CPU uint8 tensors: FP8 codes of shapes (M, K) and (N, K),
    E8M0 scale codes of shapes (M, K/32) and (N, K/32), row-major."""
    if K % 32 != 0:
        raise ValueError("K must be a multiple of 32 (the scale block)")
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    A = _draw_fp8(gen, (M, K), fmt_a)
    B = _draw_fp8(gen, (N, K), fmt_b)
    SA = _draw_scales(gen, M, K)
    SB = _draw_scales(gen, N, K)
    return A, B, SA, SB


def mx_workload_inputs(w: MxWorkload):
    return make_mx_inputs(w.M, w.N, w.K, w.seed, w.fmt_a, w.fmt_b)


# ---- Gated Delta Net prefill inputs --------------------------------------------------------------
#
# The six scenarios of the page "TIRx" (zixuwang.me), section "公开版本复测：六个场景": BF16 q/k/v,
# head dimension 128, scale 0.73; single or packed sequences; multi-head (h_v == h_qk) or grouped
# values (h_v = 2 h_qk); zero or given initial state (and then a final state out).
# Draws, in this order from one torch.Generator: packed lengths (n - 1 cut points uniform on
# 1 .. T - 1 without repeats), q and k normal(0, 1) then scaled to unit L2 norm per token and head
# (the key normalisation that keeps the delta rule contractive), v normal(0, 1), all rounded to
# bfloat16; alpha = exp(-U[0, 0.1)) and beta = sigmoid(normal(0, 1)) in float32; an initial
# state normal(0, 0.1^2) in float32 when the scenario has one.

@dataclass(frozen=True)
class GdnWorkload:
    name: str
    T: int
    n_seqs: int
    h_qk: int
    h_v: int
    state: bool
    seed: int
    dk: int = 128
    dv: int = 128
    scale: float = 0.73

    @property
    def flops(self) -> int:
        """Multiply-adds of the token recurrence, counted as two flops: per token and value head
        the prediction (dv*dk), the rank-one update (dv*dk) and the output (dv*dk)."""
        return 2 * 3 * self.T * self.h_v * self.dv * self.dk

    @property
    def min_bytes(self) -> int:
        """Bytes a call must move at least: q, k, v and o (bf16), alpha and beta (fp32), and the
        fp32 initial and final states when the scenario carries them."""
        b = 2 * self.T * (2 * self.h_qk * self.dk + 2 * self.h_v * self.dv) + 8 * self.T * self.h_v
        if self.state:
            b += 2 * 4 * self.n_seqs * self.h_v * self.dv * self.dk
        return b


GDN_WORKLOADS = {
    w.name: w
    for w in [
        GdnWorkload("single_t512_h8_mha_zero", 512, 1, 8, 8, False, 20),
        GdnWorkload("single_t1024_h8_mha_state", 1024, 1, 8, 8, True, 21),
        GdnWorkload("single_t1024_h8_hv16_gva_state", 1024, 1, 8, 16, True, 22),
        GdnWorkload("single_t4096_h16_mha_zero", 4096, 1, 16, 16, False, 23),
        GdnWorkload("packed_n10_t4096_h8_mha_state", 4096, 10, 8, 8, True, 24),
        GdnWorkload("packed_n20_t8192_h8_hv16_gva_state", 8192, 20, 8, 16, True, 25),
    ]
}

GDN_ORDER = list(GDN_WORKLOADS)


def make_gdn_inputs(T: int, n_seqs: int, h_qk: int, h_v: int, dk: int, dv: int, seed: int,
                    state: bool = False):
    """dict of CPU tensors: q, k [T, h_qk, dk] and v [T, h_v, dv] bfloat16; alpha, beta [T, h_v]
    float32; cu_seqlens [n_seqs + 1] int32; initial_state [n_seqs, h_v, dv, dk] float32 or
    None."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    if n_seqs > 1:
        cuts = torch.randperm(T - 1, generator=gen)[: n_seqs - 1] + 1
        cu = torch.cat([torch.tensor([0]), torch.sort(cuts).values, torch.tensor([T])])
    else:
        cu = torch.tensor([0, T][: n_seqs + 1]) if n_seqs == 1 else torch.tensor([0])
    cu = cu.to(torch.int32)

    def unit(shape):
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        return (x / x.norm(dim=-1, keepdim=True).clamp_min(1e-6)).to(torch.bfloat16)

    q = unit((T, h_qk, dk))
    k = unit((T, h_qk, dk))
    v = torch.randn((T, h_v, dv), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    alpha = torch.exp(-0.1 * torch.rand((T, h_v), generator=gen, dtype=torch.float32))
    beta = torch.sigmoid(torch.randn((T, h_v), generator=gen, dtype=torch.float32))
    s0 = (0.1 * torch.randn((n_seqs, h_v, dv, dk), generator=gen, dtype=torch.float32)
          if state else None)
    return {"q": q.contiguous(), "k": k.contiguous(), "v": v.contiguous(),
            "alpha": alpha.contiguous(), "beta": beta.contiguous(), "cu_seqlens": cu,
            "initial_state": s0}


def gdn_workload_inputs(w: GdnWorkload):
    return make_gdn_inputs(w.T, w.n_seqs, w.h_qk, w.h_v, w.dk, w.dv, w.seed, w.state)
