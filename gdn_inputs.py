"""Seeded synthetic inputs for the gated DeltaNet token mixer.

This module only draws random numbers and casts them; it holds none of the
method's arithmetic, so both the CUDA path's tests/benchmark and the CPU oracle
may consume what it makes.

Shapes and distributions follow the two model sizes the xwen CLAUDE.md page
describes in "Architecture cheat sheet": 27B (16 K-heads, 48 V-heads) and
35B-A3B (16 K-heads, 32 V-heads), head dim 128, fused width 128*(2*H_k+H_v).
No dataset, checkpoint or trained weight is involved: every tensor is a seeded
draw.  Distribution conventions: N(m, s) is mean m and standard deviation s;
U(lo, hi) is uniform; ssm_a = -exp(U(0, ln 16)) is in [-16, -1].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

D = 128


@dataclass
class Case:
    """One synthetic workload.  Every tensor lives on the CPU.

    x [T][C], z [T][Hv*128], a_raw/b_raw [T][Hv] in ``act_dtype``;
    conv_w [C][4], dt_bias/ssm_a [Hv], norm_w [128] fp32;
    S0 [N][Hv][128][128] fp32; conv0 [N][3][C] in ``act_dtype``;
    cu_seqlens [N+1] int32 (prefill) -- for decode/verify, N = B and each
    sequence has K tokens (x row b*K + p); accept_len [B] int32 in 1..K.
    """
    name: str
    Hk: int
    Hv: int
    act_dtype: torch.dtype
    x: torch.Tensor
    z: torch.Tensor
    a_raw: torch.Tensor
    b_raw: torch.Tensor
    conv_w: torch.Tensor
    dt_bias: torch.Tensor
    ssm_a: torch.Tensor
    norm_w: torch.Tensor
    S0: torch.Tensor
    conv0: torch.Tensor
    cu_seqlens: torch.Tensor
    K: int = 1
    accept_len: torch.Tensor | None = None
    meta: dict = field(default_factory=dict)

    @property
    def C(self) -> int:
        return D * (2 * self.Hk + self.Hv)

    @property
    def N(self) -> int:
        return self.cu_seqlens.numel() - 1

    @property
    def T(self) -> int:
        return self.x.shape[0]


def varlen_lengths(gen: torch.Generator, n: int, total: int, lo: int, hi: int) -> list[int]:
    """Seeded lengths summing to ``total``, each in [lo, hi].

    u_i ~ U(0,1); L_i = lo + floor((total - n*lo) * u_i / sum(u)) for i < n-1,
    the last absorbs the remainder; redraw while any length exceeds ``hi``.
    """
    for _ in range(1000):
        u = torch.rand(n, generator=gen, dtype=torch.float64)
        free = total - n * lo
        L = [lo + int(math.floor(free * float(u[i]) / float(u.sum()))) for i in range(n - 1)]
        L.append(total - sum(L))
        if max(L) <= hi and min(L) >= lo:
            return L
    raise RuntimeError("could not draw lengths within bounds")


def make_case(name: str, *, Hk: int, Hv: int, lengths: list[int] | None = None,
              B: int | None = None, K: int = 1, act_dtype=torch.bfloat16,
              S0: str = "randn", conv0: str = "randn", seed: int = 0,
              varlen: tuple[int, int, int, int] | None = None) -> Case:
    """Draw a case.  Order of draws: x, W, z, a, b, dt_bias, ssm_a, norm_w,
    S0, conv0, lengths, accept.

    Prefill: pass ``lengths`` (or ``varlen=(n, total, lo, hi)`` to draw them,
    after conv0).  Decode/verify: pass ``B`` and ``K`` (T = B*K).
    """
    gen = torch.Generator().manual_seed(seed)
    if varlen is not None:
        n_seq, T = varlen[0], varlen[1]
    elif lengths is not None:
        n_seq, T = len(lengths), sum(lengths)
    else:
        assert B is not None
        n_seq, T = B, B * K
    C = D * (2 * Hk + Hv)
    f32 = torch.float32
    x = torch.randn(T, C, generator=gen, dtype=f32)
    conv_w = torch.randn(C, 4, generator=gen, dtype=f32) * 0.25
    z = torch.randn(T, Hv * D, generator=gen, dtype=f32)
    a_raw = torch.randn(T, Hv, generator=gen, dtype=f32)
    b_raw = torch.randn(T, Hv, generator=gen, dtype=f32)
    dt_bias = torch.rand(Hv, generator=gen, dtype=f32) * 3.0 - 2.0
    ssm_a = -torch.exp(torch.rand(Hv, generator=gen, dtype=f32) * math.log(16.0))
    norm_w = 1.0 + 0.1 * torch.randn(D, generator=gen, dtype=f32)
    if S0 == "randn":
        S = torch.randn(n_seq, Hv, D, D, generator=gen, dtype=f32) * 0.02
    else:
        S = torch.zeros(n_seq, Hv, D, D, dtype=f32)
    if conv0 == "randn":
        cv = torch.randn(n_seq, 3, C, generator=gen, dtype=f32)
    else:
        cv = torch.zeros(n_seq, 3, C, dtype=f32)
    if varlen is not None:
        lengths = varlen_lengths(gen, *varlen)
    if lengths is not None:
        cu = torch.zeros(n_seq + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    else:
        cu = torch.arange(0, T + 1, K, dtype=torch.int32)
    accept = None
    if B is not None:
        accept = torch.randint(1, K + 1, (n_seq,), generator=gen, dtype=torch.int64).to(torch.int32)
    ad = act_dtype
    return Case(name=name, Hk=Hk, Hv=Hv, act_dtype=ad, x=x.to(ad), z=z.to(ad),
                a_raw=a_raw.to(ad), b_raw=b_raw.to(ad), conv_w=conv_w, dt_bias=dt_bias,
                ssm_a=ssm_a, norm_w=norm_w, S0=S, conv0=cv.to(ad), cu_seqlens=cu, K=K,
                accept_len=accept)


# The five named workloads (seed 1000 + index).
def tiny_fp32() -> Case:
    """One sequence, T=128, H_k=2, H_v=4, fp32, zero initial S and conv state."""
    return make_case("tiny T=128 Hk=2 Hv=4 fp32", Hk=2, Hv=4, lengths=[128],
                     act_dtype=torch.float32, S0="zero", conv0="zero", seed=1000)


def decode_b1() -> Case:
    """Decode, batch 1, H_k=16, H_v=32, bf16 activations, fp32 state."""
    return make_case("decode B=1 Hk=16 Hv=32 bf16", Hk=16, Hv=32, B=1, K=1, seed=1001)


def prefill_t8192() -> Case:
    """Prefill, one sequence of 8192 tokens, H_k=16, H_v=48, bf16, zero state."""
    return make_case("prefill T=8192 Hk=16 Hv=48 bf16", Hk=16, Hv=48, lengths=[8192],
                     S0="zero", conv0="zero", seed=1002)


def verify_b64_k3() -> Case:
    """Batched decode with speculative verify: B=64, K=3, H_k=16, H_v=32, bf16."""
    return make_case("verify B=64 K=3 Hk=16 Hv=32 bf16", Hk=16, Hv=32, B=64, K=3, seed=1003)


def decode_b64() -> Case:
    """Batched decode, B=64, one token per sequence, H_k=16, H_v=32, bf16."""
    return make_case("decode B=64 Hk=16 Hv=32 bf16", Hk=16, Hv=32, B=64, K=1, seed=1003)


def varlen_t65536() -> Case:
    """Packed varlen prefill: 8 sequences summing to 65536 (512..24576), 16/48, bf16."""
    return make_case("varlen N=8 T=65536 Hk=16 Hv=48 bf16", Hk=16, Hv=48,
                     varlen=(8, 65536, 512, 24576), seed=1004)


NAMED = {
    "tiny": tiny_fp32,
    "decode_b1": decode_b1,
    "prefill_t8192": prefill_t8192,
    "verify_b64_k3": verify_b64_k3,
    "decode_b64": decode_b64,
    "varlen_t65536": varlen_t65536,
}


@dataclass
class ProjCase:
    """Inputs of the projections either side of the mixer (all bf16, CPU): hidden [T][H],
    W_qkv [C][H], W_z [Hv*128][H], W_a / W_b [Hv][H], y [T][Hv*128], W_out [H][Hv*128]."""
    Hk: int
    Hv: int
    H: int
    hidden: torch.Tensor
    W_qkv: torch.Tensor
    W_z: torch.Tensor
    W_a: torch.Tensor
    W_b: torch.Tensor
    y: torch.Tensor
    W_out: torch.Tensor


def make_proj_case(*, T: int, H: int, Hk: int, Hv: int, seed: int = 0) -> ProjCase:
    """hidden, y ~ N(0, 1); every weight ~ N(0, 1/sqrt(fan_in)).  Hidden sizes on the page:
    5120 (27B, 16/48) and 2048 (35B-A3B, 16/32).  Draw order: hidden, W_qkv, W_z, W_a, W_b,
    y, W_out."""
    gen = torch.Generator().manual_seed(seed)
    C, HvD = D * (2 * Hk + Hv), D * Hv
    rn = lambda *s, std=1.0: (torch.randn(*s, generator=gen) * std).to(torch.bfloat16)
    hidden = rn(T, H)
    W_qkv, W_z = rn(C, H, std=H ** -0.5), rn(HvD, H, std=H ** -0.5)
    W_a, W_b = rn(Hv, H, std=H ** -0.5), rn(Hv, H, std=H ** -0.5)
    y = rn(T, HvD)
    W_out = rn(H, HvD, std=HvD ** -0.5)
    return ProjCase(Hk, Hv, H, hidden, W_qkv, W_z, W_a, W_b, y, W_out)
