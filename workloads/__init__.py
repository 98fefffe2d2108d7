"""Seeded synthetic inputs for the fp16 GEMM workloads.

This module holds no GEMM, bias or GELU arithmetic: it only names the workloads
(shapes, value distributions, seeds) and draws their inputs. Both the CUDA path's
tests/benchmark and the CPU oracle consume the identical bits it produces.

Recipe (one reading, since the pages give none): a CPU ``torch.Generator``
seeded with the workload's seed draws A, then B, then the bias (when present),
in that order, as float32; uniform[lo, hi] is ``lo + (hi - lo) * torch.rand``,
normal(0, s) is ``s * torch.randn``; each is then rounded to float16 (to
nearest, ties to even).

The shapes stand in for the pages' own GEMM examples (4096^3 and 2048^3 fp16
tiles, 128x128x32 blocking) and for the transformer shapes they motivate (an
FFN up-projection and a decode-time skinny product).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Dist:
    kind: str          # "uniform" or "normal"
    a: float           # uniform: low;  normal: mean (always 0 here)
    b: float           # uniform: high; normal: standard deviation

    def draw(self, shape, gen: torch.Generator) -> torch.Tensor:
        if self.kind == "uniform":
            x = torch.rand(shape, generator=gen, dtype=torch.float32)
            x = self.a + (self.b - self.a) * x
        elif self.kind == "normal":
            x = self.a + self.b * torch.randn(shape, generator=gen, dtype=torch.float32)
        elif self.kind == "int":
            # integer-valued entries in [a, b] (exact in fp16 and in any fp32 sum
            # of the sizes the exact tests use)
            x = torch.randint(int(self.a), int(self.b) + 1, shape, generator=gen).to(torch.float32)
        else:
            raise ValueError(self.kind)
        return x.to(torch.float16)


U1 = Dist("uniform", -1.0, 1.0)


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    seed: int
    a_dist: Dist = U1
    b_dist: Dist = U1
    bias_dist: Dist | None = None
    gelu: bool = False
    note: str = field(default="", compare=False)

    @property
    def has_bias(self) -> bool:
        return self.bias_dist is not None

    def describe(self) -> str:
        epi = ("bias+" if self.has_bias else "") + ("gelu" if self.gelu else ("none" if not self.has_bias else ""))
        return f"{self.name}: M={self.M} N={self.N} K={self.K} epilogue={epi.rstrip('+')} seed={self.seed}"

    def inputs(self, device: str = "cpu"):
        """(A, B, bias_or_None) as contiguous float16 tensors on ``device``."""
        g = torch.Generator(device="cpu")
        g.manual_seed(self.seed)
        A = self.a_dist.draw((self.M, self.K), g)
        B = self.b_dist.draw((self.K, self.N), g)
        bias = self.bias_dist.draw((self.N,), g) if self.bias_dist is not None else None
        if device != "cpu":
            A = A.to(device)
            B = B.to(device)
            bias = bias.to(device) if bias is not None else None
        return A, B, bias

    # algorithmic work: what the method must do, each operand touched once
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def bytes(self) -> int:
        n = 2 * (self.M * self.K + self.K * self.N + self.M * self.N)
        if self.has_bias:
            n += 2 * self.N
        return n


# The five workloads. Names say what they are.
SQUARE_256 = Workload("square_256", 256, 256, 256, seed=0,
                      note="fp16 GEMM 256^3, uniform[-1,1], no epilogue")
RAGGED_GELU = Workload("ragged_1000x1030x520_bias_gelu", 1000, 1030, 520, seed=1,
                       bias_dist=Dist("uniform", -0.1, 0.1), gelu=True,
                       note="ragged shape, no dimension a multiple of 64, bias + exact-erf GELU")
SQUARE_8192 = Workload("square_8192", 8192, 8192, 8192, seed=2,
                       note="fp16 GEMM 8192^3, uniform[-1,1], no epilogue; tensor-bound")
FFN_UP = Workload("ffn_up_4096x14336x4096_bias_gelu", 4096, 14336, 4096, seed=3,
                  a_dist=Dist("normal", 0.0, 1.0), b_dist=Dist("normal", 0.0, 0.02),
                  bias_dist=Dist("normal", 0.0, 0.02), gelu=True,
                  note="FFN up-projection, tokens x hidden -> 14336, fused bias + GELU")
DECODE = Workload("decode_16x28672x8192", 16, 28672, 8192, seed=4,
                  a_dist=Dist("normal", 0.0, 1.0), b_dist=Dist("normal", 0.0, 0.02),
                  note="decode-shaped skinny GEMM; HBM-bound on reading B")

ALL = (SQUARE_256, RAGGED_GELU, SQUARE_8192, FFN_UP, DECODE)


@dataclass(frozen=True)
class W4Workload:
    """A GEMM with 4-bit weights: A (M x K) fp16; B stored as N rows of K/2
    bytes, one row per output column (two's-complement 4-bit values, low
    nibble = even k), plus one fp16 scale per column and per group of `group`
    rows of K, stored ceil(K/group) x N. The draws: A, then the 4-bit values
    q[n][k] (uniform over [-8, 7], drawn N x K), then the scales, then the
    bias, from one CPU torch.Generator seeded with `seed`."""
    name: str
    M: int
    N: int
    K: int
    seed: int
    group: int = 128
    a_dist: Dist = Dist("normal", 0.0, 1.0)
    scale_lo: float = 0.002
    scale_hi: float = 0.006
    bias_dist: Dist | None = None
    gelu: bool = False
    # "uniform": scales uniform in [scale_lo, scale_hi]; "pow2": 2^e with e
    # uniform over {-2, ..., 1} (with integer A, every product and partial sum
    # is then exact in fp32)
    scale_kind: str = "uniform"
    # weight format: "int4" (two's complement, q drawn uniform over [-8, 7]) or
    # "fp4" (E2M1 codes drawn uniform over all 16 codes)
    fmt: str = "int4"

    @property
    def fmt_code(self) -> int:
        return {"int4": 0, "fp4": 1}[self.fmt]

    @property
    def has_bias(self) -> bool:
        return self.bias_dist is not None

    def describe(self) -> str:
        epi = ("bias+" if self.has_bias else "") + ("gelu" if self.gelu else ("none" if not self.has_bias else ""))
        return (f"{self.name}: M={self.M} N={self.N} K={self.K} {self.fmt} weights, group {self.group}, "
                f"epilogue={epi.rstrip('+')} seed={self.seed}")

    def inputs(self, device: str = "cpu"):
        """(A fp16, Bq uint8 N x K/2, scales fp16 ceil(K/group) x N, bias or None)."""
        g = torch.Generator(device="cpu")
        g.manual_seed(self.seed)
        A = self.a_dist.draw((self.M, self.K), g)
        if self.fmt == "fp4":
            u = torch.randint(0, 16, (self.N, self.K), generator=g, dtype=torch.int16).to(torch.uint8)
        else:
            q = torch.randint(-8, 8, (self.N, self.K), generator=g, dtype=torch.int16)
            u = (q & 0xF).to(torch.uint8)
        Bq = (u[:, 0::2] | (u[:, 1::2] << 4)).contiguous()
        groups = (self.K + self.group - 1) // self.group
        if self.scale_kind == "pow2":
            e = torch.randint(-2, 2, (groups, self.N), generator=g).to(torch.float32)
            scales = torch.pow(2.0, e).to(torch.float16)
        elif self.scale_kind == "uniform":
            scales = (self.scale_lo + (self.scale_hi - self.scale_lo) *
                      torch.rand((groups, self.N), generator=g, dtype=torch.float32)).to(torch.float16)
        else:
            raise ValueError(self.scale_kind)
        bias = self.bias_dist.draw((self.N,), g) if self.bias_dist is not None else None
        out = [A, Bq, scales, bias]
        if device != "cpu":
            out = [t.to(device) if t is not None else None for t in out]
        return tuple(out)

    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def bytes(self) -> int:
        groups = (self.K + self.group - 1) // self.group
        n = 2 * self.M * self.K + self.K * self.N // 2 + 2 * groups * self.N + 2 * self.M * self.N
        if self.has_bias:
            n += 2 * self.N
        return n


DECODE_W4 = W4Workload("decode_w4_16x28672x8192", 16, 28672, 8192, seed=5)
DECODE_FP4 = W4Workload("decode_fp4_16x28672x8192", 16, 28672, 8192, seed=6, fmt="fp4")
W4_ALL = (DECODE_W4, DECODE_FP4)
BY_NAME = {w.name: w for w in ALL + W4_ALL}


@dataclass(frozen=True)
class AttnWorkload:
    """Attention forward O = softmax(Q K^T / sqrt(D)) V (optionally causal) on
    (batch, sequence, head, dim) fp16 tensors, the layout of the bshd example
    in the pages. Q, K, V are drawn in that order from one CPU torch.Generator
    seeded with `seed`, each normal(0, 1) then rounded to fp16.

    ``k_ramp`` > 0 draws keys whose scale grows along the sequence: the drawn
    fp16 key at position s is multiplied by (1 + k_ramp * s / 128) in float32
    and rounded to fp16 again, so later blocks of 128 keys score higher than
    earlier ones (inputs that make a running row maximum rise from block to
    block)."""
    name: str
    B: int
    S: int
    H: int
    D: int
    seed: int
    causal: bool = False
    dist: Dist = Dist("normal", 0.0, 1.0)
    k_ramp: float = 0.0

    def describe(self) -> str:
        return (f"{self.name}: batch={self.B} seq={self.S} heads={self.H} dim={self.D} "
                f"{'causal' if self.causal else 'non-causal'} seed={self.seed}")

    def inputs(self, device: str = "cpu"):
        g = torch.Generator(device="cpu")
        g.manual_seed(self.seed)
        shape = (self.B, self.S, self.H, self.D)
        if self.k_ramp:
            q = self.dist.draw(shape, g)
            k = self.dist.draw(shape, g).to(torch.float32)
            ramp = 1.0 + self.k_ramp * torch.arange(self.S, dtype=torch.float32) / 128.0
            k = (k * ramp.view(1, self.S, 1, 1)).to(torch.float16)
            out = [q, k, self.dist.draw(shape, g)]
        else:
            out = [self.dist.draw(shape, g) for _ in range(3)]
        if device != "cpu":
            out = [t.to(device) for t in out]
        return tuple(out)

    def visible_pairs(self) -> int:
        return self.S * (self.S + 1) // 2 if self.causal else self.S * self.S

    # algorithmic work: two products over the visible (query, key) pairs
    def flops(self) -> int:
        return 4 * self.B * self.H * self.D * self.visible_pairs()

    def bytes(self) -> int:
        return 2 * 4 * self.B * self.S * self.H * self.D  # Q, K, V read once, O written once


ATTN_SMALL = AttnWorkload("attn_1x256x2x128", 1, 256, 2, 128, seed=20)
ATTN_SMALL_CAUSAL = AttnWorkload("attn_1x256x2x128_causal", 1, 256, 2, 128, seed=21, causal=True)
ATTN_RAGGED = AttnWorkload("attn_2x1000x3x128_causal", 2, 1000, 3, 128, seed=22, causal=True)
# the pages' attention benchmark shape: batch 1, 32 heads, head dim 128, sequence 512..4096
ATTN_4096 = AttnWorkload("attn_1x4096x32x128", 1, 4096, 32, 128, seed=23)
ATTN_4096_CAUSAL = AttnWorkload("attn_1x4096x32x128_causal", 1, 4096, 32, 128, seed=24, causal=True)
ATTN_ALL = (ATTN_SMALL, ATTN_SMALL_CAUSAL, ATTN_RAGGED, ATTN_4096, ATTN_4096_CAUSAL)
BY_NAME.update({w.name: w for w in ATTN_ALL})


@dataclass(frozen=True)
class SoftmaxWorkload:
    """Row softmax Y = softmax(X) along each row of an M x N fp16 matrix; X is
    drawn normal(0, sigma) (logit-like) from a CPU torch.Generator seeded with
    `seed`, then rounded to fp16."""
    name: str
    M: int
    N: int
    seed: int
    dist: Dist = Dist("normal", 0.0, 3.0)

    def describe(self) -> str:
        return f"{self.name}: M={self.M} N={self.N} seed={self.seed}"

    def inputs(self, device: str = "cpu"):
        g = torch.Generator(device="cpu")
        g.manual_seed(self.seed)
        X = self.dist.draw((self.M, self.N), g)
        return (X.to(device) if device != "cpu" else X,)

    def bytes(self) -> int:
        return 2 * 2 * self.M * self.N  # X read once, Y written once


SOFTMAX_RAGGED = SoftmaxWorkload("softmax_1000x1030", 1000, 1030, seed=30)
SOFTMAX_4096 = SoftmaxWorkload("softmax_32768x4096", 32768, 4096, seed=31)
SOFTMAX_VOCAB = SoftmaxWorkload("softmax_4096x32768", 4096, 32768, seed=32)
SOFTMAX_ALL = (SOFTMAX_RAGGED, SOFTMAX_4096, SOFTMAX_VOCAB)
BY_NAME.update({w.name: w for w in SOFTMAX_ALL})


def custom(M: int, N: int, K: int, seed: int, dist: Dist = U1, bias: Dist | None = None,
           gelu: bool = False) -> Workload:
    """An ad-hoc workload (edge-shape tests) with the same generator recipe."""
    return Workload(f"custom_{M}x{N}x{K}_s{seed}", M, N, K, seed=seed, a_dist=dist, b_dist=dist,
                    bias_dist=bias, gelu=gelu)
