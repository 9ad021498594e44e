"""Seeded synthetic inputs for the routed FP8 MoE FFN layer (Kimi K2 shapes).

This module is the one thing the CPU oracle and the CUDA path share. It draws
random tensors of the shapes and distributions of the workloads and stores the
expert weights in the checkpoint's storage format (e4m3 bytes with one fp32
scale per 128x128 block). It computes none of the layer's forward arithmetic:
no routing, no activation quantisation, no GEMM. The only arithmetic here is
the preparation of the synthetic FP8 checkpoint, done with torch's own
``float8_e4m3fn`` cast after clamping to the finite range.

Shapes and constants follow the pages' configuration of Kimi K2
("Kimi K2 · Architecture", Sources: config.json excerpt): hidden_size 7168,
n_routed_experts 384, num_experts_per_tok 8, moe_intermediate_size 2048,
n_shared_experts 1, routed_scaling_factor 2.827, intermediate_size 18432,
quantization_config {fmt e4m3, weight_block_size [128, 128]}.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import torch

BLOCK = 128          # weight block and activation group width (config weight_block_size)
E4M3_MAX = 448.0     # largest finite e4m3 magnitude (OCP FP8 E4M3)


@dataclass(frozen=True)
class MoEShape:
    """One routed-MoE-layer workload: T tokens through one layer."""
    name: str
    T: int
    d: int
    E: int
    topk: int
    H: int
    n_shared: int = 1
    route_scale: float = 2.827
    hot_experts: tuple = field(default_factory=tuple)   # expert ids with the hot bias
    hot_bias: float = 0.0

    @property
    def rows_routed(self) -> int:
        return self.T * self.topk


@dataclass(frozen=True)
class DenseShape:
    """The first block's dense SwiGLU FFN workload."""
    name: str
    T: int
    d: int
    H: int


def _hot(E: int, n: int) -> tuple:
    # n hot experts spread evenly over the id range
    step = E // n
    return tuple(i * step for i in range(n))


# The workloads: a toy layer the oracle runs in seconds, then the Kimi K2 layer at
# decode, prefill and two skewed-routing batches, then the dense FFN.
TOY = MoEShape("toy_t64_d1024_e32_h256", T=64, d=1024, E=32, topk=8, H=256)
DECODE = MoEShape("kimi_k2_moe_decode_t256", T=256, d=7168, E=384, topk=8, H=2048)
PREFILL = MoEShape("kimi_k2_moe_prefill_t4096", T=4096, d=7168, E=384, topk=8, H=2048)
SKEWED = MoEShape("kimi_k2_moe_skewed_t16384", T=16384, d=7168, E=384, topk=8, H=2048,
                  hot_experts=_hot(384, 16), hot_bias=0.5)
# the same mechanism with the bias that gives the hot experts about 40% of the
# routed assignments under these distributions (+0.5 gives about 90%)
SKEWED40 = MoEShape("kimi_k2_moe_skewed40_t16384", T=16384, d=7168, E=384, topk=8, H=2048,
                    hot_experts=_hot(384, 16), hot_bias=0.18)
DENSE = DenseShape("kimi_k2_dense_ffn_t8192", T=8192, d=7168, H=18432)

SHAPES = {s.name: s for s in (TOY, DECODE, PREFILL, SKEWED, SKEWED40)}


def sub_seed(seed: int, name: str, idx: int = 0) -> int:
    """Per-tensor seed derived from (seed, tensor name, index)."""
    h = hashlib.sha256(f"{seed}/{name}/{idx}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed: int, name: str, idx: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(seed, name, idx))
    return g


def randn(shape, std: float, device, seed: int, name: str, idx: int = 0,
          dtype=torch.float32) -> torch.Tensor:
    g = _gen(device, seed, name, idx)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def gen_x(T: int, d: int, seed: int = 0, device="cpu", name: str = "x") -> torch.Tensor:
    """Layer input x ~ N(0, 1), bf16 [T, d]."""
    return randn((T, d), 1.0, device, seed, name, dtype=torch.bfloat16)


def gen_residual(T: int, d: int, seed: int = 0, device="cpu", std: float = 1.0, name: str = "residual") -> torch.Tensor:
    """Residual-stream rows h ~ N(0, std^2) times a per-row factor 10^U(-1, 1)
    (rows of different magnitude, as RMSNorm sees them), bf16 [T, d]."""
    g = _gen(device, seed, name)
    f = 10.0 ** (torch.rand((T, 1), generator=g, device=device) * 2.0 - 1.0)
    return (torch.randn((T, d), generator=g, device=device) * std * f).to(torch.bfloat16)


def gen_norm_weight(d: int, seed: int = 0, device="cpu", name: str = "norm") -> torch.Tensor:
    """RMSNorm weight gamma ~ U(0.5, 1.5), bf16 [d]."""
    g = _gen(device, seed, name)
    return (torch.rand(d, generator=g, device=device) + 0.5).to(torch.bfloat16)


def gen_router(shape: MoEShape, seed: int = 0, device="cpu"):
    """Router weight W_g ~ N(0, 0.02) bf16 [E, d] and selection bias ~ N(0, 0.01) fp32 [E].

    For a skewed workload the bias of each hot expert is set to ``hot_bias``.
    """
    wg = randn((shape.E, shape.d), 0.02, device, seed, "w_gate", dtype=torch.bfloat16)
    b = randn((shape.E,), 0.01, device, seed, "e_score_correction_bias")
    if shape.hot_experts:
        b[list(shape.hot_experts)] = shape.hot_bias
    return wg, b


def fp8_blocks(w: torch.Tensor):
    """Store an fp32 matrix [R, C] as e4m3 bytes with one fp32 scale per 128x128 block.

    scale = amax(block) / 448; bytes = e4m3(w / scale) via torch's cast after
    clamping to +-448. R and C must be multiples of 128. An all-zero block gets
    scale 0 and zero bytes. Returns (uint8 [R, C], fp32 [R/128, C/128]).
    """
    R, C = w.shape
    blk = w.view(R // BLOCK, BLOCK, C // BLOCK, BLOCK)
    amax = blk.abs().amax(dim=(1, 3))
    scale = amax / E4M3_MAX
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    q = (blk / safe[:, None, :, None]).clamp_(-E4M3_MAX, E4M3_MAX)
    q = q.to(torch.float8_e4m3fn).view(torch.uint8).view(R, C)
    return q.contiguous(), scale.contiguous()


@dataclass
class ExpertWeights:
    """All experts' FP8 weights, routed experts 0..E-1 then the shared expert(s).

    w13   uint8 [E+S, 2, H, d]   gate_proj (index 0) and up_proj (index 1), nn.Linear layout
    w13_s fp32  [E+S, 2, H/128, d/128]
    w2    uint8 [E+S, d, H]      down_proj
    w2_s  fp32  [E+S, d/128, H/128]
    """
    w13: torch.Tensor
    w13_s: torch.Tensor
    w2: torch.Tensor
    w2_s: torch.Tensor

    def to(self, device) -> "ExpertWeights":
        return ExpertWeights(self.w13.to(device), self.w13_s.to(device),
                             self.w2.to(device), self.w2_s.to(device))

    def expert(self, e: int):
        """(w1, w1_s, w3, w3_s, w2, w2_s) of one expert."""
        return (self.w13[e, 0], self.w13_s[e, 0], self.w13[e, 1], self.w13_s[e, 1],
                self.w2[e], self.w2_s[e])


def gen_expert(e: int, d: int, H: int, seed: int = 0, device="cpu", std: float = 0.02, name: str = "expert"):
    """Expert e's weights: (w13 uint8 [2, H, d], w13_s [2, H/128, d/128], w2 uint8 [d, H], w2_s [d/128, H/128]).

    Each matrix has its own seed, so one expert can be regenerated alone."""
    q1, s1 = fp8_blocks(randn((H, d), std, device, seed, f"{name}.w1", e))
    q3, s3 = fp8_blocks(randn((H, d), std, device, seed, f"{name}.w3", e))
    q2, s2 = fp8_blocks(randn((d, H), std, device, seed, f"{name}.w2", e))
    return torch.stack([q1, q3]), torch.stack([s1, s3]), q2, s2


def gen_experts(n_experts: int, d: int, H: int, seed: int = 0, device="cpu",
                std: float = 0.02, name: str = "expert", only=None) -> ExpertWeights:
    """n_experts SwiGLU experts with weights ~ N(0, std) stored as block-scaled e4m3.

    ``only``: generate just these expert ids (the others stay zero)."""
    w13 = torch.zeros((n_experts, 2, H, d), dtype=torch.uint8, device=device)
    w13_s = torch.zeros((n_experts, 2, H // BLOCK, d // BLOCK), dtype=torch.float32, device=device)
    w2 = torch.zeros((n_experts, d, H), dtype=torch.uint8, device=device)
    w2_s = torch.zeros((n_experts, d // BLOCK, H // BLOCK), dtype=torch.float32, device=device)
    for e in (range(n_experts) if only is None else sorted(set(only))):
        a, b, c, f = gen_expert(e, d, H, seed, device, std, name)
        w13[e].copy_(a)
        w13_s[e].copy_(b)
        w2[e].copy_(c)
        w2_s[e].copy_(f)
    return ExpertWeights(w13, w13_s, w2, w2_s)


@dataclass
class MoEInputs:
    shape: MoEShape
    x: torch.Tensor        # bf16 [T, d]
    w_gate: torch.Tensor   # bf16 [E, d]
    bias: torch.Tensor     # fp32 [E]
    experts: ExpertWeights


def gen_moe_inputs(shape: MoEShape, seed: int = 0, device="cpu") -> MoEInputs:
    x = gen_x(shape.T, shape.d, seed, device)
    wg, b = gen_router(shape, seed, device)
    ex = gen_experts(shape.E + shape.n_shared, shape.d, shape.H, seed, device)
    return MoEInputs(shape, x, wg, b, ex)


@dataclass
class DenseInputs:
    shape: DenseShape
    x: torch.Tensor        # bf16 [T, d]
    w13: torch.Tensor      # uint8 [2, H, d]
    w13_s: torch.Tensor    # fp32 [2, H/128, d/128]
    w2: torch.Tensor       # uint8 [d, H]
    w2_s: torch.Tensor     # fp32 [d/128, H/128]


def gen_dense_inputs(shape: DenseShape, seed: int = 0, device="cpu") -> DenseInputs:
    x = gen_x(shape.T, shape.d, seed, device, name="x_dense")
    ex = gen_experts(1, shape.d, shape.H, seed, device, name="dense")
    return DenseInputs(shape, x, ex.w13[0], ex.w13_s[0], ex.w2[0], ex.w2_s[0])
