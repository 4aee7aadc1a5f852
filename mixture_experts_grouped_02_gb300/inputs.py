"""Seeded synthetic workloads for the MoE expert-FFN forward.

This module only draws inputs: activations, expert weights and the router's
top-k choice.  It holds no step of the forward pass itself, so the CUDA path
and the CPU oracle can both consume what it makes without sharing any of the
method's arithmetic.

Workload shapes (all synthetic; the pages use no dataset):

=================  ======  =====  =====  ===  ==  ======  ================
name               T       H      I      E    K   dtype   router logits
=================  ======  =====  =====  ===  ==  ======  ================
tiny               16      128    256    8    2   fp32    N(0,1)
mixtral_prefill    4096    4096   14336  8    2   bf16    N(0,1)
dsv3_prefill       8192    7168   2048   256  8   bf16    N(0,1)+Zipf bias
mixtral_decode_T*  1..128  4096   14336  8    2   bf16    N(0,1)
dsv3_decode_T*     1..128  7168   2048   256  8   bf16    N(0,1)+Zipf bias
lowp               2048    2880   2880   128  4   mxfp4   U(0,1)
lowp_oai           2048    2880   2880   128  4   mxfp4   U(0,1)
=================  ======  =====  =====  ===  ==  ======  ================

``lowp_oai`` is the same layer with GPT-OSS's expert FFN as the "MOE Bmm1
Fused Gather" example benchmarks it: the clamped SwiGLU with alpha =
U(0,1)/5 + 1 and limit = U(0,1)/5 + 1.3, gate and linear rows of w13
interleaved, a per-expert fp32 w13 bias ~ N(0,1), fp8 hidden activation
with out-scale U(0,1) + 3.5 (the example's y_scale).  The w2 bias ~ N(0,1)
is this workload's reading (the example benchmarks the first GEMM only).

Values: x ~ N(0,1); w13 ~ N(0, 1/sqrt(H)), w2 ~ N(0, 1/sqrt(I)) (standard
deviation 1/sqrt(fan_in)), drawn in fp32 and rounded to nearest-even into
the storage type.  The router takes a softmax over the experts in fp32,
keeps the k largest probabilities (ties to the lower expert id) and
renormalises them to sum to one.  The Zipf bias follows the skewed-routing
generator of the "MOE Bmm1 Fused Gather" example (make_prod_like_logits):
expert popularity p_r proportional to r^-1.1 over ranks r = 1..E, assigned to
experts by a seeded permutation, added to the logits as ln p.  Its cluster,
batch-hot and Gumbel terms are not part of these workloads.

mxfp4 weights (``lowp``) are quantised here, once, following the OCP
Microscaling v1.0 format: per block of 32 K elements the shared exponent is
floor(log2(amax)) - 2 (2 is e2m1's largest exponent), stored as e8m0; each
element is rounded to nearest-even on the e2m1 grid with saturation.  Both
sides consume the same bytes.

Every tensor is drawn from its own generator, seeded from
(seed, tensor id, expert), so one expert's weights can be drawn without the
others and the result does not depend on chunking.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    K: int
    dtype: str  # "f32" | "bf16" | "mxfp4"
    routing: str  # "normal" | "zipf" | "uniform"
    activation: str = "silu"  # "silu" | "swiglu_oai" (clamped, biases, interleaved w13)

    @property
    def n_assign(self) -> int:
        return self.T * self.K

    @property
    def flops(self) -> int:
        """Algorithmic FLOPs: 2*Na*H*2I (gate+up) + 2*Na*I*H (down)."""
        return 6 * self.T * self.K * self.H * self.I

    def with_tokens(self, T: int) -> "MoEConfig":
        return dataclasses.replace(self, T=T, name=f"{self.name}@T{T}")


_BASE = {
    "tiny": MoEConfig("tiny", 16, 128, 256, 8, 2, "f32", "normal"),
    "mixtral_prefill": MoEConfig("mixtral_prefill", 4096, 4096, 14336, 8, 2, "bf16", "normal"),
    "dsv3_prefill": MoEConfig("dsv3_prefill", 8192, 7168, 2048, 256, 8, "bf16", "zipf"),
    "lowp": MoEConfig("lowp", 2048, 2880, 2880, 128, 4, "mxfp4", "uniform"),
    "lowp_oai": MoEConfig("lowp_oai", 2048, 2880, 2880, 128, 4, "mxfp4", "uniform",
                          "swiglu_oai"),
}
DECODE_T = (1, 8, 32, 128)
for _t in DECODE_T:
    _BASE[f"mixtral_decode_T{_t}"] = MoEConfig(f"mixtral_decode_T{_t}", _t, 4096, 14336, 8, 2,
                                               "bf16", "normal")
    _BASE[f"dsv3_decode_T{_t}"] = MoEConfig(f"dsv3_decode_T{_t}", _t, 7168, 2048, 256, 8, "bf16",
                                            "zipf")
CONFIGS = dict(_BASE)


def config(name: str) -> MoEConfig:
    return CONFIGS[name]


# tensor ids for sub-seeding
_X, _W13, _W2, _LOGITS, _ZIPF, _B13, _B2, _OAI = 1, 2, 3, 4, 5, 6, 7, 8


def _generator(seed: int, tensor_id: int, part: int, device) -> torch.Generator:
    ss = np.random.SeedSequence([int(seed), tensor_id, int(part)])
    g = torch.Generator(device=device)
    g.manual_seed(int(ss.generate_state(1, dtype=np.uint64)[0] & ((1 << 63) - 1)))
    return g


@dataclasses.dataclass
class MoEInputs:
    cfg: MoEConfig
    x: torch.Tensor  # (T, H) fp32 or bf16
    w13: torch.Tensor  # (E, 2I, H) fp32/bf16, or (E, 2I, H/2) uint8 packed e2m1
    w2: torch.Tensor  # (E, H, I) fp32/bf16, or (E, H, I/2) uint8
    topk_ids: torch.Tensor  # (T, K) int32
    topk_weights: torch.Tensor  # (T, K) fp32
    w13_scale: torch.Tensor | None = None  # (E, 2I, H/32) uint8 e8m0
    w2_scale: torch.Tensor | None = None  # (E, H, I/32) uint8 e8m0
    # activation "swiglu_oai" only: rows of w13 (and w13_bias) alternate
    # gate / linear; scalars of the clamped SwiGLU and the fp8 out-scale
    w13_bias: torch.Tensor | None = None  # (E, 2I) fp32, w13's row order
    w2_bias: torch.Tensor | None = None  # (E, H) fp32
    swiglu_alpha: float = 1.0
    swiglu_limit: float = float("inf")
    h_scale: float = 1.0

    @property
    def interleaved(self) -> bool:
        return self.cfg.activation == "swiglu_oai"

    def to(self, device) -> "MoEInputs":
        mv = lambda t: None if t is None else t.to(device)
        return dataclasses.replace(
            self, x=mv(self.x), w13=mv(self.w13), w2=mv(self.w2), topk_ids=mv(self.topk_ids),
            topk_weights=mv(self.topk_weights), w13_scale=mv(self.w13_scale),
            w2_scale=mv(self.w2_scale), w13_bias=mv(self.w13_bias), w2_bias=mv(self.w2_bias))


def _storage_dtype(cfg: MoEConfig):
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


def draw_x(cfg: MoEConfig, seed: int = 0, device="cpu") -> torch.Tensor:
    g = _generator(seed, _X, 0, device)
    x = torch.randn((cfg.T, cfg.H), generator=g, device=device, dtype=torch.float32)
    return x.to(_storage_dtype(cfg))


def draw_expert_weight(cfg: MoEConfig, which: str, e: int, seed: int = 0, device="cpu"):
    """fp32 draw of one expert's w13 (2I, H) or w2 (H, I) before storage rounding."""
    if which == "w13":
        shape, fan_in, tid = (2 * cfg.I, cfg.H), cfg.H, _W13
    else:
        shape, fan_in, tid = (cfg.H, cfg.I), cfg.I, _W2
    g = _generator(seed, tid, e, device)
    w = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return w * (1.0 / math.sqrt(fan_in))


def quantize_mxfp4(w: torch.Tensor):
    """OCP MX e2m1 + e8m0 quantisation along the last dim (a multiple of 32).

    Returns (packed uint8 (..., C/2), scale uint8 (..., C/32)); the lower K
    index sits in the low nibble."""
    *lead, C = w.shape
    assert C % 32 == 0
    b = w.reshape(*lead, C // 32, 32).to(torch.float32)
    amax = b.abs().amax(dim=-1)
    # floor(log2(amax)) exactly: frexp gives amax = m * 2^ex with m in [0.5, 1)
    _, ex = torch.frexp(amax)
    shared = (ex.to(torch.int32) - 1) - 2
    code = torch.where(amax > 0, shared + 127, torch.zeros_like(shared)).clamp(0, 254)
    scale = torch.ldexp(torch.ones_like(amax), (code - 127).to(torch.float32))
    v = b / scale.unsqueeze(-1)
    grid = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], device=w.device)
    a = v.abs().clamp(max=6.0)
    # nearest grid point; on an exact tie take the even code (lower index
    # when the lower code is even)
    hi = torch.searchsorted(grid, a.contiguous()).clamp(1, 7)
    lo = hi - 1
    dlo = a - grid[lo]
    dhi = grid[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    mag = torch.where(pick_hi, hi, lo)
    mag = torch.where(a == 0, torch.zeros_like(mag), mag)
    sign = ((v < 0) & (mag > 0)).to(torch.int64)
    nib = (sign << 3 | mag).to(torch.uint8).reshape(*lead, C)
    packed = nib[..., 0::2] | (nib[..., 1::2] << 4)
    return packed.contiguous(), code.to(torch.uint8).contiguous()


def draw_weights(cfg: MoEConfig, seed: int = 0, device="cpu", experts=None):
    """(w13, w2, w13_scale, w2_scale) for all experts (or the listed ones,
    which still get the values they would get in the full draw)."""
    experts = range(cfg.E) if experts is None else experts
    w13s, w2s, s13, s2 = [], [], [], []
    for e in experts:
        a = draw_expert_weight(cfg, "w13", e, seed, device)
        b = draw_expert_weight(cfg, "w2", e, seed, device)
        if cfg.dtype == "mxfp4":
            qa, sa = quantize_mxfp4(a)
            qb, sb = quantize_mxfp4(b)
            w13s.append(qa), s13.append(sa), w2s.append(qb), s2.append(sb)
        else:
            w13s.append(a.to(_storage_dtype(cfg)))
            w2s.append(b.to(_storage_dtype(cfg)))
        del a, b
    w13 = torch.stack(w13s)
    w2 = torch.stack(w2s)
    if cfg.dtype == "mxfp4":
        return w13, w2, torch.stack(s13), torch.stack(s2)
    return w13, w2, None, None


def router_logits(cfg: MoEConfig, seed: int = 0, device="cpu") -> torch.Tensor:
    g = _generator(seed, _LOGITS, 0, device)
    if cfg.routing == "uniform":
        logits = torch.rand((cfg.T, cfg.E), generator=g, device=device, dtype=torch.float32)
    else:
        logits = torch.randn((cfg.T, cfg.E), generator=g, device=device, dtype=torch.float32)
    if cfg.routing == "zipf":
        logits = logits + zipf_bias(cfg.E, seed, device)
    return logits


def zipf_bias(E: int, seed: int = 0, device="cpu", s: float = 1.1) -> torch.Tensor:
    ranks = torch.arange(1, E + 1, dtype=torch.float64)
    p = ranks.pow(-s)
    p = p / p.sum()
    g = _generator(seed, _ZIPF, 0, "cpu")
    perm = torch.randperm(E, generator=g)
    bias = torch.empty(E, dtype=torch.float64)
    bias[perm] = p.log()
    return bias.to(torch.float32).to(device)


def route(logits: torch.Tensor, K: int):
    """softmax -> top-k (ties to the lower expert id) -> renormalise."""
    p = torch.softmax(logits.to(torch.float32), dim=-1)
    order = torch.sort(-p, dim=-1, stable=True).indices[:, :K]
    pk = torch.gather(p, 1, order)
    w = pk / pk.sum(dim=-1, keepdim=True)
    return order.to(torch.int32).contiguous(), w.to(torch.float32).contiguous()


def generate(cfg: MoEConfig | str, seed: int = 0, device="cpu") -> MoEInputs:
    if isinstance(cfg, str):
        cfg = config(cfg)
    x = draw_x(cfg, seed, device)
    w13, w2, s13, s2 = draw_weights(cfg, seed, device)
    ids, w = route(router_logits(cfg, seed, device), cfg.K)
    inp = MoEInputs(cfg, x.contiguous(), w13.contiguous(), w2.contiguous(), ids, w, s13, s2)
    if cfg.activation == "swiglu_oai":
        draw_swiglu_oai(inp, seed, device)
    return inp


def draw_swiglu_oai(inp: MoEInputs, seed: int = 0, device="cpu") -> None:
    """Biases and scalars of the GPT-OSS expert FFN (see the module doc)."""
    cfg = inp.cfg
    inp.w13_bias = torch.randn((cfg.E, 2 * cfg.I), generator=_generator(seed, _B13, 0, device),
                               device=device, dtype=torch.float32)
    inp.w2_bias = torch.randn((cfg.E, cfg.H), generator=_generator(seed, _B2, 0, device),
                              device=device, dtype=torch.float32)
    u = torch.rand(3, generator=_generator(seed, _OAI, 0, "cpu"), dtype=torch.float32)
    # held as fp32 values, the precision the GPU path takes them in
    inp.swiglu_alpha = float(np.float32(float(u[0]) / 5.0 + 1.0))
    inp.swiglu_limit = float(np.float32(float(u[1]) / 5.0 + 1.3))
    inp.h_scale = float(np.float32(float(u[2]) + 3.5))


def to_numpy_storage(t: torch.Tensor | None):
    """Raw storage view for the oracle: bf16 -> uint16 bits, others as is."""
    if t is None:
        return None
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
