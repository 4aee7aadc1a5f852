"""MoE expert-FFN forward on one GB300 (sm_103a).

The computation lives in ``libmoe_gb300.so`` (C ABI in ``include/moe.h``):
align -> gathered grouped GEMM with w13 + SiLU(gate)*up -> grouped GEMM with
w2 x routing weight -> deterministic combine.  This package is its Python
binding: :mod:`._abi` has one function per C entry point, with the same name;
the helpers below only allocate device buffers with torch and call them.
"""
from __future__ import annotations

import torch

from . import _abi
from ._abi import (MOE_ACT_SILU, MOE_ACT_SWIGLU_CLAMP, MOE_BF16, MOE_E2M1_MX, MOE_E4M3, MOE_F32,
                   MoEError, Problem, moe_abi_version,
                   moe_align, moe_align_capacity, moe_align_local, moe_combine, moe_forward,
                   moe_route_align, moe_align_scratch_bytes, moe_combine_finish,
                   moe_forward_noalloc, moe_forward_noalloc_status, moe_gather_rows, moe_gemm1_silu,
                   moe_gemm1_silu_gather, moe_gemm2_default_splits,
                   moe_gemm2_weighted, moe_get_device_status, moe_mx_packed_bytes,
                   moe_pack_mx_weights, moe_quantize_gather_x_fp8, moe_quantize_x_fp8,
                   moe_resolve_block_m, moe_workspace_offsets, moe_workspace_size)

__all__ = ["MOE_ACT_SILU", "MOE_ACT_SWIGLU_CLAMP", "MoEError", "Problem", "make_problem", "dtype_code", "align", "Workspace", "forward",
           "pack_mx", "moe_forward_noalloc", "moe_forward_noalloc_status", "moe_mx_packed_bytes", "moe_pack_mx_weights",
           "moe_quantize_gather_x_fp8", "moe_gather_rows",
           "moe_abi_version", "moe_align", "moe_align_capacity", "moe_align_local",
           "moe_align_scratch_bytes", "moe_combine_finish",
           "moe_route_align", "route_align",
           "moe_combine", "moe_forward",
           "moe_gemm1_silu", "moe_gemm1_silu_gather",
           "moe_gemm2_default_splits", "moe_gemm2_weighted",
           "moe_get_device_status", "moe_quantize_x_fp8", "moe_resolve_block_m",
           "moe_workspace_offsets", "moe_workspace_size"]


def dtype_code(dt) -> int:
    if dt in (torch.float32, "f32"):
        return MOE_F32
    if dt in (torch.bfloat16, "bf16"):
        return MOE_BF16
    if dt in ("mxfp4", MOE_E2M1_MX):
        return MOE_E2M1_MX
    raise ValueError(f"unsupported dtype {dt}")


def make_problem(T, H, I, E, K, act="bf16", weight=None, block_m=0, h_scale=1.0,
                 expert_base=0, local_experts=0, activation=MOE_ACT_SILU, swiglu_alpha=1.0,
                 swiglu_limit=float("inf"), gate_up_interleaved=False, w13_bias=None,
                 w2_bias=None, fused_combine=False) -> Problem:
    """local_experts > 0: an expert-parallel shard holding experts
    [expert_base, expert_base + local_experts) of E; its weights hold those
    experts only.  activation MOE_ACT_SWIGLU_CLAMP selects the clamped
    SwiGLU (swiglu_alpha, swiglu_limit); gate_up_interleaved: w13 rows
    alternate gate and up; w13_bias (experts, 2I) / w2_bias (experts, H):
    fp32 device tensors, kept alive by the returned problem.  fused_combine:
    GEMM2 adds its rows into an fp32 accumulator (atomics) instead of the
    separate, deterministic combine."""
    a = dtype_code(act)
    w = a if weight is None else dtype_code(weight)
    for b in (w13_bias, w2_bias):
        if b is not None and (b.dtype != torch.float32 or not b.is_contiguous()):
            raise ValueError("biases are contiguous fp32 device tensors")
    lim = swiglu_limit if activation == MOE_ACT_SWIGLU_CLAMP else 0.0
    P = Problem(T, H, I, E, K, a, w, block_m, h_scale, expert_base, local_experts, activation,
                swiglu_alpha, lim, int(gate_up_interleaved),
                None if w13_bias is None else w13_bias.data_ptr(),
                None if w2_bias is None else w2_bias.data_ptr(), int(fused_combine))
    P._keep = (w13_bias, w2_bias)
    return P


def align(topk_ids: torch.Tensor, E: int, block_m: int = 128, dev_status=None, stream=None,
          expert_base: int = 0, local_experts: int = 0, many_cta: bool = True):
    """Run moe_align_local on (T, K) int32 ids; returns the outputs as a
    dict of device tensors.  many_cta: give the call the scratch with which
    batches of 16384 or more ids are aligned by many CTAs (as moe_forward
    does); False keeps the one-CTA kernel."""
    T, K = topk_ids.shape
    L = local_experts if local_experts > 0 else E
    cap = moe_align_capacity(T, K, L, block_m)
    dev = topk_ids.device
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(counts=torch.empty(L, **i32), offsets=torch.empty(L + 1, **i32),
               padded_offsets=torch.empty(L + 1, **i32), sorted_ids=torch.empty(cap, **i32),
               inv_perm=torch.empty(T * K, **i32),
               block_info=torch.empty((cap // block_m, 4), **i32),
               num_blocks=torch.empty(1, **i32))
    nbytes = moe_align_scratch_bytes(T, K, L) if many_cta else 0
    scratch = torch.empty(nbytes // 4, **i32) if nbytes > 0 else None
    moe_align_local(topk_ids, T, K, E, expert_base, L, block_m, out["counts"], out["offsets"],
                    out["padded_offsets"], out["sorted_ids"], out["inv_perm"], out["block_info"],
                    out["num_blocks"], dev_status, stream, scratch)
    return out


def route_align(logits: torch.Tensor, K: int, block_m: int = 128, dev_status=None, stream=None,
                expert_base: int = 0, local_experts: int = 0):
    """moe_route_align on (T, E) router logits (fp32 or bf16): returns the
    top-K ids and weights and the align outputs as a dict of device
    tensors."""
    T, E = logits.shape
    L = local_experts if local_experts > 0 else E
    cap = moe_align_capacity(T, K, L, block_m)
    dev = logits.device
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(topk_ids=torch.empty((T, K), **i32),
               topk_weights=torch.empty((T, K), dtype=torch.float32, device=dev),
               counts=torch.empty(L, **i32), offsets=torch.empty(L + 1, **i32),
               padded_offsets=torch.empty(L + 1, **i32), sorted_ids=torch.empty(cap, **i32),
               inv_perm=torch.empty(T * K, **i32),
               block_info=torch.empty((cap // block_m, 4), **i32),
               num_blocks=torch.empty(1, **i32))
    moe_route_align(logits.contiguous(), dtype_code(logits.dtype), T, E, K, expert_base, L,
                    block_m, out["topk_ids"], out["topk_weights"], out["counts"], out["offsets"],
                    out["padded_offsets"], out["sorted_ids"], out["inv_perm"],
                    out["block_info"], out["num_blocks"], dev_status, stream)
    return out


def pack_mx(w: torch.Tensor, w_scale: torch.Tensor, sections: int, stream=None,
            interleaved: bool = False):
    """Packed (values, scale images) of an mxfp4 weight tensor in natural form
    (E, R, K/2) + (E, R, K/32), as the block-scaled GEMMs read it; done once
    when the model is loaded."""
    E, R, half_k = w.shape
    K = 2 * half_k
    vb, sb = moe_mx_packed_bytes(E, R, K, sections)
    # tile-major: (expert, 192-row weight tile, 128-element K tile, 192, 64)
    span = 192 // sections
    tiles = -(-(R // sections) // span)
    vals = torch.empty((E, tiles, (K + 127) // 128, 192, 64), dtype=torch.uint8, device=w.device)
    assert vals.numel() == vb
    imgs = torch.empty(sb, dtype=torch.uint8, device=w.device)
    moe_pack_mx_weights(w.contiguous(), w_scale.contiguous(), E, R, K, sections, int(interleaved),
                        vals, imgs, stream)
    return vals, imgs


class Workspace:
    """A device buffer sized for one problem, with views of its parts."""

    def __init__(self, p: Problem, device="cuda"):
        self.problem = p
        self.nbytes = moe_workspace_size(p)
        if self.nbytes == 0:
            raise MoEError(_abi.MOE_ERR_INVALID_ARG, "moe_workspace_size")
        self.buffer = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.offsets, self.sizes = moe_workspace_offsets(p)

    def part(self, idx: int, dtype=torch.uint8) -> torch.Tensor:
        off, size = self.offsets[idx], self.sizes[idx]
        return self.buffer[off:off + size].view(dtype)

    @property
    def status(self) -> torch.Tensor:
        return self.part(_abi.MOE_WS_STATUS, torch.int32)[:1]


def forward(x, topk_ids, topk_weights, w13, w2, w13_scale=None, w2_scale=None, out=None,
            workspace: Workspace | None = None, weight=None, h_scale=1.0, stream=None,
            num_experts=None, expert_base=0, intermediate=None, **activation):
    """out = MoE expert FFN of x routed by (topk_ids, topk_weights).  With
    num_experts given, w13/w2 hold the experts [expert_base, expert_base +
    w13.shape[0]) of num_experts (an expert-parallel shard) and out is this
    shard's share of the layer output.  `activation`: make_problem's
    activation, swiglu_alpha, swiglu_limit, gate_up_interleaved, w13_bias,
    w2_bias, fused_combine.  MX weights (weight="mxfp4") come packed by
    pack_mx, whose tiles do not show the intermediate size: pass it as
    `intermediate`."""
    T, H = x.shape
    if weight in ("mxfp4", MOE_E2M1_MX):
        if intermediate is None:
            raise ValueError("packed MX weights: pass the intermediate size")
        L, I = w13.shape[0], intermediate
    else:
        L, I = w13.shape[0], w13.shape[1] // 2
    E = L if num_experts is None else num_experts
    K = topk_ids.shape[1]
    p = make_problem(T, H, I, E, K, x.dtype, weight, 0, h_scale, expert_base,
                     0 if num_experts is None else L, **activation)
    if workspace is None:
        workspace = Workspace(p, x.device)
    if out is None:
        out = torch.empty((T, H), dtype=x.dtype, device=x.device)
    moe_forward(p, x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, out,
                workspace.buffer, workspace.nbytes, stream)
    return out
