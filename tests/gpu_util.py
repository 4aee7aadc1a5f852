"""Helpers for the GPU parity tests: input preparation for the oracle and the
comparison rule.  The oracle gets host copies of the very inputs the GPU got;
nothing the CUDA path computes is fed to the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mixture_experts_grouped_02_gb300 import inputs as gen

# bf16 (and tf32) output bounds stated for the workload: max-abs 2e-2 and
# relative L2 1e-2 against the fp64 oracle.
MAX_ABS = 2e-2
REL_L2 = 1e-2


def np_store(t):
    return gen.to_numpy_storage(t)


def generate(cfg, seed=0, device="cuda"):
    return gen.generate(cfg, seed=seed, device=device)


def activation_kw(inp: gen.MoEInputs, experts=None):
    """The oracle's activation arguments for `inp` (its biases restricted to
    `experts`, in that order, when given)."""
    if inp.cfg.activation != "swiglu_oai":
        return {}
    sel = slice(None) if experts is None else np.asarray(experts)
    return dict(activation=oracle.ACT_SWIGLU_CLAMP, swiglu_alpha=inp.swiglu_alpha,
                swiglu_limit=inp.swiglu_limit, gate_up_interleaved=True,
                w13_bias=inp.w13_bias.cpu().numpy()[sel], w2_bias=inp.w2_bias.cpu().numpy()[sel])


def problem_kw(inp: gen.MoEInputs):
    """The library's make_problem arguments for the activation of `inp`."""
    if inp.cfg.activation != "swiglu_oai":
        return {}
    import mixture_experts_grouped_02_gb300 as moe
    return dict(activation=moe.MOE_ACT_SWIGLU_CLAMP, swiglu_alpha=inp.swiglu_alpha,
                swiglu_limit=inp.swiglu_limit, gate_up_interleaved=True,
                w13_bias=inp.w13_bias, w2_bias=inp.w2_bias)


def oracle_problem(inp: gen.MoEInputs, E=None, quantize_x=False, h_e4m3=False, h_scale=1.0,
                   experts=None):
    c = inp.cfg
    xs = np_store(inp.x[:1])
    ws = np_store(inp.w13[:1])
    return oracle.make_problem(c.T, c.H, c.I, c.E if E is None else E, c.K, xs, ws,
                               quantize_x=quantize_x, h_e4m3=h_e4m3, h_scale=h_scale,
                               **activation_kw(inp, experts))


def oracle_forward_tokens(inp: gen.MoEInputs, tokens, mode=oracle.EXACT, **kw):
    """Oracle output rows for `tokens`, copying to the host only the experts
    those tokens use (ids are renumbered into that subset)."""
    tokens = np.asarray(tokens, np.int32)
    ids = inp.topk_ids.cpu().numpy()
    used = np.unique(ids[tokens])
    remap = np.full(inp.cfg.E, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    sub_ids = remap[ids]
    sub_ids[sub_ids < 0] = 0  # rows of tokens not evaluated
    sel = torch.as_tensor(used, device=inp.w13.device, dtype=torch.long)
    w13 = np_store(inp.w13.index_select(0, sel))
    w2 = np_store(inp.w2.index_select(0, sel))
    s13 = None if inp.w13_scale is None else np_store(inp.w13_scale.index_select(0, sel))
    s2 = None if inp.w2_scale is None else np_store(inp.w2_scale.index_select(0, sel))
    P = oracle_problem(inp, E=len(used), experts=used, **kw)
    return oracle.forward(P, np_store(inp.x), sub_ids, inp.topk_weights.cpu().numpy(), w13, w2,
                          s13, s2, mode=mode, tokens=tokens)


def errors(gpu: torch.Tensor, ref: np.ndarray):
    g = gpu.detach().to(torch.float64).cpu().numpy()
    diff = g - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(gpu, ref, max_abs=MAX_ABS, rel_l2=REL_L2, what=""):
    assert np.all(np.isfinite(gpu.detach().float().cpu().numpy())), f"{what}: non-finite output"
    m, r = errors(gpu, ref)
    assert m <= max_abs and r <= rel_l2, f"{what}: max-abs {m:.3g} (<= {max_abs}), " \
                                         f"rel-L2 {r:.3g} (<= {rel_l2})"
    return m, r


def sample_tokens(T, n, seed=0):
    rng = np.random.default_rng(seed)
    picks = {0, T - 1}
    while len(picks) < min(n, T):
        picks.add(int(rng.integers(0, T)))
    return np.array(sorted(picks), np.int32)


def block_tokens(inp: gen.MoEInputs, block_m: int, n_random: int = 8, seed: int = 0,
                 expert_base: int = 0, local_experts: int = 0):
    """Tokens that together touch every align block of the routing in `inp`:
    the token of the first and of the last valid slot of each block (so
    every active expert, every tile of the GEMMs' persistent schedule and
    every K split is reached by a checked row), plus `n_random` sampled
    tokens.  The blocks come from the oracle's align of the same ids."""
    c = inp.cfg
    ids = inp.topk_ids.cpu().numpy()
    al = oracle.align(ids, c.E, block_m, expert_base=expert_base, local_experts=local_experts)
    s = al["sorted_ids"]
    picks = set(sample_tokens(c.T, n_random, seed).tolist())
    for b in range(al["num_blocks"]):
        first, valid = int(al["block_info"][b][2]), int(al["block_info"][b][3])
        picks.add(int(s[first]) // c.K)
        picks.add(int(s[first + valid - 1]) // c.K)
    return np.array(sorted(picks), np.int32), al["num_blocks"]
