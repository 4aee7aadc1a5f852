"""moe_forward_noalloc: the forward for callers that cannot allocate device
memory where they run the layer (a framework that owns all device memory, a
serving loop that must not allocate after start-up).  It keeps its
intermediates in the library's own static scratch array instead of a
caller workspace.

Called through the C ABI and compared with moe_forward (which uses a
workspace) on two calls in a row with different inputs, so that a result
left over from the first call in the shared array would show up in the
second.  This file is collected last."""
import numpy as np
import pytest
import torch

import mixture_experts_grouped_02_gb300 as moe
from mixture_experts_grouped_02_gb300 import _abi
from mixture_experts_grouped_02_gb300 import inputs as gen
from gpu_util import MAX_ABS, REL_L2, errors

pytestmark = pytest.mark.gpu


def _reference(p, d):
    ws = moe.Workspace(p)
    out = torch.empty((p.T, p.H), dtype=d.x.dtype, device="cuda")
    moe.moe_forward(p, d.x, d.topk_ids, d.topk_weights, d.w13, None, d.w2, None, out, ws.buffer,
                    ws.nbytes)
    assert moe.moe_get_device_status(ws.status) == 0
    return out


def test_noalloc_matches_forward_on_two_calls():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    cfg = gen.MoEConfig("noalloc", 96, 256, 384, 8, 2, "bf16", "normal")
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.dtype)
    assert moe.moe_workspace_size(p) <= _abi.MOE_STATIC_SCRATCH_BYTES
    for seed in (1, 2):  # two calls in a row, different inputs
        d = gen.generate(cfg, seed=seed, device="cuda")
        ref = _reference(p, d)
        out = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        _abi.moe_forward_noalloc(p, d.x, d.topk_ids, d.topk_weights, d.w13, None, d.w2, None,
                                 out)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        m, r = errors(out, ref.double().cpu().numpy())
        assert m <= MAX_ABS and r <= REL_L2, (seed, m, r)


def test_noalloc_rejects_problems_beyond_its_scratch():
    big = moe.make_problem(4096, 4096, 14336, 8, 2, "bf16")
    assert moe.moe_workspace_size(big) > _abi.MOE_STATIC_SCRATCH_BYTES
    with pytest.raises(moe.MoEError) as ei:
        _abi.moe_forward_noalloc(big, 0, 0, 0, 0, None, 0, None, 0)
    assert ei.value.status == _abi.MOE_ERR_WORKSPACE
