"""moe_forward_noalloc: the forward for callers that cannot allocate device
memory where they run the layer -- a host framework that owns and pre-carves
all device memory, or a serving loop that must not allocate after start-up
(an allocation can block, synchronise the device or fail under memory
pressure).  It keeps its intermediates in the library's own static device
array instead of a caller workspace.

Every call here goes through the C ABI.  The array is shared by all calls and
keeps the previous call's contents, so the checks run several calls in a row
with different inputs and layouts (another T, the fused combine, a bad expert
id) and compare each with moe_forward on a workspace of its own: the default
combine runs the same deterministic launches, so the outputs must match bit
for bit.  This file is collected last."""
import numpy as np
import pytest
import torch

import mixture_experts_grouped_02_gb300 as moe
from mixture_experts_grouped_02_gb300 import _abi
from mixture_experts_grouped_02_gb300 import inputs as gen
from gpu_util import assert_close, oracle_forward_tokens

pytestmark = pytest.mark.gpu


def _problem(cfg, fused=False):
    return moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.dtype, fused_combine=fused)


def _with_workspace(p, d):
    ws = moe.Workspace(p)
    out = torch.empty((p.T, p.H), dtype=d.x.dtype, device="cuda")
    moe.moe_forward(p, d.x, d.topk_ids, d.topk_weights, d.w13, None, d.w2, None, out, ws.buffer,
                    ws.nbytes)
    assert moe.moe_get_device_status(ws.status) == 0
    return out


def _noalloc(p, d):
    out = torch.full((p.T, p.H), float("nan"), dtype=d.x.dtype, device="cuda")
    _abi.moe_forward_noalloc(p, d.x, d.topk_ids, d.topk_weights, d.w13, None, d.w2, None, out)
    assert _abi.moe_forward_noalloc_status() == 0
    return out


def _setup():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


def test_noalloc_matches_forward_on_calls_in_a_row():
    _setup()
    big = gen.MoEConfig("noalloc", 96, 256, 384, 8, 2, "bf16", "normal")
    small = gen.MoEConfig("noalloc_small", 40, 256, 384, 8, 2, "bf16", "normal")
    assert moe.moe_workspace_size(_problem(big)) <= _abi.MOE_STATIC_SCRATCH_BYTES
    # two calls with different inputs, then a smaller batch whose align
    # outputs and rows land on what the larger one left in the array
    for n, (cfg, seed) in enumerate(((big, 1), (big, 2), (small, 3))):
        inp = gen.generate(cfg, seed=seed)
        d = inp.to("cuda")
        p = _problem(cfg)
        out = _noalloc(p, d)
        assert torch.equal(out, _with_workspace(p, d)), (cfg.name, seed)
        if n == 0:  # and once against the oracle itself
            assert_close(out, oracle_forward_tokens(inp, np.arange(cfg.T)), what="noalloc")


def test_noalloc_fused_combine_after_default():
    """The fused combine's accumulator shares the array with the default
    path's y rows; its zeroing must not depend on what the last call left."""
    _setup()
    cfg = gen.MoEConfig("noalloc_fused", 96, 256, 384, 8, 2, "bf16", "normal")
    for seed, fused in ((4, False), (5, True), (6, True), (7, False)):
        inp = gen.generate(cfg, seed=seed)
        d = inp.to("cuda")
        p = _problem(cfg, fused)
        out = _noalloc(p, d)
        if fused:  # atomic adds in no fixed order: within the bounds of the oracle
            assert_close(out, oracle_forward_tokens(inp, np.arange(cfg.T)), what="fused")
            det = _with_workspace(_problem(cfg), d)
            assert_close(out, det.double().cpu().numpy(), max_abs=2e-2, rel_l2=4e-3,
                         what="fused vs default")
        else:
            assert torch.equal(out, _with_workspace(p, d))


def test_noalloc_bad_id_reported_through_its_status():
    """An expert id outside [0, E): the call returns MOE_OK (the kernels find
    the error), the array's status word says MOE_ERR_DEVICE_BAD_ID, later
    stages skip their writes; the next good call clears the word."""
    _setup()
    cfg = gen.MoEConfig("noalloc_bad", 64, 128, 256, 4, 2, "bf16", "normal")
    d = gen.generate(cfg, seed=8).to("cuda")
    p = _problem(cfg)
    bad = d.topk_ids.clone()
    bad[5, 1] = cfg.E
    out = torch.zeros((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    _abi.moe_forward_noalloc(p, d.x, bad, d.topk_weights, d.w13, None, d.w2, None, out)
    assert _abi.moe_forward_noalloc_status() == _abi.MOE_ERR_DEVICE_BAD_ID
    assert (out == 0).all()  # the combine did not run
    good = _noalloc(p, d)
    assert torch.equal(good, _with_workspace(p, d))


def test_noalloc_rejects_like_forward_and_beyond_its_scratch():
    big = moe.make_problem(4096, 4096, 14336, 8, 2, "bf16")
    assert moe.moe_workspace_size(big) > _abi.MOE_STATIC_SCRATCH_BYTES
    with pytest.raises(moe.MoEError) as ei:
        _abi.moe_forward_noalloc(big, 0, 0, 0, 0, None, 0, None, 0)
    assert ei.value.status == _abi.MOE_ERR_WORKSPACE
    # argument errors: the codes moe_forward gives
    odd = moe.make_problem(16, 100, 256, 8, 2, "bf16")  # H not a multiple of 64
    with pytest.raises(moe.MoEError) as ei:
        _abi.moe_forward_noalloc(odd, 0, 0, 0, 0, None, 0, None, 0)
    assert ei.value.status == _abi.MOE_ERR_UNSUPPORTED
