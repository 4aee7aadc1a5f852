"""The range-checked build, libmoe_gb300_checked.so (-DMOE_BOUNDS_CHECK), in
place of a memory checker: every index a kernel reads from its inputs or the
workspace is checked against the buffer it addresses before the access, and
a failure is reported as MOE_ERR_BOUNDS with the access skipped.

1. On valid inputs the checked build computes exactly what the product
   build computes (the checks add no arithmetic), bit for bit.
2. Corrupt routing tables (a block descriptor past the capacity or naming an
   expert that is not held, a block count past the block array, a slot past
   the capacity) given to the checked build come back as MOE_ERR_BOUNDS.
   Only the checked build ever receives such inputs: its checks guard every
   access they steer (the TMA loads they move read the fill value)."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import assert_close
import mixture_experts_grouped_02_gb300 as moe
from mixture_experts_grouped_02_gb300 import _abi
from mixture_experts_grouped_02_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked():
    assert torch.cuda.is_available()
    return _abi.checked_lib()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _status(L, st):
    return L.moe_get_device_status(_ptr(st), _stream())


def _forward(L, p, d, weights):
    w13, s13, w2, s2 = weights
    ws = moe.Workspace(p)
    ws.buffer.fill_(0xFF)
    out = torch.full((p.T, p.H), float("nan"), dtype=d.x.dtype, device="cuda")
    rc = L.moe_forward(ctypes.byref(p), _ptr(d.x), _ptr(d.topk_ids), _ptr(d.topk_weights),
                       _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), _ptr(out), _ptr(ws.buffer),
                       ws.nbytes, _stream())
    assert rc == 0, rc
    assert _status(L, ws.status) == 0
    return out


CASES = [
    # name, T, H, I, E, K, dtype, fused combine
    ("bf16", 300, 256, 320, 3, 2, "bf16", False),
    ("bf16_decode", 8, 256, 320, 8, 2, "bf16", False),
    ("tf32", 33, 128, 256, 8, 2, "f32", False),
    ("mx", 150, 320, 288, 3, 2, "mxfp4", False),
    ("bf16_fused", 300, 256, 320, 3, 2, "bf16", True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_checked_build_matches_product_build(checked, case):
    name, T, H, I, E, K, dt, fused = case
    mx = dt == "mxfp4"
    cfg = gen.MoEConfig(name, T, H, I, E, K, dt, "uniform" if mx else "normal")
    d = gen.generate(cfg, seed=81).to("cuda")
    p = moe.make_problem(T, H, I, E, K, "bf16" if mx else dt, "mxfp4" if mx else None,
                         h_scale=0.5 if mx else 1.0, fused_combine=fused)
    weights = (*moe.pack_mx(d.w13, d.w13_scale, 2), *moe.pack_mx(d.w2, d.w2_scale, 1)) if mx \
        else (d.w13, None, d.w2, None)
    got = _forward(checked, p, d, weights)
    ref = _forward(_abi.lib(), p, d, weights)
    if fused:  # atomic adds in no fixed order
        assert_close(got, ref.double().cpu().numpy(), max_abs=2e-2, rel_l2=4e-3, what=name)
    else:
        assert torch.equal(got, ref), name


@pytest.mark.parametrize("T,E,dt", [(3, 8, "bf16"), (300, 3, "bf16"), (40, 8, "f32")])
def test_checked_build_gather_in_gemm_matches_product_build(checked, T, E, dt):
    """The gate/up GEMM that gathers its token rows by index (its producer
    reads sorted_ids, checked against the capacity and T*K in this build):
    the same h from both builds."""
    H, I, K = 256, 320, 2
    cfg = gen.MoEConfig("gather", T, H, I, E, K, dt, "normal")
    d = gen.generate(cfg, seed=83).to("cuda")
    p = moe.make_problem(T, H, I, E, K, dt)
    bm = moe.moe_resolve_block_m(p)
    al = moe.align(d.topk_ids, E, bm)
    cap = moe.moe_align_capacity(T, K, E, bm)
    outs = []
    for L in (checked, _abi.lib()):
        h = torch.full((cap, I), float("nan"), dtype=d.x.dtype, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = L.moe_gemm1_silu_gather(ctypes.byref(p), _ptr(d.x), _ptr(d.w13),
                                     _ptr(al["sorted_ids"]), _ptr(al["block_info"]),
                                     _ptr(al["num_blocks"]), _ptr(h), _ptr(st), _stream())
        assert rc == 0
        assert _status(L, st) == 0
        outs.append(h.view(torch.int16 if dt == "bf16" else torch.int32))
    assert torch.equal(outs[0], outs[1])


def _stage_problem(mx=False):
    T, H, I, E, K = 150, 256, 320, 3, 2
    cfg = gen.MoEConfig("corrupt", T, H, I, E, K, "mxfp4" if mx else "bf16",
                        "uniform" if mx else "normal")
    d = gen.generate(cfg, seed=82).to("cuda")
    p = moe.make_problem(T, H, I, E, K, "bf16", "mxfp4" if mx else None)
    bm = moe.moe_resolve_block_m(p)
    al = moe.align(d.topk_ids, E, bm)
    cap = moe.moe_align_capacity(T, K, E, bm)
    return p, d, al, cap


@pytest.mark.parametrize("what", ["row_start_past_capacity", "expert_not_held",
                                  "block_count_past_array"])
@pytest.mark.parametrize("gemm", [1, 2])
def test_checked_build_reports_corrupt_block_table(checked, what, gemm):
    p, d, al, cap = _stage_problem()
    binfo = al["block_info"].clone()
    nblk = al["num_blocks"].clone()
    if what == "row_start_past_capacity":
        binfo[1, 2] = cap + 512
    elif what == "expert_not_held":
        binfo[0, 0] = p.E + 5
    else:
        nblk[0] = 1 << 20
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if gemm == 1:
        a_rows = torch.zeros((cap, p.H), dtype=torch.bfloat16, device="cuda")
        h = torch.zeros((cap, p.I), dtype=torch.bfloat16, device="cuda")
        rc = checked.moe_gemm1_silu(ctypes.byref(p), _ptr(a_rows), None, _ptr(d.w13), None,
                                    _ptr(al["sorted_ids"]), _ptr(binfo), _ptr(nblk), _ptr(h),
                                    _ptr(st), _stream())
    else:
        h = torch.zeros((cap, p.I), dtype=torch.bfloat16, device="cuda")
        y = torch.zeros((cap, p.H), dtype=torch.float32, device="cuda")
        rc = checked.moe_gemm2_weighted(ctypes.byref(p), _ptr(h), _ptr(d.w2), None,
                                        _ptr(d.topk_weights), _ptr(al["sorted_ids"]),
                                        _ptr(binfo), _ptr(nblk), _ptr(y), 1, _ptr(st), _stream())
    assert rc == 0
    assert _status(checked, st) == _abi.MOE_ERR_BOUNDS


def test_checked_build_reports_corrupt_block_table_mx(checked):
    p, d, al, cap = _stage_problem(mx=True)
    binfo = al["block_info"].clone()
    binfo[0, 2] = cap + 512
    xq = torch.zeros((cap, p.H), dtype=torch.uint8, device="cuda")
    xs = torch.ones(p.T, dtype=torch.float32, device="cuda")
    w13p, s13p = moe.pack_mx(d.w13, d.w13_scale, 2)
    hq = torch.zeros((cap, p.I), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = checked.moe_gemm1_silu(ctypes.byref(p), _ptr(xq), _ptr(xs), _ptr(w13p), _ptr(s13p),
                                _ptr(al["sorted_ids"]), _ptr(binfo), _ptr(al["num_blocks"]),
                                _ptr(hq), _ptr(st), _stream())
    assert rc == 0
    assert _status(checked, st) == _abi.MOE_ERR_BOUNDS


def test_checked_build_reports_slot_past_capacity(checked):
    p, d, al, cap = _stage_problem()
    inv = al["inv_perm"].clone()
    inv[7] = cap + 3
    y = torch.zeros((cap, p.H), dtype=torch.float32, device="cuda")
    out = torch.zeros((p.T, p.H), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = checked.moe_combine(_ptr(y), 1, cap, _ptr(inv), p.T, p.K, p.H, _abi.MOE_BF16, _ptr(out),
                             _ptr(st), _stream())
    assert rc == 0
    assert _status(checked, st) == _abi.MOE_ERR_BOUNDS
