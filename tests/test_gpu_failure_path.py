"""The grouped GEMMs' failure path on the GPU, driven without any risk of a
hang: moe_test_gemm_wait_timeout launches a GEMM whose producers issue no
copies at all, with a pipeline wait limit of a few milliseconds.  Nothing is
ever in flight, so the first wait of every CTA runs out; the kernel must
raise its abort flag, free its tensor memory, write MOE_ERR_TIMEOUT to the
status word and return without writing its output.  A later stage given the
same status word must skip its writes, and the next ordinary forward on the
same device must still match the oracle (the tensor memory was freed and the
context is healthy)."""
import time

import numpy as np
import pytest
import torch

from gpu_util import assert_close, oracle_forward_tokens
import mixture_experts_grouped_02_gb300 as moe
from mixture_experts_grouped_02_gb300 import _abi
from mixture_experts_grouped_02_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

WAIT_LIMIT_NS = 2_000_000  # 2 ms

CASES = [
    # name, T, H, I, E, K, dtype, gemm, k_splits
    ("bf16_gate_up", 300, 256, 320, 3, 2, "bf16", 1, 1),
    ("bf16_gate_up_decode", 8, 256, 320, 8, 2, "bf16", 1, 1),  # two K steps per stage
    ("bf16_down_split", 300, 256, 320, 3, 2, "bf16", 2, 2),
    ("tf32_down", 40, 128, 256, 8, 2, "f32", 2, 1),
    ("mx_gate_up", 150, 320, 288, 3, 2, "mxfp4", 1, 1),
    ("mx_down", 150, 320, 288, 3, 2, "mxfp4", 2, 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_gemm_wait_timeout_reports_and_recovers(case):
    name, T, H, I, E, K, dt, gemm, splits = case
    assert torch.cuda.is_available()
    mx = dt == "mxfp4"
    cfg = gen.MoEConfig(name, T, H, I, E, K, dt, "uniform" if mx else "normal")
    inp = gen.generate(cfg, seed=71)
    d = inp.to("cuda")
    p = moe.make_problem(T, H, I, E, K, "bf16" if mx else dt, "mxfp4" if mx else None)
    bm = moe.moe_resolve_block_m(p)
    al = moe.align(d.topk_ids, E, bm)
    cap = moe.moe_align_capacity(T, K, E, bm)
    act = torch.bfloat16 if (mx or dt == "bf16") else torch.float32
    # operands: never read by a starved kernel, but shaped as the call needs
    if gemm == 1:
        a_rows = torch.zeros((cap, H), dtype=torch.uint8 if mx else act, device="cuda")
        xs = torch.ones(T, dtype=torch.float32, device="cuda") if mx else None
        w, ws = moe.pack_mx(d.w13, d.w13_scale, 2) if mx else (d.w13, None)
        out = torch.full((cap, I), 0x5A, dtype=torch.uint8, device="cuda")
    else:
        a_rows = torch.zeros((cap, I), dtype=torch.uint8 if mx else act, device="cuda")
        xs = None
        w, ws = moe.pack_mx(d.w2, d.w2_scale, 1) if mx else (d.w2, None)
        out = torch.full((splits * cap * H,), float("nan"), dtype=torch.float32, device="cuda")
    before = out.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    _abi.moe_test_gemm_wait_timeout(p, gemm, a_rows, xs, w, ws, d.topk_weights,
                                    al["sorted_ids"], al["block_info"], al["num_blocks"], out,
                                    splits, WAIT_LIMIT_NS, st)
    status = moe.moe_get_device_status(st)
    elapsed = time.perf_counter() - t0
    assert status == _abi.MOE_ERR_TIMEOUT, status
    assert elapsed < 2.0, elapsed  # gave up after the short limit, not the default 2 s
    assert torch.equal(out.view(torch.uint8), before.view(torch.uint8))  # nothing written

    # a later stage that finds the status word set skips its writes
    y = torch.zeros((1, cap, H), dtype=torch.float32, device="cuda")
    o = torch.zeros((T, H), dtype=act, device="cuda")
    moe.moe_combine(y, 1, cap, al["inv_perm"], T, K, H, moe.dtype_code(act), o, st)
    assert moe.moe_get_device_status(st) == _abi.MOE_ERR_TIMEOUT
    assert (o == 0).all()
    o.fill_(1.0)
    moe.moe_combine(y, 1, cap, al["inv_perm"], T, K, H, moe.dtype_code(act), o, st)
    torch.cuda.synchronize()
    assert (o == 1.0).all()

    # the device is fine afterwards: an ordinary forward matches the oracle
    if mx:
        w13p, s13p = moe.pack_mx(d.w13, d.w13_scale, 2)
        w2p, s2p = moe.pack_mx(d.w2, d.w2_scale, 1)
        out_f = moe.forward(d.x, d.topk_ids, d.topk_weights, w13p, w2p, w13_scale=s13p,
                            w2_scale=s2p, weight="mxfp4", intermediate=I)
        ref = oracle_forward_tokens(inp, np.arange(T), mode=moe_oracle_emulate(), quantize_x=True,
                                    h_e4m3=True)
        assert_close(out_f, ref, max_abs=6e-2, rel_l2=2e-2, what=name + " after the timeout")
    else:
        out_f = moe.forward(d.x, d.topk_ids, d.topk_weights, d.w13, d.w2)
        assert_close(out_f, oracle_forward_tokens(inp, np.arange(T)),
                     what=name + " after the timeout")


def moe_oracle_emulate():
    import oracle
    return oracle.EMULATE


def test_wait_limit_outside_its_range_is_refused():
    p = moe.make_problem(16, 128, 256, 8, 2, "bf16")
    fake = 1 << 20
    for limit in (0, 999_999, 3_000_000_000):
        with pytest.raises(moe.MoEError) as ei:
            _abi.moe_test_gemm_wait_timeout(p, 1, fake, None, fake, None, fake, fake, fake, fake,
                                            fake, 1, limit, fake)
        assert ei.value.status == _abi.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoEError):
        _abi.moe_test_gemm_wait_timeout(p, 3, fake, None, fake, None, fake, fake, fake, fake,
                                        fake, 1, WAIT_LIMIT_NS, fake)
