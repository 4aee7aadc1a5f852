"""The C-ABI library on the host: it builds for sm_103a, loads, exports every
symbol include/moe.h declares, and rejects bad arguments before launching
anything.  No GPU compute is called here."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from mixture_experts_grouped_02_gb300 import _abi, make_problem

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(_abi.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = _abi.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert _abi.moe_abi_version() == 3


def test_status_strings():
    L = _abi.lib()
    for code in range(7):
        assert L.moe_status_string(code)
    assert L.moe_status_string(99) == b"unknown status"


@pytest.mark.parametrize("T,K,E,bm", [(16, 2, 8, 16), (4096, 2, 8, 128), (8192, 8, 256, 128),
                                      (1, 8, 256, 128), (0, 2, 8, 128), (5, 3, 1, 32)])
def test_capacity_matches_oracle(T, K, E, bm):
    assert _abi.moe_align_capacity(T, K, E, bm) == oracle.align_capacity(T, K, E, bm)


def test_problem_validation():
    ok = make_problem(16, 128, 256, 8, 2, "f32")
    assert _abi.moe_resolve_block_m(ok) == 128
    assert _abi.moe_workspace_size(ok) > 0
    for bad in (make_problem(-1, 128, 256, 8, 2), make_problem(16, 0, 256, 8, 2),
                make_problem(16, 128, 256, 0, 2), make_problem(16, 128, 256, 8, 2, block_m=48),
                make_problem(16, 128, 256, 8, 2, block_m=512),
                make_problem(16, 128, 256, 2048, 2)):
        assert _abi.moe_workspace_size(bad) == 0
        assert _abi.moe_resolve_block_m(bad) == -1
    bad_pair = make_problem(16, 128, 256, 8, 2, "f32", "mxfp4")
    assert _abi.moe_workspace_size(bad_pair) == 0


def test_block_m_auto_rule():
    # 256-row blocks (CTA pairs) once experts average 256 rows, mx weights 128
    assert _abi.moe_resolve_block_m(make_problem(4096, 4096, 14336, 8, 2, "bf16")) == 256
    assert _abi.moe_resolve_block_m(make_problem(8192, 7168, 2048, 256, 8, "bf16")) == 256
    assert _abi.moe_resolve_block_m(make_problem(8191, 7168, 2048, 256, 8, "bf16")) == 128
    assert _abi.moe_resolve_block_m(make_problem(128, 4096, 14336, 8, 2, "bf16")) == 128
    assert _abi.moe_resolve_block_m(make_problem(2048, 2880, 2880, 128, 4, "bf16", "mxfp4")) == 128
    assert _abi.moe_resolve_block_m(make_problem(16, 128, 256, 8, 2, "f32", block_m=64)) == 64


def test_workspace_layout_is_disjoint_and_aligned():
    p = make_problem(4096, 4096, 14336, 8, 2, "bf16")
    off, size = _abi.moe_workspace_offsets(p)
    total = _abi.moe_workspace_size(p)
    spans = sorted((o, o + s) for o, s in zip(off, size) if s > 0)
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
    assert spans[-1][1] <= total
    assert all(o % 1024 == 0 for o in off)
    bm = _abi.moe_resolve_block_m(p)
    assert bm == 256  # many tokens per expert: CTA-pair GEMMs
    cap = _abi.moe_align_capacity(4096, 2, 8, bm)
    assert size[_abi.MOE_WS_SORTED_IDS] == 4 * cap
    assert size[_abi.MOE_WS_BLOCK_INFO] == 16 * (cap // bm)
    assert size[_abi.MOE_WS_H] == 2 * cap * 14336
    splits = _abi.moe_gemm2_default_splits(p)
    assert size[_abi.MOE_WS_Y] == 4 * splits * cap * 4096
    # a fused combine keeps the (T, H) fp32 accumulator instead of y
    pf = make_problem(4096, 4096, 14336, 8, 2, "bf16", fused_combine=True)
    assert _abi.moe_workspace_offsets(pf)[1][_abi.MOE_WS_Y] == 4 * 4096 * 4096
    assert _abi.moe_workspace_size(make_problem(16, 128, 256, 8, 2, "bf16", fused_combine=2)) == 0


def test_entry_points_reject_bad_arguments_before_launch():
    L = _abi.lib()
    vp = ctypes.c_void_p
    fake = vp(1 << 20)  # never dereferenced: every call below fails its checks first
    # block_m outside {16, 32, 64, 128, 256}
    assert L.moe_align(fake, 4, 2, 8, 48, *([fake] * 7), None, None) == _abi.MOE_ERR_INVALID_ARG
    # E above the supported maximum
    assert L.moe_align(fake, 4, 2, 4096, 128, *([fake] * 7), None, None) == \
        _abi.MOE_ERR_UNSUPPORTED
    # null outputs
    assert L.moe_align(fake, 4, 2, 8, 128, *([None] * 7), None, None) == _abi.MOE_ERR_INVALID_ARG
    # T == 0 is a no-op
    assert L.moe_align(None, 0, 2, 8, 128, *([None] * 7), None, None) == _abi.MOE_OK
    p = make_problem(16, 100, 256, 8, 2, "bf16")  # H not a multiple of 64
    assert L.moe_gemm1_silu(ctypes.byref(p), *([fake] * 8), None, None) == \
        _abi.MOE_ERR_UNSUPPORTED
    p = make_problem(16, 128, 256, 8, 2, "bf16", "mxfp4", block_m=64)
    assert L.moe_gemm1_silu(ctypes.byref(p), *([fake] * 8), None, None) == \
        _abi.MOE_ERR_UNSUPPORTED  # the block-scaled GEMMs tile 128 rows
    p = make_problem(16, 128, 256, 8, 2, "bf16")
    assert L.moe_gemm2_weighted(ctypes.byref(p), *([fake] * 7), fake, 0, None, None) == \
        _abi.MOE_ERR_INVALID_ARG  # k_splits = 0
    assert L.moe_gemm2_weighted(ctypes.byref(p), *([fake] * 7), fake, 5, None, None) == \
        _abi.MOE_ERR_INVALID_ARG  # more splits than 64-wide k-tiles
    assert L.moe_combine(fake, 1, 64, fake, 4, 2, 126, _abi.MOE_BF16, fake, None, None) == \
        _abi.MOE_ERR_UNSUPPORTED
    assert L.moe_combine(fake, 1, 64, fake, 4, 2, 128, _abi.MOE_E4M3, fake, None, None) == \
        _abi.MOE_ERR_INVALID_ARG
    assert L.moe_combine_finish(fake, 4, 126, _abi.MOE_BF16, fake, None, None) == \
        _abi.MOE_ERR_UNSUPPORTED
    assert L.moe_combine_finish(fake, 4, 128, _abi.MOE_E4M3, fake, None, None) == \
        _abi.MOE_ERR_INVALID_ARG
    assert L.moe_combine_finish(vp((1 << 20) + 4), 4, 128, _abi.MOE_BF16, fake, None, None) == \
        _abi.MOE_ERR_INVALID_ARG  # the accumulator is read as 16-byte vectors
    assert L.moe_gather_rows(fake, _abi.MOE_BF16, 4, 128, 2, fake, fake, vp((1 << 20) + 4), None,
                             None) == _abi.MOE_ERR_INVALID_ARG
    # workspace too small / misaligned
    ws_ok = _abi.moe_workspace_size(p)
    assert L.moe_forward(ctypes.byref(p), *([fake] * 8), fake, ws_ok - 1, None) == \
        _abi.MOE_ERR_WORKSPACE
    assert L.moe_forward(ctypes.byref(p), *([fake] * 8), vp((1 << 20) + 16), ws_ok, None) == \
        _abi.MOE_ERR_WORKSPACE
    assert L.moe_quantize_x_fp8(fake, _abi.MOE_BF16, 4, 7, fake, fake, None) == \
        _abi.MOE_ERR_INVALID_ARG
    assert L.moe_get_device_status(None, None) == _abi.MOE_ERR_INVALID_ARG
    # routing: K within [1, min(E, 32)], logits fp32 or bf16
    args9 = [fake] * 9
    assert L.moe_route_align(fake, _abi.MOE_F32, 4, 8, 9, 0, 8, 128, *args9, None, None) == \
        _abi.MOE_ERR_INVALID_ARG
    assert L.moe_route_align(fake, _abi.MOE_F32, 4, 64, 33, 0, 64, 128, *args9, None, None) == \
        _abi.MOE_ERR_UNSUPPORTED
    assert L.moe_route_align(fake, _abi.MOE_E4M3, 4, 8, 2, 0, 8, 128, *args9, None, None) == \
        _abi.MOE_ERR_INVALID_ARG
    assert L.moe_route_align(None, _abi.MOE_F32, 0, 8, 2, 0, 8, 128, *([None] * 9), None,
                             None) == _abi.MOE_OK
    # expert shards: the range must lie inside [0, E)
    for base, local in ((-1, 2), (7, 2), (0, 0), (0, 9)):
        assert L.moe_align_local(fake, 4, 2, 8, base, local, 128, *([fake] * 7), None, 0, None,
                                 None) == _abi.MOE_ERR_INVALID_ARG
    # the many-CTA align: scratch only from 16384 assignments on, one int per
    # (warp of 256 ids, local expert) and per (CTA of 8 warps, local expert);
    # too small a scratch is refused
    assert L.moe_align_scratch_bytes(2048, 4, 64) == 0
    assert L.moe_align_scratch_bytes(4096, 4, 64) == 4 * (64 + 8) * 64
    assert L.moe_align_scratch_bytes(16384, 8, 256) == 4 * (512 + 64) * 256
    assert L.moe_align_scratch_bytes(20001, 6, 64) == 4 * (59 * 8 + 59) * 64  # 469 warps
    # at most 4864 warps: larger chunks for the largest batches
    big = L.moe_align_scratch_bytes(1 << 20, 32, 1024)
    assert big == 4 * (607 * 8 + 607) * 1024  # chunks of 6912 ids: 4855 warps
    assert L.moe_align_local(fake, 4096, 4, 64, 0, 64, 128, *([fake] * 7), fake, 64, None,
                             None) == _abi.MOE_ERR_WORKSPACE
    for base, local in ((1, 0), (-1, 3), (6, 3)):
        bad = make_problem(16, 128, 256, 8, 2, "bf16", expert_base=base, local_experts=local)
        assert _abi.moe_workspace_size(bad) == 0
    # the forward without a workspace returns moe_forward's codes for the
    # same arguments, and refuses problems beyond its static array
    for p, code in ((make_problem(16, 100, 256, 8, 2, "bf16"), _abi.MOE_ERR_UNSUPPORTED),
                    (make_problem(16, 128, 256, 2048, 2, "bf16"), _abi.MOE_ERR_UNSUPPORTED),
                    (make_problem(16, 128, 256, 8, 2, "bf16", block_m=48),
                     _abi.MOE_ERR_INVALID_ARG),
                    (make_problem(4096, 4096, 14336, 8, 2, "bf16"), _abi.MOE_ERR_WORKSPACE)):
        assert L.moe_forward_noalloc(ctypes.byref(p), *([fake] * 9)) == code
        if code != _abi.MOE_ERR_WORKSPACE:
            assert L.moe_forward(ctypes.byref(p), *([fake] * 9), 1 << 40, None) == code
    assert L.moe_forward_noalloc(None, *([fake] * 9)) == _abi.MOE_ERR_INVALID_ARG


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                       "mixture_experts_grouped_02_gb300")
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "moe_oracle" not in text, f
