"""GPU parity: every stage of the CUDA path, called through the C ABI, against
the fp64 CPU oracle on the same seeded inputs.

Integer outputs (align) must match bit for bit; floating-point outputs must be
within max-abs 2e-2 and relative L2 1e-2 of the oracle (bf16 and tf32)."""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins as pins
from gpu_util import (assert_close, block_tokens, errors, generate, np_store,
                      oracle_forward_tokens, oracle_problem, problem_kw, sample_tokens)
import mixture_experts_grouped_02_gb300 as moe
from mixture_experts_grouped_02_gb300 import _abi
from mixture_experts_grouped_02_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _abi.lib()
    yield
    torch.cuda.synchronize()


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ------------------------------------------------------------------ align

EXTRA_ALIGN = [(1, 8, 256, 128, "normal"), (3, 2, 1000, 16, "normal"),
               (2000, 4, 1024, 64, "normal"), (4096, 2, 8, 128, "normal"),
               (4096, 2, 8, 256, "normal"), (700, 3, 5, 256, "skewed")]


@pytest.mark.parametrize("case", pins.ALIGN_CASES + EXTRA_ALIGN,
                         ids=lambda c: "T%d_K%d_E%d_bm%d_%s" % c)
def test_align_bit_exact(case):
    T, K, E, bm, kind = case
    ids = pins.align_ids(T, K, E, kind)
    ref = oracle.align(ids, E, bm)
    st = _status()
    got = moe.align(torch.from_numpy(ids).cuda(), E, bm, dev_status=st)
    assert moe.moe_get_device_status(st) == 0
    for k in ("counts", "offsets", "padded_offsets", "sorted_ids", "inv_perm"):
        assert np.array_equal(got[k].cpu().numpy(), ref[k]), k
    assert np.array_equal(got["block_info"].cpu().numpy(), ref["block_info"])
    assert int(got["num_blocks"].item()) == ref["num_blocks"]


def test_align_skewed_dsv3_routing():
    cfg = gen.config("dsv3_prefill")
    ids, _ = gen.route(gen.router_logits(cfg, 0), cfg.K)
    ref = oracle.align(ids.numpy(), cfg.E, 128)
    got = moe.align(ids.cuda(), cfg.E, 128)
    assert (ref["counts"] == 0).sum() >= 0
    for k in ("counts", "offsets", "padded_offsets", "sorted_ids", "inv_perm", "block_info"):
        assert np.array_equal(got[k].cpu().numpy(), ref[k]), k


def test_align_bad_id_sets_status():
    # 6 assignments: the one-warp path of small batches
    ids = torch.tensor([[0, 1], [2, 9], [3, 4]], dtype=torch.int32, device="cuda")
    st = _status()
    got = moe.align(ids, 8, 16, dev_status=st)
    assert moe.moe_get_device_status(st) == _abi.MOE_ERR_DEVICE_BAD_ID
    assert int(got["num_blocks"].item()) == 0


def test_align_bad_id_sets_status_large_batch():
    # 3000 assignments: the per-warp histograms of the single-CTA path
    ids = torch.from_numpy(pins.align_ids(1500, 2, 8, "normal")).cuda()
    ids[777, 1] = -2
    st = _status()
    got = moe.align(ids, 8, 16, dev_status=st)
    assert moe.moe_get_device_status(st) == _abi.MOE_ERR_DEVICE_BAD_ID
    assert int(got["num_blocks"].item()) == 0


@pytest.mark.parametrize("case,shard", [((300, 4, 16, 64, "skewed"), (0, 5)),
                                        ((37, 3, 8, 32, "normal"), (3, 4)),
                                        ((2000, 8, 256, 128, "normal"), (224, 32)),
                                        ((64, 2, 8, 256, "normal"), (7, 1)),
                                        ((12, 2, 16, 32, "normal"), (4, 6))])
def test_align_local_bit_exact(case, shard):
    T, K, E, bm, kind = case
    base, L = shard
    ids = pins.align_ids(T, K, E, kind)
    ref = oracle.align(ids, E, bm, expert_base=base, local_experts=L)
    st = _status()
    got = moe.align(torch.from_numpy(ids).cuda(), E, bm, dev_status=st, expert_base=base,
                    local_experts=L)
    assert moe.moe_get_device_status(st) == 0
    for k in ("counts", "offsets", "padded_offsets", "sorted_ids", "inv_perm", "block_info"):
        assert np.array_equal(got[k].cpu().numpy(), ref[k]), k
    assert int(got["num_blocks"].item()) == ref["num_blocks"]


ALIGN_MANY_CTA_CASES = [
    # T, K, E, block_m, routing, (expert_base, local_experts); T*K >= 16384
    # assignments go to the many-CTA align (chunks of 1024 ids per warp)
    (4096, 4, 64, 128, "skewed", (0, 64)),
    (16384, 8, 256, 256, "normal", (0, 256)),
    (20001, 6, 160, 16, "skewed", (32, 64)),   # ragged last chunk, a shard
    (3000, 8, 1024, 64, "normal", (0, 1024)),  # the most experts
    (8192, 2, 8, 256, "skewed", (7, 1)),       # one local expert
]


@pytest.mark.parametrize("case,shard", [(c[:5], c[5]) for c in ALIGN_MANY_CTA_CASES],
                         ids=lambda c: "_".join(map(str, c)))
def test_align_many_cta_bit_exact(case, shard):
    T, K, E, bm, kind = case
    base, L = shard
    assert moe.moe_align_scratch_bytes(T, K, L) > 0
    ids = pins.align_ids(T, K, E, kind)
    ref = oracle.align(ids, E, bm, expert_base=base, local_experts=L)
    d_ids = torch.from_numpy(ids).cuda()
    st = _status()
    got = moe.align(d_ids, E, bm, dev_status=st, expert_base=base, local_experts=L)
    one = moe.align(d_ids, E, bm, dev_status=st, expert_base=base, local_experts=L,
                    many_cta=False)
    assert moe.moe_get_device_status(st) == 0
    for k in ("counts", "offsets", "padded_offsets", "sorted_ids", "inv_perm", "block_info"):
        assert np.array_equal(got[k].cpu().numpy(), ref[k]), k
        assert torch.equal(got[k], one[k]), k
    assert int(got["num_blocks"].item()) == ref["num_blocks"]


def test_align_many_cta_bad_id_sets_status():
    ids = pins.align_ids(4096, 4, 64, "normal")
    ids[4000, 3] = 64  # outside [0, E), in the last chunk
    st = _status()
    got = moe.align(torch.from_numpy(ids).cuda(), 64, 128, dev_status=st)
    assert moe.moe_get_device_status(st) == _abi.MOE_ERR_DEVICE_BAD_ID
    assert int(got["num_blocks"].item()) == 0


ROUTE_CASES = [
    # T, E, K, logit dtype, kind; up to 1024 tokens the align kernel routes
    (37, 8, 2, torch.float32, "normal"),
    (1000, 256, 8, torch.float32, "zipf"),
    (5000, 256, 8, torch.float32, "zipf"),     # separate routing kernel
    (2048, 128, 4, torch.bfloat16, "normal"),
    (300, 64, 6, torch.float32, "ties"),       # small integers: many equal logits
    (1, 1024, 32, torch.float32, "normal"),
]


@pytest.mark.parametrize("case", ROUTE_CASES, ids=lambda c: "T%d_E%d_K%d_%s_%s" % (
    c[0], c[1], c[2], str(c[3]).split(".")[-1], c[4]))
def test_route_align_vs_oracle(case):
    T, E, K, dt, kind = case
    g = torch.Generator().manual_seed(T + E)
    if kind == "ties":
        logits = torch.randint(-3, 4, (T, E), generator=g).to(torch.float32)
    else:
        logits = torch.randn((T, E), generator=g)
        if kind == "zipf":
            logits = logits + gen.zipf_bias(E, 1)
    logits = logits.to(dt)
    ids_ref, w_ref = oracle.route(np_store(logits), K)
    bm = 128
    st = _status()
    got = moe.route_align(logits.cuda(), K, bm, dev_status=st)
    assert moe.moe_get_device_status(st) == 0
    assert np.array_equal(got["topk_ids"].cpu().numpy(), ids_ref)
    w = got["topk_weights"].cpu().numpy().astype(np.float64)
    assert np.allclose(w, w_ref, rtol=2e-6, atol=1e-7)
    al = oracle.align(ids_ref, E, bm)
    for k in ("counts", "offsets", "padded_offsets", "sorted_ids", "inv_perm", "block_info"):
        assert np.array_equal(got[k].cpu().numpy(), al[k]), k
    assert int(got["num_blocks"].item()) == al["num_blocks"]


def test_route_align_shard():
    T, E, K = 700, 64, 4
    logits = torch.randn((T, E), generator=torch.Generator().manual_seed(3))
    ids_ref, _ = oracle.route(np_store(logits), K)
    got = moe.route_align(logits.cuda(), K, 64, expert_base=16, local_experts=16)
    al = oracle.align(ids_ref, E, 64, expert_base=16, local_experts=16)
    assert np.array_equal(got["topk_ids"].cpu().numpy(), ids_ref)
    for k in ("counts", "padded_offsets", "sorted_ids", "inv_perm", "block_info"):
        assert np.array_equal(got[k].cpu().numpy(), al[k]), k


# ------------------------------------------------------------------ stages

STAGE_CASES = [
    # T, H, I, E, K, dtype
    (300, 256, 320, 3, 2, "bf16"),   # 2 blocks per expert, ragged I tile
    (77, 192, 256, 5, 2, "bf16"),
    (40, 128, 256, 8, 2, "f32"),     # tf32 path
    # T <= 32: the decode-like launch, two K steps per stage; 5 K steps of
    # the down projection leave a last stage with one
    (8, 256, 320, 8, 2, "bf16"),
    (12, 128, 256, 4, 3, "f32"),
]


def _valid_rows(al, na):
    s = al["sorted_ids"]
    rows = np.nonzero(s < na)[0].astype(np.int32)
    return rows


def _expert_of_rows(al, rows, ids_flat):
    return ids_flat[al["sorted_ids"][rows]].astype(np.int32)


@pytest.mark.parametrize("bm", [32, 128, 256])
@pytest.mark.parametrize("case", STAGE_CASES, ids=lambda c: "T%d_H%d_I%d_E%d_K%d_%s" % c)
def test_gemm1_silu_stage(case, bm):
    T, H, I, E, K, dt = case
    cfg = gen.MoEConfig("stage", T, H, I, E, K, dt, "normal")
    inp = gen.generate(cfg, seed=21)
    d = inp.to("cuda")
    al_ref = oracle.align(inp.topk_ids.numpy(), E, bm)
    al = moe.align(d.topk_ids, E, bm)
    p = moe.make_problem(T, H, I, E, K, dt, block_m=bm)
    cap = moe.moe_align_capacity(T, K, E, bm)
    h = torch.full((cap, I), float("nan"), dtype=d.x.dtype, device="cuda")
    st = _status()
    # the GEMM reads the token rows at their sorted slots (moe_gather_rows)
    xs = np.zeros((cap, H), np.float32)
    valid = al_ref["sorted_ids"] < T * K
    xs[valid] = inp.x.float().numpy()[al_ref["sorted_ids"][valid] // K]
    x_in = torch.from_numpy(xs).to(d.x.dtype).cuda()
    moe.moe_gemm1_silu(p, x_in, None, d.w13, None, al["sorted_ids"], al["block_info"],
                       al["num_blocks"], h, st)
    assert moe.moe_get_device_status(st) == 0
    rows = _valid_rows(al_ref, T * K)
    eor = _expert_of_rows(al_ref, rows, inp.topk_ids.numpy().ravel())
    ref = oracle.gemm1_silu_rows(oracle_problem(inp), np_store(inp.x), np_store(inp.w13),
                                 al_ref["sorted_ids"], eor, rows)
    got = h[torch.from_numpy(rows).long().cuda()]
    # h is stored in bf16 (tf32 operands in the f32 case): besides the bounds on
    # the layer output, each element may carry one rounding of relative size
    # 2^-8, which exceeds 2e-2 for |h| > 5.
    g = got.double().cpu().numpy()
    assert np.all(np.abs(g - ref) <= 2e-2 + 2.0 ** -8 * np.abs(ref)), np.abs(g - ref).max()
    assert_close(got, ref, max_abs=np.inf, what="h")
    # padding rows are never written
    pad = np.nonzero(al_ref["sorted_ids"] >= T * K)[0]
    if len(pad):
        assert torch.isnan(h[torch.from_numpy(pad).long().cuda()].float()).all()


GATHER_CASES = STAGE_CASES + [
    (600, 256, 320, 3, 2, "bf16"),   # 400 rows per expert: full 256-token tiles, 128 rows per CTA
    (64, 256, 320, 8, 2, "bf16"),    # 16 rows per expert on average: decode-like, mixed tiles
]


def _raw(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("bm", [32, 128, 256])
@pytest.mark.parametrize("case", GATHER_CASES, ids=lambda c: "T%d_H%d_I%d_E%d_K%d_%s" % c)
def test_gemm1_silu_gather_matches_gather_pass(case, bm, interleaved):
    """The gate/up GEMM that gathers its token rows by index in the producer
    (tile::gather4 from x) writes h bit for bit as the GEMM over the rows
    moe_gather_rows put at their sorted slots, padding rows left unwritten,
    for tiles of 16 to 256 tokens, bf16 and fp32, w13 in halves or with the
    gate and up rows interleaved."""
    T, H, I, E, K, dt = case
    cfg = gen.MoEConfig("stage", T, H, I, E, K, dt, "normal")
    d = gen.generate(cfg, seed=24).to("cuda")
    al = moe.align(d.topk_ids, E, bm)
    p = moe.make_problem(T, H, I, E, K, dt, block_m=bm, gate_up_interleaved=interleaved)
    cap = moe.moe_align_capacity(T, K, E, bm)
    st = _status()
    xs = torch.zeros((cap, H), dtype=d.x.dtype, device="cuda")
    moe.moe_gather_rows(d.x, p.act, T, H, K, al["inv_perm"], xs, st)
    h_ref = torch.full((cap, I), float("nan"), dtype=d.x.dtype, device="cuda")
    moe.moe_gemm1_silu(p, xs, None, d.w13, None, al["sorted_ids"], al["block_info"],
                       al["num_blocks"], h_ref, st)
    h = torch.full((cap, I), float("nan"), dtype=d.x.dtype, device="cuda")
    moe.moe_gemm1_silu_gather(p, d.x, d.w13, al["sorted_ids"], al["block_info"],
                              al["num_blocks"], h, st)
    assert moe.moe_get_device_status(st) == 0
    assert torch.equal(_raw(h), _raw(h_ref))


@pytest.mark.parametrize("bm", [32, 128, 256])
@pytest.mark.parametrize("splits", [1, 2, 3])
@pytest.mark.parametrize("case", STAGE_CASES, ids=lambda c: "T%d_H%d_I%d_E%d_K%d_%s" % c)
def test_gemm2_weighted_stage(case, splits, bm):
    T, H, I, E, K, dt = case
    cfg = gen.MoEConfig("stage", T, H, I, E, K, dt, "normal")
    inp = gen.generate(cfg, seed=22)
    d = inp.to("cuda")
    cap = moe.moe_align_capacity(T, K, E, bm)
    g = torch.Generator().manual_seed(5)
    hin = torch.randn((cap, I), generator=g).to(inp.x.dtype)  # synthetic hidden rows
    al_ref = oracle.align(inp.topk_ids.numpy(), E, bm)
    al = moe.align(d.topk_ids, E, bm)
    p = moe.make_problem(T, H, I, E, K, dt, block_m=bm)
    y = torch.full((splits, cap, H), float("nan"), dtype=torch.float32, device="cuda")
    st = _status()
    moe.moe_gemm2_weighted(p, hin.cuda(), d.w2, None, d.topk_weights, al["sorted_ids"],
                           al["block_info"], al["num_blocks"], y, splits, st)
    assert moe.moe_get_device_status(st) == 0
    rows = _valid_rows(al_ref, T * K)
    eor = _expert_of_rows(al_ref, rows, inp.topk_ids.numpy().ravel())
    ref = oracle.gemm2_weighted_rows(oracle_problem(inp), np_store(hin), np_store(inp.w2),
                                     inp.topk_weights.numpy(), al_ref["sorted_ids"], eor, rows)
    got = y[:, torch.from_numpy(rows).long().cuda()].sum(0)
    tol = 1e-4 if dt == "bf16" else 5e-3  # bf16 products are exact; tf32 rounds operands
    assert_close(got, ref, max_abs=2e-2, rel_l2=tol, what="y")
    # padding rows are never written
    pad = np.nonzero(al_ref["sorted_ids"] >= T * K)[0]
    if len(pad):
        assert torch.isnan(y[:, torch.from_numpy(pad).long().cuda()]).all()


@pytest.mark.parametrize("splits", [1, 2])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_combine_stage(splits, out_dtype):
    T, K, E, H = 50, 3, 7, 96
    ids = pins.align_ids(T, K, E, "normal", seed=3)
    al_ref = oracle.align(ids, E, 16)
    cap = moe.moe_align_capacity(T, K, E, 16)
    g = torch.Generator().manual_seed(6)
    y = torch.randn((cap, H), generator=g)
    ref = oracle.combine(y.numpy(), al_ref["inv_perm"], T, K, H)
    # two splits holding y/2 each sum to y exactly
    ys = (y / splits).unsqueeze(0).repeat(splits, 1, 1).contiguous().cuda()
    inv = torch.from_numpy(al_ref["inv_perm"]).cuda()
    out = torch.empty((T, H), dtype=out_dtype, device="cuda")
    moe.moe_combine(ys, splits, cap, inv, T, K, H, moe.dtype_code(out_dtype), out)
    torch.cuda.synchronize()
    tol = 1e-6 if out_dtype == torch.float32 else 8e-3
    assert_close(out, ref, max_abs=2e-2, rel_l2=tol, what="out")


@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("case", STAGE_CASES, ids=lambda c: "T%d_H%d_I%d_E%d_K%d_%s" % c)
def test_gemm2_fused_combine_stage(case, splits):
    """GEMM2 adding its weighted rows into the (T, H) accumulator the gather
    step zeroed: every token row equals the sum of its K weighted expert rows
    (the oracle's rows, summed per token in fp64)."""
    T, H, I, E, K, dt = case
    bm = 128
    cfg = gen.MoEConfig("stage", T, H, I, E, K, dt, "normal")
    inp = gen.generate(cfg, seed=23)
    d = inp.to("cuda")
    cap = moe.moe_align_capacity(T, K, E, bm)
    hin = torch.randn((cap, I), generator=torch.Generator().manual_seed(7)).to(inp.x.dtype)
    al_ref = oracle.align(inp.topk_ids.numpy(), E, bm)
    al = moe.align(d.topk_ids, E, bm)
    p = moe.make_problem(T, H, I, E, K, dt, block_m=bm, fused_combine=True)
    acc = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    xs = torch.empty((cap, H), dtype=d.x.dtype, device="cuda")
    st = _status()
    moe.moe_gather_rows(d.x, p.act, T, H, K, al["inv_perm"], xs, st, acc_zero=acc)
    moe.moe_gemm2_weighted(p, hin.cuda(), d.w2, None, d.topk_weights, al["sorted_ids"],
                           al["block_info"], al["num_blocks"], acc, splits, st)
    assert moe.moe_get_device_status(st) == 0
    rows = _valid_rows(al_ref, T * K)
    eor = _expert_of_rows(al_ref, rows, inp.topk_ids.numpy().ravel())
    per_row = oracle.gemm2_weighted_rows(oracle_problem(inp), np_store(hin), np_store(inp.w2),
                                         inp.topk_weights.numpy(), al_ref["sorted_ids"], eor, rows)
    ref = np.zeros((T, H))
    np.add.at(ref, al_ref["sorted_ids"][rows] // K, per_row)
    tol = 1e-4 if dt == "bf16" else 5e-3
    assert_close(acc, ref, max_abs=2e-2, rel_l2=tol, what="accumulator")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_combine_finish_rounds_once(out_dtype):
    T, H = 37, 96
    acc = (torch.randn((T, H), generator=torch.Generator().manual_seed(8)) * 3).cuda()
    out = torch.empty((T, H), dtype=out_dtype, device="cuda")
    moe.moe_combine_finish(acc, T, H, moe.dtype_code(out_dtype), out)
    assert torch.equal(out, acc.to(out_dtype))  # round to nearest even, bit for bit


# ------------------------------------------------------------------ forward

FORWARD_CASES = [
    # T, H, I, E, K, dtype, routing
    (300, 256, 320, 3, 2, "bf16", "normal"),
    (64, 320, 256, 16, 4, "bf16", "zipf"),     # ragged H tile, empty experts
    (1, 256, 256, 8, 2, "bf16", "normal"),
    (513, 128, 128, 2, 1, "bf16", "normal"),   # top-1
    (33, 128, 256, 8, 2, "f32", "normal"),
]


def _run_forward(d, cfg, poison=True, block_m=0):
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.dtype, block_m=block_m)
    ws = moe.Workspace(p)
    if poison:
        ws.buffer.fill_(0xFF)  # NaN patterns everywhere the path does not write
    out = torch.full((cfg.T, cfg.H), float("nan"), dtype=d.x.dtype, device="cuda")
    moe.moe_forward(p, d.x, d.topk_ids, d.topk_weights, d.w13, None, d.w2, None, out, ws.buffer,
                    ws.nbytes)
    assert moe.moe_get_device_status(ws.status) == 0
    return out, ws


@pytest.mark.parametrize("bm", [0, 16, 256])
@pytest.mark.parametrize("case", FORWARD_CASES, ids=lambda c: "T%d_H%d_I%d_E%d_K%d_%s_%s" % c)
def test_forward_small(case, bm):
    cfg = gen.MoEConfig("fwd", *case)
    inp = gen.generate(cfg, seed=31)
    out, ws = _run_forward(inp.to("cuda"), cfg, block_m=bm)
    ref = oracle_forward_tokens(inp, np.arange(cfg.T))
    assert_close(out, ref, what=cfg.name)


def test_block_m_auto_picks_pairs_for_many_tokens_per_expert():
    assert moe.moe_resolve_block_m(moe.make_problem(4096, 4096, 14336, 8, 2, "bf16")) == 256
    assert moe.moe_resolve_block_m(moe.make_problem(8192, 7168, 2048, 256, 8, "bf16")) == 256
    assert moe.moe_resolve_block_m(moe.make_problem(8191, 7168, 2048, 256, 8, "bf16")) == 128
    assert moe.moe_resolve_block_m(moe.make_problem(128, 4096, 14336, 8, 2, "bf16")) == 128
    assert moe.moe_resolve_block_m(moe.make_problem(2048, 2880, 2880, 128, 4, "bf16",
                                                    "mxfp4")) == 128


def test_forward_tiny_config():
    cfg = gen.config("tiny")
    inp = gen.generate(cfg, seed=0)
    out, _ = _run_forward(inp.to("cuda"), cfg)
    ref = oracle_forward_tokens(inp, np.arange(cfg.T))
    assert_close(out, ref, what="tiny")


@pytest.mark.parametrize("bm", [128, 256])
def test_forward_deterministic_and_padding_untouched(bm):
    cfg = gen.MoEConfig("fwd", 300, 256, 320, 3, 2, "bf16", "normal")
    d = gen.generate(cfg, seed=32).to("cuda")
    out1, ws = _run_forward(d, cfg, block_m=bm)
    out2, _ = _run_forward(d, cfg, block_m=bm)
    assert torch.equal(out1, out2)
    h = ws.part(_abi.MOE_WS_H, torch.uint8)
    cap = moe.moe_align_capacity(cfg.T, cfg.K, cfg.E, bm)
    h = h[:cap * cfg.I * 2].view(cap, cfg.I * 2)
    s = ws.part(_abi.MOE_WS_SORTED_IDS, torch.int32)[:cap].cpu().numpy()
    pad = np.nonzero(s >= cfg.T * cfg.K)[0]
    assert len(pad) > 0
    assert (h[torch.from_numpy(pad).long().cuda()] == 0xFF).all()


def test_forward_status_blocks_later_stages():
    cfg = gen.MoEConfig("fwd", 64, 128, 128, 4, 2, "bf16", "normal")
    d = gen.generate(cfg, seed=33).to("cuda")
    d.topk_ids[5, 1] = 4  # outside [0, E)
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.dtype)
    ws = moe.Workspace(p)
    out = torch.zeros((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(p, d.x, d.topk_ids, d.topk_weights, d.w13, None, d.w2, None, out, ws.buffer,
                    ws.nbytes)
    assert moe.moe_get_device_status(ws.status) == _abi.MOE_ERR_DEVICE_BAD_ID
    assert (out == 0).all()  # combine did not run


def test_forward_zero_tokens():
    p = moe.make_problem(0, 128, 128, 4, 2, "bf16")
    moe.moe_forward(p, 0, 0, 0, 0, None, 0, None, 0, 0, 0)


# ------------------------------------------------------------- full sizes

@pytest.mark.parametrize("name", [f"mixtral_decode_T{t}" for t in gen.DECODE_T] +
                         [f"dsv3_decode_T{t}" for t in gen.DECODE_T])
def test_forward_decode_full_size(name):
    cfg = gen.config(name)
    inp = generate(cfg, seed=0, device="cuda")
    out, _ = _run_forward(inp, cfg, poison=False)
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.dtype)
    toks, _ = block_tokens(inp, moe.moe_resolve_block_m(p))
    ref = oracle_forward_tokens(inp, toks)
    assert_close(out[torch.from_numpy(toks).long().cuda()], ref, what=name)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("name", ["mixtral_prefill", "dsv3_prefill"])
def test_forward_prefill_full_size_sampled(name):
    cfg = gen.config(name)
    inp = generate(cfg, seed=0, device="cuda")
    out, ws = _run_forward(inp, cfg, poison=False)
    # a checked token in every align block: the first and last valid slot
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.dtype)
    toks, nb = block_tokens(inp, moe.moe_resolve_block_m(p), seed=1)
    assert nb > 0 and len(toks) >= nb // cfg.K
    ref = oracle_forward_tokens(inp, toks)
    assert_close(out[torch.from_numpy(toks).long().cuda()], ref, what=name)
    assert torch.isfinite(out.float()).all()
    # the align's outputs in the workspace (over many CTAs from T*K = 16384
    # on, the DeepSeek-V3 shape), bit for bit against the oracle's
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.dtype)
    al = oracle.align(inp.topk_ids.cpu().numpy(), cfg.E, moe.moe_resolve_block_m(p))
    cap = len(al["sorted_ids"])
    for k, part, n in (("counts", _abi.MOE_WS_COUNTS, cfg.E),
                       ("padded_offsets", _abi.MOE_WS_PADDED_OFFSETS, cfg.E + 1),
                       ("sorted_ids", _abi.MOE_WS_SORTED_IDS, cap),
                       ("inv_perm", _abi.MOE_WS_INV_PERM, cfg.T * cfg.K)):
        assert np.array_equal(ws.part(part, torch.int32)[:n].cpu().numpy(), al[k]), k
    assert int(ws.part(_abi.MOE_WS_NUM_BLOCKS, torch.int32)[0]) == al["num_blocks"]
    del inp, out
    torch.cuda.empty_cache()


# ------------------------------------------------------------- fp8 step

@pytest.mark.parametrize("shape", [(2048, 2880), (1, 64), (37, 4096)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_x_fp8_bit_exact(shape, dtype):
    """e4m3 codes and fp32 row scales match the oracle bit for bit: both sides
    form amax/448 and x/s in fp32 and round to nearest-even, saturating."""
    T, H = shape
    g = torch.Generator().manual_seed(T + H)
    x = torch.randn((T, H), generator=g) * torch.logspace(-3, 3, T).unsqueeze(1)
    if T > 2:
        x[1] = 0.0  # all-zero row: scale 1
        x[2, :5] = torch.tensor([1e30, -1e30, 0.5, -0.0, 3.0])  # extreme row
    x = x.to(dtype)
    xq_ref, s_ref = oracle.quantize_x_fp8(np_store(x))
    xq = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    s = torch.empty(T, dtype=torch.float32, device="cuda")
    moe.moe_quantize_x_fp8(x.cuda(), moe.dtype_code(dtype), T, H, xq, s)
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), xq_ref)


# ------------------------------------------------------------- mxfp4 path
# Bounds for the fp8 x mxfp4 path: against the oracle that rounds h to e4m3
# the way the GPU stores it (EMULATE), max-abs 6e-2 and rel-L2 2e-2; against
# the unrounded oracle (EXACT), rel-L2 6e-2 (one e4m3 rounding of h carries
# up to 2^-4 relative error per element).
MX_MAX_ABS, MX_REL_EMU, MX_REL_EXACT = 6e-2, 2e-2, 6e-2

MX_CASES = [
    # T, H, I, E, K
    (40, 256, 192, 4, 2),     # whole k-tiles, two N tiles of 96
    (150, 320, 288, 3, 2),    # K ending half-way through a 128-element tile, 2 M blocks
    (7, 2880, 192, 8, 4),     # the low-precision hidden size
]


def _mx_problem(case, seed):
    T, H, I, E, K = case
    cfg = gen.MoEConfig("mx", T, H, I, E, K, "mxfp4", "uniform")
    return cfg, gen.generate(cfg, seed=seed)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_gather_rows_bit_exact(dtype):
    """Every sorted slot of a token holds that token's row, bit for bit;
    padding slots are left alone."""
    T, H, K, E = 300, 264, 2, 3
    g = torch.Generator().manual_seed(9)
    x = torch.randn((T, H), generator=g).to(dtype)
    ids = pins.align_ids(T, K, E, "normal", seed=5)
    al = oracle.align(ids, E, 256)
    cap = len(al["sorted_ids"])
    xs = torch.zeros((cap, H), dtype=dtype, device="cuda")
    moe.moe_gather_rows(x.cuda(), moe.dtype_code(dtype), T, H, K,
                        torch.from_numpy(al["inv_perm"]).cuda(), xs)
    torch.cuda.synchronize()
    valid = al["sorted_ids"] < T * K
    got = xs.cpu()
    assert torch.equal(got[torch.from_numpy(valid)], x[al["sorted_ids"][valid] // K])
    assert (got[torch.from_numpy(~valid)] == 0).all()


@pytest.mark.parametrize("xdt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,H,K,E", [(2048, 2880, 4, 128), (37, 64, 2, 5), (19, 72, 3, 4)])
def test_quantize_gather_x_fp8_bit_exact(T, H, K, E, xdt):
    """Codes at every sorted slot of a token equal the oracle's codes of that
    token, bit for bit; the row scales too.  Rows of a multiple of 16
    elements take the 16-element-run kernel, H = 72 the general one."""
    g = torch.Generator().manual_seed(T)
    x = (torch.randn((T, H), generator=g) * 3).to(xdt)
    ids = pins.align_ids(T, K, E, "normal", seed=4)
    al = oracle.align(ids, E, 128)
    cap = len(al["sorted_ids"])
    xq_ref, s_ref = oracle.quantize_x_fp8(np_store(x))
    xs = torch.zeros((cap, H), dtype=torch.uint8, device="cuda")
    s = torch.empty(T, dtype=torch.float32, device="cuda")
    moe.moe_quantize_gather_x_fp8(x.cuda(), moe.dtype_code(xdt), T, H, K,
                                  torch.from_numpy(al["inv_perm"]).cuda(), xs, s)
    torch.cuda.synchronize()
    valid = al["sorted_ids"] < T * K
    got = xs.cpu().numpy()
    assert np.array_equal(got[valid], xq_ref[al["sorted_ids"][valid] // K])
    assert np.all(got[~valid] == 0)  # padding slots untouched
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("E,R,K,sections", [(2, 200, 320, 2), (3, 300, 128, 1), (1, 96, 2880, 1)])
def test_pack_mx_layout(E, R, K, sections):
    """The packed values and scale images hold exactly the bytes the layout in
    include/moe.h puts where (built here with numpy index arithmetic)."""
    rng = np.random.default_rng(E * R + K)
    w = rng.integers(0, 256, (E, R, K // 2)).astype(np.uint8)
    sc = rng.integers(0, 256, (E, R, K // 32)).astype(np.uint8)
    vals, imgs = moe.pack_mx(torch.from_numpy(w).cuda(), torch.from_numpy(sc).cuda(), sections)
    torch.cuda.synchronize()
    Kp = (K + 127) // 128 * 128
    rs = R // sections
    KT = Kp // 128
    span = 192 // sections
    NT = -(-rs // span)
    # values, tile-major: (expert, weight tile, K tile) tiles of 192 rows x 64
    # bytes; tile row r is section r // span, row span * n + r % span
    nat = np.zeros((E, sections, NT * span, Kp // 2), np.uint8)
    nat[:, :, :rs, :K // 2] = w.reshape(E, sections, rs, K // 2)
    tiles = nat.reshape(E, sections, NT, span, KT, 64).transpose(0, 2, 4, 1, 3, 5)
    exp_vals = tiles.reshape(E, NT, KT, 192, 64)
    assert np.array_equal(vals.cpu().numpy(), exp_vals)
    # scale images: one of 1 KB per (expert, 192-row weight tile, K tile);
    # byte 512 p + 16 l + 4 c + b is tile row 128 p + 32 c + l, K block 4 t + b
    span = 192 // sections
    NT = -(-rs // span)
    exp = np.full((E, NT, KT, 2, 32, 4, 4), 127, np.uint8)
    for n in range(NT):
        for p in range(2):
            for c in range(4):
                for l in range(32):
                    tr = 128 * p + 32 * c + l
                    if tr >= 192:
                        continue
                    sec, srow = tr // span, span * n + tr % span
                    if srow >= rs:
                        continue
                    for t in range(KT):
                        for b in range(4):
                            blk = 4 * t + b
                            if blk < K // 32:
                                exp[:, n, t, p, l, c, b] = sc[:, sec * rs + srow, blk]
    assert np.array_equal(imgs.cpu().numpy(), exp.ravel())


@pytest.mark.parametrize("case", MX_CASES, ids=lambda c: "T%d_H%d_I%d_E%d_K%d" % c)
def test_mx_gemm1_stage(case):
    cfg, inp = _mx_problem(case, 41)
    T, H, I, E, K = case
    d = inp.to("cuda")
    xq_ref, s_ref = oracle.quantize_x_fp8(np_store(inp.x))  # fp8 codes as the method forms them
    al_ref = oracle.align(inp.topk_ids.numpy(), E, 128)
    al = moe.align(d.topk_ids, E, 128)
    p = moe.make_problem(T, H, I, E, K, "bf16", "mxfp4", h_scale=0.5)
    cap = moe.moe_align_capacity(T, K, E, 128)
    hq = torch.zeros((cap, I), dtype=torch.uint8, device="cuda")
    st = _status()
    w13p, s13p = moe.pack_mx(d.w13, d.w13_scale, 2)
    # the oracle's codes placed at the sorted slots of their tokens
    xs = np.zeros((cap, H), np.uint8)
    valid = al_ref["sorted_ids"] < T * K
    xs[valid] = xq_ref[al_ref["sorted_ids"][valid] // K]
    moe.moe_gemm1_silu(p, torch.from_numpy(xs).cuda(), torch.from_numpy(s_ref).cuda(), w13p,
                       s13p, al["sorted_ids"], al["block_info"], al["num_blocks"], hq, st)
    assert moe.moe_get_device_status(st) == 0
    rows = _valid_rows(al_ref, T * K)
    eor = _expert_of_rows(al_ref, rows, inp.topk_ids.numpy().ravel())
    P = oracle_problem(inp, quantize_x=True, h_e4m3=True, h_scale=0.5)
    emu = oracle.gemm1_silu_rows(P, np_store(inp.x), np_store(inp.w13), al_ref["sorted_ids"], eor,
                                 rows, w13_scale=np_store(inp.w13_scale), mode=oracle.EMULATE)
    got = oracle.e4m3_to_float(hq[torch.from_numpy(rows).long().cuda()].cpu().numpy()) * 0.5
    # the stored codes equal the oracle's rounding of the same values, except
    # where the fp32 and fp64 sums straddle a rounding boundary (one step)
    step = np.maximum(np.abs(emu) * 2.0 ** -3, 2.0 ** -9 * 0.5)
    assert np.all(np.abs(got - emu) <= step * 1.001)
    assert (got != emu).mean() < 1e-3
    exact = oracle.gemm1_silu_rows(P, np_store(inp.x), np_store(inp.w13), al_ref["sorted_ids"],
                                   eor, rows, w13_scale=np_store(inp.w13_scale))
    assert np.linalg.norm(got - exact) / np.linalg.norm(exact) < MX_REL_EXACT


@pytest.mark.parametrize("splits", [1, 2])
@pytest.mark.parametrize("case", MX_CASES, ids=lambda c: "T%d_H%d_I%d_E%d_K%d" % c)
def test_mx_gemm2_stage(case, splits):
    cfg, inp = _mx_problem(case, 42)
    T, H, I, E, K = case
    d = inp.to("cuda")
    cap = moe.moe_align_capacity(T, K, E, 128)
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 256, (cap, I)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38  # no NaN codes: 1.0 instead
    al_ref = oracle.align(inp.topk_ids.numpy(), E, 128)
    al = moe.align(d.topk_ids, E, 128)
    p = moe.make_problem(T, H, I, E, K, "bf16", "mxfp4", h_scale=0.25)
    y = torch.full((splits, cap, H), float("nan"), dtype=torch.float32, device="cuda")
    st = _status()
    w2p, s2p = moe.pack_mx(d.w2, d.w2_scale, 1)
    moe.moe_gemm2_weighted(p, torch.from_numpy(codes).cuda(), w2p, s2p, d.topk_weights,
                           al["sorted_ids"], al["block_info"], al["num_blocks"], y, splits, st)
    assert moe.moe_get_device_status(st) == 0
    rows = _valid_rows(al_ref, T * K)
    eor = _expert_of_rows(al_ref, rows, inp.topk_ids.numpy().ravel())
    P = oracle_problem(inp, h_e4m3=True, h_scale=0.25)
    ref = oracle.gemm2_weighted_rows(P, codes, np_store(inp.w2), inp.topk_weights.numpy(),
                                     al_ref["sorted_ids"], eor, rows,
                                     w2_scale=np_store(inp.w2_scale), h_is_e4m3=True)
    got = y[:, torch.from_numpy(rows).long().cuda()].sum(0)
    # e4m3 x e2m1 x e8m0 products are exact; only the fp32 summation differs
    assert_close(got, ref, max_abs=2e-2, rel_l2=1e-4, what="y")


def _run_forward_mx(d, cfg, h_scale=1.0):
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, "bf16", "mxfp4", h_scale=h_scale)
    ws = moe.Workspace(p)
    ws.buffer.fill_(0xFF)
    out = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    w13p, s13p = moe.pack_mx(d.w13, d.w13_scale, 2)
    w2p, s2p = moe.pack_mx(d.w2, d.w2_scale, 1)
    moe.moe_forward(p, d.x, d.topk_ids, d.topk_weights, w13p, s13p, w2p, s2p, out, ws.buffer,
                    ws.nbytes)
    assert moe.moe_get_device_status(ws.status) == 0
    return out


def _check_mx(out, inp, toks, h_scale=1.0):
    emu = oracle_forward_tokens(inp, toks, mode=oracle.EMULATE, quantize_x=True, h_e4m3=True,
                                h_scale=h_scale)
    exact = oracle_forward_tokens(inp, toks, mode=oracle.EXACT, quantize_x=True, h_e4m3=True,
                                  h_scale=h_scale)
    got = out[torch.from_numpy(np.asarray(toks)).long().cuda()]
    assert_close(got, emu, max_abs=MX_MAX_ABS, rel_l2=MX_REL_EMU, what="vs emulate")
    assert_close(got, exact, max_abs=np.inf, rel_l2=MX_REL_EXACT, what="vs exact")


@pytest.mark.parametrize("case", MX_CASES, ids=lambda c: "T%d_H%d_I%d_E%d_K%d" % c)
def test_forward_mx_small(case):
    cfg, inp = _mx_problem(case, 43)
    out = _run_forward_mx(inp.to("cuda"), cfg, h_scale=0.5)
    _check_mx(out, inp, np.arange(cfg.T), h_scale=0.5)


def test_forward_lowp_full_size_sampled():
    cfg = gen.config("lowp")
    inp = generate(cfg, seed=0, device="cuda")
    out = _run_forward_mx(inp, cfg)
    assert torch.isfinite(out.float()).all()
    toks, _ = block_tokens(inp, 128, seed=2)  # every align block of the 128-row tiles
    _check_mx(out, inp, toks)


# ------------------------------------------------------------------ expert shards

def _oracle_shard(inp, base, L, tokens, mode=oracle.EXACT, **kw):
    c = inp.cfg
    P = oracle.make_problem(c.T, c.H, c.I, c.E, c.K, np_store(inp.x[:1]), np_store(inp.w13[:1]),
                            expert_base=base, local_experts=L, **kw)
    sl = slice(base, base + L)
    sc = lambda t: None if t is None else np_store(t[sl].cpu())
    return oracle.forward(P, np_store(inp.x.cpu()), inp.topk_ids.cpu().numpy(),
                          inp.topk_weights.cpu().numpy(), np_store(inp.w13[sl].cpu()),
                          np_store(inp.w2[sl].cpu()), sc(inp.w13_scale), sc(inp.w2_scale),
                          mode=mode, tokens=tokens)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_forward_expert_shards(dtype):
    """Each shard's output against the oracle's shard; the shards' outputs
    sum to the unsharded forward."""
    cfg = gen.MoEConfig("shard", 200, 256, 320, 8, 2, dtype, "normal")
    inp = gen.generate(cfg, seed=41)
    d = inp.to("cuda")
    total = torch.zeros((cfg.T, cfg.H), dtype=torch.float64, device="cuda")
    for base, L in ((0, 3), (3, 4), (7, 1)):
        out = moe.forward(d.x, d.topk_ids, d.topk_weights, d.w13[base:base + L].contiguous(),
                          d.w2[base:base + L].contiguous(), num_experts=cfg.E, expert_base=base)
        ref = _oracle_shard(inp, base, L, np.arange(cfg.T))
        assert_close(out, ref, what=f"shard {base}+{L}")
        # tokens none of whose experts live here get an exact zero row
        ids = inp.topk_ids.numpy()
        none = ~((ids >= base) & (ids < base + L)).any(1)
        assert torch.all(out[torch.from_numpy(none).cuda()] == 0)
        total += out.double()
    full, _ = _run_forward(d, cfg)
    # each shard's output is rounded once to the activation type
    assert_close(total, full.double().cpu().numpy(), max_abs=4e-2, what="sum of shards")


@pytest.mark.parametrize("fused", [False, True])
def test_forward_expert_shard_decode(fused):
    """A decode-sized batch (two K steps per stage) on one shard of 8 of 16
    experts, with either combine."""
    cfg = gen.MoEConfig("shard_dec", 8, 256, 1536, 16, 2, "bf16", "normal")
    inp = gen.generate(cfg, seed=45)
    d = inp.to("cuda")
    base, L = 4, 8
    out = moe.forward(d.x, d.topk_ids, d.topk_weights, d.w13[base:base + L].contiguous(),
                      d.w2[base:base + L].contiguous(), num_experts=cfg.E, expert_base=base,
                      fused_combine=fused)
    assert_close(out, _oracle_shard(inp, base, L, np.arange(cfg.T)), what="decode shard")


def test_forward_expert_shard_mx():
    cfg = gen.MoEConfig("shard_mx", 96, 256, 320, 16, 4, "mxfp4", "uniform")
    inp = gen.generate(cfg, seed=42)
    d = inp.to("cuda")
    base, L = 4, 8
    sl = slice(base, base + L)
    w13p, s13p = moe.pack_mx(d.w13[sl].contiguous(), d.w13_scale[sl].contiguous(), 2)
    w2p, s2p = moe.pack_mx(d.w2[sl].contiguous(), d.w2_scale[sl].contiguous(), 1)
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, "bf16", "mxfp4", expert_base=base,
                         local_experts=L)
    ws = moe.Workspace(p)
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(p, d.x, d.topk_ids, d.topk_weights, w13p, s13p, w2p, s2p, out, ws.buffer,
                    ws.nbytes)
    assert moe.moe_get_device_status(ws.status) == 0
    emu = _oracle_shard(inp, base, L, np.arange(cfg.T), mode=oracle.EMULATE, quantize_x=True,
                        h_e4m3=True)
    assert_close(out, emu, max_abs=MX_MAX_ABS, rel_l2=MX_REL_EMU, what="mx shard vs emulate")


@pytest.mark.parametrize("case", [(300, 256, 320, 3, 2, "bf16", "normal"),
                                  (8, 256, 320, 8, 2, "bf16", "normal"),
                                  (33, 128, 256, 8, 2, "f32", "normal")],
                         ids=lambda c: "T%d_H%d_I%d_E%d_K%d_%s_%s" % c)
def test_forward_cuda_graph_replay(case):
    """moe_forward captured in a CUDA graph: every replay gives the eager
    output bit for bit (the default combine is deterministic)."""
    cfg = gen.MoEConfig("graph", *case)
    d = gen.generate(cfg, seed=34).to("cuda")
    eager, _ = _run_forward(d, cfg)
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.dtype)
    ws = moe.Workspace(p)
    out = torch.full((cfg.T, cfg.H), float("nan"), dtype=d.x.dtype, device="cuda")
    s = torch.cuda.Stream()

    def fwd():
        moe.moe_forward(p, d.x, d.topk_ids, d.topk_weights, d.w13, None, d.w2, None, out,
                        ws.buffer, ws.nbytes, s)

    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fwd()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s, capture_error_mode="relaxed"):
        fwd()
    for _ in range(2):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(ws.status) == 0
        assert torch.equal(out, eager)


# ------------------------------------------------------------------ fused combine

def _run_forward_fused(d, cfg, block_m=0, **kw):
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.dtype, block_m=block_m,
                         fused_combine=True, **kw)
    ws = moe.Workspace(p)
    ws.buffer.fill_(0xFF)  # the accumulator starts as NaN: the gather step must zero it
    out = torch.full((cfg.T, cfg.H), float("nan"), dtype=d.x.dtype, device="cuda")
    moe.moe_forward(p, d.x, d.topk_ids, d.topk_weights, d.w13, None, d.w2, None, out, ws.buffer,
                    ws.nbytes)
    assert moe.moe_get_device_status(ws.status) == 0
    return out, p


@pytest.mark.parametrize("bm", [0, 16, 256])
@pytest.mark.parametrize("case", FORWARD_CASES, ids=lambda c: "T%d_H%d_I%d_E%d_K%d_%s_%s" % c)
def test_forward_fused_combine(case, bm):
    cfg = gen.MoEConfig("fused", *case)
    inp = gen.generate(cfg, seed=31)
    d = inp.to("cuda")
    out, p = _run_forward_fused(d, cfg, block_m=bm)
    # the accumulator (T rows) replaces y (k_splits x cap rows)
    assert moe.moe_workspace_size(p) <= moe.moe_workspace_size(
        moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.dtype, block_m=bm))
    assert_close(out, oracle_forward_tokens(inp, np.arange(cfg.T)), what=cfg.name)
    # the deterministic combine differs only by the order of fp32 adds
    det, _ = _run_forward(d, cfg, block_m=bm)
    assert_close(out, det.double().cpu().numpy(), max_abs=2e-2, rel_l2=4e-3, what="vs combine")


def test_forward_fused_combine_k_splits_and_biases():
    """Several K splits of the down projection add into one accumulator row;
    the w2 bias joins once (first split), with the GPT-OSS epilogue."""
    cfg = gen.MoEConfig("fused_oai", 8, 256, 1536, 8, 2, "bf16", "normal", "swiglu_oai")
    inp = gen.generate(cfg, seed=53)
    d = inp.to("cuda")
    out, p = _run_forward_fused(d, cfg, **problem_kw(d))
    assert moe.moe_gemm2_default_splits(p) > 1
    assert_close(out, oracle_forward_tokens(inp, np.arange(cfg.T)), what="fused, split K")


def test_forward_fused_combine_shard():
    cfg = gen.MoEConfig("fused_shard", 200, 256, 320, 8, 2, "bf16", "normal")
    inp = gen.generate(cfg, seed=41)
    d = inp.to("cuda")
    base, L = 3, 4
    out = moe.forward(d.x, d.topk_ids, d.topk_weights, d.w13[base:base + L].contiguous(),
                      d.w2[base:base + L].contiguous(), num_experts=cfg.E, expert_base=base,
                      fused_combine=True)
    assert_close(out, _oracle_shard(inp, base, L, np.arange(cfg.T)), what="fused shard")
    ids = inp.topk_ids.numpy()
    none = ~((ids >= base) & (ids < base + L)).any(1)
    assert torch.all(out[torch.from_numpy(none).cuda()] == 0)


def test_forward_fused_combine_mx():
    cfg, inp = _mx_problem(MX_CASES[0], 44)
    d = inp.to("cuda")
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, "bf16", "mxfp4", h_scale=0.5,
                         fused_combine=True)
    ws = moe.Workspace(p)
    ws.buffer.fill_(0xFF)
    out = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    w13p, s13p = moe.pack_mx(d.w13, d.w13_scale, 2)
    w2p, s2p = moe.pack_mx(d.w2, d.w2_scale, 1)
    moe.moe_forward(p, d.x, d.topk_ids, d.topk_weights, w13p, s13p, w2p, s2p, out, ws.buffer,
                    ws.nbytes)
    assert moe.moe_get_device_status(ws.status) == 0
    _check_mx(out, inp, np.arange(cfg.T), h_scale=0.5)


def test_forward_fused_combine_status_blocks_output():
    cfg = gen.MoEConfig("fwd", 64, 128, 128, 4, 2, "bf16", "normal")
    d = gen.generate(cfg, seed=33).to("cuda")
    d.topk_ids[5, 1] = 4  # outside [0, E)
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.dtype, fused_combine=True)
    ws = moe.Workspace(p)
    out = torch.zeros((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(p, d.x, d.topk_ids, d.topk_weights, d.w13, None, d.w2, None, out, ws.buffer,
                    ws.nbytes)
    assert moe.moe_get_device_status(ws.status) == _abi.MOE_ERR_DEVICE_BAD_ID
    assert (out == 0).all()


@pytest.mark.parametrize("name", ["mixtral_prefill", "dsv3_prefill"])
def test_forward_fused_combine_full_size_sampled(name):
    cfg = gen.config(name)
    inp = generate(cfg, seed=0, device="cuda")
    out, p = _run_forward_fused(inp, cfg)
    toks, _ = block_tokens(inp, moe.moe_resolve_block_m(p), seed=3)
    assert_close(out[torch.from_numpy(toks).long().cuda()], oracle_forward_tokens(inp, toks),
                 what=name + " fused")
    assert torch.isfinite(out.float()).all()
    del inp, out
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ GPT-OSS expert FFN

OAI_CASES = [
    # T, H, I, E, K, dtype -- clamped SwiGLU, biases, interleaved gate/linear rows
    (300, 256, 320, 3, 2, "bf16"),
    (8, 256, 1536, 8, 2, "bf16"),    # few tokens: the down projection splits K
    (40, 128, 256, 8, 2, "f32"),
]


@pytest.mark.parametrize("case", OAI_CASES, ids=lambda c: "T%d_H%d_I%d_E%d_K%d_%s" % c)
def test_forward_swiglu_oai(case):
    cfg = gen.MoEConfig("oai", *case, "normal", "swiglu_oai")
    inp = gen.generate(cfg, seed=51)
    d = inp.to("cuda")
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.dtype, **problem_kw(d))
    if cfg.T <= 8:
        assert moe.moe_gemm2_default_splits(p) > 1
    out = moe.forward(d.x, d.topk_ids, d.topk_weights, d.w13, d.w2, **problem_kw(d))
    ref = oracle_forward_tokens(inp, np.arange(cfg.T))
    assert_close(out, ref, what=cfg.name)


def test_pack_mx_interleaved_equals_halves():
    E, R, K = 3, 2 * 96, 320
    g = torch.Generator().manual_seed(9)
    w = torch.randint(0, 256, (E, R, K // 2), generator=g, dtype=torch.uint8)
    sc = torch.randint(100, 140, (E, R, K // 32), generator=g, dtype=torch.uint8)
    inter_w = torch.empty_like(w)
    inter_s = torch.empty_like(sc)
    inter_w[:, 0::2], inter_w[:, 1::2] = w[:, :R // 2], w[:, R // 2:]
    inter_s[:, 0::2], inter_s[:, 1::2] = sc[:, :R // 2], sc[:, R // 2:]
    a = moe.pack_mx(w.cuda(), sc.cuda(), 2)
    b = moe.pack_mx(inter_w.cuda(), inter_s.cuda(), 2, interleaved=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def _run_oai_mx(d, cfg):
    kw = problem_kw(d)
    w13p, s13p = moe.pack_mx(d.w13, d.w13_scale, 2, interleaved=True)
    w2p, s2p = moe.pack_mx(d.w2, d.w2_scale, 1)
    return moe.forward(d.x, d.topk_ids, d.topk_weights, w13p, w2p, w13_scale=s13p, w2_scale=s2p,
                       weight="mxfp4", h_scale=d.h_scale, intermediate=cfg.I, **kw)


@pytest.mark.parametrize("case", [(96, 256, 320, 16, 4), (5, 512, 256, 8, 2)],
                         ids=lambda c: "T%d_H%d_I%d_E%d_K%d" % c)
def test_forward_swiglu_oai_mx(case):
    cfg = gen.MoEConfig("oai_mx", *case, "mxfp4", "uniform", "swiglu_oai")
    inp = gen.generate(cfg, seed=52)
    d = inp.to("cuda")
    out = _run_oai_mx(d, cfg)
    _check_mx(out, inp, np.arange(cfg.T), h_scale=inp.h_scale)


def test_forward_lowp_oai_full_size_sampled():
    cfg = gen.config("lowp_oai")
    d = gen.generate(cfg, seed=0, device="cuda")
    out = _run_oai_mx(d, cfg)
    assert torch.isfinite(out.float()).all()
    toks, _ = block_tokens(d, 128, seed=5)
    _check_mx(out, d, toks, h_scale=d.h_scale)


# ------------------------------------------------------------------ edge cases of the method

def _scale_gate_up(inp, gate_shift, up_shift):
    """Scale w13's gate rows by 2^gate_shift and its up rows by 2^up_shift,
    exactly: bf16 weights times a power of two, or mxfp4 e8m0 codes shifted
    (the e2m1 values stay).  Rows follow the workload's layout (halves, or
    GPT-OSS's alternating rows)."""
    I = inp.cfg.I
    gate = slice(0, 2 * I, 2) if inp.interleaved else slice(0, I)
    up = slice(1, 2 * I, 2) if inp.interleaved else slice(I, 2 * I)
    if inp.w13_scale is None:
        w = inp.w13.clone()
        w[:, gate] *= 2.0 ** gate_shift
        w[:, up] *= 2.0 ** up_shift
        inp.w13 = w
    else:
        s = inp.w13_scale.to(torch.int32)
        s[:, gate] += gate_shift
        s[:, up] += up_shift
        assert int(s.min()) >= 1 and int(s.max()) <= 254
        inp.w13_scale = s.to(torch.uint8)
    return inp


@pytest.mark.parametrize("kind", ["bf16", "bf16_oai", "mxfp4", "mxfp4_oai"])
def test_forward_gate_far_past_exp_overflow(kind):
    """Gate pre-activations of |g| up to several hundred, where e^-g
    overflows fp32 for g < -88 (SiLU(g) -> -0) and SiLU(g) = g above it; for
    GPT-OSS's clamped SwiGLU the gate is also far above `limit` and the
    linear branch far outside [-limit, limit] (up rows scaled up).  The up
    rows are scaled so that the output keeps its usual magnitude."""
    oai = kind.endswith("_oai")
    mx = kind.startswith("mxfp4")
    cfg = gen.MoEConfig("edge", 96, 256, 320, 8, 2, "mxfp4" if mx else "bf16",
                        "uniform" if mx else "normal", "swiglu_oai" if oai else "silu")
    inp = _scale_gate_up(gen.generate(cfg, seed=61), 7, 3 if oai else -7)
    d = inp.to("cuda")
    # the gate reaches far past 88 in both directions
    xg = d.x.float() @ (d.w13[0, 0:2 * cfg.I:2] if oai else d.w13[0, :cfg.I]).float().T \
        if not mx else None
    if xg is not None:
        assert float(xg.max()) > 100 and float(xg.min()) < -100
    if mx:
        out = _run_oai_mx(d, cfg) if oai else _run_forward_mx(d, cfg)
        _check_mx(out, inp, np.arange(cfg.T), h_scale=inp.h_scale if oai else 1.0)
    else:
        out = moe.forward(d.x, d.topk_ids, d.topk_weights, d.w13, d.w2, **problem_kw(d))
        assert_close(out, oracle_forward_tokens(inp, np.arange(cfg.T)), what=kind)


@pytest.mark.parametrize("fused", [False, True])
def test_forward_non_finite_token_stays_in_its_row(fused):
    """A NaN and an infinity in one token's x: that token's output row is
    non-finite like the oracle's, and every other token's row matches the
    oracle (no tile mixes tokens)."""
    cfg = gen.MoEConfig("nonfinite", 64, 256, 320, 4, 2, "bf16", "normal")
    inp = gen.generate(cfg, seed=62)
    inp.x[7, 3] = float("nan")
    inp.x[20, 0] = float("inf")
    d = inp.to("cuda")
    out = moe.forward(d.x, d.topk_ids, d.topk_weights, d.w13, d.w2, fused_combine=fused)
    ref = oracle_forward_tokens(inp, np.arange(cfg.T))
    got = out.double().cpu().numpy()
    bad = np.zeros(cfg.T, bool)
    bad[[7, 20]] = True
    assert not np.isfinite(ref[bad]).any() and not np.isfinite(got[bad]).any()
    assert_close(out[torch.from_numpy(~bad).cuda()], ref[~bad], what="finite tokens")
