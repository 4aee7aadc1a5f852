"""Pins for the CPU oracle: each checks the oracle against something other than
itself -- a library routine (numpy / torch), a closed form, an invariant of the
definition, or a special case that reduces to a dense MLP.

The pins are plain functions that raise AssertionError, so that
``test_oracle_pins.py`` runs them against the real oracle and
``test_oracle_mutants.py`` runs them against copies of the oracle with a
planted mistake, to show that each plausible mistake fails at least one pin.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from mixture_experts_grouped_02_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden_constants():
    out = {}
    with open(os.path.join(GOLDEN, "page_constants.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, *vals = line.split()
            out[name] = [float(v) for v in vals]
    return out


def np_store(t):
    return gen.to_numpy_storage(t)


def rand_problem(T, H, I, E, K, dtype="f32", seed=0, routing="normal"):
    cfg = gen.MoEConfig("pin", T, H, I, E, K, dtype, routing)
    return gen.generate(cfg, seed=seed)


def prob_for(inp, **kw):
    c = inp.cfg
    return oracle.make_problem(c.T, c.H, c.I, c.E, c.K, np_store(inp.x), np_store(inp.w13), **kw)


def run_forward(inp, mode=oracle.EXACT, tokens=None, **kw):
    return oracle.forward(prob_for(inp, **kw), np_store(inp.x), inp.topk_ids.numpy(),
                          inp.topk_weights.numpy(), np_store(inp.w13), np_store(inp.w2),
                          np_store(inp.w13_scale), np_store(inp.w2_scale), mode=mode,
                          tokens=tokens)


def to64(t):
    return t.to(torch.float64) if t.dtype != torch.uint8 else None


def dense_swiglu(x64, w13_64, w2_64):
    """Dense SwiGLU MLP with torch's own silu: rows of w13 = [gate; up]."""
    I = w13_64.shape[0] // 2
    g = x64 @ w13_64[:I].T
    u = x64 @ w13_64[I:].T
    return (F.silu(g) * u) @ w2_64.T


E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # OCP MX v1.0, FP4 E2M1


def dequant_mx(packed, scale):
    """Reference dequantisation of packed e2m1 + e8m0 with torch ops."""
    lo = (packed & 15).to(torch.int64)
    hi = (packed >> 4).to(torch.int64)
    nib = torch.stack([lo, hi], dim=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    mag = torch.tensor(E2M1_GRID, dtype=torch.float64)[nib & 7]
    val = torch.where((nib & 8) != 0, -mag, mag)
    s = torch.pow(2.0, scale.to(torch.float64) - 127.0)
    return val * s.repeat_interleave(32, dim=-1)


# ---------------------------------------------------------------- align pins

ALIGN_CASES = [
    # (T, K, E, bm, kind)
    (16, 2, 8, 16, "normal"),
    (37, 3, 8, 32, "normal"),
    (64, 2, 1, 64, "normal"),
    (100, 8, 256, 128, "normal"),
    (5, 2, 256, 16, "normal"),
    (300, 4, 16, 64, "one_expert"),
    (257, 2, 32, 32, "skewed"),
    (9000, 8, 64, 128, "normal"),  # T*K = 72000 > 2^16
]


def align_ids(T, K, E, kind, seed=0):
    rng = np.random.default_rng(seed)
    if kind == "one_expert":
        # every token's first slot goes to expert 3, the rest elsewhere
        ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
        ids[:, 0] = 3 % E
        for t in range(T):
            others = [e for e in range(E) if e != 3 % E]
            ids[t, 1:] = rng.choice(others, K - 1, replace=False)
        return ids
    if kind == "skewed":
        p = 1.0 / np.arange(1, E + 1) ** 2.0
        p /= p.sum()
        return np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    if E >= K:
        return np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    return rng.integers(0, E, (T, K)).astype(np.int32)


def pin_align_vs_stable_argsort(T, K, E, bm, kind):
    ids = align_ids(T, K, E, kind)
    a = oracle.align(ids, E, bm)
    flat = ids.ravel()
    na = flat.size
    counts = np.bincount(flat, minlength=E)
    assert np.array_equal(a["counts"], counts)
    assert np.array_equal(a["offsets"], np.concatenate([[0], np.cumsum(counts)]))
    padded = -(-counts // bm) * bm
    po = np.concatenate([[0], np.cumsum(padded)])
    assert np.array_equal(a["padded_offsets"], po)
    order = np.argsort(flat, kind="stable")  # library stable sort by expert id
    cap = oracle.align_capacity(T, K, E, bm)
    assert cap == na + min(E, na) * (bm - 1)
    expect = np.full(cap, na, np.int32)
    for e in range(E):
        seg = order[np.searchsorted(flat[order], e, "left"):np.searchsorted(flat[order], e,
                                                                             "right")]
        expect[po[e]:po[e] + len(seg)] = seg
    assert np.array_equal(a["sorted_ids"], expect)
    inv = np.empty(na, np.int64)
    valid = expect < na
    inv[expect[valid]] = np.nonzero(valid)[0]
    assert np.array_equal(a["inv_perm"], inv)
    nb = int(po[-1] // bm)
    assert a["num_blocks"] == nb
    bi = a["block_info"]
    assert bi.shape == (cap // bm, 4)
    blk_expert = np.repeat(np.arange(E), padded // bm)
    assert np.array_equal(bi[:nb, 0], blk_expert)
    assert np.array_equal(bi[:nb, 2], np.arange(nb) * bm)
    for b in range(nb):
        e = blk_expert[b]
        m = (b * bm - po[e]) // bm
        assert bi[b, 1] == m
        assert bi[b, 3] == min(bm, counts[e] - m * bm) and bi[b, 3] >= 1
    assert np.all(bi[nb:] == np.array([-1, 0, 0, 0]))


def pin_align_invariants():
    for (T, K, E, bm, kind) in ALIGN_CASES[:6]:
        ids = align_ids(T, K, E, kind, seed=7)
        a = oracle.align(ids, E, bm)
        na = T * K
        s = a["sorted_ids"]
        assert a["counts"].sum() == na
        assert np.all(np.diff(a["offsets"]) >= 0)
        assert np.all(a["padded_offsets"] % bm == 0)
        # a bijection between flat indices and valid slots
        assert np.array_equal(s[a["inv_perm"]], np.arange(na))
        assert (s < na).sum() == na
        # every slot of a block belongs to the block's expert, in ascending order
        for b in range(a["num_blocks"]):
            e, m, r0, v = a["block_info"][b]
            rows = s[r0:r0 + v]
            assert np.all(ids.ravel()[rows] == e)
            assert np.all(np.diff(rows) > 0)
            assert np.all(s[r0 + v:r0 + bm] == na)


def pin_align_rejects_bad_id():
    ids = np.array([[0, 1], [2, 8]], np.int32)
    try:
        oracle.align(ids, 8, 16)
    except ValueError:
        return
    raise AssertionError("id 8 with E=8 was accepted")


# ---------------------------------------------------------------- FFN pins

def pin_identical_experts_dense_mlp():
    """All experts share weights => out = (sum_k w) * dense SwiGLU MLP."""
    for dtype in ("f32", "bf16"):
        inp = rand_problem(12, 64, 96, 4, 2, dtype, seed=3)
        inp.w13 = inp.w13[:1].repeat(4, 1, 1).contiguous()
        inp.w2 = inp.w2[:1].repeat(4, 1, 1).contiguous()
        out = run_forward(inp)
        ref = dense_swiglu(inp.x.to(torch.float64), inp.w13[0].to(torch.float64),
                           inp.w2[0].to(torch.float64))
        ref = ref * inp.topk_weights.to(torch.float64).sum(1, keepdim=True)
        assert np.allclose(out, ref.numpy(), rtol=1e-10, atol=1e-12), np.abs(out - ref.numpy()).max()


def pin_top1_unit_weight_per_expert_ffn():
    """top_k = 1 with weight 1 => out[t] = FFN of expert ids[t] on x[t]."""
    inp = rand_problem(20, 64, 32, 5, 1, "bf16", seed=4)
    inp.topk_weights = torch.ones_like(inp.topk_weights)
    out = run_forward(inp)
    x = inp.x.to(torch.float64)
    for t in range(inp.cfg.T):
        e = int(inp.topk_ids[t, 0])
        ref = dense_swiglu(x[t:t + 1], inp.w13[e].to(torch.float64), inp.w2[e].to(torch.float64))
        assert np.allclose(out[t], ref[0].numpy(), rtol=1e-10, atol=1e-12)


def pin_weighted_sum_over_slots():
    """K > 1 with distinct experts: out = sum_k w_k * FFN_{e_k}(x_t) (torch)."""
    inp = rand_problem(10, 32, 48, 6, 3, "f32", seed=5)
    out = run_forward(inp)
    x = inp.x.to(torch.float64)
    for t in range(inp.cfg.T):
        ref = torch.zeros(inp.cfg.H, dtype=torch.float64)
        for k in range(3):
            e = int(inp.topk_ids[t, k])
            ref += float(inp.topk_weights[t, k]) * dense_swiglu(
                x[t:t + 1], inp.w13[e].to(torch.float64), inp.w2[e].to(torch.float64))[0]
        assert np.allclose(out[t], ref.numpy(), rtol=1e-10, atol=1e-12)


def pin_loop_orders_agree():
    for dtype in ("f32", "bf16"):
        inp = rand_problem(24, 64, 64, 8, 2, dtype, seed=6)
        P = prob_for(inp)
        a = oracle.forward(P, np_store(inp.x), inp.topk_ids.numpy(), inp.topk_weights.numpy(),
                           np_store(inp.w13), np_store(inp.w2))
        b = oracle.forward_by_expert(P, np_store(inp.x), inp.topk_ids.numpy(),
                                     inp.topk_weights.numpy(), np_store(inp.w13),
                                     np_store(inp.w2))
        assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def pin_zero_input():
    inp = rand_problem(8, 32, 32, 4, 2, "f32", seed=8)
    inp.x = torch.zeros_like(inp.x)
    assert np.all(run_forward(inp) == 0.0)


def pin_linearity():
    inp = rand_problem(8, 32, 64, 4, 2, "f32", seed=9)
    base = run_forward(inp)
    inp2 = gen.MoEInputs(inp.cfg, inp.x, inp.w13, inp.w2 * 2.0, inp.topk_ids, inp.topk_weights)
    assert np.allclose(run_forward(inp2), 2.0 * base, rtol=1e-13, atol=0)
    inp3 = gen.MoEInputs(inp.cfg, inp.x, inp.w13, inp.w2, inp.topk_ids, inp.topk_weights * 0.5)
    assert np.allclose(run_forward(inp3), 0.5 * base, rtol=1e-13, atol=0)


def _scalar_ffn(g, u, c, w=1.0):
    """H = I = E = K = 1, x = 1: out = w * c * SiLU(g) * u."""
    cfg = gen.MoEConfig("scalar", 1, 1, 1, 1, 1, "f32", "normal")
    inp = gen.MoEInputs(cfg, torch.ones(1, 1), torch.tensor([[[g], [u]]], dtype=torch.float32),
                        torch.tensor([[[c]]], dtype=torch.float32),
                        torch.zeros(1, 1, dtype=torch.int32), torch.tensor([[w]]))
    return float(run_forward(inp)[0, 0])


def pin_silu_closed_forms():
    # g = ln 3: sigmoid(g) = 3/4, so SiLU(g) = 3/4 g; up = 2, c = 0.5
    g = float(np.float32(math.log(3.0)))
    got = _scalar_ffn(g, 2.0, 0.5)
    assert abs(got - 0.75 * g * 2.0 * 0.5) < 1e-7, got
    # gate and up are not interchangeable: SiLU(2)*ln3 differs from 0.75*ln3*2
    assert abs(_scalar_ffn(2.0, g, 0.5) - 0.75 * g * 2.0 * 0.5) > 1e-2
    assert _scalar_ffn(0.0, 5.0, 3.0) == 0.0  # SiLU(0) = 0
    assert _scalar_ffn(40.0, 1.5, 2.0) == 40.0 * 1.5 * 2.0  # SiLU(g) = g for large g
    assert abs(_scalar_ffn(-40.0, 1.5, 2.0)) < 1e-14  # SiLU(-inf) -> 0
    assert abs(_scalar_ffn(g, 2.0, 0.5, w=0.25) - 0.25 * 0.75 * g) < 1e-7


def pin_token_subset():
    inp = rand_problem(16, 32, 32, 4, 2, "bf16", seed=10)
    full = run_forward(inp)
    toks = np.array([15, 0, 7, 7], np.int32)
    assert np.array_equal(run_forward(inp, tokens=toks), full[toks])


def pin_emulate_close_to_exact():
    inp = rand_problem(16, 64, 64, 4, 2, "bf16", seed=11)
    a = run_forward(inp)
    b = run_forward(inp, mode=oracle.EMULATE)
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 0 < rel < 1e-2


def pin_stage_composition():
    """combine(gemm2(gemm1)) over the aligned slots reproduces the forward
    (fp32 intermediates, EMULATE mode rounds a to fp32 the same way)."""
    inp = rand_problem(16, 32, 64, 4, 2, "f32", seed=12)
    c = inp.cfg
    al = oracle.align(inp.topk_ids.numpy(), c.E, 16)
    P = prob_for(inp)
    rows = np.arange(len(al["sorted_ids"]), dtype=np.int32)
    flat = inp.topk_ids.numpy().ravel()
    s = al["sorted_ids"]
    eor = np.where(s < c.n_assign, flat[np.minimum(s, c.n_assign - 1)], 0).astype(np.int32)
    h = oracle.gemm1_silu_rows(P, np_store(inp.x), np_store(inp.w13), s, eor, rows)
    y = oracle.gemm2_weighted_rows(P, h.astype(np.float32), np_store(inp.w2),
                                   inp.topk_weights.numpy(), s, eor, rows)
    out = oracle.combine(y.astype(np.float32), al["inv_perm"], c.T, c.K, c.H)
    ref = run_forward(inp, mode=oracle.EMULATE)
    assert np.allclose(out, ref, rtol=1e-5, atol=1e-6)


# ---------------------------------------------------------------- format pins

def pin_e4m3_decode_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_to_float(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    k = golden_constants()["e4m3_max_code"]
    assert mine[int(k[0])] == k[1]


def pin_float_to_e4m3_vs_torch():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(2000) * 50,
        rng.standard_normal(500) * 1e-2,
        # exact midpoints between neighbouring codes, to test ties-to-even
        (oracle.e4m3_to_float(np.arange(1, 126)) + oracle.e4m3_to_float(np.arange(2, 127))) / 2,
    ]).astype(np.float32)
    vals = vals[np.abs(vals) < 464.0]  # torch's cast is not saturating above this
    mine = oracle.float_to_e4m3(vals)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # +0 / -0 both decode to zero; compare values
    assert np.array_equal(oracle.e4m3_to_float(mine), oracle.e4m3_to_float(ref))
    assert oracle.float_to_e4m3(np.array([1e6, -1e6], np.float32)).tolist() == [0x7E, 0xFE]


def pin_e2m1_e8m0():
    got = oracle.e2m1_to_float(np.arange(16))
    assert got[:8].tolist() == E2M1_GRID
    assert got[8:].tolist() == [-v for v in E2M1_GRID]
    k = golden_constants()["e8m0_unit_code"]
    assert oracle.e8m0_to_float(np.array([int(k[0])]))[0] == k[1]
    assert oracle.e8m0_to_float(np.array([0, 254])).tolist() == [2.0 ** -127, 2.0 ** 127]
    assert np.isnan(oracle.e8m0_to_float(np.array([255]))[0])


def pin_mx_weights_dense_mlp():
    """mxfp4 weights: identical experts reduce to a dense MLP on weights
    dequantised with torch ops from the OCP definition."""
    inp = rand_problem(6, 64, 64, 3, 2, "mxfp4", seed=13)
    for name in ("w13", "w2", "w13_scale", "w2_scale"):
        t = getattr(inp, name)
        setattr(inp, name, t[:1].repeat(3, 1, 1).contiguous())
    inp.x = inp.x.to(torch.float32)  # plain activations (no fp8 step here)
    out = run_forward(inp)
    w13 = dequant_mx(inp.w13[0], inp.w13_scale[0])
    w2 = dequant_mx(inp.w2[0], inp.w2_scale[0])
    ref = dense_swiglu(inp.x.to(torch.float64), w13, w2)
    ref = ref * inp.topk_weights.to(torch.float64).sum(1, keepdim=True)
    assert np.allclose(out, ref.numpy(), rtol=1e-10, atol=1e-12)


def pin_mx_scale_block_is_32():
    """Perturbing scale block 0 of the gate row changes exactly the outputs
    whose one-hot input column lies in K columns [0, 32)."""
    blk = int(golden_constants()["mx_block"][0])
    cfg = gen.MoEConfig("mxblk", 1, 64, 1, 1, 1, "mxfp4", "normal")
    w13 = torch.full((1, 2, 32), 0x22, dtype=torch.uint8)  # every element 1.0
    s13 = torch.full((1, 2, 2), 127, dtype=torch.uint8)
    changed = []
    for h in range(64):
        x = torch.zeros(1, 64)
        x[0, h] = 1.0
        P = oracle.make_problem(1, 64, 1, 1, 1, x.numpy(), w13.numpy())
        res = []
        for sc in (127, 128):
            s = s13.clone()
            s[0, 0, 0] = sc
            hrow = oracle.gemm1_silu_rows(P, x.numpy(), w13.numpy(), np.array([0], np.int32),
                                          np.array([0], np.int32), np.array([0], np.int32),
                                          w13_scale=s.numpy())
            res.append(hrow[0, 0])
        changed.append(res[0] != res[1])
    assert changed == [h < blk for h in range(64)]


def pin_mx_nibble_order():
    """Packed byte 0x21: the lower K index holds the low nibble (0.5), the
    next holds the high nibble (1.0)."""
    for h, expect_g in ((0, 0.5), (1, 1.0)):
        x = np.zeros((1, 64), np.float32)
        x[0, h] = 1.0
        w13 = np.full((1, 2, 32), 0x22, np.uint8)
        w13[0, 0, 0] = 0x21
        s = np.full((1, 2, 2), 127, np.uint8)
        P = oracle.make_problem(1, 64, 1, 1, 1, x, w13)
        hrow = oracle.gemm1_silu_rows(P, x, w13, np.array([0], np.int32), np.array([0], np.int32),
                                      np.array([0], np.int32), w13_scale=s)
        u = 1.0
        assert abs(hrow[0, 0] - expect_g / (1 + math.exp(-expect_g)) * u) < 1e-15


def pin_quantize_x_fp8():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((6, 96)) * np.array([[1], [10], [1e-3], [300], [0], [1]])).astype(
        np.float32)
    xq, s = oracle.quantize_x_fp8(x)
    xt = torch.from_numpy(x)
    amax = xt.abs().amax(1)
    s_ref = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))  # fp32 division
    assert np.array_equal(s, s_ref.numpy())
    q_ref = (xt / s_ref[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_to_float(xq), oracle.e4m3_to_float(q_ref))
    assert np.all(oracle.e4m3_to_float(xq[4]) == 0.0) and s[4] == 1.0  # (+-0 codes)
    # every row's amax lands on the largest code
    for t in (0, 1, 2, 3, 5):
        assert oracle.e4m3_to_float(np.abs(xq[t].astype(np.int64)) & 0x7F).max() == 448.0
    # error bound: half a unit in the last of 3 mantissa bits, or half the
    # subnormal step (2^-9) scaled
    deq = oracle.e4m3_to_float(xq) * s[:, None]
    bound = np.maximum(np.abs(x) * 2.0 ** -4, s[:, None] * 2.0 ** -10)
    assert np.all(np.abs(deq - x) <= bound * (1 + 1e-6))


def pin_lowp_forward_loop_orders():
    """fp8 x step + mx weights + e4m3 h: both loop orders agree, and the
    quantised forward is close to the unquantised-activation forward."""
    inp = rand_problem(10, 64, 64, 4, 2, "mxfp4", seed=14)
    P = prob_for(inp, quantize_x=True, h_e4m3=True, h_scale=1.0)
    args = (np_store(inp.x), inp.topk_ids.numpy(), inp.topk_weights.numpy(), np_store(inp.w13),
            np_store(inp.w2), np_store(inp.w13_scale), np_store(inp.w2_scale))
    a = oracle.forward(P, *args[:5], w13_scale=args[5], w2_scale=args[6], mode=oracle.EMULATE)
    b = oracle.forward_by_expert(P, *args[:5], w13_scale=args[5], w2_scale=args[6],
                                 mode=oracle.EMULATE)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)
    P0 = prob_for(inp)
    c = oracle.forward(P0, *args[:5], w13_scale=args[5], w2_scale=args[6])
    rel = np.linalg.norm(a - c) / np.linalg.norm(c)
    assert 1e-4 < rel < 0.1, rel


def _e4m3_nearest_torch(v):
    """Nearest e4m3 value of each fp32 v by torch's own cast (round to
    nearest even), after saturating to the largest finite code, 448."""
    v = np.clip(np.asarray(v, np.float32), -448.0, 448.0)
    return torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def _hidden_rows(a_over_scale, h_scale, mode):
    """h of one slot of an expert whose gate pre-activations are all 64 and
    whose up pre-activations are u_j = v_j h_scale / 64 (H = 1, x = 1).
    SiLU(64) = 64 in fp64 (e^-64 is far below half an ulp of 1), so the
    activation is a_j = 64 u_j = v_j h_scale exactly and a_j / h_scale = v_j."""
    v = np.asarray(a_over_scale, np.float64)
    I = len(v)
    u = (v * h_scale / 64.0).astype(np.float32)
    assert np.array_equal(u.astype(np.float64) * 64.0 / h_scale, v)  # dyadic, exact
    w13 = np.concatenate([np.full(I, 64.0, np.float32), u]).reshape(1, 2 * I, 1)
    x = np.ones((1, 1), np.float32)
    P = oracle.make_problem(1, 1, I, 1, 1, x, w13, h_e4m3=True, h_scale=h_scale)
    one = np.zeros(1, np.int32)
    return oracle.gemm1_silu_rows(P, x, w13, one, one, one, mode=mode)[0]


def pin_e4m3_hidden_store():
    """The e4m3 hidden activation of the low-precision path ("MOE Bmm1 Fused
    Gather", pack_fp8_out_fragment: out times 1/out_scale, then e4m3): in
    EMULATE mode the oracle keeps e4m3(a / h_scale) h_scale.  a / h_scale is
    placed on e4m3 grid points, on midpoints between neighbouring codes (ties
    go to the even code), past the saturation point 448 and below half the
    smallest subnormal; torch's float8 cast gives the expected codes."""
    grid = [1.0, 1.125, 2.0 ** -6, 2.0 ** -9, 448.0, 240.0, -3.5, 0.0]
    mids = [1.0625, 1.1875, 3.125, 3.375, -1.0625, 2.0 ** -6 + 2.0 ** -10, 232.0]
    extremes = [500.0, -1000.0, 2.0 ** -11]
    v = np.array(grid + mids + extremes)
    for h_scale in (4.0, 0.25):
        got = _hidden_rows(v, h_scale, oracle.EMULATE)
        assert np.array_equal(got, _e4m3_nearest_torch(v) * h_scale), (h_scale, got)
        # EXACT mode keeps the activation unrounded
        assert np.array_equal(_hidden_rows(v, h_scale, oracle.EXACT), v * h_scale)
    # hand-checked neighbours: ties to the even mantissa, saturation, underflow
    got = _hidden_rows([1.0625, 1.1875, 500.0, 2.0 ** -11], 4.0, oracle.EMULATE)
    assert got.tolist() == [4.0, 5.0, 448.0 * 4.0, 0.0], got


def pin_e4m3_hidden_in_down_projection():
    """The down projection reading e4m3 hidden codes decodes code x h_scale:
    against torch's float8_e4m3fn decode times h_scale, a float64 product
    with W2 (plain fp32 weights, and mxfp4 weights dequantised by torch ops)
    and the routing weight of each slot."""
    rng = np.random.default_rng(15)
    T, H, I, E, K, hs = 6, 24, 64, 3, 2, 0.25
    na = T * K
    codes = rng.integers(0, 256, (na, I)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38  # no NaN codes
    hdeq = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64) * hs
    eor = rng.integers(0, E, na).astype(np.int32)
    topk_w = rng.random(na).astype(np.float32)
    slots = np.arange(na, dtype=np.int32)
    w2_f32 = rng.standard_normal((E, H, I)).astype(np.float32)
    w2_mx = rng.integers(0, 256, (E, H, I // 2)).astype(np.uint8)
    s2_mx = rng.integers(120, 135, (E, H, I // 32)).astype(np.uint8)
    for w2, s2, W in ((w2_f32, None, torch.from_numpy(w2_f32).to(torch.float64)),
                      (w2_mx, s2_mx, dequant_mx(torch.from_numpy(w2_mx), torch.from_numpy(s2_mx)))):
        x = np.zeros((1, H), np.float32)
        # the weight format of the problem follows w13's storage type
        w13 = np.zeros((1, 2 * I, H), np.float32) if s2 is None else np.zeros((1, 2 * I, H // 2),
                                                                               np.uint8)
        P = oracle.make_problem(T, H, I, E, K, x, w13, h_e4m3=True, h_scale=hs)
        y = oracle.gemm2_weighted_rows(P, codes, w2, topk_w, slots, eor, slots, w2_scale=s2,
                                       h_is_e4m3=True)
        ref = torch.stack([float(topk_w[r]) * (W[eor[r]] @ hdeq[r]) for r in range(na)])
        assert np.allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def pin_bf16_hidden_store():
    """EMULATE mode with bf16 activations rounds each a_j once to the nearest
    bfloat16 (ties to even).  Gate 64 and up 1 + 2^-8 give a = 64.25, the
    midpoint of the bf16 neighbours 64 and 64.5: the even one, 64.  Up
    1 + 2^-8 + 2^-30 puts a 2^-24 above that midpoint: 64.5 (rounding through
    fp32 first would lose the 2^-24 and give 64)."""
    x = torch.ones(1, 3, dtype=torch.bfloat16)
    for up, want in (([1.0, 2.0 ** -8, 0.0], 64.0), ([1.0, 2.0 ** -8, 2.0 ** -30], 64.5),
                     ([1.0, 3 * 2.0 ** -9, 0.0], 64.5)):
        w13 = torch.tensor([[[64.0, 0.0, 0.0], up]], dtype=torch.bfloat16)
        assert w13.to(torch.float64)[0, 1].tolist() == up  # each entry exact in bf16
        P = oracle.make_problem(1, 3, 1, 1, 1, np_store(x), np_store(w13))
        one = np.zeros(1, np.int32)
        h = oracle.gemm1_silu_rows(P, np_store(x), np_store(w13), one, one, one,
                                   mode=oracle.EMULATE)
        assert h[0, 0] == want, (up, h[0, 0])


# ---------------------------------------------------------------- shard pins

SHARDS = [(0, 3), (3, 3), (6, 2)]  # an uneven partition of E = 8 experts


def _shard_forward(inp, base, L, **kw):
    c = inp.cfg
    P = oracle.make_problem(c.T, c.H, c.I, c.E, c.K, np_store(inp.x), np_store(inp.w13),
                            expert_base=base, local_experts=L, **kw)
    sl = slice(base, base + L)
    return oracle.forward(P, np_store(inp.x), inp.topk_ids.numpy(), inp.topk_weights.numpy(),
                          np_store(inp.w13[sl]), np_store(inp.w2[sl]))


def pin_shards_sum_to_full():
    """Expert shards partition the experts => their outputs add up to the
    unsharded output; a token none of whose experts a shard holds gets 0."""
    inp = rand_problem(40, 64, 32, 8, 2, "bf16", seed=12)
    full = run_forward(inp)
    parts = [_shard_forward(inp, b, L) for b, L in SHARDS]
    assert np.allclose(sum(parts), full, rtol=1e-12, atol=1e-13)
    ids = inp.topk_ids.numpy()
    for (b, L), part in zip(SHARDS, parts):
        none_local = ~((ids >= b) & (ids < b + L)).any(1)
        assert none_local.any()
        assert np.all(part[none_local] == 0.0)
    # a shard holding every expert is the plain forward, bit for bit
    assert np.array_equal(_shard_forward(inp, 0, 8), full)


def pin_shard_vs_torch():
    """One shard: out[t] = sum over the slots routed into the shard of
    w * FFN_e(x_t) (torch, fp64), with the shard's weights indexed from 0."""
    inp = rand_problem(12, 32, 48, 8, 3, "f32", seed=13)
    base, L = 2, 4
    out = _shard_forward(inp, base, L)
    x = inp.x.to(torch.float64)
    for t in range(inp.cfg.T):
        ref = torch.zeros(inp.cfg.H, dtype=torch.float64)
        for k in range(3):
            e = int(inp.topk_ids[t, k])
            if base <= e < base + L:
                ref += float(inp.topk_weights[t, k]) * dense_swiglu(
                    x[t:t + 1], inp.w13[e].to(torch.float64), inp.w2[e].to(torch.float64))[0]
        assert np.allclose(out[t], ref.numpy(), rtol=1e-10, atol=1e-12)


def pin_align_local_vs_stable_argsort():
    """A shard's align: numpy's stable sort of the assignments routed into
    the shard, keyed by local expert; inv_perm = -1 for the others."""
    for (T, K, E, bm, kind), (base, L) in (((37, 3, 8, 32, "normal"), (3, 4)),
                                            ((300, 4, 16, 64, "skewed"), (0, 5)),
                                            ((100, 8, 256, 128, "normal"), (200, 56))):
        ids = align_ids(T, K, E, kind, seed=3)
        a = oracle.align(ids, E, bm, expert_base=base, local_experts=L)
        flat = ids.ravel()
        na = flat.size
        local = (flat >= base) & (flat < base + L)
        counts = np.bincount(flat[local] - base, minlength=L)
        assert np.array_equal(a["counts"], counts)
        padded = -(-counts // bm) * bm
        po = np.concatenate([[0], np.cumsum(padded)])
        assert np.array_equal(a["padded_offsets"], po)
        assert np.array_equal(a["offsets"], np.concatenate([[0], np.cumsum(counts)]))
        cap = oracle.align_capacity(T, K, L, bm)
        assert len(a["sorted_ids"]) == cap
        idx = np.nonzero(local)[0]
        order = idx[np.argsort(flat[idx], kind="stable")]
        expect = np.full(cap, na, np.int32)
        pos = 0
        for e in range(L):
            seg = order[pos:pos + counts[e]]
            pos += counts[e]
            expect[po[e]:po[e] + len(seg)] = seg
        assert np.array_equal(a["sorted_ids"], expect)
        inv = np.full(na, -1, np.int64)
        valid = expect < na
        inv[expect[valid]] = np.nonzero(valid)[0]
        assert np.array_equal(a["inv_perm"], inv)
        nb = int(po[-1] // bm)
        assert a["num_blocks"] == nb
        assert np.array_equal(a["block_info"][:nb, 0], np.repeat(np.arange(L), padded // bm))


# ------------------------------------------------ clamped SwiGLU (GPT-OSS) pins

def _one_hot_problem(g, u, alpha, limit, w2_identity=True):
    """T = K = E = 1, x = e_0, gate/up rows with g_j / u_j in column 0 and
    W2 = identity (H = I), weight 1: out = a exactly as the activation
    gives it."""
    I = len(g)
    H = I
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1.0
    w13 = np.zeros((1, 2 * I, H), np.float32)
    w13[0, :I, 0] = g
    w13[0, I:, 0] = u
    w2 = np.eye(H, dtype=np.float32)[None] if w2_identity else np.zeros((1, H, I), np.float32)
    P = oracle.make_problem(1, H, I, 1, 1, x, w13, activation=oracle.ACT_SWIGLU_CLAMP,
                            swiglu_alpha=alpha, swiglu_limit=limit)
    out = oracle.forward(P, x, np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32), w13, w2)
    return out[0], w13[0, :I, 0].astype(np.float64), w13[0, I:, 0].astype(np.float64)


def pin_swiglu_clamp_closed_forms():
    """With alpha = 2 and limit = ln(3)/2, sigmoid(alpha * limit) = 3/4
    exactly: a gate above the limit gives limit * 3/4 * (u + 1); the linear
    branch is clamped to [-limit, limit]; a gate of -ln(3)/2 is not clamped
    and gives g / 4 * (u + 1); a very negative gate gives almost nothing (the
    gate has no lower clamp)."""
    lim = math.log(3.0) / 2.0
    g = [5.0, 5.0, 5.0, -lim, -5.0]
    u = [0.25, 3.0, -3.0, 0.5, 0.5]
    a, g32, u32 = _one_hot_problem(g, u, 2.0, lim)
    expect = [lim * 0.75 * 1.25, lim * 0.75 * (1 + lim), lim * 0.75 * (1 - lim),
              g32[3] * 0.25 * 1.5]
    assert np.allclose(a[:4], expect, rtol=2e-7, atol=0), (a, expect)
    assert abs(a[4]) < 1e-3, a[4]


def pin_swiglu_bias_is_a_ones_column():
    """The w13 bias equals one more input column of ones whose weights are
    the bias (the extra product is added last, as the bias is)."""
    inp = rand_problem(9, 32, 16, 4, 2, "f32", seed=14)
    rng = np.random.default_rng(3)
    b13 = rng.standard_normal((4, 32)).astype(np.float32)
    x = np_store(inp.x)
    w13 = np_store(inp.w13)
    kw = dict(activation=oracle.ACT_SWIGLU_CLAMP, swiglu_alpha=1.7, swiglu_limit=1.4)
    P = oracle.make_problem(9, 32, 16, 4, 2, x, w13, w13_bias=b13, **kw)
    got = oracle.forward(P, x, inp.topk_ids.numpy(), inp.topk_weights.numpy(), w13,
                         np_store(inp.w2))
    xa = np.concatenate([x, np.ones((9, 1), np.float32)], 1)
    w13a = np.concatenate([w13, b13[:, :, None]], 2)
    w2a = np.concatenate([np_store(inp.w2), np.zeros((4, 1, 16), np.float32)], 1)
    Pa = oracle.make_problem(9, 33, 16, 4, 2, xa, w13a, **kw)
    ref = oracle.forward(Pa, xa, inp.topk_ids.numpy(), inp.topk_weights.numpy(), w13a, w2a)
    assert np.array_equal(got, ref[:, :32])


def pin_w2_bias_closed_form():
    """W2 = 0: out[t] = sum_k w_k * b2[e_k] (numpy)."""
    inp = rand_problem(11, 16, 16, 5, 3, "f32", seed=15)
    rng = np.random.default_rng(4)
    b2 = rng.standard_normal((5, 16)).astype(np.float32)
    w2 = np.zeros((5, 16, 16), np.float32)
    x, w13 = np_store(inp.x), np_store(inp.w13)
    P = oracle.make_problem(11, 16, 16, 5, 3, x, w13, w2_bias=b2)
    out = oracle.forward(P, x, inp.topk_ids.numpy(), inp.topk_weights.numpy(), w13, w2)
    ids, w = inp.topk_ids.numpy(), inp.topk_weights.numpy().astype(np.float64)
    ref = np.einsum("tk,tkc->tc", w, b2[ids].astype(np.float64))
    assert np.allclose(out, ref, rtol=1e-14, atol=1e-15)


def pin_interleaved_gate_up():
    """w13 (and its bias) with gate/up rows interleaved give exactly the
    forward of the same rows put back into [gate; up] halves (numpy)."""
    inp = rand_problem(13, 32, 24, 3, 2, "bf16", seed=16)
    rng = np.random.default_rng(5)
    b13 = rng.standard_normal((3, 48)).astype(np.float32)
    w13 = np_store(inp.w13)  # (E, 2I, H): halves
    inter = np.empty_like(w13)
    inter[:, 0::2], inter[:, 1::2] = w13[:, :24], w13[:, 24:]
    b_inter = np.empty_like(b13)
    b_inter[:, 0::2], b_inter[:, 1::2] = b13[:, :24], b13[:, 24:]
    x, w2 = np_store(inp.x), np_store(inp.w2)
    kw = dict(activation=oracle.ACT_SWIGLU_CLAMP, swiglu_alpha=1.1, swiglu_limit=1.35)
    args = (x, inp.topk_ids.numpy(), inp.topk_weights.numpy())
    P1 = oracle.make_problem(13, 32, 24, 3, 2, x, inter, gate_up_interleaved=True,
                             w13_bias=b_inter, **kw)
    P2 = oracle.make_problem(13, 32, 24, 3, 2, x, w13, w13_bias=b13, **kw)
    a = oracle.forward(P1, *args, inter, w2)
    b = oracle.forward(P2, *args, w13, w2)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, oracle.forward(P2, *args, inter, w2))


# ---------------------------------------------------------------- router pins

def pin_route_vs_library():
    """ids: numpy's stable argsort of the negated logits, first K (ties to
    the lower id); weights: scipy's softmax over all E experts, taken at the
    chosen ids and renormalised (a different computation from the oracle's
    softmax over the K chosen logits)."""
    from scipy.special import softmax
    rng = np.random.default_rng(8)
    for T, E, K in ((37, 8, 2), (20, 256, 8), (5, 3, 3), (9, 1, 1)):
        logits = rng.standard_normal((T, E)).astype(np.float32)
        ids, w = oracle.route(logits, K)
        ref_ids = np.argsort(-logits, axis=1, kind="stable")[:, :K]
        assert np.array_equal(ids, ref_ids)
        p = softmax(logits.astype(np.float64), axis=1)
        pk = np.take_along_axis(p, ref_ids, 1)
        assert np.allclose(w, pk / pk.sum(1, keepdims=True), rtol=1e-12, atol=0)


def pin_route_ties_and_bf16():
    """Equal logits go to the lower expert id; bf16 logits are ranked at
    their stored values (two logits that round to the same bf16 tie)."""
    logits = np.array([[0.5, 2.0, 2.0, -1.0, 2.0],
                       [1.0, 1.0, 1.0, 1.0, 1.0]], np.float32)
    ids, w = oracle.route(logits, 3)
    assert ids.tolist() == [[1, 2, 4], [0, 1, 2]]
    assert np.allclose(w, 1.0 / 3.0, rtol=1e-15)
    b = torch.tensor([[1.0, 1.001, 0.5]], dtype=torch.float32).to(torch.bfloat16)
    assert float(b[0, 0]) == float(b[0, 1])  # 1.001 rounds to 1.0 in bf16
    ids, w = oracle.route(np_store(b), 2)
    assert ids.tolist() == [[0, 1]] and np.allclose(w, 0.5, rtol=1e-15)


def pin_route_matches_input_generator():
    """Without ties, the generator's route (softmax over all experts in
    fp32, stable top-k on the probabilities, renormalise) picks the same
    experts and, within fp32 rounding, the same weights."""
    cfg = gen.MoEConfig("route", 64, 8, 8, 32, 4, "f32", "zipf")
    logits = gen.router_logits(cfg, 3)
    ids, w = oracle.route(logits.numpy(), cfg.K)
    gi, gw = gen.route(logits, cfg.K)
    assert np.array_equal(ids, gi.numpy())
    assert np.allclose(w, gw.numpy(), rtol=2e-6, atol=0)


ROUTE_PINS = [pin_route_vs_library, pin_route_ties_and_bf16, pin_route_matches_input_generator]

SWIGLU_PINS = [pin_swiglu_clamp_closed_forms, pin_swiglu_bias_is_a_ones_column,
               pin_w2_bias_closed_form, pin_interleaved_gate_up]

SHARD_PINS = [pin_shards_sum_to_full, pin_shard_vs_torch, pin_align_local_vs_stable_argsort]

FFN_PINS = [
    pin_identical_experts_dense_mlp, pin_top1_unit_weight_per_expert_ffn,
    pin_weighted_sum_over_slots, pin_loop_orders_agree, pin_zero_input, pin_linearity,
    pin_silu_closed_forms, pin_token_subset, pin_emulate_close_to_exact, pin_stage_composition,
    pin_mx_weights_dense_mlp, pin_mx_scale_block_is_32, pin_mx_nibble_order,
    pin_lowp_forward_loop_orders, pin_e4m3_hidden_store, pin_e4m3_hidden_in_down_projection,
    pin_bf16_hidden_store,
]
FORMAT_PINS = [pin_e4m3_decode_vs_torch, pin_float_to_e4m3_vs_torch, pin_e2m1_e8m0,
               pin_quantize_x_fp8]
ALIGN_PINS = [pin_align_invariants, pin_align_rejects_bad_id] + [
    (lambda c=c: pin_align_vs_stable_argsort(*c)) for c in ALIGN_CASES
]
