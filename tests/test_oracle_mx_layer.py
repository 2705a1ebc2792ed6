"""The MXFP8 and fp8_bwd layer oracle against a brute-force scalar restatement on
tiny inputs, plus the bf16 rounding it uses for stored intermediates.

The brute force follows the layer's MXFP8 operand table (each GEMM operand in
32-element blocks along that GEMM's contraction axis: x, W_gate, W_up along H and
a, W_down along I in the forward; dy, W_down along H, dh, W_gate, W_up along I
for the input gradient; token-axis blocks from each expert's first row, the last
one zero-padded, for the weight gradients) one element and one block at a time.
Its e4m3 rounding is a nearest-value search over torch's float8_e4m3fn code
table; its bf16 rounding is Python's round-half-even on the scaled value.  Planted
mistakes in the oracle (a transposed block axis, a dropped quantisation, an
unrounded stored tensor) must fail the comparison.
"""
import math

import numpy as np
import pytest
import torch

import oracle.moe as om
from oracle import mx

# ------------------------------------------------------------------ scalar pieces
_codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
_vals = _codes.to(torch.float64).numpy()
E4M3_POS = np.unique(_vals[np.isfinite(_vals) & (_vals >= 0)])   # 0, 2^-9, ..., 448


def e4m3_nearest(v: float) -> float:
    a = min(abs(v), 448.0)                       # saturating
    i = int(np.searchsorted(E4M3_POS, a))
    if i < len(E4M3_POS) and E4M3_POS[i] == a:
        r = a
    else:
        lo, hi = E4M3_POS[i - 1], E4M3_POS[i]
        if a - lo < hi - a:
            r = lo
        elif hi - a < a - lo:
            r = hi
        else:                                     # tie: the even code
            r = lo if (i - 1) % 2 == 0 else hi
    return math.copysign(r, v)


def quant_block(vals):
    """One block (<= 32 values; a short block counts as zero-padded)."""
    amax = max(abs(v) for v in vals)
    if amax == 0.0:
        return [0.0] * len(vals)
    _, ex = math.frexp(amax)                      # amax = m * 2**ex, m in [0.5, 1)
    e = max(-127, min(127, (ex - 1) - 8))
    s = 2.0 ** e
    return [e4m3_nearest(v / s) * s for v in vals]


def quant_vec(vec):
    out = []
    for b in range(0, len(vec), 32):
        out += quant_block(list(vec[b:b + 32]))
    return out


def quant_rows(M):
    return np.array([quant_vec(list(r)) for r in M])


def quant_cols(M):
    return quant_rows(np.asarray(M).T).T


def bf16_scalar(v: float) -> float:
    if v == 0.0:
        return v
    _, ex = math.frexp(abs(v))
    step = 2.0 ** (max(ex - 1, -126) - 7)
    return math.copysign(round(abs(v) / step) * step, v)


bf16 = np.vectorize(bf16_scalar, otypes=[np.float64])


def sig(z):
    return 1.0 / (1.0 + math.exp(-z))


# ------------------------------------------------------------------ brute-force layer
def brute(d, prec):
    qf = prec == "mxfp8"
    qb = prec in ("mxfp8", "fp8_bwd")
    x, dy = np.asarray(d["x"], np.float64), np.asarray(d["dy"], np.float64)
    Wg, Wu, Wd = (np.asarray(d[k], np.float64) for k in ("W_gate", "W_up", "W_down"))
    idx = np.asarray(d["topk_idx"])
    w = np.asarray(d["topk_w"], np.float64)
    T, H = x.shape
    E, I, _ = Wg.shape
    k = idx.shape[1]
    y = np.zeros((T, H))
    dx = np.zeros((T, H))
    dtw = np.zeros((T, k))
    dWg, dWu, dWd = np.zeros_like(Wg), np.zeros_like(Wu), np.zeros_like(Wd)
    for e in range(E):
        rows = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        if not rows:
            continue
        n = len(rows)
        xe = np.array([x[t] for t, _ in rows])
        dye = np.array([dy[t] for t, _ in rows])
        we = np.array([w[t, j] for t, j in rows])
        # forward
        xq = quant_rows(xe) if qf else xe
        Wgq = quant_rows(Wg[e]) if qf else Wg[e]
        Wuq = quant_rows(Wu[e]) if qf else Wu[e]
        Wdq = quant_rows(Wd[e]) if qf else Wd[e]
        g = np.array([[float(np.dot(xq[r], Wgq[i])) for i in range(I)] for r in range(n)])
        u = np.array([[float(np.dot(xq[r], Wuq[i])) for i in range(I)] for r in range(n)])
        a = np.array([[g[r, i] * sig(g[r, i]) * u[r, i] for i in range(I)] for r in range(n)])
        a_in = quant_rows(bf16(a)) if qf else a
        for r, (t, j) in enumerate(rows):
            o = np.array([float(np.dot(a_in[r], Wdq[h])) for h in range(H)])
            y[t] += w[t, j] * o
        # backward (the stored h and a when the backward is MXFP8)
        if qb:
            g, u, a = bf16(g), bf16(u), bf16(a)
        dyq = quant_rows(dye) if qb else dye
        WdT = quant_cols(Wd[e]) if qb else Wd[e]          # blocks along H
        gp = np.array([[float(np.dot(dyq[r], WdT[:, i])) for i in range(I)] for r in range(n)])
        dg = np.zeros((n, I))
        du = np.zeros((n, I))
        for r in range(n):
            for i in range(I):
                s = sig(g[r, i])
                da = we[r] * gp[r, i]
                dg[r, i] = da * u[r, i] * s * (1.0 + g[r, i] * (1.0 - s))
                du[r, i] = da * g[r, i] * s
        if qb:
            dg, du = bf16(dg), bf16(du)
        dgq = quant_rows(dg) if qb else dg
        duq = quant_rows(du) if qb else du
        WgI = quant_cols(Wg[e]) if qb else Wg[e]          # blocks along I
        WuI = quant_cols(Wu[e]) if qb else Wu[e]
        for r, (t, j) in enumerate(rows):
            dx[t] += np.array([float(np.dot(dgq[r], WgI[:, h]) + np.dot(duq[r], WuI[:, h]))
                               for h in range(H)])
            dtw[t, j] = float(np.dot(a[r], gp[r]))
        # weight gradients: token-axis blocks from the expert's first row
        aw = np.array([we[r] * a[r] for r in range(n)])
        if qb:
            aw = bf16(aw)
        tq = quant_cols if qb else (lambda M: M)
        dgt, dut, xt, dyt, awt = tq(dg), tq(du), tq(xe), tq(dye), tq(aw)
        dWg[e] = np.array([[float(np.dot(dgt[:, i], xt[:, h])) for h in range(H)]
                           for i in range(I)])
        dWu[e] = np.array([[float(np.dot(dut[:, i], xt[:, h])) for h in range(H)]
                           for i in range(I)])
        dWd[e] = np.array([[float(np.dot(dyt[:, h], awt[:, i])) for i in range(I)]
                           for h in range(H)])
    return dict(y=y, dx=dx, dtopk_w=dtw, dW_gate=dWg, dW_up=dWu, dW_down=dWd)


def tiny_inputs(seed=0, T=6, H=64, I=64, E=3, k=2):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    # spread magnitudes over several binades so that block scales differ
    scale = np.exp2(rng.integers(-3, 4, size=(1, H)))
    return dict(
        x=rng.standard_normal((T, H)) * scale, dy=rng.standard_normal((T, H)),
        W_gate=rng.standard_normal((E, I, H)) * 0.1, W_up=rng.standard_normal((E, I, H)) * 0.1,
        W_down=rng.standard_normal((E, H, I)) * 0.1, topk_idx=idx,
        topk_w=rng.uniform(0.1, 1.0, size=(T, k)))


def oracle_all(d, prec):
    f = om.forward(d["x"], d["topk_idx"], d["topk_w"], d["W_gate"], d["W_up"], d["W_down"],
                   prec)
    b = om.backward(d["dy"], d["x"], d["topk_idx"], d["topk_w"], d["W_gate"], d["W_up"],
                    d["W_down"], prec, fwd=f)
    b["y"] = f["y"]
    return b


KEYS = ("y", "dx", "dtopk_w", "dW_gate", "dW_up", "dW_down")


def assert_match(d, prec):
    ref = brute(d, prec)
    got = oracle_all(d, prec)
    for key in KEYS:
        den = np.abs(ref[key]).max()
        err = np.abs(got[key] - ref[key]).max() / den
        assert err <= 1e-12, (prec, key, err)


# ------------------------------------------------------------------ tests
def test_bf16_round_matches_library():
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(20000) * np.exp2(rng.integers(-30, 30, 20000)),
                        rng.standard_normal(2000) * 2.0 ** -128])        # subnormal range
    v32 = torch.from_numpy(v).to(torch.float32)
    v = v32.double().numpy()                       # fp32 inputs: one rounding to bf16
    lib = v32.to(torch.bfloat16).double().numpy()
    assert np.array_equal(mx.bf16_round(v), lib)
    # exact ties (9 significant bits, last one set) go to the even neighbour
    t = (np.arange(256, 512) * 2 + 1) * 2.0 ** -9
    lib_t = torch.from_numpy(t).to(torch.float32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(mx.bf16_round(t), lib_t)
    assert np.array_equal(bf16(v[:3000]), lib[:3000])     # the brute force's own rounding


def test_e4m3_nearest_matches_library():
    rng = np.random.default_rng(6)
    v = rng.uniform(-448, 448, 5000)
    v = torch.from_numpy(v).to(torch.float32).double().numpy()
    lib = torch.from_numpy(v).to(torch.float32).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.array([e4m3_nearest(a) for a in v]), lib)


@pytest.mark.parametrize("prec", ["mxfp8", "fp8_bwd", "bf16"])
@pytest.mark.parametrize("seed", [0, 1])
def test_layer_matches_brute_force(prec, seed):
    assert_match(tiny_inputs(seed), prec)


def test_partial_token_blocks():
    """An expert with 37 rows: one full 32-row block and a zero-padded one."""
    d = tiny_inputs(2, T=40, H=32, I=32, E=2, k=1)
    d["topk_idx"][:37, 0] = 0
    d["topk_idx"][37:, 0] = 1
    assert_match(d, "mxfp8")


def _plant(monkeypatch, fn):
    monkeypatch.setattr(om, "expert_backward", fn)


def test_planted_transposed_block_axis_is_caught(monkeypatch):
    orig = om._q

    def wrong(v, axis, on):                       # W_down's backward blocks along I
        if on and np.ndim(v) == 2 and v.shape == (64, 64) and axis == 0:
            return orig(v, 1, on)
        return orig(v, axis, on)
    monkeypatch.setattr(om, "_q", wrong)
    with pytest.raises(AssertionError):
        assert_match(tiny_inputs(0), "mxfp8")


def test_planted_dropped_quantisation_is_caught(monkeypatch):
    orig = om.expert_forward

    def no_a_quant(xe, Wg_e, Wu_e, Wd_e, prec="bf16"):
        g, u, a, o = orig(xe, Wg_e, Wu_e, Wd_e, "bf16")
        if prec == "mxfp8":
            xq = mx.mx_qdq(xe, 1)
            g = xq @ mx.mx_qdq(Wg_e, 1).T
            u = xq @ mx.mx_qdq(Wu_e, 1).T
            a = om.swiglu(g, u)
            o = a @ mx.mx_qdq(Wd_e, 1).T              # a not quantised
        return g, u, a, o
    monkeypatch.setattr(om, "expert_forward", no_a_quant)
    with pytest.raises(AssertionError):
        assert_match(tiny_inputs(0), "mxfp8")


def test_planted_unrounded_stored_tensor_is_caught(monkeypatch):
    monkeypatch.setattr(om, "_stored", lambda v, on: v)
    with pytest.raises(AssertionError):
        assert_match(tiny_inputs(1), "fp8_bwd")
