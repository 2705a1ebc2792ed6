"""The blockwise FP8 oracle (oracle/fp8block.py and the fp8_block layer mode) against
independent facts: the scale rule on worked values, no element ever saturating,
exactness on blocks already on the grid, independence of the 128 x 128 weight blocks,
axis symmetry, and a brute-force scalar restatement of the layer on tiny inputs
(blocks walked one at a time; e4m3 by nearest search over torch's float8 code table).
Planted mistakes must fail."""
import math

import numpy as np
import pytest

import oracle.moe as om
from oracle import fp8block as fb
from tests.test_oracle_mx_layer import bf16, e4m3_nearest, oracle_all, sig


def test_scale_rule_worked_values():
    amax = np.array([448.0, 449.0, 448.0 * 2 ** 5, 1.75 * 2 ** 8 * 1.0078125, 1.0, 224.0,
                     224.5, 0.0, 2.0 ** -140, 3.0e38])
    # ceil(log2(amax / 448)): 448 -> 0; just above -> 1; exact power -> 5; 1.0 -> -8;
    # 224 -> -1; above 224 -> 0; zero block -> -127; tiny -> clipped; 3e38 -> 120
    # (448 * 2^119 = 2.98e38 < 3e38)
    assert fb.ue8m0_ceil_exponent(amax).tolist() == [0, 1, 5, 1, -8, -1, 0, -127, -127, 120]


def test_no_element_saturates_and_grid_blocks_are_exact():
    rng = np.random.default_rng(0)
    v = rng.standard_normal((16, 512)) * np.exp2(rng.integers(-20, 20, size=(16, 1)))
    q = fb.qdq_1d(v, axis=1)
    blocks = v.reshape(16, 4, 128)
    bm = np.abs(blocks).max(axis=2)
    X = np.exp2(fb.ue8m0_ceil_exponent(bm))[..., None]
    assert np.all(bm / X[..., 0] <= 448.0) and np.all(bm / X[..., 0] > 224.0)  # tightest scale
    # error within half an e4m3 step of each element (3 mantissa bits) or the subnormal step
    Xf = np.broadcast_to(X, blocks.shape).reshape(16, 512)
    assert np.all(np.abs(q - v) <= np.maximum(np.abs(v) * 2.0 ** -4, Xf * 2.0 ** -10) * (1 + 1e-12))
    # values already on the grid with block maximum in (224, 448] * 2^s are fixed points
    codes = np.array(sorted(set(abs(e4m3_nearest(x)) for x in np.linspace(0, 448, 4000))))
    g = rng.choice(codes, size=(8, 128)) * np.sign(rng.standard_normal((8, 128)))
    g[:, 0] = 256.0
    g *= np.exp2(rng.integers(-10, 10, size=(8, 1)))
    assert np.array_equal(fb.qdq_1d(g, axis=1), g)


def test_weight_blocks_are_independent_and_axis_symmetric():
    rng = np.random.default_rng(1)
    scales = np.exp2(rng.integers(-8, 8, size=(2, 3)).astype(np.float64))
    W = rng.standard_normal((256, 384)) * np.kron(scales, np.ones((128, 128)))
    q = fb.qdq_2d(W)
    for i in range(2):
        for j in range(3):
            t = W[128 * i:128 * (i + 1), 128 * j:128 * (j + 1)]
            X = 2.0 ** fb.ue8m0_ceil_exponent(np.abs(t).max())
            want = np.array([[e4m3_nearest(x / X) * X for x in row] for row in t])
            assert np.array_equal(q[128 * i:128 * (i + 1), 128 * j:128 * (j + 1)], want)
    assert np.array_equal(fb.qdq_2d(W.T), q.T)
    v = rng.standard_normal((300, 64))
    assert np.array_equal(fb.qdq_1d(v, 0), fb.qdq_1d(v.T, 1).T)


# ------------------------------------------------------------------ brute-force layer
def qblock(vals):
    amax = max(abs(x) for x in vals)
    if amax == 0.0:
        return [0.0] * len(vals)
    e = max(-127, min(127, math.ceil(math.log2(amax / 448.0))))
    X = 2.0 ** e
    return [e4m3_nearest(x / X) * X for x in vals]


def q_rows(M, B=128):
    out = []
    for r in M:
        row = []
        for b in range(0, len(r), B):
            row += qblock(list(r[b:b + B]))
        out.append(row)
    return np.array(out)


def q_cols(M, B=128):
    return q_rows(np.asarray(M).T, B).T


def q_w(W, B=128):
    W = np.asarray(W)
    out = np.zeros_like(W)
    for i in range(0, W.shape[0], B):
        for j in range(0, W.shape[1], B):
            t = W[i:i + B, j:j + B]
            flat = qblock(list(t.reshape(-1)))
            out[i:i + B, j:j + B] = np.array(flat).reshape(t.shape)
    return out


def brute_block(d):
    x, dy = np.asarray(d["x"], np.float64), np.asarray(d["dy"], np.float64)
    Wg, Wu, Wd = (np.asarray(d[k], np.float64) for k in ("W_gate", "W_up", "W_down"))
    idx, w = np.asarray(d["topk_idx"]), np.asarray(d["topk_w"], np.float64)
    T, H = x.shape
    E, I, _ = Wg.shape
    k = idx.shape[1]
    y, dx, dtw = np.zeros((T, H)), np.zeros((T, H)), np.zeros((T, k))
    dWg, dWu, dWd = np.zeros_like(Wg), np.zeros_like(Wu), np.zeros_like(Wd)
    for e in range(E):
        rows = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        if not rows:
            continue
        n = len(rows)
        xe = np.array([x[t] for t, _ in rows])
        dye = np.array([dy[t] for t, _ in rows])
        we = np.array([w[t, j] for t, j in rows])
        Wgq, Wuq, Wdq = q_w(Wg[e]), q_w(Wu[e]), q_w(Wd[e])   # the same for every GEMM
        xq = q_rows(xe)
        g = np.array([[float(np.dot(xq[r], Wgq[i])) for i in range(I)] for r in range(n)])
        u = np.array([[float(np.dot(xq[r], Wuq[i])) for i in range(I)] for r in range(n)])
        a = np.array([[g[r, i] * sig(g[r, i]) * u[r, i] for i in range(I)] for r in range(n)])
        aq = q_rows(bf16(a))
        for r, (t, j) in enumerate(rows):
            y[t] += w[t, j] * np.array([float(np.dot(aq[r], Wdq[h])) for h in range(H)])
        g, u, a = bf16(g), bf16(u), bf16(a)
        dyq = q_rows(dye)
        gp = np.array([[float(np.dot(dyq[r], Wdq[:, i])) for i in range(I)] for r in range(n)])
        dg, du = np.zeros((n, I)), np.zeros((n, I))
        for r in range(n):
            for i in range(I):
                s = sig(g[r, i])
                da = we[r] * gp[r, i]
                dg[r, i] = da * u[r, i] * s * (1.0 + g[r, i] * (1.0 - s))
                du[r, i] = da * g[r, i] * s
        dg, du = bf16(dg), bf16(du)
        dgq, duq = q_rows(dg), q_rows(du)
        for r, (t, j) in enumerate(rows):
            dx[t] += np.array([float(np.dot(dgq[r], Wgq[:, h]) + np.dot(duq[r], Wuq[:, h]))
                               for h in range(H)])
            dtw[t, j] = float(np.dot(a[r], gp[r]))
        aw = bf16(np.array([we[r] * a[r] for r in range(n)]))
        dgt, dut, xt, dyt, awt = q_cols(dg), q_cols(du), q_cols(xe), q_cols(dye), q_cols(aw)
        dWg[e] = np.array([[float(np.dot(dgt[:, i], xt[:, h])) for h in range(H)] for i in range(I)])
        dWu[e] = np.array([[float(np.dot(dut[:, i], xt[:, h])) for h in range(H)] for i in range(I)])
        dWd[e] = np.array([[float(np.dot(dyt[:, h], awt[:, i])) for i in range(I)] for h in range(H)])
    return dict(y=y, dx=dx, dtopk_w=dtw, dW_gate=dWg, dW_up=dWu, dW_down=dWd)


def tiny(seed=0, T=10, H=256, I=128, E=2, k=2):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    return dict(x=rng.standard_normal((T, H)) * np.exp2(rng.integers(-3, 4, size=(1, H))),
                dy=rng.standard_normal((T, H)), W_gate=rng.standard_normal((E, I, H)) * 0.1,
                W_up=rng.standard_normal((E, I, H)) * 0.1, W_down=rng.standard_normal((E, H, I)) * 0.1,
                topk_idx=idx, topk_w=rng.uniform(0.1, 1.0, size=(T, k)))


def assert_match(d):
    ref, got = brute_block(d), oracle_all(d, "fp8_block")
    for key in ref:
        err = np.abs(got[key] - ref[key]).max() / np.abs(ref[key]).max()
        assert err <= 1e-12, (key, err)


def test_layer_matches_brute_force():
    assert_match(tiny(0))


def test_planted_32_blocks_are_caught(monkeypatch):
    orig = fb.qdq_1d
    monkeypatch.setattr(om, "block_qdq_1d", lambda v, axis: orig(v, axis, 32))
    with pytest.raises(AssertionError):
        assert_match(tiny(1))


def test_planted_floor_scale_rule_is_caught(monkeypatch):
    def floor_rule(amax):
        amax = np.asarray(amax, dtype=np.float64)
        with np.errstate(divide="ignore"):
            e = np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8
        return np.clip(np.where(amax > 0, e, -127), -127, 127).astype(np.int64)
    monkeypatch.setattr(fb, "ue8m0_ceil_exponent", floor_rule)
    with pytest.raises(AssertionError):
        test_scale_rule_worked_values()
    with pytest.raises(AssertionError):
        assert_match(tiny(2))
