"""Pins of the oracle's update tail (the page's `_rail_equalizer` and
`_sign_aligned_decay_update` in anvil.py) against closed forms and invariants."""
import numpy as np
import pytest

import oracle

U32 = 2.0 ** -24


def f64(b):
    return oracle.bf16_to_f32(b).astype(np.float64)


def lanes(x, rows_ge_cols):
    """Mean square per lane: lanes along the longer dimension (rows when rows >= cols)."""
    return (x ** 2).mean(axis=2) if rows_ge_cols else (x ** 2).mean(axis=1)


def graded(shape, seed):
    """bf16 updates whose lanes have very different energies."""
    g, m, n = shape
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape)
    if m >= n:
        x *= np.geomspace(0.01, 10, m)[None, :, None]
    else:
        x *= np.geomspace(0.01, 10, n)[None, None, :]
    return oracle.f32_to_bf16(x.astype(np.float32))


@pytest.mark.parametrize("shape", [(2, 48, 16), (2, 16, 48), (1, 32, 32), (3, 7, 5)])
def test_equalizer_from_zero_state_equalises_lanes_and_keeps_the_norm(shape):
    """From zero lane energy: gain_l = 1/sqrt((1-b2) P_l), every lane's post power is the
    same, so each lane leaves with the mean lane power and ||v||_F is preserved."""
    g, m, n = shape
    v = graded(shape, sum(shape))
    le0 = np.zeros((g, m if m >= n else n), np.float32)
    veq, le = oracle.rail_equalizer(v, le0, 0.95)
    P = lanes(f64(v), m >= n)
    Q = lanes(f64(veq), m >= n)
    for i in range(g):
        assert np.allclose(Q[i], P[i].mean(), rtol=2e-2)
        assert abs(np.linalg.norm(f64(veq[i])) / np.linalg.norm(f64(v[i])) - 1) < 1e-2
    np.testing.assert_allclose(le, 0.05 * P, rtol=1e-5)


@pytest.mark.parametrize("shape,b2", [((2, 48, 16), 0.95), ((2, 16, 48), 0.9), ((1, 40, 40), 0.99)])
def test_equalizer_output_bits_from_the_closed_form_scale(shape, b2):
    """Bit for bit where the result is decided: from zero lane energy the lane scale is
    s_l = gain_l * ||v|| / post_norm with gain_l = 1/sqrt((1-b2) P_l), evaluated here in fp64;
    the page casts it to bf16 (torch's conversion here) and the output element is
    bf16(v * bf16(s_l)), a product of two bf16 values, exact before its one rounding.  Lanes
    whose s_l lies within 2^-14 (relative) of a bf16 rounding boundary, where fp32 evaluation
    order may decide, are skipped."""
    import torch
    g, m, n = shape
    v = graded(shape, 7 * m + n)
    rows_lanes = m >= n
    le0 = np.zeros((g, m if rows_lanes else n), np.float32)
    veq, _ = oracle.rail_equalizer(v, le0, b2)
    x = f64(v)
    P = lanes(x, rows_lanes)                                 # [g, nl]
    L = n if rows_lanes else m                               # lane length
    le = (1.0 - np.float64(np.float32(b2))) * P
    gain = 1.0 / np.sqrt(le)
    post = np.sqrt((P * L * gain ** 2).sum(axis=1, keepdims=True))
    pre = np.sqrt((P * L).sum(axis=1, keepdims=True))
    s = gain * (pre / post)
    s_bf = torch.from_numpy(s.astype(np.float32)).to(torch.bfloat16).double().numpy()
    # distance of s to the nearest bf16 rounding boundary (midpoint), relative
    e = np.floor(np.log2(s))
    ulp = 2.0 ** (e - 7)
    frac = (s / ulp) % 1.0
    robust = np.abs(frac - 0.5) * ulp > 2.0 ** -14 * s
    assert robust.mean() > 0.9
    prod = x * (s_bf[:, :, None] if rows_lanes else s_bf[:, None, :])
    want = torch.from_numpy(prod.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mask = np.broadcast_to(robust[:, :, None] if rows_lanes else robust[:, None, :], veq.shape)
    np.testing.assert_array_equal(veq[mask], want[mask])


def test_lane_energy_is_an_ema_over_steps():
    """The same update k times from zero: lane_energy_k = (1 - b2^k) P."""
    shape = (2, 24, 40)
    v = graded(shape, 3)
    le = np.zeros((2, 40), np.float32)
    P = lanes(f64(v), False)
    b2 = np.float32(0.9)
    for k in range(1, 8):
        _, le = oracle.rail_equalizer(v, le, 0.9)
        np.testing.assert_allclose(le, (1 - np.float64(b2) ** k) * P, rtol=1e-5)


def test_equalizer_zero_lane_stays_zero_and_finite():
    v = graded((1, 16, 8), 4)
    v[0, 3, :] = 0
    veq, le = oracle.rail_equalizer(v, np.zeros((1, 16), np.float32), 0.95)
    assert np.isfinite(f64(veq)).all() and not veq[0, 3].any()


def test_equalizer_with_equal_lanes_and_steady_state_is_identity_scale():
    """Lanes already equal, lane_energy at its fixed point: the scale is 1."""
    v = oracle.f32_to_bf16(np.ones((1, 12, 6), np.float32) * 0.5)
    le = np.full((1, 12), 0.25, np.float32)
    veq, le2 = oracle.rail_equalizer(v, le, 0.95)
    np.testing.assert_array_equal(veq, v)
    np.testing.assert_array_equal(le2, le)


def _master(p, mt):
    return ((p.astype(np.uint32) << 16) | mt.astype(np.uint32)).view(np.float32).astype(np.float64)


def test_decay_matches_fp64_and_gates_on_the_slow_rail_sign():
    rng = np.random.default_rng(6)
    shape = (3, 20, 30)
    w = (rng.standard_normal(shape) * 0.05).astype(np.float32)
    bits = w.view(np.uint32)
    p, mt = (bits >> 16).astype(np.uint16), (bits & 0xFFFF).astype(np.uint16)
    u = oracle.f32_to_bf16(rng.standard_normal(shape).astype(np.float32))
    gate = rng.standard_normal(shape).astype(np.float32) * 0.01
    lr = np.array([0.02, 0.0, 0.05], np.float32)
    wd = np.float32(0.1)
    p2, mt2 = oracle.sign_aligned_decay(p, mt, u, gate, float(wd), lr)
    W = _master(p, mt)
    aligned = (gate.astype(np.float64) * W) >= 0
    want = W - W * aligned * float(wd) * lr.astype(np.float64)[:, None, None] \
        - f64(u) * lr.astype(np.float64)[:, None, None]
    got = _master(p2, mt2)
    scale = np.abs(W) + np.abs(f64(u)) * np.abs(lr.astype(np.float64))[:, None, None]
    assert np.all(np.abs(got - want) <= 4 * U32 * scale + 1e-45)
    # lr = 0: the master weight is untouched, bit for bit
    np.testing.assert_array_equal(p2[1], p[1])
    np.testing.assert_array_equal(mt2[1], mt[1])
    # decay applies only where gate and weight agree in sign: flip the gate, the decay
    # term moves to the complementary elements
    p3, mt3 = oracle.sign_aligned_decay(p, mt, np.zeros_like(u), -gate, float(wd), lr)
    d3 = _master(p3, mt3) - W
    hit = d3[0] != 0
    assert np.array_equal(hit, ~aligned[0] & (W[0] != 0))


def test_decay_bit_split_round_trips():
    rng = np.random.default_rng(7)
    w = rng.standard_normal((1, 64)).astype(np.float32)
    bits = w.view(np.uint32)
    p, mt = (bits >> 16).astype(np.uint16), (bits & 0xFFFF).astype(np.uint16)
    p2, mt2 = oracle.sign_aligned_decay(p, mt, np.zeros((1, 64), np.uint16),
                                        np.ones((1, 64), np.float32), 0.0, np.zeros(1, np.float32))
    np.testing.assert_array_equal(p2, p)
    np.testing.assert_array_equal(mt2, mt)


# --------------------------------------------------------------------------- Adam

def test_adam_first_step_closed_form():
    """From zero moments: m = (1-b1) g, v = (1-b2) g^2, and with the bias-corrected step
    size lr sqrt(1-b2)/(1-b1) the update is lr g / (|g| + eps / sqrt(1-b2)) (no decay)."""
    rng = np.random.default_rng(8)
    g = (rng.standard_normal(4096) * 0.01).astype(np.float32)
    p = (rng.standard_normal(4096) * 0.1).astype(np.float32)
    b1, b2, eps, lr = 0.9, 0.95, 1e-8, 0.01
    step = lr * np.sqrt(1 - b2) / (1 - b1)
    p2, m, v = oracle.adam_step(p, g, np.zeros_like(g), np.zeros_like(g), b1, b2, eps, step, 0.0)
    G = g.astype(np.float64)
    np.testing.assert_allclose(m, (1 - np.float32(b1)) * G, rtol=1e-6)
    np.testing.assert_allclose(v, (1 - np.float64(np.float32(b2))) * G * G, rtol=1e-6)
    want = p - lr * G / (np.abs(G) + eps / np.sqrt(1 - b2))
    # a handful of fp32 roundings of values of size |p| + lr
    assert np.all(np.abs(p2 - want) <= 8 * U32 * (np.abs(p) + lr) + 1e-6 * lr)


def test_adam_cautious_decay_only_where_update_and_weight_agree():
    rng = np.random.default_rng(9)
    g = (rng.standard_normal(2048) * 0.01).astype(np.float32)
    p = (rng.standard_normal(2048) * 0.1).astype(np.float32)
    m0 = (rng.standard_normal(2048) * 0.01).astype(np.float32)
    v0 = (np.abs(rng.standard_normal(2048)) * 1e-4).astype(np.float32)
    a = oracle.adam_step(p, g, m0, v0, 0.9, 0.95, 1e-8, 0.01, 0.0)[0]
    b = oracle.adam_step(p, g, m0, v0, 0.9, 0.95, 1e-8, 0.01, 0.05)[0]
    upd = p.astype(np.float64) - a
    decayed = b != a
    assert np.array_equal(decayed, (upd * p > 0) & (p != 0))
    scale = np.abs(p) + np.abs(upd)
    assert np.all(np.abs((a - b) - 0.05 * p)[decayed] <= 8 * U32 * scale[decayed])
