"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle (oracle/anvil_oracle.c) against what the page
"modded-nanogpt track_1_short/optim/anvil.py" (function anvil_cascade and the
constants above it) and plain mathematics fix:

* bf16 rounding against torch's own fp32->bf16 conversion (a library routine);
* the momentum recurrences against their closed forms over k steps (fp64);
* the unrounded iteration against the SVD closed form U F(S/d) V^T;
* every stored stage of the bf16 path against an fp64 evaluation of that
  stage from the previous stored stage, within the fp32 / bf16 error bounds;
* bitwise invariants: transposition, zero padding, power-of-two scaling,
  zero input, batching.

Chosen so that a dropped term, a wrong sign or index, or a transposed operand
anywhere in the oracle fails at least one of them.
"""
import numpy as np
import pytest
import torch

import oracle
from polynomial_matrix_whitening_gb300 import workloads as W

U32 = 2.0 ** -24     # fp32 unit roundoff
UBF = 2.0 ** -8      # bf16 unit roundoff (8 significant bits)


def f64(bits):
    return oracle.bf16_to_f32(bits).astype(np.float64)


def composite(sig, maps):
    for a, b, c in maps:
        sig = a * sig + b * sig ** 3 + c * sig ** 5
    return sig


# --------------------------------------------------------------------------- constants

def test_constants_match_page(constants):
    maps, consts = constants
    assert len(maps) == 6
    np.testing.assert_array_equal(np.array(oracle.ANVIL_MAPS), np.array(maps))
    assert oracle.FROBENIUS_MARGIN == consts["FROBENIUS_MARGIN"]
    assert oracle.FROBENIUS_EPS == consts["FROBENIUS_EPS"]
    assert W.RAIL_FAST_BETA == consts["RAIL_FAST_BETA"]
    assert W.RAIL_SLOW_BETA == consts["RAIL_SLOW_BETA"]
    assert W.RAIL_FAST_WEIGHT == consts["RAIL_FAST_WEIGHT"]


def test_composite_map_properties(constants):
    """The six maps drive every singular value in (0, 1/margin] to ~1 (page: 'drives every
    singular value to ~1'; the margin 'puts every singular value safely below 1')."""
    maps, consts = constants
    slope = np.prod([a for a, _, _ in maps])
    assert abs(slope - 643.13) < 0.01
    sig = np.geomspace(0.01, 1.0 / consts["FROBENIUS_MARGIN"], 20001)
    F = composite(sig, maps)
    assert F.min() > 0.9995 and F.max() < 1.0005
    # F crosses 0.999 near sigma = 3.26e-3
    lo = np.geomspace(1e-4, 0.01, 4001)
    first = lo[np.argmax(composite(lo, maps) >= 0.999)]
    assert 3.0e-3 < first < 3.5e-3


# --------------------------------------------------------------------------- bf16 rounding

def _torch_bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    mag = (10.0 ** rng.integers(-30, 30, 200000)).astype(np.float32)
    vals = [rng.standard_normal(200000).astype(np.float32) * mag]
    # exact ties, both parities of the kept bit, around several exponents
    base = rng.integers(0, 2 ** 31, 50000, dtype=np.uint64).astype(np.uint32)
    ties = (base & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    near = [ties, ties - np.uint32(1), ties + np.uint32(1)]
    for t in near:
        vals.append(t.view(np.float32))
    special = np.array([0.0, -0.0, np.inf, -np.inf, 3.4028235e38, -3.4028235e38,
                        1e-45, -1e-45, 1.1754944e-38, 1.0, -1.0, 65504.0], np.float32)
    vals.append(special)
    x = np.concatenate([v.astype(np.float32, copy=False) for v in vals])
    x = x[~np.isnan(x)]
    ours = oracle.f32_to_bf16(x)
    ref = _torch_bf16_bits(x)
    np.testing.assert_array_equal(ours, ref)
    nan = np.array([np.nan, -np.nan], np.float32)
    assert np.isnan(oracle.bf16_to_f32(oracle.f32_to_bf16(nan))).all()


# --------------------------------------------------------------------------- momentum

def _f32(x):
    return float(np.float32(x))


@pytest.mark.parametrize("w", [1.0, 0.4385])
def test_momentum_closed_form_constant_grad(w):
    """Zero rails, constant g: v_f,k = (1 - bf^k) g, v_s,k = (1 - bs^k) g,
    y_k = (1 - mu) g + mu (w v_f,k + (1 - w) v_s,k)."""
    mu, bf, bs = 0.95, 0.85, 0.98
    g = W.gaussian([1], (64, 48), 0.02)
    vel = np.zeros((2,) + g.shape, np.float32)
    bf64, bs64, mu64, w64 = _f32(bf), _f32(bs), _f32(mu), _f32(w)
    for k in range(1, 11):
        X, y, vel = oracle.momentum(g, vel, mu, bf, w, bs)
        vf = (1 - bf64 ** k) * g.astype(np.float64)
        vs = (1 - bs64 ** k) * g.astype(np.float64)
        yk = (1 - mu64) * g + mu64 * (w64 * vf + (1 - w64) * vs)
        for got, want in ((vel[0], vf), (vel[1], vs), (y, yk)):
            assert np.linalg.norm(got - want) <= 1e-6 * np.linalg.norm(want)
            assert np.max(np.abs(got - want)) <= 2e-6 * np.max(np.abs(want))
        np.testing.assert_array_equal(X, oracle.f32_to_bf16(y))


def test_momentum_closed_form_general():
    """Fresh g per step, swept fast beta, non-zero initial rails:
    v_k = beta_k v_{k-1} + (1 - beta_k) g_k evaluated in fp64."""
    mu, bs, w = 0.95, 0.98, 0.4385
    shape = (3, 40, 24)
    vel = W.gaussian([2], (2,) + shape, 0.01)
    vf = vel[0].astype(np.float64)
    vs = vel[1].astype(np.float64)
    for k in range(10):
        bf = 0.6 + 0.25 * k / 9
        g = W.gaussian([3, k], shape, 0.02)
        X, y, vel = oracle.momentum(g, vel, mu, bf, w, bs)
        b1 = 1 - _f32(1 - _f32(bf))  # the fp32 lerp weight is 1 - beta rounded to fp32
        b2 = 1 - _f32(1 - _f32(bs))
        vf = b1 * vf + (1 - b1) * g
        vs = b2 * vs + (1 - b2) * g
        yk = (1 - _f32(mu)) * g + _f32(mu) * (_f32(w) * vf + (1 - _f32(w)) * vs)
        for got, want in ((vel[0], vf), (vel[1], vs), (y, yk)):
            assert np.linalg.norm(got - want) <= 1e-6 * np.linalg.norm(want)


def test_momentum_pre_engage_reads_fast_rail_only():
    g = W.gaussian([4], (16, 16), 0.02)
    vel = W.gaussian([5], (2, 16, 16), 0.01)
    _, y, v = oracle.momentum(g, vel, 0.95, 0.85, 1.0, 0.98)
    want = g.astype(np.float64) + 0.95 * (v[0].astype(np.float64) - g)
    assert np.max(np.abs(y - want)) < 1e-7


# --------------------------------------------------------------------------- SVD closed form

def closed_form(X, maps, margin, eps):
    """U F(S/d) V^T with d = margin * ||X||_F + eps (numpy SVD in fp64)."""
    U, S, Vt = np.linalg.svd(X, full_matrices=False)
    d = np.sqrt(np.sum(S ** 2)) * margin + eps
    return (U * composite(S / d, maps)) @ Vt


@pytest.mark.parametrize("shape", [(4, 3), (3, 4), (3, 3), (16, 8), (8, 16), (40, 17),
                                   (17, 40), (1, 5), (5, 1), (64, 64)])
def test_f64_iteration_equals_svd_closed_form(shape, constants):
    maps, consts = constants
    rng = np.random.default_rng(sum(shape))
    X = rng.standard_normal(shape)
    got = oracle.cascade_f64(X, maps, consts["FROBENIUS_MARGIN"], consts["FROBENIUS_EPS"])
    want = closed_form(X, maps, consts["FROBENIUS_MARGIN"], consts["FROBENIUS_EPS"])
    assert np.linalg.norm(got - want) <= 1e-11 * np.linalg.norm(want)


def test_f64_iteration_closed_form_other_maps():
    """Other map sets and margins (including a cubic map with c = 0) pin that a, b, c enter
    each step as a X + b X^3 + c X^5 and that margin and eps enter d as stated."""
    maps = [(1.5, -0.5, 0.0), (2.0, -1.5, 0.5), (1.0, 0.25, -0.125)]
    rng = np.random.default_rng(7)
    for shape in [(5, 9), (9, 5), (6, 6)]:
        X = rng.standard_normal(shape)
        got = oracle.cascade_f64(X, maps, 1.3, 0.01)
        want = closed_form(X, maps, 1.3, 0.01)
        assert np.linalg.norm(got - want) <= 1e-12 * np.linalg.norm(want)


@pytest.mark.parametrize("shape", [(64, 192), (192, 64), (96, 96)])
def test_bf16_oracle_near_closed_form_gaussian(shape):
    """Well-conditioned input: the bf16 pipeline lands within bf16 accuracy of U F(S/d) V^T
    (acceptance tolerance 3e-2 against the closed form; measured about 5e-3)."""
    g = W.gaussian([6, shape[0]], shape, 0.02)
    X = oracle.f32_to_bf16(g)
    out = f64(oracle.cascade(X))
    want = closed_form(f64(X), oracle.ANVIL_MAPS, oracle.FROBENIUS_MARGIN, oracle.FROBENIUS_EPS)
    err = np.linalg.norm(out - want) / np.linalg.norm(want)
    assert err < 1.5e-2
    # a non-square Gaussian has all sigma/d well above 3.3e-3: every output singular value ~1
    if shape[0] != shape[1]:
        s = np.linalg.svd(out, compute_uv=False)
        assert s.min() > 0.97 and s.max() < 1.03


# --------------------------------------------------------------------------- stage by stage

def _bound_round(exact, fp32_err):
    """|bf16(fp32 result) - exact| <= fp32 error + bf16 half-ulp of the result."""
    return fp32_err + UBF * (np.abs(exact) + fp32_err) + 1e-30


def _gram64(X, tall):
    return X.T @ X if tall else X @ X.T


@pytest.mark.parametrize("shape", [(24, 40), (40, 24), (32, 32), (7, 33)])
def test_stages_against_fp64(shape):
    """Each stored bf16 stage equals the fp64 value of the page's formula, evaluated from the
    oracle's previous stored stage, to within fp32 accumulation and one bf16 rounding."""
    rows, cols = shape
    tall = rows > cols
    g = W.gaussian([8, rows, cols], shape, 0.02)
    Xraw_bits = oracle.f32_to_bf16(g)
    out, t = oracle.cascade(Xraw_bits, trace=True)
    maps = [tuple(float(np.float32(v)) for v in m) for m in oracle.ANVIL_MAPS]
    Xraw = f64(Xraw_bits)
    K = rows if tall else cols
    # first Gram
    G = _gram64(Xraw, tall)
    absG = _gram64(np.abs(Xraw), tall)
    assert np.all(np.abs(f64(t["A0"]) - G) <= _bound_round(G, K * U32 * absG))
    # trace and d
    A0 = f64(t["A0"])
    s = A0.shape[0]
    tr = np.trace(A0)
    d_want = np.sqrt(tr) * 1.05 + 1e-6
    assert abs(float(t["d"][0]) - d_want) <= (s + 4) * U32 * d_want
    d = float(t["d"][0])
    # normalised X and A
    Xn = Xraw / d
    assert np.all(np.abs(f64(t["X"][0]) - Xn) <= _bound_round(Xn, 2 * U32 * np.abs(Xn)))
    An = A0 / (np.float32(d) * np.float32(d))
    assert np.all(np.abs(f64(t["A"][0]) - An) <= _bound_round(An, 3 * U32 * np.abs(An)))
    for k, (a, b, c) in enumerate(maps):
        X = f64(t["X"][k])
        if k > 0:
            G = _gram64(X, tall)
            absG = _gram64(np.abs(X), tall)
            assert np.all(np.abs(f64(t["A"][k]) - G) <= _bound_round(G, K * U32 * absG)), k
        A = f64(t["A"][k])
        Bx = b * A + c * (A @ A)
        err = U32 * (np.abs(b * A) + abs(c) * (s + 2) * (np.abs(A) @ np.abs(A)) + np.abs(Bx))
        assert np.all(np.abs(f64(t["B"][k]) - Bx) <= _bound_round(Bx, 2 * err)), k
        B = f64(t["B"][k])
        C = a * X + (X @ B if tall else B @ X)
        P = np.abs(X) @ np.abs(B) if tall else np.abs(B) @ np.abs(X)
        err = U32 * (np.abs(a * X) + (s + 2) * P + np.abs(C))
        assert np.all(np.abs(f64(t["X"][k + 1]) - C) <= _bound_round(C, 2 * err)), k
    np.testing.assert_array_equal(out, t["X"][-1])


def test_stage_check_catches_planted_mistakes():
    """The stage bounds above are tight enough to see a transposed operand or a dropped term:
    plant them in an fp64 restatement of one map and check the bound fails."""
    rng = np.random.default_rng(11)
    X = f64(oracle.f32_to_bf16(rng.standard_normal((24, 40)) * 0.05))
    B = f64(oracle.f32_to_bf16(rng.standard_normal((24, 24)) * 0.3))
    a = 3.9
    good = a * X + B @ X
    for bad in (a * X + B.T @ X, B @ X, a * X - B @ X):
        P = np.abs(B) @ np.abs(X)
        err = U32 * (np.abs(a * X) + 26 * P + np.abs(good))
        assert not np.all(np.abs(bad - good) <= _bound_round(good, 2 * err))


# --------------------------------------------------------------------------- invariants

@pytest.mark.parametrize("shape", [(24, 40), (40, 24), (7, 33), (130, 57)])
def test_transpose_symmetry_bitwise(shape):
    """oracle(X^T) = oracle(X)^T: the tall branch (X^T X, X @ B) is the wide branch
    (X X^T, B @ X) on the transpose, with identical sums."""
    X = oracle.f32_to_bf16(W.gaussian([9, *shape], shape, 0.02))
    a = oracle.cascade(X)
    b = oracle.cascade(np.ascontiguousarray(X.T))
    np.testing.assert_array_equal(a, b.T)


@pytest.mark.parametrize("shape,pad", [((24, 40), (6, 10)), ((40, 24), (9, 3)), ((32, 32), (0, 5))])
def test_zero_padding_invariance_bitwise(shape, pad):
    rows, cols = shape
    X = oracle.f32_to_bf16(W.gaussian([10, rows], shape, 0.02))
    P = np.zeros((rows + pad[0], cols + pad[1]), np.uint16)
    P[:rows, :cols] = X
    assert (P.shape[0] > P.shape[1]) == (rows > cols)
    a = oracle.cascade(X)
    b = oracle.cascade(P)
    np.testing.assert_array_equal(b[:rows, :cols], a)
    assert not b[rows:, :].any() and not b[:, cols:].any()


@pytest.mark.parametrize("nb,k", [(24, 4), (40, 16)])
def test_block_diagonal_copies_share_one_d(nb, k):
    """k copies of one block on the diagonal: the Gram, b A + c A A and a X + B X keep the
    off-diagonal blocks exactly zero, so each diagonal block goes through the method on
    its own, normalised by the whole matrix's d.  The whole trace is k times the block's,
    so (k a power of 4, sqrt exact in fp32) that d is the block's own with the margin
    multiplied by sqrt(k), up to the order in which the trace is summed."""
    X1 = oracle.f32_to_bf16(W.gaussian([13, nb, k], (nb, nb), 0.02))
    size = nb * k
    Xw = np.zeros((size, size), np.uint16)
    for b in range(k):
        Xw[b * nb:(b + 1) * nb, b * nb:(b + 1) * nb] = X1
    whole = oracle.cascade(Xw).reshape(k, nb, k, nb)
    margin = float(np.float32(np.sqrt(k)) * np.float32(oracle.FROBENIUS_MARGIN))
    want = f64(oracle.cascade(X1, margin=margin))
    for b in range(k):
        for c in range(k):
            if b != c:
                assert not f64(whole[b, :, c, :]).any()
        got = f64(whole[b, :, b, :])
        assert np.linalg.norm(got - want) <= 1e-3 * np.linalg.norm(want)


@pytest.mark.parametrize("k", [-3, 2, 5])
def test_power_of_two_scaling_bitwise(k):
    """With eps = 0, grad * 2^k leaves the output unchanged bit for bit."""
    X = oracle.f32_to_bf16(W.gaussian([12], (24, 40), 0.02))
    Xs = oracle.f32_to_bf16(oracle.bf16_to_f32(X) * np.float32(2.0 ** k))
    a = oracle.cascade(X, eps=0.0)
    b = oracle.cascade(Xs, eps=0.0)
    np.testing.assert_array_equal(a, b)


def test_zero_input_gives_zero_output():
    X = np.zeros((16, 40), np.uint16)
    out = oracle.cascade(X)
    assert not out.any()
    g = np.zeros((2, 40, 16), np.float32)
    out, vel = oracle.bank_step(g, np.zeros((2,) + g.shape, np.float32), 0.95, 0.85, 1.0, 0.98)
    assert not out.any() and not vel.any()


def test_bank_step_is_momentum_then_cascade_and_batch_invariant():
    grad, vel = W.random_case(1, 3, 24, 40)
    out, v = oracle.bank_step(grad, vel, 0.95, 0.7, 0.4385, 0.98)
    X, _, v2 = oracle.momentum(grad, vel, 0.95, 0.7, 0.4385, 0.98)
    np.testing.assert_array_equal(v, v2)
    for i in range(3):
        np.testing.assert_array_equal(out[i], oracle.cascade(X[i]))
        o1, v1 = oracle.bank_step(grad[i:i + 1], vel[:, i:i + 1], 0.95, 0.7, 0.4385, 0.98)
        np.testing.assert_array_equal(o1[0], out[i])
        np.testing.assert_array_equal(v1[:, 0], v[:, i])


def test_velocity_save_reload():
    """k steps, save the rails, reload, k more == 2k steps (the state is the rails only)."""
    shape = (2, 24, 40)
    vel = np.zeros((2,) + shape, np.float32)
    outs = []
    for s in range(4):
        g = W.gaussian([13, s], shape, 0.02)
        o, vel = oracle.bank_step(g, vel, 0.95, 0.85, 0.4385, 0.98)
        outs.append(o)
        if s == 1:
            saved = vel.copy()
    vel2 = saved
    for s in range(2, 4):
        g = W.gaussian([13, s], shape, 0.02)
        o, vel2 = oracle.bank_step(g, vel2, 0.95, 0.85, 0.4385, 0.98)
        np.testing.assert_array_equal(o, outs[s])
    np.testing.assert_array_equal(vel2, vel)


def test_split_epilogue_differs_only_by_rounding():
    """The page's two-kernel form for banks over 1024 rows rounds X @ B to bf16 before adding
    a X; it stays within bf16 accuracy of the one-rounding form on Gaussian input."""
    X = oracle.f32_to_bf16(W.gaussian([14], (96, 40), 0.02))
    a = f64(oracle.cascade(X))
    b = f64(oracle.cascade(X, split=True))
    assert 0 < np.linalg.norm(a - b) / np.linalg.norm(a) < 2e-2


def test_oracle_matches_stored_small_cases():
    """Regression: the stored bits (written by tests/golden/make_oracle_golden.py) still
    come out, on this machine's compiler and architecture."""
    import importlib.util
    import os
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("mk", os.path.join(here, "make_oracle_golden.py"))
    mk = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mk)
    got = mk.compute()
    lines = [l.split() for l in open(os.path.join(here, "oracle_small.txt")) if not l.startswith("#")]
    i = 0
    for name, g, m, n in mk.CASES:
        assert lines[i][:2] == ["case", name]
        out = np.array([int(x, 16) for x in lines[i + 1][1:]], np.uint16).reshape(g, m, n)
        vel = np.array([int(x, 16) for x in lines[i + 2][1:]], np.uint32).reshape(2, g, m, n)
        np.testing.assert_array_equal(got[name][0], out)
        np.testing.assert_array_equal(got[name][1].view(np.uint32), vel)
        i += 3
