"""GPU parity of libanvil against the CPU oracle (all tests need a GB300).

Tolerances (the acceptance bar of the build):
  * velocity rails: within 1e-6 relative of the oracle (they come out bit-identical,
    both sides doing the same fp32 operations one rounding at a time);
  * X_raw (bf16 cast of the lookahead): bit-identical;
  * every bf16 stage and the output: within 1e-2 relative Frobenius error per matrix;
  * the output against the fp64 SVD closed form: within 3e-2 (full matrix for
    well-conditioned input; on the dominant subspace for ill-conditioned input).
Inputs are seeded (polynomial_matrix_whitening_gb300.workloads); no oracle input or
expected value comes from the GPU.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from polynomial_matrix_whitening_gb300 import workloads as W  # noqa: E402

VEL_RTOL = 1e-6
OUT_RTOL = 1e-2
CLOSED_RTOL = 3e-2
U32 = 2.0 ** -24
UBF = 2.0 ** -8


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from polynomial_matrix_whitening_gb300 import anvil
    return anvil


def bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64(b):
    return oracle.bf16_to_f32(b).astype(np.float64)


def rel(a, b):
    n = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (n if n > 0 else 1.0)


# Ill-conditioned input (the power-law workload, sigma_i = i^-1.5): the cascade amplifies
# bf16-level differences in the small singular directions (F'(0) = 643), and how products
# are summed decides the bf16 roundings of the Gram.  The oracle sums in sequential fp32 with
# round-to-nearest; the tensor cores that run these products, here and in the page's own
# arrangement (torch bmm / baddbmm in bf16, i.e. cuBLAS), accumulate with a bias toward
# zero, which over the 2816-long Gram sums leaves the output 1.2-1.3% from the oracle on
# this input.  The bar there: the full-matrix error may exceed 1e-2 only up to 1.1x the
# distance between the page's arrangement run by torch on this GPU and the oracle (and
# never 3e-2), and the 1e-2 bar holds on the dominant subspace (sigma/d >= 3.3e-3, where
# F >= 0.999).  (The two tensor-core results need not be close to each other: on a
# rank-32 + noise matrix both sat 0.6% from the oracle and 1.5% from one another.)
ILL_FULL_RTOL = 3e-2
ILL_PAGE_FACTOR = 1.1


def dominant_rel(out_gpu, out_or, X_or):
    U, S, Vt = np.linalg.svd(f64(X_or), full_matrices=False)
    d = np.sqrt(np.sum(S ** 2)) * 1.05 + 1e-6
    keep = S / d >= 3.3e-3
    P = lambda o: U[:, keep].T @ f64(o) @ Vt[keep].T  # noqa: E731
    return rel(P(out_gpu), P(out_or))


def torch_arrangement(X_bits, maps=oracle.ANVIL_MAPS, margin=1.05, eps=1e-6):
    """The page's tensor operations on one bf16 matrix, run by torch on this GPU: matrix
    products in bf16 with fp32 accumulation (cuBLAS), `b A + c A A` and `a X + X B` each
    one fp32 epilogue and one bf16 rounding (baddbmm), the trace from the bf16 Gram's
    diagonal.  A measure of what tensor-core accumulation does to this input, not an
    expected value: the expected value is the oracle's."""
    prev = torch.backends.cuda.matmul.allow_bf16_reduced_precision_reduction
    torch.backends.cuda.matmul.allow_bf16_reduced_precision_reduction = False
    try:
        x = torch.from_numpy(np.ascontiguousarray(X_bits).view(np.int16)).cuda().view(torch.bfloat16)
        tall = x.shape[0] > x.shape[1]

        def gram(y):
            return (y.mT @ y) if tall else (y @ y.mT)

        a0 = gram(x)
        d = a0.diagonal().float().sum().sqrt() * np.float32(margin) + np.float32(eps)
        y = (x.float() / d).to(torch.bfloat16)
        acc = (a0.float() / (d * d)).to(torch.bfloat16)
        for k, (a, b, c) in enumerate(maps):
            a, b, c = (float(np.float32(v)) for v in (a, b, c))
            if k > 0:
                acc = gram(y)
            bm = torch.baddbmm(acc[None], acc[None], acc[None], beta=b, alpha=c)[0]
            y = (torch.baddbmm(y[None], y[None], bm[None], beta=a)[0] if tall
                 else torch.baddbmm(y[None], bm[None], y[None], beta=a)[0])
        return bits(y)
    finally:
        torch.backends.cuda.matmul.allow_bf16_reduced_precision_reduction = prev


def check_output(out_gpu, out_or, X_or, ill):
    """Returns (full-matrix rel error, dominant-subspace rel error or None, the page
    arrangement's rel error or None) after asserting the bar."""
    got, want = f64(out_gpu), f64(out_or)
    assert np.isfinite(got).all()
    full = rel(got, want)
    if not ill:
        assert full <= OUT_RTOL, full
        return full, None, None
    page = f64(torch_arrangement(X_or))
    e_page = rel(page, want)
    dom = dominant_rel(out_gpu, out_or, X_or)
    assert dom <= OUT_RTOL, dom
    assert full <= max(OUT_RTOL, ILL_PAGE_FACTOR * e_page) and full <= ILL_FULL_RTOL, (full, e_page)
    return full, dom, e_page


def gpu_bank(A, grad, vel, scal):
    dev = torch.device("cuda")
    g = torch.from_numpy(grad).to(dev)
    v = torch.from_numpy(vel).to(dev)
    out = torch.empty(grad.shape, dtype=torch.bfloat16, device=dev)
    return A.Bank(g, v, out, **scal)


def scal_dict(s):
    return dict(momentum=s.momentum, fast_beta=s.fast_beta, fast_weight=s.fast_weight,
                slow_beta=s.slow_beta)


# ------------------------------------------------------------------ failure detection

def test_bounded_wait_gives_up_and_reports(A):
    """A wait on a barrier nothing completes returns after its limit with a timeout status;
    the context stays usable."""
    assert A.device_error(clear=True) == A.OK
    A.selftest_wait_timeout(2000)
    assert A.device_error(clear=True) == A.ERR_TIMEOUT
    assert A.device_error(clear=True) == A.OK
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0


def test_last_device_error_reads_one_stream(A):
    """The per-stream read: a wait that gives up in work queued on a side stream is
    reported by anvil_last_device_error on that stream, once (the read resets the word),
    without waiting for the device."""
    s = torch.cuda.Stream()
    assert A.last_device_error(s) == A.OK
    A.selftest_wait_timeout(2000, stream=s)
    assert A.last_device_error(s) == A.ERR_TIMEOUT
    assert A.last_device_error(s) == A.OK
    assert A.device_error(clear=True) == A.OK


# ------------------------------------------------------------------ stage by stage

# Ragged and tiny shapes on both sides of every path: n % 8 != 0 writes `out` with plain
# stores, n % 8 == 0 with clipped TMA stores (wide: Y boxes; tall: transposed boxes).
SMALL = [(2, 256, 768), (2, 300, 130), (2, 130, 300), (1, 200, 200), (2, 4, 3), (2, 3, 4),
         (1, 1, 1), (1, 129, 1000), (1, 1000, 257), (3, 128, 128), (1, 64, 2048),
         (2, 1000, 264), (2, 264, 1000), (2, 4, 8), (2, 24, 16), (1, 520, 520)]


def _gemm_bound(exact, abs_terms, K):
    # any fp32 summation order: |err| <= K u sum|terms| (4x slack for the tensor-core
    # adder), then one bf16 rounding of the result
    e = 4 * K * U32 * abs_terms
    return e + UBF * (np.abs(exact) + e) + 1e-30


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_stages_match_oracle(A, shape):
    g, m, n = shape
    tall = m > n
    s_dim = min(m, n)
    grad, vel = W.random_case(sum(shape), g, m, n)
    sc = dict(momentum=0.95, fast_beta=0.8, fast_weight=0.4385, slow_beta=0.98)
    bank = gpu_bank(A, grad, vel, sc)
    ws = A.alloc_workspace([shape])
    t = A.bank_step_traced(bank, ws)
    torch.cuda.synchronize()
    assert A.device_error() == A.OK

    X_or, _, vel_or = oracle.momentum(grad, vel, sc["momentum"], sc["fast_beta"],
                                      sc["fast_weight"], sc["slow_beta"])
    vel_gpu = bank.velocity.cpu().numpy()
    assert np.max(np.abs(vel_gpu - vel_or)) <= VEL_RTOL * np.max(np.abs(vel_or))
    np.testing.assert_array_equal(bits(t["X_raw"]), X_or)
    np.testing.assert_array_equal(bank.grad.cpu().numpy(), grad)  # grad never written

    out_gpu = bits(bank.out)
    np.testing.assert_array_equal(out_gpu, bits(t["X"][-1]))
    if s_dim == 1 and m * n == 1:
        # a 1x1 matrix normalises to bf16(1/1.05) = 0.953125, just above 1/margin, where
        # the six maps diverge in bf16 (oracle and GPU alike): compare every stage bit for bit
        for i in range(g):
            o, tr = oracle.cascade(X_or[i], trace=True)
            np.testing.assert_array_equal(bits(t["X"][:, i]), tr["X"])
            np.testing.assert_array_equal(bits(t["A"][:, i]), tr["A"])
            np.testing.assert_array_equal(bits(t["B"][:, i]), tr["B"])
            np.testing.assert_array_equal(out_gpu[i], o)
        return
    for i in range(g):
        o, tr = oracle.cascade(X_or[i], trace=True)
        # d: the trace sums bf16-rounded diagonal entries whose fp32 sums are taken in a
        # different order on each side, so a few entries may round to the neighbouring bf16
        # value (2^-8 of that entry each); 1e-4 relative covers that and moves X by < 1e-4.
        assert abs(float(t["d"][i]) - tr["d"][0]) <= 1e-4 * tr["d"][0]
        assert rel(f64(bits(t["X"][0, i])), f64(tr["X"][0])) <= 1e-3
        for k in range(6):
            assert rel(f64(bits(t["A"][k, i])), f64(tr["A"][k])) <= OUT_RTOL, ("A", k)
            assert rel(f64(bits(t["B"][k, i])), f64(tr["B"][k])) <= OUT_RTOL, ("B", k)
            assert rel(f64(bits(t["X"][k + 1, i])), f64(tr["X"][k + 1])) <= OUT_RTOL, ("X", k)
        got = f64(out_gpu[i])
        assert np.isfinite(got).all()
        assert rel(got, f64(o)) <= OUT_RTOL

        # the GPU's own stages against fp64 evaluations of the page's formulas (no oracle)
        maps = [tuple(float(np.float32(v)) for v in mp) for mp in A.default_maps()]
        K = m if tall else n
        for k, (a, b, c) in enumerate(maps):
            Xk = f64(bits(t["X"][k, i]))
            Ak = f64(bits(t["A"][k, i]))
            if k > 0:
                G = Xk.T @ Xk if tall else Xk @ Xk.T
                aG = np.abs(Xk).T @ np.abs(Xk) if tall else np.abs(Xk) @ np.abs(Xk).T
                assert np.all(np.abs(Ak - G) <= _gemm_bound(G, aG, K)), ("gram", k)
            Bk = f64(bits(t["B"][k, i]))
            P = b * Ak + c * (Ak @ Ak)
            aP = np.abs(b * Ak) + abs(c) * (np.abs(Ak) @ np.abs(Ak))
            assert np.all(np.abs(Bk - P) <= _gemm_bound(P, aP, s_dim + 2)), ("sqpoly", k)
            Xn = f64(bits(t["X"][k + 1, i]))
            C = a * Xk + (Xk @ Bk if tall else Bk @ Xk)
            aC = np.abs(a * Xk) + (np.abs(Xk) @ np.abs(Bk) if tall else np.abs(Bk) @ np.abs(Xk))
            assert np.all(np.abs(Xn - C) <= _gemm_bound(C, aC, s_dim + 2)), ("xupdate", k)


# Other coefficient sets through the same kernels: the ABI takes any maps[] / nmaps.
NS_CUBIC = (1.5, -0.5, 0.0)  # the textbook cubic Newton-Schulz step x -> 1.5 x - 0.5 x^3
OTHER_MAPS = {
    "ns_cubic_x5": [NS_CUBIC] * 5,
    "single_map": [(3.923798038567, -6.095026865488, 3.905234618423)],
    "sixteen_maps": [NS_CUBIC] * 10 + [(2.0, -1.5, 0.5)] * 6,
    "mixed": [(2.0, -1.5, 0.5), (1.875, -1.25, 0.375), NS_CUBIC],
}


@pytest.mark.parametrize("name", sorted(OTHER_MAPS))
@pytest.mark.parametrize("shape", [(3, 256, 768), (2, 520, 264)], ids=lambda s: "x".join(map(str, s)))
def test_other_coefficient_sets(A, name, shape):
    maps = OTHER_MAPS[name]
    g, m, n = shape
    grad, vel = W.random_case(77 + len(maps), g, m, n)
    sc = dict(momentum=0.95, fast_beta=0.85, fast_weight=0.4385, slow_beta=0.98)
    bank = gpu_bank(A, grad, vel, sc)
    A.multi_bank_step([bank], A.alloc_workspace([shape]), maps=maps, margin=1.05, eps=1e-6)
    torch.cuda.synchronize()
    out, vel_or = oracle.bank_step(grad, vel, sc["momentum"], sc["fast_beta"], sc["fast_weight"],
                                   sc["slow_beta"], maps=maps)
    vg = bank.velocity.cpu().numpy()
    assert np.max(np.abs(vg - vel_or)) <= VEL_RTOL * np.max(np.abs(vel_or))
    got = bits(bank.out)
    for i in range(g):
        assert np.isfinite(f64(got[i])).all()
        assert rel(f64(got[i]), f64(out[i])) <= OUT_RTOL, (name, i)


@pytest.mark.parametrize("margin,eps", [(1.2, 1e-3), (2.0, 0.5)])
@pytest.mark.parametrize("shape", [(3, 256, 768), (2, 520, 264)], ids=lambda s: "x".join(map(str, s)))
def test_margin_and_eps_are_parameters(A, shape, margin, eps):
    """d = sqrt(tr) * margin + eps with the caller's margin and eps (the page's
    FROBENIUS_MARGIN and FROBENIUS_EPS made parameters): d from the traced step against the
    oracle's (eps = 0.5 is about 8% of d here, a margin of 2 almost doubles it), and the
    output within the bf16 bar."""
    g, m, n = shape
    grad, vel = W.random_case(131 + m, g, m, n)
    sc = dict(momentum=0.95, fast_beta=0.85, fast_weight=0.4385, slow_beta=0.98)
    bank = gpu_bank(A, grad, vel, sc)
    t = A.bank_step_traced(bank, A.alloc_workspace([shape]), margin=margin, eps=eps)
    torch.cuda.synchronize()
    assert A.device_error() == A.OK
    X_or, _, _ = oracle.momentum(grad, vel, **sc)
    got = bits(bank.out)
    for i in range(g):
        o, tr = oracle.cascade(X_or[i], margin=margin, eps=eps, trace=True)
        assert abs(float(t["d"][i]) - tr["d"][0]) <= 1e-4 * tr["d"][0], (i, float(t["d"][i]), tr["d"][0])
        assert rel(f64(got[i]), f64(o)) <= OUT_RTOL, i


@pytest.mark.parametrize("shape", [(22, 256, 768), (3, 300, 130), (2, 130, 257)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bf16_grad_input(A, shape):
    """The page's bank gradient is bf16: the same step from bf16 gradient bits (the oracle
    reads them as their exact fp32 values)."""
    g, m, n = shape
    grad, vel = W.random_case(90 + m, g, m, n)
    gh = oracle.f32_to_bf16(grad)
    sc = dict(momentum=0.95, fast_beta=0.85, fast_weight=0.4385, slow_beta=0.98)
    dev = torch.device("cuda")
    bank = A.Bank(torch.from_numpy(gh.view(np.int16)).to(dev).view(torch.bfloat16),
                  torch.from_numpy(vel).to(dev), torch.empty(shape, dtype=torch.bfloat16, device=dev), **sc)
    A.multi_bank_step([bank], A.alloc_workspace([shape]))
    torch.cuda.synchronize()
    out, vel_or = oracle.bank_step(oracle.bf16_to_f32(gh), vel, **sc)
    vg = bank.velocity.cpu().numpy()
    assert np.max(np.abs(vg - vel_or)) <= VEL_RTOL * np.max(np.abs(vel_or))
    got = bits(bank.out)
    for i in range(g):
        assert rel(f64(got[i]), f64(out[i])) <= OUT_RTOL


# A rank-1 X has sigma_1 = ||X||_F, so sigma_1 / d = 1/1.05 up to rounding: the edge of the
# maps' flat region (F(0.9524) = 1.015 with F' = 1.8e3, F(0.953) = 8e11).  The bf16 trace
# decides on which side it lands, so out's top singular value is anything from 1 to about
# 150 (both seen here), on the oracle and the GPU alike, and the method's own conditioning
# is poor: moving one input element by one bf16 ulp moves the oracle's dominant output by
# up to 11% (median 1e-5 to 3e-4).  Parity is held to that conditioning.
RANK1_RTOL = 0.15


@pytest.mark.parametrize("shape", [(2, 256, 768), (2, 768, 256), (1, 520, 520)],
                         ids=lambda s: "x".join(map(str, s)))
def test_rank_one_gradient(A, shape):
    """A rank-1 gradient, the most degenerate input short of zero.  Its singular value maps
    to F(1/1.05); the bf16 rounding noise of the outer product, in the null
    directions (sigma/d ~ 3e-4), is amplified by F'(0) = 643 on both sides alike, to
    singular values below 1.  Finite output, the input's singular vectors, the amplified
    noise below 1, and the oracle's top singular value and dominant direction within
    RANK1_RTOL."""
    g, m, n = shape
    rng = np.random.default_rng(140 + m + n)
    u = rng.standard_normal((g, m, 1))
    v = rng.standard_normal((g, 1, n))
    grad = (0.02 * u * v / np.sqrt(m * n) * 40).astype(np.float32)
    vel = np.zeros((2, g, m, n), np.float32)
    sc = dict(momentum=0.95, fast_beta=0.85, fast_weight=1.0, slow_beta=0.98)
    bank = gpu_bank(A, grad, vel, sc)
    A.multi_bank_step([bank], A.alloc_workspace([shape]))
    torch.cuda.synchronize()
    assert A.device_error() == A.OK
    X_or, _, _ = oracle.momentum(grad, vel, **sc)
    out_or, _ = oracle.bank_step(grad, vel, **sc)
    got = bits(bank.out)
    for i in range(g):
        o = f64(got[i])
        assert np.isfinite(o).all()
        Ux, _, Vx = np.linalg.svd(f64(X_or[i]), full_matrices=False)
        Uo, So, Vo = np.linalg.svd(o, full_matrices=False)
        S_or = np.linalg.svd(f64(out_or[i]), compute_uv=False)
        assert abs(So[0] - S_or[0]) <= RANK1_RTOL * S_or[0], (So[:3], S_or[:3])
        assert abs(Ux[:, 0] @ Uo[:, 0]) > 0.999 and abs(Vx[0] @ Vo[0]) > 0.999
        assert So[1] < 1.0, So[:3]
        dom = dominant_rel(got[i], out_or[i], X_or[i])
        assert dom <= RANK1_RTOL, dom
        print(f"rank-1 {shape} matrix {i}: top singular value {So[0]:.4f} (oracle {S_or[0]:.4f}), "
              f"dominant {dom:.2e}, full {rel(o, f64(out_or[i])):.2e}")


def test_zero_grad_gives_zero_output(A):
    shape = (2, 300, 130)
    grad = np.zeros(shape, np.float32)
    vel = np.zeros((2,) + shape, np.float32)
    bank = gpu_bank(A, grad, vel, {})
    ws = A.alloc_workspace([shape])
    A.multi_bank_step([bank], ws)
    out = bank.out.float().cpu().numpy()
    assert np.isfinite(out).all() and not out.any()


# ------------------------------------------------------------------ grouping, graphs

def _small_banks(A, seed):
    shapes = [(3, 256, 768), (2, 300, 130), (4, 130, 257)]
    banks = []
    for j, (g, m, n) in enumerate(shapes):
        grad, vel = W.random_case(seed + j, g, m, n)
        banks.append(gpu_bank(A, grad, vel, dict(momentum=0.95, fast_beta=0.7 + 0.05 * j,
                                                 fast_weight=0.4385, slow_beta=0.98)))
    return shapes, banks


def test_grouped_banks_equal_separate_calls(A):
    """One grouped call over three banks == three one-bank calls == per-matrix calls, bit
    for bit (every output tile is computed the same way whatever the grouping)."""
    shapes, banks = _small_banks(A, 50)
    _, solo = _small_banks(A, 50)
    A.multi_bank_step(banks, A.alloc_workspace(shapes))
    for b, s in zip(solo, shapes):
        A.multi_bank_step([b], A.alloc_workspace([s]))
    torch.cuda.synchronize()
    for b, s in zip(banks, solo):
        assert torch.equal(b.out.view(torch.int16), s.out.view(torch.int16))
        assert torch.equal(b.velocity, s.velocity)
    # per-matrix calls through the library-owned workspace
    _, per = _small_banks(A, 50)
    b = per[2]
    for i in range(b.grad.shape[0]):
        o = torch.empty_like(b.out[i:i + 1])
        v = b.velocity[:, i:i + 1].clone()
        A.bank_step(b.grad[i:i + 1].clone(), v, o, **b.scalars)
        assert torch.equal(o.view(torch.int16), banks[2].out[i:i + 1].view(torch.int16))


def test_eight_banks_in_one_call(A):
    """The largest call by bank count (ANVIL_MAX_BANKS = 8), tall, wide, square and ragged
    banks mixed: equal to one call per bank bit for bit, and each bank against the oracle."""
    shapes = [(3, 256, 768), (2, 768, 256), (2, 300, 130), (1, 130, 300), (2, 520, 520),
              (4, 64, 64), (1, 1000, 264), (2, 24, 16)]
    assert len(shapes) == A.MAX_BANKS
    sc = dict(momentum=0.95, fast_beta=0.85, fast_weight=0.4385, slow_beta=0.98)
    cases = [W.random_case(170 + j, *s) for j, s in enumerate(shapes)]
    banks = [gpu_bank(A, gr, ve, sc) for gr, ve in cases]
    solo = [gpu_bank(A, gr, ve, sc) for gr, ve in cases]
    A.multi_bank_step(banks, A.alloc_workspace(shapes))
    for b, s in zip(solo, shapes):
        A.multi_bank_step([b], A.alloc_workspace([s]))
    torch.cuda.synchronize()
    assert A.device_error() == A.OK
    for (gr, ve), b, s in zip(cases, banks, solo):
        assert torch.equal(b.out.view(torch.int16), s.out.view(torch.int16))
        assert torch.equal(b.velocity, s.velocity)
        out, _ = oracle.bank_step(gr, ve, **sc)
        got = bits(b.out)
        for i in range(gr.shape[0]):
            assert rel(f64(got[i]), f64(out[i])) <= OUT_RTOL


@pytest.mark.parametrize("shapes", [
    # 400 and 1000 matrices in three banks of tiny shapes: thousands of one-tile items per
    # phase, walked phase by phase
    [(200, 24, 16), (120, 8, 40), (80, 20, 20)],
    [(500, 24, 16), (300, 8, 40), (200, 20, 20)],
], ids=["400_matrices", "1000_matrices"])
def test_many_matrices_item_order(A, shapes):
    """Calls with hundreds of matrices (thousands of items in each phase, so pairs move
    between phases of different matrices all the time): the grouped call equals one call
    per bank bit for bit, and sampled matrices match the oracle."""
    banks, solo, cases = [], [], []
    for j, (g, m, n) in enumerate(shapes):
        grad, vel = W.random_case(900 + j, g, m, n)
        sc = dict(momentum=0.95, fast_beta=0.85, fast_weight=0.4385, slow_beta=0.98)
        banks.append(gpu_bank(A, grad, vel, sc))
        solo.append(gpu_bank(A, grad, vel, sc))
        cases.append((grad, vel, sc))
    A.multi_bank_step(banks, A.alloc_workspace(shapes))
    for b, s in zip(solo, shapes):
        A.multi_bank_step([b], A.alloc_workspace([s]))
    torch.cuda.synchronize()
    assert A.device_error() == A.OK
    for j, (b, s) in enumerate(zip(banks, solo)):
        assert torch.equal(b.out.view(torch.int16), s.out.view(torch.int16))
        assert torch.equal(b.velocity, s.velocity)
        grad, vel, sc = cases[j]
        g = grad.shape[0]
        pick = [0, g // 2, g - 1]
        out_or, vel_or = oracle.bank_step(grad[pick], vel[:, pick], sc["momentum"], sc["fast_beta"],
                                          sc["fast_weight"], sc["slow_beta"])
        got = bits(b.out)[pick]
        np.testing.assert_array_equal(b.velocity[:, pick].cpu().numpy(), vel_or)
        for k in range(len(pick)):
            assert rel(f64(got[k]), f64(out_or[k])) <= OUT_RTOL


@pytest.mark.parametrize("case,reps", [
    ("full_step", 20),
    ("400_matrices", 30),
    ("tiny", 100),
], ids=["full_step", "400_matrices", "tiny"])
def test_repeated_steps_are_bitwise_identical(A, case, reps):
    """The same step, repeated on the same inputs, gives the same bits every time: every
    value the cascade reads between its phases is complete when it is read (completion
    counters, publication after the stores), and every sum has a fixed order.  The bench's
    three banks, 400 small matrices (the densest dependency waits) and tiny matrices whose
    phases follow one another at once."""
    if case == "full_step":
        wl = W.workloads()["full_step"]
        sc = wl.scalars(0)
        shapes = [(b.g, b.m, b.n) for b in wl.banks]
        grads = [wl.grad(j, 0) for j in range(len(shapes))]
        vels = [wl.velocity(j) for j in range(len(shapes))]
        scal = scal_dict(sc)
    else:
        shapes = ([(200, 24, 16), (120, 8, 40), (80, 20, 20)] if case == "400_matrices"
                  else [(1, 3, 4), (2, 4, 3), (1, 1, 1), (1, 8, 2)])
        grads, vels = zip(*[W.random_case(950 + j, g, m, n) for j, (g, m, n) in enumerate(shapes)])
        scal = dict(momentum=0.95, fast_beta=0.85, fast_weight=0.4385, slow_beta=0.98)
    banks = [gpu_bank(A, gr, ve, scal) for gr, ve in zip(grads, vels)]
    vel0 = [b.velocity.clone() for b in banks]
    ws = A.alloc_workspace(shapes)
    first = None
    for r in range(reps):
        for b, v in zip(banks, vel0):
            b.velocity.copy_(v)
        A.multi_bank_step(banks, ws)
        outs = [b.out.view(torch.int16).clone() for b in banks]
        if first is None:
            first = outs
        else:
            for k, (o, f) in enumerate(zip(outs, first)):
                assert torch.equal(o, f), (r, k)
    torch.cuda.synchronize()
    assert A.device_error() == A.OK


@pytest.mark.parametrize("shape", [(1, 4096, 16384), (1, 16384, 4096), (2, 2048, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_large_shapes_singular_values(A, shape):
    """Sizes past the oracle's reach (up to 16 row blocks per matrix and the largest
    dimension): for Gaussian gradients with an aspect ratio of 4, every singular value of
    the normalised X lies in [0.01, 1/1.05], where the composite map is within 5e-4 of 1
    (the SVD form of the method), so every singular value of out must be 1 up to the bf16
    roundings of the cascade."""
    g, m, n = shape
    grad = W.gaussian([9000, 1234, 0], (g, m, n), 0.02)
    vel = np.zeros((2, g, m, n), dtype=np.float32)
    bank = gpu_bank(A, grad, vel, dict(momentum=0.95, fast_beta=0.85, fast_weight=1.0, slow_beta=0.98))
    A.multi_bank_step([bank], A.alloc_workspace([shape]))
    torch.cuda.synchronize()
    assert A.device_error() == A.OK
    for i in range(g):
        sv = torch.linalg.svdvals(bank.out[i].float())
        assert torch.isfinite(sv).all()
        assert float(sv.min()) > 0.97 and float(sv.max()) < 1.03, (float(sv.min()), float(sv.max()))


def test_largest_square_block_diagonal(A):
    """The largest small side, 16384 x 16384 (64 x 64 output tiles, 256 k-blocks per Gram
    tile), checked element by element against the oracle.  The gradient holds 64 copies of
    one 256 x 256 Gaussian block G1 on its diagonal and zeros elsewhere.  Every step of the
    method keeps that structure exactly: momentum of a zero is zero, and the off-diagonal
    blocks of X X^T, b A + c A A and a X + B X are sums of exact zeros.  The blocks share
    one d: the trace is 64 times the block's, and in fp32 sqrt(64 tr) = 8 sqrt(tr) exactly,
    so d is the oracle's d for the single block G1 with the margin multiplied by 8 (exact
    too), up to the order in which the trace is summed.  So each diagonal block of out must
    match the oracle's step on G1 with margin 8 x 1.05 within the bf16 bar, and every other
    block must be zero."""
    nb, k = 256, 64
    size = nb * k
    g1 = W.gaussian([9100, 0], (1, nb, nb), 0.02)
    scal = dict(momentum=0.95, fast_beta=0.85, fast_weight=1.0, slow_beta=0.98)
    want, _ = oracle.bank_step(g1, np.zeros((2, 1, nb, nb), np.float32), **scal,
                               margin=float(np.float32(8.0) * np.float32(oracle.FROBENIUS_MARGIN)))
    dev = torch.device("cuda")
    grad = torch.zeros((1, size, size), dtype=torch.float32, device=dev)
    blk = torch.from_numpy(g1[0]).to(dev)
    for b in range(k):
        grad[0, b * nb:(b + 1) * nb, b * nb:(b + 1) * nb] = blk
    vel = torch.zeros((2, 1, size, size), dtype=torch.float32, device=dev)
    out = torch.empty((1, size, size), dtype=torch.bfloat16, device=dev)
    bank = A.Bank(grad, vel, out, **scal)
    A.multi_bank_step([bank], A.alloc_workspace([(1, size, size)]))
    torch.cuda.synchronize()
    assert A.device_error() == A.OK
    del grad, vel
    tiles = out[0].view(k, nb, k, nb)
    amax = tiles.abs().amax(dim=(1, 3)).float()
    diag = torch.arange(k, device=dev)
    assert torch.isfinite(amax).all()
    off = amax.clone()
    off[diag, diag] = 0.0
    assert float(off.max()) == 0.0, "a block off the diagonal is not zero"
    errs = []
    for b in range(k):
        got = bits(tiles[b, :, b, :])
        errs.append(rel(f64(got), f64(want[0])))
    assert max(errs) <= OUT_RTOL, max(errs)


def test_cuda_graph_with_device_scalars(A):
    """A captured step reads the device scalar block when it runs: replays with new
    scalars equal eager calls with those scalars as host values."""
    shapes, banks = _small_banks(A, 60)
    _, eager = _small_banks(A, 60)
    ws = A.alloc_workspace(shapes)
    ws2 = A.alloc_workspace(shapes)
    dsc = torch.zeros((3, 4), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        dsc.copy_(torch.tensor([[0.95, 0.85, 1.0, 0.98]] * 3))
        A.multi_bank_step(banks, ws, d_scalars=dsc, stream=s)  # warm-up outside capture
        torch.cuda.synchronize()
        # reset state so graph replays and eager calls start from the same rails
        for b, e in zip(banks, eager):
            b.velocity.copy_(e.velocity)
        with torch.cuda.graph(graph, stream=s):
            A.multi_bank_step(banks, ws, d_scalars=dsc, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for step, (fb, fw) in enumerate([(0.6, 1.0), (0.75, 0.4385), (0.85, 0.4385)]):
        dsc.copy_(torch.tensor([[0.95, fb, fw, 0.98]] * 3))
        graph.replay()
        for e in eager:
            e.scalars.update(fast_beta=fb, fast_weight=fw)
        A.multi_bank_step(eager, ws2)
        torch.cuda.synchronize()
        for b, e in zip(banks, eager):
            assert torch.equal(b.out.view(torch.int16), e.out.view(torch.int16)), step
            assert torch.equal(b.velocity, e.velocity), step


# ------------------------------------------------------------------ full-size workloads

def _closed_form_check(X_bits, out_bits, tall, ill_conditioned):
    """fp64 SVD closed form U F(S/d) V^T of the oracle's bf16 X.  Ill-conditioned input:
    compare on the dominant subspace sigma/d >= 3.3e-3 (where F >= 0.999), as the
    bf16 pipeline cannot resolve the rest (F'(0) = 643)."""
    X = f64(X_bits)
    out = f64(out_bits)
    U, S, Vt = np.linalg.svd(X, full_matrices=False)
    d = np.sqrt(np.sum(S ** 2)) * 1.05 + 1e-6
    sig = S / d
    F = sig.copy()
    for a, b, c in oracle.ANVIL_MAPS:
        F = a * F + b * F ** 3 + c * F ** 5
    if not ill_conditioned:
        want = (U * F) @ Vt
        return rel(out, want)
    keep = sig >= 3.3e-3
    blk = U[:, keep].T @ out @ Vt[keep].T
    return rel(blk, np.diag(F[keep]))


WORKLOAD_STEPS = {"single_wide": 1, "single_wide_blend": 1, "qk_bank": 10, "vo_bank": 10,
                  "mlp_bank": 10}


@pytest.mark.parametrize("name", list(WORKLOAD_STEPS))
def test_workload_parity(A, name):
    wl = W.workloads()[name]
    steps = WORKLOAD_STEPS[name]
    b0 = wl.banks[0]
    shape = (b0.g, b0.m, b0.n)
    vel = wl.velocity(0)
    grad0 = wl.grad(0, 0)
    bank = gpu_bank(A, grad0, vel, scal_dict(wl.scalars(0)))
    ws = A.alloc_workspace([shape])
    vel_or = vel
    sample = sorted({0, b0.g // 2, b0.g - 1})
    grad = grad0
    for step in range(steps):
        if wl.fresh_per_step and step > 0:
            grad = wl.grad(0, step)
        bank.grad.copy_(torch.from_numpy(grad))
        sc = wl.scalars(step)
        bank.scalars = scal_dict(sc)
        A.multi_bank_step([bank], ws)
        X_or, _, vel_or = oracle.momentum(grad, vel_or, sc.momentum, sc.fast_beta, sc.fast_weight,
                                          sc.slow_beta)
        # the rails every step (every element), the output at the first and last step
        vg = bank.velocity.cpu().numpy()
        assert np.max(np.abs(vg - vel_or)) <= VEL_RTOL * np.max(np.abs(vel_or)), step
        if step in (0, steps - 1):
            out = bits(bank.out)
            ill = wl.kind == "power_law"
            for i in sample:
                o = oracle.cascade(X_or[i])
                full, dom, e_page = check_output(out[i], o, X_or[i], ill)
                cf = _closed_form_check(X_or[i], out[i], b0.m > b0.n, ill)
                print(f"{name} step {step} matrix {i}: vs oracle {full:.2e}"
                      f"{'' if dom is None else f' (dominant {dom:.2e}; page arrangement {e_page:.2e})'}"
                      f", vs closed form {cf:.2e}")
                assert cf <= CLOSED_RTOL


def test_full_step_graph_parity(A):
    """All three banks, the whole 100-step sequence captured in ONE CUDA graph (the grad
    pool of 4 cycled by pointer, the post-engage scalars read from a device block when the
    graph runs) and replayed once.  Inside the graph, after steps 1, 2, 50 and 100, the
    outputs and rails of matrices {0, 10, 11, 21} of every bank are copied aside; each is
    checked against the oracle run step by step: rails within 1e-6, Gaussian outputs within
    the plain 1e-2 full-matrix bar.  The rank-32 + noise matrices (11-21) are held to the
    ill-conditioned bar: once the rails mix the pool's four rank-32 gradients, their noise
    directions sit where the cascade amplifies accumulation differences (the qk bank's
    matrix 21 measured 1.02e-2 at step 50, as far from the oracle as the page's own
    arrangement on this GPU)."""
    wl = W.workloads()["full_step"]
    dev = torch.device("cuda")
    pool = [[wl.grad(j, p) for j in range(3)] for p in range(wl.pool)]
    pool_d = [[torch.from_numpy(x).to(dev) for x in p] for p in pool]
    vels = [wl.velocity(j) for j in range(3)]
    sc = wl.scalars(0)
    banks = [A.Bank(pool_d[0][j], torch.from_numpy(vels[j]).to(dev),
                    torch.empty((b.g, b.m, b.n), dtype=torch.bfloat16, device=dev), **scal_dict(sc))
             for j, b in enumerate(wl.banks)]
    ws = A.alloc_workspace([b.shape for b in banks])
    dsc = torch.tensor([[sc.momentum, sc.fast_beta, sc.fast_weight, sc.slow_beta]] * 3,
                       dtype=torch.float32, device=dev)
    check, sample = (1, 2, 50, 100), [0, 10, 11, 21]
    snap_out = {t: [torch.empty((len(sample), b.m, b.n), dtype=torch.bfloat16, device=dev)
                    for b in wl.banks] for t in check}
    snap_vel = {t: [torch.empty((2, len(sample), b.m, b.n), dtype=torch.float32, device=dev)
                    for b in wl.banks] for t in check}
    vel0 = [b.velocity.clone() for b in banks]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        A.multi_bank_step(banks, ws, d_scalars=dsc, stream=s)  # device set-up, outside capture
        s.synchronize()
        for b, v in zip(banks, vel0):
            b.velocity.copy_(v)
        with torch.cuda.graph(graph, stream=s):
            for step in range(1, 101):
                for j, b in enumerate(banks):
                    b.grad = pool_d[(step - 1) % wl.pool][j]
                A.multi_bank_step(banks, ws, d_scalars=dsc, stream=s)
                if step in check:
                    for j, b in enumerate(banks):
                        for k, i in enumerate(sample):
                            snap_out[step][j][k].copy_(b.out[i])
                            snap_vel[step][j][:, k].copy_(b.velocity[:, i])
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert A.device_error() == A.OK

    vel_or = [np.ascontiguousarray(v[:, sample]) for v in vels]
    for step in range(1, 101):
        Xs = []
        for j in range(3):
            grad = np.ascontiguousarray(pool[(step - 1) % wl.pool][j][sample])
            X, _, vel_or[j] = oracle.momentum(grad, vel_or[j], sc.momentum, sc.fast_beta,
                                              sc.fast_weight, sc.slow_beta)
            Xs.append(X)
        if step not in check:
            continue
        for j, b in enumerate(wl.banks):
            vg = snap_vel[step][j].cpu().numpy()
            assert np.max(np.abs(vg - vel_or[j])) <= VEL_RTOL * np.max(np.abs(vel_or[j])), (step, j)
            out = bits(snap_out[step][j])
            for k, i in enumerate(sample):
                o = oracle.cascade(Xs[j][k])
                full, dom, e_page = check_output(out[k], o, Xs[j][k], i >= 11)
                cf = _closed_form_check(Xs[j][k], out[k], b.m > b.n, i >= 11)
                print(f"full_step step {step} bank {j} matrix {i}: vs oracle {full:.2e}"
                      f"{'' if dom is None else f' (dominant {dom:.2e}; page arrangement {e_page:.2e})'}"
                      f", vs closed form {cf:.2e}{' (dominant subspace)' if i >= 11 else ''}")
                assert cf <= CLOSED_RTOL
