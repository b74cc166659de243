"""GPU parity of the update tail (equaliser + sign-aligned decay update) with the oracle.

Inputs are seeded synthetic arrays; the oracle never sees a GPU value.  Bars:
lane_energy within 1e-5 relative (sums in another order); the fp32 master weight within
fp32 rounding plus one bf16 ulp of the equalised update (a lane scale whose fp32 value
sits on a bf16 rounding boundary may round the other way), and bit-identical for at
least 99% of the elements.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from polynomial_matrix_whitening_gb300 import workloads as W  # noqa: E402

U32 = 2.0 ** -24


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from polynomial_matrix_whitening_gb300 import anvil
    return anvil


def tail_inputs(seed, g, m, n):
    rng = np.random.default_rng([7000, seed])
    upd = oracle.f32_to_bf16((rng.standard_normal((g, m, n)) * 0.03).astype(np.float32))
    vel = (rng.standard_normal((2, g, m, n)) * 0.01).astype(np.float32)
    nl = m if m >= n else n
    le = np.abs(rng.standard_normal((g, nl)) * 1e-3).astype(np.float32)
    le[:, : nl // 4] = 0.0                     # some lanes start from zero energy
    w = (rng.standard_normal((g, m, n)) * 0.05).astype(np.float32)
    bits = w.view(np.uint32)
    p = (bits >> 16).astype(np.uint16)
    mt = (bits & 0xFFFF).astype(np.uint16)
    lr = (rng.uniform(0.5, 2.0, g) * 0.02).astype(np.float32)
    return upd, vel, le, p, mt, lr


def to_dev(a):
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    return t.view(torch.bfloat16) if a.dtype == np.uint16 else t


def master(p, mt):
    return ((p.astype(np.uint32) << 16) | mt.astype(np.uint32)).view(np.float32).astype(np.float64)


def run_gpu(A, upd, vel, le, p, mt, lr, wd, beta2, calls=1):
    g, m, n = upd.shape
    t = A.Tail(to_dev(upd), to_dev(vel), to_dev(le), to_dev(p),
               torch.from_numpy(mt.view(np.int16)).cuda(), to_dev(lr), wd, beta2)
    ws = torch.empty(A.tail_workspace_bytes([(g, m, n)]), dtype=torch.uint8, device="cuda")
    for _ in range(calls):
        A.update_tail([t], ws)
    torch.cuda.synchronize()
    return (t.param.view(torch.int16).cpu().numpy().view(np.uint16),
            t.mantissa.cpu().numpy().view(np.uint16), t.lane_energy.cpu().numpy())


def check(p_g, mt_g, le_g, p_o, mt_o, le_o, upd, lr):
    np.testing.assert_allclose(le_g, le_o, rtol=1e-5, atol=1e-30)
    wg, wo = master(p_g, mt_g), master(p_o, mt_o)
    u = np.abs(oracle.bf16_to_f32(upd).astype(np.float64))
    bound = 8 * U32 * np.abs(wo) + 2.0 ** -7 * 2 * u * lr.astype(np.float64)[:, None, None] + 1e-40
    assert np.all(np.abs(wg - wo) <= bound)
    same = np.mean((p_g == p_o) & (mt_g == mt_o))
    assert same >= 0.99, same


@pytest.mark.parametrize("shape", [(22, 256, 768), (22, 768, 768), (22, 2816, 768), (3, 130, 300),
                                   (3, 300, 130), (2, 1, 17), (2, 40, 8), (2, 1000, 800)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tail_matches_oracle(A, shape):
    upd, vel, le, p, mt, lr = tail_inputs(sum(shape), *shape)
    wd, beta2 = 0.1, 0.95
    p_g, mt_g, le_g = run_gpu(A, upd, vel, le, p, mt, lr, wd, beta2)
    p_o, mt_o, le_o, _ = oracle.update_tail(upd, le, beta2, p, mt, vel[1], wd, lr)
    check(p_g, mt_g, le_g, p_o, mt_o, le_o, upd, lr)
    assert A.device_error() == A.OK


def test_grouped_tail_over_mixed_banks(A):
    """One tail call over four banks (lanes along rows and along columns, the 16-byte and
    the element path, a tiny bank) matches the oracle bank by bank, and equals one call
    per bank bit for bit."""
    shapes = [(5, 300, 136), (4, 72, 264), (3, 130, 99), (2, 3, 5)]
    wd, beta2 = 0.1, 0.95
    ins = [tail_inputs(700 + j, *s) for j, s in enumerate(shapes)]
    def tails():
        return [A.Tail(to_dev(u), to_dev(v), to_dev(le), to_dev(p), torch.from_numpy(mt.view(np.int16)).cuda(),
                       to_dev(lr), wd, beta2) for (u, v, le, p, mt, lr) in ins]
    grouped, solo = tails(), tails()
    A.update_tail(grouped, torch.empty(A.tail_workspace_bytes(shapes), dtype=torch.uint8, device="cuda"))
    for t, s in zip(solo, shapes):
        A.update_tail([t], torch.empty(A.tail_workspace_bytes([s]), dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert A.device_error() == A.OK
    for t, u, (upd, vel, le, p, mt, lr) in zip(grouped, solo, ins):
        assert torch.equal(t.param.view(torch.int16), u.param.view(torch.int16))
        assert torch.equal(t.mantissa, u.mantissa)
        assert torch.equal(t.lane_energy, u.lane_energy)
        p_o, mt_o, le_o, _ = oracle.update_tail(upd, le, beta2, p, mt, vel[1], wd, lr)
        check(t.param.view(torch.int16).cpu().numpy().view(np.uint16), t.mantissa.cpu().numpy().view(np.uint16),
              t.lane_energy.cpu().numpy(), p_o, mt_o, le_o, upd, lr)


def test_tail_twice_accumulates_lane_energy(A):
    shape = (3, 96, 160)
    upd, vel, le, p, mt, lr = tail_inputs(11, *shape)
    p_g, mt_g, le_g = run_gpu(A, upd, vel, le, p, mt, lr, 0.05, 0.9, calls=2)
    p1, mt1, le1, _ = oracle.update_tail(upd, le, 0.9, p, mt, vel[1], 0.05, lr)
    p_o, mt_o, le_o, _ = oracle.update_tail(upd, le1, 0.9, p1, mt1, vel[1], 0.05, lr)
    check(p_g, mt_g, le_g, p_o, mt_o, le_o, upd, lr)


def test_step_then_tail_matches_oracle_step_then_tail(A):
    """The page's whole anvil_bank_update (cascade, equaliser, decay update) on GPU and
    oracle from the same seeded inputs: the parameter moves by the same update within the
    cascade's 1e-2 bar."""
    shape = (4, 256, 768)
    grad, vel = W.random_case(31, *shape)
    _, _, le, p, mt, lr = tail_inputs(31, *shape)
    sc = dict(momentum=0.95, fast_beta=0.85, fast_weight=0.4385, slow_beta=0.98)
    dev = torch.device("cuda")
    bank = A.Bank(torch.from_numpy(grad).to(dev), torch.from_numpy(vel).to(dev),
                  torch.empty(shape, dtype=torch.bfloat16, device=dev), **sc)
    A.multi_bank_step([bank], A.alloc_workspace([shape]))
    t = A.Tail(bank.out, bank.velocity, to_dev(le), to_dev(p), torch.from_numpy(mt.view(np.int16)).cuda(),
               to_dev(lr), 0.1, 0.95)
    A.update_tail([t], torch.empty(A.tail_workspace_bytes([shape]), dtype=torch.uint8, device=dev))
    torch.cuda.synchronize()
    out_o, vel_o = oracle.bank_step(grad, vel, **sc)
    p_o, mt_o, le_o, _ = oracle.update_tail(out_o, le, 0.95, p, mt, vel_o[1], 0.1, lr)
    w0 = master(p, mt)
    dg = master(t.param.view(torch.int16).cpu().numpy().view(np.uint16),
                t.mantissa.cpu().numpy().view(np.uint16)) - w0
    do = master(p_o, mt_o) - w0
    for i in range(shape[0]):
        assert np.linalg.norm(dg[i] - do[i]) <= 1e-2 * np.linalg.norm(do[i])
    np.testing.assert_allclose(t.lane_energy.cpu().numpy(), le_o, rtol=2e-2)


# --------------------------------------------------------------------------- tail link

LINK_SHAPES = [(4, 256, 768), (3, 1000, 264), (2, 520, 520), (3, 300, 130), (2, 130, 300)]


def linked_step(A, shape, seed, link=True):
    grad, vel = W.random_case(seed, *shape)
    sc = dict(momentum=0.95, fast_beta=0.85, fast_weight=0.4385, slow_beta=0.98)
    dev = torch.device("cuda")
    bank = A.Bank(torch.from_numpy(grad).to(dev), torch.from_numpy(vel).to(dev),
                  torch.empty(shape, dtype=torch.bfloat16, device=dev), **sc,
                  tail_link=A.alloc_tail_link(shape) if link else None)
    A.multi_bank_step([bank], A.alloc_workspace([shape]))
    return bank, grad, vel, sc


@pytest.mark.parametrize("shape", LINK_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_linked_step_then_tail_matches_oracle(A, shape):
    """The step writes the tail link (the slow rail's sign bits) and the tail reads them
    instead of the fp32 rail: the parameter moves as the oracle's whole bank update within
    the cascade's 1e-2 bar, and equals the unlinked tail on the same step output bit for
    bit (the gates are the same, the lane powers are computed the same way)."""
    bank, grad, vel, sc = linked_step(A, shape, 41 + shape[1])
    _, _, le, p, mt, lr = tail_inputs(41, *shape)
    dev = torch.device("cuda")
    ws = torch.empty(A.tail_workspace_bytes([shape]), dtype=torch.uint8, device=dev)

    def tail(link):
        t = A.Tail(bank.out, bank.velocity, to_dev(le), to_dev(p), torch.from_numpy(mt.view(np.int16)).cuda(),
                   to_dev(lr), 0.1, 0.95, tail_link=bank.tail_link if link else None)
        A.update_tail([t], ws)
        torch.cuda.synchronize()
        return (t.param.view(torch.int16).cpu().numpy().view(np.uint16), t.mantissa.cpu().numpy().view(np.uint16),
                t.lane_energy.cpu().numpy())
    p_l, mt_l, le_l = tail(True)
    p_u, mt_u, le_u = tail(False)
    assert A.device_error() == A.OK
    np.testing.assert_array_equal(le_l, le_u)
    np.testing.assert_array_equal(p_l, p_u)
    np.testing.assert_array_equal(mt_l, mt_u)
    out_o, vel_o = oracle.bank_step(grad, vel, **sc)
    p_o, mt_o, le_o, _ = oracle.update_tail(out_o, le, 0.95, p, mt, vel_o[1], 0.1, lr)
    w0 = master(p, mt)
    dg, do = master(p_l, mt_l) - w0, master(p_o, mt_o) - w0
    for i in range(shape[0]):
        assert np.linalg.norm(dg[i] - do[i]) <= 1e-2 * np.linalg.norm(do[i])
    np.testing.assert_allclose(le_l, le_o, rtol=2e-2)


@pytest.mark.parametrize("n", [36, 40])
def test_link_gate_on_zero_tiny_and_huge_values(A, n):
    """The decay gate [slow rail * w >= 0] from the link's sign bits equals the one computed
    from the fp32 rail on every element, where the rail is zero, subnormal or huge and the
    master weight is zero, negative zero, tiny or huge (the cases the link sends back to the
    fp32 rail): bit-identical.  n = 36 takes the apply's element-by-element path, n = 40
    its 16-byte chunk path (vector layout)."""
    g, m = 2, 64
    rng = np.random.default_rng(77)
    grad = (rng.standard_normal((g, m, n)) * 0.02).astype(np.float32)
    vel = np.zeros((2, g, m, n), np.float32)
    # the slow rail after the step: exactly zero, subnormal, huge (fast_weight = 1, so the
    # cascade reads the fast rail only and stays finite)
    grad[0, :16] = 0.0
    vel[1, 0, 8:16] = np.float32(3e-39) * np.sign(rng.standard_normal((8, n)))
    vel[1, 1, :4] = np.float32(3e38) * np.sign(rng.standard_normal((4, n)))
    dev = torch.device("cuda")
    sc = dict(momentum=0.95, fast_beta=0.85, fast_weight=1.0, slow_beta=0.98)
    bank = A.Bank(torch.from_numpy(grad).to(dev), torch.from_numpy(vel).to(dev),
                  torch.empty((g, m, n), dtype=torch.bfloat16, device=dev), **sc,
                  tail_link=A.alloc_tail_link((g, m, n)))
    A.multi_bank_step([bank], A.alloc_workspace([(g, m, n)]))
    torch.cuda.synchronize()
    w = (rng.standard_normal((g, m, n)) * 0.05).astype(np.float32)
    w[:, :, 0] = 0.0
    w[:, :, 1] = -0.0
    w[:, :, 2] = np.float32(1e-20) * np.sign(rng.standard_normal((g, m)))
    w[:, :, 3] = np.float32(1e30)
    bits = w.view(np.uint32)
    p = (bits >> 16).astype(np.uint16)
    mt = (bits & 0xFFFF).astype(np.uint16)
    le = np.zeros((g, m), np.float32)
    lr = np.full(g, 0.02, np.float32)
    ws = torch.empty(A.tail_workspace_bytes([(g, m, n)]), dtype=torch.uint8, device=dev)
    res = []
    for link in (True, False):
        t = A.Tail(bank.out, bank.velocity, to_dev(le), to_dev(p), torch.from_numpy(mt.view(np.int16)).cuda(),
                   to_dev(lr), 0.5, 0.95, tail_link=bank.tail_link if link else None)
        A.update_tail([t], ws)
        torch.cuda.synchronize()
        res.append((t.param.view(torch.int16).cpu().numpy(), t.mantissa.cpu().numpy(), t.lane_energy.cpu().numpy()))
    assert A.device_error() == A.OK
    for a, b in zip(*res):
        np.testing.assert_array_equal(a, b)


def test_linked_tail_over_banks_equals_unlinked(A):
    """One linked tail call over banks of several shapes in the vector layout (lanes along
    rows and along columns, rows of 8 to 6144 elements) equals the unlinked tail of each
    bank alone, bit for bit."""
    shapes = [(4, 256, 768), (3, 1000, 264), (2, 5, 8), (1, 5, 6144), (2, 70, 64), (2, 900, 800)]
    dev = torch.device("cuda")
    steps = [linked_step(A, s, 900 + j) for j, s in enumerate(shapes)]
    ins = [tail_inputs(950 + j, *s) for j, s in enumerate(shapes)]

    def tails(link):
        return [A.Tail(b.out, b.velocity, to_dev(le), to_dev(p), torch.from_numpy(mt.view(np.int16)).cuda(),
                       to_dev(lr), 0.1, 0.95, tail_link=b.tail_link if link else None)
                for (b, _, _, _), (_, _, le, p, mt, lr) in zip(steps, ins)]
    grouped = tails(True)
    A.update_tail(grouped, torch.empty(A.tail_workspace_bytes(shapes), dtype=torch.uint8, device=dev))
    solo = tails(False)
    for t, s in zip(solo, shapes):
        A.update_tail([t], torch.empty(A.tail_workspace_bytes([s]), dtype=torch.uint8, device=dev))
    torch.cuda.synchronize()
    assert A.device_error() == A.OK
    for a, b in zip(grouped, solo):
        assert torch.equal(a.param.view(torch.int16), b.param.view(torch.int16))
        assert torch.equal(a.mantissa, b.mantissa)
        assert torch.equal(a.lane_energy, b.lane_energy)


# --------------------------------------------------------------------------- Adam

@pytest.mark.parametrize("count,offset", [(1 << 20, 0), (1000003, 0), (4096, 1)])
def test_adam_step_matches_oracle_bitwise(A, count, offset):
    """Same fp32 operations in the same order on both sides: identical bits.  The offset
    case starts the buffers one float off 16-byte alignment (scalar path)."""
    rng = np.random.default_rng(count)
    p = (rng.standard_normal(count) * 0.1).astype(np.float32)
    g = (rng.standard_normal(count) * 0.01).astype(np.float32)
    m = (rng.standard_normal(count) * 0.01).astype(np.float32)
    v = (np.abs(rng.standard_normal(count)) * 1e-4).astype(np.float32)
    args = (0.9, 0.95, 1e-8, 0.0123, 0.0004)
    want = oracle.adam_step(p, g, m, v, *args)
    dev = [torch.zeros(count + offset, dtype=torch.float32, device="cuda") for _ in range(4)]
    views = [d[offset:] for d in dev]
    for d, x in zip(views, (p, g, m, v)):
        d.copy_(torch.from_numpy(x))
    for _ in range(1):
        A.adam_step(views[0], views[1], views[2], views[3], *args)
    torch.cuda.synchronize()
    for got, w in zip((views[0], views[2], views[3]), want):
        np.testing.assert_array_equal(got.cpu().numpy(), w)
