"""Host-side checks of libanvil's C ABI that need no GPU: the library loads, exports
every function include/anvil.h declares, holds the page's ANVIL_MAPS, and rejects bad
arguments with the documented status before it makes any CUDA call.  Every call here
fails validation (the pointers are fake), so nothing reaches a GPU even where one is
present."""
import ctypes

import numpy as np
import pytest

anvil = pytest.importorskip("polynomial_matrix_whitening_gb300.anvil",
                            reason="libanvil.so not built")
L = anvil.library()


def test_exports_every_declared_symbol():
    names = anvil.header_functions()
    assert len(names) >= 11
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_default_maps_are_the_page_maps(constants):
    maps, _ = constants
    got = np.array(anvil.default_maps(), np.float32)
    np.testing.assert_array_equal(got, np.array(maps, np.float32))


def test_status_strings():
    for code, name in anvil.STATUS.items():
        assert L.anvil_status_string(code).decode() == name


def _call(descs, maps=None, nmaps=6, ws=1 << 40, ws_bytes=1 << 40, margin=1.05, eps=1e-6):
    arr = (anvil.BankDesc * len(descs))(*descs)
    if maps is None:
        marr, nm = anvil._maps_arg(None)
    else:
        marr, nm = maps, nmaps
    return L.anvil_multi_bank_step(arr, len(descs), None, marr, nm if maps is None else nmaps,
                                   margin, eps, ws, ws_bytes, None)


G = 1 << 32  # fake, aligned device addresses far apart


def d(g=2, m=40, n=24, grad=G, vel=2 * G, out=3 * G, grad_bf16=0, link=None):
    desc = anvil._raw_desc(g, m, n, grad, vel, out, grad_bf16)
    desc.tail_link = link
    return desc


def test_workspace_bytes():
    assert anvil.workspace_bytes([(2, 40, 24)]) > 0
    assert anvil.workspace_bytes([(0, 40, 24)]) == 0
    one = anvil.workspace_bytes([(22, 256, 768)])
    two = anvil.workspace_bytes([(22, 256, 768), (22, 2816, 768)])
    assert two > one
    # tall and wide of the same shape need the same scratch (small-side-major layout)
    assert anvil.workspace_bytes([(3, 300, 130)]) == anvil.workspace_bytes([(3, 130, 300)])


@pytest.mark.parametrize("desc,code", [
    (dict(grad=0), anvil.ERR_INVALID_ARG),
    (dict(vel=0), anvil.ERR_INVALID_ARG),
    (dict(out=0), anvil.ERR_INVALID_ARG),
    (dict(g=0), anvil.ERR_INVALID_ARG),
    (dict(m=0), anvil.ERR_INVALID_ARG),
    (dict(n=-1), anvil.ERR_INVALID_ARG),
    (dict(m=20000), anvil.ERR_UNSUPPORTED_SHAPE),
    (dict(g=65535, m=16384, n=16384), anvil.ERR_UNSUPPORTED_SHAPE),  # 2^44 elements
    (dict(grad=G + 2), anvil.ERR_ALIGNMENT),
    (dict(grad=G + 1, grad_bf16=1), anvil.ERR_ALIGNMENT),
    (dict(out=3 * G + 1), anvil.ERR_ALIGNMENT),
    (dict(out=G), anvil.ERR_ALIAS),            # out == grad
    (dict(out=2 * G + 4), anvil.ERR_ALIAS),    # out inside velocity
    (dict(vel=G + 64), anvil.ERR_ALIAS),       # velocity overlaps grad
    (dict(link=4 * G + 16), anvil.ERR_ALIGNMENT),  # the tail link wants 256-byte alignment
    (dict(link=3 * G), anvil.ERR_ALIAS),       # tail link over out
    (dict(link=2 * G - 256), anvil.ERR_ALIAS),  # tail link running into the velocity
])
def test_argument_errors(desc, code):
    assert _call([d(**desc)]) == code


def test_tail_link_bytes():
    """The step-to-tail link: two 64-bit words (the slow rail's sign bits, the bits that
    send the tail to the fp32 rail) per 64 columns of every row, rounded up to 256 bytes."""
    assert anvil.tail_link_bytes((0, 4, 4)) == 0
    assert anvil.tail_link_bytes((1, 20000, 4)) == 0
    for g, m, n in [(22, 2816, 768), (22, 768, 768), (3, 130, 300), (2, 5, 3)]:
        words = 16 * g * m * -(-n // 64)
        assert anvil.tail_link_bytes((g, m, n)) == -(-words // 256) * 256


def test_alias_across_banks_and_workspace():
    a = d()
    b = d(grad=4 * G, vel=5 * G, out=2 * G + 128)  # bank 2 writes into bank 1's velocity
    assert _call([a, b]) == anvil.ERR_ALIAS
    assert _call([d()], ws=2 * G) == anvil.ERR_ALIAS  # workspace over the velocity


def test_map_and_bank_count_errors():
    marr, _ = anvil._maps_arg(None)
    assert _call([d()], maps=marr, nmaps=0) == anvil.ERR_INVALID_ARG
    big = (anvil.Map * 17)()
    assert _call([d()], maps=big, nmaps=17) == anvil.ERR_INVALID_ARG
    descs = [d(grad=(10 + 3 * i) * G, vel=(11 + 3 * i) * G, out=(12 + 3 * i) * G) for i in range(9)]
    assert _call(descs) == anvil.ERR_INVALID_ARG


def test_workspace_errors():
    need = anvil.workspace_bytes([(2, 40, 24)])
    assert _call([d()], ws=0) == anvil.ERR_WORKSPACE
    assert _call([d()], ws=7 * G, ws_bytes=need - 1) == anvil.ERR_WORKSPACE
    assert _call([d()], ws=7 * G + 128, ws_bytes=need) == anvil.ERR_ALIGNMENT


def test_adam_argument_errors():
    f = L.anvil_adam_step
    ok = dict(p=G, g=2 * G, m=3 * G, v=4 * G)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["p"], a["g"], a["m"], a["v"], kw.get("count", 100), 0.9, 0.95, 1e-8, 0.01, 0.0, None)
    assert call(p=0) == anvil.ERR_INVALID_ARG
    assert call(count=0) == anvil.ERR_INVALID_ARG
    assert call(m=3 * G + 2) == anvil.ERR_ALIGNMENT
    assert call(m=G + 64) == anvil.ERR_ALIAS      # exp_avg overlaps the parameter
    assert call(v=2 * G + 8) == anvil.ERR_ALIAS   # exp_avg_sq overlaps the gradient


def test_tail_argument_errors():
    def tail(**kw):
        base = dict(update=G, velocity=2 * G, lane_energy=3 * G, param=4 * G, mantissa=5 * G,
                    eff_lr=6 * G, g=2, m=40, n=24, eff_wd=0.1, beta2=0.95, tail_link=None)
        base.update(kw)
        d = anvil.TailDesc(*[base[k] for k, _ in anvil.TailDesc._fields_])
        return L.anvil_update_tail(ctypes.byref(d), 1, 1 << 40, 1 << 40, None)
    assert tail(update=0) == anvil.ERR_INVALID_ARG
    assert tail(g=0) == anvil.ERR_INVALID_ARG
    assert tail(param=4 * G + 1) == anvil.ERR_ALIGNMENT
    assert tail(mantissa=4 * G + 16) == anvil.ERR_ALIAS   # mantissa over the parameter
    assert tail(lane_energy=2 * G) == anvil.ERR_ALIAS     # state written over the rails
    assert tail(tail_link=7 * G + 128) == anvil.ERR_ALIGNMENT
    assert tail(tail_link=4 * G + 256) == anvil.ERR_ALIAS  # link under the parameter being written


def test_binding_rejects_tensors_the_kernels_cannot_take():
    """The Python binding refuses, before any CUDA call (and whatever python -O strips),
    tensors whose pointers or extents the kernels would trust: host tensors, wrong dtypes
    or shapes, a workspace off the banks' device."""
    import torch
    g, m, n = 2, 8, 4
    grad = torch.zeros((g, m, n))
    vel = torch.zeros((2, g, m, n))
    out = torch.zeros((g, m, n), dtype=torch.bfloat16)
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA device"):
        anvil.multi_bank_step([anvil.Bank(grad, vel, out)], ws)
    with pytest.raises(ValueError, match="velocity must be"):
        anvil.multi_bank_step([anvil.Bank(grad, torch.zeros((g, m, n)), out)], ws)
    with pytest.raises(ValueError, match="out must be bf16"):
        anvil.multi_bank_step([anvil.Bank(grad, vel, torch.zeros((g, m, n)))], ws)
    with pytest.raises(ValueError, match="grad must be"):
        anvil.multi_bank_step([anvil.Bank(grad.double(), vel, out)], ws)
    with pytest.raises(ValueError, match="fp32 grads"):
        anvil.bank_step(grad.bfloat16(), vel, out)
    with pytest.raises(ValueError, match="CUDA device"):
        anvil.adam_step(*(torch.zeros(16) for _ in range(4)), 0.9, 0.95, 1e-8, 1e-3, 0.0)
    with pytest.raises(ValueError, match="one size"):
        anvil.adam_step(torch.zeros(16), torch.zeros(8), torch.zeros(16), torch.zeros(16), 0.9, 0.95, 1e-8, 1e-3, 0.0)
    tail = anvil.Tail(out, vel, torch.zeros((g, m)), out.clone(), torch.zeros((g, m, n), dtype=torch.int32),
                      torch.zeros(g), 0.1, 0.9)
    with pytest.raises(ValueError, match="mantissa"):
        anvil.update_tail([tail], ws)
