"""The fixed-scratch entry point, anvil_bank_step_noalloc, against anvil_bank_step.

anvil_bank_step_noalloc exists for callers that cannot allocate device memory from the
code that runs the step (memory owned by their own pool, graph capture in progress on
another thread, or no device-synchronising calls allowed); it keeps its scratch in a
fixed array the library declares on every GPU.  This file is collected last on
purpose, so a run that stops at the first failure has run every other test first; it
also passes when run on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from polynomial_matrix_whitening_gb300 import workloads as W  # noqa: E402

OUT_RTOL = 1e-2   # relative Frobenius error per matrix against the oracle, as in the parity tests


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from polynomial_matrix_whitening_gb300 import anvil
    return anvil


def _call(fn, grad, vel, out, sc):
    g, m, n = grad.shape
    return fn(ctypes.c_void_p(grad.data_ptr()), ctypes.c_void_p(vel.data_ptr()), g, m, n,
              sc[0], sc[1], sc[2], sc[3], None, 0, 1.05, 1e-6, ctypes.c_void_p(out.data_ptr()),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("shape", [(3, 300, 130), (22, 256, 768), (2, 130, 1000)])
def test_noalloc_matches_bank_step_twice(A, shape):
    """Both entry points run the same kernels on the same layout, so their rails and outputs
    must be equal bit for bit, on two calls in a row (the second sees whatever the first
    left in the fixed scratch); the ragged shape is also checked against the oracle."""
    lib = A.library()
    dev = torch.device("cuda")
    sc = (0.95, 0.85, 0.4385, 0.98)
    for call in range(2):
        grad, vel = W.random_case(700 + 10 * call + shape[1], *shape)
        g_d = torch.from_numpy(grad).to(dev)
        v_ref = torch.from_numpy(vel).to(dev)
        v_new = v_ref.clone()
        o_ref = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        o_new = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=dev)
        assert _call(lib.anvil_bank_step, g_d, v_ref, o_ref, sc) == A.OK
        assert _call(lib.anvil_bank_step_noalloc, g_d, v_new, o_new, sc) == A.OK
        torch.cuda.synchronize()
        assert torch.equal(v_new, v_ref), call
        assert torch.equal(o_new.view(torch.int16), o_ref.view(torch.int16)), call
        if shape == (3, 300, 130):
            out_or, vel_or = oracle.bank_step(grad, vel, *sc)
            np.testing.assert_array_equal(v_new.cpu().numpy(), vel_or)
            got = o_new.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
            for i in range(shape[0]):
                x = oracle.bf16_to_f32(got[i]).astype(np.float64)
                r = oracle.bf16_to_f32(out_or[i]).astype(np.float64)
                assert np.isfinite(x).all()
                assert np.linalg.norm(x - r) <= OUT_RTOL * np.linalg.norm(r), (call, i)
    assert A.device_error() == A.OK


def test_noalloc_rejects_sizes_beyond_the_fixed_scratch(A):
    lib = A.library()
    shape = (4, 2816, 768)  # needs about 44.6 MB of scratch
    assert A.workspace_bytes([shape]) > A.STATIC_SCRATCH_BYTES
    dev = torch.device("cuda")
    g_d = torch.zeros(shape, dtype=torch.float32, device=dev)
    v_d = torch.zeros((2,) + shape, dtype=torch.float32, device=dev)
    o_d = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    assert _call(lib.anvil_bank_step_noalloc, g_d, v_d, o_d, (0.95, 0.85, 0.4385, 0.98)) \
        == A.ERR_WORKSPACE
    assert b"fixed scratch" in lib.anvil_last_cuda_error()
