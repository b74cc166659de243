"""CPU oracle of the ANVIL bank step -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the bench's cpu_baseline /
reference legs may import this package.  It shares no code with the CUDA
library: the arithmetic lives in ``anvil_oracle.c`` (plain C, bf16 emulated in
software, fp32 with one rounding per operation, sequential k-order sums) and
this module only marshals numpy arrays to it.

What it computes is the page "modded-nanogpt track_1_short/optim/anvil.py",
function ``anvil_cascade`` and the constants above it (ANVIL_MAPS, the rail
betas and weight, FROBENIUS_MARGIN / FROBENIUS_EPS); see the C file's header
for the step list.  Every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, library routines); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# ANVIL_ORACLE_SRC / ANVIL_ORACLE_BUILD let the mutation test build a planted copy elsewhere.
_SRC = os.environ.get("ANVIL_ORACLE_SRC", os.path.join(_HERE, "anvil_oracle.c"))
_LIB_DIR = os.environ.get("ANVIL_ORACLE_BUILD", os.path.join(_HERE, "_build"))
_LIB = os.path.join(_LIB_DIR, "liboracle.so")

# ANVIL_MAPS as printed on the page (anvil.py, the ANVIL section: six quintic
# spectral maps (a, b, c), record #360).
ANVIL_MAPS = (
    (3.923798038567, -6.095026865488, 3.905234618423),
    (3.278126713798, -3.328923386476, 0.989127286973),
    (3.505298394150, -5.137358782410, 1.968325560615),
    (2.815058591845, -3.685181239622, 1.417196497642),
    (2.245503932403, -2.443826979899, 0.963091710461),
    (2.256537145403, -2.166840097229, 0.929501253245),
)
FROBENIUS_MARGIN = 1.05
FROBENIUS_EPS = 1e-6

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (portable flags: no -march, no FMA contraction)."""
    with _lock:
        fresh = os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)
        if fresh and not force:
            return _LIB
        os.makedirs(_LIB_DIR, exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O3", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


class _Trace(ctypes.Structure):
    _fields_ = [("A0", ctypes.c_void_p), ("X", ctypes.c_void_p), ("A", ctypes.c_void_p),
                ("B", ctypes.c_void_p), ("d", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        path = build()
        L = ctypes.CDLL(path)
        vp, i, f, l = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_long
        L.oracle_f32_to_bf16.argtypes = [vp, vp, l]
        L.oracle_momentum.argtypes = [vp, vp, vp, l, f, f, f, f, vp, vp]
        L.oracle_cascade.argtypes = [vp, i, i, vp, i, f, f, i, vp, ctypes.POINTER(_Trace)]
        L.oracle_cascade.restype = i
        L.oracle_cascade_f64.argtypes = [vp, i, i, vp, i, ctypes.c_double, ctypes.c_double, vp]
        L.oracle_cascade_f64.restype = i
        L.oracle_bank_step.argtypes = [vp, vp, i, i, i, f, f, f, f, vp, i, f, f, i, vp]
        L.oracle_bank_step.restype = i
        L.oracle_rail_equalizer.argtypes = [vp, i, i, i, vp, f, vp]
        L.oracle_sign_aligned_decay.argtypes = [vp, vp, vp, vp, i, l, f, vp]
        L.oracle_adam_step.argtypes = [vp, vp, vp, vp, l, f, f, f, f, f]
        L.oracle_num_threads.restype = i
        L.oracle_set_num_threads.argtypes = [i]
        _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _maps32(maps):
    return np.ascontiguousarray(np.asarray(maps, np.float64).reshape(-1, 3), np.float32)


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


def f32_to_bf16(x) -> np.ndarray:
    """bf16 bits (uint16) of fp32 values, round to nearest even."""
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_f32_to_bf16(_ptr(x), _ptr(out), x.size)
    return out


def bf16_to_f32(h) -> np.ndarray:
    """fp32 values of bf16 bits (exact: the bits become the top half of a binary32)."""
    h = np.ascontiguousarray(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def momentum(grad, velocity, momentum, fast_beta, fast_weight, slow_beta):
    """Twin-rail Nesterov momentum.

    grad [...] fp32; velocity [2, ...] fp32 (rail 0 fast, rail 1 slow).
    Returns (X bf16 bits, g fp32 lookahead, new velocity); inputs untouched.
    """
    grad = np.ascontiguousarray(grad, np.float32)
    vel = np.array(velocity, np.float32, copy=True, order="C")
    if vel.shape != (2,) + grad.shape:
        raise ValueError("velocity must be [2, g, m, n]")
    g = np.empty_like(grad)
    X = np.empty(grad.shape, np.uint16)
    lib().oracle_momentum(_ptr(grad), _ptr(vel[0]), _ptr(vel[1]), grad.size, momentum,
                          fast_beta, fast_weight, slow_beta, _ptr(g), _ptr(X))
    return X, g, vel


def cascade(X_bits, maps=ANVIL_MAPS, margin=FROBENIUS_MARGIN, eps=FROBENIUS_EPS, split=False,
            trace=False):
    """Normalisation + quintic cascade of one bf16 matrix [rows, cols] (bits in, bits out).

    With trace=True also returns a dict of per-stage bf16 bits in the page's layout:
    A0 [s,s] (first Gram, unnormalised), X [nmaps+1, rows, cols] (normalised X, then
    after each map), A / B [nmaps, s, s] per map, and d (fp32).
    """
    X_bits = np.ascontiguousarray(X_bits, np.uint16)
    rows, cols = X_bits.shape
    m = _maps32(maps)
    out = np.empty_like(X_bits)
    tr = None
    t = None
    if trace:
        s = min(rows, cols)
        k = m.shape[0]
        t = {"A0": np.empty((s, s), np.uint16), "X": np.empty((k + 1, rows, cols), np.uint16),
             "A": np.empty((k, s, s), np.uint16), "B": np.empty((k, s, s), np.uint16),
             "d": np.empty(1, np.float32)}
        tr = _Trace(*(t[n].ctypes.data for n in ("A0", "X", "A", "B", "d")))
    rc = lib().oracle_cascade(_ptr(X_bits), rows, cols, _ptr(m), m.shape[0], margin, eps,
                              int(split), _ptr(out), ctypes.byref(tr) if tr is not None else None)
    if rc != 0:
        raise MemoryError("oracle_cascade")
    return (out, t) if trace else out


def cascade_f64(X, maps=ANVIL_MAPS, margin=FROBENIUS_MARGIN, eps=FROBENIUS_EPS):
    """The same iteration in fp64 with no rounding (input fp64 [rows, cols])."""
    X = np.ascontiguousarray(X, np.float64)
    rows, cols = X.shape
    m = np.ascontiguousarray(np.asarray(maps, np.float64).reshape(-1, 3))
    out = np.empty_like(X)
    rc = lib().oracle_cascade_f64(_ptr(X), rows, cols, _ptr(m), m.shape[0], margin, eps, _ptr(out))
    if rc != 0:
        raise MemoryError("oracle_cascade_f64")
    return out


def bank_step(grad, velocity, momentum, fast_beta, fast_weight, slow_beta, maps=ANVIL_MAPS,
              margin=FROBENIUS_MARGIN, eps=FROBENIUS_EPS, split=False):
    """One ANVIL bank step: grad [g, m, n] fp32, velocity [2, g, m, n] fp32.

    Returns (out bf16 bits [g, m, n], new velocity); the inputs are not modified.
    """
    grad = np.ascontiguousarray(grad, np.float32)
    g, rows, cols = grad.shape
    vel = np.array(velocity, np.float32, copy=True, order="C")
    if vel.shape != (2, g, rows, cols):
        raise ValueError("velocity must be [2, g, m, n]")
    m = _maps32(maps)
    out = np.empty(grad.shape, np.uint16)
    rc = lib().oracle_bank_step(_ptr(grad), _ptr(vel), g, rows, cols, momentum, fast_beta,
                                fast_weight, slow_beta, _ptr(m), m.shape[0], margin, eps,
                                int(split), _ptr(out))
    if rc != 0:
        raise MemoryError("oracle_bank_step")
    return out, vel


def rail_equalizer(v_bits, lane_energy, beta2):
    """The equaliser on a bank of bf16 updates v [g, rows, cols]: returns (v_eq bits,
    new lane_energy).  lane_energy: fp32 [g, rows] if rows >= cols else [g, cols]."""
    v_bits = np.ascontiguousarray(v_bits, np.uint16)
    g, rows, cols = v_bits.shape
    le = np.array(lane_energy, np.float32, copy=True, order="C")
    if le.shape != (g, rows if rows >= cols else cols):
        raise ValueError("lane_energy must be [g, max(rows, cols)]")
    out = np.empty_like(v_bits)
    lib().oracle_rail_equalizer(_ptr(v_bits), g, rows, cols, _ptr(le), beta2, _ptr(out))
    return out, le


def sign_aligned_decay(p_bits, mantissa, update_bits, gate, wd, lr):
    """Decay + update of the fp32 master weight (bf16 bits p, uint16 mantissa), per matrix
    learning rates lr [g]; gate fp32 (the slow rail).  Returns (new p bits, new mantissa)."""
    p = np.array(p_bits, np.uint16, copy=True, order="C")
    mt = np.array(mantissa, np.uint16, copy=True, order="C")
    u = np.ascontiguousarray(update_bits, np.uint16)
    gt = np.ascontiguousarray(gate, np.float32)
    lr = np.ascontiguousarray(lr, np.float32)
    g = p.shape[0]
    if not (lr.shape == (g,) and p.shape == mt.shape == u.shape == gt.shape):
        raise ValueError("lr [g] and p, mantissa, update, gate of one shape")
    lib().oracle_sign_aligned_decay(_ptr(p), _ptr(mt), _ptr(u), _ptr(gt), g, p[0].size, wd, _ptr(lr))
    return p, mt


def update_tail(v_bits, lane_energy, beta2, p_bits, mantissa, gate, wd, lr):
    """The page's tail of anvil_bank_update: equaliser, then sign-aligned decay update."""
    v_eq, le = rail_equalizer(v_bits, lane_energy, beta2)
    p, mt = sign_aligned_decay(p_bits, mantissa, v_eq, gate, wd, lr)
    return p, mt, le, v_eq


def adam_step(p, g, exp_avg, exp_avg_sq, beta1, beta2, eps, step_size, eff_wd):
    """The page's Adam step with cautious weight decay (fp32, elementwise).
    Returns (p, exp_avg, exp_avg_sq) as new arrays."""
    p = np.array(p, np.float32, copy=True, order="C")
    m = np.array(exp_avg, np.float32, copy=True, order="C")
    v = np.array(exp_avg_sq, np.float32, copy=True, order="C")
    g = np.ascontiguousarray(g, np.float32)
    if not (p.shape == g.shape == m.shape == v.shape):
        raise ValueError("param, grad, exp_avg, exp_avg_sq of one shape")
    lib().oracle_adam_step(_ptr(p), _ptr(g), _ptr(m), _ptr(v), p.size, beta1, beta2, eps, step_size,
                           eff_wd)
    return p, m, v
