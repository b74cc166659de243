"""Thin ctypes binding of libanvil (include/anvil.h), the ANVIL bank step on GB300.

Argument marshalling only: every step of the computation runs in libanvil's CUDA
kernels.  Importing this module loads ``libanvil.so`` from this package directory and
raises ``ImportError`` if it has not been built (``python -c "import __graft_entry__ as
g; g.build()"``, or ``python polynomial_matrix_whitening_gb300/build.py``); there is no
fallback of any kind.

Tensors are torch tensors on the current CUDA device: grad fp32 [g, m, n], velocity
fp32 [2, g, m, n], out bf16 [g, m, n], all contiguous.  Calls are enqueued on
``torch.cuda.current_stream()`` unless a stream is given.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
# ANVIL_LIBRARY=timeline loads the timeline build (build.py --timeline) instead, for the
# cascade timeline tool; the computation is the same.
LIB_PATH = os.path.join(_HERE, "libanvil_timeline.so" if os.environ.get("ANVIL_LIBRARY") == "timeline"
                        else "libanvil.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "anvil.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libanvil.so is not built ({LIB_PATH}); run the package's build.py")

_lib = ctypes.CDLL(LIB_PATH)

STATUS = {0: "ANVIL_OK", 1: "ANVIL_ERR_INVALID_ARG", 2: "ANVIL_ERR_UNSUPPORTED_SHAPE",
          3: "ANVIL_ERR_ALIGNMENT", 4: "ANVIL_ERR_ALIAS", 5: "ANVIL_ERR_WORKSPACE",
          6: "ANVIL_ERR_CUDA", 7: "ANVIL_ERR_TIMEOUT", 8: "ANVIL_ERR_DEVICE", 9: "ANVIL_ERR_UNAVAILABLE"}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_ALIGNMENT, ERR_ALIAS, ERR_WORKSPACE, \
    ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE, ERR_UNAVAILABLE = range(10)
KERNEL_KINDS = ("momentum", "norm_d", "normalize", "gram_norm", "gram", "sqpoly", "xupdate",
                "xupdate_out", "tail_power", "tail_scale", "tail_apply", "adam", "cascade")
MAX_MAPS, MAX_BANKS = 16, 8


class AnvilError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        detail = _lib.anvil_last_cuda_error().decode() if status == ERR_CUDA else ""
        super().__init__(f"{where}: {STATUS.get(status, status)} {detail}".strip())


class Map(ctypes.Structure):
    _fields_ = [("a", ctypes.c_float), ("b", ctypes.c_float), ("c", ctypes.c_float)]


class Scalars(ctypes.Structure):
    _fields_ = [("momentum", ctypes.c_float), ("fast_beta", ctypes.c_float),
                ("fast_weight", ctypes.c_float), ("slow_beta", ctypes.c_float)]


class BankDesc(ctypes.Structure):
    _fields_ = [("grad", ctypes.c_void_p), ("velocity", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("g", ctypes.c_int), ("m", ctypes.c_int), ("n", ctypes.c_int),
                ("scalars", Scalars), ("grad_bf16", ctypes.c_int), ("tail_link", ctypes.c_void_p)]


class Trace(ctypes.Structure):
    _fields_ = [("X_raw", ctypes.c_void_p), ("d", ctypes.c_void_p), ("X", ctypes.c_void_p),
                ("A", ctypes.c_void_p), ("B", ctypes.c_void_p)]


class TailDesc(ctypes.Structure):
    _fields_ = [("update", ctypes.c_void_p), ("velocity", ctypes.c_void_p),
                ("lane_energy", ctypes.c_void_p), ("param", ctypes.c_void_p),
                ("mantissa", ctypes.c_void_p), ("eff_lr", ctypes.c_void_p),
                ("g", ctypes.c_int), ("m", ctypes.c_int), ("n", ctypes.c_int),
                ("eff_wd", ctypes.c_float), ("beta2", ctypes.c_float), ("tail_link", ctypes.c_void_p)]


class ScheduleRun(ctypes.Structure):
    _fields_ = [("phase", ctypes.c_int), ("op", ctypes.c_int), ("bank", ctypes.c_int), ("mat0", ctypes.c_int),
                ("nmat", ctypes.c_int), ("begin", ctypes.c_int), ("tiles", ctypes.c_int)]


class ProfileRecord(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("ms", ctypes.c_float)]


_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_lib.anvil_default_maps.argtypes = [ctypes.POINTER(Map), _i]
_lib.anvil_default_maps.restype = _i
_lib.anvil_workspace_bytes.argtypes = [ctypes.POINTER(BankDesc), _i]
_lib.anvil_workspace_bytes.restype = _sz
_lib.anvil_multi_bank_step.argtypes = [ctypes.POINTER(BankDesc), _i, _vp, ctypes.POINTER(Map), _i,
                                       _f, _f, _vp, _sz, _vp]
_lib.anvil_multi_bank_step.restype = _i
_lib.anvil_bank_step.argtypes = [_vp, _vp, _i, _i, _i, _f, _f, _f, _f, ctypes.POINTER(Map), _i,
                                 _f, _f, _vp, _vp]
_lib.anvil_bank_step.restype = _i
_lib.anvil_bank_step_noalloc.argtypes = _lib.anvil_bank_step.argtypes
_lib.anvil_bank_step_noalloc.restype = _i
_lib.anvil_bank_step_traced.argtypes = [ctypes.POINTER(BankDesc), _vp, ctypes.POINTER(Map), _i,
                                        _f, _f, _vp, _sz, ctypes.POINTER(Trace), _vp]
_lib.anvil_bank_step_traced.restype = _i
_lib.anvil_tail_link_bytes.argtypes = [_i, _i, _i]
_lib.anvil_tail_link_bytes.restype = _sz
_lib.anvil_tail_workspace_bytes.argtypes = [ctypes.POINTER(TailDesc), _i]
_lib.anvil_tail_workspace_bytes.restype = _sz
_lib.anvil_update_tail.argtypes = [ctypes.POINTER(TailDesc), _i, _vp, _sz, _vp]
_lib.anvil_update_tail.restype = _i
_lib.anvil_adam_step.argtypes = [_vp, _vp, _vp, _vp, _sz, _f, _f, _f, _f, _f, _vp]
_lib.anvil_adam_step.restype = _i
_lib.anvil_device_error.argtypes = [_i]
_lib.anvil_device_error.restype = _i
_lib.anvil_last_device_error.argtypes = [_vp]
_lib.anvil_last_device_error.restype = _i
_lib.anvil_selftest_wait_timeout.argtypes = [ctypes.c_uint, _vp]
_lib.anvil_selftest_wait_timeout.restype = _i
_lib.anvil_profile_begin.argtypes = [_i]
_lib.anvil_profile_begin.restype = _i
_lib.anvil_profile_end.argtypes = [ctypes.POINTER(ProfileRecord), _i]
_lib.anvil_profile_end.restype = _i
_lib.anvil_schedule_runs.argtypes = [ctypes.POINTER(BankDesc), _i, _i, ctypes.POINTER(ScheduleRun), _i]
_lib.anvil_schedule_runs.restype = _i
_lib.anvil_timeline_read.argtypes = [_vp, _sz]
_lib.anvil_timeline_read.restype = _i
_lib.anvil_timeline_clear.argtypes = []
_lib.anvil_timeline_clear.restype = _i
_lib.anvil_status_string.argtypes = [_i]
_lib.anvil_status_string.restype = ctypes.c_char_p
_lib.anvil_last_cuda_error.restype = ctypes.c_char_p


def library():
    """The loaded ctypes CDLL (for tests that call the C ABI directly)."""
    return _lib


def header_functions(path: str = HEADER):
    """Names of the functions include/anvil.h declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(anvil_[a-z0-9_]+)\s*\(", text)))


def _check(status, where):
    if status != OK:
        raise AnvilError(status, where)


def default_maps():
    """The page's six ANVIL_MAPS as (a, b, c) fp32 triples, as the library holds them."""
    arr = (Map * 6)()
    _lib.anvil_default_maps(arr, 6)
    return [(m.a, m.b, m.c) for m in arr]


def _maps_arg(maps):
    if maps is None:
        maps = default_maps()
    maps = list(maps)
    arr = (Map * len(maps))(*[Map(*[float(x) for x in m]) for m in maps])
    return arr, len(maps)


def _stream_arg(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _require(cond, what):
    """Argument check that survives python -O: the kernels trust every pointer and extent
    they are given, so a wrong tensor must stop here."""
    if not cond:
        raise ValueError(what)


def _on_one_gpu(tensors, what):
    _require(all(t.is_cuda for t in tensors), f"{what}: every tensor must be on a CUDA device")
    _require(len({t.device for t in tensors}) == 1, f"{what}: every tensor must be on the same device")
    _require(all(t.is_contiguous() for t in tensors), f"{what}: every tensor must be contiguous")


def _link_arg(link, g, m, n, ref):
    """Device pointer of a tail-link buffer (uint8 tensor of tail_link_bytes, on ref's GPU)."""
    if link is None:
        return None
    import torch
    _require(link.dtype == torch.uint8 and link.dim() == 1, "tail_link must be a 1-D uint8 tensor")
    _on_one_gpu((link, ref), "tail_link")
    _require(link.numel() >= tail_link_bytes((g, m, n)), "tail_link smaller than tail_link_bytes")
    _require(link.data_ptr() % 256 == 0, "tail_link not 256-byte aligned")
    return link.data_ptr()


def tail_link_bytes(shape):
    """Bytes of the step-to-tail link buffer of one bank of this (g, m, n) shape."""
    return int(_lib.anvil_tail_link_bytes(*[int(x) for x in shape]))


def alloc_tail_link(shape, device=None):
    """A step-to-tail link buffer for one bank (uint8 tensor, 256-byte aligned)."""
    import torch
    t = torch.empty(tail_link_bytes(shape), dtype=torch.uint8, device=device or "cuda")
    _require(t.data_ptr() % 256 == 0, "tail_link not 256-byte aligned")
    return t


def _desc(grad, velocity, out, scalars=None, tail_link=None):
    import torch
    _require(grad.dtype in (torch.float32, torch.bfloat16), "grad must be fp32 or bf16")
    _require(velocity.dtype == torch.float32, "velocity must be fp32")
    _require(out.dtype == torch.bfloat16, "out must be bf16")
    _require(grad.dim() == 3, "grad must be [g, m, n]")
    g, m, n = grad.shape
    _require(tuple(velocity.shape) == (2, g, m, n), "velocity must be [2, g, m, n]")
    _require(tuple(out.shape) == (g, m, n), "out must be [g, m, n]")
    _on_one_gpu((grad, velocity, out), "bank")
    s = scalars or {}
    return BankDesc(grad.data_ptr(), velocity.data_ptr(), out.data_ptr(), g, m, n,
                    Scalars(float(s.get("momentum", 0.95)), float(s.get("fast_beta", 0.85)),
                            float(s.get("fast_weight", 0.4385)), float(s.get("slow_beta", 0.98))),
                    1 if grad.dtype == torch.bfloat16 else 0, _link_arg(tail_link, g, m, n, grad))


def _raw_desc(g, m, n, grad=0, velocity=0, out=0, grad_bf16=0):
    return BankDesc(grad, velocity, out, g, m, n, Scalars(0.95, 0.85, 0.4385, 0.98), grad_bf16, None)


def workspace_bytes(shapes):
    """Workspace bytes for banks of the given (g, m, n) shapes."""
    descs = (BankDesc * len(shapes))(*[_raw_desc(*s) for s in shapes])
    return int(_lib.anvil_workspace_bytes(descs, len(shapes)))


def alloc_workspace(shapes, device=None):
    """A device workspace (uint8 tensor, 256-byte aligned by the caching allocator)."""
    import torch
    nbytes = workspace_bytes(shapes)
    if nbytes == 0:
        raise AnvilError(ERR_INVALID_ARG, "workspace_bytes")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
    _require(ws.data_ptr() % 256 == 0, "workspace not 256-byte aligned")
    return ws


def _workspace_arg(workspace, ref):
    """(pointer, bytes) of a workspace tensor on the same GPU as `ref`."""
    _on_one_gpu((workspace, ref), "workspace")
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


class Bank:
    """One bank of a multi-bank step: grad, velocity, out tensors and host scalars, and an
    optional step-to-tail link buffer (alloc_tail_link) for the update tail of this step."""

    def __init__(self, grad, velocity, out, momentum=0.95, fast_beta=0.85, fast_weight=0.4385,
                 slow_beta=0.98, tail_link=None):
        self.grad, self.velocity, self.out = grad, velocity, out
        self.scalars = dict(momentum=momentum, fast_beta=fast_beta, fast_weight=fast_weight,
                            slow_beta=slow_beta)
        self.tail_link = tail_link

    @property
    def shape(self):
        return tuple(self.grad.shape)

    def desc(self):
        return _desc(self.grad, self.velocity, self.out, self.scalars, self.tail_link)


def multi_bank_step(banks, workspace, maps=None, margin=1.05, eps=1e-6, d_scalars=None,
                    stream=None):
    """One ANVIL step over several banks (three launches: momentum, d, the cascade).

    d_scalars: optional fp32 CUDA tensor [nbanks, 4] (momentum, fast_beta, fast_weight,
    slow_beta) read on the device when the step runs (for CUDA-graph replays).
    """
    descs = (BankDesc * len(banks))(*[b.desc() for b in banks])
    marr, nm = _maps_arg(maps)
    dsp = None
    if d_scalars is not None:
        import torch
        _require(d_scalars.dtype == torch.float32, "d_scalars must be fp32")
        _require(tuple(d_scalars.shape) == (len(banks), 4), "d_scalars must be [nbanks, 4]")
        _on_one_gpu((d_scalars, banks[0].grad), "d_scalars")
        dsp = d_scalars.data_ptr()
    wsp, wsb = _workspace_arg(workspace, banks[0].grad)
    st = _lib.anvil_multi_bank_step(descs, len(banks), dsp, marr, nm, margin, eps, wsp, wsb,
                                    _stream_arg(stream))
    _check(st, "anvil_multi_bank_step")


def bank_step(grad, velocity, out, momentum=0.95, fast_beta=0.85, fast_weight=0.4385,
              slow_beta=0.98, maps=None, margin=1.05, eps=1e-6, stream=None):
    """One bank, host scalars, library-owned workspace (the page's anvil_cascade call)."""
    import torch
    _require(grad.dtype == torch.float32, "anvil_bank_step takes fp32 grads; use multi_bank_step for bf16")
    _desc(grad, velocity, out)
    g, m, n = grad.shape
    marr, nm = (None, 0) if maps is None else _maps_arg(maps)
    st = _lib.anvil_bank_step(grad.data_ptr(), velocity.data_ptr(), g, m, n, momentum, fast_beta,
                              fast_weight, slow_beta, marr, nm, margin, eps, out.data_ptr(),
                              _stream_arg(stream))
    _check(st, "anvil_bank_step")


STATIC_SCRATCH_BYTES = 32 << 20


def bank_step_noalloc(grad, velocity, out, momentum=0.95, fast_beta=0.85, fast_weight=0.4385,
                      slow_beta=0.98, maps=None, margin=1.05, eps=1e-6, stream=None):
    """bank_step with the library's fixed device scratch (no allocation by the call); for
    callers that cannot allocate device memory.  Calls that overlap on the GPU race."""
    import torch
    _require(grad.dtype == torch.float32, "anvil_bank_step_noalloc takes fp32 grads")
    _desc(grad, velocity, out)
    g, m, n = grad.shape
    marr, nm = (None, 0) if maps is None else _maps_arg(maps)
    st = _lib.anvil_bank_step_noalloc(grad.data_ptr(), velocity.data_ptr(), g, m, n, momentum,
                                      fast_beta, fast_weight, slow_beta, marr, nm, margin, eps,
                                      out.data_ptr(), _stream_arg(stream))
    _check(st, "anvil_bank_step_noalloc")


def bank_step_traced(bank: Bank, workspace, maps=None, margin=1.05, eps=1e-6, stream=None):
    """One bank step with per-stage dumps; returns a dict of torch tensors
    (X_raw [g,m,n] bf16, d [g] fp32, X [nmaps+1,g,m,n] bf16, A/B [nmaps,g,s,s] bf16)."""
    import torch
    g, m, n = bank.shape
    s = min(m, n)
    marr, nm = _maps_arg(maps)
    dev = bank.grad.device
    t = {"X_raw": torch.empty((g, m, n), dtype=torch.bfloat16, device=dev),
         "d": torch.empty((g,), dtype=torch.float32, device=dev),
         "X": torch.empty((nm + 1, g, m, n), dtype=torch.bfloat16, device=dev),
         "A": torch.empty((nm, g, s, s), dtype=torch.bfloat16, device=dev),
         "B": torch.empty((nm, g, s, s), dtype=torch.bfloat16, device=dev)}
    tr = Trace(*(t[k].data_ptr() for k in ("X_raw", "d", "X", "A", "B")))
    desc = bank.desc()
    wsp, wsb = _workspace_arg(workspace, bank.grad)
    st = _lib.anvil_bank_step_traced(ctypes.byref(desc), None, marr, nm, margin, eps, wsp, wsb,
                                     ctypes.byref(tr), _stream_arg(stream))
    _check(st, "anvil_bank_step_traced")
    return t


class Tail:
    """One bank of the update tail: the step's out as update, its velocity (rail 1 gates the
    decay), lane_energy [g, m] if m >= n else [g, n] fp32, param (bf16) and mantissa
    (uint16 as torch.int16) [g, m, n], eff_lr [g] fp32, and host eff_wd, beta2; tail_link:
    the link buffer the step that produced update and velocity was given, or None."""

    def __init__(self, update, velocity, lane_energy, param, mantissa, eff_lr, eff_wd, beta2,
                 tail_link=None):
        self.update, self.velocity, self.lane_energy = update, velocity, lane_energy
        self.param, self.mantissa, self.eff_lr = param, mantissa, eff_lr
        self.eff_wd, self.beta2 = float(eff_wd), float(beta2)
        self.tail_link = tail_link

    def desc(self):
        import torch
        _require(self.update.dim() == 3, "update must be [g, m, n]")
        g, m, n = self.update.shape
        _require(self.update.dtype == torch.bfloat16 and self.param.dtype == torch.bfloat16,
                 "update and param must be bf16")
        _require(tuple(self.param.shape) == (g, m, n), "param must be [g, m, n]")
        _require(self.mantissa.dtype in (torch.int16, torch.uint16) and tuple(self.mantissa.shape) == (g, m, n),
                 "mantissa must be 16-bit [g, m, n]")
        _require(tuple(self.velocity.shape) == (2, g, m, n) and self.velocity.dtype == torch.float32,
                 "velocity must be fp32 [2, g, m, n]")
        _require(tuple(self.lane_energy.shape) == (g, m if m >= n else n) and self.lane_energy.dtype == torch.float32,
                 "lane_energy must be fp32 [g, max(m, n)]")
        _require(tuple(self.eff_lr.shape) == (g,) and self.eff_lr.dtype == torch.float32, "eff_lr must be fp32 [g]")
        _on_one_gpu((self.update, self.velocity, self.lane_energy, self.param, self.mantissa, self.eff_lr), "tail")
        return TailDesc(self.update.data_ptr(), self.velocity.data_ptr(), self.lane_energy.data_ptr(),
                        self.param.data_ptr(), self.mantissa.data_ptr(), self.eff_lr.data_ptr(),
                        g, m, n, self.eff_wd, self.beta2, _link_arg(self.tail_link, g, m, n, self.update))


def tail_workspace_bytes(shapes):
    descs = (TailDesc * len(shapes))(*[TailDesc(0, 0, 0, 0, 0, 0, g, m, n, 0.0, 0.0, None)
                                       for g, m, n in shapes])
    return int(_lib.anvil_tail_workspace_bytes(descs, len(shapes)))


def update_tail(tails, workspace, stream=None):
    """The page's update tail (equaliser + sign-aligned decay) over several banks."""
    descs = (TailDesc * len(tails))(*[t.desc() for t in tails])
    wsp, wsb = _workspace_arg(workspace, tails[0].update)
    st = _lib.anvil_update_tail(descs, len(tails), wsp, wsb, _stream_arg(stream))
    _check(st, "anvil_update_tail")


def adam_step(param, grad, exp_avg, exp_avg_sq, beta1, beta2, eps, step_size, eff_wd, stream=None):
    """The page's Adam step with cautious weight decay, in place on fp32 CUDA tensors."""
    import torch
    for t in (param, grad, exp_avg, exp_avg_sq):
        _require(t.dtype == torch.float32 and t.numel() == param.numel(),
                 "adam_step: fp32 tensors of one size")
    _on_one_gpu((param, grad, exp_avg, exp_avg_sq), "adam_step")
    st = _lib.anvil_adam_step(param.data_ptr(), grad.data_ptr(), exp_avg.data_ptr(), exp_avg_sq.data_ptr(),
                              param.numel(), beta1, beta2, eps, step_size, eff_wd, _stream_arg(stream))
    _check(st, "anvil_adam_step")


def schedule_runs(shapes, nmaps=6):
    """The cascade kernel's item order for banks of these (g, m, n) shapes (host only, no
    GPU needed): a list of dicts with phase, op, bank, mat0, nmat, begin, tiles."""
    arr = (BankDesc * len(shapes))(*[_raw_desc(g, m, n) for g, m, n in shapes])
    n = _lib.anvil_schedule_runs(arr, len(shapes), nmaps, None, 0)
    if n < 0:
        raise AnvilError(ERR_INVALID_ARG, "anvil_schedule_runs")
    runs = (ScheduleRun * max(n, 1))()
    _lib.anvil_schedule_runs(arr, len(shapes), nmaps, runs, n)
    return [{f: getattr(r, f) for f, _ in ScheduleRun._fields_} for r in runs[:n]]


TIMELINE_ITEMS, TIMELINE_FIELDS = 16384, 16


def timeline_clear():
    """Zeroes the cascade timeline (timeline build only; AnvilError otherwise)."""
    _check(_lib.anvil_timeline_clear(), "anvil_timeline_clear")


def timeline_read():
    """The cascade timeline as a numpy uint64 array [TIMELINE_ITEMS, TIMELINE_FIELDS]
    (timeline build only; AnvilError otherwise)."""
    import numpy as np
    buf = np.zeros((TIMELINE_ITEMS, TIMELINE_FIELDS), dtype=np.uint64)
    _check(_lib.anvil_timeline_read(buf.ctypes.data, buf.nbytes), "anvil_timeline_read")
    return buf


def device_error(clear=True):
    """Status of the device error word (ANVIL_OK or ANVIL_ERR_TIMEOUT); synchronises."""
    return _lib.anvil_device_error(1 if clear else 0)


def last_device_error(stream=None):
    """Status of the device error word after the work queued on `stream` (default: the
    current stream); waits for that stream only and resets the word."""
    return _lib.anvil_last_device_error(_stream_arg(stream))


def selftest_wait_timeout(timeout_us, stream=None):
    _check(_lib.anvil_selftest_wait_timeout(int(timeout_us), _stream_arg(stream)),
           "anvil_selftest_wait_timeout")


class profile:
    """Context manager: per-launch CUDA-event timings of the steps run inside it.
    After exit, ``records`` is a list of (kernel kind name, milliseconds)."""

    def __init__(self, max_records=4096):
        self.max_records = max_records
        self.records = []

    def __enter__(self):
        _check(_lib.anvil_profile_begin(self.max_records), "anvil_profile_begin")
        return self

    def __exit__(self, *exc):
        arr = (ProfileRecord * self.max_records)()
        n = _lib.anvil_profile_end(arr, self.max_records)
        if n < 0:
            raise AnvilError(ERR_CUDA, "anvil_profile_end")
        self.records = [(KERNEL_KINDS[arr[i].kind], arr[i].ms) for i in range(n)]
        return False
