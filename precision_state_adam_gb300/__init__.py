"""precision_state_adam_gb300 — fused AdamW with compressed moment state on GB300.

A thin ctypes binding over libpsadam.so (the C ABI in include/psadam.h). Every function
here only marshals torch tensors into pointer tables and calls the library; the
arithmetic runs in the library's sm_103a kernels. There is no CPU fallback: importing
this package fails if the library has not been built.

Entry points (same names as the C ABI):
    adam_step_fp32(params, grads, m, v, step, ...)              fp32 moments
    adam_step_bf16m(params, grads, m, v, step, ...)             bf16 moments (torch.bfloat16 tensors)
    adam_step_q8(params, grads, m_code, v_code, m_scale, v_scale, step, ...)
    adam_step_q8v(params, grads, m, v_code, v_scale, step, ...) fp32 m, 8-bit v
    q8_quantize / q8_dequantize                                 8-bit state conversion
    state_bytes(mode, numel, block_size)                        optimizer-state footprint
and helpers to allocate fresh (zero) state with the right dtypes and shapes.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpsadam.so")
BLOCK = 2048             # the 8-bit format's default block (the specialised kernels' size)
MAX_BLOCK = 16384        # largest block size the library accepts
MAX_PERCENTILE_RANK = 4  # above this rank (or at another block size) the general kernel runs

OK, ERR_INVALID_ARG, ERR_MISALIGNED, ERR_UNSUPPORTED, ERR_CUDA = range(5)
GRAD_F32, GRAD_BF16 = 0, 1
MODES = {"fp32": 0, "bf16m": 1, "q8": 2, "q8v": 3}

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
        "(or `python precision_state_adam_gb300/build.py`). There is no CPU fallback.")


class _HParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


class _Q8Opts(ctypes.Structure):
    _fields_ = [("block_size", ctypes.c_int32), ("stochastic_rounding", ctypes.c_int32),
                ("seed", ctypes.c_uint64), ("percentile", ctypes.c_float), ("static_scales", ctypes.c_int32)]


class _List(ctypes.Structure):
    _fields_ = [("n_tensors", ctypes.c_int32), ("grad_dtype", ctypes.c_int32),
                ("numel", ctypes.POINTER(ctypes.c_int64)), ("param", ctypes.POINTER(ctypes.c_void_p)),
                ("grad", ctypes.POINTER(ctypes.c_void_p)), ("grad_unscale", ctypes.c_float),
                ("zero_grads", ctypes.c_int32), ("skip_if_set", ctypes.c_void_p), ("approx_update", ctypes.c_int32)]


_lib = ctypes.CDLL(LIB_PATH)
_vp = ctypes.c_void_p
_PP = ctypes.POINTER(ctypes.c_void_p)
_I64P = ctypes.POINTER(ctypes.c_int64)
_SIGS = {
    "adam_step_fp32": [ctypes.POINTER(_List), _PP, _PP, ctypes.c_int64, ctypes.POINTER(_HParams), _vp],
    "adam_step_bf16m": [ctypes.POINTER(_List), _PP, _PP, ctypes.c_int64, ctypes.POINTER(_HParams), _vp],
    "adam_step_q8": [ctypes.POINTER(_List), _PP, _PP, _PP, _PP, ctypes.c_int64, ctypes.POINTER(_HParams),
                     ctypes.POINTER(_Q8Opts), _vp],
    "adam_step_q8v": [ctypes.POINTER(_List), _PP, _PP, _PP, ctypes.c_int64, ctypes.POINTER(_HParams),
                      ctypes.POINTER(_Q8Opts), _vp],
    "psadam_q8_quantize": [ctypes.c_int32, _I64P, _PP, _PP, _PP, _PP, _PP, _PP, ctypes.POINTER(_Q8Opts),
                           ctypes.c_int64, _vp],
    "psadam_q8_dequantize": [ctypes.c_int32, _I64P, _PP, _PP, _PP, _PP, _PP, _PP, ctypes.c_int32, _vp],
    "psadam_check_grads": [ctypes.POINTER(_List), _vp, _vp],
    "psadam_step_from_host": [ctypes.c_int32, ctypes.POINTER(_List), _PP, _PP, _PP, _PP, _PP, _PP, ctypes.c_int64,
                              ctypes.POINTER(_HParams), ctypes.POINTER(_Q8Opts), ctypes.c_int32, _vp, _vp, _vp],
}
for _name, _args in _SIGS.items():
    getattr(_lib, _name).argtypes = _args
    getattr(_lib, _name).restype = ctypes.c_int
_lib.psadam_state_bytes.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32]
_lib.psadam_state_bytes.restype = ctypes.c_size_t
_lib.psadam_status_string.argtypes = [ctypes.c_int32]
_lib.psadam_status_string.restype = ctypes.c_char_p
_lib.psadam_selftest_bounded_wait.argtypes = [ctypes.c_int64, ctypes.c_void_p]
_lib.psadam_selftest_bounded_wait.restype = ctypes.c_int
_lib.psadam_selftest_update_math.argtypes = [ctypes.c_int32, ctypes.POINTER(ctypes.c_uint64), ctypes.c_void_p]
_lib.psadam_selftest_update_math.restype = ctypes.c_int
_lib.psadam_device_fault.argtypes = []
_lib.psadam_device_fault.restype = ctypes.c_int32
_lib.psadam_last_cuda_error.argtypes = []
_lib.psadam_last_cuda_error.restype = ctypes.c_int32


class PSAdamError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {status_string(status)}"
        if status == ERR_CUDA:
            msg += f" (cudaError {_lib.psadam_last_cuda_error()})"
        super().__init__(msg)


def status_string(status: int) -> str:
    return _lib.psadam_status_string(status).decode()


def state_bytes(mode: str | int, numel: int, block_size: int = BLOCK) -> int:
    return int(_lib.psadam_state_bytes(MODES.get(mode, mode) if isinstance(mode, str) else mode, numel, block_size))


def n_blocks(numel: int, block_size: int = BLOCK) -> int:
    return (numel + block_size - 1) // block_size


def _nb(block_size: int):
    return lambda n: n_blocks(n, block_size)


# ------------------------------------------------------------------ marshalling
def _ptrs(ts: Sequence[torch.Tensor | None]):
    arr = (ctypes.c_void_p * max(len(ts), 1))()
    for i, t in enumerate(ts):
        arr[i] = None if t is None or t.numel() == 0 else t.data_ptr()
    return arr


def _numels(ts: Sequence[torch.Tensor]):
    arr = (ctypes.c_int64 * max(len(ts), 1))()
    for i, t in enumerate(ts):
        arr[i] = t.numel()
    return arr


def _stream_handle(stream, ts) -> int | None:
    if stream is None:
        dev = next((t.device for t in ts if t is not None and t.is_cuda), None)
        stream = torch.cuda.current_stream(dev) if dev is not None else None
    if stream is None:
        return None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_layout(name: str, ts, dtype, like=None, numel_fn=None) -> None:
    """Every tensor of ``ts``: ``dtype``, contiguous, on the CUDA device of its counterpart in
    ``like`` (of ``ts[0]`` without one) and, with ``like``, one per tensor of ``like`` with the
    element count ``numel_fn`` gives (the same count by default). The library reads as many
    pointers from every table as the list has tensors, so a short table is refused here."""
    if like is not None and len(ts) != len(like):
        raise ValueError(f"{name}: {len(ts)} tensors for a list of {len(like)}")
    for i, t in enumerate(ts):
        if t.dtype != dtype:
            raise TypeError(f"{name}[{i}]: expected {dtype}, got {t.dtype}")
        if not t.is_cuda:
            raise TypeError(f"{name}[{i}]: must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name}[{i}]: must be contiguous")
        dev = like[i].device if like is not None else ts[0].device
        if t.device != dev:
            raise ValueError(f"{name}[{i}]: on {t.device}, expected {dev}")
        if like is not None:
            want = numel_fn(like[i].numel()) if numel_fn else like[i].numel()
            if t.numel() != want:
                raise ValueError(f"{name}[{i}]: expected {want} elements, got {t.numel()}")


def _hp(lr, beta1, beta2, eps, weight_decay) -> _HParams:
    return _HParams(lr, beta1, beta2, eps, weight_decay)


def _skip_ptr(skip_flag) -> int | None:
    if skip_flag is None:
        return None
    if skip_flag.dtype != torch.int32 or not skip_flag.is_cuda or skip_flag.numel() < 1:
        raise TypeError("skip_flag must be a CUDA int32 tensor")
    return skip_flag.data_ptr()


def _list(params, grads, grad_unscale: float = 1.0, zero_grads: bool = False, skip_flag=None, like=None,
          approx_update: bool = False):
    if like is None:
        like = params
        if len(params) != len(grads):
            raise ValueError("params and grads differ in length")
        _check_layout("params", params, torch.float32)
    gdt = grads[0].dtype if grads else torch.float32
    if gdt not in (torch.float32, torch.bfloat16):
        raise TypeError("grads must be float32 or bfloat16")
    _check_layout("grads", grads, gdt, like)
    keep = (_numels(like), _ptrs(params) if params is not None else None, _ptrs(grads))
    lst = _List(len(grads), GRAD_BF16 if gdt == torch.bfloat16 else GRAD_F32, keep[0],
                ctypes.cast(keep[1], _PP) if keep[1] is not None else None, ctypes.cast(keep[2], _PP),
                grad_unscale, int(bool(zero_grads)), _skip_ptr(skip_flag), int(bool(approx_update)))
    return lst, keep


def _raise(status: int, where: str) -> None:
    if status != OK:
        raise PSAdamError(status, where)


# ------------------------------------------------------------------ steps
def adam_step_fp32(params, grads, m, v, step: int, lr: float = 1e-3, beta1: float = 0.9, beta2: float = 0.999,
                   eps: float = 1e-8, weight_decay: float = 0.0, grad_unscale: float = 1.0, zero_grads: bool = False,
                   skip_flag=None, approx_update: bool = False, stream=None) -> None:
    """One AdamW step with fp32 moments, in place, enqueued on ``stream`` (default: current).
    Grad side: grads are multiplied by ``grad_unscale`` before use, overwritten with zeros
    after use when ``zero_grads``, and the whole step is skipped on the device when the
    CUDA int32 tensor ``skip_flag`` holds a nonzero value (see :func:`check_grads`).
    ``approx_update`` opts into the hardware's approximate square root and quotient in the
    parameter update (2-3 % faster for 8-bit moments; params within a few ulp of the
    update of the IEEE result, every moment, code and scale still exact)."""
    lst, keep = _list(params, grads, grad_unscale, zero_grads, skip_flag, approx_update=approx_update)
    _check_layout("m", m, torch.float32, params)
    _check_layout("v", v, torch.float32, params)
    mp, vp = _ptrs(m), _ptrs(v)
    st = _lib.adam_step_fp32(ctypes.byref(lst), ctypes.cast(mp, _PP), ctypes.cast(vp, _PP), step,
                             ctypes.byref(_hp(lr, beta1, beta2, eps, weight_decay)), _stream_handle(stream, params))
    _raise(st, "adam_step_fp32")


def adam_step_bf16m(params, grads, m, v, step: int, lr: float = 1e-3, beta1: float = 0.9, beta2: float = 0.999,
                   eps: float = 1e-8, weight_decay: float = 0.0, grad_unscale: float = 1.0, zero_grads: bool = False,
                   skip_flag=None, approx_update: bool = False, stream=None) -> None:
    """One AdamW step with bf16 moments (torch.bfloat16 tensors), in place (grad-side
    options as for :func:`adam_step_fp32`)."""
    lst, keep = _list(params, grads, grad_unscale, zero_grads, skip_flag, approx_update=approx_update)
    _check_layout("m", m, torch.bfloat16, params)
    _check_layout("v", v, torch.bfloat16, params)
    mp, vp = _ptrs(m), _ptrs(v)
    st = _lib.adam_step_bf16m(ctypes.byref(lst), ctypes.cast(mp, _PP), ctypes.cast(vp, _PP), step,
                              ctypes.byref(_hp(lr, beta1, beta2, eps, weight_decay)), _stream_handle(stream, params))
    _raise(st, "adam_step_bf16m")


def _q8(stochastic_rounding: bool, seed: int, percentile: float, block_size: int,
        static_scales: bool = False) -> _Q8Opts:
    return _Q8Opts(block_size, int(bool(stochastic_rounding)), seed, percentile, int(bool(static_scales)))


def adam_step_q8(params, grads, m_code, v_code, m_scale, v_scale, step: int, lr: float = 1e-3, beta1: float = 0.9,
                 beta2: float = 0.999, eps: float = 1e-8, weight_decay: float = 0.0, stochastic_rounding: bool = False,
                 seed: int = 42, percentile: float = 100.0, block_size: int = BLOCK, grad_unscale: float = 1.0,
                 zero_grads: bool = False, skip_flag=None, static_scales: bool = False, approx_update: bool = False,
                 stream=None) -> None:
    """One AdamW step with 8-bit block-wise moments (int8 m codes, uint8 v codes, fp32
    per-block scales), dequantize-update-requantize in one pass, in place.

    Defaults follow the 8-bit Adam PR's options list (block 2048, scales recomputed every
    step, round to nearest, seed 42) except the percentile: the options list defaults to
    99.9 (the block's 3rd-largest magnitude sets the scale); here the default is absmax
    (percentile 100), the faster kernel. Pass ``percentile=99.9`` for the listed default."""
    lst, keep = _list(params, grads, grad_unscale, zero_grads, skip_flag, approx_update=approx_update)
    _check_layout("m_code", m_code, torch.int8, params)
    _check_layout("v_code", v_code, torch.uint8, params)
    _check_layout("m_scale", m_scale, torch.float32, params, _nb(block_size))
    _check_layout("v_scale", v_scale, torch.float32, params, _nb(block_size))
    ptrs = [_ptrs(x) for x in (m_code, v_code, m_scale, v_scale)]
    st = _lib.adam_step_q8(ctypes.byref(lst), *[ctypes.cast(p, _PP) for p in ptrs], step,
                           ctypes.byref(_hp(lr, beta1, beta2, eps, weight_decay)),
                           ctypes.byref(_q8(stochastic_rounding, seed, percentile, block_size, static_scales)),
                           _stream_handle(stream, params))
    _raise(st, "adam_step_q8")


def adam_step_q8v(params, grads, m, v_code, v_scale, step: int, lr: float = 1e-3, beta1: float = 0.9,
                  beta2: float = 0.999, eps: float = 1e-8, weight_decay: float = 0.0, stochastic_rounding: bool = False,
                  seed: int = 42, percentile: float = 100.0, block_size: int = BLOCK, grad_unscale: float = 1.0,
                  zero_grads: bool = False, skip_flag=None, static_scales: bool = False, approx_update: bool = False,
                 stream=None) -> None:
    """One AdamW step with an fp32 first moment and an 8-bit block-wise second moment
    (uint8 v codes, fp32 per-block scales), in place. Defaults as :func:`adam_step_q8`
    (absmax; the options list's percentile default is 99.9)."""
    lst, keep = _list(params, grads, grad_unscale, zero_grads, skip_flag, approx_update=approx_update)
    _check_layout("m", m, torch.float32, params)
    _check_layout("v_code", v_code, torch.uint8, params)
    _check_layout("v_scale", v_scale, torch.float32, params, _nb(block_size))
    ptrs = [_ptrs(x) for x in (m, v_code, v_scale)]
    st = _lib.adam_step_q8v(ctypes.byref(lst), *[ctypes.cast(p, _PP) for p in ptrs], step,
                            ctypes.byref(_hp(lr, beta1, beta2, eps, weight_decay)),
                            ctypes.byref(_q8(stochastic_rounding, seed, percentile, block_size, static_scales)),
                            _stream_handle(stream, params))
    _raise(st, "adam_step_q8v")


def check_grads(grads, found_nonfinite, grad_unscale: float = 1.0, stream=None) -> None:
    """Set the CUDA int32 tensor ``found_nonfinite`` to 1 if any grad times ``grad_unscale``
    is +-inf or NaN, else 0 (enqueued on the stream; pass it as ``skip_flag`` to the step)."""
    if found_nonfinite.dtype != torch.int32 or not found_nonfinite.is_cuda:
        raise TypeError("found_nonfinite must be a CUDA int32 tensor")
    lst, keep = _list(None, grads, grad_unscale, like=grads)
    st = _lib.psadam_check_grads(ctypes.byref(lst), found_nonfinite.data_ptr(), _stream_handle(stream, grads))
    _raise(st, "psadam_check_grads")


def q8_quantize(m, v, m_code, v_code, m_scale, v_scale, step: int = 1, stochastic_rounding: bool = False,
                seed: int = 42, percentile: float = 100.0, block_size: int = BLOCK, stream=None) -> None:
    """Encode fp32 moments into 8-bit codes and block scales (as the step encodes m', v')."""
    _check_layout("m", m, torch.float32)
    _check_layout("v", v, torch.float32, m)
    _check_layout("m_code", m_code, torch.int8, m)
    _check_layout("v_code", v_code, torch.uint8, m)
    _check_layout("m_scale", m_scale, torch.float32, m, _nb(block_size))
    _check_layout("v_scale", v_scale, torch.float32, m, _nb(block_size))
    ptrs = [_ptrs(x) for x in (m, v, m_code, v_code, m_scale, v_scale)]
    st = _lib.psadam_q8_quantize(len(m), _numels(m), *[ctypes.cast(p, _PP) for p in ptrs],
                                 ctypes.byref(_q8(stochastic_rounding, seed, percentile, block_size)), step,
                                 _stream_handle(stream, m))
    _raise(st, "psadam_q8_quantize")


def q8_dequantize(m_code, v_code, m_scale, v_scale, m, v, block_size: int = BLOCK, stream=None) -> None:
    """Decode 8-bit codes and block scales into fp32 moments (code * scale)."""
    _check_layout("m_code", m_code, torch.int8)
    _check_layout("v_code", v_code, torch.uint8, m_code)
    _check_layout("m_scale", m_scale, torch.float32, m_code, _nb(block_size))
    _check_layout("v_scale", v_scale, torch.float32, m_code, _nb(block_size))
    _check_layout("m", m, torch.float32, m_code)
    _check_layout("v", v, torch.float32, m_code)
    ptrs = [_ptrs(x) for x in (m_code, v_code, m_scale, v_scale, m, v)]
    st = _lib.psadam_q8_dequantize(len(m_code), _numels(m_code), *[ctypes.cast(p, _PP) for p in ptrs], block_size,
                                   _stream_handle(stream, m))
    _raise(st, "psadam_q8_dequantize")


# ------------------------------------------------------------------ state allocation (caller side)
def zeros_state(params, mode: str, block_size: int = BLOCK):
    """Fresh (all-zero) optimizer state for ``params`` in moment mode ``mode``.
    fp32/bf16m: (m list, v list); q8: (m_code, v_code, m_scale, v_scale) lists;
    q8v: (m fp32, v_code, v_scale) lists (one scale per ``block_size`` elements)."""
    if mode == "fp32":
        return [torch.zeros_like(p) for p in params], [torch.zeros_like(p) for p in params]
    if mode == "bf16m":
        z = lambda p: torch.zeros(p.numel(), dtype=torch.bfloat16, device=p.device)
        return [z(p) for p in params], [z(p) for p in params]
    if mode == "q8":
        return ([torch.zeros(p.numel(), dtype=torch.int8, device=p.device) for p in params],
                [torch.zeros(p.numel(), dtype=torch.uint8, device=p.device) for p in params],
                [torch.zeros(n_blocks(p.numel(), block_size), dtype=torch.float32, device=p.device) for p in params],
                [torch.zeros(n_blocks(p.numel(), block_size), dtype=torch.float32, device=p.device) for p in params])
    if mode == "q8v":
        return ([torch.zeros_like(p) for p in params],
                [torch.zeros(p.numel(), dtype=torch.uint8, device=p.device) for p in params],
                [torch.zeros(n_blocks(p.numel(), block_size), dtype=torch.float32, device=p.device) for p in params])
    raise ValueError(f"unknown moment mode {mode!r}")


def adam_step(mode: str, params, grads, state, step: int, **kw) -> None:
    """Dispatch by moment mode name: ``state`` as returned by :func:`zeros_state`."""
    if mode == "fp32":
        adam_step_fp32(params, grads, *state, step, **kw)
    elif mode == "bf16m":
        adam_step_bf16m(params, grads, *state, step, **kw)
    elif mode == "q8":
        adam_step_q8(params, grads, *state, step, **kw)
    elif mode == "q8v":
        adam_step_q8v(params, grads, *state, step, **kw)
    else:
        raise ValueError(f"unknown moment mode {mode!r}")


class StepPlan:
    """A tensor list marshalled once for repeated steps.

    Building the pointer tables costs Python time proportional to the number of tensors;
    an optimizer calls the step with the same tensors every iteration, so the plan keeps
    the tables and each :meth:`step` is one C call. The tensors must stay alive and in
    place (same storage) for the plan's lifetime; grads may be swapped with
    :meth:`set_grads` (same shapes and dtype)."""

    def __init__(self, mode: str, params, grads, state, lr: float = 1e-3, beta1: float = 0.9,
                 beta2: float = 0.999, eps: float = 1e-8, weight_decay: float = 0.0,
                 stochastic_rounding: bool = False, seed: int = 42, percentile: float = 100.0,
                 block_size: int = BLOCK, grad_unscale: float = 1.0, zero_grads: bool = False, skip_flag=None,
                 static_scales: bool = False, approx_update: bool = False):
        if mode not in MODES:
            raise ValueError(f"unknown moment mode {mode!r}")
        self.mode = mode
        self._skip = skip_flag
        self._lst, self._keep = _list(params, grads, grad_unscale, zero_grads, skip_flag, approx_update=approx_update)
        self._grad_dtype = grads[0].dtype if grads else torch.float32
        self._params = list(params)
        if mode == "fp32":
            _check_layout("m", state[0], torch.float32, params)
            _check_layout("v", state[1], torch.float32, params)
        elif mode == "bf16m":
            _check_layout("m", state[0], torch.bfloat16, params)
            _check_layout("v", state[1], torch.bfloat16, params)
        elif mode == "q8":
            _check_layout("m_code", state[0], torch.int8, params)
            _check_layout("v_code", state[1], torch.uint8, params)
            _check_layout("m_scale", state[2], torch.float32, params, _nb(block_size))
            _check_layout("v_scale", state[3], torch.float32, params, _nb(block_size))
        else:
            _check_layout("m", state[0], torch.float32, params)
            _check_layout("v_code", state[1], torch.uint8, params)
            _check_layout("v_scale", state[2], torch.float32, params, _nb(block_size))
        self._state_ptrs = [_ptrs(x) for x in state]
        self._state_pp = [ctypes.cast(p, _PP) for p in self._state_ptrs]
        self._state = state
        self._hp = _hp(lr, beta1, beta2, eps, weight_decay)
        self._q8 = _q8(stochastic_rounding, seed, percentile, block_size, static_scales)

    def set_grads(self, grads) -> None:
        if len(grads) != len(self._params):
            raise ValueError("grads differ in length from params")
        _check_layout("grads", grads, self._grad_dtype, self._params)
        gp = _ptrs(grads)
        self._keep = (self._keep[0], self._keep[1], gp)
        self._lst.grad = ctypes.cast(gp, _PP)

    def step(self, step: int, stream=None) -> None:
        h = _stream_handle(stream, self._params)
        if self.mode == "fp32":
            st = _lib.adam_step_fp32(ctypes.byref(self._lst), *self._state_pp, step, ctypes.byref(self._hp), h)
        elif self.mode == "bf16m":
            st = _lib.adam_step_bf16m(ctypes.byref(self._lst), *self._state_pp, step, ctypes.byref(self._hp), h)
        elif self.mode == "q8":
            st = _lib.adam_step_q8(ctypes.byref(self._lst), *self._state_pp, step, ctypes.byref(self._hp),
                                   ctypes.byref(self._q8), h)
        else:
            st = _lib.adam_step_q8v(ctypes.byref(self._lst), *self._state_pp, step, ctypes.byref(self._hp),
                                    ctypes.byref(self._q8), h)
        _raise(st, f"StepPlan.step ({self.mode})")

    def step_from_host(self, step: int, host_grads, host_params, n_chunks: int = 4, stream=None, stream_in=None,
                       stream_out=None) -> None:
        """The step with host-resident grads and params: ``host_grads`` (CPU tensors like the
        plan's grads, pinned for asynchronous copies) are copied into the plan's device grads,
        the step runs, and the updated params are copied into ``host_params`` (CPU float32).
        With ``stream_in`` and ``stream_out`` the list is cut into about ``n_chunks`` chunks whose
        copies overlap the step; results equal :meth:`step` bit for bit."""
        if len(host_grads) != len(self._params) or len(host_params) != len(self._params):
            raise ValueError("host grads / params differ in length from params")
        for i, (hg, hp, p) in enumerate(zip(host_grads, host_params, self._params)):
            if hg.is_cuda or hp.is_cuda:
                raise TypeError(f"host tensor {i} is on a CUDA device")
            if hg.dtype != self._grad_dtype or hp.dtype != torch.float32:
                raise TypeError(f"host tensor {i}: expected grads {self._grad_dtype} and params float32")
            if hg.numel() != p.numel() or hp.numel() != p.numel() or not hg.is_contiguous() or not hp.is_contiguous():
                raise ValueError(f"host tensor {i}: expected {p.numel()} contiguous elements")
        key = (tuple(t.data_ptr() for t in host_grads), tuple(t.data_ptr() for t in host_params))
        if getattr(self, "_host_key", None) != key:
            self._host_key = key
            self._host_tables = (_ptrs(host_grads), _ptrs(host_params))
        hg, hp = self._host_tables
        n_state = len(self._state_pp)
        pp = list(self._state_pp) + [None] * (4 - n_state)
        if self.mode == "q8v":  # (m, v codes, v scale) -> m, v, no m scale, v scale
            pp = [self._state_pp[0], self._state_pp[1], None, self._state_pp[2]]
        h = _stream_handle(stream, self._params)
        sin = _stream_handle(stream_in, self._params) if stream_in is not None else None
        sout = _stream_handle(stream_out, self._params) if stream_out is not None else None
        q8 = ctypes.byref(self._q8) if self.mode in ("q8", "q8v") else None
        st = _lib.psadam_step_from_host(MODES[self.mode], ctypes.byref(self._lst), ctypes.cast(hg, _PP),
                                        ctypes.cast(hp, _PP), *pp, step, ctypes.byref(self._hp), q8, n_chunks, h,
                                        sin, sout)
        _raise(st, f"StepPlan.step_from_host ({self.mode})")


def selftest_update_math(full: bool = False, stream=None) -> dict:
    """Device-side counts of results of the update's own root and quotient that differ from IEEE
    sqrt / division (psadam_selftest_update_math): all four are 0 on a correct build."""
    out = (ctypes.c_uint64 * 4)()
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _raise(_lib.psadam_selftest_update_math(int(bool(full)), out, handle), "psadam_selftest_update_math")
    return {"root": int(out[0]), "quotient": int(out[1]), "scaling": int(out[2]), "update": int(out[3])}


def device_fault() -> int:
    """1 if a library kernel gave up a bounded wait since the last call (then read as 0), else 0."""
    return int(_lib.psadam_device_fault())


def cdll() -> ctypes.CDLL:
    """The loaded libpsadam.so handle (for ABI-level tests)."""
    return _lib


from .serialize import StateFormatError, load_state, save_state  # noqa: E402  (host-side state files)
