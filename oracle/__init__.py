"""CPU oracle for the fused AdamW update with compressed moment state.

TEST INFRASTRUCTURE ONLY. A plain, slow, single-threaded restatement (C, via ctypes)
of what the CUDA library computes, written from the method's sources:
AiDotNet PR #814 "add 8-bit Adam optimizer for memory efficiency" (block-wise 8-bit
moments, its sequence diagram and options), AiDotNet PR #1745 "make BF16-Adam
fused-compatible" (bf16 moment storage), textbook Adam/AdamW, and Salmon et al.
"Parallel random numbers: as easy as 1, 2, 3" (Philox4x32-10).

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg may import
this package. It shares no code with ``precision_state_adam_gb300`` and never imports it.

All array arguments are numpy arrays; state arrays are updated in place.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

BLOCK = 2048

_u32p = ctypes.POINTER(ctypes.c_uint32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_i8p = ctypes.POINTER(ctypes.c_int8)
_u8p = ctypes.POINTER(ctypes.c_uint8)


class _HP(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


class _Scalars(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in
                ("b1", "omb1", "b2", "omb2", "decay", "step_size", "inv_sqrt_bc2", "eps")]


class _Q8(ctypes.Structure):
    _fields_ = [("stochastic_rounding", ctypes.c_int), ("seed", ctypes.c_uint64),
                ("percentile", ctypes.c_float), ("static_scales", ctypes.c_int), ("block_size", ctypes.c_int)]


@dataclass(frozen=True)
class HParams:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0

    def _c(self) -> _HP:
        return _HP(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay)


@dataclass(frozen=True)
class Q8Opts:
    stochastic_rounding: bool = False
    seed: int = 42
    percentile: float = 100.0
    static_scales: bool = False
    block_size: int = BLOCK

    def _c(self) -> _Q8:
        assert self.block_size >= 1, "block size must be positive"
        return _Q8(int(self.stochastic_rounding), self.seed, self.percentile, int(self.static_scales),
                   self.block_size)


def _load() -> ctypes.CDLL:
    lib = ctypes.CDLL(_build.build())
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    hp = ctypes.POINTER(_HP)
    q8 = ctypes.POINTER(_Q8)
    sigs = {
        "orc_philox4x32_10_many": (None, [i64, _u32p, _u32p, _u32p]),
        "orc_sr_uniform": (ctypes.c_float, [ctypes.c_uint64, i64, i32, i32, i64]),
        "orc_bf16_round": (ctypes.c_uint16, [ctypes.c_float]),
        "orc_bf16_widen": (ctypes.c_float, [ctypes.c_uint16]),
        "orc_bf16_round_many": (None, [i64, _f32p, _u16p]),
        "orc_bf16_widen_many": (None, [i64, _u16p, _f32p]),
        "orc_make_scalars": (_Scalars, [hp, i64]),
        "orc_percentile_rank": (i64, [ctypes.c_float, i64]),
        "orc_kth_largest_abs": (ctypes.c_float, [_f32p, i64, i64]),
        "orc_quantize_block": (ctypes.c_float, [_f32p, i64, i32, q8, i64, i32, i64, ctypes.c_float, _i8p, _u8p]),
        "orc_quantize": (None, [i64, _f32p, _f32p, q8, i64, i32, _i8p, _u8p, _f32p, _f32p]),
        "orc_dequantize": (None, [i64, i64, _i8p, _u8p, _f32p, _f32p, _f32p, _f32p]),
        "orc_step_fp32": (None, [i64, _f32p, vp, i32, _f32p, _f32p, hp, i64]),
        "orc_step_bf16m": (None, [i64, _f32p, vp, i32, _u16p, _u16p, hp, i64]),
        "orc_step_q8": (None, [i64, _f32p, vp, i32, _i8p, _u8p, _f32p, _f32p, hp, i64, q8, i32,
                               i64, i64]),
        "orc_step_q8_block": (None, [i64, i64, _f32p, vp, i32, _i8p, _u8p, _f32p, _f32p, hp, i64, q8, i32]),
        "orc_step_q8v": (None, [i64, _f32p, vp, i32, _f32p, _u8p, _f32p, hp, i64, q8, i32, i64, i64]),
        "orc_step_q8v_block": (None, [i64, i64, _f32p, vp, i32, _f32p, _u8p, _f32p, hp, i64, q8, i32]),
        "orc_unscale_grads": (None, [i64, vp, i32, ctypes.c_float, _f32p]),
        "orc_probe_mul_add": (ctypes.c_float, [ctypes.c_float] * 3),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _check(a: np.ndarray, dtype, name: str, n: int | None = None) -> None:
    if a.dtype != dtype or not a.flags["C_CONTIGUOUS"]:
        raise TypeError(f"{name}: expected contiguous {np.dtype(dtype)}, got {a.dtype}")
    if n is not None and a.size != n:
        raise ValueError(f"{name}: expected {n} elements, got {a.size}")


def n_blocks(n: int, block_size: int = BLOCK) -> int:
    return (n + block_size - 1) // block_size


# ---------------------------------------------------------------- primitives
def philox4x32_10(ctr: np.ndarray, key: np.ndarray) -> np.ndarray:
    """Philox4x32-10 of counters ``ctr`` (n,4) under keys ``key`` (n,2) -> (n,4) uint32."""
    ctr = np.ascontiguousarray(ctr, dtype=np.uint32).reshape(-1, 4)
    key = np.ascontiguousarray(np.broadcast_to(np.asarray(key, dtype=np.uint32), (len(ctr), 2)))
    out = np.empty_like(ctr)
    _lib.orc_philox4x32_10_many(len(ctr), _ptr(ctr, ctypes.c_uint32), _ptr(key, ctypes.c_uint32),
                                _ptr(out, ctypes.c_uint32))
    return out


def sr_uniform(seed: int, step: int, tensor_idx: int, moment: int, elem: int) -> float:
    return _lib.orc_sr_uniform(seed, step, tensor_idx, moment, elem)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _lib.orc_bf16_round_many(x.size, _ptr(x, ctypes.c_float), _ptr(out, ctypes.c_uint16))
    return out


def bf16_widen(b: np.ndarray) -> np.ndarray:
    """bf16 bits (uint16) -> fp32, exact."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float32)
    _lib.orc_bf16_widen_many(b.size, _ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_float))
    return out


def scalars(hp: HParams, t: int) -> dict:
    s = _lib.orc_make_scalars(ctypes.byref(hp._c()), t)
    return {n: np.float32(getattr(s, n)) for n, _ in _Scalars._fields_}


def percentile_rank(pct: float, n: int) -> int:
    return int(_lib.orc_percentile_rank(pct, n))


def kth_largest_abs(x: np.ndarray, k: int) -> np.float32:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return np.float32(_lib.orc_kth_largest_abs(_ptr(x, ctypes.c_float), x.size, k))


def quantize_block(x: np.ndarray, signed: bool, q8: Q8Opts = Q8Opts(), step: int = 1,
                   tensor_idx: int = 0, elem0: int = 0, old_scale: float = 0.0):
    """Quantize one block of ``x.size`` values. Returns (codes, scale). ``old_scale`` is
    kept when ``q8.static_scales`` and it is nonzero."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.zeros(x.size, dtype=np.int8 if signed else np.uint8)
    i8 = _ptr(codes, ctypes.c_int8) if signed else None
    u8 = None if signed else _ptr(codes, ctypes.c_uint8)
    s = _lib.orc_quantize_block(_ptr(x, ctypes.c_float), x.size, int(signed), ctypes.byref(q8._c()),
                                step, tensor_idx, elem0, old_scale, i8, u8)
    return codes, np.float32(s)


def quantize(m: np.ndarray, v: np.ndarray, q8: Q8Opts = Q8Opts(), step: int = 1, tensor_idx: int = 0):
    """Whole-tensor quantize of a moment pair -> (m_code int8, v_code uint8, m_scale, v_scale)."""
    n = m.size
    _check(m, np.float32, "m")
    _check(v, np.float32, "v", n)
    mc = np.zeros(n, np.int8)
    vc = np.zeros(n, np.uint8)
    ms = np.zeros(n_blocks(n, q8.block_size), np.float32)
    vs = np.zeros(n_blocks(n, q8.block_size), np.float32)
    _lib.orc_quantize(n, _ptr(m, ctypes.c_float), _ptr(v, ctypes.c_float), ctypes.byref(q8._c()), step,
                      tensor_idx, _ptr(mc, ctypes.c_int8), _ptr(vc, ctypes.c_uint8),
                      _ptr(ms, ctypes.c_float), _ptr(vs, ctypes.c_float))
    return mc, vc, ms, vs


def dequantize(mc, vc, ms, vs, block_size: int = BLOCK):
    n = mc.size
    _check(mc, np.int8, "m_code")
    _check(vc, np.uint8, "v_code", n)
    _check(ms, np.float32, "m_scale", n_blocks(n, block_size))
    _check(vs, np.float32, "v_scale", n_blocks(n, block_size))
    m = np.empty(n, np.float32)
    v = np.empty(n, np.float32)
    _lib.orc_dequantize(n, block_size, _ptr(mc, ctypes.c_int8), _ptr(vc, ctypes.c_uint8), _ptr(ms, ctypes.c_float),
                        _ptr(vs, ctypes.c_float), _ptr(m, ctypes.c_float), _ptr(v, ctypes.c_float))
    return m, v


# ---------------------------------------------------------------- steps (in place)
def _grad(g: np.ndarray, n: int):
    if g.dtype == np.float32:
        _check(g, np.float32, "grad", n)
        return g.ctypes.data_as(ctypes.c_void_p), 0
    # bf16 grads travel as their raw uint16 bits
    _check(g, np.uint16, "grad (bf16 bits)", n)
    return g.ctypes.data_as(ctypes.c_void_p), 1


def step_fp32(p, g, m, v, t: int, hp: HParams) -> None:
    n = p.size
    _check(p, np.float32, "param")
    _check(m, np.float32, "m", n)
    _check(v, np.float32, "v", n)
    gp, gb = _grad(g, n)
    _lib.orc_step_fp32(n, _ptr(p, ctypes.c_float), gp, gb, _ptr(m, ctypes.c_float),
                       _ptr(v, ctypes.c_float), ctypes.byref(hp._c()), t)


def step_bf16m(p, g, m, v, t: int, hp: HParams) -> None:
    n = p.size
    _check(p, np.float32, "param")
    _check(m, np.uint16, "m (bf16 bits)", n)
    _check(v, np.uint16, "v (bf16 bits)", n)
    gp, gb = _grad(g, n)
    _lib.orc_step_bf16m(n, _ptr(p, ctypes.c_float), gp, gb, _ptr(m, ctypes.c_uint16),
                        _ptr(v, ctypes.c_uint16), ctypes.byref(hp._c()), t)


def step_q8(p, g, mc, vc, ms, vs, t: int, hp: HParams, q8: Q8Opts = Q8Opts(), tensor_idx: int = 0,
            blocks: tuple[int, int] | None = None) -> None:
    """8-bit step over blocks [b0, b1) (default: all blocks) of one tensor."""
    n = p.size
    _check(p, np.float32, "param")
    _check(mc, np.int8, "m_code", n)
    _check(vc, np.uint8, "v_code", n)
    nb = n_blocks(n, q8.block_size)
    _check(ms, np.float32, "m_scale", nb)
    _check(vs, np.float32, "v_scale", nb)
    b0, b1 = blocks if blocks is not None else (0, nb)
    assert 0 <= b0 <= b1 <= nb
    gp, gb = _grad(g, n)
    _lib.orc_step_q8(n, _ptr(p, ctypes.c_float), gp, gb, _ptr(mc, ctypes.c_int8), _ptr(vc, ctypes.c_uint8),
                     _ptr(ms, ctypes.c_float), _ptr(vs, ctypes.c_float), ctypes.byref(hp._c()), t,
                     ctypes.byref(q8._c()), tensor_idx, b0, b1)


def step_q8_block(p, g, mc, vc, ms, vs, t: int, hp: HParams, q8: Q8Opts, tensor_idx: int, elem0: int) -> None:
    """8-bit step of one block held in its own arrays: ``p, g, mc, vc`` are the block's
    elements (at most ``q8.block_size``), ``ms, vs`` one-element scale arrays, ``elem0`` the block's first
    element index within its tensor (it keys the stochastic-rounding stream)."""
    n = p.size
    assert 0 < n <= q8.block_size and elem0 % q8.block_size == 0
    _check(p, np.float32, "param")
    _check(mc, np.int8, "m_code", n)
    _check(vc, np.uint8, "v_code", n)
    _check(ms, np.float32, "m_scale", 1)
    _check(vs, np.float32, "v_scale", 1)
    gp, gb = _grad(g, n)
    _lib.orc_step_q8_block(n, elem0, _ptr(p, ctypes.c_float), gp, gb, _ptr(mc, ctypes.c_int8),
                           _ptr(vc, ctypes.c_uint8), _ptr(ms, ctypes.c_float), _ptr(vs, ctypes.c_float),
                           ctypes.byref(hp._c()), t, ctypes.byref(q8._c()), tensor_idx)


def step_q8v(p, g, m, vc, vs, t: int, hp: HParams, q8: Q8Opts = Q8Opts(), tensor_idx: int = 0,
             blocks: tuple[int, int] | None = None) -> None:
    """fp32 m, 8-bit v (CompressBothMoments = false) over blocks [b0, b1) of one tensor."""
    n = p.size
    _check(p, np.float32, "param")
    _check(m, np.float32, "m", n)
    _check(vc, np.uint8, "v_code", n)
    nb = n_blocks(n, q8.block_size)
    _check(vs, np.float32, "v_scale", nb)
    b0, b1 = blocks if blocks is not None else (0, nb)
    assert 0 <= b0 <= b1 <= nb
    gp, gb = _grad(g, n)
    _lib.orc_step_q8v(n, _ptr(p, ctypes.c_float), gp, gb, _ptr(m, ctypes.c_float), _ptr(vc, ctypes.c_uint8),
                      _ptr(vs, ctypes.c_float), ctypes.byref(hp._c()), t, ctypes.byref(q8._c()), tensor_idx, b0, b1)


def step_q8v_block(p, g, m, vc, vs, t: int, hp: HParams, q8: Q8Opts, tensor_idx: int, elem0: int) -> None:
    """One block of the fp32-m / 8-bit-v step, held in its own arrays (see step_q8_block)."""
    n = p.size
    assert 0 < n <= q8.block_size and elem0 % q8.block_size == 0
    _check(p, np.float32, "param")
    _check(m, np.float32, "m", n)
    _check(vc, np.uint8, "v_code", n)
    _check(vs, np.float32, "v_scale", 1)
    gp, gb = _grad(g, n)
    _lib.orc_step_q8v_block(n, elem0, _ptr(p, ctypes.c_float), gp, gb, _ptr(m, ctypes.c_float),
                            _ptr(vc, ctypes.c_uint8), _ptr(vs, ctypes.c_float), ctypes.byref(hp._c()), t,
                            ctypes.byref(q8._c()), tensor_idx)


# ---------------------------------------------------------------- multi-tensor lists
def step_list(mode: str, params, grads, state, t: int, hp: HParams, q8: Q8Opts = Q8Opts()) -> None:
    """Step a list of tensors; tensor i of the list is tensor_idx i of the stochastic-rounding
    stream. ``state[i]`` is (m, v) for fp32/bf16m, (mc, vc, ms, vs) for q8 and (m, vc, vs)
    for q8v (fp32 m, 8-bit v)."""
    for i, (p, g, st) in enumerate(zip(params, grads, state)):
        if mode == "fp32":
            step_fp32(p, g, *st, t, hp)
        elif mode == "bf16m":
            step_bf16m(p, g, *st, t, hp)
        elif mode == "q8":
            step_q8(p, g, *st, t, hp, q8, tensor_idx=i)
        elif mode == "q8v":
            step_q8v(p, g, *st, t, hp, q8, tensor_idx=i)
        else:
            raise ValueError(mode)


def unscale_grads(g: np.ndarray, unscale: float) -> np.ndarray:
    """The grads the update sees: g * unscale in fp32 (bf16 bits widened first)."""
    n = g.size
    gp, gb = _grad(g, n)
    out = np.empty(n, np.float32)
    _lib.orc_unscale_grads(n, gp, gb, unscale, _ptr(out, ctypes.c_float))
    return out


def probe_mul_add(a: float, b: float, c: float) -> np.float32:
    return np.float32(_lib.orc_probe_mul_add(a, b, c))


LIB_PATH = _build.LIB
