"""Helpers shared by the GPU parity tests: run the same seeded inputs through the CUDA
library and the CPU oracle, and compare element by element.

Tolerances (the contract): after a trajectory, params max relative error <= 1e-5 and
m/v (dequantized for 8-bit) <= 1e-3 relative, denominator max(|oracle|, 1e-30);
8-bit codes may differ by +-1 in at most 0.01% of elements; quantize-only codes and
scales are bit-exact. Both sides evaluate the same IEEE single-precision operations in
the same order, so in practice the results are identical, and the tests also report
the exact-match fraction.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import HParams, Q8Opts

PARAM_RTOL = 1e-5
MOMENT_RTOL = 1e-3
CODE_DIFF_FRACTION = 1e-4


def rel_err(got: np.ndarray, want: np.ndarray) -> float:
    got = got.astype(np.float64)
    want = want.astype(np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - want) / np.maximum(np.abs(want), 1e-30)))


def assert_params(got, want, what=""):
    e = rel_err(got, want)
    assert e <= PARAM_RTOL, f"{what}: params max rel err {e:.3g} > {PARAM_RTOL}"


def assert_moment(got, want, what=""):
    e = rel_err(got, want)
    assert e <= MOMENT_RTOL, f"{what}: moment max rel err {e:.3g} > {MOMENT_RTOL}"


def assert_codes(got, want, what=""):
    d = np.abs(got.astype(np.int32) - want.astype(np.int32))
    assert d.max(initial=0) <= 1, f"{what}: code differs by {d.max()}"
    frac = np.count_nonzero(d) / max(d.size, 1)
    assert frac <= CODE_DIFF_FRACTION, f"{what}: {frac:.3g} of codes differ"


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_from_bits(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(a.view(np.int16).copy()).to(device).view(torch.bfloat16)


def host_state(mode: str, sizes, block_size: int = oracle.BLOCK):
    if mode == "fp32":
        return [(np.zeros(n, np.float32), np.zeros(n, np.float32)) for n in sizes]
    if mode == "bf16m":
        return [(np.zeros(n, np.uint16), np.zeros(n, np.uint16)) for n in sizes]
    nb = lambda n: oracle.n_blocks(n, block_size)
    if mode == "q8v":
        return [(np.zeros(n, np.float32), np.zeros(n, np.uint8), np.zeros(nb(n), np.float32)) for n in sizes]
    return [(np.zeros(n, np.int8), np.zeros(n, np.uint8), np.zeros(nb(n), np.float32), np.zeros(nb(n), np.float32))
            for n in sizes]


def device_state_to_host(mode: str, state, i: int):
    if mode == "fp32":
        return state[0][i].cpu().numpy(), state[1][i].cpu().numpy()
    if mode == "bf16m":
        return bf16_bits(state[0][i]), bf16_bits(state[1][i])
    return tuple(s[i].cpu().numpy() for s in state)


def compare_state(mode: str, got, want, what: str, block_size: int = oracle.BLOCK):
    if mode == "fp32":
        assert_moment(got[0], want[0], what + " m")
        assert_moment(got[1], want[1], what + " v")
    elif mode == "bf16m":
        gm = (got[0].astype(np.uint32) << 16).view(np.float32)
        wm = (want[0].astype(np.uint32) << 16).view(np.float32)
        gv = (got[1].astype(np.uint32) << 16).view(np.float32)
        wv = (want[1].astype(np.uint32) << 16).view(np.float32)
        assert_moment(gm, wm, what + " m")
        assert_moment(gv, wv, what + " v")
    elif mode == "q8v":
        assert_moment(got[0], want[0], what + " m")
        assert_codes(got[1], want[1], what + " v codes")
        assert_moment(got[2], want[2], what + " v scales")
        same = got[1] == want[1]
        gv = got[1].astype(np.float32) * np.repeat(got[2], block_size)[: got[1].size]
        wv = want[1].astype(np.float32) * np.repeat(want[2], block_size)[: want[1].size]
        assert_moment(gv[same], wv[same], what + " v (dequantized)")
    else:
        assert_codes(got[0], want[0], what + " m codes")
        assert_codes(got[1], want[1], what + " v codes")
        gm, gv = oracle.dequantize(*got, block_size=block_size)
        wm, wv = oracle.dequantize(*want, block_size=block_size)
        # a code off by one moves its value by one scale step: compare where codes agree
        same_m = got[0] == want[0]
        same_v = got[1] == want[1]
        assert_moment(got[2], want[2], what + " m scales")
        assert_moment(got[3], want[3], what + " v scales")
        assert_moment(gm[same_m], wm[same_m], what + " m (dequantized)")
        assert_moment(gv[same_v], wv[same_v], what + " v (dequantized)")


def exact_fraction(mode: str, got, want) -> float:
    flat_g = np.concatenate([np.ascontiguousarray(a).view(np.uint8).ravel() for a in got])
    flat_w = np.concatenate([np.ascontiguousarray(a).view(np.uint8).ravel() for a in want])
    if flat_w.size == 0:
        return 1.0
    return float(np.mean(flat_g == flat_w))


def hp_kwargs(hp: HParams) -> dict:
    return dict(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, weight_decay=hp.weight_decay)


def q8_kwargs(q8: Q8Opts, step: bool = True) -> dict:
    kw = dict(stochastic_rounding=q8.stochastic_rounding, seed=q8.seed, percentile=q8.percentile,
              block_size=q8.block_size)
    if step:
        kw["static_scales"] = q8.static_scales
    return kw
