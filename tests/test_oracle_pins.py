"""Pins for the CPU oracle: each test checks it against something other than itself —
closed forms, special cases that reduce to plain arithmetic, library routines (torch's
bf16 conversion, numpy's nearest-rank percentile, Triton's Philox in its CPU
interpreter), brute force on tiny inputs, and a float64 textbook Adam.

Sources: AiDotNet PR #814 "add 8-bit Adam optimizer for memory efficiency" (block-wise
8-bit moments: block 2048, signed m / unsigned v, percentile scaling, stochastic
rounding, sequence diagram of one step); AiDotNet PR #1745 "make BF16-Adam
fused-compatible" (bf16 moment storage); Kingma & Ba, Adam, Algorithm 1; Loshchilov &
Hutter, decoupled weight decay; Salmon et al. SC'11, Philox4x32-10.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import HParams, Q8Opts
import workloads

F32 = np.float32


def ulp(x):
    return np.spacing(np.abs(np.asarray(x, dtype=np.float32))).astype(np.float64)


# --------------------------------------------------------------------------- build flags
def test_build_keeps_two_roundings():
    # a*b = 1 + 2^-11 + 2^-24 exactly; rounding the product first gives 1 + 2^-11, so
    # a*b + c is 0 with two roundings and 2^-24 when fused.
    a = b = float(F32(1 + 2 ** -12))
    c = float(F32(-(1 + 2 ** -11)))
    assert oracle.probe_mul_add(a, b, c) == 0.0
    # the fused value (exact in float64, then one rounding) is what a contracted build returns
    assert F32(np.float64(a) * np.float64(b) + np.float64(c)) == F32(2 ** -24)


# --------------------------------------------------------------------------- Philox
def _triton_philox(ctr: np.ndarray, seed: int) -> np.ndarray:
    """Philox4x32-10 from Triton's own implementation, run by its CPU interpreter."""
    os.environ["TRITON_INTERPRET"] = "1"
    triton = pytest.importorskip("triton")
    import triton.language as tl

    @triton.jit
    def kern(out_ptr, c_ptr, seed, N: tl.constexpr):
        i = tl.arange(0, N)
        c0 = tl.load(c_ptr + 4 * i + 0)
        c1 = tl.load(c_ptr + 4 * i + 1)
        c2 = tl.load(c_ptr + 4 * i + 2)
        c3 = tl.load(c_ptr + 4 * i + 3)
        a, b, c, d = tl.philox(seed, c0, c1, c2, c3)
        tl.store(out_ptr + 4 * i + 0, a)
        tl.store(out_ptr + 4 * i + 1, b)
        tl.store(out_ptr + 4 * i + 2, c)
        tl.store(out_ptr + 4 * i + 3, d)

    n = ctr.shape[0]
    c = torch.from_numpy(ctr.astype(np.uint32).view(np.int32).copy().reshape(-1))
    out = torch.empty_like(c)
    kern[(1,)](out, c, seed, N=n)
    return out.numpy().view(np.uint32).reshape(n, 4)


def test_philox_matches_triton_interpreter():
    rng = np.random.default_rng(7)
    seeds = [0, 42, 0xFFFFFFFF, 0x123456789ABCDEF0, (1 << 64) - 1]
    for seed in seeds:
        ctr = rng.integers(0, 2 ** 32, size=(64, 4), dtype=np.uint64).astype(np.uint32)
        ctr[0] = 0
        ctr[1] = 0xFFFFFFFF
        key = np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint32)
        want = _triton_philox(ctr, seed if seed < (1 << 63) else seed - (1 << 64))
        got = oracle.philox4x32_10(ctr, key)
        np.testing.assert_array_equal(got, want)


def test_philox_output_is_uniform():
    n = 1 << 16
    ctr = np.zeros((n, 4), np.uint32)
    ctr[:, 0] = np.arange(n, dtype=np.uint32)
    out = oracle.philox4x32_10(ctr, np.array([42, 0], np.uint32)).ravel()
    counts = np.bincount(out >> 24, minlength=256)
    expect = out.size / 256
    chi2 = ((counts - expect) ** 2 / expect).sum()
    assert chi2 < 255 + 6 * math.sqrt(2 * 255)  # ~6 sigma
    bits = (out[:, None] >> np.arange(32, dtype=np.uint32)) & 1
    assert np.all(np.abs(bits.mean(0) - 0.5) < 6 * 0.5 / math.sqrt(out.size))


def test_sr_uniform_stream_layout():
    # element e of tensor i, moment mo, step t draws word e%4 of Philox(ctr=(e//4, 0, t, 2i+mo), key=seed)
    seed, step, ti = 0xDEADBEEF12345678, 7, 3
    for mo in (0, 1):
        for e in (0, 1, 2, 3, 4, 5, 2049, 123457):
            ctr = np.array([[e // 4, 0, step, 2 * ti + mo]], np.uint32)
            word = oracle.philox4x32_10(ctr, np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32))[0, e % 4]
            assert oracle.sr_uniform(seed, step, ti, mo, e) == float(word >> 8) * 2.0 ** -24
    us = np.array([oracle.sr_uniform(1, 1, 0, 0, e) for e in range(20000)])
    assert us.min() >= 0.0 and us.max() < 1.0
    assert abs(us.mean() - 0.5) < 6 * math.sqrt(1 / 12 / us.size)


# --------------------------------------------------------------------------- bf16 storage
def test_bf16_round_exhaustive_against_torch():
    """All 2^32 fp32 bit patterns against torch's fp32->bf16 conversion (round to nearest
    even); NaNs must stay NaN with their sign."""
    from concurrent.futures import ThreadPoolExecutor
    chunk = 1 << 24
    base = np.arange(chunk, dtype=np.uint32)

    def check(start):
        bits = base + np.uint32(start)
        x = bits.view(np.float32)
        got = oracle.bf16_round(x)  # the C loop runs without the GIL
        want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(x)
        if not nan.any():
            return bool(np.array_equal(got, want))
        g = got[nan]
        return bool(np.array_equal(got[~nan], want[~nan])
                    and np.all((g & 0x7F80) == 0x7F80) and np.all((g & 0x007F) != 0)
                    and np.all((g & 0x8000) == ((bits[nan] >> 16) & 0x8000)))

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        ok = list(ex.map(check, range(0, 1 << 32, chunk)))
    assert all(ok), [i for i, o in enumerate(ok) if not o][:8]


def test_bf16_widen_exhaustive_against_torch():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_widen(b)
    want = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(want)
    np.testing.assert_array_equal(got.view(np.uint32)[~nan], want.view(np.uint32)[~nan])
    assert np.all(np.isnan(got[nan]))
    # widening keeps every bit: the bf16 pattern is the top half of the fp32
    np.testing.assert_array_equal(got.view(np.uint32) >> 16, b.astype(np.uint32))


# --------------------------------------------------------------------------- step constants
def test_bias_correction_special_values():
    lr = 2.0 ** -10
    s = oracle.scalars(HParams(lr=lr, beta1=0.5, beta2=0.75, eps=1e-8, weight_decay=2.0 ** -3), 1)
    assert s["step_size"] == F32(2 * lr)           # bc1 = 1 - 0.5 = 1/2
    assert s["inv_sqrt_bc2"] == F32(2.0)           # bc2 = 1 - 0.75 = 1/4
    assert s["decay"] == F32(1 - 2.0 ** -13)       # 1 - lr*wd, exact
    assert s["omb1"] == F32(0.5) and s["omb2"] == F32(0.25)
    s2 = oracle.scalars(HParams(lr=lr, beta1=0.5, beta2=0.75), 2)
    assert s2["step_size"] == F32(lr / 0.75)       # bc1 = 3/4
    assert s2["inv_sqrt_bc2"] == F32(1 / math.sqrt(1 - 0.5625))
    s_inf = oracle.scalars(HParams(lr=1e-3, beta1=0.9, beta2=0.999, weight_decay=0.0), 10 ** 6)
    assert s_inf["step_size"] == F32(1e-3) and s_inf["inv_sqrt_bc2"] == F32(1.0)
    assert s_inf["decay"] == F32(1.0)


# --------------------------------------------------------------------------- Adam/AdamW
def _textbook_adamw(p, grads, hp: HParams):
    """float64 Adam (Kingma & Ba, Algorithm 1) with decoupled weight decay; the
    hyper-parameters are the float32 values the caller passes."""
    lr, b1, b2, eps, wd = (float(F32(x)) for x in (hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay))
    p = p.astype(np.float64)
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    for t, g in enumerate(grads, start=1):
        g = g.astype(np.float64)
        m = b1 * m + (1 - b1) * g
        v = b2 * v + (1 - b2) * g * g
        m_hat = m / (1 - b1 ** t)
        v_hat = v / (1 - b2 ** t)
        p = p - lr * wd * p - lr * m_hat / (np.sqrt(v_hat) + eps)
    return p, m, v


def _fresh(n, seed=0, std=1e-2):
    rng = np.random.default_rng(seed)
    p = (rng.standard_normal(n) * 0.02).astype(F32)
    g = (rng.standard_normal(n) * std).astype(F32)
    return p, g


def test_first_step_closed_form():
    """t = 1 from zero state: m' = (1-b1) g, v' = (1-b2) g^2, so bias correction cancels and
    p' = p (1 - lr wd) - lr g / (|g| + eps)."""
    hp = HParams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    p0, g = _fresh(4096, seed=1)
    g[:4] = [0.0, 1e-9, -1e-9, 3.0]  # around eps and far above it
    for mode in ("fp32", "bf16m", "q8"):
        p = p0.copy()
        if mode == "fp32":
            oracle.step_fp32(p, g, np.zeros_like(p), np.zeros_like(p), 1, hp)
        elif mode == "bf16m":
            oracle.step_bf16m(p, g, np.zeros(p.size, np.uint16), np.zeros(p.size, np.uint16), 1, hp)
        else:
            nb = oracle.n_blocks(p.size)
            oracle.step_q8(p, g, np.zeros(p.size, np.int8), np.zeros(p.size, np.uint8),
                           np.zeros(nb, F32), np.zeros(nb, F32), 1, hp)
        lr, wd, eps = float(F32(hp.lr)), float(F32(hp.weight_decay)), float(F32(hp.eps))
        gd = g.astype(np.float64)
        want = p0 * (1 - lr * wd) - lr * gd / (np.abs(gd) + eps)
        err = np.abs(p.astype(np.float64) - want)
        assert np.all(err <= 1e-6 * lr + 2 * ulp(want)), (mode, err.max())


def test_zero_grad_is_pure_decay():
    """g = 0 from zero state: m and v stay 0, the Adam term is 0/eps = 0, and each step
    multiplies p by decay = 1 - lr*wd."""
    hp = HParams(lr=1e-3, weight_decay=0.1)
    p, _ = _fresh(3000, seed=2)
    p0 = p.copy()
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    decay = oracle.scalars(hp, 1)["decay"]
    assert decay == F32(1 - float(F32(1e-3)) * float(F32(0.1)))
    want = p0.copy()
    for t in range(1, 6):
        oracle.step_fp32(p, np.zeros_like(p), m, v, t, hp)
        want = (want * decay).astype(F32)
        np.testing.assert_array_equal(p, want)
    assert not m.any() and not v.any()
    exact = p0.astype(np.float64) * (1 - float(F32(1e-3)) * float(F32(0.1))) ** 5
    assert np.all(np.abs(p - exact) <= 4 * ulp(exact))


def test_zero_betas_give_sign_descent():
    """b1 = b2 = 0, wd = 0: m' = g, v' = g^2, bias corrections are 1, so every step is
    p' = p - lr g / (|g| + eps) regardless of history."""
    hp = HParams(lr=1e-3, beta1=0.0, beta2=0.0, eps=1e-8, weight_decay=0.0)
    p, _ = _fresh(2500, seed=3)
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    for t in range(1, 6):
        _, g = _fresh(p.size, seed=100 + t)
        prev = p.astype(np.float64)
        oracle.step_fp32(p, g, m, v, t, hp)
        gd = g.astype(np.float64)
        want = prev - float(F32(1e-3)) * gd / (np.abs(gd) + float(F32(1e-8)))
        assert np.all(np.abs(p - want) <= 1e-6 * 1e-3 + 2 * ulp(want))


@pytest.mark.parametrize("grad_bf16", [False, True])
def test_fp32_trajectory_matches_textbook_float64(grad_bf16):
    hp = HParams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    n, steps = 1000, 20
    p, _ = _fresh(n, seed=4)
    p0 = p.copy()
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    grads = []
    for t in range(1, steps + 1):
        g = workloads.grads_np([n], t, 1e-2, seed=4)[0]
        if grad_bf16:
            gb = workloads.to_bf16_bits_truncate(g)
            g = (gb.astype(np.uint32) << 16).view(F32)  # the value the step sees
            oracle.step_fp32(p, gb, m, v, t, hp)
        else:
            oracle.step_fp32(p, g, m, v, t, hp)
        grads.append(g)
    pt, mt, vt = _textbook_adamw(p0, grads, hp)
    # m is a signed sum that can cancel: bound its error by the size of what was summed
    mag = np.zeros(n)
    for g in grads:
        mag = 0.9 * mag + 0.1 * np.abs(g.astype(np.float64))
    assert np.all(np.abs(m - mt) <= 1e-6 * mag + 2e-6 * np.abs(mt))
    np.testing.assert_allclose(v, vt, rtol=2e-6, atol=1e-15)
    np.testing.assert_allclose(p - p0, pt - p0, rtol=1e-5, atol=1e-7)


def test_bf16m_step_is_fp32_step_then_torch_rounding():
    """bf16 moments: widen, take the fp32 step, store m and v rounded to bf16 (torch's
    round-to-nearest-even conversion)."""
    hp = HParams(weight_decay=0.01)
    n = 5000
    p, g = _fresh(n, seed=5)
    m32, v32 = workloads.random_moments_np(n, seed=6)
    mb = torch.from_numpy(m32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    vb = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    pa, ma, va = p.copy(), mb.copy(), vb.copy()
    oracle.step_bf16m(pa, g, ma, va, 3, hp)
    pf = p.copy()
    mf = torch.from_numpy(mb.view(np.int16)).view(torch.bfloat16).float().numpy().copy()
    vf = torch.from_numpy(vb.view(np.int16)).view(torch.bfloat16).float().numpy().copy()
    oracle.step_fp32(pf, g, mf, vf, 3, hp)
    np.testing.assert_array_equal(pa, pf)
    to_b = lambda x: torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ma, to_b(mf))
    np.testing.assert_array_equal(va, to_b(vf))


# --------------------------------------------------------------------------- quantization
def _brute_nearest(x, s, lo, hi):
    """Nearest code by exhaustive search in float64; ties to the even code."""
    codes = np.arange(lo, hi + 1, dtype=np.float64)
    d = np.abs(x.astype(np.float64)[:, None] - codes[None, :] * float(s))
    best = d.min(1, keepdims=True)
    cand = np.where(d == best, codes[None, :], np.nan)
    even = np.where(np.nanmin(cand, 1) % 2 == 0, np.nanmin(cand, 1), np.nanmax(cand, 1))
    return even


@pytest.mark.parametrize("n", [1, 2, 7, 100, 2047, 2048])
def test_quantize_block_brute_force(n):
    rng = np.random.default_rng(n)
    m = (rng.standard_normal(n) * 1e-3).astype(F32)
    v = (rng.exponential(1.0, n) * 1e-6).astype(F32)
    for x, signed, lo, hi in ((m, True, -127, 127), (v, False, 0, 255)):
        codes, s = oracle.quantize_block(x, signed)
        absmax = np.abs(x).max()
        assert s == F32(absmax) / F32(hi)
        ratio = x.astype(np.float64) / float(s)
        near_half = np.abs(ratio - np.floor(ratio) - 0.5) < 2.0 ** -16
        want = _brute_nearest(x, s, lo, hi)
        got = codes.astype(np.float64)
        assert np.all((got == want) | (near_half & (np.abs(got - ratio) <= 0.5 + 2.0 ** -16)))
        assert np.all(np.abs(x - got * float(s)) <= float(s) / 2 * (1 + 2.0 ** -20))
        i = int(np.argmax(np.abs(x)))
        assert got[i] == (np.sign(x[i]) * hi if signed else hi)
        assert got.min() >= lo and got.max() <= hi


def test_quantize_zero_and_degenerate_blocks():
    z = np.zeros(2048, F32)
    for signed in (True, False):
        codes, s = oracle.quantize_block(z, signed)
        assert s == 0.0 and not codes.any()
    one = np.array([-3e-4], F32)
    codes, s = oracle.quantize_block(one, True)
    assert codes[0] == -127 and s == F32(3e-4) / F32(127)
    eq = np.full(2048, 5e-7, F32)
    codes, s = oracle.quantize_block(eq, False)
    assert np.all(codes == 255)


def test_dequantize_is_code_times_its_block_scale():
    n = 5000
    rng = np.random.default_rng(9)
    mc = rng.integers(-127, 128, n).astype(np.int8)
    vc = rng.integers(0, 256, n).astype(np.uint8)
    ms = rng.random(oracle.n_blocks(n)).astype(F32)
    vs = rng.random(oracle.n_blocks(n)).astype(F32)
    m, v = oracle.dequantize(mc, vc, ms, vs)
    blk = np.arange(n) // 2048
    np.testing.assert_array_equal(m, mc.astype(F32) * ms[blk])
    np.testing.assert_array_equal(v, vc.astype(F32) * vs[blk])


def _np_nearest_rank(x, pct):
    return np.percentile(np.abs(x.astype(np.float64)), float(F32(pct)), method="inverted_cdf")


@pytest.mark.parametrize("pct", [100.0, 99.9, 99.5, 99.0, 90.0, 50.0])
def test_percentile_basis_matches_numpy_nearest_rank(pct):
    rng = np.random.default_rng(int(pct * 10))
    blocks = {
        "normal": (rng.standard_normal(2048) * 1e-3).astype(F32),
        "outlier": np.where(np.arange(2048) == 77, 1.0, rng.standard_normal(2048) * 1e-3).astype(F32),
        "ties": np.repeat(rng.standard_normal(16).astype(F32), 128),
        "three_nonzero": np.where(np.isin(np.arange(2048), [5, 600, 2000]), 1e-3, 0.0).astype(F32),
        "all_equal": np.full(2048, -2e-4, F32),
        "short_1000": (rng.standard_normal(1000) * 1e-3).astype(F32),
        "short_1001": (rng.standard_normal(1001) * 1e-3).astype(F32),
        "short_7": (rng.standard_normal(7) * 1e-3).astype(F32),
    }
    for name, x in blocks.items():
        k = oracle.percentile_rank(pct, x.size)
        basis = oracle.kth_largest_abs(x, k)
        assert basis == F32(_np_nearest_rank(x, pct)), name
        codes, s = oracle.quantize_block(x, True, Q8Opts(percentile=pct))
        use = basis if basis != 0 else np.abs(x).max()
        assert s == F32(use) / F32(127), name
        assert np.all(np.abs(codes.astype(np.int32)) <= 127)
    assert oracle.percentile_rank(99.9, 2048) == 3
    assert oracle.percentile_rank(100.0, 2048) == 1
    assert oracle.percentile_rank(99.9, 1000) == 1


def test_stochastic_rounding_brackets_and_is_unbiased():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(2048) * 1e-3).astype(F32)
    _, s = oracle.quantize_block(x, True)
    ratio = x.astype(np.float64) / float(s)
    trials = 2048
    acc = np.zeros(2048)
    for seed in range(trials):
        codes, s2 = oracle.quantize_block(x, True, Q8Opts(stochastic_rounding=True, seed=seed), step=1)
        assert s2 == s
        c = codes.astype(np.float64)
        assert np.all((c >= np.floor(ratio) - 1e-9) & (c <= np.floor(ratio) + 1 + 1e-9) | (np.abs(c) == 127))
        acc += c
    mean = acc / trials
    frac = ratio - np.floor(ratio)
    sigma = np.sqrt(np.maximum(frac * (1 - frac), 1e-4) / trials)
    inner = np.abs(ratio) < 126.5
    assert np.all(np.abs(mean - ratio)[inner] <= 5 * sigma[inner] + 1e-5)
    # reproducible from (seed, step, tensor index); each of them changes the stream
    base = oracle.quantize_block(x, True, Q8Opts(True, 5), step=3, tensor_idx=2)[0]
    np.testing.assert_array_equal(base, oracle.quantize_block(x, True, Q8Opts(True, 5), step=3, tensor_idx=2)[0])
    for other in (dict(q8=Q8Opts(True, 6), step=3, tensor_idx=2), dict(q8=Q8Opts(True, 5), step=4, tensor_idx=2),
                  dict(q8=Q8Opts(True, 5), step=3, tensor_idx=1)):
        assert (oracle.quantize_block(x, True, **other)[0] != base).any()


def _sr_expected_codes(x: np.ndarray, s: np.float32, seed: int, step: int, list_idx: int, moment: int,
                       elem0: int, qmin: int, qmax: int) -> np.ndarray:
    """clamp(floor(fl(fl(x / s) + u))) per element, with u drawn here straight from the Philox
    primitive (pinned to Triton's implementation): element e of list tensor i takes word e % 4
    of Philox4x32-10(counter = (e // 4 low, e // 4 high, step, 2 i + moment), key = seed) and
    u = (word >> 8) * 2^-24. e is the element's index within its whole tensor."""
    e = elem0 + np.arange(x.size, dtype=np.int64)
    grp = (e // 4).astype(np.uint64)
    ctr = np.stack([(grp & 0xFFFFFFFF).astype(np.uint32), (grp >> np.uint64(32)).astype(np.uint32),
                    np.full(x.size, step, np.uint32), np.full(x.size, 2 * list_idx + moment, np.uint32)], axis=1)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32)
    words = oracle.philox4x32_10(ctr, key)[np.arange(x.size), e % 4]
    u = ((words >> np.uint32(8)).astype(np.float64) * 2.0 ** -24).astype(F32)
    if s == 0:
        return np.zeros(x.size, np.int64)
    ratio = (x.astype(F32) / F32(s)).astype(F32)          # one IEEE fp32 division
    r = np.floor((ratio + u).astype(F32)).astype(np.int64)  # one fp32 addition, then floor
    return np.clip(r, qmin, qmax)


@pytest.mark.parametrize("mode", ["q8", "q8v"])
def test_sr_stream_keying_inside_the_step(mode):
    """The stochastic-rounding draw of every element inside a list step: element j of block b
    of list tensor i uses the stream position e = b*B + j within its whole tensor and list
    index i (PR #814 summary: stochastic rounding; the C# Random(42) replaced by a counter
    stream keyed by seed, step and index). The expected codes are built here from m', v' of
    the dequantize -> fp32 step decomposition and the Philox primitive alone, so dropping the
    block offset or keying by the wrong list index fails this test."""
    hp = HParams(lr=1e-3, weight_decay=0.01)
    seed = 0x1234_5678_9ABC_DEF1  # high key word in use
    sizes = [3000, 3 * 2048 + 77, 4 * 2048]  # list tensors 1 and 2: >= 3 blocks, a ragged tail
    q8 = Q8Opts(stochastic_rounding=True, seed=seed, percentile=100.0)
    params = [(_fresh(n, seed=40 + i)[0]) for i, n in enumerate(sizes)]
    state = []
    for n in sizes:
        nb = oracle.n_blocks(n)
        if mode == "q8":
            state.append((np.zeros(n, np.int8), np.zeros(n, np.uint8), np.zeros(nb, F32), np.zeros(nb, F32)))
        else:
            state.append((np.zeros(n, F32), np.zeros(n, np.uint8), np.zeros(nb, F32)))
    for t in (1, 2, 3):
        grads = workloads.grads_np(sizes, t, 1e-2, seed=41)
        # m', v' of this step: dequantize the state, then the fp32 step on copies
        mv_new = []
        for i, n in enumerate(sizes):
            st = state[i]
            if mode == "q8":
                m0, v0 = oracle.dequantize(st[0], st[1], st[2], st[3])
            else:
                m0 = st[0].copy()
                v0 = oracle.dequantize(np.zeros(n, np.int8), st[1], np.zeros_like(st[2]), st[2])[1]
            pf = params[i].copy()
            oracle.step_fp32(pf, grads[i], m0, v0, t, hp)
            mv_new.append((m0, v0))
        oracle.step_list(mode, params, grads, state, t, hp, q8)
        checked = 0
        for i, n in enumerate(sizes):
            m1, v1 = mv_new[i]
            st = state[i]
            for b in range(oracle.n_blocks(n)):
                lo, hi = b * 2048, min(n, (b + 1) * 2048)
                chans = [(v1[lo:hi], st[1][lo:hi], (st[3] if mode == "q8" else st[2])[b], 1, 0, 255)]
                if mode == "q8":
                    chans.append((m1[lo:hi], st[0][lo:hi], st[2][b], 0, -127, 127))
                for x, codes, s, moment, qmin, qmax in chans:
                    # absmax scale: one fp32 division of the block maximum by the code range
                    assert s == F32(F32(np.max(np.abs(x))) / F32(qmax))
                    want = _sr_expected_codes(x, s, seed, t, i, moment, lo, qmin, qmax)
                    np.testing.assert_array_equal(codes.astype(np.int64), want,
                                                  err_msg=f"{mode} step {t} tensor {i} block {b} moment {moment}")
                    checked += x.size
        assert checked >= sum(sizes)
    # the same block contents keyed by another list index or block offset give other codes
    x = mv_new[1][1][2048:4096]
    s = F32(F32(np.max(x)) / F32(255))
    base = _sr_expected_codes(x, s, seed, 3, 1, 1, 2048, 0, 255)
    assert (base != _sr_expected_codes(x, s, seed, 3, 0, 1, 2048, 0, 255)).any()
    assert (base != _sr_expected_codes(x, s, seed, 3, 1, 1, 0, 0, 255)).any()


def test_q8_step_uses_unquantized_moments_and_stores_their_codes():
    """From zero state the q8 step's params equal the fp32 step's bit for bit (the update
    reads m', v' before Quantize(m), Quantize(v)), and the stored codes are m', v'
    quantized."""
    hp = HParams(weight_decay=0.01)
    n = 2048 * 3 + 100
    p, g = _fresh(n, seed=12)
    pf, mf, vf = p.copy(), np.zeros_like(p), np.zeros_like(p)
    oracle.step_fp32(pf, g, mf, vf, 1, hp)
    nb = oracle.n_blocks(n)
    pq, mc, vc, ms, vs = p.copy(), np.zeros(n, np.int8), np.zeros(n, np.uint8), np.zeros(nb, F32), np.zeros(nb, F32)
    oracle.step_q8(pq, g, mc, vc, ms, vs, 1, hp)
    np.testing.assert_array_equal(pq, pf)
    mc2, vc2, ms2, vs2 = oracle.quantize(mf, vf, Q8Opts(), step=1)
    np.testing.assert_array_equal(mc, mc2)
    np.testing.assert_array_equal(vc, vc2)
    np.testing.assert_array_equal(ms, ms2)
    np.testing.assert_array_equal(vs, vs2)


def test_q8_block_range_equals_full_step():
    hp = HParams(weight_decay=0.1)
    n = 2048 * 5 + 17
    p, _ = _fresh(n, seed=13)
    nb = oracle.n_blocks(n)
    st_full = [p.copy(), np.zeros(n, np.int8), np.zeros(n, np.uint8), np.zeros(nb, F32), np.zeros(nb, F32)]
    st_part = [a.copy() for a in st_full]
    q8 = Q8Opts(stochastic_rounding=True, seed=42, percentile=99.9)
    for t in range(1, 4):
        g = workloads.grads_np([n], t, 1e-3, seed=13, kind="student_t_outliers")[0]
        oracle.step_q8(*st_full[:1], g, *st_full[1:], t, hp, q8, tensor_idx=4)
        for b0, b1 in ((0, 2), (2, 3), (3, nb)):
            oracle.step_q8(*st_part[:1], g, *st_part[1:], t, hp, q8, tensor_idx=4, blocks=(b0, b1))
    for a, b in zip(st_full, st_part):
        np.testing.assert_array_equal(a, b)


def test_q8_trajectory_tracks_fp32():
    """Quantized moments perturb the trajectory by at most the quantization error of m and
    v: over 20 steps the parameter changes stay close to the fp32-moment run."""
    hp = HParams(lr=1e-3)
    n = 4096
    p, _ = _fresh(n, seed=14)
    pf, mf, vf = p.copy(), np.zeros_like(p), np.zeros_like(p)
    nb = oracle.n_blocks(n)
    pq, mc, vc, ms, vs = p.copy(), np.zeros(n, np.int8), np.zeros(n, np.uint8), np.zeros(nb, F32), np.zeros(nb, F32)
    for t in range(1, 21):
        g = workloads.grads_np([n], t, 1e-3, seed=14)[0]
        oracle.step_fp32(pf, g, mf, vf, t, hp)
        oracle.step_q8(pq, g, mc, vc, ms, vs, t, hp)
    dq = pq - p
    df = pf - p
    assert np.median(np.abs(dq - df)) < 0.1 * np.median(np.abs(df))


def test_state_memory_ratio():
    """[PR #814]: 8-bit state is about 2 bytes per parameter plus the per-block scales,
    roughly 4x less than two fp32 moments."""
    n = 1 << 24
    fp32_bytes = 2 * 4 * n
    q8_bytes = 2 * n + 2 * 4 * oracle.n_blocks(n)
    assert 3.99 < fp32_bytes / q8_bytes < 4.0


def test_q8v_keeps_m_exact_and_quantizes_v_only():
    """CompressBothMoments = false (PR #814): m stays fp32, so p and m follow the fp32-moment
    step bit for bit when v's quantization is lossless; from zero state they always do at
    t = 1, and v's codes are v' quantized as the unsigned channel of an 8-bit block."""
    hp = HParams(weight_decay=0.01)
    n = 2048 * 2 + 300
    p, g = _fresh(n, seed=21)
    pf, mf, vf = p.copy(), np.zeros_like(p), np.zeros_like(p)
    oracle.step_fp32(pf, g, mf, vf, 1, hp)
    nb = oracle.n_blocks(n)
    pq, mq, vc, vs = p.copy(), np.zeros_like(p), np.zeros(n, np.uint8), np.zeros(nb, F32)
    oracle.step_q8v(pq, g, mq, vc, vs, 1, hp)
    np.testing.assert_array_equal(pq, pf)
    np.testing.assert_array_equal(mq, mf)
    for b in range(nb):
        lo, hi = b * 2048, min(n, (b + 1) * 2048)
        codes, s = oracle.quantize_block(vf[lo:hi], False)
        np.testing.assert_array_equal(vc[lo:hi], codes)
        assert vs[b] == s
    # a second step: m is never quantized, so it equals the textbook recursion on the same g
    _, g2 = _fresh(n, seed=22)
    m_expect = (F32(0.9) * mq + F32(np.float32(1.0 - np.float64(F32(0.9)))) * g2).astype(F32)
    oracle.step_q8v(pq, g2, mq, vc, vs, 2, hp)
    np.testing.assert_array_equal(mq, m_expect)


def test_q8v_block_equals_range_step():
    hp = HParams(weight_decay=0.1)
    n = 2048 * 3 + 11
    p, g = _fresh(n, seed=23)
    nb = oracle.n_blocks(n)
    a = [p.copy(), np.zeros_like(p), np.zeros(n, np.uint8), np.zeros(nb, F32)]
    b = [x.copy() for x in a]
    q8 = Q8Opts(True, 9, 99.9)
    for t in (1, 2):
        oracle.step_q8v(a[0], g, a[1], a[2], a[3], t, hp, q8, tensor_idx=3)
        for blk in range(nb):
            lo, hi = blk * 2048, min(n, (blk + 1) * 2048)
            sub = [b[0][lo:hi].copy(), b[1][lo:hi].copy(), b[2][lo:hi].copy(), b[3][blk:blk + 1].copy()]
            oracle.step_q8v_block(sub[0], g[lo:hi].copy(), sub[1], sub[2], sub[3], t, hp, q8, 3, lo)
            b[0][lo:hi], b[1][lo:hi], b[2][lo:hi], b[3][blk] = sub[0], sub[1], sub[2], sub[3][0]
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_grad_unscale_is_one_rounding_of_the_product():
    rng = np.random.default_rng(31)
    g = (rng.standard_normal(5000) * 1e3).astype(F32)
    # a power-of-two inverse loss scale is exact
    np.testing.assert_array_equal(oracle.unscale_grads(g, 2.0 ** -10), np.ldexp(g, -10).astype(F32))
    np.testing.assert_array_equal(oracle.unscale_grads(g, 1.0), g)
    # otherwise: the product rounded once (float64 product of two floats is exact)
    u = float(F32(1 / 3))
    np.testing.assert_array_equal(oracle.unscale_grads(g, u), (g.astype(np.float64) * u).astype(F32))
    # bf16 grads are widened exactly first
    gb = workloads.to_bf16_bits_truncate(g)
    wide = (gb.astype(np.uint32) << 16).view(F32)
    np.testing.assert_array_equal(oracle.unscale_grads(gb, u), (wide.astype(np.float64) * u).astype(F32))
    # overflow of the product is an inf the check must catch
    assert np.isinf(oracle.unscale_grads(np.array([3e38], F32), 10.0)[0])


def test_static_scales_freeze_after_the_first_quantization():
    """UseDynamicQuantization = false (PR #814 options): the first step sets each block's
    scale as the dynamic mode would; later steps keep it, and codes are the nearest code
    under the kept scale, saturating."""
    hp = HParams(lr=1e-3, weight_decay=0.0)
    n = 2048 * 2 + 77
    p, g1 = _fresh(n, seed=51, std=1e-3)
    nb = oracle.n_blocks(n)
    q_dyn, q_sta = Q8Opts(), Q8Opts(static_scales=True)
    sd = [p.copy(), np.zeros(n, np.int8), np.zeros(n, np.uint8), np.zeros(nb, F32), np.zeros(nb, F32)]
    ss = [x.copy() for x in sd]
    oracle.step_q8(*sd[:1], g1, *sd[1:], 1, hp, q_dyn)
    oracle.step_q8(*ss[:1], g1, *ss[1:], 1, hp, q_sta)
    for a, b in zip(sd, ss):
        np.testing.assert_array_equal(a, b)
    # step 2 with grads 4x larger: the kept scales saturate some codes
    _, g2 = _fresh(n, seed=52, std=4e-3)
    m1, v1 = oracle.dequantize(*ss[1:])
    pf, mf, vf = ss[0].copy(), m1.copy(), v1.copy()
    oracle.step_fp32(pf, g2, mf, vf, 2, hp)
    s_m, s_v = ss[3].copy(), ss[4].copy()
    oracle.step_q8(*ss[:1], g2, *ss[1:], 2, hp, q_sta)
    np.testing.assert_array_equal(ss[3], s_m)
    np.testing.assert_array_equal(ss[4], s_v)
    np.testing.assert_array_equal(ss[0], pf)
    blk = np.arange(n) // 2048
    for x, codes, s, lo, hi in ((mf, ss[1], s_m, -127, 127), (vf, ss[2], s_v, 0, 255)):
        ratio = x.astype(np.float64) / s[blk].astype(np.float64)
        want = np.clip(np.rint(ratio), lo, hi)
        near_half = np.abs(ratio - np.floor(ratio) - 0.5) < 2.0 ** -16
        got = codes.astype(np.float64)
        assert np.all((got == want) | near_half)
    assert np.any(np.abs(ss[1].astype(int)) == 127) and np.mean(np.abs(ss[1].astype(int)) == 127) > 0.01


# --------------------------------------------------------------------------- block size
@pytest.mark.parametrize("bs", [1, 3, 100, 777, 4096])
def test_quantize_any_block_size_brute_force(bs):
    """BlockSize (PR #814 options: any positive size): each block of bs consecutive
    elements, the last one partial, gets its own absmax scale; every code is the nearest
    code under that scale by exhaustive search."""
    n = 3 * bs + (bs // 2 if bs > 1 else 0) + 1
    rng = np.random.default_rng(bs)
    m = (rng.standard_normal(n) * 1e-3).astype(F32)
    v = (rng.exponential(1.0, n) * 1e-6).astype(F32)
    q8 = Q8Opts(block_size=bs)
    mc, vc, ms, vs = oracle.quantize(m, v, q8)
    nb = -(-n // bs)
    assert ms.size == vs.size == nb
    for b in range(nb):
        sl = slice(b * bs, min(n, (b + 1) * bs))
        for x, codes, s, lo, hi in ((m[sl], mc[sl], ms[b], -127, 127), (v[sl], vc[sl], vs[b], 0, 255)):
            assert s == F32(np.abs(x).max()) / F32(hi)
            ratio = x.astype(np.float64) / float(s)
            near_half = np.abs(ratio - np.floor(ratio) - 0.5) < 2.0 ** -16
            got = codes.astype(np.float64)
            assert np.all((got == _brute_nearest(x, s, lo, hi)) | near_half)
    # dequantize indexes scales by element // bs
    dm, dv = oracle.dequantize(mc, vc, ms, vs, block_size=bs)
    blk = np.arange(n) // bs
    np.testing.assert_array_equal(dm, mc.astype(F32) * ms[blk])
    np.testing.assert_array_equal(dv, vc.astype(F32) * vs[blk])


def test_block_size_one_is_sign_and_magnitude():
    """With one element per block the scale is |x|/qmax and every nonzero m codes to
    +-127, every nonzero v to 255 (|x/s| = qmax within one rounding of s)."""
    rng = np.random.default_rng(3)
    m = (rng.standard_normal(1000) * 1e-3).astype(F32)
    m[::97] = 0.0
    v = (np.abs(rng.standard_normal(1000)) * 1e-6).astype(F32)
    v[::89] = 0.0
    mc, vc, ms, vs = oracle.quantize(m, v, Q8Opts(block_size=1))
    np.testing.assert_array_equal(mc, (np.sign(m) * 127).astype(np.int8))
    np.testing.assert_array_equal(vc, np.where(v > 0, 255, 0).astype(np.uint8))
    np.testing.assert_array_equal(ms, np.abs(m) / F32(127))
    np.testing.assert_array_equal(vs, v / F32(255))


@pytest.mark.parametrize("bs", [64, 1000, 5000])
def test_q8_step_any_block_size_is_dequantize_update_quantize(bs):
    """The 8-bit step with block size bs is PR #814's diagram with that blocking: step 1
    from zero state equals the fp32 step (params bit for bit, codes = quantize(m', v')),
    and step 2 equals dequantize -> fp32 step -> quantize, all with block size bs."""
    hp = HParams(weight_decay=0.01)
    n = 2 * bs + bs // 3 + 5
    p, g1 = _fresh(n, seed=bs)
    q8 = Q8Opts(percentile=99.0, block_size=bs)
    nb = oracle.n_blocks(n, bs)
    st = [p.copy(), np.zeros(n, np.int8), np.zeros(n, np.uint8), np.zeros(nb, F32), np.zeros(nb, F32)]
    pf, mf, vf = p.copy(), np.zeros_like(p), np.zeros_like(p)
    oracle.step_fp32(pf, g1, mf, vf, 1, hp)
    oracle.step_q8(*st[:1], g1, *st[1:], 1, hp, q8)
    np.testing.assert_array_equal(st[0], pf)
    for a, b in zip(st[1:], oracle.quantize(mf, vf, q8, step=1)):
        np.testing.assert_array_equal(a, b)
    _, g2 = _fresh(n, seed=bs + 1)
    m1, v1 = oracle.dequantize(*st[1:], block_size=bs)
    pf, mf, vf = st[0].copy(), m1, v1
    oracle.step_fp32(pf, g2, mf, vf, 2, hp)
    oracle.step_q8(*st[:1], g2, *st[1:], 2, hp, q8)
    np.testing.assert_array_equal(st[0], pf)
    for a, b in zip(st[1:], oracle.quantize(mf, vf, q8, step=2)):
        np.testing.assert_array_equal(a, b)
    # percentile 99 ranks within each block of bs (the last one partial): X_v is numpy's
    # nearest-rank percentile of that block
    for b in range(nb):
        sl = slice(b * bs, min(n, (b + 1) * bs))
        assert st[4][b] == F32(_np_nearest_rank(vf[sl], 99.0)) / F32(255)


def test_q8v_step_any_block_size():
    """fp32 m / 8-bit v with block size 300: m equals the fp32 step's m exactly and v's
    codes and scales equal quantizing the fp32 step's v with that block size."""
    hp = HParams(weight_decay=0.01)
    bs, n = 300, 1000
    p, g = _fresh(n, seed=77)
    q8 = Q8Opts(block_size=bs)
    nb = oracle.n_blocks(n, bs)
    pq, m, vc, vs = p.copy(), np.zeros(n, F32), np.zeros(n, np.uint8), np.zeros(nb, F32)
    pf, mf, vf = p.copy(), np.zeros_like(p), np.zeros_like(p)
    oracle.step_fp32(pf, g, mf, vf, 1, hp)
    oracle.step_q8v(pq, g, m, vc, vs, 1, hp, q8)
    np.testing.assert_array_equal(pq, pf)
    np.testing.assert_array_equal(m, mf)
    _, vc2, _, vs2 = oracle.quantize(mf, vf, q8, step=1)
    np.testing.assert_array_equal(vc, vc2)
    np.testing.assert_array_equal(vs, vs2)
