"""GPU parity: libpsadam.so (called through its C ABI via the thin binding) against the
CPU oracle on identical seeded inputs, element by element.

Covers every moment mode (fp32, bf16, 8-bit), both grad dtypes, round-to-nearest and
stochastic rounding, absmax and percentile scaling, ragged multi-tensor lists (sizes
1, 2, 7, 2047, 2048, 2049, 4097, ...), lists longer than one launch, the quantize-only
and dequantize-only entry points (bit-exact), exhaustive bf16 rounding through the step
kernel, resume-equals-uninterrupted, and the workloads at full size (sampled blocks where
the oracle cannot run the whole tensor; the update is block-local, so a sampled block is
checked exactly).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import HParams, Q8Opts
import workloads
from parity_util import (assert_codes, assert_moment, assert_params, bf16_bits, compare_state,
                         device_state_to_host, exact_fraction, host_state, hp_kwargs, q8_kwargs)

pytestmark = pytest.mark.gpu

RAGGED = [1, 2, 7, 2047, 2048, 2049, 4097, 70001]


@pytest.fixture(scope="module")
def psa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import precision_state_adam_gb300 as psa
    return psa


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


DEV = "cuda:0"


def _to_dev(arrs, dtype=None):
    out = []
    for a in arrs:
        if a.dtype == np.uint16:  # bf16 bits
            out.append(torch.from_numpy(a.view(np.int16).copy()).to(DEV).view(torch.bfloat16))
        else:
            out.append(torch.from_numpy(a.copy()).to(DEV))
    return out


def run_both(psa, mode, sizes, steps, hp, q8=Q8Opts(), grad_dtype="f32", grad_kind="normal", grad_std=1e-2,
             seed=5, init_state=None, approx=False):
    """Run `steps` steps on the GPU and in the oracle from the same inputs; return both."""
    specs = [workloads.TensorSpec(f"t{i}", (n,)) for i, n in enumerate(sizes)]
    p_host = workloads.init_params_np(specs, seed=seed)
    params = _to_dev(p_host)
    ostate = host_state(mode, sizes, q8.block_size) if init_state is None else init_state
    state = psa.zeros_state(params, mode, q8.block_size)
    if init_state is not None:
        for k, arrs in enumerate(zip(*init_state)):
            for i, a in enumerate(arrs):
                state[k][i].copy_(_to_dev([a])[0])
    for t in range(1, steps + 1):
        g32 = workloads.grads_np(sizes, t, grad_std, seed=seed, kind=grad_kind)
        g_host = [workloads.to_bf16_bits_truncate(g) for g in g32] if grad_dtype == "bf16" else g32
        grads = _to_dev(g_host)
        kw = hp_kwargs(hp)
        if mode in ("q8", "q8v"):
            kw.update(q8_kwargs(q8))
        psa.adam_step(mode, params, grads, state, t, approx_update=approx, **kw)
        oracle.step_list(mode, p_host, g_host, ostate, t, hp, q8)
    torch.cuda.synchronize()
    got_p = [p.cpu().numpy() for p in params]
    got_s = [device_state_to_host(mode, state, i) for i in range(len(sizes))]
    return got_p, p_host, got_s, ostate


def check_all(mode, got_p, want_p, got_s, want_s, what, block_size=oracle.BLOCK, approx=False):
    """The contract's tolerances, and beyond them bit for bit: m, v, codes and scales always
    (they never depend on the update's square root or quotient), the params unless the
    approximate update ran. That one is checked normwise: its error is a few ulp of the
    update term, which is not elementwise-relative where a param passes near zero."""
    for i in range(len(got_p)):
        if approx:
            scale = max(float(np.max(np.abs(want_p[i]), initial=0.0)), 1e-30)
            err = float(np.max(np.abs(got_p[i].astype(np.float64) - want_p[i]), initial=0.0)) / scale
            assert err <= 1e-6, f"{what} tensor {i}: params normwise rel err {err:.3g} (approximate update)"
        else:
            assert_params(got_p[i], want_p[i], f"{what} tensor {i}")
            pe = exact_fraction(mode, [got_p[i]], [want_p[i]])
            assert pe == 1.0, f"{what} tensor {i}: params not bit-identical ({pe})"
        compare_state(mode, got_s[i], want_s[i], f"{what} tensor {i}", block_size)
        se = exact_fraction(mode, list(got_s[i]), list(want_s[i]))
        assert se == 1.0, f"{what} tensor {i}: moments / codes / scales not bit-identical ({se})"


# ------------------------------------------------------------------ every mode on ragged lists
@pytest.mark.parametrize("approx", [False, True])
@pytest.mark.parametrize("grad_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", ["fp32", "bf16m"])
def test_step_ragged_list(psa, mode, grad_dtype, approx):
    hp = HParams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    got_p, want_p, got_s, want_s = run_both(psa, mode, RAGGED, 5, hp, grad_dtype=grad_dtype, approx=approx)
    check_all(mode, got_p, want_p, got_s, want_s, f"{mode}/{grad_dtype}", approx=approx)


Q8_CASES = {
    "rne_absmax": Q8Opts(False, 42, 100.0),
    "sr_absmax": Q8Opts(True, 42, 100.0),
    "rne_p99.9": Q8Opts(False, 42, 99.9),   # rank 3 of a full block
    "sr_p99.9": Q8Opts(True, 7, 99.9),
    "rne_p99.95": Q8Opts(False, 42, 99.95),  # rank 2 of a full block
    "rne_p99.85": Q8Opts(False, 42, 99.85),  # rank 4: the largest rank of the 2048-block kernels
    "rne_p99.5": Q8Opts(False, 42, 99.5),   # rank 11: the general kernel's radix select
    "rne_static": Q8Opts(False, 42, 100.0, True),  # scales kept after the first step
    "sr_static_p99.9": Q8Opts(True, 5, 99.9, True),
}


@pytest.mark.parametrize("approx", [False, True])
@pytest.mark.parametrize("mode", ["q8", "q8v"])
@pytest.mark.parametrize("grad_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", sorted(Q8_CASES))
def test_q8_step_ragged_list(psa, case, grad_dtype, mode, approx):
    hp = HParams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
    got_p, want_p, got_s, want_s = run_both(psa, mode, RAGGED, 5, hp, Q8_CASES[case], grad_dtype=grad_dtype,
                                            grad_kind="student_t_outliers", grad_std=1e-3, approx=approx)
    check_all(mode, got_p, want_p, got_s, want_s, f"{mode}/{case}/{grad_dtype}", approx=approx)


# ------------------------------------------------------------------ any block size, any percentile
# Power-of-two blocks of 16..1024 elements at rank 1 (no runtime options) run in the persistent
# kernel's 2048-element tiles as sub-blocks; the rest runs the general kernel (one CTA per tile
# of whole blocks, shared-memory staging, radix-select ranks).
ANY_CASES = {
    "bs16_sr": (Q8Opts(True, 5, 100.0, block_size=16), [1, 15, 17, 2047, 2063, 9000]),
    "bs32_rne": (Q8Opts(False, 42, 100.0, block_size=32), [31, 33, 4096, 5000]),
    "bs128_sr_p99.9": (Q8Opts(True, 7, 99.9, block_size=128), [1, 127, 129, 6000]),   # rank 1 at 128
    "bs512_p99.95": (Q8Opts(False, 42, 99.95, block_size=512), [511, 513, 2048, 9999]),  # rank 1 at 512
    "bs1024_sr": (Q8Opts(True, 8, 100.0, block_size=1024), [1023, 1025, 3000, 70001]),
    "bs1_rne": (Q8Opts(False, 42, 100.0, block_size=1), [1, 2, 33, 300]),
    "bs3_sr": (Q8Opts(True, 42, 100.0, block_size=3), [1, 2, 7, 1000]),
    "bs64_rne": (Q8Opts(False, 42, 100.0, block_size=64), [1, 63, 64, 65, 5000]),
    "bs100_sr_p99": (Q8Opts(True, 9, 99.0, block_size=100), [1, 99, 100, 101, 7777]),
    "bs256_static": (Q8Opts(False, 42, 100.0, True, block_size=256), [5, 256, 70001]),
    "bs1000_p90": (Q8Opts(False, 42, 90.0, block_size=1000), [17, 999, 1000, 1001, 12345]),
    "bs4096_sr_p99.9": (Q8Opts(True, 3, 99.9, block_size=4096), [1, 4095, 4097, 20000]),
    "bs16384_rne": (Q8Opts(False, 42, 100.0, block_size=16384), [1, 16383, 16385, 40000]),  # read twice
    "bs8192_sr": (Q8Opts(True, 13, 100.0, block_size=8192), [1, 8191, 8193, 30000]),        # q8: read twice
    "bs8192_static": (Q8Opts(False, 42, 100.0, True, block_size=8192), [5, 8192, 24577]),
    "bs2048_p90": (Q8Opts(False, 42, 90.0), RAGGED),            # rank 205: general kernel at 2048
    "bs2048_sr_p50": (Q8Opts(True, 11, 50.0), [1, 2047, 2049, 9000]),
    "bs2048_p99_static": (Q8Opts(False, 42, 99.0, True), [3000, 2048]),
}


@pytest.mark.parametrize("approx", [False, True])
@pytest.mark.parametrize("mode", ["q8", "q8v"])
@pytest.mark.parametrize("case", sorted(ANY_CASES))
def test_q8_any_block_size_and_rank(psa, case, mode, approx):
    q8, sizes = ANY_CASES[case]
    hp = HParams(lr=1e-3, weight_decay=0.1)
    gd = "bf16" if case.endswith("sr") else "f32"
    got_p, want_p, got_s, want_s = run_both(psa, mode, sizes, 4, hp, q8, grad_dtype=gd,
                                            grad_kind="student_t_outliers", grad_std=1e-3, approx=approx)
    check_all(mode, got_p, want_p, got_s, want_s, f"{mode}/{case}", q8.block_size, approx=approx)


@pytest.mark.parametrize("case", ["bs1_rne", "bs100_sr_p99", "bs1000_p90", "bs16384_rne", "bs2048_sr_p50"])
def test_quantize_dequantize_any_block_size(psa, case):
    q8, sizes = ANY_CASES[case]
    bs = q8.block_size
    ms, vs = [], []
    for i, n in enumerate(sizes):
        m, v = workloads.random_moments_np(n, seed=40 + i)
        ms.append(m)
        vs.append(v)
    dm, dv = _to_dev(ms), _to_dev(vs)
    mc, vc, msc, vsc = psa.zeros_state(dm, "q8", bs)
    psa.q8_quantize(dm, dv, mc, vc, msc, vsc, step=4, **q8_kwargs(q8, step=False))
    back_m = [torch.empty_like(x) for x in dm]
    back_v = [torch.empty_like(x) for x in dv]
    psa.q8_dequantize(mc, vc, msc, vsc, back_m, back_v, block_size=bs)
    torch.cuda.synchronize()
    for i in range(len(sizes)):
        want = oracle.quantize(ms[i], vs[i], q8, step=4, tensor_idx=i)
        got = (mc[i].cpu().numpy(), vc[i].cpu().numpy(), msc[i].cpu().numpy(), vsc[i].cpu().numpy())
        for g, w, name in zip(got, want, ("m codes", "v codes", "m scales", "v scales")):
            np.testing.assert_array_equal(np.ascontiguousarray(g).view(np.uint8), np.ascontiguousarray(w).view(np.uint8),
                                          err_msg=f"{case} tensor {i} {name}")
        wm, wv = oracle.dequantize(*want, block_size=bs)
        np.testing.assert_array_equal(back_m[i].cpu().numpy().view(np.uint32), wm.view(np.uint32))
        np.testing.assert_array_equal(back_v[i].cpu().numpy().view(np.uint32), wv.view(np.uint32))


@pytest.mark.parametrize("mode", ["fp32", "bf16m", "q8", "q8v"])
def test_approximate_update_error_is_a_few_ulp(psa, mode):
    """The opt-in approximate square root and quotient: over 20 steps each param stays
    within 8 ulp of the update term's size of the IEEE oracle (|p' - p'_oracle| <= 2^-20 *
    lr/(1-beta1^t) summed over the steps), every moment, code and scale bit-identical."""
    hp = HParams(lr=1e-3, weight_decay=0.01)
    steps = 20
    got_p, want_p, got_s, want_s = run_both(psa, mode, RAGGED, steps, hp, Q8Opts(True, 3, 99.9), grad_std=1e-3,
                                            approx=True)
    check_all(mode, got_p, want_p, got_s, want_s, f"{mode} {steps} steps", approx=True)
    # the update term |lr/bc1 * m/(sqrt(v)/sqrt(bc2) + eps)| is at most about lr/bc1 * 1/sqrt(1-beta2)
    bound = sum(2.0 ** -20 * hp.lr / (1 - hp.beta1 ** t) / np.sqrt(1 - hp.beta2) for t in range(1, steps + 1))
    for g, w in zip(got_p, want_p):
        err = float(np.max(np.abs(g.astype(np.float64) - w), initial=0.0))
        assert err <= bound, f"{mode}: params max abs err {err:.3g} > {bound:.3g}"


def test_zero_grads_are_pure_decay(psa):
    n = 10000
    p0 = workloads.init_params_np([workloads.TensorSpec("w", (n,))], seed=8)[0]
    for mode in ("fp32", "bf16m", "q8", "q8v"):
        params = _to_dev([p0])
        state = psa.zeros_state(params, mode)
        want = p0.copy()
        decay = oracle.scalars(HParams(lr=1e-3, weight_decay=0.1), 1)["decay"]
        for t in range(1, 4):
            psa.adam_step(mode, params, [torch.zeros(n, device=DEV)], state, t, lr=1e-3, weight_decay=0.1)
            want = (want * decay).astype(np.float32)
        np.testing.assert_array_equal(params[0].cpu().numpy(), want)


# ------------------------------------------------------------------ long lists: several launches
def test_long_list_spans_several_launches(psa):
    rng = np.random.default_rng(3)
    sizes = [int(x) for x in rng.integers(1, 3000, size=1000)]
    sizes[10] = 0  # an empty tensor in the middle of the list
    hp = HParams(weight_decay=0.01)
    q8 = Q8Opts(True, 99, 99.9)
    got_p, want_p, got_s, want_s = run_both(psa, "q8", sizes, 2, hp, q8, grad_std=1e-3)
    check_all("q8", got_p, want_p, got_s, want_s, "q8 long list")


# ------------------------------------------------------------------ quantize / dequantize only
@pytest.mark.parametrize("case", sorted(Q8_CASES))
def test_quantize_only_is_bit_exact(psa, case):
    q8 = Q8_CASES[case]
    sizes = RAGGED + [2048 * 5, 2048 * 4]
    ms, vs = [], []
    rng = np.random.default_rng(8)
    for i, n in enumerate(sizes):
        m, v = workloads.random_moments_np(n, seed=20 + i)
        if n == 2048 * 5:
            m[2048:4096] = 0.0  # an all-zero block
            v[2048:4096] = 0.0
            m[:2048] = 3e-4     # a constant block
            v[4096] = 1.0       # a single outlier
        if n == 2048 * 4:
            # block 0: the block's 8 largest all held by one thread (elements t*4 + i and
            # 1024 + t*4 + i of thread t); block 1: the maximum 6 times over; block 2: small
            # integers (ties everywhere); block 3: two non-zeros
            for j, e in enumerate([37 * 4 + i for i in range(4)] + [1024 + 37 * 4 + i for i in range(4)]):
                m[e] = (-1) ** j * (0.01 + j * 1e-3)
                v[e] = 0.01 + j * 1e-3
            top = rng.choice(2048, 6, replace=False) + 2048
            m[top], v[top] = -0.02, 0.02
            m[4096:6144] = rng.integers(-3, 4, 2048) * 1e-3
            v[4096:6144] = rng.integers(0, 4, 2048) * 1e-6
            m[6144:], v[6144:] = 0.0, 0.0
            m[6144 + 5], v[6144 + 5] = 1e-3, 1e-6
            m[6144 + 1500], v[6144 + 1500] = -2e-3, 3e-6
        ms.append(m)
        vs.append(v)
    dm, dv = _to_dev(ms), _to_dev(vs)
    mc, vc, msc, vsc = psa.zeros_state(dm, "q8")
    psa.q8_quantize(dm, dv, mc, vc, msc, vsc, step=9, **q8_kwargs(q8, step=False))
    torch.cuda.synchronize()
    for i, n in enumerate(sizes):
        want = oracle.quantize(ms[i], vs[i], q8, step=9, tensor_idx=i)
        got = (mc[i].cpu().numpy(), vc[i].cpu().numpy(), msc[i].cpu().numpy(), vsc[i].cpu().numpy())
        for g, w, name in zip(got, want, ("m codes", "v codes", "m scales", "v scales")):
            np.testing.assert_array_equal(np.ascontiguousarray(g).view(np.uint8), np.ascontiguousarray(w).view(np.uint8),
                                          err_msg=f"{case} tensor {i} {name}")


def test_dequantize_only_is_bit_exact(psa):
    rng = np.random.default_rng(4)
    sizes = RAGGED
    mc = [rng.integers(-127, 128, n).astype(np.int8) for n in sizes]
    vc = [rng.integers(0, 256, n).astype(np.uint8) for n in sizes]
    msc = [(rng.random(oracle.n_blocks(n)) * 1e-4).astype(np.float32) for n in sizes]
    vsc = [(rng.random(oracle.n_blocks(n)) * 1e-8).astype(np.float32) for n in sizes]
    dmc, dvc, dms, dvs = _to_dev(mc), _to_dev(vc), _to_dev(msc), _to_dev(vsc)
    m = [torch.empty(n, device=DEV) for n in sizes]
    v = [torch.empty(n, device=DEV) for n in sizes]
    psa.q8_dequantize(dmc, dvc, dms, dvs, m, v)
    torch.cuda.synchronize()
    for i in range(len(sizes)):
        wm, wv = oracle.dequantize(mc[i], vc[i], msc[i], vsc[i])
        np.testing.assert_array_equal(m[i].cpu().numpy().view(np.uint32), wm.view(np.uint32))
        np.testing.assert_array_equal(v[i].cpu().numpy().view(np.uint32), wv.view(np.uint32))


# ------------------------------------------------------------------ bf16 rounding, exhaustively
def test_bf16_store_rounding_exhaustive(psa):
    """With beta1 = 0 the new m is exactly g (0*m + 1*g), so the stored bf16 m is the
    kernel's rounding of g. Sweep g over all 2^32 fp32 bit patterns (NaNs only need to
    stay NaN: GPU arithmetic returns a canonical NaN) against the oracle's rounding."""
    from concurrent.futures import ThreadPoolExecutor

    chunk = 1 << 28
    base = np.arange(chunk, dtype=np.uint32)
    p = torch.zeros(chunk, device=DEV)
    m = torch.zeros(chunk, dtype=torch.bfloat16, device=DEV)
    v = torch.zeros(chunk, dtype=torch.bfloat16, device=DEV)
    dbase = torch.arange(chunk, dtype=torch.int64, device=DEV)
    pool = ThreadPoolExecutor(max_workers=8)
    for start in range(0, 1 << 32, chunk):
        g = dbase + start
        g = torch.where(g >= 2 ** 31, g - 2 ** 32, g).to(torch.int32).view(torch.float32)
        m.zero_()  # 0 * (previous chunk's inf/NaN) would not be 0
        v.zero_()
        psa.adam_step_bf16m([p], [g], [m], [v], 1, lr=1e-3, beta1=0.0, beta2=0.0, eps=1e-8)
        got = bf16_bits(m)
        # m' = 0*0 + 1*g: g itself, except that -0 becomes +0
        with np.errstate(invalid="ignore"):
            x = (base + np.uint32(start)).view(np.float32) + np.float32(0.0)
        parts = np.array_split(np.arange(chunk), 8)
        want = np.concatenate(list(pool.map(lambda ix: oracle.bf16_round(x[ix[0]:ix[-1] + 1]), parts)))
        nan = np.isnan(x)
        np.testing.assert_array_equal(got[~nan], want[~nan], err_msg=f"chunk at {start:#x}")
        assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all((got[nan] & 0x7F) != 0)
    pool.shutdown()


# ------------------------------------------------------------------ resume
def test_resume_equals_uninterrupted(psa):
    """k steps, state copied to the host and back, then N-k steps == N straight steps,
    bit for bit (stochastic rounding is keyed by (seed, step, index) only)."""
    sizes = [5000, 2048 * 3]
    hp = HParams(weight_decay=0.01)
    q8 = Q8Opts(True, 42, 99.9)
    specs = [workloads.TensorSpec(f"t{i}", (n,)) for i, n in enumerate(sizes)]
    p0 = workloads.init_params_np(specs, seed=2)
    runs = []
    for split in (None, 3):
        params = _to_dev(p0)
        state = psa.zeros_state(params, "q8")
        for t in range(1, 7):
            if split is not None and t == split + 1:
                saved = [[s.cpu() for s in part] for part in state]
                saved_p = [p.cpu() for p in params]
                state = [[s.to(DEV) for s in part] for part in saved]
                params = [p.to(DEV) for p in saved_p]
            grads = _to_dev(workloads.grads_np(sizes, t, 1e-3, seed=2))
            psa.adam_step_q8(params, grads, *state, t, **hp_kwargs(hp), **q8_kwargs(q8))
        runs.append(([p.cpu().numpy() for p in params], [[s.cpu().numpy() for s in part] for part in state]))
    for a, b in zip(runs[0][0], runs[1][0]):
        np.testing.assert_array_equal(a, b)
    for pa, pb in zip(runs[0][1], runs[1][1]):
        for a, b in zip(pa, pb):
            np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("mode", ["fp32", "bf16m", "q8", "q8v"])
def test_resume_through_state_file(psa, mode, tmp_path):
    """k steps, state written with save_state and read back with load_state, then N-k
    steps == N straight steps, bit for bit, for every moment mode."""
    sizes = [5000, 0, 2048 * 3 + 5]
    hp = HParams(weight_decay=0.01)
    q8 = Q8Opts(True, 7, 99.9)
    specs = [workloads.TensorSpec(f"t{i}", (n,)) for i, n in enumerate(sizes)]
    p0 = workloads.init_params_np(specs, seed=4)
    step_fn = {"fp32": psa.adam_step_fp32, "bf16m": psa.adam_step_bf16m,
               "q8": psa.adam_step_q8, "q8v": psa.adam_step_q8v}[mode]
    extra = q8_kwargs(q8) if mode in ("q8", "q8v") else {}
    path = str(tmp_path / "state.bin")
    runs = []
    for split in (None, 2):
        params = _to_dev(p0)
        state = psa.zeros_state(params, mode)
        for t in range(1, 6):
            if split is not None and t == split + 1:
                psa.save_state(path, mode, state, t - 1, hparams=hp_kwargs(hp))
                del state
                mode2, state, last, _ = psa.load_state(path, device=DEV)
                assert mode2 == mode and last == t - 1
            grads = _to_dev(workloads.grads_np(sizes, t, 1e-3, seed=4))
            step_fn(params, grads, *state, t, **hp_kwargs(hp), **extra)
        runs.append(([p.cpu().numpy() for p in params],
                     [[(s.view(torch.int16) if s.dtype == torch.bfloat16 else s).cpu().numpy() for s in part]
                      for part in state]))
    for a, b in zip(runs[0][0], runs[1][0]):
        np.testing.assert_array_equal(a, b)
    for pa, pb in zip(runs[0][1], runs[1][1]):
        for a, b in zip(pa, pb):
            np.testing.assert_array_equal(a, b)


def test_runs_on_the_callers_stream(psa):
    n = 300000
    p0 = workloads.init_params_np([workloads.TensorSpec("w", (n,))], seed=6)[0]
    g = workloads.grads_np([n], 1, 1e-2, seed=6)[0]
    outs = []
    for use_side in (False, True):
        params = _to_dev([p0])
        grads = _to_dev([g])
        state = psa.zeros_state(params, "bf16m")
        s = torch.cuda.Stream() if use_side else torch.cuda.current_stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            psa.adam_step_bf16m(params, grads, *state, 1)
        s.synchronize()
        outs.append(params[0].cpu().numpy())
    np.testing.assert_array_equal(outs[0], outs[1])


# ------------------------------------------------------------------ the workloads at full size
def test_flat_1m_bf16m_full(psa):
    w = workloads.WORKLOADS["flat_1m"]
    hp = HParams(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    got_p, want_p, got_s, want_s = run_both(psa, "bf16m", w.sizes, w.steps, hp, grad_std=w.grad_std, seed=1234)
    check_all("bf16m", got_p, want_p, got_s, want_s, "flat_1m")


def test_flat_16m_q8_full(psa):
    w = workloads.WORKLOADS["flat_16m"]
    hp = HParams(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    got_p, want_p, got_s, want_s = run_both(psa, "q8", w.sizes, w.steps, hp, Q8Opts(False, 42, 100.0),
                                            grad_std=w.grad_std, seed=1234)
    check_all("q8", got_p, want_p, got_s, want_s, "flat_16m")


def _sample_blocks(nb: int):
    # block 0, the last, every 257th, and the blocks on either side of element 2^31
    edge = {b for b in ((2 ** 31 - 1) // 2048, 2 ** 31 // 2048) if b < nb}
    return sorted({0, nb - 1, *range(0, nb, 257), *edge})


def sampled_run(psa, w: workloads.Workload, mode: str, steps: int, tensor_stride: int = 1):
    """Full-size GPU run of workload `w` in moment mode `mode`, with the oracle following a
    deterministic sample of blocks (block 0, the last, every 257th) of every
    `tensor_stride`-th tensor. Inputs come from the device generators of the benchmark."""
    dev = torch.device(DEV)
    sizes = w.sizes
    params = workloads.init_params_torch(w.specs, dev)
    state = psa.zeros_state(params, mode)
    hp = HParams(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    q8 = Q8Opts(w.stochastic_rounding, w.seed, w.percentile)
    picks = []  # (tensor index, block index, start, length)
    for i in range(0, len(sizes), tensor_stride):
        nb = oracle.n_blocks(sizes[i])
        for b in _sample_blocks(nb):
            lo = b * 2048
            picks.append((i, b, lo, min(2048, sizes[i] - lo)))
    host = {}
    for (i, b, lo, ln) in picks:
        p = params[i][lo:lo + ln].cpu().numpy().copy()
        if mode == "fp32":
            st = [np.zeros(ln, np.float32), np.zeros(ln, np.float32)]
        elif mode == "bf16m":
            st = [np.zeros(ln, np.uint16), np.zeros(ln, np.uint16)]
        elif mode == "q8v":
            st = [np.zeros(ln, np.float32), np.zeros(ln, np.uint8), np.zeros(1, np.float32)]
        else:
            st = [np.zeros(ln, np.int8), np.zeros(ln, np.uint8), np.zeros(1, np.float32), np.zeros(1, np.float32)]
        host[(i, b)] = (p, st)
    gbuf = [torch.empty(n, dtype=torch.float32 if w.grad_dtype == "f32" else torch.bfloat16, device=dev)
            for n in sizes]
    for t in range(1, steps + 1):
        workloads.grads_torch(sizes, t, w.grad_std, dev, kind=w.grad_kind, dtype=w.grad_dtype, out=gbuf)
        kw = hp_kwargs(hp)
        if mode in ("q8", "q8v"):
            kw.update(q8_kwargs(q8))
        psa.adam_step(mode, params, gbuf, state, t, **kw)
        for (i, b, lo, ln) in picks:
            gs = gbuf[i][lo:lo + ln]
            g = bf16_bits(gs) if w.grad_dtype == "bf16" else gs.cpu().numpy()
            p, st = host[(i, b)]
            if mode == "fp32":
                oracle.step_fp32(p, g, *st, t, hp)
            elif mode == "bf16m":
                oracle.step_bf16m(p, g, *st, t, hp)
            elif mode == "q8v":
                oracle.step_q8v_block(p, g, *st, t, hp, q8, tensor_idx=i, elem0=lo)
            else:
                oracle.step_q8_block(p, g, *st, t, hp, q8, tensor_idx=i, elem0=lo)
    torch.cuda.synchronize()
    exact = 1.0
    for (i, b, lo, ln) in picks:
        p, st = host[(i, b)]
        got_p = params[i][lo:lo + ln].cpu().numpy()
        if mode == "q8":
            got_s = (state[0][i][lo:lo + ln].cpu().numpy(), state[1][i][lo:lo + ln].cpu().numpy(),
                     state[2][i][b:b + 1].cpu().numpy(), state[3][i][b:b + 1].cpu().numpy())
        elif mode == "q8v":
            got_s = (state[0][i][lo:lo + ln].cpu().numpy(), state[1][i][lo:lo + ln].cpu().numpy(),
                     state[2][i][b:b + 1].cpu().numpy())
        elif mode == "bf16m":
            got_s = (bf16_bits(state[0][i][lo:lo + ln]), bf16_bits(state[1][i][lo:lo + ln]))
        else:
            got_s = (state[0][i][lo:lo + ln].cpu().numpy(), state[1][i][lo:lo + ln].cpu().numpy())
        what = f"{w.name}/{mode} tensor {i} block {b}"
        assert_params(got_p, p, what)
        compare_state(mode, got_s, tuple(st), what)
        exact = min(exact, exact_fraction(mode, [got_p, *got_s], [p, *st]))
    del params, state, gbuf
    return exact, len(picks)


@pytest.mark.parametrize("mode", ["q8", "fp32"])
def test_tensor_past_2_31_elements_sampled(psa, mode):
    """One tensor of 2^31 + 2049 elements: element offsets beyond the 32-bit range, blocks
    on both sides of element 2^31 checked against the oracle (8-bit with stochastic
    rounding and percentile 99.9, and fp32 moments)."""
    n = 2 ** 31 + 2049
    w = workloads.Workload("flat_2g_edge", (workloads.TensorSpec("w", (n,)),), "q8", grad_std=1e-3,
                           weight_decay=0.01, steps=2, stochastic_rounding=True, percentile=99.9)
    ex, picks = sampled_run(psa, w, mode, 2)
    assert picks > 4000 and ex == 1.0


def test_vit_base_list_sampled(psa):
    w = workloads.WORKLOADS["vit_base"]
    for mode in ("bf16m", "fp32", "q8", "q8v"):
        exact, n = sampled_run(psa, w, mode, steps=w.steps if mode == "bf16m" else 10, tensor_stride=2)
        assert exact == 1.0 and n > 90


def test_flat_1g_heavy_tail_sr_sampled(psa):
    w = workloads.WORKLOADS["flat_1g_heavy"]
    exact, n = sampled_run(psa, w, "q8", steps=w.steps)
    assert exact == 1.0 and n > 2000


@pytest.mark.parametrize("mode", ["fp32", "bf16m", "q8", "q8v"])
def test_gpt_1p3b_bf16_grads_sampled(psa, mode):
    w = workloads.WORKLOADS["gpt_1p3b"]
    exact, n = sampled_run(psa, w, mode, steps=w.steps, tensor_stride=5)
    assert exact == 1.0 and n > 200


def test_step_plan_matches_direct_calls(psa):
    """The cached StepPlan issues the same C call as the one-shot binding: identical results."""
    sizes = [3000, 1, 2048 * 2 + 5]
    specs = [workloads.TensorSpec(f"t{i}", (n,)) for i, n in enumerate(sizes)]
    p0 = workloads.init_params_np(specs, seed=17)
    q8 = Q8Opts(True, 3, 99.9)
    for mode in ("fp32", "bf16m", "q8", "q8v"):
        runs = []
        for use_plan in (False, True):
            params = _to_dev(p0)
            state = psa.zeros_state(params, mode)
            gbufs = [_to_dev(workloads.grads_np(sizes, t, 1e-2, seed=17)) for t in (1, 2, 3)]
            kw = dict(weight_decay=0.01)
            if mode in ("q8", "q8v"):
                kw.update(q8_kwargs(q8))
            if use_plan:
                plan = psa.StepPlan(mode, params, gbufs[0], state, **kw)
                for t in (1, 2, 3):
                    plan.set_grads(gbufs[t - 1])
                    plan.step(t)
            else:
                for t in (1, 2, 3):
                    psa.adam_step(mode, params, gbufs[t - 1], state, t, **kw)
            torch.cuda.synchronize()
            runs.append([p.cpu().numpy() for p in params])
        for a, b in zip(*runs):
            np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("mode", ["fp32", "bf16m", "q8", "q8v", "q8/bs256"])
def test_steps_replay_from_a_cuda_graph(psa, mode):
    """The step calls enqueue kernels only (no host sync, no allocation, no host read of
    device data), so a stream capture records them: three steps captured into one CUDA graph
    and replayed equal three direct calls, including the grad check and skip flag."""
    base, _, bs = mode.partition("/bs")
    bs = int(bs) if bs else 2048
    sizes = [3000, 1, 2048 * 2 + 5]
    specs = [workloads.TensorSpec(f"t{i}", (n,)) for i, n in enumerate(sizes)]
    p0 = workloads.init_params_np(specs, seed=23)
    kw = dict(weight_decay=0.01)
    if base in ("q8", "q8v"):
        kw.update(stochastic_rounding=True, seed=5, percentile=99.9, block_size=bs)
    runs = []
    for use_graph in (False, True):
        params = _to_dev(p0)
        state = psa.zeros_state(params, base, bs)
        gbufs = [_to_dev(workloads.grads_np(sizes, t, 1e-2, seed=23)) for t in (1, 2, 3)]
        flag = torch.zeros(1, dtype=torch.int32, device=DEV)
        plans = [psa.StepPlan(base, params, gbufs[t - 1], state, skip_flag=flag, **kw) for t in (1, 2, 3)]

        def three_steps():
            for t in (1, 2, 3):
                psa.check_grads(gbufs[t - 1], flag)
                plans[t - 1].step(t)

        if use_graph:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    three_steps()
            torch.cuda.current_stream().wait_stream(side)
            g.replay()
        else:
            three_steps()
        torch.cuda.synchronize()
        runs.append([p.cpu().numpy() for p in params] + [s.cpu().numpy() if s.dtype != torch.bfloat16 else
                                                          s.view(torch.int16).cpu().numpy()
                                                          for part in state for s in part])
    for a, b in zip(*runs):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("flat", [False, True])
@pytest.mark.parametrize("piped", [False, True])
@pytest.mark.parametrize("mode", ["fp32", "bf16m", "q8", "q8v", "q8/bs256", "q8/p99"])
def test_step_from_host_equals_device_step(psa, mode, piped, flat):
    """psadam_step_from_host (grads uploaded from pinned host buffers, params downloaded), in
    chunks pipelined over three streams or in one piece: the same bits as device-resident steps,
    with stochastic rounding (slices keep their tensors' element offsets and list positions).
    With `flat`, params, grads and the host buffers are views of flat buffers, so the library
    merges the copies of back-to-back tensors."""
    base, _, rest = mode.partition("/")
    kw = dict(weight_decay=0.01)
    if base in ("q8", "q8v"):
        kw.update(stochastic_rounding=True, seed=9, percentile=99.9)
        if rest.startswith("bs"):
            kw["block_size"] = int(rest[2:])
        elif rest.startswith("p"):
            kw["percentile"] = float(rest[1:])
    bs = kw.get("block_size", 2048)
    sizes = [3000, 1, 2048 * 40 + 7, 70001, 0]
    specs = [workloads.TensorSpec(f"t{i}", (n,)) for i, n in enumerate(sizes)]
    p0 = workloads.init_params_np(specs, seed=29)
    gdt = torch.bfloat16 if base == "bf16m" else torch.float32
    host_grads = []
    for t in (1, 2, 3):
        g = [torch.from_numpy(x) for x in workloads.grads_np(sizes, t, 1e-2, seed=29)]
        if flat:
            _, hv = workloads.flat_views(sizes, gdt, pin=True)
            for v, x in zip(hv, g):
                v.copy_(x.to(gdt))
            host_grads.append(hv)
        else:
            host_grads.append([x.to(gdt).pin_memory() for x in g])
    runs = []
    for from_host in (False, True):
        if flat:
            _, params = workloads.flat_views(sizes, torch.float32, DEV)
            for v, a in zip(params, p0):
                v.copy_(torch.from_numpy(a))
            _, dev_g = workloads.flat_views(sizes, gdt, DEV)
            _, out = workloads.flat_views(sizes, torch.float32, pin=True)
        else:
            params = _to_dev(p0)
            dev_g = [torch.empty(n, dtype=gdt, device=DEV) for n in sizes]
            out = [torch.empty(n, dtype=torch.float32).pin_memory() for n in sizes]
        state = psa.zeros_state(params, base, bs)
        plan = psa.StepPlan(base, params, dev_g, state, **kw)
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        for t in (1, 2, 3):
            if from_host:
                plan.step_from_host(t, host_grads[t - 1], out, n_chunks=5,
                                    stream_in=s_in if piped else None, stream_out=s_out if piped else None)
            else:
                for d, h in zip(dev_g, host_grads[t - 1]):
                    d.copy_(h)
                plan.step(t)
        torch.cuda.synchronize()
        got = [p.cpu().numpy() for p in params]
        if from_host:
            for a, b in zip(got, out):
                np.testing.assert_array_equal(a, b.numpy())
        runs.append(got + [(s.view(torch.int16) if s.dtype == torch.bfloat16 else s).cpu().numpy()
                           for part in state for s in part])
    for a, b in zip(*runs):
        np.testing.assert_array_equal(a, b)
