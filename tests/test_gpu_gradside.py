"""GPU tests of the grad-side work around the update: loss-scale removal, grad zeroing, the
device skip flag, and the non-finite grad check, against the CPU oracle (the update sees
grads multiplied by the inverse loss scale, one fp32 rounding)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import HParams, Q8Opts
import workloads
from parity_util import device_state_to_host, exact_fraction, host_state, hp_kwargs, q8_kwargs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SIZES = [1, 7, 2049, 4097, 30000]
MODES = ["fp32", "bf16m", "q8", "q8v"]


@pytest.fixture(scope="module")
def psa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import precision_state_adam_gb300 as psa
    return psa


def _dev(arrs):
    out = []
    for a in arrs:
        if a.dtype == np.uint16:
            out.append(torch.from_numpy(a.view(np.int16).copy()).to(DEV).view(torch.bfloat16))
        else:
            out.append(torch.from_numpy(a.copy()).to(DEV))
    return out


def _host(x: torch.Tensor) -> np.ndarray:
    return (x.view(torch.int16) if x.dtype == torch.bfloat16 else x).cpu().numpy()


def _grads(step, bf16, scale=1.0, seed=40):
    g = [x * np.float32(scale) for x in workloads.grads_np(SIZES, step, 1e-2, seed=seed)]
    return [workloads.to_bf16_bits_truncate(x) for x in g] if bf16 else [x.astype(np.float32) for x in g]


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("unscale", [2.0 ** -10, 1.0 / 3.0])
@pytest.mark.parametrize("mode", MODES)
def test_grad_unscale_matches_oracle(psa, mode, unscale, bf16):
    hp = HParams(weight_decay=0.01)
    q8 = Q8Opts(True, 11, 99.9)
    specs = [workloads.TensorSpec(f"t{i}", (n,)) for i, n in enumerate(SIZES)]
    p_host = workloads.init_params_np(specs, seed=41)
    params = _dev(p_host)
    state = psa.zeros_state(params, mode)
    ostate = host_state(mode, SIZES)
    u = float(np.float32(unscale))
    for t in (1, 2, 3):
        g_host = _grads(t, bf16, scale=1024.0)
        kw = hp_kwargs(hp)
        if mode in ("q8", "q8v"):
            kw.update(q8_kwargs(q8))
        psa.adam_step(mode, params, _dev(g_host), state, t, grad_unscale=u, **kw)
        oracle.step_list(mode, p_host, [oracle.unscale_grads(g, u) for g in g_host], ostate, t, hp, q8)
    torch.cuda.synchronize()
    for i in range(len(SIZES)):
        got = [params[i].cpu().numpy(), *device_state_to_host(mode, state, i)]
        assert exact_fraction(mode, got, [p_host[i], *ostate[i]]) == 1.0, (mode, i)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("mode", ["q8", "q8v"])
def test_grad_side_on_blocks_larger_than_a_tile(psa, mode, bf16):
    """Blocks of 16384 with absmax scales: the general kernel reads each block twice (the
    moments for the block maxima, then the whole update). The loss-scale removal must enter
    both reads alike and the zeroing must follow the second: params, moments, codes and
    scales match the oracle bit for bit, and the grads end zero."""
    hp = HParams(weight_decay=0.01)
    bs = 16384
    q8 = Q8Opts(False, 42, 100.0, block_size=bs)
    sizes = [1, 16383, 16385, 40000]
    specs = [workloads.TensorSpec(f"t{i}", (n,)) for i, n in enumerate(sizes)]
    p_host = workloads.init_params_np(specs, seed=47)
    params = _dev(p_host)
    state = psa.zeros_state(params, mode, bs)
    ostate = host_state(mode, sizes, bs)
    u = float(np.float32(1.0 / 3.0))
    for t in (1, 2, 3):
        g = [x * np.float32(1024.0) for x in workloads.grads_np(sizes, t, 1e-2, seed=48)]
        g_host = [workloads.to_bf16_bits_truncate(x) for x in g] if bf16 else [x.astype(np.float32) for x in g]
        grads = _dev(g_host)
        kw = hp_kwargs(hp)
        kw.update(q8_kwargs(q8))
        psa.adam_step(mode, params, grads, state, t, grad_unscale=u, zero_grads=True, **kw)
        oracle.step_list(mode, p_host, [oracle.unscale_grads(x, u) for x in g_host], ostate, t, hp, q8)
        torch.cuda.synchronize()
        assert all(int(torch.count_nonzero(x)) == 0 for x in grads)
    for i in range(len(sizes)):
        got = [params[i].cpu().numpy(), *device_state_to_host(mode, state, i)]
        assert exact_fraction(mode, got, [p_host[i], *ostate[i]]) == 1.0, (mode, i)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("mode", MODES)
def test_zero_grads_zeroes_after_use(psa, mode, bf16):
    specs = [workloads.TensorSpec(f"t{i}", (n,)) for i, n in enumerate(SIZES)]
    p0 = workloads.init_params_np(specs, seed=42)
    g_host = _grads(1, bf16)
    runs = []
    for zero in (False, True):
        params = _dev(p0)
        grads = _dev(g_host)
        state = psa.zeros_state(params, mode)
        psa.adam_step(mode, params, grads, state, 1, weight_decay=0.01, zero_grads=zero)
        torch.cuda.synchronize()
        runs.append([p.cpu().numpy() for p in params])
        if zero:
            assert all(int(torch.count_nonzero(g)) == 0 for g in grads)
        else:
            assert all(int(torch.count_nonzero(g)) > 0 for g in grads if g.numel() > 1)
    for a, b in zip(*runs):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("mode", MODES)
def test_skip_flag_makes_the_step_a_no_op(psa, mode):
    specs = [workloads.TensorSpec(f"t{i}", (n,)) for i, n in enumerate(SIZES)]
    p0 = workloads.init_params_np(specs, seed=43)
    params = _dev(p0)
    state = psa.zeros_state(params, mode)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    psa.adam_step(mode, params, _dev(_grads(1, False)), state, 1, skip_flag=flag)  # flag 0: a real step
    torch.cuda.synchronize()
    before = [_host(p) for p in params] + [_host(s) for part in state for s in part]
    flag.fill_(1)
    psa.adam_step(mode, params, _dev(_grads(2, False)), state, 2, skip_flag=flag, zero_grads=True)
    torch.cuda.synchronize()
    after = [_host(p) for p in params] + [_host(s) for part in state for s in part]
    for a, b in zip(before, after):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("bf16", [False, True])
def test_check_grads_finds_planted_non_finite_values(psa, bf16):
    rng = np.random.default_rng(44)
    flag = torch.full((1,), 7, dtype=torch.int32, device=DEV)
    clean = _grads(1, bf16)
    psa.check_grads(_dev(clean), flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    for bad in (np.inf, -np.inf, np.nan):
        for trial in range(4):
            g = [x.copy() for x in clean]
            i = int(rng.integers(len(g)))
            j = int(rng.integers(g[i].size))
            if bf16:
                g[i][j] = workloads.to_bf16_bits_truncate(np.array([bad], np.float32))[0]
            else:
                g[i][j] = bad
            psa.check_grads(_dev(g), flag)
            torch.cuda.synchronize()
            assert int(flag.item()) == 1, (bad, i, j)
    # finite grads whose unscaled value overflows are caught too
    big = [np.full(n, 3e38, np.float32) for n in SIZES]
    psa.check_grads(_dev(big), flag, grad_unscale=10.0)
    torch.cuda.synchronize()
    assert int(flag.item()) == 1
    want = any(not np.isfinite(oracle.unscale_grads(x, 10.0)).all() for x in big)
    assert want


def test_mixed_precision_flow_skips_only_the_bad_step(psa):
    """check_grads -> step(skip_flag): a step whose grads hold an inf changes nothing; the
    steps around it match the oracle run that never saw it."""
    mode = "q8"
    hp = HParams(weight_decay=0.01)
    specs = [workloads.TensorSpec(f"t{i}", (n,)) for i, n in enumerate(SIZES)]
    p_host = workloads.init_params_np(specs, seed=45)
    params = _dev(p_host)
    state = psa.zeros_state(params, mode)
    ostate = host_state(mode, SIZES)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    u = 2.0 ** -8
    t_opt = 0
    for it in range(1, 5):
        g_host = _grads(it, False, scale=256.0)
        if it == 2:
            g_host[1][3] = np.inf
        grads = _dev(g_host)
        psa.check_grads(grads, flag, grad_unscale=u)
        psa.adam_step(mode, params, grads, state, t_opt + 1, grad_unscale=u, skip_flag=flag, weight_decay=0.01)
        torch.cuda.synchronize()
        if int(flag.item()) == 0:
            t_opt += 1
            oracle.step_list(mode, p_host, [oracle.unscale_grads(g, u) for g in g_host], ostate, t_opt, hp, Q8Opts())
        else:
            assert it == 2
    assert t_opt == 3
    for i in range(len(SIZES)):
        got = [params[i].cpu().numpy(), *device_state_to_host(mode, state, i)]
        assert exact_fraction(mode, got, [p_host[i], *ostate[i]]) == 1.0


def test_bounded_wait_reports_through_the_fault_word(psa):
    """A kernel wait that nothing completes gives up after its cycle limit and sets the
    library's fault word; psadam_device_fault reads it once and clears it. Steps leave it 0."""
    assert psa.device_fault() == 0
    lib = psa.cdll()
    assert lib.psadam_selftest_bounded_wait(1 << 20, None) == psa.OK
    torch.cuda.synchronize()
    assert psa.device_fault() == 1
    assert psa.device_fault() == 0
    # a real step afterwards runs normally and reports nothing
    params = [torch.randn(5000, device=DEV) * 0.02]
    state = psa.zeros_state(params, "q8")
    psa.adam_step_q8(params, [torch.randn(5000, device=DEV) * 1e-3], *state, 1)
    torch.cuda.synchronize()
    assert psa.device_fault() == 0
