"""GPU: nothing is written outside the buffers a call was given.

Every param, grad, moment, code, scale and flag buffer of a call is carved out of one large
allocation, each start 16-byte aligned, with at least 64 guard bytes before and after it; the
whole allocation is first filled with a guard pattern. After the call every byte outside the
carved buffers must still hold the pattern. The host side of psadam_step_from_host is carved
the same way from one pinned host allocation. This stands in for a memory checker: tails of
tensors (partial stores, zero-filled copies past a tensor's end, bulk copies limited to full
blocks) and slices of the host pipeline all write close to buffer ends.

Sizes 1, 7, 2047, 2049 and 4097 go in one list per call, at block sizes 3, 16, 100, 256, 2048,
4096 and 16384 (16 and 256 take the persistent kernel's sub-block path; 16384 with absmax
scales the general kernel's read-twice path), for every moment mode with
its options (stochastic rounding with percentile scales, grad zeroing, static scales, bf16
grads, the approximate update), and for quantize-only,
dequantize-only, the grad check and the host pipeline. Each step is also checked against the
CPU oracle, so a kernel that wrote nothing could not pass. Input validation follows PR #814's
review thread (block size > 0, percentile within 0..100); the guard idea itself is this
library's stand-in for a sanitizer.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import HParams, Q8Opts
import workloads
from parity_util import hp_kwargs, host_state

pytestmark = pytest.mark.gpu

SIZES = [1, 7, 2047, 2049, 4097]
# 16 and 256: sub-blocks of the persistent kernel; 16384 with absmax scales: read twice, not staged
BLOCKS = [3, 16, 100, 256, 2048, 4096, 16384]
GUARD = 64
PATTERN = 0xA5
DEV = "cuda:0"
HP = HParams(lr=1e-3, weight_decay=0.01)


@pytest.fixture(scope="module")
def psa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import precision_state_adam_gb300 as psa
    return psa


class Arena:
    """Buffers carved from one byte allocation (device or pinned host) with guard bytes."""

    def __init__(self, specs, device):
        self.offsets = []
        cur = 0
        for dtype, n in specs:
            nbytes = n * torch.empty((), dtype=dtype).element_size()
            off = (cur + GUARD + 15) // 16 * 16
            self.offsets.append((off, nbytes))
            cur = off + nbytes
        total = (cur + GUARD + 15) // 16 * 16
        if device == "host":
            self.raw = torch.full((total,), PATTERN, dtype=torch.uint8).pin_memory()
        else:
            self.raw = torch.full((total,), PATTERN, dtype=torch.uint8, device=device)
        self.views = [self.raw[o:o + nb].view(dtype) for (o, nb), (dtype, _) in zip(self.offsets, specs)]

    def check_guards(self, what: str) -> None:
        torch.cuda.synchronize()
        raw = self.raw.cpu().numpy()
        inside = np.zeros(raw.size, bool)
        for o, nb in self.offsets:
            inside[o:o + nb] = True
        bad = np.nonzero((raw != PATTERN) & ~inside)[0]
        if bad.size:
            owners = [i for i, (o, nb) in enumerate(self.offsets) if o - GUARD <= bad[0] < o + nb + GUARD]
            raise AssertionError(f"{what}: {bad.size} guard bytes overwritten, first at byte {bad[0]} "
                                 f"(near buffer {owners})")


def _dtype_of(a: np.ndarray):
    return {np.float32: torch.float32, np.int8: torch.int8, np.uint8: torch.uint8,
            np.uint16: torch.bfloat16}[a.dtype.type]


def _load(view: torch.Tensor, a: np.ndarray) -> None:
    src = torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16) if a.dtype == np.uint16 \
        else torch.from_numpy(a.copy())
    view.copy_(src)


def _host(view: torch.Tensor) -> np.ndarray:
    if view.dtype == torch.bfloat16:
        return view.view(torch.int16).cpu().numpy().view(np.uint16)
    return view.cpu().numpy()


STEP_CASES = [
    # (mode, block sizes, options)
    ("fp32", [2048], dict()),
    ("fp32", [2048], dict(zero_grads=True)),
    ("fp32", [2048], dict(grad_dtype="bf16")),
    ("bf16m", [2048], dict()),
    ("bf16m", [2048], dict(zero_grads=True, grad_dtype="bf16")),
    ("q8", BLOCKS, dict()),
    ("q8", BLOCKS, dict(stochastic_rounding=True, percentile=99.9)),
    ("q8", BLOCKS, dict(zero_grads=True, static_scales=True, grad_dtype="bf16")),
    ("q8", [2048], dict(approx_update=True, percentile=99.0)),
    ("q8v", BLOCKS, dict()),
    ("q8v", BLOCKS, dict(stochastic_rounding=True, percentile=99.9, zero_grads=True)),
]


def _case_id(c):
    mode, _, opts = c
    return mode + "".join(f"-{k}" for k in sorted(opts))


@pytest.mark.parametrize("case", STEP_CASES, ids=_case_id)
def test_steps_write_only_their_buffers(psa, case):
    mode, blocks, opts = case
    opts = dict(opts)
    grad_dtype = opts.pop("grad_dtype", "f32")
    zero = opts.pop("zero_grads", False)
    approx = opts.pop("approx_update", False)
    for bs in blocks:
        q8 = Q8Opts(stochastic_rounding=opts.get("stochastic_rounding", False), seed=77,
                    percentile=opts.get("percentile", 100.0), static_scales=opts.get("static_scales", False),
                    block_size=bs)
        specs = [workloads.TensorSpec(f"t{i}", (n,)) for i, n in enumerate(SIZES)]
        p_host = workloads.init_params_np(specs, seed=61)
        ostate = host_state(mode, SIZES, bs)
        gdt = torch.bfloat16 if grad_dtype == "bf16" else torch.float32
        k = len(SIZES)
        layout = [(torch.float32, n) for n in SIZES] + [(gdt, n) for n in SIZES]
        for arrs in zip(*ostate):
            layout += [(_dtype_of(a), a.size) for a in arrs]
        arena = Arena(layout, DEV)
        params = arena.views[:k]
        grads = arena.views[k:2 * k]
        flat_state = arena.views[2 * k:]
        n_state = len(ostate[0])
        state = [flat_state[j * k:(j + 1) * k] for j in range(n_state)]
        for v, a in zip(params, p_host):
            _load(v, a)
        for j in range(n_state):
            for i in range(k):
                _load(state[j][i], ostate[i][j])
        kw = hp_kwargs(HP)
        if mode in ("q8", "q8v"):
            kw.update(stochastic_rounding=q8.stochastic_rounding, seed=q8.seed, percentile=q8.percentile,
                      block_size=bs, static_scales=q8.static_scales)
        for t in (1, 2):
            g32 = workloads.grads_np(SIZES, t, 1e-2, seed=62)
            g_host = [workloads.to_bf16_bits_truncate(g) for g in g32] if grad_dtype == "bf16" else g32
            for v, a in zip(grads, g_host):
                _load(v, a)
            psa.adam_step(mode, params, grads, state, t, zero_grads=zero, approx_update=approx, **kw)
            oracle.step_list(mode, p_host, g_host, ostate, t, HP, q8)
            what = f"{mode} bs={bs} {opts} zero={zero} grads={grad_dtype} step {t}"
            arena.check_guards(what)
            if zero:
                assert all(float(g.float().abs().max()) == 0.0 for g in grads), what + ": grads not zeroed"
        for i in range(k):
            got = params[i].cpu().numpy()
            assert not np.array_equal(got, workloads.init_params_np(specs, seed=61)[i]), "the step wrote nothing"
            if approx:
                scale = max(float(np.abs(p_host[i]).max()), 1e-30)
                assert float(np.abs(got.astype(np.float64) - p_host[i]).max()) / scale <= 1e-6
            else:
                np.testing.assert_array_equal(got, p_host[i], err_msg=f"{mode} bs={bs} params tensor {i}")
            for j in range(n_state):
                np.testing.assert_array_equal(_host(state[j][i]), ostate[i][j],
                                              err_msg=f"{mode} bs={bs} state {j} tensor {i}")


@pytest.mark.parametrize("bs", BLOCKS)
@pytest.mark.parametrize("sr", [False, True])
def test_quantize_and_dequantize_write_only_their_buffers(psa, bs, sr):
    q8 = Q8Opts(stochastic_rounding=sr, seed=5, percentile=99.9 if sr else 100.0, block_size=bs)
    k = len(SIZES)
    mv = [workloads.random_moments_np(n, seed=70 + i) for i, n in enumerate(SIZES)]
    nb = [oracle.n_blocks(n, bs) for n in SIZES]
    layout = ([(torch.float32, n) for n in SIZES] * 2 + [(torch.int8, n) for n in SIZES] +
              [(torch.uint8, n) for n in SIZES] + [(torch.float32, b) for b in nb] * 2 +
              [(torch.float32, n) for n in SIZES] * 2)
    arena = Arena(layout, DEV)
    v = arena.views
    m_in, v_in = v[:k], v[k:2 * k]
    mc, vc, ms, vs = v[2 * k:3 * k], v[3 * k:4 * k], v[4 * k:5 * k], v[5 * k:6 * k]
    m_out, v_out = v[6 * k:7 * k], v[7 * k:8 * k]
    for i in range(k):
        _load(m_in[i], mv[i][0])
        _load(v_in[i], mv[i][1])
    psa.q8_quantize(m_in, v_in, mc, vc, ms, vs, step=3, stochastic_rounding=sr, seed=5,
                    percentile=q8.percentile, block_size=bs)
    arena.check_guards(f"quantize bs={bs} sr={sr}")
    psa.q8_dequantize(mc, vc, ms, vs, m_out, v_out, block_size=bs)
    arena.check_guards(f"dequantize bs={bs} sr={sr}")
    for i in range(k):
        want = oracle.quantize(mv[i][0], mv[i][1], q8, step=3, tensor_idx=i)
        for got, w in zip((mc[i], vc[i], ms[i], vs[i]), want):
            np.testing.assert_array_equal(_host(got), w)
        wm, wv = oracle.dequantize(*want, block_size=bs)
        np.testing.assert_array_equal(_host(m_out[i]), wm)
        np.testing.assert_array_equal(_host(v_out[i]), wv)


def test_grad_check_writes_only_its_flag(psa):
    k = len(SIZES)
    arena = Arena([(torch.float32, n) for n in SIZES] + [(torch.int32, 1)], DEV)
    grads, flag = arena.views[:k], arena.views[k]
    for g, a in zip(grads, workloads.grads_np(SIZES, 1, 1e-2, seed=63)):
        _load(g, a)
    grads[3][2048] = float("inf")
    psa.check_grads(grads, flag)
    arena.check_guards("check_grads")
    assert int(flag.item()) == 1


@pytest.mark.parametrize("piped", [False, True])
@pytest.mark.parametrize("mode,bs", [("fp32", 2048), ("bf16m", 2048), ("q8", 2048), ("q8", 100), ("q8v", 4096),
                                     ("q8", 3)])
def test_step_from_host_writes_only_its_buffers(psa, mode, bs, piped):
    """The host pipeline: device grads and params, host grads and params, all carved with
    guards; 3 chunks cut the list inside its tensors."""
    k = len(SIZES)
    gdt = torch.bfloat16 if mode == "bf16m" else torch.float32
    specs = [workloads.TensorSpec(f"t{i}", (n,)) for i, n in enumerate(SIZES)]
    p0 = workloads.init_params_np(specs, seed=64)
    ostate = host_state(mode, SIZES, bs)
    layout = [(torch.float32, n) for n in SIZES] + [(gdt, n) for n in SIZES]
    for arrs in zip(*ostate):
        layout += [(_dtype_of(a), a.size) for a in arrs]
    dev = Arena(layout, DEV)
    host = Arena([(gdt, n) for n in SIZES] + [(torch.float32, n) for n in SIZES], "host")
    params, dev_g = dev.views[:k], dev.views[k:2 * k]
    n_state = len(ostate[0])
    state = [dev.views[2 * k + j * k:2 * k + (j + 1) * k] for j in range(n_state)]
    for v, a in zip(params, p0):
        _load(v, a)
    for j in range(n_state):
        for i in range(k):
            _load(state[j][i], ostate[i][j])
    host_g, host_p = host.views[:k], host.views[k:]
    kw = dict(weight_decay=0.01)
    if mode in ("q8", "q8v"):
        kw.update(stochastic_rounding=True, seed=9, percentile=99.9, block_size=bs)
    plan = psa.StepPlan(mode, params, dev_g, state, **kw)
    s_in, s_out = (torch.cuda.Stream(), torch.cuda.Stream()) if piped else (None, None)
    for t in (1, 2):
        for hg, a in zip(host_g, workloads.grads_np(SIZES, t, 1e-2, seed=65)):
            hg.copy_(torch.from_numpy(a).to(gdt))
        plan.step_from_host(t, host_g, host_p, n_chunks=3, stream_in=s_in, stream_out=s_out)
        torch.cuda.synchronize()
        dev.check_guards(f"from_host {mode} bs={bs} piped={piped} step {t} (device)")
        host.check_guards(f"from_host {mode} bs={bs} piped={piped} step {t} (host)")
    for i in range(k):
        np.testing.assert_array_equal(host_p[i].numpy(), params[i].cpu().numpy())
