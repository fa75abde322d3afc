"""Host-side checks of libpsadam.so without a GPU: the library loads, exports every
function include/psadam.h declares, rejects bad arguments before launching anything,
and reports the state-memory closed form (AiDotNet PR #814: 8-bit state is about 2 bytes
per parameter plus per-block scales, ~4x less than fp32 Adam's two moments)."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "psadam.h")


@pytest.fixture(scope="module")
def psa():
    import __graft_entry__
    __graft_entry__.build()
    import precision_state_adam_gb300 as psa
    return psa


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted({n for n in names if n not in ("if", "while", "return")})


def test_header_declares_the_step_entry_points():
    names = declared_functions()
    for want in ("adam_step_fp32", "adam_step_bf16m", "adam_step_q8", "adam_step_q8v", "psadam_q8_quantize",
                 "psadam_q8_dequantize", "psadam_state_bytes", "psadam_status_string", "psadam_check_grads",
                 "psadam_step_from_host"):
        assert want in names


def test_library_exports_every_declared_symbol(psa):
    lib = ctypes.CDLL(psa.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_library_does_not_link_the_oracle(psa):
    data = open(psa.LIB_PATH, "rb").read()
    assert b"orc_step" not in data and b"liboracle" not in data


def test_state_bytes_closed_form(psa):
    lib = psa.cdll()
    for bs in (2048, 1, 64, 1000, 16384):
        for n in (0, 1, 2047, 2048, 2049, 1 << 24, 86_564_352):
            nb = -(-n // bs)
            assert lib.psadam_state_bytes(0, n, bs) == 8 * n
            assert lib.psadam_state_bytes(1, n, bs) == 4 * n
            assert lib.psadam_state_bytes(2, n, bs) == 2 * n + 8 * nb
            assert lib.psadam_state_bytes(3, n, bs) == 5 * n + 4 * nb
    assert lib.psadam_state_bytes(4, 10, 2048) == 0 and lib.psadam_state_bytes(0, -1, 2048) == 0
    assert lib.psadam_state_bytes(2, 10, 0) == 0 and lib.psadam_state_bytes(3, 10, -1) == 0
    assert lib.psadam_state_bytes(0, 10, 0) == 80  # block size only matters to 8-bit modes
    n = 1 << 24
    assert 3.99 < lib.psadam_state_bytes(0, n, 2048) / lib.psadam_state_bytes(2, n, 2048) < 4.0
    assert psa.state_bytes("q8", 4096, 64) == 2 * 4096 + 8 * 64


def test_status_strings(psa):
    assert psa.status_string(0) == "PSADAM_OK"
    assert psa.status_string(3) == "PSADAM_ERR_UNSUPPORTED"
    assert psa.status_string(99) == "PSADAM_ERR_UNKNOWN"


# ---------------------------------------------------------------- validation (never launches)
FAKE = 1 << 20  # aligned, never dereferenced: every call below fails validation first


def _arr(ctype, vals):
    a = (ctype * max(len(vals), 1))()
    for i, x in enumerate(vals):
        a[i] = x
    return a


def _call_q8(psa, numel=(4096,), ptr=FAKE, step=1, hp=None, block=2048, pct=100.0, sr=0, grad_dtype=0,
             n_tensors=None):
    n = len(numel) if n_tensors is None else n_tensors
    nums = _arr(ctypes.c_int64, list(numel))
    ptrs = _arr(ctypes.c_void_p, [ptr] * len(numel))
    lst = psa._List(n, grad_dtype, nums, ctypes.cast(ptrs, psa._PP), ctypes.cast(ptrs, psa._PP))
    hp = hp or psa._HParams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    q = psa._Q8Opts(block, sr, 42, pct)
    P = ctypes.cast(ptrs, psa._PP)
    return psa.cdll().adam_step_q8(ctypes.byref(lst), P, P, P, P, step, ctypes.byref(hp), ctypes.byref(q), None)


def test_validation_errors(psa):
    E = psa
    assert _call_q8(psa, n_tensors=0) == E.OK                       # empty list: no-op
    assert _call_q8(psa, numel=(0, 0)) == E.OK                      # only empty tensors: no-op
    assert _call_q8(psa, step=0) == E.ERR_INVALID_ARG
    assert _call_q8(psa, numel=(-1,)) == E.ERR_INVALID_ARG
    assert _call_q8(psa, ptr=FAKE + 4) == E.ERR_MISALIGNED
    assert _call_q8(psa, ptr=0) == E.ERR_INVALID_ARG
    assert _call_q8(psa, block=0) == E.ERR_INVALID_ARG
    assert _call_q8(psa, block=-64) == E.ERR_INVALID_ARG
    assert _call_q8(psa, block=16385) == E.ERR_UNSUPPORTED          # beyond the staged block
    assert _call_q8(psa, pct=0.0) == E.ERR_INVALID_ARG
    assert _call_q8(psa, pct=100.5) == E.ERR_INVALID_ARG
    assert _call_q8(psa, pct=float("nan")) == E.ERR_INVALID_ARG
    assert _call_q8(psa, sr=2) == E.ERR_INVALID_ARG
    assert _call_q8(psa, grad_dtype=5) == E.ERR_INVALID_ARG
    for bad in ((1e-3, 1.0, 0.999, 1e-8, 0.0), (1e-3, 0.9, -0.1, 1e-8, 0.0), (float("inf"), 0.9, 0.999, 1e-8, 0.0),
                (1e-3, 0.9, 0.999, -1.0, 0.0)):
        assert _call_q8(psa, hp=psa._HParams(*bad)) == E.ERR_INVALID_ARG
    assert psa.cdll().adam_step_q8(None, None, None, None, None, 1, None, None, None) == E.ERR_INVALID_ARG
    # numel beyond what one grid can cover, at the default and at a small block size
    assert _call_q8(psa, numel=((2 ** 31) * 2048,)) == E.ERR_UNSUPPORTED
    assert _call_q8(psa, numel=(2 ** 31,), block=1) == E.ERR_UNSUPPORTED


def test_grad_side_validation(psa):
    import ctypes as C
    nums = _arr(C.c_int64, [4096])
    ptrs = _arr(C.c_void_p, [FAKE])
    P = C.cast(ptrs, psa._PP)
    hp = psa._HParams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    q = psa._Q8Opts(2048, 0, 42, 100.0)
    lib = psa.cdll()
    for unscale, skip, want in ((float("inf"), None, psa.ERR_INVALID_ARG), (float("nan"), None, psa.ERR_INVALID_ARG),
                                (1.0, FAKE + 2, psa.ERR_MISALIGNED)):
        lst = psa._List(1, 0, nums, P, P, unscale, 0, skip)
        assert lib.adam_step_q8(C.byref(lst), P, P, P, P, 1, C.byref(hp), C.byref(q), None) == want
    lst = psa._List(1, 0, nums, P, P, 1.0, 0, None)
    assert lib.psadam_check_grads(C.byref(lst), None, None) == psa.ERR_INVALID_ARG
    assert lib.psadam_check_grads(C.byref(lst), FAKE + 1, None) == psa.ERR_MISALIGNED
    assert lib.psadam_check_grads(None, FAKE, None) == psa.ERR_INVALID_ARG


def test_dequantize_block_size_validation(psa):
    nums = _arr(ctypes.c_int64, [4096])
    P = ctypes.cast(_arr(ctypes.c_void_p, [FAKE]), psa._PP)
    lib = psa.cdll()
    assert lib.psadam_q8_dequantize(1, nums, P, P, P, P, P, P, 0, None) == psa.ERR_INVALID_ARG
    assert lib.psadam_q8_dequantize(1, nums, P, P, P, P, P, P, 16385, None) == psa.ERR_UNSUPPORTED
    assert lib.psadam_q8_dequantize(0, nums, P, P, P, P, P, P, 0, None) == psa.OK  # empty list: no-op


def test_step_from_host_validation(psa):
    """Every argument error is reported before a copy or a launch is enqueued."""
    C = ctypes
    nums = _arr(C.c_int64, [4096])
    P = C.cast(_arr(C.c_void_p, [FAKE]), psa._PP)
    lst = psa._List(1, 0, nums, P, P, 1.0, 0, None, 0)
    hp = psa._HParams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    q = psa._Q8Opts(2048, 0, 42, 100.0)
    lib = psa.cdll()
    f = lib.psadam_step_from_host
    B = C.byref
    assert f(7, B(lst), P, P, P, P, P, P, 1, B(hp), B(q), 4, None, None, None) == psa.ERR_INVALID_ARG      # mode
    assert f(2, B(lst), P, P, P, P, P, P, 1, B(hp), B(q), 0, None, None, None) == psa.ERR_INVALID_ARG      # chunks
    assert f(2, B(lst), None, P, P, P, P, P, 1, B(hp), B(q), 4, None, None, None) == psa.ERR_INVALID_ARG   # host grads
    assert f(2, B(lst), P, P, P, P, P, P, 0, B(hp), B(q), 4, None, None, None) == psa.ERR_INVALID_ARG      # step
    assert f(2, B(lst), P, P, P, P, P, P, 1, B(hp), None, 4, None, None, None) == psa.ERR_INVALID_ARG      # q8 opts
    bad = C.cast(_arr(C.c_void_p, [FAKE + 8]), psa._PP)
    assert f(2, B(lst), P, P, bad, P, P, P, 1, B(hp), B(q), 4, None, None, None) == psa.ERR_MISALIGNED
    empty = psa._List(0, 0, nums, P, P, 1.0, 0, None, 0)
    assert f(2, B(empty), None, None, None, None, None, None, 1, B(hp), B(q), 4, None, None, None) == psa.OK


def test_selftest_and_fault_validation(psa):
    lib = psa.cdll()
    assert lib.psadam_selftest_bounded_wait(-1, None) == psa.ERR_INVALID_ARG
    # no wait longer than the step kernels' own limit (2^31 SM cycles, about a second)
    assert lib.psadam_selftest_bounded_wait((1 << 31) + 1, None) == psa.ERR_INVALID_ARG
    assert lib.psadam_selftest_bounded_wait(2 ** 62, None) == psa.ERR_INVALID_ARG
    out = (ctypes.c_uint64 * 4)()
    assert lib.psadam_selftest_update_math(0, None, None) == psa.ERR_INVALID_ARG
    assert lib.psadam_selftest_update_math(2, out, None) == psa.ERR_INVALID_ARG
    assert lib.psadam_selftest_update_math(-1, out, None) == psa.ERR_INVALID_ARG


def test_binding_refuses_short_pointer_tables(psa):
    # the library reads one pointer per list tensor from every table: a state list shorter
    # than the param list is refused before any call (checked before the device checks, so
    # CPU tensors show it)
    a, b = torch.zeros(4), torch.zeros(8)
    with pytest.raises(ValueError, match="1 tensors for a list of 2"):
        psa._check_layout("m", [a], torch.float32, like=[a, b])
    with pytest.raises(ValueError, match="tensors for a list of"):
        psa._check_layout("m", [a, b, a], torch.float32, like=[a, b])
    with pytest.raises(TypeError, match="must be a CUDA tensor"):
        psa._check_layout("m", [a, b], torch.float32, like=[a, b])
    with pytest.raises(TypeError, match="expected torch.float32"):
        psa._check_layout("m", [a.double()], torch.float32)
