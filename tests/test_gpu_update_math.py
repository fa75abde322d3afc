"""The IEEE-exact step takes its square root and quotient from the hardware's reciprocal
approximations plus one fused multiply-add correction each, wherever a thread's moments lie
in the domain where that gives IEEE's bits. The library's own device-side check compares
them with IEEE sqrt and division: the root over every float of its range, the quotient over
2^36 significand pairs (every pair with full=True, about a minute, not run here), the
exponent scaling that carries those to the whole domain, and the step's arithmetic on
random elements against the per-element IEEE update, the domain switch going both ways."""
from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def psa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import precision_state_adam_gb300 as psa
    return psa


def test_fused_root_and_quotient_match_ieee(psa):
    got = psa.selftest_update_math()
    assert got == {"root": 0, "quotient": 0, "scaling": 0, "update": 0}


def _moment_hitting(target: float, beta: float, steps: int) -> list[float]:
    """fp32 moments x whose decayed value RN(beta*x) (the step's m' or v' with a zero grad)
    is `target` or one of its neighbours up to `steps` ulp away on either side (those that
    some x reaches)."""
    import numpy as np

    b = np.float32(beta)
    want = [np.float32(target)]
    lo = hi = np.float32(target)
    for _ in range(steps):
        lo, hi = np.nextafter(lo, np.float32(0)), np.nextafter(hi, np.float32(np.inf))
        want += [lo, hi]
    out = []
    for w in want:
        x = np.float32(w / b)
        for _ in range(8):  # walk x until RN(b*x) is w
            y = np.float32(b * x)
            if y == w:
                break
            x = np.nextafter(x, np.float32(np.inf) if y < w else np.float32(0))
        if np.float32(b * x) == w:
            out.append(float(x))
    return out


def test_step_at_the_edges_of_the_fused_domain(psa):
    """Moments whose m' and v' land on, just inside and just outside the fused domain's
    bounds (2^-60 and 2^64), and zeros: one fp32-moment step against the oracle, bit for bit
    (params and moments). With zero grads m' = RN(beta1*m) and v' = RN(beta2*v)."""
    import numpy as np
    import oracle
    from oracle import HParams
    from parity_util import hp_kwargs

    hp = HParams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    m_edges = _moment_hitting(2.0 ** -60, 0.9, 3) + _moment_hitting(2.0 ** 64, 0.9, 3) + [0.0]
    v_edges = _moment_hitting(2.0 ** -60, 0.999, 3) + _moment_hitting(2.0 ** 64, 0.999, 3) + [0.0]
    assert len(m_edges) >= 10 and len(v_edges) >= 10
    rng = np.random.default_rng(11)
    n = 16384
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = np.zeros(n, np.float32)
    m = (rng.uniform(1e-4, 1e-2, n) * rng.choice([-1.0, 1.0], n)).astype(np.float32)
    v = rng.uniform(1e-8, 1e-6, n).astype(np.float32)
    # one element of each thread's 8 in every other 2048-block takes an edge value: its tile
    # then switches on that one value; the rest stay inside the domain
    idx = np.arange(n)
    hit = ((idx // 2048) % 2 == 1) & (idx % 1024 < 256)
    m[hit] = rng.choice(np.array(m_edges, np.float32), hit.sum()) * rng.choice([-1.0, 1.0], hit.sum())
    hit_v = ((idx // 2048) % 2 == 1) & (idx % 1024 >= 512) & (idx % 1024 < 768)
    v[hit_v] = rng.choice(np.array(v_edges, np.float32), hit_v.sum())
    m, v = m.astype(np.float32), v.astype(np.float32)
    dev = [torch.tensor(a, device="cuda") for a in (p, g, m, v)]
    psa.adam_step_fp32([dev[0]], [dev[1]], [dev[2]], [dev[3]], step=3, **hp_kwargs(hp))
    p1, m1, v1 = p.copy(), m.copy(), v.copy()
    oracle.step_fp32(p1, g, m1, v1, 3, hp)
    for got, want in ((dev[0], p1), (dev[2], m1), (dev[3], v1)):
        assert np.array_equal(got.cpu().numpy().view(np.uint32), want.view(np.uint32))
