"""The 8-bit optimizer's options as the pages list them (AiDotNet PR #814, options list and
summary; fixture in tests/golden/pages_options.json) against what the library and its
binding expose (CPU: defaults, accepted ranges, the memory claims)."""
import inspect
import json
import os

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
PAGES = json.load(open(os.path.join(HERE, "golden", "pages_options.json")))


@pytest.fixture(scope="module")
def psa():
    import __graft_entry__
    __graft_entry__.build()
    import precision_state_adam_gb300 as psa
    return psa


def _defaults(fn):
    return {k: v.default for k, v in inspect.signature(fn).parameters.items() if v.default is not inspect.Parameter.empty}


def test_binding_defaults_follow_the_options_list(psa):
    for fn in (psa.adam_step_q8, psa.adam_step_q8v, psa.StepPlan.__init__):
        d = _defaults(fn)
        assert d["block_size"] == PAGES["block_size_default"] == psa.BLOCK
        assert d["stochastic_rounding"] is PAGES["use_stochastic_rounding_default"]
        assert d["seed"] == PAGES["random_seed"]
        # dynamic quantization (scales recomputed every step) unless static scales are asked for
        assert d["static_scales"] is (not PAGES["use_dynamic_quantization_default"])
    # compress both moments by default: the 8-bit mode keeps both moments in codes; keeping
    # m in fp32 is the separate q8v mode
    assert len(psa.zeros_state([], "q8")) == 4 and len(psa.zeros_state([], "q8v")) == 3
    # the percentile default of the options list is a documented one-argument choice here
    # (the binding's default is absmax, percentile 100)
    assert "99.9" in psa.adam_step_q8.__doc__


def test_percentile_range_of_the_options_list(orc):
    lo, hi = PAGES["quantization_percentile_range"]
    assert orc.percentile_rank(hi, 2048) == 1                      # 100: absmax
    assert orc.percentile_rank(PAGES["quantization_percentile_default"], 2048) == 3
    assert orc.percentile_rank(1e-6 + lo, 2048) == 2048            # just above 0: the minimum


def test_memory_claims(psa):
    n = 1 << 24
    fp32 = psa.state_bytes("fp32", n)
    q8 = psa.state_bytes("q8", n)
    assert 3.99 < fp32 / q8 < 4.0                                  # "about 4x"
    assert 2.0 < q8 / n < 2.01                                     # "about 2 bytes" + scales
