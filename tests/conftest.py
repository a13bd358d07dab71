import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def golden_rows(name):
    """Non-comment, non-empty lines of a golden fixture, split on whitespace."""
    with open(os.path.join(GOLDEN, name)) as fh:
        return [ln.split() for ln in fh if ln.strip() and not ln.startswith("#")]


@pytest.fixture(scope="session")
def tiny():
    """Tiny fp32 workload: its parameters (CPU), prompt and oracle models."""
    import spd_inputs as si
    from oracle import spd as ospd
    w = si.WORKLOADS["tiny_f32_n2"]
    params = si.generate_weights(w)
    prompt = si.prompt_tokens(w).tolist()
    models = ospd.build(w, params)
    return w, params, prompt, models


@pytest.fixture(scope="session")
def tiny_ar(tiny):
    from oracle import model as om
    w, params, prompt, (target, pdm) = tiny
    return om.greedy_ar(target, prompt, w.gen_len)
