import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def oracle_named(oracle_mod):
    """(q, k, v, O_ref, LSE_ref) of a named workload: inputs and the full fp64
    oracle, computed once per session and shared by the test files."""
    import time

    from attention_forward_flashattention_gb300 import inputs as I
    cache = {}

    def get(name):
        if name not in cache:
            w = I.WORKLOADS[name]
            q, k, v = I.qkv_bits(w)
            t0 = time.perf_counter()
            o_ref, l_ref = oracle_mod.attn_fwd(q, k, v, w.dtype, w.causal, w.scale)
            get.seconds[name] = time.perf_counter() - t0
            cache[name] = (q, k, v, o_ref, l_ref)
        return cache[name]
    get.seconds = {}   # wall time of each full oracle run
    return get
