"""Device-side failure path, without a fault: every wait in the library's
kernels is bounded, and a wait that gives up records MLA_ERR_DEVICE_TIMEOUT in
the device error word instead of hanging or trapping.  The probe entry point
waits on an mbarrier phase that nothing completes, the way a stalled pipeline
would; the host must read the timeout status, and the context must still run
the prefill correctly afterwards."""
import time

import numpy as np
import pytest

from latent_compressed_attention_gb300 import workloads as W
from tests.conftest import gpu_available

pytestmark = pytest.mark.gpu

ERR_DEVICE_TIMEOUT = -8
TOL_F32 = 1e-4


@pytest.fixture(scope="module")
def env():
    if not gpu_available():
        pytest.skip("no CUDA device")
    import torch

    import latent_compressed_attention_gb300 as lca
    import oracle
    from latent_compressed_attention_gb300 import _build
    _build.build()
    oracle.build()
    return torch, lca, oracle


def test_wait_that_gives_up_is_reported(env):
    torch, lca, _ = env
    assert lca.mla_get_device_error() == 0
    t0 = time.perf_counter()
    lca.mla_debug_wait_timeout(2000)   # 2 ms
    status = lca.mla_get_device_error()
    elapsed = time.perf_counter() - t0
    assert status == ERR_DEVICE_TIMEOUT
    assert lca.mla_status_string(status) == "device-side wait timed out"
    assert elapsed < 10.0                 # the wait ended by itself
    assert lca.mla_get_device_error() == 0   # reading clears the word


def test_context_still_runs_after_a_timeout(env):
    torch, lca, oracle = env
    lca.mla_debug_wait_timeout(1000)
    assert lca.mla_get_device_error() == ERR_DEVICE_TIMEOUT
    w = W.TOY_LAYER_F32
    d = W.draw_prefill_direct(w, seed=3, T=200, B=1, H=2)
    d = {k: None if v is None else W.round_f32(v) for k, v in d.items()}
    t = lambda a: None if a is None else torch.tensor(a, dtype=torch.float32, device="cuda")  # noqa: E731
    out = lca.mla_absorbed_attn_fwd(t(d["q"]), t(d["c"]), t(d["w_uk"]), t(d["w_uv"]), t(d["gate"]), w.scale)
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    ref = oracle.prefill(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], w.scale)
    got = out.double().cpu().numpy()
    assert np.max(np.abs(got - ref)) <= TOL_F32 * np.max(np.abs(ref))
