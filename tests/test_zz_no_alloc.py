"""mla_latent_decode_noalloc: the decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: a host framework may own all device
memory and hand this library only the inputs and outputs, or a serving loop
may forbid allocation once it runs.  For them the library keeps the decode's
partial results in its own device scratch array instead of a caller
workspace.  This file checks, through the C ABI, that two calls in a row
produce what mla_latent_decode produces (within the bf16 bar the other tests
use), and that a size needing more scratch than the array holds is refused
before anything is launched.  It sits in its own file, collected last.
"""
import ctypes

import numpy as np
import pytest

from latent_compressed_attention_gb300 import workloads as W
from tests.conftest import gpu_available

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
ERR_WORKSPACE = -5


@pytest.fixture(scope="module")
def env():
    if not gpu_available():
        pytest.skip("no CUDA device")
    import torch

    import latent_compressed_attention_gb300 as lca
    from latent_compressed_attention_gb300 import _build
    _build.build()
    return torch, lca


def bf(torch, a):
    return torch.tensor(np.asarray(a, np.float32), device="cuda").to(torch.bfloat16)


def call_noalloc(lca, q_abs, cache, lens, w_uv, gate, out, scale):
    """Call the C entry point directly: only inputs and outputs, no workspace."""
    B, max_len, r = cache.shape
    H, d_v = w_uv.shape[0], w_uv.shape[1]
    lib = lca.library()
    return lib.mla_latent_decode_noalloc(q_abs.data_ptr(), cache.data_ptr(), cache.stride(1), lens.data_ptr(),
                                         max_len, w_uv.data_ptr(), None if gate is None else gate.data_ptr(),
                                         ctypes.c_float(scale), out.data_ptr(), B, H, d_v, r, lca.DTYPE_BF16,
                                         None)


@pytest.mark.parametrize("H,lens,max_len,gate", [(96, [300, 1, 700, 0, 129], 800, True),
                                                  (16, [2000, 35, 1024], 2048, False)])
def test_noalloc_matches_workspace_decode_twice(env, H, lens, max_len, gate):
    torch, lca = env
    w = W.K3_DECODE_BF16
    lens = np.asarray(lens, np.int32)
    B = lens.size
    d = W.draw_decode(w, seed=11, B=B, lens=lens, gate=gate, H=H)
    cache = bf(torch, np.stack([W.decode_cache_rows(w, b, max_len, seed=11) for b in range(B)]))
    q_abs, w_uv = bf(torch, d["q_abs"]), bf(torch, d["w_uv"])
    g = None if d["gate"] is None else bf(torch, d["gate"])
    lens_dev = torch.tensor(lens, device="cuda")

    ref = lca.mla_latent_decode(q_abs, cache, lens_dev, w_uv, g, 1.0).float()
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    scale_ref = float(ref.abs().max())
    for _ in range(2):   # the scratch array keeps the previous call's contents
        out = torch.full((B, H * 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert call_noalloc(lca, q_abs, cache, lens_dev, w_uv, g, out, 1.0) == 0
        torch.cuda.synchronize()
        assert lca.mla_get_device_error() == 0
        err = float((out.float() - ref).abs().max())
        assert err <= TOL_BF16 * scale_ref


def test_noalloc_refuses_sizes_beyond_its_scratch(env):
    """A batch whose partial results exceed the fixed scratch array is refused, nothing launched."""
    torch, lca = env
    H, max_len = 96, 1
    # the smallest batch whose partial results need more than the 48 MiB array (a few hundred
    # sequences on a 152-SM GPU), so the refusal costs little device memory on a shared GPU
    B = next(b for b in range(1, 1 << 16) if lca.mla_latent_decode_workspace_size(b, H, 512, max_len) > 48 * 2**20)
    assert lca.mla_latent_decode_workspace_size(B - 1, H, 512, max_len) <= 48 * 2**20
    q_abs = torch.zeros((B, H, 512), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((B, max_len, 512), dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(B, dtype=torch.int32, device="cuda")
    w_uv = torch.zeros((H, 128, 512), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((B, H * 128), dtype=torch.bfloat16, device="cuda")
    assert call_noalloc(lca, q_abs, cache, lens, w_uv, None, out, 1.0) == ERR_WORKSPACE
    with pytest.raises(lca.MLAError):
        lca.mla_latent_decode_noalloc(q_abs, cache, lens, w_uv)
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
