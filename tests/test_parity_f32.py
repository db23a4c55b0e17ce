"""GPU parity of the fp32 prefill path against the fp64 oracle (tolerance 1e-4
of max|oracle|, the fp32 bound), through the C ABI."""
import numpy as np
import pytest

from latent_compressed_attention_gb300 import workloads as W
from tests.conftest import gpu_available

pytestmark = pytest.mark.gpu

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


def run(env, q, c, w_uk, w_uv, g, scale):
    torch, lca, _ = env
    t = lambda a: None if a is None else torch.tensor(a, dtype=torch.float32, device="cuda")  # noqa: E731
    out = lca.mla_absorbed_attn_fwd(t(q), t(c), t(w_uk), t(w_uv), t(g), scale)
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    return out.double().cpu().numpy()


def rel_err(got, ref):
    return np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30)


def test_toy_layer_f32(env):
    """The toy Gated-MLA layer (B=2, T=128, H=8, d=16, r=32), inputs through step 1."""
    _, _, oracle = env
    from oracle import layer
    w = W.TOY_LAYER_F32
    p = W.draw_layer(w)
    q, c, g = layer.step1(p["x"], p["kv_down"], p["q_down"], p["q_up"], p["gate"], w.H, w.d_q)
    w_uk, w_uv = layer.split_kv_up(p["kv_up"], w.H, w.d_q, w.d_v)
    q, c, g, w_uk, w_uv = (W.round_f32(a) for a in (q, c, g, w_uk, w_uv))
    got = run(env, q, c, w_uk, w_uv, g, w.scale)
    assert rel_err(got, oracle.prefill(q, c, w_uk, w_uv, g, w.scale)) <= TOL_F32


@pytest.mark.parametrize("B,T,H,dq,dv,r", [(1, 1, 1, 16, 16, 32), (2, 5, 3, 16, 16, 32), (1, 130, 2, 16, 16, 32),
                                           (2, 300, 2, 8, 12, 20), (1, 257, 1, 64, 64, 64), (3, 64, 4, 1, 3, 1)])
@pytest.mark.parametrize("gate", [True, False])
def test_shapes_f32(env, B, T, H, dq, dv, r, gate):
    _, _, oracle = env
    rng = np.random.default_rng(B * 1000 + T)
    q = W.round_f32(rng.standard_normal((B, T, H, dq)))
    c = W.round_f32(rng.standard_normal((B, T, r)))
    w_uk = W.round_f32(rng.standard_normal((H, dq, r)) * 0.3)
    w_uv = W.round_f32(rng.standard_normal((H, dv, r)) * 0.3)
    g = W.round_f32(rng.standard_normal((B, T, H * dv))) if gate else None
    got = run(env, q, c, w_uk, w_uv, g, 0.7)
    assert rel_err(got, oracle.prefill(q, c, w_uk, w_uv, g, 0.7)) <= TOL_F32


def test_peaky_attention_f32(env):
    """W_UK ~ N(0,1), scale 1: near one-hot attention exercises the mask and the online softmax."""
    _, _, oracle = env
    rng = np.random.default_rng(5)
    B, T, H, dq, dv, r = 2, 200, 3, 16, 16, 32
    q = W.round_f32(rng.standard_normal((B, T, H, dq)))
    c = W.round_f32(rng.standard_normal((B, T, r)))
    w_uk = W.round_f32(rng.standard_normal((H, dq, r)))
    w_uv = W.round_f32(rng.standard_normal((H, dv, r)) * 0.1)
    g = W.round_f32(rng.standard_normal((B, T, H * dv)))
    got = run(env, q, c, w_uk, w_uv, g, 1.0)
    assert rel_err(got, oracle.prefill(q, c, w_uk, w_uv, g, 1.0)) <= TOL_F32


def test_causality_bitwise_f32(env):
    rng = np.random.default_rng(6)
    B, T, H, dq, dv, r = 1, 150, 2, 16, 16, 32
    q = W.round_f32(rng.standard_normal((B, T, H, dq)))
    c = W.round_f32(rng.standard_normal((B, T, r)))
    w_uk = W.round_f32(rng.standard_normal((H, dq, r)) * 0.3)
    w_uv = W.round_f32(rng.standard_normal((H, dv, r)) * 0.3)
    g = W.round_f32(rng.standard_normal((B, T, H * dv)))
    base = run(env, q, c, w_uk, w_uv, g, 1.0)
    t0 = 77
    q2, c2 = q.copy(), c.copy()
    q2[:, t0 + 1:] = W.round_f32(q2[:, t0 + 1:] * 3 + 1)
    c2[:, t0 + 1:] = W.round_f32(c2[:, t0 + 1:] * -2)
    out = run(env, q2, c2, w_uk, w_uv, g, 1.0)
    assert np.array_equal(out[:, : t0 + 1], base[:, : t0 + 1])
