"""GPU parity of the whole Gated-MLA layer (mla_gated_layer_fwd) against the fp64 oracle.

Page "Gated MLA（矩阵吸收版）", section "完整计算流（四步）": step 1 (c = RMSNorm(x W_kv_down^T),
q = RMSNorm(x W_q_down^T) W_q_up^T, g = x W_gate^T), steps 2-4 (the absorbed attention) and
the output projection y = o W_o^T.  The oracle is ``oracle.layer_forward`` on the same
rounded inputs.  Bars: fp32 1e-4, bf16 2e-2 of max|oracle|, for y and for the
intermediate results the call leaves in its workspace (q, c, g, o).
"""
import dataclasses

import numpy as np
import pytest

from latent_compressed_attention_gb300 import workloads as W
from oracle import layer
from tests.conftest import gpu_available

pytestmark = pytest.mark.gpu

TOL_F32, TOL_BF16 = 1e-4, 2e-2


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


def rel_err(got, ref):
    return float(np.max(np.abs(got - ref)) / max(float(np.max(np.abs(ref))), 1e-30))


def run_layer(env, w, p, dtype_name):
    torch, lca, _ = env
    dt = torch.float32 if dtype_name == "f32" else torch.bfloat16
    to = lambda a: torch.tensor(np.asarray(a, np.float32), device="cuda").to(dt)  # noqa: E731
    ws = torch.empty(lca.mla_gated_layer_workspace_size(w.B, w.T, w.D, w.H, w.d_q, w.d_v, w.r, w.r_q, dt),
                     dtype=torch.uint8, device="cuda")
    y = lca.mla_gated_layer_fwd(to(p["x"]), to(p["q_down"]), to(p["q_up"]), to(p["kv_down"]), to(p["kv_up"]),
                                to(p["gate"]), to(p["o_proj"]), w.H, w.d_q, w.d_v, w.scale, workspace=ws)
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    views = lca.layer_workspace_views(ws, w.B, w.T, w.H, w.d_q, w.d_v, w.r, dt)
    f = lambda t: t.float().double().cpu().numpy()  # noqa: E731
    return f(y).reshape(w.B * w.T, w.D), [f(v) for v in views]


def rounded_layer(w, seed):
    p = W.draw_layer(w, seed=seed)
    return {k: W.round_to(v, w.dtype) for k, v in p.items()}


def check(env, w, p, rows, tol):
    _, _, oracle = env
    y, (q, c, g, o) = run_layer(env, w, p, w.dtype)
    ref = oracle.layer_forward(p["x"], p, w.H, w.d_q, w.d_v, w.scale, rows=rows)
    assert np.all(np.isfinite(y))
    assert rel_err(y[rows], ref) <= tol
    # step-1 intermediates on the same rows, and the latent for every row
    flat = p["x"].reshape(w.B * w.T, w.D)
    q_ref = layer.query(flat[rows], p["q_down"], p["q_up"])
    g_ref = layer.gate_logits(flat[rows], p["gate"])
    c_ref = layer.latent(flat, p["kv_down"])
    assert rel_err(q.reshape(w.B * w.T, -1)[rows], q_ref) <= tol
    assert rel_err(g.reshape(w.B * w.T, -1)[rows], g_ref) <= tol
    assert rel_err(c.reshape(w.B * w.T, -1), c_ref) <= tol
    return y, o


def test_toy_layer_f32_every_row(env):
    """The toy fp32 layer (B=2, T=128, D=256, H=8, d=16, r=32, r_q=64), every row."""
    w = W.TOY_LAYER_F32
    p = W.draw_layer(w, seed=0)
    check(env, w, p, np.arange(w.B * w.T), TOL_F32)


BF16_BASE = W.MID_PREFILL_BF16


@pytest.mark.parametrize("B,T,D,H,r_q", [(1, 1, 256, 2, 256), (1, 300, 512, 2, 256), (2, 129, 256, 4, 512),
                                         (1, 640, 768, 2, 768)])
def test_bf16_layer_shapes(env, B, T, D, H, r_q):
    """Ragged token counts (not multiples of the 128-row GEMM tile), small D and r_q."""
    w = dataclasses.replace(BF16_BASE, B=B, T=T, D=D, H=H, r_q=r_q, scale=1.0 / np.sqrt(128.0))
    p = rounded_layer(w, seed=B * 1000 + T)
    check(env, w, p, np.arange(w.B * w.T), TOL_BF16)


def sample_rows(B, T, n, seed):
    rng = np.random.default_rng(seed)
    t = np.unique(np.concatenate([[0, 1, 127, 128, T // 2, T - 2, T - 1], rng.integers(0, T, n)]))
    return rng.integers(0, B, t.size) * T + t


@pytest.mark.parametrize("name", ["mid_prefill_bf16", "k3_prefill_bf16"])
def test_full_size_layer_sampled_rows(env, name):
    """Configs 3 and 4 through step 1 (x ~ N(0,1), weights N(0, 0.02^2)), sampled rows."""
    w = W.WORKLOADS[name]
    p = rounded_layer(w, seed=0)
    check(env, w, p, sample_rows(w.B, w.T, 10, seed=3), TOL_BF16)
