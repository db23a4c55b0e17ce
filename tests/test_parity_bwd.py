"""GPU parity of the attention's backward (fp32, toy sizes) against the fp64
oracle's gradients, through the C ABI.

Bar: for every gradient, max|gpu - oracle| <= 1e-4 * max|oracle| (the fp32
bound), on the same fp32 inputs.  Shapes span several 16-token tiles, ragged
tails, T = 1, widths up to 64, with and without the gate, and a peaky softmax.
"""
import numpy as np
import pytest

from latent_compressed_attention_gb300 import workloads as W
from tests.conftest import gpu_available

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
KEYS = ("dq", "dc", "dw_uk", "dw_uv", "dgate")


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


def case(B, T, H, dq, dv, r, seed, gate=True, wuk_std=W.WEIGHT_STD):
    w = W.Workload(name="bwd", kind="prefill", dtype="f32", B=B, T=T, D=256, H=H, d_q=dq, d_v=dv, r=r,
                   r_q=64, scale=1.0, gate=gate, q_std=1.0)
    d = W.draw_prefill_direct(w, seed=seed, wuk_std=wuk_std)
    rng = np.random.default_rng(seed + 1000)
    d["dout"] = W.round_f32(rng.standard_normal((B, T, H * dv)))
    return d


def run(env, d, scale):
    torch, lca, oracle = env
    t = lambda a: None if a is None else torch.tensor(np.asarray(a, np.float32), device="cuda")  # noqa: E731
    got = lca.mla_absorbed_attn_bwd(t(d["q"]), t(d["c"]), t(d["w_uk"]), t(d["w_uv"]), t(d["gate"]), scale,
                                    t(d["dout"]))
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    ref = oracle.prefill_backward(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], scale, d["dout"])
    return {k: None if got[k] is None else got[k].double().cpu().numpy() for k in KEYS}, ref


def check(got, ref):
    scale = max(float(np.max(np.abs(ref[k]))) for k in KEYS if ref[k] is not None)
    for k in KEYS:
        if ref[k] is None:
            assert got[k] is None
            continue
        top = float(np.max(np.abs(ref[k])))
        if top == 0.0:
            # exactly zero in exact arithmetic (T = 1: one visible key, so the score path carries no
            # gradient to q); fp32 rounding must stay negligible against the other gradients
            assert np.max(np.abs(got[k])) <= 1e-6 * scale, k
            continue
        err = np.max(np.abs(got[k] - ref[k])) / top
        assert err <= TOL_F32, (k, err)


@pytest.mark.parametrize("B,T,H,dq,dv,r", [(2, 128, 8, 16, 16, 32), (1, 1, 1, 16, 16, 32), (2, 5, 3, 16, 16, 32),
                                           (1, 130, 2, 16, 16, 32), (1, 77, 2, 24, 40, 64), (1, 300, 1, 64, 64, 64)])
@pytest.mark.parametrize("gate", [True, False])
def test_backward_shapes(env, B, T, H, dq, dv, r, gate):
    d = case(B, T, H, dq, dv, r, seed=T + r + H, gate=gate)
    got, ref = run(env, d, 1.0)
    check(got, ref)


def test_backward_peaky_attention(env):
    d = case(1, 200, 2, 16, 16, 32, seed=7, wuk_std=0.5)
    got, ref = run(env, d, 2.0)
    check(got, ref)


def test_backward_toy_layer_inputs(env):
    """The toy layer's attention inputs (through step 1), as in the toy fp32 prefill test."""
    from oracle import layer
    w = W.TOY_LAYER_F32
    p = W.draw_layer(w)
    q, c, g = layer.step1(p["x"], p["kv_down"], p["q_down"], p["q_up"], p["gate"], w.H, w.d_q)
    w_uk, w_uv = layer.split_kv_up(p["kv_up"], w.H, w.d_q, w.d_v)
    rng = np.random.default_rng(3)
    d = dict(q=W.round_f32(q), c=W.round_f32(c), w_uk=W.round_f32(w_uk), w_uv=W.round_f32(w_uv), gate=W.round_f32(g),
             dout=W.round_f32(rng.standard_normal((w.B, w.T, w.H * w.d_v))))
    got, ref = run(env, d, w.scale)
    check(got, ref)


def test_backward_repeatable(env):
    d = case(2, 128, 8, 16, 16, 32, seed=9)
    a, _ = run(env, d, 1.0)
    b, _ = run(env, d, 1.0)
    assert np.array_equal(a["dq"], b["dq"]) and np.array_equal(a["dgate"], b["dgate"])   # no atomics
    for k in ("dc", "dw_uk", "dw_uv"):   # sums over thread blocks in any order
        assert np.max(np.abs(a[k] - b[k])) <= 1e-5 * np.max(np.abs(a[k]))


def case_bf16(B, T, H, dq, dv, r, seed, gate=True):
    w = W.Workload(name="bwd16", kind="prefill", dtype="bf16", B=B, T=T, D=256, H=H, d_q=dq, d_v=dv, r=r,
                   r_q=64, scale=1.0, gate=gate, q_std=1.0)
    d = W.draw_prefill_direct(w, seed=seed)
    rng = np.random.default_rng(seed + 2000)
    d["dout"] = W.round_bf16(rng.standard_normal((B, T, H * dv)))
    return d


def run_bf16(env, d, scale):
    torch, lca, oracle = env
    t = lambda a: None if a is None else torch.tensor(np.asarray(a, np.float32), device="cuda").to(torch.bfloat16)  # noqa: E731
    got = lca.mla_absorbed_attn_bwd(t(d["q"]), t(d["c"]), t(d["w_uk"]), t(d["w_uv"]), t(d["gate"]), scale,
                                    t(d["dout"]))
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    assert got["dq"].dtype == torch.float32
    ref = oracle.prefill_backward(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], scale, d["dout"])
    return {k: None if got[k] is None else got[k].double().cpu().numpy() for k in KEYS}, ref


@pytest.mark.parametrize("B,T,H,dq,dv,r,gate", [(2, 5, 3, 16, 16, 32, True), (1, 300, 2, 16, 16, 32, False),
                                                (1, 130, 2, 64, 32, 64, True)])
def test_backward_bf16_inputs(env, B, T, H, dq, dv, r, gate):
    """bf16 inputs are widened to fp32: the gradients meet the fp32 bar on the rounded inputs."""
    d = case_bf16(B, T, H, dq, dv, r, seed=T + H, gate=gate)
    got, ref = run_bf16(env, d, 1.0)
    check(got, ref)


def test_backward_toy_long_context_full(env):
    """The toy long-context configuration (B=4, T=2048, H=8, d=16, r=32, bf16 inputs), every gradient."""
    d = case_bf16(4, 2048, 8, 16, 16, 32, seed=1)
    got, ref = run_bf16(env, d, 1.0)
    check(got, ref)


@pytest.mark.parametrize("B,T,H,dq,dv,r", [(2, 65, 2, 16, 16, 16), (1, 70, 2, 8, 12, 20), (1, 150, 1, 33, 17, 40),
                                           (1, 64, 3, 5, 3, 1), (1, 129, 1, 64, 64, 63)])
def test_backward_padded_widths(env, B, T, H, dq, dv, r):
    """Widths that the 16-, 32- and 64-column tilings pad with zeros, and tile-edge sequence lengths."""
    d = case(B, T, H, dq, dv, r, seed=3 * T + r)
    got, ref = run(env, d, 0.7)
    check(got, ref)
