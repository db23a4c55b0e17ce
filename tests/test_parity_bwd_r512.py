"""GPU parity of the attention's backward at the real sizes (r = 512, d_q = d_v = 128, bf16 inputs, fp32
gradients, tensor cores) against the fp64 oracle's gradients (oracle.prefill_backward, pinned by finite
differences in tests/test_oracle_backward.py), through the C ABI.

Bar: the bf16 one, max|gpu - oracle| <= 2e-2 * max|oracle| for every gradient, on the same bf16 inputs.
Every product of the chain rule runs on bf16 operands (the attention matrix, its gradient and the per-head
intermediates are kept in bf16), so the gradients carry bf16-level error, not fp32's.  Shapes span several
128-token tiles and ragged tails, T = 1, with and without the gate, two softmax scales.
"""
import numpy as np
import pytest

from latent_compressed_attention_gb300 import workloads as W
from tests.conftest import gpu_available

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
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


def case(B, T, H, seed, gate=True, wuk_std=W.WEIGHT_STD):
    w = W.MID_PREFILL_BF16
    d = W.draw_prefill_direct(w, seed=seed, T=T, B=B, H=H, wuk_std=wuk_std)
    if not gate:
        d["gate"] = None
    d["dout"] = W.round_bf16(np.random.default_rng(seed + 1000).standard_normal((B, T, H * w.d_v)))
    return d


def run(env, d, scale):
    torch, lca, oracle = env
    t = lambda a: None if a is None else torch.tensor(np.asarray(a, np.float32), device="cuda").to(torch.bfloat16)  # noqa: E731
    got = lca.mla_absorbed_attn_bwd(t(d["q"]), t(d["c"]), t(d["w_uk"]), t(d["w_uv"]), t(d["gate"]), scale,
                                    t(d["dout"]))
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    ref = oracle.prefill_backward(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], scale, d["dout"])
    return {k: None if got[k] is None else got[k].double().cpu().numpy() for k in KEYS}, ref


def check(got, ref):
    """Each gradient against the bar relative to its own largest value.  Where the oracle's gradient is zero by
    a closed form (T = 1: a single visible key makes dS, dq and dW_UK vanish), the relative error is undefined;
    there the largest of all the gradients, times 1e-3, is the floor of the denominator."""
    top_all = max(float(np.max(np.abs(ref[k]))) for k in KEYS if ref[k] is not None)
    for k in KEYS:
        if ref[k] is None:
            assert got[k] is None
            continue
        assert np.all(np.isfinite(got[k])), k
        err = float(np.max(np.abs(got[k] - ref[k]))) / max(float(np.max(np.abs(ref[k]))), 1e-3 * top_all)
        assert err <= TOL_BF16, f"{k}: {err:.3e}"


@pytest.mark.parametrize("B,T,H", [(1, 512, 2), (2, 300, 2), (1, 129, 3), (1, 1, 2), (2, 640, 1)])
@pytest.mark.parametrize("scale", [1.0 / np.sqrt(128.0), 1.0])
def test_bwd_r512_shapes(env, B, T, H, scale):
    got, ref = run(env, case(B, T, H, seed=T + 7 * H), scale)
    check(got, ref)


def test_bwd_r512_no_gate(env):
    got, ref = run(env, case(1, 384, 2, seed=5, gate=False), 1.0)
    check(got, ref)


def test_bwd_r512_peaky(env):
    """W_UK ~ N(0, 0.04^2) with q ~ N(0, 1.5^2): a score spread of several natural-log units."""
    d = case(1, 400, 2, seed=9, wuk_std=0.04)
    d["q"] = W.round_bf16(d["q"] / W.MID_PREFILL_BF16.q_std * 1.5)
    got, ref = run(env, d, 1.0)
    check(got, ref)


def test_bwd_r512_repeatable(env):
    """No atomics: two calls give the same bits."""
    d = case(1, 256, 2, seed=11)
    a, _ = run(env, d, 1.0)
    b, _ = run(env, d, 1.0)
    for k in KEYS:
        assert np.array_equal(a[k], b[k]), k


def test_bwd_r512_stale_workspace(env):
    """Every workspace value a product reads was written by the same call: a workspace filled with NaN
    beforehand (a ragged T, so the last tiles have padding columns) still gives finite gradients that match."""
    torch, lca, _ = env
    d = case(1, 300, 2, seed=13)
    need = lca.library().mla_absorbed_attn_bwd_workspace_size(1, 300, 2, 128, 128, 512, lca.DTYPE_BF16)
    ws = torch.full((need // 4 + 1,), float("nan"), dtype=torch.float32, device="cuda").view(torch.uint8)
    t = lambda a: None if a is None else torch.tensor(np.asarray(a, np.float32), device="cuda").to(torch.bfloat16)  # noqa: E731
    got = lca.mla_absorbed_attn_bwd(t(d["q"]), t(d["c"]), t(d["w_uk"]), t(d["w_uv"]), t(d["gate"]), 1.0, t(d["dout"]),
                                    workspace=ws)
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    _, ref = run(env, d, 1.0)
    check({k: None if got[k] is None else got[k].double().cpu().numpy() for k in KEYS}, ref)


def test_bwd_r512_many_items_per_cta(env):
    """More work items than resident CTAs in the large products (624 attention-matrix tiles, 384 o_lat and dq_abs
    tiles, dc and the weight gradients split over K), a ragged T: each CTA's TMA ring runs on across items and
    its accumulator alternates between two TMEM halves.  Two calls give the same bits."""
    torch, lca, _ = env
    d = case(2, 1500, 4, seed=31)
    got, ref = run(env, d, 1.0 / np.sqrt(128.0))
    check(got, ref)
    t = lambda a: None if a is None else torch.tensor(np.asarray(a, np.float32), device="cuda").to(torch.bfloat16)  # noqa: E731
    again = lca.mla_absorbed_attn_bwd(t(d["q"]), t(d["c"]), t(d["w_uk"]), t(d["w_uv"]), t(d["gate"]),
                                      1.0 / np.sqrt(128.0), t(d["dout"]))
    torch.cuda.synchronize()
    for k in KEYS:
        if got[k] is not None:
            assert np.array_equal(got[k], again[k].double().cpu().numpy()), k


# ---- the forward's log-sum-exp, and the backward given the forward's output and log-sum-exp

TOL_LSE = 2e-2   # natural-log units: the relative error it puts on the softmax weights, the bf16 bar


def tensors(env, d):
    torch = env[0]
    t = lambda a: None if a is None else torch.tensor(np.asarray(a, np.float32), device="cuda").to(torch.bfloat16)  # noqa: E731
    return {k: t(d[k]) for k in ("q", "c", "w_uk", "w_uv", "gate", "dout")}


@pytest.mark.parametrize("B,T,H,scale", [(1, 300, 2, 1.0), (2, 200, 3, 1.0 / np.sqrt(128.0)), (1, 1, 2, 1.0)])
def test_fwd_lse_matches_the_oracle(env, B, T, H, scale):
    """Each row's log-sum-exp from the forward (bf16 inputs, f16 score operands) against the fp64 one; the output
    of the call is the plain forward's, bit for bit."""
    torch, lca, oracle = env
    d = case(B, T, H, seed=51 + T)
    x = tensors(env, d)
    plain = lca.mla_absorbed_attn_fwd(x["q"], x["c"], x["w_uk"], x["w_uv"], x["gate"], scale)
    out, lse = lca.mla_absorbed_attn_fwd(x["q"], x["c"], x["w_uk"], x["w_uv"], x["gate"], scale, return_lse=True)
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    assert torch.equal(out, plain)
    ref = oracle.prefill_lse(d["q"], d["c"], d["w_uk"], scale)
    got = lse.double().cpu().numpy()
    assert got.shape == ref.shape and np.all(np.isfinite(got))
    assert float(np.max(np.abs(got - ref))) <= TOL_LSE


@pytest.mark.parametrize("gate", [True, False])
def test_bwd_lse_matches_the_oracle(env, gate):
    """The backward given the forward's (out, lse): the forward is not run again, the attention matrix comes
    from lse and dgate from the gated output; every gradient against the oracle's."""
    torch, lca, oracle = env
    d = case(2, 300, 2, seed=61, gate=gate)
    x = tensors(env, d)
    out, lse = lca.mla_absorbed_attn_fwd(x["q"], x["c"], x["w_uk"], x["w_uv"], x["gate"], 1.0, return_lse=True)
    got = lca.mla_absorbed_attn_bwd(x["q"], x["c"], x["w_uk"], x["w_uv"], x["gate"], 1.0, x["dout"], out=out, lse=lse)
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    ref = oracle.prefill_backward(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], 1.0, d["dout"])
    check({k: None if got[k] is None else got[k].double().cpu().numpy() for k in KEYS}, ref)


def test_bwd_lse_peaky(env):
    """The peaky case (scores spread over several natural-log units) through the saved statistics."""
    torch, lca, oracle = env
    d = case(1, 400, 2, seed=9, wuk_std=0.04)
    d["q"] = W.round_bf16(d["q"] / W.MID_PREFILL_BF16.q_std * 1.5)
    x = tensors(env, d)
    out, lse = lca.mla_absorbed_attn_fwd(x["q"], x["c"], x["w_uk"], x["w_uv"], x["gate"], 1.0, return_lse=True)
    got = lca.mla_absorbed_attn_bwd(x["q"], x["c"], x["w_uk"], x["w_uv"], x["gate"], 1.0, x["dout"], out=out, lse=lse)
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    ref = oracle.prefill_backward(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], 1.0, d["dout"])
    check({k: None if got[k] is None else got[k].double().cpu().numpy() for k in KEYS}, ref)
