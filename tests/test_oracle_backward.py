"""Pins of the fp64 backward oracle: its gradients equal central finite
differences of the C forward oracle (an independent implementation of steps
2-4), element by element on tiny inputs, with and without the gate, at small
and large score scales."""
import numpy as np
import pytest

EPS = 1e-5


def tiny(seed, B=2, T=5, H=2, dq=3, dv=2, r=4, gate=True, wuk_std=0.5):
    rng = np.random.default_rng(seed)
    d = dict(q=rng.normal(size=(B, T, H, dq)), c=rng.normal(size=(B, T, r)),
             w_uk=rng.normal(scale=wuk_std, size=(H, dq, r)), w_uv=rng.normal(size=(H, dv, r)),
             gate=rng.normal(size=(B, T, H * dv)) if gate else None)
    dout = rng.normal(size=(B, T, H * dv))
    return d, dout


def loss(oracle, d, dout, scale):
    return float(np.sum(dout * oracle.prefill(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], scale)))


def numeric_grad(oracle, d, dout, scale, name):
    base = d[name]
    g = np.zeros_like(base)
    it = np.nditer(base, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        hi, lo = base.copy(), base.copy()
        hi[idx] += EPS
        lo[idx] -= EPS
        g[idx] = (loss(oracle, {**d, name: hi}, dout, scale) - loss(oracle, {**d, name: lo}, dout, scale)) / (2 * EPS)
    return g


@pytest.mark.parametrize("gate", [True, False])
@pytest.mark.parametrize("scale", [0.7, 3.0])
def test_gradients_match_finite_differences(oracle, gate, scale):
    d, dout = tiny(seed=11 + int(gate) + int(scale), gate=gate)
    got = oracle.prefill_backward(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], scale, dout)
    names = ["q", "c", "w_uk", "w_uv"] + (["gate"] if gate else [])
    keys = {"q": "dq", "c": "dc", "w_uk": "dw_uk", "w_uv": "dw_uv", "gate": "dgate"}
    for name in names:
        num = numeric_grad(oracle, d, dout, scale, name)
        ana = got[keys[name]]
        assert ana.shape == num.shape
        err = np.max(np.abs(ana - num)) / max(np.max(np.abs(num)), 1e-12)
        assert err < 1e-7, (name, err)
    if not gate:
        assert got["dgate"] is None


def test_first_token_gradient_has_no_score_path(oracle):
    # token 0 attends only to itself: its output is c_0 W_UV^T, whatever q_0 is, so dq at t = 0 is zero
    d, dout = tiny(seed=5, T=4)
    got = oracle.prefill_backward(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], 1.0, dout)
    assert np.all(got["dq"][:, 0] == 0.0)
    assert np.any(got["dq"][:, 1:] != 0.0)


def test_future_tokens_do_not_receive_gradient_from_the_past(oracle):
    # dout only on token t = 1: no gradient reaches q or c of tokens t > 1
    d, dout = tiny(seed=6, T=5)
    dout[:] = 0.0
    dout[:, 1] = 1.0
    got = oracle.prefill_backward(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], 1.0, dout)
    assert np.all(got["dq"][:, 2:] == 0.0) and np.all(got["dc"][:, 2:] == 0.0)


# ---- prefill_lse: each row's log-sum-exp of the scaled causal scores

def test_lse_single_token_is_the_score(oracle):
    """T = 1: one visible key, so the log-sum-exp is that key's scaled score."""
    d, _ = tiny(seed=41, T=1)
    lse = oracle.prefill_lse(d["q"], d["c"], d["w_uk"], 0.8)
    for b in range(2):
        for h in range(2):
            s = 0.8 * float((d["q"][b, 0, h] @ d["w_uk"][h]) @ d["c"][b, 0])
            assert abs(lse[b, h, 0] - s) < 1e-12


def test_lse_of_zero_queries_counts_the_visible_keys(oracle):
    """q = 0: every score is 0, so row t sums t + 1 ones."""
    d, _ = tiny(seed=42, T=6)
    lse = oracle.prefill_lse(np.zeros_like(d["q"]), d["c"], d["w_uk"], 1.3)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, 7)), lse.shape), rtol=0, atol=1e-14)


@pytest.mark.parametrize("scale", [0.5, 4.0])
def test_lse_rebuilds_the_forward_output(oracle, scale):
    """The weights exp(s - lse) applied to c, then W_UV^T and the gate, give the C forward oracle's output: lse is
    the normaliser of the same softmax (a dropped term or a wrong mask changes every row after the first)."""
    d, _ = tiny(seed=43, T=7)
    lse = oracle.prefill_lse(d["q"], d["c"], d["w_uk"], scale)
    ref = oracle.prefill(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], scale)
    B, T, H, _ = d["q"].shape
    dv = d["w_uv"].shape[1]
    out = np.zeros((B, T, H, dv))
    for b in range(B):
        for h in range(H):
            s = scale * (d["q"][b, :, h] @ d["w_uk"][h]) @ d["c"][b].T
            a = np.where(np.tril(np.ones((T, T), dtype=bool)), np.exp(s - lse[b, h][:, None]), 0.0)
            out[b, :, h] = (a @ d["c"][b]) @ d["w_uv"][h].T
    out = out.reshape(B, T, H * dv) / (1.0 + np.exp(-d["gate"]))
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
