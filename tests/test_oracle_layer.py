"""Pins of the oracle's step 1 and output projection (oracle/layer.py).

Page "Gated MLA（矩阵吸收版）" fixes c = RMSNorm(W_down x) (section "低秩压缩"),
q = W_q_up . RMSNorm(W_q_down x) viewed as [B,T,H,d_q] (section "完整计算流（四步）",
step 1, and the listing's ``view`` in section "代码对照"), g = W_g x and
y = W_o [sigmoid(g) * o] (step 4).  The pages print no values for these
projections, so each pin checks a property those formulas imply and that is a
different statement from the formula itself:

* where the norm sits: q scales with W_q_up but not with W_q_down or x; c does
  not scale with W_down or x;
* what the norm does: c has unit RMS per row and points along W_down x; with
  W_q_up = I the query is the normalised W_q_down x, with W_g = I the gate
  logits are x, with W_o = I the output is its input;
* linearity of the plain projections in their weights and inputs;
* head layout: head h of q depends only on rows h*d_q .. h*d_q+d_q-1 of W_q_up.

``test_planted_slip_is_rejected`` plants plausible slips in a private copy of
oracle/layer.py (the norm after W_q_up, no norm on c, no norm on the query path,
a norm over the token axis, heads interleaved, the gate logits squashed) and
checks that these pins reject each one.
"""
import importlib.util
import os

import numpy as np
import pytest

from oracle import layer

SRC = layer.__file__


def _rel(a, b):
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b))) / max(np.max(np.abs(b)), 1e-300))


def failed_pins(L) -> list:
    """Names of the pins that module ``L`` (oracle/layer.py or a planted variant) fails."""
    rng = np.random.default_rng(31)
    B, T, D, H, dq, dv, r, rq = 2, 5, 24, 3, 4, 5, 7, 10
    x = rng.standard_normal((B, T, D))
    kv_down = rng.standard_normal((r, D))
    q_down = rng.standard_normal((rq, D))
    q_up = rng.standard_normal((H * dq, rq))
    gate_w = rng.standard_normal((H * dv, D))
    o_proj = rng.standard_normal((D, H * dv))
    bad = []

    def check(name, fn):
        try:
            if not fn():
                bad.append(name)
        except Exception:   # a shape slip that raises is a rejection too
            bad.append(name)

    q0, c0, g0 = L.step1(x, kv_down, q_down, q_up, gate_w, H, dq)
    # (1) the norm sits between the two query projections
    check("q_linear_in_q_up", lambda: _rel(L.step1(x, kv_down, q_down, 3.0 * q_up, gate_w, H, dq)[0], 3.0 * q0) < 1e-12
          and _rel(L.step1(x, kv_down, q_down, -2.0 * q_up, gate_w, H, dq)[0], -2.0 * q0) < 1e-12)
    check("q_invariant_to_q_down_scale", lambda: _rel(L.step1(x, kv_down, 7.0 * q_down, q_up, gate_w, H, dq)[0], q0) < 1e-7)
    check("q_invariant_to_x_scale", lambda: _rel(L.step1(4.0 * x, kv_down, q_down, q_up, gate_w, H, dq)[0], q0) < 1e-7)
    # (2) the latent is normalised
    check("c_invariant_to_kv_down_scale", lambda: _rel(L.step1(x, 5.0 * kv_down, q_down, q_up, gate_w, H, dq)[1], c0) < 1e-7)
    check("c_invariant_to_x_scale", lambda: _rel(L.step1(0.25 * x, kv_down, q_down, q_up, gate_w, H, dq)[1], c0) < 1e-6)
    check("c_shape", lambda: c0.shape == (B, T, r))
    check("c_unit_rms_rows", lambda: np.max(np.abs(np.sqrt(np.mean(c0 * c0, -1)) - 1.0)) < 1e-6)
    z = x @ kv_down.T

    def c_along_z():
        # c = z / rho with one positive rho per row
        ratio = c0 / z
        return np.all(ratio > 0) and np.max(np.abs(ratio / ratio[..., :1] - 1.0)) < 1e-12
    check("c_points_along_W_down_x", c_along_z)
    # (3) closed forms with identity weights
    eye_q = np.eye(rq)   # H*dq == rq for this check: 2 heads of 5

    def q_identity():
        q = L.step1(x, kv_down, q_down, eye_q, gate_w, 2, rq // 2)[0].reshape(B, T, rq)
        zq = x @ q_down.T
        return q.shape == (B, T, rq) and _rel(q, zq / np.sqrt(np.mean(zq * zq, -1, keepdims=True) + 1e-6)) < 1e-12
    check("q_closed_form_identity_up", q_identity)

    def g_identity():
        g = L.step1(x, kv_down, q_down, q_up, np.eye(D), H, dq)[2]
        return np.array_equal(g, x)
    check("g_closed_form_identity", g_identity)
    check("g_linear", lambda: _rel(L.step1(x, kv_down, q_down, q_up, -1.5 * gate_w, H, dq)[2], -1.5 * g0) < 1e-12
          and _rel(L.step1(2.0 * x, kv_down, q_down, q_up, gate_w, H, dq)[2], 2.0 * g0) < 1e-12)
    check("g_shape", lambda: g0.shape == (B, T, H * dv))
    # (4) head layout of the query
    def q_heads():
        for h in range(H):
            qu = np.zeros_like(q_up)
            qu[h * dq:(h + 1) * dq] = q_up[h * dq:(h + 1) * dq]
            qh = L.step1(x, kv_down, q_down, qu, gate_w, H, dq)[0]
            if qh.shape != (B, T, H, dq):
                return False
            others = np.delete(qh, h, axis=2)
            if np.any(others != 0.0) or _rel(qh[:, :, h], q0[:, :, h]) > 1e-12:
                return False
        return True
    check("q_head_h_uses_rows_of_head_h", q_heads)
    # (5) output projection
    gated = rng.standard_normal((B, T, H * dv))
    y0 = L.output_projection(gated, o_proj)
    check("y_shape", lambda: y0.shape == (B, T, D))
    check("y_linear", lambda: _rel(L.output_projection(gated, 2.5 * o_proj), 2.5 * y0) < 1e-12
          and _rel(L.output_projection(-gated, o_proj), -y0) < 1e-12)
    check("y_identity", lambda: np.array_equal(L.output_projection(gated, np.eye(H * dv)), gated))
    # (6) the row-wise functions agree with step1 (the layer composition uses them on row samples)
    flat = x.reshape(B * T, D)
    check("row_functions_match_step1",
          lambda: np.array_equal(L.latent(flat, kv_down), c0.reshape(B * T, r))
          and np.array_equal(L.query(flat, q_down, q_up), q0.reshape(B * T, H * dq))
          and np.array_equal(L.gate_logits(flat, gate_w), g0.reshape(B * T, H * dv)))
    # a zero row normalises to zero, not NaN (eps > 0)
    check("zero_row_stays_finite", lambda: np.array_equal(L.rmsnorm(np.zeros((2, 6))), np.zeros((2, 6))))
    return bad


def test_step1_and_output_projection_pins():
    assert failed_pins(layer) == []


MUTATIONS = {
    "norm_after_q_up": ("return rmsnorm(_f64(x) @ _f64(q_down).T) @ _f64(q_up).T",
                        "return rmsnorm(_f64(x) @ _f64(q_down).T @ _f64(q_up).T)"),
    "no_norm_on_latent": ("return rmsnorm(_f64(x) @ _f64(kv_down).T)", "return _f64(x) @ _f64(kv_down).T"),
    "no_norm_on_query": ("return rmsnorm(_f64(x) @ _f64(q_down).T) @ _f64(q_up).T",
                         "return (_f64(x) @ _f64(q_down).T) @ _f64(q_up).T"),
    "norm_over_token_axis": ("np.mean(z * z, axis=-1, keepdims=True)", "np.mean(z * z, axis=-2, keepdims=True)"),
    "heads_interleaved": ("return q.reshape(B, T, H, d_q), latent",
                          "return q.reshape(B, T, d_q, H).transpose(0, 1, 3, 2), latent"),
    "gate_squashed": ("return _f64(x) @ _f64(gate_w).T", "return np.tanh(_f64(x) @ _f64(gate_w).T)"),
    "norm_gain_sqrt2": ("return z / np.sqrt(", "return np.sqrt(2.0) * z / np.sqrt("),
}


def _load_variant(path, name):
    spec = importlib.util.spec_from_file_location(name, path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_slip_is_rejected(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / f"layer_{name}.py"
    path.write_text(src.replace(old, new))
    assert failed_pins(_load_variant(str(path), f"layer_{name}")) != [], f"planted slip {name} passed the pins"


def test_unmutated_copy_passes(tmp_path):
    path = tmp_path / "layer_copy.py"
    path.write_text(open(SRC).read())
    assert failed_pins(_load_variant(str(path), "layer_copy")) == []
