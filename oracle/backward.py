"""fp64 gradients of the absorbed causal Gated-MLA attention (steps 2-4).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The page "Gated MLA（矩阵吸收版）" gives the forward only (section "完整计算流（四步）"
and its listing in section "代码对照").  This module takes the chain rule back
through those steps, in reverse order, per (batch, head), with the full
[T, T] score and weight matrices written out:

  step 2  q_abs = q . W_UK                  (absorb, einsum bthd,hdj->bthj)
          s     = scale * q_abs . c^T       (scores, masked above the diagonal)
          a     = softmax_rows(s)
  step 3  o_lat = a . c                     (latent weighting, same c)
          o     = o_lat . W_UV^T            (up-projection)
  step 4  out   = sigmoid(g) * o            (gate)

Given dL/dout it returns dL/dq, dL/dc, dL/dW_UK, dL/dW_UV and dL/dg.
Parity: pinned by central finite differences of the C forward oracle
(tests/test_oracle_backward.py).
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def prefill_backward(q, c, w_uk, w_uv, gate, scale: float, dout) -> dict:
    """Gradients of L = sum(dout * out) for out = prefill(q, c, w_uk, w_uv, gate, scale).

    Shapes as in ``oracle.prefill``: q [B,T,H,d_q], c [B,T,r], w_uk [H,d_q,r],
    w_uv [H,d_v,r], gate [B,T,H*d_v] or None, dout [B,T,H*d_v].
    Returns dict(dq, dc, dw_uk, dw_uv, dgate); dgate is None without a gate.
    """
    q, c, w_uk, w_uv, dout = _f64(q), _f64(c), _f64(w_uk), _f64(w_uv), _f64(dout)
    B, T, H, dq_dim = q.shape
    r = c.shape[-1]
    dv = w_uv.shape[1]
    g = None if gate is None else _f64(gate).reshape(B, T, H, dv)
    dout = dout.reshape(B, T, H, dv)
    visible = np.tril(np.ones((T, T), dtype=bool))   # key u <= query t
    dq = np.zeros_like(q)
    dc = np.zeros_like(c)
    dw_uk = np.zeros_like(w_uk)
    dw_uv = np.zeros_like(w_uv)
    dgate = None if g is None else np.zeros_like(g)
    for b in range(B):
        for h in range(H):
            # forward, kept for the backward
            q_abs = q[b, :, h, :] @ w_uk[h]                    # [T, r]
            s = np.where(visible, scale * (q_abs @ c[b].T), -np.inf)
            e = np.exp(s - s.max(axis=1, keepdims=True))
            a = e / e.sum(axis=1, keepdims=True)              # [T, T], zero above the diagonal
            o_lat = a @ c[b]                                   # [T, r]
            o = o_lat @ w_uv[h].T                              # [T, d_v]
            # step 4: out = sigmoid(g) * o
            if g is None:
                d_o = dout[b, :, h, :]
            else:
                sig = 1.0 / (1.0 + np.exp(-g[b, :, h, :]))
                dgate[b, :, h, :] = dout[b, :, h, :] * o * sig * (1.0 - sig)
                d_o = dout[b, :, h, :] * sig
            # step 3: o = o_lat . W_UV^T ; o_lat = a . c
            dw_uv[h] += d_o.T @ o_lat
            d_olat = d_o @ w_uv[h]                             # [T, r]
            d_a = d_olat @ c[b].T                              # [T, T]
            dc[b] += a.T @ d_olat
            # softmax rows: ds = a * (da - sum_u a da)
            d_s = a * (d_a - (a * d_a).sum(axis=1, keepdims=True))
            # step 2: s = scale * q_abs . c^T ; q_abs = q . W_UK
            d_qabs = scale * (d_s @ c[b])                      # [T, r]
            dc[b] += scale * (d_s.T @ q_abs)
            dq[b, :, h, :] = d_qabs @ w_uk[h].T
            dw_uk[h] += q[b, :, h, :].T @ d_qabs
    return dict(dq=dq, dc=dc, dw_uk=dw_uk, dw_uv=dw_uv,
                dgate=None if dgate is None else dgate.reshape(B, T, H * dv))


def prefill_lse(q, c, w_uk, scale: float) -> np.ndarray:
    """Each row's log-sum-exp of the scaled, causally masked scores, in fp64: the normaliser of the softmax of
    step 2 (page "Gated MLA（矩阵吸收版）", section "完整计算流（四步）"),

        lse[b, h, t] = ln sum_{u <= t} exp(scale * q_abs[b, t, h, :] . c[b, u, :]),   q_abs = q . W_UK[h]

    so that the weights are a[t, u] = exp(s[t, u] - lse[t]).  Returns [B, H, T].
    Parity: pinned by closed forms (T = 1; zero queries) and by rebuilding ``oracle.prefill``'s output from it
    (tests/test_oracle_backward.py).
    """
    q, c, w_uk = _f64(q), _f64(c), _f64(w_uk)
    B, T, H, _ = q.shape
    visible = np.tril(np.ones((T, T), dtype=bool))
    out = np.empty((B, H, T))
    for b in range(B):
        for h in range(H):
            s = np.where(visible, scale * ((q[b, :, h, :] @ w_uk[h]) @ c[b].T), -np.inf)
            m = s.max(axis=1)
            out[b, h] = m + np.log(np.exp(s - m[:, None]).sum(axis=1))
    return out

