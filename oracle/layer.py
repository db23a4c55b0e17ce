"""Step 1 and the output projection of step 4 of the Gated-MLA layer, fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Page "Gated MLA（矩阵吸收版）":
* section "低秩压缩" (low-rank compression): c = RMSNorm(W_down x), shape [B,T,r]
  (``latent``);
* section "完整计算流（四步）" step 1: q = W_q_up . RMSNorm(W_q_down x), [B,T,H,d_q]
  (``query``; the norm sits between the two projections);
* step 4: y = W_o [sigmoid(W_g x) * o_flat]; the gate logits W_g x (``gate_logits``)
  are what the hot path consumes, W_o (``output_projection``) is applied here only for
  the full-layer check;
* section "形状与参数对比" (parameter table): kv_down [r,D], kv_up [H(d_q+d_v), r],
  q_down [r_q,D], q_up [H d_q, r_q], gate [H d_v, D], o_proj [D, H d_v];
* section "代码对照" (code listing): kv_up.weight splits as a block, all heads'
  W_UK rows first, then all heads' W_UV rows; q is viewed as [B,T,H,d_q], head-major.

Readings where the page is silent: RMSNorm gain is 1 and eps = 1e-6; every
projection is bias-free.

Parity: pinned by properties the page's formulas fix, each a different statement
from the formula itself (tests/test_oracle_layer.py): q is linear in W_q_up and
invariant to positive scalings of W_q_down and of x; c is invariant to positive
scalings of W_down and of x, has unit RMS per row and points along W_down x; with
identity weights q, c and g reduce to closed forms; g and y are linear in their
weights and in their inputs; head h of q depends only on rows h*d_q .. h*d_q+d_q-1
of W_q_up.  Planted slips (the norm after W_q_up, no norm on c or on the query
path, a norm over the wrong axis, heads interleaved) are each rejected by them.
"""
from __future__ import annotations

import numpy as np

RMS_EPS = 1e-6


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def rmsnorm(z: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """Row RMS normalisation with unit gain: z / sqrt(mean(z^2) + eps) over the last axis."""
    z = _f64(z)
    return z / np.sqrt(np.mean(z * z, axis=-1, keepdims=True) + eps)


def latent(x, kv_down) -> np.ndarray:
    """c = RMSNorm(x . W_down^T): [..., D] -> [..., r] (section "低秩压缩")."""
    return rmsnorm(_f64(x) @ _f64(kv_down).T)


def query(x, q_down, q_up) -> np.ndarray:
    """q = RMSNorm(x . W_q_down^T) . W_q_up^T: [..., D] -> [..., H*d_q] (step 1)."""
    return rmsnorm(_f64(x) @ _f64(q_down).T) @ _f64(q_up).T


def gate_logits(x, gate_w) -> np.ndarray:
    """g = x . W_g^T: [..., D] -> [..., H*d_v], the pre-sigmoid gate of step 4."""
    return _f64(x) @ _f64(gate_w).T


def split_kv_up(kv_up: np.ndarray, H: int, d_q: int, d_v: int):
    """Block split of kv_up.weight [H(d_q+d_v), r] into W_UK [H,d_q,r], W_UV [H,d_v,r]."""
    r = kv_up.shape[1]
    assert kv_up.shape[0] == H * (d_q + d_v)
    return kv_up[: H * d_q].reshape(H, d_q, r), kv_up[H * d_q:].reshape(H, d_v, r)


def step1(x, kv_down, q_down, q_up, gate_w, H: int, d_q: int):
    """x [B,T,D] -> (q [B,T,H,d_q], c [B,T,r], g [B,T,H*d_v]) in fp64."""
    x = _f64(x)
    B, T, _ = x.shape
    q = query(x, q_down, q_up)
    return q.reshape(B, T, H, d_q), latent(x, kv_down), gate_logits(x, gate_w)


def output_projection(gated: np.ndarray, o_proj: np.ndarray) -> np.ndarray:
    """y = gated . W_o^T with W_o = o_proj.weight [D, H d_v]."""
    return _f64(gated) @ _f64(o_proj).T
