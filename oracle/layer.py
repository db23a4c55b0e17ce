"""Step 1 and the output projection of step 4 of the Gated-MLA layer, fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Page "Gated MLA（矩阵吸收版）":
* section "低秩压缩" (low-rank compression): c = RMSNorm(W_down x), shape [B,T,r];
* section "完整计算流（四步）" step 1: q = W_q_up . RMSNorm(W_q_down x), [B,T,H,d_q];
* step 4: y = W_o [sigmoid(W_g x) * o_flat]; the gate logits W_g x are what the
  hot path consumes, W_o is applied here only for the full-layer check;
* section "形状与参数对比" (parameter table): kv_down [r,D], kv_up [H(d_q+d_v), r],
  q_down [r_q,D], q_up [H d_q, r_q], gate [H d_v, D], o_proj [D, H d_v];
* section "代码对照" (code listing): kv_up.weight splits as a block, all heads'
  W_UK rows first, then all heads' W_UV rows.

Readings where the page is silent: RMSNorm gain is 1 and eps = 1e-6; every
projection is bias-free.  Parity of these projections is unpinned by the page
beyond shapes and the decompression cross-check (the page prints no values);
the tests pin RMSNorm's unit-RMS property and the kv_up split.
"""
from __future__ import annotations

import numpy as np

RMS_EPS = 1e-6


def rmsnorm(z: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """Row RMS normalisation with unit gain: z / sqrt(mean(z^2) + eps)."""
    z = np.asarray(z, dtype=np.float64)
    return z / np.sqrt(np.mean(z * z, axis=-1, keepdims=True) + eps)


def split_kv_up(kv_up: np.ndarray, H: int, d_q: int, d_v: int):
    """Block split of kv_up.weight [H(d_q+d_v), r] into W_UK [H,d_q,r], W_UV [H,d_v,r]."""
    r = kv_up.shape[1]
    assert kv_up.shape[0] == H * (d_q + d_v)
    return kv_up[: H * d_q].reshape(H, d_q, r), kv_up[H * d_q:].reshape(H, d_v, r)


def step1(x, kv_down, q_down, q_up, gate_w, H: int, d_q: int):
    """x [B,T,D] -> (q [B,T,H,d_q], c [B,T,r], g [B,T,H*d_v]) in fp64."""
    x = np.asarray(x, dtype=np.float64)
    B, T, _ = x.shape
    c = rmsnorm(x @ np.asarray(kv_down, np.float64).T)
    q = rmsnorm(x @ np.asarray(q_down, np.float64).T) @ np.asarray(q_up, np.float64).T
    g = x @ np.asarray(gate_w, np.float64).T
    return q.reshape(B, T, H, d_q), c, g


def output_projection(gated: np.ndarray, o_proj: np.ndarray) -> np.ndarray:
    """y = gated . W_o^T with W_o = o_proj.weight [D, H d_v]."""
    return np.asarray(gated, np.float64) @ np.asarray(o_proj, np.float64).T
