"""Pins of the fp64 oracle against what the Gated-MLA page and plain mathematics fix.

The oracle (oracle/mla_oracle.c) computes steps 2-4 of the page "Gated MLA（矩阵
吸收版）", section "完整计算流（四步）", in the absorbed order.  Each test below
checks it against something that is NOT the same formula retyped:

* explicit decompression (section "矩阵吸收的核心思路": k = c W_UK^T,
  v = c W_UV^T under ordinary causal attention), a different order of the
  products that the page states is equal (box "如果你只记一件事" and the
  associativity box "为什么可以先加权再乘 W_UV");
* a one-hot latent that makes the output equal the attention matrix itself,
  checked for rows summing to 1, zeros above the diagonal and against a
  library softmax;
* closed forms: T = 1, row 0, uniform attention (prefix mean), zero gate,
  dominant key;
* causality, head-permutation equivariance, batch independence;
* decode of token t equal to prefill row t;
* a brute-force pure-Python transcription on tiny inputs;
* a stored fixture written by tests/golden/make_golden.py.

Each pin is chosen so a plausible slip (transposed W_UK or W_UV, dropped
scale, off-by-one mask, wrong gate sign, missing normalisation, wrong flat
order of heads) fails at least one test.
"""
import json
import os

import numpy as np
import pytest
from scipy.special import expit, softmax

from latent_compressed_attention_gb300 import workloads as W
from oracle import layer

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(rng, B, T, H, dq, dv, r, gate=True, wstd=0.5):
    q = rng.standard_normal((B, T, H, dq))
    c = rng.standard_normal((B, T, r))
    w_uk = rng.standard_normal((H, dq, r)) * wstd
    w_uv = rng.standard_normal((H, dv, r)) * wstd
    g = rng.standard_normal((B, T, H * dv)) if gate else None
    return q, c, w_uk, w_uv, g


def decompressed(q, c, w_uk, w_uv, g, scale):
    """Ordinary causal MHA on explicitly decompressed keys and values."""
    B, T, H, dq = q.shape
    dv = w_uv.shape[1]
    k = np.einsum("btj,hdj->bhtd", c, w_uk)           # k_h = c W_UK,h^T
    v = np.einsum("btj,hvj->bhtv", c, w_uv)           # v_h = c W_UV,h^T
    s = scale * np.einsum("bthd,bhsd->bhts", q, k)
    s = np.where(np.triu(np.ones((T, T), bool), 1), -np.inf, s)
    o = np.einsum("bhts,bhsv->bthv", softmax(s, axis=-1), v).reshape(B, T, H * dv)
    return o if g is None else o * expit(g)


def rel_err(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# --------------------------------------------------------------------------- pin 1
@pytest.mark.parametrize("shape", [(1, 1, 1, 1, 1, 1), (2, 5, 3, 2, 3, 4), (1, 17, 2, 5, 7, 3),
                                   (2, 33, 4, 16, 16, 32), (1, 9, 2, 3, 2, 8)])
@pytest.mark.parametrize("scale", [1.0, 0.37, 2.5])
@pytest.mark.parametrize("gate", [True, False])
def test_absorbed_equals_decompressed(oracle, shape, scale, gate):
    rng = np.random.default_rng(hash((shape, scale, gate)) % 2**32)
    B, T, H, dq, dv, r = shape
    q, c, w_uk, w_uv, g = rand_case(rng, B, T, H, dq, dv, r, gate)
    got = oracle.prefill(q, c, w_uk, w_uv, g, scale)
    assert rel_err(got, decompressed(q, c, w_uk, w_uv, g, scale)) < 1e-12


def test_absorbed_equals_decompressed_toy_layer(oracle):
    """The toy fp32 layer through step 1: absorbed == decompressed, and W_o applies."""
    w = W.TOY_LAYER_F32
    p = W.draw_layer(w, T=64)
    q, c, g = layer.step1(p["x"], p["kv_down"], p["q_down"], p["q_up"], p["gate"], w.H, w.d_q)
    w_uk, w_uv = layer.split_kv_up(p["kv_up"], w.H, w.d_q, w.d_v)
    got = oracle.prefill(q, c, w_uk, w_uv, g, w.scale)
    ref = decompressed(q, c, w_uk, w_uv, g, w.scale)
    assert rel_err(got, ref) < 1e-12
    y = layer.output_projection(got, p["o_proj"])
    assert y.shape == (w.B, 64, w.D)
    assert rel_err(y, ref @ p["o_proj"].T) < 1e-12


def test_layer_forward_is_the_composition_of_its_steps(oracle):
    """layer_forward (all rows, and a row sample) == step 1, prefill, W_o composed by hand, with the
    attention replaced by its explicit-decompression form, so a slip in the composition fails here."""
    w = W.TOY_LAYER_F32
    p = W.draw_layer(w, T=48, B=2)
    q, c, g = layer.step1(p["x"], p["kv_down"], p["q_down"], p["q_up"], p["gate"], w.H, w.d_q)
    w_uk, w_uv = layer.split_kv_up(p["kv_up"], w.H, w.d_q, w.d_v)
    ref = decompressed(q, c, w_uk, w_uv, g, 0.7) @ p["o_proj"].T
    full = oracle.layer_forward(p["x"], p, w.H, w.d_q, w.d_v, 0.7)
    assert full.shape == (2, 48, w.D)
    assert rel_err(full, ref) < 1e-12
    rows = np.array([0, 5, 47, 48, 70, 95])
    part = oracle.layer_forward(p["x"], p, w.H, w.d_q, w.d_v, 0.7, rows=rows)
    assert rel_err(part, ref.reshape(96, w.D)[rows]) < 1e-12


def test_peaky_attention_equals_decompressed(oracle):
    """Stress case: W_UK ~ N(0,1) makes attention nearly one-hot; the identity still holds."""
    rng = np.random.default_rng(7)
    q, c, w_uk, w_uv, g = rand_case(rng, 2, 40, 3, 16, 16, 32, wstd=1.0)
    got = oracle.prefill(q, c, w_uk, w_uv, g, 1.0)
    assert rel_err(got, decompressed(q, c, w_uk, w_uv, g, 1.0)) < 1e-12


# --------------------------------------------------------------------------- pin 2
def attention_matrix_via_one_hot_latent(oracle, q_abs_scores_q, w_uk, scale):
    """With c[u] = e_u (r >= T), W_UV = I and no gate, out[t, h*r + u] = attn[h, t, u]."""
    B, T, H, dq = q_abs_scores_q.shape
    r = w_uk.shape[2]
    c = np.zeros((B, T, r))
    for u in range(T):
        c[:, u, u] = 1.0
    w_uv = np.broadcast_to(np.eye(r), (H, r, r)).copy()
    out = oracle.prefill(q_abs_scores_q, c, w_uk, w_uv, None, scale)
    return out.reshape(B, T, H, r)[..., :T].transpose(0, 2, 1, 3)   # [B,H,T,T]


@pytest.mark.parametrize("scale", [1.0, 3.0])
def test_softmax_rows_sum_to_one_and_causal(oracle, scale):
    rng = np.random.default_rng(11)
    B, T, H, dq, r = 2, 12, 3, 5, 16
    q = rng.standard_normal((B, T, H, dq))
    w_uk = rng.standard_normal((H, dq, r))
    a = attention_matrix_via_one_hot_latent(oracle, q, w_uk, scale)
    assert np.all(a >= 0)
    assert np.max(np.abs(a.sum(-1) - 1.0)) < 1e-13
    upper = np.triu(np.ones((T, T), bool), 1)
    assert np.all(a[..., upper] == 0.0)
    # the scores of a one-hot latent are the first T entries of q_abs
    q_abs = np.einsum("bthd,hdj->bhtj", q, w_uk)[..., :T] * scale
    ref = softmax(np.where(upper, -np.inf, q_abs), axis=-1)
    assert np.max(np.abs(a - ref)) < 1e-13


# --------------------------------------------------------------------------- pin 3
def test_T1_closed_form(oracle):
    """T = 1: the only key is the query's own token, so out = sigmoid(g) * (c_0 W_UV^T)."""
    rng = np.random.default_rng(3)
    B, H, dq, dv, r = 3, 4, 6, 5, 7
    q, c, w_uk, w_uv, g = rand_case(rng, B, 1, H, dq, dv, r)
    got = oracle.prefill(q, c, w_uk, w_uv, g, 1.7)
    ref = np.einsum("bj,hvj->bhv", c[:, 0], w_uv).reshape(B, 1, H * dv) * expit(g)
    assert rel_err(got, ref) < 1e-13


def test_row0_closed_form(oracle):
    rng = np.random.default_rng(4)
    q, c, w_uk, w_uv, g = rand_case(rng, 2, 9, 3, 4, 6, 8)
    got = oracle.prefill(q, c, w_uk, w_uv, g, 1.0)[:, 0]
    ref = np.einsum("bj,hvj->bhv", c[:, 0], w_uv).reshape(2, 18) * expit(g[:, 0])
    assert rel_err(got, ref) < 1e-13


# --------------------------------------------------------------------------- pin 4
def test_causality_future_tokens_do_not_matter(oracle):
    rng = np.random.default_rng(5)
    B, T, H, dq, dv, r = 2, 14, 2, 4, 4, 8
    q, c, w_uk, w_uv, g = rand_case(rng, B, T, H, dq, dv, r)
    base = oracle.prefill(q, c, w_uk, w_uv, g, 1.0)
    for t in (0, 5, 12):
        q2, c2, g2 = q.copy(), c.copy(), g.copy()
        q2[:, t + 1:] += rng.standard_normal(q2[:, t + 1:].shape) * 3
        c2[:, t + 1:] += rng.standard_normal(c2[:, t + 1:].shape) * 3
        g2[:, t + 1:] -= 2.0
        out = oracle.prefill(q2, c2, w_uk, w_uv, g2, 1.0)
        assert np.array_equal(out[:, : t + 1], base[:, : t + 1])
        assert not np.array_equal(out[:, t + 1:], base[:, t + 1:])


# --------------------------------------------------------------------------- pin 5
def brute_force(q, c, w_uk, w_uv, g, scale):
    """Literal loops over the page's four einsums, building the full [B,H,T,T] matrix."""
    import math
    B, T, H, dq = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    r = len(c[0][0])
    dv = len(w_uv[0])
    q_abs = [[[[sum(q[b][t][h][d] * w_uk[h][d][j] for d in range(dq)) for j in range(r)]
               for h in range(H)] for t in range(T)] for b in range(B)]
    out = [[[0.0] * (H * dv) for _ in range(T)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            score = [[scale * sum(q_abs[b][t][h][j] * c[b][s][j] for j in range(r)) if s <= t else -math.inf
                      for s in range(T)] for t in range(T)]
            for t in range(T):
                mx = max(score[t])
                e = [math.exp(x - mx) if x != -math.inf else 0.0 for x in score[t]]
                attn = [x / sum(e) for x in e]
                lat = [sum(attn[s] * c[b][s][j] for s in range(T)) for j in range(r)]
                for v in range(dv):
                    o = sum(lat[j] * w_uv[h][v][j] for j in range(r))
                    gv = g[b][t][h * dv + v]
                    out[b][t][h * dv + v] = o / (1.0 + math.exp(-gv))
    return np.array(out)


@pytest.mark.parametrize("shape", [(1, 1, 1, 1, 1, 1), (2, 3, 2, 2, 3, 4), (1, 5, 2, 3, 2, 3)])
def test_brute_force_tiny(oracle, shape):
    rng = np.random.default_rng(sum(shape))
    q, c, w_uk, w_uv, g = rand_case(rng, *shape)
    ref = brute_force(q.tolist(), c.tolist(), w_uk.tolist(), w_uv.tolist(), g.tolist(), 0.8)
    assert rel_err(oracle.prefill(q, c, w_uk, w_uv, g, 0.8), ref) < 1e-13


# --------------------------------------------------------------------------- extra closed forms
@pytest.mark.parametrize("how", ["zero_q", "zero_scale"])
def test_uniform_attention_gives_prefix_mean(oracle, how):
    rng = np.random.default_rng(6)
    B, T, H, dq, dv, r = 2, 11, 3, 4, 5, 6
    q, c, w_uk, w_uv, g = rand_case(rng, B, T, H, dq, dv, r)
    scale = 1.0
    if how == "zero_q":
        q[:] = 0.0
    else:
        scale = 0.0
    got = oracle.prefill(q, c, w_uk, w_uv, g, scale)
    prefix_mean = np.cumsum(c, axis=1) / np.arange(1, T + 1)[None, :, None]
    ref = np.einsum("btj,hvj->bthv", prefix_mean, w_uv).reshape(B, T, H * dv) * expit(g)
    assert rel_err(got, ref) < 1e-13


def test_zero_gate_halves_and_large_gate_passes(oracle):
    rng = np.random.default_rng(8)
    q, c, w_uk, w_uv, g = rand_case(rng, 2, 7, 2, 3, 4, 5)
    plain = oracle.prefill(q, c, w_uk, w_uv, None, 1.0)
    assert rel_err(oracle.prefill(q, c, w_uk, w_uv, np.zeros_like(g), 1.0), plain / 2) < 1e-15
    assert rel_err(oracle.prefill(q, c, w_uk, w_uv, np.full_like(g, 40.0), 1.0), plain) < 1e-15
    assert np.max(np.abs(oracle.prefill(q, c, w_uk, w_uv, np.full_like(g, -40.0), 1.0))) < 1e-15


def test_dominant_key(oracle):
    """q_abs aligned with one latent row and a large scale: the output is that row's value."""
    B, T, H, r, dv = 1, 6, 2, 6, 3
    c = np.eye(T, r)[None]                       # c_u = e_u
    w_uk = np.broadcast_to(np.eye(r), (H, r, r)).copy()
    target = [0, 0, 1, 3, 2, 5]                  # key each query points at (<= t)
    q = np.zeros((B, T, H, r))
    for t, u in enumerate(target):
        q[0, t, :, u] = 1.0
    rng = np.random.default_rng(9)
    w_uv = rng.standard_normal((H, dv, r))
    got = oracle.prefill(q, c, w_uk, w_uv, None, 60.0).reshape(T, H, dv)
    ref = np.stack([np.einsum("j,hvj->hv", c[0, u], w_uv) for u in target])
    assert np.max(np.abs(got - ref)) < 1e-20 + 1e-12 * np.max(np.abs(ref))


def test_head_permutation_and_batch_independence(oracle):
    rng = np.random.default_rng(10)
    B, T, H, dq, dv, r = 3, 8, 4, 3, 2, 5
    q, c, w_uk, w_uv, g = rand_case(rng, B, T, H, dq, dv, r)
    base = oracle.prefill(q, c, w_uk, w_uv, g, 1.0).reshape(B, T, H, dv)
    perm = np.array([2, 0, 3, 1])
    gp = g.reshape(B, T, H, dv)[:, :, perm].reshape(B, T, H * dv)
    out = oracle.prefill(q[:, :, perm], c, w_uk[perm], w_uv[perm], gp, 1.0).reshape(B, T, H, dv)
    assert np.array_equal(out, base[:, :, perm])
    one = oracle.prefill(q[1:2], c[1:2], w_uk, w_uv, g[1:2], 1.0).reshape(1, T, H, dv)
    assert np.array_equal(one[0], base[1])


def test_row_sampling_matches_full(oracle):
    rng = np.random.default_rng(12)
    B, T = 2, 10
    q, c, w_uk, w_uv, g = rand_case(rng, B, T, 2, 3, 3, 4)
    full = oracle.prefill(q, c, w_uk, w_uv, g, 1.0).reshape(B * T, -1)
    rows = np.array([0, 7, 12, 19, 3])
    assert np.array_equal(oracle.prefill(q, c, w_uk, w_uv, g, 1.0, rows=rows), full[rows])


# --------------------------------------------------------------------------- decode
def test_decode_equals_prefill_row(oracle):
    rng = np.random.default_rng(13)
    B, T, H, dq, dv, r = 2, 9, 3, 4, 5, 6
    q, c, w_uk, w_uv, g = rand_case(rng, B, T, H, dq, dv, r)
    pre = oracle.prefill(q, c, w_uk, w_uv, g, 0.9)
    for t in (0, 4, 8):
        q_abs = np.einsum("bhd,hdj->bhj", q[:, t], w_uk)
        cache = np.concatenate([c, rng.standard_normal((B, 3, r))], axis=1)   # rows past lens are ignored
        got = oracle.decode(q_abs, cache, np.full(B, t + 1), w_uv, g[:, t], 0.9)
        assert rel_err(got, pre[:, t]) < 1e-12


def test_decode_ragged_lens_and_zero_length(oracle):
    rng = np.random.default_rng(14)
    B, H, dv, r, L = 4, 2, 3, 5, 12
    q_abs = rng.standard_normal((B, H, r))
    cache = rng.standard_normal((B, L, r))
    w_uv = rng.standard_normal((H, dv, r))
    lens = np.array([3, 0, 12, 1])
    out = oracle.decode(q_abs, cache, lens, w_uv, None, 1.0)
    assert np.all(out[1] == 0.0)
    # lens == 1: the single row's value, independent of the query
    assert rel_err(out[3], np.einsum("j,hvj->hv", cache[3, 0], w_uv).ravel()) < 1e-14
    # explicit decompression for the others
    for b in (0, 2):
        n = lens[b]
        s = np.einsum("hj,uj->hu", q_abs[b], cache[b, :n])
        v = np.einsum("uj,hvj->huv", cache[b, :n], w_uv)
        ref = np.einsum("hu,huv->hv", softmax(s, -1), v).ravel()
        assert rel_err(out[b], ref) < 1e-12


# --------------------------------------------------------------------------- step 1 helpers
def test_rmsnorm_unit_rms_and_kv_up_split():
    rng = np.random.default_rng(15)
    z = rng.standard_normal((5, 32)) * 3
    n = layer.rmsnorm(z)
    assert np.max(np.abs(np.sqrt(np.mean(n * n, -1)) - 1.0)) < 1e-6
    H, dq, dv, r = 3, 2, 4, 5
    kv_up = np.arange(H * (dq + dv) * r, dtype=float).reshape(H * (dq + dv), r)
    w_uk, w_uv = layer.split_kv_up(kv_up, H, dq, dv)
    assert np.array_equal(w_uk[1, 0], kv_up[dq])            # head 1's first key row follows head 0's
    assert np.array_equal(w_uv[0, 0], kv_up[H * dq])         # value block starts after all key rows
    assert np.array_equal(w_uv[2, 3], kv_up[H * dq + 2 * dv + 3])


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-7, -2.5 - 2**-9, 3.0e-3])
    got = W.round_bf16(vals)
    assert list(got[:4]) == [1.0, 1.0, 1.0 + 2**-6, 1.0 + 2**-7]
    assert got[4] == -2.5
    assert abs(got[5] - 3.0e-3) <= 3.0e-3 * 2**-8


# --------------------------------------------------------------------------- golden fixture
def test_golden_fixture(oracle):
    with open(os.path.join(GOLDEN, "prefill_small.json")) as f:
        fx = json.load(f)
    a = {k: (None if fx[k] is None else np.array(fx[k])) for k in ("q", "c", "w_uk", "w_uv", "gate")}
    got = oracle.prefill(a["q"], a["c"], a["w_uk"], a["w_uv"], a["gate"], fx["scale"])
    assert np.max(np.abs(got - np.array(fx["out"]))) < 1e-12
