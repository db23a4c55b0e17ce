"""GPU parity of one decode step of the whole layer with the latent-cache append
(mla_gated_layer_decode) against the layer prefill and the fp64 oracle.

Page "Gated MLA（矩阵吸收版）": only the latent c is cached (section "低秩压缩"); a step
appends the new token's latent and attends to the cache through steps 2-4 of section
"完整计算流（四步）".  Decoding token t over the cached latents of tokens 0..t-1 must
give the layer prefill's row t.  Bar: bf16, 2e-2 of max|reference|.
"""
import dataclasses

import numpy as np
import pytest

from latent_compressed_attention_gb300 import workloads as W
from oracle import layer
from tests.conftest import gpu_available

pytestmark = pytest.mark.gpu

TOL = 2e-2


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


def bf(torch, a):
    return torch.tensor(np.asarray(a, np.float32), device="cuda").to(torch.bfloat16)


def weights(torch, p):
    return [bf(torch, p[k]) for k in ("q_down", "q_up", "kv_down", "kv_up", "gate", "o_proj")]


def test_decode_step_equals_prefill_row(env):
    """Two sequences at different positions: the appended latent and the output match the prefill."""
    torch, lca, oracle = env
    w = dataclasses.replace(W.MID_PREFILL_BF16, B=2, T=300, D=512, H=2, r_q=256, scale=1.0 / np.sqrt(128.0))
    p = {k: W.round_bf16(v) for k, v in W.draw_layer(w, seed=5).items()}
    x = bf(torch, p["x"])
    wt = weights(torch, p)
    ws = torch.empty(lca.mla_gated_layer_workspace_size(w.B, w.T, w.D, w.H, w.d_q, w.d_v, w.r, w.r_q,
                                                        torch.bfloat16), dtype=torch.uint8, device="cuda")
    y_pre = lca.mla_gated_layer_fwd(x, *wt, w.H, w.d_q, w.d_v, w.scale, workspace=ws)
    torch.cuda.synchronize()
    c_pre = lca.layer_workspace_views(ws, w.B, w.T, w.H, w.d_q, w.d_v, w.r, torch.bfloat16)[1]
    c_pre = c_pre.view(w.B, w.T, w.r)

    pos = [w.T - 1, 137]
    max_len = w.T + 8
    cache = torch.full((w.B, max_len, w.r), float("nan"), dtype=torch.bfloat16, device="cuda")
    for b, t in enumerate(pos):
        cache[b, :t] = c_pre[b, :t]          # rows past the new one stay NaN: never read
    lens = torch.tensor(pos, dtype=torch.int32, device="cuda")
    x_t = torch.stack([x[b, t] for b, t in enumerate(pos)])
    y_dec = lca.mla_gated_layer_decode(x_t, *wt, cache, lens, w.H, w.d_q, w.d_v, w.scale)
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    for b, t in enumerate(pos):
        appended = cache[b, t].float().cpu().numpy()
        assert rel_err(appended, c_pre[b, t].float().cpu().numpy()) <= TOL
        assert torch.isnan(cache[b, t + 1]).all()          # nothing else written
    got = y_dec.float().double().cpu().numpy()
    pre = np.stack([y_pre[b, t].float().double().cpu().numpy() for b, t in enumerate(pos)])
    assert rel_err(got, pre) <= TOL
    rows = [b * w.T + t for b, t in enumerate(pos)]
    ref = oracle.layer_forward(p["x"], p, w.H, w.d_q, w.d_v, w.scale, rows=rows)
    assert rel_err(got, ref) <= TOL


def decode_against_oracle(env, w, B, max_len, seed):
    """One step for B sequences at random positions, against the oracle's composition."""
    torch, lca, oracle = env
    p = {k: W.round_bf16(v) for k, v in W.draw_layer(dataclasses.replace(w, B=B, T=1), seed=seed).items()}
    x_t = p["x"].reshape(B, w.D)
    rng = np.random.default_rng(seed)
    pos = rng.integers(0, max_len - 1, B)
    dec = dataclasses.replace(W.K3_DECODE_BF16, B=B)
    cache_np = np.zeros((B, max_len, w.r))
    for b in range(B):
        cache_np[b, :pos[b]] = W.decode_cache_rows(dec, b, int(pos[b]), seed=seed)
    cache = bf(torch, cache_np)
    lens = torch.tensor(pos, dtype=torch.int32, device="cuda")
    y = lca.mla_gated_layer_decode(bf(torch, x_t), *weights(torch, p), cache, lens, w.H, w.d_q, w.d_v, w.scale)
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0

    # oracle: step 1 for the new tokens, absorb W_UK, append, decode over lens+1 rows, W_o
    c_t = layer.latent(x_t, p["kv_down"])
    q = layer.query(x_t, p["q_down"], p["q_up"]).reshape(B, w.H, w.d_q)
    g = layer.gate_logits(x_t, p["gate"])
    w_uk, w_uv = layer.split_kv_up(p["kv_up"], w.H, w.d_q, w.d_v)
    q_abs = np.einsum("bhd,hdj->bhj", q, w_uk)
    for b in range(B):
        cache_np[b, pos[b]] = c_t[b]
    o = oracle.decode(q_abs, cache_np, (pos + 1).astype(np.int32), w_uv, g, w.scale)
    ref = layer.output_projection(o, p["o_proj"])
    assert rel_err(y.float().double().cpu().numpy(), ref) <= TOL
    got_rows = np.stack([cache[b, pos[b]].float().cpu().numpy() for b in range(B)])
    assert rel_err(got_rows, c_t) <= TOL


def test_decode_step_full_size_dims(env):
    """D=7168, H=96, r_q=1536 (the K3 layer's sizes), four sequences of ragged synthetic caches."""
    decode_against_oracle(env, W.K3_PREFILL_BF16, B=4, max_len=4096, seed=9)


def test_decode_step_batch_past_one_row_tile(env):
    """130 sequences: two 128-row tiles in every projection and in the query absorption."""
    w = dataclasses.replace(W.MID_PREFILL_BF16, D=512, H=2, r_q=256, scale=1.0 / np.sqrt(128.0))
    decode_against_oracle(env, w, B=130, max_len=96, seed=4)


def test_decode_step_position_out_of_range_is_reported(env):
    torch, lca, _ = env
    w = dataclasses.replace(W.MID_PREFILL_BF16, B=2, T=1, D=256, H=2, r_q=256)
    p = {k: W.round_bf16(v) for k, v in W.draw_layer(w, seed=1).items()}
    max_len = 16
    cache = torch.zeros((2, max_len, w.r), dtype=torch.bfloat16, device="cuda")
    lens = torch.tensor([3, max_len], dtype=torch.int32, device="cuda")   # the second has no free row
    lca.mla_gated_layer_decode(bf(torch, p["x"].reshape(2, w.D)), *weights(torch, p), cache, lens, w.H, w.d_q,
                               w.d_v, 1.0)
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == -9
    assert cache[0, 3].abs().sum() > 0            # the valid sequence's latent was appended
    assert cache[1].abs().sum() == 0              # nothing written for the other
    assert lca.mla_get_device_error() == 0        # the word was cleared
