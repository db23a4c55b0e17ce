"""GPU parity of the decode over an e4m3 latent cache (mla_latent_decode_fp8) and of the cache quantiser
(mla_quantize_latent_fp8), through the C ABI.

The cache bytes are made on the host by the pinned codec (workloads.quantize_e4m3, tests/test_e4m3_codec.py)
and given to the GPU as they are; the fp64 oracle decodes over the same bytes dequantised
(cache_scale * e4m3 value).  So the bar measures the kernel's own error, on the cache it was given:
max|gpu - oracle| <= 2e-2 * max|oracle|, the bf16 bar (q_abs, W_UV, the gate and the output are bf16).
The quantiser is integer-valued work: bit-exact against the host codec.
"""
import numpy as np
import pytest

from latent_compressed_attention_gb300 import workloads as W
from tests.conftest import gpu_available

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
SCALE = 0.0625   # RMSNorm rows (|c| <= sqrt(512) = 22.6) map inside e4m3's 448


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


def bf(torch, a):
    return torch.tensor(np.asarray(a, np.float32), device="cuda").to(torch.bfloat16)


def rel_err(got, ref):
    return float(np.max(np.abs(got - ref)) / max(float(np.max(np.abs(ref))), 1e-30))


def make_case(H, lens, max_len, seed=0, gate=False, q_mul=1.0, ld=None, poison=False):
    w = W.K3_DECODE_BF16
    lens = np.asarray(lens, np.int32)
    B = lens.size
    d = W.draw_decode(w, seed=seed, B=B, lens=np.clip(lens, 0, max_len), gate=gate, H=H)
    if q_mul != 1.0:
        d = dict(d)
        d["q_abs"] = W.round_bf16(d["q_abs"] * q_mul)
    rows = np.stack([W.decode_cache_rows(w, b, max_len, seed=seed) for b in range(B)])
    inv = np.float32(1.0) / np.float32(SCALE)
    c8 = W.quantize_e4m3(rows, inv)                          # [B, max_len, r] bytes
    if poison:   # rows at or past lens[b] hold e4m3 NaN patterns: they must never reach the result
        for b in range(B):
            c8[b, max(lens[b], 0):] = 0x7F
    ld = ld or w.r
    full = np.zeros((B, max_len, ld), np.uint8)
    full[:, :, : w.r] = c8
    return d, full, lens


def run(env, d, full, lens, scale=1.0, workspace=None):
    torch, lca, _ = env
    B, max_len, ld = full.shape
    c8 = torch.tensor(full, device="cuda")[:, :, :512]
    out = lca.mla_latent_decode_fp8(bf(torch, d["q_abs"]), c8, torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                    bf(torch, d["w_uv"]), SCALE, None if d["gate"] is None else bf(torch, d["gate"]),
                                    scale, workspace=workspace)
    torch.cuda.synchronize()
    return out.float().double().cpu().numpy(), lca.mla_get_device_error()


def oracle_ref(oracle, d, full, lens, scale=1.0):
    c = W.decode_e4m3(full[:, :, :512]) * SCALE
    c = np.where(np.isfinite(c), c, 0.0)
    for b in range(len(lens)):
        c[b, max(lens[b], 0):] = 0.0
    return oracle.decode(d["q_abs"], c, lens, d["w_uv"], d["gate"], scale)


@pytest.mark.parametrize("H,lens,max_len", [
    (8, [1, 130, 300], 300),
    (96, [1, 2, 127, 128, 129, 255, 256, 257], 300),
    (96, [0, 700, 0, 1500], 1600),
    (16, [513, 1000, 64, 1999, 5], 2048),
    (1, [40, 41], 64),
    (37, [300, 280, 1], 300),
])
@pytest.mark.parametrize("gate", [False, True])
def test_fp8_decode_shapes(env, H, lens, max_len, gate):
    _, _, oracle = env
    d, full, lens = make_case(H, lens, max_len, seed=len(lens) + H, gate=gate)
    got, err = run(env, d, full, lens)
    assert err == 0
    assert rel_err(got, oracle_ref(oracle, d, full, lens)) <= TOL_BF16
    for b in np.flatnonzero(lens == 0):
        assert np.all(got[b] == 0.0)


def test_fp8_decode_poisoned_tail_and_row_stride(env):
    _, _, oracle = env
    d, full, lens = make_case(96, [5, 200, 129, 1], 256, seed=3, poison=True, ld=576)
    got, err = run(env, d, full, lens)
    assert err == 0
    assert np.all(np.isfinite(got))
    assert rel_err(got, oracle_ref(oracle, d, full, lens)) <= TOL_BF16


@pytest.mark.parametrize("q_mul,scale", [(4.0, 1.0), (1.0, 0.5), (20.0, 0.25)])
def test_fp8_decode_wider_scores(env, q_mul, scale):
    """Score spreads of about 20 natural-log units and other softmax scales: the hi + lo split of q_abs and of
    the softmax weights keeps bf16-like precision."""
    _, _, oracle = env
    d, full, lens = make_case(32, [600, 50, 3000], 3000, seed=5, q_mul=q_mul)
    got, err = run(env, d, full, lens, scale=scale)
    assert err == 0
    assert rel_err(got, oracle_ref(oracle, d, full, lens, scale=scale)) <= TOL_BF16


def test_fp8_decode_stale_workspace(env):
    torch, lca, oracle = env
    d, full, lens = make_case(96, [32768, 0, 5, 1000], 32768, seed=21)
    need = lca.library().mla_latent_decode_fp8_workspace_size(len(lens), 96, 512, full.shape[1])
    ws = torch.full((need // 4 + 1,), float("nan"), dtype=torch.float32, device="cuda")
    got, err = run(env, d, full, lens, workspace=ws.view(torch.uint8))
    assert err == 0 and np.all(np.isfinite(got))
    assert rel_err(got, oracle_ref(oracle, d, full, lens)) <= TOL_BF16


def test_fp8_decode_full_workload_sampled(env):
    """The K3 decode workload (B=64, lengths U[1024, 32768], H=96) with its cache quantised on the host; the
    oracle checks a sample of sequences, including the longest and shortest."""
    torch, lca, oracle = env
    w = W.K3_DECODE_BF16
    d = W.draw_decode(w, seed=0)
    lens = d["lens"]
    inv = np.float32(1.0) / np.float32(SCALE)
    c8 = torch.zeros((w.B, w.max_len, w.r), dtype=torch.uint8, device="cuda")
    rows = {}
    for b in range(w.B):
        q = W.quantize_e4m3(W.decode_cache_rows(w, b, int(lens[b]), seed=0), inv)
        c8[b, : lens[b]] = torch.tensor(q, device="cuda")
        rows[b] = q
    out = lca.mla_latent_decode_fp8(bf(torch, d["q_abs"]), c8, torch.tensor(lens, device="cuda"), bf(torch, d["w_uv"]),
                                    SCALE, None, w.scale)
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    got = out.float().double().cpu().numpy()
    assert np.all(np.isfinite(got))
    for b in sorted({int(np.argmax(lens)), int(np.argmin(lens)), 0, 17, 63}):
        ref = oracle.decode(d["q_abs"][b:b + 1], (W.decode_e4m3(rows[b]) * SCALE)[None], lens[b:b + 1], d["w_uv"],
                            None, w.scale)
        assert rel_err(got[b:b + 1], ref) <= TOL_BF16, f"sequence {b} (len {lens[b]})"


@pytest.mark.parametrize("scale", [0.0625, 0.3, 2.0**-12])
def test_quantize_bit_exact(env, scale):
    """The GPU quantiser against the host codec, bit for bit: ordinary values, values that round to e4m3
    subnormals, values that saturate at +-448 (the smallest scale), signed zeros."""
    torch, lca, _ = env
    rng = np.random.default_rng(7)
    c = W.round_bf16(rng.standard_normal((300, 512)) * np.exp2(rng.integers(-8, 4, (300, 1))))
    c[0, :4] = [0.0, -0.0, 1e-30, -1e-30]
    got = lca.mla_quantize_latent_fp8(bf(torch, c), scale).cpu().numpy()
    want = W.quantize_e4m3(c, np.float32(1.0) / np.float32(scale))
    # a zero result may carry either sign bit (the host codec writes +0 for every zero)
    got_z = np.where((got & 0x7F) == 0, 0, got)
    assert np.array_equal(got_z, want)
