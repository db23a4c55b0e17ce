"""GPU parity of the cached-latent decode (split + merge kernels) against the
fp64 oracle, through the C ABI.  Bar: max|gpu - oracle| <= 2e-2 * max|oracle|
(bf16 inputs)."""
import numpy as np
import pytest

from latent_compressed_attention_gb300 import workloads as W
from tests.conftest import gpu_available

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
ERR_DEVICE_BOUNDS = -9


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


def bf(torch, a, dev="cuda"):
    return torch.tensor(np.asarray(a, np.float32), device=dev).to(torch.bfloat16)


def make_case(H, lens, max_len, seed=0, gate=False, ld=None, poison=False):
    w = W.K3_DECODE_BF16
    lens = np.asarray(lens, np.int32)
    B = lens.size
    d = W.draw_decode(w, seed=seed, B=B, lens=np.clip(lens, 0, max_len), gate=gate, H=H)
    cache = np.stack([W.decode_cache_rows(w, b, max_len, seed=seed) for b in range(B)])
    if poison:   # rows at or past lens[b] must never reach the result
        for b in range(B):
            cache[b, max(lens[b], 0):] = np.nan
    return d, cache, lens, ld


def run_decode(env, d, cache, lens, ld=None, scale=1.0):
    torch, lca, _ = env
    B, max_len, r = cache.shape
    if ld is None:
        c_dev = bf(torch, cache)
    else:
        full = torch.zeros((B, max_len, ld), dtype=torch.bfloat16, device="cuda")
        full[:, :, :r] = bf(torch, cache)
        c_dev = full[:, :, :r]
    out = lca.mla_latent_decode(bf(torch, d["q_abs"]), c_dev, torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                bf(torch, d["w_uv"]), None if d["gate"] is None else bf(torch, d["gate"]), scale)
    torch.cuda.synchronize()
    err = lca.mla_get_device_error()
    return out.float().double().cpu().numpy(), err


def rel_err(got, ref):
    return float(np.max(np.abs(got - ref)) / max(float(np.max(np.abs(ref))), 1e-30))


def oracle_ref(oracle, d, cache, lens, scale=1.0):
    clean = np.nan_to_num(cache, nan=0.0)
    return oracle.decode(d["q_abs"], clean, np.clip(lens, 0, cache.shape[1]), d["w_uv"], d["gate"], scale)


@pytest.mark.parametrize("H,lens,max_len", [
    (8, [1, 130, 300], 300),
    (96, [1, 2, 127, 128, 129, 255, 256, 257], 300),
    (96, [0, 700, 0, 1500], 1600),
    (16, [513, 1000, 64, 1999, 5], 2048),
    (1, [40, 41], 64),
    (37, [300, 280, 1], 300),
])
@pytest.mark.parametrize("gate", [False, True])
def test_decode_shapes(env, H, lens, max_len, gate):
    _, _, oracle = env
    d, cache, lens, _ = make_case(H, lens, max_len, seed=len(lens) + H, gate=gate)
    got, err = run_decode(env, d, cache, lens)
    assert err == 0
    ref = oracle_ref(oracle, d, cache, lens)
    assert rel_err(got, ref) <= TOL_BF16
    for b in np.flatnonzero(lens == 0):
        assert np.all(got[b] == 0.0)


def test_decode_poisoned_tail_rows(env):
    _, _, oracle = env
    d, cache, lens, _ = make_case(96, [5, 200, 129, 1], 256, seed=3, poison=True)
    got, err = run_decode(env, d, cache, lens)
    assert err == 0
    assert np.all(np.isfinite(got))
    assert rel_err(got, oracle_ref(oracle, d, cache, lens)) <= TOL_BF16


def test_decode_row_strided_cache(env):
    _, _, oracle = env
    d, cache, lens, _ = make_case(24, [100, 333, 77], 400, seed=4)
    got, err = run_decode(env, d, cache, lens, ld=576)
    assert err == 0
    assert rel_err(got, oracle_ref(oracle, d, cache, lens)) <= TOL_BF16


def test_decode_scale_and_peaky(env):
    _, _, oracle = env
    d, cache, lens, _ = make_case(32, [600, 50], 600, seed=5)
    d = dict(d)
    d["q_abs"] = W.round_bf16(d["q_abs"] * 20.0)   # score spread about 5 natural-log units
    got, err = run_decode(env, d, cache, lens, scale=0.9)
    assert err == 0
    assert rel_err(got, oracle_ref(oracle, d, cache, lens, scale=0.9)) <= TOL_BF16


def test_decode_lens_out_of_range_is_reported(env):
    """A length past max_len is clamped on the device and reported as a bounds error."""
    _, _, oracle = env
    d, cache, lens, _ = make_case(8, [50, 64], 64, seed=6)
    bad = np.array([50, 70], np.int32)
    got, err = run_decode(env, d, cache, bad)
    assert err == ERR_DEVICE_BOUNDS
    assert rel_err(got, oracle_ref(oracle, d, cache, lens)) <= TOL_BF16
    _, err2 = run_decode(env, d, cache, lens)
    assert err2 == 0


def test_decode_repeatable(env):
    d, cache, lens, _ = make_case(96, [900, 1200, 33], 1200, seed=7)
    a, _ = run_decode(env, d, cache, lens)
    b, _ = run_decode(env, d, cache, lens)
    assert np.array_equal(a, b)


def test_decode_full_workload_sampled(env):
    """The K3 decode workload (B=64, lens U[1024, 32768], H=96) as the benchmark runs it;
    the oracle checks a sample of sequences, including the longest and shortest."""
    torch, lca, oracle = env
    w = W.K3_DECODE_BF16
    d = W.draw_decode(w, seed=0)
    lens = d["lens"]
    cache = torch.empty((w.B, w.max_len, w.r), dtype=torch.bfloat16, device="cuda")
    for b in range(w.B):
        cache[b, : lens[b]] = bf(torch, W.decode_cache_rows(w, b, int(lens[b]), seed=0))
        cache[b, lens[b]:] = float("nan")
    out = lca.mla_latent_decode(bf(torch, d["q_abs"]), cache, torch.tensor(lens, device="cuda"),
                                bf(torch, d["w_uv"]), None, w.scale)
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    got = out.float().double().cpu().numpy()
    assert np.all(np.isfinite(got))
    pick = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 0, 17, 63})
    for b in pick:
        rows = W.decode_cache_rows(w, b, int(lens[b]), seed=0)[None]
        ref = oracle.decode(d["q_abs"][b:b + 1], rows, lens[b:b + 1], d["w_uv"], None, w.scale)
        assert rel_err(got[b:b + 1], ref) <= TOL_BF16, f"sequence {b} (len {lens[b]})"


@pytest.mark.parametrize("lens", [[32768, 0, 5, 1000], [0, 3000, 1, 0, 20000, 129]])
def test_decode_stale_workspace_is_never_read(env, lens):
    """The merge reads only the partial-result slots that the split kernel of the same call wrote:
    a caller workspace filled with NaN beforehand (ragged lengths, zeros, and one sequence long enough
    to be split across far more than 32 clusters) still gives the oracle's result, finite everywhere."""
    torch, lca, oracle = env
    H, max_len = 96, max(lens)
    d, cache, lens, _ = make_case(H, lens, max_len, seed=21)
    B = lens.size
    need = lca.mla_latent_decode_workspace_size(B, H, 512, max_len)
    ws = torch.full((need // 4 + 1,), float("nan"), dtype=torch.float32, device="cuda")
    out = lca.mla_latent_decode(bf(torch, d["q_abs"]), bf(torch, cache), torch.tensor(lens, device="cuda"),
                                bf(torch, d["w_uv"]), None, 1.0, workspace=ws.view(torch.uint8))
    torch.cuda.synchronize()
    assert lca.mla_get_device_error() == 0
    got = out.float().double().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert rel_err(got, oracle_ref(oracle, d, cache, lens)) <= TOL_BF16
    for b in np.flatnonzero(lens == 0):
        assert np.all(got[b] == 0.0)
