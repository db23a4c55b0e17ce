"""C-ABI checks that need no GPU: the library builds, loads and exports every
function include/mla.h declares, and host-side validation rejects bad
arguments before any CUDA call (fault injection on the host)."""
import ctypes
import os
import re

import pytest

import latent_compressed_attention_gb300 as lca
from latent_compressed_attention_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mla.h")

OK, ERR_NULL, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_WORKSPACE, ERR_UNSUPPORTED = 0, -1, -2, -3, -4, -5, -6
BF16, F32 = 0, 1
FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced: validation fails first


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return lca.library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("mla_absorbed_attn_fwd", "mla_latent_decode", "mla_latent_decode_workspace_size",
              "mla_get_device_error", "mla_status_string", "mla_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared in mla.h but not exported: {missing}"


def test_status_strings(lib):
    for code in range(-9, 1):
        assert lca.mla_status_string(code) != "unknown status"
    assert lca.mla_status_string(-99) == "unknown status"
    assert lca.mla_version() >= 100


def prefill(lib, q=FAKE, c=FAKE, wuk=FAKE, wuv=FAKE, gate=None, out=FAKE, B=1, T=16, H=2, dq=16, dv=16, r=32,
            dtype=F32, ws=None, ws_bytes=0):
    return lib.mla_absorbed_attn_fwd(q, c, wuk, wuv, gate, 1.0, out, B, T, H, dq, dv, r, dtype, ws, ws_bytes, None)


def test_prefill_workspace_sizes(lib):
    """Only the r = 512 kernel needs a workspace: an f16 copy of c (2 bytes per latent value), one maximum
    per 32 keys of each sequence and one scale per sequence."""
    assert lib.mla_absorbed_attn_fwd_workspace_size(2, 100, 4, 16, 16, 32, F32) == 0
    assert lib.mla_absorbed_attn_fwd_workspace_size(2, 100, 4, 16, 16, 32, BF16) == 0
    B, T = 3, 300
    need = lib.mla_absorbed_attn_fwd_workspace_size(B, T, 16, 128, 128, 512, BF16)
    c16 = (B * T * 512 * 2 + 255) // 256 * 256
    assert need == c16 + B * (10 + 1) * 4   # ceil(300 / 32) = 10 groups of 32 keys, and one scale
    assert lib.mla_absorbed_attn_fwd_workspace_size(B, T, 16, 128, 128, 512, 9) == 0


def test_prefill_r512_needs_its_workspace(lib):
    kw = dict(dtype=BF16, r=512, dq=128, dv=128, T=256)
    need = lib.mla_absorbed_attn_fwd_workspace_size(1, 256, 2, 128, 128, 512, BF16)
    assert prefill(lib, **kw) == ERR_WORKSPACE
    assert prefill(lib, ws=FAKE, ws_bytes=need - 1, **kw) == ERR_WORKSPACE
    assert prefill(lib, ws=FAKE + 8, ws_bytes=need, **kw) == ERR_ALIGN


@pytest.mark.parametrize("field", ["q", "c", "wuk", "wuv", "out"])
def test_prefill_null_pointer(lib, field):
    assert prefill(lib, **{field: None}) == ERR_NULL


@pytest.mark.parametrize("field", ["q", "c", "wuk", "wuv", "out", "gate"])
def test_prefill_misaligned_pointer(lib, field):
    assert prefill(lib, **{field: FAKE + 4}) == ERR_ALIGN


@pytest.mark.parametrize("kw", [dict(B=-1), dict(T=-1), dict(H=0), dict(dq=0), dict(dv=-3), dict(r=0),
                                dict(B=1 << 20, T=1 << 20)])
def test_prefill_bad_shape(lib, kw):
    assert prefill(lib, **kw) == ERR_SHAPE


def test_prefill_bad_dtype(lib):
    assert prefill(lib, dtype=7) == ERR_DTYPE


@pytest.mark.parametrize("kw", [dict(r=65), dict(dq=100), dict(dtype=BF16, r=48, dq=16, dv=16),
                                dict(dtype=BF16, r=512, dq=64, dv=128), dict(dtype=BF16, r=32, dq=8, dv=16),
                                dict(dtype=BF16, r=64, dq=16, dv=80), dict(B=1, T=1_048_561)])
def test_prefill_unsupported_shape(lib, kw):
    assert prefill(lib, **kw) == ERR_UNSUPPORTED


def test_prefill_empty_is_noop(lib):
    assert prefill(lib, B=0) == OK
    assert prefill(lib, T=0) == OK


def decode(lib, q=FAKE, cache=FAKE, ld=512, lens=FAKE, max_len=64, wuv=FAKE, gate=None, out=FAKE, B=2, H=8,
           dv=128, r=512, dtype=BF16, ws=None, ws_bytes=0):
    return lib.mla_latent_decode(q, cache, ld, lens, max_len, wuv, gate, 1.0, out, B, H, dv, r, dtype, ws,
                                 ws_bytes, None)


@pytest.mark.parametrize("field", ["q", "cache", "lens", "wuv", "out"])
def test_decode_null_pointer(lib, field):
    assert decode(lib, **{field: None}) == ERR_NULL


@pytest.mark.parametrize("kw", [dict(B=-1), dict(H=0), dict(dv=0), dict(r=0), dict(max_len=-1), dict(ld=100)])
def test_decode_bad_shape(lib, kw):
    assert decode(lib, **kw) == ERR_SHAPE


@pytest.mark.parametrize("kw", [dict(q=FAKE + 2), dict(lens=FAKE + 4), dict(ld=520 + 4)])
def test_decode_misaligned(lib, kw):
    assert decode(lib, **kw) == ERR_ALIGN


@pytest.mark.parametrize("kw", [dict(dtype=F32), dict(H=129), dict(r=256, ld=256), dict(dv=64)])
def test_decode_unsupported(lib, kw):
    assert decode(lib, **kw) == ERR_UNSUPPORTED


def decode_fp8(lib, q=FAKE, cache=FAKE, ld=512, lens=FAKE, max_len=64, cache_scale=0.0625, wuv=FAKE, gate=None,
               out=FAKE, B=2, H=8, dv=128, r=512, ws=None, ws_bytes=0):
    return lib.mla_latent_decode_fp8(q, cache, ld, lens, max_len, cache_scale, wuv, gate, 1.0, out, B, H, dv, r, ws,
                                     ws_bytes, None)


@pytest.mark.parametrize("field", ["q", "cache", "lens", "wuv", "out"])
def test_decode_fp8_null_pointer(lib, field):
    assert decode_fp8(lib, **{field: None}) == ERR_NULL


@pytest.mark.parametrize("kw", [dict(B=-1), dict(H=0), dict(r=0), dict(max_len=-1), dict(ld=100),
                                dict(cache_scale=0.0), dict(cache_scale=-1.0), dict(cache_scale=float("inf")),
                                dict(cache_scale=float("nan"))])
def test_decode_fp8_bad_shape(lib, kw):
    assert decode_fp8(lib, **kw) == ERR_SHAPE


@pytest.mark.parametrize("kw", [dict(ld=520), dict(cache=FAKE + 8), dict(lens=FAKE + 4)])
def test_decode_fp8_misaligned(lib, kw):
    assert decode_fp8(lib, **kw) == ERR_ALIGN


@pytest.mark.parametrize("kw", [dict(H=97), dict(r=256, ld=256), dict(dv=64)])
def test_decode_fp8_unsupported(lib, kw):
    assert decode_fp8(lib, **kw) == ERR_UNSUPPORTED


def test_decode_fp8_empty_batch_is_noop(lib):
    assert decode_fp8(lib, B=0) == OK


def quantize(lib, c=FAKE, ld_c=512, c8=FAKE, ld_c8=512, rows=4, r=512, cache_scale=0.0625):
    return lib.mla_quantize_latent_fp8(c, ld_c, c8, ld_c8, rows, r, cache_scale, None)


@pytest.mark.parametrize("kw,want", [(dict(r=12, ld_c=12, ld_c8=16), ERR_SHAPE), (dict(rows=-1), ERR_SHAPE),
                                     (dict(cache_scale=0.0), ERR_SHAPE), (dict(ld_c8=100), ERR_SHAPE),
                                     (dict(ld_c8=520), ERR_ALIGN), (dict(ld_c=516), ERR_ALIGN),
                                     (dict(c=FAKE + 2), ERR_ALIGN), (dict(c=None), ERR_NULL), (dict(rows=0), OK)])
def test_quantize_fp8_validation(lib, kw, want):
    assert quantize(lib, **kw) == want


def test_decode_bad_dtype(lib):
    assert decode(lib, dtype=3) == ERR_DTYPE


def test_workspace_size_rejects_bad_sizes(lib):
    assert lib.mla_latent_decode_workspace_size(0, 8, 512, 64) == 0
    assert lib.mla_latent_decode_workspace_size(2, 0, 512, 64) == 0
    assert lib.mla_latent_decode_workspace_size(2, 8, 48, 64) == 0


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 4, 2, 16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        lca.mla_absorbed_attn_fwd(x, torch.zeros(1, 4, 32), torch.zeros(2, 16, 32), torch.zeros(2, 16, 32))


def test_binding_refuses_cpu_tensors_everywhere():
    """Every entry point checks its tensors before any call into the library: there is no CPU path."""
    torch = pytest.importorskip("torch")
    z = torch.zeros
    with pytest.raises(ValueError, match="CUDA tensor"):
        lca.mla_absorbed_attn_bwd(z(1, 4, 2, 16), z(1, 4, 32), z(2, 16, 32), z(2, 16, 32), None, 1.0, z(1, 4, 32))
    with pytest.raises(ValueError, match="CUDA tensor"):
        lca.mla_latent_decode(z(2, 8, 512), z(2, 64, 512), torch.ones(2, dtype=torch.int32), z(8, 128, 512))
    with pytest.raises(ValueError, match="CUDA tensor"):
        lca.mla_gated_layer_fwd(z(1, 4, 256), z(64, 256), z(32, 64), z(32, 256), z(64, 32), z(32, 256), z(256, 32),
                                2, 16, 16)


# ----------------------------------------------------------------------------- whole layer
def layer(lib, x=FAKE, wqd=FAKE, wqu=FAKE, wkvd=FAKE, wkvu=FAKE, wg=FAKE, wo=FAKE, y=FAKE, B=1, T=16, D=256, H=2,
          dq=128, dv=128, r=512, rq=256, dtype=BF16, ws=FAKE, ws_bytes=1 << 40):
    return lib.mla_gated_layer_fwd(x, wqd, wqu, wkvd, wkvu, wg, wo, 1.0, y, B, T, D, H, dq, dv, r, rq, dtype, ws,
                                   ws_bytes, None)


@pytest.mark.parametrize("field", ["x", "wqd", "wqu", "wkvd", "wkvu", "wg", "wo", "y"])
def test_layer_null_pointer(lib, field):
    assert layer(lib, **{field: None}) == ERR_NULL


@pytest.mark.parametrize("field", ["x", "wo", "y", "ws"])
def test_layer_misaligned(lib, field):
    assert layer(lib, **{field: FAKE + 8}) == ERR_ALIGN


@pytest.mark.parametrize("kw", [dict(B=-1), dict(D=0), dict(H=0), dict(rq=0), dict(B=1 << 20, T=1 << 20)])
def test_layer_bad_shape(lib, kw):
    assert layer(lib, **kw) == ERR_SHAPE


@pytest.mark.parametrize("kw", [dict(H=3), dict(D=320), dict(rq=320), dict(r=256), dict(dq=64),
                                dict(dtype=F32, r=128, dq=16, dv=16), dict(dtype=F32, r=32, dq=16, dv=16, B=1, T=1_048_561)])
def test_layer_unsupported(lib, kw):
    assert layer(lib, **kw) == ERR_UNSUPPORTED


def test_layer_workspace_checked_before_launch(lib):
    need = lib.mla_gated_layer_workspace_size(1, 16, 256, 2, 128, 128, 512, 256, BF16)
    assert need > 0
    assert layer(lib, ws=None) == ERR_WORKSPACE
    assert layer(lib, ws_bytes=need - 1) == ERR_WORKSPACE
    assert layer(lib, dtype=9) == ERR_DTYPE
    assert layer(lib, T=0) == OK


def test_layer_workspace_size(lib):
    # q, c, g, o, the low-rank query and the row sums, each on a 256-byte boundary
    B, T, D, H, d, r, rq = 2, 128, 256, 8, 16, 32, 64
    M = B * T
    parts = [M * H * d * 4, M * r * 4, M * H * d * 4, M * H * d * 4, M * rq * 4, M * 4]
    assert lib.mla_gated_layer_workspace_size(B, T, D, H, d, d, r, rq, F32) == sum((p + 255) // 256 * 256
                                                                                   for p in parts)
    assert lib.mla_gated_layer_workspace_size(1, 16, 256, 3, 128, 128, 512, 256, BF16) == 0
    assert lib.mla_gated_layer_workspace_size(1, 16, 256, 2, 128, 128, 512, 256, 5) == 0


def layer_decode(lib, x=FAKE, y=FAKE, cache=FAKE, ld=512, lens=FAKE, max_len=64, B=2, D=256, H=2, r=512, rq=256,
                 dtype=BF16, ws=FAKE, ws_bytes=1 << 40):
    return lib.mla_gated_layer_decode(x, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, y, cache, ld, lens, max_len, B, D,
                                      H, 128, 128, r, rq, dtype, ws, ws_bytes, None)


@pytest.mark.parametrize("kw", [dict(x=None), dict(y=None), dict(cache=None), dict(lens=None)])
def test_layer_decode_null_pointer(lib, kw):
    assert layer_decode(lib, **kw) == ERR_NULL


@pytest.mark.parametrize("kw", [dict(ld=100), dict(max_len=-1), dict(B=-1), dict(D=0)])
def test_layer_decode_bad_shape(lib, kw):
    assert layer_decode(lib, **kw) == ERR_SHAPE


@pytest.mark.parametrize("kw", [dict(dtype=F32), dict(H=3), dict(H=98), dict(rq=128), dict(r=256, ld=256)])
def test_layer_decode_unsupported(lib, kw):
    assert layer_decode(lib, **kw) == ERR_UNSUPPORTED


def test_layer_decode_checks_before_launch(lib):
    assert layer_decode(lib, lens=FAKE + 4) == ERR_ALIGN
    assert layer_decode(lib, ld=520 + 4) == ERR_ALIGN
    assert layer_decode(lib, ws=None) == ERR_WORKSPACE
    assert layer_decode(lib, B=0) == OK
    assert layer_decode(lib, dtype=4) == ERR_DTYPE


@pytest.mark.parametrize("limit_us", [0, 2000001])
def test_wait_timeout_probe_rejects_limits_out_of_range(lib, limit_us):
    assert lib.mla_debug_wait_timeout(limit_us, None) == ERR_SHAPE


# ----------------------------------------------------------------------------- backward
def bwd_call(lib, **kw):
    a = dict(q=FAKE, c=FAKE, wuk=FAKE, wuv=FAKE, gate=FAKE, dout=FAKE, dq=FAKE, dc=FAKE, dwuk=FAKE, dwuv=FAKE,
             dgate=FAKE, B=2, T=128, H=8, dq_dim=16, dv=16, r=32, dtype=F32, ws=FAKE, ws_bytes=1 << 30)
    a.update(kw)
    return lib.mla_absorbed_attn_bwd(a["q"], a["c"], a["wuk"], a["wuv"], a["gate"], 1.0, a["dout"], a["dq"], a["dc"],
                                     a["dwuk"], a["dwuv"], a["dgate"], a["B"], a["T"], a["H"], a["dq_dim"], a["dv"],
                                     a["r"], a["dtype"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("field", ["q", "c", "wuk", "wuv", "dout", "dq", "dc", "dwuk", "dwuv"])
def test_backward_null_pointer(lib, field):
    assert bwd_call(lib, **{field: None}) == ERR_NULL


@pytest.mark.parametrize("kw", [dict(gate=None), dict(dgate=None)])
def test_backward_gate_and_its_gradient_go_together(lib, kw):
    assert bwd_call(lib, **kw) == ERR_NULL


@pytest.mark.parametrize("field", ["q", "dout", "dc", "dgate", "ws"])
def test_backward_misaligned(lib, field):
    assert bwd_call(lib, **{field: FAKE + 4}) == ERR_ALIGN


@pytest.mark.parametrize("kw", [dict(r=65), dict(dq_dim=128), dict(dv=65), dict(r=512, dq_dim=128, dv=128),
                                dict(B=1, T=4_194_241)])
def test_backward_unsupported(lib, kw):
    assert bwd_call(lib, **kw) == ERR_UNSUPPORTED


@pytest.mark.parametrize("kw", [dict(B=-1), dict(H=0), dict(r=0), dict(B=1 << 20, T=1 << 20)])
def test_backward_bad_shape(lib, kw):
    assert bwd_call(lib, **kw) == ERR_SHAPE


def test_backward_bad_dtype(lib):
    assert bwd_call(lib, dtype=7) == ERR_DTYPE


def test_backward_workspace_checked_before_launch(lib):
    assert bwd_call(lib, ws=None) == ERR_WORKSPACE
    assert bwd_call(lib, ws_bytes=16) == ERR_WORKSPACE
    assert bwd_call(lib, B=0) == OK   # nothing to do


def test_backward_workspace_size(lib):
    assert lib.mla_absorbed_attn_bwd_workspace_size(2, 128, 8, 16, 16, 32, F32) == 2 * 128 * 8 * (2 * 32 + 4) * 4
    assert lib.mla_absorbed_attn_bwd_workspace_size(2, 128, 8, 16, 16, 32, BF16) == 2 * 128 * 8 * (2 * 32 + 4) * 4
    assert lib.mla_absorbed_attn_bwd_workspace_size(2, 128, 8, 16, 16, 32, 7) == 0
    assert lib.mla_absorbed_attn_bwd_workspace_size(2, 128, 8, 16, 16, 65, F32) == 0


# ----------------------------------------------------------------------------- forward with lse, backward given it
def fwd_lse_call(lib, lse=FAKE, **kw):
    a = dict(q=FAKE, c=FAKE, wuk=FAKE, wuv=FAKE, gate=None, out=FAKE, B=1, T=256, H=2, dq=128, dv=128, r=512,
             dtype=BF16, ws=FAKE, ws_bytes=1 << 30)
    a.update(kw)
    return lib.mla_absorbed_attn_fwd_lse(a["q"], a["c"], a["wuk"], a["wuv"], a["gate"], 1.0, a["out"], lse, a["B"],
                                         a["T"], a["H"], a["dq"], a["dv"], a["r"], a["dtype"], a["ws"], a["ws_bytes"],
                                         None)


def bwd_lse_call(lib, out=FAKE, lse=FAKE, **kw):
    a = dict(q=FAKE, c=FAKE, wuk=FAKE, wuv=FAKE, gate=FAKE, dout=FAKE, dq=FAKE, dc=FAKE, dwuk=FAKE, dwuv=FAKE,
             dgate=FAKE, B=1, T=256, H=2, dq_dim=128, dv=128, r=512, dtype=BF16, ws=FAKE, ws_bytes=1 << 40)
    a.update(kw)
    return lib.mla_absorbed_attn_bwd_lse(a["q"], a["c"], a["wuk"], a["wuv"], a["gate"], 1.0, a["dout"], out, lse,
                                         a["dq"], a["dc"], a["dwuk"], a["dwuv"], a["dgate"], a["B"], a["T"], a["H"],
                                         a["dq_dim"], a["dv"], a["r"], a["dtype"], a["ws"], a["ws_bytes"], None)


def test_fwd_lse_refusals(lib):
    assert fwd_lse_call(lib, lse=None) == ERR_NULL
    assert fwd_lse_call(lib, lse=FAKE + 4) == ERR_ALIGN
    # only the r = 512 bf16 kernel writes the statistics
    assert fwd_lse_call(lib, r=32, dq=16, dv=16) == ERR_UNSUPPORTED
    assert fwd_lse_call(lib, dtype=F32, r=32, dq=16, dv=16, ws=None, ws_bytes=0) == ERR_UNSUPPORTED
    assert fwd_lse_call(lib, B=0) == OK


def test_bwd_lse_refusals(lib):
    assert bwd_lse_call(lib, out=None) == ERR_NULL
    assert bwd_lse_call(lib, lse=None) == ERR_NULL
    assert bwd_lse_call(lib, lse=FAKE + 4) == ERR_ALIGN
    assert bwd_lse_call(lib, out=FAKE + 2) == ERR_ALIGN
    assert bwd_lse_call(lib, r=32, dq_dim=16, dv=16, dtype=F32) == ERR_UNSUPPORTED
    assert bwd_lse_call(lib, ws=None) == ERR_WORKSPACE
    assert bwd_lse_call(lib, B=0) == OK
