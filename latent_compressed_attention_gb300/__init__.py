"""GB300-native (sm_103a) absorbed, NoPE, causal Gated MLA forward.

A thin ctypes binding over the C ABI in ``include/mla.h`` (``libmla_gb300.so``,
built in-tree by ``_build.build()``).  The binding only marshals arguments:
PyTorch provides device memory and the current stream, and every step of the
computation runs in the library's CUDA kernels.  There is no CPU fallback: if
the library is missing or a call fails, an exception is raised.

Entry points (same names as the C functions):
    mla_absorbed_attn_fwd(q, c, w_uk, w_uv, gate=None, scale=1.0, out=None, workspace=None)
    mla_absorbed_attn_fwd_workspace_size(B, T, H, d_q, d_v, r, dtype)
    mla_latent_decode(q_abs, c_cache, lens, w_uv, gate=None, scale=1.0, out=None, workspace=None)
    mla_latent_decode_workspace_size(B, H, r, max_len)
    mla_latent_decode_fp8(q_abs, c8_cache, lens, w_uv, cache_scale, gate=None, scale=1.0, out=None, workspace=None)
    mla_quantize_latent_fp8(c, cache_scale, out=None)
    mla_get_device_error(stream=None)
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB_PATH, build

__all__ = ["MLAError", "build", "library", "library_path", "mla_absorbed_attn_fwd",
           "mla_absorbed_attn_fwd_workspace_size", "mla_latent_decode",
           "mla_latent_decode_workspace_size", "mla_latent_decode_noalloc", "mla_latent_decode_fp8",
           "mla_quantize_latent_fp8", "mla_get_device_error",
           "mla_status_string", "mla_version", "mla_kernel_launches", "mla_debug_wait_timeout",
           "mla_absorbed_attn_bwd", "mla_gated_layer_fwd", "mla_gated_layer_workspace_size",
           "mla_gated_layer_decode", "layer_workspace_views", "DTYPE_BF16", "DTYPE_F32"]

DTYPE_BF16 = 0
DTYPE_F32 = 1

_lock = threading.Lock()
_lib = None


class MLAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({mla_status_string(status)})")


def library_path() -> str:
    return LIB_PATH


def library():
    """The loaded C library (ctypes.CDLL) with argument types declared."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library {LIB_PATH} is not built; run "
                                   "`python -c 'import __graft_entry__ as g; g.build()'` first")
            lib = ctypes.CDLL(LIB_PATH)
            vp, i, f, ll, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong, ctypes.c_size_t
            lib.mla_absorbed_attn_fwd.argtypes = [vp, vp, vp, vp, vp, f, vp, i, i, i, i, i, i, i, vp, sz, vp]
            lib.mla_absorbed_attn_fwd.restype = i
            lib.mla_absorbed_attn_fwd_lse.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, i, i, i, i, i, i, i, vp, sz, vp]
            lib.mla_absorbed_attn_fwd_lse.restype = i
            lib.mla_absorbed_attn_fwd_workspace_size.argtypes = [i] * 7
            lib.mla_absorbed_attn_fwd_workspace_size.restype = sz
            lib.mla_latent_decode_workspace_size.argtypes = [i, i, i, i]
            lib.mla_latent_decode_workspace_size.restype = sz
            lib.mla_latent_decode.argtypes = [vp, vp, ll, vp, i, vp, vp, f, vp, i, i, i, i, i, vp, sz, vp]
            lib.mla_latent_decode.restype = i
            lib.mla_latent_decode_fp8_workspace_size.argtypes = [i, i, i, i]
            lib.mla_latent_decode_fp8_workspace_size.restype = sz
            lib.mla_latent_decode_fp8.argtypes = [vp, vp, ll, vp, i, f, vp, vp, f, vp, i, i, i, i, vp, sz, vp]
            lib.mla_latent_decode_fp8.restype = i
            lib.mla_quantize_latent_fp8.argtypes = [vp, ll, vp, ll, ll, i, f, vp]
            lib.mla_quantize_latent_fp8.restype = i
            lib.mla_latent_decode_noalloc.argtypes = [vp, vp, ll, vp, i, vp, vp, f, vp, i, i, i, i, i, vp]
            lib.mla_latent_decode_noalloc.restype = i
            lib.mla_gated_layer_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i]
            lib.mla_gated_layer_workspace_size.restype = sz
            lib.mla_gated_layer_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, f, vp] + [i] * 9 + [vp, sz, vp]
            lib.mla_gated_layer_fwd.restype = i
            lib.mla_gated_layer_decode_workspace_size.argtypes = [i] * 9
            lib.mla_gated_layer_decode_workspace_size.restype = sz
            lib.mla_gated_layer_decode.argtypes = [vp] * 7 + [f, vp, vp, ll, vp] + [i] * 9 + [vp, sz, vp]
            lib.mla_gated_layer_decode.restype = i
            lib.mla_absorbed_attn_bwd_workspace_size.argtypes = [i] * 7
            lib.mla_absorbed_attn_bwd_workspace_size.restype = sz
            lib.mla_absorbed_attn_bwd.argtypes = [vp] * 5 + [f] + [vp] * 6 + [i] * 7 + [vp, sz, vp]
            lib.mla_absorbed_attn_bwd.restype = i
            lib.mla_absorbed_attn_bwd_lse.argtypes = [vp] * 5 + [f] + [vp] * 8 + [i] * 7 + [vp, sz, vp]
            lib.mla_absorbed_attn_bwd_lse.restype = i
            lib.mla_debug_wait_timeout.argtypes = [ctypes.c_uint, vp]
            lib.mla_debug_wait_timeout.restype = i
            lib.mla_get_device_error.argtypes = [vp]
            lib.mla_get_device_error.restype = i
            lib.mla_status_string.argtypes = [i]
            lib.mla_status_string.restype = ctypes.c_char_p
            lib.mla_version.argtypes = []
            lib.mla_version.restype = i
            lib.mla_kernel_launches.argtypes = []
            lib.mla_kernel_launches.restype = ctypes.c_ulonglong
            _lib = lib
    return _lib


def mla_status_string(status: int) -> str:
    try:
        return library().mla_status_string(int(status)).decode()
    except RuntimeError:
        return "library not loaded"


def mla_version() -> int:
    return int(library().mla_version())


def mla_kernel_launches() -> int:
    """Kernels the library has launched in this process (a diagnostic counter)."""
    return int(library().mla_kernel_launches())


# ----------------------------------------------------------------------------- torch marshalling
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}; expected bfloat16 or float32")


def _check(t, name, dtype, device, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU fallback exists)")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _stream_ptr(stream, device):
    torch = _torch()
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def mla_absorbed_attn_fwd_workspace_size(B: int, T: int, H: int, d_q: int, d_v: int, r: int, dtype) -> int:
    """Bytes of workspace mla_absorbed_attn_fwd needs (0 when none)."""
    torch = _torch()
    code = dtype if isinstance(dtype, int) else (DTYPE_BF16 if dtype == torch.bfloat16 else
                                                 DTYPE_F32 if dtype == torch.float32 else -1)
    return int(library().mla_absorbed_attn_fwd_workspace_size(B, T, H, d_q, d_v, r, code))


def mla_absorbed_attn_fwd(q, c, w_uk, w_uv, gate=None, scale: float = 1.0, out=None, workspace=None, stream=None,
                          return_lse: bool = False):
    """Causal absorbed Gated-MLA prefill; returns out [B,T,H*d_v] (allocated if not given), or (out, lse) with
    return_lse (lse [B,H,T] fp32: each row's log-sum-exp of the scaled scores, for mla_absorbed_attn_bwd; bf16
    with r = 512, d_q = d_v = 128 only).

    q [B,T,H,d_q], c [B,T,r], w_uk [H,d_q,r], w_uv [H,d_v,r], gate [B,T,H*d_v]
    (pre-sigmoid logits) or None; all CUDA, contiguous, one dtype (bf16/fp32).
    A workspace (uint8 CUDA tensor) is allocated when the call needs one and none is given.
    """
    torch = _torch()
    B, T, H, d_q = q.shape
    r = c.shape[-1]
    d_v = w_uv.shape[1]
    dev, dt = q.device, q.dtype
    _check(q, "q", dt, dev)
    _check(c, "c", dt, dev, (B, T, r))
    _check(w_uk, "w_uk", dt, dev, (H, d_q, r))
    _check(w_uv, "w_uv", dt, dev, (H, d_v, r))
    if gate is not None:
        _check(gate, "gate", dt, dev, (B, T, H * d_v))
    if out is None:
        out = torch.empty((B, T, H * d_v), dtype=dt, device=dev)
    _check(out, "out", dt, dev, (B, T, H * d_v))
    lib = library()
    need = int(lib.mla_absorbed_attn_fwd_workspace_size(B, T, H, d_q, d_v, r, _dtype_code(q)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if return_lse:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
        rc = lib.mla_absorbed_attn_fwd_lse(q.data_ptr(), c.data_ptr(), w_uk.data_ptr(), w_uv.data_ptr(),
                                           None if gate is None else gate.data_ptr(), float(scale), out.data_ptr(),
                                           lse.data_ptr(), B, T, H, d_q, d_v, r, _dtype_code(q), ws_ptr, ws_bytes,
                                           _stream_ptr(stream, dev))
        if rc != 0:
            raise MLAError(rc, "mla_absorbed_attn_fwd_lse")
        return out, lse
    rc = lib.mla_absorbed_attn_fwd(q.data_ptr(), c.data_ptr(), w_uk.data_ptr(), w_uv.data_ptr(),
                                   None if gate is None else gate.data_ptr(), float(scale), out.data_ptr(),
                                   B, T, H, d_q, d_v, r, _dtype_code(q), ws_ptr, ws_bytes, _stream_ptr(stream, dev))
    if rc != 0:
        raise MLAError(rc, "mla_absorbed_attn_fwd")
    return out


def mla_absorbed_attn_bwd(q, c, w_uk, w_uv, gate, scale: float, dout, workspace=None, stream=None, out=None,
                          lse=None) -> dict:
    """Gradients of sum(dout * mla_absorbed_attn_fwd(q, c, w_uk, w_uv, gate, scale)): a dict with dq, dc, dw_uk,
    dw_uv and dgate (None without a gate), allocated here as fp32.  Inputs fp32 or bf16 with r, d_q, d_v <= 64,
    or bf16 with r = 512, d_q = d_v = 128 (tensor cores; the workspace is O(B H T^2)).  Given the forward's
    (out, lse) from mla_absorbed_attn_fwd(..., return_lse=True) (r = 512 only), the forward is not run again."""
    saved_out = out
    torch = _torch()
    B, T, H, d_q = q.shape
    r = c.shape[-1]
    d_v = w_uv.shape[1]
    dev, dt = q.device, q.dtype
    _check(q, "q", dt, dev)
    _check(c, "c", dt, dev, (B, T, r))
    _check(w_uk, "w_uk", dt, dev, (H, d_q, r))
    _check(w_uv, "w_uv", dt, dev, (H, d_v, r))
    _check(dout, "dout", dt, dev, (B, T, H * d_v))
    if gate is not None:
        _check(gate, "gate", dt, dev, (B, T, H * d_v))
    lib = library()
    code = _dtype_code(q)
    f32 = lambda t: torch.empty(t.shape, dtype=torch.float32, device=dev)  # noqa: E731
    out_grads = dict(dq=f32(q), dc=f32(c), dw_uk=f32(w_uk), dw_uv=f32(w_uv), dgate=None if gate is None else f32(gate))
    need = int(lib.mla_absorbed_attn_bwd_workspace_size(B, T, H, d_q, d_v, r, code))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    grads = out_grads
    if saved_out is not None or lse is not None:
        if saved_out is None or lse is None:
            raise ValueError("out and lse come together (both from mla_absorbed_attn_fwd(..., return_lse=True))")
        _check(saved_out, "out", dt, dev, (B, T, H * d_v))
        if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, T) or lse.device != dev or not lse.is_contiguous():
            raise ValueError("lse: float32 [B, H, T], contiguous, on the inputs' device")
        rc = lib.mla_absorbed_attn_bwd_lse(q.data_ptr(), c.data_ptr(), w_uk.data_ptr(), w_uv.data_ptr(), ptr(gate),
                                           float(scale), dout.data_ptr(), saved_out.data_ptr(), lse.data_ptr(),
                                           grads["dq"].data_ptr(), grads["dc"].data_ptr(), grads["dw_uk"].data_ptr(),
                                           grads["dw_uv"].data_ptr(), ptr(grads["dgate"]), B, T, H, d_q, d_v, r, code,
                                           ws_ptr, ws_bytes, _stream_ptr(stream, dev))
        if rc != 0:
            raise MLAError(rc, "mla_absorbed_attn_bwd_lse")
        return grads
    rc = lib.mla_absorbed_attn_bwd(q.data_ptr(), c.data_ptr(), w_uk.data_ptr(), w_uv.data_ptr(), ptr(gate),
                                   float(scale), dout.data_ptr(), grads["dq"].data_ptr(), grads["dc"].data_ptr(),
                                   grads["dw_uk"].data_ptr(), grads["dw_uv"].data_ptr(), ptr(grads["dgate"]),
                                   B, T, H, d_q, d_v, r, code, ws_ptr, ws_bytes, _stream_ptr(stream, dev))
    if rc != 0:
        raise MLAError(rc, "mla_absorbed_attn_bwd")
    return grads


def mla_gated_layer_workspace_size(B: int, T: int, D: int, H: int, d_q: int, d_v: int, r: int, r_q: int,
                                   dtype) -> int:
    """Workspace bytes of mla_gated_layer_fwd (0: shape or dtype unsupported); dtype a torch dtype."""
    torch = _torch()
    code = DTYPE_BF16 if dtype == torch.bfloat16 else DTYPE_F32 if dtype == torch.float32 else -1
    return int(library().mla_gated_layer_workspace_size(B, T, D, H, d_q, d_v, r, r_q, code))


def layer_workspace_views(workspace, B: int, T: int, H: int, d_q: int, d_v: int, r: int, dtype):
    """The intermediate results mla_gated_layer_fwd leaves in its workspace: q, c, g, o."""
    torch = _torch()
    es = torch.tensor([], dtype=dtype).element_size()
    M = B * T
    align = lambda n: (n + 255) // 256 * 256  # noqa: E731
    offs, sizes = [], [M * H * d_q, M * r, M * H * d_v, M * H * d_v]
    o = 0
    for n in sizes:
        offs.append(o)
        o += align(n * es)
    flat = workspace.view(torch.uint8)
    return tuple(flat[off:off + n * es].view(dtype) for off, n in zip(offs, sizes))


def mla_gated_layer_fwd(x, w_q_down, w_q_up, w_kv_down, w_kv_up, w_gate, w_o, H: int, d_q: int, d_v: int,
                        scale: float = 1.0, out=None, workspace=None, stream=None):
    """The whole Gated-MLA layer: x [B,T,D] -> y [B,T,D] (allocated if not given).

    Weights are nn.Linear weights [out, in]: w_q_down [r_q,D], w_q_up [H*d_q,r_q], w_kv_down [r,D],
    w_kv_up [H*(d_q+d_v),r] (W_UK rows, then W_UV rows), w_gate [H*d_v,D], w_o [D,H*d_v].
    A workspace (uint8 CUDA tensor) is allocated when not given; after the call it holds q, c, g
    and the gated attention output (``layer_workspace_views``).
    """
    torch = _torch()
    B, T, D = x.shape
    r_q, r = w_q_down.shape[0], w_kv_down.shape[0]
    dev, dt = x.device, x.dtype
    _check(x, "x", dt, dev)
    _check(w_q_down, "w_q_down", dt, dev, (r_q, D))
    _check(w_q_up, "w_q_up", dt, dev, (H * d_q, r_q))
    _check(w_kv_down, "w_kv_down", dt, dev, (r, D))
    _check(w_kv_up, "w_kv_up", dt, dev, (H * (d_q + d_v), r))
    _check(w_gate, "w_gate", dt, dev, (H * d_v, D))
    _check(w_o, "w_o", dt, dev, (D, H * d_v))
    if out is None:
        out = torch.empty((B, T, D), dtype=dt, device=dev)
    _check(out, "out", dt, dev, (B, T, D))
    lib = library()
    code = _dtype_code(x)
    need = int(lib.mla_gated_layer_workspace_size(B, T, D, H, d_q, d_v, r, r_q, code))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.mla_gated_layer_fwd(x.data_ptr(), w_q_down.data_ptr(), w_q_up.data_ptr(), w_kv_down.data_ptr(),
                                 w_kv_up.data_ptr(), w_gate.data_ptr(), w_o.data_ptr(), float(scale),
                                 out.data_ptr(), B, T, D, H, d_q, d_v, r, r_q, code, ws_ptr, ws_bytes,
                                 _stream_ptr(stream, dev))
    if rc != 0:
        raise MLAError(rc, "mla_gated_layer_fwd")
    return out


def mla_gated_layer_decode(x, w_q_down, w_q_up, w_kv_down, w_kv_up, w_gate, w_o, c_cache, lens, H: int, d_q: int,
                           d_v: int, scale: float = 1.0, out=None, workspace=None, stream=None):
    """One decode step of the whole layer: x [B,D] (the new tokens) -> y [B,D].

    Appends each token's latent to c_cache [B,max_len,r] (unit inner stride) at row lens[b]
    (int32 [B] on the device, read only: advance it after the step), then attends to rows
    [0, lens[b]].  Weights as in ``mla_gated_layer_fwd``.  bf16 only.
    """
    torch = _torch()
    B, D = x.shape
    r_q, r = w_q_down.shape[0], w_kv_down.shape[0]
    dev, dt = x.device, x.dtype
    _check(x, "x", dt, dev)
    for name, t, shape in (("w_q_down", w_q_down, (r_q, D)), ("w_q_up", w_q_up, (H * d_q, r_q)),
                           ("w_kv_down", w_kv_down, (r, D)), ("w_kv_up", w_kv_up, (H * (d_q + d_v), r)),
                           ("w_gate", w_gate, (H * d_v, D)), ("w_o", w_o, (D, H * d_v))):
        _check(t, name, dt, dev, shape)
    max_len = c_cache.shape[1]
    if c_cache.dtype != dt or c_cache.device != dev or c_cache.dim() != 3 or c_cache.shape[0] != B \
            or c_cache.shape[2] != r or c_cache.stride(2) != 1 or c_cache.stride(0) != max_len * c_cache.stride(1):
        raise ValueError("c_cache must be [B,max_len,r] with unit inner stride and batch stride max_len*row_stride")
    _check(lens, "lens", torch.int32, dev, (B,))
    if out is None:
        out = torch.empty((B, D), dtype=dt, device=dev)
    _check(out, "out", dt, dev, (B, D))
    lib = library()
    code = _dtype_code(x)
    need = int(lib.mla_gated_layer_decode_workspace_size(B, D, H, d_q, d_v, r, r_q, max_len, code))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.mla_gated_layer_decode(x.data_ptr(), w_q_down.data_ptr(), w_q_up.data_ptr(), w_kv_down.data_ptr(),
                                    w_kv_up.data_ptr(), w_gate.data_ptr(), w_o.data_ptr(), float(scale),
                                    out.data_ptr(), c_cache.data_ptr(), c_cache.stride(1), lens.data_ptr(), max_len,
                                    B, D, H, d_q, d_v, r, r_q, code, ws_ptr, ws_bytes, _stream_ptr(stream, dev))
    if rc != 0:
        raise MLAError(rc, "mla_gated_layer_decode")
    return out


def mla_latent_decode_workspace_size(B: int, H: int, r: int, max_len: int) -> int:
    return int(library().mla_latent_decode_workspace_size(B, H, r, max_len))


def mla_latent_decode(q_abs, c_cache, lens, w_uv, gate=None, scale: float = 1.0, out=None, workspace=None,
                      stream=None):
    """One decode step over the cached latent; returns out [B,H*d_v].

    q_abs [B,H,r], c_cache [B,max_len,r] (or a row-strided view with unit
    inner stride), lens int32 [B] on the device, w_uv [H,d_v,r], gate
    [B,H*d_v] or None.  A workspace (uint8 CUDA tensor) is allocated when not given.
    """
    torch = _torch()
    B, H, r = q_abs.shape
    max_len = c_cache.shape[1]
    d_v = w_uv.shape[1]
    dev, dt = q_abs.device, q_abs.dtype
    _check(q_abs, "q_abs", dt, dev)
    if c_cache.dtype != dt or c_cache.device != dev or c_cache.dim() != 3 or c_cache.shape[0] != B \
            or c_cache.shape[2] != r or c_cache.stride(2) != 1 or c_cache.stride(0) != max_len * c_cache.stride(1):
        raise ValueError("c_cache must be [B,max_len,r] with unit inner stride and batch stride max_len*row_stride")
    ld_cache = c_cache.stride(1)
    _check(lens, "lens", torch.int32, dev, (B,))
    _check(w_uv, "w_uv", dt, dev, (H, d_v, r))
    if gate is not None:
        _check(gate, "gate", dt, dev, (B, H * d_v))
    if out is None:
        out = torch.empty((B, H * d_v), dtype=dt, device=dev)
    _check(out, "out", dt, dev, (B, H * d_v))
    lib = library()
    need = int(lib.mla_latent_decode_workspace_size(B, H, r, max_len))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.mla_latent_decode(q_abs.data_ptr(), c_cache.data_ptr(), ld_cache, lens.data_ptr(), max_len,
                               w_uv.data_ptr(), None if gate is None else gate.data_ptr(), float(scale),
                               out.data_ptr(), B, H, d_v, r, _dtype_code(q_abs), ws_ptr, ws_bytes,
                               _stream_ptr(stream, dev))
    if rc != 0:
        raise MLAError(rc, "mla_latent_decode")
    return out


def _cache_layout(c_cache, B, r):
    if c_cache.dim() != 3 or c_cache.shape[0] != B or c_cache.shape[2] != r or c_cache.stride(2) != 1 \
            or c_cache.stride(0) != c_cache.shape[1] * c_cache.stride(1):
        raise ValueError("cache must be [B,max_len,r] with unit inner stride and batch stride max_len*row_stride")
    return c_cache.shape[1], c_cache.stride(1)


def mla_latent_decode_fp8(q_abs, c8_cache, lens, w_uv, cache_scale: float, gate=None, scale: float = 1.0, out=None,
                          workspace=None, stream=None):
    """Decode over an e4m3 latent cache; returns out [B,H*d_v] (bf16).

    c8_cache: uint8 [B,max_len,r] (or a row-strided view, row stride a multiple of 16 bytes) holding
    e4m3(c / cache_scale), e.g. from mla_quantize_latent_fp8; q_abs [B,H,r], w_uv [H,d_v,r] and gate
    [B,H*d_v] (or None) bf16; lens int32 [B].  A workspace is allocated when not given.
    """
    torch = _torch()
    B, H, r = q_abs.shape
    d_v = w_uv.shape[1]
    dev = q_abs.device
    _check(q_abs, "q_abs", torch.bfloat16, dev)
    if c8_cache.dtype != torch.uint8 or c8_cache.device != dev:
        raise TypeError("c8_cache must be a uint8 CUDA tensor on the query's device")
    max_len, ld = _cache_layout(c8_cache, B, r)
    _check(lens, "lens", torch.int32, dev, (B,))
    _check(w_uv, "w_uv", torch.bfloat16, dev, (H, d_v, r))
    if gate is not None:
        _check(gate, "gate", torch.bfloat16, dev, (B, H * d_v))
    if out is None:
        out = torch.empty((B, H * d_v), dtype=torch.bfloat16, device=dev)
    _check(out, "out", torch.bfloat16, dev, (B, H * d_v))
    lib = library()
    need = int(lib.mla_latent_decode_fp8_workspace_size(B, H, r, max_len))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.mla_latent_decode_fp8(q_abs.data_ptr(), c8_cache.data_ptr(), ld, lens.data_ptr(), max_len,
                                   float(cache_scale), w_uv.data_ptr(), None if gate is None else gate.data_ptr(),
                                   float(scale), out.data_ptr(), B, H, d_v, r, ws_ptr, ws_bytes,
                                   _stream_ptr(stream, dev))
    if rc != 0:
        raise MLAError(rc, "mla_latent_decode_fp8")
    return out


def mla_quantize_latent_fp8(c, cache_scale: float, out=None, stream=None):
    """e4m3 bytes of c / cache_scale: c bf16 [..., r] (rows contiguous) -> uint8 [..., r]."""
    torch = _torch()
    if c.dtype != torch.bfloat16 or not c.is_cuda or not c.is_contiguous():
        raise ValueError("c must be a contiguous bf16 CUDA tensor")
    r = c.shape[-1]
    rows = c.numel() // max(r, 1)
    if out is None:
        out = torch.empty(c.shape, dtype=torch.uint8, device=c.device)
    if out.dtype != torch.uint8 or tuple(out.shape) != tuple(c.shape) or not out.is_contiguous():
        raise ValueError("out must be a contiguous uint8 tensor of c's shape")
    rc = library().mla_quantize_latent_fp8(c.data_ptr(), r, out.data_ptr(), r, rows, r, float(cache_scale),
                                           _stream_ptr(stream, c.device))
    if rc != 0:
        raise MLAError(rc, "mla_quantize_latent_fp8")
    return out


def mla_latent_decode_noalloc(q_abs, c_cache, lens, w_uv, gate=None, scale: float = 1.0, out=None, stream=None):
    """mla_latent_decode without a workspace, for callers that cannot allocate device memory.

    The library keeps the partial results in its own 48 MiB device scratch
    array (reserved when the library loads); sizes that need more raise
    MLAError(MLA_ERR_WORKSPACE).  Calls that overlap on the GPU share that
    array and race; ordered calls (e.g. on one stream) are safe.  The first
    call on a device resolves the array's address there.  ``out`` is
    allocated with torch only when the caller does not pass it.
    """
    torch = _torch()
    B, H, r = q_abs.shape
    max_len = c_cache.shape[1]
    d_v = w_uv.shape[1]
    dev, dt = q_abs.device, q_abs.dtype
    _check(q_abs, "q_abs", dt, dev)
    if c_cache.dtype != dt or c_cache.device != dev or c_cache.dim() != 3 or c_cache.shape[0] != B \
            or c_cache.shape[2] != r or c_cache.stride(2) != 1 or c_cache.stride(0) != max_len * c_cache.stride(1):
        raise ValueError("c_cache must be [B,max_len,r] with unit inner stride and batch stride max_len*row_stride")
    _check(lens, "lens", torch.int32, dev, (B,))
    _check(w_uv, "w_uv", dt, dev, (H, d_v, r))
    if gate is not None:
        _check(gate, "gate", dt, dev, (B, H * d_v))
    if out is None:
        out = torch.empty((B, H * d_v), dtype=dt, device=dev)
    _check(out, "out", dt, dev, (B, H * d_v))
    rc = library().mla_latent_decode_noalloc(q_abs.data_ptr(), c_cache.data_ptr(), c_cache.stride(1),
                                             lens.data_ptr(), max_len, w_uv.data_ptr(),
                                             None if gate is None else gate.data_ptr(), float(scale),
                                             out.data_ptr(), B, H, d_v, r, _dtype_code(q_abs),
                                             _stream_ptr(stream, dev))
    if rc != 0:
        raise MLAError(rc, "mla_latent_decode_noalloc")
    return out


def mla_debug_wait_timeout(limit_us: int = 1000, stream=None, device=None) -> None:
    """Make one device-side bounded wait give up after `limit_us` (a barrier nothing completes); the device
    error word then holds MLA_ERR_DEVICE_TIMEOUT (read it with mla_get_device_error)."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    rc = library().mla_debug_wait_timeout(int(limit_us), _stream_ptr(stream, dev))
    if rc != 0:
        raise MLAError(rc, "mla_debug_wait_timeout")


def mla_get_device_error(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    return int(library().mla_get_device_error(_stream_ptr(stream, dev)))
