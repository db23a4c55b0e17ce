"""fp64 CPU oracle of the absorbed, NoPE, causal Gated MLA forward.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The CUDA library never
imports, links or runs anything here, and nothing here imports the CUDA
library.

* ``prefill`` / ``decode`` call the plain C loops in ``mla_oracle.c`` (steps
  2-4 of the page "Gated MLA（矩阵吸收版）", section "完整计算流（四步）").
* ``layer`` holds step 1 (the low-rank latent and query paths) and the output
  projection of step 4, in numpy fp64, used to build full-layer inputs;
  ``layer_forward`` composes them with ``prefill`` into the whole layer.
* ``prefill_backward`` (module ``backward``) takes the chain rule back through
  steps 2-4 in numpy fp64: the gradients of the prefill's inputs; ``prefill_lse``
  gives each row's softmax normaliser (log-sum-exp of the scaled scores).

Parity status of each function is stated in its docstring; the pins live in
``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``mla_oracle.c`` with gcc (-O2, no fast-math, OpenMP) and return the .so path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", src, "-o", tmp, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:  # OpenMP missing: the loops are still correct serially
        cmd = [a for a in cmd if a != "-fopenmp"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + res.stderr)
    os.replace(tmp, out)
    return out


def load_library(path: str):
    """Load an oracle shared library (the default build, or a test's variant of it)."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.mla_oracle_prefill.argtypes = [dp, dp, dp, dp, dp, ctypes.c_double, dp,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_longlong), ctypes.c_longlong]
    lib.mla_oracle_prefill.restype = ctypes.c_int
    lib.mla_oracle_decode.argtypes = [dp, dp, ctypes.c_longlong, ctypes.c_longlong,
                                      ctypes.POINTER(ctypes.c_int), dp, dp, ctypes.c_double, dp,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.mla_oracle_decode.restype = ctypes.c_int
    lib.mla_oracle_num_threads.argtypes = []
    lib.mla_oracle_num_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a, ctype=ctypes.c_double):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


def num_threads() -> int:
    """Threads the oracle's OpenMP regions use on this host."""
    return int(_load().mla_oracle_num_threads())


def prefill(q, c, w_uk, w_uv, gate=None, scale: float = 1.0, rows=None, lib=None) -> np.ndarray:
    """Causal absorbed Gated-MLA prefill in fp64 (steps 2-4 of sec-06).

    q [B,T,H,d_q], c [B,T,r], w_uk [H,d_q,r], w_uv [H,d_v,r], gate [B,T,H*d_v]
    (pre-sigmoid logits) or None.  Returns [B,T,H*d_v], or [len(rows), H*d_v]
    when ``rows`` lists flattened token indices b*T+t.
    Parity: pinned (tests/test_oracle.py).
    """
    q, c, w_uk, w_uv = _f64(q), _f64(c), _f64(w_uk), _f64(w_uv)
    B, T, H, dq = q.shape
    r = c.shape[-1]
    dv = w_uv.shape[1]
    assert c.shape == (B, T, r) and w_uk.shape == (H, dq, r) and w_uv.shape == (H, dv, r)
    g = None if gate is None else _f64(gate).reshape(B, T, H * dv)
    if rows is None:
        out = np.empty((B, T, H * dv), dtype=np.float64)
        rows_arr, n = None, 0
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.size
        out = np.empty((n, H * dv), dtype=np.float64)
    rc = (lib or _load()).mla_oracle_prefill(_ptr(q), _ptr(c), _ptr(w_uk), _ptr(w_uv), _ptr(g), float(scale), _ptr(out),
                                    B, T, H, dq, dv, r, _ptr(rows_arr, ctypes.c_longlong), n)
    if rc != 0:
        raise ValueError(f"oracle prefill rejected its arguments (code {rc})")
    return out


def layer_forward(x, p, H: int, d_q: int, d_v: int, scale: float = 1.0, rows=None) -> np.ndarray:
    """The whole Gated-MLA layer in fp64: x [B,T,D] -> y, for all rows or the flattened rows ``rows``.

    Page "Gated MLA（矩阵吸收版）", section "完整计算流（四步）": step 1 (``layer``:
    c = RMSNorm(x W_kv_down^T), q = RMSNorm(x W_q_down^T) W_q_up^T, g = x W_gate^T), steps
    2-4 (``prefill``), then y = o W_o^T (``layer.output_projection``).  ``p`` holds the
    weights as nn.Linear weights under the keys of ``workloads.draw_layer``: q_down, q_up,
    kv_down, kv_up, gate, o_proj.  Only the requested rows' q, g and o are formed; c is
    formed for every row (each row's attention reads all earlier latents).
    Returns [B,T,D], or [len(rows), D].
    Parity: a composition of pinned parts (``layer``'s functions are pinned in
    tests/test_oracle_layer.py; tests/test_oracle.py checks the composition against
    explicit decompression).
    """
    from . import layer
    x = _f64(x)
    B, T, D = x.shape
    flat = x.reshape(B * T, D)
    sel = np.arange(B * T) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = layer.latent(flat, p["kv_down"]).reshape(B, T, -1)
    q = np.zeros((B * T, H * d_q))
    q[sel] = layer.query(flat[sel], p["q_down"], p["q_up"])
    g = np.zeros((B * T, H * d_v))
    g[sel] = layer.gate_logits(flat[sel], p["gate"])
    w_uk, w_uv = layer.split_kv_up(_f64(p["kv_up"]), H, d_q, d_v)
    o = prefill(q.reshape(B, T, H, d_q), c, w_uk, w_uv, g.reshape(B, T, H * d_v), scale, rows=sel)
    y = layer.output_projection(o, p["o_proj"])
    return y.reshape(B, T, D) if rows is None else y


def prefill_backward(q, c, w_uk, w_uv, gate, scale: float, dout) -> dict:
    """Gradients of sum(dout * prefill(...)) in fp64; see ``oracle.backward``.
    Parity: pinned by finite differences of ``prefill`` (tests/test_oracle_backward.py).
    """
    from .backward import prefill_backward as _bwd
    return _bwd(q, c, w_uk, w_uv, gate, scale, dout)


def prefill_lse(q, c, w_uk, scale: float = 1.0) -> np.ndarray:
    """Each row's log-sum-exp of the scaled causal scores, [B,H,T] fp64; see ``oracle.backward.prefill_lse``.
    Parity: pinned by closed forms and by rebuilding ``prefill``'s output (tests/test_oracle_backward.py).
    """
    from .backward import prefill_lse as _lse
    return _lse(q, c, w_uk, scale)


def decode(q_abs, c_cache, lens, w_uv, gate=None, scale: float = 1.0) -> np.ndarray:
    """Cached-latent decode in fp64: query b attends to cache rows [0, lens[b]).

    q_abs [B,H,r] (already absorbed), c_cache [B,max_len,r], lens int [B],
    w_uv [H,d_v,r], gate [B,H*d_v] or None.  Returns [B,H*d_v].
    Parity: pinned against prefill (decode of token t == prefill row t).
    """
    q_abs, c_cache, w_uv = _f64(q_abs), _f64(c_cache), _f64(w_uv)
    B, H, r = q_abs.shape
    max_len = c_cache.shape[1]
    dv = w_uv.shape[1]
    assert c_cache.shape == (B, max_len, r) and w_uv.shape == (H, dv, r)
    lens_arr = np.ascontiguousarray(lens, dtype=np.int32)
    g = None if gate is None else _f64(gate).reshape(B, H * dv)
    out = np.empty((B, H * dv), dtype=np.float64)
    rc = _load().mla_oracle_decode(_ptr(q_abs), _ptr(c_cache), r, max_len, _ptr(lens_arr, ctypes.c_int),
                                   _ptr(w_uv), _ptr(g), float(scale), _ptr(out), B, H, dv, r)
    if rc != 0:
        raise ValueError(f"oracle decode rejected its arguments (code {rc})")
    return out


if __name__ == "__main__":  # `python -m oracle` builds the library
    print(build(force="--force" in sys.argv))
