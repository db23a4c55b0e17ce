"""Seeded synthetic workloads for the absorbed Gated-MLA forward.

This module only draws random numbers and rounds them to the kernels' input
precision.  It holds none of the method's arithmetic, so the tests (which feed
the same draws to the fp64 oracle) and the benchmark (which feeds them to the
CUDA library) share nothing but the inputs.

Sizes come from the course notes' "K3 toy 尺寸" table (page "K3 混合架构":
toy D=256, H=8, head dim 16, kv_lora_rank 32, q_lora_rank 64; real K3
D=7168, H=96, head dim 128, kv_lora_rank 512, q_lora_rank 1536).

Two recipes:

* ``draw_layer``: x ~ N(0,1) and the six projection weights ~ N(0, 0.02^2),
  drawn in the fixed order x, q_down, q_up, kv_down, kv_up, gate, o_proj.
  The oracle's step 1 turns them into q, c and the gate logits.
* ``draw_prefill_direct`` / ``draw_decode``: the hot path's own inputs drawn
  straight from the distributions step 1 produces (used where running step 1
  in fp64 on the host is too slow, and by the benchmark):
    c      rows of N(0,1) rescaled to unit RMS (what RMSNorm with gain 1 emits),
    q      N(0, r_q * 0.02^2)   (unit-RMS vector times N(0,0.02^2) weights),
    g      N(0, D * 0.02^2)     (x ~ N(0,1) times N(0,0.02^2) weights),
    W_UK, W_UV   N(0, 0.02^2)   (the two blocks of kv_up),
    q_abs  N(0, d_q * 0.02^2)   (decode: q ~ N(0,1) times W_UK ~ N(0,0.02^2)).
  Where a config gives q directly as N(0,1) (the toy long-context case) that
  is used instead.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

WEIGHT_STD = 0.02


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "prefill" | "decode"
    dtype: str                # "f32" | "bf16"
    B: int
    H: int
    d_q: int
    d_v: int
    r: int
    T: int = 0                # prefill sequence length
    D: int = 0                # hidden size (gate logits / full layer)
    r_q: int = 0              # q_lora_rank
    scale: float = 1.0
    q_std: float = 1.0        # std of directly drawn q (prefill)
    gate: bool = True
    lens_lo: int = 0          # decode: cache lengths uniform in [lens_lo, lens_hi]
    lens_hi: int = 0
    note: str = ""

    @property
    def max_len(self) -> int:
        return self.lens_hi

    def prefill_flops(self) -> float:
        """Algorithmic FLOPs of one causal prefill: B*H*[2 r T(T+1) + 2 T r (d_q+d_v)].

        QK^T and P.c over the T(T+1)/2 causal (query, key) pairs per head, 2r
        each, plus the W_UK absorb and the W_UV up-projection per row.
        """
        B, T, H, r = self.B, self.T, self.H, self.r
        return float(B) * H * (2.0 * r * T * (T + 1) + 2.0 * T * r * (self.d_q + self.d_v))


TOY_LAYER_F32 = Workload(
    name="toy_layer_f32", kind="prefill", dtype="f32", B=2, T=128, D=256, H=8, d_q=16, d_v=16, r=32, r_q=64,
    scale=1.0, note="toy Gated MLA layer, fp32, inputs through step 1")
TOY_LONG_BF16 = Workload(
    name="toy_long_bf16", kind="prefill", dtype="bf16", B=4, T=2048, D=256, H=8, d_q=16, d_v=16, r=32, r_q=64,
    scale=1.0, q_std=1.0, note="toy dims at long context, q and c given directly")
MID_PREFILL_BF16 = Workload(
    name="mid_prefill_bf16", kind="prefill", dtype="bf16", B=4, T=4096, D=2048, H=16, d_q=128, d_v=128, r=512,
    r_q=1536, scale=1.0 / math.sqrt(128.0), q_std=math.sqrt(1536) * WEIGHT_STD,
    note="mid-size absorbed prefill, scale 1/sqrt(d_q)")
K3_PREFILL_BF16 = Workload(
    name="k3_prefill_bf16", kind="prefill", dtype="bf16", B=1, T=8192, D=7168, H=96, d_q=128, d_v=128, r=512,
    r_q=1536, scale=1.0, q_std=math.sqrt(1536) * WEIGHT_STD, note="K3-size layer prefill")
K3_DECODE_BF16 = Workload(
    name="k3_decode_bf16", kind="decode", dtype="bf16", B=64, H=96, d_q=128, d_v=128, r=512, scale=1.0,
    gate=False, lens_lo=1024, lens_hi=32768, note="cached-latent decode, absorbed q per head")

WORKLOADS = {w.name: w for w in (TOY_LAYER_F32, TOY_LONG_BF16, MID_PREFILL_BF16, K3_PREFILL_BF16, K3_DECODE_BF16)}


# ----------------------------------------------------------------------------- rounding
def round_bf16(a) -> np.ndarray:
    """Nearest bfloat16 value of each element (ties to even), returned as fp64.

    The input is first rounded to fp32 (ties to even); the draws are fp32
    already, so that step is exact for them.  bf16 is the upper half of the
    fp32 bit pattern: add 0x7FFF plus the lowest kept bit, then clear the
    low 16 bits.
    """
    x = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    bits = x.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


# e4m3 (the OCP FP8 format: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinities, the all-ones
# pattern is NaN; largest finite 448, smallest normal 2^-6, subnormals k * 2^-9).
E4M3_MAX = 448.0


def encode_e4m3(a) -> np.ndarray:
    """Bytes of the nearest e4m3 value of each (finite) element, ties to even, saturating at +-448."""
    x = np.asarray(a, dtype=np.float64)
    mag = np.minimum(np.abs(x), E4M3_MAX)
    e = np.floor(np.log2(np.maximum(mag, 2.0**-40)))
    quantum = 2.0 ** (np.maximum(e, -6.0) - 3.0)          # spacing of the binade (2^-9 for subnormals)
    q = np.minimum(np.round(mag / quantum) * quantum, E4M3_MAX)   # np.round: ties to even
    code = np.zeros(x.shape, dtype=np.uint8)
    sub = q < 2.0**-6
    code[sub] = np.round(q[sub] / 2.0**-9).astype(np.uint8)
    qn = q[~sub]
    en = np.floor(np.log2(qn))
    mant = np.round((qn / 2.0**en - 1.0) * 8.0)
    code[~sub] = ((en + 7).astype(np.uint8) << 3) | mant.astype(np.uint8)
    return code | (np.signbit(x) & (q != 0)).astype(np.uint8) << 7


def decode_e4m3(codes) -> np.ndarray:
    """fp64 values of e4m3 bytes (the all-ones exponent and mantissa pattern, NaN, is not produced here)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    e, m = (c >> 3) & 15, c & 7
    v = np.where(e == 0, m * 2.0**-9, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.where(c >> 7, -v, v)


def quantize_e4m3(a, inv_scale: float) -> np.ndarray:
    """The fp8 latent cache's bytes: e4m3(fp32(a) * fp32(inv_scale)), the product rounded to fp32 first."""
    prod = np.asarray(a, np.float32) * np.float32(inv_scale)
    return encode_e4m3(prod.astype(np.float64))


def round_f32(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_to(a, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_bf16(a)
    if dtype == "f32":
        return round_f32(a)
    raise ValueError(dtype)


def _unit_rms_rows(z: np.ndarray) -> np.ndarray:
    return z / np.sqrt(np.mean(np.square(z, dtype=np.float64), axis=-1, keepdims=True))


def _normal(rng, shape, std=1.0) -> np.ndarray:
    """fp32 standard-normal draws times std (held in fp64, exactly)."""
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float64) * std


# ----------------------------------------------------------------------------- recipes
def draw_layer(w: Workload, seed: int = 0, T: int | None = None, B: int | None = None) -> dict:
    """x and the six weights of one Gated-MLA layer, fixed draw order, fp64 holding fp32 draws."""
    rng = np.random.default_rng(seed)
    B = w.B if B is None else B
    T = w.T if T is None else T
    D, H, r, rq = w.D, w.H, w.r, w.r_q
    return dict(
        x=_normal(rng, (B, T, D)),
        q_down=_normal(rng, (rq, D), WEIGHT_STD),
        q_up=_normal(rng, (H * w.d_q, rq), WEIGHT_STD),
        kv_down=_normal(rng, (r, D), WEIGHT_STD),
        kv_up=_normal(rng, (H * (w.d_q + w.d_v), r), WEIGHT_STD),
        gate=_normal(rng, (H * w.d_v, D), WEIGHT_STD),
        o_proj=_normal(rng, (D, H * w.d_v), WEIGHT_STD),
    )


def draw_prefill_direct(w: Workload, seed: int = 0, T: int | None = None, B: int | None = None,
                        wuk_std: float = WEIGHT_STD, H: int | None = None) -> dict:
    """q, c, W_UK, W_UV and gate logits drawn directly (see module docstring), rounded to w.dtype."""
    rng = np.random.default_rng(seed)
    B = w.B if B is None else B
    T = w.T if T is None else T
    H = w.H if H is None else H
    r = w.r
    g_std = math.sqrt(w.D) * WEIGHT_STD if w.D else 1.0
    out = dict(
        q=_normal(rng, (B, T, H, w.d_q), w.q_std),
        c=_unit_rms_rows(_normal(rng, (B, T, r))),
        w_uk=_normal(rng, (H, w.d_q, r), wuk_std),
        w_uv=_normal(rng, (H, w.d_v, r), WEIGHT_STD),
        gate=_normal(rng, (B, T, H * w.d_v), g_std) if w.gate else None,
    )
    return {k: (None if v is None else round_to(v, w.dtype)) for k, v in out.items()}


def draw_lens(w: Workload, seed: int = 0, B: int | None = None) -> np.ndarray:
    """Decode cache lengths, integer-uniform on [lens_lo, lens_hi] inclusive."""
    rng = np.random.default_rng([seed, 1])
    B = w.B if B is None else B
    return rng.integers(w.lens_lo, w.lens_hi, size=B, endpoint=True).astype(np.int32)


def draw_decode(w: Workload, seed: int = 0, B: int | None = None, lens=None, gate: bool | None = None,
                H: int | None = None) -> dict:
    """q_abs [B,H,r], lens [B], W_UV [H,d_v,r], optional gate logits [B,H*d_v].

    The cache itself comes from ``decode_cache_rows`` one sequence at a time.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    lens = draw_lens(w, seed, B) if lens is None else np.asarray(lens, dtype=np.int32)
    rng = np.random.default_rng([seed, 2])
    gate = w.gate if gate is None else gate
    out = dict(
        q_abs=_normal(rng, (B, H, w.r), math.sqrt(w.d_q) * WEIGHT_STD),
        w_uv=_normal(rng, (H, w.d_v, w.r), WEIGHT_STD),
        gate=_normal(rng, (B, H * w.d_v), 1.0) if gate else None,
    )
    out = {k: (None if v is None else round_to(v, w.dtype)) for k, v in out.items()}
    out["lens"] = lens
    return out


def decode_cache_rows(w: Workload, b: int, n_rows: int, seed: int = 0) -> np.ndarray:
    """Latent-cache rows [n_rows, r] of sequence b: N(0,1) rows at unit RMS, rounded.

    Drawn from a generator keyed on (seed, b), so any sequence can be rebuilt
    on its own; the first n rows do not depend on n_rows.
    """
    rng = np.random.default_rng([seed, 3, b])
    return round_to(_unit_rms_rows(_normal(rng, (n_rows, w.r))), w.dtype)
