"""The host-side e4m3 codec that builds fp8 latent caches for the tests.

The fp8 decode's parity tests quantise the cache on the host (workloads.quantize_e4m3) and give the same bytes
to the GPU and, dequantised, to the fp64 oracle; the GPU quantiser is checked bit for bit against this codec.
So the codec is pinned here against the e4m3 format's definition (OCP 8-bit floating point: 1 sign bit, 4
exponent bits with bias 7, 3 mantissa bits, no infinities, largest finite 448): every code's value, round
trips, ties to even, subnormals and saturation.
"""
import numpy as np

from latent_compressed_attention_gb300 import workloads as W


def test_every_code_decodes_to_its_definition():
    for code in range(256):
        if (code & 0x7F) == 0x7F:
            continue   # NaN patterns
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        want = (m / 8.0) * 2.0**-6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        assert W.decode_e4m3(np.array([code]))[0] == (-want if s else want)


def test_round_trip_and_ordering():
    codes = np.array([c for c in range(128) if c != 0x7F], np.uint8)
    vals = W.decode_e4m3(codes)
    assert np.all(np.diff(vals) > 0)                      # monotone in the code for positive values
    assert np.array_equal(W.encode_e4m3(vals), codes)
    assert np.array_equal(W.encode_e4m3(-vals[1:]), codes[1:] | 0x80)
    assert vals.max() == 448.0 and vals[1] == 2.0**-9 and vals[8] == 2.0**-6


def test_ties_to_even_subnormals_and_saturation():
    got = W.decode_e4m3(W.encode_e4m3([1.0625, 1.1875, 2.0**-10, 3 * 2.0**-10, 2.0**-6 + 2.0**-10, 464.0, 1e6, -1e6,
                                       0.3, -0.3]))
    assert list(got[:5]) == [1.0, 1.25, 0.0, 2 * 2.0**-9, 2.0**-6]   # halfway cases go to the even neighbour
    assert list(got[5:8]) == [448.0, 448.0, -448.0]                   # saturating, no infinities
    assert got[8] == 0.3125 and got[9] == -0.3125                     # 0.3 between 0.28125 and 0.3125


def test_nearest_value_brute_force():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(4000) * np.exp2(rng.integers(-12, 9, 4000))
    grid = W.decode_e4m3(np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8))
    got = W.decode_e4m3(W.encode_e4m3(x))
    for xi, gi in zip(x, got):
        d = np.abs(grid - np.clip(xi, -448, 448))
        assert abs(gi - np.clip(xi, -448, 448)) == d.min()


def test_quantize_rounds_the_fp32_product_first():
    c = W.round_bf16(np.array([1.0, 3.3, -0.7, 21.5]))
    inv = np.float32(1.0) / np.float32(0.0625)
    assert np.array_equal(W.quantize_e4m3(c, inv), W.encode_e4m3((c.astype(np.float32) * inv).astype(np.float64)))
