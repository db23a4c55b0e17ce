"""The oracle's pins must catch plausible slips.

Each case plants one mistake in a private copy of oracle/mla_oracle.c (on the
CPU, in a temporary directory), builds it, and checks that at least one pin of
tests/test_oracle.py (absorbed == decompressed, softmax rows, T = 1 closed form,
causality) rejects the planted variant.
"""
import os

import numpy as np
import pytest

import oracle
from tests.test_oracle import attention_matrix_via_one_hot_latent, decompressed, rand_case, rel_err

SRC = os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.c")

MUTATIONS = {
    "transposed_w_uk": ("w_uk_h[(size_t)d * r + j]", "w_uk_h[(size_t)j * dq + d]"),
    "transposed_w_uv": ("w_uv_h[(size_t)v * r + j]", "w_uv_h[(size_t)j * dv + v]"),
    "dropped_scale": ("s[u] = scale * acc;", "s[u] = acc;"),
    "mask_excludes_self": ("r, t + 1, w_uv", "r, (t > 0 ? t : 1), w_uv"),
    "gate_sign": ("exp(-g_row[v])", "exp(g_row[v])"),
    "no_normalisation": ("s[u] /= z;", "s[u] /= 1.0;"),
    "latent_not_weighted": ("o_lat[j] += s[u] * cu[j];", "o_lat[j] += cu[j] / n_keys;"),
    "wrong_head_slice": ("out + (size_t)i * H * dv + (size_t)h * dv", "out + (size_t)i * H * dv + (size_t)(H - 1 - h) * dv"),
}


def pins_reject(lib) -> bool:
    rng = np.random.default_rng(1)
    q, c, w_uk, w_uv, g = rand_case(rng, 2, 7, 3, 4, 5, 6)
    got = oracle.prefill(q, c, w_uk, w_uv, g, 0.37, lib=lib)
    if rel_err(got, decompressed(q, c, w_uk, w_uv, g, 0.37)) > 1e-12:
        return True
    q1, c1, wk1, wv1, g1 = rand_case(rng, 2, 1, 2, 3, 3, 4)
    ref = np.einsum("bj,hvj->bhv", c1[:, 0], wv1).reshape(2, 1, 6) * (1 / (1 + np.exp(-g1)))
    if rel_err(oracle.prefill(q1, c1, wk1, wv1, g1, 1.0, lib=lib), ref) > 1e-13:
        return True
    return False


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistake(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = tmp_path / "mla_oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.load_library(oracle.build(force=True, src=str(mutated), out=str(tmp_path / "libmut.so")))
    assert pins_reject(lib), f"planted mistake {name} passed the pins"


def test_unmutated_copy_passes(tmp_path):
    copy = tmp_path / "mla_oracle_copy.c"
    copy.write_text(open(SRC).read())
    lib = oracle.load_library(oracle.build(force=True, src=str(copy), out=str(tmp_path / "libcopy.so")))
    assert not pins_reject(lib)
