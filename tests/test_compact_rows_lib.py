"""The library's host encoder of compact 656-byte rows (ess_compact_rows, no
GPU) against the oracle's encoder, byte for byte ("ESS: Latent-Cache Offload",
the 656-byte latent entry)."""
import numpy as np
import pytest

from host_latent_cache_gb300 import ess
from host_latent_cache_gb300 import workloads as W
from oracle import compact_row as X


@pytest.fixture(scope="module")
def lib():
    from host_latent_cache_gb300 import build as B
    B.build()
    return ess.load()


def _rows(rng, n):
    x = (rng.standard_normal((n, 576)) * 0.5).astype(np.float32)
    x[0, :128] = 0.0                                   # an all-zero tile
    x[1, 128:256] *= 1e-4                              # values deep in the subnormal codes
    x[2, :] *= 200.0                                   # large values
    x[3, 256:384] = 0.0
    x[3, 300] = -7.0                                   # one value; the rest zero (and -0)
    x[3, 301] = -0.0
    levels = np.array([X.e4m3_value(c) for c in range(0x7F)])
    x[4, 384:512] = rng.choice(levels, 128) * 0.25     # on the grid, scale exactly 2^-2 ...
    x[4, 400] = 448.0 * 0.25                           # ... once 448 * 2^-2 is present
    mid = (levels[1:] + levels[:-1]) / 2               # the 126 exact ties between neighbours
    x[5, :126] = mid
    x[5, 126] = 0.0
    x[5, 127] = 448.0                                  # scale 1, so the ties stay ties
    return W.float_to_bf16_bits(x).reshape(n, 576)


def test_library_encoder_matches_the_oracle(lib):
    rng = np.random.default_rng(12)
    bits = _rows(rng, 64)
    got = ess.ess_compact_rows(bits)
    want = np.stack([X.encode_row(b) for b in bits])
    assert got.shape == (64, 656)
    assert np.array_equal(got, want)


def test_library_encoder_rejects_bad_arguments(lib):
    assert lib.ess_compact_rows(None, 1, None) == ess.ESS_ERR_INVALID_ARG
    assert lib.ess_compact_rows(None, -1, None) == ess.ESS_ERR_INVALID_ARG
    assert lib.ess_compact_rows(None, 0, None) == ess.ESS_OK
