"""The library's prefill binding table (ess_prefill_plan, host code, no GPU)
against the oracle's timeline model of the same schedule (FlashOffloading
analysis, section "prefill side")."""
import numpy as np
import pytest

from host_latent_cache_gb300 import ess
from oracle import prefill_schedule as S


@pytest.fixture(scope="module")
def lib():
    from host_latent_cache_gb300 import build as B
    B.build()
    return ess.load()


def test_figure3_plan(lib):
    L = 6
    m = [i + 1 if i + 1 < L else -1 for i in range(L)]
    buf, at, after = ess.ess_prefill_plan(m)
    assert buf.tolist() == [0, 1, 2, 3, 1, 2]
    assert at.tolist() == [-1, 0, 1, 2, 3, 4]
    assert after.tolist() == [-1, -1, -1, -1, 1, 2]      # B1 and B2 come back after layers 1, 2


def test_plan_matches_the_oracle_timeline(lib):
    rng = np.random.default_rng(21)
    agree = refused = 0
    for _ in range(400):
        L = int(rng.integers(1, 12))
        d = int(rng.integers(1, 5))
        m = [i + d if i + d < L else -1 for i in range(L)]
        if rng.random() < 0.3 and L > 2:                  # some layers left for up front
            m[int(rng.integers(0, L))] = -1
        R = int(rng.integers(1, 5))
        shared = bool(rng.integers(0, 2))
        try:
            t = S.simulate(L, [1.0] * L, [0.5] * L, [0.3] * L, onload_layer_map=m, rotating=R,
                           shared_copy=shared)
        except ValueError:
            t = None
        if t is None:
            with pytest.raises(ess.EssError) as e:
                ess.ess_prefill_plan(m, R, shared)
            assert e.value.code == ess.ESS_ERR_INVALID_ARG
            refused += 1
        else:
            buf, _, _ = ess.ess_prefill_plan(m, R, shared)
            assert buf.tolist() == t.buffer, (m, R, shared)
            agree += 1
    assert agree > 50 and refused > 50


def test_plan_rejects_bad_maps(lib):
    for m in ([1, 1, -1], [0, -1, -1], [3, -1, -1], [-5, -1]):
        with pytest.raises(ess.EssError):
            ess.ess_prefill_plan(m)
