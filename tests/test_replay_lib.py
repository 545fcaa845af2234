"""The library's eviction replay (ess_replay_misses, host code, no GPU)
against the oracle's replay, step by step, for every policy (FlashOffloading
analysis, section "evaluation": the decode ablation's offline simulator)."""
import numpy as np
import pytest

from host_latent_cache_gb300 import ess
from oracle import eviction_replay as R

POLICY = {"lru": ess.ESS_EVICT_LRU, "random": ess.ESS_EVICT_RANDOM,
          "score": ess.ESS_EVICT_SCORE, "lim": ess.ESS_EVICT_LIM}


@pytest.fixture(scope="module")
def lib():
    from host_latent_cache_gb300 import build as B
    B.build()
    return ess.load()


def _trace(rng, steps, T, k, M, drift):
    cur = [rng.choice(T, k, replace=False) for _ in range(M)]
    out = []
    for _ in range(steps):
        nxt = []
        for c in cur:
            keep = c[rng.random(k) > drift]
            fresh = rng.choice(np.setdiff1d(np.arange(T), keep), k - keep.shape[0], replace=False)
            nxt.append(np.concatenate([keep, fresh]))
        cur = nxt
        out.append([np.sort(c) for c in cur])
    return out


@pytest.mark.parametrize("policy", sorted(POLICY))
def test_library_replay_matches_the_oracle(lib, policy):
    rng = np.random.default_rng(17)
    for trial in range(6):
        T, k, M = 600, int(rng.integers(8, 40)), int(rng.integers(1, 4))
        C = int(rng.integers(M * k, 4 * M * k))
        tr = _trace(rng, 25, T, k, M, drift=float(rng.uniform(0.05, 0.5)))
        sc = [[rng.random(T).astype(np.float32) for _ in range(M)] for _ in tr]
        sc[3][0][:] = 0.5                                  # a step of equal scores
        want = R.replay(tr, C, policy, sc, seed=99, request=trial)
        um, wm = ess.ess_replay_misses(tr, T, C, POLICY[policy], sc, seed=99, request=trial)
        assert um.tolist() == want["union_misses"].tolist(), (policy, trial)
        assert wm.tolist() == want["way_misses"].tolist(), (policy, trial)


def test_library_replay_refuses_an_overfull_step(lib):
    tr = [[np.arange(10)]]
    with pytest.raises(ess.EssError) as e:
        ess.ess_replay_misses(tr, 20, 5, ess.ESS_EVICT_LRU)
    assert e.value.code == ess.ESS_ERR_CAPACITY
    with pytest.raises(ess.EssError):
        ess.ess_replay_misses([[np.array([25])]], 20, 5, ess.ESS_EVICT_LRU)
    with pytest.raises(ess.EssError):                      # Score needs the scores
        ess.ess_replay_misses(tr, 20, 16, ess.ESS_EVICT_SCORE)
