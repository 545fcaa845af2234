"""Pins of the eviction-policy replay (oracle/eviction_replay.py), and the
plausible mistakes they catch.

The replay restates the offline simulator of the FlashOffloading analysis,
section "evaluation" (the decode ablation and Figure 8): the same trace of
selected tokens, replayed with Random, LRU, Score or LIM eviction.  The pins
are closed forms that hold for every policy, hand-worked traces that tell the
policies apart, the published reference outputs of the random generator, a
uniformity property, and agreement of the LRU replay with the oracle's pinned
lru_update.
"""
import inspect
import sys

import numpy as np
import pytest

from oracle import ess_oracle as O
from oracle import eviction_replay as R
from host_latent_cache_gb300 import workloads as W


def _trace(rng, steps, T, k, M=1, drift=0.2):
    """Selections that drift: each step keeps most of the previous set."""
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


def test_splitmix64_reference_outputs():
    # the first five outputs of SplitMix64 seeded with 1234567, as printed by
    # the generator's reference implementation (Steele, Lea and Flood 2014)
    s, got = 1234567, []
    for _ in range(5):
        s, o = R.splitmix64(s)
        got.append(o)
    assert got == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]
    assert R.splitmix64_at(1234567, 2) == 9817491932198370423


@pytest.mark.parametrize("policy", R.POLICIES)
def test_pool_holding_every_token_has_only_first_time_misses(policy):
    rng = np.random.default_rng(5)
    tr = _trace(rng, 12, T=200, k=16, M=2)
    sc = [[rng.random(200) for _ in range(2)] for _ in tr]
    got = R.replay(tr, C=200, policy=policy, scores=sc, seed=3)["union_misses"]
    seen, want = set(), []
    for ways in tr:
        u = set(np.concatenate(ways).tolist())
        want.append(len(u - seen))
        seen |= u
    assert got.tolist() == want


@pytest.mark.parametrize("policy", R.POLICIES)
def test_pool_the_size_of_the_union_is_policy_free(policy):
    # one way of k tokens and C = k: every slot outside the union must go, so
    # the misses are |U_s \ U_{s-1}| whatever the order
    rng = np.random.default_rng(6)
    tr = _trace(rng, 15, T=120, k=24)
    sc = [[rng.random(120)] for _ in tr]
    got = R.replay(tr, C=24, policy=policy, scores=sc, seed=4)["union_misses"]
    want = [24] + [len(set(tr[s][0].tolist()) - set(tr[s - 1][0].tolist()))
                   for s in range(1, len(tr))]
    assert got.tolist() == want


def _hand(policy, s3_scores):
    # C = 3; s0 {1,2} fills slots 0, 1; s1 {2,3} puts 3 in the empty slot 2;
    # s2 {1,3} only hits (slot 1 keeps the older stamp); s3 {3,5} misses 5
    # with candidates slot 0 (token 1, stamped at s2) and slot 1 (token 2,
    # stamped at s1)
    st = R.ReplayState.empty(3)
    misses = []
    for s, u in enumerate([[1, 2], [2, 3], [1, 3], [3, 5]]):
        ts = {t: s3_scores.get(t, 0.5) for t in st.slot_of} if s == 3 else \
            {t: 0.5 for t in st.slot_of}
        misses.append(R.replay_step(st, np.array(u), policy, ts, key=R.random_key(0, 0, s)).tolist())
    return misses, st.slot_token.tolist()


def test_hand_trace_lru_evicts_the_older_stamp():
    misses, slots = _hand("lru", {})
    assert misses == [[1, 2], [3], [], [5]]
    assert slots == [1, 5, 3]


def test_hand_trace_lim_scans_in_slot_order():
    misses, slots = _hand("lim", {})
    assert misses == [[1, 2], [3], [], [5]]
    assert slots == [5, 2, 3]


def test_hand_trace_score_evicts_the_lower_score():
    assert _hand("score", {1: 0.9, 2: 0.1})[1] == [1, 5, 3]
    assert _hand("score", {1: 0.1, 2: 0.9})[1] == [5, 2, 3]
    assert _hand("score", {1: 0.3, 2: 0.3})[1] == [5, 2, 3]     # equal: the lower slot


def test_empty_slots_go_first_for_every_policy():
    for policy in R.POLICIES:
        _, slots = _hand(policy, {1: 0.9, 2: 0.1})
        assert slots[2] == 3, policy      # s1 used the empty slot, not token 1's


def test_random_choice_is_uniform_and_varies_by_step():
    # two resident candidates, 4000 steps: each goes first about half the time
    st = R.ReplayState.empty(2)
    st.slot_token[:] = [10, 11]
    st.last_used[:] = [0, 0]
    first = [int(R.victim_order("random", np.array([0, 1]), st, None, R.random_key(9, 2, s))[0])
             for s in range(4000)]
    frac = sum(1 for f in first if f == 0) / 4000
    assert 0.46 < frac < 0.54
    other = [int(R.victim_order("random", np.array([0, 1]), st, None, R.random_key(9, 3, s))[0])
             for s in range(4000)]
    assert first != other                 # requests draw independently


def test_way_misses_count_each_way():
    tr = [[np.array([1, 2]), np.array([2, 3])], [np.array([2, 4]), np.array([3, 4])]]
    r = R.replay(tr, C=8, policy="lru")
    assert r["union_misses"].tolist() == [3, 1]
    assert r["way_misses"].tolist() == [4, 2]


def test_lru_replay_matches_the_oracle_lru():
    rng = np.random.default_rng(8)
    tr = _trace(rng, 30, T=400, k=32, M=2, drift=0.3)
    st = O.CacheState.empty(400, 80)
    want = []
    for ways in tr:
        r = O.resolve_union(ways, st.cache_slots)
        O.lru_update(st, r.union, r.miss_tok)
        want.append(r.miss_tok.shape[0])
    rs = R.ReplayState.empty(80)
    got = [R.replay_step(rs, np.concatenate(w), "lru").shape[0] for w in tr]
    assert got == want
    assert rs.slot_token.tolist() == st.slot_token.tolist()


def test_replay_over_the_oracle_trace_capacity_helps_every_policy():
    # selections of the oracle on a small drifting workload (the pages' trace
    # stands in): doubling the pool never adds misses here
    cfg = W.tiny().replace(T=2048, k=64, rho=0.9, seed=77)
    ld = W.gen_layer(cfg)
    keys = W.decode_keys(cfg, ld.idx_keys)
    lay = O.OracleLayer(ld.T, 4096, cfg.k, cfg.sm_scale)
    qs = W.QueryStream(cfg)
    tr, sc = [], []
    for _ in range(40):
        q, _, _ = qs.next()
        r = lay.step(q, W.head_weights(cfg, ld.w), keys, ld.idx_scale, None, None,
                     keep_scores=True)
        tr.append(r.topk[0])
        sc.append(r.scores[0])
    for policy in R.POLICIES:
        small = R.replay(tr, 96, policy, sc, seed=1)["union_misses"].sum()
        large = R.replay(tr, 192, policy, sc, seed=1)["union_misses"].sum()
        assert large <= small, policy


# ------------------------------------------------------------------ mutants

def _order_highest_score_first(policy, cand, st, token_score, key):
    if policy == "score":
        flipped = {t: -v for t, v in token_score.items()}
        return ORIG(policy, cand, st, flipped, key)
    return ORIG(policy, cand, st, token_score, key)


def _order_lim_from_the_top(policy, cand, st, token_score, key):
    out = ORIG(policy, cand, st, token_score, key)
    if policy == "lim":
        res = st.slot_token[out] >= 0
        return np.concatenate([out[~res], out[res][::-1]])
    return out


def _order_resident_first(policy, cand, st, token_score, key):
    out = ORIG(policy, cand, st, token_score, key)
    res = st.slot_token[out] >= 0
    return np.concatenate([out[res], out[~res]])


def _order_random_ignores_key(policy, cand, st, token_score, key):
    return ORIG(policy, cand, st, token_score, 0)


def _order_lru_most_recent(policy, cand, st, token_score, key):
    out = ORIG(policy, cand, st, token_score, key)
    if policy == "lru":
        res = st.slot_token[out] >= 0
        r = out[res]
        r = r[np.lexsort((r, -st.last_used[r]))]
        return np.concatenate([out[~res], r])
    return out


ORIG = R.victim_order
MUTANTS = [_order_highest_score_first, _order_lim_from_the_top, _order_resident_first,
           _order_random_ignores_key, _order_lru_most_recent]
PINS = [f for name, f in sorted(vars(sys.modules[__name__]).items())
        if name.startswith("test_") and inspect.isfunction(f) and name != "test_pins_catch_mutant"
        and not hasattr(f, "pytestmark")]


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m.__name__ for m in MUTANTS])
def test_pins_catch_mutant(monkeypatch, mutant):
    monkeypatch.setattr(R, "victim_order", mutant)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (Exception, pytest.fail.Exception) as e:   # an assertion or a pytest.raises miss
            failed.append(f"{pin.__name__}: {type(e).__name__}")
            break
    assert failed, f"no pin notices {mutant.__name__}"
