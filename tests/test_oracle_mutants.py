"""The oracle's pins catch plausible mistakes.

Each case below replaces one oracle function with a copy that carries one
plausible mistake (a dropped term, a wrong sign, order or index, a step
out of order) and runs the pins of tests/test_oracle_pins.py against it.
At least one pin must fail for every mistake; a mistake that no pin
notices would mean the oracle is not pinned where it matters.  The
mistakes are planted in the oracle, on the CPU, through monkeypatch.
"""
from __future__ import annotations

import inspect

import numpy as np
import pytest

from oracle import ess_oracle as O
from tests import test_oracle_pins as P

PINS = [f for name, f in sorted(vars(P).items())
        if name.startswith("test_") and inspect.isfunction(f)]


# ------------------------------------------------------------- indexer score

def score_no_relu(q, w, keys, scale, check_exact=True):
    q, w, keys = (np.asarray(x, dtype=np.float64) for x in (q, w, keys))
    inner = (keys @ q.T) @ w
    return (inner.astype(np.float32).astype(np.float64)
            * np.asarray(scale, np.float32).astype(np.float64)).astype(np.float32)


def score_no_scale(q, w, keys, scale, check_exact=True):
    q, w, keys = (np.asarray(x, dtype=np.float64) for x in (q, w, keys))
    return (np.maximum(keys @ q.T, 0.0) @ w).astype(np.float32)


def score_relu_after_weights(q, w, keys, scale, check_exact=True):
    q, w, keys = (np.asarray(x, dtype=np.float64) for x in (q, w, keys))
    inner = np.maximum((keys @ q.T) @ w, 0.0)
    return (inner.astype(np.float32).astype(np.float64)
            * np.asarray(scale, np.float32).astype(np.float64)).astype(np.float32)


# ------------------------------------------------------------------- top-k

def topk_higher_index_wins(scores, k):
    scores = np.asarray(scores, dtype=np.float32)
    idx = np.arange(scores.shape[0])
    return np.lexsort((-idx, -scores.astype(np.float64)))[:min(k, len(scores))].astype(np.int64)


def topk_smallest(scores, k):
    scores = np.asarray(scores, dtype=np.float32)
    idx = np.arange(scores.shape[0])
    return np.lexsort((idx, scores.astype(np.float64)))[:min(k, len(scores))].astype(np.int64)


# ---------------------------------------------------------- resolve / union

def resolve_first_way_only(topk, cache_slots):
    return O.__dict__["_orig_resolve_union"](list(topk)[:1], cache_slots)


def resolve_slot_zero_is_miss(topk, cache_slots):
    hits, misses = [], []
    for sel in topk:
        s = cache_slots[np.asarray(sel, dtype=np.int64)]
        h = int(np.count_nonzero(s > 0))
        hits.append(h)
        misses.append(len(sel) - h)
    union = np.unique(np.concatenate([np.asarray(s, dtype=np.int64) for s in topk])) \
        if len(topk) else np.zeros(0, np.int64)
    res = cache_slots[union] > 0
    return O.Resolve(hits, misses, union, union[~res], res)


# --------------------------------------------------------------------- LRU

def _lru(state, union, miss_tok, *, mru=False, slot_desc=False, stamp_late=False,
         keep_union=False):
    C = state.slot_token.shape[0]
    step = state.step
    if union.shape[0] > C:
        raise O.CapacityError("capacity")
    slots_u = state.cache_slots[union]
    hit_slots = slots_u[slots_u >= 0]
    if not stamp_late:
        state.last_used[hit_slots] = step
    in_union = np.zeros(C, dtype=bool)
    if not keep_union:
        in_union[hit_slots] = True
    cand = np.nonzero(~in_union)[0]
    lu = state.last_used[cand]
    order = np.lexsort((-cand if slot_desc else cand, -lu if mru else lu))
    victims = cand[order[: miss_tok.shape[0]]].astype(np.int64)
    evicted = np.full(miss_tok.shape[0], -1, dtype=np.int64)
    for i, (t, v) in enumerate(zip(miss_tok.tolist(), victims.tolist())):
        old = int(state.slot_token[v])
        if old >= 0:
            state.cache_slots[old] = -1
        evicted[i] = old
        state.cache_slots[t] = v
        state.slot_token[v] = t
        state.last_used[v] = step
    if stamp_late:
        state.last_used[hit_slots] = step
    state.step += 1
    return victims, evicted


def lru_most_recent_first(state, union, miss_tok):
    return _lru(state, union, miss_tok, mru=True)


def lru_ties_to_higher_slot(state, union, miss_tok):
    return _lru(state, union, miss_tok, slot_desc=True)


def lru_evicts_selected_rows(state, union, miss_tok):
    # victims chosen among all slots before the hits are stamped, so a
    # selected row can be evicted (either change alone is harmless: stamped
    # hits sort after every other slot, and unstamped ones are excluded)
    return _lru(state, union, miss_tok, keep_union=True, stamp_late=True)


def lru_pairs_misses_in_reverse(state, union, miss_tok):
    return O.__dict__["_orig_lru_update"](state, union, miss_tok[::-1].copy())


# --------------------------------------------------------------- attention

def mla_no_max_subtraction(q, rows, sm_scale, latent_dim=512):
    q, rows = np.asarray(q, np.float64), np.asarray(rows, np.float64)
    if rows.shape[0] == 0:
        return np.zeros((q.shape[0], latent_dim), np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        p = np.exp(float(sm_scale) * (q @ rows.T))
        p /= np.sum(p, axis=1, keepdims=True)
    return (p @ rows[:, :latent_dim]).astype(np.float32)


def mla_latent_only_logits(q, rows, sm_scale, latent_dim=512):
    q, rows = np.asarray(q, np.float64), np.asarray(rows, np.float64)
    return O.__dict__["_orig_sparse_mla"](q[:, :latent_dim], rows[:, :latent_dim], sm_scale,
                                          latent_dim)


def mla_no_scale(q, rows, sm_scale, latent_dim=512):
    return O.__dict__["_orig_sparse_mla"](q, rows, 1.0, latent_dim)


def mla_values_include_rope(q, rows, sm_scale, latent_dim=512):
    rows = np.asarray(rows, np.float64)
    if rows.shape[0] == 0:
        return np.zeros((np.asarray(q).shape[0], latent_dim), np.float32)
    shifted = np.concatenate([rows[:, 64:], rows[:, :64]], axis=1)   # value dims off by 64
    q = np.asarray(q, np.float64)
    logits = float(sm_scale) * (q @ rows.T)
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return (p @ shifted[:, :latent_dim]).astype(np.float32)


# ------------------------------------------------------------------ append

def append_without_growth(T, states):
    pass


def append_new_token_resident(T, states):
    # the new token claims slot 0 as if it were already in the hot cache
    for b in range(len(T)):
        T[b] += 1
        states[b].cache_slots = np.append(states[b].cache_slots, np.int32(0))


MUTANTS = [
    ("score_indexer", score_no_relu),
    ("score_indexer", score_no_scale),
    ("score_indexer", score_relu_after_weights),
    ("topk_select", topk_higher_index_wins),
    ("topk_select", topk_smallest),
    ("resolve_union", resolve_first_way_only),
    ("resolve_union", resolve_slot_zero_is_miss),
    ("lru_update", lru_most_recent_first),
    ("lru_update", lru_ties_to_higher_slot),
    ("lru_update", lru_evicts_selected_rows),
    ("lru_update", lru_pairs_misses_in_reverse),
    ("sparse_mla", mla_no_max_subtraction),
    ("sparse_mla", mla_latent_only_logits),
    ("sparse_mla", mla_no_scale),
    ("sparse_mla", mla_values_include_rope),
    ("append_tokens", append_without_growth),
    ("append_tokens", append_new_token_resident),
]


def _pins_failing(stop_after=1):
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (Exception, pytest.fail.Exception) as e:   # an assertion, a pytest.raises miss,
            # or the mistake breaking a contract
            failed.append(f"{pin.__name__}: {type(e).__name__}")
            if len(failed) >= stop_after:
                break
    return failed


def test_pins_pass_on_the_oracle():
    assert _pins_failing() == []


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=[m.__name__ for _, m in MUTANTS])
def test_pins_catch_mutant(monkeypatch, name, mutant):
    monkeypatch.setitem(O.__dict__, "_orig_" + name, getattr(O, name))
    monkeypatch.setattr(O, name, mutant)
    failed = _pins_failing()
    assert failed, f"no pin notices the mutant {mutant.__name__} of {name}"
