"""CPU replay of hot-pool eviction policies over a trace of selections.

TEST INFRASTRUCTURE ONLY.  Only the tests may import this module.  It shares
no code with the CUDA library.

What it restates: hwcomputing.csdn.net FlashOffloading analysis, section
"evaluation", the decode ablation "capacity matters more than the eviction
policy" and its Figure 8.  The top-k indices of every layer and step are
collected once, then an offline simulator replays the same access sequence
with only the eviction policy changed: Random, LRU, Score (evict low-score
tokens) and LIM (a score threshold plus a chunk scan).  The figure plots
misses per request and layer, summed over the MTP ways, against the hot-pool
budget.

One replayed step of one request is the bookkeeping of the oracle's
resolve_union and lru_update with the victim order made a parameter:
  1. hits are the union tokens already resident; misses the others;
  2. hits are stamped with the step;
  3. the candidates are the slots whose token is not in the union (empty
     slots included); the first |Miss| of them in the policy's order are
     the victims;
  4. the i-th miss (ascending token) takes the i-th victim.

Victim orders (ties always go to the lower slot; an empty slot counts as
older, lower-scored and colder than any resident token):
  lru     last_used ascending;
  random  a priority drawn per (request, step, slot) from SplitMix64, the
          counter-based generator of Steele, Lea and Flood, "Fast Splittable
          Pseudorandom Number Generators" (OOPSLA 2014), ascending;
  score   the resident token's current score ascending (the maximum over
          the ways' scores of this step);
  lim     slot order: the page names a score threshold and a chunk scan but
          gives neither the threshold nor the chunk.  The reading taken: the
          threshold is the step's top-k cutoff, so every token outside the
          union is below it in every way, and the scan walks the slots in
          ascending order and stops once it has |Miss| victims.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np

POLICIES = ("lru", "random", "score", "lim")

_MASK = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15


def splitmix64(state: int) -> tuple[int, int]:
    """One SplitMix64 step: returns (new state, output)."""
    state = (state + _GAMMA) & _MASK
    z = state
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
    return state, z ^ (z >> 31)


def splitmix64_at(key: int, i: int) -> int:
    """The (i+1)-th output of SplitMix64 seeded with key (counter-based use)."""
    _, out = splitmix64((key + i * _GAMMA) & _MASK)
    return out


def random_key(seed: int, request: int, step: int) -> int:
    """Generator key of one (request, step) of the Random policy."""
    k = seed & _MASK
    for v in (request, step):
        _, k = splitmix64((k ^ (v & _MASK)) & _MASK)
    return k


@dataclass
class ReplayState:
    """Hot-pool bookkeeping of one request: token -> slot and slot -> token."""
    slot_of: Dict[int, int]
    slot_token: np.ndarray    # int64 [C], -1 empty
    last_used: np.ndarray     # int64 [C], -1 empty
    step: int = 0

    @staticmethod
    def empty(C: int) -> "ReplayState":
        return ReplayState({}, np.full(C, -1, np.int64), np.full(C, -1, np.int64), 0)


def victim_order(policy: str, cand: np.ndarray, st: ReplayState,
                 token_score: Optional[Dict[int, float]], key: int) -> np.ndarray:
    """Candidate slots in the policy's eviction order: empty slots first (in
    slot order), then the resident ones by the policy's key, then by slot."""
    cand = np.asarray(cand, dtype=np.int64)
    resident = (st.slot_token[cand] >= 0).astype(np.int64)
    if policy == "lru":
        primary = st.last_used[cand]
    elif policy == "random":
        primary = np.array([splitmix64_at(key, int(v)) for v in cand], dtype=np.uint64)
    elif policy == "score":
        if token_score is None:
            raise ValueError("the score policy needs this step's scores")
        primary = np.array([token_score[int(t)] if r else 0.0
                            for r, t in zip(resident, st.slot_token[cand])], dtype=np.float64)
    elif policy == "lim":
        primary = np.zeros(cand.shape[0], dtype=np.int64)
    else:
        raise ValueError(f"unknown policy {policy}")
    primary = np.where(resident == 1, primary, 0)          # empty slots: slot order
    return cand[np.lexsort((cand, primary, resident))]


def replay_step(st: ReplayState, union: np.ndarray, policy: str,
                token_score: Optional[Dict[int, float]] = None, key: int = 0) -> np.ndarray:
    """One step for one request; returns the miss tokens (ascending).
    Mutates st and advances its step."""
    C = st.slot_token.shape[0]
    union = np.unique(np.asarray(union, dtype=np.int64))
    if union.shape[0] > C:
        raise ValueError(f"union {union.shape[0]} > C {C}")
    hit = np.array([int(t) in st.slot_of for t in union], dtype=bool)
    miss = union[~hit]
    hit_slots = np.array([st.slot_of[int(t)] for t in union[hit]], dtype=np.int64)
    st.last_used[hit_slots] = st.step
    held = np.zeros(C, dtype=bool)
    held[hit_slots] = True
    cand = np.nonzero(~held)[0]
    victims = victim_order(policy, cand, st, token_score, key)[: miss.shape[0]]
    for t, v in zip(miss.tolist(), victims.tolist()):
        old = int(st.slot_token[v])
        if old >= 0:
            del st.slot_of[old]
        st.slot_of[t] = v
        st.slot_token[v] = t
        st.last_used[v] = st.step
    st.step += 1
    return miss


def replay(trace: Sequence[Sequence[np.ndarray]], C: int, policy: str,
           scores: Optional[Sequence[Sequence[np.ndarray]]] = None, seed: int = 0,
           request: int = 0) -> Dict[str, np.ndarray]:
    """Replay one request's trace: trace[s][m] holds way m's selected tokens
    at step s; scores[s][m] the way's scores of all tokens at step s (needed
    by the score policy).  Returns per step the union misses and the misses
    summed over the ways (a way's selected token that was not resident before
    the step)."""
    st = ReplayState.empty(C)
    union_miss, way_miss = [], []
    for s, ways in enumerate(trace):
        ways = [np.asarray(w, dtype=np.int64) for w in ways]
        union = np.unique(np.concatenate(ways)) if ways else np.zeros(0, np.int64)
        ts = None
        if scores is not None:
            best = np.max(np.stack([np.asarray(x, np.float64) for x in scores[s]]), axis=0)
            ts = {int(t): float(best[t]) for t in st.slot_of}
        resident = set(st.slot_of)
        way_miss.append(sum(int(np.count_nonzero([int(t) not in resident for t in w]))
                            for w in ways))
        miss = replay_step(st, union, policy, ts, random_key(seed, request, s))
        union_miss.append(miss.shape[0])
    return {"union_misses": np.asarray(union_miss), "way_misses": np.asarray(way_miss)}
