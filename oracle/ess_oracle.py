"""CPU oracle for sparse decode with a host-resident latent cache.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of the entry
module and the bench's CPU-baseline leg may import or call this module.
The product path never routes through it.  It shares no code with the
CUDA library: inputs come from the seeded generators, and nothing here
reads a value computed by the GPU.

It is a plain, slow, obviously correct restatement of what the decode
path computes, in float64 where the arithmetic is floating point:

1. indexer scores over the full context      (score_indexer)
2. exact top-k with the lower index winning ties (topk_select)
3. hit/miss resolution against cache_slots and the miss union over the
   MTP ways                                    (resolve_union)
4. LRU victim choice and the cache_slots / slot_token / last_used update
   (lru_update)
5. absorbed-MLA softmax attention over the selected latent rows, read
   straight from the full latent array, never from a pool (sparse_mla)
6. decode append: every request gains its newest token (append_tokens)

Sources (web pages on latent-cache offload for DSA sparse decode):

* hwcomputing.csdn.net FlashOffloading analysis, section
  "decode side (1): fold the miss lookup into top-k":
  - subsection "cache_slots": per request and layer an int32 token->slot
    vector, -1 when not resident; load Miss_b = T_b - C_b and evict as
    many, so the hot cache keeps its size;
  - subsection "five steps and the four-way MTP3 merge": (1) look up each
    way's top-k in cache_slots, (2) take the union of the misses, (3)
    remove the union of the top-k from C_b and pick as many victims as
    there are misses, (4) pair each miss with a victim and rewrite
    cache_slots, (5) copy the misses from DRAM into the paired slots, then
    run sparse attention;
  - the 20-candidate worked example and Figure 4 (tokens 8 and 17 miss
    and land in the evicted slots 3 and 5).
* The same page, section "account first": kappa_base = (L_KV*D_KV +
  L_index*D_index)*P per token, the decode residency formula
  M_decode ~ L(C+2b)s_KV + ..., and the OverlapRatio definition in
  section "decode side (2)".
* The same page, section "architecture: one master copy, two residency
  policies" and its Figure 2: besides the hot cache of C slots the decode
  side keeps two tail blocks that take the newly produced KV, and the host
  keeps the authoritative copy paged by token block.
* "ESS: Latent-Cache Offload" (foosynaptic tech notes): the indexer keeps
  one light vector per position and scores all positions to choose the
  top-2048; the latent entry is c^KV[512] + k^R[64]; the GPU sparse pool
  keeps a hot subset under LRU.

Readings where the pages are silent (each also listed in the design
notes): the indexer score is sum_h w_h * ReLU(q_h . k_s) times the
per-token key scale, applied once after the head sum; ties in the top-k
go to the lower token index; the LRU recency unit is a per-layer step
counter, hits are stamped before victims are chosen, and victims are
ordered by (last_used asc, slot asc) with empty slots (last_used = -1)
first; the i-th miss (ascending token) takes the i-th victim; the pool
starts empty; attention outputs are float32; a newly appended token is
not in the hot cache (it sits in a tail block), so it starts with
cache_slots = -1 and is loaded into a slot, like any miss, when a step first
selects it.

Parity pins live in tests/test_oracle_pins.py.  Every function here is
pinned by at least one value or property fixed by the pages or by
mathematics.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np

SCORE_EXACT_BOUND = 4096.0  # partial sums stay exact in fp32 below this (2^24 quanta of 2^-12)


class CapacityError(RuntimeError):
    """The union of the selected tokens does not fit in the hot pool."""


# --------------------------------------------------------------------------
# byte accounting (FlashOffloading page, section "account first")
# --------------------------------------------------------------------------

def kv_bytes_per_token(L_kv: int, D_kv: int, L_index: int, D_index: int, P: int) -> int:
    """kappa_base = (L_KV*D_KV + L_index*D_index) * P bytes per token."""
    return (L_kv * D_kv + L_index * D_index) * P


def decode_residency_bytes(L: int, C: int, b: int, s_kv: int, m_index: int = 0,
                           m_slots: int = 0, m_meta: int = 0) -> int:
    """M_decode ~ L(C + 2b) s_KV + M_index + M_slots + M_meta."""
    return L * (C + 2 * b) * s_kv + m_index + m_slots + m_meta


def overlap_ratio(t_copy: float, t_sfa: float, t_fused: float) -> float:
    """OverlapRatio = (T_copy + T_SFA - T_fused) / T_copy."""
    return (t_copy + t_sfa - t_fused) / t_copy


# --------------------------------------------------------------------------
# 1. indexer score
# --------------------------------------------------------------------------

def score_indexer(q: np.ndarray, w: np.ndarray, keys: np.ndarray, scale: np.ndarray,
                  check_exact: bool = True) -> np.ndarray:
    """Indexer scores of one way over all positions of one request.

    q      float64 [H_I][d_I]  query values
    w      float64 [H_I]       head weights
    keys   float64 [T][d_I]    key values
    scale  float32 [T]         per-token key scale
    returns float32 [T]:  fl32( scale_t * sum_h w_h * max(0, q_h . k_t) )

    The inner sum is formed in float64; under the exact-score data contract
    it is exact, and it is checked to convert to float32 without rounding.
    The scale multiply is one correctly rounded float32 product.
    """
    q = np.asarray(q, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    dots = keys @ q.T                                   # [T][H_I], a library matmul
    relu = np.maximum(dots, 0.0)
    inner = relu @ w                                    # [T]
    inner32 = inner.astype(np.float32)
    if check_exact:
        if np.any(inner >= SCORE_EXACT_BOUND):
            raise ValueError("indexer score outside the exact-score bound")
        if not np.array_equal(inner32.astype(np.float64), inner):
            raise ValueError("indexer inner sum not exact in float32")
    prod = inner32.astype(np.float64) * np.asarray(scale, dtype=np.float32).astype(np.float64)
    s = prod.astype(np.float32)        # product of two fp32 is exact in fp64: one rounding
    return s + np.float32(0.0)         # canonical +0


# --------------------------------------------------------------------------
# 2. top-k
# --------------------------------------------------------------------------

def topk_select(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores, ordered by (score desc, index asc).

    When k exceeds the number of positions every position is selected.
    """
    scores = np.asarray(scores, dtype=np.float32)
    T = scores.shape[0]
    k = min(k, T)
    idx = np.arange(T)
    order = np.lexsort((idx, -scores.astype(np.float64)))   # stable library sort
    return order[:k].astype(np.int64)


# --------------------------------------------------------------------------
# 3 + 4. cache management
# --------------------------------------------------------------------------

@dataclass
class CacheState:
    """Per-request hot-pool bookkeeping of one layer."""
    cache_slots: np.ndarray   # int32 [T]   token -> slot, -1 if not resident
    slot_token: np.ndarray    # int32 [C]   slot -> token, -1 if empty
    last_used: np.ndarray     # int32 [C]   step of last use, -1 if empty
    step: int = 0

    @staticmethod
    def empty(T: int, C: int) -> "CacheState":
        return CacheState(np.full(T, -1, np.int32), np.full(C, -1, np.int32),
                          np.full(C, -1, np.int32), 0)

    def copy(self) -> "CacheState":
        return CacheState(self.cache_slots.copy(), self.slot_token.copy(),
                          self.last_used.copy(), self.step)


@dataclass
class Resolve:
    hits: List[int]           # per way
    misses: List[int]         # per way
    union: np.ndarray         # ascending tokens selected by any way
    miss_tok: np.ndarray      # ascending tokens of the union that are not resident
    was_resident: np.ndarray  # bool per union token


def resolve_union(topk: Sequence[np.ndarray], cache_slots: np.ndarray) -> Resolve:
    """Step (1) look-up per way and step (2) the miss union over the ways."""
    hits, misses = [], []
    for sel in topk:
        s = cache_slots[np.asarray(sel, dtype=np.int64)]
        h = int(np.count_nonzero(s >= 0))
        hits.append(h)
        misses.append(len(sel) - h)
    if len(topk):
        union = np.unique(np.concatenate([np.asarray(s, dtype=np.int64) for s in topk]))
    else:
        union = np.zeros(0, np.int64)
    res = cache_slots[union] >= 0
    return Resolve(hits, misses, union, union[~res], res)


def lru_update(state: CacheState, union: np.ndarray, miss_tok: np.ndarray
               ) -> Tuple[np.ndarray, np.ndarray]:
    """Steps (3) and (4): stamp hits, choose LRU victims, pair and rewrite.

    Returns (victim_slots, evicted_tokens), aligned with miss_tok.
    Mutates state and advances its step counter.
    """
    C = state.slot_token.shape[0]
    step = state.step
    if union.shape[0] > C:
        raise CapacityError(f"union {union.shape[0]} > C {C}")
    slots_u = state.cache_slots[union]
    hit_slots = slots_u[slots_u >= 0]
    state.last_used[hit_slots] = step                   # hits are stamped first
    in_union = np.zeros(C, dtype=bool)
    in_union[hit_slots] = True
    cand = np.nonzero(~in_union)[0]                     # slots whose token is not in the union
    order = np.lexsort((cand, state.last_used[cand]))   # last_used asc, then slot asc
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
    state.step += 1
    return victims, evicted


# --------------------------------------------------------------------------
# 6. decode append
# --------------------------------------------------------------------------

def append_tokens(T: List[int], states: List[CacheState]) -> None:
    """Every request gains its newest token: T_b grows by one and the new
    token is not resident in the hot cache.

    New KV goes to the tail blocks beside the hot cache, not into one of its
    C slots, so cache_slots gets a -1 entry.  Whether the bytes sit in a tail
    block or already in the host copy changes no result, so nothing about
    them is tracked here.  Mutates T and states.
    """
    for b in range(len(T)):
        T[b] += 1
        states[b].cache_slots = np.append(states[b].cache_slots, np.int32(-1))


# --------------------------------------------------------------------------
# 5. sparse absorbed-MLA attention
# --------------------------------------------------------------------------

def sparse_mla(q: np.ndarray, rows: np.ndarray, sm_scale: float, latent_dim: int = 512
               ) -> np.ndarray:
    """Softmax attention of H heads over the selected latent rows.

    q     float64 [H][D]      absorbed query (latent + RoPE part)
    rows  float64 [n][D]      selected latent rows c^KV | k^R
    out   float32 [H][latent_dim] = softmax(sm_scale * q rows^T) rows[:, :latent_dim]
    An empty selection gives zeros.
    """
    q = np.asarray(q, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.float64)
    H = q.shape[0]
    if rows.shape[0] == 0:
        return np.zeros((H, latent_dim), dtype=np.float32)
    logits = float(sm_scale) * (q @ rows.T)            # [H][n]
    mx = np.max(logits, axis=1, keepdims=True)
    p = np.exp(logits - mx)
    p /= np.sum(p, axis=1, keepdims=True)
    return (p @ rows[:, :latent_dim]).astype(np.float32)


# --------------------------------------------------------------------------
# one decode layer, step by step
# --------------------------------------------------------------------------

@dataclass
class StepResult:
    topk: List[List[np.ndarray]]        # [b][m] selected tokens in (score desc, index asc) order
    emit_idx: List[List[np.ndarray]]    # [b][m] emitted order: misses asc, then hits asc
    emit_slot: List[List[np.ndarray]]   # [b][m] slot (hit) or ~slot (miss)
    miss_tok: List[np.ndarray]          # [b] union misses ascending
    miss_slot: List[np.ndarray]         # [b] paired slots
    hits: np.ndarray                    # [B][M]
    misses: np.ndarray                  # [B][M]
    union_size: np.ndarray              # [B]
    out: Optional[np.ndarray] = None    # float32 [B][M][H][512]
    scores: Optional[List[List[np.ndarray]]] = None


class OracleLayer:
    """One decode layer of B requests with an LRU hot pool of C slots each."""

    def __init__(self, T: Sequence[int], C: int, k: int, sm_scale: float, page: int = 64):
        self.T = [int(t) for t in T]
        self.C = int(C)
        self.k = int(k)
        self.sm_scale = float(sm_scale)
        self.page = page
        self.state = [CacheState.empty(t, C) for t in self.T]

    def append(self) -> None:
        """Decode append of one token per request (before the step that sees it)."""
        append_tokens(self.T, self.state)

    def step(self, q_idx: np.ndarray, w: np.ndarray, keys: np.ndarray, scale: np.ndarray,
             q_mla: Optional[np.ndarray], latent: Optional[np.ndarray],
             keep_scores: bool = False) -> StepResult:
        """One decode step.

        q_idx  float64 [B][M][H_I][d_I]
        w      float64 [B][M][H_I]
        keys   float64 [B][T_max][d_I]   (or a callable b -> [T_b][d_I])
        scale  float32 [B][T_max]
        q_mla  float64/bf16-valued [B][M][H][576] or None to skip attention
        latent float64/bf16-valued [B][T_max][576] logical order (or callable b, tokens -> rows)
        """
        B, M = q_idx.shape[0], q_idx.shape[1]
        topk_all, emit_i, emit_s, mt, ms = [], [], [], [], []
        hits = np.zeros((B, M), np.int64)
        misses = np.zeros((B, M), np.int64)
        usz = np.zeros(B, np.int64)
        outs = None
        if q_mla is not None:
            outs = np.zeros((B, M, q_mla.shape[2], 512), dtype=np.float32)
        all_scores = [] if keep_scores else None
        for b in range(B):
            T = self.T[b]
            kb = keys(b) if callable(keys) else keys[b, :T]
            sb = scale[b, :T]
            sel, sc = [], []
            for m in range(M):
                s = score_indexer(q_idx[b, m], w[b, m], kb, sb)
                sc.append(s)
                sel.append(topk_select(s, self.k))
            if keep_scores:
                all_scores.append(sc)
            st = self.state[b]
            r = resolve_union(sel, st.cache_slots)
            resident_before = st.cache_slots.copy()
            victims, _ = lru_update(st, r.union, r.miss_tok)
            hits[b] = r.hits
            misses[b] = r.misses
            usz[b] = r.union.shape[0]
            ei, es = [], []
            for m in range(M):
                srt = np.sort(sel[m])
                was = resident_before[srt] >= 0
                order = np.concatenate([srt[~was], srt[was]])
                slots = st.cache_slots[order].astype(np.int64)
                enc = np.where(resident_before[order] >= 0, slots, ~slots)
                ei.append(order)
                es.append(enc)
                if q_mla is not None:
                    rows = latent(b, order) if callable(latent) else latent[b, order]
                    outs[b, m] = sparse_mla(q_mla[b, m], rows, self.sm_scale)
            topk_all.append(sel)
            emit_i.append(ei)
            emit_s.append(es)
            mt.append(r.miss_tok)
            ms.append(victims)
        return StepResult(topk_all, emit_i, emit_s, mt, ms, hits, misses, usz, outs, all_scores)
