"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test pins one oracle function to something other than itself: a
value the pages print (golden fixtures under tests/golden/, each citing
its passage), a hand-derived closed form, an exact-rational or
brute-force computation on tiny inputs, or an invariant the pages state.
"""
import itertools
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

from oracle import ess_oracle as O
from host_latent_cache_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = {}
    multi = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            multi.setdefault(key, []).append(vals)
            rows[key] = vals
    return rows, multi


# --------------------------------------------------------------------------
# byte accounting and the overlap metric (FlashOffloading page, "account first"
# and "decode side (2)")
# --------------------------------------------------------------------------

def test_kv_bytes_per_token_matches_page():
    g, multi = _read_golden("byte_accounting.txt")
    L_kv, D_kv, L_i, D_i, P = (int(g[k][0]) for k in ("L_KV", "D_KV", "L_index", "D_index", "P"))
    kappa = O.kv_bytes_per_token(L_kv, D_kv, L_i, D_i, P)
    assert kappa == 95232
    assert round(kappa / 1000, 2) == float(g["kappa_base_kB"][0])
    assert round(O.kv_bytes_per_token(L_kv, D_kv, 0, 0, P) / 1000, 2) == float(g["kv_part_kB"][0])
    assert round(O.kv_bytes_per_token(0, 0, L_i, D_i, P) / 1000, 2) == float(g["index_part_kB"][0])
    for tokens, gb in multi["total_GB"]:
        assert round(int(tokens) * kappa / 1e9, 2) == float(gb)
    kv_tok = O.kv_bytes_per_token(L_kv, D_kv, 0, 0, P)
    idx_tok = O.kv_bytes_per_token(0, 0, L_i, D_i, P)
    (hot, hot_gb), = multi["hot_kv_GB"]
    (itok, igb), = multi["index_GB"]
    # the page multiplies its rounded per-token figures (89.86 kB, 5.38 kB)
    kv_kb = round(kv_tok / 1000, 2)
    idx_kb = round(idx_tok / 1000, 2)
    assert round(int(hot) * kv_kb * 1e3 / 1e9, 2) == float(hot_gb)
    assert round(int(itok) * idx_kb * 1e3 / 1e9, 2) == float(igb)
    assert abs(int(itok) * idx_tok / 1e9 - float(igb)) < 0.01
    # the decode residency formula with one layer, b = 0 and only KV data
    assert O.decode_residency_bytes(1, int(hot), 0, kv_tok) == int(hot) * kv_tok
    assert O.decode_residency_bytes(2, 10, 3, 7, 1, 2, 3) == 2 * 16 * 7 + 6


def test_overlap_ratio_matches_page():
    _, multi = _read_golden("byte_accounting.txt")
    (tc, ts, tf, r), = multi["overlap_us"]
    assert round(O.overlap_ratio(float(tc), float(ts), float(tf)), 2) == float(r)
    assert O.overlap_ratio(10.0, 5.0, 5.0) == 1.0     # copy fully hidden
    assert O.overlap_ratio(10.0, 5.0, 15.0) == 0.0    # no overlap at all


# --------------------------------------------------------------------------
# indexer score
# --------------------------------------------------------------------------

def test_score_hand_computed():
    # two heads, two dims, three positions; derived by hand:
    # t0: dots (2.5, 0)  -> 0.5*2.5 + 0.25*0 = 1.25, times scale 1   = 1.25
    # t1: dots (-0.375, -2.125) -> both clipped by ReLU             = 0
    # t2: dots (-3, 3)   -> 0.25*3 = 0.75, times scale 0.5          = 0.375
    q = np.array([[1.0, 0.5], [-1.0, 2.0]])
    w = np.array([0.5, 0.25])
    keys = np.array([[2.0, 1.0], [0.125, -1.0], [-3.0, 0.0]])
    scale = np.array([1.0, 2.0, 0.5], dtype=np.float32)
    s = O.score_indexer(q, w, keys, scale)
    assert s.dtype == np.float32
    assert s.tolist() == [1.25, 0.0, 0.375]
    assert not np.signbit(s[1])


def test_score_scale_is_one_rounding_after_head_sum():
    # inner = 3 exactly; 3 * fp32(1/3) = 1.00000002980... rounds to 1.0 in fp32
    q = np.array([[1.0]])
    w = np.array([1.0])
    keys = np.array([[3.0]])
    third = np.float32(1.0 / 3.0)
    s = O.score_indexer(q, w, keys, np.array([third], dtype=np.float32))
    assert s[0] == np.float32(1.0)
    # scale applied per head inside the ReLU would round twice; after the sum once
    q2 = np.array([[1.0], [1.0]])
    w2 = np.array([0.5, 0.5])
    keys2 = np.array([[3.0]])
    assert O.score_indexer(q2, w2, keys2, np.array([third], np.float32))[0] == np.float32(1.0)


def test_score_exact_rational_brute_force():
    rng = np.random.default_rng(5)
    lv, _ = W.key_levels()
    for _ in range(20):
        H, d, T = 3, 5, 7
        q = rng.integers(-16, 17, size=(H, d)) / 8.0
        w = rng.integers(0, 64, size=H) / 64.0
        keys = lv[rng.integers(0, len(lv), size=(T, d))]
        scale = rng.random(T).astype(np.float32) + np.float32(0.01)
        got = O.score_indexer(q, w, keys, scale)
        for t in range(T):
            inner = Fraction(0)
            for h in range(H):
                dot = sum(Fraction(q[h, j]) * Fraction(keys[t, j]) for j in range(d))
                inner += Fraction(w[h]) * max(dot, Fraction(0))
            exact = inner * Fraction(float(scale[t]))
            want = np.float32(float(exact))   # float() of a Fraction is correctly rounded
            # float(exact) rounds to double first; the exact value has at most 48
            # significant bits here, so the double is exact and the fp32 rounding single
            assert got[t] == want


def test_score_rejects_values_outside_exact_bound():
    # two heads at the largest dot (128 * 2 * 15 = 3840) sum to 7560 > 4096
    q = np.array([[2.0] * 128, [2.0] * 128])
    keys = np.array([[15.0] * 128])
    with pytest.raises(ValueError):
        O.score_indexer(q, np.array([0.984375, 0.984375]), keys, np.ones(1, np.float32))
    assert O.score_indexer(q[:1], np.array([0.984375]), keys, np.ones(1, np.float32))[0] == 3780.0


def test_score_generated_data_within_exact_bound():
    cfg = W.tiny().replace(T=512)
    ld = W.gen_layer(cfg, want_latent=False)
    qs = W.QueryStream(cfg)
    q, _, _ = qs.next()
    keys = W.decode_keys(cfg, ld.idx_keys[0])
    s = O.score_indexer(q[0, 0], ld.w[0], keys, ld.idx_scale[0])
    assert np.all(s >= 0)
    assert np.all(np.isfinite(s))


# --------------------------------------------------------------------------
# top-k
# --------------------------------------------------------------------------

def _topk_by_rank_counting(scores, k):
    """Independent definition: t is selected iff fewer than k positions beat it,
    u beating t when s_u > s_t, or s_u == s_t and u < t; order by that count."""
    T = len(scores)
    beat = []
    for t in range(T):
        c = sum(1 for u in range(T)
                if scores[u] > scores[t] or (scores[u] == scores[t] and u < t))
        beat.append(c)
    sel = [t for t in range(T) if beat[t] < k]
    return sorted(sel, key=lambda t: beat[t])


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(7)
    for _ in range(300):
        T = int(rng.integers(1, 12))
        k = int(rng.integers(0, T + 3))
        s = rng.integers(0, 3, size=T).astype(np.float32)
        got = O.topk_select(s, k).tolist()
        assert got == _topk_by_rank_counting(s.tolist(), k)


def test_topk_worked_example_ordering():
    g, _ = _read_golden("fig4_worked_example.txt")
    T = int(g["T"][0])
    top3 = [int(x) for x in g["top3"]]
    s = np.zeros(T, dtype=np.float32)
    s[top3[0]], s[top3[1]], s[top3[2]] = 3.0, 2.0, 1.0
    assert O.topk_select(s, 3).tolist() == top3


def test_topk_lower_index_wins_ties():
    s = np.array([1, 5, 5, 5, 0], dtype=np.float32)
    assert O.topk_select(s, 2).tolist() == [1, 2]
    assert O.topk_select(s, 10).tolist() == [1, 2, 3, 0, 4]


# --------------------------------------------------------------------------
# resolve + union + LRU (worked example and Figure 4)
# --------------------------------------------------------------------------

def _fig4_state():
    g, _ = _read_golden("fig4_worked_example.txt")
    T, C = int(g["T"][0]), int(g["C"][0])
    cs = np.array([int(x) for x in g["cache_slots"]], dtype=np.int32)
    st = O.CacheState.empty(T, C)
    st.cache_slots[:] = cs
    for t, s in enumerate(cs):
        if s >= 0:
            st.slot_token[s] = t
    return g, st


def test_resolve_worked_example():
    g, st = _fig4_state()
    top3 = np.array([int(x) for x in g["top3"]])
    assert st.cache_slots[top3].tolist() == [int(x) for x in g["top3_slots"]]
    r = O.resolve_union([top3], st.cache_slots)
    assert r.hits == [1] and r.misses == [2]
    assert r.miss_tok.tolist() == [int(x) for x in g["miss"]]
    assert r.union.tolist() == sorted(top3.tolist())


def test_lru_figure4_final_state():
    # The page gives no history; a history in which slots 3 and 5 are the
    # least recently used (3 older than 5) reproduces Figure 4.
    g, st = _fig4_state()
    st.last_used[:] = [5, 5, 5, 1, 5, 2, 5, 5]
    st.step = 6
    before = st.cache_slots.copy()
    top3 = np.array([int(x) for x in g["top3"]])
    r = O.resolve_union([top3], st.cache_slots)
    victims, evicted = O.lru_update(st, r.union, r.miss_tok)
    assert victims.tolist() == [int(x) for x in g["victim_slots"]]
    assert evicted.tolist() == [18, 19]
    assert st.cache_slots[8] == 3 and st.cache_slots[17] == 5
    assert st.cache_slots[18] == -1 and st.cache_slots[19] == -1
    others = [t for t in range(20) if t not in (8, 17, 18, 19)]
    assert st.cache_slots[others].tolist() == before[others].tolist()
    assert st.slot_token[3] == 8 and st.slot_token[5] == 17
    assert st.last_used[7] == 6            # the hit (token 4 in slot 7) was stamped
    assert st.last_used[3] == 6 and st.last_used[5] == 6
    assert st.step == 7
    # DRAM block of each miss (blocks of 4 tokens, 1-based) as drawn in Figure 4
    assert [t // 4 + 1 for t in r.miss_tok.tolist()] == [int(x) for x in g["miss_dram_block_1based"]]


def _check_bijection(st):
    res = np.nonzero(st.cache_slots >= 0)[0]
    assert np.array_equal(st.slot_token[st.cache_slots[res]], res)
    occ = np.nonzero(st.slot_token >= 0)[0]
    assert np.array_equal(st.cache_slots[st.slot_token[occ]], occ)
    assert len(occ) == len(res) <= st.slot_token.shape[0]


def test_lru_invariants_random_sequence():
    rng = np.random.default_rng(11)
    T, C, k = 200, 48, 16
    st = O.CacheState.empty(T, C)
    ever = set()
    for step in range(60):
        ways = [rng.choice(T, size=k, replace=False) for _ in range(2)]
        before = st.copy()
        r = O.resolve_union(ways, st.cache_slots)
        for m in range(2):
            assert r.hits[m] + r.misses[m] == k
        assert len(r.miss_tok) <= sum(r.misses)
        victims, evicted = O.lru_update(st, r.union, r.miss_tok)
        _check_bijection(st)
        ever |= set(r.union.tolist())
        occ = int(np.count_nonzero(st.slot_token >= 0))
        assert occ == min(C, len(ever)) or occ == len(set(np.nonzero(st.cache_slots >= 0)[0]))
        # every union token is resident after the step
        assert np.all(st.cache_slots[r.union] >= 0)
        # hits are never evicted in the step that uses them
        hit_slots = before.cache_slots[r.union][before.cache_slots[r.union] >= 0]
        assert not set(victims.tolist()) & set(hit_slots.tolist())
        # loads equal evictions once the pool is full: occupancy is unchanged
        if np.count_nonzero(before.slot_token >= 0) == C:
            assert np.count_nonzero(st.slot_token >= 0) == C
            assert np.all(evicted >= 0)
        # LRU: no victim was used more recently than a surviving non-union slot
        used = before.last_used.copy()
        used[hit_slots] = before.step
        vset = set(victims.tolist())
        surv = [s for s in range(C) if s not in vset and s not in set(hit_slots.tolist())]
        if len(victims) and surv:
            assert max(used[v] for v in victims) <= min(used[s] for s in surv)
        assert st.step == step + 1


def test_lru_no_eviction_when_pool_holds_everything():
    rng = np.random.default_rng(3)
    T, k = 64, 8
    st = O.CacheState.empty(T, T)
    for _ in range(40):
        sel = rng.choice(T, size=k, replace=False)
        r = O.resolve_union([sel], st.cache_slots)
        _, evicted = O.lru_update(st, r.union, r.miss_tok)
        assert np.all(evicted == -1)


def test_lru_first_fill_uses_empty_slots_in_order():
    st = O.CacheState.empty(10, 6)
    union = np.array([2, 5, 7])
    r = O.resolve_union([union], st.cache_slots)
    victims, evicted = O.lru_update(st, r.union, r.miss_tok)
    assert victims.tolist() == [0, 1, 2]
    assert evicted.tolist() == [-1, -1, -1]
    assert st.cache_slots[[2, 5, 7]].tolist() == [0, 1, 2]


def test_lru_capacity_error():
    st = O.CacheState.empty(10, 2)
    with pytest.raises(O.CapacityError):
        O.lru_update(st, np.array([1, 2, 3]), np.array([1, 2, 3]))


# --------------------------------------------------------------------------
# sparse MLA attention
# --------------------------------------------------------------------------

def test_mla_all_positions_is_dense_softmax_attention():
    rng = np.random.default_rng(1)
    H, n, D = 4, 9, 576
    q = rng.standard_normal((H, D)) * 0.5
    rows = rng.standard_normal((n, D)) * 0.5
    sc = 1.0 / 24.0
    got = O.sparse_mla(q, rows, sc)
    want = scipy.special.softmax(sc * q @ rows.T, axis=1) @ rows[:, :512]
    np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-7)


def test_mla_single_row_and_uniform_logits():
    rng = np.random.default_rng(2)
    rows = rng.standard_normal((5, 576))
    one = O.sparse_mla(rng.standard_normal((3, 576)), rows[:1], 0.1)
    np.testing.assert_allclose(one, np.repeat(rows[:1, :512], 3, 0).astype(np.float32), rtol=1e-7)
    flat = O.sparse_mla(np.zeros((2, 576)), rows, 0.1)
    np.testing.assert_allclose(flat, np.repeat(rows[:, :512].mean(0, keepdims=True), 2, 0),
                               rtol=1e-6, atol=1e-7)


def test_mla_rope_part_enters_logits_only():
    # two rows that differ only in the RoPE part: logits a = 2*sc, b = 0
    rows = np.zeros((2, 576))
    rows[0, :512] = 1.0
    rows[1, :512] = -1.0
    rows[0, 512] = 2.0
    q = np.zeros((1, 576))
    q[0, 512] = 1.0
    sc = 0.5
    got = O.sparse_mla(q, rows, sc)
    p0 = 1.0 / (1.0 + np.exp(-(2.0 * sc)))
    np.testing.assert_allclose(got[0], np.full(512, p0 - (1 - p0)), rtol=1e-7)
    assert got.shape == (1, 512)


def test_mla_permutation_invariance_and_empty():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((3, 576))
    rows = rng.standard_normal((17, 576))
    a = O.sparse_mla(q, rows, 0.05)
    b = O.sparse_mla(q, rows[rng.permutation(17)], 0.05)
    np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-7)
    assert np.all(O.sparse_mla(q, rows[:0], 0.05) == 0)


# --------------------------------------------------------------------------
# whole layer
# --------------------------------------------------------------------------

def _run_layer(cfg, steps, C=None):
    ld = W.gen_layer(cfg)
    keys = W.decode_keys(cfg, ld.idx_keys)
    lat = W.bf16_bits_to_float(ld.latent).astype(np.float64)
    lay = O.OracleLayer(ld.T, C or cfg.C, cfg.k, cfg.sm_scale)
    qs = W.QueryStream(cfg)
    res = []
    for _ in range(steps):
        q, _, qm = qs.next()
        w = W.head_weights(cfg, ld.w)
        r = lay.step(q, w, keys, ld.idx_scale, W.bf16_bits_to_float(qm).astype(np.float64), lat)
        res.append((r, q, qm))
    return ld, lay, res, keys, lat


def test_layer_losslessness_and_emitted_order():
    cfg = W.tiny().replace(T=1024, k=64, C=1024)
    ld, lay, res, keys, lat = _run_layer(cfg, 3)
    for r, q, qm in res:
        for m in range(cfg.mtp):
            sel = r.topk[0][m]
            dense = O.sparse_mla(W.bf16_bits_to_float(qm[0, m]).astype(np.float64), lat[0, sel],
                                 cfg.sm_scale)
            np.testing.assert_allclose(r.out[0, m], dense, rtol=1e-6, atol=1e-7)
            emit = r.emit_idx[0][m]
            assert sorted(emit.tolist()) == sorted(sel.tolist())
            nmiss = int(r.misses[0, m])
            assert np.all(r.emit_slot[0][m][:nmiss] < 0) and np.all(r.emit_slot[0][m][nmiss:] >= 0)
            assert np.all(np.diff(emit[:nmiss]) > 0) and np.all(np.diff(emit[nmiss:]) > 0)
            slots = np.where(r.emit_slot[0][m] < 0, ~r.emit_slot[0][m], r.emit_slot[0][m])
            assert np.array_equal(lay.state[0].cache_slots[emit], slots)
    # C >= T: nothing is ever evicted and the pool holds every token selected so far
    seen = set()
    for r, _, _ in res:
        seen |= set(r.topk[0][0].tolist())
    assert np.count_nonzero(lay.state[0].cache_slots >= 0) == len(seen)


def test_layer_first_step_is_all_misses():
    cfg = W.tiny().replace(T=2048, k=128, C=512)
    _, lay, res, _, _ = _run_layer(cfg, 2)
    r0 = res[0][0]
    assert r0.hits[0, 0] == 0 and r0.misses[0, 0] == cfg.k
    assert r0.miss_slot[0].tolist() == list(range(cfg.k))


def test_generator_contract_and_determinism():
    lv, codes = W.key_levels()
    assert len(lv) == 79 and lv.min() == -15 and lv.max() == 15
    assert np.all(lv * 8 == np.round(lv * 8))
    tab = W.e4m3_decode_table()
    assert np.array_equal(tab[codes], lv)
    assert np.array_equal(W.bf16_bits_to_float(W.float_to_bf16_bits(lv.astype(np.float32))), lv)
    cfg = W.long_128k().replace(batch=1, T=256)
    a = W.gen_layer(cfg)
    b = W.gen_layer(cfg)
    assert np.array_equal(a.idx_keys, b.idx_keys) and np.array_equal(a.host_latent, b.host_latent)
    vals = W.decode_keys(cfg, a.idx_keys)
    assert set(np.unique(vals).tolist()) <= set(lv.tolist())
    # host layout is the logical latent behind the page table
    t = np.arange(cfg.T)
    phys = a.page_table[0][t // 64] * 64 + t % 64
    assert np.array_equal(a.host_latent[0][phys], a.latent[0])
    qs = W.QueryStream(cfg)
    q, enc, qm = qs.next()
    assert np.max(np.abs(q)) == 2.0 and np.all(q * 8 == np.round(q * 8))


def test_mla_large_logits_closed_form():
    # logits 1000 and 999 (exp overflows without the max shift): weights are
    # 1/(1+e^-1) and e^-1/(1+e^-1)
    rows = np.zeros((2, 576))
    rows[0, :512] = 3.0
    rows[1, :512] = -1.0
    rows[0, 512] = 1000.0
    rows[1, 512] = 999.0
    q = np.zeros((1, 576))
    q[0, 512] = 1.0
    got = O.sparse_mla(q, rows, 1.0)
    a = 1.0 / (1.0 + np.exp(-1.0))
    np.testing.assert_allclose(got[0], np.full(512, 3.0 * a - (1.0 - a)), rtol=1e-7)


# --------------------------------------------------------------------------
# decode append (FlashOffloading page, section "architecture" and Figure 2:
# new KV goes to tail blocks beside the hot cache)
# --------------------------------------------------------------------------

def _append_run(T0, C, k, grow, seed):
    """A one-request bf16 layer that appends a token before each of `grow`
    steps; returns the layer data, the keys and latent of every token, the
    oracle layer and each step's (result, q_mla)."""
    cfg = W.tiny().replace(T=T0, k=k, C=C, grow=grow, seed=seed)
    ld = W.gen_layer(cfg)
    keys = W.decode_keys(cfg, ld.idx_keys)
    keys[:, T0:T0 + grow] = W.decode_keys(cfg, ld.app_keys)
    scale = ld.idx_scale.copy()
    scale[:, T0:T0 + grow] = ld.app_scale
    lat = W.bf16_bits_to_float(ld.latent).astype(np.float64)
    lay = O.OracleLayer(ld.T, C, k, cfg.sm_scale)
    qs = W.QueryStream(cfg)
    res = []
    for _ in range(grow):
        lay.append()
        q, _, qm = qs.next()
        r = lay.step(q, W.head_weights(cfg, ld.w), keys, scale,
                     W.bf16_bits_to_float(qm).astype(np.float64), lat)
        res.append((r, W.bf16_bits_to_float(qm).astype(np.float64)))
    return cfg, ld, lat, lay, res


def test_append_every_token_attended_when_k_covers_the_context():
    # k >= T: each step selects every token, the newest included, and the
    # output is dense softmax attention over all of them; the newest token
    # is the one miss of its step (it is not in the hot cache yet)
    T0, grow = 60, 12
    cfg, ld, lat, lay, res = _append_run(T0, C=256, k=256, grow=grow, seed=31)
    for i, (r, qm) in enumerate(res):
        T = T0 + 1 + i
        assert sorted(r.topk[0][0].tolist()) == list(range(T))
        want = scipy.special.softmax(cfg.sm_scale * qm[0, 0] @ lat[0, :T].T, axis=1) @ lat[0, :T, :512]
        np.testing.assert_allclose(r.out[0, 0], want, rtol=1e-6, atol=1e-7)
        if i > 0:
            assert r.misses[0, 0] == 1 and r.miss_tok[0].tolist() == [T - 1]
    assert lay.T == [T0 + grow]
    assert lay.state[0].cache_slots.shape == (T0 + grow,)


def test_append_keeps_the_cache_maps_consistent():
    # a small pool under appends: cache_slots and slot_token stay inverse
    # maps, the pool stays full once filled, and a selected token is resident
    _, _, _, lay, res = _append_run(500, C=96, k=64, grow=40, seed=32)
    st = lay.state[0]
    _check_bijection(st)
    assert np.all(st.cache_slots[res[-1][0].topk[0][0]] >= 0)
    assert np.count_nonzero(st.slot_token >= 0) == 96
    assert sum(int(r.miss_tok[0].shape[0]) for r, _ in res) >= 96


def test_generator_append_inputs_continue_the_same_streams():
    # the rows a decode append feeds in are the rows a longer context would
    # have had: keys, scales and latent come from the same seeded streams,
    # and the bound cache and host copy start empty past T_b
    cfg = W.long_128k().replace(batch=2, T=300, T_per_req=[300, 170], grow=40)
    ld = W.gen_layer(cfg)
    full = W.gen_layer(cfg.replace(T_per_req=[340, 210], grow=0))
    assert W.t_max_of(cfg) == W.t_max_of(cfg.replace(T_per_req=[340, 210], grow=0)) == 384
    for b, T in enumerate([300, 170]):
        assert np.array_equal(ld.app_keys[b], full.idx_keys[b, T:T + 40])
        assert np.array_equal(ld.app_scale[b], full.idx_scale[b, T:T + 40])
        assert np.all(ld.idx_keys[b, T:] == 0) and np.all(ld.idx_scale[b, T:] == 1.0)
        assert np.array_equal(ld.latent[b], full.latent[b])
        t = np.arange(W.t_max_of(cfg))
        phys = ld.page_table[b][t // cfg.page] * cfg.page + t % cfg.page
        assert np.array_equal(ld.host_latent[b][phys[:T]], ld.latent[b, :T])
        assert np.all(ld.host_latent[b][phys[T:]] == 0)
        lat, key, sc = W.appended_token(cfg, ld, 7)
        assert np.array_equal(lat[b], full.latent[b, T + 7]) and np.array_equal(key[b], full.idx_keys[b, T + 7])
        assert sc[b] == full.idx_scale[b, T + 7]
