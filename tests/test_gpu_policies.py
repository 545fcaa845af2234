"""Eviction orders in the decode kernels against the oracle's replay.

The FlashOffloading analysis (section "evaluation", the decode ablation and
its Figure 8) replays one access sequence with Random, LRU, Score and LIM
eviction.  ess_pool_set_eviction makes the selection kernels use each order;
here every step's lists (misses first, their paired slots), the miss union,
the copy triples and the whole cache state are compared bit for bit with
oracle/eviction_replay.py driven by the same selections, over enough steps
that full pools evict resident tokens, with ties in the scores so that the
slot tie-break decides some victims.
"""
import numpy as np
import pytest
import torch

from host_latent_cache_gb300 import ess
from host_latent_cache_gb300 import workloads as W
from host_latent_cache_gb300.session import Session
from oracle import ess_oracle as O
from oracle import eviction_replay as R

pytestmark = pytest.mark.gpu

POLICY = {"lru": ess.ESS_EVICT_LRU, "random": ess.ESS_EVICT_RANDOM,
          "score": ess.ESS_EVICT_SCORE, "lim": ess.ESS_EVICT_LIM}
SEED = 0x5EED1234ABCD


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_latent_cache_gb300 import build as B
    B.build()
    assert torch.cuda.is_available()
    ess.load()


def _scores(rng, B, M, Tm, levels):
    """Scores on a coarse grid of `levels` values, so that many tokens tie (at
    the top-k cutoff and among the Score order's candidates); None for
    continuous scores."""
    if levels is None:
        return rng.random((B, M, Tm), dtype=np.float32)
    return rng.integers(0, levels, size=(B, M, Tm)).astype(np.float32) / 8.0


class _Replay:
    """The oracle replay of one request, plus the emitted lists of a step."""

    def __init__(self, T, C):
        self.T = T
        self.st = R.ReplayState.empty(C)

    def step(self, sc_bm, k, policy, key):
        M = sc_bm.shape[0]
        sel = [O.topk_select(sc_bm[m, :self.T], k) for m in range(M)]
        union = np.unique(np.concatenate(sel)) if M else np.zeros(0, np.int64)
        before = dict(self.st.slot_of)
        best = np.max(sc_bm[:, :self.T].astype(np.float64), axis=0)
        ts = {t: float(best[t]) for t in self.st.slot_of}
        miss = R.replay_step(self.st, union, policy, ts, key)
        victims = np.array([self.st.slot_of[int(t)] for t in miss], dtype=np.int64)
        emit = []
        for m in range(M):
            srt = np.sort(sel[m])
            was = np.array([int(t) in before for t in srt], dtype=bool)
            order = np.concatenate([srt[~was], srt[was]])
            slots = np.array([self.st.slot_of[int(t)] for t in order], dtype=np.int64)
            enc = np.where(np.array([int(t) in before for t in order], dtype=bool), slots, ~slots)
            emit.append((order, enc, int(np.count_nonzero(~was))))
        return miss, victims, emit

    def cache_slots(self):
        cs = np.full(self.T, -1, np.int64)
        for t, v in self.st.slot_of.items():
            cs[t] = v
        return cs


def _run(policies, T_list, k, C, M, steps_each, seed, levels=24):
    cfg = W.multilayer().replace(layers=1, batch=len(T_list), T=max(max(T_list), 64),
                                 T_per_req=T_list, k=k, C=C, mtp=M, mla_heads=16)
    ld = W.gen_layer(cfg)
    sess = Session(cfg, [ld])
    reps = [_Replay(int(ld.T[b]), C) for b in range(cfg.batch)]
    rng = np.random.default_rng(seed)
    Tm = W.t_max_of(cfg)
    s = 0
    evicted = 0
    for pol in policies:
        ess.ess_pool_set_eviction(sess.pool, POLICY[pol], SEED)
        for _ in range(steps_each):
            sc = _scores(rng, cfg.batch, M, Tm, levels)
            sess.select(0, torch.from_numpy(sc).cuda())
            torch.cuda.synchronize()
            assert sess.poll() == ess.ESS_OK, (pol, s)
            ti = sess.topk_idx.cpu().numpy()
            tsl = sess.topk_slot.cpu().numpy()
            nmw = sess.n_miss_way.cpu().numpy()
            mt = sess.miss_tok.cpu().numpy()
            msl = sess.miss_slot.cpu().numpy()
            nm = sess.n_miss.cpu().numpy()
            cs, stok, lu, sp = sess.state(0)
            for b in range(cfg.batch):
                rp = reps[b]
                tok_before = rp.st.slot_token.copy()
                miss, victims, emit = rp.step(sc[b], k, pol, R.random_key(SEED, b, s))
                evicted += int(np.count_nonzero(tok_before[victims] >= 0)) if len(victims) else 0
                where = f"{pol} step {s} b={b}"
                assert nm[b] == len(miss), where
                assert np.array_equal(mt[b, :nm[b]], miss), where
                assert np.array_equal(msl[b, :nm[b]], victims), where
                for m in range(M):
                    order, enc, nmiss = emit[m]
                    n = len(order)
                    assert np.array_equal(ti[b, m, :n], order), where
                    assert np.array_equal(tsl[b, m, :n], enc), where
                    assert nmw[b, m] == nmiss, where
                Tb = int(ld.T[b])
                assert np.array_equal(cs[b, :Tb], rp.cache_slots()), where
                assert np.array_equal(stok[b], rp.st.slot_token), where
                assert np.array_equal(lu[b], rp.st.last_used), where
                assert sp[b] == rp.st.step, where
            s += 1
    sess.close()
    return evicted


@pytest.mark.parametrize("policy", ["lru", "random", "score", "lim"])
def test_policy_matches_replay_two_ways(policy):
    evicted = _run([policy], [3000, 1200], k=128, C=300, M=2, steps_each=8, seed=11)
    assert evicted > 0


@pytest.mark.parametrize("policy", ["random", "score", "lim"])
def test_policy_matches_replay_one_way_large_pool(policy):
    # 2048 new selections a step fill the 4096 slots after two steps
    evicted = _run([policy], [65536], k=2048, C=4096, M=1, steps_each=6, seed=12)
    assert evicted > 0


def test_score_keys_read_again_when_they_do_not_fit():
    # 40960 slots: the Score keys no longer fit the victim kernel's shared
    # memory beside the classes and the sort buffer, so each pass reads them
    # from the scores again (continuous scores: about 4096 new tokens a step
    # fill the pool after ten steps)
    evicted = _run(["score"], [131072], k=2048, C=40960, M=2, steps_each=14, seed=14,
                   levels=None)
    assert evicted > 0


def test_switching_policies_keeps_state_in_step():
    # Score, then LRU again (its order list rebuilt from the stamps), then LIM
    evicted = _run(["score", "lru", "lim"], [2500, 900, 64], k=96, C=128, M=1, steps_each=4,
                   seed=13)
    assert evicted > 0
