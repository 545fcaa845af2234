"""Runs the CUDA path and the CPU oracle side by side on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

from host_latent_cache_gb300 import ess
from host_latent_cache_gb300 import workloads as W
from host_latent_cache_gb300.session import Session
from oracle import compact_row as X
from oracle import ess_oracle as O

# attention tolerance: max-abs error and relative L2 error against the float64 oracle
ATOL = 2e-2
REL_L2 = 1e-3


def attn_errors(got: np.ndarray, want: np.ndarray):
    d = got.astype(np.float64) - want.astype(np.float64)
    maxabs = float(np.max(np.abs(d))) if d.size else 0.0
    nrm = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(d) / nrm) if nrm > 0 else float(np.linalg.norm(d))
    return maxabs, rel


def assert_attn_close(got, want, what=""):
    maxabs, rel = attn_errors(got, want)
    assert maxabs <= ATOL and rel <= REL_L2, f"{what}: max-abs {maxabs:.3e}, rel-L2 {rel:.3e}"
    return maxabs, rel


class Pair:
    """A GPU session and an oracle per layer, fed identical inputs."""

    def __init__(self, cfg: W.WorkloadConfig, layers: int = 1, miss_mode=ess.ESS_MISS_FUSED,
                 lds=None):
        self.cfg = cfg
        self.lds = lds if lds is not None else [W.gen_layer(cfg, l) for l in range(layers)]
        layers = len(self.lds)
        self.sess = Session(cfg, self.lds, miss_mode)
        self.orc = [O.OracleLayer(ld.T, cfg.C, cfg.k, cfg.sm_scale) for ld in self.lds]
        self.qs = [W.QueryStream(cfg, l) for l in range(layers)]
        self.keys32 = [W.decode_keys(cfg, ld.idx_keys).astype(np.float32) for ld in self.lds]
        self.errs = []
        self.evicted = []   # per step: resident tokens evicted, summed over requests

    def prime_full(self, layer=0, age=8):
        """Both sides start from the same full pool (W.full_pool_state)."""
        ps = W.full_pool_state(self.cfg, self.lds[layer], layer, age)
        self.sess.set_state(layer, ps)
        for b in range(self.cfg.batch):
            Tb = int(self.lds[layer].T[b])
            self.orc[layer].state[b] = O.CacheState(ps.cache_slots[b, :Tb].copy(),
                                                    ps.slot_token[b].copy(),
                                                    ps.last_used[b].copy(), int(ps.step[b]))
        return ps

    def oracle_inputs(self, layer):
        ld = self.lds[layer]
        keys = self.keys32[layer]
        keyf = lambda b: keys[b, : int(ld.T[b])]
        if self.cfg.compact:
            latf = lambda b, order: X.decode_rows(ld.latent_c[b, order])
        else:
            latf = lambda b, order: W.bf16_bits_to_float(ld.latent[b, order]).astype(np.float64)
        return keyf, latf

    def next_inputs(self, layer):
        q, enc, qm = self.qs[layer].next()
        w = W.head_weights(self.cfg, self.lds[layer].w)
        return q, enc, w, qm

    def run_step(self, layer=0, api="calls", check_lists=True, check_state=True,
                 check_out=True, check_scores=False):
        cfg, sess = self.cfg, self.sess
        q, enc, w, qm = self.next_inputs(layer)
        qd, wd, qmd = sess.device_inputs(enc, w, qm)
        if check_scores:
            sc = sess.scores_only(layer, qd, wd).cpu().numpy()
        if api == "calls":
            sess.indexer_topk(layer, qd, wd)
            if sess.ecfg.miss_mode == ess.ESS_MISS_STAGED:
                sess.stage(layer)
            out = sess.attention(layer, qmd)
        else:
            out = sess.step(layer, qd, wd, qmd)
        torch.cuda.synchronize()
        st = sess.poll()
        assert st == ess.ESS_OK, ess.status_string(st)
        keyf, latf = self.oracle_inputs(layer)
        ld = self.lds[layer]
        tok_before = [st_.slot_token.copy() for st_ in self.orc[layer].state]
        r = self.orc[layer].step(q.astype(np.float64), w.astype(np.float64), keyf, ld.idx_scale,
                                 W.bf16_bits_to_float(qm).astype(np.float64), latf,
                                 keep_scores=check_scores)
        self.evicted.append(sum(int(np.count_nonzero(tok_before[b][r.miss_slot[b]] >= 0))
                                for b in range(cfg.batch)))
        if check_scores:
            for b in range(cfg.batch):
                Tb = int(ld.T[b])
                for m in range(cfg.mtp):
                    assert np.array_equal(sc[b, m, :Tb], r.scores[b][m]), f"scores b={b} m={m}"
        if check_lists and api == "calls":
            self.compare_lists(r)
        if check_state:
            self.compare_state(layer)
        if check_out:
            got = out.cpu().numpy()
            self.errs.append(assert_attn_close(got, r.out, "attention"))
        return r

    def compare_lists(self, r):
        cfg, sess = self.cfg, self.sess
        ti = sess.topk_idx.cpu().numpy()
        ts = sess.topk_slot.cpu().numpy()
        nmw = sess.n_miss_way.cpu().numpy()
        mt = sess.miss_tok.cpu().numpy()
        ms = sess.miss_slot.cpu().numpy()
        nm = sess.n_miss.cpu().numpy()
        for b in range(cfg.batch):
            for m in range(cfg.mtp):
                n = len(r.emit_idx[b][m])
                assert np.array_equal(ti[b, m, :n], r.emit_idx[b][m]), f"topk_idx b={b} m={m}"
                assert np.array_equal(ts[b, m, :n], r.emit_slot[b][m]), f"topk_slot b={b} m={m}"
                assert nmw[b, m] == r.misses[b, m], f"n_miss_way b={b} m={m}"
            n = len(r.miss_tok[b])
            assert nm[b] == n, f"n_miss b={b}: {nm[b]} vs {n}"
            assert np.array_equal(mt[b, :n], r.miss_tok[b]), f"miss_tok b={b}"
            assert np.array_equal(ms[b, :n], r.miss_slot[b]), f"miss_slot b={b}"

    def compare_state(self, layer):
        cs, st, lu, sp = self.sess.state(layer)
        ld = self.lds[layer]
        for b in range(self.cfg.batch):
            o = self.orc[layer].state[b]
            Tb = int(ld.T[b])
            assert np.array_equal(cs[b, :Tb], o.cache_slots), f"cache_slots b={b}"
            assert np.all(cs[b, Tb:] == -1)
            assert np.array_equal(st[b], o.slot_token), f"slot_token b={b}"
            assert np.array_equal(lu[b], o.last_used), f"last_used b={b}"
            assert sp[b] == o.step, f"step b={b}"

    def check_pool_rows(self, layer=0):
        """Rows of resident tokens in the pool equal the host master copy."""
        rows = self.sess.pool_rows(layer)
        ld = self.lds[layer]
        for b in range(self.cfg.batch):
            o = self.orc[layer].state[b]
            occ = np.nonzero(o.slot_token >= 0)[0]
            if self.cfg.compact:
                # the widened rows: decoded values, exact in bf16
                dec = X.decode_rows(ld.latent_c[b, o.slot_token[occ]]).astype(np.float32)
                want = W.float_to_bf16_bits(dec).reshape(len(occ), -1)
            else:
                want = ld.latent[b, o.slot_token[occ]]
            assert np.array_equal(rows[b, occ], want), f"pool rows b={b}"

    def close(self):
        self.sess.close()
