"""Decode append on the GPU against the oracle.

Before each step every request appends one token: its latent row goes to the
device ring, its key to the indexer cache, and a completed page goes back to
the host copy.  Then the layer runs.  The selection lists, the cache state
and the attention output must match the oracle, which sees T_b grow by one
per step (FlashOffloading page, section "architecture" and Figure 2: two
tail blocks take the new KV beside the hot cache).  The runs are long enough
that appended tokens are loaded into the pool both from the ring and, after
their page has left it, from the host copy; the tests count both cases from
the oracle's miss lists.
"""
import numpy as np
import pytest
import torch

from host_latent_cache_gb300 import ess
from host_latent_cache_gb300 import workloads as W
from host_latent_cache_gb300.session import Session
from oracle import ess_oracle as O
from tests.parity_util import Pair, assert_attn_close

pytestmark = pytest.mark.gpu


class AppendRun:
    """A GPU session and the oracle, fed the same appends and queries."""

    def __init__(self, cfg, miss_mode=ess.ESS_MISS_FUSED):
        self.cfg = cfg
        self.ld = ld = W.gen_layer(cfg)
        self.sess = Session(cfg, [ld], miss_mode)
        self.orc = O.OracleLayer(ld.T, cfg.C, cfg.k, cfg.sm_scale)
        self.qs = W.QueryStream(cfg)
        # the oracle reads every token's key, latent and scale from full arrays
        self.keys = W.decode_keys(cfg, ld.idx_keys)
        self.scale = ld.idx_scale.copy()
        for b in range(cfg.batch):
            T = int(ld.T[b])
            self.keys[b, T:T + cfg.grow] = W.decode_keys(cfg, ld.app_keys[b])
            self.scale[b, T:T + cfg.grow] = ld.app_scale[b]
        self.lat = W.bf16_bits_to_float(ld.latent).astype(np.float64)
        self.n = 0
        self.from_ring = 0
        self.from_host = 0

    def append(self):
        self.sess.append(0, *self.sess.append_inputs(*W.appended_token(self.cfg, self.ld, self.n)))
        self.orc.append()
        self.n += 1

    def step(self, api):
        cfg, sess = self.cfg, self.sess
        q, enc, qm = self.qs.next()
        w = W.head_weights(cfg, self.ld.w)
        qd, wd, qmd = sess.device_inputs(enc, w, qm)
        if api == "calls":
            sess.indexer_topk(0, qd, wd)
            if sess.ecfg.miss_mode == ess.ESS_MISS_STAGED:
                sess.stage(0)
            out = sess.attention(0, qmd)
        else:
            out = sess.step(0, qd, wd, qmd)
        torch.cuda.synchronize()
        st = sess.poll()
        assert st == ess.ESS_OK, ess.status_string(st)
        r = self.orc.step(q.astype(np.float64), w.astype(np.float64), self.keys, self.scale,
                          W.bf16_bits_to_float(qm).astype(np.float64), self.lat)
        if api == "calls":
            Pair.compare_lists(self, r)
        self.compare_state()
        assert_attn_close(out.cpu().numpy(), r.out, f"attention after {self.n} appends")
        for b in range(cfg.batch):
            T0, Tb = int(self.ld.T[b]), self.orc.T[b]
            lo = max(T0, (Tb // cfg.page - 1) * cfg.page)   # the ring's window
            new = r.miss_tok[b][r.miss_tok[b] >= T0]
            self.from_ring += int(np.count_nonzero(new >= lo))
            self.from_host += int(np.count_nonzero(new < lo))

    def compare_state(self):
        cs, st, lu, sp = self.sess.state(0)
        for b in range(self.cfg.batch):
            o = self.orc.state[b]
            Tb = self.orc.T[b]
            assert np.array_equal(cs[b, :Tb], o.cache_slots), f"cache_slots b={b}"
            assert np.all(cs[b, Tb:] == -1)
            assert np.array_equal(st[b], o.slot_token), f"slot_token b={b}"
            assert np.array_equal(lu[b], o.last_used), f"last_used b={b}"
            assert sp[b] == o.step, f"step b={b}"

    def check_written_rows(self):
        """Appended keys sit in the indexer cache; appended rows of complete
        pages sit in the host copy (byte for byte); the newest, incomplete
        page is not written back yet."""
        cfg, ld = self.cfg, self.ld
        keys = self.sess.keys[0].cpu().numpy()
        scale = self.sess.scale[0].cpu().numpy()
        host = self.sess.host[0].array
        for b in range(cfg.batch):
            T0 = int(ld.T[b])
            Tn = T0 + self.n
            assert np.array_equal(keys[b, T0:Tn], ld.app_keys[b, :self.n]), f"keys b={b}"
            assert np.array_equal(scale[b, T0:Tn], ld.app_scale[b, :self.n]), f"scale b={b}"
            t = np.arange(Tn)
            phys = ld.page_table[b][t // cfg.page] * cfg.page + t % cfg.page
            done = max(T0, (Tn // cfg.page) * cfg.page)    # appended tokens below this are home
            assert np.array_equal(host[b][phys[:done]], ld.latent[b, :done]), f"host rows b={b}"
            assert np.all(host[b][phys[done:Tn]] == 0), f"incomplete page b={b}"

    def close(self):
        self.sess.close()


def _run(cfg, miss_mode=ess.ESS_MISS_FUSED, steps=None):
    run = AppendRun(cfg, miss_mode)
    try:
        for i in range(steps or cfg.grow):
            run.append()
            run.step("calls" if i % 2 else "step")
        run.check_written_rows()
        assert run.from_ring > 0 and run.from_host > 0, (run.from_ring, run.from_host)
    finally:
        run.close()


def test_append_parity_bf16_ragged():
    _run(W.append_ragged())


def test_append_parity_fp8_128_heads():
    _run(W.append_fp8())


def test_append_parity_staged_misses():
    _run(W.append_ragged(), ess.ESS_MISS_STAGED)


def test_append_at_capacity_is_refused():
    # one request 63 tokens short of max_T after rounding: 63 appends fit,
    # the 64th returns ESS_ERR_CAPACITY without touching the layer
    cfg = W.append_ragged().replace(T_per_req=None, batch=1, T=4033, grow=63)
    run = AppendRun(cfg)
    try:
        assert W.t_max_of(cfg) == 4096
        for _ in range(63):
            run.append()
        lat, key, sc = run.sess.append_inputs(*W.appended_token(cfg, run.ld, 62))
        with pytest.raises(ess.EssError) as e:
            run.sess.append(0, lat, key, sc)
        assert e.value.code == ess.ESS_ERR_CAPACITY
        run.step("calls")
        run.check_written_rows()
    finally:
        run.close()
