"""The allocation-free selection entry point against the ordinary one.

ess_select_manage_noalloc takes its selection scratch from a fixed array in
the library instead of the pool's workspace.  Two pools built from identical
data are driven with the same scores, one through each entry point, for two
steps in a row; every list and the whole cache state must agree exactly.  The
file is named to be collected last, so that it runs both after the other GPU
tests and, when run on its own, in a fresh process.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from host_latent_cache_gb300 import ess
from host_latent_cache_gb300 import workloads as W
from host_latent_cache_gb300.session import Session

STATIC_SCRATCH_BYTES = 2 << 20


def _scratch_need(cfg):
    bm = cfg.batch * cfg.mtp
    up = lambda x: (x + 255) // 256 * 256
    return up(bm * 4096 * 4) + up(bm * cfg.k * 4)


def _lists(s: Session):
    return [t.cpu().numpy().copy() for t in (s.topk_idx, s.topk_slot, s.n_miss_way, s.miss_tok,
                                             s.miss_slot, s.n_miss)]


def _noalloc(s: Session, layer, scores):
    ess.ess_select_manage_noalloc(s.pool, layer, scores, s.topk_idx, s.topk_slot, s.n_miss_way,
                                  s.miss_tok, s.miss_slot, s.n_miss)


def _compare(a: Session, b: Session, step):
    names = ("topk_idx", "topk_slot", "n_miss_way", "miss_tok", "miss_slot", "n_miss")
    la, lb = _lists(a), _lists(b)
    cfg = a.cfg
    nm = la[5]
    for b_ in range(cfg.batch):
        n = int(nm[b_])
        assert np.array_equal(la[3][b_, :n], lb[3][b_, :n]), f"step {step}: miss_tok b={b_}"
        assert np.array_equal(la[4][b_, :n], lb[4][b_, :n]), f"step {step}: miss_slot b={b_}"
    for i in (0, 1, 2, 5):
        assert np.array_equal(la[i], lb[i]), f"step {step}: {names[i]}"
    for x, y, what in zip(a.state(0), b.state(0), ("cache_slots", "slot_token", "last_used",
                                                   "step")):
        assert np.array_equal(x, y), f"step {step}: {what}"


@pytest.mark.parametrize("shape", [dict(), dict(batch=3, mtp=2, idx_heads=32)],
                         ids=["tiny", "tiny_b3_mtp2"])
def test_noalloc_matches_select_manage(shape):
    cfg = dataclasses.replace(W.tiny(), **shape)
    assert _scratch_need(cfg) <= STATIC_SCRATCH_BYTES
    ld = W.gen_layer(cfg, 0)
    ref = Session(cfg, [ld])
    new = Session(cfg, [ld])
    qs = W.QueryStream(cfg, 0)
    w = W.head_weights(cfg, ld.w)
    try:
        for step in range(2):
            _, enc, qm = qs.next()
            qd, wd, _ = ref.device_inputs(enc, w, qm)
            scores = ref.scores_only(0, qd, wd).clone()
            ref.select(0, scores)
            _noalloc(new, 0, scores)
            torch.cuda.synchronize()
            assert ref.poll() == ess.ESS_OK
            assert new.poll() == ess.ESS_OK
            _compare(ref, new, step)
            # the steps must move the cache, or the second step checks nothing new
            assert int(new.n_miss.sum().item()) > 0 or step > 0
    finally:
        ref.close()
        new.close()


def test_noalloc_rejects_oversized_scratch():
    # 64 requests x 2 ways: 128 histograms of 16 KiB fill the 2 MiB array alone,
    # and the victim lists do not fit beside them; the pool itself is valid
    cfg = dataclasses.replace(W.tiny(), batch=64, mtp=2, idx_heads=32, T=1024, C=256, k=128)
    assert _scratch_need(cfg) > STATIC_SCRATCH_BYTES
    from host_latent_cache_gb300.session import ess_config_of
    assert ess.ess_pool_device_bytes(ess_config_of(cfg)) > 0
    ld = W.gen_layer(cfg, 0)
    s = Session(cfg, [ld])
    try:
        s.n_miss.fill_(-7)
        before = s.state(0)
        scores = torch.zeros_like(s.scores)
        with pytest.raises(ess.EssError) as ei:
            _noalloc(s, 0, scores)
        assert ei.value.code == ess.ESS_ERR_OOM
        torch.cuda.synchronize()
        assert np.all(s.n_miss.cpu().numpy() == -7)
        for x, y in zip(before, s.state(0)):
            assert np.array_equal(x, y)
    finally:
        s.close()
