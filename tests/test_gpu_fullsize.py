"""Parity at the full workload sizes, in the launch configuration the bench
times: every step is compared in full against the oracle (top-k lists, miss
union, LRU state bit-exact; attention within tolerance).

Each workload runs its first steps from an empty pool, then both sides are
put into the same FULL pool (every slot resident, stamps of earlier steps
with many ties) and run eight more steps.  There every miss evicts a resident
token, which is the steady state of the FlashOffloading analysis (section
"decode side (1)": once the hot cache is full, loads equal evictions and its
size stays C).  The evictions are counted to show the regime was reached."""
import pytest
import torch

from host_latent_cache_gb300 import ess
from host_latent_cache_gb300 import workloads as W

from parity_util import Pair

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

FULL_POOL_STEPS = 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_latent_cache_gb300 import build as B
    B.build()
    assert torch.cuda.is_available()
    ess.load()


_layer_cache = {}


def _layer(cfg):
    """Layer data, generated once per shape (the hot-pool size is not part of it)."""
    key = (cfg.name.split("_C")[0], cfg.seed, cfg.batch, cfg.T, cfg.compact)
    if key not in _layer_cache:
        _layer_cache.clear()
        _layer_cache[key] = W.gen_layer(cfg)
    return _layer_cache[key]


def _empty_then_full(cfg, first_steps, check_scores_first=True):
    p = Pair(cfg, lds=[_layer(cfg)])
    try:
        for s in range(first_steps):
            p.run_step(check_scores=(check_scores_first and s == 0))
        p.prime_full()
        p.check_pool_rows()          # the restored rows come from the host copy
        p.evicted.clear()
        for _ in range(FULL_POOL_STEPS):
            p.run_step()
        p.check_pool_rows()
        # every step of a full pool that misses evicts as many resident tokens
        assert all(e > 0 for e in p.evicted), p.evicted
    finally:
        p.close()
    return p.evicted


def test_long_128k_first_steps_then_full_pool():
    _empty_then_full(W.long_128k(), 3)


@pytest.mark.parametrize("C", [8192, 16384])
def test_ctx_1m_then_full_pool(C):
    _empty_then_full(W.ctx_1m(C), 2)


def test_long_128k_compact_rows_then_full_pool():
    """The 128K layer with its host copy in compact 656-byte rows."""
    _empty_then_full(W.long_128k().replace(compact=True), 2, check_scores_first=False)


def test_v32_full_batch_then_full_pool():
    _empty_then_full(W.v32_32k(), 3, check_scores_first=False)


def test_v32_four_ways_then_full_pool():
    """The pages' MTP3 merge (four top-k ways, one miss union) at the V3.2
    shape, with C = 4 * k: a full pool leaves no slack beyond the union."""
    _empty_then_full(W.v32_32k().replace(mtp=4), 2)


def test_multilayer_full_shape_one_layer_then_full_pool():
    _empty_then_full(W.multilayer().replace(layers=1), 2, check_scores_first=False)
