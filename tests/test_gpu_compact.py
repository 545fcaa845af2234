"""Layers whose host master copy holds compact 656-byte rows.

"ESS: Latent-Cache Offload" quotes ~656-byte host transfers per token (its
table of mechanisms, the FlashTrans + UVA row): 512 e4m3 latent values in four
tiles with power-of-two scales and the 64 bf16 RoPE values.  The gathers widen
each miss row to bf16 on the way (exactly), so the pool rows equal the decoded
rows bit for bit, the lists and state follow the oracle bit for bit, and the
attention matches the oracle's attention over the decoded rows within the
usual tolerance; fused and staged misses, from an empty and from a full pool.
"""
import numpy as np
import pytest
import torch

from host_latent_cache_gb300 import ess
from host_latent_cache_gb300 import workloads as W

from parity_util import Pair

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_latent_cache_gb300 import build as B
    B.build()
    assert torch.cuda.is_available()
    ess.load()


@pytest.mark.parametrize("mode", [ess.ESS_MISS_FUSED, ess.ESS_MISS_STAGED], ids=["fused", "staged"])
def test_tiny_compact_rows(mode):
    cfg = W.tiny().replace(compact=True)
    p = Pair(cfg, miss_mode=mode)
    for _ in range(cfg.steps):
        p.run_step()
    p.check_pool_rows()
    p.prime_full(age=6)          # the reload of a restored state widens rows too
    p.check_pool_rows()
    for _ in range(4):
        p.run_step()
    p.check_pool_rows()
    assert sum(p.evicted) > 0
    p.close()


def test_compact_rows_fp8_indexer_two_ways_ragged():
    cfg = W.v32_32k().replace(batch=3, T=8192, T_per_req=[8192, 3001, 200], k=512, C=1024,
                              mtp=2, mla_heads=128, compact=True)
    p = Pair(cfg)
    for s in range(3):
        p.run_step(check_scores=(s == 0))
    p.prime_full(age=3)
    for _ in range(3):
        p.run_step()
    p.check_pool_rows()
    p.close()


def test_append_is_refused_on_a_compact_layer():
    cfg = W.tiny().replace(compact=True, T=1024, k=64, C=128)
    p = Pair(cfg)
    lat = torch.zeros((cfg.batch, 576), dtype=torch.int16, device="cuda")
    key = torch.zeros((cfg.batch, 128), dtype=torch.uint8, device="cuda")
    sc = torch.ones(cfg.batch, dtype=torch.float32, device="cuda")
    with pytest.raises(ess.EssError) as ei:
        ess.ess_append(p.sess.pool, 0, lat, key, sc)
    assert ei.value.code == ess.ESS_ERR_UNSUPPORTED
    p.close()
