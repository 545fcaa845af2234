"""Parity at the full workload sizes, in the launch configuration the bench
times: every step of a few is compared in full against the oracle (top-k
lists, miss union, LRU state bit-exact; attention within tolerance)."""
import pytest
import torch

from host_latent_cache_gb300 import ess
from host_latent_cache_gb300 import workloads as W

from parity_util import Pair

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_latent_cache_gb300 import build as B
    B.build()
    assert torch.cuda.is_available()
    ess.load()


def test_long_128k_first_steps():
    cfg = W.long_128k()
    p = Pair(cfg)
    for s in range(3):
        p.run_step(check_scores=(s == 0))
    p.check_pool_rows()
    p.close()


@pytest.mark.parametrize("C", [8192, 16384])
def test_ctx_1m(C):
    cfg = W.ctx_1m(C)
    p = Pair(cfg)
    for s in range(2):
        p.run_step(check_scores=(s == 0))
    p.close()


def test_v32_full_batch():
    cfg = W.v32_32k()
    p = Pair(cfg)
    for _ in range(3):
        p.run_step()
    p.close()


def test_multilayer_full_shape_one_layer():
    cfg = W.multilayer().replace(layers=1)
    p = Pair(cfg)
    for _ in range(2):
        p.run_step()
    p.close()
