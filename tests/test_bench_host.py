"""Host-side logic of bench.py that needs no GPU: the units counted per step,
the ncu traffic read from the committed profile summary (and dropped once the
indexer's sources change), and the defaults the timing rules depend on."""
import sys

import bench
from host_latent_cache_gb300 import workloads as W


def test_throughput_counts_one_layer_per_step():
    # 8 requests x 1 way, 2 ranks, 10 steps in 2 ms -> 80,000 token-layers/s
    assert bench.job_throughput(8, 2, 10, 2.0) == 8 * 2 * 10 / 2e-3
    for name in ("long_128k", "multilayer"):
        cfg = W.ALL_CONFIGS[name]()
        assert bench.config_json(cfg, 1, "fused")["layers"] == 1


def test_traffic_comes_from_the_profile_while_sources_match(monkeypatch):
    cfg = W.long_128k()
    t = bench.indexer_traffic(cfg)
    assert isinstance(t, int) and t > 138_412_032            # at least the algorithmic bytes
    monkeypatch.setattr(bench, "indexer_source_digest", lambda: "0" * 16)
    assert bench.indexer_traffic(cfg) is None               # the kernel changed: no claim
    assert bench.indexer_traffic(W.tiny()) is None           # no capture for this workload


def test_defaults_meet_the_timing_rules(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert a.warmup >= 3 and a.steps >= 32 and a.gpus == 1 and a.impl == "ours"
    assert a.workload == "long_128k" and a.miss_mode == "fused"


def test_cpu_model_is_named():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
