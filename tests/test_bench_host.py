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


def _recorded_digest(name):
    import os
    with open(os.path.join(bench.ROOT, "profiles", f"indexer_{name}.txt")) as f:
        for line in f:
            if line.startswith("source_digest"):
                return line.split("=", 1)[1].strip()


def test_traffic_comes_from_the_profile_while_sources_match(monkeypatch):
    cfg = W.long_128k()
    monkeypatch.setattr(bench, "indexer_source_digest", lambda: _recorded_digest(cfg.name))
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


def test_layer_roofline_terms():
    # 138.4 MB of keys and 15,000 hit rows at 6,781 GB/s, a 100 us step
    r = bench.layer_roofline(138_412_032, 15_000, 1_200, 100.0, 6781.1,
                             idx_flops=2 * 64 * 128 * 8 * 131072, idx_us=45.0, bf16_tflops=1907.9)
    r_idx = 138_412_032 / 6781.1e9 * 1e6
    r_hit = 15_000 * 1152 / 6781.1e9 * 1e6
    assert abs(r["R_us"] - max(r_idx, r_hit)) < 1e-9 and abs(r["frac"] - r["R_us"] / 100.0) < 1e-12
    assert abs(r["additive_us"] - (r_idx + r_hit)) < 1e-9 and r["additive_frac"] > r["frac"]
    assert r["miss_bytes_per_step"] == 1_200 * 1152
    t = r["indexer_tensor"]
    assert abs(t["achieved_tflops"] - 2 * 64 * 128 * 8 * 131072 / 45e-6 / 1e12) < 1e-9
    assert t["peak_tflops"] == 2 * 1907.9 and 0 < t["frac"] < 0.2
    assert "indexer_tensor" not in bench.layer_roofline(1, 1, 0, 1.0, 1.0)


def test_layer_roofline_link_term():
    # 1,200 miss rows over a 200 GB/s link take 6.9 us: above the hit term,
    # below the indexer's 20.4 us; the additive form adds all three
    r = bench.layer_roofline(138_412_032, 15_000, 1_200, 100.0, 6781.1, link_gbs=200.0)
    r_idx = 138_412_032 / 6781.1e9 * 1e6
    r_hit = 15_000 * 1152 / 6781.1e9 * 1e6
    r_miss = 1_200 * 1152 / 200e9 * 1e6
    assert abs(r["terms_us"]["misses_link"] - r_miss) < 1e-9
    assert abs(r["R_us"] - max(r_idx, r_hit, r_miss)) < 1e-9
    assert abs(r["additive_us"] - (r_idx + r_hit + r_miss)) < 1e-9
    # a slow link makes the miss term the bound
    r2 = bench.layer_roofline(138_412_032, 15_000, 1_200, 100.0, 6781.1, link_gbs=10.0)
    assert abs(r2["R_us"] - 1_200 * 1152 / 10e9 * 1e6) < 1e-9
