"""Benchmark of one sparse-decode layer with a host-resident latent cache.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload long_128k|...] [--miss-mode fused|staged]
                [--miss-sweep C1,C2,...]

A step is one decode step of one layer for the whole batch (the bench runs
the workload's first layer; a multi-layer workload counts one layer too): indexer scores
over the GPU-resident indexer cache, exact top-k + cache_slots resolve +
miss union + LRU update, and sparse MLA attention whose gather reads hits
from the HBM pool and misses from pinned host memory.  The workload is the
long-context layer: 8 requests x 131072 tokens, top-2048, 128 MLA heads,
64x128 e4m3 indexer, hot pool of 32768 slots, query drift rho = 0.9 with 5%
cold-miss bursts.  Inputs are seeded synthetic data; the keys read per step
(138 MB) exceed the 129 MB L2, so no flush is inserted between steps.

The timed steps are plain ess_step calls (each kernel launched as a
programmatic dependent of the previous one); per-kernel durations come from
as many further steps with events between the kernels.

One JSON line is printed by rank 0.  --impl reference times the CPU oracle
(float64 numpy) on the same workload instead; --miss-sweep prints the
distinct misses per step for several hot-pool sizes instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

_CORES = os.cpu_count() or 1
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from host_latent_cache_gb300 import workloads as W  # noqa: E402

METRIC = "decode token·layers/s at 128K,k=2048; HBM & host-link GB/s vs roofline"
UNIT = "token·layers/s"
IDX_BYTES_PER_TOKEN = 128 + 4       # e4m3 key row + fp32 scale, read once per request
ROW_BYTES = 1152


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_128k", choices=sorted(W.ALL_CONFIGS))
    ap.add_argument("--miss-mode", default="fused", choices=["fused", "staged"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-link", action="store_true", help="skip the host-link measurement")
    ap.add_argument("--compact", action="store_true",
                    help="host latent as compact 656-byte rows (e4m3 + power-of-two tile "
                         "scales + bf16 RoPE), widened to bf16 on the way in")
    ap.add_argument("--empty-pool", action="store_true",
                    help="time from an empty pool instead of filling it first")
    ap.add_argument("--prime-random", action="store_true",
                    help="start from a full pool of random resident tokens instead of filling it "
                         "by decode steps (short runs, e.g. under a profiler)")
    ap.add_argument("--cpu-steps", type=int, default=48)
    ap.add_argument("--overlap-steps", type=int, default=24)
    ap.add_argument("--pipeline", type=int, default=0,
                    help="time L layers of the workload as two micro-batches (half the "
                         "requests each) on two streams against the same work on one stream")
    ap.add_argument("--prefill", action="store_true",
                    help="time the prefill four-buffer engine over 8 layers of a 64K request")
    ap.add_argument("--append", action="store_true",
                    help="time decode steps that each append one token per request first")
    ap.add_argument("--policy", default="lru",
                    help="eviction orders of --miss-sweep, comma-separated: lru,random,score,lim")
    ap.add_argument("--miss-sweep", default=None,
                    help="comma-separated hot-pool sizes C: print the distinct miss rows per "
                         "step of the workload for each instead of the benchmark line")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_workload(cfg: W.WorkloadConfig, rank: int) -> W.WorkloadConfig:
    """Each rank serves its own independent requests (same shapes, its own
    seed): the decode path shards over requests with no exchange, so the job
    scales weakly and needs no collective on the data path."""
    return cfg.replace(seed=cfg.seed + 7919 * rank)


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise maximum of per-rank timings (a barrier-bracketed job is as
    slow as its slowest rank)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_throughput(units_per_step_per_rank: int, world: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job units per second: every rank's units over the slowest rank's time."""
    return world * units_per_step_per_rank * steps / (elapsed_ms / 1e3)


def config_json(cfg: W.WorkloadConfig, n_gpus: int, miss_mode: str):
    return {
        "workload": f"{cfg.name}: batch {cfg.batch} x T={cfg.T}, top-k {cfg.k}, "
                    f"{cfg.mla_heads} MLA heads (512+64 bf16), indexer {cfg.idx_heads}x"
                    f"{cfg.idx_dim} {'e4m3' if cfg.idx_dtype == W.FP8_E4M3 else 'bf16'}, "
                    f"C={cfg.C}, MTP={cfg.mtp}, rho={cfg.rho}, cold bursts {cfg.cold_p}",
        "batch_per_gpu": cfg.batch, "T": cfg.T, "k": cfg.k, "C": cfg.C, "mtp": cfg.mtp,
        "layers": 1, "miss_mode": miss_mode,
        "host_rows": ("compact 656 B (e4m3 + power-of-two tile scales + bf16 RoPE)"
                      if cfg.compact else "bf16 1152 B"),
        "l2": "inputs larger than L2 (keys read per step exceed the 129 MB L2); no flush",
        "parallelism": f"replicas x{n_gpus} (independent requests per GPU, no collective)",
    }


# ---------------------------------------------------------------- clocks
_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """Samples the SM clock and the clock-event reasons while the timed region
    runs: NVML through ctypes every millisecond (the timed region can be a few
    milliseconds long), else nvidia-smi every 50 ms.  Reads settings only."""

    def __init__(self, cuda_index: int):
        self.index = cuda_index
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            try:
                self.index = int(vis.split(",")[cuda_index])
            except (ValueError, IndexError):
                pass
        self.samples, self.smax, self.reasons, self.power = [], None, set(), []
        self.proc = None
        self.thread = None
        self.marks = []

    def _nvml(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvml init")
        h = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(h)) != 0:
            raise RuntimeError("nvml handle")
        return nv, h

    def __enter__(self):
        import threading
        import ctypes
        self.stop = False
        try:
            nv, h = self._nvml()
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.smax = float(mx.value)
            get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons

            def run():
                clk, rs, pw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
                while not self.stop:
                    timed = len(self.marks) == 1     # between the two marks
                    if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and timed:
                        self.samples.append(float(clk.value))
                    if get_reasons(h, ctypes.byref(rs)) == 0 and timed:
                        for bit, name in _REASONS.items():
                            if rs.value & bit:
                                self.reasons.add(name)
                    if nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 and timed:
                        self.power.append(pw.value / 1000.0)
                    time.sleep(0.001)

            self.thread = threading.Thread(target=run, daemon=True)
            self.thread.start()
            time.sleep(0.005)
        except Exception:
            self.thread = None
            fields = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                      "clocks_event_reasons.hw_thermal_slowdown,"
                      "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), f"--query-gpu={fields}",
                     "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                time.sleep(0.3)
            except Exception:
                self.proc = None
        return self

    def mark(self):
        """Start (first call) and end (second call) of the timed region."""
        self.marks.append(time.time())

    def __exit__(self, *a):
        self.stop = True
        if self.thread is not None:
            self.thread.join(timeout=2)
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.splitlines():
                p = [x.strip() for x in line.split(",")]
                if len(p) < 6:
                    continue
                try:
                    self.samples.append(float(p[0]))
                    self.smax = float(p[1])
                except ValueError:
                    continue
                for n, v in zip(names, p[2:6]):
                    if v.lower() == "active":
                        self.reasons.add(n)

    def summary(self):
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.smax, "reasons": sorted(self.reasons),
                "samples": len(self.samples),
                "power_w_max": max(self.power) if self.power else None,
                "source": "nvml" if self.thread is not None else "nvidia-smi"}


# ---------------------------------------------------------------- CPU oracle baseline
def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, else implementer/part ids)."""
    try:
        name, impl, part = None, None, None
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                k, v = k.strip(), v.strip()
                if k == "model name" and not name:
                    name = v
                elif k == "CPU implementer" and not impl:
                    impl = v
                elif k == "CPU part" and not part:
                    part = v
        return name or (f"implementer {impl} part {part}" if impl else "unknown")
    except OSError:
        return "unknown"


def run_oracle(cfg: W.WorkloadConfig, ld: W.LayerData, n_steps: int, n_req: int,
               warm: int = 1):
    """Times the CPU oracle on the first n_req requests for n_steps steps
    (after `warm` untimed steps).  Returns (token.layers/s, seconds)."""
    from oracle import ess_oracle as O
    sub = cfg.replace(batch=n_req)
    keys = W.decode_keys(cfg, ld.idx_keys[:n_req]).astype(np.float32)
    lay = O.OracleLayer(ld.T[:n_req], cfg.C, cfg.k, cfg.sm_scale)
    qs = W.QueryStream(sub)
    keyf = lambda b: keys[b, : int(ld.T[b])]
    if cfg.compact:
        from oracle import compact_row as X
        latf = lambda b, order: X.decode_rows(ld.latent_c[b, order])
    else:
        latf = lambda b, order: W.bf16_bits_to_float(ld.latent[b, order]).astype(np.float64)
    w = W.head_weights(sub, ld.w[:n_req]).astype(np.float64)
    t = 0.0
    for s in range(warm + n_steps):
        q, _, qm = qs.next()
        qmf = W.bf16_bits_to_float(qm).astype(np.float64)
        t0 = time.perf_counter()
        lay.step(q.astype(np.float64), w, keyf, ld.idx_scale, qmf, latf)
        if s >= warm:
            t += time.perf_counter() - t0
    units = n_req * cfg.mtp * n_steps          # one decode layer per step
    return units / t, t


# ---------------------------------------------------------------- reference arm
def bench_reference(args, cfg, rank, world):
    if rank != 0:
        return 0
    ld = W.gen_layer(cfg)
    steps = max(1, args.steps)
    # a bounded sample per step: all requests while that keeps the run to a few
    # minutes, fewer requests otherwise
    n_req = max(1, min(cfg.batch, (cfg.batch * 32) // max(steps, 1)))
    v, t = run_oracle(cfg, ld, steps, n_req, warm=max(1, min(args.warmup, 2)))
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": config_json(cfg, args.gpus, args.miss_mode),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": _CORES, "cpu": cpu_model(),
                         "kind": "oracle",
                         "sample": f"{n_req} of {cfg.batch} requests per step, {steps} steps "
                                   f"after warm-up, float64 numpy with {_CORES} BLAS threads"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def measure_overlap(cfg, ld, n_steps, stream, host_buffers, qs=None, start_state=None):
    """T_copy (staging kernel), T_SFA (attention with every row in the pool)
    and T_fused (attention that reads misses from host memory itself), per
    step, and OverlapRatio = (T_copy + T_SFA - T_fused) / T_copy.

    A fused and a staged pool start from the same state and take the same
    inputs, so their selections and misses are identical; they take turns step
    by step (a slow phase of the host link, which other work on the machine
    shares, then falls on both).  A host row is slower the first time it is
    read after a while (its address translation is cold), so whichever pool
    reads a step's misses second would be favoured: the steps run in two
    halves, the fused pool first in the first half and the staged pool first
    in the second, and T_fused comes from the first half, T_copy from the
    second, each on rows read cold; T_SFA reads no host memory.  With a start
    state (the main session's steady state) and its query stream both halves
    continue from where the timed run ended; otherwise the pools start empty
    and the first steps, which still fill the pool, are dropped.  Events
    between the kernels stop them from launching early, as in the separate
    calls these timings stand for."""
    import torch
    from host_latent_cache_gb300 import ess
    from host_latent_cache_gb300.session import Session
    qs = qs if qs is not None else W.QueryStream(cfg)
    wts = W.head_weights(cfg, ld.w)
    F, S = ess.ESS_MISS_FUSED, ess.ESS_MISS_STAGED
    halves = []
    state = start_state
    identical = True
    for order in ((F, S), (S, F)):
        steps = [qs.next() for _ in range(n_steps)]
        sessions, ins, evs, nms = {}, {}, {}, {}
        for mode in order:
            sess = Session(cfg, [ld], miss_mode=mode, host_buffers=host_buffers)
            if state is not None:
                sess.set_state(0, state)
            sessions[mode] = sess
            ins[mode] = [sess.device_inputs(enc, wts, qm) for (_, enc, qm) in steps]
            evs[mode] = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in steps]
            nms[mode] = torch.zeros(len(steps), dtype=torch.int64, device=sess.device)
        torch.cuda.synchronize()
        for i in range(len(steps)):
            for mode in order:
                sess, e = sessions[mode], evs[mode][i]
                qd, wd, qmd = ins[mode][i]
                sess.indexer_topk(0, qd, wd, stream)
                e[0].record(stream)
                if mode == S:
                    sess.stage(0, stream)
                e[1].record(stream)
                sess.attention(0, qmd, stream=stream)
                e[2].record(stream)
                nms[mode][i] = sess.n_miss.sum()
        torch.cuda.synchronize()
        res = {}
        for mode in order:
            sess = sessions[mode]
            assert sess.poll(stream) == ess.ESS_OK
            nmh = nms[mode].cpu().tolist()
            res[mode] = [(int(nmh[i]), e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]))
                         for i, e in enumerate(evs[mode])]
        identical = identical and bool(torch.equal(sessions[F].out, sessions[S].out))
        assert [r[0] for r in res[F]] == [r[0] for r in res[S]]
        cs_, st_, lu_, sp_ = sessions[F].state(0)
        state = W.PoolState(cs_, st_, lu_, sp_)
        for mode in order:
            sessions[mode].close()
        halves.append(res)
    # from an empty pool the first steps still miss heavily (the pool has not
    # settled into the drift's working set): they are dropped
    settle = 0 if start_state is not None else min(4, n_steps - 1)
    rng = range(settle, n_steps)
    fz = halves[0][F]                      # fused first: its rows cold
    sg = halves[1][S]                      # staged first: its copies cold
    sfa = [halves[h][S][i][2] for h in (0, 1) for i in rng]
    tf = statistics.median(fz[i][2] for i in rng)
    tc = statistics.median(sg[i][1] for i in rng)
    ts = statistics.median(sfa)
    mf = statistics.mean(fz[i][2] for i in rng)
    mc = statistics.mean(sg[i][1] for i in rng)
    ms_ = statistics.mean(sfa)
    return {"steps_per_half": len(rng), "settling_steps_dropped": settle,
            "start": "steady state of the timed run" if start_state is not None else "empty pool",
            "statistic": "median over steps (means beside)",
            "miss_rows_per_step": statistics.mean(fz[i][0] for i in rng),
            "t_copy_us": 1e3 * tc, "t_sfa_us": 1e3 * ts, "t_fused_us": 1e3 * tf,
            "overlap_ratio": (tc + ts - tf) / tc if tc > 0 else None,
            "speedup_vs_copy_then_attend": (tc + ts) / tf if tf > 0 else None,
            "mean": {"t_copy_us": 1e3 * mc, "t_sfa_us": 1e3 * ms_, "t_fused_us": 1e3 * mf,
                     "overlap_ratio": (mc + ms_ - mf) / mc if mc > 0 else None},
            "second_reader_us": {
                "fused_after_staged": 1e3 * statistics.median(halves[1][F][i][2] for i in rng),
                "copy_after_fused": 1e3 * statistics.median(halves[0][S][i][1] for i in rng)},
            "per_step_us": {"miss_rows_first_half": [fz[i][0] for i in rng],
                            "fused_first_half": [round(1e3 * fz[i][2], 1) for i in rng],
                            "miss_rows_second_half": [sg[i][0] for i in rng],
                            "copy_second_half": [round(1e3 * sg[i][1], 1) for i in rng]},
            "outputs_identical": identical}


# what the indexer kernel's device code is built from: its own file, the
# device helpers, and the compile-time constants of the shared header (the
# rest of that header declares host-side state); the DRAM traffic taken by
# ncu holds only while these are unchanged
INDEXER_SOURCES = ("ess_indexer.cu", "ess_device.cuh")
INDEXER_CONSTANTS = "ess_internal.h"


def layer_roofline(idx_bytes, hit_rows, miss_rows, step_us, hbm_gbs, idx_flops=None,
                   idx_us=None, bf16_tflops=None, link_gbs=None, miss_row_bytes=ROW_BYTES):
    """The layer's roofline terms: R = max(indexer bytes / HBM, hit bytes /
    HBM, miss bytes / host link) against the step; the stricter additive form
    (indexer and hit bytes through HBM one after the other, plus the miss
    bytes over the link); and the indexer's fraction of the FP8 tensor peak
    (the measured bf16 peak times the nominal FP8/bf16 ratio of 2).  Without
    a measured link peak the miss term is left out and only reported."""
    r_idx = idx_bytes / (hbm_gbs * 1e9) * 1e6
    r_hit = hit_rows * ROW_BYTES / (hbm_gbs * 1e9) * 1e6
    miss_bytes = miss_rows * miss_row_bytes          # over the host link
    r_miss = miss_bytes / (link_gbs * 1e9) * 1e6 if link_gbs else 0.0
    R = max(r_idx, r_hit, r_miss)
    add = r_idx + r_hit + r_miss
    out = {"R_us": R, "step_us": step_us, "frac": R / step_us,
           "additive_us": add, "additive_frac": add / step_us,
           "terms_us": {"indexer": r_idx, "hits": r_hit, "misses_link": r_miss},
           "link_peak_gbs": link_gbs,
           "miss_rows_per_step": miss_rows, "miss_bytes_per_step": miss_bytes}
    if idx_flops is not None and idx_us and bf16_tflops:
        achieved = idx_flops / (idx_us * 1e-6) / 1e12
        peak = 2.0 * bf16_tflops
        out["indexer_tensor"] = {"achieved_tflops": achieved, "peak_tflops": peak,
                                 "frac": achieved / peak,
                                 "peak_source": "measured bf16 burst x 2 (nominal fp8/bf16)"}
    return out


def indexer_source_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "host_latent_cache_gb300", "csrc")
    for name in INDEXER_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    with open(os.path.join(csrc, INDEXER_CONSTANTS), "rb") as f:
        h.update(b"".join(l for l in f.read().splitlines(True)
                          if b"constexpr" in l or l.lstrip().startswith(b"#define")))
    return h.hexdigest()[:16]


def indexer_traffic(cfg):
    """DRAM bytes (read + write) per indexer launch from the committed ncu
    summary of this workload, or None when there is none or the kernel's
    sources have changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"indexer_{cfg.name}.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                fields[k.strip()] = v.strip()
    if fields.get("source_digest") != indexer_source_digest():
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measure_link(host_buf, n_host_rows, device, stream, reps=5, row_bytes=ROW_BYTES):
    """Host-link rates through the library's own gather kernel (16-byte loads
    by the GPU's threads, as the miss path reads) and through the copy engine
    (cudaMemcpyAsync from pinned memory), each timed with CUDA events over
    `reps` launches after one untimed launch.  Returns GB/s figures; the
    largest sequential rate is the link peak of the layer roofline."""
    import torch
    from host_latent_cache_gb300 import ess
    res = {}
    n_seq = min(n_host_rows, (256 << 20) // row_bytes)
    dst = torch.empty((n_seq, row_bytes), dtype=torch.uint8, device=device)
    bad = torch.zeros(1, dtype=torch.int32, device=device)
    g = torch.Generator().manual_seed(4242)

    per_launch = {}

    def timed(fn, nbytes, name):
        fn()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        ev[0].record(stream)
        for i in range(reps):
            fn()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        per_launch[name] = [round(ev[i].elapsed_time(ev[i + 1]) * 1e3, 1) for i in range(reps)]
        return nbytes * reps / (ev[0].elapsed_time(ev[reps]) * 1e-3) / 1e9

    res["gather_seq_gbs"] = timed(
        lambda: ess.ess_host_gather(host_buf, n_host_rows, row_bytes, None, n_seq, dst, bad,
                                    stream), n_seq * row_bytes, "gather_seq")
    for n in (16384, n_seq):
        rows = torch.randint(0, n_host_rows, (n,), generator=g, dtype=torch.int64).to(device)
        res[f"gather_random_{n}_rows_gbs"] = timed(
            lambda: ess.ess_host_gather(host_buf, n_host_rows, row_bytes, rows, n, dst, bad,
                                        stream), n * row_bytes, f"gather_random_{n}")
    hsrc = torch.empty(n_seq * row_bytes, dtype=torch.uint8).pin_memory()
    dflat = dst.view(-1)
    res["copy_engine_h2d_gbs"] = timed(lambda: dflat.copy_(hsrc, non_blocking=True),
                                       n_seq * row_bytes, "copy_engine")
    torch.cuda.synchronize()
    assert int(bad.item()) == 0
    res["per_launch_us"] = per_launch
    res["bytes_per_sequential_read"] = n_seq * row_bytes
    res["row_bytes"] = row_bytes
    res["peak_gbs"] = max(res["gather_seq_gbs"], res["copy_engine_h2d_gbs"])
    res["peak_source"] = ("measured in this run: the larger of the sequential gather kernel "
                          "and the copy engine")
    return res


def warm_host(sess, layers, stream, row_bytes):
    """Every host row of the given layers read once by the GPU, in 256 MB
    chunks through the library's gather: the first device access to a pinned
    page sets up its mapping, slowly (at B=32 and 64K tokens the first
    steps that met never-read rows took milliseconds), and a running server's
    host cache has long been read."""
    import torch
    from host_latent_cache_gb300 import ess
    n_rows = sess.cfg.batch * W.t_max_of(sess.cfg)
    chunk = max(1, (256 << 20) // row_bytes)
    dst = torch.empty((min(chunk, n_rows), row_bytes), dtype=torch.uint8, device=sess.device)
    bad = torch.zeros(1, dtype=torch.int32, device=sess.device)
    for l in layers:
        for r0 in range(0, n_rows, chunk):
            n = min(chunk, n_rows - r0)
            rows = torch.arange(r0, r0 + n, dtype=torch.int64, device=sess.device)
            ess.ess_host_gather(sess.host[l], n_rows, row_bytes, rows, n, dst, bad, stream)
    torch.cuda.synchronize()
    assert int(bad.item()) == 0


def fill_pool(sess, qs, wts, stream, max_steps=1024, check_every=16):
    """Runs decode steps (untimed) until every request's hot pool is full, so
    that the timed steps see the steady state of the FlashOffloading analysis
    ("decode side (1)": loads equal evictions once the C slots are taken).
    Returns (steps run, fraction of slots resident)."""
    import numpy as np
    from host_latent_cache_gb300 import ess
    C, B = sess.cfg.C, sess.cfg.batch
    T = np.asarray(sess.T[0].numpy())
    full = float(np.minimum(T, C).sum())
    n, occ = 0, 0.0
    while n < max_steps:
        for _ in range(check_every):
            _, enc, qm = qs.next()
            qd, wd, qmd = sess.device_inputs(enc, wts, qm)
            ess.ess_step(sess.pool, 0, qd, wd, qmd, sess.out, stream)
            n += 1
        _, st, _, _ = sess.state(0)
        occ = float((st >= 0).sum()) / full if full else 1.0
        if occ >= 1.0:
            break
    return n, occ


def bench_ours(args, cfg, rank, world, local_rank):
    import torch
    from host_latent_cache_gb300 import build as B
    from host_latent_cache_gb300 import ess
    from host_latent_cache_gb300.session import Session

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if rank == 0:
        B.build()
    if dist is not None:
        dist.barrier()
    ess.load()
    # each rank serves its own independent requests (weak scaling)
    cfg_r = rank_workload(cfg, rank)
    ld = W.gen_layer(cfg_r)
    mode = ess.ESS_MISS_STAGED if args.miss_mode == "staged" else ess.ESS_MISS_FUSED
    miss_row_bytes = W.COMPACT_ROW_BYTES if cfg.compact else ROW_BYTES
    sess = Session(cfg_r, [ld], miss_mode=mode)
    qs = W.QueryStream(cfg_r)
    n_total = args.warmup + 3 * args.steps
    wts = W.head_weights(cfg_r, ld.w)
    stream = torch.cuda.current_stream()
    warm_host(sess, [0], stream, miss_row_bytes)
    # steady state: the pool is filled by real decode steps before the warm-up
    if args.prime_random:
        # a full pool of random resident tokens (short runs, e.g. under a profiler):
        # the warm-up steps then settle it into the queries' working set
        sess.set_state(0, W.full_pool_state(cfg_r, ld, 0, age=8))
        fill_steps, occupancy = 0, 1.0
    elif args.empty_pool:
        fill_steps, occupancy = 0, 0.0
    else:
        fill_steps, occupancy = fill_pool(sess, qs, wts, stream)
    dev_inputs, host_inputs = [], []
    for s in range(n_total):
        q, enc, qm = qs.next()
        if s < args.warmup + 2 * args.steps:
            dev_inputs.append(sess.device_inputs(enc, wts, qm))
        else:
            hq = torch.from_numpy(np.ascontiguousarray(enc).view(np.uint8)).pin_memory()
            hw = torch.from_numpy(wts).pin_memory()
            hqm = torch.from_numpy(np.ascontiguousarray(qm).view(np.int16)).pin_memory()
            host_inputs.append((hq, hw, hqm))
    out_host = torch.empty(tuple(sess.out.shape), dtype=torch.float32).pin_memory()
    nsteps = args.steps

    def make_events(n, k):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(k)] for _ in range(n)]
        for row in evs:
            for e in row:
                e.record(stream)        # materialise the event handles
        torch.cuda.synchronize()
        return evs

    ev = make_events(nsteps, 4)

    def one_step(i, events=None):
        qd, wd, qmd = dev_inputs[i]
        if events is None:
            ess.ess_step(sess.pool, 0, qd, wd, qmd, sess.out, stream)
        else:
            ess.ess_step_profiled(sess.pool, 0, qd, wd, qmd, sess.out, events, stream)

    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # the clock sampler starts before the warm-up, and the timed steps follow
    # the warm-up with nothing but the barrier and a synchronize in between:
    # the host-memory path of the misses is slow again after the GPU idles
    # generating the inputs above leaves the GPU idle for up to seconds (at
    # B=32 tens of ms of numpy per step), after which the first steps that
    # read host rows ran many times slower; the host rows are read once more
    # right before the warm-up, as a serving GPU reads them all the time
    warm_host(sess, [0], stream, miss_row_bytes)
    with ClockSampler(local_rank) as clk:
        for i in range(args.warmup):
            one_step(i)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        launches_before = sess.kernel_launches()
        clk.mark()
        t_start.record(stream)
        for i in range(nsteps):
            one_step(args.warmup + i)
        t_end.record(stream)
        torch.cuda.synchronize()
        clk.mark()
    if dist is not None:
        dist.barrier()
    st = sess.poll(stream)
    assert st == ess.ESS_OK, ess.status_string(st)
    elapsed_ms = t_start.elapsed_time(t_end)
    launches_timed = sess.kernel_launches() - launches_before
    # per-kernel durations and the step counters: the next steps again, with
    # events between the kernels (an event between two kernels stops the next
    # one from launching early, so these steps are kept out of the timed region)
    sess.stats(0, reset=True)
    for i in range(nsteps):
        one_step(args.warmup + nsteps + i, ev[i])
    torch.cuda.synchronize()
    assert sess.poll(stream) == ess.ESS_OK
    stats = sess.stats(0, reset=True)
    idx_ms = [e[0].elapsed_time(e[1]) for e in ev]
    sel_ms = [e[1].elapsed_time(e[2]) for e in ev]
    att_ms = [e[2].elapsed_time(e[3]) for e in ev]

    # host-link rates (the miss term of the roofline), on this session's host copy
    link = None
    if rank == 0 and not args.no_link:
        link = measure_link(sess.host[0], cfg_r.batch * W.t_max_of(cfg_r), sess.device, stream,
                            row_bytes=miss_row_bytes)


    # end to end through the public C ABI with host buffers.  The first device
    # access to a freshly pinned buffer is slow (its mapping is set up), so one
    # untimed pass goes over every buffer first, as a server's reused input
    # buffers would have been; the timed pass then runs the same calls again
    for i in range(nsteps):
        hq, hw, hqm = host_inputs[i]
        ess.ess_step_host(sess.pool, 0, hq, hw, hqm, out_host, stream)
    torch.cuda.synchronize()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for i in range(nsteps):
        hq, hw, hqm = host_inputs[i]
        ess.ess_step_host(sess.pool, 0, hq, hw, hqm, out_host, stream)
    e_end.record(stream)
    torch.cuda.synchronize()
    assert sess.poll(stream) == ess.ESS_OK
    e2e_ms = e_start.elapsed_time(e_end)

    # OverlapRatio of the fused miss path: fused and staged pools stepped in
    # lockstep on the same inputs (identical state trajectories), from the
    # state the main pool has reached, with the queries that follow
    overlap = None
    if args.overlap_steps > 0 and world == 1:
        cs_, st_, lu_, sp_ = sess.state(0)
        overlap = measure_overlap(cfg_r, ld, args.overlap_steps, stream, sess.host, qs=qs,
                                  start_state=W.PoolState(cs_, st_, lu_, sp_))

    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e_ms], dist, device="cuda")
    units_step = cfg.batch * cfg.mtp            # one decode layer of the workload per step
    value = job_throughput(units_step, world, nsteps, elapsed_ms)
    e2e_value = job_throughput(units_step, world, nsteps, e2e_ms)

    result = None
    if rank == 0:
        peaks = {}
        try:
            peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        except Exception:
            pass
        hbm_peak = peaks.get("hbm_gbs")
        peak_src = "measured" if hbm_peak else "fallback"
        hbm_peak = hbm_peak or 6800.0
        Tsum = int(ld.T.sum())
        idx_bytes = Tsum * IDX_BYTES_PER_TOKEN
        idx_avg_ms = statistics.mean(idx_ms)
        achieved = idx_bytes / (idx_avg_ms / 1e3) / 1e9
        miss_rows = stats.miss_rows / max(nsteps, 1)
        hit_rows = (stats.hits) / max(nsteps, 1)
        step_us = elapsed_ms * 1e3 / nsteps
        idx_flops = 2 * cfg.idx_heads * cfg.idx_dim * Tsum * cfg.mtp
        traffic = indexer_traffic(cfg)
        link_peak = link["peak_gbs"] if link else None
        att_avg_ms = statistics.mean(att_ms)
        if link is not None:
            # miss bytes the fused attention moved over the link per step, over
            # the attention kernel's time (attention + merge, event-timed)
            link["achieved_fused_attention_gbs"] = (miss_rows * miss_row_bytes
                                                    / (att_avg_ms * 1e-3) / 1e9)
            link["achieved_frac_of_peak"] = link["achieved_fused_attention_gbs"] / link_peak
        result = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": nsteps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / nsteps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3+bf16", "data": "synthetic",
            "config": dict(config_json(cfg, world, args.miss_mode),
                           pool_fill_steps=fill_steps, pool_occupancy_at_warmup=occupancy,
                           pool_state=("full of random tokens before the warm-up"
                                       if args.prime_random else
                                       "steady (full before the warm-up)" if occupancy >= 1.0
                                       else "filling"),
                           host_rows="every host row read once by the GPU before the first step"),
            "roofline": {"bound": "hbm", "kernel": "indexer (a1)", "achieved": achieved,
                         "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                         "traffic": traffic, "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": idx_bytes},
            "layer_roofline": layer_roofline(idx_bytes, hit_rows, miss_rows, step_us, hbm_peak,
                                             idx_flops, idx_avg_ms * 1e3,
                                             peaks.get("bf16_tflops"), link_peak,
                                             miss_row_bytes),
            "link": link,
            "kernels_ms": {"indexer": statistics.mean(idx_ms), "select": statistics.mean(sel_ms),
                           "attention": statistics.mean(att_ms)},
            "hit_rate": stats.hits / max(stats.hits + stats.misses, 1),
            "overlap": overlap,
            "e2e": {"value": e2e_value, "unit": UNIT,
                    "h2d_bytes_per_step": int(sum(x.numel() * x.element_size()
                                                  for x in host_inputs[0])),
                    "d2h_bytes_per_step": int(out_host.numel() * 4),
                    "buffers": f"{nsteps} pinned input sets and one pinned output, each "
                               "touched by one untimed pass of the same calls first"},
            "gpu_launches": launches_timed,
            "gpu_launches_note": "kernels the library launched in the timed steps, counted by "
                                 "the pool as they were enqueued",
            "clocks": clk.summary(),
        }
    sess.close()
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return result, ld


POLICIES = {"lru": 0, "random": 1, "score": 2, "lim": 3}   # ESS_EVICT_*


def miss_sweep(args, cfg):
    """Distinct miss rows per step (after the first fill) for each hot-pool
    size C and eviction order, on the same seeded query stream, through the
    CUDA path.  The FlashOffloading analysis reports how misses fall as the
    hot cache grows and how little the eviction policy matters (section
    "evaluation", the decode ablation and Figure 8)."""
    import torch
    from host_latent_cache_gb300 import ess
    from host_latent_cache_gb300.session import Session
    ess.load()
    ld = W.gen_layer(cfg)
    sizes = [int(x) for x in args.miss_sweep.split(",")]
    policies = args.policy.split(",")
    hb = [ess.HostBuffer(ld.host_latent.shape, np.uint16)]
    hb[0].array[...] = ld.host_latent
    res = {}
    for pol in policies:
        for C in sizes:
            c2 = cfg.replace(C=C)
            sess = Session(c2, [ld], host_buffers=hb)
            ess.ess_pool_set_eviction(sess.pool, POLICIES[pol], 0x5EED)
            qs = W.QueryStream(c2)
            wts = W.head_weights(c2, ld.w)
            stream = torch.cuda.current_stream()
            for s in range(args.steps):
                _, enc, qm = qs.next()
                qd, wd, qmd = sess.device_inputs(enc, wts, qm)
                if s == 1:
                    torch.cuda.synchronize()
                    sess.stats(0, reset=True)      # the first step fills the empty pool
                ess.ess_step(sess.pool, 0, qd, wd, qmd, sess.out, stream)
            torch.cuda.synchronize()
            assert sess.poll(stream) == ess.ESS_OK
            st = sess.stats(0, reset=True)
            res[(pol, C)] = st.miss_rows / max(1, args.steps - 1) / cfg.batch
            sess.close()
    hb[0].close()
    line = {"miss_sweep": {"workload": cfg.name, "steps_after_first_fill": args.steps - 1,
                           "C": sizes, "policies": policies,
                           "miss_rows_per_request_step": {
                               p: [res[(p, c)] for c in sizes] for p in policies},
                           "reduction_vs_first": {
                               p: [1.0 - res[(p, c)] / res[(p, sizes[0])] if res[(p, sizes[0])]
                                   else None for c in sizes] for p in policies}}}
    print(json.dumps(line), flush=True)
    return 0


def pipeline_bench(args, cfg):
    """The layer-wise pipeline (ess_pipeline_step): two micro-batches, half of
    the workload's requests each, every layer on its own stream per
    micro-batch, so one micro-batch's kernels fill the SMs the other leaves
    idle.  Timed against the same launches issued on a single stream."""
    import torch
    from host_latent_cache_gb300 import ess
    from host_latent_cache_gb300.session import Session
    ess.load()
    L = args.pipeline
    half = cfg.batch // 2
    cfgs = [cfg.replace(layers=L, batch=half, seed=cfg.seed + 100 * h) for h in range(2)]
    sess, ins = [], []
    for c in cfgs:
        lds = [W.gen_layer(c, l) for l in range(L)]
        s_ = Session(c, lds)
        warm_host(s_, range(L), torch.cuda.current_stream(), ROW_BYTES)
        qs = [W.QueryStream(c, l) for l in range(L)]
        steps = []
        for _ in range(2 * (args.warmup + args.steps)):
            per = []
            for l in range(L):
                _, enc, qm = qs[l].next()
                per.append(s_.device_inputs(enc, W.head_weights(c, lds[l].w), qm))
            steps.append(per)
        outs = [torch.zeros((c.batch, c.mtp, c.mla_heads, 512), dtype=torch.float32,
                            device="cuda") for _ in range(L)]
        sess.append((s_, outs))
        ins.append(steps)
        del lds
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    main_st = torch.cuda.current_stream()

    def run(step, two):
        if two:
            ess.ess_pipeline_step([s_[0].pool for s_ in sess], L,
                                  [ins[h][step][l][0] for h in range(2) for l in range(L)],
                                  [ins[h][step][l][1] for h in range(2) for l in range(L)],
                                  [ins[h][step][l][2] for h in range(2) for l in range(L)],
                                  [sess[h][1][l] for h in range(2) for l in range(L)], streams)
        else:
            for l in range(L):
                for h in range(2):
                    qd, wd, qmd = ins[h][step][l]
                    ess.ess_step(sess[h][0].pool, l, qd, wd, qmd, sess[h][1][l], main_st)

    res = {}
    nxt = 0   # every call takes the next step's inputs
    for mode, two in (("one_stream", False), ("two_streams", True)):
        for _ in range(args.warmup):
            run(nxt, two)
            nxt += 1
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            run(nxt, two)
            nxt += 1
        torch.cuda.synchronize()
        res[mode] = (time.perf_counter() - t0) / args.steps
    for s_, _ in sess:
        assert s_.poll() == ess.ESS_OK
        s_.close()
    units = cfg.batch * cfg.mtp * L
    line = {"pipeline": {"workload": cfg.name, "layers": L, "micro_batches": 2,
                         "requests_per_micro_batch": half, "steps": args.steps,
                         "timing": "host wall clock between synchronizes, per step of all layers",
                         "one_stream_us_per_step": 1e6 * res["one_stream"],
                         "two_streams_us_per_step": 1e6 * res["two_streams"],
                         "one_stream_token_layers_per_s": units / res["one_stream"],
                         "two_streams_token_layers_per_s": units / res["two_streams"]}}
    print(json.dumps(line), flush=True)
    return 0


def append_bench(args, cfg):
    """Decode with appends: a step that first appends one token per request
    (ess_append: the ring row, the indexer key, a completed page back to host
    memory), then runs the layer over the grown context.  After warm-up steps
    that fill the pool, blocks of steps with and without appends alternate
    (twice each) on the same pool, timed with CUDA events; then the append
    kernel alone, back to back."""
    import torch
    from host_latent_cache_gb300 import ess
    from host_latent_cache_gb300.session import Session
    ess.load()
    K = args.steps
    n_app = 3 * K
    c = cfg.replace(grow=n_app)
    ld = W.gen_layer(c)
    sess = Session(c, [ld])
    qs = W.QueryStream(c)
    wts = W.head_weights(c, ld.w)
    ins = []
    for _ in range(args.warmup + 4 * K):
        _, enc, qm = qs.next()
        ins.append(sess.device_inputs(enc, wts, qm))
    apps = [sess.append_inputs(*W.appended_token(c, ld, i)) for i in range(n_app)]
    del ld
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nq = na = 0

    def block(n, append, step):
        nonlocal nq, na
        torch.cuda.synchronize()
        e0.record(st)
        for _ in range(n):
            if append:
                ess.ess_append(sess.pool, 0, *apps[na], st)
                na += 1
            if step:
                qd, wd, qmd = ins[nq]
                nq += 1
                ess.ess_step(sess.pool, 0, qd, wd, qmd, sess.out, st)
        e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n

    block(args.warmup, False, True)
    runs = {"with_append": [], "without_append": []}
    for _ in range(2):
        runs["with_append"].append(block(K, True, True))
        runs["without_append"].append(block(K, False, True))
    alone = block(K, True, False)
    assert sess.poll(st) == ess.ESS_OK
    sess.close()
    units = cfg.batch * cfg.mtp
    mean = {m: sum(v) / len(v) for m, v in runs.items()}
    line = {"append": {"workload": cfg.name, "steps_per_block": K, "warmup": args.warmup,
                       "T_start": cfg.T, "tokens_appended_per_request": na,
                       "timing": "CUDA events on the launching stream around each block",
                       "with_append_us_per_step": runs["with_append"],
                       "without_append_us_per_step": runs["without_append"],
                       "append_kernel_alone_us": alone,
                       "with_append_token_layers_per_s": units / (mean["with_append"] * 1e-6),
                       "without_append_token_layers_per_s":
                           units / (mean["without_append"] * 1e-6)}}
    print(json.dumps(line), flush=True)
    return 0


def prefill_bench(args):
    """The prefill four-buffer engine (ess_prefill_run) moving whole-layer KV:
    8 layers of one request of 65536 tokens (1152-byte latent rows, 75.5 MB a
    layer) in pinned host memory, B0 + 3 rotating device buffers, the page's
    Figure 3 prefetch map, and a per-layer compute (a bf16 matmul loop on the
    compute stream standing in for the layer's prefill) sized near the load
    time.  Timed with CUDA events: one layer's H2D, D2H and compute alone, the
    engine's pass, and the same work serialised on one stream.  A pass is no
    shorter than its busiest stream; the FlashOffloading analysis ("prefill
    side") bounds each exposed load by max(0, tau_H2D - d_on * tau_compute)."""
    import torch
    from host_latent_cache_gb300 import ess
    ess.load()
    L, rows = 8, 65536
    layer_bytes = rows * ROW_BYTES
    host = [None] + [ess.HostBuffer((layer_bytes,), np.uint8) for _ in range(1, L)]
    for h in host[1:]:
        h.array[::4096] = 1
    bufs = [torch.zeros(layer_bytes, dtype=torch.uint8, device="cuda") for _ in range(4)]
    cs, hs, ds = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    n = 4096
    a = torch.randn(n, n, device="cuda", dtype=torch.bfloat16)
    bmat = torch.randn(n, n, device="cuda", dtype=torch.bfloat16)
    reps = [1]

    def work():
        for _ in range(reps[0]):
            torch.mm(a, bmat)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def timed(stream, fn, k=3):
        fn()
        torch.cuda.synchronize()
        e0, e1 = ev(), ev()
        with torch.cuda.stream(stream):
            e0.record()
            for _ in range(k):
                fn()
            e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / k * 1e3

    hb0 = torch.from_numpy(host[1].array)
    t_h2d = timed(hs, lambda: bufs[1].copy_(hb0, non_blocking=True))
    t_d2h = timed(ds, lambda: hb0.copy_(bufs[1], non_blocking=True))
    t_mm = timed(cs, lambda: torch.mm(a, bmat))
    reps[0] = max(1, int(round(t_h2d / t_mm)))
    t_c = timed(cs, work)

    def compute(layer, buf_ptr, stream_ptr):
        with torch.cuda.stream(torch.cuda.ExternalStream(stream_ptr)):
            work()

    omap = [-1, 4, 5, 6, 7, -1, -1, -1]
    res = {}
    for shared in (False, True):
        m = omap if not shared else [-1, -1, 4, 5, 6, 7, -1, -1]
        for _ in range(2):                               # warm-up, then timed
            torch.cuda.synchronize()
            e0, e1 = ev(), ev()
            e0.record(cs)
            ess.ess_prefill_run(m, host, layer_bytes, bufs, compute, cs, hs, ds,
                                shared_copy=shared)
            e1.record(cs)
            torch.cuda.synchronize()
        res["one_copy_stream" if shared else "three_streams"] = {
            "onload_layer_map": m, "pass_us": e0.elapsed_time(e1) * 1e3}

    def serial():
        with torch.cuda.stream(cs):
            work()                                       # layer 0 in B0
            for l in range(1, L):
                hb = torch.from_numpy(host[l].array)
                bufs[1].copy_(hb, non_blocking=True)
                work()
                hb.copy_(bufs[1], non_blocking=True)
    t_serial = timed(cs, serial, k=1)
    for h in host[1:]:
        h.close()
    line = {"prefill": {
        "layers": L, "tokens_per_layer": rows, "layer_bytes": layer_bytes, "buffers": "B0 + 3",
        "timing": "CUDA events; one layer alone, then the pass",
        "t_h2d_us": t_h2d, "t_d2h_us": t_d2h, "t_compute_us": t_c,
        "h2d_gbs": layer_bytes / (t_h2d * 1e-6) / 1e9,
        "engine": res, "serial_one_stream_us": t_serial,
        "compute_only_us": L * t_c,
        "lower_bound_us": {"three_streams": max(L * t_c, (L - 1) * t_h2d, (L - 1) * t_d2h),
                           "one_copy_stream": max(L * t_c, (L - 1) * (t_h2d + t_d2h))},
        "note": "a pass is no shorter than its busiest stream"}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    cfg = W.ALL_CONFIGS[args.workload]()
    if args.compact:
        cfg = cfg.replace(compact=True)
    if args.miss_sweep:
        return miss_sweep(args, cfg) if rank == 0 else 0
    if args.pipeline:
        return pipeline_bench(args, cfg) if rank == 0 else 0
    if args.append:
        return append_bench(args, cfg) if rank == 0 else 0
    if args.prefill:
        return prefill_bench(args) if rank == 0 else 0
    if args.impl == "reference":
        return bench_reference(args, cfg, rank, world)
    result, ld = bench_ours(args, cfg, rank, world, local_rank)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            n_req = min(cfg.batch, 8)
            v, t = run_oracle(cfg, ld, max(1, args.cpu_steps), n_req)
            result["cpu_baseline"] = {
                "value": v, "unit": UNIT, "cores": _CORES, "cpu": cpu_model(), "kind": "oracle",
                "sample": f"{n_req} requests x {args.cpu_steps} steps of the same workload "
                          f"after one warm-up step ({t:.1f} s), float64 numpy, "
                          f"{_CORES} BLAS threads"}
        print(json.dumps(result), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
