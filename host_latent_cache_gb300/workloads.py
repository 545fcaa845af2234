"""Seeded synthetic inputs for the sparse-decode hot path.

This module only draws inputs. It holds none of the method's arithmetic
(no scores, no selection, no cache bookkeeping, no attention), so that
the CPU oracle and the CUDA path can both consume the same arrays
without sharing any computation.

Where the inputs come from (web pages on latent-cache offload for DSA
sparse decode):

* "ESS: Latent-Cache Offload" (foosynaptic tech notes), table
  "double cache and ESS division of labour": one light indexer vector per
  position, scored over the full length; the latent entry is c^KV[512]
  plus k^R[64].
* hwcomputing.csdn.net FlashOffloading analysis, section "architecture:
  one master copy, two residency policies": the host keeps the
  authoritative KV paged by (request, layer, token block) behind a block
  table.  The synthetic page table below is a seeded permutation so that
  the indirection is exercised.

Exact-score data contract (so that a tensor-core contraction can be
checked bit for bit against a float64 oracle):

* indexer query values lie on (1/8)Z within [-2, 2];
* indexer key values lie on the e4m3 values that are multiples of 1/8
  with magnitude at most 15 (79 levels, exact in e4m3 and in bf16);
* head weights lie on (1/64)Z within [0, 1);
* the per-token key scale is an arbitrary positive fp32.

Every dot product is then a multiple of 2^-6 below 2^12 in magnitude and
every weighted ReLU term a non-negative multiple of 2^-12, so all partial
sums are exact in fp32 in any order while the total stays below 4096.

Query drift: per head, q_t = normalize(rho * q_{t-1} + (1 - rho) * g),
where the state q is a unit vector and g is isotropic Gaussian noise on the
same scale, i.e. unit expected norm (per-element variance 1/d).  Read with
per-element variance 1, the noise would outweigh the unit-norm state ten to
one in 128 dims and adjacent top-2048 sets would overlap by only about a
third, against the stated intent of a high adjacent-step overlap.  The
normalised fp32 state carries over; each step's query is then scaled so
that its largest magnitude is 2 and rounded to the grid.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

# Tensor ids for the per-tensor random streams.
_TID_KEYS, _TID_QIDX, _TID_W, _TID_QMLA, _TID_LATENT, _TID_PAGES, _TID_COLD = range(1, 8)

FP8_E4M3 = 0
BF16 = 1

LATENT_DIM = 512
ROPE_DIM = 64
ROW_DIM = LATENT_DIM + ROPE_DIM  # 576 bf16 = 1152 bytes per latent row


# --------------------------------------------------------------------------
# grids of the exact-score data contract
# --------------------------------------------------------------------------

def _e4m3_value(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    if e == 0xF and m == 0x7:
        return float("nan")
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_decode_table() -> np.ndarray:
    """float64 value of every e4m3 byte (NaN for the two NaN codes)."""
    return np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def key_levels() -> tuple[np.ndarray, np.ndarray]:
    """The 79 key levels (ascending) and their e4m3 codes."""
    tab = e4m3_decode_table()
    vals, codes = [], []
    for c in range(256):
        v = tab[c]
        if np.isnan(v) or abs(v) > 15.0:
            continue
        if (v * 8.0) != np.round(v * 8.0):
            continue
        if v == 0.0 and c != 0:
            continue  # keep +0 only
        vals.append(v)
        codes.append(c)
    order = np.argsort(vals)
    return np.asarray(vals)[order], np.asarray(codes, dtype=np.uint8)[order]


_KEY_VALS, _KEY_CODES = key_levels()
assert len(_KEY_VALS) == 79


def _round_to_levels(x: np.ndarray, levels: np.ndarray) -> np.ndarray:
    """Index of the nearest level (ties to the lower level)."""
    i = np.searchsorted(levels, x, side="left")
    i = np.clip(i, 1, len(levels) - 1)
    lo = levels[i - 1]
    hi = levels[i]
    pick_lo = (x - lo) <= (hi - x)
    return np.where(pick_lo, i - 1, i)


def e4m3_encode_grid(v: np.ndarray) -> np.ndarray:
    """Encode values already on the key/query grid as e4m3 bytes."""
    idx = np.searchsorted(_KEY_VALS, v)
    idx = np.clip(idx, 0, len(_KEY_VALS) - 1)
    if not np.all(_KEY_VALS[idx] == v):
        raise ValueError("value off the e4m3 grid")
    return _KEY_CODES[idx]


def float_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_float(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# configurations
# --------------------------------------------------------------------------

@dataclass
class WorkloadConfig:
    name: str
    layers: int
    batch: int
    T: int                      # context length per request
    steps: int
    idx_heads: int
    idx_dim: int
    idx_dtype: int              # FP8_E4M3 or BF16
    k: int
    mla_heads: int
    C: int
    page: int = 64
    mtp: int = 1
    rho: float = 0.9
    cold_p: float = 0.0         # per (request, step >= 1) chance of a fresh query
    seed: int = 1000
    T_per_req: Optional[List[int]] = None   # ragged contexts (defaults to T for all)
    grow: int = 0               # tokens appended to every request, one per step
    compact: bool = False       # host latent as compact 656-byte rows (e4m3 + scales + bf16 RoPE)
    sm_scale: float = float(np.float32(1.0 / np.sqrt(576.0)))

    def t_of(self, b: int) -> int:
        return self.T if self.T_per_req is None else int(self.T_per_req[b])

    def replace(self, **kw) -> "WorkloadConfig":
        return dataclasses.replace(self, **kw)


def tiny() -> WorkloadConfig:
    return WorkloadConfig("tiny", layers=1, batch=1, T=4096, steps=8, idx_heads=4, idx_dim=64,
                          idx_dtype=BF16, k=256, mla_heads=16, C=1024, rho=0.9, seed=1001)


def v32_32k() -> WorkloadConfig:
    return WorkloadConfig("v32_32k", layers=1, batch=16, T=32768, steps=32, idx_heads=64,
                          idx_dim=128, idx_dtype=FP8_E4M3, k=2048, mla_heads=128, C=8192,
                          rho=0.95, seed=1002)


def long_128k() -> WorkloadConfig:
    return WorkloadConfig("long_128k", layers=1, batch=8, T=131072, steps=64, idx_heads=64,
                          idx_dim=128, idx_dtype=FP8_E4M3, k=2048, mla_heads=128, C=32768,
                          rho=0.9, cold_p=0.05, seed=1003)


def ctx_1m(C: int = 8192) -> WorkloadConfig:
    return WorkloadConfig(f"ctx_1m_C{C}", layers=1, batch=1, T=1 << 20, steps=64, idx_heads=64,
                          idx_dim=128, idx_dtype=FP8_E4M3, k=2048, mla_heads=128, C=C,
                          rho=0.9, seed=1004)


def multilayer() -> WorkloadConfig:
    return WorkloadConfig("multilayer", layers=8, batch=32, T=65536, steps=32, idx_heads=64,
                          idx_dim=128, idx_dtype=FP8_E4M3, k=2048, mla_heads=128, C=16384,
                          mtp=2, rho=0.95, seed=1005)


ALL_CONFIGS = {"tiny": tiny, "v32_32k": v32_32k, "long_128k": long_128k,
               "ctx_1m": ctx_1m, "multilayer": multilayer}


def _rng(seed: int, *ids: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *ids])))


# --------------------------------------------------------------------------
# static per-layer data
# --------------------------------------------------------------------------

@dataclass
class LayerData:
    """Static inputs of one layer.

    idx_keys   uint8 [B][T_max][row_bytes] (e4m3 bytes, or bf16 bits viewed as bytes);
               rows t >= T_b are zero
    idx_scale  float32 [B][T_max]   (all ones for bf16 keys; 1 for t >= T_b)
    w          float32 [B][H_I]     head weights, on (1/64)Z in [0, 1)
    latent     uint16 [B][T_max][576] bf16 bits, LOGICAL token order
    host_latent uint16 [B][T_max][576] bf16 bits, page-permuted host layout
    page_table int32 [B][T_max / page]
    T          int32 [B]
    With cfg.grow > 0 (decode append) the rows of the tokens appended later
    are held apart: their keys in app_keys [B][grow][row_bytes] and
    app_scale [B][grow]; latent holds them in logical order; host_latent has
    zeros there (the library writes them back as their pages complete).
    """
    idx_keys: np.ndarray
    idx_scale: np.ndarray
    w: np.ndarray
    latent: np.ndarray
    host_latent: np.ndarray
    page_table: np.ndarray
    T: np.ndarray
    app_keys: Optional[np.ndarray] = None
    app_scale: Optional[np.ndarray] = None
    latent_c: Optional[np.ndarray] = None   # compact rows uint8 [B][T_max][656], logical order


def t_max_of(cfg: WorkloadConfig) -> int:
    tm = max(cfg.t_of(b) + cfg.grow for b in range(cfg.batch))
    tm = max(tm, 1)
    return ((tm + cfg.page - 1) // cfg.page) * cfg.page


def gen_keys(cfg: WorkloadConfig, layer: int, b: int, T_max: int):
    """Keys of one request: (bytes [T_max][row_bytes], scale [T_max])."""
    rng = _rng(cfg.seed, _TID_KEYS, layer, b)
    T = cfg.t_of(b) + cfg.grow      # rows that ever hold a token
    d = cfg.idx_dim
    x = rng.standard_normal((T_max, d), dtype=np.float32)
    if cfg.idx_dtype == FP8_E4M3:
        amax = np.max(np.abs(x), axis=1)
        scale = (amax / np.float32(15.0)).astype(np.float32)
        scale = np.maximum(scale, np.float32(1e-30))
        v = x / scale[:, None]
        lv = _KEY_VALS[_round_to_levels(v.astype(np.float64), _KEY_VALS)]
        codes = e4m3_encode_grid(lv)
        out = codes.reshape(T_max, d)
    else:
        lv = _KEY_VALS[_round_to_levels(x.astype(np.float64), _KEY_VALS)]
        bits = float_to_bf16_bits(lv.astype(np.float32)).reshape(T_max, d)
        out = bits.view(np.uint8).reshape(T_max, 2 * d)
        scale = np.ones(T_max, dtype=np.float32)
    if T < T_max:
        out = out.copy()
        out[T:] = 0
        scale = scale.copy()
        scale[T:] = 1.0
    return np.ascontiguousarray(out), scale.astype(np.float32)


def gen_layer(cfg: WorkloadConfig, layer: int = 0, want_latent: bool = True) -> LayerData:
    B = cfg.batch
    T_max = t_max_of(cfg)
    rb = cfg.idx_dim * (1 if cfg.idx_dtype == FP8_E4M3 else 2)
    keys = np.zeros((B, T_max, rb), dtype=np.uint8)
    scale = np.ones((B, T_max), dtype=np.float32)
    w = np.zeros((B, cfg.idx_heads), dtype=np.float32)
    npages = T_max // cfg.page
    pages = np.zeros((B, npages), dtype=np.int32)
    latent = np.zeros((B, T_max, ROW_DIM), dtype=np.uint16) if want_latent else None
    host = np.zeros((B, T_max, ROW_DIM), dtype=np.uint16) if want_latent else None
    for b in range(B):
        keys[b], scale[b] = gen_keys(cfg, layer, b, T_max)
        rw = _rng(cfg.seed, _TID_W, layer, b)
        w[b] = np.floor(rw.random(cfg.idx_heads) * 64.0) / 64.0
        rp = _rng(cfg.seed, _TID_PAGES, layer, b)
        pages[b] = rp.permutation(npages).astype(np.int32)
        if want_latent:
            rl = _rng(cfg.seed, _TID_LATENT, layer, b)
            x = rl.standard_normal((T_max, ROW_DIM), dtype=np.float32) * np.float32(0.5)
            latent[b] = float_to_bf16_bits(x).reshape(T_max, ROW_DIM)
            # physical row p holds logical token t with p = pages[t // page] * page + t % page
            t = np.arange(T_max)
            phys = pages[b][t // cfg.page] * cfg.page + (t % cfg.page)
            host[b][phys] = latent[b]
    Ts = np.array([cfg.t_of(b) for b in range(B)], dtype=np.int32)
    if cfg.compact:
        if cfg.grow:
            raise ValueError("compact host rows take no appends")
        latent_c, host = gen_compact_latent(cfg, layer, pages) if want_latent else (None, None)
        return LayerData(keys, scale, w, None, host, pages, Ts, None, None, latent_c)
    app_keys = app_scale = None
    if cfg.grow > 0:
        app_keys = np.zeros((B, cfg.grow, rb), dtype=np.uint8)
        app_scale = np.ones((B, cfg.grow), dtype=np.float32)
        for b in range(B):
            T = int(Ts[b])
            app_keys[b] = keys[b, T:T + cfg.grow]
            app_scale[b] = scale[b, T:T + cfg.grow]
            keys[b, T:] = 0
            scale[b, T:] = 1.0
            if want_latent:
                t = np.arange(T, T_max)
                host[b][pages[b][t // cfg.page] * cfg.page + t % cfg.page] = 0
    return LayerData(keys, scale, w, latent, host, pages, Ts, app_keys, app_scale)


_TID_STATE = 8
_TID_COMPACT = 9
COMPACT_ROW_BYTES = 656


@dataclass
class PoolState:
    """A hot-pool state to start from (one layer): cache_slots [B][T_max],
    slot_token [B][C], last_used [B][C] int32 and step [B] int32."""
    cache_slots: np.ndarray
    slot_token: np.ndarray
    last_used: np.ndarray
    step: np.ndarray


def full_pool_state(cfg: WorkloadConfig, ld: LayerData, layer: int = 0,
                    age: int = 8) -> PoolState:
    """A pool that has been running for `age` steps and is full: every
    request holds min(C, T_b) distinct tokens drawn at random, in random
    slots, each last used at a random earlier step in [0, age) (so many slots
    share a stamp), and the step counter stands at `age`.  Empty slots (when
    T_b < C) keep token -1 and stamp -1.  A draw of inputs only: which slots
    a step evicts from it is left to the code under test."""
    B, C, Tm = cfg.batch, cfg.C, t_max_of(cfg)
    cs = np.full((B, Tm), -1, np.int32)
    st = np.full((B, C), -1, np.int32)
    lu = np.full((B, C), -1, np.int32)
    sp = np.full(B, age, np.int32)
    for b in range(B):
        r = _rng(cfg.seed, _TID_STATE, layer, b)
        Tb = int(ld.T[b])
        n = min(C, Tb)
        toks = r.choice(Tb, size=n, replace=False).astype(np.int32)
        slots = r.permutation(C)[:n].astype(np.int32)
        st[b, slots] = toks
        cs[b, toks] = slots
        lu[b, slots] = r.integers(0, age, size=n).astype(np.int32)
    return PoolState(cs, st, lu, sp)


def gen_compact_latent(cfg: WorkloadConfig, layer: int, pages: np.ndarray):
    """Compact latent rows drawn directly in their stored form (logical order,
    and the page-permuted host copy): per token, 512 e4m3 codes (a random
    sign and a magnitude code uniform over the finite codes 0x00..0x7E, i.e.
    values spread log-uniformly from 2^-9 to 448), four tile scales 2^-9,
    2^-8 or 2^-7, and 64 RoPE values bf16 N(0, 0.5)."""
    B, Tm, page = cfg.batch, t_max_of(cfg), cfg.page
    lat = np.zeros((B, Tm, COMPACT_ROW_BYTES), dtype=np.uint8)
    host = np.zeros_like(lat)
    for b in range(B):
        r = _rng(cfg.seed, _TID_COMPACT, layer, b)
        mag = r.integers(0, 0x7F, size=(Tm, 512), dtype=np.uint8)
        sign = (r.integers(0, 2, size=(Tm, 512), dtype=np.uint8) << np.uint8(7)).astype(np.uint8)
        lat[b, :, :512] = mag | sign
        sc = np.ldexp(np.float32(1.0), r.integers(-9, -6, size=(Tm, 4))).astype("<f4")
        lat[b, :, 512:528] = sc.view(np.uint8).reshape(Tm, 16)
        rope = r.standard_normal((Tm, ROPE_DIM), dtype=np.float32) * np.float32(0.5)
        lat[b, :, 528:] = float_to_bf16_bits(rope).reshape(Tm, ROPE_DIM).astype("<u2").view(
            np.uint8).reshape(Tm, 2 * ROPE_DIM)
        t = np.arange(Tm)
        host[b][pages[b][t // page] * page + t % page] = lat[b]
    return lat, host


def appended_token(cfg: WorkloadConfig, ld: LayerData, i: int):
    """Inputs of the i-th decode append (token T_b + i of each request):
    latent rows uint16 [B][576], key rows uint8 [B][row_bytes], scales
    float32 [B]."""
    B = cfg.batch
    lat = np.stack([ld.latent[b, int(ld.T[b]) + i] for b in range(B)])
    return (np.ascontiguousarray(lat), np.ascontiguousarray(ld.app_keys[:, i]),
            np.ascontiguousarray(ld.app_scale[:, i]))


def append_ragged() -> WorkloadConfig:
    """Decode with appends: two ragged requests whose first pages are
    partial, growing by 150 tokens (several pages complete and leave the
    two-page ring)."""
    return WorkloadConfig("append_ragged", layers=1, batch=2, T=4000, steps=150, idx_heads=4,
                          idx_dim=64, idx_dtype=BF16, k=256, mla_heads=16, C=1024, rho=0.9,
                          seed=1006, T_per_req=[4000, 2500], grow=150)


def append_fp8() -> WorkloadConfig:
    """Decode with appends on the FP8 indexer and 128 MLA heads."""
    return WorkloadConfig("append_fp8", layers=1, batch=2, T=3000, steps=140, idx_heads=64,
                          idx_dim=128, idx_dtype=FP8_E4M3, k=512, mla_heads=128, C=1024,
                          rho=0.9, seed=1007, T_per_req=[3000, 2100], grow=140)


# --------------------------------------------------------------------------
# per-step queries
# --------------------------------------------------------------------------

class QueryStream:
    """Drifting indexer queries and fresh MLA queries, step by step.

    Yields for each step: q_idx (grid values, float32 [B][M][H_I][d_I]) and
    its device encoding (e4m3 bytes or bf16 bits), and q_mla (bf16 bits
    [B][M][H][576]).
    """

    def __init__(self, cfg: WorkloadConfig, layer: int = 0):
        self.cfg = cfg
        self.layer = layer
        self.step = 0
        B, H, d = cfg.batch, cfg.idx_heads, cfg.idx_dim
        self._rng = [_rng(cfg.seed, _TID_QIDX, layer, b) for b in range(B)]
        self._cold = [_rng(cfg.seed, _TID_COLD, layer, b) for b in range(B)]
        self._mla = _rng(cfg.seed, _TID_QMLA, layer)
        self.state = np.zeros((B, H, d), dtype=np.float32)
        for b in range(B):
            self.state[b] = self._normalize(self._rng[b].standard_normal((H, d), dtype=np.float32))

    @staticmethod
    def _normalize(x: np.ndarray) -> np.ndarray:
        n = np.sqrt(np.sum(x.astype(np.float64) ** 2, axis=-1, keepdims=True))
        n = np.maximum(n, 1e-30)
        return (x / n).astype(np.float32)

    @staticmethod
    def _to_grid(q: np.ndarray) -> np.ndarray:
        """Scale so that max |q| = 2, round to (1/8)Z, clip to [-2, 2]."""
        amax = float(np.max(np.abs(q)))
        s = 2.0 / amax if amax > 0 else 1.0
        g = np.round(q.astype(np.float64) * s * 8.0) / 8.0
        return np.clip(g, -2.0, 2.0).astype(np.float32)

    def next(self):
        cfg = self.cfg
        B, M, H, d = cfg.batch, cfg.mtp, cfg.idx_heads, cfg.idx_dim
        rho = np.float32(cfg.rho)
        q = np.zeros((B, M, H, d), dtype=np.float32)
        for b in range(B):
            r = self._rng[b]
            if self.step > 0:
                g = r.standard_normal((H, d), dtype=np.float32) * np.float32(1.0 / np.sqrt(d))
                cold = cfg.cold_p > 0 and self._cold[b].random() < cfg.cold_p
                if cold:
                    self.state[b] = self._normalize(g)
                else:
                    self.state[b] = self._normalize(rho * self.state[b] + (np.float32(1) - rho) * g)
            ways = [self.state[b]]
            for m in range(1, M):
                g = r.standard_normal((H, d), dtype=np.float32) * np.float32(1.0 / np.sqrt(d))
                ways.append(self._normalize(rho * ways[-1] + (np.float32(1) - rho) * g))
            for m in range(M):
                q[b, m] = self._to_grid(ways[m])
        q_mla_f = self._mla.standard_normal((B, M, cfg.mla_heads, ROW_DIM), dtype=np.float32)
        q_mla = float_to_bf16_bits(q_mla_f * np.float32(0.5)).reshape(B, M, cfg.mla_heads, ROW_DIM)
        self.step += 1
        return q, encode_query(cfg, q), q_mla


def encode_query(cfg: WorkloadConfig, q: np.ndarray) -> np.ndarray:
    """Device bytes of grid-valued indexer queries: [B][M][H_I][row_bytes]."""
    if cfg.idx_dtype == FP8_E4M3:
        return e4m3_encode_grid(q.reshape(-1)).reshape(q.shape)
    bits = float_to_bf16_bits(q.reshape(-1)).reshape(q.shape)
    return bits.view(np.uint8).reshape(*q.shape[:-1], 2 * q.shape[-1])


def decode_keys(cfg: WorkloadConfig, keys: np.ndarray) -> np.ndarray:
    """Grid values (float64) of stored key bytes [..][row_bytes]."""
    if cfg.idx_dtype == FP8_E4M3:
        return e4m3_decode_table()[keys]
    bits = np.ascontiguousarray(keys).view(np.uint16)
    return bf16_bits_to_float(bits).astype(np.float64)


def head_weights(cfg: WorkloadConfig, layer_w: np.ndarray) -> np.ndarray:
    """Per-call head weights [B][M][H_I] (the same weights for every way)."""
    return np.ascontiguousarray(np.repeat(layer_w[:, None, :], cfg.mtp, axis=1)).astype(np.float32)
