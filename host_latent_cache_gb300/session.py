"""Device memory and bindings for one pool (PyTorch is used for memory and
streams only; every step of the decode path runs in the CUDA library).

A Session owns the workspace tensor, the per-layer indexer cache on the
device, the pinned host latent cache and the pool handle, and offers the
per-step calls with torch tensors.
"""
from __future__ import annotations

from typing import List, Optional

import numpy as np
import torch

from . import ess
from . import workloads as W


def ess_config_of(cfg: W.WorkloadConfig, miss_mode: int = ess.ESS_MISS_FUSED,
                  n_layers: Optional[int] = None, batch: Optional[int] = None) -> ess.ess_config:
    return ess.make_config(
        n_layers=n_layers or cfg.layers, batch=batch or cfg.batch, max_T=W.t_max_of(cfg), C=cfg.C,
        k=cfg.k, mtp=cfg.mtp, idx_heads=cfg.idx_heads, idx_dim=cfg.idx_dim,
        idx_dtype=ess.ESS_FP8_E4M3 if cfg.idx_dtype == W.FP8_E4M3 else ess.ESS_BF16,
        mla_heads=cfg.mla_heads, sm_scale=cfg.sm_scale, page=cfg.page, miss_mode=miss_mode)


class Session:
    def __init__(self, cfg: W.WorkloadConfig, layers: List[W.LayerData],
                 miss_mode: int = ess.ESS_MISS_FUSED, device: str = "cuda",
                 host_buffers: Optional[List["ess.HostBuffer"]] = None):
        """host_buffers: latent caches already in host memory (one per layer),
        shared with another session; by default each layer gets its own."""
        ess.load()
        self.cfg = cfg
        self.device = torch.device(device)
        self.ecfg = ess_config_of(cfg, miss_mode, n_layers=len(layers))
        nbytes = ess.ess_pool_device_bytes(self.ecfg)
        self.workspace = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.workspace.data_ptr()) % 256
        self.ws_view = self.workspace[off:off + nbytes]
        self.pool = ess.ess_pool_create(self.ecfg, self.ws_view)
        self.keys, self.scale, self.pages, self.host, self.T = [], [], [], [], []
        self._own_host = []
        for l, ld in enumerate(layers):
            keys = torch.from_numpy(ld.idx_keys).to(self.device)
            scale = torch.from_numpy(ld.idx_scale).to(self.device)
            pages = torch.from_numpy(ld.page_table).to(self.device)
            if host_buffers is not None:
                host = host_buffers[l]
            else:
                host = ess.HostBuffer(ld.host_latent.shape, ld.host_latent.dtype)
                host.array[...] = ld.host_latent
                self._own_host.append(host)
            T = torch.from_numpy(ld.T.astype(np.int32))
            bind = ess.ess_pool_bind_layer_compact if cfg.compact else ess.ess_pool_bind_layer
            bind(self.pool, l, host, pages, keys, scale, T)
            self.keys.append(keys)
            self.scale.append(scale)
            self.pages.append(pages)
            self.host.append(host)
            self.T.append(T)
        B, M, k = cfg.batch, cfg.mtp, cfg.k
        dev = self.device
        self.topk_idx = torch.zeros((B, M, k), dtype=torch.int32, device=dev)
        self.topk_slot = torch.zeros((B, M, k), dtype=torch.int32, device=dev)
        self.n_miss_way = torch.zeros((B, M), dtype=torch.int32, device=dev)
        self.miss_tok = torch.zeros((B, M * k), dtype=torch.int32, device=dev)
        self.miss_slot = torch.zeros((B, M * k), dtype=torch.int32, device=dev)
        self.n_miss = torch.zeros((B,), dtype=torch.int32, device=dev)
        self.scores = torch.zeros((B, M, W.t_max_of(cfg)), dtype=torch.float32, device=dev)
        self.out = torch.zeros((B, M, cfg.mla_heads, 512), dtype=torch.float32, device=dev)

    # -------------------------------------------------------------- inputs
    def device_inputs(self, q_enc: np.ndarray, w: np.ndarray, q_mla: np.ndarray):
        q = torch.from_numpy(np.ascontiguousarray(q_enc).view(np.uint8)).to(self.device)
        wt = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).to(self.device)
        qm = torch.from_numpy(np.ascontiguousarray(q_mla).view(np.int16)).to(self.device)
        return q, wt, qm

    def append_inputs(self, latent_rows: np.ndarray, key_rows: np.ndarray, scales: np.ndarray):
        """Device copies of one decode append's inputs (see W.appended_token)."""
        lat = torch.from_numpy(np.ascontiguousarray(latent_rows).view(np.int16)).to(self.device)
        key = torch.from_numpy(np.ascontiguousarray(key_rows)).to(self.device)
        sc = torch.from_numpy(np.ascontiguousarray(scales, dtype=np.float32)).to(self.device)
        return lat, key, sc

    # -------------------------------------------------------------- calls
    def append(self, layer, latent_rows, key_rows, scales, stream=None):
        ess.ess_append(self.pool, layer, latent_rows, key_rows, scales, stream)

    def scores_only(self, layer, q, w, stream=None):
        ess.ess_indexer_scores(self.pool, layer, q, w, self.scores, stream)
        return self.scores

    def select(self, layer, scores, stream=None):
        ess.ess_select_manage(self.pool, layer, scores, self.topk_idx, self.topk_slot,
                              self.n_miss_way, self.miss_tok, self.miss_slot, self.n_miss, stream)

    def indexer_topk(self, layer, q, w, stream=None):
        ess.ess_indexer_topk(self.pool, layer, q, w, self.topk_idx, self.topk_slot,
                             self.n_miss_way, self.miss_tok, self.miss_slot, self.n_miss, stream)

    def stage(self, layer, stream=None):
        ess.ess_stage_misses(self.pool, layer, self.miss_tok, self.miss_slot, self.n_miss, stream)

    def attention(self, layer, q_mla, out=None, stream=None):
        out = self.out if out is None else out
        ess.ess_sparse_mla_decode(self.pool, layer, q_mla, self.topk_idx, self.topk_slot, out,
                                  stream)
        return out

    def step(self, layer, q, w, q_mla, out=None, stream=None):
        out = self.out if out is None else out
        ess.ess_step(self.pool, layer, q, w, q_mla, out, stream)
        return out

    def poll(self, stream=None) -> int:
        return ess.ess_pool_poll(self.pool, stream)

    def state(self, layer):
        B, T, C = self.cfg.batch, W.t_max_of(self.cfg), self.cfg.C
        cs = torch.empty((B, T), dtype=torch.int32)
        st = torch.empty((B, C), dtype=torch.int32)
        lu = torch.empty((B, C), dtype=torch.int32)
        sp = torch.empty((B,), dtype=torch.int32)
        ess.ess_pool_get_state(self.pool, layer, cs, st, lu, sp)
        return cs.numpy(), st.numpy(), lu.numpy(), sp.numpy()

    def set_state(self, layer, state: "W.PoolState"):
        """Start the layer from a given pool state; the rows of its resident
        tokens are reloaded from the host copy."""
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32))
        ess.ess_pool_set_state(self.pool, layer, t(state.cache_slots), t(state.slot_token),
                               t(state.last_used), t(state.step))

    def pool_rows(self, layer):
        """The hot pool of a layer as uint16 [B][C][576] (synchronous copy)."""
        rows = torch.empty((self.cfg.batch, self.cfg.C, W.ROW_DIM), dtype=torch.int16)
        ess.ess_pool_get_rows(self.pool, layer, rows)
        return rows.numpy().view(np.uint16)

    def kernel_launches(self) -> int:
        return ess.ess_pool_kernel_launches(self.pool)

    def stats(self, layer, reset=False):
        return ess.ess_pool_read_stats(self.pool, layer, reset)

    def close(self):
        if self.pool:
            ess.ess_pool_destroy(self.pool)
            self.pool = None
        for h in self._own_host:
            h.close()
        self._own_host = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
