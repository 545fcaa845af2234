"""Python binding of the C ABI in include/ess.h (argument marshalling only).

Every compute step runs in the CUDA library; this module converts torch
tensors to pointers and checks status codes.  Importing it needs no GPU;
loading the library does, and fails loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_lib", "libess.so")

ESS_OK = 0
ESS_ERR_INVALID_ARG = 1
ESS_ERR_CAPACITY = 2
ESS_ERR_UNSUPPORTED = 3
ESS_ERR_OOM = 4
ESS_ERR_CUDA = 5
ESS_ERR_TIMEOUT = 6
ESS_ERR_DEVICE_CHECK = 7

ESS_FP8_E4M3 = 0
ESS_BF16 = 1

ESS_EVICT_LRU, ESS_EVICT_RANDOM, ESS_EVICT_SCORE, ESS_EVICT_LIM = range(4)
ESS_MISS_FUSED = 0
ESS_MISS_STAGED = 1

# every exported symbol of include/ess.h
EXPORTS = (
    "ess_status_string", "ess_host_alloc", "ess_host_free", "ess_pool_device_bytes",
    "ess_pool_create", "ess_pool_destroy",
    "ess_pool_bind_layer", "ess_pool_reset", "ess_append", "ess_indexer_scores",
    "ess_select_manage",
    "ess_select_manage_noalloc",
    "ess_indexer_topk", "ess_stage_misses", "ess_sparse_mla_decode", "ess_step",
    "ess_step_profiled", "ess_step_host",
    "ess_pipeline_step", "ess_pool_get_state", "ess_pool_set_state", "ess_pool_get_rows",
    "ess_pool_read_stats", "ess_pool_poll", "ess_pool_kernel_launches", "ess_prefill_plan",
    "ess_compact_rows", "ess_replay_misses", "ess_host_gather", "ess_pool_set_eviction",
    "ess_pool_bind_layer_compact", "ess_prefill_run",
)

# void (*)(void* user, int32_t layer, void* buffer, void* stream)
PREFILL_COMPUTE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                      ctypes.c_void_p)


class ess_config(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("batch", ctypes.c_int32), ("max_T", ctypes.c_int32),
        ("C", ctypes.c_int32), ("page", ctypes.c_int32), ("k", ctypes.c_int32),
        ("mtp", ctypes.c_int32), ("idx_heads", ctypes.c_int32), ("idx_dim", ctypes.c_int32),
        ("idx_dtype", ctypes.c_int32), ("mla_heads", ctypes.c_int32),
        ("latent_dim", ctypes.c_int32), ("rope_dim", ctypes.c_int32),
        ("sm_scale", ctypes.c_float), ("miss_mode", ctypes.c_int32),
    ]


class ess_stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("hits", ctypes.c_int64), ("misses", ctypes.c_int64),
                ("union_size", ctypes.c_int64), ("miss_rows", ctypes.c_int64),
                ("miss_bytes", ctypes.c_int64), ("guided", ctypes.c_int64),
                ("fine_cuts", ctypes.c_int64)]


class EssError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libess.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.ess_status_string.restype = ctypes.c_char_p
    lib.ess_status_string.argtypes = [I]
    sigs = {
        "ess_host_alloc": [ctypes.c_size_t, ctypes.POINTER(P)],
        "ess_host_free": [P],
        "ess_pool_device_bytes": [ctypes.POINTER(ess_config), ctypes.POINTER(ctypes.c_size_t)],
        "ess_pool_create": [ctypes.POINTER(ess_config), P, ctypes.c_size_t, ctypes.POINTER(P)],
        "ess_pool_destroy": [P],
        "ess_pool_bind_layer": [P, I, P, P, P, P, P],
        "ess_pool_reset": [P, I, P],
        "ess_append": [P, I, P, P, P, P],
        "ess_indexer_scores": [P, I, P, P, P, P],
        "ess_select_manage": [P, I, P, P, P, P, P, P, P, P],
        "ess_select_manage_noalloc": [P, I, P, P, P, P, P, P, P, P],
        "ess_indexer_topk": [P, I, P, P, P, P, P, P, P, P, P],
        "ess_stage_misses": [P, I, P, P, P, P],
        "ess_sparse_mla_decode": [P, I, P, P, P, P, P],
        "ess_step": [P, I, P, P, P, P, P],
        "ess_step_profiled": [P, I, P, P, P, P, P, P],
        "ess_step_host": [P, I, P, P, P, P, P],
        "ess_pipeline_step": [P, I, I, P, P, P, P, P],
        "ess_pool_get_state": [P, I, P, P, P, P],
        "ess_pool_set_state": [P, I, P, P, P, P],
        "ess_pool_get_rows": [P, I, P],
        "ess_pool_read_stats": [P, I, ctypes.POINTER(ess_stats), I],
        "ess_pool_poll": [P, P],
        "ess_pool_kernel_launches": [P, ctypes.POINTER(ctypes.c_int64)],
        "ess_prefill_plan": [I, P, I, I, P, P, P],
        "ess_compact_rows": [P, ctypes.c_int64, P],
        "ess_replay_misses": [I, I, P, P, P, I, I, I, ctypes.c_uint64, ctypes.c_int64, P, P],
        "ess_host_gather": [P, ctypes.c_int64, I, P, ctypes.c_int64, P, P, P],
        "ess_pool_set_eviction": [P, I, ctypes.c_uint64],
        "ess_pool_bind_layer_compact": [P, I, P, P, P, P, P],
        "ess_prefill_run": [I, P, I, I, P, ctypes.c_size_t, ctypes.c_size_t, ctypes.c_size_t, P,
                            PREFILL_COMPUTE_FN, P, P, P, P],
    }
    for name, args in sigs.items():
        f = getattr(lib, name)
        f.restype = I
        f.argtypes = args
    _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load().ess_status_string(code).decode()
    except Exception:
        return f"status {code}"


def check(code: int, where: str) -> None:
    if code != ESS_OK:
        raise EssError(code, where)


def _p(t) -> Optional[int]:
    """Device/host address of a torch tensor (None -> NULL)."""
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class HostBuffer:
    """Pinned, device-mapped host memory from ess_host_alloc, exposed as a
    numpy array; freed with close()."""

    def __init__(self, shape, dtype):
        import numpy as np
        self.dtype = np.dtype(dtype)
        self.shape = tuple(int(x) for x in shape)
        n = int(np.prod(self.shape)) * self.dtype.itemsize
        p = ctypes.c_void_p(0)
        check(load().ess_host_alloc(max(n, 1), ctypes.byref(p)), "ess_host_alloc")
        self.ptr = p.value
        self.nbytes = n
        buf = (ctypes.c_char * max(n, 1)).from_address(self.ptr)
        self.array = np.frombuffer(buf, dtype=self.dtype, count=n // self.dtype.itemsize).reshape(self.shape)

    def data_ptr(self):
        return self.ptr

    def close(self):
        if self.ptr:
            self.array = None
            check(load().ess_host_free(self.ptr), "ess_host_free")
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def make_config(*, n_layers, batch, max_T, C, k, mtp, idx_heads, idx_dim, idx_dtype, mla_heads,
                sm_scale, page=64, miss_mode=ESS_MISS_FUSED, latent_dim=512,
                rope_dim=64) -> ess_config:
    return ess_config(n_layers, batch, max_T, C, page, k, mtp, idx_heads, idx_dim, idx_dtype,
                      mla_heads, latent_dim, rope_dim, float(sm_scale), miss_mode)


def ess_pool_device_bytes(cfg: ess_config) -> int:
    n = ctypes.c_size_t(0)
    check(load().ess_pool_device_bytes(ctypes.byref(cfg), ctypes.byref(n)), "ess_pool_device_bytes")
    return n.value


def ess_pool_create(cfg: ess_config, workspace) -> int:
    h = ctypes.c_void_p(0)
    check(load().ess_pool_create(ctypes.byref(cfg), _p(workspace), workspace.numel() *
                                 workspace.element_size(), ctypes.byref(h)), "ess_pool_create")
    return h.value


def ess_pool_destroy(pool: int) -> None:
    check(load().ess_pool_destroy(pool), "ess_pool_destroy")


def ess_pool_bind_layer(pool, layer, host_latent, page_table, idx_keys, idx_scale, T_host) -> None:
    check(load().ess_pool_bind_layer(pool, layer, _p(host_latent), _p(page_table), _p(idx_keys),
                                     _p(idx_scale), _p(T_host)), "ess_pool_bind_layer")


def ess_pool_bind_layer_compact(pool, layer, host_compact, page_table, idx_keys, idx_scale,
                                T_host) -> None:
    check(load().ess_pool_bind_layer_compact(pool, layer, _p(host_compact), _p(page_table),
                                             _p(idx_keys), _p(idx_scale), _p(T_host)),
          "ess_pool_bind_layer_compact")


def ess_pool_reset(pool, layer, stream=None) -> None:
    check(load().ess_pool_reset(pool, layer, _stream(stream)), "ess_pool_reset")


def ess_append(pool, layer, latent_row, key_row, key_scale, stream=None) -> None:
    check(load().ess_append(pool, layer, _p(latent_row), _p(key_row), _p(key_scale),
                            _stream(stream)), "ess_append")


def ess_indexer_scores(pool, layer, q_idx, w, scores, stream=None) -> None:
    check(load().ess_indexer_scores(pool, layer, _p(q_idx), _p(w), _p(scores), _stream(stream)),
          "ess_indexer_scores")


def ess_select_manage(pool, layer, scores, topk_idx, topk_slot, n_miss_way, miss_tok, miss_slot,
                      n_miss, stream=None) -> None:
    check(load().ess_select_manage(pool, layer, _p(scores), _p(topk_idx), _p(topk_slot),
                                   _p(n_miss_way), _p(miss_tok), _p(miss_slot), _p(n_miss),
                                   _stream(stream)), "ess_select_manage")


def ess_select_manage_noalloc(pool, layer, scores, topk_idx, topk_slot, n_miss_way, miss_tok,
                              miss_slot, n_miss, stream=None) -> None:
    """ess_select_manage with its scratch in the library's fixed device array
    (for callers that cannot provide device scratch)."""
    check(load().ess_select_manage_noalloc(pool, layer, _p(scores), _p(topk_idx), _p(topk_slot),
                                           _p(n_miss_way), _p(miss_tok), _p(miss_slot),
                                           _p(n_miss), _stream(stream)),
          "ess_select_manage_noalloc")


def ess_indexer_topk(pool, layer, q_idx, w, topk_idx, topk_slot, n_miss_way, miss_tok, miss_slot,
                     n_miss, stream=None) -> None:
    check(load().ess_indexer_topk(pool, layer, _p(q_idx), _p(w), _p(topk_idx), _p(topk_slot),
                                  _p(n_miss_way), _p(miss_tok), _p(miss_slot), _p(n_miss),
                                  _stream(stream)), "ess_indexer_topk")


def ess_stage_misses(pool, layer, miss_tok, miss_slot, n_miss, stream=None) -> None:
    check(load().ess_stage_misses(pool, layer, _p(miss_tok), _p(miss_slot), _p(n_miss),
                                  _stream(stream)), "ess_stage_misses")


def ess_sparse_mla_decode(pool, layer, q_mla, topk_idx, topk_slot, out, stream=None) -> None:
    check(load().ess_sparse_mla_decode(pool, layer, _p(q_mla), _p(topk_idx), _p(topk_slot),
                                       _p(out), _stream(stream)), "ess_sparse_mla_decode")


def ess_step(pool, layer, q_idx, w, q_mla, out, stream=None) -> None:
    check(load().ess_step(pool, layer, _p(q_idx), _p(w), _p(q_mla), _p(out), _stream(stream)),
          "ess_step")


def ess_step_profiled(pool, layer, q_idx, w, q_mla, out, events, stream=None) -> None:
    """events: four torch.cuda.Event (or None) recorded between the phases."""
    hs = [None if e is None else e.cuda_event for e in events]
    arr = (ctypes.c_void_p * 4)(*hs)
    check(load().ess_step_profiled(pool, layer, _p(q_idx), _p(w), _p(q_mla), _p(out),
                                   _stream(stream), arr), "ess_step_profiled")


def ess_step_host(pool, layer, q_idx, w, q_mla, out, stream=None) -> None:
    check(load().ess_step_host(pool, layer, _p(q_idx), _p(w), _p(q_mla), _p(out),
                               _stream(stream)), "ess_step_host")


def ess_pipeline_step(pools: Sequence[int], n_layers: int, q_idx, w, q_mla, out, streams) -> None:
    n = len(pools)
    arr = lambda xs, T=ctypes.c_void_p: (T * len(xs))(*xs)
    check(load().ess_pipeline_step(arr(list(pools)), n, n_layers, arr([_p(x) for x in q_idx]),
                                   arr([_p(x) for x in w]), arr([_p(x) for x in q_mla]),
                                   arr([_p(x) for x in out]), arr([_stream(s) for s in streams])),
          "ess_pipeline_step")


def ess_pool_get_state(pool, layer, cache_slots, slot_token, last_used, step) -> None:
    check(load().ess_pool_get_state(pool, layer, _p(cache_slots), _p(slot_token), _p(last_used),
                                    _p(step)), "ess_pool_get_state")


def ess_pool_set_state(pool, layer, cache_slots, slot_token, last_used, step) -> None:
    check(load().ess_pool_set_state(pool, layer, _p(cache_slots), _p(slot_token), _p(last_used),
                                    _p(step)), "ess_pool_set_state")


def ess_pool_get_rows(pool, layer, rows_host) -> None:
    check(load().ess_pool_get_rows(pool, layer, _p(rows_host)), "ess_pool_get_rows")


def ess_pool_read_stats(pool, layer, reset: bool = False) -> ess_stats:
    s = ess_stats()
    check(load().ess_pool_read_stats(pool, layer, ctypes.byref(s), int(reset)), "ess_pool_read_stats")
    return s


def ess_pool_kernel_launches(pool) -> int:
    n = ctypes.c_int64(0)
    check(load().ess_pool_kernel_launches(pool, ctypes.byref(n)), "ess_pool_kernel_launches")
    return int(n.value)


def ess_pool_poll(pool, stream=None) -> int:
    return load().ess_pool_poll(pool, _stream(stream))


def ess_prefill_plan(onload_layer_map, rotating: int = 3, shared_copy: bool = False):
    """Binding table of the prefill layer schedule: (buffer, load_at,
    reuse_after) as int32 arrays, one entry per layer."""
    import numpy as np
    m = np.ascontiguousarray(onload_layer_map, dtype=np.int32)
    L = int(m.shape[0])
    outs = [np.zeros(L, dtype=np.int32) for _ in range(3)]
    check(load().ess_prefill_plan(L, m.ctypes.data, int(rotating), int(bool(shared_copy)),
                                  *[o.ctypes.data for o in outs]), "ess_prefill_plan")
    return tuple(outs)


def ess_compact_rows(rows_bf16_bits):
    """bf16 bits [n][576] (numpy uint16) -> compact rows uint8 [n][656]."""
    import numpy as np
    rows = np.ascontiguousarray(rows_bf16_bits, dtype=np.uint16).reshape(-1, 576)
    out = np.zeros((rows.shape[0], 656), dtype=np.uint8)
    check(load().ess_compact_rows(rows.ctypes.data, rows.shape[0], out.ctypes.data),
          "ess_compact_rows")
    return out


def ess_replay_misses(trace, T: int, C: int, policy: int, scores=None, seed: int = 0,
                      request: int = 0):
    """trace[s][m]: the tokens way m selected at step s; scores[s][m]: the
    way's scores of all T tokens (Score policy).  Returns (union_misses,
    way_misses) per step as int32 arrays."""
    import numpy as np
    n_steps = len(trace)
    n_ways = len(trace[0]) if n_steps else 1
    lists = [np.asarray(w, dtype=np.int32) for ways in trace for w in ways]
    offsets = np.zeros(len(lists) + 1, dtype=np.int64)
    offsets[1:] = np.cumsum([x.shape[0] for x in lists])
    tokens = np.concatenate(lists) if lists else np.zeros(1, np.int32)
    sc = None
    if scores is not None:
        sc = np.ascontiguousarray(np.asarray(scores, dtype=np.float32).reshape(n_steps, n_ways, T))
    um = np.zeros(max(n_steps, 1), dtype=np.int32)
    wm = np.zeros(max(n_steps, 1), dtype=np.int32)
    check(load().ess_replay_misses(n_steps, n_ways, offsets.ctypes.data, tokens.ctypes.data,
                                   None if sc is None else sc.ctypes.data, T, C, policy,
                                   seed & ((1 << 64) - 1), request, um.ctypes.data,
                                   wm.ctypes.data), "ess_replay_misses")
    return um[:n_steps], wm[:n_steps]


def ess_host_gather(host_rows, n_host_rows: int, row_bytes: int, rows, n_rows: int, dst,
                    bad_row=None, stream=None) -> None:
    """Rows of pinned host memory (a HostBuffer or pinned tensor) into the
    device tensor dst; rows is a device int64 tensor or None (sequential)."""
    check(load().ess_host_gather(_p(host_rows), int(n_host_rows), int(row_bytes), _p(rows),
                                 int(n_rows), _p(dst), _p(bad_row), _stream(stream)),
          "ess_host_gather")


def ess_pool_set_eviction(pool, policy: int, seed: int = 0) -> None:
    """Victim order of the decode kernels (ESS_EVICT_*)."""
    check(load().ess_pool_set_eviction(pool, int(policy), seed & ((1 << 64) - 1)),
          "ess_pool_set_eviction")


def ess_prefill_run(onload_layer_map, host_kv, layer_bytes: int, buffers, compute,
                    compute_stream, h2d_stream, d2h_stream, rotating: int = 3,
                    shared_copy: bool = False, wb_offset: int = 0, wb_bytes=None) -> None:
    """One prefill pass.  host_kv: per layer a pinned host buffer (HostBuffer or
    tensor; entry 0 may be None); buffers: 1 + rotating device tensors;
    compute(layer, buffer_ptr, stream_ptr) enqueues the layer's work."""
    import numpy as np
    m = np.ascontiguousarray(onload_layer_map, dtype=np.int32)
    L = int(m.shape[0])
    hk = (ctypes.c_void_p * L)(*[None if h is None else _p(h) for h in host_kv])
    bf = (ctypes.c_void_p * len(buffers))(*[_p(b) for b in buffers])
    cb = PREFILL_COMPUTE_FN(lambda user, layer, buf, st: compute(int(layer), buf, st))
    wb = layer_bytes - wb_offset if wb_bytes is None else wb_bytes
    check(load().ess_prefill_run(L, m.ctypes.data, int(rotating), int(bool(shared_copy)), hk,
                                 int(layer_bytes), int(wb_offset), int(wb), bf, cb, None,
                                 _stream(compute_stream), _stream(h2d_stream),
                                 _stream(d2h_stream)), "ess_prefill_run")
