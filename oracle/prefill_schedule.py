"""Timeline model of the prefill layer schedule with four device buffers.

TEST INFRASTRUCTURE ONLY.  Only the tests may import this module.  It shares
no code with the CUDA library.

What it restates: hwcomputing.csdn.net FlashOffloading analysis, section
"prefill side: four whole-layer buffers hide the transfers":
  - buffer B0 stays bound to layer 0 for the whole prefill; B1..B3 rotate
    over the later layers through a binding table;
  - an offloaded layer (l >= 1) goes through: bind a free buffer and load
    its history (H2D), wait for that load, compute, write the updated KV
    back (D2H), and release the buffer only once both the last compute
    consumer and the write-back are done; layer 0 computes from B0 at once;
  - at layer i's scheduling point the schedule prefetches layer
    onload_layer_map[i] (not necessarily i + 1);
  - the exposed load time of a layer is at least
    max(0, tau_H2D - d_on * tau_compute), d_on being the independent layer
    compute between prefetch and use; with one serial copy path tau_H2D
    becomes tau_H2D + tau_D2H;
  - Figure 3: H2D fills B1, B2, B3 with layers 1-3 and then reuses B1, B2
    for layers 4-5; D2H idles until layer 1 has been computed.

The model (the reading taken where the page leaves steps open):
  - three in-order streams: compute, H2D and D2H (or one copy stream that
    takes loads and write-backs in issue order);
  - rotating buffers are bound round-robin in load order;
  - the load of layer j, prefetched at layer i's scheduling point, starts
    no earlier than compute(i) starts, the copy stream is free, and the
    buffer's previous layer has been released; layers no entry of the map
    prefetches are loaded from time 0, in order;
  - compute(i) waits for compute(i-1) and for load(i); write-back(i)
    follows compute(i); layer 0 is neither loaded nor written back here.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence


@dataclass
class Timeline:
    buffer: List[int]             # buffer of each layer (0 = B0)
    compute: List[tuple]          # (start, end) per layer
    load: List[Optional[tuple]]   # (start, end) per layer, None for layer 0
    save: List[Optional[tuple]]   # (start, end) per layer, None for layer 0
    exposed: List[float]          # compute(i) start - compute(i-1) end (0 for layer 0)

    @property
    def makespan(self) -> float:
        ends = [e for _, e in self.compute] + [s[1] for s in self.save if s]
        return max(ends)


def prefetch_not_before(scheduling_point_start: float) -> float:
    """Earliest start of a load prefetched at a layer's scheduling point: the
    start of that layer's compute."""
    return scheduling_point_start


def simulate(L: int, t_compute: Sequence[float], t_h2d: Sequence[float], t_d2h: Sequence[float],
             onload_layer_map: Optional[Sequence[int]] = None, rotating: int = 3,
             shared_copy: bool = False) -> Timeline:
    """Run the schedule for L layers; onload_layer_map[i] = j prefetches layer
    j at layer i's scheduling point (default j = i + 1; -1 for none)."""
    if onload_layer_map is None:
        onload_layer_map = [i + 1 if i + 1 < L else -1 for i in range(L)]
    prefetched = {j for j in onload_layer_map if j >= 1}
    initial = [j for j in range(1, L) if j not in prefetched]
    load_order = initial + [j for j in onload_layer_map if j >= 1]
    if sorted(load_order) != list(range(1, L)):
        raise ValueError("every layer >= 1 must be loaded exactly once")
    buf = [0] * L
    prev_on_buf = {}                     # layer -> layer that used the same buffer before
    last = {}
    for n, j in enumerate(load_order):
        b = 1 + n % rotating
        buf[j] = b
        prev_on_buf[j] = last.get(b)
        last[b] = j

    comp = [None] * L
    load = [None] * L
    save = [None] * L
    h2d_free = d2h_free = 0.0

    def released(j):
        p = prev_on_buf[j]
        return 0.0 if p is None else max(comp[p][1], save[p][1])

    # issue order: the initial loads, then per layer its compute, its
    # prefetch and its write-back
    def do_load(j, not_before):
        nonlocal h2d_free, d2h_free
        free = d2h_free if shared_copy else h2d_free
        s = max(free, not_before, released(j))
        load[j] = (s, s + t_h2d[j])
        if shared_copy:
            d2h_free = h2d_free = load[j][1]
        else:
            h2d_free = load[j][1]

    def do_save(i):
        nonlocal h2d_free, d2h_free
        s2 = max(d2h_free, comp[i][1])
        save[i] = (s2, s2 + t_d2h[i])
        d2h_free = save[i][1]
        if shared_copy:
            h2d_free = d2h_free

    def check_free(j, when):
        p = prev_on_buf[j]
        if p is not None and save[p] is None:
            # the buffer is still held by a layer not yet written back: on
            # separate streams that layer comes later; on one serial copy
            # stream the load would queue ahead of the write-back it waits for
            raise ValueError(f"layer {j} cannot be loaded {when}: its buffer is still held")

    def prefetch(j, i):
        check_free(j, f"at layer {i}")
        do_load(j, prefetch_not_before(comp[i][0]))

    for j in initial:
        check_free(j, "up front")
        do_load(j, 0.0)
    for i in range(L):
        s = 0.0 if i == 0 else max(comp[i - 1][1], load[i][1])
        comp[i] = (s, s + t_compute[i])
        j = onload_layer_map[i]
        if shared_copy:                  # one stream: the prefetch is issued first
            if j >= 1:
                prefetch(j, i)
            if i >= 1:
                do_save(i)
        else:                            # separate streams: issue order does not matter
            if i >= 1:
                do_save(i)
            if j >= 1:
                prefetch(j, i)
    exposed = [0.0] + [comp[i][0] - comp[i - 1][1] for i in range(1, L)]
    return Timeline(buf, comp, load, save, exposed)


def exposed_lower_bound(t_h2d: float, t_compute: float, d_on: int, t_d2h: float = 0.0,
                        shared_copy: bool = False) -> float:
    """The page's bound on the exposed load time of a layer."""
    tau = t_h2d + (t_d2h if shared_copy else 0.0)
    return max(0.0, tau - d_on * t_compute)
