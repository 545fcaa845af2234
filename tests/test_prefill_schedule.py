"""Pins of the prefill layer-schedule model (oracle/prefill_schedule.py),
and the plausible mistakes they catch.

The model restates the FlashOffloading analysis, section "prefill side: four
whole-layer buffers": B0 pinned to layer 0, B1-B3 rotating, a buffer released
only after its compute and its write-back, prefetch at a layer's scheduling
point, and the bound on exposed load time.  The pins are Figure 3's buffer
roles and write-back start, the page's bound met with equality in steady
state (separate copy streams and one shared copy path), the closed form for a
single rotating buffer, the bound as a floor for uneven layers, and the
refusal of a prefetch into a buffer that is still held.
"""
import inspect
import sys

import numpy as np
import pytest

from oracle import prefill_schedule as S


def test_figure3_buffer_roles_and_first_write_back():
    t = S.simulate(6, [1.0] * 6, [0.5] * 6, [0.3] * 6)
    assert t.buffer == [0, 1, 2, 3, 1, 2]              # B1..B3 for layers 1-3, then B1, B2
    assert t.load[0] is None and t.save[0] is None      # layer 0 computes from B0 at once
    assert t.compute[0][0] == 0.0
    first = min(s[0] for s in t.save if s)
    assert first == t.compute[1][1] and t.save[1][0] == first   # D2H waits for layer 1


@pytest.mark.parametrize("th,tc", [(1.5, 1.0), (0.6, 1.0), (2.0, 0.5)])
def test_steady_state_meets_the_bound_with_separate_streams(th, tc):
    L = 12
    t = S.simulate(L, [tc] * L, [th] * L, [0.2] * L)
    want = S.exposed_lower_bound(th, tc, d_on=1)
    assert want == max(0.0, th - tc)
    assert np.allclose(t.exposed[3:], want)


@pytest.mark.parametrize("th,td,tc", [(0.7, 0.6, 1.0), (0.3, 0.3, 1.0), (1.0, 0.8, 1.2)])
def test_one_copy_path_needs_both_directions_in_the_window(th, td, tc):
    L = 12
    t = S.simulate(L, [tc] * L, [th] * L, [td] * L, shared_copy=True)
    want = S.exposed_lower_bound(th, tc, d_on=1, t_d2h=td, shared_copy=True)
    assert want == max(0.0, th + td - tc)
    assert np.allclose(t.exposed[3:], want)


def test_one_rotating_buffer_serialises_write_back_and_load():
    L = 8
    t = S.simulate(L, [1.0] * L, [0.5] * L, [0.3] * L, rotating=1)
    assert np.allclose(t.exposed[2:], 0.5 + 0.3)       # release, then the whole load
    assert t.buffer == [0] + [1] * (L - 1)


def test_bound_is_a_floor_for_uneven_layers():
    rng = np.random.default_rng(11)
    for _ in range(30):
        L = int(rng.integers(4, 14))
        tc = rng.uniform(0.2, 2.0, L)
        th = rng.uniform(0.1, 3.0, L)
        td = rng.uniform(0.1, 1.0, L)
        d = int(rng.integers(1, 3))
        m = [i + d if i + d < L else -1 for i in range(L)]
        shared = bool(rng.integers(0, 2))
        try:
            t = S.simulate(L, tc, th, td, onload_layer_map=m, shared_copy=shared)
        except ValueError:
            continue
        for i, j in enumerate(m):
            if j < 1:
                continue
            # the compute between prefetching j and using it, and the bound
            assert t.compute[j][0] - t.compute[i][0] >= th[j] - 1e-12
            assert t.exposed[j] >= S.exposed_lower_bound(th[j], float(sum(tc[i:j])), 1) \
                - sum(t.exposed[i + 1:j]) - 1e-12


def test_prefetch_into_a_held_buffer_is_refused():
    L = 8
    far = [i + 4 if i + 4 < L else -1 for i in range(L)]     # distance 4 with 3 buffers
    with pytest.raises(ValueError):
        S.simulate(L, [1.0] * L, [0.5] * L, [0.3] * L, onload_layer_map=far)
    with pytest.raises(ValueError):                          # the load would queue ahead
        S.simulate(L, [1.0] * L, [0.5] * L, [0.3] * L, rotating=1, shared_copy=True)


# ------------------------------------------------------------------ mutants

ORIG = S.simulate


def _b0_rotates(L, tc, th, td, onload_layer_map=None, rotating=3, shared_copy=False):
    t = ORIG(L, tc, th, td, onload_layer_map, rotating + 1, shared_copy)
    t.buffer = [(b - 1) % (rotating + 1) if i else 0 for i, b in enumerate(t.buffer)]
    return t


def _release_before_write_back(L, tc, th, td, onload_layer_map=None, rotating=3,
                               shared_copy=False):
    return ORIG(L, tc, th, [0.0] * L, onload_layer_map, rotating, shared_copy)


def _shared_path_ignored(L, tc, th, td, onload_layer_map=None, rotating=3, shared_copy=False):
    if shared_copy and rotating == 1:
        raise ValueError("refused")
    return ORIG(L, tc, th, td, onload_layer_map, rotating, False)


MUTANTS = [_b0_rotates, _release_before_write_back, _shared_path_ignored]
HOOK_MUTANTS = [("prefetch_not_before", lambda start: 0.0)]   # loads ignore the scheduling point
PINS = [f for name, f in sorted(vars(sys.modules[__name__]).items())
        if name.startswith("test_") and inspect.isfunction(f)
        and name not in ("test_pins_catch_mutant", "test_pins_catch_early_prefetch")]


def _call(pin):
    sig = inspect.signature(pin)
    if not sig.parameters:
        return pin()
    marks = [m for m in getattr(pin, "pytestmark", []) if m.name == "parametrize"]
    for args in marks[0].args[1]:
        pin(*args)


def test_pins_catch_early_prefetch(monkeypatch):
    for name, mutant in HOOK_MUTANTS:
        monkeypatch.setattr(S, name, mutant)
        failed = []
        for pin in PINS:
            try:
                _call(pin)
            except (Exception, pytest.fail.Exception) as e:
                failed.append(f"{pin.__name__}: {type(e).__name__}")
                break
        assert failed, f"no pin notices {name}"


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m.__name__ for m in MUTANTS])
def test_pins_catch_mutant(monkeypatch, mutant):
    monkeypatch.setattr(S, "simulate", mutant)
    failed = []
    for pin in PINS:
        try:
            _call(pin)
        except (Exception, pytest.fail.Exception) as e:   # an assertion or a pytest.raises miss
            failed.append(f"{pin.__name__}: {type(e).__name__}")
            break
    assert failed, f"no pin notices {mutant.__name__}"
