"""The prefill four-buffer engine (ess_prefill_run) moving real layer KV.

FlashOffloading analysis, section "prefill side: four whole-layer buffers hide
the transfers": B0 keeps layer 0, B1..B3 rotate over the later layers; each
offloaded layer is loaded into a free buffer, computed, written back to the
host copy, and only then released.  Here every layer's compute adds its own
constant to the buffer it finds, on the compute stream, while the engine
moves the layers on the copy streams.  If a buffer were reused before its
previous layer's compute and write-back were done, or a compute ran before its
load landed, the host copies would not come out as original + constant; every
byte is checked, for several prefetch maps, with separate copy streams and
with one shared copy stream, and for a written-back sub-range."""
import numpy as np
import pytest
import torch

from host_latent_cache_gb300 import ess

pytestmark = pytest.mark.gpu

L = 8
WORDS = 262144                  # 1 MiB per layer


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_latent_cache_gb300 import build as B
    B.build()
    assert torch.cuda.is_available()
    ess.load()


def _run(onload_map, shared_copy, wb=None, rotating=3):
    rng = np.random.default_rng(21)
    orig = [rng.integers(0, 1 << 30, size=WORDS, dtype=np.int32) for _ in range(L)]
    host = [None] + [ess.HostBuffer((WORDS,), np.int32) for _ in range(1, L)]
    for l in range(1, L):
        host[l].array[...] = orig[l]
    bufs = [torch.zeros(WORDS, dtype=torch.int32, device="cuda") for _ in range(1 + rotating)]
    bufs[0].copy_(torch.from_numpy(orig[0]))          # B0 holds layer 0
    by_ptr = {b.data_ptr(): b for b in bufs}
    streams = [torch.cuda.Stream() for _ in range(3)]
    seen = []

    def compute(layer, buf_ptr, stream_ptr):
        seen.append(layer)
        s = torch.cuda.ExternalStream(stream_ptr)
        with torch.cuda.stream(s):
            by_ptr[buf_ptr].add_(1000 + layer)

    off, nbytes = (0, WORDS * 4) if wb is None else wb
    torch.cuda.synchronize()
    ess.ess_prefill_run(onload_map, host, WORDS * 4, bufs, compute, *streams,
                        rotating=rotating, shared_copy=shared_copy, wb_offset=off, wb_bytes=nbytes)
    streams[0].synchronize()
    assert seen == list(range(L))
    assert torch.equal(bufs[0].cpu(), torch.from_numpy(orig[0] + 1000))
    lo, hi = off // 4, (off + nbytes) // 4
    for l in range(1, L):
        want = orig[l].copy()
        want[lo:hi] += 1000 + l
        assert np.array_equal(host[l].array, want), f"layer {l}"
    for h in host[1:]:
        h.close()


def test_figure3_schedule_three_streams():
    # B1..B3 take layers 1-3 up front; points 1..4 prefetch layers 4..7, each
    # into the buffer of the layer being computed at that point: the load
    # must wait for that layer's compute and write-back
    _run([-1, 4, 5, 6, 7, -1, -1, -1], False)


def test_one_shared_copy_stream():
    # one copy stream takes the write-back of a layer after the prefetch of
    # its own point, so the prefetches come one point later
    _run([-1, -1, 4, 5, 6, 7, -1, -1], True)


def test_prefetch_far_ahead():
    _run([-1, -1, -1, 4, 5, 6, 7, -1], False)


def test_written_back_range_only():
    _run([-1, 4, 5, 6, 7, -1, -1, -1], False, wb=(WORDS, WORDS))   # the second quarter


def test_two_rotating_buffers():
    _run([-1, 3, 4, 5, 6, 7, -1, -1], False, rotating=2)
