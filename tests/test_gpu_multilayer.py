"""The multi-layer configuration at its stated shape: 8 layers, 32 requests,
two MTP ways, T = 65536, C = 16384, through the layer-wise pipeline.

"ESS: Latent-Cache Offload" (layer-wise overlap of transfers with compute):
the batch runs as two micro-batches of 16 requests on two streams, layer by
layer (ess_pipeline_step), so one micro-batch's indexer and selection overlap
the other's attention.  Every layer of both micro-batches is compared with the
oracle on each of the first eight steps: top-k lists, miss union and LRU state
bit-exact (through the state), attention within tolerance."""
import numpy as np
import pytest
import torch

from host_latent_cache_gb300 import ess
from host_latent_cache_gb300 import workloads as W

from parity_util import Pair, assert_attn_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

STEPS = 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_latent_cache_gb300 import build as B
    B.build()
    assert torch.cuda.is_available()
    ess.load()


def test_eight_layers_two_microbatches_first_steps():
    cfg = W.multilayer()
    assert (cfg.layers, cfg.batch, cfg.mtp, cfg.T, cfg.C) == (8, 32, 2, 65536, 16384)
    half = cfg.batch // 2
    halves = [cfg.replace(batch=half, seed=cfg.seed + 100 * h) for h in range(2)]
    pairs = []
    for c in halves:
        p = Pair(c, layers=cfg.layers)
        for ld in p.lds:
            ld.host_latent = None      # the session holds its own pinned copy
        pairs.append(p)
    streams = [torch.cuda.Stream() for _ in range(2)]
    L = cfg.layers
    worst = (0.0, 0.0)
    for s in range(STEPS):
        inputs = []
        for p in pairs:
            per_layer = []
            for l in range(L):
                q, enc, w, qm = p.next_inputs(l)
                qd, wd, qmd = p.sess.device_inputs(enc, w, qm)
                out = torch.zeros((half, cfg.mtp, cfg.mla_heads, 512), dtype=torch.float32,
                                  device="cuda")
                per_layer.append((q, w, qm, qd, wd, qmd, out))
            inputs.append(per_layer)
        torch.cuda.synchronize()
        ess.ess_pipeline_step([p.sess.pool for p in pairs], L,
                              [inputs[h][l][3] for h in range(2) for l in range(L)],
                              [inputs[h][l][4] for h in range(2) for l in range(L)],
                              [inputs[h][l][5] for h in range(2) for l in range(L)],
                              [inputs[h][l][6] for h in range(2) for l in range(L)], streams)
        torch.cuda.synchronize()
        for h, p in enumerate(pairs):
            assert p.sess.poll() == ess.ESS_OK
            for l in range(L):
                q, w, qm, _, _, _, out = inputs[h][l]
                keyf, latf = p.oracle_inputs(l)
                r = p.orc[l].step(q.astype(np.float64), w.astype(np.float64), keyf,
                                  p.lds[l].idx_scale, W.bf16_bits_to_float(qm).astype(np.float64),
                                  latf)
                p.compare_state(l)
                e = assert_attn_close(out.cpu().numpy(), r.out, f"step {s} half {h} layer {l}")
                worst = (max(worst[0], e[0]), max(worst[1], e[1]))
    for p in pairs:
        p.close()
    print(f"worst attention error over {STEPS} steps x {L} layers x 2 halves: "
          f"max-abs {worst[0]:.2e}, rel-L2 {worst[1]:.2e}")
