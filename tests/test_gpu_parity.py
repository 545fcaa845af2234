"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Bit-exact: indexer scores, top-k lists (misses first), topk slots, the miss
union and its paired slots, cache_slots / slot_token / last_used / step.
Within tolerance (max-abs 2e-2, relative L2 1e-3): the attention output.
"""
import numpy as np
import pytest
import torch

from host_latent_cache_gb300 import ess
from host_latent_cache_gb300 import workloads as W
from host_latent_cache_gb300.session import Session
from oracle import ess_oracle as O

from parity_util import Pair, assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from host_latent_cache_gb300 import build as B
    B.build()
    assert torch.cuda.is_available()
    ess.load()


# ------------------------------------------------------------------ indexer (a1)

def test_indexer_scores_tiny_bf16():
    p = Pair(W.tiny())
    p.run_step(check_scores=True)
    p.close()


def test_indexer_scores_fp8_ragged_two_ways():
    cfg = W.multilayer().replace(layers=1, batch=3, T=1024, T_per_req=[1000, 130, 0], k=64,
                                 C=256, mla_heads=32, steps=2)
    p = Pair(cfg)
    for _ in range(2):
        p.run_step(check_scores=True)
    p.close()


def test_indexer_scores_precision_stress():
    # one product of 30 beside many products of 1/64: an accumulator that
    # dropped low bits relative to the largest term would lose the small ones
    cfg = W.v32_32k().replace(batch=1, T=256, k=16, C=64, mla_heads=16)
    ld = W.gen_layer(cfg)
    lv, codes = W.key_levels()
    code = dict(zip(lv.tolist(), codes.tolist()))
    keys = np.full((1, 256, 128), code[0.125], dtype=np.uint8)
    keys[0, :, 0] = code[15.0]
    keys[0, 1::2, 5] = code[-15.0]
    ld.idx_keys[:] = keys
    ld.idx_scale[:] = np.float32(1.0)
    sess = Session(cfg, [ld])
    q = np.full((1, 1, 64, 128), 0.125, dtype=np.float32)
    q[:, :, :, 0] = 2.0
    q[:, :, 1::3, 7] = -2.0
    w = np.full((1, 1, 64), 1.0 / 64.0, dtype=np.float32)
    w[:, :, ::5] = 63.0 / 64.0
    enc = W.encode_query(cfg, q)
    qm = np.zeros((1, 1, 16, 576), dtype=np.uint16)
    qd, wd, _ = sess.device_inputs(enc, w, qm)
    got = sess.scores_only(0, qd, wd).cpu().numpy()[0, 0, :256]
    want = O.score_indexer(q[0, 0].astype(np.float64), w[0, 0].astype(np.float64),
                           W.decode_keys(cfg, keys[0]), ld.idx_scale[0])
    assert np.array_equal(got, want)
    sess.close()


@pytest.mark.parametrize("shape", [
    dict(mtp=3),                                       # N = 192: 64-column chunks
    dict(mtp=4),                                       # N = 256, the pages' MTP3 (4 ways)
    dict(mtp=3, idx_heads=32),                         # N = 96: 32-column chunks
    dict(mtp=4, idx_heads=32, T_per_req=[4096, 700]),  # ragged, a way per 32 columns
], ids=["3x64", "4x64", "3x32", "4x32_ragged"])
def test_three_and_four_ways(shape):
    """More MTP ways than the configs use: scores bit-exact per way, then the
    whole layer from an empty and from a full pool (FlashOffloading analysis,
    "decode side (1)": the four-way MTP3 merge into one miss union)."""
    base = dict(layers=1, batch=2, T=4096, k=256, mla_heads=32, steps=3)
    base.update(shape)
    base["C"] = base["mtp"] * base["k"]
    cfg = W.v32_32k().replace(**base)
    p = Pair(cfg)
    for s in range(2):
        p.run_step(check_scores=(s == 0))
    p.prime_full(age=4)
    for _ in range(3):
        p.run_step()
    p.check_pool_rows()
    p.close()


# ------------------------------------------------------------------ selection + LRU (a2-a4)

def _planted_ties(rng, shape, k):
    """Mostly distinct scores with a run of exact ties planted at the k-th largest."""
    sc = np.exp(rng.normal(0.0, 3.0, size=shape)).astype(np.float32)  # spread over binades
    B_, M_, T_ = shape
    for b in range(B_):
        for m in range(M_):
            kth = np.sort(sc[b, m])[::-1][min(k, T_) - 1]
            pos = rng.choice(T_, size=min(60, T_), replace=False)
            sc[b, m, pos] = kth
    return sc


def _select_case(T_list, k, C, M, steps, seed, levels=3, H=16, planted=False):
    cfg = W.multilayer().replace(layers=1, batch=len(T_list), T=max(max(T_list), 64),
                                 T_per_req=T_list, k=k, C=C, mtp=M, mla_heads=H)
    ld = W.gen_layer(cfg)
    sess = Session(cfg, [ld])
    orc = O.OracleLayer(ld.T, C, k, cfg.sm_scale)
    rng = np.random.default_rng(seed)
    Tm = W.t_max_of(cfg)
    for s in range(steps):
        if planted:
            sc = _planted_ties(rng, (cfg.batch, M, Tm), k)
        else:
            sc = rng.integers(0, levels, size=(cfg.batch, M, Tm)).astype(np.float32)
            sc[:, :, ::7] = rng.random((cfg.batch, M, len(range(0, Tm, 7)))).astype(np.float32)
        st = torch.from_numpy(sc).cuda()
        sess.select(0, st)
        torch.cuda.synchronize()
        assert sess.poll() == ess.ESS_OK
        # oracle from the same scores
        ti = sess.topk_idx.cpu().numpy()
        ts = sess.topk_slot.cpu().numpy()
        nmw = sess.n_miss_way.cpu().numpy()
        mt = sess.miss_tok.cpu().numpy()
        msl = sess.miss_slot.cpu().numpy()
        nm = sess.n_miss.cpu().numpy()
        cs, stok, lu, sp = sess.state(0)
        for b in range(cfg.batch):
            Tb = int(ld.T[b])
            o = orc.state[b]
            before = o.cache_slots.copy()
            sel = [O.topk_select(sc[b, m, :Tb], k) for m in range(M)]
            r = O.resolve_union(sel, o.cache_slots)
            victims, _ = O.lru_update(o, r.union, r.miss_tok)
            for m in range(M):
                srt = np.sort(sel[m])
                was = before[srt] >= 0
                order = np.concatenate([srt[~was], srt[was]])
                slots = o.cache_slots[order]
                enc = np.where(before[order] >= 0, slots, ~slots)
                n = len(order)
                assert np.array_equal(ti[b, m, :n], order), (s, b, m)
                assert np.array_equal(ts[b, m, :n], enc), (s, b, m)
                assert nmw[b, m] == r.misses[m]
            assert nm[b] == len(r.miss_tok)
            assert np.array_equal(mt[b, :nm[b]], r.miss_tok)
            assert np.array_equal(msl[b, :nm[b]], victims)
            assert np.array_equal(cs[b, :Tb], o.cache_slots)
            assert np.array_equal(stok[b], o.slot_token)
            assert np.array_equal(lu[b], o.last_used)
            assert sp[b] == o.step
    sess.close()


def test_select_ties_evictions_two_ways():
    _select_case([3000, 777, 64], k=128, C=300, M=2, steps=6, seed=1)


def test_select_k_at_least_T_and_empty_request():
    _select_case([100, 0, 64, 1], k=128, C=256, M=1, steps=4, seed=2)


def test_select_all_equal_scores():
    _select_case([5000, 4096], k=256, C=512, M=1, steps=5, seed=3, levels=1)


def test_select_threshold_ties_candidate_path():
    # few candidates per histogram bin: the candidate-refinement path, with
    # exact ties at the k-th score spread over every CTA's token range
    _select_case([20000, 9000], k=512, C=1200, M=2, steps=5, seed=5, planted=True)


def test_select_threshold_ties_one_way_large_T():
    _select_case([131072], k=2048, C=4096, M=1, steps=3, seed=6, planted=True)


def test_select_many_ties_small_pool():
    _select_case([20000], k=512, C=512, M=1, steps=5, seed=4, levels=2)


# ------------------------------------------------------------------ whole layer (a1-a6)

def test_tiny_all_steps_fused():
    cfg = W.tiny()
    p = Pair(cfg)
    for _ in range(cfg.steps):
        p.run_step()
    p.check_pool_rows()
    p.close()


def test_tiny_all_steps_staged():
    cfg = W.tiny()
    p = Pair(cfg, miss_mode=ess.ESS_MISS_STAGED)
    for _ in range(cfg.steps):
        p.run_step()
    p.check_pool_rows()
    p.close()


def test_ess_step_matches_separate_calls():
    cfg = W.tiny().replace(T=2048, k=256, C=512)
    a = Pair(cfg)
    b = Pair(cfg)
    for _ in range(4):
        a.run_step(api="calls")
        b.run_step(api="step")
        assert torch.equal(a.sess.out, b.sess.out)
    a.close()
    b.close()


@pytest.mark.parametrize("host_kind", ["mapped", "torch_pinned", "pageable"])
def test_step_host_matches_step(host_kind):
    """ess_step_host gives the same output and state as ess_step on device
    inputs: with mapped pinned buffers the GPU reads the inputs and writes the
    output over the host link itself; with pageable buffers the library copies
    through its staging."""
    cfg = W.tiny().replace(T=2048, k=256, C=512)
    a = Pair(cfg)
    b = Pair(cfg)
    keep = []

    def host(arr):
        arr = np.ascontiguousarray(arr)
        if host_kind == "mapped":
            hb = ess.HostBuffer(arr.shape, arr.dtype)
            hb.array[...] = arr
            keep.append(hb)
            return hb
        t = torch.from_numpy(arr.copy())
        return t.pin_memory() if host_kind == "torch_pinned" else t

    out_np = np.zeros((cfg.batch, cfg.mtp, cfg.mla_heads, 512), np.float32)
    out_h = host(out_np)
    for _ in range(4):
        _, enc, w, qm = a.next_inputs(0)
        b.next_inputs(0)
        qd, wd, qmd = a.sess.device_inputs(enc, w, qm)
        a.sess.step(0, qd, wd, qmd)
        ess.ess_step_host(b.sess.pool, 0, host(enc.view(np.uint8)), host(w.astype(np.float32)),
                          host(qm.view(np.int16)), out_h)
        torch.cuda.synchronize()
        assert a.sess.poll() == ess.ESS_OK and b.sess.poll() == ess.ESS_OK
        got = out_h.array if host_kind == "mapped" else out_h.numpy()
        assert np.array_equal(got, a.sess.out.cpu().numpy())
        for x, y in zip(a.sess.state(0), b.sess.state(0)):
            assert np.array_equal(x, y)
    for hb in keep:
        hb.close()
    out_h = None
    a.close()
    b.close()


def test_kernel_launch_count():
    """A fused step launches the indexer, the selection, the LRU finishing
    kernel, the attention and the merge; staged adds the copy."""
    cfg = W.tiny().replace(T=2048, k=256, C=512)
    counts = {}
    for mode in (ess.ESS_MISS_FUSED, ess.ESS_MISS_STAGED):
        p = Pair(cfg, miss_mode=mode)
        n0 = p.sess.kernel_launches()
        p.run_step(api="step")
        counts[mode] = p.sess.kernel_launches() - n0
        p.close()
    assert counts[ess.ESS_MISS_FUSED] == 5
    assert counts[ess.ESS_MISS_STAGED] == counts[ess.ESS_MISS_FUSED] + 1


def test_v32_shaped_reduced_batch():
    cfg = W.v32_32k().replace(batch=2, T=8192 + 64, T_per_req=[8192 + 64, 5000], steps=4)
    p = Pair(cfg)
    for _ in range(4):
        p.run_step()
    p.check_pool_rows()
    p.close()


def test_stats_counters():
    cfg = W.tiny().replace(T=2048, k=128, C=256)
    p = Pair(cfg)
    hits = misses = union = nmiss = 0
    for _ in range(3):
        r = p.run_step()
        hits += int(r.hits.sum())
        misses += int(r.misses.sum())
        union += int(r.union_size.sum())
        nmiss += sum(len(x) for x in r.miss_tok)
    s = p.sess.stats(0)
    assert (s.steps, s.hits, s.misses, s.union_size, s.miss_rows) == (3, hits, misses, union, nmiss)
    assert s.miss_bytes == nmiss * 1152
    p.close()


def _cut_bins(scores, k):
    """Coarse bin (top 12 bits of the ordered key) of the k-th largest score."""
    u = np.ascontiguousarray(scores, dtype=np.float32).view(np.uint32)
    key = np.where(u >> 31 != 0, ~u, u | np.uint32(0x80000000)).astype(np.uint32)
    return int(np.sort(key >> 20)[::-1][k - 1])


def test_guided_selection_regimes():
    """From its second step a layer's selection reads only the tokens that the
    indexer flagged at or above the previous step's cut less one bin, when
    every way's cut stays at or above that bin; a way whose cut lies in one of
    the four bins the indexer's fine histogram covers takes it from there.
    Doubled and halved head weights move every cut by eight bins (an octave):
    up out of the fine window, then down below the flagged bin (the full
    scan).  Lists, state and attention follow the oracle bit for bit at every
    step, and the layer's counters show which of the three ways each request
    took, as the oracle's own scores predict it."""
    cfg = W.v32_32k().replace(batch=3, T=8192, T_per_req=[8192, 5000, 300], k=512, C=2048,
                              mtp=2, mla_heads=32)
    p = Pair(cfg)
    base = p.next_inputs
    guess = np.zeros((cfg.batch, cfg.mtp), dtype=np.int64)
    seen = set()
    for f in [1.0, 1.0, 2.0, 2.0, 0.5, 0.5, 0.5]:
        def scaled(layer, f=f):
            q, enc, w, qm = base(layer)
            return q, enc, (w * np.float32(f)).astype(np.float32), qm
        p.next_inputs = scaled
        r = p.run_step(check_scores=True)
        want_guided = want_fine = 0
        for b in range(cfg.batch):
            if cfg.k >= int(p.lds[0].T[b]):
                guess[b] = 0                   # every token selected: no cut
                continue
            b1 = [_cut_bins(r.scores[b][m], cfg.k) for m in range(cfg.mtp)]
            if all(guess[b, m] != 0 and b1[m] >= guess[b, m] for m in range(cfg.mtp)):
                want_guided += 1
                want_fine += sum(b1[m] - guess[b, m] < 4 for m in range(cfg.mtp))
            guess[b] = [x - 1 for x in b1]
        st = ess.ess_pool_read_stats(p.sess.pool, 0, reset=True)
        assert (st.guided, st.fine_cuts) == (want_guided, want_fine), f
        seen.add((want_guided > 0, want_fine > 0))
    assert seen == {(False, False), (True, False), (True, True)}
    p.close()


def test_device_bounds_check_reports_instead_of_faulting():
    cfg = W.tiny().replace(T=1024, k=128, C=256)
    p = Pair(cfg)
    p.run_step()
    sess = p.sess
    bad = sess.topk_slot.clone()
    bad[0, 0, 3] = cfg.C + 5          # slot outside the pool: skipped and reported
    q, enc, w, qm = p.next_inputs(0)
    _, _, qmd = sess.device_inputs(enc, w, qm)
    ess.ess_sparse_mla_decode(sess.pool, 0, qmd, sess.topk_idx, bad, sess.out)
    torch.cuda.synchronize()
    assert sess.poll() == ess.ESS_ERR_DEVICE_CHECK
    assert sess.poll() == ess.ESS_OK   # cleared by the poll
    p.close()


# ------------------------------------------------------------------ layer pipeline (a7)

def test_two_microbatch_layer_pipeline():
    """Two pools (two halves of a batch) run layer by layer on two streams."""
    cfg = W.multilayer().replace(layers=2, batch=2, T=8192, k=256, C=1024, steps=3)
    halves = [cfg.replace(seed=cfg.seed + 100 * h) for h in range(2)]
    pairs = [Pair(c, layers=2) for c in halves]
    streams = [torch.cuda.Stream() for _ in range(2)]
    for _ in range(3):
        inputs, oracle_runs = [], []
        for h, p in enumerate(pairs):
            per_layer = []
            for l in range(2):
                q, enc, w, qm = p.next_inputs(l)
                qd, wd, qmd = p.sess.device_inputs(enc, w, qm)
                out = torch.zeros((cfg.batch, cfg.mtp, cfg.mla_heads, 512),
                                  dtype=torch.float32, device="cuda")
                per_layer.append((q, w, qm, qd, wd, qmd, out))
            inputs.append(per_layer)
        torch.cuda.synchronize()
        ess.ess_pipeline_step([p.sess.pool for p in pairs], 2,
                              [inputs[h][l][3] for h in range(2) for l in range(2)],
                              [inputs[h][l][4] for h in range(2) for l in range(2)],
                              [inputs[h][l][5] for h in range(2) for l in range(2)],
                              [inputs[h][l][6] for h in range(2) for l in range(2)], streams)
        torch.cuda.synchronize()
        for h, p in enumerate(pairs):
            assert p.sess.poll() == ess.ESS_OK
            for l in range(2):
                q, w, qm, _, _, _, out = inputs[h][l]
                keyf, latf = p.oracle_inputs(l)
                r = p.orc[l].step(q.astype(np.float64), w.astype(np.float64), keyf,
                                  p.lds[l].idx_scale, W.bf16_bits_to_float(qm).astype(np.float64),
                                  latf)
                p.compare_state(l)
                assert_attn_close(out.cpu().numpy(), r.out, f"pipeline h={h} l={l}")
    for p in pairs:
        p.close()


# ------------------------------------------------------------------ state set/get (resume)

def test_set_state_resumes_from_oracle_state():
    """A fresh pool given the oracle's state after some steps continues in step
    with the oracle (lists and bookkeeping; the LRU order is rebuilt)."""
    cfg = W.tiny().replace(T=2048, k=128, C=256)
    p = Pair(cfg)
    for _ in range(3):
        p.run_step()
    q = Pair(cfg)
    for _ in range(3):   # advance the second pair's query stream and oracle only
        q.next_inputs(0)
    for b in range(cfg.batch):
        q.orc[0].state[b] = p.orc[0].state[b].copy()
    st = p.orc[0].state[0]
    Tm = W.t_max_of(cfg)
    cs = np.full((1, Tm), -1, np.int32)
    cs[0, :len(st.cache_slots)] = st.cache_slots
    ess.ess_pool_set_state(q.sess.pool, 0, torch.from_numpy(cs), torch.from_numpy(st.slot_token[None].copy()),
                           torch.from_numpy(st.last_used[None].copy()),
                           torch.tensor([st.step], dtype=torch.int32))
    q.compare_state(0)
    q.check_pool_rows()              # resident rows reloaded from the host copy
    for _ in range(3):
        q.run_step()
    p.close()
    q.close()


@pytest.mark.parametrize("shape", [
    dict(),                                                     # every slot resident
    dict(batch=2, T=3072, T_per_req=[3000, 700], k=128, C=1024),  # one request smaller than C
    dict(batch=2, T=4096, mtp=2, idx_heads=32, k=256, C=512),   # two ways, C = M * k
], ids=["tiny_full", "ragged_partly_full", "two_ways_tight"])
def test_full_pool_evictions(shape):
    """From a full pool every miss evicts a resident token: lists, state and
    attention stay in step with the oracle, and the pool rows stay equal to the
    host copy."""
    cfg = W.tiny().replace(**shape)
    p = Pair(cfg)
    p.prime_full(age=5)
    p.check_pool_rows()
    for _ in range(6):
        p.run_step()
    p.check_pool_rows()
    assert sum(p.evicted) > 0
    p.close()


def test_set_state_rejects_future_stamps():
    cfg = W.tiny().replace(T=1024, k=64, C=128)
    p = Pair(cfg)
    lu = torch.full((1, cfg.C), -1, dtype=torch.int32)
    lu[0, 5] = 7
    with pytest.raises(ess.EssError):
        ess.ess_pool_set_state(p.sess.pool, 0, None, None, lu, torch.tensor([3], dtype=torch.int32))
    p.close()
