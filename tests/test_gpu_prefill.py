"""NOSA_S sparse prefill (nosa_prefill) against the CPU oracle.

The oracle runs its decode step over the prompt, one position at a time from an
empty context (the reading of sparse prefill taken here: position t gets the
selection the decode step at T = t + 1 makes, the eviction state carried from
t - 1).  The GPU selects every position in order and attends all positions in
one launch.  Compared: every checked position's selection (its query-aware and
query-agnostic picks, returned as bitmaps, with the sink and window blocks)
bit-exact, near ties logged and adopted as in the decode tests; outputs within
max-abs 2e-2 / mean-abs 2e-3 and the tighter relative bound; the layer's state
after the prompt (compressed keys, eviction bitmap, last selection; the cache holding
exactly that selection, block i in slot i) bit-exact; then a few decode steps continue from that state, which
checks the cache the prefill leaves behind.
"""
import math

import numpy as np
import pytest

from oracle import nosa_oracle as O
from synth import inputs as syn

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from tests.nosa_harness import OUT_MAX_ABS, OUT_MEAN_ABS, _near_tie_ok  # noqa: E402
from offloadable_block_sparse_gb300 import nosa as N  # noqa: E402

FUSED, UNFUSED = 0, N.NOSA_F_UNFUSED_STEP


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def _check_out(got, ref, where):
    err = np.abs(got - ref)
    assert err.max() <= OUT_MAX_ABS and err.mean() <= OUT_MEAN_ABS, f"output error {err.max():.3e} {where}"
    assert err.max() <= 2 ** -7 * np.abs(ref).max() + 1e-4, f"output error {err.max():.3e} (tight) {where}"
    return float(err.max())


def _select_and_adopt(o, sq, se, T, Q_gpu, E_gpu, k_q, k_e, ties, where):
    """The oracle's picks at context length T; a differing pick must be a near tie, then the GPU's is adopted."""
    _, C, _ = O.partition(T, o.nw, o.sink, o.block)
    Q = O.select_query_aware(sq, C, k_q)
    if Q != Q_gpu:
        assert _near_tie_ok(np.asarray(sq).astype(np.float32), Q_gpu, Q, C, k_q), f"query-aware pick {where}"
        ties.append(("q", where))
        Q = Q_gpu
    E = O.select_query_agnostic(se, C, Q, o.evicted, k_e)
    if E != E_gpu:
        pool = [b for b in C if b not in set(Q) and b not in o.evicted]
        assert _near_tie_ok(np.asarray(se).astype(np.float32), E_gpu, E, pool, k_e), f"query-agnostic pick {where}"
        ties.append(("e", where))
        E = E_gpu
    return Q, E


def run_prefill(wl, n, check_units, out_positions, flags=0, decode_steps=3, score_positions=None, cache_slots=0):
    """Prefill n tokens into an empty layer, check against the oracle, then decode_steps steps.

    score_positions (long prompts): the positions where the oracle forms its own query-aware
    scores; elsewhere it takes the GPU's query-aware picks and ranks the query-agnostic part by
    the whole prompt's pooled eviction scores (a candidate block lies before the window, so its
    windows are complete at every position where it is a candidate)."""
    B, Hq, Hkv, d, G = wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim, wl.group
    U = B * Hkv
    assert n + decode_steps <= wl.steps and wl.context == 0
    cfg = N.make_config(num_layers=1, batch=B, num_q_heads=Hq, num_kv_heads=Hkv, k_q=wl.k_q, k_e=wl.k_e,
                        window_tokens=wl.window_tokens, max_context=n + decode_steps, sink_blocks=wl.sink_blocks,
                        evict_hidden=wl.evict_hidden, flags=flags, cache_slots=cache_slots)
    stream = torch.cuda.current_stream()
    ctx = N.nosa_create(cfg, stream.cuda_stream)
    ties, max_err = [], 0.0
    try:
        sz = N.nosa_query_sizes(cfg)
        cap, cs = sz.select_slots, sz.cache_slots
        xs = {(b, g): wl.unit_inputs(0, b, g) for b in range(B) for g in range(Hkv)}
        W1 = np.stack([xs[(0, g)]["W1"] for g in range(Hkv)]).astype(np.float32)
        W2 = np.stack([xs[(0, g)]["W2"] for g in range(Hkv)]).astype(np.float32)
        N.nosa_set_eviction_head(ctx, 0, W1, W2)
        q = np.zeros((B, Hq, n, d), np.uint16)
        k = np.zeros((B, Hkv, n, d), np.uint16)
        v = np.zeros((B, Hkv, n, d), np.uint16)
        for (b, g), x in xs.items():
            q[b, g * G:(g + 1) * G] = x["Q"][:n].transpose(1, 0, 2)
            k[b, g] = x["K"][:n]
            v[b, g] = x["V"][:n]
        qd, kd, vd = _dev(q), _dev(k), _dev(v)
        out = torch.full((B, Hq, n, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        nbytes = N.nosa_prefill_scratch_bytes(ctx, n)
        W = (-(-n // 64) + 31) // 32  # bitmap words per position
        assert nbytes == 2 * U * n * W * 4  # query-aware, then query-agnostic picks
        scratch = torch.empty(nbytes // 2, dtype=torch.int16, device="cuda")
        N.nosa_prefill(ctx, 0, qd, kd, vd, n, out.view(torch.int16), scratch, nbytes)
        assert N.nosa_sync(ctx) == N.NOSA_OK
        assert N.nosa_context_length(ctx, 0) == n
        picks = scratch.view(torch.int32)[:2 * U * n * W].cpu().numpy().view(np.uint32).reshape(2, U, n, W)
        picks = np.unpackbits(picks.view(np.uint8), axis=-1, bitorder="little").astype(bool)  # [2][U][n][32 W]
        out_h = out.float().cpu().numpy()
        st = dict(sel=np.zeros((U, cap), np.int32), n_sel=np.zeros(U, np.int32), fetch=np.zeros((U, cap, 2), np.int32),
                  n_fetch=np.zeros(U, np.int32), slot_blk=np.zeros((U, cs), np.int32),
                  last_used=np.zeros((U, cs), np.int32),
                  evicted=np.zeros((U, sz.evict_words), np.uint32),
                  kt=np.zeros((U, max(sz.max_windows, 1), d), np.uint16))
        N.nosa_export_state(ctx, 0, **st)
        stats = N.nosa_get_stats(ctx)
        assert stats.selections == U * n

        oracles = {}
        for (b, g) in check_units:
            u = b * Hkv + g
            x = xs[(b, g)]
            o = O.UnitOracle(head_dim=d, k_q=wl.k_q, k_e=wl.k_e, sink_blocks=wl.sink_blocks,
                             window_tokens=wl.window_tokens, max_context=n + decode_steps, W1=x["W1"], W2=x["W2"],
                             dma_bias=bool(flags & N.NOSA_F_DMA_BIAS), cache_slots=cs)
            se_full = None
            if score_positions is not None:
                assert wl.window_tokens >= 2 * 64
                of = O.UnitOracle(head_dim=d, k_q=wl.k_q, k_e=wl.k_e, sink_blocks=wl.sink_blocks,
                                  window_tokens=wl.window_tokens, max_context=n, W1=x["W1"], W2=x["W2"])
                of.append(x["K"][:n], x["V"][:n])
                se_full = of.scores(x["Q"][n - 1])[1]
            r = None
            for t in range(n):
                o.append(x["K"][t:t + 1], x["V"][t:t + 1])
                Qg = np.flatnonzero(picks[0, u, t]).tolist()
                Eg = np.flatnonzero(picks[1, u, t]).tolist()
                sink_b, C_t, win_b = O.partition(o.T, o.nw, o.sink, o.block)
                assert not set(Qg) & set(Eg) and set(Qg) | set(Eg) <= set(C_t), f"picks of position {t} unit {u}"
                blocks = sorted(set(sink_b) | set(Qg) | set(Eg) | set(win_b))
                if score_positions is None or t in score_positions:
                    sq, se = o.scores(x["Q"][t])
                    Q, E = _select_and_adopt(o, sq, se, o.T, Qg, Eg, wl.k_q, wl.k_e, ties, (u, t))
                else:
                    _, C, _ = O.partition(o.T, o.nw, o.sink, o.block)
                    Q = Qg
                    assert len(Q) == min(wl.k_q, len(C)) and set(Q) <= set(C), f"query-aware picks {(u, t)}"
                    E = O.select_query_agnostic(se_full, C, Q, o.evicted, wl.k_e)
                    if E != Eg:
                        pool = [bb for bb in C if bb not in set(Q) and bb not in o.evicted]
                        assert _near_tie_ok(np.asarray(se_full).astype(np.float32), Eg, E, pool, wl.k_e), \
                            f"query-agnostic pick {(u, t)}"
                        ties.append(("e", (u, t)))
                        E = Eg
                r = o.commit(Q, E)
                assert blocks == r["S"], f"selection of position {t} unit {u}: {blocks} vs {r['S']}"
                if t in out_positions:
                    ref = o.attend(x["Q"][t], r["S"])
                    max_err = max(max_err, _check_out(out_h[b, g * G:(g + 1) * G, t], ref, f"unit {u} position {t}"))
            # the state after the prompt: the cache holds the last selection, block i in slot i,
            # nothing left to fetch
            o.settle_cache()
            assert np.array_equal(st["kt"][u, :o.nc], O.f64_to_bf16_bits(o.compressed_keys())), "K~"
            assert list(st["sel"][u, :st["n_sel"][u]]) == r["S"]
            assert list(st["slot_blk"][u]) == o.slot_blk, "slot map"
            assert list(st["last_used"][u]) == o.last_used, "slot recency"
            assert st["n_fetch"][u] == 0
            ev = st["evicted"][u]
            assert {bb for bb in range(o.nb) if (ev[bb >> 5] >> (bb & 31)) & 1} == o.evicted, "eviction bitmap"
            oracles[(b, g)] = o

        # decode continues from the prefill's state (cache slots refreshed from the prompt)
        for j in range(decode_steps):
            t = n + j
            qs = np.zeros((B, Hq, d), np.uint16)
            ks = np.zeros((B, Hkv, d), np.uint16)
            vs = np.zeros((B, Hkv, d), np.uint16)
            for (b, g), x in xs.items():
                qs[b, g * G:(g + 1) * G] = x["Q"][t]
                ks[b, g] = x["K"][t]
                vs[b, g] = x["V"][t]
            od = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
            N.nosa_step(ctx, 0, _dev(qs), _dev(ks), _dev(vs), od.view(torch.int16))
            assert N.nosa_sync(ctx) == N.NOSA_OK
            kinds = np.zeros((U, cap), np.int32)
            sel = np.zeros((U, cap), np.int32)
            nsel = np.zeros(U, np.int32)
            N.nosa_export_state(ctx, 0, sel=sel, sel_kind=kinds, n_sel=nsel)
            oh = od.float().cpu().numpy()
            for (b, g), o in oracles.items():
                u = b * Hkv + g
                x = xs[(b, g)]
                o.append(x["K"][t:t + 1], x["V"][t:t + 1])
                sq, se = o.scores(x["Q"][t])
                S_gpu = list(sel[u, :nsel[u]])
                Qg = sorted(int(bb) for bb, kk in zip(S_gpu, kinds[u, :nsel[u]]) if kk == 2)
                Eg = sorted(int(bb) for bb, kk in zip(S_gpu, kinds[u, :nsel[u]]) if kk == 3)
                Q, E = _select_and_adopt(o, sq, se, o.T, Qg, Eg, wl.k_q, wl.k_e, ties, (u, t))
                r = o.commit(Q, E)
                assert S_gpu == r["S"], f"decode step {j} after the prefill, unit {u}"
                max_err = max(max_err, _check_out(oh[b, g * G:(g + 1) * G], o.attend(x["Q"][t], r["S"]),
                                                  f"decode step {j} unit {u}"))
    finally:
        N.nosa_destroy(ctx)
    print(f"[prefill n={n}] units={len(check_units)} near_ties={len(ties)} max_out_abs={max_err:.2e}")
    return ties


# NOSA_F_TEST_PREFILL_WIDE: the kernel forms prompts of more than 65,536 tokens take (two positions
# per query-aware warp, two bitmap words per walk lane), here on short prompts
TILE = pytest.mark.parametrize("tile", [0, N.NOSA_F_TEST_PREFILL_WIDE], ids=["short-form", "wide-form"])


@TILE
@pytest.mark.parametrize("mode", [FUSED, UNFUSED], ids=["fused-decode", "three-kernel-decode"])
def test_prefill_640_every_position(mode, tile):
    # k = 3 with a 2-block window: the selection turns sparse once the prompt passes 6 blocks, so
    # evictions and the window sliding over the budget all happen inside the prompt
    wl = syn.Workload("pf640", layers=1, batch=2, q_heads=16, kv_heads=2, context=0, k_q=1, k_e=2,
                      window_tokens=128, steps=644, sigma=0.3)
    units = [(b, g) for b in range(2) for g in range(2)]
    run_prefill(wl, 640, units, set(range(640)), flags=mode | tile, decode_steps=4)


def test_prefill_with_a_cache_of_one_selection():
    # the pages' cache size (sink + window + k_q + k_e slots): the same state after the prompt,
    # and the decode steps after it replace exactly the slots whose blocks left the selection
    wl = syn.Workload("pf640c", layers=1, batch=2, q_heads=16, kv_heads=2, context=0, k_q=1, k_e=2,
                      window_tokens=128, steps=650, sigma=0.3)
    units = [(b, g) for b in range(2) for g in range(2)]
    run_prefill(wl, 640, units, set(range(0, 640, 7)), decode_steps=8, cache_slots=1 + 2 + 1 + 2)


@TILE
def test_prefill_ragged_group4_dma_bias(tile):
    # a prompt that ends mid-block and mid-window, 4 q heads per kv head, 6 units (two walk CTAs),
    # with the attention bias
    wl = syn.Workload("pf_ragged", layers=1, batch=3, q_heads=8, kv_heads=2, context=0, k_q=3, k_e=5,
                      window_tokens=128, steps=1004, sigma=1.0)
    units = [(b, g) for b in range(3) for g in range(2)]
    run_prefill(wl, 1001, units, set(range(1001)), flags=N.NOSA_F_DMA_BIAS | tile, decode_steps=3)


@pytest.mark.parametrize("hq", [2, 4, 6], ids=["group1", "group2", "group3"])
def test_prefill_small_groups(hq):
    # 1, 2 and 3 q heads per kv head: the tensor-core query-aware scores with 32, 64 and 96 of
    # their 128 rows in use, and the attention's last rows idle when 128 is not a multiple of G
    wl = syn.Workload(f"pf_g{hq // 2}", layers=1, batch=2, q_heads=hq, kv_heads=2, context=0, k_q=4, k_e=6,
                      window_tokens=128, steps=1203, sigma=1.0)
    units = [(b, g) for b in range(2) for g in range(2)]
    run_prefill(wl, 1200, units, set(range(0, 1200, 3)) | {1199}, decode_steps=2)


@pytest.mark.parametrize("window", [0, 64], ids=["no-window", "one-block-window"])
def test_prefill_short_window(window):
    # with a window of fewer than two blocks the last two blocks are candidates, whose pooled
    # eviction scores still change as the prompt grows: the walk re-ranks them at every position
    wl = syn.Workload(f"pf_w{window}", layers=1, batch=1, q_heads=16, kv_heads=2, context=0, k_q=2, k_e=3,
                      window_tokens=window, steps=803, sigma=1.0)
    units = [(0, 0), (0, 1)]
    run_prefill(wl, 800, units, set(range(0, 800, 7)) | {799}, decode_steps=3)


@pytest.mark.parametrize("kq,ke", [(40, 8), (0, 6), (5, 0)], ids=["kq40", "kq0", "ke0"])
def test_prefill_pick_counts(kq, ke):
    # more query-aware picks than a warp ranks in one round (40: two rounds), and either part empty
    n = 3500 if kq == 40 else 900
    wl = syn.Workload(f"pf_k{kq}_{ke}", layers=1, batch=1, q_heads=16, kv_heads=2, context=0, k_q=kq, k_e=ke,
                      window_tokens=128, steps=n + 3, sigma=1.0)
    units = [(0, 0), (0, 1)]
    run_prefill(wl, n, units, set(range(0, n, 13)) | {n - 1}, decode_steps=3)


def test_prefill_16k_prompt_sampled_positions():
    # the 1B-shaped layer (16/2 heads, k_q 16, k_e 48, 1024-token window) over a 16K prompt: one
    # unit's selection checked at every position, its outputs at sampled positions
    n = 16384
    wl = syn.Workload("pf16k", layers=1, batch=1, q_heads=16, kv_heads=2, context=0, k_q=16, k_e=48,
                      window_tokens=1024, steps=n + 2, sigma=0.3)
    pos = set(range(0, n, 61)) | set(range(n - 8, n)) | {63, 64, 65, 1023, 1024, 1025}
    run_prefill(wl, n, [(0, 1)], pos, decode_steps=2)


def test_prefill_70k_prompt_long_forms():
    # 70,000 tokens (1,094 blocks): the long-prompt kernel forms for real, block ids past 1,024 in
    # the bitmaps' second words.  Every position's query-agnostic picks, eviction state, selection
    # and slots against the oracle; the query-aware picks against the oracle's own scores at
    # sampled positions (elsewhere checked for count and range, then adopted)
    n = 70000
    wl = syn.Workload("pf70k", layers=1, batch=1, q_heads=16, kv_heads=2, context=0, k_q=16, k_e=48,
                      window_tokens=1024, steps=n + 2, sigma=0.3)
    scored = set(range(0, n, 4999)) | {65535, 65536, 65600, n - 1}
    out = set(range(0, n, 997)) | {n - 1}
    run_prefill(wl, n, [(0, 0)], out, decode_steps=2, score_positions=scored)


def test_prefill_40k_prompt_group4():
    # the 8B-shaped group (32/8 heads: 4 per kv head) over 40,000 tokens (625 blocks): the
    # tensor-core query-aware scores keep fewer positions per CTA (26) so that their pooled
    # scores fit in shared memory, the last CTA ragged
    n = 40000
    wl = syn.Workload("pf40k_g4", layers=1, batch=1, q_heads=8, kv_heads=2, context=0, k_q=16, k_e=48,
                      window_tokens=1024, steps=n + 2, sigma=0.3)
    scored = set(range(0, n, 3001)) | {25, 26, 27, 51, 52, n - 1}
    out = set(range(0, n, 499)) | {n - 1}
    run_prefill(wl, n, [(0, 1)], out, decode_steps=2, score_positions=scored)


def test_prefill_argument_checks():
    cfg = N.make_config(num_layers=2, batch=1, num_q_heads=16, num_kv_heads=2, k_q=2, k_e=2, window_tokens=128,
                        max_context=300)
    ctx = N.nosa_create(cfg, torch.cuda.current_stream().cuda_stream)
    try:
        n = 200
        q = torch.zeros((1, 16, n, 128), dtype=torch.int16, device="cuda")
        kv = torch.zeros((1, 2, n, 128), dtype=torch.int16, device="cuda")
        nb = N.nosa_prefill_scratch_bytes(ctx, n)
        scratch = torch.zeros(nb // 2 + 8, dtype=torch.int16, device="cuda")
        with pytest.raises(N.NosaError) as e:      # scratch too small
            N.nosa_prefill(ctx, 0, q, kv, kv, n, q, scratch, nb - 2)
        assert e.value.status == N.NOSA_ERR_CAPACITY
        with pytest.raises(N.NosaError) as e:      # longer than the context's capacity
            N.nosa_prefill(ctx, 0, q, kv, kv, 301, q, scratch, nb)
        assert e.value.status == N.NOSA_ERR_CAPACITY
        N.nosa_prefill(ctx, 0, q, kv, kv, n, q, scratch, nb)
        with pytest.raises(N.NosaError) as e:      # the layer is no longer empty
            N.nosa_prefill(ctx, 0, q, kv, kv, n, q, scratch, nb)
        assert e.value.status == N.NOSA_ERR_STATE
        N.nosa_prefill(ctx, 1, q, kv, kv, 1, q, scratch, nb)   # a one-token prompt
        assert N.nosa_sync(ctx) == N.NOSA_OK
        assert N.nosa_context_length(ctx, 0) == n and N.nosa_context_length(ctx, 1) == 1
    finally:
        N.nosa_destroy(ctx)
