"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Selections, fetch lists, slots, eviction bitmaps and
compressed keys bit-exact (near ties logged and adopted, see nosa_harness);
pooled scores within 1e-4 relative; outputs within 2e-2 max-abs / 2e-3 mean-abs."""
import math

import numpy as np
import pytest

from synth import inputs as syn

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # collected on CPU machines too; every test here is marked gpu
    pytest.skip("no CUDA device", allow_module_level=True)

from tests.nosa_harness import Parity  # noqa: E402
from offloadable_block_sparse_gb300 import nosa as N  # noqa: E402


FUSED, UNFUSED = 0, N.NOSA_F_UNFUSED_STEP
STEP_MODES = pytest.mark.parametrize("mode", [FUSED, UNFUSED], ids=["fused", "three-kernels"])


def run(wl, steps, samples=None, layers=None, split_calls=False, gather_ctas=0, separate_fetch=True, flags=0,
        plan=None, **sizing):
    p = Parity(wl, sample_units=samples, layers=layers, gather_ctas=gather_ctas, flags=flags, **sizing)
    try:
        if plan is not None:  # the step form the test is about is the one that runs
            assert N.nosa_step_plan(p.ctx) == plan, N.nosa_step_plan(p.ctx)
        p.load_context()
        for _ in range(steps):
            p.run_step(split_calls=split_calls, separate_fetch=separate_fetch)
        assert N.nosa_sync(p.ctx) == N.NOSA_OK
        stats = N.nosa_get_stats(p.ctx)
        return p.log, stats
    finally:
        p.close()


def _report(name, log, stats=None):
    print(f"[{name}] steps={log.steps} unit_steps={log.unit_steps} near_ties={len(log.near_ties)} "
          f"max_out_abs={log.max_out_abs:.2e} max_mean_abs={log.max_out_mean_abs:.2e} "
          f"max_score_rel={log.max_score_rel:.2e} gamma_min={min(log.gammas) if log.gammas else None}")


@STEP_MODES
def test_tiny_every_step_every_unit(mode):
    wl = syn.workload("tiny")
    log, stats = run(wl, wl.steps, flags=mode)
    _report("tiny", log, stats)
    assert log.unit_steps == wl.steps * 2
    assert min(log.gammas) >= wl.k_e / (wl.k_q + wl.k_e) - 1e-12   # Theorem 2 on the GPU path
    assert stats.gamma_min >= wl.k_e / (wl.k_q + wl.k_e) - 1e-6


def test_tiny_through_separate_calls():
    wl = syn.workload("tiny", steps=12)
    log, _ = run(wl, wl.steps, split_calls=True)
    assert log.unit_steps == 24


def test_separate_calls_attend_fetches_itself():
    # select then attend without nosa_fetch: the attention kernel copies the new blocks itself
    wl = syn.Workload("fused", layers=2, batch=2, q_heads=16, kv_heads=2, context=3001, k_q=4, k_e=8,
                      window_tokens=256, steps=40, sigma=1.0)
    log, _ = run(wl, wl.steps, split_calls=True, separate_fetch=False)
    assert log.unit_steps == 40 * 8


@STEP_MODES
def test_tiny_with_dma_attention_bias(mode):
    # attention logits get each token's eviction score added; sigma 1.0 moves the selection
    wl = syn.workload("tiny", steps=24, sigma=1.0)
    log, _ = run(wl, wl.steps, flags=mode | N.NOSA_F_DMA_BIAS)
    _report("tiny-dma", log)
    assert log.unit_steps == 48


def test_dma_bias_through_separate_calls():
    wl = syn.workload("tiny", steps=10)
    p = Parity(wl, flags=N.NOSA_F_DMA_BIAS)
    try:
        p.load_context()
        for _ in range(wl.steps):
            p.run_step(split_calls=True, separate_fetch=False)
        assert N.nosa_sync(p.ctx) == N.NOSA_OK
    finally:
        p.close()


@STEP_MODES
def test_ragged_context_group4_small_window(mode):
    # T_0 not a multiple of 64 or 16: the tail block is partial and is fetched on the first step;
    # 8 q heads over 2 kv heads (G = 4)
    wl = syn.Workload("ragged", layers=2, batch=3, q_heads=8, kv_heads=2, context=1001, k_q=3, k_e=5,
                      window_tokens=128, steps=70, sigma=1.0)
    log, _ = run(wl, wl.steps, flags=mode)
    _report("ragged", log)
    assert log.unit_steps == 70 * 12


@STEP_MODES
def test_short_context_everything_selected(mode):
    # fewer blocks than the budget: every block is selected, so attention is dense
    wl = syn.Workload("short", layers=1, batch=2, q_heads=16, kv_heads=2, context=40, k_q=4, k_e=12,
                      window_tokens=256, steps=30)
    log, _ = run(wl, wl.steps, flags=mode)
    assert log.unit_steps == 30 * 4


@STEP_MODES
def test_no_sink_no_window_query_aware_only(mode):
    wl = syn.Workload("kq_only", layers=1, batch=2, q_heads=4, kv_heads=1, context=3000, k_q=8, k_e=0,
                      window_tokens=0, sink_blocks=0, steps=20, sigma=1.0)
    log, _ = run(wl, wl.steps, flags=mode)
    assert log.unit_steps == 40


@STEP_MODES
def test_sparse_prefill_by_steps_from_one_token(mode):
    # NOSA_S prefill: the eviction constraint is defined per step, so the selection for prompt
    # position t is the decode selection at t; the prompt is fed one token at a time from a
    # one-token context.  With k = 3 the selection turns sparse once the prompt passes 6 blocks
    # (sink 1 + window 2 + k 3): the first complete windows, the first evictions and the window
    # sliding over the budget all happen inside the prompt.
    wl = syn.Workload("prefill", layers=1, batch=2, q_heads=16, kv_heads=2, context=1, k_q=1, k_e=2,
                      window_tokens=128, steps=640)
    log, stats = run(wl, wl.steps, flags=mode)
    assert log.unit_steps == 640 * 4
    assert log.gammas and min(log.gammas) >= 2 / 3 - 1e-6  # Theorem 2: gamma >= k_e / k
    assert min(log.gammas) < 1.0  # the selection moved: blocks were dropped during the prompt


@pytest.mark.parametrize("ctas", [1, 8, 64, 152])
def test_gather_cta_counts_agree(ctas):
    # the separate calls with nosa_fetch: the persistent gather kernel copies every new block
    # (the cold first step's whole selection, then the query-aware picks) at each CTA count
    wl = syn.Workload("ctas", layers=2, batch=4, q_heads=16, kv_heads=2, context=4096, k_q=4, k_e=12,
                      window_tokens=256, steps=8, sigma=1.0)
    log, stats = run(wl, wl.steps, gather_ctas=ctas, split_calls=True, separate_fetch=True)
    assert log.unit_steps == 8 * 16
    assert log.fetched > 16 * 21  # more than the cold step's blocks: later steps fetched too
    assert stats.blocks_fetched == log.fetched


# Kernel sizing overrides (nosa_config): every non-default choice against the oracle, with the
# step form it belongs to checked through nosa_step_plan.  sigma 1.0 moves the selection.
SIZING = [
    (dict(score_ctas=1), UNFUSED, (3, 0)),
    (dict(score_ctas=3), UNFUSED, (3, 0)),
    (dict(score_ctas=8), UNFUSED, (3, 0)),
    (dict(attend_blocks_per_cta=1), UNFUSED, (3, 0)),
    (dict(attend_blocks_per_cta=64), UNFUSED, (3, 0)),
    (dict(attend_merge=N.NOSA_MERGE_TICKET), UNFUSED, (2, 0)),
    (dict(attend_merge=N.NOSA_MERGE_CLUSTER), UNFUSED, (2, 0)),
    (dict(attend_merge=N.NOSA_MERGE_TICKET, attend_blocks_per_cta=3), UNFUSED, (2, 0)),
    (dict(decode_cluster=1), FUSED, (1, 1)),
    (dict(decode_cluster=2), FUSED, (1, 2)),
    (dict(decode_cluster=8), FUSED, (1, 8)),
    (dict(decode_teams=1), FUSED, None),
    (dict(decode_stages=2), FUSED, None),
    (dict(decode_teams=1, decode_stages=6), FUSED, None),
    (dict(cache_slots=21), FUSED, None),      # a cache of one selection (the pages' cache)
    (dict(cache_slots=21), UNFUSED, (3, 0)),
    (dict(cache_slots=64), FUSED, None),      # three selections' worth: fewer fetches still
    (dict(cache_slots=256), UNFUSED, (3, 0)),
]


@pytest.mark.parametrize("sizing,mode,plan", SIZING,
                         ids=["-".join(f"{k}{v}" for k, v in z.items()) for z, _, _ in SIZING])
def test_sizing_overrides(sizing, mode, plan):
    wl = syn.workload("tiny", steps=16, sigma=1.0)
    log, _ = run(wl, wl.steps, flags=mode, plan=plan, **sizing)
    assert log.unit_steps == 32
    if mode == FUSED:  # the fused kernel, not the chain, ran
        p = Parity(wl, sample_units=[], flags=mode, **sizing)
        try:
            assert N.nosa_step_plan(p.ctx)[0] == 1
        finally:
            p.close()
    # the separate calls with the same sizing
    log, _ = run(syn.workload("tiny", steps=6, sigma=1.0), 6, flags=mode, split_calls=True, **sizing)
    assert log.unit_steps == 12


@STEP_MODES
def test_radix_topk_hook(mode):
    # the warp radix select for the query-agnostic part at every step (normally only beyond 1024
    # eligible blocks): the same selections as the oracle's
    wl = syn.workload("tiny", steps=24, sigma=1.0)
    log, _ = run(wl, wl.steps, flags=mode | N.NOSA_F_TEST_RADIX_TOPK)
    assert log.unit_steps == 48


@STEP_MODES
def test_long_context_first_selection_takes_the_radix_select(mode):
    # 70,000 tokens: 1094 blocks, so the first selection after the bulk load has more than 1024
    # eligible blocks (every candidate outside the query-aware picks) and takes the warp radix
    # select without any hook; later steps rank the few never-dropped candidates directly
    wl = syn.Workload("long70k", layers=1, batch=2, q_heads=16, kv_heads=2, context=70000, k_q=16, k_e=48,
                      window_tokens=1024, steps=3, sigma=0.3)
    nb = -(-70001 // 64)
    assert nb - 16 - 1 - 16 > 1024
    log, _ = run(wl, wl.steps, flags=mode)
    assert log.unit_steps == 3 * 4


def test_capacity_error_leaves_state_unchanged():
    wl = syn.Workload("cap", layers=1, batch=1, q_heads=16, kv_heads=2, context=100, k_q=2, k_e=2,
                      window_tokens=128, steps=2)
    p = Parity(wl)
    try:
        p.load_context()
        p.run_step()
        p.run_step()
        k = torch.zeros((1, 2, 128), dtype=torch.int16, device="cuda")
        with pytest.raises(N.NosaError) as e:
            N.nosa_append_kv(p.ctx, 0, k, k, 1)
        assert e.value.status == N.NOSA_ERR_CAPACITY
        assert N.nosa_context_length(p.ctx, 0) == 102
        assert N.nosa_sync(p.ctx) == N.NOSA_OK
    finally:
        p.close()


def test_step_plan_follows_the_flag():
    wl = syn.workload("tiny")
    for flags, kernels in ((FUSED, 1), (UNFUSED, 3)):
        p = Parity(wl, flags=flags)
        try:
            k, cs = N.nosa_step_plan(p.ctx)
            assert k == kernels and (cs > 0) == (kernels == 1)
        finally:
            p.close()


def test_out_of_order_calls_are_rejected():
    wl = syn.Workload("order", layers=1, batch=1, q_heads=16, kv_heads=2, context=300, k_q=2, k_e=2,
                      window_tokens=128, steps=2)
    p = Parity(wl)
    try:
        p.load_context()
        q = torch.zeros((1, 16, 128), dtype=torch.int16, device="cuda")
        with pytest.raises(N.NosaError) as e:
            N.nosa_attend(p.ctx, 0, q, q)   # no selection for this length yet
        assert e.value.status == N.NOSA_ERR_STATE
        with pytest.raises(N.NosaError):
            N.nosa_fetch(p.ctx, 0)
        with pytest.raises(N.NosaError):
            N.nosa_step(p.ctx, 5, q, q, q, q)
    finally:
        p.close()


def _one_step(p):
    q, k, v = p.step_inputs(0)
    out = torch.empty_like(q)
    N.nosa_step(p.ctx, 0, q.view(torch.int16), k.view(torch.int16), v.view(torch.int16), out.view(torch.int16))


@pytest.mark.parametrize("flag,status", [(N.NOSA_F_TEST_ZERO_WAIT, N.NOSA_ERR_TIMEOUT),
                                         (N.NOSA_F_TEST_BAD_SLOT, N.NOSA_ERR_BOUNDS)])
def test_device_errors_are_latched_and_recoverable(flag, status):
    # Failure detection without a fault or a hang: a test hook makes the attention kernel's
    # bounded waits give up at once, or publishes an out-of-range slot that the kernel clamps.
    wl = syn.Workload("hook", layers=1, batch=2, q_heads=16, kv_heads=2, context=2048, k_q=4, k_e=12,
                      window_tokens=256, steps=4)
    p = Parity(wl, sample_units=[], flags=flag)
    try:
        p.load_context()
        got = N.NOSA_OK
        for _ in range(2):  # the first step after a cold start may read every block from host memory
            _one_step(p)
            got = N.nosa_sync(p.ctx)
            if got != N.NOSA_OK:
                break
        assert got == status
        with pytest.raises(N.NosaError) as e:     # the context stays failed ...
            _one_step(p)
        assert e.value.status == N.NOSA_ERR_STATE
        N.nosa_reset_state(p.ctx)                 # ... until the error is cleared
        assert N.nosa_sync(p.ctx) == N.NOSA_OK
    finally:
        p.close()


def test_host_pointer_step_matches_device_step():
    # nosa_step_host reads page-locked inputs in place and copies pageable ones; both must give
    # exactly the device-pointer step's outputs (same kernels, same inputs, deterministic merges).
    wl = syn.Workload("host", layers=2, batch=3, q_heads=16, kv_heads=2, context=1500, k_q=4, k_e=12,
                      window_tokens=256, steps=6)
    ps = [Parity(wl, sample_units=[]) for _ in range(3)]
    try:
        for p in ps:
            p.load_context()
        gen = torch.Generator(device="cuda").manual_seed(77)
        for t in range(wl.steps):
            for l in range(wl.layers):
                q = torch.randn((wl.batch, wl.q_heads, 128), generator=gen, device="cuda")
                q = (q / q.norm(dim=-1, keepdim=True) * math.sqrt(128)).to(torch.bfloat16)
                k = torch.randn((wl.batch, wl.kv_heads, 128), generator=gen, device="cuda").to(torch.bfloat16)
                v = torch.randn((wl.batch, wl.kv_heads, 128), generator=gen, device="cuda").to(torch.bfloat16)
                outs = []
                out_d = torch.empty_like(q)
                N.nosa_step(ps[0].ctx, l, q.view(torch.int16), k.view(torch.int16), v.view(torch.int16),
                            out_d.view(torch.int16))
                outs.append(out_d)
                for p, pin in ((ps[1], True), (ps[2], False)):
                    hq, hk, hv = (x.cpu() for x in (q, k, v))
                    ho = torch.empty_like(hq)
                    if pin:
                        hq, hk, hv, ho = hq.pin_memory(), hk.pin_memory(), hv.pin_memory(), ho.pin_memory()
                    N.nosa_step_host(p.ctx, l, hq.view(torch.int16), hk.view(torch.int16), hv.view(torch.int16),
                                     ho.view(torch.int16))
                    assert N.nosa_sync(p.ctx) == N.NOSA_OK
                    outs.append(ho)
                assert N.nosa_sync(ps[0].ctx) == N.NOSA_OK
                ref = outs[0].cpu().view(torch.int16)
                for o in outs[1:]:
                    assert torch.equal(o.view(torch.int16), ref), (t, l)
    finally:
        for p in ps:
            p.close()


@pytest.mark.parametrize("pin", [True, False], ids=["page-locked", "pageable"])
def test_whole_step_host_call_matches_per_layer_steps(pin):
    # nosa_step_host_all copies every layer's inputs at once, runs the layers and copies the
    # outputs back: the same outputs and state as nosa_step per layer on device inputs.  The
    # workload's capacity is context + steps, so the call after the last step is refused.
    wl = syn.Workload("host_all", layers=3, batch=3, q_heads=16, kv_heads=2, context=1500, k_q=4, k_e=12,
                      window_tokens=256, steps=5)
    ps = [Parity(wl, sample_units=[]) for _ in range(2)]
    try:
        for p in ps:
            p.load_context()
        gen = torch.Generator(device="cuda").manual_seed(78)
        L, B, Hq, Hkv = wl.layers, wl.batch, wl.q_heads, wl.kv_heads
        for t in range(wl.steps):
            q = torch.randn((L, B, Hq, 128), generator=gen, device="cuda")
            q = (q / q.norm(dim=-1, keepdim=True) * math.sqrt(128)).to(torch.bfloat16)
            k = torch.randn((L, B, Hkv, 128), generator=gen, device="cuda").to(torch.bfloat16)
            v = torch.randn((L, B, Hkv, 128), generator=gen, device="cuda").to(torch.bfloat16)
            out_d = torch.empty_like(q)
            for l in range(L):
                N.nosa_step(ps[0].ctx, l, q[l].view(torch.int16), k[l].view(torch.int16), v[l].view(torch.int16),
                            out_d[l].view(torch.int16))
            hq, hk, hv = (x.cpu() for x in (q, k, v))
            ho = torch.full_like(hq, float("nan"))
            if pin:
                hq, hk, hv, ho = hq.pin_memory(), hk.pin_memory(), hv.pin_memory(), ho.pin_memory()
            N.nosa_step_host_all(ps[1].ctx, hq.view(torch.int16), hk.view(torch.int16), hv.view(torch.int16),
                                 ho.view(torch.int16))
            for p in ps:
                assert N.nosa_sync(p.ctx) == N.NOSA_OK
            assert torch.equal(ho.view(torch.int16), out_d.cpu().view(torch.int16)), f"step {t}"
        for l in range(L):
            a, b = ps[0]._export(l), ps[1]._export(l)
            for key in ("sel", "sel_slot", "slot_blk", "evicted", "n_sel"):
                assert np.array_equal(a[key], b[key]), (l, key)
        T_before = [N.nosa_context_length(ps[1].ctx, l) for l in range(L)]
        hq = torch.zeros((L, B, Hq, 128), dtype=torch.bfloat16)
        hk = torch.zeros((L, B, Hkv, 128), dtype=torch.bfloat16)
        ho = torch.zeros_like(hq)
        with pytest.raises(N.NosaError) as e:
            N.nosa_step_host_all(ps[1].ctx, hq.view(torch.int16), hk.view(torch.int16), hk.view(torch.int16),
                                 ho.view(torch.int16))
        assert e.value.status == N.NOSA_ERR_CAPACITY
        assert [N.nosa_context_length(ps[1].ctx, l) for l in range(L)] == T_before
    finally:
        for p in ps:
            p.close()


# ----------------------------------------------------------------------------- forecast (SparDA)
@pytest.mark.parametrize("separate_fetch", [True, False], ids=["prefetch", "attend-fetches"])
def test_forecast_selection_every_step(separate_fetch):
    # selection one layer ahead with a forecast vector per kv head; the fetch either runs before
    # the append (as a prefetch would) or is left to the attention after it
    wl = syn.workload("tiny", steps=40, sigma=1.0)
    p = Parity(wl)
    try:
        p.load_context()
        for _ in range(wl.steps):
            p.run_forecast_step(separate_fetch=separate_fetch)
        assert N.nosa_sync(p.ctx) == N.NOSA_OK
        _report("forecast", p.log)
        assert p.log.unit_steps == 80
        assert min(p.log.gammas) >= wl.k_e / (wl.k_q + wl.k_e) - 1e-12
    finally:
        p.close()


def test_forecast_new_tail_block_is_prefetched():
    # T0 a multiple of 64: the first forecast serves the token that starts a new block
    wl = syn.Workload("fc_tail", layers=1, batch=2, q_heads=16, kv_heads=2, context=2048, k_q=4, k_e=12,
                      window_tokens=256, steps=70, sigma=1.0)
    p = Parity(wl)
    try:
        p.load_context()
        for _ in range(wl.steps):
            p.run_forecast_step()
        assert p.log.unit_steps == 70 * 4
    finally:
        p.close()


@pytest.mark.parametrize("streams", [0, 1], ids=["two-streams", "one-stream"])
def test_forecast_pipeline_overlaps_the_next_layer(streams):
    wl = syn.Workload("fc_pipe", layers=3, batch=3, q_heads=16, kv_heads=2, context=3000, k_q=4, k_e=12,
                      window_tokens=256, steps=30, sigma=1.0)
    p = Parity(wl, forecast_streams=streams)
    try:
        p.load_context()
        p.run_forecast_pipeline(wl.steps)
        _report("forecast-pipeline", p.log)
        assert p.log.unit_steps == 30 * 3 * 3 * 2
        assert min(p.log.gammas) >= wl.k_e / (wl.k_q + wl.k_e) - 1e-12
    finally:
        p.close()


def test_forecast_call_order_is_checked():
    wl = syn.Workload("fc_order", layers=2, batch=1, q_heads=16, kv_heads=2, context=500, k_q=2, k_e=2,
                      window_tokens=128, steps=2)
    p = Parity(wl)
    try:
        p.load_context()
        q = torch.zeros((1, 16, 128), dtype=torch.int16, device="cuda")
        kv = torch.zeros((1, 2, 128), dtype=torch.int16, device="cuda")
        f = torch.zeros((1, 2, 128), dtype=torch.int16, device="cuda")
        with pytest.raises(N.NosaError) as e:     # no forecast for this token yet
            N.nosa_step_forecast(p.ctx, 0, q, kv, kv, q)
        assert e.value.status == N.NOSA_ERR_STATE
        N.nosa_forecast_select(p.ctx, 0, f)
        with pytest.raises(N.NosaError) as e:     # one forecast per token
            N.nosa_forecast_select(p.ctx, 0, f)
        assert e.value.status == N.NOSA_ERR_STATE
        with pytest.raises(N.NosaError) as e:     # the next layer must differ
            N.nosa_step_forecast(p.ctx, 0, q, kv, kv, q, f, 0)
        assert e.value.status == N.NOSA_ERR_INVALID_ARG
        N.nosa_step_forecast(p.ctx, 0, q, kv, kv, q, f, 1)
        N.nosa_step_forecast(p.ctx, 1, q, kv, kv, q)
        N.nosa_forecast_join(p.ctx)
        assert N.nosa_sync(p.ctx) == N.NOSA_OK
        assert N.nosa_context_length(p.ctx, 0) == 501 and N.nosa_context_length(p.ctx, 1) == 501
    finally:
        p.close()


def test_forecast_pipeline_full_size_sampled():
    # the 1B, 16K, batch-8 workload's per-layer shape, all 28 layers pipelined, sampled units checked
    wl = syn.workload("nosa1b_16k_b8")
    p = Parity(wl, sample_units=[(0, 0, 0), (13, 5, 1), (27, 7, 0)])
    try:
        p.load_context()
        p.run_forecast_pipeline(24)
        _report("forecast-c2", p.log)
        assert p.log.unit_steps == 24 * 3
    finally:
        p.close()


# Full-size workloads, every unit run on the GPU, sampled units checked against the oracle at every
# step.  The 8B-shaped workload keeps its per-layer sizes (32 sequences x 8 kv heads x 32K tokens)
# but runs 8 of its 32 layers: its full host store (138 GB pinned) exceeds the test machine's RAM.
FULL = [
    ("nosa1b_16k_b8", 256, [(0, 0, 0), (5, 3, 1), (17, 7, 0), (27, 6, 1)], None, {}),
    ("nosa1b_16k_b8", 96, [(2, 1, 0), (26, 4, 1)], None, {"flags": UNFUSED}),
    ("nosa1b_16k_b8", 64, [(1, 2, 1), (27, 7, 0)], None, {"flags": N.NOSA_F_DMA_BIAS}),
    ("nosa1b_16k_b128", 128, [(0, 0, 0), (13, 77, 1), (27, 127, 0)], None, {}),
    ("nosa1b_16k_b128", 64, [(3, 5, 0), (20, 100, 1)], None, {"sigma": 1.0}),
    ("nosa8b_32k_b32", 128, [(0, 0, 0), (4, 17, 5), (7, 31, 7)], 8, {}),
    ("nosa1b_64k_b32", 64, [(0, 0, 0), (14, 9, 1), (27, 31, 0)], None, {}),
    ("nosa1b_64k_b32", 32, [(1, 2, 1), (26, 30, 0)], None, {"k_q": 32, "k_e": 32}),
]


@pytest.mark.parametrize("name,steps,samples,layers,over", FULL,
                         ids=[f"{n}-{s}steps-{'-'.join(f'{k}{v}' for k, v in o.items()) or 'base'}"
                              for n, s, _, _, o in FULL])
def test_full_size_sampled(name, steps, samples, layers, over):
    over = dict(over)
    flags = over.pop("flags", 0)
    wl = syn.workload(name, **over)
    log, stats = run(wl, steps, samples=samples, layers=layers, flags=flags)
    _report(name, log, stats)
    assert log.unit_steps == steps * len(samples)
    assert stats.gamma_min >= wl.k_e / (wl.k_q + wl.k_e) - 1e-6
