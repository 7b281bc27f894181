"""nosa_attend_noalloc against the CPU oracle.

The no-allocation entry point serves callers that must not call cudaMalloc
(they run inside a memory pool they do not own, under an allocator that is
being captured or audited, or on a path that may not grow the device footprint
after start-up).  It runs the split-K attention with its scratch in a fixed
device array and merges the partials in each unit's last CTA.  This test drives
a context for a few decode steps to get real selections, rebuilds that
context's block cache from the known K/V, and checks two no-allocation calls in
a row against the oracle's sparse attention (NOSA explainer, eq. 8) over the
same selection, within the parity tolerance of the decode path (max-abs 2e-2,
mean-abs 2e-3).  Each call's reported error word must be clear; a selection
count above the cache and an out-of-range slot are clamped by the kernel and
reported.  The file name sorts last so that a run stopping at the first failure
has already run every other test.
"""
import math

import numpy as np
import pytest

from oracle import nosa_oracle as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from offloadable_block_sparse_gb300 import nosa as N  # noqa: E402


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def test_noalloc_attend_matches_the_oracle_twice():
    torch.cuda.set_device(0)
    B, Hq, Hkv, d, T0, steps = 3, 16, 2, 128, 2000, 3
    G, U = Hq // Hkv, B * Hkv
    cfg = N.make_config(num_layers=1, batch=B, num_q_heads=Hq, num_kv_heads=Hkv, k_q=4, k_e=12,
                        window_tokens=256, max_context=T0 + steps)
    cfg.cache_slots = N.nosa_query_sizes(cfg).select_slots  # a cache of one selection: the entry point's layout
    stream = torch.cuda.current_stream()
    ctx = N.nosa_create(cfg, stream.cuda_stream)
    try:
        cap = N.nosa_query_sizes(cfg).cache_slots
        gen = torch.Generator(device="cuda").manual_seed(5)
        Kall = torch.randn((B, Hkv, T0 + steps, d), generator=gen, device="cuda").to(torch.bfloat16)
        Vall = torch.randn((B, Hkv, T0 + steps, d), generator=gen, device="cuda").to(torch.bfloat16)
        W1 = (torch.randn((Hkv, d, 128)) / math.sqrt(d)).float().contiguous()
        W2 = (torch.randn((Hkv, 128)) / math.sqrt(128)).float().contiguous()
        N.nosa_set_eviction_head(ctx, 0, W1.numpy(), W2.numpy())
        N.nosa_append_kv(ctx, 0, Kall[:, :, :T0].contiguous().view(torch.int16),
                         Vall[:, :, :T0].contiguous().view(torch.int16), T0)
        out_ctx = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
        for t in range(steps):
            q = torch.randn((B, Hq, d), generator=gen, device="cuda")
            q = (q / q.norm(dim=-1, keepdim=True) * math.sqrt(d)).to(torch.bfloat16)
            k = Kall[:, :, T0 + t].contiguous()
            v = Vall[:, :, T0 + t].contiguous()
            N.nosa_step(ctx, 0, q.view(torch.int16), k.view(torch.int16), v.view(torch.int16),
                        out_ctx.view(torch.int16))
        assert N.nosa_sync(ctx) == N.NOSA_OK
        T = T0 + steps
        sel = np.zeros((U, cap), np.int32)
        sel_slot = np.zeros((U, cap), np.int32)
        n_sel = np.zeros(U, np.int32)
        N.nosa_export_state(ctx, 0, sel=sel, sel_slot=sel_slot, n_sel=n_sel)
    finally:
        N.nosa_destroy(ctx)

    # the oracle: exact softmax attention of each head over the tokens of the unit's selection
    Kh = O.bf16_bits_to_f64(_bits(Kall)).reshape(U, T, d)
    Vh = O.bf16_bits_to_f64(_bits(Vall)).reshape(U, T, d)
    Qh = O.bf16_bits_to_f64(_bits(q)).reshape(U, G, d)
    ref = np.stack([O.sparse_attention(Qh[u], Kh[u], Vh[u], [int(b) for b in sel[u, :n_sel[u]]], T,
                                       1 / math.sqrt(d)) for u in range(U)])

    # the context's block cache, rebuilt from the known K/V: slot s of unit u holds
    # block sel[u][i] (K then V, rows past the context zero)
    cache = torch.zeros((U, cap, 2, 64, d), dtype=torch.bfloat16, device="cuda")
    Ku = Kall.reshape(U, T, d)
    Vu = Vall.reshape(U, T, d)
    for u in range(U):
        for i in range(n_sel[u]):
            b, sl = int(sel[u, i]), int(sel_slot[u, i])
            e = min(64 * b + 64, T)
            cache[u, sl, 0, :e - 64 * b] = Ku[u, 64 * b:e]
            cache[u, sl, 1, :e - 64 * b] = Vu[u, 64 * b:e]
    sel_d = torch.from_numpy(sel).cuda()
    slot_d = torch.from_numpy(sel_slot).cuda()
    nsel_d = torch.from_numpy(n_sel).cuda()
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    qd = q.view(torch.int16)
    for _ in range(2):  # two calls in a row share the fixed scratch
        out = torch.full((B, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        N.nosa_attend_noalloc(qd, cache.view(torch.int16), sel_d, slot_d, nsel_d, U, G, cap, T,
                              out.view(torch.int16), err_out=err, stream=stream.cuda_stream)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = out.float().cpu().numpy().reshape(U, G, d)
        e = np.abs(got - ref)
        assert np.isfinite(got).all()
        assert e.max() <= 2e-2 and e.mean() <= 2e-3, (e.max(), e.mean())
        assert e.max() <= 2 ** -7 * np.abs(ref).max() + 1e-4, e.max()
        # the context's own attention over the same selection agrees too
        assert (out.float() - out_ctx.float()).abs().max().item() <= 2e-2

    # a selection count above the cache and a slot out of range are clamped and reported (bit 1)
    for bad in ("n_sel", "slot"):
        n2, s2 = nsel_d.clone(), slot_d.clone()
        if bad == "n_sel":
            n2[U - 1] = cap + 7
        else:
            s2[0, 0] = cap + 3
        out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
        N.nosa_attend_noalloc(qd, cache.view(torch.int16), sel_d, s2, n2, U, G, cap, T, out.view(torch.int16),
                              err_out=err, stream=stream.cuda_stream)
        torch.cuda.synchronize()
        assert int(err.item()) & 1, bad
    # without an error word the call still runs, and a clean call after a flagged one reports 0
    N.nosa_attend_noalloc(qd, cache.view(torch.int16), sel_d, slot_d, nsel_d, U, G, cap, T,
                          out.view(torch.int16), stream=stream.cuda_stream)
    N.nosa_attend_noalloc(qd, cache.view(torch.int16), sel_d, slot_d, nsel_d, U, G, cap, T,
                          out.view(torch.int16), err_out=err, stream=stream.cuda_stream)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # sizes beyond the fixed scratch are refused before anything is queued
    with pytest.raises(N.NosaError) as ex:
        N.nosa_attend_noalloc(qd, cache.view(torch.int16), sel_d, slot_d, nsel_d, 5000, G, cap, T,
                              out.view(torch.int16), stream=stream.cuda_stream)
    assert ex.value.status == N.NOSA_ERR_CAPACITY
