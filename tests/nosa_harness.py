"""GPU-vs-oracle parity driver shared by the GPU tests, smoke() and the bench's
CPU-baseline leg.  The GPU side runs only through the C ABI (ctypes binding);
the oracle side runs oracle/nosa_oracle.py on the same seeded inputs.

Acceptance (the NOSA decode-path targets):
  * block selections, fetch lists, slots and eviction bitmaps bit-exact; a
    differing pick is accepted only when the oracle's float32 scores of every
    differing block lie within 1e-5 relative of the oracle's k-th score; each
    such near tie is logged and the oracle adopts the GPU's pick for that unit,
    so the sticky eviction state stays comparable;
  * compressed keys bit-exact;
  * pooled scores within 1e-4 relative, the denominator being
    max(|oracle|, 1e-3 * rms over the unit's blocks);
  * attention outputs within max-abs 2e-2 and mean-abs 2e-3 (bf16 inputs,
    fp32 accumulation), and, tighter, max-abs within 2^-7 of the output's
    largest magnitude plus 1e-4.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from oracle import nosa_oracle as O
from synth import inputs as syn

TIE_REL = 1e-5
SCORE_REL = 1e-4
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3


@dataclass
class ParityLog:
    steps: int = 0
    unit_steps: int = 0
    near_ties: list = field(default_factory=list)
    max_out_abs: float = 0.0
    max_out_mean_abs: float = 0.0
    max_score_rel: float = 0.0
    gammas: list = field(default_factory=list)
    fetched: int = 0


def _near_tie_ok(scores32, got, want, pool, k):
    """Every block in got^want has an oracle float32 score within TIE_REL of the k-th best in pool."""
    if not pool or k <= 0:
        return got == want
    ranked = sorted(pool, key=lambda b: (-float(scores32[b]), b))
    kth = float(scores32[ranked[min(k, len(ranked)) - 1]])
    tol = TIE_REL * max(abs(kth), 1e-30)
    return all(abs(float(scores32[b]) - kth) <= tol for b in set(got) ^ set(want))


def rel_err(gpu, ref):
    ref = np.asarray(ref, np.float64)
    gpu = np.asarray(gpu, np.float64)
    fin = np.isfinite(ref)
    if not np.array_equal(fin, np.isfinite(gpu)):
        return math.inf
    if not fin.any():
        return 0.0
    r, g = ref[fin], gpu[fin]
    rms = math.sqrt(float(np.mean(r * r))) if r.size else 0.0
    den = np.maximum(np.abs(r), 1e-3 * rms + 1e-30)
    return float(np.max(np.abs(g - r) / den))


class Parity:
    """Drives one context through the C ABI and checks sampled units against the oracle."""

    def __init__(self, wl: syn.Workload, sample_units=None, layers=None, gather_ctas=0, device="cuda",
                 check_scores=True, flags=0, **sizing):
        import torch
        from offloadable_block_sparse_gb300 import nosa as N
        self.torch, self.N = torch, N
        self.wl = wl
        self.L = wl.layers if layers is None else layers
        self.U = wl.batch * wl.kv_heads
        self.G = wl.group
        self.d = wl.head_dim
        self.dev = device
        self.check_scores = check_scores
        self.flags = flags
        self.cfg = N.make_config(num_layers=self.L, batch=wl.batch, num_q_heads=wl.q_heads,
                                 num_kv_heads=wl.kv_heads, k_q=wl.k_q, k_e=wl.k_e,
                                 window_tokens=wl.window_tokens, max_context=wl.max_context,
                                 sink_blocks=wl.sink_blocks, evict_hidden=wl.evict_hidden,
                                 gather_ctas=gather_ctas, flags=flags, **sizing)
        self.sizes = N.nosa_query_sizes(self.cfg)
        self.stream = torch.cuda.current_stream()
        self.ctx = N.nosa_create(self.cfg, self.stream.cuda_stream)
        if sample_units is None:
            sample_units = [(l, b, g) for l in range(self.L) for b in range(wl.batch) for g in range(wl.kv_heads)]
        self.samples = list(sample_units)
        self.log = ParityLog()
        self.oracles = {}
        self.inputs = {}
        self.t = 0

    # ------------------------------------------------------------------ setup
    def load_context(self, filler_seed=1234):
        """Bulk-append T_0 tokens to every layer; sampled units get the seeded synth values."""
        torch, N, wl = self.torch, self.N, self.wl
        T0, d = wl.context, self.d
        for l in range(self.L):
            W1 = np.zeros((wl.kv_heads, d, wl.evict_hidden), np.float32)
            W2 = np.zeros((wl.kv_heads, wl.evict_hidden), np.float32)
            for g in range(wl.kv_heads):
                W1[g], W2[g] = syn.eviction_head(wl.seed, l, g, d, wl.evict_hidden)
            N.nosa_set_eviction_head(self.ctx, l, W1, W2)
            gen = torch.Generator(device=self.dev).manual_seed(filler_seed + l)
            K = torch.randn((wl.batch, wl.kv_heads, T0, d), generator=gen, device=self.dev).to(torch.bfloat16)
            V = torch.randn((wl.batch, wl.kv_heads, T0, d), generator=gen, device=self.dev).to(torch.bfloat16)
            for (sl, b, g) in self.samples:
                if sl != l:
                    continue
                x = wl.unit_inputs(l, b, g)
                self.inputs[(l, b, g)] = x
                K[b, g] = torch.from_numpy(x["K"][:T0].view(np.int16)).view(torch.bfloat16).to(self.dev)
                V[b, g] = torch.from_numpy(x["V"][:T0].view(np.int16)).view(torch.bfloat16).to(self.dev)
                o = O.UnitOracle(head_dim=d, k_q=wl.k_q, k_e=wl.k_e, sink_blocks=wl.sink_blocks,
                                 window_tokens=wl.window_tokens, max_context=wl.max_context,
                                 W1=W1[g], W2=W2[g], dma_bias=bool(self.flags & N.NOSA_F_DMA_BIAS),
                                 cache_slots=self.sizes.cache_slots)
                o.append(x["K"][:T0], x["V"][:T0])
                self.oracles[(l, b, g)] = o
            N.nosa_append_kv(self.ctx, l, K.view(torch.int16), V.view(torch.int16), T0)
            del K, V
        self._filler = torch.Generator(device=self.dev).manual_seed(filler_seed + 10000)

    # ------------------------------------------------------------------ one decode step
    def step_inputs(self, l):
        """q [B][Hq][d], k/v [B][Hkv][d] on the device for decode step self.t+1 of layer l."""
        torch, wl = self.torch, self.wl
        gen = self._filler
        q = torch.randn((wl.batch, wl.q_heads, self.d), generator=gen, device=self.dev)
        q = (q / q.norm(dim=-1, keepdim=True) * math.sqrt(self.d)).to(torch.bfloat16)
        k = torch.randn((wl.batch, wl.kv_heads, self.d), generator=gen, device=self.dev).to(torch.bfloat16)
        v = torch.randn((wl.batch, wl.kv_heads, self.d), generator=gen, device=self.dev).to(torch.bfloat16)
        pos = wl.context + self.t
        for (sl, b, g) in self.samples:
            if sl != l:
                continue
            x = self.inputs[(l, b, g)]
            q[b, g * self.G:(g + 1) * self.G] = torch.from_numpy(x["Q"][self.t].view(np.int16)).view(
                torch.bfloat16).to(self.dev)
            k[b, g] = torch.from_numpy(x["K"][pos].view(np.int16)).view(torch.bfloat16).to(self.dev)
            v[b, g] = torch.from_numpy(x["V"][pos].view(np.int16)).view(torch.bfloat16).to(self.dev)
        return q, k, v

    def forecast_inputs(self, l, t):
        """f [B][Hkv][d] on the device: the forecast vectors for the token of decode step t+1 of layer l."""
        torch, wl = self.torch, self.wl
        f = torch.randn((wl.batch, wl.kv_heads, self.d), generator=self._filler, device=self.dev)
        f = (f / f.norm(dim=-1, keepdim=True) * math.sqrt(self.d)).to(torch.bfloat16)
        for (sl, b, g) in self.samples:
            if sl == l:
                f[b, g] = torch.from_numpy(self.inputs[(l, b, g)]["F"][t].view(np.int16)).view(
                    torch.bfloat16).to(self.dev)
        return f

    def run_forecast_step(self, check=True, separate_fetch=True):
        """One decode step with forecast selections made by separate calls, every layer checked."""
        torch, N = self.torch, self.N
        for l in range(self.L):
            q, k, v = self.step_inputs(l)
            f = self.forecast_inputs(l, self.t)
            out = torch.empty_like(q)
            N.nosa_forecast_select(self.ctx, l, f.view(torch.int16))
            if separate_fetch:
                N.nosa_fetch(self.ctx, l)
            N.nosa_append_kv(self.ctx, l, k.view(torch.int16), v.view(torch.int16), 1)
            N.nosa_attend(self.ctx, l, q.view(torch.int16), out.view(torch.int16))
            if check and any(sl == l for (sl, _, _) in self.samples):
                st = N.nosa_sync(self.ctx)
                assert st == 0, f"device error {N.STATUS_NAMES[st]}"
                self._check_layer(l, q, out, f)
        self.t += 1
        self.log.steps += 1

    def run_forecast_pipeline(self, steps):
        """Steps through nosa_step_forecast: each layer's call starts the next layer's forecast and
        prefetch on the context's prefetch stream (the last layer forecasts layer 0 of the next
        step).  Outputs of the sampled units are checked against the oracle's forecast step."""
        torch, N = self.torch, self.N
        assert self.L >= 2
        fs = [[self.forecast_inputs(l, t) for l in range(self.L)] for t in range(steps)]
        N.nosa_forecast_select(self.ctx, 0, fs[0][0].view(torch.int16))
        for t in range(steps):
            done = []
            for l in range(self.L):
                q, k, v = self.step_inputs(l)
                out = torch.empty_like(q)
                if l + 1 < self.L:
                    fn, nxt = fs[t][l + 1], l + 1
                else:
                    fn, nxt = (fs[t + 1][0], 0) if t + 1 < steps else (None, 0)
                N.nosa_step_forecast(self.ctx, l, q.view(torch.int16), k.view(torch.int16), v.view(torch.int16),
                                     out.view(torch.int16), None if fn is None else fn.view(torch.int16), nxt)
                done.append((l, q, k, v, out))
            N.nosa_forecast_join(self.ctx)
            st = N.nosa_sync(self.ctx)
            assert st == 0, f"device error {N.STATUS_NAMES[st]}"
            for (l, q, k, v, out) in done:
                f_h = fs[t][l].view(torch.int16).cpu().numpy().view(np.uint16)
                q_h = q.view(torch.int16).cpu().numpy().view(np.uint16)
                out_h = out.float().cpu().numpy()
                for (sl, b, g) in self.samples:
                    if sl != l:
                        continue
                    o, x = self.oracles[(l, b, g)], self.inputs[(l, b, g)]
                    pos = self.wl.context + self.t
                    r = o.forecast_step(f_h[b, g], q_h[b, g * self.G:(g + 1) * self.G], x["K"][pos:pos + 1],
                                        x["V"][pos:pos + 1])
                    err = np.abs(out_h[b, g * self.G:(g + 1) * self.G] - r["out"])
                    self.log.max_out_abs = max(self.log.max_out_abs, float(err.max()))
                    self.log.max_out_mean_abs = max(self.log.max_out_mean_abs, float(err.mean()))
                    assert err.max() <= OUT_MAX_ABS and err.mean() <= OUT_MEAN_ABS, f"output error {err.max():.3e}"
                    if r["gamma"] is not None:
                        self.log.gammas.append(r["gamma"])
                    self.log.unit_steps += 1
            self.t += 1
            self.log.steps += 1

    def run_step(self, check=True, split_calls=False, separate_fetch=True):
        torch, N = self.torch, self.N
        for l in range(self.L):
            q, k, v = self.step_inputs(l)
            out = torch.empty_like(q)
            if split_calls:
                N.nosa_append_kv(self.ctx, l, k.view(torch.int16), v.view(torch.int16), 1)
                N.nosa_select(self.ctx, l, q.view(torch.int16))
                if separate_fetch:
                    N.nosa_fetch(self.ctx, l)
                N.nosa_attend(self.ctx, l, q.view(torch.int16), out.view(torch.int16))
            else:
                N.nosa_step(self.ctx, l, q.view(torch.int16), k.view(torch.int16), v.view(torch.int16),
                            out.view(torch.int16))
            if check and any(sl == l for (sl, _, _) in self.samples):
                st = N.nosa_sync(self.ctx)
                assert st == 0, f"device error {N.STATUS_NAMES[st]}"
                self._check_layer(l, q, out)
        self.t += 1
        self.log.steps += 1

    # ------------------------------------------------------------------ comparison
    def _export(self, l):
        U, cap, cs, sz = self.U, self.sizes.select_slots, self.sizes.cache_slots, self.sizes
        nc = max(sz.max_windows, 1)
        st = dict(sel=np.zeros((U, cap), np.int32), sel_kind=np.zeros((U, cap), np.int32),
                  sel_slot=np.zeros((U, cap), np.int32), n_sel=np.zeros(U, np.int32),
                  fetch=np.zeros((U, cap, 2), np.int32), n_fetch=np.zeros(U, np.int32),
                  slot_blk=np.zeros((U, cs), np.int32), last_used=np.zeros((U, cs), np.int32),
                  evicted=np.zeros((U, sz.evict_words), np.uint32),
                  kt=np.zeros((U, nc, self.d), np.uint16), se_blk=np.zeros((U, sz.max_blocks), np.float32),
                  gamma=np.zeros((U, 2), np.int32))
        self.N.nosa_export_state(self.ctx, l, **st)
        sq = np.zeros((U, sz.max_blocks), np.float32)
        self.N.nosa_debug_scores(self.ctx, l, sq, None)
        st["sq_blk"] = sq
        return st

    def _check_layer(self, l, q, out, f=None):
        """Compares layer l's selection, state and output with the oracle.  With f (the forecast
        vectors of this step) the oracle selects before the append, as the forecast path does."""
        wl = self.wl
        st = self._export(l)
        out_h = out.float().cpu().numpy()
        q_h = q.view(self.torch.int16).cpu().numpy().view(np.uint16)
        f_h = None if f is None else f.view(self.torch.int16).cpu().numpy().view(np.uint16)
        for (sl, b, g) in self.samples:
            if sl != l:
                continue
            u = b * wl.kv_heads + g
            o = self.oracles[(l, b, g)]
            x = self.inputs[(l, b, g)]
            pos = wl.context + self.t
            qb = q_h[b, g * self.G:(g + 1) * self.G]
            assert np.array_equal(qb, x["Q"][self.t])
            if f is None:
                o.append(x["K"][pos:pos + 1], x["V"][pos:pos + 1])
                sq, se = o.scores(qb)
                T_sel = o.T
            else:
                fb = f_h[b, g]
                assert np.array_equal(fb, x["F"][self.t])
                sq, se = o.forecast_scores(fb)
                T_sel = o.T + 1
            _, C, _ = O.partition(T_sel, o.nw, o.sink, o.block)
            nb = O.num_blocks(T_sel, o.block)
            if self.check_scores:
                e1 = rel_err(st["sq_blk"][u, :nb], sq)
                # the forecast path appends after it selects: the token's window may move the pooled
                # s^e of window blocks, so only the candidates' scores are compared there
                cmp = slice(0, nb) if f is None else C
                e2 = rel_err(st["se_blk"][u, :nb][cmp], np.asarray(se)[cmp]) if (f is None or C) else 0.0
                self.log.max_score_rel = max(self.log.max_score_rel, e1, e2)
                assert e1 <= SCORE_REL and e2 <= SCORE_REL, f"pooled scores {e1:.2e} {e2:.2e} unit {(l, b, g)}"
            n = st["n_sel"][u]
            S_gpu = list(st["sel"][u, :n])
            kinds = st["sel_kind"][u, :n]
            Q_gpu = sorted(int(bb) for bb, kk in zip(S_gpu, kinds) if kk == 2)
            E_gpu = sorted(int(bb) for bb, kk in zip(S_gpu, kinds) if kk == 3)
            Q = O.select_query_aware(sq, C, wl.k_q)
            if Q != Q_gpu:
                ok = _near_tie_ok(np.asarray(sq).astype(np.float32), Q_gpu, Q, C, wl.k_q)
                assert ok, f"query-aware pick differs beyond a near tie: unit {(l, b, g)} step {self.t}: {Q} vs {Q_gpu}"
                self.log.near_ties.append(("q", (l, b, g), self.t, sorted(set(Q) ^ set(Q_gpu))))
                Q = Q_gpu
            E = O.select_query_agnostic(se, C, Q, o.evicted, wl.k_e)
            if E != E_gpu:
                pool = [bb for bb in C if bb not in set(Q) and bb not in o.evicted]
                ok = _near_tie_ok(np.asarray(se).astype(np.float32), E_gpu, E, pool, wl.k_e)
                assert ok, f"query-agnostic pick differs beyond a near tie: unit {(l, b, g)} step {self.t}"
                self.log.near_ties.append(("e", (l, b, g), self.t, sorted(set(E) ^ set(E_gpu))))
                E = E_gpu
            r = o.commit(Q, E, T=T_sel)
            if f is not None:
                o.append(x["K"][pos:pos + 1], x["V"][pos:pos + 1])
            nb, nc = o.nb, o.nc
            # compressed keys after the step's append: bit-exact
            kt_or = O.f64_to_bf16_bits(o.compressed_keys())
            assert np.array_equal(st["kt"][u, :nc], kt_or), f"K~ mismatch unit {(l, b, g)} step {self.t}"
            assert S_gpu == r["S"], f"selection mismatch unit {(l, b, g)} step {self.t}"
            assert list(st["sel_slot"][u, :n]) == r["slot_of"], "slot mismatch"
            nf = st["n_fetch"][u]
            assert [tuple(x) for x in st["fetch"][u, :nf]] == [tuple(x) for x in r["fetch"]], "fetch list mismatch"
            assert list(st["slot_blk"][u]) == o.slot_blk, "slot map mismatch"
            assert list(st["last_used"][u]) == o.last_used, "slot recency mismatch"
            ev = st["evicted"][u]
            ev_gpu = {bb for bb in range(nb) if (ev[bb >> 5] >> (bb & 31)) & 1}
            assert ev_gpu == o.evicted, "eviction bitmap mismatch"
            num, den = st["gamma"][u]
            assert den == len(r["D"])
            if r["gamma"] is not None and den > 0:   # gamma is undefined for an empty dynamic set
                assert abs(num / den - r["gamma"]) < 1e-12
                self.log.gammas.append(r["gamma"])
            self.log.fetched += len(r["fetch"])
            ref = o.attend(qb, r["S"])
            got = out_h[b, g * self.G:(g + 1) * self.G]
            err = np.abs(got - ref)
            self.log.max_out_abs = max(self.log.max_out_abs, float(err.max()))
            self.log.max_out_mean_abs = max(self.log.max_out_mean_abs, float(err.mean()))
            where = f"unit {(l, b, g)} step {self.t} T {o.T} max|ref| {np.abs(ref).max():.3e}"
            assert err.max() <= OUT_MAX_ABS and err.mean() <= OUT_MEAN_ABS, f"output error {err.max():.3e} {where}"
            assert err.max() <= 2 ** -7 * np.abs(ref).max() + 1e-4, f"output error {err.max():.3e} (tight) {where}"
            self.log.unit_steps += 1

    def close(self):
        if self.ctx:
            self.N.nosa_destroy(self.ctx)
            self.ctx = None
