"""CPU oracle for the NOSA decode step (NOSA wiki page; NOSA-1B blog; NOSA explainer).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
module.  It shares no code with the CUDA path and imports nothing from it.

It restates, per (layer, batch, kv-head) unit, what one decode step of
NOSA computes, in float64 numpy, in the order the pages describe it:

  1. compressed keys  K~_i = bf16(mean of keys in window i)     (CompressK)
  2. eviction score   s^e_j = softplus(v_j W1) W2               (eq. 4)
  3. query score      s^q_i = sum_h softmax_i(q_h . K~_i / sqrt d)
  4. pooling          window mean, then max onto the 64-token block grid (eq. 5-6)
  5. selection        top-k_q by s^q; those set to +inf; fill k_e by s^e among
                      blocks never dropped before; add sink + window blocks
  6. set difference   blocks to fetch = selected blocks that hold no cache slot
  7. attention        exact softmax attention over the selected tokens (eq. 8)
  8. locality         gamma(t) = |D_t intersect S_{t-1}| / |D_t|     (Theorem 2)

Readings taken where the pages leave a step open:
  * kernel 32 / stride 16 for CompressK (the wiki table prints "32 / 16" with a
    note that SparDA and InfLLM-V2 give kernel 32, stride 16; the NOSA-1B blog
    gives kernel_size=32, stride 16).
  * GQA: each q head of the group scores the windows; the per-head softmax over
    all complete windows is summed over the group (SparDA summary, "lightweight
    design": the original selector aggregates the group's heads through a softmax).
  * a window counts towards a block when the two token ranges overlap.
  * the sink is block 0, the window is the last W/64 blocks (the last one
    partial); candidates are the blocks in between.  Ties: higher score first,
    then lower block index.  Selection is decided on float32 scores, the
    precision the kernels rank in.
  * "evicted" is sticky: a candidate left out of the dynamic set at any step is
    never again eligible for the query-agnostic part; the query-aware part may
    still recall it.  With fewer than k_e eligible blocks the query-agnostic part
    comes up short.
  * the block cache has at least as many slots as a selection has blocks (as many
    is the pages' cache: exactly the last selection).  A selected block without a
    slot is fetched (this includes a newly started tail block and, on the first
    step after a bulk context load, every selected block).  The new blocks, in
    ascending order, take the slots that hold no selected block, least recently
    selected first (an empty slot counts as never selected; ties to the lower
    slot), those slots in ascending order; blocks in the other slots stay cached
    for later steps.  With exactly as many slots as the selection, the slots taken
    are those whose block left the selection.
  * after a sparse prefill the cache holds exactly the prompt's last selection,
    its i-th block (ascending) in slot i (every block of it was just written from
    the prompt, so nothing earlier is worth keeping).
  * by default no DMA attention bias in the attention step (eq. 8 prints none);
    as an option (UnitOracle(dma_bias=True)) each token's eviction score s^e_j
    is added to its scaled logit q.k_j / sqrt(d), the additive bias of DMA that
    the eviction head comes from (wiki "How NOSA works").

Parity pins for every function live in tests/test_oracle.py.
"""
from __future__ import annotations

import math

import numpy as np


# ----------------------------------------------------------------------------- numerics
def bf16_round(x):
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits and float32's exponent range; below
    2^-126 its spacing is the subnormal step 2^-133.  Scaling by a power of
    two is exact, so rint (ties-to-even) at the right scale is the rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                      # |x| in [2^(e-1), 2^e)
    q = np.maximum(e - 8, -133)             # spacing of bf16 values near x
    return np.ldexp(np.rint(np.ldexp(x, -q)), q)


def bf16_bits_to_f64(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x):
    """bf16-valued float64 -> bit pattern (x must already be bf16-representable)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def softplus(x):
    """tau in the eviction head: log(1 + e^x), evaluated without overflow."""
    return np.logaddexp(0.0, x)


# ----------------------------------------------------------------------------- geometry
def num_windows(T, kernel=32, stride=16):
    """Complete compression windows over T tokens: window i covers [stride*i, stride*i + kernel)."""
    return 0 if T < kernel else (T - kernel) // stride + 1


def num_blocks(T, block=64):
    return -(-T // block)


def window_block_overlap(nb, nc, block=64, kernel=32, stride=16):
    """Boolean [nb][nc]: does window i's token range overlap block b's token range?"""
    b = np.arange(nb)[:, None]
    i = np.arange(nc)[None, :]
    return (stride * i < block * (b + 1)) & (stride * i + kernel > block * b)


def block_pool(win_scores, nb, block=64, kernel=32, stride=16):
    """Max over the windows that overlap each block; -inf for a block with none (eq. 5-6)."""
    win_scores = np.asarray(win_scores, dtype=np.float64)
    nc = len(win_scores)
    if nb == 0:
        return np.zeros(0)
    if nc == 0:
        return np.full(nb, -np.inf)
    m = window_block_overlap(nb, nc, block, kernel, stride)
    return np.where(m, win_scores[None, :], -np.inf).max(axis=1)


def partition(T, nw, sink=1, block=64):
    """Sink blocks, candidate blocks and window blocks for a context of T tokens."""
    nb = num_blocks(T, block)
    ns = min(sink, nb)
    ws = max(nb - nw, ns)
    return list(range(ns)), list(range(sink, ws)) if ws > sink else [], list(range(ws, nb))


# ----------------------------------------------------------------------------- method steps
def compress_keys(K, kernel=32, stride=16):
    """CompressK: K~_i = bf16(mean of the kernel keys of window i), mean taken exactly in float64."""
    K = np.asarray(K, dtype=np.float64)
    nc = num_windows(len(K), kernel, stride)
    out = np.empty((nc, K.shape[1]))
    for i in range(nc):
        out[i] = bf16_round(K[stride * i: stride * i + kernel].mean(axis=0))
    return out


def eviction_scores(V, W1, W2):
    """Eq. 4: s^e_j = softplus(v_j W1) W2, per token, ranked pre-exponential (ED-DMA)."""
    V = np.asarray(V, dtype=np.float64)
    return softplus(V @ np.asarray(W1, np.float64)) @ np.asarray(W2, np.float64)


def window_means(s_tok, kernel=32, stride=16):
    """Mean-pool of per-token scores over the compression windows (eq. 5)."""
    s_tok = np.asarray(s_tok, dtype=np.float64)
    nc = num_windows(len(s_tok), kernel, stride)
    return np.array([s_tok[stride * i: stride * i + kernel].mean() for i in range(nc)])


def query_scores(Qg, Kt, scale):
    """Query-aware window score: per-head softmax over all windows, summed over the GQA group."""
    Qg = np.asarray(Qg, dtype=np.float64)
    Kt = np.asarray(Kt, dtype=np.float64)
    if len(Kt) == 0:
        return np.zeros(0)
    z = (Qg @ Kt.T) * scale                         # [G][nc]
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p = p / p.sum(axis=1, keepdims=True)
    return p.sum(axis=0)


def top_k(scores32, eligible, k):
    """The k best eligible blocks by float32 score, ties to the lower block index; ascending."""
    ranked = sorted(eligible, key=lambda b: (-float(scores32[b]), b))
    return sorted(ranked[:max(k, 0)])


def select_query_aware(sq_blk, candidates, k_q):
    """Q: the k_q candidates with the highest pooled query-aware score."""
    return top_k(np.asarray(sq_blk, np.float64).astype(np.float32), candidates, k_q)


def select_query_agnostic(se_blk, candidates, Q, evicted, k_e):
    """E: after Q is fixed (its scores set to +inf), fill k_e blocks by the pooled
    eviction score, only from candidates outside Q that were never dropped before."""
    taken = set(Q)
    eligible = [b for b in candidates if b not in taken and b not in evicted]
    return top_k(np.asarray(se_blk, np.float64).astype(np.float32), eligible, k_e)


def assign_slots(S, slot_blk, last_used=None, T=0):
    """Set difference of the selection S, made at context length T, against the block cache.

    slot_blk: the block in each slot (-1: empty); last_used: the context length of the last
    selection that held each slot's block (-1: never; None: all -1).  Selected blocks with no
    slot are new.  In ascending order they take the slots that hold no selected block, least
    recently selected first (ties to the lower slot), those slots in ascending order; the
    other slots keep their blocks.  Every slot holding a block of S is marked selected at T.
    Returns the fetch list [(block, slot)], the new slot map, the new marks and the slot of
    every block of S.
    """
    keep = set(S)
    n = len(slot_blk)
    lu = [-1] * n if last_used is None else list(last_used)
    resident = {b for b in slot_blk if b >= 0}
    new_blocks = [b for b in S if b not in resident]
    open_slots = [s for s in range(n) if not (slot_blk[s] >= 0 and slot_blk[s] in keep)]
    if len(new_blocks) > len(open_slots):
        raise ValueError("block cache too small for the selection")
    taken = sorted(sorted(open_slots, key=lambda s: (lu[s], s))[:len(new_blocks)])
    new_map = list(slot_blk)
    fetch = list(zip(new_blocks, taken))
    for b, s in fetch:
        new_map[s] = b
    where = {b: s for s, b in enumerate(new_map) if b >= 0}
    for b in S:
        lu[where[b]] = T
    return fetch, new_map, lu, [where[b] for b in S]


def sparse_attention(Qg, K, V, S, T, scale, block=64, bias=None):
    """Eq. 8: softmax attention of each head over the tokens of the selected blocks.

    bias (one value per token, natural-log units) is the DMA-style additive attention
    bias (wiki "How NOSA works": the eviction head is adapted from DMA, which adds its
    per-token score to the attention logits): token j's logit is q.k_j * scale + bias[j].
    """
    idx = np.concatenate([np.arange(block * b, min(block * (b + 1), T)) for b in S]) if S else np.zeros(0, int)
    Qg = np.asarray(Qg, np.float64)
    Ks = np.asarray(K, np.float64)[idx]
    Vs = np.asarray(V, np.float64)[idx]
    z = (Qg @ Ks.T) * scale
    if bias is not None:
        z = z + np.asarray(bias, np.float64)[idx][None, :]
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ Vs


def locality(D, S_prev):
    """gamma(t) = |D_t intersect S_{t-1}| / |D_t| (Theorem 2 bounds it below by k_e/k)."""
    if not D:
        return 1.0
    return len(set(D) & set(S_prev)) / len(D)


# ----------------------------------------------------------------------------- one unit
class UnitOracle:
    """State and steps of one (layer, batch, kv-head) unit, computed from its raw inputs."""

    def __init__(self, *, head_dim=128, block=64, kernel=32, stride=16, k_q, k_e,
                 sink_blocks=1, window_tokens, max_context, W1, W2, scale=None, dma_bias=False,
                 cache_slots=None):
        self.d, self.block, self.kernel, self.stride = head_dim, block, kernel, stride
        self.k_q, self.k_e, self.sink = k_q, k_e, sink_blocks
        self.nw = window_tokens // block
        self.cap = sink_blocks + self.nw + k_q + k_e
        self.cslots = self.cap if not cache_slots else cache_slots
        if self.cslots < self.cap:
            raise ValueError("the block cache must hold a whole selection")
        self.scale = 1.0 / math.sqrt(head_dim) if not scale else scale
        self.dma_bias = dma_bias  # attention logits get each token's eviction score added
        self.W1 = np.asarray(W1, np.float64)
        self.W2 = np.asarray(W2, np.float64)
        self.K = np.zeros((max_context, head_dim))
        self.V = np.zeros((max_context, head_dim))
        self.se_tok = np.zeros(max_context)
        self.Kt = np.zeros((num_windows(max_context, kernel, stride), head_dim))
        self.T = 0
        self.evicted: set[int] = set()
        self.slot_blk = [-1] * self.cslots
        self.last_used = [-1] * self.cslots
        self.S_prev: list[int] | None = None
        self.steps = 0

    # -- a1: append (token values are bf16 bit patterns)
    def append(self, k_bits, v_bits):
        k = bf16_bits_to_f64(k_bits).reshape(-1, self.d)
        v = bf16_bits_to_f64(v_bits).reshape(-1, self.d)
        n = len(k)
        t0 = self.T
        self.K[t0:t0 + n] = k
        self.V[t0:t0 + n] = v
        self.se_tok[t0:t0 + n] = eviction_scores(v, self.W1, self.W2)
        nc0 = num_windows(t0, self.kernel, self.stride)
        self.T = t0 + n
        nc1 = num_windows(self.T, self.kernel, self.stride)
        for i in range(nc0, nc1):           # windows completed by these tokens
            self.Kt[i] = compress_keys(self.K[self.stride * i: self.stride * i + self.kernel],
                                       self.kernel, self.stride)[0]

    @property
    def nc(self):
        return num_windows(self.T, self.kernel, self.stride)

    @property
    def nb(self):
        return num_blocks(self.T, self.block)

    def compressed_keys(self):
        return self.Kt[:self.nc]

    # -- a2: pooled block scores
    def scores(self, q_bits):
        """Pooled query-aware and query-agnostic block scores, float64 [nb] each."""
        Qg = bf16_bits_to_f64(q_bits).reshape(-1, self.d)
        sq_win = query_scores(Qg, self.compressed_keys(), self.scale)
        se_win = window_means(self.se_tok[:self.T], self.kernel, self.stride)
        return (block_pool(sq_win, self.nb, self.block, self.kernel, self.stride),
                block_pool(se_win, self.nb, self.block, self.kernel, self.stride))

    def partition(self):
        return partition(self.T, self.nw, self.sink, self.block)

    # -- a3: selection (pure: no state change)
    def select(self, sq_blk, se_blk):
        _, C, _ = self.partition()
        Q = select_query_aware(sq_blk, C, self.k_q)
        E = select_query_agnostic(se_blk, C, Q, self.evicted, self.k_e)
        return Q, E

    # -- a3/a4: commit a selection: eviction update, set difference, slots (for a context of T tokens,
    # by default the current one)
    def commit(self, Q, E, T=None):
        T = self.T if T is None else T
        sink, C, win = partition(T, self.nw, self.sink, self.block)
        D = sorted(set(Q) | set(E))
        S = sorted(set(sink) | set(D) | set(win))
        Dset = set(D)
        self.evicted |= {b for b in C if b not in Dset}
        fetch, self.slot_blk, self.last_used, slot_of = assign_slots(S, self.slot_blk, self.last_used, T)
        gamma = None if self.S_prev is None else locality(D, self.S_prev)
        self.S_prev = S
        self.steps += 1
        return dict(S=S, D=D, fetch=fetch, slot_of=slot_of, gamma=gamma,
                    short=max(0, self.k_e - len(E)))

    # -- the cache after a sparse prefill: the last selection, block i of it in slot i
    def settle_cache(self):
        S = self.S_prev or []
        self.slot_blk = list(S) + [-1] * (self.cslots - len(S))
        self.last_used = [self.T] * len(S) + [-1] * (self.cslots - len(S))

    # -- a6: attention over the selection
    def attend(self, q_bits, S):
        Qg = bf16_bits_to_f64(q_bits).reshape(-1, self.d)
        bias = self.se_tok[:self.T] if self.dma_bias else None
        return sparse_attention(Qg, self.K[:self.T], self.V[:self.T], S, self.T, self.scale, self.block, bias)

    # -- SparDA-style selection one layer ahead (SparDA summary: a forecast vector of layer l
    # picks layer l+1's blocks before layer l+1 runs; one forecast head per kv head, no softmax
    # aggregation over a group; sink and local blocks by position).  It is made before the token
    # it serves is appended: scores over the windows complete now, blocks and candidates of T+1.
    def forecast_scores(self, f_bits):
        F = bf16_bits_to_f64(f_bits).reshape(1, self.d)
        sq_win = query_scores(F, self.compressed_keys(), self.scale)
        se_win = window_means(self.se_tok[:self.T], self.kernel, self.stride)
        nb1 = num_blocks(self.T + 1, self.block)
        return (block_pool(sq_win, nb1, self.block, self.kernel, self.stride),
                block_pool(se_win, nb1, self.block, self.kernel, self.stride))

    def forecast_step(self, f_bits, q_bits, k_bits, v_bits):
        """Forecast selection for T+1, diff and slots; then append the token and attend with q."""
        sq, se = self.forecast_scores(f_bits)
        _, C, _ = partition(self.T + 1, self.nw, self.sink, self.block)
        Q = select_query_aware(sq, C, self.k_q)
        E = select_query_agnostic(se, C, Q, self.evicted, self.k_e)
        r = self.commit(Q, E, T=self.T + 1)
        self.append(k_bits, v_bits)
        r.update(Q=Q, E=E, sq_blk=sq, se_blk=se, out=self.attend(q_bits, r["S"]))
        return r

    def step(self, q_bits, k_bits, v_bits):
        """One decode step: append, score, select, diff, attend."""
        self.append(k_bits, v_bits)
        sq, se = self.scores(q_bits)
        Q, E = self.select(sq, se)
        r = self.commit(Q, E)
        r.update(Q=Q, E=E, sq_blk=sq, se_blk=se, out=self.attend(q_bits, r["S"]))
        return r
