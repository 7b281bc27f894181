"""Pins for the CPU oracle: each check ties a function of oracle/nosa_oracle.py to
something other than itself -- hand-computed values from the pages' rules, closed
forms, invariants (Theorem 2), brute force on tiny inputs, or a library routine
(torch's bf16 conversion and scaled-dot-product attention) in a special case."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import nosa_oracle as O
from synth import inputs as syn

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load_rows(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# ----------------------------------------------------------------------------- bf16
def test_bf16_round_hand_values():
    # ulp of bf16 at 1.0 is 2^-7; halfway cases go to the even mantissa
    cases = {1 + 2 ** -8: 1.0, 1 + 3 * 2 ** -8: 1 + 2 ** -6, 1 + 2 ** -9: 1.0,
             -(1 + 2 ** -8): -1.0, 1 + 2 ** -8 + 2 ** -20: 1 + 2 ** -7,
             3 * 2 ** -135: 2 ** -133, 0.0: 0.0, 255.5: 256.0, 254.5: 254.0}
    for x, want in cases.items():
        assert O.bf16_round(x) == want, (x, O.bf16_round(x), want)


def test_bf16_round_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_round(x.astype(np.float64)), want)


# ----------------------------------------------------------------------------- CompressK
def test_compress_keys_ramp_fixture():
    want = [float(v) for v in _load_rows("compress_ramp.txt")[0].split()]
    K = np.repeat(np.arange(96, dtype=np.float64)[:, None], 128, axis=1)
    Kt = O.compress_keys(K)
    assert Kt.shape == (5, 128)
    assert np.array_equal(Kt[:, 0], want) and np.all(Kt == Kt[:, :1])
    # the eviction score is mean-pooled over the same windows (eq. 5)
    assert np.array_equal(O.window_means(np.arange(96, dtype=np.float64)), want)


def test_compress_keys_rounds_exact_mean_to_even():
    # 31 ones and one 1.125: mean 1 + 2^-8, halfway -> 1.0 ; with 1.375: 1 + 3*2^-8 -> 1 + 2^-6
    for extra, want in [(1.125, 1.0), (1.375, 1 + 2 ** -6), (1.0078125, 1.0)]:
        K = np.ones((32, 4))
        K[7] = extra
        assert O.compress_keys(K)[0, 0] == want


def test_compressed_keys_are_one_sixteenth_of_K():
    c = json.load(open(os.path.join(GOLD, "page_constants.json")))
    for T in (4096, 16384, 65536):
        assert O.num_windows(T) == (T - 32) // 16 + 1
        assert abs(O.num_windows(T) / T - c["compressed_key_fraction"]) < 32 / T
    assert O.num_windows(31) == 0 and O.num_windows(32) == 1 and O.num_windows(47) == 1
    assert O.num_windows(48) == 2


# ----------------------------------------------------------------------------- eviction head
def test_eviction_score_closed_forms():
    d, h = 8, 6
    rng = np.random.default_rng(2)
    W1 = rng.standard_normal((d, h))
    W2 = rng.standard_normal(h)
    # one-hot v picks one row of W1
    for c in range(d):
        v = np.zeros((1, d)); v[0, c] = 1.0
        want = sum(W2[m] * math.log1p(math.exp(W1[c, m])) for m in range(h))
        assert abs(O.eviction_scores(v, W1, W2)[0] - want) < 1e-12
    # softplus(0) = ln 2
    assert abs(O.eviction_scores(np.ones((1, d)), np.zeros((d, h)), W2)[0] - math.log(2) * W2.sum()) < 1e-12


def test_eviction_score_hand_case_catches_transpose():
    W1 = np.array([[1.0, -1.0], [0.0, 2.0]])
    W2 = np.array([1.0, 0.5])
    # v W1 = [1, 1]; softplus(1) = ln(1 + e) = 1.3132616875182228; times (1 + 0.5)
    assert abs(O.eviction_scores(np.array([[1.0, 1.0]]), W1, W2)[0] - 1.9698925312773342) < 1e-14
    # large arguments do not overflow: softplus(x) -> x
    assert abs(O.softplus(800.0) - 800.0) < 1e-12 and O.softplus(-800.0) >= 0.0


# ----------------------------------------------------------------------------- pooling
def test_window_block_overlap_fixture():
    m = O.window_block_overlap(16, O.num_windows(1024))
    for row in _load_rows("pool_windows.txt"):
        b, ws = row.split(":")
        assert list(np.nonzero(m[int(b)])[0]) == [int(w) for w in ws.split()]
    # closed form 4b-1 .. 4b+3 for every interior block
    for b in range(1, 15):
        assert list(np.nonzero(m[b])[0]) == list(range(4 * b - 1, 4 * b + 4))


def test_block_pool_is_max_over_overlapping_windows():
    s = np.arange(63, dtype=np.float64)[::-1] * 0.5  # decreasing: max is the first window
    pooled = O.block_pool(s, 16)
    assert pooled[0] == s[0] and pooled[1] == s[3] and pooled[5] == s[19] and pooled[15] == s[59]
    # a block past the last complete window pools nothing
    assert O.block_pool(np.array([1.0]), 2)[1] == -np.inf


# ----------------------------------------------------------------------------- query score
def test_query_scores_group_softmax_invariants():
    rng = np.random.default_rng(3)
    Kt = rng.standard_normal((40, 16))
    Q = rng.standard_normal((4, 16))
    s = O.query_scores(Q, Kt, 0.25)
    assert abs(s.sum() - 4.0) < 1e-12          # each head's softmax sums to one
    assert np.all(s > 0)
    # G = 1: the softmax is monotone, so the ranking is the ranking of raw dot products
    s1 = O.query_scores(Q[:1], Kt, 0.25)
    assert np.array_equal(np.argsort(-s1, kind="stable"), np.argsort(-(Kt @ Q[0]), kind="stable"))


def test_query_scores_hand_case_two_heads_three_windows():
    # d = 4, so the temperature is 1/sqrt(4) = 1/2.  Windows K~ = 2 e0, 2 e1, 0; heads q = e0, e1.
    # Logits z = (q . K~) / 2: head 0 -> (1, 0, 0), head 1 -> (0, 1, 0).  Each head's softmax runs
    # over the windows; the group score is the sum over the heads:
    #   s = ((e + 1) / (e + 2), (e + 1) / (e + 2), 2 / (e + 2)).
    # A temperature of 1/d, a softmax over the heads instead of the windows, or a mean over the
    # heads instead of the sum gives other numbers.
    e = math.e
    Kt = np.array([[2.0, 0, 0, 0], [0, 2.0, 0, 0], [0, 0, 0, 0]])
    Q = np.array([[1.0, 0, 0, 0], [0, 1.0, 0, 0]])
    want = np.array([(e + 1) / (e + 2), (e + 1) / (e + 2), 2 / (e + 2)])
    assert np.max(np.abs(O.query_scores(Q, Kt, 1 / math.sqrt(4)) - want)) < 1e-15


def test_unit_scores_use_inverse_sqrt_d_temperature_hand_case():
    # One unit with head_dim 4 and 80 tokens: four complete windows, two blocks.  Keys come in
    # groups of 16 tokens g0..g4 = 2e0, 2e0, 2e1, 2e1, 0, so K~_i = (g_i + g_{i+1}) / 2 =
    # 2e0, e0 + e1, 2e1, e1.  Heads q0 = 2e0, q1 = 2e1 at the default temperature 1/sqrt(4):
    #   z0 = (2, 1, 0, 0), z1 = (0, 1, 2, 1)
    #   s_i = exp(z0_i) / (e^2 + e + 2) + exp(z1_i) / (1 + e)^2.
    # Block 0 (tokens 0..63) overlaps windows 0..3, block 1 (tokens 64..127) only window 3, so the
    # pooled scores are max(s) = s_0 and s_3.
    e = math.e
    d, T = 4, 80
    g = [[2, 0, 0, 0], [2, 0, 0, 0], [0, 2, 0, 0], [0, 2, 0, 0], [0, 0, 0, 0]]
    K = np.repeat(np.array(g, np.float64), 16, axis=0)
    u = O.UnitOracle(head_dim=d, k_q=1, k_e=1, window_tokens=0, max_context=T,
                     W1=np.zeros((d, 2)), W2=np.zeros(2))
    u.append(O.f64_to_bf16_bits(K), O.f64_to_bf16_bits(np.zeros((T, d))))
    assert np.array_equal(u.compressed_keys(), [[2, 0, 0, 0], [1, 1, 0, 0], [0, 2, 0, 0], [0, 1, 0, 0]])
    a, b = e ** 2 + e + 2, (1 + e) ** 2
    s0 = e ** 2 / a + 1 / b
    s3 = 1 / a + e / b
    sq, se = u.scores(O.f64_to_bf16_bits(np.array([[2.0, 0, 0, 0], [0, 2.0, 0, 0]])))
    assert abs(sq[0] - s0) < 1e-15 and abs(sq[1] - s3) < 1e-15
    assert abs(s0 - 0.6826251735421364) < 1e-15 and abs(s3 - 0.2792064726850172) < 1e-15
    # W2 = 0: every eviction score is zero, so both pooled query-agnostic scores are zero
    assert np.array_equal(se, [0.0, 0.0])


def test_single_head_query_score_is_softmax_of_mean_token_logits():
    # The explainer writes the query-aware score through per-token logits q.k_j pooled by the mean
    # over a window.  With one head and unrounded mean keys, query_scores must equal the softmax of
    # those pooled token logits at the same temperature (computed here without query_scores).
    rng = np.random.default_rng(4)
    K = rng.standard_normal((160, 16))
    q = rng.standard_normal(16)
    nc = O.num_windows(160)
    kbar = np.stack([K[16 * i:16 * i + 32].mean(0) for i in range(nc)])
    token_form = np.array([(K[16 * i:16 * i + 32] @ q).mean() for i in range(nc)]) * 0.25
    w = np.exp(token_form - token_form.max())
    assert np.max(np.abs(O.query_scores(q[None, :], kbar, 0.25) - w / w.sum())) < 1e-12


# ----------------------------------------------------------------------------- selection
def _best_subset_by_sum(scores, eligible, k):
    """Brute force: with distinct scores the top-k set is the k-subset of largest sum."""
    k = min(k, len(eligible))
    best, arg = -np.inf, None
    for sub in itertools.combinations(eligible, k):
        v = sum(float(scores[b]) for b in sub)
        if v > best:
            best, arg = v, sorted(sub)
    return arg if arg is not None else []


@pytest.mark.parametrize("seed", range(25))
def test_selection_brute_force(seed):
    rng = np.random.default_rng(seed)
    nb = int(rng.integers(6, 13))
    nw = int(rng.integers(1, 3))
    k_q, k_e = int(rng.integers(1, 4)), int(rng.integers(1, 4))
    sq = rng.permutation(nb).astype(np.float64) + 0.5    # distinct, exact in float32
    se = rng.permutation(nb).astype(np.float64) - 3.0
    _, C, _ = O.partition(nb * 64, nw)
    evicted = {b for b in C if rng.random() < 0.3}
    Q = O.select_query_aware(sq, C, k_q)
    assert Q == _best_subset_by_sum(sq, C, k_q)
    E = O.select_query_agnostic(se, C, Q, evicted, k_e)
    eligible = [b for b in C if b not in Q and b not in evicted]
    assert E == _best_subset_by_sum(se, eligible, k_e)
    assert not (set(E) & evicted) and not (set(E) & set(Q))


def test_selection_ties_go_to_lower_block():
    sq = np.zeros(10)
    assert O.select_query_aware(sq, list(range(1, 8)), 3) == [1, 2, 3]
    se = np.array([0, 5, 5, 1, 5, 5, 0, 0, 0, 0], dtype=np.float64)
    assert O.select_query_agnostic(se, list(range(1, 8)), [2], set(), 2) == [1, 4]


def test_selection_decided_in_float32():
    # two scores that differ only below float32 resolution tie, so the lower block wins
    sq = np.array([0.0, 1.0 + 1e-12, 1.0, 0.0])
    assert O.select_query_aware(sq, [1, 2], 1) == [1]
    sq = np.array([0.0, 1.0, 1.0 + 1e-12, 0.0])
    assert O.select_query_aware(sq, [1, 2], 1) == [1]


def test_partition_sink_window_candidates():
    sink, C, win = O.partition(4097, 4)          # 65 blocks, last one partial
    assert sink == [0] and win == [61, 62, 63, 64] and C == list(range(1, 61))
    assert O.partition(64 * 3, 4) == ([0], [], [1, 2])
    assert O.partition(1, 4) == ([0], [], [])


# ----------------------------------------------------------------------------- a unit over many steps
def _run_unit(T0, steps, k_q, k_e, window, sigma, seed, G=2, d=32, kernel=32, cache_slots=None):
    w = syn.Workload("t", 1, 1, G, 1, T0, k_q, k_e, window, steps, sigma=sigma, head_dim=d,
                     evict_hidden=16, seed=seed)
    x = w.unit_inputs(0, 0, 0)
    u = O.UnitOracle(head_dim=d, k_q=k_q, k_e=k_e, window_tokens=window,
                     max_context=T0 + steps, W1=x["W1"], W2=x["W2"], cache_slots=cache_slots)
    u.append(x["K"][:T0], x["V"][:T0])
    res = []
    for t in range(steps):
        p = T0 + t
        res.append(u.step(x["Q"][t], x["K"][p:p + 1], x["V"][p:p + 1]))
    return u, x, res


@pytest.mark.parametrize("sigma,seed", [(0.3, 0), (1.0, 1), (3.0, 2)])
def test_theorem2_locality_bound(sigma, seed):
    k_q, k_e = 4, 12
    _, _, res = _run_unit(2048, 70, k_q, k_e, 256, sigma, seed)
    gammas = [r["gamma"] for r in res[1:]]
    assert min(gammas) >= k_e / (k_q + k_e) - 1e-12
    c = json.load(open(os.path.join(GOLD, "page_constants.json")))
    k, kq = c["budget_tokens"] // 64, c["k_q_tokens"] // 64
    assert (k - kq) / k == c["gamma_lower_bound"]


def test_locality_hand_values():
    # gamma = |D_t & S_{t-1}| / |D_t|: D = {3, 5, 8, 9}, S_prev = {0, 3, 8, 12, 13, 14} share {3, 8}
    # -> 2 / 4.  Dividing by |S_prev| would give 2 / 6, intersecting S_t instead of D_t more.
    assert O.locality([3, 5, 8, 9], [0, 3, 8, 12, 13, 14]) == 0.5
    assert O.locality([3], [4]) == 0.0 and O.locality([], [1]) == 1.0


def test_unit_locality_over_two_hand_selections():
    # 10 blocks, window 2 blocks (8, 9), sink 0: candidates 1..7.  Selection 1: Q = {2}, E = {3, 4}
    # -> S_1 = {0, 2, 3, 4, 8, 9}.  Selection 2: Q = {5}, E = {3, 4} -> D_2 = {3, 4, 5}, of which
    # {3, 4} were in S_1: gamma = 2/3 (|S_2 & S_1| / |S_2| would be 5/6, / |S_1| would be 1/3).
    u = O.UnitOracle(head_dim=4, k_q=1, k_e=2, window_tokens=128, max_context=640,
                     W1=np.zeros((4, 2)), W2=np.zeros(2))
    u.append(np.zeros((640, 4), np.uint16), np.zeros((640, 4), np.uint16))
    r1 = u.commit([2], [3, 4])
    assert r1["S"] == [0, 2, 3, 4, 8, 9] and r1["gamma"] is None
    assert u.evicted == {1, 5, 6, 7}
    r2 = u.commit([5], [3, 4])
    assert r2["D"] == [3, 4, 5] and abs(r2["gamma"] - 2 / 3) < 1e-15
    assert r2["fetch"] == [(5, 1)]              # block 2 left its slot 1, block 5 takes it
    assert r2["gamma"] >= u.k_e / (u.k_q + u.k_e) - 1e-15


def test_eviction_is_sticky_and_fetches_follow_the_set_difference():
    k_q, k_e = 3, 6
    u, x, res = _run_unit(1500, 90, k_q, k_e, 128, 1.0, 5)
    dropped = set()
    S_prev = []
    cached = [-1] * u.cslots  # the slot map, replayed from the fetch lists
    for t, r in enumerate(res):
        assert not (set(r["E"]) & dropped)                       # never re-selected by E
        fetched = [b for b, _ in r["fetch"]]
        assert fetched == sorted(set(r["S"]) - set(cached))      # exactly the selected blocks not cached
        assert set(fetched) <= set(r["S"]) - set(S_prev)
        for b, sl in r["fetch"]:
            cached[sl] = b
        if t > 0:
            assert len(set(r["D"]) - set(S_prev)) <= k_q         # only Q can bring new dynamic blocks
        slots = r["slot_of"]
        assert len(set(slots)) == len(slots) and max(slots) < u.cap
        _, C, _ = O.partition(1500 + t + 1, 2)
        dropped |= {b for b in C if b not in set(r["D"])}
        S_prev = r["S"]
    assert len(res[0]["fetch"]) == len(res[0]["S"])              # cold first step fetches all of S_1


def test_a_larger_cache_changes_only_the_transfers():
    # twice the selection's slots: the same selections, eviction and outputs, fewer fetches; a
    # selected block is fetched exactly when it holds no slot, and every slot holds a distinct block
    k_q, k_e = 4, 12
    u1, _, r1 = _run_unit(2048, 60, k_q, k_e, 256, 1.0, 4)
    u2, _, r2 = _run_unit(2048, 60, k_q, k_e, 256, 1.0, 4, cache_slots=2 * (1 + 4 + k_q + k_e))
    assert u2.cslots == 2 * u1.cap
    cached = [-1] * u2.cslots
    for a, b in zip(r1, r2):
        assert a["S"] == b["S"] and a["D"] == b["D"] and a["gamma"] == b["gamma"]
        assert np.array_equal(a["out"], b["out"])
        assert [x for x, _ in b["fetch"]] == [x for x in b["S"] if x not in set(cached)]
        for x, sl in b["fetch"]:
            cached[sl] = x
        assert sorted(cached[sl] for sl in b["slot_of"]) == b["S"]
    assert u1.evicted == u2.evicted
    n1, n2 = sum(len(r["fetch"]) for r in r1), sum(len(r["fetch"]) for r in r2)
    assert n2 < n1


def test_budget_accounting_and_transfer_unit():
    c = json.load(open(os.path.join(GOLD, "page_constants.json")))
    bb = c["budget_blocks"]
    assert bb["sink"] + bb["window"] + bb["dynamic"] == bb["total"] == c["budget_tokens"] // c["block_tokens"]
    assert c["block_tokens"] * c["head_dim"] * 2 == c["block_transfer_bytes"]
    _, _, res = _run_unit(3000, 10, 4, 8, 256, 0.3, 3)
    # the query-agnostic part comes up short only when Q takes blocks it could have kept
    assert res[0]["short"] == 0
    for r in res:
        assert len(r["S"]) == 1 + 4 + 4 + 8 - r["short"] and len(r["Q"]) == 4


def test_k_e_zero_is_plain_top_k():
    u, x, res = _run_unit(2000, 5, 6, 0, 128, 0.3, 4)
    for r in res:
        assert r["E"] == [] and r["D"] == r["Q"]
        _, C, _ = O.partition(u.T, 2)
        order = sorted(C, key=lambda b: (-np.float32(r["sq_blk"][b]), b))
        assert r["Q"] == sorted(order[:6])


# ----------------------------------------------------------------------------- forecast (SparDA)
def _pair(T0, steps, k_q, k_e, window, sigma, seed, G, d=32):
    w = syn.Workload("f", 1, 1, G, 1, T0, k_q, k_e, window, steps, sigma=sigma, head_dim=d,
                     evict_hidden=16, seed=seed)
    x = w.unit_inputs(0, 0, 0)

    def unit():
        u = O.UnitOracle(head_dim=d, k_q=k_q, k_e=k_e, window_tokens=window, max_context=T0 + steps,
                         W1=x["W1"], W2=x["W2"])
        u.append(x["K"][:T0], x["V"][:T0])
        return u
    return unit(), unit(), x


def test_forecast_with_the_query_as_forecast_selects_what_the_plain_step_selects():
    # One q head per kv head and the forecast equal to the query: selecting before the append
    # (windows complete now, blocks of T+1) and after it differ only by the window the new token
    # completes, which overlaps window blocks only and rescales every candidate's softmax score
    # by one factor -- the same blocks are chosen, slots, fetches and outputs agree.
    T0, steps = 2000, 70                  # a new block starts at T = 2049 (step 49)
    a, b, x = _pair(T0, steps, 4, 8, 256, 1.0, 3, G=1)
    for t in range(steps):
        p = T0 + t
        ra = a.step(x["Q"][t], x["K"][p:p + 1], x["V"][p:p + 1])
        rb = b.forecast_step(x["Q"][t][0], x["Q"][t], x["K"][p:p + 1], x["V"][p:p + 1])
        for key in ("S", "D", "fetch", "slot_of"):
            assert ra[key] == rb[key], (t, key)
        assert a.evicted == b.evicted
        assert np.max(np.abs(ra["out"] - rb["out"])) < 1e-12


def test_forecast_selection_keeps_the_locality_bound_and_fetches_a_new_tail_block():
    T0, steps, k_q, k_e = 2048, 60, 4, 12  # the first forecast already serves a new block
    _, u, x = _pair(T0, steps, k_q, k_e, 256, 1.0, 4, G=2)
    gammas = []
    for t in range(steps):
        p = T0 + t
        r = u.forecast_step(x["F"][t], x["Q"][t], x["K"][p:p + 1], x["V"][p:p + 1])
        if t == 0:
            assert 32 in r["S"] and 32 in [b for b, _ in r["fetch"]]   # block 32 starts at token 2048
        if r["gamma"] is not None:
            gammas.append(r["gamma"])
        assert all(b < O.num_blocks(T0 + t + 1) for b in r["S"])
    assert min(gammas) >= k_e / (k_q + k_e) - 1e-12


# ----------------------------------------------------------------------------- attention
def _sdpa(Q, K, V, scale, mask=None):
    q = torch.from_numpy(Q)[None, :, None, :]
    k = torch.from_numpy(K)[None, None].expand(1, Q.shape[0], -1, -1)
    v = torch.from_numpy(V)[None, None].expand(1, Q.shape[0], -1, -1)
    m = None if mask is None else torch.from_numpy(mask)[None, None, None, :]
    return torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m, scale=scale)[0, :, 0].numpy()


def test_covering_budget_equals_dense_attention():
    # k covers every candidate: S is every block and the output is dense decode attention
    T0, d = 1000, 32
    u, x, res = _run_unit(T0, 4, 20, 20, 128, 0.3, 6, d=d)
    for t, r in enumerate(res):
        T = T0 + t + 1
        assert r["S"] == list(range(O.num_blocks(T)))
        Qg = O.bf16_bits_to_f64(x["Q"][t])
        K = O.bf16_bits_to_f64(x["K"][:T]); V = O.bf16_bits_to_f64(x["V"][:T])
        assert np.max(np.abs(r["out"] - _sdpa(Qg, K, V, 1 / math.sqrt(d)))) < 1e-6


def test_sparse_attention_equals_masked_dense():
    rng = np.random.default_rng(7)
    T, d = 700, 16
    K, V = rng.standard_normal((T, d)), rng.standard_normal((T, d))
    Q = rng.standard_normal((3, d))
    S = [0, 2, 5, 10]
    mask = np.zeros(T, bool)
    for b in S:
        mask[64 * b: min(64 * b + 64, T)] = True
    got = O.sparse_attention(Q, K, V, S, T, 0.3)
    assert np.max(np.abs(got - _sdpa(Q, K, V, 0.3, mask))) < 1e-12


# DMA-style additive attention bias (wiki "How NOSA works": the eviction head comes from DMA,
# which adds its per-token score to the attention logits).
def test_dma_bias_equals_sdpa_with_an_additive_float_mask():
    rng = np.random.default_rng(11)
    T, d = 700, 16
    K, V = rng.standard_normal((T, d)), rng.standard_normal((T, d))
    Q = rng.standard_normal((3, d))
    bias = rng.standard_normal(T) * 2.0
    S = [0, 2, 5, 10]
    mask = np.full(T, -np.inf)
    for b in S:
        mask[64 * b: min(64 * b + 64, T)] = bias[64 * b: min(64 * b + 64, T)]
    got = O.sparse_attention(Q, K, V, S, T, 0.3, bias=bias)
    assert np.max(np.abs(got - _sdpa(Q, K, V, 0.3, mask))) < 1e-12


def test_dma_bias_constant_shift_changes_nothing_and_two_tokens_match_the_closed_form():
    rng = np.random.default_rng(12)
    T, d = 130, 8
    K, V = rng.standard_normal((T, d)), rng.standard_normal((T, d))
    Q = rng.standard_normal((2, d))
    S = [0, 2]
    plain = O.sparse_attention(Q, K, V, S, T, 0.5)
    shifted = O.sparse_attention(Q, K, V, S, T, 0.5, bias=np.full(T, 7.25))
    assert np.max(np.abs(plain - shifted)) < 1e-12
    # two tokens (block 2 holds tokens 128, 129 only): softmax of z + b written out
    q = Q[0]
    z = np.array([q @ K[128], q @ K[129]]) * 0.5
    b = np.array([0.7, -1.9])
    w = np.exp(z + b)
    want = (w[0] * V[128] + w[1] * V[129]) / w.sum()
    bias = np.zeros(T)
    bias[128:130] = b
    got = O.sparse_attention(Q[:1], K, V, [2], T, 0.5, bias=bias)[0]
    assert np.max(np.abs(got - want)) < 1e-12


def test_unit_dma_bias_is_the_eviction_score_of_each_token():
    # One hidden unit: s^e_j = -100 * softplus(v_j[0]).  Block 3's tokens get v[0] = 20 (bias about
    # -2000: masked out), every other token v[0] = -20 (bias about -2e-7: no effect), so with the
    # bias the output is attention over the selection without block 3; with W2 = 0 it is unbiased.
    rng = np.random.default_rng(13)
    T, d = 600, 16
    K = O.bf16_round(rng.standard_normal((T, d)))
    V = O.bf16_round(rng.standard_normal((T, d)))
    V[:, 0] = -20.0
    V[192:256, 0] = 20.0
    W1 = np.zeros((d, 1)); W1[0, 0] = 1.0
    Q = O.f64_to_bf16_bits(rng.standard_normal((2, d)))
    S = [0, 1, 3, 5, 9]

    def unit(W2, dma):
        u = O.UnitOracle(head_dim=d, k_q=2, k_e=2, window_tokens=128, max_context=T, W1=W1, W2=W2,
                         dma_bias=dma)
        u.append(O.f64_to_bf16_bits(K), O.f64_to_bf16_bits(V))
        return u.attend(Q, S)

    Qg = O.bf16_bits_to_f64(Q)
    without3 = O.sparse_attention(Qg, K, V, [0, 1, 5, 9], T, 1 / math.sqrt(d))
    plain = O.sparse_attention(Qg, K, V, S, T, 1 / math.sqrt(d))
    assert np.max(np.abs(unit(np.array([-100.0]), True) - without3)) < 1e-5
    assert np.max(np.abs(unit(np.array([0.0]), True) - plain)) < 1e-12
    assert np.max(np.abs(unit(np.array([-100.0]), False) - plain)) < 1e-12


def test_assign_slots_pairs_ascending():
    fetch, m, lu, where = O.assign_slots([0, 3, 4, 9], [3, -1, 7, 0, 8], T=5)
    # open slots 1 (empty), 2 (block 7) and 4 (block 8), none selected before: the two lowest
    # go to the new blocks 4 and 9; block 8 stays cached in slot 4
    assert fetch == [(4, 1), (9, 2)] and m == [3, 4, 9, 0, 8] and where == [3, 0, 1, 2]
    assert lu == [5, 5, 5, 5, -1]


def test_assign_slots_replaces_the_least_recently_selected():
    # four slots, worked by hand: a block that left the selection stays cached while slots
    # selected longer ago (or never) are free to take, and comes back without a fetch
    m, lu = [-1] * 4, None
    fetch, m, lu, where = O.assign_slots([0, 1], m, lu, T=10)
    assert fetch == [(0, 0), (1, 1)] and m == [0, 1, -1, -1] and lu == [10, 10, -1, -1]
    fetch, m, lu, where = O.assign_slots([0, 2], m, lu, T=11)   # empty slots before block 1's
    assert fetch == [(2, 2)] and m == [0, 1, 2, -1] and lu == [11, 10, 11, -1]
    fetch, m, lu, where = O.assign_slots([0, 3, 4], m, lu, T=12)  # slot 3 (never), slot 1 (T 10)
    assert fetch == [(3, 1), (4, 3)] and m == [0, 3, 2, 4] and lu == [12, 12, 11, 12] and where == [0, 1, 3]
    fetch, m, lu, where = O.assign_slots([0, 1, 2], m, lu, T=13)  # block 2 still cached
    assert fetch == [(1, 1)] and m == [0, 1, 2, 4] and lu == [13, 13, 13, 12] and where == [0, 1, 2]


def test_assign_slots_with_a_selection_sized_cache_frees_exactly_the_blocks_that_left():
    # the pages' cache (as many slots as a full selection): written out directly, freed slots
    # (ascending) paired with new blocks (ascending) -- the same fetch lists and slot maps
    rng = np.random.default_rng(3)
    cap, m, lu, ref = 6, [-1] * 6, None, [-1] * 6
    for T in range(40):
        S = sorted(rng.choice(20, size=cap, replace=False).tolist())
        fetch, m, lu, where = O.assign_slots(S, m, lu, T)
        keep = set(S)
        resident = {b for b in ref if b >= 0}
        ref = [b if b in keep else -1 for b in ref]
        free = [s for s, b in enumerate(ref) if b < 0]
        new = [b for b in S if b not in resident]
        want = list(zip(new, free))
        for b, s in want:
            ref[s] = b
        assert fetch == want and m == ref


# ----------------------------------------------------------------------------- inputs
def test_synthetic_inputs_are_counter_based():
    a = syn.normals(0, syn.T_K, 1, 2, 3, 1001, 77)
    b = syn.normals(0, syn.T_K, 1, 2, 3, 1000, 100)[1:78]
    assert np.array_equal(a, b)
    z = syn.normals(0, syn.T_V, 0, 0, 0, 0, 1 << 18)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    q = O.bf16_bits_to_f64(syn.query_walk(0, 0, 0, 0, 4, 128, 0.3))
    assert np.allclose(np.linalg.norm(q, axis=1), math.sqrt(128), rtol=1e-2)
