"""The prefill benchmark's prompt queries (bench.prompt_queries) against the workload's query
model: the decode steps' random walk q_t = normalize(q_{t-1} + sigma N(0, I)) sqrt(d)
(synth.inputs.query_walk).  The benchmark generates its prompts in closed form rather than one
step per position; these checks hold it to the walk's norm and its correlation along the
positions, at one lag and at ten."""
import math

import numpy as np
import pytest
import torch

import bench
from oracle import nosa_oracle as O
from synth import inputs as syn


def _corr(q, lag):
    # mean cosine between positions t and t + lag, q [heads][n][d]
    a, b = q[:, lag:], q[:, :-lag]
    return float(((a * b).sum(-1) / (np.linalg.norm(a, axis=-1) * np.linalg.norm(b, axis=-1))).mean())


@pytest.mark.parametrize("sigma", [0.3, 1.0])
def test_prompt_queries_follow_the_decode_walk(sigma):
    d, n = 128, 700
    gen = torch.Generator().manual_seed(0)
    q = bench.prompt_queries(2, 8, n, d, sigma, gen, "cpu").float().numpy().reshape(16, n, d)
    assert np.allclose(np.linalg.norm(q, axis=-1), math.sqrt(d), rtol=1e-2)
    walk = np.stack([O.bf16_bits_to_f64(syn.query_walk(0, 0, 0, h, n, d, sigma)) for h in range(16)])
    for lag in (1, 10):
        want = _corr(walk, lag)
        assert abs(_corr(q, lag) - want) < 0.02, (lag, _corr(q, lag), want)
    assert abs(_corr(q, 1) - 1 / math.sqrt(1 + sigma ** 2)) < 0.01
