"""Seeded synthetic inputs for the NOSA decode path.

This module is shared by the CPU oracle tests, the GPU parity tests and the
bench's CPU-baseline leg.  It holds none of the method's arithmetic: it only
draws numbers.  Every value is a pure function of
(seed, tensor id, layer, batch, head, position, dim), so any slice of any
tensor can be regenerated on its own without generating the rest.

Generator (all integer steps are exact, so any implementation agrees bit for bit):
  * stream key   = SplitMix64 chained over (seed, tensor id, layer, batch, head)
  * raw word n   = SplitMix64(key + n)                       (64-bit wrap-around)
  * uniforms     = u1 = ((w_{2j} >> 11) + 1) * 2^-53 in (0, 1],
                   u2 = (w_{2j+1} >> 11) * 2^-53 in [0, 1)
  * normals      = Box-Muller in float64: r = sqrt(-2 ln u1),
                   element 2j = r cos(2 pi u2), element 2j+1 = r sin(2 pi u2)
  * bf16 values  = float64 -> float32 (round to nearest even) -> bf16 (RNE)

SplitMix64 is the public mixing function of Steele, Lea and Flood
("Fast splittable pseudorandom number generators", OOPSLA 2014), as
popularised by Vigna's xorshift/xoshiro seeding code.

Workload recipe (what the five benchmark shapes draw, per layer l):
  * K, V context tokens ~ N(0, 1), rounded to bf16, per (l, b, kv head g, pos)
  * eviction head W1 (d x h) ~ N(0, 1/d), W2 (h) ~ N(0, 1/h), float32, per (l, g)
  * queries: a random walk per (l, b, q head h):
        q_0 = normalize(N(0, I)) * sqrt(d)
        q_t = normalize(q_{t-1} + sigma * N(0, I)) * sqrt(d)
    carried in float64; the query used at decode step t >= 1 is bf16(q_t).
  * the token appended at decode step t sits at position T_0 + t - 1 and is
    drawn from the same K / V streams as the context.
"""
from __future__ import annotations

import numpy as np

# tensor ids (part of the stream key)
T_K, T_V, T_W1, T_W2, T_Q0, T_QN, T_F0, T_FN = 1, 2, 3, 4, 5, 6, 7, 8

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)


def splitmix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser applied elementwise to a uint64 array (wraps mod 2^64)."""
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
        return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor: int, layer: int, batch: int, head: int) -> np.uint64:
    key = splitmix64(np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))
    for field in (tensor, layer, batch, head):
        key = splitmix64(key ^ np.uint64(field & 0xFFFFFFFFFFFFFFFF))
    return key[0]


def normals(seed: int, tensor: int, layer: int, batch: int, head: int,
            start: int, count: int) -> np.ndarray:
    """Elements [start, start+count) of one stream as float64 N(0, 1) draws."""
    if count <= 0:
        return np.zeros(0, dtype=np.float64)
    key = stream_key(seed, tensor, layer, batch, head)
    j0 = start // 2
    j1 = (start + count + 1) // 2
    pairs = np.arange(j0, j1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        w1 = splitmix64(key + pairs * np.uint64(2))
        w2 = splitmix64(key + pairs * np.uint64(2) + np.uint64(1))
    u1 = ((w1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (w2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * len(pairs), dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    off = start - 2 * int(j0)
    return z[off:off + count]


# ---------------------------------------------------------------- bf16 helpers
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 draw -> float32 (RNE) -> bf16 (RNE), as bit patterns."""
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float64).astype(np.float32))


# ---------------------------------------------------------------- tensors
def kv_tokens(seed: int, which: int, layer: int, batch: int, kv_head: int,
              pos0: int, n: int, d: int) -> np.ndarray:
    """bf16 bits [n][d] of K (which=T_K) or V (which=T_V) for positions pos0..pos0+n-1."""
    return to_bf16_bits(normals(seed, which, layer, batch, kv_head, pos0 * d, n * d)).reshape(n, d)


def eviction_head(seed: int, layer: int, kv_head: int, d: int, h: int):
    """float32 W1 [d][h] ~ N(0, 1/d) and W2 [h] ~ N(0, 1/h)."""
    w1 = (normals(seed, T_W1, layer, 0, kv_head, 0, d * h) / np.sqrt(d)).astype(np.float32).reshape(d, h)
    w2 = (normals(seed, T_W2, layer, 0, kv_head, 0, h) / np.sqrt(h)).astype(np.float32)
    return w1, w2


def query_walk(seed: int, layer: int, batch: int, q_head: int, steps: int, d: int,
               sigma: float, tensors=(T_Q0, T_QN)) -> np.ndarray:
    """bf16 bits [steps][d]: row t-1 is the query of decode step t (t = 1..steps)."""
    q = normals(seed, tensors[0], layer, batch, q_head, 0, d)
    q = q / np.linalg.norm(q) * np.sqrt(d)
    out = np.empty((steps, d), dtype=np.uint16)
    noise = normals(seed, tensors[1], layer, batch, q_head, 0, steps * d).reshape(steps, d)
    for t in range(steps):
        q = q + sigma * noise[t]
        q = q / np.linalg.norm(q) * np.sqrt(d)
        out[t] = to_bf16_bits(q)
    return out


class Workload:
    """Shape of one decode workload (one of the five benchmark shapes or a test shape)."""

    def __init__(self, name, layers, batch, q_heads, kv_heads, context, k_q, k_e,
                 window_tokens, steps, sigma=0.3, head_dim=128, block=64,
                 evict_hidden=128, sink_blocks=1, seed=0):
        self.name = name
        self.layers, self.batch = layers, batch
        self.q_heads, self.kv_heads = q_heads, kv_heads
        self.context, self.k_q, self.k_e = context, k_q, k_e
        self.window_tokens, self.steps, self.sigma = window_tokens, steps, sigma
        self.head_dim, self.block, self.evict_hidden = head_dim, block, evict_hidden
        self.sink_blocks, self.seed = sink_blocks, seed

    @property
    def group(self):
        return self.q_heads // self.kv_heads

    @property
    def max_context(self):
        return self.context + self.steps

    def unit_inputs(self, layer: int, batch: int, kv_head: int):
        """Everything one (layer, batch, kv head) unit consumes, as numpy arrays."""
        d, G = self.head_dim, self.group
        n = self.context + self.steps
        K = kv_tokens(self.seed, T_K, layer, batch, kv_head, 0, n, d)
        V = kv_tokens(self.seed, T_V, layer, batch, kv_head, 0, n, d)
        W1, W2 = eviction_head(self.seed, layer, kv_head, d, self.evict_hidden)
        Q = np.stack([query_walk(self.seed, layer, batch, kv_head * G + j, self.steps, d, self.sigma)
                      for j in range(G)], axis=1)  # [steps][G][d]
        # forecast vectors (one per kv head, the same random walk on their own streams)
        F = query_walk(self.seed, layer, batch, kv_head, self.steps, d, self.sigma, (T_F0, T_FN))  # [steps][d]
        return dict(K=K, V=V, W1=W1, W2=W2, Q=Q, F=F)


# The five benchmark shapes (synthetic stand-ins for the pages' PG19 / NOSA-1B / NOSA-8B runs).
WORKLOADS = {
    "tiny": dict(layers=1, batch=1, q_heads=16, kv_heads=2, context=4096, k_q=4, k_e=12,
                 window_tokens=256, steps=32),
    "nosa1b_16k_b8": dict(layers=28, batch=8, q_heads=16, kv_heads=2, context=16384, k_q=16, k_e=48,
                          window_tokens=1024, steps=256),
    "nosa1b_16k_b128": dict(layers=28, batch=128, q_heads=16, kv_heads=2, context=16384, k_q=16, k_e=48,
                            window_tokens=1024, steps=128),
    "nosa8b_32k_b32": dict(layers=32, batch=32, q_heads=32, kv_heads=8, context=32768, k_q=16, k_e=48,
                           window_tokens=1024, steps=128),
    "nosa1b_64k_b32": dict(layers=28, batch=32, q_heads=16, kv_heads=2, context=65536, k_q=16, k_e=48,
                           window_tokens=1024, steps=64),
}


def workload(name: str, **over) -> Workload:
    kw = dict(WORKLOADS[name])
    kw.update(over)
    return Workload(name, **kw)
