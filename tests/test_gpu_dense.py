"""Dense decode attention (the full-attention comparator) against the oracle.

nosa_dense_attend attends every token of a device-resident KV store; the oracle's
attention over all blocks (a selection covering the whole context) is its
reference, which tests/test_oracle.py pins to SDPA.
"""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle import nosa_oracle as O  # noqa: E402
from offloadable_block_sparse_gb300 import nosa as N  # noqa: E402


def _case(units, group, T, max_blocks, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    d = 128
    kv = torch.randn((units, max_blocks, 2, 64, d), generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn((units, group, d), generator=g, device="cuda")
    q = (q / q.norm(dim=-1, keepdim=True) * math.sqrt(d)).to(torch.bfloat16)
    return q, kv


def _oracle(q, kv, T):
    units, group, d = q.shape
    qh = q.float().cpu().numpy().astype(np.float64)
    kvh = kv.float().cpu().numpy().astype(np.float64)
    nb = -(-T // 64)
    refs = []
    for u in range(units):
        K = kvh[u, :, 0].reshape(-1, d)[:T]
        V = kvh[u, :, 1].reshape(-1, d)[:T]
        refs.append(O.sparse_attention(qh[u], K, V, list(range(nb)), T, 1 / math.sqrt(d)))
    return np.stack(refs)


@pytest.mark.parametrize("units,group,T,max_blocks", [(6, 8, 3000, 50), (4, 4, 64, 1), (2, 8, 70000, 1100)],
                         ids=["ragged", "one-block", "long"])
def test_dense_attention_matches_the_oracle_twice(units, group, T, max_blocks):
    q, kv = _case(units, group, T, max_blocks, seed=units * 1000 + T)
    nbytes = N.nosa_dense_scratch_bytes(units, T)
    assert nbytes > 0
    scratch = torch.zeros(nbytes // 4 + 64, dtype=torch.int32, device="cuda")
    ref = _oracle(q, kv, T)
    for _ in range(2):  # the scratch is reused
        out = torch.full((units, group, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        N.nosa_dense_attend(q.view(torch.int16), kv.view(torch.int16), units, group, max_blocks, T,
                            out.view(torch.int16), scratch, nbytes, stream=torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        err = np.abs(got - ref)
        assert np.isfinite(got).all()
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
        assert err.max() <= 2 ** -7 * np.abs(ref).max() + 1e-4, err.max()
    assert int(scratch[0].item()) == 0  # no device-side error bits


def test_dense_scratch_too_small_is_refused():
    q, kv = _case(2, 8, 1000, 16, seed=1)
    nbytes = N.nosa_dense_scratch_bytes(2, 1000)
    scratch = torch.zeros(nbytes // 4 + 64, dtype=torch.int32, device="cuda")
    out = torch.empty((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(N.NosaError) as e:
        N.nosa_dense_attend(q.view(torch.int16), kv.view(torch.int16), 2, 8, 16, 1000, out.view(torch.int16),
                            scratch, nbytes - 4)
    assert e.value.status == N.NOSA_ERR_CAPACITY
    with pytest.raises(N.NosaError) as e:  # the context does not fit the store
        N.nosa_dense_attend(q.view(torch.int16), kv.view(torch.int16), 2, 8, 15, 1000, out.view(torch.int16),
                            scratch, nbytes)
    assert e.value.status == N.NOSA_ERR_INVALID_ARG
