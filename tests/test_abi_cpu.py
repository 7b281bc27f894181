"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point declared in include/nosa.h, validates configs and derives
sizes; context creation without a GPU fails with a status, not a crash."""
import ctypes
import os
import re

import pytest

from offloadable_block_sparse_gb300 import build as B
from offloadable_block_sparse_gb300 import nosa as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    if not os.path.exists(N.LIB_PATH):
        B.build()


def _declared():
    src = open(os.path.join(ROOT, "include", "nosa.h")).read()
    return sorted(set(re.findall(r"^\S.*?\b(nosa_[a-z_]+)\(", src, re.M)))


def test_header_and_binding_agree():
    assert _declared() == sorted(N.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(N.LIB_PATH)
    for name in _declared():
        assert hasattr(lib, name), name


def _cfg(**kw):
    base = dict(num_layers=2, batch=3, num_q_heads=16, num_kv_heads=2, k_q=4, k_e=12, window_tokens=256,
                max_context=5000)
    base.update(kw)
    return N.make_config(**base)


def test_validate_config():
    assert N.nosa_validate_config(_cfg()) == N.NOSA_OK
    bad = [dict(head_dim=64), dict(block_size=32), dict(cmp_kernel=16), dict(cmp_stride=8),
           dict(num_q_heads=15), dict(num_q_heads=32, num_kv_heads=2), dict(k_q=-1), dict(window_tokens=100),
           dict(max_context=0), dict(max_context=1 << 20), dict(evict_hidden=100), dict(flags=64),
           dict(k_q=200, k_e=100), dict(batch=4097, num_kv_heads=1, num_q_heads=8), dict(softmax_scale=-1.0),
           dict(score_ctas=9), dict(score_ctas=-1), dict(attend_blocks_per_cta=65), dict(attend_merge=4),
           dict(decode_cluster=9), dict(decode_teams=3), dict(decode_stages=1), dict(decode_stages=7),
           dict(forecast_streams=3), dict(cache_slots=20), dict(cache_slots=257)]
    for b in bad:
        assert N.nosa_validate_config(_cfg(**b)) == N.NOSA_ERR_INVALID_ARG, b
    c = _cfg()
    c.struct_size = 4
    assert N.nosa_validate_config(c) == N.NOSA_ERR_INVALID_ARG


def test_sizing_overrides_are_accepted():
    good = [dict(score_ctas=1), dict(score_ctas=8), dict(attend_blocks_per_cta=1), dict(attend_blocks_per_cta=64),
            dict(attend_merge=N.NOSA_MERGE_TICKET), dict(attend_merge=N.NOSA_MERGE_CLUSTER),
            dict(decode_cluster=2), dict(decode_teams=1), dict(decode_stages=6), dict(forecast_streams=1),
            dict(cache_slots=21), dict(cache_slots=256)]
    for g in good:
        assert N.nosa_validate_config(_cfg(**g)) == N.NOSA_OK, g


def test_test_hook_flags_are_accepted():
    assert N.nosa_validate_config(_cfg(flags=N.NOSA_F_TEST_ZERO_WAIT)) == N.NOSA_OK
    assert N.nosa_validate_config(_cfg(flags=N.NOSA_F_TEST_BAD_SLOT | N.NOSA_F_TEST_ZERO_WAIT)) == N.NOSA_OK
    assert N.nosa_validate_config(_cfg(flags=N.NOSA_F_UNFUSED_STEP)) == N.NOSA_OK
    assert N.nosa_validate_config(_cfg(flags=N.NOSA_F_DMA_BIAS | N.NOSA_F_UNFUSED_STEP)) == N.NOSA_OK
    assert N.nosa_validate_config(_cfg(flags=N.NOSA_F_TEST_RADIX_TOPK | N.NOSA_F_TEST_PREFILL_WIDE)) == N.NOSA_OK


def test_query_sizes_closed_forms():
    s = N.nosa_query_sizes(_cfg())
    assert s.units_per_layer == 6 and s.group == 8
    assert s.select_slots == 1 + 4 + 4 + 12
    assert s.cache_slots == 2 * s.select_slots  # the rule: twice a selection
    one = N.nosa_query_sizes(_cfg(cache_slots=21))
    assert one.cache_slots == 21 and one.select_slots == 21
    # each extra cache slot of every (layer, unit): one 32 KiB block, its block id and its last-selection mark
    assert s.device_state_bytes - one.device_state_bytes == 2 * 6 * (42 - 21) * (32768 + 4 + 4)
    assert s.max_blocks == -(-5000 // 64) and s.max_windows == (5000 - 32) // 16 + 1
    assert s.evict_words == -(-s.max_blocks // 32)
    # one block of K plus V is 2 x 16 KiB (the transfer unit on the NOSA wiki)
    assert s.host_store_bytes == 2 * 6 * s.max_blocks * 2 * 16384


def test_status_strings():
    for i, name in enumerate(N.STATUS_NAMES):
        assert N.nosa_status_string(i) and N.nosa_status_string(i) != "unknown status", name


def test_null_and_bad_arguments_are_rejected_without_a_gpu():
    lib = N.lib()
    assert lib.nosa_validate_config(None) == N.NOSA_ERR_INVALID_ARG
    assert lib.nosa_create(None, None, None) == N.NOSA_ERR_INVALID_ARG
    assert lib.nosa_destroy(None) == N.NOSA_OK
    assert lib.nosa_step(None, 0, None, None, None, None) == N.NOSA_ERR_INVALID_ARG
    assert lib.nosa_sync(None) == N.NOSA_ERR_INVALID_ARG


def test_create_without_gpu_reports_a_status():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(N.NosaError) as e:
        N.nosa_create(_cfg())
    assert e.value.status == N.NOSA_ERR_CUDA
