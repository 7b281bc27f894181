"""ctypes binding of libnosa.so: the C ABI of include/nosa.h under the same names.

Argument marshalling only -- every step of the decode path runs in the CUDA
kernels of libnosa.so.  Pointer arguments accept an integer address, a torch
tensor (``data_ptr()``), a numpy array (``ctypes.data``) or None (NULL).
If the library has not been built the first call raises ``RuntimeError``:
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnosa.so")

NOSA_OK = 0
STATUS_NAMES = ["NOSA_OK", "NOSA_ERR_INVALID_ARG", "NOSA_ERR_OOM", "NOSA_ERR_HOST_ALLOC", "NOSA_ERR_CUDA",
                "NOSA_ERR_CAPACITY", "NOSA_ERR_TIMEOUT", "NOSA_ERR_BOUNDS", "NOSA_ERR_STATE"]
globals().update({n: i for i, n in enumerate(STATUS_NAMES)})
NOSA_F_TEST_ZERO_WAIT = 1
NOSA_F_TEST_BAD_SLOT = 2
NOSA_F_UNFUSED_STEP = 4
NOSA_F_DMA_BIAS = 8
NOSA_F_TEST_RADIX_TOPK = 16
NOSA_F_TEST_PREFILL_WIDE = 32
NOSA_MERGE_AUTO, NOSA_MERGE_KERNEL, NOSA_MERGE_TICKET, NOSA_MERGE_CLUSTER = 0, 1, 2, 3

# every entry point declared in include/nosa.h
EXPORTS = ["nosa_validate_config", "nosa_query_sizes", "nosa_create", "nosa_destroy", "nosa_set_stream",
           "nosa_set_eviction_head", "nosa_append_kv", "nosa_select", "nosa_fetch", "nosa_attend", "nosa_step",
           "nosa_step_host", "nosa_step_host_all", "nosa_sync", "nosa_reset_state", "nosa_context_length", "nosa_get_stats",
           "nosa_reset_stats", "nosa_debug_scores", "nosa_export_state", "nosa_status_string",
           "nosa_attend_noalloc", "nosa_step_plan", "nosa_forecast_select", "nosa_step_forecast",
           "nosa_forecast_join", "nosa_dense_attend", "nosa_dense_scratch_bytes", "nosa_prefill",
           "nosa_prefill_scratch_bytes"]


class nosa_config(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("num_layers", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("cmp_kernel", ctypes.c_int32), ("cmp_stride", ctypes.c_int32),
                ("k_q", ctypes.c_int32), ("k_e", ctypes.c_int32), ("sink_blocks", ctypes.c_int32),
                ("window_tokens", ctypes.c_int32), ("max_context", ctypes.c_int32),
                ("evict_hidden", ctypes.c_int32), ("gather_ctas", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("flags", ctypes.c_uint32),
                ("score_ctas", ctypes.c_int32), ("attend_blocks_per_cta", ctypes.c_int32),
                ("attend_merge", ctypes.c_int32), ("decode_cluster", ctypes.c_int32),
                ("decode_teams", ctypes.c_int32), ("decode_stages", ctypes.c_int32),
                ("forecast_streams", ctypes.c_int32), ("cache_slots", ctypes.c_int32)]


class nosa_sizes(ctypes.Structure):
    _fields_ = [("units_per_layer", ctypes.c_int32), ("group", ctypes.c_int32), ("cache_slots", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32), ("max_windows", ctypes.c_int32), ("evict_words", ctypes.c_int32),
                ("host_store_bytes", ctypes.c_uint64), ("device_state_bytes", ctypes.c_uint64),
                ("select_slots", ctypes.c_int32), ("pad_", ctypes.c_int32)]


class nosa_stats(ctypes.Structure):
    _fields_ = [("selections", ctypes.c_uint64), ("gamma_samples", ctypes.c_uint64),
                ("gamma_mean", ctypes.c_double), ("gamma_min", ctypes.c_double),
                ("blocks_fetched", ctypes.c_uint64), ("bytes_fetched", ctypes.c_uint64),
                ("short_selections", ctypes.c_uint64)]


class nosa_state_view(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("sel", "sel_kind", "sel_slot", "n_sel", "fetch", "n_fetch",
                                               "slot_blk", "evicted", "kt", "se_win", "se_blk", "gamma",
                                               "last_used")]


class NosaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{where}: {name} ({_string(status)})")


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libnosa.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, p = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
        sig = {
            "nosa_validate_config": [ctypes.POINTER(nosa_config)],
            "nosa_query_sizes": [ctypes.POINTER(nosa_config), ctypes.POINTER(nosa_sizes)],
            "nosa_create": [ctypes.POINTER(nosa_config), vp, ctypes.POINTER(vp)],
            "nosa_destroy": [vp],
            "nosa_set_stream": [vp, vp],
            "nosa_set_eviction_head": [vp, i32, p, p],
            "nosa_append_kv": [vp, i32, p, p, i32, i32],
            "nosa_select": [vp, i32, p, p, p],
            "nosa_fetch": [vp, i32],
            "nosa_attend": [vp, i32, p, p],
            "nosa_step": [vp, i32, p, p, p, p],
            "nosa_step_host": [vp, i32, p, p, p, p],
            "nosa_step_host_all": [vp, p, p, p, p],
            "nosa_sync": [vp],
            "nosa_forecast_select": [vp, i32, p],
            "nosa_step_forecast": [vp, i32, p, p, p, p, p, i32],
            "nosa_forecast_join": [vp],
            "nosa_dense_attend": [p, p, i32, i32, i32, i32, ctypes.c_float, p, p, ctypes.c_size_t, vp],
            "nosa_dense_scratch_bytes": [i32, i32],
            "nosa_step_plan": [vp, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)],
            "nosa_prefill": [vp, i32, p, p, p, i32, p, p, ctypes.c_size_t],
            "nosa_prefill_scratch_bytes": [vp, i32],
            "nosa_reset_state": [vp],
            "nosa_context_length": [vp, i32, ctypes.POINTER(ctypes.c_int32)],
            "nosa_get_stats": [vp, ctypes.POINTER(nosa_stats)],
            "nosa_reset_stats": [vp],
            "nosa_debug_scores": [vp, i32, p, p],
            "nosa_export_state": [vp, i32, ctypes.POINTER(nosa_state_view)],
            "nosa_attend_noalloc": [p, p, p, p, p, i32, i32, i32, i32, ctypes.c_float, p, p, vp],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.nosa_status_string.argtypes = [ctypes.c_int]
        L.nosa_status_string.restype = ctypes.c_char_p
        L.nosa_dense_scratch_bytes.restype = ctypes.c_size_t
        L.nosa_prefill_scratch_bytes.restype = ctypes.c_size_t
        _lib = L
    return _lib


def _string(status: int) -> str:
    try:
        return lib().nosa_status_string(status).decode()
    except Exception:  # noqa: BLE001 - message only
        return "?"


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _check(st: int, where: str):
    if st != NOSA_OK:
        raise NosaError(st, where)


def make_config(*, num_layers, batch, num_q_heads, num_kv_heads, k_q, k_e, window_tokens, max_context,
                head_dim=128, block_size=64, cmp_kernel=32, cmp_stride=16, sink_blocks=1, evict_hidden=128,
                gather_ctas=0, softmax_scale=0.0, flags=0, score_ctas=0, attend_blocks_per_cta=0,
                attend_merge=0, decode_cluster=0, decode_teams=0, decode_stages=0,
                forecast_streams=0, cache_slots=0) -> nosa_config:
    return nosa_config(ctypes.sizeof(nosa_config), num_layers, batch, num_q_heads, num_kv_heads, head_dim,
                       block_size, cmp_kernel, cmp_stride, k_q, k_e, sink_blocks, window_tokens, max_context,
                       evict_hidden, gather_ctas, softmax_scale, flags, score_ctas, attend_blocks_per_cta,
                       attend_merge, decode_cluster, decode_teams, decode_stages, forecast_streams, cache_slots)


# ------------------------------------------------------------------ entry points
def nosa_status_string(status: int) -> str:
    return _string(status)


def nosa_validate_config(cfg: nosa_config) -> int:
    return lib().nosa_validate_config(ctypes.byref(cfg))


def nosa_query_sizes(cfg: nosa_config) -> nosa_sizes:
    out = nosa_sizes()
    _check(lib().nosa_query_sizes(ctypes.byref(cfg), ctypes.byref(out)), "nosa_query_sizes")
    return out


def nosa_create(cfg: nosa_config, stream=0) -> int:
    h = ctypes.c_void_p()
    _check(lib().nosa_create(ctypes.byref(cfg), stream or None, ctypes.byref(h)), "nosa_create")
    return h.value


def nosa_destroy(ctx) -> None:
    _check(lib().nosa_destroy(ctx), "nosa_destroy")


def nosa_set_stream(ctx, stream) -> None:
    _check(lib().nosa_set_stream(ctx, stream or None), "nosa_set_stream")


def nosa_set_eviction_head(ctx, layer, W1, W2) -> None:
    _check(lib().nosa_set_eviction_head(ctx, layer, _ptr(W1), _ptr(W2)), "nosa_set_eviction_head")


def nosa_append_kv(ctx, layer, k, v, n_tokens, src_is_host=False) -> None:
    _check(lib().nosa_append_kv(ctx, layer, _ptr(k), _ptr(v), n_tokens, int(bool(src_is_host))), "nosa_append_kv")


def nosa_select(ctx, layer, q, sel_out=None, nfetch_out=None) -> None:
    _check(lib().nosa_select(ctx, layer, _ptr(q), _ptr(sel_out), _ptr(nfetch_out)), "nosa_select")


def nosa_fetch(ctx, layer) -> None:
    _check(lib().nosa_fetch(ctx, layer), "nosa_fetch")


def nosa_attend(ctx, layer, q, out) -> None:
    _check(lib().nosa_attend(ctx, layer, _ptr(q), _ptr(out)), "nosa_attend")


def nosa_step(ctx, layer, q, k_new, v_new, out) -> None:
    _check(lib().nosa_step(ctx, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out)), "nosa_step")


def nosa_step_host(ctx, layer, q, k_new, v_new, out) -> None:
    _check(lib().nosa_step_host(ctx, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out)), "nosa_step_host")


def nosa_step_host_all(ctx, q, k_new, v_new, out) -> None:
    """Every layer's step from host buffers: q/out [L][B][Hq][d], k_new/v_new [L][B][Hkv][d]."""
    _check(lib().nosa_step_host_all(ctx, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out)), "nosa_step_host_all")


def nosa_forecast_select(ctx, layer, f) -> None:
    _check(lib().nosa_forecast_select(ctx, layer, _ptr(f)), "nosa_forecast_select")


def nosa_step_forecast(ctx, layer, q, k_new, v_new, out, f_next=None, next_layer=0) -> None:
    _check(lib().nosa_step_forecast(ctx, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out),
                                    _ptr(f_next) if f_next is not None else None, next_layer),
           "nosa_step_forecast")


def nosa_forecast_join(ctx) -> None:
    _check(lib().nosa_forecast_join(ctx), "nosa_forecast_join")


def nosa_dense_scratch_bytes(units, context_len) -> int:
    return int(lib().nosa_dense_scratch_bytes(units, context_len))


def nosa_dense_attend(q, kv, units, group, max_blocks, context_len, out, scratch, scratch_bytes,
                      softmax_scale=0.0, stream=0) -> None:
    """Dense decode attention over a device KV store [units][max_blocks][2][64][d] (see include/nosa.h)."""
    _check(lib().nosa_dense_attend(_ptr(q), _ptr(kv), units, group, max_blocks, context_len, softmax_scale,
                                   _ptr(out), _ptr(scratch), scratch_bytes, stream), "nosa_dense_attend")


def nosa_prefill_scratch_bytes(ctx, n_tokens) -> int:
    return int(lib().nosa_prefill_scratch_bytes(ctx, n_tokens))


def nosa_prefill(ctx, layer, q, k, v, n_tokens, out, scratch, scratch_bytes) -> None:
    """NOSA_S sparse prefill of an empty layer: q/out [B][Hq][n][d], k/v [B][Hkv][n][d] (see include/nosa.h)."""
    _check(lib().nosa_prefill(ctx, layer, _ptr(q), _ptr(k), _ptr(v), n_tokens, _ptr(out), _ptr(scratch),
                              scratch_bytes), "nosa_prefill")


def nosa_step_plan(ctx):
    """(kernels per layer of nosa_step: 1 fused or 3, cluster size of the fused kernel or 0)."""
    k, c = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().nosa_step_plan(ctx, ctypes.byref(k), ctypes.byref(c)), "nosa_step_plan")
    return k.value, c.value


def nosa_sync(ctx) -> int:
    """Returns the status (a latched device-side error is reported, not raised)."""
    return lib().nosa_sync(ctx)


def nosa_reset_state(ctx) -> None:
    _check(lib().nosa_reset_state(ctx), "nosa_reset_state")


def nosa_context_length(ctx, layer) -> int:
    t = ctypes.c_int32()
    _check(lib().nosa_context_length(ctx, layer, ctypes.byref(t)), "nosa_context_length")
    return t.value


def nosa_get_stats(ctx) -> nosa_stats:
    out = nosa_stats()
    _check(lib().nosa_get_stats(ctx, ctypes.byref(out)), "nosa_get_stats")
    return out


def nosa_reset_stats(ctx) -> None:
    _check(lib().nosa_reset_stats(ctx), "nosa_reset_stats")


def nosa_debug_scores(ctx, layer, sq_blk=None, se_blk=None) -> None:
    _check(lib().nosa_debug_scores(ctx, layer, _ptr(sq_blk), _ptr(se_blk)), "nosa_debug_scores")


def nosa_export_state(ctx, layer, **arrays) -> None:
    """Keyword arrays (host numpy) named as the fields of nosa_state_view."""
    view = nosa_state_view(**{k: _ptr(v) for k, v in arrays.items()})
    _check(lib().nosa_export_state(ctx, layer, ctypes.byref(view)), "nosa_export_state")


def nosa_attend_noalloc(q, cache, sel, sel_slot, n_sel, units, group, cache_slots, context_len, out,
                        softmax_scale=0.0, err_out=None, stream=0) -> None:
    """Attention over a caller-owned block cache without any device allocation (see include/nosa.h).
    err_out: optional device int32 that receives the call's device-side error bits."""
    _check(lib().nosa_attend_noalloc(_ptr(q), _ptr(cache), _ptr(sel), _ptr(sel_slot), _ptr(n_sel), units, group,
                                     cache_slots, context_len, softmax_scale, _ptr(out), _ptr(err_out),
                                     stream or None),
           "nosa_attend_noalloc")
