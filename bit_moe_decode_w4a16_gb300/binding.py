"""ctypes binding of libbitmoe.so: argument marshalling only.

Every function here has the name of the C entry point it calls (see
include/bitmoe.h) and does nothing but convert arguments: torch tensors to
device pointers, torch streams to cudaStream_t handles, and a non-OK status
to a ``BitMoeError``.  All of the decode step's work runs in the CUDA
library; when the library has not been built this module raises on import
of the library rather than running anything else in its place.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libbitmoe.so")

BM_OK = 0
STATUS_NAMES = {
    0: "BM_OK", 1: "BM_ERR_INVALID_ARG", 2: "BM_ERR_CTX_CAP", 3: "BM_ERR_NO_SLOT",
    4: "BM_ERR_SLOT_FREE", 5: "BM_ERR_CUDA", 6: "BM_ERR_OOM", 7: "BM_ERR_NOT_READY",
    8: "BM_ERR_DEVICE_CHECK", 9: "BM_ERR_UNSUPPORTED",
}
POLICY_AUTO, POLICY_SIMT, POLICY_TC, POLICY_MMA = 0, 1, 2, 3


class BitMoeError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


class bm_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("hidden", "q_heads", "kv_heads", "head_dim", "experts", "top_k",
                                            "ffn", "group", "vocab", "layers")] + \
               [("rope_base", ctypes.c_float), ("rms_eps", ctypes.c_float)] + \
               [(n, ctypes.c_int) for n in ("max_streams", "ctx_cap", "renorm_topk", "kernel_policy",
                                            "use_graph", "prefill_tc", "persistent_step")]


_P = ctypes.c_void_p


class bm_layer_weights(ctypes.Structure):
    _fields_ = [(n, _P) for n in ("wqkv", "wqkv_s", "wo", "wo_s", "wr", "wg", "wg_s", "wu", "wu_s",
                                  "wd", "wd_s", "attn_norm", "ffn_norm")]


class bm_moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("experts", "top_k", "hidden", "ffn", "group", "renorm_topk")] + \
               [(n, _P) for n in ("wr", "wg", "wg_s", "wu", "wu_s", "wd", "wd_s")]


class bm_kernel_profile(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 24), ("launches", ctypes.c_int), ("ms", ctypes.c_float),
                ("bytes", ctypes.c_double), ("flops", ctypes.c_double)]


class bm_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("steps", "tokens", "graph_launches", "graph_captures",
                                               "kernel_launches", "kernels_per_step")] + \
               [(n, ctypes.c_size_t) for n in ("weight_bytes", "arena_bytes", "scratch_bytes")]


_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libbitmoe.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        I, V, S, SZ = ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        PI = ctypes.POINTER(ctypes.c_int)
        sig = {
            "bm_last_error": ([], ctypes.c_char_p),
            "bm_engine_create": ([ctypes.POINTER(bm_config), ctypes.POINTER(V)], S),
            "bm_engine_destroy": ([V], None),
            "bm_engine_set_layer": ([V, I, ctypes.POINTER(bm_layer_weights), V], S),
            "bm_engine_set_embeddings": ([V, V, V, V, V], S),
            "bm_engine_sync": ([V, V], S),
            "bm_engine_stats": ([V, ctypes.POINTER(bm_stats)], S),
            "bm_engine_kernel_family": ([V], I),
            "kv_slot_seed": ([V, V, V, I, PI, V], S),
            "kv_slot_append": ([V, I, V, V, V, I, V], S),
            "kv_slot_attend": ([V, I, V, V, V, I, V], S),
            "kv_slot_advance": ([V, V, I, V], S),
            "kv_slot_release": ([V, I], S),
            "kv_slot_length": ([V, I, PI], S),
            "kv_slot_read": ([V, I, I, I, V, V, V], S),
            "w4_gemm_batched": ([V, V, V, V, V, I, I, I, I, V], S),
            "bm_moe_workspace_bytes": ([I, I, I, I, I], SZ),
            "bm_w4_repack_tc": ([V, V, I, I, I, V, V, V], S),
            "w4_gemm_batched_tc": ([V, V, V, V, V, I, I, I, I, V], S),
            "bm_w4_repack_mma": ([V, V, I, I, I, V, V, V], S),
            "w4_gemm_batched_mma": ([V, V, V, V, V, I, I, I, I, V], S),
            "w4_gemm_prompt_tc": ([V, V, V, V, V, I, I, I, I, V], S),
            "moe_grouped_w4": ([ctypes.POINTER(bm_moe_weights), V, V, V, V, V, I, V, SZ, V], S),
            "moe_grouped_w4_noalloc": ([ctypes.POINTER(bm_moe_weights), V, V, V, V, V, I, V], S),
            "bm_moe_noalloc_max_bytes": ([], SZ),
            "decode_step": ([V, I, V, V, V, V, V], S),
            "kv_slot_prefill": ([V, I, I, V, V, V, V], S),
            "bm_engine_profile_step": ([V, I, V, V, V, ctypes.POINTER(bm_kernel_profile), I, PI, V], S),
            "bm_w4_quantize": ([V, I, I, I, V, V, V], S),
            "bm_engine_moe": ([V, I, V, V, V, V, I, V], S),
            "bm_probe_tcgen05_mma": ([I, I, I, I, I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)], S),
            "bm_engine_attention": ([V, I, V, V, V, I, V], S),
            "bm_engine_read_hidden": ([V, I, V, V], S),
            "bm_engine_test_drop_expert_item": ([V, I], S),
            "bm_engine_test_drop_persist_unit": ([V, I], S),
            "bm_engine_set_persistent_step": ([V, I], S),
            "bm_slot_map_create": ([I, I, ctypes.POINTER(V)], S),
            "bm_slot_map_destroy": ([V], None),
            "bm_slot_map_acquire": ([V, I, PI], S),
            "bm_slot_map_release": ([V, I], S),
            "bm_slot_map_check_batch": ([V, V, I], S),
            "bm_slot_map_advance": ([V, V, I], S),
            "bm_slot_map_length": ([V, I, PI], S),
            "bm_slot_map_active_count": ([V], I),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def last_error():
    return lib().bm_last_error().decode()


def _check(status):
    if status != BM_OK:
        raise BitMoeError(status, last_error())
    return status


def ptr(x):
    """Device/host address of a torch tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, ctypes.Array):
        return ctypes.addressof(x)
    raise TypeError(f"cannot take the address of {type(x)}")


def stream_handle(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _i32_array(values):
    arr = (ctypes.c_int32 * len(values))(*[int(v) for v in values])
    return arr


# --------------------------------------------------------------- engine

def bm_engine_create(cfg):
    """cfg: a bm_config or a dict of its fields.  Returns the engine handle."""
    if isinstance(cfg, dict):
        c = bm_config()
        for k, v in cfg.items():
            setattr(c, k, v)
        cfg = c
    h = ctypes.c_void_p()
    _check(lib().bm_engine_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h.value


def bm_engine_destroy(e):
    lib().bm_engine_destroy(e)


def bm_engine_set_layer(e, layer, weights, stream=None):
    """weights: dict with the bm_layer_weights field names -> tensors/addresses."""
    w = bm_layer_weights(**{k: ptr(weights.get(k)) for k, _ in bm_layer_weights._fields_})
    _check(lib().bm_engine_set_layer(e, layer, ctypes.byref(w), stream_handle(stream)))


def bm_engine_set_embeddings(e, embed, lm_head, final_norm=None, stream=None):
    _check(lib().bm_engine_set_embeddings(e, ptr(embed), ptr(lm_head), ptr(final_norm), stream_handle(stream)))


def bm_engine_sync(e, stream=None):
    _check(lib().bm_engine_sync(e, stream_handle(stream)))


def bm_engine_stats(e):
    s = bm_stats()
    _check(lib().bm_engine_stats(e, ctypes.byref(s)))
    return {k: getattr(s, k) for k, _ in bm_stats._fields_}


def bm_engine_kernel_family(e):
    return lib().bm_engine_kernel_family(e)


# --------------------------------------------------------------- slots

def kv_slot_seed(e, K, V, length, stream=None):
    slot = ctypes.c_int(-1)
    _check(lib().kv_slot_seed(e, ptr(K), ptr(V), int(length), ctypes.byref(slot), stream_handle(stream)))
    return slot.value


def kv_slot_append(e, layer, slots, Knew, Vnew, stream=None):
    arr = _i32_array(slots)
    _check(lib().kv_slot_append(e, layer, ctypes.addressof(arr), ptr(Knew), ptr(Vnew), len(slots),
                                stream_handle(stream)))


def kv_slot_attend(e, layer, slots, Q, O, stream=None):
    arr = _i32_array(slots)
    _check(lib().kv_slot_attend(e, layer, ctypes.addressof(arr), ptr(Q), ptr(O), len(slots),
                                stream_handle(stream)))


def kv_slot_advance(e, slots, stream=None):
    arr = _i32_array(slots)
    _check(lib().kv_slot_advance(e, ctypes.addressof(arr), len(slots), stream_handle(stream)))


def kv_slot_release(e, slot):
    _check(lib().kv_slot_release(e, int(slot)))


def kv_slot_length(e, slot):
    n = ctypes.c_int(0)
    _check(lib().kv_slot_length(e, int(slot), ctypes.byref(n)))
    return n.value


def kv_slot_read(e, layer, slot, count, K_out, V_out, stream=None):
    _check(lib().kv_slot_read(e, layer, slot, count, ptr(K_out), ptr(V_out), stream_handle(stream)))


# --------------------------------------------------------------- ops

def w4_gemm_batched(W, S, X, Y, R, M, N, K, g, stream=None):
    _check(lib().w4_gemm_batched(ptr(W), ptr(S), ptr(X), ptr(Y), ptr(R), M, N, K, g, stream_handle(stream)))


def bm_w4_repack_tc(W, S, N, K, g, Wtc, Stc, stream=None):
    _check(lib().bm_w4_repack_tc(ptr(W), ptr(S), N, K, g, ptr(Wtc), ptr(Stc), stream_handle(stream)))


def w4_gemm_batched_tc(Wtc, Stc, X, Y, R, M, N, K, g, stream=None):
    _check(lib().w4_gemm_batched_tc(ptr(Wtc), ptr(Stc), ptr(X), ptr(Y), ptr(R), M, N, K, g, stream_handle(stream)))


def bm_w4_repack_mma(W, S, N, K, g, Wm, Sm, stream=None):
    _check(lib().bm_w4_repack_mma(ptr(W), ptr(S), N, K, g, ptr(Wm), ptr(Sm), stream_handle(stream)))


def w4_gemm_batched_mma(Wm, Sm, X, Y, R, M, N, K, g, stream=None):
    _check(lib().w4_gemm_batched_mma(ptr(Wm), ptr(Sm), ptr(X), ptr(Y), ptr(R), M, N, K, g, stream_handle(stream)))


def w4_gemm_prompt_tc(Wm, Sm, X16, Y, R, M, N, K, g, stream=None):
    _check(lib().w4_gemm_prompt_tc(ptr(Wm), ptr(Sm), ptr(X16), ptr(Y), ptr(R), M, N, K, g, stream_handle(stream)))


def bm_moe_workspace_bytes(B, experts, top_k, hidden, ffn):
    return lib().bm_moe_workspace_bytes(B, experts, top_k, hidden, ffn)


def moe_grouped_w4(weights, X, Hres, Y, topk_ids, topk_w, B, ws, ws_bytes, stream=None):
    """weights: dict with bm_moe_weights field names."""
    w = bm_moe_weights(**{k: (weights[k] if t is ctypes.c_int else ptr(weights[k]))
                          for k, t in bm_moe_weights._fields_})
    _check(lib().moe_grouped_w4(ctypes.byref(w), ptr(X), ptr(Hres), ptr(Y), ptr(topk_ids), ptr(topk_w), B,
                                ptr(ws), ws_bytes, stream_handle(stream)))


def moe_grouped_w4_noalloc(weights, X, Hres, Y, topk_ids, topk_w, B, stream=None):
    """The grouped expert op with the library's built-in workspace (no
    allocation); weights as for moe_grouped_w4."""
    w = bm_moe_weights(**{k: (weights[k] if t is ctypes.c_int else ptr(weights[k]))
                          for k, t in bm_moe_weights._fields_})
    _check(lib().moe_grouped_w4_noalloc(ctypes.byref(w), ptr(X), ptr(Hres), ptr(Y), ptr(topk_ids), ptr(topk_w), B,
                                        stream_handle(stream)))


def bm_moe_noalloc_max_bytes():
    return lib().bm_moe_noalloc_max_bytes()


def decode_step(e, slots, tokens, next_tokens, logits=None, stream=None):
    """slots: host sequence of ints; tokens / next_tokens: host or device int32."""
    arr = _i32_array(slots)
    _check(lib().decode_step(e, len(slots), ctypes.addressof(arr), ptr(tokens), ptr(next_tokens), ptr(logits),
                             stream_handle(stream)))


def kv_slot_prefill(e, slot, tokens, next_token, logits=None, stream=None):
    """tokens: host or device int32 [n]; next_token: host or device int32 [1]."""
    _check(lib().kv_slot_prefill(e, int(slot), int(tokens.numel()), ptr(tokens), ptr(next_token), ptr(logits),
                                 stream_handle(stream)))


def bm_engine_profile_step(e, slots, tokens, next_tokens, stream=None):
    """One eager decode step with per-kernel CUDA-event times; returns a list
    of dicts (name, launches, ms, bytes, flops), one per kernel class."""
    arr = _i32_array(slots)
    out = (bm_kernel_profile * 32)()
    n = ctypes.c_int(0)
    _check(lib().bm_engine_profile_step(e, len(slots), ctypes.addressof(arr), ptr(tokens), ptr(next_tokens), out,
                                        32, ctypes.byref(n), stream_handle(stream)))
    return [{"name": out[i].name.decode(), "launches": out[i].launches, "ms": out[i].ms,
             "bytes": out[i].bytes, "flops": out[i].flops} for i in range(n.value)]


def bm_engine_moe(e, layer, h, y, topk_ids=None, topk_w=None, stream=None):
    """The decode step's routing and expert kernels on one layer; h, y: bf16 [B][H]."""
    _check(lib().bm_engine_moe(e, layer, ptr(h), ptr(y), ptr(topk_ids), ptr(topk_w), int(h.shape[0]),
                               stream_handle(stream)))


def bm_engine_attention(e, layer, slots, qkv, out, stream=None):
    """The decode step's fused attention on one layer; qkv: bf16 rows, out: fp16 [B][qh][d]."""
    arr = _i32_array(slots)
    _check(lib().bm_engine_attention(e, layer, ctypes.addressof(arr), ptr(qkv), ptr(out), len(slots),
                                     stream_handle(stream)))


def bm_engine_read_hidden(e, B, out, stream=None):
    _check(lib().bm_engine_read_hidden(e, int(B), ptr(out), stream_handle(stream)))


def bm_engine_test_drop_expert_item(e, item):
    _check(lib().bm_engine_test_drop_expert_item(e, int(item)))


def bm_engine_set_persistent_step(e, enable):
    _check(lib().bm_engine_set_persistent_step(e, int(enable)))


def bm_engine_test_drop_persist_unit(e, unit):
    _check(lib().bm_engine_test_drop_persist_unit(e, int(unit)))


def bm_probe_tcgen05_mma(n, a_in_tmem, swizzle128, iters, roundtrip=0):
    """SM cycles per tcgen05 MMA (M 128 x N n x K 16): (to issue, to complete)."""
    a, b = ctypes.c_double(0), ctypes.c_double(0)
    _check(lib().bm_probe_tcgen05_mma(int(n), int(a_in_tmem), int(swizzle128), int(iters), int(roundtrip),
                                      ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def bm_w4_quantize(W, N, K, g, packed, scales, stream=None):
    _check(lib().bm_w4_quantize(ptr(W), N, K, g, ptr(packed), ptr(scales), stream_handle(stream)))


# --------------------------------------------------------------- host slot map

def bm_slot_map_create(max_streams, ctx_cap):
    h = ctypes.c_void_p()
    _check(lib().bm_slot_map_create(max_streams, ctx_cap, ctypes.byref(h)))
    return h.value


def bm_slot_map_destroy(m):
    lib().bm_slot_map_destroy(m)


def bm_slot_map_acquire(m, length):
    s = ctypes.c_int(-1)
    _check(lib().bm_slot_map_acquire(m, int(length), ctypes.byref(s)))
    return s.value


def bm_slot_map_release(m, slot):
    _check(lib().bm_slot_map_release(m, int(slot)))


def bm_slot_map_check_batch(m, slots):
    arr = _i32_array(slots)
    _check(lib().bm_slot_map_check_batch(m, ctypes.addressof(arr), len(slots)))


def bm_slot_map_advance(m, slots):
    arr = _i32_array(slots)
    _check(lib().bm_slot_map_advance(m, ctypes.addressof(arr), len(slots)))


def bm_slot_map_length(m, slot):
    n = ctypes.c_int(0)
    _check(lib().bm_slot_map_length(m, int(slot), ctypes.byref(n)))
    return n.value


def bm_slot_map_active_count(m):
    return lib().bm_slot_map_active_count(m)
