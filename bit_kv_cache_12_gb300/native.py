"""ctypes binding of libkvint2 (argument marshalling only).

The module-level functions carry the C names of ``include/kvint2.h`` and take
either integers (raw pointers) or torch tensors (their ``data_ptr()``).  Every
step of the hot path runs in the CUDA library; there is no fallback: if the
library is missing the first call raises.

``KVPool`` is a small convenience owner of a pool handle used by the tests and
``bench.py``.
"""

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libkvint2.so")

KV_OK = 0
KV_ERR_INVALID_ARG = 1
KV_ERR_OOM = 2
KV_ERR_CUDA = 3
KV_ERR_UNSUPPORTED = 4
KV_ERR_DEVICE = 5
KV_ERR_TIMEOUT = 6
KV_ERR_SCRATCH_LIMIT = 7
STATUS_NAMES = {0: "KV_OK", 1: "KV_ERR_INVALID_ARG", 2: "KV_ERR_OOM", 3: "KV_ERR_CUDA",
                4: "KV_ERR_UNSUPPORTED", 5: "KV_ERR_DEVICE", 6: "KV_ERR_TIMEOUT",
                7: "KV_ERR_SCRATCH_LIMIT"}
KV_NOALLOC_SCRATCH_BYTES = 16 << 20
KV_POOL_INT2_3TIER = 0
KV_POOL_BF16 = 1


class KvPoolConfig(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("sink_tokens", ctypes.c_int32),
                ("recent_tokens", ctypes.c_int32), ("max_seqs", ctypes.c_int32),
                ("num_pages", ctypes.c_int64)]


class KvPoolLayout(ctypes.Structure):
    _fields_ = [("hist", ctypes.c_void_p), ("hist_layer_stride", ctypes.c_size_t),
                ("hist_page_stride", ctypes.c_size_t), ("hist_head_stride", ctypes.c_size_t),
                ("tile_bytes", ctypes.c_size_t), ("sink_k", ctypes.c_void_p),
                ("sink_v", ctypes.c_void_p), ("recent_k", ctypes.c_void_p),
                ("recent_v", ctypes.c_void_p), ("tier_layer_stride", ctypes.c_size_t),
                ("recent_layer_stride", ctypes.c_size_t), ("bf16_k", ctypes.c_void_p),
                ("bf16_v", ctypes.c_void_p), ("bf16_layer_stride", ctypes.c_size_t)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SIG = {
    "kv_pool_create": (_I32, [ctypes.POINTER(KvPoolConfig), _P, ctypes.POINTER(_P)]),
    "kv_pool_destroy": (_I32, [_P]),
    "kv_pool_set_rotation": (_I32, [_P, _I32, _P, _P, _P, _P, _P]),
    "kv_pool_get_layout": (_I32, [_P, _I32, ctypes.POINTER(KvPoolLayout)]),
    "kv_pool_get_error": (_I32, [_P, ctypes.POINTER(_I32)]),
    "kv_store_tier": (_I32, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P]),
    "kv_quantize_pack_f32": (_I32, [_P, _I32, _I32, _I64, _P, _P, _P, _P]),
    "kv_append_quantize": (_I32, [_P, _I32, _I32, _P, _P, _P, _P, _P, _I32, _I32, _P]),
    "kv_append_step": (_I32, [_P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _I32, _P]),
    "kv_decode_multi_workspace_bytes": (ctypes.c_size_t, [_P, _I32, _I32, _I32]),
    "kv_decode_attention_multi": (_I32, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _I32, _I32,
                                         ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P]),
    "kv_decode_workspace_bytes": (ctypes.c_size_t, [_P, _I32, _I32]),
    "kv_decode_attention": (_I32, [_P, _I32, _I32, _P, _P, _P, _P, _P, _P, _I32, _I32,
                                   ctypes.c_float, _P, _P, ctypes.c_size_t, _P]),
    "kv_decode_attention_noalloc": (_I32, [_P, _I32, _I32, _P, _P, _P, _P, _P, _P, _I32, _I32,
                                           ctypes.c_float, _P, _P]),
    "kv_debug_stall_first_copy": (_I32, [_P, _I32, _I32]),
    "kv_append_bf16": (_I32, [_P, _I32, _I32, _P, _P, _P, _P, _P, _I32, _I32, _P]),
    "kv_decode_attention_bf16": (_I32, [_P, _I32, _I32, _P, _P, _P, _I32, _I32,
                                        ctypes.c_float, _P, _P, ctypes.c_size_t, _P]),
}

_lib = None


def lib():
    """Load libkvint2.so (build it with ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkvint2.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIG.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class KVError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


def _check(fn, st):
    if st != KV_OK:
        raise KVError(fn, st)


# ---- C-named wrappers -----------------------------------------------------

def kv_pool_create(cfg, stream=None):
    h = _P()
    _check("kv_pool_create", lib().kv_pool_create(ctypes.byref(cfg), _stream(stream), ctypes.byref(h)))
    return h.value


def kv_pool_destroy(pool):
    _check("kv_pool_destroy", lib().kv_pool_destroy(pool))


def kv_pool_set_rotation(pool, layer, R_k, R_v, clip_k, clip_v, stream=None):
    _check("kv_pool_set_rotation", lib().kv_pool_set_rotation(
        pool, layer, _ptr(R_k), _ptr(R_v), _ptr(clip_k), _ptr(clip_v), _stream(stream)))


def kv_pool_get_layout(pool, layer):
    out = KvPoolLayout()
    _check("kv_pool_get_layout", lib().kv_pool_get_layout(pool, layer, ctypes.byref(out)))
    return out


def kv_pool_get_error(pool):
    code = _I32(0)
    st = lib().kv_pool_get_error(pool, ctypes.byref(code))
    if st not in (KV_OK, KV_ERR_DEVICE):
        raise KVError("kv_pool_get_error", st)
    return code.value


def kv_store_tier(pool, layer, tier, n_rows, k, v, seq, slot, stream=None):
    _check("kv_store_tier", lib().kv_store_tier(pool, layer, tier, n_rows, _ptr(k), _ptr(v),
                                                _ptr(seq), _ptr(slot), _stream(stream)))


def kv_quantize_pack_f32(pool, layer, tensor, n_rows, x_rot, codes, scale_zero, stream=None):
    _check("kv_quantize_pack_f32", lib().kv_quantize_pack_f32(
        pool, layer, tensor, n_rows, _ptr(x_rot), _ptr(codes), _ptr(scale_zero), _stream(stream)))


def kv_append_quantize(pool, layer, n_seqs, k, v, cu_tokens, hist_start, page_table,
                       max_pages_per_seq, max_tokens_per_seq, stream=None):
    _check("kv_append_quantize", lib().kv_append_quantize(
        pool, layer, n_seqs, _ptr(k), _ptr(v), _ptr(cu_tokens), _ptr(hist_start),
        _ptr(page_table), max_pages_per_seq, max_tokens_per_seq, _stream(stream)))


def kv_append_step(pool, layer, B, k_new, v_new, sink_len, hist_len, recent_len, recent_start,
                   page_table, max_pages_per_seq, stream=None):
    _check("kv_append_step", lib().kv_append_step(
        pool, layer, B, _ptr(k_new), _ptr(v_new), _ptr(sink_len), _ptr(hist_len), _ptr(recent_len),
        _ptr(recent_start), _ptr(page_table), max_pages_per_seq, _stream(stream)))


def kv_decode_multi_workspace_bytes(pool, B, T, max_hist_len):
    return lib().kv_decode_multi_workspace_bytes(pool, B, T, max_hist_len)


def kv_decode_attention_multi(pool, layer, B, T, q, sink_len, hist_len, recent_len, recent_start,
                              page_table, max_pages_per_seq, max_hist_len, softmax_scale, out,
                              lse, workspace, workspace_bytes, stream=None):
    _check("kv_decode_attention_multi", lib().kv_decode_attention_multi(
        pool, layer, B, T, _ptr(q), _ptr(sink_len), _ptr(hist_len), _ptr(recent_len),
        _ptr(recent_start), _ptr(page_table), max_pages_per_seq, max_hist_len, softmax_scale,
        _ptr(out), _ptr(lse), _ptr(workspace), workspace_bytes, _stream(stream)))


def kv_decode_workspace_bytes(pool, B, max_len):
    return lib().kv_decode_workspace_bytes(pool, B, max_len)


def kv_decode_attention(pool, layer, B, q, sink_len, hist_len, recent_len, recent_start,
                        page_table, max_pages_per_seq, max_hist_len, softmax_scale, out,
                        workspace, workspace_bytes, stream=None):
    _check("kv_decode_attention", lib().kv_decode_attention(
        pool, layer, B, _ptr(q), _ptr(sink_len), _ptr(hist_len), _ptr(recent_len),
        _ptr(recent_start), _ptr(page_table), max_pages_per_seq, max_hist_len,
        float(softmax_scale), _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream)))


def kv_decode_attention_noalloc(pool, layer, B, q, sink_len, hist_len, recent_len, recent_start,
                                page_table, max_pages_per_seq, max_hist_len, softmax_scale, out,
                                stream=None):
    """kv_decode_attention without a workspace: for callers that cannot
    allocate device memory; uses the library's fixed 16 MiB device buffer."""
    _check("kv_decode_attention_noalloc", lib().kv_decode_attention_noalloc(
        pool, layer, B, _ptr(q), _ptr(sink_len), _ptr(hist_len), _ptr(recent_len),
        _ptr(recent_start), _ptr(page_table), max_pages_per_seq, max_hist_len,
        float(softmax_scale), _ptr(out), _stream(stream)))


def kv_debug_stall_first_copy(pool, enable, max_polls=0):
    """Test hook: later decodes of this pool make one bounded wait run out."""
    _check("kv_debug_stall_first_copy", lib().kv_debug_stall_first_copy(pool, int(enable),
                                                                         int(max_polls)))


def kv_append_bf16(pool, layer, n_seqs, k, v, cu_tokens, start_pos, page_table,
                   max_pages_per_seq, max_tokens_per_seq, stream=None):
    _check("kv_append_bf16", lib().kv_append_bf16(
        pool, layer, n_seqs, _ptr(k), _ptr(v), _ptr(cu_tokens), _ptr(start_pos),
        _ptr(page_table), max_pages_per_seq, max_tokens_per_seq, _stream(stream)))


def kv_decode_attention_bf16(pool, layer, B, q, seq_len, page_table, max_pages_per_seq,
                             max_seq_len, softmax_scale, out, workspace, workspace_bytes,
                             stream=None):
    _check("kv_decode_attention_bf16", lib().kv_decode_attention_bf16(
        pool, layer, B, _ptr(q), _ptr(seq_len), _ptr(page_table), max_pages_per_seq,
        max_seq_len, float(softmax_scale), _ptr(out), _ptr(workspace), workspace_bytes,
        _stream(stream)))


# ---- device-memory views (zero copy) ---------------------------------------

class _CudaArray:
    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(int(s) for s in shape),
                                         "typestr": typestr, "data": (int(ptr), False),
                                         "version": 3, "strides": None}


def device_view(ptr, shape, dtype):
    """A torch tensor aliasing pool memory (uint8 or bf16 via int16)."""
    import torch
    if dtype == torch.uint8:
        return torch.as_tensor(_CudaArray(ptr, shape, "|u1"), device="cuda")
    if dtype == torch.bfloat16:
        return torch.as_tensor(_CudaArray(ptr, shape, "<i2"), device="cuda").view(torch.bfloat16)
    raise ValueError(dtype)


class KVPool:
    """Owner of one pool handle with a few torch-friendly helpers."""

    def __init__(self, kind, num_layers, num_q_heads, num_kv_heads, page_size, num_pages,
                 max_seqs, group_size=128, sink_tokens=64, recent_tokens=256, stream=None):
        self.cfg = KvPoolConfig(kind, num_layers, num_q_heads, num_kv_heads, 128, page_size,
                                group_size, sink_tokens, recent_tokens, max_seqs, num_pages)
        self.handle = kv_pool_create(self.cfg, stream)

    def close(self):
        if self.handle:
            kv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def layout(self, layer=0):
        return kv_pool_get_layout(self.handle, layer)

    def hist_view(self, layer=0):
        """uint8 [num_pages, Hkv, page_size/16 * tile_bytes] view of the INT2 history."""
        import torch
        lay = self.layout(layer)
        c = self.cfg
        return device_view(lay.hist, (c.num_pages, c.num_kv_heads, lay.hist_head_stride), torch.uint8)

    def tier_views(self, layer=0):
        import torch
        lay = self.layout(layer)
        c = self.cfg
        s = (c.max_seqs, c.num_kv_heads, c.sink_tokens, 128)
        r = (c.max_seqs, c.num_kv_heads, c.recent_tokens, 128)
        return (device_view(lay.sink_k, s, torch.bfloat16), device_view(lay.sink_v, s, torch.bfloat16),
                device_view(lay.recent_k, r, torch.bfloat16), device_view(lay.recent_v, r, torch.bfloat16))

    def bf16_views(self, layer=0):
        import torch
        lay = self.layout(layer)
        c = self.cfg
        shp = (c.num_pages, c.num_kv_heads, c.page_size, 128)
        return (device_view(lay.bf16_k, shp, torch.bfloat16), device_view(lay.bf16_v, shp, torch.bfloat16))

    def error(self):
        return kv_pool_get_error(self.handle)
