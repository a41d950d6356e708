"""ctypes binding of ``libkvc.so`` (the C ABI in ``include/kvc.h``).

Argument marshalling only: every operation runs in the CUDA library.  Functions keep the
C names (``kvc_create``, ``kvc_append``, ...); they take torch CUDA tensors (or raw integer
device pointers) and a torch stream (default: the current stream), and raise
:class:`KvcError` on a nonzero status.  :class:`KVCache` is a small owner of one handle.

There is no fallback: if the library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libkvc.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "kvc.h")

KVC_BF16, KVC_F32 = 0, 1
KVC_OK, KVC_EINVAL, KVC_ENOMEM, KVC_ECUDA, KVC_ERANGE, KVC_EDEVICE, KVC_EUNSUPPORTED = range(7)
KVC_DEV_BAD_LENS, KVC_DEV_WAIT_TIMEOUT, KVC_DEV_BAD_BLOCK = 1, 2, 4
KVC_CACHE_PLAIN, KVC_CACHE_INT8, KVC_CACHE_FP8 = 0, 1, 2

_lib = None


class KvcError(RuntimeError):
    def __init__(self, status: int, what: str, detail: int = 0):
        self.status = status
        self.detail = detail
        name = load().kvc_status_str(status).decode()
        super().__init__(f"{what}: {name} (status {status}, detail {detail:#x})")


def load() -> ctypes.CDLL:
    """Load libkvc.so (raises OSError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise OSError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    P, I, U64, I64, U32P = (ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_int64,
                            ctypes.POINTER(ctypes.c_uint32))
    sig = {
        "kvc_create": (I, [ctypes.POINTER(P), I, I, I, I, I, I, I]),
        "kvc_destroy": (I, [P]),
        "kvc_prefill_write": (I, [P, I, P, P, I, P, P]),
        "kvc_append": (I, [P, I, P, P, P, P]),
        "kvc_decode_attn": (I, [P, I, P, P, P, P]),
        "kvc_decode_step": (I, [P, I, P, P, P, P, P, P]),
        "kvc_bytes": (U64, [P]),
        "kvc_bytes_formula": (U64, [I64] * 6),
        "kvc_payload_bytes": (U64, [P, P]),
        "kvc_layer_ptrs": (I, [P, I, ctypes.POINTER(P), ctypes.POINTER(P)]),
        "kvc_last_error": (I, [P, P, U32P]),
        "kvc_set_ctas": (I, [P, I]),
        "kvc_get_ctas": (I, [P]),
        "kvc_set_combine_mode": (I, [P, I]),
        "kvc_set_math": (I, [P, I]),
        "kvc_get_math": (I, [P]),
        "kvc_set_launch_overlap": (I, [P, I]),
        "kvc_get_launch_overlap": (I, [P]),
        "kvc_get_shape": (I, [P] + [ctypes.POINTER(I)] * 7),
        "kvc_plan_cta_of": (I, [I64, I64, I]),
        "kvc_plan_grain": (I, [I, I, I]),
        "kvc_plan_cuts": (I, [P, I, I, I, I, I, I, P]),
        "kvc_plan_stream_ctas": (I, [P, I, I, I, I, I, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I)]),
        "kvc_status_str": (ctypes.c_char_p, [I]),
        "kvc_decode_attn_noalloc": (I, [P, P, I, I, I, I, I, I, P, P, P, P, P]),
        "kvc_selftest_wait_timeout": (I, [P, P, ctypes.c_longlong, P]),
        "kvc_create_paged": (I, [ctypes.POINTER(P), I, I, I, I, I, I, I, I, I]),
        "kvc_create_rolling": (I, [ctypes.POINTER(P), I, I, I, I, I, I, I]),
        "kvc_create_quantized": (I, [ctypes.POINTER(P), I, I, I, I, I, I, I]),
        "kvc_layer_scales": (I, [P, I, ctypes.POINTER(P), ctypes.POINTER(P)]),
        "kvc_create_fp8": (I, [ctypes.POINTER(P), I, I, I, I, I, I, I]),
        "kvc_get_cache_format": (I, [P]),
        "kvc_append_multi": (I, [P, I, P, P, P, I, P]),
        "kvc_decode_attn_multi": (I, [P, I, P, P, P, I, P]),
        "kvc_decode_step_multi": (I, [P, I, P, P, P, P, P, I, P]),
        "kvc_get_window": (I, [P]),
        "kvc_paged_prefill_write": (I, [P, I, P, P, I, P, P, P]),
        "kvc_paged_append": (I, [P, I, P, P, P, P, P]),
        "kvc_paged_decode_attn": (I, [P, I, P, P, P, P, P]),
        "kvc_paged_decode_step": (I, [P, I, P, P, P, P, P, P, P]),
        "kvc_get_paged_shape": (I, [P] + [ctypes.POINTER(I)] * 3),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def header_symbols() -> list[str]:
    """Function names declared in include/kvc.h."""
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z0-9_]+)\s*\(", text)))


# ----------------------------------------------------------------------------- marshalling
def _ptr(x) -> int:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != KVC_OK:
        raise KvcError(status, what)


# ----------------------------------------------------------------------------- C names
def kvc_create(layers, B, H_q, H_kv, D, T_max, dtype) -> int:
    h = ctypes.c_void_p()
    _check(load().kvc_create(ctypes.byref(h), layers, B, H_q, H_kv, D, T_max, dtype), "kvc_create")
    return h.value


def kvc_destroy(h) -> None:
    _check(load().kvc_destroy(h), "kvc_destroy")


def kvc_prefill_write(h, layer, K, V, T_in, lens, stream=None) -> None:
    _check(load().kvc_prefill_write(h, layer, _ptr(K), _ptr(V), T_in, _ptr(lens), _stream(stream)),
           "kvc_prefill_write")


def kvc_append(h, layer, k_new, v_new, lens, stream=None) -> None:
    _check(load().kvc_append(h, layer, _ptr(k_new), _ptr(v_new), _ptr(lens), _stream(stream)),
           "kvc_append")


def kvc_decode_attn(h, layer, q, out, lens, stream=None) -> None:
    _check(load().kvc_decode_attn(h, layer, _ptr(q), _ptr(out), _ptr(lens), _stream(stream)),
           "kvc_decode_attn")


def kvc_decode_step(h, layer, q, k_new, v_new, out, lens, stream=None) -> None:
    _check(load().kvc_decode_step(h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out),
                                  _ptr(lens), _stream(stream)), "kvc_decode_step")


def kvc_append_multi(h, layer, k_new, v_new, lens, T_q, stream=None) -> None:
    _check(load().kvc_append_multi(h, layer, _ptr(k_new), _ptr(v_new), _ptr(lens), T_q, _stream(stream)),
           "kvc_append_multi")


def kvc_decode_attn_multi(h, layer, q, out, lens, T_q, stream=None) -> None:
    _check(load().kvc_decode_attn_multi(h, layer, _ptr(q), _ptr(out), _ptr(lens), T_q, _stream(stream)),
           "kvc_decode_attn_multi")


def kvc_decode_step_multi(h, layer, q, k_new, v_new, out, lens, T_q, stream=None) -> None:
    _check(load().kvc_decode_step_multi(h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out),
                                        _ptr(lens), T_q, _stream(stream)), "kvc_decode_step_multi")


def kvc_create_quantized(layers, B, H_q, H_kv, D, T_max, dtype) -> int:
    h = ctypes.c_void_p()
    _check(load().kvc_create_quantized(ctypes.byref(h), layers, B, H_q, H_kv, D, T_max, dtype),
           "kvc_create_quantized")
    return h.value


def kvc_create_fp8(layers, B, H_q, H_kv, D, T_max, dtype) -> int:
    h = ctypes.c_void_p()
    _check(load().kvc_create_fp8(ctypes.byref(h), layers, B, H_q, H_kv, D, T_max, dtype), "kvc_create_fp8")
    return h.value


def kvc_get_cache_format(h) -> int:
    return int(load().kvc_get_cache_format(h))


def kvc_layer_scales(h, layer):
    k, v = ctypes.c_void_p(), ctypes.c_void_p()
    _check(load().kvc_layer_scales(h, layer, ctypes.byref(k), ctypes.byref(v)), "kvc_layer_scales")
    return k.value, v.value


def kvc_create_rolling(layers, B, H_q, H_kv, D, window, dtype) -> int:
    h = ctypes.c_void_p()
    _check(load().kvc_create_rolling(ctypes.byref(h), layers, B, H_q, H_kv, D, window, dtype),
           "kvc_create_rolling")
    return h.value


def kvc_get_window(h) -> int:
    return int(load().kvc_get_window(h))


def kvc_create_paged(layers, num_blocks, block_size, B, max_blocks, H_q, H_kv, D, dtype) -> int:
    h = ctypes.c_void_p()
    _check(load().kvc_create_paged(ctypes.byref(h), layers, num_blocks, block_size, B, max_blocks,
                                   H_q, H_kv, D, dtype), "kvc_create_paged")
    return h.value


def kvc_paged_prefill_write(h, layer, K, V, T_in, block_table, lens, stream=None) -> None:
    _check(load().kvc_paged_prefill_write(h, layer, _ptr(K), _ptr(V), T_in, _ptr(block_table),
                                          _ptr(lens), _stream(stream)), "kvc_paged_prefill_write")


def kvc_paged_append(h, layer, k_new, v_new, block_table, lens, stream=None) -> None:
    _check(load().kvc_paged_append(h, layer, _ptr(k_new), _ptr(v_new), _ptr(block_table), _ptr(lens),
                                   _stream(stream)), "kvc_paged_append")


def kvc_paged_decode_attn(h, layer, q, out, block_table, lens, stream=None) -> None:
    _check(load().kvc_paged_decode_attn(h, layer, _ptr(q), _ptr(out), _ptr(block_table), _ptr(lens),
                                        _stream(stream)), "kvc_paged_decode_attn")


def kvc_paged_decode_step(h, layer, q, k_new, v_new, out, block_table, lens, stream=None) -> None:
    _check(load().kvc_paged_decode_step(h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out),
                                        _ptr(block_table), _ptr(lens), _stream(stream)),
           "kvc_paged_decode_step")


def kvc_get_paged_shape(h) -> dict:
    vals = [ctypes.c_int() for _ in range(3)]
    _check(load().kvc_get_paged_shape(h, *[ctypes.byref(v) for v in vals]), "kvc_get_paged_shape")
    return dict(zip(("num_blocks", "block_size", "max_blocks"), (v.value for v in vals)))


def kvc_bytes(h) -> int:
    return int(load().kvc_bytes(h))


def kvc_bytes_formula(L, B, H_kv, D, T, elem_bytes) -> int:
    return int(load().kvc_bytes_formula(L, B, H_kv, D, T, elem_bytes))


def kvc_payload_bytes(h, lens_host) -> int:
    import numpy as np
    arr = np.ascontiguousarray(lens_host, dtype=np.int32)
    return int(load().kvc_payload_bytes(h, arr.ctypes.data_as(ctypes.c_void_p)))


def kvc_layer_ptrs(h, layer) -> tuple[int, int]:
    k, v = ctypes.c_void_p(), ctypes.c_void_p()
    _check(load().kvc_layer_ptrs(h, layer, ctypes.byref(k), ctypes.byref(v)), "kvc_layer_ptrs")
    return k.value, v.value


def kvc_last_error(h, stream=None) -> tuple[int, int]:
    """Returns (status, detail bits); does not raise on KVC_EDEVICE."""
    detail = ctypes.c_uint32(0)
    st = load().kvc_last_error(h, _stream(stream), ctypes.byref(detail))
    return st, detail.value


def kvc_set_ctas(h, ctas) -> None:
    _check(load().kvc_set_ctas(h, ctas), "kvc_set_ctas")


def kvc_get_ctas(h) -> int:
    return int(load().kvc_get_ctas(h))


def kvc_set_combine_mode(h, mode) -> None:
    _check(load().kvc_set_combine_mode(h, mode), "kvc_set_combine_mode")


def kvc_set_math(h, mode) -> None:
    _check(load().kvc_set_math(h, mode), "kvc_set_math")


def kvc_get_math(h) -> int:
    return int(load().kvc_get_math(h))


def kvc_set_launch_overlap(h, on) -> None:
    _check(load().kvc_set_launch_overlap(h, int(on)), "kvc_set_launch_overlap")


def kvc_get_launch_overlap(h) -> int:
    return int(load().kvc_get_launch_overlap(h))


def kvc_get_shape(h) -> dict:
    vals = [ctypes.c_int() for _ in range(7)]
    _check(load().kvc_get_shape(h, *[ctypes.byref(v) for v in vals]), "kvc_get_shape")
    keys = ["layers", "B", "H_q", "H_kv", "D", "T_max", "dtype"]
    return {k: v.value for k, v in zip(keys, vals)}


def kvc_decode_attn_noalloc(K, V, B, H_q, H_kv, D, T_max, dtype, q, out, lens, err=None,
                            stream=None) -> None:
    """Decode attention with no device allocation: K, V are one layer's cache buffers owned by
    the caller; scratch lives in a fixed array inside the library (see include/kvc.h)."""
    _check(load().kvc_decode_attn_noalloc(_ptr(K), _ptr(V), B, H_q, H_kv, D, T_max, dtype, _ptr(q),
                                          _ptr(out), _ptr(lens), _ptr(err), _stream(stream)),
           "kvc_decode_attn_noalloc")


def kvc_selftest_wait_timeout(err, info, limit_ns=0, stream=None) -> None:
    """One CTA whose in-kernel wait runs out on purpose (see include/kvc.h): err (int32 [1]) gets
    KVC_DEV_WAIT_TIMEOUT, info (int64 [2]) the completed-wait count and thread 0's wait in ns."""
    _check(load().kvc_selftest_wait_timeout(_ptr(err), _ptr(info), int(limit_ns), _stream(stream)),
           "kvc_selftest_wait_timeout")


def kvc_plan_cta_of(x, U, P) -> int:
    return int(load().kvc_plan_cta_of(x, U, P))


# ----------------------------------------------------------------------------- owner class
class KVCache:
    """Owns one kvc handle: a [layers] x (K, V) cache of shape [B, H_kv, T_max, D]."""

    def __init__(self, layers, B, H_q, H_kv, D, T_max, dtype="bf16"):
        self.dtype_code = {"bf16": KVC_BF16, "f32": KVC_F32, KVC_BF16: KVC_BF16, KVC_F32: KVC_F32}[dtype]
        self.layers, self.B, self.H_q, self.H_kv, self.D, self.T_max = layers, B, H_q, H_kv, D, T_max
        self.h = kvc_create(layers, B, H_q, H_kv, D, T_max, self.dtype_code)

    @property
    def torch_dtype(self):
        import torch
        return torch.bfloat16 if self.dtype_code == KVC_BF16 else torch.float32

    def close(self):
        if self.h:
            kvc_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def nbytes(self) -> int:
        return kvc_bytes(self.h)

    def layer_views(self, layer):
        """torch views (no copy) of layer `layer`'s K and V caches."""
        import torch
        kp, vp = kvc_layer_ptrs(self.h, layer)
        shape = (self.B, self.H_kv, self.T_max, self.D)
        return _wrap_device(kp, shape, self.torch_dtype), _wrap_device(vp, shape, self.torch_dtype)

    def prefill_write(self, layer, K, V, lens, stream=None):
        kvc_prefill_write(self.h, layer, K, V, K.shape[2], lens, stream)

    def append(self, layer, k_new, v_new, lens, stream=None):
        kvc_append(self.h, layer, k_new, v_new, lens, stream)

    def decode_attn(self, layer, q, out, lens, stream=None):
        kvc_decode_attn(self.h, layer, q, out, lens, stream)

    def decode_step(self, layer, q, k_new, v_new, out, lens, stream=None):
        kvc_decode_step(self.h, layer, q, k_new, v_new, out, lens, stream)

    def last_error(self, stream=None):
        return kvc_last_error(self.h, stream)

    def set_ctas(self, ctas):
        kvc_set_ctas(self.h, ctas)

    def set_combine_mode(self, mode):
        kvc_set_combine_mode(self.h, mode)

    def set_math(self, mode):
        kvc_set_math(self.h, mode)

    def math(self) -> int:
        return kvc_get_math(self.h)

    def append_multi(self, layer, k_new, v_new, lens, stream=None):
        """k_new / v_new [B, H_kv, T_q, D] into slots [lens[b] - T_q, lens[b])."""
        kvc_append_multi(self.h, layer, k_new, v_new, lens, k_new.shape[2], stream)

    def decode_attn_multi(self, layer, q, out, lens, stream=None):
        """q, out [B, H_q, T_q, D]; new token i sees positions up to lens[b] - T_q + i."""
        kvc_decode_attn_multi(self.h, layer, q, out, lens, q.shape[2], stream)

    def decode_step_multi(self, layer, q, k_new, v_new, out, lens, stream=None):
        kvc_decode_step_multi(self.h, layer, q, k_new, v_new, out, lens, q.shape[2], stream)

    def set_launch_overlap(self, on):
        kvc_set_launch_overlap(self.h, on)

    def launch_overlap(self) -> int:
        return kvc_get_launch_overlap(self.h)


def _wrap_device(ptr: int, shape, dtype):
    """A torch tensor over library-owned device memory (the handle must outlive it)."""
    import torch

    class _Iface:
        def __init__(self):
            typestr = {torch.bfloat16: "<i2", torch.float32: "<f4", torch.int8: "|i1", torch.uint8: "|u1"}[dtype]
            self.__cuda_array_interface__ = {
                "shape": tuple(shape), "typestr": typestr, "data": (ptr, False), "version": 2,
                "strides": None,
            }

    t = torch.as_tensor(_Iface(), device="cuda")
    if dtype == torch.bfloat16:
        t = t.view(torch.bfloat16)
    return t


class PagedKVCache(KVCache):
    """Owns one paged kvc handle: per layer, K and V block pools [num_blocks, H_kv, block_size, D]
    reached through a caller-owned block table [B, max_blocks] (int32, device)."""

    def __init__(self, layers, num_blocks, block_size, B, max_blocks, H_q, H_kv, D, dtype="bf16"):
        self.dtype_code = {"bf16": KVC_BF16, "f32": KVC_F32, KVC_BF16: KVC_BF16, KVC_F32: KVC_F32}[dtype]
        self.layers, self.B, self.H_q, self.H_kv, self.D = layers, B, H_q, H_kv, D
        self.num_blocks, self.block_size, self.max_blocks = num_blocks, block_size, max_blocks
        self.T_max = max_blocks * block_size
        self.h = kvc_create_paged(layers, num_blocks, block_size, B, max_blocks, H_q, H_kv, D,
                                  self.dtype_code)

    def layer_views(self, layer):
        """torch views (no copy) of layer `layer`'s K and V block pools."""
        kp, vp = kvc_layer_ptrs(self.h, layer)
        shape = (self.num_blocks, self.H_kv, self.block_size, self.D)
        return _wrap_device(kp, shape, self.torch_dtype), _wrap_device(vp, shape, self.torch_dtype)

    def prefill_write(self, layer, K, V, block_table, lens, stream=None):
        kvc_paged_prefill_write(self.h, layer, K, V, K.shape[2], block_table, lens, stream)

    def append(self, layer, k_new, v_new, block_table, lens, stream=None):
        kvc_paged_append(self.h, layer, k_new, v_new, block_table, lens, stream)

    def decode_attn(self, layer, q, out, block_table, lens, stream=None):
        kvc_paged_decode_attn(self.h, layer, q, out, block_table, lens, stream)

    def decode_step(self, layer, q, k_new, v_new, out, block_table, lens, stream=None):
        kvc_paged_decode_step(self.h, layer, q, k_new, v_new, out, block_table, lens, stream)


class RollingKVCache(KVCache):
    """Owns one rolling kvc handle: per layer a [B, H_kv, window, D] cache, position p in slot
    p mod window; lens count positions and may exceed the window."""

    def __init__(self, layers, B, H_q, H_kv, D, window, dtype="bf16"):
        self.dtype_code = {"bf16": KVC_BF16, "f32": KVC_F32, KVC_BF16: KVC_BF16, KVC_F32: KVC_F32}[dtype]
        self.layers, self.B, self.H_q, self.H_kv, self.D = layers, B, H_q, H_kv, D
        self.window = self.T_max = window
        self.h = kvc_create_rolling(layers, B, H_q, H_kv, D, window, self.dtype_code)


class QuantKVCache(KVCache):
    """Owns one int8 kvc handle (fp8=True: an E4M3 handle): per layer, codes [B, H_kv, T_max, D]
    (int8, or uint8 E4M3 bit patterns) and row scales [B, H_kv, T_max] (fp32) for K and V; q,
    out and new rows stay bf16."""

    def __init__(self, layers, B, H_q, H_kv, D, T_max, dtype="bf16", fp8=False):
        self.dtype_code = {"bf16": KVC_BF16, KVC_BF16: KVC_BF16}[dtype]
        self.layers, self.B, self.H_q, self.H_kv, self.D, self.T_max = layers, B, H_q, H_kv, D, T_max
        self.fp8 = fp8
        create = kvc_create_fp8 if fp8 else kvc_create_quantized
        self.h = create(layers, B, H_q, H_kv, D, T_max, self.dtype_code)

    def layer_views(self, layer):
        """torch views (no copy): K codes, V codes (int8 / uint8) and K scales, V scales (fp32)."""
        import torch
        kp, vp = kvc_layer_ptrs(self.h, layer)
        ks, vs = kvc_layer_scales(self.h, layer)
        shape = (self.B, self.H_kv, self.T_max, self.D)
        cdt = torch.uint8 if self.fp8 else torch.int8
        return (_wrap_device(kp, shape, cdt), _wrap_device(vp, shape, cdt),
                _wrap_device(ks, shape[:3], torch.float32), _wrap_device(vs, shape[:3], torch.float32))
