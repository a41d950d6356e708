"""CPU oracle for the single-token KV-cache decode step (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline arm of ``bench.py``
may import this package.  The product path (the CUDA library and its binding) never
does: the two share no code.  The arithmetic lives in ``kvc_oracle.c`` (plain C,
double precision); this module builds it with gcc and marshals numpy arrays.

bf16 tensors are passed as their raw ``uint16`` bit patterns; fp32 as ``float32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvc_oracle.c")
_SO = os.path.join(_HERE, "libkvc_oracle.so")
# the same source with the planted mistakes compiled in (tests of the pins only)
_SO_PLANTED = os.path.join(_HERE, "libkvc_oracle_planted.so")

BF16, F32 = 0, 1
_lib = None
_lib_planted = None
_planted_on = False


def _compile(out: str, defines) -> None:
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", *defines, "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when the compiler has it), and its planted-mistake
    variant for the pin tests.  Returns the oracle's .so path."""
    for out, defs in ((_SO, []), (_SO_PLANTED, ["-DORACLE_PLANTED"])):
        if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
            _compile(out, defs)
    return _SO


def lib() -> ctypes.CDLL:
    """The oracle library (its planted-mistake build while a planted_fault context is open)."""
    global _lib, _lib_planted
    if _lib is None:
        build()
        _lib = _load(_SO)
        _lib_planted = _load(_SO_PLANTED)
        _lib_planted.oracle_set_fault.restype = None
        _lib_planted.oracle_set_fault.argtypes = [ctypes.c_int]
        _lib_planted.oracle_get_fault.restype = ctypes.c_int
    return _lib_planted if _planted_on else _lib


def _load(path: str) -> ctypes.CDLL:
    L = ctypes.CDLL(path)
    P, I, U64, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_int64
    L.oracle_kv_bytes.restype = U64
    L.oracle_kv_bytes.argtypes = [I64] * 6
    L.oracle_kv_bytes_ragged.restype = U64
    L.oracle_kv_bytes_ragged.argtypes = [I64, I64, I64, I64, P, I]
    L.oracle_append.restype = I
    L.oracle_append.argtypes = [P, P, P, P, P, I, I, I, I, I]
    L.oracle_prefill_write.restype = I
    L.oracle_prefill_write.argtypes = [P, P, P, P, I, P, I, I, I, I, I]
    L.oracle_decode_attn.restype = I
    L.oracle_decode_attn.argtypes = [P, P, P, P, I, I, I, I, I, I, P]
    L.oracle_layer_full.restype = None
    L.oracle_layer_full.argtypes = [P, I, I, I, I, I, I, P, P, P, P, P, P, P]
    L.oracle_layer_incremental.restype = None
    L.oracle_layer_incremental.argtypes = [P, I, I, I, I, I, I, I, P, P, P, P, P, P, P]
    L.oracle_paged_append.restype = I
    L.oracle_paged_append.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I]
    L.oracle_paged_prefill_write.restype = I
    L.oracle_paged_prefill_write.argtypes = [P, P, P, P, I, P, P, I, I, I, I, I, I, I]
    L.oracle_paged_decode_attn.restype = I
    L.oracle_paged_decode_attn.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, P]
    L.oracle_window_decode_attn.restype = I
    L.oracle_window_decode_attn.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P]
    L.oracle_rolling_append.restype = I
    L.oracle_rolling_append.argtypes = [P, P, P, P, P, I, I, I, I, I]
    L.oracle_rolling_decode_attn.restype = I
    L.oracle_rolling_decode_attn.argtypes = [P, P, P, P, I, I, I, I, I, I, P]
    L.oracle_append_multi.restype = I
    L.oracle_append_multi.argtypes = [P, P, P, P, P, I, I, I, I, I, I]
    L.oracle_decode_multi.restype = I
    L.oracle_decode_multi.argtypes = [P, P, P, P, I, I, I, I, I, I, I, P]
    L.oracle_quantize_rows.restype = None
    L.oracle_quantize_rows.argtypes = [P, I, I, I, P, P]
    L.oracle_quant_append.restype = I
    L.oracle_quant_append.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I]
    L.oracle_quant_prefill_write.restype = I
    L.oracle_quant_prefill_write.argtypes = [P, P, P, P, P, P, I, P, I, I, I, I, I]
    L.oracle_quant_decode_attn.restype = I
    L.oracle_quant_decode_attn.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P]
    L.oracle_e4m3_value.restype = ctypes.c_double
    L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    L.oracle_fp8_quantize_rows.restype = None
    L.oracle_fp8_quantize_rows.argtypes = [P, I, I, I, P, P]
    L.oracle_fp8_append.restype = I
    L.oracle_fp8_append.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I]
    L.oracle_fp8_prefill_write.restype = I
    L.oracle_fp8_prefill_write.argtypes = [P, P, P, P, P, P, I, P, I, I, I, I, I]
    L.oracle_fp8_decode_attn.restype = I
    L.oracle_fp8_decode_attn.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P]
    L.oracle_set_threads.restype = I
    L.oracle_set_threads.argtypes = [I]
    return L


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    raise TypeError(f"oracle takes bf16 bits (uint16) or float32, got {a.dtype}")


def kv_bytes(L, B, H_kv, D, T, s) -> int:
    return int(lib().oracle_kv_bytes(L, B, H_kv, D, T, s))


def kv_bytes_ragged(L, H_kv, D, s, T_i) -> int:
    t = np.ascontiguousarray(np.asarray(T_i, dtype=np.int32))
    return int(lib().oracle_kv_bytes_ragged(L, H_kv, D, s, _ptr(t), t.size))


def append(Kc, Vc, k_new, v_new, lens) -> int:
    """In place: writes k_new/v_new [B,H_kv,D] into slot lens[b]-1 of Kc/Vc [B,H_kv,T_max,D]."""
    B, H_kv, T_max, D = Kc.shape
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    return lib().oracle_append(_ptr(Kc), _ptr(Vc), _ptr(k_new), _ptr(v_new), _ptr(lens),
                               B, H_kv, T_max, D, _dtype_code(Kc))


def prefill_write(Kc, Vc, K, V, lens) -> int:
    """In place: copies K/V [B,H_kv,T_in,D] slots [0, lens[b]) into Kc/Vc."""
    B, H_kv, T_max, D = Kc.shape
    T_in = K.shape[2]
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    return lib().oracle_prefill_write(_ptr(Kc), _ptr(Vc), _ptr(K), _ptr(V), T_in, _ptr(lens),
                                      B, H_kv, T_max, D, _dtype_code(Kc))


def decode_attn(q, Kc, Vc, lens, return_bad: bool = False):
    """out[B,H_q,D] (float64) = softmax(q K^T / sqrt(D)) V over slots [0, lens[b])."""
    B, H_q, D = q.shape
    _, H_kv, T_max, D2 = Kc.shape
    assert D == D2 and Kc.shape == Vc.shape and q.dtype == Kc.dtype == Vc.dtype
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    out = np.zeros((B, H_q, D), dtype=np.float64)
    bad = lib().oracle_decode_attn(_ptr(q), _ptr(Kc), _ptr(Vc), _ptr(lens), B, H_q, H_kv, T_max,
                                   D, _dtype_code(q), _ptr(out))
    return (out, bad) if return_bad else out


def _paged_shape(Kp, table):
    num_blocks, H_kv, bs, D = Kp.shape
    B, max_blocks = table.shape
    return num_blocks, H_kv, bs, D, B, max_blocks


def paged_append(Kp, Vp, k_new, v_new, table, lens) -> int:
    """In place: token lens[b]-1 of sequence b (pool [num_blocks,H_kv,bs,D], table
    [B,max_blocks]) takes k_new/v_new [B,H_kv,D].  Returns the number of invalid rows."""
    table = np.ascontiguousarray(table, dtype=np.int32)
    nbk, H_kv, bs, D, B, mb = _paged_shape(Kp, table)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    return lib().oracle_paged_append(_ptr(Kp), _ptr(Vp), _ptr(k_new), _ptr(v_new), _ptr(table),
                                     _ptr(lens), B, H_kv, D, bs, mb, nbk, _dtype_code(Kp))


def paged_prefill_write(Kp, Vp, K, V, table, lens) -> int:
    """In place: tokens [0, lens[b]) of K/V [B,H_kv,T_in,D] into the pool through the table."""
    table = np.ascontiguousarray(table, dtype=np.int32)
    nbk, H_kv, bs, D, B, mb = _paged_shape(Kp, table)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    return lib().oracle_paged_prefill_write(_ptr(Kp), _ptr(Vp), _ptr(K), _ptr(V), K.shape[2],
                                            _ptr(table), _ptr(lens), B, H_kv, D, bs, mb, nbk,
                                            _dtype_code(Kp))


def paged_decode_attn(q, Kp, Vp, table, lens, return_bad: bool = False):
    """out[B,H_q,D] (float64): decode attention over the history read through the table."""
    table = np.ascontiguousarray(table, dtype=np.int32)
    nbk, H_kv, bs, D, B, mb = _paged_shape(Kp, table)
    Bq, H_q, Dq = q.shape
    assert Bq == B and Dq == D and Kp.shape == Vp.shape and q.dtype == Kp.dtype == Vp.dtype
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    out = np.zeros((B, H_q, D), dtype=np.float64)
    bad = lib().oracle_paged_decode_attn(_ptr(q), _ptr(Kp), _ptr(Vp), _ptr(table), _ptr(lens), B,
                                         H_q, H_kv, D, bs, mb, nbk, _dtype_code(q), _ptr(out))
    return (out, bad) if return_bad else out


def quantize_rows(x):
    """int8 codes and fp32 scales of the rows of x [..., D] (bf16 bits or float32)."""
    x = np.ascontiguousarray(x)
    D = x.shape[-1]
    n = x.size // D
    codes = np.zeros(x.shape, np.int8)
    scales = np.zeros(x.shape[:-1], np.float32)
    lib().oracle_quantize_rows(_ptr(x), n, D, _dtype_code(x), _ptr(codes), _ptr(scales))
    return codes, scales


class QuantCache:
    """One layer of a quantized cache: int8 codes [B,H_kv,T_max,D] and fp32 scales [B,H_kv,T_max]
    for K and for V."""

    def __init__(self, B, H_kv, T_max, D):
        self.Kq = np.zeros((B, H_kv, T_max, D), np.int8)
        self.Vq = np.zeros_like(self.Kq)
        self.Ks = np.zeros((B, H_kv, T_max), np.float32)
        self.Vs = np.zeros_like(self.Ks)

    def _args(self):
        return _ptr(self.Kq), _ptr(self.Ks), _ptr(self.Vq), _ptr(self.Vs)

    def append(self, k_new, v_new, lens) -> int:
        B, H_kv, T_max, D = self.Kq.shape
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        return lib().oracle_quant_append(*self._args(), _ptr(k_new), _ptr(v_new), _ptr(lens), B, H_kv,
                                         T_max, D, _dtype_code(k_new))

    def prefill_write(self, K, V, lens) -> int:
        B, H_kv, T_max, D = self.Kq.shape
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        return lib().oracle_quant_prefill_write(*self._args(), _ptr(K), _ptr(V), K.shape[2], _ptr(lens), B,
                                                H_kv, T_max, D, _dtype_code(K))

    def decode_attn(self, q, lens, return_bad: bool = False):
        B, H_kv, T_max, D = self.Kq.shape
        H_q = q.shape[1]
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        out = np.zeros((B, H_q, D), dtype=np.float64)
        bad = lib().oracle_quant_decode_attn(_ptr(q), *self._args(), _ptr(lens), B, H_q, H_kv, T_max, D,
                                             _dtype_code(q), _ptr(out))
        return (out, bad) if return_bad else out


def e4m3_value(codes) -> np.ndarray:
    """float64 values of E4M3 codes (uint8 array)."""
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib().oracle_e4m3_value(int(x)) for x in c.ravel()], dtype=np.float64).reshape(c.shape)


def e4m3_encode(x) -> np.ndarray:
    """E4M3 codes (uint8) of float32 values: nearest, ties to even, saturating at +-448."""
    a = np.asarray(x, dtype=np.float32)
    return np.array([lib().oracle_e4m3_encode(float(v)) for v in a.ravel()], dtype=np.uint8).reshape(a.shape)


def fp8_quantize_rows(x):
    """E4M3 codes (uint8) and fp32 scales of the rows of x [..., D] (bf16 bits or float32)."""
    x = np.ascontiguousarray(x)
    D = x.shape[-1]
    n = x.size // D
    codes = np.zeros(x.shape, np.uint8)
    scales = np.zeros(x.shape[:-1], np.float32)
    lib().oracle_fp8_quantize_rows(_ptr(x), n, D, _dtype_code(x), _ptr(codes), _ptr(scales))
    return codes, scales


class Fp8Cache(QuantCache):
    """One layer of an fp8 cache: E4M3 codes [B,H_kv,T_max,D] (uint8) and fp32 row scales
    [B,H_kv,T_max] for K and for V."""

    def __init__(self, B, H_kv, T_max, D):
        super().__init__(B, H_kv, T_max, D)
        self.Kq = np.zeros((B, H_kv, T_max, D), np.uint8)
        self.Vq = np.zeros_like(self.Kq)

    def append(self, k_new, v_new, lens) -> int:
        B, H_kv, T_max, D = self.Kq.shape
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        return lib().oracle_fp8_append(*self._args(), _ptr(k_new), _ptr(v_new), _ptr(lens), B, H_kv,
                                       T_max, D, _dtype_code(k_new))

    def prefill_write(self, K, V, lens) -> int:
        B, H_kv, T_max, D = self.Kq.shape
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        return lib().oracle_fp8_prefill_write(*self._args(), _ptr(K), _ptr(V), K.shape[2], _ptr(lens), B,
                                              H_kv, T_max, D, _dtype_code(K))

    def decode_attn(self, q, lens, return_bad: bool = False):
        B, H_kv, T_max, D = self.Kq.shape
        H_q = q.shape[1]
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        out = np.zeros((B, H_q, D), dtype=np.float64)
        bad = lib().oracle_fp8_decode_attn(_ptr(q), *self._args(), _ptr(lens), B, H_q, H_kv, T_max, D,
                                           _dtype_code(q), _ptr(out))
        return (out, bad) if return_bad else out


def append_multi(Kc, Vc, k_new, v_new, lens) -> int:
    """In place: the T_q rows of k_new/v_new [B,H_kv,T_q,D] into slots [lens[b]-T_q, lens[b])."""
    B, H_kv, T_max, D = Kc.shape
    T_q = k_new.shape[2]
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    return lib().oracle_append_multi(_ptr(Kc), _ptr(Vc), _ptr(k_new), _ptr(v_new), _ptr(lens), B, H_kv,
                                     T_max, D, T_q, _dtype_code(Kc))


def decode_multi(q, Kc, Vc, lens, return_bad: bool = False):
    """out[B,H_q,T_q,D] (float64): new query i of sequence b sees keys 0 .. lens[b]-T_q+i."""
    B, H_q, T_q, D = q.shape
    _, H_kv, T_max, _ = Kc.shape
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    out = np.zeros((B, H_q, T_q, D), dtype=np.float64)
    bad = lib().oracle_decode_multi(_ptr(q), _ptr(Kc), _ptr(Vc), _ptr(lens), B, H_q, H_kv, T_max, D,
                                    T_q, _dtype_code(q), _ptr(out))
    return (out, bad) if return_bad else out


def window_decode_attn(q, Kc, Vc, lens, W, return_bad: bool = False):
    """Sliding-window decode over a full-history cache [B,H_kv,T_max,D]: positions
    [max(0, L-W), L).  out [B,H_q,D] float64."""
    B, H_q, D = q.shape
    _, H_kv, T_max, _ = Kc.shape
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    out = np.zeros((B, H_q, D), dtype=np.float64)
    bad = lib().oracle_window_decode_attn(_ptr(q), _ptr(Kc), _ptr(Vc), _ptr(lens), B, H_q, H_kv,
                                          T_max, D, W, _dtype_code(q), _ptr(out))
    return (out, bad) if return_bad else out


def rolling_append(Kr, Vr, k_new, v_new, lens) -> int:
    """In place: position lens[b]-1 into slot (lens[b]-1) mod W of the rolling cache [B,H_kv,W,D]."""
    B, H_kv, W, D = Kr.shape
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    return lib().oracle_rolling_append(_ptr(Kr), _ptr(Vr), _ptr(k_new), _ptr(v_new), _ptr(lens), B,
                                       H_kv, W, D, _dtype_code(Kr))


def rolling_decode_attn(q, Kr, Vr, lens, return_bad: bool = False):
    """Decode over a rolling cache [B,H_kv,W,D]: positions [max(0, L-W), L), position p in slot
    p mod W.  out [B,H_q,D] float64."""
    B, H_q, D = q.shape
    _, H_kv, W, _ = Kr.shape
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    out = np.zeros((B, H_q, D), dtype=np.float64)
    bad = lib().oracle_rolling_decode_attn(_ptr(q), _ptr(Kr), _ptr(Vr), _ptr(lens), B, H_q, H_kv, W,
                                           D, _dtype_code(q), _ptr(out))
    return (out, bad) if return_bad else out


def layer_full(x, WQ, WK, WV, WO, H_q, H_kv, D):
    """Path A (dense causal layer).  Returns (out[B,T,hidden], K[B,H_kv,T,D], V[...])."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    B, T, hidden = x.shape
    Ws = [np.ascontiguousarray(w, dtype=np.float64) for w in (WQ, WK, WV, WO)]
    out = np.zeros((B, T, hidden))
    K = np.zeros((B, H_kv, T, D))
    V = np.zeros((B, H_kv, T, D))
    lib().oracle_layer_full(_ptr(x), B, T, hidden, H_q, H_kv, D, *[_ptr(w) for w in Ws],
                            _ptr(out), _ptr(K), _ptr(V))
    return out, K, V


def layer_incremental(x, T_p, WQ, WK, WV, WO, H_q, H_kv, D):
    """Path B (prefill T_p, then one token at a time through the cache).
    Returns (decode outputs [B, T-T_p, hidden], final K cache, final V cache)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    B, T, hidden = x.shape
    Ws = [np.ascontiguousarray(w, dtype=np.float64) for w in (WQ, WK, WV, WO)]
    out = np.zeros((B, T - T_p, hidden))
    Kc = np.zeros((B, H_kv, T, D))
    Vc = np.zeros((B, H_kv, T, D))
    lib().oracle_layer_incremental(_ptr(x), B, T_p, T, hidden, H_q, H_kv, D,
                                   *[_ptr(w) for w in Ws], _ptr(out), _ptr(Kc), _ptr(Vc))
    return out, Kc, Vc


class planted_fault:
    """Context manager that plants a known mistake in the oracle (tests only).

    1 = interleaved GQA map (j mod H_kv), 2 = score scale 1/D, 3 = append one slot late,
    4 = the new token left out of the attention, 5 = paged block stored token-major,
    6 = sliding window one position too wide,
    7 = several-query causal mask aligned to the upper left,
    8 = quantization scale max/128 instead of max/127,
    9 = E4M3 rounding ties away from zero, 10 = fp8 scale max/240 instead of max/448."""

    def __init__(self, which: int):
        self.which = which

    def __enter__(self):
        global _planted_on
        lib()
        _lib_planted.oracle_set_fault(self.which)
        _planted_on = True
        return self

    def __exit__(self, *exc):
        global _planted_on
        _lib_planted.oracle_set_fault(0)
        _planted_on = False
        return False


def set_threads(n: int) -> int:
    """Host threads for decode_attn (OpenMP over rows); returns the count in effect."""
    return int(lib().oracle_set_threads(int(n)))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
