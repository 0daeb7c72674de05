"""CPU oracle for the MoE finalize + residual + RMSNorm path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only users.  The product package never
imports this module, and this module never imports the product package.

The arithmetic lives in ``mfr_oracle.c`` (plain C, one token and one column at
a time); this file only builds/loads it and marshals NumPy arrays.  BF16 data
crosses as ``uint16`` bit patterns.

Pins: every function here is checked in ``tests/test_oracle.py``,
``tests/test_oracle_nvfp4.py`` or ``tests/test_oracle_expert_norm.py`` against
values fixed by the pages or by mathematics (a hand-worked example, closed
forms, brute force with exact rationals, a library BF16 rounding, a library
RMSNorm, invariants); ``tests/test_oracle_mutations.py`` shows that planted
mistakes in the C source fail those pins.  No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "mfr_oracle.c")
LIBRARY = os.path.join(_HERE, "libmfr_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared"]


def compile_oracle(src: str, out: str) -> str:
    """gcc with no FMA contraction and no fast-math, so FMAs are only where
    the source writes fmaf()."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIBRARY) or \
            os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE):
        compile_oracle(SOURCE, LIBRARY)
    return LIBRARY


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def bf16_bits_to_f64(b) -> np.ndarray:
    """Exact widening of BF16 bit patterns (uint16) to double (NumPy only)."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class Oracle:
    """ctypes front end of one compiled copy of the oracle."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.mfr_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.mfr_oracle_bf16_to_f64.restype = ctypes.c_double
        lib.mfr_oracle_bf16_from_f64.argtypes = [ctypes.c_double]
        lib.mfr_oracle_bf16_from_f64.restype = ctypes.c_uint16
        lib.mfr_oracle_bf16_from_f64_array.argtypes = [p, p, i64]
        lib.mfr_oracle_bf16_from_f64_array.restype = None
        lib.mfr_oracle_weighted_residual.argtypes = [i64, i64, i64, i64, p, p, p, p, p, p, i64]
        lib.mfr_oracle_weighted_residual.restype = i64
        lib.mfr_oracle_rmsnorm_f64.argtypes = [i64, i64, p, p, ctypes.c_float, p]
        lib.mfr_oracle_rmsnorm_f64.restype = None
        lib.mfr_oracle_finalize_residual_rmsnorm.argtypes = [
            i64, i64, i64, i64, p, p, p, p, p, ctypes.c_float, p, p, p, i64, p]
        lib.mfr_oracle_finalize_residual_rmsnorm.restype = i64
        lib.mfr_oracle_finalize_only.argtypes = [i64, i64, i64, i64, p, p, p, p, p, i64]
        lib.mfr_oracle_finalize_only.restype = i64
        lib.mfr_oracle_e4m3_from_f64.argtypes = [ctypes.c_double]
        lib.mfr_oracle_e4m3_from_f64.restype = ctypes.c_uint8
        lib.mfr_oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.mfr_oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.mfr_oracle_e2m1_from_f64.argtypes = [ctypes.c_double]
        lib.mfr_oracle_e2m1_from_f64.restype = ctypes.c_uint8
        lib.mfr_oracle_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        lib.mfr_oracle_e2m1_to_f64.restype = ctypes.c_double
        lib.mfr_oracle_nvfp4_quantize.argtypes = [i64, i64, p, ctypes.c_float, p, p]
        lib.mfr_oracle_nvfp4_quantize.restype = None
        lib.mfr_oracle_nvfp4_encode.argtypes = [i64, i64, p, ctypes.c_float, p, p]
        lib.mfr_oracle_nvfp4_encode.restype = None
        lib.mfr_oracle_nvfp4_swizzle_scales.argtypes = [i64, i64, p, p]
        lib.mfr_oracle_nvfp4_swizzle_scales.restype = None
        lib.mfr_oracle_finalize_residual_rmsnorm_nvfp4.argtypes = [
            i64, i64, i64, i64, p, p, p, p, p, ctypes.c_float, ctypes.c_float, p, p, p, p, i64, p, p]
        lib.mfr_oracle_finalize_residual_rmsnorm_nvfp4.restype = i64
        lib.mfr_oracle_expert_rmsnorm_f64.argtypes = [i64, i64, i64, i64, p, p, p, p, ctypes.c_float, p, p, i64]
        lib.mfr_oracle_expert_rmsnorm_f64.restype = i64
        lib.mfr_oracle_finalize_expert_rmsnorm.argtypes = [
            i64, i64, i64, i64, p, p, p, p, ctypes.c_float, p, p, i64, p]
        lib.mfr_oracle_finalize_expert_rmsnorm.restype = i64
        self.lib = lib
        self.path = path

    # -- BF16 -----------------------------------------------------------------
    def bf16_from_f64(self, x) -> np.ndarray:
        """Nearest BF16 (ties to even) of each double, one rounding; uint16."""
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.mfr_oracle_bf16_from_f64_array(_ptr(x), _ptr(out), x.size)
        return out

    def bf16_to_f64(self, b) -> np.ndarray:
        b = np.asarray(b, dtype=np.uint16)
        f = np.vectorize(self.lib.mfr_oracle_bf16_to_f64, otypes=[np.float64])
        return f(b) if b.size else b.astype(np.float64)

    # -- the path, step by step ----------------------------------------------
    @staticmethod
    def _tokens(tokens, T):
        if tokens is None:
            return None, T
        tk = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64).reshape(-1))
        if tk.size and (tk.min() < 0 or tk.max() >= T):
            raise IndexError("token index out of range")
        return tk, tk.size

    def weighted_residual(self, expert_out_bits, permuted_row_of, topk_weights,
                          residual_in, tokens: Optional[Sequence[int]] = None):
        """x = residual_in + sum_j w[t,j] * E[idx[t,j]], FP32 FMAs in slot
        order.  Returns (x float32 [n, H], number of out-of-range slots)."""
        E = _c(expert_out_bits, np.uint16)
        idx = _c(permuted_row_of, np.int32)
        w = _c(topk_weights, np.float32)
        res = _c(residual_in, np.float32)
        R, H = E.shape
        T, k = idx.shape
        assert w.shape == (T, k) and res.shape == (T, H)
        tk, n = self._tokens(tokens, T)
        x = np.empty((n, H), dtype=np.float32)
        bad = self.lib.mfr_oracle_weighted_residual(T, H, k, R, _ptr(E), _ptr(idx), _ptr(w),
                                                    _ptr(res), _ptr(x), _ptr(tk), n)
        return x, int(bad)

    def rmsnorm_f64(self, x, gamma_bits, eps: float) -> np.ndarray:
        """y = x / sqrt(mean(x^2) + eps) * gamma, in double, row by row."""
        x = _c(x, np.float32)
        g = _c(gamma_bits, np.uint16)
        n, H = x.shape
        assert g.shape == (H,)
        y = np.empty((n, H), dtype=np.float64)
        self.lib.mfr_oracle_rmsnorm_f64(n, H, _ptr(x), _ptr(g), ctypes.c_float(eps), _ptr(y))
        return y

    def finalize_residual_rmsnorm(self, expert_out_bits, permuted_row_of, topk_weights,
                                  residual_in, gamma_bits, eps: float,
                                  tokens: Optional[Sequence[int]] = None):
        """The whole path for the given tokens (all when None).

        Returns (residual_out float32 [n, H], out uint16 [n, H] BF16 bits,
        number of out-of-range slots)."""
        E = _c(expert_out_bits, np.uint16)
        idx = _c(permuted_row_of, np.int32)
        w = _c(topk_weights, np.float32)
        res = _c(residual_in, np.float32)
        g = _c(gamma_bits, np.uint16)
        R, H = E.shape
        T, k = idx.shape
        assert w.shape == (T, k) and res.shape == (T, H) and g.shape == (H,)
        tk, n = self._tokens(tokens, T)
        res_out = np.empty((n, H), dtype=np.float32)
        out = np.empty((n, H), dtype=np.uint16)
        scratch = np.empty(H, dtype=np.float64)
        bad = self.lib.mfr_oracle_finalize_residual_rmsnorm(
            T, H, k, R, _ptr(E), _ptr(idx), _ptr(w), _ptr(res), _ptr(g), ctypes.c_float(eps),
            _ptr(res_out), _ptr(out), _ptr(tk), n, _ptr(scratch))
        return res_out, out, int(bad)

    def finalize_only(self, expert_out_bits, permuted_row_of, topk_weights,
                      tokens: Optional[Sequence[int]] = None):
        """out = BF16(sum_j w[t,j] * E[idx[t,j]]), the FP32 FMA sum rounded
        once.  Returns (out uint16 [n, H], number of out-of-range slots)."""
        E = _c(expert_out_bits, np.uint16)
        idx = _c(permuted_row_of, np.int32)
        w = _c(topk_weights, np.float32)
        R, H = E.shape
        T, k = idx.shape
        tk, n = self._tokens(tokens, T)
        out = np.empty((n, H), dtype=np.uint16)
        bad = self.lib.mfr_oracle_finalize_only(T, H, k, R, _ptr(E), _ptr(idx), _ptr(w),
                                                _ptr(out), _ptr(tk), n)
        return out, int(bad)


    # -- per-expert RMSNorm before the weighted sum (a reading) ---------------
    def expert_rmsnorm_f64(self, expert_out_bits, permuted_row_of, topk_weights, gamma_bits, eps: float,
                           tokens: Optional[Sequence[int]] = None):
        """y = sum_j w[t,j] * RMSNorm(E[idx[t,j]]) * gamma, in double.
        Returns (y float64 [n, H], number of out-of-range slots)."""
        E = _c(expert_out_bits, np.uint16)
        idx = _c(permuted_row_of, np.int32)
        w = _c(topk_weights, np.float32)
        g = _c(gamma_bits, np.uint16)
        R, H = E.shape
        T, k = idx.shape
        assert w.shape == (T, k) and g.shape == (H,)
        tk, n = self._tokens(tokens, T)
        y = np.empty((n, H), dtype=np.float64)
        bad = self.lib.mfr_oracle_expert_rmsnorm_f64(T, H, k, R, _ptr(E), _ptr(idx), _ptr(w), _ptr(g),
                                                     ctypes.c_float(eps), _ptr(y), _ptr(tk), n)
        return y, int(bad)

    def finalize_expert_rmsnorm(self, expert_out_bits, permuted_row_of, topk_weights, gamma_bits, eps: float,
                                tokens: Optional[Sequence[int]] = None):
        """out = BF16(sum_j w[t,j] * RMSNorm(E[idx[t,j]]) * gamma), one
        rounding from double.  Returns (out uint16 [n, H], bad slots)."""
        E = _c(expert_out_bits, np.uint16)
        idx = _c(permuted_row_of, np.int32)
        w = _c(topk_weights, np.float32)
        g = _c(gamma_bits, np.uint16)
        R, H = E.shape
        T, k = idx.shape
        assert w.shape == (T, k) and g.shape == (H,)
        tk, n = self._tokens(tokens, T)
        out = np.empty((n, H), dtype=np.uint16)
        scratch = np.empty(H, dtype=np.float64)
        bad = self.lib.mfr_oracle_finalize_expert_rmsnorm(T, H, k, R, _ptr(E), _ptr(idx), _ptr(w), _ptr(g),
                                                          ctypes.c_float(eps), _ptr(out), _ptr(tk), n,
                                                          _ptr(scratch))
        return out, int(bad)

    # -- NVFP4 ----------------------------------------------------------------
    def e4m3_from_f64(self, x) -> np.ndarray:
        f = np.vectorize(self.lib.mfr_oracle_e4m3_from_f64, otypes=[np.uint8])
        return f(np.asarray(x, dtype=np.float64))

    def e4m3_to_f64(self, b) -> np.ndarray:
        f = np.vectorize(self.lib.mfr_oracle_e4m3_to_f64, otypes=[np.float64])
        return f(np.asarray(b, dtype=np.uint8))

    def e2m1_from_f64(self, x) -> np.ndarray:
        f = np.vectorize(self.lib.mfr_oracle_e2m1_from_f64, otypes=[np.uint8])
        return f(np.asarray(x, dtype=np.float64))

    def e2m1_to_f64(self, c) -> np.ndarray:
        f = np.vectorize(self.lib.mfr_oracle_e2m1_to_f64, otypes=[np.float64])
        return f(np.asarray(c, dtype=np.uint8))

    def nvfp4_quantize(self, y, s_enc: float):
        """y float32 [n, H] (H % 16 == 0) -> (packed codes uint8 [n, H/2],
        block scales uint8 [n, H/16])."""
        y = _c(y, np.float32)
        n, H = y.shape
        assert H % 16 == 0
        q = np.empty((n, H // 2), dtype=np.uint8)
        sf = np.empty((n, H // 16), dtype=np.uint8)
        self.lib.mfr_oracle_nvfp4_quantize(n, H, _ptr(y), ctypes.c_float(s_enc), _ptr(q), _ptr(sf))
        return q, sf

    def nvfp4_encode(self, y, s_enc: float, sf):
        """The codes of y float32 [n, H] for block scales chosen by the caller
        (sf uint8 [n, H/16]), by the quantiser's steps after its scale
        choice.  Returns packed codes uint8 [n, H/2]."""
        y = _c(y, np.float32)
        sf = _c(sf, np.uint8)
        n, H = y.shape
        assert H % 16 == 0 and sf.shape == (n, H // 16)
        q = np.empty((n, H // 2), dtype=np.uint8)
        self.lib.mfr_oracle_nvfp4_encode(n, H, _ptr(y), ctypes.c_float(s_enc), _ptr(sf), _ptr(q))
        return q

    def nvfp4_swizzle_scales(self, sf, fill: int = 0):
        """Block scales uint8 [n, S] -> the tiled layout block-scaled GEMMs
        read: uint8 [ceil(n/128)*128 * ceil(S/4)*4], padding bytes = fill."""
        sf = _c(sf, np.uint8)
        n, S = sf.shape
        out = np.full(-(-n // 128) * 128 * (-(-S // 4) * 4), fill, dtype=np.uint8)
        self.lib.mfr_oracle_nvfp4_swizzle_scales(n, S, _ptr(sf), _ptr(out))
        return out

    def finalize_residual_rmsnorm_nvfp4(self, expert_out_bits, permuted_row_of, topk_weights, residual_in,
                                        gamma_bits, eps: float, s_enc: float,
                                        tokens: Optional[Sequence[int]] = None):
        """The path with the NVFP4 epilogue.  Returns (residual_out float32
        [n, H], packed codes [n, H/2], block scales [n, H/16], bad slots)."""
        E = _c(expert_out_bits, np.uint16)
        idx = _c(permuted_row_of, np.int32)
        w = _c(topk_weights, np.float32)
        res = _c(residual_in, np.float32)
        g = _c(gamma_bits, np.uint16)
        R, H = E.shape
        T, k = idx.shape
        assert H % 16 == 0
        tk, n = self._tokens(tokens, T)
        res_out = np.empty((n, H), dtype=np.float32)
        q = np.empty((n, H // 2), dtype=np.uint8)
        sf = np.empty((n, H // 16), dtype=np.uint8)
        ys = np.empty(H, dtype=np.float64)
        y32 = np.empty(H, dtype=np.float32)
        bad = self.lib.mfr_oracle_finalize_residual_rmsnorm_nvfp4(
            T, H, k, R, _ptr(E), _ptr(idx), _ptr(w), _ptr(res), _ptr(g), ctypes.c_float(eps),
            ctypes.c_float(s_enc), _ptr(res_out), _ptr(q), _ptr(sf), _ptr(tk), n, _ptr(ys), _ptr(y32))
        return res_out, q, sf, int(bad)


def unpack_e2m1(q_packed: np.ndarray) -> np.ndarray:
    """[n, H/2] packed bytes -> [n, H] codes (element 2j = low nibble)."""
    q = np.asarray(q_packed, dtype=np.uint8)
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = q & 0xF
    out[..., 1::2] = q >> 4
    return out


_default: Optional[Oracle] = None
_lock = threading.Lock()


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def bf16_from_f64(x):
    return default().bf16_from_f64(x)


def weighted_residual(*a, **kw):
    return default().weighted_residual(*a, **kw)


def rmsnorm_f64(*a, **kw):
    return default().rmsnorm_f64(*a, **kw)


def finalize_residual_rmsnorm(*a, **kw):
    return default().finalize_residual_rmsnorm(*a, **kw)


def finalize_only(*a, **kw):
    return default().finalize_only(*a, **kw)


def nvfp4_quantize(*a, **kw):
    return default().nvfp4_quantize(*a, **kw)


def nvfp4_encode(*a, **kw):
    return default().nvfp4_encode(*a, **kw)


def nvfp4_swizzle_scales(*a, **kw):
    return default().nvfp4_swizzle_scales(*a, **kw)


def finalize_residual_rmsnorm_nvfp4(*a, **kw):
    return default().finalize_residual_rmsnorm_nvfp4(*a, **kw)


def expert_rmsnorm_f64(*a, **kw):
    return default().expert_rmsnorm_f64(*a, **kw)


def finalize_expert_rmsnorm(*a, **kw):
    return default().finalize_expert_rmsnorm(*a, **kw)
