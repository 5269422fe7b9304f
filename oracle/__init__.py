"""CPU oracle for the q4f16_1 fused dequantize + NT matmul.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg are the only callers. The CUDA
library never imports this package and shares no code with it.

The arithmetic lives in ``zq4_oracle.c`` (plain fp64 C, one function per
passage of the pages, see its header). This module compiles it with gcc,
loads it with ctypes and wraps each entry in a numpy-friendly function.
Inputs are the raw bits: packed words as uint32, scales / activations as
float16 arrays (passed bit for bit), router weights as float32.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zq4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict = {}


def lib_path(mutant: int = 0) -> str:
    name = "libzq4_oracle.so" if mutant == 0 else f"libzq4_oracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (OpenMP when the compiler has it). Returns the .so path."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", f"-DZO_MUTANT={int(mutant)}",
            _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def _load(mutant: int = 0):
    with _LOCK:
        if mutant in _LIBS:
            return _LIBS[mutant]
        lib = ctypes.CDLL(build(mutant))
        lib.zo_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.zo_f16_to_f64.restype = ctypes.c_double
        lib.zo_f64_to_f16_rn.argtypes = [ctypes.c_double]
        lib.zo_f64_to_f16_rn.restype = ctypes.c_uint16
        lib.zo_code.argtypes = [_p, _i64, _i64, _i64]
        lib.zo_code.restype = ctypes.c_int
        lib.zo_weight.argtypes = [_p, _p, _i64, _i64, _i64]
        lib.zo_weight.restype = ctypes.c_double
        lib.zo_dequant.argtypes = [_p, _p, _i64, _i64, _p]
        lib.zo_gemv_rows.argtypes = [_p, _p, _p, _i64, _i64, _i64, _p, _i64, _p, _p]
        lib.zo_gemv.argtypes = [_p, _p, _p, _i64, _i64, _i64, _p, _p]
        lib.zo_silu.argtypes = [ctypes.c_double]
        lib.zo_silu.restype = ctypes.c_double
        lib.zo_silu_deriv.argtypes = [ctypes.c_double]
        lib.zo_silu_deriv.restype = ctypes.c_double
        lib.zo_gate_up_silu.argtypes = [_p, _p, _p, _i64, _i64, _i64, ctypes.c_int,
                                        _p, _p, _p, _p, _p, _p]
        lib.zo_moe_gate_up.argtypes = [_p, _p, _i64, _p, _i64, _i64, _i64, _p, _i64,
                                       ctypes.c_int, _p, _p]
        lib.zo_moe_gate_up.restype = _i64
        lib.zo_moe_down_combine.argtypes = [_p, _p, _i64, _p, _p, _i64, _i64, _i64, _p,
                                            _i64, _p, _p]
        lib.zo_moe_down_combine.restype = _i64
        lib.zo_argmax.argtypes = [_p, _i64, _i64, _p]
        lib.zo_weight_affine.argtypes = [_p, _p, _p, _i64, _i64, _i64]
        lib.zo_weight_affine.restype = ctypes.c_double
        lib.zo_dequant_affine.argtypes = [_p, _p, _p, _i64, _i64, _p]
        lib.zo_gemv_affine_rows.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p, _i64, _p, _p]
        lib.zo_gate_up_silu_affine.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p, _p]
        lib.zo_moe_gate_up_affine.argtypes = [_p, _p, _p, _i64, _p, _i64, _i64, _i64, _p, _i64, _p, _p]
        lib.zo_moe_gate_up_affine.restype = _i64
        lib.zo_moe_down_combine_affine.argtypes = [_p, _p, _p, _i64, _p, _p, _i64, _i64, _i64, _p, _i64, _p, _p]
        lib.zo_moe_down_combine_affine.restype = _i64
        lib.zo_gemv_add_rmsnorm.argtypes = [_p, _p, _p, _p, _p, ctypes.c_double, _i64, _i64, _i64, _p, _p, _p, _p]
        lib.zo_qkv_rope.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, _i64, ctypes.c_double, _p] + [_p] * 9
        lib.zo_num_threads.restype = ctypes.c_int
        lib.zo_set_num_threads.argtypes = [ctypes.c_int]
        lib.zo_set_num_threads.restype = ctypes.c_int
        lib.zo_mutant.restype = ctypes.c_int
        _LIBS[mutant] = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _u32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint32)


def _f16(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float16)


class Oracle:
    """fp64 oracle bound to one build (``mutant=0`` is the real one)."""

    def __init__(self, mutant: int = 0):
        self.mutant = mutant
        self.lib = _load(mutant)

    # --- binary16 ---------------------------------------------------------
    def f16_to_f64(self, bits: int) -> float:
        return self.lib.zo_f16_to_f64(int(bits) & 0xFFFF)

    def f64_to_f16_bits(self, v: float) -> int:
        return int(self.lib.zo_f64_to_f16_rn(float(v)))

    def round_f16(self, a) -> np.ndarray:
        """Element-wise fp64 -> f16 (round to nearest even), via the oracle."""
        a = np.asarray(a, dtype=np.float64)
        bits = np.fromiter((self.lib.zo_f64_to_f16_rn(float(v)) for v in a.ravel()),
                           dtype=np.uint16, count=a.size)
        return bits.view(np.float16).reshape(a.shape)

    # --- format -----------------------------------------------------------
    def code(self, wq, K: int, n: int, k: int) -> int:
        wq = _u32(wq)
        return self.lib.zo_code(_ptr(wq), K, n, k)

    def dequant(self, wq, scales, N: int, K: int) -> np.ndarray:
        wq, sc = _u32(wq), _f16(scales)
        out = np.empty((N, K), dtype=np.float64)
        self.lib.zo_dequant(_ptr(wq), _ptr(sc), N, K, _ptr(out))
        return out

    # --- GEMV -------------------------------------------------------------
    def gemv(self, wq, scales, x, N: int, K: int, rows=None):
        """y_ref, S (both [M, N] or [M, len(rows)] fp64)."""
        wq, sc, xx = _u32(wq), _f16(scales), _f16(x)
        M = xx.size // K if K else 0
        if rows is None:
            R, rp = N, None
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            R, rp = rows.size, rows
        y = np.empty((M, R), dtype=np.float64)
        S = np.empty((M, R), dtype=np.float64)
        self.lib.zo_gemv_rows(_ptr(wq), _ptr(sc), _ptr(xx), M, N, K,
                              None if rp is None else _ptr(rp), R, _ptr(y), _ptr(S))
        return y, S

    def silu(self, z: float) -> float:
        return self.lib.zo_silu(float(z))

    # --- MLX affine format (w = s q + b, groups of 64) -------------------------
    def weight_affine(self, wq, scales, biases, K: int, n: int, k: int) -> float:
        wq, sc, bi = _u32(wq), _f16(scales), _f16(biases)
        return self.lib.zo_weight_affine(_ptr(wq), _ptr(sc), _ptr(bi), K, n, k)

    def dequant_affine(self, wq, scales, biases, N: int, K: int) -> np.ndarray:
        wq, sc, bi = _u32(wq), _f16(scales), _f16(biases)
        out = np.empty((N, K), dtype=np.float64)
        self.lib.zo_dequant_affine(_ptr(wq), _ptr(sc), _ptr(bi), N, K, _ptr(out))
        return out

    def gemv_affine(self, wq, scales, biases, x, N: int, K: int, rows=None):
        """y_ref, Sa (both [M, N] or [M, len(rows)] fp64); Sa = sum |x| (|s| q + |b|)."""
        wq, sc, bi, xx = _u32(wq), _f16(scales), _f16(biases), _f16(x)
        M = xx.size // K if K else 0
        if rows is None:
            R, rp = N, None
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            R, rp = rows.size, rows
        y = np.empty((M, R), dtype=np.float64)
        S = np.empty((M, R), dtype=np.float64)
        self.lib.zo_gemv_affine_rows(_ptr(wq), _ptr(sc), _ptr(bi), _ptr(xx), M, N, K,
                                     None if rp is None else _ptr(rp), R, _ptr(y), _ptr(S))
        return y, S

    def gate_up_silu_affine(self, wq, scales, biases, x, N2: int, K: int):
        """h_ref, Sh ([M, N2/2] fp64) over interleaved gate/up rows."""
        wq, sc, bi, xx = _u32(wq), _f16(scales), _f16(biases), _f16(x)
        M = xx.size // K if K else 0
        h = np.empty((M, N2 // 2), dtype=np.float64)
        Sh = np.empty((M, N2 // 2), dtype=np.float64)
        self.lib.zo_gate_up_silu_affine(_ptr(wq), _ptr(sc), _ptr(bi), _ptr(xx), M, N2, K, _ptr(h), _ptr(Sh))
        return h, Sh

    def gate_up_silu(self, wq, scales, x, N2: int, K: int, interleaved: bool = True,
                     parts: bool = False):
        """h_ref, Sh ([M, N2/2] fp64); with parts=True also g, u, Sg, Su."""
        wq, sc, xx = _u32(wq), _f16(scales), _f16(x)
        M = xx.size // K if K else 0
        I = N2 // 2
        outs = [np.empty((M, I), dtype=np.float64) for _ in range(6)]
        self.lib.zo_gate_up_silu(_ptr(wq), _ptr(sc), _ptr(xx), M, N2, K, int(interleaved),
                                 *[_ptr(o) for o in outs])
        return tuple(outs) if parts else (outs[0], outs[1])

    # --- MoE --------------------------------------------------------------
    def moe_gate_up(self, wq_bank, sc_bank, E: int, x, N2: int, K: int, ids,
                    interleaved: bool = True):
        """h_ref, Sh ([T, top_k, N2/2] fp64) and the count of invalid ids."""
        wq, sc, xx = _u32(wq_bank), _f16(sc_bank), _f16(x)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        T, top_k = ids.shape
        I = N2 // 2
        h = np.empty((T, top_k, I), dtype=np.float64)
        Sh = np.empty((T, top_k, I), dtype=np.float64)
        bad = self.lib.zo_moe_gate_up(_ptr(wq), _ptr(sc), E, _ptr(xx), T, N2, K, _ptr(ids),
                                      top_k, int(interleaved), _ptr(h), _ptr(Sh))
        return h, Sh, int(bad)

    def moe_down_combine(self, wq_bank, sc_bank, E: int, h, r, N: int, K: int, ids):
        """y_ref, S ([T, N] fp64) and the count of invalid ids. h is f16 [T, top_k, K]."""
        wq, sc, hh = _u32(wq_bank), _f16(sc_bank), _f16(h)
        rr = np.ascontiguousarray(r, dtype=np.float32)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        T, top_k = ids.shape
        y = np.empty((T, N), dtype=np.float64)
        S = np.empty((T, N), dtype=np.float64)
        bad = self.lib.zo_moe_down_combine(_ptr(wq), _ptr(sc), E, _ptr(hh), _ptr(rr), T, N, K,
                                           _ptr(ids), top_k, _ptr(y), _ptr(S))
        return y, S, int(bad)

    def moe_gate_up_affine(self, wq_bank, sc_bank, bi_bank, E: int, x, N2: int, K: int, ids):
        """h_ref, Sh ([T, top_k, N2/2]) and the count of invalid ids; affine banks."""
        wq, sc, bi, xx = _u32(wq_bank), _f16(sc_bank), _f16(bi_bank), _f16(x)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        T, top_k = ids.shape
        h = np.empty((T, top_k, N2 // 2), dtype=np.float64)
        Sh = np.empty((T, top_k, N2 // 2), dtype=np.float64)
        bad = self.lib.zo_moe_gate_up_affine(_ptr(wq), _ptr(sc), _ptr(bi), E, _ptr(xx), T, N2, K, _ptr(ids),
                                             top_k, _ptr(h), _ptr(Sh))
        return h, Sh, int(bad)

    def moe_down_combine_affine(self, wq_bank, sc_bank, bi_bank, E: int, h, r, N: int, K: int, ids):
        """y_ref, Sa ([T, N]) and the count of invalid ids; affine banks, h f16 [T, top_k, K]."""
        wq, sc, bi, hh = _u32(wq_bank), _f16(sc_bank), _f16(bi_bank), _f16(h)
        rr = np.ascontiguousarray(r, dtype=np.float32)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        T, top_k = ids.shape
        y = np.empty((T, N), dtype=np.float64)
        S = np.empty((T, N), dtype=np.float64)
        bad = self.lib.zo_moe_down_combine_affine(_ptr(wq), _ptr(sc), _ptr(bi), E, _ptr(hh), _ptr(rr), T, N, K,
                                                  _ptr(ids), top_k, _ptr(y), _ptr(S))
        return y, S, int(bad)

    # --- GEMV + residual add + RMSNorm -----------------------------------------
    def gemv_add_rmsnorm(self, wq, scales, x, resid, gamma, eps: float, N: int, K: int):
        """(r, out, S, Tn), each [M, N] fp64: r = resid + x W^T, out =
        RMSNorm(r) * gamma, S the dot products' tolerance scale and Tn the
        propagated bound on out."""
        wq, sc, xx = _u32(wq), _f16(scales), _f16(x)
        rr, gg = _f16(resid), _f16(gamma)
        M = xx.size // K if K else 0
        r, out, S, Tn = (np.empty((M, N), dtype=np.float64) for _ in range(4))
        self.lib.zo_gemv_add_rmsnorm(_ptr(wq), _ptr(sc), _ptr(xx), _ptr(rr), _ptr(gg), float(eps), M, N, K,
                                     _ptr(r), _ptr(out), _ptr(S), _ptr(Tn))
        return r, out, S, Tn

    # --- QKV + RoPE + KV append ------------------------------------------------
    def qkv_rope(self, wq, scales, x, K: int, H: int, Hkv: int, D: int, base: float, pos):
        """dict of fp64 arrays: q [M, H D], k and v [M, Hkv D] (the token's
        cache rows), S_q/S_k/S_v (dot-product scales, summed over a RoPE
        pair), A_q/A_k/A_v (|a| + |b| of the pair, |y| for V)."""
        wq, sc, xx = _u32(wq), _f16(scales), _f16(x)
        p = np.ascontiguousarray(pos, dtype=np.int32)
        M = xx.size // K
        o = {n: np.empty((M, (H if n.endswith("q") else Hkv) * D), dtype=np.float64)
             for n in ("q", "k", "v", "S_q", "S_k", "S_v", "A_q", "A_k", "A_v")}
        self.lib.zo_qkv_rope(_ptr(wq), _ptr(sc), _ptr(xx), M, K, H, Hkv, D, float(base), _ptr(p),
                             *[_ptr(o[n]) for n in ("q", "k", "v", "S_q", "S_k", "S_v", "A_q", "A_k", "A_v")])
        return o

    # --- LM head ------------------------------------------------------------
    def argmax(self, y) -> np.ndarray:
        """Per row of y [M, N] (taken as fp64): the lowest index of the largest
        value, a NaN counting as the largest."""
        yy = np.ascontiguousarray(np.atleast_2d(y), dtype=np.float64)
        M, N = yy.shape
        idx = np.empty(M, dtype=np.int32)
        self.lib.zo_argmax(_ptr(yy), M, N, _ptr(idx))
        return idx

    def num_threads(self) -> int:
        return int(self.lib.zo_num_threads())

    def set_num_threads(self, n: int) -> int:
        """Threads of the oracle's parallel loops (timing only); returns the
        count in effect."""
        return int(self.lib.zo_set_num_threads(int(n)))


_DEFAULT = None


def get() -> Oracle:
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle(0)
    return _DEFAULT


def tolerance(y_ref, S):
    """Parity bound |y - y_ref| <= 2^-10 |y_ref| + 1e-4 S + 2^-25 (fp64).

    The outputs are f16. Below 2^-14 the f16 grid is fixed-point (spacing
    2^-24), so rounding the exact result to f16 can move it by up to 2^-25
    there, which the relative term does not cover; the absolute term admits
    the correctly rounded f16 answer everywhere and changes nothing above
    the subnormal range (2^-25 < 2^-10 |y| for |y| >= 2^-15)."""
    return np.ldexp(np.abs(y_ref), -10) + 1e-4 * S + np.ldexp(1.0, -25)
