"""ctypes wrapper around the C oracle (``gq4_oracle.c``).

TEST INFRASTRUCTURE ONLY (see the package docstring).  Each wrapper takes and
returns numpy arrays; the arithmetic is all in C.  ``build()`` compiles the
shared library with gcc (``-ffp-contract=off`` so no step is fused into an
FMA, identical results on x86-64 and aarch64).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gq4_oracle.c")
_HDR = os.path.join(_HERE, "gq4_oracle.h")
_LIB_PATH = os.path.join(_HERE, "libgq4_oracle.so")
_lock = threading.Lock()
_lib = None

_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i32p = ctypes.POINTER(ctypes.c_int)
_int = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile ``libgq4_oracle.so`` next to the sources (if stale) and return its path."""
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= newest_src):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Load a compiled oracle library from ``path`` and declare its signatures."""
    lib = ctypes.CDLL(path)
    sig = {
        "gq4o_nibble": (_int, [_u32p, _int, _int, _int]),
        "gq4o_unpack": (_int, [_int, _int, _u32p, _u8p]),
        "gq4o_pack": (_int, [_int, _int, _u8p, _u32p]),
        "gq4o_dequant_f64": (_int, [_int, _int, _int, _u32p, _f32p, _f32p, _f64p]),
        "gq4o_dequant_f32": (_int, [_int, _int, _int, _u32p, _f32p, _f32p, _f32p]),
        "gq4o_matvec": (_int, [_int, _int, _int, _int, _f32p, _u32p, _f32p, _f32p,
                               _f64p, _f64p]),
        "gq4o_matvec_cols": (_int, [_int, _int, _int, _f64p, _u32p, _f32p, _f32p,
                                    _int, _i32p, _f64p, _f64p]),
        "gq4o_quad_matvec": (_int, [_int, _int, _int, _int, _int, _int, _int, _f32p,
                                    _u32p, _f32p, _f32p] + [_f64p] * 8),
        "gq4o_norm": (_int, [_int, _int, _f32p, _f32p, _f32p, ctypes.c_float, _f32p,
                             _f64p, _f64p]),
        "gq4o_norm_matvec": (_int, [_int, _int, _int, _int, _f32p, _f32p, _f32p,
                                    ctypes.c_float, _u32p, _f32p, _f32p, _f64p,
                                    _f64p, _f32p, _f64p]),
        "gq4o_gated_input_matvec": (_int, [_int, _int, _int, _int, _int, _f32p, _f32p,
                                           _u32p, _f32p, _f32p, _f64p, _f64p, _f64p]),
        "gq4o_quantize": (_int, [_int, _int, _int, _f32p, _u32p, _f32p, _f32p, _i32p]),
        "gq4o_mlx_dequant_f64": (_int, [_int, _int, _int, _u32p, _f32p, _f32p, _f64p]),
        "gq4o_from_mlx": (_int, [_int, _int, _int, _u32p, _f32p, _f32p, _u32p, _f32p,
                                 _f32p]),
        "gq4o_embedding": (_int, [_int, _int, _int, _int, _i32p, _u32p, _f32p, _f32p, _f32p,
                                  _i32p]),
        "gq4o_gated_matvec": (_int, [_int, _int, _int, _int, _f32p, _f32p, _f32p,
                                     ctypes.c_float, _u32p, _f32p, _f32p, _u32p,
                                     _f32p, _f32p, _f64p, _f64p, _f64p, _f64p,
                                     _f64p, _f32p, _f64p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load():
    """The default oracle (built from this folder's sources on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(load_library(build()))
        return _lib


def _ptr(arr, ctype):
    if arr is None:
        return None
    return arr.ctypes.data_as(ctype)


def _c(arr, dtype):
    """Contiguous array of the exact dtype (no silent conversion of the caller's data)."""
    a = np.asarray(arr)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid argument")


class Oracle:
    """The oracle's functions bound to one loaded copy of the C library."""

    def __init__(self, lib):
        self.lib = lib

    def nibble(self, Bq, K, n, k) -> int:
        Bq = _c(Bq, np.uint32)
        return int(self.lib.gq4o_nibble(_ptr(Bq, _u32p), K, n, k))

    def unpack(self, Bq, K, N):
        """q[n, k] as uint8 [N, K]."""
        Bq = _c(Bq, np.uint32)
        q = np.empty((N, K), np.uint8)
        _check(self.lib.gq4o_unpack(K, N, _ptr(Bq, _u32p), _ptr(q, _u8p)), "unpack")
        return q

    def pack(self, q):
        """Pack uint8 codes [N, K] (0..15) into u32 words [N, K/8]."""
        q = _c(q, np.uint8)
        N, K = q.shape
        Bq = np.empty((N, K // 8), np.uint32)
        _check(self.lib.gq4o_pack(K, N, _ptr(q, _u8p), _ptr(Bq, _u32p)), "pack")
        return Bq

    def dequant_f64(self, Bq, scales, zeros, K, N, gs):
        Bq, s, z = _c(Bq, np.uint32), _c(scales, np.float32), _c(zeros, np.float32)
        W = np.empty((N, K), np.float64)
        _check(self.lib.gq4o_dequant_f64(K, N, gs, _ptr(Bq, _u32p), _ptr(s, _f32p),
                                       _ptr(z, _f32p), _ptr(W, _f64p)), "dequant_f64")
        return W

    def dequant_f32(self, Bq, scales, zeros, K, N, gs):
        Bq, s, z = _c(Bq, np.uint32), _c(scales, np.float32), _c(zeros, np.float32)
        W = np.empty((N, K), np.float32)
        _check(self.lib.gq4o_dequant_f32(K, N, gs, _ptr(Bq, _u32p), _ptr(s, _f32p),
                                       _ptr(z, _f32p), _ptr(W, _f32p)), "dequant_f32")
        return W

    def matvec(self, A, Bq, scales, zeros, K, N, gs):
        """(C, S) with C[m, n] = sum_k A[m, k] w(n, k) and S the absolute sum, both [M, N] f64."""
        A = _c(A, np.float32).reshape(-1, K)
        M = A.shape[0]
        Bq, s, z = _c(Bq, np.uint32), _c(scales, np.float32), _c(zeros, np.float32)
        C = np.empty((M, N), np.float64)
        S = np.empty((M, N), np.float64)
        _check(self.lib.gq4o_matvec(M, K, N, gs, _ptr(A, _f32p), _ptr(Bq, _u32p), _ptr(s, _f32p),
                                  _ptr(z, _f32p), _ptr(C, _f64p), _ptr(S, _f64p)), "matvec")
        return C, S

    def dot_cols(self, a, Bq, scales, zeros, K, gs, cols):
        """(C, S) [M, len(cols)] for double activations a [M, K] on the listed columns."""
        a = np.ascontiguousarray(np.asarray(a, np.float64)).reshape(-1, K)
        M = a.shape[0]
        cols = np.ascontiguousarray(np.asarray(cols, np.int32))
        Bq, s, z = _c(Bq, np.uint32), _c(scales, np.float32), _c(zeros, np.float32)
        C = np.empty((M, len(cols)), np.float64)
        S = np.empty((M, len(cols)), np.float64)
        _check(self.lib.gq4o_matvec_cols(M, K, gs, _ptr(a, _f64p), _ptr(Bq, _u32p), _ptr(s, _f32p),
                                       _ptr(z, _f32p), len(cols), _ptr(cols, _i32p),
                                       _ptr(C, _f64p), _ptr(S, _f64p)), "matvec_cols")
        return C, S

    def quad_matvec(self, A, Bq, scales, zeros, K, N, gs, n0, n1, n2):
        """([out0..out3], [S0..S3]) with out_i [M, len_i] f64."""
        A = _c(A, np.float32).reshape(-1, K)
        M = A.shape[0]
        Bq, s, z = _c(Bq, np.uint32), _c(scales, np.float32), _c(zeros, np.float32)
        lens = [n0, n1 - n0, n2 - n1, N - n2]
        outs = [np.empty((M, max(n, 0)), np.float64) for n in lens]
        sabs = [np.empty((M, max(n, 0)), np.float64) for n in lens]
        ptrs = [_ptr(o, _f64p) if o.size else None for o in outs]
        sptrs = [_ptr(o, _f64p) if o.size else None for o in sabs]
        _check(self.lib.gq4o_quad_matvec(M, K, N, gs, n0, n1, n2, _ptr(A, _f32p), _ptr(Bq, _u32p),
                                       _ptr(s, _f32p), _ptr(z, _f32p), *ptrs, *sptrs), "quad")
        return outs, sabs

    def norm(self, A_a, A_b, W_norm, eps, K):
        """(x f32 [M,K], a f64 [M,K], inv_rms f64 [M]) for the RMSNorm prologue."""
        A_a = _c(A_a, np.float32).reshape(-1, K)
        M = A_a.shape[0]
        A_b = None if A_b is None else _c(A_b, np.float32).reshape(M, K)
        W = _c(W_norm, np.float32)
        x = np.empty((M, K), np.float32)
        a = np.empty((M, K), np.float64)
        inv = np.empty((M,), np.float64)
        _check(self.lib.gq4o_norm(M, K, _ptr(A_a, _f32p), _ptr(A_b, _f32p), _ptr(W, _f32p),
                                float(eps), _ptr(x, _f32p), _ptr(a, _f64p), _ptr(inv, _f64p)),
               "norm")
        return x, a, inv

    def norm_matvec(self, A_a, A_b, W_norm, eps, Bq, scales, zeros, K, N, gs):
        """(C, S, residual_out f32, norm_out f64)."""
        A_a = _c(A_a, np.float32).reshape(-1, K)
        M = A_a.shape[0]
        A_b = None if A_b is None else _c(A_b, np.float32).reshape(M, K)
        W = _c(W_norm, np.float32)
        Bq, s, z = _c(Bq, np.uint32), _c(scales, np.float32), _c(zeros, np.float32)
        C = np.empty((M, N), np.float64)
        S = np.empty((M, N), np.float64)
        res = np.empty((M, K), np.float32)
        nout = np.empty((M, K), np.float64)
        _check(self.lib.gq4o_norm_matvec(M, K, N, gs, _ptr(A_a, _f32p), _ptr(A_b, _f32p),
                                       _ptr(W, _f32p), float(eps), _ptr(Bq, _u32p),
                                       _ptr(s, _f32p), _ptr(z, _f32p), _ptr(C, _f64p),
                                       _ptr(S, _f64p), _ptr(res, _f32p), _ptr(nout, _f64p)),
               "norm_matvec")
        return C, S, res, nout

    def gated_matvec(self, A, Bq_g, s_g, z_g, Bq_u, s_u, z_u, K, N, gs,
                     A_b=None, W_norm=None, eps=1e-6):
        """dict(out, g, u, Sg, Su, residual_out, norm_out); norm keys None without W_norm."""
        A = _c(A, np.float32).reshape(-1, K)
        M = A.shape[0]
        A_b = None if A_b is None else _c(A_b, np.float32).reshape(M, K)
        W = None if W_norm is None else _c(W_norm, np.float32)
        arrs = [_c(Bq_g, np.uint32), _c(s_g, np.float32), _c(z_g, np.float32),
                _c(Bq_u, np.uint32), _c(s_u, np.float32), _c(z_u, np.float32)]
        out = {k: np.empty((M, N), np.float64) for k in ("out", "g", "u", "Sg", "Su")}
        res = np.empty((M, K), np.float32) if W is not None else None
        nout = np.empty((M, K), np.float64) if W is not None else None
        _check(self.lib.gq4o_gated_matvec(
            M, K, N, gs, _ptr(A, _f32p), _ptr(A_b, _f32p), _ptr(W, _f32p), float(eps),
            _ptr(arrs[0], _u32p), _ptr(arrs[1], _f32p), _ptr(arrs[2], _f32p),
            _ptr(arrs[3], _u32p), _ptr(arrs[4], _f32p), _ptr(arrs[5], _f32p),
            _ptr(out["out"], _f64p), _ptr(out["g"], _f64p), _ptr(out["u"], _f64p),
            _ptr(out["Sg"], _f64p), _ptr(out["Su"], _f64p), _ptr(res, _f32p),
            _ptr(nout, _f64p)), "gated_matvec")
        out["residual_out"] = res
        out["norm_out"] = nout
        return out


    def gated_input_matvec(self, kind, X, G, Bq, scales, zeros, K, N, gs):
        """(C, S, a) for the gated input a = X*sigmoid(G) ("sigmoid") or silu(G)*X ("swiglu")."""
        k = {"sigmoid": 0, "swiglu": 1}[kind]
        X = _c(X, np.float32).reshape(-1, K)
        M = X.shape[0]
        G = _c(G, np.float32).reshape(M, K)
        Bq, s, z = _c(Bq, np.uint32), _c(scales, np.float32), _c(zeros, np.float32)
        C = np.empty((M, N), np.float64)
        S = np.empty((M, N), np.float64)
        a = np.empty((M, K), np.float64)
        _check(self.lib.gq4o_gated_input_matvec(M, K, N, gs, k, _ptr(X, _f32p), _ptr(G, _f32p),
                                              _ptr(Bq, _u32p), _ptr(s, _f32p), _ptr(z, _f32p),
                                              _ptr(C, _f64p), _ptr(S, _f64p), _ptr(a, _f64p)),
               "gated_input_matvec")
        return C, S, a

    def quantize(self, W, gs):
        """(Bq [N, K/8], scales [N, G], zeros [N, G], bad_groups) for W f32 [N, K]."""
        W = _c(W, np.float32)
        N, K = W.shape
        Bq = np.empty((N, K // 8), np.uint32)
        s = np.empty((N, K // gs), np.float32)
        z = np.empty((N, K // gs), np.float32)
        bad = ctypes.c_int(0)
        _check(self.lib.gq4o_quantize(K, N, gs, _ptr(W, _f32p), _ptr(Bq, _u32p), _ptr(s, _f32p),
                                      _ptr(z, _f32p), ctypes.byref(bad)), "quantize")
        return Bq, s, z, bad.value

    def mlx_dequant_f64(self, packed, mlx_scales, mlx_biases, K, N, gs):
        """W [N, K] (double) = scale * q + bias of an MLX affine int4 matrix."""
        packed = _c(packed, np.uint32)
        ms, mb = _c(mlx_scales, np.float32), _c(mlx_biases, np.float32)
        W = np.empty((N, K), np.float64)
        _check(self.lib.gq4o_mlx_dequant_f64(K, N, gs, _ptr(packed, _u32p), _ptr(ms, _f32p),
                                             _ptr(mb, _f32p), _ptr(W, _f64p)), "mlx_dequant_f64")
        return W

    def from_mlx(self, packed, mlx_scales, mlx_biases, K, N, gs):
        """(Bq, scales, zeros) of this format for an MLX affine int4 matrix."""
        packed = _c(packed, np.uint32)
        ms, mb = _c(mlx_scales, np.float32), _c(mlx_biases, np.float32)
        Bq = np.empty((N, K // 8), np.uint32)
        s = np.empty((N, K // gs), np.float32)
        z = np.empty((N, K // gs), np.float32)
        _check(self.lib.gq4o_from_mlx(K, N, gs, _ptr(packed, _u32p), _ptr(ms, _f32p),
                                      _ptr(mb, _f32p), _ptr(Bq, _u32p), _ptr(s, _f32p),
                                      _ptr(z, _f32p)), "from_mlx")
        return Bq, s, z

    def embedding(self, ids, Bq, scales, zeros, K, gs):
        """(out f32 [T, K], bad_ids): rows ids of the int4 table dequantized in binary32."""
        ids = _c(ids, np.int32).reshape(-1)
        Bq, s, z = _c(Bq, np.uint32), _c(scales, np.float32), _c(zeros, np.float32)
        V = Bq.shape[0]
        out = np.empty((ids.size, K), np.float32)
        bad = ctypes.c_int(0)
        _check(self.lib.gq4o_embedding(ids.size, K, V, gs, _ptr(ids, _i32p), _ptr(Bq, _u32p),
                                       _ptr(s, _f32p), _ptr(z, _f32p), _ptr(out, _f32p),
                                       ctypes.byref(bad)), "embedding")
        return out, bad.value


def _default(name):
    def call(*args, **kwargs):
        return getattr(load(), name)(*args, **kwargs)
    call.__name__ = name
    call.__doc__ = getattr(Oracle, name).__doc__
    return call


nibble = _default("nibble")
unpack = _default("unpack")
pack = _default("pack")
dequant_f64 = _default("dequant_f64")
dequant_f32 = _default("dequant_f32")
matvec = _default("matvec")
dot_cols = _default("dot_cols")
quad_matvec = _default("quad_matvec")
norm = _default("norm")
norm_matvec = _default("norm_matvec")
gated_matvec = _default("gated_matvec")
gated_input_matvec = _default("gated_input_matvec")
quantize = _default("quantize")
mlx_dequant_f64 = _default("mlx_dequant_f64")
from_mlx = _default("from_mlx")
embedding = _default("embedding")
