"""Thin Python binding over the libgq4 C ABI (``include/gq4.h``).

Argument marshalling only: each function checks that the torch tensors it is
given are CUDA, contiguous and of the right dtype and shape, then passes their
device pointers and the current CUDA stream to the C entry point of the same
name.  Every step of the computation runs in the library's sm_103a kernels.
There is no CPU fallback: importing this module raises if ``libgq4.so`` has
not been built (``python -m int4_group_quantized_quant_gb300.build``).
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgq4.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -m int4_group_quantized_quant_gb300.build)")

lib = ctypes.CDLL(LIB_PATH)

MAX_LANES = 32

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_ALIAS = 3
ERR_CUDA = 4
ERR_MISALIGNED = 5

_vp = ctypes.c_void_p
_i = ctypes.c_int


class Norm(ctypes.Structure):
    """``gq4_norm``: the optional residual + RMSNorm prologue."""
    _fields_ = [("A_b", _vp), ("W_norm", _vp), ("eps", ctypes.c_float),
                ("residual_out", _vp), ("norm_out", _vp)]


_NormP = ctypes.POINTER(Norm)

OP_MATVEC, OP_QUAD, OP_NORM, OP_GATED = 0, 1, 2, 3


class Call(ctypes.Structure):
    """``gq4_call``: one one-lane call of a sequence (``gq4_run_sequence``)."""
    _fields_ = [("op", _i), ("K", _i), ("N", _i), ("group_size", _i),
                ("n0", _i), ("n1", _i), ("n2", _i),
                ("A", _vp), ("Bq", _vp * 2), ("scales", _vp * 2), ("zeros", _vp * 2),
                ("out", _vp * 4), ("has_norm", _i), ("norm", Norm)]

_SIGS = {
    "gq4_matvec": [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp],
    "gq4_quad_matvec": [_i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                        _vp, _vp],
    "gq4_norm_matvec": [_i, _i, _i, _i, _NormP, _vp, _vp, _vp, _vp, _vp, _vp],
    "gq4_gated_matvec": [_i, _i, _i, _i, _NormP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                         _vp],
    "gq4_dual_matvec": [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "gq4_sigmoid_gated_matvec": [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "gq4_swiglu_gated_matvec": [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "gq4_run_sequence": [ctypes.POINTER(Call), _i, _vp, _vp],
    "gq4_run_sequence_static": [ctypes.POINTER(Call), _i, _vp],
    "gq4_sequence_launches": [ctypes.POINTER(Call), _i, ctypes.POINTER(_i)],
    "gq4_gemm": [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp],
    "gq4_quantize": [_i, _i, _i, _vp, _vp, _vp, _vp, _vp],
    "gq4_from_mlx": [_i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "gq4_embedding": [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp],
    "gq4_unpack": [_i, _i, _vp, _vp, _vp],
    "gq4_dequant": [_i, _i, _i, _vp, _vp, _vp, _vp, _vp],
}
for _name, _args in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype = _i
    _fn.argtypes = _args
lib.gq4_status_string.restype = ctypes.c_char_p
lib.gq4_status_string.argtypes = [_i]
lib.gq4_version.restype = _i
lib.gq4_version.argtypes = []
lib.gq4_device_error.restype = _i
lib.gq4_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), _i]
lib.gq4_sequence_workspace_bytes.restype = ctypes.c_size_t
lib.gq4_sequence_workspace_bytes.argtypes = []
lib.gq4_gemm_workspace_bytes.restype = ctypes.c_size_t
lib.gq4_gemm_workspace_bytes.argtypes = [_i, _i]

EXPORTED = list(_SIGS) + ["gq4_status_string", "gq4_version", "gq4_device_error",
                          "gq4_sequence_workspace_bytes", "gq4_gemm_workspace_bytes"]


class GQ4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib.gq4_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


def _check(status: int, where: str):
    if status != OK:
        raise GQ4Error(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtypes, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")


_F32 = (torch.float32,)
_WORDS = (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())


def _weights(Bq, scales, zeros, K, group_size, tag=""):
    N = Bq.shape[0]
    _need(Bq, "Bq" + tag, _WORDS, (N, K // 8))
    _need(scales, "scales" + tag, _F32, (N, K // group_size))
    _need(zeros, "zeros" + tag, _F32, (N, K // group_size))
    return N


def _lanes(A):
    _need(A, "A", _F32)
    if A.dim() != 2:
        raise ValueError("A must be [M, K]")
    return A.shape


def matvec(A, Bq, scales, zeros, group_size, C=None, stream=None):
    """C [M, N] = A [M, K] times the int4 matrix (Bq [N, K/8], scales/zeros [N, K/gs])."""
    M, K = _lanes(A)
    N = _weights(Bq, scales, zeros, K, group_size)
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _need(C, "C", _F32, (M, N))
    _check(lib.gq4_matvec(M, K, N, group_size, _ptr(A), _ptr(Bq), _ptr(scales), _ptr(zeros),
                          _ptr(C), _stream(stream)), "gq4_matvec")
    return C


def gemm_workspace_bytes(M, K) -> int:
    return int(lib.gq4_gemm_workspace_bytes(M, K))


def gemm(A, Bq, scales, zeros, group_size, C=None, workspace=None, stream=None):
    """C [M, N] = A [M, K] times the int4 matrix, any M >= 1 (gq4_gemm; bf16 tensor cores).
    ``workspace`` (a CUDA tensor of at least gemm_workspace_bytes(M, K) bytes) enables the
    GEMM kernel for M > 32; ``workspace=False`` runs the row chunks without one."""
    _need(A, "A", _F32)
    if A.dim() != 2:
        raise ValueError("A must be [M, K]")
    M, K = A.shape
    N = _weights(Bq, scales, zeros, K, group_size)
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _need(C, "C", _F32, (M, N))
    if workspace is None:
        workspace = torch.empty(gemm_workspace_bytes(M, K), dtype=torch.uint8, device=A.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not False:
        if not (isinstance(workspace, torch.Tensor) and workspace.is_cuda and workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _check(lib.gq4_gemm(M, K, N, group_size, _ptr(A), _ptr(Bq), _ptr(scales), _ptr(zeros),
                        _ptr(C), ws_ptr, ws_bytes, _stream(stream)), "gq4_gemm")
    return C


def quad_matvec(A, Bq, scales, zeros, group_size, n0, n1, n2, outs=None, stream=None):
    """Quad-output matvec; returns the four segment outputs [M, len_i] (empty ones have 0 columns)."""
    M, K = _lanes(A)
    N = _weights(Bq, scales, zeros, K, group_size)
    lens = [n0, n1 - n0, n2 - n1, N - n2]
    if outs is None:
        outs = [torch.empty((M, max(n, 0)), dtype=torch.float32, device=A.device) for n in lens]
    ptrs = []
    for i, (o, n) in enumerate(zip(outs, lens)):
        if o is None:
            ptrs.append(None)
            continue
        _need(o, f"out{i}", _F32, (M, n) if n >= 0 else None)
        ptrs.append(_ptr(o) if o.numel() else None)
    _check(lib.gq4_quad_matvec(M, K, N, group_size, n0, n1, n2, _ptr(A), _ptr(Bq), _ptr(scales),
                               _ptr(zeros), *ptrs, _stream(stream)), "gq4_quad_matvec")
    return outs


def _norm_struct(M, K, W_norm, eps, A_b, residual_out, norm_out):
    _need(W_norm, "W_norm", _F32, (K,))
    for name, t in (("A_b", A_b), ("residual_out", residual_out), ("norm_out", norm_out)):
        if t is not None:
            _need(t, name, _F32, (M, K))
    return Norm(_ptr(A_b), _ptr(W_norm), float(eps), _ptr(residual_out), _ptr(norm_out))


def norm_matvec(A, Bq, scales, zeros, group_size, W_norm, eps=1e-6, A_b=None,
                residual_out=None, norm_out=None, C=None, stream=None):
    """C = matvec of RMSNorm(A + A_b) * W_norm; optionally writes residual_out / norm_out."""
    M, K = _lanes(A)
    N = _weights(Bq, scales, zeros, K, group_size)
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _need(C, "C", _F32, (M, N))
    nrm = _norm_struct(M, K, W_norm, eps, A_b, residual_out, norm_out)
    _check(lib.gq4_norm_matvec(M, K, N, group_size, ctypes.byref(nrm), _ptr(A), _ptr(Bq),
                               _ptr(scales), _ptr(zeros), _ptr(C), _stream(stream)),
           "gq4_norm_matvec")
    return C


def gated_matvec(A, Bq_gate, scales_gate, zeros_gate, Bq_up, scales_up, zeros_up, group_size,
                 W_norm=None, eps=1e-6, A_b=None, residual_out=None, norm_out=None, out=None,
                 stream=None):
    """out = silu(a . Wg) * (a . Wu), a = A or RMSNorm(A + A_b) * W_norm when W_norm is given."""
    M, K = _lanes(A)
    N = _weights(Bq_gate, scales_gate, zeros_gate, K, group_size, "_gate")
    if _weights(Bq_up, scales_up, zeros_up, K, group_size, "_up") != N:
        raise ValueError("gate and up must have the same N")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _need(out, "out", _F32, (M, N))
    nrm = None
    if W_norm is not None:
        nrm = _norm_struct(M, K, W_norm, eps, A_b, residual_out, norm_out)
    elif A_b is not None or residual_out is not None or norm_out is not None:
        raise ValueError("A_b / residual_out / norm_out need W_norm")
    _check(lib.gq4_gated_matvec(M, K, N, group_size, ctypes.byref(nrm) if nrm else None,
                                _ptr(A), _ptr(Bq_gate), _ptr(scales_gate), _ptr(zeros_gate),
                                _ptr(Bq_up), _ptr(scales_up), _ptr(zeros_up), _ptr(out),
                                _stream(stream)), "gq4_gated_matvec")
    return out


def dual_matvec(A, Bq0, scales0, zeros0, Bq1, scales1, zeros1, group_size, C0=None, C1=None,
                stream=None):
    """(C0, C1) = (A . W0, A . W1): two projections sharing the input (gq4_dual_matvec)."""
    M, K = _lanes(A)
    N = _weights(Bq0, scales0, zeros0, K, group_size, "0")
    if _weights(Bq1, scales1, zeros1, K, group_size, "1") != N:
        raise ValueError("both matrices must have the same N")
    if C0 is None:
        C0 = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if C1 is None:
        C1 = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _need(C0, "C0", _F32, (M, N))
    _need(C1, "C1", _F32, (M, N))
    _check(lib.gq4_dual_matvec(M, K, N, group_size, _ptr(A), _ptr(Bq0), _ptr(scales0),
                               _ptr(zeros0), _ptr(Bq1), _ptr(scales1), _ptr(zeros1), _ptr(C0),
                               _ptr(C1), _stream(stream)), "gq4_dual_matvec")
    return C0, C1


def _gated_input(fn, name, X, G, Bq, scales, zeros, group_size, C, stream):
    M, K = _lanes(X)
    _need(G, "G", _F32, (M, K))
    N = _weights(Bq, scales, zeros, K, group_size)
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=X.device)
    _need(C, "C", _F32, (M, N))
    _check(fn(M, K, N, group_size, _ptr(X), _ptr(G), _ptr(Bq), _ptr(scales), _ptr(zeros), _ptr(C),
              _stream(stream)), name)
    return C


def sigmoid_gated_matvec(X, G, Bq, scales, zeros, group_size, C=None, stream=None):
    """C = (X * sigmoid(G)) . W (gq4_sigmoid_gated_matvec)."""
    return _gated_input(lib.gq4_sigmoid_gated_matvec, "gq4_sigmoid_gated_matvec", X, G, Bq, scales,
                        zeros, group_size, C, stream)


def swiglu_gated_matvec(X, G, Bq, scales, zeros, group_size, C=None, stream=None):
    """C = (silu(G) * X) . W (gq4_swiglu_gated_matvec)."""
    return _gated_input(lib.gq4_swiglu_gated_matvec, "gq4_swiglu_gated_matvec", X, G, Bq, scales,
                        zeros, group_size, C, stream)


# ---------------------------------------------------------------------------
# Producing the format
# ---------------------------------------------------------------------------

def _format_outputs(N, K, group_size, device, Bq, scales, zeros):
    G = K // group_size
    if Bq is None:
        Bq = torch.empty((N, K // 8), dtype=torch.int32, device=device)
    if scales is None:
        scales = torch.empty((N, G), dtype=torch.float32, device=device)
    if zeros is None:
        zeros = torch.empty((N, G), dtype=torch.float32, device=device)
    _need(Bq, "Bq", _WORDS, (N, K // 8))
    _need(scales, "scales", _F32, (N, G))
    _need(zeros, "zeros", _F32, (N, G))
    return Bq, scales, zeros


def quantize(W, group_size, Bq=None, scales=None, zeros=None, stream=None):
    """(Bq, scales, zeros) of W f32 [N, K] (gq4_quantize: min/max asymmetric per group)."""
    _need(W, "W", _F32)
    if W.dim() != 2:
        raise ValueError("W must be [N, K]")
    N, K = W.shape
    if K % 8 != 0 or group_size <= 0:
        raise ValueError("K must be a multiple of 8 and group_size positive")
    Bq, scales, zeros = _format_outputs(N, K, group_size, W.device, Bq, scales, zeros)
    _check(lib.gq4_quantize(K, N, group_size, _ptr(W), _ptr(Bq), _ptr(scales), _ptr(zeros),
                            _stream(stream)), "gq4_quantize")
    return Bq, scales, zeros


def from_mlx(packed, mlx_scales, mlx_biases, group_size, Bq=None, scales=None, zeros=None,
             stream=None):
    """(Bq, scales, zeros) of an MLX affine int4 matrix (gq4_from_mlx); pass Bq=packed to
    convert the words in place."""
    _need(packed, "packed", _WORDS)
    if packed.dim() != 2:
        raise ValueError("packed must be [N, K/8]")
    N, K = packed.shape[0], packed.shape[1] * 8
    if group_size <= 0 or K % group_size != 0:
        raise ValueError("K must be a multiple of group_size")
    G = K // group_size
    _need(mlx_scales, "mlx_scales", _F32, (N, G))
    _need(mlx_biases, "mlx_biases", _F32, (N, G))
    Bq, scales, zeros = _format_outputs(N, K, group_size, packed.device, Bq, scales, zeros)
    _check(lib.gq4_from_mlx(K, N, group_size, _ptr(packed), _ptr(mlx_scales), _ptr(mlx_biases),
                            _ptr(Bq), _ptr(scales), _ptr(zeros), _stream(stream)),
           "gq4_from_mlx")
    return Bq, scales, zeros


def embedding(ids, Bq, scales, zeros, group_size, out=None, stream=None):
    """out [T, K] = the int4 table's rows ids dequantized (gq4_embedding)."""
    _need(ids, "ids", (torch.int32,))
    if ids.dim() != 1:
        raise ValueError("ids must be [T]")
    V, K = Bq.shape[0], Bq.shape[1] * 8
    _weights(Bq, scales, zeros, K, group_size)
    T = ids.shape[0]
    if out is None:
        out = torch.empty((T, K), dtype=torch.float32, device=Bq.device)
    _need(out, "out", _F32, (T, K))
    _check(lib.gq4_embedding(T, K, V, group_size, _ptr(ids), _ptr(Bq), _ptr(scales),
                             _ptr(zeros), _ptr(out), _stream(stream)), "gq4_embedding")
    return out


# ---------------------------------------------------------------------------
# Call sequences (one lane)
# ---------------------------------------------------------------------------

class SeqCall:
    """One call of a sequence: the C descriptor plus the tensors it points to
    (kept alive while the descriptor is in use)."""

    def __init__(self, desc: Call, tensors):
        self.desc = desc
        self.tensors = tensors


def _one_lane(A):
    M, K = _lanes(A)
    if M != 1:
        raise ValueError("sequence calls take one lane (A of shape [1, K])")
    return K


def _seq_norm(desc, K, W_norm, eps, A_b, residual_out, norm_out):
    desc.has_norm = 1
    desc.norm = _norm_struct(1, K, W_norm, eps, A_b, residual_out, norm_out)


def seq_matvec(A, Bq, scales, zeros, group_size, C):
    """Sequence entry of gq4_matvec (C [1, N] must be given)."""
    K = _one_lane(A)
    N = _weights(Bq, scales, zeros, K, group_size)
    _need(C, "C", _F32, (1, N))
    d = Call(op=OP_MATVEC, K=K, N=N, group_size=group_size, A=_ptr(A))
    d.Bq[0], d.scales[0], d.zeros[0], d.out[0] = _ptr(Bq), _ptr(scales), _ptr(zeros), _ptr(C)
    return SeqCall(d, (A, Bq, scales, zeros, C))


def seq_quad(A, Bq, scales, zeros, group_size, n0, n1, n2, outs):
    """Sequence entry of gq4_quad_matvec (outs: four [1, len] tensors or None for empty ones)."""
    K = _one_lane(A)
    N = _weights(Bq, scales, zeros, K, group_size)
    lens = [n0, n1 - n0, n2 - n1, N - n2]
    d = Call(op=OP_QUAD, K=K, N=N, group_size=group_size, n0=n0, n1=n1, n2=n2, A=_ptr(A))
    d.Bq[0], d.scales[0], d.zeros[0] = _ptr(Bq), _ptr(scales), _ptr(zeros)
    for i, (o, n) in enumerate(zip(outs, lens)):
        if o is not None:
            _need(o, f"out{i}", _F32, (1, n))
        d.out[i] = _ptr(o)
    return SeqCall(d, (A, Bq, scales, zeros, *outs))


def seq_norm(A, Bq, scales, zeros, group_size, W_norm, C, eps=1e-6, A_b=None,
             residual_out=None, norm_out=None):
    """Sequence entry of gq4_norm_matvec."""
    K = _one_lane(A)
    N = _weights(Bq, scales, zeros, K, group_size)
    _need(C, "C", _F32, (1, N))
    d = Call(op=OP_NORM, K=K, N=N, group_size=group_size, A=_ptr(A))
    d.Bq[0], d.scales[0], d.zeros[0], d.out[0] = _ptr(Bq), _ptr(scales), _ptr(zeros), _ptr(C)
    _seq_norm(d, K, W_norm, eps, A_b, residual_out, norm_out)
    return SeqCall(d, (A, Bq, scales, zeros, C, W_norm, A_b, residual_out, norm_out))


def seq_gated(A, Bq_gate, scales_gate, zeros_gate, Bq_up, scales_up, zeros_up, group_size, out,
              W_norm=None, eps=1e-6, A_b=None, residual_out=None, norm_out=None):
    """Sequence entry of gq4_gated_matvec."""
    K = _one_lane(A)
    N = _weights(Bq_gate, scales_gate, zeros_gate, K, group_size, "_gate")
    if _weights(Bq_up, scales_up, zeros_up, K, group_size, "_up") != N:
        raise ValueError("gate and up must have the same N")
    _need(out, "out", _F32, (1, N))
    d = Call(op=OP_GATED, K=K, N=N, group_size=group_size, A=_ptr(A))
    d.Bq[0], d.scales[0], d.zeros[0] = _ptr(Bq_gate), _ptr(scales_gate), _ptr(zeros_gate)
    d.Bq[1], d.scales[1], d.zeros[1] = _ptr(Bq_up), _ptr(scales_up), _ptr(zeros_up)
    d.out[0] = _ptr(out)
    if W_norm is not None:
        _seq_norm(d, K, W_norm, eps, A_b, residual_out, norm_out)
    elif A_b is not None or residual_out is not None or norm_out is not None:
        raise ValueError("A_b / residual_out / norm_out need W_norm")
    return SeqCall(d, (A, Bq_gate, scales_gate, zeros_gate, Bq_up, scales_up, zeros_up, out,
                       W_norm, A_b, residual_out, norm_out))


def sequence_workspace(device=None):
    """A zero-filled workspace for run_sequence (reusable on one stream)."""
    n = int(lib.gq4_sequence_workspace_bytes())
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def run_sequence(calls, workspace, stream=None):
    """Run the calls in order as one persistent launch (gq4_run_sequence)."""
    _need(workspace, "workspace", (torch.uint8,), (int(lib.gq4_sequence_workspace_bytes()),))
    arr = (Call * max(len(calls), 1))(*[c.desc for c in calls])
    _check(lib.gq4_run_sequence(arr, len(calls), _ptr(workspace), _stream(stream)),
           "gq4_run_sequence")


def sequence_launches(calls) -> int:
    """Persistent launches the calls would take (gq4_sequence_launches; 0 = run call by call)."""
    arr = (Call * max(len(calls), 1))(*[c.desc for c in calls])
    n = _i(0)
    _check(lib.gq4_sequence_launches(arr, len(calls), ctypes.byref(n)), "gq4_sequence_launches")
    return int(n.value)


def run_sequence_static(calls, stream=None):
    """Run the calls in order with the library's fixed scratch (gq4_run_sequence_static)."""
    arr = (Call * max(len(calls), 1))(*[c.desc for c in calls])
    _check(lib.gq4_run_sequence_static(arr, len(calls), _stream(stream)), "gq4_run_sequence_static")


def unpack(Bq, K, q=None, stream=None):
    """Integer unpack test kernel: codes [N, K] uint8."""
    N = Bq.shape[0]
    _need(Bq, "Bq", _WORDS, (N, K // 8))
    if q is None:
        q = torch.empty((N, K), dtype=torch.uint8, device=Bq.device)
    _need(q, "q", (torch.uint8,), (N, K))
    _check(lib.gq4_unpack(K, N, _ptr(Bq), _ptr(q), _stream(stream)), "gq4_unpack")
    return q


def dequant(Bq, scales, zeros, K, group_size, W=None, stream=None):
    """Dequant test kernel: W [N, K] = fl32(fl32(q - zero) * scale)."""
    N = _weights(Bq, scales, zeros, K, group_size)
    if W is None:
        W = torch.empty((N, K), dtype=torch.float32, device=Bq.device)
    _need(W, "W", _F32, (N, K))
    _check(lib.gq4_dequant(K, N, group_size, _ptr(Bq), _ptr(scales), _ptr(zeros), _ptr(W),
                           _stream(stream)), "gq4_dequant")
    return W


def device_error(clear: bool = True) -> int:
    """The library's sticky device error bits (bit 0: the one-lane kernel, bit 1: the
    tensor-core kernel, bit 2: a call sequence gave up a bounded wait; bit 3: the
    quantizer met a non-finite group; bit 4: the embedding gather met an id outside
    its table)."""
    bits = ctypes.c_uint(0)
    _check(lib.gq4_device_error(ctypes.byref(bits), int(clear)), "gq4_device_error")
    return int(bits.value)


def version() -> int:
    return int(lib.gq4_version())
