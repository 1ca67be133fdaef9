"""The C ABI on the host: the library builds, loads, exports every declared
symbol, and rejects invalid arguments before anything is enqueued.

The argument checks below use made-up device addresses: the library compares
addresses and sizes but never dereferences them on the host, and every case is
invalid, so nothing is launched.  They run only where no GPU is present; on a
GPU machine the same checks are exercised through the GPU tests with real buffers.
"""

import ctypes
import os
import re

import pytest
import torch

from tests.gpu_util import gq4_module

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gq4.h")

no_gpu_only = pytest.mark.skipif(torch.cuda.is_available(),
                                 reason="made-up addresses are only used where no GPU exists")


@pytest.fixture(scope="module")
def gq4():
    return gq4_module()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GQ4_API\s+[\w\s\*]*?\b(gq4_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    syms = declared_symbols()
    for name in ("gq4_matvec", "gq4_quad_matvec", "gq4_norm_matvec", "gq4_gated_matvec",
                 "gq4_unpack", "gq4_dequant", "gq4_status_string", "gq4_version"):
        assert name in syms


def test_library_exports_every_declared_symbol(gq4):
    lib = ctypes.CDLL(gq4.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} declared in gq4.h but not exported"
    assert set(declared_symbols()) <= set(gq4.EXPORTED)


def test_status_strings_and_version(gq4):
    for st in range(6):
        assert gq4.lib.gq4_status_string(st)
    assert gq4.lib.gq4_status_string(99) == b"unknown status"
    assert gq4.version() >= 100


# ---------------------------------------------------------------------------
# Argument validation with made-up addresses (never dereferenced)
# ---------------------------------------------------------------------------

BASE = 0x7F0000000000


def addr(i, off=0):
    """A fake, 256-byte aligned device address, far apart for each i."""
    return ctypes.c_void_p(BASE + i * (1 << 32) + off)


def mv(gq4, M=1, K=1024, N=64, gs=32, A=None, Bq=None, s=None, z=None, C=None):
    return gq4.lib.gq4_matvec(M, K, N, gs, A or addr(0), Bq or addr(1), s or addr(2),
                              z or addr(3), C or addr(4), None)


@no_gpu_only
@pytest.mark.parametrize("M,K,N,gs", [
    (0, 1024, 64, 32), (33, 1024, 64, 32), (1, 0, 64, 32), (1, 1024, 0, 32),
    (1, 1024, 64, 0), (1, 1024, 64, 16), (1, 1000, 64, 40), (1, 96, 64, 64),
    (1, 1024, 64, 48), (-1, 1024, 64, 32), (1, 1 << 25, 64, 32)])
def test_bad_shapes(gq4, M, K, N, gs):
    assert mv(gq4, M, K, N, gs) == gq4.ERR_INVALID_ARG


@no_gpu_only
def test_null_pointers(gq4):
    lib = gq4.lib
    assert lib.gq4_matvec(1, 1024, 64, 32, None, addr(1), addr(2), addr(3), addr(4), None) \
        == gq4.ERR_INVALID_ARG
    assert lib.gq4_matvec(1, 1024, 64, 32, addr(0), None, addr(2), addr(3), addr(4), None) \
        == gq4.ERR_INVALID_ARG
    assert lib.gq4_matvec(1, 1024, 64, 32, addr(0), addr(1), None, addr(3), addr(4), None) \
        == gq4.ERR_INVALID_ARG
    assert lib.gq4_matvec(1, 1024, 64, 32, addr(0), addr(1), addr(2), None, addr(4), None) \
        == gq4.ERR_INVALID_ARG
    assert lib.gq4_matvec(1, 1024, 64, 32, addr(0), addr(1), addr(2), addr(3), None, None) \
        == gq4.ERR_INVALID_ARG
    # norm matvec needs a norm struct with W_norm
    assert lib.gq4_norm_matvec(1, 1024, 64, 32, None, addr(0), addr(1), addr(2), addr(3),
                               addr(4), None) == gq4.ERR_INVALID_ARG
    nrm = gq4.Norm(None, None, 1e-6, None, None)
    assert lib.gq4_norm_matvec(1, 1024, 64, 32, ctypes.byref(nrm), addr(0), addr(1), addr(2),
                               addr(3), addr(4), None) == gq4.ERR_INVALID_ARG


@no_gpu_only
def test_misaligned(gq4):
    assert mv(gq4, A=addr(0, 4)) == gq4.ERR_MISALIGNED          # A needs 16 bytes
    assert mv(gq4, Bq=addr(1, 8)) == gq4.ERR_MISALIGNED         # Bq needs 16 bytes
    assert mv(gq4, s=addr(2, 2)) == gq4.ERR_MISALIGNED          # scales need 4 bytes
    assert mv(gq4, C=addr(4, 1)) == gq4.ERR_MISALIGNED


@no_gpu_only
def test_aliasing(gq4):
    M, K, N, gs = 2, 1024, 64, 32
    # C overlapping the tail of A
    a = addr(0).value
    assert mv(gq4, M, K, N, gs, A=addr(0), C=ctypes.c_void_p(a + M * K * 4 - 16)) == gq4.ERR_ALIAS
    # C overlapping the scales
    s = addr(2).value
    assert mv(gq4, M, K, N, gs, C=ctypes.c_void_p(s + 4)) == gq4.ERR_ALIAS
    # C overlapping the packed words
    assert mv(gq4, M, K, N, gs, C=addr(1, 1024)) == gq4.ERR_ALIAS


@no_gpu_only
def test_quad_splits_and_outputs(gq4):
    lib = gq4.lib
    M, K, N, gs = 1, 256, 50, 32

    def quad(n0, n1, n2, outs):
        return lib.gq4_quad_matvec(M, K, N, gs, n0, n1, n2, addr(0), addr(1), addr(2), addr(3),
                                   *outs, None)
    o = [addr(10), addr(11), addr(12), addr(13)]
    for bad in [(-1, 2, 3), (5, 4, 6), (1, 7, 6), (1, 2, 51)]:
        assert quad(*bad, o) == gq4.ERR_INVALID_ARG, bad
    # a non-empty segment needs its pointer
    assert quad(10, 20, 30, [o[0], None, o[2], o[3]]) == gq4.ERR_INVALID_ARG
    # segments overlapping each other
    assert quad(10, 20, 30, [o[0], ctypes.c_void_p(o[0].value + 8), o[2], o[3]]) \
        == gq4.ERR_ALIAS


@no_gpu_only
def test_norm_outputs_alias(gq4):
    lib = gq4.lib
    M, K, N, gs = 1, 1024, 64, 32
    # residual_out aliasing A (in-place residual update is not allowed)
    nrm = gq4.Norm(addr(5), addr(6), 1e-6, addr(0), addr(7))
    assert lib.gq4_norm_matvec(M, K, N, gs, ctypes.byref(nrm), addr(0), addr(1), addr(2),
                               addr(3), addr(4), None) == gq4.ERR_ALIAS
    # negative or NaN eps
    for eps in (-1.0, float("nan")):
        nrm = gq4.Norm(None, addr(6), eps, None, None)
        assert lib.gq4_norm_matvec(M, K, N, gs, ctypes.byref(nrm), addr(0), addr(1), addr(2),
                                   addr(3), addr(4), None) == gq4.ERR_INVALID_ARG


@no_gpu_only
def test_gated_checks(gq4):
    lib = gq4.lib
    M, K, N, gs = 1, 1024, 64, 32
    args = [addr(1), addr(2), addr(3), addr(11), addr(12), addr(13)]
    # out overlapping the up matrix
    assert lib.gq4_gated_matvec(M, K, N, gs, None, addr(0), *args, addr(11, 64), None) \
        == gq4.ERR_ALIAS
    # missing up scales
    bad = list(args)
    bad[4] = None
    assert lib.gq4_gated_matvec(M, K, N, gs, None, addr(0), *bad, addr(20), None) \
        == gq4.ERR_INVALID_ARG


@no_gpu_only
def test_dual_and_gated_input_checks(gq4):
    lib = gq4.lib
    M, K, N, gs = 1, 1024, 64, 32
    w0 = [addr(1), addr(2), addr(3)]
    w1 = [addr(11), addr(12), addr(13)]
    # the two outputs overlapping each other, or an output over the second matrix
    assert lib.gq4_dual_matvec(M, K, N, gs, addr(0), *w0, *w1, addr(20), addr(20, 64), None) \
        == gq4.ERR_ALIAS
    assert lib.gq4_dual_matvec(M, K, N, gs, addr(0), *w0, *w1, addr(20), addr(12, 16), None) \
        == gq4.ERR_ALIAS
    assert lib.gq4_dual_matvec(M, K, N, gs, addr(0), *w0, *w1, addr(20), None, None) \
        == gq4.ERR_INVALID_ARG
    for fn in (lib.gq4_sigmoid_gated_matvec, lib.gq4_swiglu_gated_matvec):
        # gate vector missing, misaligned, or overlapped by the output
        assert fn(M, K, N, gs, addr(0), None, *w0, addr(20), None) == gq4.ERR_INVALID_ARG
        assert fn(M, K, N, gs, addr(0), addr(5, 4), *w0, addr(20), None) == gq4.ERR_MISALIGNED
        assert fn(M, K, N, gs, addr(0), addr(5), *w0, addr(5, 16), None) == gq4.ERR_ALIAS
        assert fn(0, K, N, gs, addr(0), addr(5), *w0, addr(20), None) == gq4.ERR_INVALID_ARG


@no_gpu_only
def test_unpack_dequant_checks(gq4):
    lib = gq4.lib
    assert lib.gq4_unpack(100, 4, addr(0), addr(1), None) == gq4.ERR_INVALID_ARG   # K % 32
    assert lib.gq4_unpack(64, 4, addr(0, 4), addr(1), None) == gq4.ERR_MISALIGNED
    assert lib.gq4_unpack(64, 4, addr(0), addr(0, 16), None) == gq4.ERR_ALIAS
    assert lib.gq4_dequant(64, 4, 48, addr(0), addr(1), addr(2), addr(3), None) \
        == gq4.ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(gq4):
    A = torch.zeros(1, 64)
    Bq = torch.zeros(4, 8, dtype=torch.int32)
    s = torch.zeros(4, 2)
    with pytest.raises(ValueError, match="CUDA"):
        gq4.matvec(A, Bq, s, s, 32)


# ---------------------------------------------------------------------------
# Call sequences: struct layout and validation on the host
# ---------------------------------------------------------------------------

def test_call_struct_layout_matches_header(gq4, tmp_path):
    """The binding's gq4_call / gq4_norm mirror the C layout field by field."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    src = tmp_path / "layout.c"
    src.write_text(r"""
#include <stddef.h>
#include <stdio.h>
#include "gq4.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(gq4_call), offsetof(gq4_call, A),
         offsetof(gq4_call, Bq), offsetof(gq4_call, scales), offsetof(gq4_call, zeros),
         offsetof(gq4_call, out), offsetof(gq4_call, has_norm), offsetof(gq4_call, norm),
         sizeof(gq4_norm), offsetof(gq4_norm, residual_out));
  return 0;
}
""")
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe)],
                   check=True)
    got = [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    C, N = gq4.Call, gq4.Norm
    want = [ctypes.sizeof(C), C.A.offset, C.Bq.offset, C.scales.offset, C.zeros.offset,
            C.out.offset, C.has_norm.offset, C.norm.offset, ctypes.sizeof(N), N.residual_out.offset]
    assert got == want


def _seq_call(gq4, op, K=256, N=64, gs=32, base=0x7f0000000000):
    d = gq4.Call(op=op, K=K, N=N, group_size=gs, A=base)
    d.Bq[0], d.scales[0], d.zeros[0] = base + 0x100000, base + 0x200000, base + 0x300000
    d.Bq[1], d.scales[1], d.zeros[1] = base + 0x400000, base + 0x500000, base + 0x600000
    d.out[0] = base + 0x700000
    return d


def _run_seq(gq4, descs, ws=0x7e0000000000):
    arr = (gq4.Call * max(len(descs), 1))(*descs)
    return gq4.lib.gq4_run_sequence(arr, len(descs), ws, None)


@no_gpu_only
def test_sequence_validation(gq4):
    # no calls: nothing to do
    assert gq4.lib.gq4_run_sequence(None, 0, None, None) == gq4.OK
    assert gq4.lib.gq4_run_sequence(None, 1, 0x7e0000000000, None) == gq4.ERR_INVALID_ARG
    good = _seq_call(gq4, gq4.OP_MATVEC)
    assert _run_seq(gq4, [good], ws=0) == gq4.ERR_INVALID_ARG              # no workspace
    assert _run_seq(gq4, [good], ws=0x7e0000000004) == gq4.ERR_MISALIGNED  # workspace alignment
    bad_op = _seq_call(gq4, 7)
    assert _run_seq(gq4, [good, bad_op]) == gq4.ERR_INVALID_ARG
    bad_shape = _seq_call(gq4, gq4.OP_MATVEC, K=100)
    assert _run_seq(gq4, [bad_shape]) == gq4.ERR_INVALID_ARG
    no_norm = _seq_call(gq4, gq4.OP_NORM)                                  # norm op needs has_norm
    assert _run_seq(gq4, [no_norm]) == gq4.ERR_INVALID_ARG
    quad = _seq_call(gq4, gq4.OP_QUAD)
    quad.n0, quad.n1, quad.n2 = 40, 30, 64                                 # non-monotone split
    assert _run_seq(gq4, [quad]) == gq4.ERR_INVALID_ARG
    # the workspace may not overlap any call's buffers
    assert _run_seq(gq4, [good], ws=good.out[0]) == gq4.ERR_ALIAS
    # within a call, outputs may not overlap inputs
    alias = _seq_call(gq4, gq4.OP_MATVEC)
    alias.out[0] = alias.A
    assert _run_seq(gq4, [alias]) == gq4.ERR_ALIAS
    # the plan query validates the same way and enqueues nothing
    import ctypes
    n = ctypes.c_int(-1)
    arr = (gq4.Call * 1)(bad_shape)
    assert gq4.lib.gq4_sequence_launches(arr, 1, ctypes.byref(n)) == gq4.ERR_INVALID_ARG
    arr = (gq4.Call * 1)(alias)
    assert gq4.lib.gq4_sequence_launches(arr, 1, ctypes.byref(n)) == gq4.ERR_ALIAS
    assert gq4.lib.gq4_sequence_launches(None, 0, ctypes.byref(n)) == gq4.OK and n.value == 0
    assert gq4.lib.gq4_sequence_launches(None, 0, None) == gq4.ERR_INVALID_ARG


@no_gpu_only
def test_quantize_and_mlx_checks(gq4):
    lib = gq4.lib
    K, N, gs = 1024, 64, 32
    G = N * (K // gs)
    # shape rules, NULLs, alignment
    assert lib.gq4_quantize(K, N, 48, addr(0), addr(1), addr(2), addr(3), None) \
        == gq4.ERR_INVALID_ARG
    assert lib.gq4_quantize(K, N, gs, None, addr(1), addr(2), addr(3), None) == gq4.ERR_INVALID_ARG
    assert lib.gq4_quantize(K, N, gs, addr(0, 4), addr(1), addr(2), addr(3), None) \
        == gq4.ERR_MISALIGNED
    assert lib.gq4_quantize(K, N, gs, addr(0), addr(1, 4), addr(2), addr(3), None) \
        == gq4.ERR_MISALIGNED
    # outputs over W, or over each other
    assert lib.gq4_quantize(K, N, gs, addr(0), addr(0, 4096), addr(2), addr(3), None) \
        == gq4.ERR_ALIAS
    assert lib.gq4_quantize(K, N, gs, addr(0), addr(1), addr(2), addr(2, 4 * (G - 1)), None) \
        == gq4.ERR_ALIAS
    # MLX: scales converted in place over the MLX scales, zeros over the biases
    assert lib.gq4_from_mlx(K, N, gs, addr(0), addr(1), addr(2), addr(3), addr(1), addr(4),
                            None) == gq4.ERR_ALIAS
    assert lib.gq4_from_mlx(K, N, gs, addr(0), addr(1), addr(2), addr(3), addr(4), addr(2),
                            None) == gq4.ERR_ALIAS
    # words partly over the packed input (only the identical pointer is in place)
    assert lib.gq4_from_mlx(K, N, gs, addr(0), addr(1), addr(2), addr(0, 16), addr(4), addr(5),
                            None) == gq4.ERR_ALIAS
    assert lib.gq4_from_mlx(K, N, gs, addr(0), None, addr(2), addr(3), addr(4), addr(5), None) \
        == gq4.ERR_INVALID_ARG
    assert lib.gq4_from_mlx(K, N, 96, addr(0), addr(1), addr(2), addr(3), addr(4), addr(5),
                            None) == gq4.ERR_INVALID_ARG
    assert lib.gq4_from_mlx(K, N, gs, addr(0, 8), addr(1), addr(2), addr(3), addr(4), addr(5),
                            None) == gq4.ERR_MISALIGNED


@no_gpu_only
def test_embedding_checks(gq4):
    lib = gq4.lib
    T, K, V, gs = 8, 1024, 100, 32
    w = [addr(1), addr(2), addr(3)]
    assert lib.gq4_embedding(-1, K, V, gs, addr(0), *w, addr(4), None) == gq4.ERR_INVALID_ARG
    assert lib.gq4_embedding(T, K, V, 48, addr(0), *w, addr(4), None) == gq4.ERR_INVALID_ARG
    assert lib.gq4_embedding(T, K, V, gs, None, *w, addr(4), None) == gq4.ERR_INVALID_ARG
    assert lib.gq4_embedding(T, K, V, gs, addr(0, 2), *w, addr(4), None) == gq4.ERR_MISALIGNED
    assert lib.gq4_embedding(T, K, V, gs, addr(0), *w, addr(4, 4), None) == gq4.ERR_MISALIGNED
    assert lib.gq4_embedding(T, K, V, gs, addr(0), *w, addr(1, 16), None) == gq4.ERR_ALIAS
    assert lib.gq4_embedding(T, K, V, gs, addr(0), *w, addr(0, 16), None) == gq4.ERR_ALIAS
    # T = 0 validates the table and enqueues nothing
    assert lib.gq4_embedding(0, K, V, gs, None, *w, None, None) == gq4.OK


@no_gpu_only
def test_gemm_checks(gq4):
    lib = gq4.lib
    K, N, gs = 1024, 64, 32
    w = [addr(1), addr(2), addr(3)]
    ws = gq4.gemm_workspace_bytes(100, K)
    assert ws >= 100 * K * 2

    def g(M, gs_, A, C, W=None, wb=0):
        return lib.gq4_gemm(M, K, N, gs_, A, *w, C, W, wb, None)
    assert g(0, gs, addr(0), addr(4)) == gq4.ERR_INVALID_ARG
    assert g((1 << 20) + 1, gs, addr(0), addr(4)) == gq4.ERR_INVALID_ARG
    assert g(100, 48, addr(0), addr(4)) == gq4.ERR_INVALID_ARG
    assert g(100, gs, addr(0, 4), addr(4)) == gq4.ERR_MISALIGNED
    # C over the tail of A (100 rows of 4 KB)
    assert g(100, gs, addr(0), addr(0, 99 * 4096)) == gq4.ERR_ALIAS
    assert g(100, gs, addr(0), None) == gq4.ERR_INVALID_ARG
    # workspace: misaligned, or over C
    assert g(100, gs, addr(0), addr(4), addr(5, 16), ws) == gq4.ERR_MISALIGNED
    assert g(100, gs, addr(0), addr(4), addr(4, 256), ws) == gq4.ERR_ALIAS
