"""Helpers for the GPU parity tests: device transfer, tolerances, guard bands.

Tolerances (the stated parity bar for this method):
  * fp32 CUDA-core paths:   |gpu - oracle| <= 1e-4 * S + 1e-6
  * bf16 tensor-core lanes: |gpu - oracle| <= 2e-2 * S + 1e-6
  where S = sum_k |a_k * w_k| is computed by the oracle for each output.
  * norm_out:     |gpu - oracle| <= 1e-5 * |oracle| + 1e-7;  residual_out bit-exact.
  * gated out:    propagated from the two dot products (see ``tol_gated``).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

requires_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def gq4_module():
    """Build libgq4 if needed and import the binding (fails loudly otherwise)."""
    from int4_group_quantized_quant_gb300 import build as b
    b.build()
    from int4_group_quantized_quant_gb300 import gq4
    return gq4


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def wdev(w):
    """(Bq, scales, zeros) on the device for an inputs.QuantWeights."""
    return dev(w.Bq), dev(w.scales), dev(w.zeros)


def tol_fp32(S):
    return 1e-4 * S + 1e-6


def tol_bf16(S):
    return 2e-2 * S + 1e-6


def tol_gated(g, u, Sg, Su, out, eps_fn=tol_fp32):
    """Bound on |out_gpu - out_ref| for out = silu(g) * u from the dot-product tolerances.

    |silu'(t)| <= 1.1 everywhere, so an error eg in g moves silu(g) by at most
    1.1 eg; with an error eu in u the product moves by at most
    1.1 eg |u| + |silu(g)| eu + 1.1 eg eu.  The last two terms cover the
    rounding of expf, the division and the final product in binary32.
    """
    eg, eu = eps_fn(Sg), eps_fn(Su)
    silu_g = g / (1.0 + np.exp(-np.clip(g, -700, 700)))
    return 1.1 * eg * np.abs(u) + np.abs(silu_g) * eu + 1.1 * eg * eu + 1e-6 * np.abs(out) + 1e-6


def check_close(name, got, ref, tol):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    err = np.abs(got - ref)
    ratio = err / tol
    worst = float(ratio.max()) if ratio.size else 0.0
    bad = int((ratio > 1.0).sum())
    where = np.unravel_index(int(np.argmax(ratio)), ratio.shape) if ratio.size else None
    assert bad == 0, (f"{name}: {bad}/{ratio.size} outside tolerance; worst err/tol "
                      f"{worst:.3g} at {where}: gpu {got[where]!r} ref {ref[where]!r}")
    return worst


class Guarded:
    """An output tensor with canary bands on both sides, checked after the call."""

    PAD = 64
    CANARY = np.float32(-1234.5625)

    def __init__(self, shape, dtype=torch.float32):
        n = int(np.prod(shape))
        self.full = torch.full((n + 2 * self.PAD,), float(self.CANARY), dtype=dtype, device="cuda")
        # keep the inner view 16-byte aligned: PAD floats = 256 bytes
        self.t = self.full[self.PAD:self.PAD + n].view(*shape) if n else \
            torch.empty(shape, dtype=dtype, device="cuda")
        self.n = n

    def check(self):
        f = host(self.full)
        assert np.all(f[:self.PAD] == self.CANARY), "underrun: canary before the output changed"
        assert np.all(f[self.PAD + self.n:] == self.CANARY), "overrun: canary after the output changed"
