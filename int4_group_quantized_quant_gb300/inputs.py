"""Seeded synthetic inputs for the int4 group-quantized matvec family.

This module only draws random numbers with the shapes and value
distributions of the workloads; it holds none of the method's arithmetic and
is the one module that both the CUDA-side tests and the oracle-side tests use.

* Packed weights: every u32 word is drawn uniformly from [0, 2^32).  Its eight
  4-bit fields are then independent and uniform on 0..15, which is exactly
  "nibbles uniform 0..15 packed 8 per u32", without any packing step here.
* Scales and zeros: uniform on the stated ranges, one per (column, group),
  laid out [N][K/gs].
* Activations: standard normal f32, laid out [M][K].
* RMSNorm gain: uniform on [0.5, 1.5].

Streams come from ``numpy.random.default_rng`` seeded by a
``SeedSequence((base_seed, tag...))`` so each tensor has its own stream.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

BASE_SEED = 0x6751340000

# Value ranges of the workloads.
SCALE_RANGE = (0.005, 0.02)
SCALE_RANGE_GATED = (0.002, 0.01)
ZERO_RANGE = (6.0, 9.0)
NORM_GAIN_RANGE = (0.5, 1.5)
NORM_EPS = 1e-6


def rng(*tags: int) -> np.random.Generator:
    """Independent generator for the tensor identified by ``tags``."""
    return np.random.default_rng(np.random.SeedSequence([BASE_SEED, *[int(t) for t in tags]]))


def uniform_f32(shape, lo: float, hi: float, *tags: int) -> np.ndarray:
    u = rng(*tags).random(shape, dtype=np.float32)
    return (np.float32(lo) + np.float32(hi - lo) * u).astype(np.float32)


def normal_f32(shape, *tags: int) -> np.ndarray:
    return rng(*tags).standard_normal(shape, dtype=np.float32)


def words_u32(shape, *tags: int) -> np.ndarray:
    return rng(*tags).integers(0, 2**32, size=shape, dtype=np.uint32)


@dataclass
class QuantWeights:
    """One int4 matrix: Bq u32 [N][K/8], scales and zeros f32 [N][K/gs]."""
    Bq: np.ndarray
    scales: np.ndarray
    zeros: np.ndarray
    K: int
    N: int
    gs: int

    @property
    def nbytes(self) -> int:
        return self.Bq.nbytes + self.scales.nbytes + self.zeros.nbytes


def quant_weights(K: int, N: int, gs: int, *tags: int,
                  scale_range=SCALE_RANGE, zero_range=ZERO_RANGE) -> QuantWeights:
    if K % 8 or K % gs:
        raise ValueError("K must be a multiple of 8 and of group_size")
    G = K // gs
    return QuantWeights(
        Bq=words_u32((N, K // 8), *tags, 1),
        scales=uniform_f32((N, G), *scale_range, *tags, 2),
        zeros=uniform_f32((N, G), *zero_range, *tags, 3),
        K=K, N=N, gs=gs)


def activations(M: int, K: int, *tags: int) -> np.ndarray:
    return normal_f32((M, K), *tags, 10)


def float_weights(N: int, K: int, *tags: int) -> np.ndarray:
    """Unquantized linear weights f32 [N][K] (row n: output n's K inputs):
    normal with standard deviation 0.02, each row shifted by its own normal
    offset (standard deviation 0.005) so that groups are not centred."""
    w = normal_f32((N, K), *tags, 30) * np.float32(0.02)
    return (w + normal_f32((N, 1), *tags, 31) * np.float32(0.005)).astype(np.float32)


@dataclass
class MLXWeights:
    """An MLX affine int4 matrix: packed u32 [N][K/8], scales and biases f32
    [N][K/gs] with w = scale * q + bias."""
    packed: np.ndarray
    scales: np.ndarray
    biases: np.ndarray
    K: int
    N: int
    gs: int


MLX_BIAS_RANGE = (-0.18, -0.03)  # the span of -scale * zero over SCALE_RANGE x ZERO_RANGE


def mlx_weights(K: int, N: int, gs: int, *tags: int) -> MLXWeights:
    """Random words, scales uniform on SCALE_RANGE, biases uniform on
    MLX_BIAS_RANGE (drawn independently)."""
    G = K // gs
    return MLXWeights(packed=words_u32((N, K // 8), *tags, 40),
                      scales=uniform_f32((N, G), *SCALE_RANGE, *tags, 41),
                      biases=uniform_f32((N, G), *MLX_BIAS_RANGE, *tags, 42), K=K, N=N, gs=gs)


def norm_gain(K: int, *tags: int) -> np.ndarray:
    return uniform_f32((K,), *NORM_GAIN_RANGE, *tags, 20)


# ---------------------------------------------------------------------------
# The five workloads.  Each returns a plain dict of numpy arrays and ints.
# ---------------------------------------------------------------------------

def single_matvec(M=1, K=1024, N=1024, gs=32, seed=0):
    """Single int4 matvec, 1024 x 1024, group 32."""
    w = quant_weights(K, N, gs, seed, 0)
    return dict(kind="matvec", M=M, K=K, N=N, gs=gs, A=activations(M, K, seed, 0), w=w)


def quad_qkv(M=1, K=2560, N=10240, gs=64, n0=4096, n1=5120, n2=6144, seed=1):
    """Quad-output QKV matvec: 2560 -> 10240 split at 4096/5120/6144, group 64."""
    w = quant_weights(K, N, gs, seed, 0)
    return dict(kind="quad", M=M, K=K, N=N, gs=gs, n0=n0, n1=n1, n2=n2,
                A=activations(M, K, seed, 0), w=w)


def norm_prologue(M=1, K=4096, N=4096, gs=64, seed=2):
    """Norm-prologue matvec: RMSNorm(A_a + A_b) * W_norm, eps 1e-6, 4096 -> 4096, group 64."""
    w = quant_weights(K, N, gs, seed, 0)
    return dict(kind="norm", M=M, K=K, N=N, gs=gs, eps=NORM_EPS,
                A=activations(M, K, seed, 0), A_b=activations(M, K, seed, 1),
                W_norm=norm_gain(K, seed, 0), w=w)


def gated_gate_up(M=1, K=4096, N=11008, gs=128, seed=3):
    """SiLU-gated gate/up matvec: 4096 -> 2 x 11008, group 128."""
    wg = quant_weights(K, N, gs, seed, 0, scale_range=SCALE_RANGE_GATED)
    wu = quant_weights(K, N, gs, seed, 1, scale_range=SCALE_RANGE_GATED)
    return dict(kind="gated", M=M, K=K, N=N, gs=gs, A=activations(M, K, seed, 0),
                wg=wg, wu=wu)


# 7B-shaped decode layer: hidden 4096, GQA qkv 4096 -> 4096 + 1024 + 1024,
# o 4096 -> 4096, gate/up 4096 -> 2 x 11008, down 11008 -> 4096, group 128.
STACK_HIDDEN = 4096
STACK_QKV = (4096, 1024, 1024)
STACK_FFN = 11008
STACK_GS = 128
STACK_LAYERS = 32


def stack_layer(layer: int, seed=4, hidden=STACK_HIDDEN, ffn=STACK_FFN, gs=STACK_GS,
                qkv=STACK_QKV):
    """Weights of one decoder layer of the 7B-shaped stack."""
    nq = sum(qkv)
    return dict(
        qkv=quant_weights(hidden, nq, gs, seed, layer, 0),
        o=quant_weights(hidden, hidden, gs, seed, layer, 1),
        gate=quant_weights(hidden, ffn, gs, seed, layer, 2),
        up=quant_weights(hidden, ffn, gs, seed, layer, 3),
        down=quant_weights(ffn, hidden, gs, seed, layer, 4),
        W_norm=norm_gain(hidden, seed, layer, 5),
    )


def stack_input(M: int, seed=4, hidden=STACK_HIDDEN):
    """Decode-step input h [M][hidden] for the stack."""
    return activations(M, hidden, seed, 1_000_000)
