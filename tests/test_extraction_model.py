"""CPU model of the kernels' in-register code extraction (no GPU needed).

The CUDA kernels turn each 4-bit code into a float by masking it in place
and OR-ing in the exponent bits of 2^23 (codes 0..3 of a word from the word,
codes 4..7 from the word shifted right by 16), then form
d = (f - 2^23) - 16^p * zero and multiply by activations pre-scaled by
16^-p.  This test replays those bit operations in numpy binary32 and checks
the two facts the kernels rely on, against the oracle:

* (f - 2^23) * 16^-p is the code itself, for every code of every word;
* d * 16^-p == fl32(q - zero) bit for bit, for ordinary and extreme zeros.
"""

import numpy as np

import oracle
from int4_group_quantized_quant_gb300 import inputs as I

MAGIC_BITS = np.uint32(0x4B000000)
MAGIC = np.float32(8388608.0)
MASKS = [np.uint32(0xF << (4 * p)) for p in range(4)]


def model_magic_floats(words):
    """[..., 8] binary32 values 2^23 + 16^p q for the eight codes of each word."""
    w = words.astype(np.uint32)
    t = w >> np.uint32(16)
    cols = [(w & MASKS[p]) | MAGIC_BITS for p in range(4)] + \
           [(t & MASKS[p]) | MAGIC_BITS for p in range(4)]
    return np.stack(cols, axis=-1).view(np.float32)


def prescale():
    return np.array([16.0 ** -(i % 4) for i in range(8)], np.float32)


def test_extraction_recovers_codes():
    words = np.concatenate([I.words_u32((4096,), 77),
                            np.array([0, 0xFFFFFFFF, 0x76543210, 0xFEDCBA98, 0x88888888,
                                      0x0F0F0F0F, 0xF0F0F0F0], np.uint32)])
    f = model_magic_floats(words)
    q = ((f - MAGIC) * prescale()).astype(np.float32)
    codes = oracle.unpack(words.reshape(1, -1), 8 * words.size, 1).reshape(-1, 8)
    assert np.array_equal(q, codes.astype(np.float32))


def test_difference_is_exact():
    words = I.words_u32((2048,), 78)
    zeros = np.concatenate([I.uniform_f32((2000,), 6.0, 9.0, 78),
                            np.array([-3.5, 0.0, 15.0, 7.999999, 1e-7, -1e6, 100.25, 2.0 ** 20,
                                      1.5e-30, 3.3e4] * 4 + [0.1] * 8, np.float32)])
    f = model_magic_floats(words)
    zp = zeros[:, None] * np.float32(16.0) ** (np.arange(8) % 4).astype(np.float32)
    d = ((f - MAGIC) - zp.astype(np.float32)).astype(np.float32)
    got = (d * prescale()).astype(np.float32)
    codes = oracle.unpack(words.reshape(1, -1), 8 * words.size, 1).reshape(-1, 8)
    expect = (codes.astype(np.float32) - zeros[:, None]).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), expect.view(np.uint32))
