// gq4_device.cuh -- device helpers shared by the gq4 kernels (sm_103a).
//
// In-register int4 unpack.  A u32 word holds eight 4-bit codes, code i at
// bits 4i..4i+3 (low nibble first; WGSL_QUAD_MATVEC_INT4 main loop of the
// gerbil moonshine-stt bundle).  Rather than shift every code down and convert
// it with an integer-to-float instruction, each code is masked IN PLACE and
// OR-ed with the exponent bits of 2^23:
//
//     bits(f) = 0x4B000000 | (x & (0xF << 4p))   =>   f = 2^23 + 16^p * q
//
// which is exact while the code stays inside the 23-bit mantissa, i.e. for
// bit positions 0..19 (p <= 4; bit 23 is already the exponent's lowest bit).
// Codes 0..3 are masked in w itself, codes 4..7 in t = w >> 16, so every code
// sits at position p = i % 4:
//
//     p = {0, 1, 2, 3, 0, 1, 2, 3}   for codes i = 0..7 of a word,
//
// one LOP3 per code plus one shift per word.  Then
//
//     d_i = (f_i - 2^23) - 16^p_i * zero = 16^p_i * fl(q_i - zero)
//
// exactly: f_i - 2^23 is exact, 16^p * zero is exact (a power-of-two scale),
// and a difference of two values both scaled by 16^p rounds to 16^p times the
// rounded unscaled difference.  The activation that multiplies code i is
// pre-scaled by 16^-p_i (also exact), so a_scaled * d = a * fl(q - zero)
// exactly inside the FMA.  The fp32 result is therefore bit-identical to an
// FMA chain over fl(q - zero) * a, with three FP operations per code (two
// additions of pre-negated constants and an FMA), issued as packed f32x2
// instructions.  Subtractions are written as additions of negated constants
// because the packed add has no negated-operand form: a packed subtract would
// cost two extra sign flips per pair inside the inner loop.
#pragma once

#include <cstdint>

namespace gq4 {

// 2^23 as a float: the magic offset.
constexpr float kMagic = 8388608.0f;
constexpr uint32_t kMagicBits = 0x4B000000u;

// 16^-p for code i of a word (p = i % 4); the same for both float4 halves.
__host__ __device__ constexpr float code_prescale(int i)
{
    return (i & 3) == 0 ? 1.0f
         : (i & 3) == 1 ? 0.0625f
         : (i & 3) == 2 ? 0.00390625f
                        : 0.000244140625f;
}

// ---------------------------------------------------------------------------
// Packed 2 x f32 arithmetic (PTX ISA 8.6 `*.f32x2`, sm_100 and later): two
// fp32 lanes in one 64-bit register pair, one instruction issue.
// ---------------------------------------------------------------------------
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float lo, float hi)
{
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 unpack2(f32x2 v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return make_float2(lo, hi);
}

__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b)
{
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c)
{
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// The eight magic floats of one word as four pairs (codes 0,1 / 2,3 / 4,5 / 6,7).
struct CodePairs {
    f32x2 p01, p23, p45, p67;
};

// (x & MASK) | magic as ONE lop3 (LUT 0xEA = a & b | c).  `magic` must come
// from a register or a kernel parameter (constant bank): written in plain C
// with both constants as immediates the compiler emits two logic ops per
// code, which doubles the load on the half-rate ALU pipe.
template <uint32_t MASK>
__device__ __forceinline__ float masked_magic(uint32_t x, uint32_t magic)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "n"(MASK), "r"(magic));
    return __uint_as_float(d);
}

// `magic` is kMagicBits, passed in from a kernel parameter.
__device__ __forceinline__ CodePairs extract_word(uint32_t w, uint32_t magic)
{
    const uint32_t t = w >> 16;
    CodePairs c;
    c.p01 = pack2(masked_magic<0x000Fu>(w, magic), masked_magic<0x00F0u>(w, magic));
    c.p23 = pack2(masked_magic<0x0F00u>(w, magic), masked_magic<0xF000u>(w, magic));
    c.p45 = pack2(masked_magic<0x000Fu>(t, magic), masked_magic<0x00F0u>(t, magic));
    c.p67 = pack2(masked_magic<0x0F00u>(t, magic), masked_magic<0xF000u>(t, magic));
    return c;
}

// Negated zero point scaled to the code positions: -(z, 16z) for p = 0, 1 and
// -(256z, 4096z) for p = 2, 3.
struct ZeroPairs {
    f32x2 nz01, nz23;
};

__device__ __forceinline__ ZeroPairs scaled_zero(float z)
{
    ZeroPairs r;
    r.nz01 = pack2(z * -1.0f, z * -16.0f);
    r.nz23 = pack2(z * -256.0f, z * -4096.0f);
    return r;
}

// d = 16^p * fl(q - zero) for the eight codes of a word.
struct DiffPairs {
    f32x2 d01, d23, d45, d67;
};

__device__ __forceinline__ f32x2 neg_magic2()
{
    return pack2(-kMagic, -kMagic);
}

__device__ __forceinline__ DiffPairs code_minus_zero(uint32_t w, const ZeroPairs &z,
                                                     f32x2 nmagic2, uint32_t magic)
{
    const CodePairs c = extract_word(w, magic);
    DiffPairs d;
    d.d01 = add2(add2(c.p01, nmagic2), z.nz01);
    d.d23 = add2(add2(c.p23, nmagic2), z.nz23);
    d.d45 = add2(add2(c.p45, nmagic2), z.nz01);
    d.d67 = add2(add2(c.p67, nmagic2), z.nz23);
    return d;
}

// Scale group of the 32-code chunk gc (gc < 2^20): gc / (gs/32) by
// multiply-shift with magic = ceil(2^40 / (gs/32)).
__device__ __forceinline__ int chunk_group(int gc, unsigned long long magic)
{
    return (int)(((unsigned long long)gc * magic) >> 40);
}

// Shared-memory slot of activation float4 j (0..7) of chunk t: chunk groups
// of R chunks are XOR-swizzled so that 32 lanes reading 32 consecutive
// groups hit distinct banks.
template <int R>
__device__ __forceinline__ int act_index(int t, int j)
{
    return t * 8 + (j ^ ((t / R) & 7));
}

// ---------------------------------------------------------------------------
// One-lane path, integer form.  The activations of a chunk group (R
// consecutive 32-code chunks inside one scale group) are written as 24-bit
// fixed-point integers with the group's own power-of-two scale:
//
//     X_k = rint(a_k * 2^(22 - E)),   2^(E-1) <= max_k |a_k| < 2^E,
//
// so |X_k| <= 2^22 and |X_k * 2^(E-22) - a_k| <= 2^(E-23) <= max_k |a_k| * 2^-22.
// Each X_k splits exactly into three bytes, X = 65536 B2 + 256 B1 + B0 with
// B2 in [-64, 64] (signed) and B1, B0 in [0, 255] (the two's-complement
// bytes of X).  The dot product of a column's codes with one byte piece is
// then an exact integer sum, four products per dp4a instruction (PTX dp4a,
// byte lanes multiplied pairwise and added to a 32-bit accumulator):
//
//     even = w & 0x0F0F0F0F   bytes (q0, q2, q4, q6)
//     odd  = w - even         bytes (16 q1, 16 q3, 16 q5, 16 q7)
//
// against activation words holding the matching bytes of (k0, k2, k4, k6)
// and (k1, k3, k5, k7).  Per word: one logic operation, one integer add and
// six dp4a for the three pieces.  With T_p = sum_k (q_k - zi) B_p,k (exact:
// the integer zero point comes off through the group's piece sums),
//
//     sum_k a_k (q_k - z) ~= 2^(E-22) (65536 T2 + 256 T1 + T0) + (zi - z) sum_k a_k.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int dp4a_s8u8(uint32_t a_s8x4, uint32_t b_u8x4, int c)
{
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a_s8x4), "r"(b_u8x4), "r"(c));
    return d;
}

__device__ __forceinline__ int dp4a_u8u8(uint32_t a_u8x4, uint32_t b_u8x4, int c)
{
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a_u8x4), "r"(b_u8x4), "r"(c));
    return d;
}

// Integer accumulators of one weight stream over a chunk group, piece p
// (p = 0, 1, 2 for B2, B1, B0): e[p] starts at -zi * sum_k B_p,k and adds
// q * B_p over the even codes; o[p] starts at kI8Magic and adds 16 q * B_p
// over the odd codes.
struct I8Acc {
    int e[3];
    int o[3];
};

// Start value of the odd accumulators: the bits of the float 1.5 * 2^23, so
// that 16 e + o is directly the bit pattern of 1.5 * 2^23 + 16 T (exact for
// |16 T| < 2^22) and one float subtraction recovers 16 T.
constexpr int kI8Magic = 0x4B400000;
constexpr float kI8MagicF = 12582912.0f;  // 1.5 * 2^23

// acc += the eight codes of word w against the activation bytes of its
// even (ae[p]) and odd (ao[p]) codes, pieces p = 2, 1, 0 in slots 0, 1, 2.
// `mask` is 0x0F0F0F0F from a kernel parameter.
__device__ __forceinline__ void word_dot_i8(uint32_t w, uint32_t mask, uint32_t ae2, uint32_t ao2,
                                            uint32_t ae1, uint32_t ao1, uint32_t ae0, uint32_t ao0,
                                            I8Acc &acc)
{
    const uint32_t ev = w & mask;
    const uint32_t od = w - ev;
    acc.e[0] = dp4a_s8u8(ae2, ev, acc.e[0]);
    acc.o[0] = dp4a_s8u8(ao2, od, acc.o[0]);
    acc.e[1] = dp4a_u8u8(ae1, ev, acc.e[1]);
    acc.o[1] = dp4a_u8u8(ao1, od, acc.o[1]);
    acc.e[2] = dp4a_u8u8(ae0, ev, acc.e[2]);
    acc.o[2] = dp4a_u8u8(ao0, od, acc.o[2]);
}

// Integer part zi = round(clamp(z, 0, 15)) of a zero point, as an integer
// and as the float fractional correction dz = zi - z.
struct IntZero {
    int zi;
    float dz;
};

__device__ __forceinline__ IntZero int_zero(float z)
{
    const float zc = fminf(fmaxf(z, 0.0f), 15.0f);
    const float r = __fadd_rn(zc, kMagic);  // 2^23 + round(zc), exact
    IntZero iz;
    iz.zi = (int)(__float_as_uint(r) - kMagicBits);
    iz.dz = __fsub_rn(r, kMagic) - z;
    return iz;
}

// Accumulators of one stream at the start of a chunk group: the integer
// zero point comes off through the piece sums sB[p] = sum_k B_p,k of the
// group's activations (16 e + o then carries 16 sum_k (q_k - zi) B_p,k).
__device__ __forceinline__ void int_group_init(I8Acc &acc, int zi, const int (&sB)[3])
{
#pragma unroll
    for (int p = 0; p < 3; ++p) {
        acc.e[p] = -zi * sB[p];
        acc.o[p] = kI8Magic;
    }
}

// sum_k a_k (q_k - z) of one stream over a chunk group: `fac16` = 2^(E-22)/16,
// `asum` = sum_k a_k (f32), dz = zi - z.
__device__ __forceinline__ float int_group_value(const I8Acc &acc, float fac16, float dz, float asum)
{
    float f[3];
#pragma unroll
    for (int p = 0; p < 3; ++p)
        f[p] = __int_as_float(acc.e[p] * 16 + acc.o[p]) - kI8MagicF;  // 16 T_p, exact
    const float t = fmaf(fmaf(f[0], 256.0f, f[1]), 256.0f, f[2]);  // 16 (65536 T2 + 256 T1 + T0)
    return fmaf(fac16, t, dz * asum);
}

}  // namespace gq4
