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

// Per (column, group) zero-point constants.  The integer part of the zero
// is folded into the magic offset, exactly: with zi = round(clamp(z, 0, 15)),
//   f - (2^23 + 16^p zi) = 16^p (q - zi)          (an exact small integer),
// and the fractional part dz = zi - z multiplies the chunk's activation sum:
//   sum_k a_k (q_k - z) = sum_k a_k (q_k - zi) + dz * sum_k a_k.
// When the zero is an integer in 0..15 (as for codes equal to their zero),
// dz is exactly 0 and so is the correction.
struct ZeroFold {
    f32x2 nc01, nc23;  // -(2^23 + 16^p zi) for p = 0, 1 and p = 2, 3
    float dz;
};

__device__ __forceinline__ ZeroFold fold_zero(float z)
{
    const float zc = fminf(fmaxf(z, 0.0f), 15.0f);
    const float rz = zc + kMagic;  // 2^23 + round(zc)
    const uint32_t rb = __float_as_uint(rz);
    const uint32_t zi = rb - kMagicBits;
    const uint32_t nb = rb | 0x80000000u;  // bits of -(2^23 + zi)
    ZeroFold f;
    f.nc01 = pack2(__uint_as_float(nb), __uint_as_float(nb + zi * 15u));
    f.nc23 = pack2(__uint_as_float(nb + zi * 255u), __uint_as_float(nb + zi * 4095u));
    f.dz = (rz - kMagic) - z;
    return f;
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
// One-lane path: fp16 code pairs.  A LOP3 places two codes of a word as the
// low mantissa bits of the two halves of an fp16 pair whose exponent is that
// of 1024 (bits 0x6400 per half):
//
//     halves = 0x64006400 | (x & (0x000F000F << 4p))  =>  1024 + 16^p q, p in {0, 1}
//
// (exact: 16^p q <= 240 stays inside the 10-bit mantissa).  With t = w >> 8
// the four masks give the pairs (0,4) (1,5) (2,6) (3,7) of a word, codes
// 0, 2, 4, 6 at p = 0 and 1, 3, 5, 7 at p = 1: five ALU operations per word
// instead of nine.  One mixed-precision add (PTX `add.rn.f32.f16`, sm_100
// and later) then widens a half to f32 and adds -(1024 + 16^p zi) in one
// rounding, which is exact: the result 16^p (q - zi) is a small integer.
// The activation that multiplies the code is pre-scaled by 16^-p, so the
// packed FMA forms a * (q - zi) exactly before its single rounding, the same
// arithmetic as the f32 magic form above with half the logic operations.
// ---------------------------------------------------------------------------
constexpr uint32_t kHalfMagicBits = 0x64006400u;

// Per (column, group) zero-point constants of the fp16 form: the integer
// part zi = round(clamp(z, 0, 15)) goes into the widening adds, the
// fractional part dz = zi - z multiplies the chunk group's activation sum
// (sum_k a_k (q_k - z) = sum_k a_k (q_k - zi) + dz * sum_k a_k).  An integer
// zero point in 0..15 gives dz = 0 exactly.
struct HalfZero {
    float nz0;  // -(1024 + zi)       (codes at p = 0)
    float nz1;  // -(1024 + 16 zi)    (codes at p = 1)
    float dz;
};

__device__ __forceinline__ HalfZero half_zero(float z)
{
    const float zc = fminf(fmaxf(z, 0.0f), 15.0f);
    const float zi = __fsub_rn(__fadd_rn(zc, kMagic), kMagic);  // round to nearest integer
    HalfZero h;
    h.nz0 = -1024.0f - zi;
    h.nz1 = fmaf(-16.0f, zi, -1024.0f);
    h.dz = zi - z;
    return h;
}

// f32(low / high half of x, as fp16) + c, one rounding.
__device__ __forceinline__ float widen_add_lo(uint32_t x, float c)
{
    float r;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.f16 %0, l, %2;\n\t}"
        : "=f"(r) : "r"(x), "f"(c));
    return r;
}

__device__ __forceinline__ float widen_add_hi(uint32_t x, float c)
{
    float r;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.f16 %0, h, %2;\n\t}"
        : "=f"(r) : "r"(x), "f"(c));
    return r;
}

template <uint32_t MASK>
__device__ __forceinline__ uint32_t masked_magic_bits(uint32_t x, uint32_t magic)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "n"(MASK), "r"(magic));
    return d;
}

// acc += the eight products of one word with its activations.  `lo` holds
// the activations of codes (0, 4, 1, 5) and `hi` those of (2, 6, 3, 7), the
// ones of codes 1, 3, 5, 7 pre-scaled by 1/16 (see pair_activations).
// `magic` is kHalfMagicBits, passed in from a kernel parameter.
__device__ __forceinline__ f32x2 word_dot(uint32_t w, ulonglong2 lo, ulonglong2 hi, const HalfZero &z,
                                          uint32_t magic, f32x2 acc)
{
    const uint32_t t = w >> 8;
    const uint32_t h04 = masked_magic_bits<0x000F000Fu>(w, magic);
    const uint32_t h15 = masked_magic_bits<0x00F000F0u>(w, magic);
    const uint32_t h26 = masked_magic_bits<0x000F000Fu>(t, magic);
    const uint32_t h37 = masked_magic_bits<0x00F000F0u>(t, magic);
    acc = fma2(lo.x, pack2(widen_add_lo(h04, z.nz0), widen_add_hi(h04, z.nz0)), acc);
    acc = fma2(lo.y, pack2(widen_add_lo(h15, z.nz1), widen_add_hi(h15, z.nz1)), acc);
    acc = fma2(hi.x, pack2(widen_add_lo(h26, z.nz0), widen_add_hi(h26, z.nz0)), acc);
    acc = fma2(hi.y, pack2(widen_add_lo(h37, z.nz1), widen_add_hi(h37, z.nz1)), acc);
    return acc;
}

// The eight activations a0..a7 of one word (x0 = a0..a3, x1 = a4..a7) in
// the order word_dot reads them, pre-scaled: (a0, a4, a1/16, a5/16) and
// (a2, a6, a3/16, a7/16).
__device__ __forceinline__ void pair_activations(float4 x0, float4 x1, float4 &lo, float4 &hi)
{
    lo = make_float4(x0.x, x1.x, x0.y * 0.0625f, x1.y * 0.0625f);
    hi = make_float4(x0.z, x1.z, x0.w * 0.0625f, x1.w * 0.0625f);
}

// Sum of the unscaled activations held by one paired float4.
__device__ __forceinline__ float paired_sum(float4 v)
{
    return (v.x + v.y) + 16.0f * (v.z + v.w);
}

}  // namespace gq4
