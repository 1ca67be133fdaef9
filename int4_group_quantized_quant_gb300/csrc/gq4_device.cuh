// gq4_device.cuh -- device helpers shared by the gq4 kernels (sm_103a).
//
// In-register int4 unpack.  A u32 word holds eight 4-bit codes, code i at
// bits 4i..4i+3 (low nibble first; WGSL_QUAD_MATVEC_INT4 main loop of the
// gerbil moonshine-stt bundle).  Rather than shift every code down and convert
// it with an integer-to-float instruction, each code is masked IN PLACE and
// OR-ed with the exponent bits of 2^23:
//
//     bits(f_i) = 0x4B000000 | (w & (0xF << 4*p_i))   =>   f_i = 2^23 + 16^p_i * q_i
//
// which is exact for p_i <= 5 (the code stays inside the 23-bit mantissa).
// Codes 6 and 7 (bits 24..31) are first moved down by 24 bits and then
// masked at positions 0 and 1.  So the position scale p_i is
//
//     p = {0, 1, 2, 3, 4, 5, 0, 1}   for codes i = 0..7 of a word,
//
// one LOP3 per code (plus one shift per word).  Then
//
//     d_i = (f_i - 2^23) - 16^p_i * zero = 16^p_i * fl(q_i - zero)
//
// exactly: f_i - 2^23 is exact, 16^p * zero is exact (a power-of-two scale),
// and a difference of two values both scaled by 16^p rounds to 16^p times the
// rounded unscaled difference.  The activation that multiplies code i is
// pre-scaled by 16^-p_i (also exact), so a * d = a_scaled_back * fl(q - zero)
// exactly inside the FMA.  The fp32 result is therefore bit-identical to an
// FMA chain over fl(q - zero) * a, with two FP operations per code: one
// subtraction pair and one FMA, issued as packed f32x2 instructions.
#pragma once

#include <cstdint>

namespace gq4 {

// 2^23 as a float: the magic offset.
constexpr float kMagic = 8388608.0f;
constexpr uint32_t kMagicBits = 0x4B000000u;

// 16^-p for the eight codes of a word, split into the two float4 halves
// (codes 0..3 and codes 4..7).
__host__ __device__ constexpr float code_prescale(int i)
{
    return i == 0 ? 1.0f
         : i == 1 ? 0.0625f
         : i == 2 ? 0.00390625f
         : i == 3 ? 0.000244140625f
         : i == 4 ? 1.52587890625e-05f
         : i == 5 ? 9.5367431640625e-07f
         : i == 6 ? 1.0f
                  : 0.0625f;
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

__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b)
{
    f32x2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
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

__device__ __forceinline__ CodePairs extract_word(uint32_t w)
{
    const uint32_t t = w >> 24;
    CodePairs c;
    c.p01 = pack2(__uint_as_float((w & 0x0000000Fu) | kMagicBits),
                  __uint_as_float((w & 0x000000F0u) | kMagicBits));
    c.p23 = pack2(__uint_as_float((w & 0x00000F00u) | kMagicBits),
                  __uint_as_float((w & 0x0000F000u) | kMagicBits));
    c.p45 = pack2(__uint_as_float((w & 0x000F0000u) | kMagicBits),
                  __uint_as_float((w & 0x00F00000u) | kMagicBits));
    c.p67 = pack2(__uint_as_float((t & 0x0000000Fu) | kMagicBits),
                  __uint_as_float((t & 0x000000F0u) | kMagicBits));
    return c;
}

// Zero point scaled to each code position: (z, 16z), (256z, 4096z), (65536z, 2^20 z).
struct ZeroPairs {
    f32x2 z01, z23, z45;
};

__device__ __forceinline__ ZeroPairs scaled_zero(float z)
{
    ZeroPairs r;
    r.z01 = pack2(z, z * 16.0f);
    r.z23 = pack2(z * 256.0f, z * 4096.0f);
    r.z45 = pack2(z * 65536.0f, z * 1048576.0f);
    return r;
}

// d = 16^p * fl(q - zero) for the eight codes of a word.
struct DiffPairs {
    f32x2 d01, d23, d45, d67;
};

__device__ __forceinline__ DiffPairs code_minus_zero(uint32_t w, const ZeroPairs &z)
{
    const f32x2 magic2 = pack2(kMagic, kMagic);
    const CodePairs c = extract_word(w);
    DiffPairs d;
    d.d01 = sub2(sub2(c.p01, magic2), z.z01);
    d.d23 = sub2(sub2(c.p23, magic2), z.z23);
    d.d45 = sub2(sub2(c.p45, magic2), z.z45);
    d.d67 = sub2(sub2(c.p67, magic2), z.z01);
    return d;
}

}  // namespace gq4
