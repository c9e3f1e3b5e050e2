// nvfp4_encode.cuh -- the NVFP4 encode of one 16-element bf16 block
// (sm_103a), shared by the quantization kernels and the FC2 GEMM that
// quantizes its A operand as it loads it.
//
// "miniTE Technical Report" 2.2 / 5.1: block scale s_b = E4M3(bmax / (6
// s_g)), element codes E2M1(x / (s_b s_g)), every step IEEE binary32 round to
// nearest; the divisions come from fastdiv.cuh.
#pragma once

#include "common.cuh"
#include "fastdiv.cuh"

namespace nvfp4 {

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max |x| of 16 bf16 values: the magnitude bits of non-negative bf16 values
// order like unsigned integers, so a packed 16-bit unsigned max does it.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ float absmax16(const uint4& a, const uint4& b) {
    uint32_t m = max_u16x2(max_u16x2(max_u16x2(a.x & 0x7FFF7FFFu, a.y & 0x7FFF7FFFu),
                                     max_u16x2(a.z & 0x7FFF7FFFu, a.w & 0x7FFF7FFFu)),
                           max_u16x2(max_u16x2(b.x & 0x7FFF7FFFu, b.y & 0x7FFF7FFFu),
                                     max_u16x2(b.z & 0x7FFF7FFFu, b.w & 0x7FFF7FFFu)));
    m = max_u16x2(m, m >> 16);
    return __uint_as_float((m & 0xFFFFu) << 16);
}

// Four fp32 pairs -> one word of eight E2M1 codes (element 2i low nibble).
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float* e) {
    uint32_t w;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(w)
        : "f"(e[0]), "f"(e[1]), "f"(e[2]), "f"(e[3]), "f"(e[4]), "f"(e[5]), "f"(e[6]), "f"(e[7]));
    return w;
}

// Encode one 16-element block (two 16-byte halves) with the row's s_g, t and
// rt = RN(1/t).  Returns the 8 code bytes as two words; *sbyte receives the
// block scale.
__device__ __forceinline__ uint2 encode16(const uint4& lo, const uint4& hi, float bmax, float s_g, float t,
                                          float rt, uint32_t* sbyte) {
    const float u = div_block(bmax, t, rt);
    const uint32_t sb = cvt_e4m3(u);
    *sbyte = sb;
    if (sb == 0) return make_uint2(0u, 0u);
    const float d = __fmul_rn(e4m3_to_f32(sb), s_g);
    float e[16] = {bf16lo(lo.x), bf16hi(lo.x), bf16lo(lo.y), bf16hi(lo.y),
                   bf16lo(lo.z), bf16hi(lo.z), bf16lo(lo.w), bf16hi(lo.w),
                   bf16lo(hi.x), bf16hi(hi.x), bf16lo(hi.y), bf16hi(hi.y),
                   bf16lo(hi.z), bf16hi(hi.z), bf16lo(hi.w), bf16hi(hi.w)};
    if (d >= 1.17549435e-38f) {  // d normal: multiply by the correctly rounded reciprocal
        const float r = rcp_rn(d);
        // two lanes per instruction (mul.rn.f32x2: each lane rounded like the scalar multiply)
        uint64_t r2;
        asm("mov.b64 %0, {%1, %1};" : "=l"(r2) : "f"(r));
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
            uint64_t v;
            asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(e[j]), "f"(e[j + 1]));
            asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(v) : "l"(r2));
            asm("mov.b64 {%0, %1}, %2;" : "=f"(e[j]), "=f"(e[j + 1]) : "l"(v));
        }
    } else {  // d subnormal: 1/d would overflow or lose bits, divide instead
#pragma unroll
        for (int j = 0; j < 16; ++j) e[j] = __fdiv_rn(e[j], d);
    }
    return make_uint2(cvt_e2m1x8(e), cvt_e2m1x8(e + 8));
}

}  // namespace nvfp4
