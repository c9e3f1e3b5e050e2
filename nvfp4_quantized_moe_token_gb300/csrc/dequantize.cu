// dequantize.cu -- NVFP4 rows back to bf16: y = bf16(q * s_b * s_g).
//
// "Per-token NVFP4 and Dequantized Backward" (the pages' "Improving Gradient
// Stability" section): the backward pass takes BF16 operands that carry the
// forward pass's quantization decisions, DQ(Q(x)) and DQ(Q(w)), the
// BF16-dequantized value of the exact quantized tensor.  Decode as in
// "miniTE Technical Report" 2.2: x^ = q s_b s_g, here rounded once to bf16.
//
// Exactness: q s_b (E2M1 times E4M3) has at most 6 significant bits, so it is
// exact in fp32.  With p = RN32(v s_g): the bf16 midpoints lie on the fp32
// grid and RN32 is monotonic, so RN16(p) = RN16(v s_g) unless p is itself a
// bf16 midpoint (its low 16 bits are 0x8000).  The kernel converts two
// products at a time with cvt.rn.bf16x2.f32 and settles only that case
// exactly: the sign of the remainder e = fma(v, s_g, -p) decides (e = 0:
// ties to even), and products below 2^-100, where e could underflow, are
// rounded in fp64 on the bf16 grid (subnormal spacing 2^-133).  That is the
// single rounding of the exact product, zero and subnormal results
// included.
//
// Mapping: one thread per 16-element block (8 code bytes in, 32 bytes out),
// consecutive threads on consecutive blocks of a row.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int DQ_THREADS = 256;

// RN16 of a value given as its fp32 rounding p plus the exact remainder
// (e: its sign only matters, when p sits on a bf16 midpoint).
__device__ __forceinline__ uint32_t bf16_rn_split(uint32_t bits, bool e_zero, bool e_same_sign) {
    const uint32_t lo = bits & 0xFFFFu, hi = bits >> 16;
    if (lo != 0x8000u || e_zero) return (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) ? hi + 1 : hi;
    return e_same_sign ? hi + 1 : hi;  // past the midpoint, away from zero, or short of it
}

// bf16 bits of the exact product v * s (v = q s_b exact in fp32): the slow
// path, for products whose fp32 rounding sits on a bf16 midpoint.
__device__ __forceinline__ uint32_t bf16_of_product(float v, float s) {
    const float p = __fmul_rn(v, s);
    if (fabsf(p) >= 0x1p-100f) {  // the fp32 remainder is exact
        const float e = __fmaf_rn(v, s, -p);
        return bf16_rn_split(__float_as_uint(p), e == 0.0f, ((__float_as_uint(e) ^ __float_as_uint(p)) >> 31) == 0);
    }
    const double x = (double)v * (double)s;  // exact: 6 + 24 significant bits
    if (fabs(x) < 0x1p-126) {  // the bf16 subnormal grid, spacing 2^-133
        const double r = rint(x * 0x1p133);  // ties to even
        return __float_as_uint((float)(r * 0x1p-133)) >> 16;  // exact in fp32
    }
    const float pf = (float)x;      // fp32 normal here
    const double ed = x - (double)pf;  // exact in fp64
    return bf16_rn_split(__float_as_uint(pf), ed == 0.0, (ed > 0.0) == (pf > 0.0f));
}

struct DequantArgs {
    const uint8_t* codes;
    const uint8_t* sf;
    const float* scale;
    int64_t rows;
    int cols;
    int per_tensor;
    const int* goff;   // nullable: scale rows padded per group (MoE buffers)
    const int* gpoff;
    int G;
    int padded_rows;   // y rows at the padded positions too
    __nv_bfloat16* y;
    int64_t ldy;
};

// One thread per 16-element block (8 code bytes in, 32 bytes out); the CTA
// is blockDim.x blocks of a row by blockDim.y rows, so no index divides.
__global__ void __launch_bounds__(DQ_THREADS) dequantize_kernel(DequantArgs a) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.y + threadIdx.y;
    const int b = (int)(blockIdx.y * blockDim.x + threadIdx.x);
    const int nb = a.cols >> 4;
    int64_t srow = r;
    int g = 0;
    if (a.goff != nullptr) {
        // the group g with goff[g] <= r < goff[g + 1]: a warp's lanes share one row
        // whenever a row spans whole warps (blockDim.x a multiple of 32), so one lane
        // searches and the others take its answer; otherwise every lane searches
        const bool shared_row = (blockDim.x & 31) == 0;
        const int lane = threadIdx.x & 31;
        if (!shared_row || lane == 0) {
            int lo = 0, hi = a.G;
            const int64_t rr = r < a.rows ? r : a.rows - 1;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (__ldg(a.goff + mid) <= rr) lo = mid; else hi = mid;
            }
            g = lo;
        }
        if (shared_row) g = __shfl_sync(0xffffffffu, g, 0);
        srow = (int64_t)__ldg(a.gpoff + g) + (r - __ldg(a.goff + g));
    }
    if (r >= a.rows || b >= nb) return;
    const int sp4 = (nb + 3) >> 2;
    const uint32_t sbyte = __ldg(a.sf + sf_group_offset(srow, b >> 2, sp4) + (b & 3));
    // per-tensor with groups: one outer scale per group (the stacked expert weights)
    const float sg = a.per_tensor ? __ldg(a.scale + g) : __ldg(a.scale + r);
    const uint2 cw = __ldg(reinterpret_cast<const uint2*>(a.codes + r * (a.cols >> 1)) + b);
    // s_b as f16x2 (both halves): q s_b has at most 6 significant bits and lies
    // in [2^-10, 2688], so the f16 product is exact
    uint32_t sb2;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, %1;\n\t"
        "mov.b32 {lo, hi}, %0;\n\t"
        "mov.b32 %0, {lo, lo};\n\t}"
        : "=r"(sb2) : "h"((uint16_t)sbyte));
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t byte = ((i < 4 ? cw.x : cw.y) >> (8 * (i & 3))) & 0xFFu;
        uint32_t v2;
        asm("{\n\t.reg .b8 c;\n\t.reg .b32 q;\n\t"
            "cvt.u8.u32 c, %1;\n\t"
            "cvt.rn.f16x2.e2m1x2 q, c;\n\t"
            "mul.rn.f16x2 %0, q, %2;\n\t}"
            : "=r"(v2) : "r"(byte), "r"(sb2));
        const float v0 = __half2float(__ushort_as_half((unsigned short)(v2 & 0xFFFFu)));
        const float v1 = __half2float(__ushort_as_half((unsigned short)(v2 >> 16)));
        const float p0 = __fmul_rn(v0, sg), p1 = __fmul_rn(v1, sg);
        uint32_t w;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(p1), "f"(p0));  // p0 in the low half
        // a product whose fp32 value is a bf16 midpoint (low half 0x8000): settle it exactly
        const uint32_t lows = __byte_perm(__float_as_uint(p0), __float_as_uint(p1), 0x5410);
        if (__vcmpeq2(lows, 0x80008000u) != 0u)
            w = bf16_of_product(v0, sg) | (bf16_of_product(v1, sg) << 16);
        o[i] = w;
    }
    uint4* dst = reinterpret_cast<uint4*>(a.y + (a.padded_rows ? srow : r) * a.ldy + (int64_t)b * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// Zero the padding rows of the padded row layout: rows [gpoff[g] + (goff[g +
// 1] - goff[g]), gpoff[g + 1]) of group g = blockIdx.y (at most 127 rows),
// 16 bytes per thread.
__global__ void __launch_bounds__(DQ_THREADS) zero_padding_rows_kernel(DequantArgs a, int chunks_per_row) {
    const int g = blockIdx.y;
    const int64_t start = (int64_t)__ldg(a.gpoff + g) + (__ldg(a.goff + g + 1) - __ldg(a.goff + g));
    const int64_t end = __ldg(a.gpoff + g + 1);
    const int64_t i = (int64_t)blockIdx.x * DQ_THREADS + threadIdx.x;
    const int64_t pr = start + i / chunks_per_row;
    if (pr >= end) return;
    const int64_t c = i % chunks_per_row;
    reinterpret_cast<uint4*>(a.y + pr * a.ldy)[c] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

cudaError_t launch_dequantize(const DequantLaunch& d, cudaStream_t stream) {
    if (d.rows == 0 && !d.padded_rows) return cudaSuccess;
    DequantArgs a;
    a.codes = d.codes;
    a.sf = d.sf;
    a.scale = d.scale;
    a.rows = d.rows;
    a.cols = (int)d.cols;
    a.per_tensor = d.per_tensor;
    a.goff = d.goff;
    a.gpoff = d.gpoff;
    a.G = d.G;
    a.padded_rows = d.padded_rows;
    a.y = reinterpret_cast<__nv_bfloat16*>(d.y);
    a.ldy = d.ldy;
    const int nb = a.cols / 16;
    const int tx = nb < DQ_THREADS ? nb : DQ_THREADS;  // blocks of a row per CTA
    const int ty = DQ_THREADS / tx;                    // rows per CTA
    const int64_t gx = (a.rows + ty - 1) / ty;
    if (gx > 0x7FFFFFFF) return cudaErrorInvalidValue;
    if (gx > 0) dequantize_kernel<<<dim3((unsigned)gx, (unsigned)((nb + tx - 1) / tx)), dim3(tx, ty), 0, stream>>>(a);
    if (a.padded_rows) {
        // each group pads at most 127 rows
        const int chunks = a.cols / 8;
        const unsigned bx = (unsigned)((127 * (int64_t)chunks + DQ_THREADS - 1) / DQ_THREADS);
        zero_padding_rows_kernel<<<dim3(bx, (unsigned)a.G), DQ_THREADS, 0, stream>>>(a, chunks);
    }
    return cudaGetLastError();
}

}  // namespace nvfp4
