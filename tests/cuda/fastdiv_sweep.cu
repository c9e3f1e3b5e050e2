// fastdiv_sweep.cu -- test-only kernels: the library's correctly rounded
// reciprocal and division helpers (csrc/fastdiv.cuh) against CUDA's IEEE
// round-to-nearest intrinsics, bit for bit, over whole input sets.
//
// Each sweep counts the inputs whose result differs and keeps the smallest
// such input index; the kernels touch no memory but those two counters.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../nvfp4_quantized_moe_token_gb300/csrc/fastdiv.cuh"

namespace {

struct Tally {
    unsigned long long bad;
    unsigned long long first;  // smallest failing index (ULLONG_MAX if none)
};

__device__ __forceinline__ void note(Tally* t, unsigned long long i) {
    atomicAdd(&t->bad, 1ull);
    atomicMin(&t->first, i);
}

__device__ __forceinline__ float bf16_value(uint32_t b) { return __uint_as_float(b << 16); }

// kind 0: rcp_rn(d) against __frcp_rn(d) for every positive finite fp32 d
//         (index = bit pattern 1 .. 0x7F7FFFFF)
// kind 1: outer_scale(a, 2688) against __fdiv_rn(a, 2688), every positive finite a
// kind 2: outer_scale(a, 1536) against __fdiv_rn(a, 1536), every positive finite a
// kind 3: the block-scale quotient u = bmax / t as the quantizer forms it
//         (div_block with rcp_rn(t)) against __fdiv_rn(bmax, t), for every
//         non-negative finite bf16 bmax and every t = c * outer_scale(amax, s)
//         of a positive finite bf16 amax, (c, s) in {(6, 2688), (6, 1536), (4, 1536)}
// kind 4: div_block on 2^32 pseudo-random pairs of a non-negative finite fp32
//         a and a positive finite fp32 t (each side of every range condition)
__global__ void sweep_kernel(int kind, unsigned long long n, Tally* t) {
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < n; i += stride) {
        if (kind == 0) {
            const float d = __uint_as_float((uint32_t)(i + 1));
            if (__float_as_uint(nvfp4::rcp_rn(d)) != __float_as_uint(__frcp_rn(d))) note(t, i);
        } else if (kind == 1 || kind == 2) {
            const float a = __uint_as_float((uint32_t)(i + 1));
            const float c = kind == 1 ? 2688.0f : 1536.0f;
            if (__float_as_uint(nvfp4::outer_scale(a, c)) != __float_as_uint(__fdiv_rn(a, c))) note(t, i);
        } else if (kind == 4) {
            // a counter-based hash of i gives a (bits of a non-negative finite a) and t (positive finite)
            unsigned long long h = i * 0x9E3779B97F4A7C15ull;
            h ^= h >> 31; h *= 0xBF58476D1CE4E5B9ull; h ^= h >> 29; h *= 0x94D049BB133111EBull; h ^= h >> 32;
            const uint32_t ab = (uint32_t)h % 0x7F800000u, tb = (uint32_t)(h >> 32) % 0x7F7FFFFFu + 1u;
            const float a = __uint_as_float(ab), tt = __uint_as_float(tb);
            const float u = nvfp4::div_block(a, tt, nvfp4::rcp_rn(tt));
            if (__float_as_uint(u) != __float_as_uint(__fdiv_rn(a, tt))) note(t, i);
        } else {
            // i = ((form * 0x7F7F) + (amax pattern - 1)) * 0x7F80 + bmax pattern
            const uint32_t nb = 0x7F80u, na = 0x7F7Fu;
            const uint32_t bpat = (uint32_t)(i % nb);
            const unsigned long long rest = i / nb;
            const uint32_t apat = (uint32_t)(rest % na) + 1u;
            const int form = (int)(rest / na);
            const float s_g = nvfp4::outer_scale(bf16_value(apat), form == 0 ? 2688.0f : 1536.0f);
            const float tt = __fmul_rn(form == 2 ? 4.0f : 6.0f, s_g);
            const float bmax = bf16_value(bpat);
            const float u = nvfp4::div_block(bmax, tt, nvfp4::rcp_rn(tt));
            if (__float_as_uint(u) != __float_as_uint(__fdiv_rn(bmax, tt))) note(t, i);
        }
    }
}

}  // namespace

// Runs one sweep; returns 0 and fills bad / first, or a CUDA error code.
extern "C" int fastdiv_sweep(int kind, unsigned long long* bad, unsigned long long* first,
                             unsigned long long* count) {
    unsigned long long n;
    if (kind == 0 || kind == 1 || kind == 2) n = 0x7F7FFFFFull;
    else if (kind == 3) n = 3ull * 0x7F7Full * 0x7F80ull;
    else if (kind == 4) n = 1ull << 32;
    else return (int)cudaErrorInvalidValue;
    Tally* d = nullptr;
    cudaError_t e = cudaMalloc(&d, sizeof(Tally));
    if (e != cudaSuccess) return (int)e;
    Tally h = {0ull, ~0ull};
    e = cudaMemcpy(d, &h, sizeof h, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) {
        sweep_kernel<<<152 * 8, 256>>>(kind, n, d);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpy(&h, d, sizeof h, cudaMemcpyDeviceToHost);
    cudaFree(d);
    if (e != cudaSuccess) return (int)e;
    *bad = h.bad;
    *first = h.first;
    *count = n;
    return 0;
}
