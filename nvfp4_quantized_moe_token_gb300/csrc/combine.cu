// combine.cu -- router-weighted unpermute that ends the expert layer (sm_103a).
//
// out[t] = bf16( sum_{slot=0..k-1} w[t, slot] * Y2[inv[t, slot]] ), fp32
// accumulation in slot order (deterministic).  One block per token; a thread
// owns 8 consecutive columns per 2048-column step and has the k row loads of
// a step in flight together; every Y2 row read and the output row write are
// 16-byte coalesced.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;

// KMAX = the largest k the instance serves (registers for KMAX row loads):
// 8 for the common top-8 routing (64 registers, 4 blocks per SM), else 16.
template <int KMAX>
__global__ void __launch_bounds__(kThreads, KMAX <= 8 ? 4 : 3) combine_kernel(CombineLaunch c) {
    const int64_t t = blockIdx.x;
    const __nv_bfloat16* y = reinterpret_cast<const __nv_bfloat16*>(c.y);
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(c.out) + t * c.H;
    int row[KMAX];
    float w[KMAX];
#pragma unroll
    for (int s = 0; s < KMAX; ++s) {
        if (s < c.k) {
            row[s] = __ldg(c.inv + t * c.k + s);
            w[s] = c.w ? __ldg(c.w + t * c.k + s) : 1.0f;
        }
    }
    for (int64_t col = threadIdx.x * 8; col < c.H; col += kThreads * 8) {
        uint4 v[KMAX];
#pragma unroll
        for (int s = 0; s < KMAX; ++s)  // all k row loads in flight before any use
            if (s < c.k) v[s] = __ldg(reinterpret_cast<const uint4*>(y + (int64_t)row[s] * c.H + col));
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
        for (int s = 0; s < KMAX; ++s) {
            if (s < c.k) {
                const uint32_t wv[4] = {v[s].x, v[s].y, v[s].z, v[s].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[2 * j] = fmaf(w[s], __uint_as_float(wv[j] << 16), acc[2 * j]);
                    acc[2 * j + 1] = fmaf(w[s], __uint_as_float(wv[j] & 0xFFFF0000u), acc[2 * j + 1]);
                }
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
            o[j] = *reinterpret_cast<uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(out + col) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_combine(const CombineLaunch& c, cudaStream_t stream) {
    if (c.T == 0) return cudaSuccess;
    if (c.k <= 8) combine_kernel<8><<<(unsigned)c.T, kThreads, 0, stream>>>(c);
    else combine_kernel<16><<<(unsigned)c.T, kThreads, 0, stream>>>(c);
    return cudaGetLastError();
}

}  // namespace nvfp4
