// route_topk.cuh -- the router top-k of one chunk of kRouteChunk tokens, as
// a block-level device function: launched on its own (route.cu) or beside
// the per-token quantization of X in one launch (quantize.cu), whose work is
// independent of it.
//
// "miniTE Technical Report" 6.4 (D15 profiles): top-8 of 128 experts.  One
// warp per 4 tokens (their logits loaded together, their reductions
// interleaved): z = logit + bias, k rounds of warp argmax (ties to the lower
// expert), softmax over the k selected z; per-chunk expert histogram in
// shared memory.  Blocks of kTopkThreads threads.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;

template <int EPL>  // experts per lane: E = 32 * EPL
__device__ __forceinline__ void route_topk_block(const RouteLaunch& p, int chunk) {
    constexpr int TPW = kRouteChunk / kTopkWarps;  // tokens per warp, selected together
    __shared__ int scnt[32 * EPL];
    const int E = 32 * EPL;
    for (int e = threadIdx.x; e < E; e += kTopkThreads) scnt[e] = 0;
    if (chunk == 0 && threadIdx.x == 0) *p.done = 0u;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t tw = (int64_t)chunk * kRouteChunk + warp * TPW;  // this warp's first token
    // all logits of the warp's tokens in flight at once
    float z[TPW][EPL];
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = lane + 32 * j;
            const float b = p.bias ? __ldg(p.bias + e) : 0.0f;
            z[u][j] = tw + u < p.T ? __fadd_rn(__ldg(p.logits + (tw + u) * E + e), b) : 0.0f;
        }
    }
    // k rounds of warp argmax (ties to the lower expert index), the TPW
    // tokens' reductions interleaved so their shuffle latencies overlap
    uint32_t taken[TPW];
    float my_z[TPW];
    int my_id[TPW];
#pragma unroll
    for (int u = 0; u < TPW; ++u) { taken[u] = 0u; my_z[u] = 0.0f; my_id[u] = 0; }
    for (int s = 0; s < p.k; ++s) {
        float bv[TPW];
        int bi[TPW];
#pragma unroll
        for (int u = 0; u < TPW; ++u) {
            bv[u] = -INFINITY;
            bi[u] = 0x7fffffff;
#pragma unroll
            for (int j = 0; j < EPL; ++j)
                if (!((taken[u] >> j) & 1u) && z[u][j] > bv[u]) { bv[u] = z[u][j]; bi[u] = lane + 32 * j; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
            for (int u = 0; u < TPW; ++u) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv[u], o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi[u], o);
                if (ov > bv[u] || (ov == bv[u] && oi < bi[u])) { bv[u] = ov; bi[u] = oi; }
            }
        }
#pragma unroll
        for (int u = 0; u < TPW; ++u) {
            if ((bi[u] & 31) == lane) taken[u] |= 1u << (bi[u] >> 5);
            if (lane == s) { my_z[u] = bv[u]; my_id[u] = bi[u]; }
        }
    }
    // weights: softmax over the selected z, summed in slot order
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
        const int64_t t = tw + u;
        const float zmax = __shfl_sync(0xffffffffu, my_z[u], 0);
        const float ex = lane < p.k ? expf(__fsub_rn(my_z[u], zmax)) : 0.0f;
        float sum = 0.0f;
        for (int s = 0; s < p.k; ++s) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, ex, s));
        if (t < p.T && lane < p.k) {
            p.ids[t * p.k + lane] = my_id[u];
            p.w[t * p.k + lane] = __fdiv_rn(ex, sum);
            atomicAdd(&scnt[my_id[u]], 1);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kTopkThreads) p.chunk_cnt[(int64_t)chunk * E + e] = scnt[e];
}

}  // namespace nvfp4
