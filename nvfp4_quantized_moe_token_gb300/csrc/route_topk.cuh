// route_topk.cuh -- the router top-k of one chunk of kRouteChunk tokens, as
// a block-level device function: launched on its own (route.cu) or beside
// the per-token quantization of X in one launch (quantize.cu), whose work is
// independent of it.
//
// "miniTE Technical Report" 6.4 (D15 profiles): top-8 of 128 experts.  One
// warp per 4 tokens (their logits loaded together, their rounds
// interleaved): z = logit + bias, k rounds of warp argmax on order-preserving
// integer keys (ties to the lower expert), softmax over the k selected z;
// per-chunk expert histogram in shared memory.  Blocks of kTopkThreads
// threads.
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
    // tokens' rounds interleaved.  Each z becomes a 32-bit key that orders
    // like the float (sign bit flipped for z >= 0, all bits for z < 0; -0 is
    // first made +0 so that equal values share one key), so a round is one
    // warp max of keys and one warp min of the indices holding it
    // (redux.sync), not a five-level shuffle reduction.  Taken entries count
    // as key 0, below every value.
    uint32_t key[TPW][EPL];
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const uint32_t b = __float_as_uint(__fadd_rn(z[u][j], 0.0f));
            key[u][j] = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
        }
    }
    uint32_t taken[TPW], my_key[TPW];
    int my_id[TPW];
#pragma unroll
    for (int u = 0; u < TPW; ++u) { taken[u] = 0u; my_key[u] = 0u; my_id[u] = 0; }
    for (int s = 0; s < p.k; ++s) {
        uint32_t m[TPW];
#pragma unroll
        for (int u = 0; u < TPW; ++u) {
            uint32_t lm = 0u;
#pragma unroll
            for (int j = 0; j < EPL; ++j)
                if (!((taken[u] >> j) & 1u)) lm = max(lm, key[u][j]);
            m[u] = lm;
        }
#pragma unroll
        for (int u = 0; u < TPW; ++u) m[u] = __reduce_max_sync(0xffffffffu, m[u]);
        uint32_t bi[TPW];
#pragma unroll
        for (int u = 0; u < TPW; ++u) {
            uint32_t c = 0xffffffffu;  // this lane's lowest expert index holding the max
#pragma unroll
            for (int j = EPL - 1; j >= 0; --j)
                if (!((taken[u] >> j) & 1u) && key[u][j] == m[u]) c = (uint32_t)(lane + 32 * j);
            bi[u] = c;
        }
#pragma unroll
        for (int u = 0; u < TPW; ++u) bi[u] = __reduce_min_sync(0xffffffffu, bi[u]);
#pragma unroll
        for (int u = 0; u < TPW; ++u) {
            if ((int)(bi[u] & 31u) == lane) taken[u] |= 1u << (bi[u] >> 5);
            if (lane == s) { my_key[u] = m[u]; my_id[u] = (int)bi[u]; }
        }
    }
    float my_z[TPW];
#pragma unroll
    for (int u = 0; u < TPW; ++u)
        my_z[u] = __uint_as_float((my_key[u] & 0x80000000u) ? (my_key[u] & 0x7fffffffu) : ~my_key[u]);
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
