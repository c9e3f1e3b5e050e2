// route_topk.cuh -- the router top-k of one chunk of kRouteChunk tokens, as
// a block-level device function: launched on its own (route.cu) or beside
// the per-token quantization of X in one launch (quantize.cu), whose work is
// independent of it.
//
// "miniTE Technical Report" 6.4 (D15 profiles): top-8 of 128 experts.  One
// warp per 4 tokens (their logits loaded together, their rounds
// interleaved): z = logit + bias, each lane's keys sorted once, then k rounds
// of warp argmax over the lanes' largest remaining keys (order-preserving
// integer keys, ties to the lower expert), softmax over the k selected z;
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
    static_assert(EPL >= 1 && EPL <= 8, "a lane's expert slots are 4-bit fields of one word");
    __shared__ int scnt[32 * EPL];
    const int E = 32 * EPL;
    for (int e = threadIdx.x; e < E; e += kTopkThreads) scnt[e] = 0;
    if (chunk == 0 && threadIdx.x == 0) *p.done = 0u;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t tw = (int64_t)chunk * kRouteChunk + warp * TPW;  // this warp's first token
    // Lane l holds experts EPL l .. EPL l + EPL - 1 of each of the warp's
    // tokens (one 16-byte load per four of them where the logits start on a
    // 16-byte boundary); all logits in flight at once.
    const bool v4 = EPL % 4 == 0 && (reinterpret_cast<uintptr_t>(p.logits) & 15u) == 0;
    float z[TPW][EPL];
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
        const bool in = tw + u < p.T;
        const float* lg = p.logits + (tw + u) * E + lane * EPL;
        if (v4) {
#pragma unroll
            for (int j = 0; j + 3 < EPL; j += 4) {
                const float4 v = in ? __ldg(reinterpret_cast<const float4*>(lg + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
                z[u][j] = v.x; z[u][j + 1] = v.y; z[u][j + 2] = v.z; z[u][j + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < EPL; ++j) z[u][j] = in ? __ldg(lg + j) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const float b = p.bias ? __ldg(p.bias + lane * EPL + j) : 0.0f;
            z[u][j] = in ? __fadd_rn(z[u][j], b) : 0.0f;
        }
    }
    // Each z becomes a 32-bit key that orders like the float (sign bit
    // flipped for z >= 0, all bits for z < 0; -0 is first made +0 so that
    // equal values share one key).  A lane sorts its keys, largest first and
    // equal keys in expert order (odd-even transposition sort: adjacent
    // swaps on strictly larger keys only, so it is stable).  Then each of
    // the k rounds is one warp max of the lanes' first keys, one warp min
    // of the expert indices whose first key equals it (ties to the lower
    // expert: a lane's equal keys are already in expert order), and the
    // winning lane drops its first key.  Dropped slots hold key 0, below
    // every value.
    uint32_t key[TPW][EPL];
    uint32_t slot[TPW];  // 4-bit expert offsets within the lane, first key's lowest
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
        int jj[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const uint32_t b = __float_as_uint(__fadd_rn(z[u][j], 0.0f));
            key[u][j] = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
            jj[j] = j;
        }
#pragma unroll
        for (int r = 0; r < EPL; ++r) {
#pragma unroll
            for (int i = r & 1; i + 1 < EPL; i += 2) {
                const bool sw = key[u][i + 1] > key[u][i];
                const uint32_t ka = key[u][i], kb = key[u][i + 1];
                const int ja = jj[i], jb = jj[i + 1];
                key[u][i] = sw ? kb : ka;
                key[u][i + 1] = sw ? ka : kb;
                jj[i] = sw ? jb : ja;
                jj[i + 1] = sw ? ja : jb;
            }
        }
        uint32_t w = 0u;
#pragma unroll
        for (int j = 0; j < EPL; ++j) w |= (uint32_t)jj[j] << (4 * j);
        slot[u] = w;
    }
    uint32_t my_key[TPW];
    int my_id[TPW];
#pragma unroll
    for (int u = 0; u < TPW; ++u) { my_key[u] = 0u; my_id[u] = 0; }
    for (int s = 0; s < p.k; ++s) {
        uint32_t m[TPW], c[TPW];
#pragma unroll
        for (int u = 0; u < TPW; ++u) m[u] = __reduce_max_sync(0xffffffffu, key[u][0]);
#pragma unroll
        for (int u = 0; u < TPW; ++u)
            c[u] = key[u][0] == m[u] ? (uint32_t)(lane * EPL) + (slot[u] & 15u) : 0xffffffffu;
        uint32_t bi[TPW];
#pragma unroll
        for (int u = 0; u < TPW; ++u) bi[u] = __reduce_min_sync(0xffffffffu, c[u]);
#pragma unroll
        for (int u = 0; u < TPW; ++u) {
            if (c[u] == bi[u]) {  // this lane holds the round's expert: drop its first key
#pragma unroll
                for (int j = 0; j + 1 < EPL; ++j) key[u][j] = key[u][j + 1];
                key[u][EPL - 1] = 0u;
                slot[u] >>= 4;
            }
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
