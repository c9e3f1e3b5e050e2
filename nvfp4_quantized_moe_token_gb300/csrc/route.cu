// route.cu -- router top-k, device-side routing metadata, and the permute of
// the per-token quantized rows into expert order (sm_103a).
//
// "miniTE Technical Report" 5.2: expert boundaries are offsets built on the
// device (no host-to-device metadata copies, no host sync), zero-token
// experts and padding handled in the same grouped path; 5.3: the quantized
// activation travels with its scales through the reorder.  Routing: top-8 of
// 128 experts ("miniTE Technical Report" 6.4 D15 profiles).
//
// Four kernels, all deterministic:
//   1. route_topk (route_topk.cuh; in the expert layer it shares one launch
//      with the quantization of X): one warp per 4 tokens -- z = logit +
//      bias, k rounds of warp argmax (ties to the lower expert), softmax over
//      the k selected z; per-chunk expert histogram in shared memory.
//   2. route_scan: one block per expert scans its chunk counts; the last
//      block to finish turns the expert totals into offsets and padded
//      offsets.
//   3. route_scatter: one block per chunk of 32 tokens ranks each (token,
//      slot) inside its expert by a shared-memory bitmap (stable: ascending
//      token index) and writes perm / inv.
//   4. route_permute: one block per padded 128-row m-tile of an expert copies
//      its rows' codes, block scales (staged in shared memory, written as
//      whole swizzled atoms) and outer scales into the expert-ordered buffers.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "route_topk.cuh"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int EPL>
__global__ void __launch_bounds__(kTopkThreads) route_topk_kernel(RouteLaunch p) {
    route_topk_block<EPL>(p, blockIdx.x);
}

// Block-wide exclusive scan of one int per thread (kThreads threads).
__device__ __forceinline__ int block_exclusive_scan(int v, int* total) {
    __shared__ int warp_sums[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int before = 0, all = 0;
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) before += warp_sums[w];
        all += warp_sums[w];
    }
    __syncthreads();
    *total = all;
    return before + incl - v;
}

__global__ void __launch_bounds__(kThreads) route_scan_kernel(RouteLaunch p, int nchunks) {
    const int E = p.E;
    const int e = blockIdx.x;
    const int per = (nchunks + kThreads - 1) / kThreads;
    const int c0 = threadIdx.x * per;
    // up to kScanRegs chunks per thread (T <= 65536 tokens): the counts are
    // loaded once, all in flight together, and kept in registers for the bases
    constexpr int kScanRegs = 8;
    int v[kScanRegs];
    int local = 0;
    if (per <= kScanRegs) {
#pragma unroll
        for (int j = 0; j < kScanRegs; ++j)
            v[j] = (j < per && c0 + j < nchunks) ? p.chunk_cnt[(int64_t)(c0 + j) * E + e] : 0;
#pragma unroll
        for (int j = 0; j < kScanRegs; ++j) local += v[j];
    } else {
        for (int c = c0; c < c0 + per && c < nchunks; ++c) local += p.chunk_cnt[(int64_t)c * E + e];
    }
    int total;
    int base = block_exclusive_scan(local, &total);
    if (per <= kScanRegs) {
#pragma unroll
        for (int j = 0; j < kScanRegs; ++j) {
            if (j < per && c0 + j < nchunks) {
                p.chunk_base[(int64_t)(c0 + j) * E + e] = base;
                base += v[j];
            }
        }
    } else {
        for (int c = c0; c < c0 + per && c < nchunks; ++c) {
            p.chunk_base[(int64_t)c * E + e] = base;
            base += p.chunk_cnt[(int64_t)c * E + e];
        }
    }
    __shared__ int is_last;
    if (threadIdx.x == 0) {
        p.cnt[e] = total;
        __threadfence();
        is_last = atomicAdd(p.done, 1u) == (unsigned)(E - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // the last expert block: offsets and 128-padded offsets over all experts
    const int c = threadIdx.x < E ? __ldcg(p.cnt + threadIdx.x) : 0;
    int tot1, tot2;
    const int o1 = block_exclusive_scan(c, &tot1);
    const int o2 = block_exclusive_scan((c + 127) / 128 * 128, &tot2);
    if (threadIdx.x < E) { p.off[threadIdx.x] = o1; p.poff[threadIdx.x] = o2; }
    if (threadIdx.x == 0) { p.off[E] = tot1; p.poff[E] = tot2; }
}

__global__ void __launch_bounds__(kThreads) route_scatter_kernel(RouteLaunch p) {
    // one chunk of 32 tokens: bit t of bitmap[e] says token t of the chunk chose e
    extern __shared__ uint32_t bitmap[];
    const int E = p.E, k = p.k;
    const int nslot = kRouteChunk * k;
    const int64_t t0 = (int64_t)blockIdx.x * kRouteChunk;
    for (int i = threadIdx.x; i < E; i += kThreads) bitmap[i] = 0u;
    if (p.comb_cnt != nullptr) {  // the combine inside FC2: this chunk's arrival counters start at zero
        const int nb = p.comb_blocks;
        for (int i = threadIdx.x; i < kRouteChunk * nb; i += kThreads)
            if (t0 + i / nb < p.T) p.comb_cnt[t0 * nb + i] = 0;
    }
    // each thread's slots (32 tokens x k <= 16 slots over 256 threads: at most 2),
    // their experts and their rows' first positions are loaded once, before the
    // bitmap is complete
    constexpr int kSlotRegs = kRouteChunk * 16 / kThreads;
    static_assert(kSlotRegs * kThreads >= kRouteChunk * 16, "slots per thread");
    int ev[kSlotRegs], base[kSlotRegs];
#pragma unroll
    for (int j = 0; j < kSlotRegs; ++j) {
        const int i = threadIdx.x + j * kThreads;
        const bool in = i < nslot && t0 + i / k < p.T;
        ev[j] = in ? p.ids[t0 * k + i] : -1;
        const bool good = ev[j] >= 0 && ev[j] < E;
        if (in && !good) ev[j] = -1;
        base[j] = good ? __ldg(p.off + ev[j]) + p.chunk_base[(int64_t)blockIdx.x * E + ev[j]] : 0;
        if (in && !good) atomicOr(p.err, NVFP4_DEVERR_BADEXPERT);
    }
    __syncthreads();  // the bitmap is zeroed
#pragma unroll
    for (int j = 0; j < kSlotRegs; ++j)
        if (ev[j] >= 0) atomicOr(&bitmap[ev[j]], 1u << ((threadIdx.x + j * kThreads) / k));
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kSlotRegs; ++j) {
        if (ev[j] < 0) continue;
        const int i = threadIdx.x + j * kThreads;
        const int tl = i / k;
        const int64_t ts = t0 * k + i;  // = t * k + slot
        const int pos = base[j] + __popc(bitmap[ev[j]] & ((1u << tl) - 1u));
        p.perm[pos] = (int)ts;
        p.inv[ts] = pos;
        p.amax2[pos] = 0.0f;
        if (p.row_w) p.row_w[pos] = p.w[ts];
    }
}

// Permute: one CTA per 128-row padded m-tile of an expert.  Rows of the tile
// are the expert-ordered rows pos0 .. pos0 + 127 (fewer in the expert's last
// tile); row i copies the codes, the block scales and the outer scale of
// token perm[pos0 + i] / k.  The codes move row by row (1 KB per row at
// H = 2048, four rows in flight per warp).  The scales of the tile are
// gathered from the row-linear X scales (one coalesced 4-byte word per lane
// per row) into shared memory, then leave as the tile's contiguous run of
// swizzled 512-byte atoms, so every global store is a whole 16-byte line;
// rows past the expert's end get zero scales.
constexpr int kTileRows = 128;

__global__ void __launch_bounds__(kThreads) route_permute_kernel(RouteLaunch p) {
    __shared__ uint32_t ssf[kTileRows][33];  // [row][scale group], stride 33 words: no bank conflicts
    __shared__ int stok[kTileRows];
    // tiles last to first: FC1 reads them first to last, and finds the ones
    // written last still in L2
    const int E = p.E;
    // the expert whose padded rows hold the tile: the number of expert starts
    // poff[1 .. E-1] at or below its first row, one per thread (E <= 256), all
    // loaded together with the total
    const int ptotal = __ldg(p.poff + E);
    const int pstart = (int)threadIdx.x + 1 < E ? __ldg(p.poff + threadIdx.x + 1) : INT_MAX;
    const int n_tiles = ptotal / kTileRows;
    if ((int)blockIdx.x >= n_tiles) return;  // block-uniform
    const int tile = n_tiles - 1 - (int)blockIdx.x;
    const int prow0 = tile * kTileRows;
    static_assert(kThreads >= 255, "one expert start per thread");
    const int lo = __syncthreads_count(pstart <= prow0);
    const int pos0 = __ldg(p.off + lo) + (prow0 - __ldg(p.poff + lo));
    const int end = __ldg(p.off + lo + 1);
    const int nrows = end - pos0 < kTileRows ? end - pos0 : kTileRows;
    for (int i = threadIdx.x; i < kTileRows; i += kThreads) stok[i] = i < nrows ? __ldg(p.perm + pos0 + i) / p.k : -1;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int W = kThreads / 32;

    // codes: warp w copies rows w, w + W, ..., four rows per batch
    const int64_t row_bytes = p.H / 2;
    for (int i0 = warp; i0 < nrows; i0 += 4 * W) {
        for (int64_t c = lane * 16; c < row_bytes; c += 512) {
            uint4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * W;
                if (i < nrows) v[j] = __ldg(reinterpret_cast<const uint4*>(p.xq_codes + stok[i] * row_bytes + c));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * W;
                // streaming stores: the 268 MB written here would otherwise push the token rows,
                // read 8 times each, out of L2
                if (i < nrows) __stcs(reinterpret_cast<uint4*>(p.a1_codes + (int64_t)(pos0 + i) * row_bytes + c), v[j]);
            }
        }
    }
    for (int i = threadIdx.x; i < nrows; i += kThreads) p.a1_scale[pos0 + i] = __ldg(p.xq_scale + stok[i]);

    // block scales, 32 groups of 4 (128 columns of scales) per pass
    const int64_t sp4 = p.H / 64;
    const int64_t sf_ld = p.H / 16;
    uint8_t* tile_sf = p.a1_sf + (int64_t)tile * sp4 * 512;
    for (int64_t q0 = 0; q0 < sp4; q0 += 32) {
        const int nq = sp4 - q0 < 32 ? (int)(sp4 - q0) : 32;
        for (int i = warp; i < kTileRows; i += W) {
            const int t = stok[i];
            ssf[i][lane] = (t >= 0 && lane < nq)
                ? __ldg(reinterpret_cast<const uint32_t*>(p.xq_sf + (int64_t)t * sf_ld + (q0 + lane) * 4)) : 0u;
        }
        __syncthreads();
        // line c of the pass: group q0 + c / 32, line l = c % 32 holds rows l, l+32, l+64, l+96
        for (int c = threadIdx.x; c < nq * 32; c += kThreads) {
            const int q = c >> 5, l = c & 31;
            *reinterpret_cast<uint4*>(tile_sf + (q0 + q) * 512 + l * 16) =
                make_uint4(ssf[l][q], ssf[l + 32][q], ssf[l + 64][q], ssf[l + 96][q]);
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_route_topk(const RouteLaunch& r, cudaStream_t stream) {
    const int nchunks = (int)((r.T + kRouteChunk - 1) / kRouteChunk);
    switch (r.E / 32) {
        case 1: route_topk_kernel<1><<<nchunks, kTopkThreads, 0, stream>>>(r); break;
        case 2: route_topk_kernel<2><<<nchunks, kTopkThreads, 0, stream>>>(r); break;
        case 3: route_topk_kernel<3><<<nchunks, kTopkThreads, 0, stream>>>(r); break;
        case 4: route_topk_kernel<4><<<nchunks, kTopkThreads, 0, stream>>>(r); break;
        case 5: route_topk_kernel<5><<<nchunks, kTopkThreads, 0, stream>>>(r); break;
        case 6: route_topk_kernel<6><<<nchunks, kTopkThreads, 0, stream>>>(r); break;
        case 7: route_topk_kernel<7><<<nchunks, kTopkThreads, 0, stream>>>(r); break;
        case 8: route_topk_kernel<8><<<nchunks, kTopkThreads, 0, stream>>>(r); break;
        default: return cudaErrorInvalidValue;  // E is validated by the caller
    }
    return cudaGetLastError();
}

cudaError_t launch_route_rest(const RouteLaunch& r, cudaStream_t stream) {
    const int nchunks = (int)((r.T + kRouteChunk - 1) / kRouteChunk);
    route_scan_kernel<<<r.E, kThreads, 0, stream>>>(r, nchunks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    route_scatter_kernel<<<nchunks, kThreads, sizeof(uint32_t) * r.E, stream>>>(r);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // padded m-tiles: sum over experts of ceil(count / 128) <= R / 128 + E; CTAs past the last tile exit
    const int64_t R = r.T * r.k;
    route_permute_kernel<<<(unsigned)((R + kTileRows - 1) / kTileRows + r.E), kThreads, 0, stream>>>(r);
    return cudaGetLastError();
}

cudaError_t launch_route(const RouteLaunch& r, cudaStream_t stream) {
    cudaError_t e = launch_route_topk(r, stream);
    if (e != cudaSuccess) return e;
    return launch_route_rest(r, stream);
}

}  // namespace nvfp4
