// gemm_bf16.cu -- grouped BF16 GEMMs of the dequantized backward on the
// sm_103a tensor cores (tcgen05.mma kind::f16, TMA, TMEM).
//
// "Per-token NVFP4 and Dequantized Backward" (the pages' "Improving Gradient
// Stability"): the backward of y = DQ(Q(x)) . DQ(Q(w))^T runs in BF16 on the
// dequantized operands, x^ = DQ(Q(x)) and w^ = DQ(Q(w)) (nvfp4_dequantize_rows
// makes them); "miniTE Technical Report" 4.2 / 5.2: BF16 backward GEMMs of the
// MoE GroupedLinear over contiguous expert buffers.  Two products per group g:
//   dgrad   dX[rows of g] = dY[rows of g] . w^_g        w^_g stored [Nf x Kf]
//   wgrad   dW_g          = dY[rows of g]^T . x^[rows of g]
// where dY is [rows x Nf] and x^ [rows x Kf], all row-major.  dgrad contracts
// over Nf (A = dY is K-major; B = w^_g has its output dimension Kf
// contiguous: MN-major); wgrad contracts over the group's rows (A = dY and
// B = x^ both MN-major).  Groups are ranges of 128-row multiples of the
// expert-padded row layout (padded offsets poff[G + 1], padding rows zero),
// so no tile crosses a group boundary; a single group of any row count is the
// dense case (the tensor maps zero-fill rows past the end, and stores past it
// are dropped).
//
// Persistent kernel over CTA pairs (clusters of 2, one CTA per SM): a pair
// computes a 256 x 256 output tile with tcgen05.mma.cta_group::2.kind::f16
// (M = 256, N = 256, K = 16 per instruction, fp32 accumulation in TMEM),
// each CTA staging its own 128 rows of A and one 128-row half of B in 64-wide
// K-stages.  Both accumulators fit in TMEM (no scale columns), so the next
// tile's MMAs run while the epilogue drains the previous one.  Roles, 20
// warps per CTA:
//   warp 0       TMA producer: per K-stage the CTA's A tile and B half.
//   warp 1       TMEM allocation (pair-collective, 512 columns) and, in the
//                even CTA, the MMA issuer.
//   warp 2       relay: once the CTA's stage has landed it arrives on the
//                even CTA's `ready` barrier, which tells the MMA issuer that
//                both halves of the stage are in shared memory.
//   warp 3       idle.
//   warps 4-19   epilogue: each warp copies its 32 rows x 64 columns of the
//                accumulator into registers, releases them, converts to bf16
//                and stores through a shared-memory box and a TMA store.
// Every wait is bounded in time; one that runs out raises the abort flag of
// both CTAs, records NVFP4_DEVERR_TIMEOUT and lets both CTAs exit normally.
#include <cuda.h>

#include <cstddef>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int BM = 128;              // rows per CTA; a pair covers 256
constexpr int TN = 256;              // output columns per tile
constexpr int BK = 64;               // K per stage (128 bytes of bf16)
constexpr int STAGES = 4;
constexpr int EPI_WARP0 = 4;
constexpr int EPI_WARPS = 16;
constexpr int THREADS = (EPI_WARP0 + EPI_WARPS) * 32;
constexpr uint32_t TMEM_COLS = 512;  // two 256-column accumulators
constexpr int TILE_BYTES = BM * BK * 2;  // 16 KB: A tile, or B half-tile, of one stage
constexpr int BOXW = 64;                 // output columns per epilogue warp (one 32 x 64 store box)
constexpr int STG_BYTES = 32 * BOXW * 2;
constexpr int MAX_G = 256;

struct __align__(1024) Smem {
    uint8_t a[STAGES][TILE_BYTES];
    uint8_t b[STAGES][TILE_BYTES];
    uint8_t stg[EPI_WARPS][STG_BYTES];
    uint64_t full[STAGES];       // this CTA's stage landed (producer expect_tx)
    uint64_t ready[STAGES];      // (even CTA) both CTAs' stage landed: one relay arrival per CTA
    uint64_t empty[STAGES];      // the stage's MMAs done (commit, multicast to the pair)
    uint64_t tmem_full[2];       // accumulator ready (commit, multicast)
    uint64_t tmem_empty[2];      // (even CTA) accumulator drained: one arrival per epilogue warp of the pair
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int bad;                     // group offsets not multiples of 128 or not ascending: nothing is computed
    int gpoff[MAX_G + 1];
    int ppre[MAX_G + 1];         // dgrad: units of m-tile pairs before each group
    int order[MAX_G];            // wgrad: groups by decreasing row count (ties: lower index first)
};
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory per CTA");
static_assert(offsetof(Smem, stg) % 1024 == 0, "staging alignment (128B swizzle atoms)");

struct Params {
    const int* gpoff;   // nullable: one group of `rows` rows
    int64_t rows;       // rows of dY (and x^ / dX)
    int G;
    int Kc;             // dgrad: contraction (Nf)
    int Mo, No;         // output tile space: dgrad (rows, Kf); wgrad (Nf, Kf)
    uint32_t* err;
};

struct Unit {
    int g;      // group
    int m0;     // first output row of this CTA's 128 (dgrad: row of dX; wgrad: row of dW_g)
    int n0;     // first output column of the pair's 256
    int rows;   // dgrad: valid rows of this CTA's m-tile (0: the odd CTA of a group's last pair)
    int k0;     // wgrad: first row of the contraction; dgrad: 0
    int kst;    // K-stages
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void raise_abort(int* abort_flag, uint32_t rank) {
    *(volatile int*)abort_flag = 1;
    const uint32_t peer = mapa_shared(smem_u32(abort_flag), rank ^ 1u);
    asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" :: "r"(peer), "r"(1) : "memory");
}

// tcgen05.mma.cta_group::2.kind::f16: D[tmem] (+)= A[smem] x B[smem]^T, bf16
// operands, fp32 accumulation, M = 256 across the pair.
__device__ __forceinline__ void tc_mma2_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of kind::f16 with bf16 A and B and fp32 D: D format
// (bits 4-5) 1, A format (7-9) 1, B format (10-12) 1, A / B MN-major (bits 15
// / 16), N >> 3 (17-22), M >> 4 (24-28).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Work units.  dgrad: (pair of m-tiles of one group, n-tile), n fastest; the
// CTA `rank` takes m-tile 2 (pr - ppre[g]) + rank of group g, none past the
// group's end.  wgrad: (group, pair of output row tiles, n-tile), n fastest.
template <bool WGRAD>
__device__ __forceinline__ Unit decode_unit(const Smem& s, const Params& p, int u, uint32_t rank) {
    Unit x;
    const int n_tiles = p.No / TN;
    if (!WGRAD) {
        const int pr = u / n_tiles;
        x.n0 = (u - pr * n_tiles) * TN;
        int lo = 0, hi = p.G;  // the group holding pair row pr
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s.ppre[mid] <= pr) lo = mid; else hi = mid;
        }
        x.g = lo;
        const int g_rows = s.gpoff[lo + 1] - s.gpoff[lo];
        const int mt = 2 * (pr - s.ppre[lo]) + (int)rank;
        const bool none = mt * BM >= g_rows;
        const int mt_eff = none ? mt - 1 : mt;  // repeat the partner's A rows
        x.m0 = s.gpoff[lo] + mt_eff * BM;
        x.rows = none ? 0 : (g_rows - mt * BM < BM ? g_rows - mt * BM : BM);
        x.k0 = 0;
        x.kst = p.Kc / BK;
    } else {
        const int m_pairs = p.Mo / (2 * BM);
        const int per_g = m_pairs * n_tiles;
        const int gi = u / per_g;
        x.g = s.order[gi];
        const int r = u - gi * per_g;
        const int mp = r / n_tiles;
        x.n0 = (r - mp * n_tiles) * TN;
        x.m0 = mp * 2 * BM + (int)rank * BM;
        x.rows = BM;
        x.k0 = s.gpoff[x.g];
        x.kst = (s.gpoff[x.g + 1] - s.gpoff[x.g] + BK - 1) / BK;
    }
    return x;
}

template <bool WGRAD>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmO, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    const int G = p.G;

    if (p.gpoff == nullptr) {
        if (threadIdx.x == 0) { s.gpoff[0] = 0; s.gpoff[1] = (int)p.rows; }
    } else {
        for (int i = threadIdx.x; i <= G; i += THREADS) s.gpoff[i] = p.gpoff[i];
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(smem_u32(&s.full[i]), 1);
            mbar_init(smem_u32(&s.ready[i]), 2);
            mbar_init(smem_u32(&s.empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s.tmem_full[i]), 1);
            mbar_init(smem_u32(&s.tmem_empty[i]), 2 * EPI_WARPS);
        }
        mbar_init(smem_u32(&s.drain), 1);
        s.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int bad = 0;
        if (p.gpoff != nullptr)
            for (int g = 0; g < G; ++g) {
                const int n = s.gpoff[g + 1] - s.gpoff[g];
                if (n < 0 || (n & (BM - 1)) != 0 || s.gpoff[g + 1] > p.rows) bad = 1;
            }
        s.bad = bad;
        if (bad && p.err != nullptr && blockIdx.x == 0) atomicOr(p.err, NVFP4_DEVERR_BADGROUP);
    }
    if (warp == 0 && lane == 0) { prefetch_tmap(&tmA); prefetch_tmap(&tmB); prefetch_tmap(&tmO); }
    if (warp == 1) { tmem_alloc2(smem_u32(&s.tmem_base), TMEM_COLS); tmem_relinquish2(); }
    __syncthreads();
    if (WGRAD) {
        // Largest groups first: a unit's cost is its group's row count, and the
        // pairs take units in a fixed stride, so the long units start first and
        // the short ones fill the end (the skewed routing of the expert layer
        // leaves a few groups several times the mean).  Rank of g = groups with
        // more rows, or as many rows and a lower index.
        for (int g = threadIdx.x; g < G; g += THREADS) {
            const int n = s.gpoff[g + 1] - s.gpoff[g];
            int rank_g = 0;
            for (int h = 0; h < G; ++h) {
                const int m = s.gpoff[h + 1] - s.gpoff[h];
                rank_g += (m > n) || (m == n && h < g);
            }
            s.order[rank_g] = g;
        }
    }
    if (!WGRAD && warp == 0) {
        // ppre[g] = pair rows before group g; lane l holds groups 8l .. 8l + 7
        int loc[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int g = lane * 8 + j;
            loc[j] = sum;
            sum += g < G ? ((s.gpoff[g + 1] - s.gpoff[g] + BM - 1) / BM + 1) >> 1 : 0;
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int g = lane * 8 + j;
            if (g < G) s.ppre[g] = incl - sum + loc[j];
        }
        if (lane == 31) s.ppre[G] = incl;
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    volatile int* abort = &s.abort;
    const int n_tiles = p.No / TN;
    const int total = s.bad ? 0 : (WGRAD ? G * (p.Mo / (2 * BM)) * n_tiles : s.ppre[G] * n_tiles);

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------------------- producer
            int stage = 0, issued = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = pair; u < total && ok; u += n_pairs) {
                const Unit x = decode_unit<WGRAD>(s, p, u, rank);
                const int bn = x.n0 + (int)rank * BM;  // this CTA's half of the pair's 256 columns
                for (int ks = 0; ks < x.kst; ++ks) {
                    if (!mbar_wait_bounded(smem_u32(&s.empty[stage]), phase ^ 1, abort, p.err)) { ok = false; break; }
                    const uint32_t fb = smem_u32(&s.full[stage]);
                    mbar_arrive_expect_tx(fb, 2 * TILE_BYTES);
                    const uint32_t sa = smem_u32(s.a[stage]), sb = smem_u32(s.b[stage]);
                    if (!WGRAD) {
                        // A = dY rows (K-major box of 64 K x 128 rows); B = w^_g rows k (MN-major boxes)
                        tma_load_2d(sa, &tmA, fb, ks * BK, x.m0);
                        const int krow = x.g * p.Kc + ks * BK;
                        tma_load_2d(sb, &tmB, fb, bn, krow);
                        tma_load_2d(sb + TILE_BYTES / 2, &tmB, fb, bn + 64, krow);
                    } else {
                        // A = dY rows of the group (MN-major along Nf); B = x^ rows (MN-major along Kf)
                        const int krow = x.k0 + ks * BK;
                        tma_load_2d(sa, &tmA, fb, x.m0, krow);
                        tma_load_2d(sa + TILE_BYTES / 2, &tmA, fb, x.m0 + 64, krow);
                        tma_load_2d(sb, &tmB, fb, bn, krow);
                        tma_load_2d(sb + TILE_BYTES / 2, &tmB, fb, bn + 64, krow);
                    }
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                raise_abort(&s.abort, rank);
                for (int st = 0; st < STAGES && st < issued; ++st) {
                    const int idx = st + (issued - 1 - st) / STAGES * STAGES;
                    mbar_wait_drain(smem_u32(&s.full[st]), (uint32_t)(idx / STAGES) & 1u);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------------------------------------------------------- MMA issuer (even CTA)
            // K-major operand (dgrad's A): 128-byte rows, 8-row groups 1024 bytes apart, a K-step of
            // 16 elements = +32 bytes.  MN-major operands: two 8 KB boxes of 64 K-rows x 128 bytes
            // (64 columns), 8-row groups 1024 bytes apart, the second box the next 64 columns
            // (leading byte offset 8192); a K-step of 16 rows = +2048 bytes.
            constexpr bool A_MN = WGRAD;
            constexpr uint32_t IDESC = idesc_bf16(2 * BM, TN, A_MN, true);
            const uint64_t adesc0 = A_MN ? smem_desc(smem_u32(s.a[0]), TILE_BYTES / 2, 1024, 2)
                                         : smem_desc(smem_u32(s.a[0]), 0, 1024, 2);
            const uint64_t bdesc0 = smem_desc(smem_u32(s.b[0]), TILE_BYTES / 2, 1024, 2);
            constexpr int A_KSTEP = A_MN ? 2048 : 32;
            constexpr int B_KSTEP = 2048;
            int stage = 0, it = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = pair; u < total && ok; u += n_pairs) {
                const Unit x = decode_unit<WGRAD>(s, p, u, rank);
                if (x.kst == 0) continue;  // an empty group: the epilogue writes zeros
                const int ab = it & 1;
                const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
                ++it;
                if (!mbar_wait_bounded_relaxed(smem_u32(&s.tmem_empty[ab]), acc_phase ^ 1, abort, p.err)) { ok = false; break; }
                tc_fence_after();
                for (int ks = 0; ks < x.kst; ++ks) {
                    if (!mbar_wait_bounded_relaxed(smem_u32(&s.ready[stage]), phase, abort, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = adesc0 + (uint64_t)((stage * TILE_BYTES) >> 4);
                    const uint64_t bd = bdesc0 + (uint64_t)((stage * TILE_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc_mma2_bf16(tmem + ab * TN, ad + (uint64_t)((kk * A_KSTEP) >> 4),
                                     bd + (uint64_t)((kk * B_KSTEP) >> 4), IDESC, (ks | kk) != 0);
                    tc_commit2_mc(smem_u32(&s.empty[stage]), 3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit2_mc(smem_u32(&s.tmem_full[ab]), 3);
            }
            if (!ok) raise_abort(&s.abort, rank);
            tc_commit2_mc(smem_u32(&s.drain), 1);
            mbar_wait_drain(smem_u32(&s.drain), 0);
        }
    } else if (warp == 2) {
        if (lane == 0) {
            // ---------------------------------------------------------------- relay
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const uint32_t ready0 = mapa_shared(smem_u32(&s.ready[0]), 0);
            for (int u = pair; u < total && ok; u += n_pairs) {
                const Unit x = decode_unit<WGRAD>(s, p, u, rank);
                for (int ks = 0; ks < x.kst; ++ks) {
                    if (!mbar_wait_bounded(smem_u32(&s.full[stage]), phase, abort, p.err)) { ok = false; break; }
                    mbar_arrive_cluster(ready0 + stage * 8);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) raise_abort(&s.abort, rank);
        }
    } else if (warp >= EPI_WARP0) {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;                   // TMEM lane quarter of this warp
        const int cg = (warp - EPI_WARP0) >> 2;   // column group 0..3 (64 columns each)
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        const uint32_t stg = smem_u32(s.stg[warp - EPI_WARP0]);
        bool ok = true;
        int it = 0;
        for (int u = pair; u < total; u += n_pairs) {
            const Unit x = decode_unit<WGRAD>(s, p, u, rank);
            uint32_t w[32];
            if (x.kst > 0) {
                const int ab = it & 1;
                const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
                ++it;
                if (!mbar_wait_bounded_relaxed(smem_u32(&s.tmem_full[ab]), acc_phase, abort, p.err)) { ok = false; break; }
                tc_fence_after();
                uint32_t v[64];
                tmem_ld32(lane_addr + ab * TN + cg * 64, v);
                tmem_ld32(lane_addr + ab * TN + cg * 64 + 32, v + 32);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&s.tmem_empty[ab]), 0));
#pragma unroll
                for (int j = 0; j < 32; ++j) w[j] = pack_bf16(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) w[j] = 0u;  // an empty group's gradient is zero
            }
            if (x.rows == 0) continue;  // the odd CTA of a group's last pair: nothing to store
            const int orow = WGRAD ? x.g * p.Mo + x.m0 + q * 32 : x.m0 + q * 32;
            if (!WGRAD && orow >= p.rows) continue;  // a dense tail: this warp's rows are all past the end
            if (lane == 0) bulk_wait_read();  // the previous store has read the box
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t a = stg + lane * 128 + ((c ^ (lane & 7)) << 4);  // 128B swizzle
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                             :: "r"(a), "r"(w[4 * c]), "r"(w[4 * c + 1]), "r"(w[4 * c + 2]), "r"(w[4 * c + 3])
                             : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&tmO, stg, x.n0 + cg * 64, orow);
                bulk_commit();
            }
        }
        if (!ok && lane == 0) raise_abort(&s.abort, rank);
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }
    tc_fence_before();
    __syncwarp();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc2(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2D bf16 view [rows x cols] (row stride ld elements), boxes of box_cols x
// box_rows, 128B swizzle (box_cols = 64: one 128-byte swizzle span per row).
bool make_bf16_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                   int box_rows, bool load) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              load ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool WGRAD>
cudaError_t launch_kind(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to, const Params& p,
                        int num_sms, int64_t units, cudaStream_t stream) {
    const size_t smem = sizeof(Smem) + 1024;
    static std::mutex mu;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64 || !attr_set[dev]) {
            cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel<WGRAD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) attr_set[dev] = true;
        }
    }
    int pairs = num_sms / 2;
    if (units > 0 && units < pairs) pairs = (int)units;
    if (pairs < 1) pairs = 1;
    gemm_bf16_kernel<WGRAD><<<2 * pairs, THREADS, smem, stream>>>(ta, tb, to, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_bf16(const GemmBf16Launch& g, cudaStream_t stream) {
    Params p;
    p.gpoff = g.gpoff;
    p.rows = g.rows;
    p.G = g.gpoff ? g.G : 1;
    p.err = g.err;
    const int num_sms = g.num_sms > 0 ? g.num_sms : 148;
    CUtensorMap ta, tb, to;
    if (!g.wgrad) {
        // dX [rows x Kf] = dY [rows x Nf] . w^_g [Nf x Kf]
        if (g.rows <= 0) return cudaSuccess;
        p.Kc = g.nf;
        p.Mo = (int)g.rows;
        p.No = g.kf;
        if (!make_bf16_map(&ta, g.dy, g.rows, g.nf, g.nf, 64, BM, true)) return cudaErrorInvalidValue;
        if (!make_bf16_map(&tb, g.w, (int64_t)p.G * g.nf, g.kf, g.kf, 64, BK, true)) return cudaErrorInvalidValue;
        if (!make_bf16_map(&to, g.out, g.rows, g.kf, g.kf, 64, 32, false)) return cudaErrorInvalidValue;
        const int64_t units = g.gpoff ? 0 : ((g.rows + BM - 1) / BM + 1) / 2 * (g.kf / TN);
        return launch_kind<false>(ta, tb, to, p, num_sms, units, stream);
    }
    // dW_g [Nf x Kf] = dY[rows of g]^T . x^[rows of g]
    p.Kc = 0;
    p.Mo = g.nf;
    p.No = g.kf;
    const int64_t rows = g.rows > 0 ? g.rows : 1;  // a map needs a nonzero extent (no rows: no loads)
    if (!make_bf16_map(&ta, g.dy, rows, g.nf, g.nf, 64, BK, true)) return cudaErrorInvalidValue;
    if (!make_bf16_map(&tb, g.x, rows, g.kf, g.kf, 64, BK, true)) return cudaErrorInvalidValue;
    if (!make_bf16_map(&to, g.out, (int64_t)p.G * g.nf, g.kf, g.kf, 64, 32, false)) return cudaErrorInvalidValue;
    const int64_t units = (int64_t)p.G * (g.nf / (2 * BM)) * (g.kf / TN);
    return launch_kind<true>(ta, tb, to, p, num_sms, units, stream);
}

}  // namespace nvfp4
