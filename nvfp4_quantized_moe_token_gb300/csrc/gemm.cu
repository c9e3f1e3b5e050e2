// gemm.cu -- grouped / dense block-scaled NVFP4 GEMM on the sm_103a tensor
// cores (tcgen05 + TMEM + TMA), with the two epilogues of the expert layer.
//
// "miniTE Technical Report" 5.2 (one grouped scheduling path over
// contiguous buffers with device-side expert offsets; zero-token experts and
// padding inside it) and 5.4 (ACC = block-scaled GEMM(A, B); ACC x alpha_a[m]
// x alpha_b; C = gate | up; D = act(gate, up) (x prob); amax of D reduced
// concurrently across CTAs).
//
// Persistent kernel, one CTA per SM, 22 warps with fixed roles:
//   warp 0       TMA producer: per K-stage the A tile (128 rows x 256 FP4,
//                128B-swizzled), the B tile (256 rows: two 128-row boxes) and
//                the E4M3 scale atoms of both (plain bulk copies: the
//                quantizer wrote them in the MMA's layout), 4-stage ring.
//   warp 1       TMEM allocator and MMA issuer: per stage four
//                tcgen05.mma.kind::mxf4nvf4.block_scale (M=128, N=256,
//                K=64), fp32 accumulation in TMEM; tcgen05.commit frees the
//                smem stage and, after the last stage, hands the accumulator
//                to the epilogue.
//   warps 2-5    scale writers (one per TMEM lane quarter): move each stage's
//                scale atoms from shared memory into TMEM with tcgen05.st.
//                (tcgen05.cp would do the same copy, but every cp instruction
//                occupies the tensor pipe for ~55-80 cycles whatever its size,
//                three of them per MMA; tcgen05.st runs on the warps.)
//   warps 6-21   epilogue: each warp copies its 32 rows x 64 accumulator
//                columns into registers, releases TMEM at once (the next
//                tile's MMAs start), then scales and either stores bf16
//                (mode 0) or computes SwiGLU -> bf16 D + row amax (mode 1).
// Tiles are ordered (padded m-tile, n-tile) with n fastest, so CTAs running
// at the same time share the A rows and one expert's weights in L2.
// Every pipeline wait is bounded in time; a wait that runs out raises an
// abort flag, records NVFP4_DEVERR_TIMEOUT, drains what is in flight and
// lets the CTA exit normally (TMEM freed).
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

namespace {

constexpr int BM = 128;                 // rows per tile (TMEM lanes)
constexpr int BN = 256;                 // accumulator columns per tile
constexpr int BK = 256;                 // FP4 elements of K per stage (128 bytes)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK / 2;    // 16 KB
constexpr int B_BYTES = BN * BK / 2;    // 32 KB
constexpr int ATOMS = BK / 64;          // scale atoms (128 rows x 4 scales) per 128 rows per stage
constexpr int SFA_BYTES = ATOMS * 512;  // 2 KB
constexpr int SFB_BYTES = 2 * ATOMS * 512;
constexpr int EPI_WARP0 = 6;            // warps 6..21 run the epilogue (2..5 write scales)
constexpr int EPI_WARPS = 16;
constexpr int THREADS = (EPI_WARP0 + EPI_WARPS) * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;
constexpr uint32_t SF_COL = 256;        // per stage: SFA 4 atoms x 4 cols, SFB 8 atoms x 4 cols
constexpr uint32_t SF_STAGE_COLS = 48;
constexpr int MAX_G = 256;
constexpr uint32_t IDESC = idesc_nvfp4(BM, BN);

struct __align__(1024) Smem {
    uint8_t a[STAGES][A_BYTES];
    uint8_t b[STAGES][B_BYTES];
    uint8_t sfa[STAGES][SFA_BYTES];
    uint8_t sfb[STAGES][SFB_BYTES];
    uint64_t full[STAGES];      // TMA bytes landed
    uint64_t sf_full[STAGES];   // scales of the stage written to TMEM (4 warps)
    uint64_t empty[STAGES];     // MMAs of the stage done (commit)
    uint64_t tmem_full;
    uint64_t tmem_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int consumed;               // stages the MMA issuer has taken from the ring
    int goff[MAX_G + 1];
    int gpoff[MAX_G + 1];
};

struct KParams {
    const uint8_t* a_sf;
    const float* a_scale;
    const uint8_t* b_sf;
    const float* b_scale;
    const int* goff;
    const int* gpoff;
    int64_t M;
    int N, K, G;
    int mode;
    __nv_bfloat16* out;
    int64_t ldo;
    float* amax_out;
    const float* row_prob;
    float* c_debug;
    uint32_t* err;
};

struct Tile {
    int g, row0, rows, mt, nt;
};

__device__ __forceinline__ Tile decode_tile(const Smem& s, int G, int n_tiles, int t) {
    Tile x;
    x.mt = t / n_tiles;
    x.nt = t - x.mt * n_tiles;
    const int prow = x.mt * BM;
    int lo = 0, hi = G;  // last g with gpoff[g] <= prow (non-empty groups are unique)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s.gpoff[mid] <= prow) lo = mid; else hi = mid;
    }
    x.g = lo;
    x.row0 = s.goff[lo] + (prow - s.gpoff[lo]);
    const int end = s.goff[lo + 1];
    x.rows = end - x.row0 < BM ? end - x.row0 : BM;
    return x;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// silu(g) = g / (1 + exp(-g)) with the hardware exp2 and reciprocal
// approximations (a few fp32 ulps, far inside the bf16 rounding that follows);
// exp(-g) = inf for very negative g gives rcp = 0 and silu = -0, no NaN.
__device__ __forceinline__ float silu(float g) {
    return g * rcp_approx(1.0f + __expf(-g));
}

__global__ void __launch_bounds__(THREADS, 1)
gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const KParams p) {
    extern __shared__ uint8_t smem_raw[];
    Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G;

    // group table: dense calls are one group of M rows
    if (p.goff == nullptr) {
        if (threadIdx.x == 0) {
            s.goff[0] = 0; s.goff[1] = (int)p.M;
            s.gpoff[0] = 0; s.gpoff[1] = (int)((p.M + BM - 1) / BM * BM);
        }
    } else {
        for (int i = threadIdx.x; i <= G; i += THREADS) { s.goff[i] = p.goff[i]; s.gpoff[i] = p.gpoff[i]; }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(smem_u32(&s.full[i]), 1);
            mbar_init(smem_u32(&s.sf_full[i]), 4);
            mbar_init(smem_u32(&s.empty[i]), 1);
        }
        mbar_init(smem_u32(&s.tmem_full), 1);
        mbar_init(smem_u32(&s.tmem_empty), EPI_WARPS);
        mbar_init(smem_u32(&s.drain), 1);
        s.abort = 0;
        s.consumed = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) { prefetch_tmap(&tmA); prefetch_tmap(&tmB); }
    if (warp == 1) { tmem_alloc(smem_u32(&s.tmem_base), TMEM_COLS); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    volatile int* abort = &s.abort;

    const int n_tiles = p.mode == 1 ? p.N / 256 : p.N / BN;  // mode 1: 128 gate + 128 up columns per tile
    const int total = (s.gpoff[G] / BM) * n_tiles;
    const int k_atoms = p.K / 64;
    const int k_stages = (k_atoms + ATOMS - 1) / ATOMS;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ producer
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            int last_phase[STAGES];
            for (int i = 0; i < STAGES; ++i) last_phase[i] = -1;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile x = decode_tile(s, G, n_tiles, t);
                const int jb0 = p.mode == 1 ? x.g * (p.N / 128) + x.nt : x.g * (p.N / 128) + 2 * x.nt;
                const int jb1 = p.mode == 1 ? x.g * (p.N / 128) + p.N / 256 + x.nt : jb0 + 1;
                for (int ks = 0; ks < k_stages; ++ks) {
                    if (!mbar_wait_bounded(smem_u32(&s.empty[stage]), phase ^ 1, abort, p.err)) { ok = false; break; }
                    const int na = k_atoms - ks * ATOMS < ATOMS ? k_atoms - ks * ATOMS : ATOMS;
                    const uint32_t fb = smem_u32(&s.full[stage]);
                    mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES + 3 * na * 512);
                    tma_load_2d(smem_u32(s.a[stage]), &tmA, fb, ks * 128, x.row0);
                    tma_load_2d(smem_u32(s.b[stage]), &tmB, fb, ks * 128, jb0 * 128);
                    tma_load_2d(smem_u32(s.b[stage]) + B_BYTES / 2, &tmB, fb, ks * 128, jb1 * 128);
                    bulk_load(smem_u32(s.sfa[stage]), p.a_sf + ((int64_t)x.mt * k_atoms + ks * ATOMS) * 512, na * 512, fb);
                    bulk_load(smem_u32(s.sfb[stage]), p.b_sf + ((int64_t)jb0 * k_atoms + ks * ATOMS) * 512, na * 512, fb);
                    bulk_load(smem_u32(s.sfb[stage]) + SFB_BYTES / 2,
                              p.b_sf + ((int64_t)jb1 * k_atoms + ks * ATOMS) * 512, na * 512, fb);
                    last_phase[stage] = (int)phase;
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                // drain: wait (bounded) for loads the MMA issuer never consumed
                const int outstanding = issued - *(volatile int*)&s.consumed;
                int st = stage;
                for (int i = 0; i < outstanding && i < STAGES; ++i) {
                    st = st == 0 ? STAGES - 1 : st - 1;
                    if (last_phase[st] >= 0) mbar_wait_drain(smem_u32(&s.full[st]), (uint32_t)last_phase[st]);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (!mbar_wait_bounded(smem_u32(&s.tmem_empty), acc_phase ^ 1, abort, p.err)) { ok = false; break; }
                tc_fence_after();
                for (int ks = 0; ks < k_stages; ++ks) {
                    if (!mbar_wait_bounded(smem_u32(&s.full[stage]), phase, abort, p.err) ||
                        !mbar_wait_bounded(smem_u32(&s.sf_full[stage]), phase, abort, p.err)) { ok = false; break; }
                    *(volatile int*)&s.consumed += 1;
                    tc_fence_after();
                    const int na = k_atoms - ks * ATOMS < ATOMS ? k_atoms - ks * ATOMS : ATOMS;
                    const uint32_t sfc = tmem + SF_COL + stage * SF_STAGE_COLS;
                    const uint32_t a0 = smem_u32(s.a[stage]), b0 = smem_u32(s.b[stage]);
                    for (int kk = 0; kk < na; ++kk) {
                        tc_mma_nvfp4(tmem + ACC_COL, smem_desc(a0 + kk * 32, 0, 1024, 2),
                                     smem_desc(b0 + kk * 32, 0, 1024, 2), IDESC,
                                     sfc + kk * 4, sfc + 16 + kk * 8, (ks | kk) != 0);
                    }
                    tc_commit(smem_u32(&s.empty[stage]));
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit(smem_u32(&s.tmem_full));
                acc_phase ^= 1;
            }
            // every MMA issued by this thread completes before TMEM is released
            tc_commit(smem_u32(&s.drain));
            mbar_wait_drain(smem_u32(&s.drain), 0);
        }
    } else if (warp < EPI_WARP0) {
        // ---------------------------------------------------------------- scale writers
        // Warp w writes TMEM lane quarter w % 4.  Each scale atom (32 lines
        // of 16 bytes; line i holds the 4 scales of rows i, i+32, i+64, i+96)
        // goes to 4 consecutive columns of every quarter: thread i of each
        // quarter writes line i.  SFA atom kk -> columns sfc + 4kk; SFB atom kk
        // of half hh -> columns sfc + 16 + 8kk + 4hh.
        const int q = warp & 3;
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            for (int ks = 0; ks < k_stages; ++ks) {
                if (!mbar_wait_bounded(smem_u32(&s.full[stage]), phase, abort, p.err)) { ok = false; break; }
                const uint32_t sfc = lane_addr + SF_COL + stage * SF_STAGE_COLS;
#pragma unroll
                for (int kk = 0; kk < ATOMS; ++kk) {
                    const uint4 a = *reinterpret_cast<const uint4*>(s.sfa[stage] + kk * 512 + lane * 16);
                    const uint4 b0 = *reinterpret_cast<const uint4*>(s.sfb[stage] + kk * 512 + lane * 16);
                    const uint4 b1 = *reinterpret_cast<const uint4*>(s.sfb[stage] + SFB_BYTES / 2 + kk * 512 + lane * 16);
                    tmem_st4(sfc + kk * 4, a.x, a.y, a.z, a.w);
                    tmem_st4(sfc + 16 + kk * 8, b0.x, b0.y, b0.z, b0.w);
                    tmem_st4(sfc + 20 + kk * 8, b1.x, b1.y, b1.z, b1.w);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&s.sf_full[stage]));
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        // Each warp copies its 32 rows x 64 accumulator columns into registers
        // and releases TMEM at once, so the next tile's MMAs run while this
        // warp scales, activates and stores.
        const int q = warp & 3;                    // TMEM lane quarter this warp may access
        const int cg = (warp - EPI_WARP0) >> 2;    // column group 0..3
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const Tile x = decode_tile(s, G, n_tiles, t);
            const int rl = q * 32 + lane;
            const bool valid = rl < x.rows;
            const int64_t row = (int64_t)x.row0 + rl;
            // scales are fetched before the wait so their latency hides under the MMAs
            const float sa = valid ? __ldg(p.a_scale + row) : 0.0f;
            const float sbw = __ldg(p.b_scale + x.g);
            const float prob = (valid && p.row_prob) ? __ldg(p.row_prob + row) : 1.0f;
            if (!mbar_wait_bounded(smem_u32(&s.tmem_full), acc_phase, abort, p.err)) break;
            tc_fence_after();
            uint32_t v[64];
            if (p.mode == 0) {
                tmem_ld32(lane_addr + ACC_COL + cg * 64, v);
                tmem_ld32(lane_addr + ACC_COL + cg * 64 + 32, v + 32);
            } else {
                tmem_ld32(lane_addr + ACC_COL + cg * 32, v);             // gate
                tmem_ld32(lane_addr + ACC_COL + 128 + cg * 32, v + 32);  // up
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s.tmem_empty));
            acc_phase ^= 1;
            if (!valid) continue;
            const float scale = __fmul_rn(sa, sbw);
            if (p.mode == 0) {
                uint4* dst = reinterpret_cast<uint4*>(p.out + row * p.ldo + x.nt * BN + cg * 64);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float* f = reinterpret_cast<const float*>(v + c * 8);
                    dst[c] = make_uint4(pack_bf16(f[0] * scale, f[1] * scale), pack_bf16(f[2] * scale, f[3] * scale),
                                        pack_bf16(f[4] * scale, f[5] * scale), pack_bf16(f[6] * scale, f[7] * scale));
                }
            } else {
                uint4* dst = reinterpret_cast<uint4*>(p.out + row * p.ldo + x.nt * 128 + cg * 32);
                float m = 0.0f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float d[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float g = __uint_as_float(v[c * 8 + j]) * scale;
                        const float u = __uint_as_float(v[32 + c * 8 + j]) * scale;
                        float dv = silu(g) * u;
                        if (p.row_prob) dv *= prob;
                        m = fmaxf(m, fabsf(dv));
                        d[j] = dv;
                    }
                    dst[c] = make_uint4(pack_bf16(d[0], d[1]), pack_bf16(d[2], d[3]), pack_bf16(d[4], d[5]),
                                        pack_bf16(d[6], d[7]));
                }
                if (p.c_debug) {
                    float* cgp = p.c_debug + row * p.N + x.nt * 128 + cg * 32;
                    float* cup = cgp + p.N / 2;
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        *reinterpret_cast<float4*>(cgp + j) = make_float4(
                            __uint_as_float(v[j]) * scale, __uint_as_float(v[j + 1]) * scale,
                            __uint_as_float(v[j + 2]) * scale, __uint_as_float(v[j + 3]) * scale);
                        *reinterpret_cast<float4*>(cup + j) = make_float4(
                            __uint_as_float(v[32 + j]) * scale, __uint_as_float(v[33 + j]) * scale,
                            __uint_as_float(v[34 + j]) * scale, __uint_as_float(v[35 + j]) * scale);
                    }
                }
                // max |bf16(d)| = bf16(max |d|): rounding is monotone and odd
                const float mb = __bfloat162float(__float2bfloat16_rn(m));
                atomicMax(reinterpret_cast<unsigned int*>(p.amax_out + row), __float_as_uint(mb));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
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
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2D uint8 view [rows x row_bytes] of packed FP4 codes, 128-byte x 128-row boxes, 128B swizzle.
bool make_codes_map(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int device_sm_count() {
    static int cache[64] = {0};
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

cudaError_t launch_gemm(const GemmLaunch& g, cudaStream_t stream) {
    if (g.M <= 0) return cudaSuccess;
    CUtensorMap ta, tb;
    if (!make_codes_map(&ta, g.a_codes, g.M, g.K / 2)) return cudaErrorInvalidValue;
    if (!make_codes_map(&tb, g.b_codes, (int64_t)g.G * g.N, g.K / 2)) return cudaErrorInvalidValue;
    KParams p;
    p.a_sf = g.a_sf;
    p.a_scale = g.a_scale;
    p.b_sf = g.b_sf;
    p.b_scale = g.b_scale;
    p.goff = g.goff;
    p.gpoff = g.gpoff;
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.G = g.goff ? g.G : 1;
    p.mode = g.mode;
    p.out = reinterpret_cast<__nv_bfloat16*>(g.out);
    p.ldo = g.ldo;
    p.amax_out = g.amax_out;
    p.row_prob = g.row_prob;
    p.c_debug = g.c_debug;
    p.err = g.err;
    const size_t smem = sizeof(Smem) + 1024;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [&] {
        attr_err = cudaFuncSetAttribute(gemm_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    int grid = g.num_sms > 0 ? g.num_sms : 148;
    if (g.goff == nullptr) {
        const int64_t tiles = (g.M + BM - 1) / BM * (g.N / BN);
        if (tiles < grid) grid = (int)tiles;
    }
    gemm_nvfp4_kernel<<<grid, THREADS, smem, stream>>>(ta, tb, p);
    return cudaGetLastError();
}

}  // namespace nvfp4
