// gemm.cu -- grouped / dense block-scaled NVFP4 GEMM on the sm_103a tensor
// cores (tcgen05 + TMEM + TMA), with the two epilogues of the expert layer.
//
// "miniTE Technical Report" 5.2 (one grouped scheduling path over
// contiguous buffers with device-side expert offsets; zero-token experts and
// padding inside it) and 5.4 (ACC = block-scaled GEMM(A, B); ACC x alpha_a[m]
// x alpha_b; C = gate | up; D = act(gate, up) (x prob); amax of D reduced
// concurrently across CTAs).
//
// Persistent kernel over CTA pairs (clusters of 2, one CTA per SM).  A pair
// computes a 256 x 256 output tile with tcgen05.mma.cta_group::2: each CTA
// stages its own 128 rows of A and one 128-row half of the 256 weight rows,
// the tensor cores of both SMs read both halves of B, and each CTA's TMEM
// receives its own 128 rows of the accumulator.  Per SM that halves the
// weight bytes moved per tile (the single-CTA M=128 x N=256 form is limited
// by the bytes it must stage, not by the tensor pipe), and one MMA issue
// does the work of two.  Roles, 23 warps per CTA:
//   warp 0       TMA producer of A (both CTAs): per K-stage its A tile (128
//                rows, tensor copy) and the E4M3 scale atoms of those rows
//                (a plain bulk copy: the quantizer wrote them in the MMA's
//                layout).
//   warp 22      TMA producer of B (both CTAs): per K-stage its half of the
//                weight tile (128 rows) and the weight scales of both halves
//                in one tensor copy (each SM's tensor core applies the scales
//                of all 256 columns).  Every TMA instruction costs its
//                issuing thread ~65-80 cycles, so the two operands are
//                issued by two threads: one thread could not issue a K-stage's
//                copies within the 512 cycles its MMAs take.
//   warp 1       TMEM allocation (pair-collective, 512 columns) and, in the
//                even CTA only, the MMA issuer: per stage tcgen05.mma
//                .cta_group::2.kind::mxf4nvf4.block_scale (M=256, N=256,
//                K=64), fp32 accumulation; tcgen05.commit multicast to both
//                CTAs frees their smem stages and, after the last stage,
//                hands both accumulator halves to the epilogues.
//   warps 2-5    scale writers (one per TMEM lane quarter): move each stage's
//                scale atoms from shared memory into the CTA's TMEM with
//                tcgen05.st, then arrive on the even CTA's barrier.
//                (tcgen05.cp would do the same copy, but every cp instruction
//                occupies the tensor pipe for ~55-80 cycles whatever its size;
//                tcgen05.st runs on the warps.)
//   warps 6-21   epilogue: each warp copies its 32 rows x 64 accumulator
//                columns into registers and releases them with its own
//                arrival on the even CTA's barrier (the next tile's MMAs
//                start once all 32 warps of the pair have theirs), then
//                scales and either converts to bf16 (modes 0, 2, 3) or
//                computes SwiGLU -> bf16 D + row amax (mode 1).  Outputs leave
//                through a per-warp shared-memory box and a TMA tensor store;
//                a warp whose 32 rows straddle the end of an expert group
//                stores its valid rows directly.  In mode 3 these warps also
//                encode the resident A tile (and warp 0 has no role); in
//                mode 4 they also sum the router-weighted combine of the
//                tokens whose last row they write.
// Work units are (pair of m-tiles of one group, n-tile), n fastest, so pairs
// running at the same time share the A rows and one expert's weights in L2.
// A group with an odd number of m-tiles ends in a unit whose odd CTA has no
// rows: it repeats its partner's A rows for the MMA and stores nothing.
// Every pipeline wait is bounded in time; a wait that runs out raises the
// abort flag of both CTAs, records NVFP4_DEVERR_TIMEOUT, drains what is in
// flight and lets both CTAs exit normally (TMEM freed).
#include <cuda.h>

#include <cstddef>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "nvfp4_encode.cuh"

namespace nvfp4 {

namespace {

constexpr int BM = 128;                 // rows per CTA (TMEM lanes); a pair covers 2 * BM
constexpr int EPI_WARP0 = 6;            // warps 2..5 write scales, 6..21 run the epilogue
constexpr int EPI_WARPS = 16;
constexpr int PRODB_WARP = EPI_WARP0 + EPI_WARPS;  // warp 22: producer of B
constexpr int THREADS = (PRODB_WARP + 1) * 32;
constexpr int ISSUE2_WARP = PRODB_WARP + 1;          // mode 5: warp 23 issues the second half's MMAs
template <int MODE>
constexpr int threads_of() { return MODE == 5 ? (ISSUE2_WARP + 1) * 32 : THREADS; }
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;
constexpr uint32_t SF_COL = 256;
constexpr int MAX_G = 256;

// Pipeline shape.  128-byte K-stages (4 MMAs per stage and per commit, so
// the issuing thread's fixed cost per stage is spread over the stage's
// tensor-pipe cycles), 128B swizzle, plus the epilogue's TMA-store staging
// boxes.
// Mode 1 (SwiGLU, FC1: a long K loop of 8 stages): 256-column tiles (128
// gate + 128 up), one accumulator, 5 stages in flight, one box per warp.
// Mode 0 (plain, FC2: a short K loop of 3 stages): 256-column tiles, one
// accumulator, 4 stages, and each epilogue warp's 32 x 64 output block
// leaves as one TMA store of 128-byte rows (128B swizzle) from one staging
// box.  Measured on FC2 and dropped: 128-column tiles with two accumulators
// (the next tile's MMAs running while the epilogue drains; 0.37 ms against
// 0.31: twice the A tile loads and epilogue passes), 32 x 32 boxes of 64-byte
// rows (0.31 ms), stores from the warps instead of the TMA (coalesced full
// lines read back from the staging box: 0.38 ms).  The tile shape is a
// parameter (TN, ACC_BUFS): both forms pass the parity tests.
// Mode 2 is the plain epilogue for long K loops (K >= 1024, the dense
// linear): 5 stages in flight, and each warp's 64 columns leave as two
// 32-column boxes through one staging box (the smem of a fifth stage).
// Mode 3 is mode 0 with its A operand quantized in the kernel (FC2 of the
// expert layer, K <= 768): the epilogue warps read the bf16 rows of D and
// the row amax that FC1's epilogue left, encode them into a resident A tile
// (codes in the MMA's swizzled layout, block scales as atoms) and the row
// scales; a pair then runs all n-tiles of its m-tiles back to back on that
// tile.  B streams through the 4-stage ring as in mode 0.
// Mode 4 is mode 0 with the expert layer's router-weighted combine in the
// epilogue (combine_completed below).
template <int MODE>
struct Cfg {
    static constexpr int BK = 256;                      // FP4 elements of K per stage
    static constexpr int ROWB = BK / 2;                 // bytes per row per stage
    static constexpr int TN = 256;                      // accumulator columns per tile
    static constexpr int ACC_BUFS = 1;                  // accumulators in TMEM (2 fit at TN = 128)
    static constexpr int B_ROWS = TN / 2;               // weight rows staged per CTA (half the tile)
    static constexpr int SFB_BLOCKS = TN / 128;         // 128-row weight-scale blocks per tile
    static constexpr bool PLAIN = MODE != 1;            // modes 0, 2 and 3: plain bf16 out
    static constexpr bool QOL = MODE == 3;              // A quantized on load, resident across n-tiles
    static constexpr bool COMB = MODE == 4;             // mode 0 plus the combine in the epilogue
    // mode 5: mode 0 with two MMA issuers, one per 128-column half of the
    // tile, each with its own accumulator and hand-off
    static constexpr bool DUAL = MODE == 5;
    static constexpr int NACC = DUAL ? 2 : 1;           // accumulator barriers (ACC_BUFS is 1 in every mode)
    static constexpr int STAGES = (MODE == 0 || MODE == 3 || MODE == 4 || MODE == 5) ? 4 : 5;
    static constexpr int KCH = 3;                       // mode 3: K-stages of the resident A tile (K <= 768)
    static constexpr int A_SLOTS = QOL ? KCH : STAGES;  // A slots: the ring, or the resident tile's stages
    static constexpr int NBUF = 1;                      // staging boxes per epilogue warp
    static constexpr int A_BYTES = BM * ROWB;           // this CTA's 128 rows of A
    static constexpr int B_BYTES = B_ROWS * ROWB;       // this CTA's half of the weight rows
    static constexpr int ATOMS = BK / 64;               // scale atoms per 128 rows per stage
    static constexpr int SFA_BYTES = ATOMS * 512;
    static constexpr int SFB_BYTES = SFB_BLOCKS * ATOMS * 512;  // weight scales of the whole tile
    static constexpr int SWZ = 2;                       // descriptor swizzle code: 128B
    static constexpr int SBO = 8 * ROWB;                // bytes between 8-row core-matrix groups
    static constexpr uint32_t SF_STAGE_COLS = 4 * ATOMS * (1 + SFB_BLOCKS);  // SFA 4 + SFB 4 per block, per atom
    static constexpr uint32_t IDESC = idesc_nvfp4(2 * BM, DUAL ? TN / 2 : TN);
    static constexpr int CPW = PLAIN ? TN / 4 : 32;       // output columns per epilogue warp per tile
    static constexpr int BOXW = (MODE == 0 || MODE == 3 || MODE == 4 || MODE == 5) ? CPW : 32;  // store box width (columns)
    static constexpr int STG_BYTES = 32 * BOXW * 2;       // one staging box: 32 rows x BOXW bf16
    static constexpr bool STAGED = true;
    static constexpr bool TMA_STORE = true;               // false: coalesced warp stores from the staging box
    static constexpr int NSTG = EPI_WARPS * NBUF;
    static_assert(ACC_BUFS * TN <= (int)SF_COL, "accumulators overlap the scale columns");
    static_assert(SF_COL + STAGES * SF_STAGE_COLS <= TMEM_COLS, "scale columns exceed TMEM");
};

template <int MODE>
struct __align__(1024) Smem {
    using C = Cfg<MODE>;
    uint8_t a[C::A_SLOTS][C::A_BYTES];
    uint8_t b[C::STAGES][C::B_BYTES];
    uint8_t sfa[C::A_SLOTS][C::SFA_BYTES];
    uint8_t sfb[C::STAGES][C::SFB_BYTES];
    uint8_t stg[C::NSTG > 0 ? C::NSTG : 1][C::NSTG > 0 ? C::STG_BYTES : 16];
    uint64_t full_a[C::STAGES];    // this CTA's A tile and scales landed
    uint64_t full_b[C::STAGES];    // this CTA's B half and the weight scales landed
    uint64_t sf_full[C::STAGES];   // (even CTA) scales of the stage in TMEM: 4 warps of each CTA
    uint64_t empty[C::STAGES];     // MMAs of the stage done (commit, multicast to the pair)
    uint64_t tmem_full[C::NACC];   // accumulator ready (commit, multicast to the pair)
    uint64_t tmem_empty[C::NACC];  // (even CTA) accumulator drained: one arrival per epilogue warp of the pair
    uint64_t a_full[C::A_SLOTS];   // mode 3: K-stage of the resident A tile encoded (one arrival per epilogue warp)
    uint64_t drain;
    uint64_t never;                // no arrival ever: the time-out test's wait
    uint32_t tmem_base;
    int abort;
    int goff[MAX_G + 1];
    int gpoff[MAX_G + 1];
    int ppre[MAX_G + 1];           // units of m-tile pairs before each group
    float ascale[BM];              // mode 3: the resident tile's row scales (alpha of D's rows)
};
static_assert(sizeof(Smem<0>) + 1024 <= 232448 && sizeof(Smem<1>) + 1024 <= 232448 &&
              sizeof(Smem<2>) + 1024 <= 232448 && sizeof(Smem<3>) + 1024 <= 232448 &&
              sizeof(Smem<4>) + 1024 <= 232448 && sizeof(Smem<5>) + 1024 <= 232448, "shared memory per CTA");
// the two plain forms share the host-side tensor maps
static_assert(Cfg<2>::ROWB == Cfg<0>::ROWB && Cfg<2>::ATOMS == Cfg<0>::ATOMS && Cfg<2>::TN == Cfg<0>::TN &&
              Cfg<2>::B_ROWS == Cfg<0>::B_ROWS && Cfg<2>::SFB_BLOCKS == Cfg<0>::SFB_BLOCKS, "plain forms");
// the staging boxes start on 1024-byte boundaries (the TMA swizzle patterns repeat per 1024 bytes)
static_assert(offsetof(Smem<0>, stg) % 1024 == 0 && offsetof(Smem<1>, stg) % 1024 == 0 &&
              offsetof(Smem<2>, stg) % 1024 == 0 && offsetof(Smem<3>, stg) % 1024 == 0, "staging alignment");
static_assert(Cfg<3>::ROWB == Cfg<0>::ROWB && Cfg<3>::TN == Cfg<0>::TN && Cfg<3>::B_ROWS == Cfg<0>::B_ROWS &&
              Cfg<3>::BOXW == Cfg<0>::BOXW && Cfg<4>::ROWB == Cfg<0>::ROWB && Cfg<4>::TN == Cfg<0>::TN &&
              Cfg<4>::B_ROWS == Cfg<0>::B_ROWS && Cfg<4>::BOXW == Cfg<0>::BOXW &&
              offsetof(Smem<4>, stg) % 1024 == 0, "modes 3 and 4 share mode 0's tensor maps");

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
    int stall;
    // mode 3: the bf16 rows of D [M x K] and their amax (FC1's epilogue), and
    // nullable copies of what the kernel encodes (codes [M x K/2], swizzled
    // block scales of the padded rows, row scales [M]) for inspection
    const __nv_bfloat16* d_in;
    const float* d_amax;
    uint8_t* q_codes;
    uint8_t* q_sf;
    float* q_scale;
    // mode 4: the router-weighted combine in the epilogue
    const int* perm;
    const int* inv;
    const float* cw;
    __nv_bfloat16* cout;
    int* ccnt;
    int k_top;
};

struct Tile {
    int g, row0, rows, mt, nt;
    int arows;  // rows of m-tile mt (the partner's when this CTA has none): the A rows it stages
};

// Unit u = (pair row pr, n-tile nt), nt fastest.  Pair row pr lies in the
// group g with ppre[g] <= pr < ppre[g + 1]; CTA `rank` of the pair takes
// m-tile gpoff[g] / BM + 2 (pr - ppre[g]) + rank.  Past the group's last
// m-tile that CTA has no rows (rows = 0) and repeats its partner's m-tile.
template <class S>
__device__ __forceinline__ Tile decode_unit(const S& s, int G, int n_tiles, int u, uint32_t rank) {
    Tile x;
    const int pr = u / n_tiles;
    x.nt = u - pr * n_tiles;
    int lo = 0, hi = G;  // last g with ppre[g] <= pr (the group holding pair row pr)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s.ppre[mid] <= pr) lo = mid; else hi = mid;
    }
    x.g = lo;
    const int mt0 = s.gpoff[lo] / BM + 2 * (pr - s.ppre[lo]);
    const bool none = mt0 + (int)rank >= s.gpoff[lo + 1] / BM;
    x.mt = none ? mt0 : mt0 + (int)rank;
    x.row0 = s.goff[lo] + (x.mt * BM - s.gpoff[lo]);
    const int end = s.goff[lo + 1];
    x.arows = end - x.row0 < BM ? end - x.row0 : BM;
    x.rows = none ? 0 : x.arows;
    return x;
}

// Set the abort flag of both CTAs of the pair (the peer's through its
// shared-memory window), so its bounded waits give up at once.
__device__ __forceinline__ void raise_abort(int* abort_flag, uint32_t rank) {
    *(volatile int*)abort_flag = 1;
    const uint32_t peer = mapa_shared(smem_u32(abort_flag), rank ^ 1u);
    asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" :: "r"(peer), "r"(1) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// One warp's 32 rows x BOXW bf16 output columns (BOXW / 2 packed words per
// thread, thread = row).  Whole warp inside the group: stage the box in
// shared memory (swizzled as the tensor map expects: 64B for 64-byte rows,
// 128B for 128-byte rows) in the next of the warp's NBUF boxes and issue one
// TMA tensor store; otherwise each valid row is stored directly.
template <bool STAGED, int NBUF, int BOXW, bool TMA_STORE>
__device__ __forceinline__ void emit_box(const KParams& p, const CUtensorMap* tmO, uint32_t stg_base, int& nbox,
                                         const uint32_t* w, bool full_warp, bool valid, int lane, int64_t row,
                                         int col, int row_base) {
    constexpr int CHUNKS = BOXW / 8;  // 16-byte chunks per row
    if (STAGED && full_warp) {
        const uint32_t stg = stg_base + (uint32_t)((nbox % NBUF) * (32 * BOXW * 2));
        ++nbox;
        if (TMA_STORE && lane == 0) {  // the store that last used this box has read it
            if (NBUF == 2) bulk_wait_read_1(); else bulk_wait_read();
        }
        __syncwarp();
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c) {
            const int sw = CHUNKS == 4 ? ((lane >> 1) & 3) : (lane & 7);  // the 64B / 128B swizzle
            const uint32_t a = stg + lane * (BOXW * 2) + ((c ^ sw) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                         :: "r"(a), "r"(w[4 * c]), "r"(w[4 * c + 1]), "r"(w[4 * c + 2]), "r"(w[4 * c + 3])
                         : "memory");
        }
        if (TMA_STORE) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(tmO, stg, col, row_base);
                bulk_commit();
            }
        } else {
            // read back row-major: each instruction moves 32 x 16 bytes of whole
            // consecutive rows (full 128-byte lines at BOXW = 64), so the
            // stores leave the SM coalesced without occupying the TMA unit
            __syncwarp();
            constexpr int RPI = 32 / CHUNKS;  // rows per instruction
            const int rr = lane / CHUNKS, c = lane % CHUNKS;
#pragma unroll
            for (int i = 0; i < 32 / RPI; ++i) {
                const int r = i * RPI + rr;
                const int sw = CHUNKS == 4 ? ((r >> 1) & 3) : (r & 7);
                uint4 v;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                             : "r"(stg + r * (BOXW * 2) + ((c ^ sw) << 4)) : "memory");
                *reinterpret_cast<uint4*>(p.out + (int64_t)(row_base + r) * p.ldo + col + c * 8) = v;
            }
            __syncwarp();  // the box is read before the warp's next box overwrites it
        }
    } else if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + row * p.ldo + col);
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c) dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
}

// Pairs of fp32 values in one 64-bit register pair, for the packed
// two-wide fp32 multiply and add (each lane rounded to nearest like the
// scalar instruction), which halve the epilogue's multiply count.
__device__ __forceinline__ uint64_t f2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float f2_lo(uint64_t v) {
    float a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
    return a;
}
__device__ __forceinline__ float f2_hi(uint64_t v) {
    float a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
    return b;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint32_t pack_bf16x2(uint64_t v) { return pack_bf16(f2_lo(v), f2_hi(v)); }

__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// silu(g) u for a pair from the accumulators a_g, a_u and the row's scale:
// g = a_g s, u = a_u s, exp(-g) = 2^(a_g e) with e = -s log2(e) (the
// hardware exp2 and reciprocal approximations: a few fp32 ulps, far inside
// the bf16 rounding that follows); exp(-g) = inf for very negative g gives
// rcp = 0 and silu = -0, no NaN.
__device__ __forceinline__ uint64_t swiglu2(uint64_t ag, uint64_t au, uint64_t scale2, uint64_t escale2) {
    const uint64_t ea = f2_mul(ag, escale2);
    const uint64_t den = f2_add(f2(ex2_approx(f2_lo(ea)), ex2_approx(f2_hi(ea))), f2(1.0f, 1.0f));
    const uint64_t sg = f2_mul(f2_mul(ag, scale2), f2(rcp_approx(f2_lo(den)), rcp_approx(f2_hi(den))));
    return f2_mul(sg, f2_mul(au, scale2));
}

// One 16-pair SwiGLU pass of an epilogue warp: bf16 D words and the running
// max of their magnitudes (bf16 magnitude bits order like unsigned integers,
// so a packed 16-bit max of the stored values gives max |bf16(d)| exactly).
template <bool PROB>
__device__ __forceinline__ uint32_t swiglu_words(const uint32_t* v, uint64_t scale2, uint64_t escale2, uint64_t prob2,
                                                 uint32_t* w) {
    uint32_t mw = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        uint64_t dv = swiglu2(f2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])),
                              f2(__uint_as_float(v[32 + 2 * j]), __uint_as_float(v[33 + 2 * j])), scale2, escale2);
        if (PROB) dv = f2_mul(dv, prob2);
        w[j] = pack_bf16x2(dv);
        mw = __vmaxu2(mw, w[j] & 0x7FFF7FFFu);
    }
    return mw;
}

// Mode 3: encode the A rows of one m-tile into the resident tile, by the 16
// epilogue warps (wi = 0..15).  Rows row0 .. row0 + arows - 1 of D (K bf16
// columns) take their outer scale from FC1's row amax; rows past arows
// encode as zero.  Per K-stage kc: 16 lanes per row (lane j of a half-warp
// takes the stage's 16-element block j), two rows per warp, four passes of
// 32 rows.  Codes go to the stage's 128-byte rows in the 128B-swizzled
// layout the TMA would have written (16-byte chunk c of row r at chunk
// c ^ (r % 8)), block scales to the stage's 512-byte atoms (row r, block j:
// byte (r % 32) 16 + (r / 32) 4 + j % 4 of atom j / 4), row scales to
// ascale.  Each warp fences its writes to the async proxy and arrives on
// a_full[kc].  The same block encode as the quantization kernels, so the
// codes and scales are those of the separate requantization.
template <class S>
__device__ __forceinline__ void encode_a_tile(S& s, const KParams& p, int row0, int arows, int mt, int k_stages,
                                              int wi, int lane) {
    const int half = lane >> 4, b = lane & 15;
    const int64_t sp4 = p.K / 64;
    uint64_t pol;  // the rows are read once: first out of L2
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    for (int kc = 0; kc < k_stages; ++kc) {
        // the stage's four passes load before any encodes: four loads in flight per lane
        uint4 lo[4], hi[4];
        float amax[4];
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {
            const int r = pass * 32 + wi * 2 + half;
            lo[pass] = make_uint4(0u, 0u, 0u, 0u);
            hi[pass] = make_uint4(0u, 0u, 0u, 0u);
            amax[pass] = 0.0f;
            if (r < arows) {
                const __nv_bfloat16* src = p.d_in + (int64_t)(row0 + r) * p.K + kc * 256 + b * 16;
                asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8], %9;"
                             : "=r"(lo[pass].x), "=r"(lo[pass].y), "=r"(lo[pass].z), "=r"(lo[pass].w),
                               "=r"(hi[pass].x), "=r"(hi[pass].y), "=r"(hi[pass].z), "=r"(hi[pass].w)
                             : "l"(src), "l"(pol));
                amax[pass] = __ldg(p.d_amax + row0 + r);
            }
        }
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {
            const int r = pass * 32 + wi * 2 + half;
            const bool valid = r < arows;
            const float s_g = outer_scale(amax[pass], 2688.0f);  // 0 for a zero row
            uint2 w = make_uint2(0u, 0u);
            uint32_t sb = 0;
            if (s_g != 0.0f) {
                const float t = __fmul_rn(6.0f, s_g);
                w = encode16(lo[pass], hi[pass], absmax16(lo[pass], hi[pass]), s_g, t, rcp_rn(t), &sb);
            }
            *reinterpret_cast<uint2*>(s.a[kc] + r * 128 + (((b >> 1) ^ (r & 7)) << 4) + ((b & 1) << 3)) = w;
            // the 4 blocks of a 64-column atom are 4 neighbouring lanes: one scale word
            uint32_t word = sb;
            word |= __shfl_down_sync(0xffffffffu, sb, 1) << 8;
            word |= __shfl_down_sync(0xffffffffu, sb, 2) << 16;
            word |= __shfl_down_sync(0xffffffffu, sb, 3) << 24;
            if ((b & 3) == 0)
                *reinterpret_cast<uint32_t*>(s.sfa[kc] + (b >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4) = word;
            if (kc == 0 && b == 0) s.ascale[r] = valid ? s_g : 0.0f;
            if (p.q_codes != nullptr) {  // inspection copies, in the separate requantization's layout
                if (valid) *reinterpret_cast<uint2*>(p.q_codes + (int64_t)(row0 + r) * (p.K / 2) + kc * 128 + b * 8) = w;
                if (valid && (b & 3) == 0)
                    *reinterpret_cast<uint32_t*>(p.q_sf + sf_group_offset((int64_t)mt * BM + r, kc * 4 + (b >> 2), sp4)) =
                        word;
                if (valid && kc == 0 && b == 0) p.q_scale[row0 + r] = s_g;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.a_full[kc]));
    }
}

// Mode 4: the router-weighted combine of the tokens whose k-th and last
// output row of one 64-column block this warp has just written.  Each row of
// the block counts its arrival on the token's counter for the block; the
// arrival that brings it to k (whichever unit that is) sums the token's k
// rows of that block, read back from Y2, in slot order -- the same fp32
// fused multiply-adds in the same order as the combine kernel, so the output
// is bit-identical and independent of which unit arrives last.  The warp's
// own writes are complete and ordered before its counts (bulk wait, proxy
// and gpu fences); the last arriver fences again before reading.  Up to four
// completed tokens at a time, eight lanes each, 8 columns per lane.
__device__ __forceinline__ void combine_completed(const KParams& p, bool valid, int64_t row, int blk, int lane) {
    const int nblk = p.N >> 6;
    bool last = false;
    int tok = 0;
    if (valid) {
        tok = __ldg(p.perm + row) / p.k_top;
        last = atomicAdd(p.ccnt + (int64_t)tok * nblk + blk, 1) == p.k_top - 1;
    }
    __threadfence();
    uint32_t lm = __ballot_sync(0xffffffffu, last);
    const int e = lane >> 3, sub = lane & 7;
    while (lm != 0u) {
        uint32_t m = lm;
        for (int i = 0; i < e; ++i) m &= m - 1u;  // drop the e lowest completed tokens
        const bool act = m != 0u;
        const int t = __shfl_sync(0xffffffffu, tok, act ? __ffs(m) - 1 : 0);
        if (act) {
            float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
            for (int sl = 0; sl < p.k_top; ++sl) {
                const int r = __ldg(p.inv + (int64_t)t * p.k_top + sl);
                const float ws = p.cw ? __ldg(p.cw + (int64_t)t * p.k_top + sl) : 1.0f;
                const uint4 y = __ldcg(reinterpret_cast<const uint4*>(p.out + (int64_t)r * p.ldo + blk * 64 + sub * 8));
                const uint32_t wv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[2 * j] = fmaf(ws, __uint_as_float(wv[j] << 16), acc[2 * j]);
                    acc[2 * j + 1] = fmaf(ws, __uint_as_float(wv[j] & 0xFFFF0000u), acc[2 * j + 1]);
                }
            }
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) o[j] = pack_bf16(acc[2 * j], acc[2 * j + 1]);
            *reinterpret_cast<uint4*>(p.cout + (int64_t)t * p.N + blk * 64 + sub * 8) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        for (int i = 0; i < 4 && lm != 0u; ++i) lm &= lm - 1u;
    }
}

// Mode 3: pull the D rows of an m-tile into L2 ahead of its encode.
__device__ __forceinline__ void prefetch_a_rows(const KParams& p, int row0, int arows) {
    const char* src = reinterpret_cast<const char*>(p.d_in + (int64_t)row0 * p.K);
    const uint32_t bytes = (uint32_t)arows * (uint32_t)p.K * 2u;
    for (uint32_t o = 0; o < bytes; o += 16384u) prefetch_l2_keep(src + o, bytes - o < 16384u ? bytes - o : 16384u);
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(threads_of<MODE>(), 1)
gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmSFB, const __grid_constant__ CUtensorMap tmO,
                  const KParams p) {
    using C = Cfg<MODE>;
    constexpr int STAGES = C::STAGES, A_BYTES = C::A_BYTES, B_BYTES = C::B_BYTES, ATOMS = C::ATOMS;
    constexpr int SFB_BYTES = C::SFB_BYTES, ROWB = C::ROWB, SWZ = C::SWZ, SBO = C::SBO;
    constexpr uint32_t SF_STAGE_COLS = C::SF_STAGE_COLS;
    constexpr int TN = C::TN, ACC_BUFS = C::ACC_BUFS, SFB_BLOCKS = C::SFB_BLOCKS, B_ROWS = C::B_ROWS;
    extern __shared__ uint8_t smem_raw[];
    Smem<MODE>& s = *reinterpret_cast<Smem<MODE>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G;
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

    // group table: dense calls are one group of M rows
    if (p.goff == nullptr) {
        if (threadIdx.x == 0) {
            s.goff[0] = 0; s.goff[1] = (int)p.M;
            s.gpoff[0] = 0; s.gpoff[1] = (int)((p.M + BM - 1) / BM * BM);
        }
    } else {
        for (int i = threadIdx.x; i <= G; i += threads_of<MODE>()) { s.goff[i] = p.goff[i]; s.gpoff[i] = p.gpoff[i]; }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(smem_u32(&s.full_a[i]), 1);
            mbar_init(smem_u32(&s.full_b[i]), 1);
            mbar_init(smem_u32(&s.sf_full[i]), 8);
            mbar_init(smem_u32(&s.empty[i]), C::DUAL ? 2 : 1);  // mode 5: a commit from each issuer
        }
        for (int i = 0; i < C::NACC; ++i) {
            mbar_init(smem_u32(&s.tmem_full[i]), 1);
            // the epilogue warps of the pair that drain this accumulator (mode 5: half of them)
            mbar_init(smem_u32(&s.tmem_empty[i]), C::DUAL ? EPI_WARPS : 2 * EPI_WARPS);
        }
        if (C::QOL)
            for (int i = 0; i < C::A_SLOTS; ++i) mbar_init(smem_u32(&s.a_full[i]), EPI_WARPS);
        mbar_init(smem_u32(&s.drain), C::DUAL ? 2 : 1);
        mbar_init(smem_u32(&s.never), 1);
        s.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        if (!C::QOL) prefetch_tmap(&tmA);
        prefetch_tmap(&tmO);
    }
    if (warp == PRODB_WARP && lane == 0) { prefetch_tmap(&tmB); prefetch_tmap(&tmSFB); }
    if (warp == 1) { tmem_alloc2(smem_u32(&s.tmem_base), TMEM_COLS); tmem_relinquish2(); }
    __syncthreads();
    if (warp == 0) {
        // ppre[g] = sum over groups before g of ceil(m-tiles / 2); lane l holds groups 8l..8l+7
        int loc[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int g = lane * 8 + j;
            loc[j] = sum;
            sum += g < G ? ((s.gpoff[g + 1] - s.gpoff[g]) / BM + 1) >> 1 : 0;
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
    // barriers initialised and TMEM allocated in both CTAs before any remote arrival
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    volatile int* abort = &s.abort;

    const int n_tiles = p.N / TN;  // mode 1: 128 gate + 128 up columns per tile
    const int total = s.ppre[G] * n_tiles;
    const int k_atoms = p.K / 64;
    const int k_stages = (k_atoms + ATOMS - 1) / ATOMS;
    // Unit order.  Modes 0-2 deal units round-robin (u = pair, pair + n_pairs,
    // ...): the n-tiles of one m-tile pair run on neighbouring pairs at once
    // and share its A rows in L2.  Mode 3 gives each pair whole m-tile pairs,
    // all n-tiles back to back on the resident A tile.
    const int u_first = C::QOL ? pair * n_tiles : pair;
    auto u_next = [&](int u) {
        return C::QOL ? ((u + 1) % n_tiles == 0 ? u + 1 + (n_pairs - 1) * n_tiles : u + 1) : u + n_pairs;
    };

    if ((warp == 0 && !C::QOL) || warp == PRODB_WARP) {
        if (lane == 0) {
            // ------------------------------------------------------------ producers
            // warp 0: A rows + their scales; warp 22: B half + weight scales
            const bool is_a = warp == 0 && !C::QOL;  // mode 3 has no A producer (warp 0 idles)
            uint64_t* full = is_a ? s.full_a : s.full_b;
            int stage = 0, issued = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = u_first; u < total && ok; u = u_next(u)) {
                const Tile x = decode_unit(s, G, n_tiles, u, rank);
                // 128-row weight blocks of the tile: mode 1 takes 128 gate and
                // 128 up rows of the expert (one per CTA), mode 0 the tile's
                // SFB_BLOCKS adjacent blocks, each CTA staging half the rows
                const int jb0 = x.g * (p.N / 128) + (MODE == 1 ? 1 : SFB_BLOCKS) * x.nt;
                const int jb1 = x.g * (p.N / 128) + p.N / 256 + x.nt;
                const int brow = MODE == 1 ? (rank == 0 ? jb0 : jb1) * 128 : jb0 * 128 + (int)rank * B_ROWS;
                for (int ks = 0; ks < k_stages; ++ks) {
                    if (!mbar_wait_bounded(smem_u32(&s.empty[stage]), phase ^ 1, abort, p.err)) { ok = false; break; }
                    const uint32_t fb = smem_u32(&full[stage]);
                    if (is_a) {
                        const int na = k_atoms - ks * ATOMS < ATOMS ? k_atoms - ks * ATOMS : ATOMS;
                        mbar_arrive_expect_tx(fb, A_BYTES + na * 512);
                        tma_load_2d(smem_u32(s.a[stage]), &tmA, fb, ks * ROWB, x.row0);
                        bulk_load(smem_u32(s.sfa[stage]), p.a_sf + ((int64_t)x.mt * k_atoms + ks * ATOMS) * 512,
                                  na * 512, fb);
                    } else {
                        // the scale box is always whole: atoms past K are zero-filled
                        mbar_arrive_expect_tx(fb, B_BYTES + SFB_BYTES);
                        if constexpr (C::DUAL) {
                            // half h of the tile (its 128 weight rows) is split between the pair:
                            // this CTA stages rows h * 128 + rank * 64 .. + 63 at b + h * (B_BYTES / 2)
                            tma_load_2d(smem_u32(s.b[stage]), &tmB, fb, ks * ROWB, jb0 * 128 + (int)rank * 64);
                            tma_load_2d(smem_u32(s.b[stage]) + B_BYTES / 2, &tmB, fb, ks * ROWB,
                                        jb0 * 128 + 128 + (int)rank * 64);
                        } else {
                            tma_load_2d(smem_u32(s.b[stage]), &tmB, fb, ks * ROWB, brow);
                        }
                        if (MODE == 1)
                            tma_load_4d(smem_u32(s.sfb[stage]), &tmSFB, fb, 0, ks * ATOMS, x.nt, 2 * x.g);
                        else
                            tma_load_3d(smem_u32(s.sfb[stage]), &tmSFB, fb, 0, ks * ATOMS, jb0);
                    }
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                raise_abort(&s.abort, rank);
                // drain: the last load issued into each stage has landed (bounded wait)
                for (int st = 0; st < STAGES && st < issued; ++st) {
                    const int idx = st + (issued - 1 - st) / STAGES * STAGES;  // last stage issued into slot st
                    mbar_wait_drain(smem_u32(&full[st]), (uint32_t)(idx / STAGES) & 1u);
                }
            }
        }
    } else if (warp == 1 || (C::DUAL && warp == ISSUE2_WARP)) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------------------ MMA issuer (even CTA)
            // Mode 5 has two: warp 1 issues the MMAs of the tile's first 128
            // columns into accumulator 0, warp 23 those of the last 128 into
            // accumulator 1 (N = 128 each; both read the same A stage, each its
            // half of B, and both commit on the stage's empty barrier).
            // The issuing thread's instruction stream is kept short (it shares
            // its scheduler with epilogue warps): descriptors of stage 0 are
            // built once, a stage / K-step adds its byte offset >> 4 to the
            // start-address field, and the K-steps are unrolled.  The wait on
            // sf_full alone suffices: this CTA's scale writers arrive on it
            // only after both of its stage's copies have landed, the peer's
            // after the peer's have.
            const int hh = (C::DUAL && warp == ISSUE2_WARP) ? 1 : 0;  // mode 5: the half this thread issues
            const uint64_t adesc0 = smem_desc(smem_u32(s.a[0]), 0, SBO, SWZ);
            const uint64_t bdesc0 = smem_desc(smem_u32(s.b[0]) + (C::DUAL ? hh * (B_BYTES / 2) : 0), 0, SBO, SWZ);
            int stage = 0, it = 0;
            uint32_t phase = 0;
            bool ok = true;
            // the time-out test: a bounded wait for a phase that never completes
            if (p.stall && hh == 0) ok = mbar_wait_bounded_relaxed(smem_u32(&s.never), 0, abort, p.err);
            for (int u = u_first; u < total && ok; u = u_next(u), ++it) {
                // accumulator it % ACC_BUFS, in its (it / ACC_BUFS)-th use; mode 5: this half's
                const int ab = C::DUAL ? hh : (ACC_BUFS == 1 ? 0 : (it & 1));
                const uint32_t acc_phase = (uint32_t)(ACC_BUFS == 1 ? it : it >> 1) & 1u;
                if (!mbar_wait_bounded_relaxed(smem_u32(&s.tmem_empty[ab]), acc_phase ^ 1, abort, p.err)) { ok = false; break; }
                tc_fence_after();
                for (int ks = 0; ks < k_stages; ++ks) {
                    if (!mbar_wait_bounded_relaxed(smem_u32(&s.sf_full[stage]), phase, abort, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const int na = k_atoms - ks * ATOMS;
                    const uint32_t sfc = tmem + SF_COL + stage * SF_STAGE_COLS;
                    const uint64_t ad = adesc0 + (uint64_t)(((C::QOL ? ks : stage) * A_BYTES) >> 4);
                    const uint64_t bd = bdesc0 + (uint64_t)((stage * B_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < ATOMS; ++kk) {
                        if (kk < na) {
                            if constexpr (C::DUAL)  // half hh: 128 accumulator columns, its 128-row weight-scale block
                                tc_mma2_nvfp4(tmem + ACC_COL + hh * (TN / 2), ad + 2 * kk, bd + 2 * kk, C::IDESC,
                                              sfc + kk * 4, sfc + 4 * ATOMS + kk * 4 * SFB_BLOCKS + 4 * hh,
                                              (ks | kk) != 0);
                            else
                                tc_mma2_nvfp4(tmem + ACC_COL + ab * TN, ad + 2 * kk, bd + 2 * kk, C::IDESC,
                                              sfc + kk * 4, sfc + 4 * ATOMS + kk * 4 * SFB_BLOCKS, (ks | kk) != 0);
                        }
                    }
                    tc_commit2_mc(smem_u32(&s.empty[stage]), 3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit2_mc(smem_u32(&s.tmem_full[ab]), 3);
            }
            if (!ok) raise_abort(&s.abort, rank);
            // every MMA issued by this thread completes before TMEM is released
            tc_commit2_mc(smem_u32(&s.drain), 1);
            mbar_wait_drain(smem_u32(&s.drain), 0);
        }
    } else if (warp >= 2 && warp < EPI_WARP0) {
        // ---------------------------------------------------------------- scale writers
        // Warp w writes TMEM lane quarter w % 4.  Each scale atom (32 lines
        // of 16 bytes; line i holds the 4 scales of rows i, i+32, i+64, i+96)
        // goes to 4 consecutive columns of every quarter: thread i of each
        // quarter writes line i.  SFA atom kk -> columns sfc + 4kk; SFB atom kk
        // of 128-row block hh -> columns sfc + 4*ATOMS + 4*SFB_BLOCKS*kk + 4hh.
        const int q = warp & 3;
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int it = 0;
        for (int u = u_first; u < total && ok; u = u_next(u), ++it) {
            for (int ks = 0; ks < k_stages; ++ks) {
                // mode 3: stage ks of the resident A tile, encoded for this unit's m-tile (the it / n_tiles-th)
                const bool a_in = C::QOL ? mbar_wait_bounded(smem_u32(&s.a_full[ks]), (uint32_t)(it / n_tiles) & 1u, abort, p.err)
                                         : mbar_wait_bounded(smem_u32(&s.full_a[stage]), phase, abort, p.err);
                if (!a_in || !mbar_wait_bounded(smem_u32(&s.full_b[stage]), phase, abort, p.err)) { ok = false; break; }
                const uint32_t sfc = lane_addr + SF_COL + stage * SF_STAGE_COLS;
                // the stage's SFA columns (4 per atom) and SFB columns (4 per atom and 128-row
                // block) are contiguous runs: one wide store each
                uint32_t fa[4 * ATOMS], fb[4 * ATOMS * SFB_BLOCKS];
#pragma unroll
                for (int kk = 0; kk < ATOMS; ++kk) {
                    const uint4 a = *reinterpret_cast<const uint4*>(s.sfa[C::QOL ? ks : stage] + kk * 512 + lane * 16);
                    fa[4 * kk] = a.x; fa[4 * kk + 1] = a.y; fa[4 * kk + 2] = a.z; fa[4 * kk + 3] = a.w;
#pragma unroll
                    for (int hh = 0; hh < SFB_BLOCKS; ++hh) {
                        const uint4 b = *reinterpret_cast<const uint4*>(s.sfb[stage] + hh * (ATOMS * 512) + kk * 512 +
                                                                        lane * 16);
                        uint32_t* d = fb + 4 * (SFB_BLOCKS * kk + hh);
                        d[0] = b.x; d[1] = b.y; d[2] = b.z; d[3] = b.w;
                    }
                }
                static_assert(4 * ATOMS == 16 && (SFB_BLOCKS == 1 || SFB_BLOCKS == 2), "scale store widths");
                tmem_st16(sfc, fa);
                if constexpr (SFB_BLOCKS == 2) tmem_st32(sfc + 4 * ATOMS, fb);
                else tmem_st16(sfc + 4 * ATOMS, fb);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&s.sf_full[stage]), 0));
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
        }
        if (!ok && lane == 0) raise_abort(&s.abort, rank);
    } else if (warp >= EPI_WARP0 && warp < PRODB_WARP) {
        // ---------------------------------------------------------------- epilogue
        // Each warp copies its 32 rows x 64 accumulator columns into
        // registers (mode 1: 32 gate and the matching 32 up columns) and
        // releases them with one arrival on the even CTA's tmem_empty, so the
        // MMAs that need the accumulator can run while the warps scale,
        // activate and store.
        const int q = warp & 3;                    // TMEM lane quarter this warp may access
        const int cg = (warp - EPI_WARP0) >> 2;    // column group 0..3
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        bool ok = true;
        int nbox = 0;  // staged boxes this warp has stored
        int it = 0;    // tiles of this CTA so far
        const int wi = warp - EPI_WARP0;
        float sa_m = 0.0f;  // mode 3: this thread's row scale in the current m-tile
        if (C::QOL && u_first < total) {
            // the pair's first m-tile: encode it, and pull the next one's rows into L2
            const Tile x0 = decode_unit(s, G, n_tiles, u_first, rank);
            encode_a_tile(s, p, x0.row0, x0.arows, x0.mt, k_stages, wi, lane);
            const int un = u_first + n_pairs * n_tiles;
            if (wi == 0 && lane == 0 && un < total) {
                const Tile xn = decode_unit(s, G, n_tiles, un, rank);
                prefetch_a_rows(p, xn.row0, xn.arows);
            }
        }
        for (int u = u_first; u < total; u = u_next(u), ++it) {
            // mode 5: column groups 0-1 drain accumulator 0 (the tile's first 128 columns), 2-3 accumulator 1
            const int ab = C::DUAL ? (cg >> 1) : (ACC_BUFS == 1 ? 0 : (it & 1));
            const uint32_t acc_phase = (uint32_t)(ACC_BUFS == 1 ? it : it >> 1) & 1u;
            const Tile x = decode_unit(s, G, n_tiles, u, rank);
            const int rl = q * 32 + lane;
            const bool valid = rl < x.rows;
            const int64_t row = (int64_t)x.row0 + rl;
            // scales are fetched before the wait so their latency hides under the MMAs
            float sa;
            if (C::QOL) {
                // the m-tile's first unit: every warp's encode of it is complete (and its
                // row scales visible) once a_full[0] has its phase; the scale stays in a
                // register for the m-tile's units, as the next encode rewrites ascale
                if (x.nt == 0) {
                    if (!mbar_wait_bounded(smem_u32(&s.a_full[0]), (uint32_t)(it / n_tiles) & 1u, abort, p.err)) {
                        ok = false;
                        break;
                    }
                    sa_m = s.ascale[rl];
                }
                sa = valid ? sa_m : 0.0f;
            } else {
                sa = valid ? __ldg(p.a_scale + row) : 0.0f;
            }
            const float sbw = __ldg(p.b_scale + x.g);
            const float prob = (valid && p.row_prob) ? __ldg(p.row_prob + row) : 1.0f;
            if (!mbar_wait_bounded_relaxed(smem_u32(&s.tmem_full[ab]), acc_phase, abort, p.err)) { ok = false; break; }
            tc_fence_after();
            uint32_t v[C::PLAIN ? C::CPW : 64];
            if (C::PLAIN) {
#pragma unroll
                for (int h = 0; h < C::CPW / 32; ++h)
                    tmem_ld32(lane_addr + ACC_COL + (C::DUAL ? 0 : ab * TN) + cg * C::CPW + 32 * h, v + 32 * h);
            } else {
                tmem_ld32(lane_addr + ACC_COL + cg * 32, v);             // gate
                tmem_ld32(lane_addr + ACC_COL + 128 + cg * 32, v + 32);  // up
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            // Each warp releases its share of the accumulator itself: an arrival
            // on the even CTA's barrier, which completes when all 32 warps of
            // the pair have theirs in registers.  A warp arrives for tile t + 1
            // only after tile t + 1's commit, which follows that completion.
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&s.tmem_empty[ab]), 0));
            // Mode 3, the m-tile's last unit: its MMAs (done: tmem_full) no longer read
            // the resident tile, so the pair's next m-tile is encoded over it.  Run
            // after this unit's outputs have left the registers (staged and stored).
            auto encode_next = [&]() {
                if (!C::QOL || x.nt != n_tiles - 1) return;
                const int un = u_next(u);
                if (un >= total) return;
                const Tile xn = decode_unit(s, G, n_tiles, un, rank);
                encode_a_tile(s, p, xn.row0, xn.arows, xn.mt, k_stages, wi, lane);
                const int un2 = un + n_pairs * n_tiles;
                if (wi == 0 && lane == 0 && un2 < total) {
                    const Tile x2 = decode_unit(s, G, n_tiles, un2, rank);
                    prefetch_a_rows(p, x2.row0, x2.arows);
                }
            };
            if (x.rows == 0) {  // the odd CTA of a group's last pair: nothing to store
                encode_next();
                continue;
            }
            const float scale = __fmul_rn(sa, sbw);
            const uint64_t scale2 = f2(scale, scale);
            // all 32 rows of this warp inside the tile's group: TMA store; else direct
            const bool full_warp = q * 32 + 32 <= x.rows;
            const uint32_t stg = smem_u32(s.stg[(warp - EPI_WARP0) * C::NBUF]);
            if (C::PLAIN) {
                uint32_t w[C::CPW / 2];
#pragma unroll
                for (int j = 0; j < C::CPW / 2; ++j)
                    w[j] = pack_bf16x2(f2_mul(f2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), scale2));
#pragma unroll
                for (int hf = 0; hf < C::CPW / C::BOXW; ++hf)
                    emit_box<C::STAGED, C::NBUF, C::BOXW, C::TMA_STORE>(p, &tmO, stg, nbox, w + hf * (C::BOXW / 2),
                                                                         full_warp, valid, lane, row,
                                                                         x.nt * TN + cg * C::CPW + hf * C::BOXW,
                                                                         x.row0 + q * 32);
                if constexpr (C::COMB) {
                    // this warp's block of Y2 is complete and visible before its rows count
                    if (lane == 0) {
                        bulk_wait_all();
                        fence_proxy_async_global();
                        __threadfence();
                    }
                    __syncwarp();
                    fence_proxy_async_global();
                    __threadfence();
                    combine_completed(p, valid, row, (x.nt * TN + cg * C::CPW) >> 6, lane);
                }
            } else {
                if (valid && p.c_debug) {
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
                uint32_t w[16];
                const float es = __fmul_rn(scale, -1.44269504088896341f);
                const uint64_t escale2 = f2(es, es);
                uint32_t mw = p.row_prob ? swiglu_words<true>(v, scale2, escale2, f2(prob, prob), w)
                                         : swiglu_words<false>(v, scale2, escale2, 0, w);
                emit_box<C::STAGED, C::NBUF, C::BOXW, C::TMA_STORE>(p, &tmO, stg, nbox, w, full_warp, valid, lane, row,
                                                      x.nt * 128 + cg * 32, x.row0 + q * 32);
                // the row's max |bf16(d)| over this warp's 32 columns
                if (valid) {
                    mw = __vmaxu2(mw, mw >> 16);
                    const float mb = __uint_as_float((mw & 0xFFFFu) << 16);
                    atomicMax(reinterpret_cast<unsigned int*>(p.amax_out + row), __float_as_uint(mb));
                }
            }
            encode_next();
        }
        if (!ok && lane == 0) raise_abort(&s.abort, rank);
        if (C::STAGED && lane == 0) bulk_wait_all();  // this warp's tensor stores are complete before exit
        __syncwarp();
    }
    // neither CTA leaves while the pair's MMAs, commits or arrivals may still touch it
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
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2D uint8 view [rows x row_bytes] of packed FP4 codes: boxes of ROWB bytes x
// box_rows rows, swizzled to match the MMA descriptors of the mode.
bool make_codes_map(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes, int mode, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int rowb = mode == 0 ? Cfg<0>::ROWB : Cfg<1>::ROWB;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)rowb, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, rowb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Weight scales, stored as 128-row blocks of k_atoms 512-byte atoms, viewed
// as 32-bit words so one tensor copy brings a stage's atoms of the tile's
// weight rows: mode 0 (the tile's blocks from jb) as 3D {128, k_atoms, G*N/128}
// with box {128, ATOMS, blocks per tile}; mode 1 (gate block nt and up block N/256 + nt of expert
// g) as 4D {128, k_atoms, N/256, 2G} with box {128, ATOMS, 1, 2}, the up
// block being one step of the last dimension away.
bool make_sfb_map(CUtensorMap* m, const void* base, int G, int N, int K, int mode) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t k_atoms = (cuuint64_t)(K / 64);
    const cuuint32_t atoms = (cuuint32_t)(mode == 0 ? Cfg<0>::ATOMS : Cfg<1>::ATOMS);
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (mode == 0) {
        cuuint64_t dims[3] = {128, k_atoms, (cuuint64_t)G * (N / 128)};
        cuuint64_t strides[2] = {512, k_atoms * 512};
        cuuint32_t box[3] = {128, atoms, (cuuint32_t)Cfg<0>::SFB_BLOCKS};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    cuuint64_t dims[4] = {128, k_atoms, (cuuint64_t)(N / 256), 2 * (cuuint64_t)G};
    cuuint64_t strides[3] = {512, k_atoms * 512, k_atoms * 512 * (cuuint64_t)(N / 256)};
    cuuint32_t box[4] = {128, atoms, 1, 2};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D bf16 view [rows x cols] (row stride ld elements) of an output: 32-row
// boxes of box_cols columns, 64B swizzle for 32 columns, 128B for 64.
bool make_out_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Pairs that can be resident at once for the kernel of one mode (clusters of
// two CTAs of one SM each), from the occupancy calculator; 0 on failure.
template <int MODE>
int resident_pairs(size_t smem, int num_sms) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms & ~1), 1, 1);
    cfg.blockDim = dim3(threads_of<MODE>(), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_nvfp4_kernel<MODE>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsfb, const CUtensorMap& to,
                        const KParams& p,
                        int num_sms, int64_t dense_units, cudaStream_t stream) {
    const size_t smem = sizeof(Smem<MODE>) + 1024;
    static std::mutex mu;
    static int pairs_cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    int pairs = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 0 && dev < 64) pairs = pairs_cache[dev];
        if (pairs == 0) {
            cudaError_t e = cudaFuncSetAttribute(gemm_nvfp4_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
            pairs = resident_pairs<MODE>(smem, num_sms);
            if (pairs <= 0) pairs = num_sms / 2;
            if (dev >= 0 && dev < 64) pairs_cache[dev] = pairs;
        }
    }
    if (dense_units > 0 && dense_units < pairs) pairs = (int)dense_units;
    if (pairs < 1) pairs = 1;
    gemm_nvfp4_kernel<MODE><<<2 * pairs, threads_of<MODE>(), smem, stream>>>(ta, tb, tsfb, to, p);
    return cudaGetLastError();
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
    const bool qol = g.mode == 3;
    if (qol && (g.goff == nullptr || g.d_in == nullptr || g.d_amax == nullptr || g.K % 256 != 0 ||
                g.K / 256 > Cfg<3>::KCH || g.N % 256 != 0 || g.N / 256 < 2))
        return cudaErrorInvalidValue;
    if (g.mode == 4 && (g.goff == nullptr || g.perm == nullptr || g.inv == nullptr || g.cout == nullptr ||
                        g.ccnt == nullptr || g.k_top < 1 || g.K / 256 >= 4))
        return cudaErrorInvalidValue;
    const int map_mode = g.mode == 1 ? 1 : 0;  // modes 0, 2 and 3 share the plain tensor maps
    CUtensorMap ta, tb, tsfb, to;
    // plain GEMMs with long K loops (4 or more stages of 256) take the 5-stage form;
    // shorter ones the two-issuer form (mode 5)
    const int plain_mode = (g.K / 256 >= 4) ? 2 : 5;
    const bool dual = g.mode == 0 && plain_mode == 5;
    // mode 5 stages each half of a CTA's weight rows as its own 64-row box
    const int b_rows = dual ? Cfg<5>::B_ROWS / 2 : (map_mode == 0 ? Cfg<0>::B_ROWS : Cfg<1>::B_ROWS);
    if (!make_codes_map(&tb, g.b_codes, (int64_t)g.G * g.N, g.K / 2, map_mode, b_rows)) return cudaErrorInvalidValue;
    // mode 3 has no A tensor (the kernel encodes A): its map argument repeats B's, unused
    if (qol) ta = tb;
    else if (!make_codes_map(&ta, g.a_codes, g.M, g.K / 2, map_mode, BM)) return cudaErrorInvalidValue;
    if (!make_sfb_map(&tsfb, g.b_sf, g.goff ? g.G : 1, g.N, g.K, map_mode)) return cudaErrorInvalidValue;
    const int64_t out_cols = g.mode == 1 ? g.N / 2 : g.N;
    const int box_cols = g.mode == 1 ? Cfg<1>::BOXW : (g.mode == 0 && plain_mode == 2 ? Cfg<2>::BOXW : Cfg<0>::BOXW);
    if (!make_out_map(&to, g.out, g.M, out_cols, g.ldo, box_cols)) return cudaErrorInvalidValue;
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
    p.stall = g.stall;
    p.d_in = reinterpret_cast<const __nv_bfloat16*>(g.d_in);
    p.d_amax = g.d_amax;
    p.q_codes = g.q_codes;
    p.q_sf = g.q_sf;
    p.q_scale = g.q_scale;
    p.perm = g.perm;
    p.inv = g.inv;
    p.cw = g.cw;
    p.cout = reinterpret_cast<__nv_bfloat16*>(g.cout);
    p.ccnt = g.ccnt;
    p.k_top = g.k_top;
    const int num_sms = g.num_sms > 0 ? g.num_sms : 148;
    // dense calls: no more pairs than units of work (m-tile pairs x n-tiles)
    const int tn = g.mode == 1 ? Cfg<1>::TN : Cfg<0>::TN;
    const int64_t dense_units = g.goff == nullptr ? ((g.M + BM - 1) / BM + 1) / 2 * (g.N / tn) : 0;
    if (qol) return launch_mode<3>(ta, tb, tsfb, to, p, num_sms, 0, stream);
    if (g.mode == 4) return launch_mode<4>(ta, tb, tsfb, to, p, num_sms, 0, stream);
    if (g.mode == 0 && plain_mode == 2) return launch_mode<2>(ta, tb, tsfb, to, p, num_sms, dense_units, stream);
    if (dual) return launch_mode<5>(ta, tb, tsfb, to, p, num_sms, dense_units, stream);
    if (g.mode == 0) return launch_mode<0>(ta, tb, tsfb, to, p, num_sms, dense_units, stream);
    return launch_mode<1>(ta, tb, tsfb, to, p, num_sms, dense_units, stream);
}

}  // namespace nvfp4
