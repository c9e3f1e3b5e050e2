// kernels.h -- internal launch interfaces between the C ABI layer (api.cu)
// and the kernel files.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

struct QuantLaunch {
    const void* x;          // bf16 [rows x cols], row stride ld elements
    int64_t ld, rows, cols;
    const float* amax_in;   // nullable
    int per_tensor;
    uint8_t* codes;
    uint8_t* sf;
    int64_t sf_ld;          // 0: swizzled MMA layout; > 0: row-linear, sf_ld bytes per row (multiple of 4)
    float* scale;
    const int* goff;        // nullable: scale rows remapped by group padding
    const int* gpoff;
    int G;
    int reverse;            // rows taken last to first
    int fos;                // four-over-six: 0 off, 1 by MSE, 2 by MAE
    int x_once;             // the rows are read once: their L2 lines are marked evict-first, so
                            // that they do not push the outputs out of L2 before the next kernel
    int groups;             // per_tensor: one outer scale per group of rows / groups rows (0 or 1: one)
    void* ws;               // >= 16 + 4 * groups bytes when per_tensor && !amax_in
    uint32_t* err;          // nullable device error word (pipeline wait time-outs)
};
cudaError_t launch_quantize(const QuantLaunch& q, cudaStream_t stream);

// NVFP4 rows -> bf16 y = RN16(q s_b s_g) (the exact product, rounded once).
struct DequantLaunch {
    const uint8_t* codes;   // [rows x cols/2]
    const uint8_t* sf;      // swizzled block scales
    const float* scale;     // [rows]; per_tensor: [1], or [G] (one per group) when goff is given
    int64_t rows, cols;
    int per_tensor;
    const int* goff;        // nullable: scale rows padded per group (goff/gpoff [G+1])
    const int* gpoff;
    int G;
    int padded_rows;        // y rows follow the padded layout too (padding rows zeroed)
    void* y;                // bf16, row stride ldy elements
    int64_t ldy;
};
cudaError_t launch_dequantize(const DequantLaunch& d, cudaStream_t stream);

// Grouped / dense block-scaled NVFP4 GEMM on tcgen05.
//   A rows [M_total x K] (codes + swizzled scales padded per group by
//   gpoff + per-row fp32 scale); B per group [N x K] (codes + swizzled
//   scales + one fp32 scale per group).  Mode 0 writes bf16 [M x N]; mode 1
//   (SwiGLU) reads B rows [gate F | up F] (N = 2F) and writes bf16 D [M x F]
//   plus a per-row atomic amax of D.
struct GemmLaunch {
    const uint8_t* a_codes;
    const uint8_t* a_sf;
    const float* a_scale;
    int64_t M;             // rows of A (dense) or the bound on rows (grouped)
    const uint8_t* b_codes;
    const uint8_t* b_sf;
    const float* b_scale;  // [G]
    int N, K, G;
    const int* goff;       // nullable (dense: one group of M rows)
    const int* gpoff;
    int mode;              // 0 plain, 1 SwiGLU, 3 plain with A encoded from bf16 rows in the kernel, 4 plain + combine
    void* out;             // bf16
    int64_t ldo;
    float* amax_out;       // mode 1
    const float* row_prob; // mode 1, nullable: D *= row_prob[row] (router weight at FC1)
    float* c_debug;        // mode 1, nullable: fp32 [M x N] pre-activation
    uint32_t* err;         // nullable
    int num_sms;
    int stall;             // test of the time-out path: the MMA thread waits on a barrier nothing arrives at
    // mode 3 (plain out, A encoded in the kernel from bf16 rows; grouped, K a
    // multiple of 256 up to 768, N a multiple of 256 of at least 512): D
    // [M x K] bf16 and its row amax [M] stand in for a_codes / a_sf /
    // a_scale; q_codes / q_sf / q_scale (nullable) receive copies of the
    // encoded codes, swizzled padded-row block scales and row scales
    const void* d_in;
    const float* d_amax;
    uint8_t* q_codes;
    uint8_t* q_sf;
    float* q_scale;
    // mode 4 (mode 0 plus the router-weighted combine in the epilogue; grouped,
    // N a multiple of 64): perm [M] (token * k_top + slot of each row), inv
    // [T x k_top], combine weights cw [T x k_top] (nullable: 1), the layer
    // output cout bf16 [T x N], zeroed arrival counters ccnt [T x N/64]
    const int* perm;
    const int* inv;
    const float* cw;
    void* cout;
    int* ccnt;
    int k_top;
};
cudaError_t launch_gemm(const GemmLaunch& g, cudaStream_t stream);

// Grouped BF16 GEMMs of the dequantized backward (tcgen05 kind::f16), over
// row groups of the 128-row-padded expert layout (gpoff [G+1], multiples of
// 128, padding rows zero) or one dense group of `rows` rows (gpoff null):
//   dgrad (wgrad == 0): out [rows x kf] = dy [rows x nf] . w_g [nf x kf]
//   wgrad (wgrad == 1): out_g [nf x kf] = dy[rows of g]^T . x[rows of g]
struct GemmBf16Launch {
    int wgrad;
    const void* dy;        // bf16 [rows x nf]
    const void* w;         // dgrad: bf16 [G*nf x kf] (w_g = DQ(Q(W_g)) as stored, [nf x kf])
    const void* x;         // wgrad: bf16 [rows x kf]
    void* out;             // dgrad: bf16 [rows x kf]; wgrad: bf16 [G*nf x kf]
    int64_t rows;
    int nf, kf;
    const int* gpoff;      // nullable
    int G;
    uint32_t* err;         // nullable
    int num_sms;
};
cudaError_t launch_gemm_bf16(const GemmBf16Launch& g, cudaStream_t stream);

struct RouteLaunch {
    const float* logits;   // [T x E]
    const float* bias;     // nullable
    int64_t T;
    int E, k;
    int* ids;              // [T x k]
    float* w;              // [T x k]
    int* chunk_cnt;        // [nchunks x E]
    int* chunk_base;       // [nchunks x E]
    int* cnt;              // [E]
    int* off;              // [E+1]
    int* poff;             // [E+1]
    unsigned int* done;    // one counter word, zero before the call, left zero after
    int* perm;             // [T*k]
    int* inv;              // [T*k]
    uint32_t* err;
    // permute (gather quantized X rows into expert order)
    const uint8_t* xq_codes;
    const uint8_t* xq_sf;  // row-linear [T x H/16]
    const float* xq_scale;
    int64_t H;
    uint8_t* a1_codes;
    uint8_t* a1_sf;
    float* a1_scale;
    float* amax2;          // zeroed here for the FC1 epilogue ([T*k])
    float* row_w;          // nullable: [T*k] router weight of each expert-ordered row
    int* comb_cnt;         // nullable: [T x comb_blocks] arrival counters of the combine inside FC2, zeroed here
    int comb_blocks;
};
constexpr int kRouteChunk = 32;  // tokens per chunk of the stable scatter (one bitmap word)
cudaError_t launch_route(const RouteLaunch& r, cudaStream_t stream);       // top-k, then the rest
cudaError_t launch_route_topk(const RouteLaunch& r, cudaStream_t stream);  // top-k + chunk histograms
cudaError_t launch_route_rest(const RouteLaunch& r, cudaStream_t stream);  // scan, scatter, permute
// Per-token quantization of X and the router top-k in one launch (their
// blocks interleaved: independent work, both latency-bound); separate
// launches where the shapes fall outside the fused instances.
cudaError_t launch_quantize_topk(const QuantLaunch& q, const RouteLaunch& r, cudaStream_t stream);

struct CombineLaunch {
    const void* y;         // bf16 [R x H]
    const int* inv;        // [T x k]
    const float* w;        // [T x k], nullable = weights of 1
    int64_t T, H;
    int k;
    void* out;             // bf16 [T x H]
};
cudaError_t launch_combine(const CombineLaunch& c, cudaStream_t stream);

int device_sm_count();
int set_last_error(int code, const char* msg);

}  // namespace nvfp4
