/*
 * nvfp4moe.h -- C ABI of the per-token NVFP4 W4A4 forward path for GB300 (sm_103a).
 *
 * Three compute calls, following the problem statement of the pages:
 *   nvfp4_quantize_rows  bf16 rows -> packed E2M1 codes, one E4M3 scale per
 *                        16-element block (in the swizzled layout that block-
 *                        scaled tensor-core MMA reads), one fp32 scale per row
 *                        (activations) or per tensor (weights).
 *   nvfp4_linear         dense W4A4 GEMM Y = bf16(deq(X) . deq(W)^T).
 *   moe_expert_forward   route -> permute by expert -> FC1 gate/up -> SwiGLU
 *                        -> requant -> FC2 -> router-weighted combine.
 *
 * Sources (page title, section):
 *   "miniTE Technical Report: Stable and Efficient Reinforcement Learning
 *   with Native NVFP4": 2.2 (x^ = q s_b s_g), 2.3 and 5.1 (per-token outer
 *   scale), 5.2 (contiguous quantized buffers, device-side expert offsets,
 *   zero-token experts and padding in one grouped path, workspace reuse),
 *   5.3 (amax computed where data are produced and reused by the quantizer),
 *   5.4 (block-scaled GEMM epilogue ACC x alpha_a[m] x alpha_b, C = gate|up,
 *   D = act(gate, up), concurrent amax of D), 5.6 (gs = gamax / 2688, zero
 *   rows give zero).
 *   "The 4-bitter Lesson": baseline recipe (per-token activation scale fused
 *   into the quantization kernel; weights with one fp32 scale per tensor).
 *
 * Conventions for every call:
 *   - All buffers are DEVICE memory allocated and owned by the caller.  The
 *     library never allocates, frees, synchronizes or copies to the host.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream) and completes asynchronously.
 *   - Return value 0 = enqueued; negative = rejected before any launch
 *     (nothing was written), or a launch error:
 *       NVFP4_EINVAL  -1  null pointer / bad enum / negative size
 *       NVFP4_ESHAPE  -2  unsupported shape (see each call)
 *       NVFP4_EALIGN  -3  misaligned pointer or leading dimension
 *       NVFP4_EWORKSPACE -4 workspace too small
 *       NVFP4_ELAUNCH -5  CUDA error while enqueueing
 *     nvfp4_last_error() returns a message for the last failure on the
 *     calling thread.
 *   - Inputs must be finite; NaN/Inf inputs are outside the contract.
 *   - Device-side faults are never raised on purpose: a kernel that detects
 *     an inconsistency (or a pipeline wait that exceeds its time limit)
 *     ORs a bit into a device error word and returns.  The error word is
 *     the first uint32 of `ws` for nvfp4_linear (when ws_bytes >= 4) and
 *     nvfp4_quantize_rows (when ws_bytes >= 16), and the `err` slot of
 *     moe_expert_forward's workspace.  The library never clears it: the
 *     caller zeroes it and reads it when convenient.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NVFP4_API __attribute__((visibility("default")))
#else
#define NVFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4_OK 0
#define NVFP4_EINVAL (-1)
#define NVFP4_ESHAPE (-2)
#define NVFP4_EALIGN (-3)
#define NVFP4_EWORKSPACE (-4)
#define NVFP4_ELAUNCH (-5)

/* Scale modes of nvfp4_quantize_rows. */
#define NVFP4_PER_ROW 0    /* one fp32 outer scale per row (per token) */
#define NVFP4_PER_TENSOR 1 /* one fp32 outer scale for the whole matrix */
/* Four-over-six block scaling, OR-ed into the scale mode (at most one of
 * the two): per 16-block the max maps to 6 or to 4, whichever gives the
 * smaller block error ("The 4-bitter Lesson", Four-Over-Six for RL Weights
 * and Activations); see nvfp4_quantize_rows. */
#define NVFP4_FOUR_OVER_SIX_MSE 2 /* error = sum of squared differences */
#define NVFP4_FOUR_OVER_SIX_MAE 4 /* error = sum of absolute differences */
/* nvfp4_dequantize_rows only: write row r at its padded row (see there). */
#define NVFP4_DQ_PADDED_ROWS 8

/* Bits of the device error word. */
#define NVFP4_DEVERR_TIMEOUT 1u   /* a pipeline wait (GEMM or quantizer) ran past its limit */
#define NVFP4_DEVERR_BADEXPERT 2u /* a routed expert id outside [0, E) */
#define NVFP4_DEVERR_BADGROUP 4u  /* grouped BF16 GEMM: padded offsets not ascending multiples of 128 */

/*
 * An NVFP4 matrix [rows x cols] in device memory (caller-owned):
 *   codes  uint8 [rows x cols/2]: E2M1 codes, row-major, element 2i of a row
 *          in the low nibble of byte i, element 2i+1 in the high nibble;
 *          code = sign bit (8) | index into {0, .5, 1, 1.5, 2, 3, 4, 6}.
 *   sf     E4M3 block scales, nvfp4_sf_bytes(rows, cols) bytes, swizzled:
 *          the [rows x cols/16] scale matrix padded to 128-row x 4-column
 *          tiles of 512 bytes, tiles of one 128-row band consecutive, and
 *          inside a tile byte (r, c) at (r%32)*16 + ((r%128)/32)*4 + c%4.
 *   scale  fp32 outer scales s_g: [rows] (per row) or [1] (per tensor).
 * Decoding: x^[r][j] = E2M1(code) * E4M3(sf block) * s_g.
 */
typedef struct nvfp4_tensor {
    uint8_t* codes;
    uint8_t* sf;
    float* scale;
    int64_t rows;
    int64_t cols;
} nvfp4_tensor;

/* Bytes of the swizzled block-scale buffer of a [rows x cols] matrix:
 * ceil(rows/128)*128 * ceil(cols/64)*4.  Pure host function. */
NVFP4_API size_t nvfp4_sf_bytes(int64_t rows, int64_t cols);

/* Workspace bytes nvfp4_quantize_rows needs: 0 for NVFP4_PER_ROW, 256 for
 * NVFP4_PER_TENSOR (the tensor amax is reduced there when amax_in is not
 * given), with or without a four-over-six flag.  Pure host function. */
NVFP4_API size_t nvfp4_quantize_workspace(int64_t rows, int64_t cols, int scale_mode);

/*
 * nvfp4_quantize_rows: quantize a bf16 matrix x [rows x cols] (row stride
 * ld elements) to NVFP4 into `out` (out->rows/cols must equal rows/cols).
 *
 * Per row ("miniTE Technical Report" 5.1, 5.6; "The 4-bitter Lesson"):
 *   amax = max_j |x_j| over the row (NVFP4_PER_ROW) or the whole matrix
 *          (NVFP4_PER_TENSOR); amax_in (nullable, device) replaces the
 *          reduction: [rows] values for per-row, [1] for per-tensor
 *          ("miniTE Technical Report" 5.3: the producer's amax is reused).
 *   s_g  = amax / 2688 (fp32); s_g == 0 -> the row is all-zero codes/scales.
 *   per 16-block: s_b = E4M3_rne_satfinite(bmax / (6 s_g)); s_b == 0 ->
 *          codes 0; else d = s_b s_g and v = x * (1/d) (v = x / d if d is
 *          an fp32 subnormal); code = E2M1_rne_saturating(v), sign kept.
 * Every step is an IEEE fp32 operation in that order, so the result is
 * bit-identical to any implementation of the same steps.
 * With NVFP4_FOUR_OVER_SIX_MSE / _MAE ("The 4-bitter Lesson", Four-Over-Six
 * for RL Weights and Activations; the pages name but do not print the E4M3
 * ceiling, read here as 256):
 *   s_g  = amax / 1536 (= 6 * 256, so a max -> 4 block scale, 3/2 of the
 *          max -> 6 one, stays within E4M3's 448); inv = 1536 / amax.
 *   per 16-block, for c = 6 and c = 4: s_b(c) = E4M3(bmax / (c s_g)) and
 *          codes as above with d = s_b(c) s_g; err(c) = sum over j = 0..15
 *          in order of (e2m1(q_j) s_b(c) - x_j inv)^2 (MSE) or |.| (MAE),
 *          each step one fp32 operation; max -> 4 is kept only when
 *          err(4) < err(6).
 *   The decode rule is unchanged, so the GEMMs take such tensors as they are.
 * Shapes: rows >= 0, 0 < cols <= 32768, cols % 16 == 0, ld >= cols.
 * Alignment: x and ld*2 bytes 16-byte aligned; codes 16-byte aligned.
 * Scale-factor padding columns inside the last 4-column group are written 0;
 * padding rows (beyond rows, up to the 128-row tile) are not written.
 * ws: nullable when nvfp4_quantize_workspace() is 0.  When ws_bytes >= 16
 * its first uint32 is the device error word; NVFP4_PER_TENSOR without
 * amax_in reduces the tensor amax at ws + 16.
 */
NVFP4_API int nvfp4_quantize_rows(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld,
                        int scale_mode, const float* amax_in, const nvfp4_tensor* out,
                        void* ws, size_t ws_bytes, void* stream);

/*
 * nvfp4_quantize_grouped: quantize `groups` bf16 matrices stacked row-wise,
 * x [groups * rows_per_group x cols] (contiguous, row stride cols), each
 * with its own per-tensor outer scale (scale_mode must contain
 * NVFP4_PER_TENSOR; four-over-six flags as in nvfp4_quantize_rows): the
 * per-expert weights of an MoE layer, requantized after every optimizer
 * step.  Bit-identical to nvfp4_quantize_rows(NVFP4_PER_TENSOR) on each
 * group, in three launches for all groups instead of three per group.
 * out: rows = groups * rows_per_group, cols = cols; out->scale has `groups`
 * entries; the swizzled block scales of group g start at byte g *
 * nvfp4_sf_bytes(rows_per_group, cols).
 * Shapes: 1 <= groups <= 65535, rows_per_group % 128 == 0, rows_per_group
 *         >= 128, 0 < cols <= 32768, cols % 16 == 0.
 * ws: >= 16 + 4 * groups bytes, 16-byte aligned (error word, then the
 * groups' amax accumulators).
 */
NVFP4_API int nvfp4_quantize_grouped(const void* x_bf16, int groups, int64_t rows_per_group, int64_t cols,
                                     int scale_mode, const nvfp4_tensor* out, void* ws, size_t ws_bytes,
                                     void* stream);

/*
 * nvfp4_dequantize_rows: y[r][j] = bf16(q[r][j] * s_b[r][j/16] * s_g) for an
 * NVFP4 matrix `in` [rows x cols] as nvfp4_quantize_rows writes it (swizzled
 * block scales), rounded once to nearest even from the exact product.  This
 * is DQ(Q(x)), the BF16 backward operand that keeps the forward pass's
 * quantization decisions (the pages' "Improving Gradient Stability":
 * dequantized backward for weights and activations; decode as "miniTE
 * Technical Report" 2.2).  s_g = in->scale[r] (NVFP4_PER_ROW) or
 * in->scale[0] (NVFP4_PER_TENSOR; with group offsets, in->scale[g] for the
 * rows of group g: the stacked per-expert weights of nvfp4_quantize_grouped);
 * four-over-six flags are ignored (the decode rule is the same).
 * group_offsets / padded_offsets (nullable, device, [groups + 1]): the block
 * scales of row r live at padded row padded_offsets[g] + (r -
 * group_offsets[g]) for the group g holding r, as in the expert-ordered
 * buffers of moe_expert_forward (a1, a2); NULL = scale row r.
 * y is bf16 [rows x cols], row stride ldy elements.  With NVFP4_DQ_PADDED_ROWS
 * (offsets required) y follows the padded layout as well: row r goes to the
 * padded row above, and the padding rows of every group (padded_offsets[g] +
 * count .. padded_offsets[g + 1]) are written with zeros, so y must hold
 * padded_offsets[groups] rows: the operand layout of the grouped BF16 GEMMs.
 * Shapes: rows >= 0, 0 < cols <= 32768, cols % 16 == 0, ldy >= cols,
 *         ldy % 8 == 0; 1 <= groups <= 256 when offsets are given.
 *         rows == 0 is a no-op (the buffers may then be null); with
 *         NVFP4_DQ_PADDED_ROWS it writes only the zero padding rows.
 * Alignment: codes 16-byte aligned, y 16-byte aligned, scale 4-byte aligned.
 */
NVFP4_API int nvfp4_dequantize_rows(const nvfp4_tensor* in, int scale_mode, const int* group_offsets,
                                    const int* padded_offsets, int groups, void* y_bf16, int64_t ldy,
                                    void* stream);

/*
 * Grouped BF16 GEMMs of the dequantized backward (the pages' "Improving
 * Gradient Stability": the backward of y = DQ(Q(x)) . DQ(Q(w))^T runs on the
 * BF16 dequantized operands x^ = DQ(Q(x)) and w^ = DQ(Q(w)) of the exact
 * tensors the forward pass used; "miniTE Technical Report" 4.2: BF16
 * backward GEMMs).  tcgen05 kind::f16 on the tensor cores, fp32
 * accumulation, bf16 results rounded once to nearest even.
 *
 * Rows are grouped by padded_offsets (device, [groups + 1], ascending
 * multiples of 128: the 128-row-padded expert layout of moe_expert_forward's
 * scale buffers, which nvfp4_dequantize_rows with NVFP4_DQ_PADDED_ROWS
 * writes; the padding rows must hold zeros), or, with padded_offsets NULL,
 * form one group of `rows` rows (any count: the dense linear).  Offsets that
 * are not ascending multiples of 128 within `rows` set NVFP4_DEVERR_BADGROUP
 * in the error word and nothing is written.
 *
 * nvfp4_grouped_dgrad_bf16: for each group g and each of its rows r,
 *   dx[r][k] = sum_n dy[r][n] * w[g][n][k]
 * dy bf16 [rows x nf], w bf16 [groups x nf x kf] (each expert's DQ(Q(W)) in
 * its forward layout [N x K], stacked), dx bf16 [rows x kf]; all row-major,
 * contiguous.  dx rows of the padding rows are written (zero, as dy's are).
 * nvfp4_grouped_wgrad_bf16: for each group g,
 *   dw[g][n][k] = sum over the rows r of g of dy[r][n] * x[r][k]
 * dy bf16 [rows x nf], x bf16 [rows x kf], dw bf16 [groups x nf x kf]; a
 * group with no rows gets a zero dw[g].
 * Shapes: rows >= 0; kf % 256 == 0; nf % 64 == 0 (dgrad) or nf % 256 == 0
 *         (wgrad); 1 <= groups <= 256 with offsets.
 * Alignment: every operand 16-byte aligned.
 * ws: nullable; when ws_bytes >= 4 its first uint32 is the device error word.
 */
NVFP4_API int nvfp4_grouped_dgrad_bf16(const void* dy_bf16, const void* w_bf16, void* dx_bf16, int64_t rows,
                                       int64_t nf, int64_t kf, const int* padded_offsets, int groups, void* ws,
                                       size_t ws_bytes, void* stream);
NVFP4_API int nvfp4_grouped_wgrad_bf16(const void* dy_bf16, const void* x_bf16, void* dw_bf16, int64_t rows,
                                       int64_t nf, int64_t kf, const int* padded_offsets, int groups, void* ws,
                                       size_t ws_bytes, void* stream);

/*
 * nvfp4_linear: y[m][n] = bf16( s_gx[m] * s_gw * sum_k (q_x s_bx)(q_w s_bw) )
 * for x [M x K] quantized per row and w [N x K] (K-major, i.e. the weight
 * transposed) quantized per tensor.  Accumulation is fp32 on the tensor
 * cores ("miniTE Technical Report" 5.4: ACC x alpha_a[m] x alpha_b; 5.2
 * dense path).  y is bf16 [M x N] with row stride ldy elements.
 * Shapes: K % 64 == 0, N % 256 == 0, M >= 0, ldy >= N, ldy % 8 == 0.
 * Alignment: codes and sf 16-byte aligned, y 16-byte aligned.
 * ws: nullable; when ws_bytes >= 4 its first uint32 is the device error word.
 */
NVFP4_API int nvfp4_linear(const nvfp4_tensor* x, const nvfp4_tensor* w, void* y_bf16, int64_t ldy,
                 void* ws, size_t ws_bytes, void* stream);

/* Options of moe_expert_forward. */
typedef struct moe_options {
    /* 0: router weight applied in the combine (default).  1: applied to
     * the SwiGLU output before the FC2 amax / quantization ("miniTE
     * Technical Report" 5.3 weighted SwiGLU; the combine then sums the
     * expert outputs unweighted). */
    int weight_at_fc1;
    /* 0, NVFP4_FOUR_OVER_SIX_MSE or NVFP4_FOUR_OVER_SIX_MAE: four-over-six
     * block scaling of the activations (X and the FC2 input D).  Weights
     * take it through their own nvfp4_quantize_rows call. */
    int four_over_six;
    /* Where the FC2 input D is requantized ("miniTE Technical Report" 5.6:
     * moving the quantization into the consumer GEMM so that the quantized
     * copy is never written).
     *   MOE_REQUANT_AUTO (0): the library's choice: MOE_REQUANT_SEPARATE.
     *   MOE_REQUANT_SEPARATE (1): a quantization launch between FC1 and FC2
     *     reads D back and writes its codes, block scales and row scales to
     *     the workspace; FC2 loads them.
     *   MOE_REQUANT_IN_FC2 (2): FC2 reads D and FC1's row amax and encodes
     *     each 128-row tile of A in shared memory (the same codes and scales,
     *     bit for bit), reusing it for all of the tile's output columns.  Only
     *     for plain NVFP4 activations (four_over_six 0), F a multiple of 256
     *     up to 768 and H of at least 512; other layers take the separate
     *     launch.  The workspace's requantized copies (a2_codes, a2_sf,
     *     a2_scale) are then written only on request (moe_debug.requant_copy). */
    int fc2_requant;
    /* 0: the router-weighted combine is its own launch after FC2 (default).
     * 1: FC2's epilogue does it: each 64-column block of a token's output is
     * summed, in slot order, by the unit that writes the last of the token's
     * k rows of that block (arrival counters in the workspace), reading the
     * other rows back from Y2.  Bit-identical to the separate combine (the
     * same fp32 fused multiply-adds in the same order); Y2 is still written.
     * Only with the separate requantization (fc2_requant other than
     * MOE_REQUANT_IN_FC2) and F up to 768; otherwise the separate combine. */
    int fc2_combine;
} moe_options;

#define MOE_REQUANT_AUTO 0
#define MOE_REQUANT_SEPARATE 1
#define MOE_REQUANT_IN_FC2 2

/* Optional debug outputs of moe_expert_forward (all nullable, device).
 * Zero-initialise the whole struct (moe_debug d = {0};) and set only the
 * fields wanted: every field's zero value means "off". */
typedef struct moe_debug {
    /* fp32 [R x 2F], R = T*topk rows in expert order: the FC1 output after
     * the alpha scaling, before SwiGLU (gate columns then up columns). */
    float* fc1_out;
    /* MOE_STAGE_EVENTS cudaEvent_t handles (created by the caller; a NULL
     * entry is skipped) recorded on `stream` before the first stage and after
     * each stage: quantize X
     * (with the router top-k, launched together), routing metadata +
     * permute, FC1, requant, FC2, combine.  With the requantization inside
     * FC2 the requant stage is empty (its two events are recorded back to
     * back) and the FC2 stage holds both. */
    void** stage_events;
    /* Nonzero: FC1's MMA-issuing thread first waits on a barrier that
     * nothing arrives at, so that its bounded wait runs out (a test of the
     * time-out path).  The kernel then sets NVFP4_DEVERR_TIMEOUT in the
     * workspace's error word, stops all its roles, frees its tensor memory
     * and returns; the layer's outputs are undefined, the context stays
     * usable.  Takes about 2 s.  0 for normal operation. */
    int stall_fc1;
    /* Nonzero: with the requantization inside FC2 (moe_options.fc2_requant),
     * FC2 also writes the codes, block scales and row scales it encodes to
     * the workspace's a2_codes / a2_sf / a2_scale, where the separate launch
     * leaves them.  0: they are not written. */
    int requant_copy;
} moe_debug;

#define MOE_STAGE_EVENTS 7

/*
 * Offsets (bytes from the workspace base) of the intermediates that
 * moe_expert_forward leaves in its workspace, for inspection after the
 * call completes.  R = T*topk token-expert rows, Rp = padded row bound.
 */
typedef struct moe_workspace_layout {
    size_t total;        /* workspace bytes required */
    size_t err;          /* uint32 device error word (+ scratch words) */
    size_t ids;          /* int32 [T x topk] routed expert ids, descending z */
    size_t weights;      /* fp32 [T x topk] router weights (softmax over the selected) */
    size_t row_weights;  /* fp32 [R] router weight of each expert-ordered row (weight_at_fc1 only) */
    size_t counts;       /* int32 [E] rows per expert */
    size_t offsets;      /* int32 [E+1] exclusive prefix of counts */
    size_t padded_offsets; /* int32 [E+1] prefix of ceil(count/128)*128 */
    size_t perm;         /* int32 [R] t*topk+slot of each expert-ordered row */
    size_t inv;          /* int32 [T x topk] expert-ordered row of (t, slot) */
    size_t chunk_counts; /* int32 scratch for the stable scatter */
    size_t xq_codes;     /* uint8 [T x H/2] per-token quantized X */
    size_t xq_sf;        /* row-linear [T x H/16] (the permute reads whole rows) */
    size_t xq_scale;     /* fp32 [T] */
    size_t a1_codes;     /* uint8 [R x H/2] X rows in expert order */
    size_t a1_sf;        /* swizzled, expert e's rows start at padded row padded_offsets[e] */
    size_t a1_scale;     /* fp32 [R] */
    size_t d;            /* bf16 [R x F] SwiGLU output */
    size_t amax2;        /* fp32 [R] row amax of d (from the FC1 epilogue) */
    size_t a2_codes;     /* uint8 [R x F/2] requantized d */
    size_t a2_sf;        /* swizzled [Rp x F/16], padded per expert like a1_sf */
    size_t a2_scale;     /* fp32 [R] */
    size_t y2;           /* bf16 [R x H] FC2 output in expert order */
    size_t comb_cnt;     /* int32 [T x H/64] arrival counters of the combine inside FC2 */
} moe_workspace_layout;

/* Fill *layout for the given sizes; returns 0, or NVFP4_ESHAPE /
 * NVFP4_EINVAL for sizes moe_expert_forward rejects.  Pure host function. */
NVFP4_API int moe_expert_workspace_layout(int64_t T, int64_t H, int64_t F, int E, int topk,
                                moe_workspace_layout* layout);

/* Workspace bytes moe_expert_forward needs (0 for rejected sizes). */
NVFP4_API size_t moe_expert_workspace(int64_t T, int64_t H, int64_t F, int E, int topk);

/*
 * moe_expert_forward: one MoE expert layer, W4A4 forward, all on device.
 *   x              bf16 [T x H] token activations (row stride H)
 *   router_logits  fp32 [T x E]; router_bias fp32 [E] (nullable = zeros)
 *   w1             E experts stacked: rows = E*2F, cols = H; expert e owns
 *                  rows [e*2F, (e+1)*2F) = gate (F rows) then up (F rows);
 *                  scale = fp32 [E], one per-tensor scale per expert
 *   w2             rows = E*H, cols = F; expert e owns rows [e*H, (e+1)*H);
 *                  scale = fp32 [E]
 *   out            bf16 [T x H]
 * Steps: z = logit + bias; top-k of z (ties to the lower expert), weights =
 * softmax over the k selected z; expert histogram, offsets and a stable
 * (expert, token) permutation built on the device; X quantized once per
 * token and its rows gathered into expert order; FC1 grouped block-scaled
 * GEMM with the SwiGLU + row-amax epilogue writing bf16 D; D requantized per
 * row with the reused amax; FC2 grouped GEMM writing bf16 Y2; out[t] =
 * bf16( sum_slot w[t,slot] * Y2[row(t,slot)] ) accumulated in fp32 in slot
 * order.  No host synchronization anywhere.
 * Shapes: T >= 1, H % 256 == 0, F % 128 == 0, 1 <= topk <= min(E, 16),
 *         E % 32 == 0, 32 <= E <= 256.
 * Alignment: every pointer 16-byte aligned; ws 256-byte aligned.
 * ws: moe_expert_workspace() bytes; its intermediates are described by
 * moe_expert_workspace_layout().  opt and dbg are nullable.
 */
NVFP4_API int moe_expert_forward(const void* x_bf16, int64_t T, int64_t H,
                       const float* router_logits, const float* router_bias, int E, int topk,
                       const nvfp4_tensor* w1, const nvfp4_tensor* w2, int64_t F,
                       const moe_options* opt, void* out_bf16, const moe_debug* dbg,
                       void* ws, size_t ws_bytes, void* stream);

/*
 * moe_expert_forward_noalloc: moe_expert_forward for callers that must not
 * allocate device memory -- for example a plugin that its host framework
 * hands only input and output buffers, or a latency-critical step in which
 * cudaMalloc / cudaFree would synchronize the device.  The pages describe no
 * such call; it is a deployment convenience of this library.
 *   Arguments, layouts and results are those of moe_expert_forward (no
 *   debug outputs).  The workspace is a fixed 32 MiB array in device global
 *   memory inside the library, which every GPU that loads the library holds
 *   until the process exits.  Sizes whose workspace
 *   (moe_expert_workspace()) exceeds 32 MiB are rejected with
 *   NVFP4_EWORKSPACE and a message; at hidden 2048, FFN 768, 128 experts,
 *   top-8 that is more than 516 tokens.
 *   The first call on each device looks the array's device address up
 *   (cudaGetSymbolAddress) with that device current, so make it before any
 *   stream capture.  Nothing is allocated, by this call or later ones.  The
 *   address is kept for the life of the process: do not use this entry
 *   point after cudaDeviceReset or any other teardown of the device's
 *   primary context.
 *   All calls on a device share the one array: calls whose work overlaps on
 *   the GPU (different streams without ordering) race and corrupt each
 *   other.  Each call clears the device error word at the start of the
 *   array; moe_noalloc_error_word() gives its address, so that the caller
 *   can read the call's device-side error bits in stream order.
 */
NVFP4_API int moe_expert_forward_noalloc(const void* x_bf16, int64_t T, int64_t H,
                                         const float* router_logits, const float* router_bias, int E,
                                         int topk, const nvfp4_tensor* w1, const nvfp4_tensor* w2,
                                         int64_t F, const moe_options* opt, void* out_bf16, void* stream);

/*
 * moe_noalloc_error_word: *out = the device address, on the current device,
 * of moe_expert_forward_noalloc's device error word (a uint32 at the start
 * of its built-in array; bits NVFP4_DEVERR_*).  Each no-alloc call clears it
 * before its kernels run; read it after the call in the call's stream order
 * (for example a 4-byte cudaMemcpyAsync on the same stream, then a
 * synchronize).  The address stays valid for the life of the process, with
 * the same caveat as the entry point (no use after a device reset).
 * Returns NVFP4_OK, NVFP4_EINVAL for a null out, NVFP4_ELAUNCH without a
 * usable current device.
 */
NVFP4_API int moe_noalloc_error_word(uint32_t** out);

/* Message describing the last error returned on the calling thread ("" if none). */
NVFP4_API const char* nvfp4_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4MOE_H */
