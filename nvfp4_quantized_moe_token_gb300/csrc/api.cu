// api.cu -- the C ABI (include/nvfp4moe.h): argument validation, workspace
// layout and the launch sequence of each call.  No allocation, no host
// synchronization, no device-to-host copy.
#include <stdarg.h>
#include <stdio.h>

#include <string>

#include "../../include/nvfp4moe.h"
#include "kernels.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int ok() {
    g_last_error.clear();
    return NVFP4_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int64_t sf_bytes_of(int64_t rows, int64_t cols) {
    return (rows + 127) / 128 * 128 * ((cols / 16 + 3) / 4 * 4);
}

int sm_count() {
    static int n = 0;
    if (n == 0) n = nvfp4::device_sm_count();
    return n;
}

int check_tensor(const nvfp4_tensor* t, const char* name) {
    if (t == nullptr || t->codes == nullptr || t->sf == nullptr || t->scale == nullptr)
        return fail(NVFP4_EINVAL, "%s: null tensor or buffer", name);
    if (!aligned(t->codes, 16) || !aligned(t->sf, 16) || !aligned(t->scale, 4))
        return fail(NVFP4_EALIGN, "%s: codes/sf must be 16-byte aligned, scale 4-byte aligned", name);
    if (t->rows < 0 || t->cols <= 0) return fail(NVFP4_EINVAL, "%s: bad size %lld x %lld", name,
                                                 (long long)t->rows, (long long)t->cols);
    return NVFP4_OK;
}

}  // namespace

namespace nvfp4 {
// Record a message for nvfp4_last_error() from another translation unit.
int set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace nvfp4

extern "C" {

const char* nvfp4_last_error(void) { return g_last_error.c_str(); }

size_t nvfp4_sf_bytes(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 0) return 0;
    return (size_t)sf_bytes_of(rows, cols);
}

size_t nvfp4_quantize_workspace(int64_t rows, int64_t cols, int scale_mode) {
    (void)rows;
    (void)cols;
    return (scale_mode & NVFP4_PER_TENSOR) ? 256 : 0;
}

namespace {
// four-over-six selector of the quantizer (0 off, 1 MSE, 2 MAE) from the flags
int fos_of(int flags) {
    return (flags & NVFP4_FOUR_OVER_SIX_MSE) ? 1 : ((flags & NVFP4_FOUR_OVER_SIX_MAE) ? 2 : 0);
}
bool fos_flags_valid(int flags) {
    return (flags & ~(NVFP4_FOUR_OVER_SIX_MSE | NVFP4_FOUR_OVER_SIX_MAE)) == 0 &&
           (flags & (NVFP4_FOUR_OVER_SIX_MSE | NVFP4_FOUR_OVER_SIX_MAE)) !=
               (NVFP4_FOUR_OVER_SIX_MSE | NVFP4_FOUR_OVER_SIX_MAE);
}
}  // namespace

int nvfp4_quantize_rows(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld, int scale_mode,
                        const float* amax_in, const nvfp4_tensor* out, void* ws, size_t ws_bytes,
                        void* stream) {
    if (x_bf16 == nullptr) return fail(NVFP4_EINVAL, "quantize: x is null");
    if (!fos_flags_valid(scale_mode & ~NVFP4_PER_TENSOR))
        return fail(NVFP4_EINVAL, "quantize: unknown scale_mode %d", scale_mode);
    const bool per_tensor = (scale_mode & NVFP4_PER_TENSOR) != 0;
    int rc = check_tensor(out, "quantize out");
    if (rc) return rc;
    if (rows < 0 || cols <= 0 || ld < cols) return fail(NVFP4_EINVAL, "quantize: bad rows/cols/ld");
    if (out->rows != rows || out->cols != cols) return fail(NVFP4_EINVAL, "quantize: out shape mismatch");
    if (cols % 16 != 0) return fail(NVFP4_ESHAPE, "quantize: cols %% 16 != 0 (cols = %lld)", (long long)cols);
    if (rows >= (1ll << 31) || cols > 32768) return fail(NVFP4_ESHAPE, "quantize: rows >= 2^31 or cols > 32768");
    if (!aligned(x_bf16, 16) || (ld % 8) != 0) return fail(NVFP4_EALIGN, "quantize: x and ld*2 must be 16-byte aligned");
    if (amax_in != nullptr && !aligned(amax_in, 4)) return fail(NVFP4_EALIGN, "quantize: amax_in misaligned");
    if (per_tensor && amax_in == nullptr && (ws == nullptr || ws_bytes < 256))
        return fail(NVFP4_EWORKSPACE, "quantize: per-tensor needs 256 bytes of ws");
    if (ws != nullptr && !aligned(ws, 16)) return fail(NVFP4_EALIGN, "quantize: ws must be 16-byte aligned");
    nvfp4::QuantLaunch q{};
    q.x = x_bf16;
    q.ld = ld;
    q.rows = rows;
    q.cols = cols;
    q.amax_in = amax_in;
    q.per_tensor = per_tensor;
    q.fos = fos_of(scale_mode);
    q.codes = out->codes;
    q.sf = out->sf;
    q.scale = out->scale;
    q.ws = ws;
    q.err = (ws != nullptr && ws_bytes >= 16) ? reinterpret_cast<uint32_t*>(ws) : nullptr;
    cudaError_t e = nvfp4::launch_quantize(q, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(NVFP4_ELAUNCH, "quantize: %s", cudaGetErrorString(e));
    return ok();
}

int nvfp4_quantize_grouped(const void* x_bf16, int groups, int64_t rows_per_group, int64_t cols, int scale_mode,
                           const nvfp4_tensor* out, void* ws, size_t ws_bytes, void* stream) {
    if (x_bf16 == nullptr) return fail(NVFP4_EINVAL, "quantize grouped: x is null");
    if (!(scale_mode & NVFP4_PER_TENSOR) || !fos_flags_valid(scale_mode & ~NVFP4_PER_TENSOR))
        return fail(NVFP4_EINVAL, "quantize grouped: scale_mode must be NVFP4_PER_TENSOR (| four-over-six)");
    int rc = check_tensor(out, "quantize grouped out");
    if (rc) return rc;
    if (groups < 1 || groups > 65535) return fail(NVFP4_ESHAPE, "quantize grouped: groups must be in [1, 65535]");
    if (rows_per_group < 128 || rows_per_group % 128 != 0)
        return fail(NVFP4_ESHAPE, "quantize grouped: rows_per_group must be a positive multiple of 128");
    if (cols <= 0 || cols % 16 != 0 || cols > 32768)
        return fail(NVFP4_ESHAPE, "quantize grouped: cols must be a multiple of 16 in (0, 32768]");
    const int64_t rows = (int64_t)groups * rows_per_group;
    if (rows >= (1ll << 31)) return fail(NVFP4_ESHAPE, "quantize grouped: too many rows");
    if (out->rows != rows || out->cols != cols) return fail(NVFP4_EINVAL, "quantize grouped: out shape mismatch");
    if (!aligned(x_bf16, 16)) return fail(NVFP4_EALIGN, "quantize grouped: x must be 16-byte aligned");
    if (ws == nullptr || !aligned(ws, 16) || ws_bytes < 16 + 4 * (size_t)groups)
        return fail(NVFP4_EWORKSPACE, "quantize grouped: ws must hold 16 + 4 * groups bytes, 16-byte aligned");
    nvfp4::QuantLaunch q{};
    q.x = x_bf16;
    q.ld = cols;
    q.rows = rows;
    q.cols = cols;
    q.per_tensor = 1;
    q.groups = groups;
    q.fos = fos_of(scale_mode);
    q.codes = out->codes;
    q.sf = out->sf;
    q.scale = out->scale;
    q.ws = ws;
    q.err = reinterpret_cast<uint32_t*>(ws);
    cudaError_t e = nvfp4::launch_quantize(q, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(NVFP4_ELAUNCH, "quantize grouped: %s", cudaGetErrorString(e));
    return ok();
}

int nvfp4_dequantize_rows(const nvfp4_tensor* in, int scale_mode, const int* group_offsets,
                          const int* padded_offsets, int groups, void* y_bf16, int64_t ldy, void* stream) {
    const bool padded_rows = (scale_mode & NVFP4_DQ_PADDED_ROWS) != 0;
    if (in != nullptr && in->rows == 0 && !padded_rows && in->cols > 0 && in->cols % 16 == 0)
        return ok();  // nothing to write
    // with no data rows the input buffers are never read (a padded layout then gets only its zero rows)
    int rc = (in != nullptr && in->rows == 0) ? NVFP4_OK : check_tensor(in, "dequantize in");
    if (rc) return rc;
    if (in == nullptr || in->cols <= 0) return fail(NVFP4_EINVAL, "dequantize: null input or bad cols");
    if (y_bf16 == nullptr) return fail(NVFP4_EINVAL, "dequantize: y is null");
    if (!fos_flags_valid(scale_mode & ~(NVFP4_PER_TENSOR | NVFP4_DQ_PADDED_ROWS)))
        return fail(NVFP4_EINVAL, "dequantize: unknown scale_mode %d", scale_mode);
    if (padded_rows && group_offsets == nullptr)
        return fail(NVFP4_EINVAL, "dequantize: NVFP4_DQ_PADDED_ROWS needs group and padded offsets");
    const int64_t rows = in->rows, cols = in->cols;
    if (cols % 16 != 0) return fail(NVFP4_ESHAPE, "dequantize: cols %% 16 != 0 (cols = %lld)", (long long)cols);
    if (rows >= (1ll << 31) || cols > 32768) return fail(NVFP4_ESHAPE, "dequantize: rows >= 2^31 or cols > 32768");
    if (ldy < cols || ldy % 8 != 0) return fail(NVFP4_EALIGN, "dequantize: ldy must be >= cols and a multiple of 8");
    if (!aligned(y_bf16, 16)) return fail(NVFP4_EALIGN, "dequantize: y must be 16-byte aligned");
    if ((group_offsets == nullptr) != (padded_offsets == nullptr))
        return fail(NVFP4_EINVAL, "dequantize: group_offsets and padded_offsets go together");
    if (group_offsets != nullptr && (groups < 1 || groups > 256))
        return fail(NVFP4_ESHAPE, "dequantize: groups must be in [1, 256]");
    nvfp4::DequantLaunch d{};
    d.codes = in->codes;
    d.sf = in->sf;
    d.scale = in->scale;
    d.rows = rows;
    d.cols = cols;
    d.per_tensor = (scale_mode & NVFP4_PER_TENSOR) != 0;
    d.goff = group_offsets;
    d.gpoff = padded_offsets;
    d.G = group_offsets != nullptr ? groups : 0;
    d.padded_rows = padded_rows ? 1 : 0;
    d.y = y_bf16;
    d.ldy = ldy;
    cudaError_t e = nvfp4::launch_dequantize(d, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(NVFP4_ELAUNCH, "dequantize: %s", cudaGetErrorString(e));
    return ok();
}

int nvfp4_linear(const nvfp4_tensor* x, const nvfp4_tensor* w, void* y_bf16, int64_t ldy, void* ws,
                 size_t ws_bytes, void* stream) {
    int rc = check_tensor(x, "linear x");
    if (rc) return rc;
    rc = check_tensor(w, "linear w");
    if (rc) return rc;
    if (y_bf16 == nullptr) return fail(NVFP4_EINVAL, "linear: y is null");
    const int64_t M = x->rows, K = x->cols, N = w->rows;
    if (w->cols != K) return fail(NVFP4_EINVAL, "linear: x cols %lld != w cols %lld", (long long)K, (long long)w->cols);
    if (K % 64 != 0) return fail(NVFP4_ESHAPE, "linear: K %% 64 != 0 (K = %lld)", (long long)K);
    if (N <= 0 || N % 256 != 0) return fail(NVFP4_ESHAPE, "linear: N %% 256 != 0 (N = %lld)", (long long)N);
    if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 24)) return fail(NVFP4_ESHAPE, "linear: too large");
    if (ldy < N || ldy % 8 != 0) return fail(NVFP4_EALIGN, "linear: ldy must be >= N and a multiple of 8");
    if (!aligned(y_bf16, 16)) return fail(NVFP4_EALIGN, "linear: y must be 16-byte aligned");
    if (ws != nullptr && ws_bytes >= 4 && !aligned(ws, 4)) return fail(NVFP4_EALIGN, "linear: ws misaligned");
    if (sm_count() <= 0) return fail(NVFP4_ELAUNCH, "linear: no CUDA device");
    nvfp4::GemmLaunch g{};
    g.a_codes = x->codes;
    g.a_sf = x->sf;
    g.a_scale = x->scale;
    g.M = M;
    g.b_codes = w->codes;
    g.b_sf = w->sf;
    g.b_scale = w->scale;
    g.N = (int)N;
    g.K = (int)K;
    g.G = 1;
    g.goff = nullptr;
    g.gpoff = nullptr;
    g.mode = 0;
    g.out = y_bf16;
    g.ldo = ldy;
    g.err = (ws != nullptr && ws_bytes >= 4) ? reinterpret_cast<uint32_t*>(ws) : nullptr;
    g.num_sms = sm_count();
    cudaError_t e = nvfp4::launch_gemm(g, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(NVFP4_ELAUNCH, "linear: %s", cudaGetErrorString(e));
    return ok();
}

namespace {
// Shared argument checks of the two grouped BF16 GEMMs.
int bwd_check(const char* name, const void* a, const void* b, const void* c, int64_t rows, int64_t nf, int64_t kf,
              const int* padded_offsets, int groups, void* ws, size_t ws_bytes, bool wgrad) {
    if (a == nullptr || b == nullptr || c == nullptr) return fail(NVFP4_EINVAL, "%s: null operand", name);
    if (rows < 0 || rows >= (1ll << 31)) return fail(NVFP4_ESHAPE, "%s: rows must be in [0, 2^31)", name);
    if (nf <= 0 || kf <= 0 || nf >= (1 << 24) || kf >= (1 << 24))
        return fail(NVFP4_ESHAPE, "%s: bad nf / kf", name);
    if (kf % 256 != 0) return fail(NVFP4_ESHAPE, "%s: kf %% 256 != 0 (kf = %lld)", name, (long long)kf);
    if (wgrad ? nf % 256 != 0 : nf % 64 != 0)
        return fail(NVFP4_ESHAPE, "%s: nf must be a multiple of %d (nf = %lld)", name, wgrad ? 256 : 64,
                    (long long)nf);
    if (padded_offsets != nullptr && (groups < 1 || groups > 256))
        return fail(NVFP4_ESHAPE, "%s: groups must be in [1, 256]", name);
    if (padded_offsets != nullptr && !aligned(padded_offsets, 4)) return fail(NVFP4_EALIGN, "%s: offsets misaligned", name);
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(c, 16))
        return fail(NVFP4_EALIGN, "%s: operands must be 16-byte aligned", name);
    if (ws != nullptr && ws_bytes >= 4 && !aligned(ws, 4)) return fail(NVFP4_EALIGN, "%s: ws misaligned", name);
    if (sm_count() <= 0) return fail(NVFP4_ELAUNCH, "%s: no CUDA device", name);
    return NVFP4_OK;
}
}  // namespace

int nvfp4_grouped_dgrad_bf16(const void* dy_bf16, const void* w_bf16, void* dx_bf16, int64_t rows, int64_t nf,
                             int64_t kf, const int* padded_offsets, int groups, void* ws, size_t ws_bytes,
                             void* stream) {
    int rc = bwd_check("dgrad", dy_bf16, w_bf16, dx_bf16, rows, nf, kf, padded_offsets, groups, ws, ws_bytes, false);
    if (rc) return rc;
    nvfp4::GemmBf16Launch g{};
    g.wgrad = 0;
    g.dy = dy_bf16;
    g.w = w_bf16;
    g.out = dx_bf16;
    g.rows = rows;
    g.nf = (int)nf;
    g.kf = (int)kf;
    g.gpoff = padded_offsets;
    g.G = padded_offsets ? groups : 1;
    g.err = (ws != nullptr && ws_bytes >= 4) ? reinterpret_cast<uint32_t*>(ws) : nullptr;
    g.num_sms = sm_count();
    cudaError_t e = nvfp4::launch_gemm_bf16(g, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(NVFP4_ELAUNCH, "dgrad: %s", cudaGetErrorString(e));
    return ok();
}

int nvfp4_grouped_wgrad_bf16(const void* dy_bf16, const void* x_bf16, void* dw_bf16, int64_t rows, int64_t nf,
                             int64_t kf, const int* padded_offsets, int groups, void* ws, size_t ws_bytes,
                             void* stream) {
    int rc = bwd_check("wgrad", dy_bf16, x_bf16, dw_bf16, rows, nf, kf, padded_offsets, groups, ws, ws_bytes, true);
    if (rc) return rc;
    nvfp4::GemmBf16Launch g{};
    g.wgrad = 1;
    g.dy = dy_bf16;
    g.x = x_bf16;
    g.out = dw_bf16;
    g.rows = rows;
    g.nf = (int)nf;
    g.kf = (int)kf;
    g.gpoff = padded_offsets;
    g.G = padded_offsets ? groups : 1;
    g.err = (ws != nullptr && ws_bytes >= 4) ? reinterpret_cast<uint32_t*>(ws) : nullptr;
    g.num_sms = sm_count();
    cudaError_t e = nvfp4::launch_gemm_bf16(g, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(NVFP4_ELAUNCH, "wgrad: %s", cudaGetErrorString(e));
    return ok();
}

static int moe_check_sizes(int64_t T, int64_t H, int64_t F, int E, int topk) {
    if (T < 1) return fail(NVFP4_EINVAL, "moe: T must be >= 1");
    if (H <= 0 || H % 256 != 0) return fail(NVFP4_ESHAPE, "moe: H %% 256 != 0 (H = %lld)", (long long)H);
    if (F <= 0 || F % 128 != 0) return fail(NVFP4_ESHAPE, "moe: F %% 128 != 0 (F = %lld)", (long long)F);
    if (E < 32 || E > 256 || E % 32 != 0) return fail(NVFP4_ESHAPE, "moe: E must be a multiple of 32 in [32, 256]");
    if (topk < 1 || topk > 16 || topk > E) return fail(NVFP4_ESHAPE, "moe: topk must be in [1, min(E, 16)]");
    if (T * topk >= (1ll << 30) || H >= (1 << 16) || F >= (1 << 16))
        return fail(NVFP4_ESHAPE, "moe: sizes too large");
    return NVFP4_OK;
}

int moe_expert_workspace_layout(int64_t T, int64_t H, int64_t F, int E, int topk, moe_workspace_layout* L) {
    if (L == nullptr) return fail(NVFP4_EINVAL, "moe layout: null");
    int rc = moe_check_sizes(T, H, F, E, topk);
    if (rc) return rc;
    const int64_t R = T * topk;
    const int64_t Rp = (R + 127 * (int64_t)E + 127) / 128 * 128;
    const int64_t nchunks = (T + nvfp4::kRouteChunk - 1) / nvfp4::kRouteChunk;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L->err = take(256);
    L->ids = take(4 * R);
    L->weights = take(4 * R);
    L->row_weights = take(4 * R);
    L->counts = take(4 * E);
    L->offsets = take(4 * (E + 1));
    L->padded_offsets = take(4 * (E + 1));
    L->perm = take(4 * R);
    L->inv = take(4 * R);
    L->chunk_counts = take(2 * 4 * nchunks * E);
    L->xq_codes = take(T * H / 2);
    L->xq_sf = take(sf_bytes_of(T, H));
    L->xq_scale = take(4 * T);
    L->a1_codes = take(R * H / 2);
    L->a1_sf = take(Rp * H / 16);
    L->a1_scale = take(4 * R);
    L->d = take(2 * R * F);
    L->amax2 = take(4 * R);
    L->a2_codes = take(R * F / 2);
    L->a2_sf = take(Rp * ((F / 16 + 3) / 4 * 4));
    L->a2_scale = take(4 * R);
    L->y2 = take(2 * R * H);
    L->comb_cnt = take(4 * T * (H / 64));
    L->total = o;
    return ok();
}

size_t moe_expert_workspace(int64_t T, int64_t H, int64_t F, int E, int topk) {
    moe_workspace_layout L;
    return moe_expert_workspace_layout(T, H, F, E, topk, &L) == NVFP4_OK ? L.total : 0;
}

int moe_expert_forward(const void* x_bf16, int64_t T, int64_t H, const float* router_logits,
                       const float* router_bias, int E, int topk, const nvfp4_tensor* w1,
                       const nvfp4_tensor* w2, int64_t F, const moe_options* opt, void* out_bf16,
                       const moe_debug* dbg, void* ws, size_t ws_bytes, void* stream) {
    moe_workspace_layout L;
    int rc = moe_expert_workspace_layout(T, H, F, E, topk, &L);
    if (rc) return rc;
    if (x_bf16 == nullptr || router_logits == nullptr || out_bf16 == nullptr || ws == nullptr)
        return fail(NVFP4_EINVAL, "moe: null x / logits / out / ws");
    rc = check_tensor(w1, "moe w1");
    if (rc) return rc;
    rc = check_tensor(w2, "moe w2");
    if (rc) return rc;
    if (w1->rows != (int64_t)E * 2 * F || w1->cols != H)
        return fail(NVFP4_EINVAL, "moe: w1 must be [E*2F x H]");
    if (w2->rows != (int64_t)E * H || w2->cols != F) return fail(NVFP4_EINVAL, "moe: w2 must be [E*H x F]");
    if (!aligned(x_bf16, 16) || !aligned(router_logits, 16) || !aligned(out_bf16, 16) ||
        (router_bias != nullptr && !aligned(router_bias, 4)))
        return fail(NVFP4_EALIGN, "moe: x, logits and out must be 16-byte aligned");
    if (!aligned(ws, 256)) return fail(NVFP4_EALIGN, "moe: ws must be 256-byte aligned");
    if (ws_bytes < L.total)
        return fail(NVFP4_EWORKSPACE, "moe: workspace %zu < required %zu bytes", ws_bytes, L.total);
    if (dbg != nullptr && dbg->fc1_out != nullptr && !aligned(dbg->fc1_out, 16))
        return fail(NVFP4_EALIGN, "moe: dbg->fc1_out must be 16-byte aligned");
    const int fos_flags = opt != nullptr ? opt->four_over_six : 0;
    if (!fos_flags_valid(fos_flags) || (fos_flags != 0 && fos_flags != NVFP4_FOUR_OVER_SIX_MSE &&
                                        fos_flags != NVFP4_FOUR_OVER_SIX_MAE))
        return fail(NVFP4_EINVAL, "moe: four_over_six must be 0, NVFP4_FOUR_OVER_SIX_MSE or _MAE");
    const int requant = opt != nullptr ? opt->fc2_requant : MOE_REQUANT_AUTO;
    if (requant < MOE_REQUANT_AUTO || requant > MOE_REQUANT_IN_FC2)
        return fail(NVFP4_EINVAL, "moe: fc2_requant must be MOE_REQUANT_AUTO, _SEPARATE or _IN_FC2");
    const int comb_opt = opt != nullptr ? opt->fc2_combine : 0;
    if (comb_opt != 0 && comb_opt != 1) return fail(NVFP4_EINVAL, "moe: fc2_combine must be 0 or 1");
    if (sm_count() <= 0) return fail(NVFP4_ELAUNCH, "moe: no CUDA device");
    const bool at_fc1 = opt != nullptr && opt->weight_at_fc1 != 0;
    const int fos = fos_of(fos_flags);
    uint8_t* base = reinterpret_cast<uint8_t*>(ws);
    auto at = [&](size_t off) { return base + off; };
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t R = T * topk;
    cudaError_t e;
    void** ev = dbg ? dbg->stage_events : nullptr;
    int ev_i = 0;
    auto mark = [&]() -> cudaError_t {
        if (ev == nullptr) return cudaSuccess;
        void* e = ev[ev_i++];
        return e == nullptr ? cudaSuccess : cudaEventRecord(reinterpret_cast<cudaEvent_t>(e), s);
    };
    if ((e = mark()) != cudaSuccess) return fail(NVFP4_ELAUNCH, "moe event: %s", cudaGetErrorString(e));

    // 1. per-token quantization of X (once per token; the permute moves the
    //    result, scales row-linear here and swizzled in the permuted copy),
    //    in the same launch as the router top-k: the two are independent
    nvfp4::QuantLaunch qx{};
    qx.x = x_bf16;
    qx.ld = H;
    qx.rows = T;
    qx.cols = H;
    qx.codes = at(L.xq_codes);
    qx.sf = at(L.xq_sf);
    qx.sf_ld = H / 16;  // row-linear: the permute gathers whole rows of scales
    qx.fos = fos;
    qx.x_once = 1;  // X leaves L2 first: its codes stay there for the permute's 8 reads of each row
    qx.scale = reinterpret_cast<float*>(at(L.xq_scale));
    qx.err = reinterpret_cast<uint32_t*>(at(L.err));

    // 2. routing, metadata and permute
    nvfp4::RouteLaunch r{};
    r.logits = router_logits;
    r.bias = router_bias;
    r.T = T;
    r.E = E;
    r.k = topk;
    r.ids = reinterpret_cast<int*>(at(L.ids));
    r.w = reinterpret_cast<float*>(at(L.weights));
    const int64_t nchunks = (T + nvfp4::kRouteChunk - 1) / nvfp4::kRouteChunk;
    r.chunk_cnt = reinterpret_cast<int*>(at(L.chunk_counts));
    r.chunk_base = r.chunk_cnt + nchunks * E;
    r.cnt = reinterpret_cast<int*>(at(L.counts));
    r.off = reinterpret_cast<int*>(at(L.offsets));
    r.poff = reinterpret_cast<int*>(at(L.padded_offsets));
    r.done = reinterpret_cast<unsigned int*>(at(L.err) + 4);
    r.perm = reinterpret_cast<int*>(at(L.perm));
    r.inv = reinterpret_cast<int*>(at(L.inv));
    r.err = reinterpret_cast<uint32_t*>(at(L.err));
    r.xq_codes = at(L.xq_codes);
    r.xq_sf = at(L.xq_sf);
    r.xq_scale = reinterpret_cast<const float*>(at(L.xq_scale));
    r.H = H;
    r.a1_codes = at(L.a1_codes);
    r.a1_sf = at(L.a1_sf);
    r.a1_scale = reinterpret_cast<float*>(at(L.a1_scale));
    r.amax2 = reinterpret_cast<float*>(at(L.amax2));
    r.row_w = at_fc1 ? reinterpret_cast<float*>(at(L.row_weights)) : nullptr;
    // the requantization inside FC2 (plain NVFP4, F a multiple of 256 up to 768,
    // H >= 512) and the combine inside FC2's epilogue (FC2 on its 4-stage plain
    // form, F < 1024, with the separate requantization); the scatter zeroes the
    // combine's arrival counters
    const bool in_fc2 = requant == MOE_REQUANT_IN_FC2 && fos == 0 && F % 256 == 0 && F <= 768 && H >= 512;
    const bool comb_in_fc2 = comb_opt == 1 && !in_fc2 && F < 1024;
    r.comb_cnt = comb_in_fc2 ? reinterpret_cast<int*>(at(L.comb_cnt)) : nullptr;
    r.comb_blocks = (int)(H / 64);

    if ((e = nvfp4::launch_quantize_topk(qx, r, s)) != cudaSuccess)
        return fail(NVFP4_ELAUNCH, "moe quantize + top-k: %s", cudaGetErrorString(e));
    if ((e = mark()) != cudaSuccess) return fail(NVFP4_ELAUNCH, "moe event: %s", cudaGetErrorString(e));
    if ((e = nvfp4::launch_route_rest(r, s)) != cudaSuccess) return fail(NVFP4_ELAUNCH, "moe route: %s", cudaGetErrorString(e));
    if ((e = mark()) != cudaSuccess) return fail(NVFP4_ELAUNCH, "moe event: %s", cudaGetErrorString(e));

    // 3. FC1 grouped GEMM, SwiGLU + row-amax epilogue
    nvfp4::GemmLaunch g1{};
    g1.a_codes = at(L.a1_codes);
    g1.a_sf = at(L.a1_sf);
    g1.a_scale = reinterpret_cast<const float*>(at(L.a1_scale));
    g1.M = R;
    g1.b_codes = w1->codes;
    g1.b_sf = w1->sf;
    g1.b_scale = w1->scale;
    g1.N = (int)(2 * F);
    g1.K = (int)H;
    g1.G = E;
    g1.goff = r.off;
    g1.gpoff = r.poff;
    g1.mode = 1;
    g1.out = at(L.d);
    g1.ldo = F;
    g1.amax_out = reinterpret_cast<float*>(at(L.amax2));
    g1.row_prob = r.row_w;
    g1.c_debug = dbg ? dbg->fc1_out : nullptr;
    g1.stall = dbg ? dbg->stall_fc1 : 0;
    g1.err = r.err;
    g1.num_sms = sm_count();
    if ((e = nvfp4::launch_gemm(g1, s)) != cudaSuccess) return fail(NVFP4_ELAUNCH, "moe fc1: %s", cudaGetErrorString(e));
    if ((e = mark()) != cudaSuccess) return fail(NVFP4_ELAUNCH, "moe event: %s", cudaGetErrorString(e));

    // 4. requantize D per row, reusing the epilogue's amax: a separate launch,
    //    or inside FC2 (in_fc2, decided above)
    nvfp4::QuantLaunch q2{};
    q2.x = at(L.d);
    q2.ld = F;
    q2.rows = R;
    q2.cols = F;
    q2.amax_in = reinterpret_cast<const float*>(at(L.amax2));
    q2.codes = at(L.a2_codes);
    q2.sf = at(L.a2_sf);
    q2.scale = reinterpret_cast<float*>(at(L.a2_scale));
    q2.goff = r.off;
    q2.gpoff = r.poff;
    q2.G = E;
    q2.reverse = 1;  // FC1's last rows are still in L2; FC2 then starts on the rows written last
    q2.fos = fos;
    q2.err = reinterpret_cast<uint32_t*>(at(L.err));
    if (!in_fc2 && (e = nvfp4::launch_quantize(q2, s)) != cudaSuccess)
        return fail(NVFP4_ELAUNCH, "moe requant: %s", cudaGetErrorString(e));
    if ((e = mark()) != cudaSuccess) return fail(NVFP4_ELAUNCH, "moe event: %s", cudaGetErrorString(e));

    // 5. FC2 grouped GEMM -> bf16 Y2
    nvfp4::GemmLaunch g2{};
    g2.a_codes = at(L.a2_codes);
    g2.a_sf = at(L.a2_sf);
    g2.a_scale = reinterpret_cast<const float*>(at(L.a2_scale));
    g2.M = R;
    g2.b_codes = w2->codes;
    g2.b_sf = w2->sf;
    g2.b_scale = w2->scale;
    g2.N = (int)H;
    g2.K = (int)F;
    g2.G = E;
    g2.goff = r.off;
    g2.gpoff = r.poff;
    g2.mode = in_fc2 ? 3 : (comb_in_fc2 ? 4 : 0);
    if (comb_in_fc2) {
        g2.perm = r.perm;
        g2.inv = r.inv;
        g2.cw = at_fc1 ? nullptr : r.w;
        g2.cout = out_bf16;
        g2.ccnt = r.comb_cnt;
        g2.k_top = topk;
    }
    if (in_fc2) {
        g2.d_in = at(L.d);
        g2.d_amax = reinterpret_cast<const float*>(at(L.amax2));
        if (dbg != nullptr && dbg->requant_copy) {  // copies of the encoded A, where the separate launch writes them
            g2.q_codes = at(L.a2_codes);
            g2.q_sf = at(L.a2_sf);
            g2.q_scale = reinterpret_cast<float*>(at(L.a2_scale));
        }
    }
    g2.out = at(L.y2);
    g2.ldo = H;
    g2.err = r.err;
    g2.num_sms = sm_count();
    if ((e = nvfp4::launch_gemm(g2, s)) != cudaSuccess) return fail(NVFP4_ELAUNCH, "moe fc2: %s", cudaGetErrorString(e));
    if ((e = mark()) != cudaSuccess) return fail(NVFP4_ELAUNCH, "moe event: %s", cudaGetErrorString(e));

    // 6. router-weighted combine
    nvfp4::CombineLaunch c{};
    c.y = at(L.y2);
    c.inv = r.inv;
    c.w = at_fc1 ? nullptr : r.w;
    c.T = T;
    c.H = H;
    c.k = topk;
    c.out = out_bf16;
    if (!comb_in_fc2 && (e = nvfp4::launch_combine(c, s)) != cudaSuccess)
        return fail(NVFP4_ELAUNCH, "moe combine: %s", cudaGetErrorString(e));
    if ((e = mark()) != cudaSuccess) return fail(NVFP4_ELAUNCH, "moe event: %s", cudaGetErrorString(e));
    return ok();
}

}  // extern "C"
