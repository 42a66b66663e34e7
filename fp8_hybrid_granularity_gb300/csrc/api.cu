// C-ABI entry points (declared in include/fp8hg.h): argument validation, then
// one launch each.  Nothing here allocates device memory or synchronizes,
// except fp8hg_get_device_error.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/fp8hg.h"
#include "internal.h"

namespace {

inline bool aligned(const void *p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline int status_from_cuda(cudaError_t e) { return e == cudaSuccess ? FP8HG_OK : FP8HG_ERR_CUDA; }

inline bool valid_fmt(int f) { return f == FP8HG_E4M3 || f == FP8HG_E5M2; }

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s

int validate_operand(const fp8hg_operand *o) {
    if (!o || !o->codes || !o->scale) return FP8HG_ERR_INVALID_ARG;
    if (!valid_fmt(o->fmt)) return FP8HG_ERR_INVALID_ARG;
    if (o->gran < FP8HG_GRAN_ROW || o->gran > FP8HG_GRAN_MX32) return FP8HG_ERR_INVALID_ARG;
    if (o->rows <= 0 || o->k <= 0) return FP8HG_ERR_SHAPE;
    if (o->rows % 128 || o->k % 128) return FP8HG_ERR_SHAPE;
    if (o->rows > (int64_t(1) << 30) || o->k > (int64_t(1) << 30)) return FP8HG_ERR_SHAPE;
    if (o->ld < o->k || o->ld % 16) return FP8HG_ERR_ALIGNMENT;
    if (!aligned(o->codes, 16)) return FP8HG_ERR_ALIGNMENT;
    int64_t scale_cols = 1;
    switch (o->gran) {
    case FP8HG_GRAN_ROW: scale_cols = 1; break;
    case FP8HG_GRAN_1x128:
    case FP8HG_GRAN_128x128: scale_cols = o->k / 128; break;
    default: scale_cols = o->k / 32; break;
    }
    if (o->gran == FP8HG_GRAN_ROW) {
        if (o->ld_scale < 1) return FP8HG_ERR_INVALID_ARG;
    } else {
        const int64_t padded = (scale_cols + 3) / 4 * 4;
        if (o->ld_scale < padded || o->ld_scale % 4) return FP8HG_ERR_ALIGNMENT;
        if (!aligned(o->scale, 4)) return FP8HG_ERR_ALIGNMENT;
    }
    return FP8HG_OK;
}

bool gran_pair_ok(int op, int ga, int gb) {
    if (ga == FP8HG_GRAN_MX32 && gb == FP8HG_GRAN_MX32) return true;
    if (ga == FP8HG_GRAN_MX32 || gb == FP8HG_GRAN_MX32) return false;
    switch (op) {
    case FP8HG_FPROP:
    case FP8HG_DGRAD:
        return (ga == FP8HG_GRAN_ROW || ga == FP8HG_GRAN_1x128) && gb == FP8HG_GRAN_128x128;
    case FP8HG_WGRAD: return ga == FP8HG_GRAN_1x128 && gb == FP8HG_GRAN_1x128;
    default: return false;
    }
}

int check_quant_common(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                       const uint8_t *q, int64_t ld_q, const uint8_t *s) {
    if (!valid_fmt(fmt)) return FP8HG_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0) return FP8HG_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return FP8HG_OK;  // nothing is read or written
    if (!x || !q || !s) return FP8HG_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(q, 16)) return FP8HG_ERR_ALIGNMENT;
    if (ld_x % 8 || ld_q % 16) return FP8HG_ERR_ALIGNMENT;
    return FP8HG_OK;
}

// fp8hg_wait_opts -> WaitOpts (NULL = defaults).
int wait_opts(const fp8hg_wait_opts *opts, fp8hg::WaitOpts &w) {
    w = fp8hg::WaitOpts{};
    if (!opts) return FP8HG_OK;
    if (opts->inject_fault < 0 || opts->inject_fault > 1 || opts->reserved != 0)
        return FP8HG_ERR_INVALID_ARG;
    w.limit_ns = opts->wait_limit_ns;
    w.inject = opts->inject_fault;
    return FP8HG_OK;
}

}  // namespace

namespace {

// Checks shared by the GEMM entry points and the common part of GemmArgs.
int prepare_gemm(int op, const fp8hg_operand *a, const fp8hg_operand *b, fp8hg::GemmArgs &g) {
    if (op < FP8HG_FPROP || op > FP8HG_WGRAD) return FP8HG_ERR_INVALID_ARG;
    int st = validate_operand(a);
    if (st != FP8HG_OK) return st;
    st = validate_operand(b);
    if (st != FP8HG_OK) return st;
    if (a->k != b->k) return FP8HG_ERR_SHAPE;
    if (!gran_pair_ok(op, a->gran, b->gran)) return FP8HG_ERR_UNSUPPORTED;
    g = fp8hg::GemmArgs{};
    g.a_codes = a->codes;
    g.b_codes = b->codes;
    g.a_scale = a->scale;
    g.b_scale = b->scale;
    g.M = a->rows;
    g.N = b->rows;
    g.K = a->k;
    g.lda = a->ld;
    g.ldb = b->ld;
    g.ld_sa = a->ld_scale;
    g.ld_sb = b->ld_scale;
    g.fmt_a = a->fmt;
    g.fmt_b = b->fmt;
    g.gran_a = a->gran;
    g.gran_b = b->gran;
    return FP8HG_OK;
}

int run_gemm(fp8hg::GemmArgs &g, const fp8hg_gemm_opts *opts, void *stream) {
    unsigned int *err = fp8hg::device_error_word();
    if (!err) return FP8HG_ERR_CUDA;
    g.wait_limit_ns = (opts && opts->wait_limit_ns) ? opts->wait_limit_ns : kDefaultWaitNs;
    g.inject_fault = opts ? opts->inject_fault : 0;
    g.tile = opts ? opts->tile : 0;
    g.err = err;
    const int rc = fp8hg::launch_gemm_scaled(g, static_cast<cudaStream_t>(stream));
    if (rc == 1) return FP8HG_ERR_UNSUPPORTED;  // tensor map could not be encoded
    return rc == 0 ? FP8HG_OK : FP8HG_ERR_CUDA;
}

}  // namespace

extern "C" {

int fp8_quant_token_ex(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int group,
                       int transpose, int fmt, uint8_t *q, int64_t ld_q, uint8_t *scale,
                       int64_t ld_s, const fp8hg_wait_opts *opts, void *stream) {
    fp8hg::WaitOpts w;
    int st = wait_opts(opts, w);
    if (st != FP8HG_OK) return st;
    st = check_quant_common(x, rows, cols, ld_x, fmt, q, ld_q, scale);
    if (st != FP8HG_OK) return st;
    if (group != 0 && group != 128) return FP8HG_ERR_INVALID_ARG;
    if (transpose != 0 && transpose != 1) return FP8HG_ERR_INVALID_ARG;
    if (transpose && group != 128) return FP8HG_ERR_UNSUPPORTED;
    if (rows == 0 || cols == 0) return FP8HG_OK;
    if (transpose) {
        if (rows % 128 || cols % 64) return FP8HG_ERR_SHAPE;
        if (rows / 128 > 65535) return FP8HG_ERR_SHAPE;
        if (ld_x < cols || ld_q < rows || ld_s < rows / 128) return FP8HG_ERR_INVALID_ARG;
    } else {
        if (cols % 128) return FP8HG_ERR_SHAPE;
        if (ld_x < cols || ld_q < cols) return FP8HG_ERR_INVALID_ARG;
        if (ld_s < (group ? cols / 128 : 1)) return FP8HG_ERR_INVALID_ARG;
        if (group == 0 && rows > 2147483647LL) return FP8HG_ERR_SHAPE;
    }
    if (w.inject && !fp8hg::quant_token_waits(cols, group, transpose)) return FP8HG_ERR_UNSUPPORTED;
    return status_from_cuda(fp8hg::launch_quant_token(x, rows, cols, ld_x, group, transpose, fmt, q,
                                                      ld_q, scale, ld_s, w,
                                                      static_cast<cudaStream_t>(stream)));
}

int fp8_quant_token(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int group,
                    int transpose, int fmt, uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s,
                    void *stream) {
    return fp8_quant_token_ex(x, rows, cols, ld_x, group, transpose, fmt, q, ld_q, scale, ld_s,
                              nullptr, stream);
}

size_t fp8_quant_token_dual_workspace(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return fp8hg::dual_workspace_bytes(rows, cols);
}

int fp8_quant_token_dual(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                         uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s, int fmt_t,
                         uint8_t *q_t, int64_t ld_qt, uint8_t *scale_t, int64_t ld_st,
                         void *workspace, size_t workspace_bytes, const fp8hg_wait_opts *opts,
                         void *stream) {
    fp8hg::WaitOpts w;
    int st = wait_opts(opts, w);
    if (st != FP8HG_OK) return st;
    st = check_quant_common(x, rows, cols, ld_x, fmt, q, ld_q, scale);
    if (st != FP8HG_OK) return st;
    if (!valid_fmt(fmt_t)) return FP8HG_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return FP8HG_OK;
    if (!q_t || !scale_t || !workspace) return FP8HG_ERR_INVALID_ARG;
    if (!aligned(q_t, 16) || ld_qt % 16 || !aligned(workspace, 16)) return FP8HG_ERR_ALIGNMENT;
    if (rows % 128 || cols % 128) return FP8HG_ERR_SHAPE;
    if (rows > (int64_t(1) << 31) || cols > (int64_t(1) << 31)) return FP8HG_ERR_SHAPE;
    if (ld_x < cols || ld_q < cols || ld_s < 1 || ld_qt < rows || ld_st < rows / 128)
        return FP8HG_ERR_INVALID_ARG;
    if (workspace_bytes < fp8hg::dual_workspace_bytes(rows, cols)) return FP8HG_ERR_INVALID_ARG;
    return status_from_cuda(fp8hg::launch_quant_dual(
        x, rows, cols, ld_x, fmt, q, ld_q, scale, ld_s, fmt_t, q_t, ld_qt, scale_t, ld_st,
        static_cast<unsigned int *>(workspace), w, static_cast<cudaStream_t>(stream)));
}

int fp8_quant_token_dual_noalloc(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                                 int fmt, uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s,
                                 int fmt_t, uint8_t *q_t, int64_t ld_qt, uint8_t *scale_t,
                                 int64_t ld_st, const fp8hg_wait_opts *opts, void *stream) {
    fp8hg::WaitOpts w;
    int st = wait_opts(opts, w);
    if (st != FP8HG_OK) return st;
    st = check_quant_common(x, rows, cols, ld_x, fmt, q, ld_q, scale);
    if (st != FP8HG_OK) return st;
    if (!valid_fmt(fmt_t)) return FP8HG_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return FP8HG_OK;
    if (!q_t || !scale_t) return FP8HG_ERR_INVALID_ARG;
    if (!aligned(q_t, 16) || ld_qt % 16) return FP8HG_ERR_ALIGNMENT;
    if (rows % 128 || cols % 128) return FP8HG_ERR_SHAPE;
    if (rows > fp8hg::noalloc_dual_max_rows()) return FP8HG_ERR_SHAPE;   // beyond the fixed scratch
    if (cols > (int64_t(1) << 31)) return FP8HG_ERR_SHAPE;
    if (ld_x < cols || ld_q < cols || ld_s < 1 || ld_qt < rows || ld_st < rows / 128)
        return FP8HG_ERR_INVALID_ARG;
    unsigned int *ws = fp8hg::noalloc_dual_workspace();
    if (!ws) return FP8HG_ERR_CUDA;
    return status_from_cuda(fp8hg::launch_quant_dual(x, rows, cols, ld_x, fmt, q, ld_q, scale, ld_s,
                                                     fmt_t, q_t, ld_qt, scale_t, ld_st, ws, w,
                                                     static_cast<cudaStream_t>(stream)));
}

int fp8_quant_block128(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                       uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s, uint8_t *q_t,
                       int64_t ld_qt, uint8_t *scale_t, int64_t ld_st, void *stream) {
    int st = check_quant_common(x, rows, cols, ld_x, fmt, q, ld_q, scale);
    if (st != FP8HG_OK) return st;
    if (rows == 0 || cols == 0) return FP8HG_OK;
    if ((q_t == nullptr) != (scale_t == nullptr)) return FP8HG_ERR_INVALID_ARG;
    if (rows % 128 || cols % 128) return FP8HG_ERR_SHAPE;
    if (rows / 128 > 65535) return FP8HG_ERR_SHAPE;
    if (ld_x < cols || ld_q < cols || ld_s < cols / 128) return FP8HG_ERR_INVALID_ARG;
    if (q_t) {
        if (!aligned(q_t, 16) || ld_qt % 16) return FP8HG_ERR_ALIGNMENT;
        if (ld_qt < rows || ld_st < rows / 128) return FP8HG_ERR_INVALID_ARG;
    }
    return status_from_cuda(fp8hg::launch_quant_block128(x, rows, cols, ld_x, fmt, q, ld_q, scale,
                                                         ld_s, q_t, ld_qt, scale_t, ld_st,
                                                         static_cast<cudaStream_t>(stream)));
}

int fp8_quant_block128_batch(const fp8hg_block128_job *jobs, int n, int fmt, void *stream) {
    if (n < 0 || n > FP8HG_BATCH_MAX) return FP8HG_ERR_INVALID_ARG;
    if (n == 0) return FP8HG_OK;
    if (!jobs) return FP8HG_ERR_INVALID_ARG;
    static_assert(FP8HG_BATCH_MAX <= fp8hg::kBlock128BatchMax, "batch table too small");
    fp8hg::Block128Batch b{};
    int64_t blocks = 0;
    int trans = -1;
    for (int i = 0; i < n; ++i) {
        const fp8hg_block128_job &j = jobs[i];
        int st = check_quant_common(j.x, j.rows, j.cols, j.ld_x, fmt, j.q, j.ld_q, j.scale);
        if (st != FP8HG_OK) return st;
        if (j.rows == 0 || j.cols == 0) continue;   // nothing read or written
        if ((j.q_t == nullptr) != (j.scale_t == nullptr)) return FP8HG_ERR_INVALID_ARG;
        const int t = j.q_t != nullptr;
        if (trans >= 0 && t != trans) return FP8HG_ERR_INVALID_ARG;
        trans = t;
        if (j.rows % 128 || j.cols % 128) return FP8HG_ERR_SHAPE;
        if (j.ld_x < j.cols || j.ld_q < j.cols || j.ld_s < j.cols / 128) return FP8HG_ERR_INVALID_ARG;
        if (t) {
            if (!aligned(j.q_t, 16) || j.ld_qt % 16) return FP8HG_ERR_ALIGNMENT;
            if (j.ld_qt < j.rows || j.ld_st < j.rows / 128) return FP8HG_ERR_INVALID_ARG;
        }
        fp8hg::Block128Job &k = b.job[b.n++];
        k = {j.x, j.ld_x, j.q, j.ld_q, j.scale, j.ld_s, j.q_t, j.ld_qt, j.scale_t, j.ld_st,
             j.cols / 128, blocks};
        blocks += (j.rows / 128) * (j.cols / 128);
        if (blocks > 0x7FFFFFFF) return FP8HG_ERR_SHAPE;
    }
    return status_from_cuda(fp8hg::launch_quant_block128_batch(b, blocks, fmt, trans == 1,
                                                               static_cast<cudaStream_t>(stream)));
}

int fp8_quant_mx32(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt, uint8_t *q,
                   int64_t ld_q, uint8_t *scale, int64_t ld_s, unsigned long long *clamp_count,
                   void *stream) {
    int st = check_quant_common(x, rows, cols, ld_x, fmt, q, ld_q, scale);
    if (st != FP8HG_OK) return st;
    if (rows == 0 || cols == 0) return FP8HG_OK;
    if (cols % 32) return FP8HG_ERR_SHAPE;
    if (ld_x < cols || ld_q < cols || ld_s < cols / 32) return FP8HG_ERR_INVALID_ARG;
    if (clamp_count && !aligned(clamp_count, 8)) return FP8HG_ERR_ALIGNMENT;
    return status_from_cuda(fp8hg::launch_quant_mx32(x, rows, cols, ld_x, fmt, q, ld_q, scale, ld_s,
                                                     clamp_count,
                                                     static_cast<cudaStream_t>(stream)));
}

int fp8_quant_mx32_monitor(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                           uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s,
                           fp8hg_mx_stats *stats, unsigned int *row_saturated, void *stream) {
    int st = check_quant_common(x, rows, cols, ld_x, fmt, q, ld_q, scale);
    if (st != FP8HG_OK) return st;
    if (stats == nullptr) return FP8HG_ERR_INVALID_ARG;
    if (!aligned(stats, 8) || (row_saturated && !aligned(row_saturated, 4)))
        return FP8HG_ERR_ALIGNMENT;
    if (rows == 0 || cols == 0) return FP8HG_OK;
    if (cols % 32) return FP8HG_ERR_SHAPE;
    if (ld_x < cols || ld_q < cols || ld_s < cols / 32) return FP8HG_ERR_INVALID_ARG;
    return status_from_cuda(fp8hg::launch_quant_mx32_monitor(
        x, rows, cols, ld_x, fmt, q, ld_q, scale, ld_s,
        reinterpret_cast<unsigned long long *>(stats), row_saturated,
        static_cast<cudaStream_t>(stream)));
}

int fp8_requant_t_ex(const uint8_t *q, int64_t rows, int64_t cols, int64_t ld_q,
                     const uint8_t *scale, int64_t ld_s, int gran, int fmt_in, int fmt_out,
                     uint8_t *q_t, int64_t ld_qt, uint8_t *scale_t, int64_t ld_st,
                     const fp8hg_wait_opts *opts, void *stream) {
    fp8hg::WaitOpts w;
    const int wst = wait_opts(opts, w);
    if (wst != FP8HG_OK) return wst;
    if (!valid_fmt(fmt_in) || !valid_fmt(fmt_out)) return FP8HG_ERR_INVALID_ARG;
    if (gran != FP8HG_GRAN_ROW && gran != FP8HG_GRAN_1x128) return FP8HG_ERR_UNSUPPORTED;
    if (rows < 0 || cols < 0) return FP8HG_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return FP8HG_OK;
    if (!q || !scale || !q_t || !scale_t) return FP8HG_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(q_t, 16) || ld_q % 16 || ld_qt % 16) return FP8HG_ERR_ALIGNMENT;
    if (rows % 128 || cols % 128) return FP8HG_ERR_SHAPE;
    if (rows / 128 > 65535) return FP8HG_ERR_SHAPE;
    if (ld_q < cols || ld_qt < rows || ld_st < rows / 128) return FP8HG_ERR_INVALID_ARG;
    if (ld_s < (gran == FP8HG_GRAN_ROW ? 1 : cols / 128)) return FP8HG_ERR_INVALID_ARG;
    return status_from_cuda(fp8hg::launch_requant_t(q, rows, cols, ld_q, scale, ld_s,
                                                    gran == FP8HG_GRAN_ROW ? 1 : 0, fmt_in,
                                                    fmt_out, q_t, ld_qt, scale_t, ld_st, w,
                                                    static_cast<cudaStream_t>(stream)));
}

int fp8_requant_t(const uint8_t *q, int64_t rows, int64_t cols, int64_t ld_q, const uint8_t *scale,
                  int64_t ld_s, int gran, int fmt_in, int fmt_out, uint8_t *q_t, int64_t ld_qt,
                  uint8_t *scale_t, int64_t ld_st, void *stream) {
    return fp8_requant_t_ex(q, rows, cols, ld_q, scale, ld_s, gran, fmt_in, fmt_out, q_t, ld_qt,
                            scale_t, ld_st, nullptr, stream);
}

int fp8_gemm_scaled_ex(int op, const fp8hg_operand *a, const fp8hg_operand *b, void *c, int64_t ldc,
                       int out, int accumulate, const fp8hg_gemm_opts *opts, void *stream) {
    if (out != FP8HG_OUT_BF16 && out != FP8HG_OUT_FP32) return FP8HG_ERR_INVALID_ARG;
    if (accumulate != 0 && accumulate != 1) return FP8HG_ERR_INVALID_ARG;
    fp8hg::GemmArgs g;
    int st = prepare_gemm(op, a, b, g);
    if (st != FP8HG_OK) return st;
    if (!c) return FP8HG_ERR_INVALID_ARG;
    if (!aligned(c, 16)) return FP8HG_ERR_ALIGNMENT;
    if (ldc < b->rows) return FP8HG_ERR_INVALID_ARG;
    if (ldc % (out == FP8HG_OUT_BF16 ? 8 : 4)) return FP8HG_ERR_ALIGNMENT;
    if (opts && (opts->inject_fault < 0 || opts->inject_fault > 1)) return FP8HG_ERR_INVALID_ARG;
    if (opts && (opts->tile < 0 || opts->tile > 3)) return FP8HG_ERR_INVALID_ARG;
    if (opts && opts->tile >= 2 && a->rows % 256) return FP8HG_ERR_UNSUPPORTED;
    g.c = c;
    g.ldc = ldc;
    g.out_fp32 = out == FP8HG_OUT_FP32;
    g.accumulate = accumulate;
    return run_gemm(g, opts, stream);
}

size_t fp8_gemm_splitk_workspace(int64_t M, int64_t N, int64_t K, int split_k) {
    if (M <= 0 || N <= 0 || K <= 0 || M % 256 || N % 128 || K % 128) return 0;
    if (split_k < 0 || split_k > 8 || split_k > K / 128) return 0;
    return fp8hg::gemm_splitk_workspace(M, N, K, split_k);
}

int fp8_gemm_scaled_splitk(int op, const fp8hg_operand *a, const fp8hg_operand *b, void *c,
                           int64_t ldc, int out, int accumulate, int split_k, void *workspace,
                           size_t workspace_bytes, const fp8hg_gemm_opts *opts, void *stream) {
    if (out != FP8HG_OUT_BF16 && out != FP8HG_OUT_FP32) return FP8HG_ERR_INVALID_ARG;
    if (accumulate != 0 && accumulate != 1) return FP8HG_ERR_INVALID_ARG;
    if (split_k < 0 || split_k > 8) return FP8HG_ERR_INVALID_ARG;
    if (opts && (opts->inject_fault < 0 || opts->inject_fault > 2)) return FP8HG_ERR_INVALID_ARG;
    if (opts && (opts->tile < 0 || opts->tile > 3)) return FP8HG_ERR_INVALID_ARG;
    fp8hg::GemmArgs g;
    int st = prepare_gemm(op, a, b, g);
    if (st != FP8HG_OK) return st;
    if (!c) return FP8HG_ERR_INVALID_ARG;
    if (!aligned(c, 16)) return FP8HG_ERR_ALIGNMENT;
    if (ldc < b->rows) return FP8HG_ERR_INVALID_ARG;
    if (ldc % (out == FP8HG_OUT_BF16 ? 8 : 4)) return FP8HG_ERR_ALIGNMENT;
    if (workspace && !aligned(workspace, 256)) return FP8HG_ERR_ALIGNMENT;
    if (split_k > a->k / 128) return FP8HG_ERR_SHAPE;              // every part >= 1 k-block
    if (split_k >= 2) {
        // the split runs on the 256 x 224 tiles
        if (a->rows % 256 || (opts && opts->tile != 0 && opts->tile != 2))
            return FP8HG_ERR_UNSUPPORTED;
        if (!workspace ||
            workspace_bytes < fp8hg::gemm_splitk_workspace(a->rows, b->rows, a->k, split_k))
            return FP8HG_ERR_INVALID_ARG;
    }
    if (opts && opts->inject_fault == 2 && split_k < 2) return FP8HG_ERR_UNSUPPORTED;
    g.c = c;
    g.ldc = ldc;
    g.out_fp32 = out == FP8HG_OUT_FP32;
    g.accumulate = accumulate;
    g.split_k = split_k;
    g.ws = workspace;
    g.ws_bytes = workspace ? workspace_bytes : 0;
    return run_gemm(g, opts, stream);
}

int fp8_gemm_scaled_q(int op, const fp8hg_operand *a, const fp8hg_operand *b, uint8_t *c_codes,
                      int64_t ld_c, uint8_t *c_scale, int64_t ld_cs, int fmt_c, void *stream) {
    if (!valid_fmt(fmt_c)) return FP8HG_ERR_INVALID_ARG;
    fp8hg::GemmArgs g;
    int st = prepare_gemm(op, a, b, g);
    if (st != FP8HG_OK) return st;
    if (!c_codes || !c_scale) return FP8HG_ERR_INVALID_ARG;
    if (!aligned(c_codes, 16) || ld_c % 16) return FP8HG_ERR_ALIGNMENT;
    if (ld_c < b->rows || ld_cs < b->rows / 128) return FP8HG_ERR_INVALID_ARG;
    g.c = c_codes;
    g.ldc = ld_c;
    g.out_q = 1;
    g.fmt_c = fmt_c;
    g.c_scale = c_scale;
    g.ld_cs = ld_cs;
    return run_gemm(g, nullptr, stream);
}

int fp8_gemm_scaled(int op, const fp8hg_operand *a, const fp8hg_operand *b, void *c, int64_t ldc,
                    int out, int accumulate, void *stream) {
    return fp8_gemm_scaled_ex(op, a, b, c, ldc, out, accumulate, nullptr, stream);
}

int fp8_quant_token_f32s(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int group,
                         int fmt, uint8_t *q, int64_t ld_q, float *scale, int64_t ld_s,
                         void *stream) {
    int st = check_quant_common(x, rows, cols, ld_x, fmt, q, ld_q,
                                reinterpret_cast<const uint8_t *>(scale));
    if (st != FP8HG_OK) return st;
    if (group != 0 && group != 128) return FP8HG_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return FP8HG_OK;
    if (!aligned(scale, 4)) return FP8HG_ERR_ALIGNMENT;
    if (cols % 128) return FP8HG_ERR_SHAPE;
    if (ld_x < cols || ld_q < cols) return FP8HG_ERR_INVALID_ARG;
    if (ld_s < (group ? cols / 128 : 1)) return FP8HG_ERR_INVALID_ARG;
    if (group == 0 && rows > 2147483647LL) return FP8HG_ERR_SHAPE;
    return status_from_cuda(fp8hg::launch_quant_token_f32s(x, rows, cols, ld_x, group, fmt, q, ld_q,
                                                           scale, ld_s,
                                                           static_cast<cudaStream_t>(stream)));
}

int fp8_quant_block128_f32s(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                            uint8_t *q, int64_t ld_q, float *scale, int64_t ld_s, uint8_t *q_t,
                            int64_t ld_qt, float *scale_t, int64_t ld_st, void *stream) {
    int st = check_quant_common(x, rows, cols, ld_x, fmt, q, ld_q,
                                reinterpret_cast<const uint8_t *>(scale));
    if (st != FP8HG_OK) return st;
    if (rows == 0 || cols == 0) return FP8HG_OK;
    if ((q_t == nullptr) != (scale_t == nullptr)) return FP8HG_ERR_INVALID_ARG;
    if (!aligned(scale, 4) || (scale_t && !aligned(scale_t, 4))) return FP8HG_ERR_ALIGNMENT;
    if (rows % 128 || cols % 128) return FP8HG_ERR_SHAPE;
    if (rows / 128 > 65535) return FP8HG_ERR_SHAPE;
    if (ld_x < cols || ld_q < cols || ld_s < cols / 128) return FP8HG_ERR_INVALID_ARG;
    if (q_t) {
        if (!aligned(q_t, 16) || ld_qt % 16) return FP8HG_ERR_ALIGNMENT;
        if (ld_qt < rows || ld_st < rows / 128) return FP8HG_ERR_INVALID_ARG;
    }
    return status_from_cuda(fp8hg::launch_quant_block128_f32s(x, rows, cols, ld_x, fmt, q, ld_q,
                                                              scale, ld_s, q_t, ld_qt, scale_t,
                                                              ld_st,
                                                              static_cast<cudaStream_t>(stream)));
}

int fp8_gemm_scaled_f32s_ex(int op, const fp8hg_operand_f32s *a, const fp8hg_operand_f32s *b,
                            void *c, int64_t ldc, int out, const fp8hg_wait_opts *opts,
                            void *stream) {
    fp8hg::WaitOpts w;
    const int wst = wait_opts(opts, w);
    if (wst != FP8HG_OK) return wst;
    if (op < FP8HG_FPROP || op > FP8HG_WGRAD) return FP8HG_ERR_INVALID_ARG;
    if (out != FP8HG_OUT_BF16 && out != FP8HG_OUT_FP32) return FP8HG_ERR_INVALID_ARG;
    if (!a || !b) return FP8HG_ERR_INVALID_ARG;
    for (const fp8hg_operand_f32s *o : {a, b}) {
        if (!valid_fmt(o->fmt)) return FP8HG_ERR_INVALID_ARG;
        if (o->rows <= 0 || o->k <= 0 || o->rows % 128 || o->k % 128) return FP8HG_ERR_SHAPE;
        if (o->rows > 2147483647LL || o->k > 2147483647LL) return FP8HG_ERR_SHAPE;
        if (!o->codes || !o->scale) return FP8HG_ERR_INVALID_ARG;
        if (!aligned(o->codes, 16) || o->ld % 16 || !aligned(o->scale, 4))
            return FP8HG_ERR_ALIGNMENT;
        if (o->ld < o->k) return FP8HG_ERR_INVALID_ARG;
    }
    if (a->k != b->k) return FP8HG_ERR_SHAPE;
    if (op == FP8HG_WGRAD) return FP8HG_ERR_UNSUPPORTED;
    if ((a->gran != FP8HG_GRAN_ROW && a->gran != FP8HG_GRAN_1x128) || b->gran != FP8HG_GRAN_128x128)
        return FP8HG_ERR_UNSUPPORTED;
    if (a->ld_scale < (a->gran == FP8HG_GRAN_ROW ? 1 : a->k / 128)) return FP8HG_ERR_INVALID_ARG;
    if (b->ld_scale < b->k / 128) return FP8HG_ERR_INVALID_ARG;
    if (!c) return FP8HG_ERR_INVALID_ARG;
    if (!aligned(c, 16)) return FP8HG_ERR_ALIGNMENT;
    if (ldc < b->rows) return FP8HG_ERR_INVALID_ARG;
    if (ldc % (out == FP8HG_OUT_BF16 ? 8 : 4)) return FP8HG_ERR_ALIGNMENT;
    unsigned int *err = fp8hg::device_error_word();
    if (!err) return FP8HG_ERR_CUDA;
    fp8hg::GemmF32sArgs g{};
    g.a_codes = a->codes;
    g.b_codes = b->codes;
    g.a_scale = a->scale;
    g.b_scale = b->scale;
    g.M = a->rows;
    g.N = b->rows;
    g.K = a->k;
    g.lda = a->ld;
    g.ldb = b->ld;
    g.ld_sa = a->ld_scale;
    g.ld_sb = b->ld_scale;
    g.fmt_a = a->fmt;
    g.fmt_b = b->fmt;
    g.a_per_token = a->gran == FP8HG_GRAN_ROW;
    g.c = c;
    g.ldc = ldc;
    g.out_fp32 = out == FP8HG_OUT_FP32;
    g.wait_limit_ns = w.limit_ns ? w.limit_ns : kDefaultWaitNs;
    g.inject_fault = w.inject;
    g.err = err;
    const int rc = fp8hg::launch_gemm_f32s(g, static_cast<cudaStream_t>(stream));
    if (rc == 1) return FP8HG_ERR_UNSUPPORTED;
    return rc == 0 ? FP8HG_OK : FP8HG_ERR_CUDA;
}

int fp8_gemm_scaled_f32s(int op, const fp8hg_operand_f32s *a, const fp8hg_operand_f32s *b, void *c,
                         int64_t ldc, int out, void *stream) {
    return fp8_gemm_scaled_f32s_ex(op, a, b, c, ldc, out, nullptr, stream);
}

int fp8hg_get_device_error(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8HG_ERR_CUDA;
    unsigned int *err = fp8hg::device_error_word();
    if (!err) return FP8HG_ERR_CUDA;
    unsigned int host[2] = {0, 0};
    if (cudaMemcpy(host, err, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess)
        return FP8HG_ERR_CUDA;
    if (host[0] == 0) return FP8HG_OK;
    const unsigned int zero[2] = {0, 0};
    if (cudaMemcpy(err, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return FP8HG_ERR_CUDA;
    return FP8HG_ERR_TIMEOUT;
}

const char *fp8hg_status_str(int status) {
    switch (status) {
    case FP8HG_OK: return "FP8HG_OK";
    case FP8HG_ERR_INVALID_ARG: return "FP8HG_ERR_INVALID_ARG";
    case FP8HG_ERR_ALIGNMENT: return "FP8HG_ERR_ALIGNMENT";
    case FP8HG_ERR_SHAPE: return "FP8HG_ERR_SHAPE";
    case FP8HG_ERR_UNSUPPORTED: return "FP8HG_ERR_UNSUPPORTED";
    case FP8HG_ERR_CUDA: return "FP8HG_ERR_CUDA";
    case FP8HG_ERR_TIMEOUT: return "FP8HG_ERR_TIMEOUT";
    default: return "FP8HG_UNKNOWN_STATUS";
    }
}

int fp8hg_version(void) { return (1 << 16) | 0; }

}  // extern "C"
