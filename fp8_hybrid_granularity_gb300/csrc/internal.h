// Launchers shared between the C-ABI layer (api.cu) and the kernel files.
// Arguments are validated by the caller; these only configure and launch.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace fp8hg {

// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry
// point (no link against libcuda); null if the driver does not provide it.
using TensorMapEncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                       const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                       const cuuint32_t *, CUtensorMapInterleave,
                                       CUtensorMapSwizzle, CUtensorMapL2promotion,
                                       CUtensorMapFloatOOBfill);
TensorMapEncodeFn tensor_map_encoder();

// Wait options of the kernels that wait on copies: limit_ns bounds one wait
// (0 = the kernel's default, 2 s); inject = 1 withholds the first copy of
// CTA 0, so that wait can only run out (a GPU-safe test of the timeout path).
struct WaitOpts {
    uint64_t limit_ns = 0;
    int inject = 0;
};

// True when fp8_quant_token runs the bulk-copy row kernel (the only
// configuration of it that waits on copies).
bool quant_token_waits(int64_t cols, int group, int transpose);

cudaError_t launch_quant_token(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                               int group, int transpose, int fmt, uint8_t *q, int64_t ld_q,
                               uint8_t *s, int64_t ld_s, const WaitOpts &w, cudaStream_t stream);

// Both layouts of an activation from one read (per token, and 1x128 along
// the tokens transposed); ws: dual_workspace_bytes(rows, cols) of device
// memory (per-token maxima and per-stripe counters; zeroed by the launch).
size_t dual_workspace_bytes(int64_t rows, int64_t cols);
cudaError_t launch_quant_dual(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                              uint8_t *q, int64_t ld_q, uint8_t *s, int64_t ld_s, int fmt_t,
                              uint8_t *qt, int64_t ld_qt, uint8_t *st, int64_t ld_st,
                              unsigned int *ws, const WaitOpts &w, cudaStream_t stream);

// The fixed scratch of the allocation-free dual quantizer: its device address
// on the current device (looked up on the first call per device; null on
// failure) and the largest row count it serves.
unsigned int *noalloc_dual_workspace();
int64_t noalloc_dual_max_rows();

cudaError_t launch_quant_mx32(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                              uint8_t *q, int64_t ld_q, uint8_t *s, int64_t ld_s,
                              unsigned long long *cnt, cudaStream_t stream);

cudaError_t launch_quant_mx32_monitor(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                                      int fmt, uint8_t *q, int64_t ld_q, uint8_t *s, int64_t ld_s,
                                      unsigned long long *stats, unsigned int *row_sat,
                                      cudaStream_t stream);

cudaError_t launch_requant_t(const uint8_t *q, int64_t rows, int64_t cols, int64_t ld_q,
                             const uint8_t *s, int64_t ld_s, int per_token, int fmt_in,
                             int fmt_out, uint8_t *qt, int64_t ld_qt, uint8_t *st, int64_t ld_st,
                             const WaitOpts &w, cudaStream_t stream);

// Up to kBlock128BatchMax tensors' block quantization in one launch.
constexpr int kBlock128BatchMax = 8;
struct Block128Job {
    const uint16_t *x;
    int64_t ld_x;
    uint8_t *q;
    int64_t ld_q;
    uint8_t *s;
    int64_t ld_s;
    uint8_t *qt;             // transposed copy (every job or none)
    int64_t ld_qt;
    uint8_t *st;
    int64_t ld_st;
    int64_t cbs;             // column blocks: cols / 128
    int64_t first;           // the job's first block in the launch's grid
};
struct Block128Batch {
    Block128Job job[kBlock128BatchMax];
    int n;
};
cudaError_t launch_quant_block128_batch(const Block128Batch &b, int64_t blocks, int fmt, bool trans,
                                        cudaStream_t stream);
cudaError_t launch_quant_block128(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                                  int fmt, uint8_t *q, int64_t ld_q, uint8_t *s, int64_t ld_s,
                                  uint8_t *qt, int64_t ld_qt, uint8_t *st, int64_t ld_st,
                                  cudaStream_t stream);

cudaError_t launch_quant_token_f32s(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                                    int group, int fmt, uint8_t *q, int64_t ld_q, float *s,
                                    int64_t ld_s, cudaStream_t stream);

cudaError_t launch_quant_block128_f32s(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                                       int fmt, uint8_t *q, int64_t ld_q, float *s, int64_t ld_s,
                                       uint8_t *qt, int64_t ld_qt, float *st, int64_t ld_st,
                                       cudaStream_t stream);

struct GemmArgs {
    const uint8_t *a_codes, *b_codes;
    const uint8_t *a_scale, *b_scale;
    int64_t M, N, K;
    int64_t lda, ldb, ld_sa, ld_sb;
    int fmt_a, fmt_b, gran_a, gran_b;
    void *c;
    int64_t ldc;
    int out_fp32, accumulate;
    int out_q, fmt_c;        // out_q: C quantized in the epilogue (1x128 along N)
    uint8_t *c_scale;        // out_q: scale bytes [M, N/128]
    int64_t ld_cs;
    uint64_t wait_limit_ns;
    int inject_fault;
    int tile;           // 0 = choose, 1 = 128 x 256, 2 = 256 x 224
    unsigned int *err;  // device error word
    int split_k = 1;    // 1 = no split, 0 = the library's choice, >= 2 forced
    void *ws = nullptr; // split-K workspace
    size_t ws_bytes = 0;
};

// Split-K (256 x 224 tiles): the library's number of K parts for a shape on
// `sms` SMs, and the workspace bytes for `split` parts (0 = the library's).
int gemm_auto_split(int64_t M, int64_t N, int64_t K, int sms);
size_t gemm_splitk_workspace(int64_t M, int64_t N, int64_t K, int split);

// Returns 0 on success, 1 if the tensor maps could not be encoded, or a
// cudaError_t + 2 on a launch failure.
int launch_gemm_scaled(const GemmArgs &args, cudaStream_t stream);

// FP8 GEMM with FP32 scale factors (promotion on the CUDA cores): A scales
// per row (a_per_token) or per (row, 128-K block), B scales per 128x128 block.
struct GemmF32sArgs {
    const uint8_t *a_codes, *b_codes;
    const float *a_scale, *b_scale;
    int64_t M, N, K;
    int64_t lda, ldb, ld_sa, ld_sb;  // ld_sa / ld_sb in floats
    int fmt_a, fmt_b, a_per_token;
    void *c;
    int64_t ldc;
    int out_fp32;
    uint64_t wait_limit_ns;
    int inject_fault;   // 1: the producer withholds the first stage's copies
    unsigned int *err;
};
int launch_gemm_f32s(const GemmF32sArgs &args, cudaStream_t stream);

// Device address of the error word of the current device (null on failure).
unsigned int *device_error_word();

}  // namespace fp8hg
