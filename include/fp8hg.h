/*
 * fp8hg — hybrid-granularity FP8 quantization and block-scaled FP8 GEMM for
 * GB300 (sm_103a).  Plain C ABI: raw pointers, sizes and enums, no C++ or
 * framework types.
 *
 * What the library computes
 * -------------------------
 * The data-parallel hot path of the FP8 training recipe in "A Comprehensive
 * FP8 Training Recipe for Reasoning-Enhanced Language Models" ("Core claim",
 * "What carries the argument"): weights are quantized with one scale per
 * 128x128 block, activations with one scale per token (or per 1x128 group in
 * the tiled variant); every scale is an exponent-only UE8M0 power of two
 * rounded UP, so that amax/scale never exceeds the FP8 format's largest value;
 * the FP8 GEMMs of the forward and backward passes consume the codes and
 * scales and accumulate in FP32.  An MXFP8 mode ("Characterization and
 * Mitigation of Training Instabilities in Microscaling Formats", "What carries
 * the argument") shares one E8M0 scale per 32 elements, taken as
 * floor(log2 amax) - emax, and clamps scaled magnitudes beyond the largest
 * code.  The codes follow "FP8 Formats for Deep Learning" (abstract / core
 * claim): E4M3 without infinities and with a single NaN pattern, E5M2 with
 * IEEE-754 specials, round to nearest even.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers on the current CUDA device.  The
 *    caller allocates and owns every buffer; the library never allocates or
 *    frees memory and never synchronizes, except in fp8hg_get_device_error.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued asynchronously; the entry points return once it is launched.
 *  - BF16 inputs are passed as uint16_t bit patterns, row-major with a row
 *    stride `ld_*` in ELEMENTS.  FP8 codes and scale bytes are uint8_t,
 *    row-major with row strides in BYTES.
 *  - Scale byte b means 2^(b - 127) (UE8M0 / E8M0); b = 0xFF marks a group
 *    that held a NaN or an infinity, in which case every code of the group is
 *    0x7F (a NaN in both encodings).  A dequantized element is
 *    decode(code) * 2^(b - 127).
 *  - Return value: an fp8hg_status.  Argument, shape and alignment errors are
 *    reported before anything is launched and leave every buffer untouched.
 *    FP8HG_ERR_CUDA reports a failed launch (the CUDA error is left for the
 *    caller to query).  Errors raised inside a running kernel (a bounded wait
 *    that expired) are recorded in a device error word and reported by
 *    fp8hg_get_device_error.
 *  - Thread safety: entry points keep no host state and may be called from
 *    several threads.  Calls that write the same output buffers must be
 *    ordered by the caller (same stream or events).
 */
#ifndef FP8HG_H
#define FP8HG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8HG_OK = 0,
    FP8HG_ERR_INVALID_ARG = 1, /* null pointer, bad enum, negative size */
    FP8HG_ERR_ALIGNMENT = 2,   /* pointer or stride misaligned */
    FP8HG_ERR_SHAPE = 3,       /* sizes not multiples of the tile / group */
    FP8HG_ERR_UNSUPPORTED = 4, /* valid request the library does not offer */
    FP8HG_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
    FP8HG_ERR_TIMEOUT = 6      /* a kernel's bounded wait expired */
} fp8hg_status;

typedef enum { FP8HG_E4M3 = 0, FP8HG_E5M2 = 1 } fp8hg_format;

typedef enum {
    FP8HG_GRAN_ROW = 0,      /* one scale per row (per token) */
    FP8HG_GRAN_1x128 = 1,    /* one scale per 128 consecutive K elements of a row */
    FP8HG_GRAN_128x128 = 2,  /* one scale per 128x128 block (weights) */
    FP8HG_GRAN_MX32 = 3      /* MXFP8: one scale per 32 consecutive K elements */
} fp8hg_gran;

typedef enum { FP8HG_FPROP = 0, FP8HG_DGRAD = 1, FP8HG_WGRAD = 2 } fp8hg_op;

typedef enum { FP8HG_OUT_BF16 = 0, FP8HG_OUT_FP32 = 1 } fp8hg_out;

/*
 * Options of the quantizer and GEMM entry points whose kernels wait on
 * copies or on each other (the per-token quantizer's row staging, the
 * re-quantizer's tile ring, the FP32-scale GEMM's operand pipeline, the
 * single-read quantizer's second pass).  No passage: these exist to
 * bound and test the library's own waits.
 *   wait_limit_ns  upper bound on any single wait for a copy (0 = the
 *                  default, 2 s).  When it runs out the kernel records
 *                  FP8HG_ERR_TIMEOUT in the device error word, waits (bounded)
 *                  for the copies it still has in flight and returns; the
 *                  outputs are then unspecified.
 *   inject_fault   0 = none.  1 = the first CTA never issues its first copy,
 *                  so the wait for it can only run out: a host-chosen,
 *                  GPU-safe way to exercise the timeout path in tests.
 *   reserved       must be 0.
 */
typedef struct {
    uint64_t wait_limit_ns;
    int32_t inject_fault;
    int32_t reserved;
} fp8hg_wait_opts;

/*
 * fp8_quant_token — per-token (group = 0) or per-1x128-group (group = 128)
 * activation quantizer with UE8M0 round-up scales.
 *
 * Passage: "A Comprehensive FP8 Training Recipe ...", "What carries the
 * argument" (token-wise activation scales; E8M0 exponent-only scales rounded
 * up to a power of two); the 1x128 tiled variant and the transposed wgrad
 * re-quantization are this library's reading of where the recipe's
 * activations go in the weight-gradient GEMM.
 *
 * For each group the scale exponent is the smallest e in [-127, 127] with
 * amax <= FMAX * 2^e (FMAX = 448 for E4M3, 57344 for E5M2; amax = 0 gives
 * -127), and each code is the round-to-nearest-even FP8 encoding of
 * x * 2^-e, which never overflows.
 *
 *   x         [rows, cols] BF16, row stride ld_x elements
 *   group     0 (whole row) or 128
 *   transpose 0: q [rows, cols] (ld_q bytes), scale [rows, G] (ld_s), G = 1
 *                or cols/128.
 *             1 (group must be 128): the groups are 128 consecutive ROWS of
 *                one column, and the result is written transposed:
 *                q [cols, rows] (ld_q), scale [cols, rows/128] (ld_s).  This
 *                is the operand layout of the weight-gradient GEMM, whose
 *                contraction runs over tokens.
 *   fmt       FP8HG_E4M3 or FP8HG_E5M2
 * Requirements: transpose = 0: cols % 128 == 0; transpose = 1: rows % 128 == 0
 * and cols % 64 == 0.  x and q 16-byte aligned, ld_x % 8 == 0,
 * ld_q % 16 == 0; ld_s >= number of scale columns.  rows or cols may be 0.
 */
int fp8_quant_token(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int group,
                    int transpose, int fmt, uint8_t *q, int64_t ld_q, uint8_t *scale,
                    int64_t ld_s, void *stream);

/*
 * fp8_quant_token_dual — both quantizations an activation needs, from one read
 * of it: the per-token codes of fp8_quant_token(group = 0) and the transposed
 * 1x128-along-tokens codes of fp8_quant_token(group = 128, transpose = 1),
 * identical to what those two calls write.
 *
 * Passage: "A Comprehensive FP8 Training Recipe ...", "What carries the
 * argument" (token-wise activation scales, E8M0 exponent-only scales rounded
 * up); the forward and data-gradient GEMMs take the per-token operand, the
 * weight-gradient GEMM (contraction over tokens) the transposed one.
 *
 *   x         [rows = tokens, cols] BF16 (ld_x elements)
 *   fmt, q, scale      per-token codes [rows, cols] (ld_q bytes) in fmt,
 *                      scale [rows] at scale[r * ld_s]
 *   fmt_t, q_t, scale_t  transposed codes [cols, rows] (ld_qt bytes) in fmt_t,
 *                      scale_t [cols, rows/128] (ld_st bytes)
 *   workspace  device scratch of at least
 *              fp8_quant_token_dual_workspace(rows, cols) bytes, 16-byte
 *              aligned, owned by the caller; the call clears and uses it
 *              (per-token maxima and per-128-token counters), so calls that
 *              may overlap on the GPU need separate workspaces.
 *   opts       NULL or wait options (fp8hg_wait_opts; inject_fault = 1
 *              withholds one tile's completion so that the waits for it run
 *              out, for tests of the timeout path)
 * The kernel is a cooperative launch (every CTA resident at once).  Its
 * second pass over a 128-token stripe waits (bounded) for the first pass of
 * every tile of that stripe; an expired wait is FP8HG_ERR_TIMEOUT from
 * fp8hg_get_device_error.
 * Requirements: rows % 128 == 0, cols % 128 == 0; x, q, q_t 16-byte aligned;
 * ld_x % 8 == 0, ld_q % 16 == 0, ld_qt % 16 == 0; ld_s >= 1,
 * ld_st >= rows/128.
 */
size_t fp8_quant_token_dual_workspace(int64_t rows, int64_t cols);
int fp8_quant_token_dual(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                         uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s, int fmt_t,
                         uint8_t *q_t, int64_t ld_qt, uint8_t *scale_t, int64_t ld_st,
                         void *workspace, size_t workspace_bytes,
                         const fp8hg_wait_opts *opts, void *stream);

/*
 * fp8_quant_token_dual_noalloc — fp8_quant_token_dual for callers that cannot
 * hand the library any device memory of its own: code that runs inside a
 * framework whose memory pool owns the device and gives extensions no way to
 * call cudaMalloc, code that runs inside an allocator's own callbacks, or a
 * hot path that must not take the device-wide synchronization cudaMalloc and
 * cudaFree can cause.  It takes the same inputs and outputs, writes the same
 * bytes, and allocates nothing: its scratch is a fixed array inside the
 * library (about 2 MB, present on every device that loads the library until
 * the process exits).
 *
 * No passage of the paper corresponds to this entry point; it exists only for
 * the callers above.
 *
 *   arguments as fp8_quant_token_dual, without workspace / workspace_bytes
 * Limit: rows <= 65536; more rows is FP8HG_ERR_SHAPE (the fixed scratch holds
 * the per-token maxima of 65536 tokens).
 * The first call on a device, with that device current, looks up the array's
 * device address once; make that first call before any stream capture.
 * Every call on a device uses the same array: each call clears it before it
 * starts, and calls that can overlap on the GPU (different streams with no
 * ordering between them) race on it and give wrong results.
 */
int fp8_quant_token_dual_noalloc(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                                 int fmt, uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s,
                                 int fmt_t, uint8_t *q_t, int64_t ld_qt, uint8_t *scale_t,
                                 int64_t ld_st, const fp8hg_wait_opts *opts, void *stream);

/*
 * fp8_quant_block128 — weight quantizer, one UE8M0 round-up scale per
 * 128x128 block (the whole block's amax is taken before any element is cast).
 *
 * Passage: "A Comprehensive FP8 Training Recipe ...", "What carries the
 * argument" (block-wise weight scales); block size 128x128 is this library's
 * reading (the recipe leaves the block size unreported).
 *
 *   x        [rows, cols] BF16 (ld_x elements)
 *   q        [rows, cols] codes (ld_q bytes)
 *   scale    [rows/128, cols/128] (ld_s bytes)
 *   q_t      optional (may be NULL): the same codes transposed, [cols, rows]
 *            (ld_qt bytes) — the B operand of the data-gradient GEMM
 *   scale_t  optional (must be non-NULL iff q_t is): the scale grid transposed,
 *            [cols/128, rows/128] (ld_st bytes)
 * Requirements: rows % 128 == 0, cols % 128 == 0; x, q, q_t 16-byte aligned;
 * ld_x % 8 == 0, ld_q % 16 == 0, ld_qt % 16 == 0.
 */
int fp8_quant_block128(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                       uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s, uint8_t *q_t,
                       int64_t ld_qt, uint8_t *scale_t, int64_t ld_st, void *stream);

/*
 * fp8_quant_block128_batch — fp8_quant_block128 on up to FP8HG_BATCH_MAX
 * tensors in one launch (for example every weight of a layer, re-quantized
 * each training step), all in the same format.  Each job's codes, scales and
 * optional transposed copy are exactly those fp8_quant_block128 writes for
 * that tensor alone.
 *
 * Passage: as fp8_quant_block128.
 *
 *   jobs     n job descriptions (host memory, read during the call only);
 *            fields as the arguments of fp8_quant_block128
 *   n        0 .. FP8HG_BATCH_MAX (0: nothing to do)
 *   fmt      FP8HG_E4M3 or FP8HG_E5M2, for every job
 * Requirements: each job as fp8_quant_block128 requires; the transposed copy
 * is asked for by every job or by none (q_t and scale_t all NULL or all
 * non-NULL), else FP8HG_ERR_INVALID_ARG; jobs with rows or cols 0 are
 * skipped.  The outputs of different jobs must not overlap.  Every job is
 * checked before anything is launched: on an error nothing is written.
 */
#define FP8HG_BATCH_MAX 8
typedef struct {
    const uint16_t *x;
    int64_t rows, cols, ld_x;
    uint8_t *q;
    int64_t ld_q;
    uint8_t *scale;
    int64_t ld_s;
    uint8_t *q_t;
    int64_t ld_qt;
    uint8_t *scale_t;
    int64_t ld_st;
} fp8hg_block128_job;

int fp8_quant_block128_batch(const fp8hg_block128_job *jobs, int n, int fmt, void *stream);

/*
 * fp8_quant_mx32 — MXFP8 quantizer: 32 consecutive elements of a row share
 * one E8M0 scale 2^e with e = floor(log2 amax) - emax (emax = 8 for E4M3,
 * 15 for E5M2), clamped to [-127, 127]; codes are the saturating
 * round-to-nearest-even encoding of x * 2^-e (magnitudes beyond the largest
 * code clamp to it).
 *
 * Passage: "Characterization and Mitigation of Training Instabilities in
 * Microscaling Formats", "What carries the argument" (shared power-of-two
 * block scale; values beyond the representable limit clamp to the largest
 * code).  Block size 32 is this library's reading.
 *
 *   q            [rows, cols] codes (ld_q bytes); scale [rows, cols/32] (ld_s)
 *   clamp_count  optional device pointer; if non-NULL, the number of elements
 *                whose scaled magnitude exceeded the largest value is ADDED
 *                to *clamp_count (the caller zeroes it).
 * Requirements: cols % 32 == 0; x, q 16-byte aligned; ld_x % 8 == 0,
 * ld_q % 16 == 0.
 */
int fp8_quant_mx32(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                   uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s,
                   unsigned long long *clamp_count, void *stream);

/*
 * fp8_requant_t — re-quantizes a STORED FP8 activation for the
 * weight-gradient GEMM: 1x128 groups along the tokens, written transposed,
 * computed from the FP8 codes and their scales instead of the BF16 original.
 *
 * Passage: "A Comprehensive FP8 Training Recipe ...", "What carries the
 * argument" (activations kept in FP8 with fine-grained power-of-two scales;
 * the weight gradient contracts over tokens, so its operands need groups
 * that run along the tokens).  Each stored value x_hat = decode(q) *
 * 2^(byte - 127) is taken exactly; the output is the UE8M0 round-up
 * quantization of x_hat in groups of 128 consecutive tokens of one column,
 * cast to fmt_out by round-to-nearest-even.
 *
 *   q        [rows = tokens, cols] codes of format fmt_in (ld_q bytes)
 *   scale    gran = FP8HG_GRAN_ROW: [rows] (ld_s >= 1); FP8HG_GRAN_1x128:
 *            [rows, cols/128] (ld_s >= cols/128)
 *   q_t      [cols, rows] codes of format fmt_out (ld_qt bytes)
 *   scale_t  [cols, rows/128] (ld_st bytes)
 * A token whose scale byte is 0xFF, or a NaN / infinite code, makes the
 * output groups it belongs to non-finite (scale 0xFF, codes 0x7F).
 * Requirements: rows % 128 == 0, cols % 128 == 0; q, q_t 16-byte aligned;
 * ld_q % 16 == 0, ld_qt % 16 == 0; every stored value finite in FP32
 * (|x_hat| < 2^128: true of every operand quantized from BF16).
 */
int fp8_requant_t(const uint8_t *q, int64_t rows, int64_t cols, int64_t ld_q, const uint8_t *scale,
                  int64_t ld_s, int gran, int fmt_in, int fmt_out, uint8_t *q_t, int64_t ld_qt,
                  uint8_t *scale_t, int64_t ld_st, void *stream);

/*
 * FP32-scale variant ("FP8 w. FP32 scale").
 *
 * Passage: "A Comprehensive FP8 Training Recipe ...", referee comments: the
 * recipe's ablation compares its UE8M0 scales with an "FP8 w. FP32 scale"
 * arm that the setup does not define.  This library reads it as ordinary
 * FP32 scaling at the same granularities: per group
 *   d = fl32(amax / FMAX)       stored FP32 scale (x ~ decode(q) * d)
 *   q = RNE_sat(fl32(x * fl32(FMAX / amax)))
 * (amax = 0: d = 1, codes +-0; a NaN or infinity: d = NaN, codes 0x7F).
 * Scales are float arrays; their leading dimensions count floats.
 *
 * fp8_quant_token_f32s: group 0 (per token, scale [rows]) or 128 (1x128,
 *   scale [rows, cols/128]); cols % 128 == 0; alignment as fp8_quant_token,
 *   scale 4-byte aligned.  No transposed form.
 * fp8_quant_block128_f32s: one scale per 128x128 block, optional transposed
 *   copy (q_t [cols, rows], scale_t [cols/128, rows/128]); requirements as
 *   fp8_quant_block128.
 */
int fp8_quant_token_f32s(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int group,
                         int fmt, uint8_t *q, int64_t ld_q, float *scale, int64_t ld_s,
                         void *stream);
int fp8_quant_block128_f32s(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                            uint8_t *q, int64_t ld_q, float *scale, int64_t ld_s, uint8_t *q_t,
                            int64_t ld_qt, float *scale_t, int64_t ld_st, void *stream);

/* An operand with FP32 scales: as fp8hg_operand, scale a float array with
 * ld_scale counted in floats; gran ROW or 1x128 (A) / 128x128 (B). */
typedef struct {
    const uint8_t *codes;
    const float *scale;
    int64_t rows, k, ld, ld_scale;
    int32_t fmt, gran;
} fp8hg_operand_f32s;

/*
 * fp8_gemm_scaled_f32s — C = A * B^T with FP32 scale factors.  The tensor
 * cores accumulate each 128-K block's raw FP8 product in FP32; the FP32
 * factors sa * sb are applied on the CUDA cores between blocks (promotion).
 * op FPROP or DGRAD: A ROW or 1x128, B 128x128 (WGRAD returns
 * FP8HG_ERR_UNSUPPORTED).  out BF16 or FP32; M, N, K multiples of 128;
 * codes 16-byte aligned, ld % 16 == 0; scales 4-byte aligned.
 */
int fp8_gemm_scaled_f32s(int op, const fp8hg_operand_f32s *a, const fp8hg_operand_f32s *b, void *c,
                         int64_t ldc, int out, void *stream);

/*
 * Counts of the MX clamp monitor (all over the whole tensor):
 *   saturated         elements whose scaled magnitude x * 2^-e exceeded the
 *                     format's largest value (448 or 57344) and were written
 *                     as the largest code
 *   top_code          elements whose code has the largest finite magnitude
 *                     (0x7E / 0x7B, either sign): the last quantization bin,
 *                     reached by saturation or by rounding
 *   blocks_saturated  32-element blocks holding at least one saturated element
 *   blocks_collapsed  blocks whose 32 codes are one and the same byte (all
 *                     values in one bin); blocks of zeros and blocks holding a
 *                     NaN or an infinity are not counted
 * The same layout as four consecutive unsigned 64-bit integers.
 */
typedef struct {
    unsigned long long saturated;
    unsigned long long top_code;
    unsigned long long blocks_saturated;
    unsigned long long blocks_collapsed;
} fp8hg_mx_stats;

/*
 * fp8_quant_mx32_monitor — fp8_quant_mx32 (identical codes and scales) that
 * also counts how much of the tensor lands in the last quantization bin.
 *
 * Passage: "Characterization and Mitigation of Training Instabilities in
 * Microscaling Formats": tightly clustered blocks (layer-norm weights) are
 * pushed into the format's last bin and collapse onto one code ("What
 * carries the argument"); the fraction of values and of blocks clamped there
 * is the proposed early-warning signal of divergence ("What would settle
 * it", "If this is right").  The four counts above are this library's
 * reading of that signal.
 *
 *   stats          device pointer, required, 8-byte aligned; the counts are
 *                  ADDED to it (the caller zeroes it)
 *   row_saturated  optional device array [rows] of unsigned 32-bit counts;
 *                  each row's saturated elements are ADDED (caller zeroes)
 * Requirements as fp8_quant_mx32.  Counting uses atomics: concurrent calls
 * may share the same counters.
 */
int fp8_quant_mx32_monitor(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                           uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s,
                           fp8hg_mx_stats *stats, unsigned int *row_saturated, void *stream);

/*
 * One quantized GEMM operand: `rows` rows of `k` FP8 codes, K-contiguous.
 *   codes     device pointer, 16-byte aligned, row stride ld bytes (ld % 16 == 0)
 *   scale     device pointer to the scale bytes of `gran`:
 *               ROW      [rows]         at scale[r * ld_scale]
 *               1x128    [rows, k/128]  at scale[r * ld_scale + k/128]
 *               128x128  [rows/128, k/128]
 *               MX32     [rows, k/32]
 *             For 1x128, 128x128 and MX32 the GEMM reads the scale bytes four
 *             at a time: scale must be 4-byte aligned, ld_scale % 4 == 0 and
 *             ld_scale >= the column count rounded up to a multiple of 4
 *             (the padding bytes are read and ignored).
 *   fmt       FP8HG_E4M3 / FP8HG_E5M2;  gran  fp8hg_gran
 */
typedef struct {
    const uint8_t *codes;
    const uint8_t *scale;
    int64_t rows;
    int64_t k;
    int64_t ld;
    int64_t ld_scale;
    int32_t fmt;
    int32_t gran;
} fp8hg_operand;

/*
 * fp8_gemm_scaled — C = A * B^T on block-scaled FP8 operands, FP32
 * accumulation on the tensor cores, BF16 or FP32 output.
 *
 *   C[i, j] = sum_k (qa[i,k] * 2^ea(i,k)) * (qb[j,k] * 2^eb(j,k))
 *
 * Passage: "A Comprehensive FP8 Training Recipe ...", referee summary and
 * "What carries the argument" (E4M3 GEMMs in the forward and backward passes
 * over block-scaled weights and token-scaled activations; FP32 master
 * weights and weight gradients).  All three GEMMs of a linear layer reduce to
 * this one form once the quantizers have put both operands K-contiguous:
 *   FPROP  Y  = X W^T      A = X  [M, K] (ROW or 1x128), B = W  [N, K] (128x128)
 *   DGRAD  dX = dY W       A = dY [M, N] (ROW or 1x128), B = W^T [K, N] (128x128,
 *                          the transposed copy from fp8_quant_block128)
 *   WGRAD  dW = dY^T X     A = dY^T [N, M] (1x128), B = X^T [K, M] (1x128), both
 *                          from fp8_quant_token(transpose = 1)
 * MX32 x MX32 is accepted under any op.
 *
 *   op          fp8hg_op; only selects which granularity pairs are accepted
 *   a, b        operands; M = a->rows, N = b->rows, K = a->k = b->k
 *   c           device output [M, N], row stride ldc ELEMENTS, 16-byte aligned,
 *               ldc % 8 == 0 (BF16) or % 4 == 0 (FP32)
 *   out         FP8HG_OUT_BF16 (round to nearest even) or FP8HG_OUT_FP32
 *   accumulate  0: C = A B^T;  1: C = C + A B^T (gradient accumulation)
 * Requirements: M % 128 == 0, N % 128 == 0, K % 128 == 0, K > 0.
 * Scale bytes of 0xFF (non-finite groups) make the affected outputs NaN.
 */
int fp8_gemm_scaled(int op, const fp8hg_operand *a, const fp8hg_operand *b, void *c,
                    int64_t ldc, int out, int accumulate, void *stream);

/*
 * fp8_gemm_scaled_q — the scaled GEMM with its output quantized in the
 * epilogue: C = A * B^T (FP32 in tensor memory) leaves the kernel as FP8
 * codes with one UE8M0 round-up scale per 128 consecutive columns of a row,
 * i.e. directly as the 1x128 A operand of a following GEMM; no BF16 copy of
 * C is written and no separate quantization pass reads it back.
 *
 * Passage: "A Comprehensive FP8 Training Recipe ...", "What carries the
 * argument" (activations quantized per token / per 1x128 tile with
 * power-of-two scales rounded up so the FP8 range is never exceeded); the
 * fusion into the producing GEMM is this library's design.  The rounding
 * decisions are taken on the FP32 accumulator: amax over the group, e the
 * smallest integer with amax <= FMAX * 2^e (clamped to [-127, 127]),
 * code = RNE(C * 2^-e) in fmt_c; a group holding a NaN or an infinity gets
 * scale byte 0xFF and codes 0x7F.
 *
 *   a, b     as fp8_gemm_scaled (same op / granularity rules)
 *   c_codes  [M, N] codes (ld_c bytes, ld_c % 16 == 0, 16-byte aligned)
 *   c_scale  [M, N/128] scale bytes (ld_cs >= N/128; a multiple of four
 *            keeps it usable as a GEMM operand)
 *   fmt_c    FP8HG_E4M3 or FP8HG_E5M2
 */
int fp8_gemm_scaled_q(int op, const fp8hg_operand *a, const fp8hg_operand *b, uint8_t *c_codes,
                      int64_t ld_c, uint8_t *c_scale, int64_t ld_cs, int fmt_c, void *stream);

/*
 * Options for fp8_gemm_scaled_ex.
 *   wait_limit_ns  upper bound on any single pipeline wait inside the GEMM
 *                  kernel (0 = the default, 2 s).  When a wait runs out the
 *                  kernel stops, drains its in-flight copies, releases its
 *                  tensor memory, records FP8HG_ERR_TIMEOUT in the device
 *                  error word and returns; C is then unspecified.
 *   inject_fault   0 = none.  1 = the scale-loading warp withholds its first
 *                  arrival, so the first wait of the MMA warp can never
 *                  complete: a host-chosen, GPU-safe way to exercise the
 *                  timeout path in tests.
 *   tile           0 = the library's choice.  1 = 128 x 256 tiles.  2 = 256 x 224
 *                  tiles (two accumulators per B stage).  3 = 256 x 448 tiles
 *                  computed by a pair of CTAs (a two-CTA cluster sharing the
 *                  MMA).  2 and 3 are honoured when M is a multiple of 256,
 *                  else FP8HG_ERR_UNSUPPORTED.  The result does not depend on
 *                  the tile beyond FP32 accumulation order.
 */
typedef struct {
    uint64_t wait_limit_ns;
    int32_t inject_fault;
    int32_t tile;
} fp8hg_gemm_opts;

/* fp8_gemm_scaled with options (opts may be NULL = defaults). */
int fp8_gemm_scaled_ex(int op, const fp8hg_operand *a, const fp8hg_operand *b, void *c,
                       int64_t ldc, int out, int accumulate, const fp8hg_gemm_opts *opts,
                       void *stream);


/*
 * fp8_gemm_scaled_splitk — fp8_gemm_scaled with the K range of each output
 * tile divided into split_k parts that run on different CTAs, for shapes
 * whose tiles fill only a few waves of SMs (few tiles, long K).  The parts
 * other than the first write FP32 partial tiles into the workspace; the first
 * part's CTA waits for them (bounded) and adds them to its accumulator in
 * part order before the output conversion, so the result is deterministic
 * (it differs from fp8_gemm_scaled only in FP32 summation order).
 *
 * Passage: the same C as fp8_gemm_scaled ("A Comprehensive FP8 Training
 * Recipe ...", "What carries the argument"); splitting K is this library's
 * execution strategy and changes no rule of the recipe.
 *
 *   op, a, b, c, ldc, out, accumulate   as fp8_gemm_scaled
 *   split_k    0 = the library's choice (no split where it would not pay,
 *              or where the workspace is missing or too small), 1 = no
 *              split, 2..8 = that many parts (at most K/128)
 *   workspace  device scratch of fp8_gemm_splitk_workspace(M, N, K, split_k)
 *              bytes (for split_k = 0: what the library's choice needs on
 *              the current device; 0 bytes means it would not split),
 *              256-byte aligned, owned by the caller.  Its first bytes are
 *              per-tile counters that must be ZERO before the first call;
 *              every call that completes leaves them zero, so the workspace
 *              can be reused without clearing.  After FP8HG_ERR_TIMEOUT it
 *              must be cleared again.  Calls that may overlap on the GPU
 *              need separate workspaces.
 *   opts       as fp8_gemm_scaled_ex; tile must be 0 or 2 when split_k >= 2;
 *              inject_fault = 2 (split_k >= 2 only) makes one part withhold
 *              its completion count, so the first part's wait for it runs
 *              out (tests of the timeout path)
 * A split launch is cooperative (every CTA resident at once).
 * Requirements: as fp8_gemm_scaled; split_k >= 2 also needs M % 256 == 0
 * (else FP8HG_ERR_UNSUPPORTED).
 */
size_t fp8_gemm_splitk_workspace(int64_t M, int64_t N, int64_t K, int split_k);
int fp8_gemm_scaled_splitk(int op, const fp8hg_operand *a, const fp8hg_operand *b, void *c,
                           int64_t ldc, int out, int accumulate, int split_k, void *workspace,
                           size_t workspace_bytes, const fp8hg_gemm_opts *opts, void *stream);

/*
 * fp8_quant_token, fp8_requant_t and fp8_gemm_scaled_f32s with wait options
 * (opts may be NULL = defaults; an inject_fault outside {0, 1} is
 * FP8HG_ERR_INVALID_ARG).  For fp8_quant_token_ex only the per-token
 * quantizer of rows longer than 4096 elements waits on copies; asking it to
 * inject a fault in any other configuration returns FP8HG_ERR_UNSUPPORTED.
 */
int fp8_quant_token_ex(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int group,
                       int transpose, int fmt, uint8_t *q, int64_t ld_q, uint8_t *scale,
                       int64_t ld_s, const fp8hg_wait_opts *opts, void *stream);
int fp8_requant_t_ex(const uint8_t *q, int64_t rows, int64_t cols, int64_t ld_q,
                     const uint8_t *scale, int64_t ld_s, int gran, int fmt_in, int fmt_out,
                     uint8_t *q_t, int64_t ld_qt, uint8_t *scale_t, int64_t ld_st,
                     const fp8hg_wait_opts *opts, void *stream);
int fp8_gemm_scaled_f32s_ex(int op, const fp8hg_operand_f32s *a, const fp8hg_operand_f32s *b,
                            void *c, int64_t ldc, int out, const fp8hg_wait_opts *opts,
                            void *stream);

/*
 * fp8hg_get_device_error — synchronizes `stream`, then reads and clears the
 * device error word of the current device.  Returns FP8HG_OK,
 * FP8HG_ERR_TIMEOUT (a bounded wait in a GEMM, the per-token quantizer, the
 * re-quantizer or the single-read quantizer expired since the last call) or FP8HG_ERR_CUDA (the
 * synchronization itself failed).
 */
int fp8hg_get_device_error(void *stream);

/* Human-readable name of an fp8hg_status value (static storage). */
const char *fp8hg_status_str(int status);

/* ABI version of this header / library: (major << 16) | minor. */
int fp8hg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8HG_H */
