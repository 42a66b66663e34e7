// One read of an activation for both of its FP8 layouts.
//
// The recipe quantizes activations per token for the forward and data-gradient
// GEMMs ("A Comprehensive FP8 Training Recipe for Reasoning-Enhanced Language
// Models", "What carries the argument": token-wise activation scales), and the
// weight-gradient GEMM contracts over tokens, so the same tensor is also needed
// in 1x128 groups along the tokens, transposed.  Quantizing it twice reads it
// from HBM twice.  This kernel reads it once.
//
// Work unit: one 128-token x 128-column tile; a 128-token stripe is tiles
// wide.  Each thread holds an 8-token x 8-column block of its tile in
// registers for the whole unit:
//   1. the token maxima over the tile's columns are folded into a workspace
//      (integer atomic max on BF16 magnitude patterns, spread over 8
//      partitions by tile column), and the stripe's counter is bumped;
//   2. each column's amax over the tile's 128 tokens gives the transposed
//      codes and their scale (the 1x128 group lies inside the tile), written
//      through shared memory as whole 128-byte rows;
//   3. once every tile of the stripe has been counted, the token scales come
//      from the workspace and the same registers are cast per token.
// Persistent cooperative grid (every CTA resident); CTA b takes tiles b,
// b + G, ... (G = grid), so the tiles of a stripe are taken by neighbouring
// CTAs in the same round of the grid, or in two consecutive rounds.  Each
// CTA prefetches its next tile into a private shared-memory region by
// cp.async as soon as step 1 is counted, while it works on steps 2 and 3.  A CTA waits in step 3 only
// for first steps of the same round or of the next round's first CTAs, which
// never wait themselves on a later round while the stripe is at most G tiles
// wide (checked by the launcher), so the waits cannot form a cycle.  Every
// wait is bounded; on expiry the kernel records bit 8 in the device error
// word and its CTAs return.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "internal.h"
#include "quant_math.cuh"

namespace fp8hg {
namespace {

constexpr int kDT = 128;          // tokens per stripe = the 1x128 group along tokens
constexpr int kDC = 128;          // columns per tile
constexpr int kDThreads = 256;
constexpr int kParts = 8;         // partitions of the per-token maxima (by tile column)
constexpr uint64_t kDualWaitNs = 2000000000ull;  // 2 s

struct DualSmem {
    uint4 pre[8][kDThreads];        // next tile: vector k of thread t at pre[k][t] (cp.async;
                                    // consecutive threads, consecutive 16-byte slots)
    uint2 codes[kDC][kDT / 8];      // transposed codes: column c, 8-token groups XOR-swizzled
    uint32_t cred[8][4][16];        // per-warp column maxima, two columns per word:
                                    // [warp][p][v] holds columns 8 v + 2 p (low), + 1 (high)
    float cmul[kDC];                // column multipliers 2^-e
    uint32_t cnan[kDC];
    float rmul[kDT];                // token multipliers 2^-e (NaN: a non-finite token)
    int ok;
};

__device__ __forceinline__ uint32_t ld_acquire(const unsigned int *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const unsigned int *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// 16-byte asynchronous copy global -> shared (completion by wait_group).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Bounded wait for *counter >= target; false if `limit` nanoseconds ran out.
__device__ bool wait_count(const unsigned int *counter, uint32_t target, uint64_t limit) {
    if (ld_acquire(counter) >= target) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        __nanosleep(64);
        if (ld_acquire(counter) >= target) return true;
        if (ptx::globaltimer() - t0 > limit) return false;
    }
}

// 32-bit word p (BF16 elements 2 p, 2 p + 1) of a 16-byte vector
__device__ __forceinline__ uint32_t word_of(const uint4 &v, int p) {
    return p == 0 ? v.x : (p == 1 ? v.y : (p == 2 ? v.z : v.w));
}

// Two FP32 values times one factor with the packed FP32 multiply (each half
// correctly rounded, as two separate multiplies; by a power of two, exact).
__device__ __forceinline__ void mul2(float &a, float &b, float m) {
    uint64_t x, mm, r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
    asm("mov.b64 %0, {%1, %1};" : "=l"(mm) : "f"(m));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(mm));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

// Two BF16 values (lo, hi) scaled by m -> two FP8 codes (lo in the low byte);
// a NaN multiplier gives the NaN code for both.
template <int FMT>
__device__ __forceinline__ uint32_t cast_pair(float lo, float hi, float m) {
    mul2(lo, hi, m);
    return cvt2<FMT>(lo, hi);
}

// One token's 8 consecutive BF16 values -> 8 codes.
template <int FMT>
__device__ __forceinline__ uint2 cast_row8(const uint4 &v, float m) {
    uint32_t c[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t w = word_of(v, p);
        c[p] = cast_pair<FMT>(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u), m);
    }
    return make_uint2(__byte_perm(c[0], c[1], 0x5410), __byte_perm(c[2], c[3], 0x5410));
}

// FP32 value of BF16 element j (0..7) of a 16-byte vector
__device__ __forceinline__ float f32_el(const uint4 &v, int j) {
    const uint32_t w = j < 2 ? v.x : (j < 4 ? v.y : (j < 6 ? v.z : v.w));
    return __uint_as_float((j & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// F1: per-token codes; F2: transposed 1x128 codes.  Thread tid holds tokens
// 8 g .. 8 g + 7 (g = tid / 16) and columns 8 v .. 8 v + 7 (v = tid % 16) of
// the tile: vector k is token 8 g + k.
template <int F1, int F2>
__global__ void __launch_bounds__(kDThreads, 4)
    k_quant_dual(const uint16_t *__restrict__ x, int64_t ld_x, int stripes, int tiles,
                 uint8_t *__restrict__ q, int64_t ld_q, uint8_t *__restrict__ s, int64_t ld_s,
                 uint8_t *__restrict__ qt, int64_t ld_qt, uint8_t *__restrict__ st, int64_t ld_st,
                 unsigned int *__restrict__ rowmax, unsigned int *__restrict__ done,
                 uint64_t wait_ns, int inject, unsigned int *err) {
    extern __shared__ __align__(16) uint8_t dual_smem[];
    DualSmem &sm = *reinterpret_cast<DualSmem *>(dual_smem);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = tid >> 4, v = tid & 15;
    const int64_t n1 = static_cast<int64_t>(stripes) * tiles;
    const int64_t rows = static_cast<int64_t>(stripes) * kDT;
    // inject = 1 (a test of the timeout path): CTA 0 never counts its first
    // tile, so the cast of that stripe can only run out of time.
    bool withhold = inject == 1 && blockIdx.x == 0;
    auto issue = [&](int64_t t) {
        const int64_t rr0 = (t / tiles) * kDT, cc0 = (t % tiles) * kDC;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            cp_async16(ptx::smem_u32(&sm.pre[k][tid]), x + (rr0 + 8 * g + k) * ld_x + cc0 + 8 * v);
        cp_async_commit();
    };
    if (static_cast<int64_t>(blockIdx.x) < n1) issue(blockIdx.x);
    for (int64_t t = blockIdx.x; t < n1; t += gridDim.x) {
        const int stripe = static_cast<int>(t / tiles), tcol = static_cast<int>(t % tiles);
        const int64_t r0 = static_cast<int64_t>(stripe) * kDT, c0 = static_cast<int64_t>(tcol) * kDC;
        // this thread's block (its own copies), then the next tile's copies
        cp_async_wait_all();
        uint4 a[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] = sm.pre[k][tid];

        // 1. token maxima and column maxima in one pass over the |x| patterns
        // (two columns per word, sign bits cleared): the 16 threads of a
        // token group reduce its maximum over 128 columns; each column's over
        // this thread's 8 tokens, then over the two token groups of the warp
        uint32_t cp[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            uint32_t am[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                am[p] = word_of(a[k], p) & 0x7FFF7FFFu;
                cp[p] = __vmaxu2(cp[p], am[p]);
            }
            const uint32_t t2 = __vmaxu2(__vmaxu2(am[0], am[1]), __vmaxu2(am[2], am[3]));
            uint32_t m = max(t2 & 0xFFFFu, t2 >> 16);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            if (v == 0) atomicMax(rowmax + (tcol % kParts) * rows + r0 + 8 * g + k, m);
        }
#pragma unroll
        for (int p = 0; p < 4; ++p) cp[p] = __vmaxu2(cp[p], __shfl_xor_sync(0xFFFFFFFFu, cp[p], 16));
        if (lane < 16) {
#pragma unroll
            for (int p = 0; p < 4; ++p) sm.cred[warp][p][v] = cp[p];
        }
        __syncthreads();
        if (tid == 0) {
            // release: one fence, after the barrier, orders every thread's
            // token maxima of this tile before the count (a fence in every
            // thread would stall each of them on its own outstanding stores)
            __threadfence();
            if (!withhold) atomicAdd(done + stripe, 1u);
            withhold = false;
        }
        // every thread has its block in registers: the next tile's copies go
        // out now (thread 0's after its fence, which would otherwise wait for
        // them) and land while this tile is finished
        if (t + gridDim.x < n1) issue(t + gridDim.x);
        // 2. column scales and the transposed codes (staged in shared memory)
        uint32_t cbyte = 0;   // column tid's scale byte (tid < 128), stored after the count
        if (tid < kDC) {
            uint32_t m = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) m = __vmaxu2(m, sm.cred[w][(tid & 7) >> 1][tid >> 3]);
            m = (tid & 1) ? (m >> 16) : (m & 0xFFFFu);
            float mul;
            cbyte = group_scale<F2, false>(m, mul);
            sm.cmul[tid] = mul;
            sm.cnan[tid] = cbyte == 0xFFu;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = 8 * v + j;
            const float mul = sm.cmul[c];
            uint2 w;
            if (sm.cnan[c]) {
                w = make_uint2(kNanCodes, kNanCodes);
            } else {
                const uint32_t p0 = cast_pair<F2>(f32_el(a[0], j), f32_el(a[1], j), mul);
                const uint32_t p1 = cast_pair<F2>(f32_el(a[2], j), f32_el(a[3], j), mul);
                const uint32_t p2 = cast_pair<F2>(f32_el(a[4], j), f32_el(a[5], j), mul);
                const uint32_t p3 = cast_pair<F2>(f32_el(a[6], j), f32_el(a[7], j), mul);
                w = make_uint2(__byte_perm(p0, p1, 0x5410), __byte_perm(p2, p3, 0x5410));
            }
            sm.codes[c][(g ^ (c >> 3)) & 15] = w;   // token group g of column c
        }
        __syncthreads();
        if (tid < kDC) st[(c0 + tid) * ld_st + stripe] = static_cast<uint8_t>(cbyte);
        // transposed rows: column c, tokens 16 h .. 16 h + 15 (two token groups)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = tid + kDThreads * i, c = e >> 3, h = e & 7;
            const uint2 lo = sm.codes[c][(2 * h ^ (c >> 3)) & 15];
            const uint2 hi = sm.codes[c][((2 * h + 1) ^ (c >> 3)) & 15];
            *reinterpret_cast<uint4 *>(qt + (c0 + c) * ld_qt + r0 + 16 * h) =
                make_uint4(lo.x, lo.y, hi.x, hi.y);
        }
        // 3. per-token codes once the whole stripe has been counted
        if (tid == 0) sm.ok = wait_count(done + stripe, static_cast<uint32_t>(tiles), wait_ns);
        __syncthreads();
        if (!sm.ok) {
            if (tid == 0) atomicOr(err, 8u);
            cp_async_wait_all();   // no copy into this CTA's shared memory outlives it
            return;
        }
        if (tid < kDT) {
            // thread 0 read the count with acquire and the barrier orders these
            // loads after it: independent relaxed loads, one round trip (a
            // chain of acquire loads would cost one round trip each)
            uint32_t m = 0;
#pragma unroll
            for (int pt = 0; pt < kParts; ++pt) m = max(m, ld_relaxed(rowmax + pt * rows + r0 + tid));
            // a non-finite token's multiplier is NaN, which casts to NaN codes
            const GroupScale<F1, SCALE_UE8M0> gs(m);
            sm.rmul[tid] = gs.nan ? __uint_as_float(0x7FFFFFFFu) : gs.mul;
            if (tcol == 0) gs.store(s, (r0 + tid) * ld_s);
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int r = 8 * g + k;
            const uint2 code = cast_row8<F1>(a[k], sm.rmul[r]);
            *reinterpret_cast<uint2 *>(q + (r0 + r) * ld_q + c0 + 8 * v) = code;
        }
        __syncthreads();   // sm.cred / codes / rmul are rewritten by the next tile
    }
    cp_async_wait_all();
}

std::atomic<int> g_dual_sms[64];
std::atomic<int> g_dual_ready[64];

template <int F1, int F2>
cudaError_t launch_dual_t(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t *q,
                          int64_t ld_q, uint8_t *s, int64_t ld_s, uint8_t *qt, int64_t ld_qt,
                          uint8_t *st, int64_t ld_st, unsigned int *ws, const WaitOpts &w,
                          unsigned int *err, cudaStream_t stream) {
    auto kern = k_quant_dual<F1, F2>;
    const size_t smem = sizeof(DualSmem);
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    const int bit = 1 << (F1 * 2 + F2);
    int sms = g_dual_sms[dev].load(std::memory_order_acquire);
    if (sms == 0 || !(g_dual_ready[dev].load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        sms = n > 0 ? n : 1;
        g_dual_sms[dev].store(sms, std::memory_order_release);
        g_dual_ready[dev].fetch_or(bit, std::memory_order_acq_rel);
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int stripes = static_cast<int>(rows / kDT), tiles = static_cast<int>(cols / kDC);
    unsigned int *rowmax = ws, *done = ws + kParts * rows;
    e = cudaMemsetAsync(ws, 0, dual_workspace_bytes(rows, cols), stream);
    if (e != cudaSuccess) return e;
    int64_t grid = static_cast<int64_t>(sms) * per_sm;
    if (grid > static_cast<int64_t>(stripes) * tiles) grid = static_cast<int64_t>(stripes) * tiles;
    if (tiles > grid) {
        // a stripe wider than one round of the grid (more than ~77k columns
        // on GB300): the two quantizers, one read each
        const WaitOpts none{};
        e = launch_quant_token(x, rows, cols, ld_x, 0, 0, F1, q, ld_q, s, ld_s, none, stream);
        if (e != cudaSuccess) return e;
        return launch_quant_token(x, rows, cols, ld_x, 128, 1, F2, qt, ld_qt, st, ld_st, none, stream);
    }
    uint64_t wait_ns = w.limit_ns ? w.limit_ns : kDualWaitNs;
    int inject = w.inject;
    void *args[] = {&x, &ld_x, &stripes, &tiles, &q, &ld_q, &s, &ld_s, &qt, &ld_qt, &st, &ld_st,
                    &rowmax, &done, &wait_ns, &inject, &err};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern),
                                       dim3(static_cast<unsigned>(grid)), dim3(kDThreads), args,
                                       smem, stream);
}

// Scratch of fp8_quant_token_dual_noalloc, for callers that cannot give the
// library device memory: the per-token maxima (kParts partitions) and the
// per-stripe counters for up to kNoallocMaxRows tokens, about 2 MB.  Every
// device that loads the library holds it until the process exits; all calls
// on a device share it.
constexpr int64_t kNoallocMaxRows = 65536;
__device__ __align__(256) unsigned int
    g_dual_noalloc_ws[kParts * kNoallocMaxRows + kNoallocMaxRows / kDT];
std::atomic<unsigned int *> g_dual_noalloc_ptr[64];

}  // namespace

int64_t noalloc_dual_max_rows() { return kNoallocMaxRows; }

unsigned int *noalloc_dual_workspace() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    unsigned int *p = g_dual_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (p) return p;
    // Set-up, once per device, with that device current.  In host code the
    // array's name only stands in for it; its device address is asked for.
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_dual_noalloc_ws) != cudaSuccess || addr == nullptr)
        return nullptr;
    p = static_cast<unsigned int *>(addr);
    g_dual_noalloc_ptr[dev].store(p, std::memory_order_release);
    return p;
}

size_t dual_workspace_bytes(int64_t rows, int64_t cols) {
    (void)cols;
    const size_t words = static_cast<size_t>(kParts) * rows + static_cast<size_t>(rows / kDT);
    return (words * 4 + 255) / 256 * 256;
}

cudaError_t launch_quant_dual(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                              uint8_t *q, int64_t ld_q, uint8_t *s, int64_t ld_s, int fmt_t,
                              uint8_t *qt, int64_t ld_qt, uint8_t *st, int64_t ld_st,
                              unsigned int *ws, const WaitOpts &w, cudaStream_t stream) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    unsigned int *err = device_error_word();
    if (!err) return cudaErrorInvalidValue;
    if (fmt == FMT_E4M3)
        return fmt_t == FMT_E4M3
                   ? launch_dual_t<FMT_E4M3, FMT_E4M3>(x, rows, cols, ld_x, q, ld_q, s, ld_s, qt,
                                                       ld_qt, st, ld_st, ws, w, err, stream)
                   : launch_dual_t<FMT_E4M3, FMT_E5M2>(x, rows, cols, ld_x, q, ld_q, s, ld_s, qt,
                                                       ld_qt, st, ld_st, ws, w, err, stream);
    return fmt_t == FMT_E4M3
               ? launch_dual_t<FMT_E5M2, FMT_E4M3>(x, rows, cols, ld_x, q, ld_q, s, ld_s, qt, ld_qt,
                                                   st, ld_st, ws, w, err, stream)
               : launch_dual_t<FMT_E5M2, FMT_E5M2>(x, rows, cols, ld_x, q, ld_q, s, ld_s, qt, ld_qt,
                                                   st, ld_st, ws, w, err, stream);
}

}  // namespace fp8hg
