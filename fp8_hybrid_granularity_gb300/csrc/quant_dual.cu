// One read of an activation for both of its FP8 layouts.
//
// The recipe quantizes activations per token for the forward and data-gradient
// GEMMs ("A Comprehensive FP8 Training Recipe for Reasoning-Enhanced Language
// Models", "What carries the argument": token-wise activation scales), and the
// weight-gradient GEMM contracts over tokens, so the same tensor is also needed
// in 1x128 groups along the tokens, transposed.  Quantizing it twice reads it
// from HBM twice.  This kernel reads it once from HBM:
//
//   first pass, per 128-token x 128-column tile: each column's amax over the
//     tile's 128 tokens -> the transposed codes and their scale (the 1x128
//     group is wholly inside the tile); each row's amax over the tile's
//     columns is folded into a per-token maximum in a workspace (integer
//     atomic max on BF16 magnitude patterns, spread over 8 partitions by tile
//     column so that the ~150 tiles of a stripe do not all update the same
//     128 words), and the stripe's counter is bumped once the tile's maxima
//     are published;
//   second pass, per tile, once every tile of its 128-token stripe has passed
//     the first pass: the per-token scales from the workspace, and the tile
//     read again (from L2: the stripe was read moments before) and cast.
//
// Persistent cooperative grid (every CTA resident), work taken in rounds of
// one tile per CTA, first-pass and second-pass rounds alternating, the second
// passes a few rounds behind the first (see dual_round): a second pass only
// waits for first passes earlier in that order, so the waits cannot form a
// cycle, and the data it re-reads is a few rounds old (~60-80 MB), inside L2.  Every wait is bounded; on expiry the kernel
// records bit 8 in the device error word and its CTAs return.
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
constexpr int kParts = 8;         // the per-token maxima are kept in 8 partitions (by tile column)
constexpr uint64_t kDualWaitNs = 2000000000ull;  // 2 s

struct DualSmem {
    uint16_t tile[kDT][kDC + 8];   // first pass: the tile (rows padded: conflict-free columns)
    uint8_t codes[kDC][kDT + 16];  // first pass: transposed codes, one row per column
    uint32_t red[2][kDC];          // column amax of each half of the tokens
    float mul[kDT];                // second pass: per-token multipliers 2^-e
    uint32_t nan_row[kDT];         // second pass: the token holds a NaN or an infinity
    int ok;
};

__device__ __forceinline__ uint32_t ld_acquire(const unsigned int *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
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
        __nanosleep(128);
        if (ld_acquire(counter) >= target) return true;
        if (ptx::globaltimer() - t0 > limit) return false;
    }
}

// The work is cut into rounds of one item per CTA: first-pass rounds P1_j
// (tiles j*G .. j*G + G - 1 of the first pass, G = the grid) and second-pass
// rounds P2_j, in the order P1_0 .. P1_{lag-1}, then P2_m, P1_{m+lag} for
// m = 0, 1, ..., then the remaining P2 rounds.  Every CTA thus alternates
// between reading HBM (first pass) and L2 (second pass).  The second pass of
// round m needs first-pass tiles up to (m+1) G + T - 1, which lie in rounds
// P1_0 .. P1_{m+lag-1} when lag >= 1 + ceil(T / G): all of them come earlier
// in the order, so the waits cannot form a cycle.
__device__ __forceinline__ void dual_round(int r, int lag, int nrounds1, bool &first, int &block) {
    const int pre = min(lag, nrounds1);
    if (r < pre) {
        first = true;
        block = r;
        return;
    }
    const int t = r - pre, pairs = max(nrounds1 - lag, 0);
    if (t < 2 * pairs) {
        first = (t & 1) != 0;
        block = first ? t / 2 + lag : t / 2;
        return;
    }
    first = false;
    block = pairs + (t - 2 * pairs);
}

// F1: per-token codes; F2: transposed 1x128 codes.
template <int F1, int F2>
__global__ void __launch_bounds__(kDThreads, 4)
    k_quant_dual(const uint16_t *__restrict__ x, int64_t ld_x, int stripes, int tiles,
                 uint8_t *__restrict__ q, int64_t ld_q, uint8_t *__restrict__ s, int64_t ld_s,
                 uint8_t *__restrict__ qt, int64_t ld_qt, uint8_t *__restrict__ st, int64_t ld_st,
                 unsigned int *__restrict__ rowmax, unsigned int *__restrict__ done,
                 uint64_t wait_ns, int inject, unsigned int *err) {
    extern __shared__ __align__(16) uint8_t dual_smem[];
    DualSmem &sm = *reinterpret_cast<DualSmem *>(dual_smem);
    const int tid = threadIdx.x;
    const int64_t n1 = static_cast<int64_t>(stripes) * tiles;
    const int64_t rows = static_cast<int64_t>(stripes) * kDT;
    const int64_t G = gridDim.x;
    const int nrounds1 = static_cast<int>((n1 + G - 1) / G);
    const int lag = 2 + static_cast<int>((tiles + G - 1) / G);
    // inject = 1 (a test of the timeout path): CTA 0 never reports its first
    // tile, so the second passes of that stripe can only run out of time.
    bool withhold = inject == 1 && blockIdx.x == 0;
    // The first-pass tile is copied into sm.tile by cp.async as soon as the
    // buffer is free (after the previous first pass), so that its HBM latency
    // overlaps the second-pass item in between.  Thread tid copies vectors
    // e = tid + 256k: token e / 16, columns 8 (e % 16) .. +7.
    auto issue_tile = [&](int64_t tidx) {
        const int64_t rr0 = (tidx / tiles) * kDT, cc0 = (tidx % tiles) * kDC;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int e = tid + kDThreads * k, r = e >> 4, cv = e & 15;
            cp_async16(ptx::smem_u32(&sm.tile[r][cv * 8]), x + (rr0 + r) * ld_x + cc0 + cv * 8);
        }
        cp_async_commit();
    };
    // this CTA's next first-pass tile after round r (-1 if none)
    auto next_first = [&](int r) -> int64_t {
        for (int r2 = r + 1; r2 < 2 * nrounds1; ++r2) {
            bool f;
            int b;
            dual_round(r2, lag, nrounds1, f, b);
            const int64_t t = static_cast<int64_t>(b) * G + blockIdx.x;
            if (f && t < n1) return t;
        }
        return -1;
    };
    int64_t prefetched = -1;   // tile whose copy into sm.tile is in flight
    for (int r = 0; r < 2 * nrounds1; ++r) {
        bool first;
        int block;
        dual_round(r, lag, nrounds1, first, block);
        const int64_t idx = static_cast<int64_t>(block) * G + blockIdx.x;
        if (idx >= n1) continue;
        const int stripe = static_cast<int>(idx / tiles), tcol = static_cast<int>(idx % tiles);
        const int64_t r0 = static_cast<int64_t>(stripe) * kDT, c0 = static_cast<int64_t>(tcol) * kDC;
        if (first) {
            // --------------------------------------------------- first pass
            if (prefetched != idx) issue_tile(idx);
            cp_async_wait_all();
            __syncthreads();
            // the 16 lanes of a token reduce its maximum over the tile
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int e = tid + kDThreads * k, r = e >> 4, cv = e & 15;
                const uint4 v = *reinterpret_cast<const uint4 *>(&sm.tile[r][cv * 8]);
                uint32_t m = bf16_abs_max8(v);
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
                if ((tid & 15) == 0) atomicMax(rowmax + (tcol % kParts) * rows + r0 + r, m);
            }
            // column c over tokens 64 h .. 64 h + 63
            const int c = tid & (kDC - 1), h = tid >> 7;
            uint32_t vals[32];
            uint32_t m = 0;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const uint32_t lo = sm.tile[h * 64 + 2 * k][c];
                const uint32_t hi = sm.tile[h * 64 + 2 * k + 1][c];
                vals[k] = lo | (hi << 16);
                m = max(m, max(lo & 0x7FFFu, hi & 0x7FFFu));
            }
            sm.red[h][c] = m;
            // publish the tile's token maxima (the atomics above) before the
            // cast and the stores, so that no fence waits for those stores
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                if (!withhold) atomicAdd(done + stripe, 1u);
                withhold = false;
            }
            m = max(sm.red[0][c], sm.red[1][c]);
            float mul;
            const uint32_t sbyte = group_scale<F2, false>(m, mul);
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                if (sbyte == 0xFFu) {
                    w[k] = kNanCodes;
                } else {
                    const uint32_t a = vals[2 * k], b = vals[2 * k + 1];
                    const uint32_t p0 = cvt2<F2>(__uint_as_float(a << 16) * mul,
                                                 __uint_as_float(a & 0xFFFF0000u) * mul);
                    const uint32_t p1 = cvt2<F2>(__uint_as_float(b << 16) * mul,
                                                 __uint_as_float(b & 0xFFFF0000u) * mul);
                    w[k] = p0 | (p1 << 16);
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint4 *>(&sm.codes[c][h * 64 + 16 * k]) =
                    make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
            if (h == 0) st[(c0 + c) * ld_st + stripe] = static_cast<uint8_t>(sbyte);
            __syncthreads();
            // transposed rows: 128 columns x 128 tokens, whole 128-byte rows
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int e = tid + kDThreads * k, row = e >> 3, ch = e & 7;
                *reinterpret_cast<uint4 *>(qt + (c0 + row) * ld_qt + r0 + ch * 16) =
                    *reinterpret_cast<const uint4 *>(&sm.codes[row][ch * 16]);
            }
            __syncthreads();   // sm.tile / sm.codes are free again
            prefetched = next_first(r);
            if (prefetched >= 0) issue_tile(prefetched);
        } else {
            // -------------------------------------------------- second pass
            // the tile's re-read (from L2) is issued before the wait
            uint4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int e = tid + kDThreads * k, r = e >> 4, cv = e & 15;
                v[k] = ptx::ld_stream_v4(x + (r0 + r) * ld_x + c0 + cv * 8);
            }
            if (tid == 0) sm.ok = wait_count(done + stripe, static_cast<uint32_t>(tiles), wait_ns);
            __syncthreads();
            if (!sm.ok) {
                if (tid == 0) atomicOr(err, 8u);
                cp_async_wait_all();   // no copy into this CTA's shared memory outlives it
                return;
            }
            if (tid < kDT) {
                uint32_t m = 0;
#pragma unroll
                for (int pt = 0; pt < kParts; ++pt)
                    m = max(m, ld_acquire(rowmax + pt * rows + r0 + tid));
                const GroupScale<F1, SCALE_UE8M0> gs(m);
                sm.mul[tid] = gs.mul;
                sm.nan_row[tid] = gs.nan;
                if (tcol == 0) gs.store(s, (r0 + tid) * ld_s);
            }
            __syncthreads();
            uint32_t unused = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int e = tid + kDThreads * k, r = e >> 4, cv = e & 15;
                const uint2 code = sm.nan_row[r] ? make_uint2(kNanCodes, kNanCodes)
                                                 : quant8<F1, false>(v[k], sm.mul[r], unused);
                *reinterpret_cast<uint2 *>(q + (r0 + r) * ld_q + c0 + cv * 8) = code;
            }
            __syncthreads();   // sm.mul / nan_row are rewritten by the next item
        }
    }
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
    if (grid > 2 * static_cast<int64_t>(stripes) * tiles) grid = 2 * static_cast<int64_t>(stripes) * tiles;
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
