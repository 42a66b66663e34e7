// Quantizer kernels: BF16 -> FP8 codes + UE8M0 / E8M0 scale bytes.
//
// All four are HBM-bound streaming kernels (3 bytes of traffic per element:
// 2 read, 1 written, plus one scale byte per group).  Each reads every input
// element exactly once with 16-byte vector loads, reduces the group amax with
// warp shuffles (integer max on BF16 patterns), derives the scale exponent
// from the amax's bit fields and casts with the hardware RNE FP8 conversion.
//
//  k_quant_row       one scale per token ("A Comprehensive FP8 Training
//                    Recipe ...", "What carries the argument": token-wise
//                    activation scales).  Persistent CTAs stage whole rows in
//                    shared memory with bulk copies several rows ahead;
//                    rows of up to 8 KB use k_quant_row_regs (one CTA per row,
//                    row in registers).
//  k_quant_groups    one scale per 1x128 group (tiled activations) or per
//                    32-element MX block ("Characterization and Mitigation of
//                    Training Instabilities in Microscaling Formats", "What
//                    carries the argument").  A group is 16 (resp. 4) lanes.
//  k_quant_t         1x128 groups along the ROWS (tokens) of x, written
//                    transposed: the weight-gradient GEMM's operand layout.
//  k_quant_block128  one scale per 128x128 block (block-wise weights), with
//                    an optional transposed copy for the data-gradient GEMM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "quant_math.cuh"

namespace fp8hg {

// ------------------------------------------------------------------ per row
// Persistent, one CTA per SM.  Whole rows are staged in shared memory by 1-D
// bulk copies issued by one thread, up to nslots rows ahead (each slot's
// completion on its own mbarrier), so the bytes in flight do not depend on
// registers.  For each row the CTA reduces the amax from shared memory, then
// casts from shared memory and stores the codes.
constexpr int kRowThreads = 512;
constexpr int kMaxRowSlots = 8;
constexpr int kRowSmemBudget = 200 * 1024;

constexpr uint64_t kRowWaitNs = 2000000000ull;  // bound on one row's copy (2 s)

// Thread 0 waits (bounded) for a slot's copy; false when the bound ran out.
__device__ __forceinline__ bool row_wait(uint32_t bar, uint32_t parity, uint64_t limit) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity))
        if (ptx::globaltimer() - t0 > limit) return false;
    return true;
}

template <int FMT, int SM>
__global__ void __launch_bounds__(kRowThreads) k_quant_row(const uint16_t *__restrict__ x,
                                                              int64_t rows, int nvec, int64_t ld_x,
                                                              uint8_t *__restrict__ q, int64_t ld_q,
                                                              uint8_t *__restrict__ s, int64_t ld_s,
                                                              int nslots, uint64_t wait_ns,
                                                              int inject, unsigned int *err) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[kMaxRowSlots];
    __shared__ uint32_t red[kRowThreads / 32];
    __shared__ int row_ok;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const uint32_t row_bytes = static_cast<uint32_t>(nvec) * 16u;
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t fbase = ptx::smem_u32(full);
    const int64_t step = gridDim.x;
    // inject = 1 (a test of the timeout path): CTA 0 never issues the copy of
    // its first row, so the wait for it can only run out.
    const bool withhold_first = inject == 1 && blockIdx.x == 0;
    if (tid == 0) {
        for (int i = 0; i < nslots; ++i) ptx::mbar_init(fbase + 8 * i, 1);
        ptx::fence_mbar_init();
        // prologue: the first nslots - 1 rows of this CTA
        for (int i = 0; i < nslots - 1; ++i) {
            const int64_t r = blockIdx.x + i * step;
            if (r >= rows) break;
            if (i == 0 && withhold_first) continue;
            ptx::mbar_arrive_expect_tx(fbase + 8 * i, row_bytes);
            ptx::bulk_load(sbase + i * row_bytes, x + r * ld_x, row_bytes, fbase + 8 * i);
        }
    }
    __syncthreads();
    int k = 0;  // rows done by this CTA
    for (int64_t row = blockIdx.x; row < rows; row += step, ++k) {
        const int slot = k % nslots;
        // issue the row nslots - 1 ahead into the slot the previous row freed
        if (tid == 0) {
            const int64_t r = row + static_cast<int64_t>(nslots - 1) * step;
            if (r < rows && !(withhold_first && k + nslots - 1 == 0)) {
                const int sl = (k + nslots - 1) % nslots;
                ptx::mbar_arrive_expect_tx(fbase + 8 * sl, row_bytes);
                ptx::bulk_load(sbase + sl * row_bytes, x + r * ld_x, row_bytes, fbase + 8 * sl);
            }
        }
        if (tid == 0) {
            row_ok = row_wait(fbase + 8 * slot, static_cast<uint32_t>(k / nslots) & 1u, wait_ns);
            if (!row_ok) {
                atomicOr(err, 2u);
                // let this CTA's other copies in flight land before it exits
                for (int j = 1; j < nslots; ++j) {
                    const int64_t r = row + static_cast<int64_t>(j) * step;
                    if (r >= rows) break;
                    const int sl = (k + j) % nslots;
                    row_wait(fbase + 8 * sl, static_cast<uint32_t>((k + j) / nslots) & 1u, 2000000ull);
                }
            }
        }
        __syncthreads();  // also makes the copied row visible to every thread
        if (!row_ok) return;
        const uint4 *xs = reinterpret_cast<const uint4 *>(smem + static_cast<size_t>(slot) * row_bytes);
        uint32_t m = 0;
        for (int c = tid; c < nvec; c += blockDim.x) m = max(m, bf16_abs_max8(xs[c]));
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0) red[warp] = m;
        __syncthreads();
        m = 0;
        for (int w = 0; w < nwarps; ++w) m = max(m, red[w]);
        const GroupScale<FMT, SM> gs(m);
        uint2 *qr = reinterpret_cast<uint2 *>(q + row * ld_q);
        uint32_t unused = 0;
        for (int c = tid; c < nvec; c += blockDim.x)
            qr[c] = gs.nan ? make_uint2(kNanCodes, kNanCodes)
                           : quant8<FMT, false>(xs[c], gs.mul, unused);
        if (tid == 0) gs.store(s, row * ld_s);
        __syncthreads();  // the slot and red[] are free for the next row
    }
}

// Short rows (up to 8 KB): one CTA per row, the row kept in registers between
// the amax and the cast; many small CTAs keep the memory system busy.
// GV = 0: one scale for the whole row (per token).  GV = 16 (1x128) or 4
// (MX 32): one scale per group of GV consecutive 16-byte vectors; thread tid
// holds vectors tid + i * blockDim.x, so a group is GV consecutive lanes
// (blockDim.x is a multiple of 32) and is reduced with lane shuffles.
// COUNT (MX groups only): add the row's saturated elements to *cnt, one
// atomic per CTA and none for a row without any.
template <int FMT, int NV, int SM, int GV, bool COUNT = false>
__global__ void __launch_bounds__(512) k_quant_row_regs(const uint16_t *__restrict__ x, int nvec,
                                                        int64_t ld_x, uint8_t *__restrict__ q,
                                                        int64_t ld_q, uint8_t *__restrict__ s,
                                                        int64_t ld_s,
                                                        unsigned long long *__restrict__ cnt = nullptr) {
    __shared__ uint32_t red[16];
    __shared__ uint32_t bcast;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    if (COUNT && tid == 0) bcast = 0u;
    const int64_t row = blockIdx.x;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + row * ld_x);
    uint2 *qr = reinterpret_cast<uint2 *>(q + row * ld_q);
    uint4 v[NV];
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c = tid + i * blockDim.x;
        if (c < nvec) {
            v[i] = ptx::ld_stream_v4(xr + c);
            m = max(m, bf16_abs_max8(v[i]));
        }
    }
    uint32_t unused = 0, nsat = 0;
    if constexpr (GV > 0) {
        // nvec is a multiple of GV, so a group is either wholly inside the
        // row or wholly past it; every lane reaches the shuffles
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int c = tid + i * blockDim.x;
            const bool ok = c < nvec;
            uint32_t g = ok ? bf16_abs_max8(v[i]) : 0u;
#pragma unroll
            for (int o = GV / 2; o > 0; o >>= 1) g = max(g, __shfl_xor_sync(0xFFFFFFFFu, g, o));
            if (ok) {
                const GroupScale<FMT, SM> gs(g);
                qr[c] = gs.nan ? make_uint2(kNanCodes, kNanCodes)
                               : quant8<FMT, COUNT>(v[i], gs.mul, COUNT ? nsat : unused);
                if ((tid % GV) == 0) gs.store(s, row * ld_s + c / GV);
            }
        }
        if constexpr (COUNT) {
            nsat = __reduce_add_sync(0xFFFFFFFFu, nsat);
            __syncthreads();   // the counter's reset is visible
            if (lane == 0 && nsat) atomicAdd(&bcast, nsat);
            __syncthreads();
            if (tid == 0 && bcast) atomicAdd(cnt, static_cast<unsigned long long>(bcast));
        }
        return;
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (warp == 0) {
        uint32_t t = (lane < nwarps) ? red[lane] : 0u;
        t = __reduce_max_sync(0xFFFFFFFFu, t);
        if (lane == 0) bcast = t;
    }
    __syncthreads();
    const GroupScale<FMT, SM> gs(bcast);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c = tid + i * blockDim.x;
        if (c < nvec) {
            qr[c] = gs.nan ? make_uint2(kNanCodes, kNanCodes)
                           : quant8<FMT, false>(v[i], gs.mul, unused);
        }
    }
    if (tid == 0) gs.store(s, row * ld_s);
}

// Rows too long to keep in registers: the amax pass and the cast pass read the
// row twice (the second read is served from L2).
template <int FMT, int SM>
__global__ void __launch_bounds__(512) k_quant_row_2pass(const uint16_t *__restrict__ x, int nvec,
                                                         int64_t ld_x, uint8_t *__restrict__ q,
                                                         int64_t ld_q, uint8_t *__restrict__ s,
                                                         int64_t ld_s) {
    __shared__ uint32_t red[16];
    __shared__ uint32_t bcast;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int64_t row = blockIdx.x;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + row * ld_x);
    uint32_t m = 0;
    for (int c = tid; c < nvec; c += blockDim.x) m = max(m, bf16_abs_max8(xr[c]));
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (warp == 0) {
        uint32_t t = (lane < nwarps) ? red[lane] : 0u;
        t = __reduce_max_sync(0xFFFFFFFFu, t);
        if (lane == 0) bcast = t;
    }
    __syncthreads();
    const GroupScale<FMT, SM> gs(bcast);
    uint2 *qr = reinterpret_cast<uint2 *>(q + row * ld_q);
    uint32_t unused = 0;
    for (int c = tid; c < nvec; c += blockDim.x) {
        qr[c] = gs.nan ? make_uint2(kNanCodes, kNanCodes)
                       : quant8<FMT, false>(xr[c], gs.mul, unused);
    }
    if (tid == 0) gs.store(s, row * ld_s);
}

// ------------------------------------------------------ groups along a row
// Optional counters of the MX quantizer.  clamp: elements whose scaled
// magnitude exceeded the format's maximum.  Monitor (stats non-null): the
// four counts of fp8hg_mx_stats, and per-row saturated counts.
struct MxCounters {
    unsigned long long *clamp;     // COUNT: saturated elements
    unsigned long long *stats;     // MON: saturated, top code, saturated blocks, collapsed blocks
    unsigned int *row_sat;         // MON, optional: saturated elements per row
};

// Number of the eight codes whose magnitude is the format's largest code.
template <int FMT>
__device__ __forceinline__ uint32_t top_codes(const uint2 &c) {
    constexpr uint32_t T = (FMT == FMT_E4M3 ? 0x7Eu : 0x7Bu) * 0x01010101u;
    const uint32_t a = __vcmpeq4(c.x & 0x7F7F7F7Fu, T), b = __vcmpeq4(c.y & 0x7F7F7F7Fu, T);
    return (__popc(a) + __popc(b)) >> 3;
}

// GV = 16-byte vectors per group: 16 (1x128) or 4 (MX 32).  A CTA covers
// 256*U consecutive vectors of a row (blockIdx.x) for the rows blockIdx.y,
// blockIdx.y + gridDim.y, ...; lanes [g*GV, g*GV + GV) of a warp hold one
// group, and every lane reaches the shuffles.
// D: rows in flight ahead of the one being cast (1 or 2).
template <int FMT, int GV, int SM, bool COUNT, bool MON, int U, int D>
__global__ void __launch_bounds__(256) k_quant_groups(const uint16_t *__restrict__ x, int64_t rows,
                                                      int vpr, int64_t ld_x,
                                                      uint8_t *__restrict__ q, int64_t ld_q,
                                                      uint8_t *__restrict__ s, int64_t ld_s,
                                                      MxCounters cnt) {
    constexpr bool SAT = COUNT || MON;
    const int lane = threadIdx.x & 31;
    const int cv0 = blockIdx.x * (256 * U) + threadIdx.x;
    uint32_t nsat = 0, ntop = 0, nbsat = 0, ncoll = 0;
    uint4 v[U], nxt[U], nxt2[U];
    auto load = [&](int64_t r, uint4 (&dst)[U]) {
        const uint16_t *xr = x + r * ld_x;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int cv = cv0 + u * 256;
            if (cv < vpr) dst[u] = ptx::ld_stream_v4(xr + static_cast<int64_t>(cv) * 8);
        }
    };
    // D rows in flight ahead of the one being cast (with few rows per CTA,
    // each would otherwise wait a full round trip)
    const int64_t gy = gridDim.y;
    if (static_cast<int64_t>(blockIdx.y) < rows) load(blockIdx.y, nxt);
    if (D == 2 && static_cast<int64_t>(blockIdx.y) + gy < rows) load(blockIdx.y + gy, nxt2);
    for (int64_t row = blockIdx.y; row < rows; row += gy) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            v[u] = nxt[u];
            if (D == 2) nxt[u] = nxt2[u];
        }
        if (D == 2) {
            if (row + 2 * gy < rows) load(row + 2 * gy, nxt2);
        } else if (row + gy < rows) {
            load(row + gy, nxt);
        }
        uint32_t row_nsat = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int cv = cv0 + u * 256;
            const bool ok = cv < vpr;
            uint32_t m = ok ? bf16_abs_max8(v[u]) : 0u;
#pragma unroll
            for (int o = GV / 2; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            uint2 out = make_uint2(0u, 0u);
            bool group_nan = false;
            const uint32_t before = nsat;
            if (ok) {
                const GroupScale<FMT, SM> gs(m);
                group_nan = gs.nan;
                out = gs.nan ? make_uint2(kNanCodes, kNanCodes)
                             : quant8<FMT, SAT>(v[u], gs.mul, nsat);
                *reinterpret_cast<uint2 *>(q + row * ld_q + static_cast<int64_t>(cv) * 8) = out;
                if ((lane % GV) == 0) gs.store(s, row * ld_s + cv / GV);
            }
            if constexpr (MON) {
                // lanes past the row's end hold out = 0: no top codes, no saturation
                const uint32_t dsat = nsat - before;
                ntop += top_codes<FMT>(out);
                const uint32_t first = __shfl_sync(0xFFFFFFFFu, out.x, lane & ~(GV - 1)) & 0xFFu;
                const uint32_t rep = first * 0x01010101u;
                uint32_t same = (out.x == rep && out.y == rep) ? 1u : 0u, gsat = dsat;
#pragma unroll
                for (int o = GV / 2; o > 0; o >>= 1) {
                    same &= __shfl_xor_sync(0xFFFFFFFFu, same, o);
                    gsat += __shfl_xor_sync(0xFFFFFFFFu, gsat, o);
                }
                if (ok && (lane % GV) == 0) {
                    nbsat += gsat != 0u;
                    ncoll += (same && m != 0u && !group_nan) ? 1u : 0u;
                }
                row_nsat += dsat;
            }
        }
        if constexpr (MON) {
            if (cnt.row_sat != nullptr) {
                row_nsat = __reduce_add_sync(0xFFFFFFFFu, row_nsat);
                if (lane == 0 && row_nsat) atomicAdd(cnt.row_sat + row, row_nsat);
            }
        }
    }
    if constexpr (SAT) {
        nsat = __reduce_add_sync(0xFFFFFFFFu, nsat);
        unsigned long long *dst = MON ? cnt.stats : cnt.clamp;
        if (lane == 0 && nsat) atomicAdd(dst, static_cast<unsigned long long>(nsat));
    }
    if constexpr (MON) {
        ntop = __reduce_add_sync(0xFFFFFFFFu, ntop);
        nbsat = __reduce_add_sync(0xFFFFFFFFu, nbsat);
        ncoll = __reduce_add_sync(0xFFFFFFFFu, ncoll);
        if (lane == 0) {
            if (ntop) atomicAdd(cnt.stats + 1, static_cast<unsigned long long>(ntop));
            if (nbsat) atomicAdd(cnt.stats + 2, static_cast<unsigned long long>(nbsat));
            if (ncoll) atomicAdd(cnt.stats + 3, static_cast<unsigned long long>(ncoll));
        }
    }
}

// ------------------------------------------- 1x128 along rows, transposed out
// One CTA per 128-row x 64-column tile of x.  The tile is staged in shared
// memory, each column's amax over the 128 rows is reduced, and the codes are
// staged again so that the transposed output rows (64 of 128 bytes) are
// written with full, coalesced 16-byte stores.  At most 40 registers a thread
// (six CTAs per SM instead of five at 48): more tiles' loads in flight.
constexpr int kTC = 64;  // tile columns
template <int FMT>
__global__ void __launch_bounds__(256, 6) k_quant_t(const uint16_t *__restrict__ x, int64_t ld_x,
                                                 uint8_t *__restrict__ qt, int64_t ld_q,
                                                 uint8_t *__restrict__ st, int64_t ld_s) {
    __shared__ __align__(16) uint16_t tile[128][kTC + 8];
    __shared__ __align__(16) uint8_t codes[kTC][128 + 16];
    __shared__ uint32_t red[4][kTC];
    const int tid = threadIdx.x;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kTC;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = tid + 256 * i;
        const int r = idx >> 3, cv = idx & 7;
        const uint4 v = ptx::ld_stream_v4(x + (r0 + r) * ld_x + c0 + cv * 8);
        *reinterpret_cast<uint4 *>(&tile[r][cv * 8]) = v;
    }
    __syncthreads();
    const int c = tid & (kTC - 1), rq = tid >> 6;
    uint32_t vals[16];  // this thread's 32 elements, two per word
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t lo = tile[rq * 32 + 2 * i][c];
        const uint32_t hi = tile[rq * 32 + 2 * i + 1][c];
        vals[i] = lo | (hi << 16);
        m = max(m, max(lo & 0x7FFFu, hi & 0x7FFFu));
    }
    red[rq][c] = m;
    __syncthreads();
    m = max(max(red[0][c], red[1][c]), max(red[2][c], red[3][c]));
    float mul;
    const uint32_t sbyte = group_scale<FMT, false>(m, mul);
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (sbyte == 0xFFu) {
            w[j] = kNanCodes;
        } else {
            const uint32_t a = vals[2 * j], b = vals[2 * j + 1];
            const uint32_t p0 = cvt2<FMT>(__uint_as_float(a << 16) * mul,
                                          __uint_as_float(a & 0xFFFF0000u) * mul);
            const uint32_t p1 = cvt2<FMT>(__uint_as_float(b << 16) * mul,
                                          __uint_as_float(b & 0xFFFF0000u) * mul);
            w[j] = p0 | (p1 << 16);
        }
    }
    *reinterpret_cast<uint4 *>(&codes[c][rq * 32]) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4 *>(&codes[c][rq * 32 + 16]) = make_uint4(w[4], w[5], w[6], w[7]);
    if (rq == 0) st[(c0 + c) * ld_s + blockIdx.y] = static_cast<uint8_t>(sbyte);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int idx = tid + 256 * i;
        const int row = idx >> 3, ch = idx & 7;
        *reinterpret_cast<uint4 *>(qt + (c0 + row) * ld_q + r0 + ch * 16) =
            *reinterpret_cast<const uint4 *>(&codes[row][ch * 16]);
    }
}

// ------------------------------- stored FP8 codes -> 1x128 along the tokens
// Re-quantizes a stored operand (codes [tokens, cols], per-token or
// 1x128-along-K scales) for the weight-gradient GEMM.  Persistent CTAs walk
// 128-token x 128-column tiles; each tile's codes (16 KB) arrive by one 2-D
// TMA copy into one of kRqStages shared-memory stages, issued kRqStages tiles
// ahead, and the 128 tokens' scale bytes are fetched one tile ahead into
// registers.  Thread (cq, tg) owns columns 4cq..4cq+3 for the 16 tokens
// 16tg..16tg+15 and reads one 32-bit word (four columns of one token) per
// token.  Pass 1 decodes each stored value exactly in FP32 (code -> F16 ->
// F32, times the token's power-of-two scale; no FTZ, so even 2^-136 is exact)
// and keeps a NaN-propagating max of the magnitudes; the eight token groups
// of a column are combined in shared memory.  Pass 2 decodes again from the
// words held in registers and casts with the column's round-up scale.  Each
// column's 16 codes become one 16-byte chunk of the transposed tile, whose
// chunks are XOR-swizzled so that neither the chunk writes nor the row reads
// for the coalesced global stores conflict.
constexpr int kRQ = 128;          // tokens and columns per tile
constexpr int kRqStages = 4;
constexpr uint32_t kRqTileBytes = kRQ * kRQ;
constexpr uint64_t kRqWaitNs = 2000000000ull;  // bound on one tile's copy (2 s)

struct RqSmem {
    uint32_t cin[kRqStages][kRQ][kRQ / 4];   // [stage][token][4 columns]
    uint4 cout[kRQ][kRQ / 16];               // [column][swizzled 16-token chunk]
    float mul_in[kRQ];
    float red[8][kRQ];
    float mul_out[kRQ];
    uint32_t nan_col[kRQ];
    uint64_t full[kRqStages];
    int ok;
};

template <int FIN>
__device__ __forceinline__ void decode4(uint32_t w, float (&f)[4]) {
    uint32_t lo, hi;
    if constexpr (FIN == FMT_E4M3) {
        lo = ptx::cvt_f16x2_e4m3x2(static_cast<uint16_t>(w));
        hi = ptx::cvt_f16x2_e4m3x2(static_cast<uint16_t>(w >> 16));
    } else {
        lo = ptx::cvt_f16x2_e5m2x2(static_cast<uint16_t>(w));
        hi = ptx::cvt_f16x2_e5m2x2(static_cast<uint16_t>(w >> 16));
    }
    ptx::f16x2_to_f32(lo, f[0], f[1]);
    ptx::f16x2_to_f32(hi, f[2], f[3]);
}

// max(a, |b|), NaN if either is NaN.
__device__ __forceinline__ float max_abs_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(fabsf(b)));
    return r;
}

__device__ __forceinline__ float scale_mul(uint32_t b) {
    return (b == 0xFFu) ? __uint_as_float(0x7FC00000u) : pow2f(static_cast<int>(b) - 127);
}

template <int FIN, int FOUT>
__global__ void __launch_bounds__(256, 2) k_requant_t(const __grid_constant__ CUtensorMap tq,
                                                      const uint8_t *__restrict__ s, int64_t ld_s,
                                                      int scale_col_step, int tiles_x, int ntiles,
                                                      uint8_t *__restrict__ qt, int64_t ld_qt,
                                                      uint8_t *__restrict__ st, int64_t ld_st,
                                                      uint64_t wait_ns, int inject,
                                                      unsigned int *err) {
    extern __shared__ __align__(128) uint8_t rq_smem[];
    RqSmem &sm = *reinterpret_cast<RqSmem *>(rq_smem);
    const int tid = threadIdx.x;
    const int step = gridDim.x;
    const uint32_t fbar = ptx::smem_u32(&sm.full[0]);
    auto issue = [&](int tile, int stage) {
        const int bx = tile % tiles_x, by = tile / tiles_x;
        ptx::mbar_arrive_expect_tx(fbar + 8 * stage, kRqTileBytes);
        ptx::tma_load_2d(ptx::smem_u32(&sm.cin[stage][0][0]), &tq, fbar + 8 * stage, bx * kRQ,
                         by * kRQ);
    };
    auto scale_byte = [&](int tile) -> uint32_t {
        const int bx = tile % tiles_x, by = tile / tiles_x;
        return s[(static_cast<int64_t>(by) * kRQ + tid) * ld_s +
                 static_cast<int64_t>(bx) * scale_col_step];
    };
    // inject = 1 (a test of the timeout path): CTA 0 never issues the copy of
    // its first tile, so the wait for it can only run out.
    const bool withhold_first = inject == 1 && blockIdx.x == 0;
    int issued = 0;  // tiles whose copy thread 0 has issued (or withheld)
    if (tid == 0) {
        ptx::prefetch_tmap(&tq);
        for (int i = 0; i < kRqStages; ++i) ptx::mbar_init(fbar + 8 * i, 1);
        ptx::fence_mbar_init();
        for (int i = 0; i < kRqStages; ++i) {
            const int tile = blockIdx.x + i * step;
            if (tile >= ntiles) break;
            if (!(i == 0 && withhold_first)) issue(tile, i);
            ++issued;
        }
    }
    uint32_t sb = (tid < kRQ && static_cast<int>(blockIdx.x) < ntiles) ? scale_byte(blockIdx.x) : 0u;
    __syncthreads();
    const int cq = tid & 31, tg = tid >> 5;
    int k = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += step, ++k) {
        const int stage = k % kRqStages;
        const int bx = tile % tiles_x, by = tile / tiles_x;
        if (tid < kRQ) {
            sm.mul_in[tid] = scale_mul(sb);
            if (tile + step < ntiles) sb = scale_byte(tile + step);   // one tile ahead
        }
        if (tid == 0) {
            const uint32_t bar = fbar + 8 * stage, parity = static_cast<uint32_t>(k / kRqStages) & 1u;
            bool ok = ptx::mbar_try_wait(bar, parity);
            if (!ok) {
                const uint64_t t0 = ptx::globaltimer();
                while (!(ok = ptx::mbar_try_wait(bar, parity)))
                    if (ptx::globaltimer() - t0 > wait_ns) break;
            }
            sm.ok = ok;
        }
        __syncthreads();                                           // (A)
        if (!sm.ok) break;
        uint32_t w[16];
        float amax[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int t = 16 * tg + i;
            w[i] = sm.cin[stage][t][cq];
            const float mi = sm.mul_in[t];
            float f[4];
            decode4<FIN>(w[i], f);
#pragma unroll
            for (int j = 0; j < 4; ++j) amax[j] = max_abs_nan(amax[j], f[j] * mi);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) sm.red[tg][4 * cq + j] = amax[j];
        __syncthreads();                                           // (B) stage consumed
        if (tid == 0 && tile + kRqStages * step < ntiles) {
            issue(tile + kRqStages * step, stage);
            ++issued;
        }
        if (tid < kRQ) {
            float m = sm.red[0][tid];
#pragma unroll
            for (int r = 1; r < 8; ++r) m = max_abs_nan(m, sm.red[r][tid]);
            const uint32_t mb = __float_as_uint(m);
            const bool nonfinite = mb >= 0x7F800000u;
            const int e = nonfinite ? 128 : ue8m0_exponent_f32<FOUT>(mb);
            sm.mul_out[tid] = nonfinite ? 0.0f : pow2f(-e);
            sm.nan_col[tid] = nonfinite;
            st[(static_cast<int64_t>(bx) * kRQ + tid) * ld_st + by] = static_cast<uint8_t>(e + 127);
        }
        __syncthreads();                                           // (C)
        float mo[4];
        uint32_t out[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) mo[j] = sm.mul_out[4 * cq + j];
#pragma unroll
        for (int p = 0; p < 8; ++p) {       // token pairs (16tg + 2p, 16tg + 2p + 1)
            const int t = 16 * tg + 2 * p;
            const float ma = sm.mul_in[t], mb = sm.mul_in[t + 1];
            float a[4], b[4];
            decode4<FIN>(w[2 * p], a);
            decode4<FIN>(w[2 * p + 1], b);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t pair = cvt2<FOUT>((a[j] * ma) * mo[j], (b[j] * mb) * mo[j]);
                if (p & 1) out[j][p >> 1] |= pair << 16;
                else out[j][p >> 1] = pair;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = 4 * cq + j;
            const uint4 v = sm.nan_col[c] ? make_uint4(kNanCodes, kNanCodes, kNanCodes, kNanCodes)
                                          : make_uint4(out[j][0], out[j][1], out[j][2], out[j][3]);
            sm.cout[c][tg ^ (cq & 7)] = v;  // row c = 4cq + j, so (c >> 2) & 7 == cq & 7
        }
        __syncthreads();                                           // (D)
        const int64_t r0 = static_cast<int64_t>(by) * kRQ, c0 = static_cast<int64_t>(bx) * kRQ;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = tid + 256 * i;
            const int row = idx >> 3, ch = idx & 7;
            *reinterpret_cast<uint4 *>(qt + (c0 + row) * ld_qt + r0 + ch * 16) =
                sm.cout[row][ch ^ ((row >> 2) & 7)];
        }
    }
    if (tid == 0 && k < issued) {
        // a copy ran out of time: record it and wait (bounded) for the copies
        // still in flight before the CTA's shared memory is released
        atomicOr(err, 4u);
        for (int j = k; j < issued; ++j) {
            if (j == 0 && withhold_first) continue;   // never issued
            const uint32_t bar = fbar + 8 * (j % kRqStages);
            const uint32_t parity = static_cast<uint32_t>(j / kRqStages) & 1u;
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(bar, parity))
                if (ptx::globaltimer() - t0 > kRqWaitNs) break;
        }
    }
}

// ------------------------------------------------------------ 128x128 blocks
// 4x4 byte transpose of four 32-bit rows: result word j = byte j of each row.
__device__ __forceinline__ void transpose4x4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t (&c)[4]) {
    const uint32_t t0 = __byte_perm(a0, a1, 0x5140), t1 = __byte_perm(a0, a1, 0x7362);
    const uint32_t t2 = __byte_perm(a2, a3, 0x5140), t3 = __byte_perm(a2, a3, 0x7362);
    c[0] = __byte_perm(t0, t2, 0x5410);
    c[1] = __byte_perm(t0, t2, 0x7632);
    c[2] = __byte_perm(t1, t3, 0x5410);
    c[3] = __byte_perm(t1, t3, 0x7632);
}

// One CTA per 128x128 block (rb, cb); thread (rsub, csub) owns an 8x8
// sub-block.
template <int FMT, bool TRANS, int SM>
__device__ __forceinline__ void block128_body(const uint16_t *__restrict__ x, int64_t ld_x,
                                              uint8_t *__restrict__ q, int64_t ld_q,
                                              uint8_t *__restrict__ s, int64_t ld_s,
                                              uint8_t *__restrict__ qt, int64_t ld_qt,
                                              uint8_t *__restrict__ st, int64_t ld_st,
                                              int64_t rb, int64_t cb) {
    __shared__ uint32_t red[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rsub = tid >> 4, csub = tid & 15;
    const int64_t r_first = rb * 128 + rsub * 8, c_first = cb * 128 + csub * 8;
    const uint16_t *xb = x + r_first * ld_x + c_first;
    uint4 v[8];
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = ptx::ld_stream_v4(xb + i * ld_x);
        m = max(m, bf16_abs_max8(v[i]));
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) m = max(m, red[i]);
    const GroupScale<FMT, SM> gs(m);
    uint2 o[8];
    uint32_t unused = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        o[i] = gs.nan ? make_uint2(kNanCodes, kNanCodes)
                      : quant8<FMT, false>(v[i], gs.mul, unused);
        *reinterpret_cast<uint2 *>(q + (r_first + i) * ld_q + c_first) = o[i];
    }
    if (tid == 0) {
        gs.store(s, rb * ld_s + cb);
        if constexpr (TRANS) gs.store(st, cb * ld_st + rb);
    }
    if constexpr (TRANS) {
        // The transposed block is assembled in shared memory (8-byte units
        // XOR-swizzled by row group) and written as whole 128-byte rows; each
        // thread's own transposed 8x8 would otherwise go out as 8-byte pieces
        // scattered over 8 rows.
        __shared__ __align__(16) uint8_t tile_t[128 * 128];
        uint32_t lo03[4], lo47[4], hi03[4], hi47[4];
        transpose4x4(o[0].x, o[1].x, o[2].x, o[3].x, lo03);
        transpose4x4(o[4].x, o[5].x, o[6].x, o[7].x, lo47);
        transpose4x4(o[0].y, o[1].y, o[2].y, o[3].y, hi03);
        transpose4x4(o[4].y, o[5].y, o[6].y, o[7].y, hi47);
        // output row csub*8 + j of the tile, 8-byte unit rsub (tokens rsub*8..+7)
        const int unit = rsub ^ csub;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            *reinterpret_cast<uint2 *>(tile_t + (csub * 8 + j) * 128 + unit * 8) = make_uint2(lo03[j], lo47[j]);
            *reinterpret_cast<uint2 *>(tile_t + (csub * 8 + j + 4) * 128 + unit * 8) = make_uint2(hi03[j], hi47[j]);
        }
        __syncthreads();
        const int64_t r0 = rb * 128, c0 = cb * 128;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = tid + 256 * i, row = idx >> 3, c16 = idx & 7, g = row >> 3;
            const uint2 a = *reinterpret_cast<const uint2 *>(tile_t + row * 128 + ((2 * c16) ^ g) * 8);
            const uint2 b = *reinterpret_cast<const uint2 *>(tile_t + row * 128 + ((2 * c16 + 1) ^ g) * 8);
            *reinterpret_cast<uint4 *>(qt + (c0 + row) * ld_qt + r0 + c16 * 16) = make_uint4(a.x, a.y, b.x, b.y);
        }
    }
}

template <int FMT, bool TRANS, int SM>
__global__ void __launch_bounds__(256) k_quant_block128(const uint16_t *__restrict__ x,
                                                        int64_t ld_x, uint8_t *__restrict__ q,
                                                        int64_t ld_q, uint8_t *__restrict__ s,
                                                        int64_t ld_s, uint8_t *__restrict__ qt,
                                                        int64_t ld_qt, uint8_t *__restrict__ st,
                                                        int64_t ld_st) {
    block128_body<FMT, TRANS, SM>(x, ld_x, q, ld_q, s, ld_s, qt, ld_qt, st, ld_st, blockIdx.y,
                                  blockIdx.x);
}

// Several tensors' 128x128 blocks in one grid: CTA b belongs to the last job
// whose first block is <= b, and takes that job's block b - first (row-major
// over the job's block grid).
template <int FMT, bool TRANS, int SM>
__global__ void __launch_bounds__(256) k_quant_block128_batch(const __grid_constant__ Block128Batch bt) {
    int j = bt.n - 1;
    while (j > 0 && static_cast<int64_t>(blockIdx.x) < bt.job[j].first) --j;
    const Block128Job &jb = bt.job[j];
    const int64_t local = static_cast<int64_t>(blockIdx.x) - jb.first;
    block128_body<FMT, TRANS, SM>(jb.x, jb.ld_x, jb.q, jb.ld_q, jb.s, jb.ld_s, jb.qt, jb.ld_qt,
                                  jb.st, jb.ld_st, local / jb.cbs, local % jb.cbs);
}

// ------------------------------------------------------------------ launchers
TensorMapEncodeFn tensor_map_encoder() {
    static TensorMapEncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult res;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &res) == cudaSuccess &&
            res == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<TensorMapEncodeFn>(ptr);
    });
    return fn;
}

namespace {
// Per-device caches, filled on first use; concurrent first uses write the
// same values.
std::atomic<int> g_num_sms[64];

int num_sms() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    int n = g_num_sms[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
        g_num_sms[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

template <typename K>
int resident_blocks(K kernel, int threads) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1)
        n = 1;
    return n;
}

template <int FMT, int SM, int GV = 0, bool COUNT = false>
cudaError_t launch_row_regs(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t *q,
                       int64_t ld_q, uint8_t *s, int64_t ld_s, cudaStream_t stream,
                       unsigned long long *cnt = nullptr) {
    const int nvec = static_cast<int>(cols / 8);
    // Vectors per thread NV and threads T (T * NV covers the row, T <= 512):
    // the largest NV that keeps at least 96 threads per row and wastes at
    // most an eighth of the CTA's slots (fewer threads per row: more rows
    // resident per SM, more bytes in flight); failing that, the least waste.
    const int nvs[5] = {16, 8, 4, 2, 1};
    int best_nv = -1, best_t = 0;
    for (int k = 0; k < 5; ++k) {
        const int nv = nvs[k];
        int t = (nvec + nv - 1) / nv;
        t = ((t + 31) / 32) * 32;
        if (t > 512) continue;
        if (t < 96 && nv > 1) continue;
        const int64_t waste = static_cast<int64_t>(t) * nv - nvec;
        if (waste <= nvec / 8) {
            best_nv = nv;
            best_t = t;
            break;
        }
    }
    if (best_nv < 0) {
        int64_t best_waste = -1;
        for (int k = 0; k < 5; ++k) {
            const int nv = nvs[k];
            int t = (nvec + nv - 1) / nv;
            t = ((t + 31) / 32) * 32;
            if (t > 512) continue;
            const int64_t waste = static_cast<int64_t>(t) * nv - nvec;
            if (best_nv < 0 || waste < best_waste) {
                best_nv = nv;
                best_t = t;
                best_waste = waste;
            }
        }
    }
    const dim3 grid(static_cast<unsigned>(rows));
    if (best_nv < 0) {
        if (GV != 0) return cudaErrorInvalidValue;   // callers send only rows of at most 8 KB
        k_quant_row_2pass<FMT, SM><<<grid, 512, 0, stream>>>(x, nvec, ld_x, q, ld_q, s, ld_s);
        return cudaGetLastError();
    }
    switch (best_nv) {
    case 1: k_quant_row_regs<FMT, 1, SM, GV, COUNT><<<grid, best_t, 0, stream>>>(x, nvec, ld_x, q, ld_q, s, ld_s, cnt); break;
    case 2: k_quant_row_regs<FMT, 2, SM, GV, COUNT><<<grid, best_t, 0, stream>>>(x, nvec, ld_x, q, ld_q, s, ld_s, cnt); break;
    case 4: k_quant_row_regs<FMT, 4, SM, GV, COUNT><<<grid, best_t, 0, stream>>>(x, nvec, ld_x, q, ld_q, s, ld_s, cnt); break;
    case 8: k_quant_row_regs<FMT, 8, SM, GV, COUNT><<<grid, best_t, 0, stream>>>(x, nvec, ld_x, q, ld_q, s, ld_s, cnt); break;
    default: k_quant_row_regs<FMT, 16, SM, GV, COUNT><<<grid, best_t, 0, stream>>>(x, nvec, ld_x, q, ld_q, s, ld_s, cnt); break;
    }
    return cudaGetLastError();
}

template <int FMT, int SM>
cudaError_t launch_row(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t *q,
                       int64_t ld_q, uint8_t *s, int64_t ld_s, const WaitOpts &w,
                       cudaStream_t stream) {
    const int nvec = static_cast<int>(cols / 8);
    const int64_t row_bytes = cols * 2;
    if (row_bytes <= 8192) return launch_row_regs<FMT, SM>(x, rows, cols, ld_x, q, ld_q, s, ld_s, stream);
    // Several CTAs per SM (up to 4, at least 2 row slots each, at most 8),
    // ~200 KB of rows per SM in total: one CTA's per-row synchronisation then
    // overlaps the others' work.  For 37 KB rows two CTAs with two slots
    // each beat one CTA with five (6.2 vs 5.5 TB/s).
    int64_t per_sm = kRowSmemBudget / (2 * row_bytes);
    const int ctas_per_sm = static_cast<int>(per_sm < 1 ? 1 : (per_sm > 4 ? 4 : per_sm));
    int nslots = static_cast<int>(kRowSmemBudget / ctas_per_sm / row_bytes);
    if (nslots > kMaxRowSlots) nslots = kMaxRowSlots;
    if (nslots < 2) {
        // rows too long to stage two at a time: amax pass + cast pass
        k_quant_row_2pass<FMT, SM><<<static_cast<unsigned>(rows), 512, 0, stream>>>(x, nvec, ld_x, q,
                                                                                    ld_q, s, ld_s);
        return cudaGetLastError();
    }
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    static std::atomic<bool> attr_set[64];   // one flag per device and instantiation
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(k_quant_row<FMT, SM>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   kRowSmemBudget);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    int64_t grid = static_cast<int64_t>(num_sms()) * ctas_per_sm;
    if (grid > rows) grid = rows;
    int threads = kRowThreads;
    if (nvec < threads) threads = ((nvec + 31) / 32) * 32;
    unsigned int *err = device_error_word();
    if (!err) return cudaErrorInvalidValue;
    k_quant_row<FMT, SM><<<static_cast<unsigned>(grid), threads, static_cast<size_t>(nslots) * row_bytes,
                       stream>>>(x, rows, nvec, ld_x, q, ld_q, s, ld_s, nslots,
                                 w.limit_ns ? w.limit_ns : kRowWaitNs, w.inject, err);
    return cudaGetLastError();
}

template <int FMT, int GV, int SM, bool COUNT, bool MON, int U, int D>
cudaError_t launch_groups_ud(const uint16_t *x, int64_t rows, int vpr, int64_t ld_x, uint8_t *q,
                             int64_t ld_q, uint8_t *s, int64_t ld_s, MxCounters cnt,
                             cudaStream_t stream, int64_t gx, int64_t gy) {
    k_quant_groups<FMT, GV, SM, COUNT, MON, U, D>
        <<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), 256, 0, stream>>>(
            x, rows, vpr, ld_x, q, ld_q, s, ld_s, cnt);
    return cudaGetLastError();
}

// Grid: enough CTAs for every SM's resident slots.  Two rows in flight per
// CTA, except for the monitor variant when its CTAs have many rows each (its
// extra registers cost more occupancy than the deeper prefetch gains there).
template <int FMT, int GV, int SM, bool COUNT, bool MON, int U>
cudaError_t launch_groups_u(const uint16_t *x, int64_t rows, int vpr, int64_t ld_x, uint8_t *q,
                            int64_t ld_q, uint8_t *s, int64_t ld_s, MxCounters cnt,
                            cudaStream_t stream) {
    const int gx = (vpr + 256 * U - 1) / (256 * U);
    auto grid_y = [&](int res) {
        int64_t gy = (static_cast<int64_t>(num_sms()) * res + gx - 1) / gx;
        if (gy > rows) gy = rows;
        if (gy > 65535) gy = 65535;
        return gy < 1 ? int64_t(1) : gy;
    };
    const int64_t gy2 = grid_y(resident_blocks(k_quant_groups<FMT, GV, SM, COUNT, MON, U, 2>, 256));
    if (!MON || (rows + gy2 - 1) / gy2 <= 16)
        return launch_groups_ud<FMT, GV, SM, COUNT, MON, U, 2>(x, rows, vpr, ld_x, q, ld_q, s, ld_s,
                                                             cnt, stream, gx, gy2);
    const int64_t gy1 = grid_y(resident_blocks(k_quant_groups<FMT, GV, SM, COUNT, MON, U, 1>, 256));
    return launch_groups_ud<FMT, GV, SM, COUNT, MON, U, 1>(x, rows, vpr, ld_x, q, ld_q, s, ld_s, cnt,
                                                         stream, gx, gy1);
}

template <int FMT, int GV, int SM, bool COUNT, bool MON = false>
cudaError_t launch_groups(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t *q,
                          int64_t ld_q, uint8_t *s, int64_t ld_s, MxCounters cnt,
                          cudaStream_t stream) {
    const int vpr = static_cast<int>(cols / 8);
    // vectors per thread: the largest U (up to 4) that leaves no more than
    // an eighth of the CTA's slots in a row idle
    int u = 1;
    for (int cand : {4, 2}) {
        const int span = 256 * cand, gx = (vpr + span - 1) / span;
        if (static_cast<int64_t>(gx) * span - vpr <= vpr / 8) {
            u = cand;
            break;
        }
    }
    if (u == 4) return launch_groups_u<FMT, GV, SM, COUNT, MON, 4>(x, rows, vpr, ld_x, q, ld_q, s, ld_s, cnt, stream);
    if (u == 2) return launch_groups_u<FMT, GV, SM, COUNT, MON, 2>(x, rows, vpr, ld_x, q, ld_q, s, ld_s, cnt, stream);
    return launch_groups_u<FMT, GV, SM, COUNT, MON, 1>(x, rows, vpr, ld_x, q, ld_q, s, ld_s, cnt, stream);
}
}  // namespace

bool quant_token_waits(int64_t cols, int group, int transpose) {
    if (transpose || group != 0) return false;
    const int64_t row_bytes = cols * 2;
    if (row_bytes <= 8192) return false;
    int64_t per_sm = kRowSmemBudget / (2 * row_bytes);
    const int64_t ctas = per_sm < 1 ? 1 : (per_sm > 4 ? 4 : per_sm);
    return kRowSmemBudget / ctas / row_bytes >= 2;
}

cudaError_t launch_quant_token(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                               int group, int transpose, int fmt, uint8_t *q, int64_t ld_q,
                               uint8_t *s, int64_t ld_s, const WaitOpts &w, cudaStream_t stream) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    if (transpose) {
        const dim3 grid(static_cast<unsigned>(cols / kTC), static_cast<unsigned>(rows / 128));
        if (fmt == FMT_E4M3) k_quant_t<FMT_E4M3><<<grid, 256, 0, stream>>>(x, ld_x, q, ld_q, s, ld_s);
        else k_quant_t<FMT_E5M2><<<grid, 256, 0, stream>>>(x, ld_x, q, ld_q, s, ld_s);
        return cudaGetLastError();
    }
    if (group == 0) {
        return fmt == FMT_E4M3
                   ? launch_row<FMT_E4M3, SCALE_UE8M0>(x, rows, cols, ld_x, q, ld_q, s, ld_s, w, stream)
                   : launch_row<FMT_E5M2, SCALE_UE8M0>(x, rows, cols, ld_x, q, ld_q, s, ld_s, w, stream);
    }
    if (cols * 2 <= 8192)   // short rows: one row per CTA, held in registers
        return fmt == FMT_E4M3
                   ? launch_row_regs<FMT_E4M3, SCALE_UE8M0, 16>(x, rows, cols, ld_x, q, ld_q, s, ld_s, stream)
                   : launch_row_regs<FMT_E5M2, SCALE_UE8M0, 16>(x, rows, cols, ld_x, q, ld_q, s, ld_s, stream);
    const MxCounters none{nullptr, nullptr, nullptr};
    return fmt == FMT_E4M3
               ? launch_groups<FMT_E4M3, 16, SCALE_UE8M0, false>(x, rows, cols, ld_x, q, ld_q, s, ld_s,
                                                           none, stream)
               : launch_groups<FMT_E5M2, 16, SCALE_UE8M0, false>(x, rows, cols, ld_x, q, ld_q, s, ld_s,
                                                           none, stream);
}

cudaError_t launch_quant_mx32(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                              uint8_t *q, int64_t ld_q, uint8_t *s, int64_t ld_s,
                              unsigned long long *cnt, cudaStream_t stream) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    const MxCounters c{cnt, nullptr, nullptr};
    if (cnt && cols * 2 <= 8192)   // short rows with the clamp count
        return fmt == FMT_E4M3
                   ? launch_row_regs<FMT_E4M3, SCALE_MX, 4, true>(x, rows, cols, ld_x, q, ld_q, s, ld_s,
                                                                stream, cnt)
                   : launch_row_regs<FMT_E5M2, SCALE_MX, 4, true>(x, rows, cols, ld_x, q, ld_q, s, ld_s,
                                                                stream, cnt);
    if (cnt) {
        return fmt == FMT_E4M3
                   ? launch_groups<FMT_E4M3, 4, SCALE_MX, true>(x, rows, cols, ld_x, q, ld_q, s, ld_s,
                                                            c, stream)
                   : launch_groups<FMT_E5M2, 4, SCALE_MX, true>(x, rows, cols, ld_x, q, ld_q, s, ld_s,
                                                            c, stream);
    }
    if (cols * 2 <= 8192)   // short rows: one row per CTA, held in registers
        return fmt == FMT_E4M3
                   ? launch_row_regs<FMT_E4M3, SCALE_MX, 4>(x, rows, cols, ld_x, q, ld_q, s, ld_s, stream)
                   : launch_row_regs<FMT_E5M2, SCALE_MX, 4>(x, rows, cols, ld_x, q, ld_q, s, ld_s, stream);
    return fmt == FMT_E4M3
               ? launch_groups<FMT_E4M3, 4, SCALE_MX, false>(x, rows, cols, ld_x, q, ld_q, s, ld_s,
                                                         c, stream)
               : launch_groups<FMT_E5M2, 4, SCALE_MX, false>(x, rows, cols, ld_x, q, ld_q, s, ld_s,
                                                         c, stream);
}

cudaError_t launch_quant_mx32_monitor(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                                      int fmt, uint8_t *q, int64_t ld_q, uint8_t *s, int64_t ld_s,
                                      unsigned long long *stats, unsigned int *row_sat,
                                      cudaStream_t stream) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    const MxCounters c{nullptr, stats, row_sat};
    return fmt == FMT_E4M3
               ? launch_groups<FMT_E4M3, 4, SCALE_MX, false, true>(x, rows, cols, ld_x, q, ld_q, s,
                                                               ld_s, c, stream)
               : launch_groups<FMT_E5M2, 4, SCALE_MX, false, true>(x, rows, cols, ld_x, q, ld_q, s,
                                                               ld_s, c, stream);
}

cudaError_t launch_requant_t(const uint8_t *q, int64_t rows, int64_t cols, int64_t ld_q,
                             const uint8_t *s, int64_t ld_s, int per_token, int fmt_in,
                             int fmt_out, uint8_t *qt, int64_t ld_qt, uint8_t *st, int64_t ld_st,
                             const WaitOpts &w, cudaStream_t stream) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    CUtensorMap tq;
    std::memset(&tq, 0, sizeof(tq));
    TensorMapEncodeFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_q)};
    const cuuint32_t box[2] = {kRQ, kRQ};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(q), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    unsigned int *err = device_error_word();
    if (!err) return cudaErrorInvalidValue;
    const int tiles_x = static_cast<int>(cols / kRQ);
    const int64_t ntiles64 = (rows / kRQ) * static_cast<int64_t>(tiles_x);
    if (ntiles64 > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const int ntiles = static_cast<int>(ntiles64);
    const int step = per_token ? 0 : 1;
    const size_t smem = sizeof(RqSmem);
    auto run = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem);
        if (e != cudaSuccess) return e;
        int64_t grid = static_cast<int64_t>(num_sms()) * (per_sm > 0 ? per_sm : 1);
        if (grid > ntiles) grid = ntiles;
        kern<<<static_cast<unsigned>(grid), 256, smem, stream>>>(
            tq, s, ld_s, step, tiles_x, ntiles, qt, ld_qt, st, ld_st,
            w.limit_ns ? w.limit_ns : kRqWaitNs, w.inject, err);
        return cudaGetLastError();
    };
    if (fmt_in == FMT_E4M3)
        return fmt_out == FMT_E4M3 ? run(k_requant_t<FMT_E4M3, FMT_E4M3>)
                                   : run(k_requant_t<FMT_E4M3, FMT_E5M2>);
    return fmt_out == FMT_E4M3 ? run(k_requant_t<FMT_E5M2, FMT_E4M3>)
                               : run(k_requant_t<FMT_E5M2, FMT_E5M2>);
}

namespace {
template <int FMT, int SM>
void launch_block128_t(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, uint8_t *q,
                       int64_t ld_q, uint8_t *s, int64_t ld_s, uint8_t *qt, int64_t ld_qt,
                       uint8_t *st, int64_t ld_st, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(cols / 128), static_cast<unsigned>(rows / 128));
    if (qt)
        k_quant_block128<FMT, true, SM><<<grid, 256, 0, stream>>>(x, ld_x, q, ld_q, s, ld_s, qt,
                                                                  ld_qt, st, ld_st);
    else
        k_quant_block128<FMT, false, SM><<<grid, 256, 0, stream>>>(x, ld_x, q, ld_q, s, ld_s,
                                                                   nullptr, 0, nullptr, 0);
}
}  // namespace

cudaError_t launch_quant_block128(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                                  int fmt, uint8_t *q, int64_t ld_q, uint8_t *s, int64_t ld_s,
                                  uint8_t *qt, int64_t ld_qt, uint8_t *st, int64_t ld_st,
                                  cudaStream_t stream) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    if (fmt == FMT_E4M3)
        launch_block128_t<FMT_E4M3, SCALE_UE8M0>(x, rows, cols, ld_x, q, ld_q, s, ld_s, qt, ld_qt,
                                                 st, ld_st, stream);
    else
        launch_block128_t<FMT_E5M2, SCALE_UE8M0>(x, rows, cols, ld_x, q, ld_q, s, ld_s, qt, ld_qt,
                                                 st, ld_st, stream);
    return cudaGetLastError();
}

cudaError_t launch_quant_block128_batch(const Block128Batch &b, int64_t blocks, int fmt, bool trans,
                                        cudaStream_t stream) {
    if (b.n == 0 || blocks == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>(blocks));
    if (fmt == FMT_E4M3) {
        if (trans) k_quant_block128_batch<FMT_E4M3, true, SCALE_UE8M0><<<grid, 256, 0, stream>>>(b);
        else k_quant_block128_batch<FMT_E4M3, false, SCALE_UE8M0><<<grid, 256, 0, stream>>>(b);
    } else {
        if (trans) k_quant_block128_batch<FMT_E5M2, true, SCALE_UE8M0><<<grid, 256, 0, stream>>>(b);
        else k_quant_block128_batch<FMT_E5M2, false, SCALE_UE8M0><<<grid, 256, 0, stream>>>(b);
    }
    return cudaGetLastError();
}

// FP32-scale variant: per token (group 0) or 1x128 (group 128), and
// 128x128 blocks; scales are floats (ld in floats).
cudaError_t launch_quant_token_f32s(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                                    int group, int fmt, uint8_t *q, int64_t ld_q, float *sf,
                                    int64_t ld_s, cudaStream_t stream) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    uint8_t *s = reinterpret_cast<uint8_t *>(sf);
    if (group == 0)
        return fmt == FMT_E4M3
                   ? launch_row<FMT_E4M3, SCALE_F32>(x, rows, cols, ld_x, q, ld_q, s, ld_s, WaitOpts{}, stream)
                   : launch_row<FMT_E5M2, SCALE_F32>(x, rows, cols, ld_x, q, ld_q, s, ld_s, WaitOpts{}, stream);
    if (cols * 2 <= 8192)
        return fmt == FMT_E4M3
                   ? launch_row_regs<FMT_E4M3, SCALE_F32, 16>(x, rows, cols, ld_x, q, ld_q, s, ld_s, stream)
                   : launch_row_regs<FMT_E5M2, SCALE_F32, 16>(x, rows, cols, ld_x, q, ld_q, s, ld_s, stream);
    const MxCounters none{nullptr, nullptr, nullptr};
    return fmt == FMT_E4M3
               ? launch_groups<FMT_E4M3, 16, SCALE_F32, false>(x, rows, cols, ld_x, q, ld_q, s,
                                                               ld_s, none, stream)
               : launch_groups<FMT_E5M2, 16, SCALE_F32, false>(x, rows, cols, ld_x, q, ld_q, s,
                                                               ld_s, none, stream);
}

cudaError_t launch_quant_block128_f32s(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x,
                                       int fmt, uint8_t *q, int64_t ld_q, float *s, int64_t ld_s,
                                       uint8_t *qt, int64_t ld_qt, float *st, int64_t ld_st,
                                       cudaStream_t stream) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    uint8_t *sb = reinterpret_cast<uint8_t *>(s), *stb = reinterpret_cast<uint8_t *>(st);
    if (fmt == FMT_E4M3)
        launch_block128_t<FMT_E4M3, SCALE_F32>(x, rows, cols, ld_x, q, ld_q, sb, ld_s, qt, ld_qt,
                                               stb, ld_st, stream);
    else
        launch_block128_t<FMT_E5M2, SCALE_F32>(x, rows, cols, ld_x, q, ld_q, sb, ld_s, qt, ld_qt,
                                               stb, ld_st, stream);
    return cudaGetLastError();
}

}  // namespace fp8hg
