// Block-scaled FP8 GEMM on the 5th-generation tensor cores (tcgen05).
//
//   C[M, N] (+)= A[M, K] * B[N, K]^T,  A and B FP8 (E4M3 / E5M2), K-contiguous,
//   each element carrying a UE8M0 power-of-two scale.
//
// "A Comprehensive FP8 Training Recipe for Reasoning-Enhanced Language
// Models" ("What carries the argument", referee summary): the forward and
// backward GEMMs run on FP8 operands scaled per 128x128 weight block and per
// token (or 1x128 group) of the activations, with FP32 accumulation.
//
// Design (GB300, sm_103a):
//  * Every granularity becomes one UE8M0 scale per 32 K elements per row,
//    which is exactly the operand of tcgen05.mma.kind::mxf8f6f4.block_scale
//    (scale_vec::1X).  The scales are applied inside the MMA while it
//    accumulates into tensor memory in FP32: no CUDA-core promotion pass.
//      ROW      the row's byte repeated in all four 32-K slots
//      1x128    the group's byte; all four 32-K MMAs of a 128-K stage use it
//      128x128  the block's byte, the same for the tile's 128 rows
//      MX32     four distinct bytes per 128-K stage
//    The kernel reads the caller's compact scale arrays directly.  A scale
//    warp keeps, per row, four 32-bit scale words in registers and loads the
//    next group's words while it writes the current ones: for 1x128 and
//    128x128 a word holds the bytes of four consecutive 128-K blocks, so a
//    group spans 16 k-blocks of look-ahead; for MX32 a word holds the four
//    32-K slots of one block (groups of 4 k-blocks).  Per stage it writes the
//    words into the shared-memory layout tcgen05.cp expects; the MMA's
//    scale-factor id picks the byte of the word that belongs to the stage.
//  * Tile 128 x 256 x 128 (one CTA per SM, 4-stage TMA/mbarrier pipeline,
//    128-byte swizzled operand tiles), persistent over output tiles.
//  * Warp roles (256 threads): warp 0 TMA producer, warp 1 MMA issuer and
//    tensor-memory owner, warp 2 scale loader, warps 4-7 epilogue
//    (tensor memory -> registers -> BF16/FP32 global stores).
//  * Tensor memory (512 columns): accumulator in columns [0, 256), then per
//    pipeline stage 4 columns of A scales and 8 of B scales.
//  * Every wait is bounded (globaltimer); on expiry the kernel records a
//    timeout in the device error word, drains its in-flight copies and MMAs,
//    frees tensor memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"
#include "gemm_common.cuh"

namespace fp8hg {

__device__ unsigned int g_fp8hg_err[2];

namespace {

constexpr int BM = 128, BN = 256, BK = 128, STAGES = 4;
constexpr uint32_t A_TILE = BM * BK;  // bytes per stage
constexpr uint32_t B_TILE = BN * BK;
constexpr uint32_t SFA_TILE = 512;    // 128 rows x 4 scale bytes
constexpr uint32_t SFB_TILE = 1024;   // 256 rows x 4 scale bytes
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;
constexpr uint32_t SFA_COL = 256;                // + 4 * stage
constexpr uint32_t SFB_COL = 256 + 4 * STAGES;   // + 8 * stage
constexpr int NUM_THREADS = 256;

constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_TILE;
constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_TILE;
constexpr uint32_t OFF_SFB = OFF_SFA + STAGES * SFA_TILE;
constexpr uint32_t OFF_BAR = OFF_SFB + STAGES * SFB_TILE;
// Barriers (8 bytes each) from OFF_BAR: tma[STAGES] at 0 (the stage's operand
// bytes landed), empty[STAGES] at 32 (the MMAs that read the stage are done),
// tfull 64, tempty 72, drain 80, sf[STAGES] at 128 (the scale warp wrote the
// stage's scale words).  The operand copies and the scale words complete on
// separate barriers, so a CTA that stops early can wait for its own copies
// alone.
constexpr uint32_t BAR_SF = 128;
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + 96;
constexpr uint32_t OFF_ABORT = OFF_BAR + 100;
constexpr uint32_t OFF_EPI = OFF_BAR + 256;      // 4 KB per epilogue warp: store staging
constexpr uint32_t EPI_WARP_BYTES = 32 * 128;
constexpr uint32_t SMEM_USED = OFF_EPI + 4 * EPI_WARP_BYTES;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment

enum { GRAN_ROW = 0, GRAN_1x128 = 1, GRAN_128x128 = 2, GRAN_MX32 = 3 };
using gemm_common::tile_coords;
using gemm_common::desc_sw128;
using gemm_common::wait_phase;
enum { WHO_PRODUCER = 1, WHO_MMA = 2, WHO_SCALES = 3, WHO_EPILOGUE = 4 };

struct KParams {
    int M, N, nk, num_mb, num_nb, num_tiles;
    int gran_a, gran_b;
    int out_fp32, accumulate, inject;
    int out_q, fmt_c;
    uint8_t *cs;
    int64_t ld_cs;
    const uint8_t *sa, *sb;
    int64_t ld_sa, ld_sb;
    void *c;
    int64_t ldc;
    uint32_t idesc;
    uint64_t wait_limit_ns;
    unsigned int *err;
    // split-K (256 x 224 kernel only): each tile's K range in `split` parts,
    // work unit u = tile * split + j computing part split - 1 - j; parts >= 1
    // leave FP32 partial tiles in `ws`, part 0 adds them in part order.
    int split, num_units;
    float *ws;               // [num_tiles][split - 1][256][224] FP32
    unsigned int *flags;     // [num_tiles][8]: partial pieces written, per epilogue warp
};

// Bounded wait until *flag >= target, read with acquire.  Returns false if
// the CTA is aborting or the limit ran out (then the abort flag and the
// device error word are set, as by wait_phase).
__device__ bool wait_flag(const unsigned int *flag, uint32_t target, uint64_t limit,
                          volatile uint32_t *abort_flag, unsigned int *err) {
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v >= target) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > limit) {
            *abort_flag = 1u;
            atomicOr(err, 1u);
            atomicCAS(err + 1, 0u, static_cast<unsigned int>(WHO_EPILOGUE));
            return false;
        }
        __nanosleep(256);
    }
}

// Work unit -> (tile, part, k-block range [kb0, kb1)); without SPLIT a unit
// is a whole tile.
template <bool SPLIT>
__device__ __forceinline__ void unit_of(int u, const KParams &p, int &tile, int &part, int &kb0,
                                        int &kb1) {
    if constexpr (SPLIT) {
        tile = u / p.split;
        part = p.split - 1 - (u - tile * p.split);
        kb0 = part * p.nk / p.split;
        kb1 = (part + 1) * p.nk / p.split;
    } else {
        tile = u;
        part = 0;
        kb0 = 0;
        kb1 = p.nk;
    }
}

// Descriptor of a 32-row x 16-byte scale tile (no swizzle; 8-row core
// matrices of 128 contiguous bytes).
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}

// Loads issued where they stand in the program (asm volatile), so that the
// next group's scale words are in flight while the current group is written.
__device__ __forceinline__ uint32_t ld_u32_now(const uint8_t *p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_u8_now(const uint8_t *p) {
    uint16_t v;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// Scale words of one row for one group of G k-blocks (G = 16, or 4 for MX32):
// four 32-bit words at byte offsets 16*grp + 4t (t < 4) of the row's scales.
//   1x128 / 128x128 (G = 16): word t holds the bytes of k-blocks
//     16*grp + 4t .. +3; the MMA of k-block kb picks byte kb & 3.
//   MX32 (G = 4): word t holds the four 32-K slots of k-block 4*grp + t.
//   ROW: the row's single byte repeated, in every word.
// Words whose first k-block lies past K are not read (the row's scale bytes
// are padded to a multiple of four, not of sixteen).  Rows past the operand
// (B tail tile) get 2^0.
template <int G>
__device__ __forceinline__ void load_row_scales(const uint8_t *__restrict__ s, int64_t ld, int gran,
                                                int64_t r, int grp, int nk, bool valid,
                                                uint32_t (&w)[4]) {
    if (!valid) {
        w[0] = w[1] = w[2] = w[3] = 0x7F7F7F7Fu;
        return;
    }
    if (gran == GRAN_ROW) {
        w[0] = w[1] = w[2] = w[3] = ld_u8_now(s + r * ld) * 0x01010101u;
        return;
    }
    const uint8_t *row = (gran == GRAN_128x128) ? s + (r >> 7) * ld : s + r * ld;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int first_kb = (G == 4) ? 4 * grp + t : 16 * grp + 4 * t;
        w[t] = first_kb < nk ? ld_u32_now(row + 16 * grp + 4 * t) : 0x7F7F7F7Fu;
    }
}

// This lane's rows of a tile: A rows 32a + lane (a < 4), B rows 32h + lane (h < 8).
struct ScaleGroup {
    uint32_t a[4][4];
    uint32_t b[8][4];
};

template <int G>
__device__ __forceinline__ void load_group(ScaleGroup &g, const KParams &p, int tile, int grp,
                                           int lane) {
    int mb, nb;
    tile_coords(tile, p.num_mb, p.num_nb, mb, nb);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int64_t m = static_cast<int64_t>(mb) * BM + 32 * a + lane;
        load_row_scales<G>(p.sa, p.ld_sa, p.gran_a, m, grp, p.nk, true, g.a[a]);
    }
#pragma unroll
    for (int h = 0; h < 8; ++h) {
        const int64_t n = static_cast<int64_t>(nb) * BN + 32 * h + lane;
        load_row_scales<G>(p.sb, p.ld_sb, p.gran_b, n, grp, p.nk, n < p.N, g.b[h]);
    }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Coalesced store of a 32-row x 128-byte piece of the output through this
// warp's shared-memory staging area: lane l holds row l's 128 bytes; each
// global store instruction then writes four whole 128-byte row segments
// instead of 32 scattered 16-byte pieces.  The 16-byte chunks are
// XOR-swizzled by row so that neither the row writes nor the column reads
// conflict.
__device__ __forceinline__ void store_piece(uint8_t *stage, const uint4 (&v)[8], int lane,
                                            uint8_t *g_row0, int64_t ld_bytes) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4 *>(stage + lane * 128 + ((c ^ (lane & 7)) << 4)) = v[c];
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = i * 32 + lane, r = idx >> 3, c = idx & 7;
        *reinterpret_cast<uint4 *>(g_row0 + r * ld_bytes + c * 16) =
            *reinterpret_cast<const uint4 *>(stage + r * 128 + ((c ^ (r & 7)) << 4));
    }
    __syncwarp();
}

// The reverse: a 32-row x 128-byte piece of C read with whole-segment loads;
// lane l receives row l's 128 bytes.
__device__ __forceinline__ void load_piece(uint8_t *stage, uint4 (&v)[8], int lane,
                                           const uint8_t *g_row0, int64_t ld_bytes) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = i * 32 + lane, r = idx >> 3, c = idx & 7;
        *reinterpret_cast<uint4 *>(stage + r * 128 + ((c ^ (r & 7)) << 4)) =
            *reinterpret_cast<const uint4 *>(g_row0 + r * ld_bytes + c * 16);
    }
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 8; ++c)
        v[c] = *reinterpret_cast<const uint4 *>(stage + lane * 128 + ((c ^ (lane & 7)) << 4));
    __syncwarp();
}

__device__ __forceinline__ uint32_t sf_id(int gran, int kb, int j) {
    return (gran == GRAN_1x128 || gran == GRAN_128x128) ? static_cast<uint32_t>(kb & 3)
                                                        : static_cast<uint32_t>(j);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// k-blocks that share one 32-bit scale word per row: four for 1x128 / 128x128
// scales (G = 16: a word holds four k-blocks' bytes), one for MX (G = 4: a
// word holds the four 32-K slots of one k-block).
template <int G>
__device__ __forceinline__ constexpr int kScaleGroupKb() { return G == 16 ? 4 : 1; }

// G: k-blocks per scale group (16, or 4 when the operands are MX32).
// OUTQ: the epilogue quantizes C (FP8, 1x128 along N) instead of storing it.
template <int G, bool OUTQ>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_mxf8(const __grid_constant__ CUtensorMap tmap_a,
                const __grid_constant__ CUtensorMap tmap_b, const KParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sA = base + OFF_A, sB = base + OFF_B;
    const uint32_t sSFA = base + OFF_SFA, sSFB = base + OFF_SFB, sBAR = base + OFF_BAR;
    const uint32_t tfull = sBAR + 64, tempty = sBAR + 72, drain = sBAR + 80;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + OFF_TMEM_SLOT);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + OFF_ABORT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t limit = p.wait_limit_ns;
    const uint64_t drain_limit = 2000000ull;  // 2 ms: copies and MMAs finish in microseconds

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(sBAR + 8 * s, 1);            // TMA expect_tx

            ptx::mbar_init(sBAR + 32 + 8 * s, 1);       // tcgen05.commit
        }
        for (int i = 0; i < STAGES; ++i) {
            ptx::mbar_init(sBAR + BAR_SF + 8 * i, 32);      // words written: one per scale-warp lane
            ptx::mbar_init(sBAR + BAR_SF + 32 + 8 * i, 1);  // words copied: tcgen05.commit
        }
        ptx::mbar_init(tfull, 1);
        ptx::mbar_init(tempty, 128);
        ptx::mbar_init(drain, 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmap_a);
        ptx::prefetch_tmap(&tmap_b);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, p.num_mb, p.num_nb, mb, nb);
            for (int kb = 0; kb < p.nk; ++kb) {
                const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                ok = wait_phase(sBAR + 32 + 8 * s, ph ^ 1u, limit, abort_flag, p.err, WHO_PRODUCER);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) break;
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(sBAR + 8 * s, A_TILE + B_TILE);
                    ptx::tma_load_2d(sA + s * A_TILE, &tmap_a, sBAR + 8 * s, kb * BK, mb * BM);
                    ptx::tma_load_2d(sB + s * B_TILE, &tmap_b, sBAR + 8 * s, kb * BK, nb * BN);
                }
                __syncwarp();
                ++it;
            }
        }
        // wait for the last loads to land before the CTA may exit (the tma
        // barriers count the copies' bytes alone, not the scale arrivals)
        const uint32_t nd = it < static_cast<uint32_t>(STAGES) ? it : static_cast<uint32_t>(STAGES);
        for (uint32_t i = it - nd; i < it; ++i)
            wait_phase(sBAR + 8 * (i % STAGES), (i / STAGES) & 1u, drain_limit, abort_flag, p.err,
                       WHO_PRODUCER, false);
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        // scale words as in the 256 x 224 kernel: with 1x128 / 128x128 scales
        // one buffer of their own ring per four k-blocks, copied into one of
        // three tensor-memory slots once; MX words ride with the stage
        uint32_t it = 0, tcount = 0, sfi = 0, tslot = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
            ok = wait_phase(tempty, (tcount & 1u) ^ 1u, limit, abort_flag, p.err, WHO_MMA);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            for (int kb = 0; kb < p.nk; ++kb) {
                const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                const bool new_group = kb % kScaleGroupKb<G>() == 0;
                const uint32_t sl = G == 16 ? sfi % STAGES : s;
                const uint32_t sph = G == 16 ? (sfi / STAGES) & 1u : ph;
                ok = wait_phase(sBAR + 8 * s, ph, limit, abort_flag, p.err, WHO_MMA) &&
                     (!new_group ||
                      wait_phase(sBAR + BAR_SF + 8 * sl, sph, limit, abort_flag, p.err, WHO_MMA));
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) break;
                ptx::tc_fence_after();
                if (new_group) tslot = G == 16 ? sfi % 3 : s;
                if (lane == 0) {
                    const uint32_t tsfa = tmem + SFA_COL + 4 * tslot;
                    const uint32_t tsfb = tmem + SFB_COL + 8 * tslot;
                    if (new_group) {
                        ptx::tc_cp_32x128b_warpx4(tsfa, desc_sf(sSFA + sl * SFA_TILE));
                        ptx::tc_cp_32x128b_warpx4(tsfb, desc_sf(sSFB + sl * SFB_TILE));
                        ptx::tc_cp_32x128b_warpx4(tsfb + 4, desc_sf(sSFB + sl * SFB_TILE + 512));
                        if (G == 16) ptx::tc_commit(sBAR + BAR_SF + 32 + 8 * sl);   // buffer free
                    }
                    const uint64_t ad = desc_sw128(sA + s * A_TILE);
                    const uint64_t bd = desc_sw128(sB + s * B_TILE);
#pragma unroll
                    for (int j = 0; j < BK / 32; ++j) {
                        const uint32_t idesc = p.idesc | (sf_id(p.gran_a, kb, j) << 29) |
                                               (sf_id(p.gran_b, kb, j) << 4);
                        // +32 bytes along K inside the swizzled 128-byte rows
                        ptx::tc_mma_mxf8(tmem + ACC_COL, ad + 2 * j, bd + 2 * j, idesc, tsfa, tsfb,
                                         (kb | j) != 0 ? 1u : 0u);
                    }
                    ptx::tc_commit(sBAR + 32 + 8 * s);  // frees the smem stage when done
                }
                __syncwarp();
                if (new_group) ++sfi;
                ++it;
            }
            if (!ok) break;
            if (lane == 0) ptx::tc_commit(tfull);
            __syncwarp();
            ++tcount;
        }
        // all issued MMAs must finish before tensor memory is released
        if (lane == 0) ptx::tc_commit(drain);
        __syncwarp();
        wait_phase(drain, 0u, drain_limit, abort_flag, p.err, WHO_MMA, false);
    } else if (warp == 2) {
        // ------------------------------------------------------ scale loader
        // Walks the same (tile, k-block) sequence as the producer, one group
        // of G k-blocks at a time, with the next group's loads in flight.
        uint32_t it = 0;
        bool ok = true;
        const int ngrp = (p.nk + G - 1) / G;
        int tile = blockIdx.x, grp = 0;
        ScaleGroup cur, nxt;
        if (tile < p.num_tiles) load_group<G>(cur, p, tile, 0, lane);
        while (tile < p.num_tiles && ok) {
            int ntile = tile, ngrp_next = grp + 1;
            if (ngrp_next == ngrp) {
                ntile += gridDim.x;
                ngrp_next = 0;
            }
            if (ntile < p.num_tiles) load_group<G>(nxt, p, ntile, ngrp_next, lane);
#pragma unroll
            for (int t = 0; t < G; ++t) {
                if (G * grp + t >= p.nk || !ok) break;
                // one buffer per scale group (four k-blocks; MX: one)
                if ((G * grp + t) % kScaleGroupKb<G>() != 0) continue;
                constexpr int kWordStep = G / 4;  // k-blocks per scale word
                const int wi = t / kWordStep;
                // free once the MMA warp's copy of its previous group is done
                // (its own commit; MX: the operand stage's)
                const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                ok = wait_phase(sBAR + (G == 16 ? BAR_SF + 32 : 32) + 8 * s, ph ^ 1u, limit,
                                abort_flag, p.err, WHO_SCALES);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) break;
                // Row r = 32a + lane of a 128-row chunk goes to byte offset
                // lane*16 + a*4: the 32x128-bit layout tcgen05.cp broadcasts.
                const uint32_t dA = sSFA + s * SFA_TILE + lane * 16;
                const uint32_t dB = sSFB + s * SFB_TILE + lane * 16;
                st_shared_v4(dA, cur.a[0][wi], cur.a[1][wi], cur.a[2][wi], cur.a[3][wi]);
                st_shared_v4(dB, cur.b[0][wi], cur.b[1][wi], cur.b[2][wi], cur.b[3][wi]);
                st_shared_v4(dB + 512, cur.b[4][wi], cur.b[5][wi], cur.b[6][wi], cur.b[7][wi]);
                if (!(p.inject == 1 && it == 0)) {
                    ptx::fence_proxy_async_smem();  // make the words visible to tcgen05.cp
                    ptx::mbar_arrive(sBAR + BAR_SF + 8 * s);
                }
                ++it;
            }
            cur = nxt;
            tile = ntile;
            grp = ngrp_next;
        }
    } else if (warp >= 4) {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;  // tensor-memory lane quarter this warp may read
        uint8_t *stage = gbase + OFF_EPI + q * EPI_WARP_BYTES;
        uint32_t tcount = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, p.num_mb, p.num_nb, mb, nb);
            bool ok = wait_phase(tfull, tcount & 1u, limit, abort_flag, p.err, WHO_EPILOGUE);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const int64_t row = static_cast<int64_t>(mb) * BM + q * 32 + lane;
            const int64_t row0 = static_cast<int64_t>(mb) * BM + q * 32;  // this warp's first row
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + ACC_COL;
            if constexpr (OUTQ) {
                // FP8 out, one UE8M0 round-up scale per 128 columns of the row
                // (the next GEMM's 1x128 operand).  Pass 1 takes each group's
                // NaN-propagating amax (integer max of |value| patterns) from
                // tensor memory; pass 2 reads the accumulator again and casts.
                uint32_t am[BN / 128] = {};
#pragma unroll
                for (int g = 0; g < BN / 128; ++g) {
                    // a whole group's four loads in flight per wait
                    uint32_t r[4][32];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) ptx::tmem_ld_32x32b_x32(taddr + g * 128 + c4 * 32, r[c4]);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                        for (int e = 0; e < 32; ++e) am[g] = max(am[g], r[c4][e] & 0x7FFFFFFFu);
                }
                float mul[BN / 128];
                uint32_t sbyte[BN / 128];
#pragma unroll
                for (int g = 0; g < BN / 128; ++g) {
                    const bool nonfinite = am[g] >= 0x7F800000u;
                    const int e = nonfinite ? 128
                                  : (p.fmt_c == 0 ? ue8m0_exponent_f32<FMT_E4M3>(am[g])
                                                  : ue8m0_exponent_f32<FMT_E5M2>(am[g]));
                    mul[g] = nonfinite ? 0.0f : pow2f(-e);
                    sbyte[g] = static_cast<uint32_t>(e + 127);
                }
                uint32_t codes[BN / 4];
#pragma unroll
                for (int chunk = 0; chunk < BN / 32; chunk += 2) {
                    uint32_t r[2][32];
                    ptx::tmem_ld_32x32b_x32(taddr + chunk * 32, r[0]);
                    ptx::tmem_ld_32x32b_x32(taddr + chunk * 32 + 32, r[1]);
                    ptx::tmem_wait_ld();
                    const float m = mul[chunk / 4];
                    const bool nan_group = sbyte[chunk / 4] == 0xFFu;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            const float f0 = __uint_as_float(r[h][4 * v]) * m, f1 = __uint_as_float(r[h][4 * v + 1]) * m;
                            const float f2 = __uint_as_float(r[h][4 * v + 2]) * m, f3 = __uint_as_float(r[h][4 * v + 3]) * m;
                            const uint32_t lo = p.fmt_c == 0 ? ptx::cvt_e4m3x2(f0, f1) : ptx::cvt_e5m2x2(f0, f1);
                            const uint32_t hi = p.fmt_c == 0 ? ptx::cvt_e4m3x2(f2, f3) : ptx::cvt_e5m2x2(f2, f3);
                            codes[(chunk + h) * 8 + v] = nan_group ? kNanCodes : (lo | (hi << 16));
                        }
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(tempty);
#pragma unroll
                for (int g = 0; g < BN / 128; ++g) {
                    const int64_t n0 = static_cast<int64_t>(nb) * BN + g * 128;
                    if (n0 >= p.N) continue;
                    uint4 v[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        v[c] = make_uint4(codes[32 * g + 4 * c], codes[32 * g + 4 * c + 1],
                                          codes[32 * g + 4 * c + 2], codes[32 * g + 4 * c + 3]);
                    store_piece(stage, v, lane, static_cast<uint8_t *>(p.c) + row0 * p.ldc + n0, p.ldc);
                    p.cs[row * p.ld_cs + n0 / 128] = static_cast<uint8_t>(sbyte[g]);
                }
                ++tcount;
                continue;
            } else if (!p.out_fp32 && !p.accumulate) {
                // BF16 out: pull the whole accumulator row into registers
                // (packed BF16), release the accumulator to the next tile's
                // MMAs, then store while they run.
                uint32_t packed[BN / 2];
#pragma unroll
                for (int chunk = 0; chunk < BN / 32; chunk += 2) {
                    // two loads in flight per wait: the drain is latency-bound
                    uint32_t r[32], r2[32];
                    ptx::tmem_ld_32x32b_x32(taddr + chunk * 32, r);
                    ptx::tmem_ld_32x32b_x32(taddr + chunk * 32 + 32, r2);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        packed[chunk * 16 + e] =
                            ptx::cvt_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
                        packed[chunk * 16 + 16 + e] =
                            ptx::cvt_bf16x2(__uint_as_float(r2[2 * e]), __uint_as_float(r2[2 * e + 1]));
                    }
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(tempty);
#pragma unroll
                for (int pc = 0; pc < BN / 64; ++pc) {       // 64 BF16 columns = 128 bytes
                    const int64_t n0 = static_cast<int64_t>(nb) * BN + pc * 64;
                    if (n0 >= p.N) continue;
                    uint4 v[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        v[c] = make_uint4(packed[pc * 32 + 4 * c], packed[pc * 32 + 4 * c + 1],
                                          packed[pc * 32 + 4 * c + 2], packed[pc * 32 + 4 * c + 3]);
                    store_piece(stage, v, lane,
                                reinterpret_cast<uint8_t *>(static_cast<uint16_t *>(p.c) + row0 * p.ldc + n0),
                                p.ldc * 2);
                }
                ++tcount;
                continue;
            }
            // FP32 out, or accumulation into C: 64 columns at a time, the old
            // values read and the new ones written as whole 128-byte row
            // segments through the staging area; the accumulator is
            // released after its last columns are read.
#pragma unroll 1
            for (int pc = 0; pc < BN / 64; ++pc) {
                uint32_t r0[32], r1[32];
                ptx::tmem_ld_32x32b_x32(taddr + pc * 64, r0);
                ptx::tmem_ld_32x32b_x32(taddr + pc * 64 + 32, r1);
                ptx::tmem_wait_ld();
                if (pc == BN / 64 - 1) {
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(tempty);  // accumulator may be overwritten now
                }
                const int64_t n0 = static_cast<int64_t>(nb) * BN + pc * 64;
                if (n0 >= p.N) continue;
                if (p.out_fp32) {
                    auto piece = [&](const uint32_t(&rr)[32], int64_t col) {
                        uint8_t *g = reinterpret_cast<uint8_t *>(static_cast<float *>(p.c) + row0 * p.ldc + col);
                        uint4 v[8];
                        if (p.accumulate) {
                            load_piece(stage, v, lane, g, p.ldc * 4);
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                v[c] = make_uint4(__float_as_uint(__uint_as_float(rr[4 * c]) + __uint_as_float(v[c].x)),
                                                  __float_as_uint(__uint_as_float(rr[4 * c + 1]) + __uint_as_float(v[c].y)),
                                                  __float_as_uint(__uint_as_float(rr[4 * c + 2]) + __uint_as_float(v[c].z)),
                                                  __float_as_uint(__uint_as_float(rr[4 * c + 3]) + __uint_as_float(v[c].w)));
                        } else {
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                v[c] = make_uint4(rr[4 * c], rr[4 * c + 1], rr[4 * c + 2], rr[4 * c + 3]);
                        }
                        store_piece(stage, v, lane, g, p.ldc * 4);
                    };
                    piece(r0, n0);
                    piece(r1, n0 + 32);
                } else {
                    // BF16 with accumulation: add in FP32, round once
                    uint8_t *g = reinterpret_cast<uint8_t *>(static_cast<uint16_t *>(p.c) + row0 * p.ldc + n0);
                    uint4 v[8];
                    load_piece(stage, v, lane, g, p.ldc * 2);
                    auto add8 = [](const uint32_t *f32, const uint4 &old) {
                        return make_uint4(
                            ptx::cvt_bf16x2(__uint_as_float(f32[0]) + bf16_lo(old.x), __uint_as_float(f32[1]) + bf16_hi(old.x)),
                            ptx::cvt_bf16x2(__uint_as_float(f32[2]) + bf16_lo(old.y), __uint_as_float(f32[3]) + bf16_hi(old.y)),
                            ptx::cvt_bf16x2(__uint_as_float(f32[4]) + bf16_lo(old.z), __uint_as_float(f32[5]) + bf16_hi(old.z)),
                            ptx::cvt_bf16x2(__uint_as_float(f32[6]) + bf16_lo(old.w), __uint_as_float(f32[7]) + bf16_hi(old.w)));
                    };
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        v[c] = add8(r0 + 8 * c, v[c]);
                        v[c + 4] = add8(r1 + 8 * c, v[c + 4]);
                    }
                    store_piece(stage, v, lane, g, p.ldc * 2);
                }
            }
            ++tcount;
        }
    }

    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------- wide variant
// Tile 256 x 224: two M = 128 MMAs per k-step share each B tile, so every
// stage (A 32 KB + B 28 KB) feeds twice the flops of a 128 x 256 stage with
// 1.25x the bytes: 67 instead of 96 bytes per MMA cycle, for an operand feed
// that is bound by the latency of what it has in flight.  Both accumulators
// (2 x 224 columns) and the scale factors (3 stages x 16 columns) fill the
// 512 tensor-memory columns.  384 threads: warp 0 TMA producer, warp 1 MMA
// issuer, warps 2 and 3 scale loaders (A, B), warps 4-11 epilogue (two per
// 32-lane quarter, one per accumulator).  BF16 or FP32 output, with or without accumulation.
constexpr int WBM = 256, WBN = 224, WSTAGES = 3;
constexpr uint32_t WA_TILE = WBM * BK, WB_TILE = WBN * BK;
constexpr uint32_t WSF_TILE = 1024;  // 256 rows x 4 scale bytes (A, and B padded to 256)
constexpr uint32_t WACC1 = WBN;      // second accumulator's first column
constexpr uint32_t WSFA_COL = 2 * WBN;                 // + 8 * stage
constexpr uint32_t WSFB_COL = 2 * WBN + 8 * WSTAGES;   // + 8 * stage
constexpr int W_THREADS = 384;
constexpr uint32_t WOFF_A = 0;
constexpr uint32_t WOFF_B = WOFF_A + WSTAGES * WA_TILE;
constexpr int WNSF = 4;              // scale-word buffers, one per scale group
constexpr uint32_t WOFF_SFA = WOFF_B + WSTAGES * WB_TILE;
constexpr uint32_t WOFF_SFB = WOFF_SFA + WNSF * WSF_TILE;
constexpr uint32_t WOFF_BAR = WOFF_SFB + WNSF * WSF_TILE;
// barriers as in the 128 x 256 kernel: tma[3] at 0, empty[3] at 32, tfull 64,
// tempty 72, drain 80; scale words: full[4] at BAR_SF, empty[4] at BAR_SF + 32
constexpr uint32_t WOFF_TMEM_SLOT = WOFF_BAR + 96;
constexpr uint32_t WOFF_ABORT = WOFF_BAR + 100;
constexpr uint32_t WOFF_EPI = WOFF_BAR + 256;
constexpr uint32_t W_SMEM_BYTES = WOFF_EPI + 8 * EPI_WARP_BYTES + 1024;
static_assert(WSFB_COL + 8 * WSTAGES <= TMEM_COLS, "tensor memory overflow");
static_assert(W_SMEM_BYTES <= 232448, "shared memory overflow");

// One lane's scale words for one operand of a tile: A rows 32a + lane
// (a < 8, 256 rows) or B rows 32h + lane (h < 7, 224 rows; row 8 padding).
struct WScaleRows {
    uint32_t w[8][4];
};

template <int G, bool IS_A>
__device__ __forceinline__ void load_rows_wide(WScaleRows &g, const KParams &p, int tile, int grp,
                                               int lane) {
    int mb, nb;
    tile_coords(tile, p.num_mb, p.num_nb, mb, nb);
#pragma unroll
    for (int h = 0; h < 8; ++h) {
        if constexpr (IS_A) {
            const int64_t m = static_cast<int64_t>(mb) * WBM + 32 * h + lane;
            load_row_scales<G>(p.sa, p.ld_sa, p.gran_a, m, grp, p.nk, true, g.w[h]);
        } else {
            const int64_t n = static_cast<int64_t>(nb) * WBN + 32 * h + lane;
            load_row_scales<G>(p.sb, p.ld_sb, p.gran_b, n, grp, p.nk, h < 7 && n < p.N, g.w[h]);
        }
    }
}

// A piece of the wide kernel's packed BF16 rows (lane l: row l, words OFF ..
// OFF + W - 1 of its packed row; W = 32 for 64 columns, 16 for 32) written
// as whole row segments through the staging area.  The packed registers
// are read in place, so the piece needs no second copy of them.
template <int OFF, int W>
__device__ __forceinline__ void store_packed(uint8_t *stage, const uint32_t (&pk)[WBN / 2], int lane,
                                             uint8_t *g_row0, int64_t ld_bytes) {
    constexpr int V = W / 4;   // 16-byte chunks per row
#pragma unroll
    for (int c = 0; c < V; ++c)
        *reinterpret_cast<uint4 *>(stage + lane * 128 + ((c ^ (lane & 7)) << 4)) =
            make_uint4(pk[OFF + 4 * c], pk[OFF + 4 * c + 1], pk[OFF + 4 * c + 2], pk[OFF + 4 * c + 3]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int idx = i * 32 + lane, r = idx / V, c = idx % V;
        *reinterpret_cast<uint4 *>(g_row0 + r * ld_bytes + c * 16) =
            *reinterpret_cast<const uint4 *>(stage + r * 128 + ((c ^ (r & 7)) << 4));
    }
    __syncwarp();
}

// Columns col0 + PC * 64 .. + 63 of 224 packed BF16 columns (PC = 3: the
// last 32 columns).  N is a multiple of 128 and col0 a multiple of 32, so a
// 64-column piece can straddle N by exactly 32 columns: it is then written
// as a 32-column half piece.
template <int PC>
__device__ __forceinline__ void store_wide_piece(uint8_t *stage, const uint32_t (&pk)[WBN / 2], int lane,
                                                 const KParams &p, int64_t row0, int64_t col0) {
    const int64_t n0 = col0 + PC * 64;
    if (n0 >= p.N) return;
    uint8_t *g = reinterpret_cast<uint8_t *>(static_cast<uint16_t *>(p.c) + row0 * p.ldc + n0);
    if (PC < WBN / 64 && n0 + 64 <= p.N) store_packed<PC * 32, 32>(stage, pk, lane, g, p.ldc * 2);
    else store_packed<PC * 32, 16>(stage, pk, lane, g, p.ldc * 2);
}

// Half piece: 32 rows x 64 bytes through the staging area (lane l holds row
// l's four 16-byte chunks).
__device__ __forceinline__ void store_piece64(uint8_t *stage, const uint4 (&v)[4], int lane,
                                              uint8_t *g_row0, int64_t ld_bytes) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4 *>(stage + lane * 128 + ((c ^ (lane & 7)) << 4)) = v[c];
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = i * 32 + lane, r = idx >> 2, c = idx & 3;
        *reinterpret_cast<uint4 *>(g_row0 + r * ld_bytes + c * 16) =
            *reinterpret_cast<const uint4 *>(stage + r * 128 + ((c ^ (r & 7)) << 4));
    }
    __syncwarp();
}

__device__ __forceinline__ void load_piece64(uint8_t *stage, uint4 (&v)[4], int lane,
                                             const uint8_t *g_row0, int64_t ld_bytes) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = i * 32 + lane, r = idx >> 2, c = idx & 3;
        *reinterpret_cast<uint4 *>(stage + r * 128 + ((c ^ (r & 7)) << 4)) =
            *reinterpret_cast<const uint4 *>(g_row0 + r * ld_bytes + c * 16);
    }
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 4; ++c)
        v[c] = *reinterpret_cast<const uint4 *>(stage + lane * 128 + ((c ^ (lane & 7)) << 4));
    __syncwarp();
}

// SPLIT: the split-K instantiation (work units of one K part of a tile).
template <int G, bool SPLIT>
__global__ void __launch_bounds__(W_THREADS, 1)
    k_gemm_wide(const __grid_constant__ CUtensorMap tmap_a,
                const __grid_constant__ CUtensorMap tmap_b, const KParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sA = base + WOFF_A, sB = base + WOFF_B;
    const uint32_t sSFA = base + WOFF_SFA, sSFB = base + WOFF_SFB, sBAR = base + WOFF_BAR;
    const uint32_t tfull = sBAR + 64, tempty = sBAR + 72, drain = sBAR + 80;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + WOFF_TMEM_SLOT);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + WOFF_ABORT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t limit = p.wait_limit_ns;
    const uint64_t drain_limit = 2000000ull;

    if (threadIdx.x == 0) {
        for (int s = 0; s < WSTAGES; ++s) {
            ptx::mbar_init(sBAR + 8 * s, 1);            // TMA expect_tx
            ptx::mbar_init(sBAR + 32 + 8 * s, 1);       // tcgen05.commit
        }
        for (int i = 0; i < WNSF; ++i) {
            ptx::mbar_init(sBAR + BAR_SF + 8 * i, 64);      // words written: both scale warps' lanes
            ptx::mbar_init(sBAR + BAR_SF + 32 + 8 * i, 1);  // words copied: tcgen05.commit
        }
        ptx::mbar_init(tfull, 1);
        ptx::mbar_init(tempty, 256);
        ptx::mbar_init(drain, 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmap_a);
        ptx::prefetch_tmap(&tmap_b);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        uint32_t it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
            int tile, part, kb0, kb1, mb, nb;
            unit_of<SPLIT>(u, p, tile, part, kb0, kb1);
            tile_coords(tile, p.num_mb, p.num_nb, mb, nb);
            for (int kb = kb0; kb < kb1; ++kb) {
                const uint32_t s = it % WSTAGES, ph = (it / WSTAGES) & 1u;
                ok = wait_phase(sBAR + 32 + 8 * s, ph ^ 1u, limit, abort_flag, p.err, WHO_PRODUCER);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) break;
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(sBAR + 8 * s, WA_TILE + WB_TILE);
                    ptx::tma_load_2d(sA + s * WA_TILE, &tmap_a, sBAR + 8 * s, kb * BK, mb * WBM);
                    ptx::tma_load_2d(sB + s * WB_TILE, &tmap_b, sBAR + 8 * s, kb * BK, nb * WBN);
                }
                __syncwarp();
                ++it;
            }
        }
        const uint32_t nd = it < static_cast<uint32_t>(WSTAGES) ? it : static_cast<uint32_t>(WSTAGES);
        for (uint32_t i = it - nd; i < it; ++i)
            wait_phase(sBAR + 8 * (i % WSTAGES), (i / WSTAGES) & 1u, drain_limit, abort_flag, p.err,
                       WHO_PRODUCER, false);
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        // With 1x128 / 128x128 scales a row's 32-bit scale word holds four
        // k-blocks' bytes: the words come in groups of four k-blocks through
        // their own ring of WNSF buffers (the scale warps run up to WNSF
        // groups ahead of the MMAs, independently of the operand stages) and
        // each group is copied into one of three tensor-memory slots once,
        // when its first k-block comes up.  MX words change every k-block:
        // they ride with the operand stage (buffer and slot = stage), freed by
        // the stage's own commit.
        uint32_t it = 0, tcount = 0, sfi = 0, tslot = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
            int tile, part, kb0, kb1;
            unit_of<SPLIT>(u, p, tile, part, kb0, kb1);
            ok = wait_phase(tempty, (tcount & 1u) ^ 1u, limit, abort_flag, p.err, WHO_MMA);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            for (int kb = kb0; kb < kb1; ++kb) {
                const uint32_t s = it % WSTAGES, ph = (it / WSTAGES) & 1u;
                const bool new_group = kb == kb0 || kb % kScaleGroupKb<G>() == 0;
                const uint32_t sl = G == 16 ? sfi % WNSF : s;
                const uint32_t sph = G == 16 ? (sfi / WNSF) & 1u : ph;
                ok = wait_phase(sBAR + 8 * s, ph, limit, abort_flag, p.err, WHO_MMA) &&
                     (!new_group ||
                      wait_phase(sBAR + BAR_SF + 8 * sl, sph, limit, abort_flag, p.err, WHO_MMA));
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) break;
                ptx::tc_fence_after();
                if (new_group) tslot = G == 16 ? sfi % 3 : s;
                if (lane == 0) {
                    const uint32_t tsfa = tmem + WSFA_COL + 8 * tslot;
                    const uint32_t tsfb = tmem + WSFB_COL + 8 * tslot;
                    if (new_group) {
                        ptx::tc_cp_32x128b_warpx4(tsfa, desc_sf(sSFA + sl * WSF_TILE));
                        ptx::tc_cp_32x128b_warpx4(tsfa + 4, desc_sf(sSFA + sl * WSF_TILE + 512));
                        ptx::tc_cp_32x128b_warpx4(tsfb, desc_sf(sSFB + sl * WSF_TILE));
                        ptx::tc_cp_32x128b_warpx4(tsfb + 4, desc_sf(sSFB + sl * WSF_TILE + 512));
                        if (G == 16) ptx::tc_commit(sBAR + BAR_SF + 32 + 8 * sl);   // buffer free
                    }
                    const uint64_t ad0 = desc_sw128(sA + s * WA_TILE);
                    const uint64_t ad1 = desc_sw128(sA + s * WA_TILE + WA_TILE / 2);
                    const uint64_t bd = desc_sw128(sB + s * WB_TILE);
#pragma unroll
                    for (int j = 0; j < BK / 32; ++j) {
                        const uint32_t idesc = p.idesc | (sf_id(p.gran_a, kb, j) << 29) |
                                               (sf_id(p.gran_b, kb, j) << 4);
                        const uint32_t acc = (kb != kb0 || j != 0) ? 1u : 0u;
                        ptx::tc_mma_mxf8(tmem, ad0 + 2 * j, bd + 2 * j, idesc, tsfa, tsfb, acc);
                        ptx::tc_mma_mxf8(tmem + WACC1, ad1 + 2 * j, bd + 2 * j, idesc, tsfa + 4, tsfb, acc);
                    }
                    ptx::tc_commit(sBAR + 32 + 8 * s);
                }
                __syncwarp();
                if (new_group) ++sfi;
                ++it;
            }
            if (!ok) break;
            if (lane == 0) ptx::tc_commit(tfull);
            __syncwarp();
            ++tcount;
        }
        if (lane == 0) ptx::tc_commit(drain);
        __syncwarp();
        wait_phase(drain, 0u, drain_limit, abort_flag, p.err, WHO_MMA, false);
    } else if (warp == 2 || warp == 3) {
        // ------------------------------------------------- scale loaders
        // warp 2: A's 256 rows, warp 3: B's 224 rows (padded to 256); each
        // keeps its rows' words for one group of G k-blocks in registers with
        // the next group's loads in flight, and writes one buffer of the
        // scale-word ring per scale group.
        // A work unit covers k-blocks [kb0, kb1), which may start and end
        // inside a group.
        const bool is_a = warp == 2;
        uint32_t it = 0;
        bool ok = true;
        int u = blockIdx.x, tile = 0, part = 0, kb0 = 0, kb1 = 0;
        if (u < p.num_units) unit_of<SPLIT>(u, p, tile, part, kb0, kb1);
        int grp = kb0 / G;
        WScaleRows cur, nxt;
        auto load = [&](WScaleRows &dst, int t, int gr) {
            if (is_a) load_rows_wide<G, true>(dst, p, t, gr, lane);
            else load_rows_wide<G, false>(dst, p, t, gr, lane);
        };
        if (u < p.num_units) load(cur, tile, grp);
        const uint32_t sbase = is_a ? sSFA : sSFB;
        while (u < p.num_units && ok) {
            int nu = u, ntile = tile, nkb0 = kb0, nkb1 = kb1, ngrp_next = grp + 1;
            if (ngrp_next * G >= kb1) {
                nu = u + gridDim.x;
                if (nu < p.num_units) {
                    int npart;
                    unit_of<SPLIT>(nu, p, ntile, npart, nkb0, nkb1);
                    ngrp_next = nkb0 / G;
                }
            }
            if (nu < p.num_units) load(nxt, ntile, ngrp_next);
            const int t_lo = kb0 - G * grp, t_hi = kb1 - G * grp;
#pragma unroll
            for (int t = 0; t < G; ++t) {
                if (SPLIT && t < t_lo) continue;
                if (t >= t_hi || !ok) break;
                // one buffer per scale group: its first k-block (or the unit's)
                const int kb = G * grp + t;
                if (!(kb == kb0 || kb % kScaleGroupKb<G>() == 0)) continue;
                constexpr int kWordStep = G / 4;
                const int wi = t / kWordStep;
                // the buffer is free once the MMA warp's copy of its previous
                // group is done (its own commit; MX: the operand stage's)
                const uint32_t sl = G == 16 ? it % WNSF : it % WSTAGES;
                const uint32_t sph = G == 16 ? (it / WNSF) & 1u : (it / WSTAGES) & 1u;
                ok = wait_phase(sBAR + (G == 16 ? BAR_SF + 32 : 32) + 8 * sl, sph ^ 1u, limit,
                                abort_flag, p.err, WHO_SCALES);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) break;
                const uint32_t d = sbase + sl * WSF_TILE + lane * 16;
                st_shared_v4(d, cur.w[0][wi], cur.w[1][wi], cur.w[2][wi], cur.w[3][wi]);
                st_shared_v4(d + 512, cur.w[4][wi], cur.w[5][wi], cur.w[6][wi], cur.w[7][wi]);
                if (!(p.inject == 1 && it == 0)) {
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(sBAR + BAR_SF + 8 * sl);
                }
                ++it;
            }
            cur = nxt;
            u = nu;
            tile = ntile;
            kb0 = nkb0;
            kb1 = nkb1;
            grp = ngrp_next;
        }
    } else if (warp >= 4) {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3, half = (warp - 4) >> 2, ew = warp - 4;
        uint8_t *stage = gbase + WOFF_EPI + ew * EPI_WARP_BYTES;
        uint32_t tcount = 0;
        bool withhold = SPLIT && p.inject == 2 && blockIdx.x == 0 && ew == 0;
        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
            int tile, part, kb0, kb1, mb, nb;
            unit_of<SPLIT>(u, p, tile, part, kb0, kb1);
            tile_coords(tile, p.num_mb, p.num_nb, mb, nb);
            bool ok = wait_phase(tfull, tcount & 1u, limit, abort_flag, p.err, WHO_EPILOGUE);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const int64_t row0 = static_cast<int64_t>(mb) * WBM + half * 128 + q * 32;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + half * WACC1;
            // this warp's 32 rows of a partial tile of part `pt` (>= 1)
            auto partial_rows = [&](int pt) {
                return reinterpret_cast<uint8_t *>(
                    p.ws + ((static_cast<int64_t>(tile) * (p.split - 1) + (pt - 1)) * WBM +
                            half * 128 + q * 32) * WBN);
            };
            if (SPLIT && part > 0) {
                // a K part other than the first: its FP32 partial tile goes to
                // the workspace; the accumulator is free after its last read
#pragma unroll 1
                for (int chunk = 0; chunk < WBN / 32; ++chunk) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(taddr + chunk * 32, r);
                    ptx::tmem_wait_ld();
                    if (chunk == WBN / 32 - 1) {
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(tempty);
                    }
                    uint4 v[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        v[c] = make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
                    store_piece(stage, v, lane, partial_rows(part) + chunk * 128, WBN * 4);
                }
                __syncwarp();
                if (lane == 0) {
                    // release: the warp's partial rows before the count
                    __threadfence();
                    if (!withhold) atomicAdd(p.flags + tile * 8 + ew, 1u);
                }
                withhold = false;
                ++tcount;
                continue;
            }
            if (SPLIT && p.split > 1) {
                // the first K part: wait until every other part has written
                // this warp's rows (bounded), then add them chunk by chunk
                if (lane == 0)
                    ok = wait_flag(p.flags + tile * 8 + ew, static_cast<uint32_t>(p.split - 1),
                                   limit, abort_flag, p.err);
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                __syncwarp();              // lane 0's acquire orders every lane's reads below
                if (!ok) break;
            }
            // FP32 partials of parts 1 .. split-1 added to a 32-column chunk of
            // the accumulator, in part order
            auto add_partials = [&](uint32_t (&r)[32], int chunk) {
                for (int pt = 1; pt < p.split; ++pt) {
                    uint4 v[8];
                    load_piece(stage, v, lane, partial_rows(pt) + chunk * 128, WBN * 4);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        r[4 * c] = __float_as_uint(__uint_as_float(r[4 * c]) + __uint_as_float(v[c].x));
                        r[4 * c + 1] = __float_as_uint(__uint_as_float(r[4 * c + 1]) + __uint_as_float(v[c].y));
                        r[4 * c + 2] = __float_as_uint(__uint_as_float(r[4 * c + 2]) + __uint_as_float(v[c].z));
                        r[4 * c + 3] = __float_as_uint(__uint_as_float(r[4 * c + 3]) + __uint_as_float(v[c].w));
                    }
                }
            };
            if (p.out_fp32 || p.accumulate || (SPLIT && p.split > 1)) {
                // FP32 out, accumulation into C, or a split tile's first part:
                // 32 columns at a time, old values (and partial tiles) read
                // and new ones written as row segments through the staging
                // area; the accumulator is released after its last columns
                // are read.
#pragma unroll 1
                for (int chunk = 0; chunk < WBN / 32; ++chunk) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(taddr + chunk * 32, r);
                    ptx::tmem_wait_ld();
                    if (chunk == WBN / 32 - 1) {
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(tempty);
                    }
                    if constexpr (SPLIT) add_partials(r, chunk);
                    auto emit = [&](const uint32_t(&rr)[32], int cc) {
                        const int64_t n0 = static_cast<int64_t>(nb) * WBN + cc * 32;
                        if (n0 >= p.N) return;
                        if (p.out_fp32) {
                            uint8_t *g = reinterpret_cast<uint8_t *>(static_cast<float *>(p.c) + row0 * p.ldc + n0);
                            uint4 v[8];
                            if (p.accumulate) {
                                load_piece(stage, v, lane, g, p.ldc * 4);
#pragma unroll
                                for (int c = 0; c < 8; ++c)
                                    v[c] = make_uint4(__float_as_uint(__uint_as_float(rr[4 * c]) + __uint_as_float(v[c].x)),
                                                      __float_as_uint(__uint_as_float(rr[4 * c + 1]) + __uint_as_float(v[c].y)),
                                                      __float_as_uint(__uint_as_float(rr[4 * c + 2]) + __uint_as_float(v[c].z)),
                                                      __float_as_uint(__uint_as_float(rr[4 * c + 3]) + __uint_as_float(v[c].w)));
                            } else {
#pragma unroll
                                for (int c = 0; c < 8; ++c)
                                    v[c] = make_uint4(rr[4 * c], rr[4 * c + 1], rr[4 * c + 2], rr[4 * c + 3]);
                            }
                            store_piece(stage, v, lane, g, p.ldc * 4);
                        } else if (!p.accumulate) {
                            // BF16 (a split tile's first part): round once
                            uint8_t *g = reinterpret_cast<uint8_t *>(static_cast<uint16_t *>(p.c) + row0 * p.ldc + n0);
                            uint4 v[4];
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                v[c] = make_uint4(
                                    ptx::cvt_bf16x2(__uint_as_float(rr[8 * c]), __uint_as_float(rr[8 * c + 1])),
                                    ptx::cvt_bf16x2(__uint_as_float(rr[8 * c + 2]), __uint_as_float(rr[8 * c + 3])),
                                    ptx::cvt_bf16x2(__uint_as_float(rr[8 * c + 4]), __uint_as_float(rr[8 * c + 5])),
                                    ptx::cvt_bf16x2(__uint_as_float(rr[8 * c + 6]), __uint_as_float(rr[8 * c + 7])));
                            store_piece64(stage, v, lane, g, p.ldc * 2);
                        } else {
                            // BF16 with accumulation: add in FP32, round once
                            uint8_t *g = reinterpret_cast<uint8_t *>(static_cast<uint16_t *>(p.c) + row0 * p.ldc + n0);
                            uint4 v[4];
                            load_piece64(stage, v, lane, g, p.ldc * 2);
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                v[c] = make_uint4(
                                    ptx::cvt_bf16x2(__uint_as_float(rr[8 * c]) + bf16_lo(v[c].x),
                                                    __uint_as_float(rr[8 * c + 1]) + bf16_hi(v[c].x)),
                                    ptx::cvt_bf16x2(__uint_as_float(rr[8 * c + 2]) + bf16_lo(v[c].y),
                                                    __uint_as_float(rr[8 * c + 3]) + bf16_hi(v[c].y)),
                                    ptx::cvt_bf16x2(__uint_as_float(rr[8 * c + 4]) + bf16_lo(v[c].z),
                                                    __uint_as_float(rr[8 * c + 5]) + bf16_hi(v[c].z)),
                                    ptx::cvt_bf16x2(__uint_as_float(rr[8 * c + 6]) + bf16_lo(v[c].w),
                                                    __uint_as_float(rr[8 * c + 7]) + bf16_hi(v[c].w)));
                            }
                            store_piece64(stage, v, lane, g, p.ldc * 2);
                        }
                    };
                    emit(r, chunk);
                }
                if (SPLIT && lane == 0) p.flags[tile * 8 + ew] = 0u;   // clean for the next call
                ++tcount;
                continue;
            }
            uint32_t packed[WBN / 2];
#pragma unroll
            for (int chunk = 0; chunk < WBN / 32; ++chunk) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(taddr + chunk * 32, r);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    packed[chunk * 16 + e] =
                        ptx::cvt_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(tempty);
            const int64_t col0 = static_cast<int64_t>(nb) * WBN;
            store_wide_piece<0>(stage, packed, lane, p, row0, col0);
            store_wide_piece<1>(stage, packed, lane, p, row0, col0);
            store_wide_piece<2>(stage, packed, lane, p, row0, col0);
            store_wide_piece<3>(stage, packed, lane, p, row0, col0);
            ++tcount;
        }
    }

    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------- CTA-pair variant
// Tile 256 x 448 computed by a pair of CTAs (a cluster of two) with
// tcgen05.mma.cta_group::2: per 32-K step two M = 256, N = 224 MMAs, one per
// half of the tile's columns.  Each CTA holds its 128 rows of A and, of each
// column half, its 112 rows of B in its own shared memory; the MMAs issued by
// the even CTA read both CTAs' operands, and each CTA's tensor memory
// receives its 128 rows of the 256 x 448 accumulator (two 224-column
// accumulators).  A stage is then 44 KB per CTA for 128 x 448 x 128 MACs per
// SM (the single-CTA 256 x 224 kernel needs 60 KB for the same work): four
// stages fit, three in flight while one is consumed, and each SM reads 27 %
// fewer operand bytes per MAC from L2.
//   Both CTAs: warp 0 TMA producer (its A rows and B rows; completion counted
//   on the even CTA's stage barrier), warps 2 and 3 scale loaders (warp 2:
//   this CTA's 128 A rows and the first column half's 224 B rows; warp 3: the
//   second half's), writing one buffer of a four-deep ring per scale group
//   (four k-blocks for 1x128 / 128x128 scales, one for MX), warps 4-11
//   epilogue (two per tensor-memory lane quarter, one per accumulator).
//   Even CTA: warp 1 copies each scale group into tensor memory and issues
//   the MMAs for the pair, committing to both CTAs' barriers.  Odd CTA: warp
//   1 forwards each filled scale buffer to the even CTA (one cluster-scope
//   release arrival from a warp with no loads in flight).
//   The MMA issuer and the producer run on one lane: an MMA, a commit or a
//   completed barrier wait each take tens of cycles to issue, and a 32-K
//   step of this tile lasts 224 cycles.
//   Tensor memory (both CTAs): accumulators at columns 0 and 224, then three
//   slots of 4 columns of A scales and 16 of B scales (8 per column half).
constexpr int PR_BM = 256, PR_BN = 448, PR_HN = 224, PR_STAGES = 4, PR_NSF = 4;
constexpr int PR_THREADS = 384;
constexpr uint32_t PR_A_TILE = 128 * BK;                 // per CTA
constexpr uint32_t PR_BH_TILE = (PR_HN / 2) * BK;        // per CTA and column half
constexpr uint32_t PR_STAGE = PR_A_TILE + 2 * PR_BH_TILE;
constexpr uint32_t PR_SFA_TILE = 512, PR_SFB_TILE = 2048;
constexpr uint32_t PR_SFA_COL = PR_BN;                   // + 4 * slot
constexpr uint32_t PR_SFB_COL = PR_BN + 12;              // + 16 * slot
constexpr uint32_t PR_OFF_SFA = PR_STAGES * PR_STAGE;
constexpr uint32_t PR_OFF_SFB = PR_OFF_SFA + PR_NSF * PR_SFA_TILE;
constexpr uint32_t PR_OFF_BAR = PR_OFF_SFB + PR_NSF * PR_SFB_TILE;
// barriers from PR_OFF_BAR (8 bytes each): full[4] at 0 (operand bytes of both
// CTAs; even CTA), empty[4] at 32 (each CTA), sf_full[4] at 64 (scale words
// written: this CTA's 64 scale-warp lanes, plus on the even CTA the odd CTA's
// forwarder), sf_empty[4] at 96 (the pair's copy of the buffer done; each
// CTA), tfull 128 (each CTA), tempty 136 (one arrival per epilogue warp of
// both CTAs; even CTA), drain 144.
constexpr uint32_t PR_BAR_EMPTY = 32, PR_BAR_SFF = 64, PR_BAR_SFE = 96, PR_BAR_TFULL = 128,
                   PR_BAR_TEMPTY = 136, PR_BAR_DRAIN = 144;
constexpr uint32_t PR_OFF_TMEM_SLOT = PR_OFF_BAR + 160;
constexpr uint32_t PR_OFF_ABORT = PR_OFF_BAR + 164;
constexpr uint32_t PR_OFF_EPI = PR_OFF_BAR + 256;
constexpr uint32_t PR_SMEM_BYTES = PR_OFF_EPI + 8 * EPI_WARP_BYTES + 1024;
static_assert(PR_A_TILE % 1024 == 0 && PR_BH_TILE % 1024 == 0,
              "operand tiles must keep the 128-byte swizzle's 1 KB alignment");
static_assert(PR_SFB_COL + 16 * 3 <= TMEM_COLS, "tensor memory overflow");
static_assert(PR_SMEM_BYTES <= 232448, "shared memory overflow");

// Wait on a barrier of this CTA whose arrivals may come from the other CTA of
// the pair (acquire at cluster scope); bounded like wait_phase.
__device__ bool wait_phase_pair(uint32_t bar, uint32_t parity, uint64_t limit,
                                volatile uint32_t *abort_flag, unsigned int *err, uint32_t who,
                                bool check_abort = true) {
    if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    uint32_t it = 0;
    while (true) {
        if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
        if ((++it & 15u) == 0) {
            if (check_abort && *abort_flag) return false;
            if (ptx::globaltimer() - t0 > limit) {
                if (check_abort) {
                    *abort_flag = 1u;
                    atomicOr(err, 1u);
                    atomicCAS(err + 1, 0u, who);
                }
                return false;
            }
        }
    }
}

// One lane's scale words for one group of G k-blocks: up to 12 rows.
struct PairScaleRows {
    uint32_t w[12][4];
};

// Pair tile t -> (m-block of 256 rows, n-block of 448 columns); the same
// grouped order as the other kernels.
template <int G>
__global__ void __launch_bounds__(PR_THREADS, 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap tmap_a,
                const __grid_constant__ CUtensorMap tmap_b, const KParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sSFA = base + PR_OFF_SFA, sSFB = base + PR_OFF_SFB, sBAR = base + PR_OFF_BAR;
    const uint32_t empty = sBAR + PR_BAR_EMPTY, sf_full = sBAR + PR_BAR_SFF,
                   sf_empty = sBAR + PR_BAR_SFE;
    const uint32_t tfull = sBAR + PR_BAR_TFULL, tempty = sBAR + PR_BAR_TEMPTY,
                   drain = sBAR + PR_BAR_DRAIN;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + PR_OFF_TMEM_SLOT);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + PR_OFF_ABORT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();   // 0: issues the pair's MMAs
    const bool leader = rank == 0;
    const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);
    const uint64_t limit = p.wait_limit_ns;
    const uint64_t drain_limit = 2000000ull;
    // the even CTA's barriers, as seen from either CTA
    const uint32_t full_l = ptx::map_shared_rank(sBAR, 0);
    const uint32_t sf_full_l = ptx::map_shared_rank(sf_full, 0);
    const uint32_t tempty_l = ptx::map_shared_rank(tempty, 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < PR_STAGES; ++s) {
            ptx::mbar_init(sBAR + 8 * s, 1);        // even CTA's expect_tx (both CTAs' bytes)
            ptx::mbar_init(empty + 8 * s, 1);       // the pair's commit
        }
        for (int i = 0; i < PR_NSF; ++i) {
            ptx::mbar_init(sf_full + 8 * i, leader ? 65 : 64);
            ptx::mbar_init(sf_empty + 8 * i, 1);    // the pair's commit after the copy
        }
        ptx::mbar_init(tfull, 1);
        ptx::mbar_init(tempty, 16);                 // one arrival per epilogue warp of both CTAs
        ptx::mbar_init(drain, 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmap_a);
        ptx::prefetch_tmap(&tmap_b);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();   // both CTAs' barriers and tensor memory exist
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int tile = pair; tile < p.num_tiles && ok; tile += npairs) {
                int mb, nb;
                tile_coords(tile, p.num_mb, p.num_nb, mb, nb);
                const int arow = mb * PR_BM + static_cast<int>(rank) * 128;
                const int brow = nb * PR_BN + static_cast<int>(rank) * (PR_HN / 2);
                for (int kb = 0; kb < p.nk; ++kb) {
                    const uint32_t s = it % PR_STAGES, ph = (it / PR_STAGES) & 1u;
                    ok = wait_phase(empty + 8 * s, ph ^ 1u, limit, abort_flag, p.err, WHO_PRODUCER);
                    if (!ok) break;
                    const uint32_t st = base + s * PR_STAGE;
                    if (leader) ptx::mbar_arrive_expect_tx(sBAR + 8 * s, 2 * PR_STAGE);
                    ptx::tma_load_2d_pair(st, &tmap_a, full_l + 8 * s, kb * BK, arow);
                    ptx::tma_load_2d_pair(st + PR_A_TILE, &tmap_b, full_l + 8 * s, kb * BK, brow);
                    ptx::tma_load_2d_pair(st + PR_A_TILE + PR_BH_TILE, &tmap_b, full_l + 8 * s, kb * BK,
                                          brow + PR_HN);
                    ++it;
                }
            }
            // the even CTA waits until the last loads of both CTAs have landed;
            // the cluster barrier below keeps the odd CTA resident until then
            if (leader) {
                const uint32_t nd = it < static_cast<uint32_t>(PR_STAGES) ? it : static_cast<uint32_t>(PR_STAGES);
                for (uint32_t i = it - nd; i < it; ++i)
                    wait_phase(sBAR + 8 * (i % PR_STAGES), (i / PR_STAGES) & 1u, drain_limit, abort_flag,
                               p.err, WHO_PRODUCER, false);
            }
            // A CTA that stopped early cannot tell which of its last copies the
            // even CTA's barriers have counted; it gives them the drain bound
            // to land (copies take microseconds) before the pair may leave.
            if (!ok || *abort_flag) {
                const uint64_t t0 = ptx::globaltimer();
                while (ptx::globaltimer() - t0 < drain_limit) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1 && leader) {
        // ------------------------------------------- MMA issuer (even CTA)
        // Scale groups come through the ring in order (sfi); each is copied
        // into one of three tensor-memory slots when its first k-block comes
        // up, and its buffer is released by the copy's commit.
        if (lane == 0) {
            uint32_t it = 0, tcount = 0, sfi = 0, tslot = 0;
            bool ok = true;
            for (int tile = pair; tile < p.num_tiles && ok; tile += npairs) {
                ok = wait_phase_pair(tempty, (tcount & 1u) ^ 1u, limit, abort_flag, p.err, WHO_MMA);
                if (!ok) break;
                ptx::tc_fence_after();
                for (int kb = 0; kb < p.nk; ++kb) {
                    const uint32_t s = it % PR_STAGES, ph = (it / PR_STAGES) & 1u;
                    const bool new_group = kb % kScaleGroupKb<G>() == 0;
                    const uint32_t sl = sfi % PR_NSF, sph = (sfi / PR_NSF) & 1u;
                    ok = wait_phase(sBAR + 8 * s, ph, limit, abort_flag, p.err, WHO_MMA) &&
                         (!new_group ||
                          wait_phase_pair(sf_full + 8 * sl, sph, limit, abort_flag, p.err, WHO_MMA));
                    if (!ok) break;
                    ptx::tc_fence_after();
                    if (new_group) {
                        tslot = sfi % 3;
                        const uint32_t tsfa = tmem + PR_SFA_COL + 4 * tslot;
                        const uint32_t tsfb = tmem + PR_SFB_COL + 16 * tslot;
                        const uint32_t bsf = sSFB + sl * PR_SFB_TILE;
                        ptx::tc_cp_32x128b_warpx4_pair(tsfa, desc_sf(sSFA + sl * PR_SFA_TILE));
                        ptx::tc_cp_32x128b_warpx4_pair(tsfb, desc_sf(bsf));
                        ptx::tc_cp_32x128b_warpx4_pair(tsfb + 4, desc_sf(bsf + 512));
                        ptx::tc_cp_32x128b_warpx4_pair(tsfb + 8, desc_sf(bsf + 1024));
                        ptx::tc_cp_32x128b_warpx4_pair(tsfb + 12, desc_sf(bsf + 1536));
                        ptx::tc_commit_pair(sf_empty + 8 * sl, 0x3);   // the buffer, both CTAs
                        ++sfi;
                    }
                    const uint32_t tsfa = tmem + PR_SFA_COL + 4 * tslot;
                    const uint32_t tsfb = tmem + PR_SFB_COL + 16 * tslot;
                    const uint32_t st = base + s * PR_STAGE;
                    const uint64_t ad = desc_sw128(st);
                    const uint64_t bd0 = desc_sw128(st + PR_A_TILE);
                    const uint64_t bd1 = desc_sw128(st + PR_A_TILE + PR_BH_TILE);
#pragma unroll
                    for (int j = 0; j < BK / 32; ++j) {
                        const uint32_t idesc = p.idesc | (sf_id(p.gran_a, kb, j) << 29) |
                                               (sf_id(p.gran_b, kb, j) << 4);
                        const uint32_t acc = (kb | j) != 0 ? 1u : 0u;
                        ptx::tc_mma_mxf8_pair(tmem, ad + 2 * j, bd0 + 2 * j, idesc, tsfa, tsfb, acc);
                        ptx::tc_mma_mxf8_pair(tmem + PR_HN, ad + 2 * j, bd1 + 2 * j, idesc, tsfa, tsfb + 8,
                                              acc);
                    }
                    ptx::tc_commit_pair(empty + 8 * s, 0x3);   // frees the stage in both CTAs
                    ++it;
                }
                if (!ok) break;
                ptx::tc_commit_pair(tfull, 0x3);
                ++tcount;
            }
            ptx::tc_commit_pair(drain, 0x1);
            wait_phase(drain, 0u, drain_limit, abort_flag, p.err, WHO_MMA, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------ scale-buffer forwarder (odd CTA)
        if (lane == 0) {
            uint32_t sfi = 0;
            bool ok = true;
            for (int tile = pair; tile < p.num_tiles && ok; tile += npairs) {
                for (int kb = 0; kb < p.nk; kb += kScaleGroupKb<G>()) {
                    const uint32_t sl = sfi % PR_NSF, sph = (sfi / PR_NSF) & 1u;
                    ok = wait_phase(sf_full + 8 * sl, sph, limit, abort_flag, p.err, WHO_SCALES);
                    if (!ok) break;
                    ptx::mbar_arrive_cluster(sf_full_l + 8 * sl);
                    ++sfi;
                }
            }
        }
        __syncwarp();
    } else if (warp == 2 || warp == 3) {
        // ------------------------------------------------- scale loaders
        // warp 2: this CTA's 128 A rows (words 0-3) and the first column
        // half's 224 B rows, padded to 256 (words 4-11); warp 3: the second
        // half's B rows (words 0-7).  Each loads its rows' words for one group
        // of G k-blocks (four ring buffers) after writing the previous
        // group's; the ring covers the loads' latency.
        const bool w2 = warp == 2;
        uint32_t it = 0;
        bool ok = true;
        const int ngrp = (p.nk + G - 1) / G;
        int tile = pair, grp = 0;
        PairScaleRows cur;
        auto load = [&](PairScaleRows &g, int t, int gr) {
            int mb, nb;
            tile_coords(t, p.num_mb, p.num_nb, mb, nb);
            const int64_t nbase = static_cast<int64_t>(nb) * PR_BN;
            if (w2) {
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const int64_t m = static_cast<int64_t>(mb) * PR_BM + rank * 128 + 32 * a + lane;
                    load_row_scales<G>(p.sa, p.ld_sa, p.gran_a, m, gr, p.nk, true, g.w[a]);
                }
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const int64_t n = nbase + 32 * h + lane;
                    load_row_scales<G>(p.sb, p.ld_sb, p.gran_b, n, gr, p.nk, h < 7 && n < p.N, g.w[4 + h]);
                }
            } else {
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const int64_t n = nbase + PR_HN + 32 * h + lane;
                    load_row_scales<G>(p.sb, p.ld_sb, p.gran_b, n, gr, p.nk, h < 7 && n < p.N, g.w[h]);
                }
            }
        };
        while (tile < p.num_tiles && ok) {
            load(cur, tile, grp);
#pragma unroll
            for (int t = 0; t < G; ++t) {
                const int kb = G * grp + t;
                if (kb >= p.nk || !ok) break;
                if (kb % kScaleGroupKb<G>() != 0) continue;
                constexpr int kWordStep = G / 4;
                const int wi = t / kWordStep;
                const uint32_t sl = it % PR_NSF, sph = (it / PR_NSF) & 1u;
                ok = wait_phase(sf_empty + 8 * sl, sph ^ 1u, limit, abort_flag, p.err, WHO_SCALES);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) break;
                const uint32_t dB = sSFB + sl * PR_SFB_TILE + lane * 16;
                if (w2) {
                    st_shared_v4(sSFA + sl * PR_SFA_TILE + lane * 16, cur.w[0][wi], cur.w[1][wi],
                                 cur.w[2][wi], cur.w[3][wi]);
                    st_shared_v4(dB, cur.w[4][wi], cur.w[5][wi], cur.w[6][wi], cur.w[7][wi]);
                    st_shared_v4(dB + 512, cur.w[8][wi], cur.w[9][wi], cur.w[10][wi], cur.w[11][wi]);
                } else {
                    st_shared_v4(dB + 1024, cur.w[0][wi], cur.w[1][wi], cur.w[2][wi], cur.w[3][wi]);
                    st_shared_v4(dB + 1536, cur.w[4][wi], cur.w[5][wi], cur.w[6][wi], cur.w[7][wi]);
                }
                if (!(p.inject == 1 && it == 0 && leader && w2)) {
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(sf_full + 8 * sl);
                }
                ++it;
            }
            if (++grp == ngrp) {
                grp = 0;
                tile += npairs;
            }
        }
    } else if (warp >= 4) {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3, half = (warp - 4) >> 2, ew = warp - 4;
        uint8_t *stage = gbase + PR_OFF_EPI + ew * EPI_WARP_BYTES;
        uint32_t tcount = 0;
        for (int tile = pair; tile < p.num_tiles; tile += npairs) {
            int mb, nb;
            tile_coords(tile, p.num_mb, p.num_nb, mb, nb);
            bool ok = wait_phase(tfull, tcount & 1u, limit, abort_flag, p.err, WHO_EPILOGUE);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const int64_t row0 = static_cast<int64_t>(mb) * PR_BM + rank * 128 + q * 32;
            const int64_t col0 = static_cast<int64_t>(nb) * PR_BN + half * PR_HN;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + half * PR_HN;
            if (p.out_fp32 || p.accumulate) {
                // FP32 out, or accumulation into C: 32 columns at a time; the
                // accumulator is released after its last columns are read
#pragma unroll 1
                for (int chunk = 0; chunk < PR_HN / 32; ++chunk) {
                    uint32_t rr[32];
                    ptx::tmem_ld_32x32b_x32(taddr + chunk * 32, rr);
                    ptx::tmem_wait_ld();
                    if (chunk == PR_HN / 32 - 1) {
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive_cluster(tempty_l);
                    }
                    const int64_t n0 = col0 + chunk * 32;
                    if (n0 >= p.N) continue;
                    if (p.out_fp32) {
                        uint8_t *g = reinterpret_cast<uint8_t *>(static_cast<float *>(p.c) + row0 * p.ldc + n0);
                        uint4 v[8];
                        if (p.accumulate) {
                            load_piece(stage, v, lane, g, p.ldc * 4);
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                v[c] = make_uint4(__float_as_uint(__uint_as_float(rr[4 * c]) + __uint_as_float(v[c].x)),
                                                  __float_as_uint(__uint_as_float(rr[4 * c + 1]) + __uint_as_float(v[c].y)),
                                                  __float_as_uint(__uint_as_float(rr[4 * c + 2]) + __uint_as_float(v[c].z)),
                                                  __float_as_uint(__uint_as_float(rr[4 * c + 3]) + __uint_as_float(v[c].w)));
                        } else {
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                v[c] = make_uint4(rr[4 * c], rr[4 * c + 1], rr[4 * c + 2], rr[4 * c + 3]);
                        }
                        store_piece(stage, v, lane, g, p.ldc * 4);
                    } else {
                        // BF16 with accumulation: add in FP32, round once
                        uint8_t *g = reinterpret_cast<uint8_t *>(static_cast<uint16_t *>(p.c) + row0 * p.ldc + n0);
                        uint4 v[4];
                        load_piece64(stage, v, lane, g, p.ldc * 2);
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            v[c] = make_uint4(
                                ptx::cvt_bf16x2(__uint_as_float(rr[8 * c]) + bf16_lo(v[c].x),
                                                __uint_as_float(rr[8 * c + 1]) + bf16_hi(v[c].x)),
                                ptx::cvt_bf16x2(__uint_as_float(rr[8 * c + 2]) + bf16_lo(v[c].y),
                                                __uint_as_float(rr[8 * c + 3]) + bf16_hi(v[c].y)),
                                ptx::cvt_bf16x2(__uint_as_float(rr[8 * c + 4]) + bf16_lo(v[c].z),
                                                __uint_as_float(rr[8 * c + 5]) + bf16_hi(v[c].z)),
                                ptx::cvt_bf16x2(__uint_as_float(rr[8 * c + 6]) + bf16_lo(v[c].w),
                                                __uint_as_float(rr[8 * c + 7]) + bf16_hi(v[c].w)));
                        }
                        store_piece64(stage, v, lane, g, p.ldc * 2);
                    }
                }
                ++tcount;
                continue;
            }
            // BF16 out: the warp's 224 columns converted first, the
            // accumulator released, then written in 64-column pieces (N is a
            // multiple of 128 and a column half starts at a multiple of 32,
            // so a piece can straddle N by exactly 32 columns: it is then a
            // half piece) and a last 32-column half piece
            uint32_t packed[PR_HN / 2];
#pragma unroll
            for (int chunk = 0; chunk < PR_HN / 16; ++chunk) {
                uint32_t rr[16];
                ptx::tmem_ld_32x32b_x16(taddr + chunk * 16, rr);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    packed[chunk * 8 + e] =
                        ptx::cvt_bf16x2(__uint_as_float(rr[2 * e]), __uint_as_float(rr[2 * e + 1]));
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(tempty_l);
            static_assert(PR_HN == WBN, "the pair kernel's column half has the wide tile's width");
            store_wide_piece<0>(stage, packed, lane, p, row0, col0);
            store_wide_piece<1>(stage, packed, lane, p, row0, col0);
            store_wide_piece<2>(stage, packed, lane, p, row0, col0);
            store_wide_piece<3>(stage, packed, lane, p, row0, col0);
            ++tcount;
        }
    }

    // neither CTA leaves (or frees its tensor memory) while the other may still
    // read its shared memory, signal its barriers or write its tensor memory
    ptx::tc_fence_before();
    ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

bool make_tmap(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t k, uint64_t ld,
               uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {k, rows};
    const cuuint64_t strides[1] = {ld};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_sms[64] = {0};
bool g_attr_set[64] = {false};
std::mutex g_mu;

// Split-K workspace: per-tile flags (8 words per tile, padded to 256 bytes),
// then the FP32 partial tiles of parts 1 .. split-1.
size_t splitk_flag_bytes(int64_t tiles) { return (static_cast<size_t>(tiles) * 32 + 255) / 256 * 256; }
size_t splitk_bytes(int64_t tiles, int split) {
    if (split <= 1) return 0;
    return splitk_flag_bytes(tiles) +
           static_cast<size_t>(tiles) * (split - 1) * WBM * WBN * sizeof(float);
}

int device_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

}  // namespace

int64_t gemm_wide_tiles(int64_t M, int64_t N) { return (M / WBM) * ((N + WBN - 1) / WBN); }

// The library's split for a 256 x 224-tile GEMM.  Cost in k-block times:
// rounds of units x (k-blocks per unit + 13 per extra part), the exchange
// cost measured on GB300 (about 10 us per partial tile read by the first
// part's CTA while it holds its accumulator).  A split is taken only when it
// is estimated at least 20 % faster: shapes with few tiles and a long K.
int gemm_auto_split(int64_t M, int64_t N, int64_t K, int sms) {
    const int64_t tiles = gemm_wide_tiles(M, N), nk = K / BK;
    const double base = static_cast<double>((tiles + sms - 1) / sms) * static_cast<double>(nk);
    int best = 1;
    double best_cost = 0.8 * base;
    for (int sp = 2; sp <= 8; ++sp) {
        if (nk / sp < 8) break;
        const double cost = static_cast<double>((tiles * sp + sms - 1) / sms) *
                            (static_cast<double>(nk) / sp + 13.0 * (sp - 1));
        if (cost < best_cost) {
            best = sp;
            best_cost = cost;
        }
    }
    return best;
}

size_t gemm_splitk_workspace(int64_t M, int64_t N, int64_t K, int split) {
    if (split == 0) split = gemm_auto_split(M, N, K, device_sms());
    return splitk_bytes(gemm_wide_tiles(M, N), split);
}

unsigned int *device_error_word() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fp8hg_err) != cudaSuccess) return nullptr;
    return static_cast<unsigned int *>(p);
}

int launch_gemm_scaled(const GemmArgs &g, cudaStream_t stream) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_attr_set[dev]) {
            for (auto kern : {k_gemm_mxf8<16, false>, k_gemm_mxf8<4, false>, k_gemm_mxf8<16, true>,
                              k_gemm_mxf8<4, true>}) {
                const cudaError_t e = cudaFuncSetAttribute(
                    kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM_BYTES));
                if (e != cudaSuccess) return 2 + static_cast<int>(e);
            }
            for (auto kern : {k_gemm_wide<16, false>, k_gemm_wide<4, false>, k_gemm_wide<16, true>,
                              k_gemm_wide<4, true>}) {
                const cudaError_t e = cudaFuncSetAttribute(
                    kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(W_SMEM_BYTES));
                if (e != cudaSuccess) return 2 + static_cast<int>(e);
            }
            for (auto kern : {k_gemm_pair<16>, k_gemm_pair<4>}) {
                const cudaError_t e = cudaFuncSetAttribute(
                    kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(PR_SMEM_BYTES));
                if (e != cudaSuccess) return 2 + static_cast<int>(e);
            }
            int n = 0;
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
            g_sms[dev] = n > 0 ? n : 1;
            g_attr_set[dev] = true;
        }
    }
    const int sms = g_sms[dev];

    // The 256 x 224 variant where M is a multiple of 256 (not for the
    // quantized epilogue, whose 1x128 groups must not straddle tiles), unless
    // its coarser tiles fill the last wave of SMs so much worse that its
    // ~8 % faster tiles do not make up for it.
    const bool paired = g.tile == 3 && !g.out_q && g.M % PR_BM == 0 && sms >= 2;
    bool wide = !paired && !g.out_q && g.M % WBM == 0 && g.tile != 1;
    // split-K: forced (split_k >= 2, wide tiles) or chosen (split_k = 0) when
    // the workspace holds what the split needs
    int split = 1;
    if (wide && g.ws && g.split_k != 1) {
        split = g.split_k >= 2 ? g.split_k : gemm_auto_split(g.M, g.N, g.K, sms);
        if (split > 1 && g.ws_bytes < splitk_bytes(gemm_wide_tiles(g.M, g.N), split)) {
            if (g.split_k >= 2) return 1;
            split = 1;
        }
    }
    if (wide && g.tile != 2 && split == 1) {
        auto wave_eff = [&](int64_t tiles) {
            const int64_t waves = (tiles + sms - 1) / sms;
            return static_cast<double>(tiles) / static_cast<double>(waves * sms);
        };
        const int64_t t_wide = (g.M / WBM) * ((g.N + WBN - 1) / WBN);
        const int64_t t_std = (g.M / BM) * ((g.N + BN - 1) / BN);
        wide = 1.08 * wave_eff(t_wide) >= wave_eff(t_std);
    }
    CUtensorMap ta, tb;
    std::memset(&ta, 0, sizeof(ta));
    std::memset(&tb, 0, sizeof(tb));
    if (!make_tmap(&ta, g.a_codes, g.M, g.K, g.lda, paired ? 128 : (wide ? WBM : BM))) return 1;
    if (!make_tmap(&tb, g.b_codes, g.N, g.K, g.ldb, paired ? PR_HN / 2 : (wide ? WBN : BN))) return 1;

    KParams p;
    p.M = static_cast<int>(g.M);
    p.N = static_cast<int>(g.N);
    p.nk = static_cast<int>(g.K / BK);
    const int tbn = paired ? PR_BN : (wide ? WBN : BN), tbm = paired ? PR_BM : (wide ? WBM : BM);
    p.num_nb = static_cast<int>((g.N + tbn - 1) / tbn);
    p.num_mb = static_cast<int>(g.M / tbm);
    p.num_tiles = p.num_mb * p.num_nb;
    p.gran_a = g.gran_a;
    p.gran_b = g.gran_b;
    p.out_fp32 = g.out_fp32;
    p.accumulate = g.accumulate;
    p.out_q = g.out_q;
    p.fmt_c = g.fmt_c;
    p.cs = g.c_scale;
    p.ld_cs = g.ld_cs;
    p.inject = g.inject_fault;
    p.sa = g.a_scale;
    p.sb = g.b_scale;
    p.ld_sa = g.ld_sa;
    p.ld_sb = g.ld_sb;
    p.c = g.c;
    p.ldc = g.ldc;
    // instruction descriptor, kind::mxf8f6f4 with block scaling: A/B formats
    // (E4M3 = 0, E5M2 = 1) in bits 7-9 / 10-12, K-major A and B, N >> 3 in
    // bits 17-22, UE8M0 scale type in bit 23, M >> 4 in bits 24-28; the
    // scale-factor byte ids (bits 4-5 for B, 29-30 for A) are set per MMA.
    // (the pair kernel's MMA spans M = 256 rows of both CTAs)
    p.idesc = (1u << 23) | (static_cast<uint32_t>((paired ? PR_HN : tbn) >> 3) << 17) |
              (static_cast<uint32_t>((paired ? PR_BM : BM) >> 4) << 24) |
              (static_cast<uint32_t>(g.fmt_a) << 7) | (static_cast<uint32_t>(g.fmt_b) << 10);
    p.wait_limit_ns = g.wait_limit_ns;
    p.err = g.err;
    p.split = split;
    p.num_units = p.num_tiles * split;
    p.flags = split > 1 ? static_cast<unsigned int *>(g.ws) : nullptr;
    p.ws = split > 1 ? reinterpret_cast<float *>(static_cast<uint8_t *>(g.ws) +
                                                 splitk_flag_bytes(p.num_tiles))
                     : nullptr;

    const bool mx = g.gran_a == GRAN_MX32;
    if (paired) {
        // one pair of CTAs (a cluster of two) per two SMs
        int pairs = sms / 2;
        if (pairs > p.num_tiles) pairs = p.num_tiles;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
        cfg.blockDim = dim3(PR_THREADS);
        cfg.dynamicSmemBytes = PR_SMEM_BYTES;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = mx ? cudaLaunchKernelEx(&cfg, k_gemm_pair<4>, ta, tb, p)
                                 : cudaLaunchKernelEx(&cfg, k_gemm_pair<16>, ta, tb, p);
        return e == cudaSuccess ? 0 : 2 + static_cast<int>(e);
    }
    int grid = sms;
    if (grid > p.num_units) grid = p.num_units;
    if (wide && split > 1) {
        // a unit of the first K part waits for the other parts of its tile,
        // which run on other CTAs: every CTA must be resident (cooperative)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(W_THREADS);
        cfg.dynamicSmemBytes = W_SMEM_BYTES;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = mx ? cudaLaunchKernelEx(&cfg, k_gemm_wide<4, true>, ta, tb, p)
                                 : cudaLaunchKernelEx(&cfg, k_gemm_wide<16, true>, ta, tb, p);
        return e == cudaSuccess ? 0 : 2 + static_cast<int>(e);
    }
    if (wide) {
        if (mx) k_gemm_wide<4, false><<<grid, W_THREADS, W_SMEM_BYTES, stream>>>(ta, tb, p);
        else k_gemm_wide<16, false><<<grid, W_THREADS, W_SMEM_BYTES, stream>>>(ta, tb, p);
    } else if (g.out_q) {
        if (mx) k_gemm_mxf8<4, true><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(ta, tb, p);
        else k_gemm_mxf8<16, true><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(ta, tb, p);
    } else {
        if (mx) k_gemm_mxf8<4, false><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(ta, tb, p);
        else k_gemm_mxf8<16, false><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(ta, tb, p);
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? 0 : 2 + static_cast<int>(e);
}

}  // namespace fp8hg
