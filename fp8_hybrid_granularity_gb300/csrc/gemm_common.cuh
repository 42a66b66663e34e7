// Pieces shared by the tcgen05 GEMM kernels: the persistent tile order, the
// shared-memory operand descriptor and the bounded mbarrier wait.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fp8hg {
namespace gemm_common {

// Output tile t -> (m-block, n-block).  Tiles are walked in groups of
// kGroupM m-blocks, m fastest within a group: the CTAs resident at any moment
// then share a few A panels and a few B panels, which stay in L2, instead of
// sweeping every B panel once per m-block.
constexpr int kGroupM = 16;
__device__ __forceinline__ void tile_coords(int t, int num_mb, int num_nb, int &mb, int &nb) {
    const int per_group = kGroupM * num_nb;
    const int g = t / per_group, w = t - g * per_group;
    const int rows = min(kGroupM, num_mb - g * kGroupM);
    mb = g * kGroupM + w % rows;
    nb = w / rows;
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(1) << 16;                  // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                  // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
    return d;
}

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting or
// the limit ran out (then the abort flag and the device error word are set).
// check_abort = false is used while draining: keep waiting for the phase up
// to `limit` even though an abort is in progress, and report nothing.
static __device__ bool wait_phase(uint32_t bar, uint32_t parity, uint64_t limit,
                           volatile uint32_t *abort_flag, unsigned int *err, uint32_t who,
                           bool check_abort = true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    uint32_t it = 0;
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
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

}  // namespace gemm_common
}  // namespace fp8hg
