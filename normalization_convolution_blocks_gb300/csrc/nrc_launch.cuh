// Host-side planning and launch of gemm_kernel (shared by the block TUs).
#pragma once
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <utility>

#include "nrc_gemm.cuh"
#include "nrc_host.h"

namespace nrc {

struct GemmPlan {
    int BN, num_tiles, num_kiters, b_stages, x_depth;
    int split_h;            // accumulator handed over in column halves, H stages (0: whole)
    bool coop;              // cooperative launch: all CTAs resident at once (grid-wide waits)
    bool b_after_prev;      // programmatic dependent launch after the kernel writing B
    uint32_t b_stage_bytes, x_box_bytes, extra_bytes, smem_bytes;
};

// Shared-memory split.  Register-loaded A: as many B stages as fit (at most
// kMaxStages).  Staged A (x_box_bytes > 0, one slot per stage): the deepest B
// ring (at most 4) that still leaves two A-source slots, then as many slots as
// fit (at most kMaxXDepth).  b_stages < 2 or x_depth < 2 (staged) means the
// problem does not fit.
inline GemmPlan make_gemm_plan(int BN, int num_tiles, int num_kiters, int NP,
                               uint32_t extra_bytes, uint32_t x_box_bytes = 0) {
    GemmPlan g{};
    g.BN = BN;
    g.num_tiles = num_tiles;
    g.num_kiters = num_kiters;
    g.b_stage_bytes = (uint32_t)NP * (uint32_t)BN * 128u;
    g.x_box_bytes = x_box_bytes;
    g.extra_bytes = extra_bytes;
    const uint32_t fixed = 1024u + gemm_bookkeeping_bytes() + extra_bytes;
    const long long avail = (long long)kMaxSmemBytes - fixed;
    if (x_box_bytes == 0) {
        g.x_depth = 0;
        g.b_stages = (int)std::min<long long>(kMaxStages, avail / g.b_stage_bytes);
    } else {
        g.b_stages = (int)std::min<long long>(4, (avail - 2LL * x_box_bytes) / g.b_stage_bytes);
        g.x_depth = (int)std::min<long long>(
            kMaxXDepth, (avail - (long long)std::max(g.b_stages, 0) * g.b_stage_bytes) /
                            (long long)x_box_bytes);
    }
    g.smem_bytes = fixed + (uint32_t)std::max(g.b_stages, 0) * g.b_stage_bytes +
                   (uint32_t)std::max(g.x_depth, 0) * x_box_bytes;
    return g;
}

template <class Prob, int NP>
inline nrc_status launch_gemm(const char* name, const typename Prob::Params& p,
                              const GemmPlan& pl, cudaStream_t stream) {
    if (pl.b_stages < 2) return NRC_ERR_UNSUPPORTED;
    if (Prob::kStagedA != (pl.x_box_bytes > 0) || (Prob::kStagedA && pl.x_depth < 2))
        return NRC_ERR_UNSUPPORTED;
    auto kern = gemm_kernel<Prob, NP>;
    // The opt-in shared-memory size is raised once per device and kernel
    // (to the maximum), so calls issue no host API work between launches.
    static std::atomic<unsigned long long> smem_set_mask{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NRC_ERR_CUDA;
    if (!(smem_set_mask.load() & (1ull << dev))) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kMaxSmemBytes) != cudaSuccess)
            return NRC_ERR_CUDA;
        smem_set_mask.fetch_or(1ull << dev);
    }
    if (pl.smem_bytes > (uint32_t)kMaxSmemBytes) return NRC_ERR_UNSUPPORTED;
    GemmCfg cfg{};
    cfg.BN = pl.BN;
    cfg.num_tiles = pl.num_tiles;
    cfg.num_kiters = pl.num_kiters;
    cfg.b_stages = pl.b_stages;
    cfg.b_stage_bytes = pl.b_stage_bytes;
    cfg.x_depth = pl.x_depth;
    cfg.x_box_bytes = pl.x_box_bytes;
    cfg.split_h = pl.split_h;
    {   // the halves need both rings to hold H stages at once, and whole halves
        constexpr int SA = (int)((kTmemCols - kTmemARing) / (32u * NP));
        if (pl.split_h < 0 || pl.split_h > SA || pl.split_h > pl.b_stages ||
            2 * pl.split_h > pl.num_kiters || (pl.split_h > 0 && pl.BN % 128 != 0))
            return NRC_ERR_UNSUPPORTED;
    }
    cfg.status = device_status_ptr();
    cfg.timeout_ns = wait_timeout_ns();
    cfg.b_after_prev = pl.b_after_prev ? 1 : 0;
    if (cfg.status == nullptr) return NRC_ERR_CUDA;
    // Each CTA allocates all 512 TMEM columns, so one CTA per SM.
    if (pl.coop) {
        // all CTAs resident (they wait on one another): the driver refuses the
        // launch if they cannot be
        if (!device_coop_launch()) return NRC_ERR_UNSUPPORTED;
        cudaLaunchConfig_t lc{};
        lc.gridDim = dim3((unsigned)std::min(pl.num_tiles, device_sm_count()));
        lc.blockDim = dim3(kThreads);
        lc.dynamicSmemBytes = pl.smem_bytes;
        lc.stream = stream;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeCooperative;
        at[0].val.cooperative = 1;
        lc.attrs = at;
        lc.numAttrs = 1;
        TraceScope ts(name, stream);
        const cudaError_t e = cudaLaunchKernelEx(&lc, kern, p, cfg);
        if (e == cudaErrorCooperativeLaunchTooLarge) {
            // not all CTAs can be resident now (the GPU is shared): the caller
            // takes its non-cooperative path
            (void)cudaGetLastError();
            return NRC_ERR_UNSUPPORTED;
        }
        if (e != cudaSuccess) return cuda_status(e);
        return cuda_status(cudaGetLastError());
    }
    const int grid = std::min(pl.num_tiles, device_sm_count());
    if (pl.b_after_prev) {
        // may start while the kernel writing B finishes; the B producer waits
        cudaLaunchConfig_t lc{};
        lc.gridDim = dim3((unsigned)grid);
        lc.blockDim = dim3(kThreads);
        lc.dynamicSmemBytes = pl.smem_bytes;
        lc.stream = stream;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        lc.attrs = at;
        lc.numAttrs = 1;
        TraceScope ts(name, stream);
        const cudaError_t e = cudaLaunchKernelEx(&lc, kern, p, cfg);
        if (e != cudaSuccess) return cuda_status(e);
        return cuda_status(cudaGetLastError());
    }
    {
        TraceScope ts(name, stream);
        kern<<<grid, kThreads, pl.smem_bytes, stream>>>(p, cfg);
    }
    return cuda_status(cudaGetLastError());
}

// Launch that may start while the previous kernel of the stream finishes
// (programmatic dependent launch): the kernel must griddep_wait before it
// reads that kernel's results.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_after_prev(void (*kern)(KArgs...), dim3 grid, dim3 block,
                                     cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t lc{};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = 0;
    lc.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kern, std::forward<Args>(args)...);
}

inline int elementwise_grid(size_t units, int per_sm = 8) {
    const size_t g = std::min<size_t>((units + 255) / 256, (size_t)device_sm_count() * per_sm);
    return (int)std::max<size_t>(g, 1);
}

}  // namespace nrc
