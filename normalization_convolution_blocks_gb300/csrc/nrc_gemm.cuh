// Persistent, warp-specialized tcgen05 GEMM skeleton shared by the three
// blocks.  One CTA per SM walks a static round-robin list of 128 x BN output
// tiles; D = A * B^T with A (128 x K) produced in shared memory by eight
// "prologue" warps (each block's own load-and-transform), B (BN x K) bulk-copied
// from a pre-packed global image, and the fp32 accumulator in TMEM (two
// buffers, so the epilogue of one tile overlaps the mainloop of the next).
//
// fp32 storage runs three bf16 MMAs per K step (hi*hi + lo*hi + hi*lo, with
// v = hi + lo split in bf16): products exact to ~2^-16 relative, accumulated in
// fp32 on the tensor cores.  bf16 storage runs one.
//
// Warp roles (448 threads):
//   warp 0      B producer: one thread issues cp.async.bulk per stage
//   warp 1      TMEM allocator; one thread issues tcgen05.mma and commits
//   warps 2-9   A producers: warp w writes rows 32*(w%4).. of the stage, K half (w-2)/4
//   warps 10-13 epilogue: warp w drains TMEM lanes 32*(w%4).. (its lane quarter)
#pragma once
#include <cstdint>

#include "nrc_ptx.cuh"

namespace nrc {

constexpr int kThreads = 448;
constexpr int kBM = 128;            // rows of a tile (MMA M)
constexpr int kBK = 64;             // K elements per stage (one 128-byte swizzle row)
constexpr int kUMMA_K = 16;         // K of one bf16 MMA
constexpr uint32_t kATileBytes = kBM * 128;   // one bf16 part of an A stage
constexpr int kMaxStages = 8;
constexpr int kMaxSmemBytes = 232448;          // 227 KB opt-in per CTA

enum WaitSite : int {
    kSiteBEmpty = 1, kSiteAEmpty = 2, kSiteAccEmpty = 3, kSiteFullA = 4, kSiteFullB = 5,
    kSiteAccFull = 6
};

struct GemmCfg {
    int BN;                 // tile columns (multiple of 16, <= 256)
    int num_tiles;
    int num_kiters;         // K stages per tile
    int stages;             // pipeline depth
    uint32_t stage_bytes;   // NP * (kATileBytes + BN * 128)
    uint32_t tmem_cols;     // power of two >= 2 * BN
    int* status;            // device status word
    unsigned long long timeout_ns;
};

// Shared-memory footprint of the skeleton's bookkeeping after the stages.
__host__ __device__ constexpr uint32_t gemm_bookkeeping_bytes(int stages) {
    return (uint32_t)(3 * stages + 5) * 8u + 16u;
}

template <int NP>
__host__ __device__ constexpr uint32_t gemm_stage_bytes(int BN) {
    return (uint32_t)NP * (kATileBytes + (uint32_t)BN * 128u);
}

// Prob must provide:
//   struct Params;
//   static constexpr uint32_t extra_smem_bytes(const Params&)   [host]
//   static __device__ void setup(const Params&, uint8_t* extra)         (all threads)
//   static __device__ void fetch_a(const Params&, const uint8_t* extra, int tile,
//                                  int kiter, int row, int k0, float (&v)[32])
//        -> the 32 fp32 values A[row][kiter*64 + k0 .. +32) after the block's transform
//   static __device__ const void* b_src(const Params&, int tile, int kiter)
//        -> packed B image of the stage: NP parts of BN rows x 128 B, swizzled
//   static __device__ void epilogue(const Params&, const uint8_t* extra, int tile, int quarter,
//                                   int lane, uint32_t taddr, int BN)
//        -> drains TMEM columns [taddr, taddr + BN) of its lane quarter (all lanes
//           execute the tcgen05.ld calls)
template <class Prob, int NP>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const typename Prob::Params p, const GemmCfg cfg) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = cfg.stages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)S * cfg.stage_bytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * S + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint8_t* extra = reinterpret_cast<uint8_t*>(tmem_slot + 4);

    const uint32_t bar0 = smem_u32(bars);
    auto full_a = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto full_b = [&](int s) { return bar0 + 8u * (uint32_t)(S + s); };
    auto empty = [&](int s) { return bar0 + 8u * (uint32_t)(2 * S + s); };
    auto acc_full = [&](int a) { return bar0 + 8u * (uint32_t)(3 * S + a); };
    auto acc_empty = [&](int a) { return bar0 + 8u * (uint32_t)(3 * S + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (uint32_t)(3 * S + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BN = cfg.BN;
    const uint32_t b_bytes = (uint32_t)NP * (uint32_t)BN * 128u;
    WaitCtx ctx{abort_flag, cfg.status, cfg.timeout_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_a(s), 8);      // one arrival per A-producer warp
            mbar_init(full_b(s), 1);      // producer's arrive.expect_tx
            mbar_init(empty(s), 1);       // MMA commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full(a), 1);    // MMA commit
            mbar_init(acc_empty(a), 4);   // one arrival per epilogue warp
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    Prob::setup(p, extra);
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), cfg.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    auto stage_ptr = [&](int s) { return smem + (size_t)s * cfg.stage_bytes; };

    if (warp == 0) {
        // ------------------------------------------------------------ B producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed_parity[kMaxStages];
            bool armed[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) armed[s] = false;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < cfg.num_tiles; tile += gridDim.x) {
                for (int k = 0; k < cfg.num_kiters; ++k) {
                    if (!mbar_wait(empty(stage), phase ^ 1u, ctx, kSiteBEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_b(stage), b_bytes);
                    bulk_g2s(smem_u32(stage_ptr(stage) + NP * kATileBytes),
                             Prob::b_src(p, tile, k), b_bytes, full_b(stage));
                    armed[stage] = true;
                    armed_parity[stage] = phase;
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // Let every copy still in flight land before the CTA can exit.
                for (int s = 0; s < S; ++s)
                    if (armed[s]) mbar_wait_drain(full_b(s), armed_parity[s], 200000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kBM, BN);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int tile = blockIdx.x; ok && tile < cfg.num_tiles; tile += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait(acc_empty(acc), acc_phase ^ 1u, ctx, kSiteAccEmpty)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int k = 0; k < cfg.num_kiters; ++k) {
                    if (!mbar_wait(full_a(stage), phase, ctx, kSiteFullA) ||
                        !mbar_wait(full_b(stage), phase, ctx, kSiteFullB)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_hi = smem_u32(stage_ptr(stage));
                    const uint32_t b_hi = a_hi + NP * kATileBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / kUMMA_K; ++kk) {
                        const uint32_t koff = (uint32_t)kk * (kUMMA_K * 2);
                        const uint64_t ad = sw128_kmajor_desc(a_hi + koff);
                        const uint64_t bd = sw128_kmajor_desc(b_hi + koff);
                        mma_bf16_ss(d_tmem, ad, bd, idesc, (k | kk) != 0 ? 1u : 0u);
                        if constexpr (NP == 2) {
                            const uint64_t ad_lo = sw128_kmajor_desc(a_hi + kATileBytes + koff);
                            const uint64_t bd_lo =
                                sw128_kmajor_desc(b_hi + (uint32_t)BN * 128u + koff);
                            mma_bf16_ss(d_tmem, ad_lo, bd, idesc, 1u);
                            mma_bf16_ss(d_tmem, ad, bd_lo, idesc, 1u);
                        }
                    }
                    mma_commit(empty(stage));          // stage free once these MMAs finish
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(acc_full(acc));             // accumulator ready for the epilogue
            }
            if (!ok) {
                // Every MMA issued so far must finish before TMEM/smem go away.
                mma_commit(drain_bar);
                mbar_wait_drain(drain_bar, 0, 200000000ull);
            }
        }
    } else if (warp < 10) {
        // ------------------------------------------------------------ A producers
        const int quarter = warp & 3;
        const int khalf = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        int stage = 0;
        uint32_t phase = 0;
        for (int tile = blockIdx.x; tile < cfg.num_tiles; tile += gridDim.x) {
            bool ok = true;
            for (int k = 0; k < cfg.num_kiters; ++k) {
                float v[32];
                Prob::fetch_a(p, extra, tile, k, row, khalf * 32, v);
                int w_ok = 1;
                if (lane == 0) w_ok = mbar_wait(empty(stage), phase ^ 1u, ctx, kSiteAEmpty);
                w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
                if (!w_ok) { ok = false; break; }
                const uint32_t a_base = smem_u32(stage_ptr(stage));
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t off = sw128_offset((uint32_t)row, (uint32_t)(khalf * 4 + j));
                    if constexpr (NP == 2) {
                        uint32_t h[4], l[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            split_bf16x2(v[8 * j + 2 * e], v[8 * j + 2 * e + 1], h[e], l[e]);
                        st_shared_v4(a_base + off, h[0], h[1], h[2], h[3]);
                        st_shared_v4(a_base + kATileBytes + off, l[0], l[1], l[2], l[3]);
                    } else {
                        st_shared_v4(a_base + off, pack_bf16x2(v[8 * j], v[8 * j + 1]),
                                     pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                     pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                                     pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_a(stage));
                if (++stage == S) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        int it = 0;
        for (int tile = blockIdx.x; tile < cfg.num_tiles; tile += gridDim.x, ++it) {
            const int acc = it & 1;
            const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
            int w_ok = 1;
            if (lane == 0) w_ok = mbar_wait(acc_full(acc), acc_phase, ctx, kSiteAccFull);
            w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
            if (!w_ok) break;
            tc_fence_after();
            const uint32_t taddr =
                tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
            Prob::epilogue(p, extra, tile, quarter, lane, taddr, BN);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(acc));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, cfg.tmem_cols);
    }
}

// Host helpers ------------------------------------------------------------------
inline uint32_t tmem_cols_for(int BN) {
    uint32_t c = 32;
    while (c < (uint32_t)(2 * BN)) c <<= 1;
    return c;
}

}  // namespace nrc
