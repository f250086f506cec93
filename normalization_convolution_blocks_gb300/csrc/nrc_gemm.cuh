// Persistent, warp-specialized tcgen05 GEMM skeleton shared by the three
// blocks.  One CTA per SM walks a static round-robin list of 128 x BN output
// tiles and computes D[128 x BN] = A[128 x K] * B[BN x K]^T:
//
//   * A (the activation side) is produced by eight prologue warps: each block's
//     own load-and-transform, split into bf16 parts and written straight into
//     tensor memory with tcgen05.st; the MMA reads A from TMEM.  With a staged
//     A source (Prob::kStagedA) one thread copies each stage's raw input box
//     into a ring of D shared-memory slots with tiled TMA copies
//     (cp.async.bulk.tensor) and the prologue warps transform from there;
//     otherwise each prologue warp loads its raw values into registers one
//     stage ahead.
//   * B (the weight side) is bulk-copied (cp.async.bulk) from a pre-packed
//     global image into a ring of shared-memory stages in the 128-byte swizzle
//     layout the MMA's shared-memory descriptor expects.
//   * The fp32 accumulator lives in TMEM; the epilogue warps drain it.  With
//     cfg.split_h = H > 0 the accumulator's two column halves are handed over
//     separately at tile boundaries: the MMAs finish half A over the tile's
//     last H stages (all resident) before half B, so the epilogue starts on
//     half A while half B is still being computed; and the next tile's first
//     H stages run on half A as soon as it is drained, before half B is.
//
// Keeping A out of shared memory leaves shared-memory bandwidth to the weight
// stream alone, which the MMAs read at 64 B/clk at full rate.
//
// fp32 storage runs three bf16 MMAs per K step (hi*hi + lo*hi + hi*lo, with
// v = hi + lo split in bf16): products exact to ~2^-16 relative, accumulated in
// fp32.  bf16 storage runs one.
//
// Start-up: the copy warps (0, 14) issue the first stages at once while warps
// 1-13 stage the block's parameters and allocate TMEM.  A kernel launched
// behind the one writing its B image (programmatic dependent launch) waits for
// it in the B producer only; a problem that writes its B image in its own
// setup (one wave, cooperative launch) has the B producer wait for all CTAs.
//
// Warp roles (480 threads):
//   warp 0      B producer: one thread issues the bulk copies
//   warp 1      allocates all 512 TMEM columns; one thread issues the MMAs
//   warps 2-9   A producers: warp w owns TMEM lanes 32*(w%4).. (tile rows), K half (w-2)/4
//   warps 10-13 epilogue: warp w drains TMEM lanes 32*(w%4)..
//   warp 14     A-source copies (staged A): one thread issues the TMA boxes
//
// Shared memory: [B ring][A-source ring: D slots][barriers, TMEM slot, abort
// flag][the block's extra bytes].
//
// TMEM columns: [0, BN) accumulator; [256, 512) A ring, stage s at
// 256 + s*32*NP (hi part: 32 columns = 64 bf16 of K; then the lo part).
#pragma once
#include <cstdint>

#include "nrc_ptx.cuh"

namespace nrc {

constexpr int kThreads = 480;
constexpr int kBM = 128;            // rows of a tile (MMA M)
constexpr int kBK = 64;             // K elements per stage (one 128-byte swizzle row)
constexpr int kUMMA_K = 16;         // K of one bf16 MMA
constexpr int kMaxStages = 8;
constexpr int kProducerWarps = 8;
constexpr int kMaxXDepth = 8;       // A-source ring slots (staged A)
constexpr int kNumBars = 4 * kMaxStages + 5 + 2 * kMaxXDepth;
constexpr int kMaxSmemBytes = 232448;          // 227 KB opt-in per CTA
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemARing = 256;           // first column of the A ring

enum WaitSite : int {
    kSiteBEmpty = 1, kSiteAEmpty = 2, kSiteAccEmpty = 3, kSiteFullA = 4, kSiteFullB = 5,
    kSiteAccFull = 6, kSiteFullX = 7, kSiteEmptyX = 8, kSiteGridBarrier = 9, kSiteBImage = 10
};

struct GemmCfg {
    int BN;                 // tile columns (multiple of 16, <= 256)
    int num_tiles;
    int num_kiters;         // K stages per tile
    int b_stages;           // depth of the shared-memory B ring
    uint32_t b_stage_bytes; // NP * BN * 128
    int x_depth;            // A-source ring slots (0: A loaded to registers)
    uint32_t x_box_bytes;   // bytes of one slot: one stage's box (a multiple of 128)
    int split_h;            // >0: hand the accumulator over in column halves, H stages at
                            // each tile end (H <= both ring depths, 2H <= num_kiters)
    int* status;            // device status word
    unsigned long long timeout_ns;
    int b_after_prev;       // B image written by the previous kernel of the stream, which
                            // may still run (programmatic dependent launch): the B
                            // producer waits for it (griddepcontrol.wait) first
};

// Shared-memory bookkeeping after the B stages and A-source slots: barriers
// and two words.
__host__ __device__ constexpr uint32_t gemm_bookkeeping_bytes() {
    return (((uint32_t)kNumBars * 8u + 16u) + 63u) & ~63u;
}

template <int NP>
__device__ __forceinline__ void split_store_a(uint32_t taddr_hi, const float (&v)[32]) {
    uint32_t h[16];
    if constexpr (NP == 2) {
        uint32_t l[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) split_bf16x2(v[2 * e], v[2 * e + 1], h[e], l[e]);
        tmem_st16(taddr_hi, h);
        tmem_st16(taddr_hi + 32u, l);
    } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) h[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
        tmem_st16(taddr_hi, h);
    }
}

// Prob must provide:
//   struct Params; struct Tile;
//   static __device__ Tile tile_info(const Params&, int tile)
//   static __device__ void setup(const Params&, uint8_t* extra, int tid, int nthreads)
//        -> stages the block's parameters in the extra bytes; run by warps 1-13
//           (tid in [0, nthreads)) while the copy warps issue the first stages
//   static __device__ uint32_t* b_ready_counter(const Params&)
//        -> non-NULL when setup also writes part of the B image in global memory:
//           each CTA then arrives on it once setup is done and the B producer
//           waits (bounded) until all gridDim.x have (all CTAs resident)
//   static __device__ void load_a(const Params&, const Tile&, int kiter, int row, int k0,
//                                 float (&v)[32])
//        -> issues the loads of the raw values A[row][kiter*64 + k0 .. +32)
//   static __device__ void finish_a(const Params&, const uint8_t* extra, const Tile&,
//                                   int kiter, int row, int k0, float (&v)[32])
//        -> the block's transform, in place (runs after the loads have landed)
//   static constexpr bool kStagedA; and when it is true:
//   static __device__ void issue_a_box(const Params&, const Tile&, int kiter,
//                                      uint32_t dst_smem, uint32_t bar)
//        -> issues the TMA copy of the raw input of the whole stage into a slot,
//           completing on bar (the caller arms it)
//   static __device__ void read_a(const Params&, const uint8_t* extra, const Tile&,
//                                 int kiter, int row, int k0, int lane, uint32_t box_smem,
//                                 float (&v)[32])
//        -> A[row][kiter*64 + k0 .. +32) from the landed slot, transform applied
//   static __device__ const void* b_src(const Params&, const Tile&, int kiter)
//        -> packed B image of the stage: NP parts of BN rows x 128 B, swizzled
//   static constexpr bool kPackedA
//        -> (NP == 1) read_a returns the 16 bf16 pairs already packed, their bits
//           in v[0..16), stored to TMEM as they are
//   template <class Acquire, class Release>
//   static __device__ bool epilogue(const Params&, const uint8_t* extra, const Tile&,
//                                   int quarter, int lane, uint32_t taddr, int BN,
//                                   int halves, Acquire& acquire, Release& release)
//        -> may issue loads that do not need the accumulator, then for each of the
//           `halves` column halves (1: the whole tile; 2: [0, BN/2) then
//           [BN/2, BN)) calls acquire(h) before reading it (false = pipeline
//           aborted, return false) and release(h) once it has read it; drains
//           TMEM columns [taddr, taddr + BN) of its lane quarter (every lane
//           executes the tcgen05.ld calls)
template <class Prob, int NP>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ typename Prob::Params p, const GemmCfg cfg) {
    using Tile = typename Prob::Tile;
    constexpr int SA = (int)((kTmemCols - kTmemARing) / (32u * NP));   // A ring depth
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived by pointer arithmetic so every pointer
    // into it stays in the shared state space (native shared loads/stores).
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int SB = cfg.b_stages;
    uint8_t* xslots = smem + (size_t)SB * cfg.b_stage_bytes;
    const size_t x_bytes = (size_t)cfg.x_depth * cfg.x_box_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(xslots + x_bytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint8_t* extra = reinterpret_cast<uint8_t*>(bars) + gemm_bookkeeping_bytes();

    const uint32_t bar0 = smem_u32(bars);
    auto a_full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto a_empty = [&](int s) { return bar0 + 8u * (uint32_t)(kMaxStages + s); };
    auto b_full = [&](int s) { return bar0 + 8u * (uint32_t)(2 * kMaxStages + s); };
    auto b_empty = [&](int s) { return bar0 + 8u * (uint32_t)(3 * kMaxStages + s); };
    // Accumulator column half h: full (MMA commit) / empty (epilogue warps).
    const uint32_t drain_bar = bar0 + 8u * (uint32_t)(4 * kMaxStages);
    auto acc_full = [&](int h) { return drain_bar + 8u + 16u * (uint32_t)h; };
    auto acc_empty = [&](int h) { return drain_bar + 16u + 16u * (uint32_t)h; };
    // A-source slot j: full (TMA complete_tx) / empty (producer warps)
    auto x_full = [&](int j) { return bar0 + 8u * (uint32_t)(4 * kMaxStages + 5 + j); };
    auto x_empty = [&](int j) {
        return bar0 + 8u * (uint32_t)(4 * kMaxStages + 5 + kMaxXDepth + j);
    };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a kernel launched behind this one may start launching (it waits for our
    // completion before reading our results)
    griddep_launch_dependents();
    const int BN = cfg.BN;
    WaitCtx ctx{abort_flag, cfg.status, cfg.timeout_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; ++s) {
            mbar_init(a_full(s), 8);      // one arrival per A-producer warp
            mbar_init(a_empty(s), 1);     // MMA commit
        }
        for (int s = 0; s < SB; ++s) {
            mbar_init(b_full(s), 1);      // producer's arrive.expect_tx
            mbar_init(b_empty(s), 1);     // MMA commit
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(acc_full(h), 1);    // MMA commit
            mbar_init(acc_empty(h), 4);   // one arrival per epilogue warp
        }
        mbar_init(drain_bar, 1);
        for (int j = 0; j < cfg.x_depth; ++j) {
            mbar_init(x_full(j), 1);                  // the issuer's arrive.expect_tx
            mbar_init(x_empty(j), kProducerWarps);    // one arrival per A-producer warp
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();                              // barriers initialised
    // The copy warps (0 and 14) start at once; the others stage the block's
    // parameters and allocate TMEM meanwhile, then meet at named barrier 2.
    uint32_t tmem_base = 0;
    if (warp != 0 && warp != 14) {
        Prob::setup(p, extra, (int)threadIdx.x - 32, kThreads - 64);
        if (warp == 1) {
            tmem_alloc(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
        named_bar_sync(2, kThreads - 64);
        tc_fence_after();
        tmem_base = *tmem_slot;
        if (threadIdx.x == 32) {
            if (uint32_t* c = Prob::b_ready_counter(p)) {
                __threadfence();
                atomicAdd(c, 1u);
            }
        }
    }

    if (warp == 0) {
        // ------------------------------------------------------------ B producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed_parity[kMaxStages];
            bool armed[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) armed[s] = false;
            bool ok = true;
            if (cfg.b_after_prev) griddep_wait();
            if (uint32_t* c = Prob::b_ready_counter(p)) {
                // the B image is written by all CTAs' setup: wait for every one
                const uint64_t t0 = globaltimer_ns();
                while (ld_acquire_gpu(c) < gridDim.x) {
                    if (globaltimer_ns() - t0 > cfg.timeout_ns) {
                        record_status(cfg.status, kStatusTimeout, kSiteBImage);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    __nanosleep(64);
                }
                fence_proxy_async_global();
            }
            for (int tile = blockIdx.x; ok && tile < cfg.num_tiles; tile += gridDim.x) {
                const Tile tl = Prob::tile_info(p, tile);
                for (int k = 0; k < cfg.num_kiters; ++k) {
                    if (!mbar_wait(b_empty(stage), phase ^ 1u, ctx, kSiteBEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(b_full(stage), cfg.b_stage_bytes);
                    bulk_g2s(smem_u32(smem + (size_t)stage * cfg.b_stage_bytes),
                             Prob::b_src(p, tl, k), cfg.b_stage_bytes, b_full(stage));
                    armed[stage] = true;
                    armed_parity[stage] = phase;
                    if (++stage == SB) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // Let every copy still in flight land before the CTA can exit.
                for (int s = 0; s < SB; ++s)
                    if (armed[s]) mbar_wait_drain(b_full(s), armed_parity[s], 200000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const int H = cfg.split_h;
            const int HB = BN / 2;                      // columns of a half
            const uint32_t idesc_full = idesc_bf16_f32(kBM, BN);
            const uint32_t idesc_half = idesc_bf16_f32(kBM, HB);
            int sa = 0, sb = 0;
            uint32_t pha = 0, phb = 0;
            bool ok = true;
            int it = 0;
            // Ring slot and phase i stages past the cursor (i < ring depth).
            auto a_at = [&](int i, int& s, uint32_t& ph) {
                s = sa + i;
                ph = pha;
                if (s >= SA) { s -= SA; ph ^= 1u; }
            };
            auto b_at = [&](int i, int& s, uint32_t& ph) {
                s = sb + i;
                ph = phb;
                if (s >= SB) { s -= SB; ph ^= 1u; }
            };
            auto wait_stage = [&](int i) -> bool {
                int s;
                uint32_t ph;
                a_at(i, s, ph);
                if (!mbar_wait(a_full(s), ph, ctx, kSiteFullA)) return false;
                b_at(i, s, ph);
                if (!mbar_wait(b_full(s), ph, ctx, kSiteFullB)) return false;
                tc_fence_after();
                return true;
            };
            // Descriptor of B ring slot 0; slot s, row c0 lies (s*stage + c0*128)
            // bytes further, i.e. that >> 4 more in the start-address field
            // (the ring lies far below the field's 256 KB limit).
            const uint64_t bdesc0 = sw128_kmajor_desc(smem_u32(smem));
            const uint32_t a_ring = tmem_base + kTmemARing;
            // MMAs of the stage i past the cursors into columns [c0, c0 + n) (B
            // rows c0 ..); `first` starts that column range afresh.
            auto mma_stage = [&](int i, int c0, uint32_t idesc, bool first) {
                int s_a, s_b;
                uint32_t ph;
                a_at(i, s_a, ph);
                b_at(i, s_b, ph);
                const uint64_t bd =
                    bdesc0 + (uint64_t)(((uint32_t)s_b * cfg.b_stage_bytes + (uint32_t)c0 * 128u) >> 4);
                mma_stage_bf16<NP>(tmem_base + (uint32_t)c0, a_ring + (uint32_t)(s_a * 32 * NP), bd,
                                   bd + (uint64_t)(((uint32_t)BN * 128u) >> 4), idesc,
                                   first ? 0u : 1u);
            };
            // Frees the stage at the cursors once its MMAs finish; advances.
            auto retire = [&]() {
                mma_commit(a_empty(sa));
                mma_commit(b_empty(sb));
                if (++sa == SA) { sa = 0; pha ^= 1u; }
                if (++sb == SB) { sb = 0; phb ^= 1u; }
            };
            for (int tile = blockIdx.x; ok && tile < cfg.num_tiles; tile += gridDim.x, ++it) {
                const uint32_t epar = ((uint32_t)it & 1u) ^ 1u;   // previous use drained
                if (H == 0) {
                    if (!mbar_wait(acc_empty(0), epar, ctx, kSiteAccEmpty)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int k = 0; k < cfg.num_kiters; ++k) {
                        if (!wait_stage(0)) {
                            ok = false;
                            break;
                        }
                        mma_stage(0, 0, idesc_full, k == 0);
                        retire();
                    }
                    if (!ok) break;
                    mma_commit(acc_full(0));           // accumulator ready for the epilogue
                    continue;
                }
                // head: the first H stages on half A as soon as it is drained,
                // then on half B
                if (!mbar_wait(acc_empty(0), epar, ctx, kSiteAccEmpty)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int i = 0; i < H && ok; ++i) {
                    ok = wait_stage(i);
                    if (ok) mma_stage(i, 0, idesc_half, i == 0);
                }
                if (!ok) break;
                if (!mbar_wait(acc_empty(1), epar, ctx, kSiteAccEmpty)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int i = 0; i < H; ++i) {
                    mma_stage(0, HB, idesc_half, i == 0);
                    retire();
                }
                // body: full width
                for (int k = H; k < cfg.num_kiters - H; ++k) {
                    if (!wait_stage(0)) {
                        ok = false;
                        break;
                    }
                    mma_stage(0, 0, idesc_full, false);
                    retire();
                }
                if (!ok) break;
                // tail: the last H stages on half A, which is then complete,
                // then on half B
                for (int i = 0; i < H && ok; ++i) {
                    ok = wait_stage(i);
                    if (ok) mma_stage(i, 0, idesc_half, false);
                }
                if (!ok) break;
                mma_commit(acc_full(0));
                for (int i = 0; i < H; ++i) {
                    mma_stage(0, HB, idesc_half, false);
                    retire();
                }
                mma_commit(acc_full(1));
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
        const int k0 = khalf * 32;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        int sa = 0;
        uint32_t pha = 0;
        auto advance = [&](int& t, int& kk, Tile& tl) {
            if (++kk == cfg.num_kiters) {
                kk = 0;
                t += gridDim.x;
                if (t < cfg.num_tiles) tl = Prob::tile_info(p, t);
            }
        };
        // Waits for a free A-ring stage, writes v into it and publishes it.
        // Returns false when the pipeline is being aborted.
        auto store_a = [&](const float (&v)[32]) -> bool {
            int w_ok = 1;
            if (lane == 0) w_ok = mbar_wait(a_empty(sa), pha ^ 1u, ctx, kSiteAEmpty);
            w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
            if (!w_ok) return false;
            tc_fence_after();
            const uint32_t ta = tmem_base + lane_off + kTmemARing + (uint32_t)(sa * 32 * NP) +
                                (uint32_t)(k0 / 2);
            if constexpr (Prob::kPackedA && NP == 1) {
                // already packed bf16 pairs (v[0..16) hold their bits)
                uint32_t h[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) h[e] = __float_as_uint(v[e]);
                tmem_st16(ta, h);
            } else {
                split_store_a<NP>(ta, v);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full(sa));
            if (++sa == SA) { sa = 0; pha ^= 1u; }
            return true;
        };
        if constexpr (Prob::kStagedA) {
            // Stage k's raw input sits in slot k % D once x_full completes; the
            // warp reads its 32 rows x 32 channels and releases the slot.
            const int D = cfg.x_depth;
            const uint32_t slot0 = smem_u32(xslots);
            int ptile = blockIdx.x, pk = 0, pslot = 0;
            uint32_t pphase = 0;
            Tile ptl{};
            if (ptile < cfg.num_tiles) ptl = Prob::tile_info(p, ptile);
            while (ptile < cfg.num_tiles) {
                int w_ok = 1;
                if (lane == 0) w_ok = mbar_wait(x_full(pslot), pphase, ctx, kSiteFullX);
                w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
                if (!w_ok) break;
                // The phase is complete (lane 0 saw it) and stays so until the
                // slot is released: every lane's own test succeeds at once and
                // orders its reads after the copy.
                (void)mbar_try_wait(x_full(pslot), pphase);
                float v[32];
                Prob::read_a(p, extra, ptl, pk, row, k0, lane,
                             slot0 + (uint32_t)pslot * cfg.x_box_bytes, v);
                __syncwarp();
                if (lane == 0) mbar_arrive(x_empty(pslot));
                if (++pslot == D) { pslot = 0; pphase ^= 1u; }
                if (!store_a(v)) break;
                advance(ptile, pk, ptl);
            }
        } else {
            // Raw values loaded into registers, one stage ahead.
            int ltile = blockIdx.x, lk = 0;
            int ptile = blockIdx.x, pk = 0;
            Tile ltl{}, ptl{};
            if (ltile < cfg.num_tiles) ltl = Prob::tile_info(p, ltile);
            ptl = ltl;
            auto process = [&](float (&v)[32]) -> bool {
                Prob::finish_a(p, extra, ptl, pk, row, k0, v);
                if (!store_a(v)) return false;
                advance(ptile, pk, ptl);
                return true;
            };
            float v0[32], v1[32];
            if (ltile < cfg.num_tiles) {
                Prob::load_a(p, ltl, lk, row, k0, v0);
                advance(ltile, lk, ltl);
            }
            while (ptile < cfg.num_tiles) {
                if (ltile < cfg.num_tiles) {
                    Prob::load_a(p, ltl, lk, row, k0, v1);
                    advance(ltile, lk, ltl);
                }
                if (!process(v0) || ptile >= cfg.num_tiles) break;
                if (ltile < cfg.num_tiles) {
                    Prob::load_a(p, ltl, lk, row, k0, v0);
                    advance(ltile, lk, ltl);
                }
                if (!process(v1)) break;
            }
        }
    } else if (warp == 14) {
        // ------------------------------------------------------------ A-source copies
        if constexpr (Prob::kStagedA) {
            if (lane == 0) {
                const int D = cfg.x_depth;
                const uint32_t slot0 = smem_u32(xslots);
                int slot = 0;
                uint32_t phase = 0;
                uint32_t armed = 0, armed_par = 0;     // bit j: copy in flight / its parity
                bool ok = true;
                for (int tile = blockIdx.x; ok && tile < cfg.num_tiles; tile += gridDim.x) {
                    const Tile tl = Prob::tile_info(p, tile);
                    for (int k = 0; k < cfg.num_kiters; ++k) {
                        if (!mbar_wait(x_empty(slot), phase ^ 1u, ctx, kSiteEmptyX)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(x_full(slot), cfg.x_box_bytes);
                        Prob::issue_a_box(p, tl, k, slot0 + (uint32_t)slot * cfg.x_box_bytes,
                                          x_full(slot));
                        armed |= 1u << slot;
                        armed_par = (armed_par & ~(1u << slot)) | (phase << slot);
                        if (++slot == D) { slot = 0; phase ^= 1u; }
                    }
                }
                if (!ok) {
                    // Let every copy still in flight land before the CTA can exit.
                    for (int j = 0; j < D; ++j)
                        if ((armed >> j) & 1u)
                            mbar_wait_drain(x_full(j), (armed_par >> j) & 1u, 200000000ull);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        int it = 0;
        for (int tile = blockIdx.x; tile < cfg.num_tiles; tile += gridDim.x, ++it) {
            const Tile tl = Prob::tile_info(p, tile);
            // The block's epilogue calls acquire(h) once it has issued whatever
            // it can load before column half h is ready, release(h) once it
            // has read it.
            auto acquire = [&](int h) -> bool {
                int w_ok = 1;
                if (lane == 0)
                    w_ok = mbar_wait(acc_full(h), (uint32_t)it & 1u, ctx, kSiteAccFull);
                w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
                if (w_ok) tc_fence_after();
                return w_ok != 0;
            };
            auto release = [&](int h) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty(h));
            };
            if (!Prob::epilogue(p, extra, tl, quarter, lane,
                                tmem_base + ((uint32_t)(quarter * 32) << 16), BN,
                                cfg.split_h > 0 ? 2 : 1, acquire, release))
                break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace nrc
