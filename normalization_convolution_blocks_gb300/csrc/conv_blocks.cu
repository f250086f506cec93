// Conv1d blocks as implicit GEMMs on tcgen05:
//   * pre-norm residual block  out = x + Conv1d(ReLU(BN_eval(x))), k=3, pad=dil
//     ("Kimi-K2.6 l2_p12", problem statement)
//   * Conv1d(k=3, pad=1) + GroupNorm ("FW-GLM-5-1 l2_p35", problem analysis)
//
// GEMM view of one sample n: D[t][o] = sum_tap sum_c z[c][t*stride - pad + tap*dil] * W[o][c][tap]
// (the block: stride 1, three taps, pad = dil; Conv1d + GroupNorm: any kernel
// size, stride, padding and dilation).
// Tile rows are 128 consecutive t, tile columns BN output channels; the K loop
// runs over (tap, 64-channel chunk).  The A operand (activations) is produced
// in tensor memory by the prologue warps: the conv input for the tile's shifted
// window, with BN+ReLU applied (block) and the zero padding applied after it,
// split into bf16 hi/lo parts for fp32 storage.  When the rows of x are 16-byte
// aligned, each stage's shifted window (64 channels x 128 rows of one tap,
// start rounded down to 16 bytes) is gathered as one TMA box, out-of-range rows
// filled by the copy itself; otherwise the prologue warps load x directly.
// The B operand (weights) is repacked once per call into the exact
// shared-memory image the MMA reads: by a repack kernel that the GEMM is
// launched behind (programmatic dependent launch), or, when every tile has its
// own resident CTA (one wave, cooperative launch), inside the GEMM kernel.
// Conv + GroupNorm in one wave also finishes the normalization inside the
// GEMM kernel (statistics exchanged behind a grid-wide barrier); larger
// problems run a finalize kernel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "nrc_launch.cuh"

namespace nrc {

template <typename T>
__device__ __forceinline__ float load_f(const T* p);
template <>
__device__ __forceinline__ float load_f<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_f<__nv_bfloat16>(const __nv_bfloat16* p) {
    const unsigned short u = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float((uint32_t)u << 16);
}

template <typename T>
__device__ __forceinline__ void store_f(T* p, float v);
template <>
__device__ __forceinline__ void store_f<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_f<__nv_bfloat16>(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
}

enum class ConvEpi { kResidual, kGroupStats };

struct ConvParams {
    CUtensorMap xmap;       // x as (L, Cin, N) boxes of (128 + 16/esize) x 64 x 1 (staged A)
    const void* x;          // (N, Cin, L)
    void* out;              // (N, Cout, L)
    int N, Cin, Cout, L;    // L: output length (tile rows, out rows)
    int Lin;                // input length (rows of x); the block has Lin == L
    int pad, dil, stride;   // tap k of output t reads t*stride - pad + k*dil
    int ksz;                // taps of the kernel (3 for the block)
    int n_tt, n_ot, n_chunks, n_kiters, BN;
    // eval-mode BatchNorm of the block's prologue (NULL rm: no BN/ReLU)
    const float *rm, *rv, *gamma, *beta;
    float bn_eps;
    const void* bias;       // (Cout) or NULL
    int bias_off;           // float offset of the staged bias in the extra smem
    int bn2_off;            // bf16 storage: word offset of the BN scale and shift as packed
                            // bf16 pairs (channels 2i, 2i+1), n_chunks*32 words each
    int stage_off;          // byte offset of the bf16 epilogue's two chunk buffers (staged bf16)
    const uint8_t* wpack;   // packed weight image
    // in-kernel weight repack (pack_counter != NULL): every CTA packs a share of
    // the image from w_raw during setup, then arrives on pack_counter (zeroed
    // before the launch); the B producer waits for all CTAs (cooperative launch)
    const void* w_raw;
    uint8_t* wpack_out;
    uint32_t* pack_counter;
    // group statistics (conv + GroupNorm)
    float2* partials;       // [((n*G + g) * n_tt + tt) * 128 + row] = (mean, M2) of the
                            // row's cpg values (count cpg, or 0 for rows past L)
    int G, cpg;
    // conv + GroupNorm in one wave (fused): every tile on its own resident CTA;
    // the host's planning flag (the kernel variant is ConvProblem's ONE_WAVE)
    int fused;
    uint32_t* grid_counter;  // zeroed before the launch; one arrival per CTA
    float4* tile_stats;      // [(n*G + g) * n_tt + tt] = (count, mean, M2, 0) of a tile's group
    const float *gn_gamma, *gn_beta;
    float gn_eps;
    int* status;             // device status word, for the grid barrier's give-up
    unsigned long long timeout_ns;
};

// Shared memory of the fused conv + GroupNorm epilogue: per-warp group
// partials [group][4] (float4), then the per-channel scale and shift.
constexpr int kGnMaxGroups = 256;
constexpr uint32_t kGnFusedBytes = kGnMaxGroups * 4 * 16 + 2 * 256 * 4;

// Chan's pairwise merge of (count, mean, M2) b into a.
__device__ __forceinline__ void chan_merge(float& cnt, float& mean, float& m2, float nb, float mb,
                                           float qb) {
    const float nab = cnt + nb;
    if (nab > 0.f) {
        const float delta = mb - mean;
        const float fb = nb / nab;
        mean += delta * fb;
        m2 += qb + delta * delta * cnt * fb;
        cnt = nab;
    }
}

// Tile index -> (n, t tile, o tile); o tiles of one (n, t) are adjacent, then t,
// so neighbouring CTAs share the x windows (and the +-dil halos) in L2.
struct ConvTile {
    int n, tt, ot;
};
__device__ __forceinline__ ConvTile conv_tile(const ConvParams& p, int tile) {
    ConvTile r;
    r.ot = tile % p.n_ot;
    const int rest = tile / p.n_ot;
    r.tt = rest % p.n_tt;
    r.n = rest / p.n_tt;
    return r;
}

// One 16-byte chunk of the weight image: W (Cout, Cin, ksz) -> for each (o tile,
// tap, 64-channel chunk) the B-stage image, NP parts of BN rows x 64 bf16,
// 128B-swizzled (fp32 split into hi + lo bf16; bf16 copied).  Rows past Cout
// and channels past Cin are zero.  idx enumerates (o tile, K stage, row, chunk).
template <typename T, int NP>
__device__ __forceinline__ void pack_conv_chunk(const T* __restrict__ w,
                                                uint8_t* __restrict__ pack, int Cout, int Cin,
                                                int BN, int n_chunks, int ksz, size_t idx) {
    const int n_kiters = ksz * n_chunks;
    const int j = (int)(idx & 7);
    size_t rest = idx >> 3;
    const int row = (int)(rest % BN);
    rest /= BN;
    const int kiter = (int)(rest % n_kiters);
    const int ot = (int)(rest / n_kiters);
    const int tap = kiter / n_chunks, chunk = kiter % n_chunks;
    const int o = ot * BN + row;
    const int c0 = chunk * kBK + j * 8;
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int c = c0 + e;
        v[e] = (o < Cout && c < Cin) ? load_f<T>(w + ((size_t)o * Cin + c) * ksz + tap) : 0.f;
    }
    const size_t blk = ((size_t)ot * n_kiters + kiter) * NP;
    const uint32_t off = sw128_offset((uint32_t)row, (uint32_t)j);
    uint4* hi = reinterpret_cast<uint4*>(pack + (blk * BN) * 128 + off);
    if constexpr (NP == 2) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_bf16x2(v[2 * e], v[2 * e + 1], h[e], l[e]);
        *hi = make_uint4(h[0], h[1], h[2], h[3]);
        uint4* lo = reinterpret_cast<uint4*>(pack + ((blk + 1) * BN) * 128 + off);
        *lo = make_uint4(l[0], l[1], l[2], l[3]);
    } else {
        // bf16 input: values are already bf16, the repack is exact.
        *hi = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                         pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
    }
}

// Warp-level merge of (count, mean, M2) triples (Chan et al.'s pairwise
// update); every lane ends with the total.  Lanes with count 0 contribute
// nothing.  kFast: the weight nb/nab by the fast division intrinsic (a few ulp;
// both are small exact counts), for the per-tile statistics in the epilogue.
template <bool kFast = false>
__device__ __forceinline__ void warp_merge_stats(float& cnt, float& mean, float& m2) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float nb = __shfl_xor_sync(0xffffffffu, cnt, off);
        const float mb = __shfl_xor_sync(0xffffffffu, mean, off);
        const float qb = __shfl_xor_sync(0xffffffffu, m2, off);
        const float nab = cnt + nb;
        if (nab > 0.f) {
            const float delta = mb - mean;
            const float fb = kFast ? __fdividef(nb, nab) : nb / nab;
            mean = mean + delta * fb;
            m2 = m2 + qb + delta * delta * cnt * fb;
            cnt = nab;
        }
    }
}

// GroupNorm statistics of one row over a 16-channel chunk holding 16/CPG whole
// groups (CPG divides 16): for each group its (mean, M2) over the row's CPG
// values, two-pass in registers, zero for a row outside [0, L) (tw = 0).
// Groups at or past n (channels of the chunk that exist) are skipped.
template <int CPG>
__device__ __forceinline__ void gn_chunk_stats(const float (&v)[16], int n, float tw,
                                               float2* part, size_t group_stride) {
#pragma unroll
    for (int j = 0; j < 16 / CPG; ++j) {
        if (j * CPG >= n) break;
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < CPG; ++i) s += v[j * CPG + i];
        const float m = s * (1.0f / CPG);
        float q = 0.f;
#pragma unroll
        for (int i = 0; i < CPG; ++i) {
            const float d = v[j * CPG + i] - m;
            q = fmaf(d, d, q);
        }
        part[(size_t)j * group_stride] = make_float2(m * tw, q * tw);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// TMEM load of COLS (16, 32 or 64) consecutive columns, one wait.
template <int COLS>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[COLS]) {
    if constexpr (COLS == 16)
        tmem_ld16(taddr, v);
    else if constexpr (COLS == 32)
        tmem_ld32(taddr, v);
    else
        tmem_ld64(taddr, v);
}

// Fused GroupNorm, step 1 for groups of CPG channels (CPG divides 16): the
// accumulator is read COLS columns at a time (one TMEM round trip); for each
// of the NB whole groups in them, the row's mean and M2 over its CPG values
// (two-pass), then the warp's (count, mean, M2) over its valid rows by two
// warp sums, the NB groups' sums interleaved so their shuffle latencies
// overlap.  Lane 0 writes s_part[local group][quarter].
template <int CPG>
__device__ __forceinline__ void gn_tile_stats(const float* bias_s, uint32_t taddr, int ovalid,
                                              int ng, float tw, float inv_nvr, float wcount,
                                              int quarter, int lane, float4* s_part,
                                              bool has_bias) {
    constexpr int COLS = CPG == 1 ? 16 : (CPG <= 4 ? 32 : 64);
    constexpr int NB = COLS / CPG;                      // groups per batch
    for (int cb = 0; cb < ovalid; cb += COLS) {         // COLS divides 256: no batch
        float v[COLS];                                  // crosses the accumulator
        tmem_ld_cols<COLS>(taddr + (uint32_t)cb, v);
#pragma unroll
        for (int i = 0; i < COLS; ++i)
            v[i] = cb + i < ovalid ? (has_bias ? v[i] + bias_s[cb + i] : v[i]) : 0.f;
        float m[NB], q[NB];
#pragma unroll
        for (int k = 0; k < NB; ++k) {
            float s1 = 0.f;
#pragma unroll
            for (int i = 0; i < CPG; ++i) s1 += v[k * CPG + i];
            m[k] = s1 * (1.0f / CPG);
            float s2 = 0.f;
#pragma unroll
            for (int i = 0; i < CPG; ++i) {
                const float d = v[k * CPG + i] - m[k];
                s2 = fmaf(d, d, s2);
            }
            q[k] = s2;
        }
        float S[NB];
#pragma unroll
        for (int k = 0; k < NB; ++k) S[k] = m[k] * tw;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int k = 0; k < NB; ++k) S[k] += __shfl_xor_sync(0xffffffffu, S[k], off);
#pragma unroll
        for (int k = 0; k < NB; ++k) {
            S[k] *= inv_nvr;                            // the warp's mean of the group
            const float d = m[k] - S[k];
            q[k] = tw * (q[k] + (float)CPG * d * d);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int k = 0; k < NB; ++k) q[k] += __shfl_xor_sync(0xffffffffu, q[k], off);
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < NB; ++k) {
                const int gl = cb / CPG + k;
                if (gl < ng) s_part[gl * 4 + quarter] = make_float4(wcount, S[k], q[k], 0.f);
            }
        }
    }
}

// ONE_WAVE: every tile on its own CTA, all resident (cooperative launch).  The
// kernel then also repacks the weight image (see pack_counter) and, for
// GroupNorm, finishes the normalization (gn_fused).  A separate instantiation,
// so the kernels of larger problems carry none of it.
template <typename T, ConvEpi EPI, bool STAGED, bool ONE_WAVE = false>
struct ConvProblem {
    using Params = ConvParams;
    using Tile = ConvTile;
    static constexpr bool kStagedA = STAGED;
    static constexpr int kAlign = 16 / (int)sizeof(T);   // box starts on 16-byte boundaries
    static constexpr int kBoxW = kBM + kAlign;            // rows (time positions) per box
    static constexpr uint32_t kBoxBytes = (uint32_t)(kBoxW * kBK * sizeof(T));
    // Staged bf16 residual epilogue: two chunk buffers of 16 channels x 128 rows.
    static constexpr uint32_t kChunkBufBytes = 16u * kBM * 2u;

    static __device__ __forceinline__ Tile tile_info(const Params& p, int tile) {
        return conv_tile(p, tile);
    }

    // Non-NULL: the B producer waits until every CTA has packed its share.
    static __device__ __forceinline__ uint32_t* b_ready_counter(const Params& p) {
        if constexpr (ONE_WAVE)
            return p.pack_counter;
        else
            return nullptr;
    }

    static __device__ void setup(const Params& p, uint8_t* extra, int tid, int nthr) {
        if constexpr (ONE_WAVE) {
            // this CTA's share of the weight image, published to the copy engine.
            // Unit u goes to CTA u % gridDim.x, so every CTA packs about the
            // same number of units: the B producers wait for the slowest CTA.
            constexpr int NP = sizeof(T) == 4 ? 2 : 1;
            const size_t units = (size_t)p.n_ot * p.n_kiters * p.BN * 8;
            for (size_t idx = (size_t)tid * gridDim.x + blockIdx.x; idx < units;
                 idx += (size_t)gridDim.x * nthr)
                pack_conv_chunk<T, NP>(static_cast<const T*>(p.w_raw), p.wpack_out, p.Cout,
                                       p.Cin, p.BN, p.n_chunks, p.ksz, idx);
            fence_proxy_async_global();
            __threadfence();
        }
        float* ex = reinterpret_cast<float*>(extra);
        // Conv bias for every (padded) output channel, staged once per CTA so
        // the epilogue reads it from shared memory.
        const T* bias = static_cast<const T*>(p.bias);
        // (32 zero floats past the last tile, so vector reads never leave the region)
        for (int o = tid; o < p.n_ot * p.BN + 32; o += nthr)
            ex[p.bias_off + o] = (bias && o < p.Cout) ? load_f<T>(bias + o) : 0.f;
        if (p.rm == nullptr) return;
        // BN fold: z = max(0, x*scale + shift), scale = gamma/sqrt(rv+eps),
        // shift = beta - rm*scale.  Channels past Cin get 0.
        float* sc = ex;
        float* sh = sc + p.n_chunks * kBK;
        for (int c = tid; c < p.n_chunks * kBK; c += nthr) {
            float sv = 0.f, h = 0.f;
            if (c < p.Cin) {
                sv = p.gamma[c] / sqrtf(p.rv[c] + p.bn_eps);
                h = p.beta[c] - p.rm[c] * sv;
            }
            sc[c] = sv;
            sh[c] = h;
        }
        if constexpr (sizeof(T) == 2) {
            // the same fold as packed bf16 pairs for the producers' bf16x2 math
            uint32_t* sc2 = reinterpret_cast<uint32_t*>(extra) + p.bn2_off;
            uint32_t* sh2 = sc2 + p.n_chunks * (kBK / 2);
            for (int i = tid; i < p.n_chunks * (kBK / 2); i += nthr) {
                float sv[2] = {0.f, 0.f}, h[2] = {0.f, 0.f};
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int c = 2 * i + e;
                    if (c < p.Cin) {
                        sv[e] = p.gamma[c] / sqrtf(p.rv[c] + p.bn_eps);
                        h[e] = p.beta[c] - p.rm[c] * sv[e];
                    }
                }
                sc2[i] = pack_bf16x2(sv[0], sv[1]);
                sh2[i] = pack_bf16x2(h[0], h[1]);
            }
        }
    }

    // K stage -> (tap, 64-channel chunk): taps outermost.
    static __device__ __forceinline__ void stage_tap(const Params& p, int kiter, int& tap,
                                                     int& chunk) {
        tap = kiter / p.n_chunks;
        chunk = kiter - tap * p.n_chunks;
    }

    // Input position read by tap `tap` for output row t, and the channel base.
    static __device__ __forceinline__ void where(const Params& p, const Tile& tl, int kiter,
                                                 int row, int k0, int& s, int& c0) {
        int tap, chunk;
        stage_tap(p, kiter, tap, chunk);
        s = (tl.tt * kBM + row) * p.stride - p.pad + tap * p.dil;
        c0 = chunk * kBK + k0;
    }

    static __device__ __forceinline__ void load_a(const Params& p, const Tile& tl, int kiter,
                                                  int row, int k0, float (&v)[32]) {
        int s, c0;
        where(p, tl, kiter, row, k0, s, c0);
        if ((unsigned)s < (unsigned)p.Lin) {
            const T* xp = static_cast<const T*>(p.x) + ((size_t)tl.n * p.Cin + c0) * p.Lin + s;
            if (c0 + 32 <= p.Cin) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = load_f<T>(xp + (size_t)i * p.Lin);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[i] = (c0 + i < p.Cin) ? load_f<T>(xp + (size_t)i * p.Lin) : 0.f;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;   // zero padding of the conv input
        }
    }

    // Staged A (stride 1 only).  Tile rows t0 .. t0+128 read input rows from
    // s = t0 - pad + tap*dil on; the stage's box starts at s rounded down to the
    // 16-byte boundary and row r sits at offset r + s mod kAlign.  Rows outside
    // [0, L) and channels past Cin come back as the map's fill: NaN when BN
    // precedes the conv (max(NaN*scale + shift, 0) = 0, so the padding is
    // applied after BN+ReLU, as the block defines it), zero otherwise.
    static __device__ __forceinline__ int box_row0(const Params& p, const Tile& tl, int tap) {
        return tl.tt * kBM - p.pad + tap * p.dil;
    }

    static __device__ __forceinline__ void issue_a_box(const Params& p, const Tile& tl,
                                                       int kiter, uint32_t dst, uint32_t bar) {
        int tap, chunk;
        stage_tap(p, kiter, tap, chunk);
        const int s = box_row0(p, tl, tap);
        tma_load_3d(dst, &p.xmap, s & ~(kAlign - 1), chunk * kBK, tl.n, bar);
    }

    // bf16 storage with BN (staged): read_a returns the 16 packed bf16 pairs
    // (channels 2j, 2j+1 in v[j]'s bits) with BN+ReLU applied in bf16x2
    // arithmetic -- two values per instruction, nothing widened to fp32 -- so
    // the eight producer warps leave issue slots to the MMA warp.  The fold's
    // scale and shift are rounded to bf16 for it; z is rounded to bf16 for
    // the MMA in either case.
    static constexpr bool kPackedA = STAGED && sizeof(T) == 2 && EPI == ConvEpi::kResidual;

    static __device__ __forceinline__ void read_a(const Params& p, const uint8_t* extra,
                                                  const Tile& tl, int kiter, int row, int k0,
                                                  int lane, uint32_t box, float (&v)[32]) {
        int tap, chunk;
        stage_tap(p, kiter, tap, chunk);
        const int rem = box_row0(p, tl, tap) & (kAlign - 1);
        const uint32_t a = box + (uint32_t)((k0 * kBoxW + row + rem) * (int)sizeof(T));
        if constexpr (kPackedA) {
            const int c0 = chunk * kBK + k0;            // even
            const uint4* sc4 =
                reinterpret_cast<const uint4*>(reinterpret_cast<const uint32_t*>(extra) +
                                               p.bn2_off + c0 / 2);
            const uint4* sh4 = reinterpret_cast<const uint4*>(
                reinterpret_cast<const uint32_t*>(extra) + p.bn2_off + p.n_chunks * (kBK / 2) +
                c0 / 2);
            const __nv_bfloat162 zero2 = __floats2bfloat162_rn(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 s4 = sc4[q], h4 = sh4[q];
                const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w};
                const uint32_t hw[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = 4 * q + e;
                    const uint32_t lo = ld_shared_u16(a + (uint32_t)((2 * j) * kBoxW * 2));
                    const uint32_t hi = ld_shared_u16(a + (uint32_t)((2 * j + 1) * kBoxW * 2));
                    const uint32_t xw = lo | (hi << 16);
                    __nv_bfloat162 z = __hfma2(*reinterpret_cast<const __nv_bfloat162*>(&xw),
                                               *reinterpret_cast<const __nv_bfloat162*>(&sw[e]),
                                               *reinterpret_cast<const __nv_bfloat162*>(&hw[e]));
                    z = __hmax2(z, zero2);
                    v[j] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&z));
                }
            }
            return;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t ai = a + (uint32_t)(i * kBoxW * (int)sizeof(T));
            if constexpr (sizeof(T) == 4)
                v[i] = ld_shared_f32(ai);
            else
                v[i] = ld_shared_bf16(ai);
        }
        if (p.rm == nullptr) return;                   // zero fill is the padding
        const int c0 = chunk * kBK + k0;
        const float4* sc = reinterpret_cast<const float4*>(extra) + c0 / 4;
        const float4* sh = reinterpret_cast<const float4*>(extra) + (p.n_chunks * kBK + c0) / 4;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 a4 = sc[q], b4 = sh[q];
            v[4 * q] = fmaxf(fmaf(v[4 * q], a4.x, b4.x), 0.f);
            v[4 * q + 1] = fmaxf(fmaf(v[4 * q + 1], a4.y, b4.y), 0.f);
            v[4 * q + 2] = fmaxf(fmaf(v[4 * q + 2], a4.z, b4.z), 0.f);
            v[4 * q + 3] = fmaxf(fmaf(v[4 * q + 3], a4.w, b4.w), 0.f);
        }
    }

    static __device__ __forceinline__ void finish_a(const Params& p, const uint8_t* extra,
                                                    const Tile& tl, int kiter, int row, int k0,
                                                    float (&v)[32]) {
        if (p.rm == nullptr) return;                   // plain conv input
        int s, c0;
        where(p, tl, kiter, row, k0, s, c0);
        if ((unsigned)s >= (unsigned)p.Lin) return;    // padding applies to z, after BN+ReLU
        const float4* sc = reinterpret_cast<const float4*>(extra) + c0 / 4;
        const float4* sh = reinterpret_cast<const float4*>(extra) + (p.n_chunks * kBK + c0) / 4;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 a = sc[q], b = sh[q];
            v[4 * q] = fmaxf(fmaf(v[4 * q], a.x, b.x), 0.f);
            v[4 * q + 1] = fmaxf(fmaf(v[4 * q + 1], a.y, b.y), 0.f);
            v[4 * q + 2] = fmaxf(fmaf(v[4 * q + 2], a.z, b.z), 0.f);
            v[4 * q + 3] = fmaxf(fmaf(v[4 * q + 3], a.w, b.w), 0.f);
        }
    }

    static __device__ __forceinline__ const void* b_src(const Params& p, const Tile& tl,
                                                        int kiter) {
        constexpr int NP = sizeof(T) == 4 ? 2 : 1;
        return p.wpack + ((size_t)tl.ot * p.n_kiters + kiter) * NP * (size_t)p.BN * 128u;
    }

    template <class Acquire, class Release>
    static __device__ __forceinline__ bool epilogue(const Params& p, const uint8_t* extra,
                                                    const Tile& tl, int quarter, int lane,
                                                    uint32_t taddr, int BN, int halves,
                                                    Acquire& acquire, Release& release) {
        const int t = tl.tt * kBM + quarter * 32 + lane;
        const bool t_ok = t < p.L;
        T* out = static_cast<T*>(p.out);
        const int obase = tl.ot * BN;
        const size_t row0 = (size_t)tl.n * p.Cout;
        const float* bias_s = reinterpret_cast<const float*>(extra) + p.bias_off + obase;
        if constexpr (EPI == ConvEpi::kResidual) {
            // out = acc + bias + x.  The residual of the first four 16-channel
            // chunks is loaded before the accumulator is ready (this warp is
            // otherwise idle during the mainloop), later chunks four ahead of
            // the drain.  Path tests are uniform per chunk (t_ok per lane), so
            // a full chunk drains as straight-line code.
            const int ovalid = p.Cout - obase;     // channels of this tile that exist
            if constexpr (STAGED && sizeof(T) == 2) {
                // bf16 rows 16-byte aligned: a warp owns only 32 rows (half a
                // 128-byte line of one channel), so the four epilogue warps
                // move each 16-channel chunk through a shared buffer and touch
                // global memory in full lines: warp q loads/stores channel rows
                // 4q .. 4q+3 of the chunk, lane l rows 4l .. 4l+3 (8 bytes).
                // Named barrier 1 orders the four warps; whether the tile's
                // accumulator is ready is decided for all four at once (the
                // AND of their waits), so they always meet the same barriers.
                const int t0 = tl.tt * kBM;
                const bool rows_ok = t0 + 4 * lane < p.L;       // L % 8 == 0: all 4 or none
                const size_t grow = (row0 + obase + 4 * quarter) * p.L + (size_t)(t0 + 4 * lane);
                const uint2* xq = reinterpret_cast<const uint2*>(static_cast<const T*>(p.x) + grow);
                uint2* oq = reinterpret_cast<uint2*>(out + grow);
                const size_t rstride = (size_t)p.L / 4;          // one channel row, in uint2
                const uint32_t buf0 = smem_u32(extra + p.stage_off);
                const uint32_t mine = (uint32_t)(32 * quarter + lane) * 2u;   // this lane's row
                const uint32_t coop = (uint32_t)(4 * quarter * kBM + 4 * lane) * 2u;
                auto fetch = [&](int cc, uint2 (&w)[4]) {
                    if (cc >= BN) return;
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        w[r] = (rows_ok && cc + 4 * quarter + r < ovalid)
                                   ? __ldg(xq + (size_t)(cc + r) * rstride)
                                   : make_uint2(0u, 0u);
                };
                uint32_t bsel = 0;
                auto emit = [&](int cc, uint2 (&w)[4]) {
                    const uint32_t buf = buf0 + bsel * kChunkBufBytes;
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        st_shared_v2(buf + coop + (uint32_t)(r * kBM * 2), w[r].x, w[r].y);
                    fetch(cc + 64, w);          // refill this buffer four chunks ahead
                    named_bar_sync(1, 128);     // the chunk's residual is staged
                    float v[16];
                    tmem_ld16(taddr + (uint32_t)cc, v);
                    const float4* b4 = reinterpret_cast<const float4*>(bias_s + cc);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 bq = b4[q];
                        v[4 * q] += bq.x;
                        v[4 * q + 1] += bq.y;
                        v[4 * q + 2] += bq.z;
                        v[4 * q + 3] += bq.w;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint32_t a = buf + mine + (uint32_t)(i * kBM * 2);
                        const float y = v[i] + ld_shared_bf16(a);
                        st_shared_u16(a, __bfloat16_as_ushort(__float2bfloat16_rn(y)));
                    }
                    named_bar_sync(1, 128);     // the chunk's output is staged
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const uint2 o = ld_shared_v2(buf + coop + (uint32_t)(r * kBM * 2));
                        if (rows_ok && cc + 4 * quarter + r < ovalid)
                            oq[(size_t)(cc + r) * rstride] = o;
                    }
                    bsel ^= 1u;
                };
                uint2 w0[4], w1[4], w2[4], w3[4];
                fetch(0, w0);
                fetch(16, w1);
                fetch(32, w2);
                fetch(48, w3);
                if (!named_bar_and(1, 128, acquire(0))) return false;
                for (int cc = 0; cc < BN; cc += 64) {
                    if (halves == 2 && cc == BN / 2) {   // half A read: hand it back
                        release(0);
                        if (!named_bar_and(1, 128, acquire(1))) return false;
                    }
                    emit(cc, w0);
                    if (cc + 16 < BN) emit(cc + 16, w1);
                    if (cc + 32 < BN) emit(cc + 32, w2);
                    if (cc + 48 < BN) emit(cc + 48, w3);
                }
                release(halves - 1);
                return true;
            }
            const T* xr = static_cast<const T*>(p.x) + (row0 + obase) * p.L + t;
            T* outr = out + (row0 + obase) * p.L + t;
            auto fetch = [&](int cc, float (&r)[16]) {
                if (cc >= BN) return;
                const T* xp = xr + (size_t)cc * p.L;
                if (cc + 16 <= ovalid) {
                    if (t_ok) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) r[i] = load_f<T>(xp + (size_t)i * p.L);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        r[i] = (t_ok && cc + i < ovalid) ? load_f<T>(xp + (size_t)i * p.L) : 0.f;
                }
            };
            auto emit = [&](int cc, float (&r)[16]) {
                float v[16];
                tmem_ld16(taddr + (uint32_t)cc, v);
                const float4* b4 = reinterpret_cast<const float4*>(bias_s + cc);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 bq = b4[q];
                    v[4 * q] += bq.x + r[4 * q];
                    v[4 * q + 1] += bq.y + r[4 * q + 1];
                    v[4 * q + 2] += bq.z + r[4 * q + 2];
                    v[4 * q + 3] += bq.w + r[4 * q + 3];
                }
                T* op = outr + (size_t)cc * p.L;
                if (cc + 16 <= ovalid) {
                    if (t_ok) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) store_f<T>(op + (size_t)i * p.L, v[i]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (t_ok && cc + i < ovalid) store_f<T>(op + (size_t)i * p.L, v[i]);
                }
                fetch(cc + 64, r);              // refill this buffer four chunks ahead
            };
            float r0[16], r1[16], r2[16], r3[16];
            fetch(0, r0);
            fetch(16, r1);
            fetch(32, r2);
            fetch(48, r3);
            if (!acquire(0)) return false;
            for (int cc = 0; cc < BN; cc += 64) {
                if (halves == 2 && cc == BN / 2) {   // half A read: hand it back
                    release(0);
                    if (!acquire(1)) return false;
                }
                emit(cc, r0);
                if (cc + 16 < BN) emit(cc + 16, r1);
                if (cc + 32 < BN) emit(cc + 32, r2);
                if (cc + 48 < BN) emit(cc + 48, r3);
            }
            release(halves - 1);
        } else {
            // y -> out, and per-(n, group, t tile, row) statistics of y.  A
            // group's channels are contiguous.  Each run of a group inside a
            // 16-channel chunk is reduced two-pass in registers (count, mean,
            // M2), folded into the group's running triple with Chan's update,
            // and merged across the warp when the group ends.  Every test below
            // is uniform across the warp except t_ok (invalid rows count 0).
            if constexpr (ONE_WAVE) {
                // one tile per CTA: its channels' gamma and beta, staged by the
                // epilogue warps while the mainloop runs (step 3 of gn_fused
                // turns them into scale and shift, behind its first barrier)
                float* s_a =
                    reinterpret_cast<float*>(const_cast<uint8_t*>(extra) + p.stage_off +
                                             kGnMaxGroups * 4 * 16);
                for (int c = quarter * 32 + lane; c < 256; c += 128) {
                    const int o = obase + c;
                    s_a[c] = (p.gn_gamma && o < p.Cout) ? p.gn_gamma[o] : 1.f;
                    s_a[256 + c] = (p.gn_beta && o < p.Cout) ? p.gn_beta[o] : 0.f;
                }
            }
            bool acquired = true;
            for (int h = 0; h < halves && acquired; ++h) acquired = acquire(h);
            if constexpr (ONE_WAVE) {
                // gn_fused meets at named barrier 1: the four warps decide
                // together (a warp whose wait gave up would never arrive)
                if (!named_bar_and(1, 128, acquired)) return false;
                const bool ok = gn_fused(p, extra, tl, quarter, lane, taddr, BN);
                for (int h = 0; h < halves; ++h) release(h);
                return ok;
            }
            if (!acquired) return false;
            const int ovalid = p.Cout - obase;
            float cnt = 0.f, mean = 0.f, m2 = 0.f;
            const float tw = t_ok ? 1.f : 0.f;
            // first channel of the group after the current one (tiles hold whole
            // groups, so this starts at obase + cpg and steps by cpg)
            int gend = obase + p.cpg;
            // sum of the 16 values selected by [lo, hi), as a 4-level tree
            auto tree16 = [](const float (&a)[16]) {
                float b[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) b[i] = a[2 * i] + a[2 * i + 1];
#pragma unroll
                for (int i = 0; i < 4; ++i) b[i] = b[2 * i] + b[2 * i + 1];
                return (b[0] + b[1]) + (b[2] + b[3]);
            };
            for (int cc = 0; cc < BN && cc < ovalid; cc += 16) {
                float v[16];
                tmem_ld16(taddr + (uint32_t)cc, v);
                const float4* b4 = reinterpret_cast<const float4*>(bias_s + cc);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 bq = b4[q];
                    v[4 * q] += bq.x;
                    v[4 * q + 1] += bq.y;
                    v[4 * q + 2] += bq.z;
                    v[4 * q + 3] += bq.w;
                }
                T* op = out + (row0 + obase + cc) * p.L + t;
                const int n = min(16, ovalid - cc);
                if (n == 16) {
                    if (t_ok) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) store_f<T>(op + (size_t)i * p.L, v[i]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (t_ok && i < n) store_f<T>(op + (size_t)i * p.L, v[i]);
                }
                if (p.cpg <= 16 && 16 % p.cpg == 0) {
                    // whole groups inside the chunk: group (obase + cc)/cpg + j
                    const size_t gstride = (size_t)p.n_tt * kBM;
                    float2* part = p.partials +
                                   ((size_t)(tl.n * p.G + (obase + cc) / p.cpg) * p.n_tt + tl.tt) *
                                       kBM +
                                   quarter * 32 + lane;
                    switch (p.cpg) {
                        case 1: gn_chunk_stats<1>(v, n, tw, part, gstride); break;
                        case 2: gn_chunk_stats<2>(v, n, tw, part, gstride); break;
                        case 4: gn_chunk_stats<4>(v, n, tw, part, gstride); break;
                        case 8: gn_chunk_stats<8>(v, n, tw, part, gstride); break;
                        default: gn_chunk_stats<16>(v, n, tw, part, gstride); break;
                    }
                    continue;
                }
                // runs [i0, i1) of one group inside this chunk
                int i0 = 0;
                while (i0 < n) {
                    const int i1 = min(n, gend - (obase + cc));
                    float sel[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) sel[i] = (i >= i0 && i < i1) ? v[i] : 0.f;
                    const float k = (float)(i1 - i0);
                    const float sm = __fdividef(tree16(sel), k);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float d = (i >= i0 && i < i1) ? v[i] - sm : 0.f;
                        sel[i] = d * d;
                    }
                    const float sq = tree16(sel);
                    const float kb = k * tw;                           // this run's count
                    const float nab = cnt + kb;
                    if (nab > 0.f) {
                        const float delta = sm - mean;
                        const float fb = __fdividef(kb, nab);
                        mean += delta * fb;
                        m2 += sq * tw + delta * delta * cnt * fb;
                        cnt = nab;
                    }
                    if (obase + cc + i1 == gend) {                     // group complete
                        // this row's (mean, M2) over the group's channels; the
                        // rows of the tile are merged by the finalize kernel
                        const int g = gend / p.cpg - 1;
                        gend += p.cpg;
                        p.partials[((size_t)(tl.n * p.G + g) * p.n_tt + tl.tt) * kBM +
                                   quarter * 32 + lane] = make_float2(mean, m2);
                        cnt = 0.f;
                        mean = 0.f;
                        m2 = 0.f;
                    }
                    i0 = i1;
                }
            }
            for (int h = 0; h < halves; ++h) release(h);
        }
        return true;
    }

    // Conv + GroupNorm when every tile has its own CTA and all are resident
    // (cooperative launch): y = acc + bias never leaves TMEM.
    //  1. Each group's (count, mean, M2) over the tile: per row two-pass over
    //     the group's run of channels, merged over the warp's 32 rows with
    //     shuffles, then over the four epilogue warps in shared memory (fixed
    //     order), written once per (n, group, t tile).
    //  2. Grid-wide barrier: one arrival per CTA on a counter zeroed before
    //     the launch; one thread waits for all (bounded).
    //  3. Each group's statistics merged over the sample's n_tt tiles, in t
    //     order, so every CTA of the sample computes the same values; scale
    //     a = gamma*rsqrt(var + eps) and shift beta - mean*a per channel.
    //  4. out = y*a + shift, read again from TMEM.
    // The four epilogue warps meet at named barrier 1.  Tiles hold whole groups.
    static __device__ bool gn_fused(const Params& p, const uint8_t* extra, const Tile& tl,
                                    int quarter, int lane, uint32_t taddr, int BN) {
        const int t = tl.tt * kBM + quarter * 32 + lane;
        const bool t_ok = t < p.L;
        const float tw = t_ok ? 1.f : 0.f;
        const int obase = tl.ot * BN;
        const int ovalid = min(BN, p.Cout - obase);
        const int ng = ovalid / p.cpg;                 // groups of this tile
        const int g0 = obase / p.cpg;
        const int etid = quarter * 32 + lane;          // 0..127 over the four warps
        const float* bias_s = reinterpret_cast<const float*>(extra) + p.bias_off + obase;
        uint8_t* ex = const_cast<uint8_t*>(extra) + p.stage_off;
        float4* s_part = reinterpret_cast<float4*>(ex);                 // [group][warp]
        float* s_a = reinterpret_cast<float*>(ex + kGnMaxGroups * 4 * 16);
        float* s_sh = s_a + 256;

        // 1. group statistics of the tile.  Every valid row of a group has the
        //    same count (cpg), so the warp's merge of its rows is two warp sums:
        //    of the row means, then of M2_r + cpg*(mean_r - mean)^2.
        const bool has_bias = p.bias != nullptr;
        const int nvr = __popc(__ballot_sync(0xffffffffu, t_ok));   // valid rows of the warp
        const float inv_nvr = nvr > 0 ? 1.f / (float)nvr : 0.f;
        const float wcount = (float)(p.cpg * nvr);
        switch (p.cpg) {
            case 1: gn_tile_stats<1>(bias_s, taddr, ovalid, ng, tw, inv_nvr, wcount, quarter, lane, s_part, has_bias); break;
            case 2: gn_tile_stats<2>(bias_s, taddr, ovalid, ng, tw, inv_nvr, wcount, quarter, lane, s_part, has_bias); break;
            case 4: gn_tile_stats<4>(bias_s, taddr, ovalid, ng, tw, inv_nvr, wcount, quarter, lane, s_part, has_bias); break;
            case 8: gn_tile_stats<8>(bias_s, taddr, ovalid, ng, tw, inv_nvr, wcount, quarter, lane, s_part, has_bias); break;
            case 16: gn_tile_stats<16>(bias_s, taddr, ovalid, ng, tw, inv_nvr, wcount, quarter, lane, s_part, has_bias); break;
            default: {
                // groups crossing 16-channel chunks: each row's (count, mean, M2)
                // over the group's runs, then the warp sums at its last run
                float cnt = 0.f, mean = 0.f, m2 = 0.f;
                int gend = obase + p.cpg;              // first channel after the group
                for (int cc = 0; cc < ovalid; cc += 16) {
                    float v[16];
                    tmem_ld16(taddr + (uint32_t)cc, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] += bias_s[cc + i];
                    const int n = min(16, ovalid - cc);
                    int i0 = 0;
                    while (i0 < n) {                    // runs [i0, i1) of one group
                        const int i1 = min(n, gend - (obase + cc));
                        float s1 = 0.f;
#pragma unroll
                        for (int i = 0; i < 16; ++i) s1 += (i >= i0 && i < i1) ? v[i] : 0.f;
                        const float k = (float)(i1 - i0);
                        const float rm = s1 / k;
                        float sq = 0.f;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float d = (i >= i0 && i < i1) ? v[i] - rm : 0.f;
                            sq = fmaf(d, d, sq);
                        }
                        chan_merge(cnt, mean, m2, k, rm, sq);
                        if (obase + cc + i1 == gend) {  // group complete (uniform)
                            const float wm = warp_sum(mean * tw) * inv_nvr;
                            const float d = mean - wm;
                            const float wq = warp_sum(tw * (m2 + (float)p.cpg * d * d));
                            if (lane == 0)
                                s_part[(gend / p.cpg - 1 - g0) * 4 + quarter] =
                                    make_float4(wcount, wm, wq, 0.f);
                            gend += p.cpg;
                            cnt = 0.f;
                            mean = 0.f;
                            m2 = 0.f;
                        }
                        i0 = i1;
                    }
                }
            }
        }
        named_bar_sync(1, 128);
        for (int gl = etid; gl < ng; gl += 128) {
            float c = 0.f, m = 0.f, q = 0.f;
            for (int w = 0; w < 4; ++w) {
                const float4 sp = s_part[gl * 4 + w];
                chan_merge(c, m, q, sp.x, sp.y, sp.z);
            }
            p.tile_stats[((size_t)tl.n * p.G + g0 + gl) * p.n_tt + tl.tt] = make_float4(c, m, q, 0.f);
        }
        // (s_a and s_sh hold the channels' gamma and beta, staged by setup)
        __threadfence();
        named_bar_sync(1, 128);

        // 2. grid-wide barrier
        bool ok = true;
        if (etid == 0) {
            __threadfence();
            atomicAdd(p.grid_counter, 1u);
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(p.grid_counter) < gridDim.x) {
                if (globaltimer_ns() - t0 > p.timeout_ns) {
                    record_status(p.status, kStatusTimeout, kSiteGridBarrier);
                    ok = false;
                    break;
                }
                __nanosleep(128);
            }
        }
        if (!named_bar_and(1, 128, ok)) return false;

        // 3. the sample's statistics of each group of the tile
        for (int gl = etid; gl < ng; gl += 128) {
            const int g = g0 + gl;
            float c = 0.f, m = 0.f, q = 0.f;
            const float4* ts = p.tile_stats + ((size_t)tl.n * p.G + g) * p.n_tt;
            for (int t0 = 0; t0 < p.n_tt; t0 += 8) {      // eight loads in flight
                float4 sp[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    sp[k] = t0 + k < p.n_tt ? __ldcg(ts + t0 + k) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k = 0; k < 8; ++k) chan_merge(c, m, q, sp[k].x, sp[k].y, sp[k].z);
            }
            const float var = fmaxf(q / c, 0.f);      // biased variance
            const float inv = 1.0f / sqrtf(var + p.gn_eps);
            for (int i = 0; i < p.cpg; ++i) {
                const int cl = gl * p.cpg + i;             // channel within the tile
                const float a = inv * s_a[cl];
                s_a[cl] = a;
                // out = (y - mean)*a + beta with y = acc + bias: the conv bias
                // folds into the shift, so step 4 reads the accumulator alone
                s_sh[cl] = s_sh[cl] - (m - bias_s[cl]) * a;
            }
        }
        named_bar_sync(1, 128);

        // 4. normalize from TMEM, 64 columns per round trip
        T* out = static_cast<T*>(p.out);
        T* op0 = out + ((size_t)tl.n * p.Cout + obase) * p.L + t;
        for (int cb = 0; cb < ovalid; cb += 64) {          // 64 divides 256
            float v[64];
            tmem_ld64(taddr + (uint32_t)cb, v);
            T* op = op0 + (size_t)cb * p.L;
            if (cb + 64 <= ovalid) {
                if (t_ok) {
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        store_f<T>(op + (size_t)i * p.L, fmaf(v[i], s_a[cb + i], s_sh[cb + i]));
                }
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (t_ok && cb + i < ovalid)
                        store_f<T>(op + (size_t)i * p.L, fmaf(v[i], s_a[cb + i], s_sh[cb + i]));
            }
        }
        return true;
    }
};

// ---------------------------------------------------------------------------
// Weight repack: W (Cout, Cin, ksz) -> for each (o tile, tap, 64-channel chunk)
// the B-stage image: NP parts of BN rows x 64 bf16, 128B-swizzled.  fp32
// weights are split into hi + lo bf16 parts; bf16 weights are copied.  Rows
// past Cout and channels past Cin are zero.  One thread per 16-byte chunk.
// ---------------------------------------------------------------------------
template <typename T, int NP>
__global__ void pack_conv_weight_kernel(const T* __restrict__ w, uint8_t* __restrict__ pack,
                                        int Cout, int Cin, int BN, int n_ot, int n_chunks,
                                        int ksz) {
    griddep_launch_dependents();       // the GEMM may launch; it waits before reading B
    const size_t total = (size_t)n_ot * ksz * n_chunks * BN * 8;   // 16-byte chunks per part
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x)
        pack_conv_chunk<T, NP>(w, pack, Cout, Cin, BN, n_chunks, ksz, idx);
}

// ---------------------------------------------------------------------------
// GroupNorm finalize + normalize, one CTA per (n, group): merge the group's
// per-row partial (mean, M2) over its n_tt * 128 rows (count cpg per row inside
// [0, T), 0 past it) in a fixed order -- each thread a strided subset, then the
// warps, then the CTA -- and apply
// out = (y - mean) * rsqrt(var + eps) * gamma + beta in place over the group's
// contiguous (cpg x T) block.
// ---------------------------------------------------------------------------
__global__ void groupnorm_finalize_normalize_kernel(float* __restrict__ out,
                                                    const float2* __restrict__ partials,
                                                    int n_tt, int Cout, int T, int G,
                                                    const float* __restrict__ gamma,
                                                    const float* __restrict__ beta, float eps) {
    const int ng = blockIdx.x;
    const int g = ng % G;
    const int cpg = Cout / G;
    const int n_part = n_tt * kBM;
    __shared__ float s_mean, s_inv;
    __shared__ float s_w[3][32];
    {
    float cnt = 0.f, mean = 0.f, m2 = 0.f;
    for (int i = threadIdx.x; i < n_part; i += blockDim.x) {
        const float2 q = partials[(size_t)ng * n_part + i];
        const float nb = (i < T) ? (float)cpg : 0.f;        // row i of the sample
        const float nab = cnt + nb;
        if (nab > 0.f) {
            const float delta = q.x - mean;
            const float fb = nb / nab;
            mean += delta * fb;
            m2 += q.y + delta * delta * cnt * fb;
            cnt = nab;
        }
    }
    warp_merge_stats(cnt, mean, m2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        s_w[0][warp] = cnt;
        s_w[1][warp] = mean;
        s_w[2][warp] = m2;
    }
    __syncthreads();
    if (warp == 0) {
        const int nw = (int)(blockDim.x >> 5);
        cnt = lane < nw ? s_w[0][lane] : 0.f;
        mean = lane < nw ? s_w[1][lane] : 0.f;
        m2 = lane < nw ? s_w[2][lane] : 0.f;
        warp_merge_stats(cnt, mean, m2);
        if (lane == 0) {
            const float var = fmaxf(m2 / cnt, 0.f);   // biased variance
            s_mean = mean;
            s_inv = 1.0f / sqrtf(var + eps);
        }
    }
    }
    __syncthreads();
    const float mean = s_mean, inv = s_inv;
    float* base = out + (size_t)ng * cpg * T;      // channels g*cpg.. of sample n
    // channel by channel: scale and shift are uniform along a channel's T values
    for (int c = 0; c < cpg; ++c) {
        const int o = g * cpg + c;
        const float a = inv * (gamma ? gamma[o] : 1.f);
        const float sh = (beta ? beta[o] : 0.f) - mean * a;
        float* row = base + (size_t)c * T;
        if ((T & 3) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
            float4* r4 = reinterpret_cast<float4*>(row);
            for (int i = threadIdx.x; i < T / 4; i += blockDim.x) {
                float4 y = r4[i];
                y.x = fmaf(y.x, a, sh);
                y.y = fmaf(y.y, a, sh);
                y.z = fmaf(y.z, a, sh);
                y.w = fmaf(y.w, a, sh);
                r4[i] = y;
            }
        } else {
            for (int i = threadIdx.x; i < T; i += blockDim.x) row[i] = fmaf(row[i], a, sh);
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct ConvPlan {
    GemmPlan g;
    int n_ot, n_chunks, n_tt;
    int stage_off;          // byte offset of the epilogue's chunk buffers in the extra smem
    size_t wpack_bytes;
};

// Extra shared memory: BN fold (scale, shift) when present, the staged bias,
// then (128-byte aligned) stage_bytes for the epilogue's chunk buffers.
static ConvPlan plan_conv(int N, int Cin, int Cout, int L, int NP, bool with_bn,
                          uint32_t x_box_bytes = 0, uint32_t stage_bytes = 0, int ksz = 3) {
    ConvPlan pl{};
    const int BN = Cout <= 256 ? ((Cout + 15) / 16) * 16 : 256;
    pl.n_ot = ceil_div(Cout, BN);
    pl.n_chunks = ceil_div(Cin, kBK);
    pl.n_tt = ceil_div(L, kBM);
    const long long tiles = (long long)N * pl.n_tt * pl.n_ot;
    const uint32_t fold_bias = (with_bn ? (uint32_t)(2 * pl.n_chunks * kBK * 4) : 0u) +
                               (uint32_t)((pl.n_ot * BN + 32) * 4) +
                               (with_bn && NP == 1 ? (uint32_t)(pl.n_chunks * kBK * 4) : 0u);
    pl.stage_off = (int)((fold_bias + 127u) & ~127u);
    const uint32_t extra = stage_bytes ? (uint32_t)pl.stage_off + stage_bytes : fold_bias;
    pl.g = make_gemm_plan(BN, (int)std::min<long long>(tiles, 1LL << 30), ksz * pl.n_chunks, NP,
                          extra, x_box_bytes);
    pl.wpack_bytes = (size_t)pl.n_ot * pl.g.num_kiters * NP * BN * 128;
    return pl;
}

// Tensor map of x for the staged A path: (L, Cin, N) with boxes of
// (128 + 16/esize) rows x 64 channels x 1 sample.  Needs 16-byte aligned rows;
// false (use the register path) when they are not or the driver refuses.
template <typename T>
static bool make_x_map(ConvParams& p, const void* x, int N, int Cin, int L, bool nan_fill) {
    constexpr size_t es = sizeof(T);
    if (!aligned(x, 16) || ((size_t)L * es) % 16 != 0) return false;
    const uint64_t dims[3] = {(uint64_t)L, (uint64_t)Cin, (uint64_t)N};
    const uint64_t strides[2] = {(uint64_t)L * es, (uint64_t)Cin * L * es};
    const uint32_t box[3] = {(uint32_t)(kBM + 16 / es), (uint32_t)kBK, 1u};
    return encode_tensor_map_3d(
        &p.xmap, es == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x,
        dims, strides, box, nan_fill);
}

// Plans the conv GEMM (L output rows, Lin input rows, ksz taps), staged when x
// allows it (stride 1, aligned rows) and the slots fit; fills the map and
// returns whether the staged kernel runs.  p.x and p.out must be set: the
// staged bf16 residual epilogue moves x and out in 8-byte words, so it also
// needs out 8-byte aligned (x is 16-byte aligned for the map).
template <typename T>
static bool plan_conv_staged(ConvParams& p, ConvPlan& pl, int N, int Cin, int Cout, int L,
                             bool with_bn, int Lin, int stride = 1, int ksz = 3) {
    constexpr int NP = sizeof(T) == 4 ? 2 : 1;
    constexpr uint32_t box_bytes = (uint32_t)((kBM + 16 / sizeof(T)) * kBK * sizeof(T));
    // the staged bf16 residual epilogue needs its two chunk buffers, the fused
    // GroupNorm epilogue its partials and per-channel scale and shift
    const uint32_t fused_bytes = p.fused ? kGnFusedBytes : 0u;
    const uint32_t stage_bytes =
        (with_bn && sizeof(T) == 2) ? 2u * ConvProblem<T, ConvEpi::kResidual, true>::kChunkBufBytes
                                    : fused_bytes;
    const bool out_ok = !(with_bn && sizeof(T) == 2) || aligned(p.out, 8);
    if (out_ok && stride == 1 && make_x_map<T>(p, p.x, N, Cin, Lin, with_bn)) {
        pl = plan_conv(N, Cin, Cout, L, NP, with_bn, box_bytes, stage_bytes, ksz);
        if (pl.g.b_stages >= 2 && pl.g.x_depth >= 2) {
            p.stage_off = pl.stage_off;
            return true;
        }
    }
    pl = plan_conv(N, Cin, Cout, L, NP, with_bn, 0, fused_bytes, ksz);
    p.stage_off = pl.stage_off;
    return false;
}

}  // namespace nrc

using namespace nrc;

// The block's workspace: the packed weight image, then (256-byte aligned) the
// counter of the in-kernel repack.
static size_t block_counter_offset(int C, nrc_dtype dt) {
    return (plan_conv(1, C, C, 1, dt == NRC_F32 ? 2 : 1, true).wpack_bytes + 255) &
           ~(size_t)255;
}

extern "C" size_t nrc_prenorm_dilconv_residual_workspace_size(int C, nrc_dtype dt) {
    if (C <= 0 || (dt != NRC_F32 && dt != NRC_BF16)) return 0;
    return block_counter_offset(C, dt) + 256;
}

namespace {

// The block's weight image (packed once per call into wpack; depends on C only).
nrc_status block_pack(const void* conv_weight, nrc_dtype dt, int C, void* wpack,
                      cudaStream_t st) {
    const int NP = dt == NRC_F32 ? 2 : 1;
    const ConvPlan pl = plan_conv(1, C, C, 1, NP, true);
    const size_t units = pl.wpack_bytes / 16 / NP;
    TraceScope ts("pack_conv_weight", st);
    if (dt == NRC_F32)
        pack_conv_weight_kernel<float, 2><<<elementwise_grid(units), 256, 0, st>>>(
            static_cast<const float*>(conv_weight), static_cast<uint8_t*>(wpack), C, C, pl.g.BN,
            pl.n_ot, pl.n_chunks, 3);
    else
        pack_conv_weight_kernel<__nv_bfloat16, 1><<<elementwise_grid(units), 256, 0, st>>>(
            static_cast<const __nv_bfloat16*>(conv_weight), static_cast<uint8_t*>(wpack), C, C,
            pl.g.BN, pl.n_ot, pl.n_chunks, 3);
    return cuda_status(cudaGetLastError());
}

// Plans and launches the block's GEMM on device buffers; wpack holds the
// packed weight image.  Arguments already validated.
nrc_status block_gemm(const void* x, void* out, nrc_dtype dt, int N, int C, int L, int dilation,
                      int padding, const float* rm, const float* rv, const float* gamma,
                      const float* beta, float bn_eps, const void* conv_bias, uint8_t* wpack,
                      const void* w_raw, uint32_t* pack_counter, cudaStream_t st) {
    const int NP = dt == NRC_F32 ? 2 : 1;
    ConvPlan pl = plan_conv(N, C, C, L, NP, true);
    if ((long long)N * pl.n_tt * pl.n_ot >= (1LL << 30)) return NRC_ERR_UNSUPPORTED;
    ConvParams p{};
    p.x = x;
    p.out = out;
    const bool staged = dt == NRC_F32 ? plan_conv_staged<float>(p, pl, N, C, C, L, true, L)
                                      : plan_conv_staged<__nv_bfloat16>(p, pl, N, C, C, L, true, L);
    p.N = N;
    p.Cin = C;
    p.Cout = C;
    p.L = L;
    p.Lin = L;
    p.pad = padding;
    p.dil = dilation;
    p.stride = 1;
    p.ksz = 3;
    p.n_tt = pl.n_tt;
    p.n_ot = pl.n_ot;
    p.n_chunks = pl.n_chunks;
    p.n_kiters = pl.g.num_kiters;
    p.BN = pl.g.BN;
    p.rm = rm;
    p.rv = rv;
    p.gamma = gamma;
    p.beta = beta;
    p.bn_eps = bn_eps;
    p.bias = conv_bias;
    p.bias_off = 2 * pl.n_chunks * kBK;
    p.bn2_off = p.bias_off + pl.n_ot * pl.g.BN + 32;     // after the staged bias
    p.wpack = wpack;
    // w_raw given: repack it.  One wave (pack_counter given) with the staged
    // kernel: inside the GEMM kernel (cooperative launch); otherwise by the
    // repack kernel, with the GEMM launched behind it (it waits only to read B).
    // w_raw NULL: wpack already holds the image.
    const bool one_wave = w_raw != nullptr && pack_counter != nullptr && staged;
    if (one_wave) {
        ConvParams p1 = p;
        GemmPlan g1 = pl.g;
        p1.w_raw = w_raw;
        p1.wpack_out = wpack;
        p1.pack_counter = pack_counter;
        if (cudaMemsetAsync(pack_counter, 0, sizeof(uint32_t), st) != cudaSuccess)
            return NRC_ERR_CUDA;
        g1.coop = true;
        if (g1.BN % 128 == 0)
            g1.split_h = std::min(std::min(256 / (32 * NP), g1.b_stages), g1.num_kiters / 2);
        const nrc_status s =
            dt == NRC_F32
                ? launch_gemm<ConvProblem<float, ConvEpi::kResidual, true, true>, 2>(
                      "prenorm_block_gemm", p1, g1, st)
                : launch_gemm<ConvProblem<__nv_bfloat16, ConvEpi::kResidual, true, true>, 1>(
                      "prenorm_block_gemm", p1, g1, st);
        // refused (the CTAs cannot all be resident now): the two-launch path
        if (s != NRC_ERR_UNSUPPORTED) return s;
    }
    if (w_raw) {
        const nrc_status s = block_pack(w_raw, dt, C, wpack, st);
        if (s != NRC_OK) return s;
        pl.g.b_after_prev = true;
    }
    // Residual drain overlapped at tile boundaries (whole 128-column halves).
    if (pl.g.BN % 128 == 0) {
        const int SA = 256 / (32 * NP);
        pl.g.split_h = std::min(std::min(SA, pl.g.b_stages), pl.g.num_kiters / 2);
    }
    if (dt == NRC_F32) {
        if (staged)
            return launch_gemm<ConvProblem<float, ConvEpi::kResidual, true>, 2>(
                "prenorm_block_gemm", p, pl.g, st);
        return launch_gemm<ConvProblem<float, ConvEpi::kResidual, false>, 2>(
            "prenorm_block_gemm", p, pl.g, st);
    }
    if (staged)
        return launch_gemm<ConvProblem<__nv_bfloat16, ConvEpi::kResidual, true>, 1>(
            "prenorm_block_gemm", p, pl.g, st);
    return launch_gemm<ConvProblem<__nv_bfloat16, ConvEpi::kResidual, false>, 1>(
        "prenorm_block_gemm", p, pl.g, st);
}

// Shared argument checks of the block entry points (device or host buffers),
// except the workspace pointer (the allocation-free entry point has none).
nrc_status block_check_args(const void* x, const void* out, nrc_dtype dt, int N, int C, int L,
                            int kernel_size, int dilation, int padding, const void* rm,
                            const void* rv, const void* gamma, const void* beta, float bn_eps,
                            const void* conv_weight) {
    if (dt != NRC_F32 && dt != NRC_BF16) return NRC_ERR_INVALID_ARG;
    if (!x || !out || !rm || !rv || !gamma || !beta || !conv_weight) return NRC_ERR_INVALID_ARG;
    if (N <= 0 || C <= 0 || L <= 0 || dilation <= 0 || padding < 0) return NRC_ERR_INVALID_ARG;
    if (!(bn_eps >= 0.f) || !std::isfinite(bn_eps)) return NRC_ERR_INVALID_ARG;
    if (kernel_size != 3 || padding != dilation) return NRC_ERR_UNSUPPORTED;
    if (C > 2048) return NRC_ERR_UNSUPPORTED;
    const size_t bytes = (size_t)N * C * L * (dt == NRC_F32 ? 4 : 2);
    if (ranges_overlap(x, bytes, out, bytes)) return NRC_ERR_INVALID_ARG;
    return NRC_OK;
}

nrc_status block_check(const void* x, const void* out, nrc_dtype dt, int N, int C, int L,
                       int kernel_size, int dilation, int padding, const void* rm,
                       const void* rv, const void* gamma, const void* beta, float bn_eps,
                       const void* conv_weight, const void* workspace) {
    const nrc_status s = block_check_args(x, out, dt, N, C, L, kernel_size, dilation, padding,
                                          rm, rv, gamma, beta, bn_eps, conv_weight);
    if (s != NRC_OK) return s;
    if (!workspace) return NRC_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return NRC_ERR_ALIGNMENT;
    return NRC_OK;
}

}  // namespace

extern "C" nrc_status nrc_prenorm_dilconv_residual(
    const void* x, void* out, nrc_dtype dt, int N, int C, int L, int kernel_size, int dilation,
    int padding, const float* rm, const float* rv, const float* gamma, const float* beta,
    float bn_eps, const void* conv_weight, const void* conv_bias, void* workspace,
    size_t workspace_bytes, void* stream) {
    const nrc_status c = block_check(x, out, dt, N, C, L, kernel_size, dilation, padding, rm, rv,
                                     gamma, beta, bn_eps, conv_weight, workspace);
    if (c != NRC_OK) return c;
    if (workspace_bytes < nrc_prenorm_dilconv_residual_workspace_size(C, dt))
        return NRC_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    // Problems of one wave (every tile on its own CTA): one launch, the GEMM
    // kernel repacks the weights itself (this saves a launch and its gap, a
    // large share of a short call).  A longer GEMM gains nothing from it: its
    // first weight stages would wait for the whole grid's repack.
    const int n_tiles = plan_conv(N, C, C, L, dt == NRC_F32 ? 2 : 1, true).g.num_tiles;
    if (n_tiles <= device_sm_count() && device_coop_launch()) {
        // (block_gemm packs separately if the staged kernel does not apply)
        uint32_t* counter = reinterpret_cast<uint32_t*>(ws + block_counter_offset(C, dt));
        return block_gemm(x, out, dt, N, C, L, dilation, padding, rm, rv, gamma, beta, bn_eps,
                          conv_bias, ws, conv_weight, counter, st);
    }
    // the repack, then the GEMM launched behind it (it waits only to read B)
    return block_gemm(x, out, dt, N, C, L, dilation, padding, rm, rv, gamma, beta, bn_eps,
                      conv_bias, ws, conv_weight, nullptr, st);
}

// ---------------------------------------------------------------------------
// Host-buffer entry point: x and out in host memory (pinned for overlap), the
// small parameters and weights in host memory too.  The batch goes through in
// chunks of chunk_n samples and two device buffers: the copy-in of chunk j+1,
// the GEMM of chunk j and the copy-out of chunk j-1 run at once on two
// library streams and the caller's stream, ordered by events.
// ---------------------------------------------------------------------------
namespace {

struct HostLayout {
    size_t par, w, b, x[2], o[2], total;
};

HostLayout host_layout(int N, int C, int L, nrc_dtype dt, int chunk_n) {
    const size_t es = dt == NRC_F32 ? 4 : 2;
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    const size_t chunk = (size_t)chunk_n * C * L * es;
    HostLayout h{};
    h.par = up(nrc_prenorm_dilconv_residual_workspace_size(C, dt));
    h.w = up(h.par + (size_t)4 * C * sizeof(float));
    h.b = up(h.w + (size_t)C * C * 3 * es);
    h.x[0] = up(h.b + (size_t)C * es);
    h.x[1] = up(h.x[0] + chunk);
    h.o[0] = up(h.x[1] + chunk);
    h.o[1] = up(h.o[0] + chunk);
    h.total = h.o[1] + chunk;
    (void)N;
    return h;
}

// Per device: the copy-in and copy-out streams and the events of the pipeline.
struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start, join, ev_in[2], ev_gemm[2], ev_out[2];
    bool ready = false;
};
std::mutex g_host_mu;
HostPipe g_host_pipe[64];

nrc_status host_pipe(HostPipe** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NRC_ERR_CUDA;
    HostPipe& hp = g_host_pipe[dev];
    if (!hp.ready) {
        const unsigned f = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.start, f) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.join, f) != cudaSuccess)
            return NRC_ERR_CUDA;
        for (int b = 0; b < 2; ++b)
            if (cudaEventCreateWithFlags(&hp.ev_in[b], f) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.ev_gemm[b], f) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.ev_out[b], f) != cudaSuccess)
                return NRC_ERR_CUDA;
        hp.ready = true;
    }
    *out = &hp;
    return NRC_OK;
}

}  // namespace

extern "C" size_t nrc_prenorm_dilconv_residual_host_workspace_size(int N, int C, int L,
                                                                   nrc_dtype dt, int chunk_n) {
    if (N <= 0 || C <= 0 || L <= 0 || chunk_n <= 0 || (dt != NRC_F32 && dt != NRC_BF16))
        return 0;
    return host_layout(N, C, L, dt, std::min(chunk_n, N)).total;
}

extern "C" nrc_status nrc_prenorm_dilconv_residual_host(
    const void* x_host, void* out_host, nrc_dtype dt, int N, int C, int L, int kernel_size,
    int dilation, int padding, const float* rm_host, const float* rv_host,
    const float* gamma_host, const float* beta_host, float bn_eps, const void* weight_host,
    const void* bias_host, int chunk_n, void* workspace, size_t workspace_bytes, void* stream) {
    const nrc_status c = block_check(x_host, out_host, dt, N, C, L, kernel_size, dilation,
                                     padding, rm_host, rv_host, gamma_host, beta_host, bn_eps,
                                     weight_host, workspace);
    if (c != NRC_OK) return c;
    if (chunk_n <= 0) return NRC_ERR_INVALID_ARG;
    chunk_n = std::min(chunk_n, N);
    const HostLayout hl = host_layout(N, C, L, dt, chunk_n);
    if (workspace_bytes < hl.total) return NRC_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return NRC_ERR_ALIGNMENT;

    std::lock_guard<std::mutex> lk(g_host_mu);      // the per-device pipe is shared
    HostPipe* hp = nullptr;
    nrc_status s = host_pipe(&hp);
    if (s != NRC_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t es = dt == NRC_F32 ? 4 : 2;
    const size_t sample = (size_t)C * L * es;
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    // Parameters and weights: copied and packed on the caller's stream.
    float* par = reinterpret_cast<float*>(ws + hl.par);
    bool good = ok(cudaMemcpyAsync(par, rm_host, C * sizeof(float), cudaMemcpyHostToDevice, st)) &&
                ok(cudaMemcpyAsync(par + C, rv_host, C * sizeof(float), cudaMemcpyHostToDevice,
                                   st)) &&
                ok(cudaMemcpyAsync(par + 2 * C, gamma_host, C * sizeof(float),
                                   cudaMemcpyHostToDevice, st)) &&
                ok(cudaMemcpyAsync(par + 3 * C, beta_host, C * sizeof(float),
                                   cudaMemcpyHostToDevice, st)) &&
                ok(cudaMemcpyAsync(ws + hl.w, weight_host, (size_t)C * C * 3 * es,
                                   cudaMemcpyHostToDevice, st)) &&
                (!bias_host || ok(cudaMemcpyAsync(ws + hl.b, bias_host, (size_t)C * es,
                                                  cudaMemcpyHostToDevice, st)));
    if (!good) return NRC_ERR_CUDA;
    s = block_pack(ws + hl.w, dt, C, ws, st);
    if (s != NRC_OK) return s;
    // The library streams start after everything already on the caller's stream
    // (the workspace may still be in use by an earlier call).
    if (!ok(cudaEventRecord(hp->start, st)) || !ok(cudaStreamWaitEvent(hp->in, hp->start, 0)) ||
        !ok(cudaStreamWaitEvent(hp->out, hp->start, 0)))
        return NRC_ERR_CUDA;
    const uint8_t* xh = static_cast<const uint8_t*>(x_host);
    uint8_t* oh = static_cast<uint8_t*>(out_host);
    // Chunk sizes ramp up and down (chunk_n/4, chunk_n/2, chunk_n ..., chunk_n/2,
    // chunk_n/4): the first copy-in and the last copy-out overlap nothing, so
    // they are kept short.
    const std::vector<int> sizes = host_chunk_sizes(N, chunk_n);
    const int n_chunks = (int)sizes.size();
    int n0 = 0;
    for (int j = 0; j < n_chunks; n0 += sizes[j], ++j) {
        const int b = j & 1;
        const int cn = sizes[j];
        const size_t bytes = (size_t)cn * sample;
        // copy-in: buffer b is free once the GEMM of chunk j-2 has read it
        if (j >= 2 && !ok(cudaStreamWaitEvent(hp->in, hp->ev_gemm[b], 0))) return NRC_ERR_CUDA;
        if (!ok(cudaMemcpyAsync(ws + hl.x[b], xh + (size_t)n0 * sample, bytes,
                                cudaMemcpyHostToDevice, hp->in)) ||
            !ok(cudaEventRecord(hp->ev_in[b], hp->in)))
            return NRC_ERR_CUDA;
        // GEMM: after its copy-in, and after chunk j-2's copy-out read buffer b
        if (!ok(cudaStreamWaitEvent(st, hp->ev_in[b], 0)) ||
            (j >= 2 && !ok(cudaStreamWaitEvent(st, hp->ev_out[b], 0))))
            return NRC_ERR_CUDA;
        s = block_gemm(ws + hl.x[b], ws + hl.o[b], dt, cn, C, L, dilation, padding, par,
                       par + C, par + 2 * C, par + 3 * C, bn_eps,
                       bias_host ? static_cast<const void*>(ws + hl.b) : nullptr, ws, nullptr,
                       nullptr, st);
        if (s != NRC_OK) return s;
        if (!ok(cudaEventRecord(hp->ev_gemm[b], st))) return NRC_ERR_CUDA;
        // copy-out
        if (!ok(cudaStreamWaitEvent(hp->out, hp->ev_gemm[b], 0)) ||
            !ok(cudaMemcpyAsync(oh + (size_t)n0 * sample, ws + hl.o[b], bytes,
                                cudaMemcpyDeviceToHost, hp->out)) ||
            !ok(cudaEventRecord(hp->ev_out[b], hp->out)))
            return NRC_ERR_CUDA;
    }
    // The caller's stream resumes once the last copy-out has landed.
    if (!ok(cudaEventRecord(hp->join, hp->out)) || !ok(cudaStreamWaitEvent(st, hp->join, 0)))
        return NRC_ERR_CUDA;
    return NRC_OK;
}

static size_t gn_partials_offset(const ConvPlan& pl) {
    return (pl.wpack_bytes + 255) & ~(size_t)255;
}

namespace {

constexpr int kMaxConvTaps = 64;

// Output length of Conv1d (PyTorch's definition):
// floor((T + 2*padding - dilation*(kernel_size - 1) - 1) / stride) + 1, or 0
// when the arguments are out of range or the result is not positive.
long long conv1d_out_len(int T, int kernel_size, int stride, int padding, int dilation) {
    if (T <= 0 || kernel_size <= 0 || stride <= 0 || padding < 0 || dilation <= 0) return 0;
    const long long span = (long long)dilation * (kernel_size - 1) + 1;
    const long long num = (long long)T + 2LL * padding - span;
    if (num < 0) return 0;
    return num / stride + 1;
}

// Position arithmetic of the kernels (t*stride - padding + k*dilation, box
// starts) is 32-bit: every input position a tap can reach must fit.
bool conv_positions_fit(int T, int kernel_size, int stride, int padding, int dilation,
                        long long T_out) {
    const long long reach = (T_out + kBM) * (long long)stride + (long long)dilation * kernel_size;
    return reach + padding + T < (1LL << 30);
}

}  // namespace

extern "C" int nrc_conv1d_output_length(int T, int kernel_size, int stride, int padding,
                                        int dilation) {
    const long long t = conv1d_out_len(T, kernel_size, stride, padding, dilation);
    return t > 0 && t < (1LL << 30) ? (int)t : 0;
}

extern "C" size_t nrc_conv1d_groupnorm_workspace_size(int N, int C_in, int C_out, int T,
                                                      int kernel_size, int stride, int padding,
                                                      int dilation, int num_groups) {
    if (N <= 0 || C_in <= 0 || C_out <= 0 || num_groups <= 0) return 0;
    if (kernel_size > kMaxConvTaps) return 0;
    const int T_out = nrc_conv1d_output_length(T, kernel_size, stride, padding, dilation);
    if (T_out <= 0) return 0;
    const ConvPlan pl = plan_conv(N, C_in, C_out, T_out, 2, false, 0, 0, kernel_size);
    return gn_partials_offset(pl) + (size_t)N * num_groups * pl.n_tt * kBM * sizeof(float2);
}

namespace {

// The argument checks of the Conv1d + GroupNorm entries (device and host
// buffers alike); T_out receives the conv's output length.
nrc_status gn_check(const void* x, const void* out, int N, int C_in, int C_out, int T,
                    int kernel_size, int stride, int padding, int dilation,
                    const void* conv_weight, int num_groups, const float* gn_gamma,
                    const float* gn_beta, float eps, const void* workspace, int* T_out_p) {
    if (!x || !out || !conv_weight || !workspace) return NRC_ERR_INVALID_ARG;
    if (N <= 0 || C_in <= 0 || C_out <= 0 || T <= 0 || num_groups <= 0)
        return NRC_ERR_INVALID_ARG;
    if (kernel_size <= 0 || stride <= 0 || padding < 0 || dilation <= 0)
        return NRC_ERR_INVALID_ARG;
    if ((gn_gamma == nullptr) != (gn_beta == nullptr)) return NRC_ERR_INVALID_ARG;
    if (C_out % num_groups != 0) return NRC_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return NRC_ERR_INVALID_ARG;
    const long long T_out_ll = conv1d_out_len(T, kernel_size, stride, padding, dilation);
    if (T_out_ll <= 0) return NRC_ERR_INVALID_ARG;        // the kernel does not fit the input
    if (kernel_size > kMaxConvTaps) return NRC_ERR_UNSUPPORTED;
    if (!conv_positions_fit(T, kernel_size, stride, padding, dilation, T_out_ll))
        return NRC_ERR_UNSUPPORTED;
    const int T_out = (int)T_out_ll;
    const int cpg = C_out / num_groups;
    if (C_out > 256 && 256 % cpg != 0) return NRC_ERR_UNSUPPORTED;
    if (ranges_overlap(x, (size_t)N * C_in * T * 4, out, (size_t)N * C_out * T_out * 4))
        return NRC_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return NRC_ERR_ALIGNMENT;
    *T_out_p = T_out;
    return NRC_OK;
}

}  // namespace

extern "C" nrc_status nrc_conv1d_groupnorm(const float* x, float* out, int N, int C_in, int C_out,
                                           int T, int kernel_size, int stride, int padding,
                                           int dilation, const float* conv_weight,
                                           const float* conv_bias, int num_groups,
                                           const float* gn_gamma, const float* gn_beta, float eps,
                                           void* workspace, size_t workspace_bytes,
                                           void* stream) {
    int T_out = 0;
    const nrc_status chk = gn_check(x, out, N, C_in, C_out, T, kernel_size, stride, padding,
                                    dilation, conv_weight, num_groups, gn_gamma, gn_beta, eps,
                                    workspace, &T_out);
    if (chk != NRC_OK) return chk;
    const int cpg = C_out / num_groups;
    ConvPlan pl = plan_conv(N, C_in, C_out, T_out, 2, false, 0, 0, kernel_size);
    if (workspace_bytes < nrc_conv1d_groupnorm_workspace_size(N, C_in, C_out, T, kernel_size,
                                                              stride, padding, dilation,
                                                              num_groups))
        return NRC_ERR_WORKSPACE;
    if ((long long)N * pl.n_tt * pl.n_ot >= (1LL << 30)) return NRC_ERR_UNSUPPORTED;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    ConvParams p{};
    p.x = x;
    p.out = out;
    // One wave (every tile on its own CTA, all resident): the GroupNorm is
    // finished inside the GEMM kernel behind a grid-wide barrier.  Stride 1
    // with 16-byte aligned rows stages x by TMA boxes; otherwise the prologue
    // warps load x directly (either kernel also runs the one-wave path).
    p.fused = (pl.g.num_tiles <= device_sm_count() && device_coop_launch()) ? 1 : 0;
    bool staged = plan_conv_staged<float>(p, pl, N, C_in, C_out, T_out, false, T, stride,
                                          kernel_size);
    p.N = N;
    p.Cin = C_in;
    p.Cout = C_out;
    p.L = T_out;
    p.Lin = T;
    p.pad = padding;
    p.dil = dilation;
    p.stride = stride;
    p.ksz = kernel_size;
    p.n_tt = pl.n_tt;
    p.n_ot = pl.n_ot;
    p.n_chunks = pl.n_chunks;
    p.n_kiters = pl.g.num_kiters;
    p.BN = pl.g.BN;
    p.bias = conv_bias;
    p.bias_off = 0;
    p.wpack = ws;
    p.partials = reinterpret_cast<float2*>(ws + gn_partials_offset(pl));
    p.G = num_groups;
    p.cpg = cpg;
    if (p.fused) {
        // one launch: the GEMM kernel also repacks the weights
        ConvParams p1 = p;
        GemmPlan g1 = pl.g;
        uint8_t* part = ws + gn_partials_offset(pl);
        p1.grid_counter = reinterpret_cast<uint32_t*>(part);
        p1.pack_counter = reinterpret_cast<uint32_t*>(part + 4);
        p1.w_raw = conv_weight;
        p1.wpack_out = ws;
        p1.tile_stats = reinterpret_cast<float4*>(part + 256);
        p1.gn_gamma = gn_gamma;
        p1.gn_beta = gn_beta;
        p1.gn_eps = eps;
        p1.status = device_status_ptr();
        p1.timeout_ns = grid_barrier_timeout_ns();
        if (p1.status == nullptr) return NRC_ERR_CUDA;
        if (cudaMemsetAsync(p1.grid_counter, 0, 2 * sizeof(uint32_t), st) != cudaSuccess)
            return NRC_ERR_CUDA;
        g1.coop = true;
        const nrc_status s1 =
            staged ? launch_gemm<ConvProblem<float, ConvEpi::kGroupStats, true, true>, 2>(
                         "conv_gn_gemm", p1, g1, st)
                   : launch_gemm<ConvProblem<float, ConvEpi::kGroupStats, false, true>, 2>(
                         "conv_gn_gemm", p1, g1, st);
        if (s1 != NRC_ERR_UNSUPPORTED) return s1;
        // refused (the CTAs cannot all be resident now): the two-kernel path,
        // planned without the fused epilogue's shared memory
        p.fused = 0;
        staged = plan_conv_staged<float>(p, pl, N, C_in, C_out, T_out, false, T, stride,
                                         kernel_size);
    }
    {
        const size_t units = pl.wpack_bytes / 16 / 2;
        TraceScope ts("pack_conv_weight", st);
        pack_conv_weight_kernel<float, 2><<<elementwise_grid(units), 256, 0, st>>>(
            conv_weight, ws, C_out, C_in, pl.g.BN, pl.n_ot, pl.n_chunks, kernel_size);
        if (cudaGetLastError() != cudaSuccess) return NRC_ERR_CUDA;
        pl.g.b_after_prev = true;      // the GEMM launched behind the repack
    }
    nrc_status s =
        staged ? launch_gemm<ConvProblem<float, ConvEpi::kGroupStats, true>, 2>("conv_gn_gemm",
                                                                               p, pl.g, st)
               : launch_gemm<ConvProblem<float, ConvEpi::kGroupStats, false>, 2>(
                     "conv_gn_gemm", p, pl.g, st);
    if (s != NRC_OK) return s;
    {
        TraceScope ts("groupnorm_finalize_normalize", st);
        groupnorm_finalize_normalize_kernel<<<N * num_groups, 256, 0, st>>>(
            out, p.partials, pl.n_tt, C_out, T_out, num_groups, gn_gamma, gn_beta, eps);
    }
    return cuda_status(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// Conv1d + GroupNorm on host buffers: the batch in chunks of samples (a
// sample's group statistics involve that sample alone), so the copy-in of
// chunk j+1, the call on chunk j and the copy-out of chunk j-1 run at once.
// Each chunk is an ordinary call of the device entry on its samples.
// ---------------------------------------------------------------------------
namespace {

struct GnHostLayout {
    size_t par_w, par_b, par_g, par_be, x[2], o[2], total;
};

GnHostLayout gn_host_layout(int C_in, int C_out, int T, int T_out, int kernel_size,
                            size_t gn_ws, int chunk_n) {
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    GnHostLayout h{};
    h.par_w = up(gn_ws);
    h.par_b = up(h.par_w + (size_t)C_out * C_in * kernel_size * 4);
    h.par_g = up(h.par_b + (size_t)C_out * 4);
    h.par_be = up(h.par_g + (size_t)C_out * 4);
    h.x[0] = up(h.par_be + (size_t)C_out * 4);
    h.x[1] = up(h.x[0] + (size_t)chunk_n * C_in * T * 4);
    h.o[0] = up(h.x[1] + (size_t)chunk_n * C_in * T * 4);
    h.o[1] = up(h.o[0] + (size_t)chunk_n * C_out * T_out * 4);
    h.total = h.o[1] + (size_t)chunk_n * C_out * T_out * 4;
    return h;
}

}  // namespace

extern "C" size_t nrc_conv1d_groupnorm_host_workspace_size(int N, int C_in, int C_out, int T,
                                                           int kernel_size, int stride,
                                                           int padding, int dilation,
                                                           int num_groups, int chunk_n) {
    if (N <= 0 || chunk_n <= 0) return 0;
    chunk_n = std::min(chunk_n, N);
    const size_t gn_ws = nrc_conv1d_groupnorm_workspace_size(chunk_n, C_in, C_out, T, kernel_size,
                                                             stride, padding, dilation,
                                                             num_groups);
    if (gn_ws == 0) return 0;
    const int T_out = nrc_conv1d_output_length(T, kernel_size, stride, padding, dilation);
    return gn_host_layout(C_in, C_out, T, T_out, kernel_size, gn_ws, chunk_n).total;
}

extern "C" nrc_status nrc_conv1d_groupnorm_host(
    const float* x_host, float* out_host, int N, int C_in, int C_out, int T, int kernel_size,
    int stride, int padding, int dilation, const float* conv_weight_host,
    const float* conv_bias_host, int num_groups, const float* gn_gamma_host,
    const float* gn_beta_host, float eps, int chunk_n, void* workspace, size_t workspace_bytes,
    void* stream) {
    int T_out = 0;
    const nrc_status chk = gn_check(x_host, out_host, N, C_in, C_out, T, kernel_size, stride,
                                    padding, dilation, conv_weight_host, num_groups,
                                    gn_gamma_host, gn_beta_host, eps, workspace, &T_out);
    if (chk != NRC_OK) return chk;
    if (chunk_n <= 0) return NRC_ERR_INVALID_ARG;
    chunk_n = std::min(chunk_n, N);
    const size_t gn_ws = nrc_conv1d_groupnorm_workspace_size(chunk_n, C_in, C_out, T, kernel_size,
                                                             stride, padding, dilation,
                                                             num_groups);
    if (gn_ws == 0) return NRC_ERR_INVALID_ARG;
    const GnHostLayout hl = gn_host_layout(C_in, C_out, T, T_out, kernel_size, gn_ws, chunk_n);
    if (workspace_bytes < hl.total) return NRC_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return NRC_ERR_ALIGNMENT;

    std::lock_guard<std::mutex> lk(g_host_mu);      // the per-device pipe is shared
    HostPipe* hp = nullptr;
    nrc_status s = host_pipe(&hp);
    if (s != NRC_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    // Weights and affine parameters: copied once on the caller's stream.
    float* d_w = reinterpret_cast<float*>(ws + hl.par_w);
    float* d_b = reinterpret_cast<float*>(ws + hl.par_b);
    float* d_g = reinterpret_cast<float*>(ws + hl.par_g);
    float* d_be = reinterpret_cast<float*>(ws + hl.par_be);
    const size_t cb = (size_t)C_out * 4;
    const bool good =
        ok(cudaMemcpyAsync(d_w, conv_weight_host, (size_t)C_out * C_in * kernel_size * 4,
                           cudaMemcpyHostToDevice, st)) &&
        (!conv_bias_host || ok(cudaMemcpyAsync(d_b, conv_bias_host, cb, cudaMemcpyHostToDevice,
                                               st))) &&
        (!gn_gamma_host || ok(cudaMemcpyAsync(d_g, gn_gamma_host, cb, cudaMemcpyHostToDevice,
                                              st))) &&
        (!gn_beta_host ||
         ok(cudaMemcpyAsync(d_be, gn_beta_host, cb, cudaMemcpyHostToDevice, st)));
    if (!good) return NRC_ERR_CUDA;
    // The library streams start after everything already on the caller's stream.
    if (!ok(cudaEventRecord(hp->start, st)) || !ok(cudaStreamWaitEvent(hp->in, hp->start, 0)) ||
        !ok(cudaStreamWaitEvent(hp->out, hp->start, 0)))
        return NRC_ERR_CUDA;
    const size_t xs = (size_t)C_in * T * 4, os = (size_t)C_out * T_out * 4;   // per sample
    // Equal chunks, no ramp: a call costs about the same whatever its size (the
    // kernel is latency-bound), so fewer calls beat shorter first and last copies.
    std::vector<int> sizes;
    for (int r = N; r > 0; r -= chunk_n) sizes.push_back(std::min(chunk_n, r));
    const int n_chunks = (int)sizes.size();
    int n0 = 0;
    for (int j = 0; j < n_chunks; n0 += sizes[j], ++j) {
        const int b = j & 1;
        const int cn = sizes[j];
        // copy-in: buffer b is free once the call on chunk j-2 has read it
        if (j >= 2 && !ok(cudaStreamWaitEvent(hp->in, hp->ev_gemm[b], 0))) return NRC_ERR_CUDA;
        if (!ok(cudaMemcpyAsync(ws + hl.x[b], reinterpret_cast<const uint8_t*>(x_host) + n0 * xs,
                                (size_t)cn * xs, cudaMemcpyHostToDevice, hp->in)) ||
            !ok(cudaEventRecord(hp->ev_in[b], hp->in)))
            return NRC_ERR_CUDA;
        // the call: after its copy-in, and after chunk j-2's copy-out read buffer b
        if (!ok(cudaStreamWaitEvent(st, hp->ev_in[b], 0)) ||
            (j >= 2 && !ok(cudaStreamWaitEvent(st, hp->ev_out[b], 0))))
            return NRC_ERR_CUDA;
        s = nrc_conv1d_groupnorm(reinterpret_cast<const float*>(ws + hl.x[b]),
                                 reinterpret_cast<float*>(ws + hl.o[b]), cn, C_in, C_out, T,
                                 kernel_size, stride, padding, dilation, d_w,
                                 conv_bias_host ? d_b : nullptr, num_groups,
                                 gn_gamma_host ? d_g : nullptr, gn_beta_host ? d_be : nullptr,
                                 eps, ws, gn_ws, stream);
        if (s != NRC_OK) return s;
        if (!ok(cudaEventRecord(hp->ev_gemm[b], st))) return NRC_ERR_CUDA;
        // copy-out
        if (!ok(cudaStreamWaitEvent(hp->out, hp->ev_gemm[b], 0)) ||
            !ok(cudaMemcpyAsync(reinterpret_cast<uint8_t*>(out_host) + n0 * os, ws + hl.o[b],
                                (size_t)cn * os, cudaMemcpyDeviceToHost, hp->out)) ||
            !ok(cudaEventRecord(hp->ev_out[b], hp->out)))
            return NRC_ERR_CUDA;
    }
    // The caller's stream resumes once the last copy-out has landed.
    if (!ok(cudaEventRecord(hp->join, hp->out)) || !ok(cudaStreamWaitEvent(st, hp->join, 0)))
        return NRC_ERR_CUDA;
    return NRC_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of nrc_prenorm_dilconv_residual.
//
// The regular entry point takes its scratch (the repacked weight image) from a
// caller-provided workspace.  Some callers cannot provide one: their device
// memory is owned by a host framework's allocator that forbids side
// allocations, or they run in a loop where a cudaMalloc/cudaFree (and the
// device-wide synchronisation it can bring) is not acceptable.  This variant
// keeps its scratch in a fixed-size array in the library's own device memory
// instead, so it allocates nothing.
//
// The array is kNoAllocScratchBytes (4 MiB) on every GPU that loads the
// library, held until the process exits; the weight image of fp32 C <= 512
// (bf16 C <= 768) fits.  Larger C is rejected with NRC_ERR_WORKSPACE.  Every
// call rewrites the whole image it uses (padding included), so no contents
// need clearing, but all calls share the one array: calls that overlap on the
// GPU (two streams, two host threads) race on it.
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64];   // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device.  The name of a
// __device__ array in host code is only a host-side stand-in, so the address
// is looked up (once per device, with that device current) and cached.  A
// cudaDeviceReset() on the device unloads the module and makes the cached
// address stale: the entry point must not be used on that device afterwards.
nrc_status noalloc_scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NRC_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return NRC_ERR_CUDA;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return NRC_OK;
}
}  // namespace

extern "C" size_t nrc_prenorm_dilconv_residual_noalloc_max_bytes(void) {
    return kNoAllocScratchBytes;
}

extern "C" nrc_status nrc_prenorm_dilconv_residual_noalloc(
    const void* x, void* out, nrc_dtype dt, int N, int C, int L, int kernel_size, int dilation,
    int padding, const float* rm, const float* rv, const float* gamma, const float* beta,
    float bn_eps, const void* conv_weight, const void* conv_bias, void* stream) {
    // The same argument checks (and status codes) as the workspace entry point
    // come first; then the array's size limit; only then any CUDA call.
    const nrc_status c = block_check_args(x, out, dt, N, C, L, kernel_size, dilation, padding,
                                          rm, rv, gamma, beta, bn_eps, conv_weight);
    if (c != NRC_OK) return c;
    if (nrc_prenorm_dilconv_residual_workspace_size(C, dt) > kNoAllocScratchBytes)
        return NRC_ERR_WORKSPACE;
    void* scratch = nullptr;
    const nrc_status s = noalloc_scratch_address(&scratch);
    if (s != NRC_OK) return s;
    return nrc_prenorm_dilconv_residual(x, out, dt, N, C, L, kernel_size, dilation, padding, rm,
                                        rv, gamma, beta, bn_eps, conv_weight, conv_bias, scratch,
                                        kNoAllocScratchBytes, stream);
}
