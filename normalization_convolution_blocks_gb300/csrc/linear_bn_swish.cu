// Linear + BatchNorm1d + scalar bias + divide + Swish ("Kimi-K2.6 l2_p97").
//
// GEMM orientation: tile rows are 128 output features j (A = rows of the Linear
// weight, converted to bf16 hi/lo by the prologue warps straight from fp32, so
// the large weight is never rewritten), tile columns are BN batch rows b (B =
// x, split into bf16 hi/lo once per call into the shared-memory image).
// D[j][b] = y[b][j] - lin_bias[j].  When W's rows are 16-byte aligned, each
// stage's 128 x 64 block of W is copied by TMA (two 32-wide boxes in the
// 128-byte swizzle, so a lane reading its own row is bank-conflict free) and
// the prologue warps convert it from shared memory.  With features on TMEM lanes, each thread
// owns one column j of y: its epilogue stores y (coalesced across the warp)
// and keeps the column's (count, mean, M2) over the tile's batch rows, so the
// batch statistics need no cross-thread reduction.
//
// Launches per call in training mode: pack x -> GEMM (y + per-tile column
// statistics) -> finalize (batch mean/var, running-stat update) -> normalize
// + bias + divide + Swish in place.  Each of the last three is launched behind
// the one before it (programmatic dependent launch) and waits for it before
// reading its results.  In eval mode the statistics are the running buffers,
// known before the GEMM starts, so the whole chain is the GEMM's epilogue:
// pack x -> GEMM writing out directly (y never reaches memory).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "nrc_launch.cuh"

namespace nrc {

struct LinearParams {
    CUtensorMap wmap;        // W as (IN, OUT, 1) in 32 x 128 x 1 boxes, 128B-swizzled
    const float* W;          // (OUT, IN)
    const uint8_t* xpack;    // packed x image
    float* out;              // (B, OUT): receives y
    const float* lin_bias;   // (OUT) or NULL
    float4* partials;        // [bt * OUT + j] = (count, mean, M2, 0)
    // eval mode (the epilogue applies BN with the running statistics, the
    // scalar bias, the divide and Swish)
    const float* running_mean;
    const float* running_var;
    const float* gamma;      // NULL with beta NULL: affine off
    const float* beta;
    const float* add_bias;   // one element on the device
    float bn_eps, divide_value;
    int B, IN, OUT;
    int n_jt, n_bt, n_kiters, BN;
    int vec_ok;              // W 16-byte aligned and IN % 4 == 0
};

struct LinearTile {
    int jt, bt;
};

// x * sigmoid(x) = u / (1 + e^-u), with CUDA's fast exponential and division
// intrinsics (a few ulp; far inside the 1e-4 parity bar).  For u < -87 the
// denominator overflows and __fdividef returns 0, the limit of the function.
__device__ __forceinline__ float swish_f(float u) { return __fdividef(u, 1.0f + __expf(-u)); }

template <bool STAGED, bool EVAL = false>
struct LinearProblem {
    using Params = LinearParams;
    using Tile = LinearTile;
    static constexpr bool kStagedA = STAGED;
    static constexpr bool kPackedA = false;                    // read_a returns fp32 values
    static constexpr uint32_t kBoxBytes = 2u * 128u * 128u;   // two 32-float x 128-row boxes

    // Tiles of one feature block are adjacent, so the CTAs reading the same
    // weight rows run together and the weight is fetched from HBM once.
    static __device__ __forceinline__ Tile tile_info(const Params& p, int tile) {
        return Tile{tile / p.n_bt, tile % p.n_bt};
    }

    static __device__ __forceinline__ uint32_t* b_ready_counter(const Params&) { return nullptr; }

    static __device__ void setup(const Params&, uint8_t*, int, int) {}

    static __device__ __forceinline__ void load_a(const Params& p, const Tile& tl, int kiter,
                                                  int row, int k0, float (&v)[32]) {
        const int j = tl.jt * kBM + row;
        const int k = kiter * kBK + k0;
        if (j >= p.OUT) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
            return;
        }
        const float* wr = p.W + (size_t)j * p.IN + k;
        if (p.vec_ok && k + 32 <= p.IN) {
            const float4* w4 = reinterpret_cast<const float4*>(wr);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 q = __ldg(w4 + i);
                v[4 * i] = q.x;
                v[4 * i + 1] = q.y;
                v[4 * i + 2] = q.z;
                v[4 * i + 3] = q.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = (k + i < p.IN) ? __ldg(wr + i) : 0.f;
        }
    }

    static __device__ __forceinline__ void finish_a(const Params&, const uint8_t*, const Tile&,
                                                    int, int, int, float (&)[32]) {}

    // Staged A: K columns kiter*64 .. +32 and +32 .. +64 of rows jt*128 .. +128
    // as two boxes; rows past OUT and columns past IN are zero.
    static __device__ __forceinline__ void issue_a_box(const Params& p, const Tile& tl,
                                                       int kiter, uint32_t dst, uint32_t bar) {
        tma_load_3d(dst, &p.wmap, kiter * kBK, tl.jt * kBM, 0, bar);
        tma_load_3d(dst + kBoxBytes / 2, &p.wmap, kiter * kBK + 32, tl.jt * kBM, 0, bar);
    }

    static __device__ __forceinline__ void read_a(const Params&, const uint8_t*, const Tile&,
                                                  int, int row, int k0, int, uint32_t box,
                                                  float (&v)[32]) {
        const uint32_t rb = box + (uint32_t)(k0 / 32) * (kBoxBytes / 2) + (uint32_t)row * 128u;
        const uint32_t sw = (uint32_t)(row & 7);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 q = ld_shared_v4f(rb + (((uint32_t)c ^ sw) << 4));
            v[4 * c] = q.x;
            v[4 * c + 1] = q.y;
            v[4 * c + 2] = q.z;
            v[4 * c + 3] = q.w;
        }
    }

    static __device__ __forceinline__ const void* b_src(const Params& p, const Tile& tl,
                                                        int kiter) {
        return p.xpack + ((size_t)tl.bt * p.n_kiters + kiter) * 2 * (size_t)p.BN * 128u;
    }

    template <class Acquire, class Release>
    static __device__ __forceinline__ bool epilogue(const Params& p, const uint8_t*,
                                                    const Tile& tl, int quarter, int lane,
                                                    uint32_t taddr, int BN, int halves,
                                                    Acquire& acquire, Release& release) {
        const int j = tl.jt * kBM + quarter * 32 + lane;
        const bool j_ok = j < p.OUT;
        const int b0 = tl.bt * BN;
        const int bvalid = p.B - b0;               // batch rows of this tile that exist
        if constexpr (EVAL) {
            // u = (y - mu_j) * scale_j + shift_j with the running statistics
            // (the same coefficients the finalize kernel forms), out = swish(u)
            float lb = 0.f, c = 0.f, sc = 0.f, sh = 0.f;
            if (j_ok) {
                lb = p.lin_bias ? __ldg(p.lin_bias + j) : 0.f;
                c = __ldg(p.running_mean + j);
                const float inv = 1.0f / sqrtf(__ldg(p.running_var + j) + p.bn_eps);
                const float g = p.gamma ? __ldg(p.gamma + j) : 1.f;
                const float be = p.beta ? __ldg(p.beta + j) : 0.f;
                sc = g * inv / p.divide_value;
                sh = (be + __ldg(p.add_bias)) / p.divide_value;
            }
            for (int h = 0; h < halves; ++h)
                if (!acquire(h)) return false;
            float* outj = p.out + (size_t)b0 * p.OUT + j;
            for (int cc = 0; cc < BN && cc < bvalid; cc += 16) {
                float v[16];
                tmem_ld16(taddr + (uint32_t)cc, v);
                const int n = min(16, bvalid - cc);   // uniform
                float* op = outj + (size_t)cc * p.OUT;
                if (j_ok) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (i < n) op[(size_t)i * p.OUT] = swish_f(fmaf(v[i] + lb - c, sc, sh));
                }
            }
            for (int h = 0; h < halves; ++h) release(h);
            return true;
        }
        for (int h = 0; h < halves; ++h)
            if (!acquire(h)) return false;
        const float lb = (j_ok && p.lin_bias) ? __ldg(p.lin_bias + j) : 0.f;
        float cnt = 0.f, mean = 0.f, m2 = 0.f;
        float* outj = p.out + (size_t)b0 * p.OUT + j;
        for (int cc = 0; cc < BN && cc < bvalid; cc += 16) {
            float v[16];
            tmem_ld16(taddr + (uint32_t)cc, v);
            const int n = min(16, bvalid - cc);   // uniform
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] += lb;
            float* op = outj + (size_t)cc * p.OUT;
            if (j_ok) {
                if (n == 16) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) op[(size_t)i * p.OUT] = v[i];
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (i < n) op[(size_t)i * p.OUT] = v[i];
                }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (i < n) {                         // Welford over the tile's rows
                    cnt += 1.f;
                    const float d = v[i] - mean;
                    mean += d / cnt;
                    m2 += d * (v[i] - mean);
                }
            }
        }
        if (j_ok) p.partials[(size_t)tl.bt * p.OUT + j] = make_float4(cnt, mean, m2, 0.f);
        for (int h = 0; h < halves; ++h) release(h);
        return true;
    }
};

// ---------------------------------------------------------------------------
// x (B, IN) fp32 -> per (batch tile, 64-wide K chunk) the B-stage image: hi and
// lo bf16 parts of BN rows x 64, 128B-swizzled; rows past B, columns past IN 0.
// ---------------------------------------------------------------------------
__global__ void pack_rows_split_kernel(const float* __restrict__ x, uint8_t* __restrict__ pack,
                                       int B, int IN, int BN, int n_bt, int n_kiters) {
    griddep_launch_dependents();       // the GEMM may launch; it waits before reading B
    const size_t total = (size_t)n_bt * n_kiters * BN * 8;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int j = (int)(idx & 7);
        size_t rest = idx >> 3;
        const int row = (int)(rest % BN);
        rest /= BN;
        const int kiter = (int)(rest % n_kiters);
        const int bt = (int)(rest / n_kiters);
        const int b = bt * BN + row;
        const int k0 = kiter * kBK + j * 8;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            v[e] = (b < B && k0 + e < IN) ? __ldg(x + (size_t)b * IN + k0 + e) : 0.f;
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_bf16x2(v[2 * e], v[2 * e + 1], h[e], l[e]);
        const size_t blk = ((size_t)bt * n_kiters + kiter) * 2;
        const uint32_t off = sw128_offset((uint32_t)row, (uint32_t)j);
        *reinterpret_cast<uint4*>(pack + blk * BN * 128 + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(pack + (blk + 1) * BN * 128 + off) =
            make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// ---------------------------------------------------------------------------
// Per column j: merge the per-batch-tile (count, mean, M2) in a fixed order
// into the batch mean and biased variance; in training mode update the
// running statistics (unbiased variance) and num_batches_tracked; emit the
// column's (centre, scale, shift) so that
//   u = (y - centre) * scale + shift = ((y - mu)/sqrt(var + eps)*gamma + beta + bias)/div.
// ---------------------------------------------------------------------------
__global__ void bn_finalize_kernel(const float4* __restrict__ partials, int n_bt, int B, int OUT,
                                   const float* __restrict__ gamma, const float* __restrict__ beta,
                                   float* __restrict__ running_mean, float* __restrict__ running_var,
                                   long long* __restrict__ nbt, float eps, float momentum,
                                   int training, const float* __restrict__ add_bias,
                                   float divide_value, float* __restrict__ colp) {
    griddep_launch_dependents();
    griddep_wait();                    // the GEMM's partials
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (training && nbt && j == 0) *nbt += 1;
    if (j >= OUT) return;
    float mu, var;
    if (training) {
        float cnt = 0.f, mean = 0.f, m2 = 0.f;
        for (int bt = 0; bt < n_bt; ++bt) {
            const float4 q = partials[(size_t)bt * OUT + j];
            const float nab = cnt + q.x;
            if (nab > 0.f) {
                const float delta = q.y - mean;
                const float fb = q.x / nab;
                mean += delta * fb;
                m2 += q.z + delta * delta * cnt * fb;
                cnt = nab;
            }
        }
        mu = mean;
        var = fmaxf(m2 / (float)B, 0.f);
        running_mean[j] = (1.f - momentum) * running_mean[j] + momentum * mu;
        running_var[j] = (1.f - momentum) * running_var[j] +
                         momentum * (m2 / (float)(B - 1));
    } else {
        mu = running_mean[j];
        var = running_var[j];
    }
    const float inv = 1.0f / sqrtf(var + eps);
    const float g = gamma ? gamma[j] : 1.f;
    const float be = beta ? beta[j] : 0.f;
    colp[j] = mu;
    colp[OUT + j] = g * inv / divide_value;
    colp[2 * OUT + j] = (be + add_bias[0]) / divide_value;
}

// out[b][j] = swish((y - mean_j) * scale_j + shift_j), in place.  Threads of
// grid x own 4-column groups (their coefficients stay in registers), grid y
// strides over the rows.  Columns come 4 at a time when OUT % 4 == 0 and out is
// 16-byte aligned, one at a time otherwise.
__global__ void normalize_swish_kernel(float* __restrict__ out, const float* __restrict__ colp,
                                       int B, int OUT) {
    griddep_wait();                    // y from the GEMM, the column parameters
    const int vec = (OUT % 4 == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) ? 4 : 1;
    const int j = (blockIdx.x * blockDim.x + threadIdx.x) * vec;
    if (j >= OUT) return;
    if (vec == 4) {
        const float4 c = *reinterpret_cast<const float4*>(colp + j);
        const float4 s = *reinterpret_cast<const float4*>(colp + OUT + j);
        const float4 h = *reinterpret_cast<const float4*>(colp + 2 * OUT + j);
        for (int b = blockIdx.y; b < B; b += gridDim.y) {
            float4* o4 = reinterpret_cast<float4*>(out + (size_t)b * OUT + j);
            float4 y = *o4;
            y.x = swish_f(fmaf(y.x - c.x, s.x, h.x));
            y.y = swish_f(fmaf(y.y - c.y, s.y, h.y));
            y.z = swish_f(fmaf(y.z - c.z, s.z, h.z));
            y.w = swish_f(fmaf(y.w - c.w, s.w, h.w));
            *o4 = y;
        }
    } else {
        const float c = colp[j], s = colp[OUT + j], h = colp[2 * OUT + j];
        for (int b = blockIdx.y; b < B; b += gridDim.y) {
            float* o = out + (size_t)b * OUT + j;
            *o = swish_f(fmaf(*o - c, s, h));
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct LinearPlan {
    GemmPlan g;
    int n_jt, n_bt;
    size_t xpack_bytes, partials_off, colp_off, total;
};

static LinearPlan plan_linear(int B, int IN, int OUT, uint32_t x_box_bytes = 0) {
    LinearPlan pl{};
    const int BN = B <= 256 ? ((B + 15) / 16) * 16 : 256;
    pl.n_bt = ceil_div(B, BN);
    pl.n_jt = ceil_div(OUT, kBM);
    const int n_kiters = ceil_div(IN, kBK);
    const long long tiles = (long long)pl.n_jt * pl.n_bt;
    pl.g = make_gemm_plan(BN, (int)std::min<long long>(tiles, 1LL << 30), n_kiters, 2, 0,
                          x_box_bytes);
    pl.xpack_bytes = (size_t)pl.n_bt * n_kiters * 2 * BN * 128;
    pl.partials_off = (pl.xpack_bytes + 255) & ~(size_t)255;
    pl.colp_off = (pl.partials_off + (size_t)pl.n_bt * OUT * sizeof(float4) + 255) & ~(size_t)255;
    pl.total = pl.colp_off + (size_t)3 * OUT * sizeof(float);
    return pl;
}

}  // namespace nrc

using namespace nrc;

namespace {

// The Linear chain on device buffers, x already packed at ws (the plan's
// image): the GEMM, then in training mode the finalize and normalize kernels.
// W, out and the per-feature arrays cover out_f features; num_batches_tracked
// (NULL: not counted) is incremented by the finalize kernel.  b_after_prev:
// the kernel just before on the stream wrote the x image.
nrc_status linear_chain(const float* W, float* out, int B, int in_f, int out_f,
                        const float* lin_bias, const float* bn_gamma, const float* bn_beta,
                        float* bn_running_mean, float* bn_running_var,
                        int64_t* num_batches_tracked, float bn_eps, float bn_momentum,
                        int training, const float* add_bias, float divide_value, uint8_t* ws,
                        bool b_after_prev, cudaStream_t st) {
    LinearPlan pl = plan_linear(B, in_f, out_f);
    if ((long long)pl.n_jt * pl.n_bt >= (1LL << 30)) return NRC_ERR_UNSUPPORTED;
    LinearParams p{};
    p.W = W;
    p.xpack = ws;
    p.out = out;
    p.lin_bias = lin_bias;
    p.partials = reinterpret_cast<float4*>(ws + pl.partials_off);
    p.B = B;
    p.IN = in_f;
    p.OUT = out_f;
    p.n_jt = pl.n_jt;
    p.n_bt = pl.n_bt;
    p.n_kiters = pl.g.num_kiters;
    p.BN = pl.g.BN;
    p.vec_ok = (in_f % 4 == 0) && aligned(W, 16);
    // Staged A when W's rows are 16-byte aligned and the driver takes the map.
    bool staged = false;
    if (p.vec_ok) {
        const uint64_t dims[3] = {(uint64_t)in_f, (uint64_t)out_f, 1};
        const uint64_t strides[2] = {(uint64_t)in_f * 4, (uint64_t)in_f * 4 * out_f};
        const uint32_t box[3] = {32u, (uint32_t)kBM, 1u};
        if (encode_tensor_map_3d(&p.wmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, W, dims, strides,
                                 box, false, true)) {
            const LinearPlan ps = plan_linear(B, in_f, out_f, LinearProblem<true>::kBoxBytes);
            if (ps.g.b_stages >= 2 && ps.g.x_depth >= 2) {
                pl = ps;
                staged = true;
            }
        }
    }
    float* colp = reinterpret_cast<float*>(ws + pl.colp_off);
    pl.g.b_after_prev = b_after_prev;
    if (!training) {
        // eval: one GEMM whose epilogue writes out; the running statistics are
        // inputs here, so nothing else runs
        p.running_mean = bn_running_mean;
        p.running_var = bn_running_var;
        p.gamma = bn_gamma;
        p.beta = bn_beta;
        p.add_bias = add_bias;
        p.bn_eps = bn_eps;
        p.divide_value = divide_value;
        return staged ? launch_gemm<LinearProblem<true, true>, 2>("linear_gemm", p, pl.g, st)
                      : launch_gemm<LinearProblem<false, true>, 2>("linear_gemm", p, pl.g, st);
    }
    nrc_status s = staged ? launch_gemm<LinearProblem<true>, 2>("linear_gemm", p, pl.g, st)
                          : launch_gemm<LinearProblem<false>, 2>("linear_gemm", p, pl.g, st);
    if (s != NRC_OK) return s;
    {
        TraceScope ts("bn_finalize", st);
        const cudaError_t e = launch_after_prev(
            bn_finalize_kernel, dim3(ceil_div(out_f, 256)), dim3(256), st,
            static_cast<const float4*>(p.partials), pl.n_bt, B, out_f, bn_gamma, bn_beta,
            bn_running_mean, bn_running_var, reinterpret_cast<long long*>(num_batches_tracked),
            bn_eps, bn_momentum, training, add_bias, divide_value, colp);
        if (e != cudaSuccess) return cuda_status(e);
    }
    if (cudaGetLastError() != cudaSuccess) return NRC_ERR_CUDA;
    {
        TraceScope ts("normalize_swish", st);
        // enough CTAs to fill the GPU several times over: 256 threads cover 1024
        // (or 256) columns, grid y splits the rows
        const int vec = (out_f % 4 == 0 && aligned(out, 16)) ? 4 : 1;
        const int gx = ceil_div(ceil_div(out_f, vec), 256);
        const int gy = std::max(1, std::min(B, device_sm_count() * 8 / std::max(gx, 1)));
        const cudaError_t e = launch_after_prev(normalize_swish_kernel, dim3(gx, gy), dim3(256),
                                                st, out, static_cast<const float*>(colp), B,
                                                out_f);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return cuda_status(cudaGetLastError());
}

// Packs x (B x in_f, device) into the workspace's x image.
nrc_status linear_pack_x(const float* x, int B, int in_f, uint8_t* ws, cudaStream_t st) {
    const LinearPlan pl = plan_linear(B, in_f, 1);
    const size_t units = (size_t)pl.n_bt * pl.g.num_kiters * pl.g.BN * 8;
    TraceScope ts("pack_rows_split", st);
    pack_rows_split_kernel<<<elementwise_grid(units), 256, 0, st>>>(x, ws, B, in_f, pl.g.BN,
                                                                     pl.n_bt, pl.g.num_kiters);
    return cuda_status(cudaGetLastError());
}

// The argument checks shared by the device and host-buffer entries.
nrc_status linear_check(const void* x, const void* out, int B, int in_f, int out_f,
                        const void* lin_weight, const float* bn_gamma, const float* bn_beta,
                        const float* bn_running_mean, const float* bn_running_var,
                        float bn_eps, float bn_momentum, int training, const float* add_bias,
                        float divide_value, const void* workspace) {
    if (!x || !out || !lin_weight || !bn_running_mean || !bn_running_var || !add_bias ||
        !workspace)
        return NRC_ERR_INVALID_ARG;
    if (B <= 0 || in_f <= 0 || out_f <= 0) return NRC_ERR_INVALID_ARG;
    if ((bn_gamma == nullptr) != (bn_beta == nullptr)) return NRC_ERR_INVALID_ARG;
    if (!(bn_eps >= 0.f) || !std::isfinite(bn_eps)) return NRC_ERR_INVALID_ARG;
    if (!(bn_momentum >= 0.f && bn_momentum <= 1.f)) return NRC_ERR_INVALID_ARG;
    if (divide_value == 0.f || !std::isfinite(divide_value)) return NRC_ERR_INVALID_ARG;
    if (training != 0 && training != 1) return NRC_ERR_INVALID_ARG;
    if (training && B < 2) return NRC_ERR_UNSUPPORTED;
    if (ranges_overlap(x, (size_t)B * in_f * 4, out, (size_t)B * out_f * 4))
        return NRC_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return NRC_ERR_ALIGNMENT;
    return NRC_OK;
}

}  // namespace

extern "C" size_t nrc_linear_bn_swish_workspace_size(int B, int in_f, int out_f) {
    if (B <= 0 || in_f <= 0 || out_f <= 0) return 0;
    return plan_linear(B, in_f, out_f).total;
}

extern "C" nrc_status nrc_linear_bn_swish(
    const float* x, float* out, int B, int in_f, int out_f, const float* lin_weight,
    const float* lin_bias, const float* bn_gamma, const float* bn_beta, float* bn_running_mean,
    float* bn_running_var, int64_t* num_batches_tracked, float bn_eps, float bn_momentum,
    int training, const float* add_bias, float divide_value, void* workspace,
    size_t workspace_bytes, void* stream) {
    const nrc_status c = linear_check(x, out, B, in_f, out_f, lin_weight, bn_gamma, bn_beta,
                                      bn_running_mean, bn_running_var, bn_eps, bn_momentum,
                                      training, add_bias, divide_value, workspace);
    if (c != NRC_OK) return c;
    if (workspace_bytes < plan_linear(B, in_f, out_f).total) return NRC_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const nrc_status s = linear_pack_x(x, B, in_f, ws, st);
    if (s != NRC_OK) return s;
    // launched behind the x repack
    return linear_chain(lin_weight, out, B, in_f, out_f, lin_bias, bn_gamma, bn_beta,
                        bn_running_mean, bn_running_var, num_batches_tracked, bn_eps,
                        bn_momentum, training, add_bias, divide_value, ws, true, st);
}

// ---------------------------------------------------------------------------
// Host-buffer entry: the output features in chunks (each feature's batch
// statistics are independent of the others'), so the copy-in of the weight
// rows of chunk j+1, the chain of chunk j and the copy-out of chunk j-1 run at
// once.
// ---------------------------------------------------------------------------
namespace {

struct LinearHostLayout {
    size_t xdev, par, w[2], o[2], total;
};

LinearHostLayout linear_host_layout(int B, int in_f, int out_f, int chunk_f) {
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    LinearHostLayout h{};
    h.xdev = up(plan_linear(B, in_f, chunk_f).total);
    h.par = up(h.xdev + (size_t)B * in_f * 4);
    h.w[0] = up(h.par + ((size_t)3 * out_f + 4) * 4);
    h.w[1] = up(h.w[0] + (size_t)chunk_f * in_f * 4);
    h.o[0] = up(h.w[1] + (size_t)chunk_f * in_f * 4);
    h.o[1] = up(h.o[0] + (size_t)B * chunk_f * 4);
    h.total = h.o[1] + (size_t)B * chunk_f * 4;
    return h;
}

// Per device: the copy-in and copy-out streams and the events of the pipeline.
struct LinearHostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start, join, ev_in[2], ev_chain[2], ev_out[2];
    bool ready = false;
};
std::mutex g_lin_host_mu;
LinearHostPipe g_lin_host_pipe[64];

nrc_status linear_host_pipe(LinearHostPipe** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NRC_ERR_CUDA;
    LinearHostPipe& hp = g_lin_host_pipe[dev];
    if (!hp.ready) {
        const unsigned f = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.start, f) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.join, f) != cudaSuccess)
            return NRC_ERR_CUDA;
        for (int b = 0; b < 2; ++b)
            if (cudaEventCreateWithFlags(&hp.ev_in[b], f) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.ev_chain[b], f) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.ev_out[b], f) != cudaSuccess)
                return NRC_ERR_CUDA;
        hp.ready = true;
    }
    *out = &hp;
    return NRC_OK;
}

// chunk_f rounded to whole 128-feature tiles, at most out_f's tiles
int linear_chunk_tiles(int out_f, int chunk_f) {
    return std::max(1, std::min(ceil_div(out_f, kBM), ceil_div(chunk_f, kBM)));
}

}  // namespace

extern "C" size_t nrc_linear_bn_swish_host_workspace_size(int B, int in_f, int out_f,
                                                          int chunk_f) {
    if (B <= 0 || in_f <= 0 || out_f <= 0 || chunk_f <= 0) return 0;
    const int F = std::min(out_f, linear_chunk_tiles(out_f, chunk_f) * kBM);
    return linear_host_layout(B, in_f, out_f, F).total;
}

extern "C" nrc_status nrc_linear_bn_swish_host(
    const float* x_host, float* out_host, int B, int in_f, int out_f,
    const float* lin_weight_host, const float* lin_bias_host, const float* bn_gamma_host,
    const float* bn_beta_host, float* bn_running_mean, float* bn_running_var,
    int64_t* num_batches_tracked, float bn_eps, float bn_momentum, int training,
    const float* add_bias_host, float divide_value, int chunk_f, void* workspace,
    size_t workspace_bytes, void* stream) {
    const nrc_status c = linear_check(x_host, out_host, B, in_f, out_f, lin_weight_host,
                                      bn_gamma_host, bn_beta_host, bn_running_mean,
                                      bn_running_var, bn_eps, bn_momentum, training,
                                      add_bias_host, divide_value, workspace);
    if (c != NRC_OK) return c;
    if (chunk_f <= 0) return NRC_ERR_INVALID_ARG;
    const int tiles = ceil_div(out_f, kBM);
    const int chunk_t = linear_chunk_tiles(out_f, chunk_f);
    const int F = std::min(out_f, chunk_t * kBM);
    const LinearHostLayout hl = linear_host_layout(B, in_f, out_f, F);
    if (workspace_bytes < hl.total) return NRC_ERR_WORKSPACE;

    std::lock_guard<std::mutex> lk(g_lin_host_mu);   // the per-device pipe is shared
    LinearHostPipe* hp = nullptr;
    nrc_status s = linear_host_pipe(&hp);
    if (s != NRC_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    // x and the per-feature parameters: copied on the caller's stream; x packed
    // once for every chunk.
    float* xdev = reinterpret_cast<float*>(ws + hl.xdev);
    float* par = reinterpret_cast<float*>(ws + hl.par);
    float* d_bias = par;
    float* d_gamma = par + out_f;
    float* d_beta = par + 2 * (size_t)out_f;
    float* d_add = par + 3 * (size_t)out_f;
    const size_t fb = (size_t)out_f * 4;
    bool good = ok(cudaMemcpyAsync(xdev, x_host, (size_t)B * in_f * 4, cudaMemcpyHostToDevice,
                                   st)) &&
                ok(cudaMemcpyAsync(d_add, add_bias_host, 4, cudaMemcpyHostToDevice, st)) &&
                (!lin_bias_host ||
                 ok(cudaMemcpyAsync(d_bias, lin_bias_host, fb, cudaMemcpyHostToDevice, st))) &&
                (!bn_gamma_host ||
                 ok(cudaMemcpyAsync(d_gamma, bn_gamma_host, fb, cudaMemcpyHostToDevice, st))) &&
                (!bn_beta_host ||
                 ok(cudaMemcpyAsync(d_beta, bn_beta_host, fb, cudaMemcpyHostToDevice, st)));
    if (!good) return NRC_ERR_CUDA;
    s = linear_pack_x(xdev, B, in_f, ws, st);
    if (s != NRC_OK) return s;
    // The library streams start after everything already on the caller's stream
    // (the workspace may still be in use by an earlier call).
    if (!ok(cudaEventRecord(hp->start, st)) || !ok(cudaStreamWaitEvent(hp->in, hp->start, 0)) ||
        !ok(cudaStreamWaitEvent(hp->out, hp->start, 0)))
        return NRC_ERR_CUDA;
    const std::vector<int> sizes = host_chunk_sizes(tiles, chunk_t);
    const int n_chunks = (int)sizes.size();
    int t0 = 0;
    for (int j = 0; j < n_chunks; t0 += sizes[j], ++j) {
        const int b = j & 1;
        const int f0 = t0 * kBM;
        const int fc = std::min(out_f - f0, sizes[j] * kBM);     // features of the chunk
        float* wbuf = reinterpret_cast<float*>(ws + hl.w[b]);
        float* obuf = reinterpret_cast<float*>(ws + hl.o[b]);
        // copy-in of the chunk's weight rows: buffer b is free once chain j-2 ran
        if (j >= 2 && !ok(cudaStreamWaitEvent(hp->in, hp->ev_chain[b], 0))) return NRC_ERR_CUDA;
        if (!ok(cudaMemcpyAsync(wbuf, lin_weight_host + (size_t)f0 * in_f,
                                (size_t)fc * in_f * 4, cudaMemcpyHostToDevice, hp->in)) ||
            !ok(cudaEventRecord(hp->ev_in[b], hp->in)))
            return NRC_ERR_CUDA;
        // the chain: after its copy-in, and after chunk j-2's copy-out read buffer b
        if (!ok(cudaStreamWaitEvent(st, hp->ev_in[b], 0)) ||
            (j >= 2 && !ok(cudaStreamWaitEvent(st, hp->ev_out[b], 0))))
            return NRC_ERR_CUDA;
        s = linear_chain(wbuf, obuf, B, in_f, fc, lin_bias_host ? d_bias + f0 : nullptr,
                         bn_gamma_host ? d_gamma + f0 : nullptr,
                         bn_beta_host ? d_beta + f0 : nullptr, bn_running_mean + f0,
                         bn_running_var + f0, j == 0 ? num_batches_tracked : nullptr, bn_eps,
                         bn_momentum, training, d_add, divide_value, ws, false, st);
        if (s != NRC_OK) return s;
        if (!ok(cudaEventRecord(hp->ev_chain[b], st))) return NRC_ERR_CUDA;
        // copy-out of the chunk's columns into the (B, out_f) rows
        if (!ok(cudaStreamWaitEvent(hp->out, hp->ev_chain[b], 0)) ||
            !ok(cudaMemcpy2DAsync(out_host + f0, fb, obuf, (size_t)fc * 4, (size_t)fc * 4, B,
                                  cudaMemcpyDeviceToHost, hp->out)) ||
            !ok(cudaEventRecord(hp->ev_out[b], hp->out)))
            return NRC_ERR_CUDA;
    }
    // The caller's stream resumes once the last copy-out has landed.
    if (!ok(cudaEventRecord(hp->join, hp->out)) || !ok(cudaStreamWaitEvent(st, hp->join, 0)))
        return NRC_ERR_CUDA;
    return NRC_OK;
}
