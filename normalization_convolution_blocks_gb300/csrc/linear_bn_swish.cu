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
    LinearPlan pl = plan_linear(B, in_f, out_f);
    if (workspace_bytes < pl.total) return NRC_ERR_WORKSPACE;
    if ((long long)pl.n_jt * pl.n_bt >= (1LL << 30)) return NRC_ERR_UNSUPPORTED;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    LinearParams p{};
    p.W = lin_weight;
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
    p.vec_ok = (in_f % 4 == 0) && aligned(lin_weight, 16);
    // Staged A when W's rows are 16-byte aligned and the driver takes the map.
    bool staged = false;
    if (p.vec_ok) {
        const uint64_t dims[3] = {(uint64_t)in_f, (uint64_t)out_f, 1};
        const uint64_t strides[2] = {(uint64_t)in_f * 4, (uint64_t)in_f * 4 * out_f};
        const uint32_t box[3] = {32u, (uint32_t)kBM, 1u};
        if (encode_tensor_map_3d(&p.wmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, lin_weight, dims,
                                 strides, box, false, true)) {
            const LinearPlan ps = plan_linear(B, in_f, out_f, LinearProblem<true>::kBoxBytes);
            if (ps.g.b_stages >= 2 && ps.g.x_depth >= 2) {
                pl = ps;
                staged = true;
            }
        }
    }
    float* colp = reinterpret_cast<float*>(ws + pl.colp_off);

    const size_t units = (size_t)pl.n_bt * pl.g.num_kiters * pl.g.BN * 8;
    {
        TraceScope ts("pack_rows_split", st);
        pack_rows_split_kernel<<<elementwise_grid(units), 256, 0, st>>>(
            x, ws, B, in_f, pl.g.BN, pl.n_bt, pl.g.num_kiters);
    }
    if (cudaGetLastError() != cudaSuccess) return NRC_ERR_CUDA;
    pl.g.b_after_prev = true;          // launched behind the x repack
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
