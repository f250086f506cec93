// Pre-norm residual block with BatchNorm1d in training mode.
//
// Source: "Kimi-K2.6 l2_p12" (PopcornBench), the correctness discussion that
// sets batch statistics against running statistics.  In training mode channel
// c is normalized with the mean and the biased variance of x[:, c, :] over all
// N*L values.  The running buffers move toward the batch values with the
// unbiased variance ("Kimi-K2.6 l2_p97" states the same update for the
// BatchNorm1d after its Linear).
//
// Three steps on the caller's stream:
//   1. bn_row_stats_kernel: x is read once, in segments of 2 KB of a row; a
//      warp computes each segment's (mean, M2) in two passes over registers.
//   2. bn_train_finalize_kernel: one warp per channel merges its segments'
//      partials (division-free pairwise-merge form, fp32), writes the batch
//      mean and biased variance to the workspace and updates the running
//      buffers and num_batches_tracked.  It is launched behind step 1
//      (programmatic dependent launch) and waits for it at entry.
//   3. The eval-mode block (nrc_prenorm_dilconv_residual) with the batch mean
//      and variance in place of the running statistics.  Its first launch is an
//      ordinary one, so it starts after step 2 has finished.
//
// Every argument error returns before the first launch, so a rejected call
// leaves the running buffers untouched.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "nrc.h"
#include "nrc_host.h"
#include "nrc_launch.cuh"
#include "nrc_ptx.cuh"

namespace nrc {
namespace {

constexpr int kStatThreads = 256;

// 16-byte loads of x: kVW elements each, decoded to fp32 from the raw words.
template <typename T>
struct StatVec;
template <>
struct StatVec<float> {
    static constexpr int kVW = 4;
    __device__ static float get(const uint4& r, int i) {
        return __uint_as_float(i == 0 ? r.x : i == 1 ? r.y : i == 2 ? r.z : r.w);
    }
    __device__ static float one(const float* p) { return __ldcs(p); }
};
template <>
struct StatVec<__nv_bfloat16> {
    static constexpr int kVW = 8;
    __device__ static float get(const uint4& r, int i) {
        const uint32_t w = (i >> 1) == 0 ? r.x : (i >> 1) == 1 ? r.y : (i >> 1) == 2 ? r.z : r.w;
        return __uint_as_float((i & 1) ? (w & 0xffff0000u) : (w << 16));
    }
    __device__ static float one(const __nv_bfloat16* p) { return __bfloat162float(*p); }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Segments of 32*E elements (E per lane, E*sizeof(T) = 64 bytes) of each row
// (n, c) of the N samples at x (samples n0 .. n0 + N - 1 of a batch of N_all).
// Warp w of the grid takes segments w, w + G, w + 2G, ... (G = warps in the
// grid), so every SM streams the same share of x with no CTA-wide barrier.
// Per segment the warp computes its mean and M2 in two passes over registers
// (two warp sums) and lane 0 writes (mean, M2) to
// part[(c*N_all + n0 + n)*S + seg], S = segments per row; the last segment of
// a row may be short.  VEC: rows start 16-byte aligned and L is a multiple of the
// vector width, so whole 16-byte loads cover each segment (kept as raw words,
// 16 registers a lane); otherwise one element per load.  No CTA-wide barrier,
// and the fp32 vector path fits 32 registers, so 64 warps per SM keep their
// loads in flight (bf16 decodes two values per word and needs more).
template <typename T, bool VEC>
__global__ void __launch_bounds__(kStatThreads, (VEC && sizeof(T) == 4) ? 8 : 1)
    bn_row_stats_kernel(const T* __restrict__ x, float2* __restrict__ part, int N, int C, int L,
                        int S, int n_seg, int N_all, int n0) {
    griddep_launch_dependents();           // the finalize kernel may launch and wait
    constexpr int VW = StatVec<T>::kVW;
    constexpr int E = 4 * VW;              // four 16-byte loads per lane
    constexpr int W = 32 * E;              // elements per segment
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (kStatThreads / 32);
    const int first = blockIdx.x * (kStatThreads / 32) + (threadIdx.x >> 5);
    auto seg_len = [&](int item) { return min(W, L - (item % S) * W); };
    auto finish = [&](int item, float m, float q) {
        q = warp_sum(q);
        if (lane == 0) {
            const int row = item / S, seg = item - row * S;
            const int n = row / C, c = row - n * C;
            part[((size_t)c * N_all + n0 + n) * S + seg] = make_float2(m, q);
        }
    };
    if constexpr (VEC) {
        for (int item = first; item < n_seg; item += warps) {
            const int here = seg_len(item);
            const T* xs = x + (size_t)(item / S) * L + (size_t)(item % S) * W;
            uint4 r[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int e = (j * 32 + lane) * VW;
                r[j] = e < here ? __ldcs(reinterpret_cast<const uint4*>(xs + e))
                                : make_uint4(0u, 0u, 0u, 0u);      // reads as 0.0
            }
            float s = 0.f, q = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int i = 0; i < VW; ++i) s += StatVec<T>::get(r[j], i);
            const float m = warp_sum(s) / (float)here;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool ok = (j * 32 + lane) * VW < here;
#pragma unroll
                for (int i = 0; i < VW; ++i) {
                    const float d = ok ? StatVec<T>::get(r[j], i) - m : 0.f;
                    q = fmaf(d, d, q);
                }
            }
            finish(item, m, q);
        }
    } else {
        for (int item = first; item < n_seg; item += warps) {
            const int here = seg_len(item);
            const T* xs = x + (size_t)(item / S) * L + (size_t)(item % S) * W;
            float v[E];
#pragma unroll
            for (int j = 0; j < E; ++j) {
                const int e = j * 32 + lane;
                v[j] = e < here ? StatVec<T>::one(xs + e) : 0.f;
            }
            float s = 0.f, q = 0.f;
#pragma unroll
            for (int j = 0; j < E; ++j) s += v[j];
            const float m = warp_sum(s) / (float)here;
#pragma unroll
            for (int j = 0; j < E; ++j) {
                const float d = j * 32 + lane < here ? v[j] - m : 0.f;
                q = fmaf(d, d, q);
            }
            finish(item, m, q);
        }
    }
}

// Resident CTAs per SM of a statistics kernel (queried once): the grid is one
// full wave, so no CTA starts late and streams alone at the end.
template <typename T, bool VEC>
int stats_ctas_per_sm() {
    static const int n = [] {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, bn_row_stats_kernel<T, VEC>,
                                                          kStatThreads, 0) != cudaSuccess ||
            b < 1)
            b = 1;
        return b;
    }();
    return n;
}

// One warp per channel merges its N*S segment partials: with k_i values in
// segment i (W, or the row's remainder for the last one),
//   mean = sum_i k_i mean_i / (N L),   M2 = sum_i (M2_i + k_i (mean_i - mean)^2).
__global__ void __launch_bounds__(256)
    bn_train_finalize_kernel(const float2* __restrict__ part, int N, int C, int L, int S, int W,
                             float* __restrict__ batch_mean, float* __restrict__ batch_var,
                             float* running_mean, float* running_var,
                             long long* num_batches_tracked, float momentum) {
    griddep_wait();                        // the segment statistics are complete
    const int c = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (c == 0 && lane == 0 && num_batches_tracked) *num_batches_tracked += 1;
    if (c >= C) return;
    const float2* pc = part + (size_t)c * N * S;
    const int total = N * S;
    const float last = (float)(L - (S - 1) * W);   // values in a row's last segment
    float s = 0.f;
    for (int i = lane; i < total; i += 32) {
        const float k = (i % S == S - 1) ? last : (float)W;
        s = fmaf(k, pc[i].x, s);
    }
    const float cnt = (float)N * (float)L;
    const float mean = warp_sum(s) / cnt;
    float q = 0.f;
    for (int i = lane; i < total; i += 32) {
        const float k = (i % S == S - 1) ? last : (float)W;
        const float2 p = pc[i];
        const float d = p.x - mean;
        q += p.y + k * d * d;
    }
    q = warp_sum(q);
    if (lane != 0) return;
    const float var = q / cnt;             // biased: normalizes the batch
    batch_mean[c] = mean;
    batch_var[c] = var;
    if (running_mean) running_mean[c] = (1.f - momentum) * running_mean[c] + momentum * mean;
    if (running_var)
        running_var[c] = (1.f - momentum) * running_var[c] + momentum * (q / (cnt - 1.f));
}

// Segment length of the statistics kernel, in elements.
inline int stat_segment(nrc_dtype dt) { return 32 * 4 * (dt == NRC_F32 ? 4 : 8); }

inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct TrainLayout {
    size_t part, mean, var, total;
};

TrainLayout train_layout(int N, int C, int L, nrc_dtype dt) {
    TrainLayout t{};
    const size_t base = nrc_prenorm_dilconv_residual_workspace_size(C, dt);
    if (base == 0 || N <= 0 || L <= 0) return t;
    const size_t S = (size_t)ceil_div(L, stat_segment(dt));
    t.part = align256(base);
    t.mean = align256(t.part + (size_t)N * C * S * sizeof(float2));
    t.var = align256(t.mean + (size_t)C * sizeof(float));
    t.total = t.var + (size_t)C * sizeof(float);
    return t;
}


// Launches the statistics kernel over the rows of N samples at x (samples n0 ..
// of a batch of N_all; the partials go to their place in the whole batch's
// array).  One wave of resident CTAs striding over the segments.
nrc_status launch_row_stats(const void* x, float2* part, nrc_dtype dt, int N, int C, int L,
                            int N_all, int n0, int vec, cudaStream_t st) {
    const int W = stat_segment(dt);
    const int S = ceil_div(L, W);
    const long long n_seg = (long long)N * C * S;
    TraceScope ts("bn_row_stats", st);
    const int per_sm = dt == NRC_F32 ? (vec ? stats_ctas_per_sm<float, true>()
                                            : stats_ctas_per_sm<float, false>())
                                     : (vec ? stats_ctas_per_sm<__nv_bfloat16, true>()
                                            : stats_ctas_per_sm<__nv_bfloat16, false>());
    const long long want = (n_seg + kStatThreads / 32 - 1) / (kStatThreads / 32);
    const unsigned grid = (unsigned)std::max<long long>(
        1, std::min<long long>(want, (long long)device_sm_count() * per_sm));
    const float* xf = static_cast<const float*>(x);
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    if (dt == NRC_F32 && vec)
        bn_row_stats_kernel<float, true><<<grid, kStatThreads, 0, st>>>(xf, part, N, C, L, S,
                                                                         (int)n_seg, N_all, n0);
    else if (dt == NRC_F32)
        bn_row_stats_kernel<float, false><<<grid, kStatThreads, 0, st>>>(xf, part, N, C, L, S,
                                                                          (int)n_seg, N_all, n0);
    else if (vec)
        bn_row_stats_kernel<__nv_bfloat16, true><<<grid, kStatThreads, 0, st>>>(
            xb, part, N, C, L, S, (int)n_seg, N_all, n0);
    else
        bn_row_stats_kernel<__nv_bfloat16, false><<<grid, kStatThreads, 0, st>>>(
            xb, part, N, C, L, S, (int)n_seg, N_all, n0);
    return cuda_status(cudaGetLastError());
}
}  // namespace
}  // namespace nrc

using namespace nrc;

extern "C" size_t nrc_prenorm_dilconv_residual_train_workspace_size(int N, int C, int L,
                                                                   nrc_dtype dt) {
    return train_layout(N, C, L, dt).total;
}

namespace {

// The eval-mode entry's checks, made before anything is launched (shared by
// the device and host-buffer entries).
nrc_status train_check(const void* x, const void* out, nrc_dtype dt, int N, int C, int L,
                       int kernel_size, int dilation, int padding, const float* gamma,
                       const float* beta, float bn_eps, float bn_momentum,
                       const void* conv_weight, const void* workspace) {
    if (dt != NRC_F32 && dt != NRC_BF16) return NRC_ERR_INVALID_ARG;
    if (!x || !out || !gamma || !beta || !conv_weight || !workspace) return NRC_ERR_INVALID_ARG;
    if (N <= 0 || C <= 0 || L <= 0 || dilation <= 0 || padding < 0) return NRC_ERR_INVALID_ARG;
    if (!(bn_eps >= 0.f) || !std::isfinite(bn_eps)) return NRC_ERR_INVALID_ARG;
    if (!std::isfinite(bn_momentum)) return NRC_ERR_INVALID_ARG;
    if ((long long)N * L < 2) return NRC_ERR_INVALID_ARG;     // unbiased variance: N*L - 1
    if (kernel_size != 3 || padding != dilation) return NRC_ERR_UNSUPPORTED;
    if (C > 2048) return NRC_ERR_UNSUPPORTED;
    const size_t esz = dt == NRC_F32 ? 4 : 2;
    const size_t bytes = (size_t)N * C * L * esz;
    if (ranges_overlap(x, bytes, out, bytes)) return NRC_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return NRC_ERR_ALIGNMENT;
    // 32-bit segment indices with room for one grid stride (x would be ~4 TB)
    const long long n_seg = (long long)N * C * ceil_div(L, stat_segment(dt));
    if (n_seg >= (1LL << 31) - (1LL << 24)) return NRC_ERR_UNSUPPORTED;
    return NRC_OK;
}

}  // namespace

extern "C" nrc_status nrc_prenorm_dilconv_residual_train(
    const void* x, void* out, nrc_dtype dt, int N, int C, int L, int kernel_size, int dilation,
    int padding, float* running_mean, float* running_var, long long* num_batches_tracked,
    const float* gamma, const float* beta, float bn_eps, float bn_momentum,
    const void* conv_weight, const void* conv_bias, void* workspace, size_t workspace_bytes,
    void* stream) {
    const nrc_status chk = train_check(x, out, dt, N, C, L, kernel_size, dilation, padding,
                                       gamma, beta, bn_eps, bn_momentum, conv_weight, workspace);
    if (chk != NRC_OK) return chk;
    const TrainLayout lay = train_layout(N, C, L, dt);
    if (workspace_bytes < lay.total) return NRC_ERR_WORKSPACE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float2* part = reinterpret_cast<float2*>(ws + lay.part);
    float* bmean = reinterpret_cast<float*>(ws + lay.mean);
    float* bvar = reinterpret_cast<float*>(ws + lay.var);
    const int vw = dt == NRC_F32 ? 4 : 8;
    const int vec = (L % vw == 0 && aligned(x, 16)) ? 1 : 0;
    const int W = stat_segment(dt);
    const int S = ceil_div(L, W);
    if (launch_row_stats(x, part, dt, N, C, L, N, 0, vec, st) != NRC_OK) return NRC_ERR_CUDA;
    {
        TraceScope ts("bn_train_finalize", st);
        if (launch_after_prev(bn_train_finalize_kernel, dim3((unsigned)ceil_div(C, 8)), dim3(256),
                              st, (const float2*)part, N, C, L, S, W, bmean, bvar,
                              running_mean, running_var, num_batches_tracked,
                              bn_momentum) != cudaSuccess)
            return NRC_ERR_CUDA;
    }
    return nrc_prenorm_dilconv_residual(x, out, dt, N, C, L, kernel_size, dilation, padding,
                                        bmean, bvar, gamma, beta, bn_eps, conv_weight, conv_bias,
                                        ws, lay.part, stream);
}

// ---------------------------------------------------------------------------
// Host-buffer entry.  The batch statistics need every sample before the first
// value is normalized, so the pipeline has two phases over the same chunks of
// samples: x comes in chunk by chunk (into one device copy of the whole batch)
// with each chunk's statistics computed behind its copy; after the merge, the
// GEMM of chunk j runs while chunk j-1's output is copied out.
// ---------------------------------------------------------------------------
namespace {

struct TrainHostLayout {
    size_t xdev, o[2], par, w, b, total;
};

TrainHostLayout train_host_layout(int N, int C, int L, nrc_dtype dt, int chunk_n) {
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    const size_t es = dt == NRC_F32 ? 4 : 2;
    const size_t chunk = (size_t)chunk_n * C * L * es;
    TrainHostLayout h{};
    h.xdev = up(train_layout(N, C, L, dt).total);
    h.o[0] = up(h.xdev + (size_t)N * C * L * es);
    h.o[1] = up(h.o[0] + chunk);
    h.par = up(h.o[1] + chunk);
    h.w = up(h.par + (size_t)2 * C * sizeof(float));
    h.b = up(h.w + (size_t)C * C * 3 * es);
    h.total = h.b + (size_t)C * es;
    return h;
}

// Per device: the copy-in and copy-out streams and the events of the pipeline.
struct TrainHostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start, join, ev_in[2], ev_gemm[2], ev_out[2];
    bool ready = false;
};
std::mutex g_train_host_mu;
TrainHostPipe g_train_host_pipe[64];

nrc_status train_host_pipe(TrainHostPipe** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NRC_ERR_CUDA;
    TrainHostPipe& hp = g_train_host_pipe[dev];
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

extern "C" size_t nrc_prenorm_dilconv_residual_train_host_workspace_size(int N, int C, int L,
                                                                        nrc_dtype dt,
                                                                        int chunk_n) {
    if (N <= 0 || C <= 0 || L <= 0 || chunk_n <= 0 || (dt != NRC_F32 && dt != NRC_BF16))
        return 0;
    if (train_layout(N, C, L, dt).total == 0) return 0;
    return train_host_layout(N, C, L, dt, std::min(chunk_n, N)).total;
}

extern "C" nrc_status nrc_prenorm_dilconv_residual_train_host(
    const void* x_host, void* out_host, nrc_dtype dt, int N, int C, int L, int kernel_size,
    int dilation, int padding, float* running_mean, float* running_var,
    long long* num_batches_tracked, const float* gamma_host, const float* beta_host,
    float bn_eps, float bn_momentum, const void* conv_weight_host, const void* conv_bias_host,
    int chunk_n, void* workspace, size_t workspace_bytes, void* stream) {
    const nrc_status chk = train_check(x_host, out_host, dt, N, C, L, kernel_size, dilation,
                                       padding, gamma_host, beta_host, bn_eps, bn_momentum,
                                       conv_weight_host, workspace);
    if (chk != NRC_OK) return chk;
    if (chunk_n <= 0) return NRC_ERR_INVALID_ARG;
    chunk_n = std::min(chunk_n, N);
    const TrainLayout lay = train_layout(N, C, L, dt);
    const TrainHostLayout hl = train_host_layout(N, C, L, dt, chunk_n);
    if (workspace_bytes < hl.total) return NRC_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return NRC_ERR_ALIGNMENT;

    std::lock_guard<std::mutex> lk(g_train_host_mu);   // the per-device pipe is shared
    TrainHostPipe* hp = nullptr;
    nrc_status s = train_host_pipe(&hp);
    if (s != NRC_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    const size_t es = dt == NRC_F32 ? 4 : 2;
    const size_t sample = (size_t)C * L * es;
    float* d_gamma = reinterpret_cast<float*>(ws + hl.par);
    float* d_beta = d_gamma + C;
    // Parameters and weights: copied once on the caller's stream.
    const bool good =
        ok(cudaMemcpyAsync(d_gamma, gamma_host, (size_t)C * 4, cudaMemcpyHostToDevice, st)) &&
        ok(cudaMemcpyAsync(d_beta, beta_host, (size_t)C * 4, cudaMemcpyHostToDevice, st)) &&
        ok(cudaMemcpyAsync(ws + hl.w, conv_weight_host, (size_t)C * C * 3 * es,
                           cudaMemcpyHostToDevice, st)) &&
        (!conv_bias_host ||
         ok(cudaMemcpyAsync(ws + hl.b, conv_bias_host, (size_t)C * es, cudaMemcpyHostToDevice,
                            st)));
    if (!good) return NRC_ERR_CUDA;
    if (!ok(cudaEventRecord(hp->start, st)) || !ok(cudaStreamWaitEvent(hp->in, hp->start, 0)) ||
        !ok(cudaStreamWaitEvent(hp->out, hp->start, 0)))
        return NRC_ERR_CUDA;
    uint8_t* xdev = ws + hl.xdev;
    float2* part = reinterpret_cast<float2*>(ws + lay.part);
    float* bmean = reinterpret_cast<float*>(ws + lay.mean);
    float* bvar = reinterpret_cast<float*>(ws + lay.var);
    const int vw = dt == NRC_F32 ? 4 : 8;
    const int vec = (L % vw == 0) ? 1 : 0;             // xdev and every chunk 16-byte aligned
    const std::vector<int> sizes = host_chunk_sizes(N, chunk_n);
    const int n_chunks = (int)sizes.size();
    // Phase 1: copy-in, and each chunk's row statistics behind its copy.
    int n0 = 0;
    for (int j = 0; j < n_chunks; n0 += sizes[j], ++j) {
        const int b = j & 1;
        if (!ok(cudaMemcpyAsync(xdev + (size_t)n0 * sample,
                                static_cast<const uint8_t*>(x_host) + (size_t)n0 * sample,
                                (size_t)sizes[j] * sample, cudaMemcpyHostToDevice, hp->in)) ||
            !ok(cudaEventRecord(hp->ev_in[b], hp->in)) ||
            !ok(cudaStreamWaitEvent(st, hp->ev_in[b], 0)))
            return NRC_ERR_CUDA;
        if (launch_row_stats(xdev + (size_t)n0 * sample, part, dt, sizes[j], C, L, N, n0, vec,
                             st) != NRC_OK)
            return NRC_ERR_CUDA;
    }
    {
        const int W = stat_segment(dt);
        TraceScope ts("bn_train_finalize", st);
        if (launch_after_prev(bn_train_finalize_kernel, dim3((unsigned)ceil_div(C, 8)), dim3(256),
                              st, (const float2*)part, N, C, L, ceil_div(L, W), W, bmean, bvar,
                              running_mean, running_var, num_batches_tracked,
                              bn_momentum) != cudaSuccess)
            return NRC_ERR_CUDA;
    }
    // Phase 2: the block on each chunk with the batch statistics, its output
    // copied out behind it.
    n0 = 0;
    for (int j = 0; j < n_chunks; n0 += sizes[j], ++j) {
        const int b = j & 1;
        const size_t bytes = (size_t)sizes[j] * sample;
        if (j >= 2 && !ok(cudaStreamWaitEvent(st, hp->ev_out[b], 0))) return NRC_ERR_CUDA;
        s = nrc_prenorm_dilconv_residual(xdev + (size_t)n0 * sample, ws + hl.o[b], dt, sizes[j],
                                         C, L, kernel_size, dilation, padding, bmean, bvar,
                                         d_gamma, d_beta, bn_eps, ws + hl.w,
                                         conv_bias_host ? ws + hl.b : nullptr, ws, lay.part,
                                         stream);
        if (s != NRC_OK) return s;
        if (!ok(cudaEventRecord(hp->ev_gemm[b], st)) ||
            !ok(cudaStreamWaitEvent(hp->out, hp->ev_gemm[b], 0)) ||
            !ok(cudaMemcpyAsync(static_cast<uint8_t*>(out_host) + (size_t)n0 * sample,
                                ws + hl.o[b], bytes, cudaMemcpyDeviceToHost, hp->out)) ||
            !ok(cudaEventRecord(hp->ev_out[b], hp->out)))
            return NRC_ERR_CUDA;
    }
    // The caller's stream resumes once the last copy-out has landed.
    if (!ok(cudaEventRecord(hp->join, hp->out)) || !ok(cudaStreamWaitEvent(st, hp->join, 0)))
        return NRC_ERR_CUDA;
    return NRC_OK;
}
