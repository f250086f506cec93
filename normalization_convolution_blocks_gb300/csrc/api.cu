// Library-wide pieces of libnrc.so: the device status word, status queries,
// the wait-limit setting and the fault-path self test.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "nrc_host.h"
#include "nrc_ptx.cuh"

namespace nrc {

// Device status word: [0] = first error code recorded, [1] = where (wait site).
__device__ int g_status_word[2];

namespace {
constexpr int kMaxDevices = 64;
int* g_status_addr[kMaxDevices];
int g_sm_count[kMaxDevices];
int g_coop[kMaxDevices];         // 0 unknown, 1 supported, 2 not
std::mutex g_mu;
std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
// Limit of the one-wave GroupNorm kernel's grid-wide barrier only; 0: the
// general limit.
std::atomic<unsigned long long> g_grid_barrier_timeout_ns{0ull};
int g_last_site = 0;

int current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
    return d;
}
}  // namespace

int* device_status_ptr() {
    const int d = current_device();
    if (d < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_addr[d]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_addr[d] = static_cast<int*>(p);
    }
    return g_status_addr[d];
}

unsigned long long wait_timeout_ns() { return g_timeout_ns.load(); }

unsigned long long grid_barrier_timeout_ns() {
    const unsigned long long v = g_grid_barrier_timeout_ns.load();
    return v ? v : g_timeout_ns.load();
}

int device_sm_count() {
    const int d = current_device();
    if (d < 0) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[d]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
        g_sm_count[d] = n > 0 ? n : 1;
    }
    return g_sm_count[d];
}

bool device_coop_launch() {
    const int d = current_device();
    if (d < 0) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_coop[d]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrCooperativeLaunch, d);
        g_coop[d] = v ? 1 : 2;
    }
    return g_coop[d] == 1;
}

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}
}  // namespace

bool encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                          const uint64_t dims[3], const uint64_t strides[2],
                          const uint32_t box[3], bool nan_fill, bool swizzle128) {
    const EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t gdim[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t gstride[2] = {strides[0], strides[1]};
    const cuuint32_t bdim[3] = {box[0], box[1], box[2]};
    const cuuint32_t estride[3] = {1, 1, 1};
    return fn(map, dtype, 3, const_cast<void*>(base), gdim, gstride, bdim, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              nan_fill ? CU_TENSOR_MAP_FLOAT_OOB_FILL_NAN_REQUEST_ZERO_FMA
                       : CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
struct TraceRec {
    const char* name;
    cudaEvent_t start, stop;
};
std::mutex g_trace_mu;
std::atomic<bool> g_trace_on{false};
std::vector<TraceRec> g_trace;          // completed and open records
std::vector<cudaEvent_t> g_event_pool;  // recycled events

cudaEvent_t take_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}
}  // namespace

bool trace_enabled() { return g_trace_on.load(std::memory_order_relaxed); }

void trace_record(const char* name, cudaStream_t s, bool begin) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (begin) {
        TraceRec r{name, take_event(), nullptr};
        cudaEventRecord(r.start, s);
        g_trace.push_back(r);
    } else {
        // close the most recent open record of this name
        for (auto it = g_trace.rbegin(); it != g_trace.rend(); ++it) {
            if (it->name == name && it->stop == nullptr) {
                it->stop = take_event();
                cudaEventRecord(it->stop, s);
                break;
            }
        }
    }
}

// One thread waits, with a bounded limit, on an mbarrier that nothing arrives
// at; the give-up path records the timeout like a stalled pipeline would.
__global__ void selftest_wait_timeout_kernel(int* status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
        WaitCtx ctx{&abort_flag, status, limit_ns};
        mbar_wait(smem_u32(&bar), 0, ctx, 99);
    }
}

}  // namespace nrc

using namespace nrc;

extern "C" const char* nrc_status_string(nrc_status s) {
    switch (s) {
        case NRC_OK: return "NRC_OK";
        case NRC_ERR_INVALID_ARG: return "NRC_ERR_INVALID_ARG";
        case NRC_ERR_UNSUPPORTED: return "NRC_ERR_UNSUPPORTED";
        case NRC_ERR_ALIGNMENT: return "NRC_ERR_ALIGNMENT";
        case NRC_ERR_WORKSPACE: return "NRC_ERR_WORKSPACE";
        case NRC_ERR_CUDA: return "NRC_ERR_CUDA";
        case NRC_ERR_TIMEOUT: return "NRC_ERR_TIMEOUT";
    }
    return "NRC_ERR_UNKNOWN";
}

extern "C" int nrc_version(void) { return 100; }

extern "C" void nrc_set_wait_timeout_ns(uint64_t ns) {
    g_timeout_ns.store(ns > 0 ? (unsigned long long)ns : 1ull);
}

extern "C" void nrc_set_grid_barrier_timeout_ns(uint64_t ns) {
    g_grid_barrier_timeout_ns.store((unsigned long long)ns);
}

extern "C" int nrc_last_error_site(void) { return g_last_site; }

extern "C" nrc_status nrc_query_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return NRC_ERR_CUDA;
    int word[2] = {0, 0};
    if (cudaMemcpyFromSymbol(word, g_status_word, sizeof(word)) != cudaSuccess)
        return NRC_ERR_CUDA;
    if (word[0] != 0) {
        g_last_site = word[1];
        const int zero[2] = {0, 0};
        if (cudaMemcpyToSymbol(g_status_word, zero, sizeof(zero)) != cudaSuccess)
            return NRC_ERR_CUDA;
    }
    return word[0] == 0 ? NRC_OK : static_cast<nrc_status>(word[0]);
}

extern "C" nrc_status nrc_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
    int* status = device_status_ptr();
    if (!status) return NRC_ERR_CUDA;
    selftest_wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        status, (unsigned long long)limit_ns);
    return cuda_status(cudaGetLastError());
}

extern "C" void nrc_trace_enable(int on) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (on) {
        for (auto& r : g_trace) {
            if (r.start) g_event_pool.push_back(r.start);
            if (r.stop) g_event_pool.push_back(r.stop);
        }
        g_trace.clear();
    }
    g_trace_on.store(on != 0);
}

extern "C" int nrc_trace_count(void) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    return (int)g_trace.size();
}

extern "C" nrc_status nrc_trace_get(int i, const char** name, float* ms) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (i < 0 || i >= (int)g_trace.size() || !name || !ms) return NRC_ERR_INVALID_ARG;
    const TraceRec& r = g_trace[(size_t)i];
    *name = r.name;
    *ms = 0.f;
    if (!r.stop) return NRC_ERR_INVALID_ARG;
    if (cudaEventSynchronize(r.stop) != cudaSuccess) return NRC_ERR_CUDA;
    return cuda_status(cudaEventElapsedTime(ms, r.start, r.stop));
}
