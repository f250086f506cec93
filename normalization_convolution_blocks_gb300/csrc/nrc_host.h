// Host-side helpers shared by the translation units of libnrc.so.
#pragma once
#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "nrc.h"

namespace nrc {

// Device address of the status word (two ints) for the current device.
int* device_status_ptr();
// Current limit of every device-side wait (ns).
unsigned long long wait_timeout_ns();
// Current limit of the one-wave GroupNorm kernel's grid-wide barrier (ns): its
// own setting if one was made, else wait_timeout_ns().
unsigned long long grid_barrier_timeout_ns();
// Number of SMs of the current device (cached per device).
int device_sm_count();
// Whether the current device supports cooperative launches (cached per device).
bool device_coop_launch();

// Encodes a 3-D tiled tensor map (dims and box innermost first, strides in
// bytes of dims 1 and 2) through the driver's cuTensorMapEncodeTiled, reached
// via the runtime's entry-point query so the library does not link libcuda.
// nan_fill: out-of-bounds elements read as NaN instead of zero; swizzle128: the
// box lands in shared memory in the 128-byte swizzle (16-byte chunk c of 128-byte
// row r at chunk c ^ (r mod 8); box rows of exactly 128 bytes, destination
// 1024-byte aligned).  Returns false when the driver rejects the map or the
// entry point is unavailable.
bool encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                          const uint64_t dims[3], const uint64_t strides[2],
                          const uint32_t box[3], bool nan_fill, bool swizzle128 = false);

inline bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

inline bool aligned(const void* p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

inline nrc_status cuda_status(cudaError_t e) { return e == cudaSuccess ? NRC_OK : NRC_ERR_CUDA; }

// Chunk sizes of the host-buffer pipelines (in units: samples, or 128-feature
// tiles): ramp-up chunk_n/4, chunk_n/2, then chunk_n, then ramp-down
// chunk_n/2, chunk_n/4 (each at least 1; the last middle chunk shorter if N
// asks), so the first copy-in and the last copy-out, which overlap nothing,
// stay short.  chunk_n <= N.
inline std::vector<int> host_chunk_sizes(int N, int chunk_n) {
    const int r1 = std::max(1, chunk_n / 4), r2 = std::max(1, chunk_n / 2);
    std::vector<int> sizes;
    int rem = N;
    auto push = [&](int t) {
        if (t > 0) {
            sizes.push_back(t);
            rem -= t;
        }
    };
    push(std::min(r1, rem));
    push(std::min(r2, rem));
    const int tail = std::min(rem, r1 + r2);
    while (rem > tail) push(std::min(chunk_n, rem - tail));
    if (tail > r1) {
        push(tail - r1);
        push(r1);
    } else {
        push(tail);
    }
    return sizes;
}


// Launch trace: when enabled (nrc_trace_enable), every kernel launch of the
// library is bracketed by a pair of CUDA events recorded on its stream, so a
// caller can read per-kernel device durations afterwards (nrc_trace_get).
bool trace_enabled();
void trace_record(const char* name, cudaStream_t s, bool begin);

struct TraceScope {
    const char* name;
    cudaStream_t stream;
    bool on;
    TraceScope(const char* n, cudaStream_t s) : name(n), stream(s), on(trace_enabled()) {
        if (on) trace_record(name, stream, true);
    }
    ~TraceScope() {
        if (on) trace_record(name, stream, false);
    }
};

}  // namespace nrc
