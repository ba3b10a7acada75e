// Streaming-read probe: the time a plain read of N bytes of HBM takes when it is launched the way the
// decode kernels are timed (one launch between two CUDA events on the caller's stream).  It does none
// of the layer's arithmetic; benchmarks use it as the floor against which a weight-streaming kernel of
// the same byte count is judged.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>

#include "moe.h"
#include "moe_internal.h"

namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Grid-stride read of n16 16-byte words, eight loads in flight per thread.  The xor of everything read
// is stored only if it equals a constant, so the loads cannot be dropped and nothing is normally written.
__global__ void __launch_bounds__(512) stream_read_kernel(const uint4 *src, size_t n16, uint32_t *sink) {
    constexpr int kIn = 8;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (; i + (kIn - 1) * stride < n16; i += kIn * stride) {
        uint4 v[kIn];
#pragma unroll
        for (int j = 0; j < kIn; ++j) v[j] = ld_stream(src + i + j * stride);
#pragma unroll
        for (int j = 0; j < kIn; ++j) acc ^= v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = ld_stream(src + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    if (acc == 0x9E3779B9u) *sink = acc;
}

int probe_fail(int code, const char *fmt, ...) {
    char buf[256];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    moe::set_last_error(buf);
    return code;
}

}  // namespace

namespace moe {

cudaError_t ensure_dyn_smem(const void *func, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, size_t> raised;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    size_t &have = raised[{dev, func}];
    if (bytes > have) {
        e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (e != cudaSuccess) return e;
        have = bytes;
    }
    return cudaSuccess;
}

}  // namespace moe

extern "C" int moe_debug_stream_read(const void *src_dev, size_t bytes, void *sink_dev, int32_t nblocks,
                                     void *stream) {
    if (!src_dev || !sink_dev) return probe_fail(MOE_EINVAL, "src_dev and sink_dev are required");
    if (reinterpret_cast<uintptr_t>(src_dev) % 16 || bytes % 16 || reinterpret_cast<uintptr_t>(sink_dev) % 4)
        return probe_fail(MOE_EINVAL, "src_dev and bytes must be 16-byte multiples, sink_dev 4-byte aligned");
    if (nblocks < 0) return probe_fail(MOE_EINVAL, "nblocks must be >= 0");
    if (nblocks == 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                      cudaSuccess)
            return probe_fail(MOE_ECUDA, "cannot read the device's SM count");
        nblocks = 4 * sms;  // four 512-thread blocks fill an SM's 2048 threads
    }
    if (bytes == 0) return MOE_OK;
    stream_read_kernel<<<nblocks, 512, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(src_dev), bytes / 16, static_cast<uint32_t *>(sink_dev));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return probe_fail(MOE_ECUDA, "stream_read_kernel: %s", cudaGetErrorString(e));
    return MOE_OK;
}
