// Probes for benchmarks; neither does any of the layer's arithmetic.
//  * Streaming read: the time a plain read of N bytes of HBM takes when it is launched the way the decode
//    kernels are timed (one launch between two CUDA events on the caller's stream), the floor against
//    which a weight-streaming kernel of the same byte count is judged.
//  * Block-scaled MMA stream: the rate at which every SM retires the prefill GEMMs' MMA shape (M = 128,
//    N = 256, K = 32, E4M3 x E2M1 with UE8M0 scales) from operands already in shared memory, the ceiling
//    of those GEMMs with no operand traffic at all.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>

#include "moe.h"
#include "moe_internal.h"
#include "moe_tc.cuh"

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

// One CTA per SM.  The tiles hold bytes of a fixed hash (E4M3 codes without the NaN pattern, E2M1 codes in
// their one-byte-per-element shared-memory form), every scale 2^0.  Thread 0 issues iters x 4 MMAs into one
// 256-column accumulator, then one commit; the CTA waits for it (bounded) and frees tensor memory.
constexpr int kPkTileA = 128 * 128, kPkTileB = 256 * 128, kPkAtom = 512;
constexpr int kPkUsed = 1024 + kPkTileA + kPkTileB + 3 * kPkAtom;
// Launched with more shared memory than it uses, so that no SM takes two CTAs (each holds all 512 tensor-memory
// columns; a second one on the same SM would wait for the first and halve the measured rate).
constexpr int kPkSmem = 120 * 1024;
static_assert(kPkUsed <= kPkSmem, "probe shared memory");

__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, int *err) {
    using namespace moe::tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    __shared__ __align__(8) uint64_t done;
    __shared__ uint32_t tslot;
    uint8_t *sA = smem, *sB = smem + kPkTileA, *sAt = smem + kPkTileA + kPkTileB;
    for (int i = threadIdx.x; i < (kPkTileA + kPkTileB) / 4; i += blockDim.x) {
        uint32_t h = (uint32_t)i * 0x9E3779B1u;
        h ^= h >> 15;
        reinterpret_cast<uint32_t *>(smem)[i] = (h * 0x85EBCA77u) & 0x77777777u;
    }
    for (int i = threadIdx.x; i < 3 * kPkAtom / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(sAt)[i] = 0x7F7F7F7Fu;
    if (threadIdx.x < 32) tmem_alloc(&tslot, 512);
    if (threadIdx.x == 0) {
        mbar_init(&done, 1);
        fence_barrier_init();
    }
    fence_proxy_async();  // the tiles and atoms were written through the generic proxy
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tslot, sfa = tbase + 256, sfb = sfa + 4;
    if (threadIdx.x == 0) {
        atom_to_tmem(sfa, sAt);
        atom_to_tmem(sfb, sAt + kPkAtom);
        atom_to_tmem(sfb + 4, sAt + 2 * kPkAtom);
        const uint32_t idesc = mx_idesc(kFmtE4M3, kFmtE2M1, 256);
        const uint32_t aA = smem_u32(sA), aB = smem_u32(sB);
        for (int it = 0; it < iters; ++it)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_mx(tbase, sw128_desc(aA + kk * 32), sw128_desc(aB + kk * 32), idesc, kk, sfa, sfb,
                       (it | kk) ? 1u : 0u);
        mma_commit(&done);
        mbar_wait(&done, 0, err, 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x < 32) tmem_dealloc(tbase, 512);
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

extern "C" int moe_debug_mma_peak(int32_t iters, int32_t nblocks, void *err_dev, void *stream) {
    if (!err_dev || reinterpret_cast<uintptr_t>(err_dev) % 4) return probe_fail(MOE_EINVAL, "err_dev must be 4-byte aligned");
    if (iters < 1 || iters > 65536) return probe_fail(MOE_EINVAL, "iters must be in 1..65536");
    if (nblocks < 0) return probe_fail(MOE_EINVAL, "nblocks must be >= 0");
    if (nblocks == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&nblocks, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return probe_fail(MOE_ECUDA, "cannot read the device's SM count");
    }
    cudaError_t e = moe::ensure_dyn_smem(reinterpret_cast<const void *>(mma_peak_kernel), kPkSmem);
    if (e != cudaSuccess) return probe_fail(MOE_ECUDA, "mma_peak_kernel shared memory: %s", cudaGetErrorString(e));
    mma_peak_kernel<<<nblocks, 128, kPkSmem, static_cast<cudaStream_t>(stream)>>>(iters, static_cast<int *>(err_dev));
    e = cudaGetLastError();
    if (e != cudaSuccess) return probe_fail(MOE_ECUDA, "mma_peak_kernel: %s", cudaGetErrorString(e));
    return MOE_OK;
}
