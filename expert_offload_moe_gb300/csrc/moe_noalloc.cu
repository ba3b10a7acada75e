// Routing without any allocation: moe_route_noalloc (declared in include/moe.h).
//
// Some callers cannot allocate device memory at the point where they route:
// a serving process whose device memory is reserved up front by another
// allocator (its own pool holds the whole budget, so a cudaMalloc from this
// library would fail or fragment it), or a latency-critical decode loop where
// the implicit device synchronisation of cudaMalloc/cudaFree is not allowed.
// For them this entry point runs the same route kernel as moe_route, with the
// caller's own inputs and output buffers, and keeps its only scratch -- the
// partial router logits and the grid arrival counter -- in the file-scope
// device array below.  The array is part of the library's image: every GPU
// that loads the library holds it until the process exits.
//
// On the host, the name g_route_scratch is only a stand-in for the device
// symbol, not a device address; its device address is fetched once per
// device with cudaGetSymbolAddress (with that device current) and passed to
// the kernel.  All calls share the array and it keeps the last call's
// contents: the arrival counter is cleared at the start of every call, and
// calls that overlap on the GPU (different streams, no ordering) race on it.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "moe_internal.h"

namespace {

// 256 bytes for the arrival counter, then partial logits (fp32): 1 MiB in all.
constexpr size_t kScratchBytes = size_t(1) << 20;
constexpr size_t kCounterBytes = 256;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

struct DeviceSetup {
    void *scratch = nullptr;  // device address of g_route_scratch on this device
    int num_sms = 0;
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mu;

// Failures are reported through moe_last_error(), like every other call.
int noalloc_fail(int code, const char *fmt, ...) {
    char buf[384];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    moe::set_last_error(buf);
    return code;
}

// Finds (once per device, with that device current) the scratch array's device address.
int device_setup(DeviceSetup *out) {
    int dev = 0;
    cudaError_t rc = cudaGetDevice(&dev);
    if (rc != cudaSuccess) return noalloc_fail(MOE_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(rc));
    if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(MOE_EINVAL, "device %d beyond %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_setup_mu);
    DeviceSetup &s = g_setup[dev];
    if (!s.scratch) {
        void *ptr = nullptr;
        rc = cudaGetSymbolAddress(&ptr, g_route_scratch);
        if (rc != cudaSuccess || !ptr)
            return noalloc_fail(MOE_ECUDA, "cudaGetSymbolAddress(route scratch): %s", cudaGetErrorString(rc));
        int sms = 0;
        rc = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (rc != cudaSuccess) return noalloc_fail(MOE_ECUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(rc));
        s.num_sms = sms;
        s.scratch = ptr;
    }
    *out = s;
    return MOE_OK;
}

}  // namespace

extern "C" int moe_route_noalloc(const void *x_dev, int32_t M, int32_t H, const float *router_w_dev,
                                 const float *router_bias_dev, int32_t E, int32_t top_k,
                                 const int32_t *expert_to_slot_dev, const moe_route_buffers *out, void *stream) {
    moe::set_last_error("");
    if (!x_dev || !router_w_dev || !expert_to_slot_dev || !out)
        return noalloc_fail(MOE_EINVAL, "x_dev, router_w_dev, expert_to_slot_dev and out are required");
    if (!out->topk_ids || !out->topk_w || !out->hot_expert || !out->hot_token || !out->hot_w || !out->act_expert ||
        !out->act_slot || !out->act_off || !out->act_cnt || !out->cold_token || !out->cold_expert || !out->cold_w ||
        !out->hist || !out->counts)
        return noalloc_fail(MOE_EINVAL, "every output buffer in moe_route_buffers is required");
    if (H <= 0 || H % 64) return noalloc_fail(MOE_EINVAL, "H must be a positive multiple of 64 (got %d)", H);
    if (top_k < 1 || top_k > moe::kMaxTopK || E < top_k || E > moe::kMaxExperts)
        return noalloc_fail(MOE_EINVAL, "need 1 <= top_k <= %d and top_k <= E <= %d", moe::kMaxTopK, moe::kMaxExperts);
    if (M < 1 || M > moe::kMaxTokens) return noalloc_fail(MOE_EINVAL, "M = %d outside [1, %d]", M, moe::kMaxTokens);
    if (reinterpret_cast<uintptr_t>(x_dev) % 16 || reinterpret_cast<uintptr_t>(router_w_dev) % 16)
        return noalloc_fail(MOE_EINVAL, "x_dev and router_w_dev must be 16-byte aligned");
    const int nchunk = (H + moe::kRouteChunk - 1) / moe::kRouteChunk;
    const size_t need = (size_t)nchunk * M * E * sizeof(float);
    if (need > kScratchBytes - kCounterBytes)
        return noalloc_fail(MOE_EINVAL,
                            "M=%d, H=%d, E=%d need %zu bytes of route scratch; the built-in array holds %zu "
                            "(ceil(H/256) * M * E * 4 bytes must fit)",
                            M, H, E, need, kScratchBytes - kCounterBytes);

    DeviceSetup s;
    int rc = device_setup(&s);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char *base = static_cast<unsigned char *>(s.scratch);
    // The arrival counter must start at zero.  The route kernel's last block returns it to zero, so calls
    // ordered on one stream would find it so; the memset is kept because calls that overlap on the GPU
    // (documented as racing) can leave it elsewhere, and no later call would then ever find a last block.
    // It costs the route launch its programmatic overlap with the kernel before it.
    cudaError_t e = cudaMemsetAsync(base, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) return noalloc_fail(MOE_ECUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));

    moe::RouteParams p{};
    p.x = static_cast<const uint16_t *>(x_dev);
    p.Wr = router_w_dev;
    p.bias = router_bias_dev;
    p.e2s = expert_to_slot_dev;
    p.M = M;
    p.H = H;
    p.E = E;
    p.k = top_k;
    p.nchunk = nchunk;
    p.all_hot = 0;
    p.b.logit_part = reinterpret_cast<float *>(base + kCounterBytes);
    p.b.arrive = reinterpret_cast<unsigned *>(base);
    p.b.topk_ids = out->topk_ids;
    p.b.topk_w = out->topk_w;
    p.b.hot_expert = out->hot_expert;
    p.b.hot_token = out->hot_token;
    p.b.hot_w = out->hot_w;
    p.b.act_expert = out->act_expert;
    p.b.act_slot = out->act_slot;
    p.b.act_off = out->act_off;
    p.b.act_cnt = out->act_cnt;
    p.b.cold_token = out->cold_token;
    p.b.cold_expert = out->cold_expert;
    p.b.cold_w = out->cold_w;
    p.b.hist = out->hist;
    p.b.counts = out->counts;
    e = moe::launch_route(p, st, s.num_sms);
    if (e != cudaSuccess) return noalloc_fail(MOE_ECUDA, "route kernel launch: %s", cudaGetErrorString(e));
    return MOE_OK;
}
