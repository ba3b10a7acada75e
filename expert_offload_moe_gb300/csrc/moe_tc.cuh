// Device helpers for the Blackwell (sm_103a) tensor-core path: mbarriers,
// TMA tensor copies, tcgen05 MMA / TMEM, and the exact splitting of fp32 /
// bf16 values into E4M3 terms with E8M0 block scales.
//
// Layouts used with tcgen05.mma .kind::mxf8f6f4 .block_scale.scale_vec::1X
// (M = 128, cta_group::1), as verified on the GPU with exact integer data:
//  * A and B tiles are K-major, 128 bytes per row, 128-byte swizzle (16-byte
//    chunk c of row r stored at chunk c ^ (r % 8)), 8-row groups 1024 bytes
//    apart; the K step of one MMA (32 elements) advances the start address by
//    32 bytes.  E2M1 operands sit in smem as 16 codes in 8 bytes (low nibble
//    first) followed by 8 bytes of padding, i.e. one byte of smem per element.
//  * The accumulator D[m][n] is TMEM lane m, column base + n (fp32).
//  * Block scales (E8M0) of a 4-k-block step of an M=128 operand: TMEM lane
//    (32 q + m0) for every quadrant q, column base + (m / 32), byte k-block % 4
//    of row m = 32 (m / 32) + m0; the instruction's scale id picks the byte.
//    Scale addresses are 4-column aligned.  B (N <= 32) uses the same atom with
//    lane = column n.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {
namespace tc {

// Bounded waits: a spin that runs out sets an error word and returns false.
constexpr uint32_t kSpinLimit = 1u << 26;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase with the given parity; gives up after kWaitLimitNs, sets *err and returns false.
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *err, int code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 0; it < kSpinLimit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 63 && global_ns() - t0 > kWaitLimitNs) break;
    }
    if (err) atomicExch(err, code);
    return false;
}

// 3-D tiled TMA load into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_3d(const CUtensorMap *map, uint64_t *bar, void *dst, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// 16 bytes global -> shared by this thread (cp.async, generic proxy).
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// One arrival on bar once all of this thread's earlier cp.async copies have landed (counted in the
// barrier's expected arrivals, not added to them).  The consumer runs fence_proxy_async() after its wait
// before the tensor cores read the copied bytes.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// The lanes of a warp copy a rows x 128-byte tile (row stride src_stride) into the 128-byte-swizzled K-major
// layout the MMA descriptors read: 16-byte chunk c of row r lands at chunk c ^ (r % 8).
__device__ __forceinline__ void cp_async_tile_sw128(uint8_t *dst, const uint8_t *src, size_t src_stride, int rows,
                                                    int lane) {
    for (int q = lane; q < rows * 8; q += 32) {
        const int r = q >> 3, c = q & 7;
        cp_async16(dst + r * 128 + ((c ^ (r & 7)) << 4), src + (size_t)r * src_stride + c * 16);
    }
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 1-D bulk copy global -> shared completing on an mbarrier (16-byte aligned, multiple of 16 bytes).
__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Shared-memory stores that the tensor cores read through a descriptor: nothing in the program loads these
// bytes with an ordinary instruction, so they are issued as volatile stores that are never dropped or sunk.
__device__ __forceinline__ void st_shared_u8(void *p, uint32_t v) {
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_zero16(void *p) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(smem_u32(p)), "r"(0u) : "memory");
}
__device__ __forceinline__ void st_shared_fill16(void *p, uint32_t v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// ------------------------------------------------ thread-block clusters

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster; release / acquire orders shared-memory writes and reads.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of cluster_sync, for warps that reach a cluster barrier phase at different points:
// a thread arrives once per phase and waits for that phase before arriving at the next.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Barrier `id` (1..15) among `n` threads of the CTA (whole warps).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// fetch-and-add with acquire-release semantics at GPU scope
__device__ __forceinline__ unsigned atomic_add_acq_rel(unsigned *p, unsigned v) {
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.add.u32 %0, [%1], %2;" : "=r"(prev) : "l"(p), "r"(v) : "memory");
    return prev;
}

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    return a;
}

__device__ __forceinline__ float ld_dsmem(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// ------------------------------------------------ programmatic dependent launch
// wait: the grid launched before this one in the stream has completed and its writes are visible
// (no-op when this grid was launched without the programmatic-serialization attribute).
// trigger: the next grid may start launching once every CTA of this grid has triggered or exited.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t *slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot_smem)),
                 "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)(16 >> 4) << 16;    // leading byte offset (unused with swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;            // descriptor version
    d |= (uint64_t)2 << 61;            // 128-byte swizzle
    return d;
}

// Instruction descriptor, block-scaled kinds: formats (E4M3 = 0, E2M1 = 5), UE8M0 scales, M = 128.
__host__ __device__ constexpr uint32_t mx_idesc(uint32_t afmt, uint32_t bfmt, uint32_t N) {
    return (afmt << 7) | (bfmt << 10) | ((N >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24);
}

constexpr uint32_t kFmtE4M3 = 0, kFmtE2M1 = 5;

__device__ __forceinline__ void mma_mx(uint32_t tD, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfid,
                                       uint32_t tSFA, uint32_t tSFB, uint32_t accumulate) {
    const uint32_t id = idesc | (sfid << 4) | (sfid << 29);
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p; }" ::"r"(tD),
        "l"(adesc), "l"(bdesc), "r"(id), "r"(tSFA), "r"(tSFB), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Load and wait in one statement: the registers exist for the compiler only once the load has completed
// (with a separate wait, uses of the outputs may be scheduled above it).
__device__ __forceinline__ void tmem_ld8_sync(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(taddr)
        : "memory");
}

// Two 8-column loads in flight, then the wait.
__device__ __forceinline__ void tmem_ld8x2_sync(uint32_t ta, uint32_t (&a)[8], uint32_t tb, uint32_t (&b)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
          "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7])
        : "r"(ta), "r"(tb)
        : "memory");
}

// 32 consecutive columns of the warp's 32 lanes, load and wait in one statement.
__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// ------------------------------------------------ E4M3 terms of a 32-value block

// E8M0 byte of 2^e (e clamped to the E8M0 range).
__device__ __forceinline__ uint32_t e8m0_byte(int e) { return (uint32_t)min(max(e + 127, 0), 254); }

__device__ __forceinline__ float e8m0_value(uint32_t b) {
    return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

// Two fp32 values to packed E4M3 (round to nearest even, saturating).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Packed E4M3 pair back to fp32 (exact): low byte -> lo, high byte -> hi.  One asm block, no type punning.
__device__ __forceinline__ void e4m3x2_to_f32x2(uint16_t v, float &lo, float &hi) {
    asm("{\n\t.reg .b32 t;\n\t.reg .b16 a, b;\n\t"
        "cvt.rn.f16x2.e4m3x2 t, %2;\n\t"
        "mov.b32 {a, b}, t;\n\t"
        "cvt.f32.f16 %0, a;\n\t"
        "cvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "h"(v));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// floor(log2(a)) for a finite a > 0
__device__ __forceinline__ int floor_log2(float a) {
    const uint32_t u = __float_as_uint(a);
    const int e = (int)((u >> 23) & 0xff);
    if (e) return e - 127;
    return -127 - (__clz(u & 0x7fffff) - 9);  // subnormal
}

// One term of the exact E4M3 split of a 32-value block held one value per lane:
// returns this lane's code, updates the residual, and gives the block's E8M0 byte.
__device__ __forceinline__ uint8_t split_term(float &res, uint32_t &scale_byte) {
    const float amax = warp_max(fabsf(res));
    const int X = amax > 0.f ? max(floor_log2(amax) - 7, -127) : -127;  // |res| / 2^X < 256: no saturation
    scale_byte = e8m0_byte(X);
    const float inv = e8m0_value(e8m0_byte(-X));
    const float mine = res * inv;
    const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
    const int lane = threadIdx.x & 31;
    const uint16_t pk = (lane & 1) ? f32x2_to_e4m3x2(other, mine) : f32x2_to_e4m3x2(mine, other);
    const uint8_t code = (lane & 1) ? (uint8_t)(pk >> 8) : (uint8_t)(pk & 0xff);
    float lo, hi;
    e4m3x2_to_f32x2(pk, lo, hi);
    res = res - ((lane & 1) ? hi : lo) * e8m0_value(scale_byte);
    return code;
}

// ------------------------------------------------ E2M1 terms with UE4M3 scales per 16 values (NVFP4 path)

// Two fp32 values to one byte of E2M1 codes (round to nearest even, saturating at +-6): hi in the high nibble.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
    uint16_t r;
    asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u16.u8 %0, t; }" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// The two E2M1 codes of a byte back to fp32 (exact): low nibble -> lo, high nibble -> hi.
__device__ __forceinline__ void e2m1x2_to_f32x2(uint32_t byte, float &lo, float &hi) {
    asm("{\n\t.reg .b32 t;\n\t.reg .b16 a, b, c;\n\t.reg .b8 q;\n\t"
        "cvt.u16.u32 c, %2;\n\t"
        "cvt.u8.u16 q, c;\n\t"
        "cvt.rn.f16x2.e2m1x2 t, q;\n\t"
        "mov.b32 {a, b}, t;\n\t"
        "cvt.f32.f16 %0, a;\n\t"
        "cvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(byte));
}

// The smallest UE4M3 value >= s (s > 0, s <= 448) as its byte, and that value.
__device__ __forceinline__ uint32_t ue4m3_ceil(float s, float &v) {
    const uint16_t pk = f32x2_to_e4m3x2(s, s);
    uint32_t c = pk & 0xff;
    float lo, hi;
    e4m3x2_to_f32x2((uint16_t)(c | (c << 8)), lo, hi);
    if (lo < s && c < 0x7e) {
        ++c;
        e4m3x2_to_f32x2((uint16_t)(c | (c << 8)), lo, hi);
    }
    v = lo;
    return c;
}

// 2^e as fp32 for e in [-126, 127], 0 below.
__device__ __forceinline__ float pow2f(int e) { return e < -126 ? 0.f : __uint_as_float((uint32_t)(e + 127) << 23); }

// One E2M1 term of 16-value blocks held one value per lane (a half-warp per block): the block's scale
// s = the smallest UE4M3 >= max|res| / (6 G), codes RNE(res / (s G)); res loses the term exactly.  Returns the
// byte holding this lane's code with its pair lane's (even lane low nibble), and the block's scale byte
// (0 for an all-zero block or G == 0: codes 0).
__device__ __forceinline__ uint32_t split_term_e2m1(float &res, float G, uint32_t &scale_byte) {
    float bmax = fabsf(res);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
    const int lane = threadIdx.x & 31;
    float f = 0.f, sv = 0.f;
    scale_byte = 0;
    if (bmax > 0.f && G > 0.f) {
        scale_byte = ue4m3_ceil(bmax / (6.f * G), sv);
        f = res / (sv * G);
    }
    const float other = __shfl_xor_sync(0xffffffffu, f, 1);
    const uint32_t byte = (lane & 1) ? f32x2_to_e2m1x2(other, f) : f32x2_to_e2m1x2(f, other);
    float lo, hi;
    e2m1x2_to_f32x2(byte, lo, hi);
    if (sv > 0.f) res = res - ((lane & 1) ? hi : lo) * sv * G;
    return byte;
}

// ------------------------------------------------ operand tiles shared by the decode and prefill kernels

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + expf(-g)); }

// Scale atom (512 bytes in smem, 32 rows of 16 bytes) -> 4 TMEM columns in every lane quadrant.
__device__ __forceinline__ void atom_to_tmem(uint32_t tcol, const void *atom) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_u32(atom) >> 4) & 0x3FFF);
    d |= (uint64_t)(16 >> 4) << 16;
    d |= (uint64_t)(128 >> 4) << 32;  // next 8 rows
    d |= (uint64_t)1 << 46;
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tcol), "l"(d) : "memory");
}

// The last k-step of a row tile when K % 128 == 64: 64 codes per row copied by the whole warp into the
// padded, swizzled smem layout (unit u of row r at 16-byte chunk u ^ (r % 8)); all loads before any store.
__device__ __forceinline__ void load_tail_tile(uint8_t *dst, const uint8_t *codes, int rows, int row0, int K,
                                               int kstep) {
    const int lane = threadIdx.x & 31;
    constexpr int kUnits = 4, kPerLane = 128 * kUnits / 32;
    uint2 v[kPerLane];
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
        const int i = lane + 32 * j, r = i / kUnits, u = i % kUnits;
        v[j] = make_uint2(0u, 0u);
        if (row0 + r < rows)
            v[j] = __ldg(reinterpret_cast<const uint2 *>(codes + (size_t)(row0 + r) * (K / 2) + kstep * 64 + u * 8));
    }
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
        const int i = lane + 32 * j, r = i / kUnits, u = i % kUnits;
        *reinterpret_cast<uint4 *>(dst + r * 128 + ((u ^ (r & 7)) * 16)) = make_uint4(v[j].x, v[j].y, 0u, 0u);
    }
    fence_proxy_async();
    __syncwarp();
}

// 8 bytes global -> shared by this thread (cp.async, generic proxy); both addresses 8-byte aligned.
__device__ __forceinline__ void cp_async8(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// One arrival on bar once all of this thread's earlier cp.async copies have landed.  The barrier's pending
// count is raised by one when this is issued, so a barrier initialised for its other arrivals needs no
// change; issue it before the arrival that could otherwise complete the phase.
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// load_tail_tile without waiting for the loads: the 8 code bytes of unit u of row r go to 16-byte chunk
// u ^ (r % 8) by cp.async, the chunk's other 8 bytes (and whole chunks of rows past the matrix) are zeroed
// by stores.  The caller then runs fence_proxy_async() and cp_async_arrive() on the stage barrier in every
// lane; the consumer runs fence_proxy_async() after its wait, before the tensor cores read the tile.
__device__ __forceinline__ void cp_async_tail_tile(uint8_t *dst, const uint8_t *codes, int rows, int row0, int K,
                                                   int kstep) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int i = lane + 32 * j, r = i / 4, u = i % 4;
        uint8_t *d = dst + r * 128 + ((u ^ (r & 7)) * 16);
        if (row0 + r < rows) {
            cp_async8(d, codes + (size_t)(row0 + r) * (K / 2) + kstep * 64 + u * 8);
            asm volatile("st.shared.v2.u32 [%0], {%1, %1};" ::"r"(smem_u32(d + 8)), "r"(0u) : "memory");
        } else {
            st_shared_zero16(d);
        }
    }
}

}  // namespace tc
}  // namespace moe
