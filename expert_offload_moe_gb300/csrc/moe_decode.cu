// Decode expert FFN (M <= 8 tokens) straight from the MXFP4 slot bytes.
//
// gateup_kernel: for every active slot and every row i of its intermediate
//   dimension, one warp streams row i of Wg and Wu (16-byte loads = one
//   32-element MXFP4 block per lane), decodes the E2M1 codes in registers,
//   multiplies by the bf16 activations of every token routed to the slot
//   (fp32, exact products), applies the E8M0 block scale to each 32-element
//   partial, sums across the warp, and writes h = SiLU(g) * u in fp32.
//   NVFP4 weights (kNv): the same 32 codes per lane carry two E4M3 scales, one
//   per 16-element half, each applied to its half's partial.
// down_kernel: one warp per output row r: for every active slot in ascending
//   expert order and every route of it, y = Wd[r, :] . h, and the weighted
//   sum over the token's routes is formed in the same order and stored.
//   Combining in expert order (not slot order) keeps the output independent
//   of where an expert sits (xinfer docs: placement never changes precision).
//
// The work lists and counts come from the route kernel in device memory; the
// grids are fixed (persistent, sized by the SM count), so the launches are
// the same for every routing (xinfer docs "How it works").
#include <cuda_bf16.h>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
    return e ? __uint_as_float(e << 23) : __uint_as_float(0x00400000u);
}

// E4M3 byte (sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 subnormal; S.1111.111 NaN) to
// fp32, exactly: the value is placed into an fp32 bit pattern (normal) or scaled from its mantissa (subnormal).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u, sign = (b & 0x80u) << 24;
    if (e == 15u && m == 7u) return __uint_as_float(0x7fc00000u);
    const float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;  // m 2^-9
    return __uint_as_float(__float_as_uint(mag) | sign);
}

template <bool kNv>
__device__ __forceinline__ void block_scales(const uint8_t *scales, int b, float &s0, float &s1) {
    if (kNv) {  // two E4M3 bytes: columns [32 b, 32 b + 16) and [32 b + 16, 32 b + 32)
        const uint32_t two = __ldg(reinterpret_cast<const uint16_t *>(scales) + b);
        s0 = e4m3_to_f32(two & 0xffu);
        s1 = e4m3_to_f32(two >> 8);
    } else {
        s0 = s1 = e8m0_to_f32(__ldg(scales + b));
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void fill_e2m1_lut(float *lut) {
    if (threadIdx.x < 16) {
        const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
        const float m = mag[threadIdx.x & 7];
        lut[threadIdx.x] = (threadIdx.x & 8) ? -m : m;
    }
}

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + expf(-g)); }

template <int kM, bool kNv>
__global__ void __launch_bounds__(kThreads) gateup_kernel(DecodeParams p, int M) {
    extern __shared__ float sx[];  // [M][H] activations as fp32
    __shared__ float lut[16];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = p.geo.H, I = p.geo.I, nb = H / 32;
    fill_e2m1_lut(lut);
    // block-transposed: sx[t][j][b] = x[t][32 b + j], so that lane b of a warp reading element j of its
    // block hits consecutive words (no bank conflicts)
    for (int i = threadIdx.x; i < M * H; i += kThreads) {
        const int t = i / H, c = i - t * H;
        sx[t * H + (c & 31) * nb + (c >> 5)] = __uint_as_float((uint32_t)p.x[i] << 16);
    }
    __syncthreads();

    const int n_act = p.counts[2];
    const int total = n_act * I;
    for (int task = blockIdx.x * kWarps + warp; task < total; task += gridDim.x * kWarps) {
        const int a = task / I, i = task - a * I;
        const int slot = p.act_slot[a], off = p.act_off[a], cnt = p.act_cnt[a];
        const uint8_t *base = p.bank + (size_t)slot * p.geo.expert_bytes;
        const uint8_t *gq = base + p.geo.off_wg_codes + (size_t)i * (H / 2);
        const uint8_t *gs = base + p.geo.off_wg_scales + (size_t)i * (kNv ? 2 * nb : nb);
        const uint8_t *uq = base + p.geo.off_wu_codes + (size_t)i * (H / 2);
        const uint8_t *us = base + p.geo.off_wu_scales + (size_t)i * (kNv ? 2 * nb : nb);
        int tok[kM];
#pragma unroll
        for (int t = 0; t < kM; ++t) tok[t] = t < cnt ? p.hot_token[off + t] : 0;
        float g[kM], u[kM];
#pragma unroll
        for (int t = 0; t < kM; ++t) g[t] = u[t] = 0.f;

        for (int b = lane; b < nb; b += 32) {
            const uint4 qg4 = ld_stream(gq + (size_t)b * 16);
            const uint4 qu4 = ld_stream(uq + (size_t)b * 16);
            float sg0, sg1, su0, su1;
            block_scales<kNv>(gs, b, sg0, sg1);
            block_scales<kNv>(us, b, su0, su1);
            const uint32_t qg[4] = {qg4.x, qg4.y, qg4.z, qg4.w};
            const uint32_t qu[4] = {qu4.x, qu4.y, qu4.z, qu4.w};
            // partials per 16-column half (MXFP4: both halves share one scale, summed before scaling)
            float pg[2][kM], pu[2][kM];
#pragma unroll
            for (int t = 0; t < kM; ++t) pg[0][t] = pu[0][t] = pg[1][t] = pu[1][t] = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int hf = kNv ? q >> 1 : 0;
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    const float vg = lut[(qg[q] >> (4 * n)) & 15u];
                    const float vu = lut[(qu[q] >> (4 * n)) & 15u];
#pragma unroll
                    for (int t = 0; t < kM; ++t) {
                        if (t < cnt) {
                            const float xv = sx[tok[t] * H + (q * 8 + n) * nb + b];
                            pg[hf][t] = fmaf(vg, xv, pg[hf][t]);
                            pu[hf][t] = fmaf(vu, xv, pu[hf][t]);
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kM; ++t) {
                g[t] = fmaf(pg[0][t], sg0, g[t]);
                u[t] = fmaf(pu[0][t], su0, u[t]);
                if (kNv) {
                    g[t] = fmaf(pg[1][t], sg1, g[t]);
                    u[t] = fmaf(pu[1][t], su1, u[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kM; ++t) {
            if (t < cnt) {
                const float gt = warp_sum(g[t]), ut = warp_sum(u[t]);
                // h is stored block-transposed like x: h[route][i % 32][i / 32]
                if (lane == 0) p.h[(size_t)(off + t) * I + (i & 31) * (I / 32) + (i >> 5)] = silu(gt) * ut;
            }
        }
    }
}

template <int kM, bool kNv>
__global__ void __launch_bounds__(kThreads) down_kernel(DecodeParams p, int M) {
    __shared__ float lut[16];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = p.geo.H, I = p.geo.I, nb = I / 32;
    fill_e2m1_lut(lut);
    __syncthreads();
    const int n_act = p.counts[2];

    for (int r = blockIdx.x * kWarps + warp; r < H; r += gridDim.x * kWarps) {
        float acc[kM];
#pragma unroll
        for (int t = 0; t < kM; ++t) acc[t] = 0.f;
        for (int a = 0; a < n_act; ++a) {
            const int slot = p.act_slot[a], off = p.act_off[a], cnt = p.act_cnt[a];
            const uint8_t *base = p.bank + (size_t)slot * p.geo.expert_bytes;
            const uint8_t *dq = base + p.geo.off_wd_codes + (size_t)r * (I / 2);
            const uint8_t *ds = base + p.geo.off_wd_scales + (size_t)r * (kNv ? 2 * nb : nb);
            float y[kM];
#pragma unroll
            for (int t = 0; t < kM; ++t) y[t] = 0.f;
            for (int b = lane; b < nb; b += 32) {
                const uint4 q4 = ld_stream(dq + (size_t)b * 16);
                float s0, s1;
                block_scales<kNv>(ds, b, s0, s1);
                const uint32_t q[4] = {q4.x, q4.y, q4.z, q4.w};
                float py[2][kM];
#pragma unroll
                for (int t = 0; t < kM; ++t) py[0][t] = py[1][t] = 0.f;
#pragma unroll
                for (int t = 0; t < kM; ++t) {
                    if (t < cnt) {
                        const float *hp = p.h + (size_t)(off + t) * I + b;  // block-transposed h
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq) {
                            const int hf = kNv ? qq >> 1 : 0;
#pragma unroll
                            for (int n = 0; n < 8; ++n)
                                py[hf][t] = fmaf(lut[(q[qq] >> (4 * n)) & 15u], hp[(qq * 8 + n) * nb], py[hf][t]);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < kM; ++t) {
                    y[t] = fmaf(py[0][t], s0, y[t]);
                    if (kNv) y[t] = fmaf(py[1][t], s1, y[t]);
                }
            }
#pragma unroll
            for (int t = 0; t < kM; ++t) {
                if (t < cnt) {
                    const float yt = warp_sum(y[t]);
                    const int tok = p.hot_token[off + t];
                    const float wt = p.hot_w[off + t];
#pragma unroll
                    for (int tt = 0; tt < kM; ++tt)
                        if (tt == tok) acc[tt] = fmaf(wt, yt, acc[tt]);
                }
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int t = 0; t < kM; ++t) {
                if (t < M) {
                    if (p.out_f32)
                        reinterpret_cast<float *>(p.out)[(size_t)t * H + r] = acc[t];
                    else
                        reinterpret_cast<__nv_bfloat16 *>(p.out)[(size_t)t * H + r] = __float2bfloat16_rn(acc[t]);
                }
            }
        }
    }
}

}  // namespace

// The token loops are unrolled for kM tokens per slot, the smallest of
// 1, 2, 4, 8 that covers M (a slot never serves more tokens than M).
template <int kM, bool kNv>
void gateup_launch(const DecodeParams &p, int M, cudaStream_t s, int num_sms) {
    ensure_dyn_smem(reinterpret_cast<const void *>(gateup_kernel<kM, kNv>), kDecodeSmemLimit);
    gateup_kernel<kM, kNv><<<num_sms * 4, kThreads, (size_t)M * p.geo.H * sizeof(float), s>>>(p, M);
}

template <bool kNv>
void gateup_by_m(const DecodeParams &p, int M, cudaStream_t s, int num_sms) {
    if (M <= 1) gateup_launch<1, kNv>(p, M, s, num_sms);
    else if (M <= 2) gateup_launch<2, kNv>(p, M, s, num_sms);
    else if (M <= 4) gateup_launch<4, kNv>(p, M, s, num_sms);
    else gateup_launch<8, kNv>(p, M, s, num_sms);
}

template <bool kNv>
void down_by_m(const DecodeParams &p, int M, cudaStream_t s, int num_sms) {
    if (M <= 1) down_kernel<1, kNv><<<num_sms * 4, kThreads, 0, s>>>(p, M);
    else if (M <= 2) down_kernel<2, kNv><<<num_sms * 4, kThreads, 0, s>>>(p, M);
    else if (M <= 4) down_kernel<4, kNv><<<num_sms * 4, kThreads, 0, s>>>(p, M);
    else down_kernel<8, kNv><<<num_sms * 4, kThreads, 0, s>>>(p, M);
}

// NVFP4 geometry (16 columns per scale byte) takes the E4M3-scale kernels.
void launch_gateup(const DecodeParams &p, int M, cudaStream_t s, int num_sms) {
    if (p.geo.sblk == 16) gateup_by_m<true>(p, M, s, num_sms);
    else gateup_by_m<false>(p, M, s, num_sms);
}

void launch_down(const DecodeParams &p, int M, cudaStream_t s, int num_sms) {
    if (p.geo.sblk == 16) down_by_m<true>(p, M, s, num_sms);
    else down_by_m<false>(p, M, s, num_sms);
}

}  // namespace moe
