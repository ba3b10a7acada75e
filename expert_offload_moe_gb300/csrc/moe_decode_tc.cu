// Decode expert FFN (M <= 8 tokens) on the 5th-generation tensor cores.
//
// The MXFP4 weights are never decoded by the SM: TMA copies the E2M1 codes of
// a 128-row x 128-column tile straight from the slot bytes into shared memory
// (expanded to one byte per code, 128-byte swizzle), and tcgen05.mma
// .kind::mxf8f6f4.block_scale multiplies them with the activations while
// applying the E8M0 block scales of both operands from tensor memory; fp32
// accumulators live in tensor memory (tinyserve README "How it works" 2: fused
// dequantise-and-multiply, gate / up / down; xinfer docs "How it works":
// GEMMs over [num_slots, N, K] slot tensors).
//
// The activation operand must be 8-bit, so each value is split exactly into
// E4M3 terms with one E8M0 scale per 32-element block along K: x (bf16, 8-bit
// significand) = 2 terms, reproduced exactly for every element within 2^14 of
// its block's largest magnitude; h (fp32) = 4 terms (16 significant bits).
// Each term is one more column of the B operand, and the columns of a token
// are summed after the MMA.  The routing weight is folded into the down
// operand (w * h), so the down MMA accumulates sum over experts of w * Wd h
// directly: the combine happens in tensor memory, in ascending expert order.
//
// quantize_x_kernel  x -> x terms (B operand of gate/up)
// gateup_tc_kernel   one CTA per (active expert, 128-row tile of I, K split):
//                    Dg = Wg x, Du = Wu x; then h = SiLU(g) u, w h -> h terms
// down_tc_kernel     one CTA per (128-row tile of H, K split over the
//                    concatenated (expert, k-step) sequence): out = sum_e Wd_e (w h)
// K splits write fp32 partials; the last CTA of a tile (arrival counter, no
// waiting) sums them in split order, so results do not depend on timing.
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kStages = 4;
constexpr int kTileA = 128 * 128;       // one 128 x 128 E2M1 tile, one byte per code in smem
constexpr int kTileATx = 128 * 128 / 2;  // bytes a TMA copy of that tile moves (the packed codes)
constexpr uint32_t kTmemCols = 256;  // a CTA handles at most kMaxSteps k-steps
constexpr int kMaxSteps = 16;
constexpr int NBX = 16;  // B columns of gate/up: 2 x terms x <= 8 tokens
constexpr int kHTerms = 4;  // E4M3 terms of w * h: 16 significant bits
constexpr int NBH = 32;      // B columns of down: 4 h terms x <= 8 tokens
// error codes written to the error word
constexpr int kErrFull = 1, kErrEmpty = 2, kErrDone = 3, kErrScales = 4, kErrSteps = 5;

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + expf(-g)); }

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
    int X = amax > 0.f ? floor_log2(amax) - 7 : -127;  // |res| / 2^X < 256: no saturation
    X = max(X, -127);
    scale_byte = e8m0_byte(X);
    const float inv = e8m0_value(e8m0_byte(-X) < 255 ? e8m0_byte(-X) : 254);
    // pair lanes so one cvt packs two values; each lane keeps its own byte
    const float mine = res * inv;
    const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
    const int lane = threadIdx.x & 31;
    const uint16_t pk = (lane & 1) ? f32x2_to_e4m3x2(other, mine) : f32x2_to_e4m3x2(mine, other);
    const uint8_t code = (lane & 1) ? (uint8_t)(pk >> 8) : (uint8_t)(pk & 0xff);
    float lo, hi;
    e4m3x2_to_f32x2(pk, lo, hi);
    const float q = (lane & 1) ? hi : lo;
    res = res - q * e8m0_value(scale_byte);
    return code;
}

}  // namespace

// ------------------------------------------------------------------ x terms

// xq[t * 2 + term][Hpad] E4M3 codes, xs[t * 2 + term][SP] E8M0 scales; one warp per 32-block.
__global__ void __launch_bounds__(256) quantize_x_kernel(const uint16_t *x, int M, int H, uint8_t *xq, int Hpad,
                                                         uint8_t *xs, int SP) {
    const int lane = threadIdx.x & 31;
    const int nb = H / 32;
    const int task = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (task >= M * nb) return;
    const int t = task / nb, b = task - t * nb;
    float res = __uint_as_float((uint32_t)x[(size_t)t * H + b * 32 + lane] << 16);
#pragma unroll
    for (int term = 0; term < 2; ++term) {
        uint32_t sb;
        const uint8_t code = split_term(res, sb);
        xq[(size_t)(t * 2 + term) * Hpad + b * 32 + lane] = code;
        if (lane == 0) xs[(size_t)(t * 2 + term) * SP + b] = (uint8_t)sb;
    }
}

namespace {

// ---------------------------------------------------------------- warp roles
// 192 threads: warp 0 issues TMA copies (its lanes also copy a ragged last k-step), warp 1 lane 0 issues the
// MMAs and warp 1 owns the tensor memory, warps 2..5 load the block scales into tensor memory while the
// first copies are in flight, then read the accumulators (warp w reads TMEM lane quadrant w % 4).
constexpr int kRoleThreads = 192;
constexpr int kScaleWarp0 = 2;

__device__ __forceinline__ void named_sync_scale_warps() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Weight scales of one k-step for row r of a 128-row tile: 4 E8M0 bytes (k-blocks 4 kstep .. +3) as one word;
// 2^0 for rows or k-blocks outside the matrix.  nkb is even, so the byte pairs never straddle the end.
__device__ __forceinline__ uint32_t weight_scale_word(const uint8_t *scales, int rows, int nkb, int row, int kstep) {
    uint32_t v = 0x7f7f7f7fu;
    if (row < rows) {
        const int c = kstep * 4;
        const uint16_t *p = reinterpret_cast<const uint16_t *>(scales + (size_t)row * nkb + c);
        const uint32_t lo = c < nkb ? (uint32_t)__ldg(p) : 0x7f7fu;
        const uint32_t hi = c + 2 < nkb ? (uint32_t)__ldg(p + 1) : 0x7f7fu;
        v = lo | (hi << 16);
    }
    return v;
}

// Writes the scale atoms of n k-steps from s_sc[step][row] into this warp's TMEM lane quadrant:
// column base + 4 s + m1, byte kb, of row 32 m1 + lane.
__device__ __forceinline__ void store_weight_scales(uint32_t tcol, const uint32_t *s_sc, int n) {
    const int lane = threadIdx.x & 31, quad = (threadIdx.x >> 5) & 3;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    for (int s = 0; s < n; ++s)
        tmem_st4(tcol + lane_off + 4 * s, s_sc[s * 128 + lane], s_sc[s * 128 + 32 + lane], s_sc[s * 128 + 64 + lane],
                 s_sc[s * 128 + 96 + lane]);
}

// Scales of the B operand (N <= 32 columns, one row of SP bytes each, padded with 2^0 past K); column n is
// TMEM lane n of every quadrant.
__device__ __forceinline__ void store_operand_scales(uint32_t tcol, const uint8_t *scales, int SP, int NB, int kstep) {
    const int lane = threadIdx.x & 31, quad = (threadIdx.x >> 5) & 3;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    uint32_t v = 0x7f7f7f7fu;
    if (lane < NB) v = *reinterpret_cast<const uint32_t *>(scales + (size_t)lane * SP + kstep * 4);
    tmem_st1(tcol + lane_off, v);
}

// The last k-step of a row tile when K is not a multiple of 128: the codes of each row (K - 128 kstep of
// them, 8 bytes per 16) copied by the whole warp into the padded, swizzled smem layout (unit u of row r at
// 16-byte chunk u ^ (r % 8)).
__device__ __forceinline__ void load_tail_tile(uint8_t *dst, const uint8_t *codes, int rows, int row0, int K,
                                               int kstep) {
    // K is a multiple of 64, so a ragged step holds 64 codes: 4 units per row, 16 per lane; every load is
    // issued before the first store so the warp waits for memory once
    const int lane = threadIdx.x & 31;
    constexpr int kUnits = 4, kPerLane = 128 * kUnits / 32;
    (void)K;
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

struct GateUpArgs {
    const uint8_t *bank;
    size_t expert_bytes, off_g_codes, off_g_scales, off_u_codes, off_u_scales;
    int H, I, M, KS;
    const int32_t *counts, *act_slot, *act_off, *act_cnt, *hot_token;
    const float *hot_w;
    const uint8_t *xs;  // x-term scales [16][SPH]
    int SPH;
    uint8_t *hq, *hs;   // w*h terms [n_act_max][32][Ipad], scales [n_act_max][32][SPI]
    int Ipad, SPI;
    float *part;        // split-K partials
    unsigned *tile_ctr;
    int *err;
};

constexpr int kGateStage = 2 * kTileA + ((NBX * 128 + 1023) / 1024) * 1024;
constexpr int kDownStage = kTileA + ((NBH * 128 + 1023) / 1024) * 1024;

__global__ void __launch_bounds__(kRoleThreads, 1)
    gateup_tc_kernel(const __grid_constant__ CUtensorMap mapG, const __grid_constant__ CUtensorMap mapU,
                     const __grid_constant__ CUtensorMap mapX, GateUpArgs a) {
    constexpr int kB = NBX * 128;
    constexpr uint32_t kTx = 2 * kTileATx + kB;
    constexpr int T = kHTerms;  // terms of w * h in the down operand
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint32_t *s_scg = reinterpret_cast<uint32_t *>(smem + kStages * kGateStage);  // [kMaxSteps][128]
    uint32_t *s_scu = s_scg + kMaxSteps * 128;
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], done, scales_ready;
    __shared__ uint32_t tslot;
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_act = a.counts[2];
    const int ntile = (a.I + 127) / 128;
    const int aidx = blockIdx.x / (ntile * a.KS);
    if (aidx >= n_act) return;
    const int rem = blockIdx.x - aidx * ntile * a.KS;
    const int tile = rem / a.KS, ks = rem - tile * a.KS;
    const int nks = (a.H + 127) / 128;
    const int k0 = ks * nks / a.KS, k1 = (ks + 1) * nks / a.KS, nsteps = k1 - k0;
    const bool ragged = (a.H % 128) != 0;
    if (nsteps > kMaxSteps) {  // the host always splits K finely enough; refuse rather than overrun
        if (threadIdx.x == 0) atomicExch(a.err, kErrSteps);
        return;
    }
    const int slot = a.act_slot[aidx];
    const uint8_t *expert = a.bank + (size_t)slot * a.expert_bytes;
    const int row0 = tile * 128;

    if (warp == 1) tmem_alloc(&tslot, kTmemCols);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        mbar_init(&scales_ready, 128);
        fence_barrier_init();
        tma_prefetch_desc(&mapG);
        tma_prefetch_desc(&mapU);
        tma_prefetch_desc(&mapX);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tslot;
    const uint32_t tDg = tbase, tDu = tbase + 16, tSFg = tbase + 32, tSFu = tbase + 32 + 4 * kMaxSteps,
                   tSFb = tbase + 32 + 8 * kMaxSteps;

    bool ok = true;
    if (warp == 0) {
        // producer
        for (int i = 0; i < nsteps && ok; ++i) {
            const int st = i % kStages;
            const int kstep = k0 + i;
            if (lane == 0) ok = mbar_wait(&empty[st], ((i / kStages) & 1) ^ 1, a.err, kErrEmpty);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            uint8_t *sA = smem + st * kGateStage;
            const bool tail = ragged && kstep == nks - 1;
            if (tail) {
                load_tail_tile(sA, expert + a.off_g_codes, a.I, row0, a.H, kstep);
                load_tail_tile(sA + kTileA, expert + a.off_u_codes, a.I, row0, a.H, kstep);
            }
            if (lane == 0) {
                mbar_expect_tx(&full[st], tail ? (uint32_t)kB : kTx);
                if (!tail) {
                    tma_load_3d(&mapG, &full[st], sA, kstep * 128, row0, slot);
                    tma_load_3d(&mapU, &full[st], sA + kTileA, kstep * 128, row0, slot);
                }
                tma_load_3d(&mapX, &full[st], sA + 2 * kTileA, kstep * 128, 0, 0);
            }
            __syncwarp();
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = mx_idesc(kFmtE2M1, kFmtE4M3, NBX);
            ok = mbar_wait(&scales_ready, 0, a.err, kErrScales);
            tc_fence_after();
            for (int i = 0; i < nsteps && ok; ++i) {
                const int st = i % kStages;
                ok = mbar_wait(&full[st], (i / kStages) & 1, a.err, kErrFull);
                if (!ok) break;
                tc_fence_after();
                const uint32_t aG = smem_u32(smem + st * kGateStage), aU = aG + kTileA, aB = aG + 2 * kTileA;
                const bool tail = ragged && (k0 + i) == nks - 1;
                const int nk = tail ? ((a.H - (k0 + i) * 128) / 32) : 4;
                for (int kk = 0; kk < nk; ++kk) {
                    const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                    mma_mx(tDg, sw128_desc(aG + kk * 32), sw128_desc(aB + kk * 32), idesc, kk, tSFg + 4 * i,
                           tSFb + 4 * i, acc);
                    mma_mx(tDu, sw128_desc(aU + kk * 32), sw128_desc(aB + kk * 32), idesc, kk, tSFu + 4 * i,
                           tSFb + 4 * i, acc);
                }
                mma_commit(&empty[st]);
            }
            mma_commit(&done);
        }
        __syncwarp();
    } else {
        // scale warps: thread r loads row r's scale words of every step, regrouped through shared memory
        const int r = threadIdx.x - kScaleWarp0 * 32;
        const uint8_t *gsc = expert + a.off_g_scales, *usc = expert + a.off_u_scales;
        const int nkb = a.H / 32;
        uint32_t wg[kMaxSteps], wu[kMaxSteps];
#pragma unroll
        for (int s = 0; s < kMaxSteps; ++s) {
            if (s < nsteps) {
                wg[s] = weight_scale_word(gsc, a.I, nkb, row0 + r, k0 + s);
                wu[s] = weight_scale_word(usc, a.I, nkb, row0 + r, k0 + s);
            }
        }
#pragma unroll
        for (int s = 0; s < kMaxSteps; ++s) {
            if (s < nsteps) {
                s_scg[s * 128 + r] = wg[s];
                s_scu[s * 128 + r] = wu[s];
            }
        }
        named_sync_scale_warps();
        store_weight_scales(tSFg, s_scg, nsteps);
        store_weight_scales(tSFu, s_scu, nsteps);
        for (int s = 0; s < nsteps; ++s) store_operand_scales(tSFb + 4 * s, a.xs, a.SPH, NBX, k0 + s);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&scales_ready);
    }

    // ---------------- epilogue (scale warps): every thread owns one row of the tile ----------------
    const bool epi = warp >= kScaleWarp0;
    const int quad = warp & 3;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int row = row0 + quad * 32 + lane;
    const int M = a.M;
    float g[2 * kDecodeMaxTokens], u[2 * kDecodeMaxTokens];
#pragma unroll
    for (int c = 0; c < 2 * kDecodeMaxTokens; ++c) g[c] = u[c] = 0.f;
    if (epi) {
        const bool got = mbar_wait(&done, 0, a.err, kErrDone);
        tc_fence_after();
        if (got) {
            uint32_t rr[8];
#pragma unroll
            for (int c8 = 0; c8 < 2; ++c8) {
                tmem_ld8(tDg + lane_off + 8 * c8, rr);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 8; ++j) g[8 * c8 + j] = __uint_as_float(rr[j]);
                tmem_ld8(tDu + lane_off + 8 * c8, rr);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 8; ++j) u[8 * c8 + j] = __uint_as_float(rr[j]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tbase, kTmemCols);
    if (!epi) return;

    const int rloc = quad * 32 + lane;  // row within the tile
    if (a.KS > 1) {
        // partials [unit][2][2 kDecodeMaxTokens][128], summed by the last CTA of the tile in split order
        const int tile_id = aidx * ntile + tile;
        float *mine = a.part + ((size_t)tile_id * a.KS + ks) * kTcPartGateup;
#pragma unroll
        for (int c = 0; c < 2 * kDecodeMaxTokens; ++c) {
            if (c < 2 * M) {
                mine[(0 * 2 * kDecodeMaxTokens + c) * 128 + rloc] = g[c];
                mine[(1 * 2 * kDecodeMaxTokens + c) * 128 + rloc] = u[c];
            }
        }
        __threadfence();
        named_sync_scale_warps();
        if (threadIdx.x == kScaleWarp0 * 32) s_last = atomicAdd(&a.tile_ctr[tile_id], 1u) == (unsigned)(a.KS - 1);
        named_sync_scale_warps();
        if (!s_last) return;
        __threadfence();
        if (threadIdx.x == kScaleWarp0 * 32) a.tile_ctr[tile_id] = 0u;
#pragma unroll
        for (int c = 0; c < 2 * kDecodeMaxTokens; ++c) g[c] = u[c] = 0.f;
        for (int k = 0; k < a.KS; ++k) {
            const float *p = a.part + ((size_t)tile_id * a.KS + k) * kTcPartGateup;
#pragma unroll
            for (int c = 0; c < 2 * kDecodeMaxTokens; ++c) {
                if (c < 2 * M) {
                    g[c] += __ldcg(p + (0 * 2 * kDecodeMaxTokens + c) * 128 + rloc);
                    u[c] += __ldcg(p + (1 * 2 * kDecodeMaxTokens + c) * 128 + rloc);
                }
            }
        }
    }

    // h = SiLU(g) u for the tokens routed to this expert; w h split into T E4M3 terms per 32-row block
    const int off = a.act_off[aidx], cnt = a.act_cnt[aidx];
    uint8_t *hq = a.hq + (size_t)aidx * NBH * a.Ipad;
    uint8_t *hs = a.hs + (size_t)aidx * NBH * a.SPI;
    float vt[kDecodeMaxTokens];
#pragma unroll
    for (int t = 0; t < kDecodeMaxTokens; ++t) vt[t] = 0.f;
    for (int j = 0; j < cnt; ++j) {
        const int t = a.hot_token[off + j];
        const float w = a.hot_w[off + j];
#pragma unroll
        for (int tt = 0; tt < kDecodeMaxTokens; ++tt) {
            if (tt == t) {
                const float gg = g[2 * tt] + g[2 * tt + 1], uu = u[2 * tt] + u[2 * tt + 1];
                vt[tt] = w * (silu(gg) * uu);
            }
        }
    }
    if (row < a.I) {  // whole 32-row blocks are in or out (I % 64 == 0)
#pragma unroll
        for (int t = 0; t < kDecodeMaxTokens; ++t) {
            if (t >= M) break;
            float res = vt[t];
#pragma unroll
            for (int term = 0; term < T; ++term) {
                uint32_t sb;
                const uint8_t code = split_term(res, sb);
                hq[(size_t)(t * T + term) * a.Ipad + row] = code;
                if (lane == 0) hs[(size_t)(t * T + term) * a.SPI + row / 32] = (uint8_t)sb;
            }
        }
    }
}

struct DownArgs {
    const uint8_t *bank;
    size_t expert_bytes, off_d_codes, off_d_scales;
    int H, I, M, KS;
    const int32_t *counts, *act_slot;
    const uint8_t *hs;  // [n_act_max][32][SPI]
    int Ipad, SPI;
    void *out;
    int out_f32;
    float *part;
    unsigned *tile_ctr;
    int *err;
};

__global__ void __launch_bounds__(kRoleThreads, 1)
    down_tc_kernel(const __grid_constant__ CUtensorMap mapD, const __grid_constant__ CUtensorMap mapH, DownArgs a) {
    constexpr int NB = NBH;
    constexpr int kB = NB * 128;
    constexpr uint32_t kTx = kTileATx + kB;
    constexpr int T = kHTerms;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint32_t *s_sc = reinterpret_cast<uint32_t *>(smem + kStages * kDownStage);  // [kMaxSteps][128]
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], done, scales_ready;
    __shared__ uint32_t tslot;
    __shared__ int s_last;
    __shared__ int s_slot[kMaxExperts];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_act = a.counts[2];
    const int tile = blockIdx.x / a.KS, ks = blockIdx.x - tile * a.KS;
    const int nksI = (a.I + 127) / 128;
    const int total = n_act * nksI;
    const int g0 = ks * total / a.KS, g1 = (ks + 1) * total / a.KS, nsteps = g1 - g0;
    const bool ragged = (a.I % 128) != 0;
    const int row0 = tile * 128;
    if (nsteps > kMaxSteps) {
        if (threadIdx.x == 0) atomicExch(a.err, kErrSteps);
        return;
    }
    for (int i = threadIdx.x; i < n_act; i += kRoleThreads) s_slot[i] = a.act_slot[i];

    if (warp == 1) tmem_alloc(&tslot, kTmemCols);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        mbar_init(&scales_ready, 128);
        fence_barrier_init();
        tma_prefetch_desc(&mapD);
        tma_prefetch_desc(&mapH);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tslot;
    const uint32_t tD = tbase, tSFa = tbase + 32, tSFb = tbase + 32 + 4 * kMaxSteps;

    bool ok = true;
    if (warp == 0) {
        for (int i = 0; i < nsteps && ok; ++i) {
            const int st = i % kStages;
            const int g = g0 + i, e = g / nksI, s = g - e * nksI;
            if (lane == 0) ok = mbar_wait(&empty[st], ((i / kStages) & 1) ^ 1, a.err, kErrEmpty);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            uint8_t *sA = smem + st * kDownStage;
            const bool tail = ragged && s == nksI - 1;
            if (tail)
                load_tail_tile(sA, a.bank + (size_t)s_slot[e] * a.expert_bytes + a.off_d_codes, a.H, row0, a.I, s);
            if (lane == 0) {
                mbar_expect_tx(&full[st], tail ? (uint32_t)kB : kTx);
                if (!tail) tma_load_3d(&mapD, &full[st], sA, s * 128, row0, s_slot[e]);
                tma_load_3d(&mapH, &full[st], sA + kTileA, s * 128, 0, e);
            }
            __syncwarp();
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = mx_idesc(kFmtE2M1, kFmtE4M3, NB);
            ok = mbar_wait(&scales_ready, 0, a.err, kErrScales);
            tc_fence_after();
            for (int i = 0; i < nsteps && ok; ++i) {
                const int st = i % kStages;
                ok = mbar_wait(&full[st], (i / kStages) & 1, a.err, kErrFull);
                if (!ok) break;
                tc_fence_after();
                const int s = (g0 + i) % nksI;
                const uint32_t aA = smem_u32(smem + st * kDownStage), aB = aA + kTileA;
                const bool tail = ragged && s == nksI - 1;
                const int nk = tail ? ((a.I - s * 128) / 32) : 4;
                for (int kk = 0; kk < nk; ++kk) {
                    const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                    mma_mx(tD, sw128_desc(aA + kk * 32), sw128_desc(aB + kk * 32), idesc, kk, tSFa + 4 * i,
                           tSFb + 4 * i, acc);
                }
                mma_commit(&empty[st]);
            }
            mma_commit(&done);
        }
        __syncwarp();
    } else {
        const int r = threadIdx.x - kScaleWarp0 * 32;
        uint32_t w[kMaxSteps];
#pragma unroll
        for (int i = 0; i < kMaxSteps; ++i) {
            if (i < nsteps) {
                const int g = g0 + i, e = g / nksI, s = g - e * nksI;
                const uint8_t *expert = a.bank + (size_t)s_slot[e] * a.expert_bytes;
                w[i] = weight_scale_word(expert + a.off_d_scales, a.H, a.I / 32, row0 + r, s);
            }
        }
#pragma unroll
        for (int i = 0; i < kMaxSteps; ++i)
            if (i < nsteps) s_sc[i * 128 + r] = w[i];
        named_sync_scale_warps();
        store_weight_scales(tSFa, s_sc, nsteps);
        for (int i = 0; i < nsteps; ++i) {
            const int g = g0 + i, e = g / nksI, s = g - e * nksI;
            store_operand_scales(tSFb + 4 * i, a.hs + (size_t)e * NB * a.SPI, a.SPI, NB, s);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&scales_ready);
    }

    const bool epi = warp >= kScaleWarp0;
    const int quad = warp & 3;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int rloc = quad * 32 + lane;
    const int row = row0 + rloc;
    const int M = a.M;
    float d[kDecodeMaxTokens * T];
#pragma unroll
    for (int c = 0; c < kDecodeMaxTokens * T; ++c) d[c] = 0.f;
    if (epi) {
        const bool got = mbar_wait(&done, 0, a.err, kErrDone);
        tc_fence_after();
        if (got && nsteps > 0) {
            uint32_t rr[8];
#pragma unroll
            for (int c8 = 0; c8 < (kDecodeMaxTokens * T + 7) / 8; ++c8) {
                if (8 * c8 < M * T) {
                    tmem_ld8(tD + lane_off + 8 * c8, rr);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (8 * c8 + j < kDecodeMaxTokens * T) d[8 * c8 + j] = __uint_as_float(rr[j]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tbase, kTmemCols);
    if (!epi) return;

    if (a.KS > 1) {
        float *mine = a.part + ((size_t)tile * a.KS + ks) * kTcPartDown;
#pragma unroll
        for (int c = 0; c < kDecodeMaxTokens * T; ++c)
            if (c < M * T) mine[c * 128 + rloc] = d[c];
        __threadfence();
        named_sync_scale_warps();
        if (threadIdx.x == kScaleWarp0 * 32) s_last = atomicAdd(&a.tile_ctr[tile], 1u) == (unsigned)(a.KS - 1);
        named_sync_scale_warps();
        if (!s_last) return;
        __threadfence();
        if (threadIdx.x == kScaleWarp0 * 32) a.tile_ctr[tile] = 0u;
#pragma unroll
        for (int c = 0; c < kDecodeMaxTokens * T; ++c) d[c] = 0.f;
        for (int k = 0; k < a.KS; ++k) {
            const float *p = a.part + ((size_t)tile * a.KS + k) * kTcPartDown;
#pragma unroll
            for (int c = 0; c < kDecodeMaxTokens * T; ++c)
                if (c < M * T) d[c] += __ldcg(p + c * 128 + rloc);
        }
    }
    if (row < a.H) {
#pragma unroll
        for (int t = 0; t < kDecodeMaxTokens; ++t) {
            if (t >= M) break;
            float v = 0.f;
#pragma unroll
            for (int term = 0; term < T; ++term) v += d[t * T + term];
            if (a.out_f32)
                reinterpret_cast<float *>(a.out)[(size_t)t * a.H + row] = v;
            else
                reinterpret_cast<__nv_bfloat16 *>(a.out)[(size_t)t * a.H + row] = __float2bfloat16_rn(v);
        }
    }
}

template <typename K>
void set_smem(K kernel, int bytes) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

// stages + the regrouped weight scales (one [kMaxSteps][128] word table per weight matrix) + alignment slack
int tc_gateup_smem() { return kStages * kGateStage + 2 * kMaxSteps * 128 * 4 + 1024; }
int tc_down_smem() { return kStages * kDownStage + kMaxSteps * 128 * 4 + 1024; }

void launch_quantize_x(const uint16_t *x, int M, int H, uint8_t *xq, int Hpad, uint8_t *xs, int SP, cudaStream_t s) {
    const int tasks = M * (H / 32);
    quantize_x_kernel<<<(tasks + 7) / 8, 256, 0, s>>>(x, M, H, xq, Hpad, xs, SP);
}

void launch_gateup_tc(const TcLaunch &L, cudaStream_t s) {
    GateUpArgs a{};
    a.bank = L.bank;
    a.expert_bytes = L.geo.expert_bytes;
    a.off_g_codes = L.geo.off_wg_codes;
    a.off_g_scales = L.geo.off_wg_scales;
    a.off_u_codes = L.geo.off_wu_codes;
    a.off_u_scales = L.geo.off_wu_scales;
    a.H = L.geo.H;
    a.I = L.geo.I;
    a.M = L.M;
    a.KS = L.ks_gateup;
    a.counts = L.counts;
    a.act_slot = L.act_slot;
    a.act_off = L.act_off;
    a.act_cnt = L.act_cnt;
    a.hot_token = L.hot_token;
    a.hot_w = L.hot_w;
    a.xs = L.xs;
    a.SPH = L.SPH;
    a.hq = L.hq;
    a.hs = L.hs;
    a.Ipad = L.Ipad;
    a.SPI = L.SPI;
    a.part = L.part;
    a.tile_ctr = L.tile_ctr_gateup;
    a.err = L.err;
    const int ntile = (L.geo.I + 127) / 128;
    const int grid = L.n_act_max * ntile * L.ks_gateup;
    static bool cfg = false;
    if (!cfg) set_smem(gateup_tc_kernel, tc_gateup_smem()), cfg = true;
    gateup_tc_kernel<<<grid, kRoleThreads, tc_gateup_smem(), s>>>(*L.mapG, *L.mapU, *L.mapX, a);
}

void launch_down_tc(const TcLaunch &L, cudaStream_t s) {
    DownArgs a{};
    a.bank = L.bank;
    a.expert_bytes = L.geo.expert_bytes;
    a.off_d_codes = L.geo.off_wd_codes;
    a.off_d_scales = L.geo.off_wd_scales;
    a.H = L.geo.H;
    a.I = L.geo.I;
    a.M = L.M;
    a.KS = L.ks_down;
    a.counts = L.counts;
    a.act_slot = L.act_slot;
    a.hs = L.hs;
    a.Ipad = L.Ipad;
    a.SPI = L.SPI;
    a.out = L.out;
    a.out_f32 = L.out_f32;
    a.part = L.part_down;
    a.tile_ctr = L.tile_ctr_down;
    a.err = L.err;
    const int grid = ((L.geo.H + 127) / 128) * L.ks_down;
    static bool cfg = false;
    if (!cfg) set_smem(down_tc_kernel, tc_down_smem()), cfg = true;
    down_tc_kernel<<<grid, kRoleThreads, tc_down_smem(), s>>>(*L.mapD, *L.mapH, a);
}

}  // namespace moe
