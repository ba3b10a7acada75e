// Prefill expert FFN (M > 8 tokens) on the 5th-generation tensor cores: a grouped, block-scaled GEMM over
// every expert of the layer staged in one device buffer (xinfer docs "How it works", Prefill: the whole
// expert layer is staged and the GEMM runs on it; tinyserve README, batched prefill: routes are grouped by
// expert so that each expert's weights are read once per batch).
//
// The route launch has already ordered the hot routes by (expert, token), padded each active expert's
// routes to whole 128-row tiles (a tile never mixes experts) and recorded the tile list, the expert ->
// active-index map and each route's hot-list position.  Then, on one stream:
//   prefill_quant_kernel     x of every route -> MXFP8 (E4M3 codes, one E8M0 scale per 32 columns, the
//                            OCP MX v1.0 conversion rule), gathered into route order with scale atoms
//   prefill_gemm_kernel<1>   per (route tile, 128 rows of I): Dg = x Wg^T, Du = x Wu^T on tcgen05
//                            (A = E4M3 routes, B = E2M1 weights, both block-scaled), h = SiLU(g) u,
//                            h -> MXFP8 in route order (the down GEMM's A operand)
//   prefill_gemm_kernel<0>   per (route tile, 256 rows of H): y = h Wd^T, times the route's weight
//   prefill_combine_kernel   out[t] = sum over t's routes in ascending expert order of w y
// Every result is computed in a fixed order, so it does not depend on timing.
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kEpiWarps = 8;
// warp 0: copies; warp 1 lane 0: MMAs; warps 2..9: epilogue; warp 10 lane 0: the proxy fence of each stage
constexpr int kThreads = 96 + 32 * kEpiWarps;
constexpr int kProxyWarp = 2 + kEpiWarps;
constexpr int kTileA = 128 * 128;         // one 128 x 128 operand tile in smem (one byte per element)
constexpr int kTileActTx = 128 * 128;     // TMA bytes of an E4M3 activation tile
constexpr int kTileWTx = 128 * 128 / 2;   // TMA bytes of an E2M1 weight tile (packed codes)
constexpr int kAtom = kTcAtomBytes;
constexpr int kStages = 4;
// stage: [A (128 routes)][B0 (128 weight rows)][B1 (128 weight rows)][atom A][atom B0][atom B1]
constexpr int kOffB0 = kTileA, kOffB1 = 2 * kTileA, kOffAtA = 3 * kTileA, kOffAtB0 = kOffAtA + kAtom,
              kOffAtB1 = kOffAtB0 + kAtom;
constexpr int kStage = 3 * kTileA + 3 * kAtom + 512;  // 50 KB
static_assert(kStage % 1024 == 0, "stage alignment");
constexpr int kSmemBytes = 1024 + kStages * kStage;
// tensor memory: one 256-column accumulator (gate | up, or 256 rows of down), then 12 scale columns per stage.
// The kernels are persistent (one CTA per SM walks the work items); the epilogue copies the accumulator to
// registers and releases it, so the next item's MMAs overlap the previous item's epilogue.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColSF = 256;
static_assert(kColSF + 12 * kStages <= kTmemCols, "tensor memory layout");
constexpr int kErrFull = 1, kErrEmpty = 2, kErrDone = 3;

// Byte of the 512-byte scale atom that holds row m (of a 128-row tile), k-block kb (of a 128-column step).
__device__ __forceinline__ int atom_byte(int m, int kb) { return (m & 31) * 16 + (m >> 5) * 4 + kb; }

// MXFP8 shared exponent of a block whose largest magnitude is amax (OCP MX v1.0: floor(log2 amax) minus the
// largest E4M3 exponent, 8; clamped to the E8M0 range; a block of zeros gets -127).
__device__ __forceinline__ int mxfp8_exponent(float amax) {
    if (!(amax > 0.f)) return -127;
    return min(max(floor_log2(amax) - 8, -127), 127);
}

// SiLU with the quotient from the fast reciprocal (2 ulp): the result is rounded to E4M3 next, and an
// error of this size is below the spread the accumulation order already gives g and u.  For g < -88 the
// denominator is infinite and the quotient 0, the limit of SiLU.
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.f + expf(-g)); }


}  // namespace

// ------------------------------------------------------------------ x -> MXFP8, route order

// One warp per route (the warps striding over the hot list): each lane converts 8 consecutive columns
// of the route's token, four lanes make one 32-column MXFP8 block.  XP[pr][Hpad] codes,
// XA[tile][kstep][512] scales, pr = the route's padded row.
__global__ void __launch_bounds__(256) prefill_quant_kernel(const uint16_t *x, int H, const int32_t *counts,
                                                            const int32_t *hot_expert, const int32_t *hot_token,
                                                            const int32_t *act_off, const int32_t *e2a,
                                                            const int32_t *poff, uint8_t *XP, int Hpad,
                                                            uint8_t *XA, int nks) {
    const int lane = threadIdx.x & 31;
    const int n_hot = counts[0];
    const int nit = (H + 255) / 256;
    for (int p = blockIdx.x * 8 + (threadIdx.x >> 5); p < n_hot; p += gridDim.x * 8) {
        const int a = e2a[hot_expert[p]];
        const int pr = poff[a] + (p - act_off[a]);
        const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)hot_token[p] * H);
        uint8_t *xp = XP + (size_t)pr * Hpad;
        uint8_t *xa = XA + (size_t)(pr >> 7) * nks * kAtom;
        for (int it = 0; it < nit; ++it) {
            const int col = it * 256 + lane * 8;
            const bool valid = col < H;  // H % 32 == 0: a 4-lane block is all valid or all past H
            const uint4 v = valid ? __ldg(xr + col / 8) : make_uint4(0u, 0u, 0u, 0u);
            float f[8];
            f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
            f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
            f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xffff0000u);
            f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xffff0000u);
            float m = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            const int X = mxfp8_exponent(m);
            const float inv = e8m0_value(e8m0_byte(-X));  // exact: a power of two
            const uint32_t lo = f32x2_to_e4m3x2(f[0] * inv, f[1] * inv) | (f32x2_to_e4m3x2(f[2] * inv, f[3] * inv) << 16);
            const uint32_t hi = f32x2_to_e4m3x2(f[4] * inv, f[5] * inv) | (f32x2_to_e4m3x2(f[6] * inv, f[7] * inv) << 16);
            if (valid) {
                *reinterpret_cast<uint2 *>(xp + col) = make_uint2(lo, hi);
                const int b = col / 32;
                if ((lane & 3) == 0) xa[(size_t)(b >> 2) * kAtom + atom_byte(pr & 127, b & 3)] = (uint8_t)(X + 127);
            }
        }
    }
}

// ------------------------------------------------------------------ grouped GEMM

namespace {

struct GemmArgs {
    const uint8_t *bank, *atoms;  // staged experts (slot = expert id) and their weight atoms
    size_t expert_bytes, atom_slot_bytes;
    size_t off_b0_codes, off_b1_codes;  // gate/up: Wg, Wu codes; down: Wd codes (both halves)
    size_t atom_off_b0, atom_off_b1;    // gate/up: gate, up atoms; down: down atoms
    int K, Nrows;                       // contraction length; rows of the weight matrix (I or H)
    int nN;                             // weight-row tiles per route tile (128 rows gate/up, 256 rows down)
    const int32_t *ntiles, *tile_aidx, *tile_nrows, *act_expert, *act_off, *poff;
    const float *hot_w;
    const uint8_t *Aat;  // atoms of the A operand [tile][kstep][512]
    // gate/up epilogue: h in route order (A operand of down)
    uint8_t *HP, *HA;
    int Ipad, nksI;
    // down epilogue: weighted y in route order
    float *YP;
    int H;
    int *err;
};

// Before a copy warp leaves: the copies of its last stages (issued, perhaps never consumed when a wait ran
// out) have landed, so nothing is written into the CTA's shared memory after it exits.  Lane 0 waits on the
// last min(it, S) stage barriers (bounded); a stage whose copies were consumed completed long ago.
__device__ __forceinline__ void drain_copies(uint64_t *full, int S, uint32_t it, int *err) {
    if ((threadIdx.x & 31) == 0)
        for (uint32_t j = it > (uint32_t)S ? it - S : 0u; j < it; ++j)
            if (!mbar_wait(&full[j % S], (j / S) & 1, err, kErrFull)) break;
    __syncwarp();
}

// The epilogue of one work item for accumulator row r (route row pr of the tile, valid if a real route)
// and this warp's half of the 256 columns, v = those columns as fp32 bits:
//   gate/up: h = SiLU(g) u for 64 of the item's 128 columns of I, stored as MXFP8 with its scale atom;
//   down: w y for 128 of the item's 256 columns of H.
template <int kGateUp>
__device__ __forceinline__ void epilogue_item(const GemmArgs &g, const uint32_t (&v)[128], int tile, int jn, int r,
                                              int half, int aidx, bool valid, int pr) {
    constexpr int kRowsN = kGateUp ? 128 : 256;
    if (kGateUp) {
        // h = SiLU(g) u for 64 of the item's 128 columns of I, one 32-column MXFP8 block at a time
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
            float h[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
                h[j] = valid ? silu_fast(__uint_as_float(v[32 * cb + j])) * __uint_as_float(v[64 + 32 * cb + j])
                             : 0.f;
            float amax = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(h[j]));
            const int X = mxfp8_exponent(amax);
            const float inv = e8m0_value(e8m0_byte(-X));
            uint32_t q[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t lo = f32x2_to_e4m3x2(h[4 * j] * inv, h[4 * j + 1] * inv);
                const uint32_t hi = f32x2_to_e4m3x2(h[4 * j + 2] * inv, h[4 * j + 3] * inv);
                q[j] = lo | (hi << 16);
            }
            const int c = 2 * half + cb;  // 32-column block of the item
            uint4 *dst = reinterpret_cast<uint4 *>(g.HP + (size_t)pr * g.Ipad + jn * 128 + 32 * c);
            dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
            dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
            g.HA[((size_t)tile * g.nksI + jn) * kAtom + atom_byte(r, c)] = (uint8_t)(X + 127);
        }
    } else {
        // y * w for 128 of the item's 256 columns of H (rows past the tile's routes are not stored)
        const int wrow0 = jn * kRowsN;
        const float wt = valid ? g.hot_w[g.act_off[aidx] + (pr - g.poff[aidx])] : 0.f;
        if (valid) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int col = wrow0 + half * 128 + 32 * c;
                if (col < g.H) {  // H % 32 == 0
                    float4 *dst = reinterpret_cast<float4 *>(g.YP + (size_t)pr * g.H + col);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        dst[j] = make_float4(wt * __uint_as_float(v[32 * c + 4 * j]),
                                             wt * __uint_as_float(v[32 * c + 4 * j + 1]),
                                             wt * __uint_as_float(v[32 * c + 4 * j + 2]),
                                             wt * __uint_as_float(v[32 * c + 4 * j + 3]));
                }
            }
        }
    }
}

template <int kGateUp>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB0,
                        const __grid_constant__ CUtensorMap mapB1, GemmArgs g) {
    constexpr int S = kStages;
    constexpr int NB = 256;  // MMA N: gate/up = [128 rows of Wg; the same 128 rows of Wu], down = 256 rows of Wd
    constexpr int kRowsN = kGateUp ? 128 : 256;  // weight rows per work item
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    __shared__ __align__(8) uint64_t full[S], ready[S], empty[S], acc_full, acc_empty, drain;
    __shared__ uint32_t tslot;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwork = *g.ntiles * g.nN;
    const int nks = (g.K + 127) / 128;
    const bool ragged = (g.K % 128) != 0;
    const int ntW = (g.Nrows + 127) / 128;  // 128-row weight tiles (atoms)

    if (warp == 1) tmem_alloc(&tslot, kTmemCols);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1 + 32);  // the copy thread's expect_tx + the 32 lanes' atom copies
            mbar_init(&ready[s], 1);      // the proxy warp, after its fence
            mbar_init(&empty[s], 1);
        }
        mbar_init(&acc_full, 1);
        mbar_init(&acc_empty, kEpiWarps);
        mbar_init(&drain, 1);
        fence_barrier_init();
        tma_prefetch_desc(&mapA);
        tma_prefetch_desc(&mapB0);
        tma_prefetch_desc(&mapB1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tslot;

    if (warp == 0) {
        // ---------------- operand copies: one ring of stages across all work items ----------------
        bool ok = true;
        uint32_t it = 0;
        for (int w = blockIdx.x; w < nwork && ok; w += gridDim.x) {
            const int tile = w / g.nN, jn = w - tile * g.nN;
            const int expert = g.act_expert[g.tile_aidx[tile]];
            const int wrow0 = jn * kRowsN;
            const bool b1 = kGateUp || wrow0 + 128 < g.Nrows;
            const int r0 = wrow0, r1 = kGateUp ? wrow0 : wrow0 + 128;
            const uint8_t *ex = g.bank + (size_t)expert * g.expert_bytes;
            const uint8_t *exat = g.atoms + (size_t)expert * g.atom_slot_bytes;
            for (int i = 0; i < nks; ++i, ++it) {
                const int st = it % S;
                if (lane == 0) ok = mbar_wait(&empty[st], ((it / S) & 1) ^ 1, g.err, kErrEmpty);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                uint8_t *sS = smem + st * kStage;
                const bool tail = ragged && i == nks - 1;
                const size_t atom0 = g.atom_off_b0 + ((size_t)(r0 >> 7) * nks + i) * kAtom;
                const size_t atom1 = g.atom_off_b1 + ((size_t)(r1 >> 7) * nks + i) * kAtom;
                if (tail) {
                    load_tail_tile(sS + kOffB0, ex + g.off_b0_codes, g.Nrows, r0, g.K, i);
                    if (b1) load_tail_tile(sS + kOffB1, ex + g.off_b1_codes, g.Nrows, r1, g.K, i);
                }
                if (lane == 0) {
                    const uint32_t wtx = tail ? 0u : (uint32_t)kTileWTx;
                    mbar_expect_tx(&full[st], kTileActTx + wtx * (b1 ? 2u : 1u));
                    tma_load_3d(&mapA, &full[st], sS, i * 128, tile * 128, 0);
                    if (!tail) {
                        tma_load_3d(&mapB0, &full[st], sS + kOffB0, i * 128, r0, expert);
                        if (b1) tma_load_3d(&mapB1, &full[st], sS + kOffB1, i * 128, r1, expert);
                    }
                }
                // the scale atoms (512 bytes each) by the lanes, 16 bytes apiece: small copies through the
                // tensor-copy unit would each cost it a whole request
                cp_async16(sS + kOffAtA + lane * 16, g.Aat + ((size_t)tile * nks + i) * kAtom + lane * 16);
                cp_async16(sS + kOffAtB0 + lane * 16, exat + atom0 + lane * 16);
                if (b1 && (kGateUp || (r1 >> 7) < ntW)) cp_async16(sS + kOffAtB1 + lane * 16, exat + atom1 + lane * 16);
                cp_async_arrive_noinc(&full[st]);
                __syncwarp();
            }
        }
        drain_copies(full, S, it, g.err);
    } else if (warp == 1) {
        // ---------------- MMAs: one thread; the accumulator is reused once the epilogue has drained it ----
        if (lane == 0) {
            const uint32_t idesc = mx_idesc(kFmtE4M3, kFmtE2M1, NB);
            bool ok = true;
            uint32_t it = 0;
            int n = 0;
            for (int w = blockIdx.x; w < nwork && ok; w += gridDim.x, ++n) {
                if (n > 0) {
                    ok = mbar_wait(&acc_empty, (n - 1) & 1, g.err, kErrDone);
                    if (!ok) break;
                    tc_fence_after();
                }
                const int jn = w % g.nN;
                const bool b1 = kGateUp || jn * kRowsN + 128 < g.Nrows;  // the second weight half exists
                for (int i = 0; i < nks; ++i, ++it) {
                    const int st = it % S;
                    ok = mbar_wait(&ready[st], (it / S) & 1, g.err, kErrFull);
                    if (!ok) break;
                    tc_fence_after();
                    uint8_t *sS = smem + st * kStage;
                    const uint32_t sfa = tbase + kColSF + 12 * st, sfb0 = sfa + 4, sfb1 = sfa + 8;
                    atom_to_tmem(sfa, sS + kOffAtA);
                    atom_to_tmem(sfb0, sS + kOffAtB0);
                    if (b1) atom_to_tmem(sfb1, sS + kOffAtB1);
                    const uint32_t aA = smem_u32(sS), aB0 = aA + kOffB0;
                    const int nk = (ragged && i == nks - 1) ? 2 : 4;
                    // one N = 256 MMA over both weight halves (contiguous in smem), B scales in two atoms:
                    // gate/up accumulates g in columns 0..127 and u in 128..255
                    for (int kk = 0; kk < nk; ++kk) {
                        const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                        mma_mx(tbase, sw128_desc(aA + kk * 32), sw128_desc(aB0 + kk * 32), idesc, kk, sfa, sfb0, acc);
                    }
                    mma_commit(&empty[st]);
                }
                if (ok) mma_commit(&acc_full);
            }
            // every MMA issued has finished before the CTA can leave, also when a wait ran out
            mma_commit(&drain);
            mbar_wait(&drain, 0, g.err, kErrDone);
        }
        __syncwarp();
    } else if (warp == kProxyWarp) {
        // ---------------- proxy fence: the atoms (and ragged tail tiles) of each stage came through the
        // generic proxy; this warp waits for the stage, fences, and hands it to the MMA thread, which then
        // issues no fence of its own ----------------
        if (lane == 0) {
            bool ok = true;
            uint32_t it = 0;
            for (int w = blockIdx.x; w < nwork && ok; w += gridDim.x)
                for (int i = 0; i < nks; ++i, ++it) {
                    const int st = it % S;
                    ok = mbar_wait(&full[st], (it / S) & 1, g.err, kErrFull);
                    if (!ok) break;
                    fence_proxy_async();
                    mbar_arrive(&ready[st]);
                }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: row r = 32 (warp % 4) + lane (a warp reaches its own 32 lanes of
        // tensor memory); the two warps of a lane quarter take one half of the columns each ----------
        const int quarter = warp & 3, half = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        int n = 0;
        for (int w = blockIdx.x; w < nwork; w += gridDim.x, ++n) {
            const int tile = w / g.nN, jn = w - tile * g.nN;
            const int aidx = g.tile_aidx[tile], nrows = g.tile_nrows[tile];
            const bool valid = r < nrows;
            const int pr = tile * 128 + r;  // padded route row
            const bool got = __all_sync(0xffffffffu, mbar_wait(&acc_full, n & 1, g.err, kErrDone));
            if (!got) break;
            tc_fence_after();
            // drain this warp's 128 accumulator columns, then hand the accumulator back to the MMA thread
            uint32_t v[128];
            if (kGateUp) {
                tmem_ld32_sync(tbase + lane_off + half * 64, v);
                tmem_ld32_sync(tbase + lane_off + half * 64 + 32, v + 32);
                tmem_ld32_sync(tbase + lane_off + 128 + half * 64, v + 64);
                tmem_ld32_sync(tbase + lane_off + 128 + half * 64 + 32, v + 96);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32_sync(tbase + lane_off + half * 128 + 32 * c, v + 32 * c);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty);
            epilogue_item<kGateUp>(g, v, tile, jn, r, half, aidx, valid, pr);
        }
    }
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, kTmemCols);
}


}  // namespace

// ------------------------------------------------------------------ combine

// One block per token: its routes in ascending expert order (each route's padded row from its hot-list
// position), summed into out four columns per thread.
__global__ void __launch_bounds__(256) prefill_combine_kernel(const int32_t *topk_ids, int k, const int32_t *e2a,
                                                              const int32_t *act_off, const int32_t *route_pos,
                                                              const int32_t *poff, const float *YP, int H,
                                                              void *out, int out_f32) {
    __shared__ int s_pr[kMaxTopK];
    const int t = blockIdx.x;
    if (threadIdx.x < k) {
        const int j = threadIdx.x, e = topk_ids[(size_t)t * k + j];
        int rank = 0;  // the k experts of a token are distinct
        for (int i = 0; i < k; ++i) rank += topk_ids[(size_t)t * k + i] < e;
        const int a = e2a[e];
        s_pr[rank] = poff[a] + (route_pos[(size_t)t * k + j] - act_off[a]);
    }
    __syncthreads();
    for (int h4 = threadIdx.x; h4 < H / 4; h4 += blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const float4 y = __ldg(reinterpret_cast<const float4 *>(YP + (size_t)s_pr[j] * H) + h4);
            acc.x += y.x;
            acc.y += y.y;
            acc.z += y.z;
            acc.w += y.w;
        }
        if (out_f32) {
            reinterpret_cast<float4 *>(out)[(size_t)t * (H / 4) + h4] = acc;
        } else {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 v;
            v.x = (uint32_t)__bfloat16_as_ushort(lo.x) | ((uint32_t)__bfloat16_as_ushort(lo.y) << 16);
            v.y = (uint32_t)__bfloat16_as_ushort(hi.x) | ((uint32_t)__bfloat16_as_ushort(hi.y) << 16);
            reinterpret_cast<uint2 *>(out)[(size_t)t * (H / 4) + h4] = v;
        }
    }
}

// ------------------------------------------------------------------ launchers

int prefill_tiles_cap(int max_routes, int E) { return (max_routes + 127) / 128 + (E < max_routes ? E : max_routes); }

cudaError_t launch_prefill(const PrefillLaunch &P, cudaStream_t s) {
    const ExpertGeometry &geo = P.geo;
    const TcAtomLayout l = tc_atom_layout(geo.H, geo.I);
    prefill_quant_kernel<<<(unsigned)((P.max_routes + 7) / 8), 256, 0, s>>>(P.x, geo.H, P.counts, P.hot_expert, P.hot_token,
                                                                      P.act_off, P.e2a, P.poff, P.XP, P.Hpad, P.XA,
                                                                      l.nks);
    ensure_dyn_smem(reinterpret_cast<const void *>(prefill_gemm_kernel<1>), kSmemBytes);
    ensure_dyn_smem(reinterpret_cast<const void *>(prefill_gemm_kernel<0>), kSmemBytes);
    GemmArgs g{};
    g.bank = P.bank;
    g.atoms = P.atoms;
    g.expert_bytes = geo.expert_bytes;
    g.atom_slot_bytes = l.slot_bytes;
    g.ntiles = P.ntiles;
    g.tile_aidx = P.tile_aidx;
    g.tile_nrows = P.tile_nrows;
    g.act_expert = P.act_expert;
    g.act_off = P.act_off;
    g.poff = P.poff;
    g.hot_w = P.hot_w;
    g.HP = P.HP;
    g.HA = P.HA;
    g.Ipad = P.Ipad;
    g.nksI = l.nksI;
    g.YP = P.YP;
    g.H = geo.H;
    g.err = P.err;
    // gate/up: A = x (route order), B = Wg / Wu tiles of 128 rows of I
    g.off_b0_codes = geo.off_wg_codes;
    g.off_b1_codes = geo.off_wu_codes;
    g.atom_off_b0 = l.off_g;
    g.atom_off_b1 = l.off_u;
    g.K = geo.H;
    g.Nrows = geo.I;
    g.nN = l.ntI;
    g.Aat = P.XA;
    if (P.ev[0]) cudaEventRecord(P.ev[0], s);
    const int grid1 = P.tiles_cap * g.nN < P.num_sms ? P.tiles_cap * g.nN : P.num_sms;
    prefill_gemm_kernel<1><<<grid1, kThreads, kSmemBytes, s>>>(*P.mapXP, *P.mapG, *P.mapU, g);
    if (P.ev[1]) cudaEventRecord(P.ev[1], s);
    // down: A = h (route order), B = Wd tiles of 256 rows of H
    g.off_b0_codes = geo.off_wd_codes;
    g.off_b1_codes = geo.off_wd_codes;
    g.atom_off_b0 = l.off_d;
    g.atom_off_b1 = l.off_d;
    g.K = geo.I;
    g.Nrows = geo.H;
    g.nN = (geo.H + 255) / 256;
    g.Aat = P.HA;
    if (P.ev[2]) cudaEventRecord(P.ev[2], s);
    const int grid0 = P.tiles_cap * g.nN < P.num_sms ? P.tiles_cap * g.nN : P.num_sms;
    prefill_gemm_kernel<0><<<grid0, kThreads, kSmemBytes, s>>>(*P.mapHP, *P.mapD, *P.mapD, g);
    if (P.ev[3]) cudaEventRecord(P.ev[3], s);
    prefill_combine_kernel<<<P.M, 256, 0, s>>>(P.topk_ids, P.k, P.e2a, P.act_off, P.route_pos, P.poff, P.YP, geo.H,
                                               P.out, P.out_f32);
    return cudaGetLastError();
}

void launch_build_weight_atoms_bank(const uint8_t *bank, int E, const ExpertGeometry &g, uint8_t *atoms,
                                    cudaStream_t s) {
    const TcAtomLayout l = tc_atom_layout(g.H, g.I);
    for (int e = 0; e < E; ++e)
        launch_build_weight_atoms(bank + (size_t)e * g.expert_bytes, g, atoms + (size_t)e * l.slot_bytes, s);
}

}  // namespace moe
