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
// Block scales travel as 512-byte atoms, one per (128-row tile, 128-column
// k-step): byte m0*16 + m1*4 + kb holds the scale of row 32 m1 + m0 and
// k-block 4 step + kb.  An atom is bulk-copied with its operand tile and moved
// into tensor memory by tcgen05.cp (32x128b, replicated to the four lane
// quadrants) right before the MMAs that use it.  Weight atoms are built once
// when an expert lands in a slot (build_weight_atoms); activation atoms are
// written by the kernels that produce the activation terms.
//
// The activation operand must be 8-bit, so each value is split exactly into
// E4M3 terms with one E8M0 scale per 32-element block along K: x (bf16, 8-bit
// significand) = 2 terms, reproduced exactly for every element within 2^14 of
// its block's largest magnitude; w h (fp32) = 8 terms, each taking 4 more
// significant bits of the block's largest residual (32 bits below the block's
// largest magnitude: h may span a wide range within 32 consecutive rows).
// Each term is one more column of the B operand, and the columns of a token
// are summed after the MMA.  The routing weight is folded into the down
// operand (w h), so the down MMA accumulates the sum over experts of w Wd h in
// tensor memory, in ascending expert order: the combine happens there.
//
// The x terms and their atoms (B operand of gate/up) are written by the route launch.
// gateup_tc_kernel   one CTA per (active expert, 128-row tile of I, K split):
//                    Dg = Wg x, Du = Wu x; then h = SiLU(g) u, w h -> h terms
// down_tc_kernel     one CTA per (128-row tile of H, K split over the
//                    concatenated (expert, k-step) sequence): out = sum_e Wd_e (w h)
// ffn_tc_kernel      (M = 1) both in one launch per (active expert, I tile, K split):
//                    gate/up, h in shared memory, then the tile's column slice of Wd
//                    into fp32 partials; ffn_combine_kernel sums them in a fixed order
// The K splits of a tile form a thread-block cluster; their partials meet in distributed
// shared memory and are summed in rank order, so results do not depend on timing.
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kThreads = 128;           // warp 0: copies; warp 1 lane 0: MMAs; all 4 warps: epilogue
constexpr int kTileA = 128 * 128;       // one 128 x 128 E2M1 tile, one byte per code in smem
constexpr int kTileATx = 128 * 128 / 2; // bytes a TMA copy of that tile moves (the packed codes)
constexpr int kAtom = kTcAtomBytes;
constexpr int NBX = kTcXRows;           // B columns of gate/up: 2 x terms x <= 8 tokens
constexpr int NBH = kTcHRows;           // B columns of down: 8 w*h terms x <= 8 tokens
constexpr int kHTerms = 8;
constexpr int kGateStages = 3, kDownStages = 4;
// stage layout: [A tiles][B tile][atoms], 1024-aligned for the 128-byte swizzle
constexpr int kGateStage = 2 * kTileA + NBX * 128 + 3 * kAtom + 512;   // 36 KB
constexpr int kDownStage = kTileA + NBH * 128 + 2 * kAtom + 1024;       // 26 KB
static_assert(kGateStage % 1024 == 0 && kDownStage % 1024 == 0, "stage alignment");
// Accumulators per operand: MMA slice kk of a k-step accumulates into kk % kAcc (summed in the epilogue).
// More than one did not shorten a k-step on GB300 (the MMA chain is not the bottleneck), so one.
constexpr int kAcc = 1;
constexpr uint32_t tmem_cols(uint32_t need) { return need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : need <= 256 ? 256 : 512; }
constexpr uint32_t kGateTmem = tmem_cols(2 * kAcc * kTcXRows + 12 * kGateStages);
constexpr uint32_t kDownTmem = tmem_cols(kAcc * kTcHRows + 8 * kDownStages);
constexpr int kErrFull = 1, kErrEmpty = 2, kErrDone = 3;

}  // namespace

// ------------------------------------------------------------------ atoms

// Weight scale atoms of one slot: for each (row tile, k-step), byte m0*16 + m1*4 + kb = scale of row
// 128 tile + 32 m1 + m0 and k-block 4 step + kb (2^0 outside the matrix).  One warp per atom.
__global__ void __launch_bounds__(256) build_weight_atoms_kernel(const uint8_t *scales, int rows, int nkb,
                                                                 uint8_t *atoms, int ntile, int nsteps) {
    const int atom = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (atom >= ntile * nsteps) return;
    const int tile = atom / nsteps, step = atom - tile * nsteps, m0 = threadIdx.x & 31;
    uint32_t w[4];
#pragma unroll
    for (int m1 = 0; m1 < 4; ++m1) {
        const int row = tile * 128 + 32 * m1 + m0;
        uint32_t v = 0;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
            const int c = step * 4 + kb;
            const uint32_t b = (row < rows && c < nkb) ? scales[(size_t)row * nkb + c] : 127u;
            v |= b << (8 * kb);
        }
        w[m1] = v;
    }
    *reinterpret_cast<uint4 *>(atoms + (size_t)atom * kAtom + m0 * 16) = make_uint4(w[0], w[1], w[2], w[3]);
}

namespace {

constexpr int kMaxCluster = 8;  // K splits of one tile form a cluster (portable size)

struct GateUpArgs {
    const uint8_t *bank, *atoms;  // slot bank; weight atoms of each slot
    size_t expert_bytes, atom_slot_bytes, off_g_codes, off_u_codes, atom_off_g, atom_off_u;
    int H, I, M, KS;
    const int32_t *counts, *act_slot, *act_off, *act_cnt, *hot_token;
    const float *hot_w;
    const uint8_t *xat;  // x atoms [nks][512]
    uint8_t *hq, *hat;   // w*h terms [n_act_cap][64][Ipad], atoms [n_act_cap][nksI][512]
    int Ipad;
    int *err;
};

// grid: (active expert, 128-row tile of I, K split), the K splits of a tile being one cluster.
__global__ void __launch_bounds__(kThreads, 1)
    gateup_tc_kernel(const __grid_constant__ CUtensorMap mapG, const __grid_constant__ CUtensorMap mapU,
                     const __grid_constant__ CUtensorMap mapX, GateUpArgs a) {
    constexpr int S = kGateStages;
    constexpr int kB = NBX * 128;
    constexpr uint32_t kTxFull = 2 * kTileATx + kB + 3 * kAtom, kTxTail = kB + 3 * kAtom;
    constexpr int T = kHTerms;
    constexpr int C = 2 * kDecodeMaxTokens;  // accumulator columns: 2 x terms per token
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    __shared__ __align__(8) uint64_t full[S], empty[S], done;
    __shared__ uint32_t tslot;
    __shared__ float s_wtok[kDecodeMaxTokens];  // routing weight of each token routed to this expert, else 0
    __shared__ unsigned s_routed;               // bit t: token t is routed to this expert

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntile = (a.I + 127) / 128;
    const int KS = a.KS;
    const int unit = blockIdx.x / KS, ks = blockIdx.x - unit * KS;
    const int aidx = unit / ntile, tile = unit - aidx * ntile;
    const int nks = (a.H + 127) / 128;
    const int k0 = ks * nks / KS, k1 = (ks + 1) * nks / KS, nsteps = k1 - k0;
    const bool ragged = (a.H % 128) != 0;
    const int row0 = tile * 128;

    // setup that does not read the route kernel's results overlaps its tail
    if (warp == 1) tmem_alloc(&tslot, kGateTmem);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        fence_barrier_init();
        tma_prefetch_desc(&mapG);
        tma_prefetch_desc(&mapU);
        tma_prefetch_desc(&mapX);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tslot;
    pdl_wait();  // routing and x terms are complete
    pdl_trigger();
    const int slot = a.act_slot[aidx];  // -1 past the active experts
    if (slot < 0) {  // the whole cluster (one tile) leaves together
        if (warp == 1) tmem_dealloc(tbase, kGateTmem);
        return;
    }
    const uint8_t *expert = a.bank + (size_t)slot * a.expert_bytes;
    const uint8_t *gat = a.atoms + (size_t)slot * a.atom_slot_bytes + a.atom_off_g + (size_t)tile * nks * kAtom;
    const uint8_t *uat = a.atoms + (size_t)slot * a.atom_slot_bytes + a.atom_off_u + (size_t)tile * nks * kAtom;
    // columns: gate accumulators [kAcc][16], up accumulators [kAcc][16], then 12 scale columns per stage
    const uint32_t tDg = tbase, tDu = tbase + kAcc * NBX, tSF = tbase + 2 * kAcc * NBX;

    if (warp == 0) {
        bool ok = true;
        for (int i = 0; i < nsteps && ok; ++i) {
            const int st = i % S, kstep = k0 + i;
            if (lane == 0) ok = mbar_wait(&empty[st], ((i / S) & 1) ^ 1, a.err, kErrEmpty);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            uint8_t *sA = smem + st * kGateStage;
            uint8_t *sAt = sA + 2 * kTileA + kB;
            const bool tail = ragged && kstep == nks - 1;
            if (tail) {  // copied without blocking this warp; completion counted on the stage barrier
                cp_async_tail_tile(sA, expert + a.off_g_codes, a.I, row0, a.H, kstep);
                cp_async_tail_tile(sA + kTileA, expert + a.off_u_codes, a.I, row0, a.H, kstep);
                fence_proxy_async();
                cp_async_arrive(&full[st]);
                __syncwarp();
            }
            if (lane == 0) {
                mbar_expect_tx(&full[st], tail ? kTxTail : kTxFull);
                if (!tail) {
                    tma_load_3d(&mapG, &full[st], sA, kstep * 128, row0, slot);
                    tma_load_3d(&mapU, &full[st], sA + kTileA, kstep * 128, row0, slot);
                }
                tma_load_3d(&mapX, &full[st], sA + 2 * kTileA, kstep * 128, 0, 0);
                bulk_copy(sAt, gat + (size_t)kstep * kAtom, kAtom, &full[st]);
                bulk_copy(sAt + kAtom, uat + (size_t)kstep * kAtom, kAtom, &full[st]);
                bulk_copy(sAt + 2 * kAtom, a.xat + (size_t)kstep * kAtom, kAtom, &full[st]);
            }
            __syncwarp();
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = mx_idesc(kFmtE2M1, kFmtE4M3, NBX);
            unsigned init = 0;  // bit kk: accumulator kk holds a sum
            bool ok = true;
            for (int i = 0; i < nsteps && ok; ++i) {
                const int st = i % S;
                ok = mbar_wait(&full[st], (i / S) & 1, a.err, kErrFull);
                if (!ok) break;
                tc_fence_after();
                uint8_t *sA = smem + st * kGateStage;
                uint8_t *sAt = sA + 2 * kTileA + kB;
                const uint32_t sfg = tSF + 12 * st, sfu = sfg + 4, sfb = sfg + 8;
                atom_to_tmem(sfg, sAt);
                atom_to_tmem(sfu, sAt + kAtom);
                atom_to_tmem(sfb, sAt + 2 * kAtom);
                const uint32_t aG = smem_u32(sA), aU = aG + kTileA, aB = aG + 2 * kTileA;
                const bool tail = ragged && (k0 + i) == nks - 1;
                if (tail) fence_proxy_async();  // the tail tiles came by cp.async
                const int nk = tail ? 2 : 4;
                for (int kk = 0; kk < nk; ++kk) {
                    const int q = kk % kAcc;
                    const uint32_t acc = (init >> q) & 1u;
                    mma_mx(tDg + q * NBX, sw128_desc(aG + kk * 32), sw128_desc(aB + kk * 32), idesc, kk, sfg, sfb,
                           acc);
                    mma_mx(tDu + q * NBX, sw128_desc(aU + kk * 32), sw128_desc(aB + kk * 32), idesc, kk, sfu, sfb,
                           acc);
                    init |= 1u << q;
                }
                mma_commit(&empty[st]);
            }
            mma_commit(&done);
        }
        __syncwarp();
    } else if (warp == 2) {
        // the epilogue's routing data, fetched while the weights stream
        if (lane < kDecodeMaxTokens) s_wtok[lane] = 0.f;
        const int off = a.act_off[aidx], cnt = a.act_cnt[aidx];
        int t = -1;
        float w = 0.f;
        if (lane < cnt) {
            t = a.hot_token[off + lane];
            w = a.hot_w[off + lane];
        }
        __syncwarp();
        if (t >= 0) s_wtok[t] = w;
        const unsigned bits = __reduce_or_sync(0xffffffffu, t >= 0 ? 1u << t : 0u);
        if (lane == 0) s_routed = bits;
    }

    // ---------------- epilogue: every thread owns one row of its CTA's partial ----------------
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int M = a.M;
    float g[C], u[C];
#pragma unroll
    for (int c = 0; c < C; ++c) g[c] = u[c] = 0.f;
    // every lane leaves the wait at its own time: reconverge before the warp-aligned tensor-memory loads
    const bool got = __all_sync(0xffffffffu, mbar_wait(&done, 0, a.err, kErrDone));
    tc_fence_after();
    if (got) {
        // a CTA whose single k-step is a 64-column tail touches only the first two MMA slices
        const int nacc = min(kAcc, (nsteps == 1 && ragged && k0 == nks - 1) ? 2 : 4);
        uint32_t rr[8];
        for (int q = 0; q < nacc; ++q) {
#pragma unroll
            for (int c8 = 0; c8 < C / 8; ++c8) {
                if (8 * c8 < 2 * M) {
                    tmem_ld8_sync(tDg + q * NBX + lane_off + 8 * c8, rr);
#pragma unroll
                    for (int j = 0; j < 8; ++j) g[8 * c8 + j] += __uint_as_float(rr[j]);
                    tmem_ld8_sync(tDu + q * NBX + lane_off + 8 * c8, rr);
#pragma unroll
                    for (int j = 0; j < 8; ++j) u[8 * c8 + j] += __uint_as_float(rr[j]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tbase, kGateTmem);

    // K splits: partials meet in the cluster's shared memory; rank r finishes the 32-row groups
    // r, r + KS, ... and sums the ranks in order 0..KS-1, so the result does not depend on timing.
    int grp = warp;
    float *red = reinterpret_cast<float *>(smem);  // [2][C][128], over the drained pipeline stages
    if (KS > 1) {
        const int rloc = warp * 32 + lane;
#pragma unroll
        for (int c = 0; c < C; ++c)
            if (c < 2 * M) {
                red[c * 128 + rloc] = g[c];
                red[(C + c) * 128 + rloc] = u[c];
            }
        __syncwarp();
        cluster_sync();
        grp = ks + KS * warp;
        if (grp < 4) {
            const int rl = grp * 32 + lane;
#pragma unroll
            for (int c = 0; c < C; ++c) g[c] = u[c] = 0.f;
            for (int r = 0; r < KS; ++r) {
                const uint32_t base = dsmem_addr(red, (uint32_t)r);
                float gv[C], uv[C];
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    gv[c] = uv[c] = 0.f;
                    if (c < 2 * M) {
                        gv[c] = ld_dsmem(base + 4u * (c * 128 + rl));
                        uv[c] = ld_dsmem(base + 4u * ((C + c) * 128 + rl));
                    }
                }
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    g[c] += gv[c];
                    u[c] += uv[c];
                }
            }
        }
    }

    // h = SiLU(g) u for the tokens routed to this expert; w h split into T E4M3 terms per 32-row block
    if (grp < 4) {
        const int row = row0 + grp * 32 + lane;
        const int nksI = (a.I + 127) / 128;
        uint8_t *hq = a.hq + (size_t)aidx * NBH * a.Ipad;
        uint8_t *hat = a.hat + (size_t)aidx * nksI * kAtom;
        const unsigned routed = s_routed;
        float vt[kDecodeMaxTokens];
#pragma unroll
        for (int t = 0; t < kDecodeMaxTokens; ++t) {
            const float gg = g[2 * t] + g[2 * t + 1], uu = u[2 * t] + u[2 * t + 1];
            vt[t] = (routed >> t) & 1u ? s_wtok[t] * (silu(gg) * uu) : 0.f;
        }
        if (row < a.I) {  // whole 32-row groups are in or out (I % 64 == 0)
            const int kblock = row / 32;
#pragma unroll
            for (int t = 0; t < kDecodeMaxTokens; ++t) {
                if (t >= M) break;
                if (!((routed >> t) & 1u)) {  // w h = 0 (warp-uniform): zero codes, the zero block's scale byte
#pragma unroll
                    for (int term = 0; term < T; ++term) {
                        const int n = t * T + term;
                        hq[(size_t)n * a.Ipad + row] = 0;
                        if (lane == 0) hat[(size_t)(kblock / 4) * kAtom + (n & 31) * 16 + (n >> 5) * 4 + (kblock % 4)] = 0;
                    }
                    continue;
                }
                float res = vt[t];
#pragma unroll
                for (int term = 0; term < T; ++term) {
                    uint32_t sb;
                    const uint8_t code = split_term(res, sb);
                    const int n = t * T + term;
                    hq[(size_t)n * a.Ipad + row] = code;
                    // B-operand scale of column n: lane n % 32, column n / 32 of the atom
                    if (lane == 0)
                        hat[(size_t)(kblock / 4) * kAtom + (n & 31) * 16 + (n >> 5) * 4 + (kblock % 4)] = (uint8_t)sb;
                }
            }
        }
    }
    __syncwarp();
    if (KS > 1) cluster_sync();  // no CTA leaves while another still reads its shared memory
}

struct DownArgs {
    const uint8_t *bank, *atoms;
    size_t expert_bytes, atom_slot_bytes, off_d_codes, atom_off_d;
    int H, I, M, KS;
    const int32_t *counts, *act_slot;
    const uint8_t *hat;  // [n_act_cap][nksI][512]
    void *out;
    int out_f32;
    int *err;
};

// grid: (128-row tile of H, K split over the concatenated (active expert, k-step) sequence), the K
// splits of a tile being one cluster.
__global__ void __launch_bounds__(kThreads, 1)
    down_tc_kernel(const __grid_constant__ CUtensorMap mapD, const __grid_constant__ CUtensorMap mapH, DownArgs a) {
    constexpr int S = kDownStages;
    constexpr int NB = NBH;
    constexpr int kB = NB * 128;
    constexpr uint32_t kTxFull = kTileATx + kB + 2 * kAtom, kTxTail = kB + 2 * kAtom;
    constexpr int T = kHTerms;
    constexpr int C = kDecodeMaxTokens * T;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    __shared__ __align__(8) uint64_t full[S], empty[S], done;
    __shared__ uint32_t tslot;
    __shared__ int s_slot[kMaxExperts];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KS = a.KS;
    const int tile = blockIdx.x / KS, ks = blockIdx.x - tile * KS;
    const int nksI = (a.I + 127) / 128;
    const bool ragged = (a.I % 128) != 0;
    const int row0 = tile * 128;
    // The routing (counts, slots) is complete: the gate/up grid waited for it before letting this grid
    // launch.  Only the w*h terms come from the grid right before this one.
    const int n_act = a.counts[2];
    const int total = n_act * nksI;
    const int g0 = ks * total / KS, g1 = (ks + 1) * total / KS, nsteps = g1 - g0;
    for (int i = threadIdx.x; i < n_act; i += kThreads) s_slot[i] = a.act_slot[i];

    if (warp == 1) tmem_alloc(&tslot, kDownTmem);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        fence_barrier_init();
        tma_prefetch_desc(&mapD);
        tma_prefetch_desc(&mapH);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tslot;
    // columns: accumulators [kAcc][32], then 8 scale columns per stage
    const uint32_t tD = tbase, tSF = tbase + kAcc * NB;

    if (warp == 0) {
        // weights of the first stages are fetched before the gate/up grid has finished
        const int npre = nsteps < S ? nsteps : S;
        for (int i = 0; i < npre; ++i) {
            const int g = g0 + i, e = g / nksI, s = g - e * nksI;
            uint8_t *sA = smem + i * kDownStage;
            const int slot = s_slot[e];
            const bool tail = ragged && s == nksI - 1;
            if (tail) {
                cp_async_tail_tile(sA, a.bank + (size_t)slot * a.expert_bytes + a.off_d_codes, a.H, row0, a.I, s);
                fence_proxy_async();
                cp_async_arrive(&full[i]);
                __syncwarp();
            }
            if (lane == 0) {
                mbar_expect_tx(&full[i], tail ? kTxTail : kTxFull);
                if (!tail) tma_load_3d(&mapD, &full[i], sA, s * 128, row0, slot);
                bulk_copy(sA + kTileA + kB,
                          a.atoms + (size_t)slot * a.atom_slot_bytes + a.atom_off_d + ((size_t)tile * nksI + s) * kAtom,
                          kAtom, &full[i]);
            }
            __syncwarp();
        }
        pdl_wait();
        pdl_trigger();
        if (lane == 0)
            for (int i = 0; i < npre; ++i) {
                const int g = g0 + i, e = g / nksI, s = g - e * nksI;
                uint8_t *sA = smem + i * kDownStage;
                tma_load_3d(&mapH, &full[i], sA + kTileA, s * 128, 0, e);
                bulk_copy(sA + kTileA + kB + kAtom, a.hat + ((size_t)e * nksI + s) * kAtom, kAtom, &full[i]);
            }
        __syncwarp();
        bool ok = true;
        for (int i = npre; i < nsteps && ok; ++i) {
            const int st = i % S;
            const int g = g0 + i, e = g / nksI, s = g - e * nksI;
            if (lane == 0) ok = mbar_wait(&empty[st], ((i / S) & 1) ^ 1, a.err, kErrEmpty);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            uint8_t *sA = smem + st * kDownStage;
            uint8_t *sAt = sA + kTileA + kB;
            const int slot = s_slot[e];
            const bool tail = ragged && s == nksI - 1;
            if (tail) {
                cp_async_tail_tile(sA, a.bank + (size_t)slot * a.expert_bytes + a.off_d_codes, a.H, row0, a.I, s);
                fence_proxy_async();
                cp_async_arrive(&full[st]);
                __syncwarp();
            }
            if (lane == 0) {
                mbar_expect_tx(&full[st], tail ? kTxTail : kTxFull);
                if (!tail) tma_load_3d(&mapD, &full[st], sA, s * 128, row0, slot);
                tma_load_3d(&mapH, &full[st], sA + kTileA, s * 128, 0, e);
                bulk_copy(sAt, a.atoms + (size_t)slot * a.atom_slot_bytes + a.atom_off_d +
                                   ((size_t)tile * nksI + s) * kAtom,
                          kAtom, &full[st]);
                bulk_copy(sAt + kAtom, a.hat + ((size_t)e * nksI + s) * kAtom, kAtom, &full[st]);
            }
            __syncwarp();
        }
    } else {
        pdl_wait();  // out may still be read by earlier work in the stream
        pdl_trigger();
        if (warp == 1) {
            if (lane == 0) {
                const uint32_t idesc = mx_idesc(kFmtE2M1, kFmtE4M3, NB);
                unsigned init = 0;  // bit kk: accumulator kk holds a sum
                bool ok = true;
                for (int i = 0; i < nsteps && ok; ++i) {
                    const int st = i % S;
                    ok = mbar_wait(&full[st], (i / S) & 1, a.err, kErrFull);
                    if (!ok) break;
                    tc_fence_after();
                    uint8_t *sA = smem + st * kDownStage;
                    uint8_t *sAt = sA + kTileA + kB;
                    const uint32_t sfa = tSF + 8 * st, sfb = sfa + 4;
                    atom_to_tmem(sfa, sAt);
                    atom_to_tmem(sfb, sAt + kAtom);
                    const int s = (g0 + i) % nksI;
                    const uint32_t aA = smem_u32(sA), aB = aA + kTileA;
                    if (ragged && s == nksI - 1) fence_proxy_async();  // the tail tile came by cp.async
                    const int nk = (ragged && s == nksI - 1) ? 2 : 4;
                    for (int kk = 0; kk < nk; ++kk) {
                        const int q = kk % kAcc;
                        mma_mx(tD + q * NB, sw128_desc(aA + kk * 32), sw128_desc(aB + kk * 32), idesc, kk, sfa, sfb,
                               (init >> q) & 1u);
                        init |= 1u << q;
                    }
                    mma_commit(&empty[st]);
                }
                mma_commit(&done);
            }
            __syncwarp();
        }
    }

    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int rloc = warp * 32 + lane;
    const int M = a.M;
    float d[C];
#pragma unroll
    for (int c = 0; c < C; ++c) d[c] = 0.f;
    // every lane leaves the wait at its own time: reconverge before the warp-aligned tensor-memory loads
    const bool got = __all_sync(0xffffffffu, mbar_wait(&done, 0, a.err, kErrDone));
    tc_fence_after();
    if (got && nsteps > 0) {
        // a CTA whose single k-step is a 64-column tail touches only the first two MMA slices
        const int nacc = min(kAcc, (nsteps == 1 && ragged && g0 % nksI == nksI - 1) ? 2 : 4);
        uint32_t rr[8];
        for (int q = 0; q < nacc; ++q) {
#pragma unroll
            for (int c8 = 0; c8 < C / 8; ++c8) {
                if (8 * c8 < M * T) {
                    tmem_ld8_sync(tD + q * NB + lane_off + 8 * c8, rr);
#pragma unroll
                    for (int j = 0; j < 8; ++j) d[8 * c8 + j] += __uint_as_float(rr[j]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tbase, kDownTmem);

    if (KS == 1) {
        const int row = row0 + rloc;
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
        return;
    }
    // K splits: partials meet in the cluster's shared memory; rank r finishes rows [128 r / KS, 128 (r+1) / KS)
    // of every token, summing ranks 0..KS-1 in order (then the terms), so the result does not depend on timing.
    float *red = reinterpret_cast<float *>(smem);  // [C][128], over the drained pipeline stages
#pragma unroll
    for (int c = 0; c < C; ++c)
        if (c < M * T) red[c * 128 + rloc] = d[c];
    __syncwarp();
    cluster_sync();
    const int r0 = ks * 128 / KS, nrows = (ks + 1) * 128 / KS - r0;
    for (int it = threadIdx.x; it < nrows * M; it += kThreads) {
        const int t = it / nrows, rl = r0 + (it - t * nrows);
        float pv[kMaxCluster][T];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
            if (r < KS) {
                const uint32_t base = dsmem_addr(red, (uint32_t)r);
#pragma unroll
                for (int term = 0; term < T; ++term) pv[r][term] = ld_dsmem(base + 4u * ((t * T + term) * 128 + rl));
            }
        }
        float v = 0.f;
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
            if (r < KS)
#pragma unroll
                for (int term = 0; term < T; ++term) v += pv[r][term];
        const int row = row0 + rl;
        if (row < a.H) {
            if (a.out_f32)
                reinterpret_cast<float *>(a.out)[(size_t)t * a.H + row] = v;
            else
                reinterpret_cast<__nv_bfloat16 *>(a.out)[(size_t)t * a.H + row] = __float2bfloat16_rn(v);
        }
    }
    __syncwarp();
    cluster_sync();  // no CTA leaves while another still reads its shared memory
}

// ------------------------------------------------------------------ one launch for M = 1

constexpr int kFfnThreads = 192;  // warps 0-3: epilogue (TMEM lane quadrant = warp); warp 4: copies; warp 5: MMAs
constexpr int kFfnNB = 16;        // B columns of the down MMA: 8 w*h terms of the one token, 8 zero columns
constexpr int kFfnDownAcc = 8;    // down accumulators (16 columns each) in a ring: a tile's MMAs rarely wait for a drain
constexpr uint32_t kFfnTmem = 256;  // gate/up accumulators and scales in columns 0..127, the down ring in 128..255
constexpr int kErrHReady = 4, kErrAccFull = 5, kErrAccEmpty = 6;

struct FfnArgs {
    const uint8_t *bank, *atoms;
    size_t expert_bytes, atom_slot_bytes, off_g_codes, off_u_codes, off_d_codes, atom_off_g, atom_off_u, atom_off_d;
    int H, I, KS, Ucap;
    const int32_t *counts, *act_slot, *act_off, *act_cnt, *hot_token;
    const float *hot_w;
    const uint8_t *xat;
    float *part;      // [ntH][Ucap][128] down partial of each (active expert, I tile) unit
    int *err;
};

// The whole expert FFN of a one-token decode step in one launch.  grid: (active expert, 128-row tile j of I,
// K split), the K splits of a tile being one cluster.  Each cluster
//   1. computes g, u for its I tile as gate/up does (K split over the CTAs, partials summed in rank order),
//   2. forms h = w SiLU(g) u for the tile's 128 rows in every CTA and splits it into eight E4M3 terms held in
//      shared memory (the B operand of the down MMA, never written to global memory),
//   3. multiplies the tile's column slice of Wd (all H rows, 128 columns) by it: CTA r takes H tiles
//      r, r + KS, ...; its copy warp streams those weight tiles into the pipeline right behind the gate/up
//      tiles (two per stage), so they load while the gate/up MMAs and step 2 run,
//   4. stores a fp32 partial per (unit, H tile); ffn_combine_kernel, launched right behind, sums them.
// Shared memory is the gate/up pipeline's: down tiles use a stage's two A slots and two atom slots; the
// K-split partials, h terms and h atom live in the stages' x-term slots, which down tiles never touch.
__global__ void __launch_bounds__(kFfnThreads, 2)
    ffn_tc_kernel(const __grid_constant__ CUtensorMap mapG, const __grid_constant__ CUtensorMap mapU,
                  const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapD, FfnArgs a) {
    constexpr int S = kGateStages;
    constexpr int kB = NBX * 128;
    constexpr uint32_t kTxFull = 2 * kTileATx + kB + 3 * kAtom, kTxTail = kB + 3 * kAtom;
    constexpr int T = kHTerms;
    constexpr int kAtomSlot = 2 * kTileA + kB;  // first atom slot of a stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    __shared__ __align__(8) uint64_t full[S], empty[S], done, hready, acc_full[kFfnDownAcc], acc_empty[kFfnDownAcc];
    __shared__ uint32_t tslot;
    __shared__ float s_w;
    __shared__ int s_routed;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntile = (a.I + 127) / 128, nks = (a.H + 127) / 128, nksI = ntile, ntH = (a.H + 127) / 128;
    const int KS = a.KS;
    const int unit = blockIdx.x / KS, ks = blockIdx.x - unit * KS;
    const int aidx = unit / ntile, jt = unit - aidx * ntile;
    const int k0 = ks * nks / KS, k1 = (ks + 1) * nks / KS, ngu = k1 - k0;
    const bool raggedH = (a.H % 128) != 0, raggedI = (a.I % 128) != 0;
    const bool tailI = raggedI && jt == nksI - 1;
    const int row0 = jt * 128;
    const int nd = (ntH - ks + KS - 1) / KS;  // H tiles of this CTA: ks, ks + KS, ...
    const int nds = (nd + 1) / 2;             // pipeline stages they take, two tiles each

    uint8_t *red = smem + kTileA * 2;               // stage 0 x-term slot: K-split partials [4][128] fp32
    uint8_t *hB = smem + kGateStage + kTileA * 2;   // stage 1 x-term slot: h terms, 16 rows x 128 bytes
    uint8_t *hAt = smem + 2 * kGateStage + kTileA * 2;  // stage 2 x-term slot: h atom

    if (warp == 5) tmem_alloc(&tslot, kFfnTmem);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        mbar_init(&hready, 128);
        for (int b = 0; b < kFfnDownAcc; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 128);
        }
        fence_barrier_init();
        tma_prefetch_desc(&mapG);
        tma_prefetch_desc(&mapU);
        tma_prefetch_desc(&mapX);
        tma_prefetch_desc(&mapD);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tslot;
    pdl_wait();  // routing and x terms are complete
    pdl_trigger();
    const int slot = a.act_slot[aidx];  // -1 past the active experts
    if (slot < 0) {  // the whole cluster (one unit) leaves together
        __syncthreads();
        if (warp == 5) tmem_dealloc(tbase, kFfnTmem);
        return;
    }
    const uint8_t *expert = a.bank + (size_t)slot * a.expert_bytes;
    const uint8_t *slot_atoms = a.atoms + (size_t)slot * a.atom_slot_bytes;
    const uint8_t *gat = slot_atoms + a.atom_off_g + (size_t)jt * nks * kAtom;
    const uint8_t *uat = slot_atoms + a.atom_off_u + (size_t)jt * nks * kAtom;
    // columns: gate accumulator [16], up accumulator [16], 12 scale columns per stage, the h atom; the ring of
    // down accumulators from column 128
    const uint32_t tDg = tbase, tDu = tbase + NBX, tSF = tbase + 2 * NBX, tHat = tSF + 12 * S, tDown = tbase + 128;

    if (warp == 4) {
        // ---------------- copies ----------------
        bool ok = true;
        auto issue = [&](int i) {
            const int st = i % S;
            if (lane == 0) ok = mbar_wait(&empty[st], ((i / S) & 1) ^ 1, a.err, kErrEmpty);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) return;
            uint8_t *sA = smem + st * kGateStage;
            uint8_t *sAt = sA + kAtomSlot;
            if (i < ngu) {  // gate/up k-step
                const int kstep = k0 + i;
                const bool tail = raggedH && kstep == nks - 1;
                if (tail) {  // copied without blocking this warp; completion counted on the stage barrier
                    cp_async_tail_tile(sA, expert + a.off_g_codes, a.I, row0, a.H, kstep);
                    cp_async_tail_tile(sA + kTileA, expert + a.off_u_codes, a.I, row0, a.H, kstep);
                    fence_proxy_async();
                    cp_async_arrive(&full[st]);
                    __syncwarp();
                }
                if (lane == 0) {
                    mbar_expect_tx(&full[st], tail ? kTxTail : kTxFull);
                    if (!tail) {
                        tma_load_3d(&mapG, &full[st], sA, kstep * 128, row0, slot);
                        tma_load_3d(&mapU, &full[st], sA + kTileA, kstep * 128, row0, slot);
                    }
                    tma_load_3d(&mapX, &full[st], sA + 2 * kTileA, kstep * 128, 0, 0);
                    bulk_copy(sAt, gat + (size_t)kstep * kAtom, kAtom, &full[st]);
                    bulk_copy(sAt + kAtom, uat + (size_t)kstep * kAtom, kAtom, &full[st]);
                    bulk_copy(sAt + 2 * kAtom, a.xat + (size_t)kstep * kAtom, kAtom, &full[st]);
                }
            } else {  // two down tiles: Wd rows of H tile hr, columns of I tile jt
                const int d0 = 2 * (i - ngu), nt = nd - d0 < 2 ? nd - d0 : 2;
                if (tailI) {
                    for (int q = 0; q < nt; ++q)
                        cp_async_tail_tile(sA + q * kTileA, expert + a.off_d_codes, a.H, (ks + KS * (d0 + q)) * 128,
                                           a.I, jt);
                    fence_proxy_async();
                    cp_async_arrive(&full[st]);
                    __syncwarp();
                }
                if (lane == 0) {
                    mbar_expect_tx(&full[st], (uint32_t)nt * ((tailI ? 0u : (uint32_t)kTileATx) + kAtom));
                    for (int q = 0; q < nt; ++q) {
                        const int hr = ks + KS * (d0 + q);
                        if (!tailI) tma_load_3d(&mapD, &full[st], sA + q * kTileA, jt * 128, hr * 128, slot);
                        bulk_copy(sAt + q * kAtom, slot_atoms + a.atom_off_d + ((size_t)hr * nksI + jt) * kAtom, kAtom,
                                  &full[st]);
                    }
                }
            }
            __syncwarp();
        };
        // a stage whose last user was a gate/up step frees without step 2; later ones wait for the down MMAs,
        // which wait for h, which waits for every CTA of the cluster to arrive here
        const int early = ngu + (nds < S ? nds : S);
        for (int i = 0; i < early && ok; ++i) issue(i);
        __syncwarp();
        if (KS > 1) cluster_arrive_relaxed();
        for (int i = early; i < ngu + nds && ok; ++i) issue(i);
        __syncwarp();
        if (KS > 1) {
            cluster_wait();
            cluster_arrive_relaxed();
            cluster_wait();
        }
    } else if (warp == 5) {
        // ---------------- MMAs ----------------
        if (lane == 0) {
            const uint32_t idesc = mx_idesc(kFmtE2M1, kFmtE4M3, NBX);
            bool ok = true;
            for (int i = 0; i < ngu && ok; ++i) {
                const int st = i % S;
                ok = mbar_wait(&full[st], (i / S) & 1, a.err, kErrFull);
                if (!ok) break;
                tc_fence_after();
                uint8_t *sA = smem + st * kGateStage;
                uint8_t *sAt = sA + kAtomSlot;
                const uint32_t sfg = tSF + 12 * st, sfu = sfg + 4, sfb = sfg + 8;
                atom_to_tmem(sfg, sAt);
                atom_to_tmem(sfu, sAt + kAtom);
                atom_to_tmem(sfb, sAt + 2 * kAtom);
                const uint32_t aG = smem_u32(sA), aU = aG + kTileA, aB = aG + 2 * kTileA;
                const int nk = (raggedH && (k0 + i) == nks - 1) ? 2 : 4;
                if (nk == 2) fence_proxy_async();  // the tail tiles came by cp.async
                for (int kk = 0; kk < nk; ++kk) {
                    const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                    mma_mx(tDg, sw128_desc(aG + kk * 32), sw128_desc(aB + kk * 32), idesc, kk, sfg, sfb, acc);
                    mma_mx(tDu, sw128_desc(aU + kk * 32), sw128_desc(aB + kk * 32), idesc, kk, sfu, sfb, acc);
                }
                mma_commit(&empty[st]);
            }
            mma_commit(&done);
        }
        __syncwarp();
        if (KS > 1) cluster_arrive_relaxed();
        if (lane == 0) {
            const uint32_t idesc = mx_idesc(kFmtE2M1, kFmtE4M3, kFfnNB);
            bool ok = mbar_wait(&hready, 0, a.err, kErrHReady);
            tc_fence_after();
            if (ok) atom_to_tmem(tHat, hAt);
            const uint32_t aH = smem_u32(hB);
            for (int ds = 0; ds < nds && ok; ++ds) {
                const int i = ngu + ds, st = i % S;
                ok = mbar_wait(&full[st], (i / S) & 1, a.err, kErrFull);
                if (!ok) break;
                tc_fence_after();
                uint8_t *sA = smem + st * kGateStage;
                const int d0 = 2 * ds, nt = nd - d0 < 2 ? nd - d0 : 2;
                if (tailI) fence_proxy_async();  // the tail tiles came by cp.async
                for (int q = 0; q < nt && ok; ++q) {
                    const int ti = d0 + q, buf = ti % kFfnDownAcc;
                    if (ti >= kFfnDownAcc)
                        ok = mbar_wait(&acc_empty[buf], ((ti / kFfnDownAcc) - 1) & 1, a.err, kErrAccEmpty);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sfa = tSF + 12 * st + 4 * q;
                    atom_to_tmem(sfa, sA + kAtomSlot + q * kAtom);
                    const uint32_t aA = smem_u32(sA + q * kTileA);
                    const int nk = tailI ? 2 : 4;
                    for (int kk = 0; kk < nk; ++kk)
                        mma_mx(tDown + NBX * buf, sw128_desc(aA + kk * 32), sw128_desc(aH + kk * 32), idesc, kk, sfa,
                               tHat, kk > 0 ? 1u : 0u);
                    mma_commit(&acc_full[buf]);
                }
                mma_commit(&empty[st]);
            }
        }
        __syncwarp();
        if (KS > 1) {
            cluster_wait();
            cluster_arrive_relaxed();
            cluster_wait();
        }
    } else {
        // ---------------- epilogue: thread = row rloc of the I tile, then of each H tile ----------------
        const int rloc = threadIdx.x;  // warps 0-3
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        if (threadIdx.x == 0) {  // routing weight of the token for this expert
            const int off = a.act_off[aidx], cnt = a.act_cnt[aidx];
            s_routed = cnt > 0 && a.hot_token[off] == 0;
            s_w = s_routed ? a.hot_w[off] : 0.f;
        }
        float g[2] = {0.f, 0.f}, u[2] = {0.f, 0.f};
        bool got = __all_sync(0xffffffffu, mbar_wait(&done, 0, a.err, kErrDone));
        tc_fence_after();
        if (got) {
            uint32_t rg[8], ru[8];
            tmem_ld8x2_sync(tDg + lane_off, rg, tDu + lane_off, ru);
            g[0] = __uint_as_float(rg[0]);
            g[1] = __uint_as_float(rg[1]);
            u[0] = __uint_as_float(ru[0]);
            u[1] = __uint_as_float(ru[1]);
        }
        tc_fence_before();
        named_barrier(1, 128);  // s_w is set
        if (KS > 1) {
            float *rf = reinterpret_cast<float *>(red);
            rf[0 * 128 + rloc] = g[0];
            rf[1 * 128 + rloc] = g[1];
            rf[2 * 128 + rloc] = u[0];
            rf[3 * 128 + rloc] = u[1];
            __syncwarp();
            cluster_arrive();
            cluster_wait();
            // every rank's four partials are loaded before any is added (one round trip), then summed in rank order
            float pv[kMaxCluster][4];
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r)
                if (r < KS) {
                    const uint32_t base = dsmem_addr(red, (uint32_t)r);
#pragma unroll
                    for (int c = 0; c < 4; ++c) pv[r][c] = ld_dsmem(base + 4u * (c * 128 + rloc));
                }
            g[0] = g[1] = u[0] = u[1] = 0.f;
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r)
                if (r < KS) {
                    g[0] += pv[r][0];
                    g[1] += pv[r][1];
                    u[0] += pv[r][2];
                    u[1] += pv[r][3];
                }
            __syncwarp();
            cluster_arrive();  // done reading the other CTAs' partials (waited for before leaving)
        }
        // h of this row: w SiLU(g) u, split into T E4M3 terms with one scale per 32-row block (= this warp)
        {
            const float gg = g[0] + g[1], uu = u[0] + u[1];
            float res = s_routed ? s_w * (silu(gg) * uu) : 0.f;
#pragma unroll
            for (int term = 0; term < T; ++term) {
                uint32_t sb;
                const uint8_t code = split_term(res, sb);
                st_shared_u8(hB + term * 128 + ((((rloc >> 4) ^ (term & 7)) << 4) | (rloc & 15)), code);
                if (lane == 0) st_shared_u8(hAt + term * 16 + warp, sb);
            }
            if (rloc < (kFfnNB - T) * 8) st_shared_zero16(hB + T * 128 + rloc * 16);  // rows T..15: zero
            if (rloc < 32 - T) st_shared_fill16(hAt + (T + rloc) * 16, 0x7f7f7f7fu);  // their scales: 2^0
            fence_proxy_async();
            mbar_arrive(&hready);
        }
        // down partials of this CTA's H tiles
        float *part = a.part + (size_t)unit * 128;
        for (int ti = 0; ti < nd; ++ti) {
            const int buf = ti % kFfnDownAcc, hr = ks + KS * ti;
            got = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (ti / kFfnDownAcc) & 1, a.err, kErrAccFull));
            tc_fence_after();
            float v = 0.f;
            if (got) {
                uint32_t rr[8];
                tmem_ld8_sync(tDown + NBX * buf + lane_off, rr);
#pragma unroll
                for (int term = 0; term < T; ++term) v += __uint_as_float(rr[term]);
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[buf]);
            part[(size_t)hr * a.Ucap * 128 + rloc] = v;
        }
        __syncwarp();
        if (KS > 1) cluster_wait();  // no CTA leaves while another still reads its shared memory
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) tmem_dealloc(tbase, kFfnTmem);
}

constexpr int kCombineRows = 32;  // output rows per combine CTA; its 4 warps take a quarter of the units each

// out[row] = sum over the units (active expert, I tile), in that order, of the one-launch FFN's partials:
// warp q sums units [q U / 4, (q + 1) U / 4) for 32 rows with every load in flight, then the four sums are
// added in warp order, so the result does not depend on timing or on which slots hold the experts.
// Launched with programmatic serialization after ffn_tc_kernel; with no active unit the output is zero.
__global__ void __launch_bounds__(128) ffn_combine_kernel(const float *part, const int32_t *counts, int ntI, int Ucap,
                                                          int H, void *out, int out_f32) {
    __shared__ float s_sum[4][kCombineRows];
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kCombineRows + lane, hr = row >> 7, rl = row & 127;
    const int U = counts[2] * ntI;
    const int u0 = warp * U / 4, u1 = (warp + 1) * U / 4;
    float v = 0.f;
    if (row < H) {
        const float *p = part + (size_t)hr * Ucap * 128 + rl;
        constexpr int kBatch = 32;
        for (int ub = u0; ub < u1; ub += kBatch) {
            float pv[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) pv[j] = ub + j < u1 ? __ldcg(p + (size_t)(ub + j) * 128) : 0.f;
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (ub + j < u1) v += pv[j];
        }
    }
    s_sum[warp][lane] = v;
    __syncthreads();
    if (warp == 0 && row < H) {
        const float r = ((s_sum[0][lane] + s_sum[1][lane]) + s_sum[2][lane]) + s_sum[3][lane];
        if (out_f32)
            reinterpret_cast<float *>(out)[row] = r;
        else
            reinterpret_cast<__nv_bfloat16 *>(out)[row] = __float2bfloat16_rn(r);
    }
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return ensure_dyn_smem(reinterpret_cast<const void *>(kernel), (size_t)bytes);
}

// Launch with the K splits of a tile as one cluster and programmatic serialization after the previous grid.
template <typename K, typename... Args>
cudaError_t launch_ex_n(K kernel, int grid, int threads, int cluster, int smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    int n = 0;
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster > 1) {
        at[n].id = cudaLaunchAttributeClusterDimension;
        at[n].val.clusterDim.x = cluster;
        at[n].val.clusterDim.y = 1;
        at[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = at;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename K, typename... Args>
cudaError_t launch_ex(K kernel, int grid, int cluster, int smem, cudaStream_t s, Args... args) {
    return launch_ex_n(kernel, grid, kThreads, cluster, smem, s, args...);
}

}  // namespace

int tc_gateup_smem() { return kGateStages * kGateStage + 1024; }
int tc_down_smem() { return kDownStages * kDownStage + 1024; }
int tc_max_splits() { return kMaxCluster; }

TcAtomLayout tc_atom_layout(int H, int I) {
    TcAtomLayout l;
    l.ntI = (I + 127) / 128;
    l.ntH = (H + 127) / 128;
    l.nks = (H + 127) / 128;
    l.nksI = (I + 127) / 128;
    l.off_g = 0;
    l.off_u = (size_t)l.ntI * l.nks * kAtom;
    l.off_d = 2 * l.off_u;
    l.slot_bytes = l.off_d + (size_t)l.ntH * l.nksI * kAtom;
    return l;
}

void launch_build_weight_atoms(const uint8_t *expert, const ExpertGeometry &g, uint8_t *atoms, cudaStream_t s) {
    const TcAtomLayout l = tc_atom_layout(g.H, g.I);
    const int na = l.ntI * l.nks, nd = l.ntH * l.nksI;
    build_weight_atoms_kernel<<<(na + 7) / 8, 256, 0, s>>>(expert + g.off_wg_scales, g.I, g.H / 32, atoms + l.off_g,
                                                           l.ntI, l.nks);
    build_weight_atoms_kernel<<<(na + 7) / 8, 256, 0, s>>>(expert + g.off_wu_scales, g.I, g.H / 32, atoms + l.off_u,
                                                           l.ntI, l.nks);
    build_weight_atoms_kernel<<<(nd + 7) / 8, 256, 0, s>>>(expert + g.off_wd_scales, g.H, g.I / 32, atoms + l.off_d,
                                                           l.ntH, l.nksI);
}

cudaError_t launch_gateup_tc(const TcLaunch &L, cudaStream_t s) {
    const TcAtomLayout l = tc_atom_layout(L.geo.H, L.geo.I);
    GateUpArgs a{};
    a.bank = L.bank;
    a.atoms = L.atoms;
    a.expert_bytes = L.geo.expert_bytes;
    a.atom_slot_bytes = l.slot_bytes;
    a.off_g_codes = L.geo.off_wg_codes;
    a.off_u_codes = L.geo.off_wu_codes;
    a.atom_off_g = l.off_g;
    a.atom_off_u = l.off_u;
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
    a.xat = L.xat;
    a.hq = L.hq;
    a.hat = L.hat;
    a.Ipad = L.Ipad;
    a.err = L.err;
    if (a.KS < 1 || a.KS > kMaxCluster) return cudaErrorInvalidValue;
    const int grid = L.n_act_max * l.ntI * a.KS;
    if (cudaError_t e = set_smem(gateup_tc_kernel, tc_gateup_smem())) return e;
    return launch_ex(gateup_tc_kernel, grid, a.KS, tc_gateup_smem(), s, *L.mapG, *L.mapU, *L.mapX, a);
}

cudaError_t launch_down_tc(const TcLaunch &L, cudaStream_t s) {
    const TcAtomLayout l = tc_atom_layout(L.geo.H, L.geo.I);
    DownArgs a{};
    a.bank = L.bank;
    a.atoms = L.atoms;
    a.expert_bytes = L.geo.expert_bytes;
    a.atom_slot_bytes = l.slot_bytes;
    a.off_d_codes = L.geo.off_wd_codes;
    a.atom_off_d = l.off_d;
    a.H = L.geo.H;
    a.I = L.geo.I;
    a.M = L.M;
    a.KS = L.ks_down;
    a.counts = L.counts;
    a.act_slot = L.act_slot;
    a.hat = L.hat;
    a.out = L.out;
    a.out_f32 = L.out_f32;
    a.err = L.err;
    if (a.KS < 1 || a.KS > kMaxCluster) return cudaErrorInvalidValue;
    const int grid = l.ntH * a.KS;
    if (cudaError_t e = set_smem(down_tc_kernel, tc_down_smem())) return e;
    return launch_ex(down_tc_kernel, grid, a.KS, tc_down_smem(), s, *L.mapD, *L.mapH, a);
}

}  // namespace moe

namespace moe {

cudaError_t launch_ffn_tc(const TcLaunch &L, cudaStream_t s) {
    const TcAtomLayout l = tc_atom_layout(L.geo.H, L.geo.I);
    FfnArgs a{};
    a.bank = L.bank;
    a.atoms = L.atoms;
    a.expert_bytes = L.geo.expert_bytes;
    a.atom_slot_bytes = l.slot_bytes;
    a.off_g_codes = L.geo.off_wg_codes;
    a.off_u_codes = L.geo.off_wu_codes;
    a.off_d_codes = L.geo.off_wd_codes;
    a.atom_off_g = l.off_g;
    a.atom_off_u = l.off_u;
    a.atom_off_d = l.off_d;
    a.H = L.geo.H;
    a.I = L.geo.I;
    a.KS = L.ks_gateup;
    a.Ucap = L.n_act_max * l.ntI;
    a.counts = L.counts;
    a.act_slot = L.act_slot;
    a.act_off = L.act_off;
    a.act_cnt = L.act_cnt;
    a.hot_token = L.hot_token;
    a.hot_w = L.hot_w;
    a.xat = L.xat;
    a.part = L.part;
    a.err = L.err;
    if (L.M != 1 || a.KS < 1 || a.KS > kMaxCluster)
        return cudaErrorInvalidValue;
    const int grid = L.n_act_max * l.ntI * a.KS;
    if (cudaError_t e = set_smem(ffn_tc_kernel, tc_gateup_smem())) return e;
    return launch_ex_n(ffn_tc_kernel, grid, kFfnThreads, a.KS, tc_gateup_smem(), s, *L.mapG, *L.mapU, *L.mapX,
                       *L.mapD, a);
}

cudaError_t launch_ffn_combine(const TcLaunch &L, cudaStream_t s) {
    const TcAtomLayout l = tc_atom_layout(L.geo.H, L.geo.I);
    return launch_ex_n(ffn_combine_kernel, (L.geo.H + kCombineRows - 1) / kCombineRows, 128, 1, 0, s,
                       (const float *)L.part, L.counts, l.ntI, L.n_act_max * l.ntI, L.geo.H, L.out, L.out_f32);
}

}  // namespace moe
