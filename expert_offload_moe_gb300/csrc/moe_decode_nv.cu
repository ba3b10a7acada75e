// One-token decode FFN for NVFP4 experts on the 5th-generation tensor cores.
//
// NVFP4 weights are E2M1 codes with one UE4M3 scale per 16 elements (xinfer docs list NVFP4 checkpoints and
// name "NVFP4 on SM100+" as the case they do not handle).  tcgen05.mma .kind::mxf4nvf4.block_scale
// .scale_vec::4X multiplies packed E2M1 operands and applies per-16 UE4M3 scales of both, so the weights go
// from the slot bytes to the tensor cores unchanged: TMA copies 128 rows x 128 bytes (256 codes) per k-step
// into 128-byte-swizzled K-major shared memory, the MMA reads them with 64 codes (32 bytes) per instruction.
//
// The other operand must be E2M1 too.  Each activation vector is split into kNvTerms E2M1 terms: term j has
// one UE4M3 scale per 16 values (the smallest >= the block's largest residual / 6) times a power of two G_j
// shared by the whole vector, and takes the residual's value rounded to the E2M1 grid.  Every term shrinks
// a block's largest residual at least 5-fold, so sixteen terms reproduce a bf16 x exactly and an fp32 h
// to far below fp32 rounding, block by block.  Term j is B column j (M = 1, N = 16); the accumulator column
// j is multiplied by G_j when it is read.  x terms come from the route launch; h terms are formed here.
//
// Scales travel as 512-byte atoms, one per MMA (64 K elements): for a 128-row operand, byte m0*16 + m1*4 + b
// is the scale of row 32 m1 + m0 and 16-element block b; for the B operand (16 columns), byte n*16 + b.  An
// atom is moved to tensor memory by tcgen05.cp; every MMA's scales start on a 4-column boundary.
//
// ffn_nv_kernel  one CTA per (active expert, 128-row tile j of I, K split), the K splits of a unit forming
//                one cluster: gate/up of the tile (partials summed in rank order through distributed shared
//                memory), h = w SiLU(g) u, its kNvTerms terms in shared memory, then the tile's column slice
//                of Wd into fp32 partials per (unit, H tile) that ffn_combine_kernel sums in a fixed order.
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kThreads = 192;        // warps 0-3: epilogue (TMEM lane quadrant = warp); warp 4: copies; warp 5: MMAs
constexpr int T = kNvTerms;          // B columns: the terms of the one token
constexpr int kTile = 128 * 128;     // 128 rows x 128 bytes (256 packed codes) of one operand, in smem and in DRAM
constexpr int kXTile = T * 128;      // x terms of one k-step
constexpr int kAtom = kTcAtomBytes;
constexpr int kStages = 2;
// stage: [gate tile][up tile][x terms][atoms: gate 4, up 4, x 4]; down stages use the two tile slots (a 64-byte
// box each, rows padded to 128 bytes by the swizzle) and the first four atom slots
constexpr int kStage = 2 * kTile + kXTile + 12 * kAtom;  // 40 KB
static_assert(kStage % 1024 == 0, "stage alignment");
constexpr uint32_t kTmemCols = 256;  // accumulators 2 x 16, scales 48 per stage, h scales 8
constexpr int kMaxCluster = 8;
constexpr int kErrFull = 1, kErrEmpty = 2, kErrDone = 3, kErrHReady = 4, kErrAccFull = 5, kErrAccEmpty = 6;

// idesc: E2M1 x E2M1 (format 1 in the .kind::mxf4nvf4 table), UE4M3 scales (bit 23 clear), M = 128, N = 16
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void mma_nv(uint32_t tD, uint64_t adesc, uint64_t bdesc, uint32_t tSFA, uint32_t tSFB,
                                       uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %5, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%6], p; }" ::"r"(tD),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(tSFA), "r"(accumulate), "r"(tSFB)
        : "memory");
}

__device__ __forceinline__ void tmem_ld16_sync(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

}  // namespace

// UE4M3 scale atoms of one slot (built when an expert lands in it): gate and up [ntI][nks4][kk 0..3], down
// [ntH][ntI][kk 0..1]; scales of rows or blocks past the matrix are 1.0 (0x38).  One warp per atom.
__global__ void __launch_bounds__(256) build_weight_atoms_nv_kernel(const uint8_t *scales, int rows, int ncols16,
                                                                    uint8_t *atoms, int ntile, int nsteps, int nkk,
                                                                    int cols_per_step16) {
    const int atom = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (atom >= ntile * nsteps * nkk) return;
    const int tile = atom / (nsteps * nkk), rest = atom - tile * nsteps * nkk, step = rest / nkk, kk = rest - step * nkk;
    const int m0 = threadIdx.x & 31;
    uint32_t w[4];
#pragma unroll
    for (int m1 = 0; m1 < 4; ++m1) {
        const int row = tile * 128 + 32 * m1 + m0;
        uint32_t v = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int c = step * cols_per_step16 + kk * 4 + b;
            const uint32_t s = (row < rows && c < ncols16) ? scales[(size_t)row * ncols16 + c] : 0x38u;
            v |= s << (8 * b);
        }
        w[m1] = v;
    }
    *reinterpret_cast<uint4 *>(atoms + (size_t)atom * kAtom + m0 * 16) = make_uint4(w[0], w[1], w[2], w[3]);
}

namespace {

struct NvArgs {
    const uint8_t *bank, *atoms;
    size_t expert_bytes, atom_slot_bytes, atom_off_g, atom_off_u, atom_off_d;
    int H, I, KS, Ucap;
    const int32_t *counts, *act_slot, *act_off, *act_cnt, *hot_token;
    const float *hot_w;
    const uint8_t *xat;
    const float *xg;
    float *part;  // [ntH][Ucap][128]
    int *err;
};

// grid: (active expert, 128-row tile j of I, K split), the K splits of a unit being one cluster.
__global__ void __launch_bounds__(kThreads, 2)
    ffn_nv_kernel(const __grid_constant__ CUtensorMap mapG, const __grid_constant__ CUtensorMap mapU,
                  const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapD, NvArgs a) {
    constexpr int S = kStages;
    constexpr uint32_t kTxGU = 2 * kTile + kXTile + 12 * kAtom;
    constexpr uint32_t kTxDownTile = 128 * 64 + 2 * kAtom;  // a 64-byte-wide box of 128 rows + its two atoms
    constexpr int kAt = 2 * kTile + kXTile;                  // first atom slot of a stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    __shared__ __align__(8) uint64_t full[S], empty[S], done, hready, acc_full[2], acc_empty[2];
    __shared__ uint32_t tslot;
    __shared__ float s_w, s_xg[T], s_wmax[4];
    __shared__ int s_routed;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntI = (a.I + 127) / 128, ntH = (a.H + 127) / 128, nks = (a.H + 255) / 256;
    const int KS = a.KS;
    const int unit = blockIdx.x / KS, ks = blockIdx.x - unit * KS;
    const int aidx = unit / ntI, jt = unit - aidx * ntI;
    const int k0 = ks * nks / KS, k1 = (ks + 1) * nks / KS, ngu = k1 - k0;
    const int row0 = jt * 128;
    const int nd = (ntH - ks + KS - 1) / KS;  // H tiles of this CTA: ks, ks + KS, ...
    const int nds = (nd + 1) / 2;             // stages they take, two tiles each

    uint8_t *red = smem + 2 * kTile;                 // stage 0 x-term slot: K-split partials [2][128] fp32
    uint8_t *hAt = smem + 2 * kTile + 1024;          // stage 0 x-term slot, second half: h atoms [2][512]
    uint8_t *hB = smem + kStage + 2 * kTile;         // stage 1 x-term slot: h terms, 16 rows x 128 bytes

    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tslot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        mbar_init(&hready, 128);
        for (int b = 0; b < 2; ++b) {
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
        if (warp == 5) tmem_dealloc(tbase, kTmemCols);
        return;
    }
    const uint8_t *slot_atoms = a.atoms + (size_t)slot * a.atom_slot_bytes;
    const uint8_t *gat = slot_atoms + a.atom_off_g + (size_t)jt * nks * 4 * kAtom;
    const uint8_t *uat = slot_atoms + a.atom_off_u + (size_t)jt * nks * 4 * kAtom;
    // columns: gate accumulator [16], up accumulator [16] (then the two down accumulators), 48 scale columns per
    // stage (gate 16, up 16, x 16; a down stage uses the first 16), h scales [8]
    const uint32_t tDg = tbase, tDu = tbase + 16, tSF = tbase + 32, tHat = tSF + 48 * S;

    if (warp == 4) {
        // ---------------- copies ----------------
        bool ok = true;
        auto issue = [&](int i) {
            const int st = i % S;
            if (lane == 0) ok = mbar_wait(&empty[st], ((i / S) & 1) ^ 1, a.err, kErrEmpty);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) return;
            uint8_t *sA = smem + st * kStage;
            uint8_t *sAt = sA + kAt;
            if (lane == 0) {
                if (i < ngu) {  // gate/up k-step (the last one ragged: the box past the matrix is zero-filled)
                    const int kstep = k0 + i;
                    mbar_expect_tx(&full[st], kTxGU);
                    tma_load_3d(&mapG, &full[st], sA, kstep * 128, row0, slot);
                    tma_load_3d(&mapU, &full[st], sA + kTile, kstep * 128, row0, slot);
                    tma_load_3d(&mapX, &full[st], sA + 2 * kTile, kstep * 128, 0, 0);
                    bulk_copy(sAt, gat + (size_t)kstep * 4 * kAtom, 4 * kAtom, &full[st]);
                    bulk_copy(sAt + 4 * kAtom, uat + (size_t)kstep * 4 * kAtom, 4 * kAtom, &full[st]);
                    bulk_copy(sAt + 8 * kAtom, a.xat + (size_t)kstep * 4 * kAtom, 4 * kAtom, &full[st]);
                } else {  // two down tiles: Wd rows of H tile hr, the 128 columns of I tile jt (64 bytes)
                    const int d0 = 2 * (i - ngu), nt = nd - d0 < 2 ? nd - d0 : 2;
                    mbar_expect_tx(&full[st], (uint32_t)nt * kTxDownTile);
                    for (int q = 0; q < nt; ++q) {
                        const int hr = ks + KS * (d0 + q);
                        tma_load_3d(&mapD, &full[st], sA + q * kTile, jt * 64, hr * 128, slot);
                        bulk_copy(sAt + 2 * q * kAtom, slot_atoms + a.atom_off_d + ((size_t)hr * ntI + jt) * 2 * kAtom,
                                  2 * kAtom, &full[st]);
                    }
                }
            }
            __syncwarp();
        };
        // a stage whose last user was a gate/up step frees without the h hand-off; later ones wait for the down
        // MMAs, which wait for h, which waits for every CTA of the cluster to arrive here
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
            bool ok = true;
            for (int i = 0; i < ngu && ok; ++i) {
                const int st = i % S;
                ok = mbar_wait(&full[st], (i / S) & 1, a.err, kErrFull);
                if (!ok) break;
                tc_fence_after();
                uint8_t *sA = smem + st * kStage;
                uint8_t *sAt = sA + kAt;
                const uint32_t sfg = tSF + 48 * st, sfu = sfg + 16, sfx = sfg + 32;
                for (int kk = 0; kk < 4; ++kk) {
                    atom_to_tmem(sfg + 4 * kk, sAt + kk * kAtom);
                    atom_to_tmem(sfu + 4 * kk, sAt + (4 + kk) * kAtom);
                    atom_to_tmem(sfx + 4 * kk, sAt + (8 + kk) * kAtom);
                }
                const uint32_t aG = smem_u32(sA), aU = aG + kTile, aX = aG + 2 * kTile;
                const int nk = (k0 + i == nks - 1 && (a.H % 256)) ? ((a.H % 256) + 63) / 64 : 4;
                for (int kk = 0; kk < nk; ++kk) {
                    const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                    mma_nv(tDg, sw128_desc(aG + kk * 32), sw128_desc(aX + kk * 32), sfg + 4 * kk, sfx + 4 * kk, acc);
                    mma_nv(tDu, sw128_desc(aU + kk * 32), sw128_desc(aX + kk * 32), sfu + 4 * kk, sfx + 4 * kk, acc);
                }
                mma_commit(&empty[st]);
            }
            mma_commit(&done);
        }
        __syncwarp();
        if (KS > 1) cluster_arrive_relaxed();
        if (lane == 0) {
            bool ok = mbar_wait(&hready, 0, a.err, kErrHReady);
            tc_fence_after();
            if (ok) {
                atom_to_tmem(tHat, hAt);
                atom_to_tmem(tHat + 4, hAt + kAtom);
            }
            const uint32_t aH = smem_u32(hB);
            for (int ds = 0; ds < nds && ok; ++ds) {
                const int i = ngu + ds, st = i % S;
                ok = mbar_wait(&full[st], (i / S) & 1, a.err, kErrFull);
                if (!ok) break;
                tc_fence_after();
                uint8_t *sA = smem + st * kStage;
                const int d0 = 2 * ds, nt = nd - d0 < 2 ? nd - d0 : 2;
                for (int q = 0; q < nt && ok; ++q) {
                    const int ti = d0 + q, buf = ti & 1;
                    if (ti >= 2) ok = mbar_wait(&acc_empty[buf], ((ti >> 1) - 1) & 1, a.err, kErrAccEmpty);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sfa = tSF + 48 * st + 8 * q;
                    atom_to_tmem(sfa, sA + kAt + 2 * q * kAtom);
                    atom_to_tmem(sfa + 4, sA + kAt + (2 * q + 1) * kAtom);
                    const uint32_t aA = smem_u32(sA + q * kTile);
                    for (int kk = 0; kk < 2; ++kk)
                        mma_nv(tbase + 16 * buf, sw128_desc(aA + kk * 32), sw128_desc(aH + kk * 32), sfa + 4 * kk,
                               tHat + 4 * kk, kk > 0 ? 1u : 0u);
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
        if (threadIdx.x < T) s_xg[threadIdx.x] = a.xg[threadIdx.x];
        float g = 0.f, u = 0.f;
        bool got = __all_sync(0xffffffffu, mbar_wait(&done, 0, a.err, kErrDone));
        tc_fence_after();
        named_barrier(1, 128);  // s_w, s_xg are set
        if (got) {
            float v[16];
            tmem_ld16_sync(tDg + lane_off, v);
#pragma unroll
            for (int j = 0; j < T; ++j) g += s_xg[j] * v[j];
            tmem_ld16_sync(tDu + lane_off, v);
#pragma unroll
            for (int j = 0; j < T; ++j) u += s_xg[j] * v[j];
        }
        tc_fence_before();
        if (KS > 1) {
            float *rf = reinterpret_cast<float *>(red);
            rf[rloc] = g;
            rf[128 + rloc] = u;
            __syncwarp();
            cluster_arrive();
            cluster_wait();
            // every rank's partials are loaded before any is added (one round trip), then summed in rank order
            float pv[kMaxCluster][2];
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r)
                if (r < KS) {
                    const uint32_t base = dsmem_addr(red, (uint32_t)r);
                    pv[r][0] = ld_dsmem(base + 4u * rloc);
                    pv[r][1] = ld_dsmem(base + 4u * (128 + rloc));
                }
            g = u = 0.f;
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r)
                if (r < KS) {
                    g += pv[r][0];
                    u += pv[r][1];
                }
            __syncwarp();
            cluster_arrive();  // done reading the other CTAs' partials (waited for before leaving)
        }
        // h of this row: w SiLU(g) u; its terms with G_j = 2^(E0 - 2 j), 2^E0 <= max|h| / 128 over the tile
        float res = s_routed ? s_w * (silu(g) * u) : 0.f;
        const float wm = warp_max(fabsf(res));
        if (lane == 0) s_wmax[warp] = wm;
        named_barrier(1, 128);
        const float hmax = fmaxf(fmaxf(s_wmax[0], s_wmax[1]), fmaxf(s_wmax[2], s_wmax[3]));
        const int e0 = hmax > 0.f ? floor_log2(hmax) - 7 : 0;
        float hg[T];
        for (int j = 0; j < T; ++j) {
            const float G = hmax > 0.f ? pow2f(e0 - 2 * j) : 0.f;
            hg[j] = G;
            uint32_t sb;
            const uint32_t byte = split_term_e2m1(res, G, sb);
            // term j = B row j; K element rloc at byte rloc / 2 of the row, 16-byte chunk rloc / 32 swizzled
            if (!(lane & 1))
                st_shared_u8(hB + j * 128 + ((((rloc >> 5) ^ (j & 7)) << 4) | ((rloc >> 1) & 15)), byte);
            // scale of term j, 16-row block rloc / 16: atom rloc / 64, byte j * 16 + block % 4
            if ((lane & 15) == 0) st_shared_u8(hAt + (rloc >> 6) * kAtom + j * 16 + ((rloc >> 4) & 3), sb);
        }
        // the rest of every h row (K elements 128..255) is never read; the atoms' other bytes: 1.0
        for (int o = rloc; o < 2 * kAtom; o += 128) {
            const int n = (o & (kAtom - 1)) >> 4, b = o & 15;
            if (n >= T || b >= 4) st_shared_u8(hAt + o, 0x38u);
        }
        fence_proxy_async();
        mbar_arrive(&hready);
        // down partials of this CTA's H tiles: sum over the terms of G_j times accumulator column j
        float *part = a.part + (size_t)unit * 128;
        for (int ti = 0; ti < nd; ++ti) {
            const int buf = ti & 1, hr = ks + KS * ti;
            got = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (ti >> 1) & 1, a.err, kErrAccFull));
            tc_fence_after();
            float y = 0.f;
            if (got) {
                float v[16];
                tmem_ld16_sync(tbase + 16 * buf + lane_off, v);
#pragma unroll
                for (int j = 0; j < T; ++j) y += hg[j] * v[j];
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[buf]);
            part[(size_t)hr * a.Ucap * 128 + rloc] = y;
        }
        __syncwarp();
        if (KS > 1) cluster_wait();  // no CTA leaves while another still reads its shared memory
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

NvAtomLayout nv_atom_layout(int H, int I) {
    NvAtomLayout l;
    l.ntI = (I + 127) / 128;
    l.ntH = (H + 127) / 128;
    l.nks4 = (H + 255) / 256;
    l.off_g = 0;
    l.off_u = (size_t)l.ntI * l.nks4 * 4 * kAtom;
    l.off_d = 2 * l.off_u;
    l.slot_bytes = l.off_d + (size_t)l.ntH * l.ntI * 2 * kAtom;
    return l;
}

int nv_ffn_smem() { return kStages * kStage + 1024; }

void launch_build_weight_atoms_nv(const uint8_t *expert, const ExpertGeometry &g, uint8_t *atoms, cudaStream_t s) {
    const NvAtomLayout l = nv_atom_layout(g.H, g.I);
    const int ngu = l.ntI * l.nks4 * 4, nd = l.ntH * l.ntI * 2;
    build_weight_atoms_nv_kernel<<<(ngu + 7) / 8, 256, 0, s>>>(expert + g.off_wg_scales, g.I, g.H / 16,
                                                               atoms + l.off_g, l.ntI, l.nks4, 4, 16);
    build_weight_atoms_nv_kernel<<<(ngu + 7) / 8, 256, 0, s>>>(expert + g.off_wu_scales, g.I, g.H / 16,
                                                               atoms + l.off_u, l.ntI, l.nks4, 4, 16);
    build_weight_atoms_nv_kernel<<<(nd + 7) / 8, 256, 0, s>>>(expert + g.off_wd_scales, g.H, g.I / 16,
                                                              atoms + l.off_d, l.ntH, l.ntI, 2, 8);
}

cudaError_t launch_ffn_nv(const NvLaunch &L, cudaStream_t s) {
    const NvAtomLayout l = nv_atom_layout(L.geo.H, L.geo.I);
    NvArgs a{};
    a.bank = L.bank;
    a.atoms = L.atoms;
    a.expert_bytes = L.geo.expert_bytes;
    a.atom_slot_bytes = l.slot_bytes;
    a.atom_off_g = l.off_g;
    a.atom_off_u = l.off_u;
    a.atom_off_d = l.off_d;
    a.H = L.geo.H;
    a.I = L.geo.I;
    a.KS = L.ks;
    a.Ucap = L.n_act_max * l.ntI;
    a.counts = L.counts;
    a.act_slot = L.act_slot;
    a.act_off = L.act_off;
    a.act_cnt = L.act_cnt;
    a.hot_token = L.hot_token;
    a.hot_w = L.hot_w;
    a.xat = L.xat;
    a.xg = L.xg;
    a.part = L.part;
    a.err = L.err;
    if (a.KS < 1 || a.KS > kMaxCluster) return cudaErrorInvalidValue;
    if (cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void *>(ffn_nv_kernel), (size_t)nv_ffn_smem())) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(L.n_act_max * l.ntI * a.KS);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = nv_ffn_smem();
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    int n = 0;
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (a.KS > 1) {
        at[n].id = cudaLaunchAttributeClusterDimension;
        at[n].val.clusterDim.x = a.KS;
        at[n].val.clusterDim.y = 1;
        at[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = at;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, ffn_nv_kernel, *L.mapG, *L.mapU, *L.mapX, *L.mapD, a);
}

}  // namespace moe
