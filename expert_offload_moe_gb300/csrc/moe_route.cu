// Router GEMV, top-k + softmax, and slot compaction in one launch.
//
// Phase 1 (every block): one warp per (expert row, 256-column chunk) of the
// router: 128-bit loads of Wr and x, fp32 products, warp-shuffle sum, partial
// logits written to scratch.  The grid spans E x ceil(H/256) warp tasks, so
// the router is read by many thread blocks at once (NInfer-Offload v0.4.0:
// routing no longer runs in a single thread block).
//
// Phase 2 (the last block to arrive, found with a grid arrival counter; no
// block ever waits for another): per token, the partials are summed in chunk
// order, the bias added, the top-k taken by warp-shuffle arg-max rounds (ties
// to the lower expert id), and the softmax taken over the selected logits.
// Then the routes are split by expert_to_slot (onnxruntime PR #33976:
// slot < 0 is cold) and compacted with block-level prefix scans:
//   hot routes  ordered by (expert, token), grouped per active expert
//   cold routes ordered by (token, expert)
// All counts stay in device memory so the launch shape never depends on the
// routing (xinfer docs "How it works": fixed launch shapes, miss count in
// device memory, decode inside CUDA graphs).
//
// For the tensor-core decode path the same launch also writes the x terms:
// extra warp tasks split each 32-element block of x exactly into two E4M3
// terms with one E8M0 scale (the B operand of the gate/up MMAs).
//
// The kernel is launched with programmatic serialization: the router weights,
// bias and expert_to_slot map are read before it waits for the previous grid
// in the stream, x and all outputs after.
#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSmemRoutes = 1024;
constexpr int kMaxChunks = 16;  // router chunks summed with all loads in flight (H <= 4096)

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Exclusive scan of one int per thread across the block; returns the
// exclusive prefix and writes the block total to *total.
__device__ int block_scan_exclusive(int v, int *total) {
    __shared__ int warp_tot[kWarps];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[w] = x;
    __syncthreads();
    if (w == 0) {
        int t = lane < kWarps ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < kWarps; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < kWarps) warp_tot[lane] = t;
    }
    __syncthreads();
    const int base = w ? warp_tot[w - 1] : 0;
    *total = warp_tot[kWarps - 1];
    __syncthreads();
    return base + x - v;
}

// Exclusive scan in place over a[0..n) (shared memory), chunked per thread.
__device__ int block_scan_array(int *a, int n) {
    const int per = (n + kThreads - 1) / kThreads;
    const int lo = min((int)threadIdx.x * per, n), hi = min(lo + per, n);
    int s = 0;
    for (int i = lo; i < hi; ++i) s += a[i];
    int total;
    int run = block_scan_exclusive(s, &total);
    for (int i = lo; i < hi; ++i) {
        int v = a[i];
        a[i] = run;
        run += v;
    }
    __syncthreads();
    return total;
}

__device__ __forceinline__ void load_router_row(const RouteParams &p, int task, int lane, float (&w8)[8]) {
    const int e = task / p.nchunk, c = task - e * p.nchunk;
    const int col = c * kRouteChunk + lane * 8;
    if (task < p.E * p.nchunk && col < p.H) {  // H % 64 == 0, so a valid lane has all 8 columns
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p.Wr + (size_t)e * p.H + col));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p.Wr + (size_t)e * p.H + col + 4));
        w8[0] = a.x; w8[1] = a.y; w8[2] = a.z; w8[3] = a.w;
        w8[4] = b.x; w8[5] = b.y; w8[6] = b.z; w8[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w8[i] = 0.f;
    }
}

__global__ void __launch_bounds__(kThreads) route_kernel(RouteParams p) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = p.H, E = p.E, M = p.M, k = p.k;
    __shared__ int s_e2s[kMaxExperts];
    __shared__ float s_bias[kMaxExperts];

    // ---------------- before the previous grid has finished: constant inputs ----
    const int ntask = E * p.nchunk;
    const int nq = p.xq ? M * (H / 32) : 0;  // x-term tasks, one 32-element block each
    int task = blockIdx.x * kWarps + warp;
    float w8[8];
    load_router_row(p, task, lane, w8);
    for (int e = threadIdx.x; e < E; e += kThreads) {
        s_e2s[e] = p.all_hot ? e : p.e2s[e];
        s_bias[e] = p.bias ? p.bias[e] : 0.f;
    }
    tc::pdl_wait();
    tc::pdl_trigger();

    // ---------------- phase 1: partial logits; x terms -----------------------
    for (bool first = true; task < ntask + nq; task += gridDim.x * kWarps, first = false) {
        if (task >= ntask) {
            const int q = task - ntask, nb = H / 32, t = q / nb, b = q - t * nb;
            float res = __uint_as_float((uint32_t)p.x[(size_t)t * H + b * 32 + lane] << 16);
#pragma unroll
            for (int term = 0; term < 2; ++term) {
                uint32_t sb;
                const uint8_t code = tc::split_term(res, sb);
                const int n = t * 2 + term;
                p.xq[(size_t)n * p.Hpad + b * 32 + lane] = code;
                if (lane == 0) p.xat[(size_t)(b / 4) * kTcAtomBytes + n * 16 + (b % 4)] = (uint8_t)sb;
            }
            continue;
        }
        if (!first) load_router_row(p, task, lane, w8);
        const int e = task / p.nchunk, c = task - e * p.nchunk;
        const int col = c * kRouteChunk + lane * 8;
        const bool valid = col < H;
        for (int t = 0; t < M; ++t) {
            float acc = 0.f;
            if (valid) {
                const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)t * H + col));
                acc = fmaf(bf16_lo(xv.x), w8[0], acc);
                acc = fmaf(bf16_hi(xv.x), w8[1], acc);
                acc = fmaf(bf16_lo(xv.y), w8[2], acc);
                acc = fmaf(bf16_hi(xv.y), w8[3], acc);
                acc = fmaf(bf16_lo(xv.z), w8[4], acc);
                acc = fmaf(bf16_hi(xv.z), w8[5], acc);
                acc = fmaf(bf16_lo(xv.w), w8[6], acc);
                acc = fmaf(bf16_hi(xv.w), w8[7], acc);
            }
            acc = warp_sum(acc);
            if (lane == 0) p.b.logit_part[((size_t)c * M + t) * E + e] = acc;
        }
    }

    // ---------------- arrival: the last block continues --------------------
    // bar.sync orders the block's writes before thread 0's release; its acquire orders the
    // finishing block's reads after every other block's writes.
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned prev;
        asm volatile("atom.acq_rel.gpu.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(p.b.arrive) : "memory");
        s_last = prev == gridDim.x - 1;
        if (s_last) *p.b.arrive = 0u;  // every block has arrived: ready for the next launch
    }
    __syncthreads();
    if (!s_last) return;

    // ---------------- phase 2a: top-k + softmax per token -------------------
    // logits rows (top-k) and the per-token cold counts (compaction) are never live together
    __shared__ __align__(16) float s_union[kWarps * kMaxExperts > kMaxTokens ? kWarps * kMaxExperts : kMaxTokens];
    float(*s_l)[kMaxExperts] = reinterpret_cast<float(*)[kMaxExperts]>(s_union);
    int *s_cold = reinterpret_cast<int *>(s_union);
    __shared__ int s_hist[kMaxExperts];
    __shared__ int s_hot_off[kMaxExperts];
    __shared__ int s_act_pos[kMaxExperts];
    __shared__ int s_ids[kSmemRoutes];  // copy of the routes for the compaction when they fit
    __shared__ float s_w[kSmemRoutes];
    __shared__ int s_sel_id[kWarps][kMaxTopK];
    __shared__ float s_sel_l[kWarps][kMaxTopK];
    const bool routes_in_smem = M * k <= kSmemRoutes;
    int *ids = routes_in_smem ? s_ids : p.b.topk_ids;
    float *wts = routes_in_smem ? s_w : p.b.topk_w;

    for (int e = threadIdx.x; e < E; e += kThreads) s_hist[e] = 0;
    __syncthreads();

    // Decode (M <= 8): every thread sums chunk partials for some (token, expert) pairs, all loads of a
    // pair issued before the sum (in chunk order), into row t of s_l; warp t then selects from its row.
    const bool rows_by_block = M <= kWarps && p.nchunk <= kMaxChunks;
    if (rows_by_block) {
        for (int q = threadIdx.x; q < M * E; q += kThreads) {
            const int t = q / E, e = q - t * E;
            float pv[kMaxChunks];
#pragma unroll
            for (int c = 0; c < kMaxChunks; ++c)
                pv[c] = c < p.nchunk ? __ldcg(p.b.logit_part + ((size_t)c * M + t) * E + e) : 0.f;
            float v = 0.f;
#pragma unroll
            for (int c = 0; c < kMaxChunks; ++c)
                if (c < p.nchunk) v += pv[c];
            v += s_bias[e];
            s_l[t][e] = (v != v) ? -INFINITY : v;  // NaN marks a taken expert below
        }
        __syncthreads();
    }

    for (int t = warp; t < M; t += kWarps) {
        if (!rows_by_block) {
            for (int e = lane; e < E; e += 32) {
                float v = 0.f;
                for (int c = 0; c < p.nchunk; ++c) v += __ldcg(p.b.logit_part + ((size_t)c * M + t) * E + e);
                v += s_bias[e];
                s_l[warp][e] = (v != v) ? -INFINITY : v;
            }
        }
        __syncwarp();
        // k arg-max rounds (ties to the lower id); the taken expert is marked NaN in the row
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int be = 0x7fffffff;
            for (int e = lane; e < E; e += 32) {
                const float v = s_l[warp][e];
                if (v != v) continue;  // taken
                if (v > bv || (v == bv && e < be)) {
                    bv = v;
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (ov > bv || (ov == bv && oe < be)) {
                    bv = ov;
                    be = oe;
                }
            }
            // E >= k and no stored value is NaN, so a candidate always exists: be < E
            if (lane == 0) {
                s_sel_id[warp][j] = be;
                s_sel_l[warp][j] = bv;
            }
            if (lane == (be & 31)) s_l[warp][be] = __int_as_float(0x7fc00000);
            __syncwarp();
        }
        // softmax over the k selected logits, the denominator summed in selection order
        if (lane < k) {
            const float lmax = s_sel_l[warp][0];
            float den = 0.f;
            for (int j = 0; j < k; ++j) den += expf(s_sel_l[warp][j] - lmax);
            const int id = s_sel_id[warp][lane];
            const float wj = expf(s_sel_l[warp][lane] - lmax) / den;
            p.b.topk_ids[(size_t)t * k + lane] = id;
            p.b.topk_w[(size_t)t * k + lane] = wj;
            if (routes_in_smem) {
                s_ids[t * k + lane] = id;
                s_w[t * k + lane] = wj;
            }
            atomicAdd(&s_hist[id], 1);
        }
        __syncwarp();
    }
    __syncthreads();

    if (M <= kWarps) {
        // Decode: warp 0 scans the experts (each lane a run of consecutive ids), warp 1 the tokens.
        __shared__ int s_n[3];
        if (warp == 0) {
            const int per = (E + 31) / 32, e0 = min(lane * per, E), e1 = min(e0 + per, E);
            int nh = 0, na = 0;
            for (int e = e0; e < e1; ++e) {
                const int h = s_e2s[e] >= 0 ? s_hist[e] : 0;
                nh += h;
                na += h > 0;
            }
            int xh = nh, xa = na;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int yh = __shfl_up_sync(0xffffffffu, xh, o), ya = __shfl_up_sync(0xffffffffu, xa, o);
                if (lane >= o) {
                    xh += yh;
                    xa += ya;
                }
            }
            int oh = xh - nh, oa = xa - na;
            for (int e = e0; e < e1; ++e) {
                p.b.hist[e] = s_hist[e];
                const int h = s_e2s[e] >= 0 ? s_hist[e] : 0;
                s_hot_off[e] = oh;
                if (h > 0) {
                    p.b.act_expert[oa] = e;
                    p.b.act_slot[oa] = s_e2s[e];
                    p.b.act_off[oa] = oh;
                    p.b.act_cnt[oa] = h;
                    ++oa;
                }
                oh += h;
            }
            if (lane == 31) {
                s_n[0] = xh;
                s_n[1] = xa;
            }
        } else if (warp == 1) {
            // cold routes of token `lane`, ascending expert id
            int ce[kMaxTopK];
            float cw[kMaxTopK];
            int n = 0;
            if (lane < M)
                for (int j = 0; j < k; ++j) {
                    const int e = ids[lane * k + j];
                    if (s_e2s[e] >= 0) continue;
                    const float wt = wts[lane * k + j];
                    int q = n++;  // insertion by expert id
                    while (q > 0 && ce[q - 1] > e) {
                        ce[q] = ce[q - 1];
                        cw[q] = cw[q - 1];
                        --q;
                    }
                    ce[q] = e;
                    cw[q] = wt;
                }
            int x = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            const int base = x - n;
            for (int q = 0; q < n; ++q) {
                p.b.cold_token[base + q] = lane;
                p.b.cold_expert[base + q] = ce[q];
                p.b.cold_w[base + q] = cw[q];
            }
            if (lane == 31) s_n[2] = x;
        }
        __syncthreads();
        // hot routes of each active expert in token order
        for (int e = threadIdx.x; e < E; e += kThreads) {
            if (s_e2s[e] < 0 || s_hist[e] == 0) continue;
            int pos = s_hot_off[e];
            for (int t = 0; t < M; ++t)
                for (int j = 0; j < k; ++j)
                    if (ids[t * k + j] == e) {
                        p.b.hot_expert[pos] = e;
                        p.b.hot_token[pos] = t;
                        p.b.hot_w[pos] = wts[t * k + j];
                        ++pos;
                    }
        }
        if (threadIdx.x == 0) {
            p.b.counts[0] = s_n[0];
            p.b.counts[1] = s_n[2];
            p.b.counts[2] = s_n[1];
            p.b.counts[3] = M;
        }
        return;
    }

    // ---------------- phase 2b: compaction ----------------------------------
    for (int e = threadIdx.x; e < E; e += kThreads) {
        const bool hot = s_e2s[e] >= 0;
        s_hot_off[e] = hot ? s_hist[e] : 0;
        s_act_pos[e] = (hot && s_hist[e] > 0) ? 1 : 0;
    }
    __syncthreads();
    const int n_hot = block_scan_array(s_hot_off, E);
    const int n_act = block_scan_array(s_act_pos, E);

    for (int e = threadIdx.x; e < E; e += kThreads) {
        p.b.hist[e] = s_hist[e];
        const bool hot = s_e2s[e] >= 0;
        if (!hot || s_hist[e] == 0) continue;
        const int a = s_act_pos[e];
        int pos = s_hot_off[e];
        p.b.act_expert[a] = e;
        p.b.act_slot[a] = s_e2s[e];
        p.b.act_off[a] = pos;
        p.b.act_cnt[a] = s_hist[e];
        for (int t = 0; t < M; ++t)
            for (int j = 0; j < k; ++j)
                if (ids[t * k + j] == e) {
                    p.b.hot_expert[pos] = e;
                    p.b.hot_token[pos] = t;
                    p.b.hot_w[pos] = wts[t * k + j];
                    ++pos;
                }
    }

    // cold routes: per token, ascending expert
    for (int t = threadIdx.x; t < M; t += kThreads) {
        int n = 0;
        if (!p.all_hot)
            for (int j = 0; j < k; ++j) n += s_e2s[ids[t * k + j]] < 0;
        s_cold[t] = n;
    }
    __syncthreads();
    const int n_cold = block_scan_array(s_cold, M);
    if (!p.all_hot) {
        for (int t = threadIdx.x; t < M; t += kThreads) {
            int ce[kMaxTopK];
            float cw[kMaxTopK];
            int n = 0;
            for (int j = 0; j < k; ++j) {
                const int e = ids[t * k + j];
                if (s_e2s[e] >= 0) continue;
                const float wt = wts[t * k + j];
                int q = n++;  // insertion by expert id
                while (q > 0 && ce[q - 1] > e) {
                    ce[q] = ce[q - 1];
                    cw[q] = cw[q - 1];
                    --q;
                }
                ce[q] = e;
                cw[q] = wt;
            }
            const int base = s_cold[t];
            for (int q = 0; q < n; ++q) {
                p.b.cold_token[base + q] = t;
                p.b.cold_expert[base + q] = ce[q];
                p.b.cold_w[base + q] = cw[q];
            }
        }
    }
    if (threadIdx.x == 0) {
        p.b.counts[0] = n_hot;
        p.b.counts[1] = n_cold;
        p.b.counts[2] = n_act;
        p.b.counts[3] = M;
    }
}

// ---------------------------------------------------------------------------
// Prefill routing (M > 8; every expert is hot, slot = expert id).
//
// Block b owns tokens [16 b, 16 b + 16).  It stages its 16 rows of x in shared
// memory and streams the router through shared memory 128 columns x 32
// experts at a time (transposed so lane e reads expert e without bank
// conflicts); warp w accumulates 4 tokens x 32 experts over one half of each
// 128-column chunk, and the two halves are added at the end.  Each block then
// takes top-k + softmax for its tokens (ties to the lower id, as in decode),
// counts its routes per expert and ranks each route among the block's routes
// to the same expert (token order).  The last block to arrive turns the
// per-block counts into offsets and scatters every route to
//   hot position = offset(expert) + routes to that expert in earlier blocks + rank,
// i.e. the hot list ordered by (expert, token) -- a counting sort with no
// serial pass over the routes.
constexpr int kPfWc = 128;  // router columns per staged chunk
constexpr int kPfTokWarp = 4;

struct PfSmem {
    static size_t bytes(int H, int E) {
        return (size_t)kPfRouteTok * H * 2 + 2 * kPfWc * 32 * 4 + kPfRouteTok * 32 * 4 + (size_t)kPfRouteTok * E * 4;
    }
};

__device__ __forceinline__ void pf_load_w(const RouteParams &p, int eg, int c, float4 (&r)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + i * kThreads, el = idx & 31, cg = idx >> 5;
        const int e = eg * 32 + el, col = c * kPfWc + cg * 4;
        r[i] = (e < p.E && col < p.H) ? __ldg(reinterpret_cast<const float4 *>(p.Wr + (size_t)e * p.H + col))
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

__device__ __forceinline__ void pf_store_w(float *sW, const float4 (&r)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + i * kThreads, el = idx & 31, cg = idx >> 5;
        sW[(cg * 4 + 0) * 32 + el] = r[i].x;
        sW[(cg * 4 + 1) * 32 + el] = r[i].y;
        sW[(cg * 4 + 2) * 32 + el] = r[i].z;
        sW[(cg * 4 + 3) * 32 + el] = r[i].w;
    }
}

__global__ void __launch_bounds__(kThreads, 1) route_prefill_kernel(RouteParams p) {
    extern __shared__ __align__(16) unsigned char pf_smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = p.H, E = p.E, M = p.M, k = p.k;
    const int t0 = blockIdx.x * kPfRouteTok;
    uint16_t *sX = reinterpret_cast<uint16_t *>(pf_smem);                       // [16][H]
    float *sW = reinterpret_cast<float *>(pf_smem + (size_t)kPfRouteTok * H * 2);  // [2][128][32]
    float *sRed = sW + 2 * kPfWc * 32;                                           // [16][32]
    float *sL = sRed + kPfRouteTok * 32;                                         // [16][E]
    __shared__ float s_bias[kMaxExperts];
    __shared__ int s_cnt[kMaxExperts];
    __shared__ int s_off[kMaxExperts];
    __shared__ int s_act[kMaxExperts];
    __shared__ int s_ids[kPfRouteTok][kMaxTopK];
    __shared__ int s_sel_id[kWarps][kMaxTopK];
    __shared__ float s_sel_l[kWarps][kMaxTopK];

    const int nc = (H + kPfWc - 1) / kPfWc;
    float4 wr[4];
    pf_load_w(p, 0, 0, wr);  // the router is constant: read before waiting for the previous grid
    for (int e = threadIdx.x; e < E; e += kThreads) {
        s_bias[e] = p.bias ? p.bias[e] : 0.f;
        s_cnt[e] = 0;
    }
    tc::pdl_wait();
    tc::pdl_trigger();

    // x rows of the block (zeros past M)
    const int hv = H / 8;
    for (int q = threadIdx.x; q < kPfRouteTok * hv; q += kThreads) {
        const int t = q / hv, c8 = q - t * hv;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (t0 + t < M) v = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)(t0 + t) * H) + c8);
        reinterpret_cast<uint4 *>(sX + (size_t)t * H)[c8] = v;
    }

    // ---------------- logits: 32 experts at a time --------------------------
    const int g = warp & 3, hh = warp >> 2;
    const int neg = (E + 31) / 32;
    for (int eg = 0; eg < neg; ++eg) {
        if (eg > 0) pf_load_w(p, eg, 0, wr);
        pf_store_w(sW, wr);
        __syncthreads();
        float acc[kPfTokWarp] = {0.f, 0.f, 0.f, 0.f};
        for (int c = 0; c < nc; ++c) {
            if (c + 1 < nc) pf_load_w(p, eg, c + 1, wr);
            const float *w = sW + (c & 1) * kPfWc * 32;
            const int col0 = c * kPfWc + hh * (kPfWc / 2);
            if (col0 < H) {  // H % 64 == 0: a half chunk is all valid or all past H
#pragma unroll 2
                for (int j = 0; j < kPfWc / 2; j += 8) {
                    float wv[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) wv[q] = w[(hh * (kPfWc / 2) + j + q) * 32 + lane];
#pragma unroll
                    for (int t = 0; t < kPfTokWarp; ++t) {
                        const uint4 xv = *reinterpret_cast<const uint4 *>(sX + (size_t)(g * kPfTokWarp + t) * H + col0 + j);
                        float a = acc[t];
                        a = fmaf(bf16_lo(xv.x), wv[0], a);
                        a = fmaf(bf16_hi(xv.x), wv[1], a);
                        a = fmaf(bf16_lo(xv.y), wv[2], a);
                        a = fmaf(bf16_hi(xv.y), wv[3], a);
                        a = fmaf(bf16_lo(xv.z), wv[4], a);
                        a = fmaf(bf16_hi(xv.z), wv[5], a);
                        a = fmaf(bf16_lo(xv.w), wv[6], a);
                        a = fmaf(bf16_hi(xv.w), wv[7], a);
                        acc[t] = a;
                    }
                }
            }
            if (c + 1 < nc) pf_store_w(sW + ((c + 1) & 1) * kPfWc * 32, wr);
            __syncthreads();
        }
        if (hh == 1)
#pragma unroll
            for (int t = 0; t < kPfTokWarp; ++t) sRed[(g * kPfTokWarp + t) * 32 + lane] = acc[t];
        __syncthreads();
        const int e = eg * 32 + lane;
        if (hh == 0 && e < E)
#pragma unroll
            for (int t = 0; t < kPfTokWarp; ++t) {
                const float v = acc[t] + sRed[(g * kPfTokWarp + t) * 32 + lane] + s_bias[e];
                sL[(size_t)(g * kPfTokWarp + t) * E + e] = (v != v) ? -INFINITY : v;  // NaN marks a taken expert
            }
        __syncthreads();
    }

    // ---------------- top-k + softmax: two tokens per warp -------------------
    for (int tl = warp; tl < kPfRouteTok; tl += kWarps) {
        const int t = t0 + tl;
        if (t >= M) continue;  // warp-uniform
        float *row = sL + (size_t)tl * E;
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int be = 0x7fffffff;
            for (int e = lane; e < E; e += 32) {
                const float v = row[e];
                if (v != v) continue;
                if (v > bv || (v == bv && e < be)) {
                    bv = v;
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (ov > bv || (ov == bv && oe < be)) {
                    bv = ov;
                    be = oe;
                }
            }
            if (lane == 0) {
                s_sel_id[warp][j] = be;
                s_sel_l[warp][j] = bv;
            }
            if (lane == (be & 31)) row[be] = __int_as_float(0x7fc00000);
            __syncwarp();
        }
        if (lane < k) {
            const float lmax = s_sel_l[warp][0];
            float den = 0.f;
            for (int j = 0; j < k; ++j) den += expf(s_sel_l[warp][j] - lmax);
            const int id = s_sel_id[warp][lane];
            p.b.topk_ids[(size_t)t * k + lane] = id;
            p.b.topk_w[(size_t)t * k + lane] = expf(s_sel_l[warp][lane] - lmax) / den;
            s_ids[tl][lane] = id;
            atomicAdd(&s_cnt[id], 1);
        }
        __syncwarp();
    }
    __syncthreads();
    // rank of each route among the block's earlier tokens routed to the same expert
    for (int r = threadIdx.x; r < kPfRouteTok * k; r += kThreads) {
        const int tl = r / k, j = r - tl * k;
        if (t0 + tl >= M) continue;
        const int e = s_ids[tl][j];
        int n = 0;
        for (int u = 0; u < tl; ++u)
            for (int i = 0; i < k; ++i) n += s_ids[u][i] == e;
        p.b.route_rank[(size_t)(t0 + tl) * k + j] = n;
    }
    for (int e = threadIdx.x; e < E; e += kThreads) p.b.blk_cnt[(size_t)blockIdx.x * E + e] = s_cnt[e];

    // ---------------- arrival: the last block scatters ----------------------
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned prev;
        asm volatile("atom.acq_rel.gpu.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(p.b.arrive) : "memory");
        s_last = prev == gridDim.x - 1;
        if (s_last) *p.b.arrive = 0u;
    }
    __syncthreads();
    if (!s_last) return;

    // per expert: exclusive prefix of the block counts (in place), tpe lanes per expert
    const int nblk = gridDim.x;
    int tpe = 1;  // a power of two <= 32, so an expert's lanes never straddle a warp
    while (tpe < 32 && E * tpe * 2 <= kThreads) tpe *= 2;
    for (int base = 0; base < E * tpe; base += kThreads) {
        const int q = base + threadIdx.x;
        const int e = q / tpe, part = q - e * tpe;  // tpe consecutive lanes share an expert
        const int per = (nblk + tpe - 1) / tpe, b0 = min(part * per, nblk), b1 = min(b0 + per, nblk);
        int sum = 0;
        if (e < E) {
#pragma unroll 4
            for (int b = b0; b < b1; ++b) sum += __ldcg(p.b.blk_cnt + (size_t)b * E + e);
        }
        int x = sum;  // inclusive scan over the tpe lanes of this expert
        for (int o = 1; o < tpe; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (part >= o) x += y;
        }
        const int total = __shfl_sync(0xffffffffu, x, (lane | (tpe - 1)));
        int run = x - sum;
        if (e < E) {
            for (int b = b0; b < b1; ++b) {
                const int v = __ldcg(p.b.blk_cnt + (size_t)b * E + e);
                p.b.blk_cnt[(size_t)b * E + e] = run;
                run += v;
            }
            if (part == 0) {
                p.b.hist[e] = total;
                s_cnt[e] = total;
            }
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads) {
        s_off[e] = s_cnt[e];
        s_act[e] = s_cnt[e] > 0;
    }
    __syncthreads();
    block_scan_array(s_off, E);
    const int n_act = block_scan_array(s_act, E);
    for (int e = threadIdx.x; e < E; e += kThreads) {
        if (s_cnt[e] == 0) continue;
        const int a = s_act[e];
        p.b.act_expert[a] = e;
        p.b.act_slot[a] = e;
        p.b.act_off[a] = s_off[e];
        p.b.act_cnt[a] = s_cnt[e];
    }
    const int nr = M * k;
#pragma unroll 4
    for (int r = threadIdx.x; r < nr; r += kThreads) {
        const int t = r / k;
        const int e = __ldcg(p.b.topk_ids + r);
        const int pos = s_off[e] + __ldcg(p.b.blk_cnt + (size_t)(t / kPfRouteTok) * E + e) + __ldcg(p.b.route_rank + r);
        p.b.hot_expert[pos] = e;
        p.b.hot_token[pos] = t;
        p.b.hot_w[pos] = __ldcg(p.b.topk_w + r);
        p.b.route_rank[r] = pos;  // only this thread reads or writes entry r
    }

    // tile plan for the grouped GEMMs: each active expert's routes padded to whole 128-row tiles, in
    // expert order (a tile never mixes experts)
    if (p.pf_poff) {
        __shared__ int s_tiles[kMaxExperts];
        for (int e = threadIdx.x; e < E; e += kThreads) s_tiles[e] = (s_cnt[e] + 127) / 128;
        __syncthreads();
        const int total = block_scan_array(s_tiles, E);
        for (int e = threadIdx.x; e < E; e += kThreads) {
            if (s_cnt[e] == 0) {
                p.pf_e2a[e] = -1;
                continue;
            }
            const int a = s_act[e], t0e = s_tiles[e], cnt = s_cnt[e];
            p.pf_e2a[e] = a;
            p.pf_poff[a] = 128 * t0e;
            for (int i = 0; 128 * i < cnt; ++i) {
                if (t0e + i >= p.pf_tiles_cap) break;
                p.pf_tile_aidx[t0e + i] = a;
                p.pf_tile_nrows[t0e + i] = min(128, cnt - 128 * i);
            }
        }
        if (threadIdx.x == 0) *p.pf_ntiles = min(total, p.pf_tiles_cap);
    }
    if (threadIdx.x == 0) {
        p.b.counts[0] = nr;
        p.b.counts[1] = 0;
        p.b.counts[2] = n_act;
        p.b.counts[3] = M;
    }
}

constexpr int kMaxMapUpdates = 64;

struct MapUpdate {
    int n;
    int32_t expert[kMaxMapUpdates];
    int32_t slot[kMaxMapUpdates];
};

__global__ void map_update_kernel(int32_t *e2s, MapUpdate u) {
    if (threadIdx.x == 0)
        for (int i = 0; i < u.n; ++i) e2s[u.expert[i]] = u.slot[i];
}

}  // namespace

cudaError_t launch_route(const RouteParams &p, cudaStream_t s, int num_sms) {
    const size_t smem = PfSmem::bytes(p.H, p.E);
    const bool tiled = p.all_hot && p.M > kDecodeMaxTokens && p.b.blk_cnt && p.b.route_rank && smem <= 200 * 1024;
    if (p.pf_poff && !tiled) return cudaErrorNotSupported;  // only the tiled launch plans the prefill GEMMs
    if (tiled) {
        static size_t smem_set = 0;  // the kernel's dynamic shared memory limit raised so far
        if (smem > smem_set) {
            cudaError_t e = cudaFuncSetAttribute(route_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
            smem_set = smem;
        }
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((p.M + kPfRouteTok - 1) / kPfRouteTok);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, route_prefill_kernel, p);
    }
    const int ntask = p.E * p.nchunk + (p.xq ? p.M * (p.H / 32) : 0);
    int grid = (ntask + kWarps - 1) / kWarps;
    grid = grid < 1 ? 1 : (grid > 8 * num_sms ? 8 * num_sms : grid);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, route_kernel, p);
}

void launch_map_update(int32_t *e2s, int n, const int32_t *experts, const int32_t *slots, cudaStream_t s) {
    MapUpdate u;
    u.n = n < kMaxMapUpdates ? n : kMaxMapUpdates;
    for (int i = 0; i < u.n; ++i) {
        u.expert[i] = experts[i];
        u.slot[i] = slots[i];
    }
    map_update_kernel<<<1, 32, 0, s>>>(e2s, u);
}

}  // namespace moe
