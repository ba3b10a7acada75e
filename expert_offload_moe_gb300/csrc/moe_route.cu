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
#include <climits>

#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSmemRoutes = 1024;
constexpr int kMaxChunks = 16;  // router chunks summed with all loads in flight (H <= 4096)
constexpr size_t kRowTaskSmem = 48 * 1024;  // x of a decode call staged per block by row tasks (M H bf16)

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

// Demand-filled LRU slot table (xinfer docs "How it works", Decode: the routed experts are looked up in a
// per-layer LRU table kept on the GPU, misses get least-recently-used slots, expert ids become slot ids).
// The whole last block runs it once top-k has filled s_hist and before the compaction, which then reads
// the new map from s_e2s.
//   - slots whose expert this step routed (hits) get the step's clock as their stamp;
//   - misses (routed, no slot) are served most routes first, ties to the lower id;
//   - victims are the slots this step did not route: empty first, then oldest stamp, ties to the lower
//     slot; the i-th miss takes the i-th victim, and misses left over stay cold for this step.
// The fills go to a device list that the fill kernel reads.  scr: 3 * kMaxExperts + 2 * kMaxFill ints of
// shared scratch that is dead at this point.
__device__ void lru_table_step(const RouteParams &p, int *s_e2s, const int *s_hist, int *scr) {
    const LruTable &T = p.lru;
    const int E = p.E, S = T.S;
    int *s_s2e = scr, *s_key = scr + kMaxExperts, *s_off = scr + 2 * kMaxExperts;
    int *s_cand = scr + 3 * kMaxExperts, *s_vict = s_cand + kMaxFill;
    __shared__ int s_clock, s_hits, s_elig;
    if (threadIdx.x == 0) {
        s_clock = *T.clock;
        s_hits = 0;
        s_elig = 0;
    }
    for (int e = threadIdx.x; e < E; e += kThreads) {
        const int s = T.e2s[e];  // the previous step's last block wrote it; this launch has not
        s_e2s[e] = s;
        s_off[e] = (s_hist[e] > 0 && s < 0) ? 1 : 0;
    }
    for (int s = threadIdx.x; s < S; s += kThreads) s_s2e[s] = T.s2e[s];
    __syncthreads();
    const int clock = s_clock;
    int hits = 0, elig = 0;
    for (int s = threadIdx.x; s < S; s += kThreads) {
        const int o = s_s2e[s];
        const bool routed = o >= 0 && s_hist[o] > 0;
        if (routed) T.stamp[s] = clock;
        s_key[s] = routed ? INT_MAX : (o < 0 ? -2 : T.stamp[s]);
        hits += routed;
        elig += !routed;
    }
    if (hits) atomicAdd(&s_hits, hits);
    if (elig) atomicAdd(&s_elig, elig);
    const int n_cand = block_scan_array(s_off, E);  // misses, listed by ascending id
    for (int e = threadIdx.x; e < E; e += kThreads)
        if (s_hist[e] > 0 && s_e2s[e] < 0) s_cand[s_off[e]] = e;
    const int n_fill = min(n_cand, s_elig);
    if (n_cand > 0) {
        // victim ranks by (key, slot); only the first n_fill are taken
        for (int s = threadIdx.x; s < S; s += kThreads) {
            const int key = s_key[s];
            if (key == INT_MAX) continue;
            int rank = 0;
            for (int q = 0; q < S && rank < n_fill; ++q) {
                const int kq = s_key[q];
                rank += kq < key || (kq == key && q < s);
            }
            if (rank < n_fill) s_vict[rank] = s;
        }
        __syncthreads();
        // miss ranks by (routes descending, id ascending); the list is in id order
        for (int i = threadIdx.x; i < n_cand; i += kThreads) {
            const int e = s_cand[i], h = s_hist[e];
            int rank = 0;
            for (int j = 0; j < n_cand; ++j) {
                const int hj = s_hist[s_cand[j]];
                rank += hj > h || (hj == h && j < i);
            }
            if (rank >= n_fill) continue;  // stays cold this step
            const int v = s_vict[rank], old = s_s2e[v];
            if (old >= 0) {
                T.e2s[old] = -1;
                s_e2s[old] = -1;
            }
            T.e2s[e] = v;
            s_e2s[e] = v;
            T.s2e[v] = e;
            T.stamp[v] = clock;
            T.fill_expert[rank] = e;
            T.fill_slot[rank] = v;
        }
    }
    if (threadIdx.x == 0) {
        *T.n_fill = n_fill;
        *T.clock = clock + 1;
        T.stats[0] += 1;
        T.stats[1] += (unsigned long long)n_fill;
        T.stats[2] += (unsigned long long)s_hits;
        T.stats[3] += (unsigned long long)(n_cand - n_fill);
    }
    __syncthreads();
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

template <bool kRow>
__global__ void __launch_bounds__(kThreads, kRow ? 1 : 4) route_kernel(RouteParams p) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = p.H, E = p.E, M = p.M, k = p.k;
    __shared__ int s_e2s[kMaxExperts];
    __shared__ float s_bias[kMaxExperts];

    // ---------------- before the previous grid has finished: constant inputs ----
    const int ntask = kRow ? E : E * p.nchunk;  // whole router rows, or 256-column chunks of them
    const int nq = p.xq ? M * (H / 32) : 0;  // x-term tasks, one 32-element block each
    int task = blockIdx.x * kWarps + warp;
    float w8[8];
    float wrow[kRow ? kMaxChunks : 1][8];  // row tasks: the task's whole router row, chunk c in wrow[c]
    if constexpr (kRow) {
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
            const int col = c * kRouteChunk + lane * 8;
            const bool ok = task < E && c < p.nchunk && col < H;
            const float4 a = ok ? __ldg(reinterpret_cast<const float4 *>(p.Wr + (size_t)task * H + col))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 b = ok ? __ldg(reinterpret_cast<const float4 *>(p.Wr + (size_t)task * H + col + 4))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            wrow[c][0] = a.x; wrow[c][1] = a.y; wrow[c][2] = a.z; wrow[c][3] = a.w;
            wrow[c][4] = b.x; wrow[c][5] = b.y; wrow[c][6] = b.z; wrow[c][7] = b.w;
        }
    } else {
        load_router_row(p, task, lane, w8);
    }
    for (int e = threadIdx.x; e < E; e += kThreads) {
        s_e2s[e] = p.all_hot ? e : p.e2s[e];
        s_bias[e] = p.bias ? p.bias[e] : 0.f;
    }
    tc::pdl_wait();
    tc::pdl_trigger();
    extern __shared__ __align__(16) uint16_t s_xrow[];  // row tasks: x [M][H] staged once per block
    if (kRow) {
        for (int i = threadIdx.x; i < M * H / 8; i += kThreads)
            reinterpret_cast<uint4 *>(s_xrow)[i] = __ldg(reinterpret_cast<const uint4 *>(p.x) + i);
        __syncthreads();
    }

    // ---------------- phase 1: partial logits; x terms -----------------------
    for (bool first = true; task < ntask + nq; task += gridDim.x * kWarps, first = false) {
        if (task >= ntask && p.xnv) {
            // NVFP4 one-token decode: x as kNvTerms E2M1 terms, UE4M3 scale per 16 values, term j scaled by
            // G_j = 2^(E0 - 2 j) with 2^E0 <= max|x| / 128 (every block's scale stays below 448 and each term
            // shrinks the residual at least 5-fold, so G never outruns it)
            const int q = task - ntask, b = q;  // M == 1: token 0, 32-value block b
            const uint16_t xb = p.x[b * 32 + lane];
            if (p.xmir) p.xmir[b * 32 + lane] = xb;
            float am = 0.f;
            for (int i = lane; i < H / 8; i += 32) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.x) + i);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    am = fmaxf(am, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xffff0000u))));
            }
            am = tc::warp_max(am);
            const int e0 = am > 0.f ? tc::floor_log2(am) - 7 : 0;
            float res = __uint_as_float((uint32_t)xb << 16);
            const int e = b * 32 + lane, ks = e / 256, kk = (e % 256) / 64, b16 = (e % 64) / 16;
            const size_t row_bytes = (size_t)p.Hpad4 / 2;
            for (int j = 0; j < kNvTerms; ++j) {
                const float G = am > 0.f ? tc::pow2f(e0 - 2 * j) : 0.f;
                uint32_t sb;
                const uint32_t byte = tc::split_term_e2m1(res, G, sb);
                if (!(lane & 1)) p.xq[(size_t)j * row_bytes + e / 2] = (uint8_t)byte;
                if ((lane & 15) == 0) p.xat[(size_t)(ks * 4 + kk) * kTcAtomBytes + j * 16 + b16] = (uint8_t)sb;
                if (b == 0 && lane == 0) p.xg[j] = G;
            }
            continue;
        }
        if (task >= ntask) {
            const int q = task - ntask, nb = H / 32, t = q / nb, b = q - t * nb;
            const uint16_t xb = p.x[(size_t)t * H + b * 32 + lane];
            if (p.xmir) p.xmir[(size_t)t * H + b * 32 + lane] = xb;
            float res = __uint_as_float((uint32_t)xb << 16);
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
        if constexpr (kRow) {  // the logit of expert `task` for every token, summed per lane over the chunks
            float acc[kWarps];
#pragma unroll
            for (int t = 0; t < kWarps; ++t) acc[t] = 0.f;
#pragma unroll
            for (int c = 0; c < kMaxChunks; ++c) {
                const int col = c * kRouteChunk + lane * 8;
                if (c < p.nchunk && col < H) {
#pragma unroll
                    for (int t = 0; t < kWarps; ++t)
                        if (t < M) {
                            const uint4 xv = *reinterpret_cast<const uint4 *>(s_xrow + (size_t)t * H + col);
                            acc[t] = fmaf(bf16_lo(xv.x), wrow[c][0], acc[t]);
                            acc[t] = fmaf(bf16_hi(xv.x), wrow[c][1], acc[t]);
                            acc[t] = fmaf(bf16_lo(xv.y), wrow[c][2], acc[t]);
                            acc[t] = fmaf(bf16_hi(xv.y), wrow[c][3], acc[t]);
                            acc[t] = fmaf(bf16_lo(xv.z), wrow[c][4], acc[t]);
                            acc[t] = fmaf(bf16_hi(xv.z), wrow[c][5], acc[t]);
                            acc[t] = fmaf(bf16_lo(xv.w), wrow[c][6], acc[t]);
                            acc[t] = fmaf(bf16_hi(xv.w), wrow[c][7], acc[t]);
                        }
                }
            }
#pragma unroll
            for (int t = 0; t < kWarps; ++t)
                if (t < M) {
                    const float v = warp_sum(acc[t]);
                    if (lane == 0) p.b.logit_part[(size_t)t * E + task] = v;
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

    if (M <= kWarps && E <= 32 && p.nchunk <= kMaxChunks) {
        // Decode with at most 32 experts: warp t takes token t, lane e expert e.  The logit is summed from
        // the chunk partials in chunk order (all loads first), the k winners are ranked in one pass (ties
        // to the lower id, as the arg-max rounds below), then warp 0 writes the expert lists and the hot
        // routes and warp 1 the cold routes.
        if (warp < M) {
            const int t = warp;
            float v = -INFINITY;
            if (lane < E) {
                float pv[kMaxChunks];
#pragma unroll
                for (int c = 0; c < kMaxChunks; ++c)
                    pv[c] = c < p.nchunk ? __ldcg(p.b.logit_part + ((size_t)c * M + t) * E + lane) : 0.f;
                float a = 0.f;
#pragma unroll
                for (int c = 0; c < kMaxChunks; ++c)
                    if (c < p.nchunk) a += pv[c];
                a += s_bias[lane];
                v = (a != a) ? -INFINITY : a;
            }
            int rank = 0;  // experts that come before this one: larger logit, or equal and lower id
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float o = __shfl_sync(0xffffffffu, v, j);
                rank += (o > v) || (o == v && j < lane);
            }
            if (lane < E && rank < k) {
                s_sel_id[warp][rank] = lane;
                s_sel_l[warp][rank] = v;
            }
            __syncwarp();
            const float lmax = s_sel_l[warp][0];
            const float ej = lane < k ? expf(s_sel_l[warp][lane] - lmax) : 0.f;
            float den = 0.f;
            for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, ej, j);
            if (lane < k) {
                const int id = s_sel_id[warp][lane];
                const float wj = ej / den;
                p.b.topk_ids[(size_t)t * k + lane] = id;
                p.b.topk_w[(size_t)t * k + lane] = wj;
                s_ids[t * k + lane] = id;
                s_w[t * k + lane] = wj;
                atomicAdd(&s_hist[id], 1);
            }
        }
        __syncthreads();
        if (p.lru.S) lru_table_step(p, s_e2s, s_hist, reinterpret_cast<int *>(s_union));
        if (warp == 0) {
            const int e = lane;
            const int hist = e < E ? s_hist[e] : 0;
            const int h = (e < E && s_e2s[e] >= 0) ? hist : 0, act = h > 0;
            int xh = h, xa = act;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int yh = __shfl_up_sync(0xffffffffu, xh, o), ya = __shfl_up_sync(0xffffffffu, xa, o);
                if (lane >= o) {
                    xh += yh;
                    xa += ya;
                }
            }
            if (e < E) p.b.hist[e] = hist;
            if (act) {
                const int oa = xa - 1;
                int pos = xh - h;
                p.b.act_expert[oa] = e;
                p.b.act_slot[oa] = s_e2s[e];
                p.b.act_off[oa] = pos;
                p.b.act_cnt[oa] = h;
                for (int t = 0; t < M; ++t)
                    for (int j = 0; j < k; ++j)
                        if (s_ids[t * k + j] == e) {
                            p.b.hot_expert[pos] = e;
                            p.b.hot_token[pos] = t;
                            p.b.hot_w[pos] = s_w[t * k + j];
                            ++pos;
                        }
            }
            if (lane == 31) {
                p.b.counts[0] = xh;
                p.b.counts[2] = xa;
                p.b.counts[3] = M;
            }
            for (int i = __shfl_sync(0xffffffffu, xa, 31) + lane; i < p.act_pad; i += 32) p.b.act_slot[i] = -1;
        } else if (warp == 1) {
            // cold routes of token `lane`, ascending expert id
            int ce[kMaxTopK];
            float cw[kMaxTopK];
            int n = 0;
            if (lane < M)
                for (int j = 0; j < k; ++j) {
                    const int e = s_ids[lane * k + j];
                    if (s_e2s[e] >= 0) continue;
                    const float wt = s_w[lane * k + j];
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
            if (lane == 31) p.b.counts[1] = x;
        }
        return;
    }

    // Decode (M <= 8): every thread sums chunk partials for some (token, expert) pairs, all loads of a
    // pair issued before the sum (in chunk order), into row t of s_l; warp t then selects from its row.
    const bool rows_by_block = M <= kWarps && p.nchunk <= kMaxChunks;
    if (rows_by_block && kRow) {
        // whole-row logits: one load per (token, expert), all of a thread's loads (up to 16) in flight; the
        // loop runs over tokens and experts directly (a division per element made the code that the
        // finishing block fetches cold larger: 2430 -> 2518 tokens/s at E = 512, M = 8)
        for (int e0 = threadIdx.x; e0 < E; e0 += 2 * kThreads) {
            float lv[kWarps][2];
#pragma unroll
            for (int t = 0; t < kWarps; ++t)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int e = e0 + u * kThreads;
                    lv[t][u] = (t < M && e < E) ? __ldcg(p.b.logit_part + (size_t)t * E + e) : 0.f;
                }
#pragma unroll
            for (int t = 0; t < kWarps; ++t)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int e = e0 + u * kThreads;
                    if (t < M && e < E) {
                        const float v = lv[t][u] + s_bias[e];
                        s_l[t][e] = (v != v) ? -INFINITY : v;
                    }
                }
        }
        __syncthreads();
    } else if (rows_by_block) {
        // two experts of a token per thread and iteration, the loads of both issued before either sum (the
        // loop runs over tokens and experts directly: 866 -> 898 tokens/s at E = 512, M = 1, against a
        // division per element)
        for (int t = 0; t < M; ++t)
            for (int e0 = threadIdx.x; e0 < E; e0 += 2 * kThreads) {
                float pv[2][kMaxChunks];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int e = e0 + u * kThreads;
#pragma unroll
                    for (int c = 0; c < kMaxChunks; ++c)
                        pv[u][c] = (e < E && c < p.nchunk) ? __ldcg(p.b.logit_part + ((size_t)c * M + t) * E + e) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int e = e0 + u * kThreads;
                    if (e >= E) continue;
                    float v = 0.f;
#pragma unroll
                    for (int c = 0; c < kMaxChunks; ++c)
                        if (c < p.nchunk) v += pv[u][c];
                    v += s_bias[e];
                    s_l[t][e] = (v != v) ? -INFINITY : v;  // NaN marks a taken expert below
                }
            }
        __syncthreads();
    }

    if (rows_by_block && E > 32) {
        // Decode with more than 32 experts.  Top-k of token t by warp t: the k-th largest of the 32 lane maxima
        // bounds the k-th largest logit from below, so the k winners are among the logits at or above it (a
        // few more than k, as a rule); those candidates are ranked in one pass of shuffles -- larger first,
        // equal ones by lower id, the order and ties of k arg-max rounds.  With more than 32 candidates (wide
        // ties) the warp takes the k arg-max rounds over its row instead.  The row stays in shared memory and
        // the loops are rolled: this code runs once per launch, in the finishing block, from a cold
        // instruction cache, and its fetch time outweighs the loop overhead.
        constexpr int kPer = kMaxExperts / 32;
        __shared__ float s_cv[kWarps][32];
        __shared__ int s_ce[kWarps][32];
        __shared__ unsigned s_mask[kMaxExperts];  // bit t: token t routed to the expert
        __shared__ int s_tok_cold[kDecodeMaxTokens];
        for (int e = threadIdx.x; e < E; e += kThreads) s_mask[e] = 0u;
        if (threadIdx.x < kDecodeMaxTokens) s_tok_cold[threadIdx.x] = 0;
        __syncthreads();
        for (int t = warp; t < M; t += kWarps) {
            float lm = -INFINITY;
#pragma unroll 4
            for (int i = 0; i < kPer; ++i) {
                const int e = lane + 32 * i;
                lm = fmaxf(lm, e < E ? s_l[t][e] : -INFINITY);
            }
            // (the 32-step shuffle ranks fully unrolled: 839 / 2269 tokens/s at E = 512, M = 1 / 8; by 4: 875 / 2391)
            int r = 0;  // rank of this lane's maximum among the 32 (larger first, ties by lane)
#pragma unroll 4
            for (int j = 0; j < 32; ++j) {
                const float o = __shfl_sync(0xffffffffu, lm, j);
                r += (o > lm) || (o == lm && j < lane);
            }
            const float tau = __shfl_sync(0xffffffffu, lm, __ffs(__ballot_sync(0xffffffffu, r == k - 1)) - 1);
            int c = 0;
#pragma unroll 4
            for (int i = 0; i < kPer; ++i) c += (lane + 32 * i < E) && (s_l[t][lane + 32 * i] >= tau);
            int x = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            const int C = __shfl_sync(0xffffffffu, x, 31);
            if (C <= 32 && tau > -INFINITY) {
                int pos = x - c;
#pragma unroll 4
                for (int i = 0; i < kPer; ++i) {
                    const int e = lane + 32 * i;
                    const float vi = e < E ? s_l[t][e] : -INFINITY;
                    if (vi >= tau && e < E) {
                        s_cv[warp][pos] = vi;
                        s_ce[warp][pos] = e;
                        ++pos;
                    }
                }
                __syncwarp();
                const float cv = lane < C ? s_cv[warp][lane] : -INFINITY;
                const int ce = lane < C ? s_ce[warp][lane] : 0x7fffffff;
                int rk = 0;
#pragma unroll 4
                for (int j = 0; j < 32; ++j) {
                    const float ov = __shfl_sync(0xffffffffu, cv, j);
                    const int oe = __shfl_sync(0xffffffffu, ce, j);
                    rk += (ov > cv) || (ov == cv && oe < ce);
                }
                if (lane < C && rk < k) {
                    s_sel_id[warp][rk] = ce;
                    s_sel_l[warp][rk] = cv;
                }
            } else {
                // k arg-max rounds over the row (larger value, equal values to the lower id); NaN marks taken
                for (int j = 0; j < k; ++j) {
                    float bv = -INFINITY;
                    int be = 0x7fffffff;
                    for (int i = 0; i < kPer; ++i) {
                        const int e = lane + 32 * i;
                        const float vi = e < E ? s_l[t][e] : __int_as_float(0x7fc00000);
                        if (vi == vi && (vi > bv || (vi == bv && e < be))) {
                            bv = vi;
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
                    if (lane == (be & 31)) s_l[t][be] = __int_as_float(0x7fc00000);
                    __syncwarp();
                }
            }
            __syncwarp();
            {
                // softmax over the k selected logits: one exp per lane, the denominator summed in selection order
                const float lmax = s_sel_l[warp][0];
                const float ej = lane < k ? expf(s_sel_l[warp][lane] - lmax) : 0.f;
                float den = 0.f;
                for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, ej, j);
                if (lane < k) {
                    const int id = s_sel_id[warp][lane];
                    const float wj = ej / den;
                    p.b.topk_ids[(size_t)t * k + lane] = id;
                    p.b.topk_w[(size_t)t * k + lane] = wj;
                    s_ids[t * k + lane] = id;
                    s_w[t * k + lane] = wj;
                    atomicAdd(&s_hist[id], 1);
                    atomicOr(&s_mask[id], 1u << t);
                }
            }
            __syncwarp();
        }
        __syncthreads();
        if (p.lru.S) lru_table_step(p, s_e2s, s_hist, reinterpret_cast<int *>(s_union));
        // Lists: hot routes by (expert, token) at the expert's offset (a block scan of the hot counts) plus the
        // number of earlier tokens in its token mask; active experts at their index (a scan of the active
        // flags); cold routes by (token, expert) at the cold routes of earlier tokens plus the token's cold
        // routes to lower ids.
        __shared__ int s_wsum[kWarps][2];
        const int e0 = 2 * threadIdx.x;  // E <= 2 kThreads
        int hc[2], ac[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int e = e0 + u;
            hc[u] = (e < E && s_e2s[e] >= 0) ? s_hist[e] : 0;
            ac[u] = hc[u] > 0;
            if (e < E) p.b.hist[e] = s_hist[e];
        }
        int xh = hc[0] + hc[1], xa = ac[0] + ac[1];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yh = __shfl_up_sync(0xffffffffu, xh, o), ya = __shfl_up_sync(0xffffffffu, xa, o);
            if (lane >= o) {
                xh += yh;
                xa += ya;
            }
        }
        if (lane == 31) {
            s_wsum[warp][0] = xh;
            s_wsum[warp][1] = xa;
        }
        const int nr = M * k, r = threadIdx.x;
        const bool mine = r < nr;
        const int e = mine ? s_ids[r] : 0, t = mine ? r / k : 0;
        const bool hot = mine && s_e2s[e] >= 0;
        if (mine && !hot) atomicAdd(&s_tok_cold[t], 1);
        __syncthreads();
        int oh = 0, oa = 0, n_hot = 0, n_act = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            oh += w < warp ? s_wsum[w][0] : 0;
            oa += w < warp ? s_wsum[w][1] : 0;
            n_hot += s_wsum[w][0];
            n_act += s_wsum[w][1];
        }
        if (e0 < E) {
            s_hot_off[e0] = oh + xh - hc[0] - hc[1];
            s_act_pos[e0] = oa + xa - ac[0] - ac[1];
        }
        if (e0 + 1 < E) {
            s_hot_off[e0 + 1] = oh + xh - hc[1];
            s_act_pos[e0 + 1] = oa + xa - ac[1];
        }
        __syncthreads();
        if (mine) {
            const unsigned below = s_mask[e] & ((1u << t) - 1u);
            if (hot) {
                const int pos = s_hot_off[e] + __popc(below);
                p.b.hot_expert[pos] = e;
                p.b.hot_token[pos] = t;
                p.b.hot_w[pos] = s_w[r];
                if (below == 0u) {  // the expert's first token writes its active entry
                    const int ai = s_act_pos[e];
                    p.b.act_expert[ai] = e;
                    p.b.act_slot[ai] = s_e2s[e];
                    p.b.act_off[ai] = s_hot_off[e];
                    p.b.act_cnt[ai] = s_hist[e];
                }
            } else {
                int pos = 0;
                for (int t2 = 0; t2 < t; ++t2) pos += s_tok_cold[t2];
                for (int j = 0; j < k; ++j) {
                    const int e2 = s_ids[t * k + j];
                    pos += s_e2s[e2] < 0 && e2 < e;
                }
                p.b.cold_token[pos] = t;
                p.b.cold_expert[pos] = e;
                p.b.cold_w[pos] = s_w[r];
            }
        }
        for (int i = n_act + threadIdx.x; i < p.act_pad; i += kThreads) p.b.act_slot[i] = -1;
        if (threadIdx.x == 0) {
            p.b.counts[0] = n_hot;
            p.b.counts[1] = nr - n_hot;
            p.b.counts[2] = n_act;
            p.b.counts[3] = M;
        }
        return;
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
        if (p.lru.S) lru_table_step(p, s_e2s, s_hist, reinterpret_cast<int *>(s_union));
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
            for (int i = __shfl_sync(0xffffffffu, xa, 31) + lane; i < p.act_pad; i += 32) p.b.act_slot[i] = -1;
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
// Block b owns tokens [8 b, 8 b + 8).  The router, transposed once to
// [H][E32] (E rounded up to 32, zero rows), and the block's x rows are
// streamed through shared memory 128 columns at a time as fp32.  Warp w takes
// 16 columns of every chunk; each lane accumulates a tile of 2 tokens x 4
// experts (one 16-byte load of x per token and of the router per column feeds
// 8 FMAs per column), and the 8 warp sums of a (token, expert) are added in
// warp order at the end.  Each block then takes top-k + softmax for its
// tokens (ties to the lower id, as in decode), counts its routes per expert
// and ranks each route among the block's routes to the same expert (token
// order).  The last block to arrive turns the per-block counts into
//   offset(expert) + routes to that expert in earlier blocks,
// writes hist, the active-expert lists and (when asked) the prefill GEMM tile
// plan; a second launch then places every route at that offset plus its rank,
// i.e. the hot list ordered by (expert, token) -- a counting sort.
constexpr int kPfWc = 128;                  // columns per staged chunk
constexpr int kPfWarpCols = kPfWc / kWarps; // columns per warp per chunk
constexpr int kPfXs = kPfWc + 8;            // x row stride in smem (bf16): token rows on distinct banks
constexpr int kPfStages = 4;                // chunks in flight: 3 ahead of the one being summed
static_assert(kPfRouteTok == 8 && kWarps == 8, "lane tile: 4 token pairs x 8 expert quads");

struct PfSmem {
    static constexpr int kWB = kPfWc * 32 * 4;           // bytes of one router chunk [128 columns][32 experts]
    static constexpr int kXB = kPfRouteTok * kPfXs * 2;  // bytes of one x chunk [8 tokens][136] bf16
    static constexpr int kStageB = kWB + kXB;
    static constexpr int kRedB = kWarps * kPfRouteTok * 32 * 4;
    static constexpr int kFixedB = kPfStages * kStageB + kRedB;
    __host__ __device__ static size_t bytes(int E) { return (size_t)kFixedB + (size_t)kPfRouteTok * E * 4; }
};
static_assert(PfSmem::kStageB % 16 == 0 && PfSmem::kWB % 16 == 0, "16-byte copies");

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    const int n = valid ? 16 : 0;  // 0: the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Copies chunk c of expert group eg into a stage: the router block [128 columns][32 experts] of WrT and
// the block's 8 x rows (bf16), zeros past H and M (the router rows past E are zero in WrT).
__device__ __forceinline__ void pf_issue(const RouteParams &p, int t0, int eg, int c, unsigned char *stage) {
    float *sW = reinterpret_cast<float *>(stage);
    uint16_t *sX = reinterpret_cast<uint16_t *>(stage + PfSmem::kWB);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + i * kThreads, row = idx >> 3, f4 = idx & 7;
        const int col = c * kPfWc + row;
        const bool ok = col < p.H;
        cp_async16(sW + idx * 4, p.WrT + (size_t)(ok ? col : 0) * p.E32 + eg * 32 + f4 * 4, ok);
    }
    if (threadIdx.x < kPfRouteTok * (kPfWc / 8)) {
        const int t = threadIdx.x / (kPfWc / 8), c8 = threadIdx.x % (kPfWc / 8);
        const int col = c * kPfWc + c8 * 8;
        const bool ok = t0 + t < p.M && col < p.H;
        cp_async16(sX + t * kPfXs + c8 * 8, p.x + (ok ? (size_t)(t0 + t) * p.H + col : 0), ok);
    }
}

// Exclusive prefix over blocks of cnt[b][e] (row stride E) for every expert, in place; tot[e] = the sum.
// Lanes take experts, warps take contiguous ranges of blocks; the loads of 8 blocks go out before their
// stores (the compiler keeps a load behind a store to the same array).
template <bool kGlobal>
__device__ __forceinline__ int pf_ld(const int *a) {
    if constexpr (kGlobal) return __ldcg(a);  // written by other blocks
    else return *a;
}

template <bool kGlobal>
__device__ void pf_block_prefix(int *cnt, int nblk, int E, int *tot, int (*s_part)[32]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (nblk + kWarps - 1) / kWarps, b0 = min(warp * per, nblk), b1 = min(b0 + per, nblk);
    for (int eb = 0; eb < E; eb += 32) {
        const int e = eb + lane;
        int sum = 0;
        if (e < E)
            for (int bb = b0; bb < b1; bb += 8) {
                int v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = bb + i < b1 ? pf_ld<kGlobal>(cnt + (size_t)(bb + i) * E + e) : 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) sum += v[i];
            }
        s_part[warp][lane] = sum;
        __syncthreads();
        int run = 0, total = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int v = s_part[w][lane];
            run += w < warp ? v : 0;
            total += v;
        }
        if (e < E) {
            for (int bb = b0; bb < b1; bb += 8) {
                int v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = bb + i < b1 ? pf_ld<kGlobal>(cnt + (size_t)(bb + i) * E + e) : 0;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (bb + i < b1) {
                        cnt[(size_t)(bb + i) * E + e] = run;
                        run += v[i];
                    }
            }
            if (warp == 0) tot[e] = total;
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kThreads) route_prefill_kernel(RouteParams p) {
    extern __shared__ __align__(16) unsigned char pf_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int E = p.E, M = p.M, k = p.k;
    const int t0 = blockIdx.x * kPfRouteTok;
    float *sRed = reinterpret_cast<float *>(pf_raw + kPfStages * PfSmem::kStageB);  // [8 warps][8 tokens][32]
    float *sL = sRed + kWarps * kPfRouteTok * 32;                                     // [8][E]
    __shared__ float s_bias[kMaxExperts];
    __shared__ int s_cnt[kMaxExperts];
    __shared__ int s_off[kMaxExperts];
    __shared__ int s_act[kMaxExperts];
    __shared__ int s_ids[kPfRouteTok][kMaxTopK];
    __shared__ int s_sel_id[kWarps][kMaxTopK];
    __shared__ float s_sel_l[kWarps][kMaxTopK];

    const int nc = (p.H + kPfWc - 1) / kPfWc;
    for (int e = threadIdx.x; e < E; e += kThreads) {
        s_bias[e] = p.bias ? p.bias[e] : 0.f;
        s_cnt[e] = 0;
    }
    tc::pdl_wait();
    tc::pdl_trigger();

    // ---------------- logits: 32 experts at a time --------------------------
    const int tg = lane >> 3, eq = lane & 7;  // tokens 2 tg, 2 tg + 1; experts 4 eq .. 4 eq + 3 of the group
    const int neg = (E + 31) / 32;
    for (int eg = 0; eg < neg; ++eg) {
        // one commit group per chunk (empty past the last), so "all but the newest 3" is always chunk c
#pragma unroll
        for (int c = 0; c < kPfStages - 1; ++c) {
            if (c < nc) pf_issue(p, t0, eg, c, pf_raw + c * PfSmem::kStageB);
            cp_async_commit();
        }
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        for (int c = 0; c < nc; ++c) {
            cp_async_wait<kPfStages - 2>();
            __syncthreads();  // chunk c is in smem for every thread; stage (c - 1) % 4 is free
            if (c + kPfStages - 1 < nc)
                pf_issue(p, t0, eg, c + kPfStages - 1, pf_raw + ((c + kPfStages - 1) % kPfStages) * PfSmem::kStageB);
            cp_async_commit();
            const unsigned char *stage = pf_raw + (c % kPfStages) * PfSmem::kStageB;
            const float *w = reinterpret_cast<const float *>(stage) + warp * kPfWarpCols * 32 + eq * 4;
            const uint16_t *xs = reinterpret_cast<const uint16_t *>(stage + PfSmem::kWB) + 2 * tg * kPfXs +
                                 warp * kPfWarpCols;
#pragma unroll
            for (int j = 0; j < kPfWarpCols; j += 4) {
                const uint2 xa = *reinterpret_cast<const uint2 *>(xs + j);
                const uint2 xb = *reinterpret_cast<const uint2 *>(xs + kPfXs + j);
                const float xv0[4] = {bf16_lo(xa.x), bf16_hi(xa.x), bf16_lo(xa.y), bf16_hi(xa.y)};
                const float xv1[4] = {bf16_lo(xb.x), bf16_hi(xb.x), bf16_lo(xb.y), bf16_hi(xb.y)};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 wq = *reinterpret_cast<const float4 *>(w + (j + q) * 32);
                    acc[0][0] = fmaf(xv0[q], wq.x, acc[0][0]);
                    acc[0][1] = fmaf(xv0[q], wq.y, acc[0][1]);
                    acc[0][2] = fmaf(xv0[q], wq.z, acc[0][2]);
                    acc[0][3] = fmaf(xv0[q], wq.w, acc[0][3]);
                    acc[1][0] = fmaf(xv1[q], wq.x, acc[1][0]);
                    acc[1][1] = fmaf(xv1[q], wq.y, acc[1][1]);
                    acc[1][2] = fmaf(xv1[q], wq.z, acc[1][2]);
                    acc[1][3] = fmaf(xv1[q], wq.w, acc[1][3]);
                }
            }
        }
        cp_async_wait<0>();
#pragma unroll
        for (int t = 0; t < 2; ++t)
            *reinterpret_cast<float4 *>(sRed + (warp * kPfRouteTok + 2 * tg + t) * 32 + eq * 4) =
                make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
        __syncthreads();  // also: every stage is idle before the next expert group refills them
        {  // one (token, expert) per thread: the warp sums in warp order, then the bias
            const int tl = warp, e = eg * 32 + lane;
            float v = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < kWarps; ++w2) v += sRed[(w2 * kPfRouteTok + tl) * 32 + lane];
            if (e < E) {
                v += s_bias[e];
                sL[(size_t)tl * E + e] = (v != v) ? -INFINITY : v;  // NaN marks a taken expert below
            }
        }
        __syncthreads();
    }

    // ---------------- top-k + softmax: one token per warp --------------------
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
    for (int q = threadIdx.x; q < kPfRouteTok * k; q += kThreads) {
        const int tl = q / k, j = q - tl * k;
        if (t0 + tl >= M) continue;
        const int e = s_ids[tl][j];
        int n = 0;
        for (int u = 0; u < tl; ++u)
            for (int i = 0; i < k; ++i) n += s_ids[u][i] == e;
        p.b.route_rank[(size_t)(t0 + tl) * k + j] = n;
    }
    for (int e = threadIdx.x; e < E; e += kThreads) p.b.blk_cnt[(size_t)blockIdx.x * E + e] = s_cnt[e];

    // ---------------- arrival: the last block makes the offsets -------------
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

    __shared__ int s_part[kWarps][32];
    const int nblk = gridDim.x, ncnt = nblk * E;
    const bool in_smem = (size_t)ncnt * 4 <= PfSmem::bytes(E);
    int *sc = reinterpret_cast<int *>(pf_raw);  // the chunk buffers are free now
    if (in_smem) {
        for (int i0 = 0; i0 < ncnt; i0 += 8 * kThreads) {
            int v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int idx = i0 + i * kThreads + threadIdx.x;
                v[i] = idx < ncnt ? __ldcg(p.b.blk_cnt + idx) : 0;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int idx = i0 + i * kThreads + threadIdx.x;
                if (idx < ncnt) sc[idx] = v[i];
            }
        }
        __syncthreads();
        pf_block_prefix<false>(sc, nblk, E, s_cnt, s_part);
    } else {
        pf_block_prefix<true>(p.b.blk_cnt, nblk, E, s_cnt, s_part);
    }
    for (int e = threadIdx.x; e < E; e += kThreads) {
        p.b.hist[e] = s_cnt[e];
        s_off[e] = s_cnt[e];
        s_act[e] = s_cnt[e] > 0;
    }
    __syncthreads();
    block_scan_array(s_off, E);
    const int n_act = block_scan_array(s_act, E);
    // block offsets + expert offsets: the hot position of a route is this plus its rank
    for (int i0 = 0; i0 < ncnt; i0 += 8 * kThreads) {
        int v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = i0 + i * kThreads + threadIdx.x;
            v[i] = idx < ncnt ? (in_smem ? sc[idx] : __ldcg(p.b.blk_cnt + idx)) : 0;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = i0 + i * kThreads + threadIdx.x;
            if (idx < ncnt) p.b.blk_cnt[idx] = v[i] + s_off[idx % E];
        }
    }
    for (int e = threadIdx.x; e < E; e += kThreads) {
        if (s_cnt[e] == 0) continue;
        const int a = s_act[e];
        p.b.act_expert[a] = e;
        p.b.act_slot[a] = e;
        p.b.act_off[a] = s_off[e];
        p.b.act_cnt[a] = s_cnt[e];
    }
    const int nr = M * k;

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

// Second prefill routing launch: every route to its hot position (block offset from the first launch
// plus its rank within its block).
__global__ void __launch_bounds__(kThreads) route_scatter_kernel(RouteParams p) {
    const int q = blockIdx.x * kThreads + threadIdx.x;
    if (q >= p.M * p.k) return;
    const int t = q / p.k, e = p.b.topk_ids[q];
    const int pos = p.b.blk_cnt[(size_t)(t / kPfRouteTok) * p.E + e] + p.b.route_rank[q];
    p.b.hot_expert[pos] = e;
    p.b.hot_token[pos] = t;
    p.b.hot_w[pos] = p.b.topk_w[q];
    p.b.route_rank[q] = pos;
}

// Wr [E][H] -> WrT [H][E32] (experts past E are zero rows).
__global__ void router_transpose_kernel(const float *Wr, float *WrT, int E, int H, int E32) {
    const long n = (long)H * E32;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const int col = (int)(i / E32), e = (int)(i - (long)col * E32);
        WrT[i] = e < E ? Wr[(size_t)e * H + col] : 0.f;
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
    const size_t smem = PfSmem::bytes(p.E);
    const bool tiled = p.all_hot && p.M > kDecodeMaxTokens && p.b.blk_cnt && p.b.route_rank && p.WrT;
    if (p.pf_poff && !tiled) return cudaErrorNotSupported;  // only the tiled launch plans the prefill GEMMs
    if (tiled) {
        {
            cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void *>(route_prefill_kernel), smem);
            if (e != cudaSuccess) return e;
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
        cudaError_t e = cudaLaunchKernelEx(&cfg, route_prefill_kernel, p);
        if (e != cudaSuccess) return e;
        route_scatter_kernel<<<(p.M * p.k + kThreads - 1) / kThreads, kThreads, 0, s>>>(p);
        return cudaGetLastError();
    }
    // decode of 4-8 tokens with more than 32 experts: one warp per whole router row, x staged once per block
    // (the last block then reads finished logits instead of summing chunk partials, which grows with M; with
    // fewer tokens the chunk tasks, spread over more SMs, finish sooner)
    RouteParams q = p;
    q.rowtask = !p.all_hot && p.E > 32 && p.M >= 4 && p.M <= kWarps && p.nchunk <= kMaxChunks &&
                (size_t)p.M * p.H * 2 <= kRowTaskSmem;
    const int ntask = (q.rowtask ? p.E : p.E * p.nchunk) + (p.xq ? p.M * (p.H / 32) : 0);
    int grid = (ntask + kWarps - 1) / kWarps;
    grid = grid < 1 ? 1 : (grid > 8 * num_sms ? 8 * num_sms : grid);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = q.rowtask ? (size_t)p.M * p.H * 2 : 0;
    if (q.rowtask) {  // static + dynamic shared memory of the row-task form passes 48 KB
        cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void *>(route_kernel<true>), kRowTaskSmem);
        if (e != cudaSuccess) return e;
    }
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return q.rowtask ? cudaLaunchKernelEx(&cfg, route_kernel<true>, q) : cudaLaunchKernelEx(&cfg, route_kernel<false>, q);
}

cudaError_t launch_router_transpose(const float *Wr, float *WrT, int E, int H, int E32, cudaStream_t s) {
    router_transpose_kernel<<<256, 256, 0, s>>>(Wr, WrT, E, H, E32);
    return cudaGetLastError();
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
