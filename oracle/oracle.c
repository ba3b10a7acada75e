/*
 * oracle.c -- plain, slow, obviously-correct CPU model of the decode-time
 * Mixture-of-Experts layer with GPU expert slots.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library.  The CUDA path
 * never calls it and shares no code, header, table or helper with it.
 *
 * Sources (page title, section):
 *  - xinfer-ai docs/moe_offload.md, "How it works": per-layer GPU slots,
 *    routed expert ids rewritten to slot ids, GEMMs over [num_slots, N, K]
 *    slot tensors; "Placement never changes routing or precision".
 *  - onnxruntime PR #33976 "hybrid GPU/CPU expert offload for MoEPacked",
 *    "Key Changes": expert_to_slot map, slot < 0 = cold, cold routes are
 *    skipped on the GPU and handled elsewhere.
 *  - NInfer-Offload release notes v0.4.0 "expert cache": slots follow recent
 *    routing, at most two refills per layer and call, replacing the least
 *    used expert.
 *  - tinyserve README, "How it works" 2-3: fused dequantise-and-multiply over
 *    the native MXFP4 bytes (gate, up, down), frequency-recency eviction.
 *  - MXFP4 itself (E2M1 elements, one E8M0 scale per 32 elements) is named by
 *    the pages (xinfer "Supported": FusedMoeMxfp4; tinyserve README: native
 *    MXFP4) but not defined there; the OCP Microscaling Formats (MX) v1.0
 *    definition is used.
 *  - NVFP4 is named by the pages (xinfer docs: NVFP4 checkpoints, "NVFP4 on
 *    SM100+" not supported there) but not defined; NVIDIA's block format is
 *    used: the same E2M1 elements with one E4M3 scale per 16 elements.  The
 *    pages give no per-tensor scale, so none is applied (a factor of 1).
 *  - The pages define no router or FFN formula.  The plain reading used here:
 *    logits = x.Wr^T + b; the k largest logits (ties to the lower expert id);
 *    softmax over the k selected logits; expert FFN
 *    y = Wd . (SiLU(Wg . x) * (Wu . x)); output = sum of w * y over the
 *    token's hot routes.
 *
 * Arithmetic: fp32 throughout with sums taken in ascending index order; the
 * products bf16 x E2M1 x 2^k are exact in fp32.  Every function is written
 * for a reader to check by eye, not for speed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- formats */

/* E2M1 element (OCP MX v1.0): sign bit 3, exponent bits 2..1 (bias 1),
 * mantissa bit 0.  Magnitudes of codes 0..7 are listed out in full. */
static const float E2M1_MAGNITUDE[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float oracle_e2m1(uint8_t code) {
    float m = E2M1_MAGNITUDE[code & 7];
    return (code & 8) ? -m : m;
}

/* E8M0 scale (OCP MX v1.0): 2^(e - 127); e = 255 is NaN. */
float oracle_e8m0(uint8_t e) {
    if (e == 255) return NAN;
    return ldexpf(1.0f, (int)e - 127);
}

/* bf16 bit pattern -> fp32 (bf16 is the top half of an fp32). */
float oracle_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16 bit pattern, round to nearest even (NaN kept quiet). */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* One MXFP4 matrix [R, C]: codes [R, C/2] (column 2c in the low nibble of
 * byte c, column 2c+1 in the high nibble), scales [R, C/32]. */
float oracle_mxfp4_element(const uint8_t *codes, const uint8_t *scales, int C, int r, int c) {
    uint8_t byte = codes[(size_t)r * (C / 2) + c / 2];
    uint8_t code = (c & 1) ? (byte >> 4) : (byte & 15);
    uint8_t sc = scales[(size_t)r * (C / 32) + c / 32];
    return oracle_e2m1(code) * oracle_e8m0(sc);
}

/* One NVFP4 matrix [R, C]: codes [R, C/2] as in MXFP4, scales [R, C/16], each
 * an E4M3 byte (oracle_e4m3, below) for 16 consecutive columns. */
float oracle_e4m3(uint8_t code);
float oracle_nvfp4_element(const uint8_t *codes, const uint8_t *scales, int C, int r, int c) {
    uint8_t byte = codes[(size_t)r * (C / 2) + c / 2];
    uint8_t code = (c & 1) ? (byte >> 4) : (byte & 15);
    uint8_t sc = scales[(size_t)r * (C / 16) + c / 16];
    return oracle_e2m1(code) * oracle_e4m3(sc);
}

void oracle_nvfp4_dequant(const uint8_t *codes, const uint8_t *scales, int R, int C, float *W) {
    for (int r = 0; r < R; ++r)
        for (int c = 0; c < C; ++c) W[(size_t)r * C + c] = oracle_nvfp4_element(codes, scales, C, r, c);
}

void oracle_mxfp4_dequant(const uint8_t *codes, const uint8_t *scales, int R, int C, float *W) {
    for (int r = 0; r < R; ++r)
        for (int c = 0; c < C; ++c) W[(size_t)r * C + c] = oracle_mxfp4_element(codes, scales, C, r, c);
}

/* Expert record: [Wg codes, Wg scales, Wu codes, Wu scales, Wd codes, Wd scales].
 * fmt 0 = MXFP4 (a scale per 32 elements), 1 = NVFP4 (a scale per 16). */
static int scale_block(int fmt) { return fmt == 1 ? 16 : 32; }

size_t oracle_expert_bytes_fmt(int H, int I, int fmt) {
    return (size_t)3 * I * H / 2 + (size_t)3 * I * H / scale_block(fmt);
}

size_t oracle_expert_bytes(int H, int I) { return oracle_expert_bytes_fmt(H, I, 0); }

static float element(int fmt, const uint8_t *codes, const uint8_t *scales, int C, int r, int c) {
    return fmt == 1 ? oracle_nvfp4_element(codes, scales, C, r, c) : oracle_mxfp4_element(codes, scales, C, r, c);
}

static void expert_sections(const uint8_t *rec, int H, int I, int fmt, const uint8_t **gc, const uint8_t **gs,
                            const uint8_t **uc, const uint8_t **us, const uint8_t **dc, const uint8_t **ds) {
    size_t c = (size_t)I * H / 2, s = (size_t)I * H / scale_block(fmt);
    *gc = rec;
    *gs = rec + c;
    *uc = rec + c + s;
    *us = rec + 2 * c + s;
    *dc = rec + 2 * c + 2 * s;
    *ds = rec + 3 * c + 2 * s;
}

/* ----------------------------------------------------------------- router */

/* logits[t, e] = sum_h x[t, h] * Wr[e, h] + b[e], fp32, ascending h. */
void oracle_router_logits(const uint16_t *x, int M, int H, const float *Wr, const float *bias, int E,
                          float *logits) {
    for (int t = 0; t < M; ++t)
        for (int e = 0; e < E; ++e) {
            float acc = 0.0f;
            for (int h = 0; h < H; ++h) acc = acc + oracle_bf16_to_f32(x[(size_t)t * H + h]) * Wr[(size_t)e * H + h];
            logits[(size_t)t * E + e] = acc + (bias ? bias[e] : 0.0f);
        }
}

/* The k largest logits of each token, largest first; equal logits go to the
 * lower expert id.  Weights: softmax over the k selected logits (equal to the
 * softmax over all E renormalised to the selected k), max-subtracted, fp32. */
void oracle_topk_softmax(const float *logits, int M, int E, int k, int32_t *ids, float *w) {
    char *taken = (char *)malloc((size_t)E);
    for (int t = 0; t < M; ++t) {
        const float *l = logits + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e; /* strict '>' keeps the lower id on ties */
            }
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
        }
        float lmax = l[ids[(size_t)t * k]];
        float den = 0.0f;
        for (int j = 0; j < k; ++j) den = den + expf(l[ids[(size_t)t * k + j]] - lmax);
        for (int j = 0; j < k; ++j) w[(size_t)t * k + j] = expf(l[ids[(size_t)t * k + j]] - lmax) / den;
    }
    free(taken);
}

/* ------------------------------------------------------------ compaction */

/* Splits the routes by the expert_to_slot map (slot < 0 = cold).
 *  hot:    (expert, slot, token, weight), ordered by (expert, token)
 *  active: one entry per expert with at least one hot route, ascending expert,
 *          with its slot, first hot index and hot count
 *  cold:   (token, expert, weight), ordered by (token, expert)
 *  hist:   all routes (hot and cold) per expert
 * counts[0..2] = n_hot, n_cold, n_active. */
void oracle_compact(const int32_t *ids, const float *w, int M, int k, const int32_t *e2s, int E,
                    int32_t *hot_expert, int32_t *hot_slot, int32_t *hot_token, float *hot_w,
                    int32_t *act_expert, int32_t *act_slot, int32_t *act_off, int32_t *act_cnt,
                    int32_t *cold_token, int32_t *cold_expert, float *cold_w, int32_t *hist,
                    int32_t *counts) {
    int n_hot = 0, n_cold = 0, n_act = 0;
    for (int e = 0; e < E; ++e) hist[e] = 0;
    for (int i = 0; i < M * k; ++i) hist[ids[i]] += 1;
    /* hot routes: experts ascending, tokens ascending inside an expert */
    for (int e = 0; e < E; ++e) {
        if (e2s[e] < 0) continue;
        int first = n_hot;
        for (int t = 0; t < M; ++t)
            for (int j = 0; j < k; ++j)
                if (ids[t * k + j] == e) {
                    hot_expert[n_hot] = e;
                    hot_slot[n_hot] = e2s[e];
                    hot_token[n_hot] = t;
                    hot_w[n_hot] = w[t * k + j];
                    ++n_hot;
                }
        if (n_hot > first) {
            act_expert[n_act] = e;
            act_slot[n_act] = e2s[e];
            act_off[n_act] = first;
            act_cnt[n_act] = n_hot - first;
            ++n_act;
        }
    }
    /* cold routes: tokens ascending, experts ascending inside a token */
    for (int t = 0; t < M; ++t)
        for (int e = 0; e < E; ++e) {
            if (e2s[e] >= 0) continue;
            for (int j = 0; j < k; ++j)
                if (ids[t * k + j] == e) {
                    cold_token[n_cold] = t;
                    cold_expert[n_cold] = e;
                    cold_w[n_cold] = w[t * k + j];
                    ++n_cold;
                }
        }
    counts[0] = n_hot;
    counts[1] = n_cold;
    counts[2] = n_act;
}

/* ------------------------------------------------------------- expert FFN */

static float silu(float g) { return g / (1.0f + expf(-g)); }

/* h[i] = SiLU(sum_c Wg[i,c] x[c]) * (sum_c Wu[i,c] x[c]), fp32, ascending c. */
void oracle_expert_gate_up_fmt(const uint8_t *rec, int H, int I, int fmt, const uint16_t *x, float *h) {
    const uint8_t *gc, *gs, *uc, *us, *dc, *ds;
    expert_sections(rec, H, I, fmt, &gc, &gs, &uc, &us, &dc, &ds);
    for (int i = 0; i < I; ++i) {
        float g = 0.0f, u = 0.0f;
        for (int c = 0; c < H; ++c) {
            float xc = oracle_bf16_to_f32(x[c]);
            g = g + element(fmt, gc, gs, H, i, c) * xc;
            u = u + element(fmt, uc, us, H, i, c) * xc;
        }
        h[i] = silu(g) * u;
    }
}

/* y[r] = sum_i Wd[r,i] h[i], fp32, ascending i. */
void oracle_expert_down_fmt(const uint8_t *rec, int H, int I, int fmt, const float *h, float *y) {
    const uint8_t *gc, *gs, *uc, *us, *dc, *ds;
    expert_sections(rec, H, I, fmt, &gc, &gs, &uc, &us, &dc, &ds);
    for (int r = 0; r < H; ++r) {
        float acc = 0.0f;
        for (int i = 0; i < I; ++i) acc = acc + element(fmt, dc, ds, I, r, i) * h[i];
        y[r] = acc;
    }
}

void oracle_expert_ffn_fmt(const uint8_t *rec, int H, int I, int fmt, const uint16_t *x, float *y) {
    float *h = (float *)malloc(sizeof(float) * (size_t)I);
    oracle_expert_gate_up_fmt(rec, H, I, fmt, x, h);
    oracle_expert_down_fmt(rec, H, I, fmt, h, y);
    free(h);
}

void oracle_expert_gate_up(const uint8_t *rec, int H, int I, const uint16_t *x, float *h) {
    oracle_expert_gate_up_fmt(rec, H, I, 0, x, h);
}

void oracle_expert_down(const uint8_t *rec, int H, int I, const float *h, float *y) {
    oracle_expert_down_fmt(rec, H, I, 0, h, y);
}

void oracle_expert_ffn(const uint8_t *rec, int H, int I, const uint16_t *x, float *y) {
    oracle_expert_ffn_fmt(rec, H, I, 0, x, y);
}

/* ------------------------------------------------------------ whole layer */

/* One layer call: route, split by the map, run every hot route through its
 * expert, combine.  `experts` holds the records of all E experts (indexed by
 * expert id, so the result cannot depend on which slot holds an expert).
 * out_f32[t, :] = sum over t's hot routes, ascending expert, of w * y;
 * a token without hot routes gets zeros.  Also returns the routing and the
 * compaction (arrays sized M*k, E, and 3 for counts). */
void oracle_moe_layer_fmt(const uint16_t *x, int M, int H, int I, int E, int k, int fmt, const float *Wr,
                          const float *bias, const uint8_t *experts, const int32_t *e2s, float *out_f32,
                          uint16_t *out_bf16, int32_t *ids, float *w, int32_t *hot_expert, int32_t *hot_slot,
                          int32_t *hot_token, float *hot_w, int32_t *act_expert, int32_t *act_slot,
                          int32_t *act_off, int32_t *act_cnt, int32_t *cold_token, int32_t *cold_expert,
                          float *cold_w, int32_t *hist, int32_t *counts, float *logits_out) {
    size_t eb = oracle_expert_bytes_fmt(H, I, fmt);
    float *logits = (float *)malloc(sizeof(float) * (size_t)M * E);
    oracle_router_logits(x, M, H, Wr, bias, E, logits);
    if (logits_out) memcpy(logits_out, logits, sizeof(float) * (size_t)M * E);
    oracle_topk_softmax(logits, M, E, k, ids, w);
    oracle_compact(ids, w, M, k, e2s, E, hot_expert, hot_slot, hot_token, hot_w, act_expert, act_slot,
                   act_off, act_cnt, cold_token, cold_expert, cold_w, hist, counts);
    for (size_t i = 0; i < (size_t)M * H; ++i) out_f32[i] = 0.0f;
    float *y = (float *)malloc(sizeof(float) * (size_t)H);
    for (int r = 0; r < counts[0]; ++r) {
        int t = hot_token[r];
        oracle_expert_ffn_fmt(experts + (size_t)hot_expert[r] * eb, H, I, fmt, x + (size_t)t * H, y);
        for (int c = 0; c < H; ++c) out_f32[(size_t)t * H + c] = out_f32[(size_t)t * H + c] + hot_w[r] * y[c];
    }
    if (out_bf16)
        for (size_t i = 0; i < (size_t)M * H; ++i) out_bf16[i] = oracle_f32_to_bf16(out_f32[i]);
    free(y);
    free(logits);
}

void oracle_moe_layer(const uint16_t *x, int M, int H, int I, int E, int k, const float *Wr,
                      const float *bias, const uint8_t *experts, const int32_t *e2s, float *out_f32,
                      uint16_t *out_bf16, int32_t *ids, float *w, int32_t *hot_expert, int32_t *hot_slot,
                      int32_t *hot_token, float *hot_w, int32_t *act_expert, int32_t *act_slot,
                      int32_t *act_off, int32_t *act_cnt, int32_t *cold_token, int32_t *cold_expert,
                      float *cold_w, int32_t *hist, int32_t *counts, float *logits_out) {
    oracle_moe_layer_fmt(x, M, H, I, E, k, 0, Wr, bias, experts, e2s, out_f32, out_bf16, ids, w, hot_expert,
                         hot_slot, hot_token, hot_w, act_expert, act_slot, act_off, act_cnt, cold_token,
                         cold_expert, cold_w, hist, counts, logits_out);
}

/* --------------------------------------------------------------- slot cache */

/* One step of the frequency/recency slot cache for one layer (NInfer v0.4.0
 * "expert cache": experts the router keeps choosing are copied in, at most
 * R per layer and call, replacing the least used; tinyserve "GPU LFRU
 * cache": frequency with a recency component).
 *
 *  score[e] <- decay * score[e] + hist[e]          (decay = 1: plain LFU)
 *  last[e]  <- step if hist[e] > 0
 *  candidates: experts not resident and not in flight, with score above the
 *              lowest resident score, highest score first, ties lower id
 *  victims:    resident experts not in flight, lowest score first, ties to
 *              the least recently routed (smaller last), then the lower slot
 *  the i-th candidate replaces the i-th victim while its score is strictly
 *  greater, at most R pairs.
 *
 * e2s/s2e are updated in place as if every chosen copy had completed (the
 * deterministic visibility mode); in_flight (per expert, may be NULL) marks
 * experts whose copy has not landed yet in the polled mode.
 * Writes the chosen pairs to pair_expert/pair_slot/pair_victim and returns
 * their number.  Double precision, no contraction, so that decay < 1 gives
 * the same decisions on any host. */
int oracle_cache_step(double *score, int64_t *last, int32_t *e2s, int32_t *s2e, int E, int S,
                      const int32_t *hist, int64_t step, double decay, int R, const uint8_t *in_flight,
                      int32_t *pair_expert, int32_t *pair_slot, int32_t *pair_victim) {
    for (int e = 0; e < E; ++e) {
        score[e] = decay * score[e] + (double)hist[e];
        if (hist[e] > 0) last[e] = step;
    }
    char *used = (char *)calloc((size_t)E, 1);
    int n = 0;
    for (int p = 0; p < R; ++p) {
        /* best candidate */
        int cand = -1;
        for (int e = 0; e < E; ++e) {
            if (e2s[e] >= 0 || used[e] || (in_flight && in_flight[e])) continue;
            if (cand < 0 || score[e] > score[cand]) cand = e;
        }
        if (cand < 0) break;
        /* worst resident victim */
        int vic = -1;
        for (int s = 0; s < S; ++s) {
            int e = s2e[s];
            if (e < 0 || used[e] || (in_flight && in_flight[e])) continue;
            if (vic < 0 || score[e] < score[vic] || (score[e] == score[vic] && last[e] < last[vic]) ||
                (score[e] == score[vic] && last[e] == last[vic] && e2s[e] < e2s[vic]))
                vic = e;
        }
        if (vic < 0 || !(score[cand] > score[vic])) break;
        int slot = e2s[vic];
        used[cand] = 1;
        used[vic] = 1;
        pair_expert[n] = cand;
        pair_slot[n] = slot;
        pair_victim[n] = vic;
        ++n;
    }
    for (int i = 0; i < n; ++i) {
        e2s[pair_victim[i]] = -1;
        e2s[pair_expert[i]] = pair_slot[i];
        s2e[pair_slot[i]] = pair_expert[i];
    }
    free(used);
    return n;
}

/* Recency and arrival policies (tinyserve README "How it works" 3 lists lru
 * and fifo beside frequency-recency; NInfer-Offload v0.4.0: at most R
 * refills per layer and step).  policy 1 = LRU, 2 = FIFO.
 *   last[e]   : the last step that routed e (updated first, for both)
 *   loaded[e] : the step e entered a slot (FIFO; -1 for the initial ones)
 * Candidates: non-resident experts routed this step, most routes first,
 * ties to the lower id.  Victims: LRU the resident expert routed longest
 * ago, FIFO the one loaded earliest, ties to the lower slot.  LRU takes a
 * pair only while the victim was not routed this step; FIFO always.
 * Experts in flight are neither.  score keeps the decayed frequency for
 * reference only.  Returns the number of (expert, slot, victim) pairs. */
int oracle_cache_step_recency(int policy, double *score, int64_t *last, int64_t *loaded, int32_t *e2s,
                              int32_t *s2e, int E, int S, const int32_t *hist, int64_t step, double decay,
                              int R, const uint8_t *in_flight, int32_t *pair_expert, int32_t *pair_slot,
                              int32_t *pair_victim) {
    int e, s, p, n = 0;
    char *used = (char *)calloc((size_t)E, 1);
    for (e = 0; e < E; ++e) {
        score[e] = decay * score[e] + (double)hist[e];
        if (hist[e] > 0) last[e] = step;
    }
    for (p = 0; p < R; ++p) {
        int cand = -1, vic = -1;
        for (e = 0; e < E; ++e) {
            if (e2s[e] >= 0 || used[e] || hist[e] <= 0 || (in_flight && in_flight[e])) continue;
            if (cand < 0 || hist[e] > hist[cand]) cand = e; /* ascending e: ties keep the lower id */
        }
        if (cand < 0) break;
        for (s = 0; s < S; ++s) { /* ascending slot: ties keep the lower slot */
            int r = s2e[s];
            int64_t key, best;
            if (r < 0 || used[r] || (in_flight && in_flight[r])) continue;
            if (vic < 0) {
                vic = r;
                continue;
            }
            key = policy == 2 ? loaded[r] : last[r];
            best = policy == 2 ? loaded[vic] : last[vic];
            if (key < best) vic = r;
        }
        if (vic < 0) break;
        if (policy == 1 && last[vic] >= step) break; /* LRU never evicts an expert this step used */
        used[cand] = 1;
        used[vic] = 1;
        pair_expert[n] = cand;
        pair_slot[n] = e2s[vic];
        pair_victim[n] = vic;
        ++n;
    }
    for (p = 0; p < n; ++p) {
        e2s[pair_victim[p]] = -1;
        e2s[pair_expert[p]] = pair_slot[p];
        s2e[pair_slot[p]] = pair_expert[p];
        if (loaded) loaded[pair_expert[p]] = step;
    }
    free(used);
    return n;
}

/* Segmented LRU (tinyserve README "Configuration" lists slru among its cache
 * policies beside lru, lfru, lfu and fifo; "How it works" 3).  The pages
 * give no details; this follows the textbook two-segment scheme.  Resident
 * experts are either probationary (seg 0) or protected (seg 1); at most
 * pcap of them are protected.  Per step:
 *   1. last[e] = step for every routed expert; score keeps the decayed
 *      frequency for reference only.
 *   2. a routed resident expert that is probationary becomes protected;
 *   3. while more than pcap residents are protected, the protected one
 *      routed longest ago (ties: lower slot) goes back to probationary;
 *   4. candidates: non-resident experts routed this step, most routes
 *      first (ties: lower id); victims: the probationary residents, routed
 *      longest ago first (ties: lower slot), then the protected ones in the
 *      same order; experts in flight are neither.  Candidate i replaces
 *      victim i while that victim was not routed this step, at most R pairs;
 *      a new expert enters probationary.
 * Returns the number of (expert, slot, victim) pairs. */
int oracle_cache_step_slru(double *score, int64_t *last, uint8_t *seg, int32_t *e2s, int32_t *s2e, int E, int S,
                           const int32_t *hist, int64_t step, double decay, int R, int pcap,
                           const uint8_t *in_flight, int32_t *pair_expert, int32_t *pair_slot,
                           int32_t *pair_victim) {
    int e, s, p, n = 0;
    char *used = (char *)calloc((size_t)E, 1);
    for (e = 0; e < E; ++e) {
        score[e] = decay * score[e] + (double)hist[e];
        if (hist[e] > 0) last[e] = step;
    }
    /* promotion of this step's hits */
    for (e = 0; e < E; ++e)
        if (e2s[e] >= 0 && hist[e] > 0) seg[e] = 1;
    /* demotion down to the protected capacity */
    for (;;) {
        int nprot = 0, worst = -1;
        for (s = 0; s < S; ++s) {
            int r = s2e[s];
            if (r < 0 || !seg[r]) continue;
            ++nprot;
            if (worst < 0 || last[r] < last[worst]) worst = r; /* ascending slot: ties keep the lower slot */
        }
        if (nprot <= pcap) break;
        seg[worst] = 0;
    }
    for (p = 0; p < R; ++p) {
        int cand = -1, vic = -1;
        for (e = 0; e < E; ++e) {
            if (e2s[e] >= 0 || used[e] || hist[e] <= 0 || (in_flight && in_flight[e])) continue;
            if (cand < 0 || hist[e] > hist[cand]) cand = e;
        }
        if (cand < 0) break;
        for (s = 0; s < S; ++s) {
            int r = s2e[s];
            if (r < 0 || used[r] || (in_flight && in_flight[r])) continue;
            if (vic < 0 || seg[r] < seg[vic] || (seg[r] == seg[vic] && last[r] < last[vic])) vic = r;
        }
        if (vic < 0 || last[vic] >= step) break; /* never evicts an expert this step routed */
        used[cand] = 1;
        used[vic] = 1;
        pair_expert[n] = cand;
        pair_slot[n] = e2s[vic];
        pair_victim[n] = vic;
        ++n;
    }
    for (p = 0; p < n; ++p) {
        e2s[pair_victim[p]] = -1;
        seg[pair_victim[p]] = 0;
        e2s[pair_expert[p]] = pair_slot[p];
        s2e[pair_slot[p]] = pair_expert[p];
        seg[pair_expert[p]] = 0;
    }
    free(used);
    return n;
}

/* Demand-filled LRU slot table (xinfer docs "How it works", Decode: before
 * the expert GEMMs, a kernel looks the routed experts up in a per-layer LRU
 * table kept on the GPU, gives least-recently-used slots to the misses and
 * rewrites expert ids to slot ids; a second kernel copies the missing
 * experts from device-mapped page-locked host memory into their slots; the
 * step then computes every route from a slot).  The page gives no tie or
 * order rules; readings:
 *   stamp[s] : the last step slot s was used, i.e. its expert was routed
 *              while resident (a hit) or it was filled; -1 at creation.
 *              Hits are stamped before any slot is chosen.
 *   misses   : routed experts without a slot, most routes first, ties to
 *              the lower id.
 *   victims  : slots whose expert this step did not route; empty slots
 *              first (ascending slot), then the oldest stamp, ties to the
 *              lower slot.
 * The i-th miss takes the i-th victim.  A miss left without a victim (the
 * step routes more distinct experts than there are slots) stays cold for
 * this step.  No refill budget: every miss that can be served is.  Writes
 * the fills as (expert, slot) in that order and returns their number. */
int oracle_demand_lru_step(int32_t *e2s, int32_t *s2e, int64_t *stamp, int E, int S, const int32_t *hist,
                           int64_t step, int32_t *fill_expert, int32_t *fill_slot) {
    int e, s, n = 0;
    char *took_e = (char *)calloc((size_t)E, 1), *took_s = (char *)calloc((size_t)S, 1);
    for (e = 0; e < E; ++e)
        if (hist[e] > 0 && e2s[e] >= 0) stamp[e2s[e]] = step;
    for (;;) {
        int cand = -1, vic = -1;
        for (e = 0; e < E; ++e) {
            if (hist[e] <= 0 || e2s[e] >= 0 || took_e[e]) continue;
            if (cand < 0 || hist[e] > hist[cand]) cand = e; /* ascending e: ties keep the lower id */
        }
        if (cand < 0) break;
        for (s = 0; s < S; ++s) { /* ascending s: ties keep the lower slot */
            int r = s2e[s];
            if (took_s[s] || (r >= 0 && hist[r] > 0)) continue;
            if (vic < 0) {
                vic = s;
                continue;
            }
            if (s2e[vic] < 0) continue; /* an empty slot comes first */
            if (r < 0 || stamp[s] < stamp[vic]) vic = s;
        }
        if (vic < 0) break;
        took_e[cand] = 1;
        took_s[vic] = 1;
        fill_expert[n] = cand;
        fill_slot[n] = vic;
        ++n;
    }
    for (int i = 0; i < n; ++i) {
        int v = fill_slot[i], old = s2e[v];
        if (old >= 0) e2s[old] = -1;
        e2s[fill_expert[i]] = v;
        s2e[v] = fill_expert[i];
        stamp[v] = step;
    }
    free(took_e);
    free(took_s);
    return n;
}

/* Next-layer prefetch (tinyserve README "How it works" 4, FATE: the current
 * layer's activations predict the next layer's experts, and their copies to
 * the GPU overlap the current layer's work).  The prediction is the next
 * layer's own routing applied to the current layer's input; pred[e] counts
 * the predicted routes of expert e.  One prefetch step of the next layer:
 *  candidates: predicted experts (pred > 0) neither resident nor in flight,
 *              most predicted routes first, then higher score, then lower id
 *  victims:    resident experts not in flight and not predicted, lowest score
 *              first, then least recently routed, then lower slot
 *  the i-th candidate takes the i-th victim's slot, at most R pairs.
 * Scores and recency are not touched (the layer's own step does that when it
 * routes); e2s/s2e are updated as if the copies had landed.  Returns the
 * number of pairs written to pair_expert/pair_slot/pair_victim. */
int oracle_prefetch_step(const double *score, const int64_t *last, int32_t *e2s, int32_t *s2e, int E, int S,
                         const int32_t *pred, int R, const uint8_t *in_flight, int32_t *pair_expert,
                         int32_t *pair_slot, int32_t *pair_victim) {
    int n = 0;
    char *used = (char *)calloc((size_t)E, 1);
    for (int p = 0; p < R; ++p) {
        /* best remaining candidate */
        int cand = -1;
        for (int e = 0; e < E; ++e) {
            if (pred[e] <= 0 || e2s[e] >= 0 || used[e] || (in_flight && in_flight[e])) continue;
            if (cand < 0 || pred[e] > pred[cand] || (pred[e] == pred[cand] && score[e] > score[cand])) cand = e;
        }
        if (cand < 0) break;
        /* best remaining victim, scanned by slot so that ties go to the lower slot */
        int vic = -1, vslot = -1;
        for (int s = 0; s < S; ++s) {
            int e = s2e[s];
            if (e < 0 || used[e] || pred[e] > 0 || (in_flight && in_flight[e])) continue;
            if (vic < 0 || score[e] < score[vic] || (score[e] == score[vic] && last[e] < last[vic])) {
                vic = e;
                vslot = s;
            }
        }
        if (vic < 0) break;
        used[cand] = used[vic] = 1;
        pair_expert[n] = cand;
        pair_slot[n] = vslot;
        pair_victim[n] = vic;
        ++n;
    }
    for (int i = 0; i < n; ++i) {
        e2s[pair_victim[i]] = -1;
        e2s[pair_expert[i]] = pair_slot[i];
        s2e[pair_slot[i]] = pair_expert[i];
    }
    free(used);
    return n;
}

/* ------------------------------------------------ prefill activation format */

/* E4M3 element (OCP MX v1.0 / OFP8): sign bit 7, exponent bits 6..3 (bias 7),
 * mantissa bits 2..0; exponent 0 is subnormal; S.1111.111 is NaN; max 448. */
float oracle_e4m3(uint8_t code) {
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    float v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexpf((float)m, -9); /* m/8 * 2^(1-7) */
    else
        v = ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return s ? -v : v;
}

/* Nearest E4M3 code to v (ties to an even mantissa), saturating at +-448.
 * Brute force over the 254 finite codes. */
uint8_t oracle_e4m3_encode(float v) {
    uint8_t best = 0;
    double bd = INFINITY;
    for (int c = 0; c < 256; ++c) {
        float q = oracle_e4m3((uint8_t)c);
        if (isnan(q)) continue;
        if (q == 0.0f && (c & 0x80)) continue; /* keep +0 for zero */
        double d = fabs((double)q - (double)v);
        if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) {
            bd = d;
            best = (uint8_t)c;
        }
    }
    if (v > 448.0f) best = 0x7e;
    if (v < -448.0f) best = 0xfe;
    return best;
}

/* MXFP8 block (OCP MX v1.0 conversion rule): shared exponent
 * X = floor(log2(max |v|)) - 8 (8 = largest E4M3 exponent), clamped to the
 * E8M0 range; each element becomes E4M3(v / 2^X), rounding to nearest even,
 * saturating.  A block of zeros gets X = -127.  Returns the E8M0 byte. */
uint8_t oracle_mxfp8_block(const float *v, int n, uint8_t *codes) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i)
        if (fabsf(v[i]) > amax) amax = fabsf(v[i]);
    int X;
    if (amax == 0.0f)
        X = -127;
    else {
        int ex;
        frexpf(amax, &ex); /* amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1 */
        X = (ex - 1) - 8;
        if (X < -127) X = -127;
        if (X > 127) X = 127;
    }
    for (int i = 0; i < n; ++i) codes[i] = oracle_e4m3_encode(ldexpf(v[i], -X));
    return (uint8_t)(X + 127);
}

/* Prefill variant of the expert FFN: x and h pass through MXFP8 (32-element
 * blocks along the contraction) before their products with the MXFP4 weights;
 * the products of two decoded values are exact and summed in fp32. */
void oracle_expert_ffn_mxfp8(const uint8_t *rec, int H, int I, const uint16_t *x, float *y) {
    const uint8_t *gc, *gs, *uc, *us, *dc, *ds;
    expert_sections(rec, H, I, 0, &gc, &gs, &uc, &us, &dc, &ds);
    float *xq = (float *)malloc(sizeof(float) * (size_t)H);
    float *h = (float *)malloc(sizeof(float) * (size_t)I);
    float *hq = (float *)malloc(sizeof(float) * (size_t)I);
    float blk[32];
    uint8_t codes[32];
    for (int b = 0; b < H / 32; ++b) {
        for (int i = 0; i < 32; ++i) blk[i] = oracle_bf16_to_f32(x[b * 32 + i]);
        uint8_t sc = oracle_mxfp8_block(blk, 32, codes);
        for (int i = 0; i < 32; ++i) xq[b * 32 + i] = oracle_e4m3(codes[i]) * oracle_e8m0(sc);
    }
    for (int i = 0; i < I; ++i) {
        float g = 0.0f, u = 0.0f;
        for (int c = 0; c < H; ++c) {
            g = g + oracle_mxfp4_element(gc, gs, H, i, c) * xq[c];
            u = u + oracle_mxfp4_element(uc, us, H, i, c) * xq[c];
        }
        h[i] = silu(g) * u;
    }
    for (int b = 0; b < I / 32; ++b) {
        uint8_t sc = oracle_mxfp8_block(h + b * 32, 32, codes);
        for (int i = 0; i < 32; ++i) hq[b * 32 + i] = oracle_e4m3(codes[i]) * oracle_e8m0(sc);
    }
    for (int r = 0; r < H; ++r) {
        float acc = 0.0f;
        for (int i = 0; i < I; ++i) acc = acc + oracle_mxfp4_element(dc, ds, I, r, i) * hq[i];
        y[r] = acc;
    }
    free(xq);
    free(h);
    free(hq);
}
