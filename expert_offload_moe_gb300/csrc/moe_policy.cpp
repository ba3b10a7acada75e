// Slot-cache decision for one layer and one step, on the host.
//
// NInfer-Offload v0.4.0 "expert cache": slots follow recent routing; experts
// the router keeps choosing are copied to the GPU in the background, at most
// two per layer and call, replacing the least used.  tinyserve README "How it
// works" 3: frequency-recency eviction keyed by (layer, expert).
//
// Score: score = decay * score + routes this step (decay 1 = LFU).
// Candidates: experts neither resident nor in flight, best score first (ties:
// lower id).  Victims: resident experts not in flight, lowest score first
// (ties: least recently routed, then lower slot).  Pair i is taken while the
// candidate's score is strictly greater than the victim's; at most R pairs.
#include <cstdint>
#include <algorithm>
#include <vector>

#include "../../include/moe.h"

extern "C" int moe_policy_step(double *score, int64_t *last, int32_t *e2s, int32_t *s2e, int32_t E, int32_t S,
                               const int32_t *hist, int64_t step, double decay, int32_t R,
                               const uint8_t *in_flight, int32_t *pair_expert, int32_t *pair_slot,
                               int32_t *pair_victim) {
    if (!score || !last || !e2s || !s2e || !hist || E <= 0 || S <= 0 || S > E || R < 0 ||
        (R > 0 && (!pair_expert || !pair_slot || !pair_victim)))
        return -1;
    for (int32_t e = 0; e < E; ++e) {
        // a separate multiply and add, so every host compiler gives the same doubles
        const double decayed = decay * score[e];
        score[e] = decayed + static_cast<double>(hist[e]);
        if (hist[e] > 0) last[e] = step;
    }
    std::vector<char> taken(static_cast<size_t>(E), 0);
    auto busy = [&](int32_t e) { return taken[e] || (in_flight && in_flight[e]); };

    int32_t n = 0;
    for (int32_t p = 0; p < R; ++p) {
        int32_t cand = -1;
        for (int32_t e = 0; e < E; ++e) {
            if (e2s[e] >= 0 || busy(e)) continue;
            if (cand < 0 || score[e] > score[cand]) cand = e;
        }
        if (cand < 0) break;
        int32_t vic = -1;
        for (int32_t s = 0; s < S; ++s) {
            const int32_t e = s2e[s];
            if (e < 0 || busy(e)) continue;
            if (vic < 0) {
                vic = e;
                continue;
            }
            const bool lower = score[e] < score[vic];
            const bool same = score[e] == score[vic];
            if (lower || (same && last[e] < last[vic]) || (same && last[e] == last[vic] && s < e2s[vic])) vic = e;
        }
        if (vic < 0 || !(score[cand] > score[vic])) break;
        taken[cand] = taken[vic] = 1;
        pair_expert[n] = cand;
        pair_slot[n] = e2s[vic];
        pair_victim[n] = vic;
        ++n;
    }
    for (int32_t i = 0; i < n; ++i) {
        e2s[pair_victim[i]] = -1;
        e2s[pair_expert[i]] = pair_slot[i];
        s2e[pair_slot[i]] = pair_expert[i];
    }
    return n;
}

// Recency and arrival policies (tinyserve README "How it works" 3 lists lru and fifo beside
// frequency-recency).  policy MOE_POLICY_LRU: the victim is the resident expert routed longest ago, and
// an expert this step routed is never evicted; MOE_POLICY_FIFO: the victim is the resident expert that
// entered its slot first, whatever its use.  Candidates are the non-resident experts this step routed,
// most routes first; ties go to the lower id (candidates) and the lower slot (victims).  score keeps the
// decayed frequency for reference; loaded[e] (FIFO) is the step e entered a slot, -1 for the initial ones.
extern "C" int moe_policy_step_recency(int32_t policy, double *score, int64_t *last, int64_t *loaded, int32_t *e2s,
                                       int32_t *s2e, int32_t E, int32_t S, const int32_t *hist, int64_t step,
                                       double decay, int32_t R, const uint8_t *in_flight, int32_t *pair_expert,
                                       int32_t *pair_slot, int32_t *pair_victim) {
    if ((policy != MOE_POLICY_LRU && policy != MOE_POLICY_FIFO) || !score || !last || !e2s || !s2e || !hist ||
        E <= 0 || S <= 0 || S > E || R < 0 || (policy == MOE_POLICY_FIFO && !loaded) ||
        (R > 0 && (!pair_expert || !pair_slot || !pair_victim)))
        return -1;
    for (int32_t e = 0; e < E; ++e) {
        const double decayed = decay * score[e];
        score[e] = decayed + static_cast<double>(hist[e]);
        if (hist[e] > 0) last[e] = step;
    }
    auto busy = [&](int32_t e) { return in_flight && in_flight[e]; };
    // candidates in order: routes descending, then id ascending
    std::vector<int32_t> cand;
    for (int32_t e = 0; e < E; ++e)
        if (e2s[e] < 0 && hist[e] > 0 && !busy(e)) cand.push_back(e);
    std::stable_sort(cand.begin(), cand.end(), [&](int32_t a, int32_t b) { return hist[a] > hist[b]; });
    // victims in order: key ascending (last use, or load step), then slot ascending
    std::vector<int32_t> vic;
    for (int32_t s = 0; s < S; ++s)
        if (s2e[s] >= 0 && !busy(s2e[s])) vic.push_back(s2e[s]);
    auto key = [&](int32_t e) { return policy == MOE_POLICY_FIFO ? loaded[e] : last[e]; };
    std::stable_sort(vic.begin(), vic.end(), [&](int32_t a, int32_t b) { return key(a) < key(b); });
    int32_t n = 0;
    const size_t np = std::min(cand.size(), vic.size());
    for (size_t i = 0; i < np && n < R; ++i) {
        const int32_t c = cand[i], v = vic[i];
        if (policy == MOE_POLICY_LRU && last[v] >= step) break;
        pair_expert[n] = c;
        pair_slot[n] = e2s[v];
        pair_victim[n] = v;
        ++n;
    }
    for (int32_t i = 0; i < n; ++i) {
        e2s[pair_victim[i]] = -1;
        e2s[pair_expert[i]] = pair_slot[i];
        s2e[pair_slot[i]] = pair_expert[i];
        if (loaded) loaded[pair_expert[i]] = step;
    }
    return n;
}

// Segmented LRU (tinyserve README "Configuration" lists slru among the cache policies): hits are promoted
// to a protected segment of at most pcap residents, its least recently routed members fall back to the
// probationary segment, and victims come from the probationary segment before the protected one.
extern "C" int moe_policy_step_slru(double *score, int64_t *last, uint8_t *seg, int32_t *e2s, int32_t *s2e,
                                    int32_t E, int32_t S, const int32_t *hist, int64_t step, double decay,
                                    int32_t R, int32_t pcap, const uint8_t *in_flight, int32_t *pair_expert,
                                    int32_t *pair_slot, int32_t *pair_victim) {
    if (!score || !last || !seg || !e2s || !s2e || !hist || E <= 0 || S <= 0 || S > E || R < 0 || pcap < 0 ||
        pcap > S || (R > 0 && (!pair_expert || !pair_slot || !pair_victim)))
        return -1;
    for (int32_t e = 0; e < E; ++e) {
        const double decayed = decay * score[e];
        score[e] = decayed + static_cast<double>(hist[e]);
        if (hist[e] > 0) last[e] = step;
        if (hist[e] > 0 && e2s[e] >= 0) seg[e] = 1;
    }
    // residents by (last use, slot): the order of both demotion and eviction within a segment
    std::vector<int32_t> order;
    for (int32_t s = 0; s < S; ++s)
        if (s2e[s] >= 0) order.push_back(s2e[s]);
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return last[a] < last[b]; });
    int32_t nprot = 0;
    for (int32_t e : order) nprot += seg[e] ? 1 : 0;
    for (int32_t e : order) {
        if (nprot <= pcap) break;
        if (seg[e]) {
            seg[e] = 0;
            --nprot;
        }
    }
    auto busy = [&](int32_t e) { return in_flight && in_flight[e]; };
    std::vector<int32_t> cand;
    for (int32_t e = 0; e < E; ++e)
        if (e2s[e] < 0 && hist[e] > 0 && !busy(e)) cand.push_back(e);
    std::stable_sort(cand.begin(), cand.end(), [&](int32_t a, int32_t b) { return hist[a] > hist[b]; });
    std::vector<int32_t> vic;
    for (int32_t e : order)
        if (!seg[e] && !busy(e)) vic.push_back(e);
    for (int32_t e : order)
        if (seg[e] && !busy(e)) vic.push_back(e);
    int32_t n = 0;
    const size_t np = std::min(cand.size(), vic.size());
    for (size_t i = 0; i < np && n < R; ++i) {
        if (last[vic[i]] >= step) break;
        pair_expert[n] = cand[i];
        pair_slot[n] = e2s[vic[i]];
        pair_victim[n] = vic[i];
        ++n;
    }
    for (int32_t i = 0; i < n; ++i) {
        e2s[pair_victim[i]] = -1;
        seg[pair_victim[i]] = 0;
        e2s[pair_expert[i]] = pair_slot[i];
        s2e[pair_slot[i]] = pair_expert[i];
        seg[pair_expert[i]] = 0;
    }
    return n;
}

// Next-layer prefetch (tinyserve README "How it works" 4, FATE: the current layer's activations predict the
// next layer's experts; their copies overlap the current layer's work).  pred[e] counts the predicted routes
// of expert e (the next layer's routing applied to the current layer's input).  Candidates: predicted experts
// neither resident nor in flight, most predicted routes first, then higher score, then lower id.  Victims:
// resident experts neither predicted nor in flight, lowest score first, then least recently routed, then
// lower slot.  Candidate i takes victim i's slot, at most R pairs.  Scores and recency are left alone: the
// layer's own step counts the routes when they happen.
extern "C" int moe_prefetch_step(const double *score, const int64_t *last, int32_t *e2s, int32_t *s2e, int32_t E,
                                 int32_t S, const int32_t *pred, int32_t R, const uint8_t *in_flight,
                                 int32_t *pair_expert, int32_t *pair_slot, int32_t *pair_victim) {
    if (!score || !last || !e2s || !s2e || !pred || E <= 0 || S <= 0 || S > E || R < 0 ||
        (R > 0 && (!pair_expert || !pair_slot || !pair_victim)))
        return -1;
    auto busy = [&](int32_t e) { return in_flight && in_flight[e]; };
    std::vector<int32_t> cand, vic;
    for (int32_t e = 0; e < E; ++e)
        if (pred[e] > 0 && e2s[e] < 0 && !busy(e)) cand.push_back(e);
    std::stable_sort(cand.begin(), cand.end(), [&](int32_t a, int32_t b) {
        return pred[a] != pred[b] ? pred[a] > pred[b] : score[a] > score[b];
    });
    for (int32_t s = 0; s < S; ++s) {
        const int32_t e = s2e[s];
        if (e >= 0 && pred[e] <= 0 && !busy(e)) vic.push_back(e);
    }
    std::stable_sort(vic.begin(), vic.end(), [&](int32_t a, int32_t b) {
        return score[a] != score[b] ? score[a] < score[b] : last[a] < last[b];
    });
    const int32_t n = static_cast<int32_t>(std::min<size_t>({cand.size(), vic.size(), static_cast<size_t>(R)}));
    for (int32_t i = 0; i < n; ++i) {
        pair_expert[i] = cand[i];
        pair_slot[i] = e2s[vic[i]];
        pair_victim[i] = vic[i];
    }
    for (int32_t i = 0; i < n; ++i) {
        e2s[pair_victim[i]] = -1;
        e2s[pair_expert[i]] = pair_slot[i];
        s2e[pair_slot[i]] = pair_expert[i];
    }
    return n;
}
