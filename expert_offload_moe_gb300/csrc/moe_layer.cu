// The layer object and the C ABI calls (declared in include/moe.h).
//
// Streams: every compute kernel runs on the caller's stream.  Two internal
// non-blocking streams carry copies: `d2h` mirrors the cold-route list to
// page-locked host memory (forked from the caller's stream after routing,
// joined back by moe_forward_slots), and `h2d` carries slot refills from the
// page-locked host bank (onnxruntime PR #33976: pinned staging with
// CUDA_EVENT_DISABLE_TIMING events for overlap; NInfer-Offload v0.4.0: refills
// run in the background without stalling decode).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "moe_host.h"
#include "moe_internal.h"

namespace {

// out[t, :] += y[t, :] for the first M tokens (bf16 outputs are rounded once more, to nearest even).
__global__ void add_cold_kernel(void *out, const float *y, int n, int out_f32) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        if (out_f32) {
            reinterpret_cast<float *>(out)[i] += y[i];
        } else {
            __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(out);
            o[i] = __float2bfloat16_rn(__bfloat162float(o[i]) + y[i]);
        }
    }
}

// The cold routes of a decode step (ordered by (token, expert), at most 128) grouped by expert for the
// CUDA-core FFN kernels: routes ordered by (expert, token), and per expert its first route and count.
__global__ void __launch_bounds__(128) cold_lists_kernel(const int32_t *counts, const int32_t *ctok,
                                                         const int32_t *cexp, const float *cw, int32_t *act_expert,
                                                         int32_t *act_off, int32_t *act_cnt, int32_t *tok, float *w,
                                                         int32_t *c_counts) {
    __shared__ int s_e[128], s_t[128];
    __shared__ unsigned char s_first[128];
    const int n = counts[1], r = threadIdx.x;
    const bool mine = r < n;
    const int e = mine ? cexp[r] : 0, t = mine ? ctok[r] : 0;
    if (mine) {
        s_e[r] = e;
        s_t[r] = t;
    }
    __syncthreads();
    if (mine) {
        bool first = true;
        for (int q = 0; q < n; ++q)
            if (s_e[q] == e && s_t[q] < t) first = false;
        s_first[r] = first;
    }
    __syncthreads();
    if (mine) {
        int pos = 0, aidx = 0, cnt = 0;
        for (int q = 0; q < n; ++q) {
            pos += s_e[q] < e || (s_e[q] == e && s_t[q] < t);
            aidx += s_first[q] && s_e[q] < e;
            cnt += s_e[q] == e;
        }
        tok[pos] = t;
        w[pos] = cw[r];
        if (s_first[r]) {
            act_expert[aidx] = e;
            act_off[aidx] = pos;
            act_cnt[aidx] = cnt;
        }
    }
    const int n_act = __syncthreads_count(mine && s_first[r]);
    if (r == 0) {
        c_counts[0] = n;
        c_counts[1] = 0;
        c_counts[2] = n_act;
        c_counts[3] = 0;
    }
}

}  // namespace

namespace {

thread_local std::string g_err;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

#define CUDA_TRY(call)                                                                          \
    do {                                                                                        \
        cudaError_t _e = (call);                                                                \
        if (_e != cudaSuccess) return fail(MOE_ECUDA, "%s: %s", #call, cudaGetErrorString(_e)); \
    } while (0)

struct PendingCopy {
    int32_t expert, slot;
    cudaEvent_t ev;
};

}  // namespace

struct moe_layer {
    moe_layer_desc d{};
    int device = 0;
    int num_sms = 0;
    moe::ExpertGeometry geo{};
    int nchunk = 0;
    int max_hot = 0;

    uint8_t *slots = nullptr;  // [S][expert_bytes]
    float *Wr = nullptr;       // [E][H]
    float *WrT = nullptr;      // [H][E32], the router transposed for prefill routing
    float *bias = nullptr;     // [E]
    int32_t *e2s_dev = nullptr;
    const uint8_t *host_bank = nullptr;
    uint8_t *staging = nullptr;
    size_t staging_bytes = 0;
    bool staged = false;

    moe::RouteBuffers rb{};
    float *h = nullptr;  // [max_hot][I]
    // cold routes on the GPU from the page-locked bank (moe_forward_cold_gpu)
    const uint8_t *host_bank_dev = nullptr;  // the bank's device address, nullptr if the GPU cannot reach it
    void *cold_block = nullptr;              // lists of the cold routes grouped by expert, and their h
    int32_t *c_act_expert = nullptr, *c_act_off = nullptr, *c_act_cnt = nullptr, *c_token = nullptr,
            *c_counts = nullptr;
    float *c_w = nullptr, *c_h = nullptr;
    void *dev_block = nullptr;

    // page-locked mirror
    int32_t *m_counts = nullptr, *m_cold_token = nullptr, *m_cold_expert = nullptr, *m_hist = nullptr;
    float *m_cold_w = nullptr;
    // cold routes on host threads (decode): x mirrored with the route, their sums and the device copy
    uint16_t *m_x = nullptr;     // [dec_tokens][H] bf16, page-locked
    float *m_ycold = nullptr;    // [dec_tokens][H] fp32, page-locked
    float *d_ycold = nullptr;    // [dec_tokens][H] fp32
    cudaEvent_t ev_cold = nullptr;  // the last copy of m_ycold to the device
    void *pinned_block = nullptr;
    // what moe_route mirrors to the host, laid out identically on the device and in pinned_block, so that
    // one copy moves it: counts[4], hist[E], cold token/expert/w [dec k] each, x [dec][H] (decode)
    void *mir_block = nullptr;
    size_t mir_off_cold = 0, mir_off_x = 0;
    // under stream capture the mirror copy is a leaf node of the graph; the next moe_route of the layer in the
    // same capture depends on it (it must have read the route buffers before they are rewritten)
    cudaGraphNode_t cap_mirror = nullptr;
    unsigned long long cap_id = 0;

    // next-layer prefetch (moe_prefetch): route scratch of its own, so that a prediction never touches the
    // buffers of the layer's last moe_route, and the predicted histogram in page-locked memory
    moe::RouteBuffers prb{};
    void *pred_block = nullptr;
    int32_t *m_pred = nullptr;
    cudaEvent_t ev_pred = nullptr, ev_pfork = nullptr;

    cudaStream_t d2h = nullptr, h2d = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_route = nullptr, ev_fence = nullptr;
    std::vector<cudaEvent_t> ev_copy;  // deterministic mode, one per pair
    std::vector<cudaEvent_t> ev_pool;  // polled mode
    std::vector<PendingCopy> pending;

    // host policy state
    std::vector<int32_t> e2s, s2e, e2s_visible;
    std::vector<double> score;
    int policy = MOE_POLICY_FREQ;
    std::vector<int64_t> loaded;  // FIFO: the step each expert entered its slot
    std::vector<uint8_t> seg;     // SLRU: 1 while the expert is in the protected segment
    std::vector<int64_t> last;
    std::vector<uint8_t> in_flight;
    int64_t step = 0;

    // call-order state
    const void *routed_x = nullptr;
    int32_t routed_M = 0;
    bool routed_plan = false;  // the last route launch wrote the prefill tile plan
    int64_t route_seq = 0, policy_seq = 0;
    int fault = MOE_FAULT_NONE;
    int64_t stats[4] = {0, 0, 0, 0};

    // tensor-core decode path: operand buffers, split-K scratch, tensor maps
    bool tc = false;
    int n_act_cap = 0;  // most active experts a decode call can have: min(S, 8 k)
    int Hpad = 0, Ipad = 0;
    moe::TcAtomLayout atl{};
    uint8_t *atoms = nullptr;  // weight scale atoms of every slot [S][atl.slot_bytes]
    uint8_t *xq = nullptr, *xat = nullptr, *hq = nullptr, *hat = nullptr;
    int *err = nullptr;
    float *part = nullptr;      // one-launch FFN (M = 1): down partials [ntH][n_act(1) ntI][128]
    bool ffn1 = true;           // M = 1 takes the one-launch FFN (moe_debug_decode_fusion)
    void *tc_block = nullptr;
    CUtensorMap mapG{}, mapU{}, mapD{}, mapX{}, mapH{};
    // NVFP4 one-token decode on the tensor cores (the buffers above are shared with it: xq, xat, atoms, err,
    // part, tc_block): x terms as packed E2M1, their per-term powers of two, UE4M3 scale atoms, packed maps
    bool tcnv = false;
    moe::NvAtomLayout nvl{};
    float *nv_xg = nullptr;
    int Hpad4 = 0;
    CUtensorMap mapGn{}, mapUn{}, mapDn{}, mapXn{};

    // tensor-core prefill over the staged bank: scratch allocated when staging is attached
    bool pf = false;
    int tiles_cap = 0, rows_cap = 0;
    uint8_t *stage_atoms = nullptr;  // weight atoms of every staged expert [E][atl.slot_bytes]
    void *pf_block = nullptr;
    uint8_t *XP = nullptr, *XA = nullptr, *HP = nullptr, *HA = nullptr;
    float *YP = nullptr;
    int32_t *pf_poff = nullptr, *pf_e2a = nullptr, *pf_tile_aidx = nullptr, *pf_tile_nrows = nullptr, *pf_ntiles = nullptr;
    CUtensorMap mapXP{}, mapHP{}, mapSG{}, mapSU{}, mapSD{};

    // device-resident slot table (moe_layer_set_device_cache): the route kernel runs a demand-filled LRU
    // step and the fill kernel copies the misses from the bank's device address, all in stream order
    bool dev_cache = false;
    void *lru_block = nullptr;
    moe::LruTable lru{};

    // optional per-kernel timing: event pairs around route, gate/up and down launches
    bool prof = false;
    std::vector<cudaEvent_t> prof_ev[3];
    size_t prof_n[3] = {0, 0, 0};
};

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

void release(moe_layer *L) {
    if (!L) return;
    if (L->h2d) cudaStreamSynchronize(L->h2d);
    if (L->d2h) cudaStreamSynchronize(L->d2h);
    cudaFree(L->slots);
    cudaFree(L->Wr);
    cudaFree(L->WrT);
    cudaFree(L->d_ycold);
    cudaFree(L->bias);
    cudaFree(L->e2s_dev);
    cudaFree(L->dev_block);
    cudaFree(L->mir_block);
    cudaFree(L->pred_block);
    if (L->m_pred) cudaFreeHost(L->m_pred);
    if (L->ev_pred) cudaEventDestroy(L->ev_pred);
    if (L->ev_pfork) cudaEventDestroy(L->ev_pfork);
    cudaFree(L->h);
    cudaFree(L->cold_block);
    cudaFree(L->tc_block);
    cudaFree(L->atoms);
    cudaFree(L->pf_block);
    cudaFree(L->stage_atoms);
    cudaFree(L->lru_block);
    if (L->pinned_block) cudaFreeHost(L->pinned_block);
    for (auto e : {L->ev_fork, L->ev_route, L->ev_fence, L->ev_cold})
        if (e) cudaEventDestroy(e);
    for (auto e : L->ev_copy) cudaEventDestroy(e);
    for (auto e : L->ev_pool) cudaEventDestroy(e);
    for (auto &p : L->pending) cudaEventDestroy(p.ev);
    for (auto &v : L->prof_ev)
        for (auto e : v) cudaEventDestroy(e);
    if (L->d2h) cudaStreamDestroy(L->d2h);
    if (L->h2d) cudaStreamDestroy(L->h2d);
    delete L;
}

int enqueue_map(moe_layer *L, const std::vector<int32_t> &ex, const std::vector<int32_t> &sl, cudaStream_t s) {
    if (ex.empty()) return MOE_OK;
    moe::launch_map_update(L->e2s_dev, (int)ex.size(), ex.data(), sl.data(), s);
    CUDA_TRY(cudaGetLastError());
    for (size_t i = 0; i < ex.size(); ++i) L->e2s_visible[ex[i]] = sl[i];
    return MOE_OK;
}

// Records the opening or closing event of timed kernel `which` (0 route, 1 gate/up, 2 down).
cudaError_t prof_mark(moe_layer *L, int which, cudaStream_t s) {
    if (!L->prof) return cudaSuccess;
    auto &v = L->prof_ev[which];
    size_t &n = L->prof_n[which];
    if (n == v.size()) {
        cudaEvent_t e;
        cudaError_t rc = cudaEventCreate(&e);
        if (rc != cudaSuccess) return rc;
        v.push_back(e);
    }
    // under stream capture the mark becomes an event-record node of the graph, so replays record times
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t rc = cudaStreamIsCapturing(s, &cs);
    if (rc != cudaSuccess) return rc;
    return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(v[n++], s, cudaEventRecordExternal)
                                               : cudaEventRecord(v[n++], s);
}

// The next event of timed kernel `which` for a caller that records it itself (nullptr when not profiling).
cudaEvent_t prof_next(moe_layer *L, int which) {
    if (!L->prof) return nullptr;
    auto &v = L->prof_ev[which];
    size_t &n = L->prof_n[which];
    if (n == v.size()) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        v.push_back(e);
    }
    return v[n++];
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 3-D tiled map with a 128-byte swizzle: dims {d0 (elements), d1, d2}, byte strides {s1, s2}, box {b0, b1, 1}.
int encode_map(CUtensorMap *m, CUtensorMapDataType type, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, const char *what) {
    auto enc = tensor_map_encoder();
    if (!enc) return fail(MOE_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1, s2};
    const cuuint32_t box[3] = {b0, b1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, type, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOE_ECUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
    return MOE_OK;
}

// K splits: enough CTAs for about two per SM (the kernels are sized to fit two), but at least
// 4 k-steps of 128 per CTA so the pipeline has something to overlap, and at most one cluster's worth.
int choose_splits(int base_units, int steps, int num_sms) {
    int ks = (2 * num_sms) / (base_units > 0 ? base_units : 1);
    const int ks_max = steps / 4 > 1 ? steps / 4 : 1;
    if (ks > ks_max) ks = ks_max;
    if (ks > moe::tc_max_splits()) ks = moe::tc_max_splits();
    return ks < 1 ? 1 : ks;
}

int act_cap(const moe_layer *L, int M) {
    const int a = M * L->d.top_k;
    return a < L->d.num_slots ? a : L->d.num_slots;
}

int tc_splits_gateup(const moe_layer *L, int M) {
    return choose_splits(act_cap(L, M) * ((L->d.inter + 127) / 128), (L->d.hidden + 127) / 128, L->num_sms);
}

int tc_splits_down(const moe_layer *L, int M) {
    return choose_splits((L->d.hidden + 127) / 128, act_cap(L, M) * ((L->d.inter + 127) / 128), L->num_sms);
}

// Weight scale atoms of one slot, rebuilt whenever an expert lands in it (stream-ordered after the copy).
int build_slot_atoms(moe_layer *L, int slot, cudaStream_t st) {
    if (L->tcnv) {
        moe::launch_build_weight_atoms_nv(L->slots + (size_t)slot * L->geo.expert_bytes, L->geo,
                                          L->atoms + (size_t)slot * L->nvl.slot_bytes, st);
        CUDA_TRY(cudaGetLastError());
        return MOE_OK;
    }
    if (!L->tc) return MOE_OK;
    moe::launch_build_weight_atoms(L->slots + (size_t)slot * L->geo.expert_bytes, L->geo,
                                   L->atoms + (size_t)slot * L->atl.slot_bytes, st);
    CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

// Buffers and tensor maps of the tensor-core decode path.
int tc_setup(moe_layer *L, cudaStream_t st) {
    const int H = L->d.hidden, I = L->d.inter;
    L->n_act_cap = act_cap(L, moe::kDecodeMaxTokens);
    L->Hpad = (H + 127) / 128 * 128;
    L->Ipad = (I + 127) / 128 * 128;
    L->atl = moe::tc_atom_layout(H, I);
    const size_t ucap1 = (size_t)act_cap(L, 1) * L->atl.ntI;  // units of the one-launch FFN
    const size_t sz[] = {(size_t)moe::kTcXRows * L->Hpad,
                         (size_t)L->atl.nks * moe::kTcAtomBytes,
                         (size_t)L->n_act_cap * moe::kTcHRows * L->Ipad,
                         (size_t)L->n_act_cap * L->atl.nksI * moe::kTcAtomBytes,
                         sizeof(int),
                         (size_t)L->atl.ntH * ucap1 * 128 * sizeof(float)};
    size_t total = 0;
    for (size_t s : sz) total += align_up(s, 256);
    cudaError_t e = cudaMalloc(&L->tc_block, total);
    if (e == cudaSuccess) e = cudaMalloc(&L->atoms, (size_t)L->d.num_slots * L->atl.slot_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(e == cudaErrorMemoryAllocation ? MOE_ENOMEM : MOE_ECUDA, "tensor-core buffers: %s",
                    cudaGetErrorString(e));
    }
    char *p = static_cast<char *>(L->tc_block);
    void **dst[] = {(void **)&L->xq,  (void **)&L->xat,  (void **)&L->hq,  (void **)&L->hat,
                    (void **)&L->err, (void **)&L->part};
    for (size_t i = 0; i < sizeof(sz) / sizeof(sz[0]); ++i) {
        *dst[i] = p;
        p += align_up(sz[i], 256);
    }
    // operands start at zero; scale bytes never written (rows or k-blocks past the data) stay finite: 2^0
    CUDA_TRY(cudaMemsetAsync(L->tc_block, 0, total, st));
    CUDA_TRY(cudaMemsetAsync(L->xat, 0x7f, sz[1], st));
    CUDA_TRY(cudaMemsetAsync(L->hat, 0x7f, sz[3], st));
    CUDA_TRY(cudaMemsetAsync(L->atoms, 0x7f, (size_t)L->d.num_slots * L->atl.slot_bytes, st));

    const moe::ExpertGeometry &g = L->geo;
    const int S = L->d.num_slots;
    int rc;
    if ((rc = encode_map(&L->mapG, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, L->slots + g.off_wg_codes, H / 128 * 128,
                         I, S, H / 2, g.expert_bytes, 128, 128, "gate codes")))
        return rc;
    if ((rc = encode_map(&L->mapU, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, L->slots + g.off_wu_codes, H / 128 * 128,
                         I, S, H / 2, g.expert_bytes, 128, 128, "up codes")))
        return rc;
    if ((rc = encode_map(&L->mapD, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, L->slots + g.off_wd_codes, I / 128 * 128,
                         H, S, I / 2, g.expert_bytes, 128, 128, "down codes")))
        return rc;
    if ((rc = encode_map(&L->mapX, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->xq, L->Hpad, moe::kTcXRows, 1, L->Hpad,
                         (uint64_t)moe::kTcXRows * L->Hpad, 128, moe::kTcXRows, "x terms")))
        return rc;
    if ((rc = encode_map(&L->mapH, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->hq, L->Ipad, moe::kTcHRows, L->n_act_cap,
                         L->Ipad, (uint64_t)moe::kTcHRows * L->Ipad, 128, moe::kTcHRows, "h terms")))
        return rc;
    L->tc = true;
    return MOE_OK;
}

// Buffers and tensor maps of the NVFP4 one-token decode on the tensor cores (packed E2M1 operands).
int nv_setup(moe_layer *L, cudaStream_t st) {
    const int H = L->d.hidden, I = L->d.inter;
    L->Hpad4 = (H + 255) / 256 * 256;
    L->nvl = moe::nv_atom_layout(H, I);
    const size_t ucap1 = (size_t)act_cap(L, 1) * L->nvl.ntI;
    const size_t xrow = (size_t)L->Hpad4 / 2;
    const size_t sz[] = {(size_t)moe::kNvTerms * xrow, (size_t)L->nvl.nks4 * 4 * moe::kTcAtomBytes,
                         (size_t)moe::kNvTerms * sizeof(float), sizeof(int),
                         (size_t)L->nvl.ntH * ucap1 * 128 * sizeof(float)};
    size_t total = 0;
    for (size_t s : sz) total += align_up(s, 256);
    cudaError_t e = cudaMalloc(&L->tc_block, total);
    if (e == cudaSuccess) e = cudaMalloc(&L->atoms, (size_t)L->d.num_slots * L->nvl.slot_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(e == cudaErrorMemoryAllocation ? MOE_ENOMEM : MOE_ECUDA, "NVFP4 tensor-core buffers: %s",
                    cudaGetErrorString(e));
    }
    char *p = static_cast<char *>(L->tc_block);
    void **dst[] = {(void **)&L->xq, (void **)&L->xat, (void **)&L->nv_xg, (void **)&L->err, (void **)&L->part};
    for (size_t i = 0; i < sizeof(sz) / sizeof(sz[0]); ++i) {
        *dst[i] = p;
        p += align_up(sz[i], 256);
    }
    // x codes past H stay zero; scale bytes never written (blocks past H, columns past the terms) stay 1.0
    CUDA_TRY(cudaMemsetAsync(L->tc_block, 0, total, st));
    CUDA_TRY(cudaMemsetAsync(L->xat, 0x38, sz[1], st));
    CUDA_TRY(cudaMemsetAsync(L->atoms, 0x38, (size_t)L->d.num_slots * L->nvl.slot_bytes, st));
    const moe::ExpertGeometry &g = L->geo;
    const int S = L->d.num_slots;
    int rc;
    // codes as bytes: 128 rows x 128 bytes (256 codes) per gate/up box, 128 rows x 64 bytes per down box; the
    // boxes at the ragged ends of H and I are zero-filled past the matrix
    if ((rc = encode_map(&L->mapGn, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->slots + g.off_wg_codes, H / 2, I, S, H / 2,
                         g.expert_bytes, 128, 128, "gate codes (NVFP4)")))
        return rc;
    if ((rc = encode_map(&L->mapUn, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->slots + g.off_wu_codes, H / 2, I, S, H / 2,
                         g.expert_bytes, 128, 128, "up codes (NVFP4)")))
        return rc;
    if ((rc = encode_map(&L->mapDn, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->slots + g.off_wd_codes, I / 2, H, S, I / 2,
                         g.expert_bytes, 64, 128, "down codes (NVFP4)")))
        return rc;
    if ((rc = encode_map(&L->mapXn, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->xq, xrow, moe::kNvTerms, 1, xrow,
                         (uint64_t)moe::kNvTerms * xrow, 128, moe::kNvTerms, "x terms (NVFP4)")))
        return rc;
    L->tcnv = true;
    return MOE_OK;
}

// Scratch and tensor maps of the tensor-core prefill over the staging buffer `stg` (E experts).
int prefill_setup(moe_layer *L, uint8_t *stg) {
    cudaFree(L->pf_block);
    cudaFree(L->stage_atoms);
    L->pf_block = nullptr;
    L->stage_atoms = nullptr;
    L->pf = false;
    if (!L->tc || !stg) return MOE_OK;
    const int E = L->d.num_experts, H = L->d.hidden, I = L->d.inter;
    const int max_routes = L->d.max_tokens * L->d.top_k;
    L->tiles_cap = moe::prefill_tiles_cap(max_routes, E);
    L->rows_cap = L->tiles_cap * 128;
    L->Ipad = (I + 127) / 128 * 128;
    const size_t sz[] = {(size_t)L->rows_cap * L->Hpad,
                         (size_t)L->tiles_cap * L->atl.nks * moe::kTcAtomBytes,
                         (size_t)L->rows_cap * L->Ipad,
                         (size_t)L->tiles_cap * L->atl.nksI * moe::kTcAtomBytes,
                         (size_t)L->rows_cap * H * sizeof(float),
                         (size_t)E * 4, (size_t)E * 4, (size_t)L->tiles_cap * 4, (size_t)L->tiles_cap * 4, 4};
    size_t total = 0;
    for (size_t v : sz) total += align_up(v, 256);
    cudaError_t e = cudaMalloc(&L->pf_block, total);
    if (e == cudaSuccess) e = cudaMalloc(&L->stage_atoms, (size_t)E * L->atl.slot_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        cudaFree(L->pf_block);
        L->pf_block = nullptr;
        return fail(e == cudaErrorMemoryAllocation ? MOE_ENOMEM : MOE_ECUDA, "prefill buffers: %s",
                    cudaGetErrorString(e));
    }
    char *p = static_cast<char *>(L->pf_block);
    void **dst[] = {(void **)&L->XP, (void **)&L->XA, (void **)&L->HP, (void **)&L->HA, (void **)&L->YP,
                    (void **)&L->pf_poff, (void **)&L->pf_e2a, (void **)&L->pf_tile_aidx, (void **)&L->pf_tile_nrows,
                    (void **)&L->pf_ntiles};
    for (size_t i = 0; i < sizeof(sz) / sizeof(sz[0]); ++i) {
        *dst[i] = p;
        p += align_up(sz[i], 256);
    }
    // activation operands start at zero (columns past H or I are never written); unwritten scales are 2^0
    CUDA_TRY(cudaMemset(L->pf_block, 0, total));
    CUDA_TRY(cudaMemset(L->XA, 0x7f, sz[1]));
    CUDA_TRY(cudaMemset(L->HA, 0x7f, sz[3]));
    CUDA_TRY(cudaMemset(L->stage_atoms, 0x7f, (size_t)E * L->atl.slot_bytes));
    const moe::ExpertGeometry &g = L->geo;
    int rc;
    if ((rc = encode_map(&L->mapSG, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, stg + g.off_wg_codes, H / 128 * 128, I, E,
                         H / 2, g.expert_bytes, 128, 128, "staged gate codes")))
        return rc;
    if ((rc = encode_map(&L->mapSU, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, stg + g.off_wu_codes, H / 128 * 128, I, E,
                         H / 2, g.expert_bytes, 128, 128, "staged up codes")))
        return rc;
    if ((rc = encode_map(&L->mapSD, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, stg + g.off_wd_codes, I / 128 * 128, H, E,
                         I / 2, g.expert_bytes, 128, 128, "staged down codes")))
        return rc;
    if ((rc = encode_map(&L->mapXP, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->XP, L->Hpad, L->rows_cap, 1, L->Hpad,
                         (uint64_t)L->rows_cap * L->Hpad, 128, 128, "prefill x")))
        return rc;
    if ((rc = encode_map(&L->mapHP, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->HP, L->Ipad, L->rows_cap, 1, L->Ipad,
                         (uint64_t)L->rows_cap * L->Ipad, 128, 128, "prefill h")))
        return rc;
    L->pf = true;
    return MOE_OK;
}

}  // namespace

void moe::set_last_error(const char *msg) { g_err = msg ? msg : ""; }

extern "C" {

const char *moe_last_error(void) { return g_err.c_str(); }

int moe_layer_create(const moe_layer_desc *desc, const float *router_w_dev, const float *router_bias_dev,
                     const uint8_t *host_bank, const int32_t *expert_to_slot_host, void *stream,
                     moe_layer **out) {
    g_err.clear();
    if (!out) return fail(MOE_EINVAL, "out is NULL");
    *out = nullptr;
    if (!desc || !router_w_dev || !host_bank || !expert_to_slot_host)
        return fail(MOE_EINVAL, "desc, router_w_dev, host_bank and expert_to_slot_host are required");
    const moe_layer_desc d = *desc;
    if (d.hidden <= 0 || d.hidden % 64 || d.inter <= 0 || d.inter % 64)
        return fail(MOE_EINVAL, "hidden and inter must be positive multiples of 64 (got %d, %d)", d.hidden, d.inter);
    if (d.top_k < 1 || d.top_k > moe::kMaxTopK || d.num_experts < d.top_k || d.num_experts > moe::kMaxExperts)
        return fail(MOE_EINVAL, "need 1 <= top_k <= %d and top_k <= num_experts <= %d", moe::kMaxTopK,
                    moe::kMaxExperts);
    if (d.num_slots < d.top_k || d.num_slots > d.num_experts)
        return fail(MOE_EINVAL, "need top_k <= num_slots <= num_experts (got %d)", d.num_slots);
    if (d.max_tokens < 1 || d.max_tokens > moe::kMaxTokens)
        return fail(MOE_EINVAL, "max_tokens must be in [1, %d]", moe::kMaxTokens);
    if (d.out_dtype != MOE_OUT_BF16 && d.out_dtype != MOE_OUT_F32) return fail(MOE_EINVAL, "bad out_dtype");
    if (d.max_refills_per_step < 0 || d.max_refills_per_step > 16)
        return fail(MOE_EINVAL, "max_refills_per_step must be in [0, 16]");
    if (!(d.score_decay > 0.f && d.score_decay <= 1.f)) return fail(MOE_EINVAL, "score_decay must be in (0, 1]");
    if (d.visibility != MOE_VIS_DETERMINISTIC && d.visibility != MOE_VIS_POLLED)
        return fail(MOE_EINVAL, "bad visibility");
    if (d.weight_format != MOE_FMT_MXFP4 && d.weight_format != MOE_FMT_NVFP4)
        return fail(MOE_EINVAL, "bad weight_format %d", d.weight_format);
    const int dec_tokens = d.max_tokens < moe::kDecodeMaxTokens ? d.max_tokens : moe::kDecodeMaxTokens;
    if ((size_t)dec_tokens * d.hidden * sizeof(float) > (size_t)moe::kDecodeSmemLimit)
        return fail(MOE_EINVAL, "hidden %d too large for the decode kernels", d.hidden);

    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, host_bank) != cudaSuccess || pa.type != cudaMemoryTypeHost) {
        cudaGetLastError();
        return fail(MOE_EINVAL, "host_bank must be page-locked host memory (cudaHostAlloc / cudaHostRegister)");
    }
    std::vector<int32_t> e2s(expert_to_slot_host, expert_to_slot_host + d.num_experts);
    std::vector<int32_t> s2e(d.num_slots, -1);
    for (int e = 0; e < d.num_experts; ++e) {
        const int s = e2s[e];
        if (s < -1 || s >= d.num_slots) return fail(MOE_EINVAL, "expert_to_slot[%d] = %d out of range", e, s);
        if (s >= 0) {
            if (s2e[s] >= 0) return fail(MOE_EINVAL, "slot %d given to experts %d and %d", s, s2e[s], e);
            s2e[s] = e;
        }
    }

    moe_layer *L = new moe_layer();
    L->d = d;
    L->host_bank = host_bank;
    L->geo = moe::make_geometry(d.hidden, d.inter, d.weight_format == MOE_FMT_NVFP4 ? 16 : 32);
    L->nchunk = (d.hidden + moe::kRouteChunk - 1) / moe::kRouteChunk;
    L->max_hot = d.max_tokens * d.top_k;
    L->e2s = e2s;
    L->e2s_visible = e2s;
    L->s2e = s2e;
    L->score.assign(d.num_experts, 0.0);
    L->last.assign(d.num_experts, -1);
    L->loaded.assign(d.num_experts, -1);
    L->seg.assign(d.num_experts, 0);
    L->in_flight.assign(d.num_experts, 0);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    auto bail = [&](int code) {
        release(L);
        return code;
    };
#define CREATE_TRY(call)                                                         \
    do {                                                                         \
        cudaError_t _e = (call);                                                 \
        if (_e != cudaSuccess) {                                                 \
            int _c = (_e == cudaErrorMemoryAllocation) ? MOE_ENOMEM : MOE_ECUDA; \
            fail(_c, "%s: %s", #call, cudaGetErrorString(_e));                   \
            cudaGetLastError();                                                  \
            return bail(_c);                                                     \
        }                                                                        \
    } while (0)

    CREATE_TRY(cudaGetDevice(&L->device));
    CREATE_TRY(cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->device));
    const int E = d.num_experts, H = d.hidden, I = d.inter, k = d.top_k, mt = d.max_tokens;
    const size_t eb = L->geo.expert_bytes;
    CREATE_TRY(cudaMalloc(&L->slots, (size_t)d.num_slots * eb));
    CREATE_TRY(cudaMalloc(&L->Wr, (size_t)E * H * sizeof(float)));
    const int E32 = (E + 31) / 32 * 32;
    CREATE_TRY(cudaMalloc(&L->WrT, (size_t)E32 * H * sizeof(float)));
    CREATE_TRY(cudaMalloc(&L->bias, (size_t)E * sizeof(float)));
    CREATE_TRY(cudaMalloc(&L->e2s_dev, (size_t)E * sizeof(int32_t)));
    CREATE_TRY(cudaMalloc(&L->h, (size_t)L->max_hot * I * sizeof(float)));
    {  // the cold routes of a decode step, grouped by expert for the GPU (at most 8 * k of them)
        const int dec = (mt < moe::kDecodeMaxTokens ? mt : moe::kDecodeMaxTokens) * k;
        const size_t l = align_up((size_t)dec * 4, 256);
        CREATE_TRY(cudaMalloc(&L->cold_block, 6 * l + 256 + align_up((size_t)dec * I * 4, 256)));
        char *q = static_cast<char *>(L->cold_block);
        L->c_act_expert = (int32_t *)q;
        L->c_act_off = (int32_t *)(q + l);
        L->c_act_cnt = (int32_t *)(q + 2 * l);
        L->c_token = (int32_t *)(q + 3 * l);
        L->c_w = (float *)(q + 4 * l);
        L->c_counts = (int32_t *)(q + 5 * l);
        L->c_h = (float *)(q + 5 * l + 256);
    }
    {  // the device address of the page-locked bank, when the GPU can read it in place
        void *dp = nullptr;
        if (cudaHostGetDevicePointer(&dp, const_cast<uint8_t *>(host_bank), 0) == cudaSuccess)
            L->host_bank_dev = static_cast<const uint8_t *>(dp);
        else
            cudaGetLastError();  // not mappable: moe_forward_cold_gpu reports it
    }

    // route scratch in one block
    const size_t nh = (size_t)L->max_hot;
    const size_t sizes[] = {
        (size_t)L->nchunk * mt * E * 4,          // logit_part
        (size_t)mt * k * 4, (size_t)mt * k * 4,  // topk ids, w
        nh * 4, nh * 4, nh * 4,                  // hot expert/token/w
        nh * 4, nh * 4, nh * 4, nh * 4,          // act expert/slot/off/cnt
        16,                                      // arrive
        (size_t)((mt + moe::kPfRouteTok - 1) / moe::kPfRouteTok) * E * 4,  // blk_cnt
        (size_t)mt * k * 4};                     // route_rank
    size_t total = 0;
    for (size_t s : sizes) total += align_up(s, 256);
    CREATE_TRY(cudaMalloc(&L->dev_block, total));
    {
        char *p = static_cast<char *>(L->dev_block);
        void **dst[] = {(void **)&L->rb.logit_part, (void **)&L->rb.topk_ids, (void **)&L->rb.topk_w,
                        (void **)&L->rb.hot_expert, (void **)&L->rb.hot_token, (void **)&L->rb.hot_w,
                        (void **)&L->rb.act_expert, (void **)&L->rb.act_slot, (void **)&L->rb.act_off,
                        (void **)&L->rb.act_cnt, (void **)&L->rb.arrive, (void **)&L->rb.blk_cnt,
                        (void **)&L->rb.route_rank};
        for (size_t i = 0; i < sizeof(sizes) / sizeof(sizes[0]); ++i) {
            *dst[i] = p;
            p += align_up(sizes[i], 256);
        }
    }
    CREATE_TRY(cudaMemsetAsync(L->dev_block, 0, total, st));
    // The mirrored arrays: cold routes exist only in decode calls (M <= 8; prefill routes are all hot), so
    // the cold lists hold dec k entries.
    const int dec = mt < moe::kDecodeMaxTokens ? mt : moe::kDecodeMaxTokens;
    const size_t nc = (size_t)dec * k;
    L->mir_off_cold = align_up(16 + (size_t)E * 4, 16);
    L->mir_off_x = L->mir_off_cold + 3 * align_up(nc * 4, 16);
    const size_t mir_bytes = L->mir_off_x + align_up((size_t)dec * H * 2, 16);
    CREATE_TRY(cudaMalloc(&L->mir_block, mir_bytes));
    CREATE_TRY(cudaMemsetAsync(L->mir_block, 0, mir_bytes, st));
    {
        char *p = static_cast<char *>(L->mir_block);
        L->rb.counts = (int32_t *)p;
        L->rb.hist = (int32_t *)(p + 16);
        L->rb.cold_token = (int32_t *)(p + L->mir_off_cold);
        L->rb.cold_expert = (int32_t *)(p + L->mir_off_cold + align_up(nc * 4, 16));
        L->rb.cold_w = (float *)(p + L->mir_off_cold + 2 * align_up(nc * 4, 16));
    }
    // decode on the tensor cores wherever a full 128-column tile exists along H and I
    if (d.hidden >= 128 && d.inter >= 128 && d.weight_format == MOE_FMT_MXFP4) {
        const int rc = tc_setup(L, st);
        if (rc) {
            release(L);
            return rc;
        }
    } else if (d.hidden >= 256 && d.inter >= 128 && d.hidden % 64 == 0 && d.inter % 64 == 0 &&
               d.weight_format == MOE_FMT_NVFP4) {  // NVFP4: one-token decode on the tensor cores
        const int rc = nv_setup(L, st);
        if (rc) {
            release(L);
            return rc;
        }
    }

    // page-locked mirror: the device mirror block's layout, then the cold sums of the decode tokens
    const size_t psz = align_up(mir_bytes, 64) + align_up((size_t)dec * H * 4, 64);
    CREATE_TRY(cudaHostAlloc(&L->pinned_block, psz, cudaHostAllocDefault));
    memset(L->pinned_block, 0, psz);
    {
        char *p = static_cast<char *>(L->pinned_block);
        L->m_counts = (int32_t *)p;
        L->m_hist = (int32_t *)(p + 16);
        L->m_cold_token = (int32_t *)(p + L->mir_off_cold);
        L->m_cold_expert = (int32_t *)(p + L->mir_off_cold + align_up(nc * 4, 16));
        L->m_cold_w = (float *)(p + L->mir_off_cold + 2 * align_up(nc * 4, 16));
        L->m_x = (uint16_t *)(p + L->mir_off_x);
        L->m_ycold = (float *)(p + align_up(mir_bytes, 64));
    }
    CREATE_TRY(cudaMalloc(&L->d_ycold, (size_t)dec * H * 4));

    CREATE_TRY(cudaStreamCreateWithFlags(&L->d2h, cudaStreamNonBlocking));
    CREATE_TRY(cudaStreamCreateWithFlags(&L->h2d, cudaStreamNonBlocking));
    CREATE_TRY(cudaEventCreateWithFlags(&L->ev_cold, cudaEventDisableTiming));
    for (cudaEvent_t *e : {&L->ev_fork, &L->ev_route, &L->ev_fence})
        CREATE_TRY(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
    L->ev_copy.resize(d.max_refills_per_step);
    for (auto &e : L->ev_copy) CREATE_TRY(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));

    CREATE_TRY(cudaMemcpyAsync(L->Wr, router_w_dev, (size_t)E * H * sizeof(float), cudaMemcpyDeviceToDevice, st));
    CREATE_TRY(moe::launch_router_transpose(L->Wr, L->WrT, E, H, (E + 31) / 32 * 32, st));
    if (router_bias_dev)
        CREATE_TRY(cudaMemcpyAsync(L->bias, router_bias_dev, (size_t)E * sizeof(float), cudaMemcpyDeviceToDevice, st));
    else
        CREATE_TRY(cudaMemsetAsync(L->bias, 0, (size_t)E * sizeof(float), st));
    CREATE_TRY(cudaMemcpyAsync(L->e2s_dev, e2s.data(), (size_t)E * sizeof(int32_t), cudaMemcpyHostToDevice, st));
    for (int e = 0; e < E; ++e)
        if (e2s[e] >= 0)
            CREATE_TRY(cudaMemcpyAsync(L->slots + (size_t)e2s[e] * eb, host_bank + (size_t)e * eb, eb,
                                       cudaMemcpyHostToDevice, st));
    for (int e = 0; e < E; ++e)
        if (e2s[e] >= 0) {
            const int rc = build_slot_atoms(L, e2s[e], st);
            if (rc) {
                cudaStreamSynchronize(st);
                release(L);
                return rc;
            }
        }
    CREATE_TRY(cudaStreamSynchronize(st));
#undef CREATE_TRY
    *out = L;
    return MOE_OK;
}

int moe_route(moe_layer *L, const void *x_dev, int32_t M, void *stream, moe_route_result *res) {
    g_err.clear();
    if (!L || !x_dev) return fail(MOE_EINVAL, "layer and x_dev are required");
    if (M < 1 || M > L->d.max_tokens) return fail(MOE_EINVAL, "M = %d outside [1, max_tokens=%d]", M, L->d.max_tokens);
    if (reinterpret_cast<uintptr_t>(x_dev) % 16) return fail(MOE_EINVAL, "x_dev must be 16-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int E = L->d.num_experts, k = L->d.top_k;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    unsigned long long cid = 0;
    CUDA_TRY(cudaStreamGetCaptureInfo(st, &cs, &cid));
    const bool capturing = cs == cudaStreamCaptureStatusActive;
    // the previous mirror copy of this layer has read the route buffers before this launch rewrites them
    if (!capturing) {
        CUDA_TRY(cudaStreamWaitEvent(st, L->ev_route, 0));
    } else if (L->cap_mirror && L->cap_id == cid) {
        CUDA_TRY(cudaStreamUpdateCaptureDependencies(st, &L->cap_mirror, nullptr, 1, cudaStreamAddCaptureDependencies));
    }
    moe::RouteParams p{};
    p.x = static_cast<const uint16_t *>(x_dev);
    p.Wr = L->Wr;
    p.WrT = L->WrT;
    p.E32 = (L->d.num_experts + 31) / 32 * 32;
    p.bias = L->bias;
    p.e2s = L->e2s_dev;
    p.M = M;
    p.H = L->d.hidden;
    p.E = E;
    p.k = k;
    p.nchunk = L->nchunk;
    p.all_hot = M > moe::kDecodeMaxTokens;
    p.act_pad = M <= moe::kDecodeMaxTokens ? act_cap(L, M) : 0;
    p.b = L->rb;
    if (L->tc && M <= moe::kDecodeMaxTokens) {  // the route launch also writes the gate/up B operand
        p.xq = L->xq;
        p.xat = L->xat;
        p.Hpad = L->Hpad;
        p.xmir = reinterpret_cast<uint16_t *>(static_cast<char *>(L->mir_block) + L->mir_off_x);  // and copies x
    }
    if (L->tcnv && M == 1 && L->ffn1) {  // NVFP4: x as E2M1 terms for the one-token tensor-core FFN
        p.xq = L->xq;
        p.xat = L->xat;
        p.xnv = 1;
        p.xg = L->nv_xg;
        p.Hpad4 = L->Hpad4;
        p.xmir = reinterpret_cast<uint16_t *>(static_cast<char *>(L->mir_block) + L->mir_off_x);
    }
    if (M > moe::kDecodeMaxTokens && L->pf) {  // the route launch also plans the prefill GEMM tiles
        p.pf_poff = L->pf_poff;
        p.pf_e2a = L->pf_e2a;
        p.pf_tile_aidx = L->pf_tile_aidx;
        p.pf_tile_nrows = L->pf_tile_nrows;
        p.pf_ntiles = L->pf_ntiles;
        p.pf_tiles_cap = moe::prefill_tiles_cap(M * k, E);
    }
    const bool table = L->dev_cache && M <= moe::kDecodeMaxTokens;
    if (table) p.lru = L->lru;  // the route launch assigns slots to this step's misses
    L->routed_plan = false;
    CUDA_TRY(prof_mark(L, 0, st));
    CUDA_TRY(moe::launch_route(p, st, L->num_sms));
    if (table) {  // and the fill kernel copies them in before anything later on the stream runs
        moe::FillLaunch F{};
        F.bank = L->host_bank_dev;
        F.slots = L->slots;
        F.atoms = L->tc ? L->atoms : nullptr;
        F.geo = L->geo;
        F.fill_expert = L->lru.fill_expert;
        F.fill_slot = L->lru.fill_slot;
        F.n_fill = L->lru.n_fill;
        F.grid = 2 * L->num_sms;
        CUDA_TRY(moe::launch_slot_fill(F, st));
    }
    CUDA_TRY(prof_mark(L, 0, st));

    // mirror counts, histogram, cold triples and (decode) x to page-locked memory off the compute chain, in
    // one copy of the mirror block: a prefill call has only counts and histogram (every route is hot); the
    // route launch copied x into the block when it wrote the x terms, else x is copied on its own
    // Nothing on `stream` waits for the copy: the compute chain of the next calls stays kernel after kernel.
    const bool dec_call = M <= moe::kDecodeMaxTokens;
    const size_t mbytes = !dec_call ? 16 + (size_t)E * 4 : p.xmir ? L->mir_off_x + (size_t)M * L->d.hidden * 2
                                                                  : L->mir_off_x;
    const bool copy_x = dec_call && !p.xmir;  // the host computes cold routes from this copy (moe_forward_cold)
    if (capturing) {
        cudaGraph_t g = nullptr;
        const cudaGraphNode_t *deps = nullptr;
        const cudaGraphEdgeData *edges = nullptr;
        size_t nd = 0;
        CUDA_TRY(cudaStreamGetCaptureInfo(st, &cs, &cid, &g, &deps, &edges, &nd));
        cudaGraphNode_t node = nullptr;
        CUDA_TRY(cudaGraphAddMemcpyNode1D(&node, g, deps, nd, L->pinned_block, L->mir_block, mbytes,
                                          cudaMemcpyDeviceToHost));
        if (copy_x) {
            cudaGraphNode_t xn = nullptr;
            CUDA_TRY(cudaGraphAddMemcpyNode1D(&xn, g, &node, 1, L->m_x, x_dev, (size_t)M * L->d.hidden * 2,
                                              cudaMemcpyDeviceToHost));
            node = xn;
        }
        L->cap_mirror = node;
        L->cap_id = cid;
    } else {
        CUDA_TRY(cudaEventRecord(L->ev_fork, st));
        CUDA_TRY(cudaStreamWaitEvent(L->d2h, L->ev_fork, 0));
        CUDA_TRY(cudaMemcpyAsync(L->pinned_block, L->mir_block, mbytes, cudaMemcpyDeviceToHost, L->d2h));
        if (copy_x) CUDA_TRY(cudaMemcpyAsync(L->m_x, x_dev, (size_t)M * L->d.hidden * 2, cudaMemcpyDeviceToHost, L->d2h));
        CUDA_TRY(cudaEventRecord(L->ev_route, L->d2h));
    }

    L->routed_x = x_dev;
    L->routed_M = M;
    L->routed_plan = p.pf_poff != nullptr;
    L->route_seq++;
    if (res) {
        res->M = M;
        res->topk_ids = L->rb.topk_ids;
        res->topk_w = L->rb.topk_w;
        res->hot_expert = L->rb.hot_expert;
        res->hot_token = L->rb.hot_token;
        res->hot_w = L->rb.hot_w;
        res->act_expert = L->rb.act_expert;
        res->act_slot = L->rb.act_slot;
        res->act_off = L->rb.act_off;
        res->act_cnt = L->rb.act_cnt;
        res->cold_token = L->rb.cold_token;
        res->cold_expert = L->rb.cold_expert;
        res->cold_w = L->rb.cold_w;
        res->hist = L->rb.hist;
        res->counts = L->rb.counts;
        res->h_counts = L->m_counts;
        res->h_cold_token = L->m_cold_token;
        res->h_cold_expert = L->m_cold_expert;
        res->h_cold_w = L->m_cold_w;
        res->h_hist = L->m_hist;
        res->done = L->ev_route;
    }
    return MOE_OK;
}

int moe_forward_slots(moe_layer *L, const void *x_dev, void *out_dev, int32_t M, void *stream) {
    g_err.clear();
    if (!L || !x_dev || !out_dev) return fail(MOE_EINVAL, "layer, x_dev and out_dev are required");
    if (L->routed_M == 0 || L->routed_x != x_dev || L->routed_M != M)
        return fail(MOE_ESTATE, "moe_forward_slots needs the x_dev and M of the last moe_route");
    if (reinterpret_cast<uintptr_t>(out_dev) % 16) return fail(MOE_EINVAL, "out_dev must be 16-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    moe::DecodeParams p{};
    p.geo = L->geo;
    p.x = static_cast<const uint16_t *>(x_dev);
    p.counts = L->rb.counts;
    p.act_slot = L->rb.act_slot;
    p.act_off = L->rb.act_off;
    p.act_cnt = L->rb.act_cnt;
    p.hot_token = L->rb.hot_token;
    p.hot_w = L->rb.hot_w;
    p.h = L->h;
    p.out = out_dev;
    p.out_f32 = L->d.out_dtype == MOE_OUT_F32;
    if (M == 1 && L->tcnv && L->ffn1) {  // NVFP4: gate/up, SiLU and down in one launch, then the combine
        moe::NvLaunch n{};
        n.bank = L->slots;
        n.atoms = L->atoms;
        n.geo = L->geo;
        n.n_act_max = act_cap(L, 1);
        n.ks = choose_splits(n.n_act_max * L->nvl.ntI, L->nvl.nks4, L->num_sms);
        n.counts = L->rb.counts;
        n.act_slot = L->rb.act_slot;
        n.act_off = L->rb.act_off;
        n.act_cnt = L->rb.act_cnt;
        n.hot_token = L->rb.hot_token;
        n.hot_w = L->rb.hot_w;
        n.xat = L->xat;
        n.xg = L->nv_xg;
        n.part = L->part;
        n.err = L->err;
        n.mapG = &L->mapGn;
        n.mapU = &L->mapUn;
        n.mapX = &L->mapXn;
        n.mapD = &L->mapDn;
        moe::TcLaunch t{};  // the combine's arguments
        t.geo = L->geo;
        t.n_act_max = n.n_act_max;
        t.counts = L->rb.counts;
        t.part = L->part;
        t.out = out_dev;
        t.out_f32 = p.out_f32;
        CUDA_TRY(prof_mark(L, 1, st));
        CUDA_TRY(moe::launch_ffn_nv(n, st));
        CUDA_TRY(prof_mark(L, 1, st));
        CUDA_TRY(prof_mark(L, 2, st));
        CUDA_TRY(moe::launch_ffn_combine(t, st));
        CUDA_TRY(prof_mark(L, 2, st));
    } else if (M <= moe::kDecodeMaxTokens && L->tc) {
        moe::TcLaunch t{};
        t.bank = L->slots;
        t.geo = L->geo;
        t.M = M;
        t.n_act_max = act_cap(L, M);
        t.ks_gateup = tc_splits_gateup(L, M);
        t.ks_down = tc_splits_down(L, M);
        t.counts = L->rb.counts;
        t.act_slot = L->rb.act_slot;
        t.act_off = L->rb.act_off;
        t.act_cnt = L->rb.act_cnt;
        t.hot_token = L->rb.hot_token;
        t.hot_w = L->rb.hot_w;
        t.atoms = L->atoms;
        t.xat = L->xat;
        t.hq = L->hq;
        t.hat = L->hat;
        t.Ipad = L->Ipad;
        t.err = L->err;
        t.out = out_dev;
        t.out_f32 = p.out_f32;
        t.mapG = &L->mapG;
        t.mapU = &L->mapU;
        t.mapX = &L->mapX;
        t.mapD = &L->mapD;
        t.mapH = &L->mapH;
        t.part = L->part;
        if (M == 1 && L->ffn1) {  // gate/up, SiLU and down in one launch, then the combine
            CUDA_TRY(prof_mark(L, 1, st));
            CUDA_TRY(moe::launch_ffn_tc(t, st));
            CUDA_TRY(prof_mark(L, 1, st));
            CUDA_TRY(prof_mark(L, 2, st));
            CUDA_TRY(moe::launch_ffn_combine(t, st));
            CUDA_TRY(prof_mark(L, 2, st));
        } else {
            CUDA_TRY(prof_mark(L, 1, st));
            CUDA_TRY(moe::launch_gateup_tc(t, st));
            CUDA_TRY(prof_mark(L, 1, st));
            CUDA_TRY(prof_mark(L, 2, st));
            CUDA_TRY(moe::launch_down_tc(t, st));
            CUDA_TRY(prof_mark(L, 2, st));
        }
    } else if (M <= moe::kDecodeMaxTokens) {
        p.bank = L->slots;
        CUDA_TRY(prof_mark(L, 1, st));
        moe::launch_gateup(p, M, st, L->num_sms);
        CUDA_TRY(cudaGetLastError());
        CUDA_TRY(prof_mark(L, 1, st));
        CUDA_TRY(prof_mark(L, 2, st));
        moe::launch_down(p, M, st, L->num_sms);
        CUDA_TRY(cudaGetLastError());
        CUDA_TRY(prof_mark(L, 2, st));
    } else {
        if (!L->staging || !L->staged)
            return fail(MOE_ESTATE, "prefill (M > %d) needs a staging buffer filled by moe_layer_stage_all",
                        moe::kDecodeMaxTokens);
        if (!L->pf)
            return fail(MOE_ESTATE, "prefill needs hidden and inter of at least 128 (tensor-core tiles)");
        if (!L->routed_plan)
            return fail(MOE_ESTATE, "prefill needs a moe_route call made after the staging buffer was attached");
        moe::PrefillLaunch P{};
        P.bank = L->staging;
        P.atoms = L->stage_atoms;
        P.geo = L->geo;
        P.E = L->d.num_experts;
        P.k = L->d.top_k;
        P.M = M;
        P.max_routes = M * L->d.top_k;
        P.tiles_cap = moe::prefill_tiles_cap(P.max_routes, P.E);
        P.num_sms = L->num_sms;
        P.Hpad = L->Hpad;
        P.Ipad = L->Ipad;
        P.x = p.x;
        P.counts = L->rb.counts;
        P.act_expert = L->rb.act_expert;
        P.act_off = L->rb.act_off;
        P.act_cnt = L->rb.act_cnt;
        P.hot_expert = L->rb.hot_expert;
        P.hot_token = L->rb.hot_token;
        P.topk_ids = L->rb.topk_ids;
        P.route_pos = L->rb.route_rank;
        P.hot_w = L->rb.hot_w;
        P.poff = L->pf_poff;
        P.e2a = L->pf_e2a;
        P.tile_aidx = L->pf_tile_aidx;
        P.tile_nrows = L->pf_tile_nrows;
        P.ntiles = L->pf_ntiles;
        P.XP = L->XP;
        P.XA = L->XA;
        P.HP = L->HP;
        P.HA = L->HA;
        P.YP = L->YP;
        P.err = L->err;
        P.out = out_dev;
        P.out_f32 = p.out_f32;
        P.mapXP = &L->mapXP;
        P.mapHP = &L->mapHP;
        P.mapG = &L->mapSG;
        P.mapU = &L->mapSU;
        P.mapD = &L->mapSD;
        P.ev[0] = prof_next(L, 1);  // gate/up GEMM
        P.ev[1] = prof_next(L, 1);
        P.ev[2] = prof_next(L, 2);  // down GEMM
        P.ev[3] = prof_next(L, 2);
        CUDA_TRY(moe::launch_prefill(P, st));
    }
    return MOE_OK;
}

int moe_layer_set_device_cache(moe_layer *L, int32_t enable) {
    g_err.clear();
    if (!L) return fail(MOE_EINVAL, "layer is NULL");
    const int E = L->d.num_experts, S = L->d.num_slots;
    if (enable && L->d.weight_format != MOE_FMT_MXFP4) return fail(MOE_EINVAL, "the device slot table is MXFP4 only");
    if (enable && !L->dev_cache) {
        if (!L->host_bank_dev) return fail(MOE_ESTATE, "the GPU cannot address the host bank in place");
        if (reinterpret_cast<uintptr_t>(L->host_bank_dev) % 16)
            return fail(MOE_EINVAL, "the host bank must be 16-byte aligned for the device slot table");
        // every copy the host policy issued has landed once the device is idle: its map is the slots' content
        CUDA_TRY(cudaDeviceSynchronize());
        for (auto &pc : L->pending) {
            L->in_flight[pc.expert] = 0;
            L->ev_pool.push_back(pc.ev);
        }
        L->pending.clear();
        const size_t l = align_up((size_t)S * 4, 256), f = align_up((size_t)moe::kMaxFill * 4, 256);
        if (!L->lru_block) {
            CUDA_TRY(cudaMalloc(&L->lru_block, 2 * l + 2 * f + 512));
            char *q = static_cast<char *>(L->lru_block);
            L->lru.e2s = L->e2s_dev;
            L->lru.s2e = (int32_t *)q;
            L->lru.stamp = (int32_t *)(q + l);
            L->lru.fill_expert = (int32_t *)(q + 2 * l);
            L->lru.fill_slot = (int32_t *)(q + 2 * l + f);
            L->lru.clock = (int32_t *)(q + 2 * l + 2 * f);
            L->lru.n_fill = (int32_t *)(q + 2 * l + 2 * f + 4);
            L->lru.stats = (unsigned long long *)(q + 2 * l + 2 * f + 256);
            L->lru.S = S;
        }
        std::vector<int32_t> stamp((size_t)S, -1);
        const int32_t zero2[2] = {0, 0};
        const unsigned long long zero4[4] = {0, 0, 0, 0};
        CUDA_TRY(cudaMemcpy(L->e2s_dev, L->e2s.data(), (size_t)E * 4, cudaMemcpyHostToDevice));
        CUDA_TRY(cudaMemcpy(L->lru.s2e, L->s2e.data(), (size_t)S * 4, cudaMemcpyHostToDevice));
        CUDA_TRY(cudaMemcpy(L->lru.stamp, stamp.data(), (size_t)S * 4, cudaMemcpyHostToDevice));
        CUDA_TRY(cudaMemcpy(L->lru.clock, zero2, sizeof(zero2), cudaMemcpyHostToDevice));
        CUDA_TRY(cudaMemcpy(L->lru.stats, zero4, sizeof(zero4), cudaMemcpyHostToDevice));
        L->e2s_visible = L->e2s;
        L->dev_cache = true;
    } else if (!enable && L->dev_cache) {
        // the host policy takes over the device's map
        CUDA_TRY(cudaDeviceSynchronize());
        CUDA_TRY(cudaMemcpy(L->e2s.data(), L->e2s_dev, (size_t)E * 4, cudaMemcpyDeviceToHost));
        CUDA_TRY(cudaMemcpy(L->s2e.data(), L->lru.s2e, (size_t)S * 4, cudaMemcpyDeviceToHost));
        L->e2s_visible = L->e2s;
        L->seg.assign(E, 0);  // SLRU segments start over from the device's map
        L->policy_seq = L->route_seq;  // the last route's decision was the device's
        L->dev_cache = false;
    }
    return MOE_OK;
}

int moe_layer_set_policy(moe_layer *L, int32_t policy) {
    g_err.clear();
    if (!L) return fail(MOE_EINVAL, "layer is NULL");
    if (policy != MOE_POLICY_FREQ && policy != MOE_POLICY_LRU && policy != MOE_POLICY_FIFO &&
        policy != MOE_POLICY_SLRU)
        return fail(MOE_EINVAL, "unknown policy %d", policy);
    L->policy = policy;
    return MOE_OK;
}

int moe_forward_cold(moe_layer *L, const void *x_dev, void *out_dev, int32_t M, int32_t nthreads, void *stream) {
    g_err.clear();
    if (!L || !x_dev || !out_dev) return fail(MOE_EINVAL, "layer, x_dev and out_dev are required");
    if (nthreads < 0) return fail(MOE_EINVAL, "nthreads must be >= 0 (0: every host core)");
    if (L->d.weight_format != MOE_FMT_MXFP4) return fail(MOE_EINVAL, "moe_forward_cold is MXFP4 only");
    if (L->routed_M == 0 || L->routed_x != x_dev || L->routed_M != M)
        return fail(MOE_ESTATE, "moe_forward_cold needs the x_dev and M of the last moe_route");
    if (M > moe::kDecodeMaxTokens) return MOE_OK;  // prefill: every route is hot
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUDA_TRY(cudaEventSynchronize(L->ev_cold));   // the previous sums have left m_ycold
    CUDA_TRY(cudaEventSynchronize(L->ev_route));  // counts, cold triples and x are on the host
    const int n_cold = L->m_counts[1];
    if (n_cold == 0) return MOE_OK;
    moe::host::ColdJob job{};
    job.L = moe::host::record_layout(L->d.hidden, L->d.inter);
    job.bank = L->host_bank;
    job.x = L->m_x;
    job.M = M;
    job.n = n_cold;
    job.token = L->m_cold_token;
    job.expert = L->m_cold_expert;
    job.w = L->m_cold_w;
    job.y = L->m_ycold;
    moe::host::run_cold(job, nthreads);
    const size_t n = (size_t)M * L->d.hidden;
    CUDA_TRY(cudaMemcpyAsync(L->d_ycold, L->m_ycold, n * 4, cudaMemcpyHostToDevice, st));
    CUDA_TRY(cudaEventRecord(L->ev_cold, st));
    add_cold_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(out_dev, L->d_ycold, (int)n,
                                                                 L->d.out_dtype == MOE_OUT_F32);
    CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int moe_forward_cold_gpu(moe_layer *L, const void *x_dev, void *out_dev, int32_t M, void *stream) {
    g_err.clear();
    if (!L || !x_dev || !out_dev) return fail(MOE_EINVAL, "layer, x_dev and out_dev are required");
    if (L->routed_M == 0 || L->routed_x != x_dev || L->routed_M != M)
        return fail(MOE_ESTATE, "moe_forward_cold_gpu needs the x_dev and M of the last moe_route");
    if (L->d.weight_format != MOE_FMT_MXFP4) return fail(MOE_EINVAL, "moe_forward_cold_gpu is MXFP4 only");
    if (M > moe::kDecodeMaxTokens) return MOE_OK;  // prefill: every route is hot
    if (!L->host_bank_dev)
        return fail(MOE_ESTATE, "the GPU cannot address the host bank in place (cudaHostGetDevicePointer failed)");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cold_lists_kernel<<<1, 128, 0, st>>>(L->rb.counts, L->rb.cold_token, L->rb.cold_expert, L->rb.cold_w,
                                         L->c_act_expert, L->c_act_off, L->c_act_cnt, L->c_token, L->c_w,
                                         L->c_counts);
    CUDA_TRY(cudaGetLastError());
    moe::DecodeParams p{};
    p.bank = L->host_bank_dev;  // "slot" = expert id: the bank is indexed by expert
    p.geo = L->geo;
    p.x = static_cast<const uint16_t *>(x_dev);
    p.counts = L->c_counts;
    p.act_slot = L->c_act_expert;
    p.act_off = L->c_act_off;
    p.act_cnt = L->c_act_cnt;
    p.hot_token = L->c_token;
    p.hot_w = L->c_w;
    p.h = L->c_h;
    p.out = L->d_ycold;
    p.out_f32 = 1;
    moe::launch_gateup(p, M, st, L->num_sms);
    moe::launch_down(p, M, st, L->num_sms);
    const size_t n = (size_t)M * L->d.hidden;
    add_cold_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(out_dev, L->d_ycold, (int)n,
                                                                 L->d.out_dtype == MOE_OUT_F32);
    CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int moe_host_expert_ffn(const uint8_t *record, int32_t H, int32_t I, const uint16_t *x_host, float *y_host) {
    g_err.clear();
    if (!record || !x_host || !y_host) return fail(MOE_EINVAL, "record, x_host and y_host are required");
    if (H <= 0 || H % 64 || I <= 0 || I % 64) return fail(MOE_EINVAL, "H and I must be positive multiples of 64");
    std::vector<float> h((size_t)I);
    moe::host::expert_ffn(moe::host::record_layout(H, I), record, x_host, h.data(), y_host);
    return MOE_OK;
}

// Copies pairs (expert pe[i] into slot ps[i], replacing pv[i]) from the host bank on the side stream and
// makes them visible as the layer's visibility mode says (shared by the slot policy and the prefetch).
static int issue_refills(moe_layer *L, int n, const int32_t *pe, const int32_t *ps, const int32_t *pv,
                         cudaStream_t st) {
    if (n == 0) return MOE_OK;
    const size_t eb = L->geo.expert_bytes;
    std::vector<int32_t> unmap_e, unmap_s, map_e, map_s;
    for (int i = 0; i < n; ++i) {
        unmap_e.push_back(pv[i]);
        unmap_s.push_back(-1);
    }
    if (L->d.visibility == MOE_VIS_POLLED) {
        // victims leave the map in stream order before their slots are overwritten
        int rc = enqueue_map(L, unmap_e, unmap_s, st);
        if (rc) return rc;
    }
    // everything already on the compute stream (including reads of the victims' slots) precedes the copies
    CUDA_TRY(cudaEventRecord(L->ev_fence, st));
    CUDA_TRY(cudaStreamWaitEvent(L->h2d, L->ev_fence, 0));
    for (int i = 0; i < n; ++i) {
        CUDA_TRY(cudaMemcpyAsync(L->slots + (size_t)ps[i] * eb, L->host_bank + (size_t)pe[i] * eb, eb,
                                 cudaMemcpyHostToDevice, L->h2d));
        if (int rc = build_slot_atoms(L, ps[i], L->h2d)) return rc;
        L->stats[0] += 1;
        L->stats[1] += (int64_t)eb;
        if (L->d.visibility == MOE_VIS_DETERMINISTIC) {
            CUDA_TRY(cudaEventRecord(L->ev_copy[i], L->h2d));
            CUDA_TRY(cudaStreamWaitEvent(st, L->ev_copy[i], 0));
        } else {
            cudaEvent_t ev;
            if (L->ev_pool.empty()) {
                CUDA_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
            } else {
                ev = L->ev_pool.back();
                L->ev_pool.pop_back();
            }
            CUDA_TRY(cudaEventRecord(ev, L->h2d));
            L->pending.push_back({pe[i], ps[i], ev});
            L->in_flight[pe[i]] = 1;
        }
    }
    if (L->d.visibility == MOE_VIS_DETERMINISTIC) {
        map_e = unmap_e;
        map_s = unmap_s;
        for (int i = 0; i < n; ++i) {
            map_e.push_back(pe[i]);
            map_s.push_back(ps[i]);
        }
        int rc = enqueue_map(L, map_e, map_s, st);
        if (rc) return rc;
    }
    return MOE_OK;
}

int moe_cache_update(moe_layer *L, void *stream, int32_t *n_refills_out) {
    g_err.clear();
    if (n_refills_out) *n_refills_out = 0;
    if (!L) return fail(MOE_EINVAL, "layer is NULL");
    const int E = L->d.num_experts, S = L->d.num_slots;
    if (L->dev_cache) return fail(MOE_ESTATE, "the device slot table owns the slots (moe_layer_set_device_cache)");
    if (S >= E) return MOE_OK;  // every expert resident: nothing to refill
    if (L->route_seq == L->policy_seq)
        return fail(MOE_ESTATE, "moe_cache_update needs a moe_route since the last update");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUDA_TRY(cudaEventSynchronize(L->ev_route));
    L->policy_seq = L->route_seq;

    // polled mode: map the experts whose copies have landed
    if (L->d.visibility == MOE_VIS_POLLED && !L->pending.empty()) {
        std::vector<int32_t> ex, sl;
        std::vector<PendingCopy> still;
        for (auto &pc : L->pending) {
            cudaError_t q = cudaEventQuery(pc.ev);
            if (q == cudaSuccess) {
                ex.push_back(pc.expert);
                sl.push_back(pc.slot);
                L->in_flight[pc.expert] = 0;
                L->ev_pool.push_back(pc.ev);
            } else if (q == cudaErrorNotReady) {
                still.push_back(pc);
            } else {
                return fail(MOE_ECUDA, "refill copy failed: %s", cudaGetErrorString(q));
            }
        }
        L->pending.swap(still);
        int rc = enqueue_map(L, ex, sl, st);
        if (rc) return rc;
    }

    const int R = L->d.max_refills_per_step;
    std::vector<int32_t> pe(R > 0 ? R : 1), ps(pe.size()), pv(pe.size());
    // the decision runs on copies so that an injected fault leaves the state unchanged
    std::vector<double> score = L->score;
    std::vector<int64_t> last = L->last, loaded = L->loaded;
    std::vector<uint8_t> seg = L->seg;
    std::vector<int32_t> e2s = L->e2s, s2e = L->s2e;
    const int n =
        L->policy == MOE_POLICY_FREQ
            ? moe_policy_step(score.data(), last.data(), e2s.data(), s2e.data(), E, S, L->m_hist, L->step,
                              (double)L->d.score_decay, R, L->in_flight.data(), pe.data(), ps.data(), pv.data())
        : L->policy == MOE_POLICY_SLRU
            ? moe_policy_step_slru(score.data(), last.data(), seg.data(), e2s.data(), s2e.data(), E, S, L->m_hist,
                                   L->step, (double)L->d.score_decay, R, (4 * S) / 5, L->in_flight.data(), pe.data(),
                                   ps.data(), pv.data())
            : moe_policy_step_recency(L->policy, score.data(), last.data(), loaded.data(), e2s.data(), s2e.data(), E,
                                      S, L->m_hist, L->step, (double)L->d.score_decay, R, L->in_flight.data(),
                                      pe.data(), ps.data(), pv.data());
    if (n < 0) return fail(MOE_EINVAL, "policy rejected its arguments");
    if (n > 0 && L->fault == MOE_FAULT_COPY) {
        L->fault = MOE_FAULT_NONE;
        return fail(MOE_ECUDA, "injected refill copy failure (no copy issued, map unchanged)");
    }
    L->score.swap(score);
    L->last.swap(last);
    L->loaded.swap(loaded);
    L->seg.swap(seg);
    L->e2s.swap(e2s);
    L->s2e.swap(s2e);
    L->step++;
    L->stats[2] += (int64_t)L->routed_M * L->d.top_k;
    L->stats[3] += L->m_counts[0];

    if (int rc = issue_refills(L, n, pe.data(), ps.data(), pv.data(), st)) return rc;
    if (n_refills_out) *n_refills_out = n;
    return MOE_OK;
}

// Scratch of the prediction launch, allocated at the first moe_prefetch of a layer.
static int prefetch_setup(moe_layer *L) {
    const int E = L->d.num_experts, k = L->d.top_k, dec = moe::kDecodeMaxTokens;
    const size_t nh = (size_t)dec * k;
    const size_t sizes[] = {(size_t)L->nchunk * dec * E * 4,     // logit_part
                            nh * 4, nh * 4,                     // topk ids, w
                            nh * 4, nh * 4, nh * 4,             // hot expert/token/w
                            nh * 4, nh * 4, nh * 4, nh * 4,     // act expert/slot/off/cnt
                            nh * 4, nh * 4, nh * 4,             // cold token/expert/w
                            (size_t)E * 4, 16, 16};             // hist, counts, arrive
    size_t total = 0;
    for (size_t z : sizes) total += align_up(z, 256);
    cudaError_t e = cudaMalloc(&L->pred_block, total);
    if (e == cudaSuccess) e = cudaMemset(L->pred_block, 0, total);
    if (e == cudaSuccess) e = cudaHostAlloc(&L->m_pred, (size_t)E * 4, cudaHostAllocDefault);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&L->ev_pred, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&L->ev_pfork, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(e == cudaErrorMemoryAllocation ? MOE_ENOMEM : MOE_ECUDA, "prefetch scratch: %s",
                    cudaGetErrorString(e));
    }
    char *q = static_cast<char *>(L->pred_block);
    void **dst[] = {(void **)&L->prb.logit_part, (void **)&L->prb.topk_ids, (void **)&L->prb.topk_w,
                    (void **)&L->prb.hot_expert, (void **)&L->prb.hot_token, (void **)&L->prb.hot_w,
                    (void **)&L->prb.act_expert, (void **)&L->prb.act_slot, (void **)&L->prb.act_off,
                    (void **)&L->prb.act_cnt, (void **)&L->prb.cold_token, (void **)&L->prb.cold_expert,
                    (void **)&L->prb.cold_w, (void **)&L->prb.hist, (void **)&L->prb.counts, (void **)&L->prb.arrive};
    for (size_t i = 0; i < sizeof(sizes) / sizeof(sizes[0]); ++i) {
        *dst[i] = q;
        q += align_up(sizes[i], 256);
    }
    return MOE_OK;
}

int moe_prefetch(moe_layer *L, const void *x_dev, int32_t M, void *stream, int32_t *n_refills_out) {
    g_err.clear();
    if (n_refills_out) *n_refills_out = 0;
    if (!L || !x_dev) return fail(MOE_EINVAL, "layer and x_dev are required");
    const int dec = L->d.max_tokens < moe::kDecodeMaxTokens ? L->d.max_tokens : moe::kDecodeMaxTokens;
    if (M < 1 || M > dec) return fail(MOE_EINVAL, "M = %d outside [1, %d] (decode calls)", M, dec);
    if (reinterpret_cast<uintptr_t>(x_dev) % 16) return fail(MOE_EINVAL, "x_dev must be 16-byte aligned");
    if (L->dev_cache) return fail(MOE_ESTATE, "the device slot table owns the slots (moe_layer_set_device_cache)");
    const int E = L->d.num_experts, S = L->d.num_slots;
    if (S >= E) return MOE_OK;  // every expert resident: nothing to prefetch
    if (!L->pred_block)
        if (int rc = prefetch_setup(L)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // the prediction: this layer's routing of x, on the side stream (the compute stream goes on meanwhile)
    moe::RouteParams p{};
    p.x = static_cast<const uint16_t *>(x_dev);
    p.Wr = L->Wr;
    p.WrT = L->WrT;
    p.E32 = (E + 31) / 32 * 32;
    p.bias = L->bias;
    p.e2s = L->e2s_dev;
    p.M = M;
    p.H = L->d.hidden;
    p.E = E;
    p.k = L->d.top_k;
    p.nchunk = L->nchunk;
    p.b = L->prb;
    CUDA_TRY(cudaEventRecord(L->ev_pfork, st));
    CUDA_TRY(cudaStreamWaitEvent(L->d2h, L->ev_pfork, 0));
    CUDA_TRY(moe::launch_route(p, L->d2h, L->num_sms));
    CUDA_TRY(cudaMemcpyAsync(L->m_pred, L->prb.hist, (size_t)E * 4, cudaMemcpyDeviceToHost, L->d2h));
    CUDA_TRY(cudaEventRecord(L->ev_pred, L->d2h));
    CUDA_TRY(cudaEventSynchronize(L->ev_pred));

    const int R = L->d.max_refills_per_step;
    std::vector<int32_t> pe(R > 0 ? R : 1), ps(pe.size()), pv(pe.size());
    std::vector<int32_t> e2s = L->e2s, s2e = L->s2e;
    const int n = moe_prefetch_step(L->score.data(), L->last.data(), e2s.data(), s2e.data(), E, S, L->m_pred, R,
                                    L->in_flight.data(), pe.data(), ps.data(), pv.data());
    if (n < 0) return fail(MOE_EINVAL, "prefetch policy rejected its arguments");
    if (n > 0 && L->fault == MOE_FAULT_COPY) {
        L->fault = MOE_FAULT_NONE;
        return fail(MOE_ECUDA, "injected refill copy failure (no copy issued, map unchanged)");
    }
    L->e2s.swap(e2s);
    L->s2e.swap(s2e);
    for (int i = 0; i < n; ++i) L->seg[pe[i]] = L->seg[pv[i]] = 0;  // SLRU: prefetched experts are probationary
    if (int rc = issue_refills(L, n, pe.data(), ps.data(), pv.data(), st)) return rc;
    if (n_refills_out) *n_refills_out = n;
    return MOE_OK;
}

int moe_destroy(moe_layer *L) {
    g_err.clear();
    release(L);
    return MOE_OK;
}

int moe_layer_set_bias(moe_layer *L, const float *bias_dev, void *stream) {
    g_err.clear();
    if (!L) return fail(MOE_EINVAL, "layer is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t n = (size_t)L->d.num_experts * sizeof(float);
    if (bias_dev)
        CUDA_TRY(cudaMemcpyAsync(L->bias, bias_dev, n, cudaMemcpyDeviceToDevice, st));
    else
        CUDA_TRY(cudaMemsetAsync(L->bias, 0, n, st));
    return MOE_OK;
}

int moe_layer_attach_staging(moe_layer *L, void *staging_dev, size_t bytes) {
    g_err.clear();
    if (!L) return fail(MOE_EINVAL, "layer is NULL");
    if (staging_dev && L->d.weight_format != MOE_FMT_MXFP4) return fail(MOE_EINVAL, "prefill is MXFP4 only");
    if (staging_dev && bytes < (size_t)L->d.num_experts * L->geo.expert_bytes)
        return fail(MOE_EINVAL, "staging buffer needs %zu bytes, got %zu",
                    (size_t)L->d.num_experts * L->geo.expert_bytes, bytes);
    L->staging = static_cast<uint8_t *>(staging_dev);
    L->staging_bytes = staging_dev ? bytes : 0;
    L->staged = false;
    return prefill_setup(L, L->staging);
}

int moe_layer_stage_all(moe_layer *L, void *stream) {
    g_err.clear();
    if (!L) return fail(MOE_EINVAL, "layer is NULL");
    if (!L->staging) return fail(MOE_ESTATE, "no staging buffer attached");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUDA_TRY(cudaMemcpyAsync(L->staging, L->host_bank, (size_t)L->d.num_experts * L->geo.expert_bytes,
                             cudaMemcpyHostToDevice, st));
    if (L->pf) {  // block scales of every staged expert, as the prefill kernels read them
        moe::launch_build_weight_atoms_bank(L->staging, L->d.num_experts, L->geo, L->stage_atoms, st);
        CUDA_TRY(cudaGetLastError());
    }
    L->staged = true;
    return MOE_OK;
}

int moe_debug_get_map(const moe_layer *L, int32_t *out) {
    if (!L || !out) return fail(MOE_EINVAL, "layer and out are required");
    if (L->dev_cache) {  // the device owns the map: read it after everything enqueued
        CUDA_TRY(cudaDeviceSynchronize());
        CUDA_TRY(cudaMemcpy(out, L->e2s_dev, (size_t)L->d.num_experts * sizeof(int32_t), cudaMemcpyDeviceToHost));
        return MOE_OK;
    }
    memcpy(out, L->e2s_visible.data(), L->e2s_visible.size() * sizeof(int32_t));
    return MOE_OK;
}

int moe_debug_device_cache(const moe_layer *L, int64_t out[4]) {
    if (!L || !out) return fail(MOE_EINVAL, "layer and out are required");
    for (int i = 0; i < 4; ++i) out[i] = 0;
    if (!L->lru_block) return MOE_OK;
    unsigned long long v[4];
    CUDA_TRY(cudaDeviceSynchronize());
    CUDA_TRY(cudaMemcpy(v, L->lru.stats, sizeof(v), cudaMemcpyDeviceToHost));
    for (int i = 0; i < 4; ++i) out[i] = (int64_t)v[i];
    return MOE_OK;
}

int moe_debug_slot_ptr(const moe_layer *L, int32_t slot, const void **ptr) {
    if (!L || !ptr || slot < 0 || slot >= L->d.num_slots) return fail(MOE_EINVAL, "bad slot");
    *ptr = L->slots + (size_t)slot * L->geo.expert_bytes;
    return MOE_OK;
}

int moe_debug_inject_fault(moe_layer *L, int32_t fault) {
    if (!L || (fault != MOE_FAULT_NONE && fault != MOE_FAULT_COPY)) return fail(MOE_EINVAL, "bad fault");
    L->fault = fault;
    return MOE_OK;
}

int moe_debug_stats(const moe_layer *L, int64_t stats[4]) {
    if (!L || !stats) return fail(MOE_EINVAL, "layer and stats are required");
    for (int i = 0; i < 4; ++i) stats[i] = L->stats[i];
    return MOE_OK;
}

int moe_debug_check_error(moe_layer *L, int32_t *code) {
    if (!L) return fail(MOE_EINVAL, "layer is NULL");
    int32_t v = 0;
    if (L->err) {
        CUDA_TRY(cudaDeviceSynchronize());
        CUDA_TRY(cudaMemcpy(&v, L->err, sizeof(int32_t), cudaMemcpyDeviceToHost));
        CUDA_TRY(cudaMemset(L->err, 0, sizeof(int32_t)));
    }
    if (code) *code = v;
    return v ? fail(MOE_ETIMEOUT, "a tensor-core kernel gave up a bounded wait (code %d)", v) : MOE_OK;
}

int moe_debug_decode_fusion(moe_layer *L, int32_t enable) {
    if (!L) return fail(MOE_EINVAL, "layer is NULL");
    L->ffn1 = enable != 0;
    return MOE_OK;
}

int moe_debug_profile(moe_layer *L, int32_t enable) {
    if (!L) return fail(MOE_EINVAL, "layer is NULL");
    CUDA_TRY(cudaDeviceSynchronize());
    L->prof = enable != 0;
    for (auto &n : L->prof_n) n = 0;
    return MOE_OK;
}

int moe_debug_profile_read(moe_layer *L, double out[4]) {
    if (!L || !out) return fail(MOE_EINVAL, "layer and out are required");
    for (int i = 0; i < 4; ++i) out[i] = 0.0;
    for (int w = 0; w < 3; ++w) {
        for (size_t i = 0; i + 1 < L->prof_n[w]; i += 2) {
            CUDA_TRY(cudaEventSynchronize(L->prof_ev[w][i + 1]));
            float ms = 0.f;
            CUDA_TRY(cudaEventElapsedTime(&ms, L->prof_ev[w][i], L->prof_ev[w][i + 1]));
            out[w] += ms;
        }
    }
    out[3] = (double)(L->prof_n[1] / 2);
    return MOE_OK;
}

}  // extern "C"
