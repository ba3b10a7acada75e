// Internal declarations shared by the layer's host code and its kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 512;
constexpr int kMaxTokens = 4096;
constexpr int kDecodeMaxTokens = 8;            // M <= 8 takes the decode kernels
constexpr int kRouteChunk = 256;               // router columns per warp task
constexpr int kPfRouteTok = 8;                 // prefill routing: tokens per thread block
constexpr int kDecodeSmemLimit = 200 * 1024;   // decode activations staged in shared memory

// Device scratch written by the route kernel.
struct RouteBuffers {
    float *logit_part;    // [nchunk][max_tokens][E]
    int32_t *topk_ids;    // [max_tokens][k]
    float *topk_w;        // [max_tokens][k]
    int32_t *hot_expert;  // [max_tokens * k]
    int32_t *hot_token;
    float *hot_w;
    int32_t *act_expert;  // [max_tokens * k]
    int32_t *act_slot;
    int32_t *act_off;
    int32_t *act_cnt;
    int32_t *cold_token;  // [max_tokens * k]
    int32_t *cold_expert;
    float *cold_w;
    int32_t *hist;        // [E]
    int32_t *counts;      // [4] n_hot, n_cold, n_active, M
    unsigned *arrive;     // [1] grid arrival counter (reset by the last block)
    int32_t *blk_cnt;     // prefill: [ceil(max_tokens / kPfRouteTok)][E] routes per (token tile, expert)
    int32_t *route_rank;  // prefill: [max_tokens * k] rank of a route among its tile's routes to its expert,
                          // then (after the launch) the route's position in the hot list
};

// Device-resident slot table (demand-filled LRU), written only by the route kernel's last block.
struct LruTable {
    int32_t *e2s;          // [E] expert -> slot, the same array as RouteParams::e2s
    int32_t *s2e;          // [S] slot -> expert, -1 empty
    int32_t *stamp;        // [S] last step the slot was used, -1 never
    int32_t *clock;        // [1] step counter
    int32_t *fill_expert;  // [<= kMaxFill] this step's fills, in fill order
    int32_t *fill_slot;
    int32_t *n_fill;       // [1]
    unsigned long long *stats;  // [4] steps, fills, hit experts, misses left cold
    int S;                 // 0: no table
};
constexpr int kMaxFill = kDecodeMaxTokens * kMaxTopK;  // distinct experts of a decode step

struct RouteParams {
    const uint16_t *x;   // bf16 bits [M, H]
    const float *Wr;     // [E, H]
    const float *WrT;    // prefill: [H, E32] (E rounded up to 32, zero rows), or nullptr
    int E32;
    const float *bias;   // [E] or nullptr
    const int32_t *e2s;  // [E]; ignored when all_hot
    int M, H, E, k, nchunk;
    int act_pad;         // decode: act_slot[n_active .. act_pad) are set to -1 (the expert kernels read one word)
    int all_hot;         // prefill: every expert is hot, slot = expert id
    int rowtask;         // set by launch_route: one warp per whole router row (decode, E > 32), logits final
    RouteBuffers b;
    uint16_t *xmir;      // decode: x copied here by the x-term tasks (the host mirror's source), or nullptr
    uint8_t *xq;         // tensor-core decode: x terms [16][Hpad] and their atoms, or nullptr
    uint8_t *xat;
    int Hpad;
    // NVFP4 one-token decode on the tensor cores: x as kNvTerms E2M1 terms instead (xq [kNvTerms][Hpad4 / 2]
    // packed, xat [nks4][4][512] UE4M3 scale atoms), the power-of-two factor of each term in xg [kNvTerms]
    int xnv;
    float *xg;
    int Hpad4;
    // prefill tile plan (or nullptr): each active expert's routes padded to whole 128-row tiles
    int32_t *pf_poff, *pf_e2a, *pf_tile_aidx, *pf_tile_nrows, *pf_ntiles;  // [E], [E], [cap], [cap], [1]
    int pf_tiles_cap;
    LruTable lru;        // decode with the device slot table (lru.S > 0): slots assigned before compaction
};

struct ExpertGeometry {
    int H, I;
    int sblk;  // columns per scale byte: 32 (MXFP4, E8M0 scales) or 16 (NVFP4, E4M3 scales)
    size_t expert_bytes;
    size_t off_wg_codes, off_wg_scales, off_wu_codes, off_wu_scales, off_wd_codes, off_wd_scales;
};

inline ExpertGeometry make_geometry(int H, int I, int sblk = 32) {
    ExpertGeometry g;
    g.H = H;
    g.I = I;
    g.sblk = sblk;
    size_t c = (size_t)I * H / 2, s = (size_t)I * H / sblk;
    g.off_wg_codes = 0;
    g.off_wg_scales = c;
    g.off_wu_codes = c + s;
    g.off_wu_scales = 2 * c + s;
    g.off_wd_codes = 2 * c + 2 * s;
    g.off_wd_scales = 3 * c + 2 * s;
    g.expert_bytes = 3 * c + 3 * s;
    return g;
}

struct DecodeParams {
    const uint8_t *bank;    // slot bank (decode) or staging bank (prefill)
    ExpertGeometry geo;
    const uint16_t *x;      // bf16 [M, H]
    const int32_t *counts;  // device counts from the route kernel
    const int32_t *act_slot, *act_off, *act_cnt;
    const int32_t *hot_token;
    const float *hot_w;
    float *h;               // [max_hot, I] fp32 scratch
    void *out;              // [M, H]
    int out_f32;
};

// Tensor-core decode path (moe_decode_tc.cu).
constexpr int kTcAtomBytes = 512;   // block scales of a 128-row tile x 128-column k-step
constexpr int kTcXRows = 16;        // rows of the x-term operand: 2 terms x 8 tokens
constexpr int kTcHRows = 64;        // rows of the w*h-term operand: 8 terms x 8 tokens

// NVFP4 decode on the tensor cores (moe_decode_nv.cu): packed E2M1 x packed E2M1 with UE4M3 scales per 16
// elements; activations and h enter as kNvTerms E2M1 terms, one B column each, term j scaled by its own
// power of two (applied when the accumulator column is read).
constexpr int kNvTerms = 16;

struct NvAtomLayout {       // UE4M3 scale atoms of one slot (512 bytes: one MMA of 64 K elements, 128 rows)
    int ntI, ntH, nks4;     // 128-row tiles of I and H; 256-element k-steps of H
    size_t off_g, off_u, off_d, slot_bytes;  // gate/up [ntI][nks4][4], down [ntH][ntI][2]
};
NvAtomLayout nv_atom_layout(int H, int I);

struct NvLaunch {
    const uint8_t *bank, *atoms;
    ExpertGeometry geo;
    int n_act_max, ks;
    const int32_t *counts, *act_slot, *act_off, *act_cnt, *hot_token;
    const float *hot_w;
    const uint8_t *xat;
    const float *xg;
    float *part;
    int *err;
    const CUtensorMap *mapG, *mapU, *mapX, *mapD;
};
void launch_build_weight_atoms_nv(const uint8_t *expert, const ExpertGeometry &g, uint8_t *atoms, cudaStream_t s);
cudaError_t launch_ffn_nv(const NvLaunch &L, cudaStream_t s);
int nv_ffn_smem();

// Weight scale atoms of one slot: gate [ntI][nks], up [ntI][nks], down [ntH][nksI], 512 bytes each.
struct TcAtomLayout {
    int ntI, ntH, nks, nksI;
    size_t off_g, off_u, off_d, slot_bytes;
};
TcAtomLayout tc_atom_layout(int H, int I);

struct TcLaunch {
    const uint8_t *bank, *atoms;  // slot (or staging) bank and its weight atoms
    ExpertGeometry geo;
    int M, n_act_max, ks_gateup, ks_down;
    const int32_t *counts, *act_slot, *act_off, *act_cnt, *hot_token;
    const float *hot_w;
    const uint8_t *xat;           // x-term atoms [nks][512]
    uint8_t *hq, *hat;            // w*h terms [n_act_cap][64][Ipad], atoms [n_act_cap][nksI][512]
    int Ipad;
    int *err;
    void *out;
    int out_f32;
    const CUtensorMap *mapG, *mapU, *mapX, *mapD, *mapH;
    float *part;                  // one-launch FFN: down partials [ntH][n_act_max * ntI][128]
};

int tc_max_splits();  // K splits of a tile run as one thread-block cluster: at most this many
void launch_build_weight_atoms(const uint8_t *expert, const ExpertGeometry &g, uint8_t *atoms, cudaStream_t s);
// Both launched with programmatic serialization after the previous grid in the stream.
cudaError_t launch_gateup_tc(const TcLaunch &L, cudaStream_t s);
cudaError_t launch_down_tc(const TcLaunch &L, cudaStream_t s);
// M = 1: gate/up, SiLU and down in one launch (launch_ffn_tc), then the fixed-order combine of its partials
// (launch_ffn_combine), both with programmatic serialization after the previous grid.
cudaError_t launch_ffn_tc(const TcLaunch &L, cudaStream_t s);
cudaError_t launch_ffn_combine(const TcLaunch &L, cudaStream_t s);

// Prefill (M > 8) on the tensor cores over the staged bank (moe_prefill_tc.cu).
struct PrefillLaunch {
    const uint8_t *bank, *atoms;  // staged experts (slot = expert id) and their weight atoms
    ExpertGeometry geo;
    int E, k, M, max_routes, tiles_cap, Hpad, Ipad, num_sms;
    const uint16_t *x;
    const int32_t *counts, *act_expert, *act_off, *act_cnt, *hot_expert, *hot_token, *topk_ids;
    const int32_t *route_pos;  // [M * k] hot-list position of each (token, j) route
    const float *hot_w;
    const int32_t *poff, *e2a, *tile_aidx, *tile_nrows, *ntiles;  // tile plan from the route launch
    uint8_t *XP, *XA, *HP, *HA;  // MXFP8 x / h in route order (rows_cap x Hpad / Ipad) and their atoms
    float *YP;                   // weighted expert outputs in route order [rows_cap][H]
    int *err;
    void *out;
    int out_f32;
    const CUtensorMap *mapXP, *mapHP, *mapG, *mapU, *mapD;
    cudaEvent_t ev[4];  // optional (nullptr = none): recorded before/after the gate/up and the down GEMM
};
int prefill_tiles_cap(int max_routes, int E);  // 128-row route tiles the buffers must hold
cudaError_t launch_prefill(const PrefillLaunch &P, cudaStream_t s);
void launch_build_weight_atoms_bank(const uint8_t *bank, int E, const ExpertGeometry &g, uint8_t *atoms,
                                    cudaStream_t s);

// Miss-copy kernel of the device slot table (moe_fill.cu): copies this step's fills from the host bank's
// device address into their slots and builds their scale atoms.
struct FillLaunch {
    const uint8_t *bank;  // device address of the page-locked bank, 16-byte aligned
    uint8_t *slots;
    uint8_t *atoms;       // weight atoms of every slot, or nullptr
    ExpertGeometry geo;
    const int32_t *fill_expert, *fill_slot, *n_fill;
    int grid;
};
size_t slot_fill_smem(int H, int I);
cudaError_t launch_slot_fill(const FillLaunch &F, cudaStream_t s);

cudaError_t launch_route(const RouteParams &p, cudaStream_t s, int num_sms);
cudaError_t launch_router_transpose(const float *Wr, float *WrT, int E, int H, int E32, cudaStream_t s);
void launch_gateup(const DecodeParams &p, int M, cudaStream_t s, int num_sms);
void launch_down(const DecodeParams &p, int M, cudaStream_t s, int num_sms);
void launch_map_update(int32_t *e2s, int n, const int32_t *experts, const int32_t *slots, cudaStream_t s);

// Sets the thread-local message returned by moe_last_error().
void set_last_error(const char *msg);

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the current device.  Function
// attributes belong to a device's context, so the limit is tracked per (device, kernel); thread-safe.
cudaError_t ensure_dyn_smem(const void *func, size_t bytes);

}  // namespace moe
