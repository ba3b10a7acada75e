/*
 * moe.h -- C ABI of the decode-time Mixture-of-Experts layer with GPU expert
 * slots, for one GB300 GPU (sm_103a).
 *
 * What the layer computes, per call, for M tokens x[M, H]:
 *   1. router: logits[t, e] = x[t, :] . Wr[e, :] + b[e]; the top_k largest
 *      logits of each token (ties go to the lower expert id); weights =
 *      softmax over the selected logits (onnxruntime PR #33976 "Key Changes":
 *      router, then hot experts on the GPU; NInfer-Offload v0.4.0: routing on
 *      the GPU across many thread blocks).
 *   2. expert_to_slot indirection: a route to expert e is hot when
 *      expert_to_slot[e] >= 0 (the slot holding e), cold otherwise
 *      (onnxruntime PR #33976 "Slot-Compacted GPU Hot Experts +
 *      expert_to_slot Indirection": slot < 0 is skipped on the GPU).
 *   3. hot routes run the expert FFN straight from the slot's MXFP4 bytes:
 *      y = Wd . (SiLU(Wg . x) * (Wu . x)) (tinyserve README "How it works" 2:
 *      fused dequantise-and-multiply, gate, up, down; xinfer docs
 *      "How it works": GEMMs over [num_slots, N, K] slot tensors).
 *   4. out[t, :] = sum of w * y over t's hot routes; cold routes are returned
 *      as (token, expert, weight) triples for the caller to handle.
 *   5. the slot cache refills slots from a page-locked host bank with async
 *      copies, at most max_refills_per_step experts per call, replacing the
 *      least used (NInfer-Offload v0.4.0 "expert cache"; tinyserve README
 *      "How it works" 3: frequency-recency eviction; xinfer docs "Supported":
 *      host RAM holds every expert, pinned).
 *
 * Formats (MXFP4 as defined by the OCP Microscaling Formats v1.0 spec; the
 * pages name MXFP4 but do not define it):
 *   x        bf16 [M, H], row-major, device memory, 16-byte aligned
 *   out      bf16 or fp32 [M, H] (moe_layer_desc.out_dtype), row-major, device
 *   Wr       fp32 [E, H], row-major;  b: fp32 [E] (may be NULL = zeros)
 *   expert record, expert_bytes = 3 * I * H * 17 / 32 bytes:
 *     [Wg codes I x H/2][Wg scales I x H/32][Wu codes I x H/2][Wu scales I x H/32]
 *     [Wd codes H x I/2][Wd scales H x I/32]
 *   codes: E2M1, row-major, byte c of a row holds column 2c in its low nibble
 *   and column 2c+1 in its high nibble; scales: E8M0 (2^(s-127)), byte b of a
 *   row covers columns [32b, 32b+32); 255 (NaN) is not allowed.
 *   The host bank is [E][expert_bytes], indexed by expert id; a slot holds a
 *   byte-identical copy of one record.
 *
 * Requirements: H and I multiples of 64; 1 <= top_k <= 16; top_k <= E <= 512;
 * top_k <= num_slots <= E; 1 <= max_tokens <= 4096.  Decode calls use
 * M <= 8 tokens; a call with M > 8 runs the prefill path (every expert of the
 * layer staged on the GPU, see moe_layer_attach_staging).
 *
 * Threading: a layer is not thread-safe; calls on one layer must be
 * serialised by the caller.  Every call returns a status code; on failure
 * moe_last_error() gives a message (thread-local, valid until the next call
 * on the same thread).  No call throws.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum moe_status {
    MOE_OK = 0,
    MOE_EINVAL = 1,   /* bad argument (sizes, NULL, non-pinned host bank, ...) */
    MOE_ENOMEM = 2,   /* device or pinned host allocation failed */
    MOE_ECUDA = 3,    /* a CUDA runtime call failed (message says which) */
    MOE_ETIMEOUT = 4, /* a bounded device wait gave up */
    MOE_ESTATE = 5    /* call order violated (e.g. forward without route) */
};

enum { MOE_OUT_BF16 = 0, MOE_OUT_F32 = 1 };

/* Slot-cache visibility of a refill:
 *  DETERMINISTIC: a refill chosen by moe_cache_update after step t is mapped
 *                 before any work enqueued after that call (step t+1 sees it);
 *                 the compute stream waits for the copy.
 *  POLLED:        the victim is unmapped at once, the copy runs on a side
 *                 stream, and the new expert is mapped by a later
 *                 moe_cache_update once its copy has landed; decode never
 *                 waits for a copy, so which routes are hot can depend on
 *                 timing (the NInfer-Offload v0.4.0 behaviour). */
enum { MOE_VIS_DETERMINISTIC = 0, MOE_VIS_POLLED = 1 };

/* Expert weight formats.  Both hold E2M1 codes [R, C/2] (column 2c in the
 * low nibble of byte c) per matrix, followed by its block scales:
 *  MOE_FMT_MXFP4: one E8M0 byte per 32 columns (OCP MX v1.0), record
 *                 3*I*H*17/32 bytes;
 *  MOE_FMT_NVFP4: one E4M3 byte per 16 columns (NVIDIA's NVFP4 block scale;
 *                 the pages name NVFP4 -- xinfer docs -- without defining it,
 *                 and no per-tensor scale is applied), record 3*I*H*9/16
 *                 bytes.
 * NVFP4 layers run decode (M <= 8) on CUDA-core kernels that decode the codes
 * and scales in registers; the tensor-core decode, prefill (staging), the
 * cold-route computations (moe_forward_cold, moe_forward_cold_gpu) and the
 * device slot table are MXFP4 only and return MOE_EINVAL for them.  Routing,
 * the miss list and the host slot policy are the same for both. */
enum { MOE_FMT_MXFP4 = 0, MOE_FMT_NVFP4 = 1 };

/* Slot policies (tinyserve README "How it works" 3 lists lfu, lru and fifo
 * among its eviction policies, with frequency-recency as its default):
 *  MOE_POLICY_FREQ  decayed route counts, score_decay = 1 LFU, < 1 LFRU (the
 *                   default; moe_policy_step)
 *  MOE_POLICY_LRU   evict the resident expert routed longest ago, never one
 *                   this step routed
 *  MOE_POLICY_FIFO  evict the resident expert that entered its slot first
 *  MOE_POLICY_SLRU  segmented LRU (tinyserve README "Configuration" lists
 *                   slru): a probationary and a protected segment of four
 *                   fifths of the slots; a hit is protected, new experts
 *                   are probationary and probationary ones are evicted first
 *                   (moe_policy_step_slru)
 * In every policy the candidates for a slot are non-resident experts,
 * at most max_refills_per_step per step. */
enum { MOE_POLICY_FREQ = 0, MOE_POLICY_LRU = 1, MOE_POLICY_FIFO = 2, MOE_POLICY_SLRU = 3 };

typedef struct moe_layer moe_layer;

typedef struct {
    int32_t hidden;               /* H */
    int32_t inter;                /* I, expert intermediate size */
    int32_t num_experts;          /* E */
    int32_t top_k;                /* k */
    int32_t num_slots;            /* S, GPU slots of this layer */
    int32_t max_tokens;           /* largest M of any call (sizes the scratch) */
    int32_t out_dtype;            /* MOE_OUT_BF16 or MOE_OUT_F32 */
    int32_t max_refills_per_step; /* R, refills per moe_cache_update (NInfer: 2) */
    float score_decay;            /* 1.0 = LFU; in (0,1) = decayed frequency (LFRU) */
    int32_t visibility;           /* MOE_VIS_DETERMINISTIC or MOE_VIS_POLLED */
    int32_t weight_format;        /* MOE_FMT_MXFP4 (0) or MOE_FMT_NVFP4 */
} moe_layer_desc;

/* Result of moe_route.  Device arrays are owned by the layer and stay valid
 * until the next moe_route on the same layer; host arrays are a page-locked
 * mirror, valid once `done` (a cudaEvent_t) has completed (eager calls), or
 * once the launch of a graph captured from the calls has completed. */
typedef struct {
    int32_t M;
    /* device */
    const int32_t *topk_ids;   /* [M, k] experts of each token, largest logit first */
    const float *topk_w;       /* [M, k] renormalised weights, same order */
    const int32_t *hot_expert; /* [<= M*k] hot routes ordered by (expert, token) */
    const int32_t *hot_token;
    const float *hot_w;
    const int32_t *act_expert; /* [<= min(S, M*k)] experts with hot routes, ascending */
    const int32_t *act_slot;   /* their slots; after a decode call (M <= 8) entries n_active..min(S, M*k)-1 are -1 */
    const int32_t *act_off;    /* first index of each in the hot arrays */
    const int32_t *act_cnt;    /* number of hot routes of each */
    const int32_t *cold_token; /* [<= M*k] cold routes ordered by (token, expert) */
    const int32_t *cold_expert;
    const float *cold_w;
    const int32_t *hist;       /* [E] routes (hot and cold) per expert */
    const int32_t *counts;     /* [4] n_hot, n_cold, n_active, M */
    /* page-locked host mirror of counts, cold triples and hist */
    const int32_t *h_counts;
    const int32_t *h_cold_token;
    const int32_t *h_cold_expert;
    const float *h_cold_w;
    const int32_t *h_hist;
    void *done; /* cudaEvent_t recorded after the mirror copy (eager calls) */
} moe_route_result;

/* Creates a layer on the current CUDA device.
 *  router_w_dev    fp32 [E, H] device, copied (the caller may free it after)
 *  router_bias_dev fp32 [E] device or NULL, copied
 *  host_bank       [E, expert_bytes] page-locked host memory (cudaHostAlloc or
 *                  cudaHostRegister), borrowed: it must outlive the layer.
 *                  Pageable memory is rejected with MOE_EINVAL.
 *  expert_to_slot_host int32 [E]: -1 = cold, else a slot in [0, S); no slot
 *                  twice.  The named experts are copied into their slots
 *                  before this call returns (on `stream`, then synchronised).
 *  stream          cudaStream_t for the initial copies (NULL = default)
 * Allocates the slot bank (S * expert_bytes), router copy, map and scratch.
 * Errors: MOE_EINVAL, MOE_ENOMEM, MOE_ECUDA; *out is NULL on failure. */
int moe_layer_create(const moe_layer_desc *desc, const float *router_w_dev, const float *router_bias_dev,
                     const uint8_t *host_bank, const int32_t *expert_to_slot_host, void *stream,
                     moe_layer **out);

/* Routes M tokens: router GEMV, top-k + softmax, slot lookup and compaction,
 * all on `stream` (asynchronous, no host synchronisation, fixed launch
 * shapes: capturable in a CUDA graph).  One copy moves the host mirror; later
 * work on `stream` does not wait for it.  Eager calls run it on an internal
 * stream forked from `stream` (`done` marks its end) and the layer's next
 * moe_route waits for it.  Under stream capture it becomes a leaf node of the
 * graph after the route launch, and the layer's next moe_route in the same
 * capture depends on it.
 *  x_dev  bf16 [M, H] device;  1 <= M <= max_tokens
 *  res    filled with the pointers above (may be NULL)
 * With M > 8 (prefill) every expert is treated as resident in the staging
 * bank, so every route is hot and the cold list is empty.
 * Errors: MOE_EINVAL, MOE_ECUDA. */
int moe_route(moe_layer *layer, const void *x_dev, int32_t M, void *stream, moe_route_result *res);

/* Runs the hot routes of the last moe_route and combines them:
 *   out[t, :] = sum over t's hot routes, in ascending expert order, of w * y
 * where y is the expert FFN read from the expert's slot (fp32 accumulation);
 * tokens without hot routes get zeros.  x_dev and M must be those of the last
 * moe_route (MOE_ESTATE otherwise).  M <= 8: decode kernels over the slot
 * bank.  M > 8: prefill on the staging bank (MOE_ESTATE if none is attached,
 * it was not staged with moe_layer_stage_all, or the last moe_route was made
 * before it was attached: that route launch also plans the prefill tiles).
 *  out_dev  [M, H] out_dtype, device, caller-owned, 16-byte aligned
 * Asynchronous, capturable.  Errors: MOE_EINVAL, MOE_ESTATE, MOE_ECUDA. */
int moe_forward_slots(moe_layer *layer, const void *x_dev, void *out_dev, int32_t M, void *stream);

/* Computes the cold routes of the last moe_route on host threads and adds them
 * to out_dev (onnxruntime PR #33976 "Key Changes" and NInfer-Offload v0.4.0:
 * routes to experts not on the GPU are computed by CPU workers while the GPU
 * computes the resident ones).  Call it after moe_forward_slots on the same
 * stream.
 *  x_dev, M   those of the last moe_route (MOE_ESTATE otherwise); M > 8 is
 *             prefill, where every route is hot: nothing to do
 *  out_dev    the output moe_forward_slots wrote, [M, H] out_dtype
 *  nthreads   host threads to use, the calling thread included; 0 = every
 *             hardware thread
 * The calling thread blocks: it waits for the route's page-locked mirror
 * (counts, cold triples and x, copied by moe_route), then computes
 *   y[t] = sum over t's cold routes, ascending expert, of w * FFN_e(x_t)
 * from the page-locked host bank, in fp32 with h not rounded, on the
 * library's worker pool.  Every sum has a fixed order, so y does not depend
 * on the thread count.  Meanwhile the GPU works on the hot routes.
 * Then, asynchronously on `stream`, y is copied to the device and added to
 * out_dev.  Tokens with no cold route are unchanged.  With bf16 outputs the
 * sum is rounded once more; the fp32 output mode keeps hot + cold exact in
 * fp32.
 * Errors: MOE_EINVAL, MOE_ESTATE, MOE_ECUDA. */
int moe_forward_cold(moe_layer *layer, const void *x_dev, void *out_dev, int32_t M, int32_t nthreads,
                     void *stream);

/* The cold routes of the last moe_route computed on the GPU, reading the
 * expert bytes in place from the page-locked host bank through its device
 * address (NVLink-C2C on a Grace host, PCIe elsewhere), added to out_dev.
 * xinfer docs "How it works" reads missed experts from device-mapped host
 * memory; here the CUDA-core FFN kernels stream them directly, one pass per
 * step, without refilling a slot.  Call it after moe_forward_slots on the
 * same stream.
 *  x_dev, M   those of the last moe_route (MOE_ESTATE otherwise); M > 8 is
 *             prefill, where every route is hot: nothing to do
 *  out_dev    the output moe_forward_slots wrote, [M, H] out_dtype
 * Fully asynchronous and capturable: the cold lists never leave the device.
 * The cold sum is formed in fp32 in ascending expert order per token and
 * added to out_dev (bf16 outputs are rounded once more, as in
 * moe_forward_cold).  MOE_ESTATE if the GPU cannot address the bank.
 * Errors: MOE_EINVAL, MOE_ESTATE, MOE_ECUDA. */
int moe_forward_cold_gpu(moe_layer *layer, const void *x_dev, void *out_dev, int32_t M, void *stream);

/* The expert FFN used by moe_forward_cold, on one expert record (layout as
 * in moe_layer_create's host bank), on the calling thread:
 *   y = Wd (SiLU(Wg x) * (Wu x)), fp32, h not rounded.
 *  record  host, expert_bytes(H, I) bytes
 *  x_host  bf16 [H] host;  y_host fp32 [H] host
 * No GPU is involved.  Errors: MOE_EINVAL. */
int moe_host_expert_ffn(const uint8_t *record, int32_t H, int32_t I, const uint16_t *x_host, float *y_host);

/* Host-side slot-cache step after a moe_route (waits for its `done` event).
 * Scores every expert (score = decay * score + routes this step), picks at
 * most R (candidate, victim) pairs, copies each candidate from the host bank
 * into the victim's slot with cudaMemcpyAsync on the layer's side stream
 * (after the work already on `stream`, so a slot is never overwritten while
 * read), and updates expert_to_slot on `stream` per the visibility mode.
 * Does nothing when every expert is resident (S == E).
 *  n_refills_out  copies issued by this call (may be NULL)
 * Not capturable (host decisions).  Errors: MOE_ESTATE, MOE_ECUDA. */
int moe_cache_update(moe_layer *layer, void *stream, int32_t *n_refills_out);

/* Waits for the layer's copies, frees everything the layer owns.  NULL is OK. */
int moe_destroy(moe_layer *layer);

/* Thread-local message of the last failed call on this thread ("" if none). */
const char *moe_last_error(void);

/* Replaces the router bias with bias_dev (fp32 [E], device; NULL = zeros),
 * copied on `stream` in stream order (capturable).  Used when the bias moves
 * between steps.  Errors: MOE_EINVAL, MOE_ECUDA. */
int moe_layer_set_bias(moe_layer *layer, const float *bias_dev, void *stream);

/* ------------------------------------------------ expert-parallel sharding */

/* Expert parallelism over `world` ranks, one GPU each (xinfer docs "Options":
 * each rank loads and offloads its own expert shard, and NCCL combines the
 * rank-local MoE results).  The router is replicated on every rank; the E
 * experts are split into `world` contiguous ranges, the first E % world
 * ranks taking one more, and rank r owns [first, first + count).  Writes the
 * rank's expert_to_slot[E]: its own experts in slots 0..count-1 in ascending
 * id order, every other expert -1.  A layer created with this map (and
 * num_slots >= count) routes every token like the whole layer, computes the
 * routes to this rank's experts as its hot routes (moe_forward_slots) and
 * returns the routes to the other ranks' experts as its cold list; one sum
 * all-reduce of the ranks' fp32 outputs out[M, H] gives the whole layer (the
 * experts' contributions summed within each rank in ascending order, then
 * over the ranks in rank order).  first and count may be NULL.  Host only.
 * Errors: MOE_EINVAL (E < 1, world < 1 or > E, rank outside [0, world),
 * NULL map). */
int moe_ep_local_map(int32_t E, int32_t world, int32_t rank, int32_t *expert_to_slot, int32_t *first,
                     int32_t *count);

/* ------------------------------------------------ routing without allocation */

/* Caller-owned device buffers that receive a routing result; sizes as in
 * moe_route_result: [M*k] for the route lists, [E] for hist, [4] for counts. */
typedef struct {
    int32_t *topk_ids;
    float *topk_w;
    int32_t *hot_expert;
    int32_t *hot_token;
    float *hot_w;
    int32_t *act_expert;
    int32_t *act_slot;
    int32_t *act_off;
    int32_t *act_cnt;
    int32_t *cold_token;
    int32_t *cold_expert;
    float *cold_w;
    int32_t *hist;
    int32_t *counts;
} moe_route_buffers;

/* The pages have no counterpart to this call.  It routes M tokens exactly as
 * moe_route does (router GEMV, top-k + softmax, split and compaction by
 * expert_to_slot), but it never allocates: no cudaMalloc, no cudaFree, no
 * host allocation, no layer object.  It is meant for callers that cannot
 * allocate device memory where they route -- e.g. a serving process whose
 * device memory is all reserved up front by its own pool allocator, or a
 * latency-critical loop that must not take the implicit synchronisation of
 * cudaMalloc/cudaFree.
 *  x_dev, M, H          bf16 [M, H] device, 16-byte aligned; H % 64 == 0
 *  router_w_dev         fp32 [E, H] device, 16-byte aligned (read in place)
 *  router_bias_dev      fp32 [E] device, or NULL (zeros)
 *  E, top_k             1 <= top_k <= 16, top_k <= E <= 512
 *  expert_to_slot_dev   int32 [E] device; < 0 = cold (no prefill mode here)
 *  out                  caller-owned device buffers (all required)
 * Scratch: a built-in device array of 1 MiB (held by every GPU that loads the
 * library until exit) holds the partial logits, so ceil(H/256) * M * E * 4
 * must not exceed 1 MiB - 256 bytes; larger sizes return MOE_EINVAL with a
 * message saying so.  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress); make that first call before any
 * stream capture.  All calls share the array: calls that overlap on the GPU
 * (unordered streams) race and give wrong results; calls ordered on one
 * stream are fine (each clears the arrival counter it needs).
 * Errors: MOE_EINVAL, MOE_ECUDA (message in moe_last_error()). */
int moe_route_noalloc(const void *x_dev, int32_t M, int32_t H, const float *router_w_dev,
                      const float *router_bias_dev, int32_t E, int32_t top_k, const int32_t *expert_to_slot_dev,
                      const moe_route_buffers *out, void *stream);

/* ------------------------------------------------------------ prefill */

/* Attaches a caller-owned device buffer of at least E * expert_bytes bytes
 * used to stage all experts of the layer for prefill (xinfer docs "How it
 * works", Prefill: the whole expert layer is copied to a staging buffer and
 * the unmodified GEMM runs on it).  Several layers may share one buffer if
 * their calls are serialised on one stream.  NULL detaches.
 * Errors: MOE_EINVAL. */
int moe_layer_attach_staging(moe_layer *layer, void *staging_dev, size_t bytes);

/* Copies all E experts of the layer from the host bank into the attached
 * staging buffer on `stream` (asynchronous).  Errors: MOE_ESTATE, MOE_ECUDA. */
int moe_layer_stage_all(moe_layer *layer, void *stream);

/* ------------------------------------------------------- introspection */

/* expert_to_slot as last enqueued to the device (what the next moe_route on
 * the same stream sees): int32 [E]. */
int moe_debug_get_map(const moe_layer *layer, int32_t *expert_to_slot_host);

/* Device address of slot s (expert_bytes bytes), for byte comparisons. */
int moe_debug_slot_ptr(const moe_layer *layer, int32_t slot, const void **ptr);

/* Fault injection on the host: MOE_FAULT_COPY makes the next refill fail
 * before any copy is issued (the call returns MOE_ECUDA and leaves the map
 * unchanged); MOE_FAULT_NONE clears it. */
enum { MOE_FAULT_NONE = 0, MOE_FAULT_COPY = 1 };
int moe_debug_inject_fault(moe_layer *layer, int32_t fault);

/* Cumulative counters of the layer: [0] refills issued, [1] refill bytes,
 * [2] routes seen, [3] hot routes seen (updated by moe_cache_update). */
int moe_debug_stats(const moe_layer *layer, int64_t stats[4]);

/* Reads and clears the layer's device error word (synchronises the device):
 * 0 = no error; otherwise a tensor-core kernel gave up a bounded wait
 * (1: operand copy, 2: stage release, 3: accumulator; in the one-launch
 * M = 1 FFN also 4: h operand, 5: down accumulator full, 6: down accumulator
 * drained) and its output is not valid.  Returns MOE_ETIMEOUT when the word was set, MOE_OK otherwise. */
int moe_debug_check_error(moe_layer *layer, int32_t *code);

/* Kernel timing for benchmarks: with enable != 0, later route and forward
 * calls record timing events around the router, gate/up and down kernels on
 * the caller's stream (synchronises the device; resets the sums). */
int moe_debug_profile(moe_layer *layer, int32_t enable);

/* One-token decode (M = 1) on the tensor-core path runs gate/up, SiLU·up
 * and down of every active expert (tinyserve README "How it works" 2: fused
 * dequantise-and-multiply, gate / up / down) as ONE kernel launch, followed
 * by a small launch that adds the weighted per-expert results in a fixed
 * order (on by default); enable == 0 makes moe_forward_slots use the
 * separate gate/up and down launches instead (for comparison; with NVFP4
 * layers, the CUDA-core kernels).  Both give results within the same
 * tolerance of the oracle; they sum the experts' contributions in different
 * orders, so they are not bit-identical to each other.  Takes effect at the
 * next moe_forward_slots; no device work.  Errors: MOE_EINVAL (NULL layer). */
int moe_debug_decode_fusion(moe_layer *layer, int32_t enable);

/* Streaming-read probe for benchmarks (no counterpart on the pages; it does
 * none of the layer's arithmetic): one launch on `stream` that reads `bytes`
 * bytes of device memory at src_dev with 128-bit loads, the floor against
 * which a weight-streaming kernel of the same byte count is measured.
 * src_dev and bytes must be multiples of 16; sink_dev (4 bytes, device,
 * caller-owned) is written only in the unlikely case the xor of all words
 * read equals 0x9E3779B9.  nblocks = 0 picks four 512-thread blocks per SM.
 * Asynchronous; nothing is allocated.  Errors: MOE_EINVAL (NULL or unaligned
 * pointers, bytes not a multiple of 16, nblocks < 0), MOE_ECUDA. */
int moe_debug_stream_read(const void *src_dev, size_t bytes, void *sink_dev, int32_t nblocks, void *stream);

/* Block-scaled tensor-core probe for benchmarks (no counterpart on the
 * pages; none of the layer's data): one launch on `stream`, one CTA per SM
 * (nblocks = 0: the device's SM count), each issuing `iters` steps of four
 * tcgen05.mma kind::mxf8f6f4 block_scale MMAs of M = 128, N = 256, K = 32
 * (E4M3 A x E2M1 B, UE8M0 scales, fp32 accumulator in tensor memory) on
 * operand tiles held in shared memory, the shape the prefill GEMMs issue per
 * 128-column step.  The launch does nblocks * iters * 4 * 2 * 128 * 256 * 32
 * flops; its event-timed duration gives the ceiling of that MMA stream with
 * no operand traffic.  err_dev (4 bytes, device, caller-owned, set to 0 by
 * the caller) receives a nonzero code if the final completion wait ran out.
 * Asynchronous; nothing is allocated.  Errors: MOE_EINVAL (NULL or unaligned
 * err_dev, iters outside 1..65536, nblocks < 0), MOE_ECUDA. */
int moe_debug_mma_peak(int32_t iters, int32_t nblocks, void *err_dev, void *stream);

/* Sums of the timed kernels since moe_debug_profile: out[0] route ms,
 * out[1] gate/up ms (the one-launch FFN when M = 1 takes it), out[2] down
 * ms (its combine launch for one-launch calls), out[3] forward calls (waits
 * for the events). */
int moe_debug_profile_read(moe_layer *layer, double out[4]);

/* Next-layer prefetch (tinyserve README "How it works" 4, FATE: the
 * current layer's activations predict the next layer's experts, and the
 * copies overlap the current layer's work).  Call it on the NEXT layer with
 * the CURRENT layer's input x_dev [M, H] (1 <= M <= min(8, max_tokens)),
 * after the current layer's moe_forward_slots has been issued:
 *  1. the layer's own router, top-k and softmax run on x_dev (its routing of
 *     x_dev, i.e. the prediction) on an internal stream forked from `stream`,
 *     into scratch of their own (the last moe_route's results stay valid);
 *  2. the calling thread waits for the predicted per-expert route counts;
 *  3. moe_prefetch_step picks up to max_refills_per_step predicted,
 *     non-resident experts and the unpredicted resident experts they replace;
 *  4. their copies from the host bank are issued on the layer's copy stream
 *     and become visible as moe_cache_update's do (MOE_VIS_DETERMINISTIC:
 *     later work on `stream` waits for them; MOE_VIS_POLLED: they join the map
 *     once landed).
 * Scores and recency are not changed (the layer's own moe_cache_update counts
 * the routes when they happen).  Does nothing when every expert is resident.
 * *n_refills (may be NULL) receives the number of copies issued.  Not
 * capturable (the host waits for the prediction).  Errors: MOE_EINVAL,
 * MOE_ESTATE (device slot table on), MOE_ENOMEM, MOE_ECUDA. */
int moe_prefetch(moe_layer *layer, const void *x_dev, int32_t M, void *stream, int32_t *n_refills);

/* The prefetch decision on host arrays, as moe_prefetch runs it.
 *  pred[E]: predicted routes per expert.  Candidates: predicted experts
 *  neither resident nor in flight, most predicted routes first, then higher
 *  score[e], then lower id.  Victims: resident experts neither predicted nor
 *  in flight, lowest score first, then the oldest last[e], then lower slot.
 *  Candidate i takes victim i's slot; at most R pairs.  e2s[E] and s2e[S]
 *  are updated in place, score[] and last[] are only read.  Returns the
 *  number of pairs, or -1 on bad arguments. */
int moe_prefetch_step(const double *score, const int64_t *last, int32_t *e2s, int32_t *s2e, int32_t E, int32_t S,
                      const int32_t *pred, int32_t R, const uint8_t *in_flight, int32_t *pair_expert,
                      int32_t *pair_slot, int32_t *pair_victim);

/* The slot-cache decision on host arrays, as moe_cache_update runs it
 * (exported so that the policy can be checked without a GPU).
 *  score[E], last[E], e2s[E], s2e[S] are updated in place; in_flight[E]
 *  (may be NULL) marks experts whose copy has not landed; hist[E] are this
 *  step's routes per expert.  Writes up to R (expert, slot, victim) triples
 *  and returns their number, or -1 on bad arguments. */
int moe_policy_step(double *score, int64_t *last, int32_t *e2s, int32_t *s2e, int32_t E, int32_t S,
                    const int32_t *hist, int64_t step, double decay, int32_t R, const uint8_t *in_flight,
                    int32_t *pair_expert, int32_t *pair_slot, int32_t *pair_victim);

/* The same for MOE_POLICY_LRU and MOE_POLICY_FIFO.  Candidates: the
 * non-resident experts this step routed, most routes first (ties: lower id).
 * Victims: LRU the resident expert with the oldest last[e] (the last step
 * that routed it), taken only while it was not routed this step; FIFO the
 * one with the oldest loaded[e] (the step it entered a slot, -1 for experts
 * placed at creation), taken whatever its use; ties: lower slot.  Experts in
 * flight are neither.  last[] (and for FIFO loaded[], required) are updated
 * in place; score[] keeps the decayed frequency for reference.  Returns the
 * number of pairs, or -1 on bad arguments. */
int moe_policy_step_recency(int32_t policy, double *score, int64_t *last, int64_t *loaded, int32_t *e2s,
                            int32_t *s2e, int32_t E, int32_t S, const int32_t *hist, int64_t step, double decay,
                            int32_t R, const uint8_t *in_flight, int32_t *pair_expert, int32_t *pair_slot,
                            int32_t *pair_victim);

/* Segmented LRU (MOE_POLICY_SLRU; tinyserve README "Configuration" names slru
 * among its cache policies and gives no details, so the textbook two-segment
 * scheme is used).  seg[e] is 1 while resident expert e is in the protected
 * segment, 0 otherwise; at most pcap residents are protected (layers use
 * pcap = 4 S / 5, rounded down).  One step:
 *   1. last[e] = step for every expert this step routed (score[] keeps the
 *      decayed frequency for reference);
 *   2. every routed resident expert becomes protected;
 *   3. while more than pcap residents are protected, the protected one with
 *      the oldest last[e] (ties: lower slot) returns to probationary;
 *   4. candidates: non-resident experts this step routed, most routes first
 *      (ties: lower id); victims: probationary residents by oldest last[e],
 *      then protected ones by oldest last[e] (ties: lower slot); experts in
 *      flight are neither; candidate i replaces victim i while that victim
 *      was not routed this step, at most R pairs; new experts enter the
 *      probationary segment.
 * score[], last[], seg[], e2s[E] and s2e[S] are updated in place.  Returns
 * the number of (expert, slot, victim) pairs, or -1 on bad arguments
 * (NULL arrays, E, S or R out of range, pcap < 0 or > S). */
int moe_policy_step_slru(double *score, int64_t *last, uint8_t *seg, int32_t *e2s, int32_t *s2e, int32_t E, int32_t S,
                         const int32_t *hist, int64_t step, double decay, int32_t R, int32_t pcap,
                         const uint8_t *in_flight, int32_t *pair_expert, int32_t *pair_slot, int32_t *pair_victim);

/* Selects the slot policy of a layer (MOE_POLICY_*, default MOE_POLICY_FREQ)
 * for its later moe_cache_update calls.  Errors: MOE_EINVAL. */
int moe_layer_set_policy(moe_layer *layer, int32_t policy);

/* ------------------------------------------------ device-resident slot table */

/* Switches the layer's decode calls (M <= 8) to a slot table kept and run on
 * the GPU (xinfer docs "How it works", Decode: before the expert GEMMs a
 * kernel looks the routed experts up in a per-layer LRU table on the GPU,
 * gives least-recently-used slots to the misses and rewrites expert ids to
 * slot ids; a second kernel copies the missing experts from device-mapped
 * page-locked host memory into their slots; both have fixed launch shapes and
 * read the miss count from device memory, so decode stays inside CUDA graphs).
 *
 * With the table on, moe_route does both in stream order after top-k:
 *   - slots whose expert the step routed (hits) are stamped with the step;
 *   - each routed expert without a slot (a miss; most routes first, ties to
 *     the lower id) takes a slot the step did not route: empty slots first
 *     (ascending), then the oldest stamp (ties: lower slot); expert_to_slot
 *     and the route lists use the new map;
 *   - a fill kernel copies those experts from the host bank's device address
 *     into their slots (with their tensor-core scale atoms) before any later
 *     work on the stream.
 * Every route of the step is then hot, except for misses left without a slot
 * (only when a step routes more distinct experts than num_slots), which stay
 * cold for the step and are listed as usual.  There is no refill budget:
 * max_refills_per_step and the host policy do not apply, and
 * moe_cache_update returns MOE_ESTATE while the table is on.  Prefill calls
 * (M > 8) do not touch the table.  Routes to the same experts give the same
 * output whatever slots they sit in (expert-order accumulation).
 *
 * enable != 0: the table starts from the layer's current map (after every
 * copy the host policy issued has landed), every stamp -1.  enable == 0: the
 * host policy takes over the table's map.  Both synchronise the device; not
 * capturable.  The host bank must have a device address (page-locked memory
 * on a GPU that can map it: MOE_ESTATE otherwise) and be 16-byte aligned
 * (MOE_EINVAL).  While on, moe_debug_get_map reads the device's map
 * (synchronising).  In profiling mode (moe_debug_profile) the fill kernel is
 * timed with the route.  Errors: MOE_EINVAL, MOE_ESTATE, MOE_ECUDA. */
int moe_layer_set_device_cache(moe_layer *layer, int32_t enable);

/* Cumulative counters of the device slot table since it was last switched
 * on (synchronises the device): [0] decode steps, [1] experts filled,
 * [2] hits (routed experts already resident, counted once per step),
 * [3] misses left cold.  All zero if the table was never on. */
int moe_debug_device_cache(const moe_layer *layer, int64_t out[4]);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
