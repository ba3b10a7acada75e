// Host-side compute of the layer (plain C++, no CUDA): the expert FFN on MXFP4 records for cold routes,
// run on a pool of worker threads (onnxruntime PR #33976 and NInfer-Offload v0.4.0: routes to experts that
// are not on the GPU are computed by CPU workers while the GPU computes the resident ones).
#pragma once

#include <cstddef>
#include <cstdint>

namespace moe {
namespace host {

// Byte offsets of the six sections of one expert record: [Wg codes I x H/2][Wg scales I x H/32]
// [Wu codes][Wu scales][Wd codes H x I/2][Wd scales H x I/32], codes row-major, column 2c in the low nibble
// of byte c, one E8M0 scale per 32 columns.
struct RecordLayout {
    int H, I;
    size_t wg_codes, wg_scales, wu_codes, wu_scales, wd_codes, wd_scales, bytes;
};
RecordLayout record_layout(int H, int I);

// y = Wd (SiLU(Wg x) * (Wu x)) for one expert record: x bf16 bits [H], y fp32 [H]; h scratch fp32 [I].
// fp32 throughout, h not rounded.  One thread.
void expert_ffn(const RecordLayout &L, const uint8_t *rec, const uint16_t *x, float *h, float *y);

// The cold routes of one layer step: route r = (token[r], expert[r], w[r]), ordered by (token, expert).
// y [M][H] receives, for every token with cold routes, the sum over them in list order of w * FFN(x_t);
// other tokens' rows are set to zero.
struct ColdJob {
    RecordLayout L;
    const uint8_t *bank;  // [E][L.bytes], expert e at bank + e * L.bytes
    const uint16_t *x;    // bf16 bits [M][H]
    int M, n;
    const int32_t *token, *expert;
    const float *w;
    float *y;  // [M][H]
};

// Runs the job on `nthreads` workers of the process-wide pool (0: one per hardware thread).  Blocks until
// done.  Deterministic: every sum has a fixed order whatever the thread count.
void run_cold(const ColdJob &job, int nthreads);

}  // namespace host
}  // namespace moe
