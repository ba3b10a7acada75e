// Miss-copy kernel of the device-resident slot table (xinfer docs "How it works", Decode: a second kernel
// copies the missing experts straight from device-mapped page-locked host memory into their slots; both
// kernels have fixed launch shapes and read the miss count from device memory, so decode stays inside CUDA
// graphs without a host synchronisation).
//
// The route kernel's last block leaves this step's fills as an (expert, slot) list in device memory.  A
// fixed grid walks the work items of every fill:
//   - the three E2M1 code sections of the record, in 32 KB chunks: eight 16-byte loads in flight per
//     thread from the host bank's device address, then eight stores into the slot;
//   - the three E8M0 scale matrices, in 128-row bands: a band goes through shared memory on its way to the
//     slot, and the tensor-core scale atoms of that row tile (the layout build_weight_atoms_kernel writes)
//     are built from the shared copy, so the slot's atoms are ready with its bytes.
// The kernel is launched with programmatic serialization after the route kernel; the expert kernels that
// follow wait for its completion before they read a slot.
#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {
namespace {

constexpr int kFillThreads = 256;
constexpr int kFillVec = 8;                                 // 16-byte loads in flight per thread
constexpr int kFillChunk = kFillThreads * kFillVec * 16;    // bytes of one code work item
constexpr int kBandVec = 4;                                 // 16-byte loads in flight per thread in a band

struct FillArgs {
    const uint8_t *bank;  // device address of the page-locked host bank [E][eb]
    uint8_t *slots;       // [S][eb]
    uint8_t *atoms;       // [S][slot_bytes], or nullptr (no tensor-core path)
    size_t eb, atom_slot_bytes;
    size_t code_off[3], scale_off[3], code_bytes;
    size_t atom_off[3];
    int chunks_per_sec, n_code_items, n_items;  // per fill
    int ntI, ntH, nks, nksI, H, I;
    const int32_t *fill_expert, *fill_slot, *n_fill;
};

__global__ void __launch_bounds__(kFillThreads) slot_fill_kernel(FillArgs a) {
    extern __shared__ __align__(16) uint8_t band[];
    tc::pdl_trigger();
    tc::pdl_wait();
    const int n = *a.n_fill;
    const int tid = threadIdx.x;
    for (int q = blockIdx.x; q < n * a.n_items; q += gridDim.x) {
        const int i = q / a.n_items, r = q - i * a.n_items;
        const int e = a.fill_expert[i], s = a.fill_slot[i];
        const uint8_t *src = a.bank + (size_t)e * a.eb;
        uint8_t *dst = a.slots + (size_t)s * a.eb;
        if (r < a.n_code_items) {
            const int sec = r / a.chunks_per_sec, j = r - sec * a.chunks_per_sec;
            const size_t base = (size_t)j * kFillChunk;
            const size_t len = a.code_bytes - base < (size_t)kFillChunk ? a.code_bytes - base : (size_t)kFillChunk;
            const int nv = (int)(len / 16);
            const uint4 *sp = reinterpret_cast<const uint4 *>(src + a.code_off[sec] + base);
            uint4 *dp = reinterpret_cast<uint4 *>(dst + a.code_off[sec] + base);
            uint4 v[kFillVec];
#pragma unroll
            for (int u = 0; u < kFillVec; ++u) {
                const int idx = tid + u * kFillThreads;
                if (idx < nv) v[u] = __ldg(sp + idx);
            }
#pragma unroll
            for (int u = 0; u < kFillVec; ++u) {
                const int idx = tid + u * kFillThreads;
                if (idx < nv) dp[idx] = v[u];
            }
            continue;
        }
        // a 128-row band of one scale matrix: m = 0 gate, 1 up, 2 down
        const int b = r - a.n_code_items;
        const int m = b < a.ntI ? 0 : (b < 2 * a.ntI ? 1 : 2);
        const int tile = b - (m == 2 ? 2 * a.ntI : m * a.ntI);
        const int rows = m < 2 ? a.I : a.H, nkb = m < 2 ? a.H / 32 : a.I / 32, nsteps = m < 2 ? a.nks : a.nksI;
        const int nr = rows - tile * 128 < 128 ? rows - tile * 128 : 128;
        const size_t off = a.scale_off[m] + (size_t)tile * 128 * nkb;
        const int nv = nr * nkb / 16;  // rows and nkb keep every band a whole number of 16-byte vectors
        const uint4 *sp = reinterpret_cast<const uint4 *>(src + off);
        uint4 *dp = reinterpret_cast<uint4 *>(dst + off);
        uint4 *bp = reinterpret_cast<uint4 *>(band);
        for (int v0 = 0; v0 < nv; v0 += kBandVec * kFillThreads) {
            uint4 v[kBandVec];
#pragma unroll
            for (int u = 0; u < kBandVec; ++u) {
                const int idx = v0 + tid + u * kFillThreads;
                if (idx < nv) v[u] = __ldg(sp + idx);
            }
#pragma unroll
            for (int u = 0; u < kBandVec; ++u) {
                const int idx = v0 + tid + u * kFillThreads;
                if (idx < nv) {
                    dp[idx] = v[u];
                    bp[idx] = v[u];
                }
            }
        }
        __syncthreads();
        if (a.atoms) {
            // atom (tile, step): byte m0*16 + m1*4 + kb = scale of row 32 m1 + m0 of the tile and k-block
            // 4 step + kb; 127 (2^0) outside the matrix
            uint8_t *ap = a.atoms + (size_t)s * a.atom_slot_bytes + a.atom_off[m] + (size_t)tile * nsteps * 512;
            for (int idx = tid; idx < nsteps * 32; idx += kFillThreads) {
                const int step = idx >> 5, m0 = idx & 31;
                uint32_t w[4];
#pragma unroll
                for (int m1 = 0; m1 < 4; ++m1) {
                    const int row = 32 * m1 + m0;
                    uint32_t word = 0;
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb) {
                        const int c = step * 4 + kb;
                        const uint32_t sc = (row < nr && c < nkb) ? band[row * nkb + c] : 127u;
                        word |= sc << (8 * kb);
                    }
                    w[m1] = word;
                }
                *reinterpret_cast<uint4 *>(ap + (size_t)step * 512 + m0 * 16) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        __syncthreads();  // the band buffer is reused by this block's next item
    }
}

}  // namespace

size_t slot_fill_smem(int H, int I) { return (size_t)128 * ((H > I ? H : I) / 32); }

cudaError_t launch_slot_fill(const FillLaunch &F, cudaStream_t s) {
    const ExpertGeometry &g = F.geo;
    const TcAtomLayout l = tc_atom_layout(g.H, g.I);
    FillArgs a{};
    a.bank = F.bank;
    a.slots = F.slots;
    a.atoms = F.atoms;
    a.eb = g.expert_bytes;
    a.atom_slot_bytes = l.slot_bytes;
    a.code_off[0] = g.off_wg_codes;
    a.code_off[1] = g.off_wu_codes;
    a.code_off[2] = g.off_wd_codes;
    a.scale_off[0] = g.off_wg_scales;
    a.scale_off[1] = g.off_wu_scales;
    a.scale_off[2] = g.off_wd_scales;
    a.code_bytes = (size_t)g.I * g.H / 2;
    a.atom_off[0] = l.off_g;
    a.atom_off[1] = l.off_u;
    a.atom_off[2] = l.off_d;
    a.chunks_per_sec = (int)((a.code_bytes + kFillChunk - 1) / kFillChunk);
    a.n_code_items = 3 * a.chunks_per_sec;
    a.ntI = (g.I + 127) / 128;
    a.ntH = (g.H + 127) / 128;
    a.nks = l.nks;
    a.nksI = l.nksI;
    a.H = g.H;
    a.I = g.I;
    a.n_items = a.n_code_items + 2 * a.ntI + a.ntH;
    a.fill_expert = F.fill_expert;
    a.fill_slot = F.fill_slot;
    a.n_fill = F.n_fill;

    const size_t smem = slot_fill_smem(g.H, g.I);
    if (smem > 48 * 1024) {
        cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void *>(slot_fill_kernel), smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(F.grid);
    cfg.blockDim = dim3(kFillThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, slot_fill_kernel, a);
}

}  // namespace moe
