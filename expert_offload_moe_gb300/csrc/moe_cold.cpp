// Cold routes on host threads: the MXFP4 expert FFN of every route whose expert has no GPU slot, computed
// from the page-locked host bank by a pool of workers while the GPU computes the hot routes (onnxruntime
// PR #33976 "Key Changes": routes to experts not on the GPU go to CPU workers; NInfer-Offload v0.4.0:
// CPU workers take the experts that are not cached on the GPU).
//
// Arithmetic (the same reading as the GPU path): E2M1 codes through the OCP MX v1.0 table times
// 2^(scale - 127) per 32 columns, products with the bf16 activations summed in fp32, h = SiLU(g) * u kept
// in fp32.  Sums run per 32-column block in eight interleaved partial sums (so the compiler can vectorise
// them) added in a fixed order, then block by block: results do not depend on the thread count.
#include "moe_host.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <condition_variable>
#include <cstring>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

namespace moe {
namespace host {

RecordLayout record_layout(int H, int I) {
    RecordLayout L{};
    L.H = H;
    L.I = I;
    const size_t c = (size_t)I * H / 2, s = (size_t)I * H / 32;
    L.wg_codes = 0;
    L.wg_scales = c;
    L.wu_codes = c + s;
    L.wu_scales = 2 * c + s;
    L.wd_codes = 2 * c + 2 * s;
    L.wd_scales = 3 * c + 2 * s;
    L.bytes = 3 * c + 3 * s;
    return L;
}

namespace {

// OCP MX v1.0 E2M1: codes 0..7 = 0, 0.5, 1, 1.5, 2, 3, 4, 6; codes 8..15 their negatives.
constexpr float kE2M1[16] = {0.f,  0.5f,  1.f,  1.5f,  2.f,  3.f,  4.f,  6.f,
                             -0.f, -0.5f, -1.f, -1.5f, -2.f, -3.f, -4.f, -6.f};

// Decode tables built once: both elements of a code byte (low nibble first), and 2^(s - 127) for every
// E8M0 byte (the same values as ldexp: s = 0 is the subnormal 2^-127, s = 255 overflows to infinity).
struct Tables {
    float pair[256][2];
    float scale[256];
    Tables() {
        for (int b = 0; b < 256; ++b) {
            pair[b][0] = kE2M1[b & 15];
            pair[b][1] = kE2M1[b >> 4];
            scale[b] = std::ldexp(1.0f, b - 127);
        }
    }
};
const Tables kTables;

inline float e8m0(uint8_t s) { return kTables.scale[s]; }

inline float bf16_to_f32(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

// Row r of an MXFP4 matrix with C columns dotted with v[C].
inline float mxfp4_row_dot(const uint8_t *codes, const uint8_t *scales, int C, const float *v) {
    float acc = 0.f;
    for (int b = 0; b < C / 32; ++b) {
        float e[32];
        const uint8_t *cb = codes + b * 16;
        for (int j = 0; j < 16; ++j) {
            e[2 * j] = kTables.pair[cb[j]][0];
            e[2 * j + 1] = kTables.pair[cb[j]][1];
        }
        const float *vb = v + b * 32;
        float p[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int i = 0; i < 32; i += 8)
            for (int l = 0; l < 8; ++l) p[l] += e[i + l] * vb[i + l];
        const float blk = ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
        acc += blk * e8m0(scales[b]);
    }
    return acc;
}

inline float silu(float g) { return g / (1.f + std::exp(-g)); }

void gate_up_rows(const RecordLayout &L, const uint8_t *rec, const float *x, int i0, int i1, float *h) {
    const size_t cb = (size_t)L.H / 2, sb = (size_t)L.H / 32;
    for (int i = i0; i < i1; ++i) {
        const float g = mxfp4_row_dot(rec + L.wg_codes + i * cb, rec + L.wg_scales + i * sb, L.H, x);
        const float u = mxfp4_row_dot(rec + L.wu_codes + i * cb, rec + L.wu_scales + i * sb, L.H, x);
        h[i] = silu(g) * u;
    }
}

void down_rows(const RecordLayout &L, const uint8_t *rec, const float *h, int r0, int r1, float *y) {
    const size_t cb = (size_t)L.I / 2, sb = (size_t)L.I / 32;
    for (int r = r0; r < r1; ++r) y[r] = mxfp4_row_dot(rec + L.wd_codes + r * cb, rec + L.wd_scales + r * sb, L.I, h);
}

// A process-wide pool of worker threads; the calling thread works too.  One parallel region at a time.
class Pool {
public:
    explicit Pool(int n) {
        for (int i = 0; i < n; ++i) workers_.emplace_back([this, i] { loop(i); });
    }
    ~Pool() {
        {
            std::lock_guard<std::mutex> lk(m_);
            stop_ = true;
        }
        cv_.notify_all();
        for (auto &t : workers_) t.join();
    }
    int size() const { return (int)workers_.size() + 1; }

    // f(0) .. f(n-1) on at most `threads` threads (the caller included); returns when all have run.
    void parallel_for(int n, int threads, const std::function<void(int)> &f) {
        std::lock_guard<std::mutex> one(region_);
        {
            std::lock_guard<std::mutex> lk(m_);
            fn_ = &f;
            ntask_ = n;
            next_.store(0);
            want_ = threads - 1;
            ++gen_;
        }
        cv_.notify_all();
        drain(&f, n);
        std::unique_lock<std::mutex> lk(m_);
        done_.wait(lk, [&] { return active_ == 0; });
        fn_ = nullptr;
    }

private:
    void drain(const std::function<void(int)> *f, int n) {
        for (int t = next_.fetch_add(1); t < n; t = next_.fetch_add(1)) (*f)(t);
    }
    void loop(int id) {
        uint64_t seen = 0;
        std::unique_lock<std::mutex> lk(m_);
        for (;;) {
            cv_.wait(lk, [&] { return stop_ || gen_ != seen; });
            if (stop_) return;
            seen = gen_;
            if (id >= want_ || !fn_) continue;
            const std::function<void(int)> *f = fn_;
            const int n = ntask_;
            ++active_;
            lk.unlock();
            drain(f, n);
            lk.lock();
            if (--active_ == 0) done_.notify_all();
        }
    }

    std::vector<std::thread> workers_;
    std::mutex m_, region_;
    std::condition_variable cv_, done_;
    const std::function<void(int)> *fn_ = nullptr;
    std::atomic<int> next_{0};
    int ntask_ = 0, want_ = 0, active_ = 0;
    uint64_t gen_ = 0;
    bool stop_ = false;
};

Pool &pool() {
    static Pool p(std::max(1u, std::thread::hardware_concurrency()) - 1);
    return p;
}

constexpr int kRowsPerTask = 64;

}  // namespace

void expert_ffn(const RecordLayout &L, const uint8_t *rec, const uint16_t *x, float *h, float *y) {
    std::vector<float> xf((size_t)L.H);
    for (int c = 0; c < L.H; ++c) xf[c] = bf16_to_f32(x[c]);
    gate_up_rows(L, rec, xf.data(), 0, L.I, h);
    down_rows(L, rec, h, 0, L.H, y);
}

void run_cold(const ColdJob &job, int nthreads) {
    const RecordLayout &L = job.L;
    const int H = L.H, I = L.I, n = job.n;
    std::fill(job.y, job.y + (size_t)job.M * H, 0.f);
    if (n <= 0) return;
    Pool &P = pool();
    const int threads = nthreads > 0 ? std::min(nthreads, P.size()) : P.size();
    std::vector<float> xf((size_t)job.M * H), hb((size_t)n * I), yb((size_t)n * H);
    for (size_t i = 0; i < xf.size(); ++i) xf[i] = bf16_to_f32(job.x[i]);
    auto rec = [&](int r) { return job.bank + (size_t)job.expert[r] * L.bytes; };

    // gate/up: (route, 64 rows of I) per task
    const int ci = (I + kRowsPerTask - 1) / kRowsPerTask;
    P.parallel_for(n * ci, threads, [&](int task) {
        const int r = task / ci, c = task - r * ci;
        const int i0 = c * kRowsPerTask, i1 = std::min(I, i0 + kRowsPerTask);
        gate_up_rows(L, rec(r), xf.data() + (size_t)job.token[r] * H, i0, i1, hb.data() + (size_t)r * I);
    });
    // down: (route, 64 rows of H) per task
    const int ch = (H + kRowsPerTask - 1) / kRowsPerTask;
    P.parallel_for(n * ch, threads, [&](int task) {
        const int r = task / ch, c = task - r * ch;
        const int r0 = c * kRowsPerTask, r1 = std::min(H, r0 + kRowsPerTask);
        down_rows(L, rec(r), hb.data() + (size_t)r * I, r0, r1, yb.data() + (size_t)r * H);
    });
    // combine: each token's routes in list order (ascending expert), 64 rows of H per task
    std::vector<int> first((size_t)job.M + 1, 0);
    for (int r = 0; r < n; ++r) first[job.token[r] + 1]++;
    for (int t = 0; t < job.M; ++t) first[t + 1] += first[t];
    P.parallel_for(job.M * ch, threads, [&](int task) {
        const int t = task / ch, c = task - t * ch;
        const int r0 = c * kRowsPerTask, r1 = std::min(H, r0 + kRowsPerTask);
        float *yt = job.y + (size_t)t * H;
        for (int r = first[t]; r < first[t + 1]; ++r) {
            const float w = job.w[r];
            const float *yr = yb.data() + (size_t)r * H;
            for (int q = r0; q < r1; ++q) yt[q] += w * yr[q];
        }
    });
}

}  // namespace host
}  // namespace moe
