// C ABI of libcsa: argument validation, workspace layout and the launch
// sequence of every entry point declared in include/csa.h.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

using namespace csa;

static std::atomic<long long> g_launches{0};
void csa::count_launches(int n) { g_launches += n; }

namespace {

thread_local char g_err[512] = "";

csa_status fail(csa_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

}  // namespace

csa_status csa::report_error(csa_status s, const char *msg) { return fail(s, "%s", msg); }

namespace {

csa_status cuda_fail(cudaError_t e, const char *where) {
    return fail(CSA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

#define CSA_TRY_CUDA(call, where)                      \
    do {                                               \
        cudaError_t e_ = (call);                       \
        if (e_ != cudaSuccess) return cuda_fail(e_, where); \
    } while (0)

#define CSA_TRY(call)                       \
    do {                                    \
        csa_status s_ = (call);             \
        if (s_ != CSA_OK) return s_;        \
    } while (0)

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

csa_status need_ptr(const void *p, const char *name) {
    if (p == nullptr) return fail(CSA_ERR_INVALID_ARG, "%s is NULL", name);
    if (!al16(p)) return fail(CSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
    return CSA_OK;
}

size_t esize(csa_dtype dt) { return dt == CSA_BF16 ? 2 : 4; }

csa_status check_dtype(csa_dtype dt) {
    if (dt != CSA_F32 && dt != CSA_BF16) return fail(CSA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
    return CSA_OK;
}

csa_status check_c(int c) {
    if (c != 64 && c != 128 && c != 256 && c != 512)
        return fail(CSA_ERR_UNSUPPORTED, "head dim c=%d not in {64,128,256,512}", c);
    return CSA_OK;
}

csa_status check_params(const csa_params *p, int c, bool attn) {
    if (p == nullptr) return fail(CSA_ERR_INVALID_ARG, "params is NULL");
    if (p->m < 1 || p->m > 1024) return fail(CSA_ERR_UNSUPPORTED, "compression rate m=%d not in 1..1024", p->m);
    if (p->overlap != 0 && p->overlap != 1) return fail(CSA_ERR_INVALID_ARG, "overlap must be 0 or 1");
    if (p->rope_dims < 0 || (p->rope_dims & 1) || p->rope_dims > c || p->rope_dims / 2 > MAX_ROPE_PAIRS)
        return fail(CSA_ERR_UNSUPPORTED, "rope_dims=%d must be even and <= c", p->rope_dims);
    if (p->rope_dims > 0 && !(p->rope_theta > 1.0)) return fail(CSA_ERR_INVALID_ARG, "rope_theta must be > 1");
    if (p->batch_invariant != 0 && p->batch_invariant != 1)
        return fail(CSA_ERR_INVALID_ARG, "batch_invariant must be 0 or 1");
    if (p->spin_limit < 0) return fail(CSA_ERR_INVALID_ARG, "spin_limit must be >= 0");
    if (p->cache_format != CSA_CACHE_DTYPE && p->cache_format != CSA_CACHE_LOWP)
        return fail(CSA_ERR_INVALID_ARG, "cache_format must be CSA_CACHE_DTYPE or CSA_CACHE_LOWP");
    if (!(p->norm_eps >= 0.f) || std::isinf(p->norm_eps)) return fail(CSA_ERR_INVALID_ARG, "norm_eps must be finite and >= 0");
    if ((p->q_norm && !al16(p->q_norm)) || (p->kv_norm && !al16(p->kv_norm)))
        return fail(CSA_ERR_INVALID_ARG, "norm gains must be 16-byte aligned");
    if (attn) {
        if (p->n_win < 0 || p->n_win > 1024) return fail(CSA_ERR_UNSUPPORTED, "n_win=%d not in 0..1024", p->n_win);
        if (p->derotate != 0 && p->derotate != 1) return fail(CSA_ERR_INVALID_ARG, "derotate must be 0 or 1");
        if (!(p->scale >= 0.f) || std::isinf(p->scale)) return fail(CSA_ERR_INVALID_ARG, "scale must be finite and >= 0");
    }
    return CSA_OK;
}

RopeFreqs make_rope(int c, int r, double theta) {
    RopeFreqs rf;
    memset(&rf, 0, sizeof rf);
    rf.pairs = r / 2;
    rf.first = c - r;
    for (int i = 0; i < r / 2; i++) {
        rf.w[i] = pow(theta, -2.0 * i / (double)r);
        const double f = rf.w[i] / (2.0 * 3.14159265358979323846);
        rf.fh[i] = (float)f;
        rf.fl[i] = (float)(f - (double)rf.fh[i]);
    }
    return rf;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Bump allocator over a caller-provided workspace.
struct Carve {
    char *base;
    size_t off;
    void *take(size_t bytes) {
        void *p = base ? base + off : nullptr;
        off = align256(off + bytes);
        return p;
    }
};

__global__ void iota_pos_kernel(int64_t *pos, int64_t B, int64_t n) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < B * n) pos[i] = i % n;
}

cudaError_t fill_positions(int64_t *pos, int64_t B, int64_t n, cudaStream_t st) {
    if (B * n == 0) return cudaSuccess;
    iota_pos_kernel<<<(unsigned)((B * n + 255) / 256), 256, 0, st>>>(pos, B, n);
    count_launches(1);
    return cudaGetLastError();
}

csa_status check_ws(void *ws, size_t ws_bytes, size_t need) {
    if (ws == nullptr) return fail(CSA_ERR_WORKSPACE, "workspace is NULL (need %zu bytes)", need);
    if (!al16(ws)) return fail(CSA_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
    if (ws_bytes < need) return fail(CSA_ERR_WORKSPACE, "workspace has %zu bytes, need %zu", ws_bytes, need);
    return CSA_OK;
}

// ------------------------------------------------------------ stage timing

struct StageTimer {
    std::mutex mu;
    int on = 0;
    struct Pending { int stage; cudaEvent_t a, b; };
    std::vector<cudaEvent_t> pool;
    std::vector<Pending> pending;
    double ms[CSA_NUM_STAGES] = {};
    long long launches[CSA_NUM_STAGES] = {};
};
StageTimer g_timer;

// Records an event pair around one stage when timing is enabled.
struct StageScope {
    int stage;
    cudaStream_t st;
    cudaEvent_t a = nullptr, b = nullptr;
    StageScope(int s, cudaStream_t stream) : stage(s), st(stream) {
        std::lock_guard<std::mutex> g(g_timer.mu);
        if (!g_timer.on) return;
        for (cudaEvent_t *e : {&a, &b}) {
            if (!g_timer.pool.empty()) {
                *e = g_timer.pool.back();
                g_timer.pool.pop_back();
            } else if (cudaEventCreate(e) != cudaSuccess) {
                *e = nullptr;
            }
        }
        if (a && b) cudaEventRecord(a, st);
    }
    ~StageScope() {
        if (!a || !b) return;
        cudaEventRecord(b, st);
        std::lock_guard<std::mutex> g(g_timer.mu);
        g_timer.pending.push_back({stage, a, b});
    }
};

// --------------------------------------------------------------- launchers

// gain: the KV RMSNorm gains (params->kv_norm for the KV; nullptr for the
// indexer keys, which carry no norm)
csa_status do_compress(csa_dtype dt, int64_t B, int64_t n, int c, const void *C, const void *Z,
                       const float *bias, const void *Cb, const void *Zb, const float *biasb,
                       void *out, void *raw_out, const csa_params *p, int rope_dims,
                       const float *gain, cudaStream_t st) {
    RopeFreqs rf = make_rope(c, rope_dims, p->rope_theta);
    StageScope sc(CSA_STAGE_COMPRESS, st);
    if (gain && c / (dt == CSA_BF16 ? 8 : 4) > 256)
        return fail(CSA_ERR_UNSUPPORTED, "the KV norm takes c <= %d", dt == CSA_BF16 ? 2048 : 1024);
    CSA_TRY_CUDA(launch_compress(dt, B, n, c, p->m, p->overlap, C, Z, bias, Cb, Zb, biasb, out,
                                 raw_out, rf, gain, p->norm_eps > 0.f ? p->norm_eps : 1e-6f, st),
                 "csa_compress launch");
    return CSA_OK;
}

csa_status do_indexer(csa_dtype dt, int64_t B, int64_t T, int hI, int dI, int64_t E, int m,
                      const void *qI, const float *w, const void *kI, const int64_t *q_pos,
                      float *scores, int write_masked, unsigned *status, int64_t spin_limit,
                      cudaStream_t st, int max_ctas = 0) {
    StageScope sc(CSA_STAGE_INDEXER, st);
    if (dt == CSA_BF16 && indexer_tc_supported(hI, dI, B, T, E)) {
        CSA_TRY_CUDA(launch_indexer_tc(B, T, E, m, qI, w, kI, q_pos, scores, write_masked, status,
                                       max_ctas, spin_limit_of(spin_limit), st),
                     "indexer_score launch (tensor cores)");
        return CSA_OK;
    }
    CSA_TRY_CUDA(launch_indexer_simt(dt, B, T, hI, dI, E, m, qI, w, kI, q_pos, scores,
                                     write_masked, st),
                 "indexer_score launch");
    return CSA_OK;
}

csa_status do_topk(int64_t B, int64_t T, int64_t E, int k, int m, const float *scores,
                   const int64_t *q_pos, int32_t *idx, int32_t *cnt, void *scratch, cudaStream_t st,
                   int phase = 0) {
    StageScope sc(CSA_STAGE_TOPK, st);
    if (phase == 0)
        CSA_TRY_CUDA(launch_topk(B, T, E, k, m, scores, q_pos, idx, cnt, scratch, st), "topk_select launch");
    else
        CSA_TRY_CUDA(launch_topk_phase(phase, B, T, E, k, m, scores, q_pos, idx, cnt, scratch, st),
                     "topk_select launch");
    return CSA_OK;
}

// scratch bytes an attention call needs beyond the status word
size_t attn_scratch_bytes(csa_dtype dt, int64_t rows, int H, int c, int64_t E, int k, int n_win,
                          bool invariant) {
    if (!attn_tc_supported(dt, c)) return 0;
    const int64_t max_list = (k > 0 ? (int64_t)k : E) + n_win;
    const int ch = attn_tc_chunks(rows, H, max_list, invariant);
    return ch > 1 ? attn_tc_split_bytes(rows, H, c, ch) : 0;
}

csa_status do_attn(csa_dtype dt, int64_t B, int64_t T, int H, int c, int64_t E, int k, int64_t L,
                   const void *q, const int64_t *q_pos, const void *kvc, const int32_t *idx,
                   const int32_t *cnt, const void *kv_raw, const int64_t *raw_pos0,
                   const float *sink, void *out, float *lse, const csa_params *p, unsigned *status,
                   void *scratch, cudaStream_t st, int max_ctas = 0) {
    AttnArgs a;
    a.q = q; a.q_pos = q_pos; a.kvc = kvc; a.idx = idx; a.kv_raw = kv_raw; a.raw_pos0 = raw_pos0;
    a.sink = sink; a.out = out; a.lse = lse; a.status = status;
    a.Tq = T; a.H = H; a.c = c; a.E = E; a.k = k; a.L = L;
    a.m = p->m; a.n_win = p->n_win; a.derotate = p->derotate;
    a.scale = p->scale > 0.f ? p->scale : (float)(1.0 / sqrt((double)c));
    a.spin = spin_limit_of(p->spin_limit);
    a.kv8 = p->cache_format == CSA_CACHE_LOWP;
    a.q_norm = p->q_norm;
    a.norm_eps = p->norm_eps > 0.f ? p->norm_eps : 1e-6f;
    a.rope = make_rope(c, p->rope_dims, p->rope_theta);
    StageScope sc(idx ? CSA_STAGE_SPARSE_ATTN : CSA_STAGE_HCA_ATTN, st);
    // the tensor-core path addresses rows of q, kvc and kv_raw with 32-bit TMA coordinates
    const int64_t lim = 2147483647LL - 65536;
    const bool fits = B * T * H < lim && B * E < lim && B * L < lim;
    if (attn_tc_supported(dt, c) && fits) {
        const int64_t max_list = (idx ? (int64_t)k : E) + p->n_win;
        int ch = attn_tc_chunks(B * T, H, max_list, p->batch_invariant != 0);
        if (ch > 1 && scratch == nullptr) {
            // without split scratch the list runs unsplit, which changes the
            // summation order: not allowed when batch invariance was asked for
            if (p->batch_invariant)
                return fail(CSA_ERR_WORKSPACE, "batch_invariant needs the split-KV scratch of attn_ws_size");
            ch = 1;
        }
        if (ch > 1 && !p->batch_invariant) {
            // no more chunk items than the launch has CTAs for in one round:
            // each item ends in a partial-output epilogue, and a last round
            // that only some CTAs fill costs a whole item's time
            const int64_t units = B * T * ((H + 63) / 64);
            const int64_t ctas = max_ctas > 0 && max_ctas < device_sms() ? max_ctas : device_sms();
            const int64_t fit = ctas / units;
            if (fit < ch) ch = fit > 1 ? (int)fit : 1;
        }
        CSA_TRY_CUDA(launch_attn_tc(B, a, cnt, ch, scratch, max_ctas, st),
                     "attention launch (tensor cores)");
        return CSA_OK;
    }
    if (a.kv8) return fail(CSA_ERR_UNSUPPORTED, "FP8 entries need the tensor-core path");
    CSA_TRY_CUDA(launch_attn_simt(dt, B, a, st), "attention launch");
    return CSA_OK;
}

csa_status check_attn_common(csa_dtype dt, int64_t B, int64_t T, int H, int c, int64_t E, int64_t L,
                             const void *q, const int64_t *q_pos, const void *kvc, const void *kv_raw,
                             const int64_t *raw_pos0, const float *sink, const void *out,
                             const csa_params *p) {
    CSA_TRY(check_dtype(dt));
    CSA_TRY(check_c(c));
    CSA_TRY(check_params(p, c, true));
    if (B < 0 || T < 0 || E < 0 || L < 0) return fail(CSA_ERR_INVALID_ARG, "negative size");
    if (H < 1 || H > 128) return fail(CSA_ERR_UNSUPPORTED, "H=%d not in 1..128", H);
    if (p->cache_format == CSA_CACHE_LOWP && (dt != CSA_BF16 || c != 512 || p->rope_dims != 64))
        return fail(CSA_ERR_UNSUPPORTED, "FP8 entries need bf16, c = 512 and rope_dims = 64");
    if (B * T == 0) return CSA_OK;
    CSA_TRY(need_ptr(q, "q"));
    CSA_TRY(need_ptr(q_pos, "q_pos"));
    CSA_TRY(need_ptr(sink, "sink"));
    CSA_TRY(need_ptr(out, "out"));
    if (E > 0) CSA_TRY(need_ptr(kvc, "kvc"));
    if (p->n_win > 0) {
        if (L <= 0) return fail(CSA_ERR_INVALID_ARG, "n_win > 0 needs raw rows (L > 0)");
        CSA_TRY(need_ptr(kv_raw, "kv_raw"));
        if (raw_pos0 == nullptr) return fail(CSA_ERR_INVALID_ARG, "raw_pos0 is NULL");
    }
    return CSA_OK;
}

}  // namespace

namespace csa {

// One thread waits on a barrier whose single expected arrival never comes;
// the bounded wait gives up after `spin` polls and records ST_TIMEOUT.
__global__ void wait_probe_kernel(unsigned *status, long long spin) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_barrier_init();
    tc::mbar_wait(&bar, 0, status, (volatile int *)&abort_flag, spin);
}

cudaError_t launch_wait_probe(unsigned *status, long long spin, cudaStream_t st) {
    wait_probe_kernel<<<1, 32, 0, st>>>(status, spin);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace csa

// ====================================================================== ABI

extern "C" {

const char *csa_last_error(void) { return g_err; }

const char *csa_version(void) { return "csa-b300 0.1 (sm_103a)"; }

int64_t csa_launch_count(void) { return g_launches.load(); }

csa_status csa_timing_enable(int32_t on) {
    std::lock_guard<std::mutex> g(g_timer.mu);
    g_timer.on = on ? 1 : 0;
    return CSA_OK;
}

csa_status csa_timing_read(double *ms, int64_t *launches, int32_t nstages) {
    std::vector<StageTimer::Pending> pend;
    {
        std::lock_guard<std::mutex> g(g_timer.mu);
        pend.swap(g_timer.pending);
    }
    double acc[CSA_NUM_STAGES] = {};
    long long cnt[CSA_NUM_STAGES] = {};
    cudaError_t err = cudaSuccess;
    for (auto &p : pend) {
        float t = 0.f;
        cudaError_t e = cudaEventSynchronize(p.b);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&t, p.a, p.b);
        if (e != cudaSuccess) err = e;
        acc[p.stage] += t;
        cnt[p.stage] += 1;
    }
    {
        std::lock_guard<std::mutex> g(g_timer.mu);
        for (auto &p : pend) {
            g_timer.pool.push_back(p.a);
            g_timer.pool.push_back(p.b);
        }
    }
    for (int s = 0; s < nstages && s < CSA_NUM_STAGES; s++) {
        if (ms) ms[s] = acc[s];
        if (launches) launches[s] = cnt[s];
    }
    if (err != cudaSuccess) return cuda_fail(err, "timing read");
    return CSA_OK;
}

csa_status csa_workspace_init(void *ws, size_t ws_bytes, void *stream) {
    CSA_TRY(check_ws(ws, ws_bytes, CSA_STATUS_BYTES));
    CSA_TRY_CUDA(cudaMemsetAsync(ws, 0, CSA_STATUS_BYTES, (cudaStream_t)stream), "workspace init");
    return CSA_OK;
}

csa_status csa_stream_status(void *ws, void *stream) {
    if (ws == nullptr) return fail(CSA_ERR_INVALID_ARG, "workspace is NULL");
    CSA_TRY_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "stream synchronize");
    unsigned word = 0;
    CSA_TRY_CUDA(cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost), "status read");
    if (word == 0) return CSA_OK;
    CSA_TRY_CUDA(cudaMemset(ws, 0, sizeof word), "status clear");
    if (word & ST_TIMEOUT) return fail(CSA_ERR_TIMEOUT, "a bounded device wait ran out (status 0x%x)", word);
    return fail(CSA_ERR_DEVICE, "device range check: %s%s(status 0x%x)",
                (word & ST_BAD_INDEX) ? "selected index outside the cache; " : "",
                (word & ST_NO_WINDOW_ROW) ? "window position missing from kv_raw; " : "", word);
}

csa_status csa_wait_probe(int64_t spin_limit, void *ws, size_t ws_bytes, void *stream) {
    if (spin_limit < 0) return fail(CSA_ERR_INVALID_ARG, "spin_limit must be >= 0");
    CSA_TRY(check_ws(ws, ws_bytes, CSA_STATUS_BYTES));
    CSA_TRY_CUDA(launch_wait_probe((unsigned *)ws, spin_limit_of(spin_limit), (cudaStream_t)stream),
                 "wait probe launch");
    return CSA_OK;
}

csa_status csa_compress(csa_dtype dtype, int64_t B, int64_t n, int32_t c, const void *C,
                        const void *Z, const float *bias, const void *Cb, const void *Zb,
                        const float *biasb, void *out, void *raw_out, const csa_params *params,
                        void *stream) {
    CSA_TRY(check_dtype(dtype));
    if (c < 8 || c % 8 != 0 || c > 4096) return fail(CSA_ERR_UNSUPPORTED, "c=%d must be a multiple of 8 in 8..4096", c);
    CSA_TRY(check_params(params, c, false));
    if (B < 0 || n < 0) return fail(CSA_ERR_INVALID_ARG, "negative size");
    if (B * n == 0) return CSA_OK;
    CSA_TRY(need_ptr(C, "C"));
    CSA_TRY(need_ptr(Z, "Z"));
    CSA_TRY(need_ptr(bias, "bias"));
    if (params->overlap) {
        CSA_TRY(need_ptr(Cb, "Cb"));
        CSA_TRY(need_ptr(Zb, "Zb"));
        CSA_TRY(need_ptr(biasb, "biasb"));
    }
    if (n / params->m > 0) CSA_TRY(need_ptr(out, "out"));
    if (raw_out != nullptr && !al16(raw_out)) return fail(CSA_ERR_INVALID_ARG, "raw_out is not 16-byte aligned");
    return do_compress(dtype, B, n, c, C, Z, bias, Cb, Zb, biasb, out, raw_out, params,
                       params->rope_dims, params->kv_norm, (cudaStream_t)stream);
}

size_t indexer_score_ws_size(void) { return CSA_STATUS_BYTES; }

csa_status indexer_score(csa_dtype dtype, int64_t B, int64_t T, int32_t hI, int32_t dI, int64_t E,
                         int32_t m, const void *qI, const float *w, const void *kI,
                         const int64_t *q_pos, float *scores, void *ws, size_t ws_bytes,
                         void *stream) {
    CSA_TRY(check_dtype(dtype));
    if (B < 0 || T < 0 || E < 0) return fail(CSA_ERR_INVALID_ARG, "negative size");
    if (hI < 1 || hI > 64) return fail(CSA_ERR_UNSUPPORTED, "hI=%d not in 1..64", hI);
    if (dI != 32 && dI != 64 && dI != 128) return fail(CSA_ERR_UNSUPPORTED, "dI=%d not in {32,64,128}", dI);
    if (m < 1) return fail(CSA_ERR_INVALID_ARG, "m must be >= 1");
    if (E > 2147483647LL) return fail(CSA_ERR_UNSUPPORTED, "E too large");
    CSA_TRY(check_ws(ws, ws_bytes, indexer_score_ws_size()));
    if (B * T == 0 || E == 0) return CSA_OK;
    CSA_TRY(need_ptr(qI, "qI"));
    CSA_TRY(need_ptr(w, "w"));
    CSA_TRY(need_ptr(kI, "kI"));
    CSA_TRY(need_ptr(q_pos, "q_pos"));
    CSA_TRY(need_ptr(scores, "scores"));
    return do_indexer(dtype, B, T, hI, dI, E, m, qI, w, kI, q_pos, scores, 1, (unsigned *)ws, 0,
                      (cudaStream_t)stream);
}

size_t topk_select_ws_size(int64_t B, int64_t T, int64_t E, int32_t k) {
    (void)k;
    if (B < 0 || T < 0 || E < 0) return 0;
    return CSA_STATUS_BYTES + topk_scratch_bytes(B * T, E);
}

csa_status topk_select(int64_t B, int64_t T, int64_t E, int32_t k, int32_t m, const float *scores,
                       const int64_t *q_pos, int32_t *idx, int32_t *cnt, void *ws, size_t ws_bytes,
                       void *stream) {
    if (B < 0 || T < 0 || E < 0) return fail(CSA_ERR_INVALID_ARG, "negative size");
    if (k < 1 || k > 2048) return fail(CSA_ERR_UNSUPPORTED, "k=%d not in 1..2048", k);
    if (m < 1) return fail(CSA_ERR_INVALID_ARG, "m must be >= 1");
    if (E > 2147483647LL) return fail(CSA_ERR_UNSUPPORTED, "E too large");
    CSA_TRY(check_ws(ws, ws_bytes, topk_select_ws_size(B, T, E, k)));
    if (B * T == 0) return CSA_OK;
    if (E > 0) CSA_TRY(need_ptr(scores, "scores"));
    CSA_TRY(need_ptr(q_pos, "q_pos"));
    CSA_TRY(need_ptr(idx, "idx"));
    CSA_TRY(need_ptr(cnt, "cnt"));
    return do_topk(B, T, E, k, m, scores, q_pos, idx, cnt, (char *)ws + CSA_STATUS_BYTES,
                   (cudaStream_t)stream);
}

size_t attn_ws_size(csa_dtype dtype, int64_t B, int64_t T, int32_t H, int32_t c, int64_t E,
                    int32_t k, const csa_params *params) {
    if (params == nullptr || B < 0 || T < 0 || E < 0) return CSA_STATUS_BYTES;
    return CSA_STATUS_BYTES + attn_scratch_bytes(dtype, B * T, H, c, E, k, params->n_win, params->batch_invariant != 0);
}

csa_status sparse_attn(csa_dtype dtype, int64_t B, int64_t T, int32_t H, int32_t c, int64_t E,
                       int32_t k, int64_t L, const void *q, const int64_t *q_pos, const void *kvc,
                       const int32_t *idx, const void *kv_raw, const int64_t *raw_pos0,
                       const float *sink, void *out, float *lse, const csa_params *params,
                       void *ws, size_t ws_bytes, void *stream) {
    CSA_TRY(check_attn_common(dtype, B, T, H, c, E, L, q, q_pos, kvc, kv_raw, raw_pos0, sink, out,
                              params));
    if (k < 1 || k > 2048) return fail(CSA_ERR_UNSUPPORTED, "k=%d not in 1..2048", k);
    CSA_TRY(check_ws(ws, ws_bytes, attn_ws_size(dtype, B, T, H, c, E, k, params)));
    if (B * T == 0) return CSA_OK;
    CSA_TRY(need_ptr(idx, "idx"));
    if (lse != nullptr && !al16(lse)) return fail(CSA_ERR_INVALID_ARG, "lse is not 16-byte aligned");
    return do_attn(dtype, B, T, H, c, E, k, L, q, q_pos, kvc, idx, nullptr, kv_raw, raw_pos0, sink,
                   out, lse, params, (unsigned *)ws, (char *)ws + CSA_STATUS_BYTES,
                   (cudaStream_t)stream);
}

csa_status hca_attn(csa_dtype dtype, int64_t B, int64_t T, int32_t H, int32_t c, int64_t E,
                    int64_t L, const void *q, const int64_t *q_pos, const void *kvc,
                    const void *kv_raw, const int64_t *raw_pos0, const float *sink, void *out,
                    float *lse, const csa_params *params, void *ws, size_t ws_bytes, void *stream) {
    CSA_TRY(check_attn_common(dtype, B, T, H, c, E, L, q, q_pos, kvc, kv_raw, raw_pos0, sink, out,
                              params));
    CSA_TRY(check_ws(ws, ws_bytes, attn_ws_size(dtype, B, T, H, c, E, 0, params)));
    if (B * T == 0) return CSA_OK;
    if (lse != nullptr && !al16(lse)) return fail(CSA_ERR_INVALID_ARG, "lse is not 16-byte aligned");
    return do_attn(dtype, B, T, H, c, E, 0, L, q, q_pos, kvc, nullptr, nullptr, kv_raw, raw_pos0,
                   sink, out, lse, params, (unsigned *)ws, (char *)ws + CSA_STATUS_BYTES,
                   (cudaStream_t)stream);
}

// ------------------------------------------------------------ fused: CSA prefill

static size_t csa_prefill_layout(Carve &cv, csa_dtype dt, int64_t B, int64_t n, int H, int c,
                                 int dI, const csa_params *p, void **pos, void **rp0, void **kvc,
                                 void **kic, void **raw, void **sc, void **idx, void **cnt,
                                 void **tks, void **asc) {
    const int64_t E = n / p->m;
    cv.take(CSA_STATUS_BYTES);
    *pos = cv.take((size_t)B * n * 8);
    *rp0 = cv.take((size_t)B * 8);
    *kvc = cv.take((size_t)B * E * c * esize(dt));
    *kic = cv.take((size_t)B * E * dI * esize(dt));
    *raw = cv.take((size_t)B * n * c * esize(dt));
    *sc = cv.take((size_t)B * n * E * 4);
    *idx = cv.take((size_t)B * n * p->top_k * 4);
    *cnt = cv.take((size_t)B * n * 4);
    *tks = cv.take(topk_scratch_bytes(B * n, E));
    *asc = cv.take(attn_scratch_bytes(dt, B * n, H, c, E, p->top_k, p->n_win, p->batch_invariant != 0));
    return cv.off;
}

size_t csa_prefill_ws_size(csa_dtype dtype, int64_t B, int64_t n, int32_t H, int32_t c, int32_t hI,
                           int32_t dI, const csa_params *params) {
    (void)hI;
    if (params == nullptr || params->m < 1 || B < 0 || n < 0) return 0;
    Carve cv{nullptr, 0};
    void *a, *b, *d, *e, *f, *g, *h, *i, *j, *k;
    return csa_prefill_layout(cv, dtype, B, n, H, c, dI, params, &a, &b, &d, &e, &f, &g, &h, &i, &j,
                              &k);
}

csa_status csa_prefill(csa_dtype dtype, int64_t B, int64_t n, int32_t H, int32_t c, int32_t hI,
                       int32_t dI, const void *C, const void *Z, const float *bias, const void *Cb,
                       const void *Zb, const float *biasb, const void *Ck, const void *Zk,
                       const float *biask, const void *Ckb, const void *Zkb, const float *biaskb,
                       const void *q, const void *qI, const float *w, const float *sink, void *out,
                       int32_t *idx_out, const csa_params *params, void *ws, size_t ws_bytes,
                       void *stream) {
    CSA_TRY(check_dtype(dtype));
    CSA_TRY(check_c(c));
    CSA_TRY(check_params(params, c, true));
    if (B < 0 || n < 0) return fail(CSA_ERR_INVALID_ARG, "negative size");
    if (H < 1 || H > 128) return fail(CSA_ERR_UNSUPPORTED, "H=%d not in 1..128", H);
    if (hI < 1 || hI > 64) return fail(CSA_ERR_UNSUPPORTED, "hI=%d not in 1..64", hI);
    if (dI != 32 && dI != 64 && dI != 128) return fail(CSA_ERR_UNSUPPORTED, "dI=%d not in {32,64,128}", dI);
    if (params->top_k < 1 || params->top_k > 2048) return fail(CSA_ERR_UNSUPPORTED, "top_k=%d not in 1..2048", params->top_k);
    if (params->cache_format != CSA_CACHE_DTYPE) return fail(CSA_ERR_UNSUPPORTED, "csa_prefill stores caches in dtype");
    CSA_TRY(check_ws(ws, ws_bytes, csa_prefill_ws_size(dtype, B, n, H, c, hI, dI, params)));
    if (B * n == 0) return CSA_OK;
    const char *names[] = {"C", "Z", "bias", "Ck", "Zk", "biask", "q", "qI", "w", "sink", "out"};
    const void *ptrs[] = {C, Z, bias, Ck, Zk, biask, q, qI, w, sink, out};
    for (int i = 0; i < 11; i++) CSA_TRY(need_ptr(ptrs[i], names[i]));
    if (params->overlap) {
        const char *nb[] = {"Cb", "Zb", "biasb", "Ckb", "Zkb", "biaskb"};
        const void *pb[] = {Cb, Zb, biasb, Ckb, Zkb, biaskb};
        for (int i = 0; i < 6; i++) CSA_TRY(need_ptr(pb[i], nb[i]));
    }
    if (idx_out != nullptr && !al16(idx_out)) return fail(CSA_ERR_INVALID_ARG, "idx_out is not 16-byte aligned");
    cudaStream_t st = (cudaStream_t)stream;
    Carve cv{(char *)ws, 0};
    void *pos, *rp0, *kvc, *kic, *raw, *sc, *idx, *cnt, *tks, *asc;
    csa_prefill_layout(cv, dtype, B, n, H, c, dI, params, &pos, &rp0, &kvc, &kic, &raw, &sc, &idx, &cnt,
                       &tks, &asc);
    if (idx_out) idx = idx_out;
    const int64_t E = n / params->m;
    unsigned *status = (unsigned *)ws;
    CSA_TRY_CUDA(fill_positions((int64_t *)pos, B, n, st), "positions");
    CSA_TRY_CUDA(cudaMemsetAsync(rp0, 0, (size_t)B * 8, st), "raw_pos0");
    CSA_TRY(do_compress(dtype, B, n, c, C, Z, bias, Cb, Zb, biasb, kvc, raw, params,
                        params->rope_dims, params->kv_norm, st));
    CSA_TRY(do_compress(dtype, B, n, dI, Ck, Zk, biask, Ckb, Zkb, biaskb, kic, nullptr, params, 0,
                        nullptr, st));
    CSA_TRY(do_indexer(dtype, B, n, hI, dI, E, params->m, qI, w, kic, (const int64_t *)pos,
                       (float *)sc, 0, status, params->spin_limit, st));
    CSA_TRY(do_topk(B, n, E, params->top_k, params->m, (const float *)sc, (const int64_t *)pos,
                    (int32_t *)idx, (int32_t *)cnt, tks, st));
    return do_attn(dtype, B, n, H, c, E, params->top_k, n, q, (const int64_t *)pos, kvc,
                   (const int32_t *)idx, (const int32_t *)cnt, raw, (const int64_t *)rp0, sink, out,
                   nullptr, params, status, asc, st);
}

// ------------------------------------------------------------ fused: HCA prefill

static size_t hca_prefill_layout(Carve &cv, csa_dtype dt, int64_t B, int64_t n, int H, int c,
                                 const csa_params *p, void **pos, void **rp0, void **kvc,
                                 void **raw, void **asc) {
    const int64_t E = n / p->m;
    cv.take(CSA_STATUS_BYTES);
    *pos = cv.take((size_t)B * n * 8);
    *rp0 = cv.take((size_t)B * 8);
    *kvc = cv.take((size_t)B * E * c * esize(dt));
    *raw = cv.take((size_t)B * n * c * esize(dt));
    *asc = cv.take(attn_scratch_bytes(dt, B * n, H, c, E, 0, p->n_win, p->batch_invariant != 0));
    return cv.off;
}

size_t hca_prefill_ws_size(csa_dtype dtype, int64_t B, int64_t n, int32_t H, int32_t c,
                           const csa_params *params) {
    if (params == nullptr || params->m < 1 || B < 0 || n < 0) return 0;
    Carve cv{nullptr, 0};
    void *a, *b, *d, *e, *f;
    return hca_prefill_layout(cv, dtype, B, n, H, c, params, &a, &b, &d, &e, &f);
}

csa_status hca_prefill(csa_dtype dtype, int64_t B, int64_t n, int32_t H, int32_t c, const void *C,
                       const void *Z, const float *bias, const void *q, const float *sink,
                       void *out, const csa_params *params, void *ws, size_t ws_bytes,
                       void *stream) {
    CSA_TRY(check_dtype(dtype));
    CSA_TRY(check_c(c));
    CSA_TRY(check_params(params, c, true));
    if (params->overlap) return fail(CSA_ERR_UNSUPPORTED, "HCA compression has one branch (overlap = 0)");
    if (params->cache_format != CSA_CACHE_DTYPE) return fail(CSA_ERR_UNSUPPORTED, "hca_prefill stores caches in dtype");
    if (B < 0 || n < 0) return fail(CSA_ERR_INVALID_ARG, "negative size");
    if (H < 1 || H > 128) return fail(CSA_ERR_UNSUPPORTED, "H=%d not in 1..128", H);
    CSA_TRY(check_ws(ws, ws_bytes, hca_prefill_ws_size(dtype, B, n, H, c, params)));
    if (B * n == 0) return CSA_OK;
    const char *names[] = {"C", "Z", "bias", "q", "sink", "out"};
    const void *ptrs[] = {C, Z, bias, q, sink, out};
    for (int i = 0; i < 6; i++) CSA_TRY(need_ptr(ptrs[i], names[i]));
    cudaStream_t st = (cudaStream_t)stream;
    Carve cv{(char *)ws, 0};
    void *pos, *rp0, *kvc, *raw, *asc;
    hca_prefill_layout(cv, dtype, B, n, H, c, params, &pos, &rp0, &kvc, &raw, &asc);
    const int64_t E = n / params->m;
    CSA_TRY_CUDA(fill_positions((int64_t *)pos, B, n, st), "positions");
    CSA_TRY_CUDA(cudaMemsetAsync(rp0, 0, (size_t)B * 8, st), "raw_pos0");
    CSA_TRY(do_compress(dtype, B, n, c, C, Z, bias, nullptr, nullptr, nullptr, kvc, raw, params,
                        params->rope_dims, params->kv_norm, st));
    return do_attn(dtype, B, n, H, c, E, 0, n, q, (const int64_t *)pos, kvc, nullptr, nullptr, raw,
                   (const int64_t *)rp0, sink, out, nullptr, params, (unsigned *)ws, asc, st);
}

// ------------------------------------------------------------ fused: decode

static size_t decode_layout(Carve &cv, csa_dtype dt, int64_t B, int H, int c, int64_t E,
                            int64_t E2, const csa_params *p, const csa_params *p2, void **sc,
                            void **idx, void **cnt, void **tks, void **asc, void **asc2) {
    cv.take(CSA_STATUS_BYTES);
    *sc = cv.take((size_t)B * E * 4);
    *idx = cv.take((size_t)B * p->top_k * 4);
    *cnt = cv.take((size_t)B * 4);
    *tks = cv.take(topk_scratch_bytes(B, E));
    *asc = cv.take(attn_scratch_bytes(dt, B, H, c, E, p->top_k, p->n_win, p->batch_invariant != 0));
    *asc2 = cv.take(p2 ? attn_scratch_bytes(dt, B, H, c, E2, 0, p2->n_win, p2->batch_invariant != 0) : 0);
    return cv.off;
}

// Auxiliary stream sets, one per concurrent hybrid_decode call: a call takes
// a set (stream + fork/join events) from its device's pool, records fork on
// its own stream, runs the HCA layer's attention on the set's stream after
// fork, records join there and makes its own stream wait on join; then it
// returns the set.  A set is never shared by two calls in flight, so every
// call's auxiliary work waits on its own stream.  Sets are created on demand
// and kept until the process exits.
struct AuxSet {
    cudaStream_t aux = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
static std::vector<AuxSet> g_aux_free[MAX_DEVICES];
static std::mutex g_aux_mu;

struct AuxLease {
    int dev = -1;
    AuxSet set;
    cudaStream_t waiter = nullptr;   // set once work was forked onto set.aux
    // the join: record it on the auxiliary stream and make the caller's
    // stream wait on it
    cudaError_t join() {
        cudaError_t e1 = cudaEventRecord(set.join, set.aux);
        cudaError_t e2 = cudaStreamWaitEvent(waiter, set.join, 0);
        waiter = nullptr;
        return e1 != cudaSuccess ? e1 : e2;
    }
    ~AuxLease() {
        if (dev < 0) return;
        // an early return after the fork still joins, so the set goes back to
        // the pool with nothing of this call pending that the caller's stream
        // does not wait for
        if (waiter != nullptr) (void)join();
        std::lock_guard<std::mutex> g(g_aux_mu);
        g_aux_free[dev].push_back(set);
    }
};

static csa_status take_aux(AuxLease &lease) {
    int dev = 0;
    CSA_TRY_CUDA(cudaGetDevice(&dev), "get device");
    if (dev < 0 || dev >= MAX_DEVICES) return fail(CSA_ERR_UNSUPPORTED, "device index %d", dev);
    {
        std::lock_guard<std::mutex> g(g_aux_mu);
        if (!g_aux_free[dev].empty()) {
            lease.set = g_aux_free[dev].back();
            g_aux_free[dev].pop_back();
            lease.dev = dev;
            return CSA_OK;
        }
    }
    AuxSet a;
    CSA_TRY_CUDA(cudaStreamCreateWithFlags(&a.aux, cudaStreamNonBlocking), "aux stream");
    CSA_TRY_CUDA(cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming), "fork event");
    CSA_TRY_CUDA(cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming), "join event");
    lease.set = a;
    lease.dev = dev;
    return CSA_OK;
}

size_t hybrid_decode_ws_size(csa_dtype dtype, int64_t B, int32_t H, int32_t c, int32_t hI,
                             int32_t dI, int64_t E, int64_t E2, const csa_params *params,
                             const csa_params *params2) {
    (void)hI; (void)dI;
    if (params == nullptr || B < 0 || E < 0) return 0;
    Carve cv{nullptr, 0};
    void *a, *b, *d, *e, *f, *g;
    return decode_layout(cv, dtype, B, H, c, E, E2, params, params2, &a, &b, &d, &e, &f, &g);
}

csa_status hybrid_decode(csa_dtype dtype, int64_t B, int32_t H, int32_t c, int32_t hI, int32_t dI,
                         int64_t E, int64_t E2, int64_t L, const void *q, const void *qI,
                         const float *w, const void *kvc, const void *kIc, const void *kv_raw,
                         const float *sink, const void *q2, const void *kvc2, const void *kv_raw2,
                         const float *sink2, const int64_t *q_pos, const int64_t *raw_pos0,
                         void *out, void *out2, int32_t *idx_out, const csa_params *params,
                         const csa_params *params2, void *ws, size_t ws_bytes, void *stream) {
    CSA_TRY(check_attn_common(dtype, B, 1, H, c, E, L, q, q_pos, kvc, kv_raw, raw_pos0, sink, out,
                              params));
    if (hI < 1 || hI > 64) return fail(CSA_ERR_UNSUPPORTED, "hI=%d not in 1..64", hI);
    if (dI != 32 && dI != 64 && dI != 128) return fail(CSA_ERR_UNSUPPORTED, "dI=%d not in {32,64,128}", dI);
    if (params->top_k < 1 || params->top_k > 2048) return fail(CSA_ERR_UNSUPPORTED, "top_k=%d not in 1..2048", params->top_k);
    if (E > 2147483647LL) return fail(CSA_ERR_UNSUPPORTED, "E too large");
    if (params->cache_format == CSA_CACHE_LOWP && (hI != 64 || dI != 128 || B * E > 2147483647LL))
        return fail(CSA_ERR_UNSUPPORTED, "MXFP4 keys need hI = 64 and dI = 128");
    const bool hca = q2 != nullptr;
    if (hca) {
        CSA_TRY(check_attn_common(dtype, B, 1, H, c, E2, L, q2, q_pos, kvc2, kv_raw2, raw_pos0,
                                  sink2, out2, params2));
    }
    CSA_TRY(check_ws(ws, ws_bytes, hybrid_decode_ws_size(dtype, B, H, c, hI, dI, E, E2, params,
                                                         params2)));
    if (B == 0) return CSA_OK;
    if (E > 0) {
        CSA_TRY(need_ptr(qI, "qI"));
        CSA_TRY(need_ptr(w, "w"));
        CSA_TRY(need_ptr(kIc, "kIc"));
    }
    if (idx_out != nullptr && !al16(idx_out)) return fail(CSA_ERR_INVALID_ARG, "idx_out is not 16-byte aligned");
    cudaStream_t st = (cudaStream_t)stream;
    Carve cv{(char *)ws, 0};
    void *sc, *idx, *cnt, *tks, *asc, *asc2;
    decode_layout(cv, dtype, B, H, c, E, E2, params, hca ? params2 : nullptr, &sc, &idx, &cnt, &tks,
                  &asc, &asc2);
    if (idx_out) idx = idx_out;
    unsigned *status = (unsigned *)ws;
    // The HCA layer's attention does not depend on the CSA layer.  It starts
    // first, on an auxiliary stream, on a third of the SMs; the CSA indexer
    // (which streams kI at the HBM rate and needs few SMs to do so) runs
    // beside it on the rest, then the CSA top-k and sparse attention.  (The
    // Pro decode step, B = 8 at 1M positions, measured 0.183 / 0.168 / 0.170
    // ms with 32 / 48 / 64 SMs for the HCA branch: past a third the CSA chain
    // is the critical path.  It was 0.246 ms when the HCA attention waited
    // for the CSA top-k's collection.  The outputs are bitwise the same,
    // since no kernel's result depends on its grid.)
    const bool concurrent = hca && dtype == CSA_BF16 && attn_tc_supported(dtype, c);
    AuxLease ax;
    int rest = 0;
    if (concurrent) {
        CSA_TRY(take_aux(ax));
        const int sms = device_sms();
        const int hca_sms = sms / 3;
        rest = sms - hca_sms;
        CSA_TRY_CUDA(cudaEventRecord(ax.set.fork, st), "fork");
        CSA_TRY_CUDA(cudaStreamWaitEvent(ax.set.aux, ax.set.fork, 0), "fork wait");
        ax.waiter = st;
        CSA_TRY(do_attn(dtype, B, 1, H, c, E2, 0, L, q2, q_pos, kvc2, nullptr, nullptr, kv_raw2,
                        raw_pos0, sink2, out2, nullptr, params2, status, asc2, ax.set.aux, hca_sms));
    }
    if (params->cache_format == CSA_CACHE_LOWP) {
        StageScope si(CSA_STAGE_INDEXER, st);
        CSA_TRY_CUDA(launch_indexer_fp4(B, E, params->m, qI, w, kIc, q_pos, (float *)sc, status,
                                        spin_limit_of(params->spin_limit), rest, st),
                     "indexer launch (MXFP4 keys)");
    } else {
        CSA_TRY(do_indexer(dtype, B, 1, hI, dI, E, params->m, qI, w, kIc, q_pos, (float *)sc, 0, status,
                           params->spin_limit, st, rest));
    }
    CSA_TRY(do_topk(B, 1, E, params->top_k, params->m, (const float *)sc, q_pos, (int32_t *)idx,
                    (int32_t *)cnt, tks, st, 1));
    CSA_TRY(do_topk(B, 1, E, params->top_k, params->m, (const float *)sc, q_pos, (int32_t *)idx,
                    (int32_t *)cnt, tks, st, 2));
    CSA_TRY(do_attn(dtype, B, 1, H, c, E, params->top_k, L, q, q_pos, kvc, (const int32_t *)idx,
                    (const int32_t *)cnt, kv_raw, raw_pos0, sink, out, nullptr, params, status, asc,
                    st));
    if (concurrent) CSA_TRY_CUDA(ax.join(), "join");
    if (!concurrent && hca) {
        CSA_TRY(do_attn(dtype, B, 1, H, c, E2, 0, L, q2, q_pos, kvc2, nullptr, nullptr, kv_raw2,
                        raw_pos0, sink2, out2, nullptr, params2, status, asc2, st));
    }
    return CSA_OK;
}

// ------------------------------------------------------ low-precision caches

size_t index_fp4_bytes(int64_t rows) { return rows < 0 ? 0 : mxfp4_bytes(rows); }

csa_status quantize_kv_fp8(csa_dtype dtype, int64_t rows, int32_t c, int32_t rope_dims, const void *src,
                           void *dst, void *stream) {
    CSA_TRY(check_dtype(dtype));
    if (c != 512 || rope_dims != 64) return fail(CSA_ERR_UNSUPPORTED, "FP8 records hold c = 512 with 64 rotary dims");
    if (rows < 0) return fail(CSA_ERR_INVALID_ARG, "negative size");
    if (rows == 0) return CSA_OK;
    if (rows > ((int64_t)1 << 40)) return fail(CSA_ERR_UNSUPPORTED, "rows too large");
    CSA_TRY(need_ptr(src, "src"));
    CSA_TRY(need_ptr(dst, "dst"));
    CSA_TRY_CUDA(launch_quant_kv_fp8(dtype, rows, src, dst, (cudaStream_t)stream), "quantize_kv_fp8 launch");
    return CSA_OK;
}

csa_status quantize_index_fp4(csa_dtype dtype, int64_t rows, int32_t d, const void *src, void *dst,
                              void *stream) {
    CSA_TRY(check_dtype(dtype));
    if (d != 128) return fail(CSA_ERR_UNSUPPORTED, "MXFP4 rows hold d = 128 values");
    if (rows < 0) return fail(CSA_ERR_INVALID_ARG, "negative size");
    if (rows == 0) return CSA_OK;
    if (rows > ((int64_t)1 << 40)) return fail(CSA_ERR_UNSUPPORTED, "rows too large");
    CSA_TRY(need_ptr(src, "src"));
    CSA_TRY(need_ptr(dst, "dst"));
    CSA_TRY_CUDA(launch_quant_mxfp4(dtype, rows, src, dst, (cudaStream_t)stream), "quantize_index_fp4 launch");
    return CSA_OK;
}

csa_status indexer_score_fp4(int64_t B, int64_t E, int32_t m, const void *qI, const float *w,
                             const void *kI4, const int64_t *q_pos, float *scores, void *ws,
                             size_t ws_bytes, void *stream) {
    if (B < 0 || E < 0) return fail(CSA_ERR_INVALID_ARG, "negative size");
    if (m < 1) return fail(CSA_ERR_INVALID_ARG, "m must be >= 1");
    if (B * E > 2147483647LL) return fail(CSA_ERR_UNSUPPORTED, "B x E too large");
    CSA_TRY(check_ws(ws, ws_bytes, CSA_STATUS_BYTES));
    if (B == 0 || E == 0) return CSA_OK;
    const char *names[] = {"qI", "w", "kI4", "q_pos", "scores"};
    const void *ptrs[] = {qI, w, kI4, q_pos, scores};
    for (int i = 0; i < 5; i++) CSA_TRY(need_ptr(ptrs[i], names[i]));
    cudaStream_t st = (cudaStream_t)stream;
    StageScope sc(CSA_STAGE_INDEXER, st);
    CSA_TRY_CUDA(launch_indexer_fp4(B, E, m, qI, w, kI4, q_pos, scores, (unsigned *)ws, DEFAULT_SPIN_LIMIT,
                                    0, st),
                 "indexer_score_fp4 launch");
    CSA_TRY_CUDA(launch_mask_tail(scores, q_pos, B, E, m, st), "mask launch");
    return CSA_OK;
}

// ------------------------------------------------- grouped output projection

size_t out_proj_ws_size(int64_t T, int32_t H, int32_t heads_per_group, int32_t d_g) {
    if (T < 0 || H < 1 || heads_per_group < 1 || d_g < 0 || H % heads_per_group) return CSA_STATUS_BYTES;
    return CSA_STATUS_BYTES + align256((size_t)T * (H / heads_per_group) * d_g * 2);
}

csa_status out_proj(int64_t T, int32_t H, int32_t c, int32_t heads_per_group, int32_t d_g, int32_t d,
                    const void *o, const void *w_g, const void *w_o, void *y, void *ws, size_t ws_bytes,
                    void *stream) {
    if (T < 0) return fail(CSA_ERR_INVALID_ARG, "negative size");
    if (H < 1 || c < 1 || heads_per_group < 1 || H % heads_per_group)
        return fail(CSA_ERR_INVALID_ARG, "H=%d must be a multiple of heads_per_group=%d", H, heads_per_group);
    const int G = H / heads_per_group;
    const int64_t kin = (int64_t)heads_per_group * c;
    if (d_g < 256 || d_g % 256 || d < 256 || d % 256)
        return fail(CSA_ERR_UNSUPPORTED, "d_g=%d and d=%d must be positive multiples of 256", d_g, d);
    if (kin % 64 || kin > (1 << 20) || (int64_t)G * d_g > (1 << 20))
        return fail(CSA_ERR_UNSUPPORTED, "heads_per_group * c = %lld must be a multiple of 64", (long long)kin);
    CSA_TRY(check_ws(ws, ws_bytes, out_proj_ws_size(T, H, heads_per_group, d_g)));
    if (T == 0) return CSA_OK;
    const char *names[] = {"o", "w_g", "w_o", "y"};
    const void *ptrs[] = {o, w_g, w_o, y};
    for (int i = 0; i < 4; i++) CSA_TRY(need_ptr(ptrs[i], names[i]));
    cudaStream_t st = (cudaStream_t)stream;
    void *u = (char *)ws + CSA_STATUS_BYTES;
    unsigned *status = (unsigned *)ws;
    CSA_TRY_CUDA(launch_gemm_bf16(T, d_g, (int)kin, G, o, w_g, u, status, DEFAULT_SPIN_LIMIT, st),
                 "out_proj group stage");
    CSA_TRY_CUDA(launch_gemm_bf16(T, d, G * d_g, 1, u, w_o, y, status, DEFAULT_SPIN_LIMIT, st),
                 "out_proj final stage");
    return CSA_OK;
}

// ------------------------------------------------------ incremental decode

size_t decode_tail_bytes(csa_dtype dtype, int64_t B, int32_t c, int32_t dI,
                         const csa_params *params) {
    if (params == nullptr || B < 0 || c < 0 || dI < 0 || params->m < 1) return 0;
    return (size_t)B * decode_tail_slots(params->m, params->overlap) *
           decode_tail_width(c, dI, params->overlap) * esize(dtype);
}

csa_status decode_append(csa_dtype dtype, int64_t B, int32_t c, int32_t dI, const int64_t *t,
                         const void *C, const void *Z, const float *bias, const void *Cb,
                         const void *Zb, const float *biasb, const void *Ck, const void *Zk,
                         const float *biask, const void *Ckb, const void *Zkb,
                         const float *biaskb, void *win, void *tail, void *kvc, void *kIc,
                         int64_t E_cap, const csa_params *params, void *ws, size_t ws_bytes,
                         void *stream) {
    CSA_TRY(check_dtype(dtype));
    const int vec = dtype == CSA_BF16 ? 8 : 4;
    if (c < vec || c % vec != 0 || c / vec > 256)
        return fail(CSA_ERR_UNSUPPORTED, "c=%d must be a multiple of %d, at most %d", c, vec, 256 * vec);
    CSA_TRY(check_params(params, c, false));
    if (params->m > 128) return fail(CSA_ERR_UNSUPPORTED, "m=%d: the tail holds at most 128 slots", params->m);
    if (params->n_win < 0 || params->n_win > 1024) return fail(CSA_ERR_UNSUPPORTED, "n_win=%d not in 0..1024", params->n_win);
    const bool keys = Ck != nullptr;
    if (keys && (dI < vec || dI % vec != 0 || dI / vec > 256))
        return fail(CSA_ERR_UNSUPPORTED, "dI=%d must be a multiple of %d, at most %d", dI, vec, 256 * vec);
    if (!keys) dI = 0;
    if (B < 0 || E_cap < 0) return fail(CSA_ERR_INVALID_ARG, "negative size");
    if (B > 2147483647LL) return fail(CSA_ERR_UNSUPPORTED, "B too large");
    CSA_TRY(check_ws(ws, ws_bytes, CSA_STATUS_BYTES));
    if (B == 0) return CSA_OK;
    const char *names[] = {"t", "C", "Z", "bias", "tail", "kvc"};
    const void *ptrs[] = {t, C, Z, bias, tail, kvc};
    for (int i = 0; i < 6; i++) CSA_TRY(need_ptr(ptrs[i], names[i]));
    if (params->n_win > 0) CSA_TRY(need_ptr(win, "win"));
    if (keys) {
        CSA_TRY(need_ptr(Zk, "Zk"));
        CSA_TRY(need_ptr(biask, "biask"));
        CSA_TRY(need_ptr(kIc, "kIc"));
    }
    if (params->overlap) {
        CSA_TRY(need_ptr(Cb, "Cb"));
        CSA_TRY(need_ptr(Zb, "Zb"));
        CSA_TRY(need_ptr(biasb, "biasb"));
        if (keys) {
            CSA_TRY(need_ptr(Ckb, "Ckb"));
            CSA_TRY(need_ptr(Zkb, "Zkb"));
            CSA_TRY(need_ptr(biaskb, "biaskb"));
        }
    }
    DecodeAppend d;
    d.C = C; d.Z = Z; d.Cb = params->overlap ? Cb : nullptr; d.Zb = params->overlap ? Zb : nullptr;
    d.Ck = keys ? Ck : nullptr; d.Zk = keys ? Zk : nullptr;
    d.Ckb = keys && params->overlap ? Ckb : nullptr; d.Zkb = keys && params->overlap ? Zkb : nullptr;
    d.bias = bias; d.biasb = biasb; d.biask = biask; d.biaskb = biaskb;
    d.t = t; d.win = win; d.tail = tail; d.kvc = kvc; d.kIc = kIc;
    d.status = (unsigned *)ws;
    d.E_cap = E_cap; d.c = c; d.dI = dI; d.m = params->m; d.overlap = params->overlap;
    d.n_win = params->n_win;
    d.kv_norm = params->kv_norm;
    d.norm_eps = params->norm_eps > 0.f ? params->norm_eps : 1e-6f;
    d.rope = make_rope(c, params->rope_dims, params->rope_theta);
    cudaStream_t st = (cudaStream_t)stream;
    StageScope sc(CSA_STAGE_COMPRESS, st);
    CSA_TRY_CUDA(launch_decode_append(dtype, B, d, st), "decode_append launch");
    return CSA_OK;
}

}  // extern "C"
