// Per-query top-k selection: block-level radix select in shared memory.
//
// ["DeepSeek-V4: Making Million-Token Context an Architectural Problem",
// Key design 1, C_t = TopK_k(I[t,:]); DeepSeek-V4 book ch.6 "Top-k is a
// budget over compressed entries": with at most k eligible entries, all are
// kept.]  Ties go to the lower index.
//
// Scores are mapped to order-preserving uint32 keys (-0.0 folded onto +0.0).
// Three histogram passes (11 + 11 + 10 bits) find the exact k-th largest key
// tau and how many keys equal to tau must be taken; one ordered pass then
// emits every index with key > tau plus the first (in index order) keys
// equal to tau, in ascending index order, using block-wide prefix sums.
// Keys are cached in shared memory when the visible prefix fits.
#include "common.cuh"
#include "kernels.h"

namespace csa {

constexpr int TK_THREADS = 512;

// block-wide exclusive prefix sum over TK_THREADS threads; *total gets the sum
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *wsum, uint32_t *total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    constexpr int NW = TK_THREADS / 32;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[wid] = x;
    __syncthreads();
    if (wid == 0) {
        uint32_t s = lane < NW ? wsum[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < NW) wsum[lane] = s;
    }
    __syncthreads();
    uint32_t before = wid > 0 ? wsum[wid - 1] : 0u;
    *total = wsum[NW - 1];
    __syncthreads();
    return before + x - v;
}

__global__ void __launch_bounds__(TK_THREADS)
topk_kernel(const float *__restrict__ scores, const int64_t *__restrict__ q_pos,
            int32_t *__restrict__ idx, int32_t *__restrict__ cnt, int64_t E, int k, int m,
            int kcap) {
    extern __shared__ uint32_t smk[];   // cached keys [kcap]
    __shared__ uint32_t hist[2048];
    __shared__ uint32_t wsum[32];
    __shared__ uint32_t s_bin, s_above;
    const int tid = threadIdx.x;
    const int64_t row = blockIdx.x;
    const int64_t nv = visible_count(q_pos[row], m, E);
    const float *srow = scores + row * E;
    int32_t *orow = idx + row * (int64_t)k;

    if (nv <= k) {
        for (int i = tid; i < k; i += TK_THREADS) orow[i] = i < nv ? i : -1;
        if (tid == 0) cnt[row] = (int32_t)nv;
        return;
    }
    const bool cached = nv <= kcap;
    if (cached) {
        for (int64_t j = tid; j < nv; j += TK_THREADS) smk[j] = score_key(__ldcs(srow + j));
        __syncthreads();
    }
    uint32_t prefix = 0, pmask = 0;
    uint32_t remaining = (uint32_t)k;
#pragma unroll 1
    for (int pass = 0; pass < 3; pass++) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nb = pass < 2 ? 2048 : 1024;
        for (int i = tid; i < nb; i += TK_THREADS) hist[i] = 0;
        __syncthreads();
        for (int64_t j = tid; j < nv; j += TK_THREADS) {
            uint32_t key = cached ? smk[j] : score_key(srow[j]);
            if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
        }
        __syncthreads();
        // thread t owns bins [t*per, (t+1)*per); count of keys above its bins
        const int per = nb / TK_THREADS;
        uint32_t mine = 0;
        for (int i = 0; i < per; i++) mine += hist[tid * per + i];
        // above(t) = sum over threads t' > t of mine(t'): an exclusive prefix
        // sum taken in mirrored thread order, then read back mirrored
        uint32_t tot;
        __shared__ uint32_t mirror[TK_THREADS];
        mirror[TK_THREADS - 1 - tid] = mine;
        __syncthreads();
        uint32_t mv = mirror[tid];
        uint32_t ex = block_excl_scan(mv, wsum, &tot);
        mirror[tid] = ex;           // = above-count of thread TK_THREADS-1-tid
        __syncthreads();
        uint32_t above = mirror[TK_THREADS - 1 - tid];
        __syncthreads();
        for (int i = per - 1; i >= 0; i--) {
            const int bin = tid * per + i;
            const uint32_t h = hist[bin];
            if (above < remaining && above + h >= remaining) {
                s_bin = (uint32_t)bin;
                s_above = above;
            }
            above += h;
        }
        __syncthreads();
        remaining -= s_above;
        prefix |= s_bin << shift;
        pmask |= (uint32_t)(nb - 1) << shift;
        __syncthreads();
    }
    const uint32_t tau = prefix;
    const uint32_t need_eq = remaining;
    uint32_t run_sel = 0, run_eq = 0;
    for (int64_t base = 0; base < nv && run_sel < (uint32_t)k; base += TK_THREADS) {
        const int64_t j = base + tid;
        const uint32_t key = j < nv ? (cached ? smk[j] : score_key(srow[j])) : 0u;
        const uint32_t gt = (j < nv && key > tau) ? 1u : 0u;
        const uint32_t eq = (j < nv && key == tau) ? 1u : 0u;
        uint32_t eq_tot, sel_tot;
        const uint32_t eq_rank = run_eq + block_excl_scan(eq, wsum, &eq_tot);
        const uint32_t sel = (gt || (eq && eq_rank < need_eq)) ? 1u : 0u;
        const uint32_t pos = run_sel + block_excl_scan(sel, wsum, &sel_tot);
        if (sel && pos < (uint32_t)k) orow[pos] = (int32_t)j;
        run_eq += eq_tot;
        run_sel += sel_tot;
    }
    if (tid == 0) cnt[row] = k;
}

static int g_topk_smem_set = 0;

cudaError_t launch_topk(int64_t B, int64_t Tq, int64_t E, int k, int m, const float *scores,
                        const int64_t *q_pos, int32_t *idx, int32_t *cnt, cudaStream_t st) {
    if (B * Tq == 0) return cudaSuccess;
    const int kcap_max = 40960;   // 160 KB of cached keys
    int kcap = (int)(E < kcap_max ? E : kcap_max);
    size_t smem = (size_t)kcap * 4;
    if (!g_topk_smem_set) {
        cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kcap_max * 4);
        if (e != cudaSuccess) return e;
        g_topk_smem_set = 1;
    }
    topk_kernel<<<(unsigned)(B * Tq), TK_THREADS, smem, st>>>(scores, q_pos, idx, cnt, E, k, m, kcap);
    return cudaGetLastError();
}

}  // namespace csa
