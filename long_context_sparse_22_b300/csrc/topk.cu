// Per-query top-k selection: radix select on order-preserving score keys.
//
// ["DeepSeek-V4: Making Million-Token Context an Architectural Problem",
// Key design 1, C_t = TopK_k(I[t,:]); DeepSeek-V4 book ch.6 "Top-k is a
// budget over compressed entries": with at most k eligible entries, all are
// kept.]  Ties go to the lower index.
//
// Scores map to uint32 keys that order like the floats (-0.0 folded onto
// +0.0).  The exact selection: three histogram passes (11 + 11 + 10 bits)
// find the k-th largest key tau and how many keys equal to tau must be taken;
// one ordered pass then emits every index with key > tau plus the first keys
// equal to tau, in ascending index order, using block-wide prefix sums.
//
// Most of a row cannot reach the top k, so the exact selection runs on a
// short candidate list: an evenly spaced sample of the row gives a key lo that
// lies below the k-th largest with a margin of five standard deviations; the
// keys >= lo are compacted in index order and the exact selection runs on
// them.  If fewer than k keys reach lo (or too many to hold), the exact
// selection runs on the whole row instead, so the result never depends on the
// sample.
//
// Many rows (prefill): one warp per row.
// Few long rows (decode, up to 262144 entries): one launch, a cluster of eight
// CTAs per row, the row's keys in their registers; each CTA derives the row's
// sampled bound and keeps its keys >= lo in index order in shared memory, and
// the cluster's first CTA reads all of them through distributed shared memory
// and runs the exact selection.  Longer rows: two launches, (1) the row's
// chunks spread over many CTAs, each keeping its keys >= lo in global memory,
// (2) one CTA per row running the exact selection on the candidates.
#include <mutex>

#include <cooperative_groups.h>

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

struct TkShared {
    uint32_t hist[2048];
    uint32_t wsum[32];
    uint32_t mirror[TK_THREADS];
    uint32_t wcnt[2][TK_THREADS / 32];
    uint32_t bin, above, binsz;
};

// Add one to hist[bin] for every lane with `in` set; lanes of a warp that
// hit the same bin are merged into one shared-memory atomic (scores crowd
// into a few bins, so plain per-lane atomics serialise).  Warp-uniform call.
__device__ __forceinline__ void hist_add(uint32_t *hist, bool in, uint32_t bin) {
    const unsigned m_in = __ballot_sync(0xffffffffu, in);
    if (in) {
        const unsigned peers = __match_any_sync(m_in, bin);
        if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
    }
}

// Exclusive prefix over the block of per-warp counts c (lane 0 of each warp
// supplies its warp's count); returns the sum over earlier warps and sets
// *total.  Two barriers.
__device__ __forceinline__ uint32_t warp_offsets(uint32_t *wc, uint32_t c, uint32_t *total) {
    const int wid = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) wc[wid] = c;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < TK_THREADS / 32; w++) {
        const uint32_t v = wc[w];
        before += w < wid ? v : 0u;
        tot += v;
    }
    *total = tot;
    __syncthreads();
    return before;
}

// Given a histogram of nb bins (nb a multiple of TK_THREADS), find the bin
// holding the remaining-th largest key counting down from the top bin; sets
// sh.bin and sh.above (the count in the bins above it).  All threads call.
__device__ __forceinline__ void find_bin(TkShared &sh, int nb, uint32_t remaining) {
    const int tid = threadIdx.x;
    const int per = nb / TK_THREADS;
    uint32_t mine = 0;
    for (int i = 0; i < per; i++) mine += sh.hist[tid * per + i];
    // above(t) = sum over threads t' > t: an exclusive prefix sum taken in
    // mirrored thread order, then read back mirrored
    sh.mirror[TK_THREADS - 1 - tid] = mine;
    __syncthreads();
    uint32_t tot;
    const uint32_t ex = block_excl_scan(sh.mirror[tid], sh.wsum, &tot);
    sh.mirror[tid] = ex;
    __syncthreads();
    uint32_t above = sh.mirror[TK_THREADS - 1 - tid];
    __syncthreads();
    for (int i = per - 1; i >= 0; i--) {
        const int bin = tid * per + i;
        const uint32_t h = sh.hist[bin];
        if (above < remaining && above + h >= remaining) {
            sh.bin = (uint32_t)bin;
            sh.above = above;
            sh.binsz = h;
        }
        above += h;
    }
    __syncthreads();
}

// The k-th largest key tau of n > k items, how many items equal to tau the
// selection takes (need_eq), and whether that is all of them.
struct Thr {
    uint32_t tau, need_eq;
    bool all_eq;
};

template <typename KeyF>
__device__ Thr find_threshold(TkShared &sh, int64_t n, int k, KeyF key) {
    const int tid = threadIdx.x;
    uint32_t prefix = 0, pmask = 0;
    uint32_t remaining = (uint32_t)k;
    uint32_t n_eq = 0;
#pragma unroll 1
    for (int pass = 0; pass < 3; pass++) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nb = pass < 2 ? 2048 : 1024;
        for (int i = tid; i < nb; i += TK_THREADS) sh.hist[i] = 0;
        __syncthreads();
        for (int64_t base = 0; base < n; base += TK_THREADS) {
            const int64_t j = base + tid;
            const uint32_t kv = j < n ? key(j) : 0u;
            hist_add(sh.hist, j < n && (kv & pmask) == prefix, (kv >> shift) & (nb - 1));
        }
        __syncthreads();
        find_bin(sh, nb, remaining);
        remaining -= sh.above;
        prefix |= sh.bin << shift;
        pmask |= (uint32_t)(nb - 1) << shift;
        n_eq = sh.binsz;                 // after the last pass: keys equal to tau
        __syncthreads();
    }
    Thr t;
    t.tau = prefix;
    t.need_eq = remaining;
    t.all_eq = remaining == n_eq;        // every tie is kept: selection is key >= tau
    return t;
}

// Writes, in the items' order, the id of every item with key > tau and of the
// first need_eq items with key == tau (k in all) to orow.
template <typename KeyF, typename IdF>
__device__ void emit_ordered(TkShared &sh, int64_t n, int k, const Thr &th, KeyF key, IdF id,
                             int32_t *orow) {
    const int tid = threadIdx.x, lane = tid & 31;
    const unsigned lt = (1u << lane) - 1u;
    uint32_t run_sel = 0, run_eq = 0;
    for (int64_t base = 0; base < n && run_sel < (uint32_t)k; base += TK_THREADS) {
        const int64_t j = base + tid;
        const uint32_t kv = j < n ? key(j) : 0u;
        const bool gt = j < n && kv > th.tau;
        const bool eq = j < n && kv == th.tau;
        bool sel;
        if (th.all_eq) {
            sel = gt || eq;
        } else {
            const unsigned be = __ballot_sync(0xffffffffu, eq);
            uint32_t eq_tot;
            const uint32_t eq_before = warp_offsets(sh.wcnt[0], (uint32_t)__popc(be), &eq_tot);
            const uint32_t eq_rank = run_eq + eq_before + (uint32_t)__popc(be & lt);
            sel = gt || (eq && eq_rank < th.need_eq);
            run_eq += eq_tot;
        }
        const unsigned bs = __ballot_sync(0xffffffffu, sel);
        uint32_t sel_tot;
        const uint32_t pos = run_sel + warp_offsets(sh.wcnt[1], (uint32_t)__popc(bs), &sel_tot) +
                             (uint32_t)__popc(bs & lt);
        if (sel && pos < (uint32_t)k) orow[pos] = id(j);
        run_sel += sel_tot;
    }
}

// Exact top-k over n > k items given in index order: key(i) is the item's
// uint32 key, id(i) its output index.  Writes the k kept indices to orow in
// the items' order.
template <typename KeyF, typename IdF>
__device__ void select_core(TkShared &sh, int64_t n, int k, KeyF key, IdF id, int32_t *orow) {
    const Thr th = find_threshold(sh, n, k, key);
    emit_ordered(sh, n, k, th, key, id, orow);
}

// Rank in a sample of S keys (drawn from n) whose key lower-bounds the k-th
// largest of all n with a margin of five standard deviations of the number of
// sample keys above it; >= S means "no useful bound".  In fp32 (B300's fp64
// pipe is narrow, and every thread of a block evaluates this): the rank only
// sets how far below the k-th largest key the bound falls, and any rank
// leaves the selection exact.
__device__ __forceinline__ int sample_rank(int64_t n, int k, int S) {
    const float nf = n > 0x7fffffffLL ? 2147483648.0f : (float)(int)n;
    const float p = (float)k / nf;
    const float mu = (float)S * p;
    const float sd = sqrtf(mu * (1.0f - p));
    return (int)ceilf(mu + 5.0f * sd + 2.0f);
}

// ----------------------------------------------------------- one CTA per row

// ----------------------------------------------- one warp per row (prefill)
//
// Each warp selects for its own rows with warp-level synchronisation only:
// the exact threshold is a radix select with 8-bit digits (four passes) on
// a per-warp 256-bin histogram; the bin holding the remaining-th largest key
// is found by a suffix sum across the lanes, each lane owning eight bins.

constexpr int TW_WARPS = 16;                  // warps per CTA
constexpr int TW_SAMPLE = 512;                // sampled keys per row
constexpr int TW_LCAP = 2048;                 // candidates kept per warp

struct TwShared {
    uint32_t hist[256];                       // histogram of the exact whole-row fallback
    uint32_t lkey[TW_LCAP];                   // candidates, in index order
    uint16_t lidx[TW_LCAP];                   // their positions (rows of at most 65536 entries)
};

// hist[bin] += 1 for every lane with `in`, lanes of the same bin merged.
__device__ __forceinline__ void warp_hist_add(uint32_t *hist, bool in, uint32_t bin) {
    const unsigned m_in = __ballot_sync(0xffffffffu, in);
    if (in) {
        const unsigned peers = __match_any_sync(m_in, bin);
        if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
    }
    __syncwarp();
}

// The k-th largest of n keys, exact: radix select with digits of at most 8
// bits, run only over the bits in which the keys differ (bits they all share
// are found first by a warp-wide AND / OR and taken as given).
template <typename KeyF>
__device__ Thr warp_threshold(uint32_t *hist, int64_t n, int k, KeyF key) {
    const int lane = threadIdx.x & 31;
    uint32_t all1 = 0xffffffffu, any1 = 0u;
    for (int64_t j = lane; j < n; j += 32) {
        const uint32_t kv = key(j);
        all1 &= kv;
        any1 |= kv;
    }
    all1 = __reduce_and_sync(0xffffffffu, all1);
    any1 = __reduce_or_sync(0xffffffffu, any1);
    const uint32_t vary = all1 ^ any1;
    uint32_t prefix = all1 & ~vary, pmask = ~vary, remaining = (uint32_t)k;
    uint32_t n_eq = (uint32_t)n;
    int hi = vary ? 31 - __clz(vary) : -1;
#pragma unroll 1
    while (hi >= 0) {
        const int lo_bit = hi >= 7 ? hi - 7 : 0;
        const uint32_t dmask = (2u << (hi - lo_bit)) - 1u;     // digit of hi - lo_bit + 1 bits
#pragma unroll
        for (int i = 0; i < 8; i++) hist[lane * 8 + i] = 0u;
        __syncwarp();
        for (int64_t base = 0; base < n; base += 32) {
            const int64_t j = base + lane;
            const uint32_t kv = j < n ? key(j) : 0u;
            warp_hist_add(hist, j < n && (kv & pmask) == prefix, (kv >> lo_bit) & dmask);
        }
        uint32_t h[8], c = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            h[i] = hist[lane * 8 + i];
            c += h[i];
        }
        // suffix sum over lanes: keys in bins above this lane's eight
        uint32_t sfx = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_down_sync(0xffffffffu, sfx, o);
            if (lane + o < 32) sfx += t;
        }
        uint32_t above = sfx - c;
        int found = -1;
        uint32_t f_above = 0, f_size = 0;
#pragma unroll
        for (int i = 7; i >= 0; i--) {
            if (found < 0 && above < remaining && above + h[i] >= remaining) {
                found = lane * 8 + i;
                f_above = above;
                f_size = h[i];
            }
            above += h[i];
        }
        const unsigned who = __ballot_sync(0xffffffffu, found >= 0);
        const int src = __ffs(who) - 1;
        const uint32_t bin = (uint32_t)__shfl_sync(0xffffffffu, found, src);
        remaining -= __shfl_sync(0xffffffffu, f_above, src);
        n_eq = __shfl_sync(0xffffffffu, f_size, src);
        prefix |= bin << lo_bit;
        pmask |= dmask << lo_bit;
        __syncwarp();
        hi = lo_bit - 1;
    }
    Thr t;
    t.tau = prefix;
    t.need_eq = remaining;
    t.all_eq = remaining == n_eq;
    return t;
}

template <typename KeyF, typename IdF>
__device__ void warp_emit(int64_t n, int k, const Thr &th, KeyF key, IdF id, int32_t *orow) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    uint32_t run_sel = 0, run_eq = 0;
    for (int64_t base = 0; base < n && run_sel < (uint32_t)k; base += 32) {
        const int64_t j = base + lane;
        const uint32_t kv = j < n ? key(j) : 0u;
        const bool gt = j < n && kv > th.tau;
        const bool eq = j < n && kv == th.tau;
        const unsigned be = __ballot_sync(0xffffffffu, eq);
        const bool sel = gt || (eq && (th.all_eq || run_eq + (uint32_t)__popc(be & lt) < th.need_eq));
        run_eq += (uint32_t)__popc(be);
        const unsigned bs = __ballot_sync(0xffffffffu, sel);
        const uint32_t pos = run_sel + (uint32_t)__popc(bs & lt);
        if (sel && pos < (uint32_t)k) orow[pos] = id(j);
        run_sel += (uint32_t)__popc(bs);
    }
}

// Keys of the lane's NK registers that are >= t, summed over the warp
// (padding holds key 0, which no t >= 1 counts).
template <int NK>
__device__ __forceinline__ uint32_t warp_count_ge(const uint32_t (&kr)[NK], uint32_t t) {
    uint32_t c = 0;
#pragma unroll
    for (int i = 0; i < NK; i++) c += kr[i] >= t ? 1u : 0u;
    return __reduce_add_sync(0xffffffffu, c);
}

// The largest t whose low (32 - bits) bits are zero and that at least k keys
// reach: with bits = 32, the k-th largest key; with fewer bits, a lower bound
// on it.  One bit per step, decided by a count.
template <int NK>
__device__ __forceinline__ uint32_t warp_kth(const uint32_t (&kr)[NK], int k, int bits) {
    uint32_t t = 0;
#pragma unroll 1
    for (int b = 31; b >= 32 - bits; b--) {
        const uint32_t c = t | (1u << b);
        if (warp_count_ge(kr, c) >= (uint32_t)k) t = c;
    }
    return t;
}

__global__ void __launch_bounds__(TW_WARPS * 32, 1)
topk_kernel(const float *__restrict__ scores, const int64_t *__restrict__ q_pos,
            int32_t *__restrict__ idx, int32_t *__restrict__ cnt, int64_t rows, int64_t E, int k,
            int m) {
    extern __shared__ __align__(16) uint8_t tw_raw[];
    TwShared &sh = reinterpret_cast<TwShared *>(tw_raw)[threadIdx.x >> 5];
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    const int64_t nwarps = (int64_t)gridDim.x * TW_WARPS;
    for (int64_t row = (int64_t)blockIdx.x * TW_WARPS + (threadIdx.x >> 5); row < rows; row += nwarps) {
        const int64_t nv = visible_count(q_pos[row], m, E);
        const float *srow = scores + row * E;
        int32_t *orow = idx + row * (int64_t)k;
        if (nv <= k) {
            for (int i = lane; i < k; i += 32) orow[i] = i < nv ? i : -1;
            if (lane == 0) cnt[row] = (int32_t)nv;
            continue;
        }
        auto gkey = [&](int64_t j) { return score_key(__ldg(srow + j)); };
        auto gid = [](int64_t j) { return (int32_t)j; };
        bool done = false;
        const bool whole = nv <= TW_SAMPLE;                 // the row itself is the sample
        const int r = whole ? k : sample_rank(nv, k, TW_SAMPLE);
        if ((whole || r < TW_SAMPLE) && 2 * k <= TW_LCAP && nv <= 65536) {
            // sample keys (or the whole row) in registers: sk[u] is sample 32u + lane, taken at
            // position (i * nv) / TW_SAMPLE (exact in 32 bits for rows of at most 65536)
            uint32_t sk[TW_SAMPLE / 32];
#pragma unroll
            for (int u = 0; u < TW_SAMPLE / 32; u++) {
                const uint32_t i = 32 * u + lane;
                if (whole) sk[u] = i < nv ? score_key(__ldcs(srow + i)) : 0u;
                else sk[u] = gkey((int64_t)((i * (uint32_t)nv) / TW_SAMPLE));
            }
            // lo: the top 24 bits of the r-th largest sample key, a lower bound on the k-th largest key
            const uint32_t lo = warp_kth(sk, r, 24);
            // the keys >= lo, in index order, 64 loads in flight per lane
            uint32_t n = 0;
            if (whole) {
#pragma unroll
                for (int u = 0; u < TW_SAMPLE / 32; u++) {
                    const int j = 32 * u + lane;
                    const bool in = j < nv && sk[u] >= lo;
                    const unsigned bm = __ballot_sync(0xffffffffu, in);
                    const uint32_t p = n + (uint32_t)__popc(bm & lt);
                    if (in) {
                        sh.lkey[p] = sk[u];
                        sh.lidx[p] = (uint16_t)j;
                    }
                    n += (uint32_t)__popc(bm);
                }
            } else {
                constexpr int NB = 64;
                for (int64_t base = 0; base < nv && n <= (uint32_t)TW_LCAP; base += 32 * NB) {
                    uint32_t kv[NB];
#pragma unroll
                    for (int u = 0; u < NB; u++) {
                        const int64_t j = base + 32 * u + lane;
                        kv[u] = j < nv ? score_key(__ldcs(srow + j)) : 0u;
                    }
#pragma unroll
                    for (int u = 0; u < NB; u++) {
                        const int64_t j = base + 32 * u + lane;
                        const bool in = j < nv && kv[u] >= lo;
                        const unsigned bm = __ballot_sync(0xffffffffu, in);
                        const uint32_t p = n + (uint32_t)__popc(bm & lt);
                        if (in && p < (uint32_t)TW_LCAP) {
                            sh.lkey[p] = kv[u];
                            sh.lidx[p] = (uint16_t)j;
                        }
                        n += (uint32_t)__popc(bm);
                    }
                }
            }
            __syncwarp();
            if (n <= (uint32_t)TW_LCAP && n >= (uint32_t)k) {
                auto ckey = [&](int64_t j) { return sh.lkey[j]; };
                const Thr th = warp_threshold(sh.hist, n, k, ckey);
                warp_emit(n, k, th, ckey, [&](int64_t j) { return (int32_t)sh.lidx[j]; }, orow);
                done = true;
            }
        }
        if (!done) {
            // exact over the whole row, from global memory
            const Thr th = warp_threshold(sh.hist, nv, k, gkey);
            warp_emit(nv, k, th, gkey, gid, orow);
        }
        if (lane == 0) cnt[row] = k;
        __syncwarp();
    }
}

// ------------------------------------------------------- few long rows (decode)

struct TkLong {
    const float *scores;
    const int64_t *q_pos;
    uint32_t *chunk_cnt;   // [rows][CH]
    uint32_t *cand_key;    // [rows][E]: chunk c's candidates at [c*CS, ...)
    int32_t *cand_idx;     // [rows][E]
    int32_t *idx;          // [rows][k]
    int32_t *cnt;          // [rows]
    int64_t E, CS;         // CS: chunk size
    int CH, k, m;
};

constexpr int TK_LSAMPLE = 1024;              // sample keys per long row (32 per lane of warp 0)
constexpr int TK_SEG = 256;                   // candidates a warp keeps per chunk

// The k-th largest of the valid keys held in registers by the block's
// TK_THREADS threads (the first nk[t] of thread t's NK keys are valid):
// radix select with digits of at most 8 bits, over the bits in which the
// keys differ only; three barriers per digit.
template <int NK>
__device__ Thr block_threshold(const uint32_t (&kr)[NK], int nk, int k, uint32_t *hist, uint32_t *red) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    constexpr int NW = TK_THREADS / 32;
    uint32_t a1 = 0xffffffffu, o1 = 0u;
#pragma unroll
    for (int i = 0; i < NK; i++)
        if (i < nk) {
            a1 &= kr[i];
            o1 |= kr[i];
        }
    a1 = __reduce_and_sync(0xffffffffu, a1);
    o1 = __reduce_or_sync(0xffffffffu, o1);
    if (lane == 0) {
        red[wid] = a1;
        red[NW + wid] = o1;
    }
    __syncthreads();
    a1 = 0xffffffffu;
    o1 = 0u;
#pragma unroll
    for (int w = 0; w < NW; w++) {
        a1 &= red[w];
        o1 |= red[NW + w];
    }
    const uint32_t vary = a1 ^ o1;
    uint32_t prefix = a1 & ~vary, pmask = ~vary, remaining = (uint32_t)k, n_eq = 0;
    int hi = vary ? 31 - __clz(vary) : -1;
    if (hi < 0) {
        // all keys equal: count them
        uint32_t c = 0;
#pragma unroll
        for (int i = 0; i < NK; i++) c += i < nk ? 1u : 0u;
        c = __reduce_add_sync(0xffffffffu, c);
        __syncthreads();
        if (lane == 0) red[wid] = c;
        __syncthreads();
        for (int w = 0; w < NW; w++) n_eq += red[w];
    }
#pragma unroll 1
    while (hi >= 0) {
        const int lo_bit = hi >= 7 ? hi - 7 : 0;
        const uint32_t dmask = (2u << (hi - lo_bit)) - 1u;
        if (tid < 256) hist[tid] = 0u;
        __syncthreads();
#pragma unroll
        for (int i = 0; i < NK; i++) {
            const bool in = i < nk && (kr[i] & pmask) == prefix;
            const uint32_t bin = (kr[i] >> lo_bit) & dmask;
            const unsigned m_in = __ballot_sync(0xffffffffu, in);
            if (in) {
                const unsigned peers = __match_any_sync(m_in, bin);
                if (lane == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
            }
        }
        __syncthreads();
        if (wid == 0) {
            uint32_t h[8], c = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                h[i] = hist[lane * 8 + i];
                c += h[i];
            }
            uint32_t sfx = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_down_sync(0xffffffffu, sfx, o);
                if (lane + o < 32) sfx += t;
            }
            uint32_t above = sfx - c;
#pragma unroll
            for (int i = 7; i >= 0; i--) {
                if (above < remaining && above + h[i] >= remaining) {
                    red[2 * NW] = (uint32_t)(lane * 8 + i);
                    red[2 * NW + 1] = above;
                    red[2 * NW + 2] = h[i];
                }
                above += h[i];
            }
        }
        __syncthreads();
        prefix |= red[2 * NW] << lo_bit;
        remaining -= red[2 * NW + 1];
        n_eq = red[2 * NW + 2];
        pmask |= dmask << lo_bit;
        hi = lo_bit - 1;
    }
    __syncthreads();
    Thr t;
    t.tau = prefix;
    t.need_eq = remaining;
    t.all_eq = remaining == n_eq;
    return t;
}

// The k largest of n > k candidates held in registers, thread t holding
// candidates PT t .. PT t + PT - 1 in index order (nk of them valid), written
// to orow in index order; id(u) gives the index of this thread's candidate u.
// The threshold from block_threshold, then one block scan of the per-thread
// counts of keys above it and of ties places every kept index.
// Writes, in index order, the id of every key above tau and of the first
// need_eq keys equal to tau, from keys held in registers (thread t holds
// keys PT t .. PT t + PT - 1, nk of them valid): one block scan of the
// per-thread counts of keys above tau and of ties places every kept index.
template <int PT, typename IdF>
__device__ void emit_registers(const uint32_t (&ck)[PT], int nk, uint32_t t, uint32_t need_eq, IdF id,
                               uint32_t *wsum, int32_t *orow) {
    uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
    for (int u = 0; u < PT; u++) {
        n_gt += ck[u] > t && u < nk ? 1u : 0u;
        n_eq += ck[u] == t && u < nk ? 1u : 0u;
    }
    uint32_t tot2;
    const uint32_t ex2 = block_excl_scan((n_eq << 16) | n_gt, wsum, &tot2);
    uint32_t eq_before = ex2 >> 16, gt_before = ex2 & 0xffffu;
    uint32_t pos = gt_before + (eq_before < need_eq ? eq_before : need_eq);
#pragma unroll
    for (int u = 0; u < PT; u++) {
        bool sel = false;
        if (u < nk) {
            if (ck[u] > t) sel = true;
            else if (ck[u] == t) sel = eq_before++ < need_eq;
        }
        if (sel) orow[pos++] = id(u);
    }
}

// The k largest of n > k candidates held in registers (see emit_registers
// for the layout), written to orow in index order.
template <int PT, typename IdF>
__device__ void select_registers(const uint32_t (&ck)[PT], int nk, int k, IdF id, uint32_t *hist,
                                 uint32_t *red, uint32_t *wsum, int32_t *orow) {
    const Thr th = block_threshold(ck, nk, k, hist, red);
    emit_registers(ck, nk, th.tau, th.need_eq, id, wsum, orow);
}

// (1) per chunk of a long row: the row's sampled bound lo (every chunk CTA
// derives the same value from the same evenly spaced sample), then the
// chunk's keys >= lo in index order.  Each warp compacts its own contiguous
// slice into a shared-memory segment; one scan of the warp counts places the
// segments.  chunk_cnt gets the chunk's count, or ~0u if a segment overflowed.
__global__ void __launch_bounds__(TK_THREADS) topk_collect_kernel(TkLong a) {
    __shared__ uint32_t wcount[TK_THREADS / 32];
    __shared__ uint32_t skey[TK_THREADS / 32][TK_SEG];
    __shared__ int32_t sidx[TK_THREADS / 32][TK_SEG];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t row = blockIdx.y;
    const int64_t nv = visible_count(a.q_pos[row], a.m, a.E);
    if (nv <= a.k) return;
    const float *s = a.scores + row * a.E;
    // the bound: top 24 bits of the r-th largest of TK_LSAMPLE evenly spaced
    // keys, found by warp 0 alone (32 keys per lane, bit by bit)
    __shared__ uint32_t lo_s;
    if (wid == 0) {
        const int S = (int)(nv < TK_LSAMPLE ? nv : TK_LSAMPLE);
        uint32_t sk[TK_LSAMPLE / 32];
#pragma unroll
        for (int u = 0; u < TK_LSAMPLE / 32; u++) {
            const int i = 32 * u + lane;
            const int64_t pos = S == TK_LSAMPLE ? (((int64_t)i * nv) >> 10) : i;   // TK_LSAMPLE = 2^10
            sk[u] = i < S ? score_key(s[pos]) : 0u;
        }
        const int r = S < TK_LSAMPLE ? a.k : sample_rank(nv, a.k, S);
        const uint32_t lo = r < S ? warp_kth(sk, r, 24) : 0u;
        if (lane == 0) lo_s = lo;
    }
    // this warp's slice of the chunk; its first keys are loaded before the
    // bound is known, so the loads overlap warp 0's work
    const int64_t c0 = (int64_t)blockIdx.x * a.CS;
    const int64_t c1 = c0 + a.CS < nv ? c0 + a.CS : nv;
    const int64_t per = (c1 - c0 + TK_THREADS / 32 - 1) / (TK_THREADS / 32);
    const int64_t w0 = c0 + wid * per;
    const int64_t w1 = w0 + per < c1 ? w0 + per : c1;
    const unsigned lt = (1u << lane) - 1u;
    constexpr int NB = 16;
    uint32_t kv[NB];
#pragma unroll
    for (int u = 0; u < NB; u++) {
        const int64_t j = w0 + 32 * u + lane;
        kv[u] = j < w1 ? score_key(__ldcs(s + j)) : 0u;
    }
    __syncthreads();
    const uint32_t lo = lo_s;
    uint32_t n = 0;
    for (int64_t base = w0; base < w1; base += 32 * NB) {
        if (base != w0) {
#pragma unroll
            for (int u = 0; u < NB; u++) {
                const int64_t j = base + 32 * u + lane;
                kv[u] = j < w1 ? score_key(__ldcs(s + j)) : 0u;
            }
        }
#pragma unroll
        for (int u = 0; u < NB; u++) {
            const int64_t j = base + 32 * u + lane;
            const bool in = j < w1 && kv[u] >= lo;
            const unsigned bm = __ballot_sync(0xffffffffu, in);
            const uint32_t p = n + (uint32_t)__popc(bm & lt);
            if (in && p < (uint32_t)TK_SEG) {
                skey[wid][p] = kv[u];
                sidx[wid][p] = (int32_t)j;
            }
            n += (uint32_t)__popc(bm);
        }
    }
    if (lane == 0) wcount[wid] = n;
    __syncthreads();
    uint32_t before = 0, tot = 0;
    bool over = false;
#pragma unroll
    for (int w = 0; w < TK_THREADS / 32; w++) {
        const uint32_t v = wcount[w];
        before += w < wid ? v : 0u;
        tot += v;
        over |= v > (uint32_t)TK_SEG;
    }
    if (!over) {
        uint32_t *ok = a.cand_key + row * a.E + c0 + before;
        int32_t *oi = a.cand_idx + row * a.E + c0 + before;
        for (uint32_t i = lane; i < n; i += 32) {
            ok[i] = skey[wid][i];
            oi[i] = sidx[wid][i];
        }
    }
    if (tid == 0) a.chunk_cnt[row * a.CH + blockIdx.x] = over ? 0xffffffffu : tot;
}

__global__ void __launch_bounds__(TK_THREADS) topk_final_kernel(TkLong a, int cap) {
    extern __shared__ uint32_t smc[];   // [cap] keys, then [cap] indices
    __shared__ TkShared sh;
    __shared__ uint32_t offs[257];
    const int tid = threadIdx.x;
    const int64_t row = blockIdx.x;
    const int64_t nv = visible_count(a.q_pos[row], a.m, a.E);
    int32_t *orow = a.idx + row * (int64_t)a.k;
    if (nv <= a.k) {
        for (int i = tid; i < a.k; i += TK_THREADS) orow[i] = i < nv ? i : -1;
        if (tid == 0) a.cnt[row] = (int32_t)nv;
        return;
    }
    // chunk offsets: one block scan of the chunk counts (CH <= TK_THREADS)
    const uint32_t mine = tid < a.CH ? a.chunk_cnt[row * a.CH + tid] : 0u;
    const bool bad = __syncthreads_or(mine == 0xffffffffu);
    uint32_t tot_all;
    const uint32_t ex = block_excl_scan(bad ? 0u : mine, sh.wsum, &tot_all);
    if (tid <= a.CH && tid < 257) offs[tid] = ex;
    __syncthreads();
    const int64_t n = bad ? -1 : (int64_t)tot_all;
    const uint32_t *gk = a.cand_key + row * a.E;
    const int32_t *gi = a.cand_idx + row * a.E;
    if (n < a.k) {
        // the sampled bound missed (fewer than k keys reach it, or a warp's
        // segment overflowed): exact over the row
        const float *s = a.scores + row * a.E;
        select_core(sh, nv, a.k, [&](int64_t j) { return score_key(s[j]); },
                    [](int64_t j) { return (int32_t)j; }, orow);
    } else if (n <= cap) {
        // the chunks' candidates, in index order, packed into shared memory;
        // every thread locates its items' chunks by binary search so all the
        // loads are in flight together
        int32_t *si = (int32_t *)(smc + cap);
        // four items per thread per round: their sources first, then all eight
        // loads in flight together, then the stores
        for (int64_t j0 = tid; j0 < n; j0 += 4 * TK_THREADS) {
            int64_t src[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int64_t j = j0 + (int64_t)u * TK_THREADS;
                int lo = 0, hi = a.CH - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if ((int64_t)offs[mid] <= j) lo = mid; else hi = mid - 1;
                }
                src[u] = j < n ? lo * a.CS + (j - offs[lo]) : -1;
            }
            uint32_t kv[4];
            int32_t iv[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                kv[u] = src[u] >= 0 ? gk[src[u]] : 0u;
                iv[u] = src[u] >= 0 ? gi[src[u]] : 0;
            }
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int64_t j = j0 + (int64_t)u * TK_THREADS;
                if (j < n) {
                    smc[j] = kv[u];
                    si[j] = iv[u];
                }
            }
        }
        __syncthreads();
        constexpr int PT = 16;                 // candidates per thread in registers
        if (n <= PT * TK_THREADS) {
            // exact k-th largest over the candidates in registers, thread t
            // holding candidates PT t .. PT t + PT-1 (index order)
            uint32_t ck[PT];
#pragma unroll
            for (int u = 0; u < PT; u++) {
                const int64_t j = (int64_t)tid * PT + u;
                ck[u] = j < n ? smc[j] : 0u;
            }
            __shared__ uint32_t red[40];
            __shared__ uint32_t hist[256];
            const int64_t left = n - (int64_t)tid * PT;
            const int nk = (int)(left < 0 ? 0 : (left > PT ? PT : left));
            select_registers(ck, nk, a.k, [&](int u) { return si[(int64_t)tid * PT + u]; }, hist, red,
                             sh.wsum, orow);
        } else {
            select_core(sh, n, a.k, [&](int64_t j) { return smc[j]; }, [&](int64_t j) { return si[j]; },
                        orow);
        }
    } else {
        // many candidates (heavy ties): read them in place, chunk by chunk
        auto where = [&](int64_t j) {
            int c = 0;
            while (c + 1 < a.CH && (int64_t)offs[c + 1] <= j) c++;
            return c * a.CS + (j - offs[c]);
        };
        select_core(sh, n, a.k, [&](int64_t j) { return gk[where(j)]; },
                    [&](int64_t j) { return gi[where(j)]; }, orow);
    }
    if (tid == 0) a.cnt[row] = a.k;
}

// Few long rows, one launch: a cluster of TC_CL CTAs per row.  CTA r of the
// cluster holds the keys of the r-th slice of the row in registers (the
// slices cut E, so the loads start before the position is known).  Within a
// CTA, warp w owns a contiguous part of the slice, and lane l holds, for each
// step u, the four keys at u * 128 + 4 l .. + 3 of it (each warp load reads
// 512 contiguous bytes).  Every CTA derives the same sampled bound lo from the
// same evenly spaced sample and writes its keys >= lo, in index order, into
// its own region of the first CTA's shared memory.  After one cluster barrier
// the other CTAs leave; the first CTA loads the candidates (regions in rank
// order, so index order) into registers, thread t holding a contiguous run,
// and runs the exact selection.  If the sample misses (fewer than k
// candidates) or a region overflows, it runs the exact selection over the
// whole row from global memory instead.
constexpr int TC_CL = 8;              // CTAs per row
constexpr int TC_CAPR = 1024;         // candidates a CTA may keep
constexpr int TC_RSTRIDE = TC_CAPR + TC_CAPR / 8;    // a region: four pad words after every 32
constexpr int TC_PT = 16;             // candidates per thread in the first CTA's selection
constexpr int TC_SMEM = TC_CL * TC_RSTRIDE * 8;
constexpr int TC_WARPS = TK_THREADS / 32;

struct TcShared {
    uint32_t hist[2][2048];           // radix histograms, one being counted while the other is cleared
    uint32_t wtot[TC_WARPS];
    uint32_t wand[TC_WARPS], wor[TC_WARPS];
    uint32_t res[3];                  // bin, count above it, its count
    uint32_t nsmall, tau, need;       // the last bin's keys, finished by one warp
    uint32_t small[64];
    uint32_t rcount[TC_CL];           // first CTA: each region's count, ~0u on overflow
};

// Word offset of candidate p in a region: four pad words after every 32, so
// that runs of a region read by consecutive threads spread over the banks and
// groups of four stay 16-byte aligned.
__device__ __forceinline__ uint32_t padw(uint32_t p) { return p + 4u * (p >> 5); }

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// The bin of hist (2048 bins, larger keys in higher bins) that holds the
// remaining-th largest key, the count above it and its own count, into
// sh.res.  Warp w scans bins 128 w .. 128 w + 127, four per lane; a suffix sum
// over the lanes and one over the warp totals place every lane.  Two
// barriers; also clears the histogram `other` for the next pass.
__device__ __forceinline__ void lean_find(const uint32_t *hist, uint32_t *other, uint32_t remaining,
                                          TcShared &sh) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int b0 = w * 128 + lane * 4;
    const uint4 hv = *reinterpret_cast<const uint4 *>(hist + b0);
    const uint32_t h[4] = {hv.x, hv.y, hv.z, hv.w};
    const uint32_t c = h[0] + h[1] + h[2] + h[3];
    uint32_t sfx = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_down_sync(0xffffffffu, sfx, o);
        if (lane + o < 32) sfx += t;
    }
    if (lane == 0) sh.wtot[w] = sfx;
    *reinterpret_cast<uint4 *>(other + b0) = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    uint32_t above = sfx - c;
#pragma unroll
    for (int v = 0; v < TC_WARPS; v++) above += v > w ? sh.wtot[v] : 0u;
#pragma unroll
    for (int i = 3; i >= 0; i--) {
        if (above < remaining && above + h[i] >= remaining) {
            sh.res[0] = (uint32_t)(b0 + i);
            sh.res[1] = above;
            sh.res[2] = h[i];
        }
        above += h[i];
    }
    __syncthreads();
}

// The rank-th largest (1-based) of the valid keys in registers, bits stop and
// up (the lower bits of the result are those all keys share, else zero):
// radix select with 11-bit digits starting at the highest bit in which the
// keys differ, so that keys crowded into a narrow range spread over the bins;
// plain shared-memory atomics.  need gets how many keys equal to the result
// are taken (meaningful when stop = 0).  sh.hist[0] must be clear on entry,
// and is again on return.
template <int NK, typename OkF>
__device__ void radix_kth(const uint32_t (&kr)[NK], OkF ok, uint32_t rank, int stop, TcShared &sh,
                          uint32_t &tau, uint32_t &need) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    uint32_t a1 = 0xffffffffu, o1 = 0u;
#pragma unroll
    for (int u = 0; u < NK; u++)
        if (ok(u)) {
            a1 &= kr[u];
            o1 |= kr[u];
        }
    a1 = __reduce_and_sync(0xffffffffu, a1);
    o1 = __reduce_or_sync(0xffffffffu, o1);
    if (lane == 0) {
        sh.wand[w] = a1;
        sh.wor[w] = o1;
    }
    if (tid == 0) sh.nsmall = 0u;
    __syncthreads();
    a1 = 0xffffffffu;
    o1 = 0u;
#pragma unroll
    for (int v = 0; v < TC_WARPS; v++) {
        a1 &= sh.wand[v];
        o1 |= sh.wor[v];
    }
    const uint32_t vary = a1 ^ o1;
    uint32_t prefix = a1 & ~vary, pmask = ~vary, remaining = rank;
    int hi = vary ? 31 - __clz(vary) : -1;
    int buf = 0;
    bool done = false;
#pragma unroll 1
    while (hi >= stop) {
        const int lo_bit = hi - 10 > stop ? hi - 10 : stop;
        const uint32_t dmask = (2u << (hi - lo_bit)) - 1u;
        uint32_t *hcur = sh.hist[buf];
#pragma unroll
        for (int u = 0; u < NK; u++)
            if (ok(u) && (kr[u] & pmask) == prefix) atomicAdd(&hcur[(kr[u] >> lo_bit) & dmask], 1u);
        __syncthreads();
        lean_find(hcur, sh.hist[buf ^ 1], remaining, sh);
        prefix |= sh.res[0] << lo_bit;
        remaining -= sh.res[1];
        pmask |= dmask << lo_bit;
        hi = lo_bit - 1;
        buf ^= 1;
        if (stop == 0 && hi >= 0 && sh.res[2] <= 64u) {
            // few keys left in the bin: gather them, and one warp finds the
            // remaining-th largest by counting, for each key, the keys above it
            const uint32_t nb = sh.res[2];
#pragma unroll
            for (int u = 0; u < NK; u++)
                if (ok(u) && (kr[u] & pmask) == prefix) sh.small[atomicAdd(&sh.nsmall, 1u)] = kr[u];
            __syncthreads();
            if (w == 0) {
                const uint32_t x0 = (uint32_t)lane < nb ? sh.small[lane] : 0u;
                const uint32_t x1 = (uint32_t)lane + 32u < nb ? sh.small[lane + 32] : 0u;
                uint32_t g0 = 0, e0 = 0, g1 = 0, e1 = 0;
                for (int j = 0; j < 64 && (uint32_t)j < nb; j++) {
                    const uint32_t y = __shfl_sync(0xffffffffu, j < 32 ? x0 : x1, j & 31);
                    g0 += y > x0 ? 1u : 0u;
                    e0 += y == x0 ? 1u : 0u;
                    g1 += y > x1 ? 1u : 0u;
                    e1 += y == x1 ? 1u : 0u;
                }
                if ((uint32_t)lane < nb && g0 < remaining && g0 + e0 >= remaining) {
                    sh.tau = x0;
                    sh.need = remaining - g0;
                }
                if ((uint32_t)lane + 32u < nb && g1 < remaining && g1 + e1 >= remaining) {
                    sh.tau = x1;
                    sh.need = remaining - g1;
                }
            }
            __syncthreads();
            prefix = sh.tau;
            remaining = sh.need;
            done = true;
            break;
        }
    }
    if (buf) {                        // hist[0] was counted last: clear it
        for (int i = tid; i < 2048; i += TK_THREADS) sh.hist[0][i] = 0u;
        __syncthreads();
    }
    tau = done ? prefix : prefix & ~((1u << stop) - 1u & vary);
    need = remaining;
}

// Writes, in index order, the id of every key above t and of the first
// need_eq keys equal to t (keys in registers, thread t holding a contiguous
// run of PT, nk of them valid): lane prefixes of the per-thread counts from
// ballots of their bits, warp bases from one exchange.
template <int PT, typename IdF>
__device__ void emit_ballot(const uint32_t (&ck)[PT], int nk, uint32_t t, uint32_t need_eq, IdF id,
                            TcShared &sh, int32_t *orow) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const unsigned lt = (1u << lane) - 1u;
    uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
    for (int u = 0; u < PT; u++) {
        n_gt += ck[u] > t && u < nk ? 1u : 0u;
        n_eq += ck[u] == t && u < nk ? 1u : 0u;
    }
    uint32_t pg = 0, pe = 0, tg = 0, te = 0;
#pragma unroll
    for (int b = 0; b < 5; b++) {                         // counts are at most 16
        const unsigned bg = __ballot_sync(0xffffffffu, (n_gt >> b) & 1u);
        const unsigned be = __ballot_sync(0xffffffffu, (n_eq >> b) & 1u);
        pg += (uint32_t)__popc(bg & lt) << b;
        pe += (uint32_t)__popc(be & lt) << b;
        tg += (uint32_t)__popc(bg) << b;
        te += (uint32_t)__popc(be) << b;
    }
    if (lane == 0) {
        sh.wtot[w] = tg;
        sh.wand[w] = te;
    }
    __syncthreads();
#pragma unroll
    for (int v = 0; v < TC_WARPS; v++) {
        pg += v < w ? sh.wtot[v] : 0u;
        pe += v < w ? sh.wand[v] : 0u;
    }
    uint32_t eq_before = pe;
    uint32_t pos = pg + (eq_before < need_eq ? eq_before : need_eq);
#pragma unroll
    for (int u = 0; u < PT; u++) {
        bool sel = false;
        if (u < nk) {
            if (ck[u] > t) sel = true;
            else if (ck[u] == t) sel = eq_before++ < need_eq;
        }
        if (sel) orow[pos++] = id(u);
    }
}

template <int KPT>
__global__ void __cluster_dims__(TC_CL, 1, 1) __launch_bounds__(TK_THREADS, KPT <= 8 ? 2 : 1)
topk_cluster_kernel(const float *__restrict__ scores, const int64_t *__restrict__ q_pos,
                    int32_t *__restrict__ idx, int32_t *__restrict__ cnt, int64_t E, int k, int m) {
    static_assert(KPT % 4 == 0, "keys come in groups of four");
    constexpr int U = KPT / 4;        // steps per warp
    extern __shared__ __align__(16) uint8_t tc_raw[];
    uint32_t *rkey = reinterpret_cast<uint32_t *>(tc_raw);                  // first CTA: [TC_CL][TC_RSTRIDE]
    int32_t *rid = reinterpret_cast<int32_t *>(tc_raw + TC_CL * TC_RSTRIDE * 4);
    __shared__ __align__(16) TcShared sh;
    __shared__ TkShared tk;           // the whole-row fallback
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    const unsigned rank = cl.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int64_t row = blockIdx.x / TC_CL;
    // the peers' shared memory is written only after every CTA of the cluster
    // has started: arrive now, wait just before the first remote write
    cluster_arrive_relaxed();
    const float *s = scores + row * E;
    const int64_t per = (((E + TC_CL - 1) / TC_CL) + 3) & ~(int64_t)3;
    const int64_t c0 = (int64_t)rank * per;
    const int64_t c1 = c0 + per < E ? c0 + per : E;
    const int64_t wb = c0 + (int64_t)w * (32 * KPT) + 4 * lane;   // this lane's first key
    uint32_t key[KPT];
    const bool vec = (((uintptr_t)s) & 15) == 0;
#pragma unroll
    for (int u = 0; u < U; u++) {
        const int64_t j = wb + (int64_t)u * 128;
        if (vec && j + 4 <= c1) {
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(s + j));
            key[4 * u] = score_key(v.x);
            key[4 * u + 1] = score_key(v.y);
            key[4 * u + 2] = score_key(v.z);
            key[4 * u + 3] = score_key(v.w);
        } else {
#pragma unroll
            for (int e = 0; e < 4; e++) key[4 * u + e] = j + e < c1 ? score_key(__ldcs(s + j + e)) : 0u;
        }
    }
    for (int i = tid; i < 2048; i += TK_THREADS) sh.hist[0][i] = 0u;
    const int64_t nv = visible_count(q_pos[row], m, E);
    int32_t *orow = idx + row * (int64_t)k;
    if (nv <= k) {                    // the same in every CTA of the cluster
        if (rank == 0) {
            for (int i = tid; i < k; i += TK_THREADS) orow[i] = i < nv ? i : -1;
            if (tid == 0) cnt[row] = (int32_t)nv;
        }
        cluster_wait();
        return;
    }
    const int64_t cv = c1 < nv ? c1 : nv;                    // visible keys end here
    // this lane's keys are visible while their offset from wb is below lim
    const int64_t lim64 = cv - wb;
    const int lim = (int)(lim64 < 0 ? 0 : (lim64 > 0x7fffffff ? 0x7fffffff : lim64));
    // the bound: the r-th largest of TK_LSAMPLE evenly spaced keys (two per
    // thread), its bits below 12 cleared
    const int S = (int)(nv < TK_LSAMPLE ? nv : TK_LSAMPLE);
    uint32_t sk[2];
    bool sv[2];
#pragma unroll
    for (int h = 0; h < 2; h++) {
        const int i = tid + h * TK_THREADS;
        const int64_t pos = S == TK_LSAMPLE ? (((int64_t)i * nv) >> 10) : i;   // TK_LSAMPLE = 2^10
        sv[h] = i < S;
        sk[h] = sv[h] ? score_key(s[pos]) : 0u;
    }
    __syncthreads();                  // hist[0] is clear
    const int r = S < TK_LSAMPLE ? k : sample_rank(nv, k, S);
    uint32_t lo = 0, unused;
    if (r < S) radix_kth(sk, [&](int h) { return sv[h]; }, (uint32_t)r, 12, sh, lo, unused);
    // this CTA's keys >= lo, in index order: per warp, steps in order, lanes
    // in order within a step, a lane's four keys in order
    uint32_t wcount = 0;
#pragma unroll
    for (int u = 0; u < U; u++)
#pragma unroll
        for (int e = 0; e < 4; e++) wcount += u * 128 + e < lim && key[4 * u + e] >= lo ? 1u : 0u;
    wcount = __reduce_add_sync(0xffffffffu, wcount);
    if (lane == 0) sh.wtot[w] = wcount;
    __syncthreads();
    uint32_t base = 0, tot = 0;
#pragma unroll
    for (int v = 0; v < TC_WARPS; v++) {
        const uint32_t x = sh.wtot[v];
        base += v < w ? x : 0u;
        tot += x;
    }
    if (tot <= (uint32_t)TC_CAPR) {
        // staged in this CTA's own region (the first CTA's is final)
        uint32_t *dk = rkey + rank * TC_RSTRIDE;
        int32_t *di = rid + rank * TC_RSTRIDE;
        const unsigned lt = (1u << lane) - 1u;
        uint32_t run = base;
#pragma unroll
        for (int u = 0; u < U; u++) {
            bool in[4];
            uint32_t c = 0;
#pragma unroll
            for (int e = 0; e < 4; e++) {
                in[e] = u * 128 + e < lim && key[4 * u + e] >= lo;
                c += in[e] ? 1u : 0u;
            }
            // the lanes' counts (0..4) bit by bit: their prefix over the lanes
            // from three ballots
            const unsigned b0 = __ballot_sync(0xffffffffu, c & 1u), b1 = __ballot_sync(0xffffffffu, c & 2u),
                           b2 = __ballot_sync(0xffffffffu, c & 4u);
            if ((b0 | b1 | b2) == 0u) continue;
            uint32_t p = run + (uint32_t)__popc(b0 & lt) + 2u * (uint32_t)__popc(b1 & lt) +
                         4u * (uint32_t)__popc(b2 & lt);
            const int64_t j = wb + (int64_t)u * 128;
#pragma unroll
            for (int e = 0; e < 4; e++)
                if (in[e]) {
                    dk[padw(p)] = key[4 * u + e];
                    di[padw(p)] = (int32_t)(j + e);
                    p++;
                }
            run += (uint32_t)__popc(b0) + 2u * (uint32_t)__popc(b1) + 4u * (uint32_t)__popc(b2);
        }
    }
    __syncthreads();
    cluster_wait();
    if (rank != 0 && tot <= (uint32_t)TC_CAPR && tot > 0) {
        // the staged region to the first CTA, 16 bytes a store
        const uint32_t nvec = (padw(tot - 1) + 4u) >> 2;
        const uint4 *sk4 = reinterpret_cast<const uint4 *>(rkey + rank * TC_RSTRIDE);
        const uint4 *si4 = reinterpret_cast<const uint4 *>(rid + rank * TC_RSTRIDE);
        uint4 *dk4 = reinterpret_cast<uint4 *>(cl.map_shared_rank(rkey, 0) + rank * TC_RSTRIDE);
        uint4 *di4 = reinterpret_cast<uint4 *>(cl.map_shared_rank(rid, 0) + rank * TC_RSTRIDE);
        for (uint32_t i = (uint32_t)tid; i < nvec; i += TK_THREADS) {
            dk4[i] = sk4[i];
            di4[i] = si4[i];
        }
    }
    if (tid == 0) cl.map_shared_rank(sh.rcount, 0)[rank] = tot <= (uint32_t)TC_CAPR ? tot : 0xffffffffu;
    cl.sync();                        // every region is written
    if (rank != 0) return;
    uint32_t off[TC_CL + 1];
    bool bad = false;
    off[0] = 0;
#pragma unroll
    for (int q = 0; q < TC_CL; q++) {
        const uint32_t cq = sh.rcount[q];
        bad |= cq == 0xffffffffu;
        off[q + 1] = off[q] + (cq == 0xffffffffu ? 0u : cq);
    }
    const uint32_t n = off[TC_CL];
    if (!bad && n >= (uint32_t)k && n <= (uint32_t)(TC_PT * TK_THREADS)) {
        uint32_t ck[TC_PT];
        int32_t ci[TC_PT];
#pragma unroll
        for (int q = 0; q < TC_PT; q++) {
            const uint32_t g = (uint32_t)tid * TC_PT + q;
            int v = 0;
#pragma unroll
            for (int x = 1; x < TC_CL; x++) v += g >= off[x] ? 1 : 0;
            const uint32_t pr = g - off[v];
            const uint32_t at = (uint32_t)v * TC_RSTRIDE + padw(pr);
            ck[q] = g < n ? rkey[at] : 0u;
            ci[q] = g < n ? rid[at] : 0;
        }
        const int64_t l2 = (int64_t)n - (int64_t)tid * TC_PT;
        const int nk2 = (int)(l2 < 0 ? 0 : (l2 > TC_PT ? TC_PT : l2));
        uint32_t tau, need_eq;
        radix_kth(ck, [&](int q) { return q < nk2; }, (uint32_t)k, 0, sh, tau, need_eq);
        emit_ballot(ck, nk2, tau, need_eq, [&](int q) { return ci[q]; }, sh, orow);
    } else {
        select_core(tk, nv, k, [&](int64_t j) { return score_key(s[j]); },
                    [](int64_t j) { return (int32_t)j; }, orow);
    }
    if (tid == 0) cnt[row] = k;
}

// -------------------------------------------------------------------- host

static PerDevice g_final_smem;
constexpr int CAND_CAP = 24576;      // candidates cached per row (192 KB)

bool topk_use_long(int64_t rows, int64_t E) { return rows < 256 && E > 16384; }

int topk_chunks(int64_t rows, int64_t E) {
    int64_t ch = (296 + rows - 1) / rows;
    const int64_t maxch = (E + 4095) / 4096;
    if (ch > maxch) ch = maxch;
    if (ch > 256) ch = 256;
    return ch < 1 ? 1 : (int)ch;
}

static size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

// keys per thread of the cluster kernel for rows of E entries (0: too long)
static int topk_cluster_kpt(int64_t E) {
    for (int kpt = 8; kpt <= 64; kpt *= 2)
        if (E <= (int64_t)TC_CL * TK_THREADS * kpt) return kpt;
    return 0;
}

size_t topk_scratch_bytes(int64_t rows, int64_t E) {
    if (!topk_use_long(rows, E) || topk_cluster_kpt(E) > 0) return 0;
    const int ch = topk_chunks(rows, E);
    return a256((size_t)rows * ch * 4) + 2 * a256((size_t)rows * E * 4);
}

// phase 1: everything, or for long rows only the candidate collection;
// phase 2: for long rows, the exact selection (nothing otherwise).
cudaError_t launch_topk_phase(int phase, int64_t B, int64_t Tq, int64_t E, int k, int m,
                              const float *scores, const int64_t *q_pos, int32_t *idx, int32_t *cnt,
                              void *scratch, cudaStream_t st) {
    const int64_t rows = B * Tq;
    if (rows == 0) return cudaSuccess;
    if (topk_use_long(rows, E) && topk_cluster_kpt(E) > 0) {
        if (phase != 1) return cudaSuccess;
        if (rows > 65535) return cudaErrorInvalidValue;
        const dim3 g((unsigned)(rows * TC_CL));
        const int kpt = topk_cluster_kpt(E);
        const void *fn = kpt == 8 ? (const void *)topk_cluster_kernel<8>
                       : kpt == 16 ? (const void *)topk_cluster_kernel<16>
                       : kpt == 32 ? (const void *)topk_cluster_kernel<32>
                                   : (const void *)topk_cluster_kernel<64>;
        static PerDevice cl_smem[4];
        {
            cudaError_t e = smem_limit_once(cl_smem[kpt == 8 ? 0 : kpt == 16 ? 1 : kpt == 32 ? 2 : 3], fn, TC_SMEM);
            if (e != cudaSuccess) return e;
        }
        switch (kpt) {
        case 8: topk_cluster_kernel<8><<<g, TK_THREADS, TC_SMEM, st>>>(scores, q_pos, idx, cnt, E, k, m); break;
        case 16: topk_cluster_kernel<16><<<g, TK_THREADS, TC_SMEM, st>>>(scores, q_pos, idx, cnt, E, k, m); break;
        case 32: topk_cluster_kernel<32><<<g, TK_THREADS, TC_SMEM, st>>>(scores, q_pos, idx, cnt, E, k, m); break;
        default: topk_cluster_kernel<64><<<g, TK_THREADS, TC_SMEM, st>>>(scores, q_pos, idx, cnt, E, k, m); break;
        }
        count_launches(1);
        return cudaGetLastError();
    }
    if (topk_use_long(rows, E)) {
        if (scratch == nullptr) return cudaErrorInvalidValue;
        TkLong a;
        const int ch = topk_chunks(rows, E);
        char *p = (char *)scratch;
        a.chunk_cnt = (uint32_t *)p;
        p += a256((size_t)rows * ch * 4);
        a.cand_key = (uint32_t *)p;
        p += a256((size_t)rows * E * 4);
        a.cand_idx = (int32_t *)p;
        a.scores = scores; a.q_pos = q_pos; a.idx = idx; a.cnt = cnt;
        a.E = E; a.CH = ch; a.CS = (E + ch - 1) / ch; a.k = k; a.m = m;
        if (phase == 1) {
            dim3 g((unsigned)ch, (unsigned)rows);
            topk_collect_kernel<<<g, TK_THREADS, 0, st>>>(a);
            count_launches(1);
            return cudaGetLastError();
        }
        {
            cudaError_t e = smem_limit_once(g_final_smem, (const void *)topk_final_kernel, CAND_CAP * 8);
            if (e != cudaSuccess) return e;
        }
        topk_final_kernel<<<(unsigned)rows, TK_THREADS, CAND_CAP * 8, st>>>(a, CAND_CAP);
        count_launches(1);
        return cudaGetLastError();
    }
    if (phase != 1) return cudaSuccess;
    static PerDevice tw_attr;
    const size_t smem = TW_WARPS * sizeof(TwShared);
    {
        cudaError_t e = smem_limit_once(tw_attr, (const void *)topk_kernel, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int64_t blocks = (rows + TW_WARPS - 1) / TW_WARPS;
    const int64_t cap = (int64_t)device_sms();           // one resident CTA per SM
    if (blocks > cap) blocks = cap;
    topk_kernel<<<(unsigned)blocks, TW_WARPS * 32, smem, st>>>(scores, q_pos, idx, cnt, rows, E, k, m);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_topk(int64_t B, int64_t Tq, int64_t E, int k, int m, const float *scores,
                        const int64_t *q_pos, int32_t *idx, int32_t *cnt, void *scratch,
                        cudaStream_t st) {
    cudaError_t e = launch_topk_phase(1, B, Tq, E, k, m, scores, q_pos, idx, cnt, scratch, st);
    if (e != cudaSuccess) return e;
    return launch_topk_phase(2, B, Tq, E, k, m, scores, q_pos, idx, cnt, scratch, st);
}

// -------------------------------------------------- allocation-free selection
//
// Callers that cannot allocate device memory (code running where cudaMalloc
// is not available or not allowed, e.g. inside an allocator-free serving loop
// or a host that only hands over pre-registered buffers) can still select
// over long rows: topk_select_noalloc keeps its scratch (chunk counts and
// candidates) in the file-scope device array below instead of a
// caller workspace.  Limits: at most NOALLOC_MAX_ROWS rows and
// NOALLOC_MAX_ENTRIES = rows x E entries when the long-row path is taken.
constexpr int64_t NOALLOC_MAX_ROWS = 64;
constexpr int64_t NOALLOC_MAX_ENTRIES = int64_t(1) << 21;
constexpr size_t NOALLOC_BYTES = size_t(17) << 20;   // 17 MiB on every device that loads the library
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

static std::mutex g_noalloc_mu;
static void *g_noalloc_ptr[64];

// The array's device address, looked up once per device with that device
// current (host code only holds a stand-in for the symbol).
static cudaError_t noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace csa

extern "C" csa_status topk_select_noalloc(int64_t B, int64_t T, int64_t E, int32_t k, int32_t m,
                                         const float *scores, const int64_t *q_pos, int32_t *idx,
                                         int32_t *cnt, void *stream) {
    using namespace csa;
    auto bad = [](const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (B < 0 || T < 0 || E < 0) return report_error(CSA_ERR_INVALID_ARG, "negative size");
    if (k < 1 || k > 2048) return report_error(CSA_ERR_UNSUPPORTED, "k not in 1..2048");
    if (m < 1) return report_error(CSA_ERR_INVALID_ARG, "m must be >= 1");
    if (E > 2147483647LL) return report_error(CSA_ERR_UNSUPPORTED, "E too large");
    const int64_t rows = B * T;
    if (rows == 0) return CSA_OK;
    if ((E > 0 && bad(scores)) || bad(q_pos) || bad(idx) || bad(cnt))
        return report_error(CSA_ERR_INVALID_ARG, "a tensor pointer is NULL or not 16-byte aligned");
    void *scratch = nullptr;
    if (topk_use_long(rows, E)) {
        if (rows > NOALLOC_MAX_ROWS || rows * E > NOALLOC_MAX_ENTRIES ||
            topk_scratch_bytes(rows, E) > NOALLOC_BYTES)
            return report_error(CSA_ERR_UNSUPPORTED,
                                "topk_select_noalloc: rows x entries beyond its static scratch "
                                "(at most 64 rows and 2^21 entries in all); use topk_select");
        cudaError_t e = noalloc_scratch(&scratch);
        if (e != cudaSuccess) return report_error(CSA_ERR_CUDA, cudaGetErrorString(e));
    }
    cudaError_t e = launch_topk(B, T, E, k, m, scores, q_pos, idx, cnt, scratch, (cudaStream_t)stream);
    if (e != cudaSuccess) return report_error(CSA_ERR_CUDA, cudaGetErrorString(e));
    return CSA_OK;
}
