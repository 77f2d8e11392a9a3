// Lightning-indexer scores on the 5th-generation tensor cores (bf16 inputs,
// fp32 accumulation in tensor memory), fed by TMA.
//
// ["DeepSeek-V4: Making Million-Token Context an Architectural Problem",
// Key design 1 index-score equation; DeepSeek-V4 book ch.6 "The index
// score", and ch.8 "Indexer arithmetic": the indexer dominates the per-query
// arithmetic.]  scores[b,t,j] = sum_h w[b,t,h] * ReLU(qI[b,t,h,:] . kI[b,j,:]).
//
// Orientation: compressed entries on the MMA's M side (128 TMEM lanes, one
// entry per lane), (token, head) pairs on N.  One tcgen05.mma tile is
// 128 entries x (QT tokens x 64 heads) x 128 dims, so every epilogue thread
// owns one entry row and reduces sum_h w * ReLU over its own columns: no
// cross-thread reduction.
//
// Warp roles (one persistent CTA per SM):
//   warp 0     TMA producer: the query block's qI tile once per work item,
//              then a ring of kI tiles (STAGES deep);
//   warp 1     TMEM allocator and MMA issuer for the even tiles, warp 2 for the
//              odd ones (converged warps, one issuing lane each);
//   warps 3..  epilogue: tcgen05.ld of a finished accumulator, ReLU, the
//              w-weighted head sum, masked fp32 stores; two accumulators
//              alternate so the epilogue of tile i overlaps the MMA of i+1.
// Prefill (QT = 4): a work item is one block of 4 consecutive queries and
// every entry tile it can see (causal: later blocks see more); items are
// dealt to CTAs largest-first in snake order.  Decode (QT = 1, one query per
// sequence): the B x E entry tiles are split evenly over all CTAs, so one
// long sequence spreads across the whole GPU and the kI stream stays
// HBM-bound.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace csa {

struct IdxArgs {
    const float *w;          // [B, T, 64]
    const int64_t *q_pos;    // [B, T]
    float *scores;           // [B, T, E]
    unsigned *status;
    int B, T, nqb, tps;      // nqb: query blocks per sequence; tps: entry tiles per sequence
    int64_t E;
    int m;
    int write_masked;
    long long spin;          // polls before a wait between roles gives up
};

template <int QT>
struct IdxCfg {
    static constexpr int HI = 64;
    static constexpr int N = QT * HI;
    static constexpr int BM = 128;
    static constexpr int DI = 128;
    static constexpr int KH = DI / 64;
    static constexpr int STAGES = QT == 4 ? 4 : 6;
    static constexpr int A_BYTES = BM * DI * 2;
    static constexpr int B_BYTES = N * DI * 2;
    static constexpr int ACC_COLS = N;
    static constexpr int TMEM_COLS = QT == 4 ? 512 : 128;
    static constexpr int EPI_WARPS = QT == 4 ? 8 : 4;
    static constexpr int TPW = QT * 4 / EPI_WARPS;    // tokens (64 columns each) per epilogue warp
    static constexpr int EPI0 = 3;                     // first epilogue warp
    static constexpr int THREADS = (EPI0 + EPI_WARPS) * 32;
    static constexpr int W_FLOATS = TPW > 1 ? EPI_WARPS * 64 : 0;   // second token's weights per warp
    static constexpr int SMEM = STAGES * A_BYTES + B_BYTES + W_FLOATS * 4 + 256 + 1024;
};

struct Item {
    int b, qb, jt0, jt1;
};

template <int QT>
__device__ __forceinline__ bool idx_item(const IdxArgs &a, int cta, int G, int r, Item &it) {
    if (QT == 4) {
        const long long k = (long long)r * G + ((r & 1) ? (G - 1 - cta) : cta);
        if (k >= (long long)a.B * a.nqb) return false;
        const int qd = (int)(k / a.B);
        it.b = (int)(k % a.B);
        it.qb = a.nqb - 1 - qd;
        int64_t nv = 0;
        for (int u = 0; u < QT; u++) {
            const int t = it.qb * QT + u;
            if (t < a.T) {
                const int64_t v = visible_count(a.q_pos[(int64_t)it.b * a.T + t], a.m, a.E);
                nv = v > nv ? v : nv;
            }
        }
        it.jt0 = 0;
        it.jt1 = (int)((nv + 127) / 128);
        return true;
    } else {
        const long long TT = (long long)a.B * a.T * a.tps;
        const long long g0 = TT * cta / G, g1 = TT * (cta + 1) / G;
        long long g = g0;
        for (int i = 0; i < r; i++) {
            if (g >= g1) return false;
            const long long bnd = (g / a.tps + 1) * a.tps;
            g = bnd < g1 ? bnd : g1;
        }
        if (g >= g1) return false;
        const long long row = g / a.tps;         // (b, t) flattened
        it.b = (int)(row / a.T);
        it.qb = (int)(row % a.T);
        it.jt0 = (int)(g % a.tps);
        const long long end = (row + 1) * a.tps < g1 ? (row + 1) * a.tps : g1;
        it.jt1 = (int)(end - row * a.tps);
        const int64_t nv = visible_count(a.q_pos[row], a.m, a.E);
        const int lim = (int)((nv + 127) / 128);
        if (it.jt1 > lim) it.jt1 = lim;
        return true;
    }
}

template <int QT>
__global__ void __launch_bounds__(IdxCfg<QT>::THREADS, 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  IdxArgs a) {
    using Cfg = IdxCfg<QT>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;                                   // [STAGES][KH][128][128 B]
    uint8_t *sB = sA + Cfg::STAGES * Cfg::A_BYTES;        // [KH][N][128 B]
    float *w_all = (float *)(sB + Cfg::B_BYTES);          // [EPI_WARPS][64] (prefill)
    uint64_t *bars = (uint64_t *)(w_all + Cfg::W_FLOATS);
    uint64_t *full = bars;                                 // [STAGES]
    uint64_t *empty = full + Cfg::STAGES;                  // [STAGES]
    uint64_t *bfull = empty + Cfg::STAGES;
    uint64_t *bempty = bfull + 1;
    uint64_t *accfull = bempty + 1;                        // [2]
    uint64_t *accempty = accfull + 2;                      // [2]
    uint64_t *mdone = accempty + 2;                        // [2] every MMA a warp issued has completed
    uint32_t *tmem_slot = (uint32_t *)(mdone + 2);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; s++) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        tc::mbar_init(bfull, 1);
        tc::mbar_init(bempty, 2);                          // both MMA warps
        for (int i = 0; i < 2; i++) {
            tc::mbar_init(&accfull[i], 1);
            tc::mbar_init(&accempty[i], Cfg::EPI_WARPS);
        }
        tc::mbar_init(&mdone[0], 1);
        tc::mbar_init(&mdone[1], 1);
        *abort_flag = 0;
        tc::fence_barrier_init();
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_k);
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        // The whole warp runs the loop and waits; one lane issues the copies.
        const bool leader = lane == 0;
        int stage = 0;
        uint32_t phase = 0, bphase = 0;
        uint32_t issued_mask = 0, last_par = 0, b_issued = 0, b_par = 0;
        Item it;
        for (int r = 0; idx_item<QT>(a, cta, G, r, it); r++) {
            if (it.jt0 >= it.jt1) continue;
            if (!tc::warp_wait(bempty, bphase ^ 1, a.status, abort_flag, a.spin)) break;
            if (leader) {
                tc::mbar_expect_tx(bfull, Cfg::B_BYTES);
                const int qrow = (int)(((int64_t)it.b * a.T + (int64_t)it.qb * QT) * Cfg::HI);
                for (int kh = 0; kh < Cfg::KH; kh++)
                    tc::tma_load_2d(sB + kh * Cfg::N * 128, &tm_q, kh * 64, qrow, bfull);
                // the next item's queries on their way to L2: its tile loads
                // only once this item's products are done, and from HBM that
                // left the tensor pipe idle between items
                Item nx;
                if (QT == 4 && idx_item<QT>(a, cta, G, r + 1, nx)) {
                    const int nrow = (int)(((int64_t)nx.b * a.T + (int64_t)nx.qb * QT) * Cfg::HI);
                    for (int kh = 0; kh < Cfg::KH; kh++) tc::prefetch_l2_box(&tm_q, kh * 64, nrow);
                }
            }
            __syncwarp();
            b_issued = 1;
            b_par = bphase;
            bool ok = true;
            for (int jt = it.jt0; jt < it.jt1; jt++) {
                if (!tc::warp_wait(&empty[stage], phase ^ 1, a.status, abort_flag, a.spin)) { ok = false; break; }
                if (leader) {
                    tc::mbar_expect_tx(&full[stage], Cfg::A_BYTES);
                    const int krow = (int)((int64_t)it.b * a.E + (int64_t)jt * 128);
                    uint8_t *dst = sA + stage * Cfg::A_BYTES;
                    for (int kh = 0; kh < Cfg::KH; kh++)
                        if (QT == 1)   // decode: kI is read once, the scores right after
                            tc::tma_load_2d_hint(dst + kh * 128 * 128, &tm_k, kh * 64, krow, &full[stage],
                                                 tc::l2_evict_first());
                        else
                            tc::tma_load_2d(dst + kh * 128 * 128, &tm_k, kh * 64, krow, &full[stage]);
                }
                __syncwarp();
                issued_mask |= 1u << stage;
                last_par = (last_par & ~(1u << stage)) | (phase << stage);
                if (++stage == Cfg::STAGES) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            bphase ^= 1;
        }
        if (*abort_flag) {
            // let every copy this warp issued land before the CTA exits
            for (int s = 0; s < Cfg::STAGES; s++)
                if (issued_mask & (1u << s))
                    for (long long i = 0; i < tc::DRAIN_LIMIT; i++)
                        if (tc::mbar_test(&full[s], (last_par >> s) & 1u)) break;
            if (b_issued)
                for (long long i = 0; i < tc::DRAIN_LIMIT; i++)
                    if (tc::mbar_test(bfull, b_par)) break;
        }
    } else if (warp == 1 || warp == 2) {
        // --------------------------------------------------------------- MMA
        // Two issuing warps take alternate tiles (warp 1 the even ones of the
        // CTA's tile sequence, warp 2 the odd ones), so each always fills
        // the same accumulator; one warp's barrier waits overlap the other's
        // issue.  Each warp runs converged with one issuing lane.
        const int p = warp - 1;
        const bool leader = lane == 0;
        constexpr uint32_t idesc = tc::idesc_bf16_f32(128, Cfg::N);
        uint32_t g = 0, bphase = 0;
        const uint32_t aBase = tc::smem_u32(sA), bBase = tc::smem_u32(sB);
        Item it;
        for (int r = 0; idx_item<QT>(a, cta, G, r, it); r++) {
            if (it.jt0 >= it.jt1) continue;
            if (!tc::warp_wait(bfull, bphase, a.status, abort_flag, a.spin)) break;
            tc::fence_after_sync();
            bool ok = true;
            for (int jt = it.jt0; jt < it.jt1; jt++, g++) {
                if ((int)(g & 1) != p) continue;
                const int stage = (int)(g % Cfg::STAGES);
                const uint32_t phase = (g / Cfg::STAGES) & 1;
                if (!tc::warp_wait(&full[stage], phase, a.status, abort_flag, a.spin) ||
                    !tc::warp_wait(&accempty[p], ((g >> 1) & 1) ^ 1, a.status, abort_flag, a.spin)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                if (leader) {
                    const uint32_t d = tmem + p * Cfg::ACC_COLS;
                    const uint32_t aS = aBase + stage * Cfg::A_BYTES;
#pragma unroll
                    for (int kh = 0; kh < Cfg::KH; kh++)
#pragma unroll
                        for (int kk = 0; kk < 4; kk++) {
                            const uint64_t ad = tc::desc_kmajor_sw128(aS + kh * 128 * 128 + kk * 32);
                            const uint64_t bd = tc::desc_kmajor_sw128(bBase + kh * Cfg::N * 128 + kk * 32);
                            tc::mma_bf16(d, ad, bd, idesc, (kh | kk) != 0);
                        }
                    tc::mma_commit(&empty[stage]);
                    tc::mma_commit(&accfull[p]);
                }
                __syncwarp();
            }
            if (!ok) break;
            // the query tile is free once both warps' products of this item are done
            if (leader) tc::mma_commit(bempty);
            __syncwarp();
            bphase ^= 1;
        }
        // every MMA issued above has completed before TMEM is released
        if (leader) tc::mma_commit(&mdone[p]);
        __syncwarp();
        for (long long i = 0; i < tc::DRAIN_LIMIT; i++)
            if (tc::mbar_test(&mdone[p], 0)) break;
    } else {
        // ---------------------------------------------------------- epilogue
        const int ew = warp - Cfg::EPI0;         // 0 .. EPI_WARPS-1
        const int quarter = warp & 3;            // TMEM lanes this warp may read
        constexpr int TPW = Cfg::TPW;
        const int tt0 = (ew >> 2) * TPW;         // this warp's first token within the block
        const int row = quarter * 32 + lane;     // entry row within the tile
        int acc = 0;
        uint32_t accphase = 0;
        Item it;
        bool ok = true;
        for (int r = 0; ok && idx_item<QT>(a, cta, G, r, it); r++) {
            if (it.jt0 >= it.jt1) continue;
            // The first token's 64 head weights stay in registers for the
            // whole item; the second token's (prefill) sit in this warp's
            // slice of shared memory.  The MMA's operand reads keep shared
            // memory busy, and reloading all the weights from there every
            // tile left the epilogue, not the tensor core, setting the pace;
            // registers for both tokens leave only 16 columns per
            // tensor-memory load, and its round trips then hold the
            // accumulator longer.
            float wr[64];
            float *wsB = TPW > 1 ? w_all + ew * 64 : nullptr;    // prefill only
            int64_t nv[TPW];
            float *srow[TPW];
#pragma unroll
            for (int u = 0; u < TPW; u++) {
                const int t = it.qb * QT + tt0 + u;
                const bool real = t < a.T;
                const int64_t brow = (int64_t)it.b * a.T + (real ? t : 0);
                if (u == 0) {
                    const float4 *w4 = reinterpret_cast<const float4 *>(a.w + brow * Cfg::HI);
#pragma unroll
                    for (int h = 0; h < 16; h++) {
                        const float4 q = real ? __ldg(w4 + h) : make_float4(0.f, 0.f, 0.f, 0.f);
                        wr[4 * h] = q.x; wr[4 * h + 1] = q.y; wr[4 * h + 2] = q.z; wr[4 * h + 3] = q.w;
                    }
                } else {
                    __syncwarp();
                    wsB[lane] = real ? a.w[brow * Cfg::HI + lane] : 0.f;
                    wsB[lane + 32] = real ? a.w[brow * Cfg::HI + lane + 32] : 0.f;
                    __syncwarp();
                }
                nv[u] = real ? visible_count(a.q_pos[brow], a.m, a.E) : -1;
                srow[u] = a.scores + brow * a.E;
            }
            const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + tt0 * Cfg::HI;
            for (int jt = it.jt0; jt < it.jt1; jt++) {
                if (!tc::warp_wait(&accfull[acc], accphase, a.status, abort_flag, a.spin)) { ok = false; break; }
                tc::fence_after_sync();
                const int64_t j = (int64_t)jt * 128 + row;
                const uint32_t ta = tbase + acc * Cfg::ACC_COLS;
#pragma unroll
                for (int u = 0; u < TPW; u++) {
                    float v[64];
                    tc::tmem_ld32(ta + u * 64, v);
                    tc::tmem_ld32(ta + u * 64 + 32, v + 32);
                    tc::tmem_ld_wait();
                    tc::tmem_regs_ready<64>(v);
                    if (u == TPW - 1) {
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&accempty[acc]);
                    }
                    float s0 = 0.f, s1 = 0.f;
                    if (u == 0) {
#pragma unroll
                        for (int h = 0; h < 32; h++) {
                            s0 = fmaf(wr[h], fmaxf(v[h], 0.f), s0);
                            s1 = fmaf(wr[32 + h], fmaxf(v[32 + h], 0.f), s1);
                        }
                    } else {
                        const float4 *wt = reinterpret_cast<const float4 *>(wsB);
#pragma unroll
                        for (int h = 0; h < 8; h++) {
                            const float4 wa = wt[h], wb = wt[8 + h];
                            s0 = fmaf(wa.x, fmaxf(v[4 * h + 0], 0.f), s0);
                            s1 = fmaf(wb.x, fmaxf(v[32 + 4 * h + 0], 0.f), s1);
                            s0 = fmaf(wa.y, fmaxf(v[4 * h + 1], 0.f), s0);
                            s1 = fmaf(wb.y, fmaxf(v[32 + 4 * h + 1], 0.f), s1);
                            s0 = fmaf(wa.z, fmaxf(v[4 * h + 2], 0.f), s0);
                            s1 = fmaf(wb.z, fmaxf(v[32 + 4 * h + 2], 0.f), s1);
                            s0 = fmaf(wa.w, fmaxf(v[4 * h + 3], 0.f), s0);
                            s1 = fmaf(wb.w, fmaxf(v[32 + 4 * h + 3], 0.f), s1);
                        }
                    }
                    if (nv[u] >= 0 && j < a.E) {
                        if (j < nv[u]) {
                            // decode: the selection reads the scores next, from L2
                            // if the key stream has not evicted them
                            if (QT == 1) tc::st_global_hint(&srow[u][j], s0 + s1, tc::l2_evict_last());
                            else srow[u][j] = s0 + s1;
                        }
                        else if (a.write_masked) srow[u][j] = -INFINITY;
                    }
                }
                if (++acc == 2) { acc = 0; accphase ^= 1; }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

// Standalone scores are fully defined: every entry a query cannot see gets
// -inf (the fused paths skip this; their selection reads the visible prefix).
__global__ void mask_tail_kernel(float *scores, const int64_t *q_pos, int64_t rows, int64_t E, int m) {
    const int64_t row = blockIdx.y + (int64_t)blockIdx.z * 65535;
    if (row >= rows) return;
    const int64_t nv = visible_count(q_pos[row], m, E);
    for (int64_t j = nv + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < E;
         j += (int64_t)gridDim.x * blockDim.x)
        scores[row * E + j] = -INFINITY;
}

cudaError_t launch_mask_tail(float *scores, const int64_t *q_pos, int64_t rows, int64_t E, int m, cudaStream_t st) {
    if (rows == 0 || E == 0) return cudaSuccess;
    dim3 g(8, (unsigned)(rows < 65535 ? rows : 65535), (unsigned)((rows + 65534) / 65535));
    mask_tail_kernel<<<g, 256, 0, st>>>(scores, q_pos, rows, E, m);
    count_launches(1);
    return cudaGetLastError();
}

// ------------------------------------------------------------------- host

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// 2D bf16 tensor map over a row-major [rows, cols] array, box [box_rows, 64],
// 128-byte swizzle.
bool make_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                       uint32_t box_rows) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool indexer_tc_supported(int hI, int dI, int64_t B, int64_t T, int64_t E) {
    return hI == 64 && dI == 128 && B * T * 64 < (1LL << 31) && B * E < (1LL << 31) && E > 0;
}

template <int QT>
static cudaError_t launch_tc(const CUtensorMap &tq, const CUtensorMap &tk, const IdxArgs &a,
                             int grid, cudaStream_t st) {
    using Cfg = IdxCfg<QT>;
    static PerDevice attr;
    {
        cudaError_t e = smem_limit_once(attr, (const void *)indexer_tc_kernel<QT>, Cfg::SMEM);
        if (e != cudaSuccess) return e;
    }
    indexer_tc_kernel<QT><<<grid, Cfg::THREADS, Cfg::SMEM, st>>>(tq, tk, a);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_indexer_tc(int64_t B, int64_t T, int64_t E, int m, const void *qI,
                              const float *w, const void *kI, const int64_t *q_pos, float *scores,
                              int write_masked, unsigned *status, int max_ctas, long long spin,
                              cudaStream_t st) {
    if (B * T == 0 || E == 0) return cudaSuccess;
    IdxArgs a;
    a.w = w; a.q_pos = q_pos; a.scores = scores; a.status = status;
    a.B = (int)B; a.T = (int)T; a.E = E; a.m = m; a.write_masked = write_masked;
    a.spin = spin;
    a.tps = (int)((E + 127) / 128);
    const bool decode = T < 4;
    const int QT = decode ? 1 : 4;
    a.nqb = (int)((T + QT - 1) / QT);
    CUtensorMap tq, tk;
    if (!make_tmap_bf16_2d(&tq, qI, (uint64_t)(B * T * 64), 128, decode ? 64 : 256) ||
        !make_tmap_bf16_2d(&tk, kI, (uint64_t)(B * E), 128, 128))
        return cudaErrorInvalidValue;
    const int sms = max_ctas > 0 && max_ctas < device_sms() ? max_ctas : device_sms();
    cudaError_t e;
    if (decode) {
        long long tiles = (long long)B * T * a.tps;
        int grid = (int)(tiles < sms ? tiles : sms);
        e = launch_tc<1>(tq, tk, a, grid, st);
    } else {
        long long items = (long long)B * a.nqb;
        int grid = (int)(items < sms ? items : sms);
        e = launch_tc<4>(tq, tk, a, grid, st);
    }
    if (e != cudaSuccess || !write_masked) return e;
    return launch_mask_tail(scores, q_pos, B * T, E, m, st);
}

}  // namespace csa
