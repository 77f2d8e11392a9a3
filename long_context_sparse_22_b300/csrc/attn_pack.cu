// Dense attention with 128 rows per work item: every visible compressed entry
// plus the sliding window, for a layer whose head count divides 128, at
// c = 128 (the heavily compressed layer of the 16-head configuration), with
// the optional q RMSNorm ("DeepSeek-V4" book ch.7 "Query and KV normalization") and
// log-denominator output.
//
// ["DeepSeek-V4" book ch.7 "HCA's compressor": HCA attends to every visible
// compressed entry plus the window; ch.6 "Sliding-window keys and values",
// "The attention sink"; ch.7 "Partial rotary position embeddings".]
//
// An item holds 128 / H consecutive queries of one sequence; their (query,
// head) pairs are the 128 rows of every product, so the union of their lists
// (the compressed entries up to the last query, the window rows from the
// first query's window start) is read once, and each row keeps only its own
// query's entries and window rows.  Per 64-entry tile, two tcgen05 products:
// S = q~ K^T (M = 128 rows, N = 64 entries, K = 128) and O^T += V^T P^T
// (M = 128 dims, N = 128 rows, K = 64 entries); K = V is the same tile in
// shared memory.  One thread owns one row in the softmax (its 64 logits from
// one 32x32b tensor-memory load pair, no shuffles); O^T is rescaled in tensor
// memory only when some row's running max grows by more than 2^8.
//
// Warp roles (persistent CTAs, items dealt round-robin):
//   warps 0-3  loaders: q rows (box TMA, rotated at each query's position in
//              place), entry tiles (four buffers) and their presence masks;
//   warp 4     TMEM allocator and QK issuer;
//   warps 5-8  softmax (one row per thread), O rescale, epilogue (one dim per
//              thread: normalise, de-rotate per row, store);
//   warp 9     PV issuer.
// Every wait is bounded (csa_params.spin_limit) and taken by a whole warp.
#include "attn_common.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace csa {

struct PkCfg {
    static constexpr int C = 128;
    static constexpr int ROWS = 128;
    static constexpr int TE = 64;                    // entries per tile
    static constexpr int K_ATOM = TE * 128;          // 64 rows x 128 B (64 dims)
    static constexpr int K_BYTES = 2 * K_ATOM;       // 128 dims
    static constexpr int Q_ATOM = ROWS * 128;        // 128 rows x 64 dims
    static constexpr int Q_BYTES = 2 * Q_ATOM;
    static constexpr int P_BYTES = ROWS * 128;       // 128 rows x 64 entries bf16
    static constexpr int NKB = 4, QB = 2;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_Q = OFF_K + NKB * K_BYTES;
    static constexpr int OFF_P = OFF_Q + QB * Q_BYTES;
    static constexpr int OFF_MISC = OFF_P + 2 * P_BYTES;
    static constexpr int MISC_BYTES = 16384;
    static constexpr int SMEM = OFF_MISC + MISC_BYTES + 1024;
    static constexpr int S_COL = 0;                  // two S buffers: columns 0, 64
    static constexpr int O_COL = 128;                // O^T: 128 columns (one per row)
    static constexpr int TMEM_COLS = 256;
    static constexpr int NLOAD = 128;                // warps 0-3
    static constexpr int QK_WARP = 4, SM_WARP0 = 5, PV_WARP = 9;
    static constexpr int THREADS = (PV_WARP + 1) * 32;
    static constexpr int MAX_QPI = 8;                // 128 / 16
    static constexpr int MAX_PAIRS = 64;             // rotary dims up to 128
};

struct PkArgs {
    const __nv_bfloat16 *kvc;
    const __nv_bfloat16 *kv_raw;
    const int64_t *q_pos;
    const int64_t *raw_pos0;
    const float *sink;
    __nv_bfloat16 *out;
    float *lse;              // [B*T*H] log-denominators, or nullptr
    const float *q_norm;     // RMSNorm gains of q (C floats), or nullptr
    float norm_eps;
    unsigned *status;
    int64_t T, E, L;
    int H, m, n_win, derotate, qpi;
    int64_t tq_blocks, n_items;
    long long spin;
    float scale_log2;
    RopeFreqs rope;
};

struct PkItem {
    int64_t b, bt0;          // sequence, first query row
    int64_t t, tmin;         // largest and smallest position of the item's queries
    int nq;                  // queries in the item
    int64_t ncomp;           // compressed entries visible to the last query (tiles 0 .. ntc-1)
    int64_t p0, nwin;        // window rows p0 .. p0 + nwin - 1 (tiles ntc ..)
    int ntc, nt;
};

__device__ __forceinline__ void pk_item(const PkArgs &a, int64_t it, PkItem &f) {
    f.b = it / a.tq_blocks;
    const int64_t i0 = (it % a.tq_blocks) * a.qpi;
    f.bt0 = f.b * a.T + i0;
    f.nq = (int)(a.T - i0 < a.qpi ? a.T - i0 : a.qpi);
    f.t = f.tmin = a.q_pos[f.bt0];
    for (int q = 1; q < f.nq; q++) {
        const int64_t tq = a.q_pos[f.bt0 + q];
        f.t = tq > f.t ? tq : f.t;
        f.tmin = tq < f.tmin ? tq : f.tmin;
    }
    f.ncomp = visible_count(f.t, a.m, a.E);
    if (f.ncomp < 0) f.ncomp = 0;
    int64_t p0 = f.tmin - a.n_win + 1;
    if (p0 < 0) p0 = 0;
    f.p0 = p0;
    f.nwin = a.n_win > 0 && f.t >= 0 ? f.t - p0 + 1 : 0;
    f.ntc = (int)((f.ncomp + 63) / 64);
    f.nt = f.ntc + (int)((f.nwin + 63) / 64);
}

__global__ void __launch_bounds__(PkCfg::THREADS, 1)
attn_pack_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c,
                 const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ PkArgs a) {
    using Cfg = PkCfg;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sK = smem + Cfg::OFF_K;
    uint8_t *sQ = smem + Cfg::OFF_Q;
    uint8_t *sP = smem + Cfg::OFF_P;
    uint8_t *misc = smem + Cfg::OFF_MISC;
    uint64_t *bar = (uint64_t *)misc;                  // 32 barrier slots
    uint64_t *kfull = bar + 0, *kempty = bar + 4;      // [NKB]
    uint64_t *sfull = bar + 8, *sempty = bar + 10, *pfull = bar + 12, *pempty = bar + 14;
    uint64_t *qland = bar + 16, *qfull = bar + 18, *qempty = bar + 20;   // [QB]
    uint64_t *ofull = bar + 22, *oempty = bar + 23, *mdone = bar + 24;
    uint32_t *tmem_slot = (uint32_t *)(misc + 256);
    volatile int *abort_flag = (volatile int *)(misc + 260);
    uint32_t *vmask32 = (uint32_t *)(misc + 272);      // [NKB][2] presence bits of a tile's rows
    float *alpha_s = (float *)(misc + 512);            // [2][128] rescale factor of each row
    float *inv_den_s = (float *)(misc + 1536);         // [128]
    float *cs_c = (float *)(misc + 2048);              // [MAX_QPI][MAX_PAIRS] cos of the query angle
    float *cs_s = (float *)(misc + 4096);              //                      sin
    float *ep_c = (float *)(misc + 8192);              // [MAX_QPI][128] cos of -t_q at each dim
    float *ep_s = (float *)(misc + 12288);             //                sin

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::NKB; i++) {
            tc::mbar_init(&kfull[i], Cfg::NLOAD);
            tc::mbar_init(&kempty[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            tc::mbar_init(&sfull[i], 1);
            tc::mbar_init(&sempty[i], 4);
            tc::mbar_init(&pfull[i], 4);
            tc::mbar_init(&pempty[i], 1);
        }
        for (int i = 0; i < Cfg::QB; i++) {
            tc::mbar_init(&qland[i], 1);
            tc::mbar_init(&qfull[i], 1);
            tc::mbar_init(&qempty[i], 1);
        }
        tc::mbar_init(ofull, 1);
        tc::mbar_init(oempty, 4);
        tc::mbar_init(mdone, 2);
        *abort_flag = 0;
        tc::fence_barrier_init();
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_c);
        tc::prefetch_tmap(&tm_w);
    }
    if (warp == Cfg::QK_WARP) tc::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int np = a.rope.pairs;

    if (warp < 4) {
        // ------------------------------------------------------------ loaders
        const int tid = threadIdx.x;
        uint32_t g = 0, ii = 0;
        uint32_t tma_issued = 0, last_g[Cfg::NKB] = {}, q_pending = 0, q_pend_b = 0, q_pend_par = 0;
        bool ok = true;
        for (int64_t it = blockIdx.x; ok && it < a.n_items; it += G) {
            PkItem f;
            pk_item(a, it, f);
            if (f.nt == 0) continue;
            // the rotation angles of the item's queries, padding queries of a
            // short last item at the item's last position (published by the
            // barrier that ends the q-buffer wait)
            for (int i = tid; i < a.qpi * np; i += Cfg::NLOAD) {
                const int q = i / np, pi = i - q * np;
                float c_, s_;
                rope_cos_sin(a.rope, q < f.nq ? a.q_pos[f.bt0 + q] : f.t, pi, c_, s_);
                cs_c[q * Cfg::MAX_PAIRS + pi] = c_;
                cs_s[q * Cfg::MAX_PAIRS + pi] = s_;
            }
            const int qb = (int)(ii % Cfg::QB);
            const uint32_t qpar = (ii / Cfg::QB) & 1;
            uint8_t *sQb = sQ + qb * Cfg::Q_BYTES;
            if (named_bar_or(2, Cfg::NLOAD, !warp_wait(&qempty[qb], qpar ^ 1, a.status, abort_flag, a.spin))) {
                ok = false;
                break;
            }
            if (tid == 0) {
                tc::mbar_expect_tx(&qland[qb], Cfg::Q_BYTES);
                for (int at = 0; at < 2; at++)
                    for (int hf = 0; hf < 2; hf++)
                        tc::tma_load_2d(sQb + at * Cfg::Q_ATOM + hf * 8192, &tm_q, at * 64,
                                        (int)(f.bt0 * a.H + hf * 64), &qland[qb]);
                q_pending = 1;
                q_pend_b = qb;
                q_pend_par = qpar;
            }
            // q~ = RoPE(q, t_q) in place, once q has landed; runs while the item's
            // first tile is in flight
            auto rope_q = [&]() -> bool {
                if (named_bar_or(2, Cfg::NLOAD, !warp_wait(&qland[qb], qpar, a.status, abort_flag, a.spin)))
                    return false;
                if (tid == 0) q_pending = 0;
                if (a.q_norm) {
                    // RMSNorm of each row before its rotation, one row per thread
                    // (the normalised row is rounded to bf16, then rotated)
                    const int r = tid;
                    float ss = 0.f;
#pragma unroll 4
                    for (int k = 0; k < 16; k++) {
                        const int d0 = k * 8;
                        const uint4 u = *reinterpret_cast<const uint4 *>(sQb + (d0 >> 6) * Cfg::Q_ATOM + (r >> 3) * 1024 +
                                                                         swz128(r, (d0 & 63) * 2));
                        float fv[8];
                        Vec<__nv_bfloat16>::unpack(u, fv);
#pragma unroll
                        for (int e = 0; e < 8; e++) ss = fmaf(fv[e], fv[e], ss);
                    }
                    const float rs = 1.0f / sqrtf(ss / (float)Cfg::C + a.norm_eps);
#pragma unroll 4
                    for (int k = 0; k < 16; k++) {
                        const int d0 = k * 8;
                        uint4 *pu = reinterpret_cast<uint4 *>(sQb + (d0 >> 6) * Cfg::Q_ATOM + (r >> 3) * 1024 +
                                                              swz128(r, (d0 & 63) * 2));
                        float fv[8];
                        Vec<__nv_bfloat16>::unpack(*pu, fv);
                        uint4 o;
                        __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
                        for (int e = 0; e < 4; e++)
                            o2[e] = __floats2bfloat162_rn(fv[2 * e] * rs * __ldg(a.q_norm + d0 + 2 * e),
                                                          fv[2 * e + 1] * rs * __ldg(a.q_norm + d0 + 2 * e + 1));
                        *pu = o;
                    }
                    named_bar(2, Cfg::NLOAD);
                }
                if (np == 32) {
                    // one pair per lane; warp w rotates rows w, w + 4, ...
                    const int d = a.rope.first + 2 * lane;
                    uint8_t *qa = sQb + (d >> 6) * Cfg::Q_ATOM;
#pragma unroll 4
                    for (int k = 0; k < Cfg::ROWS / 4; k++) {
                        const int r = warp + 4 * k;
                        const int q = r / a.H;
                        __nv_bfloat162 *pv = (__nv_bfloat162 *)(qa + (r >> 3) * 1024 + swz128(r, (d & 63) * 2));
                        const float c_ = cs_c[q * Cfg::MAX_PAIRS + lane], s_ = cs_s[q * Cfg::MAX_PAIRS + lane];
                        const float2 v = __bfloat1622float2(*pv);
                        *pv = __floats2bfloat162_rn(v.x * c_ - v.y * s_, v.x * s_ + v.y * c_);
                    }
                } else {
                    for (int i = tid; i < Cfg::ROWS * np; i += Cfg::NLOAD) {
                        const int r = i / np, pi = i - r * np;
                        const int d = a.rope.first + 2 * pi;
                        const int q = r / a.H;
                        __nv_bfloat162 *pv = (__nv_bfloat162 *)(sQb + (d >> 6) * Cfg::Q_ATOM + (r >> 3) * 1024 +
                                                                swz128(r, (d & 63) * 2));
                        const float c_ = cs_c[q * Cfg::MAX_PAIRS + pi], s_ = cs_s[q * Cfg::MAX_PAIRS + pi];
                        const float2 v = __bfloat1622float2(*pv);
                        *pv = __floats2bfloat162_rn(v.x * c_ - v.y * s_, v.x * s_ + v.y * c_);
                    }
                }
                fence_proxy_async();
                named_bar(2, Cfg::NLOAD);
                if (tid == 0) tc::mbar_arrive(&qfull[qb]);
                return true;
            };
            const int64_t rp0 = a.raw_pos0[f.b];
            for (int j = 0; j < f.nt; j++, g++) {
                const int buf = (int)(g % Cfg::NKB);
                const uint32_t kpar = (g / Cfg::NKB) & 1;
                if (named_bar_or(2, Cfg::NLOAD, !warp_wait(&kempty[buf], kpar ^ 1, a.status, abort_flag, a.spin))) {
                    ok = false;
                    break;
                }
                // presence of the tile's rows, then its 64-row TMA boxes
                int64_t y;
                if (j < f.ntc) {
                    if (tid < 64) {
                        const bool v = (int64_t)j * 64 + tid < f.ncomp;
                        const uint32_t bal = __ballot_sync(0xffffffffu, v);
                        if (lane == 0) vmask32[buf * 2 + warp] = bal;
                    }
                    y = f.b * a.E + (int64_t)j * 64;
                } else {
                    const int64_t jw = j - f.ntc;
                    if (tid < 64) {
                        const int64_t raw = f.p0 - rp0 + jw * 64 + tid;
                        const bool in = jw * 64 + tid < f.nwin;
                        const bool v = in && raw >= 0 && raw < a.L;
                        if (in && !v) atomicOr(a.status, ST_NO_WINDOW_ROW);
                        const uint32_t bal = __ballot_sync(0xffffffffu, v);
                        if (lane == 0) vmask32[buf * 2 + warp] = bal;
                    }
                    // rows outside the array are zero-filled by the copy
                    y = f.b * a.L + f.p0 - rp0 + jw * 64;
                    if (y < -64) y = -64;
                    if (y > 0x7fff0000LL) y = 0x7fff0000LL;
                }
                if (tid == 0) {
                    tc::mbar_expect_tx(&kfull[buf], Cfg::K_BYTES);
                    for (int at = 0; at < 2; at++)
                        tc::tma_load_2d(sK + buf * Cfg::K_BYTES + at * Cfg::K_ATOM, j < f.ntc ? &tm_c : &tm_w,
                                        at * 64, (int)y, &kfull[buf]);
                    tma_issued |= 1u << buf;
                    last_g[buf] = g;
                } else {
                    tc::mbar_arrive(&kfull[buf]);
                }
                if (j == 0 && !rope_q()) {
                    ok = false;
                    break;
                }
            }
            ii++;
        }
        if (*abort_flag && tid == 0) {
            // let every copy issued by TMA land before the CTA exits
            for (int s = 0; s < Cfg::NKB; s++)
                if (tma_issued & (1u << s))
                    for (long long i = 0; i < tc::DRAIN_LIMIT; i++)
                        if (tc::mbar_test(&kfull[s], (last_g[s] / Cfg::NKB) & 1)) break;
            if (q_pending)
                for (long long i = 0; i < tc::DRAIN_LIMIT; i++)
                    if (tc::mbar_test(&qland[q_pend_b], q_pend_par)) break;
        }
    } else if (warp == Cfg::QK_WARP || warp == Cfg::PV_WARP) {
        // --------------------------------------------------------------- MMA
        const bool is_qk = warp == Cfg::QK_WARP;
        const bool leader = lane == 0;
        constexpr uint32_t idQK = tc::idesc_bf16_f32(128, 64);
        constexpr uint32_t idPV = tc::idesc_bf16_f32(128, 128) | (1u << 15);   // A (V^T) MN-major
        const uint64_t dq0 = desc_sw128(tc::smem_u32(sQ), 16, 1024);
        const uint64_t dk0 = desc_sw128(tc::smem_u32(sK), 16, 1024);
        const uint64_t dv0 = desc_sw128(tc::smem_u32(sK), Cfg::K_ATOM, 1024);
        const uint64_t dp0 = desc_sw128(tc::smem_u32(sP), 16, 1024);
        uint32_t g = 0, ii = 0;
        bool ok = true;
        for (int64_t it = blockIdx.x; ok && it < a.n_items; it += G) {
            PkItem f;
            pk_item(a, it, f);
            if (f.nt == 0) continue;
            const int nt = f.nt;
            if (is_qk) {
                const int qb = (int)(ii % Cfg::QB);
                if (!warp_wait(&qfull[qb], (ii / Cfg::QB) & 1, a.status, abort_flag, a.spin)) break;
                const uint64_t dq = dq0 + (uint64_t)((qb * Cfg::Q_BYTES) >> 4);
                for (int n = 0; n < nt; n++) {
                    const uint32_t gq = g + n;
                    const int buf = gq & 1;
                    const int kbuf = (int)(gq % Cfg::NKB);
                    if (!warp_wait(&kfull[kbuf], (gq / Cfg::NKB) & 1, a.status, abort_flag, a.spin) ||
                        !warp_wait(&sempty[buf], ((gq >> 1) & 1) ^ 1, a.status, abort_flag, a.spin)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    if (leader) {
#pragma unroll
                        for (int at = 0; at < 2; at++)
#pragma unroll
                            for (int kk = 0; kk < 4; kk++)
                                tc::mma_bf16(tmem + Cfg::S_COL + buf * 64,
                                             dq + (uint64_t)((at * Cfg::Q_ATOM + kk * 32) >> 4),
                                             dk0 + (uint64_t)((kbuf * Cfg::K_BYTES + at * Cfg::K_ATOM + kk * 32) >> 4),
                                             idQK, (at | kk) != 0);
                        tc::mma_commit(&sfull[buf]);
                        if (n == nt - 1) tc::mma_commit(&qempty[qb]);
                    }
                    __syncwarp();
                }
            } else {
                for (int n = 0; n < nt; n++) {
                    const uint32_t gp = g + n;
                    const int bp = gp & 1;
                    const int kbuf = (int)(gp % Cfg::NKB);
                    if (!warp_wait(&pfull[bp], (gp >> 1) & 1, a.status, abort_flag, a.spin) ||
                        (n == 0 && !warp_wait(oempty, (ii & 1) ^ 1, a.status, abort_flag, a.spin))) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    if (leader) {
#pragma unroll
                        for (int ks = 0; ks < 4; ks++)
                            tc::mma_bf16(tmem + Cfg::O_COL,
                                         dv0 + (uint64_t)((kbuf * Cfg::K_BYTES + ks * 2048) >> 4),
                                         dp0 + (uint64_t)((bp * Cfg::P_BYTES + ks * 32) >> 4), idPV,
                                         (n == 0 && ks == 0) ? 0u : 1u);
                        tc::mma_commit(&pempty[bp]);
                        tc::mma_commit(&kempty[kbuf]);
                    }
                    __syncwarp();
                }
                if (ok && leader) tc::mma_commit(ofull);
            }
            g += nt;
            ii++;
        }
        // every MMA issued above has completed before TMEM is released
        if (leader) tc::mma_commit(mdone);
        __syncwarp();
        if (is_qk)
            for (long long i = 0; i < tc::DRAIN_LIMIT; i++)
                if (tc::mbar_test(mdone, 0)) break;
    } else {
        // ------------------------------------------- softmax, rescale, epilogue
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        const int r = quarter * 32 + lane;       // this thread's row (softmax) and dim (epilogue)
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const int qr = r / a.H, hr = r - qr * a.H;   // the row's query in the item, its head
        const float zl = a.sink[hr] * 1.4426950408889634f;
        const bool rot = a.derotate && r >= a.rope.first;   // the epilogue dim is rotary
        uint32_t g = 0, ii = 0;
        for (int64_t it = blockIdx.x; it < a.n_items; it += G) {
            PkItem f;
            pk_item(a, it, f);
            if (f.nt == 0) continue;
            const bool real = qr < f.nq;
            const int64_t t_r = real ? a.q_pos[f.bt0 + qr] : f.t;
            // the row's own list: entries j < nv, window offsets from p0 in (wlo, whi]
            const int nv = (int)visible_count(t_r, a.m, a.E);
            const int wlo = (int)(t_r - a.n_win - f.p0), whi = (int)(t_r - f.p0);
            // the de-rotation angles of this thread's epilogue dim, per query
            if (rot)
                for (int q = 0; q < f.nq; q++) {
                    float c_, s_;
                    rope_cos_sin(a.rope, -a.q_pos[f.bt0 + q], (r - a.rope.first) >> 1, c_, s_);
                    ep_c[q * 128 + r] = c_;
                    ep_s[q * 128 + r] = s_;
                }
            float m_run = zl, l_run = 0.f;
            const uint32_t gfirst = g;
            bool fail = false;
            for (int j = 0; j < f.nt; j++, g++) {
                const int buf = g & 1;                   // S and P buffers
                const uint32_t par = (g >> 1) & 1;
                const int kbuf = (int)(g % Cfg::NKB);   // entry tile
                const uint32_t kpar = (g / Cfg::NKB) & 1;
                bool ok = warp_wait(&kfull[kbuf], kpar, a.status, abort_flag, a.spin) &&
                          warp_wait(&pempty[buf], par ^ 1, a.status, abort_flag, a.spin);
                uint32_t mlo = ok ? vmask32[kbuf * 2] : 0u, mhi = ok ? vmask32[kbuf * 2 + 1] : 0u;
                ok = ok && warp_wait(&sfull[buf], par, a.status, abort_flag, a.spin);
                float v[64];
                if (ok) {
                    tc::fence_after_sync();
                    tc::tmem_ld32(tmem + lane_base + Cfg::S_COL + buf * 64, v);
                    tc::tmem_ld32(tmem + lane_base + Cfg::S_COL + buf * 64 + 32, v + 32);
                    tc::tmem_ld_wait();
                    tc::tmem_regs_ready<64>(v);
                }
                // this row's entries of the tile: present, and in its own list
                {
                    int lo, hi;
                    if (j < f.ntc) {
                        lo = 0;
                        hi = nv - j * 64;
                    } else {
                        const int base = (j - f.ntc) * 64;
                        lo = wlo - base + 1;
                        hi = whi - base + 1;
                    }
                    lo = lo < 0 ? 0 : (lo > 64 ? 64 : lo);
                    hi = hi < 0 ? 0 : (hi > 64 ? 64 : hi);
                    const uint64_t below_hi = hi >= 64 ? ~0ull : (1ull << hi) - 1ull;
                    const uint64_t below_lo = lo >= 64 ? ~0ull : (1ull << lo) - 1ull;
                    const uint64_t im = hi > lo ? below_hi & ~below_lo : 0ull;
                    mlo &= (uint32_t)im;
                    mhi &= (uint32_t)(im >> 32);
                    if (!real) mlo = mhi = 0u;
                }
                float mx = -INFINITY;
#pragma unroll
                for (int e = 0; e < 64; e++) {
                    const uint32_t bit = e < 32 ? (mlo >> e) & 1u : (mhi >> (e - 32)) & 1u;
                    v[e] = bit ? v[e] * a.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, v[e]);
                }
                const float m_new = fmaxf(m_run, mx);
                const bool need = m_new > m_run + 8.0f;
                const float alpha = need ? ex2(m_run - m_new) : 1.0f;
                if (need) m_run = m_new;
                const float msub = m_run == -INFINITY ? 0.f : m_run;
                // P row (bf16): 16-byte chunk c of row r at chunk c ^ (r & 7)
                uint8_t *prow = sP + buf * Cfg::P_BYTES + (r >> 3) * 1024 + (r & 7) * 128;
                float ps = 0.f;
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e2 = 0; e2 < 4; e2++) {
                        const float p0 = ex2(v[8 * c + 2 * e2] - msub), p1 = ex2(v[8 * c + 2 * e2 + 1] - msub);
                        ps += p0 + p1;
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                        w4[e2] = *reinterpret_cast<uint32_t *>(&h2);
                    }
                    if (ok)
                        *reinterpret_cast<uint4 *>(prow + ((c ^ (r & 7)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
                l_run = l_run * alpha + ps;
                if (ok) alpha_s[buf * 128 + r] = alpha;
                fence_proxy_async();
                // one barrier in the common case: nothing failed, no row needs a rescale
                const bool resc = need && g != gfirst;
                if (named_bar_or(1, 128, !ok || resc)) {
                    if (named_bar_or(1, 128, !ok)) { fail = true; break; }
                    // some row's max grew: O^T was accumulated with older maxima,
                    // scale column r by alpha[r] (each warp its 32 dims)
                    const uint32_t gp = g - 1;
                    if (warp_wait(&pempty[gp & 1], (gp >> 1) & 1, a.status, abort_flag, a.spin)) {
                        tc::fence_after_sync();
                        const float *al = alpha_s + buf * 128;
#pragma unroll 1
                        for (int cb = 0; cb < 128; cb += 16) {
                            const uint32_t to = tmem + lane_base + Cfg::O_COL + cb;
                            uint32_t o[16];
                            tmem_ld16(to, o);
                            tc::tmem_ld_wait();
                            tc::tmem_regs_ready<16>(o);
#pragma unroll
                            for (int q = 0; q < 16; q++) o[q] = __float_as_uint(__uint_as_float(o[q]) * al[cb + q]);
                            tmem_st16(to, o);
                        }
                        tmem_st_wait();
                    }
                }
                // S buffer free for the QK two tiles on, P ready for this tile's PV
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&sempty[buf]);
                    tc::mbar_arrive(&pfull[buf]);
                }
            }
            if (fail) break;
            // item end: the row's denominator (the sink in it), then the epilogue
            // with one dim per thread over the 128 rows
            const float den = l_run + (zl != -INFINITY ? ex2(zl - m_run) : 0.f);
            inv_den_s[r] = (real && den > 0.f) ? 1.0f / den : 0.f;
            if (a.lse && real)
                a.lse[(f.bt0 + qr) * a.H + hr] = den > 0.f ? (m_run + log2f(den)) * 0.6931471805599453f : -INFINITY;
            const bool ok = warp_wait(ofull, ii & 1, a.status, abort_flag, a.spin);
            if (named_bar_or(1, 128, !ok)) break;
            tc::fence_after_sync();
            const int d = r;
            const int nrows = f.nq * a.H;
            __nv_bfloat16 *obase = a.out + f.bt0 * a.H * (int64_t)Cfg::C + d;
#pragma unroll 1
            for (int rb = 0; rb < 128; rb += 32) {
                float o[32];
                tc::tmem_ld32(tmem + lane_base + Cfg::O_COL + rb, o);
                tc::tmem_ld_wait();
                tc::tmem_regs_ready<32>(o);
                const float4 *id4 = reinterpret_cast<const float4 *>(inv_den_s + rb);
#pragma unroll
                for (int q4 = 0; q4 < 8; q4++) {
                    const float4 iv4 = id4[q4];
                    o[4 * q4] *= iv4.x;
                    o[4 * q4 + 1] *= iv4.y;
                    o[4 * q4 + 2] *= iv4.z;
                    o[4 * q4 + 3] *= iv4.w;
                }
                // rows rb .. rb + 31 belong to queries rb / H .. (rb + 31) / H
                // (at most two when H = 16); each is rotated back by its own
                // query's position
                const int q0 = rb / a.H, split = (q0 + 1) * a.H - rb;
                const int q1 = q0 + 1 < Cfg::MAX_QPI ? q0 + 1 : q0;
                float c0 = 1.f, s0 = 0.f, c1 = 1.f, s1 = 0.f;
                if (rot) {
                    if (q0 < f.nq) { c0 = ep_c[q0 * 128 + d]; s0 = ep_s[q0 * 128 + d]; }
                    if (q1 < f.nq) { c1 = ep_c[q1 * 128 + d]; s1 = ep_s[q1 * 128 + d]; }
                }
#pragma unroll
                for (int h = 0; h < 32; h++) {
                    const float op = __shfl_xor_sync(0xffffffffu, o[h], 1);
                    const bool second = h >= split;
                    const float ch = second ? c1 : c0, sh = second ? s1 : s0;
                    if (rot) o[h] = o[h] * ch + op * ((lane & 1) ? sh : -sh);
                }
#pragma unroll
                for (int h = 0; h < 32; h++)
                    if (rb + h < nrows) obase[(int64_t)(rb + h) * Cfg::C] = __float2bfloat16_rn(o[h]);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(oempty);
            named_bar(1, 128);                   // inv_den_s and the angles are rewritten by the next item
            ii++;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == Cfg::QK_WARP) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

bool attn_pack_supported(int64_t B, const AttnArgs &g, int n_chunks) {
    // TMA row coordinates are 32-bit
    const int64_t lim = 0x7fff0000LL;
    return g.c == 128 && !g.kv8 && g.idx == nullptr && n_chunks <= 1 && g.H >= 16 && 128 % g.H == 0 &&
           g.rope.pairs <= PkCfg::MAX_PAIRS &&
           g.Tq >= 1 && B * g.Tq * g.H < lim && B * g.E < lim && B * g.L < lim;
}

cudaError_t launch_attn_pack(int64_t B, const AttnArgs &g, int max_ctas, cudaStream_t st) {
    using Cfg = PkCfg;
    PkArgs a;
    a.kvc = (const __nv_bfloat16 *)g.kvc;
    a.kv_raw = (const __nv_bfloat16 *)g.kv_raw;
    a.q_pos = g.q_pos;
    a.raw_pos0 = g.raw_pos0;
    a.sink = g.sink;
    a.out = (__nv_bfloat16 *)g.out;
    a.lse = g.lse;
    a.q_norm = g.q_norm;
    a.norm_eps = g.norm_eps;
    a.status = g.status;
    a.T = g.Tq; a.E = g.E; a.L = g.L;
    a.H = g.H; a.m = g.m; a.n_win = g.n_win; a.derotate = g.derotate;
    a.qpi = Cfg::ROWS / g.H;
    a.tq_blocks = (g.Tq + a.qpi - 1) / a.qpi;
    a.n_items = B * a.tq_blocks;
    a.spin = g.spin;
    a.scale_log2 = g.scale * 1.4426950408889634f;
    a.rope = g.rope;
    if (a.n_items == 0) return cudaSuccess;
    const int64_t qrows = B * g.Tq * g.H;
    CUtensorMap tq, tcmp, tw;
    const bool have_c = g.E > 0 && g.kvc != nullptr;
    const bool have_w = g.L > 0 && g.kv_raw != nullptr;
    if (!make_tmap_bf16_2d(&tq, g.q, (uint64_t)qrows, Cfg::C, 64) ||
        !make_tmap_bf16_2d(&tcmp, have_c ? g.kvc : g.q, have_c ? (uint64_t)(B * g.E) : (uint64_t)qrows,
                           Cfg::C, 64) ||
        !make_tmap_bf16_2d(&tw, have_w ? g.kv_raw : g.q, have_w ? (uint64_t)(B * g.L) : (uint64_t)qrows,
                           Cfg::C, 64))
        return cudaErrorInvalidValue;
    static PerDevice attr;
    {
        cudaError_t e = smem_limit_once(attr, (const void *)attn_pack_kernel, Cfg::SMEM);
        if (e != cudaSuccess) return e;
    }
    const int sms = max_ctas > 0 && max_ctas < device_sms() ? max_ctas : device_sms();
    const int grid = (int)(a.n_items < sms ? a.n_items : sms);
    attn_pack_kernel<<<grid, Cfg::THREADS, Cfg::SMEM, st>>>(tq, tcmp, tw, a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace csa
