// Core attention on the 5th-generation tensor cores (bf16 in, fp32 out of
// tensor memory): shared-KV MQA over a per-query list of entries (selected
// or visible compressed entries, then the window rows) plus a sink logit.
//
// [DeepSeek-V4 book ch.6 "Shared key-value MQA"; ch.7 "The sliding window",
// "Partial rotary position embeddings", "Why the output is de-rotated",
// "Attention sinks"; "DeepSeek-V4: Making Million-Token Context an
// Architectural Problem", Key design 1 and 2.]
//
// Orientation: the entries of one tile (64) sit on the MMA's M side and the
// 64 heads of a head group on N, so one entry row read from HBM/L2 feeds all
// heads:
//   S^T[e, h]  = K[e, :] . q~[h, :]           M = 64 entries,  N = 64 heads
//   O^T[d, h] += V[:, d]^T . P^T[:, h]         M = 128 dims (x C/128), N = 64
// K = V is the same gathered tile; for the second product it is read as an
// MN-major operand, so no transposed copy exists.  The softmax runs across
// TMEM lanes: S^T is staged through shared memory, each head's max and
// exponentials are taken by two threads, and O^T in tensor memory is
// rescaled only when a head's running max grows by more than 2^8 (results
// are exact either way because the denominator uses the same max).  The sink
// logit seeds the running max and enters only the denominator.
//
// Warp roles (persistent CTAs, items dealt round-robin):
//   warps 0-2  q~ preparation (cp.async of the q rows into the swizzled
//              layout, then RoPE at t in place) and the cp.async gather of
//              each 64-entry tile into a 128-byte-swizzled K-major layout
//              (two tile buffers);
//   warp 3     TMEM allocator and MMA issuer: QK(j+1) is issued before
//              PV(j), so the tensor core works while tile j's softmax runs;
//   warps 4-7  softmax, O rescale, and the epilogue (normalise, de-rotate,
//              store), or fp32 partial outputs for a split-KV combine.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace csa {

template <int C>
struct AtCfg {
    static constexpr int NA = C / 64;             // 64-dim atoms
    static constexpr int NC = C / 128;            // 128-dim output chunks
    static constexpr int TE = 64;                 // entries per tile
    static constexpr int HG = 64;                 // heads per CTA item
    static constexpr int K_BYTES = NA * TE * 128; // one tile
    static constexpr int Q_BYTES = NA * HG * 128;
    static constexpr int P_BYTES = HG * 128;      // 64 heads x 64 entries bf16
    static constexpr int STAGE_LD = 65;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_Q = OFF_K + 2 * K_BYTES;
    static constexpr int OFF_P = OFF_Q + Q_BYTES;
    static constexpr int OFF_STAGE = OFF_P + 2 * P_BYTES;
    static constexpr int OFF_MISC = OFF_STAGE + TE * STAGE_LD * 4;
    static constexpr int MISC_BYTES = 2176;
    static constexpr int SMEM = OFF_MISC + MISC_BYTES;
    static constexpr int TMEM_COLS = 512;
    static constexpr int S_COL = 0;               // two S^T buffers: cols 0, 64
    static constexpr int O_COL = 128;             // O^T chunks: 128 + 64 c
    static constexpr int THREADS = 256;
};

struct AttnTcArgs {
    const __nv_bfloat16 *q;
    const int64_t *q_pos;
    const __nv_bfloat16 *kvc;
    const int32_t *idx;      // [B,T,k] or nullptr: every visible entry
    const int32_t *cnt;      // [B,T] kept count of idx rows, or nullptr (use k)
    const __nv_bfloat16 *kv_raw;
    const int64_t *raw_pos0;
    const float *sink;
    __nv_bfloat16 *out;
    float *lse;
    unsigned *status;
    float *part_o;           // split mode: [items][64][C] unnormalised
    float *part_ml;          // split mode: [items][64][2] (max in log2 units, sum)
    int64_t T, E, L;
    int H, k, m, n_win, derotate, n_hg;
    int chunk_tiles;         // > 0: split mode with this many tiles per item
    int n_chunks;
    int64_t n_items;
    float scale_log2;        // logit scale * log2(e)
    RopeFreqs rope;
};

struct ItemInfo {
    int64_t bt, b, t;
    int hg, chunk;
    int64_t ncomp, p0, total;   // list: ncomp compressed slots, then window rows p0..t
    int j0, j1;                 // tile range of this item
};

__device__ __forceinline__ void item_info(const AttnTcArgs &a, int64_t it, ItemInfo &f) {
    int64_t r = it;
    f.chunk = 0;
    if (a.chunk_tiles > 0) {
        f.chunk = (int)(r % a.n_chunks);
        r /= a.n_chunks;
    }
    f.hg = (int)(r % a.n_hg);
    f.bt = r / a.n_hg;
    f.b = f.bt / a.T;
    f.t = a.q_pos[f.bt];
    if (a.idx) f.ncomp = a.cnt ? a.cnt[f.bt] : a.k;
    else f.ncomp = visible_count(f.t, a.m, a.E);
    int64_t p0 = f.t - a.n_win + 1;
    if (p0 < 0) p0 = 0;
    f.p0 = p0;
    const int64_t nwin = a.n_win > 0 ? f.t - p0 + 1 : 0;
    f.total = f.ncomp + (nwin > 0 ? nwin : 0);
    const int nt = (int)((f.total + 63) / 64);
    if (a.chunk_tiles > 0) {
        f.j0 = f.chunk * a.chunk_tiles;
        f.j1 = f.j0 + a.chunk_tiles < nt ? f.j0 + a.chunk_tiles : nt;
        if (f.j0 > f.j1) f.j0 = f.j1;
    } else {
        f.j0 = 0;
        f.j1 = nt;
    }
}

// Row pointer of list position pos (nullptr: skipped).  Reports bad input.
// pre: the selected index already loaded for this position, or -2.
__device__ __forceinline__ const __nv_bfloat16 *entry_row(const AttnTcArgs &a, const ItemInfo &f,
                                                          int64_t pos, int C, bool report,
                                                          int32_t pre = -2) {
    if (pos < f.ncomp) {
        int64_t j = a.idx ? (pre != -2 ? (int64_t)pre : (int64_t)a.idx[f.bt * a.k + pos]) : pos;
        if (j >= 0 && j < a.E) return a.kvc + (f.b * a.E + j) * C;
        if (report && (j != -1 || !a.idx)) atomicOr(a.status, ST_BAD_INDEX);
        return nullptr;
    }
    if (pos < f.total) {
        const int64_t row = f.p0 + (pos - f.ncomp) - a.raw_pos0[f.b];
        if (row >= 0 && row < a.L) return a.kv_raw + (f.b * a.L + row) * C;
        if (report) atomicOr(a.status, ST_NO_WINDOW_ROW);
    }
    return nullptr;
}

__device__ __forceinline__ int swz128(int row, int byte) {   // within a 1024-byte atom group
    return (row & 7) * 128 + ((((byte >> 4) ^ row) & 7) << 4) + (byte & 15);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
        "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]),
        "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]),
        "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

template <int C>
__global__ void __launch_bounds__(256, 1) attn_tc_kernel(const __grid_constant__ AttnTcArgs a) {
    using Cfg = AtCfg<C>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *sK = smem + Cfg::OFF_K;
    uint8_t *sQ = smem + Cfg::OFF_Q;
    uint8_t *sP = smem + Cfg::OFF_P;
    float *stage = (float *)(smem + Cfg::OFF_STAGE);
    uint8_t *misc = smem + Cfg::OFF_MISC;
    uint64_t *bar = (uint64_t *)misc;                  // 16 barriers
    uint64_t *kfull = bar + 0, *kempty = bar + 2, *sfull = bar + 4, *sempty = bar + 6;
    uint64_t *pfull = bar + 8, *pempty = bar + 10;
    uint64_t *qfull = bar + 12, *qempty = bar + 13, *ofull = bar + 14, *oempty = bar + 15;
    uint32_t *tmem_slot = (uint32_t *)(misc + 128);
    volatile int *abort_flag = (volatile int *)(misc + 132);
    volatile int *rescale_flag = (volatile int *)(misc + 136);
    float *alpha_s = (float *)(misc + 256);            // [64]
    float *den_s = (float *)(misc + 512);              // [64]
    float *cs_s = (float *)(misc + 768);               // [64] cos, then sin
    const __nv_bfloat16 **rowp = (const __nv_bfloat16 **)(misc + 1024);   // [2][64]
    uint8_t *valid = misc + 2048;                      // [2][64] entry present

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    if ((tc::smem_u32(smem) & 1023u) != 0) {            // the layout needs 1024-byte alignment
        if (threadIdx.x == 0) atomicOr(a.status, ST_TIMEOUT);
        return;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) {
            tc::mbar_init(&kfull[i], 96);
            tc::mbar_init(&kempty[i], 1);
            tc::mbar_init(&sfull[i], 1);
            tc::mbar_init(&sempty[i], 4);
            tc::mbar_init(&pfull[i], 1);
            tc::mbar_init(&pempty[i], 1);
        }
        tc::mbar_init(qfull, 96);
        tc::mbar_init(qempty, 1);
        tc::mbar_init(ofull, 1);
        tc::mbar_init(oempty, 4);
        *abort_flag = 0;
        *rescale_flag = 0;
        tc::fence_barrier_init();
    }
    if (warp == 3) tc::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp < 3) {
        // ------------------------------------------------------ loader / q~ prep
        constexpr int NL = 96;           // loader threads
        const int tid = threadIdx.x;     // 0..95
        const uint32_t qb = tc::smem_u32(sQ);
        uint32_t g = 0, ii = 0;          // ii counts processed (non-empty) items
        for (int64_t it = blockIdx.x; it < a.n_items; it += G) {
            ItemInfo f;
            item_info(a, it, f);
            if (f.j0 >= f.j1) continue;
            // q rows -> the K-major swizzled layout [NA][64 heads][128 B] by cp.async
            tc::mbar_wait(qempty, (ii & 1) ^ 1, a.status, abort_flag);
            const int h0 = f.hg * Cfg::HG;
            for (int i = tid; i < Cfg::HG * Cfg::NA * 8; i += NL) {
                const int h = i / (Cfg::NA * 8);
                const int gr = i % (Cfg::NA * 8);           // 16-byte granule of the row
                const uint32_t dst = qb + (gr >> 3) * (Cfg::HG * 128) + (h >> 3) * 1024 + swz128(h, (gr & 7) * 16);
                const bool ok = h0 + h < a.H;
                cp_async16(dst, ok ? (const void *)(a.q + (f.bt * a.H + h0 + h) * (int64_t)C + gr * 8)
                                   : (const void *)a.q, ok ? 16u : 0u);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
            if (tid < a.rope.pairs && tid < 32) {
                float cs, sn;
                rope_cos_sin((double)f.t, a.rope.w[tid], cs, sn);
                cs_s[tid] = cs;
                cs_s[32 + tid] = sn;
            }
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            named_bar(2, NL);
            // q~ = RoPE(q, t): rotate the rotary pairs in place
            for (int i = tid; i < Cfg::HG * a.rope.pairs; i += NL) {
                const int h = i / a.rope.pairs, pi = i % a.rope.pairs;
                const int d = a.rope.first + 2 * pi;
                __nv_bfloat162 *pv = (__nv_bfloat162 *)(sQ + (d >> 6) * (Cfg::HG * 128) + (h >> 3) * 1024 +
                                                        swz128(h, (d & 63) * 2));
                const float2 x = __bfloat1622float2(*pv);
                const float c_ = cs_s[pi], s_ = cs_s[32 + pi];
                *pv = __floats2bfloat162_rn(x.x * c_ - x.y * s_, x.x * s_ + x.y * c_);
            }
            fence_proxy_async();
            tc::mbar_arrive(qfull);
            // the first 16 tiles' selected indices, loaded together up front
            int32_t pre[16];
#pragma unroll
            for (int u = 0; u < 16; u++) {
                const int64_t pos = (int64_t)(f.j0 + u) * 64 + tid;
                pre[u] = (a.idx && tid < 64 && f.j0 + u < f.j1 && pos < f.ncomp) ? a.idx[f.bt * a.k + pos] : -1;
            }
            // entry tiles
            for (int j = f.j0; j < f.j1; j++, g++) {
                const int buf = g & 1;
                tc::mbar_wait(&kempty[buf], ((g >> 1) & 1) ^ 1, a.status, abort_flag);
                if (tid < 64) {
                    int32_t jv = -2;                 // -2: not prefetched
#pragma unroll
                    for (int u = 0; u < 16; u++)
                        if (j - f.j0 == u) jv = pre[u];
                    const __nv_bfloat16 *rp = entry_row(a, f, (int64_t)j * 64 + tid, C, true, jv);
                    rowp[buf * 64 + tid] = rp;
                    valid[buf * 64 + tid] = rp != nullptr;
                }
                named_bar(2, NL);
                const uint32_t kb = tc::smem_u32(sK + buf * Cfg::K_BYTES);
                constexpr int GR = C / 8;            // granules per row
#pragma unroll 4
                for (int i = tid; i < Cfg::TE * GR; i += NL) {
                    const int r = i / GR, gr = i % GR;
                    const __nv_bfloat16 *src = rowp[buf * 64 + r];
                    const int atom = gr >> 3;
                    const uint32_t dst = kb + atom * (Cfg::TE * 128) + (r >> 3) * 1024 + swz128(r, (gr & 7) * 16);
                    cp_async16(dst, src ? (const void *)(src + gr * 8) : (const void *)a.kvc, src ? 16u : 0u);
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
                asm volatile("cp.async.wait_group 0;" ::: "memory");
                fence_proxy_async();
                tc::mbar_arrive(&kfull[buf]);
            }
            ii++;
        }
    } else if (warp == 3) {
        // ------------------------------------------------------------- MMA
        if (lane == 0) {
            constexpr uint32_t idQK = tc::idesc_bf16_f32(64, 64);
            constexpr uint32_t idPV = tc::idesc_bf16_f32(128, 64) | (1u << 15);   // A MN-major
            const uint32_t kBase = tc::smem_u32(sK), qBase = tc::smem_u32(sQ), pBase = tc::smem_u32(sP);
            uint32_t g = 0, ii = 0;
            auto issue_pv = [&](uint32_t gp, bool first) {
                const int bp = gp & 1;
                tc::fence_after_sync();
                const uint32_t kb = kBase + bp * Cfg::K_BYTES, pb = pBase + bp * Cfg::P_BYTES;
#pragma unroll
                for (int c = 0; c < Cfg::NC; c++)
#pragma unroll
                    for (int ks = 0; ks < 4; ks++) {
                        const uint64_t ad = desc_sw128(kb + (2 * c) * (Cfg::TE * 128) + ks * 2048,
                                                       Cfg::TE * 128, 1024);
                        const uint64_t bd = desc_sw128(pb + ks * 32, 16, 1024);
                        tc::mma_bf16(tmem + Cfg::O_COL + c * 64, ad, bd, idPV, (first && ks == 0) ? 0u : 1u);
                    }
                tc::mma_commit(&pempty[bp]);
                tc::mma_commit(&kempty[bp]);
            };
            for (int64_t it = blockIdx.x; it < a.n_items; it += G) {
                ItemInfo f;
                item_info(a, it, f);
                if (f.j0 >= f.j1) continue;
                tc::mbar_wait(qfull, ii & 1, a.status, abort_flag);
                const uint32_t gfirst = g;
                const int nt = f.j1 - f.j0;
                // Issue whichever product is ready: PV(j) as soon as P(j) is
                // written (it frees tile j's buffer for the loader), QK(j+1) as
                // soon as tile j+1 has landed.  A fixed order would make each
                // tile's load wait for the previous tile's load.
                int nq = 0, np = 0;
                long long idle = 0;
                while (np < nt) {
                    bool did = false;
                    if (np < nq) {
                        const uint32_t gp = gfirst + np;
                        if (tc::mbar_test(&pfull[gp & 1], (gp >> 1) & 1) &&
                            (np > 0 || tc::mbar_test(oempty, (ii & 1) ^ 1))) {
                            issue_pv(gp, np == 0);
                            np++;
                            did = true;
                        }
                    }
                    if (nq < nt && nq <= np + 1) {
                        const uint32_t gq = gfirst + nq;
                        const int buf = gq & 1;
                        if (tc::mbar_test(&kfull[buf], (gq >> 1) & 1) &&
                            tc::mbar_test(&sempty[buf], ((gq >> 1) & 1) ^ 1)) {
                            tc::fence_after_sync();
                            const uint32_t kb = kBase + buf * Cfg::K_BYTES;
#pragma unroll
                            for (int at = 0; at < Cfg::NA; at++)
#pragma unroll
                                for (int kk = 0; kk < 4; kk++) {
                                    const uint64_t ad = desc_sw128(kb + at * (Cfg::TE * 128) + kk * 32, 16, 1024);
                                    const uint64_t bd = desc_sw128(qBase + at * (Cfg::HG * 128) + kk * 32, 16, 1024);
                                    tc::mma_bf16(tmem + Cfg::S_COL + buf * 64, ad, bd, idQK, (at | kk) != 0);
                                }
                            tc::mma_commit(&sfull[buf]);
                            if (nq == nt - 1) tc::mma_commit(qempty);
                            nq++;
                            did = true;
                        }
                    }
                    if (did) {
                        idle = 0;
                    } else if (++idle > tc::SPIN_LIMIT || ((idle & 1023) == 0 && *abort_flag)) {
                        if (!*abort_flag) atomicOr(a.status, ST_TIMEOUT);
                        *abort_flag = 1;
                        break;
                    }
                }
                g = gfirst + nt;
                tc::mma_commit(ofull);
                ii++;
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------- softmax, rescale, epilogue
        const int st = threadIdx.x - 128;        // 0..127
        const int quarter = warp & 3;
        const int hh = st >> 1, half = st & 1;   // head-major role
        uint32_t g = 0, ii = 0;
        for (int64_t it = blockIdx.x; it < a.n_items; it += G) {
            ItemInfo f;
            item_info(a, it, f);
            if (f.j0 >= f.j1) continue;
            const int h0 = f.hg * Cfg::HG;
            const float zl2 = (h0 + hh < a.H) ? a.sink[h0 + hh] * 1.4426950408889634f : -INFINITY;
            float m_run = a.chunk_tiles > 0 ? -INFINITY : zl2;
            float l_part = 0.f;
            const uint32_t gfirst = g;
            for (int j = f.j0; j < f.j1; j++, g++) {
                const int buf = g & 1;
                tc::mbar_wait(&sfull[buf], (g >> 1) & 1, a.status, abort_flag);
                tc::fence_after_sync();
                float v[64];
                const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + Cfg::S_COL + buf * 64;
                tc::tmem_ld32(ta, v);
                tc::tmem_ld32(ta + 32, v + 32);
                tc::tmem_ld_wait();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&sempty[buf]);
                // the loader's presence flags for this tile (its kfull phase has
                // completed, and cannot advance again before this tile's PV)
                tc::mbar_wait(&kfull[buf], (g >> 1) & 1, a.status, abort_flag);
                if (lane < 16) {
                    const int e = quarter * 16 + lane;
                    const bool ok = valid[buf * 64 + e] != 0;
#pragma unroll
                    for (int h = 0; h < 64; h++) stage[e * Cfg::STAGE_LD + h] = ok ? v[h] * a.scale_log2 : -INFINITY;
                }
                named_bar(1, 128);
                float x[32];
                float mt = -INFINITY;
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    x[i] = stage[(half * 32 + i) * Cfg::STAGE_LD + hh];
                    mt = fmaxf(mt, x[i]);
                }
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
                const float m_new = fmaxf(m_run, mt);
                const bool need = m_new > m_run + 8.0f;
                const float alpha = need ? exp2f(m_run - m_new) : 1.0f;
                if (need) m_run = m_new;
                tc::mbar_wait(&pempty[buf], ((g >> 1) & 1) ^ 1, a.status, abort_flag);
                float ps = 0.f;
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const float p0 = m_run == -INFINITY ? 0.f : exp2f(x[2 * i] - m_run);
                    const float p1 = m_run == -INFINITY ? 0.f : exp2f(x[2 * i + 1] - m_run);
                    ps += p0 + p1;
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                    pk[i] = *reinterpret_cast<uint32_t *>(&h2);
                }
                l_part = l_part * alpha + ps;
                uint8_t *prow = sP + buf * Cfg::P_BYTES + (hh >> 3) * 1024;
#pragma unroll
                for (int c4 = 0; c4 < 4; c4++) {
                    uint4 w4 = make_uint4(pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
                    *reinterpret_cast<uint4 *>(prow + swz128(hh, (half * 4 + c4) * 16)) = w4;
                }
                if (half == 0) alpha_s[hh] = alpha;
                if (need) *rescale_flag = 1;
                fence_proxy_async();
                named_bar(1, 128);
                if (*rescale_flag && g != gfirst) {
                    // O^T was accumulated with the old maxima: scale column h by alpha[h]
                    const uint32_t gp = g - 1;
                    tc::mbar_wait(&pempty[gp & 1], (gp >> 1) & 1, a.status, abort_flag);
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < Cfg::NC; c++) {
                        const uint32_t to = tmem + ((uint32_t)(quarter * 32) << 16) + Cfg::O_COL + c * 64;
                        float o[32];
#pragma unroll
                        for (int hb = 0; hb < 64; hb += 32) {
                            tc::tmem_ld32(to + hb, o);
                            tc::tmem_ld_wait();
#pragma unroll
                            for (int u = 0; u < 32; u++) o[u] *= alpha_s[hb + u];
                            tmem_st32(to + hb, o);
                        }
                    }
                    tmem_st_wait();
                    tc::fence_before_sync();
                }
                named_bar(1, 128);
                if (st == 0) {
                    *rescale_flag = 0;
                    tc::mbar_arrive(&pfull[buf]);
                }
            }
            // item end: denominators
            const float l_tot = l_part + __shfl_xor_sync(0xffffffffu, l_part, 1);
            float den = l_tot;
            if (a.chunk_tiles == 0 && zl2 != -INFINITY) den += exp2f(zl2 - m_run);
            if (half == 0) {
                den_s[hh] = den;
                alpha_s[hh] = m_run;       // reused: final running max
                if (a.chunk_tiles > 0 && h0 + hh < a.H) {
                    a.part_ml[(it * 64 + hh) * 2] = m_run;
                    a.part_ml[(it * 64 + hh) * 2 + 1] = l_tot;
                } else if (a.lse && h0 + hh < a.H) {
                    a.lse[f.bt * a.H + h0 + hh] =
                        den > 0.f ? (m_run + log2f(den)) * 0.6931471805599453f : -INFINITY;
                }
            }
            named_bar(1, 128);
            tc::mbar_wait(ofull, ii & 1, a.status, abort_flag);
            tc::fence_after_sync();
            const int nh = a.H - h0 < 64 ? a.H - h0 : 64;
            for (int c = 0; c < Cfg::NC; c++) {
                const int d = c * 128 + quarter * 32 + lane;
                const uint32_t to = tmem + ((uint32_t)(quarter * 32) << 16) + Cfg::O_COL + c * 64;
                float o[64];
                tc::tmem_ld32(to, o);
                tc::tmem_ld32(to + 32, o + 32);
                tc::tmem_ld_wait();
                if (a.chunk_tiles > 0) {
                    float *po = a.part_o + (it * 64) * (int64_t)C + d;
#pragma unroll
                    for (int h = 0; h < 64; h++)
                        if (h < nh) po[(int64_t)h * C] = o[h];
                    continue;
                }
                float cr = 1.f, sr = 0.f;
                const bool rot = a.derotate && d >= a.rope.first;
                if (rot) rope_cos_sin(-(double)f.t, a.rope.w[(d - a.rope.first) >> 1], cr, sr);
                __nv_bfloat16 *op = a.out + (f.bt * a.H + h0) * (int64_t)C + d;
#pragma unroll
                for (int h = 0; h < 64; h++) {
                    const float dn = den_s[h];
                    float y = dn > 0.f ? o[h] / dn : 0.f;
                    const float yp = __shfl_xor_sync(0xffffffffu, y, 1);
                    if (rot) y = (lane & 1) ? (yp * sr + y * cr) : (y * cr - yp * sr);
                    if (h < nh) op[(int64_t)h * C] = __float2bfloat16_rn(y);
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(oempty);
            ii++;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 3) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

// Split-KV combine: out[bt, h] = sum_c O_c e^(m_c - M) / (e^(z - M) + sum_c l_c e^(m_c - M)),
// chunks in a fixed order, then de-rotation.  One CTA per (query, head).
template <int C>
__global__ void __launch_bounds__(128) attn_combine_kernel(const AttnTcArgs a) {
    __shared__ float s_sc[64], s_red[4];
    __shared__ float s_M, s_den;
    const int64_t bt = blockIdx.x;
    const int h = blockIdx.y;
    const int hg = h / 64, hl = h % 64;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t t = a.q_pos[bt];
    const int64_t base = (bt * a.n_hg + hg) * a.n_chunks;
    const float zl2 = a.sink[h] * 1.4426950408889634f;
    // every chunk's (max, sum) loaded at once, one per thread
    float mc = -INFINITY, lc = 0.f;
    if (tid < a.n_chunks) {
        mc = a.part_ml[((base + tid) * 64 + hl) * 2];
        lc = a.part_ml[((base + tid) * 64 + hl) * 2 + 1];
    }
    float mx = mc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_red[warp] = mx;
    __syncthreads();
    if (tid == 0) s_M = fmaxf(fmaxf(fmaxf(s_red[0], s_red[1]), fmaxf(s_red[2], s_red[3])), zl2);
    __syncthreads();
    const float M = s_M;
    const float sc = (tid < a.n_chunks && mc != -INFINITY) ? exp2f(mc - M) : 0.f;
    if (tid < 64) s_sc[tid] = sc;
    float dl = lc * sc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, o);
    __syncthreads();
    if (lane == 0) s_red[warp] = dl;
    __syncthreads();
    if (tid == 0) {
        float den = s_red[0] + s_red[1] + s_red[2] + s_red[3];
        if (zl2 != -INFINITY) den += exp2f(zl2 - M);
        s_den = den;
    }
    __syncthreads();
    const float den = s_den;
    for (int d = tid * 2; d < C; d += blockDim.x * 2) {
        float y0 = 0.f, y1 = 0.f;
#pragma unroll 4
        for (int c = 0; c < a.n_chunks; c++) {
            const float2 v = *reinterpret_cast<const float2 *>(a.part_o + ((base + c) * 64 + hl) * (int64_t)C + d);
            y0 = fmaf(v.x, s_sc[c], y0);
            y1 = fmaf(v.y, s_sc[c], y1);
        }
        y0 = den > 0.f ? y0 / den : 0.f;
        y1 = den > 0.f ? y1 / den : 0.f;
        if (a.derotate && d >= a.rope.first) {
            float cr, sr;
            rope_cos_sin(-(double)t, a.rope.w[(d - a.rope.first) >> 1], cr, sr);
            const float r0 = y0 * cr - y1 * sr, r1 = y0 * sr + y1 * cr;
            y0 = r0;
            y1 = r1;
        }
        *reinterpret_cast<__nv_bfloat162 *>(a.out + (bt * a.H + h) * (int64_t)C + d) =
            __floats2bfloat162_rn(y0, y1);
    }
    if (a.lse && tid == 0)
        a.lse[bt * a.H + h] = den > 0.f ? (M + log2f(den)) * 0.6931471805599453f : -INFINITY;
}

// ------------------------------------------------------------------- host

int device_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

bool attn_tc_supported(csa_dtype dt, int c) { return dt == CSA_BF16 && c == 512; }

size_t attn_tc_split_bytes(int64_t rows, int H, int c, int n_chunks) {
    const int64_t items = rows * ((H + 63) / 64) * n_chunks;
    return (size_t)items * 64 * c * 4 + (size_t)items * 64 * 2 * 4 + 512;
}

// Number of split-KV chunks for rows of at most max_list entries: enough items
// to cover the GPU, each at least 4 tiles; independent of the batch size when
// rows are few, so a sequence's result does not depend on the batch around it.
int attn_tc_chunks(int64_t rows, int H, int64_t max_list) {
    const int64_t tiles = (max_list + 63) / 64;
    if (rows * ((H + 63) / 64) >= 2 * 148 || tiles <= 4) return 1;
    int64_t ch = (tiles + 7) / 8;          // 8 tiles per chunk
    if (ch > 64) ch = 64;
    return (int)ch;
}

cudaError_t launch_attn_tc(int64_t B, const AttnArgs &g, const int32_t *cnt, int n_chunks,
                           void *split_ws, int max_ctas, cudaStream_t st) {
    if (B * g.Tq == 0) return cudaSuccess;
    AttnTcArgs a;
    a.q = (const __nv_bfloat16 *)g.q;
    a.q_pos = g.q_pos;
    a.kvc = (const __nv_bfloat16 *)g.kvc;
    a.idx = g.idx;
    a.cnt = cnt;
    a.kv_raw = (const __nv_bfloat16 *)g.kv_raw;
    a.raw_pos0 = g.raw_pos0;
    a.sink = g.sink;
    a.out = (__nv_bfloat16 *)g.out;
    a.lse = g.lse;
    a.status = g.status;
    a.T = g.Tq; a.E = g.E; a.L = g.L;
    a.H = g.H; a.k = g.k; a.m = g.m; a.n_win = g.n_win; a.derotate = g.derotate;
    a.n_hg = (g.H + 63) / 64;
    a.scale_log2 = g.scale * 1.4426950408889634f;
    a.rope = g.rope;
    const int64_t max_list = (g.idx ? (int64_t)g.k : g.E) + g.n_win;
    const int64_t rows = B * g.Tq;
    if (n_chunks > 1 && split_ws) {
        a.n_chunks = n_chunks;
        a.chunk_tiles = (int)(((max_list + 63) / 64 + n_chunks - 1) / n_chunks);
        a.part_o = (float *)split_ws;
        a.part_ml = (float *)((char *)split_ws + (size_t)rows * a.n_hg * n_chunks * 64 * 512 * 4);
    } else {
        a.n_chunks = 1;
        a.chunk_tiles = 0;
        a.part_o = nullptr;
        a.part_ml = nullptr;
    }
    a.n_items = rows * a.n_hg * a.n_chunks;
    using Cfg = AtCfg<512>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg::SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int sms = max_ctas > 0 && max_ctas < device_sms() ? max_ctas : device_sms();
    const int grid = (int)(a.n_items < sms ? a.n_items : sms);
    attn_tc_kernel<512><<<grid, Cfg::THREADS, Cfg::SMEM, st>>>(a);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || a.chunk_tiles == 0) return e;
    attn_combine_kernel<512><<<dim3((unsigned)rows, (unsigned)g.H), 128, 0, st>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace csa
