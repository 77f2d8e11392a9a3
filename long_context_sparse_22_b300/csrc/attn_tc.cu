// Core attention on the 5th-generation tensor cores (bf16 in, fp32 in tensor
// memory): shared-KV MQA over a per-query list of entries (selected or
// visible compressed entries, then the window rows) plus a sink logit.
// Head dims c = 512 and c = 128.
//
// [DeepSeek-V4 book ch.6 "Shared key-value MQA"; ch.7 "The sliding window",
// "Partial rotary position embeddings", "Why the output is de-rotated",
// "Attention sinks"; "DeepSeek-V4: Making Million-Token Context an
// Architectural Problem", Key design 1 and 2.]
//
// One work item is (query, group of 64 heads[, split-KV chunk]).  Its list is
// cut into 64-entry tiles: first the compressed slots (padded up to a whole
// tile), then the window rows p0..t (at most two tiles).  Per tile:
//   S[h, e]    = q~[h, :] . K[e, :]             M = 64 heads,  N = 64 entries
//   O^T[d, h] += V[:, d]^T . P^T[:, h]           M = 128 dims (x C/128), N = 64
// K = V is the same tile in shared memory; the second product reads it as an
// MN-major operand.  With heads on the rows of S, every head's logits of a
// tile sit in one thread, so the running max, the exponentials and the sum
// need no cross-thread exchange.  O^T is rescaled in tensor memory only when
// some head's running max grows by more than 2^8 (exact either way, because
// the denominator uses the same max); a barrier reduction tells the four
// softmax warps whether any head needs it.  The sink logit seeds the running
// max and enters only the denominator.
//
// Selected compressed entries are gathered by cp.async, 16 bytes per thread
// and instruction, into the 128-byte-swizzled layout (the tensor-memory
// copy engine's four-row gather sustains only about a fifth of that rate);
// contiguous rows (the window, or every visible entry of the dense variant)
// arrive as 64-row TMA boxes.  Rows that are not part of the list (padding,
// -1 slots, rows past t) are zero-filled or hold finite data, and are masked
// out of the softmax by a per-tile presence mask.
//
// Warp roles (persistent CTAs, items dealt round-robin):
//   warps 0-3  loaders: q tile (box TMA, then RoPE at t in place while the
//              item's first tile loads), the entry tiles (four buffers at
//              c = 128, two at c = 512; q has two at c = 128), the
//              presence masks;
//   warp 4     TMEM allocator and QK issuer (one lane issues);
//   warps 5-8  softmax (a head's 64 logits spread over four threads), the
//              O rescale, and the epilogue: normalise, de-rotate and store
//              straight from registers, a warp writing 64 contiguous bytes
//              of one head's row per instruction (or fp32 partial outputs
//              for a split-KV combine);
//   warp 9     PV issuer (one lane issues).
// Every wait is taken by a whole warp on an mbarrier (with an iteration cap
// after which the kernel records a timeout and unwinds), and waits whose
// phase must already have completed come before the one that can block.
#include "attn_common.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace csa {

template <int C>
struct AtCfg {
    static constexpr int NA = C / 64;             // 64-dim atoms (128-byte rows)
    static constexpr int NC = C / 128;            // 128-dim O^T chunks
    static constexpr int TE = 64;                 // entries per tile
    static constexpr int HG = 64;                 // heads per item
    static constexpr int ATOM = TE * 128;         // one atom of a tile: 64 rows x 128 B
    static constexpr int K_BYTES = NA * ATOM;
    static constexpr int Q_BYTES = NA * HG * 128;
    static constexpr int P_BYTES = HG * 128;      // 64 heads x 64 entries bf16
    // entry-tile buffers and q buffers: at c = 128 a tile is 16 KB, so four
    // tiles and two q tiles stay in flight; at c = 512 (64 KB tiles) two and one
    static constexpr int NKB = C == 128 ? 4 : 2;
    static constexpr int QB = C == 128 ? 2 : 1;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_Q = OFF_K + NKB * K_BYTES;
    static constexpr int OFF_P = OFF_Q + QB * Q_BYTES;
    static constexpr int OFF_MISC = OFF_P + 2 * P_BYTES;
    static constexpr int MISC_BYTES = 8192;       // barriers, masks, scales, angles, row pointers, q gains
    static constexpr int SMEM = OFF_MISC + MISC_BYTES + 1024;   // + alignment slack
    static constexpr int S_COL = 0;               // two S buffers: cols 0, 64
    static constexpr int O_COL = 128;             // O^T chunks: 128 + 64 c
    static constexpr int TMEM_COLS = O_COL + NC * 64 <= 256 ? 256 : 512;   // a power of two
    static constexpr int LOAD_WARPS = 4;          // warps 0-3: loaders
    static constexpr int NLOAD = LOAD_WARPS * 32;
    static constexpr int MMA_WARP = 4;            // warp 4: TMEM allocation, QK issue
    static constexpr int SM_WARP0 = 5;            // warps 5-8: softmax and epilogue
    static constexpr int PV_WARP = 9;             // warp 9: PV issue
    static constexpr int THREADS = (PV_WARP + 1) * 32;
    // one CTA per SM: at c = 128 two CTAs (registers capped at 96) spilled in the
    // softmax and measured slower than one
    static constexpr int MIN_BLOCKS = 1;
};

struct AttnTcArgs {
    const __nv_bfloat16 *kvc;
    const uint8_t *kv8;      // FP8 records of the compressed entries (the KV8 variant), or nullptr
    const void *zsrc;        // any valid 16-byte-aligned address (source of zero-filled copies)
    const int64_t *q_pos;
    const int32_t *idx;      // [B,T,k] or nullptr: every visible entry
    const int32_t *cnt;      // [B,T] kept count of idx rows, or nullptr (use k)
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
    long long spin;          // polls before a wait between roles gives up
    const float *q_norm;     // RMSNorm gains of q (C floats) or nullptr
    float norm_eps;
    float scale_log2;        // logit scale * log2(e)
    RopeFreqs rope;
};

struct ItemInfo {
    int64_t bt, b, t;        // first query row of the item, its sequence, its largest position
    int64_t tmin;            // smallest query position of the item
    int hg, chunk;
    int64_t ncomp;           // compressed slots (tiles 0 .. ntc-1)
    int64_t p0, nwin;        // window rows p0 .. p0+nwin-1 (tiles ntc ..)
    int ntc, nt;             // compressed tiles, all tiles
    int j0, j1;              // tile range of this item
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
    f.tmin = f.t;
    if (a.idx) f.ncomp = a.cnt ? a.cnt[f.bt] : a.k;
    else f.ncomp = visible_count(f.t, a.m, a.E);
    if (f.ncomp < 0) f.ncomp = 0;
    int64_t p0 = f.tmin - a.n_win + 1;
    if (p0 < 0) p0 = 0;
    f.p0 = p0;
    f.nwin = a.n_win > 0 && f.t >= 0 ? f.t - p0 + 1 : 0;
    f.ntc = (int)((f.ncomp + 63) / 64);
    f.nt = f.ntc + (int)((f.nwin + 63) / 64);
    if (a.chunk_tiles > 0) {
        f.j0 = f.chunk * a.chunk_tiles;
        f.j1 = f.j0 + a.chunk_tiles < f.nt ? f.j0 + a.chunk_tiles : f.nt;
        if (f.j0 > f.j1) f.j0 = f.j1;
    } else {
        f.j0 = 0;
        f.j1 = f.nt;
    }
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
                 : "memory");
}

// 16 E4M3 codes times their group scale -> two 16-byte chunks of 8 bf16 each
// (the code is exact in f16; the scaled value is rounded once to bf16).
__device__ __forceinline__ void fp8x16_to_bf16(const uint4 g, float sc, uint32_t *o) {
    const uint32_t w[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int q = 0; q < 4; q++)
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
            const uint16_t pair = (uint16_t)(w[q] >> (16 * hh));
            uint32_t h2;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(f.x * sc, f.y * sc);
            o[2 * q + hh] = *reinterpret_cast<const uint32_t *>(&b2);
        }
}

__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

template <int C, bool KV8>
__global__ void __launch_bounds__(AtCfg<C>::THREADS, AtCfg<C>::MIN_BLOCKS)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c,
               const __grid_constant__ CUtensorMap tm_w,
               const __grid_constant__ AttnTcArgs a) {
    using Cfg = AtCfg<C>;
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
    uint32_t *vmask32 = (uint32_t *)(misc + 272);      // [NKB buffers][2 halves] presence bits
    float *alpha_s = (float *)(misc + 512);            // [2][64]
    float *inv_den_s = (float *)(misc + 1024);         // [64]
    float *cs_s = (float *)(misc + 2048);              // [2][256]: cos, sin of the query angle
    const __nv_bfloat16 **rowp = (const __nv_bfloat16 **)(misc + 4096);   // [NKB][64] gathered rows
    float *gain_s = (float *)(misc + 6144);            // [C] RMSNorm gains of q

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
    if (warp == Cfg::MMA_WARP) tc::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    if (a.q_norm)
        for (int i = threadIdx.x; i < C; i += Cfg::THREADS) gain_s[i] = a.q_norm[i];
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp < Cfg::LOAD_WARPS) {
        // ------------------------------------------------------------ loaders
        const int tid = threadIdx.x;                     // 0 .. NLOAD-1
        const uint32_t kb0 = tc::smem_u32(sK);
        uint32_t g = 0, ii = 0;
        uint32_t tma_issued = 0, last_g[Cfg::NKB] = {}, q_pending = 0, q_pend_b = 0, q_pend_par = 0;
        // FP8 records of the next gathered tile, loaded while the current one is
        // converted and multiplied (within an item)
        uint4 pf8[KV8 ? 14 : 1], pf16[KV8 ? 4 : 1], pfs = make_uint4(0, 0, 0, 0);
        bool pf = false;
        uint32_t pf_bal = 0;
        bool ok = true;
        for (int64_t it = blockIdx.x; ok && it < a.n_items; it += G) {
            ItemInfo f;
            item_info(a, it, f);
            if (f.j0 >= f.j1) continue;
            // q rows of the next item on their way to L2 while this one runs
            if (it + G < a.n_items && tid < Cfg::NA) {
                ItemInfo fn;
                item_info(a, it + G, fn);
                const int y = (int)(fn.bt * a.H + fn.hg * Cfg::HG);
                asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                                 reinterpret_cast<uint64_t>(&tm_q)),
                             "r"(tid * 64), "r"(y)
                             : "memory");
            }
            // the cos / sin of this item's angle and its first selected indices,
            // worked out while the previous item's last QK still reads q
            for (int i = tid; i < a.rope.pairs; i += Cfg::NLOAD) {
                float c_, s_;
                rope_cos_sin(a.rope, f.t, i, c_, s_);
                cs_s[i] = c_;
                cs_s[256 + i] = s_;
            }
            int32_t iv = -1;                     // selected index of this thread's slot, next tile
            if (a.idx && tid < 64 && f.j0 < f.ntc) {
                const int64_t pos = (int64_t)f.j0 * 64 + tid;
                iv = pos < f.ncomp ? a.idx[f.bt * a.k + pos] : -1;
            }
            // this item's q rows (box TMA).  Waits are warp-uniform and the four
            // loader warps agree on a failure through a barrier reduction, so none
            // is left at a named barrier; the barrier also publishes cs_s.
            const int qb = (int)(ii % Cfg::QB);
            const uint32_t qpar = (ii / Cfg::QB) & 1;
            uint8_t *sQb = sQ + qb * Cfg::Q_BYTES;
            if (named_bar_or(2, Cfg::NLOAD, !warp_wait(&qempty[qb], qpar ^ 1, a.status, abort_flag, a.spin))) {
                ok = false;
                break;
            }
            if (tid == 0) {
                tc::mbar_expect_tx(&qland[qb], Cfg::Q_BYTES);
                for (int at = 0; at < Cfg::NA; at++)
                    tc::tma_load_2d(sQb + at * (Cfg::HG * 128), &tm_q, at * 64,
                                    (int)(f.bt * a.H + f.hg * Cfg::HG), &qland[qb]);
                q_pending = 1;
                q_pend_b = qb;
                q_pend_par = qpar;
            }
            // q~ = RoPE(q, t): once q has landed, rotate the rotary pairs in place and
            // hand q to the MMA.  Runs while the item's first tile is in flight.
            auto rope_q = [&]() -> bool {
                if (named_bar_or(2, Cfg::NLOAD, !warp_wait(&qland[qb], qpar, a.status, abort_flag, a.spin)))
                    return false;
                if (tid == 0) q_pending = 0;
                if (a.q_norm) {
                    // RMSNorm of each head's row before its rotation: two threads per
                    // head (adjacent lanes), each over half of the row's 16-byte chunks
                    const int h = tid >> 1, hf = tid & 1;
                    constexpr int CH = C / 16;           // chunks per half row
                    uint8_t *hb = sQb + (h >> 3) * 1024;
                    float ss = 0.f;
#pragma unroll 4
                    for (int k = 0; k < CH; k++) {
                        const int d0 = (hf * CH + k) * 8;
                        const uint4 u = *reinterpret_cast<const uint4 *>(hb + (d0 >> 6) * (Cfg::HG * 128) +
                                                                         swz128(h, (d0 & 63) * 2));
                        float f[8];
                        Vec<__nv_bfloat16>::unpack(u, f);
#pragma unroll
                        for (int e = 0; e < 8; e++) ss = fmaf(f[e], f[e], ss);
                    }
                    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                    const float rs = 1.0f / sqrtf(ss / (float)C + a.norm_eps);
#pragma unroll 4
                    for (int k = 0; k < CH; k++) {
                        const int d0 = (hf * CH + k) * 8;
                        uint4 *pu = reinterpret_cast<uint4 *>(hb + (d0 >> 6) * (Cfg::HG * 128) +
                                                              swz128(h, (d0 & 63) * 2));
                        float f[8];
                        Vec<__nv_bfloat16>::unpack(*pu, f);
#pragma unroll
                        for (int e = 0; e < 8; e++) f[e] = f[e] * rs * gain_s[d0 + e];
                        uint4 o;
                        __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
                        for (int e = 0; e < 4; e++) o2[e] = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
                        *pu = o;
                    }
                    named_bar(2, Cfg::NLOAD);
                }
                const int np = a.rope.pairs;
                if (np == 32) {
                    // one pair per lane, heads warp, warp + 4, ...: all loads in flight at once
                    const int d = a.rope.first + 2 * lane;
                    uint8_t *qa = sQb + (d >> 6) * (Cfg::HG * 128);
                    __nv_bfloat162 x[Cfg::HG / 4];
#pragma unroll
                    for (int k = 0; k < Cfg::HG / 4; k++) {
                        const int h = warp + 4 * k;
                        x[k] = *(const __nv_bfloat162 *)(qa + (h >> 3) * 1024 + swz128(h, (d & 63) * 2));
                    }
#pragma unroll
                    for (int k = 0; k < Cfg::HG / 4; k++) {
                        const int h = warp + 4 * k;
                        const int ci = lane;
                        const float c_ = cs_s[ci], s_ = cs_s[256 + ci];
                        const float2 v = __bfloat1622float2(x[k]);
                        *(__nv_bfloat162 *)(qa + (h >> 3) * 1024 + swz128(h, (d & 63) * 2)) =
                            __floats2bfloat162_rn(v.x * c_ - v.y * s_, v.x * s_ + v.y * c_);
                    }
                } else {
                    for (int i = tid; i < Cfg::HG * np; i += Cfg::NLOAD) {
                        const int h = i / np, pi = i - h * np;
                        const int d = a.rope.first + 2 * pi;
                        __nv_bfloat162 *pv = (__nv_bfloat162 *)(sQb + (d >> 6) * (Cfg::HG * 128) +
                                                                (h >> 3) * 1024 + swz128(h, (d & 63) * 2));
                        const float2 v = __bfloat1622float2(*pv);
                        const int ci = pi;
                        const float c_ = cs_s[ci], s_ = cs_s[256 + ci];
                        *pv = __floats2bfloat162_rn(v.x * c_ - v.y * s_, v.x * s_ + v.y * c_);
                    }
                }
                fence_proxy_async();
                named_bar(2, Cfg::NLOAD);
                if (tid == 0) tc::mbar_arrive(&qfull[qb]);
                return true;
            };
            for (int j = f.j0; j < f.j1; j++, g++) {
                const int buf = (int)(g % Cfg::NKB);
                const uint32_t kpar = (g / Cfg::NKB) & 1;
                // compressed tiles are gathered row by row: selected entries, and with
                // FP8 entries every compressed tile (its rows are dequantised here)
                const bool gather = j < f.ntc && (a.idx || KV8);
                // a gathered tile's row addresses go to shared memory before the wait
                // for its buffer (the barrier that ends the wait publishes them; the
                // gather NKB tiles back, the last reader of this slot, has been issued)
                uint32_t bal = pf ? pf_bal : 0u;
                if (gather && tid < 64 && !pf) {
                    const int64_t pos = (int64_t)j * 64 + tid;
                    const bool in = pos < f.ncomp;
                    const int64_t ent = a.idx ? (int64_t)iv : pos;
                    const bool v = in && ent >= 0 && ent < a.E;
                    if (a.idx && in && !v && iv != -1) atomicOr(a.status, ST_BAD_INDEX);
                    if constexpr (KV8)
                        rowp[buf * 64 + tid] = v ? reinterpret_cast<const __nv_bfloat16 *>(
                                                       a.kv8 + (f.b * a.E + ent) * (int64_t)KV8_BYTES)
                                                 : nullptr;
                    else
                        rowp[buf * 64 + tid] = v ? a.kvc + (f.b * a.E + ent) * (int64_t)C : nullptr;
                    bal = __ballot_sync(0xffffffffu, v);
                }
                if (named_bar_or(2, Cfg::NLOAD,
                                 !warp_wait(&kempty[buf], kpar ^ 1, a.status, abort_flag, a.spin))) {
                    ok = false;
                    break;
                }
                const uint32_t kb = kb0 + buf * Cfg::K_BYTES;
                if (gather) {
                    // gather of selected entries: cp.async, 16 bytes per thread and instruction;
                    // the presence mask is written once the softmax NKB tiles back is done with it
                    if (tid < 64 && lane == 0) vmask32[buf * 2 + warp] = bal;
                    // the next tile's selected indices, fetched while this one loads
                    if (a.idx && tid < 64 && j + 1 < f.j1 && j + 1 < f.ntc) {
                        const int64_t pos = (int64_t)(j + 1) * 64 + tid;
                        iv = pos < f.ncomp ? a.idx[f.bt * a.k + pos] : -1;
                    }
                    if constexpr (KV8) {
                        // FP8 records: two threads per row, each loading 14 granules of
                        // codes, 4 of rotary BF16 values and the group scales, then writing
                        // the row's bf16 chunks into the swizzled tile (zeros for rows
                        // that are not in the list)
                        const int r = tid >> 1, half = tid & 1;
                        auto load_rows = [&](int bsel) {
                            const uint8_t *src = reinterpret_cast<const uint8_t *>(rowp[bsel * 64 + r]);
#pragma unroll
                            for (int q = 0; q < 14; q++)
                                pf8[q] = src ? ld_nc_v4(src + (half * 14 + q) * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
                            for (int q = 0; q < 4; q++)
                                pf16[q] = src ? ld_nc_v4(src + KV8_NR + (half * 4 + q) * 16) : make_uint4(0, 0, 0, 0);
                            pfs = src ? ld_nc_v4(src + KV8_NR + 128) : make_uint4(0, 0, 0, 0);
                        };
                        if (!pf) load_rows(buf);
                        pf = false;
                        if (j == f.j0 && !rope_q()) {
                            ok = false;
                            break;
                        }
                        const float scl[4] = {__uint_as_float(pfs.x), __uint_as_float(pfs.y),
                                              __uint_as_float(pfs.z), __uint_as_float(pfs.w)};
                        uint4 *g8 = pf8, *g16 = pf16;
                        const uint32_t rb = kb + (r >> 3) * 1024;
#pragma unroll
                        for (int q = 0; q < 14; q++) {
                            const int gidx = half * 14 + q;      // dims 16 gidx .. 16 gidx + 15
                            uint32_t o[8];
                            fp8x16_to_bf16(g8[q], scl[gidx >> 3], o);
                            const uint32_t ab = rb + (gidx >> 2) * Cfg::ATOM;
                            const int c0 = (gidx & 3) * 2;
                            sts_v4(ab + swz128(r, c0 * 16), o[0], o[1], o[2], o[3]);
                            sts_v4(ab + swz128(r, (c0 + 1) * 16), o[4], o[5], o[6], o[7]);
                        }
#pragma unroll
                        for (int q = 0; q < 4; q++)      // dims 448 + 8 k .. : chunk k of the last atom
                            sts_v4(rb + (Cfg::NA - 1) * Cfg::ATOM + swz128(r, (half * 4 + q) * 16), g16[q].x,
                                   g16[q].y, g16[q].z, g16[q].w);
                        fence_proxy_async();
                        tc::mbar_arrive(&kfull[buf]);
                        if (j + 1 < f.j1 && j + 1 < f.ntc) {
                            // the next gathered tile: its row addresses into the other slot
                            // (its last reader, two tiles back, has finished), its presence
                            // bits kept, its records on their way into registers
                            const int nb = (int)((g + 1) % Cfg::NKB);
                            if (tid < 64) {
                                const int64_t pos = (int64_t)(j + 1) * 64 + tid;
                                const bool in = pos < f.ncomp;
                                const int64_t ent = a.idx ? (int64_t)iv : pos;
                                const bool v = in && ent >= 0 && ent < a.E;
                                if (a.idx && in && !v && iv != -1) atomicOr(a.status, ST_BAD_INDEX);
                                rowp[nb * 64 + tid] = v ? reinterpret_cast<const __nv_bfloat16 *>(
                                                              a.kv8 + (f.b * a.E + ent) * (int64_t)KV8_BYTES)
                                                        : nullptr;
                                pf_bal = __ballot_sync(0xffffffffu, v);
                            }
                            named_bar(2, Cfg::NLOAD);
                            load_rows(nb);
                            pf = true;
                        }
                        continue;
                    }
                    constexpr int GR = C / 8;            // 16-byte granules per row
                    const int gr = tid % GR;
                    const uint32_t dcol = (gr >> 3) * Cfg::ATOM;
#pragma unroll 8
                    for (int r = tid / GR; r < Cfg::TE; r += Cfg::NLOAD / GR) {
                        const __nv_bfloat16 *src = rowp[buf * 64 + r];
                        const uint32_t dst = kb + dcol + (r >> 3) * 1024 + swz128(r, (gr & 7) * 16);
                        cp_async16(dst, src ? (const void *)(src + gr * 8) : a.zsrc, src ? 16u : 0u);
                    }
                    asm volatile("cp.async.commit_group;" ::: "memory");
                    if (j == f.j0 && !rope_q()) {
                        ok = false;
                        break;
                    }
                    asm volatile("cp.async.wait_group 0;" ::: "memory");
                    fence_proxy_async();
                    tc::mbar_arrive(&kfull[buf]);
                } else {
                    // contiguous rows (every visible entry, or the window) as 64-row boxes
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
                        const int64_t rp0 = a.raw_pos0[f.b];
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
                        for (int at = 0; at < Cfg::NA; at++)
                            tc::tma_load_2d(sK + buf * Cfg::K_BYTES + at * Cfg::ATOM, j < f.ntc ? &tm_c : &tm_w,
                                            at * 64, (int)y, &kfull[buf]);
                        tma_issued |= 1u << buf;
                        last_g[buf] = g;
                    } else {
                        tc::mbar_arrive(&kfull[buf]);
                    }
                    if (j == f.j0 && !rope_q()) {
                        ok = false;
                        break;
                    }
                }
            }
            ii++;
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
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
    } else if (warp == Cfg::MMA_WARP || warp == Cfg::PV_WARP) {
        // --------------------------------------------------------------- MMA
        // Two issuing warps: QK on warp 4, PV on warp 9.  The whole warp runs
        // the loop and waits on the barriers; one lane issues the MMAs and
        // commits.  A tcgen05.mma of these small shapes costs more to issue
        // than to execute, so the two streams are issued side by side; the
        // barriers order them.
        {
            const bool is_qk = warp == Cfg::MMA_WARP;
            const bool leader = lane == 0;
            constexpr uint32_t idQK = tc::idesc_bf16_f32(64, 64);
            constexpr uint32_t idPV = tc::idesc_bf16_f32(128, 64) | (1u << 15);   // A MN-major
            // descriptors at the buffer bases; a byte offset o adds o >> 4
            const uint64_t dq0 = desc_sw128(tc::smem_u32(sQ), 16, 1024);
            const uint64_t dk0 = desc_sw128(tc::smem_u32(sK), 16, 1024);
            const uint64_t dv0 = desc_sw128(tc::smem_u32(sK), Cfg::ATOM, 1024);
            const uint64_t dp[2] = {desc_sw128(tc::smem_u32(sP), 16, 1024),
                                    desc_sw128(tc::smem_u32(sP + Cfg::P_BYTES), 16, 1024)};
            uint32_t g = 0, ii = 0;
            bool ok = true;
            for (int64_t it = blockIdx.x; ok && it < a.n_items; it += G) {
                ItemInfo f;
                item_info(a, it, f);
                if (f.j0 >= f.j1) continue;
                const int nt = f.j1 - f.j0;
                if (is_qk) {
                    const int qb = (int)(ii % Cfg::QB);
                    if (!warp_wait(&qfull[qb], (ii / Cfg::QB) & 1, a.status, abort_flag, a.spin)) break;
                    const uint64_t dq = dq0 + (uint64_t)((qb * Cfg::Q_BYTES) >> 4);
                    for (int n = 0; n < nt; n++) {
                        const uint32_t gq = g + n;
                        const int buf = gq & 1;                         // S buffer
                        const int kbuf = (int)(gq % Cfg::NKB);         // entry tile
                        if (!warp_wait(&kfull[kbuf], (gq / Cfg::NKB) & 1, a.status, abort_flag, a.spin) ||
                            !warp_wait(&sempty[buf], ((gq >> 1) & 1) ^ 1, a.status, abort_flag, a.spin)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        if (leader) {
#pragma unroll
                            for (int at = 0; at < Cfg::NA; at++)
#pragma unroll
                                for (int kk = 0; kk < 4; kk++)
                                    tc::mma_bf16(tmem + Cfg::S_COL + buf * 64,
                                                 dq + (uint64_t)((at * (Cfg::HG * 128) + kk * 32) >> 4),
                                                 dk0 + (uint64_t)((kbuf * Cfg::K_BYTES + at * Cfg::ATOM + kk * 32) >> 4), idQK,
                                                 (at | kk) != 0);
                            tc::mma_commit(&sfull[buf]);
                            if (n == nt - 1) tc::mma_commit(&qempty[qb]);
                        }
                        __syncwarp();
                    }
                } else {
                    for (int n = 0; n < nt; n++) {
                        const uint32_t gp = g + n;
                        const int bp = gp & 1;                          // P buffer
                        const int kbuf = (int)(gp % Cfg::NKB);         // entry tile (V)
                        if (!warp_wait(&pfull[bp], (gp >> 1) & 1, a.status, abort_flag, a.spin) ||
                            (n == 0 && !warp_wait(oempty, (ii & 1) ^ 1, a.status, abort_flag, a.spin))) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        if (leader) {
#pragma unroll
                            for (int c = 0; c < Cfg::NC; c++)
#pragma unroll
                                for (int ks = 0; ks < 4; ks++)
                                    tc::mma_bf16(tmem + Cfg::O_COL + c * 64,
                                                 dv0 + (uint64_t)((kbuf * Cfg::K_BYTES + (2 * c) * Cfg::ATOM + ks * 2048) >> 4),
                                                 dp[bp] + (uint64_t)((ks * 32) >> 4), idPV,
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
        }
    } else {
        // ------------------------------------------- softmax, rescale, epilogue
        // Waits are warp-uniform, and a failed wait never skips a named
        // barrier: the four warps agree on failure through a barrier
        // reduction and leave together.
        const int st = threadIdx.x - Cfg::SM_WARP0 * 32;   // 0 .. 127
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        // S rows (heads) of an M = 64 product sit in TMEM lanes 0-15 of each
        // quarter.  A 16x256b load spreads them over the whole warp: thread
        // t holds heads r = 16*quarter + t/4 and r + 8, entries 8i + 2(t%4)
        // and 8i + 2(t%4) + 1 for i = 0..7.  The four threads of a head
        // agree on its running max by two shuffles; the running sums stay
        // per-thread until the item ends.
        const int t4 = lane & 3;
        const int hr[2] = {quarter * 16 + (lane >> 2), quarter * 16 + (lane >> 2) + 8};
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        uint32_t g = 0, ii = 0;
        ItemInfo fn;                             // the next item, worked out during the last PV
        bool have_fn = false;
        int zl_hg = -1;                          // head group whose sink logits zl2 holds
        float zl2[2] = {-INFINITY, -INFINITY};
        for (int64_t it = blockIdx.x; it < a.n_items; it += G) {
            ItemInfo f;
            if (have_fn) f = fn;
            else item_info(a, it, f);
            have_fn = false;
            if (f.j0 >= f.j1) continue;
            const int h0 = f.hg * Cfg::HG;
            bool real[2];
            float m_run[2], l_run[2];
#pragma unroll
            for (int u = 0; u < 2; u++) {
                real[u] = h0 + hr[u] < a.H;
                if (f.hg != zl_hg) zl2[u] = real[u] ? a.sink[h0 + hr[u]] * 1.4426950408889634f : -INFINITY;
                m_run[u] = a.chunk_tiles > 0 ? -INFINITY : zl2[u];
                l_run[u] = 0.f;
            }
            zl_hg = f.hg;
            const uint32_t gfirst = g;
            bool fail = false;
            for (int j = f.j0; j < f.j1; j++, g++) {
                const int buf = g & 1;                   // S and P buffers
                const uint32_t par = (g >> 1) & 1;
                const int kbuf = (int)(g % Cfg::NKB);   // entry tile
                const uint32_t kpar = (g / Cfg::NKB) & 1;
                // the loaders' presence mask for this tile (its kfull phase has
                // completed and cannot advance again before this tile's PV) and the
                // P buffer (the PV of two tiles back has read it): both are ready
                // before this tile's logits, so they are checked first
                bool ok = warp_wait(&kfull[kbuf], kpar, a.status, abort_flag, a.spin) &&
                          warp_wait(&pempty[buf], par ^ 1, a.status, abort_flag, a.spin);
                const uint32_t mlo = ok ? vmask32[kbuf * 2] : 0u, mhi = ok ? vmask32[kbuf * 2 + 1] : 0u;
                ok = ok && warp_wait(&sfull[buf], par, a.status, abort_flag, a.spin);
                uint32_t raw[32];
                if (ok) {
                    tc::fence_after_sync();
                    asm volatile(
                        "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
                        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                        : "=r"(raw[0]), "=r"(raw[1]), "=r"(raw[2]), "=r"(raw[3]), "=r"(raw[4]), "=r"(raw[5]),
                          "=r"(raw[6]), "=r"(raw[7]), "=r"(raw[8]), "=r"(raw[9]), "=r"(raw[10]), "=r"(raw[11]),
                          "=r"(raw[12]), "=r"(raw[13]), "=r"(raw[14]), "=r"(raw[15]), "=r"(raw[16]), "=r"(raw[17]),
                          "=r"(raw[18]), "=r"(raw[19]), "=r"(raw[20]), "=r"(raw[21]), "=r"(raw[22]), "=r"(raw[23]),
                          "=r"(raw[24]), "=r"(raw[25]), "=r"(raw[26]), "=r"(raw[27]), "=r"(raw[28]), "=r"(raw[29]),
                          "=r"(raw[30]), "=r"(raw[31])
                        : "r"(tmem + lane_base + Cfg::S_COL + buf * 64));
                    tc::tmem_ld_wait();
                    tc::tmem_regs_ready<32>(raw);
                }
                // v[u][2i + e]: head hr[u], entry 8i + 2 t4 + e  (raw[4i + 2u + e])
                float v[2][16];
#pragma unroll
                for (int i = 0; i < 8; i++)
#pragma unroll
                    for (int e = 0; e < 2; e++) {
                        const int ent = 8 * i + 2 * t4 + e;
                        const uint32_t bit = i < 4 ? (mlo >> ent) & 1u : (mhi >> (ent - 32)) & 1u;
#pragma unroll
                        for (int u = 0; u < 2; u++)
                            v[u][2 * i + e] = bit ? __uint_as_float(raw[4 * i + 2 * u + e]) * a.scale_log2 : -INFINITY;
                    }
                bool need[2];
                float alpha[2];
#pragma unroll
                for (int u = 0; u < 2; u++) {
                    float mx = fmaxf(fmaxf(fmaxf(v[u][0], v[u][1]), fmaxf(v[u][2], v[u][3])),
                                     fmaxf(fmaxf(v[u][4], v[u][5]), fmaxf(v[u][6], v[u][7])));
                    mx = fmaxf(mx, fmaxf(fmaxf(fmaxf(v[u][8], v[u][9]), fmaxf(v[u][10], v[u][11])),
                                         fmaxf(fmaxf(v[u][12], v[u][13]), fmaxf(v[u][14], v[u][15]))));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    const float m_new = fmaxf(m_run[u], mx);
                    need[u] = real[u] && m_new > m_run[u] + 8.0f;
                    alpha[u] = need[u] ? ex2(m_run[u] - m_new) : 1.0f;
                    if (need[u]) m_run[u] = m_new;
                }
                // P rows (bf16): this thread's two entries of chunk i are 4 bytes
                // at byte 4 t4 of the row's (swizzled) 16-byte chunk i
#pragma unroll
                for (int u = 0; u < 2; u++) {
                    const int h = hr[u];
                    const float msub = m_run[u] == -INFINITY ? 0.f : m_run[u];
                    uint8_t *prow = sP + buf * Cfg::P_BYTES + (h >> 3) * 1024 + (h & 7) * 128 + 4 * t4;
                    float ps = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const float p0 = ex2(v[u][2 * i] - msub), p1 = ex2(v[u][2 * i + 1] - msub);
                        ps += p0 + p1;
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                        if (ok) *reinterpret_cast<uint32_t *>(prow + ((i ^ (h & 7)) << 4)) =
                            *reinterpret_cast<uint32_t *>(&h2);
                    }
                    l_run[u] = l_run[u] * alpha[u] + ps;
                    if (ok && t4 == 0) alpha_s[buf * 64 + h] = alpha[u];
                }
                fence_proxy_async();
                // one barrier in the common case: nothing failed, no head needs a rescale
                const bool resc = (need[0] || need[1]) && g != gfirst;
                if (named_bar_or(1, 128, !ok || resc)) {
                    if (named_bar_or(1, 128, !ok)) { fail = true; break; }
                    // some head's max grew: O^T was accumulated with older maxima,
                    // scale column h by alpha[h]
                    const uint32_t gp = g - 1;
                    if (warp_wait(&pempty[gp & 1], (gp >> 1) & 1, a.status, abort_flag, a.spin)) {
                        tc::fence_after_sync();
                        const float *al = alpha_s + buf * 64;
#pragma unroll 1
                        for (int cb = 0; cb < Cfg::NC * 64; cb += 16) {
                            const uint32_t to = tmem + lane_base + Cfg::O_COL + cb;
                            uint32_t o[16];
                            tmem_ld16(to, o);
                            tc::tmem_ld_wait();
                            tc::tmem_regs_ready<16>(o);
                            const float *alc = al + (cb & 63);
#pragma unroll
                            for (int q = 0; q < 16; q++) o[q] = __float_as_uint(__uint_as_float(o[q]) * alc[q]);
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
            // the next item's description, and the cos / sin of -t for this thread's
            // dim in the last chunk, worked out while the last PV runs
            if (it + G < a.n_items) {
                item_info(a, it + G, fn);
                have_fn = true;
            }
            float dcr = 1.f, dsr = 0.f;
            {
                const int dlast = (Cfg::NC - 1) * 128 + quarter * 32 + lane;
                if (a.chunk_tiles == 0 && a.derotate && dlast >= a.rope.first)
                    rope_cos_sin(a.rope, -f.t, (dlast - a.rope.first) >> 1, dcr, dsr);
            }
            // item end: the four threads of a head add their partial sums
#pragma unroll
            for (int u = 0; u < 2; u++) {
                float l = l_run[u];
                l += __shfl_xor_sync(0xffffffffu, l, 1);
                l += __shfl_xor_sync(0xffffffffu, l, 2);
                float den = l;
                if (a.chunk_tiles == 0 && zl2[u] != -INFINITY) den += ex2(zl2[u] - m_run[u]);
                const int h = hr[u];
                if (t4 == 0) {
                    inv_den_s[h] = (real[u] && den > 0.f) ? 1.0f / den : 0.f;
                    if (real[u]) {
                        if (a.chunk_tiles > 0) {
                            a.part_ml[(it * 64 + h) * 2] = m_run[u];
                            a.part_ml[(it * 64 + h) * 2 + 1] = l;
                        } else if (a.lse) {
                            a.lse[f.bt * a.H + h0 + h] =
                                den > 0.f ? (m_run[u] + log2f(den)) * 0.6931471805599453f : -INFINITY;
                        }
                    }
                }
            }
            const bool ok = warp_wait(ofull, ii & 1, a.status, abort_flag, a.spin);
            if (named_bar_or(1, 128, !ok)) break;
            tc::fence_after_sync();
            const int nh = a.H - h0 < 64 ? a.H - h0 : 64;
            const int dl = quarter * 32 + lane;                 // dim within a chunk
            for (int c = 0; c < Cfg::NC; c++) {
                const int d = c * 128 + dl;
                const uint32_t to = tmem + lane_base + Cfg::O_COL + c * 64;
                float cr = 1.f, sr = 0.f;
                const bool rot_w = a.chunk_tiles == 0 && a.derotate && c * 128 + quarter * 32 + 31 >= a.rope.first;
                const bool rot = d >= a.rope.first;
                if (rot_w && rot) {
                    if (c == Cfg::NC - 1) {
                        cr = dcr;
                        sr = dsr;
                    } else {
                        rope_cos_sin(a.rope, -f.t, (d - a.rope.first) >> 1, cr, sr);
                    }
                }
                float sgn = (lane & 1) ? sr : -sr;
#pragma unroll 1
                for (int hb = 0; hb < 64; hb += 32) {
                    float o[32];
                    tc::tmem_ld32(to + hb, o);
                    tc::tmem_ld_wait();
                    tc::tmem_regs_ready<32>(o);
                    if (a.chunk_tiles > 0) {
                        float *po = a.part_o + (it * 64 + hb) * (int64_t)C + d;
#pragma unroll
                        for (int h = 0; h < 32; h++)
                            if (hb + h < nh) po[(int64_t)h * C] = o[h];
                        continue;
                    }
                    const float4 *id4 = reinterpret_cast<const float4 *>(inv_den_s + hb);
#pragma unroll
                    for (int q4 = 0; q4 < 8; q4++) {
                        const float4 iv4 = id4[q4];
                        o[4 * q4] *= iv4.x;
                        o[4 * q4 + 1] *= iv4.y;
                        o[4 * q4 + 2] *= iv4.z;
                        o[4 * q4 + 3] *= iv4.w;
                    }
                    if (rot_w) {
#pragma unroll
                        for (int h = 0; h < 32; h++) {
                            const float op = __shfl_xor_sync(0xffffffffu, o[h], 1);
                            if (rot) o[h] = o[h] * cr + op * sgn;
                        }
                    }
                    __nv_bfloat16 *op = a.out + (f.bt * a.H + h0 + hb) * (int64_t)C + d;
                    if (nh == 64) {
#pragma unroll
                        for (int h = 0; h < 32; h += 2) {
                            const __nv_bfloat162 v2 = __floats2bfloat162_rn(o[h], o[h + 1]);
                            op[(int64_t)h * C] = v2.x;
                            op[(int64_t)(h + 1) * C] = v2.y;
                        }
                    } else {
#pragma unroll
                        for (int h = 0; h < 32; h++)
                            if (hb + h < nh) op[(int64_t)h * C] = __float2bfloat16_rn(o[h]);
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(oempty);
            named_bar(1, 128);                   // inv_den_s is rewritten by the next item
            ii++;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == Cfg::MMA_WARP) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

// Split-KV combine: out[bt, h] = sum_c O_c e^(m_c - M) / (e^(z - M) + sum_c l_c e^(m_c - M)),
// over the chunks that hold some of the query's tiles, in a fixed order, then
// de-rotation.  One CTA per (query, head).
template <int C>
__global__ void __launch_bounds__(128) attn_combine_kernel(const __grid_constant__ AttnTcArgs a) {
    __shared__ float s_sc[64], s_red[4];
    __shared__ float s_M, s_den;
    const int64_t bt = blockIdx.x;
    const int h = blockIdx.y;
    const int hg = h / 64, hl = h % 64;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t t = a.q_pos[bt];
    const int64_t base = (bt * a.n_hg + hg) * a.n_chunks;
    const float zl2 = a.sink[h] * 1.4426950408889634f;
    // chunks past this query's last tile hold no work and were never written
    ItemInfo f;
    item_info(a, base, f);
    const int64_t nlive = (f.nt + a.chunk_tiles - 1) / a.chunk_tiles;
    const int live = nlive < a.n_chunks ? (int)nlive : a.n_chunks;
    // every live chunk's (max, sum) loaded at once, one per thread
    float mc = -INFINITY, lc = 0.f;
    if (tid < live) {
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
    const float sc = (tid < live && mc != -INFINITY) ? exp2f(mc - M) : 0.f;
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
        for (int c = 0; c < live; c++) {
            const float2 v = *reinterpret_cast<const float2 *>(a.part_o + ((base + c) * 64 + hl) * (int64_t)C + d);
            y0 = fmaf(v.x, s_sc[c], y0);
            y1 = fmaf(v.y, s_sc[c], y1);
        }
        y0 = den > 0.f ? y0 / den : 0.f;
        y1 = den > 0.f ? y1 / den : 0.f;
        if (a.derotate && d >= a.rope.first) {
            float cr, sr;
            rope_cos_sin(a.rope, -t, (d - a.rope.first) >> 1, cr, sr);
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
    static std::atomic<int> n[MAX_DEVICES];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return 148;
    int v = n[dev].load();
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        n[dev].store(v);
    }
    return v;
}

cudaError_t smem_limit_once(PerDevice &once, const void *kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    const unsigned long long bit = 1ull << dev;
    if (once.done.load() & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) once.done |= bit;
    return e;
}

bool attn_tc_supported(csa_dtype dt, int c) { return dt == CSA_BF16 && (c == 512 || c == 128); }

size_t attn_tc_split_bytes(int64_t rows, int H, int c, int n_chunks) {
    const int64_t items = rows * ((H + 63) / 64) * n_chunks;
    return (size_t)items * 64 * c * 4 + (size_t)items * 64 * 2 * 4 + 512;
}

// Number of split-KV chunks for rows of at most max_list entries: enough items
// to cover the GPU, each at least 4 tiles, as a function of the list length
// alone, so a sequence's result does not depend on the batch around it.  When
// the batch alone fills the GPU the split is skipped, unless `invariant` asks
// for the same split (and so the same summation order) at every batch size.
int attn_tc_chunks(int64_t rows, int H, int64_t max_list, bool invariant) {
    const int64_t tiles = (max_list + 63) / 64 + 1;       // + 1: padding of the compressed part
    if (tiles <= 4 || (!invariant && rows * ((H + 63) / 64) >= 2 * 148)) return 1;
    // at least 4 tiles per chunk and at most 16 chunks: a function of the list
    // length alone
    int64_t per = (tiles + 15) / 16;
    if (per < 4) per = 4;
    return (int)((tiles + per - 1) / per);
}

template <int C, bool KV8>
static cudaError_t launch_attn_tc_c(int64_t B, const AttnArgs &g, const int32_t *cnt, int n_chunks,
                                    void *split_ws, int max_ctas, cudaStream_t st) {
    AttnTcArgs a;
    a.kvc = KV8 ? nullptr : (const __nv_bfloat16 *)g.kvc;
    a.kv8 = KV8 ? (const uint8_t *)g.kvc : nullptr;
    a.zsrc = g.q;
    a.q_pos = g.q_pos;
    a.idx = g.idx;
    a.cnt = cnt;
    a.raw_pos0 = g.raw_pos0;
    a.sink = g.sink;
    a.out = (__nv_bfloat16 *)g.out;
    a.lse = g.lse;
    a.status = g.status;
    a.T = g.Tq; a.E = g.E; a.L = g.L;
    a.H = g.H; a.k = g.k; a.m = g.m; a.n_win = g.n_win; a.derotate = g.derotate;
    a.n_hg = (g.H + 63) / 64;
    a.spin = g.spin;
    a.q_norm = g.q_norm;
    a.norm_eps = g.norm_eps;
    a.scale_log2 = g.scale * 1.4426950408889634f;
    a.rope = g.rope;
    const int64_t rows = B * g.Tq;
    const int64_t max_list = (g.idx ? (int64_t)g.k : g.E) + g.n_win;
    const int64_t max_tiles = (max_list + 63) / 64 + 1;
    if (n_chunks > 1 && split_ws) {
        a.n_chunks = n_chunks;
        a.chunk_tiles = (int)((max_tiles + n_chunks - 1) / n_chunks);
        a.part_o = (float *)split_ws;
        a.part_ml = (float *)((char *)split_ws + (size_t)rows * a.n_hg * n_chunks * 64 * C * 4);
    } else {
        a.n_chunks = 1;
        a.chunk_tiles = 0;
        a.part_o = nullptr;
        a.part_ml = nullptr;
    }
    a.n_items = rows * a.n_hg * a.n_chunks;
    using Cfg = AtCfg<C>;
    // tensor maps: q rows [B*T*H, C]; compressed entries [B*E, C] and raw
    // window rows [B*L, C] as 64-row boxes (a map that is never read points
    // at q).
    CUtensorMap tq, tcmp, tw;
    const bool have_c = g.E > 0 && g.kvc != nullptr && !KV8;
    const bool have_w = g.L > 0 && g.kv_raw != nullptr;
    if (!make_tmap_bf16_2d(&tq, g.q, (uint64_t)(rows * g.H), C, 64) ||
        !make_tmap_bf16_2d(&tcmp, have_c ? g.kvc : g.q, have_c ? (uint64_t)(B * g.E) : (uint64_t)(rows * g.H),
                           C, 64) ||
        !make_tmap_bf16_2d(&tw, have_w ? g.kv_raw : g.q, have_w ? (uint64_t)(B * g.L) : (uint64_t)(rows * g.H),
                           C, 64))
        return cudaErrorInvalidValue;
    static PerDevice attr;
    {
        cudaError_t e = smem_limit_once(attr, (const void *)attn_tc_kernel<C, KV8>, Cfg::SMEM);
        if (e != cudaSuccess) return e;
    }
    const int sms = (max_ctas > 0 && max_ctas < device_sms() ? max_ctas : device_sms()) * Cfg::MIN_BLOCKS;
    const int grid = (int)(a.n_items < sms ? a.n_items : sms);
    attn_tc_kernel<C, KV8><<<grid, Cfg::THREADS, Cfg::SMEM, st>>>(tq, tcmp, tw, a);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || a.chunk_tiles == 0) return e;
    attn_combine_kernel<C><<<dim3((unsigned)rows, (unsigned)g.H), 128, 0, st>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_attn_tc(int64_t B, const AttnArgs &g, const int32_t *cnt, int n_chunks,
                           void *split_ws, int max_ctas, cudaStream_t st) {
    if (B * g.Tq == 0) return cudaSuccess;
    if (attn_pack_supported(B, g, n_chunks)) return launch_attn_pack(B, g, max_ctas, st);
    if (g.kv8) {
        if (g.c != 512) return cudaErrorInvalidValue;
        return launch_attn_tc_c<512, true>(B, g, cnt, n_chunks, split_ws, max_ctas, st);
    }
    if (g.c == 128) return launch_attn_tc_c<128, false>(B, g, cnt, n_chunks, split_ws, max_ctas, st);
    if (g.c == 512) return launch_attn_tc_c<512, false>(B, g, cnt, n_chunks, split_ws, max_ctas, st);
    return cudaErrorInvalidValue;
}

}  // namespace csa
