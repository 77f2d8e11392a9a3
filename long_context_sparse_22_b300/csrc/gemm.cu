// Grouped bf16 GEMM on the 5th-generation tensor cores, for the layer's
// output projection.
//
// ["DeepSeek-V4" book ch.6 "Why output projection is a large cost": the
// heads are split into groups, each group's concatenated outputs are
// projected to a small width d_g, and the concatenation of the group results
// is projected to the hidden width d; "DeepSeek-V4 technical preview" blog:
// the group counts of the configurations.]
//
//   Y[g][m, n] = sum_k A[m, g*K + k] * W[g*N + n, k]      (g < groups)
//   Y is written at column g*N + n of a [M, groups*N] row-major output.
// A is row-major [M, groups*K] (the attention output [T, H*c] for the first
// stage), W row-major [groups*N, K] (one [N, K] matrix per group, the
// out-features-major layout of a linear layer).  bf16 in, fp32 accumulation
// in tensor memory, bf16 out.
//
// One CTA per SM, persistent over (group, n tile, m tile) work items.  A tile
// is 128 x 256 x 64: TMA brings a 128 x 64 slice of A and a 256 x 64 slice of
// W per stage (128-byte swizzle, 4 stages); one thread issues
// tcgen05.mma M = 128, N = 256, K = 16; two 256-column accumulators in
// tensor memory alternate so the epilogue of one tile (4 warps, one output
// row per thread, 16-byte stores) overlaps the MMAs of the next.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace csa {

struct GemmCfg {
    static constexpr int BM = 128, BN = 256, BK = 64;
    static constexpr int STAGES = 4;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SMEM = STAGES * STAGE_BYTES + 256 + 1024;
    static constexpr int THREADS = 192;                 // producer, MMA, 4 epilogue warps
    static constexpr int TMEM_COLS = 512;
};

struct GemmArgs {
    __nv_bfloat16 *Y;
    unsigned *status;
    int M, N, K, groups;
    int mt, nt;            // m tiles, n tiles
    long long spin;
};

__device__ __forceinline__ void gemm_item(const GemmArgs &a, long long it, int &g, int &n0, int &m0) {
    // m fastest, so consecutive CTAs share the same W slice through L2
    m0 = (int)(it % a.mt) * GemmCfg::BM;
    const long long r = it / a.mt;
    n0 = (int)(r % a.nt) * GemmCfg::BN;
    g = (int)(r / a.nt);
}

__global__ void __launch_bounds__(GemmCfg::THREADS, 1)
gemm_bf16_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                 const __grid_constant__ GemmArgs a) {
    using Cfg = GemmCfg;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = (uint64_t *)(smem + Cfg::STAGES * Cfg::STAGE_BYTES);
    uint64_t *full = bars, *empty = full + Cfg::STAGES;
    uint64_t *accfull = empty + Cfg::STAGES, *accempty = accfull + 2, *mdone = accempty + 2;
    uint32_t *tmem_slot = (uint32_t *)(mdone + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long items = (long long)a.groups * a.nt * a.mt;
    const int ksteps = a.K / Cfg::BK;
    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; s++) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; i++) {
            tc::mbar_init(&accfull[i], 1);
            tc::mbar_init(&accempty[i], 4);
        }
        tc::mbar_init(mdone, 1);
        *abort_flag = 0;
        tc::fence_barrier_init();
        tc::prefetch_tmap(&tm_a);
        tc::prefetch_tmap(&tm_w);
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (long long it = blockIdx.x; ok && it < items; it += gridDim.x) {
                int g, n0, m0;
                gemm_item(a, it, g, n0, m0);
                for (int ks = 0; ks < ksteps; ks++) {
                    if (!tc::mbar_wait(&empty[s], ph ^ 1, a.status, abort_flag, a.spin)) { ok = false; break; }
                    uint8_t *dst = smem + s * Cfg::STAGE_BYTES;
                    tc::mbar_expect_tx(&full[s], Cfg::STAGE_BYTES);
                    tc::tma_load_2d(dst, &tm_a, g * a.K + ks * Cfg::BK, m0, &full[s]);
                    tc::tma_load_2d(dst + Cfg::A_BYTES, &tm_w, ks * Cfg::BK, g * a.N + n0, &full[s]);
                    issued |= 1u << s;
                    last_par = (last_par & ~(1u << s)) | (ph << s);
                    if (++s == Cfg::STAGES) { s = 0; ph ^= 1; }
                }
            }
            if (*abort_flag)
                for (int q = 0; q < Cfg::STAGES; q++)
                    if (issued & (1u << q))
                        for (long long i = 0; i < tc::DRAIN_LIMIT; i++)
                            if (tc::mbar_test(&full[q], (last_par >> q) & 1u)) break;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(Cfg::BM, Cfg::BN);
            int s = 0, acc = 0;
            uint32_t ph = 0, accph = 0;
            const uint32_t base = tc::smem_u32(smem);
            bool ok = true;
            for (long long it = blockIdx.x; ok && it < items; it += gridDim.x) {
                if (!tc::mbar_wait(&accempty[acc], accph ^ 1, a.status, abort_flag, a.spin)) break;
                tc::fence_after_sync();
                const uint32_t d = tmem + acc * Cfg::BN;
                for (int ks = 0; ks < ksteps; ks++) {
                    if (!tc::mbar_wait(&full[s], ph, a.status, abort_flag, a.spin)) { ok = false; break; }
                    tc::fence_after_sync();
                    const uint32_t sa = base + s * Cfg::STAGE_BYTES, sb = sa + Cfg::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < 4; kk++)
                        tc::mma_bf16(d, tc::desc_kmajor_sw128(sa + kk * 32), tc::desc_kmajor_sw128(sb + kk * 32),
                                     idesc, (ks | kk) != 0);
                    tc::mma_commit(&empty[s]);
                    if (++s == Cfg::STAGES) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                tc::mma_commit(&accfull[acc]);
                if (++acc == 2) { acc = 0; accph ^= 1; }
            }
            tc::mma_commit(mdone);
            for (long long i = 0; i < tc::DRAIN_LIMIT; i++)
                if (tc::mbar_test(mdone, 0)) break;
        }
    } else {
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31, one output row per thread
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        int acc = 0;
        uint32_t accph = 0;
        for (long long it = blockIdx.x; it < items; it += gridDim.x) {
            int g, n0, m0;
            gemm_item(a, it, g, n0, m0);
            if (!tc::mbar_wait(&accfull[acc], accph, a.status, abort_flag, a.spin)) break;
            tc::fence_after_sync();
            const int m = m0 + row;
            __nv_bfloat16 *yrow = a.Y + (int64_t)m * ((int64_t)a.groups * a.N) + (int64_t)g * a.N + n0;
#pragma unroll 1
            for (int cb = 0; cb < Cfg::BN; cb += 32) {
                float v[32];
                tc::tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + acc * Cfg::BN + cb, v);
                tc::tmem_ld_wait();
                tc::tmem_regs_ready<32>(v);
                if (m < a.M) {
                    uint4 o[4];
                    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(o);
#pragma unroll
                    for (int q = 0; q < 16; q++) h[q] = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
                    uint4 *dst = reinterpret_cast<uint4 *>(yrow + cb);
#pragma unroll
                    for (int q = 0; q < 4; q++) dst[q] = o[q];
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&accempty[acc]);
            if (++acc == 2) { acc = 0; accph ^= 1; }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

cudaError_t launch_gemm_bf16(int64_t M, int N, int K, int groups, const void *A, const void *W, void *Y,
                             unsigned *status, long long spin, cudaStream_t st) {
    if (M == 0 || groups == 0) return cudaSuccess;
    using Cfg = GemmCfg;
    if (N % Cfg::BN || K % Cfg::BK || M > 2147483647LL - Cfg::BM) return cudaErrorInvalidValue;
    CUtensorMap ta, tw;
    // A [M, groups*K] with 128-row boxes; W [groups*N, K] with 256-row boxes (64 bf16 = 128 B wide)
    if (!make_tmap_bf16_2d(&ta, A, (uint64_t)M, (uint64_t)groups * K, Cfg::BM) ||
        !make_tmap_bf16_2d(&tw, W, (uint64_t)groups * N, (uint64_t)K, Cfg::BN))
        return cudaErrorInvalidValue;
    GemmArgs a;
    a.Y = (__nv_bfloat16 *)Y;
    a.status = status;
    a.M = (int)M; a.N = N; a.K = K; a.groups = groups;
    a.mt = (int)((M + Cfg::BM - 1) / Cfg::BM);
    a.nt = N / Cfg::BN;
    a.spin = spin;
    static PerDevice attr;
    cudaError_t e = smem_limit_once(attr, (const void *)gemm_bf16_kernel, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    const long long items = (long long)groups * a.nt * a.mt;
    const int sms = device_sms();
    const int grid = (int)(items < sms ? items : sms);
    gemm_bf16_kernel<<<grid, Cfg::THREADS, Cfg::SMEM, st>>>(ta, tw, a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace csa
