// Core attention on CUDA cores: the float32 path, and shapes the
// tensor-core kernels do not take.
//
// [DeepSeek-V4 book ch.6 "Shared key-value MQA"; ch.7 "The sliding window",
// "Partial rotary position embeddings", "Why the output is de-rotated",
// "Attention sinks".]
//
#include "common.cuh"
#include "kernels.h"

namespace csa {

// One warp per work item (query, group of WH heads).  The query rows live in
// shared memory (normalised when asked, rotated at t, times the logit scale in
// log2 units), read as broadcasts.  The list is walked 32 entries at a time:
//   QK  lane l takes entry base + l and dots its whole row with the WH rows;
//   softmax: the running max per head is agreed by a warp max; each lane
//       keeps its own partial denominator (rescaled with the shared max);
//   PV  lanes over dims: for each entry of the chunk, its probabilities come
//       from the owning lane by shuffle and every lane adds p * row[d] for
//       its dims d = lane + 32 i.
// No CTA-wide barrier: a warp runs its item alone, start to end.  The sink
// seeds the running max and enters only the denominator.
constexpr int AW_WARPS = 4;    // warps (items) per CTA
constexpr int AW_WH = 4;       // heads per item

template <typename T, int C>
__global__ void __launch_bounds__(AW_WARPS * 32)
attn_warp_kernel(const __grid_constant__ AttnArgs a, int64_t n_items) {
    constexpr int DPL = C / 32;                 // dims per lane in PV and the epilogue
    constexpr int VN = Vec<T>::N;
    extern __shared__ float smq[];              // [AW_WARPS][AW_WH][C]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * AW_WARPS + warp;
    if (item >= n_items) return;                // warp-uniform; nothing below syncs the CTA
    const int ng = (a.H + AW_WH - 1) / AW_WH;
    const int64_t bt = item / ng;
    const int h0 = (int)(item % ng) * AW_WH;
    const int hg = a.H - h0 < AW_WH ? a.H - h0 : AW_WH;
    const int64_t b = bt / a.Tq;
    const int64_t t = a.q_pos[bt];
    float *qs = smq + warp * AW_WH * C;
    const T *qg = (const T *)a.q + (bt * a.H + h0) * (int64_t)C;
    const float sl2 = a.scale * 1.4426950408889634f;

    // q rows: RMSNorm (when asked), RoPE at t, scale
#pragma unroll 1
    for (int h = 0; h < AW_WH; h++) {
        float v[DPL];
#pragma unroll
        for (int i = 0; i < DPL; i++) v[i] = h < hg ? to_f(qg[h * C + lane + 32 * i]) : 0.f;
        if (a.q_norm && h < hg) {
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < DPL; i++) ss = fmaf(v[i], v[i], ss);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float rs = 1.0f / sqrtf(ss / (float)C + a.norm_eps);
#pragma unroll
            for (int i = 0; i < DPL; i++) v[i] = v[i] * rs * a.q_norm[lane + 32 * i];
        }
#pragma unroll
        for (int i = 0; i < DPL; i++) {
            const int d = lane + 32 * i;       // d and d ^ 1 sit in lanes l and l ^ 1
            const float pv = __shfl_xor_sync(0xffffffffu, v[i], 1);
            if (d >= a.rope.first) {
                float cs, sn;
                rope_cos_sin(a.rope, t, (d - a.rope.first) >> 1, cs, sn);
                v[i] = (d & 1) ? pv * sn + v[i] * cs : v[i] * cs - pv * sn;
            }
            qs[h * C + d] = v[i] * sl2;
        }
    }
    __syncwarp();

    const int64_t nv = visible_count(t, a.m, a.E);
    const int64_t ncomp = a.idx ? (int64_t)a.k : nv;
    int64_t p0 = t - a.n_win + 1;
    if (p0 < 0) p0 = 0;
    const int64_t nwin = a.n_win > 0 ? t - p0 + 1 : 0;
    const int64_t total = ncomp + nwin;
    const int64_t rp0 = a.raw_pos0[b];

    float m[AW_WH], z2[AW_WH], lsum[AW_WH], acc[AW_WH][DPL];
#pragma unroll
    for (int h = 0; h < AW_WH; h++) {
        z2[h] = h < hg ? a.sink[h0 + h] * 1.4426950408889634f : -INFINITY;
        m[h] = z2[h];
        lsum[h] = 0.f;
#pragma unroll
        for (int i = 0; i < DPL; i++) acc[h][i] = 0.f;
    }
    for (int64_t base = 0; base < total; base += 32) {
        // this lane's entry of the chunk
        const int64_t e = base + lane;
        const T *row = nullptr;
        if (e < ncomp) {
            const int64_t j = a.idx ? (int64_t)a.idx[bt * a.k + e] : e;
            if (j >= 0 && j < a.E) row = (const T *)a.kvc + (b * a.E + j) * (int64_t)C;
            else if (j != -1 || !a.idx) atomicOr(a.status, ST_BAD_INDEX);
        } else if (e < total) {
            const int64_t r = p0 + (e - ncomp) - rp0;
            if (r >= 0 && r < a.L) row = (const T *)a.kv_raw + (b * a.L + r) * (int64_t)C;
            else atomicOr(a.status, ST_NO_WINDOW_ROW);
        }
        float sc[AW_WH];
#pragma unroll
        for (int h = 0; h < AW_WH; h++) sc[h] = 0.f;
        if (row) {
#pragma unroll 2
            for (int d = 0; d < C; d += VN) {
                float x[VN];
                Vec<T>::load(row + d, x);
#pragma unroll
                for (int h = 0; h < AW_WH; h++) {
#pragma unroll
                    for (int u = 0; u < VN; u += 4) {
                        const float4 qv = *reinterpret_cast<const float4 *>(qs + h * C + d + u);
                        sc[h] = fmaf(qv.x, x[u], sc[h]);
                        sc[h] = fmaf(qv.y, x[u + 1], sc[h]);
                        sc[h] = fmaf(qv.z, x[u + 2], sc[h]);
                        sc[h] = fmaf(qv.w, x[u + 3], sc[h]);
                    }
                }
            }
        }
        float p[AW_WH];
#pragma unroll
        for (int h = 0; h < AW_WH; h++) {
            const float sh = row ? sc[h] : -INFINITY;
            float mx = sh;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float mnew = fmaxf(m[h], mx);
            if (mnew == -INFINITY) {            // nothing readable yet (warp-uniform)
                p[h] = 0.f;
                continue;
            }
            const float alpha = exp2f(m[h] - mnew);
            p[h] = exp2f(sh - mnew);
            lsum[h] = fmaf(lsum[h], alpha, p[h]);
#pragma unroll
            for (int i = 0; i < DPL; i++) acc[h][i] *= alpha;
            m[h] = mnew;
        }
        const int nin = total - base < 32 ? (int)(total - base) : 32;
        for (int jj = 0; jj < nin; jj++) {
            const unsigned long long rj =
                __shfl_sync(0xffffffffu, (unsigned long long)reinterpret_cast<uintptr_t>(row), jj);
            if (rj == 0ull) continue;
            const T *r = reinterpret_cast<const T *>(rj);
            float pj[AW_WH];
#pragma unroll
            for (int h = 0; h < AW_WH; h++) pj[h] = __shfl_sync(0xffffffffu, p[h], jj);
#pragma unroll
            for (int i = 0; i < DPL; i++) {
                const float x = to_f(r[lane + 32 * i]);
#pragma unroll
                for (int h = 0; h < AW_WH; h++) acc[h][i] = fmaf(pj[h], x, acc[h][i]);
            }
        }
    }
    // finish: normalise, de-rotate by -t, store
    T *og = (T *)a.out + (bt * a.H + h0) * (int64_t)C;
#pragma unroll
    for (int h = 0; h < AW_WH; h++) {
        if (h >= hg) continue;
        float den = lsum[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        if (z2[h] != -INFINITY) den += exp2f(z2[h] - m[h]);
        const float inv = den > 0.f ? 1.0f / den : 0.f;
#pragma unroll
        for (int i = 0; i < DPL; i++) {
            const int d = lane + 32 * i;
            float o = acc[h][i] * inv;
            const float po = __shfl_xor_sync(0xffffffffu, o, 1);
            if (a.derotate && d >= a.rope.first) {
                float cs, sn;
                rope_cos_sin(a.rope, -t, (d - a.rope.first) >> 1, cs, sn);
                o = (d & 1) ? po * sn + o * cs : o * cs - po * sn;
            }
            from_f(og[h * C + d], o);
        }
        if (a.lse && lane == 0)
            a.lse[bt * a.H + h0 + h] = den > 0.f ? (m[h] + log2f(den)) * 0.6931471805599453f : -INFINITY;
    }
}

template <typename T, int C>
static cudaError_t launch_warp_c(int64_t B, const AttnArgs &a, cudaStream_t st) {
    const int64_t items = B * a.Tq * ((a.H + AW_WH - 1) / AW_WH);
    const int64_t blocks = (items + AW_WARPS - 1) / AW_WARPS;
    if (blocks > 2147483647LL) return cudaErrorInvalidValue;
    const size_t smem = (size_t)AW_WARPS * AW_WH * C * sizeof(float);
    attn_warp_kernel<T, C><<<(unsigned)blocks, AW_WARPS * 32, smem, st>>>(a, items);
    count_launches(1);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_warp_t(int64_t B, const AttnArgs &a, cudaStream_t st) {
    switch (a.c) {
        case 64: return launch_warp_c<T, 64>(B, a, st);
        case 128: return launch_warp_c<T, 128>(B, a, st);
        case 256: return launch_warp_c<T, 256>(B, a, st);
        case 512: return launch_warp_c<T, 512>(B, a, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attn_simt(csa_dtype dt, int64_t B, const AttnArgs &a, cudaStream_t st) {
    if (B * a.Tq == 0 || a.H == 0) return cudaSuccess;
    return dt == CSA_BF16 ? launch_warp_t<__nv_bfloat16>(B, a, st) : launch_warp_t<float>(B, a, st);
}

}  // namespace csa
