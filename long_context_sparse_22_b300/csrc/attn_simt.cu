// Core attention on CUDA cores: the float32 path, and shapes the
// tensor-core kernels do not take.
//
// [DeepSeek-V4 book ch.6 "Shared key-value MQA"; ch.7 "The sliding window",
// "Partial rotary position embeddings", "Why the output is de-rotated",
// "Attention sinks".]
//
// One CTA = one query and a group of up to HG heads.  Entries (selected or
// every visible compressed entry, then the window rows) stream through
// shared memory in tiles of TE rows; logits are warp-reduced dot products,
// the softmax is online (running max and denominator per head, seeded with
// the sink logit so the sink only enters the denominator), and each thread
// accumulates HG x (c/128) output columns in registers.
#include "common.cuh"
#include "kernels.h"

namespace csa {

constexpr int AT_THREADS = 128;
constexpr int AT_HG = 16;   // heads per CTA
constexpr int AT_TE = 16;   // entry rows per tile
constexpr int AT_DMAX = 4;  // c / 128 columns per thread (c <= 512)

template <typename T>
__global__ void __launch_bounds__(AT_THREADS)
attn_simt_kernel(AttnArgs a) {
    extern __shared__ float sm[];
    const int c = a.c;
    const int hg = min(AT_HG, a.H - (int)blockIdx.y * AT_HG);
    const int h0 = blockIdx.y * AT_HG;
    float *qs = sm;                       // [AT_HG][c]
    float *ks = qs + AT_HG * c;           // [AT_TE][c]
    float *lg = ks + AT_TE * c;           // [AT_HG][AT_TE]
    __shared__ const T *rowp[AT_TE];
    __shared__ float s_m[AT_HG], s_den[AT_HG], s_corr[AT_HG];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t bt = blockIdx.x;
    const int64_t b = bt / a.Tq;
    const int64_t t = a.q_pos[bt];
    const T *q = (const T *)a.q + (bt * a.H + h0) * (int64_t)c;

    // q rows -> shared float (RMSNorm per head when asked), rotated at t and scaled
    if (a.q_norm) {
        for (int i = tid; i < hg * c; i += AT_THREADS) qs[i] = to_f(q[i]);
        __syncthreads();
        for (int h = warp; h < hg; h += AT_THREADS / 32) {
            float ss = 0.f;
            for (int ch = lane; ch < c; ch += 32) ss = fmaf(qs[h * c + ch], qs[h * c + ch], ss);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float rs = 1.0f / sqrtf(ss / (float)c + a.norm_eps);
            for (int ch = lane; ch < c; ch += 32) qs[h * c + ch] = qs[h * c + ch] * rs * a.q_norm[ch] * a.scale;
        }
    } else {
        for (int i = tid; i < hg * c; i += AT_THREADS) qs[i] = to_f(q[i]) * a.scale;
    }
    __syncthreads();
    const int pairs = a.rope.pairs;
    for (int i = tid; i < hg * pairs; i += AT_THREADS) {
        const int h = i / pairs, p = i % pairs;
        float cs, sn;
        rope_cos_sin((double)t, a.rope.w[p], cs, sn);
        float *v = qs + h * c + a.rope.first + 2 * p;
        const float x0 = v[0], x1 = v[1];
        v[0] = x0 * cs - x1 * sn;
        v[1] = x0 * sn + x1 * cs;
    }
    if (tid < hg) {
        const float z = a.sink[h0 + tid];
        s_m[tid] = z;
        s_den[tid] = (z == -INFINITY) ? 0.f : 1.f;
    }

    // entry list: compressed part then window part
    const int64_t nv = visible_count(t, a.m, a.E);
    const int64_t ncomp = a.idx ? (int64_t)a.k : nv;
    int64_t p0 = t - a.n_win + 1;
    if (p0 < 0) p0 = 0;
    const int64_t nwin = a.n_win > 0 ? (t - p0 + 1) : 0;
    const int64_t total = ncomp + (nwin > 0 ? nwin : 0);
    const int64_t rp0 = a.raw_pos0[b];

    float acc[AT_HG][AT_DMAX];
#pragma unroll
    for (int h = 0; h < AT_HG; h++)
#pragma unroll
        for (int i = 0; i < AT_DMAX; i++) acc[h][i] = 0.f;
    __syncthreads();

    for (int64_t base = 0; base < total; base += AT_TE) {
        if (tid < AT_TE) {
            const int64_t e = base + tid;
            const T *p = nullptr;
            if (e < ncomp) {
                int64_t j = a.idx ? (int64_t)a.idx[bt * a.k + e] : e;
                if (j >= 0 && j < a.E) {
                    p = (const T *)a.kvc + (b * a.E + j) * (int64_t)c;
                } else if (j != -1 || !a.idx) {
                    atomicOr(a.status, ST_BAD_INDEX);
                }
            } else if (e < total) {
                const int64_t row = p0 + (e - ncomp) - rp0;
                if (row >= 0 && row < a.L) p = (const T *)a.kv_raw + (b * a.L + row) * (int64_t)c;
                else atomicOr(a.status, ST_NO_WINDOW_ROW);
            }
            rowp[tid] = p;
        }
        __syncthreads();
        // rows -> shared float (zeros for skipped rows)
        constexpr int N = Vec<T>::N;
        for (int i = tid; i < AT_TE * (c / N); i += AT_THREADS) {
            const int r = i / (c / N), cc = (i % (c / N)) * N;
            float v[N];
            if (rowp[r]) Vec<T>::load(rowp[r] + cc, v);
            else
#pragma unroll
                for (int u = 0; u < N; u++) v[u] = 0.f;
#pragma unroll
            for (int u = 0; u < N; u++) ks[r * c + cc + u] = v[u];
        }
        __syncthreads();
        // logits: warp w takes pairs w, w+4, ...
        for (int pr = warp; pr < AT_HG * AT_TE; pr += AT_THREADS / 32) {
            const int h = pr / AT_TE, e = pr % AT_TE;
            float d = 0.f;
            if (h < hg && rowp[e]) {
                for (int ch = lane; ch < c; ch += 32) d = fmaf(qs[h * c + ch], ks[e * c + ch], d);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            }
            if (lane == 0) lg[h * AT_TE + e] = (h < hg && rowp[e]) ? d : -INFINITY;
        }
        __syncthreads();
        // online softmax, one thread per head
        if (tid < hg) {
            const int h = tid;
            float mt = s_m[h];
            for (int e = 0; e < AT_TE; e++) mt = fmaxf(mt, lg[h * AT_TE + e]);
            float corr = 1.f, den = s_den[h];
            if (mt != -INFINITY) {
                corr = __expf(s_m[h] - mt);
                den *= corr;
                for (int e = 0; e < AT_TE; e++) {
                    const float p = __expf(lg[h * AT_TE + e] - mt);
                    lg[h * AT_TE + e] = p;
                    den += p;
                }
            } else {
                for (int e = 0; e < AT_TE; e++) lg[h * AT_TE + e] = 0.f;
            }
            s_m[h] = mt;
            s_den[h] = den;
            s_corr[h] = corr;
        }
        __syncthreads();
        // PV: this thread's columns d = tid + 128*i
#pragma unroll
        for (int h = 0; h < AT_HG; h++) {
            if (h < hg) {
                const float corr = s_corr[h];
#pragma unroll
                for (int i = 0; i < AT_DMAX; i++) acc[h][i] *= corr;
            }
        }
        for (int e = 0; e < AT_TE; e++) {
            float kv[AT_DMAX];
#pragma unroll
            for (int i = 0; i < AT_DMAX; i++) {
                const int d = tid + i * AT_THREADS;
                kv[i] = d < c ? ks[e * c + d] : 0.f;
            }
#pragma unroll
            for (int h = 0; h < AT_HG; h++) {
                if (h < hg) {
                    const float p = lg[h * AT_TE + e];
#pragma unroll
                    for (int i = 0; i < AT_DMAX; i++) acc[h][i] = fmaf(p, kv[i], acc[h][i]);
                }
            }
        }
        __syncthreads();
    }
    // finish: out = acc / den, de-rotate, store
#pragma unroll
    for (int h = 0; h < AT_HG; h++) {
        if (h < hg) {
            const float den = s_den[h];
            const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
            for (int i = 0; i < AT_DMAX; i++) {
                const int d = tid + i * AT_THREADS;
                if (d < c) qs[h * c + d] = acc[h][i] * inv;
            }
        }
    }
    __syncthreads();
    if (a.derotate) {
        for (int i = tid; i < hg * pairs; i += AT_THREADS) {
            const int h = i / pairs, p = i % pairs;
            float cs, sn;
            rope_cos_sin(-(double)t, a.rope.w[p], cs, sn);
            float *v = qs + h * c + a.rope.first + 2 * p;
            const float x0 = v[0], x1 = v[1];
            v[0] = x0 * cs - x1 * sn;
            v[1] = x0 * sn + x1 * cs;
        }
        __syncthreads();
    }
    T *o = (T *)a.out + (bt * a.H + h0) * (int64_t)c;
    for (int i = tid; i < hg * c; i += AT_THREADS) from_f(o[i], qs[i]);
    if (a.lse && tid < hg) {
        const float den = s_den[tid];
        a.lse[bt * a.H + h0 + tid] = den > 0.f ? s_m[tid] + logf(den) : -INFINITY;
    }
}

static PerDevice g_attn_smem[2];

cudaError_t launch_attn_simt(csa_dtype dt, int64_t B, const AttnArgs &a, cudaStream_t st) {
    if (B * a.Tq == 0 || a.H == 0) return cudaSuccess;
    dim3 grid((unsigned)(B * a.Tq), (unsigned)((a.H + AT_HG - 1) / AT_HG));
    const size_t smem = ((size_t)AT_HG * a.c + (size_t)AT_TE * a.c + AT_HG * AT_TE) * 4;
    const size_t smem_max = ((size_t)AT_HG * 512 + (size_t)AT_TE * 512 + AT_HG * AT_TE) * 4;
    const int di = dt == CSA_BF16 ? 1 : 0;
    {
        cudaError_t e = dt == CSA_BF16
            ? smem_limit_once(g_attn_smem[di], (const void *)attn_simt_kernel<__nv_bfloat16>, (int)smem_max)
            : smem_limit_once(g_attn_smem[di], (const void *)attn_simt_kernel<float>, (int)smem_max);
        if (e != cudaSuccess) return e;
    }
    if (dt == CSA_BF16) attn_simt_kernel<__nv_bfloat16><<<grid, AT_THREADS, smem, st>>>(a);
    else attn_simt_kernel<float><<<grid, AT_THREADS, smem, st>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace csa
