// Lightning-indexer scores on CUDA cores (float32 storage, and any shape the
// tensor-core kernels do not take).
//
// ["DeepSeek-V4: Making Million-Token Context an Architectural Problem",
// Key design 1 index-score equation; DeepSeek-V4 book ch.6 "The index
// score".]  scores[b,t,j] = sum_h w[b,t,h] * ReLU(qI[b,t,h,:] . kI[b,j,:]).
//
// One CTA holds one query's hI x dI indexer query in shared memory (float)
// and each thread scores one entry: its key row sits in registers and every
// shared-memory read of q is a broadcast.
#include "common.cuh"
#include "kernels.h"

namespace csa {

template <typename T, int DI>
__global__ void __launch_bounds__(128)
indexer_simt_kernel(const T *__restrict__ qI, const float *__restrict__ w,
                    const T *__restrict__ kI, const int64_t *__restrict__ q_pos,
                    float *__restrict__ scores, int64_t Tq, int hI, int64_t E, int m,
                    int write_masked) {
    extern __shared__ float sm[];
    float *qs = sm;                 // [hI][DI]
    float *ws = sm + hI * DI;       // [hI]
    const int64_t bt = blockIdx.x;  // b * Tq + t
    const int64_t b = bt / Tq;
    const int64_t nv = visible_count(q_pos[bt], m, E);
    const int64_t j0 = (int64_t)blockIdx.y * blockDim.x;
    if (j0 >= nv) {
        if (write_masked) {
            int64_t j = j0 + threadIdx.x;
            if (j < E) scores[bt * E + j] = -INFINITY;
        }
        return;
    }
    for (int i = threadIdx.x; i < hI * DI; i += blockDim.x) qs[i] = to_f(qI[bt * hI * DI + i]);
    for (int i = threadIdx.x; i < hI; i += blockDim.x) ws[i] = w[bt * hI + i];
    __syncthreads();
    const int64_t j = j0 + threadIdx.x;
    if (j >= E) return;
    if (j >= nv) {
        if (write_masked) scores[bt * E + j] = -INFINITY;
        return;
    }
    float k[DI];
    const T *kr = kI + (b * E + j) * DI;
#pragma unroll
    for (int d = 0; d < DI; d += Vec<T>::N) Vec<T>::load(kr + d, k + d);
    float s = 0.f;
    for (int h = 0; h < hI; h++) {
        const float4 *q4 = reinterpret_cast<const float4 *>(qs + h * DI);
        float dot = 0.f;
#pragma unroll
        for (int d = 0; d < DI / 4; d++) {
            float4 qv = q4[d];
            dot = fmaf(qv.x, k[4 * d], dot);
            dot = fmaf(qv.y, k[4 * d + 1], dot);
            dot = fmaf(qv.z, k[4 * d + 2], dot);
            dot = fmaf(qv.w, k[4 * d + 3], dot);
        }
        s = fmaf(ws[h], fmaxf(dot, 0.f), s);
    }
    scores[bt * E + j] = s;
}

template <typename T>
static cudaError_t launch_simt_t(int64_t B, int64_t Tq, int hI, int dI, int64_t E, int m,
                                 const void *qI, const float *w, const void *kI,
                                 const int64_t *q_pos, float *scores, int write_masked,
                                 cudaStream_t st) {
    dim3 grid((unsigned)(B * Tq), (unsigned)((E + 127) / 128));
    size_t smem = (size_t)hI * dI * 4 + (size_t)hI * 4;
    const T *q = (const T *)qI;
    const T *k = (const T *)kI;
    switch (dI) {
    case 32:
        indexer_simt_kernel<T, 32><<<grid, 128, smem, st>>>(q, w, k, q_pos, scores, Tq, hI, E, m, write_masked);
        break;
    case 64:
        indexer_simt_kernel<T, 64><<<grid, 128, smem, st>>>(q, w, k, q_pos, scores, Tq, hI, E, m, write_masked);
        break;
    default:
        indexer_simt_kernel<T, 128><<<grid, 128, smem, st>>>(q, w, k, q_pos, scores, Tq, hI, E, m, write_masked);
        break;
    }
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_indexer_simt(csa_dtype dt, int64_t B, int64_t Tq, int hI, int dI, int64_t E,
                                int m, const void *qI, const float *w, const void *kI,
                                const int64_t *q_pos, float *scores, int write_masked,
                                cudaStream_t st) {
    if (B * Tq == 0 || E == 0) return cudaSuccess;
    if (dt == CSA_BF16)
        return launch_simt_t<__nv_bfloat16>(B, Tq, hI, dI, E, m, qI, w, kI, q_pos, scores,
                                            write_masked, st);
    return launch_simt_t<float>(B, Tq, hI, dI, E, m, qI, w, kI, q_pos, scores, write_masked, st);
}

}  // namespace csa
