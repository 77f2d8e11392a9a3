// Compression of KV rows into entries: a streaming, vectorised HBM pass.
//
// ["DeepSeek-V4: Making Million-Token Context an Architectural Problem",
// Key design 1 (two-branch CSA equation) and Key design 2 (HCA equation);
// DeepSeek-V4 book ch.5 "One weight distribution per coordinate".]
//
// One thread owns one 16-byte vector of channels (8 bf16 or 4 f32) of one
// block and walks the block's m slots with a per-channel online softmax
// (running max, denominator and weighted sum), so every input byte is read
// once with coalesced 16-byte loads and m = 128 needs no second pass.  The
// same thread also writes the block's raw rows rotated at their positions
// (the stored rows a window reads), fusing that pass into this one.
#include "common.cuh"
#include "kernels.h"

namespace csa {

template <typename T>
__device__ __forceinline__ void rotate_vec(float *v, int ch0, int64_t pos, const RopeFreqs &rf) {
    constexpr int N = Vec<T>::N;
    if (ch0 + N <= rf.first) return;
#pragma unroll
    for (int q = 0; q < N / 2; q++) {
        int ch = ch0 + 2 * q;
        if (ch < rf.first) continue;
        float cs, sn;
        rope_cos_sin((double)pos, rf.w[(ch - rf.first) >> 1], cs, sn);
        float x0 = v[2 * q], x1 = v[2 * q + 1];
        v[2 * q] = x0 * cs - x1 * sn;
        v[2 * q + 1] = x0 * sn + x1 * cs;
    }
}

template <typename T>
__device__ __forceinline__ void softmax_step(float a, float v, float &mx, float &den, float &acc) {
    if (a > mx) {
        float s = __expf(mx - a);
        den = den * s + 1.0f;
        acc = acc * s + v;
        mx = a;
    } else {
        float p = __expf(a - mx);
        den += p;
        acc = fmaf(p, v, acc);
    }
}

template <typename T>
__global__ void __launch_bounds__(256)
compress_kernel(const T *__restrict__ C, const T *__restrict__ Z, const float *__restrict__ bias,
                const T *__restrict__ Cb, const T *__restrict__ Zb, const float *__restrict__ biasb,
                T *__restrict__ out, T *__restrict__ raw_out, int64_t B, int64_t n, int c, int m,
                int overlap, int64_t E, int64_t Eg, RopeFreqs rope) {
    constexpr int N = Vec<T>::N;
    const int cv = c / N;
    int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= B * Eg * cv) return;
    const int ch0 = (int)(gid % cv) * N;
    const int64_t e = (gid / cv) % Eg;
    const int64_t b = gid / ((int64_t)cv * Eg);
    const T *Cs = C + b * n * c;
    const T *Zs = Z + b * n * c;

    float mx[N], den[N], acc[N];
#pragma unroll
    for (int i = 0; i < N; i++) { mx[i] = -INFINITY; den[i] = 0.f; acc[i] = 0.f; }

    const int64_t row0 = e * m;
    const int slots = (int)((n - row0) < m ? (n - row0) : m);   // < m only for a partial tail
    for (int s = 0; s < slots; s++) {
        float z[N], v[N], bs[N];
        const int64_t row = row0 + s;
        Vec<T>::load_stream(Zs + row * c + ch0, z);
        Vec<T>::load_stream(Cs + row * c + ch0, v);
        Vec<float>::load(bias + (int64_t)s * c + ch0, bs);
        if constexpr (N == 8) Vec<float>::load(bias + (int64_t)s * c + ch0 + 4, bs + 4);
#pragma unroll
        for (int i = 0; i < N; i++) softmax_step<T>(z[i] + bs[i], v[i], mx[i], den[i], acc[i]);
        if (raw_out != nullptr) {
            rotate_vec<T>(v, ch0, row, rope);
            Vec<T>::store(raw_out + (b * n + row) * c + ch0, v);
        }
    }
    if (e >= E) return;                 // partial tail block: raw rows only
    if (overlap && e > 0) {
        const T *Cbs = Cb + b * n * c;
        const T *Zbs = Zb + b * n * c;
        for (int s = 0; s < m; s++) {
            float z[N], v[N], bs[N];
            const int64_t row = (e - 1) * m + s;
            Vec<T>::load_stream(Zbs + row * c + ch0, z);
            Vec<T>::load_stream(Cbs + row * c + ch0, v);
            Vec<float>::load(biasb + (int64_t)s * c + ch0, bs);
            if constexpr (N == 8) Vec<float>::load(biasb + (int64_t)s * c + ch0 + 4, bs + 4);
#pragma unroll
            for (int i = 0; i < N; i++) softmax_step<T>(z[i] + bs[i], v[i], mx[i], den[i], acc[i]);
        }
    }
    float o[N];
#pragma unroll
    for (int i = 0; i < N; i++) o[i] = acc[i] / den[i];
    rotate_vec<T>(o, ch0, (e + 1) * m - 1, rope);
    Vec<T>::store(out + (b * E + e) * c + ch0, o);
}

// Long blocks (m >= 16, one branch): one CTA per (sequence, block).  Thread
// (g, v) owns channel vector v and the slots s = g, g + G, ... of the block;
// each keeps a partial online softmax, and the G partials of a vector are
// merged through shared memory (max, rescaled denominators and sums).
constexpr int CW_THREADS = 256;

template <typename T>
__global__ void __launch_bounds__(CW_THREADS)
compress_wide_kernel(const T *__restrict__ C, const T *__restrict__ Z, const float *__restrict__ bias,
                     T *__restrict__ out, T *__restrict__ raw_out, int64_t n, int c, int m, int64_t E,
                     int64_t Eg, RopeFreqs rope) {
    constexpr int N = Vec<T>::N;
    __shared__ float part[CW_THREADS][3][N];
    const int V = c / N;                  // vectors per row (<= CW_THREADS)
    const int G = CW_THREADS / V;         // row groups
    const int tid = threadIdx.x;
    const int v = tid % V, grp = tid / V;
    const int64_t e = blockIdx.x % Eg, b = blockIdx.x / Eg;
    const int ch0 = v * N;
    const T *Cs = C + b * n * c;
    const T *Zs = Z + b * n * c;
    const int64_t row0 = e * m;
    const int slots = (int)((n - row0) < m ? (n - row0) : m);
    float mx[N], den[N], acc[N];
#pragma unroll
    for (int i = 0; i < N; i++) { mx[i] = -INFINITY; den[i] = 0.f; acc[i] = 0.f; }
    if (grp < G) {
        for (int s = grp; s < slots; s += G) {
            float z[N], x[N], bs[N];
            const int64_t row = row0 + s;
            Vec<T>::load_stream(Zs + row * c + ch0, z);
            Vec<T>::load_stream(Cs + row * c + ch0, x);
            Vec<float>::load(bias + (int64_t)s * c + ch0, bs);
            if constexpr (N == 8) Vec<float>::load(bias + (int64_t)s * c + ch0 + 4, bs + 4);
#pragma unroll
            for (int i = 0; i < N; i++) softmax_step<T>(z[i] + bs[i], x[i], mx[i], den[i], acc[i]);
            if (raw_out != nullptr) {
                rotate_vec<T>(x, ch0, row, rope);
                Vec<T>::store(raw_out + (b * n + row) * c + ch0, x);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < N; i++) {
        part[tid][0][i] = mx[i];
        part[tid][1][i] = den[i];
        part[tid][2][i] = acc[i];
    }
    __syncthreads();
    if (grp != 0 || e >= E) return;       // one thread per vector merges; tail block: raw rows only
#pragma unroll
    for (int i = 0; i < N; i++) {
        float M = -INFINITY;
        for (int q = 0; q < G; q++) M = fmaxf(M, part[q * V + v][0][i]);
        float d = 0.f, a = 0.f;
        for (int q = 0; q < G; q++) {
            const float mq = part[q * V + v][0][i];
            if (mq == -INFINITY) continue;
            const float sc = __expf(mq - M);
            d = fmaf(part[q * V + v][1][i], sc, d);
            a = fmaf(part[q * V + v][2][i], sc, a);
        }
        mx[i] = a / d;
    }
    rotate_vec<T>(mx, ch0, (e + 1) * m - 1, rope);
    Vec<T>::store(out + (b * E + e) * c + ch0, mx);
}

cudaError_t launch_compress(csa_dtype dt, int64_t B, int64_t n, int c, int m, int overlap,
                            const void *C, const void *Z, const float *bias, const void *Cb,
                            const void *Zb, const float *biasb, void *out, void *raw_out,
                            const RopeFreqs &rope, cudaStream_t st) {
    const int64_t E = n / m;
    const int64_t Eg = raw_out ? (n + m - 1) / m : E;
    const int N = dt == CSA_BF16 ? 8 : 4;
    const int64_t threads = B * Eg * (c / N);
    if (threads == 0) return cudaSuccess;
    if (m >= 16 && !overlap && c / N <= CW_THREADS) {
        const int64_t blocks = B * Eg;
        if (dt == CSA_BF16) {
            using T = __nv_bfloat16;
            compress_wide_kernel<T><<<(unsigned)blocks, CW_THREADS, 0, st>>>(
                (const T *)C, (const T *)Z, bias, (T *)out, (T *)raw_out, n, c, m, E, Eg, rope);
        } else {
            compress_wide_kernel<float><<<(unsigned)blocks, CW_THREADS, 0, st>>>(
                (const float *)C, (const float *)Z, bias, (float *)out, (float *)raw_out, n, c, m, E, Eg, rope);
        }
        count_launches(1);
        return cudaGetLastError();
    }
    const int tpb = 256;
    const int64_t blocks = (threads + tpb - 1) / tpb;
    if (dt == CSA_BF16) {
        using T = __nv_bfloat16;
        compress_kernel<T><<<(unsigned)blocks, tpb, 0, st>>>(
            (const T *)C, (const T *)Z, bias, (const T *)Cb, (const T *)Zb, biasb, (T *)out,
            (T *)raw_out, B, n, c, m, overlap, E, Eg, rope);
    } else {
        compress_kernel<float><<<(unsigned)blocks, tpb, 0, st>>>(
            (const float *)C, (const float *)Z, bias, (const float *)Cb, (const float *)Zb, biasb,
            (float *)out, (float *)raw_out, B, n, c, m, overlap, E, Eg, rope);
    }
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace csa
