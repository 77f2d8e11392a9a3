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
        rope_cos_sin(rf, pos, (ch - rf.first) >> 1, cs, sn);
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
__global__ void __launch_bounds__(256, 3)
compress_kernel(const T *__restrict__ C, const T *__restrict__ Z, const float *__restrict__ bias,
                const T *__restrict__ Cb, const T *__restrict__ Zb, const float *__restrict__ biasb,
                T *__restrict__ out, T *__restrict__ raw_out, int64_t B, int64_t n, int c, int m,
                int overlap, int64_t E, int64_t Eg, const __grid_constant__ RopeFreqs rope) {
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
    // the next slot's rows are loaded before this slot's arithmetic, so two
    // slots' loads are in flight per thread
    float z[N], v[N];
    if (slots > 0) {
        Vec<T>::load_stream(Zs + row0 * c + ch0, z);
        Vec<T>::load_stream(Cs + row0 * c + ch0, v);
    }
    for (int s = 0; s < slots; s++) {
        float zn[N], vn[N], bs[N];
        const int64_t row = row0 + s;
        if (s + 1 < slots) {
            Vec<T>::load_stream(Zs + (row + 1) * c + ch0, zn);
            Vec<T>::load_stream(Cs + (row + 1) * c + ch0, vn);
        }
        Vec<float>::load(bias + (int64_t)s * c + ch0, bs);
        if constexpr (N == 8) Vec<float>::load(bias + (int64_t)s * c + ch0 + 4, bs + 4);
#pragma unroll
        for (int i = 0; i < N; i++) softmax_step<T>(z[i] + bs[i], v[i], mx[i], den[i], acc[i]);
        if (raw_out != nullptr) {
            rotate_vec<T>(v, ch0, row, rope);
            Vec<T>::store(raw_out + (b * n + row) * c + ch0, v);
        }
#pragma unroll
        for (int i = 0; i < N; i++) { z[i] = zn[i]; v[i] = vn[i]; }
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
                     int64_t Eg, const __grid_constant__ RopeFreqs rope) {
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

// Sum over the CTA (every thread calls it; a fixed order, so the result does
// not depend on timing).  `red` holds one float per warp.
__device__ __forceinline__ float block_sum(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();                        // the previous sum's readers are done
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); i++) t += red[i];
    return t;
}

// RMSNorm of one vector spread over the CTA's threads (N channels each,
// zeros for threads past the row): x / sqrt(mean(x^2) + eps) * g.
template <int N>
__device__ __forceinline__ void rms_scale(float *v, bool active, int ch0, int c, const float *g, float eps,
                                          float *red) {
    float ss = 0.f;
    if (active)
#pragma unroll
        for (int i = 0; i < N; i++) ss = fmaf(v[i], v[i], ss);
    ss = block_sum(ss, red);
    const float rs = 1.0f / sqrtf(ss / (float)c + eps);
    if (active)
#pragma unroll
        for (int i = 0; i < N; i++) v[i] = v[i] * rs * g[ch0 + i];
}

// Compression with the KV RMSNorm [book ch.7 "Query and KV normalization"]:
// one CTA per (sequence, block), one thread per channel vector.  The slots
// are pooled in the order of compress_kernel; each stored raw row and the
// pooled entry are normalised over their c channels, then rotated, then
// rounded to the storage type.
template <typename T>
__global__ void __launch_bounds__(256)
compress_norm_kernel(const T *__restrict__ C, const T *__restrict__ Z, const float *__restrict__ bias,
                     const T *__restrict__ Cb, const T *__restrict__ Zb, const float *__restrict__ biasb,
                     T *__restrict__ out, T *__restrict__ raw_out, int64_t n, int c, int m, int overlap,
                     int64_t E, int64_t Eg, const __grid_constant__ RopeFreqs rope, const float *__restrict__ gain, float eps) {
    constexpr int N = Vec<T>::N;
    __shared__ float red[8];
    const int V = c / N;
    const int tid = threadIdx.x;
    const bool active = tid < V;
    const int ch0 = active ? tid * N : 0;
    const int64_t e = blockIdx.x % Eg, b = blockIdx.x / Eg;
    const T *Cs = C + b * n * c;
    const T *Zs = Z + b * n * c;
    float mx[N], den[N], acc[N];
#pragma unroll
    for (int i = 0; i < N; i++) { mx[i] = -INFINITY; den[i] = 0.f; acc[i] = 0.f; }
    const int64_t row0 = e * m;
    const int slots = (int)((n - row0) < m ? (n - row0) : m);
    for (int s = 0; s < slots; s++) {
        float z[N], v[N], bs[N];
        const int64_t row = row0 + s;
        if (active) {
            Vec<T>::load_stream(Zs + row * c + ch0, z);
            Vec<T>::load_stream(Cs + row * c + ch0, v);
            Vec<float>::load(bias + (int64_t)s * c + ch0, bs);
            if constexpr (N == 8) Vec<float>::load(bias + (int64_t)s * c + ch0 + 4, bs + 4);
#pragma unroll
            for (int i = 0; i < N; i++) softmax_step<T>(z[i] + bs[i], v[i], mx[i], den[i], acc[i]);
        }
        if (raw_out != nullptr) {
            rms_scale<N>(v, active, ch0, c, gain, eps, red);
            if (active) {
                rotate_vec<T>(v, ch0, row, rope);
                Vec<T>::store(raw_out + (b * n + row) * c + ch0, v);
            }
        }
    }
    if (e >= E) return;                     // partial tail block: raw rows only
    if (overlap && e > 0 && active) {
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
    for (int i = 0; i < N; i++) o[i] = active ? acc[i] / den[i] : 0.f;
    rms_scale<N>(o, active, ch0, c, gain, eps, red);
    if (!active) return;
    rotate_vec<T>(o, ch0, (e + 1) * m - 1, rope);
    Vec<T>::store(out + (b * E + e) * c + ch0, o);
}

cudaError_t launch_compress(csa_dtype dt, int64_t B, int64_t n, int c, int m, int overlap,
                            const void *C, const void *Z, const float *bias, const void *Cb,
                            const void *Zb, const float *biasb, void *out, void *raw_out,
                            const RopeFreqs &rope, const float *gain, float eps, cudaStream_t st) {
    if (gain != nullptr) {
        const int64_t E = n / m;
        const int64_t Eg = raw_out ? (n + m - 1) / m : E;
        const int N = dt == CSA_BF16 ? 8 : 4;
        const int V = c / N;
        if (V > 256) return cudaErrorInvalidValue;
        if (B * Eg == 0) return cudaSuccess;
        const int threads = (V + 31) / 32 * 32;
        if (dt == CSA_BF16) {
            using T = __nv_bfloat16;
            compress_norm_kernel<T><<<(unsigned)(B * Eg), threads, 0, st>>>(
                (const T *)C, (const T *)Z, bias, (const T *)Cb, (const T *)Zb, biasb, (T *)out, (T *)raw_out,
                n, c, m, overlap, E, Eg, rope, gain, eps);
        } else {
            compress_norm_kernel<float><<<(unsigned)(B * Eg), threads, 0, st>>>(
                (const float *)C, (const float *)Z, bias, (const float *)Cb, (const float *)Zb, biasb,
                (float *)out, (float *)raw_out, n, c, m, overlap, E, Eg, rope, gain, eps);
        }
        count_launches(1);
        return cudaGetLastError();
    }
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

// ------------------------------------------------------------------ decode
//
// Incremental decode state ["DeepSeek-V4" book ch.5 "What is retained during
// decode"; ch.13 "Bounded state per request"]: each arriving token's raw row
// goes into a window ring (slot t mod n_win, rotated at t), its compressor
// inputs into a tail of the current block's slots (plus, in the two-branch
// mode, the previous block's second-branch rows); when the token completes a
// block, the block is compressed into the growing caches.  The arithmetic of
// one block is exactly that of the prefill kernels above for the same (m, c,
// dtype, overlap): the slots in the same order (or, for long one-branch
// blocks, the same slot groups and the same merge), so an entry built here is
// bitwise the entry the prefill path builds.
struct AppendArgs {
    const void *C, *Z, *Cb, *Zb, *Ck, *Zk, *Ckb, *Zkb;   // new token's rows: [B, c] / [B, dI]
    const float *bias, *biasb, *biask, *biaskb;           // [m, c] / [m, dI]
    const int64_t *t;                                     // [B] position of the new token
    void *win;                                            // [B, n_win, c] window ring
    void *tail;                                           // [B, S, R] compressor inputs
    void *kvc, *kIc;                                      // [B, E_cap, c] / [B, E_cap, dI]
    unsigned *status;
    int64_t E_cap;
    int c, dI, m, overlap, n_win, S, R;
    const float *kv_norm;                                 // RMSNorm gains of the KV (or nullptr)
    float norm_eps;
    RopeFreqs rope;                                       // main KV (keys carry none)
};

// Tail row layout (elements): C | Z | Ck | Zk, then (two-branch) Cb | Zb | Ckb | Zkb.
__host__ __device__ inline int tail_off(int c, int dI, int part) {
    const int w[8] = {c, c, dI, dI, c, c, dI, dI};
    int o = 0;
    for (int i = 0; i < part; i++) o += w[i];
    return o;
}

// A coherent 16-byte load of tail rows this kernel may have just written
// (the read-only path of Vec::load is not coherent with writes of the same
// kernel).
__device__ __forceinline__ void ld_tail(const float *p, float *o) {
    asm volatile("ld.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(o[0]), "=f"(o[1]), "=f"(o[2]), "=f"(o[3])
                 : "l"(p)
                 : "memory");
}
__device__ __forceinline__ void ld_tail(const __nv_bfloat16 *p, float *o) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    Vec<__nv_bfloat16>::unpack(v, o);
}

// One block's entry over `width` channels into dst: rows of slot s at
// tail + row(s) * R (+ part offsets), the same order and merge as the prefill
// kernel that launch_compress picks for these sizes.
template <typename T>
__device__ void append_entry(const AppendArgs &a, const T *tl, int width, int offC, int offZ,
                             int offCb, int offZb, const float *bias, const float *biasb,
                             int64_t i, int base, int prev_base, const RopeFreqs *rope, T *dst,
                             const float *gain, float (*part)[3][Vec<T>::N], float *red) {
    constexpr int N = Vec<T>::N;
    const int V = width / N;
    const int tid = threadIdx.x;
    // with the KV norm, every block takes the one-thread-per-vector order of
    // the prefill norm kernel
    const bool wide = a.m >= 16 && !a.overlap && V <= CW_THREADS && gain == nullptr;
    float mx[N], den[N], acc[N];
#pragma unroll
    for (int q = 0; q < N; q++) { mx[q] = -INFINITY; den[q] = 0.f; acc[q] = 0.f; }
    if (!wide && gain != nullptr) {
        const bool active = tid < V;
        const int ch0 = active ? tid * N : 0;
        if (active) {
            for (int s = 0; s < a.m; s++) {
                float z[N], v[N], bs[N];
                const T *row = tl + (int64_t)(base + s) * a.R;
                ld_tail(row + offZ + ch0, z);
                ld_tail(row + offC + ch0, v);
                Vec<float>::load(bias + (int64_t)s * width + ch0, bs);
                if constexpr (N == 8) Vec<float>::load(bias + (int64_t)s * width + ch0 + 4, bs + 4);
#pragma unroll
                for (int q = 0; q < N; q++) softmax_step<T>(z[q] + bs[q], v[q], mx[q], den[q], acc[q]);
            }
            if (a.overlap && i > 0) {
                for (int s = 0; s < a.m; s++) {
                    float z[N], v[N], bs[N];
                    const T *row = tl + (int64_t)(prev_base + s) * a.R;
                    ld_tail(row + offZb + ch0, z);
                    ld_tail(row + offCb + ch0, v);
                    Vec<float>::load(biasb + (int64_t)s * width + ch0, bs);
                    if constexpr (N == 8) Vec<float>::load(biasb + (int64_t)s * width + ch0 + 4, bs + 4);
#pragma unroll
                    for (int q = 0; q < N; q++) softmax_step<T>(z[q] + bs[q], v[q], mx[q], den[q], acc[q]);
                }
            }
        }
        float o[N];
#pragma unroll
        for (int q = 0; q < N; q++) o[q] = active ? acc[q] / den[q] : 0.f;
        rms_scale<N>(o, active, ch0, width, gain, a.norm_eps, red);
        if (!active) return;
        if (rope) rotate_vec<T>(o, ch0, (i + 1) * a.m - 1, *rope);
        Vec<T>::store(dst + ch0, o);
        return;
    }
    if (!wide) {
        if (tid >= V) return;
        const int ch0 = tid * N;
        for (int s = 0; s < a.m; s++) {
            float z[N], v[N], bs[N];
            const T *row = tl + (int64_t)(base + s) * a.R;
            ld_tail(row + offZ + ch0, z);
            ld_tail(row + offC + ch0, v);
            Vec<float>::load(bias + (int64_t)s * width + ch0, bs);
            if constexpr (N == 8) Vec<float>::load(bias + (int64_t)s * width + ch0 + 4, bs + 4);
#pragma unroll
            for (int q = 0; q < N; q++) softmax_step<T>(z[q] + bs[q], v[q], mx[q], den[q], acc[q]);
        }
        if (a.overlap && i > 0) {
            for (int s = 0; s < a.m; s++) {
                float z[N], v[N], bs[N];
                const T *row = tl + (int64_t)(prev_base + s) * a.R;
                ld_tail(row + offZb + ch0, z);
                ld_tail(row + offCb + ch0, v);
                Vec<float>::load(biasb + (int64_t)s * width + ch0, bs);
                if constexpr (N == 8) Vec<float>::load(biasb + (int64_t)s * width + ch0 + 4, bs + 4);
#pragma unroll
                for (int q = 0; q < N; q++) softmax_step<T>(z[q] + bs[q], v[q], mx[q], den[q], acc[q]);
            }
        }
        float o[N];
#pragma unroll
        for (int q = 0; q < N; q++) o[q] = acc[q] / den[q];
        if (rope) rotate_vec<T>(o, ch0, (i + 1) * a.m - 1, *rope);
        Vec<T>::store(dst + ch0, o);
        return;
    }
    // long one-branch block: thread (g, v) takes slots g, g + G, ..., then one
    // thread per vector merges the G partial states (as compress_wide_kernel)
    const int G = CW_THREADS / V;
    const int v = tid % V, grp = tid / V;
    const int ch0 = v * N;
    if (grp < G) {
        for (int s = grp; s < a.m; s += G) {
            float z[N], x[N], bs[N];
            const T *row = tl + (int64_t)(base + s) * a.R;
            ld_tail(row + offZ + ch0, z);
            ld_tail(row + offC + ch0, x);
            Vec<float>::load(bias + (int64_t)s * width + ch0, bs);
            if constexpr (N == 8) Vec<float>::load(bias + (int64_t)s * width + ch0 + 4, bs + 4);
#pragma unroll
            for (int q = 0; q < N; q++) softmax_step<T>(z[q] + bs[q], x[q], mx[q], den[q], acc[q]);
        }
    }
#pragma unroll
    for (int q = 0; q < N; q++) {
        part[tid][0][q] = mx[q];
        part[tid][1][q] = den[q];
        part[tid][2][q] = acc[q];
    }
    __syncthreads();
    if (grp == 0) {
#pragma unroll
        for (int q = 0; q < N; q++) {
            float M = -INFINITY;
            for (int g = 0; g < G; g++) M = fmaxf(M, part[g * V + v][0][q]);
            float d = 0.f, s_ = 0.f;
            for (int g = 0; g < G; g++) {
                const float mq = part[g * V + v][0][q];
                if (mq == -INFINITY) continue;
                const float sc = __expf(mq - M);
                d = fmaf(part[g * V + v][1][q], sc, d);
                s_ = fmaf(part[g * V + v][2][q], sc, s_);
            }
            mx[q] = s_ / d;
        }
        if (rope) rotate_vec<T>(mx, ch0, (i + 1) * a.m - 1, *rope);
        Vec<T>::store(dst + ch0, mx);
    }
    __syncthreads();
}

// One CTA per sequence.
template <typename T>
__global__ void __launch_bounds__(CW_THREADS) decode_append_kernel(const __grid_constant__ AppendArgs a) {
    constexpr int N = Vec<T>::N;
    __shared__ float part[CW_THREADS][3][N];
    __shared__ float red[CW_THREADS / 32];
    const int64_t b = blockIdx.x;
    const int64_t t = a.t[b];
    const int tid = threadIdx.x;
    if (t < 0) return;
    T *tl = (T *)a.tail + b * (int64_t)a.S * a.R;
    const int slot = (int)(t % a.S);
    T *trow = tl + (int64_t)slot * a.R;
    // the new token's rows into its tail slot, and its raw row, rotated at t,
    // into the window ring
    const int nparts = a.overlap ? 8 : 4;
    const void *src[8] = {a.C, a.Z, a.Ck, a.Zk, a.Cb, a.Zb, a.Ckb, a.Zkb};
    for (int p = 0; p < nparts; p++) {
        const int wdt = (p & 2) ? a.dI : a.c;
        if (src[p] == nullptr) continue;
        const T *s = (const T *)src[p] + b * wdt;
        T *d = trow + tail_off(a.c, a.dI, p);
        if (p == 0) {
            // one vector per thread (c <= 256 vectors): the raw row, normalised
            // when asked, rotated at t, into the ring
            const bool active = tid * N < wdt;
            const int ch0 = active ? tid * N : 0;
            float v[N];
            if (active) {
                Vec<T>::load(s + ch0, v);
                Vec<T>::store(d + ch0, v);
            }
            if (a.n_win > 0) {
                if (a.kv_norm) rms_scale<N>(v, active, ch0, wdt, a.kv_norm, a.norm_eps, red);
                if (active) {
                    rotate_vec<T>(v, ch0, t, a.rope);
                    Vec<T>::store((T *)a.win + (b * a.n_win + t % a.n_win) * a.c + ch0, v);
                }
            }
            continue;
        }
        for (int ch0 = tid * N; ch0 < wdt; ch0 += CW_THREADS * N) {
            float v[N];
            Vec<T>::load(s + ch0, v);
            Vec<T>::store(d + ch0, v);
        }
    }
    if ((t + 1) % a.m != 0) return;
    __syncthreads();                        // the block's last row is in the tail
    const int64_t i = (t + 1) / a.m - 1;    // the block this token completes
    if (i >= a.E_cap) {
        if (tid == 0) atomicOr(a.status, ST_BAD_INDEX);
        return;
    }
    const int base = (int)((i * a.m) % a.S);
    const int prev_base = (int)(((i + a.S / a.m - 1) * a.m) % a.S);
    append_entry<T>(a, tl, a.c, tail_off(a.c, a.dI, 0), tail_off(a.c, a.dI, 1), tail_off(a.c, a.dI, 4),
                    tail_off(a.c, a.dI, 5), a.bias, a.biasb, i, base, prev_base, &a.rope,
                    (T *)a.kvc + (b * a.E_cap + i) * a.c, a.kv_norm, part, red);
    if (a.Ck == nullptr) return;
    __syncthreads();
    append_entry<T>(a, tl, a.dI, tail_off(a.c, a.dI, 2), tail_off(a.c, a.dI, 3), tail_off(a.c, a.dI, 6),
                    tail_off(a.c, a.dI, 7), a.biask, a.biaskb, i, base, prev_base, nullptr,
                    (T *)a.kIc + (b * a.E_cap + i) * a.dI, nullptr, part, red);
}

int decode_tail_slots(int m, int overlap) { return overlap ? 2 * m : m; }
int decode_tail_width(int c, int dI, int overlap) { return overlap ? 4 * c + 4 * dI : 2 * c + 2 * dI; }

cudaError_t launch_decode_append(csa_dtype dt, int64_t B, const DecodeAppend &d, cudaStream_t st) {
    if (B == 0) return cudaSuccess;
    AppendArgs a;
    a.C = d.C; a.Z = d.Z; a.Cb = d.Cb; a.Zb = d.Zb; a.Ck = d.Ck; a.Zk = d.Zk; a.Ckb = d.Ckb; a.Zkb = d.Zkb;
    a.bias = d.bias; a.biasb = d.biasb; a.biask = d.biask; a.biaskb = d.biaskb;
    a.t = d.t; a.win = d.win; a.tail = d.tail; a.kvc = d.kvc; a.kIc = d.kIc; a.status = d.status;
    a.E_cap = d.E_cap; a.c = d.c; a.dI = d.dI; a.m = d.m; a.overlap = d.overlap; a.n_win = d.n_win;
    a.kv_norm = d.kv_norm; a.norm_eps = d.norm_eps;
    a.S = decode_tail_slots(d.m, d.overlap);
    a.R = decode_tail_width(d.c, d.dI, d.overlap);
    a.rope = d.rope;
    if (dt == CSA_BF16) decode_append_kernel<__nv_bfloat16><<<(unsigned)B, CW_THREADS, 0, st>>>(a);
    else decode_append_kernel<float><<<(unsigned)B, CW_THREADS, 0, st>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace csa
