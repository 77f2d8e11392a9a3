// Shared device helpers of libcsa (storage types, RoPE angles, status bits).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/csa.h"

namespace csa {

// status-word bits, OR-ed by kernels into ws[0] (never a trap)
enum : unsigned {
    ST_BAD_INDEX = 1u,     // a selected index outside [0, E)
    ST_NO_WINDOW_ROW = 2u, // a window position missing from kv_raw
    ST_TIMEOUT = 4u,       // a bounded wait ran out
};

constexpr int MAX_ROPE_PAIRS = 256;

// Per-pair RoPE frequencies theta^(-2i/r), computed on the host in double.
struct RopeFreqs {
    int pairs;    // r / 2
    int first;    // c - r: first rotary channel
    double w[MAX_ROPE_PAIRS];       // theta^(-2i/r)
    float fh[MAX_ROPE_PAIRS];       // w / (2 pi) as fh + fl (fh the float
    float fl[MAX_ROPE_PAIRS];       // nearest to it, fl the float nearest the rest)
};

// cos and sin of the angle p * w_i of rotary pair i.
//
// |p| < 2^24 (every position of a 16M-token context): the angle is reduced in
// turns, in fp32 only.  With f = w / (2 pi) split as fh + fl, p * fh is split
// exactly into hi + lo by one fma (the fma two-product of Ogita, Rump and
// Oishi, 2005; p and fh are floats); hi - rint(hi) is
// exact, so t = frac(p f) = (hi - rint(hi)) + (p * fl + lo) carries one
// rounding of about 2^-25 turns, and sincospif gives sin / cos of 2 pi t.  (The
// angle itself reaches 2^20 rad, where a float product p * w would already be
// off by hundredths of a radian.)
// Larger |p|: the same reduction in double, by 2 pi split in two parts
// (Cody-Waite style), then the float sine and cosine of the reduced angle.
__device__ __forceinline__ void rope_cos_sin(const RopeFreqs &rf, int64_t p, int i, float &cs, float &sn) {
    if (p > -(1LL << 24) && p < (1LL << 24)) {
        const float pf = (float)(int)p;     // through int32: a 64-bit convert runs on the fp64 pipe
        const float fh = rf.fh[i];
        const float hi = pf * fh;
        const float lo = fmaf(pf, fh, -hi);
        const float t = (hi - rintf(hi)) + fmaf(pf, rf.fl[i], lo);
        sincospif(2.0f * t, &sn, &cs);
        return;
    }
    const double two_pi_hi = 6.283185307179586;           // 2*pi rounded to double
    const double two_pi_lo = 2.4492935982947064e-16;      // 2*pi - two_pi_hi
    const double inv_two_pi = 0.15915494309189535;
    const double a = (double)p * rf.w[i];
    const double k = rint(a * inv_two_pi);
    double r = fma(-k, two_pi_hi, a);
    r = fma(-k, two_pi_lo, r);
    sincosf((float)r, &sn, &cs);
}

// ---------------------------------------------------------------- storage
template <typename T> struct Vec;   // 16-byte vector of a storage type

template <> struct Vec<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void load(const float *p, float *o) {
        float4 v = __ldg(reinterpret_cast<const float4 *>(p));
        o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
    }
    __device__ __forceinline__ static void load_stream(const float *p, float *o) {
        float4 v = __ldcs(reinterpret_cast<const float4 *>(p));
        o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
    }
    __device__ __forceinline__ static void store(float *p, const float *o) {
        *reinterpret_cast<float4 *>(p) = make_float4(o[0], o[1], o[2], o[3]);
    }
};

template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void unpack(uint4 v, float *o) {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float2 f = __bfloat1622float2(h[i]);
            o[2 * i] = f.x; o[2 * i + 1] = f.y;
        }
    }
    __device__ __forceinline__ static void load(const __nv_bfloat16 *p, float *o) {
        unpack(__ldg(reinterpret_cast<const uint4 *>(p)), o);
    }
    __device__ __forceinline__ static void load_stream(const __nv_bfloat16 *p, float *o) {
        unpack(__ldcs(reinterpret_cast<const uint4 *>(p)), o);
    }
    __device__ __forceinline__ static void store(__nv_bfloat16 *p, const float *o) {
        uint4 v;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; i++) h[i] = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
        *reinterpret_cast<uint4 *>(p) = v;
    }
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float &d, float x) { d = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16 &d, float x) { d = __float2bfloat16_rn(x); }

// number of entries visible at position t: (j+1)*m <= t+1, clipped to [0, E]
__device__ __forceinline__ int64_t visible_count(int64_t t, int m, int64_t E) {
    int64_t v = (t + 1) / m;
    if (t + 1 < 0) v = 0;
    return v < E ? v : E;
}

// order-preserving uint32 key of a float score: larger score -> larger key;
// -0.0 is folded onto +0.0 so that the two tie.
__device__ __forceinline__ uint32_t score_key(float s) {
    uint32_t u = __float_as_uint(s);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace csa
