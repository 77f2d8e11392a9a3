// Low-precision cache formats of the production layer, written by the
// quantisers here and read by the decode indexer below and by the attention
// kernel's loaders.
//
// ["DeepSeek-V4" book ch.8 "The main compressed-entry payload": a KV entry
// keeps its 448 non-rotary dims in FP8 and its 64 rotary dims in BF16, 576
// bytes; ch.16 "The two main FP4 targets", "Why use fine-grained scales?":
// indexer queries and keys in FP4 with one scale per 1 x 32 tile; "BF16 index
// scores": the selector ranks BF16 scores.]
//
// FP8 KV record (c = 512, r = 64), 592 bytes per entry:
//   bytes   0 .. 447  E4M3 codes of dims 0 .. 447 (finite variant, largest 448)
//   bytes 448 .. 575  BF16 values of the rotary dims 448 .. 511
//   bytes 576 .. 591  four fp32 scales, one per group of dims [0,128),
//                     [128,256), [256,384), [384,448): scale = amax / 448
//                     (1 for an all-zero group); code = E4M3(x / scale),
//                     nearest-even, saturating at +-448, the quotient formed
//                     in fp32.
// MXFP4 rows of d = 128 values, planar over a whole cache of `rows` rows:
//   codes  [rows][64] bytes: value 2i in the low nibble of byte i, 2i+1 in
//          the high nibble; E2M1 (sign bit 3; magnitudes 0, .5, 1, 1.5, 2, 3,
//          4, 6), nearest-even, saturating at +-6;
//   scales [rows4][4] bytes after the codes, rows4 = rows rounded up to a
//          multiple of 4: exponent + 127 of the block's power-of-two scale
//          2^(floor(log2 amax) - 2), clipped to [-127, 127] (scale 1 for an
//          all-zero block).
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace csa {

// ---------------------------------------------------------------- encoders

// Nearest-even E4M3 code of x (finite variant, saturating at +-448): the
// spacing is 2^(e-3) in the binade [2^e, 2^(e+1)) for e >= -6 and 2^-9 below.
__device__ __forceinline__ uint32_t e4m3_encode(float x) {
    const uint32_t s = (__float_as_uint(x) >> 24) & 0x80u;
    const float a = fabsf(x);
    if (!(a < 464.f)) return s | 0x7Eu;                   // 448 (464 itself ties down to 448)
    const int e = (int)((__float_as_uint(a) >> 23) & 0xFFu) - 127;
    if (e < -6) return s | (uint32_t)rintf(a * 512.f);    // subnormal; 8 is the smallest normal
    const float q = rintf(a * __uint_as_float((uint32_t)(127 + 3 - e) << 23));   // 8 .. 16
    int mant = (int)q - 8, E = e + 7;
    if (mant == 8) { mant = 0; E += 1; }
    return s | ((uint32_t)E << 3) | (uint32_t)mant;
}

// Nearest-even E2M1 code of v (|v| < 8 here), saturating at +-6.  Ties go to
// the even mantissa: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2,
// 3.5 -> 4, 5 -> 4.
__device__ __forceinline__ uint32_t e2m1_encode(float v) {
    const uint32_t s = (__float_as_uint(v) >> 28) & 0x8u;
    const float a = fabsf(v);
    uint32_t m;
    if (a <= 0.25f) m = 0;
    else if (a < 0.75f) m = 1;
    else if (a <= 1.25f) m = 2;
    else if (a < 1.75f) m = 3;
    else if (a <= 2.5f) m = 4;
    else if (a < 3.5f) m = 5;
    else if (a <= 5.f) m = 6;
    else m = 7;
    return s | m;
}

// Exponent of a block's MXFP4 scale from its largest magnitude.
__device__ __forceinline__ int mx_exponent(float amax) {
    if (!(amax > 0.f)) return 0;
    const int E32 = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
    if (E32 == 0) return -127;                            // below 2^-126: clipped
    const int e = E32 - 127 - 2;
    return e < -127 ? -127 : e;
}

__device__ __forceinline__ float pow2f(int e) {          // 2^e for -149 <= e <= 127
    if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
    return __uint_as_float(1u << (e + 149));
}

// ------------------------------------------------------------- quantisers

// One warp per entry: lane l holds dims 16 l .. 16 l + 15.
template <typename T>
__global__ void __launch_bounds__(256) quant_kv_fp8_kernel(const T *__restrict__ src, uint8_t *__restrict__ dst,
                                                           int64_t rows) {
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const T *s = src + row * 512 + lane * 16;
    float v[16];
    if constexpr (sizeof(T) == 2) {
        Vec<T>::load(s, v);
        Vec<T>::load(s + 8, v + 8);
    } else {
#pragma unroll
        for (int q = 0; q < 4; q++) Vec<float>::load((const float *)s + 4 * q, v + 4 * q);
    }
    uint8_t *d = dst + row * KV8_BYTES;
    if (lane >= 28) {                                     // rotary dims 448 .. 511: BF16
        uint4 o[2];
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(o);
#pragma unroll
        for (int q = 0; q < 8; q++) h[q] = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
        uint4 *dd = reinterpret_cast<uint4 *>(d + 448 + (lane - 28) * 32);
        dd[0] = o[0];
        dd[1] = o[1];
    }
    // group amax over the 8 lanes of a 128-dim group (lanes 24 .. 27: 64 dims)
    float am = 0.f;
#pragma unroll
    for (int q = 0; q < 16; q++) am = fmaxf(am, fabsf(v[q]));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        const float t = __shfl_xor_sync(0xffffffffu, am, o);
        if (((lane ^ o) >> 3) == (lane >> 3) && (lane < 28) == ((lane ^ o) < 28)) am = fmaxf(am, t);
    }
    const float scale = am > 0.f ? am / 448.f : 1.f;
    if (lane < 28) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            w[q] = 0;
#pragma unroll
            for (int u = 0; u < 4; u++) w[q] |= e4m3_encode(v[4 * q + u] / scale) << (8 * u);
        }
        *reinterpret_cast<uint4 *>(d + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        if ((lane & 7) == 0) reinterpret_cast<float *>(d + 576)[lane >> 3] = scale;
    }
}

// Four threads per row of 128 values, one 32-value block each.
template <typename T>
__global__ void __launch_bounds__(256) quant_mxfp4_kernel(const T *__restrict__ src, uint8_t *__restrict__ codes,
                                                          uint8_t *__restrict__ scales, int64_t rows) {
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t row = g >> 2;
    const int blk = (int)(g & 3);
    if (row >= rows) return;
    const T *s = src + row * 128 + blk * 32;
    float v[32];
#pragma unroll
    for (int q = 0; q < 32; q += Vec<T>::N) Vec<T>::load(s + q, v + q);
    float am = 0.f;
#pragma unroll
    for (int q = 0; q < 32; q++) am = fmaxf(am, fabsf(v[q]));
    const int e = mx_exponent(am);
    const float inv = pow2f(-e);                          // exact: -e <= 127
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; q++) {
        w[q] = 0;
#pragma unroll
        for (int u = 0; u < 8; u++) w[q] |= e2m1_encode(v[8 * q + u] * inv) << (4 * u);
    }
    *reinterpret_cast<uint4 *>(codes + row * 64 + blk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    scales[row * 4 + blk] = (uint8_t)(e + 127);
}

size_t mxfp4_bytes(int64_t rows) { return (size_t)rows * 64 + (size_t)((rows + 3) / 4) * 16; }

cudaError_t launch_quant_kv_fp8(csa_dtype dt, int64_t rows, const void *src, void *dst, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((rows * 32 + 255) / 256);
    if (dt == CSA_BF16)
        quant_kv_fp8_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>((const __nv_bfloat16 *)src, (uint8_t *)dst, rows);
    else
        quant_kv_fp8_kernel<float><<<blocks, 256, 0, st>>>((const float *)src, (uint8_t *)dst, rows);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_quant_mxfp4(csa_dtype dt, int64_t rows, const void *src, void *dst, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    uint8_t *codes = (uint8_t *)dst, *scales = codes + (size_t)rows * 64;
    const unsigned blocks = (unsigned)((rows * 4 + 255) / 256);
    if (dt == CSA_BF16)
        quant_mxfp4_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>((const __nv_bfloat16 *)src, codes, scales, rows);
    else
        quant_mxfp4_kernel<float><<<blocks, 256, 0, st>>>((const float *)src, codes, scales, rows);
    count_launches(1);
    return cudaGetLastError();
}

// ---------------------------------------------------- FP4 decode indexer
//
// Decode scores over MXFP4 keys (one query per sequence, 64 heads x 128):
//   I[b, j] = bf16( sum_h w[b,h] * ReLU(q4[b,h] . k4[b,j]) )
// where q4 / k4 are qI / kI through MXFP4 (qI is quantised here, in the
// same way as quant_mxfp4).  Both operands enter a tcgen05.mma of kind f16
// exactly: a row's 4 block scales are 2^e_b, and the row is stored as
// E2M1 value * 2^(e_b - E) in f16 with E = max_b e_b (exact while a row's
// blocks span at most 23 binades; a block further below its row's largest
// contributes under 2^-24 of it, the fp32 accumulation's own resolution).
// The factors 2^E of the key row and of the query head come out of the
// product: ReLU commutes with a positive scale, so the head's factor joins
// w[h] and the key's multiplies the sum.
//
// Warp roles (one persistent CTA per SM; the B x E entry tiles are split
// evenly over the CTAs, as in the bf16 decode indexer):
//   warp 0      TMA producer: per 128-key tile, the 8 KB of codes and the
//               tile's scale bytes into a staging ring;
//   warp 1      TMEM allocator and MMA issuer for the even tiles, warp 14
//               for the odd ones (each with its own accumulator);
//   warps 2-5   epilogue: head sum, key factor, BF16 rounding, stores;
//   warps 6-13  converters in two groups of four taking alternate tiles:
//               each staged key tile into an f16 A tile (128-byte swizzle,
//               K-major); the first group also converts the item's query
//               into the f16 B tile (and the scaled head weights).
struct Fp4Cfg {
    static constexpr int AST = 3;                         // f16 A tiles
    static constexpr int SST = 8;                         // staging slots
    static constexpr int A_BYTES = 128 * 128 * 2;
    static constexpr int B_BYTES = 64 * 128 * 2;
    static constexpr int CODE_BYTES = 128 * 64;
    static constexpr int SC_ROWS = 33;                    // 16-byte scale rows covering 128 keys
    static constexpr int SC_BYTES = SC_ROWS * 16;
    static constexpr int STG_BYTES = CODE_BYTES + 640;    // codes + scales, 128-byte multiple
    static constexpr int NEK = 4;                         // ring of key-row exponents
    static constexpr int OFF_A = 0;
    static constexpr int OFF_S = OFF_A + AST * A_BYTES;
    static constexpr int OFF_B = OFF_S + SST * STG_BYTES;
    static constexpr int OFF_MISC = OFF_B + B_BYTES;
    static constexpr int MISC_BYTES = 4096;               // barriers, wq [2][64], ek [NEK][128]
    static constexpr int SMEM = OFF_MISC + MISC_BYTES + 1024;
    static constexpr int EPI0 = 2;                        // epilogue warps 2 .. 5
    static constexpr int CONV0 = 6;                       // converter warps 6 .. 13 (two groups of 4)
    static constexpr int MMA2 = 14;                       // second MMA warp (odd tiles)
    static constexpr int THREADS = 480;
    static constexpr int TMEM_COLS = 128;
};

struct Fp4IdxArgs {
    const __nv_bfloat16 *qI;   // [B, 64, 128]
    const float *w;            // [B, 64]
    const int64_t *q_pos;      // [B]
    float *scores;             // [B, E]
    unsigned *status;
    int64_t E;
    int B, m, tps;
    long long spin;
};

__device__ __forceinline__ bool fp4_item(const Fp4IdxArgs &a, int cta, int G, int r, int &b, int &jt0, int &jt1) {
    const long long TT = (long long)a.B * a.tps;
    const long long g0 = TT * cta / G, g1 = TT * (cta + 1) / G;
    long long g = g0;
    for (int i = 0; i < r; i++) {
        if (g >= g1) return false;
        const long long bnd = (g / a.tps + 1) * a.tps;
        g = bnd < g1 ? bnd : g1;
    }
    if (g >= g1) return false;
    const long long row = g / a.tps;
    b = (int)row;
    jt0 = (int)(g % a.tps);
    const long long end = (row + 1) * a.tps < g1 ? (row + 1) * a.tps : g1;
    jt1 = (int)(end - row * a.tps);
    const int64_t nv = visible_count(a.q_pos[row], a.m, a.E);
    const int lim = (int)((nv + 127) / 128);
    if (jt1 > lim) jt1 = lim;
    return true;
}

// generic-proxy shared-memory writes -> visible to the tensor core's reads
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2^rel as f16 bits (rel <= 0); 0 below the smallest subnormal.
__device__ __forceinline__ uint32_t f16_pow2(int rel) {
    if (rel >= -14) return (uint32_t)(rel + 15) << 10;
    if (rel >= -24) return 1u << (rel + 24);
    return 0u;
}

// 4 code bytes (8 E2M1 values) times 2^rel into one 16-byte f16 chunk.
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t cw, uint32_t s2, uint32_t *o) {
#pragma unroll
    for (int u = 0; u < 4; u++) {
        uint32_t h;
        asm("{\n\t.reg .b8 t;\n\t"
            "cvt.u8.u32 t, %1;\n\t"
            "cvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
            : "=r"(h)
            : "r"(cw >> (8 * u)));
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(h) : "r"(h), "r"(s2));
        o[u] = h;
    }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint32_t *v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]),
                 "r"(v[3])
                 : "memory");
}

__device__ __forceinline__ int swz_off(int row, int chunk) {   // K-major, 128-byte rows, 8-row atoms
    return (row >> 3) * 1024 + (row & 7) * 128 + (((chunk ^ row) & 7) << 4);
}

__global__ void __launch_bounds__(Fp4Cfg::THREADS, 1)
indexer_fp4_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_sc,
                   const __grid_constant__ Fp4IdxArgs a) {
    using Cfg = Fp4Cfg;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem + Cfg::OFF_A, *sS = smem + Cfg::OFF_S, *sB = smem + Cfg::OFF_B;
    uint8_t *misc = smem + Cfg::OFF_MISC;
    uint64_t *bar = (uint64_t *)misc;
    uint64_t *sfull = bar, *sempty = bar + Cfg::SST;
    uint64_t *afull = sempty + Cfg::SST, *aempty = afull + Cfg::AST;
    uint64_t *bfull = aempty + Cfg::AST, *bempty = bfull + 1;
    uint64_t *wfull = bempty + 1, *wempty = wfull + 2;
    uint64_t *accfull = wempty + 2, *accempty = accfull + 2, *mdone = accempty + 2;   // mdone [2]
    uint64_t *ekfull = mdone + 2, *ekempty = ekfull + Cfg::NEK;
    uint32_t *tmem_slot = (uint32_t *)(misc + 512);
    volatile int *abort_flag = (volatile int *)(misc + 516);
    float *wq = (float *)(misc + 1024);                   // [2][64] w[h] * 2^E_h
    int *ek = (int *)(misc + 1536);                       // [NEK][128] key-row exponents
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::SST; s++) {
            tc::mbar_init(&sfull[s], 1);
            tc::mbar_init(&sempty[s], 4);
        }
        for (int s = 0; s < Cfg::AST; s++) {
            tc::mbar_init(&afull[s], 4);
            tc::mbar_init(&aempty[s], 1);
        }
        tc::mbar_init(bfull, 4);
        tc::mbar_init(bempty, 2);                          // both MMA warps
        for (int i = 0; i < 2; i++) {
            tc::mbar_init(&wfull[i], 4);
            tc::mbar_init(&wempty[i], 4);
            tc::mbar_init(&accfull[i], 1);
            tc::mbar_init(&accempty[i], 4);
        }
        tc::mbar_init(&mdone[0], 1);
        tc::mbar_init(&mdone[1], 1);
        for (int i = 0; i < Cfg::NEK; i++) {
            tc::mbar_init(&ekfull[i], 4);
            tc::mbar_init(&ekempty[i], 4);
        }
        *abort_flag = 0;
        tc::fence_barrier_init();
        tc::prefetch_tmap(&tm_codes);
        tc::prefetch_tmap(&tm_sc);
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued = 0, last_par = 0;
            int b, jt0, jt1;
            bool ok = true;
            for (int r = 0; ok && fp4_item(a, cta, G, r, b, jt0, jt1); r++) {
                for (int jt = jt0; jt < jt1; jt++) {
                    if (!tc::mbar_wait(&sempty[s], ph ^ 1, a.status, abort_flag, a.spin)) { ok = false; break; }
                    const int64_t key0 = (int64_t)b * a.E + (int64_t)jt * 128;
                    tc::mbar_expect_tx(&sfull[s], Cfg::CODE_BYTES + Cfg::SC_BYTES);
                    uint8_t *dst = sS + s * Cfg::STG_BYTES;
                    // the keys are read once, the scores right after (kept in L2)
                    const uint64_t pol = tc::l2_evict_first();
                    tc::tma_load_2d_hint(dst, &tm_codes, 0, (int)key0, &sfull[s], pol);
                    tc::tma_load_2d_hint(dst + Cfg::CODE_BYTES, &tm_sc, 0, (int)(key0 >> 2), &sfull[s], pol);
                    issued |= 1u << s;
                    last_par = (last_par & ~(1u << s)) | (ph << s);
                    if (++s == Cfg::SST) { s = 0; ph ^= 1; }
                }
            }
            if (*abort_flag)
                for (int q = 0; q < Cfg::SST; q++)
                    if (issued & (1u << q))
                        for (long long i = 0; i < tc::DRAIN_LIMIT; i++)
                            if (tc::mbar_test(&sfull[q], (last_par >> q) & 1u)) break;
        }
    } else if (warp == 1 || warp == Cfg::MMA2) {
        // ------------------------------------------------------------ MMA
        // Two issuing warps take alternate tiles (warp 1 the even ones of the
        // CTA's tile sequence, warp MMA2 the odd ones), each always with the
        // same accumulator: one warp's barrier waits overlap the other's issue.
        const int p = warp == 1 ? 0 : 1;
        if (lane == 0) {
            // kind::f16 with f16 A and B (format fields 0), fp32 accumulation
            constexpr uint32_t idesc = (1u << 4) | ((uint32_t)(64 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
            uint32_t g = 0, bph = 0;
            const uint32_t aBase = tc::smem_u32(sA), bBase = tc::smem_u32(sB);
            int b, jt0, jt1;
            bool ok = true;
            for (int r = 0; ok && fp4_item(a, cta, G, r, b, jt0, jt1); r++) {
                if (jt0 >= jt1) continue;
                if (!tc::mbar_wait(bfull, bph, a.status, abort_flag, a.spin)) break;
                for (int jt = jt0; jt < jt1; jt++, g++) {
                    if ((int)(g & 1) != p) continue;
                    const int st = (int)(g % Cfg::AST);
                    if (!tc::mbar_wait(&afull[st], (g / Cfg::AST) & 1, a.status, abort_flag, a.spin) ||
                        !tc::mbar_wait(&accempty[p], ((g >> 1) & 1) ^ 1, a.status, abort_flag, a.spin)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t d = tmem + p * 64;
                    const uint32_t aS = aBase + st * Cfg::A_BYTES;
#pragma unroll
                    for (int kh = 0; kh < 2; kh++)
#pragma unroll
                        for (int kk = 0; kk < 4; kk++)
                            tc::mma_bf16(d, tc::desc_kmajor_sw128(aS + kh * 16384 + kk * 32),
                                         tc::desc_kmajor_sw128(bBase + kh * 8192 + kk * 32), idesc, (kh | kk) != 0);
                    tc::mma_commit(&aempty[st]);
                    tc::mma_commit(&accfull[p]);
                }
                if (!ok) break;
                // the query tile is free once both warps' products of this item are done
                tc::mma_commit(bempty);
                bph ^= 1;
            }
            // every MMA issued above has completed before TMEM is released
            tc::mma_commit(&mdone[p]);
            for (long long i = 0; i < tc::DRAIN_LIMIT; i++)
                if (tc::mbar_test(&mdone[p], 0)) break;
        }
    } else if (warp < Cfg::CONV0) {
        // -------------------------------------------------------- epilogue
        // each warp one TMEM lane quarter; the two accumulators alternate
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        uint32_t g = 0, ii = 0;
        int b, jt0, jt1;
        bool ok = true;
        for (int r = 0; ok && fp4_item(a, cta, G, r, b, jt0, jt1); r++) {
            if (jt0 >= jt1) continue;
            const int wb = ii & 1;
            if (!tc::mbar_wait(&wfull[wb], (ii >> 1) & 1, a.status, abort_flag, a.spin)) break;
            const float *wt = wq + wb * 64;
            const int64_t nv = visible_count(a.q_pos[b], a.m, a.E);
            for (int jt = jt0; jt < jt1; jt++, g++) {
                const int acc = (int)(g & 1);
                const uint32_t accph = (g >> 1) & 1;
                const int q = g % Cfg::NEK;
                if (!tc::mbar_wait(&accfull[acc], accph, a.status, abort_flag, a.spin) ||
                    !tc::mbar_wait(&ekfull[q], (g / Cfg::NEK) & 1, a.status, abort_flag, a.spin)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + acc * 64;
                // 32 columns (heads) at a time keeps the registers low
                float s0 = 0.f, s1 = 0.f;
                const float4 *wt4 = reinterpret_cast<const float4 *>(wt);
#pragma unroll
                for (int half = 0; half < 2; half++) {
                    float v[32];
                    tc::tmem_ld32(taddr + 32 * half, v);
                    tc::tmem_ld_wait();
                    tc::tmem_regs_ready<32>(v);
                    float sh = 0.f;
#pragma unroll
                    for (int h4 = 0; h4 < 8; h4++) {
                        const float4 wa = wt4[8 * half + h4];
                        sh = fmaf(wa.x, fmaxf(v[4 * h4], 0.f), sh);
                        sh = fmaf(wa.y, fmaxf(v[4 * h4 + 1], 0.f), sh);
                        sh = fmaf(wa.z, fmaxf(v[4 * h4 + 2], 0.f), sh);
                        sh = fmaf(wa.w, fmaxf(v[4 * h4 + 3], 0.f), sh);
                    }
                    if (half == 0) s0 = sh; else s1 = sh;
                }
                const int64_t j = (int64_t)jt * 128 + row;
                const float sc = (s0 + s1) * pow2f(ek[q * 128 + row]);
                if (j < nv)
                    tc::st_global_hint(a.scores + (int64_t)b * a.E + j, __bfloat162float(__float2bfloat16_rn(sc)),
                                       tc::l2_evict_last());
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&accempty[acc]);
                    tc::mbar_arrive(&ekempty[q]);
                }
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&wempty[wb]);
            ii++;
        }
    } else {
        // ------------------------------------------------------ converters
        // two groups of four warps take alternate tiles; group 0 also converts
        // each item's query (its 64 threads of one head each)
        const int cgrp = (warp - Cfg::CONV0) >> 2;
        const int ct = (threadIdx.x - Cfg::CONV0 * 32) & 127;   // the tile row this thread converts
        const uint32_t aBase = tc::smem_u32(sA), bBase = tc::smem_u32(sB);
        uint32_t bph = 0;
        uint32_t g = 0, ii = 0;
        int b, jt0, jt1;
        bool ok = true;
        for (int r = 0; ok && fp4_item(a, cta, G, r, b, jt0, jt1); r++) {
            if (jt0 >= jt1) continue;
            const int wb = ii & 1;
            if (cgrp == 0) {
                if (!tc::mbar_wait(bempty, bph ^ 1, a.status, abort_flag, a.spin) ||
                    !tc::mbar_wait(&wempty[wb], ((ii >> 1) & 1) ^ 1, a.status, abort_flag, a.spin)) {
                    ok = false;
                    break;
                }
                if (ct < 64) {
                    // head h = ct: block exponents from a first pass over its 128 values,
                    // then each block quantised and expanded (second pass, from cache)
                    const int h = ct;
                    const __nv_bfloat16 *src = a.qI + ((int64_t)b * 64 + h) * 128;
                    int eb[4], E = -127;
#pragma unroll
                    for (int blk = 0; blk < 4; blk++) {
                        float am = 0.f;
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            float v[8];
                            Vec<__nv_bfloat16>::load(src + 32 * blk + 8 * q, v);
#pragma unroll
                            for (int t = 0; t < 8; t++) am = fmaxf(am, fabsf(v[t]));
                        }
                        eb[blk] = mx_exponent(am);
                        E = max(E, eb[blk]);
                    }
#pragma unroll 1
                    for (int blk = 0; blk < 4; blk++) {
                        const float inv = pow2f(-eb[blk]);
                        const uint32_t s1 = f16_pow2(eb[blk] - E);
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            float v[8];
                            Vec<__nv_bfloat16>::load(src + 32 * blk + 8 * q, v);
                            uint32_t wv = 0;
#pragma unroll
                            for (int t = 0; t < 8; t++) wv |= e2m1_encode(v[t] * inv) << (4 * t);
                            uint32_t o[4];
                            e2m1x8_to_f16(wv, s1 | (s1 << 16), o);
                            st_shared_v4(bBase + (blk >> 1) * 8192 + swz_off(h, (blk & 1) * 4 + q), o);
                        }
                    }
                    wq[wb * 64 + h] = a.w[(int64_t)b * 64 + h] * pow2f(E);
                }
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(bfull);
                    tc::mbar_arrive(&wfull[wb]);
                }
                bph ^= 1;
            }
            ii++;
            // the key tiles of this group: 128 rows, one per thread
            const int64_t first = (int64_t)b * a.E;
            for (int jt = jt0; jt < jt1; jt++, g++) {
                if ((int)(g & 1) != cgrp) continue;
                const int s = g % Cfg::SST, st = g % Cfg::AST, qe = g % Cfg::NEK;
                if (!tc::mbar_wait(&sfull[s], (g / Cfg::SST) & 1, a.status, abort_flag, a.spin) ||
                    !tc::mbar_wait(&aempty[st], ((g / Cfg::AST) & 1) ^ 1, a.status, abort_flag, a.spin) ||
                    !tc::mbar_wait(&ekempty[qe], ((g / Cfg::NEK) & 1) ^ 1, a.status, abort_flag, a.spin)) {
                    ok = false;
                    break;
                }
                const uint8_t *stg = sS + s * Cfg::STG_BYTES;
                const int64_t key0 = first + (int64_t)jt * 128;
                const int sc0 = (int)(key0 & 3);          // key0's place in its 16-byte scale row
                const uint32_t aS = aBase + st * Cfg::A_BYTES;
                {
                    // key row rw = ct: its 64 code bytes and 4 scale bytes, all four
                    // blocks converted in this thread (independent of one another);
                    // stores of consecutive rows land in distinct banks (swizzle)
                    const int rw = ct;
                    const uint32_t sc4 = *reinterpret_cast<const uint32_t *>(stg + Cfg::CODE_BYTES + (sc0 + rw) * 4);
                    int E = -127;
#pragma unroll
                    for (int blk = 0; blk < 4; blk++) E = max(E, (int)((sc4 >> (8 * blk)) & 0xFFu) - 127);
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        // block (k + rw) & 3: the lanes' loads spread over the banks
                        const int blk = (k + rw) & 3;
                        const uint4 cw = *reinterpret_cast<const uint4 *>(stg + rw * 64 + blk * 16);
                        const int e = (int)((sc4 >> (8 * blk)) & 0xFFu) - 127;
                        const uint32_t s1 = f16_pow2(e - E);
                        const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            uint32_t o[4];
                            e2m1x8_to_f16(cws[q], s1 | (s1 << 16), o);
                            st_shared_v4(aS + (blk >> 1) * 16384 + swz_off(rw, (blk & 1) * 4 + q), o);
                        }
                    }
                    ek[qe * 128 + rw] = E;
                }
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&afull[st]);
                    tc::mbar_arrive(&sempty[s]);
                    tc::mbar_arrive(&ekfull[qe]);
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// 2D byte tensor map [rows, cols] with box [box_rows, cols], no swizzle;
// rows outside the array read as zero.
static bool make_tmap_u8_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {(cuuint32_t)cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_indexer_fp4(int64_t B, int64_t E, int m, const void *qI, const float *w, const void *kI4,
                               const int64_t *q_pos, float *scores, unsigned *status, long long spin,
                               int max_ctas, cudaStream_t st) {
    if (B == 0 || E == 0) return cudaSuccess;
    Fp4IdxArgs a;
    a.qI = (const __nv_bfloat16 *)qI; a.w = w; a.q_pos = q_pos; a.scores = scores; a.status = status;
    a.E = E; a.B = (int)B; a.m = m; a.tps = (int)((E + 127) / 128); a.spin = spin;
    const int64_t rows = B * E;
    const uint8_t *codes = (const uint8_t *)kI4;
    CUtensorMap tc_, ts_;
    if (!make_tmap_u8_2d(&tc_, codes, (uint64_t)rows, 64, 128) ||
        !make_tmap_u8_2d(&ts_, codes + (size_t)rows * 64, (uint64_t)((rows + 3) / 4), 16, Fp4Cfg::SC_ROWS))
        return cudaErrorInvalidValue;
    static PerDevice attr;
    cudaError_t e = smem_limit_once(attr, (const void *)indexer_fp4_kernel, Fp4Cfg::SMEM);
    if (e != cudaSuccess) return e;
    const int sms = max_ctas > 0 && max_ctas < device_sms() ? max_ctas : device_sms();
    const long long tiles = (long long)B * a.tps;
    const int grid = (int)(tiles < sms ? tiles : sms);
    indexer_fp4_kernel<<<grid, Fp4Cfg::THREADS, Fp4Cfg::SMEM, st>>>(tc_, ts_, a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace csa
