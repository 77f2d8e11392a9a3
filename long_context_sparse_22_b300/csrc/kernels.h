// Internal launcher declarations of libcsa (not part of the C ABI).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/csa.h"
#include "common.cuh"

namespace csa {

// Every kernel launch of the library is counted (csa_launch_count).
void count_launches(int n);

// Record a failure message for csa_last_error() and return s.
csa_status report_error(csa_status s, const char *msg);

// Devices a process may address (device ordinals 0 .. MAX_DEVICES-1).
constexpr int MAX_DEVICES = 64;

// One-time set-up done separately on every device: bit d is set once the
// set-up has run with device d current.
struct PerDevice {
    std::atomic<unsigned long long> done{0};
};

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, the first time this kernel is launched there (the attribute is per
// device).
cudaError_t smem_limit_once(PerDevice &once, const void *kernel, int bytes);

// Polls of a bounded wait: params->spin_limit, or the default when it is 0.
constexpr long long DEFAULT_SPIN_LIMIT = 1LL << 24;
inline long long spin_limit_of(int64_t v) { return v > 0 ? (long long)v : DEFAULT_SPIN_LIMIT; }

struct AttnArgs {
    const void *q;
    const int64_t *q_pos;
    const void *kvc;
    const int32_t *idx;   // nullptr: every visible entry (HCA)
    const void *kv_raw;
    const int64_t *raw_pos0;
    const float *sink;
    void *out;
    float *lse;
    unsigned *status;
    int64_t Tq;
    int H, c;
    int64_t E;
    int k;
    int64_t L;
    int m, n_win, derotate;
    float scale;
    long long spin;        // polls before a bounded wait gives up
    int kv8;               // kvc holds FP8 records (c = 512, 64 rotary dims)
    const float *q_norm;   // RMSNorm gains of q (c floats) or nullptr
    float norm_eps;
    RopeFreqs rope;
};

// gain != nullptr: the KV RMSNorm of every stored raw row and entry, before
// its rotation (one CTA per block).
cudaError_t launch_compress(csa_dtype dt, int64_t B, int64_t n, int c, int m, int overlap,
                            const void *C, const void *Z, const float *bias, const void *Cb,
                            const void *Zb, const float *biasb, void *out, void *raw_out,
                            const RopeFreqs &rope, const float *gain, float eps, cudaStream_t st);

// Low-precision caches.  FP8 KV record of a c = 512 entry with 64 rotary
// dims: 448 E4M3 codes, 64 BF16 rotary values, 4 fp32 group scales.
constexpr int KV8_BYTES = 592;
constexpr int KV8_NR = 448;
// MXFP4 rows of 128 values: codes (64 bytes a row) then scale bytes (4 a row,
// the row count rounded up to a multiple of 4).
size_t mxfp4_bytes(int64_t rows);
cudaError_t launch_quant_kv_fp8(csa_dtype dt, int64_t rows, const void *src, void *dst, cudaStream_t st);
cudaError_t launch_quant_mxfp4(csa_dtype dt, int64_t rows, const void *src, void *dst, cudaStream_t st);
// -inf into every score past a row's visible prefix.
cudaError_t launch_mask_tail(float *scores, const int64_t *q_pos, int64_t rows, int64_t E, int m, cudaStream_t st);
// Decode scores (one query per sequence, 64 x 128 indexer) over MXFP4 keys,
// rounded to BF16 (kept as fp32 values).
cudaError_t launch_indexer_fp4(int64_t B, int64_t E, int m, const void *qI, const float *w, const void *kI4,
                               const int64_t *q_pos, float *scores, unsigned *status, long long spin,
                               int max_ctas, cudaStream_t st);

// Y[:, g*N + n] = A[:, g*K : (g+1)*K] . W[g*N + n, :] for g < groups (bf16, fp32
// accumulation): A [M, groups*K], W [groups*N, K], Y [M, groups*N] row-major.
// N a multiple of 256, K of 64.
cudaError_t launch_gemm_bf16(int64_t M, int N, int K, int groups, const void *A, const void *W, void *Y,
                             unsigned *status, long long spin, cudaStream_t st);

// Incremental decode: one arriving token per sequence into the window ring and
// the compression tail; a completed block is compressed into the caches.
struct DecodeAppend {
    const void *C, *Z, *Cb, *Zb, *Ck, *Zk, *Ckb, *Zkb;
    const float *bias, *biasb, *biask, *biaskb;
    const int64_t *t;
    void *win, *tail, *kvc, *kIc;
    unsigned *status;
    int64_t E_cap;
    int c, dI, m, overlap, n_win;
    const float *kv_norm;
    float norm_eps;
    RopeFreqs rope;
};
int decode_tail_slots(int m, int overlap);
int decode_tail_width(int c, int dI, int overlap);
cudaError_t launch_decode_append(csa_dtype dt, int64_t B, const DecodeAppend &d, cudaStream_t st);

cudaError_t launch_indexer_simt(csa_dtype dt, int64_t B, int64_t Tq, int hI, int dI, int64_t E,
                                int m, const void *qI, const float *w, const void *kI,
                                const int64_t *q_pos, float *scores, int write_masked,
                                cudaStream_t st);

bool indexer_tc_supported(int hI, int dI, int64_t B, int64_t T, int64_t E);

// max_ctas > 0 caps the persistent grid (to leave SMs to a concurrent kernel)
cudaError_t launch_indexer_tc(int64_t B, int64_t T, int64_t E, int m, const void *qI,
                              const float *w, const void *kI, const int64_t *q_pos, float *scores,
                              int write_masked, unsigned *status, int max_ctas, long long spin,
                              cudaStream_t st);

// scratch: topk_scratch_bytes(B*Tq, E) bytes of device memory (0 for the
// one-CTA-per-row path, used for rows of at most 16384 entries or many rows)
size_t topk_scratch_bytes(int64_t rows, int64_t E);
cudaError_t launch_topk(int64_t B, int64_t Tq, int64_t E, int k, int m, const float *scores,
                        const int64_t *q_pos, int32_t *idx, int32_t *cnt, void *scratch,
                        cudaStream_t st);
// The same in two phases: 1 = everything, or for few long rows only the
// candidate collection (every SM); 2 = the long rows' exact selection (one
// CTA per row), nothing otherwise.
cudaError_t launch_topk_phase(int phase, int64_t B, int64_t Tq, int64_t E, int k, int m,
                              const float *scores, const int64_t *q_pos, int32_t *idx, int32_t *cnt,
                              void *scratch, cudaStream_t st);

cudaError_t launch_attn_simt(csa_dtype dt, int64_t B, const AttnArgs &a, cudaStream_t st);

// Tensor-core attention (bf16, c = 128 or 512).  n_chunks > 1 splits each query's
// entry list over several CTAs (decode) and needs attn_tc_split_bytes of
// scratch; cnt (nullable) gives the number of valid leading slots of idx.
bool attn_tc_supported(csa_dtype dt, int c);
int attn_tc_chunks(int64_t rows, int H, int64_t max_list, bool invariant);
size_t attn_tc_split_bytes(int64_t rows, int H, int c, int n_chunks);
cudaError_t launch_attn_tc(int64_t B, const AttnArgs &a, const int32_t *cnt, int n_chunks,
                           void *split_ws, int max_ctas, cudaStream_t st);
// Dense attention with 128 (query, head) rows per item (c = 128, H dividing
// 128, no split): attn_pack.cu.
bool attn_pack_supported(int64_t B, const AttnArgs &g, int n_chunks);
cudaError_t launch_attn_pack(int64_t B, const AttnArgs &g, int max_ctas, cudaStream_t st);

// SM count of the current device (cached per device).
int device_sms();

// A kernel that waits on a barrier nothing completes, for at most `spin`
// polls, then records ST_TIMEOUT in *status.
cudaError_t launch_wait_probe(unsigned *status, long long spin, cudaStream_t st);

}  // namespace csa
