// Internal declarations shared by the librsa translation units: launch
// parameter blocks, the launchers each kernel file exports, and status helpers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/rsa.h"

namespace rsa {

// Device error word values (OR-ed with a site code in the low byte).
constexpr unsigned int kDevErrTimeout = 0x100u;
constexpr unsigned int kDevErrBounds = 0x200u;  // a bounds check of an RSA_DEBUG build failed

// The device-side error record.  Kernels get a pointer to `word` and OR codes
// into it; builds with RSA_DEBUG also keep the first out-of-range index (plus
// one, so that 0 means none) of a failed bounds check.
struct DeviceError {
    unsigned int word;
    unsigned int pad;
    unsigned long long bad_index_plus1;
};

#ifdef RSA_DEBUG
// Bounds check of an RSA_DEBUG build: false (and recorded, without a trap) if
// `ok` is false; the caller then skips the access.
__device__ __forceinline__ bool debug_check(bool ok, unsigned int *err, unsigned int site, long long idx)
{
    if (!ok && err) {
        atomicOr(err, kDevErrBounds | site);
        atomicCAS(&reinterpret_cast<DeviceError *>(err)->bad_index_plus1, 0ull, (unsigned long long)idx + 1ull);
    }
    return ok;
}
#define RSA_DCHECK(cond, err, site, idx) ::rsa::debug_check((cond), (err), (site), (long long)(idx))
#else
#define RSA_DCHECK(cond, err, site, idx) true
#endif

// Most pairs one kernel launch takes; longer pair lists are split.
constexpr int kMaxPairsPerLaunch = 32;

// What a block-attention epilogue does with a pair's (o, lse).
enum EpilogueMode : int {
    kStore = 0,       // write (o, lse) to out/lse
    kMergeAcc = 1,    // fold into the fp32 accumulator in place: acc/lse <- merge(acc/lse, o/lse)
    kMergeFinal = 2,  // fold with the accumulator and write the result to out/lse (acc read only)
};

// One (query chunk, KV chunk) pair inside a block-attention launch.  Output
// row r of head bh goes to out[(bh * out_T + out_t0 + r) * d] and
// lse[bh * out_T + out_t0 + r]; a merging epilogue reads the accumulator row
// at the same index of `acc` (and the running lse from `lse`).
struct PairDesc {
    int64_t q_off;   // global position of the first query row
    int64_t q_row0;  // row of the first query inside each head of the Q tensor
    int64_t kv_off;  // global position of the first key (causal mask)
    int64_t kv_row0; // row of the first key inside each head of the K/V tensors
    void *out;       // bf16 or fp32 (out_f32)
    float *lse;
    int64_t out_T;   // row pitch of out/lse per head
    int64_t out_t0;  // first row of this pair inside each head
    int out_f32;     // 1: fp32 output, 0: bf16 output
    int mode;        // EpilogueMode
    const float *acc;  // fp32 accumulator (kMergeAcc: same as out; kMergeFinal: read only)
    int64_t split_stride;  // out/lse rows between consecutive key splits of this pair
    int64_t out_rows;      // rows out, lse (and acc) hold from their base pointers (bounds checks)
};

struct BlockParams {
    int B, H;
    int64_t T;              // rows per head of K and V
    int64_t q_T;            // rows per head of the Q tensor (T, or the decode rows)
    int d;
    int causal;
    int64_t q_len, kv_len;  // rows per pair, keys per pair
    int64_t kv_split;       // keys per split of a pair's key range (0: one split)
    int n_split;            // splits per pair; split s covers keys [s*kv_split, (s+1)*kv_split)
    int npairs;
    int n_qgroups;          // query-row groups per pair (rows per CTA granularity)
    uint64_t wait_limit_ns;
    int tc_kernel;          // tensor-core kernel choice: 0 automatic (one-SM), 1 one-SM, 2 two-SM where it applies
    int acc_staged;         // set by the one-SM launcher: merging epilogues read the accumulator staged by TMA
    unsigned int *err;      // device error word
    PairDesc pairs[kMaxPairsPerLaunch];
};

// One pair's rows inside a merge launch.  Row rr (0 <= rr < rows_per_pair)
// of the pair is head bh = rr / Tc, position t = rr % Tc; its accumulator row
// is bh * T + acc_t0 + t and its partial row is rr.
struct MergePair {
    int64_t acc_t0;
    const void *o_blk;
    const float *lse_blk;
    int final_;  // 1: write out/lse_out, 0: update o_acc/lse_acc in place
    int pad_;
};

struct MergeParams {
    int64_t rows_per_pair, Tc, T;
    int npairs, d;
    int blk_f32, out_f32;
    float *o_acc;
    float *lse_acc;
    void *out;
    float *lse_out;
    unsigned int *err;  // device error word (bounds checks of RSA_DEBUG builds)
    MergePair pairs[kMaxPairsPerLaunch];
};

// Launchers (no validation; the C ABI layer validates).  They return the
// cudaError_t of the launch.
cudaError_t launch_block_attn_bf16(const void *q, const void *k, const void *v,
                                   const BlockParams &p, cudaStream_t s);
cudaError_t launch_block_attn_f32(const float *q, const float *k, const float *v,
                                  const BlockParams &p, cudaStream_t s);
cudaError_t launch_merge(const MergeParams &p, cudaStream_t s);
// Fold S partials [S][rows][d] (fp32 o, fp32 lse) into out [rows][d] and lse [rows].
cudaError_t launch_merge_splits(const float *o_part, const float *lse_part, int S, int64_t rows, int d,
                                void *out, int out_f32, float *lse, cudaStream_t s);
cudaError_t launch_selftest_wait(uint64_t limit_ns, unsigned int *err, cudaStream_t s);
// Two-pass ring self-attention (bf16, d = 128, T/N a multiple of 128): per
// query chunk, score pass into S [BH, Tc, T] fp32 (and per-tile row
// statistics [BH, Tc, T/128] float2), row softmax into P [BH, Tc, T] bf16
// (and lse), output pass into out.
cudaError_t launch_two_pass(const void *q, const void *k, const void *v, int64_t BH, int64_t T, int N, int causal,
                            void *out, float *lse, float *S, void *P, void *stats, uint64_t wait_limit_ns,
                            unsigned int *err, cudaStream_t s);

// bf16 TMA tensor map with 128-byte swizzle: dims and box innermost first,
// strides in bytes for dimensions 1..rank-1.  False if the driver rejects it.
bool make_bf16_map_sw128(CUtensorMap *m, const void *ptr, int rank, const uint64_t *dims,
                         const uint64_t *strides_bytes, const uint32_t *box);
// The same for fp32 elements.
bool make_f32_map_sw128(CUtensorMap *m, const void *ptr, int rank, const uint64_t *dims,
                        const uint64_t *strides_bytes, const uint32_t *box);

// Rows of one CTA of the tensor-core kernel (two 128-row tiles).
constexpr int kBf16RowsPerCta = 256;
// Rows of one CTA pair of the two-SM tensor-core kernel.
constexpr int kBf16RowsPerCluster = 512;

// The two-SM kernel serves d = 128 launches without key splits whose pairs
// have at least one full cluster of rows; launch_block_attn_bf16 picks it for
// those when BlockParams::tc_kernel asks for it (2), else the one-SM kernel.
bool block_attn_2sm_applies(const BlockParams &p);
cudaError_t launch_block_attn_bf16_2sm(const void *q, const void *k, const void *v, const BlockParams &p,
                                       cudaStream_t s);

// Device address of the __device__ variable at host-side stand-in `symbol`
// in the calling thread's current CUDA context, looked up with
// cudaGetSymbolAddress once per context.  The cache is keyed by the driver's
// unique context id, so a context created later (after cudaDeviceReset, for
// instance) gets a fresh lookup instead of a stale address.
rsa_status symbol_address(const void *symbol, void **out);

// Set the thread's last-error text and return `st`.
rsa_status fail(rsa_status st, const char *fmt, ...);

}  // namespace rsa
