// Block attention on the sm_103a tensor cores, two SMs per work unit: the same
// result as the one-SM kernel (o_blk = softmax(Q_i K_j^T / sqrt(d)) V_j and
// the row log-sum-exp for every (query chunk, KV chunk) pair of a launch),
// computed by clusters of two CTAs that share each K/V tile.
//
// Pages: "Sequence parallelism -- splitting the token dimension across GPUs"
// (llmdaily, day 58): the attention equation of "Attention wants keys and
// values from other tokens", the running (m, l, o) statistics and the
// e^{m - m_new} rescale of "But softmax seems to require all attention scores
// at once" (applied between 128-key tiles inside one pair), and the
// lower-triangular mask of "Causal attention gives us another optimization".
//
// Why two SMs.  With one SM per unit, the S = Q K^T MMA reads both operands
// from shared memory (8 KB per M128 N128 K16 step, one step per 64 cycles),
// which is all the shared-memory bandwidth an SM has; the K/V fills and the
// V reads of the PV MMA then slow the tensor core down.  A cta_group::2 MMA
// over a CTA pair has M = 256: each CTA supplies its own 128 query rows and
// half of B (64 keys of K, or 64 of the d columns of V), so each SM reads and
// fills half as much K/V per FLOP.
//
// Layout (d = 128 only).  A cluster covers 512 query rows of one (pair,
// head): CTA r holds rows [256 r, 256 r + 256) of the cluster as two 128-row
// tiles t = 0, 1; MMA tile t spans tile t of both CTAs.
//   warp 8 (both CTAs)  TMA producer: its own Q tiles, then per 128-key step
//                       its half of K (64 keys, all of d) and its half of V
//                       (128 keys, 64 of the d columns); every copy signals
//                       the even CTA's full-barrier, which the even CTA arms
//                       with the bytes of both halves.
//   warp 9              TMEM allocation in both CTAs (cta_group::2); in the
//                       even CTA one thread issues every MMA and commits to
//                       both CTAs' barriers (multicast).
//   warps 0-7 (both)    softmax of the CTA's own 128-row tiles, as in the
//                       one-SM kernel (two threads per row, one per 64-key
//                       half); each warp reports its finished part of P_t to
//                       the even CTA's P-full barrier.
// TMEM (each CTA): S0 | S1 | O0 | O1, 128 columns each.
#include <cuda_bf16.h>

#include <cmath>

#include "ptx_sm103.cuh"
#include "rsa_internal.h"
#include "tc_common.cuh"
#include "tc_softmax.cuh"

namespace rsa {
namespace {

using namespace tc;

constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr int D = 128;

struct Cfg {
    static constexpr uint32_t kQBox = 128u * 128u;     // 128 rows x 128 bytes
    static constexpr uint32_t kQTile = 2 * kQBox;      // 128 rows x 128 columns
    static constexpr uint32_t kKBox = 64u * 128u;      // 64 keys x 128 bytes
    static constexpr uint32_t kStageBytes = 16384;     // K half (64 keys x 128) or V half (128 keys x 64)
    static constexpr int kStages = 8;
    static constexpr uint32_t kQOff = 0;
    static constexpr uint32_t kKVOff = 2 * kQTile;
    static constexpr uint32_t kBarOff = kKVOff + kStages * kStageBytes;
    static constexpr uint32_t kXchOff = kBarOff + 256;  // [2 tiles][2 halves][128 rows] floats
    static constexpr uint32_t kSmemBytes = kXchOff + 2048 + 1024;
    static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384;
    // barrier indices
    static constexpr int kQF = 0;
    static constexpr int kKVF = 1;
    static constexpr int kKVE = kKVF + kStages;
    static constexpr int kSF = kKVE + kStages;
    static constexpr int kPF = kSF + 2;
    static constexpr int kOF = kPF + 2;
    static constexpr int kDrain = kOF + 2;
    static constexpr int kNumBars = kDrain + 1;
    static_assert(kNumBars * 8 + 8 <= 256, "barrier area");
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    block_attn_bf16_2sm_kernel(const __grid_constant__ CUtensorMap tm_q,
                               const __grid_constant__ CUtensorMap tm_k,
                               const __grid_constant__ CUtensorMap tm_v,
                               const __grid_constant__ BlockParams p)
{
    using C = Cfg;
    extern __shared__ uint8_t smem_raw[];
    // Both CTAs run the same kernel, so this offset (and every one below) is
    // the same in both: the pair MMA addresses the peer's operands by it.
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sQ = base + C::kQOff;
    const uint32_t sKV = base + C::kKVOff;
    const uint32_t bars = base + C::kBarOff;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + C::kBarOff + 8 * C::kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::kBarOff + 8 * C::kNumBars + 4);
    auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = rank == 0;
    const uint32_t bars0 = ptx::mapa_shared(bars, 0);  // the even CTA's barriers
    auto BAR0 = [&](int i) -> uint32_t { return bars0 + 8u * (uint32_t)i; };

    // ---- which pair, head and 512-row group (one per cluster) -------------------
    // The clusters of one (pair, head) are consecutive, heaviest causal groups first.
    const int64_t L = blockIdx.x >> 1;
    const int64_t unit = L / p.n_qgroups;
    const int qg = p.n_qgroups - 1 - (int)(L - unit * p.n_qgroups);
    const int pi = (int)(unit % p.npairs);
    const int bh = (int)(unit / p.npairs);
    const PairDesc &pr = p.pairs[pi];
    const int64_t kv_off = pr.kv_off;    // global position (mask)
    const int64_t kv_row = pr.kv_row0;   // row in the K/V tensors
    const int64_t kv_len = p.kv_len;
    const int64_t qc0 = (int64_t)qg * 512;               // first row of the cluster
    const int64_t rows_valid = min((int64_t)512, p.q_len - qc0);
    int64_t kv_end = kv_len;
    if (p.causal)
        kv_end = min(kv_end, pr.q_off + qc0 + rows_valid - kv_off);
    const int n = kv_end > 0 ? (int)((kv_end + 127) / 128) : 0;  // same in both CTAs
    const int64_t q0 = qc0 + 256 * (int64_t)rank;        // first row of this CTA

    if (threadIdx.x == 0) {
        ptx::mbar_init(BAR(C::kQF), 1);
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(BAR(C::kKVF + s), 1);
            ptx::mbar_init(BAR(C::kKVE + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(BAR(C::kSF + t), 1);
            ptx::mbar_init(BAR(C::kPF + t), 16);  // one arrival per softmax warp of both CTAs
            ptx::mbar_init(BAR(C::kOF + t), 1);
        }
        ptx::mbar_init(BAR(C::kDrain), 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 9) {
        ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    if (warp == 8 && lane == 0) {
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_k);
        ptx::tma_prefetch_desc(&tm_v);
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();  // both CTAs' barriers and TMEM are ready before any cross-CTA use
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t lim_ns = p.wait_limit_ns;

    if (warp == 8) {
        // =========================== TMA producer ===========================
        if (lane == 0 && n > 0) {
            int last_use[C::kStages];
            for (int s = 0; s < C::kStages; ++s)
                last_use[s] = -1;
            if (leader)
                ptx::mbar_arrive_expect_tx(BAR(C::kQF), 2 * 2 * C::kQTile);
            for (int t = 0; t < 2; ++t)
                for (int b = 0; b < 2; ++b)
                    ptx::tma_load_3d_pair(sQ + t * C::kQTile + b * C::kQBox, &tm_q, BAR0(C::kQF), b * 64,
                                          (int)(pr.q_row0 + q0 + t * 128), bh);
            for (int ld = 0; ld < 2 * n; ++ld) {
                const int slot = ld % C::kStages;
                const int use = ld / C::kStages;
                if (use > 0 &&
                    !ptx::mbar_wait(BAR(C::kKVE + slot), (use - 1) & 1, lim_ns, abort_flag, p.err, 1))
                    break;
                const int row = (int)(kv_row + (int64_t)(ld >> 1) * 128);
                const uint32_t dst = sKV + slot * C::kStageBytes;
                if (leader)
                    ptx::mbar_arrive_expect_tx(BAR(C::kKVF + slot), 2 * C::kStageBytes);
                if ((ld & 1) == 0) {
                    // K: keys [row + 64 rank, +64), both 64-column boxes
                    for (int b = 0; b < 2; ++b)
                        ptx::tma_load_3d_pair(dst + b * C::kKBox, &tm_k, BAR0(C::kKVF + slot), b * 64,
                                              row + 64 * (int)rank, bh);
                } else {
                    // V: keys [row, row + 128), columns [64 rank, 64 rank + 64)
                    ptx::tma_load_3d_pair(dst, &tm_v, BAR0(C::kKVF + slot), 64 * (int)rank, row, bh);
                }
                last_use[slot] = use;
            }
            // The even CTA's full-barriers count the bytes of both CTAs: once
            // they complete, every copy either CTA started has landed.
            if (leader) {
                volatile int no_abort = 0;
                ptx::mbar_wait(BAR(C::kQF), 0, lim_ns, &no_abort, p.err, 2);
                for (int s = 0; s < C::kStages; ++s)
                    if (last_use[s] >= 0)
                        ptx::mbar_wait(BAR(C::kKVF + s), last_use[s] & 1, lim_ns, &no_abort, p.err, 3);
            }
        }
    } else if (warp == 9) {
        // ============================ MMA issuer ============================
        if (leader && lane == 0) {
            if (n > 0) {
                const uint32_t idesc_qk = ptx::idesc_bf16_f32(256, 128, false);
                const uint32_t idesc_pv = ptx::idesc_bf16_f32(256, D, true);
                // First K step of each operand; later steps only move the start
                // address field, which never carries out inside a tile.
                const uint64_t dq0 = ptx::smem_desc_sw128(sQ, 16, 1024);
                const uint64_t dk0 = ptx::smem_desc_sw128(sKV, 16, 1024);
                const uint64_t dv0 = ptx::smem_desc_sw128(sKV, C::kStageBytes, 1024);
                const uint16_t both = 0x3;
                auto issue_qk = [&](int t, int slot) {
                    const uint64_t qa = dq0 + ((t * C::kQTile) >> 4);
                    const uint64_t kb = dk0 + ((slot * C::kStageBytes) >> 4);
                    const uint32_t dst = tmem + (t ? C::kColS1 : C::kColS0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t aoff = ((kk >> 2) * C::kQBox + (kk & 3) * 32) >> 4;
                        const uint32_t boff = ((kk >> 2) * C::kKBox + (kk & 3) * 32) >> 4;
                        ptx::mma_ss_pair(dst, qa + aoff, kb + boff, idesc_qk, kk > 0);
                    }
                };
                auto issue_pv = [&](int t, int slot, bool acc) {
                    const uint64_t vb = dv0 + ((slot * C::kStageBytes) >> 4);
                    const uint32_t dst = tmem + (t ? C::kColO1 : C::kColO0);
                    const uint32_t pa = tmem + (t ? C::kColS1 : C::kColS0);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        ptx::mma_ts_pair(dst, pa + kk * 8, vb + ((kk * 2048) >> 4), idesc_pv,
                                         (acc || kk > 0) ? 1u : 0u);
                };
                // P_t(j) complete in both CTAs (every softmax warp arrived): O_t += P_t V_j.
                auto pv_tile = [&](int t, int slot, int j) -> bool {
                    if (!ptx::mbar_wait(BAR(C::kPF + t), j & 1, lim_ns, abort_flag, p.err, 13 + 2 * t))
                        return false;
                    ptx::tc_fence_after();
                    issue_pv(t, slot, j > 0);
                    return true;
                };
                bool ok = ptx::mbar_wait(BAR(C::kQF), 0, lim_ns, abort_flag, p.err, 10);
                int kslot = 0;
                if (ok)
                    ok = ptx::mbar_wait(BAR(C::kKVF + 0), 0, lim_ns, abort_flag, p.err, 11);
                if (ok) {
                    ptx::tc_fence_after();
                    issue_qk(0, 0);
                    ptx::mma_commit_pair(BAR(C::kSF + 0), both);
                    issue_qk(1, 0);
                    ptx::mma_commit_pair(BAR(C::kSF + 1), both);
                    ptx::mma_commit_pair(BAR(C::kKVE + 0), both);
                }
                for (int j = 0; ok && j < n; ++j) {
                    const int vld = 2 * j + 1;
                    const int vslot = vld % C::kStages;
                    ok = ptx::mbar_wait(BAR(C::kKVF + vslot), (vld / C::kStages) & 1, lim_ns, abort_flag,
                                        p.err, 12);
                    if (!ok)
                        break;
                    // tile 0
                    ok = pv_tile(0, vslot, j);
                    if (!ok)
                        break;
                    const bool more = j + 1 < n;
                    if (more) {
                        const int kld = 2 * (j + 1);
                        kslot = kld % C::kStages;
                        ok = ptx::mbar_wait(BAR(C::kKVF + kslot), (kld / C::kStages) & 1, lim_ns, abort_flag,
                                            p.err, 14);
                        if (!ok)
                            break;
                        issue_qk(0, kslot);
                        ptx::mma_commit_pair(BAR(C::kSF + 0), both);
                    } else {
                        ptx::mma_commit_pair(BAR(C::kOF + 0), both);
                    }
                    // tile 1
                    ok = pv_tile(1, vslot, j);
                    if (!ok)
                        break;
                    ptx::mma_commit_pair(BAR(C::kKVE + vslot), both);
                    if (more) {
                        issue_qk(1, kslot);
                        ptx::mma_commit_pair(BAR(C::kSF + 1), both);
                        ptx::mma_commit_pair(BAR(C::kKVE + kslot), both);
                    } else {
                        ptx::mma_commit_pair(BAR(C::kOF + 1), both);
                    }
                }
            }
            // Drain: both CTAs learn that every MMA has finished before TMEM is freed.
            ptx::mma_commit_pair(BAR(C::kDrain), 0x3);
        }
        if (lane == 0) {
            volatile int no_abort = 0;
            ptx::mbar_wait(BAR(C::kDrain), 0, lim_ns, &no_abort, p.err, 16);
        }
        __syncwarp();
    } else {
        // ============================== softmax ==============================
        // This CTA's own two 128-row tiles; each warp reports a finished
        // quarter of P to the even CTA's P-full barrier.
        SoftmaxCtx ctx;
        ctx.tmem = tmem;
        ctx.col_s[0] = C::kColS0;
        ctx.col_s[1] = C::kColS1;
        ctx.col_o[0] = C::kColO0;
        ctx.col_o[1] = C::kColO1;
        for (int t = 0; t < 2; ++t) {
            ctx.bar_sf[t] = BAR(C::kSF + t);
            ctx.bar_of[t] = BAR(C::kOF + t);
        }
        ctx.xch = reinterpret_cast<float *>(gbase + C::kXchOff);
        ctx.abort_flag = abort_flag;
        ctx.lim_ns = lim_ns;
        softmax_warps<D, 2>(ctx, p, pr, q0, n, n, kv_off, kv_len, bh, 0, [&](int t) {
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive_remote(BAR0(C::kPF + t));
        });
    }

    // ---- teardown --------------------------------------------------------------
    // Every MMA has finished (warp 9 waited on the drain in both CTAs); the
    // cluster barrier also keeps each CTA's shared memory alive until the
    // peer's last remote arrival and copy into it are done.
    ptx::tc_fence_before();
    ptx::cluster_sync();
    if (warp == 9) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem, kTmemCols);
    }
}

// [B*H, T, d] bf16 view with box_rows x 64-column boxes and 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *ptr, int64_t BH, int64_t T, int d, uint32_t box_rows)
{
    const uint64_t dims[3] = {(uint64_t)d, (uint64_t)T, (uint64_t)BH};
    const uint64_t strides[2] = {(uint64_t)d * 2, (uint64_t)T * d * 2};
    const uint32_t box[3] = {64, box_rows, 1};
    return make_bf16_map_sw128(m, ptr, 3, dims, strides, box);
}

}  // namespace

bool block_attn_2sm_applies(const BlockParams &p)
{
    return p.d == D && p.n_split == 1 && p.kv_split == 0 && p.q_len >= kBf16RowsPerCluster;
}

cudaError_t launch_block_attn_bf16_2sm(const void *q, const void *k, const void *v, const BlockParams &p0,
                                       cudaStream_t s)
{
    if (p0.d != D || p0.n_split != 1)
        return cudaErrorInvalidValue;
    BlockParams p = p0;
    p.n_qgroups = (int)((p.q_len + kBf16RowsPerCluster - 1) / kBf16RowsPerCluster);
    const int64_t BH = (int64_t)p.B * p.H;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, BH, p.q_T, D, 128) || !make_map(&mk, k, BH, p.T, D, 64) ||
        !make_map(&mv, v, BH, p.T, D, 128))
        return cudaErrorInvalidValue;
    const int64_t grid = 2 * (int64_t)p.n_qgroups * p.npairs * BH;
    if (grid <= 0)
        return cudaSuccess;
    if (grid > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const uint32_t smem = Cfg::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(block_attn_bf16_2sm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    block_attn_bf16_2sm_kernel<<<(unsigned)grid, kThreads, smem, s>>>(mq, mk, mv, p);
    return cudaGetLastError();
}

}  // namespace rsa
