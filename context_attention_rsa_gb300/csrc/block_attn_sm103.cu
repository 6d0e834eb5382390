// Block attention on the sm_103a tensor cores: one launch computes, for every
// (query chunk, KV chunk) pair it is given, o_blk = softmax(Q_i K_j^T / sqrt(d)) V_j
// and the row log-sum-exp.
//
// Pages: "Sequence parallelism -- splitting the token dimension across GPUs"
// (llmdaily, day 58): the attention equation of "Attention wants keys and
// values from other tokens", the running (m, l, o) statistics and the
// e^{m - m_new} rescale of "But softmax seems to require all attention scores
// at once" (applied here between 128-key tiles inside one pair), and the
// lower-triangular mask of "Causal attention gives us another optimization".
//
// Design (one CTA = 256 query rows of one pair and one head, as two 128-row
// tiles that share every K/V tile):
//   warp 8      TMA producer: Q tiles once, then K(j), V(j) through a ring of
//               shared-memory slots (128-byte swizzle).
//   warp 9      TMEM allocator and the single MMA-issuing thread:
//                 S_t = Q_t K_j^T   (tcgen05.mma, A and B from shared memory)
//                 O_t += P_t V_j    (tcgen05.mma, A = P from TMEM, B = V from
//                                    shared memory, MN-major)
//   warps 0-7   softmax, on tile 0's S and then on tile 1's: two threads per
//               query row (TMEM lane = row), each with one 64-key half of the
//               row; they agree on the row max through shared memory, rescale
//               O when the max rose by more than 2^8, write P = 2^{x - m} as
//               bf16 back over S, and finally write o = O / l and
//               lse = (m + log2 l) ln 2.
// TMEM: S0 | S1 | O0 | O1 (128 + 128 + d + d columns of the 512).
// The kept maximum m only moves when the new one exceeds it by more than 8
// (log2 units); o, l and lse all use the same m, so the result is exact up to
// rounding whatever m is kept.
#include <cuda_bf16.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "ptx_sm103.cuh"
#include "rsa_internal.h"
#include "tc_common.cuh"
#include "tc_softmax.cuh"

namespace rsa {
namespace {

using namespace tc;

constexpr uint32_t kTmemCols = 512;

template <int D>
struct Cfg {
    // Threads per query row in the softmax (8 softmax warps), then one TMA
    // warp and one MMA warp.  Four threads per row (16 softmax warps) was
    // measured slower: more exchange and TMEM instructions per tile.
    static constexpr int kTPR = 2;
    static constexpr int kSoftmaxWarps = 4 * kTPR;
    static constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
    static constexpr int kProducerWarp = kSoftmaxWarps;
    static constexpr int kMmaWarp = kSoftmaxWarps + 1;
    static constexpr int kThreads = 32 * (kSoftmaxWarps + 2);
    static constexpr int kBoxes = D / 64;            // 128-byte-wide TMA boxes per tile
    static constexpr uint32_t kBoxBytes = 128u * 128u; // 128 rows x 128 bytes
    static constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;
    static constexpr int kStages = D == 128 ? 4 : 6;
    static constexpr uint32_t kQOff = 0;
    static constexpr uint32_t kKVOff = 2 * kTileBytes;
    static constexpr uint32_t kBarOff = kKVOff + kStages * kTileBytes;
    static constexpr uint32_t kXchOff = kBarOff + 256;  // [2 tiles][kTPR parts][128 rows] floats
    static constexpr uint32_t kSmemBytes = kXchOff + 2 * kTPR * 128 * 4 + 1024;
    static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
    // barrier indices
    static constexpr int kQF = 0;
    static constexpr int kKVF = 1;
    static constexpr int kKVE = kKVF + kStages;
    static constexpr int kSF = kKVE + kStages;
    static constexpr int kPF = kSF + 2;
    static constexpr int kOF = kPF + 2;
    static constexpr int kDrain = kOF + 2;
    static constexpr int kQFree = kDrain + 1;   // every MMA but the last step's PVs has completed
    static constexpr int kAccFull = kQFree + 1; // the staged accumulator rows have landed
    static constexpr int kNumBars = kAccFull + 1;
    // Merging epilogues stage the CTA's fp32 accumulator rows in shared memory:
    // tile 0 over Q, tile 1 over two K/V slots, in 32-column boxes of 128 rows
    // (128-byte swizzle).
    static constexpr int kAccBoxes = D / 32;
    static constexpr uint32_t kAccBoxBytes = 128u * 32u * 4u;
    static_assert(kAccBoxes * kAccBoxBytes == 2 * kTileBytes, "an accumulator tile fills two K/V slots");
    static_assert(kStages % 2 == 0, "two consecutive slots never wrap");
    static_assert(kNumBars * 8 + 8 <= 256, "barrier area");
};

template <int D>
__global__ void __launch_bounds__(Cfg<D>::kThreads, 1)
    block_attn_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_acc,
                           const __grid_constant__ BlockParams p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
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

    // ---- which pair, head and 256-row group ------------------------------------
    // All row groups of one (pair, head) are consecutive blocks, so the CTAs
    // running at the same time stream the same K/V chunk and share it in L2.
    // Inside a (pair, head) the heaviest causal groups come first.
    // A pair's key range may be cut into n_split splits (decode): each split
    // is its own work unit and writes its own partial rows.
    const int64_t L = blockIdx.x;
    const int64_t unit = L / p.n_qgroups;
    const int qg = p.n_qgroups - 1 - (int)(L - unit * p.n_qgroups);
    const int sp = (int)(unit % p.n_split);
    const int64_t unit2 = unit / p.n_split;
    const int pi = (int)(unit2 % p.npairs);
    const int bh = (int)(unit2 / p.npairs);
    const PairDesc &pr = p.pairs[pi];
    const int64_t kv_off = pr.kv_off + (int64_t)sp * p.kv_split;   // global position (mask)
    const int64_t kv_row = pr.kv_row0 + (int64_t)sp * p.kv_split;  // row in the K/V tensors
    const int64_t kv_len = p.kv_split > 0 ? min(p.kv_split, p.kv_len - (int64_t)sp * p.kv_split) : p.kv_len;
    const int64_t q0 = (int64_t)qg * kBf16RowsPerCta;
    const int64_t rows_valid = min((int64_t)kBf16RowsPerCta, p.q_len - q0);
    int64_t kv_end = kv_len;
    if (p.causal)
        kv_end = min(kv_end, pr.q_off + q0 + rows_valid - kv_off);
    const int n = kv_end > 0 ? (int)((kv_end + 127) / 128) : 0;
    // Tile 0 (the CTA's first 128 rows) may need one key tile fewer: under the
    // causal mask a key tile that starts after its last row is all masked
    // (the last step of every CTA on a diagonal pair), so tile 0 skips it.
    int n0 = n;
    if (p.causal && n > 0) {
        const int64_t e0 = min(kv_len, pr.q_off + q0 + min((int64_t)128, rows_valid) - kv_off);
        n0 = e0 > 0 ? (int)((e0 + 127) / 128) : 0;
    }
    // The fold into the accumulator reads its rows from shared memory, staged
    // by TMA while the last step runs.
    const bool stage_acc = p.acc_staged && pr.mode != kStore && n > 0;
    const uint32_t acc_stage[2] = {sQ, sKV + (uint32_t)((2 * n) % C::kStages) * C::kTileBytes};

    if (threadIdx.x == 0) {
        ptx::mbar_init(BAR(C::kQF), 1);
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(BAR(C::kKVF + s), 1);
            ptx::mbar_init(BAR(C::kKVE + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(BAR(C::kSF + t), 1);
            ptx::mbar_init(BAR(C::kPF + t), C::kSoftmaxThreads);
            ptx::mbar_init(BAR(C::kOF + t), 1);
        }
        ptx::mbar_init(BAR(C::kDrain), 1);
        ptx::mbar_init(BAR(C::kQFree), 1);
        ptx::mbar_init(BAR(C::kAccFull), 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == C::kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp == C::kProducerWarp && lane == 0) {
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_k);
        ptx::tma_prefetch_desc(&tm_v);
        if (p.acc_staged)
            ptx::tma_prefetch_desc(&tm_acc);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t lim_ns = p.wait_limit_ns;

    if (warp == C::kProducerWarp) {
        // =========================== TMA producer ===========================
        if (lane == 0 && n > 0) {
            int last_use[C::kStages];
            for (int s = 0; s < C::kStages; ++s)
                last_use[s] = -1;
            ptx::mbar_arrive_expect_tx(BAR(C::kQF), 2 * C::kTileBytes);
            for (int t = 0; t < 2; ++t)
                for (int b = 0; b < C::kBoxes; ++b)
                    ptx::tma_load_3d(sQ + t * C::kTileBytes + b * C::kBoxBytes, &tm_q, BAR(C::kQF),
                                     b * 64, (int)(pr.q_row0 + q0 + t * 128), bh);
            // The accumulator rows a merging epilogue will stage: into L2 now,
            // so that their load at the end of the main loop is an L2 hit.
            if (stage_acc)
                for (int t = 0; t < 2; ++t)
                    for (int b = 0; b < C::kAccBoxes; ++b)
                        ptx::tma_prefetch_l2_3d(&tm_acc, b * 32, (int)(pr.out_t0 + q0 + t * 128), bh);
            for (int ld = 0; ld < 2 * n; ++ld) {
                const int slot = ld % C::kStages;
                const int use = ld / C::kStages;
                if (use > 0 &&
                    !ptx::mbar_wait(BAR(C::kKVE + slot), (use - 1) & 1, lim_ns, abort_flag, p.err, 1))
                    break;
                const CUtensorMap *m = (ld & 1) ? &tm_v : &tm_k;
                const int row = (int)(kv_row + (int64_t)(ld >> 1) * 128);
                ptx::mbar_arrive_expect_tx(BAR(C::kKVF + slot), C::kTileBytes);
                for (int b = 0; b < C::kBoxes; ++b)
                    ptx::tma_load_3d(sKV + slot * C::kTileBytes + b * C::kBoxBytes, m,
                                     BAR(C::kKVF + slot), b * 64, row, bh);
                last_use[slot] = use;
            }
            // Accumulator rows of a merging epilogue: once every MMA but the
            // last PVs has completed, Q and every slot but V(n-1)'s are free.
            bool acc_issued = false;
            if (stage_acc && ptx::mbar_wait(BAR(C::kQFree), 0, lim_ns, abort_flag, p.err, 4)) {
                ptx::mbar_arrive_expect_tx(BAR(C::kAccFull), 2 * C::kAccBoxes * C::kAccBoxBytes);
                for (int t = 0; t < 2; ++t)
                    for (int b = 0; b < C::kAccBoxes; ++b)
                        ptx::tma_load_3d(acc_stage[t] + b * C::kAccBoxBytes, &tm_acc, BAR(C::kAccFull), b * 32,
                                         (int)(pr.out_t0 + q0 + t * 128), bh);
                acc_issued = true;
            }
            // Let every copy this thread started land before the CTA can exit.
            volatile int no_abort = 0;
            ptx::mbar_wait(BAR(C::kQF), 0, lim_ns, &no_abort, p.err, 2);
            for (int s = 0; s < C::kStages; ++s)
                if (last_use[s] >= 0)
                    ptx::mbar_wait(BAR(C::kKVF + s), last_use[s] & 1, lim_ns, &no_abort, p.err, 3);
            if (acc_issued)
                ptx::mbar_wait(BAR(C::kAccFull), 0, lim_ns, &no_abort, p.err, 5);
        }
    } else if (warp == C::kMmaWarp) {
        // ============================ MMA issuer ============================
        if (lane == 0 && n > 0) {
            const uint32_t idesc_qk = ptx::idesc_bf16_f32(128, 128, false);
            const uint32_t idesc_pv = ptx::idesc_bf16_f32(128, D, true);
            // Descriptors of the first K step of each operand; a later step only
            // moves the start address (the low 14 bits, in 16-byte units), which
            // never carries out of the field inside one tile.
            const uint64_t dq0 = ptx::smem_desc_sw128(sQ, 16, 1024);
            const uint64_t dkv0 = ptx::smem_desc_sw128(sKV, 16, 1024);
            const uint64_t dv0 = ptx::smem_desc_sw128(sKV, C::kBoxBytes, 1024);
            auto issue_qk = [&](int t, int slot) {
                const uint64_t qa = dq0 + ((t * C::kTileBytes) >> 4);
                const uint64_t kb = dkv0 + ((slot * C::kTileBytes) >> 4);
                const uint32_t dst = tmem + (t ? C::kColS1 : C::kColS0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
                    ptx::mma_ss(dst, qa + off, kb + off, idesc_qk, kk > 0);
                }
            };
            auto issue_pv = [&](int t, int slot, bool acc) {
                const uint64_t vb = dv0 + ((slot * C::kTileBytes) >> 4);
                const uint32_t dst = tmem + (t ? C::kColO1 : C::kColO0);
                const uint32_t pa = tmem + (t ? C::kColS1 : C::kColS0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    ptx::mma_ts(dst, pa + kk * 8, vb + ((kk * 2048) >> 4), idesc_pv, (acc || kk > 0) ? 1u : 0u);
            };
            // P_t(j) complete (every softmax thread arrived): O_t += P_t V_j.
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
                if (n0 > 0) {
                    issue_qk(0, 0);
                    ptx::mma_commit(BAR(C::kSF + 0));
                } else {
                    ptx::mma_commit(BAR(C::kOF + 0));  // tile 0 sees no key at all
                }
                issue_qk(1, 0);
                ptx::mma_commit(BAR(C::kSF + 1));
                ptx::mma_commit(BAR(C::kKVE + 0));
                if (n == 1)
                    ptx::mma_commit(BAR(C::kQFree));  // that was the last S MMA
            }
            for (int j = 0; ok && j < n; ++j) {
                const int vld = 2 * j + 1;
                const int vslot = vld % C::kStages;
                ok = ptx::mbar_wait(BAR(C::kKVF + vslot), (vld / C::kStages) & 1, lim_ns, abort_flag, p.err, 12);
                if (!ok)
                    break;
                // tile 0
                const bool more = j + 1 < n;
                if (j < n0) {
                    ok = pv_tile(0, vslot, j);
                    if (!ok)
                        break;
                    if (j + 1 < n0) {
                        const int kld = 2 * (j + 1);
                        kslot = kld % C::kStages;
                        ok = ptx::mbar_wait(BAR(C::kKVF + kslot), (kld / C::kStages) & 1, lim_ns, abort_flag,
                                            p.err, 14);
                        if (!ok)
                            break;
                        issue_qk(0, kslot);
                        ptx::mma_commit(BAR(C::kSF + 0));
                    } else {
                        ptx::mma_commit(BAR(C::kOF + 0));
                    }
                }
                // tile 1
                ok = pv_tile(1, vslot, j);
                if (!ok)
                    break;
                ptx::mma_commit(BAR(C::kKVE + vslot));
                if (more) {
                    if (j + 1 >= n0) {  // tile 0 did not wait for K(j+1)
                        const int kld = 2 * (j + 1);
                        kslot = kld % C::kStages;
                        ok = ptx::mbar_wait(BAR(C::kKVF + kslot), (kld / C::kStages) & 1, lim_ns, abort_flag,
                                            p.err, 14);
                        if (!ok)
                            break;
                    }
                    issue_qk(1, kslot);
                    ptx::mma_commit(BAR(C::kSF + 1));
                    ptx::mma_commit(BAR(C::kKVE + kslot));
                    if (j + 2 == n)
                        ptx::mma_commit(BAR(C::kQFree));  // that was the last S MMA
                } else {
                    ptx::mma_commit(BAR(C::kOF + 1));
                }
            }
            // Drain: every MMA this thread issued has finished before TMEM is freed.
            ptx::mma_commit(BAR(C::kDrain));
            volatile int no_abort = 0;
            ptx::mbar_wait(BAR(C::kDrain), 0, lim_ns, &no_abort, p.err, 16);
        }
        __syncwarp();
    } else {
        // ============================== softmax ==============================
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
        ctx.acc_staged = stage_acc;
        ctx.acc_smem[0] = acc_stage[0];
        ctx.acc_smem[1] = acc_stage[1];
        ctx.acc_box_bytes = C::kAccBoxBytes;
        ctx.bar_acc = BAR(C::kAccFull);
        ctx.abort_flag = abort_flag;
        ctx.lim_ns = lim_ns;
        softmax_warps<D, C::kTPR>(ctx, p, pr, q0, n, n0, kv_off, kv_len, bh, (int64_t)sp * pr.split_stride,
                         [&](int t) { ptx::mbar_arrive(BAR(C::kPF + t)); });
    }

    // ---- teardown --------------------------------------------------------------
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// [B*H, T, d] bf16 view with 128-row x 64-column boxes and 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *ptr, int64_t BH, int64_t T, int d)
{
    const uint64_t dims[3] = {(uint64_t)d, (uint64_t)T, (uint64_t)BH};
    const uint64_t strides[2] = {(uint64_t)d * 2, (uint64_t)T * d * 2};
    const uint32_t box[3] = {64, 128, 1};
    return make_bf16_map_sw128(m, ptr, 3, dims, strides, box);
}

// [B*H, out_T, d] fp32 accumulator view with 128-row x 32-column boxes and
// 128-byte swizzle.
bool make_acc_map(CUtensorMap *m, const float *acc, int64_t BH, int64_t out_T, int d)
{
    const uint64_t dims[3] = {(uint64_t)d, (uint64_t)out_T, (uint64_t)BH};
    const uint64_t strides[2] = {(uint64_t)d * 4, (uint64_t)out_T * d * 4};
    const uint32_t box[3] = {32, 128, 1};
    return make_f32_map_sw128(m, acc, 3, dims, strides, box);
}

template <int D>
cudaError_t launch_d(const void *q, const void *k, const void *v, const BlockParams &p_in, cudaStream_t s)
{
    const int64_t BH = (int64_t)p_in.B * p_in.H;
    CUtensorMap mq, mk, mv, macc;
    if (!make_map(&mq, q, BH, p_in.q_T, D) || !make_map(&mk, k, BH, p_in.T, D) || !make_map(&mv, v, BH, p_in.T, D))
        return cudaErrorInvalidValue;
    // Merging pairs stage their accumulator rows by TMA when they all fold into
    // one accumulator of one row pitch, unsplit (else the epilogue reads them
    // from global memory).
    BlockParams p = p_in;
    const PairDesc *first = nullptr;
    bool same = true;
    for (int i = 0; i < p.npairs; ++i) {
        const PairDesc &pr = p.pairs[i];
        if (pr.mode == kStore)
            continue;
        if (!first)
            first = &pr;
        else if (pr.acc != first->acc || pr.out_T != first->out_T)
            same = false;
        if (pr.split_stride != 0 || (reinterpret_cast<uintptr_t>(pr.acc) & 15u))
            same = false;
    }
    p.acc_staged = first && same && p.n_split == 1 && make_acc_map(&macc, first->acc, BH, first->out_T, D) ? 1 : 0;
    if (!p.acc_staged)
        memset(&macc, 0, sizeof macc);
    const int64_t grid = (int64_t)p.n_qgroups * p.npairs * BH * p.n_split;
    if (grid <= 0)
        return cudaSuccess;
    if (grid > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const uint32_t smem = Cfg<D>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(block_attn_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    block_attn_bf16_kernel<D><<<(unsigned)grid, Cfg<D>::kThreads, smem, s>>>(mq, mk, mv, macc, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_attn_bf16(const void *q, const void *k, const void *v, const BlockParams &p,
                                   cudaStream_t s)
{
    if (p.tc_kernel == 2 && block_attn_2sm_applies(p))
        return launch_block_attn_bf16_2sm(q, k, v, p, s);
    if (p.d == 128)
        return launch_d<128>(q, k, v, p, s);
    if (p.d == 64)
        return launch_d<64>(q, k, v, p, s);
    return cudaErrorInvalidValue;
}

}  // namespace rsa
