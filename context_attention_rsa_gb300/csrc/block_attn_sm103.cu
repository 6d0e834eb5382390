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
#include <mutex>

#include "ptx_sm103.cuh"
#include "rsa_internal.h"

namespace rsa {
namespace {

constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 256x

template <int D>
struct Cfg {
    static constexpr int kBoxes = D / 64;            // 128-byte-wide TMA boxes per tile
    static constexpr uint32_t kBoxBytes = 128u * 128u; // 128 rows x 128 bytes
    static constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;
    static constexpr int kStages = D == 128 ? 4 : 6;
    static constexpr uint32_t kQOff = 0;
    static constexpr uint32_t kKVOff = 2 * kTileBytes;
    static constexpr uint32_t kBarOff = kKVOff + kStages * kTileBytes;
    static constexpr uint32_t kXchOff = kBarOff + 256;  // [2 tiles][2 halves][128 rows] floats
    static constexpr uint32_t kSmemBytes = kXchOff + 2048 + 1024;
    static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
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

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Named barrier 1 over the 256 softmax threads (warps 0-7).
__device__ __forceinline__ void softmax_bar_sync()
{
    asm volatile("barrier.cta.sync 1, 256;" ::: "memory");
}

// The same barrier, returning whether `v` holds in every softmax thread, so
// that a decision to give up is taken by all of them together.
__device__ __forceinline__ bool softmax_bar_and(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "barrier.cta.red.and.pred po, 1, 256, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Keep uses of r[0..31] after a preceding volatile asm (the TMEM load wait).
__device__ __forceinline__ void tie32(uint32_t *r)
{
#pragma unroll
    for (int i = 0; i < 32; ++i)
        asm volatile("" : "+r"(r[i]));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    block_attn_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
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
    const int64_t kv_off = pr.kv_off + (int64_t)sp * p.kv_split;
    const int64_t kv_len = p.kv_split > 0 ? min(p.kv_split, p.kv_len - (int64_t)sp * p.kv_split) : p.kv_len;
    const int64_t q0 = (int64_t)qg * kBf16RowsPerCta;
    const int64_t rows_valid = min((int64_t)kBf16RowsPerCta, p.q_len - q0);
    int64_t kv_end = kv_len;
    if (p.causal)
        kv_end = min(kv_end, pr.q_off + q0 + rows_valid - kv_off);
    const int n = kv_end > 0 ? (int)((kv_end + 127) / 128) : 0;

    if (threadIdx.x == 0) {
        ptx::mbar_init(BAR(C::kQF), 1);
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(BAR(C::kKVF + s), 1);
            ptx::mbar_init(BAR(C::kKVE + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(BAR(C::kSF + t), 1);
            ptx::mbar_init(BAR(C::kPF + t), 256);
            ptx::mbar_init(BAR(C::kOF + t), 1);
        }
        ptx::mbar_init(BAR(C::kDrain), 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 9) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        ptx::tma_prefetch_desc(&tm_q);
        ptx::tma_prefetch_desc(&tm_k);
        ptx::tma_prefetch_desc(&tm_v);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t lim_ns = p.wait_limit_ns;

    if (warp == 8) {
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
            for (int ld = 0; ld < 2 * n; ++ld) {
                const int slot = ld % C::kStages;
                const int use = ld / C::kStages;
                if (use > 0 &&
                    !ptx::mbar_wait(BAR(C::kKVE + slot), (use - 1) & 1, lim_ns, abort_flag, p.err, 1))
                    break;
                const CUtensorMap *m = (ld & 1) ? &tm_v : &tm_k;
                const int row = (int)(kv_off + (int64_t)(ld >> 1) * 128);
                ptx::mbar_arrive_expect_tx(BAR(C::kKVF + slot), C::kTileBytes);
                for (int b = 0; b < C::kBoxes; ++b)
                    ptx::tma_load_3d(sKV + slot * C::kTileBytes + b * C::kBoxBytes, m,
                                     BAR(C::kKVF + slot), b * 64, row, bh);
                last_use[slot] = use;
            }
            // Let every copy this thread started land before the CTA can exit.
            volatile int no_abort = 0;
            ptx::mbar_wait(BAR(C::kQF), 0, lim_ns, &no_abort, p.err, 2);
            for (int s = 0; s < C::kStages; ++s)
                if (last_use[s] >= 0)
                    ptx::mbar_wait(BAR(C::kKVF + s), last_use[s] & 1, lim_ns, &no_abort, p.err, 3);
        }
    } else if (warp == 9) {
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
            bool ok = ptx::mbar_wait(BAR(C::kQF), 0, lim_ns, abort_flag, p.err, 10);
            int kslot = 0;
            if (ok)
                ok = ptx::mbar_wait(BAR(C::kKVF + 0), 0, lim_ns, abort_flag, p.err, 11);
            if (ok) {
                issue_qk(0, 0);
                ptx::mma_commit(BAR(C::kSF + 0));
                issue_qk(1, 0);
                ptx::mma_commit(BAR(C::kSF + 1));
                ptx::mma_commit(BAR(C::kKVE + 0));
            }
            for (int j = 0; ok && j < n; ++j) {
                const int vld = 2 * j + 1;
                const int vslot = vld % C::kStages;
                ok = ptx::mbar_wait(BAR(C::kKVF + vslot), (vld / C::kStages) & 1, lim_ns, abort_flag, p.err, 12);
                if (!ok)
                    break;
                // tile 0
                ok = ptx::mbar_wait(BAR(C::kPF + 0), j & 1, lim_ns, abort_flag, p.err, 13);
                if (!ok)
                    break;
                ptx::tc_fence_after();
                issue_pv(0, vslot, j > 0);
                const bool more = j + 1 < n;
                if (more) {
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
                // tile 1
                ok = ptx::mbar_wait(BAR(C::kPF + 1), j & 1, lim_ns, abort_flag, p.err, 15);
                if (!ok)
                    break;
                ptx::tc_fence_after();
                issue_pv(1, vslot, j > 0);
                ptx::mma_commit(BAR(C::kKVE + vslot));
                if (more) {
                    issue_qk(1, kslot);
                    ptx::mma_commit(BAR(C::kSF + 1));
                    ptx::mma_commit(BAR(C::kKVE + kslot));
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
        // All eight warps work on tile 0's S, then on tile 1's (the tiles
        // alternate on the tensor cores).  Two threads share a row: warp w
        // holds TMEM lanes 32*(w%4).. and column half h = w/4, i.e. keys
        // [64h, 64h+64) of every 128-key step and output columns
        // [h*d/2, (h+1)*d/2).  The two halves of a row agree on the row max
        // through shared memory; each keeps its own part of the row sum.
        const int h = warp >> 2;
        const int wi = warp & 3;
        const int row = wi * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(wi * 32) << 16;
        float *xch = reinterpret_cast<float *>(gbase + C::kXchOff);  // [tile][half][row]
        const float sl2 = 1.4426950408889634f / sqrtf((float)D);   // log2(e) / sqrt(d)
        float m_used[2] = {-INFINITY, -INFINITY};                    // kept maxima, log2 units
        float l[2] = {0.f, 0.f};                                     // this half's row sums
        int64_t allowed[2];  // keys [0, allowed) of this split visible to the row, per tile
        for (int t = 0; t < 2; ++t) {
            const int64_t qpos = pr.q_off + q0 + t * 128 + row;
            allowed[t] = p.causal ? min(kv_len, qpos - kv_off + 1) : kv_len;
        }
        bool ok = true;
        for (int j = 0; ok && j < n; ++j) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const uint32_t tS = tmem + lane_addr + (t ? C::kColS1 : C::kColS0);
                const uint32_t tO = tmem + lane_addr + (t ? C::kColO1 : C::kColO0);
                bool got = ptx::mbar_wait(BAR(C::kSF + t), j & 1, lim_ns, abort_flag, p.err, 20);
                got = __all_sync(0xffffffffu, got);
                uint32_t s[64];
                float mx = -INFINITY;
                if (got) {
                    ptx::tc_fence_after();
                    ptx::tmem_ld32(tS + 64 * h, s);
                    ptx::tmem_ld32(tS + 64 * h + 32, s + 32);
                    ptx::tmem_ld_wait(s);
                    tie32(s + 32);
                    const int64_t lim = allowed[t] - (int64_t)j * 128 - 64 * h;
                    if (lim < 64) {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            if ((int64_t)i >= lim)
                                s[i] = f2u(-INFINITY);
                    }
                    // row max of this half: four independent chains of three-input max
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int i = 0; i < 64; i += 8) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            m4[c] = fmax3(m4[c], u2f(s[i + 2 * c]), u2f(s[i + 2 * c + 1]));
                    }
                    mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
                    xch[(t * 2 + h) * 128 + row] = mx;
                }
                // Every S load of this tile is done (and every thread knows
                // whether all waits succeeded) before any half writes P over S.
                ptx::tc_fence_before();
                ok = softmax_bar_and(got);
                ptx::tc_fence_after();
                if (!ok)
                    break;
                mx = fmaxf(mx, xch[(t * 2 + (h ^ 1)) * 128 + row]);
                const float mnew = mx * sl2;
                const bool need =
                    (mnew > -INFINITY) && (m_used[t] == -INFINITY || mnew > m_used[t] + kRescaleThreshold);
                if (__any_sync(0xffffffffu, need)) {
                    float alpha = 1.f;
                    if (need) {
                        alpha = (m_used[t] == -INFINITY) ? 0.f : ptx::ex2(m_used[t] - mnew);
                        l[t] *= alpha;
                        m_used[t] = mnew;
                    }
                    if (j > 0) {
                        // the commit that signalled S_t(j) also covered PV_t(j-1): O_t is stable
                        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
                        for (int c = 0; c < D / 64; ++c) {
                            uint32_t o[32];
                            const uint32_t ta = tO + h * (D / 2) + c * 32;
                            ptx::tmem_ld32(ta, o);
                            ptx::tmem_ld_wait(o);
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                const float2 r = __fmul2_rn(make_float2(u2f(o[i]), u2f(o[i + 1])), a2);
                                o[i] = f2u(r.x);
                                o[i + 1] = f2u(r.y);
                            }
                            ptx::tmem_st32(ta, o);
                        }
                    }
                }
                // p = 2^(s * log2(e)/sqrt(d) - m), written over S as bf16 pairs:
                // keys [64h, 64h+64) are packed columns [32h, 32h+32)
                const float neg = (m_used[t] == -INFINITY) ? 0.f : -m_used[t];
                const float2 c2 = make_float2(sl2, sl2);
                const float2 n2 = make_float2(neg, neg);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float2 x = __ffma2_rn(make_float2(u2f(s[2 * i]), u2f(s[2 * i + 1])), c2, n2);
                    const float p0 = ptx::ex2(x.x);
                    const float p1 = ptx::ex2(x.y);
                    acc[i & 3] = __fadd2_rn(acc[i & 3], make_float2(p0, p1));
                    pk[i] = pack_bf16(p0, p1);
                }
                ptx::tmem_st32(tS + 32 * h, pk);
                const float2 a01 = __fadd2_rn(acc[0], acc[1]);
                const float2 a23 = __fadd2_rn(acc[2], acc[3]);
                const float2 a = __fadd2_rn(a01, a23);
                l[t] += a.x + a.y;
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(BAR(C::kPF + t));
            }
        }
        // ---- epilogue: O / l and lse for both tiles --------------------------------
        bool fin = ok;
        for (int t = 0; t < 2 && fin && n > 0; ++t) {
            fin = ptx::mbar_wait(BAR(C::kOF + t), 0, lim_ns, abort_flag, p.err, 21);
            fin = __all_sync(0xffffffffu, fin);
        }
        softmax_bar_sync();  // the exchange slots are free again
        if (ok) {
            xch[(0 * 2 + h) * 128 + row] = l[0];
            xch[(1 * 2 + h) * 128 + row] = l[1];
        }
        fin = softmax_bar_and(fin && ok);
        if (fin) {
            ptx::tc_fence_after();
#pragma unroll 1
            for (int t = 0; t < 2; ++t) {
                const float lt = l[t] + xch[(t * 2 + (h ^ 1)) * 128 + row];
                const uint32_t tO = tmem + lane_addr + (t ? C::kColO1 : C::kColO0);
                const int64_t rg = q0 + t * 128 + row;  // row inside the pair
                const bool valid = rg < p.q_len;
                const int64_t orow = (int64_t)bh * pr.out_T + pr.out_t0 + rg + (int64_t)sp * pr.split_stride;
                // This pair's result is (O / l, lse_b).  A merging epilogue folds it
                // into the running (acc, lse) as the merge kernel does:
                // M = max(a, b), L = M + ln(e^{a-M} + e^{b-M}), o = acc e^{a-L} + o_b e^{b-L}.
                const bool empty = !(lt > 0.f);
                const float lse_b = empty ? -INFINITY : (m_used[t] + ptx::lg2(lt)) * 0.69314718055994531f;
                float wa = 0.f;                     // weight of the accumulator row
                float wb = empty ? 0.f : 1.f / lt;  // weight of the unnormalised O row
                float lse_out = lse_b;
                const bool merging = pr.mode != kStore;
                if (merging && valid) {
                    const float a = pr.lse[orow];
                    const float M = fmaxf(a, lse_b);
                    if (M > -INFINITY) {
                        const float ea = ptx::ex2((a - M) * 1.4426950408889634f);
                        const float eb = ptx::ex2((lse_b - M) * 1.4426950408889634f);
                        const float tot = ea + eb;
                        const float inv = 1.f / tot;
                        lse_out = M + ptx::lg2(tot) * 0.69314718055994531f;
                        wa = ea * inv;
                        wb = empty ? 0.f : eb * inv / lt;
                    } else {
                        lse_out = -INFINITY;
                        wb = 0.f;
                    }
                }
                softmax_bar_sync();  // both halves have read the running lse
                if (valid && h == 0)
                    pr.lse[orow] = lse_out;
#pragma unroll 1
                for (int c = 0; c < D / 64; ++c) {
                    const int col = h * (D / 2) + c * 32;  // first output column of this chunk
                    uint32_t o[32];
                    if (n > 0) {
                        ptx::tmem_ld32(tO + col, o);
                        ptx::tmem_ld_wait(o);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = 0u;
                    }
                    if (valid) {
                        float v[32];
                        if (merging) {
                            const float4 *src = reinterpret_cast<const float4 *>(pr.acc + orow * D + col);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float4 x = src[i];
                                v[4 * i] = fmaf(u2f(o[4 * i]), wb, x.x * wa);
                                v[4 * i + 1] = fmaf(u2f(o[4 * i + 1]), wb, x.y * wa);
                                v[4 * i + 2] = fmaf(u2f(o[4 * i + 2]), wb, x.z * wa);
                                v[4 * i + 3] = fmaf(u2f(o[4 * i + 3]), wb, x.w * wa);
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                v[i] = u2f(o[i]) * wb;
                        }
                        if (pr.out_f32) {
                            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(pr.out) + orow * D + col);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                        } else {
                            uint4 *dst =
                                reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(pr.out) + orow * D + col);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                dst[i] = make_uint4(pack_bf16(v[8 * i], v[8 * i + 1]), pack_bf16(v[8 * i + 2], v[8 * i + 3]),
                                                    pack_bf16(v[8 * i + 4], v[8 * i + 5]),
                                                    pack_bf16(v[8 * i + 6], v[8 * i + 7]));
                        }
                    }
                }
            }
        }
    }

    // ---- teardown --------------------------------------------------------------
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 9) {
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

template <int D>
cudaError_t launch_d(const void *q, const void *k, const void *v, const BlockParams &p, cudaStream_t s)
{
    const int64_t BH = (int64_t)p.B * p.H;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, BH, p.q_T, D) || !make_map(&mk, k, BH, p.T, D) || !make_map(&mv, v, BH, p.T, D))
        return cudaErrorInvalidValue;
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
    block_attn_bf16_kernel<D><<<(unsigned)grid, kThreads, smem, s>>>(mq, mk, mv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_attn_bf16(const void *q, const void *k, const void *v, const BlockParams &p,
                                   cudaStream_t s)
{
    if (p.d == 128)
        return launch_d<128>(q, k, v, p, s);
    if (p.d == 64)
        return launch_d<64>(q, k, v, p, s);
    return cudaErrorInvalidValue;
}

}  // namespace rsa
