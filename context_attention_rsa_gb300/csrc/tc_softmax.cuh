// The softmax warps of the two tensor-core block-attention kernels (one-SM and
// two-SM): per 128-key step, read S = Q K^T of each 128-row tile from TMEM,
// mask, keep the running row maximum, rescale O when it grows, write
// P = 2^{s log2(e)/sqrt(d) - m} as bf16 back over S for the PV MMA, and at
// the end write o = O / l and lse (or fold them into a ring accumulator).
//
// Pages: "Sequence parallelism -- splitting the token dimension across GPUs"
// (llmdaily, day 58): softmax(Q K^T / sqrt(d_k)) V of "Attention wants keys
// and values from other tokens", the running (m, l, o) statistics and the
// e^{m - m_new} rescale of "But softmax seems to require all attention scores
// at once" (here between 128-key tiles), and the causal mask of "Causal
// attention gives us another optimization".
//
// Thread layout (warps 0-7 of the CTA): warp w reads TMEM lanes
// 32*(w%4).. (one query row per lane) and takes column half h = w/4 of every
// step: keys [64h, 64h+64), output columns [h*d/2, (h+1)*d/2).  The two
// halves of a row agree on the row max through shared memory behind a named
// barrier and keep their own part of the row sum l.
//
// Each thread packs its P values into bf16 pairs and writes them with one
// TMEM store (32 packed columns for 64 keys), waits for it, and calls
// arrive(t): once every softmax thread has arrived, P_t and the rescaled O_t
// are complete in TMEM for the PV MMA.
// The kept maximum m only moves when the new one exceeds it by more than 8
// (log2 units); o, l and lse all use the same m, so the result is exact up
// to rounding whatever m is kept.
#pragma once

#include <cuda_bf16.h>

#include <cmath>

#include "ptx_sm103.cuh"
#include "rsa_internal.h"
#include "tc_common.cuh"

namespace rsa {
namespace tc {

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 256x

// Where one CTA's softmax warps find their TMEM tiles, barriers and scratch.
struct SoftmaxCtx {
    uint32_t tmem;        // TMEM base address of this CTA
    uint32_t col_s[2];    // S (and P) columns of tiles 0 and 1
    uint32_t col_o[2];    // O columns of tiles 0 and 1
    uint32_t bar_sf[2];   // S-full barriers of this CTA (one arrival per S_t(j))
    uint32_t bar_of[2];   // O-final barriers of this CTA
    float *xch;           // shared scratch: [2 tiles][2 halves][128 rows] floats
    volatile int *abort_flag;
    uint64_t lim_ns;
    // A merging epilogue with staged accumulator rows: tile t's rows are at
    // acc_smem[t] as 32-column boxes of 128 rows x 128 bytes (128-byte
    // swizzle), acc_box_bytes apart, complete once bar_acc's phase 0 is.
    bool acc_staged = false;
    uint32_t acc_smem[2] = {0u, 0u};
    uint32_t acc_box_bytes = 0;
    uint32_t bar_acc = 0;
};

// A load issued where it stands (the value is needed much later).
__device__ __forceinline__ float ld_global_early(const float *p)
{
    float v;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// Rows [q0, q0 + 256) of pair `pr` (two tiles of 128), keys [kv_off,
// kv_off + kv_len) in n steps of 128; tile 0 takes only the first n0 <= n of
// them (the MMA issuer computes no S, P or PV of tile 0 after those).  Output row r of the pair goes to row
// bh * out_T + out_t0 + r + row_off.  TPR threads share each query row (TPR =
// 2 or 4): the first 128 * TPR threads of the CTA call this, and all leave it
// together.  Thread (warp w, lane) reads TMEM lane 32 (w mod 4) + lane and takes
// part h = w / 4 of every step: keys [h K, h K + K) with K = 128 / TPR, and
// output columns [h D / TPR, (h + 1) D / TPR).
template <int D, int TPR, class Arrive>
__device__ __forceinline__ void softmax_warps(const SoftmaxCtx &c, const BlockParams &p, const PairDesc &pr,
                                              int64_t q0, int n, int n0, int64_t kv_off, int64_t kv_len,
                                              int bh, int64_t row_off, Arrive arrive)
{
    static_assert(TPR == 2 || TPR == 4, "two or four threads per query row");
    constexpr int NT = 128 * TPR;     // softmax threads
    constexpr int K = 128 / TPR;      // keys of a step per thread
    constexpr int OC = D / TPR;       // output columns per thread
    static_assert(OC % 32 == 0, "output columns come in 32-column TMEM loads");
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int h = warp >> 2;
    const int wi = warp & 3;
    const int row = wi * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(wi * 32) << 16;
    float *xch = c.xch;  // [2 tiles][TPR parts][128 rows]
    const float sl2 = 1.4426950408889634f / sqrtf((float)D);  // log2(e) / sqrt(d)
    float m_used[2] = {-INFINITY, -INFINITY};                   // kept maxima, log2 units
    float l[2] = {0.f, 0.f};                                    // this part's row sums
    int64_t allowed[2];  // keys [0, allowed) of the key range visible to the row, per tile
    float lse_run[2] = {-INFINITY, -INFINITY};  // the running lse a merging epilogue folds into
    for (int t = 0; t < 2; ++t) {
        const int64_t qpos = pr.q_off + q0 + t * 128 + row;
        allowed[t] = p.causal ? min(kv_len, qpos - kv_off + 1) : kv_len;
        // Only this CTA writes its rows' running lse, and only in the epilogue:
        // load it now so that its latency hides under the main loop.
        const int64_t rg = q0 + t * 128 + row;
        const int64_t orow = (int64_t)bh * pr.out_T + pr.out_t0 + rg + row_off;
        if (pr.mode != kStore && rg < p.q_len && RSA_DCHECK(orow >= 0 && orow < pr.out_rows, p.err, 0x32, orow))
            lse_run[t] = ld_global_early(pr.lse + orow);
    }
    bool ok = true;
    for (int j = 0; ok && j < n; ++j) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (t == 0 && j >= n0)
                continue;  // the same for every softmax thread
            const uint32_t tS = c.tmem + lane_addr + c.col_s[t];
            const uint32_t tO = c.tmem + lane_addr + c.col_o[t];
            bool got = ptx::mbar_wait(c.bar_sf[t], j & 1, c.lim_ns, c.abort_flag, p.err, 20);
            got = __all_sync(0xffffffffu, got);
            uint32_t s[K];
            float mx = -INFINITY;
            if (got) {
                ptx::tc_fence_after();
                if constexpr (K == 64) {
                    ptx::tmem_ld64(tS + K * h, s);
                    ptx::tmem_ld_wait64(s);
                } else {
                    ptx::tmem_ld32(tS + K * h, s);
                    ptx::tmem_ld_wait(s);
                }
                const int64_t lim = allowed[t] - (int64_t)j * 128 - K * h;
                if (lim < K) {
#pragma unroll
                    for (int i = 0; i < K; ++i)
                        if ((int64_t)i >= lim)
                            s[i] = f2u(-INFINITY);
                }
                // row max of this part: four independent chains of three-input max
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < K; i += 8) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        m4[k] = fmax3(m4[k], u2f(s[i + 2 * k]), u2f(s[i + 2 * k + 1]));
                }
                mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
                xch[(t * TPR + h) * 128 + row] = mx;
            }
            // Every S load of this tile is done (and every softmax thread knows
            // whether every wait succeeded) before any part writes P over S.
            ptx::tc_fence_before();
            ok = softmax_bar_and<NT>(got);
            ptx::tc_fence_after();
            if (!ok)
                break;
#pragma unroll
            for (int o = 1; o < TPR; ++o)
                mx = fmaxf(mx, xch[(t * TPR + ((h + o) % TPR)) * 128 + row]);
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
                    for (int k = 0; k < OC / 32; ++k) {
                        uint32_t o[32];
                        const uint32_t ta = tO + h * OC + k * 32;
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
            // p = 2^(s * log2(e)/sqrt(d) - m) as bf16 pairs over S: keys
            // [K h, K h + K) go to packed columns [K h / 2, K h / 2 + K / 2).
            const float neg = (m_used[t] == -INFINITY) ? 0.f : -m_used[t];
            const float2 c2 = make_float2(sl2, sl2);
            const float2 n2 = make_float2(neg, neg);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
            uint32_t pk[K / 2];
#pragma unroll
            for (int i = 0; i < K / 2; ++i) {
                const float2 x = __ffma2_rn(make_float2(u2f(s[2 * i]), u2f(s[2 * i + 1])), c2, n2);
                const float p0 = ptx::ex2(x.x);
                const float p1 = ptx::ex2(x.y);
                acc[i & 3] = __fadd2_rn(acc[i & 3], make_float2(p0, p1));
                pk[i] = pack_bf16(p0, p1);
            }
            if constexpr (K == 64)
                ptx::tmem_st32(tS + (K / 2) * h, pk);
            else
                ptx::tmem_st16(tS + (K / 2) * h, pk);
            // P and the rescaled O complete before the MMA may read them
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            arrive(t);
            const float2 a01 = __fadd2_rn(acc[0], acc[1]);
            const float2 a23 = __fadd2_rn(acc[2], acc[3]);
            const float2 a = __fadd2_rn(a01, a23);
            l[t] += a.x + a.y;
        }
    }
    // ---- epilogue: O / l and lse for both tiles --------------------------------
    bool fin = ok;
    for (int t = 0; t < 2 && fin && n > 0; ++t) {
        fin = ptx::mbar_wait(c.bar_of[t], 0, c.lim_ns, c.abort_flag, p.err, 21);
        fin = __all_sync(0xffffffffu, fin);
    }
    if (c.acc_staged && fin) {
        fin = ptx::mbar_wait(c.bar_acc, 0, c.lim_ns, c.abort_flag, p.err, 22);
        fin = __all_sync(0xffffffffu, fin);
    }
    softmax_bar_sync<NT>();  // the exchange slots are free again
    if (ok) {
        xch[(0 * TPR + h) * 128 + row] = l[0];
        xch[(1 * TPR + h) * 128 + row] = l[1];
    }
    fin = softmax_bar_and<NT>(fin && ok);
    if (!fin)
        return;
    ptx::tc_fence_after();
#pragma unroll 1
    for (int t = 0; t < 2; ++t) {
        float lt = l[t];
#pragma unroll
        for (int o = 1; o < TPR; ++o)
            lt += xch[(t * TPR + ((h + o) % TPR)) * 128 + row];
        const uint32_t tO = c.tmem + lane_addr + c.col_o[t];
        const int64_t rg = q0 + t * 128 + row;  // row inside the pair
        const int64_t orow = (int64_t)bh * pr.out_T + pr.out_t0 + rg + row_off;
        const bool valid = rg < p.q_len && RSA_DCHECK(orow >= 0 && orow < pr.out_rows, p.err, 0x31, orow);
        // This pair's result is (O / l, lse_b).  A merging epilogue folds it
        // into the running (acc, lse) as the merge kernel does:
        // M = max(a, b), L = M + ln(e^{a-M} + e^{b-M}), o = acc e^{a-L} + o_b e^{b-L}.
        const bool empty = !(lt > 0.f);
        const float lse_b = empty ? -INFINITY : (m_used[t] + ptx::lg2(lt)) * 0.69314718055994531f;
        float wa = 0.f;                     // weight of the accumulator row
        float wb = empty ? 0.f : 1.f / lt;  // weight of the unnormalised O row
        float lse_out = lse_b;
        const bool merging = pr.mode != kStore;
        bool use_acc = false;  // an accumulator row with lse = -inf is empty: not read
        if (merging && valid) {
            const float a = lse_run[t];
            use_acc = a > -INFINITY;
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
        if (valid && h == 0)
            pr.lse[orow] = lse_out;
#pragma unroll 1
        for (int k = 0; k < OC / 32; ++k) {
            const int col = h * OC + k * 32;  // first output column of this chunk
            uint32_t o[32];
            if ((t == 0 ? n0 : n) > 0) {  // a tile with no key step has no O
                ptx::tmem_ld32(tO + col, o);
                ptx::tmem_ld_wait(o);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    o[i] = 0u;
            }
            if (valid) {
                float v[32];
                if (use_acc) {
                    const float4 *src = reinterpret_cast<const float4 *>(pr.acc + orow * D + col);
                    // staged: row `row` of box col/32, 16-byte piece i at i ^ (row & 7)
                    const uint32_t line = c.acc_smem[t] + (uint32_t)(col / 32) * c.acc_box_bytes + (uint32_t)row * 128u;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 x = c.acc_staged ? ld_shared_v4(line + ((uint32_t)(i ^ (row & 7)) << 4)) : src[i];
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
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(pr.out) + orow * D + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(pack_bf16(v[8 * i], v[8 * i + 1]), pack_bf16(v[8 * i + 2], v[8 * i + 3]),
                                            pack_bf16(v[8 * i + 4], v[8 * i + 5]), pack_bf16(v[8 * i + 6], v[8 * i + 7]));
                }
            }
        }
    }
}

}  // namespace tc
}  // namespace rsa
