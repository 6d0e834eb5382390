// Two-pass Ring Self-Attention on the GPU.
//
// Page: "Sequence Parallelism" (glossary entry, zhongzhoutan-coder terms),
// section "How It Works": the key chunks circulate first, so each query chunk
// n builds its full score rows S^n (L/N x L); the value chunks then circulate
// and chunk n accumulates the weighted sums over them to produce O^n.  Softmax
// is taken over each full row between the two passes.
//
// Unlike the online-softmax ring, this form materialises S^n: per query chunk
// an fp32 [B*H, Tc, T] score buffer and a bf16 [B*H, Tc, T] probability
// buffer -- the O(L/N * L) memory the online merge avoids.  Chunks are done one
// after another, reusing the buffers:
//   score kernel   S^n = Q_n K^T / sqrt(d) (tcgen05, 128x128 tiles, one
//                  persistent CTA per SM), causal entries set to -inf.  Each
//                  tile is staged in shared memory and written by TMA stores;
//                  each row also leaves, per 64 keys, (max, sum of e^{s - max})
//                  in a small statistics buffer
//   softmax kernel row max and sum over the whole row from those statistics
//                  (one warp per row), then one pass over the row:
//                  P^n = e^{s - m} / l in bf16, lse = m + ln l
//   PV kernel      O^n = sum over key chunks in ring order (n - r) mod N of
//                  P^n_j V_j (tcgen05, 128 rows per CTA, fp32 accumulator)
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "ptx_sm103.cuh"
#include "rsa_internal.h"
#include "tc_common.cuh"

namespace rsa {
namespace {

constexpr int D = 128;
constexpr uint32_t kBoxBytes = 128u * 128u;  // 128 rows x 128 bytes (64 bf16)
constexpr uint32_t kTileBytes = 2 * kBoxBytes;  // 128 rows x 128 bf16

struct TwoPassParams {
    int64_t BH, T, Tc;
    int n;        // query chunk
    int N;
    int causal;
    float *S;              // [BH, Tc, T] fp32 scores of chunk n
    float2 *stats;         // [BH, Tc, T/64]: per row and 64 keys, (max, sum of e^{s - max})
    __nv_bfloat16 *out;    // [BH, T, d]
    uint64_t wait_limit_ns;
    unsigned int *err;
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void st_shared_v4(uint32_t addr, float a, float b, float c, float d)
{
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// Named barrier 1 over the 256 epilogue threads of the score kernel (warps 0-7);
// it returns whether `v` holds in all of them.
__device__ __forceinline__ bool epi_bar_and(bool v)
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

// ---- score pass ---------------------------------------------------------------
// One persistent CTA per SM walks a contiguous range of the chunk's score tiles
// (head, query tile, key tile), key tile fastest, so Q is loaded once per run of
// key tiles.  Warp 8 issues the TMA loads (Q, and K through two stages), warp 9
// the MMAs into two TMEM accumulators of 128 columns, and warps 0-7 the
// epilogue: warp w takes the rows 32 (w mod 4) .. +31 and the 64-key half
// h = w / 4 of each tile.  It scales and masks its half, leaves the half's
// (max, sum of e^{s - max}) per row in the statistics buffer, and stages its two
// 32-column fp32 chunks for the TMA stores.  Staging holds two tiles, so the
// stores of one tile run while the next is formed.
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kScoreThreads = kEpiThreads + 64;
constexpr int kKStages = 2;  // K tiles in flight
constexpr uint32_t kChunkBytes = 128u * 32u * 4u;  // 128 rows x 32 fp32 columns
constexpr uint32_t kScoreSQ = 0, kScoreSK = kTileBytes, kScoreOut = (1 + kKStages) * kTileBytes;
constexpr uint32_t kScoreBars = kScoreOut + 2 * 4 * kChunkBytes;  // two tiles of four chunks
// mbarriers: Q full/empty, K full/empty per stage, accumulator full/empty (two), done
constexpr int kBarKF = 2, kBarKE = kBarKF + kKStages, kBarAF = kBarKE + kKStages, kBarAE = kBarAF + 2,
              kBarDone = kBarAE + 2, kNumBars = kBarDone + 1;
static_assert(8 * kNumBars + 8 <= 128, "score kernel barrier area");
constexpr uint32_t kScoreSmem = kScoreBars + 128 + 1024;
static_assert(kScoreSmem <= 227u * 1024u, "score kernel shared memory");

// Wait until at most N bulk store groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Position in the chunk's tile order (head, query tile, key tile), key tile
// fastest; one division to start, then counters.
struct TileWalk {
    int bh, qt, kt;
    __device__ __forceinline__ void start(int64_t t, int n_qt, int n_kt)
    {
        bh = (int)(t / ((int64_t)n_qt * n_kt));
        const int64_t r = t - (int64_t)bh * n_qt * n_kt;
        qt = (int)(r / n_kt);
        kt = (int)(r - (int64_t)qt * n_kt);
    }
    __device__ __forceinline__ void next(int n_qt, int n_kt)
    {
        if (++kt == n_kt) {
            kt = 0;
            if (++qt == n_qt) {
                qt = 0;
                ++bh;
            }
        }
    }
};

// Causal and every key of the tile after every query of it.  Such tiles end a
// run of key tiles; key tile 0 never is one.
__device__ __forceinline__ bool tile_masked(const TwoPassParams &p, int qt, int kt)
{
    return p.causal && (int64_t)kt * 128 > (int64_t)p.n * p.Tc + (int64_t)qt * 128 + 127;
}

__global__ void __launch_bounds__(kScoreThreads)
    score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ TwoPassParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *g = smem_raw + (base - raw);
    const uint32_t bars = base + kScoreBars;
    const uint32_t Q_FULL = bars, Q_EMPTY = bars + 8, DONE = bars + 8u * kBarDone;
    auto K_FULL = [&](int s) { return bars + 8u * (kBarKF + s); };
    auto K_EMPTY = [&](int s) { return bars + 8u * (kBarKE + s); };
    auto A_FULL = [&](int a) { return bars + 8u * (kBarAF + a); };
    auto A_EMPTY = [&](int a) { return bars + 8u * (kBarAE + a); };
    uint32_t *tslot = reinterpret_cast<uint32_t *>(g + kScoreBars + 8 * kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(g + kScoreBars + 8 * kNumBars + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_qt = (int)(p.Tc / 128), n_kt = (int)(p.T / 128);
    const int64_t total = p.BH * n_qt * n_kt;
    const int64_t t0 = total * blockIdx.x / gridDim.x, t1 = total * (blockIdx.x + 1) / gridDim.x;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i)  // A_EMPTY counts every epilogue thread
            ptx::mbar_init(bars + 8 * i, (i == kBarAE || i == kBarAE + 1) ? kEpiThreads : 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kEpiWarps + 1) {
        ptx::tmem_alloc(ptx::smem_u32(tslot), 256);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == kEpiWarps) {
        if (lane == 0) {
            TileWalk w;
            w.start(t0, n_qt, n_kt);
            int q_bh = -1, q_qt = -1, qloads = 0;
            int64_t ki = 0;  // key tiles loaded so far
            bool ok = true;
            for (int64_t t = t0; ok && t < t1; ++t, w.next(n_qt, n_kt)) {
                if (tile_masked(p, w.qt, w.kt))
                    continue;
                if (w.bh != q_bh || w.qt != q_qt) {
                    // the MMAs on the previous Q are done before it is overwritten
                    if (qloads > 0 &&
                        !(ok = ptx::mbar_wait(Q_EMPTY, (uint32_t)((qloads - 1) & 1), p.wait_limit_ns, abort_flag, p.err, 40)))
                        break;
                    ptx::mbar_arrive_expect_tx(Q_FULL, kTileBytes);
                    for (int b = 0; b < 2; ++b)
                        ptx::tma_load_3d(base + kScoreSQ + b * kBoxBytes, &tm_q, Q_FULL, b * 64,
                                         (int)((int64_t)p.n * p.Tc + (int64_t)w.qt * 128), w.bh);
                    q_bh = w.bh;
                    q_qt = w.qt;
                    ++qloads;
                }
                const int s = (int)(ki % kKStages);
                if (ki >= kKStages &&
                    !(ok = ptx::mbar_wait(K_EMPTY(s), (uint32_t)((ki / kKStages - 1) & 1), p.wait_limit_ns, abort_flag,
                                          p.err, 41)))
                    break;
                ptx::mbar_arrive_expect_tx(K_FULL(s), kTileBytes);
                for (int b = 0; b < 2; ++b)
                    ptx::tma_load_3d(base + kScoreSK + s * kTileBytes + b * kBoxBytes, &tm_k, K_FULL(s), b * 64,
                                     w.kt * 128, w.bh);
                ++ki;
            }
            // no copy is still in flight when the CTA exits: the last fill of
            // each buffer has landed (earlier fills were consumed before it)
            volatile int no_abort = 0;
            if (qloads > 0)
                ptx::mbar_wait(Q_FULL, (uint32_t)((qloads - 1) & 1), p.wait_limit_ns, &no_abort, p.err, 42);
            for (int64_t last = ki - 1; last >= 0 && last >= ki - kKStages; --last)
                ptx::mbar_wait(K_FULL((int)(last % kKStages)), (uint32_t)((last / kKStages) & 1), p.wait_limit_ns,
                               &no_abort, p.err, 42);
        }
        __syncwarp();
    } else if (warp == kEpiWarps + 1) {
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16_f32(128, 128, false);
            const uint64_t dq = ptx::smem_desc_sw128(base + kScoreSQ, 16, 1024);
            TileWalk w;
            w.start(t0, n_qt, n_kt);
            int q_bh = -1, q_qt = -1, qidx = 0;
            int64_t ki = 0, li = 0;
            bool ok = true;
            for (int64_t t = t0; ok && t < t1; ++t, ++li, w.next(n_qt, n_kt)) {
                const int a = (int)(li & 1);
                // the epilogue has read this accumulator's previous tile
                if (li >= 2 &&
                    !(ok = ptx::mbar_wait(A_EMPTY(a), (uint32_t)(((li >> 1) - 1) & 1), p.wait_limit_ns, abort_flag, p.err, 43)))
                    break;
                if (tile_masked(p, w.qt, w.kt)) {
                    ptx::mbar_arrive(A_FULL(a));
                    continue;
                }
                if (w.bh != q_bh || w.qt != q_qt) {
                    if (!(ok = ptx::mbar_wait(Q_FULL, (uint32_t)(qidx & 1), p.wait_limit_ns, abort_flag, p.err, 44)))
                        break;
                    q_bh = w.bh;
                    q_qt = w.qt;
                    ++qidx;
                }
                const int s = (int)(ki % kKStages);
                if (!(ok = ptx::mbar_wait(K_FULL(s), (uint32_t)((ki / kKStages) & 1), p.wait_limit_ns, abort_flag, p.err,
                                          45)))
                    break;
                ptx::tc_fence_after();
                const uint64_t dk = ptx::smem_desc_sw128(base + kScoreSK + s * kTileBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
                    ptx::mma_ss(tmem + (uint32_t)(a * 128), dq + off, dk + off, idesc, kk > 0);
                }
                ptx::mma_commit(K_EMPTY(s));
                // the next tile with an MMA reads another Q: free this one once these MMAs end
                TileWalk y = w;
                y.next(n_qt, n_kt);
                int64_t nx = t + 1;
                while (nx < t1 && tile_masked(p, y.qt, y.kt)) {
                    ++nx;
                    y.next(n_qt, n_kt);
                }
                if (nx < t1 && (y.bh != w.bh || y.qt != w.qt))
                    ptx::mma_commit(Q_EMPTY);
                ptx::mma_commit(A_FULL(a));
                ++ki;
            }
            // every MMA issued has completed before TMEM is released
            ptx::mma_commit(DONE);
            volatile int no_abort = 0;
            ptx::mbar_wait(DONE, 0, p.wait_limit_ns, &no_abort, p.err, 46);
        }
        __syncwarp();
    } else {
        const int quarter = warp & 3, h = warp >> 2;
        const int row = quarter * 32 + lane;
        const float scale = 1.0f / sqrtf((float)D);
        const int64_t n_half = p.T / 64;
        TileWalk w;
        w.start(t0, n_qt, n_kt);
        bool ok = true;
        int64_t li = 0;
        for (int64_t t = t0; ok && t < t1; ++t, ++li, w.next(n_qt, n_kt)) {
            const int a = (int)(li & 1);
            const bool masked_tile = tile_masked(p, w.qt, w.kt);
            bool got = ptx::mbar_wait(A_FULL(a), (uint32_t)((li >> 1) & 1), p.wait_limit_ns, abort_flag, p.err, 47);
            got = __all_sync(0xffffffffu, got);
            ptx::tc_fence_after();
            const int64_t qpos = (int64_t)p.n * p.Tc + (int64_t)w.qt * 128 + row;
            const int64_t k_h = (int64_t)w.kt * 128 + 64 * h;  // first key of this half
            uint32_t s[64];
            if (got && !masked_tile) {
                ptx::tmem_ld64(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(a * 128 + 64 * h), s);
                ptx::tmem_ld_wait64(s);
            }
            // the accumulator is free for the tile after next
            ptx::tc_fence_before();
            if (got)
                ptx::mbar_arrive(A_EMPTY(a));
            // s / sqrt(d), -inf after the row's query position (causal)
            if (!got || masked_tile) {
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    s[i] = tc::f2u(-INFINITY);
            } else {
                const float2 sc2 = make_float2(scale, scale);
#pragma unroll
                for (int i = 0; i < 64; i += 2) {
                    const float2 r = __fmul2_rn(make_float2(u2f(s[i]), u2f(s[i + 1])), sc2);
                    s[i] = tc::f2u(r.x);
                    s[i + 1] = tc::f2u(r.y);
                }
                if (p.causal && qpos - k_h < 63) {
                    // keys k_h + i with i > lim are masked (all of them when lim < 0)
                    const int lim = (int)(qpos - k_h);
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        if (i > lim)
                            s[i] = tc::f2u(-INFINITY);
                }
            }
            // max and sum of e^{s - max} over the half, four chains each
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < 64; i += 8) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    m4[k] = tc::fmax3(m4[k], u2f(s[i + 2 * k]), u2f(s[i + 2 * k + 1]));
            }
            const float hm = tc::fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
            float hl = 0.f;
            if (hm > -INFINITY) {
                const float2 l2e = make_float2(kLog2e, kLog2e);
                const float2 nb = make_float2(-hm * kLog2e, -hm * kLog2e);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float2 e = __ffma2_rn(make_float2(u2f(s[2 * i]), u2f(s[2 * i + 1])), l2e, nb);
                    acc[i & 3] = __fadd2_rn(acc[i & 3], make_float2(ptx::ex2(e.x), ptx::ex2(e.y)));
                }
                const float2 a2 = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
                hl = a2.x + a2.y;
            }
            // this half's two chunks into the tile's staging slot: 128-byte rows,
            // 16-byte pieces swizzled by the row (the map's 128-byte swizzle)
            const uint32_t slot = base + kScoreOut + (uint32_t)(li & 1) * 4u * kChunkBytes;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const uint32_t line = slot + (uint32_t)(2 * h + c) * kChunkBytes + (uint32_t)row * 128u;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(line + ((uint32_t)(j ^ (row & 7)) << 4), u2f(s[32 * c + 4 * j]),
                                 u2f(s[32 * c + 4 * j + 1]), u2f(s[32 * c + 4 * j + 2]), u2f(s[32 * c + 4 * j + 3]));
            }
            ptx::fence_proxy_async_smem();
            // the other slot (the previous tile's stores) has been read
            if (threadIdx.x == 0)
                bulk_wait_group_read<0>();
            ok = epi_bar_and(got);  // every epilogue warp goes on, or none
            if (!ok)
                break;
            if (threadIdx.x == 0) {
                for (int c = 0; c < 4; ++c)
                    ptx::tma_store_3d(&tm_s, slot + (uint32_t)c * kChunkBytes, w.kt * 128 + 32 * c, w.qt * 128, w.bh);
                ptx::bulk_commit_group();
            }
            const int64_t si = ((int64_t)w.bh * p.Tc + (int64_t)w.qt * 128 + row) * n_half + 2 * w.kt + h;
            if (RSA_DCHECK(si >= 0 && si < p.BH * p.Tc * n_half, p.err, 0x61, si))
                p.stats[si] = make_float2(hm, hl);
        }
        if (threadIdx.x == 0)
            bulk_wait_group_read<0>();  // shared memory stays in use until the stores have read it
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kEpiWarps + 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 256);
    }
}

// Softmax over each full score row of chunk n (one warp per row): the row's
// max M and sum L from the per-tile statistics, then one pass over the row,
// P = e^{s-M}/L in bf16, and lse = M + ln L into the output lse.
__global__ void __launch_bounds__(256)
    softmax_rows_kernel(const float *__restrict__ S, const float2 *__restrict__ stats, __nv_bfloat16 *__restrict__ P,
                        float *__restrict__ lse, int64_t BH, int64_t Tc, int64_t T, int n, unsigned int *err)
{
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= BH * Tc)
        return;
    const int64_t n_st = T / 64;  // statistics entries of the row
    // the row's statistics, scores and probabilities lie inside their buffers
    if (!RSA_DCHECK(row < BH * Tc && (T & 3) == 0, err, 0x62, row))
        return;
    const float2 *st = stats + row * n_st;
    float M = -INFINITY;
    for (int64_t i = lane; i < n_st; i += 32)
        M = fmaxf(M, st[i].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    if (M > -INFINITY) {
        for (int64_t i = lane; i < n_st; i += 32) {
            const float2 x = st[i];
            if (x.x > -INFINITY)
                L += x.y * ptx::ex2((x.x - M) * kLog2e);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        L += __shfl_xor_sync(0xffffffffu, L, o);
    const bool empty = !(L > 0.f);
    const float inv = empty ? 0.f : 1.f / L;
    const float mM = empty ? 0.f : M * kLog2e;
    const float4 *src = reinterpret_cast<const float4 *>(S + row * T);
    uint2 *dst = reinterpret_cast<uint2 *>(P + row * T);
    for (int64_t i = lane; i < T / 4; i += 32) {
        const float4 x = src[i];
        float e[4] = {0.f, 0.f, 0.f, 0.f};
        if (!empty) {
            e[0] = ptx::ex2(fmaf(x.x, kLog2e, -mM)) * inv;
            e[1] = ptx::ex2(fmaf(x.y, kLog2e, -mM)) * inv;
            e[2] = ptx::ex2(fmaf(x.z, kLog2e, -mM)) * inv;
            e[3] = ptx::ex2(fmaf(x.w, kLog2e, -mM)) * inv;
        }
        __nv_bfloat162 a = __floats2bfloat162_rn(e[0], e[1]), b = __floats2bfloat162_rn(e[2], e[3]);
        dst[i] = make_uint2(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&b));
    }
    if (lane == 0) {
        const int64_t bh = row / Tc, r = row - bh * Tc;
        const int64_t li = bh * T + (int64_t)n * Tc + r;
        if (RSA_DCHECK(li >= 0 && li < BH * T, err, 0x63, li))
            lse[li] = empty ? -INFINITY : M + ptx::lg2(L) * 0.69314718055994531f;
    }
}

// O^n rows qt*128.. of head bh: sum over key chunks j in ring order (n - r) mod N
// of P^n_j V_j, 128 keys per step, kPvStages shared-memory stages.  The loader
// warp refills a stage as soon as the MMAs on it end, so every stage keeps
// loading while the MMA warp waits (one thread doing both held the next load
// back until the current tile had arrived).
constexpr int kPvStages = 3;
constexpr int kPvThreads = 192;  // warps 0-3 epilogue, warp 4 TMA loads, warp 5 MMA

__global__ void __launch_bounds__(kPvThreads)
    pv_kernel(const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ TwoPassParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *g = smem_raw + (base - raw);
    // stage s: P tile at base + s*2*kTileBytes, V tile right after it
    const uint32_t bars = base + 2 * kPvStages * kTileBytes;  // full[kPvStages], empty[kPvStages], done
    uint32_t *tslot = reinterpret_cast<uint32_t *>(g + 2 * kPvStages * kTileBytes + 16 * kPvStages + 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(g + 2 * kPvStages * kTileBytes + 16 * kPvStages + 20);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = blockIdx.x, bh = blockIdx.y;
    const int64_t tiles_per_chunk = p.Tc / 128;
    const int chunks = p.causal ? p.n + 1 : p.N;  // causal: chunks after n are all zero
    const int64_t nt = tiles_per_chunk * chunks;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * kPvStages + 1; ++i)
            ptx::mbar_init(bars + 8 * i, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 4) {
        ptx::tmem_alloc(ptx::smem_u32(tslot), 128);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tslot;
    auto FULL = [&](int s) { return bars + 8u * s; };
    auto EMPTY = [&](int s) { return bars + 8u * kPvStages + 8u * s; };
    const uint32_t DONE = bars + 16u * kPvStages;

    if (warp == 4) {
        if (lane == 0) {
            // key tile i: ring round r = i / tiles_per_chunk visits chunk (n - r) mod N
            auto key0 = [&](int64_t i) -> int64_t {
                const int64_t r = i / tiles_per_chunk;
                const int64_t j = ((p.n - r) % p.N + p.N) % p.N;
                return j * p.Tc + (i - r * tiles_per_chunk) * 128;
            };
            auto load = [&](int64_t i) {
                const int s = (int)(i % kPvStages);
                const uint32_t sp = base + s * 2 * kTileBytes, sv = sp + kTileBytes;
                const int64_t kk0 = key0(i);
                ptx::mbar_arrive_expect_tx(FULL(s), 2 * kTileBytes);
                for (int b = 0; b < 2; ++b) {
                    ptx::tma_load_3d(sp + b * kBoxBytes, &tm_p, FULL(s), (int)(kk0 + b * 64), qt * 128, (int)bh);
                    ptx::tma_load_3d(sv + b * kBoxBytes, &tm_v, FULL(s), b * 64, (int)kk0, (int)bh);
                }
            };
            // loads run as far ahead as the stages allow; the MMA warp frees them
            int64_t issued = 0;
            for (; issued < nt; ++issued) {
                const int s = (int)(issued % kPvStages);
                if (issued >= kPvStages &&
                    !ptx::mbar_wait(EMPTY(s), (uint32_t)((issued / kPvStages - 1) & 1), p.wait_limit_ns, abort_flag,
                                    p.err, 50))
                    break;
                load(issued);
            }
            // copies still in flight after an abort land before the CTA exits
            volatile int no_abort = 0;
            for (int64_t i = (issued > kPvStages ? issued - kPvStages : 0); i < issued; ++i)
                ptx::mbar_wait(FULL((int)(i % kPvStages)), (uint32_t)((i / kPvStages) & 1), p.wait_limit_ns, &no_abort,
                               p.err, 53);
        }
        __syncwarp();
    } else if (warp == 5) {
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16_f32(128, D, true);
            const uint64_t dp0 = ptx::smem_desc_sw128(base, 16, 1024);
            const uint64_t dv0 = ptx::smem_desc_sw128(base + kTileBytes, kBoxBytes, 1024);
            bool ok = true;
            for (int64_t i = 0; ok && i < nt; ++i) {
                const int s = (int)(i % kPvStages);
                if (!(ok = ptx::mbar_wait(FULL(s), (uint32_t)((i / kPvStages) & 1), p.wait_limit_ns, abort_flag, p.err,
                                          51)))
                    break;
                ptx::tc_fence_after();
                const uint64_t pa = dp0 + ((s * 2 * kTileBytes) >> 4);
                const uint64_t vb = dv0 + ((s * 2 * kTileBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
                    ptx::mma_ss(tmem, pa + off, vb + ((kk * 2048) >> 4), idesc, (i > 0 || kk > 0) ? 1u : 0u);
                }
                ptx::mma_commit(EMPTY(s));
            }
            ptx::mma_commit(DONE);
            volatile int no_abort = 0;
            ptx::mbar_wait(DONE, 0, p.wait_limit_ns, &no_abort, p.err, 52);
        }
        __syncwarp();
    } else {
        const int row = warp * 32 + lane;
        bool ok = ptx::mbar_wait(DONE, 0, p.wait_limit_ns, abort_flag, p.err, 54);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            ptx::tc_fence_after();
            const int64_t orow = (int64_t)bh * p.T + (int64_t)p.n * p.Tc + (int64_t)qt * 128 + row;
            const bool valid = (int64_t)qt * 128 + row < p.Tc &&
                               RSA_DCHECK(orow >= 0 && orow < p.BH * p.T, p.err, 0x64, orow);
            __nv_bfloat16 *dst = p.out + orow * D;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                if (nt > 0) {
                    ptx::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, o);
                    ptx::tmem_ld_wait(o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] = 0u;
                }
                if (valid) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        __nv_bfloat162 h[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            h[e] = __floats2bfloat162_rn(u2f(o[8 * i + 2 * e]), u2f(o[8 * i + 2 * e + 1]));
                        d4[i] = make_uint4(*reinterpret_cast<uint32_t *>(&h[0]), *reinterpret_cast<uint32_t *>(&h[1]),
                                           *reinterpret_cast<uint32_t *>(&h[2]), *reinterpret_cast<uint32_t *>(&h[3]));
                    }
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 128);
    }
}

}  // namespace

cudaError_t launch_two_pass(const void *q, const void *k, const void *v, int64_t BH, int64_t T, int N, int causal,
                            void *out, float *lse, float *S, void *P, void *stats, uint64_t wait_limit_ns,
                            unsigned int *err, cudaStream_t s)
{
    const int64_t Tc = T / N;
    CUtensorMap mq, mk, mv, mp, ms;
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)T, (uint64_t)BH};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)T * D * 2};
    const uint32_t box[3] = {64, 128, 1};
    const uint64_t pdims[3] = {(uint64_t)T, (uint64_t)Tc, (uint64_t)BH};
    const uint64_t pstrides[2] = {(uint64_t)T * 2, (uint64_t)Tc * T * 2};
    if (!make_bf16_map_sw128(&mq, q, 3, dims, strides, box) || !make_bf16_map_sw128(&mk, k, 3, dims, strides, box) ||
        !make_bf16_map_sw128(&mv, v, 3, dims, strides, box) || !make_bf16_map_sw128(&mp, P, 3, pdims, pstrides, box))
        return cudaErrorInvalidValue;
    // S [BH][Tc][T] fp32, written in 32-column x 128-row boxes (128 bytes wide)
    const uint64_t sstrides[2] = {(uint64_t)T * 4, (uint64_t)Tc * T * 4};
    const uint32_t sbox[3] = {32, 128, 1};
    if (!make_f32_map_sw128(&ms, S, 3, pdims, sstrides, sbox))
        return cudaErrorInvalidValue;
    const uint32_t smem_score = kScoreSmem,
                   smem_pv = 2 * kPvStages * kTileBytes + 16 * kPvStages + 32 + 1024;
    cudaError_t e = cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_score);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(pv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_pv);
    if (e != cudaSuccess)
        return e;
    const int64_t n_qt = (Tc + 127) / 128, n_kt = T / 128;
    if (BH > 65535 || n_kt > 65535)
        return cudaErrorInvalidConfiguration;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    // one CTA per SM (its shared memory allows no second one)
    const int64_t score_ctas = std::min<int64_t>(BH * n_qt * n_kt, std::max(sms, 1));
    for (int n = 0; n < N; ++n) {
        TwoPassParams p;
        p.BH = BH;
        p.T = T;
        p.Tc = Tc;
        p.n = n;
        p.N = N;
        p.causal = causal ? 1 : 0;
        p.S = S;
        p.stats = static_cast<float2 *>(stats);
        p.out = static_cast<__nv_bfloat16 *>(out);
        p.wait_limit_ns = wait_limit_ns;
        p.err = err;
        score_kernel<<<(unsigned)score_ctas, kScoreThreads, smem_score, s>>>(mq, mk, ms, p);
        const int64_t rows = BH * Tc;
        softmax_rows_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(
            S, static_cast<const float2 *>(stats), static_cast<__nv_bfloat16 *>(P), lse, BH, Tc, T, n, err);
        pv_kernel<<<dim3((unsigned)n_qt, (unsigned)BH), kPvThreads, smem_pv, s>>>(mp, mv, p);
        e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace rsa
