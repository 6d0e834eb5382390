// Online-softmax merge of partial attention results, HBM-bound.
//
// Page: "Sequence parallelism -- splitting the token dimension across GPUs"
// (llmdaily, day 58), section "But softmax seems to require all attention
// scores at once": with running maximum m and a new block's maximum m',
// m_new = max(m, m'), the old terms are rescaled by e^{m - m_new} and the new
// ones by e^{m' - m_new}.  The partials here are normalised (o, lse) pairs, for
// which that rule reads
//   M = max(a, b),  L = M + ln(e^{a-M} + e^{b-M}),
//   o = o_acc e^{a-L} + o_blk e^{b-L}             (a = lse_acc, b = lse_blk).
//
// Layout: d/8 threads per row, each owning 8 consecutive columns, so a warp
// reads whole rows with 16-byte vector accesses (two for fp32, one for bf16).
// Streaming cache hints keep the one-touch data from displacing L2.  Each
// (pair, head) segment is contiguous in memory, so indices need no division.
#include <cuda_bf16.h>

#include <cmath>

#include "rsa_internal.h"

namespace rsa {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 2;  // 8-column vectors per thread

__device__ __forceinline__ void load8_f32(const float *p, float *x)
{
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void load8_bf16(const __nv_bfloat16 *p, float *x)
{
    const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ void store8_f32(float *p, const float *x)
{
    __stcs(reinterpret_cast<float4 *>(p), make_float4(x[0], x[1], x[2], x[3]));
    __stcs(reinterpret_cast<float4 *>(p) + 1, make_float4(x[4], x[5], x[6], x[7]));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void store8_bf16(__nv_bfloat16 *p, const float *x)
{
    __stcs(reinterpret_cast<uint4 *>(p),
           make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7])));
}

// blockIdx.y walks the (pair, head) segments of the launch; inside a segment
// the Tc rows are contiguous both in the accumulator and in the partial, so a
// block covers kThreads * kUnroll consecutive 8-column vectors of one segment.
__global__ void __launch_bounds__(kThreads)
    merge_kernel(const __grid_constant__ MergeParams p, int log2_tpr)
{
    const int64_t BH = p.rows_per_pair / p.Tc;
    const int64_t nseg = (int64_t)p.npairs * BH;
    const int64_t nvec = p.Tc << log2_tpr;  // 8-column vectors per segment
    const int tpr_mask = (1 << log2_tpr) - 1;
    for (int64_t seg = blockIdx.y; seg < nseg; seg += gridDim.y) {
        const int pi = (int)(seg / BH);
        const int64_t bh = seg - (int64_t)pi * BH;
        const MergePair &mp = p.pairs[pi];
        const int64_t arow0 = bh * p.T + mp.acc_t0;  // first accumulator row of the segment
        const int64_t brow0 = bh * p.Tc;             // first partial row of the segment
        float a[kUnroll], b[kUnroll], x[kUnroll][8], y[kUnroll][8];
        int64_t vv[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            vv[u] = ((int64_t)blockIdx.x * kUnroll + u) * kThreads + threadIdx.x;
            if (vv[u] < nvec &&
                !(RSA_DCHECK(mp.acc_t0 + (vv[u] >> log2_tpr) < p.T, p.err, 0x51, arow0 + (vv[u] >> log2_tpr)) &&
                  RSA_DCHECK(brow0 + (vv[u] >> log2_tpr) < p.rows_per_pair, p.err, 0x52,
                             brow0 + (vv[u] >> log2_tpr))))
                vv[u] = nvec;  // out of range: skipped
            if (vv[u] < nvec) {
                const int64_t r = vv[u] >> log2_tpr;
                const int col = (int)(vv[u] & tpr_mask) * 8;
                a[u] = p.lse_acc[arow0 + r];
                b[u] = mp.lse_blk[brow0 + r];
                load8_f32(p.o_acc + (arow0 + r) * p.d + col, x[u]);
                if (p.blk_f32)
                    load8_f32(static_cast<const float *>(mp.o_blk) + (brow0 + r) * p.d + col, y[u]);
                else
                    load8_bf16(static_cast<const __nv_bfloat16 *>(mp.o_blk) + (brow0 + r) * p.d + col, y[u]);
            }
        }
        // Every thread of a row has read lse_acc before one of them overwrites it.
        __syncwarp();
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (vv[u] >= nvec)
                continue;
            const int64_t r = vv[u] >> log2_tpr;
            const int col = (int)(vv[u] & tpr_mask) * 8;
            const float M = fmaxf(a[u], b[u]);
            float L = -INFINITY;
            if (M > -INFINITY) {
                const float ea = __expf(a[u] - M);
                const float eb = __expf(b[u] - M);
                const float sum = ea + eb;
                const float inv = 1.f / sum;
                L = M + __logf(sum);
                const float wa = ea * inv, wb = eb * inv;
                // A side with lse = -inf is empty: its o is not read (it may
                // hold anything), rather than multiplied by a zero weight.
                const bool ua = a[u] > -INFINITY, ub = b[u] > -INFINITY;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    x[u][i] = (ua ? x[u][i] * wa : 0.f) + (ub ? y[u][i] * wb : 0.f);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    x[u][i] = 0.f;  // both sides empty: o = 0, lse = -inf
            }
            const int64_t arow = arow0 + r;
            if (mp.final_) {
                if (p.out_f32)
                    store8_f32(static_cast<float *>(p.out) + arow * p.d + col, x[u]);
                else
                    store8_bf16(static_cast<__nv_bfloat16 *>(p.out) + arow * p.d + col, x[u]);
                if (col == 0)
                    p.lse_out[arow] = L;
            } else {
                store8_f32(p.o_acc + arow * p.d + col, x[u]);
                if (col == 0)
                    p.lse_acc[arow] = L;
            }
        }
        __syncwarp();
    }
}

// Fold S partial results of the same rows (split-KV decode): one CTA per row.
// M = max_s lse_s, L = M + ln sum_s e^{lse_s - M}, o = sum_s o_s e^{lse_s - L};
// rows whose partials are all empty stay (0, -inf).  The eight warps share
// the splits (warp w takes s = w, w + 8, ...), so their loads are in flight
// together, and add their partial sums through shared memory.
constexpr int kSplitWarps = 8;

__device__ __forceinline__ float block_max(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kSplitWarps; ++w)
        r = fmaxf(r, red[w]);
    return r;
}

__device__ __forceinline__ float block_sum(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = 0.f;
#pragma unroll
    for (int w = 0; w < kSplitWarps; ++w)
        r += red[w];
    return r;
}

template <int PER>
__global__ void __launch_bounds__(32 * kSplitWarps)
    merge_splits_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part, int S, int64_t rows,
                        void *out, int out_f32, float *lse)
{
    constexpr int D = PER * 32;
    __shared__ float red[kSplitWarps];
    __shared__ float part[kSplitWarps][D];
    const int64_t row = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float m = -INFINITY;
    for (int s = threadIdx.x; s < S; s += 32 * kSplitWarps)
        m = fmaxf(m, lse_part[(int64_t)s * rows + row]);
    const float M = block_max(m, red);
    float acc[PER];
#pragma unroll
    for (int c = 0; c < PER; ++c)
        acc[c] = 0.f;
    float L = -INFINITY;
    if (M > -INFINITY) {
        float sum = 0.f;
        for (int s = threadIdx.x; s < S; s += 32 * kSplitWarps)
            sum += expf(lse_part[(int64_t)s * rows + row] - M);
        L = M + logf(block_sum(sum, red));
        // an empty split has lse = -inf (weight 0) and o = 0
#pragma unroll 4
        for (int s = warp; s < S; s += kSplitWarps) {
            const float w = expf(lse_part[(int64_t)s * rows + row] - L);
            const float *src = o_part + ((int64_t)s * rows + row) * D + lane * PER;
#pragma unroll
            for (int c = 0; c < PER; ++c)
                acc[c] = fmaf(w, src[c], acc[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < PER; ++c)
        part[warp][lane * PER + c] = acc[c];
    __syncthreads();
    if (warp != 0)
        return;
#pragma unroll
    for (int c = 0; c < PER; ++c) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kSplitWarps; ++w)
            v += part[w][lane * PER + c];
        acc[c] = v;
    }
    if (out_f32) {
        float *dst = static_cast<float *>(out) + row * D + lane * PER;
#pragma unroll
        for (int c = 0; c < PER; ++c)
            dst[c] = acc[c];
    } else {
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(out) + row * D + lane * PER;
#pragma unroll
        for (int c = 0; c < PER; c += 2)
            *reinterpret_cast<uint32_t *>(dst + c) = pack2(acc[c], acc[c + 1]);
    }
    if (lane == 0)
        lse[row] = L;
}

}  // namespace

cudaError_t launch_merge_splits(const float *o_part, const float *lse_part, int S, int64_t rows, int d, void *out,
                                int out_f32, float *lse, cudaStream_t s)
{
    if (rows <= 0 || S <= 0)
        return cudaSuccess;
    if (rows > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    if (d == 128)
        merge_splits_kernel<4><<<(unsigned)rows, 32 * kSplitWarps, 0, s>>>(o_part, lse_part, S, rows, out, out_f32, lse);
    else if (d == 64)
        merge_splits_kernel<2><<<(unsigned)rows, 32 * kSplitWarps, 0, s>>>(o_part, lse_part, S, rows, out, out_f32, lse);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_merge(const MergeParams &p, cudaStream_t s)
{
    if (p.npairs <= 0 || p.rows_per_pair <= 0 || p.Tc <= 0)
        return cudaSuccess;
    if (p.d != 64 && p.d != 128)
        return cudaErrorInvalidValue;
    const int log2_tpr = p.d == 128 ? 4 : 3;
    const int64_t nvec = p.Tc << log2_tpr;
    const int64_t per_block = (int64_t)kThreads * kUnroll;
    const int64_t bx = (nvec + per_block - 1) / per_block;
    const int64_t nseg = (int64_t)p.npairs * (p.rows_per_pair / p.Tc);
    if (bx > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)bx, (unsigned)(nseg < 65535 ? nseg : 65535));
    merge_kernel<<<grid, kThreads, 0, s>>>(p, log2_tpr);
    return cudaGetLastError();
}

}  // namespace rsa
