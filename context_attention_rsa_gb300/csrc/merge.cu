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
// Streaming cache hints keep the one-touch data from displacing L2.
// Grid-stride loop over rows of all pairs in the launch.
#include <cuda_bf16.h>

#include <cmath>

#include "rsa_internal.h"

namespace rsa {
namespace {

constexpr int kThreads = 256;

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

__global__ void __launch_bounds__(kThreads)
    merge_kernel(const __grid_constant__ MergeParams p)
{
    const int tpr = p.d >> 3;  // threads per row
    const int64_t total = (int64_t)p.npairs * p.rows_per_pair * tpr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += stride) {
        const int64_t row = g / tpr;
        const int col = (int)(g - row * tpr) * 8;
        const int pi = (int)(row / p.rows_per_pair);
        const int64_t rr = row - (int64_t)pi * p.rows_per_pair;
        const int64_t bh = rr / p.Tc;
        const int64_t t = rr - bh * p.Tc;
        const MergePair &mp = p.pairs[pi];
        const int64_t arow = bh * p.T + mp.acc_t0 + t;

        const float a = p.lse_acc[arow];
        const float b = mp.lse_blk[rr];
        const float M = fmaxf(a, b);
        float wa = 0.f, wb = 0.f, L = -INFINITY;
        if (M > -INFINITY) {
            const float ea = __expf(a - M);
            const float eb = __expf(b - M);
            const float s = ea + eb;
            const float inv = 1.f / s;
            L = M + __logf(s);
            wa = ea * inv;
            wb = eb * inv;
        }
        float x[8], y[8];
        load8_f32(p.o_acc + arow * p.d + col, x);
        if (p.blk_f32)
            load8_f32(static_cast<const float *>(mp.o_blk) + rr * p.d + col, y);
        else
            load8_bf16(static_cast<const __nv_bfloat16 *>(mp.o_blk) + rr * p.d + col, y);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            x[i] = x[i] * wa + y[i] * wb;
        // Every thread of the row has read lse_acc before one of them overwrites it.
        __syncwarp(__activemask());
        if (mp.final_) {
            if (p.out_f32)
                store8_f32(static_cast<float *>(p.out) + arow * p.d + col, x);
            else
                store8_bf16(static_cast<__nv_bfloat16 *>(p.out) + arow * p.d + col, x);
            if (col == 0)
                p.lse_out[arow] = L;
        } else {
            store8_f32(p.o_acc + arow * p.d + col, x);
            if (col == 0)
                p.lse_acc[arow] = L;
        }
    }
}

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, cudaStream_t s)
{
    const int64_t threads = (int64_t)p.npairs * p.rows_per_pair * (p.d >> 3);
    if (threads <= 0)
        return cudaSuccess;
    static int sms = sm_count();
    int64_t blocks = (threads + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)sms * (2048 / kThreads);
    if (blocks > cap)
        blocks = cap;
    merge_kernel<<<(unsigned)blocks, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace rsa
