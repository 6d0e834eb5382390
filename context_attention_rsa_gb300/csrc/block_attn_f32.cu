// Block attention for fp32 inputs on the CUDA cores (SIMT).  fp32 results
// must stay within 1e-4 of the fp64 definition, which rules out the tf32
// tensor-core path, so this kernel is the correctness path for fp32; it makes
// no throughput claim.
//
// Pages: "Sequence parallelism -- splitting the token dimension across GPUs"
// (llmdaily, day 58): the attention equation of "Attention wants keys and
// values from other tokens"; the running max / normaliser / accumulator and
// the e^{m - m_new} rescale of "But softmax seems to require all attention
// scores at once", applied per block of 32 keys; the causal mask of "Causal
// attention gives us another optimization".
//
// One warp owns one query row.  For each block of 32 keys, lane i scores key
// i (a full dot product against the row's query, held in shared memory);
// the block max and sum are warp-shuffle reductions; lane i then owns output
// columns i, i+32, ... and accumulates p_k v_k for the 32 keys, p_k broadcast
// by shuffle.
#include <cmath>

#include "rsa_internal.h"

namespace rsa {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
    block_attn_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                          const float *__restrict__ v, const __grid_constant__ BlockParams p)
{
    constexpr int PER = D / 32;
    __shared__ float qs[kWarps][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kWarps + warp;
    const int bh = blockIdx.y;
    const int sp = blockIdx.z / p.npairs;  // key split (decode), 0 otherwise
    const PairDesc &pr = p.pairs[blockIdx.z - sp * p.npairs];
    if (r >= p.q_len)
        return;  // whole warp leaves together
    const int64_t qpos = pr.q_off + r;
    const int64_t head = (int64_t)bh * p.T;
    const int64_t kv_off = pr.kv_off + (int64_t)sp * p.kv_split;   // global position (mask)
    const int64_t kv_row = pr.kv_row0 + (int64_t)sp * p.kv_split;  // row in the K/V tensors
    const int64_t kv_len = p.kv_split > 0 ? min(p.kv_split, p.kv_len - (int64_t)sp * p.kv_split) : p.kv_len;
    const float scale = 1.0f / sqrtf((float)D);
    if (!RSA_DCHECK(pr.q_row0 + r < p.q_T, p.err, 0x41, pr.q_row0 + r))
        return;
    const float *qrow = q + ((int64_t)bh * p.q_T + pr.q_row0 + r) * D;
#pragma unroll
    for (int i = 0; i < PER; ++i)
        qs[warp][lane + 32 * i] = qrow[lane + 32 * i];
    __syncwarp();

    int64_t kv_end = kv_len;
    if (p.causal)
        kv_end = min(kv_end, qpos - kv_off + 1);
    float m = -INFINITY, l = 0.f;
    float o[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i)
        o[i] = 0.f;

    for (int64_t j0 = 0; j0 < kv_end; j0 += 32) {
        const int64_t j = j0 + lane;
        float s = -INFINITY;
        if (j < kv_end && RSA_DCHECK(kv_row + j < p.T, p.err, 0x42, kv_row + j)) {
            const float4 *kr = reinterpret_cast<const float4 *>(k + (head + kv_row + j) * D);
            const float4 *qv = reinterpret_cast<const float4 *>(qs[warp]);
            float dot = 0.f;
#pragma unroll 8
            for (int x = 0; x < D / 4; ++x) {
                const float4 a = qv[x], b = kr[x];
                dot = fmaf(a.x, b.x, dot);
                dot = fmaf(a.y, b.y, dot);
                dot = fmaf(a.z, b.z, dot);
                dot = fmaf(a.w, b.w, dot);
            }
            s = dot * scale;
        }
        const float m_new = fmaxf(m, warp_max(s));  // finite: lane 0 always has a key here
        const float alpha = expf(m - m_new);       // 0 on the first block (m = -inf)
        const float pj = (j < kv_end) ? expf(s - m_new) : 0.f;
        l = l * alpha + warp_sum(pj);
#pragma unroll
        for (int i = 0; i < PER; ++i)
            o[i] *= alpha;
        int nk = (int)min((int64_t)32, kv_end - j0);
        if (!RSA_DCHECK(kv_row + j0 + nk <= p.T, p.err, 0x43, kv_row + j0 + nk - 1))
            nk = 0;
        const float *vb = v + (head + kv_row + j0) * D;
        for (int kk = 0; kk < nk; ++kk) {
            const float pk = __shfl_sync(0xffffffffu, pj, kk);
#pragma unroll
            for (int i = 0; i < PER; ++i)
                o[i] = fmaf(pk, vb[(int64_t)kk * D + lane + 32 * i], o[i]);
        }
        m = m_new;
    }

    const int64_t orow = (int64_t)bh * pr.out_T + pr.out_t0 + r + (int64_t)sp * pr.split_stride;
    if (!RSA_DCHECK(orow >= 0 && orow < pr.out_rows, p.err, 0x44, orow))
        return;
    const bool empty = !(l > 0.f);
    const float lse_b = empty ? -INFINITY : m + logf(l);
    float wa = 0.f, wb = empty ? 0.f : 1.f / l, lse_out = lse_b;
    bool use_acc = false;  // an accumulator row with lse = -inf is empty: not read
    if (pr.mode != kStore) {
        // fold into the running (acc, lse): M = max(a, b), L = M + ln(e^{a-M} + e^{b-M})
        const float a = pr.lse[orow];
        use_acc = a > -INFINITY;
        const float M = fmaxf(a, lse_b);
        if (M > -INFINITY) {
            const float ea = expf(a - M), eb = expf(lse_b - M);
            lse_out = M + logf(ea + eb);
            wa = ea / (ea + eb);
            wb = empty ? 0.f : eb / (ea + eb) / l;
        } else {
            lse_out = -INFINITY;
            wb = 0.f;
        }
    }
    float *out = static_cast<float *>(pr.out) + orow * D;
    const float *acc = pr.acc + orow * D;
#pragma unroll
    for (int i = 0; i < PER; ++i)
        out[lane + 32 * i] = use_acc ? fmaf(o[i], wb, acc[lane + 32 * i] * wa) : o[i] * wb;
    __syncwarp();  // every lane has read lse[orow] before lane 0 replaces it
    if (lane == 0)
        pr.lse[orow] = lse_out;
}

}  // namespace

cudaError_t launch_block_attn_f32(const float *q, const float *k, const float *v, const BlockParams &p,
                                  cudaStream_t s)
{
    const int64_t bx = (p.q_len + kWarps - 1) / kWarps;
    const int64_t BH = (int64_t)p.B * p.H;
    if (bx <= 0 || BH <= 0 || p.npairs <= 0)
        return cudaSuccess;
    const int64_t bz = (int64_t)p.npairs * p.n_split;
    if (bx > 0x7fffffffLL || BH > 65535 || bz > 65535)
        return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)bx, (unsigned)BH, (unsigned)bz);
    if (p.d == 64)
        block_attn_f32_kernel<64><<<grid, kWarps * 32, 0, s>>>(q, k, v, p);
    else if (p.d == 128)
        block_attn_f32_kernel<128><<<grid, kWarps * 32, 0, s>>>(q, k, v, p);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace rsa
