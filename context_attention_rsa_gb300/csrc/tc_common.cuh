// Register-level helpers shared by the tensor-core kernels: bit casts, bf16
// packing, three-input max and the named barrier of the softmax threads of
// the block-attention kernels (one-SM and two-SM).
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace rsa {
namespace tc {

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

// Named barrier 1 over the NT softmax threads (the first NT / 32 warps).
template <int NT = 256>
__device__ __forceinline__ void softmax_bar_sync()
{
    asm volatile("barrier.cta.sync 1, %0;" ::"n"(NT) : "memory");
}

// The same barrier, returning whether `v` holds in every softmax thread, so
// that a decision to give up is taken by all of them together.
template <int NT = 256>
__device__ __forceinline__ bool softmax_bar_and(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "barrier.cta.red.and.pred po, 1, %2, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(NT)
        : "memory");
    return r != 0;
}

// 16-byte shared-memory load (a staged row piece).
__device__ __forceinline__ float4 ld_shared_v4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

}  // namespace tc
}  // namespace rsa
