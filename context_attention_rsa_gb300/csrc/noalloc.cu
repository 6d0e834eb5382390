// rsa_ring_attn_fwd_noalloc: the whole ring with the library's own scratch.
//
// rsa_ring_attn_fwd needs a caller-provided device workspace (the fp32
// accumulator and one round's partials).  Some callers cannot allocate device
// memory when they need attention: code whose device memory is owned by
// another allocator that must not be bypassed, code running where a
// cudaMalloc (and the device-wide synchronisation it may imply) is not
// allowed or would stall a latency-critical stream.  For them this entry
// point uses a fixed scratch array compiled into the library instead.
//
// The scratch is a file-scope __device__ array of kScratchBytes.  It is
// reserved on a device when the library's device code is loaded into that
// device's context -- at the latest on this entry point's first call there,
// and on every initialised device under eager module loading -- and stays
// until the process exits.  In host code the array's name is only a host-side
// stand-in, so its device address is looked up with cudaGetSymbolAddress on
// the first call in each CUDA context (with that context current) and cached
// under the context's unique id; make that first call before any stream
// capture.
//
// Every call shares the one array and leaves its contents behind.  Nothing in
// it needs to start at zero: the ring writes each accumulator row and each
// partial before reading it.  Calls that overlap on the GPU (different
// streams, or different host threads without ordering between them) race on
// the array and corrupt each other's results.
#include <cstdio>

#include "rsa_internal.h"

namespace {

constexpr size_t kScratchBytes = 64ull << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_ring_scratch[kScratchBytes];

}  // namespace

extern "C" rsa_status rsa_ring_attn_fwd_noalloc(const void *q, const void *k, const void *v, rsa_dtype dt, int B,
                                                int H, int64_t T, int d, int N, int causal, void *out, float *lse,
                                                rsa_stream_t stream)
{
    size_t need = 0;
    rsa_status st = rsa_ring_attn_workspace_size(dt, B, H, T, d, N, causal, &need);
    if (st != RSA_OK)
        return st;
    if (need > kScratchBytes)
        return rsa::fail(RSA_ERR_INVALID_ARG,
                         "rsa_ring_attn_fwd_noalloc: this shape needs %zu bytes of scratch, the built-in "
                         "scratch holds %zu; use rsa_ring_attn_fwd with a caller workspace",
                         need, kScratchBytes);
    // The array's name is only a host-side stand-in here; the kernels need its
    // device address in the current context.
    void *scratch = nullptr;
    st = rsa::symbol_address(reinterpret_cast<const void *>(g_ring_scratch), &scratch);
    if (st != RSA_OK)
        return st;
    return rsa_ring_attn_fwd(q, k, v, dt, B, H, T, d, N, causal, out, lse, scratch, kScratchBytes, stream);
}
