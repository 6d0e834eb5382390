// C ABI of librsa and the single-GPU ring scheduler.
//
// Pages: "Sequence parallelism -- splitting the token dimension across GPUs"
// (llmdaily, day 58): contiguous chunks of T/N tokens ("Split tokens across
// four GPUs"); the ring in which GPU i sees KV block (i - r) mod N in round
// r+1 ("A better mental model: move blocks past the queries", the round
// table); chunk i never needs a later chunk under the causal mask ("Causal
// attention gives us another optimization"); partials folded with the
// running-statistics rescale ("But softmax seems to require all attention
// scores at once").
//
// Here every chunk is resident on the one GPU, so "sending a KV block to the
// next GPU" becomes pointing the next round's pairs at another chunk's base
// offset: no copy, no collective.  One block-attention launch covers all pairs
// of a round.  By default its epilogue folds each pair into the fp32
// accumulator; with RSA_RING_SEPARATE_MERGE the round's partials go to the
// workspace in fp32 (a bf16 partial would add a second rounding on top of the
// final bf16 output) and one merge launch folds them in.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "rsa_internal.h"

#define RSA_TRY(x)                     \
    do {                               \
        rsa_status st_ = (x);          \
        if (st_ != RSA_OK)             \
            return st_;                \
    } while (0)

namespace rsa {

static thread_local char g_last_error[512] = "";

rsa_status fail(rsa_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

struct CtxFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

// Driver calls reached through the runtime's entry-point query, so the
// library does not link the driver library directly.
const CtxFns &ctx_fns()
{
    static CtxFns f;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    return f;
}

// Unique id of the calling thread's current context; *have = false when no
// context is current yet.
rsa_status current_context_id(unsigned long long *id, bool *have)
{
    const CtxFns &f = ctx_fns();
    if (!f.get_current || !f.get_id)
        return fail(RSA_ERR_CUDA, "the CUDA driver lacks cuCtxGetCurrent/cuCtxGetId");
    CUcontext ctx = nullptr;
    if (f.get_current(&ctx) != CUDA_SUCCESS)
        return fail(RSA_ERR_CUDA, "cuCtxGetCurrent failed");
    *have = ctx != nullptr;
    if (ctx && f.get_id(ctx, id) != CUDA_SUCCESS)
        return fail(RSA_ERR_CUDA, "cuCtxGetId failed");
    return RSA_OK;
}

}  // namespace

rsa_status symbol_address(const void *symbol, void **out)
{
    struct Entry {
        const void *sym;
        unsigned long long ctx;
        void *addr;
    };
    constexpr int kEntries = 128;
    static Entry cache[kEntries] = {};
    static int next = 0;
    static std::mutex mu;
    unsigned long long id = 0;
    bool have = false;
    rsa_status st = current_context_id(&id, &have);
    if (st != RSA_OK)
        return st;
    if (have) {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry &e : cache)
            if (e.sym == symbol && e.addr && e.ctx == id) {
                *out = e.addr;
                return RSA_OK;
            }
    }
    // Not yet looked up in this context (this also creates the device's
    // primary context when none is current).
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, symbol);
    if (e != cudaSuccess || !p)
        return fail(RSA_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    st = current_context_id(&id, &have);
    if (st != RSA_OK)
        return st;
    if (!have)
        return fail(RSA_ERR_CUDA, "no current CUDA context after the symbol lookup");
    std::lock_guard<std::mutex> lock(mu);
    cache[next] = Entry{symbol, id, p};
    next = (next + 1) % kEntries;
    *out = p;
    return RSA_OK;
}

}  // namespace rsa

using namespace rsa;

namespace {

__device__ DeviceError g_device_error;

std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_tc_kernel{0};

// Host-side failure injection (off: -1).  When it reaches zero, the launch
// wrapper reports a launch failure instead of launching, then disarms.
std::atomic<int> g_inject_countdown{-1};

// True if this launch is to fail (and the failure has been recorded).
bool injected_failure(const char *what, rsa_status *st)
{
    int c = g_inject_countdown.load();
    while (c >= 0) {
        if (g_inject_countdown.compare_exchange_weak(c, c - 1)) {
            if (c > 0)
                return false;
            *st = fail(RSA_ERR_CUDA, "%s: injected launch failure (rsa_debug_inject_launch_failure)", what);
            return true;
        }
    }
    return false;
}

constexpr int kMaxDevices = 64;

rsa_status device_error_word(unsigned int **out)
{
    void *p = nullptr;
    RSA_TRY(symbol_address(reinterpret_cast<const void *>(&g_device_error), &p));
    *out = static_cast<unsigned int *>(p);
    return RSA_OK;
}

// The bf16 kernels are built for sm_103a only.
rsa_status check_device_for(rsa_dtype dt)
{
    if (dt != RSA_BF16)
        return RSA_OK;
    static std::mutex mu;
    static int cc[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(RSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(RSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (!cc[dev]) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return fail(RSA_ERR_CUDA, "cannot query compute capability of device %d", dev);
        cc[dev] = major * 10 + minor;
    }
    if (cc[dev] != 103)
        return fail(RSA_ERR_UNSUPPORTED, "bf16 tensor-core path needs sm_103 (device is sm_%d)", cc[dev]);
    return RSA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

rsa_status check_shape(rsa_dtype dt, int B, int H, int64_t T, int d)
{
    if (dt != RSA_F32 && dt != RSA_BF16)
        return fail(RSA_ERR_INVALID_ARG, "dtype %d is not RSA_F32 or RSA_BF16", (int)dt);
    if (B < 1 || H < 1 || T < 1)
        return fail(RSA_ERR_INVALID_ARG, "B, H, T must be >= 1 (got %d, %d, %lld)", B, H, (long long)T);
    if (d != 64 && d != 128)
        return fail(RSA_ERR_UNSUPPORTED, "head dimension d=%d not supported (64 or 128)", d);
    if (T > 0x7fffffffLL)
        return fail(RSA_ERR_UNSUPPORTED, "T=%lld exceeds 2^31-1", (long long)T);
    const int64_t BH = (int64_t)B * H;
    if (BH > 0x7fffffffLL || (dt == RSA_F32 && BH > 65535))
        return fail(RSA_ERR_UNSUPPORTED, "B*H=%lld too large", (long long)BH);
    return RSA_OK;
}

rsa_status check_ptr(const void *p, const char *name)
{
    if (!p)
        return fail(RSA_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned16(p))
        return fail(RSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
    return RSA_OK;
}

int round_pairs(int N, int causal, int r, int *qi, int *kj)
{
    int n = 0;
    for (int i = 0; i < N; ++i) {
        const int j = ((i - r) % N + N) % N;
        if (causal && j > i)
            continue;
        if (qi)
            qi[n] = i;
        if (kj)
            kj[n] = j;
        ++n;
    }
    return n;
}

int visits(int N, int causal, int i) { return causal ? i + 1 : N; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
    size_t acc, oblk, lblk, total;
    int maxp;
};

WsLayout ws_layout(rsa_dtype dt, int B, int H, int64_t T, int d, int N, int causal, bool fused)
{
    WsLayout w{};
    const size_t BH = (size_t)B * H;
    const size_t Tc = (size_t)(T / N);
    const size_t esz = 4;  // partials stay fp32 whatever the input dtype
    (void)dt;
    int maxp = 0;
    for (int r = 1; r < N; ++r) {
        const int np = round_pairs(N, causal, r, nullptr, nullptr);
        maxp = np > maxp ? np : maxp;
    }
    if (fused)
        maxp = 0;  // partials go straight into the accumulator
    w.maxp = maxp;
    w.acc = N > 1 ? align256(BH * (size_t)T * d * 4) : 0;
    w.oblk = align256((size_t)maxp * BH * Tc * d * esz);
    w.lblk = align256((size_t)maxp * BH * Tc * 4);
    w.total = w.acc + w.oblk + w.lblk;
    return w;
}

int launch_count(int N, int causal, bool fused)
{
    int n = (N + kMaxPairsPerLaunch - 1) / kMaxPairsPerLaunch;
    for (int r = 1; r < N; ++r) {
        const int np = round_pairs(N, causal, r, nullptr, nullptr);
        n += (fused ? 1 : 2) * ((np + kMaxPairsPerLaunch - 1) / kMaxPairsPerLaunch);
    }
    return n;
}

struct Recorder {
    rsa_event_t *start = nullptr, *stop = nullptr;
    int *kind = nullptr;
    int n = 0;
};

rsa_status record(rsa_event_t ev, cudaStream_t s)
{
    cudaError_t e = cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev), s);
    if (e != cudaSuccess)
        return fail(RSA_ERR_CUDA, "cudaEventRecord: %s", cudaGetErrorString(e));
    return RSA_OK;
}

rsa_status launch_block(const void *q, const void *k, const void *v, rsa_dtype dt, const BlockParams &p,
                        cudaStream_t s, Recorder *rec)
{
    rsa_status inj;
    if (injected_failure("block attention launch", &inj))
        return inj;
    if (rec)
        RSA_TRY(record(rec->start[rec->n], s));
    cudaError_t e = dt == RSA_BF16
                        ? launch_block_attn_bf16(q, k, v, p, s)
                        : launch_block_attn_f32(static_cast<const float *>(q), static_cast<const float *>(k),
                                                static_cast<const float *>(v), p, s);
    if (e != cudaSuccess)
        return fail(RSA_ERR_CUDA, "block attention launch: %s", cudaGetErrorString(e));
    if (rec) {
        RSA_TRY(record(rec->stop[rec->n], s));
        rec->kind[rec->n++] = 0;
    }
    return RSA_OK;
}

rsa_status launch_merge_rec(const MergeParams &p, cudaStream_t s, Recorder *rec)
{
    rsa_status inj;
    if (injected_failure("merge launch", &inj))
        return inj;
    if (rec)
        RSA_TRY(record(rec->start[rec->n], s));
    cudaError_t e = launch_merge(p, s);
    if (e != cudaSuccess)
        return fail(RSA_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
    if (rec) {
        RSA_TRY(record(rec->stop[rec->n], s));
        rec->kind[rec->n++] = 1;
    }
    return RSA_OK;
}

BlockParams base_params(rsa_dtype dt, int B, int H, int64_t T, int d, int causal, int64_t q_len,
                        int64_t kv_len, unsigned int *err)
{
    BlockParams p;
    memset(&p, 0, sizeof p);
    p.B = B;
    p.H = H;
    p.T = T;
    p.d = d;
    p.causal = causal ? 1 : 0;
    p.q_len = q_len;
    p.kv_len = kv_len;
    p.q_T = T;
    p.n_split = 1;
    p.n_qgroups = (int)((q_len + kBf16RowsPerCta - 1) / kBf16RowsPerCta);
    p.wait_limit_ns = g_wait_limit_ns.load();
    p.tc_kernel = g_tc_kernel.load();
    p.err = err;
    (void)dt;
    return p;
}

rsa_status validate_ring(const void *q, const void *k, const void *v, rsa_dtype dt, int B, int H, int64_t T,
                         int d, int N, void *out, float *lse, void *ws, size_t ws_bytes, int causal,
                         bool fused, WsLayout *lay)
{
    RSA_TRY(check_shape(dt, B, H, T, d));
    RSA_TRY(check_ptr(q, "q"));
    RSA_TRY(check_ptr(k, "k"));
    RSA_TRY(check_ptr(v, "v"));
    RSA_TRY(check_ptr(out, "out"));
    RSA_TRY(check_ptr(lse, "lse"));
    if (N < 1 || N > T || T % N != 0)
        return fail(RSA_ERR_INVALID_ARG, "N=%d must be >= 1 and divide T=%lld", N, (long long)T);
    if (N > 1024)
        return fail(RSA_ERR_UNSUPPORTED, "N=%d exceeds 1024 chunks", N);
    *lay = ws_layout(dt, B, H, T, d, N, causal, fused);
    if (lay->total > 0) {
        RSA_TRY(check_ptr(ws, "workspace"));
        if (ws_bytes < lay->total)
            return fail(RSA_ERR_INVALID_ARG, "workspace holds %zu bytes, %zu needed", ws_bytes, lay->total);
    }
    return check_device_for(dt);
}

rsa_status ring_run(const void *q, const void *k, const void *v, rsa_dtype dt, int B, int H, int64_t T, int d,
                    int N, int causal, void *out, float *lse, void *ws, const WsLayout &lay, bool fused,
                    cudaStream_t s, Recorder *rec)
{
    unsigned int *err = nullptr;
    RSA_TRY(device_error_word(&err));
    causal = causal ? 1 : 0;
    const int64_t Tc = T / N;
    const int64_t BH = (int64_t)B * H;
    const size_t esz = 4;  // fp32 partials
    char *wsb = static_cast<char *>(ws);
    float *o_acc = lay.acc ? reinterpret_cast<float *>(wsb) : nullptr;
    char *oblk = wsb + lay.acc;
    float *lblk = reinterpret_cast<float *>(wsb + lay.acc + lay.oblk);

    // Round 0: the diagonal pairs (i, i).
    for (int g0 = 0; g0 < N; g0 += kMaxPairsPerLaunch) {
        BlockParams p = base_params(dt, B, H, T, d, causal, Tc, Tc, err);
        for (int i = g0; i < N && p.npairs < kMaxPairsPerLaunch; ++i) {
            PairDesc &pd = p.pairs[p.npairs++];
            const bool once = visits(N, causal, i) == 1;
            pd.q_off = i * Tc;
            pd.q_row0 = pd.q_off;
            pd.kv_off = i * Tc;
            pd.kv_row0 = pd.kv_off;
            pd.out = once ? out : static_cast<void *>(o_acc);
            pd.lse = lse;
            pd.out_T = T;
            pd.out_t0 = i * Tc;
            pd.out_rows = BH * T;
            pd.out_f32 = once ? (dt == RSA_F32) : 1;
        }
        RSA_TRY(launch_block(q, k, v, dt, p, s, rec));
    }
    // Rounds 1..N-1: partials into the workspace, then merge -- or, fused,
    // each pair's epilogue folds its result into the accumulator directly.
    int qi[1024], kj[1024];
    for (int r = 1; r < N; ++r) {
        const int np = round_pairs(N, causal, r, qi, kj);
        if (fused) {
            for (int g0 = 0; g0 < np; g0 += kMaxPairsPerLaunch) {
                BlockParams p = base_params(dt, B, H, T, d, causal, Tc, Tc, err);
                for (int x = g0; x < np && p.npairs < kMaxPairsPerLaunch; ++x) {
                    const int i = qi[x], j = kj[x];
                    const bool last = r == visits(N, causal, i) - 1;
                    PairDesc &pd = p.pairs[p.npairs++];
                    pd.q_off = i * Tc;
                    pd.q_row0 = pd.q_off;
                    pd.kv_off = j * Tc;
                    pd.kv_row0 = pd.kv_off;
                    pd.out = last ? out : static_cast<void *>(o_acc);
                    pd.lse = lse;
                    pd.out_T = T;
                    pd.out_t0 = i * Tc;
                    pd.out_rows = BH * T;
                    pd.out_f32 = last ? (dt == RSA_F32) : 1;
                    pd.mode = last ? kMergeFinal : kMergeAcc;
                    pd.acc = o_acc;
                }
                RSA_TRY(launch_block(q, k, v, dt, p, s, rec));
            }
            continue;
        }
        for (int g0 = 0; g0 < np; g0 += kMaxPairsPerLaunch) {
            const int gn = np - g0 < kMaxPairsPerLaunch ? np - g0 : kMaxPairsPerLaunch;
            BlockParams p = base_params(dt, B, H, T, d, causal, Tc, Tc, err);
            MergeParams m;
            memset(&m, 0, sizeof m);
            m.rows_per_pair = BH * Tc;
            m.Tc = Tc;
            m.T = T;
            m.d = d;
            m.blk_f32 = 1;
            m.out_f32 = dt == RSA_F32;
            m.o_acc = o_acc;
            m.lse_acc = lse;
            m.out = out;
            m.lse_out = lse;
            m.err = err;
            for (int x = 0; x < gn; ++x) {
                const int slot = g0 + x;
                const int i = qi[slot], j = kj[slot];
                void *ob = oblk + (size_t)slot * (size_t)BH * Tc * d * esz;
                float *lb = lblk + (size_t)slot * (size_t)BH * Tc;
                PairDesc &pd = p.pairs[p.npairs++];
                pd.q_off = i * Tc;
                pd.q_row0 = pd.q_off;
                pd.kv_off = j * Tc;
                pd.kv_row0 = pd.kv_off;
                pd.out = ob;
                pd.lse = lb;
                pd.out_T = Tc;
                pd.out_t0 = 0;
                pd.out_rows = BH * Tc;
                pd.out_f32 = 1;
                MergePair &mp = m.pairs[m.npairs++];
                mp.acc_t0 = i * Tc;
                mp.o_blk = ob;
                mp.lse_blk = lb;
                mp.final_ = (r == visits(N, causal, i) - 1) ? 1 : 0;
            }
            RSA_TRY(launch_block(q, k, v, dt, p, s, rec));
            RSA_TRY(launch_merge_rec(m, s, rec));
        }
    }
    return RSA_OK;
}

// Split-KV decode layout.  The cache of T keys is cut into N shards of T/N
// keys; each shard is cut further into splits of kv_split keys (a multiple of
// 128, at least 1024 unless a shard is shorter) so that about 2048 CTAs run.
// Every split writes an fp32 partial (o, lse) for every query row.
struct DecodeLayout {
    int64_t kv_split;
    int sps;  // splits per shard
    int S;    // splits in total
    size_t part_o, part_lse, total;
};

DecodeLayout decode_layout(int B, int H, int64_t T, int d, int64_t q_len, int N)
{
    DecodeLayout L{};
    const int64_t Tc = T / N;
    const int64_t BH = (int64_t)B * H;
    const int64_t groups = (q_len + kBf16RowsPerCta - 1) / kBf16RowsPerCta;
    int64_t want = (2048 + BH * N * groups - 1) / (BH * N * groups);
    if (want < 1)
        want = 1;
    int64_t ks = ((Tc + want - 1) / want + 127) / 128 * 128;
    if (ks < 1024)
        ks = 1024;
    if (ks > Tc)
        ks = Tc;
    L.kv_split = ks;
    L.sps = (int)((Tc + ks - 1) / ks);
    L.S = N * L.sps;
    L.part_o = align256((size_t)L.S * BH * q_len * d * 4);
    L.part_lse = align256((size_t)L.S * BH * q_len * 4);
    L.total = L.part_o + L.part_lse;
    return L;
}

rsa_status check_decode(rsa_dtype dt, int B, int H, int64_t T, int d, int q_len, int N)
{
    RSA_TRY(check_shape(dt, B, H, T, d));
    if (q_len < 1 || q_len > T)
        return fail(RSA_ERR_INVALID_ARG, "q_len=%d must be in [1, T=%lld]", q_len, (long long)T);
    if (N < 1 || N > T || T % N != 0)
        return fail(RSA_ERR_INVALID_ARG, "N=%d must be >= 1 and divide T=%lld", N, (long long)T);
    if (N > 1024)
        return fail(RSA_ERR_UNSUPPORTED, "N=%d exceeds 1024 shards", N);
    return RSA_OK;
}

}  // namespace

extern "C" {

static rsa_status check_two_pass(rsa_dtype dt, int B, int H, int64_t T, int d, int N)
{
    RSA_TRY(check_shape(dt, B, H, T, d));
    if (N < 1 || N > T || T % N != 0)
        return fail(RSA_ERR_INVALID_ARG, "N=%d must be >= 1 and divide T=%lld", N, (long long)T);
    if (dt != RSA_BF16 || d != 128)
        return fail(RSA_ERR_UNSUPPORTED, "two-pass attention is built for bf16 with d = 128");
    if ((T / N) % 128 != 0)
        return fail(RSA_ERR_UNSUPPORTED, "two-pass attention needs chunks T/N that are a multiple of 128");
    if ((int64_t)B * H > 65535 || T / 128 > 65535)
        return fail(RSA_ERR_UNSUPPORTED, "two-pass attention grid too large");
    return RSA_OK;
}

rsa_status rsa_two_pass_workspace_size(rsa_dtype dt, int B, int H, int64_t T, int d, int N, size_t *bytes)
{
    if (!bytes)
        return fail(RSA_ERR_INVALID_ARG, "bytes is NULL");
    RSA_TRY(check_two_pass(dt, B, H, T, d, N));
    const size_t rows = (size_t)B * H * (size_t)(T / N);
    *bytes = align256(rows * (size_t)T * 4) + align256(rows * (size_t)T * 2) + align256(rows * (size_t)(T / 64) * 8);
    return RSA_OK;
}

rsa_status rsa_two_pass_attn_fwd(const void *q, const void *k, const void *v, rsa_dtype dt, int B, int H, int64_t T,
                                 int d, int N, int causal, void *out, float *lse, void *workspace, size_t ws_bytes,
                                 rsa_stream_t stream)
{
    RSA_TRY(check_two_pass(dt, B, H, T, d, N));
    RSA_TRY(check_ptr(q, "q"));
    RSA_TRY(check_ptr(k, "k"));
    RSA_TRY(check_ptr(v, "v"));
    RSA_TRY(check_ptr(out, "out"));
    RSA_TRY(check_ptr(lse, "lse"));
    RSA_TRY(check_ptr(workspace, "workspace"));
    size_t need = 0;
    RSA_TRY(rsa_two_pass_workspace_size(dt, B, H, T, d, N, &need));
    if (ws_bytes < need)
        return fail(RSA_ERR_INVALID_ARG, "workspace holds %zu bytes, %zu needed", ws_bytes, need);
    RSA_TRY(check_device_for(dt));
    unsigned int *err = nullptr;
    RSA_TRY(device_error_word(&err));
    const size_t rows = (size_t)B * H * (size_t)(T / N);
    float *S = static_cast<float *>(workspace);
    void *P = static_cast<char *>(workspace) + align256(rows * (size_t)T * 4);
    void *stats = static_cast<char *>(P) + align256(rows * (size_t)T * 2);
    rsa_status inj;
    if (injected_failure("two-pass launch", &inj))
        return inj;
    cudaError_t e = launch_two_pass(q, k, v, (int64_t)B * H, T, N, causal, out, lse, S, P, stats,
                                    g_wait_limit_ns.load(), err, stream);
    if (e != cudaSuccess)
        return fail(RSA_ERR_CUDA, "two-pass launch: %s", cudaGetErrorString(e));
    return RSA_OK;
}

rsa_status rsa_decode_workspace_size(rsa_dtype dt, int B, int H, int64_t T, int d, int q_len, int N, size_t *bytes)
{
    if (!bytes)
        return fail(RSA_ERR_INVALID_ARG, "bytes is NULL");
    RSA_TRY(check_decode(dt, B, H, T, d, q_len, N));
    *bytes = decode_layout(B, H, T, d, q_len, N).total;
    return RSA_OK;
}

rsa_status rsa_decode_attn_fwd(const void *q, const void *k, const void *v, rsa_dtype dt, int B, int H, int64_t T,
                               int d, int q_len, int N, int causal, void *out, float *lse, void *workspace,
                               size_t ws_bytes, rsa_stream_t stream)
{
    RSA_TRY(check_decode(dt, B, H, T, d, q_len, N));
    RSA_TRY(check_ptr(q, "q"));
    RSA_TRY(check_ptr(k, "k"));
    RSA_TRY(check_ptr(v, "v"));
    RSA_TRY(check_ptr(out, "out"));
    RSA_TRY(check_ptr(lse, "lse"));
    const DecodeLayout lay = decode_layout(B, H, T, d, q_len, N);
    RSA_TRY(check_ptr(workspace, "workspace"));
    if (ws_bytes < lay.total)
        return fail(RSA_ERR_INVALID_ARG, "workspace holds %zu bytes, %zu needed", ws_bytes, lay.total);
    RSA_TRY(check_device_for(dt));
    unsigned int *err = nullptr;
    RSA_TRY(device_error_word(&err));
    const int64_t Tc = T / N;
    const int64_t BH = (int64_t)B * H;
    float *part_o = static_cast<float *>(workspace);
    float *part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + lay.part_o);
    // Shards are the pairs of the block kernel: query rows T-q_len..T-1 (the
    // newest tokens) against keys [i*Tc, (i+1)*Tc), cut into splits.
    for (int g0 = 0; g0 < N; g0 += kMaxPairsPerLaunch) {
        BlockParams p = base_params(dt, B, H, T, d, causal, q_len, Tc, err);
        p.q_T = q_len;
        p.kv_split = lay.kv_split;
        p.n_split = lay.sps;
        for (int i = g0; i < N && p.npairs < kMaxPairsPerLaunch; ++i) {
            PairDesc &pd = p.pairs[p.npairs++];
            pd.q_off = T - q_len;
            pd.q_row0 = 0;
            pd.kv_off = i * Tc;
            pd.kv_row0 = pd.kv_off;
            pd.out = part_o + (size_t)i * lay.sps * BH * q_len * d;
            pd.lse = part_lse + (size_t)i * lay.sps * BH * q_len;
            pd.out_T = q_len;
            pd.out_t0 = 0;
            pd.out_rows = (int64_t)lay.sps * BH * q_len;
            pd.out_f32 = 1;
            pd.mode = kStore;
            pd.split_stride = BH * q_len;
        }
        RSA_TRY(launch_block(q, k, v, dt, p, stream, nullptr));
    }
    rsa_status inj;
    if (injected_failure("merge of decode splits", &inj))
        return inj;
    cudaError_t e = launch_merge_splits(part_o, part_lse, lay.S, BH * q_len, d, out, dt == RSA_F32, lse, stream);
    if (e != cudaSuccess)
        return fail(RSA_ERR_CUDA, "merge of decode splits: %s", cudaGetErrorString(e));
    return RSA_OK;
}

rsa_status rsa_block_attn_fwd(const void *q, const void *k, const void *v, rsa_dtype dt, int B, int H, int64_t T,
                              int d, int64_t q_off, int64_t q_len, int64_t kv_off, int64_t kv_len, int causal,
                              void *o_blk, float *lse_blk, rsa_stream_t stream)
{
    RSA_TRY(check_shape(dt, B, H, T, d));
    RSA_TRY(check_ptr(q, "q"));
    RSA_TRY(check_ptr(k, "k"));
    RSA_TRY(check_ptr(v, "v"));
    RSA_TRY(check_ptr(o_blk, "o_blk"));
    RSA_TRY(check_ptr(lse_blk, "lse_blk"));
    if (q_len < 1 || kv_len < 1 || q_off < 0 || kv_off < 0 || q_off + q_len > T || kv_off + kv_len > T)
        return fail(RSA_ERR_INVALID_ARG, "pair [q_off=%lld, q_len=%lld, kv_off=%lld, kv_len=%lld] outside T=%lld",
                    (long long)q_off, (long long)q_len, (long long)kv_off, (long long)kv_len, (long long)T);
    RSA_TRY(check_device_for(dt));
    unsigned int *err = nullptr;
    RSA_TRY(device_error_word(&err));
    BlockParams p = base_params(dt, B, H, T, d, causal, q_len, kv_len, err);
    PairDesc &pd = p.pairs[p.npairs++];
    pd.q_off = q_off;
    pd.q_row0 = pd.q_off;
    pd.kv_off = kv_off;
    pd.kv_row0 = pd.kv_off;
    pd.out = o_blk;
    pd.lse = lse_blk;
    pd.out_T = q_len;
    pd.out_t0 = 0;
    pd.out_rows = (int64_t)B * H * q_len;
    pd.out_f32 = dt == RSA_F32;
    return launch_block(q, k, v, dt, p, stream, nullptr);
}

rsa_status rsa_block_attn_fold(const void *q, int64_t q_rows, const void *k, const void *v, int64_t kv_rows,
                               rsa_dtype dt, int B, int H, int d, int64_t q_row0, int64_t q_pos, int64_t q_len,
                               int64_t kv_row0, int64_t kv_pos, int64_t kv_len, int causal, int fold, float *acc,
                               float *lse, void *out, rsa_stream_t stream)
{
    RSA_TRY(check_shape(dt, B, H, q_rows, d));
    RSA_TRY(check_shape(dt, B, H, kv_rows, d));
    RSA_TRY(check_ptr(q, "q"));
    RSA_TRY(check_ptr(k, "k"));
    RSA_TRY(check_ptr(v, "v"));
    RSA_TRY(check_ptr(lse, "lse"));
    if (fold < RSA_FOLD_FIRST || fold > RSA_FOLD_ONLY)
        return fail(RSA_ERR_INVALID_ARG, "fold=%d is not one of RSA_FOLD_FIRST..RSA_FOLD_ONLY", fold);
    if (fold != RSA_FOLD_ONLY)
        RSA_TRY(check_ptr(acc, "acc"));
    if (fold == RSA_FOLD_LAST || fold == RSA_FOLD_ONLY)
        RSA_TRY(check_ptr(out, "out"));
    if (q_len < 1 || kv_len < 1 || q_row0 < 0 || kv_row0 < 0 || q_row0 + q_len > q_rows ||
        kv_row0 + kv_len > kv_rows || q_pos < 0 || kv_pos < 0)
        return fail(RSA_ERR_INVALID_ARG,
                    "pair rows [%lld, +%lld) of %lld query rows, [%lld, +%lld) of %lld key rows, positions "
                    "%lld, %lld: outside the tensors or negative",
                    (long long)q_row0, (long long)q_len, (long long)q_rows, (long long)kv_row0, (long long)kv_len,
                    (long long)kv_rows, (long long)q_pos, (long long)kv_pos);
    RSA_TRY(check_device_for(dt));
    unsigned int *err = nullptr;
    RSA_TRY(device_error_word(&err));
    BlockParams p = base_params(dt, B, H, kv_rows, d, causal, q_len, kv_len, err);
    p.q_T = q_rows;
    PairDesc &pd = p.pairs[p.npairs++];
    pd.q_off = q_pos;
    pd.q_row0 = q_row0;
    pd.kv_off = kv_pos;
    pd.kv_row0 = kv_row0;
    const bool to_out = fold == RSA_FOLD_LAST || fold == RSA_FOLD_ONLY;
    pd.out = to_out ? out : static_cast<void *>(acc);
    pd.lse = lse;
    pd.out_T = q_rows;
    pd.out_t0 = q_row0;
    pd.out_rows = (int64_t)B * H * q_rows;
    pd.out_f32 = to_out ? (dt == RSA_F32) : 1;
    pd.mode = fold == RSA_FOLD_MERGE ? kMergeAcc : (fold == RSA_FOLD_LAST ? kMergeFinal : kStore);
    pd.acc = acc;
    return launch_block(q, k, v, dt, p, stream, nullptr);
}

static rsa_status merge_common(const float *o_acc, const float *lse_acc, const void *o_blk, rsa_dtype blk_dt,
                               const float *lse_blk, int64_t rows, int d, void *out, rsa_dtype out_dt,
                               float *lse_out, int final_, cudaStream_t s)
{
    RSA_TRY(check_ptr(o_acc, "o_acc"));
    RSA_TRY(check_ptr(lse_acc, "lse_acc"));
    RSA_TRY(check_ptr(o_blk, "o_blk"));
    RSA_TRY(check_ptr(lse_blk, "lse_blk"));
    if (final_) {
        RSA_TRY(check_ptr(out, "out"));
        RSA_TRY(check_ptr(lse_out, "lse_out"));
    }
    if ((blk_dt != RSA_F32 && blk_dt != RSA_BF16) || (out_dt != RSA_F32 && out_dt != RSA_BF16))
        return fail(RSA_ERR_INVALID_ARG, "bad dtype");
    if (rows < 1)
        return fail(RSA_ERR_INVALID_ARG, "rows must be >= 1");
    if (d != 64 && d != 128)
        return fail(RSA_ERR_UNSUPPORTED, "d=%d not supported (64 or 128)", d);
    MergeParams m;
    memset(&m, 0, sizeof m);
    m.rows_per_pair = rows;
    m.Tc = rows;
    m.T = rows;
    m.d = d;
    m.npairs = 1;
    m.blk_f32 = blk_dt == RSA_F32;
    m.out_f32 = out_dt == RSA_F32;
    m.o_acc = const_cast<float *>(o_acc);
    m.lse_acc = const_cast<float *>(lse_acc);
    m.out = out;
    m.lse_out = lse_out;
    RSA_TRY(device_error_word(&m.err));
    m.pairs[0].acc_t0 = 0;
    m.pairs[0].o_blk = o_blk;
    m.pairs[0].lse_blk = lse_blk;
    m.pairs[0].final_ = final_;
    return launch_merge_rec(m, s, nullptr);
}

rsa_status rsa_merge(float *o_acc, float *lse_acc, const void *o_blk, rsa_dtype blk_dt, const float *lse_blk,
                     int64_t rows, int d, rsa_stream_t stream)
{
    return merge_common(o_acc, lse_acc, o_blk, blk_dt, lse_blk, rows, d, nullptr, RSA_F32, nullptr, 0, stream);
}

rsa_status rsa_merge_finalize(const float *o_acc, const float *lse_acc, const void *o_blk, rsa_dtype blk_dt,
                              const float *lse_blk, int64_t rows, int d, void *out, rsa_dtype out_dt,
                              float *lse_out, rsa_stream_t stream)
{
    return merge_common(o_acc, lse_acc, o_blk, blk_dt, lse_blk, rows, d, out, out_dt, lse_out, 1, stream);
}

rsa_status rsa_ring_attn_workspace_size(rsa_dtype dt, int B, int H, int64_t T, int d, int N, int causal,
                                        size_t *bytes)
{
    if (!bytes)
        return fail(RSA_ERR_INVALID_ARG, "bytes is NULL");
    RSA_TRY(check_shape(dt, B, H, T, d));
    if (N < 1 || N > T || T % N != 0)
        return fail(RSA_ERR_INVALID_ARG, "N=%d must be >= 1 and divide T=%lld", N, (long long)T);
    *bytes = ws_layout(dt, B, H, T, d, N, causal, true).total;
    return RSA_OK;
}

rsa_status rsa_ring_attn_fwd(const void *q, const void *k, const void *v, rsa_dtype dt, int B, int H, int64_t T,
                             int d, int N, int causal, void *out, float *lse, void *workspace, size_t ws_bytes,
                             rsa_stream_t stream)
{
    WsLayout lay;
    RSA_TRY(validate_ring(q, k, v, dt, B, H, T, d, N, out, lse, workspace, ws_bytes, causal, true, &lay));
    return ring_run(q, k, v, dt, B, H, T, d, N, causal, out, lse, workspace, lay, true, stream, nullptr);
}

// Which merge a ring variant uses: the fold in the block epilogue (the
// default, RSA_RING_FUSED_MERGE) or partials and the merge kernel
// (RSA_RING_SEPARATE_MERGE).
static rsa_status ring_flags(unsigned flags, bool *fused)
{
    const unsigned known = RSA_RING_FUSED_MERGE | RSA_RING_SEPARATE_MERGE;
    if (flags & ~known)
        return fail(RSA_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    if ((flags & RSA_RING_FUSED_MERGE) && (flags & RSA_RING_SEPARATE_MERGE))
        return fail(RSA_ERR_INVALID_ARG, "RSA_RING_FUSED_MERGE and RSA_RING_SEPARATE_MERGE exclude each other");
    *fused = (flags & RSA_RING_SEPARATE_MERGE) == 0;
    return RSA_OK;
}

static rsa_status ring_profiled(const void *q, const void *k, const void *v, rsa_dtype dt, int B, int H,
                                int64_t T, int d, int N, int causal, unsigned flags, void *out, float *lse,
                                void *workspace, size_t ws_bytes, rsa_stream_t stream, rsa_event_t *ev_start,
                                rsa_event_t *ev_stop, int *kind, int cap, int *n_launches)
{
    bool fused = true;
    RSA_TRY(ring_flags(flags, &fused));
    WsLayout lay;
    RSA_TRY(validate_ring(q, k, v, dt, B, H, T, d, N, out, lse, workspace, ws_bytes, causal, fused, &lay));
    const bool timed = ev_start || ev_stop || kind;
    if (timed && (!ev_start || !ev_stop || !kind))
        return fail(RSA_ERR_INVALID_ARG, "event and kind arrays must be given together");
    const int need = launch_count(N, causal, fused);
    if (n_launches)
        *n_launches = need;
    if (!timed)
        return ring_run(q, k, v, dt, B, H, T, d, N, causal, out, lse, workspace, lay, fused, stream, nullptr);
    if (cap < need)
        return fail(RSA_ERR_INVALID_ARG, "cap=%d but the ring makes %d launches", cap, need);
    Recorder rec;
    rec.start = ev_start;
    rec.stop = ev_stop;
    rec.kind = kind;
    rsa_status st = ring_run(q, k, v, dt, B, H, T, d, N, causal, out, lse, workspace, lay, fused, stream, &rec);
    if (n_launches)
        *n_launches = rec.n;
    return st;
}

rsa_status rsa_ring_attn_fwd_timed(const void *q, const void *k, const void *v, rsa_dtype dt, int B, int H,
                                   int64_t T, int d, int N, int causal, void *out, float *lse, void *workspace,
                                   size_t ws_bytes, rsa_stream_t stream, rsa_event_t *ev_start,
                                   rsa_event_t *ev_stop, int *kind, int cap, int *n_launches)
{
    if (!ev_start || !ev_stop || !kind || !n_launches)
        return fail(RSA_ERR_INVALID_ARG, "event/kind/count arrays must not be NULL");
    return ring_profiled(q, k, v, dt, B, H, T, d, N, causal, 0u, out, lse, workspace, ws_bytes, stream, ev_start,
                         ev_stop, kind, cap, n_launches);
}

rsa_status rsa_ring_attn_workspace_size_ex(rsa_dtype dt, int B, int H, int64_t T, int d, int N, int causal,
                                           unsigned flags, size_t *bytes)
{
    if (!bytes)
        return fail(RSA_ERR_INVALID_ARG, "bytes is NULL");
    bool fused = true;
    RSA_TRY(ring_flags(flags, &fused));
    RSA_TRY(check_shape(dt, B, H, T, d));
    if (N < 1 || N > T || T % N != 0)
        return fail(RSA_ERR_INVALID_ARG, "N=%d must be >= 1 and divide T=%lld", N, (long long)T);
    *bytes = ws_layout(dt, B, H, T, d, N, causal, fused).total;
    return RSA_OK;
}

rsa_status rsa_ring_attn_fwd_ex(const void *q, const void *k, const void *v, rsa_dtype dt, int B, int H,
                                int64_t T, int d, int N, int causal, unsigned flags, void *out, float *lse,
                                void *workspace, size_t ws_bytes, rsa_stream_t stream, rsa_event_t *ev_start,
                                rsa_event_t *ev_stop, int *kind, int cap, int *n_launches)
{
    return ring_profiled(q, k, v, dt, B, H, T, d, N, causal, flags, out, lse, workspace, ws_bytes, stream,
                         ev_start, ev_stop, kind, cap, n_launches);
}

rsa_status rsa_ring_schedule(int N, int causal, int round, int *q_chunk, int *kv_chunk, int cap, int *n_pairs)
{
    if (N < 1 || N > 1024 || round < 0 || round >= N || !n_pairs)
        return fail(RSA_ERR_INVALID_ARG, "need 1 <= N <= 1024, 0 <= round < N, n_pairs != NULL");
    const int n = round_pairs(N, causal ? 1 : 0, round, nullptr, nullptr);
    *n_pairs = n;
    if (n > cap || (n > 0 && (!q_chunk || !kv_chunk)))
        return fail(RSA_ERR_INVALID_ARG, "round has %d pairs; cap=%d", n, cap);
    round_pairs(N, causal ? 1 : 0, round, q_chunk, kv_chunk);
    return RSA_OK;
}

rsa_status rsa_set_wait_limit_ns(uint64_t limit_ns)
{
    if (limit_ns < 1000000ull)
        return fail(RSA_ERR_INVALID_ARG, "wait limit must be >= 1 ms");
    g_wait_limit_ns.store(limit_ns);
    return RSA_OK;
}

int rsa_debug_checks(void)
{
#ifdef RSA_DEBUG
    return 1;
#else
    return 0;
#endif
}

rsa_status rsa_debug_inject_launch_failure(int countdown)
{
    g_inject_countdown.store(countdown < 0 ? -1 : countdown);
    return RSA_OK;
}

rsa_status rsa_set_block_kernel(int which)
{
    if (which < RSA_BLOCK_KERNEL_AUTO || which > RSA_BLOCK_KERNEL_TWO_SM)
        return fail(RSA_ERR_INVALID_ARG, "block kernel choice %d is not 0, 1 or 2", which);
    g_tc_kernel.store(which);
    return RSA_OK;
}

rsa_status rsa_check_device_error(rsa_stream_t stream)
{
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return fail(RSA_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    DeviceError rec{};
    e = cudaMemcpyFromSymbol(&rec, g_device_error, sizeof rec);
    if (e != cudaSuccess)
        return fail(RSA_ERR_CUDA, "read error word: %s", cudaGetErrorString(e));
    const unsigned int v = rec.word;
    if (v == 0)
        return RSA_OK;
    const DeviceError zero{};
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    if (e != cudaSuccess)
        return fail(RSA_ERR_CUDA, "clear error word: %s", cudaGetErrorString(e));
    if (v & kDevErrTimeout)
        return fail(RSA_ERR_TIMEOUT, "a device wait exceeded its limit (site code 0x%02x)", v & 0xffu);
    if (v & kDevErrBounds)
        return fail(RSA_ERR_CUDA, "a device bounds check failed (site code 0x%02x, first bad index %lld)", v & 0xffu,
                    (long long)rec.bad_index_plus1 - 1);
    return fail(RSA_ERR_CUDA, "device error word 0x%x", v);
}

rsa_status rsa_selftest_wait_timeout(rsa_stream_t stream)
{
    unsigned int *err = nullptr;
    RSA_TRY(device_error_word(&err));
    cudaError_t e = launch_selftest_wait(g_wait_limit_ns.load(), err, stream);
    if (e != cudaSuccess)
        return fail(RSA_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
    return RSA_OK;
}

const char *rsa_status_string(rsa_status status)
{
    switch (status) {
    case RSA_OK: return "RSA_OK";
    case RSA_ERR_INVALID_ARG: return "RSA_ERR_INVALID_ARG";
    case RSA_ERR_UNSUPPORTED: return "RSA_ERR_UNSUPPORTED";
    case RSA_ERR_CUDA: return "RSA_ERR_CUDA";
    case RSA_ERR_TIMEOUT: return "RSA_ERR_TIMEOUT";
    }
    return "RSA_ERR_UNKNOWN";
}

const char *rsa_last_error_string(void) { return g_last_error; }

int rsa_version(void) { return 10000; }

}  // extern "C"
