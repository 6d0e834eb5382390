// Host-to-host ring attention: Q, K, V in host memory in, out and lse back to
// host memory, with the copies overlapped with the ring.
//
// Page: "Sequence parallelism -- splitting the token dimension across GPUs"
// (llmdaily, day 58), section "A better mental model: move blocks past the
// queries": blocks stream past queries that stay put.  Here the streaming is
// between host and device: the B*H heads are independent attention problems,
// so they are cut into slabs that flow through the GPU.  While the ring runs
// on slab g (on the caller's stream), slab g+1 is copied in on one library
// stream and slab g-1 is copied out on another.  Device slabs are double
// buffered, so a slab's copy in only has to wait for the ring two slabs back.
//
// Slab sizes ramp: the first slab's copy in and the last slab's copy out
// cannot hide under any ring, so they are small (an eighth of the largest
// slab), and slabs grow by about 1.6x at a time so that each copy hides under
// the ring of the slab before it (copying one head in takes less time than
// its ring).
//
// Host memory: copies from page-locked memory on 64 KiB base pages have been
// measured to lose most of their copy-engine bandwidth after the memory sat
// idle for some seconds on this machine class (211 GB/s falling towards
// 10-20 GB/s), while page-locked memory on transparent huge pages kept its
// speed -- as long as the kernel kept those pages huge, which it does not
// always do.  rsa_host_alloc therefore hands out huge-page-backed memory,
// registered with the driver, and each call picks how to move each tensor:
// the copy engines for a block that is still on huge pages (they run beside
// the ring almost for free), otherwise a copy kernel whose SM loads and
// stores reach the page-locked memory through its mapped address (measured
// at full link speed from such memory, at the price of slowing the ring by
// about a tenth while both run).
#include <fcntl.h>
#include <sys/ioctl.h>
#include <sys/mman.h>
#include <unistd.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <thread>
#include <vector>

#include "rsa_internal.h"

using rsa::fail;

namespace {

#define TRY(x)                         \
    do {                               \
        rsa_status st_ = (x);          \
        if (st_ != RSA_OK)             \
            return st_;                \
    } while (0)

// ---------------------------------------------------------------------------
// Page-locked host memory on transparent huge pages
// ---------------------------------------------------------------------------

struct HostBlock {
    void *map_base;   // whole mapping, guards included (huge kind)
    size_t map_len;
    size_t bytes;     // usable bytes at the block's address
    int kind;         // RSA_HOST_HUGE or RSA_HOST_PINNED
};

std::atomic<int> g_copy_mode{RSA_HOST_COPY_AUTO};

std::mutex g_host_mu;
std::map<uintptr_t, HostBlock> g_host_blocks;

size_t read_size_file(const char *path, size_t fallback)
{
    FILE *f = fopen(path, "r");
    if (!f)
        return fallback;
    unsigned long long v = 0;
    const int n = fscanf(f, "%llu", &v);
    fclose(f);
    return (n == 1 && v > 0) ? (size_t)v : fallback;
}

size_t huge_page_bytes()
{
    static const size_t h = read_size_file("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", 2u << 20);
    return h;
}

// AnonHugePages of the mapping that starts exactly at `start` (the guards
// keep the block's mapping from merging with its neighbours); 0 if unknown.
size_t smaps_huge_bytes(const void *start)
{
    FILE *f = fopen("/proc/self/smaps", "r");
    if (!f)
        return 0;
    char line[512];
    bool inside = false;
    size_t huge = 0;
    const uintptr_t want = reinterpret_cast<uintptr_t>(start);
    while (fgets(line, sizeof line, f)) {
        unsigned long long lo = 0, hi = 0;
        char dash = 0;
        if (sscanf(line, "%llx%c%llx", &lo, &dash, &hi) == 3 && dash == '-' && strchr(line, ':') &&
            strchr(line, ':') > strchr(line, ' ')) {
            inside = lo == want;
            continue;
        }
        unsigned long long kb = 0;
        if (inside && sscanf(line, "AnonHugePages: %llu kB", &kb) == 1) {
            huge = (size_t)kb * 1024;
            break;
        }
    }
    fclose(f);
    return huge;
}

// The kernel's page-table scan of one address range (the PAGEMAP_SCAN ioctl
// of /proc/self/pagemap, Linux 6.7 on), declared here so that older headers
// build.  Its cost grows with the range scanned, where a read of
// /proc/self/smaps walks every mapping of the process (tens of milliseconds
// in a process holding some GB of base pages).  Regions whose pages are
// mapped as huge pages carry kScanHuge.
struct ScanRegion {
    uint64_t start, end, categories;
};
struct ScanArg {
    uint64_t size, flags, start, end, walk_end, vec, vec_len, max_pages;
    uint64_t category_inverted, category_mask, category_anyof_mask, return_mask;
};
constexpr uint64_t kScanHuge = 1u << 6;
const unsigned long kPagemapScan = _IOWR('f', 16, ScanArg);

using Regions = std::vector<std::pair<uintptr_t, uintptr_t>>;

// The regions of [lo, hi) mapped by huge pages, in address order (adjacent
// huge pages come back as one region); false if the kernel cannot say.
// /proc/self/pagemap is opened per call: a descriptor kept open would go on
// describing the parent after a fork.  The cost grows with the page-table
// entries walked: a few for a range on huge pages, one per base page where
// the kernel has split them.
bool huge_regions(const void *p, size_t len, Regions *out)
{
    out->clear();
    const int fd = open("/proc/self/pagemap", O_RDONLY | O_CLOEXEC);
    if (fd < 0)
        return false;
    ScanRegion reg[32];
    uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    const uintptr_t hi = lo + len;
    bool ok = true;
    while (lo < hi) {
        ScanArg a{};
        a.size = sizeof a;
        a.start = lo;
        a.end = hi;
        a.vec = reinterpret_cast<uint64_t>(reg);
        a.vec_len = sizeof reg / sizeof reg[0];
        a.category_mask = kScanHuge;
        a.return_mask = kScanHuge;
        const int n = ioctl(fd, kPagemapScan, &a);
        if (n < 0) {
            ok = false;
            break;
        }
        for (int i = 0; i < n; ++i) {
            if (!out->empty() && out->back().second == reg[i].start)
                out->back().second = reg[i].end;
            else
                out->emplace_back(reg[i].start, reg[i].end);
        }
        if (a.walk_end <= lo)
            break;
        lo = a.walk_end;
    }
    close(fd);
    return ok;
}

// Bytes of [lo, lo + len) inside the regions.
size_t bytes_in(const Regions &r, uintptr_t lo, size_t len)
{
    const uintptr_t hi = lo + len;
    size_t b = 0;
    for (const auto &x : r) {
        const uintptr_t a = x.first > lo ? x.first : lo, e = x.second < hi ? x.second : hi;
        if (e > a)
            b += e - a;
    }
    return b;
}

// Huge-page bytes of a library block: the range scan where the kernel has
// it, else the AnonHugePages of its mapping.
size_t block_huge_bytes(const void *blk, size_t bytes)
{
    Regions r;
    if (huge_regions(blk, bytes, &r))
        return bytes_in(r, reinterpret_cast<uintptr_t>(blk), bytes);
    return smaps_huge_bytes(blk);
}

// Zero the block with a few threads so that every page exists (and is a huge
// page where the kernel can provide one) before it is registered.
void touch(void *p, size_t len)
{
    const size_t chunk = 256u << 20;
    const size_t n = (len + chunk - 1) / chunk;
    unsigned nt = std::thread::hardware_concurrency();
    nt = nt < 1 ? 1 : (nt > 8 ? 8 : nt);
    if (n < 2 || nt < 2) {
        memset(p, 0, len);
        return;
    }
    std::vector<std::thread> pool;
    for (unsigned t = 0; t < nt; ++t)
        pool.emplace_back([=] {
            for (size_t i = t; i < n; i += nt) {
                const size_t off = i * chunk;
                memset(static_cast<char *>(p) + off, 0, len - off < chunk ? len - off : chunk);
            }
        });
    for (auto &th : pool)
        th.join();
}

// ---------------------------------------------------------------------------
// Moving a slab: copy engines or a copy kernel
// ---------------------------------------------------------------------------

// 16-byte units from src to dst, one of them page-locked host memory reached
// through its mapped address.  CTAs of 256 threads of 32 registers, which fit
// beside a block-attention CTA (it leaves that much free), on half as many
// CTAs as the GPU has SMs: beside the page-1 ring with every tensor moved
// this way a step took 123.7-124.7 ms, against 128.5-129.2 ms with one CTA
// per SM and 138-154 ms with one per four SMs.
constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
    slab_copy_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src, size_t n16)
{
    size_t i = (size_t)blockIdx.x * kCopyThreads + threadIdx.x;
    const size_t stride = (size_t)gridDim.x * kCopyThreads;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride)
        dst[i] = src[i];
}

// How one host tensor of a call moves.  In automatic mode a tensor in a
// library block is decided copy by copy: its huge-page regions are read once
// per call, and each copy goes by the copy engines while its own range lies
// (90%) on huge pages, else by the copy kernel -- a block the kernel has
// split in a few places then moves mostly by the engines.
struct HostPath {
    int path = RSA_HOST_PATH_ENGINES;  // the tensor as a whole
    char *mapped = nullptr;            // mapped device address (page-locked memory)
    uintptr_t host = 0;                // the tensor's host address
    bool per_copy = false;             // decide each copy from `huge`
    Regions huge;                      // the tensor's huge-page regions (per_copy)
};

constexpr double kHugeShare = 0.9;  // engines at or above this huge-page share

// The library block containing [p, p + bytes), if any.
bool find_block(const void *p, size_t bytes, uintptr_t *start, HostBlock *hb)
{
    std::lock_guard<std::mutex> lock(g_host_mu);
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    auto it = g_host_blocks.upper_bound(a);
    if (it == g_host_blocks.begin())
        return false;
    --it;
    if (a < it->first || a + bytes > it->first + it->second.bytes)
        return false;
    *start = it->first;
    *hb = it->second;
    return true;
}

rsa_status choose_path(const void *p, size_t bytes, int mode, HostPath *hp)
{
    hp->path = RSA_HOST_PATH_ENGINES;
    hp->mapped = nullptr;
    hp->host = reinterpret_cast<uintptr_t>(p);
    hp->per_copy = false;
    hp->huge.clear();
    cudaPointerAttributes attr{};
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();  // pageable memory on older runtimes
        return RSA_OK;
    }
    if (attr.type != cudaMemoryTypeHost || !attr.devicePointer)
        return RSA_OK;  // pageable: the runtime stages the copy
    const char *mapped = static_cast<const char *>(attr.devicePointer);
    if ((reinterpret_cast<uintptr_t>(mapped) & 15u) != 0)
        return RSA_OK;  // the copy kernel moves 16-byte units
    hp->mapped = const_cast<char *>(mapped);
    bool kernel = mode == RSA_HOST_COPY_SM;
    if (mode == RSA_HOST_COPY_AUTO) {
        uintptr_t start = 0;
        HostBlock hb{};
        kernel = true;  // page-locked memory on base pages
        if (find_block(p, bytes, &start, &hb) && hb.kind == RSA_HOST_HUGE) {
            if (huge_regions(p, bytes, &hp->huge)) {
                hp->per_copy = true;
                kernel = (double)bytes_in(hp->huge, hp->host, bytes) < kHugeShare * (double)bytes;
            } else {  // no range scan: the whole block's count
                kernel = (double)smaps_huge_bytes(reinterpret_cast<void *>(start)) < kHugeShare * (double)hb.bytes;
            }
        }
    }
    hp->path = kernel ? RSA_HOST_PATH_KERNEL : RSA_HOST_PATH_ENGINES;
    return RSA_OK;
}

// The path of one copy of `bytes` at offset `off` into the tensor.
int copy_path(const HostPath &hp, size_t off, size_t bytes)
{
    if (!hp.per_copy || !hp.mapped)
        return hp.path;
    const bool huge = (double)bytes_in(hp.huge, hp.host + off, bytes) >= kHugeShare * (double)bytes;
    return huge ? RSA_HOST_PATH_ENGINES : RSA_HOST_PATH_KERNEL;
}

// Copy `bytes` (a multiple of 16) between device memory and host memory at
// host offset `off`, by the tensor's path, on stream s.
rsa_status move(const HostPath &hp, void *dev, const void *host_src, void *host_dst, size_t off, size_t bytes,
                bool to_device, int n_sm, cudaStream_t s)
{
    if (copy_path(hp, off, bytes) == RSA_HOST_PATH_KERNEL && hp.mapped && (bytes & 15u) == 0 &&
        (reinterpret_cast<uintptr_t>(dev) & 15u) == 0 && (off & 15u) == 0) {
        char *h = hp.mapped + off;
        const int ctas = (n_sm + 1) / 2;
        if (to_device)
            slab_copy_kernel<<<ctas, kCopyThreads, 0, s>>>(static_cast<uint4 *>(dev), reinterpret_cast<const uint4 *>(h),
                                                          bytes / 16);
        else
            slab_copy_kernel<<<ctas, kCopyThreads, 0, s>>>(reinterpret_cast<uint4 *>(h),
                                                          static_cast<const uint4 *>(dev), bytes / 16);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return fail(RSA_ERR_CUDA, "copy kernel launch: %s", cudaGetErrorString(e));
        return RSA_OK;
    }
    cudaError_t e = to_device ? cudaMemcpyAsync(dev, static_cast<const char *>(host_src) + off, bytes,
                                                cudaMemcpyHostToDevice, s)
                              : cudaMemcpyAsync(static_cast<char *>(host_dst) + off, dev, bytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess)
        return fail(RSA_ERR_CUDA, "cudaMemcpyAsync: %s", cudaGetErrorString(e));
    return RSA_OK;
}

// ---------------------------------------------------------------------------
// Slab plan
// ---------------------------------------------------------------------------

constexpr int kDefaultGroups = 8;

std::vector<int> slab_plan(int BH, int groups, bool ramp)
{
    std::vector<int> plan;
    if (BH <= 0)
        return plan;
    int g = groups < 1 ? 1 : (groups > BH ? BH : groups);
    const int cap = (BH + g - 1) / g;  // heads of the largest slab
    if (!ramp || cap < 8) {
        for (int left = BH; left > 0; left -= cap)
            plan.push_back(left < cap ? left : cap);
        return plan;
    }
    std::vector<int> up;
    for (int x = cap / 8 > 1 ? cap / 8 : 1; x < cap;) {
        up.push_back(x);
        const int nx = (x * 8) / 5;
        x = nx > x + 1 ? nx : x + 1;
    }
    const int down[3] = {cap / 2 > 1 ? cap / 2 : 1, cap / 4 > 1 ? cap / 4 : 1, cap / 8 > 1 ? cap / 8 : 1};
    int sum_up = 0;
    for (int x : up)
        sum_up += x;
    const int sum_down = down[0] + down[1] + down[2];
    if (sum_up + sum_down >= BH)
        return slab_plan(BH, groups, false);
    const int mid = BH - sum_up - sum_down;
    const int k = (mid + cap - 1) / cap;  // middle slabs, as equal as possible
    plan = up;
    for (int i = 0; i < k; ++i)
        plan.push_back(mid / k + (i < mid % k ? 1 : 0));
    for (int x : down)
        plan.push_back(x);
    return plan;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct HostWs {
    size_t in_bytes;    // one tensor slab [hg, T, d]
    size_t lse_bytes;   // one lse slab [hg, T]
    size_t ring_bytes;  // ring workspace of one slab of hg heads
    size_t total;
};

rsa_status host_ws(rsa_dtype dt, int B, int H, int64_t T, int d, int N, int causal, int hg, HostWs *w)
{
    const size_t esz = dt == RSA_BF16 ? 2 : 4;
    size_t ring = 0;
    TRY(rsa_ring_attn_workspace_size(dt, 1, hg, T, d, N, causal, &ring));
    (void)B;
    (void)H;
    w->in_bytes = align256((size_t)hg * (size_t)T * (size_t)d * esz);
    w->lse_bytes = align256((size_t)hg * (size_t)T * 4);
    w->ring_bytes = align256(ring);
    // two slots of {q, k, v, out, lse}, then the ring workspace
    w->total = 2 * (4 * w->in_bytes + w->lse_bytes) + w->ring_bytes;
    return RSA_OK;
}

// Copy streams and events of one device, created on the first call there and
// kept until the process exits.  The mutex is held while a call enqueues its
// work: a wait on an event binds to the record before it, so the events can be
// reused by the next call as soon as its predecessor has finished enqueuing.
struct DeviceStreams {
    std::mutex mu;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    std::vector<cudaEvent_t> ev;
};

constexpr int kMaxDevices = 64;
DeviceStreams g_dev_streams[kMaxDevices];

rsa_status cuda_ok(cudaError_t e, const char *what)
{
    if (e != cudaSuccess)
        return fail(RSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return RSA_OK;
}

rsa_status ensure_streams(DeviceStreams &ds, size_t n_events)
{
    if (!ds.s_in) {
        TRY(cuda_ok(cudaStreamCreateWithFlags(&ds.s_in, cudaStreamNonBlocking), "cudaStreamCreate (copy in)"));
        TRY(cuda_ok(cudaStreamCreateWithFlags(&ds.s_out, cudaStreamNonBlocking), "cudaStreamCreate (copy out)"));
    }
    while (ds.ev.size() < n_events) {
        cudaEvent_t e = nullptr;
        TRY(cuda_ok(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "cudaEventCreate"));
        ds.ev.push_back(e);
    }
    return RSA_OK;
}

}  // namespace

extern "C" {

rsa_status rsa_host_alloc(size_t bytes, void **ptr)
{
    if (!ptr)
        return fail(RSA_ERR_INVALID_ARG, "ptr is NULL");
    *ptr = nullptr;
    if (bytes == 0)
        return fail(RSA_ERR_INVALID_ARG, "bytes must be >= 1");
    const size_t huge = huge_page_bytes();
    const size_t page = (size_t)sysconf(_SC_PAGESIZE);
    const size_t len = (bytes + huge - 1) / huge * huge;
    const size_t map_len = len + huge + 2 * page;
    // Registering pins the pages for the long term, and the kernel may first
    // migrate them (out of a movable zone, for instance) and split huge pages
    // on the way.  So the huge-page share is measured after registering, and
    // a block that lost it is given back and tried again (a few times; the
    // best attempt is kept).
    constexpr int kAttempts = 4;
    void *best_base = nullptr, *best_blk = nullptr;
    size_t best_huge = 0;
    for (int attempt = 0; attempt < kAttempts; ++attempt) {
        // A huge-page-aligned block with a guard page (no access) on each
        // side; the guards keep its mapping separate from its neighbours'.
        void *base = mmap(nullptr, map_len, PROT_NONE, MAP_PRIVATE | MAP_ANONYMOUS | MAP_NORESERVE, -1, 0);
        if (base == MAP_FAILED)
            break;
        const uintptr_t b = reinterpret_cast<uintptr_t>(base);
        void *blk = reinterpret_cast<void *>((b + page + huge - 1) / huge * huge);
        if (mprotect(blk, len, PROT_READ | PROT_WRITE) != 0) {
            munmap(base, map_len);
            break;
        }
        madvise(blk, len, MADV_HUGEPAGE);
        touch(blk, len);
        if (cudaHostRegister(blk, len, cudaHostRegisterDefault) != cudaSuccess) {
            munmap(base, map_len);
            break;
        }
        const size_t h = block_huge_bytes(blk, len);
        if (!best_blk || h > best_huge) {
            if (best_blk) {
                cudaHostUnregister(best_blk);
                munmap(best_base, map_len);
            }
            best_base = base;
            best_blk = blk;
            best_huge = h;
        } else {
            cudaHostUnregister(blk);
            munmap(base, map_len);
        }
        if (best_huge >= len / 10 * 9)
            break;
    }
    HostBlock hb{best_base, map_len, len, RSA_HOST_HUGE};
    void *blk = best_blk;
    if (!blk || best_huge < len / 10 * 9) {
        // Mostly small pages: a driver-pinned block copies faster than a
        // registered one of small pages.
        if (blk) {
            cudaHostUnregister(blk);
            munmap(best_base, map_len);
        }
        void *p = nullptr;
        cudaError_t e = cudaHostAlloc(&p, len, cudaHostAllocDefault);
        if (e != cudaSuccess)
            return fail(RSA_ERR_CUDA, "cudaHostAlloc of %zu bytes: %s", len, cudaGetErrorString(e));
        blk = p;
        hb = HostBlock{nullptr, 0, len, RSA_HOST_PINNED};
    }
    std::lock_guard<std::mutex> lock(g_host_mu);
    g_host_blocks[reinterpret_cast<uintptr_t>(blk)] = hb;
    *ptr = blk;
    return RSA_OK;
}

rsa_status rsa_host_free(void *ptr)
{
    HostBlock hb{};
    {
        std::lock_guard<std::mutex> lock(g_host_mu);
        auto it = g_host_blocks.find(reinterpret_cast<uintptr_t>(ptr));
        if (!ptr || it == g_host_blocks.end())
            return fail(RSA_ERR_INVALID_ARG, "pointer %p was not returned by rsa_host_alloc", ptr);
        hb = it->second;
        g_host_blocks.erase(it);
    }
    if (hb.kind == RSA_HOST_PINNED)
        return cuda_ok(cudaFreeHost(ptr), "cudaFreeHost");
    cudaError_t e = cudaHostUnregister(ptr);
    munmap(hb.map_base, hb.map_len);
    return cuda_ok(e, "cudaHostUnregister");
}

rsa_status rsa_host_info(const void *ptr, size_t *bytes, size_t *huge_bytes, int *kind)
{
    HostBlock hb{};
    {
        std::lock_guard<std::mutex> lock(g_host_mu);
        auto it = g_host_blocks.find(reinterpret_cast<uintptr_t>(ptr));
        if (!ptr || it == g_host_blocks.end())
            return fail(RSA_ERR_INVALID_ARG, "pointer %p was not returned by rsa_host_alloc", ptr);
        hb = it->second;
    }
    if (bytes)
        *bytes = hb.bytes;
    if (kind)
        *kind = hb.kind;
    if (huge_bytes)
        *huge_bytes = hb.kind == RSA_HOST_HUGE ? block_huge_bytes(ptr, hb.bytes) : 0;
    return RSA_OK;
}

rsa_status rsa_set_host_copy_mode(int mode)
{
    if (mode < RSA_HOST_COPY_AUTO || mode > RSA_HOST_COPY_SM)
        return fail(RSA_ERR_INVALID_ARG, "host copy mode %d is not 0, 1 or 2", mode);
    g_copy_mode.store(mode);
    return RSA_OK;
}

rsa_status rsa_host_copy_path(const void *ptr, size_t bytes, int *path)
{
    if (!ptr || !path)
        return fail(RSA_ERR_INVALID_ARG, "ptr and path must not be NULL");
    HostPath hp;
    rsa_status st = choose_path(ptr, bytes, g_copy_mode.load(), &hp);
    if (st != RSA_OK)
        return st;
    *path = hp.path;
    return RSA_OK;
}

rsa_status rsa_host_slab_plan(int BH, int groups, int ramp, int *slabs, int cap, int *n_slabs)
{
    if (BH < 1 || groups < 1 || !n_slabs)
        return fail(RSA_ERR_INVALID_ARG, "need BH >= 1, groups >= 1, n_slabs != NULL");
    const std::vector<int> plan = slab_plan(BH, groups, ramp != 0);
    *n_slabs = (int)plan.size();
    if ((int)plan.size() > cap || !slabs)
        return fail(RSA_ERR_INVALID_ARG, "the plan has %zu slabs; cap=%d", plan.size(), cap);
    for (size_t i = 0; i < plan.size(); ++i)
        slabs[i] = plan[i];
    return RSA_OK;
}

rsa_status rsa_ring_attn_host_workspace_size(rsa_dtype dt, int B, int H, int64_t T, int d, int N, int causal,
                                             size_t *bytes)
{
    if (!bytes)
        return fail(RSA_ERR_INVALID_ARG, "bytes is NULL");
    if (B < 1 || H < 1)
        return fail(RSA_ERR_INVALID_ARG, "B, H must be >= 1");
    const int64_t BH = (int64_t)B * H;
    if (BH > 0x7fffffffLL)
        return fail(RSA_ERR_UNSUPPORTED, "B*H too large");
    const std::vector<int> plan = slab_plan((int)BH, kDefaultGroups, true);
    int hg = 0;
    for (int x : plan)
        hg = x > hg ? x : hg;
    HostWs w{};
    TRY(host_ws(dt, B, H, T, d, N, causal, hg, &w));
    *bytes = w.total;
    return RSA_OK;
}

rsa_status rsa_ring_attn_fwd_host(const void *q_host, const void *k_host, const void *v_host, rsa_dtype dt, int B,
                                  int H, int64_t T, int d, int N, int causal, void *out_host, float *lse_host,
                                  void *workspace, size_t ws_bytes, rsa_stream_t stream)
{
    if (!q_host || !k_host || !v_host || !out_host || !lse_host)
        return fail(RSA_ERR_INVALID_ARG, "host pointers must not be NULL");
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(RSA_ERR_INVALID_ARG, "workspace must be a non-NULL, 256-byte-aligned device pointer");
    size_t need = 0;
    TRY(rsa_ring_attn_host_workspace_size(dt, B, H, T, d, N, causal, &need));
    if (ws_bytes < need)
        return fail(RSA_ERR_INVALID_ARG, "workspace holds %zu bytes, %zu needed", ws_bytes, need);
    const int BH = B * H;
    const std::vector<int> plan = slab_plan(BH, kDefaultGroups, true);
    int hg = 0;
    for (int x : plan)
        hg = x > hg ? x : hg;
    HostWs w{};
    TRY(host_ws(dt, B, H, T, d, N, causal, hg, &w));
    int dev = 0;
    TRY(cuda_ok(cudaGetDevice(&dev), "cudaGetDevice"));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(RSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    if (dt == RSA_BF16) {  // checked here too, so that nothing is enqueued on a device the ring rejects
        int major = 0, minor = 0;
        TRY(cuda_ok(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "cudaDeviceGetAttribute"));
        TRY(cuda_ok(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "cudaDeviceGetAttribute"));
        if (major * 10 + minor != 103)
            return fail(RSA_ERR_UNSUPPORTED, "bf16 tensor-core path needs sm_103 (device is sm_%d%d)", major, minor);
    }
    DeviceStreams &ds = g_dev_streams[dev];
    std::lock_guard<std::mutex> lock(ds.mu);
    const size_t G = plan.size();
    TRY(ensure_streams(ds, 1 + 3 * G));
    cudaStream_t main = reinterpret_cast<cudaStream_t>(stream);
    cudaEvent_t ev_start = ds.ev[0];
    cudaEvent_t *ev_in = &ds.ev[1];
    cudaEvent_t *ev_comp = &ds.ev[1 + G];
    cudaEvent_t *ev_out = &ds.ev[1 + 2 * G];

    const size_t esz = dt == RSA_BF16 ? 2 : 4;
    const size_t head_bytes = (size_t)T * (size_t)d * esz;
    const size_t total_bytes = (size_t)BH * head_bytes;
    int n_sm = 0;
    TRY(cuda_ok(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute"));
    const int mode = g_copy_mode.load();
    HostPath hp[5];
    const void *host_ptr[5] = {q_host, k_host, v_host, out_host, lse_host};
    const size_t host_bytes[5] = {total_bytes, total_bytes, total_bytes, total_bytes, (size_t)BH * (size_t)T * 4};
    for (int i = 0; i < 5; ++i)
        TRY(choose_path(host_ptr[i], host_bytes[i], mode, &hp[i]));
    char *wsb = static_cast<char *>(workspace);
    char *slot_base[2] = {wsb, wsb + 4 * w.in_bytes + w.lse_bytes};
    void *ring_ws = wsb + 2 * (4 * w.in_bytes + w.lse_bytes);
    const char *src[3] = {static_cast<const char *>(q_host), static_cast<const char *>(k_host),
                          static_cast<const char *>(v_host)};

    // The copies may only start once the caller's earlier work on `stream`
    // is done (it may still be writing the host inputs' producers or reading
    // the workspace).
    TRY(cuda_ok(cudaEventRecord(ev_start, main), "cudaEventRecord"));
    TRY(cuda_ok(cudaStreamWaitEvent(ds.s_in, ev_start, 0), "cudaStreamWaitEvent"));
    TRY(cuda_ok(cudaStreamWaitEvent(ds.s_out, ev_start, 0), "cudaStreamWaitEvent"));
    int h0 = 0;
    for (size_t g = 0; g < G; ++g) {
        const int n = plan[g];
        char *slot = slot_base[g % 2];
        char *dq = slot, *dk = slot + w.in_bytes, *dv = slot + 2 * w.in_bytes, *dout = slot + 3 * w.in_bytes;
        float *dlse = reinterpret_cast<float *>(slot + 4 * w.in_bytes);
        const size_t off = (size_t)h0 * head_bytes, nbytes = (size_t)n * head_bytes;
        // copy in (slot reuse: the ring two slabs back has read it)
        if (g >= 2)
            TRY(cuda_ok(cudaStreamWaitEvent(ds.s_in, ev_comp[g - 2], 0), "cudaStreamWaitEvent"));
        char *dst[3] = {dq, dk, dv};
        for (int t = 0; t < 3; ++t)
            TRY(move(hp[t], dst[t], src[t], nullptr, off, nbytes, true, n_sm, ds.s_in));
        TRY(cuda_ok(cudaEventRecord(ev_in[g], ds.s_in), "cudaEventRecord"));
        // ring on the caller's stream (slot reuse: slab g-2's outputs are out)
        TRY(cuda_ok(cudaStreamWaitEvent(main, ev_in[g], 0), "cudaStreamWaitEvent"));
        if (g >= 2)
            TRY(cuda_ok(cudaStreamWaitEvent(main, ev_out[g - 2], 0), "cudaStreamWaitEvent"));
        TRY(rsa_ring_attn_fwd(dq, dk, dv, dt, 1, n, T, d, N, causal, dout, dlse, ring_ws, w.ring_bytes, stream));
        TRY(cuda_ok(cudaEventRecord(ev_comp[g], main), "cudaEventRecord"));
        // copy out
        TRY(cuda_ok(cudaStreamWaitEvent(ds.s_out, ev_comp[g], 0), "cudaStreamWaitEvent"));
        TRY(move(hp[3], dout, nullptr, out_host, off, nbytes, false, n_sm, ds.s_out));
        TRY(move(hp[4], dlse, nullptr, lse_host, (size_t)h0 * (size_t)T * 4, (size_t)n * (size_t)T * 4, false, n_sm,
                 ds.s_out));
        TRY(cuda_ok(cudaEventRecord(ev_out[g], ds.s_out), "cudaEventRecord"));
        h0 += n;
    }
    // `stream` passes this point once the last copy out is done.
    return cuda_ok(cudaStreamWaitEvent(main, ev_out[G - 1], 0), "cudaStreamWaitEvent");
}

}  // extern "C"
