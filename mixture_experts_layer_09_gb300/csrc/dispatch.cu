// dispatch.cu -- stage 2 of the routed MoE layer: token-to-expert dispatch.
//
// Per-expert histogram, exclusive prefix scan and a stable permutation of the T*k slots,
// without atomics (daScript PR #3988 "dasLLAMA vulkan: a MoE that fits the card ...",
// routed-block commit: MoeSched counts each expert's slots and places the buckets with
// exclusive scans; the slot map lands in slot order).  Each warp owns a contiguous run of
// slots and a private histogram row in shared memory; within a warp, slots with the same
// expert are grouped with __match_any_sync and ranked by lane order, so the permutation is
// stable and identical on every run.
//
// Small batches (T*k <= kSmallSlots) run one CTA that does all three phases.  Larger ones
// run count -> scatter with per-CTA counts in the workspace; each scatter CTA derives its own
// starting positions from the whole count table (column totals, their exclusive scan over the
// experts, and the sum over the CTAs before it), so no scan launch sits between the two.  A
// CTA takes as few slots as keeps the table (CTAs x E) within 16384 entries and 256 rows.
//
// Besides offsets/perm/inv the dispatch writes the list of experts that received at least
// one slot (ascending) and its length; the expert kernels iterate over that list.
#include "common.cuh"
#include "internal.h"
#include "route_core.cuh"

namespace moe {

constexpr int kSmallSlots = 2048;
constexpr int kBigWarps = 8;            // warps per CTA in the multi-CTA path
constexpr int kMinSlotsPerCta = 256;    // one 32-slot walk per warp
constexpr int kMaxTableRows = 256;      // CTAs of the multi-CTA path
constexpr int kMaxTableInts = 16384;    // count table entries (every scatter CTA reads it whole)

// Slots per CTA of the multi-CTA path: the smallest power-of-two multiple of 256 whose CTA
// count n / spc fits both the table bounds.
__host__ __device__ inline int slots_per_cta(int n, int E) {
    const int max_rows = min(kMaxTableRows, kMaxTableInts / E);
    int spc = kMinSlotsPerCta;
    while ((n + spc - 1) / spc > max_rows) spc *= 2;
    return spc;
}

// One CTA of 1024 threads (32 warps) for T*k <= kSmallSlots.
__global__ void __launch_bounds__(1024) dispatch_small_kernel(
    const int32_t* __restrict__ ids, int n, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
    int32_t* inv, int32_t* active, int32_t* n_active, int* status) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int hist[];  // [32][E]
    __shared__ int scratch[9];
    const int w = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int per = ((n + 31) / 32 + 31) / 32 * 32;
    const int begin = min(n, w * per), end = min(n, begin + per);
    warp_walk(ids, begin, end, E, hist + w * E, 0, perm, inv, status);
    __syncthreads();
    finalize_plan(hist, 32, E, n, counts, offsets, active, n_active, scratch);
    __syncthreads();
    warp_walk(ids, begin, end, E, hist + w * E, 1, perm, inv, status);
}

// Multi-CTA path, phase 1: per-CTA histogram.
__global__ void __launch_bounds__(kBigWarps * 32) dispatch_count_kernel(
    const int32_t* __restrict__ ids, int n, int E, int spc, int* __restrict__ cta_cnt, int* status) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int hist[];  // [kBigWarps][E]
    const int w = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kBigWarps * E; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int spw = spc / kBigWarps;
    const int begin = min(n, blockIdx.x * spc + w * spw);
    const int end = min(n, begin + spw);
    warp_walk(ids, begin, end, E, hist + w * E, 0, nullptr, nullptr, status);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int s = 0;
        for (int q = 0; q < kBigWarps; ++q) s += hist[q * E + e];
        cta_cnt[static_cast<size_t>(blockIdx.x) * E + e] = s;
    }
}

// Phase 2: stable scatter.  The CTA loads the whole count table into shared memory (coalesced,
// sixteen loads in flight per thread), then sums each expert's column in parallel parts: the
// expert's total and the part of it counted by the CTAs before this one.  The totals' exclusive
// scan over the experts gives the bucket offsets, which CTA 0 also writes out with the counts
// and the active-expert list.
__global__ void __launch_bounds__(kBigWarps * 32) dispatch_scatter_kernel(
    const int32_t* __restrict__ ids, int n, int E, int spc, int nblk, const int* __restrict__ cta_cnt,
    int32_t* counts, int32_t* offsets, int32_t* active, int32_t* n_active, int32_t* perm, int32_t* inv,
    int* status, int* tiles, int* n_tiles) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int hist[];  // [kBigWarps][E] | the count table [nblk][E]
    int* tbl = hist + kBigWarps * E;
    __shared__ int scratch[9];
    __shared__ int base_e[MOE_MAX_E];
    __shared__ int part_tot[kBigWarps * 32], part_bef[kBigWarps * 32];
    const int w = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kBigWarps * E; i += blockDim.x) hist[i] = 0;
    const int nt = nblk * E;
    for (int i0 = 0; i0 < nt; i0 += 16 * kBigWarps * 32) {
        int v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int i = i0 + u * kBigWarps * 32 + static_cast<int>(threadIdx.x);
            v[u] = i < nt ? __ldg(cta_cnt + i) : 0;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int i = i0 + u * kBigWarps * 32 + static_cast<int>(threadIdx.x);
            if (i < nt) tbl[i] = v[u];
        }
    }
    __syncthreads();
    const int P = kBigWarps * 32 / E;  // threads per column (E <= 256)
    {
        const int e = threadIdx.x % E, q = threadIdx.x / E;
        if (q < P) {
            int tot = 0, bef = 0;
            for (int r = q; r < nblk; r += P) {
                const int c = tbl[r * E + e];
                tot += c;
                if (r < static_cast<int>(blockIdx.x)) bef += c;
            }
            part_tot[q * E + e] = tot;
            part_bef[q * E + e] = bef;
        }
    }
    __syncthreads();
    {
        const int e = threadIdx.x;
        int total = 0, before = 0;
        if (e < E) {
            for (int q = 0; q < P; ++q) {
                total += part_tot[q * E + e];
                before += part_bef[q * E + e];
            }
        }
        int sum, nact;
        const int off = cta_exclusive_scan_256(e < E ? total : 0, scratch, &sum);
        const int flag = (e < E && total > 0) ? 1 : 0;
        const int apos = cta_exclusive_scan_256(flag, scratch, &nact);
        if (e < E) {
            base_e[e] = off + before;
            if (blockIdx.x == 0) {
                offsets[e] = off;
                if (counts) counts[e] = total;
                if (flag) active[apos] = e;
            }
        }
        if (blockIdx.x == 0 && e == 0) {
            offsets[E] = sum;
            *n_active = nact;
        }
        if (tiles && blockIdx.x == 0) {
            // the tensor arm's tile list (as build_tiles_kernel): a bucket of c rows takes
            // ceil(c / kGemmTileN) tiles of equal size
            const int nt = (e < E) ? (total + kGemmTileN - 1) / kGemmTileN : 0;
            int ntot;
            const int tb = cta_exclusive_scan_256(nt, scratch, &ntot);
            if (e < E) {
                const int per = nt > 0 ? (total + nt - 1) / nt : 0;
                for (int j = 0; j < nt; ++j) {
                    tiles[3 * (tb + j)] = e;
                    tiles[3 * (tb + j) + 1] = off + j * per;
                    tiles[3 * (tb + j) + 2] = max(0, min(per, total - j * per));
                }
            }
            if (e == 0) *n_tiles = ntot;
        }
    }
    __syncthreads();
    const int spw = spc / kBigWarps;
    const int begin = min(n, blockIdx.x * spc + w * spw);
    const int end = min(n, begin + spw);
    warp_walk(ids, begin, end, E, hist + w * E, 0, nullptr, nullptr, nullptr);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = base_e[e];
        for (int q = 0; q < kBigWarps; ++q) {
            const int tmp = hist[q * E + e];
            hist[q * E + e] = run;
            run += tmp;
        }
    }
    __syncthreads();
    warp_walk(ids, begin, end, E, hist + w * E, 1, perm, inv, status);
}

// Shared memory of the scatter: the per-warp histograms and the whole count table.
static size_t scatter_smem(int nblk, int E) {
    return (static_cast<size_t>(kBigWarps) + nblk) * E * sizeof(int);
}
static cudaError_t scatter_attr() {
    static const cudaError_t once = cudaFuncSetAttribute(
        dispatch_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>((static_cast<size_t>(kBigWarps) * MOE_MAX_E + kMaxTableInts) * sizeof(int)));
    return once;
}

size_t dispatch_scratch_bytes(int n, int E) {
    if (n <= kSmallSlots) return 0;
    const int spc = slots_per_cta(n, E);
    const size_t nblk = (n + spc - 1) / spc;
    return align_up(nblk * E * sizeof(int), kWsAlign);
}

cudaError_t launch_dispatch(const int32_t* ids, int n, int E, int32_t* counts, int32_t* offsets,
                            int32_t* perm, int32_t* inv, int32_t* active, int32_t* n_active,
                            void* scratch, int* status, cudaStream_t st) {
    if (n <= kSmallSlots) {
        const size_t smem = 32 * E * sizeof(int);
        {
            KernelScope ks_("dispatch_small", st);
            return launch_pdl(dispatch_small_kernel, dim3(1), dim3(1024), smem, st, ids, n, E, counts, offsets, perm,
                              inv, active, n_active, status);
        }
    }
    const int spc = slots_per_cta(n, E);
    const int nblk = (n + spc - 1) / spc;
    int* cnt = static_cast<int*>(scratch);
    const size_t smem = kBigWarps * E * sizeof(int);
    {
        KernelScope ks_("dispatch_count", st);
        cudaError_t e = launch_pdl(dispatch_count_kernel, dim3(nblk), dim3(kBigWarps * 32), smem, st, ids, n, E, spc,
                                   cnt, status);
        if (e != cudaSuccess) return e;
    }
    {
        cudaError_t e = scatter_attr();
        if (e != cudaSuccess) return e;
        KernelScope ks_("dispatch_scatter", st);
        return launch_pdl(dispatch_scatter_kernel, dim3(nblk), dim3(kBigWarps * 32), scatter_smem(nblk, E), st, ids, n,
                          E, spc, nblk,
                          static_cast<const int*>(cnt), counts, offsets, active, n_active, perm, inv, status,
                          static_cast<int*>(nullptr), static_cast<int*>(nullptr));
    }
}

bool dispatch_counted_supported(int nblk, int E) {
    return nblk >= 1 && nblk <= kMaxTableRows && static_cast<long>(nblk) * E <= kMaxTableInts;
}

cudaError_t launch_dispatch_counted(const int32_t* ids, int n, int E, int spc, int nblk, const int* cta_cnt,
                                    int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* active,
                                    int32_t* n_active, int* status, int* tiles, int* n_tiles, cudaStream_t st) {
    if (spc % kBigWarps || !dispatch_counted_supported(nblk, E)) return cudaErrorInvalidValue;
    cudaError_t e = scatter_attr();
    if (e != cudaSuccess) return e;
    KernelScope ks_("dispatch_scatter+tiles", st);
    return launch_pdl(dispatch_scatter_kernel, dim3(nblk), dim3(kBigWarps * 32), scatter_smem(nblk, E), st, ids,
                      n, E, spc, nblk, cta_cnt, counts, offsets, active, n_active, perm, inv, status, tiles, n_tiles);
}

}  // namespace moe

// ------------------------------------------------------------------ allocation-free variant
// moe_dispatch_static: the same dispatch kernels, with their scratch (status word,
// active-expert list, per-CTA count table) in one fixed array compiled into the library
// instead of a caller workspace.  It serves callers that must not allocate device memory at
// call time: code running under a framework whose device pool is fixed at start-up, plugin
// callbacks of a serving runtime that forbid allocation, or latency-critical loops where an
// allocation's implicit device synchronisation cannot be paid.  Every GPU that loads the
// library holds the array (about 66 KiB) until the process exits.
#include <mutex>

namespace moe {
namespace {
constexpr size_t kStaticStatusBytes = 256;
constexpr size_t kStaticActiveBytes = 2048;  // active list: E + 1 <= 257 ints
constexpr size_t kStaticTableBytes = static_cast<size_t>(kMaxTableInts) * sizeof(int);  // nblk * E bound
constexpr size_t kStaticBytes = kStaticStatusBytes + kStaticActiveBytes + kStaticTableBytes;
}  // namespace
}  // namespace moe

static __device__ __align__(256) unsigned char g_dispatch_scratch[moe::kStaticBytes];

namespace {
constexpr int kMaxDevices = 128;
std::mutex g_static_mu;
void* g_static_addr[kMaxDevices] = {};

// Device address of g_dispatch_scratch on the current device.  The name is only a host-side
// stand-in for the array, so the address is looked up with that device current.  It is looked
// up again on every call whose stream is not being captured (a device reset reloads the
// library's module, which moves the array), and the last address is kept for calls made while
// a capture is in progress, where the lookup is not made.
int static_scratch_address(cudaStream_t st, void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (cap == cudaStreamCaptureStatusNone || !g_static_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_static_addr[dev] = p;
    }
    *out = g_static_addr[dev];
    return MOE_OK;
}
}  // namespace

extern "C" MOE_API int moe_dispatch_static(const int32_t* topk_ids, int T, int k, int E, int32_t* counts,
                                           int32_t* offsets, int32_t* perm, int32_t* inv, moe_stream_t stream) {
    if (T < 0 || k < 1 || k > MOE_MAX_K || E < 1 || E > MOE_MAX_E) return MOE_ERR_INVALID_ARG;
    if (static_cast<long long>(T) * k > MOE_DISPATCH_STATIC_MAX_SLOTS) return MOE_ERR_INVALID_ARG;
    if (!offsets || (T > 0 && (!topk_ids || !perm || !inv))) return MOE_ERR_INVALID_ARG;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;
    void* base = nullptr;
    if (int s = static_scratch_address(static_cast<cudaStream_t>(stream), &base)) return s;
    char* p = static_cast<char*>(base);
    int* status = reinterpret_cast<int*>(p);
    int32_t* active = reinterpret_cast<int32_t*>(p + moe::kStaticStatusBytes);
    void* table = p + moe::kStaticStatusBytes + moe::kStaticActiveBytes;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the kernels record a fault only into a zero status word: clear the previous call's
    if (cudaMemsetAsync(status, 0, moe::kStaticStatusBytes, st) != cudaSuccess) return MOE_ERR_CUDA;
    return moe::launch_dispatch(topk_ids, T * k, E, counts, offsets, perm, inv, active, active + E, table, status,
                                st) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}
