// slot_copy.cu -- kda_slot_copy: one launch that clears, copies and fans out
// state slots over several pools.
//
// "State semantics" page, section 2: rollback is an exact block copy, and the
// engines fold the per-tensor clear/copy replays into a single launch driven
// by per-tensor pointer / stride / length arrays; section 3: a fork copies the
// full parent state to every candidate (copy-on-write is off for state).
//
// Design: a one-block check kernel first proves the copy sets disjoint (a
// bitmap over slot ids in caller-provided scratch) and writes a verdict word;
// the copy kernel then streams every (operation, pool, 16 KiB piece) work item
// with 16-byte vector loads and stores.  A fan-out source piece is read once
// into registers and written to each of its destinations.  The copy kernel
// reads the verdict first and does nothing if the check failed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"
#include "kda_host.h"

namespace kda {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kVecPerThread = 4;  // 4 x 16 B per thread per piece
constexpr int64_t kPieceBytes = (int64_t)kCopyThreads * kVecPerThread * 16;  // 16 KiB

struct PoolSet {
    kda_pool_desc d[KDA_MAX_POOLS];
    int64_t piece_off[KDA_MAX_POOLS + 1];  // prefix sum of pieces per slot
    int n;
};

__global__ void __launch_bounds__(1024) slot_copy_check_kernel(
    const int32_t* __restrict__ clear, int32_t n_clear, const int32_t* __restrict__ src,
    const int32_t* __restrict__ offs, const int32_t* __restrict__ dst, int32_t n_src, int32_t n_dst,
    int64_t min_slots, uint32_t* __restrict__ bitmap, int64_t n_words, int32_t* __restrict__ verdict,
    int32_t* __restrict__ dev_status) {
    __shared__ int bad;
    if (threadIdx.x == 0) bad = 0;
    for (int64_t i = threadIdx.x; i < n_words; i += blockDim.x) bitmap[i] = 0u;
    __syncthreads();
    int mine = 0;
    // CSR shape
    for (int i = threadIdx.x; i < n_src; i += blockDim.x)
        if (offs[i] > offs[i + 1]) mine |= KDA_DEV_BAD_SLOT;
    if (threadIdx.x == 0 && (offs[0] != 0 || offs[n_src] != n_dst)) mine |= KDA_DEV_BAD_SLOT;
    // destinations and clears: in range and pairwise distinct
    const int n_mark = n_dst + n_clear;
    for (int i = threadIdx.x; i < n_mark; i += blockDim.x) {
        const int s = i < n_dst ? dst[i] : clear[i - n_dst];
        if (s < 0 || s >= min_slots) {
            mine |= KDA_DEV_BAD_SLOT;
            continue;
        }
        const uint32_t bit = 1u << (s & 31);
        if (atomicOr(&bitmap[s >> 5], bit) & bit) mine |= KDA_DEV_OVERLAP;
    }
    __syncthreads();
    // sources: in range and not written by anything
    for (int i = threadIdx.x; i < n_src; i += blockDim.x) {
        const int s = src[i];
        if (s < 0 || s >= min_slots) {
            mine |= KDA_DEV_BAD_SLOT;
            continue;
        }
        if (__ldcg(&bitmap[s >> 5]) & (1u << (s & 31))) mine |= KDA_DEV_OVERLAP;
    }
    if (mine) atomicOr(&bad, mine);
    __syncthreads();
    if (threadIdx.x == 0) {
        *verdict = bad;
        if (bad) report(dev_status, bad);
    }
}

__global__ void __launch_bounds__(kCopyThreads) slot_copy_kernel(
    PoolSet ps, const int32_t* __restrict__ clear, int32_t n_clear, const int32_t* __restrict__ src,
    const int32_t* __restrict__ offs, const int32_t* __restrict__ dst, int32_t n_src,
    const int32_t* __restrict__ verdict) {
    if (*verdict != 0) return;
    const int64_t per_op = ps.piece_off[ps.n];
    const int64_t n_items = (int64_t)(n_clear + n_src) * per_op;
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int op = (int)(item / per_op);
        const int64_t rem = item - (int64_t)op * per_op;
        int p = 0;
        while (rem >= ps.piece_off[p + 1]) ++p;
        const int64_t piece = rem - ps.piece_off[p];
        const kda_pool_desc& d = ps.d[p];
        const int64_t byte0 = piece * kPieceBytes;
        char* base = static_cast<char*>(d.base);
        if (op < n_clear) {
            char* slot = base + (int64_t)clear[op] * d.slot_stride_bytes;
#pragma unroll
            for (int j = 0; j < kVecPerThread; ++j) {
                const int64_t b = byte0 + ((int64_t)j * kCopyThreads + threadIdx.x) * 16;
                if (b < d.slot_bytes) *reinterpret_cast<uint4*>(slot + b) = make_uint4(0, 0, 0, 0);
            }
        } else {
            const int i = op - n_clear;
            const char* from = base + (int64_t)src[i] * d.slot_stride_bytes;
            uint4 v[kVecPerThread];
#pragma unroll
            for (int j = 0; j < kVecPerThread; ++j) {
                const int64_t b = byte0 + ((int64_t)j * kCopyThreads + threadIdx.x) * 16;
                if (b < d.slot_bytes) v[j] = __ldcs(reinterpret_cast<const uint4*>(from + b));
            }
            const int e0 = offs[i], e1 = offs[i + 1];
            for (int e = e0; e < e1; ++e) {
                char* to = base + (int64_t)dst[e] * d.slot_stride_bytes;
#pragma unroll
                for (int j = 0; j < kVecPerThread; ++j) {
                    const int64_t b = byte0 + ((int64_t)j * kCopyThreads + threadIdx.x) * 16;
                    if (b < d.slot_bytes) __stcs(reinterpret_cast<uint4*>(to + b), v[j]);
                }
            }
        }
    }
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" size_t kda_slot_copy_workspace_size(int64_t num_slots) {
    if (num_slots < 0) return 0;
    // verdict word (padded to 16 B) + one bit per slot, rounded to 16 B
    return 16 + (size_t)((num_slots + 127) / 128) * 16;
}

extern "C" kda_status kda_slot_copy(const kda_pool_desc* pools, int32_t n_pools,
                                    const int32_t* clear_slots, int32_t n_clear,
                                    const int32_t* src_slots, const int32_t* dst_offsets,
                                    const int32_t* dst_slots, int32_t n_src, int32_t n_dst,
                                    void* workspace, size_t ws_bytes, int32_t* dev_status,
                                    void* stream) {
    KDA_REQUIRE(pools != nullptr && n_pools > 0 && n_pools <= KDA_MAX_POOLS, KDA_ERR_INVALID_ARG);
    KDA_REQUIRE(n_clear >= 0 && n_src >= 0 && n_dst >= 0, KDA_ERR_INVALID_ARG);
    KDA_REQUIRE(n_clear == 0 || clear_slots != nullptr, KDA_ERR_INVALID_ARG);
    KDA_REQUIRE(dst_offsets != nullptr, KDA_ERR_INVALID_ARG);
    KDA_REQUIRE(n_src == 0 || src_slots != nullptr, KDA_ERR_INVALID_ARG);
    KDA_REQUIRE(n_dst == 0 || dst_slots != nullptr, KDA_ERR_INVALID_ARG);
    PoolSet ps;
    ps.n = n_pools;
    ps.piece_off[0] = 0;
    int64_t min_slots = INT64_MAX, max_slots = 0;
    for (int i = 0; i < n_pools; ++i) {
        const kda_pool_desc& d = pools[i];
        KDA_REQUIRE(d.base != nullptr && aligned16(d.base), KDA_ERR_INVALID_ARG);
        KDA_REQUIRE(d.slot_bytes > 0 && d.slot_bytes % 16 == 0, KDA_ERR_INVALID_ARG);
        KDA_REQUIRE(d.slot_stride_bytes >= d.slot_bytes && d.slot_stride_bytes % 16 == 0,
                    KDA_ERR_INVALID_ARG);
        KDA_REQUIRE(d.num_slots > 0, KDA_ERR_INVALID_ARG);
        ps.d[i] = d;
        ps.piece_off[i + 1] = ps.piece_off[i] + (d.slot_bytes + kPieceBytes - 1) / kPieceBytes;
        min_slots = d.num_slots < min_slots ? d.num_slots : min_slots;
        max_slots = d.num_slots > max_slots ? d.num_slots : max_slots;
    }
    const size_t need = kda_slot_copy_workspace_size(min_slots);
    KDA_REQUIRE(workspace != nullptr && aligned16(workspace) && ws_bytes >= need,
                KDA_ERR_INVALID_ARG);
    (void)max_slots;
    cudaStream_t s = as_stream(stream);
    int32_t* verdict = static_cast<int32_t*>(workspace);
    uint32_t* bitmap = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + 16);
    const int64_t n_words = (min_slots + 31) / 32;
    slot_copy_check_kernel<<<1, 1024, 0, s>>>(clear_slots, n_clear, src_slots, dst_offsets,
                                              dst_slots, n_src, n_dst, min_slots, bitmap, n_words,
                                              verdict, dev_status);
    const int64_t n_items = (int64_t)(n_clear + n_src) * ps.piece_off[n_pools];
    if (n_items == 0) return launch_status();
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t grid = n_items < (int64_t)sms * 8 ? n_items : (int64_t)sms * 8;
    slot_copy_kernel<<<(unsigned)grid, kCopyThreads, 0, s>>>(ps, clear_slots, n_clear, src_slots,
                                                             dst_offsets, dst_slots, n_src,
                                                             verdict);
    return launch_status();
}

extern "C" const char* kda_status_string(kda_status st) {
    switch (st) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: null pointer, bad size or misaligned buffer";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: shape or dtype outside the supported set";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: a CUDA launch or runtime call failed";
    }
    return "KDA_ERR_UNKNOWN";
}

extern "C" int32_t kda_abi_version(void) { return 105; }

// ----------------------------------------------------------------------------
// Allocation-free variant.
//
// Some callers cannot hand the library a workspace: an engine that gives all
// device memory to its own pool allocator when it starts and forbids any other
// allocation afterwards, or a latency-critical path where a cudaMalloc (which
// may synchronise the device) is not acceptable.  kda_slot_copy_noalloc uses a
// fixed scratch array that lives in the library's own device memory instead.
// The array is sized for KDA_SLOT_COPY_NOALLOC_MAX_SLOTS slots; every GPU that
// loads the library holds it until the process exits.

namespace {

constexpr size_t kNoallocScratchBytes = 16 + ((size_t)KDA_SLOT_COPY_NOALLOC_MAX_SLOTS + 127) / 128 * 16;

static __device__ __align__(256) unsigned char g_slot_copy_scratch[kNoallocScratchBytes];

// A symbol's device address belongs to a CUDA context, not to a device: a context made
// after cudaDeviceReset, or a non-primary context the caller made current, has its own copy
// of the array.  Addresses are therefore cached under the current context's unique id
// (cuCtxGetId never reuses an id within a process, even when a context handle is reused).
constexpr int kCacheSlots = 64;
std::mutex g_scratch_mu;
unsigned long long g_cache_ctx[kCacheSlots] = {};  // 0 = empty (context ids start at 1)
void* g_cache_ptr[kCacheSlots] = {};
int g_cache_next = 0;

struct CtxFns {
    PFN_cuCtxGetCurrent_v4000 current = nullptr;
    PFN_cuCtxGetId_v12000 id = nullptr;
};

CtxFns lookup_ctx_fns() {
    CtxFns f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        f.current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        f.id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    return f;
}

// Unique id of the context current on this thread (made current by the runtime if none is).
kda_status current_context_id(unsigned long long* id) {
    static const CtxFns fns = lookup_ctx_fns();
    if (fns.current == nullptr || fns.id == nullptr) return KDA_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (fns.current(&ctx) != CUDA_SUCCESS) return KDA_ERR_CUDA;
    if (ctx == nullptr) {
        // no context yet on this thread: a runtime call that needs one makes the device's
        // primary context current (the lookup below is repeated under the lock anyway)
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_slot_copy_scratch) != cudaSuccess) return KDA_ERR_CUDA;
        if (fns.current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return KDA_ERR_CUDA;
    }
    if (fns.id(ctx, id) != CUDA_SUCCESS || *id == 0) return KDA_ERR_CUDA;
    return KDA_OK;
}

// Device address of the scratch array in the current context (looked up once per context,
// with that context current; the name alone is only a host-side stand-in).
kda_status scratch_address(void** out) {
    unsigned long long id = 0;
    const kda_status st = current_context_id(&id);
    if (st != KDA_OK) return st;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    for (int i = 0; i < kCacheSlots; ++i) {
        if (g_cache_ctx[i] == id) {
            *out = g_cache_ptr[i];
            return KDA_OK;
        }
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_slot_copy_scratch) != cudaSuccess || p == nullptr) return KDA_ERR_CUDA;
    g_cache_ctx[g_cache_next] = id;
    g_cache_ptr[g_cache_next] = p;
    g_cache_next = (g_cache_next + 1) % kCacheSlots;
    *out = p;
    return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_slot_copy_noalloc(const kda_pool_desc* pools, int32_t n_pools,
                                            const int32_t* clear_slots, int32_t n_clear,
                                            const int32_t* src_slots, const int32_t* dst_offsets,
                                            const int32_t* dst_slots, int32_t n_src, int32_t n_dst,
                                            int32_t* dev_status, void* stream) {
    KDA_REQUIRE(pools != nullptr && n_pools > 0 && n_pools <= KDA_MAX_POOLS, KDA_ERR_INVALID_ARG);
    int64_t min_slots = INT64_MAX;
    for (int i = 0; i < n_pools; ++i)
        min_slots = pools[i].num_slots < min_slots ? pools[i].num_slots : min_slots;
    // the disjointness bitmap covers slot ids below the smallest pool's size
    KDA_REQUIRE(min_slots <= KDA_SLOT_COPY_NOALLOC_MAX_SLOTS, KDA_ERR_UNSUPPORTED);
    void* scratch = nullptr;
    const kda_status st = scratch_address(&scratch);
    if (st != KDA_OK) return st;
    return kda_slot_copy(pools, n_pools, clear_slots, n_clear, src_slots, dst_offsets, dst_slots,
                         n_src, n_dst, scratch, kNoallocScratchBytes, dev_status, stream);
}
