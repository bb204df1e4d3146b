// pkv_alloc.cu -- block allocation with prefix sharing on the device.
//
// TensorSharp "高级功能", section "连续批处理与分页 KV 缓存": KV blocks of a fixed size
// come from one shared pool, and every full block is content-hashed so that identical
// prefixes map to the same physical blocks; a partial block is never shared.  The keys
// come from paged_block_hashes (chained, so a key names its block's whole prefix).
//
// The result is defined as the sequential engine step (sequences in order, blocks in
// order, the free stack popped from its top), and the kernels reproduce it exactly
// whatever order their threads run in:
//  1. probe: one thread per table entry (s, j) to allocate.  A full block looks its key
//     up in the open-addressing index (linear probing, lock-free insert by CAS).  A key
//     that already has a block is a hit.  A key without one (new in this call, or whose
//     allocation failed in an earlier call) is pending: every pending entry of the key
//     takes atomicMax on the slot's id field with -(2 + e), e = s * max_blocks + j, so
//     the field ends at -(2 + first entry in sequential order): that entry owns the key.
//  2. rank: one CTA scans the entries in sequential order; owners and private blocks
//     take the free stack's next ids (rank k -> free_ids[F - 1 - k]); owners write their
//     id into the slot; the stack's count drops by the pops.
//  3. resolve: every entry reads its id (hits and duplicates from the slot), bumps the
//     slot's reference count, and writes its table entry and fresh flag.
// Reference counts are sums, so their order does not matter; which slot a key lands in
// depends on the insertion race, but the key -> (id, refcount) map does not.
#include <climits>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr uint64_t kKeyEmpty = PKV_BLOCK_KEY_EMPTY;
constexpr int32_t kIdNone = INT_MIN;   // an empty slot, or a key without a block
constexpr int kRankThreads = 1024;

enum : int32_t { kSkip = 0, kHit = 1, kPending = 2, kOwner = 3, kPrivate = 4 };

__device__ __forceinline__ uint32_t home_slot(uint64_t key, uint32_t mask)
{
    return (uint32_t)((key * 0x9E3779B97F4A7C15ull) >> 32) & mask;   // Fibonacci hashing
}

// Geometry of sequence s's allocation: blocks [first, nb), of which those below nk are full.
__device__ __forceinline__ void seq_range(const int32_t *context_lens, const int32_t *first_block, int s,
                                          int block_size, int max_blocks, int &first, int &nb, int &nk,
                                          bool &overrun)
{
    long long L = __ldg(context_lens + s);
    L = L < 0 ? 0 : L;
    long long b = (L + block_size - 1) / block_size, k = L / block_size;
    overrun = b > max_blocks;
    if (overrun)
        b = max_blocks;
    if (k > b)
        k = b;
    nb = (int)b;
    nk = (int)k;
    first = max(__ldg(first_block + s), 0);
}

__global__ void index_init_kernel(uint64_t *keys, int32_t *ids, int32_t *refs, int32_t capacity,
                                  int32_t *free_count, int32_t num_free)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < capacity; i += gridDim.x * blockDim.x) {
        keys[i] = kKeyEmpty;
        ids[i] = kIdNone;
        refs[i] = 0;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *free_count = num_free;
}

__global__ void alloc_probe_kernel(pkv_block_index ix, const uint64_t *__restrict__ block_keys,
                                   const int32_t *__restrict__ context_lens, const int32_t *__restrict__ first_block,
                                   int num_seqs, int block_size, int max_blocks, int32_t *kind_ws, int32_t *val_ws,
                                   int32_t *status)
{
    const long long n = (long long)num_seqs * max_blocks;
    const uint32_t mask = (uint32_t)ix.capacity - 1u;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        const int s = (int)(e / max_blocks), j = (int)(e - (long long)s * max_blocks);
        int first, nb, nk;
        bool overrun;
        seq_range(context_lens, first_block, s, block_size, max_blocks, first, nb, nk, overrun);
        if (overrun && j == 0)
            atomicOr(status, PKV_DEV_TABLE_OVERRUN);
        int32_t kind = kSkip, val = 0;
        if (j >= first && j < nb) {
            const uint64_t key = j < nk ? __ldg(reinterpret_cast<const unsigned long long *>(block_keys) + e)
                                        : kKeyEmpty;
            kind = kPrivate;
            if (key != kKeyEmpty) {
                // linear probing; an empty slot is claimed by CAS (a concurrent insert of the
                // same key finds it, another key moves on)
                uint32_t slot = home_slot(key, mask);
                int found = -1;
                for (int32_t probe = 0; probe < ix.capacity; ++probe) {
                    unsigned long long *kp = reinterpret_cast<unsigned long long *>(ix.keys) + slot;
                    unsigned long long k = *reinterpret_cast<volatile unsigned long long *>(kp);
                    if (k == kKeyEmpty)
                        k = atomicCAS(kp, (unsigned long long)kKeyEmpty, (unsigned long long)key);
                    if (k == kKeyEmpty || k == key) {
                        found = (int)slot;
                        break;
                    }
                    slot = (slot + 1u) & mask;
                }
                if (found < 0) {
                    atomicOr(status, PKV_DEV_INDEX_FULL);   // no slot: the block stays private
                } else {
                    // ids >= 0 exist only from earlier calls while this kernel runs
                    const int32_t id = *reinterpret_cast<volatile int32_t *>(ix.block_ids + found);
                    if (id >= 0) {
                        kind = kHit;
                    } else {
                        kind = kPending;
                        atomicMax(ix.block_ids + found, -(int32_t)(2 + e));
                    }
                    val = found;
                }
            }
        }
        kind_ws[e] = kind;
        val_ws[e] = val;
    }
}

// One CTA: entries in sequential order, each thread a contiguous run of them.
__global__ void __launch_bounds__(kRankThreads) alloc_rank_kernel(pkv_block_index ix, long long n,
                                                                 int32_t *kind_ws, int32_t *val_ws, int32_t *status)
{
    __shared__ long long warp_sum[kRankThreads / 32];
    __shared__ long long total_s;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const long long per = (n + kRankThreads - 1) / kRankThreads;
    const long long e0 = min(n, (long long)t * per), e1 = min(n, e0 + per);
    const int32_t F = *ix.free_count;
    // owners: the pending entry whose -(2 + e) won the slot's atomicMax
    long long cnt = 0;
    for (long long e = e0; e < e1; ++e) {
        const int32_t k = kind_ws[e];
        if (k == kPending && ix.block_ids[val_ws[e]] == -(int32_t)(2 + e)) {
            kind_ws[e] = kOwner;
            ++cnt;
        } else if (k == kPrivate) {
            ++cnt;
        }
    }
    // exclusive scan of the per-thread counts
    long long x = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off)
            x += y;
    }
    if (lane == 31)
        warp_sum[warp] = x;
    __syncthreads();   // also: every owner test above is done before any slot is written
    if (warp == 0) {
        long long w = lane < kRankThreads / 32 ? warp_sum[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off)
                w += y;
        }
        if (lane < kRankThreads / 32)
            warp_sum[lane] = w;   // inclusive over warps
        if (lane == kRankThreads / 32 - 1)
            total_s = w;
    }
    __syncthreads();
    long long rank = (warp > 0 ? warp_sum[warp - 1] : 0) + x - cnt;
    for (long long e = e0; e < e1; ++e) {
        const int32_t k = kind_ws[e];
        if (k != kOwner && k != kPrivate)
            continue;
        const int32_t id = rank < F ? ix.free_ids[F - 1 - rank] : -1;
        ++rank;
        if (k == kOwner)
            ix.block_ids[val_ws[e]] = id >= 0 ? id : kIdNone;   // a key whose pop failed keeps no block
        else
            val_ws[e] = id;
    }
    if (t == 0) {
        const long long P = total_s;
        *ix.free_count = P < F ? (int32_t)(F - P) : 0;
        if (P > F)
            atomicOr(status, PKV_DEV_OUT_OF_BLOCKS);
    }
}

__global__ void alloc_resolve_kernel(pkv_block_index ix, long long n, const int32_t *kind_ws, const int32_t *val_ws,
                                     int32_t *block_tables, int32_t *fresh)
{
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        const int32_t k = kind_ws[e], v = val_ws[e];
        int32_t f = 0;
        if (k != kSkip) {
            int32_t id;
            if (k == kPrivate) {
                id = v;
                f = id >= 0;
            } else {
                id = ix.block_ids[v];
                if (id >= 0) {
                    atomicAdd(ix.refcounts + v, 1);
                    f = k == kOwner;
                } else {
                    id = -1;
                }
            }
            block_tables[e] = id;
        }
        if (fresh)
            fresh[e] = f;
    }
}

int check_index(const char *who, const pkv_block_index *ix)
{
    if (!ix)
        return set_error(PKV_ERR_NULL, "%s: index is NULL", who);
    if (!ix->keys || !ix->block_ids || !ix->refcounts || !ix->free_count)
        return set_error(PKV_ERR_NULL, "%s: index arrays are required", who);
    if (ix->capacity < 1 || (ix->capacity & (ix->capacity - 1)))
        return set_error(PKV_ERR_SHAPE, "%s: capacity %d is not a positive power of two", who, ix->capacity);
    if ((reinterpret_cast<uintptr_t>(ix->keys) & 7u) || (reinterpret_cast<uintptr_t>(ix->block_ids) & 3u) ||
        (reinterpret_cast<uintptr_t>(ix->refcounts) & 3u) || (reinterpret_cast<uintptr_t>(ix->free_ids) & 3u) ||
        (reinterpret_cast<uintptr_t>(ix->free_count) & 3u))
        return set_error(PKV_ERR_ALIGN, "%s: index arrays must be aligned to their element size", who);
    return PKV_OK;
}

size_t alloc_ws_bytes(long long n) { return round_up((size_t)n * 2 * sizeof(int32_t), 256); }

}  // namespace
}  // namespace pkv

extern "C" int paged_block_index_init(const pkv_block_index *ix, int32_t num_free, void *stream)
{
    using namespace pkv;
    clear_error();
    int rc = check_index("paged_block_index_init", ix);
    if (rc)
        return rc;
    if (num_free < 0 || (num_free > 0 && !ix->free_ids))
        return set_error(PKV_ERR_SHAPE, "paged_block_index_init: num_free %d needs free_ids", num_free);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int grid = (int)std::min<long long>((ix->capacity + 255) / 256, 4LL * sm_count());
    index_init_kernel<<<grid, 256, 0, st>>>(ix->keys, ix->block_ids, ix->refcounts, ix->capacity, ix->free_count,
                                            num_free);
    return check_cuda(cudaGetLastError(), "paged_block_index_init: launch");
}

extern "C" size_t paged_block_allocate_workspace_size(int32_t num_seqs, int32_t max_blocks_per_seq)
{
    if (num_seqs < 0 || max_blocks_per_seq < 0)
        return 0;
    return pkv::alloc_ws_bytes((long long)num_seqs * max_blocks_per_seq);
}

extern "C" int paged_block_allocate(const pkv_block_index *ix, const uint64_t *block_keys,
                                    const int32_t *context_lens, const int32_t *first_block, int32_t num_seqs,
                                    int32_t block_size, int32_t max_blocks_per_seq, int32_t *block_tables,
                                    int32_t *fresh, void *workspace, size_t workspace_bytes, void *stream)
{
    using namespace pkv;
    clear_error();
    const char *who = "paged_block_allocate";
    int rc = check_index(who, ix);
    if (rc)
        return rc;
    if (num_seqs < 0 || max_blocks_per_seq < 0)
        return set_error(PKV_ERR_SHAPE, "%s: negative size", who);
    if (block_size < 1)
        return set_error(PKV_ERR_SHAPE, "%s: block_size %d must be positive", who, block_size);
    const long long n = (long long)num_seqs * max_blocks_per_seq;
    if (n == 0)
        return PKV_OK;
    if (n > INT_MAX - 2)
        return set_error(PKV_ERR_UNSUPPORTED, "%s: num_seqs x max_blocks_per_seq above 2^31 - 3", who);
    if (!block_keys || !context_lens || !first_block || !block_tables || !workspace)
        return set_error(PKV_ERR_NULL, "%s: a required pointer is NULL", who);
    if ((reinterpret_cast<uintptr_t>(block_keys) & 7u) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(fresh) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return set_error(PKV_ERR_ALIGN, "%s: keys 8-byte, tables / fresh 4-byte, workspace 256-byte aligned", who);
    if (workspace_bytes < alloc_ws_bytes(n))
        return set_error(PKV_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", who, workspace_bytes,
                         alloc_ws_bytes(n));
    int32_t *status = device_status_word();
    if (!status)
        return set_error(PKV_ERR_CUDA, "%s: device status word unavailable", who);
    int32_t *kind_ws = static_cast<int32_t *>(workspace);
    int32_t *val_ws = kind_ws + n;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int grid = (int)std::min<long long>((n + 255) / 256, 8LL * sm_count());
    alloc_probe_kernel<<<grid, 256, 0, st>>>(*ix, block_keys, context_lens, first_block, num_seqs, block_size,
                                             max_blocks_per_seq, kind_ws, val_ws, status);
    rc = check_cuda(cudaGetLastError(), "paged_block_allocate: probe launch");
    if (rc)
        return rc;
    alloc_rank_kernel<<<1, kRankThreads, 0, st>>>(*ix, n, kind_ws, val_ws, status);
    rc = check_cuda(cudaGetLastError(), "paged_block_allocate: rank launch");
    if (rc)
        return rc;
    alloc_resolve_kernel<<<grid, 256, 0, st>>>(*ix, n, kind_ws, val_ws, block_tables, fresh);
    return check_cuda(cudaGetLastError(), "paged_block_allocate: resolve launch");
}
