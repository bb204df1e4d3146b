// pkv_append.cu -- paged K/V scatter-append.
//
// TensorSharp "高级功能", "批量前向" paragraph: the batched forward pairs its
// projections with a paged K/V scatter-write.  New token i of sequence s sits at
// position p = context_lens_old[s] + i and lands in slot p % block_size of block
// block_tables[s][p / block_size], for every KV head, in both pools.
//
// One warp per (new row, KV head): the K row and the V row (head_dim bf16 each)
// are moved with 16-byte vector loads/stores.  Pure data movement, bit-exact.
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ __forceinline__ int find_seq(const int32_t *__restrict__ starts, int num_seqs, int row)
{
    // last s with starts[s] <= row  (starts is non-decreasing, starts[0] == 0)
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(starts + mid) <= row)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(128)
paged_kv_append_kernel(uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool,
                       const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                       const int32_t *__restrict__ block_tables, int max_blocks_per_seq,
                       const int32_t *__restrict__ context_lens_old,
                       const int32_t *__restrict__ new_starts, int num_seqs, int total_rows,
                       int num_blocks, int block_size, int num_kv_heads, int vecs_per_row,
                       int32_t *__restrict__ status)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int row = warp / num_kv_heads;
    const int h = warp - row * num_kv_heads;
    if (row >= total_rows)
        return;
    const int s = find_seq(new_starts, num_seqs, row);
    const long long p = (long long)__ldg(context_lens_old + s) + (row - __ldg(new_starts + s));
    const long long logical = p / block_size;
    if (p < 0 || logical >= max_blocks_per_seq) {
        if (lane == 0)
            atomicOr(status, PKV_DEV_TABLE_OVERRUN);
        return;
    }
    const int blk = __ldg(block_tables + (long long)s * max_blocks_per_seq + logical);
    if (blk < 0 || blk >= num_blocks) {
        if (lane == 0)
            atomicOr(status, PKV_DEV_BAD_BLOCK);
        return;
    }
    const size_t dst = ((((size_t)blk * num_kv_heads) + h) * block_size + (size_t)(p % block_size)) *
                       vecs_per_row;
    const size_t src = ((size_t)row * num_kv_heads + h) * vecs_per_row;
    for (int i = lane; i < vecs_per_row; i += 32) {
        k_pool[dst + i] = __ldg(k_new + src + i);
        v_pool[dst + i] = __ldg(v_new + src + i);
    }
}

}  // namespace
}  // namespace pkv

extern "C" int paged_kv_append(const pkv_pool *pool, const int32_t *block_tables,
                               int32_t max_blocks_per_seq, const int32_t *context_lens_old,
                               const int32_t *new_starts, const void *k_new, const void *v_new,
                               int32_t num_seqs, int32_t total_new_rows, void *stream)
{
    using namespace pkv;
    clear_error();
    if (!pool)
        return set_error(PKV_ERR_NULL, "paged_kv_append: pool is NULL");
    if (num_seqs < 0 || total_new_rows < 0 || max_blocks_per_seq <= 0)
        return set_error(PKV_ERR_SHAPE, "paged_kv_append: negative sizes or max_blocks_per_seq <= 0");
    if (pool->num_blocks <= 0 || pool->block_size <= 0 || pool->num_kv_heads <= 0 || pool->head_dim <= 0)
        return set_error(PKV_ERR_SHAPE, "paged_kv_append: pool dimensions must be positive");
    if (pool->head_dim % 8 != 0)
        return set_error(PKV_ERR_UNSUPPORTED, "paged_kv_append: head_dim %d is not a multiple of 8",
                         pool->head_dim);
    if (total_new_rows == 0 || num_seqs == 0)
        return PKV_OK;
    if (!pool->k_pool || !pool->v_pool || !block_tables || !context_lens_old || !new_starts || !k_new ||
        !v_new)
        return set_error(PKV_ERR_NULL, "paged_kv_append: a required pointer is NULL");
    if (!aligned16(pool->k_pool) || !aligned16(pool->v_pool) || !aligned16(k_new) || !aligned16(v_new))
        return set_error(PKV_ERR_ALIGN, "paged_kv_append: pools and k_new/v_new must be 16-byte aligned");
    int32_t *status = device_status_word();
    if (!status)
        return set_error(PKV_ERR_CUDA, "paged_kv_append: no device status word");
    const long long warps = (long long)total_new_rows * pool->num_kv_heads;
    const long long blocks = (warps * 32 + 127) / 128;
    if (blocks > 0x7fffffffLL)
        return set_error(PKV_ERR_SHAPE, "paged_kv_append: too many rows");
    paged_kv_append_kernel<<<(unsigned)blocks, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4 *>(pool->k_pool), static_cast<uint4 *>(pool->v_pool),
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), block_tables,
        max_blocks_per_seq, context_lens_old, new_starts, num_seqs, total_new_rows, pool->num_blocks,
        pool->block_size, pool->num_kv_heads, pool->head_dim / 8, status);
    return check_cuda(cudaGetLastError(), "paged_kv_append launch");
}
