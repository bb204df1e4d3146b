// pkv_attention.cu -- bf16 paged attention: the K/V pools are read with TMA tiles.
//
// TensorSharp "高级功能", section "原生分页注意力": attention of each sequence's
// query rows over K/V gathered from the paged block pool (with the per-head sink
// variant), and the TensorFold article, section "先记住一条铁律" (verify rows use
// the serial step's arithmetic; a batched row equals the row alone).  The kernels
// and the shared argument checks are in pkv_attention_impl.cuh.
#include <atomic>

#include "pkv_attention_tc.cuh"

// Which kernel serves the bf16 paths (decode, verify windows, draft trees, prefill chunks,
// the index-list gather): pkv_set_attention_kernel() chooses, process-wide, between the
// mma.sync kernel (the default) and the tcgen05 kernel of pkv_attention_tc.cuh.  Each keeps
// every row's arithmetic a function of its own sequence, but their arithmetic differs, so a
// row computed by one is not bit-identical to the row computed by the other.  The mma.sync
// kernel is the default because it is faster at these row counts: a tcgen05 MMA of 128 keys
// costs about 55 SM cycles for any N up to 64, and one softmax pipeline per SM (its 64 KB
// K / V stages leave room for no second) cannot hide the latency that many small mma.sync
// CTAs hide.  The quantised pools always use the mma.sync kernel.
static std::atomic<int> g_attention_kernel{PKV_KERNEL_MMA_SYNC};

namespace pkv {
namespace {

// Unit-pass arguments of an attention call; num_src = sequences, or query rows for the
// index-list gather.
UnitPassParams unit_pass_params(const AttnParams &prm, int num_src)
{
    UnitPassParams up;
    memset(&up, 0, sizeof up);
    up.q_starts = prm.q_starts;
    up.context_lens = prm.context_lens;
    up.key_counts = prm.key_counts;
    up.units = const_cast<int4 *>(prm.units);
    up.ctl = prm.unit_ctl;
    up.status = prm.status;
    up.num_src = num_src;
    up.num_seqs = prm.num_seqs;
    up.total_rows = prm.total_rows;
    up.max_rows = prm.max_rows;
    up.group = prm.group;
    up.num_kv_heads = prm.num_kv_heads;
    up.max_keys = prm.max_keys;
    up.L_cap = (int)std::min<long long>(prm.max_context_len, (long long)prm.max_blocks_per_seq * prm.block_size);
    up.n_max = prm.n_max;
    up.unit_cap = prm.unit_cap;
    return up;
}

int tc_limits(const char *who, int num_src, int n_max)
{
    if (num_src > kTcMaxSeqs)
        return set_error(PKV_ERR_UNSUPPORTED, "%s: %d sequences (or gather rows) in one call; at most %d", who,
                         num_src, kTcMaxSeqs);
    if (n_max > kTcMaxSplits)
        return set_error(PKV_ERR_UNSUPPORTED, "%s: contexts up to %d tokens in one call", who,
                         kTcMaxSplits * kSplitTokens);
    return PKV_OK;
}

// ---------------------------------------------------------------- host side --
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2-D map over a pool seen as rows of head_dim bf16: [num_blocks*H_kv*block_size][head_dim],
// box = 64 columns (128 B, the swizzle span) x block_size rows.
int make_pool_map(CUtensorMap *map, void *base, const pkv_pool &pool)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return set_error(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t rows = (cuuint64_t)pool.num_blocks * pool.num_kv_heads * pool.block_size;
    cuuint64_t dims[2] = {(cuuint64_t)pool.head_dim, rows};
    cuuint64_t strides[1] = {(cuuint64_t)pool.head_dim * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)pool.block_size};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return PKV_OK;
}

int launch_bf16(const PoolView &pv, AttnParams &prm, int rows, long long pairs, int n_max, cudaStream_t st)
{
    pkv_pool pool;
    pool.k_pool = const_cast<void *>(pv.k_pool);
    pool.v_pool = const_cast<void *>(pv.v_pool);
    pool.num_blocks = pv.num_blocks;
    pool.block_size = pv.block_size;
    pool.num_kv_heads = pv.num_kv_heads;
    pool.head_dim = pv.head_dim;
    CUtensorMap mk, mv;
    int rc = make_pool_map(&mk, pool.k_pool, pool);
    if (rc)
        return rc;
    rc = make_pool_map(&mv, pool.v_pool, pool);
    if (rc)
        return rc;
    const int D = pv.head_dim, BS = pv.block_size;
    if (g_attention_kernel.load(std::memory_order_relaxed) == PKV_KERNEL_TCGEN05) {
        rc = tc_limits("paged attention", prm.num_seqs, n_max);
        if (rc)
            return rc;
        const UnitPassParams up = unit_pass_params(prm, prm.num_seqs);
        if (D == 64 && BS == 16) return launch_tc<64, 16, false>(rows, mk, mv, prm, up, st);
        if (D == 64 && BS == 32) return launch_tc<64, 32, false>(rows, mk, mv, prm, up, st);
        if (D == 128 && BS == 16) return launch_tc<128, 16, false>(rows, mk, mv, prm, up, st);
        return launch_tc<128, 32, false>(rows, mk, mv, prm, up, st);
    }
    if (D == 64 && BS == 16) return launch_d_bs<64, 16, 16, true>(rows, mk, mv, prm, pairs, n_max, st);
    if (D == 64 && BS == 32) return launch_d_bs<64, 32, 16, true>(rows, mk, mv, prm, pairs, n_max, st);
    if (D == 128 && BS == 16) return launch_d_bs<128, 16, 16, true>(rows, mk, mv, prm, pairs, n_max, st);
    return launch_d_bs<128, 32, 16, true>(rows, mk, mv, prm, pairs, n_max, st);
}

#ifndef PKV_GATHER_DEEP
#define PKV_GATHER_DEEP 0
#endif
// Index-list gather: one unit per (query row, KV head); the grid's second dimension
// runs over 512-entry slices of the longest list.
template <int D>
int launch_gather_d(int rows, AttnParams prm, long long pairs, int n_max, cudaStream_t st)
{
    CUtensorMap none;   // the gather copies rows with cp.async, not tensor maps
    memset(&none, 0, sizeof none);
    const int per_cta = rows <= 8 ? 8 : 8 * PKV_WIDE_NN * PKV_WIDE_NMT;
    prm.row_groups = (rows + per_cta - 1) / per_cta;
    const long long gx = pairs * prm.row_groups;
    if (gx > 0x7fffffffLL || n_max > 65535)
        return set_error(PKV_ERR_SHAPE, "paged_attention_forward_gather: grid too large");
    const dim3 grid((unsigned)gx, (unsigned)n_max);
    // (a deeper ring was measured slower here: 1024 CTAs need the occupancy more than the
    // bytes in flight; PKV_GATHER_DEEP=1 selects it)
    if (rows <= 8)
        return launch_t<D, 16, 1, 1, false, 16, true, PKV_GATHER_DEEP != 0>(none, none, prm, grid, st);
    return launch_t<D, 16, PKV_WIDE_NN, PKV_WIDE_NMT, false, 16, true, PKV_GATHER_DEEP != 0>(none, none, prm, grid, st);
}

int launch_gather(const PoolView &pv, AttnParams &prm, int rows, long long /*pairs*/, int n_max, cudaStream_t st)
{
    const long long pairs = (long long)prm.total_rows * pv.num_kv_heads;
    if (g_attention_kernel.load(std::memory_order_relaxed) == PKV_KERNEL_TCGEN05) {
        int rc = tc_limits("paged_attention_forward_gather", prm.total_rows, n_max);
        if (rc)
            return rc;
        CUtensorMap none;
        memset(&none, 0, sizeof none);
        const UnitPassParams up = unit_pass_params(prm, prm.total_rows);
        if (pv.head_dim == 64)
            return launch_tc<64, 16, true>(rows, none, none, prm, up, st);
        return launch_tc<128, 16, true>(rows, none, none, prm, up, st);
    }
    if (pv.head_dim == 64)
        return launch_gather_d<64>(rows, prm, pairs, n_max, st);
    return launch_gather_d<128>(rows, prm, pairs, n_max, st);
}

int attention_impl(const char *who, const pkv_pool *pool, const void *q, const int32_t *q_starts,
                   const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                   int32_t num_seqs, int32_t total_q_rows, int32_t max_context_len,
                   int32_t max_q_rows_per_seq, int32_t num_q_heads, const int32_t *kv_head_of_q_head,
                   const float *sinks, int32_t causal, const uint32_t *tree_masks, float scale, void *out,
                   int32_t out_dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    if (!pool)
        return set_error(PKV_ERR_NULL, "%s: pool is NULL", who);
    PoolView pv = {pool->num_blocks, pool->block_size, pool->num_kv_heads, pool->head_dim, 16,
                   pool->k_pool, pool->v_pool, nullptr};
    return attention_run(who, pv, q, q_starts, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                         total_q_rows, max_context_len, max_q_rows_per_seq, num_q_heads, kv_head_of_q_head,
                         sinks, causal, tree_masks, scale, out, out_dtype, workspace, workspace_bytes, stream,
                         launch_bf16);
}

}  // namespace
}  // namespace pkv

extern "C" size_t paged_attention_workspace_size(int32_t num_seqs, int32_t total_q_rows,
                                                 int32_t num_q_heads, int32_t num_kv_heads,
                                                 int32_t head_dim, int32_t max_context_len)
{
    if (num_seqs < 0 || total_q_rows < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return 0;
    return pkv::ws_layout(num_seqs, total_q_rows, num_q_heads, num_kv_heads, head_dim, max_context_len).total;
}

extern "C" int paged_attention_workspace_init(void *workspace, size_t workspace_bytes, void *stream)
{
    pkv::clear_error();
    if (!workspace)
        return pkv::set_error(PKV_ERR_NULL, "paged_attention_workspace_init: workspace is NULL");
    return pkv::check_cuda(cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)),
                           "paged_attention_workspace_init");
}

extern "C" int paged_attention_forward(const pkv_pool *pool, const void *q, const int32_t *q_starts,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       const int32_t *context_lens, int32_t num_seqs,
                                       int32_t total_q_rows, int32_t max_context_len,
                                       int32_t max_q_rows_per_seq, int32_t num_q_heads,
                                       const int32_t *kv_head_of_q_head, const float *sinks,
                                       int32_t causal, float scale, void *out, int32_t out_dtype,
                                       void *workspace, size_t workspace_bytes, void *stream)
{
    pkv::clear_error();
    return pkv::attention_impl("paged_attention_forward", pool, q, q_starts, block_tables, max_blocks_per_seq,
                               context_lens, num_seqs, total_q_rows, max_context_len, max_q_rows_per_seq,
                               num_q_heads, kv_head_of_q_head, sinks, causal, nullptr, scale, out, out_dtype,
                               workspace, workspace_bytes, stream);
}

extern "C" int paged_tree_attention_forward(const pkv_pool *pool, const void *q, const int32_t *q_starts,
                                            const int32_t *block_tables, int32_t max_blocks_per_seq,
                                            const int32_t *context_lens, int32_t num_seqs,
                                            int32_t total_q_rows, int32_t max_context_len,
                                            int32_t max_q_rows_per_seq, int32_t num_q_heads,
                                            const int32_t *kv_head_of_q_head, const float *sinks,
                                            const uint32_t *tree_masks, float scale, void *out,
                                            int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                            void *stream)
{
    pkv::clear_error();
    if (num_seqs > 0 && total_q_rows > 0 && !tree_masks)
        return pkv::set_error(PKV_ERR_NULL, "paged_tree_attention_forward: tree_masks is NULL");
    if (max_q_rows_per_seq > 32)
        return pkv::set_error(PKV_ERR_UNSUPPORTED,
                              "paged_tree_attention_forward: at most 32 verify rows per sequence (got %d)",
                              max_q_rows_per_seq);
    return pkv::attention_impl("paged_tree_attention_forward", pool, q, q_starts, block_tables,
                               max_blocks_per_seq, context_lens, num_seqs, total_q_rows, max_context_len,
                               max_q_rows_per_seq, num_q_heads, kv_head_of_q_head, sinks, 0, tree_masks, scale,
                               out, out_dtype, workspace, workspace_bytes, stream);
}

// ------------------------------------------------ allocation-free variant --
// Some callers cannot call cudaMalloc: code that runs inside a CUDA-graph
// capture that must not allocate, inference runtimes that hand out all device
// memory up front from their own arena, and plug-in hosts whose allocator is
// not reachable from this library.  For them paged_attention_forward_noalloc
// runs the same kernel with its workspace in this fixed device array instead of
// a caller-provided buffer.  The array is part of the loaded module, so every
// GPU that loads the library holds PKV_NOALLOC_SCRATCH_BYTES of it until the
// process exits.
static __device__ __align__(256) uint8_t g_pkv_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace pkv {
namespace {
// Device address of the scratch array in the caller's current context.  In host code
// the array's name is only a host-side stand-in, never a device address, so it is
// looked up with cudaGetSymbolAddress -- on every call, with the caller's device and
// context current: each context (a new one after cudaDeviceReset, or a driver-API
// context other than the primary one) loads the module, and the array with it, at its
// own address, so an address kept from an earlier call could name unmapped memory.
// The lookup is a host-side query, not a stream operation.
int noalloc_scratch(uint8_t **ptr)
{
    void *p = nullptr;
    const int rc = check_cuda(cudaGetSymbolAddress(&p, g_pkv_noalloc_scratch),
                              "cudaGetSymbolAddress of the allocation-free scratch");
    if (rc)
        return rc;
    *ptr = static_cast<uint8_t *>(p);
    return PKV_OK;
}
}  // namespace
}  // namespace pkv

extern "C" int paged_attention_forward_noalloc(const pkv_pool *pool, const void *q, const int32_t *q_starts,
                                               const int32_t *block_tables, int32_t max_blocks_per_seq,
                                               const int32_t *context_lens, int32_t num_seqs,
                                               int32_t total_q_rows, int32_t max_context_len,
                                               int32_t max_q_rows_per_seq, int32_t num_q_heads,
                                               const int32_t *kv_head_of_q_head, const float *sinks,
                                               int32_t causal, float scale, void *out, int32_t out_dtype,
                                               void *stream)
{
    using namespace pkv;
    clear_error();
    if (!pool)
        return set_error(PKV_ERR_NULL, "paged_attention_forward_noalloc: pool is NULL");
    if (num_seqs == 0 || total_q_rows == 0)
        return paged_attention_forward(pool, q, q_starts, block_tables, max_blocks_per_seq, context_lens,
                                       num_seqs, total_q_rows, max_context_len, max_q_rows_per_seq,
                                       num_q_heads, kv_head_of_q_head, sinks, causal, scale, out, out_dtype,
                                       nullptr, 0, stream);
    const size_t need = paged_attention_workspace_size(num_seqs, total_q_rows, num_q_heads, pool->num_kv_heads,
                                                       pool->head_dim, max_context_len);
    if (need == 0)
        return set_error(PKV_ERR_SHAPE, "paged_attention_forward_noalloc: invalid sizes");
    if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES)
        return set_error(PKV_ERR_WORKSPACE,
                         "paged_attention_forward_noalloc: these sizes need %zu bytes of scratch but the "
                         "built-in scratch holds %zu; use paged_attention_forward with a caller workspace",
                         need, (size_t)PKV_NOALLOC_SCRATCH_BYTES);
    uint8_t *scratch = nullptr;
    int rc = noalloc_scratch(&scratch);
    if (rc)
        return rc;
    return paged_attention_forward(pool, q, q_starts, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                   total_q_rows, max_context_len, max_q_rows_per_seq, num_q_heads,
                                   kv_head_of_q_head, sinks, causal, scale, out, out_dtype, scratch,
                                   (size_t)PKV_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" int paged_attention_forward_gather(const pkv_pool *pool, const void *q, const int32_t *q_starts,
                                              const int32_t *block_tables, int32_t max_blocks_per_seq,
                                              const int32_t *context_lens, int32_t num_seqs, int32_t total_q_rows,
                                              const int32_t *key_idx, const int32_t *key_counts, int32_t max_keys,
                                              int32_t num_q_heads, const int32_t *kv_head_of_q_head,
                                              const float *sinks, float scale, void *out, int32_t out_dtype,
                                              void *workspace, size_t workspace_bytes, void *stream)
{
    using namespace pkv;
    clear_error();
    const char *who = "paged_attention_forward_gather";
    if (!pool)
        return set_error(PKV_ERR_NULL, "%s: pool is NULL", who);
    if (max_keys < 0)
        return set_error(PKV_ERR_SHAPE, "%s: max_keys %d is negative", who, max_keys);
    if (num_seqs > 0 && total_q_rows > 0 && max_keys > 0 && (!key_idx || !key_counts))
        return set_error(PKV_ERR_NULL, "%s: key_idx and key_counts are required", who);
    if (num_seqs > 0 && total_q_rows > 0 && max_keys == 0)
        return set_error(PKV_ERR_SHAPE, "%s: max_keys must be positive", who);
    PoolView pv = {pool->num_blocks, pool->block_size, pool->num_kv_heads, pool->head_dim, 16,
                   pool->k_pool, pool->v_pool, nullptr};
    pv.key_idx = key_idx;
    pv.key_counts = key_counts;
    pv.max_keys = max_keys;
    return attention_run(who, pv, q, q_starts, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                         total_q_rows, max_keys, 1, num_q_heads, kv_head_of_q_head, sinks, 0, nullptr, scale, out,
                         out_dtype, workspace, workspace_bytes, stream, launch_gather);
}

extern "C" int pkv_set_attention_kernel(int32_t which)
{
    pkv::clear_error();
    if (which != PKV_KERNEL_MMA_SYNC && which != PKV_KERNEL_TCGEN05)
        return pkv::set_error(PKV_ERR_SHAPE, "pkv_set_attention_kernel: unknown kernel %d", which);
    g_attention_kernel.store(which, std::memory_order_relaxed);
    return PKV_OK;
}
