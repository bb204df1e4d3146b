// pkv_attention_quant.cu -- quantised KV blocks: the quantising scatter-append and
// attention over the record pool.
//
// TensorSharp "高级功能", section "内存优化", the KV block codec item: blocks may be
// compressed in place to 8, 4 or 2 bits per value (Q8 / Q4 / Q2), trading a small
// accuracy cost for the footprint.  The codec built here (the pages give none): each
// (token, KV head) row of head_dim values gets one float32 scale s = max|x| / Q
// (Q = 2^(bits-1) - 1: 127, 7 or 1) and codes c = clamp(rint(x / s), -Q, Q), every step
// a correctly rounded float32 operation; the value read back is c * s.  The record
// layout (pkv.h) keeps each (block, KV head) in one contiguous record, so the
// attention kernel fetches a block with a single bulk copy.
// Splits of quantised records are 1024 keys (a build-time constant of this file,
// PKV_QUANT_SPLIT_TOKENS): a record's split CTA pays its start-up (length, block
// table and q loads, the first copies) and its key-share merge once per 1024 keys
// instead of per 512.  Measured on GB300 against 512-key splits: a Q8 cb_mix call
// 233 -> 225 us, Q4 236 -> 214 us, Q8 verify windows 325 -> 294 us, sinks_scale
// Q8 253 -> 217 us; the smallest calls (4 sequences of about 800 keys) lose about
// a microsecond.  Verify rows and decode rows of a codec share it, so every rule of
// bit identity holds within the codec; the workspace needed is at most what
// paged_attention_workspace_size returns.
#ifndef PKV_QUANT_SPLIT_TOKENS
#define PKV_QUANT_SPLIT_TOKENS 1024
#endif
#undef PKV_SPLIT_TOKENS
#define PKV_SPLIT_TOKENS PKV_QUANT_SPLIT_TOKENS
#include "pkv_attention_impl.cuh"

namespace pkv {
namespace {

// Byte of a record holding the code of (slot t, dim i): K section, then V section
// (for 4-bit codes the byte of the nibble; the nibble pairs dims i and i + 8; for
// 2-bit codes the byte of the bit pair, shared by dims i, i + 8, i + 16, i + 24 for K
// and by dims i, i + 8, i + 16, i + 24 of the same row half for V).
template <int BITS>
__device__ __forceinline__ uint32_t k_code_byte(int t, int i, int D)
{
    const int mt = t >> 4, g = (t & 15) >> 1, r = t & 1;
    const int j = i >> 4, s = i & 15, c = (s & 7) >> 1, h = s >> 3, e = s & 1, u = 4 * g + c;
    if constexpr (BITS == 8)
        return ((mt * (D / 32) + (j >> 1)) * 32 + u) * 16 + ((j & 1) * 2 + r) * 4 + h + 2 * e;
    else if constexpr (BITS == 2)
        return (mt * 32 + u) * (D / 8) + (j >> 1) * 4 + r + 2 * e;
    else
        return ((mt * (D / 64) + (j >> 2)) * 32 + u) * 16 + (j & 3) * 4 + ((4 * (2 * r + h) + 16 * e) >> 3);
}

template <int BITS>
__device__ __forceinline__ uint32_t v_code_byte(int t, int i, int D, int BS)
{
    const int kk = t >> 4, tt = t & 15, m = (tt >> 1) + 8 * (tt & 1);
    const int h = m >> 3, c = (m & 7) >> 1, e = m & 1;
    const int dm = i >> 4, g = i & 7, r = (i & 15) >> 3, u = 4 * g + c;
    const uint32_t C = (uint32_t)BS * D * BITS / 8;
    if constexpr (BITS == 8)
        return C + ((kk * (D / 32) + (dm >> 1)) * 32 + u) * 16 + ((dm & 1) * 2 + r) * 4 + h + 2 * e;
    else if constexpr (BITS == 2)
        return C + (kk * 32 + u) * (D / 8) + (dm >> 1) * 4 + h + 2 * e;
    else
        return C + ((kk * (D / 64) + (dm >> 2)) * 32 + u) * 16 + (dm & 3) * 4 + ((4 * (2 * h + r) + 16 * e) >> 3);
}

// c = clamp(rint(x / s), -Q, Q), 0 when s is not positive (a zero row)
__device__ __forceinline__ int quant_code(float x, float s, float Q)
{
    if (!(s > 0.f))
        return 0;
    float y = rintf(__fdiv_rn(x, s));
    if (y > Q)
        y = Q;
    if (y < -Q)
        y = -Q;
    return y == y ? (int)y : 0;
}

__device__ __forceinline__ uint8_t q8_byte(int c) { return (uint8_t)(c + 128); }

__device__ __forceinline__ int find_seq(const int32_t *__restrict__ starts, int num_seqs, int row)
{
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

// One warp per (new row, KV head): stage the K and V rows in shared memory as
// float32, reduce max|x|, then every lane writes whole bytes of the record (a byte
// never holds codes of two slots, so rows of one block append independently).
template <int BITS>
__global__ void __launch_bounds__(128)
paged_kv_append_quant_kernel(uint8_t *__restrict__ records, const uint16_t *__restrict__ k_new,
                             const uint16_t *__restrict__ v_new, const int32_t *__restrict__ block_tables,
                             int max_blocks_per_seq, const int32_t *__restrict__ context_lens_old,
                             const int32_t *__restrict__ new_starts, int num_seqs, int total_rows, int num_blocks,
                             int block_size, int num_kv_heads, int head_dim, int rec_bytes,
                             int32_t *__restrict__ status)
{
    __shared__ float xs[4][2][128];
    const int wib = threadIdx.x >> 5;
    const int warp = blockIdx.x * 4 + wib;
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
    const int D = head_dim;
    const size_t src = ((size_t)row * num_kv_heads + h) * D;
    float ak = 0.f, av = 0.f;
    for (int i = lane; i < D; i += 32) {
        const float xk = __uint_as_float((uint32_t)__ldg(k_new + src + i) << 16);
        const float xv = __uint_as_float((uint32_t)__ldg(v_new + src + i) << 16);
        xs[wib][0][i] = xk;
        xs[wib][1][i] = xv;
        ak = fmaxf(ak, fabsf(xk));
        av = fmaxf(av, fabsf(xv));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        ak = fmaxf(ak, __shfl_xor_sync(0xffffffffu, ak, off));
        av = fmaxf(av, __shfl_xor_sync(0xffffffffu, av, off));
    }
    __syncwarp();
    const float Q = BITS == 8 ? 127.f : BITS == 4 ? 7.f : 1.f;
    const float sk = __fdiv_rn(ak, Q), sv = __fdiv_rn(av, Q);
    uint8_t *rec = records + ((size_t)blk * num_kv_heads + h) * rec_bytes;
    const int t = (int)(p % block_size);
    if constexpr (BITS == 8) {
        for (int i = lane; i < D; i += 32) {
            rec[k_code_byte<8>(t, i, D)] = q8_byte(quant_code(xs[wib][0][i], sk, Q));
            rec[v_code_byte<8>(t, i, D, block_size)] = q8_byte(quant_code(xs[wib][1][i], sv, Q));
        }
    } else if constexpr (BITS == 2) {
        // byte task k: K dims 32 (k/8) + 2 ((k%8)/2) + k%2 + {0, 8, 16, 24} (the k-step pair's
        // h and parity, bit pairs 2 (2q + h)); V dims 32 (k/8) + k%8 + {0, 8, 16, 24} (r and
        // parity, bit pairs 2 (2q + r))
        for (int k = lane; k < D / 4; k += 32) {
            const int ik = 32 * (k >> 3) + 2 * ((k & 7) >> 1) + (k & 1);
            const int iv = 32 * (k >> 3) + (k & 7);
            uint32_t bk = 0, bv = 0;
#pragma unroll
            for (int f = 0; f < 4; ++f) {   // f = 2q + (h or r): dim offset 16 q + 8 (h or r)
                const int off = 16 * (f >> 1) + 8 * (f & 1);
                bk |= (uint32_t)(quant_code(xs[wib][0][ik + off], sk, Q) + 2) << (2 * f);
                bv |= (uint32_t)(quant_code(xs[wib][1][iv + off], sv, Q) + 2) << (2 * f);
            }
            rec[k_code_byte<2>(t, ik, D)] = (uint8_t)bk;
            rec[v_code_byte<2>(t, iv, D, block_size)] = (uint8_t)bv;
        }
    } else {
        // byte task k: K dims (16 (k/8) + 2 ((k%8)/2) + k%2, + 8); V dims (16 (k/8) + k%8, + 8)
        for (int k = lane; k < D / 2; k += 32) {
            const int ik = 16 * (k >> 3) + 2 * ((k & 7) >> 1) + (k & 1);
            const int iv = 16 * (k >> 3) + (k & 7);
            rec[k_code_byte<4>(t, ik, D)] =
                (uint8_t)((quant_code(xs[wib][0][ik], sk, Q) + 8) | ((quant_code(xs[wib][0][ik + 8], sk, Q) + 8) << 4));
            rec[v_code_byte<4>(t, iv, D, block_size)] =
                (uint8_t)((quant_code(xs[wib][1][iv], sv, Q) + 8) | ((quant_code(xs[wib][1][iv + 8], sv, Q) + 8) << 4));
        }
    }
    if (lane == 0) {
        const uint32_t C = (uint32_t)block_size * D * BITS / 8;
        reinterpret_cast<float *>(rec + 2 * C)[t] = sk;
        reinterpret_cast<float *>(rec + 2 * C + 4 * block_size)[t] = sv;
    }
}

int launch_quant(const PoolView &pv, AttnParams &prm, int rows, long long pairs, int n_max, cudaStream_t st)
{
    CUtensorMap none;   // the quantised path reads records with bulk copies, not tensor maps
    memset(&none, 0, sizeof none);
    const int D = pv.head_dim, BS = pv.block_size;
    if (pv.bits == 8) {
        if (D == 64 && BS == 16) return launch_d_bs<64, 16, 8, false>(rows, none, none, prm, pairs, n_max, st);
        if (D == 64 && BS == 32) return launch_d_bs<64, 32, 8, false>(rows, none, none, prm, pairs, n_max, st);
        if (D == 128 && BS == 16) return launch_d_bs<128, 16, 8, false>(rows, none, none, prm, pairs, n_max, st);
        return launch_d_bs<128, 32, 8, false>(rows, none, none, prm, pairs, n_max, st);
    }
    if (pv.bits == 2) {
        if (D == 64 && BS == 16) return launch_d_bs<64, 16, 2, false>(rows, none, none, prm, pairs, n_max, st);
        if (D == 64 && BS == 32) return launch_d_bs<64, 32, 2, false>(rows, none, none, prm, pairs, n_max, st);
        if (D == 128 && BS == 16) return launch_d_bs<128, 16, 2, false>(rows, none, none, prm, pairs, n_max, st);
        return launch_d_bs<128, 32, 2, false>(rows, none, none, prm, pairs, n_max, st);
    }
    if (D == 64 && BS == 16) return launch_d_bs<64, 16, 4, false>(rows, none, none, prm, pairs, n_max, st);
    if (D == 64 && BS == 32) return launch_d_bs<64, 32, 4, false>(rows, none, none, prm, pairs, n_max, st);
    if (D == 128 && BS == 16) return launch_d_bs<128, 16, 4, false>(rows, none, none, prm, pairs, n_max, st);
    return launch_d_bs<128, 32, 4, false>(rows, none, none, prm, pairs, n_max, st);
}

}  // namespace
}  // namespace pkv

extern "C" size_t pkv_qrecord_bytes(int32_t block_size, int32_t head_dim, int32_t bits)
{
    if (block_size <= 0 || head_dim <= 0 || (bits != 8 && bits != 4 && bits != 2))
        return 0;
    return 2 * (size_t)block_size * head_dim * bits / 8 + 8 * (size_t)block_size;
}

extern "C" int paged_kv_append_quant(const pkv_qpool *pool, const int32_t *block_tables,
                                     int32_t max_blocks_per_seq, const int32_t *context_lens_old,
                                     const int32_t *new_starts, const void *k_new, const void *v_new,
                                     int32_t num_seqs, int32_t total_new_rows, void *stream)
{
    using namespace pkv;
    clear_error();
    if (!pool)
        return set_error(PKV_ERR_NULL, "paged_kv_append_quant: pool is NULL");
    if (num_seqs < 0 || total_new_rows < 0 || max_blocks_per_seq <= 0)
        return set_error(PKV_ERR_SHAPE, "paged_kv_append_quant: negative sizes or max_blocks_per_seq <= 0");
    if (pool->num_blocks <= 0 || pool->num_kv_heads <= 0)
        return set_error(PKV_ERR_SHAPE, "paged_kv_append_quant: pool dimensions must be positive");
    if (pool->bits != 8 && pool->bits != 4 && pool->bits != 2)
        return set_error(PKV_ERR_UNSUPPORTED, "paged_kv_append_quant: bits %d (built: 8, 4, 2)", pool->bits);
    if (!(pool->head_dim == 64 || pool->head_dim == 128) || !(pool->block_size == 16 || pool->block_size == 32))
        return set_error(PKV_ERR_UNSUPPORTED,
                         "paged_kv_append_quant: head_dim %d / block_size %d (built: 64 or 128 / 16 or 32)",
                         pool->head_dim, pool->block_size);
    if (total_new_rows == 0 || num_seqs == 0)
        return PKV_OK;
    if (!pool->records || !block_tables || !context_lens_old || !new_starts || !k_new || !v_new)
        return set_error(PKV_ERR_NULL, "paged_kv_append_quant: a required pointer is NULL");
    if (!aligned16(pool->records) || (reinterpret_cast<uintptr_t>(k_new) & 1u) ||
        (reinterpret_cast<uintptr_t>(v_new) & 1u))
        return set_error(PKV_ERR_ALIGN, "paged_kv_append_quant: records must be 16-byte aligned");
    int32_t *status = device_status_word();
    if (!status)
        return set_error(PKV_ERR_CUDA, "paged_kv_append_quant: no device status word");
    const long long warps = (long long)total_new_rows * pool->num_kv_heads;
    const long long blocks = (warps + 3) / 4;
    if (blocks > 0x7fffffffLL)
        return set_error(PKV_ERR_SHAPE, "paged_kv_append_quant: too many rows");
    const int rb = (int)pkv_qrecord_bytes(pool->block_size, pool->head_dim, pool->bits);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto kern = pool->bits == 8 ? paged_kv_append_quant_kernel<8>
              : pool->bits == 4 ? paged_kv_append_quant_kernel<4> : paged_kv_append_quant_kernel<2>;
    kern<<<(unsigned)blocks, 128, 0, st>>>(static_cast<uint8_t *>(pool->records),
                                           static_cast<const uint16_t *>(k_new), static_cast<const uint16_t *>(v_new),
                                           block_tables, max_blocks_per_seq, context_lens_old, new_starts, num_seqs,
                                           total_new_rows, pool->num_blocks, pool->block_size, pool->num_kv_heads,
                                           pool->head_dim, rb, status);
    return check_cuda(cudaGetLastError(), "paged_kv_append_quant launch");
}

extern "C" int paged_attention_forward_quant(const pkv_qpool *pool, const void *q, const int32_t *q_starts,
                                             const int32_t *block_tables, int32_t max_blocks_per_seq,
                                             const int32_t *context_lens, int32_t num_seqs, int32_t total_q_rows,
                                             int32_t max_context_len, int32_t max_q_rows_per_seq,
                                             int32_t num_q_heads, const int32_t *kv_head_of_q_head,
                                             const float *sinks, int32_t causal, float scale, void *out,
                                             int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                             void *stream)
{
    using namespace pkv;
    clear_error();
    const char *who = "paged_attention_forward_quant";
    if (!pool)
        return set_error(PKV_ERR_NULL, "%s: pool is NULL", who);
    if (pool->bits != 8 && pool->bits != 4 && pool->bits != 2)
        return set_error(PKV_ERR_UNSUPPORTED, "%s: bits %d (built: 8, 4, 2)", who, pool->bits);
    PoolView pv = {pool->num_blocks, pool->block_size, pool->num_kv_heads, pool->head_dim, pool->bits,
                   nullptr, nullptr, pool->records};
    return attention_run(who, pv, q, q_starts, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                         total_q_rows, max_context_len, max_q_rows_per_seq, num_q_heads, kv_head_of_q_head, sinks,
                         causal, nullptr, scale, out, out_dtype, workspace, workspace_bytes, stream, launch_quant);
}
