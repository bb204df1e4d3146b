// pkv_hash.cu -- chained content keys of full KV blocks (prefix sharing).
//
// TensorSharp "高级功能", section "连续批处理与分页 KV 缓存": every full block is
// content-hashed, so identical prefixes (system prompts, shared context) map to
// the same blocks.  A block's key names its whole prefix:
//   c_i = FNV-1a 64 over the little-endian bytes of block i's token ids,
//   h_{i+1} = mix(h_i ^ c_i) (SplitMix64 output function), key_i = h_{i+1}.
//
// One warp per sequence.  The content hashes of 32 blocks are computed in
// parallel (lane j hashes block 32 q + j); the chain through them is serial
// by nature, so every lane runs the 32 mixes of the chunk on the broadcast
// content hashes and lane j keeps the key after step j.
#include <cstdint>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr uint64_t kFnvOffset = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

__device__ __forceinline__ uint64_t splitmix64_mix(uint64_t z)
{
    z ^= z >> 30;
    z *= 0xbf58476d1ce4e5b9ull;
    z ^= z >> 27;
    z *= 0x94d049bb133111ebull;
    z ^= z >> 31;
    return z;
}

__device__ __forceinline__ uint64_t fnv1a_word(uint64_t h, uint32_t v)
{
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        h ^= (v >> (8 * b)) & 0xffu;
        h *= kFnvPrime;
    }
    return h;
}

__global__ void __launch_bounds__(128)
block_hash_kernel(const int32_t *__restrict__ tokens, const int32_t *__restrict__ token_starts,
                  int32_t num_seqs, int32_t total_tokens, int32_t block_size, uint64_t seed,
                  const uint64_t *__restrict__ chain_in, uint64_t *__restrict__ hashes_out,
                  int32_t max_blocks_per_seq, int32_t *status)
{
    const int s = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (s >= num_seqs)
        return;
    uint64_t *row = hashes_out + (size_t)s * max_blocks_per_seq;
    const int a = __ldg(token_starts + s);
    const int b = __ldg(token_starts + s + 1);
    int full = 0;
    if (a < 0 || b > total_tokens || b < a) {
        if (lane == 0)
            atomicOr(status, PKV_DEV_BAD_RANGE);
    } else {
        full = (b - a) / block_size;
        if (full > max_blocks_per_seq) {
            if (lane == 0)
                atomicOr(status, PKV_DEV_TABLE_OVERRUN);
            full = max_blocks_per_seq;
        }
    }
    const uint32_t *tok = reinterpret_cast<const uint32_t *>(tokens) + (a < 0 ? 0 : a);
    uint64_t h = chain_in ? __ldg(reinterpret_cast<const unsigned long long *>(chain_in) + s) : seed;
    for (int q0 = 0; q0 < full; q0 += 32) {
        const int i = q0 + lane;
        uint64_t c = kFnvOffset;
        if (i < full) {
            const uint32_t *blk = tok + (size_t)i * block_size;
            int t = 0;
            for (; t + 4 <= block_size; t += 4) {
                const uint32_t v0 = __ldg(blk + t), v1 = __ldg(blk + t + 1);
                const uint32_t v2 = __ldg(blk + t + 2), v3 = __ldg(blk + t + 3);
                c = fnv1a_word(fnv1a_word(fnv1a_word(fnv1a_word(c, v0), v1), v2), v3);
            }
            for (; t < block_size; ++t)
                c = fnv1a_word(c, __ldg(blk + t));
        }
        const int n = min(32, full - q0);
        uint64_t mine = 0;
        for (int j = 0; j < n; ++j) {
            h = splitmix64_mix(h ^ __shfl_sync(0xffffffffu, c, j));
            if (j == lane)
                mine = h;
        }
        if (i < full)
            row[i] = mine;
    }
    for (int i = full + lane; i < max_blocks_per_seq; i += 32)
        row[i] = 0;
}

}  // namespace
}  // namespace pkv

extern "C" int paged_block_hashes(const int32_t *tokens, const int32_t *token_starts, int32_t num_seqs,
                                  int32_t total_tokens, int32_t block_size, uint64_t seed,
                                  const uint64_t *chain_in, uint64_t *hashes_out,
                                  int32_t max_blocks_per_seq, void *stream)
{
    using namespace pkv;
    clear_error();
    if (!token_starts || !hashes_out)
        return set_error(PKV_ERR_NULL, "paged_block_hashes: token_starts and hashes_out are required");
    if (num_seqs < 0 || total_tokens < 0 || max_blocks_per_seq < 0)
        return set_error(PKV_ERR_SHAPE, "paged_block_hashes: negative size");
    if (block_size < 1 || block_size > 1024)
        return set_error(PKV_ERR_UNSUPPORTED, "paged_block_hashes: block_size %d outside [1, 1024]",
                         block_size);
    if (total_tokens > 0 && !tokens)
        return set_error(PKV_ERR_NULL, "paged_block_hashes: tokens is NULL");
    if ((reinterpret_cast<uintptr_t>(hashes_out) & 7u) || (reinterpret_cast<uintptr_t>(chain_in) & 7u) ||
        (reinterpret_cast<uintptr_t>(tokens) & 3u) || (reinterpret_cast<uintptr_t>(token_starts) & 3u))
        return set_error(PKV_ERR_ALIGN, "paged_block_hashes: pointers must be aligned to their element size");
    if (num_seqs == 0 || max_blocks_per_seq == 0)
        return PKV_OK;
    int32_t *status = device_status_word();
    if (!status)
        return set_error(PKV_ERR_CUDA, "paged_block_hashes: device status word unavailable");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int grid = (num_seqs + 3) / 4;
    block_hash_kernel<<<grid, 128, 0, st>>>(tokens, token_starts, num_seqs, total_tokens, block_size, seed,
                                            chain_in, hashes_out, max_blocks_per_seq, status);
    return check_cuda(cudaGetLastError(), "paged_block_hashes: launch");
}
