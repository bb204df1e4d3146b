/*
 * pkv.h -- C ABI of libpkv.so: batched paged-KV attention for continuous
 * batching on NVIDIA GB300 (sm_103a).
 *
 * Three operations (with tree variants), each one or two hand-written CUDA kernels:
 *   paged_kv_append          scatter new tokens' K/V rows into the block pool
 *   paged_attention_forward  decode / causal verify-window attention over K/V
 *                            gathered through per-sequence block tables, with
 *                            optional per-head sink logits
 *   spec_accept_greedy       per-row argmax of verify logits, then a walk of
 *                            each draft chain to its first mismatch
 *
 * Conventions shared by every entry point
 *  - Pointers are DEVICE pointers unless the argument says HOST.  The library
 *    allocates no memory and owns no buffer: the caller owns every input,
 *    output and workspace, and must keep them alive until the stream reaches
 *    the launched work.
 *  - bf16 arrays are IEEE bfloat16 (the high 16 bits of a binary32).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every call is asynchronous on it, except pkv_device_status().
 *  - Every call returns a pkv_status.  Argument errors are found on the host
 *    before anything is launched; the text of the last error of the calling
 *    thread is available from pkv_last_error_string().  Conditions that only
 *    the device can see (a block id outside the pool, a context longer than
 *    the table or than max_context_len, a sequence with more query rows than
 *    max_q_rows_per_seq) never fault: the kernel clamps the access, records a
 *    bit in a device status word and carries on; pkv_device_status() reports
 *    and clears it.  Outputs of the affected rows are then unspecified.
 *  - Block pool layout: K and V are separate pools, each
 *    bf16 [num_blocks][num_kv_heads][block_size][head_dim], so one block of one
 *    KV head is block_size * head_dim contiguous values.  Identical prefixes
 *    may be shared by pointing several block tables at the same physical
 *    block ids.
 *  - Block tables: int32 [num_seqs][max_blocks_per_seq]; logical token t of
 *    sequence s is slot t % block_size of block block_tables[s][t / block_size].
 *
 * Sources (page title, section): TensorSharp "高级功能" (advanced features),
 * sections "连续批处理与分页 KV 缓存" (continuous batching and the paged KV
 * cache: fixed-size blocks from a shared pool, full blocks content-hashed and
 * shared across requests), "原生分页注意力" (native paged attention, gathering
 * K/V from the paged buffers; the WithSinks variant for GPT OSS) and the
 * "批量前向" (batched forward) paragraph (paged K/V scatter-write);
 * TensorFold article, sections "先记住一条铁律" (every verify-window row uses the
 * serial step's arithmetic) and "接受规则：GPU 上的 accept 内核" (the accept
 * kernel); TensorSharp "高级功能", section "MTP / NextN 推测解码" (verify all
 * drafts in one batched forward, commit the accepted prefix).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_NULL = -1,        /* a required pointer is NULL                          */
    PKV_ERR_SHAPE = -2,       /* sizes inconsistent or out of range                  */
    PKV_ERR_UNSUPPORTED = -3, /* head_dim / block_size / group x window not built    */
    PKV_ERR_WORKSPACE = -4,   /* workspace too small                                 */
    PKV_ERR_BAD_BLOCK = -5,   /* (device) block id outside the pool / table overrun  */
    PKV_ERR_CUDA = -6,        /* a CUDA runtime call or kernel launch failed         */
    PKV_ERR_ALIGN = -7,       /* a pointer is not 16-byte aligned                    */
    PKV_ERR_TIMEOUT = -8,     /* (device) a bounded wait inside a kernel expired     */
    PKV_ERR_OUT_OF_BLOCKS = -9 /* (device) the free stack or the block index ran out */
} pkv_status;

enum { PKV_DTYPE_BF16 = 0, PKV_DTYPE_F32 = 1 };

/* Bits of the device status word (see pkv_device_status). */
enum {
    PKV_DEV_BAD_BLOCK = 1,     /* a block id outside [0, num_blocks)                      */
    PKV_DEV_TABLE_OVERRUN = 2, /* a length past max_blocks_per_seq * block_size or
                                  past max_context_len                                    */
    PKV_DEV_TOO_MANY_ROWS = 4, /* a sequence with more rows than max_q_rows_per_seq       */
    PKV_DEV_WORKSPACE = 8,     /* (reserved)                                              */
    PKV_DEV_TIMEOUT = 16,      /* a bounded wait expired                                  */
    PKV_DEV_BAD_TREE = 32,     /* a draft tree whose parent indices are not topological   */
    PKV_DEV_BAD_RANGE = 64,    /* a token range outside [0, total_tokens]                 */
    PKV_DEV_OUT_OF_BLOCKS = 128, /* the block allocator's free stack ran out               */
    PKV_DEV_INDEX_FULL = 256   /* the block index had no free slot for a new key          */
};

/* One layer's K/V block pool (host struct holding device pointers).
 * k_pool, v_pool: bf16 [num_blocks][num_kv_heads][block_size][head_dim],
 * 16-byte aligned. */
typedef struct pkv_pool {
    void *k_pool;
    void *v_pool;
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
} pkv_pool;

/* Version of this ABI (incremented on any incompatible change). */
int pkv_abi_version(void);

/*
 * Paged K/V scatter-append ("批量前向": the batched forward pairs its
 * projections with a paged K/V scatter-write).
 *
 * New token i of sequence s (rows new_starts[s] .. new_starts[s+1]-1 of k_new /
 * v_new) sits at position p = context_lens_old[s] + i and is copied, bit for
 * bit and for every KV head, to slot p % block_size of block
 * block_tables[s][p / block_size] of both pools.  The caller must already have
 * placed a private block at that table entry: shared (hashed, full) blocks are
 * never appended to.  Rollback of rejected speculative tokens needs no call:
 * the caller simply does not advance its context length past them.
 *
 *   pool             HOST struct; pools as described above
 *   block_tables     int32 [num_seqs][max_blocks_per_seq]
 *   context_lens_old int32 [num_seqs], tokens cached before this append
 *   new_starts       int32 [num_seqs + 1], prefix sums of new tokens per sequence
 *   k_new, v_new     bf16 [total_new_rows][num_kv_heads][head_dim], 16-byte aligned
 *   total_new_rows   HOST; equals new_starts[num_seqs]
 * head_dim must be a multiple of 8.  Launches one kernel (none if
 * total_new_rows == 0).  Device-side checks: table overrun, bad block id.
 */
int paged_kv_append(const pkv_pool *pool,
                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *context_lens_old, const int32_t *new_starts,
                    const void *k_new, const void *v_new,
                    int32_t num_seqs, int32_t total_new_rows, void *stream);

/*
 * Bytes of workspace paged_attention_forward needs for these sizes (a
 * multiple of 256): the per-split partial results (running max, sum and
 * unnormalised output of every query row, q head and 512-token split).  Its
 * contents on entry do not matter.  One workspace serves any sequence of calls
 * on one stream; calls that may overlap on the GPU need separate workspaces.
 */
size_t paged_attention_workspace_size(int32_t num_seqs, int32_t total_q_rows,
                                      int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t max_context_len);

/* Zero a workspace (cudaMemsetAsync on `stream`); optional, kept for callers that
 * want deterministic workspace contents. */
int paged_attention_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/*
 * Batched paged attention ("原生分页注意力", with the GPT OSS sinks variant; the
 * causal verify window per "先记住一条铁律").
 *
 * For query row r of sequence s (W = q_starts[s+1] - q_starts[s] rows,
 * w = r - q_starts[s]) and q head h reading KV head g = map(h):
 *   n   = causal ? L - W + w + 1 : L,   L = context_lens[s]
 *   x_t = scale * q[r][h] . K_s[t][g]                      for t < n
 *   out[r][h] = sum_t e^{x_t} V_s[t][g] / (sum_t e^{x_t} + e^{sinks[h]})
 * (the sink term only when sinks != NULL; a row that sees no key and has no
 * sink outputs zeros).  K_s/V_s are read through the block table.
 *
 *   pool               HOST struct; head_dim in {64, 128}, block_size in {16, 32}
 *   q                  bf16 [total_q_rows][num_q_heads][head_dim]
 *   q_starts           int32 [num_seqs + 1], rows of each sequence
 *   block_tables       int32 [num_seqs][max_blocks_per_seq]
 *   context_lens       int32 [num_seqs], keys in the cache INCLUDING the tokens
 *                      appended for this step (decode token / verify window)
 *   max_context_len    HOST upper bound of context_lens (sizes the grid)
 *   max_q_rows_per_seq HOST upper bound of rows per sequence; G * it <= 8192
 *                      where G = num_q_heads / num_kv_heads (decode: 1 row;
 *                      verify windows: up to 16; prefill chunks: more)
 *   kv_head_of_q_head  HOST int32 [num_q_heads] or NULL (NULL: h -> h / G).
 *                      Each KV head must serve exactly G q heads.
 *   sinks              float32 [num_q_heads] or NULL: one logit per q head in
 *                      the units of the scaled scores
 *   causal             0: every row sees all L keys; 1: verify-window mask
 *   scale              > 0, or <= 0 for 1/sqrt(head_dim)
 *   out                [total_q_rows][num_q_heads][head_dim], bf16 or float32
 *                      (out_dtype = PKV_DTYPE_BF16 / PKV_DTYPE_F32)
 *   workspace          >= paged_attention_workspace_size(...) bytes, 256-byte
 *                      aligned
 * Every row's arithmetic depends only on its own sequence (its length fixes
 * the split of the keys into fixed 512-token chunks and the order in which the
 * chunks' partials merge), so a row computed in any batch is bit-identical to the same row
 * computed alone, and row w of a causal window is bit-identical to a one-row
 * decode over the first L - W + w + 1 keys.  Launches two kernels: the split
 * kernel and, as its programmatic dependent, the merge.
 */
int paged_attention_forward(const pkv_pool *pool,
                            const void *q, const int32_t *q_starts,
                            const int32_t *block_tables, int32_t max_blocks_per_seq,
                            const int32_t *context_lens,
                            int32_t num_seqs, int32_t total_q_rows,
                            int32_t max_context_len, int32_t max_q_rows_per_seq,
                            int32_t num_q_heads, const int32_t *kv_head_of_q_head,
                            const float *sinks, int32_t causal, float scale,
                            void *out, int32_t out_dtype,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * Tree verify attention (TensorFold article, "接受规则：GPU 上的 accept 内核": the
 * verify rows form a chain or a tree of drafts).  Same computation and
 * arguments as paged_attention_forward, except that row w of sequence s sees
 * every cached key t < L - W and the window key L - W + i exactly when bit i of
 * tree_masks[q_starts[s] + w] is set (the node's ancestors and itself).  A chain
 * is the mask (1 << (w + 1)) - 1 and gives the causal window bit for bit.
 *   tree_masks          uint32 [total_q_rows]
 *   max_q_rows_per_seq  at most 32
 */
int paged_tree_attention_forward(const pkv_pool *pool,
                                 const void *q, const int32_t *q_starts,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *context_lens,
                                 int32_t num_seqs, int32_t total_q_rows,
                                 int32_t max_context_len, int32_t max_q_rows_per_seq,
                                 int32_t num_q_heads, const int32_t *kv_head_of_q_head,
                                 const float *sinks, const uint32_t *tree_masks, float scale,
                                 void *out, int32_t out_dtype,
                                 void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace spec_accept_greedy needs (a multiple of 256). */
size_t spec_accept_workspace_size(int32_t total_rows, int32_t vocab);

/*
 * Greedy speculative accept ("接受规则：GPU 上的 accept 内核": compare each draft
 * with the target's choice and follow the chain to the first mismatch).
 *
 * Sequence s owns rows q_starts[s] .. q_starts[s+1]-1 (W rows).  Row 0 is the
 * query of the last committed token; row j >= 1 carries draft token
 * d_j = draft_tokens[q_starts[s] + j] (slot 0 is ignored).
 *   a_j           = argmax_v logits[q_starts[s] + j][v], ties to the lowest v
 *   accept_len[s] = n, the largest n <= W-1 with d_i == a_{i-1} for all i <= n
 *   out_tokens    = d_1 .. d_n, a_n at q_starts[s] + 0 .. n, then -1
 * A sequence with no rows gets accept_len = -1.  NaN logits give an
 * unspecified argmax.
 *
 *   logits        float32 [total_rows][vocab], 16-byte aligned
 *   q_starts      int32 [num_seqs + 1]; draft_tokens int32 [total_rows]
 *   argmax_out    int32 [total_rows]; accept_len int32 [num_seqs];
 *   out_tokens    int32 [total_rows]
 *   workspace     >= spec_accept_workspace_size(total_rows, vocab) bytes
 * Launches two kernels.  Results are exact (integer) and independent of the
 * batch.
 */
int spec_accept_greedy(const float *logits, int32_t vocab,
                       const int32_t *q_starts, const int32_t *draft_tokens,
                       int32_t num_seqs, int32_t total_rows,
                       int32_t *argmax_out, int32_t *accept_len, int32_t *out_tokens,
                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * Allocation-free paged attention: the same computation and arguments as
 * paged_attention_forward, minus the workspace, for callers that cannot
 * allocate device memory (a stream being captured into a CUDA graph that must
 * not allocate, runtimes that own all device memory through their own arena,
 * plug-in hosts whose allocator this library cannot reach).  The pages have no
 * counterpart of this entry point; it exists for those callers only.
 *
 * The workspace lives in a fixed device array of PKV_NOALLOC_SCRATCH_BYTES
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  Sizes whose paged_attention_workspace_size exceeds it are
 * rejected with PKV_ERR_WORKSPACE before anything is launched.  Every call
 * looks the array's device address up (cudaGetSymbolAddress) in the caller's
 * current device and context, so a context created after cudaDeviceReset, or a
 * driver-API context other than the primary one, gets its own copy of the
 * array; the first call in a context may load the library's module there, so
 * make that first call before any stream capture.  Each call launches the
 * attention kernels with the array as their workspace (whose contents on entry
 * do not matter: every partial is written before it is read); it calls no
 * allocator.  All calls in a context
 * share the one array, which keeps the last call's contents: calls that may
 * overlap on the GPU (different streams without ordering) race and corrupt
 * each other's results.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (32u << 20)
int paged_attention_forward_noalloc(const pkv_pool *pool,
                                    const void *q, const int32_t *q_starts,
                                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                                    const int32_t *context_lens,
                                    int32_t num_seqs, int32_t total_q_rows,
                                    int32_t max_context_len, int32_t max_q_rows_per_seq,
                                    int32_t num_q_heads, const int32_t *kv_head_of_q_head,
                                    const float *sinks, int32_t causal, float scale,
                                    void *out, int32_t out_dtype, void *stream);

/*
 * Greedy accept over draft trees (TensorFold article, "接受规则：GPU 上的 accept
 * 内核": from the root, follow the child whose token equals the target's
 * choice).  Sequence s owns nodes j = 0..W-1 at rows q_starts[s] + j; node 0 is
 * the last committed token; node j >= 1 carries draft token d_j and has parent
 * node parents[q_starts[s] + j] in [0, j).  From u = 0, with a_u the argmax of
 * row u (ties to the lowest id), the walk moves to the lowest-index child c of
 * u with d_c == a_u and stops at a node with no such child.
 *   accept_len[s]    number of accepted drafts n (-1: no rows, or a bad tree,
 *                    which also sets PKV_DEV_BAD_TREE)
 *   out_tokens       the n accepted drafts, then a_u of the final node, then -1
 *   accepted_rows    the n accepted node indices (rows to keep), then -1
 * At most 1024 nodes per sequence.  A chain (parents[j] = j - 1) gives
 * spec_accept_greedy's result.  Uses spec_accept_workspace_size bytes of
 * workspace; launches two kernels.
 */
int spec_accept_tree_greedy(const float *logits, int32_t vocab,
                            const int32_t *q_starts, const int32_t *draft_tokens,
                            const int32_t *parents, int32_t num_seqs, int32_t total_rows,
                            int32_t *argmax_out, int32_t *accept_len, int32_t *out_tokens,
                            int32_t *accepted_rows, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * Sampled accept (TensorFold article, "先记住一条铁律": every draw is keyed by
 * seed, absolute position and token id, and a draft is accepted only when it
 * equals the target's own draw; "接受规则": the top-k, top-p and min_p filters
 * are part of the keyed rule).  The target's draw at row r:
 *   temperature == 0: the argmax (ties to the lowest id);
 *   otherwise the lowest v maximising l_v / temperature + g(seed, positions[r], v)
 *   over the kept v: those passing all three filters, each defined on the whole
 *   row.  With the order "logit descending, token id ascending": top-k keeps the
 *   first top_k tokens (off when top_k <= 0 or >= vocab); top-p keeps the
 *   shortest prefix whose integer weight reaches ceil(p_fix * total / 2^32),
 *   p_fix = floor(top_p * 2^32), total = the row's weight (off unless
 *   0 < top_p < 1), the weight of v being floor(2^32 * exp2(((l_v - l_max) / T)
 *   * log2 e)) with exp2 a fixed float32 sequence (0 below 2^-32; else the
 *   degree-8 Taylor polynomial of 2^f, f the fraction, by Horner's rule, times
 *   2^floor); min_p keeps l_v >= l_max + temperature * logf(min_p) (off when
 *   min_p <= 0);
 *   g = -log(-log(u)), u = ((w >> 9) + 1/2) / 2^23 and w is word (v mod 4)
 *   of Philox4x32-10(counter = (v / 4, pos, 0x6b657964, 0), key = seed); the
 *   logs are a fixed float32 operation sequence (atanh series) and every step is
 *   a correctly rounded float32 operation, so the draw is reproducible exactly.
 * The walk is the greedy accept's (chain when parents is NULL, else tree) with
 * the draw in place of the argmax; outputs as spec_accept_tree_greedy, with
 * sampled_out holding every row's draw.
 *   positions   int32 [total_rows]: absolute position of the token each row draws
 *   workspace   >= 2 * spec_accept_workspace_size(total_rows, vocab) + 8 * total_rows
 *               bytes (the last part rounded up to 256)
 * Launches three kernels (two when temperature == 0), four with top-k / top-p.
 */
int spec_accept_sampled(const float *logits, int32_t vocab,
                        const int32_t *q_starts, const int32_t *draft_tokens,
                        const int32_t *parents, const int32_t *positions,
                        uint64_t seed, float temperature, int32_t top_k, float top_p, float min_p,
                        int32_t num_seqs, int32_t total_rows,
                        int32_t *sampled_out, int32_t *accept_len, int32_t *out_tokens,
                        int32_t *accepted_rows, void *workspace, size_t workspace_bytes,
                        void *stream);

/*
 * Chained content keys of full KV blocks, for prefix sharing (TensorSharp
 * "高级功能", section "连续批处理与分页 KV 缓存": every full block is
 * content-hashed, so identical prefixes map to the same blocks).  For sequence s
 * with tokens tokens[token_starts[s] .. token_starts[s+1]) (starting at a block
 * boundary), block i of its floor(n / block_size) full blocks gets
 *   c_i = FNV-1a 64 over the little-endian bytes of the block's token ids,
 *   h_0 = chain_in[s] (seed when chain_in is NULL), h_{i+1} = mix(h_i ^ c_i),
 *   hashes_out[s][i] = h_{i+1},
 * mix being the SplitMix64 output function.  The rest of row s is set to 0 (a
 * partial block is never shared).  Passing the key of the last block already
 * hashed as chain_in[s] continues the chain, so a decode step re-hashes nothing.
 *   tokens        int32 [total_tokens]            (device)
 *   token_starts  int32 [num_seqs + 1]            (device)
 *   chain_in      uint64 [num_seqs] or NULL       (device)
 *   hashes_out    uint64 [num_seqs][max_blocks_per_seq] (device, written)
 * block_size in [1, 1024].  A sequence with more full blocks than
 * max_blocks_per_seq gets keys for the first max_blocks_per_seq and sets
 * PKV_DEV_TABLE_OVERRUN; a token range outside [0, total_tokens] leaves its row
 * zero and sets PKV_DEV_BAD_RANGE.  One kernel launch, no workspace.
 */
int paged_block_hashes(const int32_t *tokens, const int32_t *token_starts, int32_t num_seqs,
                       int32_t total_tokens, int32_t block_size, uint64_t seed,
                       const uint64_t *chain_in, uint64_t *hashes_out,
                       int32_t max_blocks_per_seq, void *stream);

/*
 * Index-list gather (TensorSharp "高级功能", the DeepSeek V4 executor item: decode
 * attention reads a compact [ring | top-k] set of keys through an index-gather
 * instead of the whole context).  Query row r of sequence s attends to the keys
 * at positions key_idx[r][0 .. key_counts[r]-1] of s, read through the block
 * table; a position listed twice counts twice; there is no causal mask (the list
 * says what the row sees); sinks as in paged_attention_forward.
 *   key_idx     int32 [total_q_rows][max_keys] (device); entries past a row's
 *               count are not read
 *   key_counts  int32 [total_q_rows] (device), each in [0, max_keys]
 *   max_keys    at most max_blocks_per_seq * block_size
 * A listed position outside [0, context_lens[s]) contributes a zero key and value
 * and sets PKV_DEV_TABLE_OVERRUN (the row's output is then not meaningful); a
 * count outside [0, max_keys] is clamped and sets the same bit.  Workspace:
 * paged_attention_workspace_size(num_seqs, total_q_rows, num_q_heads,
 * num_kv_heads, head_dim, max_keys).  Within a row the arithmetic depends only
 * on its own list, so a row computed in a batch equals the row alone.  Launches
 * two kernels.
 */
int paged_attention_forward_gather(const pkv_pool *pool, const void *q, const int32_t *q_starts,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *context_lens, int32_t num_seqs, int32_t total_q_rows,
                                   const int32_t *key_idx, const int32_t *key_counts, int32_t max_keys,
                                   int32_t num_q_heads, const int32_t *kv_head_of_q_head,
                                   const float *sinks, float scale, void *out, int32_t out_dtype,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * Quantised KV blocks (TensorSharp "高级功能", section "内存优化", the KV block
 * codec item: blocks may be compressed in place to 8, 4 or 2 bits per value,
 * Q8 / Q4 / Q2, for a fraction of the footprint at an accuracy cost).  The
 * pages give no codec internals; this library's codec:
 *   each (token, KV head) row x of head_dim bf16 values is stored as one float32
 *   scale s = max_i |x_i| / Q (Q = 2^(bits-1) - 1: 127 for 8 bits, 7 for 4 bits,
 *   1 for 2 bits, whose codes are -1, 0, 1) and codes
 *   c_i = clamp(rint(x_i / s), -Q, Q) (all 0 when s == 0), every step a correctly
 *   rounded float32 operation (rint ties to even); it reads back as c_i * s.
 *   Non-finite inputs give unspecified (but in-range) codes.
 * Pool: records uint8 [num_blocks][num_kv_heads][R], R = pkv_qrecord_bytes(),
 * 16-byte aligned.  Record = [K codes | V codes | K scales | V scales]:
 *   C = block_size * head_dim * bits / 8 bytes of codes per section; the K scale
 *   of slot t at byte 2C + 4t, the V scale at 2C + 4 block_size + 4t (float32).
 *   8-bit codes: bytes holding c + 128.  4-bit codes: nibbles holding c + 8.
 *   2-bit codes: bit pairs holding c + 2.
 *   Position of the code of slot t, dim i (16-byte units of 4 little-endian
 *   32-bit words, laid out in the order the attention kernel's tensor-core
 *   operands consume them):
 *   K: mt = t/16, g = (t%16)/2, r = t%2, j = i/16, s = i%16,
 *      c = (s%8)/2, h = s/8, e = s%2, u = 4g + c
 *      8-bit: byte ((mt*(D/32) + j/2)*32 + u)*16 + ((j%2)*2 + r)*4 + h + 2e
 *      4-bit: word ((mt*(D/64) + j/4)*32 + u)*16 + (j%4)*4, bits 4(2r + h) + 16e
 *      2-bit: word (mt*32 + u)*(D/8) + (j/2)*4, bits 8r + 2(2(j%2) + h) + 16e
 *   V: kk = t/16, m = (t%16)/2 + 8(t%2), h = m/8, c = (m%8)/2, e = m%2,
 *      dm = i/16, g = i%8, r = (i%16)/8, u = 4g + c
 *      8-bit: byte C + ((kk*(D/32) + dm/2)*32 + u)*16 + ((dm%2)*2 + r)*4 + h + 2e
 *      4-bit: word C + ((kk*(D/64) + dm/4)*32 + u)*16 + (dm%4)*4, bits 4(2h + r) + 16e
 *      2-bit: word C + (kk*32 + u)*(D/8) + (dm/2)*4, bits 8h + 2(2(dm%2) + r) + 16e
 *   (D = head_dim).  A byte never holds codes of two slots.
 * Built for head_dim 64 / 128 and block_size 16 / 32.
 */
typedef struct pkv_qpool {
    void *records;
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t bits;   /* 8, 4 or 2 */
} pkv_qpool;

/* Bytes of one (block, KV head) record; 0 for unsupported arguments. */
size_t pkv_qrecord_bytes(int32_t block_size, int32_t head_dim, int32_t bits);

/*
 * paged_kv_append with quantisation: the slot of every new row is found as in
 * paged_kv_append and its K and V rows (bf16 [total_new_rows][num_kv_heads]
 * [head_dim], any 2-byte alignment) are quantised into that slot of the
 * record of (block, KV head).  Other slots are untouched; rows of one call may
 * share a block.  Device-side errors as paged_kv_append.  One kernel launch.
 */
int paged_kv_append_quant(const pkv_qpool *pool, const int32_t *block_tables,
                          int32_t max_blocks_per_seq, const int32_t *context_lens_old,
                          const int32_t *new_starts, const void *k_new, const void *v_new,
                          int32_t num_seqs, int32_t total_new_rows, void *stream);

/*
 * paged_attention_forward over a quantised pool: the same definition with K
 * and V read back as c * s; every other argument, the workspace
 * (paged_attention_workspace_size, of which it uses at most that much), the
 * split / merge structure and the batch-invariance rules are those of
 * paged_attention_forward, except that the keys split into fixed 1024-token
 * chunks.  Within one codec the arithmetic is fixed by the row's own sequence,
 * so a row computed in a batch equals the row alone, bit for bit, and row w of
 * a causal window equals the one-row decode over its keys.
 */
int paged_attention_forward_quant(const pkv_qpool *pool, const void *q, const int32_t *q_starts,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *context_lens, int32_t num_seqs, int32_t total_q_rows,
                                  int32_t max_context_len, int32_t max_q_rows_per_seq,
                                  int32_t num_q_heads, const int32_t *kv_head_of_q_head,
                                  const float *sinks, int32_t causal, float scale, void *out,
                                  int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * Block allocation with prefix sharing (TensorSharp "高级功能", section "连续批处理与分页
 * KV 缓存": KV blocks of a fixed size come from one shared pool; every full block is
 * content-hashed so that identical prefixes map to the same physical blocks; a partial
 * block is never shared).
 *
 * The index (all arrays device memory, owned by the caller):
 *   keys       uint64 [capacity]: a block key (from paged_block_hashes), or
 *              PKV_BLOCK_KEY_EMPTY in a free slot
 *   block_ids  int32 [capacity]: the physical block holding the key's contents
 *              (negative: the key has no block, e.g. its allocation ran out)
 *   refcounts  int32 [capacity]: how many block-table entries name that block
 *   capacity   slots, a power of two; keep the index at most about half full
 *              (open addressing with linear probing)
 *   free_ids   int32 [...]: a stack of free physical block ids, free_ids[0 .. *free_count)
 *   free_count int32 [1]: ids on the stack
 * The caller fills free_ids; paged_block_index_init empties every slot and sets
 * *free_count.  A key equal to PKV_BLOCK_KEY_EMPTY cannot be indexed: its block is
 * allocated as a private one.
 */
#define PKV_BLOCK_KEY_EMPTY 0xFFFFFFFFFFFFFFFFull
typedef struct pkv_block_index {
    uint64_t *keys;
    int32_t *block_ids;
    int32_t *refcounts;
    int32_t capacity;
    int32_t *free_ids;
    int32_t *free_count;
} pkv_block_index;

/* Empty every slot of the index and set *free_count = num_free.  One launch. */
int paged_block_index_init(const pkv_block_index *index, int32_t num_free, void *stream);

/* Workspace bytes paged_block_allocate needs for num_seqs x max_blocks_per_seq entries. */
size_t paged_block_allocate_workspace_size(int32_t num_seqs, int32_t max_blocks_per_seq);

/*
 * Fill block tables from the index and the free stack.  Sequence s holds
 * L = context_lens[s] tokens in nb = ceil(L / block_size) blocks; the first
 * nk = floor(L / block_size) are full and carry the keys block_keys[s][j] (the layout
 * paged_block_hashes writes); entries j < first_block[s] are already allocated and
 * are left alone.  For j = first_block[s] .. nb - 1:
 *   - a full block whose key has a block in the index shares it (table entry = that
 *     id, its reference count + 1, fresh 0);
 *   - a full block whose key has none takes a block from the free stack; later blocks
 *     with the same key in this call share it (fresh 1 for the first, 0 for the rest);
 *   - a partial block takes a private block from the free stack (fresh 1).
 * The result is the sequential engine step: sequences in order, blocks in order, the
 * k-th pop of the call taking free_ids[F - 1 - k] (F = *free_count on entry), however
 * the kernels' threads interleave.  fresh[s][j] (may be NULL) is set for every entry:
 * 1 where this call allocated a block the caller must fill, else 0.  A pop past the
 * stack's end gives -1 (the key, if any, stays without a block) and sets
 * PKV_DEV_OUT_OF_BLOCKS; a key that finds no free slot gets a private block and sets
 * PKV_DEV_INDEX_FULL (the results are then not the sequential ones); a length past
 * max_blocks_per_seq * block_size is cut there and sets PKV_DEV_TABLE_OVERRUN.
 *   block_keys    uint64 [num_seqs][max_blocks_per_seq] (device, 8-byte aligned)
 *   context_lens, first_block   int32 [num_seqs] (device)
 *   block_tables  int32 [num_seqs][max_blocks_per_seq] (device, in / out)
 *   workspace     paged_block_allocate_workspace_size bytes, 256-byte aligned; its
 *                 contents on entry do not matter
 * Calls that use one index must be ordered on the GPU (one stream).  Three launches.
 */
int paged_block_allocate(const pkv_block_index *index, const uint64_t *block_keys,
                         const int32_t *context_lens, const int32_t *first_block, int32_t num_seqs,
                         int32_t block_size, int32_t max_blocks_per_seq, int32_t *block_tables,
                         int32_t *fresh, void *workspace, size_t workspace_bytes, void *stream);

/* Text of the calling thread's last error ("" if none). */
const char *pkv_last_error_string(void);

/*
 * Synchronise `stream`, then read and clear the device status word of the
 * current device.  Returns PKV_OK, PKV_ERR_BAD_BLOCK (bad block id or table
 * overrun), PKV_ERR_SHAPE (too many rows, a bad draft tree or a bad token
 * range), PKV_ERR_TIMEOUT, PKV_ERR_OUT_OF_BLOCKS (the allocator ran out),
 * or PKV_ERR_CUDA; *bits (if not NULL) receives the raw PKV_DEV_* bits.
 */
int pkv_device_status(void *stream, int32_t *bits);

/*
 * The kernel that serves the bf16 attention calls (paged_attention_forward and its
 * allocation-free variant, paged_tree_attention_forward, paged_attention_forward_gather),
 * process-wide, for the calls launched after it:
 *   PKV_KERNEL_MMA_SYNC (the default): warp-level mma.sync tiles of 16 keys, many small
 *     CTAs per SM;
 *   PKV_KERNEL_TCGEN05: 5th-generation tensor cores (tcgen05.mma, accumulators in tensor
 *     memory), 128-key tiles, one persistent CTA per SM fed by a one-CTA unit pass.
 * Both give results within the same tolerance of the exact attention, and with either a
 * row's arithmetic depends only on its own sequence (batch / solo and verify-row / decode
 * invariance hold), but the two kernels round differently: switch only between workloads,
 * never between calls whose rows must agree bit for bit.  The quantised pools always use
 * the mma.sync kernel.  Returns PKV_OK, or PKV_ERR_SHAPE for an unknown value.  (No passage
 * of the pages; it selects between two implementations of the same operation.)
 */
enum { PKV_KERNEL_MMA_SYNC = 0, PKV_KERNEL_TCGEN05 = 1 };
int pkv_set_attention_kernel(int32_t which);

/*
 * Test hook for the failure path of the attention kernels' bounded waits.  Sets
 * the limit, in SM clock cycles, that each stage wait of the attention pipeline
 * (the consumer's wait for a staged tile, the producer's wait for a free stage)
 * may take in the calls launched after it, process-wide.  0 makes every such wait
 * give up at once, without testing its barrier: the kernel then records
 * PKV_DEV_TIMEOUT, stops issuing copies, waits for the copies it already issued
 * (that final wait always keeps the default limit) and returns, so the copies
 * land and the context stays usable; the call's output is undefined.  A negative
 * value restores the default (about two seconds of SM clock).  Not thread-safe
 * with respect to calls launched concurrently from other threads.  Returns PKV_OK.
 * (No passage of the pages; it exists to test the library's own error path.)
 */
int pkv_debug_set_wait_limit(long long cycles);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
