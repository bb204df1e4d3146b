/*
 * pkv_oracle.c -- float64 CPU oracle for batched paged-KV attention, the paged
 * K/V scatter-append and the greedy speculative accept step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain statement of what the
 * GPU path computes.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline / reference arm may build, load or call it.  It shares no code,
 * header, table or helper with the CUDA library, and the CUDA library never
 * calls it: there is no CPU fallback.
 *
 * Sources (page title, section):
 *  - TensorSharp "高级功能" (advanced features), section "连续批处理与分页 KV 缓存"
 *    (continuous batching and paged KV cache): the KV cache is cut into
 *    fixed-size blocks drawn from a shared pool; every full block is
 *    content-hashed so identical prefixes share physical blocks.
 *  - same page, section "原生分页注意力" (native paged attention): K/V are
 *    gathered from the paged buffers per sequence and fed to an ordinary
 *    attention; a variant carries per-head attention-sink logits (GPT OSS).
 *  - same page, section "批量前向" (batched forward, the paragraph on
 *    ForwardBatch): new tokens' K/V are scattered into their paged slots.
 *  - TensorFold article, section "接受规则：GPU 上的 accept 内核" (the accept
 *    rule: the accept kernel on the GPU): each draft token is compared with the
 *    target's choice and the accepted path follows the child whose token equals
 *    that choice, i.e. the chain is walked to the first mismatch.
 *  - TensorSharp page, section "MTP / NextN 推测解码": lossless speculative
 *    decoding verifies all drafts in one batched forward and commits the
 *    accepted prefix; verification follows the target greedily.
 *
 * Conventions fixed where the pages are silent (listed with reasons in the
 * design notes): K/V pools are bf16 [num_blocks][H_kv][block_size][head_dim];
 * q is bf16 [R][H_q][head_dim] with rows of sequence s at q_starts[s] ..
 * q_starts[s+1]-1; the default GQA map is h -> h / (H_q/H_kv); the score scale
 * multiplies q.k in float64; a sink is one logit per q head, in the units of
 * the scaled scores, adding exp(sink) to the softmax denominator only; with the
 * causal window, row w of a W-row window of a sequence of length L sees keys
 * t < L - W + w + 1; a row that sees no key and has no sink outputs zeros;
 * argmax ties go to the lowest index.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> float64: the 16 stored bits are the high half of an IEEE binary32;
 * the widening is exact. */
static double bf16_bits_to_f64(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_version(void) { return 1; }

/*
 * Paged K/V scatter-append.  New token i of sequence s sits at absolute
 * position p = context_lens_old[s] + i.  Its slot is block
 * block_tables[s][p / block_size], offset p % block_size.  The K and V rows of
 * each KV head are copied there bit for bit.
 * Returns 0, or -1 if a position falls beyond the table, -2 for a block id
 * outside [0, num_blocks).
 */
int oracle_paged_kv_append(uint16_t *k_pool, uint16_t *v_pool,
                           int32_t num_blocks, int32_t block_size,
                           int32_t num_kv_heads, int32_t head_dim,
                           const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens_old, const int32_t *new_starts,
                           const uint16_t *k_new, const uint16_t *v_new,
                           int32_t num_seqs)
{
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t n_new = new_starts[s + 1] - new_starts[s];
        for (int32_t i = 0; i < n_new; ++i) {
            int64_t p = (int64_t)context_lens_old[s] + i;
            int64_t logical = p / block_size;
            int64_t offset = p % block_size;
            if (logical >= max_blocks_per_seq)
                return -1;
            int32_t blk = block_tables[(int64_t)s * max_blocks_per_seq + logical];
            if (blk < 0 || blk >= num_blocks)
                return -2;
            int64_t row = (int64_t)new_starts[s] + i;
            for (int32_t h = 0; h < num_kv_heads; ++h) {
                size_t dst = ((((size_t)blk * num_kv_heads) + h) * block_size + offset) * head_dim;
                size_t src = (((size_t)row * num_kv_heads) + h) * head_dim;
                memcpy(k_pool + dst, k_new + src, (size_t)head_dim * sizeof(uint16_t));
                memcpy(v_pool + dst, v_new + src, (size_t)head_dim * sizeof(uint16_t));
            }
        }
    }
    return 0;
}

/*
 * Attention over the paged pool, by the definition:
 *   for each query row r of sequence s and q head h (KV head g = map[h]):
 *     n   = causal ? L - W + w + 1 : L        (w = r - q_starts[s], W = rows of s)
 *     x_t = scale * sum_k q[r][h][k] * K_s[t][g][k],        t < n
 *     M   = max(max_t x_t, sink_h)                           (sink only if given)
 *     out = sum_t e^{x_t - M} V_s[t][g] / (sum_t e^{x_t - M} + e^{sink_h - M})
 * K_s and V_s are first materialised contiguously from the block table
 * (logical token t -> block block_tables[s][t / B], slot t % B).
 * Everything is float64.  out is float64 [R][H_q][head_dim].
 * kv_head_of_q_head may be NULL (contiguous groups); sinks may be NULL.
 * Tree verify (TensorFold article, "接受规则": the verify rows may form a draft
 * tree): with tree_masks != NULL, row w of sequence s sees every cached key
 * t < L - W and the window key L - W + i exactly when bit i of tree_masks[r]
 * is set (its ancestors and itself); `causal` is then ignored.
 * Returns 0, -1 (position beyond table), -2 (block id out of range),
 * -3 (bad head map), -4 (out of memory), -5 (tree window wider than 32).
 */
/* Where attention reads K/V rows from: bf16 pools, or quantised block records
 * (see the quantised KV section below). */
struct kv_source {
    const uint16_t *k_pool, *v_pool;   /* bf16 pools, or NULL */
    const uint8_t *records;            /* quantised records, or NULL */
    int32_t bits;
};

static void kv_read_row(const struct kv_source *src, int32_t blk, int32_t g, int32_t off,
                        int32_t Hkv, int32_t B, int32_t D, double *k, double *v);

static int attention_core(const struct kv_source *src,
                          int32_t num_blocks, int32_t block_size,
                          int32_t num_kv_heads, int32_t head_dim,
                          const uint16_t *q, const int32_t *q_starts,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *context_lens, int32_t num_seqs,
                          int32_t num_q_heads, const int32_t *kv_head_of_q_head,
                          const float *sinks, int32_t causal, const uint32_t *tree_masks,
                          double scale, double *out, int32_t num_threads)
{
    const int32_t B = block_size, D = head_dim, Hkv = num_kv_heads, Hq = num_q_heads;
    if (Hkv <= 0 || Hq % Hkv != 0)
        return -3;
    const int32_t group = Hq / Hkv;
    for (int32_t h = 0; h < Hq; ++h) {
        int32_t g = kv_head_of_q_head ? kv_head_of_q_head[h] : h / group;
        if (g < 0 || g >= Hkv)
            return -3;
    }
    /* validate every table entry that will be read */
    for (int32_t s = 0; s < num_seqs; ++s) {
        if (tree_masks && q_starts[s + 1] - q_starts[s] > 32)
            return -5;
        int64_t L = context_lens[s];
        int64_t nblk = (L + B - 1) / B;
        if (nblk > max_blocks_per_seq)
            return -1;
        for (int64_t j = 0; j < nblk; ++j) {
            int32_t blk = block_tables[(int64_t)s * max_blocks_per_seq + j];
            if (blk < 0 || blk >= num_blocks)
                return -2;
        }
    }

    int failed = 0;
    const int64_t pairs = (int64_t)num_seqs * Hkv;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
    for (int64_t pg = 0; pg < pairs; ++pg) {
        const int32_t s = (int32_t)(pg / Hkv), g = (int32_t)(pg % Hkv);
        const int64_t L = context_lens[s];
        const int32_t row0 = q_starts[s], W = q_starts[s + 1] - q_starts[s];
        if (W <= 0)
            continue;
        /* step 1: materialise contiguous K_s, V_s for KV head g */
        double *K = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D);
        double *V = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D);
        double *x = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        if (!K || !V || !x) {
            free(K); free(V); free(x);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
            continue;
        }
        for (int64_t t = 0; t < L; ++t) {
            int32_t blk = block_tables[(int64_t)s * max_blocks_per_seq + t / B];
            kv_read_row(src, blk, g, (int32_t)(t % B), Hkv, B, D, K + t * D, V + t * D);
        }
        /* step 2: every query row of s, every q head that reads KV head g */
        for (int32_t w = 0; w < W; ++w) {
            const int64_t r = (int64_t)row0 + w;
            int64_t n = causal ? L - W + w + 1 : L;
            if (tree_masks)
                n = L;
            if (n < 0) n = 0;
            if (n > L) n = L;
            const int64_t win0 = L - W;   /* first key of the verify window */
            for (int32_t h = 0; h < Hq; ++h) {
                int32_t gh = kv_head_of_q_head ? kv_head_of_q_head[h] : h / group;
                if (gh != g)
                    continue;
                const uint16_t *qv = q + ((size_t)r * Hq + h) * D;
                double *o = out + ((size_t)r * Hq + h) * D;
                double M = -INFINITY;
                for (int64_t t = 0; t < n; ++t) {
                    if (tree_masks && t >= win0 && !((tree_masks[r] >> (t - win0)) & 1u)) {
                        x[t] = -INFINITY;   /* not an ancestor of this node: invisible */
                        continue;
                    }
                    double dot = 0.0;
                    for (int32_t k = 0; k < D; ++k)
                        dot += bf16_bits_to_f64(qv[k]) * K[t * D + k];
                    x[t] = scale * dot;
                    if (x[t] > M)
                        M = x[t];
                }
                const int has_sink = sinks != NULL;
                const double sink = has_sink ? (double)sinks[h] : 0.0;
                if (has_sink && sink > M)
                    M = sink;
                double den = 0.0;
                for (int32_t k = 0; k < D; ++k)
                    o[k] = 0.0;
                for (int64_t t = 0; t < n; ++t) {
                    if (x[t] == -INFINITY)
                        continue;
                    double e = exp(x[t] - M);
                    den += e;
                    for (int32_t k = 0; k < D; ++k)
                        o[k] += e * V[t * D + k];
                }
                if (has_sink)
                    den += exp(sink - M);
                for (int32_t k = 0; k < D; ++k)
                    o[k] = den > 0.0 ? o[k] / den : 0.0;
            }
        }
        free(K);
        free(V);
        free(x);
    }
    return failed ? -4 : 0;
}

int oracle_paged_attention(const uint16_t *k_pool, const uint16_t *v_pool,
                           int32_t num_blocks, int32_t block_size,
                           int32_t num_kv_heads, int32_t head_dim,
                           const uint16_t *q, const int32_t *q_starts,
                           const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens, int32_t num_seqs,
                           int32_t num_q_heads, const int32_t *kv_head_of_q_head,
                           const float *sinks, int32_t causal, const uint32_t *tree_masks,
                           double scale, double *out, int32_t num_threads)
{
    struct kv_source src = {k_pool, v_pool, NULL, 16};
    return attention_core(&src, num_blocks, block_size, num_kv_heads, head_dim, q, q_starts,
                          block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                          kv_head_of_q_head, sinks, causal, tree_masks, scale, out, num_threads);
}

/*
 * Row argmax over the vocabulary, ties to the lowest index: scan v = 0..V-1 and
 * replace the best only on a strictly greater value.
 */
void oracle_argmax_rows(const float *logits, int64_t rows, int32_t vocab, int32_t *argmax_out)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *row = logits + (size_t)r * vocab;
        int32_t best = 0;
        for (int32_t v = 1; v < vocab; ++v)
            if (row[v] > row[best])
                best = v;
        argmax_out[r] = best;
    }
}

/*
 * Greedy accept over draft chains.  Sequence s owns rows q_starts[s] ..
 * q_starts[s+1]-1 (W rows).  Row 0 is the query of the last committed token;
 * row j >= 1 carries draft d_j = draft_tokens[q_starts[s] + j].  With a_j the
 * target argmax of row j, draft d_j is accepted while d_i == a_{i-1} for every
 * i <= j.  accept_len[s] = n, the number of accepted drafts; the emitted tokens
 * are d_1..d_n followed by the target's own choice a_n (n + 1 tokens), written
 * to out_tokens[q_starts[s] + 0 .. n]; the remaining slots of the sequence are
 * set to -1.  A sequence with no rows gets accept_len = -1.
 */
void oracle_spec_accept_greedy(const float *logits, int32_t vocab,
                               const int32_t *q_starts, const int32_t *draft_tokens,
                               int32_t num_seqs, int32_t *argmax_out,
                               int32_t *accept_len, int32_t *out_tokens)
{
    const int64_t total = q_starts[num_seqs];
    oracle_argmax_rows(logits, total, vocab, argmax_out);
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int32_t r0 = q_starts[s], W = q_starts[s + 1] - q_starts[s];
        if (W <= 0) {
            accept_len[s] = -1;
            continue;
        }
        int32_t n = 0;
        while (n + 1 < W && draft_tokens[r0 + n + 1] == argmax_out[r0 + n])
            ++n;
        accept_len[s] = n;
        for (int32_t j = 0; j < W; ++j)
            out_tokens[r0 + j] = -1;
        for (int32_t j = 0; j < n; ++j)
            out_tokens[r0 + j] = draft_tokens[r0 + j + 1];
        out_tokens[r0 + n] = argmax_out[r0 + n];
    }
}

/*
 * Greedy accept over a draft tree (TensorFold article, "接受规则：GPU 上的 accept
 * 内核": the verify rows form a chain or a tree; the accepted path follows, from
 * the root, the child whose token equals the target's choice).  Sequence s owns
 * nodes 0..W-1 (rows q_starts[s] + j); node 0 is the last committed token, node
 * j >= 1 carries draft token d_j and has parent parents[r] (a node index < j).
 * From u = 0: a_u = argmax of row u; the next node is the lowest-index child c
 * of u with d_c == a_u; the walk stops at a node with no such child.
 * accept_len[s] = the number of accepted drafts n; out_tokens holds their tokens
 * then a_u of the final node (n + 1 tokens), then -1; accepted_rows holds the
 * accepted node indices (n of them), then -1.  A chain is parents[j] = j - 1.
 * Returns 0, or -1 if a parent index is not smaller than its node's index.
 */
int oracle_spec_accept_tree_greedy(const float *logits, int32_t vocab,
                                   const int32_t *q_starts, const int32_t *draft_tokens,
                                   const int32_t *parents, int32_t num_seqs,
                                   int32_t *argmax_out, int32_t *accept_len,
                                   int32_t *out_tokens, int32_t *accepted_rows)
{
    const int64_t total = q_starts[num_seqs];
    oracle_argmax_rows(logits, total, vocab, argmax_out);
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int32_t r0 = q_starts[s], W = q_starts[s + 1] - q_starts[s];
        if (W <= 0) {
            accept_len[s] = -1;
            continue;
        }
        for (int32_t j = 1; j < W; ++j)
            if (parents[r0 + j] < 0 || parents[r0 + j] >= j)
                return -1;
        for (int32_t j = 0; j < W; ++j) {
            out_tokens[r0 + j] = -1;
            accepted_rows[r0 + j] = -1;
        }
        int32_t u = 0, n = 0;
        for (;;) {
            int32_t next = -1;
            for (int32_t c = u + 1; c < W; ++c)
                if (parents[r0 + c] == u && draft_tokens[r0 + c] == argmax_out[r0 + u]) {
                    next = c;
                    break;
                }
            if (next < 0)
                break;
            out_tokens[r0 + n] = draft_tokens[r0 + next];
            accepted_rows[r0 + n] = next;
            ++n;
            u = next;
        }
        out_tokens[r0 + n] = argmax_out[r0 + u];
        accept_len[s] = n;
    }
    return 0;
}

/* ---------------------------------------------------------- keyed sampling -- */
/*
 * Philox4x32-10, the counter-based generator of Salmon, Moraes, Dror and Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3" (SC'11): ten rounds of
 * (hi, lo) = M * c on words 0 and 2 with M0 = 0xD2511F53, M1 = 0xCD9E8D57, the
 * output words being (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0); the key is bumped
 * by the Weyl constants 0x9E3779B9, 0xBB67AE85 before every round but the first.
 */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        const uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/*
 * Natural logarithm in float32 by a fixed sequence of correctly rounded float32
 * operations (no fused multiply-add), so that any IEEE implementation of the
 * same steps gives the same bits: x = m 2^e with m in [sqrt(1/2), sqrt(2)),
 * s = (m - 1) / (m + 1), log x = e ln 2 + 2 s (1 + s^2/3 + s^4/5 + ... + s^10/11)
 * (the atanh series), with the coefficients rounded to float32.  x > 0, finite.
 */
float oracle_keyed_log(float x)
{
    uint32_t b;
    memcpy(&b, &x, 4);
    int e;
    if ((b >> 23) == 0) {   /* subnormal: scale by 2^23 (exact) */
        x = x * 8388608.0f;
        memcpy(&b, &x, 4);
        e = (int)(b >> 23) - 127 - 23;
    } else {
        e = (int)(b >> 23) - 127;
    }
    const uint32_t mb = (b & 0x7fffffu) | 0x3f800000u;
    float m;
    memcpy(&m, &mb, 4);
    if (m > 0x1.6a09e6p+0f) {
        m = m * 0.5f;
        e += 1;
    }
    const float s = (m - 1.0f) / (m + 1.0f);
    const float z = s * s;
    float p = 0x1.745d18p-4f;        /* 1/11 */
    p = p * z + 0x1.c71c72p-4f;      /* 1/9  */
    p = p * z + 0x1.24924ap-3f;      /* 1/7  */
    p = p * z + 0x1.99999ap-3f;      /* 1/5  */
    p = p * z + 0x1.555556p-2f;      /* 1/3  */
    p = p * z + 1.0f;
    const float r = (s + s) * p;
    return (float)e * 0x1.62e43p-1f + r;   /* ln 2 */
}

/*
 * The 23-bit uniform code of token v at absolute position pos under `seed`: the top
 * 23 bits (w >> 9) of word (v mod 4) of Philox4x32-10 with counter
 * (v / 4, pos, 0x6b657964, 0) and key (seed low word, seed high word).  One generator
 * call keys four consecutive tokens, which lets a GPU thread draw a group of four
 * tokens with one call.  (TensorFold article, section "先记住一条铁律": a draw depends
 * on seed, absolute position and token id only.)
 */
uint32_t oracle_keyed_uniform_bits(uint64_t seed, int32_t pos, int32_t v)
{
    const uint32_t ctr[4] = {(uint32_t)v >> 2, (uint32_t)pos, 0x6b657964u, 0u};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t o[4];
    oracle_philox4x32_10(ctr, key, o);
    return o[(uint32_t)v & 3u] >> 9;
}

/*
 * Keyed Gumbel noise of token v at position pos under `seed`: u = (code + 1/2) / 2^23
 * with the code above, and g = -log(-log(u)) with the fixed float32 log.
 */
float oracle_keyed_gumbel(uint64_t seed, int32_t pos, int32_t v)
{
    const float u = ((float)oracle_keyed_uniform_bits(seed, pos, v) + 0.5f) * 0x1p-23f;
    const float E = -oracle_keyed_log(u);
    return -oracle_keyed_log(E);
}

/*
 * 2^y for y <= 0 as a fixed float32 operation sequence, so that every platform
 * computes the same bits: y < -32 gives 0 (such a weight is below the 2^-32
 * resolution of the integer weights below); otherwise n = floor(y), f = y - n in
 * [0, 1), and 2^f = e^{f ln 2} is the Taylor polynomial of degree 8,
 * sum_k (ln 2)^k / k! f^k, with float32 coefficients, evaluated by Horner's rule
 * with separately rounded multiplies and adds; the result is scaled by 2^n exactly.
 */
float oracle_keyed_exp2(float y)
{
    static const float c[9] = {0x1p+0f, 0x1.62e430p-1f, 0x1.ebfbe0p-3f, 0x1.c6b08ep-5f, 0x1.3b2ab6p-7f,
                               0x1.5d87fep-10f, 0x1.430912p-13f, 0x1.ffcbfcp-17f, 0x1.62c022p-20f};
    if (!(y >= -32.0f))
        return 0.0f;
    if (y >= 0.0f)
        return 1.0f;
    const float n = floorf(y);
    const float f = y - n;
    float p = c[8];
    for (int k = 7; k >= 0; --k) {
        const float t = p * f;
        p = t + c[k];
    }
    return ldexpf(p, (int)n);
}

/* Integer weight of token v in a row with maximum l_max at temperature T:
 * floor(2^32 * keyed_exp2(((l_v - l_max) / T) * log2(e))), every step a correctly
 * rounded float32 operation.  The probability of v is its weight over the row's
 * total; integer weights make every sum exact, whatever the order. */
static uint64_t keyed_weight(float l, float l_max, float temperature)
{
    const float d = l - l_max;
    const float z = d / temperature;
    const float y = z * 0x1.715476p+0f;
    const float w = oracle_keyed_exp2(y);
    return (uint64_t)(w * 4294967296.0f);
}

/* The weight the top-p prefix must reach: ceil(p_fix * total / 2^32), with the
 * product taken exactly (128 bits). */
uint64_t oracle_topp_threshold(uint64_t p_fix, uint64_t total)
{
    const unsigned __int128 prod = (unsigned __int128)p_fix * total;
    return (uint64_t)((prod + 0xFFFFFFFFu) >> 32);
}

/* the order tokens are filtered in: logit descending, then token id ascending */
static const float *g_sort_row;
static int order_cmp(const void *a, const void *b)
{
    const int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    const float lx = g_sort_row[x], ly = g_sort_row[y];
    if (lx > ly)
        return -1;
    if (lx < ly)
        return 1;
    return x < y ? -1 : (x > y ? 1 : 0);
}

/*
 * Tokens kept by top-k and top-p, as a count n: the kept tokens are the first n of
 * the order (logit descending, id ascending).  top-k keeps k tokens (k <= 0 or
 * k >= vocab: all).  top-p keeps the shortest prefix whose weight reaches
 * ceil(p_fix * total / 2^32), p_fix = floor(p * 2^32), total = the row's weight
 * (0 < p < 1; otherwise all).  n = min of the two.  order_out (vocab entries) may
 * be NULL; it receives the order.  Returns n, or -1 when out of memory.
 */
int32_t oracle_topkp_kept(const float *row, int32_t vocab, float temperature, int32_t top_k, float top_p,
                          int32_t *order_out)
{
    int32_t *order = order_out ? order_out : (int32_t *)malloc(sizeof(int32_t) * (size_t)vocab);
    if (!order)
        return -1;
    for (int32_t v = 0; v < vocab; ++v)
        order[v] = v;
    g_sort_row = row;
    qsort(order, (size_t)vocab, sizeof(int32_t), order_cmp);
    int32_t n = vocab;
    if (top_k > 0 && top_k < n)
        n = top_k;
    if (top_p > 0.0f && top_p < 1.0f) {
        const float l_max = row[order[0]];
        uint64_t total = 0;
        for (int32_t v = 0; v < vocab; ++v)
            total += keyed_weight(row[v], l_max, temperature);
        const uint64_t thr = oracle_topp_threshold((uint64_t)(top_p * 4294967296.0f), total);
        uint64_t cum = 0;
        int32_t np = vocab;
        for (int32_t i = 0; i < vocab; ++i) {
            cum += keyed_weight(row[order[i]], l_max, temperature);
            if (cum >= thr) {
                np = i + 1;
                break;
            }
        }
        if (np < n)
            n = np;
    }
    if (!order_out)
        free(order);
    return n;
}

/*
 * The target's keyed draw for one row (TensorFold article, "先记住一条铁律": every
 * draw is keyed by seed, absolute position and token id; "接受规则": the top-k,
 * top-p and min_p filters are part of the keyed rule).  temperature == 0: the
 * greedy argmax.  Otherwise the kept tokens are those that pass all three filters,
 * each defined on the whole row: the first n of the order by oracle_topkp_kept, and
 * l_v >= thr with thr = l_max + temperature * log(min_p) (no filter when min_p <= 0;
 * log(min_p) is the host libm's logf).  The draw is the lowest v maximising
 * l_v / temperature + g(seed, pos, v) over the kept v, all in float32.
 */
static int32_t keyed_draw(const float *row, int32_t vocab, uint64_t seed, int32_t pos, float temperature,
                          int32_t top_k, float top_p, float min_p, uint8_t *kept)
{
    int32_t best = 0;
    for (int32_t v = 1; v < vocab; ++v)
        if (row[v] > row[best])
            best = v;
    if (temperature == 0.0f)
        return best;
    const float l_max = row[best];
    const float thr = min_p > 0.0f ? l_max + temperature * logf(min_p) : -INFINITY;
    const int filtered = (top_k > 0 && top_k < vocab) || (top_p > 0.0f && top_p < 1.0f);
    if (filtered) {
        int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)vocab);
        if (!order)
            return -1;
        const int32_t n = oracle_topkp_kept(row, vocab, temperature, top_k, top_p, order);
        memset(kept, 0, (size_t)vocab);
        for (int32_t i = 0; i < n; ++i)
            kept[order[i]] = 1;
        free(order);
    }
    int32_t pick = -1;
    float top = -INFINITY;
    for (int32_t v = 0; v < vocab; ++v) {
        if (!(row[v] >= thr))
            continue;
        if (filtered && !kept[v])
            continue;
        const float sc = row[v] / temperature + oracle_keyed_gumbel(seed, pos, v);
        if (pick < 0 || sc > top) {
            top = sc;
            pick = v;
        }
    }
    return pick;
}

/*
 * Sampled accept (TensorFold article, "先记住一条铁律" and "接受规则"): the target's
 * token at row r is keyed_draw(row r, positions[r]); drafts are accepted along
 * the chain (parents == NULL) or the tree exactly as in the greedy accept, with
 * the draw in place of the argmax.  Outputs as oracle_spec_accept_tree_greedy,
 * sampled_out holding each row's draw.  Returns 0 or -1 (bad parent index).
 */
int oracle_spec_accept_sampled(const float *logits, int32_t vocab, const int32_t *q_starts,
                               const int32_t *draft_tokens, const int32_t *parents,
                               const int32_t *positions, uint64_t seed, float temperature,
                               int32_t top_k, float top_p, float min_p,
                               int32_t num_seqs, int32_t *sampled_out, int32_t *accept_len,
                               int32_t *out_tokens, int32_t *accepted_rows)
{
    const int64_t total = q_starts[num_seqs];
    uint8_t *kept = (uint8_t *)malloc((size_t)vocab);
    if (!kept)
        return -2;
    for (int64_t r = 0; r < total; ++r)
        sampled_out[r] = keyed_draw(logits + (size_t)r * vocab, vocab, seed, positions[r], temperature, top_k,
                                    top_p, min_p, kept);
    free(kept);
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int32_t r0 = q_starts[s], W = q_starts[s + 1] - q_starts[s];
        if (W <= 0) {
            accept_len[s] = -1;
            continue;
        }
        for (int32_t j = 1; j < W; ++j) {
            const int32_t par = parents ? parents[r0 + j] : j - 1;
            if (par < 0 || par >= j)
                return -1;
        }
        for (int32_t j = 0; j < W; ++j) {
            out_tokens[r0 + j] = -1;
            accepted_rows[r0 + j] = -1;
        }
        int32_t u = 0, n = 0;
        for (;;) {
            int32_t next = -1;
            for (int32_t c = u + 1; c < W; ++c) {
                const int32_t par = parents ? parents[r0 + c] : c - 1;
                if (par == u && draft_tokens[r0 + c] == sampled_out[r0 + u]) {
                    next = c;
                    break;
                }
            }
            if (next < 0)
                break;
            out_tokens[r0 + n] = draft_tokens[r0 + next];
            accepted_rows[r0 + n] = next;
            ++n;
            u = next;
        }
        out_tokens[r0 + n] = sampled_out[r0 + u];
        accept_len[s] = n;
    }
    return 0;
}

/* -------------------------------------------------------- block hashing -- */
/*
 * Content keys of full KV blocks for prefix sharing (TensorSharp "高级功能",
 * "连续批处理与分页 KV 缓存": every full block is content-hashed, so identical
 * prefixes, such as a shared system prompt, map to the same blocks).  A block is
 * only interchangeable with another if everything before it matches too, so a
 * block's key names its whole prefix by chaining:
 *   c_i = FNV-1a 64 over the little-endian bytes of the block's B token ids
 *         (offset basis 0xcbf29ce484222325, prime 0x100000001b3);
 *   h_0 = chain_in[s] (or `seed` when chain_in is NULL);
 *   h_{i+1} = mix(h_i ^ c_i), mix = the SplitMix64 output function
 *         z ^= z >> 30; z *= 0xbf58476d1ce4e5b9; z ^= z >> 27;
 *         z *= 0x94d049bb133111eb; z ^= z >> 31;
 *   key of block i = h_{i+1}.
 * Sequence s's tokens [token_starts[s], token_starts[s+1]) start at a block
 * boundary; only its floor(n / B) full blocks get keys (a partial block is never
 * shared), written to hashes_out[s][0 ..]; the rest of the row is set to 0.
 * Passing the key of the last block already hashed as chain_in continues a chain,
 * so a decode step hashes only the blocks that have just filled up.
 */
uint64_t oracle_fnv1a64(const uint8_t *bytes, int64_t n)
{
    uint64_t h = 0xcbf29ce484222325ull;
    for (int64_t i = 0; i < n; ++i) {
        h ^= bytes[i];
        h *= 0x100000001b3ull;
    }
    return h;
}

uint64_t oracle_splitmix64_mix(uint64_t z)
{
    z ^= z >> 30;
    z *= 0xbf58476d1ce4e5b9ull;
    z ^= z >> 27;
    z *= 0x94d049bb133111ebull;
    z ^= z >> 31;
    return z;
}

int oracle_block_hashes(const int32_t *tokens, const int32_t *token_starts, int32_t num_seqs,
                        int32_t block_size, uint64_t seed, const uint64_t *chain_in,
                        uint64_t *hashes_out, int32_t max_blocks_per_seq)
{
    if (block_size <= 0 || block_size > 1024)
        return -2;
    uint8_t *buf = (uint8_t *)malloc(4 * (size_t)block_size);
    if (!buf)
        return -3;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int64_t n = (int64_t)token_starts[s + 1] - token_starts[s];
        const int64_t full = n > 0 ? n / block_size : 0;
        if (full > max_blocks_per_seq) {
            free(buf);
            return -1;
        }
        uint64_t *row = hashes_out + (int64_t)s * max_blocks_per_seq;
        for (int64_t i = 0; i < max_blocks_per_seq; ++i)
            row[i] = 0;
        uint64_t h = chain_in ? chain_in[s] : seed;
        for (int64_t i = 0; i < full; ++i) {
            const int32_t *blk = tokens + token_starts[s] + i * block_size;
            for (int32_t t = 0; t < block_size; ++t) {
                const uint32_t v = (uint32_t)blk[t];
                buf[4 * t + 0] = (uint8_t)(v & 0xffu);
                buf[4 * t + 1] = (uint8_t)((v >> 8) & 0xffu);
                buf[4 * t + 2] = (uint8_t)((v >> 16) & 0xffu);
                buf[4 * t + 3] = (uint8_t)((v >> 24) & 0xffu);
            }
            h = oracle_splitmix64_mix(h ^ oracle_fnv1a64(buf, 4 * (int64_t)block_size));
            row[i] = h;
        }
    }
    free(buf);
    return 0;
}

/* ----------------------------------------------------- quantised KV blocks -- */
/*
 * TensorSharp "高级功能", section "内存优化", the KV block codec item: blocks may
 * be compressed in place to 8, 4 or 2 bits per value (Q8 / Q4 / Q2, selected by
 * --paged-kv-quant-bits), trading a small accuracy cost for half or a quarter of
 * the footprint.  The pages give no codec internals.  The plainest codec with
 * that footprint, and the one built here:
 *   every (token, KV head) row x of head_dim bf16 values is quantised
 *   symmetrically with one float32 scale,
 *     Q = 2^(bits-1) - 1: 127 (8 bits), 7 (4 bits) or 1 (2 bits: codes -1, 0, 1),
 *     amax  = max_i |x_i|                       (float32, exact)
 *     scale = amax / Q                          (float32 division, round to nearest)
 *     c_i   = clamp(rint(x_i / scale), -Q, Q)   (float32 division; rint ties to even)
 *             (c_i = 0 for every i when scale == 0),
 *   and is read back as c_i * scale.  Every step is a correctly rounded float32
 *   operation, so the codes are reproducible exactly.
 *
 * Record layout (our own; one record per (block, KV head), records of a block's
 * heads adjacent, record = [K codes | V codes | K scales | V scales]):
 *   C = block_size * head_dim * bits / 8 bytes of codes per section;
 *   K scale of slot t at byte 2C + 4t, V scale at 2C + 4 block_size + 4t
 *   (float32, little-endian).
 *   8-bit codes are bytes holding c + 128; 4-bit codes are nibbles holding c + 8;
 *   2-bit codes are bit pairs holding c + 2.
 *   Code positions, for slot t and dim i, with 16-byte units of 4 little-endian
 *   32-bit words:
 *   K: mt = t/16, g = (t%16)/2, r = t%2, j = i/16, s = i%16,
 *      c = (s%8)/2, h = s/8, e = s%2, u = 4g + c;
 *      8-bit: byte ((mt*D/32 + j/2)*32 + u)*16 + ((j%2)*2 + r)*4 + h + 2e
 *      4-bit: word ((mt*D/64 + j/4)*32 + u)*16 + (j%4)*4, bits 4(2r + h) + 16e
 *      2-bit: word (mt*32 + u)*(D/8) + (j/2)*4, bits 8r + 2(2(j%2) + h) + 16e
 *   V: kk = t/16, m = (t%16)/2 + 8(t%2), h = m/8, c = (m%8)/2, e = m%2,
 *      dm = i/16, g = i%8, r = (i%16)/8, u = 4g + c;
 *      8-bit: byte C + ((kk*D/32 + dm/2)*32 + u)*16 + ((dm%2)*2 + r)*4 + h + 2e
 *      4-bit: word C + ((kk*D/64 + dm/4)*32 + u)*16 + (dm%4)*4, bits 4(2h + r) + 16e
 *      2-bit: word C + (kk*32 + u)*(D/8) + (dm/2)*4, bits 8h + 2(2(dm%2) + r) + 16e
 *   (the 2-bit units are D/8 bytes: 8 at head_dim 64, 16 at 128).
 * Every byte holds codes of one slot only, so tokens of one block can be
 * appended independently.
 */
static int qmax_of(int32_t bits) { return (1 << (bits - 1)) - 1; }

static int bits_ok(int32_t bits) { return bits == 8 || bits == 4 || bits == 2; }

static float bf16_bits_to_f32(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

size_t oracle_qrecord_bytes(int32_t block_size, int32_t head_dim, int32_t bits)
{
    return 2 * (size_t)block_size * head_dim * bits / 8 + 8 * (size_t)block_size;
}

int oracle_kv_quantize_row(const uint16_t *x, int32_t d, int32_t bits, int32_t *codes, float *scale_out)
{
    if (!bits_ok(bits))
        return -1;
    float amax = 0.0f;
    for (int32_t i = 0; i < d; ++i) {
        const float a = fabsf(bf16_bits_to_f32(x[i]));
        if (a > amax)
            amax = a;
    }
    const float qm = (float)qmax_of(bits);
    const float scale = amax / qm;
    for (int32_t i = 0; i < d; ++i) {
        int32_t c = 0;
        if (scale > 0.0f) {
            float y = rintf(bf16_bits_to_f32(x[i]) / scale);
            if (y > qm)
                y = qm;
            if (y < -qm)
                y = -qm;
            c = (y == y) ? (int32_t)y : 0;
        }
        codes[i] = c;
    }
    *scale_out = scale;
    return 0;
}

/* byte offset of the code of (slot t, dim i) in section sec (0 = K, 1 = V), and
 * the shift of a 4-bit code within that byte */
static size_t qcode_pos(int sec, int32_t t, int32_t i, int32_t D, int32_t BS, int32_t bits, int *shift)
{
    const size_t C = (size_t)BS * D * bits / 8;
    size_t byte;
    if (sec == 0) {
        const int mt = t / 16, g = (t % 16) / 2, r = t % 2;
        const int j = i / 16, s = i % 16, c = (s % 8) / 2, h = s / 8, e = s % 2, u = 4 * g + c;
        if (bits == 8) {
            byte = ((size_t)(mt * (D / 32) + j / 2) * 32 + u) * 16 + (size_t)((j % 2) * 2 + r) * 4 + h + 2 * e;
            *shift = 0;
        } else if (bits == 2) {
            const int bit = 8 * r + 2 * (2 * (j % 2) + h) + 16 * e;
            byte = (size_t)(mt * 32 + u) * (D / 8) + (size_t)(j / 2) * 4 + bit / 8;
            *shift = bit % 8;
        } else {
            const int bit = 4 * (2 * r + h) + 16 * e;
            byte = ((size_t)(mt * (D / 64) + j / 4) * 32 + u) * 16 + (size_t)(j % 4) * 4 + bit / 8;
            *shift = bit % 8;
        }
    } else {
        const int kk = t / 16, m = (t % 16) / 2 + 8 * (t % 2), h = m / 8, c = (m % 8) / 2, e = m % 2;
        const int dm = i / 16, g = i % 8, r = (i % 16) / 8, u = 4 * g + c;
        if (bits == 8) {
            byte = C + ((size_t)(kk * (D / 32) + dm / 2) * 32 + u) * 16 + (size_t)((dm % 2) * 2 + r) * 4 + h + 2 * e;
            *shift = 0;
        } else if (bits == 2) {
            const int bit = 8 * h + 2 * (2 * (dm % 2) + r) + 16 * e;
            byte = C + (size_t)(kk * 32 + u) * (D / 8) + (size_t)(dm / 2) * 4 + bit / 8;
            *shift = bit % 8;
        } else {
            const int bit = 4 * (2 * h + r) + 16 * e;
            byte = C + ((size_t)(kk * (D / 64) + dm / 4) * 32 + u) * 16 + (size_t)(dm % 4) * 4 + bit / 8;
            *shift = bit % 8;
        }
    }
    return byte;
}

/* offset of the code of (sec, t, i) in a record; exported so tests can check the
 * layout is a bijection onto the code sections */
int64_t oracle_qcode_offset(int32_t sec, int32_t t, int32_t i, int32_t head_dim, int32_t block_size,
                            int32_t bits, int32_t *shift)
{
    int sh = 0;
    const size_t b = qcode_pos(sec, t, i, head_dim, block_size, bits, &sh);
    if (shift)
        *shift = sh;
    return (int64_t)b;
}

static void qrecord_put(uint8_t *rec, int sec, int32_t t, const int32_t *codes, float scale,
                        int32_t D, int32_t BS, int32_t bits)
{
    for (int32_t i = 0; i < D; ++i) {
        int shift = 0;
        const size_t b = qcode_pos(sec, t, i, D, BS, bits, &shift);
        if (bits == 8) {
            rec[b] = (uint8_t)(codes[i] + 128);
        } else {
            const int q = qmax_of(bits) + 1, mask = 2 * q - 1;   /* field c + q: 0xF or 0x3 */
            const uint8_t field = (uint8_t)(codes[i] + q);
            rec[b] = (uint8_t)((rec[b] & ~(mask << shift)) | (field << shift));
        }
    }
    const size_t C = (size_t)BS * D * bits / 8;
    memcpy(rec + 2 * C + (size_t)sec * 4 * BS + 4 * (size_t)t, &scale, sizeof scale);
}

static double qrecord_get(const uint8_t *rec, int sec, int32_t t, int32_t i, int32_t D, int32_t BS, int32_t bits)
{
    int shift = 0;
    const size_t b = qcode_pos(sec, t, i, D, BS, bits, &shift);
    int32_t c;
    if (bits == 8) {
        c = (int32_t)rec[b] - 128;
    } else {
        const int q = qmax_of(bits) + 1;
        c = (int32_t)((rec[b] >> shift) & (2 * q - 1)) - q;
    }
    float scale;
    const size_t C = (size_t)BS * D * bits / 8;
    memcpy(&scale, rec + 2 * C + (size_t)sec * 4 * BS + 4 * (size_t)t, sizeof scale);
    return (double)c * (double)scale;
}

static void kv_read_row(const struct kv_source *src, int32_t blk, int32_t g, int32_t off,
                        int32_t Hkv, int32_t B, int32_t D, double *k, double *v)
{
    if (src->records) {
        const size_t rb = oracle_qrecord_bytes(B, D, src->bits);
        const uint8_t *rec = src->records + ((size_t)blk * Hkv + g) * rb;
        for (int32_t i = 0; i < D; ++i) {
            k[i] = qrecord_get(rec, 0, off, i, D, B, src->bits);
            v[i] = qrecord_get(rec, 1, off, i, D, B, src->bits);
        }
        return;
    }
    const size_t base = ((((size_t)blk * Hkv) + g) * B + (size_t)off) * D;
    for (int32_t i = 0; i < D; ++i) {
        k[i] = bf16_bits_to_f64(src->k_pool[base + i]);
        v[i] = bf16_bits_to_f64(src->v_pool[base + i]);
    }
}

/*
 * Quantising scatter-append: the slot of new token i of sequence s is found as in
 * oracle_paged_kv_append; its K row and V row of every KV head are quantised as
 * above and written into the record of (block, head).  Returns 0, -1 (position
 * beyond the table), -2 (block id out of range), -3 (bits not 8, 4 or 2).
 */
int oracle_paged_kv_append_quant(uint8_t *records, int32_t num_blocks, int32_t block_size,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t bits,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *context_lens_old, const int32_t *new_starts,
                                 const uint16_t *k_new, const uint16_t *v_new, int32_t num_seqs)
{
    if (!bits_ok(bits))
        return -3;
    const size_t rb = oracle_qrecord_bytes(block_size, head_dim, bits);
    int32_t *codes = (int32_t *)malloc(sizeof(int32_t) * (size_t)head_dim);
    if (!codes)
        return -4;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int32_t n_new = new_starts[s + 1] - new_starts[s];
        for (int32_t i = 0; i < n_new; ++i) {
            const int64_t p = (int64_t)context_lens_old[s] + i;
            const int64_t logical = p / block_size;
            if (logical >= max_blocks_per_seq) {
                free(codes);
                return -1;
            }
            const int32_t blk = block_tables[(int64_t)s * max_blocks_per_seq + logical];
            if (blk < 0 || blk >= num_blocks) {
                free(codes);
                return -2;
            }
            const int64_t row = (int64_t)new_starts[s] + i;
            for (int32_t h = 0; h < num_kv_heads; ++h) {
                uint8_t *rec = records + ((size_t)blk * num_kv_heads + h) * rb;
                const size_t src = (((size_t)row * num_kv_heads) + h) * head_dim;
                float scale;
                oracle_kv_quantize_row(k_new + src, head_dim, bits, codes, &scale);
                qrecord_put(rec, 0, (int32_t)(p % block_size), codes, scale, head_dim, block_size, bits);
                oracle_kv_quantize_row(v_new + src, head_dim, bits, codes, &scale);
                qrecord_put(rec, 1, (int32_t)(p % block_size), codes, scale, head_dim, block_size, bits);
            }
        }
    }
    free(codes);
    return 0;
}

/* Every record read back: k_out, v_out float64 [num_blocks][H_kv][block_size][head_dim]. */
void oracle_qpool_dequant(const uint8_t *records, int32_t num_blocks, int32_t block_size,
                          int32_t num_kv_heads, int32_t head_dim, int32_t bits,
                          double *k_out, double *v_out)
{
    struct kv_source src = {NULL, NULL, records, bits};
    for (int32_t b = 0; b < num_blocks; ++b)
        for (int32_t g = 0; g < num_kv_heads; ++g)
            for (int32_t t = 0; t < block_size; ++t) {
                const size_t o = ((((size_t)b * num_kv_heads) + g) * block_size + t) * head_dim;
                kv_read_row(&src, b, g, t, num_kv_heads, block_size, head_dim, k_out + o, v_out + o);
            }
}

/*
 * Attention over quantised blocks: the definition of oracle_paged_attention with
 * K and V read back from the records (c * scale, exact in float64).
 */
int oracle_paged_attention_quant(const uint8_t *records, int32_t bits,
                                 int32_t num_blocks, int32_t block_size,
                                 int32_t num_kv_heads, int32_t head_dim,
                                 const uint16_t *q, const int32_t *q_starts,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *context_lens, int32_t num_seqs,
                                 int32_t num_q_heads, const int32_t *kv_head_of_q_head,
                                 const float *sinks, int32_t causal, const uint32_t *tree_masks,
                                 double scale, double *out, int32_t num_threads)
{
    if (!bits_ok(bits))
        return -6;
    struct kv_source src = {NULL, NULL, records, bits};
    return attention_core(&src, num_blocks, block_size, num_kv_heads, head_dim, q, q_starts,
                          block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                          kv_head_of_q_head, sinks, causal, tree_masks, scale, out, num_threads);
}

/* ------------------------------------------------- index-list (sparse) gather -- */
/*
 * Attention over an explicit list of key positions (TensorSharp "高级功能", the
 * DeepSeek V4 executor item: decode attention takes a compact [ring | top-512]
 * set of keys through a fused index-gather instead of scanning the whole
 * context).  Query row r of sequence s, q head h (KV head g = map[h]) attends to
 * the keys at positions key_idx[r][0 .. key_counts[r]-1] of s, each read through
 * the block table (block_tables[s][t / B], slot t % B):
 *   x_j = scale * q[r][h] . K_s[key_idx[r][j]][g]
 *   out = sum_j e^{x_j - M} V_s[key_idx[r][j]][g] / (sum_j e^{x_j - M} + e^{sink_h - M})
 * over j in list order (a position listed twice counts twice); M = max(x_j, sink_h).
 * No causal mask: the list says what the row sees.  key_idx is int32
 * [R][max_keys]; rows of s are q_starts[s] .. q_starts[s+1]-1.  Every position must
 * lie in [0, context_lens[s]).  Returns 0, -1 (a position outside [0, L) or past
 * the table), -2 (block id out of range), -3 (bad head map), -4 (out of memory),
 * -6 (a count outside [0, max_keys]).
 */
int oracle_paged_attention_sparse(const uint16_t *k_pool, const uint16_t *v_pool,
                                  int32_t num_blocks, int32_t block_size,
                                  int32_t num_kv_heads, int32_t head_dim,
                                  const uint16_t *q, const int32_t *q_starts,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *context_lens, int32_t num_seqs,
                                  const int32_t *key_idx, const int32_t *key_counts, int32_t max_keys,
                                  int32_t num_q_heads, const int32_t *kv_head_of_q_head,
                                  const float *sinks, double scale, double *out)
{
    const int32_t B = block_size, D = head_dim, Hkv = num_kv_heads, Hq = num_q_heads;
    if (Hkv <= 0 || Hq % Hkv != 0)
        return -3;
    const int32_t group = Hq / Hkv;
    for (int32_t h = 0; h < Hq; ++h) {
        const int32_t g = kv_head_of_q_head ? kv_head_of_q_head[h] : h / group;
        if (g < 0 || g >= Hkv)
            return -3;
    }
    double *K = (double *)malloc(sizeof(double) * (size_t)(max_keys > 0 ? max_keys : 1) * D);
    double *V = (double *)malloc(sizeof(double) * (size_t)(max_keys > 0 ? max_keys : 1) * D);
    double *x = (double *)malloc(sizeof(double) * (size_t)(max_keys > 0 ? max_keys : 1));
    if (!K || !V || !x) {
        free(K); free(V); free(x);
        return -4;
    }
    int rc = 0;
    for (int32_t s = 0; s < num_seqs && rc == 0; ++s) {
        const int64_t L = context_lens[s];
        for (int64_t r = q_starts[s]; r < q_starts[s + 1] && rc == 0; ++r) {
            const int32_t n = key_counts[r];
            if (n < 0 || n > max_keys) {
                rc = -6;
                break;
            }
            for (int32_t g = 0; g < Hkv && rc == 0; ++g) {
                /* gather this row's keys for KV head g */
                for (int32_t j = 0; j < n; ++j) {
                    const int64_t t = key_idx[r * (int64_t)max_keys + j];
                    if (t < 0 || t >= L || t / B >= max_blocks_per_seq) {
                        rc = -1;
                        break;
                    }
                    const int32_t blk = block_tables[(int64_t)s * max_blocks_per_seq + t / B];
                    if (blk < 0 || blk >= num_blocks) {
                        rc = -2;
                        break;
                    }
                    const size_t base = ((((size_t)blk * Hkv) + g) * B + (size_t)(t % B)) * D;
                    for (int32_t i = 0; i < D; ++i) {
                        K[(size_t)j * D + i] = bf16_bits_to_f64(k_pool[base + i]);
                        V[(size_t)j * D + i] = bf16_bits_to_f64(v_pool[base + i]);
                    }
                }
                if (rc)
                    break;
                for (int32_t h = 0; h < Hq; ++h) {
                    const int32_t gh = kv_head_of_q_head ? kv_head_of_q_head[h] : h / group;
                    if (gh != g)
                        continue;
                    const uint16_t *qv = q + ((size_t)r * Hq + h) * D;
                    double *o = out + ((size_t)r * Hq + h) * D;
                    double M = -INFINITY;
                    for (int32_t j = 0; j < n; ++j) {
                        double dot = 0.0;
                        for (int32_t i = 0; i < D; ++i)
                            dot += bf16_bits_to_f64(qv[i]) * K[(size_t)j * D + i];
                        x[j] = scale * dot;
                        if (x[j] > M)
                            M = x[j];
                    }
                    const int has_sink = sinks != NULL;
                    const double sink = has_sink ? (double)sinks[h] : 0.0;
                    if (has_sink && sink > M)
                        M = sink;
                    double den = 0.0;
                    for (int32_t i = 0; i < D; ++i)
                        o[i] = 0.0;
                    for (int32_t j = 0; j < n; ++j) {
                        const double e = exp(x[j] - M);
                        den += e;
                        for (int32_t i = 0; i < D; ++i)
                            o[i] += e * V[(size_t)j * D + i];
                    }
                    if (has_sink)
                        den += exp(sink - M);
                    for (int32_t i = 0; i < D; ++i)
                        o[i] = den > 0.0 ? o[i] / den : 0.0;
                }
            }
        }
    }
    free(K);
    free(V);
    free(x);
    return rc;
}

/*
 * Block allocation with prefix sharing (TensorSharp "高级功能", section "连续批处理与分页
 * KV 缓存": KV blocks of fixed size come from one shared pool, and every full block is
 * content-hashed so that identical prefixes share physical blocks; a partial block is
 * never shared).  This is the sequential engine step the GPU call replaces, written as a
 * plain loop over the sequences in order and, within a sequence, over its blocks in order:
 *
 *   sequence s holds L = context_lens[s] tokens in nb = ceil(L / B) blocks, of which the
 *   first nk = floor(L / B) are full and carry the keys block_keys[s][j] (the chained
 *   keys of paged_block_hashes); blocks j < first_block[s] are already allocated and
 *   are left alone.  For j = first_block[s] .. nb - 1:
 *     - a full block whose key is in the index with a block id: that block is shared
 *       (table entry = its id, its reference count + 1, not fresh);
 *     - a full block whose key is not (or whose earlier allocation failed in a previous
 *       call): the key enters the index and takes a block popped from the free stack
 *       (reference count 1, fresh: the caller must fill it); later blocks with that key
 *       in this call share it;
 *     - a partial block, or a full block whose key equals the reserved empty key
 *       (all bits set), takes a private block popped from the stack (fresh).
 *   The free stack holds free_ids[0 .. F-1]; the k-th pop of the call (k = 0, 1, ...)
 *   takes free_ids[F - 1 - k].  A pop past the stack's end gives -1 and sets the
 *   out-of-blocks bit (128); a key whose pop failed stays in the index without a block
 *   (id -1) and its later occurrences in this call get -1 too.  A length needing more
 *   than max_blocks blocks is cut to max_blocks and sets the table-overrun bit (2).
 *
 * The index is a list of n entries (key, id, refcount) with room for cap; it is searched
 * linearly (this is the definition, not a fast map).  fresh [S][max_blocks] is set to 1
 * for every block this call allocated and 0 elsewhere.  Returns 0, or -1 when the index
 * has no room (cap entries) for a new key.
 */
int oracle_block_allocate(uint64_t *ix_keys, int32_t *ix_ids, int32_t *ix_refs, int32_t *n_entries, int32_t cap,
                          const int32_t *free_ids, int32_t *free_count, const uint64_t *block_keys,
                          const int32_t *context_lens, const int32_t *first_block, int32_t num_seqs,
                          int32_t block_size, int32_t max_blocks, int32_t *block_tables, int32_t *fresh,
                          int32_t *status_bits)
{
    const uint64_t kEmpty = ~0ull;
    const int32_t F = *free_count;
    int64_t pops = 0;
    int32_t n = *n_entries;
    int32_t bits = 0;
    uint8_t *touched = (uint8_t *)calloc((size_t)(cap > 0 ? cap : 1), 1);
    if (!touched)
        return -1;
    for (int64_t e = 0; e < (int64_t)num_seqs * max_blocks; ++e)
        fresh[e] = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int64_t L = context_lens[s] < 0 ? 0 : context_lens[s];
        int64_t nb = (L + block_size - 1) / block_size;
        int64_t nk = L / block_size;
        if (nb > max_blocks) {
            nb = max_blocks;
            bits |= 2;
        }
        if (nk > nb)
            nk = nb;
        const int64_t j0 = first_block[s] < 0 ? 0 : first_block[s];
        for (int64_t j = j0; j < nb; ++j) {
            const int64_t e = (int64_t)s * max_blocks + j;
            int32_t id = -1;
            int32_t is_fresh = 0;
            const uint64_t key = block_keys[e];
            if (j < nk && key != kEmpty) {
                int32_t i = -1;
                for (int32_t k = 0; k < n; ++k)
                    if (ix_keys[k] == key) {
                        i = k;
                        break;
                    }
                if (i >= 0 && ix_ids[i] >= 0) {          /* shared: an earlier allocation of this key */
                    id = ix_ids[i];
                    ix_refs[i] += 1;
                } else if (i >= 0 && touched[i]) {       /* its allocation failed earlier in this call */
                    id = -1;
                } else {                                 /* a new key: pop a block for it */
                    if (i < 0) {
                        if (n >= cap) {
                            free(touched);
                            return -1;
                        }
                        i = n++;
                        ix_keys[i] = key;
                        ix_ids[i] = -1;
                        ix_refs[i] = 0;
                    }
                    touched[i] = 1;
                    if (pops < F) {
                        id = free_ids[F - 1 - pops];
                        ix_ids[i] = id;
                        ix_refs[i] = 1;
                        is_fresh = 1;
                    } else {
                        bits |= 128;
                    }
                    ++pops;
                }
            } else {                                     /* a private block */
                if (pops < F) {
                    id = free_ids[F - 1 - pops];
                    is_fresh = 1;
                } else {
                    bits |= 128;
                }
                ++pops;
            }
            block_tables[e] = id;
            fresh[e] = is_fresh;
        }
    }
    *free_count = pops < F ? (int32_t)(F - pops) : 0;
    *n_entries = n;
    *status_bits = bits;
    free(touched);
    return 0;
}
