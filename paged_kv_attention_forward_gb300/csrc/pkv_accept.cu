// pkv_accept.cu -- greedy speculative accept on the device.
//
// TensorFold article, section "接受规则：GPU 上的 accept 内核": the accept kernel
// compares each draft token with the target's choice and follows the chain to
// the first mismatch, writing its outcome to a small arena; TensorSharp
// "高级功能", DFlash paragraph: the argmax runs on the device so the
// vocabulary-wide block never crosses PCIe.
//
// Kernel 1 (argmax_chunks): grid (chunks, rows).  Each CTA scans one slice of one
//   row with 16-byte loads and reduces (value, index) pairs -- larger value wins,
//   equal values go to the lower index -- with warp shuffles, then across warps.
//   That order is total, so the result does not depend on the slicing.
// Kernel 2 (accept_walk): one warp per sequence merges the slices of each row
//   (same order), writes argmax_out, finds the first mismatching draft with a
//   ballot, and writes accept_len and out_tokens.
#include <cfloat>
#include <mutex>

#include "pkv_internal.h"

namespace pkv {
namespace {

struct Best {
    float v;
    int i;
};

__device__ __forceinline__ Best better(Best a, Best b)
{
    // b wins on a strictly larger value, or an equal value at a lower index
    return (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
}

__device__ __forceinline__ Best warp_best(Best b)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Best o;
        o.v = __shfl_xor_sync(0xffffffffu, b.v, off);
        o.i = __shfl_xor_sync(0xffffffffu, b.i, off);
        b = better(b, o);
    }
    return b;
}

constexpr int kArgmaxThreads = 256;
constexpr int kNoIndex = 0x7fffffff;

__global__ void __launch_bounds__(kArgmaxThreads)
argmax_chunks_kernel(const float *__restrict__ logits, int vocab, int chunk, int n_chunks,
                     float2 *__restrict__ part, int vec_ok)
{
    const int c = blockIdx.x, r = blockIdx.y;
    const int lo = c * chunk;
    const int hi = min(vocab, lo + chunk);
    const float *row = logits + (size_t)r * vocab;
    Best b = {-INFINITY, kNoIndex};
    if (vec_ok) {
        // lo and hi are multiples of 4 except possibly hi == vocab (vocab % 4 == 0 when vec_ok)
        const float4 *row4 = reinterpret_cast<const float4 *>(row);
        const int lo4 = lo >> 2, hi4 = hi >> 2;
#pragma unroll 8
        for (int i = lo4 + threadIdx.x; i < hi4; i += kArgmaxThreads) {
            const float4 x = __ldcs(row4 + i);
            const int base = i << 2;
            b = better(b, Best{x.x, base});
            b = better(b, Best{x.y, base + 1});
            b = better(b, Best{x.z, base + 2});
            b = better(b, Best{x.w, base + 3});
        }
    } else {
        for (int i = lo + threadIdx.x; i < hi; i += kArgmaxThreads)
            b = better(b, Best{__ldcs(row + i), i});
    }
    b = warp_best(b);
    __shared__ Best sm[kArgmaxThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        sm[warp] = b;
    __syncthreads();
    if (warp == 0) {
        b = lane < kArgmaxThreads / 32 ? sm[lane] : Best{-INFINITY, kNoIndex};
        b = warp_best(b);
        if (lane == 0)
            part[(size_t)r * n_chunks + c] = make_float2(b.v, __int_as_float(b.i));
    }
}

__global__ void __launch_bounds__(32)
accept_walk_kernel(const float2 *__restrict__ part, int n_chunks, const int32_t *__restrict__ q_starts,
                   const int32_t *__restrict__ drafts, int total_rows, int32_t *__restrict__ argmax_out,
                   int32_t *__restrict__ accept_len, int32_t *__restrict__ out_tokens,
                   int32_t *__restrict__ status)
{
    const int s = blockIdx.x, lane = threadIdx.x;
    const int r0 = q_starts[s], W = q_starts[s + 1] - r0;
    if (W <= 0) {
        if (lane == 0)
            accept_len[s] = -1;
        return;
    }
    if (r0 < 0 || r0 + W > total_rows) {   // q_starts inconsistent with total_rows
        if (lane == 0) {
            accept_len[s] = -1;
            atomicOr(status, PKV_DEV_TOO_MANY_ROWS);
        }
        return;
    }
    int n = -1, a_n = 0;
    for (int base = 0; base < W; base += 32) {
        const int j = base + lane;
        int a = 0;
        bool stop = false;
        if (j < W) {
            Best b = {-INFINITY, kNoIndex};
            const float2 *pr = part + (size_t)(r0 + j) * n_chunks;
            for (int c = 0; c < n_chunks; ++c) {
                const float2 x = pr[c];
                b = better(b, Best{x.x, __float_as_int(x.y)});
            }
            a = b.i == kNoIndex ? 0 : b.i;
            argmax_out[r0 + j] = a;
            stop = (j == W - 1) || (drafts[r0 + j + 1] != a);
        }
        if (n < 0) {
            const unsigned m = __ballot_sync(0xffffffffu, stop);
            if (m) {
                const int first = __ffs(m) - 1;
                n = base + first;
                a_n = __shfl_sync(0xffffffffu, a, first);
            }
        }
    }
    // n is found: every row stops at the window end at the latest
    for (int j = lane; j < W; j += 32)
        out_tokens[r0 + j] = j < n ? drafts[r0 + j + 1] : (j == n ? a_n : -1);
    if (lane == 0)
        accept_len[s] = n;
}

// ---- keyed sampling (draws keyed by seed, absolute position and token id) ----
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): 10 rounds of multiply-xor on
// words 0 and 2, key bumped by the Weyl constants before every round but the first.
__device__ __forceinline__ void philox4x32_10(uint32_t (&c)[4], uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c[0], hi0 = __umulhi(0xD2511F53u, c[0]);
        const uint32_t lo1 = 0xCD9E8D57u * c[2], hi1 = __umulhi(0xCD9E8D57u, c[2]);
        const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
    }
}

// Natural log in float32 as a fixed sequence of correctly rounded operations (no
// contraction into FMA): x = m 2^e, m in [sqrt(1/2), sqrt(2)), s = (m-1)/(m+1),
// log x = e ln2 + 2s (1 + s^2/3 + ... + s^10/11) with float32 coefficients.
__device__ __forceinline__ float keyed_log(float x)
{
    uint32_t b = __float_as_uint(x);
    int e;
    if ((b >> 23) == 0) {
        x = __fmul_rn(x, 8388608.0f);
        b = __float_as_uint(x);
        e = (int)(b >> 23) - 127 - 23;
    } else {
        e = (int)(b >> 23) - 127;
    }
    float m = __uint_as_float((b & 0x7fffffu) | 0x3f800000u);
    if (m > 0x1.6a09e6p+0f) {
        m = __fmul_rn(m, 0.5f);
        e += 1;
    }
    const float sv = __fdiv_rn(__fsub_rn(m, 1.0f), __fadd_rn(m, 1.0f));
    const float z = __fmul_rn(sv, sv);
    float q = 0x1.745d18p-4f;
    q = __fadd_rn(__fmul_rn(q, z), 0x1.c71c72p-4f);
    q = __fadd_rn(__fmul_rn(q, z), 0x1.24924ap-3f);
    q = __fadd_rn(__fmul_rn(q, z), 0x1.99999ap-3f);
    q = __fadd_rn(__fmul_rn(q, z), 0x1.555556p-2f);
    q = __fadd_rn(__fmul_rn(q, z), 1.0f);
    const float rr = __fmul_rn(__fadd_rn(sv, sv), q);
    return __fadd_rn(__fmul_rn(__int2float_rn(e), 0x1.62e43p-1f), rr);
}

// Gumbel noise from the top 23 bits of one Philox output word.
__device__ __forceinline__ float gumbel_of(uint32_t w)
{
    const float u = __fmul_rn(__fadd_rn(__uint2float_rn(w >> 9), 0.5f), 0x1p-23f);
    return -keyed_log(-keyed_log(u));
}

// ---- top-k / top-p: the kept tokens are a prefix of the order (logit descending,
// token id ascending).  A token's place in that order is its 64-bit key
// (~ascending-float-bits(l) << 32) | v, so the kept set is {v : key_v <= cut}.
__device__ __forceinline__ uint64_t order_key(float l, int v)
{
    uint32_t b = __float_as_uint(l == 0.f ? 0.f : l);   // -0 and +0 are one logit
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);     // ascending with the float
    return ((uint64_t)~b << 32) | (uint32_t)v;
}

// 2^y for y <= 0 as a fixed float32 sequence: 0 below -32; else n = floor(y),
// f = y - n, the degree-8 Taylor polynomial of e^{f ln 2} (float32 coefficients
// (ln 2)^k / k!) by Horner's rule with separately rounded steps, times 2^n.
__device__ __forceinline__ float keyed_exp2(float y)
{
    if (!(y >= -32.0f))
        return 0.0f;
    if (y >= 0.0f)
        return 1.0f;
    const float n = floorf(y);
    const float f = __fsub_rn(y, n);
    float p = 0x1.62c022p-20f;
    p = __fadd_rn(__fmul_rn(p, f), 0x1.ffcbfcp-17f);
    p = __fadd_rn(__fmul_rn(p, f), 0x1.430912p-13f);
    p = __fadd_rn(__fmul_rn(p, f), 0x1.5d87fep-10f);
    p = __fadd_rn(__fmul_rn(p, f), 0x1.3b2ab6p-7f);
    p = __fadd_rn(__fmul_rn(p, f), 0x1.c6b08ep-5f);
    p = __fadd_rn(__fmul_rn(p, f), 0x1.ebfbe0p-3f);
    p = __fadd_rn(__fmul_rn(p, f), 0x1.62e430p-1f);
    p = __fadd_rn(__fmul_rn(p, f), 1.0f);
    return __fmul_rn(p, __int_as_float((127 + (int)n) << 23));
}

// Integer weight floor(2^32 * 2^(((l - l_max) / T) log2 e)): sums of weights are exact.
__device__ __forceinline__ uint64_t keyed_weight(float l, float l_max, float temperature)
{
    const float y = __fmul_rn(__fdiv_rn(__fsub_rn(l, l_max), temperature), 0x1.715476p+0f);
    return __float2ull_rz(__fmul_rn(keyed_exp2(y), 4294967296.0f));
}

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelCap = 2048;   // candidates kept in shared memory once they are this few
constexpr int kSelBins = 16;    // 4-bit digits: every thread keeps its own histogram
static_assert(kSelWarps % kSelBins == 0, "whole warps sum each bin");

struct SelSmem {
    unsigned long long hw[kSelBins][kSelThreads];   // per-thread weight histograms
    unsigned int hc[kSelBins][kSelThreads];         // per-thread candidate counts
    float cl[kSelCap];                               // compacted candidates: logit, token
    int cv[kSelCap];
    unsigned long long pw[kSelWarps];                // per-warp shares of the bin sums
    unsigned int pc[kSelWarps];
    unsigned long long bw[kSelBins];                 // the pass's totals per bin
    unsigned int bc[kSelBins];
    uint64_t bcast[3];
    unsigned int n_list;
};

// Smallest key K with (sum of w_v over key_v <= K) >= need, w_v = the token's weight
// (or 1 when COUNT).  Sixteen passes of 4 bits from the top; in each, every thread
// histograms the candidates it visits into its own row of shared memory (no atomics),
// and the 16 bins are then summed.  Once the candidates are at most kSelCap they are
// copied to shared memory and later passes read only them.  For the weighted select
// `need` comes from the row total, found in pass 0: ceil(p_fix * total / 2^32) (at
// least 1).  Integer sums make the result independent of the order of the adds.
// prelisted: the candidates are already in sm.cl / sm.cv and `need` is final.
template <bool COUNT>
__device__ uint64_t select_key(const float *__restrict__ row, int vocab, float l_max, float temperature,
                               uint64_t need, uint64_t p_fix, SelSmem &sm, bool prelisted = false)
{
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    uint64_t prefix = 0;
    bool listed = prelisted;        // candidates live in sm.cl / sm.cv
    uint32_t n_cand = prelisted ? sm.n_list : (uint32_t)vocab;
    __syncthreads();
    if (t == 0 && !prelisted)
        sm.n_list = 0;
    for (int pass = 0; pass < 16; ++pass) {
        const int shift = 60 - 4 * pass;
        const bool compact = !listed && n_cand <= (uint32_t)kSelCap;
#pragma unroll
        for (int b = 0; b < kSelBins; ++b) {
            if (!COUNT)
                sm.hw[b][t] = 0ull;
            sm.hc[b][t] = 0u;
        }
        __syncthreads();
        auto visit = [&](float l, int v) {
            const uint64_t key = order_key(l, v);
            if (pass > 0 && (key >> (shift + 4)) != prefix)
                return;
            if (compact) {
                const unsigned int at = atomicAdd(&sm.n_list, 1u);
                sm.cl[at] = l;
                sm.cv[at] = v;
            }
            const int bin = (int)((key >> shift) & 15);
            if (!COUNT)
                sm.hw[bin][t] += keyed_weight(l, l_max, temperature);
            sm.hc[bin][t] += 1u;
        };
        if (listed) {
            const int n = (int)sm.n_list;
            for (int i = t; i < n; i += kSelThreads)
                visit(sm.cl[i], sm.cv[i]);
        } else if ((vocab & 3) == 0) {
            // the whole row: four 16-byte loads in flight per thread
            const float4 *row4 = reinterpret_cast<const float4 *>(row);
            const int n4 = vocab >> 2;
            for (int i0 = t; i0 < n4; i0 += 4 * kSelThreads) {
                float4 x[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * kSelThreads;
                    x[u] = i < n4 ? __ldg(row4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * kSelThreads;
                    if (i < n4) {
                        visit(x[u].x, 4 * i);
                        visit(x[u].y, 4 * i + 1);
                        visit(x[u].z, 4 * i + 2);
                        visit(x[u].w, 4 * i + 3);
                    }
                }
            }
        } else {
            for (int i = t; i < vocab; i += kSelThreads)
                visit(__ldg(row + i), i);
        }
        __syncthreads();
        // the warps of group w sum bin w over the threads, each warp a share of them
        {
            constexpr int kPer = kSelWarps / kSelBins;
            const int bin = warp / kPer, part = warp % kPer;
            unsigned long long sw = 0;
            unsigned int sc = 0;
            for (int i = part * 32 + lane; i < kSelThreads; i += 32 * kPer) {
                if (!COUNT)
                    sw += sm.hw[bin][i];
                sc += sm.hc[bin][i];
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                sw += __shfl_xor_sync(0xffffffffu, sw, off);
                sc += __shfl_xor_sync(0xffffffffu, sc, off);
            }
            if (lane == 0) {
                sm.pw[warp] = COUNT ? (unsigned long long)sc : sw;
                sm.pc[warp] = sc;
            }
        }
        __syncthreads();
        if (t < kSelBins) {
            constexpr int kPer = kSelWarps / kSelBins;
            unsigned long long sw = 0;
            unsigned int sc = 0;
            for (int q = 0; q < kPer; ++q) {
                sw += sm.pw[t * kPer + q];
                sc += sm.pc[t * kPer + q];
            }
            sm.bw[t] = sw;
            sm.bc[t] = sc;
        }
        __syncthreads();
        if (t == 0) {
            if (!COUNT && pass == 0 && !prelisted) {
                // the row total is the sum of every bin: the top-p threshold
                uint64_t total = 0;
                for (int b = 0; b < kSelBins; ++b)
                    total += sm.bw[b];
                const uint64_t lo = p_fix * total, hi = __umul64hi(p_fix, total);
                const uint64_t lo2 = lo + 0xFFFFFFFFull;
                need = ((hi + (lo2 < lo ? 1ull : 0ull)) << 32) | (lo2 >> 32);
                need = need ? need : 1ull;   // a zero threshold keeps the first token, as 1 does
            }
            uint64_t cum = 0;
            int b = 0;
            for (; b < kSelBins - 1; ++b) {
                if (cum + sm.bw[b] >= need)
                    break;
                cum += sm.bw[b];
            }
            sm.bcast[0] = (prefix << 4) | (uint64_t)b;
            sm.bcast[1] = need - cum;
            sm.bcast[2] = sm.bc[b];
        }
        __syncthreads();
        prefix = sm.bcast[0];
        need = sm.bcast[1];
        n_cand = (uint32_t)sm.bcast[2];
        listed = listed || compact;
        __syncthreads();
    }
    return prefix;
}

// One CTA per row: the cut key of top-k (k tokens) and of top-p (the shortest prefix
// whose weight reaches ceil(p_fix * total / 2^32)); the kept set is key <= min of the two.
__global__ void __launch_bounds__(kSelThreads)
topkp_cut_kernel(const float *__restrict__ logits, int vocab, const float2 *__restrict__ part_max, int n_chunks,
                 float temperature, int top_k, int use_p, unsigned long long p_fix,
                 unsigned long long *__restrict__ cut)
{
    extern __shared__ __align__(16) uint8_t sel_raw[];
    SelSmem &sm = *reinterpret_cast<SelSmem *>(sel_raw);
    const int r = blockIdx.x;
    const float *row = logits + (size_t)r * vocab;
    float l_max = -INFINITY;
    for (int i = 0; i < n_chunks; ++i)
        l_max = fmaxf(l_max, part_max[(size_t)r * n_chunks + i].x);
    uint64_t c = ~0ull;
    if (top_k > 0 && top_k < vocab)
        c = select_key<true>(row, vocab, l_max, temperature, (uint64_t)top_k, 0ull, sm);
    if (use_p && top_k > 0 && top_k <= kSelCap && c != ~0ull) {
        // top-p can only cut inside the k kept tokens: one scan for the row total and those
        // tokens, then the weighted select over them alone
        __shared__ unsigned long long tot_sh, kept_sh;
        __syncthreads();
        if (threadIdx.x == 0) {
            tot_sh = 0ull;
            kept_sh = 0ull;
            sm.n_list = 0;
        }
        __syncthreads();
        unsigned long long tot = 0, kept = 0;
        for (int v = threadIdx.x; v < vocab; v += kSelThreads) {
            const float l = __ldg(row + v);
            const uint64_t w = keyed_weight(l, l_max, temperature);
            tot += w;
            if (order_key(l, v) <= c) {
                kept += w;
                const unsigned int at = atomicAdd(&sm.n_list, 1u);
                sm.cl[at] = l;
                sm.cv[at] = v;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            tot += __shfl_xor_sync(0xffffffffu, tot, off);
            kept += __shfl_xor_sync(0xffffffffu, kept, off);
        }
        if ((threadIdx.x & 31) == 0) {
            atomicAdd(&tot_sh, tot);
            atomicAdd(&kept_sh, kept);
        }
        __syncthreads();
        const uint64_t total = tot_sh;
        const uint64_t lo = p_fix * total, hi = __umul64hi(p_fix, total);
        const uint64_t lo2 = lo + 0xFFFFFFFFull;
        uint64_t need = ((hi + (lo2 < lo ? 1ull : 0ull)) << 32) | (lo2 >> 32);
        need = need ? need : 1ull;
        if (need <= (uint64_t)kept_sh) {   // else top-p keeps all k tokens
            const uint64_t cp = select_key<false>(row, vocab, l_max, temperature, need, p_fix, sm, true);
            c = cp < c ? cp : c;
        }
    } else if (use_p) {
        const uint64_t cp = select_key<false>(row, vocab, l_max, temperature, 0ull, p_fix, sm);
        c = cp < c ? cp : c;
    }
    if (threadIdx.x == 0)
        cut[r] = c;
}

// Sampling pass: per (slice, row), the best l/T + g(seed, pos, v) over the kept tokens
// (l >= l_max + off, off = T log(min_p) or -inf, and key_v <= cut[r] when top-k / top-p
// are on), ties to the lowest token.  The row maximum comes from the argmax pass's
// slices.  Token v is keyed by word (v mod 4) of Philox(ctr = (v / 4, pos,
// 0x6b657964, 0), key = seed).
__global__ void __launch_bounds__(kArgmaxThreads)
sample_chunks_kernel(const float *__restrict__ logits, int vocab, int chunk, int n_chunks,
                     const float2 *__restrict__ part_max, float2 *__restrict__ part,
                     const int32_t *__restrict__ positions, uint32_t seed_lo, uint32_t seed_hi,
                     float temperature, float off, int vec_ok, const unsigned long long *__restrict__ cut)
{
    const int c = blockIdx.x, r = blockIdx.y;
    const int lo = c * chunk;
    const int hi = min(vocab, lo + chunk);
    const float *row = logits + (size_t)r * vocab;
    float l_max = -INFINITY;
    for (int i = 0; i < n_chunks; ++i)
        l_max = fmaxf(l_max, part_max[(size_t)r * n_chunks + i].x);
    const float thr = off == -INFINITY ? -INFINITY : __fadd_rn(l_max, off);
    const uint64_t kcut = cut ? cut[r] : ~0ull;
    const uint32_t pos = (uint32_t)__ldg(positions + r);
    Best b = {-INFINITY, kNoIndex};
    if (vec_ok) {
        const float4 *row4 = reinterpret_cast<const float4 *>(row);
        // four float4 loads in flight per thread, then the (rare) kept tokens; the result does
        // not depend on the visiting order (better() is a total order on (value, index))
        constexpr int U = 4;
        const int hi4 = hi >> 2;
        for (int i0 = (lo >> 2) + threadIdx.x; i0 < hi4; i0 += U * kArgmaxThreads) {
            float4 xv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = i0 + u * kArgmaxThreads;
                xv[u] = i < hi4 ? __ldcs(row4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = i0 + u * kArgmaxThreads;
                if (i >= hi4)
                    break;
                const float xs[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
                bool keep[4], any = false;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    keep[j] = xs[j] >= thr && order_key(xs[j], 4 * i + j) <= kcut;
                    any = any || keep[j];
                }
                if (!any)   // a token's draw depends only on (seed, position, token): skip unkept groups
                    continue;
                uint32_t w[4] = {(uint32_t)i, pos, 0x6b657964u, 0u};
                philox4x32_10(w, seed_lo, seed_hi);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (keep[j])
                        b = better(b, Best{__fadd_rn(__fdiv_rn(xs[j], temperature), gumbel_of(w[j])), 4 * i + j});
            }
        }
    } else {
        for (int v = lo + threadIdx.x; v < hi; v += kArgmaxThreads) {
            const float x = __ldcs(row + v);
            if (!(x >= thr) || order_key(x, v) > kcut)
                continue;
            uint32_t w[4] = {(uint32_t)v >> 2, pos, 0x6b657964u, 0u};
            philox4x32_10(w, seed_lo, seed_hi);
            const uint32_t word = (v & 3) == 0 ? w[0] : (v & 3) == 1 ? w[1] : (v & 3) == 2 ? w[2] : w[3];
            b = better(b, Best{__fadd_rn(__fdiv_rn(x, temperature), gumbel_of(word)), v});
        }
    }
    b = warp_best(b);
    __shared__ Best sm[kArgmaxThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        sm[warp] = b;
    __syncthreads();
    if (warp == 0) {
        b = lane < kArgmaxThreads / 32 ? sm[lane] : Best{-INFINITY, kNoIndex};
        b = warp_best(b);
        if (lane == 0)
            part[(size_t)r * n_chunks + c] = make_float2(b.v, __int_as_float(b.i));
    }
}

constexpr int kTreeMaxNodes = 1024;

// Accept over draft trees (or chains when parents is null): one warp per sequence.  The slices of each row are
// merged into argmax_out (and shared memory), then from the root the walk takes, at
// node u, the lowest-index child c (parents[c] == u) whose draft equals a_u, found by
// a ballot over 32 candidates at a time.
__global__ void __launch_bounds__(32)
accept_tree_walk_kernel(const float2 *__restrict__ part, int n_chunks, const int32_t *__restrict__ q_starts,
                        const int32_t *__restrict__ drafts, const int32_t *__restrict__ parents,
                        int total_rows, int32_t *__restrict__ argmax_out, int32_t *__restrict__ accept_len,
                        int32_t *__restrict__ out_tokens, int32_t *__restrict__ accepted_rows,
                        int32_t *__restrict__ status)
{
    __shared__ int32_t a_s[kTreeMaxNodes];
    const int s = blockIdx.x, lane = threadIdx.x;
    const int r0 = q_starts[s], W = q_starts[s + 1] - r0;
    if (W <= 0) {
        if (lane == 0)
            accept_len[s] = -1;
        return;
    }
    bool bad = r0 < 0 || r0 + W > total_rows || W > kTreeMaxNodes;
    for (int j = 1 + lane; parents && !bad && j < W; j += 32)
        if (parents[r0 + j] < 0 || parents[r0 + j] >= j)
            bad = true;
    if (__any_sync(0xffffffffu, bad)) {
        if (lane == 0) {
            accept_len[s] = -1;
            atomicOr(status, PKV_DEV_BAD_TREE);
        }
        return;
    }
    for (int j = lane; j < W; j += 32) {
        Best b = {-INFINITY, kNoIndex};
        const float2 *pr = part + (size_t)(r0 + j) * n_chunks;
        for (int c = 0; c < n_chunks; ++c) {
            const float2 x = pr[c];
            b = better(b, Best{x.x, __float_as_int(x.y)});
        }
        const int a = b.i == kNoIndex ? 0 : b.i;
        a_s[j] = a;
        argmax_out[r0 + j] = a;
        out_tokens[r0 + j] = -1;
        accepted_rows[r0 + j] = -1;
    }
    __syncwarp();
    int u = 0, n = 0;
    for (;;) {
        const int target = a_s[u];
        int next = -1;
        for (int base = u + 1; base < W && next < 0; base += 32) {
            const int c = base + lane;
            const bool hit = c < W && (parents ? parents[r0 + c] : c - 1) == u && drafts[r0 + c] == target;
            const unsigned m = __ballot_sync(0xffffffffu, hit);
            if (m)
                next = base + __ffs(m) - 1;
        }
        if (next < 0)
            break;
        if (lane == 0) {
            out_tokens[r0 + n] = drafts[r0 + next];
            accepted_rows[r0 + n] = next;
        }
        ++n;
        u = next;
    }
    if (lane == 0) {
        out_tokens[r0 + n] = a_s[u];
        accept_len[s] = n;
    }
}

int accept_chunks(int32_t total_rows, int32_t vocab, int sms)
{
    // enough CTAs to cover the GPU about four times, slices of at least 8192 values
    const int max_chunks = (vocab + 8191) / 8192;
    int want = (4 * sms + total_rows - 1) / (total_rows > 0 ? total_rows : 1);
    if (want < 1)
        want = 1;
    return want < max_chunks ? want : (max_chunks > 0 ? max_chunks : 1);
}

}  // namespace
}  // namespace pkv

extern "C" size_t spec_accept_workspace_size(int32_t total_rows, int32_t vocab)
{
    if (total_rows < 0 || vocab <= 0)
        return 0;
    const int max_chunks = (vocab + 8191) / 8192;
    return pkv::round_up((size_t)total_rows * max_chunks * sizeof(float2), 256) + 256;
}

extern "C" int spec_accept_greedy(const float *logits, int32_t vocab, const int32_t *q_starts,
                                  const int32_t *draft_tokens, int32_t num_seqs, int32_t total_rows,
                                  int32_t *argmax_out, int32_t *accept_len, int32_t *out_tokens,
                                  void *workspace, size_t workspace_bytes, void *stream)
{
    using namespace pkv;
    clear_error();
    if (num_seqs < 0 || total_rows < 0 || vocab <= 0)
        return set_error(PKV_ERR_SHAPE, "spec_accept_greedy: bad sizes (num_seqs %d, rows %d, vocab %d)",
                         num_seqs, total_rows, vocab);
    if (num_seqs == 0)
        return PKV_OK;
    if (!q_starts || !accept_len || (total_rows > 0 && (!logits || !draft_tokens || !argmax_out ||
                                                        !out_tokens || !workspace)))
        return set_error(PKV_ERR_NULL, "spec_accept_greedy: a required pointer is NULL");
    if (total_rows > 0 && !aligned16(logits))
        return set_error(PKV_ERR_ALIGN, "spec_accept_greedy: logits must be 16-byte aligned");
    if (workspace_bytes < spec_accept_workspace_size(total_rows, vocab))
        return set_error(PKV_ERR_WORKSPACE, "spec_accept_greedy: workspace %zu < %zu bytes", workspace_bytes,
                         spec_accept_workspace_size(total_rows, vocab));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int n_chunks = accept_chunks(total_rows, vocab, sm_count());
    float2 *part = static_cast<float2 *>(workspace);
    if (total_rows > 0) {
        if (total_rows > 65535)
            return set_error(PKV_ERR_SHAPE, "spec_accept_greedy: at most 65535 rows per call");
        int chunk = (vocab + n_chunks - 1) / n_chunks;
        chunk = (chunk + 3) & ~3;
        const int vec_ok = (vocab % 4) == 0;
        argmax_chunks_kernel<<<dim3(n_chunks, total_rows), kArgmaxThreads, 0, st>>>(logits, vocab, chunk,
                                                                                   n_chunks, part, vec_ok);
        const int rc = check_cuda(cudaGetLastError(), "spec_accept_greedy argmax launch");
        if (rc)
            return rc;
    }
    int32_t *status = device_status_word();
    if (!status)
        return set_error(PKV_ERR_CUDA, "spec_accept_greedy: no device status word");
    accept_walk_kernel<<<num_seqs, 32, 0, st>>>(part, n_chunks, q_starts, draft_tokens, total_rows, argmax_out,
                                                accept_len, out_tokens, status);
    return check_cuda(cudaGetLastError(), "spec_accept_greedy walk launch");
}

extern "C" int spec_accept_tree_greedy(const float *logits, int32_t vocab, const int32_t *q_starts,
                                       const int32_t *draft_tokens, const int32_t *parents, int32_t num_seqs,
                                       int32_t total_rows, int32_t *argmax_out, int32_t *accept_len,
                                       int32_t *out_tokens, int32_t *accepted_rows, void *workspace,
                                       size_t workspace_bytes, void *stream)
{
    using namespace pkv;
    clear_error();
    if (num_seqs < 0 || total_rows < 0 || vocab <= 0)
        return set_error(PKV_ERR_SHAPE, "spec_accept_tree_greedy: bad sizes (num_seqs %d, rows %d, vocab %d)",
                         num_seqs, total_rows, vocab);
    if (num_seqs == 0)
        return PKV_OK;
    if (!q_starts || !accept_len || (total_rows > 0 && (!logits || !draft_tokens || !parents || !argmax_out ||
                                                        !out_tokens || !accepted_rows || !workspace)))
        return set_error(PKV_ERR_NULL, "spec_accept_tree_greedy: a required pointer is NULL");
    if (total_rows > 0 && !aligned16(logits))
        return set_error(PKV_ERR_ALIGN, "spec_accept_tree_greedy: logits must be 16-byte aligned");
    if (workspace_bytes < spec_accept_workspace_size(total_rows, vocab))
        return set_error(PKV_ERR_WORKSPACE, "spec_accept_tree_greedy: workspace %zu < %zu bytes",
                         workspace_bytes, spec_accept_workspace_size(total_rows, vocab));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int n_chunks = accept_chunks(total_rows, vocab, sm_count());
    float2 *part = static_cast<float2 *>(workspace);
    if (total_rows > 0) {
        if (total_rows > 65535)
            return set_error(PKV_ERR_SHAPE, "spec_accept_tree_greedy: at most 65535 rows per call");
        int chunk = (vocab + n_chunks - 1) / n_chunks;
        chunk = (chunk + 3) & ~3;
        argmax_chunks_kernel<<<dim3(n_chunks, total_rows), kArgmaxThreads, 0, st>>>(logits, vocab, chunk, n_chunks,
                                                                                   part, (vocab % 4) == 0);
        const int rc = check_cuda(cudaGetLastError(), "spec_accept_tree_greedy argmax launch");
        if (rc)
            return rc;
    }
    int32_t *status = device_status_word();
    if (!status)
        return set_error(PKV_ERR_CUDA, "spec_accept_tree_greedy: no device status word");
    accept_tree_walk_kernel<<<num_seqs, 32, 0, st>>>(part, n_chunks, q_starts, draft_tokens, parents, total_rows,
                                                     argmax_out, accept_len, out_tokens, accepted_rows, status);
    return check_cuda(cudaGetLastError(), "spec_accept_tree_greedy walk launch");
}

extern "C" int spec_accept_sampled(const float *logits, int32_t vocab, const int32_t *q_starts,
                                   const int32_t *draft_tokens, const int32_t *parents, const int32_t *positions,
                                   uint64_t seed, float temperature, int32_t top_k, float top_p, float min_p,
                                   int32_t num_seqs,
                                   int32_t total_rows, int32_t *sampled_out, int32_t *accept_len,
                                   int32_t *out_tokens, int32_t *accepted_rows, void *workspace,
                                   size_t workspace_bytes, void *stream)
{
    using namespace pkv;
    clear_error();
    if (num_seqs < 0 || total_rows < 0 || vocab <= 0)
        return set_error(PKV_ERR_SHAPE, "spec_accept_sampled: bad sizes (num_seqs %d, rows %d, vocab %d)",
                         num_seqs, total_rows, vocab);
    if (!(temperature >= 0.0f) || !(temperature < INFINITY) || !(min_p <= 1.0f) || !(top_p == top_p))
        return set_error(PKV_ERR_SHAPE, "spec_accept_sampled: temperature %g must be finite and >= 0, "
                         "min_p %g at most 1, top_p %g a number", (double)temperature, (double)min_p,
                         (double)top_p);
    if (num_seqs == 0)
        return PKV_OK;
    if (!q_starts || !accept_len || (total_rows > 0 && (!logits || !draft_tokens || !positions || !sampled_out ||
                                                        !out_tokens || !accepted_rows || !workspace)))
        return set_error(PKV_ERR_NULL, "spec_accept_sampled: a required pointer is NULL");
    if (total_rows > 0 && !aligned16(logits))
        return set_error(PKV_ERR_ALIGN, "spec_accept_sampled: logits must be 16-byte aligned");
    const size_t one = spec_accept_workspace_size(total_rows, vocab);
    const size_t need_ws = 2 * one + round_up((size_t)total_rows * 8, 256);
    if (workspace_bytes < need_ws)
        return set_error(PKV_ERR_WORKSPACE, "spec_accept_sampled: workspace %zu < %zu bytes", workspace_bytes,
                         need_ws);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int n_chunks = accept_chunks(total_rows, vocab, sm_count());
    float2 *part_max = static_cast<float2 *>(workspace);
    float2 *part = reinterpret_cast<float2 *>(static_cast<uint8_t *>(workspace) + one);
    if (total_rows > 0) {
        if (total_rows > 65535)
            return set_error(PKV_ERR_SHAPE, "spec_accept_sampled: at most 65535 rows per call");
        int chunk = (vocab + n_chunks - 1) / n_chunks;
        chunk = (chunk + 3) & ~3;
        const int vec_ok = (vocab % 4) == 0;
        argmax_chunks_kernel<<<dim3(n_chunks, total_rows), kArgmaxThreads, 0, st>>>(logits, vocab, chunk, n_chunks,
                                                                                   part_max, vec_ok);
        int rc = check_cuda(cudaGetLastError(), "spec_accept_sampled argmax launch");
        if (rc)
            return rc;
        if (temperature > 0.0f) {
            // the min_p threshold's offset T log(min_p), rounded once here and once in the kernel's add
            const float off = min_p > 0.0f ? temperature * logf(min_p) : -INFINITY;
            unsigned long long *cut = nullptr;
            const bool use_k = top_k > 0 && top_k < vocab;
            const bool use_p = top_p > 0.0f && top_p < 1.0f;
            if (use_k || use_p) {
                cut = reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(workspace) + 2 * one);
                const unsigned long long p_fix = use_p ? (unsigned long long)(top_p * 4294967296.0f) : 0ull;
                // set before every launch: the attribute belongs to the current context
                rc = check_cuda(cudaFuncSetAttribute(topkp_cut_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     (int)sizeof(SelSmem)),
                                "spec_accept_sampled: shared memory attribute");
                if (rc)
                    return rc;
                topkp_cut_kernel<<<total_rows, kSelThreads, sizeof(SelSmem), st>>>(
                    logits, vocab, part_max, n_chunks, temperature, use_k ? top_k : 0, use_p ? 1 : 0, p_fix, cut);
                rc = check_cuda(cudaGetLastError(), "spec_accept_sampled top-k / top-p launch");
                if (rc)
                    return rc;
            }
            sample_chunks_kernel<<<dim3(n_chunks, total_rows), kArgmaxThreads, 0, st>>>(
                logits, vocab, chunk, n_chunks, part_max, part, positions, (uint32_t)seed, (uint32_t)(seed >> 32),
                temperature, off, vec_ok, cut);
            rc = check_cuda(cudaGetLastError(), "spec_accept_sampled sample launch");
            if (rc)
                return rc;
        } else {
            part = part_max;   // temperature 0: the greedy draw
        }
    }
    int32_t *status = device_status_word();
    if (!status)
        return set_error(PKV_ERR_CUDA, "spec_accept_sampled: no device status word");
    accept_tree_walk_kernel<<<num_seqs, 32, 0, st>>>(part, n_chunks, q_starts, draft_tokens, parents, total_rows,
                                                     sampled_out, accept_len, out_tokens, accepted_rows, status);
    return check_cuda(cudaGetLastError(), "spec_accept_sampled walk launch");
}
