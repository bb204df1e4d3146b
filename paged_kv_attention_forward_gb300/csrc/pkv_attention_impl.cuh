// pkv_attention_impl.cuh -- the paged-attention kernels (split + merge) and the host
// checks shared by the bf16 and the quantised-KV entry points.
//
// What it computes: TensorSharp "高级功能", section "原生分页注意力" -- attention of
// each sequence's query rows over K/V gathered from the paged block pool, with a
// variant carrying one sink logit per head (GPT OSS).  The causal verify window
// and the bit-identity rule come from the TensorFold article, section
// "先记住一条铁律": a verify row uses exactly the serial step's arithmetic, and a
// row computed in a batch equals the row computed alone.
//
// Design (two kernels per call: splits, then merge):
//  * Work unit = (sequence s, KV head g, split i).  Split i covers keys
//    [512 i, 512 i + 512) of s.  The split grid depends on the sequence's own
//    length only, never on the batch, so every row's arithmetic is fixed by
//    its own sequence.  Grid = (num_seqs * H_kv, ceil(max_context_len / 512)),
//    split-major, so the first splits of all sequences (where shared prefix
//    blocks live) run together and re-read shared blocks from L2.
//  * One producer warp: a single lane reads the block table and issues TMA
//    tile loads (cp.async.bulk.tensor, 128-byte swizzle) of each K and V block
//    of the split into an NST-stage shared-memory ring, completion tracked by
//    mbarriers.
//  * Consumer warps, each owning 8 * NN query rows of the (s, g) pair: the G q heads
//    of KV head g times the W rows of s, flattened row = w * G + head_in_group.  A
//    pair with more rows than one CTA holds is served by adjacent row-group CTAs
//    that read the same K/V tiles (the second and later from L2).
//    Per KV block, on mma.sync m16n8k16 (bf16 in, fp32 out) with keys / head dims
//    on the M side and query rows on the N side (decode has at most 8 rows per KV
//    head, so nothing is padded to 16 rows): S^T = K q^T, scale, causal / length
//    mask, online softmax in base 2 (running max m, running sum l of the
//    bf16-rounded weights), P^T transposed in registers (movmatrix) and
//    O^T += V^T P^T.
//    Keys past a row's limit get weight exactly 0, so a verify-window row and the
//    same row decoded alone go through identical operations.
//  * Partials (m, l, O) of every split go to the workspace.  A second kernel,
//    two warps per (query row, q head), merges them in an order fixed by the
//    row's own length (each warp one half in split order, then the halves):
//    M = max(m_i, sink), out = sum_i 2^{m_i-M} O_i / (sum_i 2^{m_i-M} l_i + 2^{sink-M}).
//    It is launched as a programmatic dependent of the split kernel, so its launch
//    overlaps the split grid's tail.
//  * Bounded waits only; block ids and lengths are range-checked on the device
//    (clamped + status bit, never a fault).
//  * Quantised KV blocks (TensorSharp "高级功能", section "内存优化", the KV block
//    codec item): the same kernel with BITS = 8, 4 or 2 reads one record per
//    (block, KV head) with a single bulk copy (codes of K and V + per-key
//    scales), widens the codes to f16 in registers, folds each key's K scale
//    into its score and log2 of its V scale into its logit, so the weights meet the
//    raw codes and P V accumulates straight into O.
#pragma once

#include <cmath>
#include <cstring>
#include <mutex>
#include <type_traits>

#include <cuda_bf16.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned long long kGatherBad = ~0ull;

// Accumulation chains of the S^T = K q^T k-steps, per codec (chosen by measurement:
// four chains gain 12 % on Q8 records, whose k-steps carry more latency, and lose 1 %
// on bf16 pools).  One value per codec keeps every CTA shape on one arithmetic.
#ifndef PKV_QK_CHAINS_BF16
#define PKV_QK_CHAINS_BF16 2
#endif
#ifndef PKV_QK_CHAINS_QUANT
#define PKV_QK_CHAINS_QUANT 4
#endif
template <int BITS>
constexpr int kQkChainsOf = BITS == 16 ? PKV_QK_CHAINS_BF16 : PKV_QK_CHAINS_QUANT;

// 16-key quantised records fetched per ring stage (1 or 2): two per stage pay the
// per-stage softmax bookkeeping once per 32 keys (Q8 cb_mix call 269 -> 251 us with a
// 4-stage ring, Q8 verify windows 504 -> 411 us)
#ifndef PKV_QUANT_RECS_PER_STAGE
#define PKV_QUANT_RECS_PER_STAGE 2
#endif
static_assert(PKV_QUANT_RECS_PER_STAGE == 1 || PKV_QUANT_RECS_PER_STAGE == 2, "records per stage");
// 16-key bf16 blocks per ring stage (1 or 2).  This sets the granularity of the online
// softmax update, so it is one constant for every CTA shape (decode, verify, prefill,
// gather): a verify row must take the same steps as the same row decoded alone.
// Two: the bookkeeping is paid once per 32 keys (with 2-stage decode and wide rings:
// cb_mix call 341.4 -> 338.7 us, spec_verify 275.0 -> 242.4 us, spec_tree 315.4 -> 279.3 us,
// ministral 23.2 -> 17.5 us per layer, prefill_mix 1780 -> 1486 us with a 3-stage ring).
#ifndef PKV_BF16_BLOCKS_PER_STAGE
#define PKV_BF16_BLOCKS_PER_STAGE 2
#endif
static_assert(PKV_BF16_BLOCKS_PER_STAGE == 1 || PKV_BF16_BLOCKS_PER_STAGE == 2, "bf16 blocks per stage");
// blocks per ring stage: 32-key blocks always go one at a time
template <int BITS, int BS>
constexpr int kBlocksPerStage = BS != 16 ? 1 : BITS != 16 ? PKV_QUANT_RECS_PER_STAGE : PKV_BF16_BLOCKS_PER_STAGE;
static_assert((PKV_QK_CHAINS_BF16 == 2 || PKV_QK_CHAINS_BF16 == 4) &&
              (PKV_QK_CHAINS_QUANT == 2 || PKV_QK_CHAINS_QUANT == 4), "QK chains");

struct AttnParams {
    const uint16_t *q;            // bf16 [R][Hq][D]
    const int32_t *q_starts;      // [S+1]
    const int32_t *block_tables;  // [S][max_blocks]
    const int32_t *context_lens;  // [S]
    const float *sinks;           // [Hq] or null
    const uint32_t *tree_masks;   // [R] or null: bit i = the row sees window token i
    void *out;                    // [R][Hq][D] bf16 or f32
    float2 *part_ml;              // [R*Hq*n_max] (m in log2 units, l)
    float *part_o;                // [R*Hq*n_max][D]
    const uint8_t *qrec;          // quantised pool: records [num_blocks][H_kv][QRec::kBytes], or null
    const uint16_t *kpool, *vpool;   // bf16 pools, read by the index-list gather
    const int32_t *key_idx;       // [R][max_keys] key positions of each row (index-list gather), or null
    const int32_t *key_counts;    // [R]
    int32_t max_keys;
    int32_t *status;
    long long wait_limit;         // SM cycles a pipeline stage wait may take (<= 0: give up at once)
    const int4 *units;            // (tensor-core path) the unit list: (s, split, KV head, row group)
    int32_t *unit_ctl;            // [0] work counter, [1] unit count
    long long unit_cap;           // entries the unit list has room for
    int32_t num_seqs, max_blocks_per_seq, num_blocks, num_q_heads, num_kv_heads, group, block_size;
    int32_t n_max, max_context_len, max_rows, total_rows;
    int32_t row_groups;           // CTAs per (s, g, split), each taking 8 * NN * NMT rows
    int32_t causal, out_f32;
    float scale_log2;             // scale * log2(e)
    int16_t q_head_of[kMaxQHeads];  // q head of (kv head g, member j): q_head_of[g*group + j]
};

template <int D, int BS>
struct Tile {
    static constexpr int kHalves = D / 64;              // 128-byte column boxes per row
    static constexpr int kBoxBytes = BS * 128;          // one box: BS rows x 128 B
    static constexpr int kTileBytes = BS * D * 2;       // one KV block of one head
    static_assert(kSplitTokens % BS == 0, "split must be whole blocks");
    static_assert(D % 64 == 0, "head_dim multiple of 64");
    static_assert(BS % 16 == 0, "block size multiple of 16");
};

// Byte offset of logical (token, 16-byte chunk) inside a swizzled tile:
// chunk ch of token t lives in box ch/8, row t, at chunk position (ch%8) ^ (t%8).
template <int BS>
__device__ __forceinline__ uint32_t tile_off(int tok, int ch)
{
    return (uint32_t)((ch >> 3) * (BS * 128) + tok * 128 + (((ch & 7) ^ (tok & 7)) << 4));
}

// ---- quantised records ------------------------------------------------------
// One record per (block, KV head): [K codes | V codes | K scales | V scales], the
// codes of each section in "fragment order": 16-byte units, unit (tile16, u, lane)
// holding exactly the 4 words lane `lane` feeds to the mma A operand, so a warp
// reads a section with conflict-free 16-byte loads.  For the 16-key tile mt, A row
// g + 8r of K is key 16 mt + 2g + r and A column s is dim s of the k-step; the V^T
// operand uses column s = key 16 kk + (s < 8 ? 2s : 2(s - 8) + 1), the order in
// which the transposed P^T fragment of K's S^T arrives.  8-bit codes are bytes of
// c + 128 (word bytes 0, 2 feed a0/a1, bytes 1, 3 feed a2/a3); 4-bit codes are
// nibbles holding c + 8; 2-bit codes are bit pairs holding c + 2, one lane's codes
// of a 16-key group in D / 8 contiguous bytes (two k-steps per word, a byte per
// key).  Full byte-level formula in pkv.h.
template <int D, int BS, int BITS>
struct QRec {
    static constexpr int kCodeBytes = BS * D * BITS / 8;          // one section
    static constexpr int kK = 0, kV = kCodeBytes;
    static constexpr int kKs = 2 * kCodeBytes, kVs = 2 * kCodeBytes + 4 * BS;
    static constexpr int kBytes = 2 * kCodeBytes + 8 * BS;
    static constexpr int kWords = D * BITS / 64;                  // 32-bit words per lane per 16 keys
    static constexpr int kGroupBytes = kWords * 4 * 32;           // a 16-key group of one section
    static_assert(BITS == 8 || BITS == 4 || BITS == 2, "codec width");
    static_assert(kBytes % 16 == 0, "record must stay 16-byte aligned");
};

// The lane's words of one 16-key group (g: the group's first byte): 16-byte units
// interleaved across the warp for 8 / 4 bits, one contiguous run for 2 bits.
template <int D, int BITS>
__device__ __forceinline__ void load_group(const uint8_t *g, int lane, uint32_t (&w)[D * BITS / 64])
{
    constexpr int NW = D * BITS / 64;
    if constexpr (BITS == 2 && NW == 2) {
        const uint2 u = *reinterpret_cast<const uint2 *>(g + lane * 8);
        w[0] = u.x;
        w[1] = u.y;
    } else {
#pragma unroll
        for (int k = 0; k < NW / 4; ++k) {
            const uint4 u = *reinterpret_cast<const uint4 *>(g + (BITS == 2 ? lane * 16 : (k * 32 + lane) * 16));
            w[4 * k] = u.x;
            w[4 * k + 1] = u.y;
            w[4 * k + 2] = u.z;
            w[4 * k + 3] = u.w;
        }
    }
}

// Codes become f16 operands with one logic op: a field u at bits p .. of the low byte
// of each 16-bit half, under the exponent bits 0x6400, is the f16 1024 + u * 2^p
// exactly.  A byte code (u = c + 128, p = 0) is 1024 + u; a nibble (c + 8) or bit pair
// (c + 2) sits at p = fpos(step, half) of its byte (bytes 1 and 3 are first moved down by
// one prmt), so its operand is 1024 + 2^p (c + off).  The factor 2^p is taken out exactly
// (K: the matching q dims are scaled by 2^-p; V: the PV product by 2^-p at the end), and
// the kernel removes the offset in fp32: sum(q' * (1024 + 2^p off)) from each score (the
// first accumulation chain starts there) and, every ring stage, (1024 + 2^p off) * sum(P)
// over the stage's weights from each output element.
template <int BITS>
constexpr int kCodeOff = 1 << (BITS - 1);   // 128, 8, 2: the stored field is c + off

// Floor of log2 of a V scale folded into a logit: keeps p = 2^(x - m) below 2^100 for a
// key whose V row is zero (scale 0) or tiny, so the denominator stays finite.
constexpr float kVlogFloor = -100.f;

// bit position, within its byte, of the field that feeds k-step (K) or dim m-tile (V)
// `step`, column half (K) or row half (V) `half`
template <int BITS>
__device__ __forceinline__ constexpr int fpos(int step, int half)
{
    return BITS == 8 ? 0 : BITS == 4 ? 4 * half : 4 * (step & 1) + 2 * half;
}

// A operand of k-step ks of a K tile, or of 16-dim m-tile ks of a V^T tile, from the
// lane's words of that 16-key group.
template <int BITS, bool IS_V, int NW>
__device__ __forceinline__ void q_frag(const uint32_t (&cw)[NW], int ks, uint32_t (&a)[4])
{
    if constexpr (BITS == 8) {
        const uint32_t w0 = cw[2 * ks], w1 = cw[2 * ks + 1];
        a[0] = __byte_perm(w0, 0x64646464u, 0x4240);   // bytes 0, 2
        a[1] = __byte_perm(w1, 0x64646464u, 0x4240);
        a[2] = __byte_perm(w0, 0x64646464u, 0x4341);   // bytes 1, 3
        a[3] = __byte_perm(w1, 0x64646464u, 0x4341);
    } else {
        // K: byte = A row half r, field = A column half h; V: byte = A column half h,
        // field = A row half r (the fields of one k-step / m-tile sit at fpos(step, 0 / 1))
        const uint32_t lo = BITS == 4 ? cw[ks] : cw[ks >> 1];
        const uint32_t hi = __byte_perm(lo, 0u, 0x3311);   // bytes 1, 3 -> 0, 2
        constexpr uint32_t f = BITS == 4 ? 0x000F000Fu : 0x00030003u;
        const uint32_t m0 = f << fpos<BITS>(ks, 0), m1 = f << fpos<BITS>(ks, 1);
        if constexpr (!IS_V) {
            a[0] = (lo & m0) | 0x64006400u;   // r 0, h 0
            a[1] = (hi & m0) | 0x64006400u;   // r 1, h 0
            a[2] = (lo & m1) | 0x64006400u;   // r 0, h 1
            a[3] = (hi & m1) | 0x64006400u;   // r 1, h 1
        } else {
            a[0] = (lo & m0) | 0x64006400u;   // r 0, h 0
            a[1] = (lo & m1) | 0x64006400u;   // r 1, h 0
            a[2] = (hi & m0) | 0x64006400u;   // r 0, h 1
            a[3] = (hi & m1) | 0x64006400u;   // r 1, h 1
        }
    }
}

// NN: n-tiles of 8 query rows per consumer warp; NMT: consumer warps.  A CTA serves
// up to 8 * NN * NMT rows (the G q heads of one KV head times the sequence's rows).
// TREE: rows carry ancestor masks over the window keys (tree verify); a separate
// instantiation so the decode / causal path carries no mask test.
// BITS: 16 = bf16 pools read by TMA tiles; 8 / 4 / 2 = quantised records, one bulk copy
// per (block, KV head), codes widened to f16 in registers.
// KW: consumer warps that share each row group's keys: warp (kw, mw) takes the split's
// blocks kw, kw + KW, ... for the rows of row warp mw, with its own softmax state; the
// KW states are merged in kw order at the end.  KW depends only on the codec, and
// which warp sees which key only on the key's position, so a row's arithmetic is
// still fixed by its own sequence, whatever the CTA shape.
// GATHER: the index-list gather.  The work unit is (query row, KV head); its keys are
// the row's list entries, 16 per stage, each row fetched through the block table with
// 16-byte cp.async copies into the same swizzled tile layout the TMA path fills.
// Residency hints: by default the compiler picks the register count (94-126 for the
// bf16 kernels at d 128); PKV_MIN_CTAS_WIDE / PKV_MIN_CTAS_DECODE request that many
// resident CTAs of the wide-row / decode shapes, capping the registers to fit.
// Quantised records: PKV_MIN_CTAS_Q8 / PKV_MIN_CTAS_QNARROW (decode shapes of 8-bit /
// 4- and 2-bit records) and PKV_MIN_CTAS_QWIDE (their wide-row shapes), when above 0,
// launch through a second entry point that asks for that many resident CTAs.  (A
// minimum of 1 is not the same as none: it changes the compiler's register choice.)
#ifndef PKV_MIN_CTAS_Q8
#define PKV_MIN_CTAS_Q8 0
#endif
#ifndef PKV_MIN_CTAS_QNARROW
#define PKV_MIN_CTAS_QNARROW 0
#endif
#ifndef PKV_MIN_CTAS_QWIDE
#define PKV_MIN_CTAS_QWIDE 0
#endif
template <int BITS, int NMT>
constexpr int kMinCtas()
{
    return BITS == 16 ? 0 : NMT > 1 ? PKV_MIN_CTAS_QWIDE : BITS == 8 ? PKV_MIN_CTAS_Q8 : PKV_MIN_CTAS_QNARROW;
}
#if defined(PKV_MIN_CTAS_WIDE) && defined(PKV_MIN_CTAS_DECODE)
#define PKV_KERNEL_BOUNDS(NMT, KW) __launch_bounds__(((NMT) * (KW) + 1) * 32, (NMT) > 1 ? PKV_MIN_CTAS_WIDE : PKV_MIN_CTAS_DECODE)
#else
#define PKV_KERNEL_BOUNDS(NMT, KW) __launch_bounds__(((NMT) * (KW) + 1) * 32)
#endif
template <int D, int BS, int NN, int NMT, int NST, bool TREE, int BITS, int KW, bool GATHER>
__device__ __forceinline__ void split_kernel_body(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const AttnParams &p)
{
    static_assert(!GATHER || (BITS == 16 && !TREE && KW == 1 && BS == 16), "index-list gather: bf16, 16-key tiles");
    static_assert(!(TREE && BITS != 16), "tree masks are built for bf16 pools only");
    // Every use of a stage must belong to one key-share warp: stage st holds blocks
    // st, st + NST, ..., all of share st % KW only when KW divides NST.  Otherwise a
    // warp could wait for a stage's next phase while another warp's phase of it is
    // still pending, and a parity wait cannot tell those phases apart.
    static_assert(NST % KW == 0, "ring depth must be a multiple of the key-share warps");
    constexpr int kQkChains = kQkChainsOf<BITS>;
    using T = Tile<D, BS>;
    constexpr int MT = BS / 16;   // 16-key m-tiles per block
    // blocks per ring stage: 16-key blocks may go two at a time, so the per-stage
    // softmax bookkeeping is paid once per 32 keys
    constexpr int TB = kBlocksPerStage<BITS, BS>;
    constexpr int MTE = MT * TB;  // 16-key m-tiles per stage
    constexpr int KS = D / 16;    // k-steps of K q^T
    constexpr int DM = D / 16;    // 16-dim m-tiles of V^T P^T
    constexpr int C = kSplitTokens;
    constexpr int RPW = 8 * NN;   // rows per consumer warp
    constexpr int NBW = (C / BS + 31) / 32;   // block ids per producer lane
    // Row sums of a stage's rounded weights (for the code offset): Q8 takes them from the tensor
    // core, one more MMA per 16-key tile with an A operand of ones (Q8 verify call 299 -> 292 us,
    // sinks_scale 217 -> 214 us); 4- and 2-bit records add the lanes' weights (the MMA made a Q4
    // cb_mix call 218 -> 223 us)
    constexpr bool kMmaRowSum = BITS == 8;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    constexpr int RECB = QRec<D, BS, (BITS == 16 ? 8 : BITS)>::kBytes;
    constexpr int STAGE = BITS == 16 ? 2 * TB * T::kTileBytes : TB * RECB;
    uint8_t *k_tiles = smem;                              // bf16: the TB K tiles of every stage,
    uint8_t *v_tiles = smem + NST * TB * T::kTileBytes;   // then the V tiles; quantised: TB records per stage
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + NST * STAGE);
    uint64_t *empty = full + NST;
    volatile int32_t *s_flag = reinterpret_cast<volatile int32_t *>(empty + NST);
    // s_flag[1]: abort; [2]: stages issued
    // (gather) the slice's resolved row offsets, in elements; kGatherBad marks a bad entry
    unsigned long long *g_off = reinterpret_cast<unsigned long long *>(empty + NST + 8);

    const int pair = blockIdx.x / p.row_groups;
    const int rg = blockIdx.x - pair * p.row_groups;
    const int s = pair / p.num_kv_heads;
    const int g = pair - s * p.num_kv_heads;
    // highest split indices first: only the longest sequences have them, so the grid ends
    // on every sequence's first split (uniform, and sharing the prefix blocks through L2)
    const int split = gridDim.y - 1 - blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    int L;        // keys of the unit: the context length, or (gather) the row's list length
    int seq = s;  // (gather) the sequence of query row s
    if constexpr (GATHER) {
        int lo = 0, hi = p.num_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.q_starts + mid) <= s)
                lo = mid;
            else
                hi = mid - 1;
        }
        seq = lo;
        L = s < p.total_rows ? __ldg(p.key_counts + s) : 0;
        if (L > p.max_keys || L < 0) {
            if (split == 0 && threadIdx.x == 0)
                atomicOr(p.status, PKV_DEV_TABLE_OVERRUN);
            L = L < 0 ? 0 : p.max_keys;
        }
    } else {
        L = __ldg(p.context_lens + s);
        const int L_cap = (int)min((long long)p.max_context_len, (long long)p.max_blocks_per_seq * BS);
        if (L > L_cap || L < 0) {
            if (split == 0 && threadIdx.x == 0)
                atomicOr(p.status, PKV_DEV_TABLE_OVERRUN);
            L = L < 0 ? 0 : L_cap;
        }
    }
    // the dependent merge kernel may be scheduled once every CTA of this grid has started
    asm volatile("griddepcontrol.launch_dependents;");
    const int n_splits = (L + C - 1) / C;
    if (split >= n_splits)
        return;
    const int row0 = GATHER ? s : __ldg(p.q_starts + s);
    int W = GATHER ? 1 : __ldg(p.q_starts + s + 1) - row0;
    if (W <= 0)
        return;
    if (row0 < 0 || row0 + W > p.total_rows) {   // q_starts inconsistent with total_q_rows
        if (split == 0 && g == 0 && threadIdx.x == 0)
            atomicOr(p.status, PKV_DEV_TOO_MANY_ROWS);
        return;
    }
    if (W > p.max_rows) {
        if (split == 0 && threadIdx.x == 0)
            atomicOr(p.status, PKV_DEV_TOO_MANY_ROWS);
        W = p.max_rows;
    }
    const int M = p.group * W;               // query rows of this (s, g)
    const int r_lo = rg * RPW * NMT;         // first row of this CTA's row group
    if (r_lo >= M)
        return;
    const int n_act = (min(M - r_lo, RPW * NMT) + RPW - 1) / RPW;   // consumer warps with rows

    const int t0 = split * C;
    const int t1 = min(t0 + C, L);
    const int blk0 = t0 / BS;
    const int nblk = (t1 - t0 + BS - 1) / BS;
    const int nstage = (nblk + TB - 1) / TB;   // ring stages of this split

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], GATHER ? 32 : 1);   // gather: every producer lane arrives
            mbar_init(&empty[i], n_act);
        }
        mbar_fence_init();
        s_flag[1] = 0;
        s_flag[2] = 0;
    }
    __syncthreads();

    if (GATHER && warp == NMT * KW) {
        // ---------------- producer warp (gather): list -> block table -> cp.async ----------------
        constexpr int CH = D / 8;             // 16-byte chunks per key row
        constexpr int KSTEP = 32 / CH;        // keys a lane steps over
        constexpr int KPL = 16 / KSTEP;       // keys per lane per tile
        const int ch = lane % CH, kq = lane / CH;
        const long long ctx_cap = (long long)p.max_blocks_per_seq * p.block_size;
        long long ctx = __ldg(p.context_lens + seq);
        ctx = ctx < 0 ? 0 : (ctx > ctx_cap ? ctx_cap : ctx);
        const int32_t *lst = p.key_idx + (size_t)s * p.max_keys;
        // resolve every entry of the slice first: all of the lane's list loads, then all
        // of its (dependent) block-table loads, so the slice costs two round trips
        constexpr int EPL = C / 32;   // entries per lane
        int pos[EPL], blk[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = t0 + j * 32 + lane;
            pos[j] = e < t1 ? __ldg(lst + e) : -1;
        }
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const bool in = pos[j] >= 0 && pos[j] < ctx;
            blk[j] = in ? __ldg(p.block_tables + (size_t)seq * p.max_blocks_per_seq + pos[j] / p.block_size) : -1;
        }
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int i = j * 32 + lane;
            if (t0 + i >= t1)
                break;
            unsigned long long off = kGatherBad;
            if (pos[j] >= 0 && pos[j] < ctx) {
                if (blk[j] >= 0 && blk[j] < p.num_blocks)
                    off = ((((unsigned long long)blk[j] * p.num_kv_heads) + g) * p.block_size + pos[j] % p.block_size) * D;
                else
                    atomicOr(p.status, PKV_DEV_BAD_BLOCK);
            } else {
                atomicOr(p.status, PKV_DEV_TABLE_OVERRUN);   // a listed position outside the context
            }
            g_off[i] = off;
        }
        __syncwarp();
        int k = 0;
        for (; k < nstage; ++k) {
            const int st = k % NST;
            bool ok = true;
            if (k >= NST)
                ok = mbar_wait_bounded(&empty[st], ((k / NST) + 1) & 1, p.wait_limit);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok || s_flag[1]) {
                if (lane == 0) {
                    if (!ok)
                        atomicOr(p.status, PKV_DEV_TIMEOUT);
                    s_flag[1] = 1;
                }
                break;
            }
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                const int tt = k * TB + b;   // 16-entry tile of the slice
                uint8_t *kt = k_tiles + (st * TB + b) * T::kTileBytes;
                uint8_t *vt = v_tiles + (st * TB + b) * T::kTileBytes;
#pragma unroll
                for (int i = 0; i < KPL; ++i) {
                    const int key = kq + i * KSTEP;
                    if (t0 + tt * 16 + key < t1) {   // entries past the list's end are masked, not copied
                        const unsigned long long o = g_off[tt * 16 + key];
                        const bool vld = o != kGatherBad;   // a bad entry copies zeros from the pool's start
                        cp_async_16(kt + tile_off<16>(key, ch), p.kpool + (vld ? o : 0ull) + ch * 8, vld ? 16u : 0u);
                        cp_async_16(vt + tile_off<16>(key, ch), p.vpool + (vld ? o : 0ull) + ch * 8, vld ? 16u : 0u);
                    }
                }
            }
            cp_async_arrive(&full[st]);
        }
        if (lane == 0)
            s_flag[2] = k;
    } else if (!GATHER && warp == NMT * KW) {
        // ---------------- producer warp: block table -> TMA ring ----------------
        // lane l holds the ids of the split's blocks l, l + 32, ... (one coalesced load each)
        int my_blk[NBW];
#pragma unroll
        for (int r = 0; r < NBW; ++r) {
            my_blk[r] = 0;
            const int j = r * 32 + lane;
            if (j < nblk) {
                my_blk[r] = __ldg(p.block_tables + (size_t)s * p.max_blocks_per_seq + blk0 + j);
                if (my_blk[r] < 0 || my_blk[r] >= p.num_blocks) {
                    atomicOr(p.status, PKV_DEV_BAD_BLOCK);
                    my_blk[r] = 0;
                }
            }
        }
        if (BITS == 16 && lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        int k = 0;   // stages issued
        for (; k < nstage; ++k) {
            int blks[TB];
#pragma unroll
            for (int i = 0; i < TB; ++i) {
                const int idx = k * TB + i;
                int mine = 0;
#pragma unroll
                for (int r = 0; r < NBW; ++r)
                    if (r == (idx >> 5))
                        mine = my_blk[r];
                const int b = __shfl_sync(0xffffffffu, mine, idx & 31);
                blks[i] = idx < nblk ? b : -1;
            }
            bool stop = false;
            if (lane == 0) {
                const int st = k % NST;
                bool ok = true;
                if (k >= NST)
                    ok = mbar_wait_bounded(&empty[st], ((k / NST) + 1) & 1, p.wait_limit);
                if (!ok)
                    atomicOr(p.status, PKV_DEV_TIMEOUT);
                if (!ok || s_flag[1]) {
                    s_flag[1] = 1;
                    stop = true;
                } else if constexpr (BITS == 16) {
                    uint32_t bytes = 0;
#pragma unroll
                    for (int i = 0; i < TB; ++i)
                        bytes += blks[i] >= 0 ? 2 * T::kTileBytes : 0;
                    mbar_arrive_expect_tx(&full[st], bytes);
#pragma unroll
                    for (int i = 0; i < TB; ++i) {
                        if (blks[i] < 0)   // past the split's last block: the keys are masked
                            continue;
                        const int y = (blks[i] * p.num_kv_heads + g) * BS;
                        uint8_t *kt = k_tiles + (st * TB + i) * T::kTileBytes;
                        uint8_t *vt = v_tiles + (st * TB + i) * T::kTileBytes;
#pragma unroll
                        for (int h = 0; h < T::kHalves; ++h) {
                            tma_load_2d(kt + h * T::kBoxBytes, &tm_k, &full[st], h * 64, y);
                            tma_load_2d(vt + h * T::kBoxBytes, &tm_v, &full[st], h * 64, y);
                        }
                    }
                } else {
                    uint32_t bytes = 0;
#pragma unroll
                    for (int i = 0; i < TB; ++i)
                        bytes += blks[i] >= 0 ? RECB : 0;
                    mbar_arrive_expect_tx(&full[st], bytes);
#pragma unroll
                    for (int i = 0; i < TB; ++i)
                        if (blks[i] >= 0)
                            bulk_load(smem + st * STAGE + i * RECB,
                                      p.qrec + ((size_t)blks[i] * p.num_kv_heads + g) * RECB, RECB, &full[st]);
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0))
                break;
        }
        if (lane == 0)
            s_flag[2] = k;
    } else if (warp % NMT >= n_act) {
        if constexpr (KW > 1) {   // row warps without rows still take part in the merge barriers
            asm volatile("bar.sync 1, %0;" ::"r"(NMT * KW * 32) : "memory");
            asm volatile("bar.sync 1, %0;" ::"r"(NMT * KW * 32) : "memory");
        }
    } else {
        // ---------------- consumer warps ----------------
        // S^T = K q^T and O^T += V^T P^T on mma.sync m16n8k16: keys / head dims on M,
        // query rows on N.  Lane l owns rows 2(l%4) and 2(l%4)+1 of each n-tile for the
        // softmax and the output, keys l/4 and l/4+8 of each 16-key m-tile.
        const int cr = 2 * (lane & 3);   // first row of this lane within an n-tile
        const int kr = lane >> 2;        // key (row of the C fragment) within 8
        const int kw = warp / NMT;        // key share of this warp
        const int mw = warp % NMT;        // row warp
        const int row_base = r_lo + mw * RPW;
        uint32_t qf[NN][KS][2];
        int lim[NN][2], win0[NN][2];   // keys t < lim are candidates; t >= win0 need their mask bit
        uint32_t tmk[NN][2];
#pragma unroll
        for (int nn = 0; nn < NN; ++nn) {
            const int jq = row_base + nn * 8 + kr;   // B fragment: lane l carries row l/4
            const uint32_t *qrow = nullptr;
            if (jq < M) {
                const int w = jq / p.group;
                const int h = p.q_head_of[g * p.group + (jq - w * p.group)];
                qrow = reinterpret_cast<const uint32_t *>(p.q + ((size_t)(row0 + w) * p.num_q_heads + h) * D);
            }
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                qf[nn][ks][0] = qrow ? __ldg(qrow + ((ks * 16 + cr) >> 1)) : 0u;
                qf[nn][ks][1] = qrow ? __ldg(qrow + ((ks * 16 + 8 + cr) >> 1)) : 0u;
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = row_base + nn * 8 + cr + e;
                lim[nn][e] = (p.causal && j < M) ? L - W + j / p.group + 1 : L;
                win0[nn][e] = L;
                tmk[nn][e] = 0u;
                if (TREE && j < M) {   // tree verify: the window keys a row sees are its ancestors
                    win0[nn][e] = L - W;
                    tmk[nn][e] = __ldg(p.tree_masks + row0 + j / p.group);
                }
            }
        }
        // keys below every row's limit (and, for a tree, below every window) need no mask: a
        // stage entirely below it skips the per-key test (warp-uniform)
        int vis_all = 0x7fffffff;
#pragma unroll
        for (int nn = 0; nn < NN; ++nn)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                vis_all = min(vis_all, TREE ? min(lim[nn][e], win0[nn][e]) : lim[nn][e]);
        vis_all = __reduce_min_sync(0xffffffffu, vis_all);
        // Quantised: q goes to f16, scaled per row by the power of two 2^e that puts its
        // largest |value| in [2^14, 2^15) (exact: a bf16 value has 8 significant bits), and
        // by 2^-fpos more where its codes carry 2^fpos; qbias is the code offset's share of
        // every score (see q_frag), qscale =
        // scale * log2(e) * 2^-e.  Both are needed for the rows cr, cr + 1 of this lane's
        // S^T elements, so they are taken from the lanes that hold those rows' q.
        float qbias[NN][2], qscale[NN][2];
        if constexpr (BITS != 16) {
#pragma unroll
            for (int nn = 0; nn < NN; ++nn) {
                float amax = 0.f;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        amax = fmaxf(amax, fmaxf(fabsf(bf16_lo_to_f32(qf[nn][ks][j])),
                                                 fabsf(bf16_hi_to_f32(qf[nn][ks][j]))));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                const int ex = (__float_as_int(amax) >> 23) & 0xFF;
                const int e2 = amax > 0.f ? min(141 - ex, 126) : 0;   // amax * 2^e2 in [2^14, 2^15)
                // dims of column half j of k-step ks meet codes scaled by 2^fpos: q' takes 2^-fpos
                constexpr int QB = BITS == 16 ? 8 : BITS;
                float qsum[4] = {0.f, 0.f, 0.f, 0.f};   // per field position class
#pragma unroll
                for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float up = __int_as_float((127 + e2 - fpos<QB>(ks, j)) << 23);
                        const uint32_t h2 = pack_f16x2(bf16_lo_to_f32(qf[nn][ks][j]) * up,
                                                       bf16_hi_to_f32(qf[nn][ks][j]) * up);
                        qf[nn][ks][j] = h2;
                        qsum[QB == 2 ? 2 * (ks & 1) + j : QB == 4 ? j : 0] += f16_lo_to_f32(h2) + f16_hi_to_f32(h2);
                    }
                // the code offset's share of the score: sum over dims of q' (1024 + 2^fpos off)
                float bias_r;
                if constexpr (QB == 8) {
                    float q0 = qsum[0];
                    q0 += __shfl_xor_sync(0xffffffffu, q0, 1);
                    q0 += __shfl_xor_sync(0xffffffffu, q0, 2);
                    bias_r = (1024.f + kCodeOff<8>) * q0;
                } else {
                    bias_r = 0.f;
#pragma unroll
                    for (int c = 0; c < (QB == 2 ? 4 : 2); ++c)
                        bias_r += qsum[c] * (1024.f + (float)((1 << fpos<QB>(c >> 1, c & 1)) * kCodeOff<QB>));
                    bias_r += __shfl_xor_sync(0xffffffffu, bias_r, 1);
                    bias_r += __shfl_xor_sync(0xffffffffu, bias_r, 2);
                }
                const float scale_r = p.scale_log2 * __int_as_float((127 - e2) << 23);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    qbias[nn][e] = __shfl_sync(0xffffffffu, bias_r, 4 * (cr + e));
                    qscale[nn][e] = __shfl_sync(0xffffffffu, scale_r, 4 * (cr + e));
                }
            }
        }
        float o[DM][NN][4];
#pragma unroll
        for (int dm = 0; dm < DM; ++dm)
#pragma unroll
            for (int nn = 0; nn < NN; ++nn)
                o[dm][nn][0] = o[dm][nn][1] = o[dm][nn][2] = o[dm][nn][3] = 0.f;
        float mrow[NN][2], lrow[NN][2];
#pragma unroll
        for (int nn = 0; nn < NN; ++nn)
            mrow[nn][0] = mrow[nn][1] = -INFINITY, lrow[nn][0] = lrow[nn][1] = 0.f;

        // per-lane ldmatrix address parts (matrix mi = lane / 8, row lane % 8)
        const int k_key = 8 * ((lane >> 3) & 1) + (lane & 7);   // K: keys of matrices 0/1 vs 2/3
        const int k_chs = lane >> 4;
        const int v_key = 8 * (lane >> 4) + (lane & 7);         // V: keys of matrices 0/1 vs 2/3
        const int v_chs = (lane >> 3) & 1;

        for (int k = kw; k < nstage; k += KW) {
            const int st = k % NST;
            if (!mbar_wait_bounded(&full[st], (k / NST) & 1, p.wait_limit)) {
                if (lane == 0) {
                    atomicOr(p.status, PKV_DEV_TIMEOUT);
                    s_flag[1] = 1;
                }
                break;
            }
            const uint32_t kb = smem_addr(k_tiles + st * TB * T::kTileBytes);   // m-tile mt: tile mt / MT
            const uint32_t vb = smem_addr(v_tiles + st * TB * T::kTileBytes);
            const uint8_t *rec = smem + st * STAGE;   // quantised record of this stage
            const int tbase = (blk0 + k * TB) * BS;

            // S^T for the BS keys of this block; even and odd k-steps in separate chains
            // (four chains: k-steps ks % 4, summed (a + b) + (c + d))
            // (quantised: the first chain starts at minus the code offset's share of the score)
            float sa[MTE][NN][4], sb[MTE][NN][4], sc[MTE][NN][4], sd[MTE][NN][4];
#pragma unroll
            for (int mt = 0; mt < MTE; ++mt)
#pragma unroll
                for (int nn = 0; nn < NN; ++nn)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        sa[mt][nn][c] = BITS != 16 ? -qbias[nn][c & 1] : 0.f;
                        sb[mt][nn][c] = sc[mt][nn][c] = sd[mt][nn][c] = 0.f;
                    }
            // quantised: scales of this lane's keys 2 kr, 2 kr + 1, log2 of their V scales
            // (floored) and 2^-log2
            float2 kscale[MTE], vlog[MTE], vunlog[MTE];
            if constexpr (BITS == 16) {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
                    for (int mt = 0; mt < MTE; ++mt) {
                        uint32_t a[4];
                        ldsm_x4(kb + (mt / MT) * T::kTileBytes + tile_off<BS>((mt % MT) * 16 + k_key, ks * 2 + k_chs),
                                a[0], a[1], a[2], a[3]);
#pragma unroll
                        for (int nn = 0; nn < NN; ++nn) {
                            const int chain = ks % kQkChains;
                            mma_bf16_16x8x16(chain == 0 ? sa[mt][nn] : chain == 1 ? sb[mt][nn] : chain == 2 ? sc[mt][nn] : sd[mt][nn],
                                             a, qf[nn][ks][0], qf[nn][ks][1]);
                        }
                    }
                }
            } else {
                using QR = QRec<D, BS, BITS>;
#pragma unroll
                for (int mt = 0; mt < MTE; ++mt) {
                    const uint8_t *rm = rec + (mt / MT) * RECB;   // the record holding m-tile mt
                    const int mi = mt % MT;
                    kscale[mt] = *reinterpret_cast<const float2 *>(rm + QR::kKs + (mi * 16 + 2 * kr) * 4);
                    const float2 vs = *reinterpret_cast<const float2 *>(rm + QR::kVs + (mi * 16 + 2 * kr) * 4);
                    vlog[mt] = make_float2(fmaxf(__log2f(vs.x), kVlogFloor), fmaxf(__log2f(vs.y), kVlogFloor));
                    vunlog[mt] = make_float2(fast_exp2(-vlog[mt].x), fast_exp2(-vlog[mt].y));
                    uint32_t cw[QR::kWords];
                    load_group<D, BITS>(rm + QR::kK + mi * QR::kGroupBytes, lane, cw);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        uint32_t a[4];
                        q_frag<BITS, false>(cw, ks, a);
#pragma unroll
                        for (int nn = 0; nn < NN; ++nn) {
                            const int chain = ks % kQkChains;
                            mma_f16_16x8x16(chain == 0 ? sa[mt][nn] : chain == 1 ? sb[mt][nn] : chain == 2 ? sc[mt][nn] : sd[mt][nn],
                                            a, qf[nn][ks][0], qf[nn][ks][1]);
                        }
                    }
                }
            }
            // scale into base-2 units; keys at or past a row's limit get -inf
            float mx[NN][2];
#pragma unroll
            for (int nn = 0; nn < NN; ++nn)
                mx[nn][0] = mx[nn][1] = -INFINITY;
            auto scale_scores = [&](auto masked) {
#pragma unroll
                for (int mt = 0; mt < MTE; ++mt)
#pragma unroll
                    for (int nn = 0; nn < NN; ++nn)
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const float qk = kQkChains == 4 ? (sa[mt][nn][c] + sb[mt][nn][c]) + (sc[mt][nn][c] + sd[mt][nn][c])
                                                            : sa[mt][nn][c] + sb[mt][nn][c];
                            float x;
                            if constexpr (BITS == 16)
                                x = qk * p.scale_log2;
                            else   // the logit plus log2 of the key's V scale (see below)
                                x = fmaf(qk, ((c >> 1) ? kscale[mt].y : kscale[mt].x) * qscale[nn][c & 1],
                                         (c >> 1) ? vlog[mt].y : vlog[mt].x);
                            if constexpr (decltype(masked)::value) {
                                // bf16 tiles: A row kr + 8 j is key kr + 8 j; quantised: key 2 kr + j
                                const int t = BITS == 16 ? tbase + mt * 16 + kr + 8 * (c >> 1)
                                                         : tbase + mt * 16 + 2 * kr + (c >> 1);
                                const int e = c & 1;
                                bool vis = t < lim[nn][e];
                                if (TREE)
                                    vis = vis && (t < win0[nn][e] || ((tmk[nn][e] >> (t - win0[nn][e])) & 1u));
                                x = vis ? x : -INFINITY;
                            }
                            sa[mt][nn][c] = x;
                            mx[nn][c & 1] = fmaxf(mx[nn][c & 1], x);
                        }
            };
            if (tbase + BS * TB <= vis_all)
                scale_scores(std::false_type{});
            else
                scale_scores(std::true_type{});
            float alpha[NN][2], base[NN][2];
#pragma unroll
            for (int nn = 0; nn < NN; ++nn)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float v = mx[nn][e];
                    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
                    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
                    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                    const float m_new = fmaxf(mrow[nn][e], v);
                    base[nn][e] = (m_new == -INFINITY) ? 0.f : m_new;
                    alpha[nn][e] = fast_exp2(mrow[nn][e] - base[nn][e]);
                    mrow[nn][e] = m_new;
                }
            const bool tail = tbase + BS * TB > L;
            // P = 2^(S - m) rounded to bf16 (packed per 8x8 fragment); l sums the rounded weights.
            // Quantised: each logit x carries log2 of its key's V scale s_v (floored at
            // kVlogFloor), so the running max m is taken over x + log2 s_v and
            // P = 2^(x + log2 s_v - m) <= 1 is the key's weight times its V scale.  P in f16
            // meets the raw codes in the MMA, which accumulates straight into O; l sums the
            // softmax weights 2^(x - m) = P * 2^-log2 s_v on the same reference.  Every step
            // depends only on the keys the row sees, so a verify row and the same row
            // decoded alone agree; keys at or past L get P exactly 0 whatever their stored
            // scale holds.
            uint32_t pk[MTE][NN][2];
            float sum[NN][2], psum[NN][2];
#pragma unroll
            for (int nn = 0; nn < NN; ++nn)
                sum[nn][0] = sum[nn][1] = psum[nn][0] = psum[nn][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < MTE; ++mt)
#pragma unroll
                for (int nn = 0; nn < NN; ++nn) {
                    if constexpr (BITS == 16) {
                        pk[mt][nn][0] = pack_bf16x2(fast_exp2(sa[mt][nn][0] - base[nn][0]), fast_exp2(sa[mt][nn][1] - base[nn][1]));
                        pk[mt][nn][1] = pack_bf16x2(fast_exp2(sa[mt][nn][2] - base[nn][0]), fast_exp2(sa[mt][nn][3] - base[nn][1]));
                        sum[nn][0] += bf16_lo_to_f32(pk[mt][nn][0]) + bf16_lo_to_f32(pk[mt][nn][1]);
                        sum[nn][1] += bf16_hi_to_f32(pk[mt][nn][0]) + bf16_hi_to_f32(pk[mt][nn][1]);
                    } else {
                        // P = 2^(x + log2 s_v - m) (keys past a row's limit: exactly 0); the
                        // softmax weight 2^(x - m) = P * 2^-log2 s_v goes to l
                        const float w0 = fast_exp2(sa[mt][nn][0] - base[nn][0]), w1 = fast_exp2(sa[mt][nn][1] - base[nn][1]);
                        const float w2 = fast_exp2(sa[mt][nn][2] - base[nn][0]), w3 = fast_exp2(sa[mt][nn][3] - base[nn][1]);
                        pk[mt][nn][0] = pack_f16x2(w0, w1);
                        pk[mt][nn][1] = pack_f16x2(w2, w3);
                        sum[nn][0] = fmaf(w0, vunlog[mt].x, fmaf(w2, vunlog[mt].y, sum[nn][0]));
                        sum[nn][1] = fmaf(w1, vunlog[mt].x, fmaf(w3, vunlog[mt].y, sum[nn][1]));
                        if constexpr (!kMmaRowSum) {   // the rounded weights, for the code offset
                            psum[nn][0] += f16_lo_to_f32(pk[mt][nn][0]) + f16_lo_to_f32(pk[mt][nn][1]);
                            psum[nn][1] += f16_hi_to_f32(pk[mt][nn][0]) + f16_hi_to_f32(pk[mt][nn][1]);
                        }
                    }
                }
            bool moved = false;   // did any row's running max change?
#pragma unroll
            for (int nn = 0; nn < NN; ++nn) {
                lrow[nn][0] = lrow[nn][0] * alpha[nn][0] + sum[nn][0];
                lrow[nn][1] = lrow[nn][1] * alpha[nn][1] + sum[nn][1];
                moved = moved || alpha[nn][0] != 1.f || alpha[nn][1] != 1.f;
            }
            // o *= alpha; skipped when every alpha is exactly 1 (then it changes no bit)
            if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
                for (int nn = 0; nn < NN; ++nn)
#pragma unroll
                    for (int dm = 0; dm < DM; ++dm) {
                        o[dm][nn][0] *= alpha[nn][0];
                        o[dm][nn][1] *= alpha[nn][1];
                        o[dm][nn][2] *= alpha[nn][0];
                        o[dm][nn][3] *= alpha[nn][1];
                    }
            }

            // O^T += V^T P^T.  (Q8: the stage's rounded weights are also summed per row by the
            // tensor core, through an A operand whose first row is all ones: pc row 0.)
            float pc[NN][4];
            if constexpr (kMmaRowSum) {
#pragma unroll
                for (int nn = 0; nn < NN; ++nn)
                    pc[nn][0] = pc[nn][1] = pc[nn][2] = pc[nn][3] = 0.f;
            }
#pragma unroll
            for (int kk = 0; kk < MTE; ++kk) {
                uint32_t b[NN][2];
#pragma unroll
                for (int nn = 0; nn < NN; ++nn) {
                    b[nn][0] = movmatrix_trans(pk[kk][nn][0]);   // keys 0-7 of the m-tile
                    b[nn][1] = movmatrix_trans(pk[kk][nn][1]);   // keys 8-15
                }
                if constexpr (BITS != 16) {
                    using QR = QRec<D, BS, BITS>;
                    uint32_t cw[QR::kWords];
                    load_group<D, BITS>(rec + (kk / MT) * RECB + QR::kV + (kk % MT) * QR::kGroupBytes, lane, cw);
#pragma unroll
                    for (int dm = 0; dm < DM; ++dm) {
                        uint32_t a[4];
                        q_frag<BITS, true>(cw, dm, a);
#pragma unroll
                        for (int nn = 0; nn < NN; ++nn)   // row half c >> 1 carries 2^fpos, taken out at the end
                            mma_f16_16x8x16(o[dm][nn], a, b[nn][0], b[nn][1]);
                    }
                    if constexpr (kMmaRowSum) {
                        const uint32_t ones = lane < 4 ? 0x3C003C00u : 0u;   // f16 1.0 pairs in A row 0
                        const uint32_t a1[4] = {ones, 0u, ones, 0u};
#pragma unroll
                        for (int nn = 0; nn < NN; ++nn)
                            mma_f16_16x8x16(pc[nn], a1, b[nn][0], b[nn][1]);
                    }
                } else {
                    // keys at or past L may hold anything (even NaN): a tail stage zeroes them
                    auto pv_tiles = [&](auto in_tail) {
                        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
                        if constexpr (decltype(in_tail)::value) {
                            const int t = tbase + kk * 16 + cr;
                            mlo = (t < L ? 0x0000ffffu : 0u) | (t + 1 < L ? 0xffff0000u : 0u);
                            mhi = (t + 8 < L ? 0x0000ffffu : 0u) | (t + 9 < L ? 0xffff0000u : 0u);
                        }
#pragma unroll
                        for (int dm = 0; dm < DM; ++dm) {
                            uint32_t a[4];
                            ldsm_x4_trans(vb + (kk / MT) * T::kTileBytes + tile_off<BS>((kk % MT) * 16 + v_key, dm * 2 + v_chs),
                                          a[0], a[1], a[2], a[3]);
                            if constexpr (decltype(in_tail)::value) {
                                a[0] &= mlo;
                                a[1] &= mlo;
                                a[2] &= mhi;
                                a[3] &= mhi;
                            }
#pragma unroll
                            for (int nn = 0; nn < NN; ++nn)
                                mma_bf16_16x8x16(o[dm][nn], a, b[nn][0], b[nn][1]);
                        }
                    };
                    if (tail)
                        pv_tiles(std::true_type{});
                    else
                        pv_tiles(std::false_type{});
                }
            }
            // Remove this stage's code offset: each weight P met 1024 + 2^fpos (c + off), so the O^T
            // elements of dims whose field sits at fpos also gained (1024 + 2^fpos off) * sum(P).
            // Removed every stage, the offset never builds up in the accumulator against the far
            // smaller sum of P c.  (Q8: the row sums sit in row 0 of pc, lanes 0-3, columns 2 l + e;
            // otherwise the lanes' sums are added across the 8 lanes of a row.)
            if constexpr (BITS != 16) {
#pragma unroll
                for (int nn = 0; nn < NN; ++nn)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float v;
                        if constexpr (kMmaRowSum) {
                            v = __shfl_sync(0xffffffffu, pc[nn][e], lane & 3);
                        } else {
                            v = psum[nn][e];
                            v += __shfl_xor_sync(0xffffffffu, v, 4);
                            v += __shfl_xor_sync(0xffffffffu, v, 8);
                            v += __shfl_xor_sync(0xffffffffu, v, 16);
                        }
#pragma unroll
                        for (int dm = 0; dm < DM; ++dm) {
                            o[dm][nn][e] = fmaf(-(1024.f + (float)((1 << fpos<BITS>(dm, 0)) * kCodeOff<BITS>)), v, o[dm][nn][e]);
                            o[dm][nn][2 + e] =
                                fmaf(-(1024.f + (float)((1 << fpos<BITS>(dm, 1)) * kCodeOff<BITS>)), v, o[dm][nn][2 + e]);
                        }
                    }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[st]);
        }

        bool write_out = true;
        if constexpr (KW > 1) {
            // merge the KW key shares in kw order, through the (now idle) stage ring
            asm volatile("bar.sync 1, %0;" ::"r"(NMT * KW * 32) : "memory");
            constexpr int NV = DM * NN * 4 + 4 * NN;
            static_assert((size_t)(KW - 1) * NMT * NV * 32 * 4 <= (size_t)NST * STAGE, "merge needs the ring");
            float *xs = reinterpret_cast<float *>(smem);
            const bool aborted = s_flag[1] != 0;
            if (!aborted && kw > 0) {
                float *dst = xs + (size_t)((kw - 1) * NMT + mw) * NV * 32 + lane;
                int v = 0;
#pragma unroll
                for (int dm = 0; dm < DM; ++dm)
#pragma unroll
                    for (int nn = 0; nn < NN; ++nn)
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            dst[(v++) * 32] = o[dm][nn][c];
#pragma unroll
                for (int nn = 0; nn < NN; ++nn)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        dst[(v++) * 32] = mrow[nn][e];
                        dst[(v++) * 32] = lrow[nn][e];
                    }
            }
            asm volatile("bar.sync 1, %0;" ::"r"(NMT * KW * 32) : "memory");
            write_out = !aborted && kw == 0;
        }
        if (KW > 1 && write_out) {
            constexpr int NV = DM * NN * 4 + 4 * NN;
            const float *xs = reinterpret_cast<const float *>(smem);
            float f[KW][NN][2];
#pragma unroll
            for (int nn = 0; nn < NN; ++nn)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float mx = mrow[nn][e];
#pragma unroll
                    for (int j = 1; j < KW; ++j)
                        mx = fmaxf(mx, xs[((size_t)((j - 1) * NMT + mw) * NV + DM * NN * 4 + nn * 4 + e * 2) * 32 + lane]);
                    f[0][nn][e] = mrow[nn][e] == -INFINITY ? 0.f : fast_exp2(mrow[nn][e] - mx);
#pragma unroll
                    for (int j = 1; j < KW; ++j) {
                        const float mj = xs[((size_t)((j - 1) * NMT + mw) * NV + DM * NN * 4 + nn * 4 + e * 2) * 32 + lane];
                        f[j][nn][e] = mj == -INFINITY ? 0.f : fast_exp2(mj - mx);
                    }
                    lrow[nn][e] *= f[0][nn][e];
#pragma unroll
                    for (int j = 1; j < KW; ++j) {
                        const float *src = xs + ((size_t)((j - 1) * NMT + mw) * NV + DM * NN * 4 + nn * 4 + e * 2) * 32 + lane;
                        lrow[nn][e] += f[j][nn][e] * src[32];
                    }
                    mrow[nn][e] = mx;
                }
#pragma unroll
            for (int dm = 0; dm < DM; ++dm)
#pragma unroll
                for (int nn = 0; nn < NN; ++nn)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float acc = o[dm][nn][c] * f[0][nn][c & 1];
#pragma unroll
                        for (int j = 1; j < KW; ++j)
                            acc += f[j][nn][c & 1] * xs[((size_t)((j - 1) * NMT + mw) * NV + (dm * NN + nn) * 4 + c) * 32 + lane];
                        o[dm][nn][c] = acc;
                    }
        }
        // this split's partial for the rows this warp owns
        if (write_out) {
#pragma unroll
        for (int nn = 0; nn < NN; ++nn)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float v = lrow[nn][e];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                lrow[nn][e] = v;
            }
        if constexpr (BITS != 16) {
            // take out the fields' 2^fpos (exact)
            constexpr int QB = BITS == 16 ? 8 : BITS;
#pragma unroll
            for (int nn = 0; nn < NN; ++nn)
#pragma unroll
                for (int dm = 0; dm < DM; ++dm) {
                    const float u0 = __int_as_float((127 - fpos<QB>(dm, 0)) << 23);
                    const float u1 = __int_as_float((127 - fpos<QB>(dm, 1)) << 23);
                    o[dm][nn][0] *= u0;
                    o[dm][nn][1] *= u0;
                    o[dm][nn][2] *= u1;
                    o[dm][nn][3] *= u1;
                }
        }
#pragma unroll
        for (int nn = 0; nn < NN; ++nn)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = row_base + nn * 8 + cr + e;
                if (j >= M)
                    continue;
                const int w = j / p.group;
                const int h = p.q_head_of[g * p.group + (j - w * p.group)];
                const size_t slot = ((size_t)(row0 + w) * p.num_q_heads + h) * p.n_max + split;
                if (kr == 0)
                    p.part_ml[slot] = make_float2(mrow[nn][e], lrow[nn][e]);
                float *dst = p.part_o + slot * D;
#pragma unroll
                for (int dm = 0; dm < DM; ++dm) {
                    dst[dm * 16 + kr] = o[dm][nn][e];
                    dst[dm * 16 + kr + 8] = o[dm][nn][2 + e];
                }
            }
        }
    }

    // a wait expired: wait (bounded) for the last copy issued into each stage before leaving
    __syncthreads();
    if (s_flag[1] && threadIdx.x == 0) {
        const int issued = s_flag[2];
        for (int st = 0; st < NST && st < issued; ++st) {
            const int k_last = st + ((issued - 1 - st) / NST) * NST;
            if (!mbar_wait_bounded(&full[st], (k_last / NST) & 1, kWaitLimitCycles))
                break;
        }
    }
}

template <int D, int BS, int NN, int NMT, int NST, bool TREE, int BITS, int KW, bool GATHER = false>
__global__ void PKV_KERNEL_BOUNDS(NMT, KW)
paged_attention_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ AttnParams p)
{
    split_kernel_body<D, BS, NN, NMT, NST, TREE, BITS, KW, GATHER>(tm_k, tm_v, p);
}

template <int D, int BS, int NN, int NMT, int NST, bool TREE, int BITS, int KW, bool GATHER = false>
__global__ void __launch_bounds__((NMT * KW + 1) * 32, kMinCtas<BITS, NMT>() > 0 ? kMinCtas<BITS, NMT>() : 1)
paged_attention_kernel_bounded(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                             const __grid_constant__ AttnParams p)
{
    split_kernel_body<D, BS, NN, NMT, NST, TREE, BITS, KW, GATHER>(tm_k, tm_v, p);
}

// Merge of the split partials of one (query row, q head) with the head's sink:
// M = max(m_i, sink), out = sum_i 2^{m_i - M} O_i / (sum_i 2^{m_i - M} l_i + 2^{sink - M}).
// Two warps serve a (row, head): warp h sums, in split order, the partials of its half
// [0, n0) or [n0, n) (n0 = ceil(n / 2)), and the second half's sums are added to the
// first's.  The order depends only on n, i.e. on the row's own length.  Launched as a
// programmatic dependent of the split kernel: it may start early and waits for the
// partials with griddepcontrol.wait.
#ifndef PKV_MERGE_BATCH
#define PKV_MERGE_BATCH 8
#endif
#ifndef PKV_MERGE_MIN_CTAS
#define PKV_MERGE_MIN_CTAS 7
#endif
template <int D>
__global__ void __launch_bounds__(128, PKV_MERGE_MIN_CTAS)
paged_attention_combine_kernel(const AttnParams p)
{
    constexpr int VEC = D / 32;   // output values per lane
    __shared__ float hand[2][VEC + 1][32];   // per pair: the second half's numerators and denominator
    // Everything up to the partials reads only the call's inputs (q_starts, lengths, masks,
    // lists, sinks), which the split kernel does not write and which every earlier kernel on
    // the stream finished writing before the split grid started: that part runs while the
    // split grid drains, and griddepcontrol.wait comes just before the first partial load.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pr = warp >> 1, half = warp & 1;
    const long long wid = (long long)blockIdx.x * 2 + pr;
    if (wid >= (long long)p.total_rows * p.num_q_heads)
        return;   // both warps of the pair leave together
    const int r = (int)(wid / p.num_q_heads);
    const int h = (int)(wid - (long long)r * p.num_q_heads);
    // sequence of row r: the last s with q_starts[s] <= r, by a 32-way search (the table
    // is non-decreasing; q_starts[lo] <= r holds throughout)
    int lo = 0, hi = p.num_seqs - 1;
    while (hi - lo >= 32) {
        const int step = (hi - lo + 32) / 32;
        const int j = lo + lane * step;
        const unsigned m = __ballot_sync(0xffffffffu, j <= hi && __ldg(p.q_starts + j) <= r);
        const int last = m ? 31 - __clz(m) : 0;
        lo += last * step;
        hi = min(hi, lo + step - 1);
    }
    {
        const int j = lo + lane;
        const unsigned m = __ballot_sync(0xffffffffu, j <= hi && __ldg(p.q_starts + j) <= r);
        lo += m ? 31 - __clz(m) : 0;
    }
    const int s = lo;
    const int row0 = __ldg(p.q_starts + s);
    const int W = min(__ldg(p.q_starts + s + 1) - row0, p.max_rows);
    const int w = r - row0;
    if (!p.key_counts && (w < 0 || w >= W))
        return;   // rows past max_q_rows_per_seq were never computed (status already set)
    const int L_cap = (int)min((long long)p.max_context_len, (long long)p.max_blocks_per_seq * p.block_size);
    int L = __ldg(p.context_lens + s);
    L = L < 0 ? 0 : (L > L_cap ? L_cap : L);
    int lim = p.causal ? L - W + w + 1 : L;
    if (p.tree_masks) {   // the row's last visible key is its highest visible window token
        uint32_t m = __ldg(p.tree_masks + r);
        if (W < 32)
            m &= (1u << W) - 1u;
        lim = L - W + (m ? 32 - __clz(m) : 0);
    }
    if (p.key_counts) {   // index-list gather: the row's list length
        const int c = __ldg(p.key_counts + r);
        lim = c < 0 ? 0 : (c > p.max_keys ? p.max_keys : c);
    }
    const int n = lim > 0 ? (lim + kSplitTokens - 1) / kSplitTokens : 0;
    const int n0 = (n + 1) / 2;
    const int i_begin = half ? n0 : 0, i_end = half ? n : n0;
    const size_t base = ((size_t)r * p.num_q_heads + h) * p.n_max;
    const float *src0 = p.part_o + base * D + lane * VEC;
    constexpr int BATCH = PKV_MERGE_BATCH;   // partial rows in flight per lane
    float sink2 = 0.f;
    const bool has_sink = p.sinks != nullptr;
    if (has_sink)
        sink2 = __ldg(p.sinks + h) * kLog2e;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // the first batch of this half's partial rows goes out with the (m, l) loads
    float x0[BATCH][VEC];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
        const int i = i_begin + b;
        if (i < i_end) {
            const float *src = src0 + (size_t)i * D;
            if constexpr (VEC == 4) {
                const float4 t = __ldcg(reinterpret_cast<const float4 *>(src));
                x0[b][0] = t.x, x0[b][1] = t.y, x0[b][2] = t.z, x0[b][3] = t.w;
            } else {
                const float2 t = __ldcg(reinterpret_cast<const float2 *>(src));
                x0[b][0] = t.x, x0[b][1] = t.y;
            }
        }
    }
    // lane i holds (m, l) of partials i, i + 32, ...; both warps find the same M
    constexpr int MAXC = 2;   // partials cached per lane (n <= 64); longer rows reload (m, l)
    float2 mlc[MAXC];
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
        const int i = c * 32 + lane;
        mlc[c] = i < n ? __ldcg(&p.part_ml[base + i]) : make_float2(-INFINITY, 0.f);
    }
    float Mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < MAXC; ++c)
        Mx = fmaxf(Mx, mlc[c].x);
    for (int i = MAXC * 32 + lane; i < n; i += 32)
        Mx = fmaxf(Mx, __ldcg(&p.part_ml[base + i]).x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, off));
    if (has_sink)
        Mx = fmaxf(Mx, sink2);
    float wc[MAXC], lc[MAXC];
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
        wc[c] = fast_exp2(mlc[c].x - Mx);
        lc[c] = mlc[c].y;
    }
    float den = 0.f;
    float num[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v)
        num[v] = 0.f;
    auto accumulate = [&](int i, const float (&xv)[VEC]) {
        float wgt, l_i;
        if (i < MAXC * 32) {
            const int c = i >> 5, srcl = i & 31;
            float wsel = wc[0], lsel = lc[0];
#pragma unroll
            for (int cc = 1; cc < MAXC; ++cc)
                if (c == cc)
                    wsel = wc[cc], lsel = lc[cc];
            wgt = __shfl_sync(0xffffffffu, wsel, srcl);
            l_i = __shfl_sync(0xffffffffu, lsel, srcl);
        } else {
            const float2 ml = __ldcg(&p.part_ml[base + i]);
            wgt = fast_exp2(ml.x - Mx);
            l_i = ml.y;
        }
        den += wgt * l_i;
#pragma unroll
        for (int v = 0; v < VEC; ++v)
            num[v] += wgt * xv[v];
    };
#pragma unroll
    for (int b = 0; b < BATCH; ++b)
        if (i_begin + b < i_end)
            accumulate(i_begin + b, x0[b]);
    for (int i0 = i_begin + BATCH; i0 < i_end; i0 += BATCH) {
        float x[BATCH][VEC];
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
            const int i = i0 + b;
            if (i < i_end) {
                const float *src = src0 + (size_t)i * D;
                if constexpr (VEC == 4) {
                    const float4 t = __ldcg(reinterpret_cast<const float4 *>(src));
                    x[b][0] = t.x, x[b][1] = t.y, x[b][2] = t.z, x[b][3] = t.w;
                } else {
                    const float2 t = __ldcg(reinterpret_cast<const float2 *>(src));
                    x[b][0] = t.x, x[b][1] = t.y;
                }
            }
        }
#pragma unroll
        for (int b = 0; b < BATCH; ++b)
            if (i0 + b < i_end)
                accumulate(i0 + b, x[b]);
    }
    // the second half hands its sums to the first, which adds them after its own
    if (half) {
#pragma unroll
        for (int v = 0; v < VEC; ++v)
            hand[pr][v][lane] = num[v];
        hand[pr][VEC][lane] = den;
    }
    if (pr == 0)   // one named barrier per pair of warps
        asm volatile("bar.sync 1, 64;" ::: "memory");
    else
        asm volatile("bar.sync 2, 64;" ::: "memory");
    if (half)
        return;
#pragma unroll
    for (int v = 0; v < VEC; ++v)
        num[v] += hand[pr][v][lane];
    den += hand[pr][VEC][lane];
    if (has_sink)
        den += fast_exp2(sink2 - Mx);
    float res[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v)
        res[v] = den > 0.f ? num[v] / den : 0.f;
    const size_t oidx = ((size_t)r * p.num_q_heads + h) * D + lane * VEC;
    if (p.out_f32) {
        float *dst = static_cast<float *>(p.out) + oidx;
        if constexpr (VEC == 4)
            *reinterpret_cast<float4 *>(dst) = make_float4(res[0], res[1], res[2], res[3]);
        else
            *reinterpret_cast<float2 *>(dst) = make_float2(res[0], res[1]);
    } else {
        uint16_t *dst = static_cast<uint16_t *>(p.out) + oidx;
        if constexpr (VEC == 4) {
            uint2 pk;
            pk.x = pack_bf16x2(res[0], res[1]);
            pk.y = pack_bf16x2(res[2], res[3]);
            *reinterpret_cast<uint2 *>(dst) = pk;
        } else {
            *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(res[0], res[1]);
        }
    }
}

// ---------------------------------------------------------------- host side --
#ifndef PKV_STAGES_DECODE
#define PKV_STAGES_DECODE 2
#endif
#ifndef PKV_STAGES_WIDE
#define PKV_STAGES_WIDE 2
#endif
// bf16 prefill CTAs (16-row warps; 2 stages: 1521 us, 3: 1486 us)
#ifndef PKV_STAGES_PREFILL
#define PKV_STAGES_PREFILL 3
#endif
#ifndef PKV_STAGES_QUANT
#define PKV_STAGES_QUANT 6
#endif
#ifndef PKV_STAGES_QUANT_WIDE
#define PKV_STAGES_QUANT_WIDE 6
#endif
#ifndef PKV_KW_BF16
#define PKV_KW_BF16 1
#endif
#ifndef PKV_KW_QUANT
#define PKV_KW_QUANT 2
#endif
// key-share warps over 4- and 2-bit records (their per-block work is longer still:
// a Q4 cb_mix call 273 -> 255 us with three)
#ifndef PKV_KW_QUANT_NARROW
#define PKV_KW_QUANT_NARROW 3
#endif
// Ring depth and key-share warps, chosen by measurement on GB300: decode CTAs are many
// and small, wide-row CTAs hold several consumer warps on one ring; a quantised record
// is half or a quarter of a bf16 stage, so its ring can be deeper at the same shared
// memory.  Key-share warps pay off for quantised records (their per-block work is
// longer: two took a Q8 cb_mix call 394 -> 309 us; 4- and 2-bit records take three) but
// not for bf16 pools, whose verify windows lose a third of their speed with two while
// decode gains 1 %.
template <int BITS>
constexpr int kKeyWarps();

#ifndef PKV_STAGES_DEEP
#define PKV_STAGES_DEEP 8
#endif
// DEEP: a grid of at most two CTAs per SM (a few long sequences, e.g. one layer of a
// 4-sequence decode) is bound by the bytes each CTA keeps in flight, not by occupancy:
// such calls get a deeper ring.  Ring depth does not change any row's arithmetic.
// Quantised rings take six stages (from four: a Q8 verify call 366 -> 324 us, a Q8
// cb_mix call 244 -> 233 us; eight cost cb_mix a CTA per SM) and hold at least
// PKV_QUANT_RING_BYTES: a record of fewer bits gets more stages, so each CTA keeps as
// many bytes in flight as a Q8 one (48 KB: Q4 cb_mix 239 -> 236 us, Q2 234 -> 230 us).
// A deep ring is never shallower than that.
#ifndef PKV_QUANT_RING_BYTES
#define PKV_QUANT_RING_BYTES 49152
#endif
// ring depth of the index-list gather (its producer fills stages with 16-byte copies; with
// two blocks per stage: 2 stages 45.7 us, 3: 43.3 us, 4: 60.7 us per sparse_gather call)
#ifndef PKV_STAGES_GATHER
#define PKV_STAGES_GATHER 3
#endif
template <int D, int BS, int NN, int NMT, int BITS, bool DEEP = false, bool GATHER = false>
constexpr int kStages()
{
    constexpr int tb = kBlocksPerStage<BITS, BS>;
    constexpr int stage = BITS == 16 ? 2 * tb * Tile<D, BS>::kTileBytes : tb * QRec<D, BS, (BITS == 16 ? 8 : BITS)>::kBytes;
    constexpr int by_bytes = BITS != 16 ? (PKV_QUANT_RING_BYTES + stage - 1) / stage : 0;
    constexpr int quant_base = NMT > 1 ? PKV_STAGES_QUANT_WIDE : PKV_STAGES_QUANT;
    constexpr int quant = quant_base > by_bytes ? quant_base : by_bytes;
    constexpr int deep = BITS != 16 && quant > PKV_STAGES_DEEP ? quant : PKV_STAGES_DEEP;
    constexpr int base = DEEP ? deep : BITS != 16 ? quant : GATHER ? PKV_STAGES_GATHER : NMT == 1 ? PKV_STAGES_DECODE
                                                         : NN > 1 ? PKV_STAGES_PREFILL : PKV_STAGES_WIDE;
    // the KW - 1 key shares' states pass through the ring at the end: make it big enough
    constexpr int merge = (kKeyWarps<BITS>() - 1) * NMT * (D / 16 * 4 + 4) * NN * 32 * 4;
    constexpr int need = (merge + stage - 1) / stage;
    constexpr int kw = kKeyWarps<BITS>();
    constexpr int n = base > need ? base : need;
    return (n + kw - 1) / kw * kw;   // a multiple of the key-share warps (see the kernel)
}

// consumer warps sharing each row group's keys (the same for every CTA shape of a codec)
template <int BITS>
constexpr int kKeyWarps()
{
    return BITS == 16 ? PKV_KW_BF16 : BITS == 8 ? PKV_KW_QUANT : PKV_KW_QUANT_NARROW;
}

template <int D, int BS, int NN, int NMT, int BITS, bool DEEP = false, bool GATHER = false>
constexpr size_t smem_bytes()
{
    constexpr int NST = kStages<D, BS, NN, NMT, BITS, DEEP, GATHER>();
    constexpr size_t tb = kBlocksPerStage<BITS, BS>;
    constexpr size_t stage = BITS == 16 ? 2 * tb * (size_t)Tile<D, BS>::kTileBytes
                                        : tb * (size_t)QRec<D, BS, (BITS == 16 ? 8 : BITS)>::kBytes;
    // + the flags (64 B) and, for the index-list gather, a split's row offsets
    return 1024 + (size_t)NST * stage + 2 * NST * sizeof(uint64_t) + 64 + (GATHER ? (size_t)kSplitTokens * 8 : 0);
}

template <int D, int BS, int NN, int NMT, bool TREE, int BITS, bool GATHER = false, bool DEEP = false>
int launch_t(const CUtensorMap &mk, const CUtensorMap &mv, const AttnParams &prm, dim3 grid,
             cudaStream_t st)
{
    constexpr int NST = kStages<D, BS, NN, NMT, BITS, DEEP, GATHER>();
    constexpr int KW = GATHER ? 1 : kKeyWarps<BITS>();
    void (*kern)(const CUtensorMap, const CUtensorMap, const AttnParams);
    if constexpr (kMinCtas<BITS, NMT>() > 0)
        kern = paged_attention_kernel_bounded<D, BS, NN, NMT, NST, TREE, BITS, KW, GATHER>;
    else
        kern = paged_attention_kernel<D, BS, NN, NMT, NST, TREE, BITS, KW, GATHER>;
    constexpr size_t smem = smem_bytes<D, BS, NN, NMT, BITS, DEEP, GATHER>();
    static_assert(smem <= 232448, "split kernel: shared memory per CTA");
    // A function attribute belongs to a context: set it before every launch, so that a
    // second device, or a context created after a reset, gets it too (the call is cheap).
    const cudaError_t attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (attr_err != cudaSuccess)
        return check_cuda(attr_err, "cudaFuncSetAttribute(max dynamic smem)");
    kern<<<grid, (NMT * KW + 1) * 32, smem, st>>>(mk, mv, prm);
    int rc = check_cuda(cudaGetLastError(), "paged attention split launch");
    if (rc)
        return rc;
    // merge, as a programmatic dependent launch (its launch overlaps the split grid's tail);
    // a CTA of four warps serves two (row, q head) units
    const long long units = (long long)prm.total_rows * prm.num_q_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((units + 1) / 2));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return check_cuda(cudaLaunchKernelEx(&cfg, paged_attention_combine_kernel<D>, prm),
                      "paged attention merge launch");
}

// Rows of one (s, g) (G * max rows per sequence) -> one consumer warp per CTA with 8
// rows (decode) or several consumer warps in several row-group CTAs (verify windows).
// Row-group CTAs of one split are adjacent in launch order and share each K/V tile
// through L2.
#ifndef PKV_WIDE_NN
#define PKV_WIDE_NN 1
#endif
#ifndef PKV_WIDE_NMT
#define PKV_WIDE_NMT 3
#endif
// Prefill chunks (more than PKV_PREFILL_ROWS rows per (sequence, KV head), beyond any
// verify window) get 16 rows per consumer warp: each K / V fragment then feeds two MMAs
// (prefill_mix 2.11 -> 1.88 ms per call); verify windows keep 8 (16 made them 14 % slower).
// Which n-tile a row lands in does not change its arithmetic.
#ifndef PKV_PREFILL_ROWS
#define PKV_PREFILL_ROWS 64
#endif
// row warps of a wide-row CTA over quantised records, each with the codec's key shares
// (Q8, two key shares: 2 row warps -> a verify call 358 us, 3 -> 408 us, 1 -> 418 us;
// Q4 / Q2, three key shares: 1 row warp -> a Q4 verify call 442 us, 2 -> 514 us)
#ifndef PKV_WIDE_NMT_QUANT
#define PKV_WIDE_NMT_QUANT 2
#endif
#ifndef PKV_WIDE_NMT_QUANT_NARROW
#define PKV_WIDE_NMT_QUANT_NARROW 1
#endif
// 8-row n-tiles per row warp of a wide CTA over Q8 / Q4 and Q2 records: a 4- or 2-bit
// warp widens each code for two n-tiles (Q4 verify call 365 -> 331 us, Q2 349 -> 328 us;
// Q8 300 -> 401 us, so it keeps one)
#ifndef PKV_WIDE_NN_QUANT
#define PKV_WIDE_NN_QUANT 1
#endif
#ifndef PKV_WIDE_NN_QUANT_NARROW
#define PKV_WIDE_NN_QUANT_NARROW 2
#endif
template <int D, int BS, int BITS, bool WITH_TREE>
int launch_d_bs(int rows, const CUtensorMap &mk, const CUtensorMap &mv, AttnParams prm,
                long long pairs, int n_max, cudaStream_t st)
{
    constexpr int WIDE_NMT = BITS == 16 ? PKV_WIDE_NMT : BITS == 8 ? PKV_WIDE_NMT_QUANT : PKV_WIDE_NMT_QUANT_NARROW;
    constexpr int WIDE_NN = BITS == 16 ? PKV_WIDE_NN : BITS == 8 ? PKV_WIDE_NN_QUANT : PKV_WIDE_NN_QUANT_NARROW;
    const bool prefill = BITS == 16 && !prm.tree_masks && rows > PKV_PREFILL_ROWS;
    const int per_cta = rows <= 8 ? 8 : prefill ? 8 * 2 * PKV_WIDE_NMT : 8 * WIDE_NN * WIDE_NMT;
    prm.row_groups = (rows + per_cta - 1) / per_cta;
    const long long gx = pairs * prm.row_groups;
    if (gx > 0x7fffffffLL || n_max > 65535)
        return set_error(PKV_ERR_SHAPE, "paged attention: grid too large");
    const dim3 grid((unsigned)gx, (unsigned)n_max);
    const bool deep = gx * n_max <= 2LL * sm_count();   // few, long CTAs: keep more bytes in flight
    if constexpr (WITH_TREE) {
        if (prm.tree_masks)
            return rows <= 8 ? launch_t<D, BS, 1, 1, true, BITS>(mk, mv, prm, grid, st)
                             : launch_t<D, BS, PKV_WIDE_NN, PKV_WIDE_NMT, true, BITS>(mk, mv, prm, grid, st);
    }
    if (rows <= 8)
        return deep ? launch_t<D, BS, 1, 1, false, BITS, false, true>(mk, mv, prm, grid, st)
                    : launch_t<D, BS, 1, 1, false, BITS>(mk, mv, prm, grid, st);
    if constexpr (BITS == 16) {
        if (prefill)
            return launch_t<D, BS, 2, PKV_WIDE_NMT, false, BITS>(mk, mv, prm, grid, st);
    }
    return launch_t<D, BS, WIDE_NN, WIDE_NMT, false, BITS>(mk, mv, prm, grid, st);
}

struct WsLayout {
    size_t ml, o, units, ctl, total;
};

// Workspace: the split partials (m, l) and O, then (tensor-core path) the unit list and its
// counters.  A sequence of W rows has ceil(G W / 16) row groups at most, so the units of a
// split number at most H_kv (G R / 16 + S') with S' = max(S, R) (the index-list gather
// lists rows, not sequences).
WsLayout ws_layout(int32_t num_seqs, int32_t total_q_rows, int32_t num_q_heads, int32_t num_kv_heads,
                   int32_t head_dim, int32_t max_context_len)
{
    const size_t n_max = (size_t)(max_context_len > 0 ? (max_context_len + kSplitTokens - 1) / kSplitTokens : 1);
    const size_t slots = (size_t)total_q_rows * num_q_heads * n_max;
    const size_t G = (size_t)(num_q_heads / (num_kv_heads > 0 ? num_kv_heads : 1));
    const size_t src = (size_t)(num_seqs > total_q_rows ? num_seqs : total_q_rows);
    const size_t units = n_max * (size_t)num_kv_heads * ((G * total_q_rows + 15) / 16 + src);
    WsLayout w;
    w.ml = 0;
    w.o = round_up(slots * sizeof(float2), 256);
    w.units = w.o + round_up(slots * head_dim * sizeof(float), 256);
    w.ctl = w.units + round_up(units * 16, 256);
    w.total = w.ctl + 256;
    return w;
}


// What a pool gives the attention: geometry, and either bf16 K/V pools or records.
struct PoolView {
    int32_t num_blocks, block_size, num_kv_heads, head_dim, bits;   // bits: 16, 8 or 4
    const void *k_pool, *v_pool;   // bits == 16
    const void *records;           // bits 8 / 4
    const int32_t *key_idx = nullptr;      // index-list gather: [R][max_keys], or null
    const int32_t *key_counts = nullptr;   // [R]
    int32_t max_keys = 0;
};

// Called with validated parameters: launches the split and merge kernels.
using LaunchFn = int (*)(const PoolView &pv, AttnParams &prm, int rows, long long pairs, int n_max,
                         cudaStream_t st);

// Argument checks shared by every attention entry point, then the launch.
inline int attention_run(const char *who, const PoolView &pv, const void *q, const int32_t *q_starts,
                         const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                         int32_t num_seqs, int32_t total_q_rows, int32_t max_context_len,
                         int32_t max_q_rows_per_seq, int32_t num_q_heads, const int32_t *kv_head_of_q_head,
                         const float *sinks, int32_t causal, const uint32_t *tree_masks, float scale, void *out,
                         int32_t out_dtype, void *workspace, size_t workspace_bytes, void *stream, LaunchFn launch)
{
    const int D = pv.head_dim, BS = pv.block_size, Hkv = pv.num_kv_heads;
    if (num_seqs < 0 || total_q_rows < 0 || max_context_len < 0 || max_q_rows_per_seq < 0)
        return set_error(PKV_ERR_SHAPE, "%s: negative size", who);
    if (pv.num_blocks <= 0 || Hkv <= 0 || max_blocks_per_seq <= 0)
        return set_error(PKV_ERR_SHAPE, "%s: pool sizes and max_blocks_per_seq must be positive", who);
    if (!(D == 64 || D == 128))
        return set_error(PKV_ERR_UNSUPPORTED, "%s: head_dim %d (built: 64, 128)", who, D);
    if (!(BS == 16 || BS == 32))
        return set_error(PKV_ERR_UNSUPPORTED, "%s: block_size %d (built: 16, 32)", who, BS);
    if (num_q_heads <= 0 || num_q_heads > kMaxQHeads || num_q_heads % Hkv != 0)
        return set_error(PKV_ERR_SHAPE,
                         "%s: num_q_heads %d must be a positive multiple of "
                         "num_kv_heads %d and at most %d", who, num_q_heads, Hkv, kMaxQHeads);
    if (out_dtype != PKV_DTYPE_BF16 && out_dtype != PKV_DTYPE_F32)
        return set_error(PKV_ERR_SHAPE, "%s: out_dtype %d", who, out_dtype);
    if ((long long)max_blocks_per_seq * BS < max_context_len)
        return set_error(PKV_ERR_SHAPE,
                         "%s: max_context_len %d exceeds max_blocks_per_seq * "
                         "block_size = %lld", who, max_context_len, (long long)max_blocks_per_seq * BS);
    if ((long long)pv.num_blocks * Hkv * BS > 0x7fffffffLL)
        return set_error(PKV_ERR_UNSUPPORTED,
                         "%s: pool too large for 32-bit TMA row coordinates", who);
    const int G = num_q_heads / Hkv;
    if (num_seqs == 0 || total_q_rows == 0)
        return PKV_OK;
    if (max_q_rows_per_seq <= 0)
        return set_error(PKV_ERR_SHAPE, "%s: max_q_rows_per_seq must be >= 1", who);
    if ((long long)G * max_q_rows_per_seq > kMaxGroupRows)
        return set_error(PKV_ERR_UNSUPPORTED,
                         "%s: group %d x max rows %d exceeds %d", who, G,
                         max_q_rows_per_seq, kMaxGroupRows);
    const bool pools_ok = pv.bits == 16 ? (pv.k_pool && pv.v_pool) : pv.records != nullptr;
    if (!pools_ok || !q || !q_starts || !block_tables || !context_lens || !out || !workspace)
        return set_error(PKV_ERR_NULL, "%s: a required pointer is NULL", who);
    const bool pools_aligned = pv.bits == 16 ? (aligned16(pv.k_pool) && aligned16(pv.v_pool))
                                             : aligned16(pv.records);
    if (!pools_aligned || !aligned16(q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return set_error(PKV_ERR_ALIGN,
                         "%s: pools, q and out must be 16-byte aligned, "
                         "workspace 256-byte aligned", who);
    const WsLayout wl = ws_layout(num_seqs, total_q_rows, num_q_heads, Hkv, D, max_context_len);
    if (workspace_bytes < wl.total)
        return set_error(PKV_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", who,
                         workspace_bytes, wl.total);

    AttnParams prm;
    memset(&prm, 0, sizeof prm);
    // GQA map: q heads of each KV head, in increasing q-head order
    {
        int fill[kMaxQHeads] = {0};
        for (int h = 0; h < num_q_heads; ++h) {
            const int gg = kv_head_of_q_head ? kv_head_of_q_head[h] : h / G;
            if (gg < 0 || gg >= Hkv || fill[gg] >= G)
                return set_error(PKV_ERR_SHAPE,
                                 "%s: kv_head_of_q_head must give each of the %d "
                                 "KV heads exactly %d q heads (entry %d = %d)", who, Hkv, G, h, gg);
            prm.q_head_of[gg * G + fill[gg]++] = (int16_t)h;
        }
    }
    int32_t *status = device_status_word();
    if (!status)
        return set_error(PKV_ERR_CUDA, "%s: no device status word", who);

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int n_max = max_context_len > 0 ? (max_context_len + kSplitTokens - 1) / kSplitTokens : 1;
    prm.q = static_cast<const uint16_t *>(q);
    prm.q_starts = q_starts;
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.sinks = sinks;
    prm.tree_masks = tree_masks;
    prm.out = out;
    prm.part_ml = reinterpret_cast<float2 *>(ws + wl.ml);
    prm.part_o = reinterpret_cast<float *>(ws + wl.o);
    prm.units = reinterpret_cast<const int4 *>(ws + wl.units);
    prm.unit_ctl = reinterpret_cast<int32_t *>(ws + wl.ctl);
    prm.unit_cap = (long long)((wl.ctl - wl.units) / 16);
    prm.qrec = static_cast<const uint8_t *>(pv.records);
    prm.kpool = static_cast<const uint16_t *>(pv.k_pool);
    prm.vpool = static_cast<const uint16_t *>(pv.v_pool);
    prm.key_idx = pv.key_idx;
    prm.key_counts = pv.key_counts;
    prm.max_keys = pv.max_keys;
    prm.status = status;
    prm.wait_limit = pipeline_wait_limit();
    prm.num_seqs = num_seqs;
    prm.max_blocks_per_seq = max_blocks_per_seq;
    prm.num_blocks = pv.num_blocks;
    prm.num_q_heads = num_q_heads;
    prm.num_kv_heads = Hkv;
    prm.block_size = BS;
    prm.group = G;
    prm.n_max = n_max;
    prm.max_context_len = max_context_len;
    prm.max_rows = max_q_rows_per_seq;
    prm.total_rows = total_q_rows;
    prm.causal = causal ? 1 : 0;
    prm.out_f32 = out_dtype == PKV_DTYPE_F32;
    const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
    prm.scale_log2 = sc * kLog2e;

    const int rows = G * max_q_rows_per_seq;
    const long long pairs = (long long)num_seqs * Hkv;
    return launch(pv, prm, rows, pairs, n_max, static_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace pkv
