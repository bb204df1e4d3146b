// pkv_attention_tc.cuh -- bf16 paged attention on the 5th-generation tensor cores
// (tcgen05.mma with tensor-memory accumulators), for decode rows, verify windows, draft
// trees, prefill chunks and the index-list gather alike.
//
// What it computes: TensorSharp "高级功能", section "原生分页注意力" -- each sequence's
// query rows attend over K/V gathered from the paged block pool through its block table
// (with the per-head sink variant, merged by the merge kernel); TensorFold article,
// section "先记住一条铁律" -- a verify row takes exactly the serial step's arithmetic and
// a row computed in a batch equals the row computed alone.
//
// Work unit = (sequence s, KV head g, 512-key split i, row group): up to RPU query rows
// (the G q heads of g times the sequence's rows, flattened row = w * G + head_in_group).
// A one-CTA pass lists the units (splits in decreasing order, so the grid ends on every
// sequence's first splits, where shared prefix blocks live); a persistent grid of one CTA
// per SM takes them from an atomic counter.  Inside a CTA:
//  * a scheduler warp takes units, writes each unit's query rows into shared memory in
//    the MMA's operand layout and resolves its block ids (one unit ahead);
//  * two producer warps stream the split's K blocks and V blocks through the block table
//    with TMA tile loads (or, for the index-list gather, cp.async row copies) into two
//    rings of 128-key tiles, so K tiles, which the QK products consume first, turn over
//    without waiting for V;
//  * the MMA warp (one thread) issues, per 128-key tile t of a split, S_t^T = K_t q^T on
//    the tensor core (keys on the MMA's M side, query rows on N) into its own
//    tensor-memory slot, and later O^T += V_t^T P_t^T (head dims on M, rows on N), which
//    accumulates over the split's tiles in tensor memory;
//  * four softmax warps, thread = tensor-memory lane (a key of the tile for S, a head dim
//    for O), take a split in two passes: pass 1 reads every tile's scores, scales and
//    masks them (length, causal window, tree ancestors) and forms each row's maximum over
//    the split in base 2 (a warp reduce-scatter, then the four warps' maxima -- one
//    exchange per split); pass 2 writes the weights p = 2^(x - m), rounded to bf16, into
//    shared memory for the PV product and keeps per-thread partial sums of them.
// A split's partial (m, l, O) goes to the workspace; the merge kernel combines a row's
// splits in an order fixed by its own length, with the sink.
//
// Invariance: a row's operations depend only on its own sequence -- the split grid and
// the 128-key tiles are anchored at token 0, the MMA computes each output column from
// that column's operands only (the same bits at any N), the max is exact, and every sum
// (the weights' partials and their final reduction, the PV accumulation over the tiles)
// runs in a fixed order.  Keys past a row's limit get weight exactly 0, and V rows past
// the keys of the unit are zeroed in shared memory before the PV product (0 * NaN would
// not be 0).
#pragma once

#include <climits>

#include "pkv_attention_impl.cuh"
#include "pkv_tc.cuh"

namespace pkv {
namespace {

constexpr int kTileKeys = 128;                        // keys per MMA tile (the M side of S^T)
constexpr int kTilesPerSplit = kSplitTokens / kTileKeys;
static_assert(kSplitTokens % kTileKeys == 0, "a split is whole 128-key tiles");
constexpr int kTcMaxSeqs = 8192;                      // sequences (or gather rows) the unit pass sorts
constexpr int kTcMaxSplits = 4096;                    // 512-key splits of the longest context

// ---------------------------------------------------------------- unit pass --
struct UnitPassParams {
    const int32_t *q_starts, *context_lens, *key_counts;
    int4 *units;         // out: (s, split, g, row group)
    int32_t *ctl;        // out: [0] the CTAs' work counter (set to 0), [1] unit count
    int32_t *status;
    int32_t num_src;     // sequences (or query rows, for the index-list gather)
    int32_t num_seqs, total_rows, max_rows, group, num_kv_heads, rpu, max_keys;
    int32_t L_cap, n_max;
    long long unit_cap;  // entries the unit list has room for
};

// One CTA of 1024 threads.  Sequences sorted by split count (descending, then index) make
// the sequences that reach split i a prefix of the order, so split i's units are the first
// cum[c_i] entries of one running sum; the list is written split by split, highest first.
__global__ void __launch_bounds__(1024) attention_unit_pass(const UnitPassParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const int S = p.num_src;
    int P2 = 1;
    while (P2 < S)
        P2 <<= 1;
    unsigned long long *key = reinterpret_cast<unsigned long long *>(smem_raw);   // [P2]
    int32_t *rgs = reinterpret_cast<int32_t *>(key + P2);                         // [S] row groups per seq
    int32_t *cum = rgs + S;                                                       // [S + 1]
    int32_t *cnt = cum + S + 1;                                                   // [n_max] units of split i
    int32_t *base = cnt + p.n_max;                                                // [n_max] first unit of split i
    __shared__ int32_t warp_sum[32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const bool gather = p.key_counts != nullptr;
    // the attention grid may start its set-up now; it waits for this grid before reading the list
    asm volatile("griddepcontrol.launch_dependents;");
    for (int s = t; s < P2; s += blockDim.x) {
        if (s >= S) {
            key[s] = ~0ull;
            continue;
        }
        int L, W;
        if (gather) {
            L = __ldg(p.key_counts + s);
            if (L < 0 || L > p.max_keys) {
                atomicOr(p.status, PKV_DEV_TABLE_OVERRUN);
                L = L < 0 ? 0 : p.max_keys;
            }
            W = 1;
        } else {
            L = __ldg(p.context_lens + s);
            if (L < 0 || L > p.L_cap) {
                atomicOr(p.status, PKV_DEV_TABLE_OVERRUN);
                L = L < 0 ? 0 : p.L_cap;
            }
            const int r0 = __ldg(p.q_starts + s);
            W = __ldg(p.q_starts + s + 1) - r0;
            if (W > 0 && (r0 < 0 || r0 + W > p.total_rows)) {
                atomicOr(p.status, PKV_DEV_TOO_MANY_ROWS);
                W = 0;
            }
            if (W > p.max_rows) {
                atomicOr(p.status, PKV_DEV_TOO_MANY_ROWS);
                W = p.max_rows;
            }
        }
        const int n = W > 0 ? (L + kSplitTokens - 1) / kSplitTokens : 0;
        rgs[s] = W > 0 ? (p.group * W + p.rpu - 1) / p.rpu : 0;
        key[s] = ((unsigned long long)(0xFFFFu - (unsigned)n) << 32) | (unsigned)s;
    }
    __syncthreads();
    // bitonic sort, ascending keys = split count descending, then sequence ascending
    for (int k = 2; k <= P2; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = t; i < P2; i += blockDim.x) {
                const int ij = i ^ j;
                if (ij > i) {
                    const unsigned long long a = key[i], b = key[ij];
                    if (((i & k) == 0) == (a > b)) {
                        key[i] = b;
                        key[ij] = a;
                    }
                }
            }
            __syncthreads();
        }
    // cum[k] = units of the first k sorted sequences (H_kv * row groups each)
    int carry = 0;
    for (int c0 = 0; c0 < S; c0 += blockDim.x) {
        const int k = c0 + t;
        const int v = k < S ? p.num_kv_heads * rgs[(int)(unsigned)key[k]] : 0;
        int x = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off)
                x += y;
        }
        if (lane == 31)
            warp_sum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = warp_sum[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off)
                    w += y;
            }
            warp_sum[lane] = w;
        }
        __syncthreads();
        if (k < S)
            cum[k] = carry + (warp > 0 ? warp_sum[warp - 1] : 0) + x - v;
        carry += warp_sum[31];
        __syncthreads();
    }
    if (t == 0)
        cum[S] = carry;
    __syncthreads();
    // units of split i: the sorted sequences with more than i splits are a prefix
    for (int i = t; i < p.n_max; i += blockDim.x) {
        int lo = 0, hi = S;   // first k whose split count is <= i
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            const int n_mid = (int)(0xFFFFu - (unsigned)(key[mid] >> 32));
            if (n_mid > i)
                lo = mid + 1;
            else
                hi = mid;
        }
        cnt[i] = cum[lo];
    }
    __syncthreads();
    if (t == 0) {   // splits in decreasing order
        long long b = 0;
        for (int i = p.n_max - 1; i >= 0; --i) {
            base[i] = (int)min(b, (long long)INT_MAX);
            b += cnt[i];
        }
        if (b > p.unit_cap) {   // only when q_starts is not increasing (row ranges overlap)
            atomicOr(p.status, PKV_DEV_TOO_MANY_ROWS);
            b = p.unit_cap;
        }
        p.ctl[0] = 0;
        p.ctl[1] = (int)b;
        warp_sum[0] = (int)b;
    }
    __syncthreads();
    const int U = warp_sum[0];
    for (int u = t; u < U; u += blockDim.x) {
        // base[] does not increase with i: the unit's split is the smallest i with base[i] <= u
        int lo = 0, hi = p.n_max - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (base[mid] <= u)
                hi = mid;
            else
                lo = mid + 1;
        }
        const int i = lo;
        const int r = u - base[i];
        int a = 0, b = S - 1;   // the last k with cum[k] <= r
        while (a < b) {
            const int mid = (a + b + 1) >> 1;
            if (cum[mid] <= r)
                a = mid;
            else
                b = mid - 1;
        }
        const int s = (int)(unsigned)key[a];
        const int rem = r - cum[a];
        const int rg = rgs[s];
        p.units[u] = make_int4(s, i, rem / rg, rem % rg);
    }
}

inline size_t unit_pass_smem(int num_src, int n_max)
{
    int P2 = 1;
    while (P2 < num_src)
        P2 <<= 1;
    return (size_t)P2 * 8 + (size_t)num_src * 4 + (size_t)(num_src + 1) * 4 + (size_t)n_max * 8 + 64;
}

// ---------------------------------------------------------------- main kernel --
template <int D, int RPU>
struct TcLayout {
    static constexpr int kHalves = D / 64;
    static constexpr int kKvTile = kTileKeys * D * 2;          // one K (or V) tile: 128 keys x D bf16
    static constexpr int kQBuf = RPU * D * 2;                  // query rows of a unit
    static constexpr int kPBuf = RPU * kTileKeys * 2;          // bf16 weights of a tile
    static_assert(RPU == 16 || RPU == 32 || RPU == 64, "rows per unit");
};

struct UnitDesc {
    int32_t valid, s, g, split, L, W, row0, m_rows, t0, ntile, n_mma;
};

// unit slots (descriptor, query rows) and weight buffers: more for the short rows of decode
template <int RPU>
constexpr int kUnitSlots = RPU == 16 ? 3 : 2;
template <int RPU>
constexpr int kPBufs = RPU == 16 ? 4 : 2;

template <int D, int BS, int RPU, int NK, int NV, bool TREE, bool GATHER>
constexpr size_t tc_smem_bytes()
{
    using Y = TcLayout<D, RPU>;
    constexpr int NU = kUnitSlots<RPU>, NPB = kPBufs<RPU>;
    return 1024 + (size_t)(NK + NV) * Y::kKvTile + (size_t)NU * Y::kQBuf + (size_t)NPB * Y::kPBuf
           + 4 * RPU * 4       // red: per-column maxima / sums of the four softmax warps
           + RPU * 4           // each row's maximum over the split
           + NU * RPU * 12     // per-unit column limits, tree masks, output rows
           + kMaxQHeads * 2    // the GQA head map
           + NU * sizeof(UnitDesc) + NU * (kSplitTokens / BS) * 4 + 512   // unit slots, block ids, barriers, flags
           + (GATHER ? (size_t)NU * kSplitTokens * 8 : 0);
}

// Lane quarter of warp w's tensor-memory accesses, and a column address.
__device__ __forceinline__ uint32_t tmem_at(uint32_t base, int quarter, int col)
{
    return base + ((uint32_t)(32 * quarter) << 16) + (uint32_t)col;
}

// 16 columns' maxima (or sums) over the warp's 32 lanes, reduced and scattered: afterwards
// lane l holds the result for column ((l >> 4) & 1) * 8 + ((l >> 3) & 1) * 4 +
// ((l >> 2) & 1) * 2 + ((l >> 1) & 1) (lanes l and l ^ 1 agree).  A fixed pattern, so a
// sum's order of operations is fixed too.
template <bool MAX>
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane)
{
    float a[8], b[4], c[2];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const bool hi = lane & 16;
        const float send = hi ? v[k] : v[k + 8];
        const float keep = hi ? v[k + 8] : v[k];
        const float got = __shfl_xor_sync(0xffffffffu, send, 16);
        a[k] = MAX ? fmaxf(keep, got) : keep + got;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const bool hi = lane & 8;
        const float send = hi ? a[k] : a[k + 4];
        const float keep = hi ? a[k + 4] : a[k];
        const float got = __shfl_xor_sync(0xffffffffu, send, 8);
        b[k] = MAX ? fmaxf(keep, got) : keep + got;
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const bool hi = lane & 4;
        const float send = hi ? b[k] : b[k + 2];
        const float keep = hi ? b[k + 2] : b[k];
        const float got = __shfl_xor_sync(0xffffffffu, send, 4);
        c[k] = MAX ? fmaxf(keep, got) : keep + got;
    }
    const bool hi = lane & 2;
    const float send = hi ? c[0] : c[1];
    const float keep = hi ? c[1] : c[0];
    const float got = __shfl_xor_sync(0xffffffffu, send, 2);
    const float r = MAX ? fmaxf(keep, got) : keep + got;
    const float o = __shfl_xor_sync(0xffffffffu, r, 1);
    return MAX ? fmaxf(r, o) : r + o;   // (a + b == b + a: both lanes agree)
}

__device__ __forceinline__ int rs_col(int lane)
{
    return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

// Named barrier of the softmax warps that also ORs a predicate over them: every thread gets
// the same answer, so the four warps take the same branch after it.
__device__ __forceinline__ bool softmax_bar_any(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, 1, 128, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

// Warp roles: 0 K side (K tile loads and the QK products; owns the tensor memory), 1 V side
// (V tile loads and the PV products), 2..5 softmax, 6 scheduler.  Each side's loads run
// ahead of its products by its ring depth, at most NU - 1 units ahead.
constexpr int kTcThreads = 224;

// A position in the stream of (unit, tile) pairs a CTA works through, reading the units'
// descriptors from the unit slots.
struct TileCursor {
    int uidx, t;     // unit (in this CTA's order) and tile within it
    bool valid;      // false once the stream has ended
    UnitDesc d;
};

template <int D, int BS, int RPU, int NK, int NV, bool TREE, bool GATHER>
__global__ void __launch_bounds__(kTcThreads, 1)
paged_attention_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          const AttnParams p)
{
    using Y = TcLayout<D, RPU>;
    constexpr int C = kSplitTokens;
    constexpr int BPT = kTileKeys / BS;     // blocks per 128-key tile
    constexpr int NBS = C / BS;             // blocks per split
    constexpr int NCH = RPU / 16;           // 16-column chunks of a unit
    constexpr int TPS = kTilesPerSplit;     // tile slots (S buffers) of a split
    constexpr int NU = kUnitSlots<RPU>;     // unit slots
    constexpr int NPB = kPBufs<RPU>;        // weight buffers
    constexpr bool KEEP = NCH == 1;         // one chunk: the split's scores stay in registers
    constexpr uint32_t kTmemNeed = (TPS + 1) * RPU;   // S slots, then O
    constexpr uint32_t kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                 : kTmemNeed <= 256 ? 256 : 512;
    static_assert(!(GATHER && (TREE || BS != 16)), "index-list gather: 16-key blocks");
    static_assert(!KEEP || NPB >= TPS, "decode keeps a weight buffer per tile");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *kring = smem;
    uint8_t *vring = kring + NK * Y::kKvTile;
    uint8_t *qbuf = vring + NV * Y::kKvTile;
    uint8_t *pbuf = qbuf + NU * Y::kQBuf;
    float *red = reinterpret_cast<float *>(pbuf + NPB * Y::kPBuf);   // [RPU][4]
    float *mbuf = red + 4 * RPU;                                      // [RPU]
    int32_t *lim_s = reinterpret_cast<int32_t *>(mbuf + RPU);        // [NU][RPU]
    uint32_t *tmk_s = reinterpret_cast<uint32_t *>(lim_s + NU * RPU);  // [NU][RPU]
    int32_t *orow_s = reinterpret_cast<int32_t *>(tmk_s + NU * RPU);   // [NU][RPU] output row * H_q + q head
    int16_t *hmap_s = reinterpret_cast<int16_t *>(orow_s + NU * RPU);  // [kMaxQHeads]
    UnitDesc *udesc = reinterpret_cast<UnitDesc *>(hmap_s + kMaxQHeads);  // [NU]
    int32_t *blk_s = reinterpret_cast<int32_t *>(udesc + NU);          // [NU][NBS] block ids of a unit's split
    uint64_t *bars = reinterpret_cast<uint64_t *>(
        (reinterpret_cast<uintptr_t>(blk_s + NU * NBS) + 7) & ~uintptr_t(7));
    uint64_t *k_full = bars, *k_empty = k_full + NK;
    uint64_t *v_full = k_empty + NK, *v_empty = v_full + NV;
    uint64_t *q_full = v_empty + NV, *q_empty = q_full + NU;
    uint64_t *u_full = q_empty + NU, *u_empty = u_full + NU;
    uint64_t *s_full = u_empty + NU, *s_empty = s_full + TPS;
    uint64_t *p_full = s_empty + TPS, *p_empty = p_full + NPB;
    uint64_t *o_full = p_empty + NPB, *o_empty = o_full + 1;
    uint64_t *mma_done = o_empty + 1;                     // [2]: the K side and the V side
    volatile int32_t *flag = reinterpret_cast<volatile int32_t *>(mma_done + 2);   // [0] abort, [1] K, [2] V tiles issued
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 2) + 3;
    unsigned long long *g_off = reinterpret_cast<unsigned long long *>(mma_done + 4);   // (gather) [NU][C]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int h = threadIdx.x; h < p.num_q_heads; h += blockDim.x)
        hmap_s[h] = p.q_head_of[h];
    if (threadIdx.x == 0) {
        for (int i = 0; i < NK; ++i) {
            mbar_init(&k_full[i], GATHER ? 32 : 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&v_full[i], GATHER ? 32 : 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int b = 0; b < NU; ++b) {
            mbar_init(&q_full[b], 1);
            mbar_init(&q_empty[b], 1);
            mbar_init(&u_full[b], 1);
            mbar_init(&u_empty[b], 6);   // the K and V sides and the four softmax warps
        }
        for (int t = 0; t < TPS; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&s_empty[t], 4);
        }
        for (int b = 0; b < NPB; ++b) {
            mbar_init(&p_full[b], 4);
            mbar_init(&p_empty[b], 1);
        }
        mbar_init(o_full, 1);
        mbar_init(o_empty, 4);
        mbar_init(&mma_done[0], 1);
        mbar_init(&mma_done[1], 1);
        mbar_fence_init();
        flag[0] = 0;
        flag[1] = 0;
        flag[2] = 0;
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tO = tmem + TPS * RPU;   // S slot t at columns [t RPU, (t + 1) RPU), O after
    // the unit list comes from the unit pass, launched just before this grid
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const long long wl = p.wait_limit;

    if (warp == 6) {
        // ================= scheduler: units -> descriptors, query rows, block ids =================
        const int U = *reinterpret_cast<volatile const int32_t *>(p.unit_ctl + 1);
        int u_next = U;   // the next unit's index, fetched one unit ahead
        if (lane == 0 && !flag[0])
            u_next = atomicAdd(p.unit_ctl, 1);
        for (int uidx = 0;; ++uidx) {
            const int ub = uidx % NU;
            bool ok = true;
            if (uidx >= NU && lane == 0)
                ok = mbar_wait_bounded(&u_empty[ub], ((uidx / NU) + 1) & 1, wl);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            int u = __shfl_sync(0xffffffffu, u_next, 0);
            if (lane == 0 && ok && u < U && !flag[0])
                u_next = atomicAdd(p.unit_ctl, 1);
            if (!ok && lane == 0) {
                atomicOr(p.status, PKV_DEV_TIMEOUT);
                flag[0] = 1;
            }
            if (u >= U || !ok) {
                if (lane == 0) {
                    udesc[ub].valid = 0;
                    mbar_arrive(&u_full[ub]);
                }
                break;
            }
            const int4 e = __ldcg(p.units + u);
            const int s = e.x, split = e.y, g = e.z, rgi = e.w;
            int L, W, row0;
            if (GATHER) {
                L = __ldg(p.key_counts + s);
                L = L < 0 ? 0 : (L > p.max_keys ? p.max_keys : L);
                W = 1;
                row0 = s;
            } else {
                L = __ldg(p.context_lens + s);
                const int L_cap = (int)min((long long)p.max_context_len, (long long)p.max_blocks_per_seq * BS);
                L = L < 0 ? 0 : (L > L_cap ? L_cap : L);
                row0 = __ldg(p.q_starts + s);
                W = min(__ldg(p.q_starts + s + 1) - row0, p.max_rows);
            }
            const int r_lo = rgi * RPU;
            const int m_rows = min(p.group * W - r_lo, RPU);
            const int t0 = split * C, t1 = min(t0 + C, L);
            const int ntile = (t1 - t0 + kTileKeys - 1) / kTileKeys;
            const int blk0 = t0 / BS;
            const int nblk = (t1 - t0 + BS - 1) / BS;
            if constexpr (!GATHER) {
                // the split's block ids (loads first, checks after)
                int my = 0, my2 = 0;
                if (lane < nblk)
                    my = __ldg(p.block_tables + (size_t)s * p.max_blocks_per_seq + blk0 + lane);
                if (NBS > 32 && lane + 32 < nblk)
                    my2 = __ldg(p.block_tables + (size_t)s * p.max_blocks_per_seq + blk0 + lane + 32);
                if (lane < nblk && (my < 0 || my >= p.num_blocks)) {
                    atomicOr(p.status, PKV_DEV_BAD_BLOCK);
                    my = 0;
                }
                if (NBS > 32 && lane + 32 < nblk && (my2 < 0 || my2 >= p.num_blocks)) {
                    atomicOr(p.status, PKV_DEV_BAD_BLOCK);
                    my2 = 0;
                }
                if (lane < NBS)
                    blk_s[ub * NBS + lane] = lane < nblk ? my : -1;
                if (NBS > 32 && lane + 32 < NBS)
                    blk_s[ub * NBS + lane + 32] = lane + 32 < nblk ? my2 : -1;
            } else {
                // resolve the slice's list entries: all list loads, then all table loads
                constexpr int EPL = C / 32;
                const long long ctx_cap = (long long)p.max_blocks_per_seq * p.block_size;
                int seq = 0;
                {
                    int lo = 0, hi = p.num_seqs - 1;
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (__ldg(p.q_starts + mid) <= s)
                            lo = mid;
                        else
                            hi = mid - 1;
                    }
                    seq = lo;
                }
                long long ctx = __ldg(p.context_lens + seq);
                ctx = ctx < 0 ? 0 : (ctx > ctx_cap ? ctx_cap : ctx);
                const int32_t *lst = p.key_idx + (size_t)s * p.max_keys;
                int pos[EPL], blk[EPL];
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    const int en = t0 + j * 32 + lane;
                    pos[j] = en < t1 ? __ldg(lst + en) : -1;
                }
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    const bool in = pos[j] >= 0 && pos[j] < ctx;
                    blk[j] = in ? __ldg(p.block_tables + (size_t)seq * p.max_blocks_per_seq + pos[j] / p.block_size)
                                : -1;
                }
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    const int i = j * 32 + lane;
                    if (t0 + i >= t1)
                        break;
                    unsigned long long off = kGatherBad;
                    if (pos[j] >= 0 && pos[j] < ctx) {
                        if (blk[j] >= 0 && blk[j] < p.num_blocks)
                            off = ((((unsigned long long)blk[j] * p.num_kv_heads) + g) * p.block_size +
                                   pos[j] % p.block_size) * D;
                        else
                            atomicOr(p.status, PKV_DEV_BAD_BLOCK);
                    } else {
                        atomicOr(p.status, PKV_DEV_TABLE_OVERRUN);
                    }
                    g_off[ub * C + i] = off;
                }
            }
            // per-column key limits (and tree masks) and output rows of this unit
            for (int n = lane; n < RPU; n += 32) {
                int lim = 0, orow = 0;
                uint32_t tm = 0u;
                if (n < m_rows) {
                    const int r = r_lo + n, w = r / p.group;
                    lim = p.causal ? L - W + w + 1 : L;
                    if (TREE)
                        tm = __ldg(p.tree_masks + row0 + w);
                    orow = (row0 + w) * p.num_q_heads + hmap_s[g * p.group + (r - w * p.group)];
                }
                lim_s[ub * RPU + n] = lim;
                tmk_s[ub * RPU + n] = tm;
                orow_s[ub * RPU + n] = orow;
            }
            if (lane == 0) {
                UnitDesc &d = udesc[ub];
                d.valid = 1;
                d.s = s;
                d.g = g;
                d.split = split;
                d.L = L;
                d.W = W;
                d.row0 = row0;
                d.m_rows = m_rows;
                d.t0 = t0;
                d.ntile = ntile;
                d.n_mma = (m_rows + 15) / 16 * 16;
            }
            // query rows -> shared memory, 128-byte swizzled K-major rows (64 dims per row)
            bool okq = true;
            if (uidx >= NU && lane == 0)
                okq = mbar_wait_bounded(&q_empty[ub], ((uidx / NU) + 1) & 1, wl);
            okq = __shfl_sync(0xffffffffu, okq, 0);
            if (!okq) {
                if (lane == 0) {
                    atomicOr(p.status, PKV_DEV_TIMEOUT);
                    flag[0] = 1;
                    udesc[ub].valid = 0;
                    mbar_arrive(&u_full[ub]);
                }
                break;
            }
            {
                constexpr int CH = D / 8;   // 16-byte chunks per row
                constexpr int PER = (RPU * CH + 31) / 32;
                uint8_t *qb = qbuf + ub * Y::kQBuf;
                __syncwarp();   // orow_s of this unit is written
                uint4 v[PER];
#pragma unroll
                for (int k = 0; k < PER; ++k) {   // every load first, then every store
                    const int idx = lane + 32 * k;
                    if (idx < m_rows * CH) {
                        const int n = idx / CH, ch = idx - n * CH;
                        v[k] = __ldg(reinterpret_cast<const uint4 *>(p.q + (size_t)orow_s[ub * RPU + n] * D) + ch);
                    }
                }
#pragma unroll
                for (int k = 0; k < PER; ++k) {
                    const int idx = lane + 32 * k;
                    if (idx < m_rows * CH) {
                        const int n = idx / CH, ch = idx - n * CH;
                        const int half = ch >> 3, c8 = ch & 7;
                        *reinterpret_cast<uint4 *>(qb + half * RPU * 128 + n * 128 + ((c8 ^ (n & 7)) << 4)) = v[k];
                    }
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&q_full[ub]);
                    mbar_arrive(&u_full[ub]);
                }
            }
        }
    } else if (warp == 0 || warp == 1) {
        // ================= K side (warp 0) / V side (warp 1): tile loads and MMA products =================
        const bool is_k = warp == 0;
        const int NR = is_k ? NK : NV;
        uint8_t *ring = is_k ? kring : vring;
        uint64_t *full = is_k ? k_full : v_full;
        uint64_t *empty = is_k ? k_empty : v_empty;
        const CUtensorMap *map = is_k ? &tm_k : &tm_v;
        const uint16_t *pool = is_k ? p.kpool : p.vpool;
        if (!GATHER && lane == 0)
            prefetch_tensormap(map);
        bool aborted = false;
        // descriptor of unit uidx (the warp waits for its slot, lane 0 testing the barrier)
        auto load_unit = [&](TileCursor &c, int uidx) {
            c.uidx = uidx;
            c.t = 0;
            bool ok = true;
            if (lane == 0)
                ok = mbar_wait_bounded(&u_full[uidx % NU], (uidx / NU) & 1, wl);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok)
                aborted = true;
            c.d = udesc[uidx % NU];
            c.valid = ok && c.d.valid;
        };
        TileCursor ld, mm;   // the load cursor runs ahead of the product cursor
        load_unit(ld, 0);
        mm = ld;
        // The load cursor waits at the end of a unit (t = -1) until the next unit's slot is
        // within NU - 1 units of the product cursor and its descriptor is written; it never
        // blocks there, so the products go on meanwhile.
        auto try_advance_ld = [&]() {
            const int nxt = ld.uidx + 1;
            if (nxt > mm.uidx + NU - 1)
                return;
            bool ready = false;
            if (lane == 0)
                ready = mbar_test_wait(&u_full[nxt % NU], (nxt / NU) & 1);
            if (__shfl_sync(0xffffffffu, ready, 0))
                load_unit(ld, nxt);
        };
        int issued = 0, done = 0;   // tiles loaded / multiplied
        int scnt[TPS];              // (K side) uses of each S slot so far
#pragma unroll
        for (int t = 0; t < TPS; ++t)
            scnt[t] = 0;
        int pc = 0;                 // (V side) weight tiles consumed
        while (!aborted && mm.valid) {
            if (!ld.valid && ld.t == -1)
                try_advance_ld();
            // 1) loads, up to the ring depth ahead
            while (!aborted && ld.valid && issued < done + NR) {
                const int st = issued % NR;
                bool okw = true;
                if (issued >= NR && lane == 0)
                    okw = mbar_wait_bounded(&empty[st], ((issued / NR) + 1) & 1, wl);
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (!okw || flag[0]) {
                    aborted = true;
                    break;
                }
                const int ub = ld.uidx % NU;
                uint8_t *tile = ring + st * Y::kKvTile;
                if constexpr (GATHER) {
                    constexpr int CH = D / 8;
                    const int t1 = min(ld.d.t0 + C, ld.d.L);
                    for (int idx = lane; idx < kTileKeys * CH; idx += 32) {
                        const int key = idx / CH, ch = idx - key * CH;
                        const int en = ld.t * kTileKeys + key;
                        if (ld.d.t0 + en < t1) {
                            const unsigned long long o = g_off[ub * C + en];
                            const bool vld = o != kGatherBad;
                            const uint32_t so = (ch >> 3) * (kTileKeys * 128) + key * 128 + (((ch & 7) ^ (key & 7)) << 4);
                            cp_async_16(tile + so, pool + (vld ? o : 0ull) + ch * 8, vld ? 16u : 0u);
                        }
                    }
                    cp_async_arrive(&full[st]);
                } else if (lane == 0) {
                    int ids[BPT];
                    uint32_t bytes = 0;
#pragma unroll
                    for (int b = 0; b < BPT; ++b) {
                        ids[b] = blk_s[ub * NBS + ld.t * BPT + b];
                        bytes += ids[b] >= 0 ? BS * D * 2 : 0;
                    }
                    mbar_arrive_expect_tx(&full[st], bytes);
#pragma unroll
                    for (int b = 0; b < BPT; ++b) {
                        if (ids[b] < 0)
                            continue;
                        const int y = (ids[b] * p.num_kv_heads + ld.d.g) * BS;
#pragma unroll
                        for (int h = 0; h < Y::kHalves; ++h)
                            tma_load_2d(tile + h * (kTileKeys * 128) + b * BS * 128, map, &full[st], h * 64, y);
                    }
                }
                ++issued;
                if (++ld.t == ld.d.ntile) {
                    ld.valid = false;
                    ld.t = -1;
                    try_advance_ld();
                }
            }
            if (aborted)
                break;
            // 2) the product of the current tile
            const int ub = mm.uidx % NU;
            if (lane == 0) {
                bool ok = true;
                if (is_k) {
                    // S_t^T = K_t q^T into S slot t, once the softmax warps have read the slot
                    const int st = done % NK, t = mm.t;
                    ok = (t > 0 || mbar_wait_bounded(&q_full[ub], (mm.uidx / NU) & 1, wl)) &&
                         mbar_wait_bounded(&k_full[st], (done / NK) & 1, wl) &&
                         (scnt[t] == 0 || mbar_wait_bounded(&s_empty[t], (scnt[t] - 1) & 1, wl));
                    if (ok) {
                        ++scnt[t];
                        tc::fence_after_sync();
                        // A = K: keys on M (K-major, 8-row atoms 1 KB apart), dims on K; B = q: rows
                        // on N, dims on K.  A k-step moves the start address (the low field).
                        const uint64_t a0 = tc::smem_desc_sw128(smem_addr(kring + st * Y::kKvTile), 16, 1024);
                        const uint64_t b0 = tc::smem_desc_sw128(smem_addr(qbuf + ub * Y::kQBuf), 16, 1024);
                        const uint32_t idesc = tc::idesc_bf16_f32(128, mm.d.n_mma, 0, 0);
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks)
                            tc::mma_bf16(tS + t * RPU, a0 + (uint64_t)(((ks >> 2) * (kTileKeys * 128) + (ks & 3) * 32) >> 4),
                                         b0 + (uint64_t)(((ks >> 2) * RPU * 128 + (ks & 3) * 32) >> 4), idesc, ks > 0);
                        tc::mma_commit(&s_full[t]);
                        tc::mma_commit(&k_empty[st]);
                        if (t == mm.d.ntile - 1)
                            tc::mma_commit(&q_empty[ub]);
                    }
                } else {
                    // O^T (+)= V_t^T P_t^T once the softmax warps have written P_t (and read
                    // the unit before's O)
                    const int b = pc % NPB, st = done % NV, t = mm.t;
                    ok = (t > 0 || mm.uidx == 0 || mbar_wait_bounded(o_empty, (mm.uidx - 1) & 1, wl)) &&
                         mbar_wait_bounded(&p_full[b], (pc / NPB) & 1, wl) &&
                         mbar_wait_bounded(&v_full[st], (done / NV) & 1, wl);
                    if (ok) {
                        tc::fence_after_sync();
                        // A = V^T: head dims on M (MN-major, 64-dim blocks 16 KB apart; at D 64 the
                        // second block repeats the first and its rows are not read), keys on K.
                        // B = P: rows on N, keys on K (K-major, two 64-key halves).
                        const uint64_t a0 = tc::smem_desc_sw128(smem_addr(vring + st * Y::kKvTile),
                                                                D == 128 ? kTileKeys * 128 : 0, 1024);
                        const uint64_t b0 = tc::smem_desc_sw128(smem_addr(pbuf + b * Y::kPBuf), 16, 1024);
                        const uint32_t idesc = tc::idesc_bf16_f32(128, mm.d.n_mma, 1, 0);
#pragma unroll
                        for (int kk = 0; kk < kTileKeys / 16; ++kk)
                            tc::mma_bf16(tO, a0 + (uint64_t)((kk * 2048) >> 4),
                                         b0 + (uint64_t)(((kk >> 2) * RPU * 128 + (kk & 3) * 32) >> 4), idesc,
                                         (t > 0 || kk > 0) ? 1u : 0u);
                        tc::mma_commit(&p_empty[b]);
                        tc::mma_commit(&v_empty[st]);
                        if (t == mm.d.ntile - 1)
                            tc::mma_commit(o_full);
                    }
                }
                if (!ok)
                    flag[0] = 1;
            }
            __syncwarp();
            if (flag[0]) {
                aborted = true;
                break;
            }
            ++done;
            if (!is_k)
                ++pc;
            if (++mm.t == mm.d.ntile) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&u_empty[ub]);
                load_unit(mm, mm.uidx + 1);
            }
        }
        if (aborted && lane == 0) {
            atomicOr(p.status, PKV_DEV_TIMEOUT);
            flag[0] = 1;
        }
        if (lane == 0) {
            flag[is_k ? 1 : 2] = issued;
            // every MMA this thread issued has completed before the tensor memory is released
            tc::mma_commit(&mma_done[is_k ? 0 : 1]);
            mbar_wait_bounded(&mma_done[is_k ? 0 : 1], 0, kWaitLimitCycles);
        }
        __syncwarp();
    } else {
        // ================= softmax warps =================
        // A failed wait makes the warp skip its work up to the next barrier; the barriers
        // OR the failures over the four warps, so they all leave at the same point.
        const int quarter = warp & 3;            // tensor-memory lane quarter of this warp
        const int kl = 32 * quarter + lane;      // key of the tile (S) / head dim (O) of this thread
        const int wg_t = (warp - 2) * 32 + lane; // 0..127 within the softmax warps
        const bool o_lane = kl < D;
        int scnt[TPS];                           // completions of each S slot seen
#pragma unroll
        for (int t = 0; t < TPS; ++t)
            scnt[t] = 0;
        int pc = 0, vc = 0;
        bool bad = false;                        // a wait of this warp gave up
        auto give_up = [&]() {
            if (!bad && lane == 0) {
                atomicOr(p.status, PKV_DEV_TIMEOUT);
                flag[0] = 1;
            }
            bad = true;
        };
        for (int uidx = 0;; ++uidx) {
            const int ub = uidx % NU;
            if (!mbar_wait_bounded(&u_full[ub], (uidx / NU) & 1, wl))
                give_up();
            if (softmax_bar_any(bad))
                break;
            const UnitDesc d = udesc[ub];
            if (!d.valid)
                break;
            const int nch = (d.m_rows + 15) >> 4;
            const int32_t *lim = lim_s + ub * RPU;
            const uint32_t *tmk = tmk_s + ub * RPU;
            const int win0 = d.L - d.W;   // (tree) window keys start here
            // visibility of this thread's key in tile t to chunk c's columns
            auto vis_of = [&](int t, int c) -> uint32_t {
                const int kp = d.t0 + t * kTileKeys + kl;
                uint32_t v = 0u;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int4 l4 = *reinterpret_cast<const int4 *>(lim + c * 16 + 4 * q4);
                    uint32_t v4 = (uint32_t)(kp < l4.x) | ((uint32_t)(kp < l4.y) << 1) | ((uint32_t)(kp < l4.z) << 2) |
                                  ((uint32_t)(kp < l4.w) << 3);
                    if (TREE && kp >= win0) {
                        const uint4 m4 = *reinterpret_cast<const uint4 *>(tmk + c * 16 + 4 * q4);
                        const int sh = kp - win0 < 32 ? kp - win0 : 31;
                        v4 &= ((m4.x >> sh) & 1u) | (((m4.y >> sh) & 1u) << 1) | (((m4.z >> sh) & 1u) << 2) |
                              (((m4.w >> sh) & 1u) << 3);
                    }
                    v |= v4 << (4 * q4);
                }
                return v;
            };
            // ---- pass 1: every tile's scaled, masked scores -> each row's maximum ----
            // (the thread's own maximum over the split's tiles first, then one reduction)
            float xmax[NCH][16];
#pragma unroll
            for (int c = 0; c < NCH; ++c)
#pragma unroll
                for (int n = 0; n < 16; ++n)
                    xmax[c][n] = -INFINITY;
            uint32_t vbk[KEEP ? TPS : 1];   // (one chunk: each tile's visibility bits, kept for pass 2)
            if constexpr (KEEP) {
                // one chunk: wait for every tile's scores, load them all, one wait
                uint32_t (&vb)[KEEP ? TPS : 1] = vbk;
#pragma unroll
                for (int t = 0; t < TPS; ++t)
                    vb[t] = t < d.ntile ? vis_of(t, 0) : 0u;
#pragma unroll
                for (int t = 0; t < TPS; ++t) {
                    if (t >= d.ntile)
                        break;
                    if (!bad && !mbar_wait_bounded(&s_full[t], scnt[t] & 1, wl))
                        give_up();
                    ++scnt[t];
                }
                if (!bad) {
                    tc::fence_after_sync();
                    uint32_t r[TPS][16];
#pragma unroll
                    for (int t = 0; t < TPS; ++t)
                        if (t < d.ntile)
                            tc::tmem_ld16(tmem_at(tS + t * RPU, quarter, 0), r[t]);
                    tc::tmem_wait(r);
#pragma unroll
                    for (int t = 0; t < TPS; ++t)
#pragma unroll
                        for (int n = 0; n < 16; ++n) {
                            const float x = (t < d.ntile && ((vb[t] >> n) & 1u)) ? __uint_as_float(r[t][n]) * p.scale_log2
                                                                               : -INFINITY;
                            xmax[0][n] = fmaxf(xmax[0][n], x);
                        }
                }
            } else {
#pragma unroll
            for (int t = 0; t < TPS; ++t) {
                if (t >= d.ntile)
                    break;
                uint32_t vb[NCH];
#pragma unroll
                for (int c = 0; c < NCH; ++c)
                    vb[c] = c < nch ? vis_of(t, c) : 0u;
                if (!bad && !mbar_wait_bounded(&s_full[t], scnt[t] & 1, wl))
                    give_up();
                ++scnt[t];
                if (bad)
                    continue;
                tc::fence_after_sync();
                uint32_t rn[16];
                tc::tmem_ld16(tmem_at(tS + t * RPU, quarter, 0), rn);
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    if (c >= nch)
                        break;
                    uint32_t r[16];
                    tc::tmem_wait(rn);
#pragma unroll
                    for (int n = 0; n < 16; ++n)
                        r[n] = rn[n];
                    if (c + 1 < nch)
                        tc::tmem_ld16(tmem_at(tS + t * RPU, quarter, (c + 1) * 16), rn);
#pragma unroll
                    for (int n = 0; n < 16; ++n) {
                        const float x = ((vb[c] >> n) & 1u) ? __uint_as_float(r[n]) * p.scale_log2 : -INFINITY;
                        xmax[c][n] = fmaxf(xmax[c][n], x);
                    }
                }
            }
            }
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                if (c >= nch)
                    break;
                const float mx = reduce_scatter16<true>(xmax[c], lane);
                if (!(lane & 1))
                    red[(c * 16 + rs_col(lane)) * 4 + quarter] = mx;
            }
            if (softmax_bar_any(bad))
                break;
            if (wg_t < d.n_mma) {   // one thread per MMA column: the four warps' maxima
                const float4 r4 = *reinterpret_cast<const float4 *>(red + wg_t * 4);
                mbuf[wg_t] = fmaxf(fmaxf(r4.x, r4.y), fmaxf(r4.z, r4.w));
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            // ---- pass 2: weights 2^(x - m) in bf16 -> P (row n, key kl); partial sums ----
            float l_part[NCH][16];
#pragma unroll
            for (int c = 0; c < NCH; ++c)
#pragma unroll
                for (int n = 0; n < 16; ++n)
                    l_part[c][n] = 0.f;
            const int kc8 = (kl & 63) >> 3, kb2 = (kl & 7) * 2;
            if constexpr (KEEP) {
                // one chunk, a weight buffer per tile: every tile's weights, then the signals
                static_assert(!KEEP || NPB >= TPS, "decode keeps a weight buffer per tile");
#pragma unroll
                for (int t = 0; t < TPS; ++t) {
                    if (t >= d.ntile)
                        break;
                    const int b = (pc + t) % NPB;
                    if (!bad && pc + t >= NPB && !mbar_wait_bounded(&p_empty[b], (((pc + t) / NPB) + 1) & 1, wl))
                        give_up();
                }
                float mb[16];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(mbuf + 4 * q4);
                    mb[4 * q4] = m4.x == -INFINITY ? 0.f : m4.x, mb[4 * q4 + 1] = m4.y == -INFINITY ? 0.f : m4.y;
                    mb[4 * q4 + 2] = m4.z == -INFINITY ? 0.f : m4.z, mb[4 * q4 + 3] = m4.w == -INFINITY ? 0.f : m4.w;
                }
                if (!bad) {
                    // the scores again (every tile at once, one wait)
                    uint32_t r[TPS][16];
#pragma unroll
                    for (int t = 0; t < TPS; ++t)
                        if (t < d.ntile)
                            tc::tmem_ld16(tmem_at(tS + t * RPU, quarter, 0), r[t]);
                    tc::tmem_wait(r);
#pragma unroll
                    for (int t = 0; t < TPS; ++t) {
                        if (t >= d.ntile)
                            break;
                        uint8_t *pb = pbuf + ((pc + t) % NPB) * Y::kPBuf + (kl >> 6) * RPU * 128;
#pragma unroll
                        for (int n = 0; n < 16; ++n) {
                            const float x = ((vbk[t] >> n) & 1u) ? __uint_as_float(r[t][n]) * p.scale_log2 : -INFINITY;
                            const __nv_bfloat16 pw = __float2bfloat16_rn(fast_exp2(x - mb[n]));
                            *reinterpret_cast<__nv_bfloat16 *>(pb + n * 128 + ((kc8 ^ (n & 7)) << 4) + kb2) = pw;
                            l_part[0][n] += __bfloat162float(pw);
                        }
                    }
                }
                // every S slot is read and every tile but the last is ready: signal those first
                // (the last tile's V load may wait for the first tile's product)
                tc::fence_before_sync();
                tc::fence_proxy_async_smem();  // P -> the MMA's operand reads
                __syncwarp();
                if (lane == 0) {
#pragma unroll
                    for (int t = 0; t < TPS; ++t) {
                        if (t >= d.ntile)
                            break;
                        mbar_arrive(&s_empty[t]);
                        if (t < d.ntile - 1)
                            mbar_arrive(&p_full[(pc + t) % NPB]);
                    }
                }
                // V rows of keys past the unit's keys: zero (the last tile may hold anything there)
                {
                    const int t = d.ntile - 1;
                    const int kp = d.t0 + t * kTileKeys + kl;
                    if (!bad && d.t0 + (t + 1) * kTileKeys > d.L) {
                        const int st = (vc + t) % NV;
                        if (!mbar_wait_bounded(&v_full[st], ((vc + t) / NV) & 1, wl))
                            give_up();
                        else if (kp >= d.L) {
                            uint8_t *vrow = vring + st * Y::kKvTile + kl * 128;
#pragma unroll
                            for (int h = 0; h < Y::kHalves; ++h)
#pragma unroll
                                for (int q16 = 0; q16 < 8; ++q16)
                                    *reinterpret_cast<uint4 *>(vrow + h * (kTileKeys * 128) + q16 * 16) = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                tc::fence_proxy_async_smem();  // the zeroed V rows -> the MMA's operand reads
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&p_full[(pc + d.ntile - 1) % NPB]);
                pc += d.ntile;
                vc += d.ntile;
            } else {
#pragma unroll
            for (int t = 0; t < TPS; ++t) {
                if (t >= d.ntile)
                    break;
                const int b = pc % NPB;
                if (!bad && pc >= NPB && !mbar_wait_bounded(&p_empty[b], ((pc / NPB) + 1) & 1, wl))
                    give_up();
                uint8_t *pb = pbuf + b * Y::kPBuf + (kl >> 6) * RPU * 128;
                uint32_t rn[16];
                if (!bad)
                    tc::tmem_ld16(tmem_at(tS + t * RPU, quarter, 0), rn);
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    if (c >= nch || bad)
                        break;
                    float x[16];
                    {
                        uint32_t r[16];
                        tc::tmem_wait(rn);
#pragma unroll
                        for (int n = 0; n < 16; ++n)
                            r[n] = rn[n];
                        if (c + 1 < nch)
                            tc::tmem_ld16(tmem_at(tS + t * RPU, quarter, (c + 1) * 16), rn);
                        const uint32_t vb = vis_of(t, c);
#pragma unroll
                        for (int n = 0; n < 16; ++n)
                            x[n] = ((vb >> n) & 1u) ? __uint_as_float(r[n]) * p.scale_log2 : -INFINITY;
                    }
                    float mb[16];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const float4 m4 = *reinterpret_cast<const float4 *>(mbuf + c * 16 + 4 * q4);
                        mb[4 * q4] = m4.x, mb[4 * q4 + 1] = m4.y, mb[4 * q4 + 2] = m4.z, mb[4 * q4 + 3] = m4.w;
                    }
#pragma unroll
                    for (int n = 0; n < 16; ++n) {
                        const int col = c * 16 + n;
                        const float base = mb[n] == -INFINITY ? 0.f : mb[n];
                        const __nv_bfloat16 pw = __float2bfloat16_rn(fast_exp2(x[n] - base));
                        *reinterpret_cast<__nv_bfloat16 *>(pb + col * 128 + ((kc8 ^ (col & 7)) << 4) + kb2) = pw;
                        l_part[c][n] += __bfloat162float(pw);
                    }
                }
                // S slot t is read: the QK issuer may reuse it
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&s_empty[t]);
                // V rows of keys past the unit's keys: zero (the tile may hold anything there)
                const int kp = d.t0 + t * kTileKeys + kl;
                if (!bad && d.t0 + (t + 1) * kTileKeys > d.L) {
                    const int st = vc % NV;
                    if (!mbar_wait_bounded(&v_full[st], (vc / NV) & 1, wl))
                        give_up();
                    else if (kp >= d.L) {
                        uint8_t *vrow = vring + st * Y::kKvTile + kl * 128;
#pragma unroll
                        for (int h = 0; h < Y::kHalves; ++h)
#pragma unroll
                            for (int q16 = 0; q16 < 8; ++q16)
                                *reinterpret_cast<uint4 *>(vrow + h * (kTileKeys * 128) + q16 * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                tc::fence_proxy_async_smem();  // P and the zeroed V rows -> the MMA's operand reads
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&p_full[b]);
                ++pc;
                ++vc;
            }
            }
            // ---- the unit's partial: O from tensor memory, l = sum over the key lanes, m ----
            if (!bad && !mbar_wait_bounded(o_full, uidx & 1, wl))
                give_up();
            const int32_t *orow = orow_s + ub * RPU;
            if (!bad && o_lane) {
                tc::fence_after_sync();
                uint32_t rn[16];
                tc::tmem_ld16(tmem_at(tO, quarter, 0), rn);
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    if (c >= nch)
                        break;
                    uint32_t r[16];
                    tc::tmem_wait(rn);
#pragma unroll
                    for (int n = 0; n < 16; ++n)
                        r[n] = rn[n];
                    if (c + 1 < nch)
                        tc::tmem_ld16(tmem_at(tO, quarter, (c + 1) * 16), rn);
#pragma unroll
                    for (int n = 0; n < 16; ++n) {
                        const int col = c * 16 + n;
                        if (col < d.m_rows)
                            __stcg(p.part_o + ((size_t)orow[col] * p.n_max + d.split) * D + kl, __uint_as_float(r[n]));
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(o_empty);
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                if (c >= nch)
                    break;
                const float sm = reduce_scatter16<false>(l_part[c], lane);
                if (!(lane & 1))
                    red[(c * 16 + rs_col(lane)) * 4 + quarter] = sm;
            }
            if (softmax_bar_any(bad))
                break;
            if (wg_t < d.m_rows) {
                const float4 r4 = *reinterpret_cast<const float4 *>(red + wg_t * 4);
                const float l = ((r4.x + r4.y) + r4.z) + r4.w;   // warp quarters 0, 1, 2, 3 in order
                p.part_ml[(size_t)orow[wg_t] * p.n_max + d.split] = make_float2(mbuf[wg_t], l);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");   // red and mbuf are read: free for the next unit
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&u_empty[ub]);
        }
    }

    // leave: every copy issued into the rings has landed, every MMA has completed
    tc::fence_before_sync();
    __syncthreads();
    if (flag[0] && threadIdx.x == 0) {
        for (int r = 0; r < 2; ++r) {
            const int NR = r == 0 ? NK : NV;
            uint64_t *full = r == 0 ? k_full : v_full;
            const int issued = flag[1 + r];
            for (int st = 0; st < NR && st < issued; ++st) {
                const int k_last = st + ((issued - 1 - st) / NR) * NR;
                if (!mbar_wait_bounded(&full[st], (k_last / NR) & 1, kWaitLimitCycles))
                    break;
            }
        }
    }
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side --
template <int D, int BS, int RPU, int NK, int NV, bool TREE, bool GATHER>
int launch_tc_t(const CUtensorMap &mk, const CUtensorMap &mv, const AttnParams &prm, const UnitPassParams &up,
                cudaStream_t st)
{
    const size_t smem_up = unit_pass_smem(up.num_src, up.n_max);
    int rc = check_cuda(cudaFuncSetAttribute(attention_unit_pass, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem_up),
                        "cudaFuncSetAttribute(unit pass)");
    if (rc)
        return rc;
    attention_unit_pass<<<1, 1024, smem_up, st>>>(up);
    rc = check_cuda(cudaGetLastError(), "paged attention unit pass launch");
    if (rc)
        return rc;
    auto kern = paged_attention_tc_kernel<D, BS, RPU, NK, NV, TREE, GATHER>;
    constexpr size_t smem = tc_smem_bytes<D, BS, RPU, NK, NV, TREE, GATHER>();
    static_assert(smem <= 232448, "shared memory of the tensor-core attention kernel");
    rc = check_cuda(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                    "cudaFuncSetAttribute(tensor-core attention)");
    if (rc)
        return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sm_count());
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    rc = check_cuda(cudaLaunchKernelEx(&cfg, kern, mk, mv, prm), "paged attention (tensor cores) launch");
    if (rc)
        return rc;
    const long long units = (long long)prm.total_rows * prm.num_q_heads;
    cudaLaunchConfig_t mc = {};
    mc.gridDim = dim3((unsigned)((units + 1) / 2));
    mc.blockDim = dim3(128);
    mc.stream = st;
    mc.attrs = attr;
    mc.numAttrs = 1;
    return check_cuda(cudaLaunchKernelEx(&mc, paged_attention_combine_kernel<D>, prm), "paged attention merge launch");
}

// Ring depths (K tiles, V tiles): a tile is 128 keys (32 KB at head_dim 128, 16 KB at 64);
// the rings fill what shared memory the query and weight buffers leave (a V tile stays
// until its PV product, a K tile only until its QK product, so V gets the extra stage).
template <int D, int RPU, bool GATHER>
constexpr int kTcKStages = D == 128 ? (RPU == 16 ? (GATHER ? 2 : 3) : 2) : (RPU == 16 ? (GATHER ? 5 : 6) : 5);
template <int D, int RPU, bool GATHER>
constexpr int kTcVStages = D == 128 ? (RPU == 16 ? 3 : 2) : (RPU == 16 ? 6 : 5);

template <int D, int BS, bool GATHER>
int launch_tc(int rows_per_pair, const CUtensorMap &mk, const CUtensorMap &mv, AttnParams prm,
              UnitPassParams up, cudaStream_t st)
{
    const bool tree = prm.tree_masks != nullptr;
    if (rows_per_pair <= 16) {
        up.rpu = 16;
        if (tree)
            return launch_tc_t<D, BS, 16, kTcKStages<D, 16, false>, kTcVStages<D, 16, false>, true, false>(mk, mv, prm, up, st);
        return launch_tc_t<D, BS, 16, kTcKStages<D, 16, GATHER>, kTcVStages<D, 16, GATHER>, false, GATHER>(mk, mv, prm, up, st);
    }
    up.rpu = 64;
    if (tree)
        return launch_tc_t<D, BS, 64, kTcKStages<D, 64, false>, kTcVStages<D, 64, false>, true, false>(mk, mv, prm, up, st);
    return launch_tc_t<D, BS, 64, kTcKStages<D, 64, GATHER>, kTcVStages<D, 64, GATHER>, false, GATHER>(mk, mv, prm, up, st);
}

}  // namespace
}  // namespace pkv
