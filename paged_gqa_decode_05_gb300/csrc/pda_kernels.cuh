// pda_kernels.cuh -- split-KV paged GQA decode kernels for sm_103a.
//
// Split kernel (one persistent CTA per resident slot; grid = SMs x CTAs/SM):
//   * the warp after the consumers is the producer: it walks the CTA's share of the
//     flattened (sequence, kv head, block) space (pda_plan.h), looks every
//     block up in the block table and copies whole K/V block rows of one kv
//     head into a ring of shared-memory stages with one 5-D TMA tensor copy
//     per block and pool (128-byte swizzle; rows gathered for block sizes
//     below 8), plus the group's q rows with one bulk copy at the start of
//     each segment.  Stage completion is tracked by mbarriers.
//   * ST/16 consumer warps read a stage of ST rows (64; 32 for head_dim 256
//     with block sizes below 8), 16 rows each.  The GQA group
//     (G <= 8 q heads of one kv head) shares every K/V load: S^T = K q^T is a
//     16x8 tile per warp (mma.sync m16n8k16, tokens as M, heads as N), the
//     online-softmax update runs on the accumulator fragments (warp-shuffle
//     max over tokens), P is transposed in registers (movmatrix) and
//     O^T += V^T P^T accumulates over D in 16-row slabs.
//   * causal multi-query with more than 8 q rows per sequence (head sizes up
//     to 128) takes the row form instead (run_consumer_rows): the packed q
//     rows are the MMA's M (S = Q K^T, O += P V), one KV walk serving up to
//     32 of them.  A tcgen05 version of it at head size 128 (run_mma_tc /
//     run_consumer_tc: tensor-memory accumulators, one MMA-issuing thread) is
//     switched on per context.
//   * a last, optional warp prefetches the CTA's first stages into L2 before
//     the kernel's dependency wait, while the previous kernel finishes
//     (prefetch_first_stages), and exits.
//   * at the end of a segment the consumer warps' states are merged in shared
//     memory; a segment that covers its whole unit writes bf16 o / l
//     directly (or folds its state into the running state, in tiled steps).
//     The pieces of a unit split across CTAs draw tickets: all but the last
//     store an fp32 partial (m, l, o) state and signal it; the last merges
//     them with its own and writes o / l (or folds).  One launch per call.
//
// Method sources: tiled_attention.rs (spark_storage) for the (m, l, o) state,
// its reset values and o / l finalize; AstrAI "CUDA Kernels" (Overview:
// split-KV paged decode with MMA) for splitting the KV walk.  Scores are kept
// in base-2 units (scale * log2 e folded in), an exact rewrite of exp().
#pragma once

#include "pda_params.h"
#include "pda_ptx.cuh"

namespace pda {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // each mbarrier wait gives up after 2 s
// How far (base-2 units) a q row's softmax reference may lag its running max
// before o is rescaled: the reference m of a row moves only when a stage's max
// exceeds it by more than this, so the weights p = 2^(s - m) stay below 2^8
// (well inside fp32 and the bf16 hi + lo split of P), and (m, l, o), which
// means the same for any reference, is rescaled a few times per segment
// instead of whenever a max grows.
constexpr float kLazyLog2 = 8.f;
#define kNegInf (-__int_as_float(0x7f800000))

#define PDA_DEVERR_BAD_BLOCK_ID_ 0x1u
#define PDA_DEVERR_BAD_LENGTH_ 0x2u
#define PDA_DEVERR_TIMEOUT_ 0x4u

// Pipeline depth per head size (tuning constants).
#ifndef PDA_STAGES_D64
#define PDA_STAGES_D64 6
#endif
#ifndef PDA_STAGES_D128
#define PDA_STAGES_D128 3
#endif
#ifndef PDA_STAGES_D256
#define PDA_STAGES_D256 3
#endif
// 32-row stages (head_dim 256, block sizes below 8).
#ifndef PDA_STAGES_D256_ST32
#define PDA_STAGES_D256_ST32 3
#endif

// Register cap of the split kernel (see split_kernel).  An SM's registers
// are four 16K quarters, one per scheduler, and a warp takes its registers
// from its scheduler's quarter: with 9 or 10 warps per SM (one CTA of 9 warps,
// or two of 5) a quarter holds 3 warps, at most 168 registers per thread.
constexpr int split_max_regs(int D, int mode) { return D == 256 && q_tiles(mode) == 0 ? 255 : 168; }

// Row form of multi-query (q rows as the MMA's M): one q tile runs two CTAs
// per SM like plain decode; two q tiles (8 consumer warps) run one CTA per
// SM with a deeper ring.
#ifndef PDA_STAGES_ROWS16_D64
#define PDA_STAGES_ROWS16_D64 5
#endif
#ifndef PDA_STAGES_ROWS16_D128
#define PDA_STAGES_ROWS16_D128 3
#endif
#ifndef PDA_STAGES_ROWS32_D64
#define PDA_STAGES_ROWS32_D64 10
#endif
#ifndef PDA_STAGES_ROWS32_D128
#define PDA_STAGES_ROWS32_D128 5
#endif
// tcgen05 form (head size 128): one CTA per SM (a kernel with tcgen05
// instructions gets one CTA per SM), five 40 KB stages.
#ifndef PDA_STAGES_TC_D128
#define PDA_STAGES_TC_D128 5
#endif

// Split-kernel shape: head size D, ST KV rows per stage, MODE (the row form
// of multi-query has its own warp count and q area).
template <int D, int ST, int MODE>
struct Cfg {
    static constexpr int kST = ST;                       // KV rows per stage (64 or 32)
    static constexpr int kLogST = ST == 64 ? 6 : 5;
    static constexpr int kQTiles = q_tiles(MODE);        // 16-row q tiles (0: n8 form)
    static constexpr int kConsumerWarps = consumer_warps(ST, MODE);  // 16 KV rows each (per q tile)
    static constexpr bool kTc = is_tc(MODE);
    // + the producer warp (warp kConsumerWarps) and the tcgen05 form's MMA warp
    static constexpr int kMainThreads = (kConsumerWarps + 1 + (kTc ? 1 : 0)) * 32;
    static constexpr int kThreads = kMainThreads + 32;              // + the prefetch warp
    static constexpr int kHalves = D / 64;               // 64-column swizzled slabs per row
    static constexpr int kHalfBytes = ST * 128;          // ST rows of one slab
    static constexpr int kTileBytes = kHalves * kHalfBytes;
    static constexpr int kStageBytes = 2 * kTileBytes + stage_q_rows(MODE) * D * 2;
    static constexpr int kStages = kTc ? PDA_STAGES_TC_D128
                                 : kQTiles == 1 ? (D == 64 ? PDA_STAGES_ROWS16_D64 : PDA_STAGES_ROWS16_D128)
                                 : kQTiles == 2 ? (D == 64 ? PDA_STAGES_ROWS32_D64 : PDA_STAGES_ROWS32_D128)
                                 : D == 64 ? PDA_STAGES_D64
                                 : D == 128 ? PDA_STAGES_D128
                                 : ST == 32 ? PDA_STAGES_D256_ST32 : PDA_STAGES_D256;
    static constexpr int kKSteps = D / 16;
    static_assert(ST == 64 || ST == 32, "stage rows");
    static_assert(kQTiles == 0 || (ST == 64 && D <= 128), "row form: 64-row stages, head size <= 128");
    // tcgen05 form: tensor-memory columns (two S buffers, O^T, Q)
    static constexpr uint32_t kTmemCols = 256u;
    static_assert(!kTc || D == 128, "tcgen05 form: head size 128");
};

// Causal multi-query decode packs qp queries of a sequence into one launch
// row (the MMA's N = qp*G columns: column n is query n / G, head n % G).  A
// sequence has Qr = ceil(q_len / qp) rows, ordered row-major over the batch:
// launch sequence s is row s / Bs of sequence s % Bs (Bs = B / Qr), which
// makes each row index one group of the split plan.  Plain decode (MQ false,
// every mode but kMulti): Qr = 1 and row s is sequence s, fixed at compile
// time so the single-query kernels carry none of the packing arithmetic.
struct RowInfo {
    int b;      // sequence (table row, lens index)
    int first;  // first query of the row
    int cnt;    // queries in the row
};

template <bool MQ>
__device__ __forceinline__ int rows_per_seq(const SplitParams& p) {
    if constexpr (!MQ) return 1;
    else return (p.q_len + p.qp - 1) / p.qp;
}

template <bool MQ>
__device__ __forceinline__ RowInfo row_info(const SplitParams& p, int s) {
    RowInfo r;
    if constexpr (!MQ) { r.b = s; r.first = 0; r.cnt = 1; return r; }
    const int Bs = p.B / rows_per_seq<MQ>(p);
    r.b = s % Bs;
    r.first = (s / Bs) * p.qp;
    r.cnt = min(p.qp, p.q_len - r.first);
    return r;
}

// Element offset of q/out row (query qi of sequence b, q head h).
template <bool MQ>
__device__ __forceinline__ int64_t qo_offset(const SplitParams& p, int b, int qi, int h, int D) {
    const int ql = MQ ? p.q_len : 1;
    return (((int64_t)b * ql + qi) * p.Hq + h) * D;
}

// The length entry of launch sequence s (tokens; blocks in tiled steps).
template <bool MQ>
__device__ __forceinline__ int32_t len_entry(const SplitParams& p, int s) {
    return p.lens[row_info<MQ>(p, s).b];
}

// Tokens read for launch sequence s with length entry L: L itself, or for a
// row of causal queries the prefix its last query sees, L - q_len + first +
// cnt (>= 0).
template <bool MQ>
__device__ __forceinline__ int32_t tokens_of(const SplitParams& p, int s, int32_t L) {
    if constexpr (!MQ) return L;
    const RowInfo r = row_info<MQ>(p, s);
    const int32_t len = L - p.q_len + r.first + r.cnt;
    return len < 0 ? 0 : len;
}

// Blocks of sequence b with length entry L, validated and clamped (flags
// bad lengths, unless FLAG is false: a speculative read).
template <bool MQ, bool FLAG = true>
__device__ __forceinline__ int32_t blocks_of(const SplitParams& p, int b, int32_t L) {
    int32_t len = p.lens_are_blocks ? L : tokens_of<MQ>(p, b, L);
    if (p.lens_are_blocks) {
        if (len < 0 || len > p.table_stride) {
            if (FLAG) atomicOr(p.err, PDA_DEVERR_BAD_LENGTH_);
            len = len < 0 ? 0 : p.table_stride;
        }
        return len;
    }
    if (len < 0) {
        if (FLAG) atomicOr(p.err, PDA_DEVERR_BAD_LENGTH_);
        len = 0;
    }
    int32_t nb = blocks_for_tokens(len, p.bs);
    if (nb > p.table_stride) {
        if (FLAG) atomicOr(p.err, PDA_DEVERR_BAD_LENGTH_);
        nb = p.table_stride;
    }
    return nb;
}

// The entry the valid-slot count of sequence b's last block comes from: its
// length entry, or in tiled steps its last_valid entry (bs when none given).
// Loaded apart from its use so that the load's latency overlaps other loads.
template <bool MQ>
__device__ __forceinline__ int32_t last_entry(const SplitParams& p, int b) {
    if (p.lens_are_blocks) return p.last_valid ? p.last_valid[b] : p.bs;
    return len_entry<MQ>(p, b);
}

// Valid slots of sequence b's last block (1..bs) from its last_entry e.
template <bool MQ>
__device__ __forceinline__ int32_t last_block_slots(const SplitParams& p, int b, int32_t nb, int32_t e) {
    if (p.lens_are_blocks) {
        if (e < 1 || e > p.bs) {
            atomicOr(p.err, PDA_DEVERR_BAD_LENGTH_);
            e = e < 1 ? 1 : p.bs;
        }
        return e;
    }
    const int32_t v = tokens_of<MQ>(p, b, e) - (nb - 1) * p.bs;
    return v > p.bs ? p.bs : v;
}

// Exclusive prefix of plan blocks per sequence (blocks plus the unit cost)
// into shared pfx[0..B] (B <= 1024); returns the largest plan-block count of
// a sequence.
// Thread t owns sequences [t*per, t*per + per): it loads all their length
// entries at once (one memory round trip), stores their plan blocks in pfx,
// and the per-thread sums are scanned with warp shuffles and the warp totals.
// Run by the kThreads threads of the consumer and producer warps (threads
// 0 .. kThreads-1), synchronised by named barrier 1; ends with that barrier
// (which also publishes the stage barriers).
template <bool MQ, int kThreads>
__device__ __forceinline__ int32_t build_prefix(const SplitParams& p, int32_t* pfx, int32_t* scan) {
    constexpr int kPer = (kMaxLaunchBatch + kThreads - 1) / kThreads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (p.B + kThreads - 1) / kThreads;  // <= kPer
    const int lo = min(p.B, tid * per), hi = min(p.B, lo + per);
    int32_t L[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) L[k] = lo + k < hi ? len_entry<MQ>(p, lo + k) : 0;
    int32_t sum = 0, big = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k)
        if (lo + k < hi) {
            const int32_t v = plan_blocks(blocks_of<MQ>(p, lo + k, L[k]), p.unit_cost);
            pfx[lo + k] = v;
            sum += v;
            big = max(big, v);
        }
    int32_t x = sum;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
        big = max(big, __shfl_xor_sync(0xffffffffu, big, o));
    }
    if (lane == 31) {
        scan[warp] = x;
        scan[16 + warp] = big;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
    int32_t run = x - sum;
    for (int w = 0; w < warp; ++w) run += scan[w];
    for (int w = 0; w < kThreads / 32; ++w) big = max(big, scan[16 + w]);
    if (tid == kThreads - 1) pfx[p.B] = run + sum;
#pragma unroll
    for (int k = 0; k < kPer; ++k)
        if (lo + k < hi) {
            const int32_t v = pfx[lo + k];
            pfx[lo + k] = run;
            run += v;
        }
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
    return big;
}

// ------------------------------------------------------------------ producer

template <int D, int ST, int MODE>
__device__ __forceinline__ void run_producer(const SplitParams& p, uint32_t base_s, const SmemLayout& L,
                                             const int32_t* pfx, StageMeta* meta,
                                             volatile int* abort_flag, int64_t begin, int64_t end,
                                             int lane) {
    // The whole warp walks the plan in lockstep; lane 0 issues the barrier
    // operations, the lanes issue the copies.  Block ids come from registers,
    // loaded well before they are used so that table reads do not stall the
    // copies: w[0..3] hold the 128-entry window [win, win + 128) of the
    // current table row (lane i of w[k]: entry win + 32k + i), f[] the first
    // 128 entries of the current sequence's row (the next kv head starts
    // there) and nx[] those of the next non-empty sequence, loaded one unit
    // ahead together with the entry its last block's valid slots come from.
    using C = Cfg<D, ST, MODE>;
    constexpr int S = C::kStages;
    constexpr bool MQ = is_multi(MODE);
    const uint32_t full0 = base_s + L.bars, empty0 = full0 + 8 * S;
    const bool leader = lane == 0;
    // K/V are read once: evict them first.  With several query rows per
    // sequence each block is read once per row at nearly the same time; keep
    // it normal.
    const uint64_t pol = rows_per_seq<MQ>(p) > 1 ? policy_evict_normal() : policy_evict_first();
    const int bs = p.bs, Hkv = p.Hkv;
    const int NB = C::kST / bs;  // blocks per stage (the host keeps bs <= ST)

    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_parity = 0;  // per-stage bits, for the drain after an abort
    bool ok = true;

    int64_t pos = begin;
    int b = 0, kvh = 0;
    int32_t j = 0, nb = 0, nv = 0;  // j: block of the unit; nb blocks, nv plan blocks
    int32_t win = 0;
    int32_t w[4], f[4], nx[4];
    int32_t lv = bs;   // valid slots of this sequence's last block
    int32_t nle = 0;   // the next sequence's last_entry, loaded a unit ahead
    int bn = p.B;               // next non-empty sequence
    // The launch rows of b and bn (multi-query: table row, first query, query
    // count) and b's causal limit, computed once per sequence, not per stage.
    RowInfo ri = row_info<MQ>(p, 0), rn = ri;
    int32_t lim = 0x7fffffff;
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = f[k] = nx[k] = 0;
    // entry idx of table row `row` (contiguous cache: block row * stride + idx)
    auto table_at = [&](int row, int32_t idx) -> int32_t {
        if (p.table == nullptr) return row * p.table_stride + idx;
        return p.table[(int64_t)row * p.table_stride + idx];
    };
    // entries [from, from + 128) of table row `row` (nbs blocks), lane-strided
    auto load_ids = [&](int32_t* dst, int row, int32_t from, int32_t nbs) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int32_t e = from + 32 * k + lane;
            dst[k] = e < nbs ? table_at(row, e) : 0;
        }
    };
    auto next_seq = [&](int s) {
        do { ++s; } while (s < p.B && pfx[s + 1] == pfx[s]);
        return s;
    };
    // The id of window entry idx (lane-varying).  A stage reads entries
    // j - win .. j - win + n - 1 < 64: the blocks per stage NB = ST / bs is a
    // power of two, j - win stays a multiple of NB (the window starts at a
    // segment start or a unit start and slides by 64) and n <= NB.  So only
    // w[0] and w[1] are read; w[2] and w[3], loaded at a slide, are first read
    // a whole window later, after the next slide has moved them down.
    auto win_id = [&](int idx) {
        const int32_t a = __shfl_sync(0xffffffffu, w[0], idx & 31);
        const int32_t c = __shfl_sync(0xffffffffu, w[1], idx & 31);
        return idx < 32 ? a : c;
    };
    if (pos < end) {
        int lo = 0, hi = p.B - 1;  // largest b with pfx[b]*Hkv <= pos
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)pfx[mid] * Hkv <= pos) lo = mid; else hi = mid - 1;
        }
        b = lo;
        nv = pfx[b + 1] - pfx[b];
        nb = real_blocks(nv, p.unit_cost);
        const int64_t rem = pos - (int64_t)pfx[b] * Hkv;
        kvh = (int)(rem / nv);
        j = (int32_t)(rem % nv);  // may lie in the unit's cost tail (j >= nb)
        win = j;
        // every load first (one round trip), their uses after
        bn = next_seq(b);
        ri = row_info<MQ>(p, b);
        rn = bn < p.B ? row_info<MQ>(p, bn) : ri;
        const int32_t e_cur = last_entry<MQ>(p, b);
        nle = bn < p.B ? last_entry<MQ>(p, bn) : 0;
        load_ids(w, ri.b, win, nb);
        if (win == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) f[k] = w[k];
        } else {
            load_ids(f, ri.b, 0, nb);
        }
        if (bn < p.B) load_ids(nx, rn.b, 0, real_blocks(pfx[bn + 1] - pfx[bn], p.unit_cost));
        lv = last_block_slots<MQ>(p, b, nb, e_cur);
        if constexpr (MQ) lim = e_cur - p.q_len + ri.first;
    }
    // Past a unit's last block: skip its cost tail and move to the next unit
    // (the next kv head reuses the row's first ids; the next sequence's ids
    // were loaded a unit ago).
    auto next_unit = [&]() {
        pos += nv - j;
        j = 0;
        win = 0;
        if (++kvh == Hkv) {
            kvh = 0;
            b = bn;
            nv = b < p.B ? pfx[b + 1] - pfx[b] : 0;
            nb = real_blocks(nv, p.unit_cost);
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = f[k] = nx[k];
            if (b < p.B && pos < end) {
                ri = rn;
                lv = last_block_slots<MQ>(p, b, nb, nle);
                if constexpr (MQ) lim = nle - p.q_len + ri.first;
                bn = next_seq(b);
                if (bn < p.B) {
                    rn = row_info<MQ>(p, bn);
                    nle = last_entry<MQ>(p, bn);
                    load_ids(nx, rn.b, 0, real_blocks(pfx[bn + 1] - pfx[bn], p.unit_cost));
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = f[k];
        }
    };
    bool seg_begin = true;
    bool whole = false;
    while (pos < end) {
        const int stop = __shfl_sync(0xffffffffu, leader ? *abort_flag : 0, 0);
        if (stop) { ok = false; break; }
        if (j >= nb) {  // the unit's last block is issued (or the range starts in its tail)
            if (b >= p.B) break;  // no units left (not reached: end <= the plan's size)
            next_unit();
            continue;
        }
        const int32_t n = (int32_t)min((int64_t)min(NB, nb - j), end - pos);
        const bool unit_end = (j + n == nb);
        const bool seg_end = unit_end || (pos + n == end);
        if (seg_begin)
            whole = (j == 0) && ((int64_t)pfx[b] * Hkv + (int64_t)kvh * nv + nb <= end);

        const int32_t lastv = unit_end ? lv : bs;

        bool got = true;
        if (leader) got = mbar_wait_bounded(empty0 + 8 * stage, phase ^ 1u, kWaitLimitNs);
        got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
        if (!got) { ok = false; break; }

        const uint32_t full = full0 + 8 * stage;
        const uint32_t sK = base_s + (uint32_t)stage * C::kStageBytes;
        const uint32_t sV = sK + C::kTileBytes;
        if (leader) {
            StageMeta m;
            m.b = b;
            m.kvh = kvh;
            m.n_valid = (n - 1) * bs + lastv;
            m.flags = (seg_begin ? kSegBegin : 0) | (seg_end ? kSegEnd : 0) | (whole ? kWholeUnit : 0);
            m.slot = b * Hkv + kvh + (int)blockIdx.x;
            m.j0 = j;
            m.lim = lim;
            m.nr = MQ ? ri.cnt * p.G : p.G;
            meta[stage] = m;
            const bool load_q = seg_begin && MODE != kGather;
            const int rows = (n - 1) * bs + lastv;
            const uint32_t kv_bytes =
                p.row_gather == 0 ? (uint32_t)n * 2u * (uint32_t)bs * D * 2u
                : p.row_gather == 1 ? (uint32_t)((rows + 3) >> 2) * 2u * 4u * D * 2u
                                    : 0u;  // cp.async completions arrive instead
            const uint32_t bytes = kv_bytes + (load_q ? (uint32_t)(m.nr * D * 2) : 0u);
            mbar_arrive_expect_tx(full, bytes);
            if (load_q) {  // the G q rows of kv head kvh for each packed query
                if constexpr (MQ) {
                    for (int k = 0; k < ri.cnt; ++k)
                        bulk_load(sV + C::kTileBytes + (uint32_t)(k * p.G * D * 2),
                                  p.q + qo_offset<MQ>(p, ri.b, ri.first + k, kvh * p.G, D),
                                  (uint32_t)(p.G * D * 2), full);
                } else {
                    bulk_load(sV + C::kTileBytes, p.q + qo_offset<MQ>(p, b, 0, kvh * p.G, D),
                              (uint32_t)(p.G * D * 2), full);
                }
            }
        }
        __syncwarp();
        if (p.row_gather == 1) {
            // Rows of small blocks, 4 per TMA gather4 copy of one 64-column slab:
            // group g covers stage rows 4g..4g+3 (the tail repeats the last row,
            // which the consumers mask), written as one ST-row block.
            constexpr int H = C::kHalves;
            const int lbs = 31 - __clz(bs);
            const int rows = (n - 1) * bs + lastv;
            const int groups = (rows + 3) >> 2;
            for (int o0 = 0; o0 < (C::kST / 4) * H; o0 += 32) {
                const int o = o0 + lane;
                const int g = o / H, h = o - g * H;
                int32_t r[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int t = min(4 * g + k, rows - 1);
                    const int i = t >> lbs;  // block of the stage (< ST)
                    int32_t id = win_id(j - win + i);
                    if (o < groups * H && (id < 0 || (int64_t)id >= p.num_blocks)) {
                        atomicOr(p.err, PDA_DEVERR_BAD_BLOCK_ID_);
                        id = 0;
                    }
                    r[k] = (int32_t)((int64_t)id * p.row_blk + (int64_t)(t & (bs - 1)) * p.row_tok +
                                     (int64_t)kvh * p.row_kvh);
                }
                if (o < groups * H) {
                    const uint32_t dst = (uint32_t)h * C::kHalfBytes + (uint32_t)(4 * g) * 128u;
                    tma_gather4(sK + dst, &p.tm_k, h * 64, r[0], r[1], r[2], r[3], full, pol);
                    tma_gather4(sV + dst, &p.tm_v, h * 64, r[0], r[1], r[2], r[3], full, pol);
                }
            }
        } else if (p.row_gather == 2) {
            // Rows of small blocks: 16-byte cp.async chunks, CH per row, written
            // in the layout of one ST-row block ([slab][row][128 B], swizzled).
            constexpr int CH = D / 8;
            constexpr int RPI = 32 / CH;  // rows per pass of the warp
            const int c = lane % CH, sub = lane / CH;
            const int lbs = 31 - __clz(bs);
            const int rows = (n - 1) * bs + lastv;
            const uint16_t* kb = p.k_base + (int64_t)kvh * p.kvh_s + c * 8;
            const uint16_t* vb = p.v_base + (int64_t)kvh * p.kvh_s + c * 8;
            for (int t0 = 0; t0 < rows; t0 += RPI) {
                const int t = t0 + sub;
                const int i = min(t, rows - 1) >> lbs;  // block of the stage (< ST)
                const int32_t wid = win_id(j - win + i);
                if (t < rows) {
                    int32_t id = wid;
                    if (id < 0 || (int64_t)id >= p.num_blocks) {
                        atomicOr(p.err, PDA_DEVERR_BAD_BLOCK_ID_);
                        id = 0;
                    }
                    const int64_t off = (int64_t)id * p.blk_s + (int64_t)(t & (bs - 1)) * p.tok_s;
                    const uint32_t dst = (uint32_t)(c >> 3) * C::kHalfBytes + (uint32_t)t * 128u +
                                         (uint32_t)(((c & 7) ^ (t & 7)) << 4);
                    cp_async_16(sK + dst, kb + off);
                    cp_async_16(sV + dst, vb + off);
                }
            }
            cp_async_mbar_arrive_noinc(full);
        } else
        // lane i copies block i of the stage (its id comes from the window)
        {
            const int32_t wid = win_id(j - win + min(lane, n - 1));
            if (lane < n) {
                int32_t id = wid;
                if (id < 0 || (int64_t)id >= p.num_blocks) {
                    atomicOr(p.err, PDA_DEVERR_BAD_BLOCK_ID_);
                    id = 0;  // stays in bounds; the flag marks the result invalid
                }
                if constexpr (is_tc(MODE) && D == 128) {
                    // one box per slab: the stage tile is [slab][64 rows][128 B]
                    const uint32_t off = (uint32_t)(lane * bs) * 128u;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        tma_load_5d(sK + off + (uint32_t)h * C::kHalfBytes, &p.tm_k1, 0, 0, h, kvh, id, full, pol);
                        tma_load_5d(sV + off + (uint32_t)h * C::kHalfBytes, &p.tm_v1, 0, 0, h, kvh, id, full, pol);
                    }
                } else {
                    const uint32_t off = (uint32_t)(lane * bs) * (uint32_t)(D * 2);
                    tma_load_5d(sK + off, &p.tm_k, 0, 0, 0, kvh, id, full, pol);
                    tma_load_5d(sV + off, &p.tm_v, 0, 0, 0, kvh, id, full, pol);
                }
            }
        }
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);

        pos += n;
        j += n;
        seg_begin = seg_end;
        if (!unit_end && j - win >= 64) {
            // first half consumed: slide by 64 and fetch the 64 entries after
            // the window (needed no sooner than the next stage)
            win += 64;
            w[0] = w[2];
            w[1] = w[3];
#pragma unroll
            for (int k = 2; k < 4; ++k) {
                const int32_t e = win + 32 * k + lane;
                w[k] = e < nb ? table_at(ri.b, e) : 0;
            }
        }
        if (++stage == S) { stage = 0; phase ^= 1u; }
    }
    if (!leader) return;
    if (ok) {
        if (mbar_wait_bounded(empty0 + 8 * stage, phase ^ 1u, kWaitLimitNs)) {
            meta[stage].flags = kDone;
            // every arrival the stage's barrier expects (33 for cp.async rows)
            mbar_arrive_count(full0 + 8 * stage, p.row_gather == 2 ? 33u : 1u);
        } else {
            ok = false;
        }
    }
    if (!ok) {
        atomicOr(p.err, PDA_DEVERR_TIMEOUT_);
        *abort_flag = 1;
        // Wait (bounded) for every copy this warp issued to land before the
        // CTA may exit.  A phase that already completed passes at once.
        for (int s = 0; s < S; ++s)
            if (issued & (1u << s))
                mbar_wait_bounded(full0 + 8 * s, (issued_parity >> s) & 1u, kWaitLimitNs);
    }
}

// ------------------------------------------------------------------ consumers

// Stage tiles hold the stage's blocks back to back; block i is one TMA box
// laid out [D/64 slabs][bs rows][128 bytes], 128-byte swizzled, so row t of
// the stage, slab h, 16-byte chunk c sits at
//   row_off(t) + h * bs * 128 + ((c ^ swz(t, h)) << 4)
// with row_off(t) = (t / bs) * bs * D * 2 + (t % bs) * 128.  The swizzle XORs
// the chunk with bits 7..9 of the shared-memory address; a box starts on a
// 1024-byte span, so those bits are (t % bs + h * bs) mod 8: t & 7 from block
// size 8 up, (t & (bs - 1)) ^ (h * bs & 7) for blocks of 2 or 4 rows.  Rows
// gathered one by one are laid out as one block of ST rows.
__device__ __forceinline__ int swz(int t, int h, int lbs) {
    return lbs >= 3 ? (t & 7) : (t & ((1 << lbs) - 1)) ^ ((h << lbs) & 7);
}

template <int D>
__device__ __forceinline__ uint32_t row_off(int t, int lbs) {
    const int bs = 1 << lbs;
    return (uint32_t)(t >> lbs) * (uint32_t)(bs * D * 2) + (uint32_t)(t & (bs - 1)) * 128u;
}

// Zeroes V rows [from, r0+16) of the warp's tile (masked rows may hold any
// bits, and 0 * NaN would poison the P.V product).
template <int D>
__device__ __forceinline__ void zero_rows(uint32_t sV, int from, int to, int lbs, int lane) {
    constexpr int kHalves = D / 64;
    const uint32_t hs = (uint32_t)(128 << lbs);
    const int units = (to - from) * kHalves * 8;
    for (int u = lane; u < units; u += 32) {
        const int r = from + u / (kHalves * 8);
        const int rem = u % (kHalves * 8);
        const uint32_t a = sV + row_off<D>(r, lbs) + (uint32_t)(rem >> 3) * hs + ((rem & 7) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
    }
}

template <int D>
__device__ __forceinline__ void gather_rows(const SplitParams& p, uint32_t base_s, const uint8_t* base,
                                            uint32_t sK, uint32_t sV, const StageMeta& m, int r0,
                                            int lbs, int lane) {
    constexpr int kHalves = D / 64;
    const uint32_t hs = (uint32_t)(128 << lbs);
    const int rows = min(16, m.n_valid - r0);
    if (rows <= 0) return;
    const int units = rows * kHalves * 8;
    const int64_t row0 = ((int64_t)m.b * p.Hkv + m.kvh) * p.dbg_row_tokens + (int64_t)m.j0 * p.bs + r0;
    for (int u = lane; u < units; u += 32) {
        const int r = u / (kHalves * 8);
        const int rem = u % (kHalves * 8);
        const int h = rem >> 3, c = rem & 7;
        const int rr = r0 + r;
        const uint32_t off = row_off<D>(rr, lbs) + (uint32_t)h * hs + (uint32_t)((c ^ swz(rr, h, lbs)) << 4);
        const uint4 kv = *reinterpret_cast<const uint4*>(base + (sK - base_s) + off);
        const uint4 vv = *reinterpret_cast<const uint4*>(base + (sV - base_s) + off);
        const int64_t dst = (row0 + r) * D + h * 64 + c * 8;
        *reinterpret_cast<uint4*>(p.dbg_k + dst) = kv;
        *reinterpret_cast<uint4*>(p.dbg_v + dst) = vv;
    }
}

// Barrier among the 128 consumer threads (an mbarrier, so the wait is
// bounded: a warp that gave up cannot leave the others waiting forever).
__device__ __forceinline__ bool consumer_sync(uint32_t cbar, uint32_t& cphase, uint32_t* err,
                                              volatile int* abort_flag) {
    mbar_arrive(cbar);
    const bool ok = mbar_wait_bounded(cbar, cphase, kWaitLimitNs);
    cphase ^= 1u;
    if (!ok) {
        atomicOr(err, PDA_DEVERR_TIMEOUT_);
        *abort_flag = 1;
    }
    return ok;
}

// Combines a partial state (mi, li, oi) into (M, Ls, Os).
__device__ __forceinline__ void merge_state(float& M, float& Ls, float4& Os, float mi, float li,
                                            const float4& oi) {
    const float Mn = fmaxf(M, mi);
    if (Mn == kNegInf) return;  // both states empty
    const float fa = ex2(M - Mn), fb = ex2(mi - Mn);
    Ls = Ls * fa + li * fb;
    Os.x = Os.x * fa + oi.x * fb;
    Os.y = Os.y * fa + oi.y * fb;
    Os.z = Os.z * fa + oi.z * fb;
    Os.w = Os.w * fa + oi.w * fb;
    M = Mn;
}

// Segment-end roles (see the epilogue in run_consumer).
enum SegRole : int32_t { kRoleWhole = 0, kRoleStore = 1, kRoleMerge = 2, kRoleAbort = -1 };

template <int D, int ST, int MODE>
__device__ __forceinline__ void run_consumer(const SplitParams& p, uint32_t base_s, uint8_t* base,
                                             const SmemLayout& L, const StageMeta* meta,
                                             const int32_t* pfx, const GroupRange& gr,
                                             volatile int* abort_flag, int warp, int lane) {
    using C = Cfg<D, ST, MODE>;
    constexpr int S = C::kStages;
    constexpr int KS = C::kKSteps;
    const uint32_t full0 = base_s + L.bars, empty0 = full0 + 8 * S;
    const int g = lane >> 2, t = lane & 3;
    const int r0 = warp * 16;
    constexpr bool MQ = MODE == kMulti;
    static_assert(C::kQTiles == 0, "n8 form");
    const int G = p.G;
    const float sl2 = p.scale_log2;
    // multi-query: the queries of this lane's two score columns (column n is
    // query n / G of the row), fixed for the whole launch
    const int qc0 = MQ ? (2 * t) / G : 0, qc1 = MQ ? (2 * t + 1) / G : 0;
    // ldmatrix row addresses: QK reads K as the A operand (rows = tokens),
    // PV reads V transposed as the A operand (rows of V = tokens = k index).
    const int qk_row = r0 + (lane & 7) + (((lane >> 3) & 1) << 3);
    const int qk_cpar = lane >> 4;
    const int pv_row = r0 + (lane & 7) + ((lane >> 4) << 3);
    const int pv_cpar = (lane >> 3) & 1;
    const int lbs = p.row_gather ? C::kLogST : 31 - __clz(p.bs);  // gathered rows: one ST-row block
    // swizzle of this lane's ldmatrix rows in slab h, swz(row, h) (both patterns
    // have row & 7 == lane & 7), fixed for the launch
    int swh[C::kHalves];
#pragma unroll
    for (int h = 0; h < C::kHalves; ++h) swh[h] = swz(lane, h, lbs);
    const uint32_t hs = (uint32_t)(128 << lbs);  // bytes between 64-column slabs of a block
    const uint32_t qk_off = row_off<D>(qk_row, lbs);
    const uint32_t pv_off = row_off<D>(pv_row, lbs);

    float o[KS][4];
    uint32_t qf[KS][2];
    float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int i = 0; i < KS; ++i) {
        o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        qf[i][0] = qf[i][1] = 0u;
    }

    const uint32_t cbar = base_s + L.cbar;
    uint32_t cphase = 0;
    int stage = 0;
    uint32_t phase = 0;
    int32_t ticket = 0;  // consumer thread 0: this piece's ticket for its split unit
    // an early tile step waits for the previous kernel before its first segment end
    bool waited = !(MODE == kTiled && p.early_inputs != 0);

    if constexpr (writes_output(MODE)) {
        // A unit with no tokens has no segment: its output rows are zero.  Such
        // units are shared round-robin over the grid; the stores overlap the
        // wait for the first stage.
        const int ct = warp * 32 + lane;
        for (int u = blockIdx.x; u < p.B * p.Hkv; u += gridDim.x) {
            const int sq = u / p.Hkv, kvh = u - sq * p.Hkv;
            if (pfx[sq + 1] != pfx[sq]) continue;
            const RowInfo ri = row_info<MQ>(p, sq);
            const int NR = ri.cnt * G;
            for (int i4 = ct; i4 < NR * D / 4; i4 += C::kConsumerWarps * 32) {
                const int h = (4 * i4) / D, d4 = 4 * i4 - h * D;
                const int64_t o = MQ ? qo_offset<MQ>(p, ri.b, ri.first + h / G, kvh * G + h % G, D) + d4
                                     : qo_offset<MQ>(p, sq, 0, kvh * G, D) + 4 * i4;
                if (p.out_f32) *reinterpret_cast<float4*>(p.out_f32 + o) = make_float4(0.f, 0.f, 0.f, 0.f);
                else *reinterpret_cast<uint2*>(p.out + o) = make_uint2(0u, 0u);
            }
        }
    }

    while (true) {
        if (*abort_flag) break;
        if (!mbar_wait_bounded(full0 + 8 * stage, phase, kWaitLimitNs)) {
            atomicOr(p.err, PDA_DEVERR_TIMEOUT_);
            *abort_flag = 1;
            break;
        }
        const StageMeta m = meta[stage];
        if (m.flags & kDone) break;
        if (!waited && (m.flags & kSegEnd)) {  // the tickets, slots and running state come next
            pdl_wait_primary();
            waited = true;
        }
        // The last stage of a piece of a split unit: take the piece's ticket now, so
        // that the atomic's round trip overlaps this stage's math.  Tickets only
        // assign roles: the piece that draws the last one merges all pieces.
        if (MODE != kGather && warp == 0 && lane == 0 && (m.flags & kSegEnd) && !(m.flags & kWholeUnit))
            ticket = atomicAdd(p.unit_sync + 2 * (m.b * p.Hkv + m.kvh), 1);
        const uint32_t sK = base_s + (uint32_t)stage * C::kStageBytes;
        const uint32_t sV = sK + C::kTileBytes;

        if constexpr (MODE == kGather) {
            gather_rows<D>(p, base_s, base, sK, sV, m, r0, lbs, lane);
        } else {
            if (m.flags & kSegBegin) {
                m0 = m1 = kNegInf;
                l0 = l1 = 0.f;
                const uint8_t* sq = base + (sV - base_s) + C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    o[kk][0] = o[kk][1] = o[kk][2] = o[kk][3] = 0.f;
                    if (g < (MQ ? m.nr : G)) {
                        const uint8_t* r = sq + (size_t)(g * D + 16 * kk + 2 * t) * 2;
                        qf[kk][0] = *reinterpret_cast<const uint32_t*>(r);
                        qf[kk][1] = *reinterpret_cast<const uint32_t*>(r + 16);
                    } else {
                        qf[kk][0] = qf[kk][1] = 0u;
                    }
                }
            }
            if (r0 < m.n_valid) {
                const bool partial = r0 + 16 > m.n_valid;
                if (partial) {
                    zero_rows<D>(sV, m.n_valid, r0 + 16, lbs, lane);
                    __syncwarp();
                }
                // S^T (16 tokens x 8 heads) = K q^T in two independent chains
                // (more chains shorten the MMA dependency but cost adds to combine;
                // fewer instructions measured faster)
                float acc[2][4];
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) acc[ch][0] = acc[ch][1] = acc[ch][2] = acc[ch][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    uint32_t a[4];
                    const int cc = (((kk & 3) << 1) + qk_cpar) ^ swh[kk >> 2];
                    ldsm_x4(sK + qk_off + (uint32_t)(kk >> 2) * hs + (cc << 4), a);
                    mma_16816(acc[kk & 1], a, qf[kk][0], qf[kk][1]);
                }
                float s0 = (acc[0][0] + acc[1][0]) * sl2;
                float s1 = (acc[0][1] + acc[1][1]) * sl2;
                float s2 = (acc[0][2] + acc[1][2]) * sl2;
                float s3 = (acc[0][3] + acc[1][3]) * sl2;
                if (m.n_valid < C::kST) {  // a stage that ends mid-way: mask the rows past it
                    if (r0 + g >= m.n_valid) { s0 = kNegInf; s1 = kNegInf; }
                    if (r0 + g + 8 >= m.n_valid) { s2 = kNegInf; s3 = kNegInf; }
                }
                if constexpr (MQ) {  // column n = query n / G may not see the later tokens
                    const int pos0 = m.j0 * p.bs + r0;  // the warp's first token
                    if (pos0 + 15 > m.lim) {  // only rows past the row's first query's limit
                        const int pos = pos0 + g;
                        const int lim0 = m.lim + qc0, lim1 = m.lim + qc1;
                        if (pos > lim0) s0 = kNegInf;
                        if (pos > lim1) s1 = kNegInf;
                        if (pos + 8 > lim0) s2 = kNegInf;
                        if (pos + 8 > lim1) s3 = kNegInf;
                    }
                }
                // column max over the 16 tokens (lanes sharing t)
                float x0 = fmaxf(s0, s2), x1 = fmaxf(s1, s3);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
                    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
                }
                // lazy reference (kLazyLog2): o is rescaled only when a column's max
                // runs more than 2^8 past its reference
                const bool up0 = x0 > m0 + kLazyLog2, up1 = x1 > m1 + kLazyLog2;
                if (__any_sync(0xffffffffu, up0 || up1)) {
                    const float a0 = up0 ? ex2(m0 - x0) : 1.f;  // an empty column (m = -inf): 0
                    const float a1 = up1 ? ex2(m1 - x1) : 1.f;
                    if (up0) m0 = x0;
                    if (up1) m1 = x1;
                    l0 *= a0;
                    l1 *= a1;
#pragma unroll
                    for (int i = 0; i < KS; ++i) {
                        o[i][0] *= a0; o[i][1] *= a1; o[i][2] *= a0; o[i][3] *= a1;
                    }
                }
                const float u0 = m0 == kNegInf ? 0.f : m0;
                const float u1 = m1 == kNegInf ? 0.f : m1;
                // P enters the tensor core as bf16 hi + lo parts (p = hi + lo to
                // about 2^-17 relative), so P.V keeps fp32-level accuracy whatever
                // running maximum the weights were taken against.
                const float p0 = ex2(s0 - u0), p1 = ex2(s1 - u1);
                const float p2 = ex2(s2 - u0), p3 = ex2(s3 - u1);
                const uint32_t px = pack_bf16x2(p0, p1), py = pack_bf16x2(p2, p3);
                const uint32_t qx = pack_bf16x2(p0 - bf16_lo(px), p1 - bf16_hi(px));
                const uint32_t qy = pack_bf16x2(p2 - bf16_lo(py), p3 - bf16_hi(py));
                // l sums the fp32 weights; the ones that multiply V (hi + lo)
                // equal them to about 2^-17 relative
                l0 += p0 + p2;
                l1 += p1 + p3;
                const uint32_t pb0 = movmatrix_trans(px), pb1 = movmatrix_trans(py);
                const uint32_t pc0 = movmatrix_trans(qx), pc1 = movmatrix_trans(qy);
                // O^T (D x 8 heads) += V^T P^T, 16 rows of D per mma
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    uint32_t a[4];
                    const int cc = (((mt & 3) << 1) + pv_cpar) ^ swh[mt >> 2];
                    ldsm_x4_trans(sV + pv_off + (uint32_t)(mt >> 2) * hs + (cc << 4), a);
                    mma_16816(o[mt], a, pb0, pb1);
                    mma_16816(o[mt], a, pc0, pc1);
                }
                if (partial) fence_proxy_async_smem();  // generic writes before the next TMA
            }
        }
        if (MODE != kGather && (m.flags & kSegEnd)) {
            // ---- segment end.  The consumer warps' states merge through this
            // stage's own K/V memory (the stage is released only afterwards).
            // Then, by role:
            //   whole unit (the unit lies in this CTA): write o / l, or fold the
            //     state into the running state (tiled steps);
            //   piece of a split unit that did not draw the last ticket: store
            //     the partial (m, l, o) in slot u + blockIdx.x and signal it with
            //     a release increment of the unit's stored count;
            //   piece that drew the last ticket: wait (bounded) until the other
            //     pieces' partials are stored, merge them with its own state,
            //     write o / l (or fold), and zero the unit's counters for the
            //     next launch.
            // The last-ticket piece only waits for pieces that have already
            // drawn their tickets, i.e. are running towards their own store, so
            // the wait cannot deadlock whichever CTAs are resident.
            float* st_m = reinterpret_cast<float*>(base + L.st_m);
            float* st_l = reinterpret_cast<float*>(base + L.st_l);
            float* st_x = reinterpret_cast<float*>(base + L.st_x);  // old running m [8], l [8]
            int32_t* st_role = reinterpret_cast<int32_t*>(st_x + 2 * kMaxGroup);
            float* st_o = reinterpret_cast<float*>(base + (sK - base_s));
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, off);
                l1 += __shfl_xor_sync(0xffffffffu, l1, off);
            }
            if (!consumer_sync(cbar, cphase, p.err, abort_flag)) break;  // all reads of the stage done
            const int h0 = 2 * t, h1 = 2 * t + 1;
            const int NR = MQ ? m.nr : G;  // q rows of the unit
            if (g == 0) {
                if (h0 < NR) { st_m[warp * kMaxGroup + h0] = m0; st_l[warp * kMaxGroup + h0] = l0; }
                if (h1 < NR) { st_m[warp * kMaxGroup + h1] = m1; st_l[warp * kMaxGroup + h1] = l1; }
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const int d = 16 * mt + g;
                if (h0 < NR) {
                    float* r = st_o + (size_t)(warp * NR + h0) * (D + 4);
                    r[d] = o[mt][0];
                    r[d + 8] = o[mt][2];
                }
                if (h1 < NR) {
                    float* r = st_o + (size_t)(warp * NR + h1) * (D + 4);
                    r[d] = o[mt][1];
                    r[d + 8] = o[mt][3];
                }
            }
            const bool whole = (m.flags & kWholeUnit) != 0;
            const int u = m.b * p.Hkv + m.kvh;
            UnitPieces pc;
            pc.cf = 0; pc.su = 0; pc.n = 1; pc.every = true;
            if (!whole) pc = unit_pieces(pfx, m.b, m.kvh, p.Hkv, p.unit_cost, gr);
            const int ct = warp * 32 + lane;
            if constexpr (MODE == kTiled) {
                // the running state's (m, l) of the unit's rows, read before any is rewritten
                if (ct < NR) {
                    const int64_t row = (int64_t)m.b * p.Hq + (int64_t)m.kvh * G + ct;
                    st_x[ct] = p.m_state[row];
                    st_x[kMaxGroup + ct] = p.l_state[row];
                }
            }
            if (ct == 0) {
                int32_t role = whole ? kRoleWhole : ticket == pc.n - 1 ? kRoleMerge : kRoleStore;
                if (role == kRoleMerge) {
                    int32_t* cnt = p.unit_sync + 2 * u;
                    bool ready = ld_acquire_gpu(cnt + 1) == pc.n - 1;
                    if (!ready) {
                        const uint64_t t0 = global_ns();
                        while (!(ready = ld_acquire_gpu(cnt + 1) == pc.n - 1) && global_ns() - t0 <= kWaitLimitNs) {
                        }
                    }
                    if (ready) {
                        cnt[0] = 0;  // every piece has drawn and stored: reset for the next launch
                        cnt[1] = 0;
                    } else {
                        atomicOr(p.err, PDA_DEVERR_TIMEOUT_);
                        *abort_flag = 1;
                        role = kRoleAbort;
                    }
                }
                *st_role = role;
            }
            if (!consumer_sync(cbar, cphase, p.err, abort_flag)) break;
            const int role = *st_role;
            if (role == kRoleAbort) break;
            const RowInfo ri = row_info<MQ>(p, m.b);
            const int SR = MQ ? p.rows_per_slot : G;  // rows per partial slot
            for (int i4 = ct; i4 < NR * D / 4; i4 += C::kConsumerWarps * 32) {
                const int h = (4 * i4) / D, d4 = 4 * i4 - h * D;  // h: q row of the unit
                float M = kNegInf;
#pragma unroll
                for (int w = 0; w < C::kConsumerWarps; ++w) M = fmaxf(M, st_m[w * kMaxGroup + h]);
                float Ls = 0.f;
                float4 Os = make_float4(0.f, 0.f, 0.f, 0.f);
                if (M != kNegInf) {
#pragma unroll
                    for (int w = 0; w < C::kConsumerWarps; ++w) {
                        const float f = ex2(st_m[w * kMaxGroup + h] - M);
                        const float4 v = *reinterpret_cast<const float4*>(st_o + (size_t)(w * NR + h) * (D + 4) + d4);
                        Ls += st_l[w * kMaxGroup + h] * f;
                        Os.x += v.x * f; Os.y += v.y * f; Os.z += v.z * f; Os.w += v.w * f;
                    }
                }
                if (role == kRoleStore) {
                    const int64_t r = (int64_t)(u + (int)blockIdx.x) * SR + h;
                    *reinterpret_cast<float4*>(p.part_o + r * D + d4) = Os;
                    if (d4 == 0) {
                        p.part_ml[r * 2] = M;
                        p.part_ml[r * 2 + 1] = Ls;
                    }
                    continue;
                }
                if (role == kRoleMerge) {
                    // every piece in piece order (this piece's own state in its
                    // place), so the result does not depend on which piece
                    // finished last; the others' partials are loaded up to eight
                    // per memory round trip
                    float Mr = kNegInf, Lr = 0.f;
                    float4 Or = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int i0 = 0; i0 < pc.n; i0 += 8) {
                        float mi[8], li[8];
                        float4 oi[8];
                        bool own[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            mi[k] = kNegInf;
                            li[k] = 0.f;
                            oi[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                            const int64_t c = piece_cta(pc, i0 + k, gr);
                            own[k] = i0 + k < pc.n && c == (int64_t)blockIdx.x;
                            if (i0 + k >= pc.n || own[k]) continue;
                            const int64_t r = (u + c) * SR + h;
                            mi[k] = ld_cg(p.part_ml + r * 2);
                            li[k] = ld_cg(p.part_ml + r * 2 + 1);
                            oi[k] = __ldcg(reinterpret_cast<const float4*>(p.part_o + r * D + d4));
                        }
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            if (own[k]) merge_state(Mr, Lr, Or, M, Ls, Os);
                            else merge_state(Mr, Lr, Or, mi[k], li[k], oi[k]);
                        }
                    }
                    M = Mr;
                    Ls = Lr;
                    Os = Or;
                }
                if constexpr (MODE == kTiled) {
                    // fold into the running state (plain decode rows: b*Hq + kvh*G + h)
                    const int64_t row = (int64_t)m.b * p.Hq + (int64_t)m.kvh * G + h;
                    float Mo = st_x[h], Lo = st_x[kMaxGroup + h];
                    float4* so = reinterpret_cast<float4*>(p.o_state + row * D + d4);
                    float4 Oo = *so;
                    merge_state(Mo, Lo, Oo, M, Ls, Os);
                    *so = Oo;
                    if (d4 == 0) {
                        p.m_state[row] = Mo;
                        p.l_state[row] = Lo;
                    }
                } else {
                    const float4 v = Ls > 0.f ? make_float4(Os.x / Ls, Os.y / Ls, Os.z / Ls, Os.w / Ls)
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
                    const int64_t o = MQ ? qo_offset<MQ>(p, ri.b, ri.first + h / G, m.kvh * G + h % G, D) + d4
                                         : qo_offset<MQ>(p, m.b, 0, m.kvh * G, D) + 4 * i4;
                    if (p.out_f32) {
                        *reinterpret_cast<float4*>(p.out_f32 + o) = v;
                    } else {
                        uint2 w2;
                        w2.x = pack_bf16x2(v.x, v.y);
                        w2.y = pack_bf16x2(v.z, v.w);
                        *reinterpret_cast<uint2*>(p.out + o) = w2;
                    }
                }
            }
            if (!consumer_sync(cbar, cphase, p.err, abort_flag)) break;
            // a stored piece signals after every consumer thread's stores (ordered
            // before this thread's release by the consumer barrier)
            if (role == kRoleStore && ct == 0) red_release_gpu_add(p.unit_sync + 2 * u + 1, 1);
            fence_proxy_async_smem();  // staging writes before the next TMA into this stage
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);
        if (++stage == S) { stage = 0; phase ^= 1u; }
    }
}

// ------------------------------------------------------- row-form consumer
//
// Causal multi-query with more than 8 q rows per KV walk (head sizes up to
// 128).  The launch row's packed q rows (row r: query r / G, head r % G) are
// the MMA's M, so one walk over the KV serves up to 32 of them.  Consumer
// warp w takes token slice ts = w % (ST/16), the stage rows 16 ts .. 16 ts +
// 15, and q tile qt = w / (ST/16), the q rows 16 qt .. 16 qt + 15:
//   S (16 q rows x 16 tokens) = Q K^T as two n8 tiles of tokens, K read as the
//     B operand (ldmatrix, rows = tokens);
//   the online-softmax update runs per q row on the accumulator fragments
//     (max over the tokens: the four lanes of a quad);
//   O (16 q rows x D) += P V, the score fragments serving as P's A fragments
//     where they stand (bf16 hi + lo parts), V read transposed as the B operand.
// Each warp keeps (m, l, o) of its q rows over its token slice.  At a segment
// end the slices of each q tile merge in shared memory, one q tile at a time,
// and the unit roles follow as in the n8 form (run_consumer).

// Zero output rows of the units with no tokens (they have no segment), shared
// round-robin over the grid: the stores overlap the wait for the first stage.
template <int D, int kThreadsC>
__device__ __forceinline__ void zero_empty_rows(const SplitParams& p, const int32_t* pfx, int ct) {
    for (int u = blockIdx.x; u < p.B * p.Hkv; u += gridDim.x) {
        const int sq = u / p.Hkv, kvh = u - sq * p.Hkv;
        if (pfx[sq + 1] != pfx[sq]) continue;
        const RowInfo ri = row_info<true>(p, sq);
        const int NR = ri.cnt * p.G;
        for (int i4 = ct; i4 < NR * D / 4; i4 += kThreadsC) {
            const int h = (4 * i4) / D, d4 = 4 * i4 - h * D;
            const int64_t o = qo_offset<true>(p, ri.b, ri.first + h / p.G, kvh * p.G + h % p.G, D) + d4;
            if (p.out_f32) *reinterpret_cast<float4*>(p.out_f32 + o) = make_float4(0.f, 0.f, 0.f, 0.f);
            else *reinterpret_cast<uint2*>(p.out + o) = make_uint2(0u, 0u);
        }
    }
}

// One 16-row q tile of a row-form segment end, once the consumers have
// staged their token slices' states: st_m / st_l [slice][32 q rows], st_o
// [slice][16 rows of the tile][D + 8].  The first tile decides the piece's
// role (whole unit, stored partial, or the last piece, which merges every
// stored partial with its own); each (row, 4 columns) of the tile is then
// combined over the slices and written (bf16 o / l, or the fp32 partial).
// Returns false when the CTA aborts.
template <int D, int kSlices, int kThreadsC>
__device__ __forceinline__ bool rows_tile_merge(const SplitParams& p, const StageMeta& m, int tile, int ct,
                                                int32_t ticket, const UnitPieces& pc, const GroupRange& grs,
                                                const RowInfo& ri, const float* st_m, const float* st_l,
                                                const float* st_o, int32_t* st_role, uint32_t cbar,
                                                uint32_t& cphase, volatile int* abort_flag, int& role) {
    constexpr int kOStride = D + 8;
    const bool whole = (m.flags & kWholeUnit) != 0;
    const int u = m.b * p.Hkv + m.kvh;
    const int NR = m.nr, SR = p.rows_per_slot, G = p.G;
        if (tile == 0 && ct == 0) {
            int32_t r = whole ? kRoleWhole : ticket == pc.n - 1 ? kRoleMerge : kRoleStore;
            if (r == kRoleMerge) {
                int32_t* cnt = p.unit_sync + 2 * u;
                bool ready = ld_acquire_gpu(cnt + 1) == pc.n - 1;
                if (!ready) {
                    const uint64_t t0 = global_ns();
                    while (!(ready = ld_acquire_gpu(cnt + 1) == pc.n - 1) &&
                           global_ns() - t0 <= kWaitLimitNs) {
                    }
                }
                if (ready) {
                    cnt[0] = 0;  // every piece has drawn and stored: reset for the next launch
                    cnt[1] = 0;
                } else {
                    atomicOr(p.err, PDA_DEVERR_TIMEOUT_);
                    *abort_flag = 1;
                    r = kRoleAbort;
                }
            }
            *st_role = r;
        }
        if (!consumer_sync(cbar, cphase, p.err, abort_flag)) return false;
        role = *st_role;
        if (role == kRoleAbort) return false;
        const int h0 = tile * 16, nrt = min(16, NR - h0);
        for (int i4 = ct; i4 < nrt * D / 4; i4 += kThreadsC) {
            const int hr = (4 * i4) / D, d4 = 4 * i4 - hr * D;
            const int h = h0 + hr;  // q row of the unit
            float M = kNegInf;
#pragma unroll
            for (int w = 0; w < kSlices; ++w) M = fmaxf(M, st_m[w * kMaxRowsPerWalk + h]);
            float Ls = 0.f;
            float4 Os = make_float4(0.f, 0.f, 0.f, 0.f);
            if (M != kNegInf) {
#pragma unroll
                for (int w = 0; w < kSlices; ++w) {
                    const float f = ex2(st_m[w * kMaxRowsPerWalk + h] - M);
                    const float4 v =
                        *reinterpret_cast<const float4*>(st_o + (size_t)(w * 16 + hr) * kOStride + d4);
                    Ls += st_l[w * kMaxRowsPerWalk + h] * f;
                    Os.x += v.x * f; Os.y += v.y * f; Os.z += v.z * f; Os.w += v.w * f;
                }
            }
            if (role == kRoleStore) {
                const int64_t r = (int64_t)(u + (int)blockIdx.x) * SR + h;
                *reinterpret_cast<float4*>(p.part_o + r * D + d4) = Os;
                if (d4 == 0) {
                    p.part_ml[r * 2] = M;
                    p.part_ml[r * 2 + 1] = Ls;
                }
                continue;
            }
            if (role == kRoleMerge) {
                // every piece in piece order, this piece's own state in its
                // place, up to four partials per memory round trip (the
                // row form's registers allow four)
                float Mr = kNegInf, Lr = 0.f;
                float4 Or = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int i0 = 0; i0 < pc.n; i0 += 4) {
                    float mi[4], li[4];
                    float4 oi[4];
                    bool own[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        mi[k] = kNegInf;
                        li[k] = 0.f;
                        oi[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                        const int64_t c = piece_cta(pc, i0 + k, grs);
                        own[k] = i0 + k < pc.n && c == (int64_t)blockIdx.x;
                        if (i0 + k >= pc.n || own[k]) continue;
                        const int64_t r = (u + c) * SR + h;
                        mi[k] = ld_cg(p.part_ml + r * 2);
                        li[k] = ld_cg(p.part_ml + r * 2 + 1);
                        oi[k] = __ldcg(reinterpret_cast<const float4*>(p.part_o + r * D + d4));
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if (own[k]) merge_state(Mr, Lr, Or, M, Ls, Os);
                        else merge_state(Mr, Lr, Or, mi[k], li[k], oi[k]);
                    }
                }
                M = Mr;
                Ls = Lr;
                Os = Or;
            }
            const float4 v = Ls > 0.f ? make_float4(Os.x / Ls, Os.y / Ls, Os.z / Ls, Os.w / Ls)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
            const int64_t oo = qo_offset<true>(p, ri.b, ri.first + h / G, m.kvh * G + h % G, D) + d4;
            if (p.out_f32) {
                *reinterpret_cast<float4*>(p.out_f32 + oo) = v;
            } else {
                uint2 w2;
                w2.x = pack_bf16x2(v.x, v.y);
                w2.y = pack_bf16x2(v.z, v.w);
                *reinterpret_cast<uint2*>(p.out + oo) = w2;
            }
        }
    return true;
}

template <int D, int ST, int MODE>
__device__ __forceinline__ void run_consumer_rows(const SplitParams& p, uint32_t base_s, uint8_t* base,
                                                  const SmemLayout& L, const StageMeta* meta,
                                                  const int32_t* pfx, volatile int* abort_flag, int warp,
                                                  int lane) {
    using C = Cfg<D, ST, MODE>;
    constexpr int S = C::kStages;
    constexpr int KS = C::kKSteps;       // 16-column steps of D
    constexpr int NT = D / 8;            // n8 tiles of O over D
    constexpr int kSlices = ST / 16;     // token slices of a stage
    constexpr int kThreadsC = C::kConsumerWarps * 32;
    constexpr int kOStride = D + 8;      // staged o row (floats): quads of rows fall in distinct banks
    static_assert(C::kQTiles > 0, "row form");
    static_assert(kSlices * 16 * kOStride * 4 <= C::kStageBytes, "one q tile's staged states fit a stage");
    static_assert(kSlices <= 4 && C::kQTiles * 16 <= kMaxRowsPerWalk, "st_m / st_l capacity");
    const uint32_t full0 = base_s + L.bars, empty0 = full0 + 8 * S;
    const int g = lane >> 2, t = lane & 3;
    const int ts = warp % kSlices, qt = warp / kSlices;
    const int r0 = ts * 16;                          // the warp's first row of a stage
    const int G = p.G;
    const float sl2 = p.scale_log2;
    const int row0 = qt * 16 + g, row1 = row0 + 8;   // this lane's q rows
    const int qc0 = row0 / G, qc1 = row1 / G;        // their queries within the launch row
    // ldmatrix row addresses: QK reads K as the B operand (matrices: tokens
    // 0-7 / 8-15 by columns lo / hi), PV reads V transposed as the B operand
    // (matrices: tokens 0-7 / 8-15 of columns lo, then of columns hi).
    const int k_row = r0 + (lane & 7) + ((lane >> 4) << 3);
    const int k_cpar = (lane >> 3) & 1;
    const int v_row = r0 + (lane & 7) + (((lane >> 3) & 1) << 3);
    const int v_cpar = lane >> 4;
    const int lbs = p.row_gather ? C::kLogST : 31 - __clz(p.bs);
    int swh[C::kHalves];  // swizzle of this lane's ldmatrix rows in slab h (row & 7 == lane & 7)
#pragma unroll
    for (int h = 0; h < C::kHalves; ++h) swh[h] = swz(lane, h, lbs);
    const uint32_t hs = (uint32_t)(128 << lbs);
    const uint32_t k_off = row_off<D>(k_row, lbs);
    const uint32_t v_off = row_off<D>(v_row, lbs);

    float o[NT][4];      // rows row0 ([0], [1]) and row1 ([2], [3]), columns 8i + 2t, + 1
    uint32_t qa[KS][4];  // Q's A fragments
    float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) qa[kk][0] = qa[kk][1] = qa[kk][2] = qa[kk][3] = 0u;

    const uint32_t cbar = base_s + L.cbar;
    uint32_t cphase = 0;
    int stage = 0;
    uint32_t phase = 0;
    int32_t ticket = 0;  // consumer thread 0: this piece's ticket for its split unit
    const int ct = warp * 32 + lane;
    zero_empty_rows<D, kThreadsC>(p, pfx, ct);

    while (true) {
        if (*abort_flag) break;
        if (!mbar_wait_bounded(full0 + 8 * stage, phase, kWaitLimitNs)) {
            atomicOr(p.err, PDA_DEVERR_TIMEOUT_);
            *abort_flag = 1;
            break;
        }
        const StageMeta m = meta[stage];
        if (m.flags & kDone) break;
        if (warp == 0 && lane == 0 && (m.flags & kSegEnd) && !(m.flags & kWholeUnit))
            ticket = atomicAdd(p.unit_sync + 2 * (m.b * p.Hkv + m.kvh), 1);
        const uint32_t sK = base_s + (uint32_t)stage * C::kStageBytes;
        const uint32_t sV = sK + C::kTileBytes;

        if (m.flags & kSegBegin) {  // (m, l, o) are reset: at the start and after each segment end
            const uint8_t* sq = base + (sV - base_s) + C::kTileBytes;  // [nr][D] bf16
            const bool v0 = row0 < m.nr, v1 = row1 < m.nr;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                const uint8_t* ra = sq + (size_t)(row0 * D + 16 * kk + 2 * t) * 2;
                const uint8_t* rb = sq + (size_t)(row1 * D + 16 * kk + 2 * t) * 2;
                qa[kk][0] = v0 ? *reinterpret_cast<const uint32_t*>(ra) : 0u;
                qa[kk][1] = v1 ? *reinterpret_cast<const uint32_t*>(rb) : 0u;
                qa[kk][2] = v0 ? *reinterpret_cast<const uint32_t*>(ra + 16) : 0u;
                qa[kk][3] = v1 ? *reinterpret_cast<const uint32_t*>(rb + 16) : 0u;
            }
        }
        // a q tile past the launch row's rows has nothing to compute
        if (r0 < m.n_valid && qt * 16 < m.nr) {
            const bool partial = r0 + 16 > m.n_valid;
            if (partial) {  // V rows past the valid ones may hold anything: P V must see zeros
                zero_rows<D>(sV, m.n_valid, r0 + 16, lbs, lane);
                __syncwarp();
            }
            // S = Q K^T: s[j] holds tokens r0 + 8j .. r0 + 8j + 7 (two independent chains)
            float s[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                uint32_t b[4];
                const int cc = (((kk & 3) << 1) + k_cpar) ^ swh[kk >> 2];
                ldsm_x4(sK + k_off + (uint32_t)(kk >> 2) * hs + (cc << 4), b);
                mma_16816(s[0], qa[kk], b[0], b[1]);
                mma_16816(s[1], qa[kk], b[2], b[3]);
            }
            // element [j][e]: q row e < 2 ? row0 : row1, stage row r0 + 8j + 2t + (e & 1)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[j][e] *= sl2;
            // Masks: the rows past the stage's valid ones and, causally, the tokens
            // past a row's query (query qi of the launch row sees tokens up to
            // m.lim + qi).  Element [j][e] stays iff 8j + (e & 1) <= th(e); the
            // thresholds are taken once, and stages that need no mask skip it.
            const int pos0 = m.j0 * p.bs + r0;  // the warp's first token
            if (partial || pos0 + 15 > m.lim) {
                const int tv = m.n_valid - 1 - r0 - 2 * t;
                const int th0 = min(tv, m.lim + qc0 - pos0 - 2 * t);
                const int th1 = min(tv, m.lim + qc1 - pos0 - 2 * t);
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (8 * j + (e & 1) > (e < 2 ? th0 : th1)) s[j][e] = kNegInf;
            }
            // row max over the 16 tokens (the quad's lanes)
            float x0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
            float x1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 1));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 1));
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 2));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 2));
            // lazy reference (kLazyLog2): o is rescaled only when a row's max
            // runs more than 2^8 past its reference
            const bool up0 = x0 > m0 + kLazyLog2, up1 = x1 > m1 + kLazyLog2;
            if (__any_sync(0xffffffffu, up0 || up1)) {
                const float a0 = up0 ? ex2(m0 - x0) : 1.f;  // an empty row (m = -inf): 0
                const float a1 = up1 ? ex2(m1 - x1) : 1.f;
                if (up0) m0 = x0;
                if (up1) m1 = x1;
                l0 *= a0;
                l1 *= a1;
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    o[i][0] *= a0; o[i][1] *= a0; o[i][2] *= a1; o[i][3] *= a1;
                }
            }
            const float u0 = m0 == kNegInf ? 0.f : m0;  // a row with no token yet: every p is 0
            const float u1 = m1 == kNegInf ? 0.f : m1;
            float pr[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                pr[j][0] = ex2(s[j][0] - u0);
                pr[j][1] = ex2(s[j][1] - u0);
                pr[j][2] = ex2(s[j][2] - u1);
                pr[j][3] = ex2(s[j][3] - u1);
            }
            // P's A fragments (rows row0 / row1, tokens 2t.. / 8 + 2t..) as bf16
            // hi + lo parts (p = hi + lo to about 2^-17 relative)
            uint32_t ah[4], al[4];
            ah[0] = pack_bf16x2(pr[0][0], pr[0][1]);
            ah[1] = pack_bf16x2(pr[0][2], pr[0][3]);
            ah[2] = pack_bf16x2(pr[1][0], pr[1][1]);
            ah[3] = pack_bf16x2(pr[1][2], pr[1][3]);
            al[0] = pack_bf16x2(pr[0][0] - bf16_lo(ah[0]), pr[0][1] - bf16_hi(ah[0]));
            al[1] = pack_bf16x2(pr[0][2] - bf16_lo(ah[1]), pr[0][3] - bf16_hi(ah[1]));
            al[2] = pack_bf16x2(pr[1][0] - bf16_lo(ah[2]), pr[1][1] - bf16_hi(ah[2]));
            al[3] = pack_bf16x2(pr[1][2] - bf16_lo(ah[3]), pr[1][3] - bf16_hi(ah[3]));
            // l sums the fp32 weights (this lane's four tokens; the quad is summed at the end)
            l0 += (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
            l1 += (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
            // O += P V over 16 columns of D per ldmatrix
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                uint32_t b[4];
                const int cc = (((mt & 3) << 1) + v_cpar) ^ swh[mt >> 2];
                ldsm_x4_trans(sV + v_off + (uint32_t)(mt >> 2) * hs + (cc << 4), b);
                mma_16816(o[2 * mt], ah, b[0], b[1]);
                mma_16816(o[2 * mt + 1], ah, b[2], b[3]);
                mma_16816(o[2 * mt], al, b[0], b[1]);
                mma_16816(o[2 * mt + 1], al, b[2], b[3]);
            }
            if (partial) fence_proxy_async_smem();  // generic writes before the next TMA
        }
        if (m.flags & kSegEnd) {
            // ---- segment end: per q tile, the token slices' states merge
            // through this stage's memory (released only afterwards); roles as
            // in run_consumer.
            float* st_m = reinterpret_cast<float*>(base + L.st_m);  // [slice][32 q rows]
            float* st_l = reinterpret_cast<float*>(base + L.st_l);
            int32_t* st_role = reinterpret_cast<int32_t*>(base + L.st_x) + 2 * kMaxGroup;
            float* st_o = reinterpret_cast<float*>(base + (sK - base_s));  // [slice][16][kOStride]
            // the next segment loads its own q fragments (no live values across the epilogue)
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) qa[kk][0] = qa[kk][1] = qa[kk][2] = qa[kk][3] = 0u;
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
            if (!consumer_sync(cbar, cphase, p.err, abort_flag)) break;  // all reads of the stage done
            const bool whole = (m.flags & kWholeUnit) != 0;
            const int u = m.b * p.Hkv + m.kvh;
            UnitPieces pc;
            pc.cf = 0; pc.su = 0; pc.n = 1; pc.every = true;
            // the CTA's group, recomputed here rather than kept in registers over the loop
            const GroupRange grs = group_of_cta(blockIdx.x, pfx, p.B, rows_per_seq<true>(p), p.Hkv, gridDim.x);
            if (!whole) pc = unit_pieces(pfx, m.b, m.kvh, p.Hkv, p.unit_cost, grs);
            const RowInfo ri = row_info<true>(p, m.b);
            int role = kRoleAbort;
            bool stop = false;
            for (int tile = 0; tile < C::kQTiles && !stop; ++tile) {
                // the previous tile's staged states are read: overwrite them
                if (tile > 0 && !consumer_sync(cbar, cphase, p.err, abort_flag)) { stop = true; break; }
                if (qt == tile) {
                    if (t == 0) {
                        st_m[ts * kMaxRowsPerWalk + row0] = m0;
                        st_m[ts * kMaxRowsPerWalk + row1] = m1;
                        st_l[ts * kMaxRowsPerWalk + row0] = l0;
                        st_l[ts * kMaxRowsPerWalk + row1] = l1;
                    }
                    float* ra = st_o + (size_t)(ts * 16 + g) * kOStride + 2 * t;
                    float* rb = ra + 8 * kOStride;
#pragma unroll
                    for (int i = 0; i < NT; ++i) {
                        *reinterpret_cast<float2*>(ra + 8 * i) = make_float2(o[i][0], o[i][1]);
                        *reinterpret_cast<float2*>(rb + 8 * i) = make_float2(o[i][2], o[i][3]);
                        o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;  // the next segment's start
                    }
                    m0 = m1 = kNegInf;
                    l0 = l1 = 0.f;
                }
                if (!rows_tile_merge<D, kSlices, kThreadsC>(p, m, tile, ct, ticket, pc, grs, ri, st_m, st_l, st_o,
                                                            st_role, cbar, cphase, abort_flag, role)) {
                    stop = true;
                    break;
                }
            }
            if (stop) break;
            if (!consumer_sync(cbar, cphase, p.err, abort_flag)) break;
            // a stored piece signals after every consumer thread's stores (ordered
            // before this thread's release by the consumer barrier)
            if (role == kRoleStore && ct == 0) red_release_gpu_add(p.unit_sync + 2 * u + 1, 1);
            fence_proxy_async_smem();  // staging writes before the next TMA into this stage
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);
        if (++stage == S) { stage = 0; phase ^= 1u; }
    }
}

// ------------------------------------------------------------ tcgen05 form
//
// Row form of causal multi-query on the tcgen05 tensor cores, for up to 32 q
// rows per launch row at head size 128 (switched on per context).  Two groups
// of four softmax warps take the even and the odd stages.  Per stage of 64 KV
// rows:
//   S = Q K^T     (M = 128: Q in four copies of the launch row's 32 q rows, one
//                  per tensor-memory lane quarter, as the A operand in tensor
//                  memory; N = the stage's 64 tokens, K from shared memory;
//                  fp32 in the group's tensor-memory S buffer)
//   softmax       (warp w of the group, lane r: q row r over the 16 tokens of
//                  slice w, read from lanes 32w + r, columns 16w..16w+15; the
//                  four slices' row maxima meet in shared memory, so a row
//                  keeps one reference per group)
//   O^T += V^T P^T (M = D = 128: V as an MN-major A operand; N = the 32 q rows:
//                  P as bf16 hi and lo parts, [q row][token], written into the
//                  stage's q area once the stage's q rows are in tensor memory;
//                  the group's O^T in 32 tensor-memory columns: lane =
//                  head-dim element)
// At a segment end the two groups' states merge as two slices.  One thread of
// the MMA warp issues every MMA, S up to one stage ahead of P V; the
// tcgen05.commit arrivals tell the softmax warps that S (and every MMA issued
// before it) is done or that a P V is, and the producer that a stage is free.
// A kernel with tcgen05 instructions runs one CTA per SM.  The stage tiles are
// [slab][64 rows][128 B] for every loader (one TMA box per block and slab at
// head size 128).

// Tensor-memory columns (256 allocated): an S buffer and an O^T per group of
// softmax warps, Q.
constexpr uint32_t kTmS = 0, kTmO = 128, kTmQ = 192;

// The stage tiles are [slab][64 rows][128 B], 128-byte swizzled, for every
// loader: one box per block and slab, or rows gathered one by one.  So the
// 64 rows of a slab are one K-major operand of N = 64 (8-row groups 1024
// bytes apart), and token chunk c of V, as the MN-major A operand of O^T,
// starts at c * 2048 (its 64-element slabs kHalfBytes apart).
#ifndef PDA_TC_P_LO
#define PDA_TC_P_LO 1  // P V also over the bf16 low parts of P (p = hi + lo)
#endif
constexpr uint32_t kTcPLo = 4096;  // the lo part of P after the hi part ([32][64] bf16 each)

// Barriers of the tcgen05 form (base + L.tcb), each at most one phase ahead of
// its waiter: Q ready (a group of softmax warps, once per segment); for the
// even / odd stages (the two groups) S done (commit), P ready (the group) and
// P V done (commit); finish (commit); each group's own barrier (its four
// warps); then the tensor-memory base address.
enum TcBar : uint32_t { kTcQ = 0, kTcS = 8, kTcP = 24, kTcPV = 40, kTcFin = 56, kTcG = 64, kTcSlot = 80 };

// A bounded barrier wait whose outcome the whole warp shares (the warp then
// reaches the warp-wide tensor-memory loads together, or leaves together).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, kWaitLimitNs) ? 1 : 0) != 0;
}

template <int D, int ST, int MODE>
__device__ __forceinline__ void run_mma_tc(const SplitParams& p, uint32_t base_s, const SmemLayout& L,
                                           const StageMeta* meta, volatile int* abort_flag, uint32_t tmem) {
    using C = Cfg<D, ST, MODE>;
    constexpr int S = C::kStages;
    constexpr int KS = C::kKSteps;
    constexpr uint32_t idS = umma_idesc_bf16(128, 64, false);
    constexpr uint32_t idO = umma_idesc_bf16(D, kMaxRowsPerWalk, false, true);
    static_assert(D == 128, "O^T takes the head dimension as the MMA's M = 128");
    const uint32_t full0 = base_s + L.bars, empty0 = full0 + 8 * S, tcb = base_s + L.tcb;
    // S cursor (next stage whose S to issue) and P V cursor, as counts and ring slots
    uint32_t sit = 0, pit = 0, segs = 0;
    uint32_t fresh = 3u;  // bit g: group g's O^T holds nothing of the current segment yet
    int ss = 0, ps = 0;
    uint32_t sph = 0;
    bool ok = true, done = false;
    auto issue_s = [&](const StageMeta& m) {
        tc_fence_after();
        const uint32_t sK = base_s + (uint32_t)ss * C::kStageBytes;
        const uint32_t tS = tmem + kTmS + 64u * (sit & 1u);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const uint64_t b = umma_sdesc(sK + (uint32_t)(ks >> 2) * C::kHalfBytes + (uint32_t)(ks & 3) * 32u, 16u,
                                          1024u);
            umma_bf16_ts(tS, tmem + kTmQ + 8u * ks, b, idS, ks > 0);
        }
        umma_commit(tcb + kTcS + 8u * (sit & 1u));
        if (m.flags & kSegBegin) ++segs;
        ++sit;
        if (++ss == S) { ss = 0; sph ^= 1u; }
    };
    // Polls for whichever is ready: the next stage's S (its rows landed, its Q
    // written at a segment start, and its S buffer read: at most one S ahead of
    // the P V cursor), then the pending P V (its P written).  S goes first: the
    // softmax warps wait for it.
    uint64_t idle_since = 0;
    bool idle = false;
    while (true) {
        if (*abort_flag) break;
        bool progressed = false;
        if (!done && sit <= pit + 1 && mbar_test_wait(full0 + 8 * ss, sph)) {
            const StageMeta m = meta[ss];
            if (m.flags & kDone) {
                done = true;
            } else if (!(m.flags & kSegBegin) || mbar_test_wait(tcb + kTcQ, segs & 1u)) {
                issue_s(m);
                progressed = true;
            }
        }
        if (pit < sit && mbar_test_wait(tcb + kTcP + 8u * (pit & 1u), (pit >> 1) & 1u)) {
            tc_fence_after();
            const StageMeta m = meta[ps];
            const uint32_t sV = base_s + (uint32_t)ps * C::kStageBytes + C::kTileBytes;
            const uint32_t sP = sV + C::kTileBytes;  // the stage's q area holds P
            const int nch = (m.n_valid + 15) >> 4;
            if (m.flags & kSegBegin) fresh = 3u;
            const uint32_t tO = tmem + kTmO + 32u * (pit & 1u);  // the stage's group's O^T
            bool acc = ((fresh >> (pit & 1u)) & 1u) == 0u;
            fresh &= ~(1u << (pit & 1u));
            for (int c = 0; c < nch; ++c) {
                const uint64_t a = umma_sdesc(sV + 2048u * c, C::kHalfBytes, 1024u);
                umma_bf16_ss(tO, a, umma_sdesc(sP + 32u * c, 16u, 1024u), idO, acc);
                if (PDA_TC_P_LO) umma_bf16_ss(tO, a, umma_sdesc(sP + kTcPLo + 32u * c, 16u, 1024u), idO, true);
                acc = true;
            }
            umma_commit(tcb + kTcPV + 8u * (pit & 1u));
            umma_commit(empty0 + 8 * ps);
            ++pit;
            if (++ps == S) ps = 0;
            progressed = true;
        }
        if (done && pit == sit) break;
        if (progressed) {
            idle = false;
        } else if (!idle) {
            idle = true;
            idle_since = global_ns();
        } else if (global_ns() - idle_since > kWaitLimitNs) {
            ok = false;
            break;
        }
    }
    if (!ok) {
        atomicOr(p.err, PDA_DEVERR_TIMEOUT_);
        *abort_flag = 1;
    }
    // every MMA issued has completed before the tensor memory is freed
    umma_commit(tcb + kTcFin);
    if (!mbar_wait_bounded(tcb + kTcFin, 0, kWaitLimitNs)) {
        atomicOr(p.err, PDA_DEVERR_TIMEOUT_);
        *abort_flag = 1;
    }
}

template <int D, int ST, int MODE>
__device__ __forceinline__ void run_consumer_tc(const SplitParams& p, uint32_t base_s, uint8_t* base,
                                                const SmemLayout& L, const StageMeta* meta,
                                                const int32_t* pfx, volatile int* abort_flag, int warp,
                                                int lane, uint32_t tmem) {
    using C = Cfg<D, ST, MODE>;
    constexpr int S = C::kStages;
    constexpr int kThreadsC = C::kConsumerWarps * 32;
    constexpr int kOStride = D + 8;
    static_assert(C::kConsumerWarps == 8 && ST == 64 && D == 128, "tcgen05 form: two groups of four slice warps");
    static_assert(2 * 2 * 16 * kOStride * 4 <= C::kStageBytes, "both groups' staged o rows fit a stage");
    const uint32_t full0 = base_s + L.bars, empty0 = full0 + 8 * S, tcb = base_s + L.tcb;
    const int g = warp >> 2;                              // group: the stages whose index has parity g
    const int w = warp & 3;                               // token slice and lane quarter
    const uint32_t tl = tmem + ((uint32_t)(32 * w) << 16);  // this warp's tensor-memory lanes
    const uint32_t tS = tl + kTmS + 64u * g + 16u * w;    // this group's S buffer, this slice's columns
    const uint32_t tO = tl + kTmO + 32u * g;              // this group's O^T (lane: head-dim element)
    const int r = lane;                                   // this thread's q row (S, P)
    const int qi = r / p.G;                               // its query within the launch row
    const float sl2 = p.scale_log2;
    const int lbs = C::kLogST;  // one 64-row block per stage tile
    float* xmax = reinterpret_cast<float*>(base + L.tcx);  // [group][2][4 slices][32 rows]
    float* lpart = xmax + 2 * 2 * 4 * kMaxRowsPerWalk;    // [8 warps][32 rows]
    float mref = kNegInf;  // the row's reference in this group (the same in its four warps)
    float lw = 0.f;        // the row's weight sum over this warp's slice of this group's stages
    bool active = false;   // this group has a stage in the current segment

    const uint32_t cbar = base_s + L.cbar;           // the eight softmax warps
    const uint32_t gbar = tcb + kTcG + 8u * g;       // this group's four warps
    uint32_t cphase = 0, gphase = 0, it = 0;
    int stage = 0;
    uint32_t phase = 0;
    int32_t ticket = 0;
    const int ct = warp * 32 + lane;
    zero_empty_rows<D, kThreadsC>(p, pfx, ct);

    auto give_up = [&]() {
        atomicOr(p.err, PDA_DEVERR_TIMEOUT_);
        *abort_flag = 1;
    };
    // Barriers among the softmax warps (all eight; this group's four) whose
    // outcome each warp shares.
    auto sync_all = [&]() -> bool {
        const bool ok = consumer_sync(cbar, cphase, p.err, abort_flag);
        return __all_sync(0xffffffffu, ok ? 1 : 0) != 0;
    };
    auto sync_group = [&]() -> bool {
        const bool ok = consumer_sync(gbar, gphase, p.err, abort_flag);
        return __all_sync(0xffffffffu, ok ? 1 : 0) != 0;
    };
    // This warp's copy of a segment's q rows (the q area of stage st, nr rows)
    // into tensor memory (lane r: q row r, zero past the launch row's rows),
    // once every S of the previous segment is done; then Q ready.  Rows are
    // D * 2 bytes apart: lane r reads the 16-byte chunks of each 128-byte half
    // in the order c ^ (r & 7), so that 8 lanes in a row hit 8 different
    // banks, and swaps them back into place.
    auto write_q = [&](int st, int nr) {
        const uint8_t* sq = base + (uint32_t)st * C::kStageBytes + 2 * C::kTileBytes + (size_t)r * D * 2;
        const int x = r & 7;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
            uint4 t[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
                t[c] = r < nr ? *reinterpret_cast<const uint4*>(sq + 128 * h + 16 * (c ^ x))
                              : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int bit = 1; bit < 8; bit <<= 1) {
                const bool sw = (x & bit) != 0;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    if (!(c & bit)) {
                        const uint4 a = t[c], d = t[c | bit];
                        t[c] = sw ? d : a;
                        t[c | bit] = sw ? a : d;
                    }
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                uint32_t v[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 y = t[4 * k + j];
                    v[4 * j] = y.x; v[4 * j + 1] = y.y; v[4 * j + 2] = y.z; v[4 * j + 3] = y.w;
                }
                tmem_st16u(tl + kTmQ + 32u * h + 16u * k, v);
            }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tcb + kTcQ);
    };
    bool q_written = false;  // this group wrote the next segment's Q before the segment's end
    // Every warp of both groups walks every stage: its own group's stages in
    // full, the other group's for their flags (a segment end gathers both).
    while (true) {
        if (*abort_flag) break;
        if (!warp_wait(full0 + 8 * stage, phase)) { give_up(); break; }
        const StageMeta m = meta[stage];
        if (m.flags & kDone) break;
        const uint32_t sK = base_s + (uint32_t)stage * C::kStageBytes;
        const uint32_t sV = sK + C::kTileBytes;
        const uint32_t sP = sV + C::kTileBytes;  // the q area; P once Q is in tensor memory
        if ((it & 1u) == (uint32_t)g) {
            if (m.flags & kSegBegin) {
                if (!q_written) write_q(stage, m.nr);
                q_written = false;
            }
            active = true;
            if (!warp_wait(tcb + kTcS + 8u * g, (it >> 1) & 1u)) { give_up(); break; }
            tc_fence_after();
            float s[16];
            tmem_ld16(tS, s);
            // Masks: the slice's rows past the stage's valid ones, the launch row's
            // rows past its own, and causally the tokens past the row's query
            // (query qi of the launch row sees tokens up to m.lim + qi).
            const int pos0 = m.j0 * p.bs + 16 * w;  // the slice's first token
            const int th = r < m.nr ? min(m.n_valid - 1 - 16 * w, m.lim + qi - pos0) : -1;
            float xw = kNegInf;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                s[i] = i <= th ? s[i] * sl2 : kNegInf;
                xw = fmaxf(xw, s[i]);
            }
            // the row's max over the stage: the group's four slice maxima meet in
            // shared memory (the barrier also ends every read of the stage's q
            // rows, so P may overwrite them)
            float* xm = xmax + (size_t)((2 * g + ((it >> 1) & 1u)) * 4) * kMaxRowsPerWalk;
            xm[32 * w + r] = xw;
            if (!sync_group()) break;
            const float x = fmaxf(fmaxf(xm[r], xm[32 + r]), fmaxf(xm[64 + r], xm[96 + r]));
            // lazy reference: o is rescaled only when the max runs more than 2^8
            // past the reference (a row with no weight yet has o = 0: nothing to
            // scale); this group's previous P V is done (it was issued before this
            // stage's S); every warp scales its lanes of the group's O^T for all 32
            // rows
            const bool up = x > mref + kLazyLog2;
            const bool scale_o = up && mref != kNegInf;
            if (__any_sync(0xffffffffu, scale_o)) {
                const float a = scale_o ? ex2(mref - x) : 1.f;
                lw *= a;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    float o[16];
                    tmem_ld16(tO + 16u * k, o);
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[i] *= __shfl_sync(0xffffffffu, a, 16 * k + i);
                    tmem_st16(tO + 16u * k, o);
                }
            }
            if (up) mref = x;
            const float u = mref == kNegInf ? 0.f : mref;
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float p0 = ex2(s[2 * i] - u), p1 = ex2(s[2 * i + 1] - u);
                lw += p0 + p1;
                hi[i] = pack_bf16x2(p0, p1);
                lo[i] = PDA_TC_P_LO ? pack_bf16x2(p0 - bf16_lo(hi[i]), p1 - bf16_hi(hi[i])) : 0u;
            }
            // P row r, this slice's 16 tokens: [32 rows][64 tokens] bf16, K-major, swizzled
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint32_t off = (uint32_t)r * 128u + (uint32_t)(((2 * w + k) ^ (r & 7)) << 4);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(sP + off), "r"(hi[4 * k]),
                             "r"(hi[4 * k + 1]), "r"(hi[4 * k + 2]), "r"(hi[4 * k + 3])
                             : "memory");
                if (PDA_TC_P_LO)
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(sP + kTcPLo + off),
                                 "r"(lo[4 * k]), "r"(lo[4 * k + 1]), "r"(lo[4 * k + 2]), "r"(lo[4 * k + 3])
                                 : "memory");
            }
            // V rows past the valid ones may hold anything: P V must see zeros
            if (16 * w < m.n_valid && m.n_valid < 16 * w + 16) zero_rows<D>(sV, m.n_valid, 16 * w + 16, lbs, lane);
            fence_proxy_async_smem();  // P and the zeroed rows, before the MMA reads them
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tcb + kTcP + 8u * g);
        }
        if (m.flags & kSegEnd) {
            // ---- segment end, both groups.  First all eight warps meet: the
            // stage's own group arrives only after its S wait, which makes its
            // previous P V complete, so the P V barrier of the stage's parity is at
            // this stage's phase for either group to wait on (a parity wait on a
            // barrier one phase behind would pass at once).  Once this stage's P V
            // is done (and so every MMA of the segment, issued before it: no S still
            // reads the segment's Q and no MMA reads the stage), the group whose
            // stage is next writes the next segment's Q, so that its S runs during
            // this epilogue; then each group's o / l as one slice through this
            // stage's memory, and the unit roles of the row forms
            const bool whole = (m.flags & kWholeUnit) != 0;
            const int u = m.b * p.Hkv + m.kvh;
            if (ct == 0 && !whole) ticket = atomicAdd(p.unit_sync + 2 * u, 1);
            if (!sync_all()) break;
            if (!warp_wait(tcb + kTcPV + 8u * (it & 1u), (it >> 1) & 1u)) { give_up(); break; }
            tc_fence_after();
            if (((it + 1u) & 1u) == (uint32_t)g) {
                const int ns = stage + 1 == S ? 0 : stage + 1;
                if (!warp_wait(full0 + 8 * ns, ns == 0 ? phase ^ 1u : phase)) { give_up(); break; }
                const StageMeta mn = meta[ns];
                if ((mn.flags & (kDone | kSegBegin)) == kSegBegin) {
                    write_q(ns, mn.nr);
                    q_written = true;
                }
            }
            float* st_m = reinterpret_cast<float*>(base + L.st_m);  // [group][32 q rows]
            float* st_l = reinterpret_cast<float*>(base + L.st_l);
            int32_t* st_role = reinterpret_cast<int32_t*>(base + L.st_x) + 2 * kMaxGroup;
            float* st_o = reinterpret_cast<float*>(base + (sK - base_s));  // [tile][group][16][kOStride]
            lpart[32 * warp + r] = lw;
#pragma unroll
            for (int k = 0; k < 2; ++k) {  // q rows 16k..16k+15: tile k
                float o[16];
                tmem_ld16(tO + 16u * k, o);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    st_o[(size_t)((2 * k + g) * 16 + i) * kOStride + 32 * w + lane] = active ? o[i] : 0.f;
            }
            if (!sync_all()) break;
            if (w == 0) {
                st_m[32 * g + r] = mref;
                st_l[32 * g + r] = (lpart[32 * (4 * g) + r] + lpart[32 * (4 * g + 1) + r]) +
                                   (lpart[32 * (4 * g + 2) + r] + lpart[32 * (4 * g + 3) + r]);
            }
            if (!sync_all()) break;
            UnitPieces pc;
            pc.cf = 0; pc.su = 0; pc.n = 1; pc.every = true;
            const GroupRange grs = group_of_cta(blockIdx.x, pfx, p.B, rows_per_seq<true>(p), p.Hkv, gridDim.x);
            if (!whole) pc = unit_pieces(pfx, m.b, m.kvh, p.Hkv, p.unit_cost, grs);
            const RowInfo ri = row_info<true>(p, m.b);
            int role = kRoleAbort;
            bool stop = false;
            for (int tile = 0; tile < 2; ++tile) {
                const bool merged = rows_tile_merge<D, 2, kThreadsC>(p, m, tile, ct, ticket, pc, grs, ri, st_m, st_l,
                                                                     st_o + (size_t)tile * 2 * 16 * kOStride, st_role,
                                                                     cbar, cphase, abort_flag, role);
                if (!__all_sync(0xffffffffu, merged ? 1 : 0)) { stop = true; break; }
            }
            if (stop) break;
            if (!sync_all()) break;
            if (role == kRoleStore && ct == 0) red_release_gpu_add(p.unit_sync + 2 * u + 1, 1);
            fence_proxy_async_smem();  // staging writes before the next TMA into this stage
            mref = kNegInf;
            lw = 0.f;
            active = false;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);
        ++it;
        if (++stage == S) { stage = 0; phase ^= 1u; }
    }
    tc_fence_before();
}

// ------------------------------------------------------------------ kernels

// The flattened range [begin, end) of this CTA (pda_plan.h): in unit mode CTA
// c takes unit c whole, otherwise its share of its row group's range.  Returns
// the CTA's group (not used in unit mode).
template <int MODE>
__device__ __forceinline__ GroupRange cta_range(const SplitParams& p, const int32_t* pfx, int32_t nv_max,
                                                int stage_rows, int64_t* begin, int64_t* end) {
    const GroupRange gr = group_of_cta(blockIdx.x, pfx, p.B, rows_per_seq<is_multi(MODE)>(p), p.Hkv,
                                       gridDim.x);
    const int64_t units = (int64_t)p.B * p.Hkv;
    if (unit_mode(units, gridDim.x, real_blocks(nv_max, p.unit_cost), stage_rows, p.bs)) {
        *begin = *end = 0;
        if ((int64_t)blockIdx.x < units) {
            const int b = blockIdx.x / p.Hkv, kvh = blockIdx.x - b * p.Hkv;
            const int32_t nv = pfx[b + 1] - pfx[b];
            *begin = (int64_t)pfx[b] * p.Hkv + (int64_t)kvh * nv;
            *end = *begin + nv;
        }
    } else {
        group_cta_range(gr, blockIdx.x, begin, end);
    }
    return gr;
}

#ifndef PDA_PREFETCH_STAGES
#define PDA_PREFETCH_STAGES 8
#endif
constexpr int kPrefetchStages = PDA_PREFETCH_STAGES;  // stages of blocks prefetched

// The prefetch warp: a speculative L2 prefetch of the blocks of the CTA's
// first stages, before the grid-dependency wait, so that while the previous
// kernel finishes, those blocks' K/V rows move towards L2.  It builds its own
// plan in registers (lengths read from L2, so no L1 line of them outlives the
// wait; no flags raised), reads the first block ids from L2 and prefetches
// their boxes, then exits: it shares no barrier with the other warps, which
// wait and run the decode as without it.  What it reads may be stale (the
// previous kernel may still be writing it): it only chooses which boxes to
// prefetch, every index is kept inside the CTA's table row and the pool, and
// the decode itself reads everything after the wait.  Single-query launches
// of block boxes (multi-query with one launch row per sequence).
template <int D, int ST, int MODE, int KPER>
__device__ __noinline__ void prefetch_first_stages_k(const SplitParams& p, int lane) {
    using C = Cfg<D, ST, MODE>;
    const int per = (p.B + 31) / 32;  // <= KPER
    const int lo = min(p.B, lane * per), hi = min(p.B, lo + per);
    const int lbs = 31 - __clz(p.bs);  // block sizes are powers of two
    int32_t v[KPER];  // plan blocks of this lane's sequences
#pragma unroll
    for (int k = 0; k < KPER; ++k) v[k] = lo + k < hi ? __ldcg(p.lens + lo + k) : 0;
    int32_t sum = 0, big = 0;
#pragma unroll
    for (int k = 0; k < KPER; ++k) {
        int32_t nb = v[k];  // blocks (tile steps) or tokens -> blocks, clamped to the table
        if (!p.lens_are_blocks) nb = nb > 0 ? (int32_t)(((int64_t)nb + p.bs - 1) >> lbs) : 0;
        nb = nb < 0 ? 0 : nb > p.table_stride ? p.table_stride : nb;
        v[k] = lo + k < hi ? plan_blocks(nb, p.unit_cost) : 0;
        sum += v[k];
        big = max(big, v[k]);
    }
    int32_t x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
        big = max(big, __shfl_xor_sync(0xffffffffu, big, o));
    }
    const int32_t base = x - sum;  // plan blocks before this lane's sequences
    const int64_t Hkv = p.Hkv, W = (int64_t)__shfl_sync(0xffffffffu, x, 31) * Hkv;
    const int64_t units = (int64_t)p.B * Hkv, c = blockIdx.x;
    int64_t begin, end;
    int32_t b = 0, nvb = 0, pfb = 0;
    if (unit_mode(units, gridDim.x, real_blocks(big, p.unit_cost), C::kST, p.bs)) {
        if (c >= units) return;
        b = (int32_t)(c / Hkv);
        int32_t pf = base;
#pragma unroll
        for (int k = 0; k < KPER; ++k) {
            if (lo + k == b) { pfb = pf; nvb = v[k]; }
            pf += v[k];
        }
        const int owner = b / per;  // per >= 1: b < B
        pfb = __shfl_sync(0xffffffffu, pfb, owner);
        nvb = __shfl_sync(0xffffffffu, nvb, owner);
        begin = (int64_t)pfb * Hkv + (c - (int64_t)b * Hkv) * nvb;
        end = begin + nvb;
    } else {
        begin = cta_begin(c, W, gridDim.x);
        end = cta_begin(c + 1, W, gridDim.x);
        const bool mine = sum > 0 && (int64_t)base * Hkv <= begin && begin < (int64_t)(base + sum) * Hkv;
        const unsigned who = __ballot_sync(0xffffffffu, mine);
        if (begin >= end || who == 0u) return;
        const int sel = __ffs(who) - 1;
        int32_t pf = base;
        bool found = false;
#pragma unroll
        for (int k = 0; k < KPER; ++k) {
            if (!found && v[k] > 0 && begin < (int64_t)(pf + v[k]) * Hkv) {
                b = lo + k; nvb = v[k]; pfb = pf; found = true;
            }
            pf += v[k];
        }
        b = __shfl_sync(0xffffffffu, b, sel);
        nvb = __shfl_sync(0xffffffffu, nvb, sel);
        pfb = __shfl_sync(0xffffffffu, pfb, sel);
    }
    const int64_t rem = begin - (int64_t)pfb * Hkv;
    if (nvb <= 0 || rem < 0 || b < 0 || b >= p.B) return;
    const int64_t kvh = rem / nvb, j = rem % nvb;
    if (kvh >= p.Hkv || j >= p.table_stride) return;
    const int64_t n = min(min(min((int64_t)real_blocks(nvb, p.unit_cost) - j, end - begin),
                              (int64_t)(kPrefetchStages * (C::kST / p.bs))),
                          (int64_t)p.table_stride - j);
    const int64_t row = (int64_t)b * p.table_stride + j;
    for (int64_t i = lane; i < n; i += 32) {  // the unit's next n blocks (one unit at most)
        const int64_t id = p.table ? (int64_t)__ldcg(p.table + row + i) : row + i;
        if (id >= 0 && id < p.num_blocks) {
            tma_prefetch_5d(&p.tm_k, 0, 0, 0, (int32_t)kvh, (int32_t)id);
            tma_prefetch_5d(&p.tm_v, 0, 0, 0, (int32_t)kvh, (int32_t)id);
        }
    }
}

// The plan in registers is sized to the batch (up to 1, 4 or 32 sequences a
// lane).  Not inlined: kept out of the split kernel's own code, whose start
// every launch fetches (inlined, it cost small batches 0.4 us a call).
template <int D, int ST, int MODE>
__device__ __noinline__ void prefetch_first_stages(const SplitParams& p, int lane) {
    // multi-query: one launch row per sequence only (then row s is sequence s
    // and reads its whole length, like plain decode)
    if (is_multi(MODE) && rows_per_seq<is_multi(MODE)>(p) != 1) return;
    if (p.B <= 32) prefetch_first_stages_k<D, ST, MODE, 1>(p, lane);
    else if (p.B <= 128) prefetch_first_stages_k<D, ST, MODE, 4>(p, lane);
    else prefetch_first_stages_k<D, ST, MODE, kMaxLaunchBatch / 32>(p, lane);
}

// Register cap: for D <= 128 two CTAs share an SM (two 3-stage rings keep as
// many bytes in flight as one 6-stage ring, and a second set of consumer warps
// hides the MMA/shuffle latency; measured 4 % faster than one CTA with six
// stages), which needs each 16K-register quarter of the SM to hold 3 of the
// 10 warps: at most 168 registers per thread.  D = 256
// runs one CTA per SM; with 32-row stages (block sizes below 8) a CTA has two
// consumer warps and one producer warp, and two CTAs share an SM.
template <int D, int ST, int MODE>
__global__ void __maxnreg__(split_max_regs(D, MODE)) split_kernel(const __grid_constant__ SplitParams p) {
    using C = Cfg<D, ST, MODE>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
    const SmemLayout L = smem_layout(D, ST, MODE, C::kStages, p.B);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t* pfx = reinterpret_cast<int32_t*>(base + L.pfx);
    int32_t* scan = reinterpret_cast<int32_t*>(base + L.scan);
    StageMeta* meta = reinterpret_cast<StageMeta*>(base + L.meta);

    // Programmatic dependent launch: barriers and descriptors are set up while
    // the previous kernel finishes; global memory is read only after
    // griddepcontrol.wait (the previous kernel complete, its writes visible),
    // and only then may the next kernel launch (its CTAs are scheduled as
    // this kernel's exit), so a kernel launched early behind this one knows
    // every kernel before this one complete.
    // A tile step right behind another tile step of the same step on the same
    // stream (p.early_inputs) instead lets the next kernel launch at once and
    // reads its inputs (lengths, tile lists, q, K/V) without waiting: the
    // first tile step of a chain waited for everything before it, so the
    // kernels that may still run beside this one are tile steps of the same
    // step, and no tile step writes another's inputs.  Its consumers wait
    // before their first access to what a tile step writes (the unit
    // counters, the partial slots, the running state).
    const bool early = MODE == kTiled && p.early_inputs != 0;
    if (early) pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            // full: the producer's arrive (+ one cp.async arrival per lane when
            // rows are copied with cp.async); empty: one arrival per consumer warp
            // (+ the MMA warp's commit in the tcgen05 form)
            mbar_init(base_s + L.bars + 8 * s, p.row_gather == 2 ? 33 : 1);
            mbar_init(base_s + L.bars + 8 * (C::kStages + s), C::kConsumerWarps + (C::kTc ? 1 : 0));
        }
        mbar_init(base_s + L.cbar, C::kConsumerWarps * 32);
        if constexpr (C::kTc) {
            mbar_init(base_s + L.tcb + kTcQ, C::kConsumerWarps / 2);
            for (int b = 0; b < 2; ++b) {
                mbar_init(base_s + L.tcb + kTcS + 8 * b, 1);
                mbar_init(base_s + L.tcb + kTcP + 8 * b, C::kConsumerWarps / 2);
                mbar_init(base_s + L.tcb + kTcPV + 8 * b, 1);
                mbar_init(base_s + L.tcb + kTcG + 8 * b, C::kConsumerWarps / 2 * 32);
            }
            mbar_init(base_s + L.tcb + kTcFin, 1);
        }
        fence_mbar_init();
        abort_flag = 0;
    }
    if (tid == C::kConsumerWarps * 32) {
        prefetch_tensormap(&p.tm_k);
        prefetch_tensormap(&p.tm_v);
    }
    if (warp == C::kMainThreads / 32) {  // the prefetch warp: joins nothing below
        // (not in the two-q-tile row forms: the call alone costs its main loop
        // registers, and its consumers set its time)
        if constexpr (MODE != kGather && MODE != kMultiRows32 && !C::kTc)
            if (!early && p.prefetch) prefetch_first_stages<D, ST, MODE>(p, lane);
        return;
    }
    if constexpr (C::kTc) {
        if (warp == C::kConsumerWarps + 1) {  // the MMA warp holds the tensor memory
            tmem_alloc(base_s + L.tcb + kTcSlot, C::kTmemCols);
            tmem_relinquish();
            tc_fence_before();
        }
    }
    if (!early) {
        pdl_wait_primary();
        if (MODE != kGather) pdl_launch_dependents();
    }
    // ends with the main warps' barrier (which also publishes the stage barriers)
    const int32_t nv_max = build_prefix<is_multi(MODE), C::kMainThreads>(p, pfx, scan);
    int64_t begin, end;
    const GroupRange gr = cta_range<MODE>(p, pfx, nv_max, C::kST, &begin, &end);

    if (warp == C::kConsumerWarps) {
        run_producer<D, ST, MODE>(p, base_s, L, pfx, meta, &abort_flag, begin, end, lane);
        return;
    }
    if constexpr (C::kTc) {
        // the softmax warps and the MMA warp meet once more before the tensor
        // memory is freed (named barrier 2: 4 + 1 warps)
        tc_fence_after();
        const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base + L.tcb + kTcSlot);
        if (warp == C::kConsumerWarps + 1) {
            if (lane == 0) run_mma_tc<D, ST, MODE>(p, base_s, L, meta, &abort_flag, tmem);
            __syncwarp();
            asm volatile("bar.sync 2, %0;" ::"n"((C::kConsumerWarps + 1) * 32) : "memory");
            tc_fence_after();
            tmem_dealloc(tmem, C::kTmemCols);
        } else {
            run_consumer_tc<D, ST, MODE>(p, base_s, base, L, meta, pfx, &abort_flag, warp, lane, tmem);
            asm volatile("bar.sync 2, %0;" ::"n"((C::kConsumerWarps + 1) * 32) : "memory");
        }
    } else if constexpr (q_tiles(MODE) > 0) {
        run_consumer_rows<D, ST, MODE>(p, base_s, base, L, meta, pfx, &abort_flag, warp, lane);
    } else {
        run_consumer<D, ST, MODE>(p, base_s, base, L, meta, pfx, gr, &abort_flag, warp, lane);
    }
}

// Host side of one split-kernel shape: its entry points by mode, their
// pipeline depth and their launch (programmatic stream serialization: the
// prologue may overlap the previous kernel; the kernel waits with
// griddepcontrol.wait before reading global memory).  The row forms of
// multi-query (mma.sync and tcgen05) exist for 64-row stages at head sizes up
// to 128.
template <int D, int ST>
constexpr bool has_rows_form() { return ST == 64 && D <= 128; }
template <int D, int ST>
constexpr bool has_tc_form() { return ST == 64 && D == 128; }

template <int D, int ST>
const void* split_fn_of(int mode) {
    switch (mode) {
        case kOneShot: return reinterpret_cast<const void*>(&split_kernel<D, ST, kOneShot>);
        case kTiled: return reinterpret_cast<const void*>(&split_kernel<D, ST, kTiled>);
        case kGather: return reinterpret_cast<const void*>(&split_kernel<D, ST, kGather>);
        case kMulti: return reinterpret_cast<const void*>(&split_kernel<D, ST, kMulti>);
        case kMultiRows16:
            if constexpr (has_rows_form<D, ST>())
                return reinterpret_cast<const void*>(&split_kernel<D, ST, kMultiRows16>);
            return nullptr;
        case kMultiRows32:
            if constexpr (has_rows_form<D, ST>())
                return reinterpret_cast<const void*>(&split_kernel<D, ST, kMultiRows32>);
            return nullptr;
        case kMultiTc:
            if constexpr (has_tc_form<D, ST>())
                return reinterpret_cast<const void*>(&split_kernel<D, ST, kMultiTc>);
            return nullptr;
        default: return nullptr;
    }
}

template <int D, int ST>
int split_stages_of(int mode) {
    if (q_tiles(mode) > 0 && !has_rows_form<D, ST>()) return 0;
    switch (mode) {
        case kMultiRows16: return Cfg<D, ST, has_rows_form<D, ST>() ? kMultiRows16 : kOneShot>::kStages;
        case kMultiRows32: return Cfg<D, ST, has_rows_form<D, ST>() ? kMultiRows32 : kOneShot>::kStages;
        case kMultiTc: return has_tc_form<D, ST>() ? Cfg<D, ST, has_tc_form<D, ST>() ? kMultiTc : kOneShot>::kStages : 0;
        default: return Cfg<D, ST, kOneShot>::kStages;
    }
}

template <int D, int ST, int MODE>
cudaError_t launch_split_mode(const SplitParams& p, int grid, size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    // the prefetch warp is launched only when the call prefetches
    cfg.blockDim = dim3(p.prefetch ? Cfg<D, ST, MODE>::kThreads : Cfg<D, ST, MODE>::kMainThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_kernel<D, ST, MODE>, p);
}

template <int D, int ST>
cudaError_t launch_split_of(int mode, const SplitParams& p, int grid, size_t smem, cudaStream_t stream) {
    switch (mode) {
        case kOneShot: return launch_split_mode<D, ST, kOneShot>(p, grid, smem, stream);
        case kTiled: return launch_split_mode<D, ST, kTiled>(p, grid, smem, stream);
        case kGather: return launch_split_mode<D, ST, kGather>(p, grid, smem, stream);
        case kMulti: return launch_split_mode<D, ST, kMulti>(p, grid, smem, stream);
        case kMultiRows16:
            if constexpr (has_rows_form<D, ST>()) return launch_split_mode<D, ST, kMultiRows16>(p, grid, smem, stream);
            return cudaErrorInvalidValue;
        case kMultiRows32:
            if constexpr (has_rows_form<D, ST>()) return launch_split_mode<D, ST, kMultiRows32>(p, grid, smem, stream);
            return cudaErrorInvalidValue;
        case kMultiTc:
            if constexpr (has_tc_form<D, ST>()) return launch_split_mode<D, ST, kMultiTc>(p, grid, smem, stream);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pda
