// pda_params.h -- kernel parameter blocks and the shared-memory layout of the
// split kernel (shared by the kernels and the host API).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pda_plan.h"

namespace pda {

// Split-kernel shape: a pipeline stage holds ST KV rows, read by ST / 16
// consumer warps of 16 rows; one more warp is the TMA producer.  ST = 64,
// except for head_dim 256 with rows gathered one by one (block size 1): there
// the producer copies rows (4 per gather4 copy, or 16-byte cp.async) and is
// bound by its instruction rate, and with 64-row stages only one CTA (one
// producer) fits on an SM; ST = 32 fits two.  (For head_dim 128, already two
// CTAs per SM, 32-row stages were measured slower.)
constexpr int kMaxLaunchBatch = 1024;                    // sequences per kernel launch
constexpr int kMaxGroup = 8;                             // q heads per kv head (n8 MMA)
constexpr int kMaxRowsPerWalk = 32;                      // q rows one KV walk serves (row form)

// kOneShot: decode, output written; kTiled: fold a tile into the running
// state; kGather: copy the staged rows out (loader check); kMulti: causal
// multi-query decode, output written (the other modes see one query per
// sequence, known at compile time).  kMulti packs at most 8 q rows (queries
// x G heads) into the MMA's N (the n8 form).  kMultiRows16 / kMultiRows32
// are the row form for head sizes up to 128: the packed q rows are the MMA's
// M, in one or two tiles of 16 rows, so that one walk over the KV serves up
// to 32 q rows.  kMultiTc is the row form of 32 q rows on the tcgen05
// tensor cores: accumulators in tensor memory, one thread issues the MMAs.
enum Mode : int {
    kOneShot = 0, kTiled = 1, kGather = 2, kMulti = 3, kMultiRows16 = 4, kMultiRows32 = 5, kMultiTc = 6
};
constexpr int kNumModes = 7;
__host__ __device__ constexpr bool is_multi(int mode) {
    return mode == kMulti || mode == kMultiRows16 || mode == kMultiRows32 || mode == kMultiTc;
}
__host__ __device__ constexpr bool is_tc(int mode) { return mode == kMultiTc; }
__host__ __device__ constexpr bool writes_output(int mode) { return mode == kOneShot || is_multi(mode); }
// 16-row q tiles of the row form (0: the n8 form); the tcgen05 form's segment
// end merges its 32 rows in two such tiles.
__host__ __device__ constexpr int q_tiles(int mode) {
    return mode == kMultiRows16 ? 1 : (mode == kMultiRows32 || mode == kMultiTc) ? 2 : 0;
}
// q rows a stage's q area holds.
__host__ __device__ constexpr int stage_q_rows(int mode) { return q_tiles(mode) ? 16 * q_tiles(mode) : kMaxGroup; }
// Consumer warps: one per 16 KV rows of a stage, times the q tiles in the
// mma.sync row form; the tcgen05 form's eight softmax warps, two groups (even
// and odd stages) of one per 16-row token slice and tensor-memory lane
// quarter.
__host__ __device__ constexpr int consumer_warps(int st, int mode) {
    return is_tc(mode) ? 8 : (st / 16) * (q_tiles(mode) ? q_tiles(mode) : 1);
}
constexpr int kMaxConsumerWarps = 8;
// Threads of a split CTA as launched at most: the consumer warps, the
// producer warp and the prefetch warp (the tcgen05 form: the MMA warp
// instead; it launches no prefetch warp).
PDA_HD int split_threads(int st, int mode) { return (consumer_warps(st, mode) + 2) * 32; }
// Stage rows for a head size and block size.
PDA_HD int stage_tokens(int D, int block_size) { return D == 256 && !block_boxes(D, block_size) ? 32 : 64; }
// Sequences (launch rows) per launch of a mode: the row form with one q tile
// runs two CTAs per SM with three 36 KB stages at head size 128, the tcgen05
// form one CTA with five 40 KB stages, which leaves room for a 512-entry
// block prefix.
PDA_HD int max_launch_rows(int mode) { return (mode == kMultiRows16 || mode == kMultiTc) ? 512 : kMaxLaunchBatch; }
// The unit-cost class of a mode (pda_plan.h).
PDA_HD int32_t cost_class(int mode) {
    return mode == kMulti ? kCostMultiN8 : mode == kMultiRows16 ? kCostRows16
         : (mode == kMultiRows32 || mode == kMultiTc) ? kCostRows32 : mode == kTiled ? kCostTiled : kCostDecode;
}

// Per-stage record the producer writes before arming the stage's barrier.
struct StageMeta {
    int32_t b;        // sequence
    int32_t kvh;      // kv head
    int32_t n_valid;  // valid rows (a prefix of the stage's 64 rows)
    int32_t flags;    // kSegBegin | kSegEnd | kWholeUnit | kDone
    int32_t slot;     // partial-state slot of the segment (u + c)
    int32_t j0;       // index of the stage's first block within the sequence
    int32_t lim;      // causal limit of the row's first query (token index)
    int32_t nr;       // q rows of the unit (packed queries x G)
};
enum MetaFlags : int32_t { kSegBegin = 1, kSegEnd = 2, kWholeUnit = 4, kDone = 8 };

struct SplitParams {
    CUtensorMap tm_k;            // K pool, 5-D {64, bs, D/64, Hkv, num_blocks}, box {64, bs, D/64, 1, 1};
                                 // for gather4 2-D {D, rows}, box {64, 1}
    CUtensorMap tm_v;            // V pool, same shape
    CUtensorMap tm_k1;           // head size 128, tcgen05 form: box {64, bs, 1, 1, 1} (one slab), so
    CUtensorMap tm_v1;           // that a stage tile is [slab][64 rows][128 B]
    const uint16_t* q;           // [B, Hq, D] bf16
    const int32_t* table;        // [B, table_stride] block ids; null = contiguous cache
    const int32_t* lens;         // [B] tokens (one-shot) or block counts (tiled)
    const int32_t* last_valid;   // [B] valid slots of the last listed block (tiled) or null
    uint16_t* out;               // [B, Hq, D] bf16 (one-shot)
    float* out_f32;              // [B, Hq, D] fp32 instead of out when non-null
    float* part_o;               // [slots, rows_per_slot, D]
    float* part_ml;              // [slots, rows_per_slot, 2] (m in base-2 units, l)
    int32_t* unit_sync;          // [B*Hkv][2] per split unit: pieces that drew a ticket, pieces
                                 // whose partial state is stored (0 between launches)
    float* m_state;              // tiled: running state [B*Hq], [B*Hq], [B*Hq*D]
    float* l_state;
    float* o_state;
    uint32_t* err;               // device error flags
    uint16_t* dbg_k;             // gather check outputs
    uint16_t* dbg_v;
    const uint16_t* k_base;      // pool base pointers and element strides, for the
    const uint16_t* v_base;      // row-gather loader (block sizes below 8)
    int64_t blk_s, tok_s, kvh_s;
    int64_t num_blocks;
    int32_t table_stride;
    int32_t row_gather;          // 0: one 5-D TMA box per block; rows one by one: 1: TMA
                                 // gather4; 2: 16-byte cp.async
    int64_t row_blk, row_tok, row_kvh;  // strides in rows of D elements (gather4)
    int32_t lens_are_blocks;
    int32_t q_len;               // causal queries per sequence (0 or 1: plain decode)
    int32_t qp;                  // queries packed into one launch row (qp*G q rows: <= 8 in
                                 // the n8 form, <= 32 in the row form)
    int32_t rows_per_slot;       // rows of a partial-state slot (0: G)
    int32_t B, Hq, Hkv, G, bs;
    int32_t unit_cost;           // plan blocks added to every non-empty unit
    int32_t dbg_row_tokens;      // tokens per (b, kvh) row of the gather output
    int32_t prefetch;            // speculative L2 prefetch of the first stages before the wait
    int32_t early_inputs;        // tiled: read the inputs before the previous kernel completes
                                 // (a tile step right behind another of the same step)
    float scale_log2;            // softmax scale * log2(e)
};

struct SmemLayout {
    uint32_t bars, cbar, tcb, tcx, meta, scan, st_m, st_l, st_x, pfx, total;
};

// K and V tiles of ST rows plus the stage's q rows (stage_q_rows x D bf16).
PDA_HD uint32_t stage_bytes(int D, int st, int mode) {
    return 2u * (uint32_t)(D / 64) * (uint32_t)st * 128u + (uint32_t)stage_q_rows(mode) * D * 2u;
}

// Dynamic shared memory of the split kernel (the +1024 pays for aligning the
// base to the 128-byte-swizzle atom).  The segment epilogue stages its o tiles
// in the finished stage: n8 form, ST/16 warps x 8 rows x (D+4) floats <=
// 2 * ST * D * 2 bytes; row form, one q tile at a time, ST/16 warps x 16 rows
// x (D+4) floats <= the stage with its q area.  st_m / st_l hold one (m, l)
// per consumer warp and q row: [ST/16 token slices][32 rows] in the row form.
PDA_HD SmemLayout smem_layout(int D, int st, int mode, int stages, int B) {
    SmemLayout L;
    uint32_t off = (uint32_t)stages * stage_bytes(D, st, mode);
    L.bars = off;  off += 2u * stages * 8u;
    L.cbar = off;  off += 8u;
    L.tcb = off;   off += is_tc(mode) ? 96u : 0u;  // tcgen05 form: 10 barriers, the tensor-memory base
    // tcgen05 form: row maxima of the slices [group][2][4][32], weight sums [8 warps][32]
    L.tcx = off;   off += is_tc(mode) ? (2u * 2u * 4u + 8u) * kMaxRowsPerWalk * 4u : 0u;
    L.meta = off;  off += (uint32_t)stages * (uint32_t)sizeof(StageMeta);
    L.scan = off;  off += 128u;  // per warp: block-prefix sum [16], largest unit [16]
    L.st_m = off;  off += 4u * kMaxRowsPerWalk * 4u;
    L.st_l = off;  off += 4u * kMaxRowsPerWalk * 4u;
    L.st_x = off;  off += 2u * kMaxGroup * 4u + 16u;  // old running (m, l) of a unit's rows; role word
    L.pfx = off;   off += (uint32_t)(B + 1) * 4u;
    L.total = off + 1024u;
    return L;
}

}  // namespace pda
