// pda_plan.h -- the split plan shared by the host API and the kernels.
//
// The work of one call is the flattened index space of W plan blocks ordered
// (sequence b, kv head g, block j): unit u = b*Hkv + g owns the W-range
// [pfx[b]*Hkv + g*nv_b, pfx[b]*Hkv + (g+1)*nv_b), where nv_b = nb_b + c for a
// sequence of nb_b > 0 blocks (0 for an empty one) and pfx is the exclusive
// prefix sum of nv.  The first nb_b positions of a unit are its blocks; the c
// after them are a cost placeholder read by nobody: every segment takes a
// fixed time beyond its blocks (its partial last stage, the consumer warps'
// state merge and store, the next unit's q rows), and counting that cost in
// the plan gives a CTA that covers many short units fewer blocks.  A grid of
// P CTAs splits the range evenly: CTA c takes [floor(c*W/P),
// floor((c+1)*W/P)).  Each maximal run of one unit's blocks inside one CTA's
// range is a "segment" with its own online-softmax state; the state of the
// segment of unit u in CTA c is stored in slot u + c, which is unique because
// moving to the next segment always advances u, c or both.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define PDA_HD __host__ __device__ __forceinline__
#else
#define PDA_HD inline
#endif

namespace pda {

// floor(a / b) for a >= 0, b > 0.  Operands that fit in 32 bits take the
// 32-bit division: a 64-bit division is a long instruction sequence on the GPU.
PDA_HD int64_t div_floor(int64_t a, int64_t b) {
    if (((uint64_t)a | (uint64_t)b) <= 0xffffffffull) return (int64_t)((uint32_t)a / (uint32_t)b);
    return a / b;
}

// First flattened block of CTA c.
PDA_HD int64_t cta_begin(int64_t c, int64_t W, int64_t P) { return div_floor(c * W, P); }

// The CTA whose range contains flattened block s (0 <= s < W): the largest c
// with floor(c*W/P) <= s, i.e. floor(((s+1)*P - 1) / W).
PDA_HD int64_t cta_of_block(int64_t s, int64_t W, int64_t P) { return div_floor((s + 1) * P - 1, W); }

// Grouped split, for several causal queries per sequence: the launch's B
// sequences form Q equal groups (group g = sequences [g*B/Q, (g+1)*B/Q), in
// the same sequence order), each walked by its own P/Q CTAs over its own
// flattened range [F_g, F_{g+1}), F_g = pfx[g*B/Q]*Hkv.  Every group visits
// the same (sequence, kv head, block) positions at nearly the same time.
// With Q = 1 this is the plain split above.  CTAs past Q*(P/Q) stay idle.
struct GroupRange {
    int64_t F0;   // first flattened block of the group
    int64_t W;    // blocks of the group
    int64_t Pg;   // CTAs of the group
    int64_t g;    // group index (>= Q for an idle CTA)
};

template <typename Pfx>
PDA_HD GroupRange group_of_cta(int64_t c, const Pfx& pfx, int64_t B, int64_t Q, int64_t Hkv,
                               int64_t P) {
    GroupRange r;
    r.Pg = div_floor(P, Q);
    r.g = div_floor(c, r.Pg);
    if (r.g >= Q) { r.F0 = 0; r.W = 0; return r; }
    const int64_t Bg = div_floor(B, Q);
    r.F0 = (int64_t)pfx[r.g * Bg] * Hkv;
    r.W = (int64_t)pfx[(r.g + 1) * Bg] * Hkv - r.F0;
    return r;
}

// Flattened range [begin, end) of CTA c within its group (empty when idle).
PDA_HD void group_cta_range(const GroupRange& r, int64_t c, int64_t* begin, int64_t* end) {
    if (r.W == 0) { *begin = *end = r.F0; return; }
    const int64_t cl = c - r.g * r.Pg;
    *begin = r.F0 + cta_begin(cl, r.W, r.Pg);
    *end = r.F0 + cta_begin(cl + 1, r.W, r.Pg);
}

// The pieces of a unit split across CTAs: the CTAs of its group that hold
// its blocks (the cost positions after them belong to no piece).  With
// W >= Pg every CTA range is non-empty, so the pieces are the CTAs cf .. cl
// between the owners of the unit's first and last block; with W < Pg a CTA
// holds at most one block, so piece i is the owner of block su + i.  The
// piece in CTA c keeps its partial state in slot u + c.
struct UnitPieces {
    int64_t cf;   // CTA of the first piece
    int64_t su;   // the unit's first flattened block
    int32_t n;    // pieces (1: the unit lies in one CTA)
    bool every;   // the pieces are the CTAs cf .. cf + n - 1
};

template <typename Pfx>
PDA_HD UnitPieces unit_pieces(const Pfx& pfx, int64_t b, int64_t kvh, int64_t Hkv, int32_t unit_cost,
                              const GroupRange& gr);

// CTA of piece i of a unit.
PDA_HD int64_t piece_cta(const UnitPieces& u, int64_t i, const GroupRange& gr) {
    return u.every ? u.cf + i : gr.g * gr.Pg + cta_of_block(u.su + i - gr.F0, gr.W, gr.Pg);
}

// Plan blocks c added to every non-empty unit: a segment's fixed cost in
// quarter stages, measured per loader and form (each value the fastest of a
// sweep on ragged and uniform batches).  TMA block boxes: two stages.  Row
// gathers of blocks below 8 tokens, whose stages take longer: half a stage.
// Causal multi-query, n8 form, whose CTAs cover about q_len times more
// segments and read most stages from L2: four stages.  Row form (q rows as
// the MMA's M), whose segments end in a merge of 16 or 32 q rows: four
// stages with one q tile, six with two.  Tile steps of block boxes, whose
// segments end in a fold into the running state: six stages.
constexpr int32_t kUnitCostX4 = 8;
constexpr int32_t kUnitCostGatherX4 = 2;
constexpr int32_t kUnitCostMultiX4 = 16;
constexpr int32_t kUnitCostRows16X4 = 16;
constexpr int32_t kUnitCostRows32X4 = 24;
constexpr int32_t kUnitCostTiledX4 = 24;
// Cost classes of unit_cost_blocks.
enum UnitCostClass : int32_t { kCostDecode = 0, kCostMultiN8 = 1, kCostRows16 = 2, kCostRows32 = 3, kCostTiled = 4 };

// Whether a block's rows are loaded with one TMA box per block and pool: a
// block of bs rows of D bf16 lands as [D/64 slabs][bs rows][128 bytes] and
// must fill whole 1024-byte spans of the 128-byte swizzle, so that every box
// starts on a span (block sizes from 8; 4 for head sizes from 128; 2 for head
// size 256).  Otherwise the rows are gathered one by one.
PDA_HD bool block_boxes(int32_t head_dim, int32_t block_size) {
    return block_size >= 8 || (block_size * head_dim * 2) % 1024 == 0;
}

PDA_HD int32_t unit_cost_blocks(int32_t stage_rows, int32_t head_dim, int32_t block_size, int32_t cost_class) {
    const int32_t nb = stage_rows / block_size;
    const bool boxes = block_boxes(head_dim, block_size);
    const int32_t x4 = cost_class == kCostMultiN8 ? kUnitCostMultiX4
                     : cost_class == kCostRows16 ? kUnitCostRows16X4
                     : cost_class == kCostRows32 ? kUnitCostRows32X4
                     : cost_class == kCostTiled && boxes ? kUnitCostTiledX4
                     : boxes ? kUnitCostX4 : kUnitCostGatherX4;
    return (nb < 1 ? 1 : nb) * x4 / 4;
}

// Small batches ("unit mode").  When there are no more units than CTAs and no
// unit holds more than kUnitModeStages stages of rows, CTA c processes unit c
// whole: no unit is split and nothing merges (splitting units of a few stages
// over many CTAs would buy no bandwidth and cost a merge each).  Otherwise the
// flattened range is split evenly over all CTAs.
constexpr int32_t kUnitModeStages = 4;
PDA_HD bool unit_mode(int64_t units, int64_t ctas, int32_t max_unit_blocks, int32_t stage_rows,
                      int32_t block_size) {
    return units <= ctas && (int64_t)max_unit_blocks * block_size <= (int64_t)kUnitModeStages * stage_rows;
}

// Plan blocks of a unit with nb blocks.
PDA_HD int32_t plan_blocks(int32_t nb, int32_t unit_cost) { return nb > 0 ? nb + unit_cost : 0; }

// Blocks of a unit with nv plan blocks.
PDA_HD int32_t real_blocks(int32_t nv, int32_t unit_cost) { return nv > 0 ? nv - unit_cost : 0; }

// Blocks needed for a length in tokens.
PDA_HD int32_t blocks_for_tokens(int32_t len, int32_t block_size) {
    return len <= 0 ? 0 : (len + block_size - 1) / block_size;
}

template <typename Pfx>
PDA_HD UnitPieces unit_pieces(const Pfx& pfx, int64_t b, int64_t kvh, int64_t Hkv, int32_t unit_cost,
                              const GroupRange& gr) {
    const int32_t lo = pfx[b], hi = pfx[b + 1];
    const int32_t nb = real_blocks(hi - lo, unit_cost);
    UnitPieces r;
    r.su = (int64_t)lo * Hkv + kvh * (hi - lo);
    const int64_t eu = r.su + nb;
    r.cf = gr.g * gr.Pg + cta_of_block(r.su - gr.F0, gr.W, gr.Pg);
    const int64_t cl = gr.g * gr.Pg + cta_of_block(eu - 1 - gr.F0, gr.W, gr.Pg);
    r.every = gr.W >= gr.Pg;
    r.n = (int32_t)(r.every ? cl - r.cf + 1 : nb);
    return r;
}

}  // namespace pda
