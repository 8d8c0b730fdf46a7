/*
 * pda.h -- paged grouped-query decode attention on GB300 (sm_103a): C ABI.
 *
 * One query token per sequence attends over a bf16 KV cache scattered across
 * a pool of fixed-size blocks and addressed through a per-sequence block
 * table.  The KV walk is split into tiles; each tile keeps an fp32
 * online-softmax state (m, l, o); a separate merge/finalize step combines the
 * states and writes o / l as bf16.
 *
 * Sources (page title, then section or item):
 *   [TA]  tiled_attention.rs (spark_storage) -- the (m, l, o) lifecycle
 *         begin_step / step_tile / finalize, TiledAttentionDims, its
 *         validate() checks, the state sizes and paged_strides /
 *         scratch_pool_strides.
 *   [CK]  AstrAI "CUDA Kernels" -- Overview (split-KV paged decode),
 *         Python Wrappers (scale 1/sqrt(head_dim); wrappers fail loudly when
 *         the compiled library is missing).
 *
 * Conventions for every call below:
 *   - Pointers named q, k_pool, v_pool, out, tile_*, block_table, seq_lens
 *     are DEVICE pointers owned by the caller; the library never frees them.
 *     bf16 tensors are passed as raw 16-bit patterns (pda_bf16).
 *   - q, k_pool, v_pool and out must be 16-byte aligned; int32 arrays
 *     4-byte aligned.
 *   - stream is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call that takes a stream only enqueues work and returns; argument
 *     errors are returned at once, kernel launch errors when they are
 *     detected at enqueue time.  Device-side data errors (a block id outside
 *     [0, num_blocks), a length beyond the table width) never fault: they
 *     set a flag read by pda_read_device_errors().
 *   - All state belongs to the pda_ctx.  Calls on one context must be
 *     ordered (one stream, or explicit events); use one context per
 *     concurrent stream.  A context also keeps the TMA descriptors of the
 *     last KV pool it read (pointers, block count and strides); a call with
 *     another pool re-encodes them, so neither calls nor host threads may
 *     share a context concurrently.
 *   - Errors: every call returns a pda_status; pda_last_error() gives the
 *     message of the last failed call on the calling thread.
 */
#ifndef PDA_H
#define PDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PDA_ABI_VERSION 5

typedef struct pda_ctx pda_ctx;
typedef void* pda_stream;      /* cudaStream_t */
typedef uint16_t pda_bf16;     /* bf16 bit pattern */
typedef int32_t pda_status;

enum {
    PDA_OK = 0,
    PDA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or stride   */
    PDA_ERR_UNSUPPORTED = 2,   /* valid per [TA] but not built (see pda_create) */
    PDA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed             */
    PDA_ERR_NO_DEVICE = 4,     /* no usable sm_103 device is current            */
    PDA_ERR_DEVICE_DATA = 5    /* pda_read_device_errors() found a flag set      */
};

/* Device-side flags (bit mask) reported by pda_read_device_errors(). */
#define PDA_DEVERR_BAD_BLOCK_ID 0x1u  /* a listed block id was outside [0, num_blocks); that
                                         block's rows read as zeros                       */
#define PDA_DEVERR_BAD_LENGTH   0x2u  /* seq_len < 0, a length beyond table width * block
                                         size, or a tile count outside [0, tile_capacity];
                                         the length was clamped                           */
#define PDA_DEVERR_TIMEOUT      0x4u  /* a bounded wait inside a kernel gave up (the kernel
                                         returned early; its output is not valid)         */

/*
 * Static sizes a context is built for -- [TA] TiledAttentionDims.
 *   max_seqs       most sequences one call may carry (>= 1).
 *   num_q_heads    Hq; must be a multiple of num_kv_heads ([TA] validate).
 *   num_kv_heads   Hkv.  The group size G = Hq / Hkv ([TA] gqa_ratio) must be
 *                  1..8 in this build.  q head h reads KV head h / G.
 *   head_dim       D; [TA] validate caps it at 256; this build has kernels for
 *                  64, 128 and 256.
 *   block_size     tokens per KV block: 1, 2, 4, 8, 16, 32 or 64 in this build
 *                  (one TMA copy per block and pool when a block's rows fill
 *                  whole 1024-byte swizzle spans: block sizes from 8, 4 with
 *                  head_dim 128 or 256, 2 with head_dim 256; otherwise the
 *                  rows are gathered, four per TMA gather4 copy when the pool
 *                  strides are multiples of head_dim, else with 16-byte
 *                  copies).  block_size 1 is the token-granular page of [CK]
 *                  Attention Backend.
 *   tile_capacity  most block ids per sequence in one pda_step_tile call.
 */
typedef struct pda_dims {
    int32_t max_seqs;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    int32_t tile_capacity;
} pda_dims;

/* Library ABI version (PDA_ABI_VERSION). Host only. */
int32_t pda_abi_version(void);

/* Static text for a status code. Host only. */
const char* pda_status_string(pda_status status);

/* Message of the last failed call on this thread ("" if none). Host only. */
const char* pda_last_error(void);

/*
 * Checks dims without touching the GPU -- [TA] TiledAttentionDims::validate
 * (Hq % Hkv == 0, head_dim <= 256) plus this build's supported set.
 * Returns PDA_ERR_INVALID_ARG for dims [TA] rejects, PDA_ERR_UNSUPPORTED for
 * dims [TA] accepts that have no kernel here.
 */
pda_status pda_check_dims(const pda_dims* dims);

/*
 * Element-stride triples (block, token, kv-head), in bf16 elements, of the two
 * pool layouts -- [TA] paged_strides and scratch_pool_strides:
 *   paged: [num_blocks, block_size, Hkv, D]        -> (bs*Hkv*D, Hkv*D, D)
 *   slot : [slot, K|V, Hkv, block_size, D]         -> (2*Hkv*bs*D, D, bs*D)
 * In the slot layout the V pool pointer is the K pool pointer + Hkv*bs*D.
 * Host only; out receives 3 values.
 */
pda_status pda_paged_strides(const pda_dims* dims, int64_t out[3]);
pda_status pda_slot_strides(const pda_dims* dims, int64_t out[3]);

/*
 * Creates a context on the CURRENT CUDA device -- [TA] TiledAttention::new.
 * Allocates the fp32 running state m, l [max_seqs*Hq] and o [max_seqs*Hq*D]
 * ([TA] m_bytes / l_bytes / o_bytes) and the split workspace; they are reused
 * by every later call and freed by pda_destroy.  Fails with
 * PDA_ERR_NO_DEVICE when the current device is not compute capability 10.3.
 */
pda_status pda_create(const pda_dims* dims, pda_ctx** out_ctx);

/* Frees the context and its device buffers (synchronises the device first). */
void pda_destroy(pda_ctx* ctx);

/*
 * One-shot decode:
 *   out[b, h, :] = softmax(scale * q[b, h, :] . K_t) V_t  over t < seq_lens[b],
 * where K_t / V_t is row (block_table[b, t / bs], t % bs, h / G) of k_pool /
 * v_pool ([CK] Overview: paged split-KV decode; the result equals the
 * finalize of [TA]'s state after all blocks).
 *   q            [batch, Hq, D] bf16, dense.
 *   k_pool,
 *   v_pool       [num_blocks, block_size, Hkv, D] bf16, dense ([TA] paged layout).
 *   block_table  [batch, max_blocks] int32; only the first
 *                ceil(seq_lens[b] / bs) entries of row b are read.
 *   seq_lens     [batch] int32 token counts (device); 0 gives a zero row.
 *   scale        softmax scale; NaN selects the default 1/sqrt(D) ([CK]).
 *   out          [batch, Hq, D] bf16, written completely.
 *   batch        0 .. max_seqs (0 returns PDA_OK without launching).
 * The work is split over the flattened (sequence, kv head, block) space so
 * every SM gets an equal share (its blocks plus a fixed cost per unit it
 * covers; see pda_plan_units), whatever the lengths; no host copy of
 * seq_lens is needed and the call can be captured in a CUDA graph.
 */
pda_status pda_decode(pda_ctx* ctx, const pda_bf16* q, const pda_bf16* k_pool,
                      const pda_bf16* v_pool, int64_t num_blocks,
                      const int32_t* block_table, int32_t max_blocks,
                      const int32_t* seq_lens, int32_t batch, float scale,
                      pda_bf16* out, pda_stream stream);

/*
 * pda_decode with an explicit pool stride triple (block, token, kv-head) in
 * bf16 elements, e.g. pda_slot_strides() -- [TA] step_tile's stride triple.
 * Each stride must be a positive multiple of 8; rows stay D-contiguous.
 */
pda_status pda_decode_strided(pda_ctx* ctx, const pda_bf16* q, const pda_bf16* k_pool,
                              const pda_bf16* v_pool, int64_t num_blocks,
                              int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride,
                              const int32_t* block_table, int32_t max_blocks,
                              const int32_t* seq_lens, int32_t batch, float scale,
                              pda_bf16* out, pda_stream stream);

/*
 * Decode over a contiguous (unpaged) cache -- [CK] Overview (attn_decode:
 * GQA decode over a contiguous KV cache) and Python Wrappers (layout
 * [batch, seq_len, n_heads, head_dim]).  It is the paged kernel with the
 * identity block table: token t of sequence b is row (b, t) of
 *   k, v         [batch, max_seq_len, Hkv, D] bf16, dense;
 * max_seq_len must be a multiple of the context's block_size; seq_lens[b]
 * (device) <= max_seq_len tokens are read.  q, out and scale as pda_decode;
 * batch <= min(max_seqs, 1024).
 */
pda_status pda_decode_contiguous(pda_ctx* ctx, const pda_bf16* q, const pda_bf16* k,
                                 const pda_bf16* v, int32_t max_seq_len,
                                 const int32_t* seq_lens, int32_t batch, float scale,
                                 pda_bf16* out, pda_stream stream);

/*
 * Multi-query decode with a causal mask (speculative verify, short prefill
 * chunks) -- [CK] Overview (attn_paged_decode / attn_paged_prefill) and
 * Python Wrappers (is_causal).  The last q_len tokens of each sequence are the
 * queries: query i of sequence b is token seq_lens[b] - q_len + i and attends
 * to tokens 0 .. seq_lens[b] - q_len + i of the paged cache (which already
 * holds the new tokens' K/V).  A sequence shorter than q_len gives its first
 * queries fewer (or no) tokens; no tokens give a zero row.
 *   q, out   [batch, q_len, Hq, D] bf16, dense.
 *   seq_lens [batch] total tokens per sequence (device).
 *   batch * q_len <= max_seqs; other arguments as pda_decode.
 * The queries of a sequence are packed G q heads each into launch rows, each
 * row split over the GPU like a sequence of its own with one walk over the
 * sequence's KV: up to 8 q rows per walk with the q rows as the MMA's N
 * ("n8 form"); with more than 8 q rows per sequence (q_len * G > 8) and head
 * sizes up to 128, up to 32 per walk with the q rows as the MMA's M ("row
 * form", [CK] Overview: split-Q MMA).  Rows of one sequence read the same
 * blocks at nearly the same time, so repeated walks read mostly from L2.
 * pda_get_multi_info tells the shape a q_len takes.
 */
pda_status pda_decode_multi(pda_ctx* ctx, const pda_bf16* q, const pda_bf16* k_pool,
                            const pda_bf16* v_pool, int64_t num_blocks,
                            const int32_t* block_table, int32_t max_blocks,
                            const int32_t* seq_lens, int32_t batch, int32_t q_len, float scale,
                            pda_bf16* out, pda_stream stream);

/*
 * Tiled lifecycle, step 1 -- [TA] begin_step: resets the running state of
 * sequences 0..num_seqs-1 to (m, l, o) = (-inf, 0, 0).  num_seqs > max_seqs
 * is PDA_ERR_INVALID_ARG.
 */
pda_status pda_begin_step(pda_ctx* ctx, int32_t num_seqs, pda_stream stream);

/*
 * Tiled lifecycle, step 2 -- [TA] step_tile: folds one tile of blocks per
 * sequence into the running state.
 *   tile_blocks        [num_seqs, tile_capacity] int32 block ids; sequence s
 *                      lists tile_block_counts[s] ids (0 leaves its state as it
 *                      is).
 *   tile_last_valid    [num_seqs] int32 in 1..block_size: valid token slots of
 *                      the LAST listed block of each sequence (the other
 *                      listed blocks are full), or NULL when every listed
 *                      block is full.  [TA] passes one scalar for all
 *                      sequences; a per-sequence array also serves ragged
 *                      batches in one call.
 *   blk/tok/kvh_stride pool stride triple in bf16 elements ([TA] paged_strides
 *                      or scratch_pool_strides); positive multiples of 8.
 *   scale              NaN selects 1/sqrt(D).  [TA] passes no scale.
 * Tiles of one step may be given in any order of blocks; the state after all
 * tiles equals the one-shot result up to fp32 rounding.
 *
 * Overlap: a tile step issued right behind another tile step of the same
 * step (same context, same stream) starts reading its inputs -- q, the pools,
 * tile_blocks, tile_block_counts, tile_last_valid -- while the previous one
 * is still finishing, and waits for it only before it touches the running
 * state.  So a kernel that the caller launches between two tile steps of a
 * step on that stream must not write the second step's inputs while
 * triggering its dependents early (programmatic dependent launch); kernels
 * launched without such a trigger, copies and host-side changes between the
 * calls are always waited for.  The first tile step of a step waits for
 * whatever precedes it.  pda_set_tile_overlap(ctx, 0) makes every tile step
 * wait.
 */
pda_status pda_step_tile(pda_ctx* ctx, const pda_bf16* q, const pda_bf16* k_pool,
                         const pda_bf16* v_pool, int64_t num_blocks,
                         const int32_t* tile_blocks, const int32_t* tile_block_counts,
                         const int32_t* tile_last_valid, int32_t num_seqs,
                         int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride,
                         float scale, pda_stream stream);
/* Tile-step overlap on (enable != 0, the default) or off.  Host only. */
pda_status pda_set_tile_overlap(pda_ctx* ctx, int32_t enable);

/*
 * Tiled lifecycle, step 3 -- [TA] finalize: out[s, h, :] = bf16(o / l) for
 * s < num_seqs (round to nearest even); l == 0 (nothing folded) gives zeros.
 * out is [num_seqs, Hq, D].  pda_finalize_f32 writes the same quotient in fp32
 * without rounding (for comparing tiled and one-shot runs).
 */
pda_status pda_finalize(pda_ctx* ctx, pda_bf16* out, int32_t num_seqs, pda_stream stream);
pda_status pda_finalize_f32(pda_ctx* ctx, float* out, int32_t num_seqs, pda_stream stream);

/*
 * Partial states from several contexts -- context-parallel decode, where each
 * context (one per GPU, say) folds a shard of every sequence's blocks with
 * the tiled lifecycle.  [CK] Overview: split-KV partial states combined by a
 * merge; [TA] module comment: the running state (m, l, o).
 *
 * pda_export_state copies the running state of sequences [0, num_seqs) into
 * caller-owned DEVICE buffers m, l [num_seqs*Hq] and o [num_seqs*Hq*D] (fp32,
 * 4-byte aligned), in natural-log units of the scaled scores:
 *   l = sum_t exp(s_t - m),  o = sum_t exp(s_t - m) v_t,
 * s_t = scale * q . K_t over the tokens folded so far ((-inf, 0, 0) when
 * none), where m is the reference the kernels keep: the running max of s_t,
 * or at most 8 ln 2 below it (the reference moves only when the max runs
 * past it by more than that).  o / l and the merge below do not depend on
 * which reference a state was taken against.  num_seqs must be <= max_seqs.
 *
 * pda_merge_states combines n_parts (>= 1) such states per (sequence, q head)
 * row, laid out part-major: m_parts, l_parts [n_parts][num_seqs*Hq] and
 * o_parts [n_parts][num_seqs*Hq*D] (DEVICE; o_parts 16-byte aligned):
 *   M = max_i m_i,  L = sum_i l_i exp(m_i - M),  O = sum_i o_i exp(m_i - M),
 *   out[s, h, :] = bf16(O / L)   (0 when L == 0)
 * into out [num_seqs, Hq, D] (16-byte aligned).  States whose token sets
 * partition a sequence merge to the decode over all of them.
 * pda_merge_states_f32 writes O / L in fp32.  Moving states between devices
 * (an all-gather of Hq*(D+2)*4 bytes per sequence and part) is the caller's;
 * the Python binding has one over torch.distributed (gather_states).
 */
pda_status pda_export_state(pda_ctx* ctx, int32_t num_seqs, float* m, float* l, float* o,
                            pda_stream stream);
pda_status pda_merge_states(pda_ctx* ctx, int32_t n_parts, int32_t num_seqs, const float* m_parts,
                            const float* l_parts, const float* o_parts, pda_bf16* out,
                            pda_stream stream);
pda_status pda_merge_states_f32(pda_ctx* ctx, int32_t n_parts, int32_t num_seqs,
                                const float* m_parts, const float* l_parts, const float* o_parts,
                                float* out, pda_stream stream);

/*
 * One-shot decode writing the fp32 quotient o / l instead of bf16 (same
 * arguments as pda_decode_strided; out is [batch, Hq, D] float).  Used to
 * compare the one-shot and tiled paths before output rounding.
 */
pda_status pda_decode_f32(pda_ctx* ctx, const pda_bf16* q, const pda_bf16* k_pool,
                          const pda_bf16* v_pool, int64_t num_blocks,
                          int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride,
                          const int32_t* block_table, int32_t max_blocks,
                          const int32_t* seq_lens, int32_t batch, float scale,
                          float* out, pda_stream stream);

/*
 * Gather check: runs the decode kernel's own loader (block-table lookup, TMA
 * copies into shared memory, per-stage masking) and writes every valid K and
 * V row it staged to k_rows / v_rows, laid out [batch, Hkv, max_blocks*bs, D]
 * bf16 (token t of sequence b, kv head g at ((b*Hkv + g)*max_blocks*bs + t)*D).
 * Rows past seq_lens[b] are left untouched.  Same pool arguments as
 * pda_decode_strided.
 */
pda_status pda_debug_gather(pda_ctx* ctx, const pda_bf16* k_pool, const pda_bf16* v_pool,
                            int64_t num_blocks, int64_t blk_stride, int64_t tok_stride,
                            int64_t kvh_stride, const int32_t* block_table,
                            int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                            pda_bf16* k_rows, pda_bf16* v_rows, pda_stream stream);

/*
 * Reads (and with clear != 0 resets) the device error flags of this context
 * (PDA_DEVERR_* bits).  Synchronises `stream`.  Returns PDA_ERR_DEVICE_DATA
 * when any flag was set, PDA_OK otherwise.  Clearing also zeroes the
 * counters through which the pieces of a split unit find the one that merges
 * them: a kernel that gave up (PDA_DEVERR_TIMEOUT) may leave them behind, and
 * later calls are valid again only after a clearing read.
 */
pda_status pda_read_device_errors(pda_ctx* ctx, uint32_t* flags, int32_t clear,
                                  pda_stream stream);

/*
 * Failure-detection check: launches one CTA that waits on a barrier phase
 * nothing completes, through the same bounded wait every decode kernel uses
 * for its TMA and consumer barriers.  After limit_ns (1 us .. 2 s) the wait
 * gives up, PDA_DEVERR_TIMEOUT is set in the context's flags and the kernel
 * returns; the context stays usable.  Read the flag with
 * pda_read_device_errors().
 */
pda_status pda_check_wait_timeout(pda_ctx* ctx, int64_t limit_ns, pda_stream stream);

/*
 * Timing hook: when the three events (cudaEvent_t) are non-NULL, every later
 * one-shot decode records ev_begin before its kernel and ev_split and ev_end
 * after it (a decode is one kernel launch: the split pieces of a unit merge
 * inside it), on the call's stream; NULLs turn it off.  The events between
 * calls stop the next call's early (programmatic) launch, so timed calls are
 * measured on their own.
 */
pda_status pda_set_timing_events(pda_ctx* ctx, void* ev_begin, void* ev_split, void* ev_end);

/*
 * Describes the launch the context would make (host only, after pda_create):
 * split-kernel CTAs (a multiple of the SM count), CTAs per SM, pipeline
 * stages, dynamic shared memory bytes per CTA, partial-state slots and the
 * plan's unit cost (see pda_plan_units).
 */
typedef struct pda_launch_info {
    int32_t split_ctas;
    int32_t ctas_per_sm;
    int32_t num_sms;
    int32_t stages;
    int32_t smem_bytes;
    int32_t stage_tokens;
    int64_t partial_slots;
    int32_t unit_cost;
} pda_launch_info;
pda_status pda_get_launch_info(const pda_ctx* ctx, pda_launch_info* info);

/*
 * The launch pda_decode_multi makes for q_len queries per sequence (host
 * only): the form (0: n8, q rows as the MMA's N; 1: row form, q rows as its
 * M, on mma.sync; 2: the row form on the tcgen05 tensor cores at head size
 * 128, for launch rows of 17 to 32 q rows, accumulators in tensor memory,
 * when switched on with pda_set_multi_tc), queries per launch
 * row and their q rows (queries x G), launch rows (KV walks) per sequence,
 * the grid and the pipeline depth.  q_len outside [1, split_ctas] is
 * PDA_ERR_INVALID_ARG; q_len 1 describes plain decode.
 */
typedef struct pda_multi_info {
    int32_t form;
    int32_t queries_per_walk;
    int32_t rows_per_walk;
    int32_t walks_per_seq;
    int32_t split_ctas;
    int32_t stages;
} pda_multi_info;
pda_status pda_get_multi_info(const pda_ctx* ctx, int32_t q_len, pda_multi_info* info);
/*
 * Whether pda_decode_multi takes the tcgen05 row form where it applies
 * (enable != 0) or the mma.sync row form (0, the default).  The form exists
 * for head size 128 with blocks of 8+ rows or rows gathered one by one
 * (block sizes below 8 whose blocks are not whole 1024-byte boxes).  Both
 * forms compute the same function (up to fp32 summation order).  The tcgen05
 * form measures 15-20 % slower on the multi-query workloads tried, hence off
 * by default.  Host only.
 */
pda_status pda_set_multi_tc(pda_ctx* ctx, int32_t enable);

/*
 * The split plan on its own (host only; no GPU needed).  The decode kernel
 * walks the flattened index space of W = Hkv * sum_b nv_b plan blocks,
 * ordered (sequence, kv head, block): a unit with nb_b blocks,
 * nb_b = ceil(max(len_b, 0) / block_size) (or the tile count when
 * blocks_given != 0), spans nv_b = nb_b + unit_cost positions (0 when
 * nb_b = 0), its blocks first.  The unit cost stands for the fixed work of a
 * segment, so that CTAs covering many short units get fewer blocks; a
 * context's value is in pda_launch_info.unit_cost.  CTA c takes positions
 * [floor(c*W/P), floor((c+1)*W/P)).  Small batches are planned by unit
 * instead: when batch*Hkv <= P and no unit holds more than 4 stages of rows
 * (4 * stage_tokens tokens; pda_launch_info.stage_tokens), CTA u processes
 * unit u whole.  For unit u = b*Hkv + g this reports the first and last CTA
 * holding one of its blocks (-1, -1 when it has none); a CTA's partial state
 * for unit u goes to slot u + c.
 *   lens         [batch] host int32 (tokens, or block counts).
 *   unit_cost    >= 0.
 *   stage_tokens rows per pipeline stage; 0 plans every batch by the even
 *                split.
 *   first_cta,
 *   last_cta     [batch*Hkv] outputs.
 *   total_blocks receives W.
 */
pda_status pda_plan_units(const int32_t* lens, int32_t batch, int32_t blocks_given,
                          int32_t block_size, int32_t num_kv_heads, int32_t split_ctas,
                          int32_t unit_cost, int32_t stage_tokens, int32_t* first_cta,
                          int32_t* last_cta, int64_t* total_blocks);

/*
 * One-shot decode that allocates nothing -- no counterpart on the pages; it
 * exists for callers that cannot allocate device memory.
 *
 * Some callers cannot call cudaMalloc (or anything that allocates) at the
 * point where they decode: code running inside a CUDA-graph capture they do
 * not control, allocators that forbid outside allocations, or embedders with
 * a fixed memory budget set up before any model runs.  pda_create allocates
 * the context's state and workspace, so those callers use this entry point
 * instead.  It needs no context: its scratch (the split kernel's partial
 * states and block prefix) lives in one statically sized device array
 * (PDA_NOALLOC_SCRATCH_BYTES) that every GPU loading this library holds
 * until the process exits.
 *
 * Arguments and layout are those of pda_decode (default pool layout
 * [num_blocks, block_size, Hkv, D], every block size pda_check_dims
 * accepts); the sizes that pda_create would take come as arguments, and the
 * call launches the same kernels, with the same loader for the block size,
 * as a context would.  device_flags is a required device word (4-byte
 * aligned) that receives PDA_DEVERR_* bits; the caller zeroes it and reads
 * it after the call has run.  A kernel that met a bad block id or length, or
 * whose bounded wait gave up (its output is then not valid), says so there;
 * NULL is refused so that no failure goes unreported.
 *
 * Rules: a call whose scratch need exceeds PDA_NOALLOC_SCRATCH_BYTES returns
 * PDA_ERR_INVALID_ARG with the size in pda_last_error(); batch is limited
 * to 1024 sequences.  The first call on each device finds the scratch's
 * device address and sets the split kernels' shared-memory attributes there
 * (to the same values pda_create sets): make that first call before any
 * stream capture.  All calls share the one scratch array and keep the last
 * call's contents (every call rewrites what it reads, so nothing needs
 * clearing): two calls that can overlap on the GPU (different streams
 * without ordering, or several threads) race and corrupt each other's
 * results, so order them on one stream.
 */
#define PDA_NOALLOC_SCRATCH_BYTES (4u << 20)
pda_status pda_decode_noalloc(const pda_bf16* q, const pda_bf16* k_pool, const pda_bf16* v_pool,
                              int64_t num_blocks, const int32_t* block_table, int32_t max_blocks,
                              const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              float scale, pda_bf16* out, uint32_t* device_flags,
                              pda_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* PDA_H */
