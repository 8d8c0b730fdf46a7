// pda_api.cu -- the C ABI of include/pda.h: argument checks, context and
// workspace ownership, TMA descriptor encoding and kernel launches.
//
// Lifecycle and checks follow tiled_attention.rs (spark_storage):
// TiledAttentionDims::validate (head divisibility, head_dim <= 256),
// TiledAttention::new (state buffers sized for the maximum dims, reused),
// begin_step (num_seqs <= max_seqs, reset to (-inf, 0, 0)), step_tile,
// finalize.  Errors are returned as status codes, never thrown.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "pda.h"
#include "pda_launch.h"

#define PDA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

thread_local std::string g_last_error;

pda_status fail(pda_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

pda_status cuda_fail(cudaError_t e, const char* what) {
    return fail(PDA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace

struct pda_pool_key {  // what a pool's tensor maps are encoded from
    const void* k = nullptr;
    const void* v = nullptr;
    int64_t num_blocks = 0, blk = 0, tok = 0, kvh = 0;
};

struct pda_ctx {
    pda_dims dims;
    int32_t G = 0;
    int device = 0;
    int num_sms = 0;
    int stages = 0;
    int stage_rows = 64;  // split-kernel shape: KV rows per stage
    int ctas_per_sm = 0;
    int split_ctas = 0;
    int smem_max = 0;
    int64_t slots = 0;
    int64_t part_rows = 0;  // q rows the partial-state buffers hold (all slots)
    // Row form of multi-query (one / two 16-row q tiles): grid and pipeline
    // depth; a grid of 0 when the shape does not exist (head size 256).
    int rows_ctas[2] = {0, 0};
    int rows_stages[2] = {0, 0};
    // The tcgen05 row form (launch rows of 17 to 32 q rows): grid and depth
    // (0: not on this shape), and whether calls take it (pda_set_multi_tc; off
    // by default: measured slower than the mma.sync row form).
    int tc_ctas = 0;
    int tc_stages = 0;
    bool multi_tc = false;
    float* part_o = nullptr;
    float* part_ml = nullptr;
    int32_t* unit_sync = nullptr;  // [chunk_b*Hkv][2] split-unit tickets and stored counts
    int64_t unit_sync_bytes = 0;
    uint32_t* err = nullptr;
    float* m_state = nullptr;
    float* l_state = nullptr;
    float* o_state = nullptr;
    cudaEvent_t ev_begin = nullptr, ev_split = nullptr, ev_end = nullptr;
    // Tiled lifecycle: tile steps since the last begin_step and the stream of
    // the last one; a tile step right behind another on the same stream reads
    // its inputs early (pda_set_tile_overlap turns that off).
    int64_t tile_steps = 0;
    cudaStream_t tile_stream = nullptr;
    bool tile_overlap = true;
    // The last pool's tensor maps: a decode loop over one cache encodes them
    // once (encoding costs host time on every call otherwise).
    bool maps_valid = false;
    pda_pool_key maps_key;
    int32_t maps_row_mode = 0;
    CUtensorMap map_k, map_v;
    CUtensorMap map_k1, map_v1;  // one-slab boxes (head size 128, block boxes): the tcgen05 form
};

namespace {

struct PoolArgs {
    const pda_bf16* k;
    const pda_bf16* v;
    int64_t num_blocks;
    int64_t blk, tok, kvh;
};

// One 5-D tiled view per pool, {64 columns, block_size slots, D/64 column
// slabs, Hkv heads, num_blocks}, whose box {64, bs, D/64, 1, 1} is one kv
// head's rows of one block: a single TMA copy per block and pool, landing in
// shared memory as [slab][slot][128 bytes] with the 128-byte swizzle.  The
// stride triple (block, token, kv head) places any row layout in this view.
pda_status encode_pool(const pda_dims& d, const void* base, const PoolArgs& a, CUtensorMap* tm,
                       bool one_slab = false) {
    auto enc = tensor_map_encoder();
    if (!enc) return fail(PDA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[5] = {64, (cuuint64_t)d.block_size, (cuuint64_t)(d.head_dim / 64),
                                (cuuint64_t)d.num_kv_heads, (cuuint64_t)a.num_blocks};
    const cuuint64_t strides[4] = {(cuuint64_t)a.tok * 2, 128, (cuuint64_t)a.kvh * 2,
                                   (cuuint64_t)a.blk * 2};
    const cuuint32_t box[5] = {64, (cuuint32_t)d.block_size, one_slab ? 1u : (cuuint32_t)(d.head_dim / 64), 1,
                               1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PDA_ERR_INVALID_ARG, "cuTensorMapEncodeTiled rejected the pool layout (CUresult %d)",
                    (int)r);
    return PDA_OK;
}

// For block sizes below 8: a 2-D view {D, rows} of a pool whose three strides
// are multiples of D, box {64, 1}, for TMA gather4 (four rows per copy).
// Returns false (no error) when the layout does not fit that view.
bool encode_rows(const pda_dims& d, const void* base, const PoolArgs& a, CUtensorMap* tm) {
    auto enc = tensor_map_encoder();
    const int64_t D = d.head_dim;
    if (!enc || a.blk % D || a.tok % D || a.kvh % D) return false;
    const int64_t rows = (a.num_blocks - 1) * (a.blk / D) + (int64_t)(d.block_size - 1) * (a.tok / D) +
                         (int64_t)(d.num_kv_heads - 1) * (a.kvh / D) + 1;
    if (rows >= INT32_MAX) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, 1};
    const cuuint32_t estr[2] = {1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

pda_status check_pool(const PoolArgs& a) {
    if (!a.k || !a.v) return fail(PDA_ERR_INVALID_ARG, "k_pool / v_pool must not be NULL");
    if (!aligned(a.k, 16) || !aligned(a.v, 16))
        return fail(PDA_ERR_INVALID_ARG, "k_pool / v_pool must be 16-byte aligned");
    if (a.num_blocks < 1 || a.num_blocks > INT32_MAX)
        return fail(PDA_ERR_INVALID_ARG, "num_blocks %lld outside [1, 2^31)", (long long)a.num_blocks);
    const int64_t s[3] = {a.blk, a.tok, a.kvh};
    for (int i = 0; i < 3; ++i)
        if (s[i] <= 0 || s[i] % 8 != 0 || s[i] >= (int64_t(1) << 38))
            return fail(PDA_ERR_INVALID_ARG,
                        "pool strides must be positive multiples of 8 elements (got %lld, %lld, %lld)",
                        (long long)a.blk, (long long)a.tok, (long long)a.kvh);
    return PDA_OK;
}

// The split kernel's KV loader for a pool, with its two tensor maps: one 5-D
// box per block and pool where a block fills whole 1024-byte swizzle spans
// (row mode 0, see block_boxes); otherwise the rows are gathered, with TMA
// gather4 when the three strides are multiples of D (row mode 1), else with
// 16-byte cp.async (row mode 2, maps unused).  The consumers' shared-memory
// layout depends on this choice, so every launch path takes it from here.
pda_status encode_loader(const pda_dims& d, const PoolArgs& a, CUtensorMap* tk, CUtensorMap* tv,
                         int32_t* row_mode) {
    if (pda::block_boxes(d.head_dim, d.block_size)) {
        pda_status st = encode_pool(d, a.k, a, tk);
        if (st == PDA_OK) st = encode_pool(d, a.v, a, tv);
        *row_mode = 0;
        return st;
    }
    *row_mode = encode_rows(d, a.k, a, tk) && encode_rows(d, a.v, a, tv) ? 1 : 2;
    return PDA_OK;
}

// The pool fields of the split kernel's parameters for a loader row mode.
void set_pool_params(pda::SplitParams& p, const pda_dims& d, const PoolArgs& a, int32_t row_mode) {
    p.num_blocks = a.num_blocks;
    p.k_base = a.k;
    p.v_base = a.v;
    p.blk_s = a.blk;
    p.tok_s = a.tok;
    p.kvh_s = a.kvh;
    p.row_gather = row_mode;
    p.row_blk = a.blk / d.head_dim;
    p.row_tok = a.tok / d.head_dim;
    p.row_kvh = a.kvh / d.head_dim;
}

// Dynamic shared memory allowed for a split-kernel shape and mode: what a
// launch of a full batch (max_launch_rows(mode) sequences) uses, so every
// caller sets the same value and none lowers it below what another launches
// with.
int split_smem_limit(int D, int st, int mode) {
    return (int)pda::smem_layout(D, st, mode, pda::split_stages(D, st, mode), pda::max_launch_rows(mode)).total;
}

// Sets the shared-memory attributes of every mode of a split-kernel shape on
// the current device (modes the shape does not have are skipped).
pda_status set_split_attributes(int D, int st, int optin) {
    for (int mode = 0; mode < pda::kNumModes; ++mode) {
        const void* fn = pda::split_kernel_fn(D, st, mode);
        if (!fn) continue;
        const int limit = split_smem_limit(D, st, mode);
        if (limit > optin)
            return fail(PDA_ERR_UNSUPPORTED, "needs %d bytes of shared memory per CTA (device allows %d)",
                        limit, optin);
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    }
    return PDA_OK;
}

pda_status check_scale(float scale, int D, float* scale_log2) {
    if (std::isnan(scale)) scale = 1.0f / std::sqrt((float)D);
    if (std::isinf(scale)) return fail(PDA_ERR_INVALID_ARG, "scale must be finite (NaN = default)");
    *scale_log2 = scale * kLog2e;
    return PDA_OK;
}

struct RunArgs {
    int mode;
    const pda_bf16* q;
    PoolArgs pool;
    const int32_t* table;
    int32_t table_stride;
    const int32_t* lens;
    int32_t lens_are_blocks;
    const int32_t* last_valid;
    int32_t batch;
    float scale;
    pda_bf16* out;
    float* out_f32;
    pda_bf16* dbg_k;
    pda_bf16* dbg_v;
    cudaStream_t stream;
    bool contiguous = false;  // no table: block b*table_stride + j (contiguous cache)
    int32_t q_len = 1;        // causal queries per sequence (q, out: [batch, q_len, Hq, D])
    bool early_inputs = false;  // tiled: a tile step right behind another of the same step
};

// The kernels keep a launch's plan-block prefix in int32: up to
// kMaxLaunchBatch rows of at most table_width + unit_cost plan blocks each.
pda_status check_plan_size(int64_t rows, int32_t table_width, int32_t unit_cost) {
    const int64_t most = std::min<int64_t>(rows, pda::kMaxLaunchBatch) * ((int64_t)table_width + unit_cost);
    if (most > 0x7fffffffLL)
        return fail(PDA_ERR_INVALID_ARG,
                    "block table width %d is too large: %lld rows per launch could hold %lld "
                    "blocks, more than a 32-bit prefix holds",
                    table_width, (long long)std::min<int64_t>(rows, pda::kMaxLaunchBatch), (long long)most);
    return PDA_OK;
}

// The launch shape of a call: the mode, queries per launch row (qp), grid
// and pipeline depth.  Multi-query calls with more than 8 q rows per
// sequence (q_len * G) take the row form when the context's shape has it.
struct MultiShape {
    int mode, qp, grid, stages;
};
// The tcgen05 form lands every stage tile as [slab][64 rows][128 B]: with one
// box per block and slab, each box must fill whole 1024-byte swizzle atoms
// (blocks of 8+ rows); smaller blocks qualify when their rows are gathered one
// by one (blocks that are not whole 1024-byte boxes).
bool tc_layout_ok(const pda_dims& d) {
    return d.block_size >= 8 || !pda::block_boxes(d.head_dim, d.block_size);
}

MultiShape multi_shape(const pda_ctx* ctx, int mode, int32_t q_len) {
    MultiShape s = {mode, 1, ctx->split_ctas, ctx->stages};
    if (mode != pda::kMulti) return s;
    const int G = ctx->G;
    if (q_len * G > pda::kMaxGroup && ctx->rows_ctas[1] > 0) {
        s.qp = std::min(q_len, pda::kMaxRowsPerWalk / G);
        const int k = s.qp * G <= 16 && ctx->rows_ctas[0] > 0 ? 0 : 1;
        s.mode = k ? pda::kMultiRows32 : pda::kMultiRows16;
        s.grid = ctx->rows_ctas[k];
        s.stages = ctx->rows_stages[k];
        if (k == 1 && ctx->multi_tc && ctx->tc_ctas > 0 && tc_layout_ok(ctx->dims)) {
            s.mode = pda::kMultiTc;
            s.grid = ctx->tc_ctas;
            s.stages = ctx->tc_stages;
        }
    } else {
        s.qp = std::max(1, std::min(q_len, pda::kMaxGroup / G));
    }
    return s;
}

pda_status run(pda_ctx* ctx, const RunArgs& r) {
    if (!ctx) return fail(PDA_ERR_INVALID_ARG, "ctx is NULL");
    const pda_dims& d = ctx->dims;
    if (r.q_len < 1 || r.q_len > std::min(pda::kMaxLaunchBatch, ctx->split_ctas))
        return fail(PDA_ERR_INVALID_ARG, "q_len %d outside [1, %d]", r.q_len,
                    std::min(pda::kMaxLaunchBatch, ctx->split_ctas));
    if (r.batch < 0 || (int64_t)r.batch * r.q_len > d.max_seqs)
        return fail(PDA_ERR_INVALID_ARG, "batch %d x q_len %d outside [0, max_seqs=%d]", r.batch,
                    r.q_len, d.max_seqs);
    if (r.batch == 0) return PDA_OK;
    pda_status st = check_pool(r.pool);
    if (st != PDA_OK) return st;
    if (r.mode != pda::kGather) {
        if (!r.q || !aligned(r.q, 16)) return fail(PDA_ERR_INVALID_ARG, "q must be non-NULL and 16-byte aligned");
    }
    if (pda::writes_output(r.mode)) {
        if (r.out_f32 ? !aligned(r.out_f32, 16) : (!r.out || !aligned(r.out, 16)))
            return fail(PDA_ERR_INVALID_ARG, "out must be non-NULL and 16-byte aligned");
    }
    if (r.mode == pda::kGather && (!r.dbg_k || !r.dbg_v || !aligned(r.dbg_k, 16) || !aligned(r.dbg_v, 16)))
        return fail(PDA_ERR_INVALID_ARG, "k_rows / v_rows must be non-NULL and 16-byte aligned");
    if ((!r.table && !r.contiguous) || !r.lens || !aligned(r.table, 4) || !aligned(r.lens, 4) ||
        (r.last_valid && !aligned(r.last_valid, 4)))
        return fail(PDA_ERR_INVALID_ARG, "table / length arrays must be non-NULL and 4-byte aligned");
    if (r.table_stride < 1)
        return fail(PDA_ERR_INVALID_ARG, "block table width must be >= 1 (got %d)", r.table_stride);
    st = check_plan_size((int64_t)r.batch * r.q_len, r.table_stride,
                         pda::unit_cost_blocks(ctx->stage_rows, d.head_dim, d.block_size,
                                               pda::cost_class(multi_shape(ctx, r.mode, r.q_len).mode)));
    if (st != PDA_OK) return st;
    float scale_log2 = 0.f;
    st = check_scale(r.scale, d.head_dim, &scale_log2);
    if (st != PDA_OK) return st;

    pda::SplitParams p;
    std::memset(&p, 0, sizeof p);
    const pda_pool_key key = {r.pool.k, r.pool.v, r.pool.num_blocks, r.pool.blk, r.pool.tok, r.pool.kvh};
    const pda_pool_key& mk = ctx->maps_key;
    if (!(ctx->maps_valid && mk.k == key.k && mk.v == key.v && mk.num_blocks == key.num_blocks &&
          mk.blk == key.blk && mk.tok == key.tok && mk.kvh == key.kvh)) {
        ctx->maps_valid = false;
        st = encode_loader(d, r.pool, &ctx->map_k, &ctx->map_v, &ctx->maps_row_mode);
        if (st == PDA_OK && ctx->maps_row_mode == 0 && d.head_dim == 128 && ctx->tc_ctas > 0) {
            st = encode_pool(d, r.pool.k, r.pool, &ctx->map_k1, true);
            if (st == PDA_OK) st = encode_pool(d, r.pool.v, r.pool, &ctx->map_v1, true);
        }
        if (st != PDA_OK) return st;
        ctx->maps_key = key;
        ctx->maps_valid = true;
    }
    p.tm_k = ctx->map_k;
    p.tm_v = ctx->map_v;
    p.tm_k1 = ctx->map_k1;
    p.tm_v1 = ctx->map_v1;
    const int32_t row_mode = ctx->maps_row_mode;

    const int32_t Hq = d.num_q_heads, Hkv = d.num_kv_heads, D = d.head_dim;
    const bool timing = ctx->ev_begin && ctx->ev_split && ctx->ev_end && pda::writes_output(r.mode);
    const int64_t dbg_row_tokens = (int64_t)r.table_stride * d.block_size;
    // Causal multi-query: qp queries of a sequence share one launch row of
    // qp*G q rows; a sequence has Qr launch rows.  Up to 8 q rows take the n8
    // form; more take the row form where the shape has it (head sizes up to
    // 128): one KV walk for up to 32 q rows, one or two 16-row q tiles.
    const MultiShape ms = multi_shape(ctx, r.mode, r.q_len);
    const int mode = ms.mode, qp = ms.qp, grid = ms.grid, stages = ms.stages;
    const int32_t Qr = (r.q_len + qp - 1) / qp;
    const int32_t SR = r.q_len > 1 ? qp * ctx->G : ctx->G;  // q rows per partial-state slot
    const int32_t rows_total = r.batch * Qr;
    // Launch rows per chunk (whole sequences): at most max_launch_rows(mode),
    // and the partial states of (rows x Hkv + grid) slots of SR rows must fit
    // the context's buffers.
    const int64_t fit = (ctx->part_rows / SR - grid) / Hkv;
    const int32_t chunk_rows = (int32_t)(std::min<int64_t>(pda::max_launch_rows(mode), fit) / Qr) * Qr;
    if (chunk_rows < 1)
        return fail(PDA_ERR_UNSUPPORTED, "q_len %d: a sequence's %d launch rows exceed the partial-state buffers",
                    r.q_len, Qr);
    for (int32_t c0 = 0; c0 < rows_total; c0 += chunk_rows) {
        const int32_t cb = std::min(chunk_rows, rows_total - c0);
        const int32_t s0 = c0 / Qr;  // first sequence of the chunk
        p.q = r.q ? r.q + (int64_t)s0 * r.q_len * Hq * D : nullptr;
        p.table = r.contiguous ? nullptr : r.table + (int64_t)s0 * r.table_stride;
        p.lens = r.lens + s0;
        p.q_len = r.q_len;
        p.qp = qp;
        p.rows_per_slot = SR;
        p.last_valid = r.last_valid ? r.last_valid + s0 : nullptr;
        p.out = r.out ? r.out + (int64_t)s0 * r.q_len * Hq * D : nullptr;
        p.out_f32 = r.out_f32 ? r.out_f32 + (int64_t)s0 * r.q_len * Hq * D : nullptr;
        p.part_o = ctx->part_o;
        p.part_ml = ctx->part_ml;
        p.unit_sync = ctx->unit_sync;
        p.m_state = ctx->m_state + (int64_t)s0 * Hq;  // tiled path (q_len 1)
        p.l_state = ctx->l_state + (int64_t)s0 * Hq;
        p.o_state = ctx->o_state + (int64_t)s0 * Hq * D;
        p.err = ctx->err;
        p.dbg_k = r.dbg_k ? r.dbg_k + (int64_t)s0 * Hkv * dbg_row_tokens * D : nullptr;
        p.dbg_v = r.dbg_v ? r.dbg_v + (int64_t)s0 * Hkv * dbg_row_tokens * D : nullptr;
        set_pool_params(p, d, r.pool, row_mode);
        p.table_stride = r.table_stride;
        p.lens_are_blocks = r.lens_are_blocks;
        p.B = cb;
        p.Hq = Hq;
        p.Hkv = Hkv;
        p.G = ctx->G;
        p.bs = d.block_size;
        p.unit_cost = pda::unit_cost_blocks(ctx->stage_rows, d.head_dim, d.block_size, pda::cost_class(mode));
        p.dbg_row_tokens = (int32_t)dbg_row_tokens;
        // a later chunk is right behind this call's previous chunk
        p.early_inputs = mode == pda::kTiled && (r.early_inputs || c0 > 0) ? 1 : 0;
        // Speculative prefetch of the first stages before the grid-dependency
        // wait (the prefetch warp): for launches that wait for their
        // predecessor, of block boxes of 8+ rows (smaller blocks spend the TMA
        // issue slots) and one launch row per sequence.
        p.prefetch = mode != pda::kGather && mode != pda::kMultiRows32 && mode != pda::kMultiTc &&
                     !p.early_inputs && Qr == 1 &&
                     d.block_size >= 8 && row_mode == 0;
        p.scale_log2 = scale_log2;
        const size_t smem = pda::smem_layout(D, ctx->stage_rows, mode, stages, cb).total;

        cudaError_t e;
        if (timing && c0 == 0 && (e = cudaEventRecord(ctx->ev_begin, r.stream)) != cudaSuccess)
            return cuda_fail(e, "cudaEventRecord");
        e = pda::launch_split(D, ctx->stage_rows, mode, p, grid, smem, r.stream);
        if (e != cudaSuccess) return cuda_fail(e, "split kernel launch");
        if (mode == pda::kGather) continue;
        if (timing && ((e = cudaEventRecord(ctx->ev_split, r.stream)) != cudaSuccess ||
                       (e = cudaEventRecord(ctx->ev_end, r.stream)) != cudaSuccess))
            return cuda_fail(e, "cudaEventRecord");
    }
    return PDA_OK;
}

}  // namespace

PDA_EXPORT int32_t pda_abi_version(void) { return PDA_ABI_VERSION; }

PDA_EXPORT const char* pda_status_string(pda_status s) {
    switch (s) {
        case PDA_OK: return "ok";
        case PDA_ERR_INVALID_ARG: return "invalid argument";
        case PDA_ERR_UNSUPPORTED: return "unsupported configuration";
        case PDA_ERR_CUDA: return "CUDA error";
        case PDA_ERR_NO_DEVICE: return "no usable sm_103 device";
        case PDA_ERR_DEVICE_DATA: return "device-side data error flagged";
        default: return "unknown status";
    }
}

PDA_EXPORT const char* pda_last_error(void) { return g_last_error.c_str(); }

PDA_EXPORT pda_status pda_check_dims(const pda_dims* d) {
    if (!d) return fail(PDA_ERR_INVALID_ARG, "dims is NULL");
    if (d->max_seqs < 1 || d->num_q_heads < 1 || d->num_kv_heads < 1 || d->head_dim < 1 ||
        d->block_size < 1 || d->tile_capacity < 1)
        return fail(PDA_ERR_INVALID_ARG, "every dim must be >= 1");
    // The check of TiledAttentionDims::validate (its message words the
    // divisibility the other way round; the check is what counts).
    if (d->num_q_heads % d->num_kv_heads != 0)
        return fail(PDA_ERR_INVALID_ARG, "num_kv_heads (%d) must divide num_q_heads (%d)",
                    d->num_kv_heads, d->num_q_heads);
    if (d->head_dim > 256)
        return fail(PDA_ERR_INVALID_ARG, "head_dim %d exceeds the maximum of 256", d->head_dim);
    if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256)
        return fail(PDA_ERR_UNSUPPORTED, "head_dim %d: kernels exist for 64, 128 and 256", d->head_dim);
    const int bs = d->block_size;
    if (bs != 1 && bs != 2 && bs != 4 && bs != 8 && bs != 16 && bs != 32 && bs != 64)
        return fail(PDA_ERR_UNSUPPORTED, "block_size %d: kernels exist for 1, 2, 4, 8, 16, 32 and 64",
                    bs);
    const int G = d->num_q_heads / d->num_kv_heads;
    if (G > pda::kMaxGroup)
        return fail(PDA_ERR_UNSUPPORTED, "group size %d: at most %d q heads per kv head", G, pda::kMaxGroup);
    return PDA_OK;
}

PDA_EXPORT pda_status pda_paged_strides(const pda_dims* d, int64_t out[3]) {
    if (!d || !out) return fail(PDA_ERR_INVALID_ARG, "NULL argument");
    out[0] = (int64_t)d->block_size * d->num_kv_heads * d->head_dim;
    out[1] = (int64_t)d->num_kv_heads * d->head_dim;
    out[2] = d->head_dim;
    return PDA_OK;
}

PDA_EXPORT pda_status pda_slot_strides(const pda_dims* d, int64_t out[3]) {
    if (!d || !out) return fail(PDA_ERR_INVALID_ARG, "NULL argument");
    const int64_t stripe = (int64_t)d->num_kv_heads * d->block_size * d->head_dim;
    out[0] = 2 * stripe;
    out[1] = d->head_dim;
    out[2] = (int64_t)d->block_size * d->head_dim;
    return PDA_OK;
}

PDA_EXPORT void pda_destroy(pda_ctx* ctx) {
    if (!ctx) return;
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != ctx->device) cudaSetDevice(ctx->device);
    cudaDeviceSynchronize();
    cudaFree(ctx->part_o);
    cudaFree(ctx->part_ml);
    cudaFree(ctx->unit_sync);
    cudaFree(ctx->err);
    cudaFree(ctx->m_state);
    cudaFree(ctx->l_state);
    cudaFree(ctx->o_state);
    if (prev >= 0 && prev != ctx->device) cudaSetDevice(prev);
    delete ctx;
}

PDA_EXPORT pda_status pda_create(const pda_dims* dims, pda_ctx** out_ctx) {
    if (!out_ctx) return fail(PDA_ERR_INVALID_ARG, "out_ctx is NULL");
    *out_ctx = nullptr;
    pda_status st = pda_check_dims(dims);
    if (st != PDA_OK) return st;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(PDA_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    cudaDeviceProp prop;
    if ((e = cudaGetDeviceProperties(&prop, dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    if (prop.major != 10 || prop.minor != 3)
        return fail(PDA_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                    prop.major, prop.minor);
    if (!tensor_map_encoder()) return fail(PDA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");

    pda_ctx* ctx = new pda_ctx();
    ctx->dims = *dims;
    ctx->G = dims->num_q_heads / dims->num_kv_heads;
    ctx->device = dev;
    ctx->num_sms = prop.multiProcessorCount;
    const int D = dims->head_dim;
    ctx->stage_rows = pda::stage_tokens(D, dims->block_size);
    ctx->stages = pda::split_stages(D, ctx->stage_rows, pda::kOneShot);
    const int chunk_b = std::min(dims->max_seqs, pda::kMaxLaunchBatch);
    ctx->smem_max = (int)pda::smem_layout(D, ctx->stage_rows, pda::kOneShot, ctx->stages, chunk_b).total;
    if (ctx->smem_max > (int)prop.sharedMemPerBlockOptin) {
        delete ctx;
        return fail(PDA_ERR_UNSUPPORTED, "needs %d bytes of shared memory per CTA (device allows %d)",
                    ctx->smem_max, (int)prop.sharedMemPerBlockOptin);
    }
    if ((st = set_split_attributes(D, ctx->stage_rows, (int)prop.sharedMemPerBlockOptin)) != PDA_OK) {
        delete ctx;
        return st;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm,
                                                      pda::split_kernel_fn(D, ctx->stage_rows, pda::kOneShot),
                                                      pda::split_threads(ctx->stage_rows, pda::kOneShot),
                                                      ctx->smem_max);
    if (e != cudaSuccess) { delete ctx; return cuda_fail(e, "occupancy query"); }
    if (per_sm < 1) { delete ctx; return fail(PDA_ERR_UNSUPPORTED, "split kernel does not fit on an SM"); }
    ctx->ctas_per_sm = per_sm;
    ctx->split_ctas = per_sm * ctx->num_sms;
    ctx->slots = (int64_t)chunk_b * dims->num_kv_heads + ctx->split_ctas;
    // The row form of multi-query, where the shape has it: its own occupancy.
    for (int k = 0; k < 2; ++k) {
        const int mode = k ? pda::kMultiRows32 : pda::kMultiRows16;
        const void* fn = pda::split_kernel_fn(D, ctx->stage_rows, mode);
        if (!fn) continue;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, pda::split_threads(ctx->stage_rows, mode),
                                                          split_smem_limit(D, ctx->stage_rows, mode));
        if (e != cudaSuccess) { delete ctx; return cuda_fail(e, "occupancy query"); }
        ctx->rows_ctas[k] = n * ctx->num_sms;
        ctx->rows_stages[k] = pda::split_stages(D, ctx->stage_rows, mode);
    }
    if (const void* fn = pda::split_kernel_fn(D, ctx->stage_rows, pda::kMultiTc)) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, pda::split_threads(ctx->stage_rows, pda::kMultiTc),
                                                          split_smem_limit(D, ctx->stage_rows, pda::kMultiTc));
        if (e != cudaSuccess) { delete ctx; return cuda_fail(e, "occupancy query"); }
        ctx->tc_ctas = n * ctx->num_sms;
        ctx->tc_stages = pda::split_stages(D, ctx->stage_rows, pda::kMultiTc);
    }
    // Partial states: slots of G <= 8 rows for plain decode and the n8 form
    // (chunk_b x Hkv units plus one slot per CTA).  The row form's launch
    // rows hold up to 32 q rows, but a full batch of max_seqs <= 1024
    // sequences has launch rows x Hkv x rows per slot below 2 x max_seqs x
    // Hq <= 16 x chunk_b x Hkv, plus 32 rows per CTA of its grid: with that
    // room every call runs in one launch.
    ctx->part_rows = ctx->slots * pda::kMaxGroup;
    if (ctx->rows_ctas[1] > 0)
        ctx->part_rows = std::max<int64_t>(ctx->part_rows,
                                           (int64_t)chunk_b * dims->num_kv_heads * 2 * pda::kMaxGroup +
                                               (int64_t)std::max({ctx->rows_ctas[0], ctx->rows_ctas[1],
                                                                  ctx->tc_ctas}) *
                                                   pda::kMaxRowsPerWalk);

    const int64_t nq = (int64_t)dims->max_seqs * dims->num_q_heads;
    struct { void** ptr; size_t bytes; } allocs[] = {
        {(void**)&ctx->part_o, (size_t)ctx->part_rows * D * sizeof(float)},
        {(void**)&ctx->part_ml, (size_t)ctx->part_rows * 2 * sizeof(float)},
        {(void**)&ctx->unit_sync, (size_t)chunk_b * dims->num_kv_heads * 2 * sizeof(int32_t)},
        {(void**)&ctx->err, sizeof(uint32_t)},
        {(void**)&ctx->m_state, (size_t)nq * sizeof(float)},
        {(void**)&ctx->l_state, (size_t)nq * sizeof(float)},
        {(void**)&ctx->o_state, (size_t)nq * D * sizeof(float)},
    };
    for (auto& a : allocs) {
        e = cudaMalloc(a.ptr, a.bytes);
        if (e != cudaSuccess) { pda_destroy(ctx); return cuda_fail(e, "cudaMalloc"); }
    }
    ctx->unit_sync_bytes = (int64_t)chunk_b * dims->num_kv_heads * 2 * sizeof(int32_t);
    if ((e = cudaMemset(ctx->err, 0, sizeof(uint32_t))) != cudaSuccess ||
        (e = cudaMemset(ctx->unit_sync, 0, (size_t)ctx->unit_sync_bytes)) != cudaSuccess) {
        pda_destroy(ctx);
        return cuda_fail(e, "cudaMemset");
    }
    // An empty running state until the first begin_step.
    e = pda::launch_reset_state(ctx->m_state, ctx->l_state, ctx->o_state, nq, D, nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { pda_destroy(ctx); return cuda_fail(e, "state reset"); }
    *out_ctx = ctx;
    return PDA_OK;
}

PDA_EXPORT pda_status pda_decode_strided(pda_ctx* ctx, const pda_bf16* q, const pda_bf16* k_pool,
                                         const pda_bf16* v_pool, int64_t num_blocks,
                                         int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride,
                                         const int32_t* block_table, int32_t max_blocks,
                                         const int32_t* seq_lens, int32_t batch, float scale,
                                         pda_bf16* out, pda_stream stream) {
    RunArgs r = {pda::kOneShot, q, {k_pool, v_pool, num_blocks, blk_stride, tok_stride, kvh_stride},
                 block_table, max_blocks, seq_lens, 0, nullptr, batch, scale, out, nullptr,
                 nullptr, nullptr, (cudaStream_t)stream};
    return run(ctx, r);
}

PDA_EXPORT pda_status pda_decode(pda_ctx* ctx, const pda_bf16* q, const pda_bf16* k_pool,
                                 const pda_bf16* v_pool, int64_t num_blocks,
                                 const int32_t* block_table, int32_t max_blocks,
                                 const int32_t* seq_lens, int32_t batch, float scale, pda_bf16* out,
                                 pda_stream stream) {
    if (!ctx) return fail(PDA_ERR_INVALID_ARG, "ctx is NULL");
    int64_t s[3];
    pda_paged_strides(&ctx->dims, s);
    return pda_decode_strided(ctx, q, k_pool, v_pool, num_blocks, s[0], s[1], s[2], block_table,
                              max_blocks, seq_lens, batch, scale, out, stream);
}

PDA_EXPORT pda_status pda_decode_f32(pda_ctx* ctx, const pda_bf16* q, const pda_bf16* k_pool,
                                     const pda_bf16* v_pool, int64_t num_blocks, int64_t blk_stride,
                                     int64_t tok_stride, int64_t kvh_stride,
                                     const int32_t* block_table, int32_t max_blocks,
                                     const int32_t* seq_lens, int32_t batch, float scale, float* out,
                                     pda_stream stream) {
    if (!out && batch > 0) return fail(PDA_ERR_INVALID_ARG, "out is NULL");
    RunArgs r = {pda::kOneShot, q, {k_pool, v_pool, num_blocks, blk_stride, tok_stride, kvh_stride},
                 block_table, max_blocks, seq_lens, 0, nullptr, batch, scale, nullptr, out,
                 nullptr, nullptr, (cudaStream_t)stream};
    return run(ctx, r);
}

PDA_EXPORT pda_status pda_begin_step(pda_ctx* ctx, int32_t num_seqs, pda_stream stream) {
    if (!ctx) return fail(PDA_ERR_INVALID_ARG, "ctx is NULL");
    if (num_seqs < 0 || num_seqs > ctx->dims.max_seqs)
        return fail(PDA_ERR_INVALID_ARG, "begin_step num_seqs %d > max_seqs %d", num_seqs,
                    ctx->dims.max_seqs);
    cudaError_t e = pda::launch_reset_state(ctx->m_state, ctx->l_state, ctx->o_state,
                                            (int64_t)num_seqs * ctx->dims.num_q_heads,
                                            ctx->dims.head_dim, (cudaStream_t)stream);
    ctx->tile_steps = 0;
    return e == cudaSuccess ? PDA_OK : cuda_fail(e, "state reset launch");
}

PDA_EXPORT pda_status pda_step_tile(pda_ctx* ctx, const pda_bf16* q, const pda_bf16* k_pool,
                                    const pda_bf16* v_pool, int64_t num_blocks,
                                    const int32_t* tile_blocks, const int32_t* tile_block_counts,
                                    const int32_t* tile_last_valid, int32_t num_seqs,
                                    int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride,
                                    float scale, pda_stream stream) {
    if (!ctx) return fail(PDA_ERR_INVALID_ARG, "ctx is NULL");
    RunArgs r = {pda::kTiled, q, {k_pool, v_pool, num_blocks, blk_stride, tok_stride, kvh_stride},
                 tile_blocks, ctx->dims.tile_capacity, tile_block_counts, 1, tile_last_valid,
                 num_seqs, scale, nullptr, nullptr, nullptr, nullptr, (cudaStream_t)stream};
    r.early_inputs = ctx->tile_overlap && ctx->tile_steps > 0 && ctx->tile_stream == (cudaStream_t)stream;
    const pda_status st = run(ctx, r);
    if (st == PDA_OK) {
        ++ctx->tile_steps;
        ctx->tile_stream = (cudaStream_t)stream;
    }
    return st;
}

PDA_EXPORT pda_status pda_set_tile_overlap(pda_ctx* ctx, int32_t enable) {
    if (!ctx) return fail(PDA_ERR_INVALID_ARG, "ctx is NULL");
    ctx->tile_overlap = enable != 0;
    return PDA_OK;
}

PDA_EXPORT pda_status pda_set_multi_tc(pda_ctx* ctx, int32_t enable) {
    if (!ctx) return fail(PDA_ERR_INVALID_ARG, "ctx is NULL");
    ctx->multi_tc = enable != 0;
    return PDA_OK;
}

static pda_status finalize_impl(pda_ctx* ctx, pda_bf16* out, float* out_f32, int32_t num_seqs,
                                pda_stream stream) {
    if (!ctx) return fail(PDA_ERR_INVALID_ARG, "ctx is NULL");
    if (num_seqs < 0 || num_seqs > ctx->dims.max_seqs)
        return fail(PDA_ERR_INVALID_ARG, "finalize num_seqs %d outside [0, max_seqs=%d]", num_seqs,
                    ctx->dims.max_seqs);
    if (num_seqs == 0) return PDA_OK;
    if (out_f32 ? !aligned(out_f32, 4) : (!out || !aligned(out, 2)))
        return fail(PDA_ERR_INVALID_ARG, "out must be non-NULL and aligned");
    cudaError_t e = pda::launch_finalize(ctx->l_state, ctx->o_state, out, out_f32,
                                         (int64_t)num_seqs * ctx->dims.num_q_heads,
                                         ctx->dims.head_dim, (cudaStream_t)stream);
    return e == cudaSuccess ? PDA_OK : cuda_fail(e, "finalize launch");
}

PDA_EXPORT pda_status pda_finalize(pda_ctx* ctx, pda_bf16* out, int32_t num_seqs, pda_stream stream) {
    if (!out && num_seqs > 0) return fail(PDA_ERR_INVALID_ARG, "out is NULL");
    return finalize_impl(ctx, out, nullptr, num_seqs, stream);
}

PDA_EXPORT pda_status pda_finalize_f32(pda_ctx* ctx, float* out, int32_t num_seqs, pda_stream stream) {
    if (!out && num_seqs > 0) return fail(PDA_ERR_INVALID_ARG, "out is NULL");
    return finalize_impl(ctx, nullptr, out, num_seqs, stream);
}

PDA_EXPORT pda_status pda_export_state(pda_ctx* ctx, int32_t num_seqs, float* m, float* l, float* o,
                                       pda_stream stream) {
    if (!ctx) return fail(PDA_ERR_INVALID_ARG, "ctx is NULL");
    if (num_seqs < 0 || num_seqs > ctx->dims.max_seqs)
        return fail(PDA_ERR_INVALID_ARG, "num_seqs %d outside [0, max_seqs=%d]", num_seqs,
                    ctx->dims.max_seqs);
    if (num_seqs == 0) return PDA_OK;
    if (!m || !l || !o || !aligned(m, 4) || !aligned(l, 4) || !aligned(o, 4))
        return fail(PDA_ERR_INVALID_ARG, "m / l / o must be non-NULL and 4-byte aligned");
    const cudaError_t e = pda::launch_export_state(ctx->m_state, ctx->l_state, ctx->o_state, m, l, o,
                                                   (int64_t)num_seqs * ctx->dims.num_q_heads,
                                                   ctx->dims.head_dim, (cudaStream_t)stream);
    return e == cudaSuccess ? PDA_OK : cuda_fail(e, "state export launch");
}

namespace {

pda_status merge_states_impl(pda_ctx* ctx, int32_t n_parts, int32_t num_seqs, const float* m_parts,
                             const float* l_parts, const float* o_parts, pda_bf16* out, float* out_f32,
                             pda_stream stream) {
    if (!ctx) return fail(PDA_ERR_INVALID_ARG, "ctx is NULL");
    if (n_parts < 1 || num_seqs < 0)
        return fail(PDA_ERR_INVALID_ARG, "n_parts %d must be >= 1 and num_seqs %d >= 0", n_parts, num_seqs);
    if (num_seqs == 0) return PDA_OK;
    if (!m_parts || !l_parts || !o_parts || !aligned(m_parts, 4) || !aligned(l_parts, 4) ||
        !aligned(o_parts, 16))
        return fail(PDA_ERR_INVALID_ARG,
                    "m_parts / l_parts must be 4-byte and o_parts 16-byte aligned, non-NULL");
    if (out_f32 ? !aligned(out_f32, 16) : (!out || !aligned(out, 16)))
        return fail(PDA_ERR_INVALID_ARG, "out must be non-NULL and 16-byte aligned");
    const cudaError_t e = pda::launch_merge_states(
        m_parts, l_parts, o_parts, n_parts, (int64_t)num_seqs * ctx->dims.num_q_heads, ctx->dims.head_dim,
        out, out_f32, (cudaStream_t)stream);
    return e == cudaSuccess ? PDA_OK : cuda_fail(e, "state merge launch");
}

}  // namespace

PDA_EXPORT pda_status pda_merge_states(pda_ctx* ctx, int32_t n_parts, int32_t num_seqs,
                                       const float* m_parts, const float* l_parts, const float* o_parts,
                                       pda_bf16* out, pda_stream stream) {
    return merge_states_impl(ctx, n_parts, num_seqs, m_parts, l_parts, o_parts, out, nullptr, stream);
}

PDA_EXPORT pda_status pda_merge_states_f32(pda_ctx* ctx, int32_t n_parts, int32_t num_seqs,
                                           const float* m_parts, const float* l_parts,
                                           const float* o_parts, float* out, pda_stream stream) {
    if (!out && num_seqs > 0) return fail(PDA_ERR_INVALID_ARG, "out is NULL");
    return merge_states_impl(ctx, n_parts, num_seqs, m_parts, l_parts, o_parts, nullptr, out, stream);
}

PDA_EXPORT pda_status pda_debug_gather(pda_ctx* ctx, const pda_bf16* k_pool, const pda_bf16* v_pool,
                                       int64_t num_blocks, int64_t blk_stride, int64_t tok_stride,
                                       int64_t kvh_stride, const int32_t* block_table,
                                       int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                                       pda_bf16* k_rows, pda_bf16* v_rows, pda_stream stream) {
    RunArgs r = {pda::kGather, nullptr, {k_pool, v_pool, num_blocks, blk_stride, tok_stride, kvh_stride},
                 block_table, max_blocks, seq_lens, 0, nullptr, batch, NAN, nullptr, nullptr,
                 k_rows, v_rows, (cudaStream_t)stream};
    return run(ctx, r);
}

PDA_EXPORT pda_status pda_read_device_errors(pda_ctx* ctx, uint32_t* flags, int32_t clear,
                                             pda_stream stream) {
    if (!ctx || !flags) return fail(PDA_ERR_INVALID_ARG, "NULL argument");
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, ctx->err, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && clear) {
        // a launch that gave up may have left split-unit counters behind
        e = cudaMemsetAsync(ctx->err, 0, sizeof(uint32_t), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(ctx->unit_sync, 0, (size_t)ctx->unit_sync_bytes, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "reading device error flags");
    *flags = v;
    if (v) return fail(PDA_ERR_DEVICE_DATA, "device error flags 0x%x", v);
    return PDA_OK;
}

PDA_EXPORT pda_status pda_check_wait_timeout(pda_ctx* ctx, int64_t limit_ns, pda_stream stream) {
    if (!ctx) return fail(PDA_ERR_INVALID_ARG, "ctx is NULL");
    if (limit_ns < 1000 || limit_ns > 2000000000LL)
        return fail(PDA_ERR_INVALID_ARG, "limit_ns %lld outside [1 us, 2 s]", (long long)limit_ns);
    cudaError_t e = pda::launch_wait_timeout_probe(ctx->err, (uint64_t)limit_ns, (cudaStream_t)stream);
    return e == cudaSuccess ? PDA_OK : cuda_fail(e, "wait probe launch");
}

PDA_EXPORT pda_status pda_set_timing_events(pda_ctx* ctx, void* ev_begin, void* ev_split, void* ev_end) {
    if (!ctx) return fail(PDA_ERR_INVALID_ARG, "ctx is NULL");
    ctx->ev_begin = (cudaEvent_t)ev_begin;
    ctx->ev_split = (cudaEvent_t)ev_split;
    ctx->ev_end = (cudaEvent_t)ev_end;
    return PDA_OK;
}

PDA_EXPORT pda_status pda_get_launch_info(const pda_ctx* ctx, pda_launch_info* info) {
    if (!ctx || !info) return fail(PDA_ERR_INVALID_ARG, "NULL argument");
    info->split_ctas = ctx->split_ctas;
    info->ctas_per_sm = ctx->ctas_per_sm;
    info->num_sms = ctx->num_sms;
    info->stages = ctx->stages;
    info->smem_bytes = ctx->smem_max;
    info->stage_tokens = ctx->stage_rows;
    info->partial_slots = ctx->slots;
    info->unit_cost = pda::unit_cost_blocks(ctx->stage_rows, ctx->dims.head_dim, ctx->dims.block_size, pda::kCostDecode);
    return PDA_OK;
}

PDA_EXPORT pda_status pda_get_multi_info(const pda_ctx* ctx, int32_t q_len, pda_multi_info* info) {
    if (!ctx || !info) return fail(PDA_ERR_INVALID_ARG, "NULL argument");
    if (q_len < 1 || q_len > std::min(pda::kMaxLaunchBatch, ctx->split_ctas))
        return fail(PDA_ERR_INVALID_ARG, "q_len %d outside [1, %d]", q_len,
                    std::min(pda::kMaxLaunchBatch, ctx->split_ctas));
    const MultiShape ms = multi_shape(ctx, q_len > 1 ? pda::kMulti : pda::kOneShot, q_len);
    info->form = pda::is_tc(ms.mode) ? 2 : pda::q_tiles(ms.mode) > 0 ? 1 : 0;
    info->queries_per_walk = ms.qp;
    info->rows_per_walk = ms.qp * ctx->G;
    info->walks_per_seq = (q_len + ms.qp - 1) / ms.qp;
    info->split_ctas = ms.grid;
    info->stages = ms.stages;
    return PDA_OK;
}

PDA_EXPORT pda_status pda_plan_units(const int32_t* lens, int32_t batch, int32_t blocks_given,
                                     int32_t block_size, int32_t num_kv_heads, int32_t split_ctas,
                                     int32_t unit_cost, int32_t stage_tokens, int32_t* first_cta,
                                     int32_t* last_cta, int64_t* total_blocks) {
    if (batch < 0 || block_size < 1 || num_kv_heads < 1 || split_ctas < 1 || unit_cost < 0 ||
        stage_tokens < 0 || (batch > 0 && (!lens || !first_cta || !last_cta)) || !total_blocks)
        return fail(PDA_ERR_INVALID_ARG, "bad plan arguments");
    auto blocks = [&](int32_t b) {
        return blocks_given ? std::max(lens[b], 0) : pda::blocks_for_tokens(lens[b], block_size);
    };
    int64_t sum = 0;
    int32_t nb_max = 0;
    for (int32_t b = 0; b < batch; ++b) {
        sum += pda::plan_blocks(blocks(b), unit_cost);
        nb_max = std::max(nb_max, blocks(b));
    }
    const int64_t W = sum * num_kv_heads, P = split_ctas;
    *total_blocks = W;
    const bool by_unit = stage_tokens > 0 &&
                         pda::unit_mode((int64_t)batch * num_kv_heads, P, nb_max, stage_tokens, block_size);
    int64_t pfx = 0;
    for (int32_t b = 0; b < batch; ++b) {
        const int32_t nb = blocks(b), nv = pda::plan_blocks(nb, unit_cost);
        for (int32_t g = 0; g < num_kv_heads; ++g) {
            const int64_t u = (int64_t)b * num_kv_heads + g;
            if (nb == 0) {
                first_cta[u] = last_cta[u] = -1;
                continue;
            }
            if (by_unit) {
                first_cta[u] = last_cta[u] = (int32_t)u;
                continue;
            }
            const int64_t su = pfx * num_kv_heads + (int64_t)g * nv;
            first_cta[u] = (int32_t)pda::cta_of_block(su, W, P);
            last_cta[u] = (int32_t)pda::cta_of_block(su + nb - 1, W, P);
        }
        pfx += nv;
    }
    return PDA_OK;
}

PDA_EXPORT pda_status pda_decode_contiguous(pda_ctx* ctx, const pda_bf16* q, const pda_bf16* k,
                                            const pda_bf16* v, int32_t max_seq_len,
                                            const int32_t* seq_lens, int32_t batch, float scale,
                                            pda_bf16* out, pda_stream stream) {
    if (!ctx) return fail(PDA_ERR_INVALID_ARG, "ctx is NULL");
    const pda_dims& d = ctx->dims;
    if (max_seq_len < 1 || max_seq_len % d.block_size != 0)
        return fail(PDA_ERR_INVALID_ARG, "max_seq_len %d must be a positive multiple of block_size %d",
                    max_seq_len, d.block_size);
    const int32_t per_seq = max_seq_len / d.block_size;
    // [batch, S, Hkv, D] read as blocks of block_size tokens: block b*(S/bs)+j.
    RunArgs r = {pda::kOneShot, q,
                 {k, v, (int64_t)batch * per_seq, (int64_t)d.block_size * d.num_kv_heads * d.head_dim,
                  (int64_t)d.num_kv_heads * d.head_dim, (int64_t)d.head_dim},
                 nullptr, per_seq, seq_lens, 0, nullptr, batch, scale, out, nullptr, nullptr, nullptr,
                 (cudaStream_t)stream, true};
    if (batch > pda::kMaxLaunchBatch)
        return fail(PDA_ERR_INVALID_ARG, "contiguous decode carries at most %d sequences per call",
                    pda::kMaxLaunchBatch);
    return run(ctx, r);
}

PDA_EXPORT pda_status pda_decode_multi(pda_ctx* ctx, const pda_bf16* q, const pda_bf16* k_pool,
                                       const pda_bf16* v_pool, int64_t num_blocks,
                                       const int32_t* block_table, int32_t max_blocks,
                                       const int32_t* seq_lens, int32_t batch, int32_t q_len,
                                       float scale, pda_bf16* out, pda_stream stream) {
    if (!ctx) return fail(PDA_ERR_INVALID_ARG, "ctx is NULL");
    int64_t s[3];
    pda_paged_strides(&ctx->dims, s);
    // one query per sequence is plain decode; more take the causal kernels
    RunArgs r = {q_len > 1 ? pda::kMulti : pda::kOneShot, q,
                 {k_pool, v_pool, num_blocks, s[0], s[1], s[2]},
                 block_table, max_blocks, seq_lens, 0, nullptr, batch, scale, out, nullptr,
                 nullptr, nullptr, (cudaStream_t)stream, false, q_len};
    return run(ctx, r);
}

// ---------------------------------------------------------------------------
// pda_decode_noalloc: the one-shot decode for callers that cannot allocate.
// Its scratch is this file-scope device array; host code reaches it only
// through the address cudaGetSymbolAddress returns for the current device.

static __device__ __align__(256) unsigned char g_noalloc_scratch[PDA_NOALLOC_SCRATCH_BYTES];

namespace {

struct NoallocDevice {
    bool ready = false;
    unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
    int num_sms = 0;
};

std::mutex g_noalloc_mutex;
NoallocDevice g_noalloc_devices[64];

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Once per device, with that device current: the scratch's device address,
// the SM count, and the shared-memory attributes of every split-kernel shape
// (the same values pda_create sets, so neither lowers the other's).
pda_status noalloc_setup(int dev, NoallocDevice& nd) {
    int major = 0, minor = 0, optin = 0;
    cudaError_t e;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&nd.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_fail(e, "device attributes");
    if (major != 10 || minor != 3)
        return fail(PDA_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                    major, minor);
    if (!tensor_map_encoder()) return fail(PDA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const int shapes[4][2] = {{64, 64}, {128, 64}, {256, 64}, {256, 32}};
    for (const auto& sh : shapes) {
        const pda_status st = set_split_attributes(sh[0], sh[1], optin);
        if (st != PDA_OK) return st;
    }
    void* ptr = nullptr;
    if ((e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch)) != cudaSuccess)
        return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    nd.scratch = static_cast<unsigned char*>(ptr);
    nd.ready = true;
    return PDA_OK;
}

}  // namespace

PDA_EXPORT pda_status pda_decode_noalloc(const pda_bf16* q, const pda_bf16* k_pool,
                                         const pda_bf16* v_pool, int64_t num_blocks,
                                         const int32_t* block_table, int32_t max_blocks,
                                         const int32_t* seq_lens, int32_t batch,
                                         int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t block_size, float scale,
                                         pda_bf16* out, uint32_t* device_flags,
                                         pda_stream stream) {
    if (batch < 0 || batch > pda::kMaxLaunchBatch)
        return fail(PDA_ERR_INVALID_ARG, "batch %d outside [0, %d]", batch, pda::kMaxLaunchBatch);
    const pda_dims dims = {batch > 0 ? batch : 1, num_q_heads, num_kv_heads, head_dim, block_size, 1};
    pda_status st = pda_check_dims(&dims);
    if (st != PDA_OK) return st;
    if (!device_flags || !aligned(device_flags, 4))
        return fail(PDA_ERR_INVALID_ARG,
                    "device_flags must be a non-NULL, 4-byte aligned device word (a call whose "
                    "kernel gives up or meets a bad block id reports it there)");
    if (batch == 0) return PDA_OK;

    const int G = num_q_heads / num_kv_heads, D = head_dim;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(PDA_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(PDA_ERR_UNSUPPORTED, "device index %d beyond 63", dev);

    unsigned char* scratch = nullptr;
    int num_sms = 0;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        NoallocDevice& nd = g_noalloc_devices[dev];
        if (!nd.ready && (st = noalloc_setup(dev, nd)) != PDA_OK) return st;
        scratch = nd.scratch;
        num_sms = nd.num_sms;
    }

    const int rows = pda::stage_tokens(D, block_size);  // split-kernel shape, as pda_create picks it
    const int stages = pda::split_stages(D, rows, pda::kOneShot);
    const size_t smem = pda::smem_layout(D, rows, pda::kOneShot, stages, batch).total;
    const void* split_fn = pda::split_kernel_fn(D, rows, pda::kOneShot);
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, split_fn,
                                                           pda::split_threads(rows, pda::kOneShot), smem)) !=
        cudaSuccess)
        return cuda_fail(e, "occupancy query");
    if (per_sm < 1) return fail(PDA_ERR_UNSUPPORTED, "split kernel does not fit on an SM");
    const int split_ctas = per_sm * num_sms;

    // Scratch: split-unit counters, partial states (m, l) and o, as a context's workspace.
    const int64_t slots = (int64_t)batch * num_kv_heads + split_ctas;
    const size_t off_sync = 0;
    const size_t sync_bytes = (size_t)batch * num_kv_heads * 2 * sizeof(int32_t);
    const size_t off_ml = off_sync + round256(sync_bytes);
    const size_t off_o = off_ml + round256((size_t)slots * G * 2 * sizeof(float));
    const size_t need = off_o + (size_t)slots * G * D * sizeof(float);
    if (need > PDA_NOALLOC_SCRATCH_BYTES)
        return fail(PDA_ERR_INVALID_ARG,
                    "this call needs %zu bytes of scratch; the static scratch holds %u "
                    "(reduce batch or use pda_create / pda_decode)",
                    need, (unsigned)PDA_NOALLOC_SCRATCH_BYTES);

    if (!q || !aligned(q, 16) || !out || !aligned(out, 16))
        return fail(PDA_ERR_INVALID_ARG, "q and out must be non-NULL and 16-byte aligned");
    if (!block_table || !seq_lens || !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return fail(PDA_ERR_INVALID_ARG, "block_table / seq_lens must be non-NULL and 4-byte aligned");
    if (max_blocks < 1) return fail(PDA_ERR_INVALID_ARG, "max_blocks must be >= 1");
    const int32_t unit_cost = pda::unit_cost_blocks(rows, D, block_size, pda::kCostDecode);
    if ((st = check_plan_size(batch, max_blocks, unit_cost)) != PDA_OK) return st;
    PoolArgs pool = {k_pool, v_pool, num_blocks, (int64_t)block_size * num_kv_heads * head_dim,
                     (int64_t)num_kv_heads * head_dim, (int64_t)head_dim};
    if ((st = check_pool(pool)) != PDA_OK) return st;
    float scale_log2 = 0.f;
    if ((st = check_scale(scale, D, &scale_log2)) != PDA_OK) return st;

    pda::SplitParams p;
    std::memset(&p, 0, sizeof p);
    int32_t row_mode = 0;
    if ((st = encode_loader(dims, pool, &p.tm_k, &p.tm_v, &row_mode)) != PDA_OK) return st;
    set_pool_params(p, dims, pool, row_mode);
    cudaStream_t s = (cudaStream_t)stream;
    p.q = q;
    p.table = block_table;
    p.lens = seq_lens;
    p.out = out;
    p.part_o = reinterpret_cast<float*>(scratch + off_o);
    p.part_ml = reinterpret_cast<float*>(scratch + off_ml);
    p.unit_sync = reinterpret_cast<int32_t*>(scratch + off_sync);
    p.err = device_flags;
    p.table_stride = max_blocks;
    p.B = batch;
    p.Hq = num_q_heads;
    p.Hkv = num_kv_heads;
    p.G = G;
    p.bs = block_size;
    p.q_len = 1;
    p.qp = 1;
    p.rows_per_slot = G;
    p.unit_cost = unit_cost;
    p.scale_log2 = scale_log2;
    // The counters start at zero (a launch that gave up may have left some behind).
    if ((e = cudaMemsetAsync(scratch + off_sync, 0, sync_bytes, s)) != cudaSuccess)
        return cuda_fail(e, "clearing the scratch counters");
    if ((e = pda::launch_split(D, rows, pda::kOneShot, p, split_ctas, smem, s)) != cudaSuccess)
        return cuda_fail(e, "split kernel launch");
    return PDA_OK;
}
