// State-reset, finalize, export and merge-states kernels, and the head_dim
// dispatch of the split kernel.
#include "pda_aux.cuh"
#include "pda_launch.h"

namespace pda {

namespace {
// Launch with programmatic stream serialization (see pda_aux.cuh).
template <typename... Args>
cudaError_t launch_pdl(void (*kernel)(Args...), int grid, int block, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)block, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}
}  // namespace

#define PDA_DECLARE_D(D)                                                                     \
    const void* split_kernel_fn_d##D(int st, int mode);                                     \
    int split_stages_d##D(int st, int mode);                                                 \
    cudaError_t launch_split_d##D(int st, int mode, const SplitParams& p, int grid,          \
                                  size_t smem, cudaStream_t stream);
PDA_DECLARE_D(64)
PDA_DECLARE_D(128)
PDA_DECLARE_D(256)

int split_stages(int D, int st, int mode) {
    switch (D) {
        case 64: return split_stages_d64(st, mode);
        case 128: return split_stages_d128(st, mode);
        case 256: return split_stages_d256(st, mode);
        default: return 0;
    }
}

const void* split_kernel_fn(int D, int st, int mode) {
    switch (D) {
        case 64: return split_kernel_fn_d64(st, mode);
        case 128: return split_kernel_fn_d128(st, mode);
        case 256: return split_kernel_fn_d256(st, mode);
        default: return nullptr;
    }
}

cudaError_t launch_split(int D, int st, int mode, const SplitParams& p, int grid, size_t smem,
                         cudaStream_t stream) {
    switch (D) {
        case 64: return launch_split_d64(st, mode, p, grid, smem, stream);
        case 128: return launch_split_d128(st, mode, p, grid, smem, stream);
        case 256: return launch_split_d256(st, mode, p, grid, smem, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_reset_state(float* m, float* l, float* o, int64_t n_q, int32_t D,
                               cudaStream_t stream) {
    if (n_q <= 0) return cudaSuccess;
    const int64_t n = n_q * D;
    const int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    return launch_pdl(reset_state_kernel, grid, 256, stream, m, l, o, n_q, D);
}

cudaError_t launch_finalize(const float* l, const float* o, uint16_t* out, float* out_f32,
                            int64_t n_q, int32_t D, cudaStream_t stream) {
    if (n_q <= 0) return cudaSuccess;
    const int64_t n = n_q * D;
    const int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    return launch_pdl(finalize_kernel, grid, 256, stream, l, o, out, out_f32, n_q, D);
}

}  // namespace pda

namespace pda {
// Failure-detection check: waits on an mbarrier phase that nothing completes,
// with the same bounded wait the decode kernels use; the wait gives up after
// limit_ns, sets the timeout flag and the kernel returns.
__global__ void wait_timeout_probe_kernel(uint32_t* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (!mbar_wait_bounded(b, 0, limit_ns) && threadIdx.x == 0) atomicOr(err, PDA_DEVERR_TIMEOUT_);
}

cudaError_t launch_wait_timeout_probe(uint32_t* err, uint64_t limit_ns, cudaStream_t stream) {
    wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}
cudaError_t launch_export_state(const float* m2, const float* l, const float* o, float* m_out,
                                float* l_out, float* o_out, int64_t n_q, int32_t D, cudaStream_t stream) {
    if (n_q <= 0) return cudaSuccess;
    const int64_t n = n_q * D;
    const int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    return launch_pdl(export_state_kernel, grid, 256, stream, m2, l, o, m_out, l_out, o_out, n_q, D);
}

cudaError_t launch_merge_states(const float* m_parts, const float* l_parts, const float* o_parts,
                                int32_t n_parts, int64_t n_q, int32_t D, uint16_t* out, float* out_f32,
                                cudaStream_t stream) {
    if (n_q <= 0) return cudaSuccess;
    const int64_t n4 = n_q * D / 4;
    const int grid = (int)((n4 + 255) / 256 < 4096 ? (n4 + 255) / 256 : 4096);
    return launch_pdl(merge_states_kernel, grid, 256, stream, m_parts, l_parts, o_parts, n_parts, n_q, D,
                      out, out_f32);
}

}  // namespace pda
