// pda_launch.h -- host-side launch entry points of the kernels (defined in
// pda_kernels_d*.cu and pda_launch.cu), called by the C API.
#pragma once

#include "pda_params.h"

namespace pda {

// Entry points defined per head_dim (pda_kernels_d*.cu).
// st: stage rows of the split kernel's shape (stage_tokens(D, block_size));
// a mode whose shape does not exist has 0 stages and a null entry point.
int split_stages(int D, int st, int mode);
const void* split_kernel_fn(int D, int st, int mode);
cudaError_t launch_split(int D, int st, int mode, const SplitParams& p, int grid, size_t smem,
                         cudaStream_t stream);
cudaError_t launch_reset_state(float* m, float* l, float* o, int64_t n_q, int32_t D,
                               cudaStream_t stream);
cudaError_t launch_wait_timeout_probe(uint32_t* err, uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_finalize(const float* l, const float* o, uint16_t* out, float* out_f32,
                            int64_t n_q, int32_t D, cudaStream_t stream);
cudaError_t launch_export_state(const float* m2, const float* l, const float* o, float* m_out,
                                float* l_out, float* o_out, int64_t n_q, int32_t D, cudaStream_t stream);
cudaError_t launch_merge_states(const float* m_parts, const float* l_parts, const float* o_parts,
                                int32_t n_parts, int64_t n_q, int32_t D, uint16_t* out, float* out_f32,
                                cudaStream_t stream);

}  // namespace pda
