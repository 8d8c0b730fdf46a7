// Split-kernel instantiations for head_dim 128 (one translation unit per head
// size so the build compiles them in parallel): 64-row stages, every mode
// including the row form of multi-query.
#include "pda_kernels.cuh"

namespace pda {

const void* split_kernel_fn_d128(int st, int mode) {
    return st == 64 ? split_fn_of<128, 64>(mode) : nullptr;
}

int split_stages_d128(int st, int mode) { return st == 64 ? split_stages_of<128, 64>(mode) : 0; }

cudaError_t launch_split_d128(int st, int mode, const SplitParams& p, int grid, size_t smem,
                             cudaStream_t stream) {
    if (st != 64) return cudaErrorInvalidValue;
    return launch_split_of<128, 64>(mode, p, grid, smem, stream);
}

}  // namespace pda
