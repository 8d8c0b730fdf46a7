// Split-kernel instantiations for head_dim 256 (one translation unit per head
// size so the build compiles them in parallel): 64-row stages (block sizes
// >= 8) and 32-row stages (block sizes below 8, two CTAs per SM).
#include "pda_kernels.cuh"

namespace pda {

const void* split_kernel_fn_d256(int st, int mode) {
    return st == 32 ? split_fn_of<256, 32>(mode) : st == 64 ? split_fn_of<256, 64>(mode) : nullptr;
}

int split_stages_d256(int st, int mode) {
    return st == 32 ? split_stages_of<256, 32>(mode) : st == 64 ? split_stages_of<256, 64>(mode) : 0;
}

cudaError_t launch_split_d256(int st, int mode, const SplitParams& p, int grid, size_t smem,
                             cudaStream_t stream) {
    if (st == 32) return launch_split_of<256, 32>(mode, p, grid, smem, stream);
    if (st == 64) return launch_split_of<256, 64>(mode, p, grid, smem, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pda
