// Split-kernel instantiations for head_dim 64 (one translation unit per head
// size so the build compiles them in parallel).
#include "pda_kernels.cuh"

namespace pda {

const void* split_kernel_fn_d64(int mode) {
    switch (mode) {
        case kOneShot: return reinterpret_cast<const void*>(&split_kernel<64, kOneShot>);
        case kTiled: return reinterpret_cast<const void*>(&split_kernel<64, kTiled>);
        case kGather: return reinterpret_cast<const void*>(&split_kernel<64, kGather>);
        default: return nullptr;
    }
}

int split_stages_d64() { return Cfg<64>::kStages; }

cudaError_t launch_split_d64(int mode, const SplitParams& p, int grid, size_t smem, cudaStream_t stream) {
    switch (mode) {
        case kOneShot: split_kernel<64, kOneShot><<<grid, kThreads, smem, stream>>>(p); break;
        case kTiled: split_kernel<64, kTiled><<<grid, kThreads, smem, stream>>>(p); break;
        case kGather: split_kernel<64, kGather><<<grid, kThreads, smem, stream>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace pda
