// Split-kernel instantiations for head_dim 128 (one translation unit per head
// size so the build compiles them in parallel).
#include "pda_kernels.cuh"

namespace pda {

const void* split_kernel_fn_d128(int mode) {
    switch (mode) {
        case kOneShot: return reinterpret_cast<const void*>(&split_kernel<128, kOneShot>);
        case kTiled: return reinterpret_cast<const void*>(&split_kernel<128, kTiled>);
        case kGather: return reinterpret_cast<const void*>(&split_kernel<128, kGather>);
        case kMulti: return reinterpret_cast<const void*>(&split_kernel<128, kMulti>);
        default: return nullptr;
    }
}

int split_stages_d128() { return Cfg<128>::kStages; }

// Launched with programmatic stream serialization: the kernel's prologue may
// overlap the previous kernel; it waits (griddepcontrol.wait) before reading
// global memory.
cudaError_t launch_split_d128(int mode, const SplitParams& p, int grid, size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (mode) {
        case kOneShot: return cudaLaunchKernelEx(&cfg, split_kernel<128, kOneShot>, p);
        case kTiled: return cudaLaunchKernelEx(&cfg, split_kernel<128, kTiled>, p);
        case kGather: return cudaLaunchKernelEx(&cfg, split_kernel<128, kGather>, p);
        case kMulti: return cudaLaunchKernelEx(&cfg, split_kernel<128, kMulti>, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pda
