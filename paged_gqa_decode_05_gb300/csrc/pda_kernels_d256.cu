// Split-kernel instantiations for head_dim 256 (one translation unit per head
// size so the build compiles them in parallel).
#include "pda_kernels.cuh"

namespace pda {

const void* split_kernel_fn_d256(int mode) {
    switch (mode) {
        case kOneShot: return reinterpret_cast<const void*>(&split_kernel<256, kOneShot>);
        case kTiled: return reinterpret_cast<const void*>(&split_kernel<256, kTiled>);
        case kGather: return reinterpret_cast<const void*>(&split_kernel<256, kGather>);
        case kMulti: return reinterpret_cast<const void*>(&split_kernel<256, kMulti>);
        default: return nullptr;
    }
}

int split_stages_d256() { return Cfg<256>::kStages; }

// Launched with programmatic stream serialization: the kernel's prologue may
// overlap the previous kernel; it waits (griddepcontrol.wait) before reading
// global memory.
cudaError_t launch_split_d256(int mode, const SplitParams& p, int grid, size_t smem, cudaStream_t stream) {
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
        case kOneShot: return cudaLaunchKernelEx(&cfg, split_kernel<256, kOneShot>, p);
        case kTiled: return cudaLaunchKernelEx(&cfg, split_kernel<256, kTiled>, p);
        case kGather: return cudaLaunchKernelEx(&cfg, split_kernel<256, kGather>, p);
        case kMulti: return cudaLaunchKernelEx(&cfg, split_kernel<256, kMulti>, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pda
