// pda_aux.cuh -- elementwise kernels around the decode path: the tiled
// state's reset and finalize, and the export and merge of partial states
// across contexts.  Included by one translation unit (pda_launch.cu).
//
// Each is launched with programmatic dependent launch: it touches global
// memory only after the previous kernel has completed (griddepcontrol.wait),
// and only then lets the next kernel in the stream launch, so that a kernel
// launched early behind it knows every kernel before this one complete.
#pragma once

#include "pda_kernels.cuh"

namespace pda {

// (m, l, o) = (-inf, 0, 0) for n_q query slots.
__global__ void reset_state_kernel(float* m, float* l, float* o, int64_t n_q, int32_t D) {
    pdl_wait_primary();
    pdl_launch_dependents();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_q * D; i += stride) {
        o[i] = 0.f;
        if (i < n_q) {
            m[i] = kNegInf;
            l[i] = 0.f;
        }
    }
}

// State export: (m, l, o) with m from base-2 units (the kernels' scores carry
// scale * log2 e) to natural-log units of the scaled scores.
__global__ void export_state_kernel(const float* m2, const float* l, const float* o, float* m_out,
                                    float* l_out, float* o_out, int64_t n_q, int32_t D) {
    pdl_wait_primary();
    pdl_launch_dependents();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_q * D; i += stride) {
        o_out[i] = o[i];
        if (i < n_q) {
            m_out[i] = m2[i] * 0.69314718055994531f;  // ln 2; -inf stays -inf
            l_out[i] = l[i];
        }
    }
}

// Merge of n_parts exported states per (sequence, q head) row r:
// M = max_i m_i, L = sum_i l_i e^(m_i - M), O = sum_i o_i e^(m_i - M),
// out = O / L (0 when L == 0).  One thread per 4 consecutive outputs.
__global__ void merge_states_kernel(const float* m_parts, const float* l_parts, const float* o_parts,
                                    int32_t n_parts, int64_t n_q, int32_t D, uint16_t* out,
                                    float* out_f32) {
    pdl_wait_primary();
    pdl_launch_dependents();
    const int64_t n4 = n_q * D / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i4 < n4; i4 += stride) {
        const int64_t r = 4 * i4 / D;
        float M = kNegInf;
        for (int32_t k = 0; k < n_parts; ++k) M = fmaxf(M, m_parts[(int64_t)k * n_q + r]);
        float Ls = 0.f;
        float4 Os = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != kNegInf) {
            for (int32_t k = 0; k < n_parts; ++k) {
                const float f = ex2((m_parts[(int64_t)k * n_q + r] - M) * 1.4426950408889634f);
                const float4 o = reinterpret_cast<const float4*>(o_parts + (int64_t)k * n_q * D)[i4];
                Ls += l_parts[(int64_t)k * n_q + r] * f;
                Os.x += o.x * f;
                Os.y += o.y * f;
                Os.z += o.z * f;
                Os.w += o.w * f;
            }
        }
        const float4 v = Ls > 0.f ? make_float4(Os.x / Ls, Os.y / Ls, Os.z / Ls, Os.w / Ls)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        if (out_f32) {
            reinterpret_cast<float4*>(out_f32)[i4] = v;
        } else {
            uint2 w;
            w.x = pack_bf16x2(v.x, v.y);
            w.y = pack_bf16x2(v.z, v.w);
            reinterpret_cast<uint2*>(out)[i4] = w;
        }
    }
}

// out = o / l (bf16 round-to-nearest-even, or fp32); l == 0 gives 0.
__global__ void finalize_kernel(const float* l, const float* o, uint16_t* out, float* out_f32,
                                int64_t n_q, int32_t D) {
    pdl_wait_primary();
    pdl_launch_dependents();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_q * D; i += stride) {
        const float li = l[i / D];
        const float r = li > 0.f ? o[i] / li : 0.f;
        if (out_f32) out_f32[i] = r;
        else out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(r));
    }
}

}  // namespace pda
