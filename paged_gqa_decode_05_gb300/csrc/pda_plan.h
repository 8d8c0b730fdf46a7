// pda_plan.h -- the split plan shared by the host API and the kernels.
//
// The work of one call is the flattened index space of W blocks ordered
// (sequence b, kv head g, block j): unit u = b*Hkv + g owns the W-range
// [pfx[b]*Hkv + g*nb_b, pfx[b]*Hkv + (g+1)*nb_b), where nb_b is the number of
// blocks of sequence b and pfx its exclusive prefix sum.  A grid of P CTAs
// splits the range evenly: CTA c takes [floor(c*W/P), floor((c+1)*W/P)).  Each
// maximal run of one unit inside one CTA's range is a "segment" with its own
// online-softmax state; the state of the segment of unit u in CTA c is stored
// in slot u + c, which is unique because moving to the next segment always
// advances u, c or both.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define PDA_HD __host__ __device__ __forceinline__
#else
#define PDA_HD inline
#endif

namespace pda {

// First flattened block of CTA c.
PDA_HD int64_t cta_begin(int64_t c, int64_t W, int64_t P) { return c * W / P; }

// The CTA whose range contains flattened block s (0 <= s < W): the largest c
// with floor(c*W/P) <= s, i.e. floor(((s+1)*P - 1) / W).
PDA_HD int64_t cta_of_block(int64_t s, int64_t W, int64_t P) { return ((s + 1) * P - 1) / W; }

// Blocks needed for a length in tokens.
PDA_HD int32_t blocks_for_tokens(int32_t len, int32_t block_size) {
    return len <= 0 ? 0 : (len + block_size - 1) / block_size;
}

}  // namespace pda
