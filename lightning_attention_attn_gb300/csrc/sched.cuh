// Work ordering for packed variable-length prefill.
//
// Each CTA owns one (sequence, head[, value slice]) and walks that sequence's
// chunks serially, so a CTA's running time is proportional to its sequence
// length.  CTAs are dispatched roughly in blockIdx order; mapping low block
// indices to the longest sequences (longest-processing-time-first) keeps the
// last wave short.  The rank of every sequence is recomputed by each CTA from
// cu_seqlens (O(nseq) per thread, no scratch memory); above kMaxSortedSeqs
// sequences the natural order is used.
#pragma once

#include <cstdint>

namespace la {

constexpr int kMaxSortedSeqs = 128;

// Returns the sequence whose length rank is `r` (0 = longest; ties keep the
// lower index first).  Must be called by all threads of the block; needs
// blockDim.x >= min(nseq, kMaxSortedSeqs).  `slot` is one int of shared memory.
__device__ inline int sequence_of_rank(const int32_t *__restrict__ cu, int nseq,
                                       int r, int *slot) {
    if (nseq > kMaxSortedSeqs || nseq <= 1) return r;
    if (threadIdx.x == 0) *slot = r;  // fallback if no match (cannot happen)
    __syncthreads();
    const int s = threadIdx.x;
    if (s < nseq) {
        const int ls = __ldg(cu + s + 1) - __ldg(cu + s);
        int rank = 0;
        for (int s2 = 0; s2 < nseq; ++s2) {
            const int l2 = __ldg(cu + s2 + 1) - __ldg(cu + s2);
            rank += (l2 > ls) || (l2 == ls && s2 < s);
        }
        if (rank == r) *slot = s;
    }
    __syncthreads();
    const int out = *slot;
    __syncthreads();
    return out;
}

}  // namespace la
