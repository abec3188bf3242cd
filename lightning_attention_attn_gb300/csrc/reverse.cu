// Time reversal of packed sequences: out row (cu[s] + cu[s+1] - 1 - t) =
// in row t for every token t of sequence s.  The gradients of the causal
// form with respect to k and v are causal sums in reversed time
// (dk_u = sum_{t >= u} lambda^(t-u) (dout_t . v_u) q_t, and likewise dv), so
// the backward pass runs the forward kernels on time-reversed operands and
// reverses their outputs back.  A pure copy: memory-bound, 16-byte accesses,
// one CTA per token row.
#include <cstdint>

#include <cuda_runtime.h>

#include "la_internal.h"

namespace la {
namespace {

constexpr int kRevThreads = 256;

__global__ void __launch_bounds__(kRevThreads)
reverse_rows_kernel(const uint4 *__restrict__ in, uint4 *__restrict__ out,
                    const int32_t *__restrict__ cu, int nseq, int T, int row_vecs) {
    __shared__ int dst_row;
    const int t = blockIdx.x;
    if (threadIdx.x == 0) {
        // the sequence holding row t: the last s with cu[s] <= t (binary
        // search; cu is non-decreasing, and reads are clamped to [0, T])
        int lo = 0, hi = nseq - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (min(max(__ldg(cu + mid), 0), T) <= t) lo = mid;
            else hi = mid - 1;
        }
        const int t0 = min(max(__ldg(cu + lo), 0), T);
        const int t1 = min(max(__ldg(cu + lo + 1), t0), T);
        // rows outside every sequence (malformed cu) stay where they are
        dst_row = (t >= t0 && t < t1) ? t0 + t1 - 1 - t : t;
    }
    __syncthreads();
    const uint4 *src = in + (long)t * row_vecs;
    uint4 *dst = out + (long)dst_row * row_vecs;
    for (int c = threadIdx.x; c < row_vecs; c += kRevThreads) dst[c] = __ldg(src + c);
}

}  // namespace

cudaError_t reverse_sequences(const void *in, void *out, const int32_t *cu_seqlens, int nseq,
                              int total_tokens, size_t row_bytes, cudaStream_t stream) {
    if (total_tokens <= 0 || nseq <= 0) return cudaSuccess;
    if (row_bytes % 16 != 0) return cudaErrorInvalidValue;
    reverse_rows_kernel<<<(unsigned)total_tokens, kRevThreads, 0, stream>>>(
        static_cast<const uint4 *>(in), static_cast<uint4 *>(out), cu_seqlens, nseq,
        total_tokens, (int)(row_bytes / 16));
    return cudaGetLastError();
}

}  // namespace la
