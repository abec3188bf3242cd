// Internal interface between the C-ABI front end (api.cu) and the kernels.
// Not installed; the public interface is include/lightning_attn.h.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "lightning_attn.h"

namespace la {

// Launches `kern` with programmatic stream serialization: it may be scheduled
// while the kernel before it in the stream is finishing, and waits
// (grid_dependency_wait) before its first global-memory access, so stream
// order is kept for every memory effect.  Only kernels that begin with that
// wait are launched this way.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), unsigned grid, unsigned block,
                                    size_t smem, cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

struct PrefillArgs {
    const void *q, *k, *v;      // [T, H, D]
    const float *decay;         // [H]
    const int32_t *cu_seqlens;  // [nseq + 1], device
    int nseq, total_tokens, num_heads, head_dim, chunk;
    void *out;                  // [T, H, D]
    float *final_state;         // [nseq, H, D, D] or nullptr
    cudaStream_t stream;
    const float *initial_state; // [nseq, H, D, D] or nullptr (zero state)
    bool reverse_out = false;   // write o_t of sequence s to row cu[s] + cu[s+1] - 1 - t
    int min_len = 0;            // sequences shorter than this are left untouched
    // > 0: launch only the work of the rank_limit longest sequences (ranks
    // are in order of length, longest first, for nseq <= kMaxSortedSeqs)
    int rank_limit = 0;
    bool channel_decay = false; // decay is [H, D]: one lambda per key channel
    // Anti-causal sum o_t = sum_{u >= t} lambda^(u-t) (q_t . k_u) v_u (the
    // backward pass's reversed-time products), output rows in place; the
    // final state is then sum_u lambda^(u - t0) k_u^T v_u.  Tensor-core
    // kernel only, zero initial state.
    bool anti_causal = false;
    // Per-block state snapshots (nullptr: none): the state after every
    // snapshot_interval tokens of each sequence, [N, H, D, D] fp32, sequence
    // s's snapshots from index sum_{s' < s} floor(L_s' / snapshot_interval).
    // snapshot_interval is a multiple of the kernel's chunk.
    float *snapshots = nullptr;
    int snapshot_interval = 0;
};

struct DecodeArgs {
    const void *q, *k, *v;      // [B, H, D]
    const float *decay;         // [H]
    float *state;               // [B, H, D, D]
    int batch, num_heads, head_dim;
    void *out;                  // [B, H, D]
    cudaStream_t stream;
    // Packed mode (cu_seqlens != nullptr): entry b is sequence b of a packed
    // batch; its token row is cu_seqlens[b], and only sequences of length
    // exactly 1 are stepped (the others are left untouched).
    const int32_t *cu_seqlens = nullptr;
    int total_tokens = 0;
    bool channel_decay = false; // decay is [H, D]: one lambda per key channel (state row)
};

// Whether a (scalar-decay) call runs on the tensor-core kernel: bf16,
// head_dim 128 and a block size of 16, 32, 64, 128 or 256 (chunk 0 = 128).
inline bool uses_tensor_cores(bool bf16, int head_dim, int chunk) {
    return bf16 && head_dim == 128 &&
           (chunk == 0 || chunk == 16 || chunk == 32 || chunk == 64 || chunk == 128 ||
            chunk == 256);
}

// CUDA-core chunkwise prefill; chunk in {16, 32, 64}, head_dim in {64, 128};
// also the channel-wise decay variant.
cudaError_t prefill_simt_f32(const PrefillArgs &a);
cudaError_t prefill_simt_bf16(const PrefillArgs &a);

// tcgen05 / TMEM / TMA prefill; bf16, head_dim 128, block size 16-256.
// Returns cudaErrorNotSupported when the tensor-map encoder is unavailable.
cudaError_t prefill_tc_bf16(const PrefillArgs &a);

// tcgen05 / TMEM / TMA prefill with the channel-wise decay; bf16, head_dim
// 128, block size 64 (chunk 0 or 64), scalar-decay features (snapshots,
// anti-causal, mixed-step ranks) excluded.
cudaError_t prefill_cw_tc_bf16(const PrefillArgs &a);
// Reads and clears the channel-wise kernel's device error word (the caller
// has synchronised the stream).
cudaError_t take_cw_device_error(unsigned int *err);

// Synchronises `stream`, then reads and clears the device error word.
cudaError_t take_device_error(cudaStream_t stream, unsigned int *err);
// Launches a kernel whose bounded wait must time out after timeout_ns.
cudaError_t selftest_wait_timeout(uint64_t timeout_ns, cudaStream_t stream);

// out row (cu[s] + cu[s+1] - 1 - t) = in row t for every token t of
// sequence s; rows are row_bytes long (a multiple of 16).  in != out.
cudaError_t reverse_sequences(const void *in, void *out, const int32_t *cu_seqlens, int nseq,
                              int total_tokens, size_t row_bytes, cudaStream_t stream);

// Every host-side check of lightning_attn_backward except those of the
// workspace.  Returns an error status, or LA_OK with *work = false when there
// is nothing to compute, or LA_OK with *work = true and *needs_workspace
// telling whether the path that serves the call reads a workspace.
la_status backward_check(const void *q, const void *k, const void *v, const float *decay,
                         const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                         int32_t num_heads, int32_t head_dim, int32_t chunk, la_dtype dtype,
                         const void *d_out, void *d_q, void *d_k, void *d_v, bool *work,
                         bool *needs_workspace);

// Sets the message lightning_attn_last_error() returns on this host thread.
void set_last_error(const char *fmt, ...) __attribute__((format(printf, 1, 2)));

// Memory-bound decode step; head_dim in {64, 128}.
cudaError_t decode_f32(const DecodeArgs &a);
cudaError_t decode_bf16(const DecodeArgs &a);

}  // namespace la
