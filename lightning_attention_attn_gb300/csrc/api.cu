// C-ABI front end of liblightning_attn.so: argument validation on the host,
// dispatch to the kernels, status mapping.  See include/lightning_attn.h for
// the contract of every entry point.
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include <cuda_runtime.h>

#include "lightning_attn.h"
#include "la_internal.h"
#include "sched.cuh"

namespace {

thread_local std::string g_last_error;

la_status fail(la_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
la_status fail(la_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

la_status from_cuda(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return LA_OK;
    if (e == cudaErrorNotSupported)
        return fail(LA_ERR_UNSUPPORTED, "%s: no kernel for this configuration", what);
    return fail(LA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Runs the forward kernel that serves (dtype, head_dim, chunk); arguments
// already validated.
la_status run_prefill(const la::PrefillArgs &a, la_dtype dtype) {
    const bool tc = la::uses_tensor_cores(dtype == LA_DTYPE_BF16, a.head_dim, a.chunk);
    if (tc) return from_cuda(la::prefill_tc_bf16(a), "prefill (tcgen05)");
    if (a.anti_causal)
        return fail(LA_ERR_UNSUPPORTED, "the anti-causal form runs on the tensor-core path only");
    if (a.chunk == 128 || a.chunk == 256)
        return fail(LA_ERR_UNSUPPORTED, "chunk %d needs the tensor-core path (bf16, head_dim 128)",
                    a.chunk);
    if (dtype == LA_DTYPE_FP32) return from_cuda(la::prefill_simt_f32(a), "prefill (fp32)");
    return from_cuda(la::prefill_simt_bf16(a), "prefill (bf16, CUDA cores)");
}

size_t elem_bytes(la_dtype dtype) { return dtype == LA_DTYPE_FP32 ? 4 : 2; }

// Fork/join events of the two-stream mixed step, one pair per device,
// created on first use; the mutex makes each call's record/wait sequence
// atomic with respect to other host threads.
constexpr int kMaxDevices = 64;
std::mutex g_mixed_mu;
cudaEvent_t g_fork[kMaxDevices] = {}, g_join[kMaxDevices] = {};

// Workspace of the backward pass: three [T, H, d] arrays, each 256-byte aligned.
size_t backward_slot_bytes(int32_t total_tokens, int32_t num_heads, int32_t head_dim,
                           la_dtype dtype) {
    const size_t b = (size_t)total_tokens * num_heads * head_dim * elem_bytes(dtype);
    return (b + 255) & ~(size_t)255;
}

// Argument checks shared by the prefill entry points.  Returns an error, or
// LA_OK with *work = false when there is nothing to launch (no sequences, or
// every sequence empty: then the final states have been set here).
la_status check_prefill(const void *q, const void *k, const void *v, const float *decay,
                        const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                        int32_t num_heads, int32_t head_dim, int32_t chunk, la_dtype dtype,
                        const float *initial_state, void *out, float *final_state,
                        void *stream, bool *work) {
    *work = false;
    if (num_seqs < 0) return fail(LA_ERR_INVALID_ARG, "num_seqs < 0 (%d)", num_seqs);
    if (total_tokens < 0) return fail(LA_ERR_INVALID_ARG, "total_tokens < 0 (%d)", total_tokens);
    if (num_heads < 1) return fail(LA_ERR_INVALID_ARG, "num_heads < 1 (%d)", num_heads);
    if (head_dim != 64 && head_dim != 128)
        return fail(LA_ERR_INVALID_ARG, "head_dim must be 64 or 128 (got %d)", head_dim);
    if (dtype != LA_DTYPE_BF16 && dtype != LA_DTYPE_FP32)
        return fail(LA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (chunk != 0 && chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128 && chunk != 256)
        return fail(LA_ERR_INVALID_ARG, "chunk must be 0, 16, 32, 64, 128 or 256 (got %d)", chunk);
    if (num_seqs == 0) return LA_OK;
    if (!cu_seqlens || !decay) return fail(LA_ERR_INVALID_ARG, "null decay or cu_seqlens");
    if (total_tokens > 0 && (!q || !k || !v || !out))
        return fail(LA_ERR_INVALID_ARG, "null q, k, v or out");
    if ((q && !aligned16(q)) || (k && !aligned16(k)) || (v && !aligned16(v)) ||
        (out && !aligned16(out)) || (final_state && !aligned16(final_state)) ||
        (initial_state && !aligned16(initial_state)) || !aligned16(decay) ||
        !aligned16(cu_seqlens))
        return fail(LA_ERR_INVALID_ARG, "every pointer must be 16-byte aligned");
    if ((long long)num_seqs * num_heads > 0x7fffffffLL / 4)
        return fail(LA_ERR_INVALID_ARG, "num_seqs * num_heads too large");
    const size_t state_bytes = (size_t)num_seqs * num_heads * head_dim * head_dim * sizeof(float);
    if (initial_state && final_state && initial_state != final_state) {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(initial_state);
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(final_state);
        if (a0 < b0 + state_bytes && b0 < a0 + state_bytes)
            return fail(LA_ERR_INVALID_ARG,
                        "initial_state and final_state overlap without being the same array");
    }
    if (total_tokens == 0) {  // every sequence is empty: each state is its cached state
        const cudaStream_t st = static_cast<cudaStream_t>(stream);
        if (!final_state || final_state == initial_state) return LA_OK;
        if (initial_state)
            return from_cuda(cudaMemcpyAsync(final_state, initial_state, state_bytes,
                                             cudaMemcpyDeviceToDevice, st),
                             "prefill (empty)");
        return from_cuda(cudaMemsetAsync(final_state, 0, state_bytes, st), "prefill (empty)");
    }
    *work = true;
    return LA_OK;
}

}  // namespace

namespace la {
void set_last_error(const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
}
}  // namespace la

extern "C" {

const char *lightning_attn_status_string(la_status s) {
    switch (s) {
        case LA_OK: return "LA_OK";
        case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG";
        case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED";
        case LA_ERR_CUDA: return "LA_ERR_CUDA";
        case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT";
    }
    return "LA_ERR_UNKNOWN";
}

const char *lightning_attn_last_error(void) { return g_last_error.c_str(); }

int32_t lightning_attn_version(void) { return LIGHTNING_ATTN_VERSION; }

la_status lightning_attn_prefill_with_state(const void *q, const void *k, const void *v,
                                            const float *decay, const int32_t *cu_seqlens,
                                            int32_t num_seqs, int32_t total_tokens,
                                            int32_t num_heads, int32_t head_dim,
                                            int32_t chunk, la_dtype dtype,
                                            const float *initial_state, void *out,
                                            float *final_state, void *stream) {
    bool work = false;
    const la_status st = check_prefill(q, k, v, decay, cu_seqlens, num_seqs, total_tokens,
                                       num_heads, head_dim, chunk, dtype, initial_state, out,
                                       final_state, stream, &work);
    if (st != LA_OK || !work) return st;
    la::PrefillArgs a{q, k, v, decay, cu_seqlens, num_seqs, total_tokens, num_heads,
                      head_dim, chunk, out, final_state, static_cast<cudaStream_t>(stream),
                      initial_state};
    return run_prefill(a, dtype);
}

la_status lightning_attn_prefill_snapshots(const void *q, const void *k, const void *v,
                                           const float *decay, const int32_t *cu_seqlens,
                                           int32_t num_seqs, int32_t total_tokens,
                                           int32_t num_heads, int32_t head_dim, int32_t chunk,
                                           la_dtype dtype, const float *initial_state, void *out,
                                           float *final_state, int32_t snapshot_interval,
                                           float *snapshots, void *stream) {
    if (snapshot_interval <= 0)
        return fail(LA_ERR_INVALID_ARG, "snapshot_interval must be > 0 (got %d)", snapshot_interval);
    bool work = false;
    const la_status st = check_prefill(q, k, v, decay, cu_seqlens, num_seqs, total_tokens,
                                       num_heads, head_dim, chunk, dtype, initial_state, out,
                                       final_state, stream, &work);
    if (st != LA_OK || !work) return st;
    if (!snapshots || !aligned16(snapshots))
        return fail(LA_ERR_INVALID_ARG, "snapshots must be a 16-byte aligned device array");
    // the kernel that serves the call and its block
    const bool tc = la::uses_tensor_cores(dtype == LA_DTYPE_BF16, head_dim, chunk);
    const int block = chunk != 0 ? chunk : tc ? 128 : 64;
    if (!tc && (chunk == 128 || chunk == 256))
        return fail(LA_ERR_UNSUPPORTED, "chunk %d needs the tensor-core path (bf16, head_dim 128)",
                    chunk);
    if (snapshot_interval % block != 0)
        return fail(LA_ERR_INVALID_ARG,
                    "snapshot_interval %d is not a multiple of the block (%d tokens) this "
                    "call runs with", snapshot_interval, block);
    la::PrefillArgs a{q, k, v, decay, cu_seqlens, num_seqs, total_tokens, num_heads,
                      head_dim, chunk, out, final_state, static_cast<cudaStream_t>(stream),
                      initial_state};
    a.snapshots = snapshots;
    a.snapshot_interval = snapshot_interval;
    return run_prefill(a, dtype);
}

int64_t lightning_attn_snapshot_count(const int32_t *cu_seqlens_host, int32_t num_seqs,
                                      int32_t snapshot_interval) {
    if (num_seqs < 0 || snapshot_interval <= 0 || (num_seqs > 0 && !cu_seqlens_host)) return -1;
    int64_t n = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int64_t L = (int64_t)cu_seqlens_host[s + 1] - cu_seqlens_host[s];
        if (L < 0) return -1;
        n += L / snapshot_interval;
    }
    return n;
}

la_status lightning_attn_prefill(const void *q, const void *k, const void *v,
                                 const float *decay, const int32_t *cu_seqlens,
                                 int32_t num_seqs, int32_t total_tokens,
                                 int32_t num_heads, int32_t head_dim,
                                 int32_t chunk, la_dtype dtype, void *out,
                                 float *final_state, void *stream) {
    return lightning_attn_prefill_with_state(q, k, v, decay, cu_seqlens, num_seqs, total_tokens,
                                             num_heads, head_dim, chunk, dtype, nullptr, out,
                                             final_state, stream);
}

la_status lightning_attn_prefill_channel_decay(const void *q, const void *k, const void *v,
                                               const float *decay, const int32_t *cu_seqlens,
                                               int32_t num_seqs, int32_t total_tokens,
                                               int32_t num_heads, int32_t head_dim, int32_t chunk,
                                               la_dtype dtype, const float *initial_state,
                                               void *out, float *final_state, void *stream) {
    bool work = false;
    const la_status st = check_prefill(q, k, v, decay, cu_seqlens, num_seqs, total_tokens,
                                       num_heads, head_dim, chunk, dtype, initial_state, out,
                                       final_state, stream, &work);
    if (st != LA_OK || !work) return st;
    if (chunk == 128 || chunk == 256)
        return fail(LA_ERR_UNSUPPORTED,
                    "channel-wise decay takes chunk 0, 16, 32 or 64");
    la::PrefillArgs a{q, k, v, decay, cu_seqlens, num_seqs, total_tokens, num_heads,
                      head_dim, chunk, out, final_state, static_cast<cudaStream_t>(stream),
                      initial_state};
    a.channel_decay = true;
    // bf16 with head_dim 128 and 64-token blocks: the tensor-core kernel
    if (dtype == LA_DTYPE_BF16 && head_dim == 128 && (chunk == 0 || chunk == 64))
        return from_cuda(la::prefill_cw_tc_bf16(a), "prefill (channel-wise decay, tcgen05)");
    if (dtype == LA_DTYPE_FP32)
        return from_cuda(la::prefill_simt_f32(a), "prefill (channel-wise decay, fp32)");
    return from_cuda(la::prefill_simt_bf16(a), "prefill (channel-wise decay, bf16)");
}

la_status lightning_attn_decode_channel_decay(const void *q, const void *k, const void *v,
                                              const float *decay, float *state, int32_t batch,
                                              int32_t num_heads, int32_t head_dim,
                                              la_dtype dtype, void *out, void *stream) {
    if (batch < 0) return fail(LA_ERR_INVALID_ARG, "batch < 0 (%d)", batch);
    if (num_heads < 1) return fail(LA_ERR_INVALID_ARG, "num_heads < 1 (%d)", num_heads);
    if (head_dim != 64 && head_dim != 128)
        return fail(LA_ERR_INVALID_ARG, "head_dim must be 64 or 128 (got %d)", head_dim);
    if (dtype != LA_DTYPE_BF16 && dtype != LA_DTYPE_FP32)
        return fail(LA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (batch == 0) return LA_OK;
    if (!q || !k || !v || !decay || !state || !out)
        return fail(LA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(decay) ||
        !aligned16(state) || !aligned16(out))
        return fail(LA_ERR_INVALID_ARG, "every pointer must be 16-byte aligned");
    if ((long long)batch * num_heads > 0x7fffffffLL)
        return fail(LA_ERR_INVALID_ARG, "batch * num_heads too large");
    la::DecodeArgs a{q, k, v, decay, state, batch, num_heads, head_dim, out,
                     static_cast<cudaStream_t>(stream)};
    a.channel_decay = true;
    if (dtype == LA_DTYPE_FP32) return from_cuda(la::decode_f32(a), "decode (channel-wise, fp32)");
    return from_cuda(la::decode_bf16(a), "decode (channel-wise, bf16)");
}

la_status lightning_attn_decode(const void *q, const void *k, const void *v,
                                const float *decay, float *state, int32_t batch,
                                int32_t num_heads, int32_t head_dim, la_dtype dtype,
                                void *out, void *stream) {
    if (batch < 0) return fail(LA_ERR_INVALID_ARG, "batch < 0 (%d)", batch);
    if (num_heads < 1) return fail(LA_ERR_INVALID_ARG, "num_heads < 1 (%d)", num_heads);
    if (head_dim != 64 && head_dim != 128)
        return fail(LA_ERR_INVALID_ARG, "head_dim must be 64 or 128 (got %d)", head_dim);
    if (dtype != LA_DTYPE_BF16 && dtype != LA_DTYPE_FP32)
        return fail(LA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (batch == 0) return LA_OK;
    if (!q || !k || !v || !decay || !state || !out)
        return fail(LA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(decay) ||
        !aligned16(state) || !aligned16(out))
        return fail(LA_ERR_INVALID_ARG, "every pointer must be 16-byte aligned");
    if ((long long)batch * num_heads > 0x7fffffffLL)
        return fail(LA_ERR_INVALID_ARG, "batch * num_heads too large");
    la::DecodeArgs a{q, k, v, decay, state, batch, num_heads, head_dim, out,
                     static_cast<cudaStream_t>(stream)};
    if (dtype == LA_DTYPE_FP32) return from_cuda(la::decode_f32(a), "decode (fp32)");
    return from_cuda(la::decode_bf16(a), "decode (bf16)");
}

int64_t lightning_attn_backward_workspace_bytes(int32_t total_tokens, int32_t num_heads,
                                                int32_t head_dim, la_dtype dtype) {
    if (total_tokens < 0 || num_heads < 1 || (head_dim != 64 && head_dim != 128) ||
        (dtype != LA_DTYPE_BF16 && dtype != LA_DTYPE_FP32))
        return -1;
    return (int64_t)(3 * backward_slot_bytes(total_tokens, num_heads, head_dim, dtype));
}

}  // extern "C"

namespace la {

la_status backward_check(const void *q, const void *k, const void *v, const float *decay,
                         const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                         int32_t num_heads, int32_t head_dim, int32_t chunk, la_dtype dtype,
                         const void *d_out, void *d_q, void *d_k, void *d_v, bool *work,
                         bool *needs_workspace) {
    *work = false;
    *needs_workspace = false;
    if (num_seqs < 0) return fail(LA_ERR_INVALID_ARG, "num_seqs < 0 (%d)", num_seqs);
    if (total_tokens < 0) return fail(LA_ERR_INVALID_ARG, "total_tokens < 0 (%d)", total_tokens);
    if (num_heads < 1) return fail(LA_ERR_INVALID_ARG, "num_heads < 1 (%d)", num_heads);
    if (head_dim != 64 && head_dim != 128)
        return fail(LA_ERR_INVALID_ARG, "head_dim must be 64 or 128 (got %d)", head_dim);
    if (dtype != LA_DTYPE_BF16 && dtype != LA_DTYPE_FP32)
        return fail(LA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (chunk != 0 && chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128 && chunk != 256)
        return fail(LA_ERR_INVALID_ARG, "chunk must be 0, 16, 32, 64, 128 or 256 (got %d)", chunk);
    if (num_seqs == 0 || total_tokens == 0) return LA_OK;
    if (!cu_seqlens || !decay) return fail(LA_ERR_INVALID_ARG, "null decay or cu_seqlens");
    const void *ptrs[] = {q, k, v, d_out, d_q, d_k, d_v};
    for (const void *p : ptrs)
        if (!p) return fail(LA_ERR_INVALID_ARG, "null tensor pointer");
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(LA_ERR_INVALID_ARG, "every pointer must be 16-byte aligned");
    if (!aligned16(decay) || !aligned16(cu_seqlens))
        return fail(LA_ERR_INVALID_ARG, "every pointer must be 16-byte aligned");
    if ((long long)num_seqs * num_heads > 0x7fffffffLL / 4)
        return fail(LA_ERR_INVALID_ARG, "num_seqs * num_heads too large");
    // outputs are distinct arrays, none of them an input
    const void *outs[] = {d_q, d_k, d_v};
    const void *ins[] = {q, k, v, d_out};
    for (int i = 0; i < 3; ++i) {
        for (int j = 0; j < 4; ++j)
            if (outs[i] == ins[j]) return fail(LA_ERR_INVALID_ARG, "a gradient aliases an input");
        for (int j = i + 1; j < 3; ++j)
            if (outs[i] == outs[j]) return fail(LA_ERR_INVALID_ARG, "two gradients share an array");
    }
    // the tensor-core path computes dk and dv in place and needs no
    // workspace; off it, blocks of 128 and 256 tokens have no kernel
    const bool tc = uses_tensor_cores(dtype == LA_DTYPE_BF16, head_dim, chunk);
    if (!tc && (chunk == 128 || chunk == 256))
        return fail(LA_ERR_UNSUPPORTED,
                    "chunk %d needs the tensor-core path (bf16, head_dim 128)", chunk);
    *work = true;
    *needs_workspace = !tc;
    return LA_OK;
}

}  // namespace la

extern "C" {

la_status lightning_attn_backward(const void *q, const void *k, const void *v,
                                  const float *decay, const int32_t *cu_seqlens,
                                  int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                  int32_t head_dim, int32_t chunk, la_dtype dtype,
                                  const void *d_out, void *d_q, void *d_k, void *d_v,
                                  void *workspace, int64_t workspace_bytes, void *stream) {
    bool work = false, needs_ws = false;
    const la_status chk = la::backward_check(q, k, v, decay, cu_seqlens, num_seqs, total_tokens,
                                             num_heads, head_dim, chunk, dtype, d_out, d_q, d_k,
                                             d_v, &work, &needs_ws);
    if (chk != LA_OK || !work) return chk;
    const bool tc = !needs_ws;
    const size_t slot = backward_slot_bytes(total_tokens, num_heads, head_dim, dtype);
    if (!tc) {
        if (!workspace) return fail(LA_ERR_INVALID_ARG, "null workspace (CUDA-core path)");
        if (workspace_bytes < 0 || (size_t)workspace_bytes < 3 * slot)
            return fail(LA_ERR_INVALID_ARG, "workspace too small: %lld bytes, %zu needed",
                        (long long)workspace_bytes, 3 * slot);
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return fail(LA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    }

    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    void *rq = ws, *rg = ws + slot, *rkv = ws + 2 * slot;
    const size_t row = (size_t)num_heads * head_dim * elem_bytes(dtype);
    auto fwd = [&](const void *a, const void *b, const void *c, void *o, bool reverse_out) {
        la::PrefillArgs pa{a, b, c, decay, cu_seqlens, num_seqs, total_tokens, num_heads,
                           head_dim, chunk, o, nullptr, st, nullptr, reverse_out};
        return run_prefill(pa, dtype);
    };
    // o_t = sum_{u >= t} lambda^(u-t) (a_t . b_u) c_u, rows in place
    auto anti = [&](const void *a, const void *b, const void *c, void *o) {
        la::PrefillArgs pa{a, b, c, decay, cu_seqlens, num_seqs, total_tokens, num_heads,
                           head_dim, chunk, o, nullptr, st, nullptr};
        pa.anti_causal = true;
        return run_prefill(pa, dtype);
    };
    auto rev = [&](const void *in, void *out) {
        return from_cuda(la::reverse_sequences(in, out, cu_seqlens, num_seqs, total_tokens, row, st),
                         "backward (time reversal)");
    };
    la_status r;
    // dq_t = sum_{u<=t} lambda^(t-u) (dout_t . v_u) k_u: the forward form
    // with (q, k, v) -> (dout, v, k)
    if ((r = fwd(d_out, v, k, d_q, false)) != LA_OK) return r;
    if (tc) {
        // tensor-core path: dv_u = sum_{t>=u} lambda^(t-u) (q_t . k_u) dout_t and
        // dk_u = sum_{t>=u} lambda^(t-u) (dout_t . v_u) q_t are anti-causal
        // forms, computed in place (the workspace is not touched)
        if ((r = anti(k, q, d_out, d_v)) != LA_OK) return r;
        return anti(v, d_out, q, d_k);
    }
    // CUDA-core path: the anti-causal sums as the forward form in reversed time
    // dv_u = sum_{t>=u} lambda^(t-u) (q_t . k_u) dout_t: the forward form in
    // reversed time with (q, k, v) -> (k, q, dout); the launch writes its
    // output rows back in forward time order
    if ((r = rev(q, rq)) != LA_OK || (r = rev(d_out, rg)) != LA_OK || (r = rev(k, rkv)) != LA_OK)
        return r;
    if ((r = fwd(rkv, rq, rg, d_v, true)) != LA_OK) return r;
    // dk_u = sum_{t>=u} lambda^(t-u) (dout_t . v_u) q_t: reversed time with
    // (q, k, v) -> (v, dout, q)
    if ((r = rev(v, rkv)) != LA_OK) return r;
    if ((r = fwd(rkv, rg, rq, d_k, true)) != LA_OK) return r;
    return LA_OK;
}

la_status lightning_attn_mixed_step(const void *q, const void *k, const void *v,
                                    const float *decay, const int32_t *cu_seqlens,
                                    int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                    int32_t head_dim, la_dtype dtype, float *state, void *out,
                                    const int32_t *cu_seqlens_host, void *prefill_stream,
                                    void *decode_stream) {
    if (num_seqs < 0) return fail(LA_ERR_INVALID_ARG, "num_seqs < 0 (%d)", num_seqs);
    if (total_tokens < 0) return fail(LA_ERR_INVALID_ARG, "total_tokens < 0 (%d)", total_tokens);
    if (num_heads < 1) return fail(LA_ERR_INVALID_ARG, "num_heads < 1 (%d)", num_heads);
    if (head_dim != 64 && head_dim != 128)
        return fail(LA_ERR_INVALID_ARG, "head_dim must be 64 or 128 (got %d)", head_dim);
    if (dtype != LA_DTYPE_BF16 && dtype != LA_DTYPE_FP32)
        return fail(LA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (num_seqs == 0 || total_tokens == 0) return LA_OK;
    if (!q || !k || !v || !out || !decay || !cu_seqlens || !state)
        return fail(LA_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
        !aligned16(decay) || !aligned16(cu_seqlens) || !aligned16(state))
        return fail(LA_ERR_INVALID_ARG, "every pointer must be 16-byte aligned");
    if ((long long)num_seqs * num_heads > 0x7fffffffLL / 4)
        return fail(LA_ERR_INVALID_ARG, "num_seqs * num_heads too large");

    const cudaStream_t ps = static_cast<cudaStream_t>(prefill_stream);
    const cudaStream_t ds = static_cast<cudaStream_t>(decode_stream);
    // sequences of >= 2 new tokens: chunkwise prefill continuing from their
    // cached state, updated in place
    la::PrefillArgs pa{q, k, v, decay, cu_seqlens, num_seqs, total_tokens, num_heads, head_dim,
                       0, out, state, ps, state, false, 2};
    // With the lengths on the host, launch prefill work only for the
    // sequences that need it: the kernels take sequences longest first, so
    // the first n_long ranks are exactly those with >= 2 new tokens.
    bool any_long = true;
    if (cu_seqlens_host && num_seqs <= la::kMaxSortedSeqs) {
        int n_long = 0;
        for (int s = 0; s < num_seqs; ++s) n_long += cu_seqlens_host[s + 1] - cu_seqlens_host[s] >= 2;
        pa.rank_limit = n_long;
        any_long = n_long > 0;
    }
    // sequences of exactly 1 new token: the decode step
    la::DecodeArgs da{q, k, v, decay, state, num_seqs, num_heads, head_dim, out, ds,
                      cu_seqlens, total_tokens};
    auto decode = [&]() {
        return from_cuda(dtype == LA_DTYPE_FP32 ? la::decode_f32(da) : la::decode_bf16(da),
                         "mixed step (decode)");
    };
    if (ps == ds) {
        la_status r = decode();
        return (r != LA_OK || !any_long) ? r : run_prefill(pa, dtype);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return from_cuda(e, "mixed step");
    if (dev < 0 || dev >= kMaxDevices) return fail(LA_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lock(g_mixed_mu);
    if (!g_fork[dev]) {
        if ((e = cudaEventCreateWithFlags(&g_fork[dev], cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&g_join[dev], cudaEventDisableTiming)) != cudaSuccess)
            return from_cuda(e, "mixed step (events)");
    }
    // fork: the decode stream starts after the work already queued on the
    // prefill stream; join: the prefill stream continues after the decode
    if ((e = cudaEventRecord(g_fork[dev], ps)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(ds, g_fork[dev], 0)) != cudaSuccess)
        return from_cuda(e, "mixed step (fork)");
    la_status r = decode();
    if (r != LA_OK) return r;
    if (any_long && (r = run_prefill(pa, dtype)) != LA_OK) return r;
    if ((e = cudaEventRecord(g_join[dev], ds)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(ps, g_join[dev], 0)) != cudaSuccess)
        return from_cuda(e, "mixed step (join)");
    return LA_OK;
}

la_status lightning_attn_device_status(void *stream) {
    unsigned int err = 0, err_cw = 0;
    la_status st =
        from_cuda(la::take_device_error(static_cast<cudaStream_t>(stream), &err), "device_status");
    if (st != LA_OK) return st;
    st = from_cuda(la::take_cw_device_error(&err_cw), "device_status");
    if (st != LA_OK) return st;
    err |= err_cw;
    if (err) return fail(LA_ERR_TIMEOUT, "a bounded device-side wait gave up");
    return LA_OK;
}

la_status lightning_attn_selftest_wait_timeout(uint64_t timeout_ns, void *stream) {
    return from_cuda(la::selftest_wait_timeout(timeout_ns, static_cast<cudaStream_t>(stream)),
                     "selftest_wait_timeout");
}

}  // extern "C"
