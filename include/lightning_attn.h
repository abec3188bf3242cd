/*
 * lightning_attn.h -- C ABI of the GB300 (sm_103a) lightning-attention library
 * (liblightning_attn.so).
 *
 * The operation (MiniMax-01 technical report, CSDN full translation, §2.2.1
 * "Lightning Attention", eqs. 4-5, with the per-head diagonal decay of the
 * Fig. 12 caption): for every sequence and head h, with lambda = decay[h],
 *
 *     o_t = sum_{u <= t} lambda^(t-u) (q_t . k_u) v_u            (left product)
 *         = q_t kv_t,  kv_t = lambda kv_{t-1} + k_t^T v_t,  kv_{-1} = 0
 *                                                         (right product)
 *
 * computed chunkwise: inside a chunk the masked left product
 * [(Q_i K_i^T) (.) M] V_i, across chunks the right product through a d x d
 * state carried on chip (§2.2.1 "intra-block" / "inter-block").  Packed
 * variable-length batches follow §3.2 ("data packing"): each sequence starts
 * from a zero state.  Decode is the recursion applied to one new token per
 * sequence, updating a cached state in place (§3.3.1 fused decode KV update,
 * §3.3.2 separate prefill and decode kernels).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates no device memory and keeps no per-call state.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL means
 *     the legacy default stream).  Calls never synchronise; results are ready
 *     when the stream reaches that point.
 *   - Argument errors are detected on the host before anything is launched
 *     and return LA_ERR_INVALID_ARG / LA_ERR_UNSUPPORTED with nothing written.
 *     A failed launch returns LA_ERR_CUDA.  Errors that only the GPU can see
 *     (e.g. a cu_seqlens array that is not monotone) are not checked: results
 *     are then unspecified but every access stays inside the buffers whose
 *     sizes the arguments state.
 *   - Every pointer must be 16-byte aligned.  Outputs must not alias inputs.
 *   - No C++ exception crosses this boundary.
 *   - lightning_attn_last_error() returns a human-readable reason for the
 *     last non-LA_OK status returned on the calling host thread.
 */
#ifndef LIGHTNING_ATTN_H
#define LIGHTNING_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum la_status {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad size or dtype */
    LA_ERR_UNSUPPORTED = 2,   /* valid request the library has no kernel for */
    LA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed          */
    LA_ERR_TIMEOUT = 4        /* reserved: a bounded device-side wait gave up  */
} la_status;

typedef enum la_dtype {
    LA_DTYPE_BF16 = 0,        /* q, k, v, out are bf16; fp32 accumulation */
    LA_DTYPE_FP32 = 1         /* q, k, v, out are fp32; fp32 FFMA throughout */
} la_dtype;

/*
 * Chunkwise prefill over a packed batch of sequences.
 *   (MiniMax-01 report §2.2.1 block split; §3.2 data packing; §3.3.1 fused
 *    prefill preprocessing -- here the tile staging and the decay values are
 *    produced inside the kernel.)
 *
 * q, k, v      [total_tokens, num_heads, head_dim], dtype `dtype`, row-major;
 *              token-major packed: sequence s owns rows
 *              [cu_seqlens[s], cu_seqlens[s+1]).
 * decay        [num_heads] fp32, lambda_h, each in (0, 1] (not checked here:
 *              this entry point does not read device memory on the host;
 *              values outside give the formula's value, possibly inf/nan.
 *              The Python binding checks the range before the call).
 * cu_seqlens   [num_seqs + 1] int32 DEVICE array, cu_seqlens[0] = 0,
 *              non-decreasing, cu_seqlens[num_seqs] = total_tokens.  Empty
 *              sequences are allowed (their final state is zero).
 * num_seqs     >= 0 (0: nothing is done).
 * total_tokens >= 0.
 * num_heads    >= 1.
 * head_dim     64 or 128.
 * chunk        block size B: 0 picks the default for the path
 *              (128 on the tensor-core path, 64 otherwise).  The
 *              tensor-core path (bf16, head_dim 128) takes 16, 32, 64, 128
 *              or 256 (its tiles are 128 tokens; a smaller block runs as
 *              masked tiles advancing B tokens, at 128 / B times the
 *              tensor-core work; a 256-token block as two tiles whose
 *              coupling term goes through the state after the first, the
 *              same sum regrouped); the fp32 / head_dim 64 CUDA-core path
 *              takes 16, 32 or 64 (128 and 256: LA_ERR_UNSUPPORTED).  The
 *              result does
 *              not depend on B beyond rounding (K3 report reading notes, CP
 *              for linear attention: any chunk split is mathematically
 *              equivalent).
 * dtype        LA_DTYPE_BF16 or LA_DTYPE_FP32.
 * out          [total_tokens, num_heads, head_dim], dtype `dtype`: o_t.
 * final_state  nullable; [num_seqs, num_heads, head_dim, head_dim] fp32:
 *              final_state[s][h][i][j] = sum_u lambda_h^(L_s-1-u) k_u[i] v_u[j]
 *              (the state after the last token of sequence s, i.e. the prefix
 *              cache a following decode step continues from).
 * stream       cudaStream_t as void*.
 */
la_status lightning_attn_prefill(const void *q, const void *k, const void *v,
                                 const float *decay, const int32_t *cu_seqlens,
                                 int32_t num_seqs, int32_t total_tokens,
                                 int32_t num_heads, int32_t head_dim,
                                 int32_t chunk, la_dtype dtype, void *out,
                                 float *final_state, void *stream);

/*
 * Prefill that continues every sequence from a cached state (the prefix KV
 * cache of MiniMax-01 report §3.3.1: a new segment of a sequence whose
 * earlier tokens were already consumed into a d x d state).  With S0 =
 * initial_state[s][h] the recursion starts at kv_{-1} = S0, so
 *
 *     o_t = sum_{u <= t} lambda^(t-u) (q_t . k_u) v_u + lambda^(t+1) q_t S0
 *     final_state = lambda^L S0 + sum_u lambda^(L-1-u) k_u^T v_u
 *
 * (the result of one prefill over the earlier tokens and this segment
 * together).  Arguments are those of lightning_attn_prefill plus
 *
 * initial_state  nullable; [num_seqs, num_heads, head_dim, head_dim] fp32,
 *                same layout as final_state; NULL means zero states (then
 *                the call equals lightning_attn_prefill).  It may be the
 *                same array as final_state (the cache is updated in place:
 *                every state is read before it is overwritten); any other
 *                overlap of the two is rejected with LA_ERR_INVALID_ARG.  An
 *                empty sequence's final state is its initial state.
 */
la_status lightning_attn_prefill_with_state(const void *q, const void *k, const void *v,
                                            const float *decay, const int32_t *cu_seqlens,
                                            int32_t num_seqs, int32_t total_tokens,
                                            int32_t num_heads, int32_t head_dim,
                                            int32_t chunk, la_dtype dtype,
                                            const float *initial_state, void *out,
                                            float *final_state, void *stream);

/*
 * Prefill that also keeps the state at every block boundary: the prefix cache
 * of a linear-attention layer kept once per block of tokens (K3 report notes
 * on the inference engine: storing every step's state would give up linear
 * attention's advantage, storing none gives no prefix reuse, so one cache
 * entry per block).  Arguments and results are those of
 * lightning_attn_prefill_with_state, plus
 *
 * snapshot_interval  tokens per block, > 0 and a multiple of the block the
 *                    call computes with (the chunk; for chunk 0, 128 on the
 *                    tensor-core path -- bf16, head_dim 128 -- and 64
 *                    otherwise); LA_ERR_INVALID_ARG otherwise.
 * snapshots          [N, num_heads, head_dim, head_dim] fp32 device array,
 *                    16-byte aligned, N = lightning_attn_snapshot_count(...)
 *                    of the same cu_seqlens (host copy).  Sequence s owns
 *                    entries [b_s, b_s + floor(L_s / snapshot_interval)) with
 *                    b_s = sum_{s' < s} floor(L_s' / snapshot_interval); entry
 *                    b_s + j holds the state after the first
 *                    (j + 1) * snapshot_interval tokens of s -- the final_state
 *                    a prefill of those tokens alone (from the same initial
 *                    state) returns.  A trailing partial block gets none.
 */
la_status lightning_attn_prefill_snapshots(const void *q, const void *k, const void *v,
                                           const float *decay, const int32_t *cu_seqlens,
                                           int32_t num_seqs, int32_t total_tokens,
                                           int32_t num_heads, int32_t head_dim, int32_t chunk,
                                           la_dtype dtype, const float *initial_state, void *out,
                                           float *final_state, int32_t snapshot_interval,
                                           float *snapshots, void *stream);

/* Number of snapshots lightning_attn_prefill_snapshots writes for these
 * sequences (host copy of cu_seqlens, num_seqs + 1 entries): the sum of
 * floor(L_s / snapshot_interval).  -1 for invalid arguments. */
int64_t lightning_attn_snapshot_count(const int32_t *cu_seqlens_host, int32_t num_seqs,
                                      int32_t snapshot_interval);

/*
 * Prefill with a channel-wise decay: one lambda per head and KEY channel
 * (K3 report reading notes: the scalar decay generalised to a channel-wise
 * one that can fall back to the uniform decay; it acts on the channels Q and
 * K share).  With lam_i = decay[h * head_dim + i] the state recursion is
 *     kv_t[i][j] = lam_i kv_{t-1}[i][j] + k_t[i] v_t[j],   o_t = q_t kv_t
 * i.e. o_t = sum_{u <= t} (sum_i q_t[i] k_u[i] lam_i^(t-u)) v_u
 *            + sum_i q_t[i] lam_i^(t+1) S0[i][:]  (from a cached state S0).
 * Arguments as for lightning_attn_prefill_with_state, except
 *   decay  [num_heads, head_dim] fp32, each in (0, 1].
 * Kernels: bf16 with head_dim 128 and chunk 0 or 64 runs the tensor-core
 * kernel (64-token blocks; intra-block scores from 16-token sub-blocks whose
 * decay factors are split between the query and key sides, every operand a
 * hi/lo bf16 pair but the key side of the off-diagonal scores).  For its
 * diagonal sub-blocks lambda is raised to 2^-12 where smaller: a score term
 * at distance 1..15 then moves by less than 2^-12 |q_t[i] k_u[i]|.  Those
 * factors reach mu_i^-8 on the query side and mu_i^-7 on the key side, with
 * mu_i = max(lambda_i, 2^-12), so the kernel needs |q_t[i]| mu_i^-8 and
 * |k_u[i]| mu_i^-7 below the bf16 maximum (about 3.4e38): always true for
 * |q| < 2^32 and |k| < 2^44.  Every other case
 * runs the CUDA-core (FFMA) kernel: chunk 0 (= 64), 16, 32 or 64 (fp32, or
 * head_dim 64); 128 and 256 return LA_ERR_UNSUPPORTED.
 */
la_status lightning_attn_prefill_channel_decay(const void *q, const void *k, const void *v,
                                               const float *decay, const int32_t *cu_seqlens,
                                               int32_t num_seqs, int32_t total_tokens,
                                               int32_t num_heads, int32_t head_dim, int32_t chunk,
                                               la_dtype dtype, const float *initial_state,
                                               void *out, float *final_state, void *stream);

/*
 * Decode step with a channel-wise decay (decay [num_heads, head_dim]):
 *     state[b][h][i][j] <- lam_i state[b][h][i][j] + k[i] v[j],  out = q state.
 * Other arguments as for lightning_attn_decode.
 */
la_status lightning_attn_decode_channel_decay(const void *q, const void *k, const void *v,
                                              const float *decay, float *state, int32_t batch,
                                              int32_t num_heads, int32_t head_dim,
                                              la_dtype dtype, void *out, void *stream);

/*
 * One decode step for a batch of sequences, each with one new token.
 *   (MiniMax-01 report §3.3.2: length-1 inputs get their own memory-bound
 *    kernel; §3.3.1: the KV computation and the prefix-KV-cache update are
 *    fused into one kernel.)
 *
 * For every b < batch, h < num_heads, with lambda = decay[h]:
 *     state[b][h] <- lambda * state[b][h] + k[b][h]^T v[b][h]     (in place)
 *     out[b][h]    = q[b][h] . state[b][h]                 (after the update)
 *
 * q, k, v, out [batch, num_heads, head_dim], dtype `dtype`.
 * decay        [num_heads] fp32.
 * state        [batch, num_heads, head_dim, head_dim] fp32, read and written.
 * batch >= 0 (0: nothing is done), num_heads >= 1, head_dim 64 or 128.
 */
la_status lightning_attn_decode(const void *q, const void *k, const void *v,
                                const float *decay, float *state,
                                int32_t batch, int32_t num_heads,
                                int32_t head_dim, la_dtype dtype, void *out,
                                void *stream);

/*
 * Gradients for training (MiniMax-01 report §2.2.1; §2.2.2 measures the
 * training speed of lightning attention): given dout = dL/do for the outputs
 * of lightning_attn_prefill on the same arguments (zero initial states),
 *
 *     dq_t = sum_{u <= t} lambda^(t-u) (dout_t . v_u) k_u
 *     dk_u = sum_{t >= u} lambda^(t-u) (dout_t . v_u) q_t
 *     dv_u = sum_{t >= u} lambda^(t-u) (q_t . k_u) dout_t
 *
 * per sequence and head.  dq is the forward form applied to (dout, v, k);
 * dk and dv are anti-causal forms (sums over t >= u).  On the tensor-core
 * path (bf16, head_dim 128, chunk 0-128) the call makes three launches of
 * the prefill kernel, one causal and two anti-causal, and does not touch
 * `workspace`; on the CUDA-core path it runs the forward form in reversed
 * time, with four time-reversal copies through `workspace`.  Same dtype /
 * head_dim / chunk rules and precision as lightning_attn_prefill.
 *
 * q, k, v, d_out          [total_tokens, num_heads, head_dim], dtype `dtype`
 * d_q, d_k, d_v           outputs, same shape and dtype; distinct arrays,
 *                         none of them equal to an input
 * workspace               caller-owned device memory, 256-byte aligned, of at
 *                         least lightning_attn_backward_workspace_bytes(...)
 *                         bytes; its contents are scratch (overwritten).  Not
 *                         used on the tensor-core path, where it may be NULL
 *                         with workspace_bytes 0.
 * other arguments         as for lightning_attn_prefill.
 * Gradients with respect to decay, to a cached initial state or from a
 * final-state loss are not computed.
 */
la_status lightning_attn_backward(const void *q, const void *k, const void *v,
                                  const float *decay, const int32_t *cu_seqlens,
                                  int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                  int32_t head_dim, int32_t chunk, la_dtype dtype,
                                  const void *d_out, void *d_q, void *d_k, void *d_v,
                                  void *workspace, int64_t workspace_bytes, void *stream);

/* Bytes of workspace lightning_attn_backward needs (three [T, H, d] arrays,
 * each rounded up to 256 bytes); -1 for invalid arguments. */
int64_t lightning_attn_backward_workspace_bytes(int32_t total_tokens, int32_t num_heads,
                                                int32_t head_dim, la_dtype dtype);

/*
 * lightning_attn_backward without a caller workspace (the paper has no
 * counterpart; this is a convenience of this library).  For callers that
 * cannot allocate device memory at call time -- code under another
 * framework's memory manager that forbids raw cudaMalloc, or a loop that
 * must not call cudaMalloc because it can synchronise the device -- the
 * scratch comes from one fixed array of lightning_attn_backward_noalloc_max_bytes()
 * bytes (64 MiB) that every GPU loading the library holds until the process
 * exits.  Arguments and results are those of lightning_attn_backward.  On the
 * tensor-core path (bf16, head_dim 128, chunk 0-128) no scratch is used
 * and no size limit applies; otherwise a call whose
 * lightning_attn_backward_workspace_bytes() exceeds the array returns
 * LA_ERR_INVALID_ARG before touching the GPU (argument errors, empty calls
 * and unsupported block sizes are reported first, exactly as by
 * lightning_attn_backward).  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current, and so does
 * the first call after the device's context has been destroyed and made
 * again (cudaDeviceReset); make such a call before any stream capture.  The
 * array is shared by all calls: calls that overlap on the GPU race on it;
 * calls ordered on one stream do not.  Nothing is allocated.
 */
la_status lightning_attn_backward_noalloc(const void *q, const void *k, const void *v,
                                          const float *decay, const int32_t *cu_seqlens,
                                          int32_t num_seqs, int32_t total_tokens,
                                          int32_t num_heads, int32_t head_dim, int32_t chunk,
                                          la_dtype dtype, const void *d_out, void *d_q,
                                          void *d_k, void *d_v, void *stream);

/* Size in bytes of the fixed scratch array of lightning_attn_backward_noalloc. */
int64_t lightning_attn_backward_noalloc_max_bytes(void);

/*
 * One serving step over a packed batch in which every sequence continues from
 * its cached state (MiniMax-01 report §3.3.2: inputs of length 1 and of
 * length > 1 get separate kernels on separate CUDA streams; §3.3.1 prefix KV
 * cache).  For every sequence s with L_s = cu_seqlens[s+1] - cu_seqlens[s]
 * new tokens, the result is that of lightning_attn_prefill_with_state with
 * initial_state = final_state = state:
 *   L_s == 1: the decode step (kv <- lambda kv + k^T v, o = q kv) on
 *             decode_stream;
 *   L_s >= 2: the chunkwise prefill on prefill_stream, state updated in place;
 *   L_s == 0: nothing (the state is unchanged).
 * Both launches read cu_seqlens on the device, so no host copy of the lengths
 * is needed.  The decode launch waits for the work already queued on
 * prefill_stream and prefill_stream waits for the decode launch before its
 * next work, so the whole step is ordered on prefill_stream (two events per
 * device are created on first use for this fork and join; calls from
 * several host threads are serialised while they enqueue).  With
 * decode_stream == prefill_stream the two launches simply run one after the
 * other.  A decode_stream of higher priority than prefill_stream lets the
 * decode kernel's small blocks start before the prefill's large ones occupy
 * the SMs (measured: 20 sequences x 64 heads, 2 with 50 new tokens, 45 ->
 * 37 us).  chunk is the path's default; dtype rules as for prefill.
 *
 * q, k, v, out    [total_tokens, num_heads, head_dim], dtype `dtype`
 * state           [num_seqs, num_heads, head_dim, head_dim] fp32, read and written
 * cu_seqlens_host nullable HOST copy of cu_seqlens.  When given (and
 *                 num_seqs <= 128) the prefill launch covers only the
 *                 sequences with >= 2 new tokens; without it every sequence
 *                 gets prefill CTAs that exit at once for the short ones.
 */
la_status lightning_attn_mixed_step(const void *q, const void *k, const void *v,
                                    const float *decay, const int32_t *cu_seqlens,
                                    int32_t num_seqs, int32_t total_tokens, int32_t num_heads,
                                    int32_t head_dim, la_dtype dtype, float *state, void *out,
                                    const int32_t *cu_seqlens_host, void *prefill_stream,
                                    void *decode_stream);

/*
 * Synchronises `stream`, then reports whether a kernel of this library raised
 * its device error word since the last call (and clears it).  The
 * tensor-core prefill bounds every wait of its pipeline (about 2 s); a wait
 * that gives up ends the kernel cleanly (the context stays usable), leaves the
 * outputs of that launch unspecified and makes this call return
 * LA_ERR_TIMEOUT.  Returns LA_ERR_CUDA if the synchronisation fails.
 */
la_status lightning_attn_device_status(void *stream);

/*
 * Failure-detection self test: launches one CTA that waits on a barrier
 * nothing will ever complete, with the same bounded wait the prefill
 * pipeline uses, giving up after timeout_ns.  A following
 * lightning_attn_device_status() must return LA_ERR_TIMEOUT.
 */
la_status lightning_attn_selftest_wait_timeout(uint64_t timeout_ns, void *stream);

/* Static English name of a status code; never NULL. */
const char *lightning_attn_status_string(la_status status);

/* Reason for the last non-OK status on this host thread ("" if none). */
const char *lightning_attn_last_error(void);

/* ABI version of this header: (major << 16) | minor. */
int32_t lightning_attn_version(void);

#define LIGHTNING_ATTN_VERSION ((1 << 16) | 5)

#ifdef __cplusplus
}
#endif

#endif /* LIGHTNING_ATTN_H */
