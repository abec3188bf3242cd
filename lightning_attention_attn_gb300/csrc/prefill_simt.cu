// CUDA-core (FFMA) chunkwise lightning-attention prefill.
//
// This is the fp32 path (tensor-core tf32 would not meet a 1e-4 relative
// bound) and the path for head_dim 64.  One CTA owns one (sequence, head)
// and walks its chunks in order, keeping the d x d state in shared memory:
//   MiniMax-01 report (CSDN translation) §2.2.1 -- intra-block left product
//   [(Q_i K_i^T) (.) M] V_i, inter-block right product Q_i KV_{i-1} and the
//   recursive state update KV_i = lambda^{B_i} KV_{i-1} + (Lambda_K K_i)^T V_i,
//   with the decay values (§3.3.1) computed in the kernel.
// A sequence may continue from a cached state (initial_state): KV_{-1} = S0.
// Exponents of lambda are never negative (lambda^(j-l) for j >= l,
// lambda^(j+1), lambda^(B_i-1-l), lambda^(B_i)), so no factor can overflow;
// B_i is the true length of the (possibly short) last chunk.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "la_internal.h"
#include "sched.cuh"

namespace la {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

template <int D, int B, bool CW>
struct SimtSmem {
    static constexpr int DP = D + 1;  // padded row: conflict-free column walks
    float q[B][DP];
    float k[B][DP];
    float v[B][D];
    float kv[D][D];
    float p[B][B + 1];
    float pw[B + 1];  // pw[e] = lambda^e, e = 0..B
    float gk[B];      // lambda^(B_i-1-l) for l < B_i, else 0
    // channel-wise decay: pwc[e][i] = lambda_i^e, e = 0..B
    float pwc[CW ? B + 1 : 1][CW ? D : 1];
    int slot;
};

template <typename T, int D, int B, bool CW>
__global__ void __launch_bounds__(kThreads)
prefill_simt_kernel(const T *__restrict__ q, const T *__restrict__ k,
                    const T *__restrict__ v, const float *__restrict__ decay,
                    const int32_t *__restrict__ cu, int nseq, int T_total, int H,
                    const float *initial_state, T *__restrict__ out, float *final_state,
                    int reverse_out, int min_len) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<SimtSmem<D, B, CW> *>(smem_raw);
    const int tid = threadIdx.x;

    const int h = blockIdx.x % H;
    const int s = sequence_of_rank(cu, nseq, blockIdx.x / H, &sm.slot);
    // Clamp so that a malformed cu_seqlens can never index outside [0, T).
    int t0 = __ldg(cu + s), t1 = __ldg(cu + s + 1);
    t0 = min(max(t0, 0), T_total);
    t1 = min(max(t1, t0), T_total);
    const int L = t1 - t0;
    if (L < min_len) return;  // a mixed step's decode launch owns this sequence
    const float lam = CW ? 1.f : __ldg(decay + h);

    for (int e = tid; e <= B; e += kThreads) sm.pw[e] = powf(lam, (float)e);
    if constexpr (CW) {
        // channel-wise decay (K3 report reading notes): lambda per key
        // channel i, decay[h * D + i]; every factor below is lambda_i^e with
        // e >= 0 from this table
        for (int e = tid; e < (B + 1) * D; e += kThreads)
            sm.pwc[e / D][e % D] = powf(__ldg(decay + (long)h * D + e % D), (float)(e / D));
    }
    // KV_{-1}: the sequence's cached state (prefix KV cache, §3.3.1), else 0.
    // initial_state may be final_state itself: it is read here, before any
    // write of this CTA's final state.
    const float *s0 = initial_state ? initial_state + ((long)s * H + h) * D * D : nullptr;
    for (int e = tid; e < D * D; e += kThreads) (&sm.kv[0][0])[e] = s0 ? s0[e] : 0.f;
    __syncthreads();

    const long row_stride = (long)H * D;
    for (int c0 = 0; c0 < L; c0 += B) {
        const int Lc = min(B, L - c0);
        // ---- stage the chunk (rows >= Lc are zero) ----
        for (int e = tid; e < B * D; e += kThreads) {
            const int l = e / D, i = e % D;
            float qv = 0.f, kv_ = 0.f, vv = 0.f;
            if (l < Lc) {
                const long g = (long)(t0 + c0 + l) * row_stride + (long)h * D + i;
                qv = to_f(q[g]);
                kv_ = to_f(k[g]);
                vv = to_f(v[g]);
            }
            sm.q[l][i] = qv;
            sm.k[l][i] = kv_;
            sm.v[l][i] = vv;
        }
        for (int l = tid; l < B; l += kThreads)
            sm.gk[l] = (l < Lc) ? sm.pw[Lc - 1 - l] : 0.f;
        __syncthreads();

        // ---- intra-block scores with the decay mask: P = (Q K^T) (.) M ----
        for (int e = tid; e < B * B; e += kThreads) {
            const int j = e / B, l = e % B;
            float acc = 0.f;
            if (l <= j && j < Lc) {
                if constexpr (CW) {
                    const float *w = sm.pwc[j - l];
#pragma unroll 8
                    for (int i = 0; i < D; ++i) acc = fmaf(sm.q[j][i] * w[i], sm.k[l][i], acc);
                } else {
#pragma unroll 8
                    for (int i = 0; i < D; ++i) acc = fmaf(sm.q[j][i], sm.k[l][i], acc);
                    acc *= sm.pw[j - l];
                }
            }
            sm.p[j][l] = acc;
        }
        __syncthreads();

        // ---- output: P V_i + lambda^(j+1) Q_i KV_{i-1} ----
        for (int e = tid; e < B * D; e += kThreads) {
            const int j = e / D, n = e % D;
            if (j >= Lc) continue;
            float intra = 0.f;
            for (int l = 0; l <= j; ++l) intra = fmaf(sm.p[j][l], sm.v[l][n], intra);
            float inter = 0.f;
            float o;
            if constexpr (CW) {
                const float *w = sm.pwc[j + 1];
#pragma unroll 8
                for (int i = 0; i < D; ++i) inter = fmaf(sm.q[j][i] * w[i], sm.kv[i][n], inter);
                o = intra + inter;
            } else {
#pragma unroll 8
                for (int i = 0; i < D; ++i) inter = fmaf(sm.q[j][i], sm.kv[i][n], inter);
                o = fmaf(sm.pw[j + 1], inter, intra);
            }
            // with reverse_out the sequence is written back to front
            const long row = reverse_out ? (long)(t1 - 1 - c0 - j) : (long)(t0 + c0 + j);
            out[row * row_stride + (long)h * D + n] = from_f<T>(o);
        }
        __syncthreads();  // everyone has read KV_{i-1}

        // ---- state: KV_i = lambda^{Lc} KV_{i-1} + (gk (.) K_i)^T V_i ----
        const float dec = sm.pw[Lc];
        for (int e = tid; e < D * D; e += kThreads) {
            const int i = e / D, n = e % D;
            float acc = 0.f;
            if constexpr (CW) {
                for (int l = 0; l < Lc; ++l)
                    acc = fmaf(sm.pwc[Lc - 1 - l][i] * sm.k[l][i], sm.v[l][n], acc);
                sm.kv[i][n] = fmaf(sm.pwc[Lc][i], sm.kv[i][n], acc);
            } else {
                for (int l = 0; l < Lc; ++l) acc = fmaf(sm.gk[l] * sm.k[l][i], sm.v[l][n], acc);
                sm.kv[i][n] = fmaf(dec, sm.kv[i][n], acc);
            }
        }
        __syncthreads();
    }

    if (final_state) {
        float *dst = final_state + ((long)s * H + h) * D * D;
        for (int e = tid; e < D * D; e += kThreads) dst[e] = (&sm.kv[0][0])[e];
    }
}

template <typename T, int D, int B, bool CW>
cudaError_t launch(const PrefillArgs &a) {
    auto kern = prefill_simt_kernel<T, D, B, CW>;
    const size_t smem = sizeof(SimtSmem<D, B, CW>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const long grid = (long)(a.rank_limit > 0 ? a.rank_limit : a.nseq) * a.num_heads;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, kThreads, smem, a.stream>>>(
        static_cast<const T *>(a.q), static_cast<const T *>(a.k),
        static_cast<const T *>(a.v), a.decay, a.cu_seqlens, a.nseq, a.total_tokens,
        a.num_heads, a.initial_state, static_cast<T *>(a.out), a.final_state,
        a.reverse_out ? 1 : 0, a.min_len);
    return cudaGetLastError();
}

template <typename T, bool CW>
cudaError_t dispatch(const PrefillArgs &a) {
    const int B = a.chunk == 0 ? 64 : a.chunk;
    if (a.head_dim == 64) {
        if (B == 16) return launch<T, 64, 16, CW>(a);
        if (B == 32) return launch<T, 64, 32, CW>(a);
        if (B == 64) return launch<T, 64, 64, CW>(a);
    } else if (a.head_dim == 128) {
        if (B == 16) return launch<T, 128, 16, CW>(a);
        if (B == 32) return launch<T, 128, 32, CW>(a);
        if (B == 64) return launch<T, 128, 64, CW>(a);
    }
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t prefill_simt_f32(const PrefillArgs &a) {
    return a.channel_decay ? dispatch<float, true>(a) : dispatch<float, false>(a);
}
cudaError_t prefill_simt_bf16(const PrefillArgs &a) {
    return a.channel_decay ? dispatch<__nv_bfloat16, true>(a) : dispatch<__nv_bfloat16, false>(a);
}

}  // namespace la
