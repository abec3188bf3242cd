// Lightning-attention decode step: one new token per sequence.
//
// MiniMax-01 report (CSDN translation) §3.3.2: the length-1 case is
// memory-bound and gets its own kernel; §3.3.1: the KV computation and the
// prefix-KV-cache update are one fused kernel.  Per (sequence b, head h):
//     S <- lambda_h S + k^T v        (S is the d x d fp32 state, in place)
//     o  = q S                        (read after the update)
// The state read-modify-write (2 * d^2 * 4 bytes) is the whole cost, so the
// kernel is a streaming pass: each warp owns d/4 rows of S, each lane a
// 16-byte (d = 128) or 8-byte (d = 64) column slice of a row, so every warp
// load/store instruction covers one whole contiguous row (512 / 256 bytes).
// All rows of a thread are loaded before any is used, keeping 8-16 vector
// loads in flight per thread; the four per-warp partial outputs are summed
// through shared memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "la_internal.h"

namespace la {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

template <int VEC> struct VecT;
template <> struct VecT<4> { using type = float4; };
template <> struct VecT<2> { using type = float2; };

__device__ __forceinline__ void vset(float4 &x, int c, float val) {
    (c == 0 ? x.x : c == 1 ? x.y : c == 2 ? x.z : x.w) = val;
}
__device__ __forceinline__ float vget(const float4 &x, int c) {
    return c == 0 ? x.x : c == 1 ? x.y : c == 2 ? x.z : x.w;
}
__device__ __forceinline__ void vset(float2 &x, int c, float val) { (c == 0 ? x.x : x.y) = val; }
__device__ __forceinline__ float vget(const float2 &x, int c) { return c == 0 ? x.x : x.y; }

// Rows are processed in groups of kRowsPerPass to bound registers while
// keeping that many independent 16-byte loads in flight per thread.
template <typename T, int D, bool CW>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
              const float *__restrict__ decay, float *__restrict__ state, int H,
              T *__restrict__ out, const int32_t *__restrict__ cu, int T_total) {
    constexpr int VEC = D / 32;             // columns per lane
    constexpr int RPW = D / kWarps;         // rows per warp
    constexpr int kRowsPerPass = 16;
    using V = typename VecT<VEC>::type;

    // launched as a dependent launch: wait for the previous kernel in the
    // stream (e.g. the step before, which wrote this state) to complete and
    // its writes to be visible, then let the next step be scheduled
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    __shared__ float qs[D], ks[D];
    __shared__ float red[kWarps][D];

    const long pair = blockIdx.x;           // b * H + h
    const int h = (int)(pair % H);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // one lambda per head, or per key channel (state row) with CW
    const float lam = CW ? 0.f : __ldg(decay + h);

    // token row of entry b: b itself, or in a packed batch (mixed prefill +
    // decode step, §3.3.2) the start of sequence b when it has exactly one
    // new token; other sequences belong to the prefill launch
    long row = pair / H;
    if (cu) {
        const int t0 = __ldg(cu + row), t1 = __ldg(cu + row + 1);
        if (t1 - t0 != 1 || t0 < 0 || t0 >= T_total) return;
        row = t0;
    }
    const long io = (row * H + h) * D;
    const T *qp = q + io, *kp = k + io, *vp = v + io;
    for (int i = threadIdx.x; i < D; i += kThreads) {
        qs[i] = to_f(qp[i]);
        ks[i] = to_f(kp[i]);
    }
    float vj[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) vj[c] = to_f(vp[lane * VEC + c]);
    __syncthreads();

    V *S = reinterpret_cast<V *>(state + pair * D * D);  // row i: D / VEC vectors
    float acc[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) acc[c] = 0.f;

#pragma unroll
    for (int r0 = 0; r0 < RPW; r0 += kRowsPerPass) {
        V sv[kRowsPerPass];
#pragma unroll
        for (int r = 0; r < kRowsPerPass; ++r) {
            const int i = warp * RPW + r0 + r;
            sv[r] = __ldcs(S + (long)i * 32 + lane);  // streaming: read once
        }
#pragma unroll
        for (int r = 0; r < kRowsPerPass; ++r) {
            const int i = warp * RPW + r0 + r;
            const float ki = ks[i], qi = qs[i];
            const float li = CW ? __ldg(decay + (long)h * D + i) : lam;
#pragma unroll
            for (int c = 0; c < VEC; ++c) {
                const float nv = fmaf(li, vget(sv[r], c), ki * vj[c]);
                vset(sv[r], c, nv);
                acc[c] = fmaf(qi, nv, acc[c]);
            }
            __stcs(S + (long)i * 32 + lane, sv[r]);
        }
    }

#pragma unroll
    for (int c = 0; c < VEC; ++c) red[warp][lane * VEC + c] = acc[c];
    __syncthreads();
    for (int j = threadIdx.x; j < D; j += kThreads) {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) o += red[w][j];
        out[io + j] = from_f<T>(o);
    }
}

template <typename T, int D>
cudaError_t launch(const DecodeArgs &a) {
    const long grid = (long)a.batch * a.num_heads;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    auto kern = a.channel_decay ? decode_kernel<T, D, true> : decode_kernel<T, D, false>;
    const cudaError_t e = launch_dependent(
        kern, (unsigned)grid, kThreads, 0, a.stream, static_cast<const T *>(a.q),
        static_cast<const T *>(a.k), static_cast<const T *>(a.v), a.decay, a.state, a.num_heads,
        static_cast<T *>(a.out), a.cu_seqlens, a.total_tokens);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(const DecodeArgs &a) {
    if (a.head_dim == 128) return launch<T, 128>(a);
    if (a.head_dim == 64) return launch<T, 64>(a);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t decode_f32(const DecodeArgs &a) { return dispatch<float>(a); }
cudaError_t decode_bf16(const DecodeArgs &a) { return dispatch<__nv_bfloat16>(a); }

}  // namespace la
