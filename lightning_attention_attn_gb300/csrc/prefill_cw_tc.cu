// Tensor-core (tcgen05 + TMEM + TMA) chunkwise prefill with a channel-wise
// decay: bf16 inputs, head_dim 128, blocks of 64 tokens, on sm_103a.
//
// The recursion (K3 report reading notes, gated DeltaNet: the scalar decay
// generalised to one decay per key channel) is
//     kv_t[i][:] = lambda_i kv_{t-1}[i][:] + k_t[i] v_t,    o_t = q_t kv_t,
// and in blocks of B tokens (MiniMax-01 report, §2.2.1 block split):
//     O_c  = intra_c + Q~_c KV_{c-1},            Q~_j[i] = q_j[i] lambda_i^(j+1)
//     KV_c = Lambda^{Lc} KV_{c-1} + K~_c^T V_c,  K~_l[i] = k_l[i] lambda_i^(Lc-1-l)
//     intra_jl = sum_i q_j[i] k_l[i] lambda_i^(j-l)      (l <= j)
// with Lc the true length of the block.  The decay sits inside the channel
// sum of the intra-block scores, so they are no plain product.  Each block is
// split into four 16-token sub-blocks; for a query j in sub-block bj and a key
// l in an earlier sub-block bl, with m = bj - bl - 1 in {0, 1, 2},
//     lambda^(j-l) = lambda^(j mod 16) * lambda^(16 m + 16 - l mod 16),
// both exponents >= 0, so the score is Q^_j . K^_{m,l} with
//     Q^_j[i] = q_j[i] lambda_i^(j mod 16),  K^_{m,l}[i] = k_l[i] lambda_i^(16m+16-l mod 16).
// Distance m only needs the keys of sub-blocks 0 .. 2 - m, so the three slabs
// concatenate into one 96-row B operand and a single MMA group (N = 96) gives
// every off-diagonal score.  The four diagonal 16 x 16 sub-blocks have no
// factoring with non-negative exponents; they are summed exactly in fp32 on
// CUDA cores.  Every exponent anywhere is >= 0, so no factor can overflow for
// any lambda in (0, 1].
//
// One CTA per (sequence, head, 64-wide value slice), 512 threads, the steps
// of a block separated by CTA barriers:
//   A  wait for the block's Q, K (one slot) and V (two slots) tiles (TMA);
//   B  all threads: Q^, Q~ (hi/lo bf16), K^ slabs, K~ (hi/lo) into shared
//      memory; the diagonal sub-block scores, 4 x 4 tiles over 16 channels
//      per thread, summed across eight threads;
//   C  thread 0: S = Q^ K^^T (N = 96), O2 = Q~_hi KV + Q~_lo KV with the state
//      copy as a hi/lo pair along N, dKV += K~_hi^T V + K~_lo^T V onto the
//      decayed state in TMEM; the next block's loads;
//   D  the warps of TMEM lane quadrants 0 and 1 (rows 0..63) assemble P from
//      S and the diagonal sums, as a hi/lo bf16 pair in TMEM; then
//      O1 = P_hi V + P_lo V;
//   E  all warps: fold (state row i in TMEM lane i: KV_c read out, its hi/lo
//      copy for the next block's O2, lambda_i^{L_{c+1}} KV_c written back);
//      rows 0..63: o = O1 + O2 -> bf16.
// Precision: P, Q~, K~ and the state copy enter the tensor core as hi + lo
// bf16 pairs (about 16 significant bits); Q^ and K^ as single bf16 (the
// scores they give carry about 2^-8 relative error per term, within the
// bf16 path's bound).  Every wait is bounded; on a timeout the CTA finishes
// its block, leaves the loop at the next barrier, drains its copies and MMAs,
// frees TMEM and raises the device error word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "la_internal.h"
#include "sched.cuh"
#include "sm100_ptx.cuh"

namespace la {

__device__ unsigned int g_cw_error = 0;  // bit 0: a bounded wait gave up

namespace {

using namespace ptx;

constexpr int D = 128;       // head dim
constexpr int DV = 64;       // value columns per CTA
constexpr int NVS = D / DV;  // value slices per head
constexpr int BC = 64;       // block size
constexpr int kThreads = 512;
constexpr int kMaxExp = 64;  // largest exponent of lambda used
// Diagonal sub-blocks factor around their middle (exponents -8 .. 8) with
// mu = max(lambda, 2^-12): every factor stays below 2^96 in magnitude.
constexpr float kMuMin = 1.0f / 4096.0f;
constexpr uint64_t kTimeoutNs = 2000000000ull;
// Issuing warps, both idle during the diagonal sums: warp 12 (lane quadrant
// 0) issues S, P V and the TMA loads; warp 14 issues Q~ KV and the state update.
constexpr int kWarpS = 12, kWarpKV = 14;

// Shared memory (offsets from a 1024-byte aligned base).  Every operand uses
// 128-byte swizzled rows of 64 16-bit values in 8-row, 1024-byte atoms; a
// 64-row, 64-column piece is 8 KB.
constexpr uint32_t kPiece = BC * 128;                // 8 KB
constexpr uint32_t kOffQ = 0;                        // raw Q: 2 pieces (channels 0-63, 64-127)
constexpr uint32_t kOffK = kOffQ + 2 * kPiece;       // raw K: 2 pieces
constexpr uint32_t kOffV = kOffK + 2 * kPiece;       // V: 2 slots x 1 piece
constexpr uint32_t kOffQh = kOffV + 2 * kPiece;      // Q^ (A, K-major, two 8 KB halves)
constexpr uint32_t kOffQt = kOffQh + 2 * kPiece;     // Q~ hi, then Q~ lo (16 KB each)
constexpr uint32_t kOffKh = kOffQt + 4 * kPiece;     // K^ slabs (B, K-major, 96 rows, 12 KB halves)
constexpr uint32_t kKhHalf = 96 * 128;
constexpr uint32_t kOffKt = kOffKh + 2 * kKhHalf;    // K~ hi, then K~ lo (MN-major A, 16 KB each)
constexpr uint32_t kOffKVb = kOffKt + 4 * kPiece;    // state copy: hi atom, lo atom (16 KB each)
constexpr uint32_t kKVAtom = D * 128;
constexpr uint32_t kOffPw = kOffKVb + 2 * kKVAtom;   // pw[e][i] = lambda_i^e, fp32
constexpr uint32_t kPwRow = D;
constexpr uint32_t kPwBytes = (kMaxExp + 1) * kPwRow * 4;
// pd[e + 8][i] = mu_i^e, e = -8 .. 8, mu_i = max(lambda_i, 2^-12): the factors
// of the diagonal sub-blocks (rows padded so that rows start on different banks)
constexpr uint32_t kOffPd = kOffPw + kPwBytes;
constexpr uint32_t kPdRow = D + 4;
constexpr uint32_t kOffCtrl = kOffPd + 17 * kPdRow * 4;
// The Q^ and Q~ MMAs read 128 rows of which only 0..63 are the block's; rows
// 64..127 of each half fall on the next 8 KB, which is always inside the
// buffers above (results of those rows are never used).

struct Ctrl {
    uint64_t full_qk, full_v[2], s_done, mma_done, pv_done, drained;
    uint32_t tmem_base;
    int abort;
    int seq_slot;
};
constexpr uint32_t kSmemBytes = kOffCtrl + sizeof(Ctrl) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// TMEM columns (512 allocated)
constexpr uint32_t kColS = 0;     // 96: off-diagonal scores, slabs m = 0, 1, 2 at 0, 48, 80
constexpr uint32_t kColPh = 96;   // 32: P hi (bf16 pairs, 64 keys)
constexpr uint32_t kColPl = 128;  // 32: P lo
constexpr uint32_t kColO1 = 160;  // 64: P V
constexpr uint32_t kColO2 = 224;  // 128: Q~ [KV_hi | KV_lo]
constexpr uint32_t kColKV = 352;  // 64: state
constexpr uint32_t kColSd = 416;  // 64: scores of the diagonal sub-blocks
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t slab_col(int m) { return m == 0 ? 0u : m == 1 ? 48u : 80u; }

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 96, 0, 0);   // Q^ (K-major) x K^ (K-major)
constexpr uint32_t kIdescSd = idesc_bf16_f32(128, 64, 0, 0);  // Q'' (K-major) x K'' (K-major)
constexpr uint32_t kIdescO2 = idesc_bf16_f32(128, 128, 0, 1); // Q~ (K-major) x KV (N-major)
constexpr uint32_t kIdescKV = idesc_bf16_f32(128, 64, 1, 1);  // K~^T (M-major) x V (N-major)
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 64, 0, 1);  // P (TMEM) x V (N-major)

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
    const uint4 u = ld_shared_v4(addr);
    return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                       __uint_as_float(u.w));
}
// 32 lanes x 8 consecutive 32-bit columns from registers.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&u)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
            taddr),
        "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7])
        : "memory");
}
// bf16 pair of (a, b), a in the low half, round to nearest even
__device__ __forceinline__ uint32_t pack_bf16_rn(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
// hi = the top 16 bits of a and b (bf16, exact); lo = the rest, also cut to
// bf16: hi + lo = x to about 2^-16 relative
__device__ __forceinline__ void split_pair(float a, float b, uint32_t &hi, uint32_t &lo) {
    const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
    hi = __byte_perm(ua, ub, 0x7632);
    const float2 l2 = f2_sub(make_float2(a, b), make_float2(__uint_as_float(ua & 0xffff0000u),
                                                            __uint_as_float(ub & 0xffff0000u)));
    lo = __byte_perm(__float_as_uint(l2.x), __float_as_uint(l2.y), 0x7632);
}
// the 8 bf16 of a 16-byte piece as fp32
__device__ __forceinline__ void unpack8(const uint4 &u, float (&x)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        x[2 * m] = __uint_as_float(w[m] << 16);
        x[2 * m + 1] = __uint_as_float(w[m] & 0xffff0000u);
    }
}
// byte offset of 16-byte piece cc (channels 8 cc .. 8 cc + 7) of row r in a
// swizzled operand whose two 64-channel halves are `half` bytes apart
__device__ __forceinline__ uint32_t swz(int r, int cc, uint32_t half) {
    return (uint32_t)(cc >> 3) * half + (uint32_t)r * 128u +
           (uint32_t)((((cc & 7) ^ (r & 7))) << 4);
}
__device__ __forceinline__ bool cw_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    return mbar_wait(bar, parity, abort, kTimeoutNs);
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_cw_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const float *__restrict__ decay,
                     const int32_t *__restrict__ cu, int nseq, int T, int H,
                     const float *initial_state, __nv_bfloat16 *__restrict__ out,
                     float *final_state) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctrl &cs = *reinterpret_cast<Ctrl *>(base + kOffCtrl);
    const uint32_t sb = smem_u32(base);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int vs = blockIdx.x % NVS;
    const int h = (blockIdx.x / NVS) % H;
    const int s = sequence_of_rank(cu, nseq, blockIdx.x / (NVS * H), &cs.seq_slot);
    int t0 = __ldg(cu + s), t1 = __ldg(cu + s + 1);
    t0 = min(max(t0, 0), T);
    t1 = min(max(t1, t0), T);
    const int L = t1 - t0;
    const int nch = (L + BC - 1) / BC;
    auto len_of = [&](int c) { return min(BC, L - c * BC); };
    const bool has_init = initial_state != nullptr;
    auto bar = [&](const uint64_t &b) { return smem_u32(&b); };
    const uint32_t pw_s = sb + kOffPw;  // lambda_i^e at pw_s + 4 (e kPwRow + i)
    const float *pw = reinterpret_cast<const float *>(base + kOffPw);
    const uint32_t pd_s = sb + kOffPd;  // mu_i^e at pd_s + 4 ((e + 8) kPdRow + i)
    volatile int *abort_flag = &cs.abort;

    // ---- set-up ----
    if (tid == 0) {
        mbar_init(bar(cs.full_qk), 1);
        mbar_init(bar(cs.full_v[0]), 1);
        mbar_init(bar(cs.full_v[1]), 1);
        mbar_init(bar(cs.s_done), 1);
        mbar_init(bar(cs.mma_done), 1);
        mbar_init(bar(cs.pv_done), 1);
        mbar_init(bar(cs.drained), 2);  // one commit per issuing warp
        cs.abort = 0;
        fence_mbar_init();
    }
    {
        float *pwm = reinterpret_cast<float *>(base + kOffPw);
        for (int idx = tid; idx < (kMaxExp + 1) * D; idx += kThreads) {
            const int e = idx / D, i = idx % D;
            pwm[e * kPwRow + i] = powf(__ldg(decay + h * D + i), (float)e);
        }
        float *pdm = reinterpret_cast<float *>(base + kOffPd);
        for (int idx = tid; idx < 17 * D; idx += kThreads) {
            const int e = idx / D - 8, i = idx % D;
            const float mu = fmaxf(__ldg(decay + h * D + i), kMuMin);
            pdm[(e + 8) * kPdRow + i] = powf(mu, (float)e);
        }
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&cs.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, cs.tmem_base, 0);
    const bool tmem_ok = tmem == 0;  // an allocation of all 512 columns starts at 0

    // TMA loads: issued by one elected lane of warp kWarpS; every lane of
    // that warp keeps the counts
    int n_qk = 0, n_v = 0;
    auto load_qk = [&](int c) {
        mbar_arrive_expect_tx(bar(cs.full_qk), 4 * kPiece);
        const int row = t0 + c * BC;
        tma_load_2d(sb + kOffQ, &tmQ, bar(cs.full_qk), h * D, row);
        tma_load_2d(sb + kOffQ + kPiece, &tmQ, bar(cs.full_qk), h * D + 64, row);
        tma_load_2d(sb + kOffK, &tmK, bar(cs.full_qk), h * D, row);
        tma_load_2d(sb + kOffK + kPiece, &tmK, bar(cs.full_qk), h * D + 64, row);
    };
    auto load_v = [&](int c) {
        const int st = c & 1;
        mbar_arrive_expect_tx(bar(cs.full_v[st]), kPiece);
        tma_load_2d(sb + kOffV + st * kPiece, &tmV, bar(cs.full_v[st]), h * D + vs * DV,
                    t0 + c * BC);
    };
    if (warp == kWarpS && tmem_ok && nch > 0) {
        if (elect_one()) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            load_qk(0);
            load_v(0);
            if (nch > 1) load_v(1);
        }
        __syncwarp();
        n_qk = 1;
        n_v = nch > 1 ? 2 : 1;
    }

    // ---- the state before the first block: KV_{-1} = S0 or 0 ----
    // Thread (warp, lane) owns state row i = 32 (warp % 4) + lane (TMEM lane
    // i) and value columns 16 (warp / 4) .. + 15 of the CTA's slice.
    const int qd = warp & 3, wq = warp >> 2;
    const int srow = qd * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const uint32_t tkv = tmem + lane_off + kColKV + 16 * wq;
    auto state_ptr = [&](float *p) {
        return reinterpret_cast<float4 *>(p + (((long)s * H + h) * D + srow) * D + vs * DV + 16 * wq);
    };
    // hi/lo copy of this thread's 16 state values into the O2 operand
    auto store_kv_copy = [&](const float(&kv)[16]) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) split_pair(kv[8 * u + 2 * m], kv[8 * u + 2 * m + 1], hi[m], lo[m]);
            const uint32_t a = sb + kOffKVb + (uint32_t)srow * 128u +
                               (uint32_t)((((2 * wq + u) ^ (srow & 7))) << 4);
            st_shared_v4(a, hi[0], hi[1], hi[2], hi[3]);
            st_shared_v4(a + kKVAtom, lo[0], lo[1], lo[2], lo[3]);
        }
    };
    // lambda_i^e kv into the state accumulator
    auto write_back = [&](const float(&kv)[16], int e) {
        const float g = pw[e * kPwRow + srow];
        uint32_t w[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) w[m] = __float_as_uint(kv[m] * g);
        tmem_st16(tkv, w);
    };
    if (tmem_ok) {
        float x[16];
        if (has_init) {
            const float4 *src = state_ptr(const_cast<float *>(initial_state));
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float4 f = src[m];
                x[4 * m] = f.x;
                x[4 * m + 1] = f.y;
                x[4 * m + 2] = f.z;
                x[4 * m + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int m = 0; m < 16; ++m) x[m] = 0.f;
        }
        if (nch == 0) {
            if (final_state) {
                float4 *dst = state_ptr(final_state);
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    dst[m] = make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
            }
        } else {
            store_kv_copy(x);
            if (has_init) write_back(x, len_of(0));
            fence_proxy_async_smem();
            tmem_wait_st();
        }
    }
    tc_fence_before();
    __syncthreads();

    for (int c = 0; tmem_ok && c < nch; ++c) {
        const int Lc = len_of(c);
        const bool last = c + 1 == nch;
        const uint32_t ph = c & 1;
        // ---- A: this block's tiles ----
        cw_wait(bar(cs.full_qk), ph, abort_flag);
        cw_wait(bar(cs.full_v[c & 1]), (c >> 1) & 1, abort_flag);

        // ---- B: derived operands ----
        // Q items: (row j, 8-channel piece cc), two per thread
#pragma unroll 1
        for (int it = tid; it < BC * 16; it += kThreads) {
            const int j = it >> 4, cc = it & 15;
            const uint32_t off = swz(j, cc, kPiece);
            uint32_t qh[4] = {0u, 0u, 0u, 0u}, th[4] = {0u, 0u, 0u, 0u}, tl[4] = {0u, 0u, 0u, 0u};
            uint32_t qd2[4] = {0u, 0u, 0u, 0u};
            if (j < Lc) {
                float q[8];
                unpack8(ld_shared_v4(sb + kOffQ + off), q);
                {  // Q''_j = q_j mu^(j mod 16 - 8), over the raw row
                    const uint32_t r = pd_s + 4u * (uint32_t)((j & 15) * kPdRow + 8 * cc);
                    const float4 m0 = ld_shared_f4(r), m1 = ld_shared_f4(r + 16);
                    const float gm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        qd2[m] = pack_bf16_rn(q[2 * m] * gm[2 * m], q[2 * m + 1] * gm[2 * m + 1]);
                }
                const float4 a0 = ld_shared_f4(pw_s + 4u * (uint32_t)((j & 15) * kPwRow + 8 * cc));
                const float4 a1 = ld_shared_f4(pw_s + 4u * (uint32_t)((j & 15) * kPwRow + 8 * cc + 4));
                const float4 b0 = ld_shared_f4(pw_s + 4u * (uint32_t)((j + 1) * kPwRow + 8 * cc));
                const float4 b1 = ld_shared_f4(pw_s + 4u * (uint32_t)((j + 1) * kPwRow + 8 * cc + 4));
                const float ga[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float gb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    qh[m] = pack_bf16_rn(q[2 * m] * ga[2 * m], q[2 * m + 1] * ga[2 * m + 1]);
                    split_pair(q[2 * m] * gb[2 * m], q[2 * m + 1] * gb[2 * m + 1], th[m], tl[m]);
                }
            }
            st_shared_v4(sb + kOffQh + off, qh[0], qh[1], qh[2], qh[3]);
            st_shared_v4(sb + kOffQ + off, qd2[0], qd2[1], qd2[2], qd2[3]);
            st_shared_v4(sb + kOffQt + off, th[0], th[1], th[2], th[3]);
            st_shared_v4(sb + kOffQt + 2 * kPiece + off, tl[0], tl[1], tl[2], tl[3]);
        }
        // K items: K~ (hi/lo) and the K^ slab rows of key l
#pragma unroll 1
        for (int it = tid; it < BC * 16; it += kThreads) {
            const int l = it >> 4, cc = it & 15;
            const uint32_t off = swz(l, cc, kPiece);
            const bool live = l < Lc;
            float k[8];
            unpack8(ld_shared_v4(sb + kOffK + off), k);
            {  // K''_l = k_l mu^(8 - l mod 16), over the raw row
                uint32_t kd2[4] = {0u, 0u, 0u, 0u};
                if (live) {
                    const uint32_t r = pd_s + 4u * (uint32_t)((16 - (l & 15)) * kPdRow + 8 * cc);
                    const float4 m0 = ld_shared_f4(r), m1 = ld_shared_f4(r + 16);
                    const float gm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        kd2[m] = pack_bf16_rn(k[2 * m] * gm[2 * m], k[2 * m + 1] * gm[2 * m + 1]);
                }
                st_shared_v4(sb + kOffK + off, kd2[0], kd2[1], kd2[2], kd2[3]);
            }
            {
                uint32_t th[4] = {0u, 0u, 0u, 0u}, tl[4] = {0u, 0u, 0u, 0u};
                if (live) {
                    const int e = Lc - 1 - l;
                    const float4 b0 = ld_shared_f4(pw_s + 4u * (uint32_t)(e * kPwRow + 8 * cc));
                    const float4 b1 = ld_shared_f4(pw_s + 4u * (uint32_t)(e * kPwRow + 8 * cc + 4));
                    const float gb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        split_pair(k[2 * m] * gb[2 * m], k[2 * m + 1] * gb[2 * m + 1], th[m], tl[m]);
                }
                st_shared_v4(sb + kOffKt + off, th[0], th[1], th[2], th[3]);
                st_shared_v4(sb + kOffKt + 2 * kPiece + off, tl[0], tl[1], tl[2], tl[3]);
            }
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                if ((l >> 4) > 2 - m) continue;  // slab m holds the keys of sub-blocks 0 .. 2 - m
                const int n = (int)slab_col(m) + l;
                uint32_t kh[4] = {0u, 0u, 0u, 0u};
                if (live) {
                    const int e = 16 * m + 16 - (l & 15);
                    const float4 a0 = ld_shared_f4(pw_s + 4u * (uint32_t)(e * kPwRow + 8 * cc));
                    const float4 a1 = ld_shared_f4(pw_s + 4u * (uint32_t)(e * kPwRow + 8 * cc + 4));
                    const float ga[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        kh[u] = pack_bf16_rn(k[2 * u] * ga[2 * u], k[2 * u + 1] * ga[2 * u + 1]);
                }
                st_shared_v4(sb + kOffKh + swz(n, cc, kKhHalf), kh[0], kh[1], kh[2], kh[3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- C: the block's MMAs ----
        // Each issuing warp is converged and issues from one elected lane, so
        // the operands are warp-uniform values and each tcgen05.mma is a
        // single issue.
        if (warp == kWarpS) {
            tc_fence_after();
            const bool go_w = __shfl_sync(0xffffffffu, (int)!*abort_flag, 0) != 0;
            const uint64_t dqh = sdesc_sw128(sb + kOffQh, 16, 1024);
            const uint64_t dkh = sdesc_sw128(sb + kOffKh, 16, 1024);
            // (the Q and K load of block c + 1 waits until S has read Q'' and K'')
            if (go_w && c + 1 < nch && c + 1 >= 2) ++n_v;
            const uint64_t dqd = sdesc_sw128(sb + kOffQ, 16, 1024);
            const uint64_t dkd = sdesc_sw128(sb + kOffK, 16, 1024);
            if (go_w && elect_one()) {
                mma_group_ss<2, kPiece / 16, 2, kKhHalf / 16>(tmem + kColS, dqh, dkh, kIdescS, 0u);
                mma_group_ss<2, kPiece / 16, 2, kPiece / 16>(tmem + kColSd, dqd, dkd, kIdescSd, 0u);
                mma_commit(bar(cs.s_done));
                // V slot (c + 1) & 1 was released by block c - 1's MMAs
                if (c + 1 < nch && c + 1 >= 2) load_v(c + 1);
            }
            __syncwarp();
        } else if (warp == kWarpKV) {
            tc_fence_after();
            const bool go_w = __shfl_sync(0xffffffffu, (int)!*abort_flag, 0) != 0;
            const uint64_t dkvb = sdesc_sw128(sb + kOffKVb, kKVAtom, 1024);
            const uint64_t dqth = sdesc_sw128(sb + kOffQt, 16, 1024);
            const uint64_t dqtl = sdesc_sw128(sb + kOffQt + 2 * kPiece, 16, 1024);
            const uint64_t dv = sdesc_sw128(sb + kOffV + (c & 1) * kPiece, kPiece, 1024);
            const uint64_t dkth = sdesc_sw128(sb + kOffKt, kPiece, 1024);
            const uint64_t dktl = sdesc_sw128(sb + kOffKt + 2 * kPiece, kPiece, 1024);
            const uint32_t acc0 = (c > 0 || has_init) ? 1u : 0u;
            if (go_w && elect_one()) {
                mma_group_ss<2, kPiece / 16, kMNMajorS1, kMNMajorS2>(tmem + kColO2, dqth, dkvb,
                                                                    kIdescO2, 0u);
                mma_group_ss<2, kPiece / 16, kMNMajorS1, kMNMajorS2>(tmem + kColO2, dqtl, dkvb,
                                                                    kIdescO2, 1u);
#pragma unroll
                for (uint32_t kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + kColKV, dkth + 128u * kk, dv + 128u * kk, kIdescKV,
                             kk > 0 ? 1u : acc0);
#pragma unroll
                for (uint32_t kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + kColKV, dktl + 128u * kk, dv + 128u * kk, kIdescKV, 1u);
                mma_commit(bar(cs.mma_done));
            }
            __syncwarp();
        }
        // ---- D: P from S and the diagonal sums; P V ----
        if (qd < 2) {
            cw_wait(bar(cs.s_done), ph, abort_flag);
            tc_fence_after();
            if (warp == kWarpS) {  // S has read Q'' and K'' (the raw tiles)
                if (__shfl_sync(0xffffffffu, (int)!*abort_flag, 0) && c + 1 < nch) {
                    if (elect_one()) load_qk(c + 1);
                    __syncwarp();
                    ++n_qk;
                }
            }
            const int j = qd * 32 + lane;  // query row = TMEM lane
            const int bj = j >> 4;
            const int b = wq;               // key sub-block of this warp
            const uint32_t srow_t = tmem + lane_off + kColS + 16 * b;
            float sv[16];
            {
                // the two halves of the warp sit in sub-blocks 2 qd and 2 qd + 1
                const int m_lo = 2 * qd - b - 1, m_hi = 2 * qd - b;
                float s_lo[16], s_hi[16], s_d[16];
                if (m_lo >= 0 && m_lo <= 2) tmem_ld16(srow_t + slab_col(m_lo), s_lo);
                if (m_hi >= 0 && m_hi <= 2) tmem_ld16(srow_t + slab_col(m_hi), s_hi);
                if (b == 2 * qd || b == 2 * qd + 1)  // this warp's block is a diagonal one
                    tmem_ld16(tmem + lane_off + kColSd + 16 * b, s_d);
                tmem_wait_ld();
                const bool lo_half = lane < 16;
                if (b < bj) {
#pragma unroll
                    for (int x = 0; x < 16; ++x) sv[x] = lo_half ? s_lo[x] : s_hi[x];
                } else if (b == bj) {
#pragma unroll
                    for (int x = 0; x < 16; ++x) sv[x] = s_d[x];
                } else {
#pragma unroll
                    for (int x = 0; x < 16; ++x) sv[x] = 0.f;
                }
            }
            const int lim = min(j, Lc - 1) - 16 * b;  // last key of this sub-block with l <= j, l < Lc
            uint32_t ph8[8], pl8[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const float a = (2 * x <= lim && j < Lc) ? sv[2 * x] : 0.f;
                const float bb = (2 * x + 1 <= lim && j < Lc) ? sv[2 * x + 1] : 0.f;
                split_pair(a, bb, ph8[x], pl8[x]);
            }
            tmem_st8(tmem + lane_off + kColPh + 8 * b, ph8);
            tmem_st8(tmem + lane_off + kColPl + 8 * b, pl8);
            tmem_wait_st();
            tc_fence_before();
            named_barrier_sync(1, 256);
            if (warp == kWarpS) {
                tc_fence_after();
                const bool go = !*abort_flag;
                const uint64_t dv = sdesc_sw128(sb + kOffV + (c & 1) * kPiece, kPiece, 1024);
                if (__shfl_sync(0xffffffffu, (int)go, 0) && elect_one()) {
#pragma unroll
                    for (uint32_t kk = 0; kk < 4; ++kk)
                        mma_bf16_tmem_a(tmem + kColO1, tmem + kColPh + 8 * kk, dv + 128u * kk,
                                        kIdescPV, kk > 0 ? 1u : 0u);
#pragma unroll
                    for (uint32_t kk = 0; kk < 4; ++kk)
                        mma_bf16_tmem_a(tmem + kColO1, tmem + kColPl + 8 * kk, dv + 128u * kk,
                                        kIdescPV, 1u);
                    mma_commit(bar(cs.pv_done));
                }
                __syncwarp();
            }
        }

        // ---- E: fold; output ----
        cw_wait(bar(cs.mma_done), ph, abort_flag);
        tc_fence_after();
        {
            float kv[16];
            tmem_ld16(tkv, kv);
            tmem_wait_ld();
            if (last) {
                if (final_state) {
                    float4 *dst = state_ptr(final_state);
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        dst[m] = make_float4(kv[4 * m], kv[4 * m + 1], kv[4 * m + 2], kv[4 * m + 3]);
                }
            } else {
                store_kv_copy(kv);
                write_back(kv, len_of(c + 1));
            }
        }
        if (qd < 2) {
            cw_wait(bar(cs.pv_done), ph, abort_flag);
            tc_fence_after();
            const int j = qd * 32 + lane;
            float o1[16], oh[16], ol[16];
            tmem_ld16(tmem + lane_off + kColO1 + 16 * wq, o1);
            tmem_ld16(tmem + lane_off + kColO2 + 16 * wq, oh);
            tmem_ld16(tmem + lane_off + kColO2 + 64 + 16 * wq, ol);
            tmem_wait_ld();
            if (j < Lc) {
                uint32_t w[8];
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    w[m] = pack_bf16_rn(o1[2 * m] + oh[2 * m] + ol[2 * m],
                                        o1[2 * m + 1] + oh[2 * m + 1] + ol[2 * m + 1]);
                uint4 *dst = reinterpret_cast<uint4 *>(
                    out + ((long)(t0 + c * BC + j) * H + h) * D + vs * DV + 16 * wq);
                dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        if (__syncthreads_or(*abort_flag != 0)) break;
    }

    // ---- teardown: no copy may still be landing, no MMA still running ----
    if (warp == kWarpKV && tmem_ok) {
        if (elect_one()) mma_commit(bar(cs.drained));
        __syncwarp();
    }
    if (warp == kWarpS && tmem_ok) {
        int no_abort = 0;
        if (elect_one()) mma_commit(bar(cs.drained));
        __syncwarp();
        mbar_wait(bar(cs.drained), 0, &no_abort, kTimeoutNs);
        // the latest load on each barrier (the only ones that can still be
        // in flight after an abort)
        if (n_qk > 0) mbar_wait(bar(cs.full_qk), (n_qk - 1) & 1, &no_abort, kTimeoutNs);
        for (int c = max(0, n_v - 2); c < n_v; ++c)
            mbar_wait(bar(cs.full_v[c & 1]), (c >> 1) & 1, &no_abort, kTimeoutNs);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0 && (cs.abort || !tmem_ok)) atomicOr(&g_cw_error, 1u);
}

// ------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [T, H*D] bf16 row-major, box = 64 columns x 64 rows, 128-byte swizzle.
bool make_map64(CUtensorMap *m, const void *ptr, int T, int H) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)H * D, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)H * D * 2};
    const cuuint32_t box[2] = {64, BC};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t take_cw_device_error(unsigned int *err) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_cw_error, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_cw_error, &zero, sizeof(zero));
        if (e != cudaSuccess) return e;
    }
    *err = v;
    return cudaSuccess;
}

cudaError_t prefill_cw_tc_bf16(const PrefillArgs &a) {
    if (!a.channel_decay || a.head_dim != D || !(a.chunk == 0 || a.chunk == BC) || a.reverse_out ||
        a.anti_causal || a.snapshots || a.min_len > 0 || a.rank_limit > 0)
        return cudaErrorNotSupported;
    CUtensorMap mq, mk, mv;
    if (!make_map64(&mq, a.q, a.total_tokens, a.num_heads) ||
        !make_map64(&mk, a.k, a.total_tokens, a.num_heads) ||
        !make_map64(&mv, a.v, a.total_tokens, a.num_heads))
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<unsigned long long> attr_set{0};
    if (dev >= 64 || !(attr_set.load(std::memory_order_acquire) & (1ull << dev))) {
        e = cudaFuncSetAttribute(prefill_cw_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set.fetch_or(1ull << dev, std::memory_order_release);
    }
    const long grid = (long)a.nseq * a.num_heads * NVS;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    prefill_cw_tc_kernel<<<(unsigned)grid, kThreads, kSmemBytes, a.stream>>>(
        mq, mk, mv, a.decay, a.cu_seqlens, a.nseq, a.total_tokens, a.num_heads, a.initial_state,
        static_cast<__nv_bfloat16 *>(a.out), a.final_state);
    return cudaGetLastError();
}

}  // namespace la
