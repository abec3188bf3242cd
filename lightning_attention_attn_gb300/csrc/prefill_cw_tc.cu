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
// split into four 16-token sub-blocks.  For a query j in sub-block bj and a
// key l in an earlier sub-block bl, with m = bj - bl - 1 in {0, 1, 2},
//     lambda^(j-l) = lambda^(j mod 16) * lambda^(16 m + 16 - l mod 16),
// both exponents >= 0, so the score is Q^_j . K^_{m,l} with
//     Q^_j[i] = q_j[i] lambda_i^(j mod 16),  K^_{m,l}[i] = k_l[i] lambda_i^(16m+16-l mod 16).
// Distance m only needs the keys of sub-blocks 0 .. 2 - m, so the three slabs
// concatenate into one 96-row B operand and a single MMA group (N = 96) gives
// every off-diagonal score.  A diagonal 16 x 16 sub-block factors around its
// middle a = 16 bj + 8:
//     lambda^(j-l) = mu^(j-a) * mu^(a-l),   Q''_j = q_j mu^(j-a),  K''_l = k_l mu^(a-l),
// exponents -8 .. 8, with mu = max(lambda, 2^-12) so that no factor exceeds
// 2^96.  For lambda < 2^-12 this changes a score term by less than 2^-12
// times |q_j[i] k_l[i]| (only l = j is untouched: mu^0 = 1), below the bf16
// rounding of the inputs.
//
// Operands as hi/lo bf16 pairs on the M rows.  A block has 64 queries but an
// MMA has M = 128 rows, so every query-side A operand is stacked: rows 0..63
// hold the hi halves (top 16 bits of the fp32 value), rows 64..127 the lo
// halves (the rest, cut to bf16).  One MMA then gives both products, and the
// output sums row j and row 64 + j:
//   S   = [Q^ hi; Q^ lo] K^^T                  (N = 96)
//   Sd  = [Q'' hi; Q'' lo] [K'' hi; K'' lo]^T  (N = 128: hi and lo keys side by side)
//   O   = [Q~ hi; Q~ lo] [KV hi | KV lo]       (N = 128)
//   P   = the masked scores of each row, itself a hi/lo pair in TMEM
//   O  += P V                                  (A from TMEM, two K = 64 passes)
//   KV += K~ hi^T V + K~ lo^T V                (M = 128 channels)
// Every product carries about 16 significant bits but K^ (single bf16), so
// off-diagonal scores have about 2^-9 relative error per term.
//
// One CTA per (sequence, head, 64-wide value slice), 512 threads; the steps
// of a block:
//   A  wait for the block's Q and K tiles (TMA, into the hi rows of the Q''
//      and K'' operands);
//   B  all threads: thread t < 256 prepares query rows, the others key rows;
//      each owns channels 8 cc .. 8 cc + 7 of rows r, r + 16, r + 32, r + 48,
//      so its decay factors depend on (r, channel) alone and sit in registers;
//   C  warp 12 issues S and Sd, then Q~ KV and the state update, and once P
//      is written, P V; warp 14 issues the next block's loads;
//   D  twelve warps: warp (TMEM lane quadrant q, w) builds P for key sub-block
//      w of the 32 lanes of quadrant q (rows 64..127 from the lo products).
//      The P tiles of queries 0..31 against keys 32..63 are zero in every
//      block, so warps 8, 10, 12 and 14 write theirs once, before the first;
//   E  all warps: fold (state row i in TMEM lane i: KV_c read out, its hi/lo
//      copy for the next block's Q~ KV, lambda_i^{L_{c+1}} KV_c written
//      back); rows 64..127 of O through shared memory to rows 0..63, which
//      round o to bf16 into a tile that all threads store as whole rows.
// Every wait is bounded; on a timeout the CTA finishes its block, leaves the
// loop at the next barrier, drains its copies and MMAs, frees TMEM and raises
// the device error word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <type_traits>

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
constexpr float kMuMin = 1.0f / 4096.0f;
constexpr uint64_t kTimeoutNs = 2000000000ull;
// Warp 12 issues every MMA, warp 14 every TMA load.  Neither builds P: their
// P tiles (queries 0..31 against keys 32..63, quadrants 0 and 2) are always
// zero, so they are written once and the two warps are free to issue.
constexpr int kWarpMma = 12, kWarpLoad = 14;

// Shared memory (offsets from a 1024-byte aligned base).  Every operand uses
// 128-byte swizzled rows of 64 16-bit values in 8-row, 1024-byte atoms.  A
// stacked operand has 128 rows (hi rows 0..63, lo rows 64..127) in two
// 16 KB halves (channels 0-63, 64-127); a 64-row piece is 8 KB.
constexpr uint32_t kPiece = BC * 128;                // 8 KB
constexpr uint32_t kHalf = 2 * kPiece;               // 16 KB: half of a stacked operand
constexpr uint32_t kOffQd = 0;                       // [Q'' hi; Q'' lo]; raw Q lands in the hi rows
constexpr uint32_t kOffQh = kOffQd + 2 * kHalf;      // [Q^ hi; Q^ lo]; later the row transfer
constexpr uint32_t kOffQt = kOffQh + 2 * kHalf;      // [Q~ hi; Q~ lo]; later the output tile
constexpr uint32_t kOffKd = kOffQt + 2 * kHalf;      // [K'' hi; K'' lo]; raw K lands in the hi rows
constexpr uint32_t kOffKh = kOffKd + 2 * kHalf;      // K^ slabs (96 rows, 12 KB halves)
constexpr uint32_t kKhHalf = 96 * 128;
constexpr uint32_t kOffKt = kOffKh + 2 * kKhHalf;    // K~ hi, then K~ lo (MN-major A, 16 KB each)
constexpr uint32_t kOffV = kOffKt + 4 * kPiece;      // V (B, MN-major)
constexpr uint32_t kOffKVb = kOffV + kPiece;         // state copy: hi atom, lo atom (16 KB each)
constexpr uint32_t kKVAtom = D * 128;
constexpr uint32_t kOffCtrl = kOffKVb + 2 * kKVAtom;
// rows 64..127 of O on their way to rows 0..63: 64 rows x 64 fp32,
// rows padded so that eight consecutive rows start on different banks
constexpr uint32_t kXferRow = DV + 4;
static_assert(BC * kXferRow * 4 <= 2 * kHalf, "row transfer fits the Q^ operand");

struct Ctrl {
    uint64_t full_qk, full_v, s_done, mma_done, pv_done, drained;
    uint32_t tmem_base;
    int abort;
    int seq_slot;
};
constexpr uint32_t kSmemBytes = kOffCtrl + sizeof(Ctrl) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// TMEM columns (512 allocated)
constexpr uint32_t kColS = 0;     // 96: off-diagonal scores, slabs m = 0, 1, 2 at 0, 48, 80
constexpr uint32_t kColSd = 96;   // 128: diagonal scores against K'' hi (0..63) and lo (64..127)
constexpr uint32_t kColP = 224;   // 64: P hi at 0..31, lo at 32..63 (bf16 pairs, 64 keys)
constexpr uint32_t kColO = 288;   // 128: Q~ KV_hi + P V (0..63), Q~ KV_lo (64..127)
constexpr uint32_t kColKV = 416;  // 64: state
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t slab_col(int m) { return m == 0 ? 0u : m == 1 ? 48u : 80u; }

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 96, 0, 0);    // Q^ (K-major) x K^ (K-major)
constexpr uint32_t kIdescSd = idesc_bf16_f32(128, 128, 0, 0);  // Q'' (K-major) x K'' (K-major)
constexpr uint32_t kIdescO = idesc_bf16_f32(128, 128, 0, 1);  // Q~ (K-major) x [KV hi | KV lo] (N-major)
constexpr uint32_t kIdescKV = idesc_bf16_f32(128, 64, 1, 1);   // K~^T (M-major) x V (N-major)
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 64, 0, 1);   // P (TMEM) x V (N-major)

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

// arrive on a named barrier without waiting for it
__device__ __forceinline__ void named_barrier_arrive(uint32_t id, uint32_t count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// byte offset of 16-byte piece cc of hi row r in a stacked operand (the lo
// row is kPiece further on)
__device__ __forceinline__ uint32_t stk(int r, int cc) {
    return (uint32_t)(cc >> 3) * kHalf + (uint32_t)r * 128u + (uint32_t)((((cc & 7) ^ (r & 7))) << 4);
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
    grid_dependency_wait();    // the previous kernel's writes are visible from here on
    grid_launch_dependents();  // the next dependent launch may be scheduled

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
    volatile int *abort_flag = &cs.abort;

    // ---- set-up ----
    if (tid == 0) {
        mbar_init(bar(cs.full_qk), 1);
        mbar_init(bar(cs.full_v), 1);
        mbar_init(bar(cs.s_done), 1);
        mbar_init(bar(cs.mma_done), 1);
        mbar_init(bar(cs.pv_done), 1);
        mbar_init(bar(cs.drained), 1);
        cs.abort = 0;
        fence_mbar_init();
    }
    // Operand preparation: thread tid < 256 prepares query rows, the others
    // key rows; each owns channels 8 cc .. 8 cc + 7 of the four rows
    // r + 16 b (b = 0..3) of every block, so its decay factors depend on
    // (r, channel) only and are computed once, here.
    const bool q_role = tid < 256;
    const int cc = tid & 15, r16 = (tid & 255) >> 4;
    const float *lam_h = decay + h * D;
    // query rows: f[0] = lambda^r (Q^), f[1] = mu^(r - 8) (Q''),
    //             f[2 + b] = lambda^(16 b + r + 1) (Q~ of row 16 b + r)
    // key rows:   f[0] = mu^(8 - r) (K''), f[1 + m] = lambda^(16 m + 16 - r)
    //             (slab m), f[4] = lambda^15, f[5] = lambda^(15 - r)
    float f[6][8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const float lam = __ldg(lam_h + 8 * cc + u), mu = fmaxf(lam, kMuMin);
        if (q_role) {
            f[0][u] = powf(lam, (float)r16);
            f[1][u] = powf(mu, (float)(r16 - 8));
#pragma unroll
            for (int b = 0; b < 4; ++b) f[2 + b][u] = powf(lam, (float)(16 * b + r16 + 1));
        } else {
            f[0][u] = powf(mu, (float)(8 - r16));
#pragma unroll
            for (int m = 0; m < 3; ++m) f[1 + m][u] = powf(lam, (float)(16 * m + 16 - r16));
            f[4][u] = powf(lam, 15.f);
            f[5][u] = powf(lam, (float)(15 - r16));
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

    // TMA loads: issued by one elected lane of warp kWarpLoad; every lane of
    // that warp keeps the counts
    int n_qk = 0, n_v = 0;
    auto load_qk = [&](int c) {
        mbar_arrive_expect_tx(bar(cs.full_qk), 4 * kPiece);
        const int row = t0 + c * BC;
        tma_load_2d(sb + kOffQd, &tmQ, bar(cs.full_qk), h * D, row);
        tma_load_2d(sb + kOffQd + kHalf, &tmQ, bar(cs.full_qk), h * D + 64, row);
        tma_load_2d(sb + kOffKd, &tmK, bar(cs.full_qk), h * D, row);
        tma_load_2d(sb + kOffKd + kHalf, &tmK, bar(cs.full_qk), h * D + 64, row);
    };
    auto load_v = [&](int c) {
        mbar_arrive_expect_tx(bar(cs.full_v), kPiece);
        tma_load_2d(sb + kOffV, &tmV, bar(cs.full_v), h * D + vs * DV, t0 + c * BC);
    };
    if (warp == kWarpLoad && tmem_ok && nch > 0) {
        if (elect_one()) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            load_qk(0);
            load_v(0);
        }
        __syncwarp();
        n_qk = 1;
        n_v = 1;
    }

    const int qd = warp & 3, wq = warp >> 2;  // TMEM lane quadrant, column group

    // ---- the state before the first block: KV_{-1} = S0 or 0 ----
    // Thread (warp, lane) owns state row i = 32 (warp % 4) + lane (TMEM lane
    // i) and value columns 16 (warp / 4) .. + 15 of the CTA's slice.
    const int srow = qd * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const uint32_t tkv = tmem + lane_off + kColKV + 16 * wq;
    auto state_ptr = [&](float *p) {
        return reinterpret_cast<float4 *>(p + (((long)s * H + h) * D + srow) * D + vs * DV + 16 * wq);
    };
    // hi/lo copy of this thread's 16 state values into the Q~ KV operand
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
    // lambda_i^e kv into the state accumulator (i = srow); e is the length
    // of the next block: BC, or that of the sequence's last block
    const float lam_row = __ldg(lam_h + srow);
    const float lam_row64 = powf(lam_row, (float)BC);
    const float lam_row_last = nch > 0 ? powf(lam_row, (float)len_of(nch - 1)) : 1.f;
    auto write_back = [&](const float(&kv)[16], int e) {
        const float g = e == BC ? lam_row64 : lam_row_last;
        uint32_t w[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) w[m] = __float_as_uint(kv[m] * g);
        tmem_st16(tkv, w);
    };
    // the P tiles of warps 8, 10, 12, 14 (queries 0..31 in TMEM lanes 0-31
    // and 64-95, keys 32..63) are zero for every block
    const bool builds_p = !((qd & 1) == 0 && wq >= 2);
    if (tmem_ok && !builds_p) {
        const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        const uint32_t t = tmem + ((uint32_t)(qd * 32) << 16) + kColP + 8 * wq;
        tmem_st8(t, z);
        tmem_st8(t + 32, z);
        tmem_wait_st();
    }
    if (tmem_ok) {
        float x[16];
        if (has_init) {
            const float4 *src = state_ptr(const_cast<float *>(initial_state));
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float4 f4 = src[m];
                x[4 * m] = f4.x;
                x[4 * m + 1] = f4.y;
                x[4 * m + 2] = f4.z;
                x[4 * m + 3] = f4.w;
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
        // ---- A: this block's Q and K tiles ----
        cw_wait(bar(cs.full_qk), ph, abort_flag);

        // ---- B: derived operands ----
        // x * g for 8 channels into 4 bf16 pairs (rounded), or a hi/lo pair
        auto scaled = [&](const float(&x)[8], const float(&g)[8], int m) {
            return f2_mul(make_float2(x[2 * m], x[2 * m + 1]), make_float2(g[2 * m], g[2 * m + 1]));
        };
        auto put_rn = [&](uint32_t dst, const float(&x)[8], const float(&g)[8]) {
            uint32_t w[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float2 y = scaled(x, g, m);
                w[m] = pack_bf16_rn(y.x, y.y);
            }
            st_shared_v4(dst, w[0], w[1], w[2], w[3]);
        };
        auto put_split = [&](uint32_t dst_hi, uint32_t dst_lo, const float(&x)[8], const float(&g)[8]) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float2 y = scaled(x, g, m);
                split_pair(y.x, y.y, hi[m], lo[m]);
            }
            st_shared_v4(dst_hi, hi[0], hi[1], hi[2], hi[3]);
            st_shared_v4(dst_lo, lo[0], lo[1], lo[2], lo[3]);
        };
        if (q_role) {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int j = 16 * b + r16;
                const uint32_t off = stk(j, cc);
                float q[8];
                unpack8(ld_shared_v4(sb + kOffQd + off), q);
                if (j >= Lc) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) q[u] = 0.f;
                }
                put_split(sb + kOffQh + off, sb + kOffQh + kPiece + off, q, f[0]);
                put_split(sb + kOffQd + off, sb + kOffQd + kPiece + off, q, f[1]);
                put_split(sb + kOffQt + off, sb + kOffQt + kPiece + off, q, f[2 + b]);
            }
        } else {
            // K~ factor lambda^(Lc - 1 - l): from the slab factors for a full
            // block; the last, partial block of a sequence computes it
            auto key_rows = [&](auto full) {
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int l = 16 * b + r16;
                    const uint32_t off = stk(l, cc);
                    float k[8], g[8];
                    unpack8(ld_shared_v4(sb + kOffKd + off), k);
                    if (!full.value && l >= Lc) {
#pragma unroll
                        for (int u = 0; u < 8; ++u) k[u] = 0.f;
                    }
                    put_split(sb + kOffKd + off, sb + kOffKd + kPiece + off, k, f[0]);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (full.value)
                            g[u] = b < 3 ? f[3 - b][u] * f[4][u] : f[5][u];
                        else  // lambda^e as 2^(e log2 lambda), e = 0 exact
                            g[u] = l >= Lc - 1 ? 1.f
                                               : exp2f((float)(Lc - 1 - l) * log2f(__ldg(lam_h + 8 * cc + u)));
                    }
                    const uint32_t o8 = swz(l, cc, kPiece);
                    put_split(sb + kOffKt + o8, sb + kOffKt + 2 * kPiece + o8, k, g);
                    // slab m holds the keys of sub-blocks 0 .. 2 - m
#pragma unroll
                    for (int m = 0; m < 3; ++m)
                        if (b <= 2 - m)
                            put_rn(sb + kOffKh + swz((int)slab_col(m) + l, cc, kKhHalf), k, f[1 + m]);
                }
            };
            if (Lc == BC)
                key_rows(std::true_type{});
            else
                key_rows(std::false_type{});
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        const bool go_w = __shfl_sync(0xffffffffu, (int)!*abort_flag, 0) != 0;

        // ---- C and D: MMAs (warp 12), P (the builders) ----
        if (warp == kWarpMma) {
            // The warp is converged and issues from one elected lane, so the
            // operands are warp-uniform values and each tcgen05.mma is a
            // single issue.  MMAs of one thread run in issue order: S and Sd
            // first (P waits for them), then Q~ KV and the state update, then
            // P V on top of Q~ KV.
            tc_fence_after();
            const uint64_t dqh = sdesc_sw128(sb + kOffQh, 16, 1024);
            const uint64_t dkh = sdesc_sw128(sb + kOffKh, 16, 1024);
            const uint64_t dqd = sdesc_sw128(sb + kOffQd, 16, 1024);
            const uint64_t dkd = sdesc_sw128(sb + kOffKd, 16, 1024);
            const uint64_t dqt = sdesc_sw128(sb + kOffQt, 16, 1024);
            const uint64_t dkvb = sdesc_sw128(sb + kOffKVb, kKVAtom, 1024);
            const uint64_t dv = sdesc_sw128(sb + kOffV, kPiece, 1024);
            const uint64_t dkth = sdesc_sw128(sb + kOffKt, kPiece, 1024);
            const uint64_t dktl = sdesc_sw128(sb + kOffKt + 2 * kPiece, kPiece, 1024);
            const uint32_t acc0 = (c > 0 || has_init) ? 1u : 0u;
            if (go_w && elect_one()) {
                mma_group_ss<2, kHalf / 16, 2, kKhHalf / 16>(tmem + kColS, dqh, dkh, kIdescS, 0u);
                mma_group_ss<2, kHalf / 16, 2, kHalf / 16>(tmem + kColSd, dqd, dkd, kIdescSd, 0u);
                mma_commit(bar(cs.s_done));
                mma_group_ss<2, kHalf / 16, kMNMajorS1, kMNMajorS2>(tmem + kColO, dqt, dkvb, kIdescO, 0u);
            }
            __syncwarp();
            cw_wait(bar(cs.full_v), ph, abort_flag);  // one V load per block
            tc_fence_after();
            const bool go_v = __shfl_sync(0xffffffffu, (int)!*abort_flag, 0) != 0;
            if (go_w && elect_one()) {
                if (go_v) {
#pragma unroll
                    for (uint32_t kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + kColKV, dkth + 128u * kk, dv + 128u * kk, kIdescKV,
                                 kk > 0 ? 1u : acc0);
#pragma unroll
                    for (uint32_t kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + kColKV, dktl + 128u * kk, dv + 128u * kk, kIdescKV, 1u);
                }
                mma_commit(bar(cs.mma_done));
            }
            __syncwarp();
            named_barrier_sync(1, 13 * 32);  // the twelve P-building warps have written P
            tc_fence_after();
            const bool go_p = __shfl_sync(0xffffffffu, (int)!*abort_flag, 0) != 0;
            if (go_p && elect_one()) {
#pragma unroll
                for (uint32_t kk = 0; kk < 4; ++kk)
                    mma_bf16_tmem_a(tmem + kColO, tmem + kColP + 8 * kk, dv + 128u * kk, kIdescPV, 1u);
#pragma unroll
                for (uint32_t kk = 0; kk < 4; ++kk)
                    mma_bf16_tmem_a(tmem + kColO, tmem + kColP + 32 + 8 * kk, dv + 128u * kk, kIdescPV,
                                    1u);
                mma_commit(bar(cs.pv_done));
            }
            __syncwarp();
        } else if (warp == kWarpLoad) {
            cw_wait(bar(cs.s_done), ph, abort_flag);
            // Sd has read the hi rows that the next Q and K tiles land in
            if (__shfl_sync(0xffffffffu, (int)!*abort_flag, 0) && c + 1 < nch) {
                if (elect_one()) load_qk(c + 1);
                __syncwarp();
                ++n_qk;
            }
        } else if (builds_p) {
            cw_wait(bar(cs.s_done), ph, abort_flag);
            tc_fence_after();
            // TMEM lane = row: rows 0..63 hold the hi products of query
            // j = row, rows 64..127 the lo products of query j = row - 64.
            // Warp (quadrant qd, wq) covers key sub-block b = wq; its lanes
            // 0-15 sit in query sub-block bq0, lanes 16-31 in bq0 + 1.
            const int j = (qd & 1) * 32 + lane;
            const int b = wq;
            const int bq0 = 2 * (qd & 1), bq1 = bq0 + 1;
            const bool lo_has = b <= bq0, hi_has = b <= bq1;
            const bool lo_diag = b == bq0, hi_diag = b == bq1;
            const uint32_t trow = tmem + lane_off;
            const bool lo_half = lane < 16;
            const bool has = lo_half ? lo_has : hi_has, diag = lo_half ? lo_diag : hi_diag;
            float sv[16];
            {
                float x0[16], x1[16];
                if (lo_has)
                    tmem_ld16(trow + (lo_diag ? kColSd + 16 * b : kColS + slab_col(bq0 - b - 1) + 16 * b), x0);
                if (hi_has)
                    tmem_ld16(trow + (hi_diag ? kColSd + 16 * b : kColS + slab_col(bq1 - b - 1) + 16 * b), x1);
                tmem_wait_ld();
#pragma unroll
                for (int x = 0; x < 16; ++x) sv[x] = lo_half ? x0[x] : x1[x];
            }
            if (lo_diag || hi_diag) {  // the diagonal half adds its products with K'' lo
                float x2[16];
                tmem_ld16(trow + kColSd + 64 + 16 * b, x2);
                tmem_wait_ld();
                if (diag) {
#pragma unroll
                    for (int x = 0; x < 16; ++x) sv[x] += x2[x];
                }
            }
            const int lim = min(j, Lc - 1) - 16 * b;  // last key of this sub-block with l <= j, l < Lc
            uint32_t ph8[8], pl8[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const float a = (has && 2 * x <= lim && j < Lc) ? sv[2 * x] : 0.f;
                const float bb = (has && 2 * x + 1 <= lim && j < Lc) ? sv[2 * x + 1] : 0.f;
                split_pair(a, bb, ph8[x], pl8[x]);
            }
            tmem_st8(trow + kColP + 8 * b, ph8);
            tmem_st8(trow + kColP + 32 + 8 * b, pl8);
            tmem_wait_st();
            tc_fence_before();
            named_barrier_arrive(1, 13 * 32);
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
                fence_proxy_async_smem();  // the copy, for the next block's Q~ KV
                tmem_wait_st();
            }
        }
        cw_wait(bar(cs.pv_done), ph, abort_flag);
        tc_fence_after();
        if (warp == kWarpLoad) {  // P V and the state update have read V
            if (__shfl_sync(0xffffffffu, (int)!*abort_flag, 0) && c + 1 < nch) {
                if (elect_one()) load_v(c + 1);
                __syncwarp();
                ++n_v;
            }
        }
        {
            // o_j = O[j] + O[64 + j] (each the sum of its two column halves):
            // rows 64..127 reach rows 0..63 through
            // shared memory
            const int j = (qd & 1) * 32 + lane;
            const uint32_t xf = sb + kOffQh + 4u * (uint32_t)(j * kXferRow + 16 * wq);
            float o[16];
            {
                float o2[16];
                tmem_ld16(tmem + lane_off + kColO + 16 * wq, o);
                tmem_ld16(tmem + lane_off + kColO + 64 + 16 * wq, o2);
                tmem_wait_ld();
#pragma unroll
                for (int x = 0; x < 16; ++x) o[x] += o2[x];
            }
            if (qd >= 2) {
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    st_shared_v4(xf + 16u * m, __float_as_uint(o[4 * m]), __float_as_uint(o[4 * m + 1]),
                                 __float_as_uint(o[4 * m + 2]), __float_as_uint(o[4 * m + 3]));
                named_barrier_arrive(3, kThreads);
            } else {
                named_barrier_sync(3, kThreads);
                uint32_t w[8];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint4 p = ld_shared_v4(xf + 16u * m);
                    w[2 * m] = pack_bf16_rn(o[4 * m] + __uint_as_float(p.x), o[4 * m + 1] + __uint_as_float(p.y));
                    w[2 * m + 1] =
                        pack_bf16_rn(o[4 * m + 2] + __uint_as_float(p.z), o[4 * m + 3] + __uint_as_float(p.w));
                }
                // the bf16 row into the output tile (row j: 128 bytes, 16-byte
                // pieces swizzled by j mod 8)
                st_shared_v4(sb + kOffQt + (uint32_t)j * 128u + (uint32_t)(((2 * wq) ^ (j & 7)) << 4), w[0],
                             w[1], w[2], w[3]);
                st_shared_v4(sb + kOffQt + (uint32_t)j * 128u + (uint32_t)(((2 * wq + 1) ^ (j & 7)) << 4),
                             w[4], w[5], w[6], w[7]);
            }
        }
        // every thread stores one 16-byte piece of the tile; eight lanes
        // write one 128-byte output row
        named_barrier_sync(4, kThreads);
        {
            const int row = tid >> 3, piece = tid & 7;
            if (row < Lc) {
                const uint4 v = ld_shared_v4(sb + kOffQt + (uint32_t)row * 128u +
                                             (uint32_t)((piece ^ (row & 7)) << 4));
                *reinterpret_cast<uint4 *>(out + ((long)(t0 + c * BC + row) * H + h) * D + vs * DV +
                                           8 * piece) = v;
            }
        }
        tc_fence_before();
        if (__syncthreads_or(*abort_flag != 0)) break;
    }

    // ---- teardown: no copy may still be landing, no MMA still running ----
    if (warp == kWarpMma && tmem_ok) {
        if (elect_one()) mma_commit(bar(cs.drained));
        __syncwarp();
    }
    if (warp == kWarpLoad && tmem_ok) {
        int no_abort = 0;
        mbar_wait(bar(cs.drained), 0, &no_abort, kTimeoutNs);
        // the latest load on each barrier (the only ones that can still be
        // in flight after an abort)
        if (n_qk > 0) mbar_wait(bar(cs.full_qk), (n_qk - 1) & 1, &no_abort, kTimeoutNs);
        if (n_v > 0) mbar_wait(bar(cs.full_v), (n_v - 1) & 1, &no_abort, kTimeoutNs);
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
    e = launch_dependent(prefill_cw_tc_kernel, (unsigned)grid, kThreads, kSmemBytes, a.stream, mq,
                         mk, mv, a.decay, a.cu_seqlens, a.nseq, a.total_tokens, a.num_heads,
                         a.initial_state, static_cast<__nv_bfloat16 *>(a.out), a.final_state);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace la
