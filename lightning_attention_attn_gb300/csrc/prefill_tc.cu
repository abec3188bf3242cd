// Tensor-core (tcgen05 + TMEM + TMA) chunkwise lightning-attention prefill
// for bf16 inputs, head_dim 128, chunk 128, on sm_103a.
//
// The method (MiniMax-01 report, CSDN translation, §2.2.1): split each
// sequence into blocks of B tokens; inside a block use the masked left product
// [(Q_i K_i^T) (.) M] V_i, across blocks the right product with the carried
// d x d state:
//     O_i  = [(Q_i K_i^T) (.) M] V_i + Lambda_Q Q_i KV_{i-1}
//     KV_i = lambda^{B_i} KV_{i-1} + (Lambda_K K_i)^T V_i
// with M_jl = lambda^(j-l) [j >= l], Lambda_Q = diag(lambda^(j+1)),
// Lambda_K = diag(lambda^(B_i-1-l)) and B_i the true length of the block
// (the last block of a sequence may be short).  The decay values are made in
// the kernel (§3.3.1 fuses them into prefill); all exponents are >= 0.
//
// Work decomposition.  One CTA per (sequence, head, 64-wide value slice):
// o[:, j] and KV[:, j] only depend on v[:, j], so splitting d_v = 128 in two
// doubles the CTAs (128 for one 64-head sequence) while Q/K tiles are shared
// by the two sibling CTAs through L2.  Per 128-token chunk the CTA issues 32
// tcgen05 MMAs (M = 128, fp32 accumulators in TMEM):
//     S   = Q K^T                   128x128x128  bf16   (double buffered)
//     dKV = K^T [Vhat_hi | Vhat_lo] 128x128x128  bf16   (Vhat = Lambda_K V)
//     O2  = Q [KV_hi | KV_lo]       128x128x128  bf16   (KV = state after i-1)
//     O1  = P V                     128x 64x128  fp16   (P read from TMEM)
// A tcgen05.mma instruction costs about the same for N = 64 and N = 128, so
// the values the tensor core can only take at 8 significant bits (Vhat and
// the fp32 state copy) are passed as hi = bf16(x), lo = bf16(x - hi)
// concatenated along N: one N = 128 instruction instead of two N = 64 ones,
// and the two halves of the result are summed in fp32.  P and V go through
// the tensor core as fp16 (11 significant bits), each with an exact
// power-of-two scale chosen so the values sit at the top of the fp16 range
// (P per row, V per chunk): no overflow, no subnormal loss, and the scale is
// undone in fp32 in the epilogue.  The fp32 state itself lives in registers
// of the state warpgroup for the whole sequence.  Nothing but q, k, v (read
// once per CTA) and out / final state (written once) touches HBM.
//
// TMEM (512 columns): S buffer b = columns [128b, 128b + 128): S (fp32), then
// P (fp16 pairs) over its first 64 columns and O1 (fp32) in its last 64;
// O2 = [256, 384); dKV = [384, 512).
//
// Warp roles (320 threads):
//   warps 0-3  mask warpgroup: S -> P = fp16(2^-e_j S (.) M) into TMEM
//   warps 4-7  state warpgroup: Vhat / fp16 V, KV update, KV copy, output
//   warp  8    TMA producer: Q, K, V two-slot rings
//   warp  9    MMA issuer (one thread)
// Every wait is bounded and warp-uniform: a wait that gives up sets a CTA-wide
// abort flag, all roles leave their loops, in-flight TMA copies and MMAs are
// drained, TMEM is freed, and a device error word is raised for
// lightning_attn_device_status.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "la_internal.h"
#include "sched.cuh"
#include "sm100_ptx.cuh"

namespace la {

__device__ unsigned int g_tc_error = 0;  // bit 0: a bounded wait gave up

namespace {

using namespace ptx;

constexpr int D = 128;       // head dim (d_k = d_v)
constexpr int DV = 64;       // value columns per CTA
constexpr int NVS = D / DV;  // value slices per head
constexpr int BC = 128;      // chunk (block) size
constexpr int kThreads = 512;      // 16 warps: 4 per SM sub-partition, 128 registers
constexpr int kStateWarp0 = 4;
constexpr int kVWarp0 = 8;
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

// Shared memory (offsets from a 1024-byte aligned base).  Operand tiles are
// 128-byte swizzled rows of 64 16-bit values in 8-row, 1024-byte atoms.
constexpr uint32_t kHalf = BC * 128;            // 128 rows x 128 B = 16 KB
constexpr uint32_t kOffQ = 0;                   // 2 slots x (two 64-col halves)
constexpr uint32_t kOffK = kOffQ + 4 * kHalf;   // 2 slots x (two halves)
constexpr uint32_t kOffV = kOffK + 4 * kHalf;   // 2 slots x 64 cols; fp16 after
                                                // conversion
constexpr uint32_t kOffVhat = kOffV + 2 * kHalf;   // hi, lo: 128 tokens x 64
constexpr uint32_t kOffKVb = kOffVhat + 2 * kHalf; // hi, lo: 128 d_k x 64
constexpr uint32_t kOffCtrl = kOffKVb + 2 * kHalf;

struct Ctrl {
    uint64_t full_q[2], full_k[2], full_v[2], empty_q[2], empty_k[2], empty_v[2];
    uint64_t s_full[2], s_free[2], p_full[2], vmax_ready[2], vconv_full[2];
    uint64_t o_full, o2_free, dkv_full, dkv_free, vhat_full, kv_full, kv_free, mma_done;
    uint32_t tmem_base;
    int abort;
    int seq_slot;
    int pad;
    float pw[BC + 4];         // pw[e] = lambda^e, e = 0..BC
    float rowscale[2][BC];    // 2^e_j of P's rows, per S buffer
    float vmax[2][4];         // per-warp max |v| of a chunk, double buffered
    float vscale[4];          // 2^f of V's fp16 scale, ring indexed by chunk & 3
};
constexpr uint32_t kSmemBytes = kOffCtrl + sizeof(Ctrl) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO2 = 256, kColDKV = 384;

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0, 0);   // Q (K-major) x K (K-major)
constexpr uint32_t kIdescKV = idesc_bf16_f32(128, 128, 1, 1);  // K^T (M-major) x Vhat (N-major)
constexpr uint32_t kIdescO2 = idesc_bf16_f32(128, 128, 0, 1);  // Q (K-major) x KV (N-major)
constexpr uint32_t kIdescPV = idesc_fp16_f32(128, DV, 0, 1);   // P (TMEM) x V (N-major)

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(v);
}
// hi = bf16(x), lo = bf16(x - hi), packed in pairs
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat16 ha = __float2bfloat16_rn(a), hb = __float2bfloat16_rn(b);
    hi = (uint32_t)__bfloat16_as_ushort(ha) | ((uint32_t)__bfloat16_as_ushort(hb) << 16);
    lo = pack_bf16(a - __bfloat162float(ha), b - __bfloat162float(hb));
}
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
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Exact power-of-two scale exponent: for m > 0 finite, returns e with
// m * 2^-e in [2^top, 2^(top+1)), clamped to [-126, 126] so that both 2^e and
// 2^-e are normal floats; 0 for m == 0 or a non-finite m.
__device__ __forceinline__ int fp16_scale_exp(float m, int top) {
    if (!(m > 0.f) || m > 3.0e38f) return 0;
    const int eb = (int)((__float_as_uint(m) >> 23) & 0xff);
    const int e = (eb == 0 ? -126 : eb - 127) - top;
    return max(-126, min(126, e));
}
__device__ __forceinline__ float exp2i(int e) {  // 2^e for -126 <= e <= 127
    return __uint_as_float((uint32_t)(e + 127) << 23);
}
// A bounded wait whose outcome is the same for every lane of the warp (so
// the warp stays converged for the .sync.aligned tcgen05 instructions).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    const bool ok = mbar_wait(bar, parity, abort, kTimeoutNs);
    return __all_sync(0xffffffffu, ok);
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const float *__restrict__ decay, const int32_t *__restrict__ cu, int nseq, int T,
                  int H, __nv_bfloat16 *__restrict__ out, float *__restrict__ final_state) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctrl &cs = *reinterpret_cast<Ctrl *>(base + kOffCtrl);
    const uint32_t sb = smem_u32(base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- which (sequence, head, value slice) ----
    const int vs = blockIdx.x % NVS;
    const int h = (blockIdx.x / NVS) % H;
    const int s = sequence_of_rank(cu, nseq, blockIdx.x / (NVS * H), &cs.seq_slot);
    int t0 = __ldg(cu + s), t1 = __ldg(cu + s + 1);
    t0 = min(max(t0, 0), T);
    t1 = min(max(t1, t0), T);
    const int L = t1 - t0;
    const int nch = (L + BC - 1) / BC;
    const float lam = __ldg(decay + h);

    auto bar = [&](const uint64_t &b) { return smem_u32(&b); };
    const uint32_t pw_s = smem_u32(&cs.pw[0]);          // lambda^e at pw_s + 4 e
    const uint32_t rowscale_s = smem_u32(&cs.rowscale[0][0]);
    const uint32_t vmax_s = smem_u32(&cs.vmax[0][0]);
    auto pw = [&](int e) { return ld_shared_f32(pw_s + 4u * (uint32_t)e); };
    auto qslot = [&](int st) { return sb + kOffQ + st * 2 * kHalf; };
    auto kslot = [&](int st) { return sb + kOffK + st * 2 * kHalf; };
    auto vslot = [&](int st) { return sb + kOffV + st * kHalf; };

    // ---- set-up ----
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(cs.full_q[i]), 1);
            mbar_init(bar(cs.full_k[i]), 1);
            mbar_init(bar(cs.full_v[i]), 1);
            mbar_init(bar(cs.empty_q[i]), 1);
            mbar_init(bar(cs.empty_k[i]), 1);
            mbar_init(bar(cs.empty_v[i]), 1);
            mbar_init(bar(cs.s_full[i]), 1);
            mbar_init(bar(cs.s_free[i]), 128);
            mbar_init(bar(cs.p_full[i]), 128);
            mbar_init(bar(cs.vmax_ready[i]), 128);
            mbar_init(bar(cs.vconv_full[i]), 128);
        }
        mbar_init(bar(cs.o_full), 1);
        mbar_init(bar(cs.o2_free), 128);
        mbar_init(bar(cs.dkv_full), 1);
        mbar_init(bar(cs.dkv_free), 128);
        mbar_init(bar(cs.vhat_full), 128);
        mbar_init(bar(cs.kv_full), 128);
        mbar_init(bar(cs.kv_free), 1);
        mbar_init(bar(cs.mma_done), 1);
        cs.abort = 0;
        fence_mbar_init();
    }
    for (int e = threadIdx.x; e <= BC; e += kThreads) cs.pw[e] = powf(lam, (float)e);
    if (warp == 0) {
        tmem_alloc(smem_u32(&cs.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = cs.tmem_base;
    volatile int *abort_flag = &cs.abort;

    if (warp == kTmaWarp) {
        // ================= TMA producer =================
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmO);
            int nq = 0, nk = 0, nv = 0;
            bool ok = true;
            for (int i = 0; i < nch && ok; ++i) {
                const int st = i & 1;
                const uint32_t sph = (i >> 1) & 1;
                const int y = t0 + i * BC;
                if (!(ok = mbar_wait(bar(cs.empty_q[st]), sph ^ 1, abort_flag, kTimeoutNs))) break;
                mbar_arrive_expect_tx(bar(cs.full_q[st]), 2 * kHalf);
                tma_load_2d(qslot(st), &tmQ, bar(cs.full_q[st]), h * D, y);
                tma_load_2d(qslot(st) + kHalf, &tmQ, bar(cs.full_q[st]), h * D + 64, y);
                ++nq;
                if (!(ok = mbar_wait(bar(cs.empty_k[st]), sph ^ 1, abort_flag, kTimeoutNs))) break;
                mbar_arrive_expect_tx(bar(cs.full_k[st]), 2 * kHalf);
                tma_load_2d(kslot(st), &tmK, bar(cs.full_k[st]), h * D, y);
                tma_load_2d(kslot(st) + kHalf, &tmK, bar(cs.full_k[st]), h * D + 64, y);
                ++nk;
                if (!(ok = mbar_wait(bar(cs.empty_v[st]), sph ^ 1, abort_flag, kTimeoutNs))) break;
                mbar_arrive_expect_tx(bar(cs.full_v[st]), kHalf);
                tma_load_2d(vslot(st), &tmV, bar(cs.full_v[st]), h * D + vs * DV, y);
                ++nv;
            }
            // Never leave with a load still landing in shared memory.
            int no_abort = 0;
            for (int c = max(0, nq - 2); c < nq; ++c)
                mbar_wait(bar(cs.full_q[c & 1]), (c >> 1) & 1, &no_abort, kTimeoutNs);
            for (int c = max(0, nk - 2); c < nk; ++c)
                mbar_wait(bar(cs.full_k[c & 1]), (c >> 1) & 1, &no_abort, kTimeoutNs);
            for (int c = max(0, nv - 2); c < nv; ++c)
                mbar_wait(bar(cs.full_v[c & 1]), (c >> 1) & 1, &no_abort, kTimeoutNs);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ================= MMA issuer =================
        // Per chunk i: dKV_i, O2_i, then the next chunk's S_{i+1}, then P_i V_i.
        // S_{i+1} goes before P_i V_i so that the mask warpgroup turns
        // S_{i+1} into P_{i+1} while the tensor core runs P_i V_i, dKV_{i+1}
        // and O2_{i+1}.
        if (lane == 0) {
            const uint32_t vha = sb + kOffVhat, kvb = sb + kOffKVb;
            auto issue_s = [&](int i) -> bool {  // S_i = Q_i K_i^T
                const int st = i & 1;
                const uint32_t sph = (i >> 1) & 1;
                // buffer st is free once chunk i-2's P V and epilogue are done
                if (!mbar_wait(bar(cs.full_q[st]), sph, abort_flag, kTimeoutNs)) return false;
                if (!mbar_wait(bar(cs.full_k[st]), sph, abort_flag, kTimeoutNs)) return false;
                if (!mbar_wait(bar(cs.s_free[st]), sph ^ 1, abort_flag, kTimeoutNs)) return false;
                tc_fence_after();
                mma8_k_k(tmem + st * 128, sdesc_sw128(qslot(st), 16, 1024),
                         sdesc_sw128(kslot(st), 16, 1024), kIdescS);
                mma_commit(bar(cs.s_full[st]));
                return true;
            };
            bool ok = nch > 0 ? issue_s(0) : true;
            for (int i = 0; ok && i < nch; ++i) {
                const int st = i & 1;
                const uint32_t sph = (i >> 1) & 1, ph = i & 1;
                const uint32_t qa = qslot(st), ka = kslot(st), va = vslot(st);
                const uint32_t colS = st * 128;
                // dKV_i = K_i^T [Vhat_hi | Vhat_lo]
                if (!mbar_wait(bar(cs.vhat_full), ph, abort_flag, kTimeoutNs)) break;
                if (!mbar_wait(bar(cs.dkv_free), ph ^ 1, abort_flag, kTimeoutNs)) break;
                tc_fence_after();
                mma8_mn_mn(tmem + kColDKV, sdesc_sw128(ka, kHalf, 1024),
                           sdesc_sw128(vha, kHalf, 1024), kIdescKV);
                mma_commit(bar(cs.dkv_full));
                mma_commit(bar(cs.empty_k[st]));
                // O2_i = Q_i [KV_hi | KV_lo] (the state after chunk i-1)
                if (!mbar_wait(bar(cs.kv_full), ph, abort_flag, kTimeoutNs)) break;
                if (!mbar_wait(bar(cs.o2_free), ph ^ 1, abort_flag, kTimeoutNs)) break;
                tc_fence_after();
                mma8_k_mn(tmem + kColO2, sdesc_sw128(qa, 16, 1024),
                          sdesc_sw128(kvb, kHalf, 1024), kIdescO2);
                mma_commit(bar(cs.kv_free));
                mma_commit(bar(cs.empty_q[st]));
                // S_{i+1}
                if (i + 1 < nch && !(ok = issue_s(i + 1))) break;
                // O1_i = P_i V_i (fp16; P in the first half of the S buffer,
                // O1 into its second half)
                if (!mbar_wait(bar(cs.p_full[st]), sph, abort_flag, kTimeoutNs)) break;
                if (!mbar_wait(bar(cs.vconv_full[st]), sph, abort_flag, kTimeoutNs)) break;
                tc_fence_after();
                mma8_t_mn(tmem + colS + 64, tmem + colS, sdesc_sw128(va, kHalf, 1024), kIdescPV);
                mma_commit(bar(cs.o_full));
                mma_commit(bar(cs.empty_v[st]));
            }
            // All MMAs must be finished before TMEM is released.
            mma_commit(bar(cs.mma_done));
            int no_abort = 0;
            mbar_wait(bar(cs.mma_done), 0, &no_abort, kTimeoutNs);
        }
        __syncwarp();
    } else if (warp < kStateWarp0) {
        // ================= mask warpgroup: S -> P =================
        // Thread j owns row j of the chunk (TMEM lane j).  p_jl = S_jl
        // lambda^(j-l) for l <= j, l < Lc, else 0.  P goes to TMEM as fp16
        // scaled by 2^-e_j, a power of two chosen from an upper bound of the
        // row's |p| (pass 1: max |S| of each column block times the block's
        // largest decay factor) so the row's values sit below 2^12: no
        // overflow, and 11 significant bits for everything within 2^25 of
        // the bound.  Pass 2 masks, scales and packs one 32-column block at a
        // time into TMEM columns [16 cb, 16 cb + 16) of the S buffer: blocks
        // are visited in increasing cb, so block cb overwrites S columns of
        // block cb / 2 <= cb, already read.
        const int j = warp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        float colf[32];  // lambda^(31-c): off the diagonal block,
#pragma unroll           // lambda^(j-l) = lambda^(j-(32cb+31)) lambda^(31-c)
        for (int c = 0; c < 32; ++c) colf[c] = pw(31 - c);
        uint32_t zero[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) zero[m] = 0u;
        for (int i = 0; i < nch; ++i) {
            const int st = i & 1;
            const uint32_t sph = (i >> 1) & 1;
            const int Lc = min(BC, L - i * BC);
            const uint32_t scol = tmem + lane_off + st * 128;
            if (!warp_wait(bar(cs.s_full[st]), sph, abort_flag)) break;
            tc_fence_after();
            // pass 1: bound of max |p| over the row
            float bound = 0.f;
#pragma unroll 1
            for (int cb = 0; cb <= warp; ++cb) {
                float sv[32];
                tmem_ld32(scol + cb * 32, sv);
                tmem_wait_ld();
                const int lim = min(cb == warp ? lane : 31, Lc - 1 - cb * 32);  // last valid c
                float m = 0.f;
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (c <= lim) m = fmaxf(m, fabsf(sv[c]));
                bound = fmaxf(bound, cb == warp ? m : m * pw(j - cb * 32 - 31));
            }
            const int e = fp16_scale_exp(bound, 11);
            const float inv = exp2i(-e);
            // pass 2: the blocks below the diagonal in increasing order, then
            // the diagonal block (P block cb lands in S block cb / 2 <= cb,
            // which has been read by then)
#pragma unroll 1
            for (int cb = 0; cb < warp; ++cb) {
                float sv[32];
                tmem_ld32(scol + cb * 32, sv);
                tmem_wait_ld();
                const float rowf = pw(j - cb * 32 - 31) * inv;
                const int lim = Lc - 1 - cb * 32;
                uint32_t pk[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const int c = 2 * m;
                    const float a = (c <= lim) ? sv[c] * (rowf * colf[c]) : 0.f;
                    const float b = (c + 1 <= lim) ? sv[c + 1] * (rowf * colf[c + 1]) : 0.f;
                    pk[m] = pack_f16(a, b);
                }
                tmem_st16(scol + cb * 16, pk);
            }
            {
                float sv[32];
                tmem_ld32(scol + warp * 32, sv);
                tmem_wait_ld();
                const int lim = min(lane, Lc - 1 - warp * 32);
                uint32_t pk[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const int c = 2 * m;
                    const float a = (c <= lim) ? sv[c] * (pw(max(lane - c, 0)) * inv) : 0.f;
                    const float b = (c + 1 <= lim) ? sv[c + 1] * (pw(max(lane - c - 1, 0)) * inv) : 0.f;
                    pk[m] = pack_f16(a, b);
                }
                tmem_st16(scol + warp * 16, pk);
            }
#pragma unroll 1
            for (int cb = warp + 1; cb < 4; ++cb) tmem_st16(scol + cb * 16, zero);
            st_shared_f32(rowscale_s + 4u * (uint32_t)(st * BC + j), exp2i(e));
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(cs.p_full[st]));
        }
    } else if (warp < kVWarp0) {
        // ================= state warpgroup =================
        const int w4 = warp - kStateWarp0;
        const int r = w4 * 32 + lane;  // TMEM lane: d_k row / token row
        const uint32_t lane_off = (uint32_t)(w4 * 32) << 16;
        const uint32_t kvb = sb + kOffKVb;
        const uint32_t vscale_s = smem_u32(&cs.vscale[0]);
        float kv[DV];
#pragma unroll
        for (int c = 0; c < DV; ++c) kv[c] = 0.f;
        // KV_{-1} = 0
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            st_shared_v4(kvb + r * 128 + c * 16, 0u, 0u, 0u, 0u);
            st_shared_v4(kvb + kHalf + r * 128 + c * 16, 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(cs.kv_full));

        for (int i = 0; i < nch; ++i) {
            const int st = i & 1;
            const uint32_t sph = (i >> 1) & 1, ph = i & 1;
            const int Lc = min(BC, L - i * BC);
            // ---- KV_i = lambda^{Lc} KV_{i-1} + dKV_hi + dKV_lo ----
            if (!warp_wait(bar(cs.dkv_full), ph, abort_flag)) break;
            tc_fence_after();
            const float dec = pw(Lc);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float a[16], b[16];
                tmem_ld16(tmem + lane_off + kColDKV + q * 16, a);
                tmem_ld16(tmem + lane_off + kColDKV + 64 + q * 16, b);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    kv[q * 16 + c] = fmaf(dec, kv[q * 16 + c], a[c] + b[c]);
            }
            tc_fence_before();
            mbar_arrive(bar(cs.dkv_free));
            // ---- hi/lo copy of KV_i for the next chunk's Q KV (after O2_i read KV_{i-1}) ----
            if (!warp_wait(bar(cs.kv_free), ph, abort_flag)) break;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t phys = (uint32_t)(c ^ (r & 7));
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    // hi = x with the low 16 bits cleared (a bf16, exact);
                    // lo = x - hi (exact in fp32), also truncated to bf16:
                    // hi + lo = x to about 2^-14 relative
                    const uint32_t ua = __float_as_uint(kv[8 * c + 2 * q]);
                    const uint32_t ub = __float_as_uint(kv[8 * c + 2 * q + 1]);
                    hi[q] = __byte_perm(ua, ub, 0x7632);
                    const float la = __uint_as_float(ua) - __uint_as_float(ua & 0xffff0000u);
                    const float lb = __uint_as_float(ub) - __uint_as_float(ub & 0xffff0000u);
                    lo[q] = __byte_perm(__float_as_uint(la), __float_as_uint(lb), 0x7632);
                }
                st_shared_v4(kvb + r * 128 + phys * 16, hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(kvb + kHalf + r * 128 + phys * 16, lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(cs.kv_full));
            // ---- output: o_j = 2^(e_j + f) O1_j + lambda^(j+1) (O2hi_j + O2lo_j) ----
            if (!warp_wait(bar(cs.o_full), ph, abort_flag)) break;
            if (!warp_wait(bar(cs.p_full[st]), sph, abort_flag)) break;  // orders rowscale
            tc_fence_after();
            const float s1 = ld_shared_f32(rowscale_s + 4u * (uint32_t)(st * BC + r)) *
                             ld_shared_f32(vscale_s + 4u * (uint32_t)(i & 3));
            const float qf = pw(r + 1);
            uint4 *orow = reinterpret_cast<uint4 *>(out + ((long)(t0 + i * BC + r) * H + h) * D +
                                                    vs * DV);
#pragma unroll 1
            for (int g = 0; g < 8; ++g) {
                float a[8], b[8], c2[8];
                tmem_ld8(tmem + lane_off + st * 128 + 64 + g * 8, a);
                tmem_ld8(tmem + lane_off + kColO2 + g * 8, b);
                tmem_ld8(tmem + lane_off + kColO2 + 64 + g * 8, c2);
                tmem_wait_ld();
                if (g == 7) {  // all TMEM reads of this chunk are done
                    tc_fence_before();
                    mbar_arrive(bar(cs.o2_free));
                    mbar_arrive(bar(cs.s_free[st]));
                }
                uint32_t w[4];
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    w[m] = pack_bf16(fmaf(qf, b[2 * m] + c2[2 * m], s1 * a[2 * m]),
                                     fmaf(qf, b[2 * m + 1] + c2[2 * m + 1], s1 * a[2 * m + 1]));
                if (r < Lc) orow[g] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        if (final_state && !*abort_flag) {
            float4 *dst = reinterpret_cast<float4 *>(final_state + (((long)s * H + h) * D + r) * D +
                                                     vs * DV);
#pragma unroll
            for (int c = 0; c < DV / 4; ++c)
                dst[c] = make_float4(kv[4 * c], kv[4 * c + 1], kv[4 * c + 2], kv[4 * c + 3]);
        }
    } else if (warp < kVWarp0 + 4) {
        // ================= V-tile warpgroup =================
        // Chunk i's V tile, one row (token) per thread, in two steps:
        //  1. Vhat = Lambda_K V as a hi/lo bf16 pair for the dKV MMA (Vhat_i
        //     may be written once dKV_{i-1} has read Vhat_{i-1});
        //  2. V itself, converted in place to fp16 with the chunk's
        //     power-of-two scale (a max over the tile) for the P V MMA.
        // Rows past the chunk end are zero in both.
        const int w4 = warp - kVWarp0;
        const int vr = w4 * 32 + lane;
        const uint32_t vha = sb + kOffVhat;
        const uint32_t vscale_s = smem_u32(&cs.vscale[0]);
        for (int i = 0; i < nch; ++i) {
            const int st = i & 1;
            if (i > 0 && !warp_wait(bar(cs.dkv_full), (i - 1) & 1, abort_flag)) break;
            if (!warp_wait(bar(cs.full_v[st]), (i >> 1) & 1, abort_flag)) break;
            const int Lc = min(BC, L - i * BC);
            const bool live = vr < Lc;
            const uint32_t row = vslot(st) + vr * 128;
            uint4 x[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) x[c] = ld_shared_v4(row + (uint32_t)((c + vr) & 7) * 16);
            // ---- 1: Vhat.  lambda^(Lc-1-l) split as g_hi + g_lo (bf16
            // each) so that the packed bf16 FMAs give hi + lo = v g to ~16 bits.
            {
                const float g = live ? pw(Lc - 1 - vr) : 0.f;
                const __nv_bfloat16 ghb = __float2bfloat16_rn(g);
                const __nv_bfloat16 glb = __float2bfloat16_rn(g - __bfloat162float(ghb));
                const __nv_bfloat162 gh = __halves2bfloat162(ghb, ghb);
                const __nv_bfloat162 gl = __halves2bfloat162(glb, glb);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t ch = (uint32_t)((c + vr) & 7) * 16;
                    const uint32_t w[4] = {x[c].x, x[c].y, x[c].z, x[c].w};
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162 *>(&w[q]);
                        const __nv_bfloat162 h2 = __hmul2(v2, gh);
                        // exact residual of the rounded product, plus the g_lo term
                        __nv_bfloat162 l2 = __hfma2(v2, gh, __hneg2(h2));
                        l2 = __hfma2(v2, gl, l2);
                        hi[q] = *reinterpret_cast<const uint32_t *>(&h2);
                        lo[q] = *reinterpret_cast<const uint32_t *>(&l2);
                    }
                    st_shared_v4(vha + vr * 128 + ch, hi[0], hi[1], hi[2], hi[3]);
                    st_shared_v4(vha + kHalf + vr * 128 + ch, lo[0], lo[1], lo[2], lo[3]);
                }
                fence_proxy_async_smem();
                mbar_arrive(bar(cs.vhat_full));
            }
            // ---- 2: fp16 V for P V
            uint32_t mbits = 0;  // max |v| as packed bf16 magnitudes
            if (live) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    mbits = __vmaxu2(mbits, x[c].x & 0x7fff7fffu);
                    mbits = __vmaxu2(mbits, x[c].y & 0x7fff7fffu);
                    mbits = __vmaxu2(mbits, x[c].z & 0x7fff7fffu);
                    mbits = __vmaxu2(mbits, x[c].w & 0x7fff7fffu);
                }
            }
            float m = fmaxf(__uint_as_float(mbits << 16), __uint_as_float(mbits & 0xffff0000u));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) st_shared_f32(vmax_s + 4u * (uint32_t)((i & 1) * 4 + w4), m);
            mbar_arrive(bar(cs.vmax_ready[i & 1]));
            if (!warp_wait(bar(cs.vmax_ready[i & 1]), (i >> 1) & 1, abort_flag)) break;
            const uint32_t vm = vmax_s + 16u * (uint32_t)(i & 1);
            const float mt = fmaxf(fmaxf(ld_shared_f32(vm), ld_shared_f32(vm + 4)),
                                   fmaxf(ld_shared_f32(vm + 8), ld_shared_f32(vm + 12)));
            // no scale when the tile is comfortably inside fp16's normal
            // range, else 2^-f with max |v| 2^-f in [2^14, 2^15)
            const int f = (mt <= 1024.f && mt >= 0.0625f) ? 0 : fp16_scale_exp(mt, 14);
            if (threadIdx.x == kVWarp0 * 32)
                st_shared_f32(vscale_s + 4u * (uint32_t)(i & 3), exp2i(f));
            const float sc = live ? exp2i(-f) : 0.f;
            const bool unscaled = f == 0 && live;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t ch = (uint32_t)((c + vr) & 7) * 16;
                const uint32_t w[4] = {x[c].x, x[c].y, x[c].z, x[c].w};
                uint32_t hv[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    hv[q] = unscaled ? pack_f16(__uint_as_float(w[q] << 16),
                                                __uint_as_float(w[q] & 0xffff0000u))
                                     : pack_f16(__uint_as_float(w[q] << 16) * sc,
                                                __uint_as_float(w[q] & 0xffff0000u) * sc);
                st_shared_v4(row + ch, hv[0], hv[1], hv[2], hv[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(cs.vconv_full[st]));
        }
    }
    // warps 14 and 15 have no role

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && cs.abort) atomicOr(&g_tc_error, 1u);
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

// [T, H*D] bf16 row-major, box = 64 columns x 128 rows, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *ptr, int T, int H) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)H * D, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)H * D * 2};
    const cuuint32_t box[2] = {64, BC};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------- bounded-wait self test
// One CTA waits on an mbarrier that nothing ever arrives on; the bounded
// wait must give up after timeout_ns and raise the device error word.
__global__ void wait_timeout_selftest_kernel(uint64_t timeout_ns) {
    __shared__ uint64_t b;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        abort = 0;
        mbar_init(smem_u32(&b), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(smem_u32(&b), 0, &abort, timeout_ns))
        atomicOr(&g_tc_error, 1u);
}

}  // namespace

cudaError_t prefill_tc_bf16(const PrefillArgs &a) {
    if (a.head_dim != D || (a.chunk != 0 && a.chunk != BC)) return cudaErrorNotSupported;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, a.q, a.total_tokens, a.num_heads) ||
        !make_map(&mk, a.k, a.total_tokens, a.num_heads) ||
        !make_map(&mv, a.v, a.total_tokens, a.num_heads) ||
        !make_map(&mo, a.out, a.total_tokens, a.num_heads))
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static int attr_set_for[64] = {0};
    if (dev < 64 && !attr_set_for[dev]) {
        e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set_for[dev] = 1;
    }
    const long grid = (long)a.nseq * a.num_heads * NVS;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    prefill_tc_kernel<<<(unsigned)grid, kThreads, kSmemBytes, a.stream>>>(
        mq, mk, mv, mo, a.decay, a.cu_seqlens, a.nseq, a.total_tokens, a.num_heads,
        static_cast<__nv_bfloat16 *>(a.out), a.final_state);
    return cudaGetLastError();
}

cudaError_t take_device_error(cudaStream_t stream, unsigned int *err) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    unsigned int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(zero));
        if (e != cudaSuccess) return e;
    }
    *err = v;
    return cudaSuccess;
}

cudaError_t selftest_wait_timeout(uint64_t timeout_ns, cudaStream_t stream) {
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(timeout_ns);
    return cudaGetLastError();
}

}  // namespace la
