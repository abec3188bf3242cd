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
// undone in fp32 in the epilogue.  The fp32 state itself lives in TMEM for
// the whole sequence, as the sum of the two halves of the dKV accumulator:
// the worker warps write lambda^{B_{i+1}} KV_i back into it and the next
// dKV MMA accumulates onto that.  Nothing but q, k, v (read once per CTA)
// and out / final state (written once) touches HBM.
//
// TMEM (512 columns): S buffer b = columns [128b, 128b + 128): S (fp32), then
// P (fp16 pairs) over its first 64 columns and O1 (fp32) in its last 64;
// O2 = [256, 384); dKV / state = [384, 512).
//
// Warp roles (512 threads, 128 registers each):
//   warps 0-3    mask: S -> P = fp16(2^-e_j S (.) M) into TMEM, one lane
//                quadrant each, helped by warps 14 and 15 on the two
//                quadrants with the most blocks below the diagonal
//   warps 4-11   workers, two threads per row (token / state row), each with
//                32 of the 64 value columns: KV fold + write-back, the V tile
//                (Vhat hi/lo, fp16 V), KV copy, output
//   warp  12     MMA stream A (one thread): S and P V; TMA loads of the V ring
//   warp  13     MMA stream B (one thread): dKV and Q KV; TMA loads of the Q
//                and K rings
// (the anti-causal instantiation swaps warps 12/13 with 14/15: its heavy
// mask quadrants are 0 and 1, and a helper must sit on its quadrant)
// Each ring slot is reloaded, by a role that waits for that event anyway, as
// soon as the last MMA reading it has finished.
// Two issuing threads keep the tensor pipe fed while either one waits: the
// tcgen05 instruction queue is short, so a wait between two groups of MMAs
// from a single issuer leaves the pipe idle.
// Every wait is bounded and warp-uniform: a wait that gives up sets a CTA-wide
// abort flag, all roles leave their loops, in-flight TMA copies and MMAs are
// drained, TMEM is freed, and a device error word is raised for
// lightning_attn_device_status.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
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
constexpr int kThreads = 512;  // 16 warps: 4 per SM sub-partition, 128 registers
constexpr int kMaskWarps = 4;   // warps 0-3: one per TMEM lane quadrant
constexpr int kWorkWarp0 = 4;   // warps 4-11: fold, V tile, copy, output
constexpr int kWorkWarps = 8;
// Warps 12-15: two MMA issuers and two mask helpers.  A helper must sit on
// the TMEM lane quadrant it helps (a warp reads lanes 32 (warp % 4) ..), and
// the quadrants with the most mask blocks are 2 and 3 in the causal
// direction, 1 and 0 in the anti-causal one; the issuers take the other two.
template <bool kAnti> struct Roles {
    static constexpr int mma_a = kAnti ? 14 : 12;  // S and P V
    static constexpr int mma_b = kAnti ? 15 : 13;  // dKV and Q KV
    static constexpr int help2 = kAnti ? 13 : 14;  // second warp of the 3-block quadrant
    static constexpr int help3 = kAnti ? 12 : 15;  // second warp of the 4-block quadrant
};
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
    alignas(16) float pw[BC + 4];  // pw[e] = lambda^e, e = 0..BC
    float pwt[64];                 // pwt[32 + d] = lambda^d for d >= 0, 0 for d < 0
    uint64_t full_q[2], full_k[2], full_v[2], empty_q[2], empty_k[2], empty_v[2];
    uint64_t s_full[2], s_free[2], pv_ready[2], vmax_ready[2], pair[2], o_full[2];
    uint64_t o2_full, o2_ready, dkv_full, dkv_ready, done_a, done_b;
    uint32_t tmem_base;
    int abort;
    int seq_slot;
    int snap_base;                 // first snapshot of this CTA's sequence
    int pad;
    alignas(16) float vmax[2][8];  // per-warp max |v| of a chunk, double buffered
    float vscale[4];               // 2^f of V's fp16 scale, ring indexed by chunk & 3
    signed char rowe[2][BC];       // e_j of P's rows (scale 2^-e_j), per S buffer
    uint16_t mpart[2][2][2][32];   // [pair][chunk & 1][owner, helper][lane]: partial
                                   // row bounds, top 16 bits of the float
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
// 32 bytes to global memory: one 256-bit store when the address is 32-byte
// aligned (aligned32), else two 128-bit stores.
__device__ __forceinline__ void st_global_32B(void *p, const uint32_t *w, bool aligned32) {
    if (aligned32) {
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
                     "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
    } else {
        uint4 *q = reinterpret_cast<uint4 *>(p);
        q[0] = make_uint4(w[0], w[1], w[2], w[3]);
        q[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
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

// kAnti = false: o_t = sum_{u <= t} lambda^(t-u) (q_t . k_u) v_u (the method);
// kAnti = true: the anti-causal sum over u >= t with lambda^(u-t), for the
// reversed-time products of the backward pass.  Chunks keep their places
// (chunk c covers tokens [t0 + c B, t0 + c B + B)) and are walked last to
// first; inside a chunk the mask is the upper triangle lambda^(l-j), the
// carried state after chunk c is G_c = sum_{u >= start_c} lambda^(u-start_c)
// k_u^T v_u (G_c = lambda^{B_c} G_{c+1} + (Lambda_K K_c)^T V_c with
// Lambda_K = diag(lambda^l)), and row j of a chunk that has a successor gains
// lambda^(B - j) q_j G_{c+1}.  Every exponent is again >= 0.
// kSnap (causal only): the state after every snap_interval tokens of a
// sequence (a multiple of B) is also written to `snapshots` (per-block
// prefix cache, K3 report notes); sequence s's snapshots start at index
// sum_{s' < s} floor(L_s' / snap_interval).
// kCS: the block size B of the method (128, 64, 32 or 16).  Tiles are always
// 128 rows; a block of B < 128 tokens is a tile whose rows past B are masked
// exactly like the short last block of a sequence, and the next block's tile
// starts B tokens later (128 / B times the tensor-core work per token).
template <bool kAnti, bool kSnap, int kCS>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV,
                  const float *__restrict__ decay, const int32_t *__restrict__ cu, int nseq, int T,
                  int H, const float *initial_state, __nv_bfloat16 *__restrict__ out,
                  float *final_state, int min_len, float *snapshots, int snap_interval) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctrl &cs = *reinterpret_cast<Ctrl *>(base + kOffCtrl);
    const uint32_t sb = smem_u32(base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_dependency_wait();    // the previous kernel's writes are visible from here on
    grid_launch_dependents();  // the next dependent launch may be scheduled

    // ---- which (sequence, head, value slice) ----
    const int vs = blockIdx.x % NVS;
    const int h = (blockIdx.x / NVS) % H;
    const int s = sequence_of_rank(cu, nseq, blockIdx.x / (NVS * H), &cs.seq_slot);
    int t0 = __ldg(cu + s), t1 = __ldg(cu + s + 1);
    t0 = min(max(t0, 0), T);
    t1 = min(max(t1, t0), T);
    const int L = t1 - t0;
    if (L < min_len) return;  // a mixed step's decode launch owns this sequence
    static_assert(kCS == 128 || kCS == 64 || kCS == 32 || kCS == 16, "block size");
    const int nch = (L + kCS - 1) / kCS;
    // chunk processed at step i, and the length of chunk c (only the last
    // chunk of a sequence may be short)
    auto chunk_of = [&](int i) { return kAnti ? nch - 1 - i : i; };
    auto len_of = [&](int c) { return min(kCS, L - c * kCS); };
    using R = Roles<kAnti>;
    const float lam = __ldg(decay + h);
    // A sequence may continue from a cached state S0 (prefix KV cache,
    // §3.3.1): KV_{-1} = S0 instead of 0.  initial_state may be final_state
    // itself: every CTA reads its slice of S0 before it writes that slice.
    const bool has_init = initial_state != nullptr;
    const bool out32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;

    auto bar = [&](const uint64_t &b) { return smem_u32(&b); };
    const uint32_t pw_s = smem_u32(&cs.pw[0]);          // lambda^e at pw_s + 4 e
    const uint32_t rowe_s = smem_u32(&cs.rowe[0][0]);
    const uint32_t vmax_s = smem_u32(&cs.vmax[0][0]);
    const uint32_t vscale_s = smem_u32(&cs.vscale[0]);
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
            mbar_init(bar(cs.empty_q[i]), 2);  // S_i (stream A) and Q_i KV (stream B)
            mbar_init(bar(cs.empty_k[i]), 2);  // S_i (stream A) and dKV_i (stream B)
            mbar_init(bar(cs.empty_v[i]), 1);
            mbar_init(bar(cs.s_full[i]), 1);
            mbar_init(bar(cs.s_free[i]), kWorkWarps * 32);
            mbar_init(bar(cs.pv_ready[i]), 6 * 32 + kWorkWarps * 32);  // mask + worker warps
            mbar_init(bar(cs.vmax_ready[i]), kWorkWarps * 32);
            mbar_init(bar(cs.pair[i]), 64);
            // by chunk parity: near the end of a sequence stream A may finish
            // two P V groups before the state warps wait for the first
            mbar_init(bar(cs.o_full[i]), 1);
        }
        mbar_init(bar(cs.o2_full), 1);
        mbar_init(bar(cs.o2_ready), kWorkWarps * 32);
        mbar_init(bar(cs.dkv_full), 1);
        mbar_init(bar(cs.dkv_ready), kWorkWarps * 32);  // Vhat and write-back, per worker
        mbar_init(bar(cs.done_a), 1);
        mbar_init(bar(cs.done_b), 1);
        cs.abort = 0;
        fence_mbar_init();
    }
    if constexpr (kSnap) {
        // snapshots of the sequences before s (lengths clamped as above)
        if (threadIdx.x == 0) cs.snap_base = 0;
        __syncthreads();
        int part = 0;
        for (int s2 = threadIdx.x; s2 < s; s2 += kThreads) {
            int a0 = __ldg(cu + s2), a1 = __ldg(cu + s2 + 1);
            a0 = min(max(a0, 0), T);
            a1 = min(max(a1, a0), T);
            part += (a1 - a0) / snap_interval;
        }
        if (part) atomicAdd(&cs.snap_base, part);
    }
    for (int e = threadIdx.x; e <= BC; e += kThreads) cs.pw[e] = powf(lam, (float)e);
    if (threadIdx.x < 64) cs.pwt[threadIdx.x] = threadIdx.x < 32 ? 0.f : powf(lam, (float)(threadIdx.x - 32));
    if (warp == 0) {
        tmem_alloc(smem_u32(&cs.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // An allocation of all 512 columns can only start at lane 0, column 0.
    // The MMA issuers use that constant (their operands must be provably
    // warp-uniform to issue quickly); the TMEM loads and stores use the
    // allocated address.
    constexpr uint32_t tmem_mma = 0;
    const uint32_t tmem = __shfl_sync(0xffffffffu, cs.tmem_base, 0);
    volatile int *abort_flag = &cs.abort;
    const bool tmem_ok = tmem == tmem_mma;  // never expected to fail

    if (!tmem_ok) {
        // leave TMEM alone; the error word is raised below
    } else if (warp == R::mma_a) {
        // ================= MMA stream A: S and P V =================
        // Per chunk i: S_{i+1}, then P_i V_i, so that the mask warps turn
        // S_{i+1} into P_{i+1} while the tensor core runs P_i V_i and stream
        // B's dKV / Q KV.  The whole warp waits; lane 0 issues.
        // V ring: slot c & 1 is reloaded for chunk c as soon as P_{c-2} V_{c-2}
        // has finished reading it.
        int nv = 0;
        auto load_v = [&](int c) -> bool {
            const int st = c & 1;
            if (!warp_wait(bar(cs.empty_v[st]), ((c >> 1) & 1) ^ 1, abort_flag)) return false;
            if (elect_one()) {
                mbar_arrive_expect_tx(bar(cs.full_v[st]), kHalf);
                tma_load_2d(vslot(st), &tmV, bar(cs.full_v[st]), h * D + vs * DV,
                            t0 + chunk_of(c) * kCS);
            }
            __syncwarp();
            ++nv;
            return true;
        };
        if (elect_one()) tma_prefetch_desc(&tmV);
        __syncwarp();
        for (int c = 0; c < min(nch, 2); ++c) load_v(c);
        auto issue_s = [&](int i) -> bool {  // S_i = Q_i K_i^T
            const int st = i & 1;
            const uint32_t sph = (i >> 1) & 1;
            if (!warp_wait(bar(cs.full_q[st]), sph, abort_flag)) return false;
            if (!warp_wait(bar(cs.full_k[st]), sph, abort_flag)) return false;
            // buffer st is free once chunk i-2's output has read its O1
            if (!warp_wait(bar(cs.s_free[st]), sph ^ 1, abort_flag)) return false;
            tc_fence_after();
            const uint64_t dq = sdesc_sw128(qslot(st), 16, 1024);
            const uint64_t dk = sdesc_sw128(kslot(st), 16, 1024);
            if (elect_one()) {
                mma_group_ss<kKMajorS1, kKMajorS2, kKMajorS1, kKMajorS2>(tmem_mma + st * 128, dq, dk,
                                                                         kIdescS, 0u);
                mma_commit(bar(cs.s_full[st]));
                mma_commit(bar(cs.empty_q[st]));
                mma_commit(bar(cs.empty_k[st]));
            }
            __syncwarp();
            return true;
        };
        for (int i = -1; i < nch; ++i) {
            if (i + 1 < nch && !issue_s(i + 1)) break;
            if (i < 0) continue;
            const int st = i & 1;
            const uint32_t sph = (i >> 1) & 1;
            // O1_i = P_i V_i (fp16; P in the first half of the S buffer, O1
            // into its second half)
            if (!warp_wait(bar(cs.pv_ready[st]), sph, abort_flag)) break;
            tc_fence_after();
            const uint64_t dv = sdesc_sw128(vslot(st), kHalf, 1024);
            if (elect_one()) {
                mma_group_ts(tmem_mma + st * 128 + 64, tmem_mma + st * 128, dv, kIdescPV, 0u);
                mma_commit(bar(cs.o_full[st]));
                mma_commit(bar(cs.empty_v[st]));
            }
            __syncwarp();
            if (i + 2 < nch && !load_v(i + 2)) break;
        }
        // All MMAs must be finished before TMEM is released, and no load
        // may still be landing in shared memory when the CTA exits.
        if (elect_one()) mma_commit(bar(cs.done_a));
        __syncwarp();
        int no_abort = 0;
        warp_wait(bar(cs.done_a), 0, &no_abort);
        for (int c = max(0, nv - 2); c < nv; ++c)
            warp_wait(bar(cs.full_v[c & 1]), (c >> 1) & 1, &no_abort);
    } else if (warp == R::mma_b) {
        // ================= MMA stream B: dKV and Q KV =================
        // Also the Q and K rings: slot c & 1 is reloaded for chunk c as soon
        // as the MMAs of chunk c - 2 reading it have finished (S and Q KV for
        // Q, S and dKV for K; dKV and Q KV are issued here, Q KV last), a
        // whole chunk before S_c needs it.
        const uint32_t vha = sb + kOffVhat, kvb = sb + kOffKVb;
        int nq = 0;
        auto load_qk = [&](int c) -> bool {
            const int st = c & 1;
            if (!warp_wait(bar(cs.empty_k[st]), ((c >> 1) & 1) ^ 1, abort_flag)) return false;
            if (elect_one()) {
                mbar_arrive_expect_tx(bar(cs.full_k[st]), 2 * kHalf);
                const int row = t0 + chunk_of(c) * kCS;
                tma_load_2d(kslot(st), &tmK, bar(cs.full_k[st]), h * D, row);
                tma_load_2d(kslot(st) + kHalf, &tmK, bar(cs.full_k[st]), h * D + 64, row);
            }
            __syncwarp();
            if (!warp_wait(bar(cs.empty_q[st]), ((c >> 1) & 1) ^ 1, abort_flag)) return false;
            if (elect_one()) {
                mbar_arrive_expect_tx(bar(cs.full_q[st]), 2 * kHalf);
                const int row = t0 + chunk_of(c) * kCS;
                tma_load_2d(qslot(st), &tmQ, bar(cs.full_q[st]), h * D, row);
                tma_load_2d(qslot(st) + kHalf, &tmQ, bar(cs.full_q[st]), h * D + 64, row);
            }
            __syncwarp();
            ++nq;
            return true;
        };
        if (elect_one()) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
        }
        __syncwarp();
        for (int c = 0; c < min(nch, 2); ++c) load_qk(c);
        for (int i = 0; i < nch; ++i) {
            const int st = i & 1;
            const uint32_t sph = (i >> 1) & 1, ph = i & 1;
            // dKV += K_i^T [Vhat_hi | Vhat_lo]: the accumulator holds
            // lambda^{B_i} KV_{i-1}, written back by the worker warps
            if (!warp_wait(bar(cs.full_k[st]), sph, abort_flag)) break;
            if (!warp_wait(bar(cs.dkv_ready), ph, abort_flag)) break;
            tc_fence_after();
            const uint64_t dk = sdesc_sw128(kslot(st), kHalf, 1024);
            const uint64_t dvh = sdesc_sw128(vha, kHalf, 1024);
            if (elect_one()) {
                mma_group_ss<kMNMajorS1, kMNMajorS2, kMNMajorS1, kMNMajorS2>(
                    tmem_mma + kColDKV, dk, dvh, kIdescKV, (i > 0 || has_init) ? 1u : 0u);
                mma_commit(bar(cs.dkv_full));
                mma_commit(bar(cs.empty_k[st]));
            }
            __syncwarp();
            // O2_i = Q_i [KV_hi | KV_lo] (the state after chunk i-1)
            if (!warp_wait(bar(cs.full_q[st]), sph, abort_flag)) break;
            if (!warp_wait(bar(cs.o2_ready), ph, abort_flag)) break;
            tc_fence_after();
            const uint64_t dq = sdesc_sw128(qslot(st), 16, 1024);
            const uint64_t dkv = sdesc_sw128(kvb, kHalf, 1024);
            if (elect_one()) {
                mma_group_ss<kKMajorS1, kKMajorS2, kMNMajorS1, kMNMajorS2>(tmem_mma + kColO2, dq, dkv,
                                                                           kIdescO2, 0u);
                mma_commit(bar(cs.o2_full));
                mma_commit(bar(cs.empty_q[st]));
            }
            __syncwarp();
            if (i + 2 < nch && !load_qk(i + 2)) break;
        }
        if (elect_one()) mma_commit(bar(cs.done_b));
        __syncwarp();
        int no_abort = 0;
        warp_wait(bar(cs.done_b), 0, &no_abort);
        for (int c = max(0, nq - 2); c < nq; ++c) {  // no load may still be landing
            warp_wait(bar(cs.full_k[c & 1]), (c >> 1) & 1, &no_abort);
            warp_wait(bar(cs.full_q[c & 1]), (c >> 1) & 1, &no_abort);
        }
    } else if (warp < kMaskWarps || warp == R::help2 || warp == R::help3) {
        // ================= mask warps: S -> P =================
        // Row j of the chunk is TMEM lane j; the warps of lane quadrant q
        // (rows 32q .. 32q + 31) hold that quadrant's 32-column S blocks
        // cb <= q in registers, two at most per warp (quadrants 2 and 3 are
        // split between an owner warp, which has the diagonal block, and a
        // helper warp).  p_jl = S_jl lambda^(j-l) for l <= j, l < Lc, else 0,
        // goes to TMEM as fp16 scaled by 2^-e_j, a power of two chosen from
        // the row's max |p| (the two warps of a split quadrant exchange their
        // partial maxima) so that the row sits below 2^12: no overflow, and
        // 11 significant bits for everything within 2^25 of the maximum.
        //   pass 1: the decay goes into the held registers, p' = S f, with
        //     f = lambda^(lane - c) (masked) on the diagonal block and
        //     f = lambda^(32 (q - cb) - 1 - c) below it, where the rest of
        //     lambda^(j-l), lambda^(lane+1), is a row constant; max |p|;
        //   pass 2: p = p' 2^-e_j (times lambda^(lane+1) below the diagonal)
        //     to fp16.
        // P block cb lands in TMEM columns [16 cb, 16 cb + 16) of the S
        // buffer, written after every S block of the quadrant has been read
        // (the exchange orders the two warps of a pair).
        // Anti-causal: quadrant q holds the blocks cb >= q and
        // p_jl = S_jl lambda^(l-j) for l >= j; it is the causal quadrant
        // qm = 3 - q mirrored (block cb <-> 3 - cb), with
        //     f = lambda^(c - lane) (masked) on the diagonal block,
        //     f = lambda^(32 (cb - q - 1) + c) above it, row constant lambda^(32 - lane).
        const int q = warp & 3;                 // TMEM lane quadrant
        const int qm = kAnti ? 3 - q : q;       // the same quadrant in causal terms
        const bool owner = warp < kMaskWarps;
        const int j = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        // Blocks (causal terms): register set A holds a block below the
        // diagonal (none for the quadrant-0 owner); set B holds the owner's
        // diagonal block, or the quadrant-3 helper's second block.
        const bool has_a = !(owner && qm == 0);
        const int cba = owner ? qm - 1 : 0;
        const bool has_b = owner || qm == 3;
        const int cbb = owner ? qm : 1;
        const int pba = kAnti ? 3 - cba : cba;  // their blocks in the S buffer
        const int pbb = kAnti ? 3 - cbb : cbb;
        const int pr = qm - 2;  // pair index of a split quadrant
        const uint32_t pwt_s = smem_u32(&cs.pwt[32]);  // masked table: lambda^d at pwt_s + 4 d
        const float rowlam = kAnti ? pw(32 - lane) : pw(lane + 1);
        // p' = S f for a block dd >= 1 blocks off the diagonal (physical
        // block pb); returns max |p'| over the valid columns.
        auto decay_below = [&](float(&sv)[32], int dd, int pb, int Lc) -> float {
            float m = 0.f;
            if constexpr (kAnti) {
                // lambda^(32 (dd - 1) + c), c = 4g .. 4g + 3: four consecutive entries
                const uint32_t tab = pw_s + 4u * (uint32_t)(32 * (dd - 1));
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const uint4 f4 = ld_shared_v4(tab + 16u * (uint32_t)g);
                    const float2 x0 = f2_mul(make_float2(sv[4 * g], sv[4 * g + 1]),
                                             make_float2(__uint_as_float(f4.x), __uint_as_float(f4.y)));
                    const float2 x1 = f2_mul(make_float2(sv[4 * g + 2], sv[4 * g + 3]),
                                             make_float2(__uint_as_float(f4.z), __uint_as_float(f4.w)));
                    sv[4 * g] = x0.x;
                    sv[4 * g + 1] = x0.y;
                    sv[4 * g + 2] = x1.x;
                    sv[4 * g + 3] = x1.y;
                }
            } else {
                const uint32_t tab = pw_s + 4u * (uint32_t)(32 * dd - 32);
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    // lambda^(32 dd - 1 - c), c = 4g .. 4g + 3: the four
                    // table entries from 32 dd - 4 - 4g, reversed
                    const uint4 f4 = ld_shared_v4(tab + 16u * (uint32_t)(7 - g));
                    const float2 x0 = f2_mul(make_float2(sv[4 * g], sv[4 * g + 1]),
                                             make_float2(__uint_as_float(f4.w), __uint_as_float(f4.z)));
                    const float2 x1 = f2_mul(make_float2(sv[4 * g + 2], sv[4 * g + 3]),
                                             make_float2(__uint_as_float(f4.y), __uint_as_float(f4.x)));
                    sv[4 * g] = x0.x;
                    sv[4 * g + 1] = x0.y;
                    sv[4 * g + 2] = x1.x;
                    sv[4 * g + 3] = x1.y;
                }
            }
            const int lim = Lc - 1 - pb * 32;  // last valid column
            if (lim < 31) {  // ragged last chunk
#pragma unroll
                for (int c = 0; c < 32; ++c) sv[c] = c <= lim ? sv[c] : 0.f;
            }
#pragma unroll
            for (int c = 0; c < 32; ++c) m = fmaxf(m, fabsf(sv[c]));
            return m;
        };
        // p' = S lambda^(lane - c) for c <= lane, 0 above the diagonal
        // (anti-causal: lambda^(c - lane) for c >= lane, 0 below).
        auto decay_diag = [&](float(&sv)[32], int pb, int Lc) -> float {
            float m = 0.f;
            if constexpr (kAnti) {
                const uint32_t tab = pwt_s - 4u * (uint32_t)lane;
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    const float2 x = f2_mul(make_float2(sv[c], sv[c + 1]),
                                            make_float2(ld_shared_f32(tab + 4u * c),
                                                        ld_shared_f32(tab + 4u * (c + 1))));
                    sv[c] = x.x;
                    sv[c + 1] = x.y;
                }
            } else {
                const uint32_t tab = pwt_s + 4u * (uint32_t)lane;
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    const float2 x = f2_mul(make_float2(sv[c], sv[c + 1]),
                                            make_float2(ld_shared_f32(tab - 4u * c),
                                                        ld_shared_f32(tab - 4u * (c + 1))));
                    sv[c] = x.x;
                    sv[c + 1] = x.y;
                }
            }
            const int lim = Lc - 1 - pb * 32;
            if (lim < 31) {
#pragma unroll
                for (int c = 0; c < 32; ++c) sv[c] = c <= lim ? sv[c] : 0.f;
            }
#pragma unroll
            for (int c = 0; c < 32; ++c) m = fmaxf(m, fabsf(sv[c]));
            return m;
        };
        // p = p' * scale to fp16, into TMEM columns [16 cb, 16 cb + 16)
        auto store_block = [&](const float(&sv)[32], int cb, float scale, uint32_t scol) {
            const float2 s2 = make_float2(scale, scale);
            uint32_t pk[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float2 x = f2_mul(make_float2(sv[2 * m], sv[2 * m + 1]), s2);
                pk[m] = pack_f16(x.x, x.y);
            }
            tmem_st16(scol + cb * 16, pk);
        };
        uint32_t zero[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) zero[m] = 0u;
        for (int i = 0; i < nch; ++i) {
            const int st = i & 1;
            const uint32_t sph = (i >> 1) & 1;
            const int Lc = len_of(chunk_of(i));
            const uint32_t scol = tmem + lane_off + st * 128;
            if (!warp_wait(bar(cs.s_full[st]), sph, abort_flag)) break;
            tc_fence_after();
            float sa[32], sb2[32];
            if (has_a) tmem_ld32(scol + pba * 32, sa);
            if (has_b) tmem_ld32(scol + pbb * 32, sb2);
            tmem_wait_ld();
            // pass 1
            float mb = 0.f, md = 0.f;  // max |p'| off the diagonal, on it
            if (has_a) mb = decay_below(sa, qm - cba, pba, Lc);
            if (owner) md = decay_diag(sb2, pbb, Lc);
            else if (has_b) mb = fmaxf(mb, decay_below(sb2, qm - cbb, pbb, Lc));
            float bound = fmaxf(mb * rowlam, md);
            if (qm >= 2) {  // exchange with the other warp of the quadrant
                // Only the exponent of the bound matters: pass its top 16 bits
                // (a nonzero bound stays nonzero), so both warps pick the same e.
                const uint32_t ub = __float_as_uint(bound);
                const uint16_t mine = (uint16_t)((ub >> 16) | ((ub >> 16) == 0u && ub != 0u ? 1u : 0u));
                cs.mpart[pr][i & 1][owner ? 0 : 1][lane] = mine;
                mbar_arrive(bar(cs.pair[pr]));
                if (!warp_wait(bar(cs.pair[pr]), (uint32_t)(i & 1), abort_flag)) break;
                const uint32_t theirs = *reinterpret_cast<volatile uint16_t *>(
                    &cs.mpart[pr][i & 1][owner ? 1 : 0][lane]);
                bound = fmaxf(__uint_as_float((uint32_t)mine << 16), __uint_as_float(theirs << 16));
            }
            const int e = fp16_scale_exp(bound, 11);
            const float inv = exp2i(-e);
            // pass 2
            if (has_a) store_block(sa, pba, rowlam * inv, scol);
            if (has_b) store_block(sb2, pbb, owner ? inv : rowlam * inv, scol);
            if (owner) {  // the blocks on the masked side of the diagonal are zero
#pragma unroll 1
                for (int cb = qm + 1; cb < 4; ++cb) tmem_st16(scol + (kAnti ? 3 - cb : cb) * 16, zero);
                cs.rowe[st][j] = (signed char)e;
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(cs.pv_ready[st]));
        }
    } else if (warp < kWorkWarp0 + kWorkWarps) {
        // ================= worker warps =================
        // Thread (warp, lane) owns TMEM lane r = 32 (warp % 4) + lane -- token
        // r of the chunk and row r (a d_k index) of the state -- and the 32
        // value columns [c0, c0 + 32) of the CTA's 64-wide slice, c0 = 0 for
        // warps 4-7 and 32 for warps 8-11.  The fp32 state lives in the dKV
        // accumulator as the sum of its two 64-column halves.  Per chunk i:
        //   fold:   KV_i = sum of the halves; lambda^{B_{i+1}} KV_i / 2 is
        //           written back into both halves for dKV_{i+1} to accumulate
        //           onto;
        //   V tile: chunk i+1's V row segment, read from shared memory once:
        //           max |v| (for the tile's fp16 scale, exchanged among the
        //           eight warps), Vhat = lambda^(Lc-1-l) v as a hi/lo bf16 pair
        //           (dKV_{i+1} may go once every worker has written its part
        //           and its write-back), then V in place as fp16 with the
        //           tile's power-of-two scale (for P V);
        //   copy:   once Q_i KV_{i-1} has finished, a hi/lo bf16 copy of KV_i
        //           for Q_{i+1} KV_i, and Q_i KV_{i-1} (hi + lo) into registers;
        //   out:    once P_i V_i has finished, o = 2^(e + f) O1 + lambda^(r+1) O2.
        // Splitting the value columns between two threads per row halves the
        // latency of each step; the steps that gate the next MMA come first.
        const int wq = warp & 3;
        const int half = (warp - kWorkWarp0) >> 2;
        const int r = wq * 32 + lane;
        const int c0 = 32 * half;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t kvb = sb + kOffKVb, vha = sb + kOffVhat;
        const uint32_t tkv = tmem + lane_off + kColDKV + c0;  // hi half; lo half at + 64
        const uint32_t to2 = tmem + lane_off + kColO2 + c0;   // hi half; lo half at + 64
        // byte offset of the row's 16-byte piece 4 half + m (value columns
        // c0 + 8m .. c0 + 8m + 7) in a 128-byte swizzled row
        auto piece = [&](int m) { return (uint32_t)(((4 * half + m) ^ (r & 7)) * 16); };
        // hi/lo bf16 copy of 8 state values: hi = x with the low 16 bits
        // cleared (a bf16, exact); lo = x - hi (exact in fp32), also
        // truncated: hi + lo = x to about 2^-14 relative
        auto split8 = [&](const float *x, uint32_t(&hi)[4], uint32_t(&lo)[4]) {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t ua = __float_as_uint(x[2 * m]);
                const uint32_t ub = __float_as_uint(x[2 * m + 1]);
                hi[m] = __byte_perm(ua, ub, 0x7632);
                const float2 l2 = f2_sub(make_float2(__uint_as_float(ua), __uint_as_float(ub)),
                                         make_float2(__uint_as_float(ua & 0xffff0000u),
                                                     __uint_as_float(ub & 0xffff0000u)));
                lo[m] = __byte_perm(__float_as_uint(l2.x), __float_as_uint(l2.y), 0x7632);
            }
        };
        // the copy of this thread's 32 state values for the Q KV MMA
        auto store_kv_copy = [&](const float(&kv)[32]) {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                uint32_t hi[4], lo[4];
                split8(&kv[8 * m], hi, lo);
                st_shared_v4(kvb + r * 128 + piece(m), hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(kvb + kHalf + r * 128 + piece(m), lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_smem();
        };
        // lambda^{Lc} KV / 2 into both halves of the dKV accumulator, for the
        // next dKV MMA to accumulate onto
        auto write_back = [&](const float(&kv)[32], float decay_to_next) {
            const float dh = 0.5f * decay_to_next;
            const float2 d2 = make_float2(dh, dh);
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float2 x = f2_mul(make_float2(kv[2 * c], kv[2 * c + 1]), d2);
                w[2 * c] = __float_as_uint(x.x);
                w[2 * c + 1] = __float_as_uint(x.y);
            }
            tmem_st32(tkv, w);
            tmem_st32(tkv + 64, w);
            tmem_wait_st();
        };
        auto state_row = [&](float *base, long idx) {  // this thread's 32 values of a state
            return reinterpret_cast<float4 *>(base + ((idx * H + h) * D + r) * D + vs * DV + c0);
        };
        // V tile of the chunk processed at step j, part 1: max |v| of the
        // row segment (published for the tile's scale), Vhat hi/lo.  Keeps the
        // bf16 values in xv for part 2.
        uint4 xv[4];
        auto vtile_hat = [&](int j) -> bool {
            const int st = j & 1;
            if (!warp_wait(bar(cs.full_v[st]), (j >> 1) & 1, abort_flag)) return false;
            const int Lc = len_of(chunk_of(j));
            const bool live = r < Lc;
            const uint32_t row = vslot(st) + r * 128;
#pragma unroll
            for (int m = 0; m < 4; ++m) xv[m] = ld_shared_v4(row + piece(m));
            {  // max |v| (bf16 magnitudes, packed)
                uint32_t mbits = 0;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    mbits = __vmaxu2(__vmaxu2(mbits, xv[m].x & 0x7fff7fffu), xv[m].y & 0x7fff7fffu);
                    mbits = __vmaxu2(__vmaxu2(mbits, xv[m].z & 0x7fff7fffu), xv[m].w & 0x7fff7fffu);
                }
                if (!live) mbits = 0;
                float mx = fmaxf(__uint_as_float(mbits << 16), __uint_as_float(mbits & 0xffff0000u));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                if (lane == 0)
                    st_shared_f32(vmax_s + 4u * (uint32_t)((j & 1) * kWorkWarps + warp - kWorkWarp0),
                                  mx);
                mbar_arrive(bar(cs.vmax_ready[j & 1]));
            }
            // Vhat: lambda^(Lc-1-l) split as g_hi + g_lo (bf16 each) so that
            // the packed bf16 FMAs give hi + lo = v g to about 16 bits
            const float g = live ? pw(kAnti ? r : Lc - 1 - r) : 0.f;
            const __nv_bfloat16 ghb = __float2bfloat16_rn(g);
            const __nv_bfloat16 glb = __float2bfloat16_rn(g - __bfloat162float(ghb));
            const __nv_bfloat162 gh = __halves2bfloat162(ghb, ghb);
            const __nv_bfloat162 gl = __halves2bfloat162(glb, glb);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t w[4] = {xv[m].x, xv[m].y, xv[m].z, xv[m].w};
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
                st_shared_v4(vha + r * 128 + piece(m), hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(vha + kHalf + r * 128 + piece(m), lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_smem();
            return true;
        };
        // part 2: V itself, written back in place as fp16 with the tile's
        // power-of-two scale; rows past the chunk end become zero
        auto vtile_f16 = [&](int j) -> bool {
            if (!warp_wait(bar(cs.vmax_ready[j & 1]), (j >> 1) & 1, abort_flag)) return false;
            const uint32_t vm = vmax_s + 4u * (uint32_t)((j & 1) * kWorkWarps);
            const uint4 ma = ld_shared_v4(vm), mb = ld_shared_v4(vm + 16);
            const float mt = fmaxf(
                fmaxf(fmaxf(__uint_as_float(ma.x), __uint_as_float(ma.y)),
                      fmaxf(__uint_as_float(ma.z), __uint_as_float(ma.w))),
                fmaxf(fmaxf(__uint_as_float(mb.x), __uint_as_float(mb.y)),
                      fmaxf(__uint_as_float(mb.z), __uint_as_float(mb.w))));
            // no scale when the tile is comfortably inside fp16's normal
            // range, else 2^-f with max |v| 2^-f in [2^14, 2^15)
            const int f = (mt <= 1024.f && mt >= 0.0625f) ? 0 : fp16_scale_exp(mt, 14);
            if (threadIdx.x == kWorkWarp0 * 32) st_shared_f32(vscale_s + 4u * (uint32_t)(j & 3), exp2i(f));
            const bool live = r < len_of(chunk_of(j));
            const float sc = live ? exp2i(-f) : 0.f;
            const float2 sc2 = make_float2(sc, sc);
            const uint32_t row = vslot(j & 1) + r * 128;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t w[4] = {xv[m].x, xv[m].y, xv[m].z, xv[m].w};
                uint32_t hv[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 y = f2_mul(make_float2(__uint_as_float(w[q] << 16),
                                                        __uint_as_float(w[q] & 0xffff0000u)),
                                            sc2);
                    hv[q] = pack_f16(y.x, y.y);
                }
                st_shared_v4(row + piece(m), hv[0], hv[1], hv[2], hv[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(cs.pv_ready[j & 1]));
            return true;
        };

        // ---- prologue: the initial state, chunk 0's V tile ----
        if (has_init) {
            // KV_{-1} = S0: row r, this thread's 32 value columns
            const float4 *src = state_row(const_cast<float *>(initial_state), s);
            float4 *dst = (nch == 0 && final_state) ? state_row(final_state, s) : nullptr;
            float x[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 f = src[c];
                x[4 * c] = f.x;
                x[4 * c + 1] = f.y;
                x[4 * c + 2] = f.z;
                x[4 * c + 3] = f.w;
            }
            if (dst) {  // empty sequence: the state is the cached one
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dst[c] = make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
            }
            store_kv_copy(x);
            if (nch > 0) write_back(x, pw(len_of(chunk_of(0))));
        } else {
            // KV_{-1} = 0
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                st_shared_v4(kvb + r * 128 + piece(m), 0u, 0u, 0u, 0u);
                st_shared_v4(kvb + kHalf + r * 128 + piece(m), 0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(bar(cs.o2_ready));  // Q_0 KV_{-1} may go
        bool ok = true;
        if (nch > 0) {
            ok = vtile_hat(0);
            if (ok) {
                tc_fence_before();
                mbar_arrive(bar(cs.dkv_ready));  // dKV_0 accumulates onto lambda^{B_0} S0 (or overwrites)
                ok = vtile_f16(0);
            }
        }

        for (int i = 0; ok && i < nch; ++i) {
            const int st = i & 1;
            const uint32_t sph = (i >> 1) & 1, ph = i & 1;
            const int Lc = len_of(chunk_of(i));
            const bool last = i + 1 == nch;
            // ---- fold ----
            if (!warp_wait(bar(cs.dkv_full), ph, abort_flag)) break;
            tc_fence_after();
            float kv[32];
            {
                float b[32];
                tmem_ld32(tkv, kv);
                tmem_ld32(tkv + 64, b);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float2 x = f2_add(make_float2(kv[2 * c], kv[2 * c + 1]),
                                            make_float2(b[2 * c], b[2 * c + 1]));
                    kv[2 * c] = x.x;
                    kv[2 * c + 1] = x.y;
                }
            }
            if constexpr (kSnap) {
                // the state after the first (i + 1) B tokens closes a block
                const int end = (i + 1) * kCS;
                if (end <= L && end % snap_interval == 0) {
                    float4 *dst = state_row(snapshots, cs.snap_base + end / snap_interval - 1);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        dst[c] = make_float4(kv[4 * c], kv[4 * c + 1], kv[4 * c + 2], kv[4 * c + 3]);
                }
            }
            if (!last) {
                write_back(kv, pw(len_of(chunk_of(i + 1))));
            } else if (final_state) {
                float4 *dst = state_row(final_state, s);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dst[c] = make_float4(kv[4 * c], kv[4 * c + 1], kv[4 * c + 2], kv[4 * c + 3]);
            }
            // ---- V tile of the next chunk ----
            if (!last) {
                // Vhat_{i+1} may overwrite Vhat_i: dKV_i has finished
                if (!vtile_hat(i + 1)) break;
                tc_fence_before();
                mbar_arrive(bar(cs.dkv_ready));
                if (!vtile_f16(i + 1)) break;
            }
            // ---- copy, O2 ----
            if (!warp_wait(bar(cs.o2_full), ph, abort_flag)) break;
            tc_fence_after();
            if (!last) store_kv_copy(kv);
            float o2[32];
            {
                float b[32];
                tmem_ld32(to2, o2);
                tmem_ld32(to2 + 64, b);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float2 x = f2_add(make_float2(o2[2 * c], o2[2 * c + 1]),
                                            make_float2(b[2 * c], b[2 * c + 1]));
                    o2[2 * c] = x.x;
                    o2[2 * c + 1] = x.y;
                }
            }
            tc_fence_before();
            mbar_arrive(bar(cs.o2_ready));
            // ---- out: o_r = 2^(e_r + f) O1_r + lambda^(r+1) O2_r ----
            if (!warp_wait(bar(cs.o_full[st]), sph, abort_flag)) break;
            if (!warp_wait(bar(cs.pv_ready[st]), sph, abort_flag)) break;  // orders the scales
            tc_fence_after();
            const float s1 = exp2i((int)*reinterpret_cast<volatile signed char *>(&cs.rowe[st][r])) *
                             ld_shared_f32(vscale_s + 4u * (uint32_t)(i & 3));
            // lambda^(r+1) Q KV_{i-1}; anti-causal: lambda^(B-r) Q G_{c+1}
            // (G is zero before the first step, when chunk c may be short)
            const float qf = kAnti ? pw(kCS - r) : pw(r + 1);
            const float2 s12 = make_float2(s1, s1), qf2 = make_float2(qf, qf);
            float a[32];
            tmem_ld32(tmem + lane_off + st * 128 + 64 + c0, a);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(cs.s_free[st]));  // all TMEM reads of this chunk are done
            uint32_t w[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float2 y = f2_fma(qf2, make_float2(o2[2 * m], o2[2 * m + 1]),
                                        f2_mul(s12, make_float2(a[2 * m], a[2 * m + 1])));
                w[m] = pack_bf16(y.x, y.y);
            }
            // Lanes 2k and 2k+1 (rows r and r+1) swap halves so that each
            // store instruction writes whole 64-byte row pieces: the first
            // writes row 2k (the even lane its bytes 0-31, the odd lane the
            // even lane's bytes 32-63), the second row 2k+1; 16 rows per
            // instruction instead of 32 half sectors.
            const bool odd = lane & 1;
            uint32_t mine[8], other[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const uint32_t send = odd ? w[m] : w[8 + m];  // even: bytes 32-63; odd: 0-31
                other[m] = __shfl_xor_sync(0xffffffffu, send, 1);
                mine[m] = odd ? w[8 + m] : w[m];
            }
            const int rbase = wq * 32 + (lane & ~1);
            const long trow = (long)(t0 + chunk_of(i) * kCS + rbase);
            __nv_bfloat16 *o0 = out + (trow * H + h) * D + vs * DV + c0 + (odd ? 16 : 0);
            __nv_bfloat16 *o1 = o0 + (long)H * D;
            // row rbase: even lane's own low half, odd lane the received high half;
            // row rbase + 1: even lane the received low half, odd lane its own high half
            const uint32_t *r0 = odd ? other : mine;
            const uint32_t *r1 = odd ? mine : other;
            if (rbase < Lc) st_global_32B(o0, r0, out32);
            if (rbase + 1 < Lc) st_global_32B(o1, r1, out32);
        }
        if (nch == 0 && final_state && !has_init) {  // empty sequence: the state stays zero
            float4 *dst = state_row(final_state, s);
#pragma unroll
            for (int c = 0; c < 8; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && (cs.abort || !tmem_ok)) atomicOr(&g_tc_error, 1u);
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

using TcKernel = decltype(&prefill_tc_kernel<false, false, BC>);

template <int CS>
TcKernel pick_kernel(bool anti, bool snap) {
    return anti ? prefill_tc_kernel<true, false, CS>
           : snap ? prefill_tc_kernel<false, true, CS>
                  : prefill_tc_kernel<false, false, CS>;
}

}  // namespace

// A block of 256 tokens (the MiniMax-01 report's block, §3.2 and §3.3.3) is
// computed as two 128-row tiles: the term that couples its halves,
// [(Q_b K_a^T) (.) M] V_a for the second half b and the first half a, is
// taken through the state carried after a, Lambda_Q Q_b (Lambda_K K_a)^T V_a,
// which is the same sum regrouped (equal in exact arithmetic), and the
// block's state update lambda^256 KV + (Lambda_K K)^T V is the two tile
// updates composed.  A 256-row left product in one piece would need a third
// 128-column S tile in TMEM, whose 512 columns already hold two S tiles, O2
// and the state.
cudaError_t prefill_tc_bf16(const PrefillArgs &a) {
    const int cs = a.chunk == 0 ? BC : a.chunk;  // the method's block size
    if (a.head_dim != D || (cs != 256 && cs != 128 && cs != 64 && cs != 32 && cs != 16))
        return cudaErrorNotSupported;
    // rows are written in place; the anti-causal kernel starts from a zero state
    if (a.reverse_out || (a.anti_causal && a.initial_state)) return cudaErrorNotSupported;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, a.total_tokens, a.num_heads) ||
        !make_map(&mk, a.k, a.total_tokens, a.num_heads) ||
        !make_map(&mv, a.v, a.total_tokens, a.num_heads))
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool snap = a.snapshots != nullptr;
    if (snap && (a.anti_causal || a.snapshot_interval <= 0 || a.snapshot_interval % cs != 0))
        return cudaErrorNotSupported;
    const int csi = cs >= 128 ? 0 : cs == 64 ? 1 : cs == 32 ? 2 : 3;
    const TcKernel kern = csi == 0   ? pick_kernel<128>(a.anti_causal, snap)
                          : csi == 1 ? pick_kernel<64>(a.anti_causal, snap)
                          : csi == 2 ? pick_kernel<32>(a.anti_causal, snap)
                                     : pick_kernel<16>(a.anti_causal, snap);
    // The shared-memory opt-in is set once per device and instantiation (one
    // bit each: (causal, anti-causal, causal with snapshots) x block size);
    // concurrent first calls may both set it, which is harmless.
    static std::atomic<int> attr_set_for[64];
    const int bit = 1 << ((a.anti_causal ? 1 : snap ? 2 : 0) * 4 + csi);
    if (dev >= 64 || !(attr_set_for[dev].load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set_for[dev].fetch_or(bit, std::memory_order_release);
    }
    const long grid = (long)(a.rank_limit > 0 ? a.rank_limit : a.nseq) * a.num_heads * NVS;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    e = launch_dependent(kern, (unsigned)grid, kThreads, kSmemBytes, a.stream, mq, mk, mv, a.decay,
                         a.cu_seqlens, a.nseq, a.total_tokens, a.num_heads, a.initial_state,
                         static_cast<__nv_bfloat16 *>(a.out), a.final_state, a.min_len,
                         a.snapshots, a.snapshot_interval);
    return e != cudaSuccess ? e : cudaGetLastError();
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
