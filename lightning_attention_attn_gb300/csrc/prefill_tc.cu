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
// by the two sibling CTAs through L2.  Per 128-token chunk the CTA runs four
// tcgen05 MMAs (M = 128):
//     S   = Q K^T          128x128x128  -> TMEM (double buffered)
//     dKV = K^T Vhat       128x 64x128  -> TMEM   (Vhat = Lambda_K V)
//     O2  = Q KVb          128x 64x128  -> TMEM   (KVb = bf16 copy of KV_{i-1})
//     O1  = P V            128x 64x128  -> TMEM   (P = bf16 of S (.) M)
// and the fp32 state lives in registers of the state warpgroup for the
// whole sequence; only a bf16 copy of it (the MMA operand) goes to shared
// memory.  Nothing but q, k, v (read once per CTA) and out / final state
// (written once) touches HBM.
//
// Warp roles (320 threads):
//   warps 0-3  mask warpgroup: S -> P = bf16(S (.) M) into shared memory
//   warps 4-7  state warpgroup: Vhat, KV update, KVb, output epilogue
//   warp  8    TMA producer (2-stage ring of Q, K, V tiles)
//   warp  9    MMA issuer (one thread)
// Every wait is bounded: a wait that gives up sets a CTA-wide abort flag, all
// roles leave their loops, in-flight TMA loads and MMAs are drained, TMEM is
// freed, and a device error word is raised for lightning_attn_device_status.
#include <cuda.h>
#include <cuda_bf16.h>
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
constexpr int kThreads = 320;
constexpr int kStateWarp0 = 4;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

// Shared memory (offsets from a 1024-byte aligned base).  Operand tiles are
// 128-byte swizzled rows of 64 bf16, 8-row atoms of 1024 bytes.
constexpr uint32_t kHalf = BC * 128;                  // 128 rows x 128 B = 16 KB
constexpr uint32_t kQBytes = 2 * kHalf;               // Q: d split in two 64-col halves
constexpr uint32_t kKBytes = 2 * kHalf;
constexpr uint32_t kVBytes = kHalf;                   // V slice: 64 cols
constexpr uint32_t kStageBytes = kQBytes + kKBytes + kVBytes;  // 80 KB
constexpr int kStages = 2;
constexpr uint32_t kOffP = kStages * kStageBytes;     // P: 128 x 128 bf16, two halves
constexpr uint32_t kOffVhat = kOffP + 2 * kHalf;      // Vhat: 128 tokens x 64
constexpr uint32_t kOffKVb = kOffVhat + kHalf;        // KVb: 128 d_k x 64
constexpr uint32_t kOffCtrl = kOffKVb + kHalf;

struct Ctrl {
    uint64_t full[kStages], empty[kStages];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full, p_free, o_full, o_free;
    uint64_t dkv_full, dkv_free, vhat_full, kv_full, kv_free, mma_done;
    uint32_t tmem_base;
    int abort;
    int seq_slot;
    int pad;
    float pw[BC + 4];  // pw[e] = lambda^e, e = 0..BC
};
constexpr uint32_t kSmemBytes = kOffCtrl + sizeof(Ctrl) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

// TMEM columns (fp32 accumulators, lane = row).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO1 = 256, kColO2 = 320, kColDKV = 384;

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0, 0);   // Q (K-major) x K (K-major)
constexpr uint32_t kIdescKV = idesc_bf16_f32(128, DV, 1, 1);   // K^T (M-major) x Vhat (N-major)
constexpr uint32_t kIdescO2 = idesc_bf16_f32(128, DV, 0, 1);   // Q (K-major) x KVb (N-major)
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, DV, 0, 1);   // P (K-major) x V (N-major)

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(v);
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

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const float *__restrict__ decay,
                  const int32_t *__restrict__ cu, int nseq, int T, int H,
                  __nv_bfloat16 *__restrict__ out, float *__restrict__ final_state) {
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

    // ---- set-up ----
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(bar(cs.full[i]), 1);
            mbar_init(bar(cs.empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(cs.s_full[i]), 1);
            mbar_init(bar(cs.s_free[i]), 128);
        }
        mbar_init(bar(cs.p_full), 128);
        mbar_init(bar(cs.p_free), 1);
        mbar_init(bar(cs.o_full), 1);
        mbar_init(bar(cs.o_free), 128);
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
    // P's blocks strictly above the diagonal are never written: zero them once.
    for (int e = threadIdx.x; e < (int)(2 * kHalf / 16); e += kThreads)
        st_shared_v4(sb + kOffP + e * 16, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
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
            int issued = 0;
            for (int i = 0; i < nch; ++i) {
                const int st = i & 1;
                const uint32_t sph = (i >> 1) & 1;
                if (!mbar_wait(bar(cs.empty[st]), sph ^ 1, abort_flag, kTimeoutNs)) break;
                const uint32_t stage = sb + st * kStageBytes;
                const uint32_t fb = bar(cs.full[st]);
                mbar_arrive_expect_tx(fb, kStageBytes);
                const int y = t0 + i * BC;
                tma_load_2d(stage, &tmQ, fb, h * D, y);
                tma_load_2d(stage + kHalf, &tmQ, fb, h * D + 64, y);
                tma_load_2d(stage + kQBytes, &tmK, fb, h * D, y);
                tma_load_2d(stage + kQBytes + kHalf, &tmK, fb, h * D + 64, y);
                tma_load_2d(stage + kQBytes + kKBytes, &tmV, fb, h * D + vs * DV, y);
                ++issued;
            }
            // Never leave with a load still landing in shared memory.
            int no_abort = 0;
            for (int i = max(0, issued - kStages); i < issued; ++i)
                mbar_wait(bar(cs.full[i & 1]), (i >> 1) & 1, &no_abort, kTimeoutNs);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ================= MMA issuer =================
        if (lane == 0) {
            const uint32_t pa = sb + kOffP, vha = sb + kOffVhat, kvb = sb + kOffKVb;
            for (int i = 0; i < nch; ++i) {
                const int st = i & 1;
                const uint32_t sph = (i >> 1) & 1, ph = i & 1;
                const uint32_t qa = sb + st * kStageBytes, ka = qa + kQBytes, va = ka + kKBytes;
                const uint32_t colS = st ? kColS1 : kColS0;
                if (!mbar_wait(bar(cs.full[st]), sph, abort_flag, kTimeoutNs)) break;
                // S_i = Q_i K_i^T
                if (!mbar_wait(bar(cs.s_free[st]), sph ^ 1, abort_flag, kTimeoutNs)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                    mma_bf16(tmem + colS, sdesc_sw128(qa + off, 16, 1024),
                             sdesc_sw128(ka + off, 16, 1024), kIdescS, kk > 0);
                }
                mma_commit(bar(cs.s_full[st]));
                // dKV_i = K_i^T Vhat_i
                if (!mbar_wait(bar(cs.vhat_full), ph, abort_flag, kTimeoutNs)) break;
                if (!mbar_wait(bar(cs.dkv_free), ph ^ 1, abort_flag, kTimeoutNs)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BC / 16; ++kk)
                    mma_bf16(tmem + kColDKV, sdesc_sw128(ka + kk * 2048, kHalf, 1024),
                             sdesc_sw128(vha + kk * 2048, kHalf, 1024), kIdescKV, kk > 0);
                mma_commit(bar(cs.dkv_full));
                // O2_i = Q_i KVb_{i-1}
                if (!mbar_wait(bar(cs.kv_full), ph, abort_flag, kTimeoutNs)) break;
                if (!mbar_wait(bar(cs.o_free), ph ^ 1, abort_flag, kTimeoutNs)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                    mma_bf16(tmem + kColO2, sdesc_sw128(qa + off, 16, 1024),
                             sdesc_sw128(kvb + kk * 2048, kHalf, 1024), kIdescO2, kk > 0);
                }
                mma_commit(bar(cs.kv_free));
                // O1_i = P_i V_i
                if (!mbar_wait(bar(cs.p_full), ph, abort_flag, kTimeoutNs)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BC / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                    mma_bf16(tmem + kColO1, sdesc_sw128(pa + off, 16, 1024),
                             sdesc_sw128(va + kk * 2048, kHalf, 1024), kIdescPV, kk > 0);
                }
                mma_commit(bar(cs.o_full));
                mma_commit(bar(cs.p_free));
                mma_commit(bar(cs.empty[st]));
            }
            // All MMAs must be finished before TMEM is released.
            mma_commit(bar(cs.mma_done));
            int no_abort = 0;
            mbar_wait(bar(cs.mma_done), 0, &no_abort, kTimeoutNs);
        }
        __syncwarp();
    } else if (warp < kStateWarp0) {
        // ================= mask warpgroup: S -> P =================
        const int j = warp * 32 + lane;  // token row within the chunk
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        float colf[32];  // lambda^(31-c)
#pragma unroll
        for (int c = 0; c < 32; ++c) colf[c] = cs.pw[31 - c];
        for (int i = 0; i < nch; ++i) {
            const int sbuf = i & 1;
            const uint32_t sph = (i >> 1) & 1, ph = i & 1;
            const int Lc = min(BC, L - i * BC);
            const uint32_t colS = sbuf ? kColS1 : kColS0;
            if (!mbar_wait(bar(cs.s_full[sbuf]), sph, abort_flag, kTimeoutNs)) break;
            tc_fence_after();
            if (!mbar_wait(bar(cs.p_free), ph ^ 1, abort_flag, kTimeoutNs)) break;
            for (int cb = 0; cb <= warp; ++cb) {  // column blocks on/below the diagonal
                float sv[32];
                tmem_ld32(tmem + lane_off + colS + cb * 32, sv);
                tmem_wait_ld();
                float p[32];
                if (cb < warp) {
                    // lambda^(j-l) = lambda^(j-(32cb+31)) * lambda^(31-c), both exponents >= 0
                    const float rowf = cs.pw[j - cb * 32 - 31];
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        p[c] = (cb * 32 + c < Lc) ? sv[c] * (rowf * colf[c]) : 0.f;
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float m = cs.pw[max(lane - c, 0)];
                        p[c] = (c <= lane && cb * 32 + c < Lc) ? sv[c] * m : 0.f;
                    }
                }
                const uint32_t row = sb + kOffP + (cb >> 1) * kHalf + j * 128;
#pragma unroll
                for (int c16 = 0; c16 < 4; ++c16) {
                    const uint32_t phys = (uint32_t)(((cb & 1) * 4 + c16) ^ (j & 7));
                    st_shared_v4(row + phys * 16, pack_bf16(p[8 * c16 + 0], p[8 * c16 + 1]),
                                 pack_bf16(p[8 * c16 + 2], p[8 * c16 + 3]),
                                 pack_bf16(p[8 * c16 + 4], p[8 * c16 + 5]),
                                 pack_bf16(p[8 * c16 + 6], p[8 * c16 + 7]));
                }
            }
            tc_fence_before();
            mbar_arrive(bar(cs.s_free[sbuf]));
            fence_proxy_async_smem();
            mbar_arrive(bar(cs.p_full));
        }
    } else {
        // ================= state warpgroup =================
        const int r = (warp - kStateWarp0) * 32 + lane;  // TMEM lane: d_k row / token row
        const uint32_t lane_off = (uint32_t)((warp - kStateWarp0) * 32) << 16;
        const uint32_t vha = sb + kOffVhat, kvb = sb + kOffKVb;
        float kv[DV];
#pragma unroll
        for (int c = 0; c < DV; ++c) kv[c] = 0.f;
        // KV_{-1} = 0
#pragma unroll
        for (int c = 0; c < 8; ++c) st_shared_v4(kvb + r * 128 + c * 16, 0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
        mbar_arrive(bar(cs.kv_full));

        // Vhat_i = Lambda_K V_i: row r (token r) scaled by lambda^(Lc-1-r).
        auto make_vhat = [&](int i) -> bool {
            const int st = i & 1;
            if (!mbar_wait(bar(cs.full[st]), (i >> 1) & 1, abort_flag, kTimeoutNs)) return false;
            const int Lc = min(BC, L - i * BC);
            const float g = (r < Lc) ? cs.pw[Lc - 1 - r] : 0.f;
            const uint32_t src = sb + st * kStageBytes + kQBytes + kKBytes + r * 128;
            const uint32_t dst = vha + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t ch = (uint32_t)((c + r) & 7) * 16;  // rotate: no bank conflicts
                const uint4 x = ld_shared_v4(src + ch);
                float2 a = unpack_bf16(x.x), b = unpack_bf16(x.y), e = unpack_bf16(x.z),
                       f = unpack_bf16(x.w);
                st_shared_v4(dst + ch, pack_bf16(a.x * g, a.y * g), pack_bf16(b.x * g, b.y * g),
                             pack_bf16(e.x * g, e.y * g), pack_bf16(f.x * g, f.y * g));
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(cs.vhat_full));
            return true;
        };

        bool ok = nch > 0 ? make_vhat(0) : true;
        for (int i = 0; ok && i < nch; ++i) {
            const uint32_t ph = i & 1;
            const int Lc = min(BC, L - i * BC);
            // ---- KV_i = lambda^{Lc} KV_{i-1} + dKV_i ----
            if (!mbar_wait(bar(cs.dkv_full), ph, abort_flag, kTimeoutNs)) break;
            tc_fence_after();
            const float dec = cs.pw[Lc];
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                float d32[32];
                tmem_ld32(tmem + lane_off + kColDKV + hlf * 32, d32);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) kv[hlf * 32 + c] = fmaf(dec, kv[hlf * 32 + c], d32[c]);
            }
            tc_fence_before();
            mbar_arrive(bar(cs.dkv_free));
            // ---- bf16 copy of KV_i for the next chunk's Q KV (after O2_i read KV_{i-1}) ----
            if (!mbar_wait(bar(cs.kv_free), ph, abort_flag, kTimeoutNs)) break;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t phys = (uint32_t)(c ^ (r & 7));
                st_shared_v4(kvb + r * 128 + phys * 16, pack_bf16(kv[8 * c + 0], kv[8 * c + 1]),
                             pack_bf16(kv[8 * c + 2], kv[8 * c + 3]),
                             pack_bf16(kv[8 * c + 4], kv[8 * c + 5]),
                             pack_bf16(kv[8 * c + 6], kv[8 * c + 7]));
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(cs.kv_full));
            // ---- next chunk's Vhat, so its dKV MMA can start early ----
            if (i + 1 < nch && !make_vhat(i + 1)) break;
            // ---- output: o_j = O1_j + lambda^(j+1) O2_j ----
            if (!mbar_wait(bar(cs.o_full), ph, abort_flag, kTimeoutNs)) break;
            tc_fence_after();
            const float qf = cs.pw[r + 1];
            __nv_bfloat16 *orow = out + ((long)(t0 + i * BC + r) * H + h) * D + vs * DV;
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                float a[32], b[32];
                tmem_ld32(tmem + lane_off + kColO1 + hlf * 32, a);
                tmem_ld32(tmem + lane_off + kColO2 + hlf * 32, b);
                tmem_wait_ld();
                if (r < Lc) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + hlf * 32);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 w;
                        w.x = pack_bf16(fmaf(qf, b[8 * c + 0], a[8 * c + 0]), fmaf(qf, b[8 * c + 1], a[8 * c + 1]));
                        w.y = pack_bf16(fmaf(qf, b[8 * c + 2], a[8 * c + 2]), fmaf(qf, b[8 * c + 3], a[8 * c + 3]));
                        w.z = pack_bf16(fmaf(qf, b[8 * c + 4], a[8 * c + 4]), fmaf(qf, b[8 * c + 5], a[8 * c + 5]));
                        w.w = pack_bf16(fmaf(qf, b[8 * c + 6], a[8 * c + 6]), fmaf(qf, b[8 * c + 7], a[8 * c + 7]));
                        dst[c] = w;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(cs.o_free));
        }
        if (final_state && !*abort_flag) {
            float4 *dst = reinterpret_cast<float4 *>(final_state + (((long)s * H + h) * D + r) * D +
                                                     vs * DV);
#pragma unroll
            for (int c = 0; c < DV / 4; ++c)
                dst[c] = make_float4(kv[4 * c], kv[4 * c + 1], kv[4 * c + 2], kv[4 * c + 3]);
        }
    }

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
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, a.total_tokens, a.num_heads) ||
        !make_map(&mk, a.k, a.total_tokens, a.num_heads) ||
        !make_map(&mv, a.v, a.total_tokens, a.num_heads))
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
        mq, mk, mv, a.decay, a.cu_seqlens, a.nseq, a.total_tokens, a.num_heads,
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
