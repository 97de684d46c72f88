// tc_bwd.cu -- tensor-core (tcgen05 / TMEM / TMA) PSA backward, bf16 storage.
//
// "Struct PsaFa2Backward" (vision_rs yolo attention psa): the backward of the
// lo/hi pair of FA2 calls that share Q and K.  Here the pair runs as ONE
// attention with a 2d-wide value [V_lo | V_hi]:
//   dS = P o (dO_lo V_lo^T + dO_hi V_hi^T - D),  D = rowsum(dO_lo o O_lo) + rowsum(dO_hi o O_hi)
// so S and P are recomputed once for both calls and dQ, dK come out already
// summed (the page's atomic_add into the shared dQ/dK sections is not needed
// for that).
//
// Decomposition: one CTA per (batch*head, 128-key tile).  The CTA keeps K_j,
// V_lo,j, V_hi,j in shared memory and its dV_lo, dV_hi, dK accumulators in
// TMEM, and walks over all 128-query tiles i (the page's "dK_n / dV_n by
// iterating over all Q rows"):
//   S^T  = K_j Q_i^T                 (M = 128 keys, N = 128 queries, K = d)
//   dP^T = V_lo,j dO_lo,i^T + V_hi,j dO_hi,i^T          (K = 2d)
//   P^T  = exp2(S^T * scale*log2e - LSE_i*log2e),  dS^T = P^T o (dP^T - D_i)
//   dV_h += P^T dO_h,i ;  dK += dS^T Q_i ;  dQ_i(partial) = dS_i K_j
// The dQ partial of each (key tile, query tile) is added into an fp32
// accumulator in the workspace; a last kernel scales and casts it into d_packed.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer (one
// thread) and TMEM owner, warps 2-5 softmax-gradient (one key row per
// thread), warps 6-9 dQ drain (one query row per thread).
//
// Every mbarrier wait is bounded (kTimeoutNs); on timeout the CTA sets a device
// error word (read by psa_attn_sync_status), skips the rest of its work, waits
// (bounded) for its own TMA copies in flight, frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdio>
#include <mutex>
#include <string>

#include "common.cuh"
#include "psa_attn.h"
#include "psa_internal.h"
#include "tc_ptx.cuh"

namespace psa {
namespace {

using namespace psa::tc;
using bf16 = __nv_bfloat16;

__device__ int g_tc_error = 0;  // 0 = fine; else (1 + role) << 24 | tile

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr int kThreads = 320;

template <int D>
struct Cfg {
    static constexpr int BM = 128;            // keys per CTA (MMA M)
    static constexpr int BQ = 128;            // queries per tile
    static constexpr int ROWB = D * 2;        // bytes per [*, D] bf16 row
    static constexpr int TILE = 128 * ROWB;   // bytes per [128, D] tile
    static constexpr uint32_t SW = D == 64 ? 2u : D == 32 ? 4u : 6u;  // swizzle code of [*, D] tiles
    static constexpr int OFF_K = 0;
    static constexpr int OFF_VL = TILE;
    static constexpr int OFF_VH = 2 * TILE;
    static constexpr int OFF_STAGE = 3 * TILE;     // stage s: Q, dO_lo, dO_hi at +s*3*TILE
    static constexpr int STAGE = 3 * TILE;
    static constexpr int OFF_PT = 9 * TILE;        // P^T  [128 keys][128 queries] bf16, 2 x 16 KB blocks
    static constexpr int OFF_DST = OFF_PT + 32768; // dS^T same layout
    static constexpr int OFF_L2 = OFF_DST + 32768; // 2 stages x 128 fp32: LSE * log2(e)
    static constexpr int OFF_DD = OFF_L2 + 1024;   // 2 stages x 128 fp32: D
    static constexpr int OFF_BAR = OFF_DD + 1024;  // 16 mbarriers
    static constexpr int OFF_MISC = OFF_BAR + 128;
    static constexpr int USED = OFF_MISC + 64;
    // + 1 KB for aligning the dynamic smem base to 1024; at least 116 KB so
    // that one CTA owns an SM (its TMEM allocation is all 512 columns)
    static constexpr int SMEM = (USED + 1024) > 118784 ? (USED + 1024) : 118784;
    // TMEM columns (fp32): S^T, dP^T, dV_lo, dV_hi, dK, dQ
    static constexpr uint32_t C_S = 0, C_DP = 128, C_DVL = 256, C_DVH = 256 + D, C_DK = 256 + 2 * D,
                              C_DQ = 256 + 3 * D;
    static constexpr uint32_t TMEM_COLS = 512;
};

enum Bar { B_KV = 0, B_QF0 = 1, B_QE0 = 3, B_SF = 5, B_PF = 6, B_DQF = 7, B_DQE = 8, B_ACC = 9 };

struct Sync {
    uint32_t bar0;
    volatile int* abort;
    __device__ uint32_t bar(int i) const { return bar0 + 8u * i; }
};

// Bounded wait on a barrier phase, by one thread.  Returns false on timeout or
// when another thread of the CTA has already aborted.
__device__ __noinline__ bool wait_bounded(const Sync& s, uint32_t bar, uint32_t parity, int role, int tile) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15) == 15) {
            if (*s.abort) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kTimeoutNs) {
                *s.abort = 1;
                atomicCAS(&g_tc_error, 0, ((1 + role) << 24) | (tile & 0xFFFFFF));
                return false;
            }
        }
    }
}

// Whole-warp wait: every lane waits, the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(const Sync& s, uint32_t bar, uint32_t parity, int role, int tile) {
    const bool ok = wait_bounded(s, bar, parity, role, tile);
    return __all_sync(0xffffffffu, ok);
}

// Wait without the abort short-cut (used only to drain copies after an abort).
__device__ bool wait_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kTimeoutNs) return false;
    return true;
}

template <int D>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, uint32_t* v) {
    if constexpr (D == 16) {
        tmem_ld_32x32b_x16(taddr, v);
    } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + 32 * c, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[32 * c + e] = r[e];
        }
    }
}

// ---------------------------------------------------------------- main kernel
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
bwd_main_kernel(const __grid_constant__ CUtensorMap tm_packed, const __grid_constant__ CUtensorMap tm_do_lo,
                const __grid_constant__ CUtensorMap tm_do_hi, const float* __restrict__ lse,
                const float* __restrict__ Drow, float* __restrict__ dq_acc, bf16* __restrict__ d_packed, int N,
                int nkt, int nqt, float scale, float scale_log2) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    Sync sy{sb + C::OFF_BAR, reinterpret_cast<volatile int*>(smem + C::OFF_MISC)};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x / nkt, kt = blockIdx.x % nkt;
    const int k0 = kt * C::BM;

    if (threadIdx.x == 0) {
        mbar_init(sy.bar(B_KV), 1);
        mbar_init(sy.bar(B_QF0), 32);
        mbar_init(sy.bar(B_QF0 + 1), 32);
        mbar_init(sy.bar(B_QE0), 1);
        mbar_init(sy.bar(B_QE0 + 1), 1);
        mbar_init(sy.bar(B_SF), 1);
        mbar_init(sy.bar(B_PF), 128);
        mbar_init(sy.bar(B_DQF), 1);
        mbar_init(sy.bar(B_DQE), 128);
        mbar_init(sy.bar(B_ACC), 1);
        *sy.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_packed);
        tma_prefetch_desc(&tm_do_lo);
        tma_prefetch_desc(&tm_do_hi);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // issued-copy bookkeeping for the abort drain (producer lane 0 only)
    int last_issued[2] = {-1, -1};

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            mbar_arrive_expect_tx(sy.bar(B_KV), 3 * C::TILE);
            tma_load_3d(sb + C::OFF_K, &tm_packed, 0, k0, bh * 4 + 1, sy.bar(B_KV));
            tma_load_3d(sb + C::OFF_VL, &tm_packed, 0, k0, bh * 4 + 2, sy.bar(B_KV));
            tma_load_3d(sb + C::OFF_VH, &tm_packed, 0, k0, bh * 4 + 3, sy.bar(B_KV));
        }
        float* L2s = reinterpret_cast<float*>(smem + C::OFF_L2);
        float* Ds = reinterpret_cast<float*>(smem + C::OFF_DD);
        for (int t = 0; t < nqt; ++t) {
            const int s = t & 1;
            if (!warp_wait(sy, sy.bar(B_QE0 + s), ((t >> 1) & 1) ^ 1, 0, t)) break;
            if (lane == 0) {
                const uint32_t st = sb + C::OFF_STAGE + s * C::STAGE;
                mbar_expect_tx(sy.bar(B_QF0 + s), 3 * C::TILE);
                tma_load_3d(st, &tm_packed, 0, t * C::BQ, bh * 4 + 0, sy.bar(B_QF0 + s));
                tma_load_3d(st + C::TILE, &tm_do_lo, 0, t * C::BQ, bh, sy.bar(B_QF0 + s));
                tma_load_3d(st + 2 * C::TILE, &tm_do_hi, 0, t * C::BQ, bh, sy.bar(B_QF0 + s));
                last_issued[s] = t;
            }
            // row statistics of the 128 queries: 4 per lane; padded rows get
            // LSE = +inf (so P = 0) and D = 0
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int q = lane * 4 + e;
                const int i = t * C::BQ + q;
                const bool v = i < N;
                L2s[s * 128 + q] = v ? lse[(size_t)bh * N + i] * kLog2e : INFINITY;
                Ds[s * 128 + q] = v ? Drow[(size_t)bh * N + i] : 0.f;
            }
            mbar_arrive(sy.bar(B_QF0 + s));
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(128, 128, 0, 0);   // S^T, dP^T
            constexpr uint32_t ID_KN = idesc_bf16(128, D, 0, 1);    // dV, dK: A K-major, B MN-major
            constexpr uint32_t ID_DQ = idesc_bf16(128, D, 1, 1);    // dQ: A, B MN-major
            const uint32_t sK = sb + C::OFF_K, sVL = sb + C::OFF_VL, sVH = sb + C::OFF_VH;
            const uint32_t sPT = sb + C::OFF_PT, sDST = sb + C::OFF_DST;
            auto issue_s_dp = [&](int s) {
                const uint32_t sQ = sb + C::OFF_STAGE + s * C::STAGE;
                const uint32_t sGL = sQ + C::TILE, sGH = sQ + 2 * C::TILE;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_ss(tmem + C::C_S, smem_desc(sK + 32 * kk, 16, 8 * C::ROWB, C::SW),
                                smem_desc(sQ + 32 * kk, 16, 8 * C::ROWB, C::SW), ID_S, kk > 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_ss(tmem + C::C_DP, smem_desc(sVL + 32 * kk, 16, 8 * C::ROWB, C::SW),
                                smem_desc(sGL + 32 * kk, 16, 8 * C::ROWB, C::SW), ID_S, kk > 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_ss(tmem + C::C_DP, smem_desc(sVH + 32 * kk, 16, 8 * C::ROWB, C::SW),
                                smem_desc(sGH + 32 * kk, 16, 8 * C::ROWB, C::SW), ID_S, 1);
            };
            bool ok = wait_bounded(sy, sy.bar(B_KV), 0, 1, -1) && wait_bounded(sy, sy.bar(B_QF0), 0, 1, 0);
            if (ok) {
                tc_fence_after();
                issue_s_dp(0);
                mma_commit(sy.bar(B_SF));
            }
            for (int t = 0; t < nqt && ok; ++t) {
                const int s = t & 1;
                ok = wait_bounded(sy, sy.bar(B_PF), t & 1, 1, t);
                if (ok && t > 0) ok = wait_bounded(sy, sy.bar(B_DQE), (t - 1) & 1, 1, t);
                if (!ok) break;
                tc_fence_after();
                const uint32_t sQ = sb + C::OFF_STAGE + s * C::STAGE;
                const uint32_t sGL = sQ + C::TILE, sGH = sQ + 2 * C::TILE;
#pragma unroll
                for (int kk = 0; kk < C::BQ / 16; ++kk) {
                    // A = P^T / dS^T (K-major, 2 blocks of 64 queries); B = [16 queries, D] rows (MN-major)
                    const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint32_t boff = kk * 16 * C::ROWB;
                    const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
                    mma_bf16_ss(tmem + C::C_DVL, smem_desc(sPT + aoff, 16, 1024, 2),
                                smem_desc(sGL + boff, 16, 8 * C::ROWB, C::SW), ID_KN, acc);
                    mma_bf16_ss(tmem + C::C_DVH, smem_desc(sPT + aoff, 16, 1024, 2),
                                smem_desc(sGH + boff, 16, 8 * C::ROWB, C::SW), ID_KN, acc);
                    mma_bf16_ss(tmem + C::C_DK, smem_desc(sDST + aoff, 16, 1024, 2),
                                smem_desc(sQ + boff, 16, 8 * C::ROWB, C::SW), ID_KN, acc);
                }
#pragma unroll
                for (int kk = 0; kk < C::BM / 16; ++kk) {
                    // A = dS (queries x keys): the dS^T buffer read MN-major, two 64-query atoms
                    // 16 KB apart; B = K_j rows kk*16.. (MN-major)
                    mma_bf16_ss(tmem + C::C_DQ, smem_desc(sDST + kk * 2048, 16384, 1024, 2),
                                smem_desc(sK + kk * 16 * C::ROWB, 16, 8 * C::ROWB, C::SW), ID_DQ, kk > 0);
                }
                mma_commit(sy.bar(B_QE0 + s));
                mma_commit(sy.bar(B_DQF));
                if (t + 1 < nqt) {
                    const int s1 = (t + 1) & 1;
                    ok = wait_bounded(sy, sy.bar(B_QF0 + s1), ((t + 1) >> 1) & 1, 1, t + 1);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s_dp(s1);
                    mma_commit(sy.bar(B_SF));
                }
            }
            if (ok) {
                mma_commit(sy.bar(B_ACC));
            } else {
                // aborted: let the MMAs already issued finish before TMEM is freed
                mma_commit(sy.bar(B_ACC));
                wait_drain(sy.bar(B_ACC), 0);
            }
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------------ softmax gradient
        const int q4 = warp & 3;                 // TMEM lane quarter of this warp
        const int jl = q4 * 32 + lane;           // key row within the tile
        const bool kvalid = k0 + jl < N;
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        const float* L2s = reinterpret_cast<const float*>(smem + C::OFF_L2);
        const float* Ds = reinterpret_cast<const float*>(smem + C::OFF_DD);
        const uint32_t pt_row = sb + C::OFF_PT + jl * 128;
        const uint32_t ds_row = sb + C::OFF_DST + jl * 128;
        bool ok = true;
        for (int t = 0; t < nqt; ++t) {
            const int s = t & 1;
            // S/dP of tile t in TMEM; the row statistics of stage s written
            ok = warp_wait(sy, sy.bar(B_SF), t & 1, 2, t) && warp_wait(sy, sy.bar(B_QF0 + s), (t >> 1) & 1, 2, t);
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < C::BQ / 32; ++c) {
                uint32_t sr[32], pr[32];
                tmem_ld_32x32b_x32(trow + C::C_S + 32 * c, sr);
                tmem_ld_32x32b_x32(trow + C::C_DP + 32 * c, pr);
                tmem_wait_ld();
                uint32_t pk[16], dk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 l4 = *reinterpret_cast<const float4*>(L2s + s * 128 + 32 * c + e);
                    const float4 d4 = *reinterpret_cast<const float4*>(Ds + s * 128 + 32 * c + e);
                    float p0 = exp2f(fmaf(__uint_as_float(sr[e + 0]), scale_log2, -l4.x));
                    float p1 = exp2f(fmaf(__uint_as_float(sr[e + 1]), scale_log2, -l4.y));
                    float p2 = exp2f(fmaf(__uint_as_float(sr[e + 2]), scale_log2, -l4.z));
                    float p3 = exp2f(fmaf(__uint_as_float(sr[e + 3]), scale_log2, -l4.w));
                    if (!kvalid) p0 = p1 = p2 = p3 = 0.f;
                    const float g0 = p0 * (__uint_as_float(pr[e + 0]) - d4.x);
                    const float g1 = p1 * (__uint_as_float(pr[e + 1]) - d4.y);
                    const float g2 = p2 * (__uint_as_float(pr[e + 2]) - d4.z);
                    const float g3 = p3 * (__uint_as_float(pr[e + 3]) - d4.w);
                    pk[e / 2] = pack_bf16x2(p0, p1);
                    pk[e / 2 + 1] = pack_bf16x2(p2, p3);
                    dk[e / 2] = pack_bf16x2(g0, g1);
                    dk[e / 2 + 1] = pack_bf16x2(g2, g3);
                }
                // 32 queries = four 16-byte chunks of row jl; 128B-swizzled position
                const uint32_t blk = (c >> 1) * 16384;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t ch = (uint32_t)(((c & 1) * 4 + u) ^ (jl & 7)) << 4;
                    st_shared_v4(pt_row + blk + ch, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                    st_shared_v4(ds_row + blk + ch, dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            mbar_arrive(sy.bar(B_PF));
        }
        // epilogue: dV_lo, dV_hi, dK rows of this thread's key
        if (ok) ok = warp_wait(sy, sy.bar(B_ACC), 0, 2, nqt);
        if (ok) {
            tc_fence_after();
            uint32_t v[D];
            const size_t sec = (size_t)N * D;
            bf16* out = d_packed + (size_t)bh * 4 * sec + (size_t)(k0 + jl) * D;
#pragma unroll
            for (int which = 0; which < 3; ++which) {
                const uint32_t col = which == 0 ? C::C_DK : which == 1 ? C::C_DVL : C::C_DVH;
                const float mul = which == 0 ? scale : 1.f;
                tmem_ld_row<D>(trow + col, v);
                tmem_wait_ld();
                if (kvalid) {
                    bf16* o = out + (size_t)(1 + which) * sec;
#pragma unroll
                    for (int e = 0; e < D; e += 8) {
                        uint4 u;
                        u.x = pack_bf16x2(__uint_as_float(v[e + 0]) * mul, __uint_as_float(v[e + 1]) * mul);
                        u.y = pack_bf16x2(__uint_as_float(v[e + 2]) * mul, __uint_as_float(v[e + 3]) * mul);
                        u.z = pack_bf16x2(__uint_as_float(v[e + 4]) * mul, __uint_as_float(v[e + 5]) * mul);
                        u.w = pack_bf16x2(__uint_as_float(v[e + 6]) * mul, __uint_as_float(v[e + 7]) * mul);
                        *reinterpret_cast<uint4*>(o + e) = u;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ dQ drain
        const int q4 = warp & 3;
        const int il = q4 * 32 + lane;           // query row within the tile
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        for (int t = 0; t < nqt; ++t) {
            if (!warp_wait(sy, sy.bar(B_DQF), t & 1, 3, t)) break;
            tc_fence_after();
            uint32_t v[D];
            tmem_ld_row<D>(trow + C::C_DQ, v);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(sy.bar(B_DQE));
            const int i = t * C::BQ + il;
            if (i < N) {
                float4* dst = reinterpret_cast<float4*>(dq_acc + ((size_t)bh * N + i) * D);
#pragma unroll
                for (int e = 0; e < D; e += 4)
                    atomicAdd(dst + e / 4, make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                                                       __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])));
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (*sy.abort && warp == 0 && lane == 0) {
        // let this CTA's own copies land before its shared memory is released
        wait_drain(sy.bar(B_KV), 0);
        for (int s = 0; s < 2; ++s)
            if (last_issued[s] >= 0) wait_drain(sy.bar(B_QF0 + s), (last_issued[s] >> 1) & 1);
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---------------------------------------------------------------- D and dQ-accumulator reset
template <int D>
__global__ void __launch_bounds__(256)
pre_kernel(const bf16* __restrict__ o_lo, const bf16* __restrict__ o_hi, const bf16* __restrict__ do_lo,
           const bf16* __restrict__ do_hi, float* __restrict__ Drow, float* __restrict__ dq_acc, long long rows) {
    constexpr int TPR = D / 8;                // threads per row, 8 bf16 (16 B) each
    constexpr int RPB = 256 / TPR;
    const long long row = (long long)blockIdx.x * RPB + threadIdx.x / TPR;
    const int part = threadIdx.x % TPR;
    float acc = 0.f;
    if (row < rows) {
        const size_t off = (size_t)row * D + part * 8;
        const uint4 a = *reinterpret_cast<const uint4*>(o_lo + off);
        const uint4 b = *reinterpret_cast<const uint4*>(do_lo + off);
        const uint4 c = *reinterpret_cast<const uint4*>(o_hi + off);
        const uint4 d = *reinterpret_cast<const uint4*>(do_hi + off);
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
        const __nv_bfloat162* pc = reinterpret_cast<const __nv_bfloat162*>(&c);
        const __nv_bfloat162* pd = reinterpret_cast<const __nv_bfloat162*>(&d);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 fa = __bfloat1622float2(pa[k]), fb = __bfloat1622float2(pb[k]);
            const float2 fc = __bfloat1622float2(pc[k]), fd = __bfloat1622float2(pd[k]);
            acc = fmaf(fa.x, fb.x, acc);
            acc = fmaf(fa.y, fb.y, acc);
            acc = fmaf(fc.x, fd.x, acc);
            acc = fmaf(fc.y, fd.y, acc);
        }
        float4* z = reinterpret_cast<float4*>(dq_acc + (size_t)row * D);
#pragma unroll
        for (int k = part; k < D / 4; k += TPR) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, TPR);
    if (row < rows && part == 0) Drow[row] = acc;
}

// ---------------------------------------------------------------- dQ = scale * acc -> bf16
template <int D>
__global__ void __launch_bounds__(256)
dq_finalize_kernel(const float* __restrict__ dq_acc, bf16* __restrict__ d_packed, long long rows, int N,
                   float scale) {
    constexpr int PPR = D / 8;  // 8-element parts per row
    const long long idx = (long long)blockIdx.x * 256 + threadIdx.x;
    if (idx >= rows * PPR) return;
    const long long row = idx / PPR;
    const int part = (int)(idx % PPR);
    const long long bh = row / N, i = row % N;
    const float4* src = reinterpret_cast<const float4*>(dq_acc + (size_t)row * D + part * 8);
    const float4 a = src[0], b = src[1];
    uint4 u;
    u.x = pack_bf16x2(a.x * scale, a.y * scale);
    u.y = pack_bf16x2(a.z * scale, a.w * scale);
    u.z = pack_bf16x2(b.x * scale, b.y * scale);
    u.w = pack_bf16x2(b.z * scale, b.w * scale);
    *reinterpret_cast<uint4*>(d_packed + ((size_t)bh * 4 * N + i) * D + part * 8) = u;
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode(std::string* err) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    static cudaError_t st = cudaSuccess;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        st = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (st == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!fn) *err = std::string("cuTensorMapEncodeTiled unavailable: ") + cudaGetErrorString(st);
    return fn;
}

// 3-D map over a [Z, N, D] bf16 tensor, box [1, 128, D], swizzle matching D.
bool encode_3d(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* base, int D, int N, long long Z,
               std::string* err) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)Z};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
    const cuuint32_t box[3] = {(cuuint32_t)D, 128u, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUtensorMapSwizzle sw = D == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : D == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_32B;
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")";
        return false;
    }
    return true;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

template <int D>
int launch(const BwdArgs& a, std::string* err) {
    using C = Cfg<D>;
    auto enc = get_encode(err);
    if (!enc) return PSA_ERR_CUDA;
    CUtensorMap tm_packed, tm_lo, tm_hi;
    if (!encode_3d(enc, &tm_packed, a.packed, D, a.N, a.BH * 4, err) ||
        !encode_3d(enc, &tm_lo, a.do_lo, D, a.N, a.BH, err) || !encode_3d(enc, &tm_hi, a.do_hi, D, a.N, a.BH, err))
        return PSA_ERR_CUDA;
    static std::once_flag attr_once;
    static cudaError_t attr_st = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_st = cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    });
    if (attr_st != cudaSuccess) {
        *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(attr_st);
        return PSA_ERR_CUDA;
    }
    const long long rows = a.BH * a.N;
    float* Drow = static_cast<float*>(a.workspace);
    float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + align256((size_t)rows * 4));
    const int nkt = (a.N + C::BM - 1) / C::BM;
    const int nqt = (a.N + C::BQ - 1) / C::BQ;
    const long long grid = a.BH * nkt;
    const long long pre_grid = (rows + 256 / (D / 8) - 1) / (256 / (D / 8));
    const long long fin_grid = (rows * (D / 8) + 255) / 256;
    if (grid > 0x7fffffffll || pre_grid > 0x7fffffffll || fin_grid > 0x7fffffffll) {
        *err = "grid too large";
        return PSA_ERR_UNSUPPORTED;
    }
    const bf16* o_lo = static_cast<const bf16*>(a.o_lo);
    const bf16* o_hi = static_cast<const bf16*>(a.o_hi);
    const bf16* do_lo = static_cast<const bf16*>(a.do_lo);
    const bf16* do_hi = static_cast<const bf16*>(a.do_hi);
    bf16* dp = static_cast<bf16*>(a.d_packed);
    {
        ProfScope prof(kSlotPre, a.stream);
        pre_kernel<D><<<(unsigned)pre_grid, 256, 0, a.stream>>>(o_lo, o_hi, do_lo, do_hi, Drow, dq_acc, rows);
    }
    {
        ProfScope prof(kSlotMain, a.stream);
        bwd_main_kernel<D><<<(unsigned)grid, kThreads, C::SMEM, a.stream>>>(
            tm_packed, tm_lo, tm_hi, a.lse, Drow, dq_acc, dp, a.N, nkt, nqt, a.scale, a.scale * kLog2e);
    }
    {
        ProfScope prof(kSlotDq, a.stream);
        dq_finalize_kernel<D><<<(unsigned)fin_grid, 256, 0, a.stream>>>(dq_acc, dp, rows, a.N, a.scale);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = std::string("tensor-core backward launch: ") + cudaGetErrorString(e);
        return PSA_ERR_CUDA;
    }
    return PSA_OK;
}

}  // namespace

bool tc_supported(int dtype, int d) { return dtype == PSA_BF16 && (d == 16 || d == 32 || d == 64); }

size_t tc_workspace_bytes(long long BH, int N, int d) {
    const size_t rows = (size_t)BH * (size_t)N;
    return align256(rows * 4) + rows * (size_t)d * 4;
}

int tc_bwd_launch(const BwdArgs& a, std::string* err) {
    switch (a.d) {
        case 16: return launch<16>(a, err);
        case 32: return launch<32>(a, err);
        case 64: return launch<64>(a, err);
        default: *err = "unsupported head_dim"; return PSA_ERR_UNSUPPORTED;
    }
}

int tc_take_device_error(std::string* err) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(int));
    if (e != cudaSuccess || v == 0) return 0;
    const int zero = 0;
    cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(int));
    static const char* roles[] = {"?", "producer", "mma", "softmax", "dq"};
    const int role = (v >> 24) & 0xff;
    *err = std::string("tensor-core backward: a bounded wait gave up (") + roles[role < 5 ? role : 0] +
           " warp, query tile " + std::to_string(v & 0xFFFFFF) + ")";
    return 1;
}

}  // namespace psa
