// tc_pair.cu -- two-pass tensor-core backward of PSA attention on SM pairs
// (bf16, head_dim 32 or 64).
//
// "Struct PsaFa2Backward" (description): key-row gradients come from a sweep
// over the queries, query-row gradients from a sweep over the keys.  Both
// sweeps here run
// on clusters of two CTAs whose tcgen05.mma instructions span the pair
// (cta_group::2, M = 256).  Each SM still does its own 128 rows of every
// instruction at the single-SM rate; what the pair halves is the number of
// instructions, commits and barrier waits one issuing thread goes through,
// which with d = 32 or 64 (every MMA has N <= 128) is where the time goes.
//
// Pass 1 (key-outer, bwd_kv_pair_kernel): the pair owns 256 keys (128 per CTA)
// and walks over the queries in 64-query sub-tiles u:
//   S^T  = K Q_u^T - 1 (LSE/scale)^T     (M = 256 keys, N = 64 queries, K = d)
//   dP^T = V_lo dO_lo,u^T + V_hi dO_hi,u^T - 1 D^T                (K = 2d)
//   P^T  = exp2(S^T scale log2e),  dS^T = P^T o dP^T
//   [dV_lo | dV_hi] += P^T [dO_lo,u | dO_hi,u]   (A = P^T from TMEM, N = 2d)
//   dK += dS^T Q_u                               (A = dS^T from TMEM, N = d)
// Pass 2 (query-outer, bwd_q_pair_kernel): the pair owns 256 queries and walks
// over the keys in 64-key sub-tiles v:
//   S = Q K_v^T,  dP = dO_lo V_lo,v^T + dO_hi V_hi,v^T,  dS = P o (dP - D)
//   dQ += dS K_v                                 (A = dS from TMEM, N = d)
// Every output element is summed in one fixed order: no atomics, results are
// reproducible bit for bit.  In pass 1 the per-query statistics enter through
// one extra K-step of 16 in each of the S^T and dP^T products: A is a constant
// tile whose columns 0 and 1 are ones, B holds -LSE/scale (resp. -D) split
// into two bf16 terms (high part and rounded remainder, 16 significant bits),
// so the softmax warps read no per-query values from shared memory.
//
// Operand placement for a pair instruction: A rows come from each CTA's own
// shared memory or TMEM (its 128 rows); B is split along N, columns [0, N/2)
// from CTA 0 and [N/2, N) from CTA 1, at the same shared-memory offset.  So
// for S^T CTA r loads queries [32r, 32r + 32) of the sub-tile, for dV it
// loads dO_lo (r = 0) or dO_hi (r = 1), for dK it loads feature columns
// [r d/2, (r + 1) d/2) of Q; pass 2 splits K and V the same way.
//
// Warp roles (352 threads per CTA): warp 0 TMA producer; warps 1 and 10 the
// MMA issuers (in CTA 0 only; both CTAs' warp 1 allocate TMEM); warps 2-9 two
// softmax-gradient warpgroups taking alternate sub-tiles, one TMEM lane (key
// row in pass 1, query row in pass 2) per thread.  Two threads issue MMAs:
// warp 10 the S/dP products, warp 1 the accumulating products.  A thread that
// waits on a barrier first waits for its own MMAs in flight, so with one
// issuer the tensor pipe would drain at every wait; with two, each one's
// waits are covered by the other's MMAs.  The softmax warps of both CTAs
// arrive on CTA 0's barrier before the issuer consumes a sub-tile;
// tcgen05.commit multicasts completion to both CTAs.  Every wait is bounded
// (tc_sync.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>
#include <string>

#include "common.cuh"
#include "psa_attn.h"
#include "psa_internal.h"
#include "tc_ptx.cuh"
#include "tc_sync.cuh"
#include "tc_tmap.h"

namespace psa {
namespace {

using namespace psa::tc;
using bf16 = __nv_bfloat16;

__device__ int g_pair_error = 0;  // (1 + role) << 24 | tile of the first wait that gave up

constexpr int kPairThreads = 352;

// Shared-memory and TMEM layout common to both passes.  "Stationary" tiles
// are [128, D] (A operands); a stage holds one 64-row sub-tile's B operands.
template <int D>
struct PairCfg {
    static constexpr int ROWB = 2 * D;                 // bytes per [*, D] bf16 row
    static constexpr int TILE = 128 * ROWB;            // [128, D]
    static constexpr int HALF = 32 * ROWB;             // [32, D]: a pair's B half, K-major
    static constexpr int FULL64 = 64 * ROWB;           // [64, D]
    static constexpr int HCOL = 64 * D;                // [64, D/2]: feature half, MN-major
    static constexpr uint32_t SW = D == 64 ? 2u : 4u;  // swizzle of [*, D] tiles (128B / 64B)
    static constexpr uint32_t SWH = D == 64 ? 4u : 6u; // swizzle of [*, D/2] tiles (64B / 32B)
    static constexpr int NB = D == 64 ? 2 : 3;         // S/dP buffers in TMEM
    static constexpr uint32_t C_ACC = 128 * NB;        // first accumulator column
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(HALF % 1024 == 0 && HCOL % 1024 == 0, "stage pieces stay on 1 KB boundaries");
};

// pass 1 layout
template <int D>
struct KvCfg : PairCfg<D> {
    using P = PairCfg<D>;
    static constexpr int NST = D == 64 ? 4 : 6;        // Q/dO stages (> NB)
    // stage: Q half (S^T) | dO_lo half | dO_hi half (dP^T) | dO_r (dV) | Q feature half (dK) |
    // statistics columns of S^T and of dP^T ([32 queries, 16] each, 32-byte swizzle)
    static constexpr int S_Q = 0, S_GL = P::HALF, S_GH = 2 * P::HALF, S_GV = 3 * P::HALF;
    static constexpr int S_QK = S_GV + P::FULL64;
    static constexpr int S_LX = S_QK + P::HCOL, S_DX = S_LX + 1024;
    static constexpr int STAGE = S_DX + 1024;
    static constexpr int TMA_BYTES = S_LX;                  // the stage's bytes that TMA writes
    static constexpr int OFF_K = 0, OFF_VL = P::TILE, OFF_VH = 2 * P::TILE;
    static constexpr int OFF_ONES = 3 * P::TILE;             // [128, 16] bf16: columns 0, 1 = 1
    static constexpr int OFF_STAGE = OFF_ONES + 4096;
    static constexpr int OFF_BAR = OFF_STAGE + NST * STAGE;
    static constexpr int OFF_MISC = OFF_BAR + 256;
    static constexpr int USED = OFF_MISC + 64;
    static constexpr int SMEM = (USED + 1024) > 118784 ? (USED + 1024) : 118784;  // one CTA per SM
    static constexpr uint32_t C_DV = P::C_ACC, C_DK = C_DV + 2 * D;
    static_assert(C_DK + D <= P::TMEM_COLS, "TMEM budget");
    static_assert(NST > P::NB, "the stage of u+NB must differ from u's");
    static_assert(USED + 1024 <= 232448, "shared memory budget");
};

// pass 2 layout
template <int D>
struct QCfg : PairCfg<D> {
    using P = PairCfg<D>;
    static constexpr int NST = 6;                      // K/V stages (> NB)
    // stage: K half (S) | V_lo half | V_hi half (dP) | K feature half (dQ)
    static constexpr int S_K = 0, S_VL = P::HALF, S_VH = 2 * P::HALF, S_KH = 3 * P::HALF;
    static constexpr int STAGE = S_KH + P::HCOL;
    static constexpr int OFF_Q = 0, OFF_GL = P::TILE, OFF_GH = 2 * P::TILE, OFF_STAGE = 3 * P::TILE;
    static constexpr int OFF_BAR = OFF_STAGE + NST * STAGE;
    static constexpr int OFF_MISC = OFF_BAR + 256;
    static constexpr int USED = OFF_MISC + 64;
    static constexpr int SMEM = (USED + 1024) > 118784 ? (USED + 1024) : 118784;
    static constexpr uint32_t C_DQ = P::C_ACC;
    static_assert(C_DQ + D <= P::TMEM_COLS, "TMEM budget");
    static_assert(NST > P::NB, "the stage of v+NB must differ from v's");
    static_assert(USED + 1024 <= 232448, "shared memory budget");
};

// barriers (same indices in both passes): stationary tiles loaded, S/dP ready
// (per buffer), softmax done (a ring of 4 over the sub-tiles, CTA 0 only, 256
// arrivals: one warpgroup of each CTA), accumulators final, pair ready (CTA 0
// only: both CTAs' first stages loaded), stage full / empty
enum { P_IN = 0, P_SF = 1, P_PF = 4, P_ACC = 8, P_RDY = 9, P_FULL = 10, P_EMPTY = 16, P_DRAIN = 22 };
static_assert(P_FULL + 6 <= P_EMPTY && P_EMPTY + 6 <= P_DRAIN && P_DRAIN < 32, "barrier indices");
// The softmax-done barriers form a ring of 4 (sub-tile u uses P_PF + u % 4).  A
// warp can start sub-tile u only after S/dP(u) was issued, which waited for
// dV/dK(u - NB), which waited for every softmax warp of sub-tile u - NB; with
// NB <= 3 no warp is ever 4 sub-tiles ahead of another, so a barrier never
// receives arrivals for two of its phases at once (with a ring of 2, a warp
// two sub-tiles ahead of a slow one would complete the slow one's phase).
constexpr int kPfRing = 4;

__device__ __forceinline__ bool warp_wait_cluster(const Sync& s, uint32_t bar, uint32_t parity, int role, int tile) {
    const bool ok = wait_bounded_cluster(s, bar, parity, role, tile);
    return __all_sync(0xffffffffu, ok);
}

// P and dS of one 32-column chunk of pass 1 (columns are queries), packed to
// bf16 pairs.  S^T and dP^T arrive with -LSE/scale and -D already added, so
// P = exp2(S^T scale log2e) and dS = P dP^T; keys past N get P = 0.
__device__ __forceinline__ void pair_softmax_chunk(const uint32_t (&sr)[32], const uint32_t (&pr)[32],
                                                   float scale_log2, float kmask, uint32_t (&pk)[16],
                                                   uint32_t (&dk)[16]) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        const float p0 = kmask * ex2_approx(__uint_as_float(sr[e]) * scale_log2);
        const float p1 = kmask * ex2_approx(__uint_as_float(sr[e + 1]) * scale_log2);
        pk[e / 2] = pack_bf16x2(p0, p1);
        dk[e / 2] = pack_bf16x2(p0 * __uint_as_float(pr[e]), p1 * __uint_as_float(pr[e + 1]));
    }
}

// Byte offset of element (row, col), col < 16, in a [rows, 16] bf16 tile with
// 32-byte rows and the 32-byte swizzle (16-byte chunk index ^= row bit 2).
__device__ __forceinline__ uint32_t sw32_offset(int row, int col) {
    return (uint32_t)(32 * row) + ((uint32_t)(col * 2) ^ ((uint32_t)((row >> 2) & 1) << 4));
}

// v as two bf16 terms, high part and rounded remainder, packed as a pair.
__device__ __forceinline__ uint32_t split_bf16x2(float v) {
    const float hi = __bfloat162float(__float2bfloat16_rn(v));
    return pack_bf16x2(hi, v - hi);
}

// Stores one thread's row of an fp32 TMEM accumulator (D columns) times `mul`
// as bf16 (whole warp loads; only `valid` rows are stored).
template <int D>
__device__ __forceinline__ void store_row(uint32_t taddr, float mul, bool valid, bf16* out) {
    uint32_t v[D];
    tmem_ld_row<D>(taddr, v);
    tmem_wait_ld();
    if (valid) {
#pragma unroll
        for (int e = 0; e < D; e += 8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[e + 0]) * mul, __uint_as_float(v[e + 1]) * mul);
            w.y = pack_bf16x2(__uint_as_float(v[e + 2]) * mul, __uint_as_float(v[e + 3]) * mul);
            w.z = pack_bf16x2(__uint_as_float(v[e + 4]) * mul, __uint_as_float(v[e + 5]) * mul);
            w.w = pack_bf16x2(__uint_as_float(v[e + 6]) * mul, __uint_as_float(v[e + 7]) * mul);
            *reinterpret_cast<uint4*>(out + e) = w;
        }
    }
}

// Collective set-up of a pair CTA: barriers, TMEM (both CTAs' warp 1), and a
// cluster barrier so that the peer's barriers exist before anything arrives.
__device__ __forceinline__ uint32_t pair_setup(const Sync& sy, uint32_t* tmem_slot, int warp, int nst, int nb) {
    if (threadIdx.x == 0) {
        mbar_init(sy.bar(P_IN), 1);
        for (int b = 0; b < nb; ++b) mbar_init(sy.bar(P_SF + b), 1);
        for (int x = 0; x < kPfRing; ++x) mbar_init(sy.bar(P_PF + x), 256);
        mbar_init(sy.bar(P_ACC), 1);
        mbar_init(sy.bar(P_RDY), 2);
        mbar_init(sy.bar(P_DRAIN), 1);
        for (int s = 0; s < nst; ++s) {
            mbar_init(sy.bar(P_FULL + s), 32);
            mbar_init(sy.bar(P_EMPTY + s), 1);
        }
        *sy.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    return *tmem_slot;
}

__device__ __forceinline__ void pair_teardown(uint32_t tmem, int warp) {
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

// ---------------------------------------------------------------- pass 1: dK, dV
template <int D>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
bwd_kv_pair_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_q32,
                   const __grid_constant__ CUtensorMap tm_lo32, const __grid_constant__ CUtensorMap tm_hi32,
                   const __grid_constant__ CUtensorMap tm_lo64, const __grid_constant__ CUtensorMap tm_hi64,
                   const __grid_constant__ CUtensorMap tm_qh, const float* __restrict__ lse,
                   const float* __restrict__ Drow, bf16* __restrict__ d_packed, int N, int npair, float scale,
                   float scale_log2) {
    using C = KvCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    Sync sy{sb + C::OFF_BAR, reinterpret_cast<volatile int*>(smem + C::OFF_MISC), &g_pair_error};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = (int)cluster_ctarank();
    const int pair = blockIdx.x >> 1;
    const int bh = pair / npair;
    const int k0 = (pair % npair) * 256 + 128 * r;     // this CTA's first key
    const int nsub = (N + 63) / 64;
    const int nready = nsub < C::NB ? nsub : C::NB;

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tm_kv);
        tma_prefetch_desc(&tm_q32);
        tma_prefetch_desc(&tm_lo32);
        tma_prefetch_desc(&tm_hi32);
        tma_prefetch_desc(r ? &tm_hi64 : &tm_lo64);
        tma_prefetch_desc(&tm_qh);
    }
    // the constant A tile of the statistics K-step and zeroed statistics
    // tiles (only their columns 0 and 1 are rewritten per sub-tile)
    for (int x = threadIdx.x; x < 4096 / 16; x += kPairThreads) {
        const int row = x >> 1, chunk = x & 1;
        const uint32_t one2 = 0x3F803F80u;  // bf16 pair (1, 1)
        const bool has = chunk == ((row >> 2) & 1);  // the physical chunk holding columns 0-7
        st_shared_v4(sb + C::OFF_ONES + 16 * x, has ? one2 : 0u, 0u, 0u, 0u);
    }
    for (int x = threadIdx.x; x < C::NST * 128; x += kPairThreads) {
        const int st = x >> 7, piece = x & 127;
        st_shared_v4(sb + C::OFF_STAGE + st * C::STAGE + C::S_LX + 16 * piece, 0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    const uint32_t tmem = pair_setup(sy, tmem_slot, warp, C::NST, C::NB);

    if (warp == 0) {
        // ------------------------------------------------------------ producer (own shared memory)
        int last[C::NST];
#pragma unroll
        for (int s = 0; s < C::NST; ++s) last[s] = -1;
        if (lane == 0) {
            mbar_arrive_expect_tx(sy.bar(P_IN), 3 * C::TILE);
            tma_load_3d(sb + C::OFF_K, &tm_kv, 0, k0, bh * 4 + 1, sy.bar(P_IN));
            tma_load_3d(sb + C::OFF_VL, &tm_kv, 0, k0, bh * 4 + 2, sy.bar(P_IN));
            tma_load_3d(sb + C::OFF_VH, &tm_kv, 0, k0, bh * 4 + 3, sy.bar(P_IN));
        }
        const CUtensorMap* tm_g = r ? &tm_hi64 : &tm_lo64;
        const float inv_scale = 1.f / scale;
        // a padded query's shift: -29952 (bf16) times the sign of the scale, so
        // that (S + shift) * scale * log2(e) is hugely negative and P = 0
        const uint32_t pad_shift = scale > 0.f ? 0x0000C6EAu : 0x000046EAu;
        bool ok = true;
        int s = 0, ph = 0;
        for (int u = 0; u < nsub; ++u) {
            if (!warp_wait_cluster(sy, sy.bar(P_EMPTY + s), ph ^ 1, 0, u)) { ok = false; break; }
            if (lane == 0) {
                const uint32_t st = sb + C::OFF_STAGE + s * C::STAGE;
                const uint32_t fb = sy.bar(P_FULL + s);
                const int q = u * 64;
                mbar_expect_tx(fb, C::TMA_BYTES);
                tma_load_3d(st + C::S_Q, &tm_q32, 0, q + 32 * r, bh * 4 + 0, fb);
                tma_load_3d(st + C::S_GL, &tm_lo32, 0, q + 32 * r, bh, fb);
                tma_load_3d(st + C::S_GH, &tm_hi32, 0, q + 32 * r, bh, fb);
                tma_load_3d(st + C::S_GV, tm_g, 0, q, bh, fb);
                tma_load_3d(st + C::S_QK, &tm_qh, r * (D / 2), q, bh * 4 + 0, fb);
            }
#pragma unroll
            for (int x = 0; x < C::NST; ++x)
                if (x == s) last[x] = u;
            {
                // statistics columns of this CTA's 32 queries (one per lane): -LSE/scale
                // and -D as bf16 (high, remainder) pairs; a padded query gets a large
                // shift against the scale's sign (P = 0) and D = 0
                const int i = u * 64 + 32 * r + lane;
                const bool v = i < N;
                const uint32_t lx = v ? split_bf16x2(-lse[(size_t)bh * N + i] * inv_scale) : pad_shift;
                const uint32_t dx = v ? split_bf16x2(-Drow[(size_t)bh * N + i]) : 0u;
                const uint32_t st = sb + C::OFF_STAGE + s * C::STAGE;
                asm volatile("st.shared.b32 [%0], %1;" ::"r"(st + C::S_LX + sw32_offset(lane, 0)), "r"(lx) : "memory");
                asm volatile("st.shared.b32 [%0], %1;" ::"r"(st + C::S_DX + sw32_offset(lane, 0)), "r"(dx) : "memory");
                fence_proxy_async_smem();
            }
            mbar_arrive(sy.bar(P_FULL + s));
            if (u == nready - 1) {
                // this CTA's stationary tiles and first stages are in: tell CTA 0's issuer
                __syncwarp();
                if (lane == 0) {
                    bool rd = wait_bounded(sy, sy.bar(P_IN), 0, 0, -1);
                    for (int x = 0; x < nready && rd; ++x) rd = wait_bounded(sy, sy.bar(P_FULL + x), 0, 0, x);
                    if (rd) mbar_arrive_cluster(mapa_shared(sy.bar(P_RDY), 0));
                }
                __syncwarp();
            }
            if (++s == C::NST) { s = 0; ph ^= 1; }
        }
        __syncwarp();
        if ((!ok || *sy.abort) && lane == 0) {
            // let this CTA's own copies land before its shared memory is released
            wait_drain(sy.bar(P_IN), 0);
#pragma unroll
            for (int x = 0; x < C::NST; ++x)
                if (last[x] >= 0) wait_drain(sy.bar(P_FULL + x), (last[x] / C::NST) & 1);
        }
    } else if (warp == 1 || warp == 10) {
        // ------------------------------------------------------------ MMA issuers (CTA 0 issues for the pair)
        if (r == 0 && lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(256, 64, 0, 0);      // S^T, dP^T: 64 queries
            constexpr uint32_t ID_DV = idesc_bf16(256, 2 * D, 0, 1);  // [dV_lo | dV_hi]: B MN-major
            constexpr uint32_t ID_DK = idesc_bf16(256, D, 0, 1);      // dK: B MN-major
            constexpr uint32_t SBO = 8 * C::ROWB, SBOH = 8 * D;
            constexpr uint32_t STAGE_U = C::STAGE >> 4;
            constexpr uint32_t KSTEP = (16 * C::ROWB) >> 4, KSTEPH = (16 * D) >> 4;
            if (warp == 10) {
                // S^T(u), dP^T(u) into TMEM buffer u % NB, once both CTAs' stage u is
                // loaded and the buffer's previous sub-tile u-NB has been consumed:
                // the commit of dV/dK(u-NB) certifies both (dV/dK(u-NB) was issued
                // after both CTAs' softmax warps, which had waited for stage u)
                const uint64_t dK = smem_desc(sb + C::OFF_K, 16, SBO, C::SW);
                const uint64_t dVL = smem_desc(sb + C::OFF_VL, 16, SBO, C::SW);
                const uint64_t dVH = smem_desc(sb + C::OFF_VH, 16, SBO, C::SW);
                const uint64_t dQ0 = smem_desc(sb + C::OFF_STAGE + C::S_Q, 16, SBO, C::SW);
                const uint64_t dGL0 = smem_desc(sb + C::OFF_STAGE + C::S_GL, 16, SBO, C::SW);
                const uint64_t dGH0 = smem_desc(sb + C::OFF_STAGE + C::S_GH, 16, SBO, C::SW);
                const uint64_t dOnes = smem_desc(sb + C::OFF_ONES, 16, 256, 6);
                const uint64_t dLX0 = smem_desc(sb + C::OFF_STAGE + C::S_LX, 16, 256, 6);
                const uint64_t dDX0 = smem_desc(sb + C::OFF_STAGE + C::S_DX, 16, 256, 6);
                bool ok = wait_bounded_cluster(sy, sy.bar(P_RDY), 0, 1, -1);
                for (int u = 0; u < nsub && ok; ++u) {
                    if (u >= C::NB) {
                        const int w = u - C::NB;
                        ok = wait_bounded_cluster(sy, sy.bar(P_EMPTY + w % C::NST), (w / C::NST) & 1, 1, u);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const uint32_t so = STAGE_U * (u % C::NST);
                    const uint32_t tS = tmem + 128u * (u % C::NB), tDP = tS + 64;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) mma_pair_ss(tS, dK + 2 * kk, dQ0 + so + 2 * kk, ID_S, kk);
                    mma_pair_ss(tS, dOnes, dLX0 + so, ID_S, 1);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_pair_ss(tDP, dVL + 2 * kk, dGL0 + so + 2 * kk, ID_S, kk);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_pair_ss(tDP, dVH + 2 * kk, dGH0 + so + 2 * kk, ID_S, 1);
                    mma_pair_ss(tDP, dOnes, dDX0 + so, ID_S, 1);
                    mma_commit_pair(sy.bar(P_SF + u % C::NB));
                }
                // this thread's MMAs are done before TMEM is released
                mma_commit_pair(sy.bar(P_DRAIN));
                wait_drain(sy.bar(P_DRAIN), 0);
            } else {
                // dV/dK(u) once PF(u) certifies P^T(u), dS^T(u) written by both CTAs
                const uint64_t dGV0 = smem_desc(sb + C::OFF_STAGE + C::S_GV, 16, SBO, C::SW);
                const uint64_t dQK0 = smem_desc(sb + C::OFF_STAGE + C::S_QK, 16, SBOH, C::SWH);
                bool ok = true;
                for (int u = 0; u < nsub && ok; ++u) {
                    ok = wait_bounded_cluster(sy, sy.bar(P_PF + u % kPfRing), (u / kPfRing) & 1, 1, u);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t so = STAGE_U * (u % C::NST);
                    const uint32_t tP = tmem + 128u * (u % C::NB), tDS = tP + 64;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t acc = (u > 0 || kk > 0) ? 1u : 0u;
                        mma_pair_ts(tmem + C::C_DV, tP + 8 * kk, dGV0 + so + KSTEP * kk, ID_DV, acc);
                        mma_pair_ts(tmem + C::C_DK, tDS + 8 * kk, dQK0 + so + KSTEPH * kk, ID_DK, acc);
                    }
                    mma_commit_pair(sy.bar(P_EMPTY + u % C::NST));
                }
                mma_commit_pair(sy.bar(P_ACC));
                if (!ok) wait_drain(sy.bar(P_ACC), 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax-gradient warpgroups
        const int grp = (warp - 2) >> 2;
        const int q4 = warp & 3;
        const int jl = q4 * 32 + lane;
        const bool kvalid = k0 + jl < N;
        const float kmask = kvalid ? 1.f : 0.f;
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        const uint32_t pf0 = mapa_shared(sy.bar(P_PF), 0);
        bool ok = true;
        for (int u = grp; u < nsub; u += 2) {
            const int s = u % C::NST, buf = u % C::NB;
            ok = warp_wait_cluster(sy, sy.bar(P_SF + buf), (u / C::NB) & 1, 2, u) &&
                 warp_wait(sy, sy.bar(P_FULL + s), (u / C::NST) & 1, 2, u);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tS = trow + 128u * buf, tDP = tS + 64;
// both chunks unrolled: the second chunk's work can overlap the first's
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t sr[32], pr[32];
                tmem_ld_32x32b_x32(tS + 32 * c, sr);
                tmem_ld_32x32b_x32(tDP + 32 * c, pr);
                tmem_wait_ld();
                uint32_t pk[16], dk[16];
                pair_softmax_chunk(sr, pr, scale_log2, kmask, pk, dk);
                // P^T over the S^T columns, dS^T over the dP^T columns already read
                tmem_st_32x32b_x16(tS + 16 * c, pk);
                tmem_st_32x32b_x16(tDP + 16 * c, dk);
            }
            tmem_wait_st();
            tc_fence_before();
            // stand-in wait for the issuer: this CTA's stage of u+NB is loaded
            if (u + C::NB < nsub)
                ok = warp_wait(sy, sy.bar(P_FULL + (u + C::NB) % C::NST), ((u + C::NB) / C::NST) & 1, 2, u);
            mbar_arrive_cluster(pf0 + 8u * (u % kPfRing));
            if (!ok) break;
        }
        // epilogue (warpgroup 0): dK, dV_lo, dV_hi rows of this thread's key
        if (grp == 0) {
            if (ok) ok = warp_wait_cluster(sy, sy.bar(P_ACC), 0, 2, nsub);
            if (ok) {
                tc_fence_after();
                const size_t sec = (size_t)N * D;
                bf16* out = d_packed + (size_t)bh * 4 * sec + (size_t)(k0 + jl) * D;
                store_row<D>(trow + C::C_DK, scale, kvalid, out + sec);
                store_row<D>(trow + C::C_DV, 1.f, kvalid, out + 2 * sec);
                store_row<D>(trow + C::C_DV + D, 1.f, kvalid, out + 3 * sec);
            }
        }
    }
    pair_teardown(tmem, warp);
}

// ---------------------------------------------------------------- pass 2: dQ
template <int D>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
bwd_q_pair_kernel(const __grid_constant__ CUtensorMap tm_q128, const __grid_constant__ CUtensorMap tm_lo128,
                  const __grid_constant__ CUtensorMap tm_hi128, const __grid_constant__ CUtensorMap tm_k32,
                  const __grid_constant__ CUtensorMap tm_kh, const float* __restrict__ lse,
                  const float* __restrict__ Drow, bf16* __restrict__ d_packed, int N, int npair, float scale,
                  float scale_log2) {
    using C = QCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    Sync sy{sb + C::OFF_BAR, reinterpret_cast<volatile int*>(smem + C::OFF_MISC), &g_pair_error};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = (int)cluster_ctarank();
    const int pair = blockIdx.x >> 1;
    const int bh = pair / npair;
    const int q0 = (pair % npair) * 256 + 128 * r;     // this CTA's first query
    const int nsub = (N + 63) / 64;
    const int nready = nsub < C::NB ? nsub : C::NB;

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tm_q128);
        tma_prefetch_desc(&tm_lo128);
        tma_prefetch_desc(&tm_hi128);
        tma_prefetch_desc(&tm_k32);
        tma_prefetch_desc(&tm_kh);
    }
    const uint32_t tmem = pair_setup(sy, tmem_slot, warp, C::NST, C::NB);

    if (warp == 0) {
        // ------------------------------------------------------------ producer (own shared memory)
        int last[C::NST];
#pragma unroll
        for (int s = 0; s < C::NST; ++s) last[s] = -1;
        if (lane == 0) {
            mbar_arrive_expect_tx(sy.bar(P_IN), 3 * C::TILE);
            tma_load_3d(sb + C::OFF_Q, &tm_q128, 0, q0, bh * 4 + 0, sy.bar(P_IN));
            tma_load_3d(sb + C::OFF_GL, &tm_lo128, 0, q0, bh, sy.bar(P_IN));
            tma_load_3d(sb + C::OFF_GH, &tm_hi128, 0, q0, bh, sy.bar(P_IN));
        }
        bool ok = true;
        int s = 0, ph = 0;
        for (int v = 0; v < nsub; ++v) {
            if (!warp_wait_cluster(sy, sy.bar(P_EMPTY + s), ph ^ 1, 0, v)) { ok = false; break; }
            if (lane == 0) {
                const uint32_t st = sb + C::OFF_STAGE + s * C::STAGE;
                const uint32_t fb = sy.bar(P_FULL + s);
                const int k = v * 64;
                mbar_expect_tx(fb, C::STAGE);
                tma_load_3d(st + C::S_K, &tm_k32, 0, k + 32 * r, bh * 4 + 1, fb);
                tma_load_3d(st + C::S_VL, &tm_k32, 0, k + 32 * r, bh * 4 + 2, fb);
                tma_load_3d(st + C::S_VH, &tm_k32, 0, k + 32 * r, bh * 4 + 3, fb);
                tma_load_3d(st + C::S_KH, &tm_kh, r * (D / 2), k, bh * 4 + 1, fb);
            }
#pragma unroll
            for (int x = 0; x < C::NST; ++x)
                if (x == s) last[x] = v;
            mbar_arrive(sy.bar(P_FULL + s));
            if (v == nready - 1) {
                __syncwarp();
                if (lane == 0) {
                    bool rd = wait_bounded(sy, sy.bar(P_IN), 0, 0, -1);
                    for (int x = 0; x < nready && rd; ++x) rd = wait_bounded(sy, sy.bar(P_FULL + x), 0, 0, x);
                    if (rd) mbar_arrive_cluster(mapa_shared(sy.bar(P_RDY), 0));
                }
                __syncwarp();
            }
            if (++s == C::NST) { s = 0; ph ^= 1; }
        }
        __syncwarp();
        if ((!ok || *sy.abort) && lane == 0) {
            wait_drain(sy.bar(P_IN), 0);
#pragma unroll
            for (int x = 0; x < C::NST; ++x)
                if (last[x] >= 0) wait_drain(sy.bar(P_FULL + x), (last[x] / C::NST) & 1);
        }
    } else if (warp == 1 || warp == 10) {
        // ------------------------------------------------------------ MMA issuers (CTA 0 issues for the pair)
        if (r == 0 && lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(256, 64, 0, 0);   // S, dP: 64 keys
            constexpr uint32_t ID_Q = idesc_bf16(256, D, 0, 1);    // dQ: A = dS (TMEM), B = K MN-major
            constexpr uint32_t SBO = 8 * C::ROWB, SBOH = 8 * D;
            constexpr uint32_t STAGE_U = C::STAGE >> 4;
            constexpr uint32_t KSTEPH = (16 * D) >> 4;
            if (warp == 10) {
                // S(v), dP(v) into buffer v % NB (same conditions as in pass 1)
                const uint64_t dQ = smem_desc(sb + C::OFF_Q, 16, SBO, C::SW);
                const uint64_t dGL = smem_desc(sb + C::OFF_GL, 16, SBO, C::SW);
                const uint64_t dGH = smem_desc(sb + C::OFF_GH, 16, SBO, C::SW);
                const uint64_t dK0 = smem_desc(sb + C::OFF_STAGE + C::S_K, 16, SBO, C::SW);
                const uint64_t dVL0 = smem_desc(sb + C::OFF_STAGE + C::S_VL, 16, SBO, C::SW);
                const uint64_t dVH0 = smem_desc(sb + C::OFF_STAGE + C::S_VH, 16, SBO, C::SW);
                bool ok = wait_bounded_cluster(sy, sy.bar(P_RDY), 0, 1, -1);
                for (int v = 0; v < nsub && ok; ++v) {
                    if (v >= C::NB) {
                        const int w = v - C::NB;
                        ok = wait_bounded_cluster(sy, sy.bar(P_EMPTY + w % C::NST), (w / C::NST) & 1, 1, v);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const uint32_t so = STAGE_U * (v % C::NST);
                    const uint32_t tS = tmem + 128u * (v % C::NB), tDP = tS + 64;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) mma_pair_ss(tS, dQ + 2 * kk, dK0 + so + 2 * kk, ID_S, kk);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_pair_ss(tDP, dGL + 2 * kk, dVL0 + so + 2 * kk, ID_S, kk);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_pair_ss(tDP, dGH + 2 * kk, dVH0 + so + 2 * kk, ID_S, 1);
                    mma_commit_pair(sy.bar(P_SF + v % C::NB));
                }
                mma_commit_pair(sy.bar(P_DRAIN));
                wait_drain(sy.bar(P_DRAIN), 0);
            } else {
                const uint64_t dKH0 = smem_desc(sb + C::OFF_STAGE + C::S_KH, 16, SBOH, C::SWH);
                bool ok = true;
                for (int v = 0; v < nsub && ok; ++v) {
                    ok = wait_bounded_cluster(sy, sy.bar(P_PF + v % kPfRing), (v / kPfRing) & 1, 1, v);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t so = STAGE_U * (v % C::NST);
                    const uint32_t tDS = tmem + 128u * (v % C::NB);
                    // dQ += dS(v) K_v: A = dS over S(v)'s columns, 4 k-steps of 16 keys
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_pair_ts(tmem + C::C_DQ, tDS + 8 * kk, dKH0 + so + KSTEPH * kk, ID_Q,
                                    (v > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_pair(sy.bar(P_EMPTY + v % C::NST));
                }
                mma_commit_pair(sy.bar(P_ACC));
                if (!ok) wait_drain(sy.bar(P_ACC), 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax (one query row per thread)
        const int grp = (warp - 2) >> 2;
        const int q4 = warp & 3;
        const int il = q4 * 32 + lane;
        const int i = q0 + il;
        const bool qvalid = i < N;
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        const uint32_t pf0 = mapa_shared(sy.bar(P_PF), 0);
        // padded query rows: LSE = +inf makes P = 0
        const float L2 = qvalid ? lse[(size_t)bh * N + i] * kLog2e : INFINITY;
        const float Di = qvalid ? Drow[(size_t)bh * N + i] : 0.f;
        bool ok = true;
        for (int v = grp; v < nsub; v += 2) {
            const int buf = v % C::NB;
            ok = warp_wait_cluster(sy, sy.bar(P_SF + buf), (v / C::NB) & 1, 2, v);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tS = trow + 128u * buf, tDP = tS + 64;
            const int nvalid = N - v * 64;   // keys of this sub-tile that exist
// both chunks unrolled: the second chunk's work can overlap the first's
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t sr[32], pr[32];
                tmem_ld_32x32b_x32(tS + 32 * c, sr);
                tmem_ld_32x32b_x32(tDP + 32 * c, pr);
                tmem_wait_ld();
                uint32_t dk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float p0 = ex2_approx(fmaf(__uint_as_float(sr[e]), scale_log2, -L2));
                    float p1 = ex2_approx(fmaf(__uint_as_float(sr[e + 1]), scale_log2, -L2));
                    if (32 * c + e >= nvalid) p0 = 0.f;
                    if (32 * c + e + 1 >= nvalid) p1 = 0.f;
                    dk[e / 2] =
                        pack_bf16x2(p0 * (__uint_as_float(pr[e]) - Di), p1 * (__uint_as_float(pr[e + 1]) - Di));
                }
                // dS over the S columns already read
                tmem_st_32x32b_x16(tS + 16 * c, dk);
            }
            tmem_wait_st();
            tc_fence_before();
            // stand-in wait for the issuer: this CTA's stage of v+NB is loaded
            if (v + C::NB < nsub)
                ok = warp_wait(sy, sy.bar(P_FULL + (v + C::NB) % C::NST), ((v + C::NB) / C::NST) & 1, 2, v);
            mbar_arrive_cluster(pf0 + 8u * (v % kPfRing));
            if (!ok) break;
        }
        if (grp == 0) {
            if (ok) ok = warp_wait_cluster(sy, sy.bar(P_ACC), 0, 2, nsub);
            if (ok) {
                tc_fence_after();
                store_row<D>(trow + C::C_DQ, scale, qvalid, d_packed + ((size_t)bh * 4 * N + i) * D);
            }
        }
    }
    pair_teardown(tmem, warp);
}

// ---------------------------------------------------------------- host side
template <int D>
int launch_pair(const BwdArgs& a, std::string* err) {
    const long long Z = a.BH * 4;
    CUtensorMap p128, p32, ph, lo32, hi32, lo64, hi64, lo128, hi128;
    if (!encode_bf16_rows(&p128, a.packed, D, a.N, Z, 128, D, err) ||
        !encode_bf16_rows(&p32, a.packed, D, a.N, Z, 32, D, err) ||
        !encode_bf16_rows(&ph, a.packed, D, a.N, Z, 64, D / 2, err) ||
        !encode_bf16_rows(&lo32, a.do_lo, D, a.N, a.BH, 32, D, err) ||
        !encode_bf16_rows(&hi32, a.do_hi, D, a.N, a.BH, 32, D, err) ||
        !encode_bf16_rows(&lo64, a.do_lo, D, a.N, a.BH, 64, D, err) ||
        !encode_bf16_rows(&hi64, a.do_hi, D, a.N, a.BH, 64, D, err) ||
        !encode_bf16_rows(&lo128, a.do_lo, D, a.N, a.BH, 128, D, err) ||
        !encode_bf16_rows(&hi128, a.do_hi, D, a.N, a.BH, 128, D, err))
        return PSA_ERR_CUDA;
    if (!set_max_dynamic_smem((const void*)bwd_kv_pair_kernel<D>, KvCfg<D>::SMEM, err) ||
        !set_max_dynamic_smem((const void*)bwd_q_pair_kernel<D>, QCfg<D>::SMEM, err))
        return PSA_ERR_CUDA;
    float* Drow = static_cast<float*>(a.workspace);
    int rc = tc_pre_d_launch(a, Drow, err);
    if (rc != PSA_OK) return rc;
    const int npair = (a.N + 255) / 256;
    const long long grid = a.BH * npair * 2;
    if (grid > 0x7fffffffll) {
        *err = "grid too large";
        return PSA_ERR_UNSUPPORTED;
    }
    bf16* dp = static_cast<bf16*>(a.d_packed);
    const float sl2 = a.scale * kLog2e;
    {
        ProfScope prof(kSlotMain, a.stream);
        bwd_kv_pair_kernel<D><<<(unsigned)grid, kPairThreads, KvCfg<D>::SMEM, a.stream>>>(
            p128, p32, lo32, hi32, lo64, hi64, ph, a.lse, Drow, dp, a.N, npair, a.scale, sl2);
    }
    {
        ProfScope prof(kSlotDq, a.stream);
        bwd_q_pair_kernel<D><<<(unsigned)grid, kPairThreads, QCfg<D>::SMEM, a.stream>>>(
            p128, lo128, hi128, p32, ph, a.lse, Drow, dp, a.N, npair, a.scale, sl2);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = std::string("tensor-core pair backward launch: ") + cudaGetErrorString(e);
        return PSA_ERR_CUDA;
    }
    return PSA_OK;
}

}  // namespace

bool tc_pair_supported(int dtype, int d) { return dtype == PSA_BF16 && (d == 32 || d == 64); }

int tc_pair_launch(const BwdArgs& a, std::string* err) {
    switch (a.d) {
        case 32: return launch_pair<32>(a, err);
        case 64: return launch_pair<64>(a, err);
        default: *err = "unsupported head_dim for the pair kernels"; return PSA_ERR_UNSUPPORTED;
    }
}

int tc_pair_take_device_error(std::string* err) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_pair_error, sizeof(int)) != cudaSuccess || v == 0) return 0;
    const int zero = 0;
    cudaMemcpyToSymbol(g_pair_error, &zero, sizeof(int));
    static const char* roles[] = {"?", "producer", "mma", "softmax"};
    const int role = (v >> 24) & 0xff;
    *err = std::string("tensor-core pair backward: a bounded wait gave up (") + roles[role < 4 ? role : 0] +
           " warp, tile " + std::to_string(v & 0xFFFFFF) + ")";
    return 1;
}

}  // namespace psa
