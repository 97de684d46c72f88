// tc_fwd.cu -- tensor-core (tcgen05 / TMEM / TMA) PSA forward, bf16 storage.
//
// Produces what the backward consumes: O_lo = P V_lo, O_hi = P V_hi and the
// natural-log row statistic LSE of P = softmax(scale Q K^T) ("Struct
// PsaFa2Backward", "Grid" paragraph: the backward shares the forward's
// decomposition).  As in the backward, lo and hi run as one attention with a
// 2d-wide value [V_lo | V_hi].
//
// One CTA per (batch*head, 128-query tile), one pass over 64-key tiles j with
// an online softmax (per query row a running max m and sum l, log2 domain):
//   S = Q K_j^T                      (M = 128 queries, N = 64 keys, K = d)
//   m' = max(m, max_k S c) if that exceeds m by more than 8, else m
//        (a stale max keeps P <= 2^8; when m moves, l and O are scaled by
//        exp2(m - m'), O read and written back in TMEM)
//   P = exp2(S c - m) written over S in TMEM as bf16 pairs,  l += sum P
//   [O_lo | O_hi] += P [V_lo,j | V_hi,j]   (A = P from TMEM, N = 2d)
// and at the end O / l and LSE = (m + log2 l) ln 2.  c = scale log2(e).
//
// Warp roles (192 threads): warp 0 TMA producer (lane 0 Q and K, lane 1 V),
// warp 1 MMA issuer (one thread) and TMEM owner, warps 2-5 softmax (one query
// row per thread, the warp's TMEM lane quarter).  A CTA holds 256 TMEM columns
// (NSB 64-column S buffers, then O), so two CTAs share an SM.  S(j+1) .. S(j+NSB-1)
// are computed while the softmax works on S(j), and S(j+NSB) once P(j) V_j has
// read P(j); the other CTA's softmax and MMAs fill the remaining gaps of the
// tensor pipe and the exp2 unit.  A row max that moves by more than 2^8 makes
// the softmax rescale O, after waiting for P(j-1) V_{j-1} to finish (rare after
// the first tiles).  K tiles rotate through NSB shared-memory stages,
// [V_lo | V_hi] through two; the softmax warps wait for K_{j+NSB} and the
// current V before they release P, so the issuing thread waits once per key
// tile.  All waits are bounded (tc_sync.cuh).
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

__device__ int g_fwd_error = 0;

constexpr int kFwdThreads = 192;
constexpr float kRescaleLog2 = 8.f;   // keep a stale row max while the new one is at most 2^8 larger

template <int D>
struct FwdCfg {
    static constexpr int BQ = 128;                 // queries per CTA (MMA M)
    static constexpr int BK = 64;                  // keys per tile
    static constexpr int ROWB = D * 2;
    static constexpr int TILE = 128 * ROWB;        // [128, D] bf16 tile (Q)
    static constexpr int KT = BK * ROWB;           // [64, D] bf16 tile (K, V_lo, V_hi)
    static constexpr uint32_t SW = D == 64 ? 2u : D == 32 ? 4u : 6u;
    // S buffers: three at d <= 32 (3 x 64 columns next to O's 2d fit the CTA's
    // 256), two at d = 64.  S(j + NSB) is issued after P(j) V_j, so the loop
    // softmax -> P V -> next S spans NSB tiles: a deeper ring hides more of it.
    static constexpr int NSB = D == 64 ? 2 : 3;
    // K stages: as many as S buffers.  The softmax of tile j waits for
    // K_{j+NSB} in stage (j+NSB) % NK; with NK = NSB that stage last held K_j,
    // whose copy completed before S(j) ran, so the parity test never meets a
    // stage two copies behind (with NK = 2 < NSB it could, and pass early).
    static constexpr int NK = NSB;
    static constexpr int NV = 2;                   // [V_lo | V_hi] stages
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = TILE;             // K stage s at +s*KT
    static constexpr int OFF_V = OFF_K + NK * KT;  // V stage s: V_lo, V_hi at +s*2*KT
    static constexpr int OFF_BAR = OFF_V + NV * 2 * KT;
    static constexpr int OFF_MISC = OFF_BAR + 256;
    static constexpr int OFF_EPI = OFF_MISC + 64;  // 2 KB per softmax warp: coalesced O stores
    static constexpr int USED = OFF_EPI + 4 * 2048;
    static constexpr int SMEM = USED + 1024;       // two CTAs per SM
    static constexpr uint32_t C_O = 64 * NSB;      // S buffers at 0, 64 (, 128); O_lo | O_hi at C_O
    static constexpr uint32_t TMEM_COLS = 256;
    static_assert(C_O + 2 * D <= TMEM_COLS, "TMEM budget");
    static_assert(2 * (SMEM + 1024) <= 233472, "two CTAs per SM");
};

// barriers: Q loaded, O final, S ready[NSB], P written[NSB] (softmax done), K
// full/empty[NK], V full/empty[2], O updated after P(j) V_j at OD + (j & 1): a
// rescale at tile j waits for P(j-1) V_{j-1} on a barrier whose previous phase,
// P(j-3) V_{j-3}, finished before S(j) (issued after it) did, so the parity
// test cannot pass a phase early even with three S buffers (a single barrier
// could: P(j-2) V_{j-2} may still run when the softmax of j starts)
enum { F_Q = 0, F_ACC = 1, F_SF = 2, F_PF = 5, F_KF = 8, F_KE = 11, F_VF = 14, F_VE = 16, F_OD = 18 };

// x = S * c over one key tile, written back over sr, and max x over the keys
// that exist (the first nvalid; all of them when !MASK).  Masked keys get
// x = -inf, so that their probability below is exactly 0.  Packed f32x2
// multiplies and three-input maxima: the softmax is issue-bound, and per-key
// mask tests on every tile had kept the ALU pipe 62% busy.
template <bool MASK, int BK>
__device__ __forceinline__ float fwd_scale_max(uint32_t (&sr)[BK], float c, int nvalid) {
    const uint64_t c2 = f2_pack(c, c);
    float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
    for (int e = 0; e < BK; e += 4) {
        float x0, x1, x2, x3;
        f2_unpack(f2_mul(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2), x0, x1);
        f2_unpack(f2_mul(f2_pack(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), c2), x2, x3);
        if (MASK) {
            if (e + 0 >= nvalid) x0 = -INFINITY;
            if (e + 1 >= nvalid) x1 = -INFINITY;
            if (e + 2 >= nvalid) x2 = -INFINITY;
            if (e + 3 >= nvalid) x3 = -INFINITY;
        }
        ma = fmax3(ma, x0, x1);
        mb = fmax3(mb, x2, x3);
        sr[e] = __float_as_uint(x0);
        sr[e + 1] = __float_as_uint(x1);
        sr[e + 2] = __float_as_uint(x2);
        sr[e + 3] = __float_as_uint(x3);
    }
    return fmaxf(ma, mb);
}

// P = exp2(x - m) over one key tile (x from fwd_scale_max), stored over S in
// TMEM as bf16 pairs (all of S is in registers); returns the tile's sum of P.
template <int BK>
__device__ __forceinline__ float fwd_probs(const uint32_t (&sr)[BK], float m, uint32_t tS) {
    const uint64_t m2 = f2_pack(m, m), one2 = f2_pack(1.f, 1.f);
    uint64_t la = f2_pack(0.f, 0.f), lb = la;
#pragma unroll
    for (int c = 0; c < BK / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const int k = 32 * c + e;
            float p0, p1, p2, p3;
            f2_unpack(f2_sub(f2_pack(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), m2), p0, p1);
            f2_unpack(f2_sub(f2_pack(__uint_as_float(sr[k + 2]), __uint_as_float(sr[k + 3])), m2), p2, p3);
            p0 = ex2_approx(p0);
            p1 = ex2_approx(p1);
            p2 = ex2_approx(p2);
            p3 = ex2_approx(p3);
            la = f2_fma(f2_pack(p0, p1), one2, la);
            lb = f2_fma(f2_pack(p2, p3), one2, lb);
            pk[e / 2] = pack_bf16x2(p0, p1);
            pk[e / 2 + 1] = pack_bf16x2(p2, p3);
        }
        tmem_st_32x32b_x16(tS + 16 * c, pk);
    }
    float a0, a1, b0, b1;
    f2_unpack(la, a0, a1);
    f2_unpack(lb, b0, b1);
    return (a0 + a1) + (b0 + b1);
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 2)
fwd_kernel(const __grid_constant__ CUtensorMap tm_pk, const __grid_constant__ CUtensorMap tm_kv, bf16* __restrict__ o_lo, bf16* __restrict__ o_hi,
           float* __restrict__ lse, int N, int nqt, float scale_log2) {
    using C = FwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    Sync sy{sb + C::OFF_BAR, reinterpret_cast<volatile int*>(smem + C::OFF_MISC), &g_fwd_error};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x / nqt, qt = blockIdx.x % nqt;
    const int q0 = qt * C::BQ;
    const int nk = (N + C::BK - 1) / C::BK;

    if (threadIdx.x == 0) {
        mbar_init(sy.bar(F_Q), 1);
        mbar_init(sy.bar(F_ACC), 1);
        mbar_init(sy.bar(F_OD), 1);
        mbar_init(sy.bar(F_OD + 1), 1);
        for (int s = 0; s < C::NSB; ++s) {
            mbar_init(sy.bar(F_SF + s), 1);
            mbar_init(sy.bar(F_PF + s), 128);
        }
        for (int s = 0; s < C::NK; ++s) {
            mbar_init(sy.bar(F_KF + s), 1);
            mbar_init(sy.bar(F_KE + s), 1);
        }
        for (int s = 0; s < C::NV; ++s) {
            mbar_init(sy.bar(F_VF + s), 1);
            mbar_init(sy.bar(F_VE + s), 1);
        }
        *sy.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_pk);
        tma_prefetch_desc(&tm_kv);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // lane 0 loads Q and the K tiles, lane 1 the [V_lo | V_hi] tiles: the two
        // streams run ahead independently (the softmax of tile j waits for
        // K_{j+NSB} before releasing P(j), whose P V frees a V stage)
        if (lane == 0) {
            int lastk[C::NK];
#pragma unroll
            for (int x = 0; x < C::NK; ++x) lastk[x] = -1;
            mbar_arrive_expect_tx(sy.bar(F_Q), C::TILE);
            tma_load_3d(sb + C::OFF_Q, &tm_pk, 0, q0, bh * 4 + 0, sy.bar(F_Q));
            for (int j = 0; j < nk; ++j) {
                const int sk = j % C::NK;
                if (!wait_bounded(sy, sy.bar(F_KE + sk), ((j / C::NK) & 1) ^ 1, 0, j)) break;
                mbar_arrive_expect_tx(sy.bar(F_KF + sk), C::KT);
                tma_load_3d(sb + C::OFF_K + sk * C::KT, &tm_kv, 0, j * C::BK, bh * 4 + 1, sy.bar(F_KF + sk));
#pragma unroll
                for (int x = 0; x < C::NK; ++x)
                    if (x == sk) lastk[x] = j;
            }
            if (*sy.abort) {
                wait_drain(sy.bar(F_Q), 0);
#pragma unroll
                for (int x = 0; x < C::NK; ++x)
                    if (lastk[x] >= 0) wait_drain(sy.bar(F_KF + x), (lastk[x] / C::NK) & 1);
            }
        } else if (lane == 1) {
            int lastv[C::NV];
#pragma unroll
            for (int x = 0; x < C::NV; ++x) lastv[x] = -1;
            for (int j = 0; j < nk; ++j) {
                const int sv = j % C::NV;
                if (!wait_bounded(sy, sy.bar(F_VE + sv), ((j / C::NV) & 1) ^ 1, 0, j)) break;
                const uint32_t vs = sb + C::OFF_V + sv * 2 * C::KT;
                mbar_arrive_expect_tx(sy.bar(F_VF + sv), 2 * C::KT);
                tma_load_3d(vs, &tm_kv, 0, j * C::BK, bh * 4 + 2, sy.bar(F_VF + sv));
                tma_load_3d(vs + C::KT, &tm_kv, 0, j * C::BK, bh * 4 + 3, sy.bar(F_VF + sv));
#pragma unroll
                for (int x = 0; x < C::NV; ++x)
                    if (x == sv) lastv[x] = j;
            }
            if (*sy.abort) {
#pragma unroll
                for (int x = 0; x < C::NV; ++x)
                    if (lastv[x] >= 0) wait_drain(sy.bar(F_VF + x), (lastv[x] / C::NV) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(128, 64, 0, 0);
            constexpr uint32_t ID_O = idesc_bf16(128, 2 * D, 0, 1);   // A = P (TMEM), B = [V_lo | V_hi] MN-major
            constexpr uint32_t SBO = 8 * C::ROWB;
            constexpr uint32_t KSTEP = (16 * C::ROWB) >> 4;
            const uint64_t dQ = smem_desc(sb + C::OFF_Q, 16, SBO, C::SW);
            const uint64_t dK0 = smem_desc(sb + C::OFF_K, 16, SBO, C::SW);
            const uint64_t dV0 = smem_desc(sb + C::OFF_V, C::KT, SBO, C::SW);
            constexpr uint32_t KT_U = C::KT >> 4;
            // S(j) = Q K_j^T into buffer j % NSB; K_j is known to be loaded (the
            // prologue waits for the first K tiles, up to NSB; later the softmax
            // warps wait for K_{j+NSB} before releasing P(j))
            auto issue_s = [&](int j) {
                const int sk = j % C::NK;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_ss(tmem + 64u * (j % C::NSB), dQ + 2 * kk, dK0 + KT_U * sk + 2 * kk, ID_S, kk);
                mma_commit(sy.bar(F_SF + j % C::NSB));
                mma_commit(sy.bar(F_KE + sk));
            };
            bool ok = wait_bounded(sy, sy.bar(F_Q), 0, 1, -1);
            // the first NSB S products; with NSB > NK, K_j of j >= NK arrives once
            // S(j - NK) has freed its stage, which the loop below issues in order
            for (int j = 0; j < C::NSB && j < nk && ok; ++j) {
                ok = wait_bounded(sy, sy.bar(F_KF + j % C::NK), (j / C::NK) & 1, 1, j);
                if (ok) {
                    tc_fence_after();
                    issue_s(j);
                }
            }
            for (int j = 0; j < nk && ok; ++j) {
                // P(j) written over S(j), O rescaled if a row max moved, V_j and
                // K_{j+NSB} loaded (the softmax warps waited for both)
                ok = wait_bounded(sy, sy.bar(F_PF + j % C::NSB), (j / C::NSB) & 1, 1, j);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dV = dV0 + 2 * KT_U * (j % C::NV);
#pragma unroll
                for (int kk = 0; kk < C::BK / 16; ++kk)
                    mma_bf16_ts(tmem + C::C_O, tmem + 64u * (j % C::NSB) + 8 * kk, dV + KSTEP * kk, ID_O,
                                (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(sy.bar(F_VE + j % C::NV));
                mma_commit(sy.bar(F_OD + (j & 1)));
                // S(j+NSB) overwrites P(j): issued after P(j) V_j, the pipe keeps issue order
                if (j + C::NSB < nk) issue_s(j + C::NSB);
            }
            mma_commit(sy.bar(F_ACC));
            if (!ok) wait_drain(sy.bar(F_ACC), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax (one query row per thread)
        const int q4 = warp & 3;
        const int il = q4 * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        float m = -INFINITY, l = 0.f;              // log2-domain row max in use and row sum
        bool ok = true;
        for (int j = 0; j < nk; ++j) {
            const uint32_t tS = trow + 64u * (j % C::NSB);
            ok = warp_wait(sy, sy.bar(F_SF + j % C::NSB), (j / C::NSB) & 1, 2, j);
            if (!ok) break;
            tc_fence_after();
            const int nvalid = N - j * C::BK;      // keys of this tile that exist (>= 1)
            uint32_t sr[C::BK];
#pragma unroll
            for (int c = 0; c < C::BK / 32; ++c)
                tmem_ld_32x32b_x32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sr + 32 * c));
            tmem_wait_ld();
            // scaled scores and their max (masked keys -> -inf, whose exp2 is 0);
            // only the ragged last tile pays for the key mask
            const float mt = nvalid >= C::BK ? fwd_scale_max<false>(sr, scale_log2, nvalid)
                                             : fwd_scale_max<true>(sr, scale_log2, nvalid);
            const bool move = mt > m + kRescaleLog2;
            const float m_new = move ? mt : m;
            const float alpha = move ? ex2_approx(m - m_new) : 1.f;   // 0 on the first tile
            l *= alpha;
            if (j > 0 && __any_sync(0xffffffffu, move)) {
                // O *= alpha on this warp's rows, once P(j-1) V_{j-1} has finished
                // (every lane loads and stores: .sync.aligned)
                ok = warp_wait(sy, sy.bar(F_OD + ((j - 1) & 1)), ((j - 1) >> 1) & 1, 2, j);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2 * D; h += 32) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(trow + C::C_O + h, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st_32x32b_x16(trow + C::C_O + h, o);
                    tmem_st_32x32b_x16(trow + C::C_O + h + 16, o + 16);
                }
                tmem_wait_st();
            }
            m = m_new;
            l += fwd_probs(sr, m, tS);
            tmem_wait_st();
            tc_fence_before();
            // stand-in waits for the issuer: V_j and K_{j+NSB} are in shared memory
            ok = warp_wait(sy, sy.bar(F_VF + j % C::NV), (j / C::NV) & 1, 2, j);
            if (ok && j + C::NSB < nk)
                ok = warp_wait(sy, sy.bar(F_KF + (j + C::NSB) % C::NK), ((j + C::NSB) / C::NK) & 1, 2, j);
            mbar_arrive(sy.bar(F_PF + j % C::NSB));
            if (!ok) break;
        }
        if (ok) ok = warp_wait(sy, sy.bar(F_ACC), 0, 2, nk);
        if (ok) {
            // TMEM loads are warp-collective (.sync.aligned): every lane loads,
            // only rows that exist are stored
            tc_fence_after();
            const int i = q0 + il;
            const bool valid = i < N;
            const size_t row = (size_t)bh * N + (valid ? i : 0);
            if (valid) lse[row] = (m + __log2f(l)) * kLn2;
            const float inv_l = 1.f / l;
            // the warp's 32 query rows, coalesced through its staging buffer
            const int r0 = q0 + q4 * 32;
            uint32_t v[D];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                tmem_ld_row<D>(trow + C::C_O + h * D, v);
                tmem_wait_ld();
                uint32_t w[D / 2];
#pragma unroll
                for (int e = 0; e < D / 2; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * inv_l, __uint_as_float(v[2 * e + 1]) * inv_l);
                store_rows_staged<D>(sb + C::OFF_EPI + 2048u * (warp - 2), w,
                                     reinterpret_cast<uint16_t*>((h == 0 ? o_lo : o_hi) + ((size_t)bh * N + r0) * D), D,
                                     N - r0, lane);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D>
int launch_fwd(const void* packed, void* o_lo, void* o_hi, float* lse, long long BH, int N, float scale,
               cudaStream_t stream, std::string* err) {
    using C = FwdCfg<D>;
    // two maps over packed [BH*4, N, D]: 128-row boxes (Q) and 64-row boxes (K, V)
    CUtensorMap tm, tm_kv;
    if (!encode_bf16_rows(&tm, packed, D, N, BH * 4, C::BQ, D, err) ||
        !encode_bf16_rows(&tm_kv, packed, D, N, BH * 4, C::BK, D, err))
        return PSA_ERR_CUDA;
    if (!set_max_dynamic_smem((const void*)fwd_kernel<D>, C::SMEM, err)) return PSA_ERR_CUDA;
    const int nqt = (N + C::BQ - 1) / C::BQ;
    const long long grid = BH * nqt;
    if (grid > 0x7fffffffll) {
        *err = "grid too large";
        return PSA_ERR_UNSUPPORTED;
    }
    {
        ProfScope prof(kSlotFwd, stream);
        fwd_kernel<D><<<(unsigned)grid, kFwdThreads, C::SMEM, stream>>>(
            tm, tm_kv, static_cast<bf16*>(o_lo), static_cast<bf16*>(o_hi), lse, N, nqt, scale * kLog2e);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = std::string("tensor-core forward launch: ") + cudaGetErrorString(e);
        return PSA_ERR_CUDA;
    }
    return PSA_OK;
}

}  // namespace

bool tc_fwd_supported(int dtype, int d) { return dtype == PSA_BF16 && (d == 16 || d == 32 || d == 64); }

int tc_fwd_launch(const void* packed, void* o_lo, void* o_hi, float* lse, long long BH, int N, int d, float scale,
                  cudaStream_t stream, std::string* err) {
    switch (d) {
        case 16: return launch_fwd<16>(packed, o_lo, o_hi, lse, BH, N, scale, stream, err);
        case 32: return launch_fwd<32>(packed, o_lo, o_hi, lse, BH, N, scale, stream, err);
        case 64: return launch_fwd<64>(packed, o_lo, o_hi, lse, BH, N, scale, stream, err);
        default: *err = "unsupported head_dim"; return PSA_ERR_UNSUPPORTED;
    }
}

int tc_fwd_take_device_error(std::string* err) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fwd_error, sizeof(int)) != cudaSuccess || v == 0) return 0;
    const int zero = 0;
    cudaMemcpyToSymbol(g_fwd_error, &zero, sizeof(int));
    *err = "tensor-core forward: a bounded wait gave up (role " + std::to_string(((v >> 24) & 0xff) - 1) +
           ", tile " + std::to_string(v & 0xFFFFFF) + ")";
    return 1;
}

}  // namespace psa
