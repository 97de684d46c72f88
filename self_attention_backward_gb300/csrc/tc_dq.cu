// tc_dq.cu -- tensor-core dQ pass of the PSA backward (bf16), query-outer.
//
// "Struct PsaFa2Backward" (description): the gradient of a query row needs a
// sweep over every key of its slice.  Here one CTA owns a 128-query tile of one
// (batch, head) and makes that sweep in 64-key sub-tiles v:
//   S    = Q K_v^T                    (M = 128 queries, N = 64 keys, K = d)
//   dP   = dO_lo V_lo,v^T + dO_hi V_hi,v^T             (K = 2d)
//   P    = exp2(S * scale*log2e - LSE*log2e),  dS = P o (dP - D)
//   dQ  += dS K_v                      (A = dS from TMEM, K = 64 keys)
// and writes scale * dQ as bf16 into section 0 of d_packed.  Each thread of the
// softmax warps owns one query row, so LSE and D are registers, and dS goes
// back into TMEM over its S columns: the softmax touches no shared memory.
// No atomics: the result does not depend on scheduling (the dK/dV pass, run
// with its dQ work switched off, is deterministic too).
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer (one
// thread) and TMEM owner, warps 2-5 softmax.  S/dP are triple-buffered in TMEM
// (3 x 128 columns) next to the dQ accumulator; K/V sub-tiles rotate through
// four shared-memory stages.  All waits are bounded (tc_sync.cuh).
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

__device__ int g_dq_error = 0;

constexpr int kDqThreads = 192;

template <int D>
struct DqCfg {
    static constexpr int BQ = 128;                 // queries per CTA (MMA M)
    static constexpr int BK = 64;                  // keys per sub-tile
    static constexpr int NB = 3;                   // S/dP buffers in TMEM
    static constexpr int NST = 4;                  // K/V stages (> NB: the stage of v+NB must differ from v's)
    static constexpr int ROWB = D * 2;
    static constexpr int QT = 128 * ROWB;          // [128, D] tile (Q, dO_lo, dO_hi)
    static constexpr int KT = 64 * ROWB;           // [64, D] sub-tile (K, V_lo, V_hi)
    static constexpr uint32_t SW = D == 64 ? 2u : D == 32 ? 4u : 6u;
    static constexpr int OFF_Q = 0;                // Q, dO_lo, dO_hi
    static constexpr int OFF_STAGE = 3 * QT;       // stage s: K, V_lo, V_hi at +s*STAGE
    static constexpr int STAGE = 3 * KT;
    static constexpr int OFF_BAR = OFF_STAGE + NST * STAGE;
    static constexpr int OFF_MISC = OFF_BAR + 256;
    static constexpr int USED = OFF_MISC + 64;
    static constexpr int SMEM = (USED + 1024) > 118784 ? (USED + 1024) : 118784;  // one CTA per SM
    // TMEM: buffer b = [128b, 128b+128): S (64 keys), dP (64 keys); dQ after the buffers
    static constexpr uint32_t C_DQ = 128 * NB;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(C_DQ + D <= TMEM_COLS, "TMEM budget");
    static_assert(NST > NB, "the softmax's wait for the stage of v+NB would wait on its own release");
};

// barriers: Q/dO loaded, stage full/empty, S/dP ready (per buffer), dS written (per buffer), dQ done
enum { Q_IN = 0, Q_FULL = 1, Q_EMPTY = 5, Q_SF = 9, Q_SD = 12, Q_ACC = 15 };

template <int D>
__global__ void __launch_bounds__(kDqThreads, 1)
dq_kernel(const __grid_constant__ CUtensorMap tm_q128, const __grid_constant__ CUtensorMap tm_k64,
          const __grid_constant__ CUtensorMap tm_lo, const __grid_constant__ CUtensorMap tm_hi,
          const float* __restrict__ lse, const float* __restrict__ Drow, bf16* __restrict__ d_packed, int N,
          int nqt, float scale, float scale_log2) {
    using C = DqCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    Sync sy{sb + C::OFF_BAR, reinterpret_cast<volatile int*>(smem + C::OFF_MISC), &g_dq_error};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x / nqt, qt = blockIdx.x % nqt;
    const int q0 = qt * C::BQ;
    const int nsub = (N + C::BK - 1) / C::BK;

    if (threadIdx.x == 0) {
        mbar_init(sy.bar(Q_IN), 1);
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(sy.bar(Q_FULL + s), 1);
            mbar_init(sy.bar(Q_EMPTY + s), 1);
        }
        for (int b = 0; b < C::NB; ++b) {
            mbar_init(sy.bar(Q_SF + b), 1);
            mbar_init(sy.bar(Q_SD + b), 128);
        }
        mbar_init(sy.bar(Q_ACC), 1);
        *sy.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q128);
        tma_prefetch_desc(&tm_k64);
        tma_prefetch_desc(&tm_lo);
        tma_prefetch_desc(&tm_hi);
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
        if (lane == 0) {
            int last[C::NST];
#pragma unroll
            for (int s = 0; s < C::NST; ++s) last[s] = -1;
            mbar_arrive_expect_tx(sy.bar(Q_IN), 3 * C::QT);
            tma_load_3d(sb + C::OFF_Q, &tm_q128, 0, q0, bh * 4 + 0, sy.bar(Q_IN));
            tma_load_3d(sb + C::OFF_Q + C::QT, &tm_lo, 0, q0, bh, sy.bar(Q_IN));
            tma_load_3d(sb + C::OFF_Q + 2 * C::QT, &tm_hi, 0, q0, bh, sy.bar(Q_IN));
            int s = 0, ph = 0;
            for (int v = 0; v < nsub; ++v) {
                if (!wait_bounded(sy, sy.bar(Q_EMPTY + s), ph ^ 1, 0, v)) break;
                const uint32_t st = sb + C::OFF_STAGE + s * C::STAGE;
                mbar_arrive_expect_tx(sy.bar(Q_FULL + s), 3 * C::KT);
                tma_load_3d(st, &tm_k64, 0, v * C::BK, bh * 4 + 1, sy.bar(Q_FULL + s));
                tma_load_3d(st + C::KT, &tm_k64, 0, v * C::BK, bh * 4 + 2, sy.bar(Q_FULL + s));
                tma_load_3d(st + 2 * C::KT, &tm_k64, 0, v * C::BK, bh * 4 + 3, sy.bar(Q_FULL + s));
#pragma unroll
                for (int x = 0; x < C::NST; ++x)
                    if (x == s) last[x] = v;
                if (++s == C::NST) { s = 0; ph ^= 1; }
            }
            if (*sy.abort) {
                wait_drain(sy.bar(Q_IN), 0);
#pragma unroll
                for (int x = 0; x < C::NST; ++x)
                    if (last[x] >= 0) wait_drain(sy.bar(Q_FULL + x), (last[x] / C::NST) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(128, 64, 0, 0);    // S, dP: 64 keys
            constexpr uint32_t ID_Q = idesc_bf16(128, D, 0, 1);     // dQ: A = dS (TMEM), B = K rows MN-major
            constexpr uint32_t SBO = 8 * C::ROWB;
            constexpr uint32_t KSTEP = (16 * C::ROWB) >> 4;
            constexpr uint32_t STAGE_U = C::STAGE >> 4, KT_U = C::KT >> 4, QT_U = C::QT >> 4;
            const uint64_t dQt = smem_desc(sb + C::OFF_Q, 16, SBO, C::SW);       // Q, then dO_lo, dO_hi (+QT)
            const uint64_t dStage0 = smem_desc(sb + C::OFF_STAGE, 16, SBO, C::SW);  // K, then V_lo, V_hi (+KT)
            // S(v), dP(v) into TMEM buffer v % 3 (the stage is known loaded: the prologue
            // waits for it, later the softmax thread that arrives SD(v-3) waited first)
            auto issue_s_dp = [&](int v) {
                const int s = v % C::NST;
                const uint64_t dK = dStage0 + STAGE_U * s;
                const uint32_t tS = tmem + 128u * (v % C::NB), tDP = tS + 64;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_bf16_ss(tS, dQt + 2 * kk, dK + 2 * kk, ID_S, kk);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_ss(tDP, dQt + QT_U + 2 * kk, dK + KT_U + 2 * kk, ID_S, kk);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_ss(tDP, dQt + 2 * QT_U + 2 * kk, dK + 2 * KT_U + 2 * kk, ID_S, 1);
                mma_commit(sy.bar(Q_SF + v % C::NB));
            };
            bool ok = wait_bounded(sy, sy.bar(Q_IN), 0, 1, -1);
            for (int v = 0; v < C::NB && v < nsub && ok; ++v) ok = wait_bounded(sy, sy.bar(Q_FULL + v), 0, 1, v);
            if (ok) {
                tc_fence_after();
                for (int v = 0; v < C::NB && v < nsub; ++v) issue_s_dp(v);
            }
            for (int v = 0; v < nsub && ok; ++v) {
                const int b = v % C::NB, s = v % C::NST;
                ok = wait_bounded(sy, sy.bar(Q_SD + b), (v / C::NB) & 1, 1, v);
                if (!ok) break;
                tc_fence_after();
                // dQ += dS(v) K_v : A = dS over S(v)'s columns, 4 k-steps of 16 keys
                const uint64_t dKmn = dStage0 + STAGE_U * s;
#pragma unroll
                for (int kk = 0; kk < C::BK / 16; ++kk)
                    mma_bf16_ts(tmem + C::C_DQ, tmem + 128u * b + 8 * kk, dKmn + KSTEP * kk, ID_Q,
                                (v > 0 || kk > 0) ? 1u : 0u);
                mma_commit(sy.bar(Q_EMPTY + s));
                if (v + C::NB < nsub) issue_s_dp(v + C::NB);
            }
            mma_commit(sy.bar(Q_ACC));
            if (!ok) wait_drain(sy.bar(Q_ACC), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax (one query row per thread)
        const int q4 = warp & 3;
        const int il = q4 * 32 + lane;
        const int i = q0 + il;
        const bool qvalid = i < N;
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        // padded query rows: LSE = +inf makes P = 0
        const float L2 = qvalid ? lse[(size_t)bh * N + i] * kLog2e : INFINITY;
        const float Di = qvalid ? Drow[(size_t)bh * N + i] : 0.f;
        bool ok = true;
        for (int v = 0; v < nsub; ++v) {
            const int b = v % C::NB;
            ok = warp_wait(sy, sy.bar(Q_SF + b), (v / C::NB) & 1, 2, v);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tS = trow + 128u * b, tDP = tS + 64;
            const int nvalid = N - v * C::BK;        // keys of this sub-tile that exist
#pragma unroll 1
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
                    dk[e / 2] = pack_bf16x2(p0 * (__uint_as_float(pr[e]) - Di), p1 * (__uint_as_float(pr[e + 1]) - Di));
                }
                // dS over the S columns already read
                tmem_st_32x32b_x16(tS + 16 * c, dk);
            }
            tmem_wait_st();
            tc_fence_before();
            // stand-in wait for the MMA issuer: the K/V stage of v+3 is loaded
            if (v + C::NB < nsub)
                ok = warp_wait(sy, sy.bar(Q_FULL + (v + C::NB) % C::NST), ((v + C::NB) / C::NST) & 1, 2, v);
            mbar_arrive(sy.bar(Q_SD + b));
            if (!ok) break;
        }
        if (ok) ok = warp_wait(sy, sy.bar(Q_ACC), 0, 2, nsub);
        if (ok) {
            tc_fence_after();
            uint32_t vq[D];
            tmem_ld_row<D>(trow + C::C_DQ, vq);       // whole warp; only existing rows are stored
            tmem_wait_ld();
            if (qvalid) {
                bf16* o = d_packed + ((size_t)bh * 4 * N + i) * D;
#pragma unroll
                for (int e = 0; e < D; e += 8) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(vq[e + 0]) * scale, __uint_as_float(vq[e + 1]) * scale);
                    w.y = pack_bf16x2(__uint_as_float(vq[e + 2]) * scale, __uint_as_float(vq[e + 3]) * scale);
                    w.z = pack_bf16x2(__uint_as_float(vq[e + 4]) * scale, __uint_as_float(vq[e + 5]) * scale);
                    w.w = pack_bf16x2(__uint_as_float(vq[e + 6]) * scale, __uint_as_float(vq[e + 7]) * scale);
                    *reinterpret_cast<uint4*>(o + e) = w;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D>
int launch_dq(const BwdArgs& a, const float* Drow, std::string* err) {
    using C = DqCfg<D>;
    CUtensorMap tq, tk, tlo, thi;
    if (!encode_bf16_rows(&tq, a.packed, D, a.N, a.BH * 4, C::BQ, D, err) ||
        !encode_bf16_rows(&tk, a.packed, D, a.N, a.BH * 4, C::BK, D, err) ||
        !encode_bf16_rows(&tlo, a.do_lo, D, a.N, a.BH, C::BQ, D, err) ||
        !encode_bf16_rows(&thi, a.do_hi, D, a.N, a.BH, C::BQ, D, err))
        return PSA_ERR_CUDA;
    if (!set_max_dynamic_smem((const void*)dq_kernel<D>, C::SMEM, err)) return PSA_ERR_CUDA;
    const int nqt = (a.N + C::BQ - 1) / C::BQ;
    const long long grid = a.BH * nqt;
    if (grid > 0x7fffffffll) {
        *err = "grid too large";
        return PSA_ERR_UNSUPPORTED;
    }
    {
        ProfScope prof(kSlotDq, a.stream);
        dq_kernel<D><<<(unsigned)grid, kDqThreads, C::SMEM, a.stream>>>(
            tq, tk, tlo, thi, a.lse, Drow, static_cast<bf16*>(a.d_packed), a.N, nqt, a.scale, a.scale * kLog2e);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = std::string("tensor-core dQ launch: ") + cudaGetErrorString(e);
        return PSA_ERR_CUDA;
    }
    return PSA_OK;
}

}  // namespace

int tc_dq_launch(const BwdArgs& a, const float* Drow, std::string* err) {
    switch (a.d) {
        case 16: return launch_dq<16>(a, Drow, err);
        case 32: return launch_dq<32>(a, Drow, err);
        case 64: return launch_dq<64>(a, Drow, err);
        default: *err = "unsupported head_dim"; return PSA_ERR_UNSUPPORTED;
    }
}

int tc_dq_take_device_error(std::string* err) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_dq_error, sizeof(int)) != cudaSuccess || v == 0) return 0;
    const int zero = 0;
    cudaMemcpyToSymbol(g_dq_error, &zero, sizeof(int));
    *err = "tensor-core dQ pass: a bounded wait gave up (role " + std::to_string(((v >> 24) & 0xff) - 1) +
           ", tile " + std::to_string(v & 0xFFFFFF) + ")";
    return 1;
}

}  // namespace psa
