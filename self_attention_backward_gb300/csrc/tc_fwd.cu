// tc_fwd.cu -- tensor-core (tcgen05 / TMEM / TMA) PSA forward, bf16 storage.
//
// Produces what the backward consumes: O_lo = P V_lo, O_hi = P V_hi and the
// natural-log row statistic LSE of P = softmax(scale Q K^T) ("Struct
// PsaFa2Backward", "Grid" paragraph: the backward shares the forward's
// decomposition).  As in the backward, lo and hi run as one attention with a
// 2d-wide value [V_lo | V_hi].
//
// One CTA per (batch*head, 128-query tile), two passes over 128-key tiles:
//   pass 1: S = Q K_j^T (M = 128 queries, N = 128 keys) -> per query row the
//           running max and sum of exp2(S * scale*log2e) -> LSE;
//   pass 2: S again, P = exp2(S * scale*log2e - LSE*log2e) (already
//           normalised) written over S in TMEM as bf16 pairs, then
//           [O_lo | O_hi] += P [V_lo,j | V_hi,j] with P as the MMA's A operand
//           from TMEM (one N = 2d MMA per 16-key step).
// Two passes recompute S once more than an online softmax would, and in
// exchange O never needs rescaling.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer (one
// thread) and TMEM owner, warps 2-5 softmax (one query row per thread, the
// warp's TMEM lane quarter).  S is double-buffered in TMEM; K (and in pass 2
// V_lo, V_hi) tiles are double-buffered in shared memory.  All waits are
// bounded (tc_sync.cuh).
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

namespace psa {
namespace {

using namespace psa::tc;
using bf16 = __nv_bfloat16;

__device__ int g_fwd_error = 0;

constexpr int kFwdThreads = 192;

template <int D>
struct FwdCfg {
    static constexpr int BQ = 128;                 // queries per CTA (MMA M)
    static constexpr int BK = 128;                 // keys per tile
    static constexpr int ROWB = D * 2;
    static constexpr int TILE = 128 * ROWB;        // [128, D] bf16 tile
    static constexpr uint32_t SW = D == 64 ? 2u : D == 32 ? 4u : 6u;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_STAGE = TILE;         // stage s: K, V_lo, V_hi at +s*STAGE
    static constexpr int STAGE = 3 * TILE;
    static constexpr int OFF_BAR = OFF_STAGE + 2 * STAGE;
    static constexpr int OFF_MISC = OFF_BAR + 128;
    static constexpr int USED = OFF_MISC + 64;
    static constexpr int SMEM = (USED + 1024) > 118784 ? (USED + 1024) : 118784;  // one CTA per SM
    static constexpr uint32_t C_O = 256;          // S buffers at 0 and 128; O_lo | O_hi at 256
    static constexpr uint32_t TMEM_COLS = 512;
};

// barriers: Q loaded, stage full[2], stage empty[2], S ready[2], S done[2], O ready
enum { F_Q = 0, F_FULL = 1, F_EMPTY = 3, F_SF = 5, F_SD = 7, F_ACC = 9 };

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tm_pk, bf16* __restrict__ o_lo, bf16* __restrict__ o_hi,
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
    const int total = 2 * nk;                      // pass 1 tiles, then pass 2 tiles

    if (threadIdx.x == 0) {
        mbar_init(sy.bar(F_Q), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(sy.bar(F_FULL + s), 1);
            mbar_init(sy.bar(F_EMPTY + s), 1);
            mbar_init(sy.bar(F_SF + s), 1);
            mbar_init(sy.bar(F_SD + s), 128);
        }
        mbar_init(sy.bar(F_ACC), 1);
        *sy.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_pk);
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
            int last[2] = {-1, -1};
            mbar_arrive_expect_tx(sy.bar(F_Q), C::TILE);
            tma_load_3d(sb + C::OFF_Q, &tm_pk, 0, q0, bh * 4 + 0, sy.bar(F_Q));
            for (int it = 0; it < total; ++it) {
                const int s = it & 1, j = it < nk ? it : it - nk;
                const bool pass2 = it >= nk;
                if (!wait_bounded(sy, sy.bar(F_EMPTY + s), ((it >> 1) & 1) ^ 1, 0, it)) break;
                const uint32_t st = sb + C::OFF_STAGE + s * C::STAGE;
                mbar_arrive_expect_tx(sy.bar(F_FULL + s), (pass2 ? 3 : 1) * C::TILE);
                tma_load_3d(st, &tm_pk, 0, j * C::BK, bh * 4 + 1, sy.bar(F_FULL + s));
                if (pass2) {
                    tma_load_3d(st + C::TILE, &tm_pk, 0, j * C::BK, bh * 4 + 2, sy.bar(F_FULL + s));
                    tma_load_3d(st + 2 * C::TILE, &tm_pk, 0, j * C::BK, bh * 4 + 3, sy.bar(F_FULL + s));
                }
                last[s] = it;
            }
            if (*sy.abort) {
                wait_drain(sy.bar(F_Q), 0);
                for (int s = 0; s < 2; ++s)
                    if (last[s] >= 0) wait_drain(sy.bar(F_FULL + s), (last[s] >> 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t ID_O = idesc_bf16(128, 2 * D, 0, 1);   // A = P (TMEM), B = [V_lo | V_hi] MN-major
            constexpr uint32_t SBO = 8 * C::ROWB;
            constexpr uint32_t KSTEP = (16 * C::ROWB) >> 4;
            const uint64_t dQ = smem_desc(sb + C::OFF_Q, 16, SBO, C::SW);
            const uint64_t dStage0 = smem_desc(sb + C::OFF_STAGE, 16, SBO, C::SW);
            const uint64_t dV0 = smem_desc(sb + C::OFF_STAGE + C::TILE, C::TILE, SBO, C::SW);
            constexpr uint32_t STAGE_U = C::STAGE >> 4;
            auto issue_s = [&](int it) -> bool {
                const int s = it & 1;
                if (!wait_bounded(sy, sy.bar(F_FULL + s), (it >> 1) & 1, 1, it)) return false;
                tc_fence_after();
                const uint64_t dK = dStage0 + STAGE_U * s;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_ss(tmem + 128u * s, dQ + 2 * kk, dK + 2 * kk, ID_S, kk);
                mma_commit(sy.bar(F_SF + s));
                if (it < nk) mma_commit(sy.bar(F_EMPTY + s));    // pass 1: the stage held only K
                return true;
            };
            bool ok = wait_bounded(sy, sy.bar(F_Q), 0, 1, -1);
            if (ok) ok = issue_s(0);
            if (ok && total > 1) ok = issue_s(1);
            for (int it = 0; it < total && ok; ++it) {
                const int s = it & 1;
                // softmax is done with S buffer s (pass 1: statistics read; pass 2: P written)
                ok = wait_bounded(sy, sy.bar(F_SD + s), (it >> 1) & 1, 1, it);
                if (!ok) break;
                tc_fence_after();
                if (it >= nk) {
                    const uint64_t dV = dV0 + STAGE_U * s;
#pragma unroll
                    for (int kk = 0; kk < C::BK / 16; ++kk)
                        mma_bf16_ts(tmem + C::C_O, tmem + 128u * s + 8 * kk, dV + KSTEP * kk, ID_O,
                                    (it > nk || kk > 0) ? 1u : 0u);
                    mma_commit(sy.bar(F_EMPTY + s));
                }
                if (it + 2 < total) ok = issue_s(it + 2);
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
        float m = -INFINITY, l = 0.f, L2 = 0.f;   // log2-domain running max and sum; then LSE * log2(e)
        bool ok = true;
        for (int it = 0; it < total; ++it) {
            const int s = it & 1, j = it < nk ? it : it - nk;
            ok = warp_wait(sy, sy.bar(F_SF + s), (it >> 1) & 1, 2, it);
            if (!ok) break;
            tc_fence_after();
            const int nvalid = N - j * C::BK;      // keys of this tile that exist (>= 1)
            const uint32_t tS = trow + 128u * s;
            if (it == nk) L2 = m + __log2f(l);
#pragma unroll 1
            for (int c = 0; c < C::BK / 32; ++c) {
                uint32_t sr[32];
                tmem_ld_32x32b_x32(tS + 32 * c, sr);
                tmem_wait_ld();
                if (it < nk) {
                    float mt = m;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (32 * c + e < nvalid) mt = fmaxf(mt, __uint_as_float(sr[e]) * scale_log2);
                    l *= ex2_approx(m - mt);
                    m = mt;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (32 * c + e < nvalid) l += ex2_approx(fmaf(__uint_as_float(sr[e]), scale_log2, -m));
                } else {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float p0 = ex2_approx(fmaf(__uint_as_float(sr[e]), scale_log2, -L2));
                        float p1 = ex2_approx(fmaf(__uint_as_float(sr[e + 1]), scale_log2, -L2));
                        if (32 * c + e >= nvalid) p0 = 0.f;
                        if (32 * c + e + 1 >= nvalid) p1 = 0.f;
                        pk[e / 2] = pack_bf16x2(p0, p1);
                    }
                    // P over the S columns already read
                    tmem_st_32x32b_x16(tS + 16 * c, pk);
                }
            }
            if (it >= nk) tmem_wait_st();
            tc_fence_before();
            mbar_arrive(sy.bar(F_SD + s));
        }
        if (ok && total == nk) L2 = m + __log2f(l);
        if (ok) ok = warp_wait(sy, sy.bar(F_ACC), 0, 2, total);
        if (ok) {
            // TMEM loads are warp-collective (.sync.aligned): every lane loads,
            // only rows that exist are stored
            tc_fence_after();
            const int i = q0 + il;
            const bool valid = i < N;
            const size_t row = (size_t)bh * N + (valid ? i : 0);
            if (valid) lse[row] = L2 * kLn2;
            uint32_t v[D];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                tmem_ld_row<D>(trow + C::C_O + h * D, v);
                tmem_wait_ld();
                if (valid) {
                    bf16* o = (h == 0 ? o_lo : o_hi) + row * D;
#pragma unroll
                    for (int e = 0; e < D; e += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(v[e + 0]), __uint_as_float(v[e + 1]));
                        w.y = pack_bf16x2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
                        w.z = pack_bf16x2(__uint_as_float(v[e + 4]), __uint_as_float(v[e + 5]));
                        w.w = pack_bf16x2(__uint_as_float(v[e + 6]), __uint_as_float(v[e + 7]));
                        *reinterpret_cast<uint4*>(o + e) = w;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fwd(std::string* err) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    static cudaError_t st = cudaSuccess;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        st = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (st == cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!fn) *err = std::string("cuTensorMapEncodeTiled unavailable: ") + cudaGetErrorString(st);
    return fn;
}

template <int D>
int launch_fwd(const void* packed, void* o_lo, void* o_hi, float* lse, long long BH, int N, float scale,
               cudaStream_t stream, std::string* err) {
    using C = FwdCfg<D>;
    auto enc = get_encode_fwd(err);
    if (!enc) return PSA_ERR_CUDA;
    CUtensorMap tm;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)(BH * 4)};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
    const cuuint32_t box[3] = {(cuuint32_t)D, 128u, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUtensorMapSwizzle sw = D == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : D == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_32B;
    const CUresult r = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(packed), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")";
        return PSA_ERR_CUDA;
    }
    static std::once_flag attr_once;
    static cudaError_t attr_st = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_st = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    });
    if (attr_st != cudaSuccess) {
        *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(attr_st);
        return PSA_ERR_CUDA;
    }
    const int nqt = (N + C::BQ - 1) / C::BQ;
    const long long grid = BH * nqt;
    if (grid > 0x7fffffffll) {
        *err = "grid too large";
        return PSA_ERR_UNSUPPORTED;
    }
    {
        ProfScope prof(kSlotFwd, stream);
        fwd_kernel<D><<<(unsigned)grid, kFwdThreads, C::SMEM, stream>>>(
            tm, static_cast<bf16*>(o_lo), static_cast<bf16*>(o_hi), lse, N, nqt, scale * kLog2e);
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
