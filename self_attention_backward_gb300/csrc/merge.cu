// merge.cu -- the PSA attention merge's backward ("Struct
// PsaMergeAttnRuntimeOp": d_merged -> d_lo, d_hi) and the strided-view gather
// it is built from.
//
// The merged tensor is [B, c, H, W] with c = 2 * heads * d: the lo outputs of
// every head in the low half of the channels, the hi outputs in the high half,
// head-major in each half (the pages name the backward's arguments -- d_merged,
// d_lo, d_hi, c, H, W, num_heads -- not the order; this is the reading taken).
// So dO_s of slice b*heads + h is the [d, N] channel-major block of channels
// s*heads*d + h*d .. + d - 1 of batch b, and the backward is a transposing
// gather.  The attention backward can also read those blocks in place
// (psa_merge_attn_bwd); this file provides the plain gather for the unfused
// path and for the CUDA-core backward, which takes contiguous dO only.
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "psa_attn.h"
#include "psa_internal.h"

namespace psa {
namespace {

constexpr int kTileN = 64;  // positions per block

// One block per (slice, 64 positions): the tile goes through shared memory so
// that both the strided reads (along whichever of n or j has unit stride) and
// the contiguous [N, d] writes are coalesced.
template <typename T>
__global__ void __launch_bounds__(256)
gather_view_kernel(const T* __restrict__ base, long long sB, long long sH, long long sN, long long sJ,
                   T* __restrict__ dst, int heads, int N, int d, int ntiles) {
    extern __shared__ unsigned char smem_raw[];
    T* tile = reinterpret_cast<T*>(smem_raw);  // [kTileN][d + 1]
    const long long bh = blockIdx.x / ntiles;
    const int n0 = (int)(blockIdx.x % ntiles) * kTileN;
    const long long b = bh / heads, h = bh % heads;
    const T* src = base + b * sB + h * sH;
    const int tot = kTileN * d;
    const bool pos_fast = sN == 1;  // channel-major: consecutive positions are adjacent
    for (int idx = threadIdx.x; idx < tot; idx += blockDim.x) {
        const int n = pos_fast ? idx % kTileN : idx / d;
        const int j = pos_fast ? idx / kTileN : idx % d;
        if (n0 + n < N) tile[n * (d + 1) + j] = src[(long long)(n0 + n) * sN + (long long)j * sJ];
    }
    __syncthreads();
    T* out = dst + ((size_t)bh * N + n0) * d;
    for (int idx = threadIdx.x; idx < tot; idx += blockDim.x) {
        const int n = idx / d, j = idx % d;
        if (n0 + n < N) out[(size_t)n * d + j] = tile[n * (d + 1) + j];
    }
}

}  // namespace

int gather_view_launch(const View& v, void* dst, long long BH, int heads, int N, int d, int esize,
                       cudaStream_t stream, std::string* err) {
    if (BH == 0 || N == 0) return PSA_OK;
    const int ntiles = (N + kTileN - 1) / kTileN;
    const long long grid = BH * ntiles;
    if (grid > 0x7fffffffll) {
        *err = "grid too large";
        return PSA_ERR_UNSUPPORTED;
    }
    const size_t smem = (size_t)kTileN * (d + 1) * esize;
    if (esize == 2)
        gather_view_kernel<uint16_t><<<(unsigned)grid, 256, smem, stream>>>(
            static_cast<const uint16_t*>(v.base), v.sB, v.sH, v.sN, v.sJ, static_cast<uint16_t*>(dst), heads, N, d,
            ntiles);
    else
        gather_view_kernel<float><<<(unsigned)grid, 256, smem, stream>>>(
            static_cast<const float*>(v.base), v.sB, v.sH, v.sN, v.sJ, static_cast<float*>(dst), heads, N, d,
            ntiles);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = std::string("gather launch: ") + cudaGetErrorString(e);
        return PSA_ERR_CUDA;
    }
    return PSA_OK;
}

// The views of dO_lo / dO_hi inside a merged [B, 2*heads*d, N] tensor.
void merged_views(const void* d_merged, int heads, int N, int d, int esize, View* lo, View* hi) {
    const long long c = 2ll * heads * d;
    *lo = View{d_merged, c * N, (long long)d * N, 1, N};
    *hi = View{static_cast<const char*>(d_merged) + (size_t)heads * d * N * esize, c * N, (long long)d * N, 1, N};
}

}  // namespace psa

extern "C" int psa_merge_bwd(const void* d_merged, void* d_lo, void* d_hi, int B, int heads, int H, int W,
                             int head_dim, int dtype, void* stream) {
    if (dtype != PSA_F32 && dtype != PSA_BF16)
        return psa::set_last_error(PSA_ERR_ARG, "dtype is not PSA_F32 or PSA_BF16");
    if (B < 0 || heads < 0 || H < 0 || W < 0 || head_dim <= 0)
        return psa::set_last_error(PSA_ERR_ARG, "negative size or head_dim <= 0");
    if (head_dim > 128) return psa::set_last_error(PSA_ERR_UNSUPPORTED, "head_dim > 128");
    const long long N = (long long)H * W, BH = (long long)B * heads;
    if (N > 0x7fffffffll) return psa::set_last_error(PSA_ERR_UNSUPPORTED, "H*W too large");
    if (BH == 0 || N == 0) return psa::set_last_error(PSA_OK, "");
    if (!d_merged || !d_lo || !d_hi) return psa::set_last_error(PSA_ERR_ARG, "NULL pointer");
    const int esize = dtype == PSA_F32 ? 4 : 2;
    psa::View lo, hi;
    psa::merged_views(d_merged, heads, (int)N, head_dim, esize, &lo, &hi);
    std::string err;
    int rc = psa::gather_view_launch(lo, d_lo, BH, heads, (int)N, head_dim, esize, (cudaStream_t)stream, &err);
    if (rc == PSA_OK)
        rc = psa::gather_view_launch(hi, d_hi, BH, heads, (int)N, head_dim, esize, (cudaStream_t)stream, &err);
    return psa::set_last_error(rc, rc ? err : std::string());
}
