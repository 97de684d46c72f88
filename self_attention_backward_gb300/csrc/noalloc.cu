// noalloc.cu -- psa_attn_bwd_noalloc: the CUDA-core backward without a
// caller-supplied workspace.
//
// The only scratch the CUDA-core backward needs is the per-query row statistic
// D_i = <dO_lo[i], O_lo[i]> + <dO_hi[i], O_hi[i]> (fp32, one value per query
// row).  Here it lives in a fixed-size array in the library's own device
// memory, so the call itself allocates nothing.  That array exists once per
// GPU that loads this library and stays resident until the process exits.
#include <cmath>
#include <map>
#include <mutex>
#include <string>

#include "psa_attn.h"
#include "psa_internal.h"
#include "simt_kernels.cuh"

namespace {

// Capacity of the static scratch, in query rows (B * heads * N): 2 MiB of fp32.
constexpr long long kNoallocMaxRows = 1ll << 19;

static __device__ __align__(256) float g_noalloc_scratch[kNoallocMaxRows];

// Device address of g_noalloc_scratch, looked up once per device.  In host
// code the symbol name is only a host-side handle, never a device address.
std::mutex g_scratch_mu;
std::map<int, float*> g_scratch_ptr;

int scratch_for_current_device(float** out, std::string* err) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return PSA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> g(g_scratch_mu);
    auto it = g_scratch_ptr.find(dev);
    if (it == g_scratch_ptr.end()) {
        float* p = nullptr;
        e = cudaGetSymbolAddress((void**)&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            *err = std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e);
            return PSA_ERR_CUDA;
        }
        it = g_scratch_ptr.emplace(dev, p).first;
    }
    *out = it->second;
    return PSA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T, int D>
int launch(const void* packed, const void* o_lo, const void* o_hi, const float* lse, const void* do_lo,
           const void* do_hi, void* d_packed, float* Drow, long long BH, int N, float scale, cudaStream_t st) {
    using namespace psa::simt;
    const long long rows = BH * N;
    const long long pre_grid = (rows + kThreads / 32 - 1) / (kThreads / 32);
    const int ntiles = (N + kRows - 1) / kRows;
    const long long grid = BH * ntiles;
    // D is fully rewritten by pre_kernel before it is read, so nothing left in
    // the scratch by an earlier call needs clearing.
    pre_kernel<T, D><<<(unsigned)pre_grid, kThreads, 0, st>>>((const T*)o_lo, (const T*)o_hi, (const T*)do_lo,
                                                             (const T*)do_hi, Drow, rows);
    dkdv_kernel<T, D><<<(unsigned)grid, kThreads, 0, st>>>((const T*)packed, (const T*)do_lo, (const T*)do_hi, lse,
                                                          Drow, (T*)d_packed, N, ntiles, scale, scale * psa::kLog2e);
    dq_kernel<T, D><<<(unsigned)grid, kThreads, 0, st>>>((const T*)packed, (const T*)do_lo, (const T*)do_hi, lse,
                                                        Drow, (T*)d_packed, N, ntiles, scale, scale * psa::kLog2e);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return psa::set_last_error(PSA_ERR_CUDA, std::string("psa_attn_bwd_noalloc launch: ") + cudaGetErrorString(e));
    return PSA_OK;
}

}  // namespace

extern "C" long long psa_attn_bwd_noalloc_max_rows(void) { return kNoallocMaxRows; }

extern "C" int psa_attn_bwd_noalloc(const void* packed, const void* o_lo, const void* o_hi, const float* lse,
                                    const void* do_lo, const void* do_hi, void* d_packed, int B, int heads, int N,
                                    int head_dim, float scale, int dtype, void* stream) {
    if (dtype != PSA_F32 && dtype != PSA_BF16) return psa::set_last_error(PSA_ERR_ARG, "dtype is not PSA_F32 or PSA_BF16");
    if (B < 0 || heads < 0 || N < 0) return psa::set_last_error(PSA_ERR_ARG, "negative size");
    if (head_dim != 16 && head_dim != 32 && head_dim != 64)
        return psa::set_last_error(PSA_ERR_UNSUPPORTED, "head_dim not in {16, 32, 64}");
    if (!std::isfinite(scale)) return psa::set_last_error(PSA_ERR_ARG, "scale is not finite");
    const long long BH = (long long)B * heads;
    if (BH == 0 || N == 0) return psa::set_last_error(PSA_OK, "");
    if (BH * (long long)N > kNoallocMaxRows)
        return psa::set_last_error(PSA_ERR_UNSUPPORTED,
                                   "psa_attn_bwd_noalloc: B*heads*N = " + std::to_string(BH * (long long)N) +
                                       " exceeds its static scratch of " + std::to_string(kNoallocMaxRows) +
                                       " rows; use psa_attn_bwd with a caller-allocated workspace");
    const void* ptrs[] = {packed, o_lo, o_hi, lse, do_lo, do_hi, d_packed};
    for (const void* p : ptrs) {
        if (!p) return psa::set_last_error(PSA_ERR_ARG, "psa_attn_bwd_noalloc: NULL tensor pointer");
        if (!aligned16(p)) return psa::set_last_error(PSA_ERR_ALIGN, "psa_attn_bwd_noalloc: pointer not 16-byte aligned");
    }
    float* Drow = nullptr;
    std::string err;
    int rc = scratch_for_current_device(&Drow, &err);
    if (rc) return psa::set_last_error(rc, err);
    const cudaStream_t st = (cudaStream_t)stream;
    if (dtype == PSA_F32) {
        rc = head_dim == 16   ? launch<float, 16>(packed, o_lo, o_hi, lse, do_lo, do_hi, d_packed, Drow, BH, N, scale, st)
             : head_dim == 32 ? launch<float, 32>(packed, o_lo, o_hi, lse, do_lo, do_hi, d_packed, Drow, BH, N, scale, st)
                              : launch<float, 64>(packed, o_lo, o_hi, lse, do_lo, do_hi, d_packed, Drow, BH, N, scale, st);
    } else {
        using bf = __nv_bfloat16;
        rc = head_dim == 16   ? launch<bf, 16>(packed, o_lo, o_hi, lse, do_lo, do_hi, d_packed, Drow, BH, N, scale, st)
             : head_dim == 32 ? launch<bf, 32>(packed, o_lo, o_hi, lse, do_lo, do_hi, d_packed, Drow, BH, N, scale, st)
                              : launch<bf, 64>(packed, o_lo, o_hi, lse, do_lo, do_hi, d_packed, Drow, BH, N, scale, st);
    }
    return rc ? rc : psa::set_last_error(PSA_OK, "");
}
