// tc_tmap.cu -- TMA tensor-map encoding (driver entry point looked up once).
#include "tc_tmap.h"

#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <set>
#include <utility>

namespace psa {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder(std::string* err) {
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

__device__ unsigned g_smem_base;

// Writes the shared-window address of its dynamic shared memory.
__global__ void smem_base_probe_kernel() {
    extern __shared__ __align__(16) unsigned char dyn[];
    if (threadIdx.x == 0) {
        unsigned a;
        asm volatile("{ .reg .u64 p; cvta.to.shared.u64 p, %1; cvt.u32.u64 %0, p; }" : "=r"(a) : "l"(dyn));
        g_smem_base = a;
    }
}

}  // namespace

static bool encode_rows(CUtensorMap* map, CUtensorMapDataType type, int esize, const void* base, int D, int N, long long Z,
                 int rows, int cols, std::string* err, long long ld = 0) {
    auto enc = encoder(err);
    if (!enc) return false;
    if (ld == 0) ld = D;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)Z};
    const cuuint64_t strides[2] = {(cuuint64_t)ld * esize, (cuuint64_t)N * ld * esize};
    const cuuint32_t box[3] = {(cuuint32_t)cols, (cuuint32_t)rows, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const int rowb = cols * esize;
    const CUtensorMapSwizzle sw = rowb == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : rowb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
    const CUresult r = enc(map, type, 3, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")";
        return false;
    }
    return true;
}

bool encode_bf16_rows(CUtensorMap* map, const void* base, int D, int N, long long Z, int rows, int cols,
                      std::string* err) {
    return encode_rows(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, D, N, Z, rows, cols, err);
}

bool encode_f32_rows(CUtensorMap* map, const void* base, int D, int N, long long Z, int rows, int cols,
                     std::string* err) {
    return encode_rows(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, D, N, Z, rows, cols, err);
}

bool encode_bf16_rows_ld(CUtensorMap* map, const void* base, int D, long long ld, int N, long long Z, int rows,
                         int cols, std::string* err) {
    return encode_rows(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, D, N, Z, rows, cols, err, ld);
}

bool encode_bf16_4d(CUtensorMap* map, const void* base, long long inner, long long outer, long long heads,
                    long long B, long long s_outer, long long s_head, long long s_batch, int box_inner,
                    int box_outer, std::string* err) {
    auto enc = encoder(err);
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)heads, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)s_outer * 2, (cuuint64_t)s_head * 2, (cuuint64_t)s_batch * 2};
    const cuuint32_t box[4] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer, 1u, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const int rowb = box_inner * 2;
    const CUtensorMapSwizzle sw = rowb == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : rowb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled (4-d) failed (" + std::to_string((int)r) + ")";
        return false;
    }
    return true;
}

bool set_max_dynamic_smem(const void* kernel, int bytes, std::string* err) {
    static std::mutex mu;
    static std::set<std::pair<int, const void*>> done;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return false;
    }
    std::lock_guard<std::mutex> g(mu);
    if (done.count({dev, kernel})) return true;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) {
        *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
        return false;
    }
    done.insert({dev, kernel});
    return true;
}

}  // namespace psa

namespace psa {

int dyn_smem_base_aligned(std::string* err) {
    static std::mutex mu;
    static std::map<int, int> known;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
        return -1;
    }
    std::lock_guard<std::mutex> g(mu);
    auto it = known.find(dev);
    if (it != known.end()) return it->second;
    // a private stream, and this thread's capture mode relaxed for the probe, so
    // that a first call made while the caller's stream is being captured works
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    cudaStream_t st = nullptr;
    unsigned base = 1;
    e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e == cudaSuccess) {
        smem_base_probe_kernel<<<1, 32, 1024, st>>>();
        e = cudaGetLastError();
        if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(&base, g_smem_base, sizeof(base), 0, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        cudaStreamDestroy(st);
    }
    cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) {
        *err = std::string("shared memory base probe: ") + cudaGetErrorString(e);
        return -1;
    }
    const int ok = (base & 1023u) == 0 ? 1 : 0;
    known[dev] = ok;
    return ok;
}

}  // namespace psa
