// psa_attn.cu -- C-ABI front end: argument checks, kernel choice, launches.
//
// The entry points are declared, with their contracts, in include/psa_attn.h.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "psa_attn.h"
#include "psa_internal.h"
#include "simt_kernels.cuh"

namespace psa {
namespace {
std::atomic<bool> g_prof_on{false};
std::mutex g_prof_mu;
struct ProfRec { int slot; cudaEvent_t a, b; };
std::vector<ProfRec> g_prof;
}  // namespace

bool prof_enabled() { return g_prof_on.load(std::memory_order_relaxed); }

ProfScope::ProfScope(int slot, cudaStream_t st) : slot_(slot), st_(st) {
    if (!g_prof_on.load(std::memory_order_relaxed)) return;
    if (cudaEventCreate(&a_) != cudaSuccess || cudaEventCreate(&b_) != cudaSuccess) {
        if (a_) cudaEventDestroy(a_);
        a_ = b_ = nullptr;
        return;
    }
    cudaEventRecord(a_, st_);
}

ProfScope::~ProfScope() {
    if (!a_) return;
    cudaEventRecord(b_, st_);
    std::lock_guard<std::mutex> g(g_prof_mu);
    g_prof.push_back({slot_, a_, b_});
}
}  // namespace psa

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int ok() {
    g_last_error.clear();
    return PSA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Largest supported problem: every element index of a [BH, 4, N, d] tensor and
// every CTA count fits comfortably in 62 / 31 bits.
constexpr long long kMaxElems = 1ll << 40;

struct Shape {
    long long BH;
    int N, d;
    bool empty;
};

int check_shape(int B, int heads, int N, int head_dim, float scale, int dtype, Shape* s) {
    if (dtype != PSA_F32 && dtype != PSA_BF16) return fail(PSA_ERR_ARG, "dtype %d is not PSA_F32 or PSA_BF16", dtype);
    if (B < 0 || heads < 0 || N < 0) return fail(PSA_ERR_ARG, "negative size (B=%d heads=%d N=%d)", B, heads, N);
    if (head_dim != 16 && head_dim != 32 && head_dim != 64)
        return fail(PSA_ERR_UNSUPPORTED, "head_dim %d not in {16, 32, 64}", head_dim);
    if (!std::isfinite(scale)) return fail(PSA_ERR_ARG, "scale is not finite");
    s->BH = (long long)B * heads;
    s->N = N;
    s->d = head_dim;
    s->empty = s->BH == 0 || N == 0;
    if (!s->empty && s->BH * 4ll * N * head_dim > kMaxElems)
        return fail(PSA_ERR_UNSUPPORTED, "problem too large (BH=%lld N=%d d=%d)", s->BH, N, head_dim);
    return PSA_OK;
}

int check_ptrs(std::initializer_list<std::pair<const char*, const void*>> ptrs) {
    for (auto& p : ptrs) {
        if (!p.second) return fail(PSA_ERR_ARG, "%s is NULL", p.first);
        if (!aligned16(p.second)) return fail(PSA_ERR_ALIGN, "%s is not 16-byte aligned", p.first);
    }
    return PSA_OK;
}

int cuda_check(const char* what) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return PSA_OK;
}

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

template <typename T, int D>
int launch_fwd(const void* packed, void* o_lo, void* o_hi, float* lse, long long BH, int N, float scale,
               cudaStream_t st) {
    const int ntiles = ceil_div(N, psa::simt::kRows);
    const long long grid = BH * ntiles;
    if (grid > 0x7fffffffll) return fail(PSA_ERR_UNSUPPORTED, "grid too large");
    psa::ProfScope prof(psa::kSlotFwd, st);
    psa::simt::fwd_kernel<T, D><<<(unsigned)grid, psa::simt::kThreads, 0, st>>>(
        (const T*)packed, (T*)o_lo, (T*)o_hi, lse, N, ntiles, scale * psa::kLog2e);
    return cuda_check("psa_attn_fwd launch");
}

template <typename T, int D>
int launch_bwd_simt(const psa::BwdArgs& a) {
    using namespace psa::simt;
    const long long rows = a.BH * a.N;
    float* Drow = (float*)a.workspace;
    const long long pre_grid = (rows + kThreads / 32 - 1) / (kThreads / 32);
    const int ntiles = ceil_div(a.N, kRows);
    const long long grid = a.BH * ntiles;
    if (grid > 0x7fffffffll || pre_grid > 0x7fffffffll) return fail(PSA_ERR_UNSUPPORTED, "grid too large");
    {
        psa::ProfScope prof(psa::kSlotPre, a.stream);
        pre_kernel<T, D><<<(unsigned)pre_grid, kThreads, 0, a.stream>>>(
            (const T*)a.o_lo, (const T*)a.o_hi, (const T*)a.do_lo, (const T*)a.do_hi, Drow, rows);
    }
    {
        psa::ProfScope prof(psa::kSlotMain, a.stream);
        dkdv_kernel<T, D><<<(unsigned)grid, kThreads, 0, a.stream>>>(
            (const T*)a.packed, (const T*)a.do_lo, (const T*)a.do_hi, a.lse, Drow, (T*)a.d_packed, a.N, ntiles,
            a.scale, a.scale * psa::kLog2e);
    }
    {
        psa::ProfScope prof(psa::kSlotDq, a.stream);
        dq_kernel<T, D><<<(unsigned)grid, kThreads, 0, a.stream>>>(
            (const T*)a.packed, (const T*)a.do_lo, (const T*)a.do_hi, a.lse, Drow, (T*)a.d_packed, a.N, ntiles,
            a.scale, a.scale * psa::kLog2e);
    }
    return cuda_check("psa_attn_bwd (simt) launch");
}

size_t simt_workspace_bytes(long long BH, int N) { return (size_t)BH * (size_t)N * sizeof(float); }

#define PSA_DISPATCH(dtype, d, FN, ...)                                                          \
    ((dtype) == PSA_F32                                                                          \
         ? ((d) == 16 ? FN<float, 16>(__VA_ARGS__)                                               \
                      : (d) == 32 ? FN<float, 32>(__VA_ARGS__) : FN<float, 64>(__VA_ARGS__))     \
         : ((d) == 16 ? FN<__nv_bfloat16, 16>(__VA_ARGS__)                                       \
                      : (d) == 32 ? FN<__nv_bfloat16, 32>(__VA_ARGS__)                           \
                                  : FN<__nv_bfloat16, 64>(__VA_ARGS__)))

bool is_bwd_algo(int algo) {
    return algo == PSA_ALGO_AUTO || algo == PSA_ALGO_SIMT || algo == PSA_ALGO_TC || algo == PSA_ALGO_TC_2PASS;
}

int resolve_algo(int dtype, int d, int algo) {
    if (algo == PSA_ALGO_AUTO) return psa::tc_supported(dtype, d) ? PSA_ALGO_TC : PSA_ALGO_SIMT;
    return algo;
}

size_t workspace_for(const Shape& s, int dtype, int algo) {
    if (s.empty) return 0;
    algo = resolve_algo(dtype, s.d, algo);
    if (algo == PSA_ALGO_SIMT) return simt_workspace_bytes(s.BH, s.N);
    if (algo == PSA_ALGO_TC && psa::tc_supported(dtype, s.d)) return psa::tc_workspace_bytes(s.BH, s.N, s.d);
    if (algo == PSA_ALGO_TC_2PASS && psa::tc_supported(dtype, s.d)) return psa::tc_two_pass_workspace_bytes(s.BH, s.N);
    return 0;
}

bool view_contiguous(const psa::View& v, int heads, int N, int d) {
    return v.sJ == 1 && v.sN == d && v.sH == (long long)N * d && v.sB == (long long)heads * N * d;
}

// Checks a dO view: aligned base, row-major (sJ = 1, sN >= d) or channel-major
// (sN = 1, sJ >= N), non-negative strides; with `tma`, every non-unit stride a
// multiple of 16 bytes.
int check_view(const char* name, const psa_attn_view* v, int N, int d, int esize, bool tma) {
    if (!v || !v->base) return fail(PSA_ERR_ARG, "%s view is NULL", name);
    if (!aligned16(v->base)) return fail(PSA_ERR_ALIGN, "%s view base is not 16-byte aligned", name);
    if (v->batch_stride < 0 || v->head_stride < 0 || v->pos_stride < 0 || v->feat_stride < 0)
        return fail(PSA_ERR_ARG, "%s view has a negative stride", name);
    const bool rows = v->feat_stride == 1 && v->pos_stride >= d;
    const bool chans = v->pos_stride == 1 && v->feat_stride >= N && !rows;
    if (!rows && !chans)
        return fail(PSA_ERR_UNSUPPORTED, "%s view is neither row-major (feat_stride 1, pos_stride >= d) nor "
                    "channel-major (pos_stride 1, feat_stride >= N)", name);
    if (tma) {
        const long long outer = rows ? v->pos_stride : v->feat_stride;
        for (long long st : {outer, v->head_stride, v->batch_stride})
            if ((st * esize) % 16 != 0)
                return fail(PSA_ERR_ALIGN, "%s view: strides must be multiples of 16 bytes on the tensor-core path",
                            name);
    }
    return PSA_OK;
}

psa::View to_view(const psa_attn_view* v) {
    return psa::View{v->base, v->batch_stride, v->head_stride, v->pos_stride, v->feat_stride};
}

// Workspace of psa_attn_bwd_ex: the kernel family's own, then (CUDA-core path
// with non-contiguous dO) room for the gathered dO_lo and dO_hi.
size_t ex_workspace(const Shape& s, int heads, int dtype, int algo, bool gather) {
    if (s.empty) return 0;
    algo = resolve_algo(dtype, s.d, algo);
    size_t w = (workspace_for(s, dtype, algo) + 255) & ~size_t(255);
    if (algo == PSA_ALGO_SIMT && gather)
        w += 2 * (((size_t)s.BH * s.N * s.d * (dtype == PSA_F32 ? 4 : 2) + 255) & ~size_t(255));
    (void)heads;
    return w;
}

// psa_attn_bwd_ex with views already built (also behind psa_merge_attn_bwd).
int bwd_ex(const void* packed, long long ldq, const void* o_lo, const void* o_hi, long long ldo, const float* lse,
           const psa_attn_view* do_lo, const psa_attn_view* do_hi, void* d_packed, void* workspace,
           size_t workspace_bytes, int B, int heads, int N, int head_dim, float scale, int dtype, int algo,
           void* stream) {
    Shape s;
    int rc = check_shape(B, heads, N, head_dim, scale, dtype, &s);
    if (rc) return rc;
    if (!is_bwd_algo(algo)) return fail(PSA_ERR_ARG, "algo %d is not a psa_algo", algo);
    algo = resolve_algo(dtype, head_dim, algo);
    if (algo == PSA_ALGO_TC_2PASS)
        return fail(PSA_ERR_UNSUPPORTED, "the two-pass mode takes contiguous tensors (psa_attn_bwd_algo)");
    if (algo == PSA_ALGO_TC && !psa::tc_supported(dtype, head_dim))
        return fail(PSA_ERR_UNSUPPORTED, "no tensor-core backward for dtype %d, head_dim %d", dtype, head_dim);
    const bool tc = algo == PSA_ALGO_TC;
    const int esize = dtype == PSA_F32 ? 4 : 2;
    if (ldq < head_dim || ldo < head_dim)
        return fail(PSA_ERR_ARG, "row strides must be >= head_dim (qkv %lld, o %lld)", ldq, ldo);
    if (tc && ((ldq * esize) % 16 || (ldo * esize) % 16))
        return fail(PSA_ERR_ALIGN, "row strides must be multiples of 16 bytes on the tensor-core path");
    if (!tc && (ldq != head_dim || ldo != head_dim))
        return fail(PSA_ERR_UNSUPPORTED, "the CUDA-core path takes packed and O rows of head_dim elements");
    if (s.empty) return ok();
    rc = check_view("do_lo", do_lo, N, head_dim, esize, tc);
    if (!rc) rc = check_view("do_hi", do_hi, N, head_dim, esize, tc);
    if (rc) return rc;
    if ((do_lo->pos_stride == 1) != (do_hi->pos_stride == 1))
        return fail(PSA_ERR_UNSUPPORTED, "do_lo and do_hi must both be row-major or both channel-major");
    rc = check_ptrs({{"packed", packed}, {"o_lo", o_lo}, {"o_hi", o_hi}, {"lse", lse}, {"d_packed", d_packed}});
    if (rc) return rc;
    const psa::View vlo = to_view(do_lo), vhi = to_view(do_hi);
    const bool gather = !view_contiguous(vlo, heads, N, head_dim) || !view_contiguous(vhi, heads, N, head_dim);
    const size_t need = ex_workspace(s, heads, dtype, algo, gather);
    if (workspace_bytes < need) return fail(PSA_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
    if (need > 0) {
        rc = check_ptrs({{"workspace", workspace}});
        if (rc) return rc == PSA_ERR_ARG ? fail(PSA_ERR_WORKSPACE, "workspace is NULL") : rc;
    }
    psa::BwdArgs a{packed, o_lo, o_hi, lse, vlo.base, vhi.base, d_packed, workspace, workspace_bytes,
                   s.BH, N, head_dim, scale, dtype, (cudaStream_t)stream};
    a.heads = heads;
    a.ld_qkv = ldq;
    a.ld_o = ldo;
    a.views = true;
    a.vlo = vlo;
    a.vhi = vhi;
    std::string err;
    if (tc) {
        rc = psa::tc_bwd_launch(a, &err);
        return rc ? fail(rc, "%s", err.c_str()) : ok();
    }
    // CUDA-core path: contiguous dO, gathered into the workspace when needed
    if (gather) {
        const size_t base = (workspace_for(s, dtype, algo) + 255) & ~size_t(255);
        const size_t one = ((size_t)s.BH * N * head_dim * esize + 255) & ~size_t(255);
        char* g = static_cast<char*>(workspace) + base;
        rc = psa::gather_view_launch(vlo, g, s.BH, heads, N, head_dim, esize, (cudaStream_t)stream, &err);
        if (!rc) rc = psa::gather_view_launch(vhi, g + one, s.BH, heads, N, head_dim, esize, (cudaStream_t)stream, &err);
        if (rc) return fail(rc, "%s", err.c_str());
        a.do_lo = g;
        a.do_hi = g + one;
    }
    a.views = false;
    rc = PSA_DISPATCH(dtype, head_dim, launch_bwd_simt, a);
    return rc ? rc : ok();
}

}  // namespace

int psa::set_last_error(int code, const std::string& msg) {
    g_last_error = msg;
    return code;
}

extern "C" {

int psa_attn_version(void) { return 100; }

const char* psa_attn_last_error(void) { return g_last_error.c_str(); }

int psa_attn_fwd_algo(const void* packed, void* o_lo, void* o_hi, float* lse, int B, int heads, int N,
                      int head_dim, float scale, int dtype, int algo, void* stream) {
    Shape s;
    int rc = check_shape(B, heads, N, head_dim, scale, dtype, &s);
    if (rc) return rc;
    if (algo != PSA_ALGO_AUTO && algo != PSA_ALGO_SIMT && algo != PSA_ALGO_TC)
        return fail(PSA_ERR_ARG, "algo %d is not a psa_algo", algo);
    if (algo == PSA_ALGO_AUTO) algo = psa::tc_fwd_supported(dtype, head_dim) ? PSA_ALGO_TC : PSA_ALGO_SIMT;
    if (algo == PSA_ALGO_TC && !psa::tc_fwd_supported(dtype, head_dim))
        return fail(PSA_ERR_UNSUPPORTED, "no tensor-core forward for dtype %d, head_dim %d", dtype, head_dim);
    if (s.empty) return ok();
    rc = check_ptrs({{"packed", packed}, {"o_lo", o_lo}, {"o_hi", o_hi}, {"lse", lse}});
    if (rc) return rc;
    if (algo == PSA_ALGO_TC) {
        std::string err;
        rc = psa::tc_fwd_launch(packed, o_lo, o_hi, lse, s.BH, N, head_dim, scale, (cudaStream_t)stream, &err);
        return rc ? fail(rc, "%s", err.c_str()) : ok();
    }
    rc = PSA_DISPATCH(dtype, head_dim, launch_fwd, packed, o_lo, o_hi, lse, s.BH, N, scale, (cudaStream_t)stream);
    return rc ? rc : ok();
}

int psa_attn_fwd(const void* packed, void* o_lo, void* o_hi, float* lse, int B, int heads, int N, int head_dim,
                 float scale, int dtype, void* stream) {
    return psa_attn_fwd_algo(packed, o_lo, o_hi, lse, B, heads, N, head_dim, scale, dtype, PSA_ALGO_AUTO, stream);
}

size_t psa_attn_bwd_workspace_bytes_algo(int B, int heads, int N, int head_dim, int dtype, int algo) {
    Shape s;
    const std::string keep = g_last_error;
    const int rc = check_shape(B, heads, N, head_dim, 1.0f, dtype, &s);
    g_last_error = keep;
    if (rc) return 0;
    if (!is_bwd_algo(algo)) return 0;
    return workspace_for(s, dtype, algo);
}

size_t psa_attn_bwd_workspace_bytes(int B, int heads, int N, int head_dim, int dtype) {
    return psa_attn_bwd_workspace_bytes_algo(B, heads, N, head_dim, dtype, PSA_ALGO_AUTO);
}

int psa_attn_bwd_algo(const void* packed, const void* o_lo, const void* o_hi, const float* lse, const void* do_lo,
                      const void* do_hi, void* d_packed, void* workspace, size_t workspace_bytes, int B, int heads,
                      int N, int head_dim, float scale, int dtype, int algo, void* stream) {
    Shape s;
    int rc = check_shape(B, heads, N, head_dim, scale, dtype, &s);
    if (rc) return rc;
    if (!is_bwd_algo(algo)) return fail(PSA_ERR_ARG, "algo %d is not a psa_algo", algo);
    algo = resolve_algo(dtype, head_dim, algo);
    if ((algo == PSA_ALGO_TC || algo == PSA_ALGO_TC_2PASS) && !psa::tc_supported(dtype, head_dim))
        return fail(PSA_ERR_UNSUPPORTED, "no tensor-core backward for dtype %d, head_dim %d", dtype, head_dim);
    if (s.empty) return ok();
    rc = check_ptrs({{"packed", packed}, {"o_lo", o_lo}, {"o_hi", o_hi}, {"lse", lse}, {"do_lo", do_lo},
                     {"do_hi", do_hi}, {"d_packed", d_packed}});
    if (rc) return rc;
    const size_t need = workspace_for(s, dtype, algo);
    if (workspace_bytes < need) return fail(PSA_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
    if (need > 0) {
        rc = check_ptrs({{"workspace", workspace}});
        if (rc) return rc == PSA_ERR_ARG ? fail(PSA_ERR_WORKSPACE, "workspace is NULL") : rc;
    }
    psa::BwdArgs a{packed, o_lo, o_hi, lse, do_lo, do_hi, d_packed, workspace, workspace_bytes,
                   s.BH, N, head_dim, scale, dtype, (cudaStream_t)stream};
    if (algo == PSA_ALGO_TC || algo == PSA_ALGO_TC_2PASS) {
        std::string err;
        if (algo == PSA_ALGO_TC)
            rc = psa::tc_bwd_launch(a, &err);
        else if (psa::tc_pair_supported(dtype, head_dim) && std::fabs(scale) >= 1e-30f)
            rc = psa::tc_pair_launch(a, &err);   // folds -LSE/scale into its MMAs: needs scale != 0
        else
            rc = psa::tc_two_pass_launch(a, &err);
        if (rc) return fail(rc, "%s", err.c_str());
        return ok();
    }
    rc = PSA_DISPATCH(dtype, head_dim, launch_bwd_simt, a);
    return rc ? rc : ok();
}

int psa_attn_bwd(const void* packed, const void* o_lo, const void* o_hi, const float* lse, const void* do_lo,
                 const void* do_hi, void* d_packed, void* workspace, size_t workspace_bytes, int B, int heads, int N,
                 int head_dim, float scale, int dtype, void* stream) {
    return psa_attn_bwd_algo(packed, o_lo, o_hi, lse, do_lo, do_hi, d_packed, workspace, workspace_bytes, B, heads,
                             N, head_dim, scale, dtype, PSA_ALGO_AUTO, stream);
}

int psa_attn_bwd_ex(const void* packed, long long qkv_row_stride, const void* o_lo, const void* o_hi,
                    long long o_row_stride, const float* lse, const psa_attn_view* do_lo,
                    const psa_attn_view* do_hi, void* d_packed, void* workspace, size_t workspace_bytes, int B,
                    int heads, int N, int head_dim, float scale, int dtype, int algo, void* stream) {
    return bwd_ex(packed, qkv_row_stride, o_lo, o_hi, o_row_stride, lse, do_lo, do_hi, d_packed, workspace,
                  workspace_bytes, B, heads, N, head_dim, scale, dtype, algo, stream);
}

size_t psa_attn_bwd_ex_workspace_bytes(const psa_attn_view* do_lo, const psa_attn_view* do_hi, int B, int heads,
                                       int N, int head_dim, int dtype, int algo) {
    Shape s;
    const std::string keep = g_last_error;
    const int rc = check_shape(B, heads, N, head_dim, 1.0f, dtype, &s);
    g_last_error = keep;
    if (rc || !is_bwd_algo(algo) || !do_lo || !do_hi) return 0;
    const bool gather = !view_contiguous(to_view(do_lo), heads, N, head_dim) ||
                        !view_contiguous(to_view(do_hi), heads, N, head_dim);
    return ex_workspace(s, heads, dtype, algo, gather);
}

size_t psa_merge_attn_bwd_workspace_bytes(int B, int heads, int H, int W, int head_dim, int dtype, int algo) {
    if ((long long)H * W > 0x7fffffffll || H < 0 || W < 0) return 0;
    Shape s;
    const std::string keep = g_last_error;
    const int rc = check_shape(B, heads, H * W, head_dim, 1.0f, dtype, &s);
    g_last_error = keep;
    if (rc || !is_bwd_algo(algo)) return 0;
    return ex_workspace(s, heads, dtype, algo, true);
}

int psa_merge_attn_bwd(const void* packed, const void* o_lo, const void* o_hi, const float* lse,
                       const void* d_merged, void* d_packed, void* workspace, size_t workspace_bytes, int B,
                       int heads, int H, int W, int head_dim, float scale, int dtype, int algo, void* stream) {
    if (H < 0 || W < 0 || (long long)H * W > 0x7fffffffll) return fail(PSA_ERR_ARG, "bad H, W (%d, %d)", H, W);
    if (!d_merged && B > 0 && heads > 0 && H > 0 && W > 0) return fail(PSA_ERR_ARG, "d_merged is NULL");
    const int N = H * W;
    psa::View lo{}, hi{};
    if (d_merged) psa::merged_views(d_merged, heads, N, head_dim, dtype == PSA_F32 ? 4 : 2, &lo, &hi);
    const psa_attn_view vlo{lo.base, lo.sB, lo.sH, lo.sN, lo.sJ}, vhi{hi.base, hi.sB, hi.sH, hi.sN, hi.sJ};
    return bwd_ex(packed, head_dim, o_lo, o_hi, head_dim, lse, &vlo, &vhi, d_packed, workspace, workspace_bytes, B,
                  heads, N, head_dim, scale, dtype, algo, stream);
}

int psa_attn_profile_enable(int on) {
    psa::g_prof_on.store(on != 0);
    return ok();
}

const char* psa_attn_profile_slot_name(int slot) {
    static const char* names[psa::kNumSlots] = {"fwd", "bwd_pre", "bwd_main", "bwd_dq"};
    return (slot >= 0 && slot < psa::kNumSlots) ? names[slot] : "";
}

int psa_attn_profile_read(float* total_ms, int* launches, int n_slots) {
    if (!total_ms || !launches || n_slots < psa::kNumSlots)
        return fail(PSA_ERR_ARG, "profile_read needs arrays of length >= %d", (int)psa::kNumSlots);
    std::vector<psa::ProfRec> recs;
    {
        std::lock_guard<std::mutex> g(psa::g_prof_mu);
        recs.swap(psa::g_prof);
    }
    for (int i = 0; i < psa::kNumSlots; ++i) { total_ms[i] = 0.f; launches[i] = 0; }
    int rc = PSA_OK;
    for (auto& r : recs) {
        float ms = 0.f;
        cudaError_t e = cudaEventSynchronize(r.b);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.a, r.b);
        if (e != cudaSuccess) rc = fail(PSA_ERR_CUDA, "profile events: %s", cudaGetErrorString(e));
        total_ms[r.slot] += ms;
        launches[r.slot] += 1;
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    return rc ? rc : psa::kNumSlots;
}

int psa_attn_selftest_wait_timeout(void* stream) {
    std::string err;
    const int rc = psa::tc_wait_selftest((cudaStream_t)stream, &err);
    return rc ? fail(rc, "%s", err.c_str()) : ok();
}

int psa_attn_sync_status(void* stream) {
    const cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return fail(PSA_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    std::string err;
    if (psa::tc_take_device_error(&err)) return fail(PSA_ERR_TIMEOUT, "%s", err.c_str());
    if (psa::tc_fwd_take_device_error(&err)) return fail(PSA_ERR_TIMEOUT, "%s", err.c_str());
    if (psa::tc_dq_take_device_error(&err)) return fail(PSA_ERR_TIMEOUT, "%s", err.c_str());
    if (psa::tc_pair_take_device_error(&err)) return fail(PSA_ERR_TIMEOUT, "%s", err.c_str());
    return ok();
}

}  // extern "C"
