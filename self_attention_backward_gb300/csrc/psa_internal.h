// psa_internal.h -- host-side interface between the C-ABI front end
// (psa_attn.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <string>

namespace psa {

// A strided view of a [B, heads, N, d] tensor: element (b, h, n, j) at
// base + b*sB + h*sH + n*sN + j*sJ (elements).
struct View {
    const void* base;
    long long sB, sH, sN, sJ;
};

struct BwdArgs {
    const void* packed;
    const void* o_lo;
    const void* o_hi;
    const float* lse;
    const void* do_lo;
    const void* do_hi;
    void* d_packed;
    void* workspace;
    size_t workspace_bytes;
    long long BH;
    int N;
    int d;
    float scale;
    int dtype;
    cudaStream_t stream;
    // Layouts (psa_attn_bwd_ex); the defaults describe contiguous tensors.
    int heads = 1;               // B = BH / heads, for the views' batch / head strides
    long long ld_qkv = 0;        // row stride of packed and d_packed (0: d)
    long long ld_o = 0;          // row stride of o_lo, o_hi (0: d)
    bool views = false;          // true: dO_lo / dO_hi are read through vlo / vhi
    View vlo{}, vhi{};
    long long qkv_ld() const { return ld_qkv ? ld_qkv : d; }
    long long o_ld() const { return ld_o ? ld_o : d; }
    // dO_lo / dO_hi as views (a contiguous [BH, N, d] tensor when !views)
    View do_view(int which) const {
        if (views) return which ? vhi : vlo;
        return View{which ? do_hi : do_lo, (long long)heads * N * d, (long long)N * d, d, 1};
    }
};

// Kernel timing scope (psa_attn_profile_enable): records a CUDA event pair
// around the launches made while it is alive, when profiling is on.  While it
// is on, launches that would overlap the kernel before them (programmatic
// dependent launch) are made plain, so that each event pair times one kernel.
enum ProfSlot { kSlotFwd = 0, kSlotPre = 1, kSlotMain = 2, kSlotDq = 3, kNumSlots = 4 };
bool prof_enabled();
class ProfScope {
  public:
    ProfScope(int slot, cudaStream_t st);
    ~ProfScope();
    ProfScope(const ProfScope&) = delete;
    ProfScope& operator=(const ProfScope&) = delete;

  private:
    int slot_;
    cudaStream_t st_;
    cudaEvent_t a_ = nullptr, b_ = nullptr;
};

// Tensor-core (tcgen05) forward: tc_fwd.cu.
bool tc_fwd_supported(int dtype, int d);
int tc_fwd_launch(const void* packed, void* o_lo, void* o_hi, float* lse, long long BH, int N, int d, float scale,
                  cudaStream_t stream, std::string* err);
int tc_fwd_take_device_error(std::string* err);

// Tensor-core (tcgen05) backward: tc_bwd.cu.
bool tc_supported(int dtype, int d);
size_t tc_workspace_bytes(long long BH, int N, int d);
// Waves of the fused backward kernel for `units` (batch*head, 128-key tile)
// units on `sms` SMs, its last-wave split included (a fraction for a split wave).
double tc_bwd_waves(long long units, int N, int sms);
// Returns 0 or a psa_status; `err` receives a message on failure.
int tc_bwd_launch(const BwdArgs& a, std::string* err);
// Two-pass tensor-core backward (no atomics, reproducible bit for bit): D,
// the key-outer dK/dV pass (tc_bwd.cu), the query-outer dQ pass (tc_dq.cu).
size_t tc_two_pass_workspace_bytes(long long BH, int N);
int tc_two_pass_launch(const BwdArgs& a, std::string* err);
// D = rowsum(dO_lo o O_lo + dO_hi o O_hi) into `Drow` ([BH*N] fp32), bf16 inputs.
int tc_pre_d_launch(const BwdArgs& a, float* Drow, std::string* err);
// Two-pass backward on SM pairs (cta_group::2, tc_pair.cu), head_dim 32 or 64;
// same workspace as tc_two_pass_launch.
bool tc_pair_supported(int dtype, int d);
int tc_pair_launch(const BwdArgs& a, std::string* err);
int tc_pair_take_device_error(std::string* err);
// The query-outer dQ pass alone; `Drow` = [BH*N] fp32 row statistics D.
int tc_dq_launch(const BwdArgs& a, const float* Drow, std::string* err);
int tc_dq_take_device_error(std::string* err);
// Launches a kernel whose bounded wait is made to run out (20 ms).
int tc_wait_selftest(cudaStream_t stream, std::string* err);
// Reads and clears the device-side timeout flag of the tensor-core kernels
// (call after the stream is synchronised).  Returns 1 if a wait gave up.
int tc_take_device_error(std::string* err);

// Gathers a strided view of a [BH, N, d] tensor (elements of `esize` bytes,
// 2 or 4) into a contiguous [BH, N, d] buffer on `stream` (merge.cu).
int gather_view_launch(const View& v, void* dst, long long BH, int heads, int N, int d, int esize,
                       cudaStream_t stream, std::string* err);
// The views of dO_lo / dO_hi inside a merged [B, 2*heads*d, N] tensor (merge.cu).
void merged_views(const void* d_merged, int heads, int N, int d, int esize, View* lo, View* hi);

// Sets the calling thread's psa_attn_last_error() message ("" clears it) and
// returns `code`; for entry points defined outside psa_attn.cu.
int set_last_error(int code, const std::string& msg);

}  // namespace psa
