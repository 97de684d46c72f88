// host_pipe.cu -- the PSA backward on HOST buffers (psa_attn_bwd_host).
//
// The (batch*head) slices of a PSA problem are independent ("Struct
// PsaFa2Backward": the backward runs per (batch, head) slice), so the copies in,
// the backward and the copy back are pipelined over groups of slices ("chunks"):
// while the kernels of chunk c run on the caller's stream, chunk c+1 is copied
// to the device on one stream of this library and chunk c-1 back to the host
// on another.  The library allocates no device memory: the caller's device
// buffer holds the device copy of every input, d_packed and the workspace.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <string>
#include <vector>

#include "psa_attn.h"
#include "psa_internal.h"

namespace {

constexpr int kMaxChunks = 64;

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

// Per-device copy streams and events, created on the first call on the device
// and kept for the life of the process.
struct Pipe {
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_in_end = nullptr, ev_done = nullptr;
    cudaEvent_t ev_in[kMaxChunks] = {}, ev_k[kMaxChunks] = {};
    std::mutex mu;  // one call enqueues at a time (the events are shared)
    bool ready = false;
};

std::mutex g_pipes_mu;
std::vector<Pipe*> g_pipes;

Pipe* pipe_for_device(int dev, std::string* err) {
    Pipe* p = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_pipes_mu);
        if ((int)g_pipes.size() <= dev) g_pipes.resize(dev + 1, nullptr);
        if (!g_pipes[dev]) g_pipes[dev] = new Pipe();
        p = g_pipes[dev];
    }
    std::lock_guard<std::mutex> lk(p->mu);
    if (p->ready) return p;
    auto ev = [](cudaEvent_t* e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming); };
    cudaError_t e = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = ev(&p->ev_start);
    if (e == cudaSuccess) e = ev(&p->ev_in_end);
    if (e == cudaSuccess) e = ev(&p->ev_done);
    for (int c = 0; c < kMaxChunks && e == cudaSuccess; ++c) {
        e = ev(&p->ev_in[c]);
        if (e == cudaSuccess) e = ev(&p->ev_k[c]);
    }
    if (e != cudaSuccess) {
        *err = std::string("creating the copy streams: ") + cudaGetErrorString(e);
        return nullptr;
    }
    p->ready = true;
    return p;
}

struct Layout {
    size_t packed, o_lo, o_hi, do_lo, do_hi, lse, d_packed, ws, ws_bytes, total;
};

Layout layout(long long BH, int N, int d, int dtype, int algo) {
    const size_t es = dtype == PSA_BF16 ? 2 : 4;
    const size_t sec = (size_t)BH * N * d * es;
    Layout L{};
    size_t off = 0;
    L.packed = off;   off += a256(4 * sec);
    L.o_lo = off;     off += a256(sec);
    L.o_hi = off;     off += a256(sec);
    L.do_lo = off;    off += a256(sec);
    L.do_hi = off;    off += a256(sec);
    L.lse = off;      off += a256((size_t)BH * N * 4);
    L.d_packed = off; off += a256(4 * sec);
    L.ws = off;
    L.ws_bytes = psa_attn_bwd_workspace_bytes_algo((int)BH, 1, N, d, dtype, algo);
    off += a256(L.ws_bytes);
    L.total = off;
    return L;
}

// Chunk count for chunks = 0: the smallest modelled time of
//   sum over chunks of the fused kernel's waves (its last-wave split included)
//     x the time of one unit (N/64 query sub-tiles at about 1.0 us each for
//     d <= 32, 1.3 us for d = 64, on GB300, plus 3 us per unit)
//   + the first chunk's copy in and the last chunk's copy back (~200 GB/s
//     each way over the host link, measured with page-locked buffers)
//   + ~8 us of launch and copy set-up per chunk.
// A heuristic: the chunk count changes only the schedule, never the result.
int auto_chunks(long long BH, int N, int d, int dtype) {
    if (N % 4) return 1;  // every chunk's lse must start on a 16-byte boundary
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    const double es = dtype == PSA_BF16 ? 2.0 : 4.0;
    const double in_bytes = (double)BH * N * (8.0 * d * es + 4.0), out_bytes = (double)BH * N * 4.0 * d * es;
    const int nkt = (N + 127) / 128;
    const double t_unit = (N + 63) / 64 * (d == 64 ? 1.3e-6 : 1.0e-6) + 3e-6;
    const double bw = 200e9;
    int best = 1;
    double best_t = 1e30;
    const int cmax = BH < 16 ? (int)BH : 16;
    for (int c = 1; c <= cmax; ++c) {
        double t = (in_bytes + out_bytes) / c / bw + 8e-6 * c;
        for (int k = 0; k < c; ++k) {
            const long long b0 = BH * k / c, b1 = BH * (k + 1) / c;
            t += psa::tc_bwd_waves((b1 - b0) * nkt, N, sms) * t_unit;
        }
        if (t < best_t * 0.98) {  // prefer fewer chunks unless clearly faster
            best_t = t;
            best = c;
        }
    }
    return best;
}

bool check_shape_args(int B, int heads, int N, int head_dim, int dtype, std::string* err) {
    if (B < 0 || heads < 0 || N < 0) { *err = "negative size"; return false; }
    if (dtype != PSA_F32 && dtype != PSA_BF16) { *err = "bad dtype"; return false; }
    if (head_dim != 16 && head_dim != 32 && head_dim != 64) { *err = "head_dim not in {16, 32, 64}"; return false; }
    return true;
}

}  // namespace

extern "C" {

size_t psa_attn_bwd_host_buffer_bytes(int B, int heads, int N, int head_dim, int dtype, int algo) {
    std::string err;
    if (!check_shape_args(B, heads, N, head_dim, dtype, &err)) return 0;
    const long long BH = (long long)B * heads;
    if (BH == 0 || N == 0) return 0;
    // every valid non-empty problem needs a workspace: 0 = invalid (algo,
    // dtype, head_dim) or sizes over the limits
    if (psa_attn_bwd_workspace_bytes_algo(B, heads, N, head_dim, dtype, algo) == 0) return 0;
    return layout(BH, N, head_dim, dtype, algo).total;
}

int psa_attn_bwd_host_chunks(int B, int heads, int N, int head_dim, int dtype, int algo) {
    (void)algo;
    std::string err;
    if (!check_shape_args(B, heads, N, head_dim, dtype, &err)) return 1;
    const long long BH = (long long)B * heads;
    if (BH <= 0 || N <= 0) return 1;
    return auto_chunks(BH, N, head_dim, dtype);
}

int psa_attn_bwd_host(const void* packed, const void* o_lo, const void* o_hi, const float* lse, const void* do_lo,
                      const void* do_hi, void* d_packed, void* dev_buf, size_t dev_buf_bytes, int B, int heads, int N,
                      int head_dim, float scale, int dtype, int algo, int chunks, void* stream) {
    if (!std::isfinite(scale)) return psa::set_last_error(PSA_ERR_ARG, "scale is not finite");
    if (chunks < 0 || chunks > kMaxChunks)
        return psa::set_last_error(PSA_ERR_ARG, "chunks must be 0 (automatic) or 1.." + std::to_string(kMaxChunks));
    const size_t need = psa_attn_bwd_host_buffer_bytes(B, heads, N, head_dim, dtype, algo);
    if (need == 0) {
        // an empty or invalid problem: the device entry point checks sizes,
        // dtype and algo before any pointer, so it returns 0 for an empty call
        // and the right status for an invalid one
        return psa_attn_bwd_algo(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0, B,
                                 heads, N, head_dim, scale, dtype, algo, stream);
    }
    const long long BH = (long long)B * heads;
    if (!packed || !o_lo || !o_hi || !lse || !do_lo || !do_hi || !d_packed)
        return psa::set_last_error(PSA_ERR_ARG, "a host buffer is NULL");
    std::string err;
    if (!dev_buf || dev_buf_bytes < need)
        return psa::set_last_error(PSA_ERR_WORKSPACE, "device buffer of " + std::to_string(dev_buf_bytes) +
                                                          " bytes < " + std::to_string(need) + " needed");
    if (reinterpret_cast<uintptr_t>(dev_buf) & 255u)
        return psa::set_last_error(PSA_ERR_ALIGN, "device buffer is not 256-byte aligned");
    if (chunks == 0) chunks = auto_chunks(BH, N, head_dim, dtype);
    if (N % 4) chunks = 1;  // chunk starts of lse must stay 16-byte aligned
    if (chunks > BH) chunks = (int)BH;

    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return psa::set_last_error(PSA_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
    Pipe* p = pipe_for_device(dev, &err);
    if (!p) return psa::set_last_error(PSA_ERR_CUDA, err);
    std::lock_guard<std::mutex> lk(p->mu);

    const Layout L = layout(BH, N, head_dim, dtype, algo);
    char* base = static_cast<char*>(dev_buf);
    const size_t es = dtype == PSA_BF16 ? 2 : 4;
    const size_t row = (size_t)N * head_dim * es;  // bytes of one [N, d] slice
    cudaStream_t main = static_cast<cudaStream_t>(stream);
    auto cuda_fail = [&](const char* what, cudaError_t e) {
        return psa::set_last_error(PSA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
    };

    // the staging buffers are free once the caller's stream got here
    ce = cudaEventRecord(p->ev_start, main);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(p->s_in, p->ev_start, 0);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(p->s_out, p->ev_start, 0);
    if (ce != cudaSuccess) return cuda_fail("ordering the copy streams after the caller's stream", ce);

    int rc = PSA_OK;
    for (int c = 0; c < chunks; ++c) {
        const long long b0 = BH * c / chunks, b1 = BH * (c + 1) / chunks, nb = b1 - b0;
        if (nb == 0) continue;
        struct Cp { size_t dev_off; const void* host; size_t slice; };
        const Cp ins[6] = {{L.packed, packed, 4 * row}, {L.o_lo, o_lo, row}, {L.o_hi, o_hi, row},
                           {L.lse, lse, (size_t)N * 4}, {L.do_lo, do_lo, row}, {L.do_hi, do_hi, row}};
        for (const Cp& x : ins) {
            ce = cudaMemcpyAsync(base + x.dev_off + b0 * x.slice, static_cast<const char*>(x.host) + b0 * x.slice,
                                 nb * x.slice, cudaMemcpyHostToDevice, p->s_in);
            if (ce != cudaSuccess) break;
        }
        if (ce == cudaSuccess) ce = cudaEventRecord(p->ev_in[c], p->s_in);
        if (ce == cudaSuccess) ce = cudaStreamWaitEvent(main, p->ev_in[c], 0);
        if (ce != cudaSuccess) { rc = cuda_fail("copy to the device", ce); break; }
        rc = psa_attn_bwd_algo(base + L.packed + b0 * 4 * row, base + L.o_lo + b0 * row, base + L.o_hi + b0 * row,
                               reinterpret_cast<const float*>(base + L.lse + b0 * (size_t)N * 4),
                               base + L.do_lo + b0 * row, base + L.do_hi + b0 * row,
                               base + L.d_packed + b0 * 4 * row, base + L.ws, L.ws_bytes, (int)nb, 1, N, head_dim,
                               scale, dtype, algo, stream);
        if (rc) break;
        ce = cudaEventRecord(p->ev_k[c], main);
        if (ce == cudaSuccess) ce = cudaStreamWaitEvent(p->s_out, p->ev_k[c], 0);
        if (ce == cudaSuccess)
            ce = cudaMemcpyAsync(static_cast<char*>(d_packed) + b0 * 4 * row, base + L.d_packed + b0 * 4 * row,
                                 nb * 4 * row, cudaMemcpyDeviceToHost, p->s_out);
        if (ce != cudaSuccess) { rc = cuda_fail("copy to the host", ce); break; }
    }
    // the caller's stream continues after every copy this call enqueued (also
    // after an error, so that a later call may reuse the buffers)
    const std::string keep = rc ? std::string(psa_attn_last_error()) : std::string();
    ce = cudaEventRecord(p->ev_in_end, p->s_in);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(main, p->ev_in_end, 0);
    if (ce == cudaSuccess) ce = cudaEventRecord(p->ev_done, p->s_out);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(main, p->ev_done, 0);
    if (rc) return psa::set_last_error(rc, keep);
    if (ce != cudaSuccess) return cuda_fail("ordering the caller's stream after the copies", ce);
    return psa::set_last_error(PSA_OK, "");
}

}  // extern "C"
