// simt_kernels.cuh -- CUDA-core (FFMA) PSA attention kernels.
//
// These are the fp32-storage path (fp32 parity needs full fp32 products, which
// the bf16 tensor-core path does not give) and the cross-check path for the
// tensor-core kernels.  Same mathematics as the tensor-core path, written as
// plain per-row loops:
//   forward  : online softmax over key tiles -> O_lo, O_hi, LSE
//   pre      : D_i = <dO_lo[i], O_lo[i]> + <dO_hi[i], O_hi[i]>
//   dK / dV  : one CTA per 64-key tile iterates over all queries
//   dQ       : one CTA per 64-query tile iterates over all keys
// "Struct PsaFa2Backward" (description): a query row's gradient is a sweep over
// the keys, a key row's gradients a sweep over the queries.  Here the two
// sweeps are separate kernels, so nothing is added atomically and the result
// is deterministic.
//
// Thread layout: 4 threads per row; thread `sub` owns the 4-float chunks
// g = sub + 4c (c < D/16) of a d-row, so the 4 threads of a row read 64
// consecutive bytes of shared memory per step (no bank conflicts), and a dot
// product over d is a partial sum per thread plus two xor-shuffles.
#pragma once

#include "common.cuh"

namespace psa {
namespace simt {

constexpr int kThreads = 256;
constexpr int kRows = 64;  // rows (queries or keys) owned per CTA

template <int D>
__device__ __forceinline__ float dot_part(const float (&a)[D / 16][4], const float* row, int sub) {
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
        const float4 b = *reinterpret_cast<const float4*>(row + 4 * (sub + 4 * c));
        acc = fmaf(a[c][0], b.x, acc);
        acc = fmaf(a[c][1], b.y, acc);
        acc = fmaf(a[c][2], b.z, acc);
        acc = fmaf(a[c][3], b.w, acc);
    }
    return acc;
}

__device__ __forceinline__ float quad_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    return x;
}

template <int D>
__device__ __forceinline__ void axpy_part(float (&acc)[D / 16][4], float a, const float* row, int sub) {
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
        const float4 b = *reinterpret_cast<const float4*>(row + 4 * (sub + 4 * c));
        acc[c][0] = fmaf(a, b.x, acc[c][0]);
        acc[c][1] = fmaf(a, b.y, acc[c][1]);
        acc[c][2] = fmaf(a, b.z, acc[c][2]);
        acc[c][3] = fmaf(a, b.w, acc[c][3]);
    }
}

template <typename T, int D>
__device__ __forceinline__ void load_row_part(float (&dst)[D / 16][4], const T* row, int sub) {
#pragma unroll
    for (int c = 0; c < D / 16; ++c) load4(row + 4 * (sub + 4 * c), dst[c]);
}

template <typename T, int D>
__device__ __forceinline__ void store_row_part(T* row, const float (&src)[D / 16][4], float mul, int sub) {
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
        float v[4] = {src[c][0] * mul, src[c][1] * mul, src[c][2] * mul, src[c][3] * mul};
        store4(row + 4 * (sub + 4 * c), v);
    }
}

// Cooperative copy of rows [r0, r0 + ROWS) of up to three [N, D] tensors into
// fp32 shared tiles; rows >= N are zero.
template <typename T, int D, int ROWS>
__device__ __forceinline__ void load_tiles(float* s0, float* s1, float* s2, const T* g0, const T* g1,
                                           const T* g2, int r0, int N) {
    for (int idx = threadIdx.x; idx < ROWS * (D / 4); idx += kThreads) {
        const int row = idx / (D / 4), g = idx % (D / 4);
        const int r = r0 + row;
        float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f}, c[4] = {0.f, 0.f, 0.f, 0.f};
        if (r < N) {
            load4(g0 + (size_t)r * D + 4 * g, a);
            load4(g1 + (size_t)r * D + 4 * g, b);
            load4(g2 + (size_t)r * D + 4 * g, c);
        }
        *reinterpret_cast<float4*>(s0 + row * D + 4 * g) = make_float4(a[0], a[1], a[2], a[3]);
        *reinterpret_cast<float4*>(s1 + row * D + 4 * g) = make_float4(b[0], b[1], b[2], b[3]);
        *reinterpret_cast<float4*>(s2 + row * D + 4 * g) = make_float4(c[0], c[1], c[2], c[3]);
    }
}

// ---------------------------------------------------------------- forward
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
fwd_kernel(const T* __restrict__ packed, T* __restrict__ o_lo, T* __restrict__ o_hi,
           float* __restrict__ lse, int N, int ntiles, float scale_log2) {
    constexpr int BK = 32, NC = D / 16;
    __shared__ __align__(16) float Ks[BK * D];
    __shared__ __align__(16) float Vl[BK * D];
    __shared__ __align__(16) float Vh[BK * D];
    const int bh = blockIdx.x / ntiles, tile = blockIdx.x % ntiles;
    const int r = threadIdx.x >> 2, sub = threadIdx.x & 3;
    const int i = tile * kRows + r;
    const bool valid = i < N;
    const size_t sec = (size_t)N * D;
    const T* Q = packed + (size_t)bh * 4 * sec;
    const T* K = Q + sec;
    const T* VL = Q + 2 * sec;
    const T* VH = Q + 3 * sec;

    float q[NC][4], ol[NC][4], oh[NC][4];
    load_row_part<T, D>(q, Q + (size_t)(valid ? i : N - 1) * D, sub);
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) ol[c][e] = oh[c][e] = 0.f;
    float m = -INFINITY, l = 0.f;

    for (int k0 = 0; k0 < N; k0 += BK) {
        __syncthreads();
        load_tiles<T, D, BK>(Ks, Vl, Vh, K, VL, VH, k0, N);
        __syncthreads();
        float s[BK];
        float mt = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < BK; ++jj) {
            const float part = quad_sum(dot_part<D>(q, Ks + jj * D, sub));
            s[jj] = (k0 + jj < N) ? part * scale_log2 : -INFINITY;
            mt = fmaxf(mt, s[jj]);
        }
        const float mn = fmaxf(m, mt);          // finite: the tile has a valid key
        const float alpha = exp2f(m - mn);      // 0 on the first tile
        l *= alpha;
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e) { ol[c][e] *= alpha; oh[c][e] *= alpha; }
#pragma unroll
        for (int jj = 0; jj < BK; ++jj) {
            const float p = exp2f(s[jj] - mn);
            l += p;
            axpy_part<D>(ol, p, Vl + jj * D, sub);
            axpy_part<D>(oh, p, Vh + jj * D, sub);
        }
        m = mn;
    }
    if (valid) {
        const float inv = 1.f / l;
        const size_t row = (size_t)bh * N + i;
        store_row_part<T, D>(o_lo + row * D, ol, inv, sub);
        store_row_part<T, D>(o_hi + row * D, oh, inv, sub);
        if (sub == 0) lse[row] = (m + log2f(l)) * kLn2;
    }
}

// ---------------------------------------------------------------- D_i
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
pre_kernel(const T* __restrict__ o_lo, const T* __restrict__ o_hi, const T* __restrict__ do_lo,
           const T* __restrict__ do_hi, float* __restrict__ Drow, long long rows) {
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    float acc = 0.f;
    for (int c = lane; c < D; c += 32) {
        const size_t x = (size_t)row * D + c;
        acc = fmaf(to_f32(do_lo[x]), to_f32(o_lo[x]), acc);
        acc = fmaf(to_f32(do_hi[x]), to_f32(o_hi[x]), acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) Drow[row] = acc;
}

// ---------------------------------------------------------------- dK, dV
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
dkdv_kernel(const T* __restrict__ packed, const T* __restrict__ do_lo, const T* __restrict__ do_hi,
            const float* __restrict__ lse, const float* __restrict__ Drow, T* __restrict__ d_packed,
            int N, int ntiles, float scale, float scale_log2) {
    constexpr int BQ = 32, NC = D / 16;
    __shared__ __align__(16) float Qs[BQ * D];
    __shared__ __align__(16) float Gl[BQ * D];
    __shared__ __align__(16) float Gh[BQ * D];
    __shared__ float Ls[BQ], Ds[BQ];
    const int bh = blockIdx.x / ntiles, tile = blockIdx.x % ntiles;
    const int r = threadIdx.x >> 2, sub = threadIdx.x & 3;
    const int j = tile * kRows + r;
    const int jc = j < N ? j : N - 1;
    const size_t sec = (size_t)N * D;
    const T* Q = packed + (size_t)bh * 4 * sec;
    const T* K = Q + sec;
    const T* VL = Q + 2 * sec;
    const T* VH = Q + 3 * sec;
    const T* GL = do_lo + (size_t)bh * sec;
    const T* GH = do_hi + (size_t)bh * sec;

    float k[NC][4], vl[NC][4], vh[NC][4], dk[NC][4], dvl[NC][4], dvh[NC][4];
    load_row_part<T, D>(k, K + (size_t)jc * D, sub);
    load_row_part<T, D>(vl, VL + (size_t)jc * D, sub);
    load_row_part<T, D>(vh, VH + (size_t)jc * D, sub);
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) dk[c][e] = dvl[c][e] = dvh[c][e] = 0.f;

    for (int q0 = 0; q0 < N; q0 += BQ) {
        __syncthreads();
        load_tiles<T, D, BQ>(Qs, Gl, Gh, Q, GL, GH, q0, N);
        if (threadIdx.x < BQ) {
            const int i = q0 + threadIdx.x;
            // a padded query row gets LSE = +inf, so its P is exactly 0
            Ls[threadIdx.x] = i < N ? lse[(size_t)bh * N + i] * kLog2e : INFINITY;
            Ds[threadIdx.x] = i < N ? Drow[(size_t)bh * N + i] : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int ii = 0; ii < BQ; ++ii) {
            const float s = quad_sum(dot_part<D>(k, Qs + ii * D, sub));
            const float p = exp2f(fmaf(s, scale_log2, -Ls[ii]));
            const float dp = quad_sum(dot_part<D>(vl, Gl + ii * D, sub) + dot_part<D>(vh, Gh + ii * D, sub));
            const float ds = p * (dp - Ds[ii]);
            axpy_part<D>(dvl, p, Gl + ii * D, sub);
            axpy_part<D>(dvh, p, Gh + ii * D, sub);
            axpy_part<D>(dk, ds, Qs + ii * D, sub);
        }
    }
    if (j < N) {
        T* out = d_packed + (size_t)bh * 4 * sec + (size_t)j * D;
        store_row_part<T, D>(out + sec, dk, scale, sub);
        store_row_part<T, D>(out + 2 * sec, dvl, 1.f, sub);
        store_row_part<T, D>(out + 3 * sec, dvh, 1.f, sub);
    }
}

// ---------------------------------------------------------------- dQ
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
dq_kernel(const T* __restrict__ packed, const T* __restrict__ do_lo, const T* __restrict__ do_hi,
          const float* __restrict__ lse, const float* __restrict__ Drow, T* __restrict__ d_packed,
          int N, int ntiles, float scale, float scale_log2) {
    constexpr int BK = 32, NC = D / 16;
    __shared__ __align__(16) float Ks[BK * D];
    __shared__ __align__(16) float Vl[BK * D];
    __shared__ __align__(16) float Vh[BK * D];
    const int bh = blockIdx.x / ntiles, tile = blockIdx.x % ntiles;
    const int r = threadIdx.x >> 2, sub = threadIdx.x & 3;
    const int i = tile * kRows + r;
    const int ic = i < N ? i : N - 1;
    const size_t sec = (size_t)N * D;
    const T* Q = packed + (size_t)bh * 4 * sec;
    const T* K = Q + sec;
    const T* VL = Q + 2 * sec;
    const T* VH = Q + 3 * sec;
    const size_t row = (size_t)bh * N + ic;

    float q[NC][4], gl[NC][4], gh[NC][4], dq[NC][4];
    load_row_part<T, D>(q, Q + (size_t)ic * D, sub);
    load_row_part<T, D>(gl, do_lo + row * D, sub);
    load_row_part<T, D>(gh, do_hi + row * D, sub);
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) dq[c][e] = 0.f;
    const float L2 = lse[row] * kLog2e;
    const float Di = Drow[row];

    for (int k0 = 0; k0 < N; k0 += BK) {
        __syncthreads();
        load_tiles<T, D, BK>(Ks, Vl, Vh, K, VL, VH, k0, N);
        __syncthreads();
#pragma unroll 4
        for (int jj = 0; jj < BK; ++jj) {
            const float s = quad_sum(dot_part<D>(q, Ks + jj * D, sub));
            const float p = (k0 + jj < N) ? exp2f(fmaf(s, scale_log2, -L2)) : 0.f;
            const float dp = quad_sum(dot_part<D>(gl, Vl + jj * D, sub) + dot_part<D>(gh, Vh + jj * D, sub));
            axpy_part<D>(dq, p * (dp - Di), Ks + jj * D, sub);
        }
    }
    if (i < N) store_row_part<T, D>(d_packed + (size_t)bh * 4 * sec + (size_t)i * D, dq, scale, sub);
}

}  // namespace simt
}  // namespace psa
