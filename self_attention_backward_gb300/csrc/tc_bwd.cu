// tc_bwd.cu -- tensor-core (tcgen05 / TMEM / TMA) PSA backward, bf16 storage.
//
// "Struct PsaFa2Backward" (vision_rs yolo attention psa): the backward of the
// lo/hi pair of FA2 calls that share Q and K.  Here the pair runs as ONE
// attention with a 2d-wide value [V_lo | V_hi]:
//   dS = P o (dO_lo V_lo^T + dO_hi V_hi^T - D),  D = rowsum(dO_lo o O_lo) + rowsum(dO_hi o O_hi)
// so S and P are recomputed once for both calls and dQ, dK come out already
// summed (the page's atomic_add into the shared dQ/dK sections is not needed
// for that).
//
// Decomposition: one work unit per (batch*head, 128-key tile j).  Its CTA keeps
// K_j, V_lo,j, V_hi,j in shared memory and its dV_lo|dV_hi and dK accumulators
// in TMEM, and sweeps over every query of its slice ("Struct PsaFa2Backward",
// description: key-row gradients come from such a sweep) in 64-query
// sub-tiles u:
//   S^T  = K_j Q_u^T                 (M = 128 keys, N = 64 queries, K = d)
//   dP^T = V_lo,j dO_lo,u^T + V_hi,j dO_hi,u^T          (K = 2d)
//   P^T  = exp2(S^T * scale*log2e - LSE*log2e),  dS^T = P^T o (dP^T - D)
//   [dV_lo | dV_hi] += P^T [dO_lo,u | dO_hi,u]          (one N = 2d MMA)
//   dK += dS^T Q_u
// and per pair of sub-tiles (128 queries g), dQ_g(partial) = dS_g K_j, added
// into an fp32 accumulator in the workspace; a last kernel scales and casts it
// into d_packed.
//
// Pipelining.  S^T/dP^T live in NB TMEM buffers (buffer u % NB; NB = 3 for
// d <= 32, 2 for d = 64, where the accumulators take the rest of TMEM), and two
// softmax-gradient warpgroups take alternate sub-tiles, so the tensor core
// works on later sub-tiles while a warpgroup turns S/dP(u) into P and dS.  P^T
// is written over the first 32 columns of its S^T buffer as bf16 pairs (the A
// operand of the dV MMA).  dS^T goes into a 4-block shared ring (block
// 2 (g & 1) + the sub-tile's place in its pair) for the dQ MMA, which needs it
// with queries as rows, and which the dK MMA reads too for d <= 32; for d = 64
// dS^T also goes over the first 32 columns of its dP^T buffer as dK's A
// operand.  S^T(u+NB) reuses u's buffer and is issued right after dV(u), the
// last reader of P^T(u); dP^T(u+NB) right after dK(u); the pipe keeps issue
// order.  A block of the ring is rewritten only after its dQ (and dK) MMA has
// read it.
//
// Cost model that shaped it (measured on GB300): a tcgen05.mma with M = 128,
// K = 16 costs about max(46, N/2) cycles, so the MMA count, not the flop
// count, bounds small head dims; a barrier wait of the issuing thread first
// waits for its own MMAs in flight.  The issuing thread precomputes every
// descriptor so that issuing an MMA is one add per operand.
//
// Persistent: one CTA per SM walks work items (units of one (batch*head,
// 128-key tile), or pieces of one along the queries) in turn (see the kernel);
// for d <= 32 the next item's K/V tile loads into a second buffer while the
// current item runs.  The kernel is a programmatic dependent of the
// statistics kernel before it (it reads the statistics and the zeroed dQ
// accumulator only after griddepcontrol.wait).
//
// Warp roles: warp 0 TMA producer (each item's K/V tile; the Q/dO stages: Q,
// dO_lo, dO_hi and the sub-tile's row statistics), warp 1 MMA issuer (one thread) and TMEM owner,
// warps 2-5 / 6-9 softmax-gradient warpgroups 0 / 1 (one key row per thread),
// warps 10-13 dQ drain (one query row per thread; the partials go to the fp32
// accumulator by TMA bulk reduce) and then each item's dK/dV epilogue (one key
// row per thread), warp 14 the dQ MMA issuer; warp 15 issues the odd
// sub-tiles' main MMAs and warp 1 the even ones (512 threads).
//
// Every mbarrier wait is bounded (kTimeoutNs); on timeout the CTA sets a device
// error word (read by psa_attn_sync_status), skips the rest of its work, waits
// (bounded) for its own TMA copies and MMAs in flight, frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdio>
#include <mutex>
#include <string>
#include <utility>

#include "common.cuh"
#include "psa_attn.h"
#include "psa_internal.h"
#include "tc_ptx.cuh"
#include "tc_sync.cuh"
#include "tc_tmap.h"

#pragma nv_diag_suppress 177  // per-variant tile constants not all used by every head_dim

namespace psa {
namespace {

using namespace psa::tc;
using bf16 = __nv_bfloat16;

__device__ int g_tc_error = 0;  // 0 = fine; else (1 + role) << 24 | tile


template <int D>
struct Cfg {
    static constexpr int BM = 128;                 // keys per CTA (MMA M)
    static constexpr int BS = 64;                  // queries per sub-tile
    static constexpr int ROWB = D * 2;             // bytes per [*, D] bf16 row
    static constexpr int KTILE = BM * ROWB;        // [128, D] tile
    static constexpr int QTILE = BS * ROWB;        // [64, D] tile
    static constexpr int NB = D == 64 ? 2 : 3;     // S^T/dP^T buffers in TMEM
    static constexpr int NST = D == 64 ? 4 : 6;    // Q/dO stages
    // warps: 0 producer, 1 the main MMA issuer (with TWO_ISSUERS: of the even
    // sub-tiles, and warp 15 of the odd ones), 2-9 softmax, 10-13 dQ drain, 14
    // the dQ MMA issuer.  Two main issuers: 1% at head_dim 32 (N = 6400); at
    // head_dim 64 they cost 5% while the drain added dQ with vector atomics and
    // gain 6% (N = 1600 0.210 -> 0.196 ms) since it uses bulk reduces, measured.
    static constexpr bool TWO_ISSUERS = true;
    static constexpr int THREADS = TWO_ISSUERS ? 512 : 480;
    static constexpr uint32_t SW = D == 64 ? 2u : D == 32 ? 4u : 6u;  // swizzle code of [*, D] tiles
    // K, V_lo, V_hi of an item at OFF_K / OFF_VL / OFF_VH of K/V buffer
    // it % KVBUF.  Two buffers where shared memory has room for them (head_dim
    // <= 32): the next item's tiles then load while the current item runs,
    // instead of after its last dQ product.
    static constexpr int KVBUF = D == 64 ? 1 : 2;
    // Where the dK product reads dS^T: from the sub-tile's dS ring block in
    // shared memory (which the dQ product reads too), sparing the softmax a
    // TMEM store per element, or from the dP^T half of its TMEM buffer.
    // Measured: the ring at head_dim <= 32 (N = 6400: bwd_main 0.3714 ->
    // 0.3678 ms), TMEM at head_dim 64 (the ring there: N = 1600 0.1905 ->
    // 0.193 ms per step).
    static constexpr bool DK_SMEM = D <= 32;
    // A P-ready barrier (PR) per sub-tile: the issuer starts dV(u) and
    // S^T(u+NB) once the softmax has written P(u), before its second phase,
    // and dK(u), dP^T(u+NB) after it (PF).  Measured: at head_dim 64 N = 1600
    // 0.1780 -> 0.1662 ms, N = 400 0.0908 -> 0.0893 ms; at head_dim 32 the
    // issuer's second wait per sub-tile cost more than it gained (N = 6400
    // bwd_main 0.3425 -> 0.3674 ms).
    static constexpr bool P_READY = D == 64;
    static constexpr int KVSET = 3 * KTILE;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_VL = KTILE;
    static constexpr int OFF_VH = 2 * KTILE;
    static constexpr int OFF_STAGE = KVBUF * KVSET;  // stage s: Q, dO_lo, dO_hi at +s*STAGE
    static constexpr int STAGE = 3 * QTILE;
    static constexpr int OFF_DS = OFF_STAGE + NST * STAGE;  // dS^T ring: 4 x [128 keys][64 queries] bf16
    // dQ drain: each 128-query partial is staged here in boxes of BOXC columns
    // (128-byte or 64-byte rows, swizzled as the tensor map expects) and added
    // to the fp32 accumulator by TMA bulk reduces.  Vector atomics, one row per
    // thread, put 32 separate 16-byte requests per warp instruction into the
    // SM's load/store path, where they held up the softmax's dS stores to
    // shared memory by ~2 K cycles per 128-query group at head_dim 64
    // (measured).  NDQS staging buffers of one box of min(D, 32) columns each:
    // two, or one at head_dim 64 (what shared memory leaves room for; the drain
    // warps also stage the dK/dV epilogue there).
    static constexpr int BOXC = D < 32 ? D : 32;
    static constexpr int NDQS = D == 64 ? 1 : 2;
    static constexpr int DQS_BYTES = 128 * BOXC * 4;
    static constexpr int OFF_DQS = OFF_DS + 4 * 16384;
    // NST x 32 float4, one per query pair c of the stage's 64 queries:
    // {-LSE_2c log2(e), -LSE_2c+1 log2(e), D_2c, D_2c+1}
    static constexpr int OFF_ST = OFF_DQS + NDQS * DQS_BYTES;
    static constexpr int OFF_BAR = OFF_ST + NST * 512;     // mbarriers (64)
    static constexpr int OFF_MISC = OFF_BAR + 512;
    static constexpr int USED = OFF_MISC + 64;
    // + 1 KB to align the base to 1024 where that fits; at head_dim 64 it does
    // not, and the host checks once per device that the base is aligned
    // (dyn_smem_base_aligned).  At least 116 KB so that one CTA owns an SM (its
    // TMEM allocation is all 512 columns).
    static constexpr bool SLACK = USED + 1024 <= 232448;
    static constexpr int SMEM_A = SLACK ? USED + 1024 : USED;
    static constexpr int SMEM = SMEM_A > 118784 ? SMEM_A : 118784;
    // TMEM columns (fp32): buffer b = [128b, 128b+128): S^T (64), dP^T (64)
    // (P^T is written over the first 32 columns of its S^T as bf16 pairs); then
    // dV_lo|dV_hi, dK, dQ
    static constexpr uint32_t C_DV = 128 * NB;
    static constexpr uint32_t C_DK = C_DV + 2 * D, C_DQ = C_DV + 3 * D;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(C_DQ + D <= TMEM_COLS, "TMEM budget");
    static_assert(USED <= 232448, "shared memory budget");
    static_assert(NDQS * DQS_BYTES >= 4 * 2048, "the epilogue stages 2 KB per drain warp");
    static_assert(NST > NB, "the softmax's wait for the stage of u+NB would wait on its own release");
};

// barrier indices (SF: one per S/dP buffer; PF: softmax done, a ring of 4 over
// the sub-tiles; QF/QE: one per Q/dO stage).  A warp starts sub-tile u only
// after S/dP(u) was issued, which followed the issuer's wait on PF(u - NB); so
// with NB <= 3 no warp runs 4 sub-tiles ahead of a slower one and a PF barrier
// never gets arrivals for two of its phases at once (a ring of 2 would allow a
// warp two sub-tiles ahead to complete a slower warp's phase).
// DQF: the dQ product of 128-query group g is done, at DQF + (g & 1); DQE: the
// drain has read group g from the dQ accumulator, at DQE + (g & 1).  Each pair
// alternates by group so that a waiter on group g finds the barrier at most one
// phase on: the barrier's previous phase (group g-2) is known complete when the
// wait starts, and its next one (group g+2) cannot complete before the waiter
// has acted (see each wait).  DQA: the dQ issuer's final commit.
enum { B_KV = 0, B_SF = 1, B_PF = 4, B_ACC = 9, B_DQA = 10, B_QF = 11, B_QE = 17, B_DQF = 23, B_DQE = 25 };
constexpr int kPfRing = 4;
static_assert(B_DQE + 2 <= 32, "barrier area holds 32 barriers");

// The fused kernel's barriers.  Two threads issue its main MMAs: the one for
// sub-tiles of parity p issues dV/dK(u) for its u and then S/dP(u + NB) (so
// buffer reuse stays in one thread's issue order), each waiting only for its
// own sub-tiles' PF.  PF is a ring of 8: PF(u + 8) needs S/dP(u + 8), which the
// thread of u + 5 issues after PF(u + 5), whose S/dP(u + 5) the thread of u + 2
// -- the same parity as u -- issued after it had seen PF(u + 2), hence PF(u);
// so no PF phase completes before each of its waiters (the issuer of its parity
// and the dQ issuer) has seen the previous one.  ACC / ACCB: each main issuer's
// final commit.  S^T(u) and dP^T(u) signal separately, SFS and SFD: rings of
// 2 NB over the sub-tiles (u % 2NB).  With NB odd the sub-tiles of one buffer
// alternate between the issuers, and two issuers give no order between their
// commits; with the ring each barrier has one committing thread (the issuer of
// u - NB) and one waiting warpgroup (u's), which saw its previous phase
// (u - 2NB) before this one.  DQF, DQE, DQA as above.
// KV / KVE: K/V buffer b loaded, and no MMA reads it any more (F_KV and F_KVE
// for buffer 0, F_KV1 and F_KVE1 for buffer 1); buffer it % KVBUF holds item
// it, phase it / KVBUF.
enum {
    F_KV = 0, F_SFS = 1, F_SFD = 7, F_PF = 13, F_ACC = 21, F_ACCB = 22, F_DQA = 23, F_QF = 24, F_QE = 30, F_DQF = 36,
    F_DQE = 38, F_KVE = 40, F_EPI = 41, F_KV1 = 42, F_KVE1 = 43, F_PR = 44
};
constexpr int kPfRingF = 8;
static_assert(F_PR + kPfRingF <= 64, "barrier area holds 64 barriers");
__device__ __forceinline__ int kv_full(int b) { return b ? F_KV1 : F_KV; }
__device__ __forceinline__ int kv_empty(int b) { return b ? F_KVE1 : F_KVE; }

// P and dS of one 32-query chunk of this thread's key row, packed to bf16
// pairs: P = exp2(S * scale*log2e - L), dS = P (dP - D).
template <bool MASK>
__device__ __forceinline__ void softmax_vals(const uint32_t (&sr)[32], const uint32_t (&pr)[32], const float* L2s,
                                             const float* Ds, float scale_log2, bool kvalid, uint32_t (&pk)[16],
                                             uint32_t (&dk)[16]) {
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(L2s + e);
        const float4 d4 = *reinterpret_cast<const float4*>(Ds + e);
        float p0 = ex2_approx(fmaf(__uint_as_float(sr[e + 0]), scale_log2, -l4.x));
        float p1 = ex2_approx(fmaf(__uint_as_float(sr[e + 1]), scale_log2, -l4.y));
        float p2 = ex2_approx(fmaf(__uint_as_float(sr[e + 2]), scale_log2, -l4.z));
        float p3 = ex2_approx(fmaf(__uint_as_float(sr[e + 3]), scale_log2, -l4.w));
        if (MASK && !kvalid) p0 = p1 = p2 = p3 = 0.f;
        pk[e / 2] = pack_bf16x2(p0, p1);
        pk[e / 2 + 1] = pack_bf16x2(p2, p3);
        dk[e / 2] = pack_bf16x2(p0 * (__uint_as_float(pr[e + 0]) - d4.x), p1 * (__uint_as_float(pr[e + 1]) - d4.y));
        dk[e / 2 + 1] =
            pack_bf16x2(p2 * (__uint_as_float(pr[e + 2]) - d4.z), p3 * (__uint_as_float(pr[e + 3]) - d4.w));
    }
}

// The epilogue of one warp: dK (scaled), dV_lo, dV_hi of the warp's 32 key
// rows (TMEM lane quarter q4) as bf16 into d_packed sections 1-3, coalesced
// through the warp's 2 KB staging buffer stg; or, for a piece of a split unit,
// the fp32 partials into dkv_part.  Every main MMA of the item must be
// complete.  Each chunk of the accumulators is zeroed once read (the next
// item's products accumulate onto it), and each thread arrives on epi_bar once
// its rows are read and zeroed.
template <int D, typename C>
__device__ __forceinline__ void dkdv_epilogue(uint32_t tmem, int q4, int lane, uint32_t stg, uint32_t epi_bar,
                                              bf16* d_packed, int bh, int k0, int N, long long ldq, float scale,
                                              int piece, float* dkv_part) {
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const int jl = q4 * 32 + lane;
    const size_t sec = (size_t)N * ldq;
    // row 0 of this warp's 32 key rows in section 0 of the slice
    bf16* wrow0 = d_packed + (size_t)bh * 4 * sec + (size_t)(k0 + q4 * 32) * ldq;
    // 32 columns (16 at head_dim 16) at a time
    constexpr int W = D < 32 ? D : 32;
#pragma unroll
    for (int which = 0; which < 3; ++which) {
        const uint32_t col = which == 0 ? C::C_DK : C::C_DV + (which - 1) * D;
        const float mul = which == 0 ? scale : 1.f;
#pragma unroll
        for (int h = 0; h < D / W; ++h) {
            uint32_t v[W];
            tmem_ld_row<W>(trow + col + W * h, v);
            tmem_wait_ld();
            const uint32_t zero[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
            for (int z = 0; z < W / 16; ++z) tmem_st_32x32b_x16(trow + col + W * h + 16 * z, zero);
            if (which == 2 && h == D / W - 1) {
                // every accumulator column of this thread's row is read and zeroed
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(epi_bar);
            }
            if (piece >= 0) {
                // a piece's partial: [piece][key row][dK | dV_lo | dV_hi] fp32
                float4* o = reinterpret_cast<float4*>(dkv_part + ((size_t)piece * C::BM + jl) * 3 * D + which * D +
                                                      W * h);
#pragma unroll
                for (int e = 0; e < W; e += 4)
                    o[e / 4] = make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                                           __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
            } else {
                uint32_t w[W / 2];
#pragma unroll
                for (int e = 0; e < W / 2; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
                store_rows_staged<W>(stg, w, reinterpret_cast<uint16_t*>(wrow0 + (size_t)(1 + which) * sec) + W * h,
                                     ldq, N - (k0 + q4 * 32), lane);
            }
        }
    }
}

// A work item of the fused kernel: a (batch*head, 128-key tile) unit, or, for
// the units of the last, partial wave, one of tail_f pieces of a unit along
// the query axis (whole 128-query groups); a piece writes its dK/dV as fp32
// partials, summed by the finalize kernel.  nsub 64-query sub-tiles starting
// at sub-tile ubase of the slice.
struct Item {
    int bh, k0, ubase, nsub, piece;
};
__device__ __forceinline__ Item decode_item(int x, int nfull, int tail_f, int nsub_all, int nkt) {
    Item t;
    int unit = x;
    t.ubase = 0;
    t.nsub = nsub_all;
    t.piece = -1;
    if (unit >= nfull) {
        t.piece = unit - nfull;
        unit = nfull + t.piece / tail_f;
        const int p = t.piece % tail_f, ng = (nsub_all + 1) / 2;
        const int gb = p * ng / tail_f, ge = (p + 1) * ng / tail_f;
        t.ubase = 2 * gb;
        t.nsub = min(2 * ge, nsub_all) - t.ubase;
    }
    t.bh = unit / nkt;
    t.k0 = (unit % nkt) * 128;
    return t;
}

// ---------------------------------------------------------------- main kernel
// Persistent: CTA b walks the work items b, b + gridDim.x, ... in turn.  Every
// ring of the CTA (Q/dO stages, S/dP buffers, their barriers, PF, the dS ring,
// the dQ barriers) runs on sub-tile and 128-query-group numbers U and G counted
// across its items, so the producer fetches the next item's stages while the
// current item ends, and the next item's K/V tile, S/dP products and softmax
// overlap the current item's last dQ products, drain and epilogue.  Per item:
// KV (its K/V tile landed) and KVE (the dQ issuer's commit after the item's
// last dQ product: no MMA reads that tile any more); ACC / ACCB (each main
// issuer's commit after its last dV/dK of the item); EPI (the drain warps have
// read the item's dK/dV accumulators, which the next item's first dV/dK
// overwrite).
// CM: dO_lo / dO_hi come as channel-major [d, N] blocks (4-D maps over
// [B][heads][d][N]); else as rows (4-D maps over [B][heads][N][d]).  The
// stage's dO tiles then hold [d][64 queries] (128-byte rows), which the dP^T
// product reads MN-major and the dV product K-major.
template <int D, bool CM>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
bwd_main_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_do_lo, const __grid_constant__ CUtensorMap tm_do_hi,
                const __grid_constant__ CUtensorMap tm_dq, int heads, long long ldq, const float4* __restrict__ stats,
                bf16* __restrict__ d_packed, int N, int nkt, float scale, float scale_log2, int nfull, int tail_f,
                int nitems, float* __restrict__ dkv_part) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = C::SLACK ? reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023))
                             : smem_raw;  // the host checked the base's alignment
    const uint32_t sb = smem_u32(smem);
    Sync sy{sb + C::OFF_BAR, reinterpret_cast<volatile int*>(smem + C::OFF_MISC), &g_tc_error};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsub_all = (N + C::BS - 1) / C::BS;
    // sub-tiles over all of this CTA's items
    int UT = 0;
    for (int x = blockIdx.x; x < nitems; x += gridDim.x) UT += decode_item(x, nfull, tail_f, nsub_all, nkt).nsub;

    if (threadIdx.x == 0) {
        for (int b = 0; b < C::KVBUF; ++b) {
            mbar_init(sy.bar(kv_full(b)), 1);
            mbar_init(sy.bar(kv_empty(b)), 1);
        }
        mbar_init(sy.bar(F_EPI), 128);
        for (int b = 0; b < 2 * C::NB; ++b) {
            mbar_init(sy.bar(F_SFS + b), 1);
            mbar_init(sy.bar(F_SFD + b), 1);
        }
        for (int x = 0; x < kPfRingF; ++x) {
            mbar_init(sy.bar(F_PF + x), 128);
            mbar_init(sy.bar(F_PR + x), 128);
        }
        mbar_init(sy.bar(F_DQF), 1);
        mbar_init(sy.bar(F_DQF + 1), 1);
        mbar_init(sy.bar(F_DQE), 128);
        mbar_init(sy.bar(F_DQE + 1), 128);
        mbar_init(sy.bar(F_ACC), 1);
        mbar_init(sy.bar(F_ACCB), 1);
        mbar_init(sy.bar(F_DQA), 1);
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(sy.bar(F_QF + s), 1);
            mbar_init(sy.bar(F_QE + s), 1);
        }
        *sy.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_kv);
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_do_lo);
        tma_prefetch_desc(&tm_do_hi);
    }
    // the dS ring starts zeroed: a half-filled 128-query group (an item's last)
    // reads a block its second sub-tile did not write (rows of queries past the
    // item, discarded, but finite)
    for (int x = threadIdx.x; x < 4 * 16384 / 16; x += C::THREADS)
        st_shared_v4(sb + C::OFF_DS + 16 * x, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
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
        // Per item: its K/V tile, once no MMA reads the buffer's previous one
        // (KVE of item it - KVBUF), then its Q/dO stages in turn (Q, dO_lo, dO_hi
        // and the sub-tile's statistics: 32 float4 per 64-query sub-tile, padded
        // rows -inf and 0, written by the preprocess kernel), each as soon as the
        // stage is free (QE).  The whole warp waits, lane 0 issues: a single
        // polling lane fed the pipeline measurably later.  With one K/V buffer an
        // item's stages are not fetched before the previous item has finished
        // with its K/V tile; nothing of that item waits for them (the softmax
        // fetches its next sub-tile's statistics early only within an item).
        int last_issued[C::NST];
#pragma unroll
        for (int s = 0; s < C::NST; ++s) last_issued[s] = -1;
        int U = 0, it = 0;
        bool ok = true, dep = false;
        for (int x = blockIdx.x; x < nitems && ok; x += gridDim.x, ++it) {
            const Item t = decode_item(x, nfull, tail_f, nsub_all, nkt);
            const int kvb = it % C::KVBUF;
            if (it >= C::KVBUF && !warp_wait(sy, sy.bar(kv_empty(kvb)), (it / C::KVBUF - 1) & 1, 0, -1)) break;
            if (lane == 0) {
                const uint32_t kvs = sb + kvb * C::KVSET, full = sy.bar(kv_full(kvb));
                mbar_arrive_expect_tx(full, 3 * C::KTILE);
                tma_load_3d(kvs + C::OFF_K, &tm_kv, 0, t.k0, t.bh * 4 + 1, full);
                tma_load_3d(kvs + C::OFF_VL, &tm_kv, 0, t.k0, t.bh * 4 + 2, full);
                tma_load_3d(kvs + C::OFF_VH, &tm_kv, 0, t.k0, t.bh * 4 + 3, full);
            }
            const float4* st_slice = stats + (size_t)t.bh * nsub_all * 32;
            const int hh = t.bh % heads, bb = t.bh / heads;
            for (int u = 0; u < t.nsub; ++u, ++U) {
                const int s = U % C::NST;
                if (!warp_wait(sy, sy.bar(F_QE + s), ((U / C::NST) & 1) ^ 1, 0, U)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t st = sb + C::OFF_STAGE + s * C::STAGE;
                    mbar_arrive_expect_tx(sy.bar(F_QF + s), 3 * C::QTILE + 512);
                    const int q0 = (t.ubase + u) * C::BS;
                    tma_load_3d(st, &tm_q, 0, q0, t.bh * 4 + 0, sy.bar(F_QF + s));
                    tma_load_4d(st + C::QTILE, &tm_do_lo, CM ? q0 : 0, CM ? 0 : q0, hh, bb, sy.bar(F_QF + s));
                    tma_load_4d(st + 2 * C::QTILE, &tm_do_hi, CM ? q0 : 0, CM ? 0 : q0, hh, bb, sy.bar(F_QF + s));
                    if (!dep) {
                        // the statistics come from the preprocess kernel, which
                        // may still be running (programmatic dependent launch)
                        griddep_wait();
                        dep = true;
                    }
                    bulk_load(sb + C::OFF_ST + s * 512, st_slice + (size_t)(t.ubase + u) * 32, 512, sy.bar(F_QF + s));
                }
#pragma unroll
                for (int y = 0; y < C::NST; ++y)
                    if (y == s) last_issued[y] = U;
            }
        }
        __syncwarp();
        if (*sy.abort && lane == 0) {
            // let this CTA's own copies land before its shared memory is released
            // (items 0 .. it-1 were loaded; the latest of each buffer)
            for (int j = it - 1; j >= 0 && j >= it - C::KVBUF; --j)
                wait_drain(sy.bar(kv_full(j % C::KVBUF)), (j / C::KVBUF) & 1);
#pragma unroll
            for (int y = 0; y < C::NST; ++y)
                if (last_issued[y] >= 0) wait_drain(sy.bar(F_QF + y), (last_issued[y] / C::NST) & 1);
        }
    } else if (warp == 1 || warp == 15) {
        // ------------------------------------------------------------ main MMA issuers
        // With two issuers warp 1 takes the even sub-tiles U, warp 15 the odd ones
        // (numbered across items).  Each issues, per sub-tile U of its parity,
        // dV/dK(U) once PF(U) shows P/dS(U) ready (with P_READY: dV(U) and
        // S^T(U + NB) once PR(U) shows P(U) ready, dK(U) and dP^T(U + NB) after
        // PF(U)), and S/dP(U + NB) into the buffer dV/dK(U) just read when U + NB
        // is in the same item: one thread's MMAs run in issue order, so the buffer
        // is reused only after its last reader.  Warp 1 issues each item's first NB S/dP products (the item
        // prologue), after the other issuer's last dV/dK of the previous item
        // (whose buffers they reuse; its QE commit), the item's K/V and stages.
        // While one thread waits for its next PF (such a wait first lets its own
        // MMAs in flight finish), the other's keep the tensor core fed.
        const int par = warp == 1 ? 0 : 1;
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(128, 64, 0, 0);     // S^T: 64 queries
            // dP^T: B = dO rows (K-major), or MN-major from channel-major tiles
            constexpr uint32_t ID_DP = idesc_bf16(128, 64, 0, CM ? 1 : 0);
            // dV_lo | dV_hi: B MN-major (rows), or K-major from channel-major tiles
            constexpr uint32_t ID_DV = idesc_bf16(128, 2 * D, 0, CM ? 0 : 1);
            constexpr uint32_t ID_DK = idesc_bf16(128, D, 0, 1);     // dK: A K-major, B MN-major
            constexpr uint32_t SBO = 8 * C::ROWB;
            constexpr uint32_t KSTEP = (16 * C::ROWB) >> 4;          // 16 rows, in descriptor address units
            // every descriptor is built once; an MMA adds its k-step offset to the address field
            // (of K/V buffer 0; kvo, in descriptor address units, selects the item's)
            const uint64_t dK = smem_desc(sb + C::OFF_K, 16, SBO, C::SW);
            const uint64_t dVL = smem_desc(sb + C::OFF_VL, 16, SBO, C::SW);
            const uint64_t dVH = smem_desc(sb + C::OFF_VH, 16, SBO, C::SW);
            uint32_t kvo = 0;
            const uint64_t dStage0 = smem_desc(sb + C::OFF_STAGE, 16, SBO, C::SW);
            const uint64_t dStage0mn = smem_desc(sb + C::OFF_STAGE + C::QTILE, C::QTILE, SBO, C::SW);
            constexpr uint32_t STAGE_U = C::STAGE >> 4, QTILE_U = C::QTILE >> 4;
            // channel-major dO tiles: [D features][64 queries], 128-byte rows,
            // 128B swizzle.  dP^T reads one as B MN-major (8 feature rows per
            // 1024-byte atom, a K-step of 16 features = 2048 bytes); dV reads the
            // lo and hi tiles, adjacent, as one K-major B of 2D rows (a K-step of
            // 16 queries = 32 bytes inside the row)
            const uint64_t dDoCm = smem_desc(sb + C::OFF_STAGE + C::QTILE, 8192, 1024, 2);
            const uint64_t dDvCm = smem_desc(sb + C::OFF_STAGE + C::QTILE, 16, 1024, 2);

            // S^T(U) and dP^T(U) into the two halves of TMEM buffer U % NB, each with
            // its own barrier.  Their Q/dO stage is known to be loaded: the item
            // prologue waits for it, later the softmax warpgroup that arrives
            // PF(U-NB) has waited for it first.
            auto issue_s = [&](int u) {
                const uint64_t dQs = dStage0 + STAGE_U * (u % C::NST);
                const uint32_t tS = tmem + 128u * (u % C::NB);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_bf16_ss(tS, dK + kvo + 2 * kk, dQs + 2 * kk, ID_S, kk);
                mma_commit(sy.bar(F_SFS + u % (2 * C::NB)));
            };
            auto issue_dp = [&](int u) {
                const uint32_t tDP = tmem + 128u * (u % C::NB) + 64;
                if constexpr (CM) {
                    const uint64_t dLo = dDoCm + STAGE_U * (u % C::NST);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_bf16_ss(tDP, dVL + kvo + 2 * kk, dLo + 128 * kk, ID_DP, kk);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_bf16_ss(tDP, dVH + kvo + 2 * kk, dLo + QTILE_U + 128 * kk, ID_DP, 1);
                } else {
                    const uint64_t dQs = dStage0 + STAGE_U * (u % C::NST);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_bf16_ss(tDP, dVL + kvo + 2 * kk, dQs + QTILE_U + 2 * kk, ID_DP, kk);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_bf16_ss(tDP, dVH + kvo + 2 * kk, dQs + 2 * QTILE_U + 2 * kk, ID_DP, 1);
                }
                mma_commit(sy.bar(F_SFD + u % (2 * C::NB)));
            };
            // dV of sub-tile u (A = P^T from the S half, 64 queries = 4 k-steps),
            // added to the accumulators (which the drain warps zero for each item)
            auto issue_dv = [&](int u) {
                // [dO_lo | dO_hi]: MN-major rows, or K-major channel-major tiles
                const uint64_t dG = (CM ? dDvCm : dStage0mn) + STAGE_U * (u % C::NST);
                constexpr uint32_t DV_STEP = CM ? 2u : KSTEP;
#pragma unroll
                for (int kk = 0; kk < C::BS / 16; ++kk)
                    mma_bf16_ts(tmem + C::C_DV, tmem + 128u * (u % C::NB) + 8 * kk, dG + DV_STEP * kk, ID_DV, 1u);
            };
            // dK of sub-tile u, B = Q.  A = dS^T: with DK_SMEM from its dS ring
            // block blk ([128 keys][64 queries] bf16, 128-byte rows, 128B swizzle:
            // K-major, a k-step of 16 queries = 32 bytes), else from the dP half of
            // its TMEM buffer.  Then the stage (and the block) are free.
            const uint64_t dDSk = smem_desc(sb + C::OFF_DS, 16, 1024, 2);
            auto issue_dk = [&](int u, int blk) {
                const uint64_t dQmn = dStage0 + STAGE_U * (u % C::NST);     // Q rows, MN-major
                if constexpr (C::DK_SMEM) {
                    const uint64_t dA = dDSk + (16384u >> 4) * blk;
#pragma unroll
                    for (int kk = 0; kk < C::BS / 16; ++kk)
                        mma_bf16_ss(tmem + C::C_DK, dA + 2 * kk, dQmn + KSTEP * kk, ID_DK, 1u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < C::BS / 16; ++kk)
                        mma_bf16_ts(tmem + C::C_DK, tmem + 128u * (u % C::NB) + 64 + 8 * kk, dQmn + KSTEP * kk,
                                    ID_DK, 1u);
                }
                mma_commit(sy.bar(F_QE + u % C::NST));
            };
            const uint32_t acc_bar = sy.bar(par == 0 ? F_ACC : F_ACCB);
            bool ok = true;
            // kb: items so far in which the odd issuer has a sub-tile (its ACCB
            // phases: it commits ACCB only for those); G0: the item's first group
            int U0 = 0, G0 = 0, it = 0, kb = 0;
            for (int x = blockIdx.x; x < nitems; x += gridDim.x, ++it) {
                const Item t = decode_item(x, nfull, tail_f, nsub_all, nkt);
                const bool odd_in = !C::TWO_ISSUERS || t.nsub >= 2 || (U0 & 1);
                kvo = (uint32_t)((it % C::KVBUF) * (C::KVSET >> 4));
                if (par == 0) {
                    // item prologue: S/dP of the first NB sub-tiles, into buffers whose
                    // last readers were dV/dK of earlier items: the other issuer's are
                    // done once its latest ACCB phase is (ACCB commits track all its
                    // MMAs; a wait on one of its QE commits could meet a stage barrier
                    // two phases behind with 4 stages)
                    if (C::TWO_ISSUERS && kb > 0) ok = wait_bounded(sy, sy.bar(F_ACCB), (kb - 1) & 1, 1, -1);
                    if (ok) ok = wait_bounded(sy, sy.bar(kv_full(it % C::KVBUF)), (it / C::KVBUF) & 1, 1, -1);
                    for (int j = 0; j < C::NB && j < t.nsub && ok; ++j)
                        ok = wait_bounded(sy, sy.bar(F_QF + (U0 + j) % C::NST), ((U0 + j) / C::NST) & 1, 1, U0 + j);
                    if (!ok) break;
                    tc_fence_after();
                    for (int j = 0; j < C::NB && j < t.nsub; ++j) {
                        issue_s(U0 + j);
                        issue_dp(U0 + j);
                    }
                }
                // PF(U) (with P_READY: PR(U)) also certifies that the stage of U+NB is
                // loaded (the softmax warpgroup waited for it).  S^T(U+NB) follows dV(U), the last reader
                // of the S half, and dP^T(U+NB) follows dK(U), the last reader of the
                // dP half when dK takes dS^T from there (dK first measured faster with
                // the ring too); the softmax of U+NB starts on S^T while dK(U) and
                // dP^T(U+NB) run.  Every dV/dK product accumulates: before its first
                // one of an item a thread waits for EPI phase `it` (phase 0: the drain
                // warps zeroed the accumulators at the start; phase i + 1: they read
                // item i's and zeroed them again).
                bool first = true;
                for (int ul = 0; ul < t.nsub; ++ul) {
                    const int U = U0 + ul;
                    if (C::TWO_ISSUERS && (U & 1) != par) continue;
                    // PF(U), or with P_READY first PR(U): P(U) is in TMEM and the
                    // stage of U+NB is loaded
                    ok = wait_bounded(sy, sy.bar((C::P_READY ? F_PR : F_PF) + U % kPfRingF), (U / kPfRingF) & 1, 1, U);
                    if (ok && first) {
                        ok = wait_bounded(sy, sy.bar(F_EPI), it & 1, 1, U);
                        first = false;
                    }
                    if (!ok) break;
                    tc_fence_after();
                    const bool more = ul + C::NB < t.nsub;
                    issue_dv(U);
                    if (more) issue_s(U + C::NB);
                    if constexpr (C::P_READY) {
                        // PF(U): dS(U) is written and dP^T(U) read
                        ok = wait_bounded(sy, sy.bar(F_PF + U % kPfRingF), (U / kPfRingF) & 1, 1, U);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    issue_dk(U, 2 * ((G0 + (ul >> 1)) & 1) + (ul & 1));
                    if (more) issue_dp(U + C::NB);
                }
                if (!ok) break;
                if (par == 0) {
                    // ACC every item; without a sub-tile, after the zeroing for this
                    // item, so that its phases keep in step with the drain's waits
                    if (first) ok = wait_bounded(sy, sy.bar(F_EPI), it & 1, 1, -1);
                    if (!ok) break;
                    mma_commit(acc_bar);
                } else if (!first) {
                    mma_commit(acc_bar);
                }
                if (odd_in) ++kb;
                U0 += t.nsub;
                G0 += (t.nsub + 1) / 2;
            }
            // all of this thread's MMAs done before TMEM is freed (also on abort)
            const int ncommit = par == 0 ? it : kb;
            if (ok) {
                if (ncommit > 0) wait_drain(acc_bar, (ncommit - 1) & 1);
            } else {
                mma_commit(acc_bar);
                wait_drain(acc_bar, ncommit & 1);
            }
        }
        __syncwarp();
    } else if (warp < 10) {
        // ------------------------------------------------------------ softmax-gradient warpgroups
        // Warpgroup grp takes the sub-tiles U of parity grp (numbered across items).
        // TMEM fragments of the 16x256b shape: in each 16-lane half hb of the
        // warp's lane quarter, thread t holds key rows 16 hb + t/4 and 16 hb + 8 + t/4
        // and, of the sub-tile's 64 queries, the pairs 8k + 2(t%4), +1 (k < 8).  So
        // a thread needs the statistics of 16 queries (8 pairs), which it loads once
        // per sub-tile into registers, instead of all 64.
        const int grp = (warp - 2) >> 2;         // 0: even sub-tiles, 1: odd
        const int q4 = warp & 3;                 // TMEM lane quarter of this warp
        const int tq = lane & 3, tr = lane >> 2;
        const uint64_t cs2 = f2_pack(scale_log2, scale_log2);
        // this thread's 8 query pairs of a stage: {-LSE log2(e) x2, D x2} (the
        // producer writes a stage's statistics before its QF arrive, and the stage
        // is not refilled before this warpgroup's PF arrive for that sub-tile)
        float4 stat[8];
        auto load_stats = [&](int u) {
            const float4* St = reinterpret_cast<const float4*>(smem + C::OFF_ST) + (u % C::NST) * 32 + tq;
#pragma unroll
            for (int k = 0; k < 8; ++k) stat[k] = St[4 * k];
        };
        bool ok = true;
        if (grp < UT) {
            ok = warp_wait(sy, sy.bar(F_QF + grp % C::NST), (grp / C::NST) & 1, 2, grp);
            if (ok) load_stats(grp);
        }
        // the item holding sub-tile U: t, its first sub-tile U0 and group G0
        int xi = blockIdx.x, U0 = 0, G0 = 0;
        Item t = decode_item(xi, nfull, tail_f, nsub_all, nkt);
        for (int U = grp; U < UT && ok; U += 2) {
            while (U >= U0 + t.nsub) {
                U0 += t.nsub;
                G0 += (t.nsub + 1) / 2;
                xi += gridDim.x;
                t = decode_item(xi, nfull, tail_f, nsub_all, nkt);
            }
            const int ul = U - U0, G = G0 + (ul >> 1);
            const int k0 = t.k0;
            const bool full = k0 + C::BM <= N;   // uniform: no padded keys in this tile
            if (ul < 2 && U != grp) {
                // this warpgroup's first sub-tile of a later item: its statistics
                // were not fetched ahead (the stage may load only after the
                // previous item's last sub-tiles)
                ok = warp_wait(sy, sy.bar(F_QF + U % C::NST), (U / C::NST) & 1, 2, U);
                if (!ok) break;
                load_stats(U);
            }
            const int buf = U % C::NB;
            // One round trip for S^T(U) and the dQ product that last read the
            // sub-tile's dS ring block 2 (G & 1) + (ul & 1): dQ(G-2).  The parity
            // test on DQF + (G & 1) is exact: dQ(G-4) was waited for by this
            // warpgroup earlier, and dQ(G) needs PF(U).  (The product is almost
            // always complete by now.)
            const uint32_t bsf = sy.bar(F_SFS + U % (2 * C::NB)), psf = (U / (2 * C::NB)) & 1;
            uint32_t bdq = bsf, pdq = psf;
            if (G >= 2) {
                const int h = G - 2;
                bdq = sy.bar(F_DQF + (h & 1));
                pdq = (h >> 1) & 1;
            }
            // With DK_SMEM the dK products read the dS ring too: before this
            // sub-tile's block is written, the dK of the block's previous
            // sub-tile must be done.  From the item's fifth sub-tile on that is
            // U-4 (the item's groups before its last have two sub-tiles): its
            // QE, waited for here (its next phase needs this warpgroup's
            // PF(U+2)).  Before that it belongs to an earlier item, whose dK
            // products all completed before S^T(U) did: the item prologue
            // followed the prologue thread's own dK products and waited for the
            // other issuer's last ACCB, and every later S^T of the item follows
            // a PF of the item.
            uint32_t bqe = bsf, pqe = psf;
            if (C::DK_SMEM && ul >= 4) {
                bqe = sy.bar(F_QE + (U - 4) % C::NST);
                pqe = ((U - 4) / C::NST) & 1;
            }
            ok = warp_wait_all(sy, bsf, psf, bdq, pdq, bqe, pqe, bsf, psf, 2, U);
            if (!ok) break;
            tc_fence_after();
            const uint32_t ds_blk = sb + C::OFF_DS + 16384 * (2 * (G & 1) + (ul & 1));
            // phase 1: P = exp2(S scale log2(e) - LSE log2(e)) as bf16 pairs, over
            // the S^T columns already read (the dP^T products may still run)
            uint32_t pk[2][2][8];
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                const int r0 = q4 * 32 + 16 * hb + tr;          // key rows r0, r0 + 8 of the tile
                const bool kv0 = full || k0 + r0 < N, kv1 = full || k0 + r0 + 8 < N;
                const uint32_t tS = tmem + ((uint32_t)(q4 * 32 + 16 * hb) << 16) + 128u * buf;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t sr[16];
                    tmem_ld_16x256b_x4(tS + 32 * c, sr);
                    tmem_wait_ld();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const float4 st = stat[4 * c + kk];
                        const uint64_t nl = f2_pack(st.x, st.y);
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const uint64_t x = f2_fma(f2_pack(__uint_as_float(sr[4 * kk + 2 * e]),
                                                              __uint_as_float(sr[4 * kk + 2 * e + 1])),
                                                      cs2, nl);
                            float x0, x1;
                            f2_unpack(x, x0, x1);
                            pk[hb][c][2 * kk + e] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
                        }
                    }
                    if (!full) {
                        // keys past the slice's end (its last tile only): P = 0
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            if (!kv0) pk[hb][c][2 * kk] = 0u;
                            if (!kv1) pk[hb][c][2 * kk + 1] = 0u;
                        }
                    }
                    // packed pair 4k + t%4 over the S^T columns
                    tmem_st_16x128b_x4(tS + 16 * c, pk[hb][c]);
                }
            }
            if constexpr (C::P_READY) {
                // P(U) is in TMEM: the issuer of U may start dV(U) and S^T(U+NB)
                // (PR), once the stage of U+NB is loaded (waited for here in its
                // stead)
                if (ul + C::NB < t.nsub)
                    ok = warp_wait(sy, sy.bar(F_QF + (U + C::NB) % C::NST), ((U + C::NB) / C::NST) & 1, 2, U);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(sy.bar(F_PR + U % kPfRingF));
                if (!ok) {
                    mbar_arrive(sy.bar(F_PF + U % kPfRingF));
                    break;
                }
            }
            // phase 2: dS = P (dP - D), with P as rounded for the dV product
            ok = warp_wait(sy, sy.bar(F_SFD + U % (2 * C::NB)), (U / (2 * C::NB)) & 1, 2, U);
            if (!ok) {
                mbar_arrive(sy.bar(F_PF + U % kPfRingF));
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                const uint32_t tDP = tmem + ((uint32_t)(q4 * 32 + 16 * hb) << 16) + 128u * buf + 64;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t pr[16];
                    tmem_ld_16x256b_x4(tDP + 32 * c, pr);
                    tmem_wait_ld();
                    uint32_t dk[8];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const float4 st = stat[4 * c + kk];
                        const uint64_t dd = f2_pack(st.z, st.w);
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const uint64_t t = f2_sub(f2_pack(__uint_as_float(pr[4 * kk + 2 * e]),
                                                              __uint_as_float(pr[4 * kk + 2 * e + 1])),
                                                      dd);
                            float t0, t1;
                            f2_unpack(t, t0, t1);
                            // dP - D rounded to bf16, times the bf16 P pair
                            dk[2 * kk + e] = bf16x2_mul(pk[hb][c][2 * kk + e], pack_bf16x2(t0, t1));
                        }
                    }
                    // dS over the dP^T columns already read, for the dK product
                    if constexpr (!C::DK_SMEM) tmem_st_16x128b_x4(tDP + 16 * c, dk);
                    // dS to the 128B-swizzled ring block (row = key, 16-byte chunk =
                    // query / 8 xor row % 8) for the dQ product (and dK with
                    // DK_SMEM).  The fragment is the MMA layout of 8x8 tiles (tile
                    // kk: key rows 16 hb + 8 e + 0..7, queries 8 (4 c + kk) + 0..7), so
                    // one stmatrix per e stores four tiles; lane l addresses row
                    // l % 8 of tile l / 8 (the XOR spreads a tile's rows over the
                    // banks)
                    {
                        const int tm = lane >> 3, rr = lane & 7;
                        const uint32_t row = ds_blk + (uint32_t)(q4 * 32 + 16 * hb + rr) * 128u +
                                             ((uint32_t)((4 * c + tm) ^ rr) << 4);
                        stmatrix_x4(row, dk[0], dk[2], dk[4], dk[6]);
                        stmatrix_x4(row + 8 * 128, dk[1], dk[3], dk[5], dk[7]);
                    }
                }
            }
            tmem_wait_st();
            tc_fence_before();
            fence_proxy_async_smem();
            if constexpr (C::P_READY) {
                // the stage of U+2, this warpgroup's next sub-tile, whose
                // statistics it loads now, when U+2 is in this item (the stage of
                // U+NB was waited for before PR)
                if (ul + 2 < t.nsub)
                    ok = warp_wait(sy, sy.bar(F_QF + (U + 2) % C::NST), ((U + 2) / C::NST) & 1, 2, U);
            } else {
                // One round trip for: (a) a stand-in wait for the MMA issuer of U
                // (see its loop): the stage of U+NB is loaded, when U+NB is in this
                // item; (b) the stage of U+2, this warpgroup's next sub-tile, whose
                // statistics it loads now, when U+2 is in this item.
                const bool v0 = ul + C::NB < t.nsub, v1 = ul + 2 < t.nsub;
                uint32_t b0 = sy.bar(F_QF + (U + C::NB) % C::NST), p0 = ((U + C::NB) / C::NST) & 1;
                uint32_t b1 = sy.bar(F_QF + (U + 2) % C::NST), p1 = ((U + 2) / C::NST) & 1;
                if (v0 || v1) {
                    // a phase that is not needed is replaced by one that is
                    if (!v0) { b0 = b1; p0 = p1; }
                    if (!v1) { b1 = b0; p1 = p0; }
                    ok = warp_wait_all(sy, b0, p0, b1, p1, b0, p0, b0, p0, 2, U);
                }
            }
            if (ok && ul + 2 < t.nsub) load_stats(U + 2);
            mbar_arrive(sy.bar(F_PF + U % kPfRingF));
            if (!ok) break;
        }
    } else if (warp < 14) {
        // ------------------------------------------------------------ dQ drain, then each item's dK/dV epilogue
        const int q4 = warp & 3;
        const int il = q4 * 32 + lane;           // query row within the 128-query group
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        const bool elected = warp == 10 && lane == 0;
        // row il of a box of BOXC fp32 columns, swizzled as the tensor map expects
        // (16-byte chunk c of a row at c xor the row bits above the 128-byte line)
        constexpr uint32_t RB = C::BOXC * 4, M = RB == 128 ? 7u : RB == 64 ? 3u : 1u;
        {
            // the dK/dV accumulators start at zero (EPI phase 0); the issuers'
            // products all accumulate
            const uint32_t zero[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
            for (int z = 0; z < 3 * D / 16; ++z) tmem_st_32x32b_x16(trow + C::C_DV + 16 * z, zero);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(sy.bar(F_EPI));
        }
        griddep_wait();                          // dq_acc is zeroed by the preprocess kernel
        bool okd = true;
        int G0 = 0, U0 = 0, it = 0, kb = 0;
        for (int x = blockIdx.x; x < nitems && okd; x += gridDim.x, ++it) {
            const Item t = decode_item(x, nfull, tail_f, nsub_all, nkt);
            const int ngrp = (t.nsub + 1) / 2;
            // the odd issuer commits ACCB only for items it has a sub-tile in
            const bool odd_in = !C::TWO_ISSUERS || t.nsub >= 2 || (U0 & 1);
            if (odd_in) ++kb;
            for (int gl = 0; gl < ngrp; ++gl) {
                const int G = G0 + gl;
                okd = warp_wait(sy, sy.bar(F_DQF + (G & 1)), (G >> 1) & 1, 3, G);
                // the four drain warps decide together (they meet at named barriers below)
                okd = named_bar_and(2, 128, okd);
                if (!okd) break;
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < D / C::BOXC; ++h) {
                    uint32_t v[C::BOXC];
                    tmem_ld_row<C::BOXC>(trow + C::C_DQ + C::BOXC * h, v);
                    tmem_wait_ld();
                    if (h == D / C::BOXC - 1) {
                        // the group's accumulator is read
                        tc_fence_before();
                        mbar_arrive(sy.bar(F_DQE + (G & 1)));
                    }
                    // staging buffer of box b: the reduce that last read it (box b - NDQS)
                    // must be done reading
                    const int bx = G * (D / C::BOXC) + h;
                    const uint32_t buf = sb + C::OFF_DQS + (bx % C::NDQS) * C::DQS_BYTES;
                    if (elected) bulk_wait_group_read<C::NDQS - 1>();
                    named_bar_sync(1, 128);
#pragma unroll
                    for (int c = 0; c < C::BOXC / 4; ++c) {
                        const uint32_t a = (uint32_t)il * RB + 16u * c;
                        st_shared_v4(buf + (a ^ (((a >> 7) & M) << 4)), v[4 * c], v[4 * c + 1], v[4 * c + 2],
                                     v[4 * c + 3]);
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(1, 128);
                    // rows past N lie outside the tensor and are skipped
                    if (elected) {
                        tma_reduce_add_3d(&tm_dq, buf, h * C::BOXC, (t.ubase / 2 + gl) * 128, t.bh);
                        bulk_commit_group();
                    }
                }
            }
            if (!okd) break;
            // epilogue: dK, dV_lo, dV_hi rows of this warp's 32 keys, once every main
            // MMA of the item is done; the staging buffers are free once the last
            // reduce read them.  EPI: the accumulators are read.
            okd = warp_wait(sy, sy.bar(F_ACC), it & 1, 3, -1) &&
                  (!C::TWO_ISSUERS || !odd_in || warp_wait(sy, sy.bar(F_ACCB), (kb - 1) & 1, 3, -1));
            okd = named_bar_and(2, 128, okd);
            if (!okd) break;
            if (elected) bulk_wait_group_read<0>();
            named_bar_sync(1, 128);
            tc_fence_after();
            dkdv_epilogue<D, C>(tmem, q4, lane, sb + C::OFF_DQS + 2048u * (warp - 10), sy.bar(F_EPI), d_packed,
                                t.bh, t.k0, N, ldq, scale, t.piece, dkv_part);
            G0 += ngrp;
            U0 += t.nsub;
        }
        // every reduce has written global memory and read its staging buffer
        if (elected) bulk_wait_group<0>();
    } else if (warp == 14) {
        // ------------------------------------------------------------ dQ issuer
        // dQ of the 128-query group G = an item's sub-tiles 2g, 2g+1: A = dS
        // (queries x keys) read MN-major from the group's two dS^T blocks 2 (G & 1)
        // and 2 (G & 1) + 1 (16 KB apart), B = K rows (MN-major).  It waits for the
        // group's softmax (PF) and for the drain to have read group G-1 (DQE).  A
        // PF phase cannot run a full ring ahead of this thread: the softmax of a
        // sub-tile of group G+2 first waits for DQF(G).  After an item's last group
        // it commits the KVE of the item's K/V buffer: no MMA reads the item's K/V
        // tile any more (the item's S/dP products completed before its softmax,
        // which this thread waited for).
        if (lane == 0) {
            constexpr uint32_t ID_DQ = idesc_bf16(128, D, 1, 1);
            constexpr uint32_t KSTEP = (16 * C::ROWB) >> 4;
            constexpr uint32_t BLK_U = 16384 >> 4;
            const uint64_t dK0 = smem_desc(sb + C::OFF_K, 16, 8 * C::ROWB, C::SW);
            const uint64_t dDS0mn = smem_desc(sb + C::OFF_DS, 16384, 1024, 2);
            bool ok = true;
            int U0 = 0, G0 = 0;
            for (int x = blockIdx.x, it = 0; x < nitems && ok; x += gridDim.x, ++it) {
                const Item t = decode_item(x, nfull, tail_f, nsub_all, nkt);
                const int ngrp = (t.nsub + 1) / 2;
                const uint64_t dK = dK0 + (uint32_t)((it % C::KVBUF) * (C::KVSET >> 4));
                const int nkk = (min(C::BM, N - t.k0) + 15) / 16;
                for (int gl = 0; gl < ngrp; ++gl) {
                    const int G = G0 + gl, u0 = U0 + 2 * gl, u1 = u0 + 1;
                    ok = wait_bounded(sy, sy.bar(F_PF + u0 % kPfRingF), (u0 / kPfRingF) & 1, 5, u0);
                    if (ok && 2 * gl + 1 < t.nsub)
                        ok = wait_bounded(sy, sy.bar(F_PF + u1 % kPfRingF), (u1 / kPfRingF) & 1, 5, u1);
                    // the drain of group G-1 (this thread waited for G-2's before
                    // issuing dQ(G-1); group G+1's drain needs dQ(G+1))
                    if (ok && G > 0) ok = wait_bounded(sy, sy.bar(F_DQE + ((G - 1) & 1)), ((G - 1) >> 1) & 1, 5, G);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t dA = dDS0mn + BLK_U * (2 * (G & 1));
                    // K = the tile's keys: k-steps past the last key that exists add
                    // nothing (its dS and K rows are zero), so a ragged last tile
                    // (16 keys at N = 400) takes one MMA here instead of eight
#pragma unroll
                    for (int kk = 0; kk < C::BM / 16; ++kk)
                        if (kk < nkk) mma_bf16_ss(tmem + C::C_DQ, dA + 128 * kk, dK + KSTEP * kk, ID_DQ, kk);
                    mma_commit(sy.bar(F_DQF + (G & 1)));
                }
                if (!ok) break;
                mma_commit(sy.bar(kv_empty(it % C::KVBUF)));
                U0 += t.nsub;
                G0 += ngrp;
            }
            // this thread's MMAs are done before TMEM is freed (also on abort)
            mma_commit(sy.bar(F_DQA));
            wait_drain(sy.bar(F_DQA), 0);
        }
        __syncwarp();
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---------------------------------------------------------------- dK/dV pass (deterministic mode)
// The key-outer pass without its dQ work: the same walk over 64-query
// sub-tiles, but P^T and dS^T both stay in TMEM (P over the S^T columns, dS
// over the dP^T columns) as the A operands of the dV and dK MMAs, so the
// softmax warps issue no shared-memory stores; dK and dV accumulate in TMEM in
// a fixed order.  dQ comes from the query-outer pass (tc_dq.cu).
template <int D>
struct CfgS {
    static constexpr int BM = 128, BS = 64;
    static constexpr int ROWB = D * 2;
    static constexpr int KTILE = BM * ROWB, QTILE = BS * ROWB;
    static constexpr int NB = D <= 32 ? 3 : 2;    // S^T/dP^T buffers in TMEM
    static constexpr int NST = D <= 32 ? 6 : 4;   // Q/dO stages (> NB)
    static constexpr uint32_t SW = D == 64 ? 2u : D == 32 ? 4u : 6u;
    static constexpr int OFF_K = 0, OFF_VL = KTILE, OFF_VH = 2 * KTILE;
    static constexpr int OFF_STAGE = 3 * KTILE, STAGE = 3 * QTILE;
    static constexpr int OFF_L2 = OFF_STAGE + NST * STAGE;
    static constexpr int OFF_DD = OFF_L2 + NST * 256;
    static constexpr int OFF_BAR = OFF_DD + NST * 256;
    static constexpr int OFF_MISC = OFF_BAR + 256;
    static constexpr int USED = OFF_MISC + 64;
    static constexpr int SMEM = (USED + 1024) > 118784 ? (USED + 1024) : 118784;
    static constexpr uint32_t C_DV = 128 * NB, C_DK = C_DV + 2 * D;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(C_DK + D <= TMEM_COLS, "TMEM budget");
    static_assert(NST > NB, "the softmax's wait for the stage of u+NB would wait on its own release");
    static_assert(USED + 1024 <= 232448, "shared memory budget");
};
constexpr int kThreadsS = 320;

template <int D>
__global__ void __launch_bounds__(kThreadsS, 1)
bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_do_lo, const __grid_constant__ CUtensorMap tm_do_hi,
                const float* __restrict__ lse, const float* __restrict__ Drow, bf16* __restrict__ d_packed, int N,
                int nkt, float scale, float scale_log2) {
    using C = CfgS<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    Sync sy{sb + C::OFF_BAR, reinterpret_cast<volatile int*>(smem + C::OFF_MISC), &g_tc_error};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x / nkt, kt = blockIdx.x % nkt;
    const int k0 = kt * C::BM;
    const int nsub = (N + C::BS - 1) / C::BS;

    if (threadIdx.x == 0) {
        mbar_init(sy.bar(B_KV), 1);
        for (int b = 0; b < C::NB; ++b) mbar_init(sy.bar(B_SF + b), 1);
        for (int x = 0; x < kPfRing; ++x) mbar_init(sy.bar(B_PF + x), 128);
        mbar_init(sy.bar(B_ACC), 1);
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(sy.bar(B_QF + s), 32);
            mbar_init(sy.bar(B_QE + s), 1);
        }
        *sy.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_kv);
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_do_lo);
        tma_prefetch_desc(&tm_do_hi);
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
        int last_issued[C::NST];
#pragma unroll
        for (int s = 0; s < C::NST; ++s) last_issued[s] = -1;
        if (lane == 0) {
            mbar_arrive_expect_tx(sy.bar(B_KV), 3 * C::KTILE);
            tma_load_3d(sb + C::OFF_K, &tm_kv, 0, k0, bh * 4 + 1, sy.bar(B_KV));
            tma_load_3d(sb + C::OFF_VL, &tm_kv, 0, k0, bh * 4 + 2, sy.bar(B_KV));
            tma_load_3d(sb + C::OFF_VH, &tm_kv, 0, k0, bh * 4 + 3, sy.bar(B_KV));
        }
        float* L2s = reinterpret_cast<float*>(smem + C::OFF_L2);
        float* Ds = reinterpret_cast<float*>(smem + C::OFF_DD);
        int s = 0, ph = 0;
        for (int u = 0; u < nsub; ++u) {
            if (!warp_wait(sy, sy.bar(B_QE + s), ph ^ 1, 0, u)) break;
            if (lane == 0) {
                const uint32_t st = sb + C::OFF_STAGE + s * C::STAGE;
                mbar_expect_tx(sy.bar(B_QF + s), 3 * C::QTILE);
                tma_load_3d(st, &tm_q, 0, u * C::BS, bh * 4 + 0, sy.bar(B_QF + s));
                tma_load_3d(st + C::QTILE, &tm_do_lo, 0, u * C::BS, bh, sy.bar(B_QF + s));
                tma_load_3d(st + 2 * C::QTILE, &tm_do_hi, 0, u * C::BS, bh, sy.bar(B_QF + s));
            }
#pragma unroll
            for (int x = 0; x < C::NST; ++x)
                if (x == s) last_issued[x] = u;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int q = lane * 2 + e;
                const int i = u * C::BS + q;
                const bool v = i < N;
                L2s[s * 64 + q] = v ? lse[(size_t)bh * N + i] * kLog2e : INFINITY;
                Ds[s * 64 + q] = v ? Drow[(size_t)bh * N + i] : 0.f;
            }
            mbar_arrive(sy.bar(B_QF + s));
            if (++s == C::NST) { s = 0; ph ^= 1; }
        }
        __syncwarp();
        if (*sy.abort && lane == 0) {
            wait_drain(sy.bar(B_KV), 0);
#pragma unroll
            for (int x = 0; x < C::NST; ++x)
                if (last_issued[x] >= 0) wait_drain(sy.bar(B_QF + x), (last_issued[x] / C::NST) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(128, 64, 0, 0);
            constexpr uint32_t ID_DV = idesc_bf16(128, 2 * D, 0, 1);
            constexpr uint32_t ID_DK = idesc_bf16(128, D, 0, 1);
            constexpr uint32_t SBO = 8 * C::ROWB;
            constexpr uint32_t KSTEP = (16 * C::ROWB) >> 4;
            constexpr uint32_t STAGE_U = C::STAGE >> 4, QTILE_U = C::QTILE >> 4;
            const uint64_t dK = smem_desc(sb + C::OFF_K, 16, SBO, C::SW);
            const uint64_t dVL = smem_desc(sb + C::OFF_VL, 16, SBO, C::SW);
            const uint64_t dVH = smem_desc(sb + C::OFF_VH, 16, SBO, C::SW);
            const uint64_t dStage0 = smem_desc(sb + C::OFF_STAGE, 16, SBO, C::SW);
            const uint64_t dStage0mn = smem_desc(sb + C::OFF_STAGE + C::QTILE, C::QTILE, SBO, C::SW);
            auto issue_s_dp = [&](int u) {
                const int s = u % C::NST;
                const uint64_t dQs = dStage0 + STAGE_U * s;
                const uint32_t tS = tmem + 128u * (u % C::NB), tDP = tS + 64;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_bf16_ss(tS, dK + 2 * kk, dQs + 2 * kk, ID_S, kk);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_ss(tDP, dVL + 2 * kk, dQs + QTILE_U + 2 * kk, ID_S, kk);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_ss(tDP, dVH + 2 * kk, dQs + 2 * QTILE_U + 2 * kk, ID_S, 1);
                mma_commit(sy.bar(B_SF + u % C::NB));
            };
            bool ok = wait_bounded(sy, sy.bar(B_KV), 0, 1, -1);
            for (int u = 0; u < C::NB && u < nsub && ok; ++u) ok = wait_bounded(sy, sy.bar(B_QF + u), 0, 1, u);
            if (ok) {
                tc_fence_after();
                for (int u = 0; u < C::NB && u < nsub; ++u) issue_s_dp(u);
            }
            for (int u = 0; u < nsub && ok; ++u) {
                const int b = u % C::NB, s = u % C::NST;
                ok = wait_bounded(sy, sy.bar(B_PF + u % kPfRing), (u / kPfRing) & 1, 1, u);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dGmn = dStage0mn + STAGE_U * s;
                const uint64_t dQmn = dStage0 + STAGE_U * s;
                const uint32_t tP = tmem + 128u * b, tDS = tP + 64;
#pragma unroll
                for (int kk = 0; kk < C::BS / 16; ++kk) {
                    const uint32_t acc = (u > 0 || kk > 0) ? 1u : 0u;
                    mma_bf16_ts(tmem + C::C_DV, tP + 8 * kk, dGmn + KSTEP * kk, ID_DV, acc);
                    mma_bf16_ts(tmem + C::C_DK, tDS + 8 * kk, dQmn + KSTEP * kk, ID_DK, acc);
                }
                mma_commit(sy.bar(B_QE + s));
                if (u + C::NB < nsub) issue_s_dp(u + C::NB);
            }
            mma_commit(sy.bar(B_ACC));
            if (!ok) wait_drain(sy.bar(B_ACC), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax-gradient warpgroups
        const int grp = (warp - 2) >> 2;
        const int q4 = warp & 3;
        const int jl = q4 * 32 + lane;
        const bool kvalid = k0 + jl < N;
        const bool full = k0 + C::BM <= N;
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        bool ok = true;
        for (int u = grp; u < nsub; u += 2) {
            const int s = u % C::NST, buf = u % C::NB;
            ok = warp_wait(sy, sy.bar(B_SF + buf), (u / C::NB) & 1, 2, u) &&
                 warp_wait(sy, sy.bar(B_QF + s), (u / C::NST) & 1, 2, u);
            if (!ok) break;
            tc_fence_after();
            const float* L2s = reinterpret_cast<const float*>(smem + C::OFF_L2) + s * 64;
            const float* Ds = reinterpret_cast<const float*>(smem + C::OFF_DD) + s * 64;
            const uint32_t tS = trow + 128u * buf, tDP = tS + 64;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                uint32_t sr[32], pr[32];
                tmem_ld_32x32b_x32(tS + 32 * c, sr);
                tmem_ld_32x32b_x32(tDP + 32 * c, pr);
                tmem_wait_ld();
                uint32_t pk[16], dk[16];
                if (full)
                    softmax_vals<false>(sr, pr, L2s + 32 * c, Ds + 32 * c, scale_log2, kvalid, pk, dk);
                else
                    softmax_vals<true>(sr, pr, L2s + 32 * c, Ds + 32 * c, scale_log2, kvalid, pk, dk);
                // P over the S^T columns, dS over the dP^T columns (chunk c's values are in registers)
                tmem_st_32x32b_x16(tS + 16 * c, pk);
                tmem_st_32x32b_x16(tDP + 16 * c, dk);
            }
            tmem_wait_st();
            tc_fence_before();
            if (u + C::NB < nsub)
                ok = warp_wait(sy, sy.bar(B_QF + (u + C::NB) % C::NST), ((u + C::NB) / C::NST) & 1, 2, u);
            mbar_arrive(sy.bar(B_PF + u % kPfRing));
            if (!ok) break;
        }
        if (grp == 0) {
            if (ok) ok = warp_wait(sy, sy.bar(B_ACC), 0, 2, nsub);
            if (ok) {
                tc_fence_after();
                uint32_t v[D];
                const size_t sec = (size_t)N * D;
                bf16* out = d_packed + (size_t)bh * 4 * sec + (size_t)(k0 + jl) * D;
#pragma unroll
                for (int which = 0; which < 3; ++which) {
                    const uint32_t col = which == 0 ? C::C_DK : C::C_DV + (which - 1) * D;
                    const float mul = which == 0 ? scale : 1.f;
                    tmem_ld_row<D>(trow + col, v);
                    tmem_wait_ld();
                    if (kvalid) {
                        bf16* o = out + (size_t)(1 + which) * sec;
#pragma unroll
                        for (int e = 0; e < D; e += 8) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(v[e + 0]) * mul, __uint_as_float(v[e + 1]) * mul);
                            w.y = pack_bf16x2(__uint_as_float(v[e + 2]) * mul, __uint_as_float(v[e + 3]) * mul);
                            w.z = pack_bf16x2(__uint_as_float(v[e + 4]) * mul, __uint_as_float(v[e + 5]) * mul);
                            w.w = pack_bf16x2(__uint_as_float(v[e + 6]) * mul, __uint_as_float(v[e + 7]) * mul);
                            *reinterpret_cast<uint4*>(o + e) = w;
                        }
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

// ---------------------------------------------------------------- bounded-wait self-test
// One CTA waits, through the same bounded wait as the backward kernel, on a
// barrier that nothing arrives on, with a short limit: the wait gives up, the
// device error word is set, and the kernel returns normally.
__global__ void wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        Sync sy{smem_u32(&bar), &abort_flag, &g_tc_error};
        wait_slow(sy, smem_u32(&bar), 0, 4, 0, limit_ns);
    }
}

// ---------------------------------------------------------------- D and dQ-accumulator reset
template <int D>
__global__ void __launch_bounds__(256)
pre_kernel(const bf16* __restrict__ o_lo, const bf16* __restrict__ o_hi, const bf16* __restrict__ do_lo,
           const bf16* __restrict__ do_hi, float* __restrict__ Drow, float* __restrict__ dq_acc, long long rows) {
    constexpr int TPR = D / 8;                // threads per row, 8 bf16 (16 B) each
    constexpr int RPB = 256 / TPR;
    const long long row = (long long)blockIdx.x * RPB + threadIdx.x / TPR;
    const int part = threadIdx.x % TPR;
    float acc = 0.f;
    if (row < rows) {
        const size_t off = (size_t)row * D + part * 8;
        const uint4 a = *reinterpret_cast<const uint4*>(o_lo + off);
        const uint4 b = *reinterpret_cast<const uint4*>(do_lo + off);
        const uint4 c = *reinterpret_cast<const uint4*>(o_hi + off);
        const uint4 d = *reinterpret_cast<const uint4*>(do_hi + off);
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
        const __nv_bfloat162* pc = reinterpret_cast<const __nv_bfloat162*>(&c);
        const __nv_bfloat162* pd = reinterpret_cast<const __nv_bfloat162*>(&d);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 fa = __bfloat1622float2(pa[k]), fb = __bfloat1622float2(pb[k]);
            const float2 fc = __bfloat1622float2(pc[k]), fd = __bfloat1622float2(pd[k]);
            acc = fmaf(fa.x, fb.x, acc);
            acc = fmaf(fa.y, fb.y, acc);
            acc = fmaf(fc.x, fd.x, acc);
            acc = fmaf(fc.y, fd.y, acc);
        }
        if (dq_acc) {  // null in the two-pass mode, which has no dQ accumulator
            float4* z = reinterpret_cast<float4*>(dq_acc + (size_t)row * D);
#pragma unroll
            for (int k = part; k < D / 4; k += TPR) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, TPR);
    if (row < rows && part == 0) Drow[row] = acc;
}

// ---------------------------------------------------------------- statistics for the fused kernel
// Per (batch*head) slice, its queries padded to whole 64-query sub-tiles
// (npad = 64 * ceil(N / 64)): for each query pair c one float4
//   {-LSE_2c log2(e), -LSE_2c+1 log2(e), D_2c, D_2c+1},  D_i = <dO_lo, O_lo> + <dO_hi, O_hi>
// with -inf and 0 for padded queries (so P = 0 there), the layout the fused
// kernel copies into shared memory per sub-tile; also zeroes the dQ accumulator.
template <int D>
__global__ void __launch_bounds__(256)
pre_stats_kernel(const bf16* __restrict__ o_lo, const bf16* __restrict__ o_hi, const bf16* __restrict__ do_lo,
                 const bf16* __restrict__ do_hi, const float* __restrict__ lse, float4* __restrict__ stats,
                 float* __restrict__ dq_acc, long long rows_pad, int N, int npad) {
    // the fused kernel may be scheduled once every block of this one has
    // started; it waits for this grid's results before it reads them
    griddep_launch_dependents();
    constexpr int TPR = D / 8;                // threads per row, 8 bf16 (16 B) each
    constexpr int RPB = 256 / TPR;
    const long long row = (long long)blockIdx.x * RPB + threadIdx.x / TPR;
    const int part = threadIdx.x % TPR;
    const long long bh = row / npad;
    const int i = (int)(row % npad);
    const bool valid = row < rows_pad && i < N;
    float acc = 0.f;
    if (valid) {
        const size_t off = ((size_t)bh * N + i) * D + part * 8;
        const uint4 a = *reinterpret_cast<const uint4*>(o_lo + off);
        const uint4 b = *reinterpret_cast<const uint4*>(do_lo + off);
        const uint4 c = *reinterpret_cast<const uint4*>(o_hi + off);
        const uint4 d = *reinterpret_cast<const uint4*>(do_hi + off);
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
        const __nv_bfloat162* pc = reinterpret_cast<const __nv_bfloat162*>(&c);
        const __nv_bfloat162* pd = reinterpret_cast<const __nv_bfloat162*>(&d);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 fa = __bfloat1622float2(pa[k]), fb = __bfloat1622float2(pb[k]);
            const float2 fc = __bfloat1622float2(pc[k]), fd = __bfloat1622float2(pd[k]);
            acc = fmaf(fa.x, fb.x, acc);
            acc = fmaf(fa.y, fb.y, acc);
            acc = fmaf(fc.x, fd.x, acc);
            acc = fmaf(fc.y, fd.y, acc);
        }
        float4* z = reinterpret_cast<float4*>(dq_acc + ((size_t)bh * N + i) * D);
#pragma unroll
        for (int k = part; k < D / 4; k += TPR) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, TPR);
    const float nl = valid ? -lse[(size_t)bh * N + i] * kLog2e : -INFINITY;
    // the odd row of the pair is the next TPR lanes of the same warp (npad and
    // the rows of a block are even)
    const float nl1 = __shfl_down_sync(0xffffffffu, nl, TPR);
    const float d1 = __shfl_down_sync(0xffffffffu, acc, TPR);
    if (row < rows_pad && part == 0 && (i & 1) == 0) stats[row >> 1] = make_float4(nl, nl1, acc, d1);
}

// The same statistics for strided layouts (psa_attn_bwd_ex): O rows `ldo`
// elements apart, dO_lo / dO_hi read through views.  One thread per query row;
// a channel-major dO view makes consecutive threads read consecutive positions.
template <int D>
__global__ void __launch_bounds__(256)
pre_stats_view_kernel(const bf16* __restrict__ o_lo, const bf16* __restrict__ o_hi, long long ldo, View vlo,
                      View vhi, int heads, const float* __restrict__ lse, float4* __restrict__ stats,
                      float* __restrict__ dq_acc, long long rows_pad, int N, int npad) {
    griddep_launch_dependents();
    const long long row = (long long)blockIdx.x * 256 + threadIdx.x;
    const long long bh = row / npad;
    const int i = (int)(row % npad);
    const bool valid = row < rows_pad && i < N;
    float acc = 0.f;
    if (valid) {
        const long long b = bh / heads, h = bh % heads;
        const bf16* gl = static_cast<const bf16*>(vlo.base) + b * vlo.sB + h * vlo.sH + (long long)i * vlo.sN;
        const bf16* gh = static_cast<const bf16*>(vhi.base) + b * vhi.sB + h * vhi.sH + (long long)i * vhi.sN;
        const bf16* ol = o_lo + ((size_t)bh * N + i) * ldo;
        const bf16* oh = o_hi + ((size_t)bh * N + i) * ldo;
#pragma unroll 8
        for (int j = 0; j < D; ++j) {
            acc = fmaf(__bfloat162float(ol[j]), __bfloat162float(gl[j * vlo.sJ]), acc);
            acc = fmaf(__bfloat162float(oh[j]), __bfloat162float(gh[j * vhi.sJ]), acc);
        }
        float4* z = reinterpret_cast<float4*>(dq_acc + ((size_t)bh * N + i) * D);
#pragma unroll
        for (int k = 0; k < D / 4; ++k) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float nl = valid ? -lse[(size_t)bh * N + i] * kLog2e : -INFINITY;
    // the odd row of the pair is the next lane (npad and 256 are even)
    const float nl1 = __shfl_down_sync(0xffffffffu, nl, 1);
    const float d1 = __shfl_down_sync(0xffffffffu, acc, 1);
    if (row < rows_pad && (i & 1) == 0) stats[row >> 1] = make_float4(nl, nl1, acc, d1);
}

// ---------------------------------------------------------------- dQ = scale * acc -> bf16
// Blocks [0, nmain) convert dQ: R passes of 256 16-byte output parts each, all
// loads of a thread issued first.  Blocks from nmain on write the dK, dV_lo,
// dV_hi rows of the split units, one part per thread.
template <int D, int R>
__global__ void __launch_bounds__(256)
dq_finalize_kernel(const float* __restrict__ dq_acc, bf16* __restrict__ d_packed, long long ldq, long long rows,
                   int N, float scale, const float* __restrict__ dkv_part, int nfull, int ntail, int tail_f,
                   int nkt, int nmain) {
    griddep_wait();             // the fused kernel's dQ sums and partials
    constexpr int PPR = D / 8;  // 8-element parts per row
    if ((int)blockIdx.x >= nmain) {
        // dK, dV_lo, dV_hi of the split units: the sum of their pieces'
        // partials, in piece order
        const long long t = (long long)(blockIdx.x - nmain) * 256 + threadIdx.x;
        if (t >= (long long)ntail * 128 * 3 * PPR) return;
        const int part = (int)(t % PPR);
        const int which = (int)(t / PPR % 3);
        const int jl = (int)(t / (3 * PPR) % 128);
        const int r = (int)(t / (3 * PPR * 128));
        const int unit = nfull + r, bh = unit / nkt, key = (unit % nkt) * 128 + jl;
        if (key >= N) return;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int p = 0; p < tail_f; ++p) {
            const float4* src = reinterpret_cast<const float4*>(
                dkv_part + ((size_t)(r * tail_f + p) * 128 + jl) * 3 * D + which * D + part * 8);
            const float4 a = src[0], b = src[1];
            acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
            acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
        }
        const float mul = which == 0 ? scale : 1.f;
        uint4 u;
        u.x = pack_bf16x2(acc[0] * mul, acc[1] * mul);
        u.y = pack_bf16x2(acc[2] * mul, acc[3] * mul);
        u.z = pack_bf16x2(acc[4] * mul, acc[5] * mul);
        u.w = pack_bf16x2(acc[6] * mul, acc[7] * mul);
        *reinterpret_cast<uint4*>(d_packed + (((size_t)bh * 4 + 1 + which) * N + key) * ldq + part * 8) = u;
        return;
    }
    const long long total = rows * PPR;
    float4 a[R], b[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const long long idx = ((long long)blockIdx.x * R + r) * 256 + threadIdx.x;
        if (idx < total) {
            const float4* src = reinterpret_cast<const float4*>(dq_acc + (size_t)idx * 8);
            a[r] = src[0];
            b[r] = src[1];
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const long long idx = ((long long)blockIdx.x * R + r) * 256 + threadIdx.x;
        if (idx >= total) continue;
        const long long row = idx / PPR;
        const int part = (int)(idx % PPR);
        const long long bh = row / N, i = row % N;
        uint4 u;
        u.x = pack_bf16x2(a[r].x * scale, a[r].y * scale);
        u.y = pack_bf16x2(a[r].z * scale, a[r].w * scale);
        u.z = pack_bf16x2(b[r].x * scale, b[r].y * scale);
        u.w = pack_bf16x2(b[r].z * scale, b[r].w * scale);
        *reinterpret_cast<uint4*>(d_packed + ((size_t)bh * 4 * N + i) * ldq + part * 8) = u;
    }
}
constexpr int kFinParts = 4;  // parts per thread of dq_finalize_kernel

// ---------------------------------------------------------------- host side
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The fused kernel's units (one per batch*head and 128-key tile) all take the
// same time, so with U units on S SMs the last wave holds U mod S of them and
// leaves the other SMs idle.  Those ntail units are split into f query ranges
// (f pieces of whole 128-query groups each, ntail*f <= min(S, kMaxPieces)).
constexpr int kMaxPieces = 256;
struct TailSplit {
    int ntail = 0, f = 1;
};
TailSplit tail_split(long long units, int N, int sms) {
    TailSplit t;
    if (sms <= 0 || units <= 0) return t;
    const int cap = sms < kMaxPieces ? sms : kMaxPieces;
    const long long rem = units % sms;
    const int ngrp = (N + 127) / 128;
    if (rem == 0 || rem > cap / 2 || ngrp < 2) return t;
    t.ntail = (int)rem;
    t.f = cap / t.ntail < ngrp ? cap / t.ntail : ngrp;
    if (t.f < 2) t = TailSplit{};
    return t;
}
// Bytes of partials the split can need, whatever the SM count (kMaxPieces bounds it)
size_t tail_part_bytes(long long BH, int N, int d) {
    const long long units = BH * ((N + 127) / 128);
    const int ngrp = (N + 127) / 128;
    if (ngrp < 2) return 0;
    const long long pieces = units * ngrp < kMaxPieces ? units * ngrp : kMaxPieces;
    return (size_t)pieces * 128 * 3 * (size_t)d * 4;
}

// Launches `kern` on `st`; with `dependent`, as a programmatic dependent of
// the kernel before it on the stream, so that its blocks can be scheduled (and
// run their set-up) while that kernel finishes.  The kernel orders its reads
// of the earlier kernel's results with griddep_wait.
template <typename... P, typename... A>
cudaError_t launch_kernel(void (*kern)(P...), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                          bool dependent, A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

template <int D, bool CM>
int launch_impl(const BwdArgs& a, std::string* err) {
    using M = Cfg<D>;
    // K/V tiles: 128 rows; Q/dO sub-tiles: 64 rows (the byte counts the
    // kernel's barriers expect)
    const long long rows = a.BH * a.N;
    const int npad = (a.N + M::BS - 1) / M::BS * M::BS;
    const long long rows_pad = a.BH * npad;
    const long long ldq = a.qkv_ld(), ldo = a.o_ld();
    float4* stats = static_cast<float4*>(a.workspace);
    char* ws = static_cast<char*>(a.workspace) + align256((size_t)rows_pad * 8);
    float* dq_acc = reinterpret_cast<float*>(ws);
    const View vlo = a.do_view(0), vhi = a.do_view(1);
    const long long nb = a.BH / a.heads;
    // dq_acc in 128-query boxes of BOXC columns (the drain's bulk reduces)
    CUtensorMap tm_kv, tm_q, tm_lo, tm_hi, tm_dq;
    if (!encode_bf16_rows_ld(&tm_kv, a.packed, D, ldq, a.N, a.BH * 4, M::BM, D, err) ||
        !encode_bf16_rows_ld(&tm_q, a.packed, D, ldq, a.N, a.BH * 4, M::BS, D, err) ||
        !(CM ? encode_bf16_4d(&tm_lo, vlo.base, a.N, D, a.heads, nb, vlo.sJ, vlo.sH, vlo.sB, M::BS, D, err)
             : encode_bf16_4d(&tm_lo, vlo.base, D, a.N, a.heads, nb, vlo.sN, vlo.sH, vlo.sB, D, M::BS, err)) ||
        !(CM ? encode_bf16_4d(&tm_hi, vhi.base, a.N, D, a.heads, nb, vhi.sJ, vhi.sH, vhi.sB, M::BS, D, err)
             : encode_bf16_4d(&tm_hi, vhi.base, D, a.N, a.heads, nb, vhi.sN, vhi.sH, vhi.sB, D, M::BS, err)) ||
        !encode_f32_rows(&tm_dq, dq_acc, D, a.N, a.BH, 128, M::BOXC, err))
        return PSA_ERR_CUDA;
    if (!set_max_dynamic_smem((const void*)bwd_main_kernel<D, CM>, M::SMEM, err)) return PSA_ERR_CUDA;
    if constexpr (!M::SLACK) {
        const int al = dyn_smem_base_aligned(err);
        if (al < 0) return PSA_ERR_CUDA;
        if (al == 0) {
            *err = "the fused kernel at this head_dim needs a 1024-byte aligned dynamic shared memory base";
            return PSA_ERR_UNSUPPORTED;
        }
    }
    float* dkv_part = reinterpret_cast<float*>(ws + align256((size_t)rows * D * 4));
    const int nkt = (a.N + M::BM - 1) / M::BM;
    const long long units = a.BH * nkt;
    // split the last wave's units along the query axis so that it fills the SMs
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 0;
    const TailSplit ts = tail_split(units, a.N, sms);
    const long long nfull = units - ts.ntail;
    const long long nitems = nfull + (long long)ts.ntail * ts.f;
    // persistent: one CTA per SM (shared memory and TMEM hold one), each
    // walking items b, b + grid, ...
    const long long grid = sms > 0 && nitems > sms ? sms : nitems;
    const bool plain = !a.views && ldo == D;   // contiguous O and dO: the vectorised statistics kernel
    const long long pre_grid = plain ? (rows_pad + 256 / (D / 8) - 1) / (256 / (D / 8)) : (rows_pad + 255) / 256;
    const long long fin_main = (rows * (D / 8) + 256 * kFinParts - 1) / (256 * kFinParts);
    const long long fin_grid = fin_main + ((long long)ts.ntail * 128 * 3 * (D / 8) + 255) / 256;
    if (nitems > 0x7fffffffll || pre_grid > 0x7fffffffll || fin_grid > 0x7fffffffll) {
        *err = "grid too large";
        return PSA_ERR_UNSUPPORTED;
    }
    const bf16* o_lo = static_cast<const bf16*>(a.o_lo);
    const bf16* o_hi = static_cast<const bf16*>(a.o_hi);
    bf16* dp = static_cast<bf16*>(a.d_packed);
    {
        ProfScope prof(kSlotPre, a.stream);
        if (plain)
            pre_stats_kernel<D><<<(unsigned)pre_grid, 256, 0, a.stream>>>(
                o_lo, o_hi, static_cast<const bf16*>(vlo.base), static_cast<const bf16*>(vhi.base), a.lse, stats,
                dq_acc, rows_pad, a.N, npad);
        else
            pre_stats_view_kernel<D><<<(unsigned)pre_grid, 256, 0, a.stream>>>(o_lo, o_hi, ldo, vlo, vhi, a.heads,
                                                                               a.lse, stats, dq_acc, rows_pad, a.N,
                                                                               npad);
    }
    // The fused kernel and the finalize kernel start as programmatic dependents
    // of the kernel before them, except while kernels are timed one by one
    // (events between them would stand in the way).
    const bool dependent = !prof_enabled();
    cudaError_t e = cudaSuccess;
    {
        ProfScope prof(kSlotMain, a.stream);
        e = launch_kernel(bwd_main_kernel<D, CM>, (unsigned)grid, M::THREADS, M::SMEM, a.stream, dependent, tm_kv,
                          tm_q, tm_lo, tm_hi, tm_dq, a.heads, ldq, (const float4*)stats, dp, a.N, nkt, a.scale,
                          a.scale * kLog2e, (int)nfull, ts.f, (int)nitems, dkv_part);
    }
    if (e == cudaSuccess) {
        ProfScope prof(kSlotDq, a.stream);
        e = launch_kernel(dq_finalize_kernel<D, kFinParts>, (unsigned)fin_grid, 256, 0, a.stream, dependent,
                          (const float*)dq_acc, dp, ldq, rows, a.N, a.scale, (const float*)dkv_part, (int)nfull,
                          ts.ntail, ts.f, nkt, (int)fin_main);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = std::string("tensor-core backward launch: ") + cudaGetErrorString(e);
        return PSA_ERR_CUDA;
    }
    return PSA_OK;
}

// dO read as rows, or as channel-major [d, N] blocks (position stride 1).
template <int D>
int launch(const BwdArgs& a, std::string* err) {
    const View v = a.do_view(0);
    return (v.sN == 1 && v.sJ != 1) ? launch_impl<D, true>(a, err) : launch_impl<D, false>(a, err);
}

template <int D>
int launch_two_pass(const BwdArgs& a, std::string* err) {
    using M = CfgS<D>;
    CUtensorMap tm_kv, tm_q, tm_lo, tm_hi;
    if (!encode_bf16_rows(&tm_kv, a.packed, D, a.N, a.BH * 4, M::BM, D, err) ||
        !encode_bf16_rows(&tm_q, a.packed, D, a.N, a.BH * 4, M::BS, D, err) ||
        !encode_bf16_rows(&tm_lo, a.do_lo, D, a.N, a.BH, M::BS, D, err) ||
        !encode_bf16_rows(&tm_hi, a.do_hi, D, a.N, a.BH, M::BS, D, err))
        return PSA_ERR_CUDA;
    if (!set_max_dynamic_smem((const void*)bwd_dkdv_kernel<D>, M::SMEM, err)) return PSA_ERR_CUDA;
    const long long rows = a.BH * a.N;
    float* Drow = static_cast<float*>(a.workspace);
    const int nkt = (a.N + M::BM - 1) / M::BM;
    const long long grid = a.BH * nkt;
    const long long pre_grid = (rows + 256 / (D / 8) - 1) / (256 / (D / 8));
    if (grid > 0x7fffffffll || pre_grid > 0x7fffffffll) {
        *err = "grid too large";
        return PSA_ERR_UNSUPPORTED;
    }
    bf16* dp = static_cast<bf16*>(a.d_packed);
    {
        ProfScope prof(kSlotPre, a.stream);
        pre_kernel<D><<<(unsigned)pre_grid, 256, 0, a.stream>>>(
            static_cast<const bf16*>(a.o_lo), static_cast<const bf16*>(a.o_hi), static_cast<const bf16*>(a.do_lo),
            static_cast<const bf16*>(a.do_hi), Drow, nullptr, rows);
    }
    {
        ProfScope prof(kSlotMain, a.stream);
        bwd_dkdv_kernel<D><<<(unsigned)grid, kThreadsS, M::SMEM, a.stream>>>(
            tm_kv, tm_q, tm_lo, tm_hi, a.lse, Drow, dp, a.N, nkt, a.scale, a.scale * kLog2e);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = std::string("tensor-core dK/dV launch: ") + cudaGetErrorString(e);
        return PSA_ERR_CUDA;
    }
    return tc_dq_launch(a, Drow, err);
}

}  // namespace

bool tc_supported(int dtype, int d) { return dtype == PSA_BF16 && (d == 16 || d == 32 || d == 64); }

double tc_bwd_waves(long long units, int N, int sms) {
    if (units <= 0) return 0.0;
    if (sms <= 0) return (double)units;
    const TailSplit t = tail_split(units, N, sms);
    if (t.ntail == 0) return (double)((units + sms - 1) / sms);
    const int ngrp = (N + 127) / 128;
    return (double)((units - t.ntail) / sms) + (double)((ngrp + t.f - 1) / t.f) / ngrp;
}

size_t tc_workspace_bytes(long long BH, int N, int d) {
    // statistics (8 bytes per query, padded to whole 64-query sub-tiles), the
    // fp32 dQ accumulator, the dK/dV partials of split units
    const size_t rows = (size_t)BH * (size_t)N;
    const size_t rows_pad = (size_t)BH * (size_t)((N + 63) / 64 * 64);
    return align256(rows_pad * 8) + align256(rows * (size_t)d * 4) + tail_part_bytes(BH, N, d);
}

size_t tc_two_pass_workspace_bytes(long long BH, int N) { return align256((size_t)BH * (size_t)N * 4); }

int tc_pre_d_launch(const BwdArgs& a, float* Drow, std::string* err) {
    const long long rows = a.BH * a.N;
    const int rpb = 256 / (a.d / 8);
    const long long grid = (rows + rpb - 1) / rpb;
    if (grid > 0x7fffffffll) {
        *err = "grid too large";
        return PSA_ERR_UNSUPPORTED;
    }
    const bf16* o_lo = static_cast<const bf16*>(a.o_lo);
    const bf16* o_hi = static_cast<const bf16*>(a.o_hi);
    const bf16* do_lo = static_cast<const bf16*>(a.do_lo);
    const bf16* do_hi = static_cast<const bf16*>(a.do_hi);
    {
        ProfScope prof(kSlotPre, a.stream);
        switch (a.d) {
            case 16: pre_kernel<16><<<(unsigned)grid, 256, 0, a.stream>>>(o_lo, o_hi, do_lo, do_hi, Drow, nullptr, rows); break;
            case 32: pre_kernel<32><<<(unsigned)grid, 256, 0, a.stream>>>(o_lo, o_hi, do_lo, do_hi, Drow, nullptr, rows); break;
            case 64: pre_kernel<64><<<(unsigned)grid, 256, 0, a.stream>>>(o_lo, o_hi, do_lo, do_hi, Drow, nullptr, rows); break;
            default: *err = "unsupported head_dim"; return PSA_ERR_UNSUPPORTED;
        }
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = std::string("row-statistics launch: ") + cudaGetErrorString(e);
        return PSA_ERR_CUDA;
    }
    return PSA_OK;
}

int tc_two_pass_launch(const BwdArgs& a, std::string* err) {
    switch (a.d) {
        case 16: return launch_two_pass<16>(a, err);
        case 32: return launch_two_pass<32>(a, err);
        case 64: return launch_two_pass<64>(a, err);
        default: *err = "unsupported head_dim"; return PSA_ERR_UNSUPPORTED;
    }
}

int tc_bwd_launch(const BwdArgs& a, std::string* err) {
    switch (a.d) {
        case 16: return launch<16>(a, err);
        case 32: return launch<32>(a, err);
        case 64: return launch<64>(a, err);
        default: *err = "unsupported head_dim"; return PSA_ERR_UNSUPPORTED;
    }
}

int tc_wait_selftest(cudaStream_t stream, std::string* err) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(20000000ull);  // 20 ms
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *err = std::string("self-test launch: ") + cudaGetErrorString(e);
        return PSA_ERR_CUDA;
    }
    return PSA_OK;
}

int tc_take_device_error(std::string* err) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(int));
    if (e != cudaSuccess || v == 0) return 0;
    const int zero = 0;
    cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(int));
    static const char* roles[] = {"?", "producer", "mma", "softmax", "dq", "self-test", "dq-mma"};
    const int role = (v >> 24) & 0xff;
    *err = std::string("tensor-core backward: a bounded wait gave up (") + roles[role < 7 ? role : 0] +
           " warp, query tile " + std::to_string(v & 0xFFFFFF) + ")";
    return 1;
}

}  // namespace psa
