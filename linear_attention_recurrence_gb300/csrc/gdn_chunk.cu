// Chunked (32-token WY) Gated DeltaNet recurrence for sm_103a.
//
// The math ("#1372 DeltaNet recurrence: STRATA_GDN_CHUNKED=1 - the prompt's
// recurrence in 32-token chunks", section "What it does"), per value head, with
// gamma_t the running sum of the gate inside the chunk and S0 the state before it:
//     A[t][i] = beta_t e^(gamma_t - gamma_i) k_t.k_i   (i < t)
//     T = (I + A)^-1,  T' = T diag(beta)
//     U' = V - diag(e^gamma) K S0,  D = T' U'
//     O = diag(e^gamma) Q S0 + P D,   P[t][i] = e^(gamma_t - gamma_i) q_t.k_i  (i <= t)
//     S_end = e^gamma_last S0 + K^T diag(e^(gamma_last - gamma)) D
// All exponents are <= 0.  A last chunk with r < 32 tokens is padded with zero
// k, q, v, g and beta, which leaves every product above unchanged.
//
// Two kernels per 2048-token super-block, as on the page:
//  * prep: one CTA per (chunk, key head) forms K K^T and Q K^T once for the key
//    head's three value heads, the gates' running sums, A and P, and solves for T
//    (one lane per column of T).  It writes a record per (chunk, value head):
//    T'^T, P^T, e^gamma and e^(gamma_last - gamma).
//  * scan: one CTA per (key head, 16 value columns) walks the super-block's
//    chunks with its slice of the three heads' state in registers (and a
//    transposed copy in shared memory for the K S0 / Q S0 product).  Each chunk's
//    k and q tiles (TMA, 128-byte swizzle), v columns (TMA) and prep records
//    (bulk copies) land in a double buffer while the chunk before computes.
// When the SMs the scan leaves free number at least n_kh, one cooperative launch
// runs both: the prep on those SMs, chunk by chunk ahead of the scan, which waits
// on a per-(chunk, key head) flag instead of a kernel boundary (gdn_chunk_fused_kernel).
// By default every product (K K^T and Q K^T in the prep; K S0, Q S0, T'U', P D and
// K^T D' in the scan) runs on the tensor cores as warp-level m16n8k8 TF32 MMAs on
// split operands (three MMAs per FP32 product, see "products on the tensor cores"
// below): plain TF32 inputs would miss the 2e-6 tolerance (relative to FP64) the
// path is held to by three orders of magnitude.  The scan's products as
// register-tiled packed FP32x2 FMAs remain selectable (the FMA form).
#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_norm_row.cuh"
#include "gdn_chunk_prep.cuh"

namespace gdn {
namespace {


// One CTA per (chunk, key head).
__global__ void __launch_bounds__(PREP_THREADS) gdn_chunk_prep_kernel(const ChunkPrepParams p) {
    PrepSmemT<1>& sm = *aligned_dynamic_smem<PrepSmemT<1>, 16>();
    prep_load(p, sm, 0, blockIdx.x, blockIdx.y);
    cp_async_wait<0>();
    __syncthreads();
    prep_task(p, sm, 0, blockIdx.x, blockIdx.y);
}

// ============================ scan ============================
constexpr int SCAN_THREADS = 256;
constexpr int NC = 16;        // value columns per CTA (per head)
constexpr int NCC = kHeadsPerKey * NC;  // 48 columns of the CTA
constexpr int SST = D + 4;    // row stride of the transposed state copy

struct __align__(1024) ScanBuf {
    float K[D / 32][C][32];        // 4 TMA boxes of [32 rows][32 floats], 128-byte swizzled
    float Q[D / 32][C][32];
    float V[kHeadsPerKey][C][NC];  // TMA boxes [32 rows][16 floats]
    float rec[kHeadsPerKey][REC];  // prep records (bulk copies)
};
constexpr uint32_t kScanTxBytes = 2 * C * D * 4 + kHeadsPerKey * C * NC * 4 + kHeadsPerKey * REC * 4;

constexpr int WST = NCC + 8;  // row stride of W and Dp: 16-byte aligned rows on which the
                              // MMA form's fragment accesses hit 32 distinct banks

struct ScanSmem {
    ScanBuf buf[2];
    float SsT[NCC][SST];        // S0 transposed: [head*16 + col][key dim]
    float W[2 * C][WST];        // rows 0..31: U'; rows 32..63: e^gamma (Q S0)
    float Dm[C][WST];           // D
    float Dp[C][WST];           // e^(gamma_last - gamma) D
    uint64_t full[2];
    int copy_gave_up;           // 1 + the chunk whose copy wait ran out, else 0
    int flag_gave_up;           // a prep flag wait ran out (later ones are skipped)
};
static_assert(sizeof(ScanSmem) + 1024 <= 227 * 1024, "scan shared memory");
static_assert(kHeadsPerKey * C * C % 256 == 0, "prep A / P loop");
// g1_mma's exchange of partial sums: 8 warps x 12 floats x 32 lanes in Dm, Dp
static_assert(offsetof(ScanSmem, Dp) == offsetof(ScanSmem, Dm) + sizeof(float) * C * WST &&
                  2 * C * WST >= 8 * 12 * 32,
              "g1_mma exchange space");

// byte offset of float4 chunk `cc` (0..7) of row `r` in a 128-byte-swizzled box
__device__ __forceinline__ int swz(int r, int cc) { return r * 128 + ((cc ^ (r & 7)) << 4); }

__device__ __forceinline__ float ldsf(const unsigned char* p) { return *reinterpret_cast<const float*>(p); }

// The CTA's 128 x 48 slice of the state (key dims x the 16 columns of each of the
// three heads), 24 floats per thread, in the layout each form of the update uses:
//  * FMA: thread (it = tid / 16, jj = tid % 16) holds key dims 8 it .. 8 it + 7 of
//    column jj of each head, as pairs of consecutive key dims;
//  * MMA: warp w holds 16 key dims (mma_key) of all 48 columns as six m16n8
//    accumulator tiles (rows = key dims, columns = the CTA's columns 8n .. 8n + 7);
//    the update reloads them from SsT, so between updates they are dead.
template <bool kMma>
struct ScanState;
template <>
struct ScanState<false> {
    float2 v[kHeadsPerKey][4];
};
template <>
struct ScanState<true> {
    float v[NCC / 8][4];
};

// Key dim of accumulator row `row` (0..15) in warp w's update tile.  Warps 2b and
// 2b + 1 share the 32 key dims of k-tile box b, each taking four of its 16-byte
// chunks, {0, 1, 4, 5} or {2, 3, 6, 7}: rows g and g + 8 of a fragment then fall in
// chunks four apart, so a warp's loads of K^T from the swizzled box hit 32 banks.
__device__ __forceinline__ int mma_key(const int w, const int row) {
    return 32 * (w >> 1) + 4 * (2 * (w & 1) + 4 * ((row >> 2) & 1) + (row >> 3)) + (row & 3);
}

// state slice -> registers and the transposed copy SsT
__device__ __forceinline__ void state_load(const ChunkScanParams& p, ScanSmem& sm, ScanState<false>& S, const int kh,
                                           const int c0) {
    const int tid = threadIdx.x, it = tid >> 4, jj = tid & 15;
#pragma unroll
    for (int m = 0; m < kHeadsPerKey; ++m) {
        const float* sh = p.state + (static_cast<int64_t>(kh + m * p.n_kh) * D + 8 * it) * D + c0 + jj;
#pragma unroll
        for (int q = 0; q < 4; ++q) S.v[m][q] = make_float2(sh[(2 * q) * D], sh[(2 * q + 1) * D]);
#pragma unroll
        for (int h4 = 0; h4 < 2; ++h4)
            *reinterpret_cast<float4*>(&sm.SsT[m * NC + jj][8 * it + 4 * h4]) =
                make_float4(S.v[m][2 * h4].x, S.v[m][2 * h4].y, S.v[m][2 * h4 + 1].x, S.v[m][2 * h4 + 1].y);
    }
}
__device__ __forceinline__ void state_load(const ChunkScanParams& p, ScanSmem& sm, ScanState<true>& S, const int kh,
                                           const int c0) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int key = mma_key(threadIdx.x >> 5, g);  // rows g; rows g + 8 are key + 4
#pragma unroll
    for (int n = 0; n < NCC / 8; ++n) {
        const int col = 8 * n + 2 * t;  // the CTA's column: head col / 16, column c0 + col % 16
        const float* sh = p.state + (static_cast<int64_t>(kh + (n >> 1) * p.n_kh) * D + key) * D + c0 + (col & 15);
        const float2 lo = *reinterpret_cast<const float2*>(sh);
        const float2 hi = *reinterpret_cast<const float2*>(sh + 4 * D);
        S.v[n][0] = lo.x;
        S.v[n][1] = lo.y;
        S.v[n][2] = hi.x;
        S.v[n][3] = hi.y;
        sm.SsT[col][key] = lo.x;
        sm.SsT[col + 1][key] = lo.y;
        sm.SsT[col][key + 4] = hi.x;
        sm.SsT[col + 1][key + 4] = hi.y;
    }
}

__device__ __forceinline__ void state_store(const ChunkScanParams& p, const ScanState<false>& S, const int kh,
                                            const int c0) {
    const int tid = threadIdx.x, it = tid >> 4, jj = tid & 15;
#pragma unroll
    for (int m = 0; m < kHeadsPerKey; ++m) {
        float* sh = p.state + (static_cast<int64_t>(kh + m * p.n_kh) * D + 8 * it) * D + c0 + jj;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            sh[(2 * q) * D] = S.v[m][q].x;
            sh[(2 * q + 1) * D] = S.v[m][q].y;
        }
    }
}
__device__ __forceinline__ void state_store(const ChunkScanParams& p, const ScanState<true>& S, const int kh,
                                            const int c0) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int key = mma_key(threadIdx.x >> 5, g);
#pragma unroll
    for (int n = 0; n < NCC / 8; ++n) {
        const int col = 8 * n + 2 * t;
        float* sh = p.state + (static_cast<int64_t>(kh + (n >> 1) * p.n_kh) * D + key) * D + c0 + (col & 15);
        *reinterpret_cast<float2*>(sh) = make_float2(S.v[n][0], S.v[n][1]);
        *reinterpret_cast<float2*>(sh + 4 * D) = make_float2(S.v[n][2], S.v[n][3]);
    }
}

// ---- G1: W = [K; Q] S0 (64 x 48), then U' = V - e^gamma K S0 and e^gamma Q S0 into W ----

// FMA form: packed over even/odd key dims, the key dims split over the two
// half-warps and their partial sums added once.  Warp tg takes X rows
// 8*(tg&3)..+7 of K (tg < 4) or Q (tg >= 4); lane bit 4 picks the key-dim half
// kgrp (dims 0..63 or 64..127) and the low four bits the column jw of each head.
// Each quarter-warp shares its rows and half, so the X loads are broadcasts; the
// halves' partial sums meet by a shuffle.
__device__ __forceinline__ void g1_fma(const ScanBuf& b, ScanSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tg = warp, kgrp = (lane >> 4) & 1, jw = lane & 15;
    const unsigned char* xb = reinterpret_cast<const unsigned char*>(tg < 4 ? &b.K[0][0][0] : &b.Q[0][0][0]) +
                              (8 * (tg & 3)) * 128;
    float2 acc[8][kHeadsPerKey];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m) acc[r][m] = make_float2(0.f, 0.f);
#pragma unroll
    for (int bh = 0; bh < 2; ++bh) {
        const int bx = 2 * kgrp + bh;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            float4 s4[kHeadsPerKey];
#pragma unroll
            for (int m = 0; m < kHeadsPerKey; ++m)
                s4[m] = *reinterpret_cast<const float4*>(&sm.SsT[m * NC + jw][32 * bx + 4 * cc]);
#pragma unroll
            for (int r = 0; r < 8; ++r) {  // row 8*(tg&3) + r has (row & 7) == r
                const float4 a = *reinterpret_cast<const float4*>(xb + bx * (C * 128) + r * 128 + ((cc ^ r) << 4));
#pragma unroll
                for (int m = 0; m < kHeadsPerKey; ++m) {
                    acc[r][m] = ffma2(make_float2(a.x, a.y), make_float2(s4[m].x, s4[m].y), acc[r][m]);
                    acc[r][m] = ffma2(make_float2(a.z, a.w), make_float2(s4[m].z, s4[m].w), acc[r][m]);
                }
            }
        }
    }
    // reduce-scatter with lane ^ 16: kgrp 0 finishes the even rows, kgrp 1 the odd
    // ones, each as (dims 0..63) + (dims 64..127)
#pragma unroll
    for (int r2 = 0; r2 < 4; ++r2) {
        const int t = 8 * (tg & 3) + 2 * r2 + kgrp;
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m) {
            const float ev = acc[2 * r2][m].x + acc[2 * r2][m].y;
            const float od = acc[2 * r2 + 1][m].x + acc[2 * r2 + 1][m].y;
            const float other = __shfl_xor_sync(0xffffffffu, kgrp ? ev : od, 16);
            const float x = kgrp ? other + od : ev + other;
            const float eg = b.rec[m][REC_EG + t];
            if (tg < 4)
                sm.W[t][m * NC + jw] = b.V[m][t][jw] - eg * x;
            else
                sm.W[C + t][m * NC + jw] = eg * x;
        }
    }
}

// MMA form: warp w sums key dims 64 (w >> 2) .. +63 (8 k8 steps) for the 32 rows of
// K (w & 1 == 0) or Q times the CTA's columns 24 ((w >> 1) & 1) .. +23: two m16
// tiles x three n8 tiles, so each split fragment feeds two or three MMAs (0.78
// splits per MMA instead of 1.11 with one m16 tile over all key dims; the splits'
// integer work bounds the issue rate).  A from the swizzled k / q box (row & 7 ==
// g: the fragment loads hit 32 banks), B from SsT (row stride 132: 32 banks); each
// step's operands load while the step before issues its MMAs.  The two key-dim
// halves meet through shared memory (the Dm / Dp space, free until P2): warp w
// finishes row tile w >> 2 and hands the other to warp w ^ 4, so the result is the
// same sum in the same order for every element.
__device__ __forceinline__ void g1_mma(const ScanBuf& b, ScanSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int h = warp >> 2, xq = warp & 1, ng = (warp >> 1) & 1;  // key-dim half, K or Q, column group
    const unsigned char* xa = reinterpret_cast<const unsigned char*>(xq ? &b.Q[0][0][0] : &b.K[0][0][0]) +
                              g * 128 + 4 * t;
    const float* sb = &sm.SsT[24 * ng + g][t];
    auto load = [&](const int j, float (&av)[8], float (&bv)[6]) {
        const unsigned char* xr = xa + (j >> 2) * (C * 128);
        const int ca = ((2 * (j & 3)) ^ g) << 4, cb = ((2 * (j & 3) + 1) ^ g) << 4;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            av[4 * r + 0] = ldsf(xr + 2048 * r + ca);
            av[4 * r + 1] = ldsf(xr + 2048 * r + 1024 + ca);
            av[4 * r + 2] = ldsf(xr + 2048 * r + cb);
            av[4 * r + 3] = ldsf(xr + 2048 * r + 1024 + cb);
        }
#pragma unroll
        for (int n = 0; n < 3; ++n) {
            bv[2 * n] = sb[8 * n * SST + 8 * j];
            bv[2 * n + 1] = sb[8 * n * SST + 8 * j + 4];
        }
    };
    float acc[2][3][4], accx[2][3][4];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int n = 0; n < 3; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[r][n][i] = accx[r][n][i] = 0.f;
    float av[2][8], bv[2][6];
    load(8 * h, av[0], bv[0]);
#pragma unroll
    for (int jj = 0; jj < D / 16; ++jj) {
        const int j = 8 * h + jj, cur = jj & 1;
        if (jj + 1 < D / 16) load(j + 1, av[cur ^ 1], bv[cur ^ 1]);
        uint32_t ah[2][4], al[2][4], bh[3][2], bl[3][2];
#pragma unroll
        for (int i = 0; i < 8; ++i) split_tf32(av[cur][i], ah[i >> 2][i & 3], al[i >> 2][i & 3]);
#pragma unroll
        for (int i = 0; i < 6; ++i) split_tf32(bv[cur][i], bh[i >> 1][i & 1], bl[i >> 1][i & 1]);
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int n = 0; n < 3; ++n) mma_tf32(acc[r][n], ah[r], bh[n]);
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int n = 0; n < 3; ++n) mma_tf32(accx[r][n], ah[r], bl[n]);
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int n = 0; n < 3; ++n) mma_tf32(accx[r][n], al[r], bh[n]);
    }
    // the partner's row tile (1 - h) out, then this warp's row tile h in (half 0 + half 1)
    float* xchg = &sm.Dm[0][0];
#pragma unroll
    for (int n = 0; n < 3; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            xchg[(warp * 12 + 4 * n + i) * 32 + lane] = h ? acc[0][n][i] + accx[0][n][i] : acc[1][n][i] + accx[1][n][i];
    __syncthreads();
    // every load of the epilogue first, then the stores (the compiler cannot tell
    // the stores into W from the loads of xchg, V and the records apart)
    float xo[3][4], eg[3][2];
    float2 vv[3][2];
#pragma unroll
    for (int n = 0; n < 3; ++n) {
        const int col = 24 * ng + 8 * n + 2 * t, m = col >> 4, jc = col & 15;
#pragma unroll
        for (int i = 0; i < 4; ++i) xo[n][i] = xchg[((warp ^ 4) * 12 + 4 * n + i) * 32 + lane];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int tk = 16 * h + g + 8 * hf;
            eg[n][hf] = b.rec[m][REC_EG + tk];
            vv[n][hf] = xq ? make_float2(0.f, 0.f) : *reinterpret_cast<const float2*>(&b.V[m][tk][jc]);
        }
    }
#pragma unroll
    for (int n = 0; n < 3; ++n) {
        const int col = 24 * ng + 8 * n + 2 * t;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int tk = 16 * h + g + 8 * hf;
            float x[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int i = 2 * hf + e;
                const float own = h ? acc[1][n][i] + accx[1][n][i] : acc[0][n][i] + accx[0][n][i];
                x[e] = own + xo[n][i];
            }
            if (!xq) {
                *reinterpret_cast<float2*>(&sm.W[tk][col]) =
                    make_float2(vv[n][hf].x - eg[n][hf] * x[0], vv[n][hf].y - eg[n][hf] * x[1]);
            } else {
                *reinterpret_cast<float2*>(&sm.W[C + tk][col]) = make_float2(eg[n][hf] * x[0], eg[n][hf] * x[1]);
            }
        }
    }
}

// ---- P2 / P3 on the tensor cores: the chunk's two small products per head, in
// transposed form (rows = the head's 16 columns, columns = tokens), so that the
// A operands (U', D) come from W / Dm with 32-bank fragment loads:
//     D^T = U'^T T'^T,   O^T = (e^gamma Q S0)^T + D^T P^T.
// T' and P are lower triangular (the records hold their zeros), so token tile nn
// needs only the k steps kk <= nn: 10 of 16.  Warp w < 6 takes head w / 2 and the
// token tiles {w % 2, 3 - w % 2}: five k steps per warp.
__device__ __forceinline__ void load_a_cols(const float (*x)[WST], const int kk, const int col0, const int g,
                                            const int t, uint32_t (&ah)[4], uint32_t (&al)[4]) {
    split_tf32(x[8 * kk + t][col0 + g], ah[0], al[0]);
    split_tf32(x[8 * kk + t][col0 + g + 8], ah[1], al[1]);
    split_tf32(x[8 * kk + t + 4][col0 + g], ah[2], al[2]);
    split_tf32(x[8 * kk + t + 4][col0 + g + 8], ah[3], al[3]);
}
__device__ __forceinline__ void load_b_rec(const float* r, const int kk, const int nn, const int g, const int t,
                                           uint32_t (&bh)[2], uint32_t (&bl)[2]) {
    split_tf32(r[(8 * kk + t) * C + 8 * nn + g], bh[0], bl[0]);
    split_tf32(r[(8 * kk + t + 4) * C + 8 * nn + g], bh[1], bl[1]);
}

// D^T tiles of head w / 2 -> Dm (D) and Dp (e^(gamma_last - gamma) D), [token][column]
__device__ __forceinline__ void p2_mma(const ScanBuf& b, ScanSmem& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int m = warp >> 1, na = warp & 1, nb = 3 - na;
    const float* tp = &b.rec[m][REC_TP];
    float acc[2][4], accx[2][4], accy[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][e] = accx[i][e] = accy[i][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < C / 8; ++kk) {
        if (kk > nb) break;
        uint32_t ah[4], al[4], bh[2][2], bl[2][2];
        load_a_cols(sm.W, kk, m * NC, g, t, ah, al);
        const bool both = kk <= na;  // tile nb (> na) takes every k step up to nb
        load_b_rec(tp, kk, nb, g, t, bh[1], bl[1]);
        if (both) load_b_rec(tp, kk, na, g, t, bh[0], bl[0]);
        mma_tf32(acc[1], ah, bh[1]);
        if (both) mma_tf32(acc[0], ah, bh[0]);
        mma_tf32(accx[1], ah, bl[1]);
        if (both) mma_tf32(accx[0], ah, bl[0]);
        mma_tf32(accy[1], al, bh[1]);
        if (both) mma_tf32(accy[0], al, bh[0]);
    }
    // the records' e^(gamma_last - gamma) first, then the stores
    float er[2][2];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int e = 0; e < 2; ++e) er[i][e] = b.rec[m][REC_ER + 8 * (i ? nb : na) + 2 * t + e];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int nn = i ? nb : na;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int col = m * NC + g + 8 * (e >> 1), tok = 8 * nn + 2 * t + (e & 1);
            const float d = acc[i][e] + (accx[i][e] + accy[i][e]);
            sm.Dm[tok][col] = d;
            sm.Dp[tok][col] = er[i][e & 1] * d;
        }
    }
}

// O^T tiles of head w / 2 -> out (tokens < nt)
__device__ __forceinline__ void p3_mma(const ChunkScanParams& p, const ScanBuf& b, const ScanSmem& sm, const int kh,
                                       const int c0, const int c, const int nt) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int m = warp >> 1, na = warp & 1, nb = 3 - na;
    const float* pt = &b.rec[m][REC_PT];
    float acc[2][4], accx[2][4], accy[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int nn = i ? nb : na;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc[i][e] = sm.W[C + 8 * nn + 2 * t + (e & 1)][m * NC + g + 8 * (e >> 1)];
            accx[i][e] = accy[i][e] = 0.f;
        }
    }
#pragma unroll
    for (int kk = 0; kk < C / 8; ++kk) {
        if (kk > nb) break;
        uint32_t ah[4], al[4], bh[2][2], bl[2][2];
        load_a_cols(sm.Dm, kk, m * NC, g, t, ah, al);
        const bool both = kk <= na;  // tile nb (> na) takes every k step up to nb
        load_b_rec(pt, kk, nb, g, t, bh[1], bl[1]);
        if (both) load_b_rec(pt, kk, na, g, t, bh[0], bl[0]);
        mma_tf32(acc[1], ah, bh[1]);
        if (both) mma_tf32(acc[0], ah, bh[0]);
        mma_tf32(accx[1], ah, bl[1]);
        if (both) mma_tf32(accx[0], ah, bl[0]);
        mma_tf32(accy[1], al, bh[1]);
        if (both) mma_tf32(accy[0], al, bh[0]);
    }
    const int h = kh + m * p.n_kh;
    float* o = p.out + ((p.t_begin + static_cast<int64_t>(c) * C) * p.n_vh + h) * D + c0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int nn = i ? nb : na;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int tok = 8 * nn + 2 * t + (e & 1);
            if (tok < nt) o[static_cast<int64_t>(tok) * p.n_vh * D + g + 8 * (e >> 1)] = acc[i][e] + (accx[i][e] + accy[i][e]);
        }
    }
}

// ---- G4: S_end = e^gamma_last S0 + K^T (e^(gamma_last-gamma) D), and its transposed copy ----

// FMA form: packed over key-dim pairs, 8 key dims x 3 columns per thread.
__device__ __forceinline__ void g4_fma(const ScanBuf& b, ScanSmem& sm, ScanState<false>& S) {
    const int tid = threadIdx.x, it = tid >> 4, jj = tid & 15;
    const unsigned char* kb = reinterpret_cast<const unsigned char*>(&b.K[it >> 2][0][0]);
    const int cc0 = 2 * (it & 3);
    float2 acc[kHeadsPerKey][4];
#pragma unroll
    for (int m = 0; m < kHeadsPerKey; ++m) {
        const float el = b.rec[m][REC_EG + C - 1];
        const float2 el2 = make_float2(el, el);
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[m][q] = fmul2(el2, S.v[m][q]);
    }
#pragma unroll 8
    for (int t = 0; t < C; ++t) {
        const float4 klo = *reinterpret_cast<const float4*>(kb + swz(t, cc0));
        const float4 khi = *reinterpret_cast<const float4*>(kb + swz(t, cc0 + 1));
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m) {
            const float dv = sm.Dp[t][m * NC + jj];
            const float2 d2 = make_float2(dv, dv);
            acc[m][0] = ffma2(make_float2(klo.x, klo.y), d2, acc[m][0]);
            acc[m][1] = ffma2(make_float2(klo.z, klo.w), d2, acc[m][1]);
            acc[m][2] = ffma2(make_float2(khi.x, khi.y), d2, acc[m][2]);
            acc[m][3] = ffma2(make_float2(khi.z, khi.w), d2, acc[m][3]);
        }
    }
#pragma unroll
    for (int m = 0; m < kHeadsPerKey; ++m) {
#pragma unroll
        for (int q = 0; q < 4; ++q) S.v[m][q] = acc[m][q];
#pragma unroll
        for (int h4 = 0; h4 < 2; ++h4)
            *reinterpret_cast<float4*>(&sm.SsT[m * NC + jj][8 * it + 4 * h4]) =
                make_float4(acc[m][2 * h4].x, acc[m][2 * h4].y, acc[m][2 * h4 + 1].x, acc[m][2 * h4 + 1].y);
    }
}

// MMA form: warp w updates its 16 key dims (mma_key) of all 48 columns, K^T from
// the swizzled k box (A: key dims x tokens), D' from Dp (B: tokens x columns, row
// stride 56: 32 banks), the state itself the accumulator; each step's operands
// are loaded while the step before issues its MMAs.
__device__ __forceinline__ void g4_mma(const ScanBuf& b, ScanSmem& sm, ScanState<true>& S) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int ch = 2 * (warp & 1) + 4 * (g >> 2);  // 16-byte chunk of key row g; row g + 8: ch + 1
    const unsigned char* ka = reinterpret_cast<const unsigned char*>(&b.K[warp >> 1][0][0]) + 4 * (g & 3);
    auto load = [&](const int j, float (&av)[4], float (&bv)[2 * NCC / 8]) {
        const unsigned char* r0 = ka + (8 * j + t) * 128;  // token 8j + t: row & 7 == t
        const unsigned char* r1 = r0 + 4 * 128;            // token 8j + t + 4: row & 7 == t + 4
        av[0] = ldsf(r0 + ((ch ^ t) << 4));
        av[1] = ldsf(r0 + (((ch + 1) ^ t) << 4));
        av[2] = ldsf(r1 + ((ch ^ (t + 4)) << 4));
        av[3] = ldsf(r1 + (((ch + 1) ^ (t + 4)) << 4));
#pragma unroll
        for (int n = 0; n < NCC / 8; ++n) {
            bv[2 * n] = sm.Dp[8 * j + t][8 * n + g];
            bv[2 * n + 1] = sm.Dp[8 * j + t + 4][8 * n + g];
        }
    };
    float av[2][4], bv[2][2 * NCC / 8];
    load(0, av[0], bv[0]);
    // the state from its transposed copy (the values the registers held: left dead
    // through the phases before, they free 24 registers there)
    const int key = mma_key(warp, g);
    float sx[NCC / 8][4];
#pragma unroll
    for (int n = 0; n < NCC / 8; ++n) {
        const float el = b.rec[n >> 1][REC_EG + C - 1];
        const int col = 8 * n + 2 * t;
        S.v[n][0] = sm.SsT[col][key] * el;
        S.v[n][1] = sm.SsT[col + 1][key] * el;
        S.v[n][2] = sm.SsT[col][key + 4] * el;
        S.v[n][3] = sm.SsT[col + 1][key + 4] * el;
#pragma unroll
        for (int i = 0; i < 4; ++i) sx[n][i] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < C / 8; ++j) {  // tokens 8j .. 8j + 7
        const int cur = j & 1;
        if (j + 1 < C / 8) load(j + 1, av[cur ^ 1], bv[cur ^ 1]);
        uint32_t ah[4], al[4], bh[NCC / 8][2], bl[NCC / 8][2];
#pragma unroll
        for (int i = 0; i < 4; ++i) split_tf32(av[cur][i], ah[i], al[i]);
#pragma unroll
        for (int i = 0; i < 2 * NCC / 8; ++i) split_tf32(bv[cur][i], bh[i >> 1][i & 1], bl[i >> 1][i & 1]);
#pragma unroll
        for (int n = 0; n < NCC / 8; ++n) mma_tf32(S.v[n], ah, bh[n]);
#pragma unroll
        for (int n = 0; n < NCC / 8; ++n) mma_tf32(sx[n], ah, bl[n]);
#pragma unroll
        for (int n = 0; n < NCC / 8; ++n) mma_tf32(sx[n], al, bh[n]);
    }
#pragma unroll
    for (int n = 0; n < NCC / 8; ++n) {
#pragma unroll
        for (int i = 0; i < 4; ++i) S.v[n][i] += sx[n][i];
        const int col = 8 * n + 2 * t;
        sm.SsT[col][key] = S.v[n][0];
        sm.SsT[col + 1][key] = S.v[n][1];
        sm.SsT[col][key + 4] = S.v[n][2];
        sm.SsT[col + 1][key + 4] = S.v[n][3];
    }
}

// The scan of key head `kh`, value columns c0..c0+15 of its three heads, over the
// super-block's chunks, with the products as FP32 FMAs (kMma false) or all of them
// as split-TF32 tensor-core MMAs (kMma true).  With `flags` set, chunk c's prep
// records are read only once flags[c * n_kh + kh] == gen (records written by
// other CTAs of the same launch); a flag wait that runs out records the flag's
// index, its last value and `gen` in diag[0..2].  A wait that runs out is
// reported in the status word and the state is left as it was; every thread still
// takes the same path through the chunk loop (a thread that gave up computes on
// whatever landed), so the CTA's barriers stay matched and the CTA ends.
template <bool kMma>
__device__ __forceinline__ void scan_body(const ChunkScanParams& p, ScanSmem& sm, const int kh, const int c0,
                                          const uint32_t* flags, uint32_t* diag, const uint32_t gen,
                                          uint32_t* out_flags = nullptr) {
    const int tid = threadIdx.x;
    const int n_kh = p.n_kh, n_vh = p.n_vh;
    const int nch = (p.n_tokens + C - 1) / C;

    if (tid == 0) {
        mbar_init(&sm.full[0], 1);
        mbar_init(&sm.full[1], 1);
        mbar_init_fence();
        sm.copy_gave_up = 0;
        sm.flag_gave_up = 0;
    }

    ScanState<kMma> S;
    state_load(p, sm, S, kh, c0);
    __syncthreads();

    // k, q and v tiles of chunk c (TMA), on the chunk's buffer barrier, which expects
    // the records too
    auto issue_tiles = [&](int c) {
        ScanBuf& b = sm.buf[c & 1];
        uint64_t* bar = &sm.full[c & 1];
        const int y = static_cast<int>(p.t_begin + static_cast<int64_t>(c) * C);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(bar, kScanTxBytes);
#pragma unroll
        for (int bx = 0; bx < D / 32; ++bx) {
            tma_load_2d(&b.K[bx][0][0], &p.tm_k, bar, kh * D + 32 * bx, y);
            tma_load_2d(&b.Q[bx][0][0], &p.tm_q, bar, kh * D + 32 * bx, y);
        }
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m) tma_load_2d(&b.V[m][0][0], &p.tm_v, bar, (kh + m * n_kh) * D + c0, y);
    };
    // prep records of chunk c (bulk copies); with flags, once the prep task has published them
    auto issue_records = [&](int c) {
        ScanBuf& b = sm.buf[c & 1];
        uint64_t* bar = &sm.full[c & 1];
        if (flags) {
            // records from another CTA: acquire its flag, then read them through the async proxy
            uint32_t seen = 0;
            if (!sm.flag_gave_up && !wait_flag(flags + c * n_kh + kh, gen, &seen)) {
                sm.flag_gave_up = 1;
                report_error(p.status, kDevErrFlagTimeout);
                if (diag) {
                    diag[0] = static_cast<uint32_t>(c * n_kh + kh);
                    diag[1] = seen;
                    diag[2] = gen;
                }
            }
            fence_proxy_async_global();
        }
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m)
            bulk_load(&b.rec[m][0], p.prep + (static_cast<int64_t>(c) * n_vh + kh + m * n_kh) * REC, REC * 4, bar);
    };
    // The issuing lane's warp waits for it at __syncwarp: left to spin on the copy
    // barrier while lane 0 spins on a prep flag, the other lanes can starve lane 0
    // of issue slots until their own wait runs out.
    const int warp = tid >> 5, lane = tid & 31;
    if (warp == 0) {
        if (lane == 0) {
            issue_tiles(0);
            issue_records(0);
        }
        __syncwarp();
    }

    // P2 / P3 tile: head pm, rows 4*pti..+3, columns 2*pjp, 2*pjp+1
    const int pm = tid >> 6, pti = (tid >> 3) & 7, pjp = tid & 7;

    for (int c = 0; c < nch; ++c) {
        // once a copy wait has run out (seen by all after the previous chunk's last
        // barrier), nothing more is issued or waited for
        if (!sm.copy_gave_up && !mbar_wait(&sm.full[c & 1], static_cast<uint32_t>((c >> 1) & 1))) {
            sm.copy_gave_up = c + 1;
            report_timeout(p.status);
        }
        const ScanBuf& b = sm.buf[c & 1];
        const int nt = min(C, p.n_tokens - c * C);

        if constexpr (kMma)
            g1_mma(b, sm);
        else
            g1_fma(b, sm);
        __syncthreads();

        // ---- P2: D = T' U' per head (32x32 by 32x16); warp 7, idle here, loads the next
        //      chunk's tiles into the buffer chunk c-1 last read (and its records, unless
        //      they come from another CTA: those follow in P3, off this phase's barrier) ----
        const bool next = c + 1 < nch && !sm.copy_gave_up;  // copy_gave_up is fixed until the next chunk
        if (warp == SCAN_THREADS / 32 - 1) {
            if (lane == 0 && next) {
                issue_tiles(c + 1);
                if (!flags) issue_records(c + 1);
            }
            // chunk c-1's outputs are stored (barriers since): tell its norm
            if (lane == 0 && out_flags && c > 0) st_release_gpu(out_flags + ((c - 1) * n_kh + kh) * 8 + c0 / NC, gen);
            __syncwarp();
        }
        if constexpr (kMma) {
            if (warp < 2 * kHeadsPerKey) p2_mma(b, sm);
        } else if (tid < kHeadsPerKey * 64) {
            const float* tp = &b.rec[pm][REC_TP];
            float acc[4][2];
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[r][0] = acc[r][1] = 0.f;
#pragma unroll 8
            for (int s = 0; s < C; ++s) {
                const float4 a = *reinterpret_cast<const float4*>(tp + s * C + 4 * pti);
                const float2 u = *reinterpret_cast<const float2*>(&sm.W[s][pm * NC + 2 * pjp]);
                acc[0][0] = fmaf(a.x, u.x, acc[0][0]);
                acc[0][1] = fmaf(a.x, u.y, acc[0][1]);
                acc[1][0] = fmaf(a.y, u.x, acc[1][0]);
                acc[1][1] = fmaf(a.y, u.y, acc[1][1]);
                acc[2][0] = fmaf(a.z, u.x, acc[2][0]);
                acc[2][1] = fmaf(a.z, u.y, acc[2][1]);
                acc[3][0] = fmaf(a.w, u.x, acc[3][0]);
                acc[3][1] = fmaf(a.w, u.y, acc[3][1]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * pti + r;
                const float er = b.rec[pm][REC_ER + t];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int col = pm * NC + 2 * pjp + q;
                    sm.Dm[t][col] = acc[r][q];
                    sm.Dp[t][col] = er * acc[r][q];
                }
            }
        }
        __syncthreads();

        // ---- P3: O = e^gamma Q S0 + P D per head -> out ----
        if (kMma && warp < 2 * kHeadsPerKey) {
            p3_mma(p, b, sm, kh, c0, c, nt);
        } else if (!kMma && tid < kHeadsPerKey * 64) {
            const float* pt = &b.rec[pm][REC_PT];
            float acc[4][2];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float2 w = *reinterpret_cast<const float2*>(&sm.W[C + 4 * pti + r][pm * NC + 2 * pjp]);
                acc[r][0] = w.x;
                acc[r][1] = w.y;
            }
#pragma unroll 8
            for (int s = 0; s < C; ++s) {
                const float4 a = *reinterpret_cast<const float4*>(pt + s * C + 4 * pti);
                const float2 d = *reinterpret_cast<const float2*>(&sm.Dm[s][pm * NC + 2 * pjp]);
                acc[0][0] = fmaf(a.x, d.x, acc[0][0]);
                acc[0][1] = fmaf(a.x, d.y, acc[0][1]);
                acc[1][0] = fmaf(a.y, d.x, acc[1][0]);
                acc[1][1] = fmaf(a.y, d.y, acc[1][1]);
                acc[2][0] = fmaf(a.z, d.x, acc[2][0]);
                acc[2][1] = fmaf(a.z, d.y, acc[2][1]);
                acc[3][0] = fmaf(a.w, d.x, acc[3][0]);
                acc[3][1] = fmaf(a.w, d.y, acc[3][1]);
            }
            const int h = kh + pm * n_kh;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * pti + r;
                if (t < nt) {
                    float* o = p.out + ((p.t_begin + static_cast<int64_t>(c) * C + t) * n_vh + h) * D + c0 + 2 * pjp;
                    *reinterpret_cast<float2*>(o) = make_float2(acc[r][0], acc[r][1]);
                }
            }
        } else if (flags && warp == SCAN_THREADS / 32 - 1) {
            // warp 7 is idle in P3: wait here for the next chunk's prep flag and copy its records
            if (lane == 0 && next) issue_records(c + 1);
            __syncwarp();
        }

        if constexpr (kMma)
            g4_mma(b, sm, S);
        else
            g4_fma(b, sm, S);
        __syncthreads();
    }

    // (the loop ended on a barrier, so copy_gave_up and flag_gave_up are final here)
    if (out_flags && tid == SCAN_THREADS - 32) st_release_gpu(out_flags + ((nch - 1) * n_kh + kh) * 8 + c0 / NC, gen);
    if (sm.copy_gave_up) {
        const int cf = sm.copy_gave_up - 1;  // the one chunk whose copies may still be landing
        if (tid == 0) mbar_wait(&sm.full[cf & 1], static_cast<uint32_t>((cf >> 1) & 1));
        return;
    }
    if (sm.flag_gave_up) return;
    state_store(p, S, kh, c0);
}

// One CTA per (key head, 16 value columns); the prep kernel has run before.
template <bool kMma>
__global__ void __launch_bounds__(SCAN_THREADS, 1) gdn_chunk_scan_kernel(const __grid_constant__ ChunkScanParams p) {
    scan_body<kMma>(p, *aligned_dynamic_smem<ScanSmem, 1024>(), blockIdx.x, blockIdx.y * NC, nullptr, nullptr, 0u);
}

// 16-byte load through L2 only: out is written by other CTAs of the same launch.
__device__ __forceinline__ float4 ld_cg4(const float* ptr) {
    float4 r;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(ptr));
    return r;
}

// The norm of the super-block's outputs by one prep CTA: units (chunk c, key head
// kh) = b, b + n_prep, ... in chunk order; a unit waits until the 8 scan CTAs of
// kh have published chunk c, then norms its 3 heads x (up to) 32 token rows, one
// warp per row (12 rows per warp, six loaded at a time).
__device__ __forceinline__ void norm_units(const ChunkFusedParams& p, const int b, const uint32_t gen) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_kh = p.scan.n_kh, n_vh = p.scan.n_vh;
    const int nch = (p.scan.n_tokens + C - 1) / C;
    const float4 w4 = __ldg(reinterpret_cast<const float4*>(p.w) + lane);
    for (int u = b; u < nch * n_kh; u += p.n_prep) {
        const int c = u / n_kh, kh = u % n_kh;
        if (warp == 0) {
            uint32_t seen = 0;
            bool ok = true;
            if (lane < 8) ok = wait_flag(p.out_flags + (c * n_kh + kh) * 8 + lane, gen, &seen);
            if (!ok) {
                report_error(p.scan.status, kDevErrFlagTimeout);
                p.sync[2] = static_cast<uint32_t>(0x80000000u | ((c * n_kh + kh) * 8 + lane));
                p.sync[3] = seen;
                p.sync[4] = gen;
            }
            __syncwarp();
        }
        __syncthreads();  // the acquires above order the scan CTAs' stores before every warp's loads
        const int nt = min(C, p.scan.n_tokens - c * C);
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            float4 ov[6], zv[6];
            int64_t rows[6];
#pragma unroll
            for (int j = 0; j < 6; ++j) {
                const int i = warp + 8 * (6 * pass + j);  // 0..95: head m = i / 32, token t = i % 32
                const int m = i >> 5, t = i & 31;
                rows[j] = (t < nt) ? (p.scan.t_begin + static_cast<int64_t>(c) * C + t) * n_vh + kh + m * n_kh : -1;
                if (rows[j] >= 0) {
                    ov[j] = ld_cg4(p.scan.out + rows[j] * D + 4 * lane);
                    zv[j] = __ldg(reinterpret_cast<const float4*>(p.z + rows[j] * D) + lane);
                }
            }
#pragma unroll
            for (int j = 0; j < 6; ++j)
                if (rows[j] >= 0)
                    __stcs(reinterpret_cast<uint2*>(p.y) + rows[j] * (D / 4) + lane, norm_row_lane(ov[j], zv[j], w4, p.eps));
        }
    }
}

// ====================== prep and scan in one launch ======================
// The scan occupies 8 n_kh SMs for the whole super-block, the prep only a short
// burst before it.  Here the remaining SMs run the prep while the scan runs: CTAs
// 0..n_prep-1 take the (chunk, key head) prep tasks in chunk order, each
// publishing its records with a release store of this launch's generation
// number; the scan CTAs acquire that flag before copying a chunk's records.  The
// prep CTAs wait on nothing, so the scan's waits end as long as every CTA is
// resident (a cooperative launch guarantees it).  The generation number lives in
// device memory and the last CTA to finish advances it, so a replayed CUDA graph
// of this launch never matches a stale flag.
template <bool kMma>
__global__ void __launch_bounds__(SCAN_THREADS, 1) gdn_chunk_fused_kernel(const __grid_constant__ ChunkFusedParams p) {
    __shared__ uint32_t s_gen;
    const int tid = threadIdx.x;
    if (tid == 0) s_gen = ld_acquire_gpu(p.sync) + 1u;
    __syncthreads();
    const uint32_t gen = s_gen;
    const int b = static_cast<int>(blockIdx.x);
    if (b < p.n_prep) {
        PrepSmemT<2>& sm = *aligned_dynamic_smem<PrepSmemT<2>, 1024>();
        const int n_kh = p.prep.n_kh;
        const int tasks = ((p.prep.n_tokens + C - 1) / C) * n_kh;
        // software pipeline: task i computes from buffer i & 1 while task i+1's tiles load
        if (b < tasks) prep_load(p.prep, sm, 0, b / n_kh, b % n_kh);
        for (int task = b, i = 0; task < tasks; task += p.n_prep, ++i) {
            const int next = task + p.n_prep;
            if (next < tasks) {
                prep_load(p.prep, sm, (i + 1) & 1, next / n_kh, next % n_kh);  // its buffer was freed by task i-1
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            prep_task(p.prep, sm, i & 1, task / n_kh, task % n_kh);
            fence_proxy_async_global();
            __syncthreads();
            if (tid == 0 && task != p.withhold_task) st_release_gpu(p.flags + task, gen);
        }
        if (p.y) norm_units(p, b, gen);
    } else {
        const int s = b - p.n_prep, n_kh = p.scan.n_kh;
        scan_body<kMma>(p.scan, *aligned_dynamic_smem<ScanSmem, 1024>(), s % n_kh, (s / n_kh) * NC, p.flags, p.sync + 2,
                  gen, p.y ? p.out_flags : nullptr);
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(p.sync + 1, 1u) == gridDim.x - 1) {
            p.sync[1] = 0u;
            st_release_gpu(p.sync, gen);
        }
    }
}

}  // namespace

int chunk_scan_box_cols() { return NC; }

cudaError_t launch_chunk_prep(const ChunkPrepParams& p, cudaStream_t s) {
    const size_t smem = sizeof(PrepSmemT<1>) + 16;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(gdn_chunk_prep_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid((p.n_tokens + C - 1) / C, p.n_kh);
    gdn_chunk_prep_kernel<<<grid, PREP_THREADS, smem, s>>>(p);
    return cudaGetLastError();
}

int chunk_fused_prep_ctas(int n_kh, int sm_count) {
    const int n_prep = sm_count - (D / NC) * n_kh;
    return n_prep >= n_kh ? n_prep : 0;
}

cudaError_t launch_chunk_fused(const ChunkFusedParams& p, const bool mma, cudaStream_t s) {
    constexpr size_t body = sizeof(ScanSmem) > sizeof(PrepSmemT<2>) ? sizeof(ScanSmem) : sizeof(PrepSmemT<2>);
    const size_t smem = body + 1024;
    const auto kernel = mma ? gdn_chunk_fused_kernel<true> : gdn_chunk_fused_kernel<false>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_prep + (D / NC) * p.scan.n_kh);
    cfg.blockDim = dim3(SCAN_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t preload_two_launch_chunk_kernels() {
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(gdn_chunk_prep_kernel),
                                  static_cast<int>(sizeof(PrepSmemT<1>) + 16));
    if (e != cudaSuccess) return e;
    const int smem = static_cast<int>(sizeof(ScanSmem) + 1024);
    e = set_smem_once(reinterpret_cast<const void*>(gdn_chunk_scan_kernel<true>), smem);
    if (e != cudaSuccess) return e;
    return set_smem_once(reinterpret_cast<const void*>(gdn_chunk_scan_kernel<false>), smem);
}

cudaError_t launch_chunk_scan(const ChunkScanParams& p, const bool mma, cudaStream_t s) {
    const size_t smem = sizeof(ScanSmem) + 1024;
    const auto kernel = mma ? gdn_chunk_scan_kernel<true> : gdn_chunk_scan_kernel<false>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_kh, D / NC);
    kernel<<<grid, SCAN_THREADS, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
