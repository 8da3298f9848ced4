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
// The large products (K S0, Q S0, K^T D) run as register-tiled packed FP32x2 FMAs;
// the tolerance the path is held to (2e-6 relative to FP64) leaves no room for
// TF32 tensor-core inputs there.
#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_norm_row.cuh"

namespace gdn {
namespace {

constexpr int D = kD;
constexpr int C = kChunk;
constexpr int REC = kPrepRecordFloats;
constexpr int REC_TP = kRecTP;
constexpr int REC_PT = kRecPT;
constexpr int REC_EG = kRecEG;
constexpr int REC_ER = kRecER;

// ============================ prep ============================
constexpr int PREP_THREADS = 256;
constexpr int KP = D + 4;  // padded row stride of the k / q tiles

// NB tile buffers: two when a CTA runs several tasks (a task's tiles load while
// the task before computes), one for the one-task-per-CTA prep kernel.
template <int NB>
struct PrepSmemT {
    float K[NB][C][KP];
    float Q[NB][C][KP];
    float graw[NB][kHeadsPerKey][C];
    float braw[NB][kHeadsPerKey][C];
    float KK[C][C + 1];
    float QK[C][C + 1];
    float A[kHeadsPerKey][C][C + 1];
    float gam[kHeadsPerKey][C];
    float bet[kHeadsPerKey][C];
};

// Asynchronous copies (cp.async) of `bytes` (16 or 4) from global memory; with
// `valid` false nothing is read and the destination is zero-filled.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Starts the copies of chunk `ci`'s k and q rows of key head `kh` and the gates
// of its three value heads into buffer `buf` (one commit group; rows past the
// super-block's end are zero-filled: exactly neutral, see the file comment).
template <class PrepSmem>
__device__ __forceinline__ void prep_load(const ChunkPrepParams& p, PrepSmem& sm, const int buf, const int ci,
                                          const int kh) {
    const int tid = threadIdx.x;
    const int t0 = ci * C;
    const int n = min(C, p.n_tokens - t0);
    const int64_t tb = p.t_begin + t0;
    for (int idx = tid; idx < C * (D / 4); idx += PREP_THREADS) {
        const int r = idx / (D / 4), c4 = idx % (D / 4);
        const int64_t off = ((tb + min(r, n - 1)) * p.n_kh + kh) * D + 4 * c4;  // in bounds even when unused
        cp_async16(&sm.K[buf][r][4 * c4], p.k + off, r < n);
        cp_async16(&sm.Q[buf][r][4 * c4], p.q + off, r < n);
    }
    if (tid < kHeadsPerKey * C) {
        const int m = tid / C, t = tid % C;
        const int64_t off = (tb + min(t, n - 1)) * p.n_vh + kh + m * p.n_kh;
        cp_async4(&sm.graw[buf][m][t], p.g + off, t < n);
        cp_async4(&sm.braw[buf][m][t], p.beta + off, t < n);
    }
    cp_async_commit();
}

// Prep records of chunk `ci` (within the super-block) for key head `kh` and its
// three value heads, by the CTA's PREP_THREADS threads, from buffer `buf` (whose
// copies the caller has waited for and made visible with a barrier).  Ends
// without a barrier (the caller syncs before reusing `sm`).
template <class PrepSmem>
__device__ __forceinline__ void prep_task(const ChunkPrepParams& p, PrepSmem& sm, const int buf, const int ci,
                                          const int kh) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float (*const K)[KP] = sm.K[buf];
    float (*const Q)[KP] = sm.Q[buf];
    if (warp < kHeadsPerKey) {
        const float gv = sm.graw[buf][warp][lane], bv = sm.braw[buf][warp][lane];
        // inclusive running sum of the gate over the chunk (fixed shuffle order)
        float x = gv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        sm.gam[warp][lane] = x;
        sm.bet[warp][lane] = bv;
    }
    __syncthreads();

    // K K^T and Q K^T, shared by the key head's three value heads.
    {
        const int t = tid >> 3, ig = tid & 7;
        float kk[4] = {0.f, 0.f, 0.f, 0.f}, qk[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int c4 = 0; c4 < D / 4; ++c4) {
            const float4 kt = *reinterpret_cast<const float4*>(&K[t][4 * c4]);
            const float4 qt = *reinterpret_cast<const float4*>(&Q[t][4 * c4]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 ki = *reinterpret_cast<const float4*>(&K[ig + 8 * u][4 * c4]);
                kk[u] = fmaf(kt.x, ki.x, kk[u]);
                kk[u] = fmaf(kt.y, ki.y, kk[u]);
                kk[u] = fmaf(kt.z, ki.z, kk[u]);
                kk[u] = fmaf(kt.w, ki.w, kk[u]);
                qk[u] = fmaf(qt.x, ki.x, qk[u]);
                qk[u] = fmaf(qt.y, ki.y, qk[u]);
                qk[u] = fmaf(qt.z, ki.z, qk[u]);
                qk[u] = fmaf(qt.w, ki.w, qk[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            sm.KK[t][ig + 8 * u] = kk[u];
            sm.QK[t][ig + 8 * u] = qk[u];
        }
    }
    __syncthreads();

    // A (shared memory) and P^T, e^gamma, e^(gamma_last - gamma) (records).
    for (int idx = tid; idx < kHeadsPerKey * C * C; idx += PREP_THREADS) {
        const int m = idx / (C * C), i = (idx / C) % C, t = idx % C;
        float* rec = p.prep + (static_cast<int64_t>(ci) * p.n_vh + kh + m * p.n_kh) * REC;
        const float e = (i <= t) ? expf(sm.gam[m][t] - sm.gam[m][i]) : 0.f;
        sm.A[m][t][i] = (i < t) ? sm.bet[m][t] * e * sm.KK[t][i] : 0.f;
        rec[REC_PT + i * C + t] = e * sm.QK[t][i];
    }
    if (tid < kHeadsPerKey * C) {
        const int m = tid / C, t = tid % C;
        float* rec = p.prep + (static_cast<int64_t>(ci) * p.n_vh + kh + m * p.n_kh) * REC;
        rec[REC_EG + t] = expf(sm.gam[m][t]);
        rec[REC_ER + t] = expf(sm.gam[m][C - 1] - sm.gam[m][t]);
    }
    __syncthreads();

    // T = (I + A)^-1 by forward substitution, lane j owning column j; then
    // row j of T'^T is T[:, j] * beta_j.
    if (warp < kHeadsPerKey) {
        const int m = warp, j = lane;
        float Tc[C];
#pragma unroll
        for (int t = 0; t < C; ++t) {
            float s = (t == j) ? 1.f : 0.f;
#pragma unroll
            for (int i = 0; i < t; ++i) s = fmaf(-sm.A[m][t][i], Tc[i], s);
            Tc[t] = s;
        }
        const float bj = sm.bet[m][j];
        float* rec = p.prep + (static_cast<int64_t>(ci) * p.n_vh + kh + m * p.n_kh) * REC;
        float4* dst = reinterpret_cast<float4*>(rec + REC_TP + j * C);
#pragma unroll
        for (int t4 = 0; t4 < C / 4; ++t4)
            dst[t4] = make_float4(Tc[4 * t4] * bj, Tc[4 * t4 + 1] * bj, Tc[4 * t4 + 2] * bj, Tc[4 * t4 + 3] * bj);
    }
}

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

struct ScanSmem {
    ScanBuf buf[2];
    float SsT[NCC][SST];     // S0 transposed: [head*16 + col][key dim]
    float W[2 * C][NCC];     // rows 0..31: U'; rows 32..63: e^gamma (Q S0)
    float Dm[C][NCC];        // D
    float Dp[C][NCC];        // e^(gamma_last - gamma) D
    uint64_t full[2];
    int copy_gave_up;        // 1 + the chunk whose copy wait ran out, else 0
    int flag_gave_up;        // a prep flag wait ran out (later ones are skipped)
};

// byte offset of float4 chunk `cc` (0..7) of row `r` in a 128-byte-swizzled box
__device__ __forceinline__ int swz(int r, int cc) { return r * 128 + ((cc ^ (r & 7)) << 4); }

// The scan of key head `kh`, value columns c0..c0+15 of its three heads, over the
// super-block's chunks.  With `flags` set, chunk c's prep records are read only
// once flags[c * n_kh + kh] == gen (records written by other CTAs of the same
// launch); a flag wait that runs out records the flag's index, its last value and
// `gen` in diag[0..2].  A wait that runs out is reported in the status word and
// the state is left as it was; every thread still takes the same path through
// the chunk loop (a thread that gave up computes on whatever landed), so the
// CTA's barriers stay matched and the CTA ends.
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

    // state slice -> registers (G4 tile: rows 8*it..8*it+7, column c0+j of each head)
    const int it = tid >> 4, jj = tid & 15;
    float2 Sreg[kHeadsPerKey][4];
#pragma unroll
    for (int m = 0; m < kHeadsPerKey; ++m) {
        const float* sh = p.state + (static_cast<int64_t>(kh + m * n_kh) * D + 8 * it) * D + c0 + jj;
#pragma unroll
        for (int q = 0; q < 4; ++q) Sreg[m][q] = make_float2(sh[(2 * q) * D], sh[(2 * q + 1) * D]);
#pragma unroll
        for (int h4 = 0; h4 < 2; ++h4)
            *reinterpret_cast<float4*>(&sm.SsT[m * NC + jj][8 * it + 4 * h4]) =
                make_float4(Sreg[m][2 * h4].x, Sreg[m][2 * h4].y, Sreg[m][2 * h4 + 1].x, Sreg[m][2 * h4 + 1].y);
    }
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

    // G1 tile: warp tg takes X rows 8*(tg&3)..+7 of K (tg < 4) or Q (tg >= 4); lane
    // bit 4 picks the key-dim half kgrp (dims 0..63 or 64..127) and the low four bits
    // the column jw of each head.  Each quarter-warp shares its rows and half, so the
    // X loads are broadcasts; the halves' partial sums meet by a shuffle.
    const int tg = warp, kgrp = (lane >> 4) & 1, jw = lane & 15;
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

        // ---- G1: W = [K; Q] S0 (64 x 48), packed over even/odd key dims, the key dims
        //      split over the two half-warps and their partial sums added once ----
        {
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
        if (tid < kHeadsPerKey * 64) {
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
        if (tid < kHeadsPerKey * 64) {
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

        // ---- G4: S_end = e^gamma_last S0 + K^T (e^(gamma_last-gamma) D), packed over key-dim pairs ----
        {
            const unsigned char* kb = reinterpret_cast<const unsigned char*>(&b.K[it >> 2][0][0]);
            const int cc0 = 2 * (it & 3);
            float2 acc[kHeadsPerKey][4];
#pragma unroll
            for (int m = 0; m < kHeadsPerKey; ++m) {
                const float el = b.rec[m][REC_EG + C - 1];
                const float2 el2 = make_float2(el, el);
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[m][q] = fmul2(el2, Sreg[m][q]);
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
                for (int q = 0; q < 4; ++q) Sreg[m][q] = acc[m][q];
#pragma unroll
                for (int h4 = 0; h4 < 2; ++h4)
                    *reinterpret_cast<float4*>(&sm.SsT[m * NC + jj][8 * it + 4 * h4]) =
                        make_float4(acc[m][2 * h4].x, acc[m][2 * h4].y, acc[m][2 * h4 + 1].x, acc[m][2 * h4 + 1].y);
            }
        }
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
#pragma unroll
    for (int m = 0; m < kHeadsPerKey; ++m) {
        float* sh = p.state + (static_cast<int64_t>(kh + m * n_kh) * D + 8 * it) * D + c0 + jj;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            sh[(2 * q) * D] = Sreg[m][q].x;
            sh[(2 * q + 1) * D] = Sreg[m][q].y;
        }
    }
}

// One CTA per (key head, 16 value columns); the prep kernel has run before.
__global__ void __launch_bounds__(SCAN_THREADS, 1) gdn_chunk_scan_kernel(const __grid_constant__ ChunkScanParams p) {
    scan_body(p, *aligned_dynamic_smem<ScanSmem, 1024>(), blockIdx.x, blockIdx.y * NC, nullptr, nullptr, 0u);
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
        scan_body(p.scan, *aligned_dynamic_smem<ScanSmem, 1024>(), s % n_kh, (s / n_kh) * NC, p.flags, p.sync + 2,
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

cudaError_t launch_chunk_fused(const ChunkFusedParams& p, cudaStream_t s) {
    constexpr size_t body = sizeof(ScanSmem) > sizeof(PrepSmemT<2>) ? sizeof(ScanSmem) : sizeof(PrepSmemT<2>);
    const size_t smem = body + 1024;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(gdn_chunk_fused_kernel), static_cast<int>(smem));
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
    return cudaLaunchKernelEx(&cfg, gdn_chunk_fused_kernel, p);
}

cudaError_t launch_chunk_scan(const ChunkScanParams& p, cudaStream_t s) {
    const size_t smem = sizeof(ScanSmem) + 1024;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(gdn_chunk_scan_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_kh, D / NC);
    gdn_chunk_scan_kernel<<<grid, SCAN_THREADS, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
