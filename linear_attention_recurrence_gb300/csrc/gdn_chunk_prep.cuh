// The chunked form's prep ("#1372 DeltaNet recurrence: STRATA_GDN_CHUNKED=1 - the
// prompt's recurrence in 32-token chunks", section "What it does"), shared by the
// scan kernels of gdn_chunk.cu and gdn_chunk_tmem.cu: per (chunk, key head) K K^T
// and Q K^T once for the key head's three value heads, the gates' running sums,
// A and P, and T = (I + A)^-1 by forward substitution.  It writes either the
// records the CUDA-core / warp-MMA scans read (PrepOut::kRecords) or the operand
// tiles of the tensor-memory scan (PrepOut::kTiles).
#pragma once

#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int D = kD;
constexpr int C = kChunk;
constexpr int REC = kPrepRecordFloats;
constexpr int REC_TP = kRecTP;
constexpr int REC_PT = kRecPT;
constexpr int REC_EG = kRecEG;
constexpr int REC_ER = kRecER;

// ---- products on the tensor cores (warp-level m16n8k8 TF32 MMAs) ----
//
// Each FP32 operand x is split as hi = x rounded to TF32 and lo = x - hi (exact),
// and a product a b is taken as hi_a hi_b + (hi_a lo_b + lo_a hi_b): the dropped
// lo_a lo_b and the MMA's truncation of lo to TF32 are below 2^-21 of |a b|, so
// with FP32 accumulation the products keep FP32-level accuracy.  The cross terms
// go to an accumulator of their own and join the main one once.  Operands are
// stored in FP32 and split as they are loaded (three integer / FP32 operations).

// D += A B for one m16n8k8 tile; fragments as the PTX ISA lays them out for .tf32:
// A rows g, g+8 x cols t, t+4; B rows t, t+4 x col g; D rows g, g+8 x cols 2t, 2t+1
// (g = lane / 4, t = lane % 4).
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// hi: x rounded to TF32, to nearest with ties away from zero, by adding half a TF32
// ulp to the bit pattern and clearing the 13 bits below it (two integer operations:
// the conversion instruction issues at a quarter of their rate); finite |x| < 2^127.
// lo: x - hi, exact, whose low 13 bits the MMA ignores.
__device__ __forceinline__ void split_tf32(const float x, uint32_t& hi, uint32_t& lo) {
    hi = (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
    lo = __float_as_uint(x - __uint_as_float(hi));
}

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
    float KK[2][C][C + 1];  // K K^T (lower triangle), partial sums over key dims 0..63 and 64..127
    float QK[2][C][C + 1];  // Q K^T (lower triangle), the same
    float A[kHeadsPerKey][C][C + 4];
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

// How a prep task's threads meet: the whole CTA (the prep kernels, whose CTAs
// are all prep threads), or the first PREP_THREADS threads by a named barrier
// (the tensor-memory kernel, whose CTAs have two more warps that the prep leaves idle).
struct PrepSyncCta {
    static __device__ __forceinline__ void sync() { __syncthreads(); }
};
struct PrepSyncNamed {
    static __device__ __forceinline__ void sync() { asm volatile("bar.sync 1, %0;" ::"n"(PREP_THREADS) : "memory"); }
};

// What a prep task writes: the records of the CUDA-core / warp-MMA scans, or the
// operand tiles of the tensor-memory scan (gdn_internal.h, "tiles of the
// tensor-memory scan", for the layout).
enum class PrepOut { kRecords, kTiles };

// x as TF32 hi (to nearest, ties away: the same integer rounding as split_tf32)
// and lo = x - hi, as FP32 values.
__device__ __forceinline__ void split_f(const float x, float& hi, float& lo) {
    hi = __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
    lo = x - hi;
}
__device__ __forceinline__ void split_f4(const float4 x, float4& hi, float4& lo) {
    split_f(x.x, hi.x, lo.x);
    split_f(x.y, hi.y, lo.y);
    split_f(x.z, hi.z, lo.z);
    split_f(x.w, hi.w, lo.w);
}

// Float offset of element (row, k), k < 32, in a K-major tile of 32-float rows
// with the 128-byte swizzle (16-byte chunk index XOR row % 8).
__device__ __forceinline__ int swf(const int row, const int k) { return row * 32 + ((((k >> 2) ^ row) & 7) << 2) + (k & 3); }

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

// Prep records (or tiles) of chunk `ci` (within the super-block) for key head `kh`
// and its three value heads, by the CTA's PREP_THREADS threads, from buffer `buf`
// (whose copies the caller has waited for and made visible with a barrier).  Ends
// without a barrier (the caller syncs before reusing `sm`).
template <PrepOut OUT = PrepOut::kRecords, class Sync = PrepSyncCta, class PrepSmem>
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
    if constexpr (OUT == PrepOut::kTiles) {
        // [K; Q] (64 rows x 128 key dims, 4 blocks of 32 key dims; per block the 64 hi
        // rows, then the 64 lo rows) and K^T (128 key dims x 32 tokens), split into TF32
        // hi / lo, in the swizzled tile layout
        float* kt = key_tiles(p.prep, p.n_kh, ci, kh);
        for (int it = tid; it < 2 * C * (D / 4); it += PREP_THREADS) {
            const int n = it >> 5, c4 = it & 31;  // row, 16-byte chunk along the key dims
            const float4 x = *reinterpret_cast<const float4*>(&(n < C ? K[n] : Q[n - C])[4 * c4]);
            float4 h, l;
            split_f4(x, h, l);
            float* blk = kt + kTileKQ + (c4 >> 3) * (4 * C * 32);
            *reinterpret_cast<float4*>(blk + swf(n, 4 * (c4 & 7))) = h;
            *reinterpret_cast<float4*>(blk + swf(kTileKQLoRow + n, 4 * (c4 & 7))) = l;
        }
        for (int it = tid; it < D * (C / 4); it += PREP_THREADS) {
            const int r = it & (D - 1), j4 = it >> 7;  // key dim, 4 tokens
            const float4 x = make_float4(K[4 * j4][r], K[4 * j4 + 1][r], K[4 * j4 + 2][r], K[4 * j4 + 3][r]);
            float4 h, l;
            split_f4(x, h, l);
            const int off = swf(r, 4 * j4);
            *reinterpret_cast<float4*>(kt + kTileKTH + off) = h;
            *reinterpret_cast<float4*>(kt + kTileKTL + off) = l;
        }
    }
    Sync::sync();

    // K K^T and Q K^T (only the tiles on or below the diagonal), shared by the key
    // head's three value heads, as split-TF32 MMAs: warp w sums key dims
    // 64 (w >> 2) .. +63 for three 16 x 8 tiles of K K^T (w & 3 < 2) or Q K^T, rows
    // t, columns i: (t 0..15, i 0..7), (0..15, 8..15), (16..31, 0..7) for even w & 3,
    // (16..31, 8..15), (16..31, 16..23), (16..31, 24..31) for odd.  The two halves'
    // sums go to KK[0 / 1] and QK[0 / 1] and are added in a fixed order below.
    {
        const int g = lane >> 2, t4 = lane & 3;
        const int h = warp >> 2, odd = warp & 1;
        const float (*X)[KP] = (warp & 2) ? Q : K;
        const int mt0 = odd ? 1 : 0, mt1 = 1;           // A row tiles of the three MMA tiles
        const int nb0 = odd ? 1 : 0, nb1 = odd ? 2 : 1;  // B column tiles
        const int nb2 = odd ? 3 : 0;                     // third tile: (mt1, nb2)
        float acc[3][4], accx[3][4];
#pragma unroll
        for (int u = 0; u < 3; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[u][e] = accx[u][e] = 0.f;
#pragma unroll 2
        for (int j = 8 * h; j < 8 * h + 8; ++j) {
            uint32_t ah[2][4], al[2][4], bh[3][2], bl[3][2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int row = 16 * (r ? mt1 : mt0) + g;
                split_tf32(X[row][8 * j + t4], ah[r][0], al[r][0]);
                split_tf32(X[row + 8][8 * j + t4], ah[r][1], al[r][1]);
                split_tf32(X[row][8 * j + t4 + 4], ah[r][2], al[r][2]);
                split_tf32(X[row + 8][8 * j + t4 + 4], ah[r][3], al[r][3]);
            }
#pragma unroll
            for (int u = 0; u < 3; ++u) {
                const int col = 8 * (u == 0 ? nb0 : u == 1 ? nb1 : nb2) + g;
                split_tf32(K[col][8 * j + t4], bh[u][0], bl[u][0]);
                split_tf32(K[col][8 * j + t4 + 4], bh[u][1], bl[u][1]);
            }
            // tiles (mt0, nb0), (mt0 or mt1, nb1), (mt1, nb2): for even w the first two
            // share row tile 0, for odd w all three share row tile 1
            uint32_t mh[4], ml[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                mh[e] = odd ? ah[1][e] : ah[0][e];
                ml[e] = odd ? al[1][e] : al[0][e];
            }
            mma_tf32(acc[0], ah[0], bh[0]);
            mma_tf32(acc[1], mh, bh[1]);
            mma_tf32(acc[2], ah[1], bh[2]);
            mma_tf32(accx[0], ah[0], bl[0]);
            mma_tf32(accx[1], mh, bl[1]);
            mma_tf32(accx[2], ah[1], bl[2]);
            mma_tf32(accx[0], al[0], bh[0]);
            mma_tf32(accx[1], ml, bh[1]);
            mma_tf32(accx[2], al[1], bh[2]);
        }
        float (*const dst)[C + 1] = (warp & 2) ? sm.QK[h] : sm.KK[h];
#pragma unroll
        for (int u = 0; u < 3; ++u) {
            const int rt = u == 0 ? mt0 : u == 1 ? (odd ? mt1 : mt0) : mt1;
            const int ct = u == 0 ? nb0 : u == 1 ? nb1 : nb2;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                dst[16 * rt + g + 8 * (e >> 1)][8 * ct + 2 * t4 + (e & 1)] = acc[u][e] + accx[u][e];
        }
    }
    Sync::sync();

    // A (shared memory) and P^T, e^gamma, e^(gamma_last - gamma) (records), four
    // entries per thread at a time: their shared loads first, then the stores (the
    // compiler cannot tell the stores into A from the loads apart)
    // (records: consecutive threads take consecutive rows t of P^T's row i; tiles:
    // consecutive columns i of P's row t, so each warp's stores fill whole rows)
#pragma unroll 1
    for (int r0 = 0; r0 < kHeadsPerKey * C * C / PREP_THREADS; r0 += 4) {
        float av[4], pv[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int idx = tid + (r0 + r) * PREP_THREADS;
            const int m = idx / (C * C);
            const int i = (OUT == PrepOut::kTiles) ? idx % C : (idx / C) % C;
            const int t = (OUT == PrepOut::kTiles) ? (idx / C) % C : idx % C;
            const bool lower = i <= t;
            const float e = lower ? expf(sm.gam[m][t] - sm.gam[m][i]) : 0.f;
            const float kk = sm.KK[0][t][i] + sm.KK[1][t][i], qk = sm.QK[0][t][i] + sm.QK[1][t][i];
            av[r] = (i < t) ? sm.bet[m][t] * e * kk : 0.f;
            pv[r] = lower ? e * qk : 0.f;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int idx = tid + (r0 + r) * PREP_THREADS;
            const int m = idx / (C * C);
            const int i = (OUT == PrepOut::kTiles) ? idx % C : (idx / C) % C;
            const int t = (OUT == PrepOut::kTiles) ? (idx / C) % C : idx % C;
            sm.A[m][t][i] = av[r];
            if constexpr (OUT == PrepOut::kTiles) {
                float* ht = head_tiles(p.prep, p.n_kh, p.n_vh, ci, kh + m * p.n_kh);
                float h, l;
                split_f(pv[r], h, l);
                ht[kTilePH + swf(t, i)] = h;
                ht[kTilePL + swf(t, i)] = l;
            } else {
                float* rec = p.prep + (static_cast<int64_t>(ci) * p.n_vh + kh + m * p.n_kh) * REC;
                rec[REC_PT + i * C + t] = pv[r];
            }
        }
    }
    if (tid < kHeadsPerKey * C) {
        const int m = tid / C, t = tid % C;
        float* eg;
        float* er;
        if constexpr (OUT == PrepOut::kTiles) {
            float* ht = head_tiles(p.prep, p.n_kh, p.n_vh, ci, kh + m * p.n_kh);
            eg = ht + kTileEG;
            er = ht + kTileER;
        } else {
            float* rec = p.prep + (static_cast<int64_t>(ci) * p.n_vh + kh + m * p.n_kh) * REC;
            eg = rec + REC_EG;
            er = rec + REC_ER;
        }
        eg[t] = expf(sm.gam[m][t]);
        er[t] = expf(sm.gam[m][C - 1] - sm.gam[m][t]);
    }
    Sync::sync();

    // T = (I + A)^-1 by forward substitution, lane j owning column j, each row's
    // sum taken as four partial sums over i mod 4 (A is zero from the diagonal on,
    // and so is Tc beyond the rows done); then row j of T'^T is T[:, j] * beta_j.
    if (warp < kHeadsPerKey) {
        const int m = warp, j = lane;
        float Tc[C];
#pragma unroll
        for (int t = 0; t < C; ++t) Tc[t] = 0.f;
#pragma unroll
        for (int t = 0; t < C; ++t) {
            float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i4 = 0; i4 < (t + 3) / 4; ++i4) {
                const float4 a = *reinterpret_cast<const float4*>(&sm.A[m][t][4 * i4]);
                s[0] = fmaf(-a.x, Tc[4 * i4], s[0]);
                s[1] = fmaf(-a.y, Tc[4 * i4 + 1], s[1]);
                s[2] = fmaf(-a.z, Tc[4 * i4 + 2], s[2]);
                s[3] = fmaf(-a.w, Tc[4 * i4 + 3], s[3]);
            }
            Tc[t] = ((t == j) ? 1.f : 0.f) + ((s[0] + s[1]) + (s[2] + s[3]));
        }
        const float bj = sm.bet[m][j];
        if constexpr (OUT == PrepOut::kTiles) {
            // T' row-major: lane j writes column j, so each t fills one tile row
            float* ht = head_tiles(p.prep, p.n_kh, p.n_vh, ci, kh + m * p.n_kh);
#pragma unroll
            for (int t = 0; t < C; ++t) {
                float h, l;
                split_f(Tc[t] * bj, h, l);
                ht[kTileTPH + swf(t, j)] = h;
                ht[kTileTPL + swf(t, j)] = l;
            }
        } else {
            float* rec = p.prep + (static_cast<int64_t>(ci) * p.n_vh + kh + m * p.n_kh) * REC;
            float4* dst = reinterpret_cast<float4*>(rec + REC_TP + j * C);
#pragma unroll
            for (int t4 = 0; t4 < C / 4; ++t4)
                dst[t4] = make_float4(Tc[4 * t4] * bj, Tc[4 * t4 + 1] * bj, Tc[4 * t4 + 2] * bj, Tc[4 * t4 + 3] * bj);
        }
    }
}


}  // namespace
}  // namespace gdn
