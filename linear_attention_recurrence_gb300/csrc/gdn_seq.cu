// Sequential Gated DeltaNet scan for sm_103a.
//
// Computes, per value head h (key head kh = h % n_kh) and token t, exactly one
// token at a time ("#413 prefill: DeltaNet recurrence with the three value heads
// of a key head in one thread", section "What changes"):
//     sk_j = sum_i S[i][j] k_i,  sq_j = sum_i S[i][j] q_i      (state before t)
//     delta_j = beta (v_j - e^g sk_j)
//     o_j = e^g sq_j + (k.q) delta_j                            (= S_t^T q)
//     S[i][j] <- e^g S[i][j] + k_i delta_j
// One pass over the state gives both sums, because S_t^T q = e^g S^T q +
// (k.q) delta; the Metal scan of "Round 20 Track C Audit: gdn_pre ... gdn_scan_r
// ..." section 1 feeds a precomputed k.q into its scan for the same purpose.
//
// Work split (GB300-first, not the pages' 64-block layout): one CTA per (key
// head, 16 value columns) covers those columns in the key head's three value
// heads, so every k/q value a thread loads feeds three heads.  A column's 128
// rows are split over G = 128/R lanes of one warp (R rows per lane, interleaved
// in groups of four so that the lanes' float4 loads of k and q are conflict
// free); the column sums are reduced with a fixed xor-shuffle tree, so every lane
// of the column ends with bit-identical sums and no CTA barrier is needed per
// token.  The state slice lives in registers for the whole call.  A producer warp
// stages B-token blocks of k, q and v with TMA into a 4-deep ring and fills in
// e^g, beta and k.q for each token; consumer warps run ahead of each other
// within the ring.  Per token every lane does its arithmetic in the same order,
// independent of the token's position in the block or the call, so a sequence
// split over calls gives the same bits as one call.
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int D = kD;
constexpr int NCOL = 16;  // value columns per CTA (per head)
constexpr int B = 16;     // tokens per stage (the producer's k.q reduce-scatter assumes 16)
static_assert(B == 16, "k.q reduce-scatter layout");
constexpr int NS = 4;     // stages in the ring

template <int R>
struct SeqShape {
    static_assert(R % 4 == 0 && D % R == 0, "rows per lane");
    static constexpr int G = D / R;          // lanes per column
    static constexpr int CPW = 32 / G;       // columns per warp
    static constexpr int NCW = NCOL / CPW;   // consumer warps
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int P4 = R / 4;         // float4 row groups per lane
};

struct __align__(128) Stage {
    float k[B][D];          // TMA: k rows of the key head
    float q[B][D];          // TMA: q rows of the key head
    float v[kHeadsPerKey][B][NCOL];  // TMA: the CTA's value columns of each head
    float a[B][4];          // producer: e^g per head
    float b[B][4];          // producer: beta per head
    float kq[B];            // producer: k . q
};
constexpr uint32_t kStageTxBytes = 2 * B * D * 4 + kHeadsPerKey * B * NCOL * 4;

struct SeqSmem {
    Stage st[NS];
    uint64_t full[NS];   // TMA bytes landed
    uint64_t ready[NS];  // producer's per-token scalars written
    uint64_t empty[NS];  // every consumer warp is done with the stage
};

template <int R>
__global__ void __launch_bounds__(SeqShape<R>::THREADS, 1) gdn_seq_kernel(const __grid_constant__ SeqParams p) {
    using Sh = SeqShape<R>;
    SeqSmem& sm = *aligned_dynamic_smem<SeqSmem, 1024>();
    const int kh = blockIdx.x;
    const int c0 = blockIdx.y * NCOL;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t T = p.T;
    const int n_kh = p.n_kh, n_vh = p.n_vh;
    const int64_t nst = (T + B - 1) / B;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.ready[s], 1);
            mbar_init(&sm.empty[s], Sh::NCW);
        }
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == Sh::NCW) {
        // ---------------- producer warp ----------------
        auto issue = [&](int64_t s) {
            Stage& st = sm.st[s % NS];
            uint64_t* bar = &sm.full[s % NS];
            const int y = static_cast<int>(s * B);
            mbar_arrive_expect_tx(bar, kStageTxBytes);
            tma_load_2d(st.k, &p.tm_k, bar, kh * D, y);
            tma_load_2d(st.q, &p.tm_q, bar, kh * D, y);
#pragma unroll
            for (int m = 0; m < kHeadsPerKey; ++m)
                tma_load_2d(st.v[m], &p.tm_v, bar, (kh + m * n_kh) * D + c0, y);
        };
        int64_t issued = nst < NS ? nst : NS;
        if (lane == 0)
            for (int64_t s = 0; s < issued; ++s) issue(s);
        __syncwarp();  // lanes 1..31 must not spin on a barrier while lane 0 still has copies to issue
        int64_t landed = 0;  // stages whose full barrier this warp has observed
        bool ok = true;
        for (int64_t s = 0; s < nst && ok; ++s) {
            const int buf = static_cast<int>(s % NS);
            Stage& st = sm.st[buf];
            for (int idx = lane; idx < kHeadsPerKey * B; idx += 32) {
                const int tt = idx / kHeadsPerKey, m = idx % kHeadsPerKey;
                const int64_t t = s * B + tt;
                float gv = 0.f, bv = 0.f;
                if (t < T) {
                    gv = __ldg(p.g + t * n_vh + kh + m * n_kh);
                    bv = __ldg(p.beta + t * n_vh + kh + m * n_kh);
                }
                st.a[tt][m] = expf(gv);
                st.b[tt][m] = bv;
            }
            if (!mbar_wait(&sm.full[buf], static_cast<uint32_t>((s / NS) & 1))) { ok = false; break; }
            landed = s + 1;
            // k.q of the block's 16 tokens: lane partials over dims 4*lane..4*lane+3, then
            // a reduce-scatter over the warp (keep half the tokens at each xor level),
            // so lanes 2u and 2u+1 end with token 8*b4 + 4*b3 + 2*b2 + b1 of lane 2u.
            float kqv[B];
#pragma unroll
            for (int tt = 0; tt < B; ++tt) {
                const float4 k4 = reinterpret_cast<const float4*>(st.k[tt])[lane];
                const float4 q4 = reinterpret_cast<const float4*>(st.q[tt])[lane];
                kqv[tt] = fmaf(k4.w, q4.w, fmaf(k4.z, q4.z, fmaf(k4.y, q4.y, k4.x * q4.x)));
            }
#pragma unroll
            for (int lvl = 0; lvl < 4; ++lvl) {
                const int off = 16 >> lvl, half = B >> (lvl + 1);
                const bool upper = (lane & off) != 0;
#pragma unroll
                for (int i = 0; i < half; ++i) {
                    const float send = upper ? kqv[i] : kqv[i + half];
                    const float keep = upper ? kqv[i + half] : kqv[i];
                    kqv[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            kqv[0] += __shfl_xor_sync(0xffffffffu, kqv[0], 1);
            if ((lane & 1) == 0)
                st.kq[((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1)] = kqv[0];
            __threadfence_block();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.ready[buf]);
            // Refill the buffer the consumers finished last.
            if (s >= 1 && s - 1 + NS < nst) {
                const int64_t r = s - 1;
                if (!mbar_wait(&sm.empty[r % NS], static_cast<uint32_t>((r / NS) & 1))) { ok = false; break; }
                if (lane == 0) issue(r + NS);
                __syncwarp();
                issued = r + NS + 1;
            }
        }
        if (!ok) {
            // Record the failure, then let every issued copy land before the CTA exits.
            if (lane == 0) report_timeout(p.status);
            for (int64_t s = landed; s < issued; ++s)
                mbar_wait(&sm.full[s % NS], static_cast<uint32_t>((s / NS) & 1));
        }
        return;
    }

    // ---------------- consumer warps ----------------
    const int colw = lane / Sh::G;
    const int rg = lane % Sh::G;
    const int cl = warp * Sh::CPW + colw;  // column within the CTA
    const int c = c0 + cl;
    // rows of this lane: 4*rg + 4*G*pp + u, pp < R/4, u < 4
    float2 S[kHeadsPerKey][Sh::P4][2];
#pragma unroll
    for (int m = 0; m < kHeadsPerKey; ++m) {
        const float* sh = p.state + static_cast<int64_t>(kh + m * n_kh) * D * D + c;
#pragma unroll
        for (int pp = 0; pp < Sh::P4; ++pp) {
            const int row = 4 * rg + 4 * Sh::G * pp;
            S[m][pp][0] = make_float2(sh[(row + 0) * D], sh[(row + 1) * D]);
            S[m][pp][1] = make_float2(sh[(row + 2) * D], sh[(row + 3) * D]);
        }
    }
    float* out_col = p.out + static_cast<int64_t>(kh + (rg < kHeadsPerKey ? rg : 0) * n_kh) * D + c;

    // One token's operands, loaded from the stage one token ahead of use.
    struct Ops {
        float4 k[Sh::P4], q[Sh::P4];
        float a[kHeadsPerKey], b[kHeadsPerKey], v[kHeadsPerKey], kq;
    };
    auto load = [&](Ops& o, const Stage& st, int tt) {
        const float4* k4 = reinterpret_cast<const float4*>(st.k[tt]);
        const float4* q4 = reinterpret_cast<const float4*>(st.q[tt]);
#pragma unroll
        for (int pp = 0; pp < Sh::P4; ++pp) {
            o.k[pp] = k4[rg + Sh::G * pp];
            o.q[pp] = q4[rg + Sh::G * pp];
        }
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m) {
            o.a[m] = st.a[tt][m];
            o.b[m] = st.b[tt][m];
            o.v[m] = st.v[m][tt][cl];
        }
        o.kq = st.kq[tt];
    };
    // One token: both column sums from one pass over the state (12 independent
    // packed accumulator chains), the k-sum reduction first (it gates delta), the
    // decay product a*S formed while the shuffles are in flight, then the update;
    // the q-sum reduction and the output come last, off the state's critical path.
    auto token = [&](const Ops& o, int64_t t) {
        float2 ak[kHeadsPerKey][2], aq[kHeadsPerKey][2];
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m)
            ak[m][0] = ak[m][1] = aq[m][0] = aq[m][1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int pp = 0; pp < Sh::P4; ++pp) {
            const float2 k01 = make_float2(o.k[pp].x, o.k[pp].y), k23 = make_float2(o.k[pp].z, o.k[pp].w);
            const float2 q01 = make_float2(o.q[pp].x, o.q[pp].y), q23 = make_float2(o.q[pp].z, o.q[pp].w);
#pragma unroll
            for (int m = 0; m < kHeadsPerKey; ++m) {
                ak[m][0] = ffma2(S[m][pp][0], k01, ak[m][0]);
                ak[m][1] = ffma2(S[m][pp][1], k23, ak[m][1]);
                aq[m][0] = ffma2(S[m][pp][0], q01, aq[m][0]);
                aq[m][1] = ffma2(S[m][pp][1], q23, aq[m][1]);
            }
        }
        float sk[kHeadsPerKey], sq[kHeadsPerKey];
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m) {
            sk[m] = (ak[m][0].x + ak[m][0].y) + (ak[m][1].x + ak[m][1].y);
            sq[m] = (aq[m][0].x + aq[m][0].y) + (aq[m][1].x + aq[m][1].y);
        }
#pragma unroll
        for (int off = 1; off < Sh::G; off <<= 1) {
#pragma unroll
            for (int m = 0; m < kHeadsPerKey; ++m) sk[m] += __shfl_xor_sync(0xffffffffu, sk[m], off);
        }
        float delta[kHeadsPerKey];
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m) {
            const float a = o.a[m];
            const float2 a2 = make_float2(a, a);
#pragma unroll
            for (int pp = 0; pp < Sh::P4; ++pp) {
                S[m][pp][0] = fmul2(a2, S[m][pp][0]);
                S[m][pp][1] = fmul2(a2, S[m][pp][1]);
            }
            delta[m] = o.b[m] * (o.v[m] - a * sk[m]);
        }
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m) {
            const float2 d2 = make_float2(delta[m], delta[m]);
#pragma unroll
            for (int pp = 0; pp < Sh::P4; ++pp) {
                S[m][pp][0] = ffma2(make_float2(o.k[pp].x, o.k[pp].y), d2, S[m][pp][0]);
                S[m][pp][1] = ffma2(make_float2(o.k[pp].z, o.k[pp].w), d2, S[m][pp][1]);
            }
        }
#pragma unroll
        for (int off = 1; off < Sh::G; off <<= 1) {
#pragma unroll
            for (int m = 0; m < kHeadsPerKey; ++m) sq[m] += __shfl_xor_sync(0xffffffffu, sq[m], off);
        }
        float o_mine = 0.f;
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m) {
            const float out = fmaf(o.kq, delta[m], o.a[m] * sq[m]);
            if (rg == m) o_mine = out;
        }
        if (rg < kHeadsPerKey) out_col[t * static_cast<int64_t>(n_vh) * D] = o_mine;
    };

    for (int64_t s = 0; s < nst; ++s) {
        const int buf = static_cast<int>(s % NS);
        const uint32_t par = static_cast<uint32_t>((s / NS) & 1);
        if (!mbar_wait(&sm.full[buf], par) || !mbar_wait(&sm.ready[buf], par)) {
            if (lane == 0) report_timeout(p.status);
            return;
        }
        const Stage& st = sm.st[buf];
        const int64_t rem = T - s * B;
        const int nt = rem < B ? static_cast<int>(rem) : B;
        const int64_t t0 = s * B;
        Ops x0, x1;
        load(x0, st, 0);
        int tt = 0;
#pragma unroll 1
        for (; tt + 1 < nt; tt += 2) {
            load(x1, st, tt + 1);
            token(x0, t0 + tt);
            if (tt + 2 < nt) load(x0, st, tt + 2);
            token(x1, t0 + tt + 1);
        }
        if (tt < nt) token(x0, t0 + tt);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[buf]);
    }

#pragma unroll
    for (int m = 0; m < kHeadsPerKey; ++m) {
        float* sh = p.state + static_cast<int64_t>(kh + m * n_kh) * D * D + c;
#pragma unroll
        for (int pp = 0; pp < Sh::P4; ++pp) {
            const int row = 4 * rg + 4 * Sh::G * pp;
            sh[(row + 0) * D] = S[m][pp][0].x;
            sh[(row + 1) * D] = S[m][pp][0].y;
            sh[(row + 2) * D] = S[m][pp][1].x;
            sh[(row + 3) * D] = S[m][pp][1].y;
        }
    }
}

template <int R>
cudaError_t launch_seq_t(const SeqParams& p, cudaStream_t s) {
    using Sh = SeqShape<R>;
    const size_t smem = sizeof(SeqSmem) + 1024;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(gdn_seq_kernel<R>), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_kh, D / NCOL);
    gdn_seq_kernel<R><<<grid, Sh::THREADS, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

int seq_tokens_per_stage() { return B; }
int seq_box_cols() { return NCOL; }

cudaError_t launch_seq(const SeqParams& p, int rows_per_thread, cudaStream_t s) {
    if (rows_per_thread == 8) return launch_seq_t<8>(p, s);
    return launch_seq_t<16>(p, s);
}

}  // namespace gdn
