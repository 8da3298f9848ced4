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
// e^g, beta and k.q for each token; consumer warps run ahead of each other within
// the ring.
//
// With the gated RMSNorm fused in (gdn_recurrence_norm, "#413 ..." section "What
// changes": the FP32 output is only the norm's input), the consumers write each
// block's outputs to shared memory and four more warps per CTA (one per SM
// sub-partition, each a quarter of the block's rows) norm them: per (token,
// head) row a norm warp publishes the sums of squares of its CTA's four 4-column
// groups in global memory (a release counter per row), gathers the other seven
// CTAs' of the key head (acquire), adds the row's 32 group sums in the order
// gdn_out_norm's warp does (so y has that kernel's bits), and writes y (FP16);
// the producer loads z and stores the FP32 output by TMA, or not at all.  That form is a
// cooperative launch, so the eight CTAs of a key head are resident together and
// their waits end.  (Eight-CTA clusters with distributed shared memory would
// avoid the global round trip, but at one CTA per SM a GB300 holds only 15 such
// clusters at once, one short of 16 key heads.)
//
// Per token every lane does its arithmetic in the same order, independent of
// the token's position in the block or the call, so a sequence split over calls
// gives the same bits as one call.
#include <cstddef>

#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_norm_row.cuh"

namespace gdn {
namespace {

constexpr int D = kD;
constexpr int NCOL = 16;  // value columns per CTA (per head)
constexpr int B = 16;     // tokens per stage (the producer's k.q reduce-scatter assumes 16)
static_assert(B == 16, "k.q reduce-scatter layout");
constexpr int NS = 4;     // stages in the ring
constexpr int SLICES = D / NCOL;           // CTAs (column slices) of a key head
constexpr int ROWS = kHeadsPerKey * B;     // (head, token) rows of a stage
constexpr int NSX = 2;                     // slots of the exchange between the CTAs of a key head
constexpr int kNormWarps = 2;              // norm warps per CTA (one per SM sub-partition)
constexpr int NROWS = ROWS / kNormWarps;   // rows of a stage each norm warp norms
static_assert(NROWS <= 32 && NROWS * kNormWarps == ROWS, "rows per norm warp");

template <int R, bool NORM>
struct SeqShape {
    static_assert(R % 4 == 0 && D % R == 0, "rows per lane");
    static constexpr int G = D / R;          // lanes per column
    static constexpr int CPW = 32 / G;       // columns per warp
    static constexpr int NCW = NCOL / CPW;   // consumer warps
    static constexpr int PRODUCER = NCW;     // warp index of the producer
    static constexpr int NORM0 = NCW + 1;    // warp index of the first norm warp (NORM only)
    static constexpr int THREADS = (NCW + 1 + (NORM ? kNormWarps : 0)) * 32;
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

// The fused norm's buffers.
struct __align__(128) NormBufs {
    float z[NS][kHeadsPerKey][B][NCOL];       // TMA: the gate z of the stage's rows and columns
    float r[kNormWarps][NROWS];               // per row: 1 / sqrt(mean o^2 + eps)
};
constexpr uint32_t kZTxBytes = kHeadsPerKey * B * NCOL * 4;

// The plain scan uses the members up to `o` only, and is launched with that much.
struct SeqSmem {
    Stage st[NS];
    uint64_t full[NS];    // TMA bytes landed
    uint64_t ready[NS];   // producer's per-token scalars written (and the stage's output tiles free)
    uint64_t empty[NS];   // every consumer warp is done with the stage's inputs and has written its outputs
    uint64_t zfull[NS];   // norm: z tile landed
    uint64_t normed[NS];  // norm: every norm warp is done with the stage's output and z tiles
    alignas(128) float o[NS][kHeadsPerKey][B][NCOL];  // norm: each stage's outputs
    NormBufs nb;                                      // norm
};

// ---------------- producer warp ----------------
template <int R, bool NORM>
__device__ void producer_role(const SeqParams& p, SeqSmem& sm, int kh, int c0, int lane) {
    // parameters read once into registers (see consumer_role)
    const int64_t T = p.T;
    const int n_kh = p.n_kh, n_vh = p.n_vh;
    const float* const gp = p.g;
    const float* const betap = p.beta;
    const bool store_out = NORM && p.out != nullptr;
    int* const status = p.status;
    const int64_t nst = (T + B - 1) / B;
    auto issue = [&](int64_t s) {
        Stage& st = sm.st[s % NS];
        uint64_t* bar = &sm.full[s % NS];
        const int y = static_cast<int>(s * B);
        mbar_arrive_expect_tx(bar, kStageTxBytes);
        tma_load_2d(st.k, &p.tm_k, bar, kh * D, y);
        tma_load_2d(st.q, &p.tm_q, bar, kh * D, y);
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m) tma_load_2d(st.v[m], &p.tm_v, bar, (kh + m * n_kh) * D + c0, y);
    };
    auto issue_z = [&](int64_t s) {  // with the norm: the gate z of stage s
        uint64_t* bar = &sm.zfull[s % NS];
        mbar_arrive_expect_tx(bar, kZTxBytes);
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m)
            tma_load_2d(&sm.nb.z[s % NS][m][0][0], &p.tm_z, bar, (kh + m * n_kh) * D + c0, static_cast<int>(s * B));
    };
    auto store_outputs = [&](int64_t r) {  // with the norm (else the consumers store their outputs)
        if (store_out) {
#pragma unroll
            for (int m = 0; m < kHeadsPerKey; ++m)
                tma_store_2d(&p.tm_o, &sm.o[r % NS][m][0][0], (kh + m * n_kh) * D + c0, static_cast<int>(r * B));
            bulk_commit_group();
        }
    };
    int64_t issued = nst < NS ? nst : NS;
    if (lane == 0)
        for (int64_t s = 0; s < issued; ++s) {
            issue(s);
            if (NORM) issue_z(s);
        }
    __syncwarp();  // lanes 1..31 must not spin on a barrier while lane 0 still has copies to issue
    int64_t z_issued = NORM ? issued : 0;
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
                gv = __ldg(gp + t * n_vh + kh + m * n_kh);
                bv = __ldg(betap + t * n_vh + kh + m * n_kh);
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
        // With the norm the consumers write this stage's output tile once 'ready'
        // arrives; it was last read by the TMA store of stage s - NS (the stores
        // committed so far are those of stages <= s - 2) and by the epilogue.
        if (NORM && lane == 0) bulk_wait_group_read<NS - 2>();
        if (NORM && s >= NS) {
            if (!mbar_wait(&sm.normed[buf], static_cast<uint32_t>(((s - NS) / NS) & 1))) {
                ok = false;
                break;
            }
            if (lane == 0) issue_z(s);  // stage s - NS's z tile is read
            z_issued = s + 1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.ready[buf]);
        // Store the outputs of the stage the consumers finished last, then refill its buffer.
        if (s >= 1) {
            const int64_t r = s - 1;
            if (!mbar_wait(&sm.empty[r % NS], static_cast<uint32_t>((r / NS) & 1))) { ok = false; break; }
            if (lane == 0) {
                store_outputs(r);
                if (r + NS < nst) issue(r + NS);
            }
            __syncwarp();
            if (r + NS < nst) issued = r + NS + 1;
        }
    }
    if (ok) {
        const int64_t r = nst - 1;
        if (!mbar_wait(&sm.empty[r % NS], static_cast<uint32_t>((r / NS) & 1)))
            ok = false;
        else if (lane == 0)
            store_outputs(r);
    }
    if (NORM && lane == 0) bulk_wait_group_all();  // every output store has landed before the CTA exits
    __syncwarp();
    if (!ok) {
        // Record the failure, then let every issued copy land before the CTA exits.
        if (lane == 0) report_timeout(status);
        for (int64_t s = landed; s < issued; ++s) mbar_wait(&sm.full[s % NS], static_cast<uint32_t>((s / NS) & 1));
    }
    if (NORM) {
        // z tiles nobody waited for (the norm warps stopped early) land before the CTA exits
        for (int64_t s = (z_issued > NS ? z_issued - NS : 0); s < z_issued; ++s)
            mbar_wait(&sm.zfull[s % NS], static_cast<uint32_t>((s / NS) & 1));
    }
}

// ---------------- consumer warps ----------------
template <int R, bool NORM>
__device__ void consumer_role(const SeqParams& p, SeqSmem& sm, int kh, int c0, int warp, int lane) {
    using Sh = SeqShape<R, NORM>;
    // parameters read once into registers (p is the kernel's parameter block, seen
    // here through a reference; reads of it inside the loop could not be hoisted
    // past the output stores)
    const int64_t T = p.T;
    const int n_kh = p.n_kh;
    const int64_t out_stride = static_cast<int64_t>(p.n_vh) * D;
    float* const state = p.state;
    int* const status = p.status;
    const int64_t nst = (T + B - 1) / B;
    const int colw = lane / Sh::G;
    const int rg = lane % Sh::G;
    const int cl = warp * Sh::CPW + colw;  // column within the CTA
    const int c = c0 + cl;
    // rows of this lane: 4*rg + 4*G*pp + u, pp < R/4, u < 4
    float2 S[kHeadsPerKey][Sh::P4][2];
#pragma unroll
    for (int m = 0; m < kHeadsPerKey; ++m) {
        const float* sh = state + static_cast<int64_t>(kh + m * n_kh) * D * D + c;
#pragma unroll
        for (int pp = 0; pp < Sh::P4; ++pp) {
            const int row = 4 * rg + 4 * Sh::G * pp;
            S[m][pp][0] = make_float2(sh[(row + 0) * D], sh[(row + 1) * D]);
            S[m][pp][1] = make_float2(sh[(row + 2) * D], sh[(row + 3) * D]);
        }
    }

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
    // Output destination of token tt of a stage (lanes rg < 3): with the norm the
    // shared output tile (indexing the shared array itself keeps the store a
    // shared-memory store that the compiler can tell apart from the operand
    // loads), else out.
    float* const o_all = &sm.o[0][0][0][0];
    float* const out_col = NORM ? nullptr : p.out + static_cast<int64_t>(kh + (rg < kHeadsPerKey ? rg : 0) * n_kh) * D + c;
    const int my_m = rg < kHeadsPerKey ? rg : 0;
    // One token: both column sums from one pass over the state (12 independent
    // packed accumulator chains), the k-sum reduction first (it gates delta), the
    // decay product a*S formed while the shuffles are in flight, then the update;
    // the q-sum reduction and the output come last, off the state's critical path.
    auto token = [&](const Ops& o, int64_t dst) {
        float2 ak[kHeadsPerKey][2], aq[kHeadsPerKey][2];
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m) ak[m][0] = ak[m][1] = aq[m][0] = aq[m][1] = make_float2(0.f, 0.f);
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
        if (rg < kHeadsPerKey) {
            if (NORM)
                o_all[dst] = o_mine;
            else
                out_col[dst * out_stride] = o_mine;
        }
    };

    bool ok = true;
    for (int64_t s = 0; s < nst; ++s) {
        const int buf = static_cast<int>(s % NS);
        const uint32_t par = static_cast<uint32_t>((s / NS) & 1);
        if (!mbar_wait(&sm.full[buf], par) || !mbar_wait(&sm.ready[buf], par)) {
            if (lane == 0) report_timeout(status);
            ok = false;
            break;
        }
        const Stage& st = sm.st[buf];
        // destination of token tt's output: o_base + tt * o_step
        const int64_t o_base = NORM ? ((buf * kHeadsPerKey + my_m) * B) * NCOL + cl : s * B;
        const int64_t o_step = NORM ? NCOL : 1;
        const int64_t rem = T - s * B;
        const int nt = rem < B ? static_cast<int>(rem) : B;
        Ops x0, x1;
        load(x0, st, 0);
        int tt = 0;
#pragma unroll 1
        for (; tt + 1 < nt; tt += 2) {
            load(x1, st, tt + 1);
            token(x0, o_base + tt * o_step);
            if (tt + 2 < nt) load(x0, st, tt + 2);
            token(x1, o_base + (tt + 1) * o_step);
        }
        if (tt < nt) token(x0, o_base + tt * o_step);
        // The stage's inputs are read and its outputs written: hand it back (with the
        // norm, after making the output tile visible to the TMA store's async proxy).
        if (NORM) fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[buf]);
    }
    if (!ok) return;  // the state is left as it was

#pragma unroll
    for (int m = 0; m < kHeadsPerKey; ++m) {
        float* sh = state + static_cast<int64_t>(kh + m * n_kh) * D * D + c;
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

// ---------------- norm warps ----------------
// Norm warp i of a CTA norms rows 12 i .. 12 i + 11 of every stage ((head, token)
// row m * 16 + tt).  Per stage: wait for the output tile; per row compute the sums
// of squares of the CTA's four 4-column groups (each as gdn_out_norm's lane does
// for its 4 columns) and publish them in global memory at [key head][slot][slice];
// gather all eight slices' once their per-row publication counters show the
// stage; add a row's 32 group sums in the order of gdn_out_norm's xor tree
// (offsets 16, 8, 4, 2, 1); form r and write y for the CTA's 16 columns with the
// row code's expression.  The gather and the norm of a stage run one stage after its
// publication, so the round trip through L2 overlaps the next stage's work.  The
// counters hold (generation << 32 | stages), so a replayed launch never takes an
// earlier launch's values for its own.
__device__ void norm_role(const SeqParams& p, SeqSmem& sm, int kh, int c0, int slice, int wi, int lane,
                          unsigned long long gen) {
    // parameters read once into registers (see consumer_role)
    const int64_t T = p.T;
    const int n_kh = p.n_kh;
    const int64_t y_stride = static_cast<int64_t>(p.n_vh) * D;
    const float eps = p.eps;
    float* const xg = p.xg;
    uint16_t* const yp = p.y;
    int* const status = p.status;
    const int64_t nst = (T + B - 1) / B;
    NormBufs& nb = sm.nb;
    const int row0 = wi * NROWS;
    const int q = lane & 3;  // 4-column group of this lane in the y phase
    const float4 wq = *reinterpret_cast<const float4*>(p.w + c0 + 4 * q);
    // Counters (stages, tagged with the generation): per (key head, slice, row) the
    // stages whose group sums of that row are published, and per (key head, slice,
    // norm warp) the stages that warp has gathered.  A lane releases its own row's
    // counter after storing the row's sums (release orders its own earlier store),
    // and a lane that gathers a row acquires that row's counters itself, so no
    // fence is needed.
    unsigned long long* const pub = p.xflags;
    unsigned long long* const con = p.xflags + static_cast<int64_t>(n_kh) * SLICES * ROWS;
    auto pub_at = [&](int sl, int row) { return pub + (static_cast<int64_t>(kh) * SLICES + sl) * ROWS + row; };
    auto con_at = [&](int sl) { return con + (static_cast<int64_t>(kh) * SLICES + sl) * kNormWarps + wi; };
    auto xslot = [&](int64_t s, int sl) {  // slice sl's group sums of this warp's rows, in the stage's slot
        return reinterpret_cast<float4*>(xg) + ((static_cast<int64_t>(kh) * NSX + s % NSX) * SLICES + sl) * ROWS + row0;
    };
    bool ok = true;
    for (int64_t s = 0; s <= nst; ++s) {
        if (s < nst) {
            const int slot = static_cast<int>(s % NS);
            // (1) the stage's outputs are in the tile
            if (!mbar_wait(&sm.empty[slot], static_cast<uint32_t>((s / NS) & 1))) ok = false;
            if (!__all_sync(0xffffffffu, ok)) break;
            // (2) group sums of row row0 + lane
            float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
            if (lane < NROWS) {
                const int row = row0 + lane;
                const float4* orow = reinterpret_cast<const float4*>(&sm.o[slot][row / B][row % B][0]);
                float g4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 o4 = orow[u];
                    float ss = o4.x * o4.x;
                    ss = fmaf(o4.y, o4.y, ss);
                    ss = fmaf(o4.z, o4.z, ss);
                    ss = fmaf(o4.w, o4.w, ss);
                    g4[u] = ss;
                }
                part = make_float4(g4[0], g4[1], g4[2], g4[3]);
            }
            // (3) the slot is free once the same warp of every slice has gathered stage
            // s - NSX: lanes 0..7 watch one slice each; the warp barrier orders the other
            // lanes' stores after what they saw
            if (s >= NSX && lane < SLICES && !wait_counter(con_at(lane), (gen << 32) | static_cast<uint64_t>(s - NSX + 1)))
                ok = false;
            if (!__all_sync(0xffffffffu, ok)) break;
            __syncwarp();
            // (4) publish: each lane its row's sums, then that row's counter
            if (lane < NROWS) {
                xslot(s, slice)[lane] = part;
                st_release_gpu_u64(pub_at(slice, row0 + lane), (gen << 32) | static_cast<uint64_t>(s + 1));
            }
        }
        if (s == 0) continue;
        const int64_t u = s - 1;  // the stage normed in this iteration
        const int slot = static_cast<int>(u % NS);
        // (5) gather: lane = row row0 + lane; acquire its 8 counters, then load
        if (lane < NROWS) {
            const unsigned long long want = (gen << 32) | static_cast<uint64_t>(u + 1);
#pragma unroll 1
            for (int sl = 0; sl < SLICES && ok; ++sl)
                if (!wait_counter(pub_at(sl, row0 + lane), want)) ok = false;
        }
        if (!__all_sync(0xffffffffu, ok)) break;
        if (lane < NROWS) {
            float g[32];
#pragma unroll
            for (int sl = 0; sl < SLICES; ++sl) {
                const float4 v = __ldcg(xslot(u, sl) + lane);
                g[4 * sl] = v.x;
                g[4 * sl + 1] = v.y;
                g[4 * sl + 2] = v.z;
                g[4 * sl + 3] = v.w;
            }
            // lane 0's view of the xor tree: level 16, 8, 4, 2, 1
#pragma unroll
            for (int j = 0; j < 16; ++j) g[j] = g[j] + g[j + 16];
#pragma unroll
            for (int j = 0; j < 8; ++j) g[j] = g[j] + g[j + 8];
#pragma unroll
            for (int j = 0; j < 4; ++j) g[j] = g[j] + g[j + 4];
#pragma unroll
            for (int j = 0; j < 2; ++j) g[j] = g[j] + g[j + 2];
            const float ss = g[0] + g[1];
            nb.r[wi][lane] = rsqrtf(fmaf(ss, 1.0f / 128.0f, eps));
        }
        // (6) this warp has read stage u's slot (its loads are complete: their values
        // are in r); the warp barrier orders them before lane 0's release
        __syncwarp();
        if (lane == 0) st_release_gpu_u64(con_at(slice), (gen << 32) | static_cast<uint64_t>(u + 1));
        // (7) z landed
        if (!mbar_wait(&sm.zfull[slot], static_cast<uint32_t>((u / NS) & 1))) ok = false;
        if (!__all_sync(0xffffffffu, ok)) break;
        // (8) y of the CTA's columns: lane = 4-column group q of rows row0 + (lane >> 2) + 8 j
#pragma unroll
        for (int j = 0; j < (NROWS + 7) / 8; ++j) {
            const int rl = (lane >> 2) + 8 * j;
            if (rl < NROWS) {
                const int row = row0 + rl;
                const int m = row / B, tt = row % B;
                const int64_t t = u * B + tt;
                if (t < T) {
                    const float4 o4 = *reinterpret_cast<const float4*>(&sm.o[slot][m][tt][4 * q]);
                    const float4 z4 = *reinterpret_cast<const float4*>(&nb.z[slot][m][tt][4 * q]);
                    const float r = nb.r[wi][rl];
                    const __half2 lo =
                        __floats2half2_rn(o4.x * r * wq.x * norm_silu(z4.x), o4.y * r * wq.y * norm_silu(z4.y));
                    const __half2 hi =
                        __floats2half2_rn(o4.z * r * wq.z * norm_silu(z4.z), o4.w * r * wq.w * norm_silu(z4.w));
                    uint2 pkd;
                    pkd.x = *reinterpret_cast<const uint32_t*>(&lo);
                    pkd.y = *reinterpret_cast<const uint32_t*>(&hi);
                    *reinterpret_cast<uint2*>(yp + t * y_stride + static_cast<int64_t>(kh + m * n_kh) * D + c0 +
                                              4 * q) = pkd;
                }
            }
        }
        // (9) done with stage u's output and z tiles
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.normed[slot]);
    }
    if (!ok && lane == 0) report_error(status, kDevErrNormTimeout);
}

template <int R, bool NORM>
__global__ void __launch_bounds__(SeqShape<R, NORM>::THREADS, 1) gdn_seq_kernel(const __grid_constant__ SeqParams p) {
    using Sh = SeqShape<R, NORM>;
    SeqSmem& sm = *aligned_dynamic_smem<SeqSmem, 1024>();
    const int kh = blockIdx.x;
    const int c0 = blockIdx.y * NCOL;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ uint32_t s_gen;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.ready[s], 1);
            mbar_init(&sm.empty[s], Sh::NCW);
            mbar_init(&sm.zfull[s], 1);
            mbar_init(&sm.normed[s], kNormWarps);
        }
        mbar_init_fence();
        // this launch's generation: one more than the last finished launch's
        if (NORM) s_gen = ld_acquire_gpu(p.sync) + 1u;
    }
    __syncthreads();

    if (warp == Sh::PRODUCER)
        producer_role<R, NORM>(p, sm, kh, c0, lane);
    else if (NORM && warp >= Sh::NORM0)
        norm_role(p, sm, kh, c0, blockIdx.y, warp - Sh::NORM0, lane, s_gen);
    else
        consumer_role<R, NORM>(p, sm, kh, c0, warp, lane);
    if (NORM) {
        // the last CTA to finish advances the generation
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            if (atomicAdd(p.sync + 1, 1u) == gridDim.x * gridDim.y - 1) {
                p.sync[1] = 0u;
                st_release_gpu(p.sync, s_gen);
            }
        }
    }
}

template <int R, bool NORM>
cudaError_t launch_seq_t(const SeqParams& p, cudaStream_t s) {
    using Sh = SeqShape<R, NORM>;
    const size_t smem = (NORM ? sizeof(SeqSmem) : offsetof(SeqSmem, o)) + 1024;
    const auto kernel = gdn_seq_kernel<R, NORM>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_kh, SLICES);
    cfg.blockDim = dim3(Sh::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // the fused norm's CTAs wait for each other
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = NORM ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace

int seq_tokens_per_stage() { return B; }
size_t seq_norm_scratch_bytes(int n_kh) {
    // counters first (8-byte aligned), then sync words, then the group sums (16-byte aligned)
    return static_cast<size_t>(seq_norm_counters(n_kh)) * 8 + 16 +
           static_cast<size_t>(n_kh) * NSX * SLICES * ROWS * 16;
}
int seq_norm_counters(int n_kh) { return n_kh * SLICES * (ROWS + kNormWarps); }
int seq_box_cols() { return NCOL; }

cudaError_t launch_seq(const SeqParams& p, int rows_per_thread, cudaStream_t s) {
    const bool norm = p.y != nullptr;
    if (rows_per_thread == 8) return norm ? launch_seq_t<8, true>(p, s) : launch_seq_t<8, false>(p, s);
    return norm ? launch_seq_t<16, true>(p, s) : launch_seq_t<16, false>(p, s);
}

}  // namespace gdn
