// Chunked Gated DeltaNet recurrence with the state in tensor memory (sm_103a).
//
// Same math as gdn_chunk.cu ("#1372 DeltaNet recurrence: STRATA_GDN_CHUNKED=1 - the
// prompt's recurrence in 32-token chunks", section "What it does"); per value head
// and chunk, with gamma the running gate sum inside the chunk and S0 the state
// before it, in transposed form (value columns first):
//     X^T   = S0^T [K; Q]^T                          128 x 64, K = 128 key dims
//     U'^T  = V^T - X_K^T diag(e^gamma)              (epilogue)
//     D^T   = U'^T T'^T                               128 x 32, K = 32
//     O^T   = X_Q^T diag(e^gamma) + D^T P^T           128 x 32, K = 32 (+ epilogue)
//     S^T   = e^gamma_last S0^T + D'^T K,  D' = diag(e^(gamma_last - gamma)) D
//                                                     128 x 128, K = 32
// One CTA per value head keeps S^T in tensor memory (value column j = lane j, key
// dim i = column i) as the FP32 accumulator of the update.  Every product is a
// tcgen05.mma with M = 128 over those lanes: its A operand (S0^T, U'^T, D^T, D'^T)
// comes from tensor memory, its B operand ([K; Q], T', P, K^T) from shared memory,
// where the prep's swizzled tiles land by bulk copies.  Products are split TF32:
// x = hi + lo, and a.b is accumulated in FP32 as hi_a hi_b in one accumulator and
// hi_a lo_b + lo_a hi_b in another (joined in the epilogue); plain TF32 would miss
// the 2e-6 tolerance against FP64 by three orders of magnitude.  The tensor cores
// read an FP32 operand as TF32 by dropping its low 13 bits (measured on GB300 for
// both operand sources), so the state's hi part is the accumulator itself and
// only its lo part, x - hi rounded to TF32, is written out; the B operands and the
// chunk's intermediates are split with hi rounded to nearest.  Where one MMA can
// take both, hi_a (hi_b, lo_b) is a single MMA over the stacked [hi; lo] operand.
// The gate scalings act in the epilogues, so one key head's tiles serve its three
// value heads unchanged.
//
// Warp roles (352 threads): warps 0-7 move values between tensor memory and
// registers (warp w: lanes 32 (w % 4) .. +31, half w / 4 of each step's columns);
// lane 0 of warp 8 issues the copies; lane 0 of warp 9 issues the MMAs but P D, which
// lane 0 of warp 10 issues (a tcgen05.mma blocks its thread while the tensor pipe's
// queue is full, and P D must not hold up the MMAs the chunk waits for).  Per chunk:
//   MMA: X's hi.(hi, lo) terms from the state as it stands, while the epilogue
//   writes the state's lo part (in two halves); MMA: X's lo.hi terms, then the
//   chunk before's P D -> epilogue: U', then e^gamma_last S in place -> MMA: D ->
//   epilogue: D', then D -> MMA: the state update, while the epilogue writes the
//   chunk before's O to out.
// For gdn_recurrence_norm a second instance of the kernel (NORM) also writes the
// gated RMSNorm of the output to y from the output epilogue: a scan CTA holds whole
// 128-column rows of its value head, so each row's sum of squares is formed inside
// the CTA, in the order of gdn_out_norm's warp (norm lane l = j / 4 sums the squares
// of columns 4l .. 4l+3 in turn, then the 32 lanes' sums meet in an xor butterfly),
// and y has that kernel's bits; z arrives by TMA like v.  The FP32 output is then
// optional.  To make room for z, that instance keeps v in one buffer, and its
// epilogue loop is rotated: a chunk's O is read during the update, the next chunk's
// state split follows, and the norm of those rows runs while the X product does.
// The CTAs before the scan CTAs run the prep of the same super-block (one task per
// (chunk, key head), in chunk order) and publish a flag per task, as the one-launch
// kernel of gdn_chunk.cu does; the cooperative launch keeps every CTA resident.
#include "gdn_chunk_prep.cuh"
#include "gdn_norm_row.cuh"

namespace gdn {
namespace {

constexpr int TM_THREADS = 352;
constexpr int kEpiWarps = 8;
constexpr int kProducerWarp = 8, kMmaWarp = 9, kOWarp = 10;
constexpr uint32_t TMEM_COLS = 512;

// tensor-memory columns
constexpr uint32_t TM_S = 0;    // S^T, the update's accumulator (128 key dims); also X's TF32 hi operand
constexpr uint32_t TM_L = 128;  // S^T's TF32 lo part; once X is done: U' hi [0,32), U' lo [32,64); the D
                                // product [64,128) (hi.hi [64,96), cross terms [96,128)), then D' hi
                                // [64,96), D' lo [96,128)
constexpr uint32_t TM_X = 256;  // chunk parity p: 128 columns at TM_X + 128 p: X's hi.hi terms [0,64)
                                // (k tokens, then q) and cross terms [64,128); then O's accumulators,
                                // e^gamma X_Q [0,32) and zeros [32,64), and D hi [64,96), D lo [96,128)

// shared memory (bytes from a 1024-aligned base); the instance with the norm keeps v
// in one buffer and adds z's buffer and the norm's exchange space
template <bool NORM>
struct Smem {
    static constexpr uint32_t KQ = 0;          // [2 buffers][4 key-dim blocks][128 rows: hi 64, lo 64][128 B]
    static constexpr uint32_t KT = 131072;     // K^T hi 16 KB | lo 16 KB: [128 key dims][128 B]
    static constexpr uint32_t TP = 163840;     // T' hi 4 KB | lo 4 KB: [32 rows][128 B] (one 64-row operand [hi; lo])
    static constexpr uint32_t P = 172032;      // [2 buffers][P hi 4 KB | lo 4 KB], the same
    static constexpr uint32_t V = 188416;      // [2 buffers (NORM: 1)][32 tokens][128 columns] floats (TMA)
    static constexpr uint32_t Z = V + 16384;   // (NORM) [32 tokens][128 columns] floats of z (TMA)
    static constexpr uint32_t G = V + 32768;   // [2 buffers][e^gamma 32 | e^(gamma_last - gamma) 32] floats
    static constexpr uint32_t NP = G + 512;    // (NORM) [2 halves][16 tokens][32 norm lanes, row stride 40]
    static constexpr uint32_t NR = NP + (NORM ? 5120 : 0);   // (NORM) [2 halves][16 tokens] 1 / rms
    static constexpr uint32_t BAR = NR + (NORM ? 128 : 0);   // mbarriers, the tensor-memory address, the abort word
    static constexpr uint32_t TOTAL = BAR + (NORM ? 512 : 256);
};
// (the instance without the norm is kept at about 218 KB, so that a 128-thread CTA of
// the norm kernel launched on another stream still fits on an SM beside its CTA)
enum {
    B_KQ0, B_KQ1, B_P0, B_P1, B_VG0, B_VG1, B_TP, B_KT,  // copies landed
    B_MX0, B_MX1, B_MD, B_MS, B_MO, B_MO0, B_MO1,        // MMA groups done (tcgen05.commit; B_MO0 / B_MO1:
    B_FIN, B_FINO,                                       //   P D again, per P buffer)
    B_ESA, B_ESB, B_EU, B_ED, B_EDO0, B_EDO1, B_EO,      // epilogue steps done (one arrival per epilogue warp)
    B_VF0, B_VF1,                                        // v / gates buffer read for the last time (the same)
    NBAR_PLAIN,
    B_Z = NBAR_PLAIN,                                    // (NORM) z copy landed
    B_ZF,                                                // (NORM) z read (one arrival per epilogue warp)
    B_NP0, B_NP1, B_NR0, B_NR1,                          // (NORM) norm exchange, per half (one arrival per warp of it)
    NBAR_NORM
};
static_assert(NBAR_PLAIN * 8 + 8 <= 256 && NBAR_NORM * 8 + 8 <= 512, "barrier space");
constexpr uint32_t TX_KQ = 2 * 2 * C * D * 4, TX_TP = 2 * C * C * 4, TX_P = 2 * C * C * 4, TX_KT = 2 * D * C * 4;
constexpr uint32_t TX_VG = C * D * 4 + 2 * C * 4, TX_Z = C * D * 4;

constexpr uint32_t IDESC_N32 = umma_idesc_tf32(128, 32);
constexpr uint32_t IDESC_N64 = umma_idesc_tf32(128, 64);
constexpr uint32_t IDESC_N128 = umma_idesc_tf32(128, 128);

struct TmemShared {
    uint64_t* bar;
    volatile int* abort_flag;  // set once a wait gave up: every later wait returns at once
    int* status;
};

// Waits for the phase of `bar` with the given parity.  Returns false when the
// wait gives up (poll limit: the abort word is set and the status reported) or
// when another role already gave up.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool wait_ab(const TmemShared& sh, int b, uint32_t parity) {
    if (mbar_test(&sh.bar[b], parity)) return true;  // the common case: no suspend
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(&sh.bar[b], parity)) return true;
        if ((i & 255u) == 255u) {
            if (*sh.abort_flag) return false;
            if (i >= kWaitPolls) {
                *sh.abort_flag = 1;
                report_timeout(sh.status);
                return false;
            }
        }
    }
}

// The same for a whole warp.  Every lane waits: only a thread that observes the
// phase completing is guaranteed to see the copies' data (lanes that learnt of it
// from another lane by a shuffle read stale shared memory on GB300).  The warp
// agrees on the outcome, so its .sync.aligned tensor-memory accesses stay converged.
__device__ __forceinline__ bool warp_wait_ab(const TmemShared& sh, int b, uint32_t parity) {
    const bool ok = wait_ab(sh, b, parity);
    return __all_sync(0xffffffffu, ok) != 0;
}

// Tell the MMA issuer that this warp's tensor-memory stores have landed.
__device__ __forceinline__ void epi_arrive(const TmemShared& sh, int b) {
    tmem_wait_st();
    tc_fence_before_sync();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.bar[b]);
}

__device__ __forceinline__ float rna_tf32(const float x) {
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}
// TF32 hi (to nearest, ties away: integer operations on the bits) and lo = x - hi
// (exact; one packed FMA per pair).
__device__ __forceinline__ void split_pair(const float x0, const float x1, float& h0, float& h1, float& l0, float& l1) {
    h0 = rna_tf32(x0);
    h1 = rna_tf32(x1);
    const float2 l = ffma2(make_float2(h0, h1), make_float2(-1.f, -1.f), make_float2(x0, x1));
    l0 = l.x;
    l1 = l.y;
}
__device__ __forceinline__ void split16(const float (&x)[16], float (&hi)[16], float (&lo)[16]) {
#pragma unroll
    for (int i = 0; i < 16; i += 2) split_pair(x[i], x[i + 1], hi[i], hi[i + 1], lo[i], lo[i + 1]);
}
// The state's lo part: x - (x with its low 13 bits cleared, which the tensor cores
// take as its TF32 hi), rounded to TF32.
__device__ __forceinline__ void state_lo32(const float (&s)[32], float (&lo)[32]) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float t0 = __uint_as_float(__float_as_uint(s[i]) & 0xFFFFE000u);
        const float t1 = __uint_as_float(__float_as_uint(s[i + 1]) & 0xFFFFE000u);
        const float2 d = ffma2(make_float2(t0, t1), make_float2(-1.f, -1.f), make_float2(s[i], s[i + 1]));
        lo[i] = rna_tf32(d.x);
        lo[i + 1] = rna_tf32(d.y);
    }
}

// ---- the scan of value head vh ----
template <bool NORM>
__device__ __forceinline__ void tmem_scan(const ChunkTmemParams& p, unsigned char* sm, const int vh,
                                          const uint32_t gen) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_kh = p.prep.n_kh, n_vh = p.prep.n_vh;
    const int kh = vh % n_kh;
    const int n_tokens = p.prep.n_tokens;
    const int nch = (n_tokens + C - 1) / C;
    using L = Smem<NORM>;
    constexpr int NBAR = NORM ? NBAR_NORM : NBAR_PLAIN;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BAR + NBAR * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::BAR + NBAR * 8 + 4);
    const TmemShared sh{bar, abort_flag, p.status};

    if (tid == 0) {
        for (int b = 0; b < B_ESA; ++b) mbar_init(&bar[b], 1);
        for (int b = B_ESA; b < NBAR_PLAIN; ++b) mbar_init(&bar[b], kEpiWarps);
        if constexpr (NORM) {
            mbar_init(&bar[B_Z], 1);
            mbar_init(&bar[B_ZF], kEpiWarps);
            for (int b = B_NP0; b <= B_NR1; ++b) mbar_init(&bar[b], kEpiWarps / 2);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == kMmaWarp) tmem_alloc(tslot, TMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tbase = *tslot;

    if (warp == kProducerWarp) {
        // ---------------- copies ----------------
        // Each buffer is refilled once the MMA group or epilogue step that last reads it
        // has finished.  The order below also keeps every wait at most one phase behind
        // its barrier: the phase after the awaited one depends on a copy issued later in
        // the same iteration (or, for z, in the next one).
        if (lane == 0) {
            int armed[B_KT + 1];  // last chunk whose copies each load barrier was armed for (-1: none)
#pragma unroll
            for (int b = 0; b <= B_KT; ++b) armed[b] = -1;
            int armed_z = -1;     // (NORM) the same for z
            float* tiles = p.prep.prep;
            for (int c = 0; c < nch && !*abort_flag; ++c) {
                // the prep task of (c, kh) has published its tiles
                uint32_t seen = 0;
                if (!wait_flag(p.flags + c * n_kh + kh, gen, &seen)) {
                    *abort_flag = 1;
                    report_error(p.status, kDevErrFlagTimeout);
                    p.sync[2] = static_cast<uint32_t>(c * n_kh + kh);
                    p.sync[3] = seen;
                    p.sync[4] = gen;
                    break;
                }
                fence_proxy_async_global();
                const float* kt = key_tiles(tiles, n_kh, c, kh);
                const float* ht = head_tiles(tiles, n_kh, n_vh, c, vh);
                const int s = c & 1;
                const uint32_t par2 = static_cast<uint32_t>(((c - 2) >> 1) & 1);
                const int row = static_cast<int>(p.prep.t_begin + static_cast<int64_t>(c) * C);
                // v and the gates of chunk c (v: slot s of two, or the one buffer)
                auto copy_vg = [&]() {
                    mbar_arrive_expect_tx(&bar[B_VG0 + s], TX_VG);
                    tma_load_2d(sm + L::V + (NORM ? 0 : s * (C * D * 4)), &p.tm_v, &bar[B_VG0 + s], vh * D, row);
                    bulk_load(sm + L::G + s * 256, ht + kTileEG, 2 * C * 4, &bar[B_VG0 + s]);
                    if (s) armed[B_VG1] = c; else armed[B_VG0] = c;
                };
                if constexpr (!NORM) {
                    // the buffer's chunk c-2 has been read for the last time
                    if (c >= 2 && !wait_ab(sh, B_VF0 + s, par2)) break;
                    copy_vg();
                }
                // [K; Q] of chunk c: the buffer's chunk c-2 X product is done
                if (c >= 2 && !wait_ab(sh, B_MX0 + s, par2)) break;
                mbar_arrive_expect_tx(&bar[B_KQ0 + s], TX_KQ);
                bulk_load(sm + L::KQ + s * 65536, kt + kTileKQ, TX_KQ, &bar[B_KQ0 + s]);
                if (s) armed[B_KQ1] = c; else armed[B_KQ0] = c;
                // P of chunk c: the buffer's chunk c-2 P D is done
                if (c >= 2 && !wait_ab(sh, B_MO0 + s, par2)) break;
                mbar_arrive_expect_tx(&bar[B_P0 + s], TX_P);
                bulk_load(sm + L::P + s * TX_P, ht + kTilePH, TX_P, &bar[B_P0 + s]);
                if (s) armed[B_P1] = c; else armed[B_P0] = c;
                if constexpr (NORM) {
                    // one v buffer: chunk c-1's v and gates have been read for the last time
                    // (after [K; Q] and P, which the next MMAs wait for sooner)
                    if (c >= 1 && !wait_ab(sh, B_VF0 + (s ^ 1), static_cast<uint32_t>(((c - 1) >> 1) & 1))) break;
                    copy_vg();
                }
                // T' of chunk c: chunk c-1's D product is done
                if (c >= 1 && !wait_ab(sh, B_MD, static_cast<uint32_t>((c - 1) & 1))) break;
                mbar_arrive_expect_tx(&bar[B_TP], TX_TP);
                bulk_load(sm + L::TP, ht + kTileTPH, TX_TP, &bar[B_TP]);
                armed[B_TP] = c;
                // K^T of chunk c: chunk c-1's update is done
                if (c >= 1 && !wait_ab(sh, B_MS, static_cast<uint32_t>((c - 1) & 1))) break;
                mbar_arrive_expect_tx(&bar[B_KT], TX_KT);
                bulk_load(sm + L::KT, kt + kTileKTH, TX_KT, &bar[B_KT]);
                armed[B_KT] = c;
                if constexpr (NORM) {
                    // z of chunk c-1 (one buffer, needed a chunk later): chunk c-2's z has been read
                    if (c >= 1) {
                        if (c >= 2 && !wait_ab(sh, B_ZF, static_cast<uint32_t>((c - 2) & 1))) break;
                        mbar_arrive_expect_tx(&bar[B_Z], TX_Z);
                        tma_load_2d(sm + L::Z, &p.tm_z, &bar[B_Z], vh * D, row - C);
                        armed_z = c - 1;
                    }
                }
            }
            if constexpr (NORM) {
                // z of the last chunk
                if (!*abort_flag && armed_z == nch - 2 &&
                    (nch < 2 || wait_ab(sh, B_ZF, static_cast<uint32_t>((nch - 2) & 1)))) {
                    mbar_arrive_expect_tx(&bar[B_Z], TX_Z);
                    tma_load_2d(sm + L::Z, &p.tm_z, &bar[B_Z], vh * D,
                                static_cast<int>(p.prep.t_begin + static_cast<int64_t>(nch - 1) * C));
                    armed_z = nch - 1;
                }
            }
            // before the CTA ends: every copy issued has landed (bounded waits; normally
            // these phases completed long ago and the waits return at once)
#pragma unroll
            for (int b = 0; b <= B_KT; ++b) {
                if (armed[b] < 0) continue;
                const bool two = b < B_TP;  // double-buffered: one phase per two chunks
                mbar_wait(&bar[b], static_cast<uint32_t>((two ? armed[b] >> 1 : armed[b]) & 1));
            }
            if (armed_z >= 0) mbar_wait(&bar[B_Z], static_cast<uint32_t>(armed_z & 1));
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---------------- MMAs ----------------
        if (lane == 0) {
            const uint64_t kq_desc = umma_desc_sw128(sm + L::KQ);
            const uint64_t kt_desc = umma_desc_sw128(sm + L::KT);
            const uint64_t tp_desc = umma_desc_sw128(sm + L::TP);
            const uint64_t p_desc = umma_desc_sw128(sm + L::P);
            // descriptor start addresses count 16-byte units: +2 per 8-float k step
            auto kq_b = [&](int c, int ks) {  // [K; Q] block of k step ks: 128 rows [hi; lo]
                return kq_desc + static_cast<uint64_t>(((c & 1) * 65536 + (ks >> 2) * 16384 + (ks & 3) * 32) >> 4);
            };
            bool alive = true;
            for (int c = 0; c < nch && alive; ++c) {
                const uint32_t pp = static_cast<uint32_t>(c & 1);
                const uint32_t tX = tbase + TM_X + 128 * pp;
                alive = false;
                // (for c >= 1 the checks that [K; Q] has landed and that X's buffer is free were
                // made while chunk c-1's update ran, below); the state after chunk c-1 is final
                // (chunk 0: the starting state is in place)
                if (c == 0 && !wait_ab(sh, B_KQ0, 0)) break;
                if (!wait_ab(sh, c == 0 ? B_ESB : B_MS, c == 0 ? 0u : pp ^ 1)) break;
                tc_fence_after_sync();
                // X = S0^T [K; Q]^T, N = 64 tokens (k then q), 16 k steps of 8 key dims:
                // hi . [hi; lo] (N = 128) from the state itself
#pragma unroll
                for (int ks = 0; ks < D / 8; ++ks)
                    umma_tf32_ts(tX, tbase + TM_S + 8 * ks, kq_b(c, ks), IDESC_N128, ks > 0);
                // lo . hi (N = 64, onto the cross terms): key dims 0-31 and 64-95 first
                if (!wait_ab(sh, B_ESA, pp)) break;
                tc_fence_after_sync();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int ks = (i & 3) + 8 * (i >> 2);  // 0-3, 8-11
                    umma_tf32_ts(tX + 64, tbase + TM_L + 8 * ks, kq_b(c, ks), IDESC_N64, true);
                }
                if (!wait_ab(sh, B_ESB, pp)) break;
                tc_fence_after_sync();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int ks = 4 + (i & 3) + 8 * (i >> 2);  // 4-7, 12-15
                    umma_tf32_ts(tX + 64, tbase + TM_L + 8 * ks, kq_b(c, ks), IDESC_N64, true);
                }
                umma_commit(&bar[B_MX0 + (c & 1)]);
                // D^T = U'^T T'^T (K = 32 tokens): per k step U' hi . [T' hi; T' lo] (N = 64: hi.hi
                // terms to columns 64-95 of L, hi.lo to 96-127) and U' lo . T' hi (N = 32, to 96-127)
                if (!wait_ab(sh, B_TP, pp)) break;
                if (!wait_ab(sh, B_EU, pp)) break;
                tc_fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks) {
                    const uint64_t b = tp_desc + static_cast<uint64_t>((ks * 32) >> 4);
                    umma_tf32_ts(tbase + TM_L + 64, tbase + TM_L + 8 * ks, b, IDESC_N64, ks > 0);
                    umma_tf32_ts(tbase + TM_L + 96, tbase + TM_L + 32 + 8 * ks, b, IDESC_N32, true);
                }
                umma_commit(&bar[B_MD]);
                // S^T += D'^T K (N = 128 key dims; the accumulator holds e^gamma_last S0^T)
                if (!wait_ab(sh, B_KT, pp)) break;
                if (!wait_ab(sh, B_ED, pp)) break;
                tc_fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks) {
                    const uint64_t bh = kt_desc + static_cast<uint64_t>((ks * 32) >> 4);
                    const uint64_t bl = bh + (16384 >> 4);
                    umma_tf32_ts(tbase + TM_S, tbase + TM_L + 64 + 8 * ks, bl, IDESC_N128, true);
                    umma_tf32_ts(tbase + TM_S, tbase + TM_L + 96 + 8 * ks, bh, IDESC_N128, true);
                }
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks)
                    umma_tf32_ts(tbase + TM_S, tbase + TM_L + 64 + 8 * ks, kt_desc + static_cast<uint64_t>((ks * 32) >> 4),
                                 IDESC_N128, true);
                umma_commit(&bar[B_MS]);
                // while the update runs: chunk c+1's [K; Q] has landed and its X buffer is free
                // (chunk c-1's O is out)
                if (c + 1 < nch) {
                    if (!wait_ab(sh, B_KQ0 + ((c + 1) & 1), static_cast<uint32_t>(((c + 1) >> 1) & 1))) break;
                    if (c >= 1 && !wait_ab(sh, B_EO, pp ^ 1)) break;
                }
                alive = true;
            }
            (void)alive;
            // every MMA issued has completed before the tensor memory is freed
            umma_commit(&bar[B_FIN]);
            mbar_wait(&bar[B_FIN], 0);
        }
        __syncwarp();
    } else if (warp == kOWarp) {
        // ---------------- P D ----------------
        // P D of chunk c, once its D and O's accumulators are in place and its P has landed,
        // and (but for the last chunk) after chunk c+1's X product, so it fills the tensor
        // pipe while the epilogue forms U': per k step D hi . [P hi; P lo] (N = 64: hi.hi
        // onto e^gamma X_Q, hi.lo onto the zeros) and D lo . P hi (N = 32, onto the second
        // half).  Every barrier awaited here is one of a pair used by alternate chunks, whose
        // next phase needs this chunk's P D first.
        if (lane == 0) {
            const uint64_t p_desc = umma_desc_sw128(sm + L::P);
            for (int c = 0; c < nch; ++c) {
                const uint32_t par = static_cast<uint32_t>((c >> 1) & 1);
                if (!wait_ab(sh, B_EDO0 + (c & 1), par)) break;
                if (!wait_ab(sh, B_P0 + (c & 1), par)) break;
                if (c + 1 < nch && !wait_ab(sh, B_MX0 + ((c + 1) & 1), static_cast<uint32_t>(((c + 1) >> 1) & 1))) break;
                tc_fence_after_sync();
                const uint32_t tXc = tbase + TM_X + 128 * static_cast<uint32_t>(c & 1);
                const uint64_t pb = p_desc + static_cast<uint64_t>(((c & 1) * TX_P) >> 4);
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks) {
                    const uint64_t b = pb + static_cast<uint64_t>((ks * 32) >> 4);
                    umma_tf32_ts(tXc, tXc + 64 + 8 * ks, b, IDESC_N64, true);
                    umma_tf32_ts(tXc + 32, tXc + 96 + 8 * ks, b, IDESC_N32, true);
                }
                umma_commit(&bar[B_MO]);
                umma_commit(&bar[B_MO0 + (c & 1)]);
                // every copy of chunk c has landed: P (awaited above), V and the gates (U' read
                // them before D's epilogue), T' (the D product), [K; Q] and K^T (chunk c+1's X
                // product follows chunk c's update, which follows chunk c's X): the chunk's ring
                // slot is free as far as this value head goes (the last chunk's is not needed)
                if (c + 1 < nch)
                    st_release_gpu_u64(p.ring + (c % kTileRing) * n_vh + vh,
                                       (static_cast<unsigned long long>(gen) << 32) | static_cast<uint32_t>(c));
            }
            umma_commit(&bar[B_FINO]);
            mbar_wait(&bar[B_FINO], 0);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue warps 0-7 ----------------
        const int q = warp & 3, hc = warp >> 2;
        const int j = 32 * q + lane;                        // value column = tensor-memory lane
        const uint32_t tl = tbase + (static_cast<uint32_t>(32 * q) << 16);  // this warp's lanes
        const float* Vb = reinterpret_cast<const float*>(sm + L::V);
        const float* Gb = reinterpret_cast<const float*>(sm + L::G);
        float* state = p.state + static_cast<int64_t>(vh) * D * D;
        bool ok = true;
        // (NORM) the exchange space of this warp's half, z and w of column j
        constexpr int NPS = 40;  // row stride of NP (floats): the row sums' loads hit 32 banks
        float* NP = reinterpret_cast<float*>(sm + L::NP) + hc * (16 * NPS);
        float* NR = reinterpret_cast<float*>(sm + L::NR) + hc * 16;
        const float* Zs = reinterpret_cast<const float*>(sm + L::Z);
        const float wj = NORM ? __ldg(p.w + j) : 0.f;

        // O of chunk cc (its two accumulators) -> out; with `arrive`, X's buffer is released
        // (B_EO) as soon as the values are in registers, before the stores
        auto o_out = [&](int cc, bool arrive) {
            const uint32_t tX = tl + TM_X + 128 * static_cast<uint32_t>(cc & 1);
            float a[16], b2[16];
            tmem_ld16x2(tX + 16 * hc, tX + 32 + 16 * hc, a, b2);
            if (arrive) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[B_EO]);
            }
            const int nt = min(C, n_tokens - cc * C);
            float* o = p.out + ((p.prep.t_begin + static_cast<int64_t>(cc) * C) * n_vh + vh) * D + j;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int t = 16 * hc + i;
                if (t < nt) o[static_cast<int64_t>(t) * n_vh * D] = a[i] + b2[i];
            }
        };
        // (NORM) The same in two steps.  o_read: O of chunk cc -> a (and out, if given);
        // o_norm, once the next chunk's state split is out of the way: the gated RMSNorm of
        // those rows -> y, with gdn_out_norm's arithmetic: norm lane l = j / 4 sums the
        // squares of columns 4l .. 4l+3 in turn (lanes 4l .. 4l+3 of this warp), the 32 norm
        // lanes' sums of a row meet in an xor butterfly (16, 8, 4, 2, 1) over shared memory,
        // and y = fp16(o r w silu(z)).  o_norm returns false if a wait gave up.
        auto o_read = [&](int cc, bool arrive, float (&a)[16]) {
            const uint32_t tX = tl + TM_X + 128 * static_cast<uint32_t>(cc & 1);
            float b2[16];
            tmem_ld16x2(tX + 16 * hc, tX + 32 + 16 * hc, a, b2);
            if (arrive) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[B_EO]);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) a[i] += b2[i];
            if (p.out) {
                const int nt = min(C, n_tokens - cc * C);
                float* o = p.out + ((p.prep.t_begin + static_cast<int64_t>(cc) * C) * n_vh + vh) * D + j;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int t = 16 * hc + i;
                    if (t < nt) o[static_cast<int64_t>(t) * n_vh * D] = a[i];
                }
            }
        };
        // silu(z) of this lane's 16 rows of chunk cc (waits for z; its buffer is then free)
        auto z_silu = [&](int cc, float (&sz)[16]) {
            if (!warp_wait_ab(sh, B_Z, static_cast<uint32_t>(cc & 1))) return false;
#pragma unroll
            for (int i = 0; i < 16; ++i) sz[i] = Zs[(16 * hc + i) * D + j];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_ZF]);  // z of chunk cc is read
#pragma unroll
            for (int i = 0; i < 16; ++i) sz[i] = norm_silu(sz[i]);
            return true;
        };
        auto o_norm = [&](int cc, const float (&a)[16], const float (&sz)[16]) {
            const uint32_t par = static_cast<uint32_t>(cc & 1);
            const int nt = min(C, n_tokens - cc * C);
            // Each quad of lanes holds one norm lane's four columns.  Per group of 4 rows the
            // quad transposes its 4 x 4 values (lane k of the quad gathers the four columns of
            // row 4g + k), so each lane sums the squares of one row in column order.
            const int k = lane & 3, quad = lane & ~3;
            auto pick = [](int i, float v0, float v1, float v2, float v3) {  // v_i, branch-free
                const float lo = (i & 1) ? v1 : v0, hi = (i & 1) ? v3 : v2;
                return (i & 2) ? hi : lo;
            };
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float v0 = a[4 * g], v1 = a[4 * g + 1], v2 = a[4 * g + 2], v3 = a[4 * g + 3];
                float x[4];  // x[r]: column (k + r) & 3 of row 4g + k
                x[0] = pick(k, v0, v1, v2, v3);
#pragma unroll
                for (int r = 1; r < 4; ++r)
                    x[r] = __shfl_sync(0xffffffffu, pick((k - r) & 3, v0, v1, v2, v3), quad | ((k + r) & 3));
                const float c0 = pick((0 - k) & 3, x[0], x[1], x[2], x[3]);
                const float c1 = pick((1 - k) & 3, x[0], x[1], x[2], x[3]);
                const float c2 = pick((2 - k) & 3, x[0], x[1], x[2], x[3]);
                const float c3 = pick((3 - k) & 3, x[0], x[1], x[2], x[3]);
                float ss = c0 * c0;
                ss = fmaf(c1, c1, ss);
                ss = fmaf(c2, c2, ss);
                ss = fmaf(c3, c3, ss);
                NP[(4 * g + k) * NPS + 8 * q + (lane >> 2)] = ss;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_NP0 + hc]);
            if (!warp_wait_ab(sh, B_NP0 + hc, par)) return false;
            // this warp's 4 of the half's 16 rows, 8 lanes a row: lane 8u + m adds norm lanes
            // m, m + 16 and m + 8, m + 24 of row 4q + u, then those two sums, as the xor
            // butterfly's levels 16 and 8 do; levels 4, 2, 1 are shuffles among the 8 lanes
            {
                const int m = lane & 7, row = 4 * q + (lane >> 3);
                const float* src = NP + row * NPS;
                float v = (src[m] + src[m + 16]) + (src[m + 8] + src[m + 24]);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                if (m == 0) NR[row] = rsqrtf(fmaf(v, 1.0f / 128.0f, p.eps));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_NR0 + hc]);
            if (!warp_wait_ab(sh, B_NR0 + hc, par)) return false;
            float r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = NR[i];
            unsigned short yv[16];
#pragma unroll
            for (int i = 0; i < 16; i += 2) {  // two rows per conversion (each rounded to nearest)
                const __half2 h2 = __floats2half2_rn(a[i] * r[i] * wj * sz[i], a[i + 1] * r[i + 1] * wj * sz[i + 1]);
                yv[i] = __half_as_ushort(__low2half(h2));
                yv[i + 1] = __half_as_ushort(__high2half(h2));
            }
            uint16_t* yo = p.y + ((p.prep.t_begin + static_cast<int64_t>(cc) * C) * n_vh + vh) * D + j;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int t = 16 * hc + i;
                if (t < nt) yo[static_cast<int64_t>(t) * n_vh * D] = yv[i];
            }
            return true;
        };
        // the lo part of the state after chunk cc (cc >= 0), in two halves
        auto split_state = [&](int cc) {
            if (!warp_wait_ab(sh, B_MS, static_cast<uint32_t>(cc & 1))) return false;
            tc_fence_after_sync();
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                float s[32], lo[32];
                tmem_ld32(tl + TM_S + 64 * hc + 32 * b, s);
                state_lo32(s, lo);
                tmem_st32(tl + TM_L + 64 * hc + 32 * b, lo);
                epi_arrive(sh, b ? B_ESB : B_ESA);
            }
            return true;
        };

        // the starting state and its lo part (key dims 64 hc + 32 b .. +31)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            float s[32], lo[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) s[i] = state[static_cast<int64_t>(64 * hc + 32 * b + i) * D + j];
            state_lo32(s, lo);
            tmem_st32(tl + TM_S + 64 * hc + 32 * b, s);
            tmem_st32(tl + TM_L + 64 * hc + 32 * b, lo);
            epi_arrive(sh, b ? B_ESB : B_ESA);
        }
        for (int c = 0; c < nch && ok; ++c) {
            const uint32_t pp = static_cast<uint32_t>(c & 1);
            const uint32_t tX = tl + TM_X + 128 * pp;
            const float* V = Vb + (NORM ? 0 : (c & 1) * (C * D));
            const float* eg = Gb + (c & 1) * 64;
            const float* er = eg + C;
            if (!NORM && c >= 1) {
                // the lo part of the state after chunk c-1, in two halves
                if (!(ok = warp_wait_ab(sh, B_MS, pp ^ 1))) break;
                tc_fence_after_sync();
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    float s[32], lo[32];
                    tmem_ld32(tl + TM_S + 64 * hc + 32 * b, s);
                    state_lo32(s, lo);
                    tmem_st32(tl + TM_L + 64 * hc + 32 * b, lo);
                    epi_arrive(sh, b ? B_ESB : B_ESA);
                }
            }

            // U' = V - e^gamma X_K (tokens 16 hc .. +15), split -> U' hi / lo; e^gamma X_Q and
            // zeros, the start of O's two accumulators, in X's place
            if (!(ok = warp_wait_ab(sh, B_VG0 + (c & 1), static_cast<uint32_t>((c >> 1) & 1)))) break;
            float vv[16], ev[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                vv[i] = V[(16 * hc + i) * D + j];
                ev[i] = eg[16 * hc + i];
            }
            const float el = eg[C - 1];
            if (!(ok = warp_wait_ab(sh, B_MX0 + (c & 1), static_cast<uint32_t>((c >> 1) & 1)))) break;
            tc_fence_after_sync();
            {
                float xk[16], ck[16], h[16], l[16];
                tmem_ld16x2(tX + 16 * hc, tX + 64 + 16 * hc, xk, ck);
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const float2 k2 = make_float2(xk[i] + ck[i], xk[i + 1] + ck[i + 1]);
                    const float2 u = ffma2(make_float2(-ev[i], -ev[i + 1]), k2, make_float2(vv[i], vv[i + 1]));
                    xk[i] = u.x;
                    xk[i + 1] = u.y;
                }
                split16(xk, h, l);
                tmem_st16(tl + TM_L + 16 * hc, h);
                tmem_st16(tl + TM_L + 32 + 16 * hc, l);
                epi_arrive(sh, B_EU);
                // O's accumulators (next needed by P D, after the D step below): e^gamma X_Q, zeros
                float xq[16], cq[16];
                tmem_ld16x2(tX + 32 + 16 * hc, tX + 96 + 16 * hc, xq, cq);
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const float2 o = fmul2(make_float2(ev[i], ev[i + 1]), make_float2(xq[i] + cq[i], xq[i + 1] + cq[i + 1]));
                    xq[i] = o.x;
                    xq[i + 1] = o.y;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) l[i] = 0.f;
                tmem_st16(tX + 16 * hc, xq);
                tmem_st16(tX + 32 + 16 * hc, l);
            }
            // the update's accumulator: S0 -> e^gamma_last S0 (X has read S0)
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                float s[32];
                tmem_ld32(tl + TM_S + 64 * hc + 32 * b, s);
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float2 e = fmul2(make_float2(s[i], s[i + 1]), make_float2(el, el));
                    s[i] = e.x;
                    s[i + 1] = e.y;
                }
                tmem_st32(tl + TM_S + 64 * hc + 32 * b, s);
            }
            // D (its two accumulators) -> D hi / lo (for P D), D' = e^(gamma_last - gamma) D -> hi / lo
            float rv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) rv[i] = er[16 * hc + i];
            if (!(ok = warp_wait_ab(sh, B_MD, pp))) break;
            tc_fence_after_sync();
            {
                float d[16], x[16], e[16], h[16], l[16];
                tmem_ld16x2(tl + TM_L + 64 + 16 * hc, tl + TM_L + 96 + 16 * hc, d, x);
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    d[i] += x[i];
                    d[i + 1] += x[i + 1];
                    const float2 f = fmul2(make_float2(d[i], d[i + 1]), make_float2(rv[i], rv[i + 1]));
                    e[i] = f.x;
                    e[i + 1] = f.y;
                }
                // D' first (the update waits for it), then D (for P D)
                split16(e, h, l);
                tmem_st16(tl + TM_L + 64 + 16 * hc, h);
                tmem_st16(tl + TM_L + 96 + 16 * hc, l);
                epi_arrive(sh, B_ED);
                if (lane == 0) mbar_arrive(&bar[B_VF0 + (c & 1)]);  // chunk c's v and gates are read
                split16(d, h, l);
                tmem_st16(tX + 64 + 16 * hc, h);
                tmem_st16(tX + 96 + 16 * hc, l);
                epi_arrive(sh, B_EDO0 + (c & 1));
            }
            // O of chunk c-1, while the tensor pipe runs the update
            if constexpr (!NORM) {
                if (c >= 1) {
                    if (!(ok = warp_wait_ab(sh, B_MO, pp ^ 1))) break;
                    tc_fence_after_sync();
                    o_out(c - 1, true);
                }
            } else {
                // (NORM) O of chunk c-1 into registers while the update runs, then the next
                // chunk's state split (the X product waits for it), then the norm of those
                // rows while X runs
                float a[16], sz[16];
                if (c >= 1) {
                    if (!(ok = warp_wait_ab(sh, B_MO, pp ^ 1))) break;
                    tc_fence_after_sync();
                    o_read(c - 1, true, a);
                    if (!(ok = z_silu(c - 1, sz))) break;
                }
                if (c + 1 < nch && !(ok = split_state(c))) break;
                if (c >= 1 && !(ok = o_norm(c - 1, a, sz))) break;
            }
        }
        if (ok) {
            // the state after the last chunk, then its outputs
            ok = warp_wait_ab(sh, B_MS, static_cast<uint32_t>((nch - 1) & 1));
            if (ok) {
                tc_fence_after_sync();
                float a[32], b2[32];
                tmem_ld32(tl + TM_S + 64 * hc, a);
                tmem_ld32(tl + TM_S + 64 * hc + 32, b2);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    state[static_cast<int64_t>(64 * hc + i) * D + j] = a[i];
                    state[static_cast<int64_t>(64 * hc + 32 + i) * D + j] = b2[i];
                }
                ok = warp_wait_ab(sh, B_MO, static_cast<uint32_t>((nch - 1) & 1));
            }
            if (ok) {
                tc_fence_after_sync();
                if constexpr (NORM) {
                    float a[16], sz[16];
                    o_read(nch - 1, false, a);
                    ok = z_silu(nch - 1, sz) && o_norm(nch - 1, a, sz);
                } else {
                    o_out(nch - 1, false);
                }
            }
        }
        tc_fence_before_sync();
    }
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tbase, TMEM_COLS);
    }
}

// Waits until *flag >= value, polling at a slow rate (the prep runs ahead of the scan,
// so this wait is never on the critical path, and slow polls leave L2 to the scan's
// copies).  Returns false if the poll limit (about 0.1 s) ran out.
__device__ __forceinline__ bool wait_ring(const unsigned long long* flag, unsigned long long value) {
    for (uint32_t i = 0; i < kFlagPolls / 4; ++i) {
        if (ld_acquire_gpu_u64(flag) >= value) return true;
        __nanosleep(400);
    }
    return false;
}

template <bool NORM>
__global__ void __launch_bounds__(TM_THREADS, 1) gdn_chunk_tmem_kernel(const __grid_constant__ ChunkTmemParams p) {
    __shared__ uint32_t s_gen;
    const int tid = threadIdx.x;
    if (tid == 0) s_gen = ld_acquire_gpu(p.sync) + 1u;
    __syncthreads();
    const uint32_t gen = s_gen;
    const int b = static_cast<int>(blockIdx.x);
    if (b < p.n_prep) {
        // prep CTA: tasks (chunk, key head) = b, b + n_prep, ... on threads 0-255
        if (tid < PREP_THREADS) {
            PrepSmemT<2>& sm = *aligned_dynamic_smem<PrepSmemT<2>, 1024>();
            const int n_kh = p.prep.n_kh;
            const int tasks = ((p.prep.n_tokens + C - 1) / C) * n_kh;
            if (b < tasks) prep_load(p.prep, sm, 0, b / n_kh, b % n_kh);
            bool ring_gave_up = false;
            for (int task = b, i = 0; task < tasks; task += p.n_prep, ++i) {
                const int next = task + p.n_prep;
                if (next < tasks) {
                    prep_load(p.prep, sm, (i + 1) & 1, next / n_kh, next % n_kh);
                    cp_async_wait<1>();
                } else {
                    cp_async_wait<0>();
                }
                // the ring slot of chunk ci: the three value heads' scan CTAs have copied out the
                // tiles of chunk ci - kTileRing (bounded; once a wait gives up, the CTA waits no
                // more)
                const int ci = task / n_kh, kh = task % n_kh;
                if (tid == 0 && ci >= kTileRing && !ring_gave_up) {
                    const unsigned long long want =
                        (static_cast<unsigned long long>(gen) << 32) | static_cast<uint32_t>(ci - kTileRing);
                    for (int m = 0; m < kHeadsPerKey && !ring_gave_up; ++m)
                        if (!wait_ring(p.ring + ((ci - kTileRing) % kTileRing) * p.prep.n_vh + kh + m * n_kh, want)) {
                            ring_gave_up = true;
                            report_error(p.status, kDevErrRingTimeout);
                        }
                }
                PrepSyncNamed::sync();
                prep_task<PrepOut::kTiles, PrepSyncNamed>(p.prep, sm, i & 1, task / n_kh, task % n_kh);
                fence_proxy_async_global();
                PrepSyncNamed::sync();
                if (tid == 0 && task != p.withhold_task) st_release_gpu(p.flags + task, gen);
            }
        }
    } else {
        tmem_scan<NORM>(p, aligned_dynamic_smem<unsigned char, 1024>(), b - p.n_prep, gen);
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

template <bool NORM>
constexpr size_t tmem_smem() {
    return (Smem<NORM>::TOTAL > sizeof(PrepSmemT<2>) ? Smem<NORM>::TOTAL : sizeof(PrepSmemT<2>)) + 1024;
}
static_assert(tmem_smem<true>() <= 227 * 1024, "tensor-memory kernel shared memory");
static_assert(tmem_smem<false>() == 221952 + 1024, "the instance without the norm keeps its size");

}  // namespace

int chunk_tmem_prep_ctas(int n_kh, int n_vh, int sm_count) {
    const int n_prep = sm_count - n_vh;
    return n_prep >= n_kh ? n_prep : 0;
}

cudaError_t preload_chunk_tmem() {
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(gdn_chunk_tmem_kernel<false>),
                                  static_cast<int>(tmem_smem<false>()));
    if (e != cudaSuccess) return e;
    return set_smem_once(reinterpret_cast<const void*>(gdn_chunk_tmem_kernel<true>), static_cast<int>(tmem_smem<true>()));
}

cudaError_t launch_chunk_tmem(const ChunkTmemParams& p, cudaStream_t s) {
    cudaError_t e = preload_chunk_tmem();
    if (e != cudaSuccess) return e;
    const bool norm = p.y != nullptr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_prep + p.prep.n_vh);
    cfg.blockDim = dim3(TM_THREADS);
    cfg.dynamicSmemBytes = norm ? tmem_smem<true>() : tmem_smem<false>();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return norm ? cudaLaunchKernelEx(&cfg, gdn_chunk_tmem_kernel<true>, p)
                : cudaLaunchKernelEx(&cfg, gdn_chunk_tmem_kernel<false>, p);
}

}  // namespace gdn
