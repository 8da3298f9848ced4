// Chunked Gated DeltaNet scan with the chunk's large products on the tensor cores.
//
// Same math and prep records as gdn_chunk.cu ("#1372 DeltaNet recurrence:
// STRATA_GDN_CHUNKED=1 - the prompt's recurrence in 32-token chunks", section
// "What it does"); per value head and chunk, with S0 the state before the chunk:
//     W    = [K; Q] S0                           (64 x 48 per CTA, K = 128)  -> tcgen05
//     U'   = V - diag(e^gamma) W_K,  QS' = diag(e^gamma) W_Q
//     D    = T' U'                               (CUDA cores)
//     O    = QS' + P D                           (CUDA cores)
//     S    = e^gamma_last S0 + K^T D',  D' = diag(e^(gamma_last - gamma)) D   -> tcgen05
// The two tensor-core products run as split TF32: every FP32 operand x is written
// as hi + lo with hi = TF32(x) (round to nearest) and lo = x - hi, and the product
// accumulates hi.lo + lo.hi + hi.hi in FP32 in tensor memory (small terms first).
// Plain TF32 inputs would miss the 2e-6 FP32 tolerance by three orders of
// magnitude; the split keeps the chunked path at the FP32 CUDA-core accuracy.
//
// One CTA per (key head, 16 value columns) as in the CUDA-core scan.  Warps 0-3
// own the state in the layout of the 128-lane tensor-memory accumulator (thread i
// holds row i of the 3 heads x 16 columns); one thread issues the MMAs; all eight
// warps share the split, the D and O products and the epilogues.  Operand tiles
// live in shared memory in the K-major 128-byte-swizzled layout both TMA and the
// MMA descriptors use; k/q tiles, v columns and prep records for the next chunk are
// loaded as soon as their buffers are free.

#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int D = kD;
constexpr int C = kChunk;
constexpr int REC = kPrepRecordFloats;
constexpr int NC = 16;                  // value columns per CTA (per head)
constexpr int NCC = kHeadsPerKey * NC;  // 48 columns: head m, column j -> m*16 + j
constexpr int THREADS = 256;
constexpr uint32_t TMEM_COLS = 128;     // W at columns [0, 48), the state update at [64, 112)
constexpr uint32_t TM_W = 0, TM_S = 64;

// Shared memory (bytes from a 1024-aligned base).
constexpr uint32_t OFF_XR = 0;        // [kb 4][64 rows][128 B]: k rows 0-31, q rows 32-63 (TMA), then TF32 hi
constexpr uint32_t OFF_XL = 32768;    // same layout: lo parts
constexpr uint32_t OFF_KTH = 65536;   // K^T [128 rows i][32 t], hi
constexpr uint32_t OFF_KTL = 81920;   // lo
constexpr uint32_t OFF_SH = 98304;    // S0^T [kb 4][48 rows][128 B], hi
constexpr uint32_t OFF_SL = 122880;   // lo
constexpr uint32_t OFF_DTH = 147456;  // D'^T [48 rows][32 t], hi
constexpr uint32_t OFF_DTL = 153600;  // lo
constexpr uint32_t OFF_V = 159744;    // [3][32][16] floats (TMA)
constexpr uint32_t OFF_REC = 165888;  // [3][REC] floats (bulk copies)
constexpr uint32_t OFF_W = 191232;    // [64][48] floats: U' (rows 0-31), QS' (rows 32-63)
constexpr uint32_t OFF_DM = 203520;   // [32][48] floats: D
constexpr uint32_t OFF_BAR = 209664;  // 5 mbarriers + the tensor-memory address
constexpr uint32_t SMEM_BYTES = OFF_BAR + 64;
enum { BAR_KQ = 0, BAR_V = 1, BAR_REC = 2, BAR_G1 = 3, BAR_G4 = 4 };
constexpr uint32_t TX_KQ = 2 * C * D * 4, TX_V = kHeadsPerKey * C * NC * 4, TX_REC = kHeadsPerKey * REC * 4;

__device__ __forceinline__ float4 tf32_rna4(float4 x) {
    return make_float4(tf32_rna(x.x), tf32_rna(x.y), tf32_rna(x.z), tf32_rna(x.w));
}

__global__ void __launch_bounds__(THREADS, 1) gdn_chunk_scan_tc_kernel(const __grid_constant__ ChunkScanParams p) {
    unsigned char* sm = aligned_dynamic_smem<unsigned char, 1024>();
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 48);
    float* V = reinterpret_cast<float*>(sm + OFF_V);
    float* R = reinterpret_cast<float*>(sm + OFF_REC);
    float* W = reinterpret_cast<float*>(sm + OFF_W);
    float* Dm = reinterpret_cast<float*>(sm + OFF_DM);
    const int kh = blockIdx.x;
    const int c0 = blockIdx.y * NC;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_kh = p.n_kh, n_vh = p.n_vh;
    const int nch = (p.n_tokens + C - 1) / C;

    if (tid == 0) {
        for (int b = 0; b < 5; ++b) mbar_init(&bar[b], 1);
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(tslot, TMEM_COLS);

    // S0^T as TF32 hi / lo for the W product (thread i of warps 0-3 writes row i's 48 columns).
    auto write_state_split = [&](const float* Srow, int i) {
        const uint32_t base = (i >> 5) * 6144;
#pragma unroll
        for (int c = 0; c < NCC; ++c) {
            const float h = tf32_rna(Srow[c]);
            const uint32_t off = base + sw128(c, i & 31);
            *reinterpret_cast<float*>(sm + OFF_SH + off) = h;
            *reinterpret_cast<float*>(sm + OFF_SL + off) = Srow[c] - h;
        }
    };

    float Sreg[NCC];  // warps 0-3: row i = tid of the state, columns m*16 + j
    if (warp < 4) {
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m) {
            const float4* src =
                reinterpret_cast<const float4*>(p.state + (static_cast<int64_t>(kh + m * n_kh) * D + tid) * D + c0);
#pragma unroll
            for (int j4 = 0; j4 < NC / 4; ++j4) {
                const float4 v = src[j4];
                Sreg[m * NC + 4 * j4 + 0] = v.x;
                Sreg[m * NC + 4 * j4 + 1] = v.y;
                Sreg[m * NC + 4 * j4 + 2] = v.z;
                Sreg[m * NC + 4 * j4 + 3] = v.w;
            }
        }
        write_state_split(Sreg, tid);
    }

    auto issue_kq = [&](int c) {
        const int y = static_cast<int>(p.t_begin + static_cast<int64_t>(c) * C);
        mbar_arrive_expect_tx(&bar[BAR_KQ], TX_KQ);
#pragma unroll
        for (int kb = 0; kb < D / 32; ++kb) {
            tma_load_2d(sm + OFF_XR + kb * 8192, &p.tm_k, &bar[BAR_KQ], kh * D + 32 * kb, y);
            tma_load_2d(sm + OFF_XR + kb * 8192 + 4096, &p.tm_q, &bar[BAR_KQ], kh * D + 32 * kb, y);
        }
    };
    auto issue_v = [&](int c) {
        const int y = static_cast<int>(p.t_begin + static_cast<int64_t>(c) * C);
        mbar_arrive_expect_tx(&bar[BAR_V], TX_V);
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m)
            tma_load_2d(V + m * C * NC, &p.tm_v, &bar[BAR_V], (kh + m * n_kh) * D + c0, y);
    };
    auto issue_rec = [&](int c) {
        mbar_arrive_expect_tx(&bar[BAR_REC], TX_REC);
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m)
            bulk_load(R + m * REC, p.prep + (static_cast<int64_t>(c) * n_vh + kh + m * n_kh) * REC, REC * 4,
                      &bar[BAR_REC]);
    };

    fence_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tbase = *tslot;
    if (tid == 0) {
        issue_kq(0);
        issue_v(0);
        issue_rec(0);
    }
    __syncwarp();  // warp 0's other lanes wait for lane 0's issues before spinning on barriers

    const int pm = tid >> 6, pti = (tid >> 3) & 7, pjp = tid & 7;  // D and O tiles (threads 0..191)
    float el[kHeadsPerKey] = {1.f, 1.f, 1.f};
    bool failed = false;

    for (int c = 0; c < nch; ++c) {
        const uint32_t par = static_cast<uint32_t>(c & 1);
        const int nt = min(C, p.n_tokens - c * C);

        // ---- split the k / q tile into TF32 hi (in place) and lo; K^T hi / lo ----
        if (!mbar_wait(&bar[BAR_KQ], par)) failed = true;
        if (!failed) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {  // k rows: lane = token row t, 16-byte chunk q of the key dim
                const int q = warp + 8 * u, kb = q >> 3, cc = q & 7, t = lane;
                const uint32_t off = kb * 8192 + t * 128 + ((cc ^ (t & 7)) << 4);
                const float4 x = *reinterpret_cast<const float4*>(sm + OFF_XR + off);
                const float4 h = tf32_rna4(x);
                const float4 l = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
                *reinterpret_cast<float4*>(sm + OFF_XR + off) = h;
                *reinterpret_cast<float4*>(sm + OFF_XL + off) = l;
                const int i0 = 32 * kb + 4 * cc;
                const float hv[4] = {h.x, h.y, h.z, h.w}, lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t ko = sw128(i0 + e, t);
                    *reinterpret_cast<float*>(sm + OFF_KTH + ko) = hv[e];
                    *reinterpret_cast<float*>(sm + OFF_KTL + ko) = lv[e];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {  // q rows
                const int idx = tid + THREADS * u, row = 32 + (idx & 31), q = idx >> 5, kb = q >> 3, cc = q & 7;
                const uint32_t off = kb * 8192 + row * 128 + ((cc ^ (row & 7)) << 4);
                const float4 x = *reinterpret_cast<const float4*>(sm + OFF_XR + off);
                const float4 h = tf32_rna4(x);
                *reinterpret_cast<float4*>(sm + OFF_XR + off) = h;
                *reinterpret_cast<float4*>(sm + OFF_XL + off) = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
            }
        }
        fence_async_smem();
        tc_fence_before_sync();
        if (__syncthreads_or(failed)) break;

        // ---- W = [K; Q] S0 on the tensor cores: M = 64, N = 48, K = 128, three passes ----
        if (tid == 0) {
            tc_fence_after_sync();
            const uint32_t id = umma_idesc_tf32(64, NCC);
            const uint32_t a_off[3] = {OFF_XR, OFF_XL, OFF_XR}, b_off[3] = {OFF_SL, OFF_SH, OFF_SH};
#pragma unroll
            for (int pass = 0; pass < 3; ++pass)
#pragma unroll
                for (int ks = 0; ks < D / 8; ++ks) {
                    const uint64_t a = umma_desc_sw128(sm + a_off[pass] + (ks >> 2) * 8192 + (ks & 3) * 32);
                    const uint64_t b = umma_desc_sw128(sm + b_off[pass] + (ks >> 2) * 6144 + (ks & 3) * 32);
                    umma_tf32(tbase + TM_W, a, b, id, pass > 0 || ks > 0);
                }
            umma_commit(&bar[BAR_G1]);
        }
        __syncwarp();
        if (!mbar_wait(&bar[BAR_G1], par)) failed = true;
        tc_fence_after_sync();
        if (tid == 0 && !failed && c + 1 < nch) issue_kq(c + 1);  // the product has read the k / q tile
        __syncwarp();
        if (!mbar_wait(&bar[BAR_V], par) || !mbar_wait(&bar[BAR_REC], par)) failed = true;
        // ---- U' = V - e^gamma W_K and QS' = e^gamma W_Q (warps 0-3; W row r sits in lane 32*(r/16) + r%16) ----
        if (warp < 4 && !__any_sync(0xffffffffu, failed)) {
            float w[NCC];
            const uint32_t ta = tbase + (static_cast<uint32_t>(32 * warp) << 16) + TM_W;
            tmem_ld16(ta, w);
            tmem_ld16(ta + 16, w + 16);
            tmem_ld16(ta + 32, w + 32);
            if (lane < 16) {
                const int r = 16 * warp + lane;
                if (r < C) {
#pragma unroll
                    for (int m = 0; m < kHeadsPerKey; ++m) {
                        const float eg = R[m * REC + kRecEG + r];
#pragma unroll
                        for (int j = 0; j < NC; ++j)
                            W[r * NCC + m * NC + j] = V[(m * C + r) * NC + j] - eg * w[m * NC + j];
                    }
                } else {
                    const int t = r - C;
#pragma unroll
                    for (int m = 0; m < kHeadsPerKey; ++m) {
                        const float eg = R[m * REC + kRecEG + t];
#pragma unroll
                        for (int j = 0; j < NC; ++j) W[r * NCC + m * NC + j] = eg * w[m * NC + j];
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < kHeadsPerKey; ++m) el[m] = R[m * REC + kRecEG + C - 1];
        }
        tc_fence_before_sync();
        if (__syncthreads_or(failed)) break;
        if (tid == 0 && c + 1 < nch) issue_v(c + 1);
        __syncwarp();

        // ---- D = T' U' per head (threads 0..191); D'^T = (e^(gamma_last - gamma) D)^T as TF32 hi / lo ----
        if (tid < kHeadsPerKey * 64) {
            const float* tp = R + pm * REC + kRecTP;
            float acc[4][2];
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[r][0] = acc[r][1] = 0.f;
#pragma unroll 8
            for (int s = 0; s < C; ++s) {
                const float4 a = *reinterpret_cast<const float4*>(tp + s * C + 4 * pti);
                const float2 u = *reinterpret_cast<const float2*>(W + s * NCC + pm * NC + 2 * pjp);
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
                const float er = R[pm * REC + kRecER + t];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int col = pm * NC + 2 * pjp + q;
                    Dm[t * NCC + col] = acc[r][q];
                    const float dd = er * acc[r][q];
                    const float h = tf32_rna(dd);
                    const uint32_t off = sw128(col, t);
                    *reinterpret_cast<float*>(sm + OFF_DTH + off) = h;
                    *reinterpret_cast<float*>(sm + OFF_DTL + off) = dd - h;
                }
            }
        }
        fence_async_smem();
        tc_fence_before_sync();
        __syncthreads();

        // ---- state update K^T D' on the tensor cores (M = 128, N = 48, K = 32) while P D runs ----
        if (tid == 0) {
            tc_fence_after_sync();
            const uint32_t id = umma_idesc_tf32(128, NCC);
            const uint32_t a_off[3] = {OFF_KTH, OFF_KTL, OFF_KTH}, b_off[3] = {OFF_DTL, OFF_DTH, OFF_DTH};
#pragma unroll
            for (int pass = 0; pass < 3; ++pass)
#pragma unroll
                for (int ks = 0; ks < C / 8; ++ks)
                    umma_tf32(tbase + TM_S, umma_desc_sw128(sm + a_off[pass] + ks * 32),
                              umma_desc_sw128(sm + b_off[pass] + ks * 32), id, pass > 0 || ks > 0);
            umma_commit(&bar[BAR_G4]);
        }
        __syncwarp();
        // ---- O = QS' + P D per head -> out (threads 0..191) ----
        if (tid < kHeadsPerKey * 64) {
            const float* pt = R + pm * REC + kRecPT;
            float acc[4][2];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float2 w = *reinterpret_cast<const float2*>(W + (C + 4 * pti + r) * NCC + pm * NC + 2 * pjp);
                acc[r][0] = w.x;
                acc[r][1] = w.y;
            }
#pragma unroll 8
            for (int s = 0; s < C; ++s) {
                const float4 a = *reinterpret_cast<const float4*>(pt + s * C + 4 * pti);
                const float2 d = *reinterpret_cast<const float2*>(Dm + s * NCC + pm * NC + 2 * pjp);
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
        }
        __syncthreads();
        if (tid == 0 && c + 1 < nch) issue_rec(c + 1);  // the records of this chunk are no longer read
        __syncwarp();

        // ---- S = e^gamma_last S0 + K^T D' (warps 0-3), then S^T as TF32 hi / lo for the next chunk ----
        if (warp < 4) {
            if (!mbar_wait(&bar[BAR_G4], par)) failed = true;
            tc_fence_after_sync();
            if (!__any_sync(0xffffffffu, failed)) {
                float u[NCC];
                const uint32_t ta = tbase + (static_cast<uint32_t>(32 * warp) << 16) + TM_S;
                tmem_ld16(ta, u);
                tmem_ld16(ta + 16, u + 16);
                tmem_ld16(ta + 32, u + 32);
#pragma unroll
                for (int cc = 0; cc < NCC; ++cc) Sreg[cc] = fmaf(el[cc / NC], Sreg[cc], u[cc]);
                write_state_split(Sreg, tid);
            }
        }
        fence_async_smem();
        tc_fence_before_sync();
        if (__syncthreads_or(failed)) break;
    }

    if (failed) {
        if (tid == 0) report_timeout(p.status);
    } else if (warp < 4) {
#pragma unroll
        for (int m = 0; m < kHeadsPerKey; ++m) {
            float4* dst = reinterpret_cast<float4*>(p.state + (static_cast<int64_t>(kh + m * n_kh) * D + tid) * D + c0);
#pragma unroll
            for (int j4 = 0; j4 < NC / 4; ++j4)
                dst[j4] = make_float4(Sreg[m * NC + 4 * j4], Sreg[m * NC + 4 * j4 + 1], Sreg[m * NC + 4 * j4 + 2],
                                      Sreg[m * NC + 4 * j4 + 3]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tbase, TMEM_COLS);
    }
}

}  // namespace

cudaError_t preload_chunk_scan_tc() {
    return set_smem_once(reinterpret_cast<const void*>(gdn_chunk_scan_tc_kernel), static_cast<int>(SMEM_BYTES + 1024));
}

cudaError_t launch_chunk_scan_tc(const ChunkScanParams& p, cudaStream_t s) {
    const size_t smem = SMEM_BYTES + 1024;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(gdn_chunk_scan_tc_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_kh, D / NC);
    gdn_chunk_scan_tc_kernel<<<grid, THREADS, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_chunk_scan_default(const ChunkScanParams& p, cudaStream_t s) {
    const ScanKind k = chunk_scan_kind();
    return k == ScanKind::kTcgen05 ? launch_chunk_scan_tc(p, s) : launch_chunk_scan(p, k != ScanKind::kFma, s);
}

}  // namespace gdn
