// One decode step of the Gated DeltaNet recurrence for a batch of independent
// sequences, each with its own state (the same per-token update as the prefill
// recurrence, "#413 prefill: DeltaNet recurrence with the three value heads of a
// key head in one thread", section "What changes", applied to T = 1).
//
// Bound by HBM: every step reads and rewrites every sequence's 48 x 64 KB of
// state.  One CTA per (sequence, value head) holds that head's 128 x 128 state in
// registers between the column sums and the update, so the state crosses HBM
// exactly once each way.  Thread (warp w, lane l) owns rows w, w+8, ..., w+120 and
// columns 4l..4l+3 (row-major float4 loads, fully coalesced).  Column sums S^T k
// and S^T q are reduced over the 8 warps through shared memory in a fixed order;
// then delta and the output follow, and the state is updated and written back.
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int D = kD;
constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int RPT = D / WARPS;  // rows per thread (16)

__global__ void __launch_bounds__(THREADS) gdn_decode_kernel(const DecodeParams p) {
    __shared__ float part_k[WARPS][D];
    __shared__ float part_q[WARPS][D];
    __shared__ float delta_s[D];
    __shared__ float kq_s;
    const int h = blockIdx.x, b = blockIdx.y;
    const int kh = h % p.n_kh;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t sbase = (static_cast<int64_t>(b) * p.n_vh + h) * D * D;
    const float* kv = p.k + (static_cast<int64_t>(b) * p.n_kh + kh) * D;
    const float* qv = p.q + (static_cast<int64_t>(b) * p.n_kh + kh) * D;

    float4 S[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r)
        S[r] = __ldcs(reinterpret_cast<const float4*>(p.state + sbase + static_cast<int64_t>(warp + WARPS * r) * D) +
                      lane);
    float kr[RPT], qr[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        kr[r] = __ldg(kv + warp + WARPS * r);
        qr[r] = __ldg(qv + warp + WARPS * r);
    }
    const float a = expf(__ldg(p.g + static_cast<int64_t>(b) * p.n_vh + h));
    const float bt = __ldg(p.beta + static_cast<int64_t>(b) * p.n_vh + h);
    if (warp == 0) {  // k . q, fixed shuffle order
        const float4 k4 = reinterpret_cast<const float4*>(kv)[lane];
        const float4 q4 = reinterpret_cast<const float4*>(qv)[lane];
        float s = fmaf(k4.w, q4.w, fmaf(k4.z, q4.z, fmaf(k4.y, q4.y, k4.x * q4.x)));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) kq_s = s;
    }

    // partial column sums over this thread's rows
    float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sq = sk;
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        sk.x = fmaf(S[r].x, kr[r], sk.x);
        sk.y = fmaf(S[r].y, kr[r], sk.y);
        sk.z = fmaf(S[r].z, kr[r], sk.z);
        sk.w = fmaf(S[r].w, kr[r], sk.w);
        sq.x = fmaf(S[r].x, qr[r], sq.x);
        sq.y = fmaf(S[r].y, qr[r], sq.y);
        sq.z = fmaf(S[r].z, qr[r], sq.z);
        sq.w = fmaf(S[r].w, qr[r], sq.w);
    }
    reinterpret_cast<float4*>(part_k[warp])[lane] = sk;
    reinterpret_cast<float4*>(part_q[warp])[lane] = sq;
    __syncthreads();

    // column j = threadIdx.x (< 128): sum the 8 warp partials in order, then delta and o
    if (threadIdx.x < D) {
        const int j = threadIdx.x;
        float tk = 0.f, tq = 0.f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            tk += part_k[w][j];
            tq += part_q[w][j];
        }
        const float vj = __ldg(p.v + (static_cast<int64_t>(b) * p.n_vh + h) * D + j);
        const float delta = bt * (vj - a * tk);
        delta_s[j] = delta;
        p.out[(static_cast<int64_t>(b) * p.n_vh + h) * D + j] = fmaf(kq_s, delta, a * tq);
    }
    __syncthreads();

    const float4 d4 = reinterpret_cast<const float4*>(delta_s)[lane];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        float4 s = S[r];
        s.x = fmaf(kr[r], d4.x, a * s.x);
        s.y = fmaf(kr[r], d4.y, a * s.y);
        s.z = fmaf(kr[r], d4.z, a * s.z);
        s.w = fmaf(kr[r], d4.w, a * s.w);
        __stcs(reinterpret_cast<float4*>(p.state + sbase + static_cast<int64_t>(warp + WARPS * r) * D) + lane, s);
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s) {
    dim3 grid(p.n_vh, p.batch);
    gdn_decode_kernel<<<grid, THREADS, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
