// Pre-stage: the recurrence's inputs from a layer's projections ("Round 20 Track C
// Audit: gdn_pre Key-Head t >= 3 Vectorized conv_w Fast Path + gdn_scan_r ...",
// section 1 "Summary of Changes": a 4-tap causal convolution per channel of the
// packed qkv rows, q of key head kh at channels kh*d, k at (n_kh + kh)*d, taps on
// rows t-3 .. t, then the normalised q, k, the convolved v and the gates).
//
// Bound by HBM: every qkv row is read once and every output row written once.
// One warp per (run of kRun consecutive tokens, 128-channel head slot): lane l
// owns channels 4l..4l+3 of the slot, keeps the three previous rows in
// registers (a sliding window, so a run reads only three extra rows) and the
// next kAhead rows in flight while it works on the current one.  Head slots of q and k add
// their squares across the warp by xor shuffles for the L2 norm.  Further warps
// compute the gates of kGateRows tokens each (contiguous, coalesced) and copy the
// last three rows into the history handed to the next call.
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int D = kD;
constexpr int kRun = 128;       // tokens per convolution warp
constexpr int kAhead = 4;       // qkv rows each convolution lane keeps in flight
constexpr int kGateRows = 64;   // tokens per gate warp
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// x sigmoid(x) = x / (1 + e^-x) with the hardware exponential and the fast
// division (a few FP32 ulp each at these arguments; for x -> -inf the quotient
// is -0): the kernel is issue-bound, and the outputs stay within a few 1e-7 of
// the FP64 values relative to their largest magnitude (the tests hold them to
// 2e-6).
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.f + __expf(-x)); }

__device__ __forceinline__ float softplus(float x) { return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))); }

__device__ __forceinline__ float4 ld4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

// Row r (may be -3..-1: the history, or zeros without one) of the slot's 4 channels.
__device__ __forceinline__ float4 row4(const PrestageParams& p, int64_t r, int64_t col) {
    if (r >= 0) return ld4(p.qkv + r * p.cw + col);
    if (p.hist_in) return ld4(p.hist_in + (3 + r) * p.cw + col);
    return make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ float conv1(float w0, float w1, float w2, float w3, float x0, float x1, float x2,
                                       float x3) {
    float x = w0 * x0;
    x = fmaf(w1, x1, x);
    x = fmaf(w2, x2, x);
    return fmaf(w3, x3, x);
}

__global__ void __launch_bounds__(kThreads) gdn_prestage_kernel(const PrestageParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t task = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const int nb = 2 * p.n_kh + p.n_vh;  // head slots per row
    const int64_t n_runs = (p.T + kRun - 1) / kRun;
    const int64_t conv_tasks = n_runs * nb;
    const int64_t gate_tasks = (p.T + kGateRows - 1) / kGateRows;

    if (task < conv_tasks) {
        const int hs = static_cast<int>(task % nb);
        const int64_t t0 = (task / nb) * kRun;
        const int64_t t1 = min(t0 + kRun, p.T);
        const int64_t col = static_cast<int64_t>(hs) * D + 4 * lane;
        // taps of the lane's 4 channels: w[i] = conv_w[col + i][0..3]
        const float4 w0 = ld4(p.conv_w + (col + 0) * 4), w1 = ld4(p.conv_w + (col + 1) * 4);
        const float4 w2 = ld4(p.conv_w + (col + 2) * 4), w3 = ld4(p.conv_w + (col + 3) * 4);
        float4 xm3 = row4(p, t0 - 3, col), xm2 = row4(p, t0 - 2, col), xm1 = row4(p, t0 - 1, col);
        const bool is_q = hs < p.n_kh, is_k = !is_q && hs < 2 * p.n_kh;
        float* dst;
        int64_t dst_stride;
        if (is_q) {
            dst = p.q + static_cast<int64_t>(hs) * D + 4 * lane;
            dst_stride = static_cast<int64_t>(p.n_kh) * D;
        } else if (is_k) {
            dst = p.k + static_cast<int64_t>(hs - p.n_kh) * D + 4 * lane;
            dst_stride = static_cast<int64_t>(p.n_kh) * D;
        } else {
            dst = p.v + static_cast<int64_t>(hs - 2 * p.n_kh) * D + 4 * lane;
            dst_stride = static_cast<int64_t>(p.n_vh) * D;
        }
        dst += t0 * dst_stride;
        // rows t0 .. t0+kAhead-1 in flight; each step consumes one and loads the row
        // kAhead further on, so every lane keeps kAhead 16-byte loads outstanding
        const float* src = p.qkv + t0 * p.cw + col;
        const int n = static_cast<int>(t1 - t0);
        float4 ahead[kAhead];
#pragma unroll
        for (int i = 0; i < kAhead; ++i) ahead[i] = (i < n) ? ld4(src + i * p.cw) : make_float4(0.f, 0.f, 0.f, 0.f);
        src += kAhead * p.cw;
        for (int i0 = 0; i0 < n; i0 += kAhead) {
#pragma unroll
            for (int i = 0; i < kAhead; ++i) {
                if (i0 + i < n) {
                    const float4 xc = ahead[i];
                    if (i0 + i + kAhead < n) ahead[i] = ld4(src);
                    src += p.cw;
                    float u[4];
                    u[0] = conv1(w0.x, w0.y, w0.z, w0.w, xm3.x, xm2.x, xm1.x, xc.x);
                    u[1] = conv1(w1.x, w1.y, w1.z, w1.w, xm3.y, xm2.y, xm1.y, xc.y);
                    u[2] = conv1(w2.x, w2.y, w2.z, w2.w, xm3.z, xm2.z, xm1.z, xc.z);
                    u[3] = conv1(w3.x, w3.y, w3.z, w3.w, xm3.w, xm2.w, xm1.w, xc.w);
                    if (p.activation) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) u[j] = silu(u[j]);
                    }
                    if (is_q || is_k) {
                        float ss = u[0] * u[0];
                        ss = fmaf(u[1], u[1], ss);
                        ss = fmaf(u[2], u[2], ss);
                        ss = fmaf(u[3], u[3], ss);
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                        float r = rsqrtf(ss + p.eps);
                        if (is_q) r *= p.q_scale;
#pragma unroll
                        for (int j = 0; j < 4; ++j) u[j] *= r;
                    }
                    __stcs(reinterpret_cast<float4*>(dst), make_float4(u[0], u[1], u[2], u[3]));
                    dst += dst_stride;
                    xm3 = xm2;
                    xm2 = xm1;
                    xm1 = xc;
                }
            }
        }
        return;
    }

    const int64_t gt = task - conv_tasks;
    if (gt < gate_tasks) {
        // gates of tokens [gt * kGateRows, ...), all value heads: contiguous in [T][n_vh]
        const int64_t e0 = gt * kGateRows * p.n_vh;
        const int64_t e1 = min((gt + 1) * kGateRows, p.T) * p.n_vh;
        for (int64_t e = e0 + lane; e < e1; e += 32) {
            const int h = static_cast<int>(e % p.n_vh);
            const float x = __ldg(p.a + e) + __ldg(p.dt_bias + h);
            p.g[e] = -expf(__ldg(p.A_log + h)) * softplus(x);
            p.beta[e] = 1.f / (1.f + expf(-__ldg(p.b + e)));
        }
        return;
    }

    const int64_t ht = gt - gate_tasks;  // history rows handed to the next call
    if (p.hist_out && ht < 3 * static_cast<int64_t>(nb)) {
        const int i = static_cast<int>(ht / nb), hs = static_cast<int>(ht % nb);
        const int64_t col = static_cast<int64_t>(hs) * D + 4 * lane;
        *reinterpret_cast<float4*>(p.hist_out + i * p.cw + col) = row4(p, p.T - 3 + i, col);
    }
}

}  // namespace

cudaError_t launch_prestage(const PrestageParams& p, cudaStream_t s) {
    const int nb = 2 * p.n_kh + p.n_vh;
    const int64_t tasks = ((p.T + kRun - 1) / kRun) * nb + (p.T + kGateRows - 1) / kGateRows + 3 * nb;
    const int64_t blocks = (tasks + kWarps - 1) / kWarps;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    gdn_prestage_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
