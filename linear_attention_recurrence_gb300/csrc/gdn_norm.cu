// Gated RMSNorm of the recurrence output to FP16 ("#413 prefill: DeltaNet
// recurrence with the three value heads of a key head in one thread", section
// "What changes": gdn_out_norm_kernel writes only the FP16 copy y_h that the
// output projection reads).  Per (token, value head) row of 128 values:
//     r = 1 / sqrt(mean_j o_j^2 + eps),  y_j = fp16_rn(o_j * r * w_j * silu(z_j)).
//
// HBM-bound (per row: 512 B of o, 512 B of z read, 256 B of y written).  One warp
// per row, one float4 of o and of z per lane, streamed past L1; two rows in flight
// per warp and a grid of 8 CTAs of 128 threads per SM, grid-striding.
#include <cuda_fp16.h>

#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_norm_row.cuh"

namespace gdn {
namespace {

// 128-thread CTAs (8 per SM): small enough (threads, registers, no shared memory)
// for one to run beside a one-launch chunked recurrence CTA (256 threads of up to
// 208 registers), so a norm on a second stream overlaps the next recurrence call
// instead of delaying its launch.
constexpr int kThreads = 128;
constexpr int kCtasPerSm = 8;
constexpr int kRowsInFlight = 2;

__device__ __forceinline__ float4 ld_stream(const float* p) {
    float4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p));
    return r;
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) gdn_out_norm_kernel(const float* __restrict__ o,
                                                                 const float* __restrict__ z,
                                                                 const float* __restrict__ w, float eps,
                                                                 uint2* __restrict__ y, int64_t rows) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
    const float4 w4 = reinterpret_cast<const float4*>(w)[lane];
    for (int64_t base = warp0; base < rows; base += nwarps * kRowsInFlight) {
        float4 ov[kRowsInFlight], zv[kRowsInFlight];
#pragma unroll
        for (int u = 0; u < kRowsInFlight; ++u) {
            const int64_t row = base + u * nwarps;
            if (row < rows) {
                ov[u] = ld_stream(o + row * kD + 4 * lane);
                zv[u] = ld_stream(z + row * kD + 4 * lane);
            }
        }
#pragma unroll
        for (int u = 0; u < kRowsInFlight; ++u) {
            const int64_t row = base + u * nwarps;
            if (row >= rows) break;  // uniform across the warp
            __stcs(y + row * (kD / 4) + lane, norm_row_lane(ov[u], zv[u], w4, eps));
        }
    }
}

}  // namespace

cudaError_t launch_out_norm(const float* out, const float* z, const float* w, float eps, uint16_t* y,
                            int64_t rows, int sm_count, cudaStream_t s) {
    const int64_t warps_per_cta = kThreads / 32;
    int64_t want = (rows + warps_per_cta * kRowsInFlight - 1) / (warps_per_cta * kRowsInFlight);
    const int64_t cap = static_cast<int64_t>(sm_count) * kCtasPerSm;
    const int grid = static_cast<int>(want < cap ? want : cap);
    gdn_out_norm_kernel<<<grid, kThreads, 0, s>>>(out, z, w, eps, reinterpret_cast<uint2*>(y), rows);
    return cudaGetLastError();
}

}  // namespace gdn
