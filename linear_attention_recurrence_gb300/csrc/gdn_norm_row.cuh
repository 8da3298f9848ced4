// The gated RMSNorm of one 128-value row by one warp ("#413 prefill: DeltaNet
// recurrence with the three value heads of a key head in one thread", section
// "What changes": the FP16 normed copy y_h of the recurrence output):
//     r = 1 / sqrt(mean_j o_j^2 + eps),   y_j = fp16_rn(o_j * r * w_j * silu(z_j)).
// Lane l holds o, z and w of columns 4l..4l+3 and receives the FP16 bits of its 4
// outputs.  Every kernel that norms rows calls this one function, so they agree
// bit for bit.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

namespace gdn {

// silu(z) = z / (1 + e^-z), with the fast exponential and division (relative
// error a few FP32 ulp, far below the FP16 output's half ulp).
__device__ __forceinline__ float norm_silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__device__ __forceinline__ uint2 norm_row_lane(const float4 o, const float4 z, const float4 w, const float eps) {
    float ss = o.x * o.x;
    ss = fmaf(o.y, o.y, ss);
    ss = fmaf(o.z, o.z, ss);
    ss = fmaf(o.w, o.w, ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float r = rsqrtf(fmaf(ss, 1.0f / 128.0f, eps));
    const __half2 lo = __floats2half2_rn(o.x * r * w.x * norm_silu(z.x), o.y * r * w.y * norm_silu(z.y));
    const __half2 hi = __floats2half2_rn(o.z * r * w.z * norm_silu(z.z), o.w * r * w.w * norm_silu(z.w));
    uint2 pkd;
    pkd.x = *reinterpret_cast<const uint32_t*>(&lo);
    pkd.y = *reinterpret_cast<const uint32_t*>(&hi);
    return pkd;
}

}  // namespace gdn
