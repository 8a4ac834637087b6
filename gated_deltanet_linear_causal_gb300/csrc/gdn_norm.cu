// gdn_norm.cu -- gated RMSNorm of the layer output (MNN discussion "MNN Model
// Support: Qwen3.5", section 2): y = weight * o / sqrt(mean(o^2) + eps) * silu(z)
// per row of head_v_dim values.  HBM-bound: one read of o (fp32) and z, one write
// of y, per element.
#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kNormThreads = 256;

// One warp per row, grid-stride over rows; each lane holds dv/32 values as
// groups of 4 (dv a multiple of 128) or single values.
template <typename T>
__global__ void __launch_bounds__(kNormThreads) gated_rmsnorm_kernel(long long rows, int dv, const float* __restrict__ o,
                                                                    const T* __restrict__ z,
                                                                    const float* __restrict__ weight, float eps,
                                                                    T* __restrict__ y) {
    const int lane = threadIdx.x & 31;
    const long long w0 = ((long long)blockIdx.x * kNormThreads + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * kNormThreads) >> 5;
    const float inv_dv = 1.f / (float)dv;
    for (long long r = w0; r < rows; r += nw) {
        const float* orow = o + r * dv;
        float ss = 0.f;
        for (int j = lane; j < dv; j += 32) ss = fmaf(orow[j], orow[j], ss);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float rinv = rsqrtf(fmaf(ss, inv_dv, eps));
        for (int j = lane; j < dv; j += 32) {
            const float zv = to_f32(z[r * dv + j]);
            const float v = __fmul_rn(__fmul_rn(weight[j], __fmul_rn(orow[j], rinv)), silu(zv));
            y[r * dv + j] = from_f32<T>(v);
        }
    }
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const Geom& g, long long rows, const float* o, const void* z, const float* weight,
                                 float eps, void* y, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const long long warps = rows;
    const int blocks = (int)std::min<long long>((warps * 32 + kNormThreads - 1) / kNormThreads, 152LL * 16);
    if (g.io_bf16)
        gated_rmsnorm_kernel<__nv_bfloat16><<<blocks, kNormThreads, 0, stream>>>(
            rows, g.dv, o, static_cast<const __nv_bfloat16*>(z), weight, eps, static_cast<__nv_bfloat16*>(y));
    else
        gated_rmsnorm_kernel<float><<<blocks, kNormThreads, 0, stream>>>(rows, g.dv, o, static_cast<const float*>(z),
                                                                        weight, eps, static_cast<float*>(y));
    return cudaGetLastError();
}

}  // namespace gdn
