// gdn_common.cuh -- device helpers shared by the Gated DeltaNet kernels.
//
// The per-token arithmetic of the gated delta rule (MNN discussion "MNN Model
// Support: Qwen3.5", section 1.2, Step 5) for the slice kernels of
// gdn_step.cu lives here, in `StateSlice::step`, with explicit roundings that
// match the streaming kernel's `Tile::step`: decode and verify run the same
// instructions in the same order, so a verify snapshot after t tokens is
// bitwise equal to t decode calls.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kStepThreads = 128;  // threads of one state-slice CTA
constexpr int kSliceCols = 32;     // value columns held by one CTA
constexpr int kMaxConv = 8;        // largest supported conv width K
constexpr int kMaxVerify = 16;     // largest verify block L

// ---- element I/O ----------------------------------------------------------
template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

template <typename T>
__device__ __forceinline__ T zero_elem();
template <>
__device__ __forceinline__ float zero_elem<float>() { return 0.f; }
template <>
__device__ __forceinline__ __nv_bfloat16 zero_elem<__nv_bfloat16>() { return __float2bfloat16_rn(0.f); }

// Streaming (evict-first) 128-bit global access for data touched once per call.
__device__ __forceinline__ float4 ld_stream(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st_stream(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }

__device__ __forceinline__ float silu(float y) { return y / (1.f + expf(-y)); }
// SiLU from the fast exponential and division intrinsics, for the output gate of the
// prefill's fused norm, where it is one factor of a product that is then rounded to
// the io type: relative error about 1e-6 for |y| < 10 (the exact form's IEEE division
// costs several times the instructions).  Below y = -87 the denominator passes 2^126
// and __fdividef gives 0, where silu(y) is under 1e-35.
__device__ __forceinline__ float silu_fast(float y) { return __fdividef(y, 1.f + __expf(-y)); }
// silu_fast of N values as separate passes (the exponentials, then the quotients), so
// the N special-function chains overlap; written as one loop of silu_fast calls they
// were compiled to run one after another, at several times the cost.  s may be y.
template <int N>
__device__ __forceinline__ void silu_fast_n(const float (&y)[N], float (&s)[N]) {
    float e[N];
#pragma unroll
    for (int j = 0; j < N; ++j) e[j] = __expf(-y[j]);
#pragma unroll
    for (int j = 0; j < N; ++j) s[j] = __fdividef(y[j], 1.f + e[j]);
}

// Gate parameterisation of section 1.2: with per-value-head A_log and dt_bias
// set, the gate input is the raw projection a and the log-decay is
// -exp(A_log[h]) * softplus(a + dt_bias[h]), softplus(x) = log(1 + e^x) (x
// itself above 20, where the two agree in fp32); the beta input is the raw b
// and the rate is sigmoid(b).  Without them the inputs are used as they are.
__device__ __forceinline__ float gate_of(const float* A_log, const float* dt_bias, float raw, int h) {
    if (!A_log) return raw;
    const float x = raw + dt_bias[h];
    const float sp = x > 20.f ? x : log1pf(expf(x));
    return -expf(A_log[h]) * sp;
}
__device__ __forceinline__ float beta_of(const float* A_log, float raw) {
    return A_log ? 1.f / (1.f + expf(-raw)) : raw;
}

// ---- thread-block cluster barrier (sm_90+) ----------------------------------
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}

// ---- causal conv window ------------------------------------------------------
// The last KMAX raw samples of one channel, newest in raw[KMAX-1], for a conv
// width K <= KMAX.  The weights are right-aligned the same way with zeros in
// front, so the K-tap cross-correlation (tap K-1 on the newest sample) is a
// KMAX-term FMA chain whose leading terms are exact zeros: every KMAX gives the
// same bits for finite inputs.
template <typename T, int KMAX = kMaxConv>
struct ConvWindow {
    static constexpr int kMaxConv = KMAX;
    T raw[KMAX];    // samples in storage type (also the state written back)
    float w[KMAX];

    __device__ __forceinline__ void load(const T* state, const T* weight, int K) {
#pragma unroll
        for (int j = 0; j < kMaxConv; ++j) {
            const int s = j - (kMaxConv + 1 - K);  // index into state [K-1]
            raw[j] = (s >= 0) ? state[s] : zero_elem<T>();
            const int wi = j - (kMaxConv - K);     // index into weight [K]
            w[j] = (wi >= 0) ? to_f32(weight[wi]) : 0.f;
        }
    }
    // Push the next sample; return the conv sum (before the SiLU) for the token it completes.
    __device__ __forceinline__ float push_pre(T v) {
#pragma unroll
        for (int j = 0; j < kMaxConv - 1; ++j) raw[j] = raw[j + 1];
        raw[kMaxConv - 1] = v;
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxConv; ++j) acc = fmaf(w[j], to_f32(raw[j]), acc);
        return acc;
    }
    // Push the next sample; return silu(conv) for the token it completes.
    __device__ __forceinline__ float push(T v) { return silu(push_pre(v)); }
    // Write the K-1 sample conv state after the last push (oldest first) to dst.
    // Loop bounds and register indices are compile-time: the window stays in
    // registers.
    __device__ __forceinline__ void store_state(T* dst, int K) const {
#pragma unroll
        for (int j = 0; j < kMaxConv; ++j) {
            const int e = j - (kMaxConv + 1 - K);
            if (e >= 0) dst[e] = raw[j];
        }
    }
};

// ---- one 32-column slice of a value head's state ------------------------------
// dk rows x 32 columns of S, row-major in global memory with row stride dv.
// Thread t holds column quad cq = t % 8 (columns 4cq..4cq+3) of rows
// rg + 16m, rg = t / 8, m = 0..DK/16-1.
template <int DK>
struct StateSlice {
    static constexpr int RPT = DK / 16;
    float4 s[RPT];

    __device__ __forceinline__ static int cq() { return threadIdx.x & 7; }
    __device__ __forceinline__ static int rg() { return threadIdx.x >> 3; }

    __device__ __forceinline__ void load(const float* base, int dv) {
#pragma unroll
        for (int m = 0; m < RPT; ++m) s[m] = ld_stream(base + (size_t)(rg() + 16 * m) * dv + 4 * cq());
    }
    __device__ __forceinline__ void store(float* base, int dv) const {
#pragma unroll
        for (int m = 0; m < RPT; ++m) st_stream(base + (size_t)(rg() + 16 * m) * dv + 4 * cq(), s[m]);
    }

    // One token of the gated delta rule on this slice.
    //   k, q : the token's normalised key and scaled query (shared memory, DK floats)
    //   v4   : this thread's 4 value entries; alpha = exp(g); beta; kq = k.q
    //   red  : shared scratch of 4 warps x 64 floats (alternate two buffers by token)
    // Returns this thread's 4 output columns.  With S the state before the token:
    //   a = (alpha S)^T k, delta = beta (v - a), S' = alpha S + k delta^T,
    //   o = S'^T q = alpha S^T q + delta (k.q).
    __device__ __forceinline__ float4 step(const float* k, const float* q, float4 v4, float alpha,
                                           float beta, float kq, float* red) {
        float a[4] = {0.f, 0.f, 0.f, 0.f}, c[4] = {0.f, 0.f, 0.f, 0.f};
        float kr[RPT];
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            kr[m] = k[rg() + 16 * m];
            const float qr = q[rg() + 16 * m];
            a[0] = fmaf(s[m].x, kr[m], a[0]); a[1] = fmaf(s[m].y, kr[m], a[1]);
            a[2] = fmaf(s[m].z, kr[m], a[2]); a[3] = fmaf(s[m].w, kr[m], a[3]);
            c[0] = fmaf(s[m].x, qr, c[0]); c[1] = fmaf(s[m].y, qr, c[1]);
            c[2] = fmaf(s[m].z, qr, c[2]); c[3] = fmaf(s[m].w, qr, c[3]);
        }
        // lanes of a warp: (rg % 4) * 8 + cq; fold the 4 row groups of the warp
#pragma unroll
        for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                a[j] += __shfl_xor_sync(0xffffffffu, a[j], off);
                c[j] += __shfl_xor_sync(0xffffffffu, c[j], off);
            }
        }
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        if (lane < 8) {
            float4* r = reinterpret_cast<float4*>(red + warp * 64 + lane * 8);
            r[0] = make_float4(a[0], a[1], a[2], a[3]);
            r[1] = make_float4(c[0], c[1], c[2], c[3]);
        }
        __syncthreads();
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f), C = A;
#pragma unroll
        for (int w = 0; w < kStepThreads / 32; ++w) {
            const float4* r = reinterpret_cast<const float4*>(red + w * 64 + cq() * 8);
            const float4 ra = r[0], rc = r[1];
            A.x += ra.x; A.y += ra.y; A.z += ra.z; A.w += ra.w;
            C.x += rc.x; C.y += rc.y; C.z += rc.z; C.w += rc.w;
        }
        // Explicit roundings (no compiler contraction) keep every caller bitwise identical.
        float4 d, o;
        d.x = __fmul_rn(beta, fmaf(-alpha, A.x, v4.x)); d.y = __fmul_rn(beta, fmaf(-alpha, A.y, v4.y));
        d.z = __fmul_rn(beta, fmaf(-alpha, A.z, v4.z)); d.w = __fmul_rn(beta, fmaf(-alpha, A.w, v4.w));
        o.x = fmaf(d.x, kq, __fmul_rn(alpha, C.x)); o.y = fmaf(d.y, kq, __fmul_rn(alpha, C.y));
        o.z = fmaf(d.z, kq, __fmul_rn(alpha, C.z)); o.w = fmaf(d.w, kq, __fmul_rn(alpha, C.w));
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            s[m].x = fmaf(kr[m], d.x, __fmul_rn(alpha, s[m].x)); s[m].y = fmaf(kr[m], d.y, __fmul_rn(alpha, s[m].y));
            s[m].z = fmaf(kr[m], d.z, __fmul_rn(alpha, s[m].z)); s[m].w = fmaf(kr[m], d.w, __fmul_rn(alpha, s[m].w));
        }
        return o;
    }
};

}  // namespace gdn
