// gdn_prefill.cu -- prefill over cu_seqlens-packed sequences, resident form.
//
// Two launches:
//   prep      steps 1-4 of the MNN "Qwen3.5" page, section 1.2, for every packed
//             token: causal conv + SiLU from the raw qkv [D, T] (channel-major, as
//             the page lays out qkv [B, D, L]) with each sequence's carried conv
//             state (section 1.4), then per-head L2 norms and the 1/sqrt(dk)
//             scale.  Writes token-major fp32 rows y [T, D] to the workspace.
//   resident  step 5, the gated delta rule: one CTA per (sequence, value head,
//             32-column slice) keeps its slice of S in registers across the whole
//             sequence (StateSlice::step, the same arithmetic as decode), with the
//             next 16 (8 for dk=256) tokens' q/k/v prefetched into registers while the current
//             16 run from shared memory.  It also writes each sequence's new conv
//             state: the prep launch has finished reading the old one by then.
// The resident form is serial in the sequence length: each token waits on the
// previous one's reductions over dk.
#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kPrepTokens = 32;
constexpr int kPrepThreads = 256;

// Sequence of packed token t: the last n with cu[n] <= t (empty sequences skipped).
__device__ __forceinline__ int seq_of(const int32_t* cu, int N, int t) {
    int lo = 0, hi = N;  // cu[lo] <= t < cu[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid;
        else hi = mid;
    }
    return lo;
}

template <typename T>
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const PrefillArgs a, float* __restrict__ y) {
    extern __shared__ float4 smem_f4[];
    float* tile = reinterpret_cast<float*>(smem_f4);  // [nch][kPrepTokens + 1]
    __shared__ int s_seq[kPrepTokens], s_pos[kPrepTokens], s_start[kPrepTokens];
    __shared__ float s_part[kPrepThreads / kPrepTokens][kPrepTokens];
    __shared__ float s_fac[kPrepTokens];
    const Geom& g = a.g;
    const int t0 = blockIdx.x * kPrepTokens;
    const int grp = blockIdx.y;
    int cbase, nch, kind;  // kind 0: q head, 1: k head, 2: v group of 32 channels
    if (grp < g.Hk) { cbase = grp * g.dk; nch = g.dk; kind = 0; }
    else if (grp < 2 * g.Hk) { cbase = grp * g.dk; nch = g.dk; kind = 1; }
    else { cbase = 2 * g.Hk * g.dk + (grp - 2 * g.Hk) * kSliceCols; nch = kSliceCols; kind = 2; }
    const int tid = threadIdx.x;
    if (tid < kPrepTokens) {
        const int t = t0 + tid;
        if (t < a.T) {
            const int n = seq_of(a.cu, a.N, t);
            s_seq[tid] = n;
            s_start[tid] = a.cu[n];
            s_pos[tid] = t - a.cu[n];
        }
    }
    __syncthreads();
    const T* qkv = static_cast<const T*>(a.qkv);
    const T* w = static_cast<const T*>(a.w);
    const T* cst = static_cast<const T*>(a.conv_state);
    const int K = g.K;
    for (int idx = tid; idx < nch * kPrepTokens; idx += kPrepThreads) {
        const int cl = idx / kPrepTokens, tl = idx - cl * kPrepTokens;
        const int t = t0 + tl;
        float v = 0.f;
        if (t < a.T) {
            const int c = cbase + cl, n = s_seq[tl], pos = s_pos[tl], st = s_start[tl];
            float acc = 0.f;
            for (int j = 0; j < K; ++j) {
                const int p = pos - (K - 1) + j;  // position in the sequence
                const T xv = p >= 0 ? qkv[(size_t)c * a.T + st + p] : cst[((size_t)n * g.D + c) * (K - 1) + (pos + j)];
                acc = fmaf(to_f32(w[(size_t)c * K + j]), to_f32(xv), acc);
            }
            v = silu(acc);
        }
        tile[cl * (kPrepTokens + 1) + tl] = v;
    }
    __syncthreads();
    if (kind < 2) {
        const int tl = tid % kPrepTokens, part = tid / kPrepTokens;
        float sum = 0.f;
        for (int cl = part; cl < nch; cl += kPrepThreads / kPrepTokens) {
            const float v = tile[cl * (kPrepTokens + 1) + tl];
            sum = fmaf(v, v, sum);
        }
        s_part[part][tl] = sum;
        __syncthreads();
        if (tid < kPrepTokens) {
            float tot = 0.f;
            for (int p = 0; p < kPrepThreads / kPrepTokens; ++p) tot += s_part[p][tid];
            const float r = g.use_l2 ? rsqrtf(tot + g.eps) : 1.f;
            s_fac[tid] = kind == 0 ? __fmul_rn(g.q_scale, r) : r;
        }
    } else if (tid < kPrepTokens) {
        s_fac[tid] = 1.f;
    }
    __syncthreads();
    for (int idx = tid; idx < nch * kPrepTokens; idx += kPrepThreads) {
        const int tl = idx / nch, cl = idx - tl * nch;
        const int t = t0 + tl;
        if (t < a.T) y[(size_t)t * g.D + cbase + cl] = __fmul_rn(tile[cl * (kPrepTokens + 1) + tl], s_fac[tl]);
    }
}

template <typename T, int DK>
__global__ void __launch_bounds__(kStepThreads) resident_kernel(const PrefillArgs a, const float* __restrict__ y) {
    constexpr int kResTokens = DK <= 128 ? 16 : 8;  // tokens staged per round (static smem < 48 KB)
    constexpr int ROW = 2 * DK + kSliceCols + 4;      // q, k, v slice, alpha, beta, k.q, pad
    constexpr int NV4 = (2 * DK + kSliceCols) / 4;     // float4 per staged token
    constexpr int PER = (kResTokens * NV4 + kStepThreads - 1) / kStepThreads;
    __shared__ __align__(16) float buf[2][kResTokens][ROW];
    __shared__ __align__(16) float red[2][4 * 64];
    const Geom& g = a.g;
    const int slice = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int hk = h / g.f, col0 = slice * kSliceCols;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tb = a.cu[n], te = a.cu[n + 1];
    const int len = te - tb;
    float* Sg = a.ssm_state + (size_t)(n * g.Hv + h) * DK * g.dv + col0;

    // New conv state of sequence n: channels split over the CTAs of the sequence.
    {
        const int nct = gridDim.x * gridDim.y, r = h * gridDim.x + slice;
        const int per = (g.D + nct - 1) / nct;
        T* cst = static_cast<T*>(a.conv_state);
        const T* qkv = static_cast<const T*>(a.qkv);
        if (len > 0)
            for (int c = r * per + tid; c < min(g.D, (r + 1) * per); c += kStepThreads) {
                T* s = cst + ((size_t)n * g.D + c) * (g.K - 1);
                for (int i = 0; i < g.K - 1; ++i) {
                    const int p = len + i;  // index into [old state (K-1), sequence (len)]
                    s[i] = p < g.K - 1 ? s[p] : qkv[(size_t)c * a.T + tb + p - (g.K - 1)];
                }
            }
    }
    if (len <= 0) return;

    StateSlice<DK> S;
    S.load(Sg, g.dv);

    float4 pre[PER];
    auto fetch = [&](int t0) {
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int idx = tid + j * kStepThreads;
            const int tl = idx / NV4, part = idx - tl * NV4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (idx < kResTokens * NV4 && t0 + tl < te) {
                const float* row = y + (size_t)(t0 + tl) * g.D;
                const float* src = part < DK / 4 ? row + hk * DK + 4 * part
                                 : part < DK / 2 ? row + g.Hk * DK + hk * DK + 4 * (part - DK / 4)
                                                 : row + 2 * g.Hk * DK + h * g.dv + col0 + 4 * (part - DK / 2);
                v = __ldg(reinterpret_cast<const float4*>(src));
            }
            pre[j] = v;
        }
    };
    auto stage = [&](int t0, int bsel) {
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int idx = tid + j * kStepThreads;
            if (idx < kResTokens * NV4) {
                const int tl = idx / NV4, part = idx - tl * NV4;
                *reinterpret_cast<float4*>(&buf[bsel][tl][4 * part]) = pre[j];
            }
        }
        __syncthreads();
        // per-token scalars: alpha = exp(g), beta, k.q (warp w handles tokens w, w+4, ...)
        for (int tl = warp; tl < kResTokens; tl += kStepThreads / 32) {
            float kq = 0.f;
            for (int i = lane; i < DK; i += 32) kq = fmaf(buf[bsel][tl][DK + i], buf[bsel][tl][i], kq);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
            if (lane == 0) {
                const int t = t0 + tl;
                const bool ok = t < te;
                buf[bsel][tl][2 * DK + kSliceCols + 0] = ok ? expf(a.gate[(size_t)t * g.Hv + h]) : 1.f;
                buf[bsel][tl][2 * DK + kSliceCols + 1] = ok ? a.beta[(size_t)t * g.Hv + h] : 0.f;
                buf[bsel][tl][2 * DK + kSliceCols + 2] = kq;
            }
        }
        __syncthreads();
    };

    const int cq = StateSlice<DK>::cq(), rg = StateSlice<DK>::rg();
    fetch(tb);
    stage(tb, 0);
    int bsel = 0;
    for (int t0 = tb; t0 < te; t0 += kResTokens) {
        const bool more = t0 + kResTokens < te;
        if (more) fetch(t0 + kResTokens);
        const int cnt = min(kResTokens, te - t0);
        for (int tl = 0; tl < cnt; ++tl) {
            const float* row = buf[bsel][tl];
            const float4 v4 = *reinterpret_cast<const float4*>(row + 2 * DK + 4 * cq);
            const float4 o = S.step(row + DK, row, v4, row[2 * DK + kSliceCols], row[2 * DK + kSliceCols + 1],
                                    row[2 * DK + kSliceCols + 2], red[tl & 1]);
            if (rg == 0) st_stream(a.out + ((size_t)(t0 + tl) * g.Hv + h) * g.dv + col0 + 4 * cq, o);
        }
        if (more) {
            bsel ^= 1;
            stage(t0 + kResTokens, bsel);
        }
    }
    S.store(Sg, g.dv);
}

template <typename T, int DK>
cudaError_t launch_resident_t(const PrefillArgs& a, cudaStream_t stream) {
    const Geom& g = a.g;
    float* y = static_cast<float*>(a.ws);
    const int ngrp = 2 * g.Hk + g.Hv * (g.dv / kSliceCols);
    const size_t prep_smem = (size_t)std::max(g.dk, kSliceCols) * (kPrepTokens + 1) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(prep_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prep_smem);
    if (e != cudaSuccess) return e;
    prep_kernel<T><<<dim3((a.T + kPrepTokens - 1) / kPrepTokens, ngrp), kPrepThreads, prep_smem, stream>>>(a, y);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    resident_kernel<T, DK><<<dim3(g.dv / kSliceCols, g.Hv, a.N), kStepThreads, 0, stream>>>(a, y);
    return cudaGetLastError();
}

}  // namespace

size_t prefill_resident_workspace(const Geom& g, int /*N*/, long long T) {
    return (size_t)T * g.D * sizeof(float);
}

cudaError_t launch_prefill_resident(const PrefillArgs& a, cudaStream_t s) {
    if (a.g.io_bf16) {
        switch (a.g.dk) {
            case 32: return launch_resident_t<__nv_bfloat16, 32>(a, s);
            case 64: return launch_resident_t<__nv_bfloat16, 64>(a, s);
            case 128: return launch_resident_t<__nv_bfloat16, 128>(a, s);
            case 256: return launch_resident_t<__nv_bfloat16, 256>(a, s);
        }
    } else {
        switch (a.g.dk) {
            case 32: return launch_resident_t<float, 32>(a, s);
            case 64: return launch_resident_t<float, 64>(a, s);
            case 128: return launch_resident_t<float, 128>(a, s);
            case 256: return launch_resident_t<float, 256>(a, s);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdn
