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

// Block-sequential form of the gated delta rule (section 1.2, Step 5) for one
// (sequence, value head, 16-column slice).  For a block of kBM tokens starting
// from state S0, with G_t the running sum of the block's log-decays and
// gamma_t = exp(G_t), unrolling Step 5 gives, per value column j:
//   a_t     = gamma_t (S0^T k_t)_j + sum_{s<t} e^{G_t-G_s} (k_s.k_t) delta_s
//   delta_t = beta_t (v_t - a_t)
//   o_t     = gamma_t (S0^T q_t)_j + sum_{s<=t} e^{G_t-G_s} (k_s.q_t) delta_s
//   S_end   = gamma_last S0 + sum_s e^{G_last-G_s} k_s delta_s^T.
// So the 2*kBM dot products against S0 are independent (one reduction round
// per block instead of per token), the kBM deltas are resolved per column with
// the block's small decay-weighted Gram matrices, and S is rewritten once.
constexpr int kBM = 8;    // tokens per block
constexpr int kBC = 16;   // value columns per CTA
constexpr int kBT = 128;  // threads per CTA

template <typename T, int DK>
__global__ void __launch_bounds__(kBT) block_kernel(const PrefillArgs a, const float* __restrict__ y) {
    constexpr int RG = kBT / (kBC / 2);          // row groups: 16
    constexpr int RPT = DK / RG;                 // rows per thread
    constexpr int NV4 = (2 * DK + kBC) / 4;      // float4 per staged token: q, k, v slice
    constexpr int PER = (kBM * NV4 + kBT - 1) / kBT;
    constexpr int QS = 2 * DK + 4;               // padded row of s_qk (q then k)
    __shared__ __align__(16) float s_qk[kBM][QS];
    __shared__ __align__(16) float s_v[kBM][kBC];
    __shared__ __align__(16) float s_kt[kBM][DK];   // e^{G_last-G_s} k_s
    __shared__ float s_g[kBM], s_b[kBM], s_gam[kBM], s_c[kBM];
    __shared__ float s_Gkk[kBM][kBM], s_Gkq[kBM][kBM];
    __shared__ __align__(16) float s_red[RG][2 * kBM][kBC];
    __shared__ float s_D[2 * kBM][kBC];
    __shared__ float s_dl[kBM][kBC];
    const Geom& g = a.g;
    const int slice = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int hk = h / g.f, col0 = slice * kBC;
    const int tid = threadIdx.x, lane = tid & 31;
    const int cp = tid & (kBC / 2 - 1), rg = tid / (kBC / 2);
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
            for (int c = r * per + tid; c < min(g.D, (r + 1) * per); c += kBT) {
                T* st = cst + ((size_t)n * g.D + c) * (g.K - 1);
                for (int i = 0; i < g.K - 1; ++i) {
                    const int p = len + i;  // index into [old state (K-1), sequence (len)]
                    st[i] = p < g.K - 1 ? st[p] : qkv[(size_t)c * a.T + tb + p - (g.K - 1)];
                }
            }
    }
    if (len <= 0) return;

    float2 S[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) S[r] = *reinterpret_cast<const float2*>(Sg + (size_t)(rg + RG * r) * g.dv + 2 * cp);

    float4 pre[PER];
    float pg = 0.f, pb = 0.f;
    auto fetch = [&](int t0) {
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int idx = tid + j * kBT;
            const int tl = idx / NV4, part = idx - tl * NV4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (idx < kBM * NV4 && t0 + tl < te) {
                const float* row = y + (size_t)(t0 + tl) * g.D;
                const float* src = part < DK / 4 ? row + hk * DK + 4 * part
                                 : part < DK / 2 ? row + g.Hk * DK + hk * DK + 4 * (part - DK / 4)
                                                 : row + 2 * g.Hk * DK + h * g.dv + col0 + 4 * (part - DK / 2);
                v = __ldg(reinterpret_cast<const float4*>(src));
            }
            pre[j] = v;
        }
        const bool ok = tid < kBM && t0 + tid < te;
        pg = ok ? a.gate[(size_t)(t0 + tid) * g.Hv + h] : 0.f;
        pb = ok ? a.beta[(size_t)(t0 + tid) * g.Hv + h] : 0.f;
    };

    fetch(tb);
    for (int t0 = tb; t0 < te; t0 += kBM) {
        const int cnt = min(kBM, te - t0);
        // ---- stage the block ----
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int idx = tid + j * kBT;
            if (idx < kBM * NV4) {
                const int tl = idx / NV4, part = idx - tl * NV4;
                if (part < DK / 2) *reinterpret_cast<float4*>(&s_qk[tl][4 * part]) = pre[j];
                else *reinterpret_cast<float4*>(&s_v[tl][4 * (part - DK / 2)]) = pre[j];
            }
        }
        if (tid < kBM) {
            s_g[tid] = pg;
            s_b[tid] = pb;
        }
        __syncthreads();
        if (t0 + kBM < te) fetch(t0 + kBM);  // next block's loads fly under this block

        // ---- block coefficients ----
        if (tid < 32) {
            float G = lane < kBM ? s_g[lane] : 0.f;  // inclusive prefix sum over the block
#pragma unroll
            for (int off = 1; off < kBM; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, G, off);
                if (lane >= off) G += o;
            }
            const float Glast = __shfl_sync(0xffffffffu, G, kBM - 1);
            if (lane < kBM) {
                s_gam[lane] = expf(G);
                s_c[lane] = expf(Glast - G);
                s_g[lane] = G;  // now the running sum
            }
        }
        {   // Gram entries: 2 threads per (t, s) pair, each half of dk
            const int pair = tid >> 1, half = tid & 1;
            const int t = pair >> 3, s = pair & 7;  // 64 pairs; row 0..3 use kk, the dot of q is done too
            float kk = 0.f, kq = 0.f;
            for (int e = half * (DK / 2); e < (half + 1) * (DK / 2); ++e) {
                const float ks = s_qk[s][DK + e];
                kk = fmaf(ks, s_qk[t][DK + e], kk);
                kq = fmaf(ks, s_qk[t][e], kq);
            }
            kk += __shfl_xor_sync(0xffffffffu, kk, 1);
            kq += __shfl_xor_sync(0xffffffffu, kq, 1);
            __syncthreads();  // s_g holds the running sums
            if (half == 0) {
                const float dec = s <= t ? expf(s_g[t] - s_g[s]) : 0.f;
                s_Gkk[t][s] = s < t ? __fmul_rn(dec, kk) : 0.f;
                s_Gkq[t][s] = __fmul_rn(dec, kq);
            }
        }
        for (int idx = tid; idx < kBM * DK; idx += kBT) {
            const int s = idx / DK, e = idx - s * DK;
            s_kt[s][e] = __fmul_rn(s_c[s], s_qk[s][DK + e]);
        }

        // ---- dot products against the block-start state ----
        float pk[kBM][2], pq[kBM][2];
#pragma unroll
        for (int t = 0; t < kBM; ++t) pk[t][0] = pk[t][1] = pq[t][0] = pq[t][1] = 0.f;
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int row = rg + RG * r;
#pragma unroll
            for (int t = 0; t < kBM; ++t) {
                const float kv = s_qk[t][DK + row], qv = s_qk[t][row];
                pk[t][0] = fmaf(S[r].x, kv, pk[t][0]); pk[t][1] = fmaf(S[r].y, kv, pk[t][1]);
                pq[t][0] = fmaf(S[r].x, qv, pq[t][0]); pq[t][1] = fmaf(S[r].y, qv, pq[t][1]);
            }
        }
#pragma unroll
        for (int t = 0; t < kBM; ++t) {
            *reinterpret_cast<float2*>(&s_red[rg][t][2 * cp]) = make_float2(pk[t][0], pk[t][1]);
            *reinterpret_cast<float2*>(&s_red[rg][kBM + t][2 * cp]) = make_float2(pq[t][0], pq[t][1]);
        }
        __syncthreads();
        for (int o = tid; o < 2 * kBM * kBC; o += kBT) {
            const int vec = o / kBC, col = o - vec * kBC;
            float sum = 0.f;
#pragma unroll
            for (int gq = 0; gq < RG; ++gq) sum += s_red[gq][vec][col];
            s_D[vec][col] = sum;
        }
        __syncthreads();

        // ---- resolve the block's deltas and outputs, one thread per column ----
        if (tid < kBC) {
            const int col = tid;
            float dl[kBM];
#pragma unroll
            for (int t = 0; t < kBM; ++t) {
                float acc = __fmul_rn(s_gam[t], s_D[t][col]);
#pragma unroll
                for (int s2 = 0; s2 < t; ++s2) acc = fmaf(s_Gkk[t][s2], dl[s2], acc);
                dl[t] = t < cnt ? __fmul_rn(s_b[t], s_v[t][col] - acc) : 0.f;
                float o = __fmul_rn(s_gam[t], s_D[kBM + t][col]);
#pragma unroll
                for (int s2 = 0; s2 <= t; ++s2) o = fmaf(s_Gkq[t][s2], dl[s2], o);
                if (t < cnt) a.out[((size_t)(t0 + t) * g.Hv + h) * g.dv + col0 + col] = o;
                s_dl[t][col] = dl[t];
            }
        }
        __syncthreads();

        // ---- S <- gamma_last S + sum_s c_s k_s delta_s^T ----
        const float gl = s_gam[kBM - 1];
        float d0[kBM], d1[kBM];
#pragma unroll
        for (int t = 0; t < kBM; ++t) {
            d0[t] = s_dl[t][2 * cp];
            d1[t] = s_dl[t][2 * cp + 1];
        }
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int row = rg + RG * r;
            float x = __fmul_rn(gl, S[r].x), z = __fmul_rn(gl, S[r].y);
#pragma unroll
            for (int t = 0; t < kBM; ++t) {
                const float kt = s_kt[t][row];
                x = fmaf(kt, d0[t], x);
                z = fmaf(kt, d1[t], z);
            }
            S[r] = make_float2(x, z);
        }
        __syncthreads();  // the block's shared data is consumed
    }
#pragma unroll
    for (int r = 0; r < RPT; ++r) *reinterpret_cast<float2*>(Sg + (size_t)(rg + RG * r) * g.dv + 2 * cp) = S[r];
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
    block_kernel<T, DK><<<dim3(g.dv / kBC, g.Hv, a.N), kBT, 0, stream>>>(a, y);
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
