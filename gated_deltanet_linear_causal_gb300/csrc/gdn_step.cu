// gdn_step.cu -- decode (L = 1, states updated in place) and MTP verify
// (L <= 16 tokens, per-token snapshots) for the Gated DeltaNet layer.
//
// One CTA owns one 32-column slice of one value head's fp32 state S [dk, dv]
// (MNN discussion "MNN Model Support: Qwen3.5", section 1.4: the recurrent
// state [B, H, d_k, d_v]) and runs all five steps of section 1.2 for it:
//   1. conv + SiLU of the 2*dk Q/K channels of its key head and its 32 V
//      channels, from the carried conv state (section 1.4) and the new tokens;
//   2-4. split, reverse GQA (value head h reads key head h / f, section 1.3),
//      L2 norms and the 1/sqrt(dk) scale;
//   5. the gated delta rule, one token at a time, on the slice held in
//      registers (StateSlice::step).
// The slice is read from HBM once and written once per call (decode) or once
// per token (verify snapshots): the kernel is bound by HBM bandwidth.
//
// Decode rewrites the conv state in place.  The Q/K channels of one key head
// are read by all f value heads x (dv/32) slices that share it, so those CTAs
// form one thread-block cluster; each CTA arrives on the cluster barrier once
// it has read the old conv state and waits on it before writing its share of
// the new one.  Verify reads the live states only and needs no cluster.
#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

template <typename T, int DK, bool IN_PLACE>
__global__ void __launch_bounds__(kStepThreads) step_kernel(const StepArgs a, const GateParams gp) {
    extern __shared__ float4 smem_f4[];
    float* sm = reinterpret_cast<float*>(smem_f4);
    const Geom& g = a.g;
    const int L = a.L;
    constexpr int NCH = 2 * DK + kSliceCols;  // channels this CTA convolves
    float* qk_s = sm;                                   // [L][2*DK]: q then k
    float* v_s = qk_s + L * 2 * DK;                     // [L][32]
    float* nred = v_s + L * kSliceCols;                 // [4][3*kMaxVerify]
    float* coef = nred + 4 * 3 * kMaxVerify;            // [kMaxVerify][3]: fq, fk, k.q
    float* red = coef + 3 * kMaxVerify;                 // [2][4*64]
    T* cs_new = reinterpret_cast<T*>(red + 2 * 4 * 64);  // IN_PLACE: [NCH][K-1]

    const int slice = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int hk = h / g.f;
    const int col0 = slice * kSliceCols;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const T* qkv = static_cast<const T*>(a.qkv);
    const T* w = static_cast<const T*>(a.w);
    const T* cin = static_cast<const T*>(a.conv_in);

    // Issue the state loads first; the prologue below runs under their latency.
    StateSlice<DK> S;
    S.load(a.S_in + (size_t)(b * g.Hv + h) * DK * g.dv + col0, g.dv);

    // ---- step 1: causal conv + SiLU of the CTA's channels, all L tokens ----
    const bool owns_qk = (h % g.f == 0) && slice == 0;  // verify: writes Q/K conv snapshots
    for (int ch = tid; ch < NCH; ch += kStepThreads) {
        int c;
        if (ch < DK) c = hk * DK + ch;
        else if (ch < 2 * DK) c = g.Hk * DK + hk * DK + (ch - DK);
        else c = 2 * g.Hk * DK + h * g.dv + col0 + (ch - 2 * DK);
        ConvWindow<T> win;
        win.load(cin + ((size_t)b * g.D + c) * (g.K - 1), w + (size_t)c * g.K, g.K);
        const T* x = qkv + ((size_t)b * g.D + c) * L;
        for (int t = 0; t < L; ++t) {
            const float y = win.push(x[t]);
            if (ch < 2 * DK) qk_s[t * 2 * DK + ch] = y;
            else v_s[t * kSliceCols + (ch - 2 * DK)] = y;
            if (!IN_PLACE && (ch >= 2 * DK || owns_qk))
                win.store_state(static_cast<T*>(a.conv_out) + (((size_t)b * L + t) * g.D + c) * (g.K - 1), g.K);
        }
        if (IN_PLACE) win.store_state(cs_new + ch * (g.K - 1), g.K);
    }
    __syncthreads();
    if (IN_PLACE) cluster_arrive_release();  // this CTA is done reading the old conv state

    // ---- steps 3-4: per-token L2 norms of q and k, 1/sqrt(dk) on q, and k.q ----
    for (int t = 0; t < L; ++t) {
        float sq = 0.f, sk = 0.f, skq = 0.f;
        for (int i = tid; i < DK; i += kStepThreads) {
            const float qv = qk_s[t * 2 * DK + i], kv = qk_s[t * 2 * DK + DK + i];
            sq = fmaf(qv, qv, sq);
            sk = fmaf(kv, kv, sk);
            skq = fmaf(kv, qv, skq);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, off);
            sk += __shfl_xor_sync(0xffffffffu, sk, off);
            skq += __shfl_xor_sync(0xffffffffu, skq, off);
        }
        if (lane == 0) {
            nred[warp * 3 * kMaxVerify + 3 * t + 0] = sq;
            nred[warp * 3 * kMaxVerify + 3 * t + 1] = sk;
            nred[warp * 3 * kMaxVerify + 3 * t + 2] = skq;
        }
    }
    __syncthreads();
    if (tid < L) {
        float sq = 0.f, sk = 0.f, skq = 0.f;
#pragma unroll
        for (int wi = 0; wi < kStepThreads / 32; ++wi) {
            sq += nred[wi * 3 * kMaxVerify + 3 * tid + 0];
            sk += nred[wi * 3 * kMaxVerify + 3 * tid + 1];
            skq += nred[wi * 3 * kMaxVerify + 3 * tid + 2];
        }
        const float rq = g.use_l2 ? rsqrtf(sq + g.eps) : 1.f;
        const float rk = g.use_l2 ? rsqrtf(sk + g.eps) : 1.f;
        const float fq = __fmul_rn(g.q_scale, rq);
        coef[3 * tid + 0] = fq;
        coef[3 * tid + 1] = rk;
        coef[3 * tid + 2] = __fmul_rn(__fmul_rn(skq, fq), rk);
    }
    __syncthreads();
    for (int idx = tid; idx < L * 2 * DK; idx += kStepThreads) {
        const int t = idx / (2 * DK), i = idx - t * 2 * DK;
        qk_s[idx] = __fmul_rn(qk_s[idx], coef[3 * t + (i < DK ? 0 : 1)]);
    }
    __syncthreads();

    // ---- step 5: gated delta rule, token by token ----
    const int cq = StateSlice<DK>::cq(), rg = StateSlice<DK>::rg();
    for (int t = 0; t < L; ++t) {
        const size_t gi = ((size_t)b * L + t) * g.Hv + h;
        const float alpha = expf(gate_of(gp.A_log, gp.dt_bias, a.gate[gi], h));
        const float bt = beta_of(gp.A_log, a.beta[gi]);
        const float4 v4 = *reinterpret_cast<const float4*>(v_s + t * kSliceCols + 4 * cq);
        const float4 o = S.step(qk_s + t * 2 * DK + DK, qk_s + t * 2 * DK, v4, alpha, bt, coef[3 * t + 2],
                                red + (t & 1) * 256);
        if (rg == 0) st_stream(a.out + gi * g.dv + col0 + 4 * cq, o);
        if (!IN_PLACE) S.store(a.S_out + (gi * DK) * g.dv + col0, g.dv);
    }
    if (IN_PLACE) {
        S.store(a.S_out + (size_t)(b * g.Hv + h) * DK * g.dv + col0, g.dv);
        // New conv state: wait until every CTA sharing the key head has read the old one.
        cluster_wait_acquire();
        const int nrank = g.f * gridDim.x;
        const int rank = (h % g.f) * gridDim.x + slice;
        const int per = (2 * DK + nrank - 1) / nrank;
        const int lo = rank * per, hi = min(2 * DK, lo + per);
        T* cout = static_cast<T*>(a.conv_out);
        for (int ch = lo + tid; ch < hi; ch += kStepThreads) {
            const int c = ch < DK ? hk * DK + ch : g.Hk * DK + hk * DK + (ch - DK);
            for (int i = 0; i < g.K - 1; ++i)
                cout[((size_t)b * g.D + c) * (g.K - 1) + i] = cs_new[ch * (g.K - 1) + i];
        }
        for (int ch = 2 * DK + tid; ch < NCH; ch += kStepThreads) {
            const int c = 2 * g.Hk * DK + h * g.dv + col0 + (ch - 2 * DK);
            for (int i = 0; i < g.K - 1; ++i)
                cout[((size_t)b * g.D + c) * (g.K - 1) + i] = cs_new[ch * (g.K - 1) + i];
        }
    }
}

template <typename T, int DK, bool IN_PLACE>
cudaError_t launch_step_t(const StepArgs& a, const GateParams& gp, cudaStream_t stream) {
    const Geom& g = a.g;
    const int NS = g.dv / kSliceCols;
    const size_t floats = (size_t)a.L * (2 * DK + kSliceCols) + 4 * 3 * kMaxVerify + 3 * kMaxVerify + 2 * 4 * 64;
    const size_t smem = floats * sizeof(float) + (IN_PLACE ? (size_t)(2 * DK + kSliceCols) * (g.K - 1) * sizeof(T) : 0);
    auto kern = step_kernel<T, DK, IN_PLACE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(NS, g.Hv, a.B);
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (IN_PLACE) {
        const int csize = NS * g.f;
        if (csize > 8) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = NS;
        attr[0].val.clusterDim.y = g.f;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a, gp);
}

template <bool IN_PLACE>
cudaError_t dispatch_step(const StepArgs& a, const GateParams& gp, cudaStream_t s) {
    if (a.g.io_bf16) {
        switch (a.g.dk) {
            case 32: return launch_step_t<__nv_bfloat16, 32, IN_PLACE>(a, gp, s);
            case 64: return launch_step_t<__nv_bfloat16, 64, IN_PLACE>(a, gp, s);
            case 128: return launch_step_t<__nv_bfloat16, 128, IN_PLACE>(a, gp, s);
            case 256: return launch_step_t<__nv_bfloat16, 256, IN_PLACE>(a, gp, s);
        }
    } else {
        switch (a.g.dk) {
            case 32: return launch_step_t<float, 32, IN_PLACE>(a, gp, s);
            case 64: return launch_step_t<float, 64, IN_PLACE>(a, gp, s);
            case 128: return launch_step_t<float, 128, IN_PLACE>(a, gp, s);
            case 256: return launch_step_t<float, 256, IN_PLACE>(a, gp, s);
        }
    }
    return cudaErrorInvalidValue;
}

// ---- verify commit: copy snapshot accepted-1 into the live states ----------------
__global__ void commit_kernel(const CommitArgs a) {
    const int b = blockIdx.y;
    const int acc = a.accepted[b];
    if (acc < 0 || acc > a.L) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && a.status) atomicExch(a.status, 10 /* GDN_ERR_RANGE */);
        return;
    }
    if (acc == 0) return;
    const size_t snap = (size_t)b * a.L + (acc - 1);
    const float4* src = reinterpret_cast<const float4*>(a.ssm_snap + snap * a.ssm_floats);
    float4* dst = reinterpret_cast<float4*>(a.ssm_state + (size_t)b * a.ssm_floats);
    const size_t n4 = a.ssm_floats / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = __ldcs(src + i);
    const unsigned char* cs = static_cast<const unsigned char*>(a.conv_snap) + snap * a.conv_bytes;
    unsigned char* cd = static_cast<unsigned char*>(a.conv_state) + (size_t)b * a.conv_bytes;
    if (a.conv_vec16) {
        const uint4* s4 = reinterpret_cast<const uint4*>(cs);
        uint4* d4 = reinterpret_cast<uint4*>(cd);
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.conv_bytes / 16;
             i += (size_t)gridDim.x * blockDim.x)
            d4[i] = s4[i];
    } else {
        const uint16_t* s2 = reinterpret_cast<const uint16_t*>(cs);
        uint16_t* d2 = reinterpret_cast<uint16_t*>(cd);
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.conv_bytes / 2;
             i += (size_t)gridDim.x * blockDim.x)
            d2[i] = s2[i];
    }
}

// Zero `bytes` bytes at p: 16-byte stores over the aligned middle, byte stores
// over the unaligned head and tail (each under 16 bytes).
__global__ void zero_kernel(unsigned char* p, size_t head, size_t n16, size_t tail) {
    uint4* mid = reinterpret_cast<uint4*>(p + head);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
        mid[i] = make_uint4(0u, 0u, 0u, 0u);
    if (blockIdx.x == 0) {
        if (threadIdx.x < head) p[threadIdx.x] = 0;
        if (threadIdx.x < tail) p[head + n16 * 16 + threadIdx.x] = 0;
    }
}

}  // namespace

bool slice_step_supported(const Geom& g) { return (g.dv / kSliceCols) * g.f <= 16; }

cudaError_t launch_step(const StepArgs& a, const GateParams& gp, bool in_place, cudaStream_t stream,
                        const NormParams& np) {
    int ns = 0;
    size_t smem = 0;
    if (stream_step_supported(a, &ns, &smem)) return launch_stream_step(a, gp, in_place, stream, np);
    if (np.z) return cudaErrorInvalidValue;  // the fused norm lives in the streaming kernel only
    return in_place ? dispatch_step<true>(a, gp, stream) : dispatch_step<false>(a, gp, stream);
}

cudaError_t launch_commit(const CommitArgs& a, cudaStream_t stream) {
    const int per_seq_blocks = (int)std::min<size_t>(64, (a.ssm_floats / 4 + 255) / 256 + 1);
    commit_kernel<<<dim3(per_seq_blocks, a.B), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t stream) {
    if (bytes == 0) return cudaSuccess;
    unsigned char* c = static_cast<unsigned char*>(p);
    size_t head = (16 - (reinterpret_cast<uintptr_t>(c) & 15)) & 15;
    if (head > bytes) head = bytes;
    const size_t n16 = (bytes - head) / 16, tail = bytes - head - n16 * 16;
    const int blocks = (int)std::max<size_t>(1, std::min<size_t>(152 * 8, (n16 + 255) / 256));
    zero_kernel<<<blocks, 256, 0, stream>>>(c, head, n16, tail);
    return cudaGetLastError();
}

}  // namespace gdn
