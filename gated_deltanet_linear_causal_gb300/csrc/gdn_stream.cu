// gdn_stream.cu -- decode and MTP verify as one persistent, TMA-fed kernel.
//
// Work item = (sequence b, key head hk): the f = Hv/Hk value heads that share
// key head hk (reverse GQA, MNN "Qwen3.5" page, section 1.3).  One CTA per SM
// walks its items; for each it
//   1. convolves + SiLUs the 2*dk Q/K channels of hk and the f*dv V channels of
//      its value heads from the carried conv state (section 1.2 Step 1, section
//      1.4), L2-normalises q and k and scales q (Steps 2-4), and rewrites the
//      conv state in place (decode) or writes its per-token snapshots (verify);
//      because an item owns all channels it reads, no other CTA touches them;
//   2. streams the item's state tiles (dk rows x 128 columns of one value head)
//      through a ring of shared-memory stages filled by bulk asynchronous copies
//      (cp.async.bulk + mbarrier), nstage tiles ahead of the compute;
//   3. runs the gated delta rule (section 1.2 Step 5) on each tile held in
//      registers, one token at a time, and stores the new state (decode, in
//      place) or every per-token snapshot (verify) straight from registers.
// Every byte of state is read from HBM once and written once per token written.
// Thread (warp w, lane l) of the 8-warp CTA holds columns 4l..4l+3 of rows
// w + 8m; the reductions over dk go through shared memory in a fixed order, so
// decode and verify produce identical bits for identical inputs.
#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tma.cuh"

namespace gdn {

static __device__ int32_t g_stream_error;  // set to GDN_ERR_DEVICE_TIMEOUT (7) by a stuck wait

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTileCols = 128;

template <int DK>
struct Tile {
    static constexpr int RPT = DK / kWarps;  // rows per thread
    float4 s[RPT];

    __device__ __forceinline__ static int row(int m) { return (threadIdx.x >> 5) + kWarps * m; }
    __device__ __forceinline__ static int col4() { return 4 * (threadIdx.x & 31); }

    __device__ __forceinline__ void load_smem(const float* stage) {
#pragma unroll
        for (int m = 0; m < RPT; ++m) s[m] = *reinterpret_cast<const float4*>(stage + row(m) * kTileCols + col4());
    }
    __device__ __forceinline__ void store_global(float* base, int dv) const {
#pragma unroll
        for (int m = 0; m < RPT; ++m) st_stream(base + (size_t)row(m) * dv + col4(), s[m]);
    }

    // One token of the gated delta rule on the tile (same algebra as
    // StateSlice::step): a = (alpha S)^T k, delta = beta (v - a),
    // S' = alpha S + k delta^T, o = alpha S^T q + delta (k.q).
    // red: [kWarps][256] shared floats, not in use by any thread.
    __device__ __forceinline__ float4 step(const float* k, const float* q, float4 v4, float alpha, float beta,
                                           float kq, float* red) {
        float a[4] = {0.f, 0.f, 0.f, 0.f}, c[4] = {0.f, 0.f, 0.f, 0.f};
        float kr[RPT];
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            kr[m] = k[row(m)];
            const float qr = q[row(m)];
            a[0] = fmaf(s[m].x, kr[m], a[0]); a[1] = fmaf(s[m].y, kr[m], a[1]);
            a[2] = fmaf(s[m].z, kr[m], a[2]); a[3] = fmaf(s[m].w, kr[m], a[3]);
            c[0] = fmaf(s[m].x, qr, c[0]); c[1] = fmaf(s[m].y, qr, c[1]);
            c[2] = fmaf(s[m].z, qr, c[2]); c[3] = fmaf(s[m].w, qr, c[3]);
        }
        const int warp = threadIdx.x >> 5;
        *reinterpret_cast<float4*>(red + warp * 256 + col4()) = make_float4(a[0], a[1], a[2], a[3]);
        *reinterpret_cast<float4*>(red + warp * 256 + 128 + col4()) = make_float4(c[0], c[1], c[2], c[3]);
        __syncthreads();
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f), C = A;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float4 ra = *reinterpret_cast<const float4*>(red + w * 256 + col4());
            const float4 rc = *reinterpret_cast<const float4*>(red + w * 256 + 128 + col4());
            A.x += ra.x; A.y += ra.y; A.z += ra.z; A.w += ra.w;
            C.x += rc.x; C.y += rc.y; C.z += rc.z; C.w += rc.w;
        }
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

struct Smem {
    float* stage;  // [nstage][DK * 128]
    float* qk;     // [L][2*DK]  q then k
    float* v;      // [L][f*dv]
    float* coef;   // [kMaxVerify][3]  q factor, k factor, k.q
    float* nred;   // [kWarps][3*kMaxVerify]
    float* red;    // [2][kWarps][256]
    uint64_t* full;  // [nstage]
};

__host__ __device__ inline size_t smem_floats(int DK, int nstage, int L, int f, int dv) {
    return (size_t)nstage * DK * kTileCols + (size_t)L * 2 * DK + (size_t)L * f * dv + 3 * kMaxVerify +
           kWarps * 3 * kMaxVerify + 2 * kWarps * 256;
}

template <typename T, int DK, bool IN_PLACE>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(const StepArgs a, const int nstage) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ int s_abort;
    const Geom& g = a.g;
    const int L = a.L;
    constexpr int TILE = DK * kTileCols;
    const int nsl = g.dv / kTileCols;  // column tiles per value head
    const int tpi = g.f * nsl;         // tiles per item
    const int nitems = a.B * g.Hk;
    const int my_items = (nitems - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    const int ntiles = my_items * tpi;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    Smem sm;
    sm.stage = reinterpret_cast<float*>(smem_raw);
    sm.qk = sm.stage + (size_t)nstage * TILE;
    sm.v = sm.qk + L * 2 * DK;
    sm.coef = sm.v + L * g.f * g.dv;
    sm.nred = sm.coef + 3 * kMaxVerify;
    sm.red = sm.nred + kWarps * 3 * kMaxVerify;
    sm.full = reinterpret_cast<uint64_t*>(sm.red + 2 * kWarps * 256);

    const T* qkv = static_cast<const T*>(a.qkv);
    const T* w = static_cast<const T*>(a.w);
    const T* cin = static_cast<const T*>(a.conv_in);
    T* cout = static_cast<T*>(a.conv_out);

    // Issue the bulk copies of tile j (warp 0 only).
    auto issue = [&](int j) {
        const int item = (int)blockIdx.x + (j / tpi) * (int)gridDim.x;
        const int r = j % tpi;
        const int b = item / g.Hk, hk = item % g.Hk;
        const int h = hk * g.f + r / nsl, col0 = (r % nsl) * kTileCols;
        const float* src = a.S_in + ((size_t)(b * g.Hv + h) * DK) * g.dv + col0;
        float* dst = sm.stage + (size_t)(j % nstage) * TILE;
        uint64_t* bar = sm.full + (j % nstage);
        if (nsl == 1) {
            if (lane == 0) {
                mbar_arrive_expect_tx(bar, TILE * 4);
                bulk_g2s(dst, src, TILE * 4, bar);
            }
        } else {
            if (lane == 0) mbar_arrive_expect_tx(bar, TILE * 4);
            __syncwarp();
            for (int row = lane; row < DK; row += 32)
                bulk_g2s(dst + row * kTileCols, src + (size_t)row * g.dv, kTileCols * 4, bar);
        }
    };

    if (tid == 0) {
        for (int s = 0; s < nstage; ++s) mbar_init(sm.full + s, 1);
        fence_mbar_init();
        s_abort = 0;
    }
    __syncthreads();
    if (warp == 0)
        for (int j = 0; j < min(nstage, ntiles); ++j) issue(j);

    for (int i = 0; i < my_items; ++i) {
        const int item = (int)blockIdx.x + i * (int)gridDim.x;
        const int b = item / g.Hk, hk = item % g.Hk;

        // ---- steps 1-4 for the item's channels (runs under the tile loads) ----
        const int nch = 2 * DK + g.f * g.dv;
        for (int ch = tid; ch < nch; ch += kThreads) {
            int c;
            if (ch < DK) c = hk * DK + ch;
            else if (ch < 2 * DK) c = g.Hk * DK + hk * DK + (ch - DK);
            else c = 2 * g.Hk * DK + hk * g.f * g.dv + (ch - 2 * DK);
            ConvWindow<T> win;
            win.load(cin + ((size_t)b * g.D + c) * (g.K - 1), w + (size_t)c * g.K, g.K);
            const T* x = qkv + ((size_t)b * g.D + c) * L;
            for (int t = 0; t < L; ++t) {
                const float y = win.push(x[t]);
                if (ch < 2 * DK) sm.qk[t * 2 * DK + ch] = y;
                else sm.v[t * g.f * g.dv + (ch - 2 * DK)] = y;
                if (!IN_PLACE) {
                    T* snap = cout + (((size_t)b * L + t) * g.D + c) * (g.K - 1);
                    for (int e = 0; e < g.K - 1; ++e) snap[e] = win.state(e, g.K);
                }
            }
            if (IN_PLACE) {
                T* st = cout + ((size_t)b * g.D + c) * (g.K - 1);
                for (int e = 0; e < g.K - 1; ++e) st[e] = win.state(e, g.K);
            }
        }
        __syncthreads();
        for (int t = 0; t < L; ++t) {
            float sq = 0.f, sk = 0.f, skq = 0.f;
            for (int e = tid; e < DK; e += kThreads) {
                const float qv = sm.qk[t * 2 * DK + e], kv = sm.qk[t * 2 * DK + DK + e];
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
                sm.nred[warp * 3 * kMaxVerify + 3 * t + 0] = sq;
                sm.nred[warp * 3 * kMaxVerify + 3 * t + 1] = sk;
                sm.nred[warp * 3 * kMaxVerify + 3 * t + 2] = skq;
            }
        }
        __syncthreads();
        if (tid < L) {
            float sq = 0.f, sk = 0.f, skq = 0.f;
#pragma unroll
            for (int wi = 0; wi < kWarps; ++wi) {
                sq += sm.nred[wi * 3 * kMaxVerify + 3 * tid + 0];
                sk += sm.nred[wi * 3 * kMaxVerify + 3 * tid + 1];
                skq += sm.nred[wi * 3 * kMaxVerify + 3 * tid + 2];
            }
            const float rq = g.use_l2 ? rsqrtf(sq + g.eps) : 1.f;
            const float rk = g.use_l2 ? rsqrtf(sk + g.eps) : 1.f;
            const float fq = __fmul_rn(g.q_scale, rq);
            sm.coef[3 * tid + 0] = fq;
            sm.coef[3 * tid + 1] = rk;
            sm.coef[3 * tid + 2] = __fmul_rn(__fmul_rn(skq, fq), rk);
        }
        __syncthreads();
        for (int idx = tid; idx < L * 2 * DK; idx += kThreads) {
            const int t = idx / (2 * DK), e = idx - t * 2 * DK;
            sm.qk[idx] = __fmul_rn(sm.qk[idx], sm.coef[3 * t + (e < DK ? 0 : 1)]);
        }
        __syncthreads();

        // ---- step 5 over the item's tiles ----
        for (int r = 0; r < tpi; ++r) {
            const int j = i * tpi + r;
            const int hl = r / nsl, col0 = (r % nsl) * kTileCols;
            const int h = hk * g.f + hl;
            Tile<DK> S;
            const bool ok = mbar_wait_bounded(sm.full + (j % nstage), (uint32_t)((j / nstage) & 1));
            if (!ok) s_abort = 1;
            S.load_smem(sm.stage + (size_t)(j % nstage) * TILE);
            __syncthreads();  // the stage is free again; s_abort is visible
            if (s_abort) {
                if (tid == 0) {
                    flag_device_error(&g_stream_error, 7);
                    // let the copies still in flight land before the CTA exits
                    for (int jj = j + 1; jj < min(ntiles, j + nstage); ++jj)
                        mbar_wait_bounded(sm.full + (jj % nstage), (uint32_t)((jj / nstage) & 1));
                }
                return;
            }
            if (warp == 0 && j + nstage < ntiles) {
                fence_proxy_async_smem();
                issue(j + nstage);
            }
            for (int t = 0; t < L; ++t) {
                const size_t gi = ((size_t)b * L + t) * g.Hv + h;
                const float alpha = expf(a.gate[gi]);
                const float bt = a.beta[gi];
                const float4 v4 =
                    *reinterpret_cast<const float4*>(sm.v + t * g.f * g.dv + hl * g.dv + col0 + Tile<DK>::col4());
                const float4 o = S.step(sm.qk + t * 2 * DK + DK, sm.qk + t * 2 * DK, v4, alpha, bt,
                                        sm.coef[3 * t + 2], sm.red + (t & 1) * kWarps * 256);
                if (warp == 0) st_stream(a.out + gi * g.dv + col0 + Tile<DK>::col4(), o);
                if (!IN_PLACE) S.store_global(a.S_out + (gi * DK) * g.dv + col0, g.dv);
            }
            if (IN_PLACE) S.store_global(a.S_out + ((size_t)(b * g.Hv + h) * DK) * g.dv + col0, g.dv);
        }
        __syncthreads();  // q/k/v buffers are rewritten by the next item
    }
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 132;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 132;
        cached[dev] = n;
    }
    return cached[dev];
}

template <typename T, int DK, bool IN_PLACE>
cudaError_t launch_t(const StepArgs& a, int nstage, size_t smem, cudaStream_t stream) {
    auto kern = stream_kernel<T, DK, IN_PLACE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int nitems = a.B * a.g.Hk;
    const int grid = std::min(nitems, sm_count());
    kern<<<grid, kThreads, smem, stream>>>(a, nstage);
    return cudaGetLastError();
}

}  // namespace

bool stream_step_supported(const StepArgs& a, int* nstage_out, size_t* smem_out) {
    const Geom& g = a.g;
    if (g.dv % kTileCols != 0 || (g.dk != 64 && g.dk != 128)) return false;
    const int max_stage = g.dk == 64 ? 4 : 3;
    for (int ns = max_stage; ns >= 2; --ns) {
        const size_t bytes = smem_floats(g.dk, ns, a.L, g.f, g.dv) * 4 + (size_t)ns * 8;
        if (bytes <= 227 * 1024) {
            *nstage_out = ns;
            *smem_out = bytes;
            return true;
        }
    }
    return false;
}

cudaError_t launch_stream_step(const StepArgs& a, bool in_place, cudaStream_t s) {
    int ns = 0;
    size_t smem = 0;
    if (!stream_step_supported(a, &ns, &smem)) return cudaErrorInvalidValue;
    const bool bf = a.g.io_bf16;
    if (a.g.dk == 128) {
        if (bf) return in_place ? launch_t<__nv_bfloat16, 128, true>(a, ns, smem, s)
                                : launch_t<__nv_bfloat16, 128, false>(a, ns, smem, s);
        return in_place ? launch_t<float, 128, true>(a, ns, smem, s) : launch_t<float, 128, false>(a, ns, smem, s);
    }
    if (bf) return in_place ? launch_t<__nv_bfloat16, 64, true>(a, ns, smem, s)
                            : launch_t<__nv_bfloat16, 64, false>(a, ns, smem, s);
    return in_place ? launch_t<float, 64, true>(a, ns, smem, s) : launch_t<float, 64, false>(a, ns, smem, s);
}

cudaError_t stream_error_read(int32_t* value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_stream_error, sizeof(int32_t));
    if (e != cudaSuccess || !clear) return e;
    const int32_t zero = 0;
    return cudaMemcpyToSymbol(g_stream_error, &zero, sizeof(int32_t));
}

}  // namespace gdn
