// gdn_chunked.cu -- prefill in the chunked (WY/UT) form on the 5th-generation
// tensor cores (tcgen05): GDN_PREFILL_CHUNKED.
//
// Step 5 of the MNN "Qwen3.5" page (section 1.2) over a chunk of C tokens that
// starts from state S0.  With G_t the running sum of the chunk's log-decays,
// gamma_t = exp(G_t) and c_t = exp(G_last - G_t), unrolling the recurrence gives
//   U     = T R,  R = diag(beta) (V - diag(gamma) K S0),
//   T     = (I + A)^-1,  A[t][s] = beta_t e^{G_t-G_s} (k_t.k_s) for s < t,
//   O     = diag(gamma) Q S0 + P U,  P[t][s] = e^{G_t-G_s} (q_t.k_s) for s <= t,
//   S_end = gamma_last S0 + K^T diag(c) U,
// where row t of U is the token's delta (beta_t (v_t - v_pred)).  T and P do
// not depend on S0, so:
//   chunk_prep_kernel  (every chunk x key head in parallel) forms the Gram
//       matrices K K^T and Q K^T on the tensor cores, then T and P for each value
//       head of the key head, and writes them, with the chunk's K and Q, as
//       tensor-core operand images to the workspace;
//   chain_kernel  (one CTA per sequence x value head x 32 value columns) walks
//       the chunks in order, three tensor-core rounds per chunk:
//         [K S0, Q S0] -> R -> [T R] -> U -> [P U, K^T diag(c) U] -> O, S_end.
// Every product takes fp32 operands as bf16 hi/lo pairs and accumulates
// hi*hi + hi*lo + lo*hi in fp32 (gdn_umma.cuh): a single bf16 or tf32 pass
// misses the output and state tolerances on this recurrence.
// The path covers head_k_dim = 128 and head_v_dim a multiple of 32.
#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tma.cuh"
#include "gdn_umma.cuh"

namespace gdn {

static __device__ int32_t g_chunk_error;  // set to GDN_ERR_DEVICE_TIMEOUT (7) by a stuck wait

namespace {

constexpr int kC = 64;     // chunk length
constexpr int kDK = 128;   // head_k_dim handled here
constexpr int kNS = 32;    // value columns per chain CTA
constexpr int kCT = 128;   // threads per CTA
constexpr uint32_t kKTokBytes = kC * 2 * kDK * 2;       // one split [64 tokens][2*128] image: 32 KB
constexpr uint32_t kKQBytes = 2 * kKTokBytes;           // K and Q images of a (chunk, key head)
constexpr uint32_t kTBytes = kC * 2 * kC * 2;           // one split [64][2*64] image: 16 KB
constexpr uint32_t kTPBytes = 2 * kTBytes;              // T and P images of a (chunk, value head)

// Chunk offsets: coff[n] = number of chunks of the sequences before n.
__global__ void plan_kernel(const int32_t* __restrict__ cu, int N, int32_t* __restrict__ coff) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        int acc = 0;
        for (int n = 0; n < N; ++n) {
            coff[n] = acc;
            acc += (cu[n + 1] - cu[n] + kC - 1) / kC;
        }
        coff[N] = acc;
    }
}

// Sequence that owns chunk `chunk`: the last n with coff[n] <= chunk.
__device__ __forceinline__ int seq_of_chunk(const int32_t* coff, int N, int chunk) {
    int lo = 0, hi = N;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (coff[mid] <= chunk) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Inclusive prefix sum of g[0..63] in shared memory by warps 0 and 1 (the others
// pass through); result in G[0..63].
__device__ __forceinline__ void scan64(const float* g, float* G, float* carry) {
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid < 64) {
        float v = g[tid];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += o;
        }
        if (tid == 31) *carry = v;
        G[tid] = v;
    }
    __syncthreads();
    if (tid >= 32 && tid < 64) G[tid] += *carry;
    __syncthreads();
}

// ---- chunk prep ----------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kCT, 1) chunk_prep_kernel(const PrefillArgs a, const float* __restrict__ y,
                                                            const int32_t* __restrict__ coff,
                                                            unsigned char* __restrict__ kq,
                                                            unsigned char* __restrict__ tp) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* ktok = smem;                                         // 32 KB
    unsigned char* qtok = smem + kKTokBytes;                            // 32 KB
    float* kk = reinterpret_cast<float*>(smem);                         // [64][65], after the MMAs
    float* qk = kk + kC * (kC + 1);                                     // [64][65]
    // after the MMAs: kk, qk [64][65] over the images, then A and T [64][65] and the
    // T and P operand images (32 KB)
    float* Ab = qk + kC * (kC + 1);
    float* Tb = Ab + kC * (kC + 1);
    unsigned char* img = reinterpret_cast<unsigned char*>(Tb + kC * (kC + 1));
    __shared__ float s_g[kC], s_b[kC], s_G[kC], s_carry;
    __shared__ uint32_t s_tmem;
    __shared__ __align__(8) uint64_t s_bar;
    const Geom& g = a.g;
    const int chunk = blockIdx.x, hk = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = seq_of_chunk(coff, a.N, chunk);
    const int t0 = a.cu[n] + (chunk - coff[n]) * kC;
    const int cnt = min(kC, a.cu[n + 1] - t0);

    // K and Q of the chunk as split operand images [token][dk]
    for (int idx = tid; idx < kC * kDK / 8; idx += kCT) {  // 8 consecutive key dims per step
        const int t = idx / (kDK / 8), i0 = 8 * (idx - t * (kDK / 8));
        float kv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, qv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (t < cnt) {
            const float* row = y + (size_t)(t0 + t) * g.D;
            const float4* kr = reinterpret_cast<const float4*>(row + g.Hk * kDK + hk * kDK + i0);
            const float4* qr = reinterpret_cast<const float4*>(row + hk * kDK + i0);
            const float4 k0 = kr[0], k1 = kr[1], q0 = qr[0], q1 = qr[1];
            kv[0] = k0.x; kv[1] = k0.y; kv[2] = k0.z; kv[3] = k0.w; kv[4] = k1.x; kv[5] = k1.y; kv[6] = k1.z; kv[7] = k1.w;
            qv[0] = q0.x; qv[1] = q0.y; qv[2] = q0.z; qv[3] = q0.w; qv[4] = q1.x; qv[5] = q1.y; qv[6] = q1.z; qv[7] = q1.w;
        }
        umma::store_split8(ktok, t, i0, kDK, kv);
        umma::store_split8(qtok, t, i0, kDK, qv);
    }
    if (warp == 0) umma::tmem_alloc(&s_tmem, 128);
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        fence_mbar_init();
    }
    fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = s_tmem;
    if (tid == 0) {
        umma::mma_split_kk(tmem + 0, ktok, ktok, kC, kC, kDK, false);   // K K^T
        umma::mma_split_kk(tmem + 64, qtok, ktok, kC, kC, kDK, false);  // Q K^T
        umma::commit(&s_bar);
    }
    // the operand images go to the workspace for the chain kernel meanwhile
    {
        const uint4* src = reinterpret_cast<const uint4*>(smem);
        uint4* dst = reinterpret_cast<uint4*>(kq + ((size_t)chunk * g.Hk + hk) * kKQBytes);
        for (int i = tid; i < (int)(kKQBytes / 16); i += kCT) dst[i] = src[i];
    }
    const bool ok = !__syncthreads_or(!mbar_wait_bounded(&s_bar, 0));
    umma::fence_after_sync();
    float vk[32], vq[32];
    const int row = 16 * warp + (lane & 15);  // M = 64 layout: lanes 0-15 of each warp
    for (int half = 0; half < 2; ++half) {
        umma::tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 0 + 32 * half, vk);
        umma::tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 64 + 32 * half, vq);
        __syncthreads();  // everyone is past the MMAs' reads of the images before kk/qk overwrite them
        if (lane < 16 && ok)
            for (int j = 0; j < 32; ++j) {
                kk[row * (kC + 1) + 32 * half + j] = vk[j];
                qk[row * (kC + 1) + 32 * half + j] = vq[j];
            }
    }
    if (!ok && tid == 0) {
        flag_device_error(&g_chunk_error, 7);
        mbar_wait_bounded(&s_bar, 0);  // give the MMAs a last chance to finish before TMEM is freed
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_free(tmem, 128);
    if (!ok) return;

    // ---- T and P for each value head of the key head ----
    for (int hl = 0; hl < g.f; ++hl) {
        const int h = hk * g.f + hl;
        if (tid < kC) {
            const bool in = tid < cnt;
            s_g[tid] = in ? a.gate[(size_t)(t0 + tid) * g.Hv + h] : 0.f;
            s_b[tid] = in ? a.beta[(size_t)(t0 + tid) * g.Hv + h] : 0.f;
        }
        __syncthreads();
        scan64(s_g, s_G, &s_carry);
        for (int idx = tid; idx < kC * kC / 8; idx += kCT) {  // 8 consecutive s per step
            const int t = idx / (kC / 8), s0 = 8 * (idx - t * (kC / 8));
            float pv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int s = s0 + e;
                const float dec = s <= t ? expf(s_G[t] - s_G[s]) : 0.f;
                Ab[t * (kC + 1) + s] = s < t ? __fmul_rn(__fmul_rn(s_b[t], dec), kk[t * (kC + 1) + s]) : 0.f;
                pv[e] = __fmul_rn(dec, qk[t * (kC + 1) + s]);
            }
            umma::store_split8(img + kTBytes, t, s0, kC, pv);  // P
        }
        __syncthreads();
        // T = (I + A)^-1, A strictly lower: blocked by 16.  Diagonal blocks by forward
        // substitution (one thread per column of each block), then the block
        // sub-diagonals d = 1, 2, 3: T_ij = -T_ii * sum_{k=j}^{i-1} A_ik T_kj.
        constexpr int BB = 16, NB = kC / BB;
        if (tid < kC) {
            const int blk = tid / BB, u = tid % BB, o = blk * BB;
            for (int i = 0; i < BB; ++i) {
                float v = i == u ? 1.f : 0.f;
                if (i > u) {
                    float acc = 0.f;
                    for (int s2 = u; s2 < i; ++s2) acc = fmaf(Ab[(o + i) * (kC + 1) + o + s2], Tb[(o + s2) * (kC + 1) + o + u], acc);
                    v = -acc;
                }
                Tb[(o + i) * (kC + 1) + o + u] = v;
            }
            for (int i = 0; i < BB; ++i)  // zero the block row's entries right of the diagonal
                for (int jb = blk + 1; jb < NB; ++jb) Tb[(o + i) * (kC + 1) + jb * BB + u] = 0.f;
        }
        __syncthreads();
        // scratch [NB-1][16][16] in the T half of the image buffer, which is written last
        float* Xb = reinterpret_cast<float*>(img);
        for (int d = 1; d < NB; ++d) {
            const int npair = NB - d;
            // X_p = sum_{k=j}^{i-1} A_ik T_kj for pair p: (i, j) = (j + d, j), j = p
            for (int idx = tid; idx < npair * BB * BB; idx += kCT) {
                const int p = idx / (BB * BB), r = (idx / BB) % BB, cc = idx % BB;
                const int bi = p + d, bj = p;
                float acc = 0.f;
                for (int kb = bj; kb < bi; ++kb)
                    for (int m = 0; m < BB; ++m)
                        acc = fmaf(Ab[(bi * BB + r) * (kC + 1) + kb * BB + m], Tb[(kb * BB + m) * (kC + 1) + bj * BB + cc], acc);
                Xb[idx] = acc;
            }
            __syncthreads();
            for (int idx = tid; idx < npair * BB * BB; idx += kCT) {
                const int p = idx / (BB * BB), r = (idx / BB) % BB, cc = idx % BB;
                const int bi = p + d, bj = p;
                float acc = 0.f;
                for (int m = 0; m <= r; ++m)
                    acc = fmaf(Tb[(bi * BB + r) * (kC + 1) + bi * BB + m], Xb[p * BB * BB + m * BB + cc], acc);
                Tb[(bi * BB + r) * (kC + 1) + bj * BB + cc] = -acc;
            }
            __syncthreads();
        }
        for (int idx = tid; idx < kC * kC / 8; idx += kCT) {
            const int t = idx / (kC / 8), s0 = 8 * (idx - t * (kC / 8));
            float tv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) tv[e] = Tb[t * (kC + 1) + s0 + e];
            umma::store_split8(img, t, s0, kC, tv);
        }
        __syncthreads();
        const uint4* src = reinterpret_cast<const uint4*>(img);
        uint4* dst = reinterpret_cast<uint4*>(tp + ((size_t)chunk * g.Hv + h) * kTPBytes);
        for (int i = tid; i < (int)(kTPBytes / 16); i += kCT) dst[i] = src[i];
        __syncthreads();
    }
}

// ---- chain ----------------------------------------------------------------------
// Loads run ahead of the rounds: T and P are double-buffered (chunk c+1's copy is
// issued when chunk c starts), Q for chunk c+1 is copied as soon as round 1 of
// chunk c has read it, K as soon as round 3 has, and the V slice and gates of
// chunk c+1 are fetched into registers while chunk c computes.
template <typename T>
__global__ void __launch_bounds__(kCT, 1) chain_kernel(const PrefillArgs a, const float* __restrict__ y,
                                                       const int32_t* __restrict__ coff,
                                                       const unsigned char* __restrict__ kq,
                                                       const unsigned char* __restrict__ tp) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* ktok = smem;                        // 32 KB  K   [64 tok][2*128]
    unsigned char* qtok = ktok + kKTokBytes;           // 32 KB  Q   [64 tok][2*128]
    unsigned char* tpb = qtok + kKTokBytes;            // 2 x 32 KB  T, P [64][2*64]
    // B operands stored MN-major (rows along K, each thread writes its own row as
    // 16-byte vectors): S0 [128 key rows][2*32], R, U, diag(c) U [64 tokens][2*32]
    unsigned char* s0t = tpb + 2 * kTPBytes;           // 16 KB  S0
    unsigned char* rt = s0t + kNS * 2 * kDK * 2;       //  8 KB  R
    unsigned char* ut = rt + kNS * 2 * kC * 2;         //  8 KB  U
    unsigned char* cut = ut + kNS * 2 * kC * 2;        //  8 KB  diag(c) U
    float* vv = reinterpret_cast<float*>(cut + kNS * 2 * kC * 2);  // [64][32]
    __shared__ float s_g[kC], s_b[kC], s_G[kC], s_carry;
    __shared__ uint32_t s_tmem;
    __shared__ __align__(8) uint64_t s_k, s_q, s_tp[2], s_mma;
    __shared__ int s_abort;
    const Geom& g = a.g;
    const int slice = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int hk = h / g.f, col0 = slice * kNS;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tb = a.cu[n], te = a.cu[n + 1], len = te - tb;

    // New conv state of sequence n: channels split over the CTAs of the sequence.
    {
        const int nct = gridDim.x * gridDim.y, r = h * gridDim.x + slice;
        const int per = (g.D + nct - 1) / nct;
        T* cst = static_cast<T*>(a.conv_state);
        const T* qkv = static_cast<const T*>(a.qkv);
        if (len > 0)
            for (int c = r * per + tid; c < min(g.D, (r + 1) * per); c += kCT) {
                T* st = cst + ((size_t)n * g.D + c) * (g.K - 1);
                for (int i = 0; i < g.K - 1; ++i) {
                    const int p = len + i;
                    st[i] = p < g.K - 1 ? st[p] : qkv[(size_t)c * a.T + tb + p - (g.K - 1)];
                }
            }
    }
    if (len <= 0) return;
    const int nchunks = coff[n + 1] - coff[n];
    const int chunk0 = coff[n];

    // state rows: thread i holds row i (key dim) of the 32-column slice
    float* Sg = a.ssm_state + ((size_t)(n * g.Hv + h) * kDK + tid) * g.dv + col0;
    float S[kNS];
#pragma unroll
    for (int j = 0; j < kNS; j += 4) {
        const float4 v = *reinterpret_cast<const float4*>(Sg + j);
        S[j] = v.x; S[j + 1] = v.y; S[j + 2] = v.z; S[j + 3] = v.w;
    }
#pragma unroll
    for (int j = 0; j < kNS; j += 8) umma::store_split8(s0t, tid, j, kNS, S + j);

    if (warp == 0) umma::tmem_alloc(&s_tmem, 256);
    if (tid == 0) {
        mbar_init(&s_k, 1);
        mbar_init(&s_q, 1);
        mbar_init(&s_tp[0], 1);
        mbar_init(&s_tp[1], 1);
        mbar_init(&s_mma, 1);
        fence_mbar_init();
        s_abort = 0;
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = s_tmem;
    const uint32_t tDk = tmem + 0, tDq = tmem + 32, tU = tmem + 64, tO = tmem + 96, tS = tmem + 128;
    const uint32_t wl = (uint32_t)(32 * warp) << 16;   // this warp's TMEM lane base
    const int trow = 16 * warp + (lane & 15);         // M = 64 accumulator row held by lanes 0-15

    // thread 0's bookkeeping of copies and MMAs in flight (for a clean exit on abort)
    int k_iss = 0, q_iss = 0, tp_iss[2] = {0, 0}, mma_iss = 0;
    auto load_k = [&](int c) {
        mbar_arrive_expect_tx(&s_k, kKTokBytes);
        bulk_g2s(ktok, kq + ((size_t)(chunk0 + c) * g.Hk + hk) * kKQBytes, kKTokBytes, &s_k);
        ++k_iss;
    };
    auto load_q = [&](int c) {
        mbar_arrive_expect_tx(&s_q, kKTokBytes);
        bulk_g2s(qtok, kq + ((size_t)(chunk0 + c) * g.Hk + hk) * kKQBytes + kKTokBytes, kKTokBytes, &s_q);
        ++q_iss;
    };
    auto load_tp = [&](int c) {
        const int b = c & 1;
        mbar_arrive_expect_tx(&s_tp[b], kTPBytes);
        bulk_g2s(tpb + b * kTPBytes, tp + ((size_t)(chunk0 + c) * g.Hv + h) * kTPBytes, kTPBytes, &s_tp[b]);
        ++tp_iss[b];
    };
    // V slice (16 values per thread) and gates of a chunk, into registers
    float pv[kC * kNS / kCT], pg = 0.f, pb = 0.f;
    auto fetch = [&](int c) {
        const int t0 = tb + c * kC, cnt = min(kC, te - t0);
#pragma unroll
        for (int k = 0; k < kC * kNS / kCT; ++k) {
            const int idx = tid + k * kCT, t = idx / kNS, j = idx - t * kNS;
            pv[k] = t < cnt ? y[(size_t)(t0 + t) * g.D + 2 * g.Hk * kDK + h * g.dv + col0 + j] : 0.f;
        }
        const bool in = tid < cnt;
        pg = tid < kC && in ? a.gate[(size_t)(t0 + tid) * g.Hv + h] : 0.f;
        pb = tid < kC && in ? a.beta[(size_t)(t0 + tid) * g.Hv + h] : 0.f;
    };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        if (!mbar_wait_bounded(bar, parity)) s_abort = 1;
    };

    if (tid == 0) {
        load_k(0);
        load_q(0);
        load_tp(0);
    }
    fetch(0);
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = tb + c * kC, cnt = min(kC, te - t0);
        const unsigned char* tpi = tpb + (c & 1) * kTPBytes;
        if (tid == 0 && c + 1 < nchunks) load_tp(c + 1);  // its buffer's last reader, chunk c-1, is done
#pragma unroll
        for (int k = 0; k < kC * kNS / kCT; ++k) vv[tid + k * kCT] = pv[k];
        if (tid < kC) {
            s_g[tid] = pg;
            s_b[tid] = pb;
        }
        __syncthreads();
        if (c + 1 < nchunks) fetch(c + 1);
        scan64(s_g, s_G, &s_carry);  // running log-decay; ends with a barrier

        // ---- round 1: K S0 and Q S0 ----
        wait_all(&s_k, (uint32_t)(c & 1));
        wait_all(&s_q, (uint32_t)(c & 1));
        wait_all(&s_tp[c & 1], (uint32_t)((c >> 1) & 1));
        fence_proxy_async_smem();  // s0t was written by the generic proxy
        umma::fence_before_sync();
        __syncthreads();
        if (s_abort) break;
        umma::fence_after_sync();
        if (tid == 0) {
            umma::mma_split(tDk, ktok, false, s0t, true, kC, kNS, kDK, false);
            umma::mma_split(tDq, qtok, false, s0t, true, kC, kNS, kDK, false);
            umma::commit(&s_mma);
            ++mma_iss;
        }
        wait_all(&s_mma, (uint32_t)((3 * c) & 1));
        umma::fence_after_sync();
        if (tid == 0 && c + 1 < nchunks) load_q(c + 1);  // round 1 was Q's last reader
        float dk[kNS], dq[kNS];
        umma::tmem_ld32(tDk + wl, dk);
        umma::tmem_ld32(tDq + wl, dq);
        const float gam_t = expf(s_G[trow]);
        if (lane < 16) {
            const float b = s_b[trow];
            float rr[kNS];
#pragma unroll
            for (int j = 0; j < kNS; ++j) rr[j] = __fmul_rn(b, fmaf(-gam_t, dk[j], vv[trow * kNS + j]));
#pragma unroll
            for (int j = 0; j < kNS; j += 8) umma::store_split8(rt, trow, j, kNS, rr + j);
        }
        fence_proxy_async_smem();
        umma::fence_before_sync();
        __syncthreads();
        if (s_abort) break;
        umma::fence_after_sync();

        // ---- round 2: U = T R ----
        if (tid == 0) {
            umma::mma_split(tU, tpi, false, rt, true, kC, kNS, kC, false);
            umma::commit(&s_mma);
            ++mma_iss;
        }
        wait_all(&s_mma, (uint32_t)((3 * c + 1) & 1));
        umma::fence_after_sync();
        float uu[kNS];
        umma::tmem_ld32(tU + wl, uu);
        if (lane < 16) {
            const float cdec = expf(s_G[kC - 1] - s_G[trow]);
            float cu[kNS];
#pragma unroll
            for (int j = 0; j < kNS; ++j) cu[j] = __fmul_rn(cdec, uu[j]);
#pragma unroll
            for (int j = 0; j < kNS; j += 8) {
                umma::store_split8(ut, trow, j, kNS, uu + j);
                umma::store_split8(cut, trow, j, kNS, cu + j);
            }
        }
        fence_proxy_async_smem();
        umma::fence_before_sync();
        __syncthreads();
        if (s_abort) break;
        umma::fence_after_sync();

        // ---- round 3: O = diag(gamma) Q S0 + P U;  S += K^T diag(c) U ----
        if (tid == 0) {
            umma::mma_split(tO, tpi + kTBytes, false, ut, true, kC, kNS, kC, false);
            umma::mma_split(tS, ktok, true, cut, true, kDK, kNS, kC, false);
            umma::commit(&s_mma);
            ++mma_iss;
        }
        wait_all(&s_mma, (uint32_t)((3 * c + 2) & 1));
        umma::fence_after_sync();
        if (tid == 0 && c + 1 < nchunks) load_k(c + 1);  // round 3 was K's last reader
        float oo[kNS], ss[kNS];
        umma::tmem_ld32(tO + wl, oo);
        umma::tmem_ld32(tS + wl, ss);
        if (lane < 16 && trow < cnt) {
            float* orow = a.out + ((size_t)(t0 + trow) * g.Hv + h) * g.dv + col0;
#pragma unroll
            for (int j = 0; j < kNS; j += 4) {
                float4 o;
                o.x = fmaf(gam_t, dq[j], oo[j]); o.y = fmaf(gam_t, dq[j + 1], oo[j + 1]);
                o.z = fmaf(gam_t, dq[j + 2], oo[j + 2]); o.w = fmaf(gam_t, dq[j + 3], oo[j + 3]);
                st_stream(orow + j, o);
            }
        }
        const float gl = expf(s_G[kC - 1]);
#pragma unroll
        for (int j = 0; j < kNS; ++j) S[j] = fmaf(gl, S[j], ss[j]);
#pragma unroll
        for (int j = 0; j < kNS; j += 8) umma::store_split8(s0t, tid, j, kNS, S + j);
        umma::fence_before_sync();
        __syncthreads();  // this chunk's operand reads are complete
        if (s_abort) break;
        umma::fence_after_sync();
    }
    if (s_abort && tid == 0) {
        flag_device_error(&g_chunk_error, 7);
        // let copies and MMAs still in flight land before TMEM and shared memory are released:
        // wait for the last issued phase of each barrier (a completed phase returns at once)
        if (k_iss) mbar_wait_bounded(&s_k, (uint32_t)((k_iss - 1) & 1));
        if (q_iss) mbar_wait_bounded(&s_q, (uint32_t)((q_iss - 1) & 1));
        for (int b = 0; b < 2; ++b)
            if (tp_iss[b]) mbar_wait_bounded(&s_tp[b], (uint32_t)((tp_iss[b] - 1) & 1));
        if (mma_iss) mbar_wait_bounded(&s_mma, (uint32_t)((mma_iss - 1) & 1));
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_free(tmem, 256);
    if (s_abort) return;
#pragma unroll
    for (int j = 0; j < kNS; j += 4) *reinterpret_cast<float4*>(Sg + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
}

constexpr size_t kChainSmem = 2 * kKTokBytes + 2 * kTPBytes + kNS * 2 * kDK * 2 + 3 * (kNS * 2 * kC * 2) + kC * kNS * 4;
constexpr size_t kPrepSmem = (4 * kC * (kC + 1) * 4 + kTPBytes) > kKQBytes ? (4 * kC * (kC + 1) * 4 + kTPBytes) : kKQBytes;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct ChunkWs {
    size_t y, coff, kq, tp, total;
    ChunkWs(const Geom& g, int N, long long T, int nchunk) {
        size_t o = 0;
        y = o;    o = align256(o + (size_t)T * g.D * 4);
        coff = o; o = align256(o + (size_t)(N + 1) * 4);
        kq = o;   o = align256(o + (size_t)nchunk * g.Hk * kKQBytes);
        tp = o;   o = align256(o + (size_t)nchunk * g.Hv * kTPBytes);
        total = o;
    }
};

}  // namespace

bool prefill_chunked_supported(const Geom& g) { return g.dk == kDK && g.dv % kNS == 0; }

int prefill_chunk_count(const int32_t* cu_host, int N) {
    int acc = 0;
    for (int n = 0; n < N; ++n) acc += (cu_host[n + 1] - cu_host[n] + kC - 1) / kC;
    return acc;
}

size_t prefill_chunked_workspace(const Geom& g, int N, long long T, int nchunk) {
    return ChunkWs(g, N, T, nchunk).total;
}

// The chunk-count-free upper bound used by gdn_prefill_workspace_size:
// every sequence adds at most one partial chunk.
size_t prefill_chunked_workspace_bound(const Geom& g, int N, long long T) {
    const long long nchunk = (T + kC - 1) / kC + N;
    return ChunkWs(g, N, T, (int)std::min<long long>(nchunk, 1ll << 30)).total;
}

cudaError_t launch_prefill_chunked(const PrefillArgs& a, cudaStream_t stream) {
    const Geom& g = a.g;
    const int nchunk = prefill_chunk_count(a.cu_host, a.N);
    const ChunkWs ws(g, a.N, a.T, nchunk);
    unsigned char* base = static_cast<unsigned char*>(a.ws);
    float* y = reinterpret_cast<float*>(base + ws.y);
    int32_t* coff = reinterpret_cast<int32_t*>(base + ws.coff);
    unsigned char* kq = base + ws.kq;
    unsigned char* tp = base + ws.tp;
    cudaError_t e = launch_prefill_prep(a, y, stream);
    if (e != cudaSuccess) return e;
    plan_kernel<<<1, 32, 0, stream>>>(a.cu, a.N, coff);
    e = cudaGetLastError();
    if (e != cudaSuccess || nchunk == 0) return e;
    if (a.g.io_bf16) {
        e = cudaFuncSetAttribute(chunk_prep_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kPrepSmem);
        if (e != cudaSuccess) return e;
        chunk_prep_kernel<__nv_bfloat16><<<dim3(nchunk, g.Hk), kCT, kPrepSmem, stream>>>(a, y, coff, kq, tp);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(chain_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kChainSmem);
        if (e != cudaSuccess) return e;
        chain_kernel<__nv_bfloat16><<<dim3(g.dv / kNS, g.Hv, a.N), kCT, kChainSmem, stream>>>(a, y, coff, kq, tp);
    } else {
        e = cudaFuncSetAttribute(chunk_prep_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem);
        if (e != cudaSuccess) return e;
        chunk_prep_kernel<float><<<dim3(nchunk, g.Hk), kCT, kPrepSmem, stream>>>(a, y, coff, kq, tp);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(chain_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kChainSmem);
        if (e != cudaSuccess) return e;
        chain_kernel<float><<<dim3(g.dv / kNS, g.Hv, a.N), kCT, kChainSmem, stream>>>(a, y, coff, kq, tp);
    }
    return cudaGetLastError();
}

cudaError_t chunk_error_read(int32_t* value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_chunk_error, sizeof(int32_t));
    if (e != cudaSuccess || !clear) return e;
    const int32_t zero = 0;
    return cudaMemcpyToSymbol(g_chunk_error, &zero, sizeof(int32_t));
}

}  // namespace gdn
