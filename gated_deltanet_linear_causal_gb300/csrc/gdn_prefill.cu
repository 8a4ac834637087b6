// gdn_prefill.cu -- prefill over cu_seqlens-packed sequences, resident form
// (GDN_PREFILL_RESIDENT).
//
// Three launches:
//   prep   steps 1-4 of the MNN "Qwen3.5" page, section 1.2, for every packed
//          token: causal conv + SiLU from the raw qkv [D, T] (channel-major, as
//          the page lays out qkv [B, D, L]) with each sequence's carried conv
//          state (section 1.4), then per-head L2 norms and the 1/sqrt(dk)
//          scale.  Writes token-major fp32 rows y [T, D] to the workspace.
//   gram   the lagged dot products q_t.k_{t-d} and k_t.k_{t-d} (d < 8) that the
//          block recurrence needs, per token and key head.
//   block  step 5, the gated delta rule: one CTA per (sequence, value head,
//          column group) keeps its columns of S in registers across the whole
//          sequence and advances 8 tokens per reduction round (the block form
//          below).  It also writes each sequence's new conv state: the prep
//          launch has finished reading the old one by then.
// The resident form stays serial in the sequence length, 8 tokens at a time.
// With the gated RMSNorm fused (section 2), the dv/16 block CTAs of a value head
// form a cluster and exchange the rows' sums of squares (see block_kernel).
#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tma.cuh"

namespace gdn {

static __device__ int32_t g_prefill_error;  // set to GDN_ERR_DEVICE_TIMEOUT (7) by a stuck wait

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
    // One thread per (channel, group of kConvRun consecutive tokens): when the group
    // lies inside one sequence past its first K-1 tokens, the K-1+kConvRun window
    // samples and the K weights are loaded once for the whole group.
    constexpr int kConvRun = 8;
    for (int idx = tid; idx < nch * (kPrepTokens / kConvRun); idx += kPrepThreads) {
        const int cl = idx / (kPrepTokens / kConvRun), tg = idx - cl * (kPrepTokens / kConvRun);
        const int c = cbase + cl, tl0 = tg * kConvRun, t = t0 + tl0;
        float wr[kMaxConv];
#pragma unroll
        for (int j = 0; j < kMaxConv; ++j) wr[j] = j < K ? to_f32(w[(size_t)c * K + j]) : 0.f;
        const int last = min(t + kConvRun, a.T) - 1;  // last token of the group in range
        const bool fast = t < a.T && s_seq[tl0] == s_seq[last - t0] && s_pos[tl0] >= K - 1;
        if (fast) {
            const T* xs = qkv + (size_t)c * a.T + t - (K - 1);
            float xw[kConvRun + kMaxConv - 1];
#pragma unroll
            for (int j = 0; j < kConvRun + kMaxConv - 1; ++j)
                xw[j] = (j < kConvRun + K - 1 && t - (K - 1) + j <= last) ? to_f32(xs[j]) : 0.f;
#pragma unroll
            for (int r = 0; r < kConvRun; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < kMaxConv; ++j)
                    if (j < K) acc = fmaf(wr[j], xw[r + j], acc);
                tile[cl * (kPrepTokens + 1) + tl0 + r] = t + r <= last ? silu(acc) : 0.f;
            }
        } else {
            for (int r = 0; r < kConvRun; ++r) {
                const int tl = tl0 + r, tt = t + r;
                float v = 0.f;
                if (tt < a.T) {
                    const int n = s_seq[tl], pos = s_pos[tl], st = s_start[tl];
                    float acc = 0.f;
                    for (int j = 0; j < K; ++j) {
                        const int p = pos - (K - 1) + j;  // position in the sequence
                        const T xv = p >= 0 ? qkv[(size_t)c * a.T + st + p]
                                            : cst[((size_t)n * g.D + c) * (K - 1) + (pos + j)];
                        acc = fmaf(wr[j], to_f32(xv), acc);
                    }
                    v = silu(acc);
                }
                tile[cl * (kPrepTokens + 1) + tl] = v;
            }
        }
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
    // nch is a power of two (dk or 32): rows of 4 channels go out as 16-byte stores
    const int lg4 = __ffs(nch / 4) - 1;
    for (int idx = tid; idx < (nch / 4) * kPrepTokens; idx += kPrepThreads) {
        const int tl = idx >> lg4, c4 = idx & (nch / 4 - 1);
        const int t = t0 + tl;
        if (t < a.T) {
            const float f = s_fac[tl];
            const float* col = tile + 4 * c4 * (kPrepTokens + 1) + tl;
            const float4 v = make_float4(__fmul_rn(col[0], f), __fmul_rn(col[kPrepTokens + 1], f),
                                         __fmul_rn(col[2 * (kPrepTokens + 1)], f),
                                         __fmul_rn(col[3 * (kPrepTokens + 1)], f));
            *reinterpret_cast<float4*>(y + (size_t)t * g.D + cbase + 4 * c4) = v;
        }
    }
}

// ---- lagged Gram entries -------------------------------------------------------
// For every packed token t and key head: gram[t][hk][d] = q_t . k_{t-d}
// (d = 0..7) and gram[t][hk][8+d] = k_t . k_{t-d} (d = 1..7), from the
// normalised rows prep_kernel wrote; entries reaching before the start of t's
// sequence are 0.  The block kernel combines them with the decays of each
// value head sharing the key head.
constexpr int kBM = 8;          // tokens per block of the block-sequential kernel
constexpr int kGramTok = 32;    // tokens per gram CTA

template <int DK>
__global__ void __launch_bounds__(256) gram_kernel(const PrefillArgs a, const float* __restrict__ y,
                                                   float* __restrict__ gram) {
    constexpr int KR = DK + 4;  // padded row
    extern __shared__ float4 smem_f4[];
    float* sk = reinterpret_cast<float*>(smem_f4);          // [kGramTok + kBM - 1][KR]  k rows
    float* sq = sk + (kGramTok + kBM - 1) * KR;             // [kGramTok][KR]           q rows
    __shared__ int s_start[kGramTok];
    const Geom& g = a.g;
    const int t0 = blockIdx.x * kGramTok, hk = blockIdx.y, tid = threadIdx.x;
    if (tid < kGramTok && t0 + tid < a.T) s_start[tid] = a.cu[seq_of(a.cu, a.N, t0 + tid)];
    for (int idx = tid; idx < (kGramTok + kBM - 1) * (DK / 4); idx += 256) {
        const int r = idx / (DK / 4), c4 = idx - r * (DK / 4);
        const int t = t0 - (kBM - 1) + r;
        float4 kv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t >= 0 && t < a.T) kv = __ldg(reinterpret_cast<const float4*>(y + (size_t)t * g.D + g.Hk * DK + hk * DK) + c4);
        *reinterpret_cast<float4*>(sk + r * KR + 4 * c4) = kv;
    }
    for (int idx = tid; idx < kGramTok * (DK / 4); idx += 256) {
        const int r = idx / (DK / 4), c4 = idx - r * (DK / 4);
        const int t = t0 + r;
        float4 qv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < a.T) qv = __ldg(reinterpret_cast<const float4*>(y + (size_t)t * g.D + hk * DK) + c4);
        *reinterpret_cast<float4*>(sq + r * KR + 4 * c4) = qv;
    }
    __syncthreads();
    // 32 tokens x 16 entries = 512 dots; 2 per thread
    for (int job = tid; job < kGramTok * 16; job += 256) {
        const int tl = job >> 4, e = job & 15;
        const int t = t0 + tl;
        if (t >= a.T) continue;
        const int d = e & 7;
        const bool kk = e >= 8;
        const float* u = kk ? sk + (tl + kBM - 1) * KR : sq + tl * KR;
        const float* v = sk + (tl + kBM - 1 - d) * KR;
        float acc = 0.f;
        if ((!kk || d > 0) && t - d >= s_start[tl]) {
            float acc2 = 0.f;
#pragma unroll 8
            for (int i = 0; i < DK; i += 8) {
                const float4 u0 = *reinterpret_cast<const float4*>(u + i), u1 = *reinterpret_cast<const float4*>(u + i + 4);
                const float4 v0 = *reinterpret_cast<const float4*>(v + i), v1 = *reinterpret_cast<const float4*>(v + i + 4);
                acc = fmaf(u0.x, v0.x, acc); acc2 = fmaf(u0.y, v0.y, acc2);
                acc = fmaf(u0.z, v0.z, acc); acc2 = fmaf(u0.w, v0.w, acc2);
                acc = fmaf(u1.x, v1.x, acc); acc2 = fmaf(u1.y, v1.y, acc2);
                acc = fmaf(u1.z, v1.z, acc); acc2 = fmaf(u1.w, v1.w, acc2);
            }
            acc += acc2;
        }
        gram[((size_t)t * g.Hk + hk) * 16 + e] = acc;
    }
}

// ---- block-sequential gated delta rule (section 1.2, Step 5) -----------------
// For a block of kBM tokens starting from state S0, with G_t the running sum of
// the block's log-decays and gamma_t = exp(G_t), unrolling Step 5 gives, per
// value column j:
//   a_t     = gamma_t (S0^T k_t)_j + sum_{s<t} e^{G_t-G_s} (k_s.k_t) delta_s
//   delta_t = beta_t (v_t - a_t)
//   o_t     = gamma_t (S0^T q_t)_j + sum_{s<=t} e^{G_t-G_s} (k_s.q_t) delta_s
//   S_end   = gamma_last S0 + sum_s e^{G_last-G_s} k_s delta_s^T.
// The 2*kBM dot products against S0 are independent, so each block needs one
// reduction round instead of one per token.  The lanes of a warp that share a
// value column split its dk rows and reduce with shuffles only (BlockCfg).
constexpr int kBW = 4;                  // warps per CTA
constexpr int kBT = kBW * 32;

// Lane layout of the block kernel: LPC lanes share one value column and split its
// dk rows (RPL consecutive rows each); a warp owns CPW columns, a CTA BC.  Rows
// of the shared q/k tiles are padded by 4 floats after every RPL rows so that the
// LPC lanes' 16-byte loads of one column group hit distinct banks.
template <int DK>
struct BlockCfg {
    static constexpr int LPC = 8;  // 16 doubles the warps, and with them the per-warp delta chain
    static constexpr int CPW = 32 / LPC;
    static constexpr int RPL = DK / LPC;
    static constexpr int BC = CPW * kBW;
    static constexpr int KR = DK + LPC * 4;
    __device__ __forceinline__ static int at(int row) { return row + (row / RPL) * 4; }
};

// NORM: the output rows get the gated RMSNorm, which needs each row's sum of squares
// over all dv columns: the dv/16 CTAs of a value head form a cluster; after a block,
// each CTA sends its rows' partial sums (over its 16 columns) to every CTA of the
// cluster (asynchronous stores into their shared memory that complete bytes on their
// barriers).  The exchange rides on the block's own barriers: at block e, warp 3
// waits for the partials of block e-2 after the first barrier (while warp 0 computes
// the block's coefficients), every thread reads their sums after the second (the
// barrier makes them visible), and after the third the CTA sends its partials of
// block e-1 and normalises and stores block e-2, whose raw outputs and z values wait
// in registers.  A peer's buffer is thus rewritten only after its reads of the
// buffer's previous use (they precede the send this CTA waited for), and the
// partials have a whole block to arrive.
template <typename T, int DK, bool NORM>
__global__ void __launch_bounds__(kBT) block_kernel(const PrefillArgs a, const GateParams gp, const float* __restrict__ y,
                                                    const float* __restrict__ gram) {
    using R = BlockCfg<DK>;
    constexpr int RPL = R::RPL, KR = R::KR, LPC = R::LPC, CPW = R::CPW, kBC = R::BC;
    constexpr int NV4 = (2 * DK + kBC) / 4;      // float4 per staged token: q, k, v slice
    constexpr int PER = (kBM * NV4 + kBT - 1) / kBT;
    __shared__ __align__(16) float s_q[kBM][KR], s_k[kBM][KR], s_kt[kBM][KR];
    __shared__ __align__(16) float s_v[kBM][kBC];
    __shared__ float s_gram[kBM][16];
    __shared__ float s_g[kBM], s_b[kBM], s_gam[kBM], s_c[kBM];
    __shared__ __align__(16) float s_Gkk[kBM][kBM], s_Gkq[kBM][kBM];
    // NORM: per-warp partial sums of the block's rows, and the cluster's partials by block parity
    __shared__ float s_wss[2][kBW][kBM];  // by block parity
    __shared__ float s_np[NORM ? 2 : 1][NORM ? 8 : 1][kBM];
    __shared__ __align__(8) uint64_t s_nb[2];
    __shared__ int s_nfail;  // NORM: a wait for the partials gave up (read after barriers only)
    const Geom& g = a.g;
    const int slice = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int hk = h / g.f, col0 = slice * kBC;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cw = lane / LPC, rl = lane % LPC;  // column in warp, row lane
    const int col = warp * CPW + cw;             // column in the CTA slice
    const int tb = a.cu[n], te = a.cu[n + 1];
    const int len = te - tb;
    float* Sg = a.ssm_state + (size_t)(n * g.Hv + h) * DK * g.dv + col0 + col;

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
    const int ncta = g.dv / kBC;  // CTAs of the cluster (NORM)
    if (NORM) {
        if (tid == 0) {
            s_nfail = 0;
            mbar_init(&s_nb[0], 1);  // one local arrive.expect_tx; the bytes come from the whole cluster
            mbar_init(&s_nb[1], 1);
            fence_mbar_init();
        }
        cluster_arrive_release();  // every CTA's barriers exist before any remote arrive
        cluster_wait_acquire();
    }
    const uint32_t crank = NORM ? cluster_ctarank() : 0;
    // the raw outputs of the last two blocks this thread holds (1: the block before, 2: the
    // one before that), their z values (io type, converted at use so that no thread waits
    // on the load) and token ranges, and the norm weight of its column
    float o1 = 0.f, o2 = 0.f;
    T z1 = T(), z2 = T();
    int t01 = 0, cnt1 = 0, t02 = 0, cnt2 = 0, e = 0;
    const float w_col = NORM ? a.norm.weight[col0 + col] : 0.f;
    // warp 3: wait until every CTA's partials of block pe have landed (gives up for good,
    // flagged, on a stuck wait)
    auto norm_wait = [&](int pe) {
        if (!s_nfail && !mbar_wait_cluster(&s_nb[pe & 1], (uint32_t)((pe >> 1) & 1), nullptr)) {
            flag_device_error(&g_prefill_error, 7);
            s_nfail = 1;
        }
    };
    // 1/RMS of row rl of block pe, after a barrier that follows norm_wait(pe); -1 after a failed wait
    auto norm_scale = [&](int pe) {
        const int bn = pe & 1;
        if (s_nfail) return -1.f;
        float tot = 0.f;
        for (int q = 0; q < ncta; ++q) tot += s_np[bn][q][rl];
        return rsqrtf(fmaf(tot, 1.f / (float)g.dv, a.norm.eps));
    };
    auto norm_store = [&](int pt0, int pcnt, float o, T z, float rinv) {
        if (rinv >= 0.f && rl < pcnt) {
            const size_t at = ((size_t)(pt0 + rl) * g.Hv + h) * g.dv + col0 + col;
            static_cast<T*>(a.norm.y)[at] =
                from_f32<T>(__fmul_rn(__fmul_rn(w_col, __fmul_rn(o, rinv)), silu_fast(to_f32(z))));
        }
    };
    // this CTA's partial sums of block pe's rows (in s_wss) to every CTA of the cluster
    auto norm_send = [&](int pe) {
        if (tid < kBM) {
            const int bn = pe & 1;
            const float p = (s_wss[bn][0][tid] + s_wss[bn][1][tid]) + (s_wss[bn][2][tid] + s_wss[bn][3][tid]);
            if (tid == 0) mbar_arrive_expect_tx(&s_nb[bn], (uint32_t)(4 * kBM * ncta));
            for (int q = 0; q < ncta; ++q)
                st_async_cluster(cluster_addr(&s_np[bn][crank][tid], q), p, cluster_addr(&s_nb[bn], q));
        }
    };

    float S[RPL];
#pragma unroll
    for (int r = 0; r < RPL; ++r) S[r] = Sg[(size_t)(rl * RPL + r) * g.dv];

    float4 pre[PER];
    float pg = 0.f, pb = 0.f, pgr = 0.f;
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
        pg = ok ? gate_of(gp.A_log, gp.dt_bias, a.gate[(size_t)(t0 + tid) * g.Hv + h], h) : 0.f;
        pb = ok ? beta_of(gp.A_log, a.beta[(size_t)(t0 + tid) * g.Hv + h]) : 0.f;
        pgr = (tid < kBM * 16 && t0 + (tid >> 4) < te) ? __ldg(gram + ((size_t)(t0 + (tid >> 4)) * g.Hk + hk) * 16 + (tid & 15))
                                                      : 0.f;
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
                if (part < DK / 4) *reinterpret_cast<float4*>(&s_q[tl][R::at(4 * part)]) = pre[j];
                else if (part < DK / 2) *reinterpret_cast<float4*>(&s_k[tl][R::at(4 * (part - DK / 4))]) = pre[j];
                else *reinterpret_cast<float4*>(&s_v[tl][4 * (part - DK / 2)]) = pre[j];
            }
        }
        if (tid < kBM) {
            s_g[tid] = pg;
            s_b[tid] = pb;
        }
        if (tid < kBM * 16) s_gram[tid >> 4][tid & 15] = pgr;
        __syncthreads();
        if (t0 + kBM < te) fetch(t0 + kBM);  // next block's loads fly under this block
        if (NORM && e >= 2 && warp == 3) norm_wait(e - 2);

        // ---- block coefficients (warp 0) ----
        if (warp == 0) {
            float G = lane < kBM ? s_g[lane] : 0.f;  // inclusive prefix sum of the log-decays
#pragma unroll
            for (int off = 1; off < kBM; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, G, off);
                if (lane >= off) G += o;
            }
            const float Glast = __shfl_sync(0xffffffffu, G, kBM - 1);
            if (lane < kBM) {
                s_gam[lane] = expf(G);
                s_c[lane] = expf(Glast - G);
            }
            // lane handles (t, s) pairs lane and lane + 32 of the 8x8 grid
#pragma unroll
            for (int p = lane; p < kBM * kBM; p += 32) {
                const int t = p >> 3, s2 = p & 7;
                const float Gt = __shfl_sync(0xffffffffu, G, t), Gs = __shfl_sync(0xffffffffu, G, s2);
                const float dec = s2 <= t ? expf(Gt - Gs) : 0.f;
                s_Gkq[t][s2] = s2 <= t ? __fmul_rn(dec, s_gram[t][t - s2]) : 0.f;
                s_Gkk[t][s2] = s2 < t ? __fmul_rn(dec, s_gram[t][8 + t - s2]) : 0.f;
            }
        }
        __syncthreads();
        if (NORM && e >= 2) norm_store(t02, cnt2, o2, z2, norm_scale(e - 2));  // warp 3 waited before the barrier
        for (int idx = tid; idx < kBM * (DK / 4); idx += kBT) {
            const int s2 = idx / (DK / 4), c4 = idx - s2 * (DK / 4);
            const int at = R::at(4 * c4);
            const float cs = s_c[s2];
            float4 kv = *reinterpret_cast<const float4*>(&s_k[s2][at]);
            kv.x = __fmul_rn(cs, kv.x); kv.y = __fmul_rn(cs, kv.y);
            kv.z = __fmul_rn(cs, kv.z); kv.w = __fmul_rn(cs, kv.w);
            *reinterpret_cast<float4*>(&s_kt[s2][at]) = kv;
        }

        // ---- dot products of the block's keys and queries with S0 ----
        float dk[kBM], dq[kBM];
#pragma unroll
        for (int t = 0; t < kBM; ++t) dk[t] = dq[t] = 0.f;
#pragma unroll
        for (int r4 = 0; r4 < RPL / 4; ++r4) {
            const int at = R::at(rl * RPL + 4 * r4);
#pragma unroll
            for (int t = 0; t < kBM; ++t) {
                const float4 kv = *reinterpret_cast<const float4*>(&s_k[t][at]);
                const float4 qv = *reinterpret_cast<const float4*>(&s_q[t][at]);
                dk[t] = fmaf(S[4 * r4 + 0], kv.x, dk[t]); dk[t] = fmaf(S[4 * r4 + 1], kv.y, dk[t]);
                dk[t] = fmaf(S[4 * r4 + 2], kv.z, dk[t]); dk[t] = fmaf(S[4 * r4 + 3], kv.w, dk[t]);
                dq[t] = fmaf(S[4 * r4 + 0], qv.x, dq[t]); dq[t] = fmaf(S[4 * r4 + 1], qv.y, dq[t]);
                dq[t] = fmaf(S[4 * r4 + 2], qv.z, dq[t]); dq[t] = fmaf(S[4 * r4 + 3], qv.w, dq[t]);
            }
        }
#pragma unroll
        for (int off = 1; off < LPC; off <<= 1) {
#pragma unroll
            for (int t = 0; t < kBM; ++t) {
                dk[t] += __shfl_xor_sync(0xffffffffu, dk[t], off);
                dq[t] += __shfl_xor_sync(0xffffffffu, dq[t], off);
            }
        }
        __syncthreads();  // s_kt, s_Gkk, s_Gkq are ready
        if (NORM && e >= 1) norm_send(e - 1);  // every thread has read block e-2's sums

        // ---- resolve the block's deltas and outputs for this lane's column ----
        float dl[kBM];
        float o_mine = 0.f;
#pragma unroll
        for (int t = 0; t < kBM; ++t) {
            float acc = __fmul_rn(s_gam[t], dk[t]);
#pragma unroll
            for (int s2 = 0; s2 < t; ++s2) acc = fmaf(s_Gkk[t][s2], dl[s2], acc);
            dl[t] = t < cnt ? __fmul_rn(s_b[t], s_v[t][col] - acc) : 0.f;
            float o = __fmul_rn(s_gam[t], dq[t]);
#pragma unroll
            for (int s2 = 0; s2 <= t; ++s2) o = fmaf(s_Gkq[t][s2], dl[s2], o);
            if (t == rl) o_mine = o;
        }
        if (NORM) {
            // this CTA's partial of row rl: the warp's 4 columns (lanes rl + 8 cw), then the 4 warps
            // (summed and sent at the next block, after its first barrier)
            float ss = __fmul_rn(o_mine, o_mine);
            ss += __shfl_xor_sync(0xffffffffu, ss, 8);
            ss += __shfl_xor_sync(0xffffffffu, ss, 16);
            if (cw == 0) s_wss[e & 1][warp][rl] = ss;
            o2 = o1, z2 = z1, t02 = t01, cnt2 = cnt1;
            o1 = o_mine, t01 = t0, cnt1 = cnt;
            if (rl < cnt) z1 = static_cast<const T*>(a.norm.z)[((size_t)(t0 + rl) * g.Hv + h) * g.dv + col0 + col];
            ++e;
        } else if (rl < cnt) {
            a.out[((size_t)(t0 + rl) * g.Hv + h) * g.dv + col0 + col] = o_mine;
        }

        // ---- S <- gamma_last S + sum_s c_s k_s delta_s^T ----
        const float gl = s_gam[kBM - 1];
#pragma unroll
        for (int r4 = 0; r4 < RPL / 4; ++r4) {
            const int at = R::at(rl * RPL + 4 * r4);
            float x0 = __fmul_rn(gl, S[4 * r4 + 0]), x1 = __fmul_rn(gl, S[4 * r4 + 1]);
            float x2 = __fmul_rn(gl, S[4 * r4 + 2]), x3 = __fmul_rn(gl, S[4 * r4 + 3]);
#pragma unroll
            for (int t = 0; t < kBM; ++t) {
                const float4 kt = *reinterpret_cast<const float4*>(&s_kt[t][at]);
                x0 = fmaf(kt.x, dl[t], x0); x1 = fmaf(kt.y, dl[t], x1);
                x2 = fmaf(kt.z, dl[t], x2); x3 = fmaf(kt.w, dl[t], x3);
            }
            S[4 * r4 + 0] = x0; S[4 * r4 + 1] = x1; S[4 * r4 + 2] = x2; S[4 * r4 + 3] = x3;
        }
        __syncthreads();  // the block's shared data is consumed
    }
    if (NORM) {  // blocks e-2 and e-1 (e = the block count); the last block's partials are in s_wss
        if (e >= 2 && warp == 3) norm_wait(e - 2);
        __syncthreads();
        if (e >= 2) norm_store(t02, cnt2, o2, z2, norm_scale(e - 2));
        __syncthreads();
        norm_send(e - 1);
        if (warp == 3) norm_wait(e - 1);
        __syncthreads();
        norm_store(t01, cnt1, o1, z1, norm_scale(e - 1));
        cluster_arrive_release();  // no CTA leaves while a peer may still write into its shared memory
        cluster_wait_acquire();
    }
#pragma unroll
    for (int r = 0; r < RPL; ++r) Sg[(size_t)(rl * RPL + r) * g.dv] = S[r];
}

template <typename T>
cudaError_t launch_prep_t(const PrefillArgs& a, float* y, cudaStream_t stream) {
    const Geom& g = a.g;
    const int ngrp = 2 * g.Hk + g.Hv * (g.dv / kSliceCols);
    const size_t prep_smem = (size_t)std::max(g.dk, kSliceCols) * (kPrepTokens + 1) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(prep_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prep_smem);
    if (e != cudaSuccess) return e;
    prep_kernel<T><<<dim3((a.T + kPrepTokens - 1) / kPrepTokens, ngrp), kPrepThreads, prep_smem, stream>>>(a, y);
    return cudaGetLastError();
}

template <typename T, int DK>
cudaError_t launch_resident_t(const PrefillArgs& a, const GateParams& gp, cudaStream_t stream) {
    const Geom& g = a.g;
    float* y = static_cast<float*>(a.ws);
    float* gram = y + (size_t)a.T * g.D;
    cudaError_t e = launch_prep_t<T>(a, y, stream);
    if (e != cudaSuccess) return e;
    const size_t gram_smem = (size_t)(2 * kGramTok + kBM - 1) * (DK + 4) * sizeof(float);
    e = cudaFuncSetAttribute(gram_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gram_smem);
    if (e != cudaSuccess) return e;
    gram_kernel<DK><<<dim3((a.T + kGramTok - 1) / kGramTok, g.Hk), 256, gram_smem, stream>>>(a, y, gram);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const dim3 grid(g.dv / BlockCfg<DK>::BC, g.Hv, a.N);
    if (!a.norm.z) {
        block_kernel<T, DK, false><<<grid, kBT, 0, stream>>>(a, gp, y, gram);
        return cudaGetLastError();
    }
    // the gated RMSNorm fused: the dv/16 CTAs of a value head form one cluster
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kBT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = grid.x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, block_kernel<T, DK, true>, a, gp, static_cast<const float*>(y),
                              static_cast<const float*>(gram));
}

}  // namespace

cudaError_t launch_prefill_prep(const PrefillArgs& a, float* y, cudaStream_t s) {
    return a.g.io_bf16 ? launch_prep_t<__nv_bfloat16>(a, y, s) : launch_prep_t<float>(a, y, s);
}

size_t prefill_resident_workspace(const Geom& g, int /*N*/, long long T) {
    return (size_t)T * g.D * sizeof(float) + (size_t)T * g.Hk * 16 * sizeof(float);
}

// Fused norm: one cluster per value head, dv/16 CTAs (resident) or dv/32 (chunked),
// at most the portable cluster size of 8.
bool prefill_norm_supported(const Geom& g, int variant) {
    if (variant == 0) return g.dv / 16 <= 8;
    return prefill_chunked_supported(g);
}

cudaError_t prefill_error_read(int32_t* value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_prefill_error, sizeof(int32_t));
    if (e != cudaSuccess || !clear) return e;
    const int32_t zero = 0;
    return cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(int32_t));
}

cudaError_t launch_prefill_resident(const PrefillArgs& a, const GateParams& gp, cudaStream_t s) {
    if (a.g.io_bf16) {
        switch (a.g.dk) {
            case 32: return launch_resident_t<__nv_bfloat16, 32>(a, gp, s);
            case 64: return launch_resident_t<__nv_bfloat16, 64>(a, gp, s);
            case 128: return launch_resident_t<__nv_bfloat16, 128>(a, gp, s);
            case 256: return launch_resident_t<__nv_bfloat16, 256>(a, gp, s);
        }
    } else {
        switch (a.g.dk) {
            case 32: return launch_resident_t<float, 32>(a, gp, s);
            case 64: return launch_resident_t<float, 64>(a, gp, s);
            case 128: return launch_resident_t<float, 128>(a, gp, s);
            case 256: return launch_resident_t<float, 256>(a, gp, s);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdn
