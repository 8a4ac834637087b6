/*
 * gdn.h -- C ABI of the Gated DeltaNet linear-attention layer for one NVIDIA
 * GB300 (sm_103a).
 *
 * The layer (MNN discussion "MNN Model Support: Qwen3.5", section 1.2) takes
 * qkv [B, D, L], gate [B, L, H], beta [B, L, H] and conv_weight [D, 1, K], with
 * D = 2*Hk*dk + Hv*dv, and runs five steps:
 *   1. stateful depthwise causal Conv1D over the D channels, then SiLU;
 *   2. split into Q = channels [0, Hk*dk), K = [Hk*dk, 2*Hk*dk), V = the rest,
 *      head-major, with reverse GQA: value head h reads key head h/(Hv/Hk)
 *      (section 1.3, repeat_interleave);
 *   3. optional per-head L2 normalisation of Q and K: x * 1/sqrt(sum x^2 + eps);
 *   4. Q scaled by 1/sqrt(dk);
 *   5. the gated delta rule on a per-value-head fp32 state S [dk, dv]:
 *        S = S*exp(g_t); v_pred = S^T k_t; delta = beta_t (v_t - v_pred);
 *        S = S + k_t delta^T; o_t = S^T q_t.
 * Two states persist between calls (section 1.4): the conv state [B, D, K-1]
 * (raw pre-conv inputs of the last K-1 tokens, oldest first, in the io dtype)
 * and the recurrent state [B, Hv, dk, dv] (fp32, row i = key dimension).
 *
 * Conventions common to every entry point:
 *   - The caller owns every buffer.  Device pointers are device memory of the
 *     current CUDA device; the library allocates nothing.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and never synchronises the host.
 *   - Errors are returned, never thrown: host-side argument checks run before
 *     any launch, so a call that returns an error has launched nothing;
 *     GDN_ERR_CUDA reports a failed launch (gdn_last_cuda_error() gives the
 *     CUDA error code of the calling thread's last failure).
 *   - Alignment: qkv, the fp32 states, snapshots, out and workspace must be
 *     16-byte aligned (GDN_ERR_ALIGN otherwise); gate, beta, conv_weight and
 *     conv states need their element alignment.
 *   - Supported shapes: head_k_dim in {32, 64, 128, 256}; head_v_dim a
 *     multiple of 32 up to 512; num_v_heads a multiple of num_k_heads; conv
 *     kernel 1..8; for decode either head_k_dim in {64, 128} with head_v_dim
 *     a multiple of 128, or (head_v_dim/32) * (num_v_heads/num_k_heads) <= 16.
 *     Others return GDN_ERR_UNSUPPORTED.
 *   - With conv_kernel K = 1 the conv state is empty and its pointers may be
 *     NULL.
 *   - The output is fp32, token-major [.., L, Hv, dv]: the layout the next
 *     step of the layer (gated RMSNorm over value_dim, section 2) reads.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *gdn_stream_t; /* a cudaStream_t */

typedef enum {
    GDN_OK = 0,
    GDN_ERR_NULL = 1,           /* a required pointer is NULL */
    GDN_ERR_SHAPE = 2,          /* a size is negative, zero where it must not be, or inconsistent */
    GDN_ERR_ALIGN = 3,          /* a pointer is not aligned as required */
    GDN_ERR_DTYPE = 4,          /* io_dtype is not a gdn_dtype_t */
    GDN_ERR_SEQLENS = 5,        /* cu_seqlens does not start at 0 or is not non-decreasing */
    GDN_ERR_CUDA = 6,           /* a CUDA launch failed; see gdn_last_cuda_error() */
    GDN_ERR_DEVICE_TIMEOUT = 7, /* a bounded device-side wait gave up (see gdn_device_error) */
    GDN_ERR_UNSUPPORTED = 8,    /* valid but not built (head size, GQA ratio, variant) */
    GDN_ERR_WORKSPACE = 9,      /* workspace missing or smaller than gdn_prefill_workspace_size() */
    GDN_ERR_RANGE = 10          /* device-side: an accepted length outside [0, L] */
} gdn_status_t;

typedef enum { GDN_BF16 = 0, GDN_F32 = 1 } gdn_dtype_t;

/* The operator record: MNN's LinearAttentionParam (section 1.4: num_k_heads,
 * num_v_heads, head_k_dim, head_v_dim, use_qk_l2norm) plus the conv width, the
 * L2-norm epsilon and the storage type of qkv, conv_weight and the conv state. */
typedef struct {
    int32_t num_k_heads;
    int32_t num_v_heads;
    int32_t head_k_dim;
    int32_t head_v_dim;
    int32_t conv_kernel;   /* K */
    int32_t use_qk_l2norm; /* 0 or 1 */
    float l2norm_eps;      /* eps in x / sqrt(sum x^2 + eps); 1e-6 is the usual value */
    int32_t io_dtype;      /* gdn_dtype_t */
    /* Gate parameterisation (section 1.2, "gate is carefully parameterized").
     * Both NULL: the `gate` and `beta` arguments of every call are the log-decay
     * g_t (<= 0) and the rate beta_t themselves.  Both set: they are the raw
     * projections a_t and b_t, and the kernels form, per value head h,
     *   gate = -exp(A_log[h]) * softplus(a + dt_bias[h]),  beta = sigmoid(b),
     * with softplus(x) = log(1 + e^x) (x itself above 20).  Device arrays of
     * num_v_heads fp32, 4-byte aligned, caller-owned, read by every call that
     * uses the config.  Only one of the two set: GDN_ERR_NULL. */
    const float *A_log;
    const float *dt_bias;
} gdn_config_t;

/* Prefill variants. */
#define GDN_PREFILL_RESIDENT 0 /* state held on chip across each sequence */
#define GDN_PREFILL_CHUNKED 1  /* chunked (WY/UT) form on tensor cores */

/*
 * Zero both persistent states (section 1.4: states start at zero on the first
 * inference step).  conv_state: device [batch, D, K-1] io dtype; ssm_state:
 * device [batch, Hv, dk, dv] fp32.  Either pointer may be NULL to skip it.
 */
gdn_status_t gdn_conv_state_init(const gdn_config_t *cfg, int32_t batch,
                                 void *conv_state, float *ssm_state,
                                 gdn_stream_t stream);

/*
 * One decode step (L = 1) for `batch` independent sequences: all five steps of
 * section 1.2 for one new token each, with both states updated in place.
 *   qkv         device [batch, D] io dtype (16-byte aligned)
 *   conv_weight device [D, K] io dtype (the [D, 1, K] weight)
 *   gate, beta  device [batch, Hv] fp32; gate <= 0 is expected (exp(gate) is the decay)
 *   conv_state  device [batch, D, K-1] io dtype, read and rewritten in place
 *   ssm_state   device [batch, Hv, dk, dv] fp32, read and rewritten in place
 *   out         device [batch, Hv, dv] fp32
 * batch = 0 is a no-op.  out must not overlap the inputs or states.
 */
gdn_status_t gdn_forward_decode(const gdn_config_t *cfg, int32_t batch,
                                const void *qkv, const void *conv_weight,
                                const float *gate, const float *beta,
                                void *conv_state, float *ssm_state, float *out,
                                gdn_stream_t stream);

/*
 * Bytes of device workspace gdn_forward_prefill needs for `total_tokens`
 * packed tokens over `num_seqs` sequences with the given variant (0 if the
 * shape is invalid).
 */
size_t gdn_prefill_workspace_size(const gdn_config_t *cfg, int32_t num_seqs,
                                  int64_t total_tokens, int32_t variant);

/*
 * Prefill of `num_seqs` sequences packed back to back: sequence n is tokens
 * [cu[n], cu[n+1]) and runs exactly as if alone, from its own states; the
 * conv window never crosses a sequence boundary.  (MNN "Qwen3.5" page: section
 * 1.2 gives the layer over qkv [B, D, L] with all five steps per token, and
 * section 1.4 the per-sequence conv state [B, D, K-1] and recurrent state
 * [B, H, d_k, d_v] that carry across calls; the pages state no packing, so a
 * packed sequence is read as an independent batch entry of length L_n.)
 *   cu_seqlens       device [num_seqs+1] int32 (same values as the host copy)
 *   cu_seqlens_host  host   [num_seqs+1] int32, cu[0] = 0, non-decreasing;
 *                    used for validation and launch sizing (T = cu[num_seqs])
 *   qkv              device [D, T] io dtype, channel-major (the [1, D, T] view
 *                    of the page's [B, D, L] layout); 16-byte aligned
 *   conv_weight      device [D, K] io dtype
 *   gate, beta       device [T, Hv] fp32
 *   conv_state       device [num_seqs, D, K-1] io dtype, in/out
 *   ssm_state        device [num_seqs, Hv, dk, dv] fp32, in/out
 *   out              device [T, Hv, dv] fp32
 *   variant          GDN_PREFILL_RESIDENT (any supported shape) or
 *                    GDN_PREFILL_CHUNKED (tensor cores; head_k_dim = 128 only,
 *                    GDN_ERR_UNSUPPORTED otherwise)
 *   workspace        device scratch of at least gdn_prefill_workspace_size()
 *                    bytes, 16-byte aligned, not shared with a concurrent call
 * Empty sequences (cu[n] == cu[n+1]) keep their states.  T = 0 is a no-op.
 */
gdn_status_t gdn_forward_prefill(const gdn_config_t *cfg, int32_t num_seqs,
                                 const int32_t *cu_seqlens,
                                 const int32_t *cu_seqlens_host,
                                 const void *qkv, const void *conv_weight,
                                 const float *gate, const float *beta,
                                 void *conv_state, float *ssm_state, float *out,
                                 int32_t variant, void *workspace,
                                 size_t workspace_bytes, gdn_stream_t stream);

/*
 * Prefill with the gated RMSNorm of section 2 ("Gated RMSNorm": the linear
 * attention layer applies attn_out = norm(attn_out, z) right after the
 * recurrence) fused into the output epilogue: as gdn_forward_prefill, but instead
 * of the fp32 output it writes
 *   y    device [T, Hv, dv] io dtype, gdn_gated_rmsnorm of the call's output
 * from z (device [T, Hv, dv] io dtype), norm_weight (device [dv] fp32) and
 * norm_eps.  z, y and norm_weight are 16-byte aligned; y must not overlap the
 * other buffers.  The CTAs that hold one value head's columns form a thread-block
 * cluster and exchange the rows' sums of squares, so the row is normalised without
 * writing the fp32 output to memory.  Both variants; head_v_dim <= 128
 * (GDN_ERR_UNSUPPORTED otherwise: call gdn_forward_prefill, then
 * gdn_gated_rmsnorm).  Workspace, states, sizes and errors as gdn_forward_prefill.
 */
gdn_status_t gdn_forward_prefill_gated(const gdn_config_t *cfg, int32_t num_seqs,
                                       const int32_t *cu_seqlens,
                                       const int32_t *cu_seqlens_host,
                                       const void *qkv, const void *conv_weight,
                                       const float *gate, const float *beta,
                                       void *conv_state, float *ssm_state,
                                       const void *z, const float *norm_weight,
                                       float norm_eps, void *y, int32_t variant,
                                       void *workspace, size_t workspace_bytes,
                                       gdn_stream_t stream);

/*
 * Prefill for callers that cannot allocate device memory.  (The pages have no
 * counterpart: this is a deployment convenience, not part of the layer.)
 *
 * gdn_forward_prefill needs a workspace from the caller.  A caller that runs
 * inside a host framework owning all device memory through its own pool, or a
 * serving loop that may not call cudaMalloc (which can synchronise the device),
 * has no way to provide one.  This entry point runs the same resident prefill
 * (GDN_PREFILL_RESIDENT) with its workspace in a fixed array of
 * GDN_NOALLOC_SCRATCH_BYTES compiled into the library; every GPU that loads
 * the library holds that memory until the process exits.  It calls no
 * allocator.  Arguments, layouts and results are those of gdn_forward_prefill.
 *
 *   - Limit: the call needs gdn_prefill_workspace_size(cfg, num_seqs, T,
 *     GDN_PREFILL_RESIDENT) = T * (4 * D + 64 * Hk) bytes (T =
 *     cu_seqlens_host[num_seqs]) to fit GDN_NOALLOC_SCRATCH_BYTES (at D = 8192,
 *     Hk = 16: T <= 496).  Larger calls return GDN_ERR_WORKSPACE and launch
 *     nothing.
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.  GDN_ERR_CUDA if the lookup
 *     fails.  Under lazy module loading (the CUDA default since 12.2) the
 *     library's device code, this array with it, is loaded on that first
 *     lookup, so the first call on each device can itself allocate device
 *     memory and synchronise.  A caller that needs a steady state without
 *     either makes one warm-up call per device at start-up.
 *   - Sharing: every call on a device uses the same array, which keeps the last
 *     call's contents.  Calls that can overlap on the GPU (different streams
 *     without ordering between them) race on it; order them.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (16u << 20)
gdn_status_t gdn_forward_prefill_noalloc(const gdn_config_t *cfg, int32_t num_seqs,
                                         const int32_t *cu_seqlens,
                                         const int32_t *cu_seqlens_host,
                                         const void *qkv, const void *conv_weight,
                                         const float *gate, const float *beta,
                                         void *conv_state, float *ssm_state, float *out,
                                         gdn_stream_t stream);

/*
 * MTP verify: run L draft tokens per sequence from the live states, which are
 * only read, and write the state after every token so that a rejected suffix
 * can be dropped exactly (the verify forward of an MTP round processes its
 * tokens in sequence, as the mlxcel benchmark notes observe for GDN targets).
 *   qkv         device [batch, D, L] io dtype; gate, beta device [batch, L, Hv] fp32
 *   conv_state  device [batch, D, K-1] (read only); ssm_state device [batch, Hv, dk, dv] (read only)
 *   conv_snap   device [batch, L, D, K-1] io dtype: conv state after tokens 0..t
 *   ssm_snap    device [batch, L, Hv, dk, dv] fp32: recurrent state after tokens 0..t
 *   out         device [batch, L, Hv, dv] fp32
 * 1 <= L <= 16.  Snapshot t is bitwise equal to the state t+1 calls of
 * gdn_forward_decode would leave.
 */
gdn_status_t gdn_forward_verify(const gdn_config_t *cfg, int32_t batch, int32_t L,
                                const void *qkv, const void *conv_weight,
                                const float *gate, const float *beta,
                                const void *conv_state, const float *ssm_state,
                                void *conv_snap, float *ssm_snap, float *out,
                                gdn_stream_t stream);

/*
 * Commit an MTP round: sequence b keeps the first accepted[b] draft tokens.
 * (mlxcel benchmark notes, "MTP speculative decoding": the target verifies a
 * drafted block in one forward pass and keeps the accepted prefix, the
 * "accepted draft tokens per verify"; the recurrent and conv states must then
 * be those after the last accepted token, which this call restores from the
 * verify's snapshots.)
 * accepted[b] = a in 1..L copies snapshot a-1 into the live conv and recurrent
 * states; a = 0 leaves them as they were before the verify.
 *   accepted  device [batch] int32
 *   status    device int32, optional: set to GDN_ERR_RANGE if some
 *             accepted[b] is outside [0, L] (that sequence is left untouched);
 *             never written otherwise, so the caller zeroes it first.
 */
gdn_status_t gdn_verify_commit(const gdn_config_t *cfg, int32_t batch, int32_t L,
                               const int32_t *accepted, const void *conv_snap,
                               const float *ssm_snap, void *conv_state,
                               float *ssm_state, int32_t *status,
                               gdn_stream_t stream);

/*
 * Gated RMSNorm of the layer output (section 2, "Gated RMSNorm", as the linear
 * attention layer applies it: attn_out = norm(attn_out, z)).  For every row r
 * (one token of one value head):
 *   y[r][j] = weight[j] * o[r][j] / sqrt(mean_i o[r][i]^2 + eps) * silu(z[r][j]),
 * silu(x) = x / (1 + e^-x); the norm runs over head_v_dim, the last axis of
 * the output as laid out ([.., Hv, dv]), and weight is shared by the heads.
 *   rows     number of rows: tokens * num_v_heads (0 is a no-op)
 *   o        device [rows, dv] fp32 (the output of any forward call), 16-byte aligned
 *   z        device [rows, dv] io dtype (the gate projection), 16-byte aligned
 *   weight   device [dv] fp32, 16-byte aligned
 *   eps      >= 0
 *   y        device [rows, dv] io dtype (bf16 output for bf16 io), 16-byte aligned;
 *            may be o itself only for fp32 io
 */
gdn_status_t gdn_gated_rmsnorm(const gdn_config_t *cfg, int64_t rows, const float *o,
                               const void *z, const float *weight, float eps, void *y,
                               gdn_stream_t stream);

/*
 * A decode step with the gated RMSNorm fused into the output epilogue: as
 * gdn_forward_decode, but instead of the fp32 output it writes
 *   y    device [batch, Hv, dv] io dtype, gdn_gated_rmsnorm of the step's output
 * from z (device [batch, Hv, dv] io dtype), norm_weight (device [dv] fp32) and
 * norm_eps.  Built for the persistent decode kernel with head_v_dim = 128 (one
 * state tile per value head holds the whole row being normalised); other shapes
 * return GDN_ERR_UNSUPPORTED (call gdn_forward_decode, then gdn_gated_rmsnorm).
 */
gdn_status_t gdn_forward_decode_gated(const gdn_config_t *cfg, int32_t batch,
                                      const void *qkv, const void *conv_weight,
                                      const float *gate, const float *beta,
                                      void *conv_state, float *ssm_state,
                                      const void *z, const float *norm_weight,
                                      float norm_eps, void *y, gdn_stream_t stream);

/* Static description of a status code. */
const char *gdn_status_string(gdn_status_t status);

/* CUDA error code (cudaError_t) behind the calling thread's last GDN_ERR_CUDA. */
int32_t gdn_last_cuda_error(void);

/*
 * Diagnostic, synchronous: read (and with clear != 0, reset) the library's
 * device-side error word of the current device.  Kernels never wait without a
 * bound: a wait on an asynchronous copy that gives up sets the word to
 * GDN_ERR_DEVICE_TIMEOUT and the kernel returns early, leaving that call's
 * outputs incomplete.  0 means no such event since the last reset.
 */
gdn_status_t gdn_device_error(int32_t *value, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
