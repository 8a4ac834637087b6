// gdn_api.cu -- the C ABI declared in include/gdn.h: argument validation on
// the host, then kernel launches on the caller's stream.  No compute entry point
// allocates, synchronises or copies on the host (gdn_device_error, a diagnostic,
// is the one synchronous call).
#include <cmath>
#include <cstdint>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

thread_local int32_t g_last_cuda_error = 0;

gdn_status_t cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return GDN_OK;
    g_last_cuda_error = (int32_t)e;
    return GDN_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t elem_bytes(const gdn_config_t* c) { return c->io_dtype == GDN_BF16 ? 2 : 4; }

// Checks every field of the operator record; fills the kernel geometry.
gdn_status_t check_config(const gdn_config_t* c, gdn::Geom* g) {
    if (!c) return GDN_ERR_NULL;
    if (c->io_dtype != GDN_BF16 && c->io_dtype != GDN_F32) return GDN_ERR_DTYPE;
    if (c->num_k_heads <= 0 || c->num_v_heads <= 0 || c->head_k_dim <= 0 || c->head_v_dim <= 0 ||
        c->conv_kernel <= 0 || (c->use_qk_l2norm != 0 && c->use_qk_l2norm != 1) || !(c->l2norm_eps >= 0.f) ||
        !std::isfinite(c->l2norm_eps))
        return GDN_ERR_SHAPE;
    if (c->num_v_heads % c->num_k_heads != 0) return GDN_ERR_UNSUPPORTED;
    if (c->head_k_dim != 32 && c->head_k_dim != 64 && c->head_k_dim != 128 && c->head_k_dim != 256)
        return GDN_ERR_UNSUPPORTED;
    if (c->head_v_dim % 32 != 0 || c->head_v_dim > 512) return GDN_ERR_UNSUPPORTED;
    if (c->conv_kernel > 8) return GDN_ERR_UNSUPPORTED;
    const long long D = 2LL * c->num_k_heads * c->head_k_dim + (long long)c->num_v_heads * c->head_v_dim;
    if (D > (1LL << 30)) return GDN_ERR_SHAPE;
    g->Hk = c->num_k_heads;
    g->Hv = c->num_v_heads;
    g->dk = c->head_k_dim;
    g->dv = c->head_v_dim;
    g->K = c->conv_kernel;
    g->D = (int)D;
    g->f = c->num_v_heads / c->num_k_heads;
    g->use_l2 = c->use_qk_l2norm;
    g->eps = c->l2norm_eps;
    g->q_scale = (float)(1.0 / std::sqrt((double)c->head_k_dim));
    g->io_bf16 = c->io_dtype == GDN_BF16;
    if ((c->A_log == nullptr) != (c->dt_bias == nullptr)) return GDN_ERR_NULL;
    if (c->A_log && (!aligned(c->A_log, 4) || !aligned(c->dt_bias, 4))) return GDN_ERR_ALIGN;
    return GDN_OK;
}

}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status_t s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_ERR_NULL: return "a required pointer is NULL";
        case GDN_ERR_SHAPE: return "invalid or inconsistent size";
        case GDN_ERR_ALIGN: return "pointer not aligned as required";
        case GDN_ERR_DTYPE: return "unknown io dtype";
        case GDN_ERR_SEQLENS: return "cu_seqlens must start at 0 and be non-decreasing";
        case GDN_ERR_CUDA: return "CUDA launch failed";
        case GDN_ERR_DEVICE_TIMEOUT: return "bounded device-side wait gave up";
        case GDN_ERR_UNSUPPORTED: return "shape or variant not supported by this library";
        case GDN_ERR_WORKSPACE: return "workspace missing or too small";
        case GDN_ERR_RANGE: return "accepted length outside [0, L]";
    }
    return "unknown status";
}

int32_t gdn_last_cuda_error(void) { return g_last_cuda_error; }

gdn_status_t gdn_device_error(int32_t* value, int32_t clear) {
    if (!value) return GDN_ERR_NULL;
    int32_t a = 0, b = 0, c = 0;
    gdn_status_t st = cuda_status(gdn::stream_error_read(&a, clear != 0));
    if (st != GDN_OK) return st;
    st = cuda_status(gdn::chunk_error_read(&b, clear != 0));
    if (st != GDN_OK) return st;
    st = cuda_status(gdn::prefill_error_read(&c, clear != 0));
    *value = a ? a : b ? b : c;
    return st;
}

gdn_status_t gdn_conv_state_init(const gdn_config_t* cfg, int32_t batch, void* conv_state, float* ssm_state,
                                 gdn_stream_t stream) {
    gdn::Geom g;
    gdn_status_t st = check_config(cfg, &g);
    if (st != GDN_OK) return st;
    if (batch < 0) return GDN_ERR_SHAPE;
    if (conv_state && !aligned(conv_state, elem_bytes(cfg))) return GDN_ERR_ALIGN;
    if (ssm_state && !aligned(ssm_state, 4)) return GDN_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (conv_state) {
        st = cuda_status(gdn::launch_zero(conv_state, (size_t)batch * g.D * (g.K - 1) * elem_bytes(cfg), s));
        if (st != GDN_OK) return st;
    }
    if (ssm_state) return cuda_status(gdn::launch_zero(ssm_state, (size_t)batch * g.Hv * g.dk * g.dv * 4, s));
    return GDN_OK;
}

gdn_status_t gdn_forward_decode(const gdn_config_t* cfg, int32_t batch, const void* qkv, const void* conv_weight,
                                const float* gate, const float* beta, void* conv_state, float* ssm_state, float* out,
                                gdn_stream_t stream) {
    gdn::Geom g;
    gdn_status_t st = check_config(cfg, &g);
    if (st != GDN_OK) return st;
    if (batch < 0 || batch > 65535) return GDN_ERR_SHAPE;
    {
        gdn::StepArgs probe{};
        probe.g = g;
        probe.B = batch;
        probe.L = 1;
        int ns = 0;
        size_t sm = 0;
        if (!gdn::stream_step_supported(probe, &ns, &sm) && !gdn::slice_step_supported(g)) return GDN_ERR_UNSUPPORTED;
    }
    if (batch == 0) return GDN_OK;
    if (!qkv || !conv_weight || !gate || !beta || (!conv_state && g.K > 1) || !ssm_state || !out) return GDN_ERR_NULL;
    const size_t eb = elem_bytes(cfg);
    if (!aligned(qkv, 16) || !aligned(ssm_state, 16) || !aligned(out, 16) || !aligned(conv_weight, eb) ||
        !aligned(conv_state, eb) || !aligned(gate, 4) || !aligned(beta, 4))
        return GDN_ERR_ALIGN;
    gdn::StepArgs a{};
    a.g = g;
    a.B = batch;
    a.L = 1;
    a.qkv = qkv;
    a.w = conv_weight;
    a.gate = gate;
    a.beta = beta;
    a.conv_in = conv_state;
    a.S_in = ssm_state;
    a.conv_out = conv_state;
    a.S_out = ssm_state;
    a.out = out;
    return cuda_status(gdn::launch_step(a, gdn::GateParams{cfg->A_log, cfg->dt_bias}, true, reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status_t gdn_gated_rmsnorm(const gdn_config_t* cfg, int64_t rows, const float* o, const void* z,
                               const float* weight, float eps, void* y, gdn_stream_t stream) {
    gdn::Geom g;
    gdn_status_t st = check_config(cfg, &g);
    if (st != GDN_OK) return st;
    if (rows < 0 || !(eps >= 0.f) || !std::isfinite(eps)) return GDN_ERR_SHAPE;
    if (rows == 0) return GDN_OK;
    if (!o || !z || !weight || !y) return GDN_ERR_NULL;
    if (!aligned(o, 16) || !aligned(z, 16) || !aligned(weight, 16) || !aligned(y, 16)) return GDN_ERR_ALIGN;
    return cuda_status(gdn::launch_gated_rmsnorm(g, rows, o, z, weight, eps, y, reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status_t gdn_forward_decode_gated(const gdn_config_t* cfg, int32_t batch, const void* qkv, const void* conv_weight,
                                      const float* gate, const float* beta, void* conv_state, float* ssm_state,
                                      const void* z, const float* norm_weight, float norm_eps, void* y,
                                      gdn_stream_t stream) {
    gdn::Geom g;
    gdn_status_t st = check_config(cfg, &g);
    if (st != GDN_OK) return st;
    if (batch < 0 || batch > 65535 || !(norm_eps >= 0.f) || !std::isfinite(norm_eps)) return GDN_ERR_SHAPE;
    {
        gdn::StepArgs probe{};
        probe.g = g;
        probe.B = batch;
        probe.L = 1;
        int ns = 0;
        size_t sm = 0;
        if (g.dv != 128 || !gdn::stream_step_supported(probe, &ns, &sm)) return GDN_ERR_UNSUPPORTED;
    }
    if (batch == 0) return GDN_OK;
    if (!qkv || !conv_weight || !gate || !beta || (!conv_state && g.K > 1) || !ssm_state || !z || !norm_weight || !y)
        return GDN_ERR_NULL;
    const size_t eb = elem_bytes(cfg);
    if (!aligned(qkv, 16) || !aligned(ssm_state, 16) || !aligned(z, 16) || !aligned(y, 16) || !aligned(norm_weight, 16) ||
        !aligned(conv_weight, eb) || !aligned(conv_state, eb) || !aligned(gate, 4) || !aligned(beta, 4))
        return GDN_ERR_ALIGN;
    gdn::StepArgs a{};
    a.g = g;
    a.B = batch;
    a.L = 1;
    a.qkv = qkv;
    a.w = conv_weight;
    a.gate = gate;
    a.beta = beta;
    a.conv_in = conv_state;
    a.S_in = ssm_state;
    a.conv_out = conv_state;
    a.S_out = ssm_state;
    a.out = nullptr;
    const gdn::NormParams np{z, norm_weight, norm_eps, y};
    return cuda_status(gdn::launch_step(a, gdn::GateParams{cfg->A_log, cfg->dt_bias}, true,
                                        reinterpret_cast<cudaStream_t>(stream), np));
}

gdn_status_t gdn_forward_verify(const gdn_config_t* cfg, int32_t batch, int32_t L, const void* qkv,
                                const void* conv_weight, const float* gate, const float* beta,
                                const void* conv_state, const float* ssm_state, void* conv_snap, float* ssm_snap,
                                float* out, gdn_stream_t stream) {
    gdn::Geom g;
    gdn_status_t st = check_config(cfg, &g);
    if (st != GDN_OK) return st;
    if (batch < 0 || batch > 65535 || L < 1 || L > 16) return GDN_ERR_SHAPE;
    if (batch == 0) return GDN_OK;
    if (!qkv || !conv_weight || !gate || !beta || (g.K > 1 && (!conv_state || !conv_snap)) || !ssm_state ||
        !ssm_snap || !out)
        return GDN_ERR_NULL;
    const size_t eb = elem_bytes(cfg);
    if (!aligned(qkv, 16) || !aligned(ssm_state, 16) || !aligned(ssm_snap, 16) || !aligned(out, 16) ||
        !aligned(conv_weight, eb) || !aligned(conv_state, eb) || !aligned(conv_snap, eb) || !aligned(gate, 4) ||
        !aligned(beta, 4))
        return GDN_ERR_ALIGN;
    gdn::StepArgs a{};
    a.g = g;
    a.B = batch;
    a.L = L;
    a.qkv = qkv;
    a.w = conv_weight;
    a.gate = gate;
    a.beta = beta;
    a.conv_in = conv_state;
    a.S_in = ssm_state;
    a.conv_out = conv_snap;
    a.S_out = ssm_snap;
    a.out = out;
    return cuda_status(gdn::launch_step(a, gdn::GateParams{cfg->A_log, cfg->dt_bias}, false, reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status_t gdn_verify_commit(const gdn_config_t* cfg, int32_t batch, int32_t L, const int32_t* accepted,
                               const void* conv_snap, const float* ssm_snap, void* conv_state, float* ssm_state,
                               int32_t* status, gdn_stream_t stream) {
    gdn::Geom g;
    gdn_status_t st = check_config(cfg, &g);
    if (st != GDN_OK) return st;
    if (batch < 0 || batch > 65535 || L < 1 || L > 16) return GDN_ERR_SHAPE;
    if (batch == 0) return GDN_OK;
    if (!accepted || (g.K > 1 && (!conv_snap || !conv_state)) || !ssm_snap || !ssm_state) return GDN_ERR_NULL;
    const size_t eb = elem_bytes(cfg);
    if (!aligned(accepted, 4) || !aligned(ssm_snap, 16) || !aligned(ssm_state, 16) || !aligned(conv_snap, eb) ||
        !aligned(conv_state, eb) || (status && !aligned(status, 4)))
        return GDN_ERR_ALIGN;
    gdn::CommitArgs a{};
    a.B = batch;
    a.L = L;
    a.conv_bytes = (size_t)g.D * (g.K - 1) * eb;
    a.ssm_floats = (size_t)g.Hv * g.dk * g.dv;
    a.conv_vec16 = (a.conv_bytes % 16 == 0) && aligned(conv_snap, 16) && aligned(conv_state, 16);
    a.accepted = accepted;
    a.conv_snap = conv_snap;
    a.ssm_snap = ssm_snap;
    a.conv_state = conv_state;
    a.ssm_state = ssm_state;
    a.status = status;
    return cuda_status(gdn::launch_commit(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t gdn_prefill_workspace_size(const gdn_config_t* cfg, int32_t num_seqs, int64_t total_tokens, int32_t variant) {
    gdn::Geom g;
    if (check_config(cfg, &g) != GDN_OK || num_seqs < 0 || total_tokens < 0) return 0;
    if (variant == GDN_PREFILL_RESIDENT) return gdn::prefill_resident_workspace(g, num_seqs, total_tokens);
    if (variant == GDN_PREFILL_CHUNKED && gdn::prefill_chunked_supported(g))
        return gdn::prefill_chunked_workspace_bound(g, num_seqs, total_tokens);
    return 0;
}

namespace {
// Shared by gdn_forward_prefill and gdn_forward_prefill_gated: np.z set writes the
// gated-RMSNorm output y instead of out.
gdn_status_t prefill_call(const gdn_config_t* cfg, int32_t num_seqs, const int32_t* cu_seqlens,
                          const int32_t* cu_seqlens_host, const void* qkv, const void* conv_weight, const float* gate,
                          const float* beta, void* conv_state, float* ssm_state, float* out, int32_t variant,
                          void* workspace, size_t workspace_bytes, gdn_stream_t stream, const gdn::NormParams& np) {
    gdn::Geom g;
    gdn_status_t st = check_config(cfg, &g);
    if (st != GDN_OK) return st;
    if (num_seqs < 0 || num_seqs > 65535) return GDN_ERR_SHAPE;
    if (variant != GDN_PREFILL_RESIDENT && variant != GDN_PREFILL_CHUNKED) return GDN_ERR_SHAPE;
    if (num_seqs == 0) return GDN_OK;
    if (!cu_seqlens || !cu_seqlens_host) return GDN_ERR_NULL;
    if (cu_seqlens_host[0] != 0) return GDN_ERR_SEQLENS;
    int max_len = 0;
    for (int n = 0; n < num_seqs; ++n) {
        const int32_t len = cu_seqlens_host[n + 1] - cu_seqlens_host[n];
        if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return GDN_ERR_SEQLENS;
        if (len > max_len) max_len = len;
    }
    const int64_t T = cu_seqlens_host[num_seqs];
    if (T == 0) return GDN_OK;
    if (variant == GDN_PREFILL_CHUNKED && !gdn::prefill_chunked_supported(g)) return GDN_ERR_UNSUPPORTED;
    if (np.z && !gdn::prefill_norm_supported(g, variant)) return GDN_ERR_UNSUPPORTED;
    if (!qkv || !conv_weight || !gate || !beta || (!conv_state && g.K > 1) || !ssm_state || (!out && !np.z))
        return GDN_ERR_NULL;
    if (np.z && (!np.weight || !np.y)) return GDN_ERR_NULL;
    const size_t eb = elem_bytes(cfg);
    if (!aligned(cu_seqlens, 4) || !aligned(qkv, 16) || !aligned(ssm_state, 16) || !aligned(out, 16) ||
        !aligned(conv_weight, eb) || !aligned(conv_state, eb) || !aligned(gate, 4) || !aligned(beta, 4) ||
        !aligned(np.z, 16) || !aligned(np.y, 16) || !aligned(np.weight, 16))
        return GDN_ERR_ALIGN;
    const size_t need = gdn_prefill_workspace_size(cfg, num_seqs, T, variant);
    if (need > 0 && (!workspace || workspace_bytes < need)) return GDN_ERR_WORKSPACE;
    if (workspace && !aligned(workspace, 16)) return GDN_ERR_ALIGN;
    gdn::PrefillArgs a{};
    a.g = g;
    a.N = num_seqs;
    a.T = (int)T;
    a.max_len = max_len;
    a.cu = cu_seqlens;
    a.cu_host = cu_seqlens_host;
    a.qkv = qkv;
    a.w = conv_weight;
    a.gate = gate;
    a.beta = beta;
    a.conv_state = conv_state;
    a.ssm_state = ssm_state;
    a.out = out;
    a.ws = workspace;
    a.ws_bytes = workspace_bytes;
    a.norm = np;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const gdn::GateParams gp{cfg->A_log, cfg->dt_bias};
    return cuda_status(variant == GDN_PREFILL_CHUNKED ? gdn::launch_prefill_chunked(a, gp, s)
                                                      : gdn::launch_prefill_resident(a, gp, s));
}
}  // namespace

gdn_status_t gdn_forward_prefill(const gdn_config_t* cfg, int32_t num_seqs, const int32_t* cu_seqlens,
                                 const int32_t* cu_seqlens_host, const void* qkv, const void* conv_weight,
                                 const float* gate, const float* beta, void* conv_state, float* ssm_state, float* out,
                                 int32_t variant, void* workspace, size_t workspace_bytes, gdn_stream_t stream) {
    return prefill_call(cfg, num_seqs, cu_seqlens, cu_seqlens_host, qkv, conv_weight, gate, beta, conv_state,
                        ssm_state, out, variant, workspace, workspace_bytes, stream, gdn::NormParams{});
}

gdn_status_t gdn_forward_prefill_gated(const gdn_config_t* cfg, int32_t num_seqs, const int32_t* cu_seqlens,
                                       const int32_t* cu_seqlens_host, const void* qkv, const void* conv_weight,
                                       const float* gate, const float* beta, void* conv_state, float* ssm_state,
                                       const void* z, const float* norm_weight, float norm_eps, void* y,
                                       int32_t variant, void* workspace, size_t workspace_bytes,
                                       gdn_stream_t stream) {
    if (!(norm_eps >= 0.f) || !std::isfinite(norm_eps)) return GDN_ERR_SHAPE;
    if (!z || !norm_weight || !y) return GDN_ERR_NULL;
    return prefill_call(cfg, num_seqs, cu_seqlens, cu_seqlens_host, qkv, conv_weight, gate, beta, conv_state,
                        ssm_state, nullptr, variant, workspace, workspace_bytes, stream,
                        gdn::NormParams{z, norm_weight, norm_eps, y});
}

}  // extern "C"
