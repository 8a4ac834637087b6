// gdn_internal.h -- launch interfaces between the C-ABI layer (gdn_api.cu) and
// the kernels.  Arguments here are already validated.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

// Geometry shared by every launch.
struct Geom {
    int Hk, Hv, dk, dv, K, D, f;  // f = Hv / Hk
    int use_l2;
    float eps;
    float q_scale;  // 1/sqrt(dk) rounded to fp32
    int io_bf16;    // 1: bf16 storage, 0: fp32 storage
};

// Gate parameterisation (section 1.2): per-value-head A_log and dt_bias, or both
// NULL when the gate/beta inputs are the log-decay and rate themselves.  Passed
// to the kernels as a parameter of its own: the argument structs stay as they are
// (growing StepArgs by these 16 bytes cost the decode kernel about 5 %).
struct GateParams {
    const float* A_log;    // [Hv]
    const float* dt_bias;  // [Hv]
};

// Decode (in place, L = 1) and verify (snapshots, L tokens) share one kernel.
struct StepArgs {
    Geom g;
    int B, L;
    const void* qkv;      // [B, D, L]
    const void* w;        // [D, K]
    const float* gate;    // [B, L, Hv]
    const float* beta;    // [B, L, Hv]
    const void* conv_in;  // [B, D, K-1]
    const float* S_in;    // [B, Hv, dk, dv]
    void* conv_out;       // decode: conv_in; verify: [B, L, D, K-1]
    float* S_out;         // decode: S_in;    verify: [B, L, Hv, dk, dv]
    float* out;           // [B, L, Hv, dv]
};
// Decode / verify.  launch_step picks the persistent TMA-fed kernel
// (gdn_stream.cu) when stream_step_supported() accepts the shape, else the
// cluster-per-key-head slice kernel (gdn_step.cu).
// Gated RMSNorm (section 2) fused into the decode output epilogue: y instead of out.
struct NormParams {
    const void* z;         // [B, Hv, dv] io dtype; NULL: no fused norm
    const float* weight;   // [dv]
    float eps;
    void* y;               // [B, Hv, dv] io dtype
};
cudaError_t launch_step(const StepArgs& a, const GateParams& gp, bool in_place, cudaStream_t stream,
                        const NormParams& np = NormParams{});
bool stream_step_supported(const StepArgs& a, int* nstage, size_t* smem_bytes);
cudaError_t launch_stream_step(const StepArgs& a, const GateParams& gp, bool in_place, cudaStream_t stream,
                               const NormParams& np = NormParams{});
// Standalone gated RMSNorm over rows of dv (gdn_norm.cu).
cudaError_t launch_gated_rmsnorm(const Geom& g, long long rows, const float* o, const void* z, const float* weight,
                                 float eps, void* y, cudaStream_t stream);
bool slice_step_supported(const Geom& g);
cudaError_t stream_error_read(int32_t* value, bool clear);

struct CommitArgs {
    int B, L;
    size_t conv_bytes;    // bytes of one sequence's conv state
    size_t ssm_floats;    // floats of one sequence's recurrent state
    int conv_vec16;       // conv bytes and both conv pointers allow 16-byte copies
    const int32_t* accepted;
    const void* conv_snap;
    const float* ssm_snap;
    void* conv_state;
    float* ssm_state;
    int32_t* status;
};
cudaError_t launch_commit(const CommitArgs& a, cudaStream_t stream);

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t stream);

struct PrefillArgs {
    Geom g;
    int N;                     // sequences
    int T;                     // packed tokens
    int max_len;               // longest sequence
    const int32_t* cu;         // device [N+1]
    const int32_t* cu_host;    // host [N+1]
    const void* qkv;           // [D, T]
    const void* w;             // [D, K]
    const float* gate;         // [T, Hv]
    const float* beta;         // [T, Hv]
    void* conv_state;          // [N, D, K-1]
    float* ssm_state;          // [N, Hv, dk, dv]
    float* out;                // [T, Hv, dv]
    void* ws;                  // workspace
    size_t ws_bytes;
    NormParams norm;           // z set: the gated RMSNorm fused, y written instead of out
};
size_t prefill_resident_workspace(const Geom& g, int N, long long T);
cudaError_t launch_prefill_resident(const PrefillArgs& a, const GateParams& gp, cudaStream_t stream);
// Steps 1-4 for every packed token into token-major normalised fp32 rows y [T, D].
cudaError_t launch_prefill_prep(const PrefillArgs& a, float* y, cudaStream_t stream);

// The gated RMSNorm fused into a prefill form's output epilogue: the CTAs that hold
// one head's columns form a cluster and exchange the rows' sums of squares.
bool prefill_norm_supported(const Geom& g, int variant);
cudaError_t prefill_error_read(int32_t* value, bool clear);

// Chunked (tensor-core) prefill, gdn_chunked.cu.
bool prefill_chunked_supported(const Geom& g);
size_t prefill_chunked_workspace_bound(const Geom& g, int N, long long T);
cudaError_t launch_prefill_chunked(const PrefillArgs& a, const GateParams& gp, cudaStream_t stream);
cudaError_t chunk_error_read(int32_t* value, bool clear);

}  // namespace gdn
