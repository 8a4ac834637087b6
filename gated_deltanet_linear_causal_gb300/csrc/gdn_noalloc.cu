// gdn_noalloc.cu -- a prefill entry point for callers that cannot allocate
// device memory.
//
// gdn_forward_prefill needs a caller-provided workspace.  Some callers cannot
// get one: a host framework that owns all device memory through its own pool
// and forbids outside cudaMalloc, or a latency-critical serving loop that may
// not call the allocator at all (cudaMalloc/cudaFree can synchronise the
// device).  gdn_forward_prefill_noalloc runs the same resident prefill with its
// workspace in a fixed array compiled into this library instead.  The array
// holds GDN_NOALLOC_SCRATCH_BYTES of device memory on every GPU that loads the
// library, until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "gdn.h"

namespace {

// The fixed workspace.  In host code this name is only a stand-in for the
// device array; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the fixed workspace on the current device, looked up once
// per device (with that device current) and cached.
gdn_status_t scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return GDN_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status_t gdn_forward_prefill_noalloc(const gdn_config_t* cfg, int32_t num_seqs,
                                                    const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                                                    const void* qkv, const void* conv_weight, const float* gate,
                                                    const float* beta, void* conv_state, float* ssm_state,
                                                    float* out, gdn_stream_t stream) {
    if (!cfg) return GDN_ERR_NULL;
    if (num_seqs < 0) return GDN_ERR_SHAPE;
    if (num_seqs > 0) {
        if (!cu_seqlens_host) return GDN_ERR_NULL;
        const int64_t T = cu_seqlens_host[num_seqs];
        if (T > 0) {
            const size_t need = gdn_prefill_workspace_size(cfg, num_seqs, T, GDN_PREFILL_RESIDENT);
            if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
        }
    }
    void* scratch = nullptr;
    const gdn_status_t st = scratch_address(&scratch);
    if (st != GDN_OK) return st;
    return gdn_forward_prefill(cfg, num_seqs, cu_seqlens, cu_seqlens_host, qkv, conv_weight, gate, beta, conv_state,
                               ssm_state, out, GDN_PREFILL_RESIDENT, scratch, (size_t)GDN_NOALLOC_SCRATCH_BYTES,
                               stream);
}
