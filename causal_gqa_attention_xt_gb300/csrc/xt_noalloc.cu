// xt_noalloc.cu -- a backward entry point that allocates nothing.
//
// Some callers cannot hand the library a workspace: a host application that
// owns all device memory through its own pool and offers plugins no way to
// allocate, or a latency-critical loop where cudaMalloc (which may block and
// synchronize the device, and may fail once memory is fragmented) is not
// allowed. For them, xt_attn_bwd_noalloc runs the regular backward with its
// scratch taken from a fixed array of this library's device memory instead
// of a caller-provided workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it until the process exits. On the host its name is only a
// stand-in for the device object, so the device address is fetched once per
// device with cudaGetSymbolAddress (with that device current) and passed to
// the kernels.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/xt_attn.h"

namespace {

// Largest scratch the no-allocation backward can use (bytes).
constexpr size_t kStaticScratchBytes = (size_t)16 << 20;   // 16 MiB

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device, looked up on the
// first call per device.
int static_scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return XT_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return XT_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
            return XT_ECUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return XT_OK;
}

}  // namespace

extern "C" int xt_attn_bwd_noalloc(int B, int S, int n_heads, int n_kv_heads, int head_dim,
                                   double eps, double theta, const void *q, const void *k,
                                   const void *v, const float *gamma_q, const float *gamma_k,
                                   int dtype, const void *out, const float *lse,
                                   const void *q_hat, const void *k_hat, const float *rstd_q,
                                   const float *rstd_k, const void *dout, void *dq, void *dk,
                                   void *dv, float *dgamma_q, float *dgamma_k, void *stream) {
    // Problems whose scratch exceeds the static array are refused up front.
    // (Invalid arguments give a need of 0 and are rejected by xt_attn_bwd.)
    const size_t need = xt_attn_workspace_bytes(B, S, n_heads, n_kv_heads, head_dim, dtype, 1);
    if (need > kStaticScratchBytes) return XT_EWORKSPACE;
    void *scratch = nullptr;
    const int st = static_scratch_address(&scratch);
    if (st != XT_OK) return st;
    // On a call that completes normally every region of the backward's scratch
    // is written before it is read, so the array needs no clearing between
    // calls. A call whose bounded waits run out (xt_attn_check() reports
    // XT_ETIMEOUT) stops writing partway: a later kernel of that call may then
    // read the previous call's scratch, and every output of that call (dq, dk,
    // dv, dgamma_q, dgamma_k) is unspecified.
    return xt_attn_bwd(B, S, n_heads, n_kv_heads, head_dim, eps, theta, q, k, v, gamma_q, gamma_k,
                       dtype, out, lse, q_hat, k_hat, rstd_q, rstd_k, dout, dq, dk, dv, dgamma_q,
                       dgamma_k, scratch, kStaticScratchBytes, stream);
}
