// dsa_sparse_mla_fwd_noalloc: the sparse latent attention with its scratch
// held in a fixed array that is part of the library's device image, for
// callers that cannot hand the library a workspace.
//
// Why it exists: some callers have no way to obtain device memory at the
// point where they run the attention.  A serving runtime that carves all of
// HBM into its own KV-cache pool at start-up leaves nothing for a late
// cudaMalloc (and forbids one, since it would stall every stream on the
// device); a plugin or callback invoked from such a runtime is handed only
// the tensors it reads and writes, never an allocator.  For them this entry
// point takes only inputs and outputs and computes in DSA_NOALLOC_SCRATCH_BYTES
// of scratch that the library reserves once per device.
//
// The scratch is a file-scope __device__ array.  In host code its name is
// only a host-side stand-in for the symbol, not a device address, so the
// device address is looked up with cudaGetSymbolAddress once per device,
// with that device current, on the first call that runs on it, and cached.
#include <mutex>

#include "dsa_common.cuh"

namespace dsa {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on the
// first call per device).
int scratch_on_current_device(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return DSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return fail_cuda(e);
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_sparse_mla_fwd_noalloc(const void *q_nope, const void *q_pe, int dtype, const void *kv_cache,
                                          int64_t ld_kv, const void *k_pe, int64_t ld_pe, const void *W_UK,
                                          const void *W_UV, int H, int d_n, int d_r, int d_c, int d_v,
                                          const int32_t *idx, int k, const dsa_seqs *seqs, float softmax_scale,
                                          void *out, float *lse, void *stream) {
    reset_trace();
    Batch bt;
    int rc = validate_mla_call(q_nope, q_pe, dtype, kv_cache, ld_kv, k_pe, ld_pe, W_UK, W_UV, H, d_n, d_r, d_c, d_v,
                               idx, k, seqs, out, bt);
    if (rc || bt.total_q == 0) return rc;
    // Every byte of the scratch that the attention reads is written earlier in
    // the same call, so nothing has to be cleared between calls.
    if (mla_workspace_bytes(H, d_c, bt.total_q) > (size_t)DSA_NOALLOC_SCRATCH_BYTES) return DSA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if ((rc = scratch_on_current_device(&scratch))) return rc;
    return run_mla(q_nope, q_pe, dtype, kv_cache, ld_kv, k_pe, ld_pe, W_UK, W_UV, H, d_n, d_r, d_c, d_v, idx, k, bt,
                   softmax_scale, out, lse, (char *)scratch, (cudaStream_t)stream);
}
