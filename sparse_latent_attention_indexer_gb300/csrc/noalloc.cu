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
// only a host-side stand-in for the symbol, not a device address, so every
// call looks up the device address with cudaGetSymbolAddress, with the call's
// device current.  Once the module is loaded on a device that lookup is a
// host-side table read; looking it up per call (instead of caching it) keeps
// the address right after the caller resets the device.
//
// When the array is reserved: it is part of this library's device code, which
// CUDA loads on a device lazily by default -- at the first use of the module
// there, i.e. the first call of this entry point on that device (a call with no
// query rows does this set-up too and launches nothing).  A caller that hands
// the rest of HBM to its own pool must make that first call before carving the
// pool, or run with CUDA_MODULE_LOADING=EAGER (modules loaded with the context).
#include "dsa_common.cuh"

namespace dsa {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.
int scratch_on_current_device(void **out) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda(e);
    *out = p;
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
    if (rc) return rc;
    // Every byte of the scratch that the attention reads is written earlier in
    // the same call, so nothing has to be cleared between calls.
    if (mla_workspace_bytes(H, d_c, bt.total_q) > (size_t)DSA_NOALLOC_SCRATCH_BYTES) return DSA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if ((rc = scratch_on_current_device(&scratch))) return rc;
    if (bt.total_q == 0) return DSA_OK;  // set-up only
    return run_mla(q_nope, q_pe, dtype, kv_cache, ld_kv, k_pe, ld_pe, W_UK, W_UV, H, d_n, d_r, d_c, d_v, idx, k, bt,
                   softmax_scale, out, lse, (char *)scratch, (cudaStream_t)stream);
}
