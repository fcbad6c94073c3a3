// Shared internals of libdsa: the per-launch sequence table, element loads,
// launch bookkeeping and the declarations of every kernel launcher.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dsa.h"

namespace dsa {

// Sequence table passed BY VALUE in kernel parameters (about 6 KB), so the
// library needs no device copy of the batch description.
struct SeqTab {
    int B;
    int q_off[DSA_MAX_SEQS + 1];  // cumulative query rows of the launch
    int k_base[DSA_MAX_SEQS];     // first cache row of each sequence
    int k_len[DSA_MAX_SEQS];      // keys of each sequence
    int start_pos[DSA_MAX_SEQS];  // position of each sequence's first row in this launch
};
static_assert(sizeof(SeqTab) + 1024 <= 32764, "a sequence table travels in a kernel's launch parameters");

// Largest b with q_off[b] <= r: the sequence that owns query row r (empty
// sequences are skipped because their successor has the same offset).
__device__ __forceinline__ int seq_of_row(const SeqTab &st, int r) {
    int lo = 0, hi = st.B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (st.q_off[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Per-row facts every stage needs.
struct RowInfo {
    int b;      // sequence
    int t;      // query index within the sequence
    int p;      // absolute position
    int S;      // keys of the sequence
    int kbase;  // first cache row of the sequence
};

__device__ __forceinline__ RowInfo row_info(const SeqTab &st, int r) {
    RowInfo ri;
    ri.b = seq_of_row(st, r);
    ri.t = r - st.q_off[ri.b];
    ri.p = st.start_pos[ri.b] + ri.t;
    ri.kbase = st.k_base[ri.b];
    ri.S = st.k_len[ri.b];
    return ri;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Exponent e of the ue8m0 block scale 2^e: the smallest integer with amax <= 448 * 2^e, clamped to
// the ue8m0 range (amax = 0 gives 0).  With amax = m * 2^E, m in [0.5, 1) and 448 = 0.875 * 2^9:
// e = E - 9 when m <= 0.875, else E - 8.  Exact for every finite fp32 amax.
__device__ __forceinline__ int ue8m0_exponent(float amax) {
    if (!(amax > 0.0f)) return 0;
    int E;
    float m = frexpf(amax, &E);
    int e = (m <= 0.875f) ? E - 9 : E - 8;
    return max(-127, min(127, e));
}

// Order-preserving map of an fp32 score to uint32 (larger float -> larger
// key); -0 is folded onto +0 first so equal values get equal keys.
__device__ __forceinline__ uint32_t ordered_key(float f) {
    f = f + 0.0f;
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------
// Host-side bookkeeping and shared host logic (dsa_api.cu)
// ---------------------------------------------------------------------------
void note_launch(uint32_t kernel_bit);

// Programmatic dependent launch: the kernel may be scheduled while the kernel before it on the
// stream drains (its on-chip set-up overlaps that tail).  Such a kernel executes pdl_wait() in
// every thread before its first global-memory access, which waits for the previous grid to
// complete and its writes to be visible, and pdl_trigger() in every thread once it needs no more
// SM resources for new work, which lets the next kernel be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}
void reset_trace();
int fail_cuda(cudaError_t e);

// Wait limit of the tensor-core kernels' bounded waits, in SM clock cycles: about two seconds by
// default; dsa_set_wait_limit changes it for the launches that follow (the waits that drain copies
// and MMAs already in flight keep the default).
constexpr long long kDefaultWaitLimitCycles = 4LL << 30;
long long wait_limit_cycles();
// Streaming multiprocessors of the current device (152 on a GB300).
int device_sm_count();

// A validated batch: the kernel table for all rows plus summary sizes.
struct Batch {
    SeqTab st;
    int total_q = 0;
    int64_t total_k = 0;
    int max_S = 0;
};
int build_batch(const dsa_seqs *s, Batch &b);
int check_mla_shape(int dtype, int H, int d_n, int d_r, int d_c, int d_v, int k);

// Scratch layout of the attention stage.
struct MlaWs {
    size_t qt = 0, olat = 0, part = 0, total = 0;
};
MlaWs mla_ws_layout(int H, int d_c, int64_t total_q);
size_t mla_workspace_bytes(int H, int d_c, int64_t total_q);
// Every host-side check of dsa_sparse_mla_fwd except the workspace ones.
int validate_mla_call(const void *q_nope, const void *q_pe, int dtype, const void *kv_cache, int64_t ld_kv,
                      const void *k_pe, int64_t ld_pe, const void *W_UK, const void *W_UV, int H, int d_n, int d_r,
                      int d_c, int d_v, const int32_t *idx, int k, const dsa_seqs *seqs, void *out, Batch &bt);
// The attention stage (q~ absorb, sparse attention, W_UV) with scratch `ws`.
int run_mla(const void *q_nope, const void *q_pe, int dtype, const void *kv, int64_t ld_kv, const void *k_pe,
            int64_t ld_pe, const void *W_UK, const void *W_UV, int H, int d_n, int d_r, int d_c, int d_v,
            const int32_t *idx, int k, const Batch &bt, float scale, void *out, float *lse, char *ws,
            cudaStream_t s, bool mark = false, bool prefix_valid = false, const void *wo = nullptr,
            int d_model = 0, void *y = nullptr, char *obuf = nullptr, const float *kv_scale = nullptr);
// Rows per chunk of the W_UV -> wo sequence: the chunk's [rows, H * d_v] bf16 attention output
// (64 MB at the 671B shapes) is read back by the wo GEMM while it is still in L2.
constexpr int kWoChunkRows = 2048;

// ---------------------------------------------------------------------------
// Kernel launchers.  Each returns the cudaError_t of its launch.
// ---------------------------------------------------------------------------
cudaError_t launch_quant_e4m3(const void *x, int x_dtype, int64_t n_blocks, uint8_t *codes, float *scales,
                              cudaStream_t s);

// Generic SIMT indexer: any H_I <= 128, D_I <= 256; F32, BF16 or E4M3 inputs.
cudaError_t launch_indexer_simt(const void *q, const float *q_scale, const void *k, const float *k_scale,
                                int dtype, const float *w, int H_I, int D_I, const SeqTab &st, int total_q,
                                int max_S, float *scores, int64_t ld, cudaStream_t s);

// tcgen05 indexer for H_I = 64, D_I = 128 (BF16 or E4M3 inputs).
bool indexer_tc_supported(int dtype, int H_I, int D_I);
cudaError_t launch_indexer_tc(const void *q, const float *q_scale, const void *k, const float *k_scale, int dtype,
                              const float *w, const SeqTab &st, int64_t total_k, float *scores, int64_t ld,
                              bool fill_future, cudaStream_t s, int dense_k = 0);
int indexer_tc_read_error(int *site);
// The indexer and the top-k in one persistent kernel (prefill-sized batches): per SM one slot of 4
// fp32 score rows of ld columns (indexer_topk_slot_bytes) instead of a [rows, ld] buffer.
bool indexer_topk_fused_ok(int dtype, int H_I, int D_I, const SeqTab &st, int k);
size_t indexer_topk_slot_bytes(const SeqTab &st, int64_t ld);
cudaError_t launch_indexer_topk_tc(const void *q, const float *q_scale, const void *k, const float *k_scale, int dtype,
                                   const float *w, const SeqTab &st, int64_t total_k, float *slots, int64_t ld,
                                   int topk, int32_t *idx, cudaStream_t s);

// DSA_FORCE_GENERIC=1 in the environment routes every stage to the generic
// CUDA-core kernels (used by the tests to cross-check the tensor-core ones).
bool force_generic();

cudaError_t launch_dense_idx(const SeqTab &st, int total_q, int k, int32_t *idx, cudaStream_t s);
cudaError_t launch_topk(const float *scores, int64_t ld, const SeqTab &st, int total_q, int k, int32_t *idx,
                        cudaStream_t s);

// Batched per-head GEMM C[m, h, :] = A[m, h, :] . B[h] (B row-major K x N).
cudaError_t launch_absorb_simt(const void *A, int a_dtype, int64_t lda_row, const void *Bm, int b_dtype, void *C,
                               int c_dtype, int64_t ldc_row, int M, int H, int K, int N, cudaStream_t s);

// Generic SIMT sparse attention in the latent space: per (row, head) online
// softmax over the selected keys.  qt rows [M, H, qt_ld] (qt_dtype) hold q~ in
// their first d_c columns; q_pe rows [M, H, qpe_ld]; the latent context is
// written [M, H, d_c] as olat_dtype.
cudaError_t launch_mla_simt(const void *qt, int qt_dtype, int qt_ld, const void *q_pe, int qpe_ld, int dtype,
                            const void *kv, int64_t ld_kv, const void *k_pe, int64_t ld_pe, const int32_t *idx, int k,
                            const SeqTab &st, int total_q, int H, int d_r, int d_c, float scale, void *olat,
                            int olat_dtype, float *lse, cudaStream_t s);

// tcgen05 absorption GEMMs (bf16, d_n = 128, d_c = 512, d_v = 128):
// qt [M, H, 512] = q_nope W_UK;  out [M, H, 128] = olat W_UV.
bool absorb_tc_supported(int dtype, int H, int d_n, int d_r, int d_c, int d_v);
cudaError_t launch_absorb_q_tc(const void *q_nope, const void *W_UK, void *qt, int M, int H, cudaStream_t s);
cudaError_t launch_absorb_v_tc(const void *olat, const void *W_UV, void *out, int M, int H, cudaStream_t s);
int absorb_tc_read_error(int *site);

// tcgen05 sparse latent attention (bf16, H = 128, d_c = 512, d_r = 64): q~ rows
// [M, 128, 512] and q_pe rows [M, 128, 64] -> olat [M, 128, 512] bf16 and lse.  Rows with
// few entries per split write fp32 partials to part_ws (mla_tc_partial_bytes)
// and a combine kernel merges them.
bool mla_tc_supported(int dtype, int H, int d_n, int d_r, int d_c, int d_v);
int mla_tc_splits(int M);
size_t mla_tc_partial_bytes(int M);
cudaError_t launch_mla_tc(const void *qt, const void *qpe, const void *kv, int64_t ld_kv, const void *kpe, int64_t ld_pe,
                          const int32_t *idx, int k, const SeqTab &st, int64_t total_k, int M, float scale,
                          bool prefix_valid, void *olat, float *lse, void *part_ws, cudaStream_t s,
                          const float *kv_scale = nullptr);
int mla_tc_read_error(int *site);

// tcgen05 dense GEMM C[M, N] = A[M, K] B[N, K]^T (bf16 in, fp32 accumulation, C bf16 or fp32);
// N and K multiples of 64, rows 16-byte aligned.
bool gemm_tc_supported(int M, int N, int K);
cudaError_t launch_gemm_tc(const void *A, int64_t lda, const void *B, int64_t ldb, void *C, int64_t ldc, bool c_f32,
                           int M, int N, int K, cudaStream_t s);
int gemm_tc_read_error(int *site);

// Bounded-wait self-test (selftest.cu): one CTA whose first wait runs out after limit_cycles.
cudaError_t launch_bounded_wait_selftest(long long limit_cycles, int *completed_ok, cudaStream_t s);
int selftest_read_error(int *site);

}  // namespace dsa
