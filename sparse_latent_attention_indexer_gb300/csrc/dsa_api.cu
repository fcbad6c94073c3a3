// The C ABI of libdsa: argument validation, workspace carving, the row-chunk
// loop of the whole path and the dispatch between the tensor-core kernels and
// the generic ones.  Host code only; every arithmetic step runs in the kernels.
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <map>

#include "dsa_common.cuh"

namespace dsa {

thread_local int g_last_cuda = 0;
thread_local uint32_t g_kernels = 0;
thread_local int g_launches = 0;
thread_local cudaEvent_t g_stage_events[DSA_STAGE_EVENTS] = {};
thread_local bool g_stage_on = false;
// dsa_forward_host: the event that marks its query copies of q_nope and q_pe done on the side stream;
// the attention stage waits for it before its first read of them (null: nothing to wait for).
thread_local cudaEvent_t g_query_in = nullptr;

// Records stage boundary i on `s` when the timing hook is on.
void stage_mark(int i, cudaStream_t s) {
    if (g_stage_on) cudaEventRecord(g_stage_events[i], s);
}

void reset_trace() {
    g_kernels = 0;
    g_launches = 0;
}

bool force_generic() {
    const char *v = getenv("DSA_FORCE_GENERIC");
    return v && v[0] == '1';
}

int fail_cuda(cudaError_t e) {
    g_last_cuda = (int)e;
    return DSA_ERR_CUDA;
}

int device_sm_count() {
    static int n[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (n[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 152;
        n[dev] = v;
    }
    return n[dev];
}

std::atomic<long long> g_wait_limit{kDefaultWaitLimitCycles};
long long wait_limit_cycles() { return g_wait_limit.load(std::memory_order_relaxed); }

namespace {

constexpr size_t WS_ALIGN = 256;
inline size_t align_up(size_t x, size_t a = WS_ALIGN) { return (x + a - 1) / a * a; }
inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

int build_batch(const dsa_seqs *s, Batch &b) {
    if (!s || s->B < 1 || s->B > DSA_MAX_SEQS || !s->cu_q || !s->cu_k || !s->start_pos) return DSA_ERR_INVALID_ARG;
    if (s->cu_q[0] != 0 || s->cu_k[0] != 0) return DSA_ERR_INVALID_ARG;
    memset(&b.st, 0, sizeof(b.st));
    b.st.B = s->B;
    b.max_S = 0;
    for (int i = 0; i < s->B; ++i) {
        const int64_t T = (int64_t)s->cu_q[i + 1] - s->cu_q[i];
        const int64_t S = (int64_t)s->cu_k[i + 1] - s->cu_k[i];
        const int64_t p0 = s->start_pos[i];
        if (T < 0 || S < 0 || p0 < 0 || p0 + T > S) return DSA_ERR_INVALID_ARG;
        b.st.q_off[i] = s->cu_q[i];
        b.st.k_base[i] = s->cu_k[i];
        b.st.k_len[i] = (int)S;
        b.st.start_pos[i] = (int)p0;
        b.max_S = std::max<int>(b.max_S, (int)S);
    }
    b.st.q_off[s->B] = s->cu_q[s->B];
    b.total_q = s->cu_q[s->B];
    b.total_k = s->cu_k[s->B];
    return DSA_OK;
}

namespace {

// The table of rows [r0, r1) of a validated batch: each sequence that overlaps
// the range contributes its overlapping rows, with start_pos advanced to the
// first of them.  Row r of the range is row r - r0 of the table.
void sub_batch(const dsa_seqs *s, int r0, int r1, SeqTab &st, int &max_S) {
    st.B = 0;
    st.q_off[0] = 0;
    max_S = 0;
    for (int b = 0; b < s->B; ++b) {
        const int lo = std::max(s->cu_q[b], r0), hi = std::min(s->cu_q[b + 1], r1);
        if (lo >= hi) continue;
        const int i = st.B++;
        st.q_off[i + 1] = st.q_off[i] + (hi - lo);
        st.k_base[i] = s->cu_k[b];
        st.k_len[i] = s->cu_k[b + 1] - s->cu_k[b];
        st.start_pos[i] = s->start_pos[b] + (lo - s->cu_q[b]);
        max_S = std::max(max_S, st.k_len[i]);
    }
}

bool valid_dtype(int t) { return t == DSA_F32 || t == DSA_BF16 || t == DSA_E4M3; }
size_t dtype_bytes(int t) { return t == DSA_F32 ? 4 : (t == DSA_BF16 ? 2 : 1); }

int check_indexer_shape(int idx_dtype, int H_I, int D_I) {
    if (!valid_dtype(idx_dtype) || H_I < 1 || D_I < 1) return DSA_ERR_INVALID_ARG;
    if (H_I > 128 || D_I > 256) return DSA_ERR_UNSUPPORTED;
    if (idx_dtype == DSA_E4M3 && D_I != 128) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

}  // namespace

int check_mla_shape(int dtype, int H, int d_n, int d_r, int d_c, int d_v, int k) {
    if (H < 1 || d_n < 1 || d_r < 0 || d_c < 1 || d_v < 1 || k < 1) return DSA_ERR_INVALID_ARG;
    if (dtype != DSA_F32 && dtype != DSA_BF16) return DSA_ERR_UNSUPPORTED;
    if (H > 256 || d_n > 256 || d_r > 128 || d_c > 1024 || d_v > 256) return DSA_ERR_UNSUPPORTED;
    // rows of the latent cache must stay 16-byte aligned for vector loads
    if ((d_c * dtype_bytes(dtype)) % 16 != 0) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

void note_launch(uint32_t kernel_bit) {
    g_kernels |= kernel_bit;
    ++g_launches;
}

}  // namespace dsa

using namespace dsa;

namespace dsa {

// Scratch of the attention stage: q~ = q_nope W_UK and the latent context,
// both fp32 [M, H, d_c] on the generic path.
MlaWs mla_ws_layout(int H, int d_c, int64_t total_q) {
    // Generic path: q~ and the latent context in fp32.  Tensor-core path: the
    // bf16 q~ rows and bf16 context fit in the same two regions, plus the split
    // partials of short batches.
    MlaWs w;
    const size_t per = align_up((size_t)total_q * H * d_c * sizeof(float));
    w.qt = 0;
    w.olat = per;
    w.part = 2 * per;
    w.total = w.part + align_up(mla_tc_partial_bytes((int)total_q));
    return w;
}

int run_mla(const void *q_nope, const void *q_pe, int dtype, const void *kv, int64_t ld_kv, const void *k_pe,
            int64_t ld_pe, const void *W_UK, const void *W_UV, int H, int d_n, int d_r, int d_c, int d_v,
            const int32_t *idx, int k, const Batch &bt, float scale, void *out, float *lse, char *ws,
            cudaStream_t s, bool mark, bool prefix_valid, const void *wo, int d_model, void *y, char *obuf,
            const float *kv_scale) {
    const MlaWs L = mla_ws_layout(H, d_c, bt.total_q);
    const int M = bt.total_q;
    if (g_query_in) {  // q_nope and q_pe are still being copied in on dsa_forward_host's side stream
        const cudaError_t ew = cudaStreamWaitEvent(s, g_query_in, 0);
        if (ew != cudaSuccess) return fail_cuda(ew);
    }
    cudaError_t e;
    const bool fast = !force_generic() && absorb_tc_supported(dtype, H, d_n, d_r, d_c, d_v) && aligned(q_nope, 16) &&
                      aligned(q_pe, 16) && aligned(W_UK, 16) && aligned(W_UV, 16) && aligned(out, 16);
    if (kv_scale && !(fast && mla_tc_supported(dtype, H, d_n, d_r, d_c, d_v))) return DSA_ERR_UNSUPPORTED;
    if (fast) {
        // q~ rows [M, H, d_c] bf16 = q_nope W_UK (q_pe is read in place); latent context bf16 [M, H, d_c].
        __nv_bfloat16 *qt = (__nv_bfloat16 *)(ws + L.qt);
        __nv_bfloat16 *olat = (__nv_bfloat16 *)(ws + L.olat);
        e = launch_absorb_q_tc(q_nope, W_UK, qt, M, H, s);
        if (e != cudaSuccess) return fail_cuda(e);
        if (mark) stage_mark(3, s);
        if (kv_scale)  // FP8 latent rows: validated by the caller for the tensor-core kernel
            e = launch_mla_tc(qt, q_pe, kv, ld_kv, k_pe, ld_pe, idx, k, bt.st, bt.total_k, M, scale, prefix_valid, olat,
                              lse, ws + L.part, s, kv_scale);
        else if (mla_tc_supported(dtype, H, d_n, d_r, d_c, d_v) && aligned(kv, 16) && aligned(k_pe, 16) &&
                 ld_kv % 8 == 0 && ld_pe % 8 == 0)
            e = launch_mla_tc(qt, q_pe, kv, ld_kv, k_pe, ld_pe, idx, k, bt.st, bt.total_k, M, scale, prefix_valid, olat,
                              lse, ws + L.part, s);
        else
            e = launch_mla_simt(qt, DSA_BF16, d_c, q_pe, d_r, dtype, kv, ld_kv, k_pe, ld_pe, idx, k, bt.st, M, H, d_r,
                                d_c, scale, olat, DSA_BF16, lse, s);
        if (e != cudaSuccess) return fail_cuda(e);
        if (mark) stage_mark(4, s);
        if (!wo) {
            e = launch_absorb_v_tc(olat, W_UV, out, M, H, s);
            if (e != cudaSuccess) return fail_cuda(e);
        } else {
            // The step after the path: y = out wo^T, chunk by chunk, so that each chunk of the
            // attention output is read back by the wo GEMM from L2 right after W_UV wrote it.
            const int64_t hv = (int64_t)H * d_v;
            for (int r0 = 0; r0 < M; r0 += kWoChunkRows) {
                const int m = std::min(kWoChunkRows, M - r0);
                void *o = out ? (void *)((__nv_bfloat16 *)out + r0 * hv) : (void *)obuf;
                e = launch_absorb_v_tc(olat + (int64_t)r0 * H * d_c, W_UV, o, m, H, s);
                if (e != cudaSuccess) return fail_cuda(e);
                e = launch_gemm_tc(o, hv, wo, hv, (__nv_bfloat16 *)y + (int64_t)r0 * d_model, d_model, false, m,
                                   d_model, (int)hv, s);
                if (e != cudaSuccess) return fail_cuda(e);
            }
        }
        if (mark) stage_mark(5, s);
        return DSA_OK;
    }
    float *qt = (float *)(ws + L.qt);
    float *olat = (float *)(ws + L.olat);
    // q~[m,h,:] = q_nope[m,h,:] . W_UK[h]    (K = d_n, N = d_c)
    e = launch_absorb_simt(q_nope, dtype, (int64_t)H * d_n, W_UK, dtype, qt, DSA_F32, (int64_t)H * d_c, M, H, d_n,
                           d_c, s);
    if (e != cudaSuccess) return fail_cuda(e);
    if (mark) stage_mark(3, s);
    e = launch_mla_simt(qt, DSA_F32, d_c, q_pe, d_r, dtype, kv, ld_kv, k_pe, ld_pe, idx, k, bt.st, M, H, d_r, d_c,
                        scale, olat, DSA_F32, lse, s);
    if (e != cudaSuccess) return fail_cuda(e);
    if (mark) stage_mark(4, s);
    // out[m,h,:] = o_lat[m,h,:] . W_UV[h]    (K = d_c, N = d_v)
    e = launch_absorb_simt(olat, DSA_F32, (int64_t)H * d_c, W_UV, dtype, out, dtype, (int64_t)H * d_v, M, H, d_c,
                           d_v, s);
    if (e != cudaSuccess) return fail_cuda(e);
    if (mark) stage_mark(5, s);
    return DSA_OK;
}

size_t mla_workspace_bytes(int H, int d_c, int64_t total_q) { return mla_ws_layout(H, d_c, total_q).total; }

int validate_mla_call(const void *q_nope, const void *q_pe, int dtype, const void *kv_cache, int64_t ld_kv,
                      const void *k_pe, int64_t ld_pe, const void *W_UK, const void *W_UV, int H, int d_n, int d_r,
                      int d_c, int d_v, const int32_t *idx, int k, const dsa_seqs *seqs, void *out, Batch &bt) {
    int rc = build_batch(seqs, bt);
    if (rc) return rc;
    if ((rc = check_mla_shape(dtype, H, d_n, d_r, d_c, d_v, k))) return rc;
    if (ld_kv < d_c || ld_pe < d_r) return DSA_ERR_INVALID_ARG;
    if (bt.total_q == 0) return DSA_OK;
    // idx may be null: the dense causal selection (entry e of a row is key e)
    if (!q_nope || (d_r > 0 && (!q_pe || !k_pe)) || !kv_cache || !W_UK || !W_UV || !out) return DSA_ERR_INVALID_ARG;
    return DSA_OK;
}

namespace {

int run_indexer(const void *q, const float *q_scale, const void *k, const float *k_scale, int idx_dtype,
                const float *w, int H_I, int D_I, const SeqTab &st, int rows, int max_S, int64_t total_k,
                float *scores, int64_t ld, bool fill_future, cudaStream_t s, int dense_k = 0) {
    cudaError_t e;
    if (!force_generic() && indexer_tc_supported(idx_dtype, H_I, D_I) && aligned(q, 16) && aligned(k, 16))
        e = launch_indexer_tc(q, q_scale, k, k_scale, idx_dtype, w, st, total_k, scores, ld, fill_future, s,
                              dense_k);
    else
        e = launch_indexer_simt(q, q_scale, k, k_scale, idx_dtype, w, H_I, D_I, st, rows, max_S, scores, ld, s);
    return e == cudaSuccess ? DSA_OK : fail_cuda(e);
}

}  // namespace
}  // namespace dsa

extern "C" {

const char *dsa_status_string(int status) {
    switch (status) {
        case DSA_OK: return "DSA_OK";
        case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
        case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
        case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
        case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
        case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
        default: return "DSA_ERR_UNKNOWN";
    }
}

int dsa_last_cuda_error(void) { return g_last_cuda; }

int dsa_set_stage_events(void *const *events, int n_events) {
    if (!events) {
        g_stage_on = false;
        return DSA_OK;
    }
    if (n_events != DSA_STAGE_EVENTS) return DSA_ERR_INVALID_ARG;
    for (int i = 0; i < DSA_STAGE_EVENTS; ++i) {
        if (!events[i]) return DSA_ERR_INVALID_ARG;
        g_stage_events[i] = (cudaEvent_t)events[i];
    }
    g_stage_on = true;
    return DSA_OK;
}
uint32_t dsa_last_kernels(void) { return g_kernels; }
int dsa_last_launch_count(void) { return g_launches; }

int dsa_check_device_error(void *stream, int *site) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e);
    if (site) *site = 0;
    // Every kernel family keeps its own error word; all of them are read and cleared, and the
    // first one that recorded a timeout gives the site.
    int (*readers[])(int *) = {indexer_tc_read_error, absorb_tc_read_error, mla_tc_read_error, gemm_tc_read_error,
                               selftest_read_error};
    int result = DSA_OK;
    for (auto rd : readers) {
        int s = 0;
        const int rc = rd(&s);
        if (rc == DSA_ERR_CUDA) return rc;
        if (rc != DSA_OK && result == DSA_OK) {
            result = rc;
            if (site) *site = s;
        }
    }
    return result;
}

int dsa_set_wait_limit(int64_t cycles) {
    if (cycles < 0 || cycles > kDefaultWaitLimitCycles) return DSA_ERR_INVALID_ARG;
    g_wait_limit.store(cycles == 0 ? kDefaultWaitLimitCycles : (long long)cycles, std::memory_order_relaxed);
    return DSA_OK;
}

int dsa_selftest_bounded_wait(int64_t limit_cycles, int *completed_ok, void *stream) {
    reset_trace();
    if (limit_cycles < 1 || limit_cycles > (int64_t(1) << 32)) return DSA_ERR_INVALID_ARG;
    cudaError_t e = launch_bounded_wait_selftest((long long)limit_cycles, completed_ok, (cudaStream_t)stream);
    return e == cudaSuccess ? DSA_OK : fail_cuda(e);
}

int dsa_quant_e4m3_ue8m0(const void *x, int x_dtype, int64_t n_blocks, uint8_t *codes, float *scales, void *stream) {
    reset_trace();
    if (n_blocks < 0) return DSA_ERR_INVALID_ARG;
    if (n_blocks > 0 && (!x || !codes || !scales)) return DSA_ERR_INVALID_ARG;
    if (x_dtype != DSA_F32 && x_dtype != DSA_BF16) return DSA_ERR_UNSUPPORTED;
    if (!aligned(codes, 4)) return DSA_ERR_INVALID_ARG;
    cudaError_t e = launch_quant_e4m3(x, x_dtype, n_blocks, codes, scales, (cudaStream_t)stream);
    return e == cudaSuccess ? DSA_OK : fail_cuda(e);
}

int dsa_indexer_scores(const void *q_idx, const float *q_scale, const void *k_idx, const float *k_scale, int idx_dtype,
                       const float *w, int H_I, int D_I, const dsa_seqs *seqs, float *scores, int64_t ld_scores,
                       void *stream) {
    reset_trace();
    Batch bt;
    int rc = build_batch(seqs, bt);
    if (rc) return rc;
    if ((rc = check_indexer_shape(idx_dtype, H_I, D_I))) return rc;
    if (ld_scores < bt.max_S || ld_scores % 4 != 0) return DSA_ERR_INVALID_ARG;
    if (bt.total_q > 0 && (!q_idx || !k_idx || !w || !scores)) return DSA_ERR_INVALID_ARG;
    if (idx_dtype == DSA_E4M3 && bt.total_q > 0 && (!q_scale || !k_scale)) return DSA_ERR_INVALID_ARG;
    if (!aligned(scores, 16)) return DSA_ERR_INVALID_ARG;
    return run_indexer(q_idx, idx_dtype == DSA_E4M3 ? q_scale : nullptr, k_idx,
                       idx_dtype == DSA_E4M3 ? k_scale : nullptr, idx_dtype, w, H_I, D_I, bt.st, bt.total_q, bt.max_S,
                       bt.total_k, scores, ld_scores, true, (cudaStream_t)stream);
}

int dsa_topk_select(const float *scores, int64_t ld_scores, const dsa_seqs *seqs, int k, int32_t *idx, void *stream) {
    reset_trace();
    Batch bt;
    int rc = build_batch(seqs, bt);
    if (rc) return rc;
    if (k < 1 || k > 16384 || ld_scores < bt.max_S) return DSA_ERR_INVALID_ARG;
    if (bt.total_q > 0 && (!scores || !idx)) return DSA_ERR_INVALID_ARG;
    cudaError_t e = launch_topk(scores, ld_scores, bt.st, bt.total_q, k, idx, (cudaStream_t)stream);
    return e == cudaSuccess ? DSA_OK : fail_cuda(e);
}

size_t dsa_sparse_mla_workspace_size(int dtype, int H, int d_n, int d_r, int d_c, int d_v, int k,
                                     const dsa_seqs *seqs) {
    (void)dtype; (void)d_n; (void)d_r; (void)d_v; (void)k;
    Batch bt;
    if (build_batch(seqs, bt) || H < 1 || d_c < 1) return 0;
    return mla_ws_layout(H, d_c, bt.total_q).total;
}

int dsa_sparse_mla_fwd(const void *q_nope, const void *q_pe, int dtype, const void *kv_cache, int64_t ld_kv,
                       const void *k_pe, int64_t ld_pe, const void *W_UK, const void *W_UV, int H, int d_n, int d_r,
                       int d_c, int d_v, const int32_t *idx, int k, const dsa_seqs *seqs, float softmax_scale,
                       void *out, float *lse, void *workspace, size_t ws_bytes, void *stream) {
    reset_trace();
    Batch bt;
    int rc = validate_mla_call(q_nope, q_pe, dtype, kv_cache, ld_kv, k_pe, ld_pe, W_UK, W_UV, H, d_n, d_r, d_c, d_v,
                               idx, k, seqs, out, bt);
    if (rc || bt.total_q == 0) return rc;
    if (!workspace || !aligned(workspace, WS_ALIGN)) return DSA_ERR_WORKSPACE;
    if (ws_bytes < mla_workspace_bytes(H, d_c, bt.total_q)) return DSA_ERR_WORKSPACE;
    return run_mla(q_nope, q_pe, dtype, kv_cache, ld_kv, k_pe, ld_pe, W_UK, W_UV, H, d_n, d_r, d_c, d_v, idx, k, bt,
                   softmax_scale, out, lse, (char *)workspace, (cudaStream_t)stream);
}

int dsa_sparse_mla_fwd_fp8kv(const void *q_nope, const void *q_pe, const uint8_t *kv_codes, int64_t ld_kv,
                             const float *kv_scale, const void *k_pe, int64_t ld_pe, const void *W_UK, const void *W_UV,
                             int H, int d_n, int d_r, int d_c, int d_v, const int32_t *idx, int k,
                             const dsa_seqs *seqs, float softmax_scale, void *out, float *lse, void *workspace,
                             size_t ws_bytes, void *stream) {
    reset_trace();
    Batch bt;
    int rc = validate_mla_call(q_nope, q_pe, DSA_BF16, kv_codes, ld_kv, k_pe, ld_pe, W_UK, W_UV, H, d_n, d_r, d_c, d_v,
                               idx, k, seqs, out, bt);
    if (rc) return rc;
    if (!mla_tc_supported(DSA_BF16, H, d_n, d_r, d_c, d_v)) return DSA_ERR_UNSUPPORTED;
    if (bt.total_q == 0) return DSA_OK;
    if (!kv_scale || ld_kv % 16 != 0 || !aligned(kv_codes, 16) || !aligned(k_pe, 16) || ld_pe % 8 != 0)
        return DSA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, WS_ALIGN)) return DSA_ERR_WORKSPACE;
    if (ws_bytes < mla_workspace_bytes(H, d_c, bt.total_q)) return DSA_ERR_WORKSPACE;
    return run_mla(q_nope, q_pe, DSA_BF16, kv_codes, ld_kv, k_pe, ld_pe, W_UK, W_UV, H, d_n, d_r, d_c, d_v, idx, k, bt,
                   softmax_scale, out, lse, (char *)workspace, (cudaStream_t)stream, false, false, nullptr, 0, nullptr,
                   nullptr, kv_scale);
}

}  // extern "C"

namespace dsa {
namespace {

// Bound on the fp32 score buffer of one chunk of query rows.  Larger chunks give the indexer and
// the top-k more rows per launch (more query groups, so the indexer leaves the split-table mode and
// balances better); on GB300 the long prefills ran faster up to the largest size measured: 32768
// rows of 32768 keys spent 8.5 / 7.6 / 7.5 ms in indexer + top-k with 256 MB / 512 MB / 1 GB
// chunks, and the chunked FP8 prefill 29.8 / 25.5 / 24.9 ms.  1 GB of a GB300's HBM is small.
constexpr size_t SCORE_CHUNK_BYTES = size_t(1024) << 20;

struct FwdWs {
    int64_t ld = 0;
    int rows_per_chunk = 0;
    bool fused = false;  // the indexer selects the top-k itself (one launch, per-SM score slots)
    size_t qcodes = 0, qscale = 0, kcodes = 0, kscale = 0, idx = 0, scores = 0, mla = 0, obuf = 0, total = 0;
};

int check_problem(const dsa_problem *p) {
    if (!p) return DSA_ERR_INVALID_ARG;
    if (p->dtype != DSA_F32 && p->dtype != DSA_BF16) return DSA_ERR_UNSUPPORTED;
    int rc = check_indexer_shape(p->idx_fp8 ? DSA_E4M3 : p->dtype, p->H_I, p->D_I);
    if (rc) return rc;
    rc = check_mla_shape(p->dtype, p->H, p->d_n, p->d_r, p->d_c, p->d_v, p->top_k);
    if (rc) return rc;
    if (p->top_k > 16384) return DSA_ERR_INVALID_ARG;
    if (p->ld_kv < p->d_c || p->ld_pe < p->d_r) return DSA_ERR_INVALID_ARG;
    if (p->kv_fp8) {  // e4m3 latent rows: the tensor-core attention only
        if (p->dtype != DSA_BF16 || !mla_tc_supported(p->dtype, p->H, p->d_n, p->d_r, p->d_c, p->d_v))
            return DSA_ERR_UNSUPPORTED;
        if (p->ld_kv % 16 != 0) return DSA_ERR_INVALID_ARG;
    }
    if (p->wo) {  // the output projection runs on the bf16 tensor-core GEMM only
        if (p->d_model < 1) return DSA_ERR_INVALID_ARG;
        if (p->dtype != DSA_BF16 || !gemm_tc_supported(1, p->d_model, p->H * p->d_v) ||
            !absorb_tc_supported(p->dtype, p->H, p->d_n, p->d_r, p->d_c, p->d_v))
            return DSA_ERR_UNSUPPORTED;
    }
    return DSA_OK;
}

FwdWs fwd_ws_layout(const dsa_problem *p, const Batch &bt) {
    FwdWs w;
    w.ld = ((int64_t)std::max(bt.max_S, 1) + 3) / 4 * 4;
    const int64_t per_row = w.ld * (int64_t)sizeof(float);
    // Batches with enough query groups take the fused indexer + top-k, whose score slots are much
    // smaller than a chunk; if it cannot run after all (misaligned inputs) the unfused path chunks
    // its rows to fit the same region.
    w.fused = !force_generic() && indexer_topk_fused_ok(p->idx_fp8 ? DSA_E4M3 : p->dtype, p->H_I, p->D_I, bt.st,
                                                        p->top_k);
    const int64_t region = w.fused ? (int64_t)indexer_topk_slot_bytes(bt.st, w.ld)
                                   : (int64_t)std::min<size_t>(SCORE_CHUNK_BYTES, (size_t)bt.total_q * per_row);
    w.rows_per_chunk = (int)std::max<int64_t>(1, std::min<int64_t>(bt.total_q, region / per_row));
    size_t off = 0;
    if (p->idx_fp8) {
        w.qcodes = off; off += align_up((size_t)bt.total_q * p->H_I * p->D_I);
        w.qscale = off; off += align_up((size_t)bt.total_q * p->H_I * sizeof(float));
        w.kcodes = off; off += align_up((size_t)bt.total_k * p->D_I);
        w.kscale = off; off += align_up((size_t)bt.total_k * sizeof(float));
    }
    if (!p->idx_out) {
        w.idx = off; off += align_up((size_t)bt.total_q * p->top_k * sizeof(int32_t));
    }
    w.scores = off; off += align_up(std::max<size_t>((size_t)w.rows_per_chunk * per_row, w.fused ? region : 0));
    w.mla = off; off += mla_ws_layout(p->H, p->d_c, bt.total_q).total;
    if (p->wo && !p->out) {  // one chunk of the attention output between W_UV and wo
        w.obuf = off; off += align_up((size_t)std::min(bt.total_q, kWoChunkRows) * p->H * p->d_v * 2);
    }
    w.total = off;
    return w;
}

// The cache rows a host-buffer call appends, staged in one piece in the workspace, go to their rows:
// appended row r (counted over the batch) of sequence b lands at dst0[b] + r - app_off[b].
struct AppendParams {
    int B;
    int app_off[DSA_MAX_SEQS + 1];
    int64_t dst0[DSA_MAX_SEQS];
};
static_assert(sizeof(AppendParams) + 256 <= 32764, "launch parameters");

// One warp per row, 16-byte chunks (row_bytes a multiple of 16, both sides 16-byte aligned).
__global__ void __launch_bounds__(256) append_rows_kernel(const __grid_constant__ AppendParams P,
                                                          const uint4 *__restrict__ src, char *__restrict__ dst,
                                                          int64_t row_bytes, int64_t rows) {
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= rows) return;
    int lo = 0, hi = P.B - 1;  // the sequence that owns row r: the last b with app_off[b] <= r
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.app_off[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const int64_t chunks = row_bytes / 16;
    const uint4 *in = src + r * chunks;
    uint4 *out = (uint4 *)(dst + (P.dst0[lo] + (r - P.app_off[lo])) * row_bytes);
    for (int64_t c = threadIdx.x & 31; c < chunks; c += 32) out[c] = in[c];
}

cudaError_t launch_append_rows(const AppendParams &P, const void *src, void *dst, int64_t row_bytes, int64_t rows,
                               cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    append_rows_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(P, (const uint4 *)src, (char *)dst, row_bytes, rows);
    note_launch(DSA_KERNEL_APPEND);
    return cudaGetLastError();
}

int forward_impl(const dsa_problem *p, const dsa_seqs *seqs, void *workspace, size_t ws_bytes, void *stream);
int check_forward(const dsa_problem *p, const Batch &bt, const void *workspace, size_t ws_bytes);

}  // namespace
}  // namespace dsa

extern "C" {

size_t dsa_forward_workspace_size(const dsa_problem *p, const dsa_seqs *seqs) {
    Batch bt;
    if (check_problem(p) || build_batch(seqs, bt)) return 0;
    return fwd_ws_layout(p, bt).total;
}

int dsa_forward(const dsa_problem *p, const dsa_seqs *seqs, void *workspace, size_t ws_bytes, void *stream) {
    reset_trace();
    return dsa::forward_impl(p, seqs, workspace, ws_bytes, stream);
}

}  // extern "C"

namespace dsa {
namespace {

// The checks of a forward call on a non-empty batch that need no GPU (the problem itself is checked by
// check_problem first).
int check_forward(const dsa_problem *p, const Batch &bt, const void *workspace, size_t ws_bytes) {
    if (!p->q_idx || !p->k_idx || !p->w || !p->q_nope || !p->kv_cache || !p->W_UK || !p->W_UV ||
        (!p->out && !p->wo) || (p->d_r > 0 && (!p->q_pe || !p->k_pe)))
        return DSA_ERR_INVALID_ARG;
    if (p->wo && (!p->y || !aligned(p->wo, 16) || !aligned(p->y, 16))) return DSA_ERR_INVALID_ARG;
    if (p->kv_fp8 && (!p->kv_scale || !aligned(p->kv_cache, 16))) return DSA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, WS_ALIGN) || ws_bytes < fwd_ws_layout(p, bt).total) return DSA_ERR_WORKSPACE;
    return DSA_OK;
}

int forward_impl(const dsa_problem *p, const dsa_seqs *seqs, void *workspace, size_t ws_bytes, void *stream) {
    int rc = check_problem(p);
    if (rc) return rc;
    Batch bt;
    if ((rc = build_batch(seqs, bt))) return rc;
    if (bt.total_q == 0) return DSA_OK;
    if ((rc = check_forward(p, bt, workspace, ws_bytes))) return rc;
    const FwdWs L = fwd_ws_layout(p, bt);
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = (char *)workspace;
    cudaError_t e;
    stage_mark(0, s);

    // A row whose causal prefix holds at most top_k keys selects all of them, in ascending order.
    // When every row of the batch does (the last row of each sequence is enough to check), the
    // selection is known without scores: the quantiser, indexer and top-k do not run, the attention
    // reads the dense causal pattern directly, and the index output is filled only if asked for.
    bool all_dense = true;
    for (int b = 0; b < bt.st.B && all_dense; ++b) {
        const int Tb = bt.st.q_off[b + 1] - bt.st.q_off[b];
        if (Tb > 0 && std::min(bt.st.start_pos[b] + Tb, bt.st.k_len[b]) > p->top_k) all_dense = false;
    }
    if (all_dense) {
        stage_mark(1, s);
        if (p->idx_out) {
            e = launch_dense_idx(bt.st, bt.total_q, p->top_k, p->idx_out, s);
            if (e != cudaSuccess) return fail_cuda(e);
        }
        stage_mark(2, s);
        return run_mla(p->q_nope, p->q_pe, p->dtype, p->kv_cache, p->ld_kv, p->k_pe, p->ld_pe, p->W_UK, p->W_UV,
                       p->H, p->d_n, p->d_r, p->d_c, p->d_v, nullptr, p->top_k, bt, p->softmax_scale, p->out, p->lse,
                       ws + L.mla, s, true, true, p->wo, p->d_model, p->y, ws + L.obuf,
                       p->kv_fp8 ? p->kv_scale : nullptr);
    }

    const void *q_idx = p->q_idx, *k_idx = p->k_idx;
    const float *q_scale = nullptr, *k_scale = nullptr;
    int idx_dtype = p->dtype;
    if (p->idx_fp8) {
        uint8_t *qc = (uint8_t *)(ws + L.qcodes), *kc = (uint8_t *)(ws + L.kcodes);
        float *qs = (float *)(ws + L.qscale), *ks = (float *)(ws + L.kscale);
        e = launch_quant_e4m3(p->q_idx, p->dtype, (int64_t)bt.total_q * p->H_I, qc, qs, s);
        if (e != cudaSuccess) return fail_cuda(e);
        e = launch_quant_e4m3(p->k_idx, p->dtype, bt.total_k, kc, ks, s);
        if (e != cudaSuccess) return fail_cuda(e);
        q_idx = qc; k_idx = kc; q_scale = qs; k_scale = ks;
        idx_dtype = DSA_E4M3;
    }
    stage_mark(1, s);
    int32_t *idx = p->idx_out ? p->idx_out : (int32_t *)(ws + L.idx);
    float *scores = (float *)(ws + L.scores);
    const size_t qrow = dtype_bytes(idx_dtype) * p->H_I * p->D_I;
    if (L.fused && aligned(q_idx, 16) && aligned(k_idx, 16)) {
        // one launch over the whole batch: scores into per-SM slots, the top-k selected from them
        e = launch_indexer_topk_tc(q_idx, q_scale, k_idx, k_scale, idx_dtype, p->w, bt.st, bt.total_k, scores, L.ld,
                                   p->top_k, idx, s);
        if (e != cudaSuccess) return fail_cuda(e);
        stage_mark(2, s);
        return run_mla(p->q_nope, p->q_pe, p->dtype, p->kv_cache, p->ld_kv, p->k_pe, p->ld_pe, p->W_UK, p->W_UV, p->H,
                       p->d_n, p->d_r, p->d_c, p->d_v, idx, p->top_k, bt, p->softmax_scale, p->out, p->lse,
                       ws + L.mla, s, true, true, p->wo, p->d_model, p->y, ws + L.obuf,
                       p->kv_fp8 ? p->kv_scale : nullptr);
    }
    for (int r0 = 0; r0 < bt.total_q; r0 += L.rows_per_chunk) {
        const int r1 = std::min(bt.total_q, r0 + L.rows_per_chunk);
        SeqTab st;
        int max_S = 0;
        sub_batch(seqs, r0, r1, st, max_S);
        rc = run_indexer((const char *)q_idx + qrow * r0, q_scale ? q_scale + (size_t)r0 * p->H_I : nullptr, k_idx,
                         k_scale, idx_dtype, p->w + (size_t)r0 * p->H_I, p->H_I, p->D_I, st, r1 - r0, max_S,
                         bt.total_k, scores, L.ld, false, s, p->top_k);
        if (rc) return rc;
        e = launch_topk(scores, L.ld, st, r1 - r0, p->top_k, idx + (size_t)r0 * p->top_k, s);
        if (e != cudaSuccess) return fail_cuda(e);
    }
    stage_mark(2, s);
    return run_mla(p->q_nope, p->q_pe, p->dtype, p->kv_cache, p->ld_kv, p->k_pe, p->ld_pe, p->W_UK, p->W_UV, p->H,
                   p->d_n, p->d_r, p->d_c, p->d_v, idx, p->top_k, bt, p->softmax_scale, p->out, p->lse, ws + L.mla, s,
                   true, true, p->wo, p->d_model, p->y, ws + L.obuf, p->kv_fp8 ? p->kv_scale : nullptr);
}

// dsa_forward_host's side stream, one per host thread and device: the copies of q_nope and q_pe,
// which only the attention stage reads, run on it while the indexer and top-k run on the caller's
// stream.  Created on first use and kept for the thread's life; null when it cannot be created
// (the copies then stay on the caller's stream).
struct QueryCopyStream {
    cudaStream_t st = nullptr;
    cudaEvent_t main_in = nullptr, query_in = nullptr;  // the caller stream's inputs are in; q_nope, q_pe are
};

QueryCopyStream *query_copy_stream() {
    thread_local std::map<int, QueryCopyStream> tab;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    QueryCopyStream &q = tab[dev];
    if (!q.st) {
        cudaStream_t st = nullptr;
        cudaEvent_t ev[2] = {nullptr, nullptr};
        bool ok = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) == cudaSuccess;
        for (int i = 0; ok && i < 2; ++i) ok = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            for (cudaEvent_t x : ev)
                if (x) cudaEventDestroy(x);
            if (st) cudaStreamDestroy(st);
            cudaGetLastError();
            return nullptr;
        }
        q.st = st;
        q.main_in = ev[0];
        q.query_in = ev[1];
    }
    return &q;
}

// Sets the attention stage's wait for the side stream's query copies for one forward, and clears it
// on every way out.
struct QueryInScope {
    explicit QueryInScope(cudaEvent_t ev) { g_query_in = ev; }
    ~QueryInScope() { g_query_in = nullptr; }
};

}  // namespace
}  // namespace dsa

extern "C" {

int dsa_forward_host(const dsa_problem *p, const dsa_seqs *seqs, const dsa_host_io *io, void *workspace,
                     size_t ws_bytes, void *stream) {
    reset_trace();
    if (!io) return DSA_ERR_INVALID_ARG;
    int rc = check_problem(p);
    if (rc) return rc;
    Batch bt;
    if ((rc = build_batch(seqs, bt))) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t esz = p->dtype == DSA_F32 ? 4 : 2;
    const size_t T = (size_t)bt.total_q;
    const bool appends = io->kv_new || io->k_pe_new || io->k_idx_new || io->kv_scale_new;
    if (appends)
        for (int b = 0; b < bt.st.B; ++b)
            if (bt.st.start_pos[b] > bt.st.k_len[b]) return DSA_ERR_INVALID_ARG;
    if ((io->kv_new && !p->kv_cache) || (io->k_pe_new && !p->k_pe) || (io->k_idx_new && !p->k_idx) ||
        (io->kv_scale_new && (!p->kv_fp8 || !p->kv_scale)) || (io->lse && !p->lse) || (io->idx && !p->idx_out) ||
        (io->out && !(p->wo ? p->y : p->out)))
        return DSA_ERR_INVALID_ARG;
    // everything the forward would refuse is refused before any copy is enqueued
    if (bt.total_q > 0 && (rc = check_forward(p, bt, workspace, ws_bytes))) return rc;
    cudaError_t e = cudaSuccess;
    if (io->copy_after) e = cudaStreamWaitEvent(s, (cudaEvent_t)io->copy_after, 0);
    auto put_on = [&](const void *dev, const void *host, size_t bytes, cudaStream_t on) {
        if (e == cudaSuccess && host && bytes) e = cudaMemcpyAsync((void *)dev, host, bytes, cudaMemcpyHostToDevice, on);
    };
    auto put = [&](const void *dev, const void *host, size_t bytes) { put_on(dev, host, bytes, s); };
    put(p->q_idx, io->q_idx, T * p->H_I * p->D_I * esz);
    put(p->w, io->w, T * p->H_I * sizeof(float));
    // Appended cache rows.  Staged: each array in one copy into the workspace (free until the forward
    // starts), then a kernel puts the rows in place -- a decode batch appends one row per sequence, and
    // a copy per row would cost more than the rows.  Otherwise one copy per sequence and array.
    const size_t kv_row = (size_t)p->ld_kv * (p->kv_fp8 ? 1 : esz), pe_row = (size_t)p->ld_pe * esz,
                 ki_row = (size_t)p->D_I * esz, sc_row = (size_t)(p->d_c / 128) * sizeof(float);
    struct Arr {
        const void *host;
        void *dev;
        size_t row;
    } arrs[4] = {{io->kv_new, (void *)p->kv_cache, kv_row},
                 {io->k_pe_new, (void *)p->k_pe, pe_row},
                 {io->k_idx_new, (void *)p->k_idx, ki_row},
                 {io->kv_scale_new, (void *)p->kv_scale, sc_row}};
    size_t app_rows = 0, stage_bytes = 0;
    bool staged = appends && workspace && aligned(workspace, 256);
    for (int b = 0; b < bt.st.B && appends; ++b) app_rows += (size_t)(bt.st.k_len[b] - bt.st.start_pos[b]);
    for (const Arr &a : arrs)
        if (a.host) {
            staged = staged && a.row % 16 == 0 && aligned(a.dev, 16);
            stage_bytes += (a.row * app_rows + 255) / 256 * 256;
        }
    staged = staged && stage_bytes <= ws_bytes;
    if (staged && app_rows > 0) {
        static thread_local AppendParams AP;  // ~12 KB: keep it off the host stack
        AP.B = bt.st.B;
        AP.app_off[0] = 0;
        for (int b = 0; b < bt.st.B; ++b) {
            AP.app_off[b + 1] = AP.app_off[b] + (bt.st.k_len[b] - bt.st.start_pos[b]);
            AP.dst0[b] = (int64_t)bt.st.k_base[b] + bt.st.start_pos[b];
        }
        char *stage = (char *)workspace;
        for (const Arr &a : arrs)
            if (a.host) {
                put(stage, a.host, a.row * app_rows);
                if (e == cudaSuccess) e = launch_append_rows(AP, stage, a.dev, (int64_t)a.row, (int64_t)app_rows, s);
                stage += (a.row * app_rows + 255) / 256 * 256;
            }
    }
    size_t done = 0;  // appended rows before sequence b
    for (int b = 0; b < bt.st.B && appends && !staged; ++b) {
        const size_t r0 = (size_t)bt.st.k_base[b] + bt.st.start_pos[b];
        const size_t n = (size_t)(bt.st.k_len[b] - bt.st.start_pos[b]);
        if (io->kv_new) put((const char *)p->kv_cache + r0 * kv_row, (const char *)io->kv_new + done * kv_row, n * kv_row);
        if (io->k_pe_new)
            put((const char *)p->k_pe + r0 * pe_row, (const char *)io->k_pe_new + done * pe_row, n * pe_row);
        if (io->k_idx_new)
            put((const char *)p->k_idx + r0 * ki_row, (const char *)io->k_idx_new + done * ki_row, n * ki_row);
        if (io->kv_scale_new)
            put((const char *)p->kv_scale + r0 * sc_row, (const char *)io->kv_scale_new + done * sc_row, n * sc_row);
        done += n;
    }
    // q_nope and q_pe, which only the attention stage reads, go in last and on the side stream: their
    // transfer overlaps the quantiser, indexer and top-k, which start once the inputs above are in;
    // the attention stage waits for query_in.
    QueryCopyStream *qs = (io->q_nope || io->q_pe) && T > 0 && e == cudaSuccess ? query_copy_stream() : nullptr;
    if (qs) {
        e = cudaEventRecord(qs->main_in, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(qs->st, qs->main_in, 0);
    }
    put_on(p->q_nope, io->q_nope, T * p->H * p->d_n * esz, qs ? qs->st : s);
    put_on(p->q_pe, io->q_pe, T * p->H * p->d_r * esz, qs ? qs->st : s);
    if (qs && e == cudaSuccess) e = cudaEventRecord(qs->query_in, qs->st);
    if (e == cudaSuccess && io->copy_done) e = cudaEventRecord((cudaEvent_t)io->copy_done, qs ? qs->st : s);
    if (e == cudaSuccess && io->compute_after) e = cudaStreamWaitEvent(s, (cudaEvent_t)io->compute_after, 0);
    if (e != cudaSuccess) return fail_cuda(e);
    {
        QueryInScope scope(qs ? qs->query_in : nullptr);
        if ((rc = forward_impl(p, seqs, workspace, ws_bytes, stream))) return rc;
    }
    // Nothing on `s` after this point reads q_nope or q_pe; a later call's copies into them wait for
    // this call's forward through main_in, recorded on its stream after this forward.
    if (io->compute_done && (e = cudaEventRecord((cudaEvent_t)io->compute_done, s)) != cudaSuccess) return fail_cuda(e);
    auto get = [&](void *host, const void *dev, size_t bytes) {
        if (e == cudaSuccess && host && bytes) e = cudaMemcpyAsync(host, dev, bytes, cudaMemcpyDeviceToHost, s);
    };
    if (p->wo)
        get(io->out, p->y, T * p->d_model * esz);
    else
        get(io->out, p->out, T * p->H * p->d_v * esz);
    get(io->lse, p->lse, T * p->H * sizeof(float));
    get(io->idx, p->idx_out, T * p->top_k * sizeof(int32_t));
    return e == cudaSuccess ? DSA_OK : fail_cuda(e);
}

}  // extern "C"
