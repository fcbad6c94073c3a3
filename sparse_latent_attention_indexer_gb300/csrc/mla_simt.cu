// Generic (CUDA-core) kernels of the latent attention, for shapes and dtypes
// the tensor-core kernels do not specialise (the tiny fp32 workload).
//
//  * absorb GEMM: C[m,h,:] = A[m,h,:] . B[h]   (B row-major K x N), used for
//    q~ = q_nope W_UK (K = d_n, N = d_c) and out = o_lat W_UV (K = d_c, N = d_v).
//  * sparse attention in the latent space: per query row and head,
//      z_j = scale (q~ . c[s_j] + q_pe . k_pe[s_j])  over the selected keys,
//      online softmax, o_lat = sum_j P_j c[s_j], lse = log sum_j exp(z_j).
// (DeepSeek-V3.2-Exp atlas page, MoE transformer block: k^C = c^KV W_UK,
// v = c^KV W_UV, K_i = [K^C_i; k^R], M^sel; regrouped into the absorbed form.)
#include "dsa_common.cuh"

namespace dsa {
namespace {

// ---------------------------------------------------------------------------
// Batched per-head SIMT GEMM: 64 x 64 tiles, K steps of 16, 4 x 4 per thread.
// ---------------------------------------------------------------------------
template <typename TA, typename TB, typename TC>
__global__ void __launch_bounds__(256) absorb_simt_kernel(const TA *__restrict__ A, int64_t lda_row,
                                                          const TB *__restrict__ Bm, TC *__restrict__ C,
                                                          int64_t ldc_row, int M, int H, int K, int N) {
    __shared__ float As[16][64 + 4];
    __shared__ float Bs[16][64 + 4];
    const int h = blockIdx.z;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += 16) {
        for (int i = threadIdx.x; i < 64 * 16; i += 256) {
            const int mm = i / 16, kk = i % 16;
            const int m = m0 + mm, kq = k0 + kk;
            As[kk][mm] = (m < M && kq < K) ? to_f32(A[(int64_t)m * lda_row + (int64_t)h * K + kq]) : 0.0f;
            const int kb = i / 64, nn = i % 64;
            const int n = n0 + nn, kr = k0 + kb;
            Bs[kb][nn] = (n < N && kr < K) ? to_f32(Bm[((int64_t)h * K + kr) * N + n]) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n < N) C[(int64_t)m * ldc_row + (int64_t)h * N + n] = from_f32<TC>(acc[i][j]);
        }
    }
}

template <typename TA, typename TB>
cudaError_t absorb_dispatch_c(const TA *A, int64_t lda, const TB *Bm, void *C, int c_dtype, int64_t ldc, int M, int H,
                              int K, int N, cudaStream_t s) {
    dim3 grid((N + 63) / 64, (M + 63) / 64, H);
    if (c_dtype == DSA_BF16)
        absorb_simt_kernel<TA, TB, __nv_bfloat16><<<grid, 256, 0, s>>>(A, lda, Bm, (__nv_bfloat16 *)C, ldc, M, H, K, N);
    else
        absorb_simt_kernel<TA, TB, float><<<grid, 256, 0, s>>>(A, lda, Bm, (float *)C, ldc, M, H, K, N);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Sparse latent attention, SIMT: one CTA = one query row x HG heads, one warp
// per head.  Selected keys are gathered 32 at a time into shared memory (fp32,
// padded rows); lane j scores key j, the warp runs the online softmax and
// each lane accumulates d_c / 32 latent columns in registers.
// ---------------------------------------------------------------------------
constexpr int HG = 8;             // heads per CTA (one warp each)
constexpr int KC = 32;            // keys per chunk
constexpr int MAX_PER_LANE = 32;  // d_c <= 1024

template <typename TQ, typename T, typename TO>
__global__ void __launch_bounds__(HG * 32) mla_simt_kernel(const TQ *__restrict__ qt, int qt_ld,
                                                           const T *__restrict__ q_pe, int qpe_ld,
                                                           const T *__restrict__ kv, int64_t ld_kv,
                                                           const T *__restrict__ kpe, int64_t ld_pe,
                                                           const int32_t *__restrict__ idx, int k,
                                                           const __grid_constant__ SeqTab st, int H, int d_r, int d_c,
                                                           float scale, TO *__restrict__ olat,
                                                           float *__restrict__ lse) {
    extern __shared__ float smem[];
    __shared__ int keys[KC];
    const int r = blockIdx.x;
    const int h0 = blockIdx.y * HG;
    const RowInfo ri = row_info(st, r);
    const int W = d_c + d_r, WP = W + 1;
    float *qs = smem;               // [HG][W]
    float *cs = qs + HG * W;        // [KC][WP]
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int h = h0 + wid;
    for (int i = threadIdx.x; i < HG * W; i += blockDim.x) {
        const int hh = i / W, c = i - hh * W;
        float v = 0.0f;
        if (h0 + hh < H)
            v = c < d_c ? to_f32(qt[((int64_t)r * H + h0 + hh) * qt_ld + c])
                        : to_f32(q_pe[((int64_t)r * H + h0 + hh) * qpe_ld + (c - d_c)]);
        qs[i] = v;
    }
    float o[MAX_PER_LANE];
#pragma unroll
    for (int i = 0; i < MAX_PER_LANE; ++i) o[i] = 0.0f;
    float m = -INFINITY, l = 0.0f;
    const int32_t *row_idx = idx ? idx + (int64_t)r * k : nullptr;  // none: entry j is key j (dense causal)
    for (int j0 = 0; j0 < k; j0 += KC) {
        __syncthreads();
        if (threadIdx.x < KC) {
            const int j = j0 + threadIdx.x;
            int s = j < k ? (row_idx ? row_idx[j] : j) : -1;
            if (s < 0 || s >= ri.S || s > ri.p) s = -1;
            keys[threadIdx.x] = s;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < KC * W; i += blockDim.x) {
            const int jj = i / W, c = i - jj * W;
            const int s = keys[jj];
            float v = 0.0f;
            if (s >= 0) {
                const int64_t row = ri.kbase + s;
                v = c < d_c ? to_f32(kv[row * ld_kv + c]) : to_f32(kpe[row * ld_pe + (c - d_c)]);
            }
            cs[jj * WP + c] = v;
        }
        __syncthreads();
        if (h >= H) continue;
        float z = -INFINITY;
        if (keys[lane] >= 0) {
            float dot = 0.0f;
            const float *q = qs + wid * W, *c = cs + lane * WP;
            for (int d = 0; d < W; ++d) dot = fmaf(q[d], c[d], dot);
            z = dot * scale;
        }
        float zmax = z;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, off));
        const float m_new = fmaxf(m, zmax);
        if (m_new == -INFINITY) continue;  // nothing live yet
        const float corr = expf(m - m_new);
        const float p = (z == -INFINITY) ? 0.0f : expf(z - m_new);
        float psum = p;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l = l * corr + psum;
        m = m_new;
#pragma unroll
        for (int i = 0; i < MAX_PER_LANE; ++i) o[i] *= corr;
        for (int jj = 0; jj < KC; ++jj) {
            const float pj = __shfl_sync(0xffffffffu, p, jj);
            if (pj == 0.0f) continue;
            const float *c = cs + jj * WP;
#pragma unroll
            for (int i = 0; i < MAX_PER_LANE; ++i) {
                const int d = lane + 32 * i;
                if (d < d_c) o[i] = fmaf(pj, c[d], o[i]);
            }
        }
    }
    if (h >= H) return;
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
    for (int i = 0; i < MAX_PER_LANE; ++i) {
        const int d = lane + 32 * i;
        if (d < d_c) olat[((int64_t)r * H + h) * d_c + d] = from_f32<TO>(o[i] * inv);
    }
    if (lse && lane == 0) lse[(int64_t)r * H + h] = l > 0.0f ? m + logf(l) : -INFINITY;
}

template <typename TQ, typename T, typename TO>
cudaError_t mla_simt_typed(const void *qt, int qt_ld, const void *q_pe, int qpe_ld, const void *kv, int64_t ld_kv,
                           const void *k_pe, int64_t ld_pe, const int32_t *idx, int k, const SeqTab &st, dim3 grid,
                           size_t smem, int H, int d_r, int d_c, float scale, void *olat, float *lse, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(mla_simt_kernel<TQ, T, TO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    mla_simt_kernel<TQ, T, TO><<<grid, HG * 32, smem, s>>>((const TQ *)qt, qt_ld, (const T *)q_pe, qpe_ld,
                                                           (const T *)kv, ld_kv, (const T *)k_pe, ld_pe, idx, k, st,
                                                           H, d_r, d_c, scale, (TO *)olat, lse);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_absorb_simt(const void *A, int a_dtype, int64_t lda_row, const void *Bm, int b_dtype, void *C,
                               int c_dtype, int64_t ldc_row, int M, int H, int K, int N, cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    cudaError_t e;
    if (a_dtype == DSA_BF16 && b_dtype == DSA_BF16)
        e = absorb_dispatch_c((const __nv_bfloat16 *)A, lda_row, (const __nv_bfloat16 *)Bm, C, c_dtype, ldc_row, M, H,
                              K, N, s);
    else if (a_dtype == DSA_F32 && b_dtype == DSA_BF16)
        e = absorb_dispatch_c((const float *)A, lda_row, (const __nv_bfloat16 *)Bm, C, c_dtype, ldc_row, M, H, K, N,
                              s);
    else if (a_dtype == DSA_F32 && b_dtype == DSA_F32)
        e = absorb_dispatch_c((const float *)A, lda_row, (const float *)Bm, C, c_dtype, ldc_row, M, H, K, N, s);
    else
        e = absorb_dispatch_c((const __nv_bfloat16 *)A, lda_row, (const float *)Bm, C, c_dtype, ldc_row, M, H, K, N,
                              s);
    note_launch(DSA_KERNEL_ABSORB_SIMT);
    return e;
}

cudaError_t launch_mla_simt(const void *qt, int qt_dtype, int qt_ld, const void *q_pe, int qpe_ld, int dtype,
                            const void *kv, int64_t ld_kv, const void *k_pe, int64_t ld_pe, const int32_t *idx, int k,
                            const SeqTab &st, int total_q, int H, int d_r, int d_c, float scale, void *olat,
                            int olat_dtype, float *lse, cudaStream_t s) {
    if (total_q == 0) return cudaSuccess;
    dim3 grid(total_q, (H + HG - 1) / HG);
    const int W = d_c + d_r;
    const size_t smem = ((size_t)HG * W + (size_t)KC * (W + 1)) * sizeof(float);
    cudaError_t e;
    if (qt_dtype == DSA_F32 && dtype == DSA_F32)
        e = mla_simt_typed<float, float, float>(qt, qt_ld, q_pe, qpe_ld, kv, ld_kv, k_pe, ld_pe, idx, k, st, grid,
                                                smem, H, d_r, d_c, scale, olat, lse, s);
    else if (qt_dtype == DSA_F32)
        e = mla_simt_typed<float, __nv_bfloat16, float>(qt, qt_ld, q_pe, qpe_ld, kv, ld_kv, k_pe, ld_pe, idx, k, st,
                                                        grid, smem, H, d_r, d_c, scale, olat, lse, s);
    else if (olat_dtype == DSA_BF16)
        e = mla_simt_typed<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16>(qt, qt_ld, q_pe, qpe_ld, kv, ld_kv, k_pe,
                                                                        ld_pe, idx, k, st, grid, smem, H, d_r, d_c,
                                                                        scale, olat, lse, s);
    else
        e = mla_simt_typed<__nv_bfloat16, __nv_bfloat16, float>(qt, qt_ld, q_pe, qpe_ld, kv, ld_kv, k_pe, ld_pe, idx,
                                                                k, st, grid, smem, H, d_r, d_c, scale, olat, lse, s);
    note_launch(DSA_KERNEL_MLA_SIMT);
    return e;
}

}  // namespace dsa
