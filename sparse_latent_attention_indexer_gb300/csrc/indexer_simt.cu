// Generic (CUDA-core) lightning indexer: any H_I <= 128, D_I <= 256, fp32,
// bf16 or e4m3 inputs.  Used for shapes the tensor-core kernel does not
// specialise (the tiny fp32 workload) and as a cross-check of it.
//
//   S~^I_{t,s} = 1/(sqrt(H_I) sqrt(D_I)) sum_h w_{t,h} ReLU(q^I_{h,t} . k^I_s) + M_{t,s}
// (DeepSeek-V3.2-Exp atlas page, MoE transformer block, indexer equations.)
//
// One CTA takes one query row and a chunk of 256 keys in tiles of 64.  The
// row's q^I (and w, with the constant and the q block scales folded in) sit
// in shared memory as fp32; 256 threads = 64 keys x 4 head groups, each
// thread accumulating its heads' dot products in fp32, then the four groups
// are summed through shared memory.
#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int KT = 64;        // keys per tile
constexpr int CHUNK = 256;    // keys per CTA
constexpr int NG = 4;         // head groups

template <typename T> __device__ __forceinline__ float ld_val(const T *p, int64_t i) { return to_f32(p[i]); }
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
    // Bit-level decode of an e4m3 code (1-4-3, bias 7, no infinities).
    const int E = (c >> 3) & 15, m = c & 7;
    float mag = (E == 0) ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), E - 10);
    if (E == 15 && m == 7) mag = __int_as_float(0x7fc00000);
    return (c & 0x80) ? -mag : mag;
}
template <> __device__ __forceinline__ float ld_val<uint8_t>(const uint8_t *p, int64_t i) { return e4m3_to_f32(p[i]); }

template <typename T>
__global__ void __launch_bounds__(256) indexer_simt_kernel(const T *__restrict__ q, const float *__restrict__ q_scale,
                                                           const T *__restrict__ k, const float *__restrict__ k_scale,
                                                           const float *__restrict__ w, int H_I, int D_I,
                                                           const __grid_constant__ SeqTab st,
                                                           float *__restrict__ scores, int64_t ld) {
    extern __shared__ float smem[];
    const int r = blockIdx.x;
    const RowInfo ri = row_info(st, r);
    const int chunk0 = blockIdx.y * CHUNK;
    if (chunk0 >= ri.S) return;
    float *out = scores + (int64_t)r * ld;
    const int chunk_end = min(chunk0 + CHUNK, ri.S);
    // Keys past the query position are masked: -inf, no arithmetic.
    if (chunk0 > ri.p) {
        for (int s = chunk0 + threadIdx.x; s < chunk_end; s += blockDim.x) out[s] = -INFINITY;
        return;
    }
    const int DP = D_I + 1;
    float *qs = smem;                    // [H_I][DP]
    float *ks = qs + H_I * DP;           // [KT][DP]
    float *ws = ks + KT * DP;            // [H_I]
    float *part = ws + H_I;              // [NG][KT]
    const float c = rsqrtf((float)H_I) * rsqrtf((float)D_I);
    for (int i = threadIdx.x; i < H_I * D_I; i += blockDim.x) {
        const int h = i / D_I, d = i - h * D_I;
        qs[h * DP + d] = ld_val(q, (int64_t)r * H_I * D_I + i);
    }
    for (int h = threadIdx.x; h < H_I; h += blockDim.x)
        ws[h] = w[(int64_t)r * H_I + h] * c * (q_scale ? q_scale[(int64_t)r * H_I + h] : 1.0f);
    const int j = threadIdx.x % KT, g = threadIdx.x / KT;
    for (int s0 = chunk0; s0 < chunk_end; s0 += KT) {
        __syncthreads();
        for (int i = threadIdx.x; i < KT * D_I; i += blockDim.x) {
            const int jj = i / D_I, d = i - jj * D_I;
            const int s = s0 + jj;
            ks[jj * DP + d] = (s < chunk_end) ? ld_val(k, (int64_t)(ri.kbase + s) * D_I + d) : 0.0f;
        }
        __syncthreads();
        float acc = 0.0f;
        for (int h = g; h < H_I; h += NG) {
            float dot = 0.0f;
            const float *qh = qs + h * DP, *kj = ks + j * DP;
            for (int d = 0; d < D_I; ++d) dot = fmaf(qh[d], kj[d], dot);
            acc = fmaf(ws[h], fmaxf(dot, 0.0f), acc);
        }
        part[g * KT + j] = acc;
        __syncthreads();
        if (g == 0) {
            const int s = s0 + j;
            if (s < chunk_end) {
                float v = part[j] + part[KT + j] + part[2 * KT + j] + part[3 * KT + j];
                if (k_scale) v *= k_scale[ri.kbase + s];
                out[s] = (s <= ri.p) ? v : -INFINITY;
            }
        }
    }
}

template <typename T>
cudaError_t launch_typed(const T *q, const float *q_scale, const T *k, const float *k_scale, const float *w, int H_I,
                         int D_I, const SeqTab &st, dim3 grid, size_t smem, float *scores, int64_t ld,
                         cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(indexer_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    indexer_simt_kernel<T><<<grid, 256, smem, s>>>(q, q_scale, k, k_scale, w, H_I, D_I, st, scores, ld);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_simt(const void *q, const float *q_scale, const void *k, const float *k_scale, int dtype,
                                const float *w, int H_I, int D_I, const SeqTab &st, int total_q, int max_S,
                                float *scores, int64_t ld, cudaStream_t s) {
    if (total_q == 0 || max_S == 0) return cudaSuccess;
    dim3 grid(total_q, (max_S + CHUNK - 1) / CHUNK);
    const size_t smem = ((size_t)(H_I + KT) * (D_I + 1) + H_I + NG * KT) * sizeof(float);
    cudaError_t e;
    if (dtype == DSA_F32)
        e = launch_typed((const float *)q, q_scale, (const float *)k, k_scale, w, H_I, D_I, st, grid, smem, scores,
                         ld, s);
    else if (dtype == DSA_BF16)
        e = launch_typed((const __nv_bfloat16 *)q, q_scale, (const __nv_bfloat16 *)k, k_scale, w, H_I, D_I, st, grid,
                         smem, scores, ld, s);
    else
        e = launch_typed((const uint8_t *)q, q_scale, (const uint8_t *)k, k_scale, w, H_I, D_I, st, grid, smem,
                         scores, ld, s);
    note_launch(DSA_KERNEL_INDEXER_SIMT);
    return e;
}

}  // namespace dsa
