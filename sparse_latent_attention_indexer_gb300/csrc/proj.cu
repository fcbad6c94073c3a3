// The projections on either side of the path, as library entry points:
//
//   * the step before it -- the key side of the new tokens and their append to
//     the caches ("DeepSeek-V3.2-Exp - Attention input" page, mla-init and
//     mla-kv excerpts; "Block input" page, RMSNorm excerpt; nnterp deepseek_v32
//     printout of the indexer and its note on the de-interleaved rotary part):
//         Y       = x . [wkv_a; wk; weights_proj]^T      (one stacked GEMM, fp32)
//         latent  = kv_norm(Y[:, 0:d_c])                 RMSNorm, gain, eps 1e-6
//         k_pe    = rotary(Y[:, d_c:d_c+d_r], position)  pair (2i, 2i+1) -> dims i, d_r/2 + i
//         k^I     = k_norm(Y[:, ... D_I])                LayerNorm, gain and bias, eps 1e-6
//         w       = Y[:, ... H_I]                        the indexer's per-head weights
//     then [latent | k_pe] (bf16) and k^I (bf16, or e4m3 codes + ue8m0 scale)
//     are written to the token's cache row;
//   * the step after it -- the output projection y = out . wo^T on the
//     attention output with the heads side by side (mla-init excerpt, wo).
//
// The GEMMs run on the tcgen05 kernel of gemm_tc.cu; the per-token norms, the
// rotation and the append run in prologue_kernel below (one warp per token;
// HBM-bound: about 3 KB of fp32 read and 1.4 KB written per token).
#include <cuda_fp8.h>

#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr float kNormEps = 1e-6f;  // kv_norm and k_norm (printout: eps=1e-06)

struct ProParams {
    SeqTab st;
    int n;          // tokens
    int ldy;        // columns of Y
    int d_c, d_r, D_I, H_I;
    int64_t ld_kv;
    int k_fp8;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(256) prologue_kernel(const float *__restrict__ Y, const float *__restrict__ kv_gain,
                                                       const float *__restrict__ k_gain,
                                                       const float *__restrict__ k_bias,
                                                       const float *__restrict__ rope_cos,
                                                       const float *__restrict__ rope_sin,
                                                       const __grid_constant__ ProParams P,
                                                       __nv_bfloat16 *__restrict__ kv_cache, void *__restrict__ k_cache,
                                                       float *__restrict__ k_scale, float *__restrict__ w) {
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= P.n) return;
    const RowInfo ri = row_info(P.st, r);
    const int64_t slot = (int64_t)ri.kbase + ri.p;  // the token's cache row
    const float *y = Y + (int64_t)r * P.ldy;
    __nv_bfloat16 *kv = kv_cache + slot * P.ld_kv;

    // kv_norm: RMSNorm of the latent, in fp32
    float ss = 0.0f;
    for (int i = lane; i < P.d_c; i += 32) ss = fmaf(y[i], y[i], ss);
    const float inv = rsqrtf(warp_sum(ss) / (float)P.d_c + kNormEps);
    for (int i = lane; i < P.d_c; i += 32) kv[i] = __float2bfloat16_rn(kv_gain[i] * (y[i] * inv));

    // rotary k_pe, de-interleaved: pair (2i, 2i+1) -> dims i and half + i
    const int half = P.d_r / 2;
    const float *pe = y + P.d_c;
    for (int i = lane; i < half; i += 32) {
        const float a = pe[2 * i], b = pe[2 * i + 1];
        const float c = rope_cos[(int64_t)ri.p * half + i], s = rope_sin[(int64_t)ri.p * half + i];
        kv[P.d_c + i] = __float2bfloat16_rn(a * c - b * s);
        kv[P.d_c + half + i] = __float2bfloat16_rn(a * s + b * c);
    }

    // k_norm: LayerNorm of the indexer key (two passes: mean, then the mean square deviation)
    const float *ky = y + P.d_c + P.d_r;
    constexpr int KMAX = 8;  // D_I <= 256
    float kvv[KMAX];
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        const int i = lane + 32 * j;
        kvv[j] = i < P.D_I ? ky[i] : 0.0f;
        sum += kvv[j];
    }
    const float mean = warp_sum(sum) / (float)P.D_I;
    float dev = 0.0f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        const int i = lane + 32 * j;
        const float d = i < P.D_I ? kvv[j] - mean : 0.0f;
        dev = fmaf(d, d, dev);
    }
    const float kinv = rsqrtf(warp_sum(dev) / (float)P.D_I + kNormEps);
    float kn[KMAX];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        const int i = lane + 32 * j;
        // the cache holds the key rounded to bf16; the FP8 codes are taken from that bf16 value
        kn[j] = i < P.D_I ? __bfloat162float(__float2bfloat16_rn((kvv[j] - mean) * kinv * k_gain[i] + k_bias[i]))
                          : 0.0f;
        amax = fmaxf(amax, fabsf(kn[j]));
    }
    if (P.k_fp8) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int e = ue8m0_exponent(amax);
        const float sc = ldexpf(1.0f, -e);  // exact power of two
        uint8_t *kc = (uint8_t *)k_cache + slot * P.D_I;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            const int i = lane + 32 * j;
            if (i < P.D_I) kc[i] = (uint8_t)__nv_cvt_float_to_fp8(kn[j] * sc, __NV_SATFINITE, __NV_E4M3);
        }
        if (lane == 0) k_scale[slot] = ldexpf(1.0f, e);
    } else {
        __nv_bfloat16 *kb = (__nv_bfloat16 *)k_cache + slot * P.D_I;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            const int i = lane + 32 * j;
            if (i < P.D_I) kb[i] = __float2bfloat16_rn(kn[j]);
        }
    }

    // the indexer's per-head weights, as the projection gives them
    const float *wy = ky + P.D_I;
    for (int i = lane; i < P.H_I; i += 32) w[(int64_t)r * P.H_I + i] = wy[i];
}

inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }
inline bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

int check_prologue(int dim, int d_c, int d_r, int D_I, int H_I, int k_dtype) {
    if (dim < 64 || d_c < 1 || d_r < 0 || D_I < 1 || H_I < 1) return DSA_ERR_INVALID_ARG;
    if (dim % 64 || (d_c + d_r + D_I + H_I) % 64 || d_r % 2) return DSA_ERR_UNSUPPORTED;
    if (D_I > 256 || d_c > 4096 || d_r > 256) return DSA_ERR_UNSUPPORTED;
    if (k_dtype != DSA_BF16 && k_dtype != DSA_E4M3) return DSA_ERR_UNSUPPORTED;
    if (k_dtype == DSA_E4M3 && D_I != 128) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

size_t dsa_kv_prologue_workspace_size(int dim, int d_c, int d_r, int D_I, int H_I, const dsa_seqs *seqs) {
    Batch bt;
    if (check_prologue(dim, d_c, d_r, D_I, H_I, DSA_BF16) || build_batch(seqs, bt)) return 0;
    return align256((size_t)bt.total_q * (d_c + d_r + D_I + H_I) * sizeof(float)) + 256;
}

int dsa_kv_prologue(const void *x, int dim, const void *W_proj, const float *kv_gain, const float *k_gain,
                    const float *k_bias, const float *rope_cos, const float *rope_sin, int n_pos, int d_c, int d_r,
                    int D_I, int H_I, const dsa_seqs *seqs, void *kv_cache, int64_t ld_kv, void *k_cache, int k_dtype,
                    float *k_scale, float *w, void *workspace, size_t ws_bytes, void *stream) {
    reset_trace();
    int rc = check_prologue(dim, d_c, d_r, D_I, H_I, k_dtype);
    if (rc) return rc;
    Batch bt;
    if ((rc = build_batch(seqs, bt))) return rc;
    if (ld_kv < d_c + d_r) return DSA_ERR_INVALID_ARG;
    if (bt.total_q == 0) return DSA_OK;
    if (!x || !W_proj || !kv_gain || !k_gain || !k_bias || !kv_cache || !k_cache || !w) return DSA_ERR_INVALID_ARG;
    if (d_r > 0 && (!rope_cos || !rope_sin)) return DSA_ERR_INVALID_ARG;
    if (k_dtype == DSA_E4M3 && !k_scale) return DSA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W_proj)) return DSA_ERR_INVALID_ARG;
    // every position the batch appends must have a rotary angle
    for (int b = 0; b < bt.st.B; ++b) {
        const int Tb = bt.st.q_off[b + 1] - bt.st.q_off[b];
        if (Tb > 0 && bt.st.start_pos[b] + Tb > n_pos) return DSA_ERR_INVALID_ARG;
    }
    const int N = d_c + d_r + D_I + H_I;
    const size_t need = align256((size_t)bt.total_q * N * sizeof(float)) + 256;
    if (!workspace || ((uintptr_t)workspace & 255) || ws_bytes < need) return DSA_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    float *Y = (float *)workspace;
    cudaError_t e = launch_gemm_tc(x, dim, W_proj, dim, Y, N, true, bt.total_q, N, dim, s);
    if (e != cudaSuccess) return fail_cuda(e);
    static thread_local ProParams P;
    P.st = bt.st;
    P.n = bt.total_q;
    P.ldy = N;
    P.d_c = d_c;
    P.d_r = d_r;
    P.D_I = D_I;
    P.H_I = H_I;
    P.ld_kv = ld_kv;
    P.k_fp8 = k_dtype == DSA_E4M3 ? 1 : 0;
    const unsigned grid = (unsigned)((bt.total_q + 7) / 8);
    prologue_kernel<<<grid, 256, 0, s>>>(Y, kv_gain, k_gain, k_bias, rope_cos, rope_sin, P, (__nv_bfloat16 *)kv_cache,
                                         k_cache, k_scale, w);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e);
    note_launch(DSA_KERNEL_PROLOGUE);
    return DSA_OK;
}

int dsa_output_proj(const void *out, const void *wo, int M, int in_features, int d_model, void *y, void *stream) {
    reset_trace();
    if (M < 0 || in_features < 1 || d_model < 1) return DSA_ERR_INVALID_ARG;
    if (!gemm_tc_supported(M, d_model, in_features)) return DSA_ERR_UNSUPPORTED;
    if (M == 0) return DSA_OK;
    if (!out || !wo || !y || !aligned16(out) || !aligned16(wo) || !aligned16(y)) return DSA_ERR_INVALID_ARG;
    cudaError_t e = launch_gemm_tc(out, in_features, wo, in_features, y, d_model, false, M, d_model, in_features,
                                   (cudaStream_t)stream);
    return e == cudaSuccess ? DSA_OK : fail_cuda(e);
}

}  // extern "C"
