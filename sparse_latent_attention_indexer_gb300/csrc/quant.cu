// FP8 e4m3 quantisation with power-of-two (ue8m0) scales per block of 128
// values: the indexer inputs in the released configuration's fp8 / ue8m0
// format (config_671B_v3.2.json excerpt, "DeepSeek-V3.2-Exp - Block input").
//
// One warp per block: each lane holds 4 consecutive values, the warp takes
// the absolute maximum with shuffles, the exponent is found exactly from the
// binary exponent of amax (no division), and each value is scaled by an exact
// power of two and converted with the hardware's round-to-nearest-even,
// saturating e4m3 conversion.  HBM-bound: 2 (or 4) bytes read + 1 byte
// written per value.
#include <cuda_fp8.h>

#include "dsa_common.cuh"

namespace dsa {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) quant_e4m3_kernel(const T *__restrict__ x, int64_t n_blocks,
                                                         uint8_t *__restrict__ codes, float *__restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (blk >= n_blocks) return;
    const T *src = x + blk * 128 + lane * 4;
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = to_f32(src[i]);
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int e = ue8m0_exponent(amax);
    const float inv = ldexpf(1.0f, -e);  // exact power of two
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(v[i] * inv, __NV_SATFINITE, __NV_E4M3);
        packed |= (uint32_t)c << (8 * i);
    }
    reinterpret_cast<uint32_t *>(codes + blk * 128)[lane] = packed;
    if (lane == 0) scales[blk] = ldexpf(1.0f, e);
}

}  // namespace

cudaError_t launch_quant_e4m3(const void *x, int x_dtype, int64_t n_blocks, uint8_t *codes, float *scales,
                              cudaStream_t s) {
    if (n_blocks == 0) return cudaSuccess;
    const int per_cta = 8;
    const int64_t grid = (n_blocks + per_cta - 1) / per_cta;
    if (x_dtype == DSA_BF16)
        quant_e4m3_kernel<__nv_bfloat16><<<(unsigned)grid, 256, 0, s>>>((const __nv_bfloat16 *)x, n_blocks, codes,
                                                                       scales);
    else
        quant_e4m3_kernel<float><<<(unsigned)grid, 256, 0, s>>>((const float *)x, n_blocks, codes, scales);
    note_launch(DSA_KERNEL_QUANT);
    return cudaGetLastError();
}

}  // namespace dsa
