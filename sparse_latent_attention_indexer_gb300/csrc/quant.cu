// FP8 e4m3 quantisation with power-of-two (ue8m0) scales per block of 128
// values: the indexer inputs in the released configuration's fp8 / ue8m0
// format (config_671B_v3.2.json excerpt, "DeepSeek-V3.2-Exp - Block input").
//
// One warp per block: each lane holds 4 consecutive values, the warp takes
// the absolute maximum with shuffles, the exponent is found exactly from the
// binary exponent of amax (no division), and each value is scaled by an exact
// power of two and converted with the hardware's round-to-nearest-even,
// saturating e4m3 conversion.  A warp takes BPW consecutive blocks and loads
// all of them (one 8- or 16-byte load per lane and block) before converting
// the first, so enough bytes are in flight to keep HBM busy.  HBM-bound: 2 (or
// 4) bytes read + 1 byte written per value.
#include <cuda_fp8.h>

#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int BPW = 4;  // blocks per warp

template <typename T>
__device__ __forceinline__ void load4(const T *p, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16 *p, float (&v)[4]) {
    const uint2 u = __ldg((const uint2 *)p);  // 8-byte aligned: checked on the host
    const __nv_bfloat162 a = *(const __nv_bfloat162 *)&u.x, b = *(const __nv_bfloat162 *)&u.y;
    v[0] = __low2float(a);
    v[1] = __high2float(a);
    v[2] = __low2float(b);
    v[3] = __high2float(b);
}
template <>
__device__ __forceinline__ void load4<float>(const float *p, float (&v)[4]) {
    const float4 u = __ldg((const float4 *)p);  // 16-byte aligned: checked on the host
    v[0] = u.x;
    v[1] = u.y;
    v[2] = u.z;
    v[3] = u.w;
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(256) quant_e4m3_kernel(const T *__restrict__ x, int64_t n_blocks,
                                                         uint8_t *__restrict__ codes, float *__restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t blk0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * BPW;
    float v[BPW][4];
#pragma unroll
    for (int b = 0; b < BPW; ++b) {
        const int64_t blk = blk0 + b;
        if (blk < n_blocks) {
            const T *src = x + blk * 128 + lane * 4;
            if (VEC) {
                load4<T>(src, v[b]);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) v[b][i] = to_f32(src[i]);
            }
        }
    }
#pragma unroll
    for (int b = 0; b < BPW; ++b) {
        const int64_t blk = blk0 + b;
        if (blk >= n_blocks) break;  // warp-uniform
        float amax = fmaxf(fmaxf(fabsf(v[b][0]), fabsf(v[b][1])), fmaxf(fabsf(v[b][2]), fabsf(v[b][3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int e = ue8m0_exponent(amax);
        const float inv = ldexpf(1.0f, -e);  // exact power of two
        uint32_t packed = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(v[b][i] * inv, __NV_SATFINITE, __NV_E4M3);
            packed |= (uint32_t)c << (8 * i);
        }
        reinterpret_cast<uint32_t *>(codes + blk * 128)[lane] = packed;
        if (lane == 0) scales[blk] = ldexpf(1.0f, e);
    }
}

}  // namespace

cudaError_t launch_quant_e4m3(const void *x, int x_dtype, int64_t n_blocks, uint8_t *codes, float *scales,
                              cudaStream_t s) {
    if (n_blocks == 0) return cudaSuccess;
    const int per_cta = 8 * BPW;  // blocks per CTA of 8 warps
    const int64_t grid = (n_blocks + per_cta - 1) / per_cta;
    const uintptr_t a = (uintptr_t)x;
    if (x_dtype == DSA_BF16) {
        auto *p = (const __nv_bfloat16 *)x;
        if (a % 8 == 0)
            quant_e4m3_kernel<__nv_bfloat16, true><<<(unsigned)grid, 256, 0, s>>>(p, n_blocks, codes, scales);
        else
            quant_e4m3_kernel<__nv_bfloat16, false><<<(unsigned)grid, 256, 0, s>>>(p, n_blocks, codes, scales);
    } else {
        auto *p = (const float *)x;
        if (a % 16 == 0)
            quant_e4m3_kernel<float, true><<<(unsigned)grid, 256, 0, s>>>(p, n_blocks, codes, scales);
        else
            quant_e4m3_kernel<float, false><<<(unsigned)grid, 256, 0, s>>>(p, n_blocks, codes, scales);
    }
    note_launch(DSA_KERNEL_QUANT);
    return cudaGetLastError();
}

}  // namespace dsa
