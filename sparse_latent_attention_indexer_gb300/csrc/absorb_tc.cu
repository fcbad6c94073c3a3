// Per-head absorption GEMMs of the latent attention on tcgen05 tensor cores:
//   q~[m,h,:]  = q_nope[m,h,:] . W_UK[h]   (K = d_n = 128, N = d_c = 512)
//   out[m,h,:] = o_lat[m,h,:]  . W_UV[h]   (K = d_c = 512, N = d_v = 128)
// (DeepSeek-V3.2-Exp atlas page, MoE transformer block: k^C = c^KV W_UK and
// v = c^KV W_UV, with W_UK folded into the query and W_UV applied to the
// latent context -- the absorbed form.)
//
// A CTA owns one head h and one N tile; the head's weight tile
// (N_TILE x K_TOTAL bf16) is loaded once by TMA and stays in shared memory,
// while 128-row blocks of A stream through a ring of 64-column slabs.  The
// weights are stored [K][N] (N contiguous), so the B operand is read
// MN-major straight from the TMA tile; A rows are K-major.  The fp32
// accumulators live in tensor memory (two buffers, so the epilogue of one
// row block overlaps the MMAs of the next); the epilogue converts to bf16 and
// stores.  For q~ the CTA holding the last N tile also copies q_pe into
// columns d_c .. d_c + d_r of the q~ row, so the attention kernel reads one
// contiguous [q~ | q_pe] row per head.
#include "tc_common.cuh"

namespace dsa {

__device__ int g_absorb_tc_error = 0;

namespace {

constexpr int BM = 128;
constexpr int NUM_THREADS = 384;
constexpr int EPI_WARP0 = 4;
constexpr int STAGES = 4;
constexpr int SLAB = BM * 128;  // one 64-column bf16 slab of a 128-row block: 16 KB

struct AbsorbParams {
    int M, H;
    int n_tiles;         // N / N_TILE
    int msplit;          // CTAs per (head, n tile); row blocks are strided across them
    int64_t ldc_row;     // elements between rows m and m+1 of C
    int ldc_head;        // elements between heads h and h+1 of C
    int d_r;             // q_pe width copied after the GEMM columns (0: none)
    int n_total;         // N of the whole GEMM (column offset of the q_pe copy)
};

template <int K_TOTAL, int N_TILE>
struct ACfg {
    static constexpr int B_BYTES = N_TILE * K_TOTAL * 2;
    static constexpr int SLABS = K_TOTAL / 64;
    static constexpr int SMEM = 1024 + B_BYTES + STAGES * SLAB + 256;
    static constexpr uint32_t IDESC = tc::instr_desc(tc::kFmtBF16, tc::kFmtBF16, BM, N_TILE, 0, 1);
};

template <int K_TOTAL, int N_TILE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    absorb_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ AbsorbParams P, __nv_bfloat16 *__restrict__ C,
                     const __nv_bfloat16 *__restrict__ pe_src) {
    using G = ACfg<K_TOTAL, N_TILE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *Bt = base;                  // [N_TILE/64 MN blocks][K_TOTAL rows][128 B]
    uint8_t *As = Bt + G::B_BYTES;       // [STAGES][128 rows][128 B]
    uint64_t *bars = (uint64_t *)(As + STAGES * SLAB);
    uint64_t *full = bars, *empty = bars + STAGES, *bfull = bars + 2 * STAGES;
    uint64_t *tfull = bfull + 1, *tempty = tfull + 2, *mmadone = tempty + 2;
    uint32_t *tmem_slot = (uint32_t *)(mmadone + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    __shared__ int never;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ms = blockIdx.x % P.msplit;
    const int nt = (blockIdx.x / P.msplit) % P.n_tiles;
    const int h = blockIdx.x / (P.msplit * P.n_tiles);
    const int n0 = nt * N_TILE;
    const int mblocks = (P.M + BM - 1) / BM;
    const int mine = ms < mblocks ? (mblocks - ms + P.msplit - 1) / P.msplit : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], 1);
        }
        tc::mbar_init(bfull, 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&tfull[i], 1);
            tc::mbar_init(&tempty[i], 8);
        }
        tc::mbar_init(mmadone, 1);
        *abort_flag = 0;
        never = 0;
        tc::fence_mbar_init();
    }
    if (warp == 2) {
        tc::tmem_alloc(tmem_slot, 2 * N_TILE);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    volatile int *nv = (volatile int *)&never;

    if (mine > 0) {
        if (warp == 0 && lane == 0) {
            tc::prefetch_tmap(&tm_a);
            tc::prefetch_tmap(&tm_b);
            // B: N_TILE/64 column blocks x K_TOTAL/128 row boxes of [128 rows][64 cols]
            tc::mbar_arrive_expect_tx(bfull, G::B_BYTES);
            for (int nb = 0; nb < N_TILE / 64; ++nb)
                for (int kb = 0; kb < K_TOTAL / 128; ++kb)
                    tc::tma_load_3d(Bt + (nb * K_TOTAL + kb * 128) * 128, &tm_b, bfull, n0 + nb * 64, kb * 128, h);
            int issued = 0;
            for (int i = 0; i < mine; ++i) {
                const int m0 = (ms + i * P.msplit) * BM;
                for (int j = 0; j < G::SLABS; ++j) {
                    const int it = i * G::SLABS + j, st = it % STAGES;
                    if (!tc::mbar_wait(&empty[st], ((it / STAGES) & 1) ^ 1, abort_flag, &g_absorb_tc_error, 11))
                        goto producer_done;
                    tc::mbar_arrive_expect_tx(&full[st], SLAB);
                    tc::tma_load_3d(As + st * SLAB, &tm_a, &full[st], j * 64, h, m0);
                    ++issued;
                }
            }
        producer_done:
            tc::mbar_wait(bfull, 0, nv, &g_absorb_tc_error, 12);
            for (int j = max(0, issued - STAGES); j < issued; ++j)
                tc::mbar_wait(&full[j % STAGES], (j / STAGES) & 1, nv, &g_absorb_tc_error, 13);
        } else if (warp == 1 && lane == 0) {
            bool ok = tc::mbar_wait(bfull, 0, abort_flag, &g_absorb_tc_error, 14);
            const uint32_t b0 = tc::smem_u32(Bt);
            int issued = 0;
            for (int i = 0; ok && i < mine; ++i) {
                const int acc = i & 1;
                if (!tc::mbar_wait(&tempty[acc], ((i >> 1) & 1) ^ 1, abort_flag, &g_absorb_tc_error, 15)) break;
                const uint32_t d = tmem + acc * N_TILE;
                for (int j = 0; ok && j < G::SLABS; ++j) {
                    const int it = i * G::SLABS + j, st = it % STAGES;
                    if (!tc::mbar_wait(&full[st], (it / STAGES) & 1, abort_flag, &g_absorb_tc_error, 16)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t a0 = tc::smem_u32(As + st * SLAB);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const int krow = j * 64 + kk * 16;  // K rows of the MN-major B tile
                        const uint64_t ad = tc::smem_desc(a0 + kk * 32, 16, 1024);
                        const uint64_t bd = tc::smem_desc(b0 + krow * 128, K_TOTAL * 128, 1024);
                        tc::mma_f16(d, ad, bd, G::IDESC, (j | kk) != 0);
                    }
                    tc::mma_commit(&empty[st]);
                    ++issued;
                }
                if (!ok) break;
                tc::mma_commit(&tfull[acc]);
            }
            if (issued > 0) {
                tc::mma_commit(mmadone);
                tc::mbar_wait(mmadone, 0, nv, &g_absorb_tc_error, 17);
            }
        } else if (warp >= EPI_WARP0) {
            const int q = warp & 3, half = (warp - EPI_WARP0) >> 2;
            constexpr int COLS = N_TILE / 2;  // columns per epilogue warp
            for (int i = 0; i < mine; ++i) {
                const int acc = i & 1;
                if (!tc::mbar_wait(&tfull[acc], (i >> 1) & 1, abort_flag, &g_absorb_tc_error, 18)) break;
                tc::tc_fence_after();
                const int m = (ms + i * P.msplit) * BM + q * 32 + lane;
                __nv_bfloat16 *crow = C + (int64_t)m * P.ldc_row + (int64_t)h * P.ldc_head + n0 + half * COLS;
#pragma unroll 1
                for (int c0 = 0; c0 < COLS; c0 += 32) {
                    float v[32];
                    tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + acc * N_TILE + half * COLS + c0, v);
                    tc::tmem_ld_wait();
                    if (m < P.M) {
                        uint4 pk[4];
                        uint32_t *pw = (uint32_t *)pk;
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            __nv_bfloat162 t2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                            pw[e] = *(uint32_t *)&t2;
                        }
                        uint4 *dst = (uint4 *)(crow + c0);
#pragma unroll
                        for (int e = 0; e < 4; ++e) dst[e] = pk[e];
                    }
                }
                if (pe_src && nt == P.n_tiles - 1 && half == 1 && m < P.M) {
                    const uint4 *src = (const uint4 *)(pe_src + ((int64_t)m * P.H + h) * P.d_r);
                    uint4 *dst = (uint4 *)(C + (int64_t)m * P.ldc_row + (int64_t)h * P.ldc_head + P.n_total);
                    for (int e = 0; e < P.d_r / 8; ++e) dst[e] = src[e];
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&tempty[acc]);
            }
        }
    }
    __syncthreads();
    if (warp == 2) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 2 * N_TILE);
    }
}

template <int K_TOTAL, int N_TILE>
cudaError_t launch_absorb(const void *A, const void *W, void *C, int M, int H, int N, int64_t ldc_row, int ldc_head,
                          const void *pe_src, int d_r, cudaStream_t s) {
    using G = ACfg<K_TOTAL, N_TILE>;
    CUtensorMap ta, tb;
    {
        uint64_t dims[3] = {(uint64_t)K_TOTAL, (uint64_t)H, (uint64_t)M};
        uint64_t strides[2] = {(uint64_t)K_TOTAL * 2, (uint64_t)H * K_TOTAL * 2};
        uint32_t box[3] = {64, 1, BM};
        if (!make_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, A, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        uint64_t dims[3] = {(uint64_t)N, (uint64_t)K_TOTAL, (uint64_t)H};
        uint64_t strides[2] = {(uint64_t)N * 2, (uint64_t)K_TOTAL * N * 2};
        uint32_t box[3] = {64, 128, 1};
        if (!make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, W, dims, strides, box)) return cudaErrorInvalidValue;
    }
    AbsorbParams P;
    P.M = M;
    P.H = H;
    P.n_tiles = N / N_TILE;
    const int mblocks = (M + BM - 1) / BM;
    const int base_ctas = H * P.n_tiles;
    // Enough CTAs to fill the GPU about twice, without splitting a head's rows finer than 2 blocks per CTA.
    P.msplit = std::max(1, std::min((2 * 152 + base_ctas - 1) / base_ctas, std::max(1, mblocks / 2)));
    P.ldc_row = ldc_row;
    P.ldc_head = ldc_head;
    P.d_r = d_r;
    P.n_total = N;
    cudaError_t e = cudaFuncSetAttribute(absorb_tc_kernel<K_TOTAL, N_TILE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
    if (e != cudaSuccess) return e;
    absorb_tc_kernel<K_TOTAL, N_TILE><<<base_ctas * P.msplit, NUM_THREADS, G::SMEM, s>>>(
        ta, tb, P, (__nv_bfloat16 *)C, (const __nv_bfloat16 *)pe_src);
    note_launch(DSA_KERNEL_ABSORB_TC);
    return cudaGetLastError();
}

}  // namespace

bool absorb_tc_supported(int dtype, int H, int d_n, int d_r, int d_c, int d_v) {
    return dtype == DSA_BF16 && d_n == 128 && d_c == 512 && d_v == 128 && d_r % 8 == 0 && H >= 1;
}

cudaError_t launch_absorb_q_tc(const void *q_nope, const void *W_UK, const void *q_pe, void *qt, int M, int H,
                               int d_r, cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    const int W = 512 + d_r;  // q~ row: [q_nope W_UK (512) | q_pe (d_r)]
    return launch_absorb<128, 256>(q_nope, W_UK, qt, M, H, 512, (int64_t)H * W, W, q_pe, d_r, s);
}

cudaError_t launch_absorb_v_tc(const void *olat, const void *W_UV, void *out, int M, int H, cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    return launch_absorb<512, 128>(olat, W_UV, out, M, H, 128, (int64_t)H * 128, 128, nullptr, 0, s);
}

int absorb_tc_read_error(int *site) {
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_absorb_tc_error, sizeof(int));
    if (e != cudaSuccess) return fail_cuda(e);
    if (v) {
        e = cudaMemcpyToSymbol(g_absorb_tc_error, &zero, sizeof(int));
        if (e != cudaSuccess) return fail_cuda(e);
        if (site) *site = v;
        return DSA_ERR_TIMEOUT;
    }
    return DSA_OK;
}

}  // namespace dsa
