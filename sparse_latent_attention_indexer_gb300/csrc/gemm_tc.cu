// Dense bf16 GEMM on tcgen05 tensor cores for the projections on either side
// of the path:
//   C[M, N] = A[M, K] . B[N, K]^T      (fp32 accumulation; C stored bf16 or fp32)
// B is an nn.Linear weight stored [out, in], so both operands are K-major.
// Used for the stacked key-side projections of the new tokens (wkv_a, wk,
// weights_proj: "DeepSeek-V3.2-Exp - Attention input" page, mla-init and
// mla-kv excerpts; nnterp deepseek_v32 printout of the indexer) and for the
// output projection wo after the attention (mla-init excerpt, wo).
//
// Design: a persistent grid, one CTA per SM, walks 128 x 256 output tiles.
// Consecutive tiles take up to eight row blocks before the next column block,
// so the tiles in flight at once share their A and B panels in L2.  Per tile:
//   * warp 0 (one thread) streams 64-wide K slabs of A (128 rows) and B (256
//     rows) by TMA, 128-byte swizzled, through a 4-stage ring;
//   * warp 1 (one thread) issues the MMAs (M = 128, N = 256, K = 16 each, four
//     per slab) into one of two fp32 accumulators in tensor memory (2 x 256
//     columns), so the epilogue of a tile overlaps the MMAs of the next;
//   * warps 4..11 read the accumulator back (two warps per 32-lane quarter,
//     each half of the columns), convert, stage 32 KB at a time in shared
//     memory in the 128-byte-swizzled layout of the TMA store, and one thread
//     writes each chunk with two TMA tensor stores.
// Rows of A past M read as zero and rows of C past M are not written, so M is
// free; N and K must be multiples of 64.  Every wait is bounded.
#include "tc_common.cuh"

namespace dsa {

__device__ int g_gemm_tc_error = 0;

namespace {

constexpr int BM = 128, BN = 256;
constexpr int STAGES = 4;
constexpr int A_SLAB = BM * 128;                // 16 KB: 128 rows x 64 bf16
constexpr int B_SLAB = BN * 128;                // 32 KB: 256 rows x 64 bf16
constexpr int STAGE_BYTES = A_SLAB + B_SLAB;
constexpr int C_STAGE = BM * 256;               // 32 KB: 128 rows x 256 bytes of output
constexpr int NUM_THREADS = 384;                // 0 TMA, 1 MMA, 2 TMEM owner, 3 idle, 4-11 epilogue
constexpr int EPI_WARP0 = 4;
constexpr int EPI_THREADS = 256;
constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + C_STAGE + 256;
static_assert(SMEM <= 232448, "shared memory per CTA");
constexpr uint32_t IDESC = tc::instr_desc(tc::kFmtBF16, tc::kFmtBF16, BM, BN, 0, 0);
constexpr int GROUP_M = 8;                      // row blocks per tile group

struct GemmParams {
    int M, N, K;
    int mt, nt;       // row blocks, column blocks
    int tiles;
    int kslabs;       // K / 64
    int c_f32;        // 1: C is fp32, else bf16
    long long wait_limit;
};

__device__ __forceinline__ void tile_of(const GemmParams &P, int u, int &m0, int &n0) {
    const int per_group = GROUP_M * P.nt;
    const int grp = u / per_group, r = u - grp * per_group;
    const int gm = min(GROUP_M, P.mt - grp * GROUP_M);
    m0 = (grp * GROUP_M + r % gm) * BM;
    n0 = (r / gm) * BN;
}

// The epilogue's 256 threads arrive on named barrier 1; returns the AND of `v` over them.
__device__ __forceinline__ bool epi_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"((uint32_t)EPI_THREADS)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void epi_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"((uint32_t)EPI_THREADS) : "memory");
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ GemmParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *ring = base;                        // [STAGES][A slab | B slab]
    uint8_t *Cs = ring + STAGES * STAGE_BYTES;   // [2 boxes][128 rows][128 B], 128-byte swizzle
    uint64_t *bars = (uint64_t *)(Cs + C_STAGE);
    uint64_t *full = bars, *empty = bars + STAGES, *tfull = bars + 2 * STAGES, *tempty = tfull + 2;
    uint64_t *mmadone = tempty + 2;
    uint32_t *tmem_slot = (uint32_t *)(mmadone + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    __shared__ int never;
    volatile int *nv = (volatile int *)&never;
    int *err = &g_gemm_tc_error;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grid = (int)gridDim.x;
    const int mine = P.tiles > (int)blockIdx.x ? (P.tiles - (int)blockIdx.x + grid - 1) / grid : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], 1);
        }
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
        tc::tmem_alloc(tmem_slot, 2 * BN);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // the set-up above overlapped the previous kernel; global memory only from here

    if (mine > 0) {
        if (warp == 0 && lane == 0) {
            // ---------------- TMA producer ----------------
            tc::prefetch_tmap(&tm_a);
            tc::prefetch_tmap(&tm_b);
            int it = 0;
            bool ok = true;
            for (int i = 0; ok && i < mine; ++i) {
                int m0, n0;
                tile_of(P, (int)blockIdx.x + i * grid, m0, n0);
                for (int ks = 0; ks < P.kslabs; ++ks, ++it) {
                    const int st = it % STAGES;
                    if (!(ok = tc::mbar_wait(&empty[st], ((it / STAGES) & 1) ^ 1, abort_flag, err, 51, P.wait_limit)))
                        break;
                    uint8_t *sa = ring + st * STAGE_BYTES;
                    tc::mbar_arrive_expect_tx(&full[st], STAGE_BYTES);
                    tc::tma_load_2d(sa, &tm_a, &full[st], ks * 64, m0);
                    tc::tma_load_2d(sa + A_SLAB, &tm_b, &full[st], ks * 64, n0);
                }
            }
            // Drain: nothing may still be landing in shared memory when the CTA exits.
            for (int j = max(0, it - STAGES); j < it; ++j)
                tc::mbar_wait(&full[j % STAGES], (j / STAGES) & 1, nv, err, 52);
        } else if (warp == 1 && lane == 0) {
            // ---------------- MMA issuer ----------------
            int it = 0, issued = 0;
            bool ok = true;
            for (int i = 0; ok && i < mine; ++i) {
                const int acc = i & 1;
                if (!(ok = tc::mbar_wait(&tempty[acc], ((i >> 1) & 1) ^ 1, abort_flag, err, 53, P.wait_limit))) break;
                const uint32_t d = tmem + acc * BN;
                for (int ks = 0; ks < P.kslabs; ++ks, ++it) {
                    const int st = it % STAGES;
                    if (!(ok = tc::mbar_wait(&full[st], (it / STAGES) & 1, abort_flag, err, 54, P.wait_limit))) break;
                    tc::tc_fence_after();
                    const uint32_t a0 = tc::smem_u32(ring + st * STAGE_BYTES), b0 = a0 + A_SLAB;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = tc::smem_desc(a0 + kk * 32, 16, 1024);
                        const uint64_t bd = tc::smem_desc(b0 + kk * 32, 16, 1024);
                        tc::mma_f16(d, ad, bd, IDESC, (ks | kk) != 0);
                    }
                    tc::mma_commit(&empty[st]);
                    ++issued;
                }
                if (!ok) break;
                tc::mma_commit(&tfull[acc]);
            }
            // No MMA may still be running when the tensor memory is released.
            if (issued > 0) {
                tc::mma_commit(mmadone);
                tc::mbar_wait(mmadone, 0, nv, err, 55);
            }
        } else if (warp >= EPI_WARP0) {
            // ---------------- epilogue ----------------
            // Warp (q, half): TMEM lanes (rows) 32q .. 32q+31, and half of each staged chunk's columns.
            const int q = warp & 3, half = (warp - EPI_WARP0) >> 2;
            const int row = q * 32 + lane;
            const bool leader = threadIdx.x == EPI_WARP0 * 32;
            const uint32_t lane_off = (uint32_t)(q * 32) << 16;
            const int chunk = P.c_f32 ? 64 : 128;   // columns per 32 KB chunk (256 bytes a row)
            const int hcols = chunk / 2;            // columns of one warp = one 128-byte box column
            uint8_t *dst = Cs + half * (BM * 128) + row * 128;
            for (int i = 0; i < mine; ++i) {
                const int acc = i & 1;
                const bool ok = tc::mbar_wait(&tfull[acc], (i >> 1) & 1, abort_flag, err, 56, P.wait_limit);
                if (!epi_and(ok)) break;
                tc::tc_fence_after();
                int m0, n0;
                tile_of(P, (int)blockIdx.x + i * grid, m0, n0);
                for (int c0 = 0; c0 < BN; c0 += chunk) {
                    if (n0 + c0 >= P.N) break;  // a partial last column block
                    // the previous chunk's stores have read the staging before it is rewritten
                    if (leader) tc::bulk_wait_read_all();
                    epi_sync();
                    const uint32_t col = (uint32_t)(acc * BN + c0 + half * hcols);
                    if (P.c_f32) {
                        float v[32];
                        tc::tmem_ld32(tmem + lane_off + col, v);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *(uint4 *)(dst + ((j ^ (row & 7)) << 4)) =
                                make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                           __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
                    } else {
#pragma unroll
                        for (int sub = 0; sub < 2; ++sub) {
                            float v[32];
                            tc::tmem_ld32(tmem + lane_off + col + sub * 32, v);
                            tc::tmem_ld_wait();
                            uint32_t pw[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const __nv_bfloat162 t2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                                pw[e] = *(const uint32_t *)&t2;
                            }
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                *(uint4 *)(dst + (((sub * 4 + j) ^ (row & 7)) << 4)) =
                                    make_uint4(pw[4 * j], pw[4 * j + 1], pw[4 * j + 2], pw[4 * j + 3]);
                        }
                    }
                    tc::fence_proxy_async_smem();  // the staging is read by the TMA stores (async proxy)
                    epi_sync();
                    if (leader) {
                        tc::tma_store_2d(&tm_c, Cs, n0 + c0, m0);
                        tc::tma_store_2d(&tm_c, Cs + BM * 128, n0 + c0 + hcols, m0);
                        tc::bulk_commit_group();
                    }
                }
                // every column of this accumulator has been read
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&tempty[acc]);
            }
            if (leader) tc::bulk_wait_all();
        }
    }
    __syncthreads();
    if (warp == 2) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 2 * BN);
    }
}

}  // namespace

bool gemm_tc_supported(int M, int N, int K) { return M >= 0 && N > 0 && K > 0 && N % 64 == 0 && K % 64 == 0; }

cudaError_t launch_gemm_tc(const void *A, int64_t lda, const void *B, int64_t ldb, void *C, int64_t ldc, bool c_f32,
                           int M, int N, int K, cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    if (!gemm_tc_supported(M, N, K)) return cudaErrorInvalidValue;
    CUtensorMap ta, tb, tcm;
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
        const uint64_t strides[1] = {(uint64_t)lda * 2};
        const uint32_t box[2] = {64, BM};
        if (!make_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)N};
        const uint64_t strides[1] = {(uint64_t)ldb * 2};
        const uint32_t box[2] = {64, BN};
        if (!make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[2] = {(uint64_t)N, (uint64_t)M};
        const uint64_t strides[1] = {(uint64_t)ldc * (c_f32 ? 4 : 2)};
        const uint32_t box[2] = {c_f32 ? 32u : 64u, BM};
        if (!make_tmap(&tcm, c_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, dims,
                       strides, box))
            return cudaErrorInvalidValue;
    }
    GemmParams P;
    P.M = M;
    P.N = N;
    P.K = K;
    P.mt = (M + BM - 1) / BM;
    P.nt = (N + BN - 1) / BN;
    P.tiles = P.mt * P.nt;
    P.kslabs = K / 64;
    P.c_f32 = c_f32 ? 1 : 0;
    P.wait_limit = wait_limit_cycles();
    const int grid = std::min(P.tiles, device_sm_count());
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    e = launch_pdl(gemm_tc_kernel, dim3(grid), dim3(NUM_THREADS), SMEM, s, ta, tb, tcm, P);
    if (e != cudaSuccess) return e;
    note_launch(DSA_KERNEL_GEMM_TC);
    return cudaGetLastError();
}

int gemm_tc_read_error(int *site) {
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemm_tc_error, sizeof(int));
    if (e != cudaSuccess) return fail_cuda(e);
    if (v) {
        e = cudaMemcpyToSymbol(g_gemm_tc_error, &zero, sizeof(int));
        if (e != cudaSuccess) return fail_cuda(e);
        if (site) *site = v;
        return DSA_ERR_TIMEOUT;
    }
    return DSA_OK;
}

}  // namespace dsa
