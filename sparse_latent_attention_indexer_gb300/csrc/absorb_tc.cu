// Per-head absorption GEMMs of the latent attention on tcgen05 tensor cores:
//   q~[m,h,:]  = q_nope[m,h,:] . W_UK[h]   (K = d_n = 128, N = d_c = 512)
//   out[m,h,:] = o_lat[m,h,:]  . W_UV[h]   (K = d_c = 512, N = d_v = 128)
// (DeepSeek-V3.2-Exp atlas page, MoE transformer block: k^C = c^KV W_UK and
// v = c^KV W_UV, with W_UK folded into the query and W_UV applied to the
// latent context -- the absorbed form.)
//
// Both GEMMs move far more bytes than they compute (q~ alone is 1 KB of
// output per head row), so the kernel is built around HBM traffic:
//   * Work unit = (head h, N tile, 128-row block).  The grid is persistent,
//     one CTA per SM, and each CTA takes a contiguous range of units, so it
//     meets at most a few (head, N tile) pairs; the pair's weight tile
//     (N_TILE x K_TOTAL bf16) is loaded by TMA when the pair changes and stays
//     in shared memory.  The weights are stored [K][N] (N contiguous), so the
//     B operand is read MN-major straight from the TMA tile; A rows are
//     K-major and stream through a ring of 64-column slabs.
//   * The fp32 accumulators live in tensor memory, double-buffered, so the
//     epilogue of one unit overlaps the MMAs of the next.
//   * Epilogue: eight warps convert to bf16 into a 128-byte-swizzled staging
//     tile in shared memory, and one thread writes it with TMA tensor stores
//     (whole 128-byte row segments instead of 32 scattered rows per store
//     instruction).
// Warp roles: 0 TMA loads, 1 MMA issue, 2 tensor-memory owner, 4-11 epilogue.
// Every wait is bounded; a timeout records its site in the device error word.
#include "tc_common.cuh"

namespace dsa {

__device__ int g_absorb_tc_error = 0;

namespace {

constexpr int BM = 128;
constexpr int NUM_THREADS = 384;
constexpr int EPI_WARP0 = 4;
constexpr int HALF_THREADS = 128;  // the four epilogue warps of one column half
constexpr int STAGES = 4;
constexpr int SLAB = BM * 128;  // one 64-column bf16 slab of a 128-row block: 16 KB

struct AbsorbParams {
    int M, H;
    int n_tiles;  // N / N_TILE
    int mblocks;  // 128-row blocks of M
    int units;    // H * n_tiles * mblocks
    long long wait_limit;  // SM cycles a wait may take before the CTA gives up (the drains keep the default)
};

template <int K_TOTAL, int N_TILE>
struct ACfg {
    static constexpr int B_BYTES = N_TILE * K_TOTAL * 2;
    static constexpr int SLABS = K_TOTAL / 64;
    static constexpr int C_BYTES = BM * N_TILE * 2;  // bf16 staging of one output tile
    static constexpr int SMEM = 1024 + B_BYTES + STAGES * SLAB + C_BYTES + 256;
    static constexpr uint32_t IDESC = tc::instr_desc(tc::kFmtBF16, tc::kFmtBF16, BM, N_TILE, 0, 1);
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

// The HALF_THREADS threads of one column half arrive; returns the AND of `v` over them.
__device__ __forceinline__ bool epi_bar_and(uint32_t id, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"((uint32_t)HALF_THREADS)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void epi_bar(uint32_t id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"((uint32_t)HALF_THREADS) : "memory");
}

struct Unit {
    int pair, h, n0, m0;
};
template <int N_TILE>
__device__ __forceinline__ Unit unit_of(const AbsorbParams &P, int u) {
    Unit x;
    x.pair = u / P.mblocks;
    x.m0 = (u - x.pair * P.mblocks) * BM;
    x.h = x.pair / P.n_tiles;
    x.n0 = (x.pair - x.h * P.n_tiles) * N_TILE;
    return x;
}

template <int K_TOTAL, int N_TILE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    absorb_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ AbsorbParams P) {
    using G = ACfg<K_TOTAL, N_TILE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *Bt = base;                  // [N_TILE/64 MN blocks][K_TOTAL rows][128 B]
    uint8_t *As = Bt + G::B_BYTES;       // [STAGES][128 rows][128 B]
    uint8_t *Cs = As + STAGES * SLAB;    // [N_TILE/64 column blocks][128 rows][128 B], 128-byte swizzle
    uint64_t *bars = (uint64_t *)(Cs + G::C_BYTES);
    uint64_t *full = bars, *empty = bars + STAGES, *bfull = bars + 2 * STAGES, *bfree = bfull + 1;
    uint64_t *tfull = bfree + 1, *tempty = tfull + 2, *mmadone = tempty + 2;
    uint32_t *tmem_slot = (uint32_t *)(mmadone + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    __shared__ int never;
    int *err = &g_absorb_tc_error;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int u0 = (int)((int64_t)blockIdx.x * P.units / gridDim.x);
    const int u1 = (int)((int64_t)(blockIdx.x + 1) * P.units / gridDim.x);
    const int mine = u1 - u0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], 1);
        }
        tc::mbar_init(bfull, 1);
        tc::mbar_init(bfree, 1);
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
    pdl_wait();  // the set-up above overlapped the previous kernel; global memory only from here

    if (mine > 0) {
        if (warp == 0 && lane == 0) {
            // ---------------- TMA producer ----------------
            tc::prefetch_tmap(&tm_a);
            tc::prefetch_tmap(&tm_b);
            int prev = -1, nb = 0, issued = 0;
            for (int i = 0; i < mine; ++i) {
                const Unit x = unit_of<N_TILE>(P, u0 + i);
                if (x.pair != prev) {
                    // the MMAs that read the previous pair's weights must be done before they are replaced
                    if (nb > 0 && !tc::mbar_wait(bfree, (nb - 1) & 1, abort_flag, err, 11, P.wait_limit)) break;
                    // B: N_TILE/64 column blocks x K_TOTAL/128 row boxes of [128 rows][64 cols]
                    tc::mbar_arrive_expect_tx(bfull, G::B_BYTES);
                    for (int c = 0; c < N_TILE / 64; ++c)
                        for (int kb = 0; kb < K_TOTAL / 128; ++kb)
                            tc::tma_load_3d(Bt + (c * K_TOTAL + kb * 128) * 128, &tm_b, bfull, x.n0 + c * 64,
                                            kb * 128, x.h);
                    ++nb;
                    prev = x.pair;
                }
                bool ok = true;
                for (int j = 0; j < G::SLABS; ++j) {
                    const int it = i * G::SLABS + j, st = it % STAGES;
                    if (!(ok = tc::mbar_wait(&empty[st], ((it / STAGES) & 1) ^ 1, abort_flag, err, 12, P.wait_limit))) break;
                    tc::mbar_arrive_expect_tx(&full[st], SLAB);
                    tc::tma_load_3d(As + st * SLAB, &tm_a, &full[st], j * 64, x.h, x.m0);
                    ++issued;
                }
                if (!ok) break;
            }
            // Drain: nothing may still be landing in shared memory when the CTA exits.
            if (nb > 0) tc::mbar_wait(bfull, (nb - 1) & 1, nv, err, 13);
            for (int j = max(0, issued - STAGES); j < issued; ++j)
                tc::mbar_wait(&full[j % STAGES], (j / STAGES) & 1, nv, err, 14);
        } else if (warp == 1 && lane == 0) {
            // ---------------- MMA issuer ----------------
            const uint32_t b0 = tc::smem_u32(Bt);
            int prev = -1, nb = 0, issued = 0;
            bool ok = true;
            for (int i = 0; ok && i < mine; ++i) {
                const Unit x = unit_of<N_TILE>(P, u0 + i);
                if (x.pair != prev) {
                    if (nb > 0) tc::mma_commit(bfree);  // arrives once every MMA on the old weights is done
                    if (!(ok = tc::mbar_wait(bfull, nb & 1, abort_flag, err, 15, P.wait_limit))) break;
                    ++nb;
                    prev = x.pair;
                }
                const int acc = i & 1;
                if (!(ok = tc::mbar_wait(&tempty[acc], ((i >> 1) & 1) ^ 1, abort_flag, err, 16, P.wait_limit))) break;
                const uint32_t d = tmem + acc * N_TILE;
                for (int j = 0; j < G::SLABS; ++j) {
                    const int it = i * G::SLABS + j, st = it % STAGES;
                    if (!(ok = tc::mbar_wait(&full[st], (it / STAGES) & 1, abort_flag, err, 17, P.wait_limit))) break;
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
                tc::mbar_wait(mmadone, 0, nv, err, 18);
            }
        } else if (warp >= EPI_WARP0) {
            // ---------------- epilogue ----------------
            // The two column halves (four warps each) run independently: each stages its half of
            // the tile and one of its threads stores that half, so neither waits for the other.
            const int q = warp & 3, half = (warp - EPI_WARP0) >> 2;
            const int row = q * 32 + lane;
            const bool leader = lane == 0 && q == 0;  // warp 4 (half 0) or warp 8 (half 1)
            const uint32_t bar_free = 1 + 2 * half, bar_done = 2 + 2 * half;
            constexpr int COLS = N_TILE / 2;  // columns per epilogue thread
            for (int i = 0; i < mine; ++i) {
                const int acc = i & 1;
                bool ok = tc::mbar_wait(&tfull[acc], (i >> 1) & 1, abort_flag, err, 19, P.wait_limit);
                // The previous unit's TMA stores must have read the staging tile before it is rewritten.
                if (leader) tc::bulk_wait_read_all();
                if (!epi_bar_and(bar_free, ok)) break;
                tc::tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < COLS; c0 += 32) {
                    float v[32];
                    tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + acc * N_TILE + half * COLS + c0, v);
                    tc::tmem_ld_wait();
                    uint32_t pw[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const __nv_bfloat162 t2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                        pw[e] = *(const uint32_t *)&t2;
                    }
                    // 32 columns = half of a 128-byte row segment of column block cb (chunks j0..j0+3)
                    const int col = half * COLS + c0, cb = col >> 6, j0 = (col & 63) >> 3;
                    uint8_t *dst = Cs + cb * (BM * 128) + row * 128;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        *(uint4 *)(dst + (((j0 + e) ^ (row & 7)) << 4)) =
                            make_uint4(pw[4 * e], pw[4 * e + 1], pw[4 * e + 2], pw[4 * e + 3]);
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&tempty[acc]);
                tc::fence_proxy_async_smem();  // the staging tile is read by the TMA store (async proxy)
                epi_bar(bar_done);
                if (leader) {
                    const Unit x = unit_of<N_TILE>(P, u0 + i);
                    for (int cb = half * (COLS / 64); cb < (half + 1) * (COLS / 64); ++cb)
                        tc::tma_store_3d(&tm_c, Cs + cb * (BM * 128), x.n0 + cb * 64, x.h, x.m0);
                    tc::bulk_commit_group();
                }
            }
            if (leader) tc::bulk_wait_all();
        }
    }
    __syncthreads();
    if (warp == 2) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 2 * N_TILE);
    }
}

int sm_count() {
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

template <int K_TOTAL, int N_TILE>
cudaError_t launch_absorb(const void *A, const void *W, void *C, int M, int H, int N, cudaStream_t s) {
    using G = ACfg<K_TOTAL, N_TILE>;
    CUtensorMap ta, tb, tcm;
    {
        // A rows [M, H, K_TOTAL]: boxes of 64 columns x 1 head x 128 rows
        uint64_t dims[3] = {(uint64_t)K_TOTAL, (uint64_t)H, (uint64_t)M};
        uint64_t strides[2] = {(uint64_t)K_TOTAL * 2, (uint64_t)H * K_TOTAL * 2};
        uint32_t box[3] = {64, 1, BM};
        if (!make_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, A, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        // weights [H, K_TOTAL, N]: boxes of 64 columns x 128 K rows
        uint64_t dims[3] = {(uint64_t)N, (uint64_t)K_TOTAL, (uint64_t)H};
        uint64_t strides[2] = {(uint64_t)N * 2, (uint64_t)K_TOTAL * N * 2};
        uint32_t box[3] = {64, 128, 1};
        if (!make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, W, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        // C rows [M, H, N]: stored as boxes of 64 columns x 1 head x 128 rows (rows past M are not written)
        uint64_t dims[3] = {(uint64_t)N, (uint64_t)H, (uint64_t)M};
        uint64_t strides[2] = {(uint64_t)N * 2, (uint64_t)H * N * 2};
        uint32_t box[3] = {64, 1, BM};
        if (!make_tmap(&tcm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, C, dims, strides, box)) return cudaErrorInvalidValue;
    }
    AbsorbParams P;
    P.M = M;
    P.H = H;
    P.n_tiles = N / N_TILE;
    P.mblocks = (M + BM - 1) / BM;
    P.units = H * P.n_tiles * P.mblocks;
    P.wait_limit = wait_limit_cycles();
    const int grid = std::min(P.units, sm_count());
    cudaError_t e = cudaFuncSetAttribute(absorb_tc_kernel<K_TOTAL, N_TILE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
    if (e != cudaSuccess) return e;
    e = launch_pdl(absorb_tc_kernel<K_TOTAL, N_TILE>, dim3(grid), dim3(NUM_THREADS), G::SMEM, s, ta, tb, tcm, P);
    if (e != cudaSuccess) return e;
    note_launch(DSA_KERNEL_ABSORB_TC);
    return cudaGetLastError();
}

}  // namespace

bool absorb_tc_supported(int dtype, int H, int d_n, int d_r, int d_c, int d_v) {
    return dtype == DSA_BF16 && d_n == 128 && d_c == 512 && d_v == 128 && d_r % 8 == 0 && H >= 1;
}

cudaError_t launch_absorb_q_tc(const void *q_nope, const void *W_UK, void *qt, int M, int H, cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    return launch_absorb<128, 256>(q_nope, W_UK, qt, M, H, 512, s);
}

cudaError_t launch_absorb_v_tc(const void *olat, const void *W_UV, void *out, int M, int H, cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    return launch_absorb<512, 128>(olat, W_UV, out, M, H, 128, s);
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
