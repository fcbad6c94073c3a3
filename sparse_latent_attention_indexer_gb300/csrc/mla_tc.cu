// Sparse multi-head latent attention in absorbed form on tcgen05 tensor cores.
//
// For one query row (all 128 heads) and its selected keys s_j:
//   z[h,j]   = scale (q~[h] . c[s_j] + q_pe[h] . k_pe[s_j])      (576-wide dot)
//   P        = online softmax over j (running max, lazily rescaled)
//   o_lat[h] = sum_j P[h,j] c[s_j]                               (512-wide)
// (DeepSeek-V3.2-Exp atlas page, MoE transformer block: Q = [Q^C; Q^R],
// K_i = [K^C_i; k^R], v = c^KV W_UV, M^sel; W_UK folded into q~ beforehand
// and W_UV applied afterwards.)
//
// The 128 x 512 fp32 context alone fills a CTA's tensor memory, so a query
// row is handled by a cluster of two CTAs on two SMs.  CTA c owns latent
// columns 256c..256c+255 and rope columns 32c..32c+31 of q~ and of every key,
// so both gather the same 576 bytes per key.
//   * q~ slice: loaded once into tensor memory (the A operand of the latent
//     part of QK^T); the rope slice of q_pe sits in shared memory (A operand
//     of the two rope MMAs).
//   * Key tiles (64 keys): four gathering warps copy the selected rows with
//     cp.async (8 lanes per 128-byte segment, 128-byte swizzle for the latent
//     slabs, 64-byte swizzle for the rope half) into a 4-stage ring; a copy's
//     completion arrives on the stage's barrier by itself.
//   * One thread issues S_c = Q_c K_c^T (M = 128 heads, N = 64 keys) into one
//     of two score buffers in tensor memory, another O_c += P V_c (N = 256,
//     V read MN-major straight from the gathered tile, P from shared memory),
//     each as its inputs become ready.
//   * Two softmax groups of four warps take alternate tiles, one thread per
//     head row and 64 keys each, so one group's exchange and exponentials
//     overlap the other's.  A group rounds its CTA's partial scores
//     (log2-scaled) to fp16 and bulk-copies them into the peer's shared
//     memory; both CTAs then add the same two rounded halves, so they hold
//     bit-identical scores and take identical softmax decisions.  The
//     probabilities (bf16) overwrite the received half in place and are the
//     A operand of that tile's PV product.
//   * Lazy rescaling: the running maximum moves (and O is rescaled in tensor
//     memory) only when a tile's maximum exceeds it by more than 2^8; each
//     group hands the row maxima it used to the group of the next tile.
// Waits are bounded; a timeout records its site in the device error word and
// both CTAs drain and exit.
//
// Short batches split each row's keys across up to 8 clusters so that one
// wave fills the GPU; each split writes a normalised partial context and its
// lse, and a small combine kernel merges them.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "tc_common.cuh"

namespace dsa {

__device__ int g_mla_tc_error = 0;

namespace {

constexpr int NH = 128;                      // heads (MMA M)
constexpr int DC = 512;                      // latent width
constexpr int DR = 64;                       // rope width (q_pe rows)
constexpr int BK = 64;                       // keys per tile (MMA N of QK^T, K of PV)
// Each CTA of the pair holds 4 latent slabs (64 columns, 128-byte rows) and half of the rope
// part (32 columns, 64-byte rows) of every key: CTA c owns latent 256c..256c+255, rope 32c..32c+31.
constexpr int NSLAB = 4;
constexpr int SLAB_K = BK * 128;             // 8 KB: 64 keys x 64 columns, 128-byte swizzle
constexpr int ROPE_K = BK * 64;              // 4 KB: 64 keys x 32 rope columns, 64-byte swizzle
constexpr int KV_STAGE = NSLAB * SLAB_K + ROPE_K;  // 36 KB (a multiple of 1 KB: swizzle atoms stay aligned)
constexpr int NSTAGE = 4;
// One tile of one group: 128 head rows x 64 keys x 16 bits = 128-byte rows, 128-byte swizzle
// (chunk c of row h at c ^ (h & 7)): fp16 partial scores in flight, then bf16 probabilities.
constexpr int X_BYTES = NH * BK * 2;
constexpr int Q_BOX = NH * 128;              // 16 KB: 128 heads x 64 bf16 columns (one TMA box of q~ or o_lat)
constexpr int QR_BYTES = NH * 64;            // 8 KB: 128 heads x this CTA's 32 rope columns, 64-byte swizzle
static_assert(4 * Q_BOX <= 4 * X_BYTES, "the q~ slice is staged in the four exchange buffers");
static_assert(4 * Q_BOX <= NSTAGE * KV_STAGE, "the context is staged in the key stages");
constexpr int SMEM = 1024 + NSTAGE * KV_STAGE + 4 * X_BYTES + QR_BYTES + NSTAGE * BK + 2 * NH * 4 + 4 * NH * 4 + 320;
static_assert(SMEM <= 232448, "shared memory per CTA");
constexpr int NUM_THREADS = 448;             // warps 0, 3, 12, 13: gather; 1: QK^T; 2: TMEM, PV; 4-7, 8-11: softmax groups
constexpr uint32_t SOFT_BAR = 1;             // named barrier of the eight softmax warps (start and end only)
constexpr int NPROD = 4;                     // gathering warps
// Tensor-memory columns (512 per CTA): two score buffers (one per softmax group), the resident
// q~ slice (bf16 pairs, A operand of QK^T) and the context.
constexpr uint32_t COL_S = 0, COL_Q = 128, COL_O = 256;
constexpr uint32_t IDESC_QK = tc::instr_desc(tc::kFmtBF16, tc::kFmtBF16, NH, BK, 0, 0);
constexpr uint32_t IDESC_PV = tc::instr_desc(tc::kFmtBF16, tc::kFmtBF16, NH, 256, 0, 1);
constexpr float RESCALE_LOG2 = 8.0f;
constexpr long long kAbortQuietCycles = 1LL << 18;  // ~130 us: the wait before the final cluster barrier after an abort
constexpr float LN2 = 0.69314718055994530942f;

struct MlaParams {
    int B;
    int q_off[DSA_MAX_SEQS + 1];
    int k_base[DSA_MAX_SEQS];
    int k_len[DSA_MAX_SEQS];
    int start_pos[DSA_MAX_SEQS];
    int total_q;
    int k;             // entries per selection row
    int splits;        // clusters per row
    int prefix_valid;  // rows list their min(k, p+1) keys first (the top-k output)
    float scale_log2;  // softmax scale * log2(e)
    long long wait_limit;  // SM cycles a wait may take before the CTA gives up (the drains keep the default)
};
static_assert(sizeof(MlaParams) + 256 <= 32764, "launch parameters");

__device__ __forceinline__ int find_seq(const MlaParams &P, int r) {
    int lo = 0, hi = P.B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.q_off[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Index [g] is the softmax group (tile parity); hand[q][g] carries group g's row maxima of lane
// quarter q to the other group.
struct Bars {
    uint64_t q_stage, q_ready, kv_full[NSTAGE], kv_empty[NSTAGE], s_full[2], s_empty[2], p_full[2], p_empty[2],
        xfull[2], xempty[2], yfree[2], hand[4][2], qk_done, o_done;
};
static_assert(sizeof(Bars) + 8 <= 320, "barrier area");

// KV8: the latent rows are e4m3 codes (ld_kv in bytes) with one power-of-two (ue8m0) scale per 128
// values (kv_scale [rows, d_c / 128] fp32); the gathering warps load and dequantise them into the same
// bf16 stage layout (e4m3 times a power of two is exact in bf16).  Otherwise the rows are bf16.
template <bool KV8>
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(128)  // 14 warps: at most 4 per SM sub-partition x 128 regs
    mla_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
                  const void *__restrict__ kv_rows, int64_t ld_kv, const float *__restrict__ kv_scale,
                  const __nv_bfloat16 *__restrict__ kpe,
                  int64_t ld_pe, const __nv_bfloat16 *__restrict__ qt, const __nv_bfloat16 *__restrict__ qpe,
                  const int32_t *__restrict__ idx,
                  const __grid_constant__ MlaParams P, __nv_bfloat16 *__restrict__ olat, float *__restrict__ lse,
                  float *__restrict__ opart, float *__restrict__ lpart) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *KV = base;
    uint8_t *X = KV + NSTAGE * KV_STAGE;               // [group] the peer's partial scores land here, then P
    uint8_t *Y = X + 2 * X_BYTES;                      // [group] this CTA's partial scores, sent from here
    uint8_t *QR = Y + 2 * X_BYTES;                     // rope slice of q_pe (A operand)
    uint8_t *kvalid = QR + QR_BYTES;                   // [NSTAGE][BK]
    float *m_pub = (float *)(kvalid + NSTAGE * BK);    // [group][NH] row maxima handed to the other group
    float *lm = m_pub + 2 * NH;                        // [group][NH][2] final (row sum, reference) per group
    Bars *bar = (Bars *)(lm + 4 * NH);
    uint32_t *tmem_slot = (uint32_t *)(bar + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    __shared__ int never;
    volatile int *nv = (volatile int *)&never;
    int *err = &g_mla_tc_error;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_rank(), peer = rank ^ 1u;

    // Work item: heavier rows (later positions) first.
    const int w = (int)(gridDim.x / 2) - 1 - (int)(blockIdx.x / 2);
    const int r = w / P.splits, split = w % P.splits;
    const int b = find_seq(P, r);
    const int p = P.start_pos[b] + (r - P.q_off[b]);
    const int S = P.k_len[b], kbase = P.k_base[b];
    const int len = P.prefix_valid ? min(P.k, p + 1) : P.k;
    const int per = (len + P.splits - 1) / P.splits;
    const int chunk = (per + BK - 1) / BK * BK;
    const int e0 = split * chunk, e1 = min(len, e0 + chunk);
    const int n = e1 > e0 ? (e1 - e0 + BK - 1) / BK : 0;

    if (threadIdx.x == 0) {
        tc::mbar_init(&bar->q_stage, 1);
        tc::mbar_init(&bar->q_ready, 8);
        for (int i = 0; i < NSTAGE; ++i) {
            // every gathering thread arrives twice: when its copies land, and to publish the mask bytes
            tc::mbar_init(&bar->kv_full[i], 2 * NPROD * 32);
            tc::mbar_init(&bar->kv_empty[i], 1);
        }
        for (int g = 0; g < 2; ++g) {
            tc::mbar_init(&bar->s_full[g], 1);
            tc::mbar_init(&bar->s_empty[g], 4);  // the group's four warps have read the scores
            tc::mbar_init(&bar->p_full[g], 4);   // ... have written the probabilities
            tc::mbar_init(&bar->p_empty[g], 1);
            tc::mbar_init(&bar->xfull[g], 1);    // armed locally with the 16 KB the peer sends
            // phase 0: the peer's q~ staging (below) has been read; then one phase per PV product
            // of the peer on this buffer (its X[g] is free again)
            tc::mbar_init(&bar->xempty[g], 1);
            tc::mbar_init(&bar->yfree[g], 1);    // the peer has received our previous tile of group g
            for (int qq = 0; qq < 4; ++qq) tc::mbar_init(&bar->hand[qq][g], 1);
        }
        tc::mbar_init(&bar->qk_done, 1);
        tc::mbar_init(&bar->o_done, 1);
        *abort_flag = 0;
        never = 0;
        tc::fence_mbar_init();
    }
    if (warp == 2) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    tc::cluster_sync();  // both CTAs' barriers exist before any remote arrive
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // the set-up above overlapped the previous kernel; global memory only from here
    // This CTA's q~ slice (128 heads x 256 latent columns) comes in by TMA as four 128-byte-swizzled
    // boxes of 64 columns, staged in the exchange buffers, which carry no scores yet.
    if (warp == 2 && lane == 0 && n > 0) {
        tc::prefetch_tmap(&tm_q);
        tc::mbar_arrive_expect_tx(&bar->q_stage, 4 * Q_BOX);
        for (int js = 0; js < 4; ++js) tc::tma_load_3d(X + js * Q_BOX, &tm_q, &bar->q_stage, rank * 256 + js * 64, 0, r);
    }

    if ((warp == 0 || warp == 3 || warp >= 12) && n > 0) {
        // ---------------- producers: gather the selected key rows with cp.async ----------------
        // Eight lanes cover one 128-byte segment of a row, so a warp instruction
        // moves four full segments; the 128-byte swizzle of the MMA operand
        // layout is applied to the 16-byte chunk index.
        const int pw = warp == 0 ? 0 : (warp == 3 ? 1 : warp - 10), c = lane & 7, jr = pw * 4 + (lane >> 3);
        // no selection array: the dense causal pattern, entry e is key e
        const int32_t *row_idx = idx ? idx + (int64_t)r * P.k : nullptr;
        const int last = min(p, S - 1);
        const uint32_t kv_s = tc::smem_u32(KV);
        constexpr int PASSES = BK / (NPROD * 4);
        int rows[PASSES];
        auto fetch = [&](int i) {  // cache rows of this thread's keys of tile i
#pragma unroll
            for (int ps = 0; ps < PASSES; ++ps) {
                const int e = e0 + i * BK + ps * NPROD * 4 + jr;
                const int sidx = e < e1 ? (row_idx ? __ldg(row_idx + e) : e) : -1;
                rows[ps] = (sidx >= 0 && sidx <= last) ? sidx : -1;
            }
        };
        fetch(0);
        for (int i = 0; i < n; ++i) {
            const int st = i % NSTAGE;
            if (!tc::mbar_wait(&bar->kv_empty[st], ((i / NSTAGE) & 1) ^ 1, abort_flag, err, 21, P.wait_limit)) break;
            if constexpr (KV8) {
                // Codes: thread c loads bytes 8c .. 8c+7 of each 64-value slab (the same columns its 16-byte
                // chunk of the bf16 layout holds), every pass's loads issued before the first is used.
                const uint8_t *kv8 = (const uint8_t *)kv_rows;
                uint2 code[PASSES][NSLAB];
                float scl[PASSES][2];
#pragma unroll
                for (int ps = 0; ps < PASSES; ++ps) {
                    const int64_t row = kbase + (rows[ps] >= 0 ? rows[ps] : 0);
                    const uint8_t *lat = kv8 + row * ld_kv + rank * 256 + c * 8;
#pragma unroll
                    for (int js = 0; js < NSLAB; ++js) code[ps][js] = __ldg((const uint2 *)(lat + js * 64));
                    scl[ps][0] = __ldg(kv_scale + row * (DC / 128) + rank * 2);
                    scl[ps][1] = __ldg(kv_scale + row * (DC / 128) + rank * 2 + 1);
                }
#pragma unroll
                for (int ps = 0; ps < PASSES; ++ps) {
                    const int j = ps * NPROD * 4 + jr;
                    const int64_t row = kbase + (rows[ps] >= 0 ? rows[ps] : 0);
                    const uint32_t dst = kv_s + st * KV_STAGE + j * 128 + ((c ^ (j & 7)) << 4);
#pragma unroll
                    for (int js = 0; js < NSLAB; ++js) {
                        const float sc = scl[ps][js >> 1];  // slabs 0, 1: block 2 * rank; 2, 3: block 2 * rank + 1
                        const uint32_t wd[2] = {code[ps][js].x, code[ps][js].y};
                        uint32_t o[4];
#pragma unroll
                        for (int h2 = 0; h2 < 4; ++h2) {
                            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
                                (__nv_fp8x2_storage_t)((wd[h2 >> 1] >> (16 * (h2 & 1))) & 0xffffu), __NV_E4M3);
                            const float2 f = __half22float2(*(const __half2 *)&hr);
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(f.x * sc, f.y * sc);
                            o[h2] = *(const uint32_t *)&b2;
                        }
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + js * SLAB_K), "r"(o[0]),
                                     "r"(o[1]), "r"(o[2]), "r"(o[3])
                                     : "memory");
                    }
                    if (c < 4)
                        tc::cp_async16(kv_s + st * KV_STAGE + NSLAB * SLAB_K + j * 64 + ((c ^ ((j >> 1) & 3)) << 4),
                                       kpe + row * ld_pe + rank * 32 + c * 8);
                    if (c == 0) kvalid[st * BK + j] = rows[ps] >= 0 ? 1 : 0;
                }
            } else {
                const __nv_bfloat16 *kv = (const __nv_bfloat16 *)kv_rows;
#pragma unroll
                for (int ps = 0; ps < PASSES; ++ps) {
                    const int j = ps * NPROD * 4 + jr;
                    const int64_t row = kbase + (rows[ps] >= 0 ? rows[ps] : 0);
                    const __nv_bfloat16 *lat = kv + row * ld_kv + rank * 256 + c * 8;
                    const uint32_t dst = kv_s + st * KV_STAGE + j * 128 + ((c ^ (j & 7)) << 4);
#pragma unroll
                    for (int js = 0; js < NSLAB; ++js) tc::cp_async16(dst + js * SLAB_K, lat + js * 64);
                    // rope half: 64-byte rows, chunk c of row j at c ^ ((j >> 1) & 3)
                    if (c < 4)
                        tc::cp_async16(kv_s + st * KV_STAGE + NSLAB * SLAB_K + j * 64 + ((c ^ ((j >> 1) & 3)) << 4),
                                       kpe + row * ld_pe + rank * 32 + c * 8);
                    if (c == 0) kvalid[st * BK + j] = rows[ps] >= 0 ? 1 : 0;
                }
            }
            tc::cp_async_arrive_noinc(&bar->kv_full[st]);  // arrives when this thread's copies have landed
            tc::mbar_arrive(&bar->kv_full[st]);            // releases the mask bytes
            if (i + 1 < n) fetch(i + 1);
        }
        tc::cp_async_wait<0>();  // nothing may still be copying when the CTA exits
    } else if (warp == 1 && lane == 0 && n > 0) {
        // ---------------- QK^T issuer ----------------
        // QK^T(j) needs tile j gathered and its score buffer (j & 1) read by the group of tile j-2.
        // The PV products come from another thread (warp 2): an MMA issue blocks while the tensor
        // pipe is busy, so one thread for both streams would hold each up behind the other.
        bool ok = tc::mbar_wait(&bar->q_ready, 0, abort_flag, err, 24, P.wait_limit);
        const uint32_t kv0 = tc::smem_u32(KV), qr0 = tc::smem_u32(QR);
        for (int j = 0; ok && j < n; ++j) {
            const int st = j % NSTAGE;
            if (j >= 2 && !(ok = tc::mbar_wait(&bar->s_empty[j & 1], ((j >> 1) - 1) & 1, abort_flag, err, 26, P.wait_limit))) break;
            if (!(ok = tc::mbar_wait(&bar->kv_full[st], (j / NSTAGE) & 1, abort_flag, err, 25, P.wait_limit))) break;
            // the gathered rows were written by cp.async (generic proxy); the MMA reads them through
            // the async proxy
            tc::fence_proxy_async_smem();
            tc::tc_fence_after();
            const uint32_t d = tmem + COL_S + (j & 1) * BK;
#pragma unroll
            for (int js = 0; js < NSLAB; ++js)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t bd = tc::smem_desc(kv0 + st * KV_STAGE + js * SLAB_K + kk * 32, 16, 1024);
                    tc::mma_f16_ts(d, tmem + COL_Q + js * 32 + kk * 8, bd, IDESC_QK, (js | kk) != 0);
                }
            // rope half: both operands K-major with the 64-byte swizzle (8-row atoms of 512 bytes)
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const uint64_t ad = tc::smem_desc(qr0 + kk * 32, 16, 512, tc::kSwizzle64B);
                const uint64_t bd = tc::smem_desc(kv0 + st * KV_STAGE + NSLAB * SLAB_K + kk * 32, 16, 512,
                                                  tc::kSwizzle64B);
                tc::mma_f16(d, ad, bd, IDESC_QK, 1);
            }
            tc::mma_commit(&bar->s_full[j & 1]);
        }
        // No MMA of this thread may still be running when the tensor memory is released (after an
        // abort the loop can stop with score tiles in flight).
        tc::mma_commit(&bar->qk_done);
        tc::mbar_wait(&bar->qk_done, 0, nv, err, 39);
    } else if (warp == 2 && lane == 0 && n > 0) {
        // ---------------- PV issuer ----------------
        // PV(j) once P(j) is written; its completion frees the key stage, this CTA's X buffer (the
        // peer may send the next tile of that group) and, for a rescale, the context.
        const uint32_t kv0 = tc::smem_u32(KV), x0 = tc::smem_u32(X);
        const uint16_t peer_mask = (uint16_t)(1u << peer);
        for (int j = 0; j < n; ++j) {
            if (!tc::mbar_wait(&bar->p_full[j & 1], (j >> 1) & 1, abort_flag, err, 27, P.wait_limit)) break;
            tc::tc_fence_after();
            const int st = j % NSTAGE;
            const uint32_t pa = x0 + (j & 1) * X_BYTES;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                // P: K-major rows of 64 keys (128-byte swizzle); V: MN-major view of latent slabs
                // 0..3 of the tile (LBO = slab stride, SBO = 8 keys).
                const uint64_t ad = tc::smem_desc(pa + kk * 32, 16, 1024);
                const uint64_t bd = tc::smem_desc(kv0 + st * KV_STAGE + kk * 16 * 128, SLAB_K, 1024);
                tc::mma_f16(tmem + COL_O, ad, bd, IDESC_PV, (j | kk) != 0);
            }
            tc::mma_commit(&bar->kv_empty[st]);
            tc::mma_commit(&bar->p_empty[j & 1]);
            tc::mma_commit_multicast(&bar->xempty[j & 1], peer_mask);  // the peer may refill our X
        }
        tc::mma_commit(&bar->o_done);
        tc::mbar_wait(&bar->o_done, 0, nv, err, 28);
        // The q~ staging load this thread issued must have landed before the CTA exits (after an
        // abort nobody else may have waited for it).
        tc::mbar_wait(&bar->q_stage, 0, nv, err, 29);
    } else if (warp >= 4 && warp < 12) {
        // ---------------- softmax: group g takes tiles g, g+2, ...; one thread per head row ----------------
        const int q = warp & 3, g = (warp - 4) >> 2, h = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const unsigned FULL = 0xffffffffu;
        float m_g = -INFINITY, l_g = 0.0f;  // this group's part of the row sum, relative to 2^m_g
        bool done_ok = true;
        if (n > 0) {
            // This CTA's slice of the head's q~ row -> tensor memory (A operand of QK^T): latent
            // columns as 4 slabs of 32 packed columns (from the TMA staging; chunk e of row h sits at
            // e ^ (h & 7)); group g moves slabs 2g and 2g+1.  Group 1 also puts the rope slice of
            // q_pe (read in place) into shared memory, K-major with the 64-byte swizzle.
            uint4 rq[4];
            if (g) {
                const uint4 *rsrc = (const uint4 *)(qpe + ((int64_t)r * NH + h) * DR + rank * 32);
#pragma unroll
                for (int e = 0; e < 4; ++e) rq[e] = __ldg(rsrc + e);
            }
            if (!tc::mbar_wait(&bar->q_stage, 0, abort_flag, err, 23, P.wait_limit)) done_ok = false;
            if (done_ok) {
                for (int js = g * 2; js < g * 2 + 2; ++js) {
                    const uint8_t *srow = X + js * Q_BOX + h * 128;
                    uint32_t qv[32];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const uint4 t4 = *(const uint4 *)(srow + ((e ^ (h & 7)) << 4));
                        qv[4 * e] = t4.x;
                        qv[4 * e + 1] = t4.y;
                        qv[4 * e + 2] = t4.z;
                        qv[4 * e + 3] = t4.w;
                    }
                    tc::tmem_st32(tmem + lane_off + COL_Q + js * 32, qv);
                }
                tc::tmem_st_wait();
            }
            if (g) {
#pragma unroll
                for (int e = 0; e < 4; ++e) *(uint4 *)(QR + h * 64 + ((e ^ ((h >> 1) & 3)) << 4)) = rq[e];
                tc::fence_proxy_async_smem();  // read by the rope MMAs (async proxy)
            }
            tc::tc_fence_before();
            // Every softmax warp has read its part of the staging before any of them writes a score
            // tile into Y, and then the peer learns that this CTA's X buffers may receive scores.
            asm volatile("bar.sync %0, %1;" ::"r"(SOFT_BAR), "r"(8 * 32) : "memory");
            if (lane == 0) tc::mbar_arrive(&bar->q_ready);
            if (threadIdx.x == 4 * 32) {
                tc::mbar_arrive_remote(tc::map_peer(tc::smem_u32(&bar->xempty[0]), peer));
                tc::mbar_arrive_remote(tc::map_peer(tc::smem_u32(&bar->xempty[1]), peer));
            }
        }
        const float sl2 = P.scale_log2;
        const uint32_t hsw = (uint32_t)(h & 7);
        uint8_t *Xg = X + g * X_BYTES, *Yg = Y + g * X_BYTES;
        const int roff = h * 128, wblk = q * 32 * 128;  // this row; this warp's 32 rows (4 KB)
        int sent = 0;  // tiles this group has copied into the peer's X[g]
        for (int t = g, k = 0; done_ok && t < n; t += 2, ++k) {
            const uint32_t ph = (uint32_t)k & 1u;
            // --- this CTA's partial scores of tile t -> fp16 of the log2-scaled values ---
            if (!__all_sync(FULL, tc::mbar_wait(&bar->s_full[g], ph, abort_flag, err, 31, P.wait_limit))) { done_ok = false; break; }
            tc::tc_fence_after();
            uint32_t cur[32];
            {
                float sa[32], sb[32];
                tc::tmem_ld32(tmem + lane_off + COL_S + g * BK, sa);
                tc::tmem_ld32(tmem + lane_off + COL_S + g * BK + 32, sb);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    cur[j] = tc::f16x2_satfinite(sa[2 * j] * sl2, sa[2 * j + 1] * sl2);
                    cur[16 + j] = tc::f16x2_satfinite(sb[2 * j] * sl2, sb[2 * j + 1] * sl2);
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bar->s_empty[g]);  // the MMA may compute tile t+2 into this buffer
            // --- ship: Y[g] -> the peer's X[g]; the peer's half of this tile arrives in ours ---
            if (q == 0 && lane == 0) tc::mbar_arrive_expect_tx(&bar->xfull[g], X_BYTES);
            // Y[g] may be rewritten once the peer has received the group's previous tile from it (the
            // copy has then finished reading it).
            if (k > 0 && !__all_sync(FULL, tc::mbar_wait_cluster(&bar->yfree[g], (k - 1) & 1, abort_flag, err, 38, P.wait_limit))) {
                done_ok = false;
                break;
            }
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *(uint4 *)(Yg + roff + ((c ^ hsw) << 4)) = make_uint4(cur[4 * c], cur[4 * c + 1], cur[4 * c + 2], cur[4 * c + 3]);
            tc::fence_proxy_async_smem();  // the stores are read by the bulk copy (async proxy)
            // The peer's X[g] is free once the peer has read its q~ staging (first tile of the group)
            // or its PV product of tile t-2 is done.
            bool ok = true;
            if (lane == 0) ok = tc::mbar_wait_cluster(&bar->xempty[g], ph, abort_flag, err, 32, P.wait_limit);
            __syncwarp();
            if (!__shfl_sync(FULL, ok, 0)) { done_ok = false; break; }
            if (lane == 0)
                tc::bulk_copy_to_peer(tc::map_peer(tc::smem_u32(Xg) + wblk, peer), Yg + wblk, 32 * 128,
                                      tc::map_peer(tc::smem_u32(&bar->xfull[g]), peer));
            ++sent;
            // --- own half in fp32 and the mask (entries that are padding, future or outside the sequence),
            // while the peer's half is in flight ---
            float v[64];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                v[2 * j] = tc::f16_to_f32((uint16_t)(cur[j] & 0xffffu));
                v[2 * j + 1] = tc::f16_to_f32((uint16_t)(cur[j] >> 16));
            }
            const int st = t % NSTAGE;
            if (!__all_sync(FULL, tc::mbar_wait(&bar->kv_full[st], (t / NSTAGE) & 1, abort_flag, err, 34, P.wait_limit))) { done_ok = false; break; }
            {
                const uint4 *kv4 = (const uint4 *)(kvalid + st * BK);
                const uint4 m0 = kv4[0], m1 = kv4[1], m2 = kv4[2], m3 = kv4[3];
                const uint32_t all = m0.x & m0.y & m0.z & m0.w & m1.x & m1.y & m1.z & m1.w & m2.x & m2.y & m2.z &
                                     m2.w & m3.x & m3.y & m3.z & m3.w;
                if (all != 0x01010101u) {
                    const uint32_t *kvw = (const uint32_t *)(kvalid + st * BK);
#pragma unroll
                    for (int wd = 0; wd < 16; ++wd) {
                        const uint32_t bits = kvw[wd];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            if (!((bits >> (8 * u)) & 0xffu)) v[4 * wd + u] = -INFINITY;
                    }
                }
            }
            // --- + peer half, one rounding in fp32 (addition commutes: both CTAs get the same sum; a
            // masked entry stays -inf) ---
            if (!__all_sync(FULL, tc::mbar_wait_cluster(&bar->xfull[g], ph, abort_flag, err, 33, P.wait_limit))) { done_ok = false; break; }
            // all four copies of the peer's half have landed: its Y[g] may be rewritten
            if (q == 0 && lane == 0) tc::mbar_arrive_remote(tc::map_peer(tc::smem_u32(&bar->yfree[g]), peer));
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 x = *(const uint4 *)(Xg + roff + ((c ^ hsw) << 4));
                const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    v[8 * c + 2 * e] = tc::add_f16_f32((uint16_t)(xs[e] & 0xffffu), v[8 * c + 2 * e]);
                    v[8 * c + 2 * e + 1] = tc::add_f16_f32((uint16_t)(xs[e] >> 16), v[8 * c + 2 * e + 1]);
                }
            }
            // row maximum as a tree (depth 4)
            float mt;
            {
                float a[22], b8[8];
#pragma unroll
                for (int i = 0; i < 21; ++i) a[i] = tc::max3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
                a[21] = v[63];
#pragma unroll
                for (int i = 0; i < 7; ++i) b8[i] = tc::max3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
                b8[7] = a[21];
                mt = tc::max3(tc::max3(b8[0], b8[1], b8[2]), tc::max3(b8[3], b8[4], b8[5]), fmaxf(b8[6], b8[7]));
            }
            // --- running maximum: the one used for tile t-1 comes from the other group ---
            float m_prev = -INFINITY;
            if (t > 0) {
                if (!__all_sync(FULL, tc::mbar_wait(&bar->hand[q][1 - g], ((t - 1) >> 1) & 1, abort_flag, err, 37, P.wait_limit))) {
                    done_ok = false;
                    break;
                }
                m_prev = m_pub[(1 - g) * NH + h];
            }
            float m_now = m_prev;  // the scores are already in log2 units
            bool rescale = false;
            if (mt != -INFINITY) {
                if (m_prev == -INFINITY) {
                    m_now = mt;
                } else if (mt > m_prev + RESCALE_LOG2) {
                    m_now = mt;
                    rescale = true;
                }
            }
            if (t + 1 < n) {
                m_pub[g * NH + h] = m_now;
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bar->hand[q][g]);
            }
            if (m_now != m_g) {
                if (m_g != -INFINITY) l_g *= tc::ex2_approx(m_g - m_now);
                m_g = m_now;
            }
            const float neg_m = m_now == -INFINITY ? 0.0f : -m_now;
            uint32_t pk[32];
            float psum0 = 0.0f, psum1 = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float p0 = tc::ex2_approx(v[2 * j] + neg_m);
                const float p1 = tc::ex2_approx(v[2 * j + 1] + neg_m);
                const __nv_bfloat162 t2 = __floats2bfloat162_rn(p0, p1);
                pk[j] = *(const uint32_t *)&t2;
                // the row sum takes the rounded probabilities that the PV product uses
                psum0 = tc::add_bf16_f32((uint16_t)(pk[j] & 0xffffu), psum0);
                psum1 = tc::add_bf16_f32((uint16_t)(pk[j] >> 16), psum1);
            }
            l_g += psum0 + psum1;
            // --- O is rescaled after PV(t-1) and before PV(t); tcgen05.ld/st are warp-wide, so the
            // whole warp takes part when any of its rows moves (the others keep alpha = 1) ---
            if (__any_sync(FULL, rescale)) {
                const float alpha = rescale ? tc::ex2_approx(m_prev - m_now) : 1.0f;
                if (!__all_sync(FULL, tc::mbar_wait(&bar->p_empty[(t - 1) & 1], ((t - 1) >> 1) & 1, abort_flag, err, 35, P.wait_limit))) {
                    done_ok = false;
                    break;
                }
                tc::tc_fence_after();
#pragma unroll 1
                for (int cc = 0; cc < 8; ++cc) {
                    float o[32];
                    uint32_t ob[32];
                    tc::tmem_ld32(tmem + lane_off + COL_O + cc * 32, o);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) ob[j] = __float_as_uint(o[j] * alpha);
                    tc::tmem_st32(tmem + lane_off + COL_O + cc * 32, ob);
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
            }
            // --- P(t) overwrites the received half (each row is read and written by its own thread) ---
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *(uint4 *)(Xg + roff + ((c ^ hsw) << 4)) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            tc::fence_proxy_async_smem();  // read by the PV product (async proxy)
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bar->p_full[g]);
        }
        // The peer acknowledges every tile it has received (yfree); the acknowledgement of the last
        // tile this group sent says that none of its copies is still landing in the peer's shared
        // memory.  (A peer that aborted sends none: the wait then gives up, and the quiet period
        // below covers the copies.)
        if (sent > 0)
            (void)__all_sync(FULL, tc::mbar_wait_cluster(&bar->yfree[g], (sent - 1) & 1, abort_flag, err, 40,
                                                         P.wait_limit));
        // ---------------- epilogue: normalise and store this thread's 128 columns ----------------
        // The row sum of each group is relative to the last maximum that group used; the context is
        // relative to the last maximum of all (the running maximum never decreases).
        lm[(g * NH + h) * 2] = l_g;
        lm[(g * NH + h) * 2 + 1] = m_g;
        asm volatile("bar.sync %0, %1;" ::"r"(SOFT_BAR), "r"(8 * 32) : "memory");
        const float la = lm[h * 2], ma = lm[h * 2 + 1], lb = lm[(NH + h) * 2], mb = lm[(NH + h) * 2 + 1];
        const float m_f = fmaxf(ma, mb);
        const float lrow = (ma == -INFINITY ? 0.0f : la * tc::ex2_approx(ma - m_f)) +
                           (mb == -INFINITY ? 0.0f : lb * tc::ex2_approx(mb - m_f));
        const int64_t rh = (int64_t)r * NH + h;
        const bool have = __all_sync(FULL, n > 0 && done_ok && tc::mbar_wait(&bar->o_done, 0, abort_flag, err, 36, P.wait_limit));
        const float inv = (have && lrow > 0.0f) ? 1.0f / lrow : 0.0f;
        const float row_lse = (have && lrow > 0.0f) ? (m_f + log2f(lrow)) * LN2 : -INFINITY;
        if (have) tc::tc_fence_after();
        if (P.splits == 1) {
            // bf16 context -> the key stages (free: every PV product is done), as four 128-byte-
            // swizzled boxes of 64 columns, then out by TMA tensor stores.
#pragma unroll 1
            for (int cc = g * 4; cc < g * 4 + 4; ++cc) {
                float o[32];
                if (have) {
                    tc::tmem_ld32(tmem + lane_off + COL_O + cc * 32, o);
                    tc::tmem_ld_wait();
                }
                uint32_t pw[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const __nv_bfloat162 t2 = have ? __floats2bfloat162_rn(o[2 * e] * inv, o[2 * e + 1] * inv)
                                                   : __floats2bfloat162_rn(0.0f, 0.0f);
                    pw[e] = *(const uint32_t *)&t2;
                }
                uint8_t *srow = KV + (cc >> 1) * Q_BOX + h * 128;
                const int j0 = (cc & 1) * 4;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    *(uint4 *)(srow + (((j0 + e) ^ (h & 7)) << 4)) =
                        make_uint4(pw[4 * e], pw[4 * e + 1], pw[4 * e + 2], pw[4 * e + 3]);
            }
            tc::fence_proxy_async_smem();  // the staging is read by the TMA stores (async proxy)
            asm volatile("bar.sync %0, %1;" ::"r"(SOFT_BAR), "r"(8 * 32) : "memory");
            if (threadIdx.x == 4 * 32) {
                for (int cb = 0; cb < 4; ++cb) tc::tma_store_3d(&tm_o, KV + cb * Q_BOX, rank * 256 + cb * 64, 0, r);
                tc::bulk_commit_group();
                tc::bulk_wait_read_all();  // the staging must outlive the stores' reads (the CTA exits next)
            }
            if (rank == 0 && g == 0 && lse) lse[rh] = row_lse;
        } else {
            const int64_t part = ((int64_t)r * P.splits + split) * NH + h;
            float *dst = opart + part * DC + rank * 256;
#pragma unroll 1
            for (int cc = g * 4; cc < g * 4 + 4; ++cc) {
                float o[32];
                if (have) {
                    tc::tmem_ld32(tmem + lane_off + COL_O + cc * 32, o);
                    tc::tmem_ld_wait();
                }
                float4 *d4 = (float4 *)(dst + cc * 32);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    d4[e] = have ? make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv, o[4 * e + 3] * inv)
                                 : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
            if (rank == 0 && g == 0) lpart[part] = row_lse;
        }
    }
    __syncthreads();
    if (*abort_flag) {
        // After an abort, a partial-score copy issued into the peer before its waits gave up may still
        // be in flight, unacknowledged; such a copy lands within microseconds.  The CTA arrives at the
        // cluster barrier (which lets the peer exit) only after a quiet period far longer than that.
        const long long t0 = clock64();
        while (clock64() - t0 < kAbortQuietCycles) {
        }
    }
    tc::cluster_sync();  // no DSMEM traffic may target a CTA that has exited
    if (warp == 2) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// Merge the normalised partial contexts of the splits of one row:
// lse = log sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s.  One warp per (row, head).
__global__ void __launch_bounds__(256) mla_combine_kernel(const float *__restrict__ opart,
                                                          const float *__restrict__ lpart, int M, int splits,
                                                          __nv_bfloat16 *__restrict__ olat, float *__restrict__ lse) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t rh = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (rh >= (int64_t)M * NH) return;
    const int64_t r = rh / NH, h = rh % NH;
    float mx = -INFINITY;
    for (int s = 0; s < splits; ++s) mx = fmaxf(mx, lpart[(r * splits + s) * NH + h]);
    float wsum = 0.0f;
    for (int s = 0; s < splits; ++s) {
        const float ls = lpart[(r * splits + s) * NH + h];
        wsum += ls == -INFINITY ? 0.0f : expf(ls - mx);
    }
    const float tot = wsum > 0.0f ? mx + logf(wsum) : -INFINITY;
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
    for (int s = 0; s < splits; ++s) {
        const float ls = lpart[(r * splits + s) * NH + h];
        if (ls == -INFINITY) continue;
        const float wgt = expf(ls - tot);
        const float4 *src = (const float4 *)(opart + ((r * splits + s) * NH + h) * DC) + lane * 4;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 x = src[j];
            acc[4 * j] += wgt * x.x;
            acc[4 * j + 1] += wgt * x.y;
            acc[4 * j + 2] += wgt * x.z;
            acc[4 * j + 3] += wgt * x.w;
        }
    }
    uint32_t pw[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const __nv_bfloat162 t2 = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
        pw[e] = *(const uint32_t *)&t2;
    }
    uint4 *dst = (uint4 *)(olat + rh * DC + lane * 16);
    dst[0] = make_uint4(pw[0], pw[1], pw[2], pw[3]);
    dst[1] = make_uint4(pw[4], pw[5], pw[6], pw[7]);
    if (lse && lane == 0) lse[rh] = tot;
}

}  // namespace

bool mla_tc_supported(int dtype, int H, int d_n, int d_r, int d_c, int d_v) {
    return dtype == DSA_BF16 && H == NH && d_n == 128 && d_r == 64 && d_c == DC && d_v == 128;
}

// Clusters per row: enough rows fill the GPU on their own; a few long rows
// (decode) are split so that about two clusters per SM pair run.
int mla_tc_splits(int M) {
    // One CTA per SM (shared memory) and two per cluster: 76 clusters run at once.  Splitting a
    // row's keys pays only while the clusters still fit one wave; beyond that it adds waves of
    // proportionally shorter work plus a pipeline fill per wave.
    const int wave = 152 / 2;
    return M >= wave ? 1 : std::min(8, std::max(1, wave / M));
}

size_t mla_tc_partial_bytes(int M) {
    const int s = mla_tc_splits(M);
    if (s == 1) return 0;
    return (size_t)M * s * NH * DC * sizeof(float) + 256 + (size_t)M * s * NH * sizeof(float);
}

cudaError_t launch_mla_tc(const void *qt, const void *qpe, const void *kv, int64_t ld_kv, const void *kpe, int64_t ld_pe,
                          const int32_t *idx, int k, const SeqTab &st, int64_t total_k, int M, float scale,
                          bool prefix_valid, void *olat, float *lse, void *part_ws, cudaStream_t s,
                          const float *kv_scale) {
    if (M == 0) return cudaSuccess;
    static thread_local MlaParams P;
    P.B = st.B;
    for (int i = 0; i < st.B; ++i) {
        P.q_off[i] = st.q_off[i];
        P.k_base[i] = st.k_base[i];
        P.k_len[i] = st.k_len[i];
        P.start_pos[i] = st.start_pos[i];
    }
    P.q_off[st.B] = st.q_off[st.B];
    P.total_q = M;
    P.k = k;
    P.splits = mla_tc_splits(M);
    P.prefix_valid = prefix_valid ? 1 : 0;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.wait_limit = wait_limit_cycles();
    float *opart = nullptr, *lpart = nullptr;
    if (P.splits > 1) {
        opart = (float *)part_ws;
        lpart = (float *)((char *)part_ws + (((size_t)M * P.splits * NH * DC * sizeof(float) + 255) / 256) * 256);
    }
    // q~ rows [M, 128, 512] (loaded) and the latent context [M, 128, 512] (stored): boxes of
    // 64 columns x 128 heads x 1 row, 128-byte swizzle.
    CUtensorMap tq, to;
    {
        const uint64_t dims[3] = {(uint64_t)DC, (uint64_t)NH, (uint64_t)M};
        const uint64_t strides[2] = {(uint64_t)DC * 2, (uint64_t)NH * DC * 2};
        const uint32_t box[3] = {64, (uint32_t)NH, 1};
        if (!make_tmap(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, qt, dims, strides, box)) return cudaErrorInvalidValue;
        if (!make_tmap(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, olat, dims, strides, box)) return cudaErrorInvalidValue;
    }
    const unsigned grid = (unsigned)M * P.splits * 2;
    auto kern = kv_scale ? mla_tc_kernel<true> : mla_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(grid), dim3(NUM_THREADS), SMEM, s, tq, to, kv, ld_kv, kv_scale,
                   (const __nv_bfloat16 *)kpe, ld_pe, (const __nv_bfloat16 *)qt, (const __nv_bfloat16 *)qpe, idx, P,
                   (__nv_bfloat16 *)olat, lse, opart, lpart);
    if (e != cudaSuccess) return e;
    note_launch(DSA_KERNEL_MLA_TC);
    if (P.splits == 1) return cudaSuccess;
    const unsigned cgrid = (unsigned)(((int64_t)M * NH + 7) / 8);
    e = launch_pdl(mla_combine_kernel, dim3(cgrid), dim3(256), 0, s, (const float *)opart, (const float *)lpart, M,
                   P.splits, (__nv_bfloat16 *)olat, lse);
    if (e != cudaSuccess) return e;
    note_launch(DSA_KERNEL_COMBINE);
    return cudaGetLastError();
}

int mla_tc_read_error(int *site) {
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_mla_tc_error, sizeof(int));
    if (e != cudaSuccess) return fail_cuda(e);
    if (v) {
        e = cudaMemcpyToSymbol(g_mla_tc_error, &zero, sizeof(int));
        if (e != cudaSuccess) return fail_cuda(e);
        if (site) *site = v;
        return DSA_ERR_TIMEOUT;
    }
    return DSA_OK;
}

}  // namespace dsa
