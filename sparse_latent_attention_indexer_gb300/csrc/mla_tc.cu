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
// row is handled by a cluster of two CTAs on two SMs:
//   * CTA 0 holds latent columns 0..255, CTA 1 latent 256..511 and the rope
//     part -- of q~ (resident, loaded once by TMA) and of each gathered key
//     tile (64 keys, rows gathered with cp.async by two producer warps).
//   * Each CTA computes a partial score tile S_c = Q_c K_c^T (M = 128 heads,
//     N = 64 keys) over its columns; the softmax warps swap partial tiles
//     through distributed shared memory and both add them (in the same
//     order), so both CTAs hold the identical full score tile.
//   * Both run the same online softmax (identical decisions), write
//     P (bf16) to shared memory, and accumulate O_c += P V_c for their own 256
//     latent columns in tensor memory (N = 256, V read MN-major straight from
//     the gathered tile).
// The running maximum is only moved (and O rescaled in tensor memory) when
// a tile's maximum exceeds it by more than 2^8, which after the first tiles
// almost never happens.  Key tiles are double-buffered in shared memory and
// score tiles in tensor memory, so the QK^T of tile i+1 overlaps the
// softmax of tile i.  Waits are bounded; a timeout records its site in the
// device error word and both CTAs drain and exit.
//
// Long rows can be split across several clusters (decode: few rows, many
// keys); each split writes a normalised partial context and its lse, and a
// small combine kernel merges them.
#include "tc_common.cuh"

namespace dsa {

__device__ int g_mla_tc_error = 0;

namespace {

constexpr int NH = 128;                      // heads (MMA M)
constexpr int DC = 512;                      // latent width
constexpr int QW = 576;                      // q~ row: [q~ (512) | q_pe (64)]
constexpr int BK = 64;                       // keys per tile (MMA N of QK^T, K of PV)
constexpr int NSLAB_MAX = 5;                 // 64-column slabs per CTA (CTA 1: 4 latent + rope)
constexpr int SLAB_K = BK * 128;             // 8 KB: 64 keys x 64 columns, 128-byte swizzle
constexpr int KV_STAGE = NSLAB_MAX * SLAB_K; // 40 KB
constexpr int NSTAGE = 3;
constexpr int X_BYTES = NH * BK * 4;         // 32 KB: partial scores (received X, sent Y)
constexpr int SMEM = 1024 + NSTAGE * KV_STAGE + 2 * X_BYTES + NSTAGE * BK + 3 * 2 * NH * 4 + 256;
constexpr int NUM_THREADS = 448;             // warps 0, 3, 12, 13: gather; 1: MMA; 2: TMEM; 4-11: softmax
constexpr int NPROD = 4;                     // gathering warps
// Tensor-memory columns (512 per CTA): scores, probabilities (bf16 pairs),
// the resident q~ slice (bf16 pairs, A operand of QK^T) and the context.
constexpr uint32_t COL_S = 0, COL_P = 64, COL_Q = 96, COL_O = 256;
constexpr uint32_t IDESC_QK = tc::instr_desc(tc::kFmtBF16, tc::kFmtBF16, NH, BK, 0, 0);
constexpr uint32_t IDESC_PV = tc::instr_desc(tc::kFmtBF16, tc::kFmtBF16, NH, 256, 0, 1);
constexpr float RESCALE_LOG2 = 8.0f;
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
};

__device__ __forceinline__ int find_seq(const MlaParams &P, int r) {
    int lo = 0, hi = P.B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.q_off[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

struct Bars {
    uint64_t q_ready, kv_full[NSTAGE], kv_empty[NSTAGE], s_full, s_empty, p_full, p_empty, xfull, xempty, o_done;
};

__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(128)  // 14 warps: at most 4 per SM sub-partition x 128 regs
    mla_tc_kernel(const __nv_bfloat16 *__restrict__ kv, int64_t ld_kv, const __nv_bfloat16 *__restrict__ kpe,
                  int64_t ld_pe, const __nv_bfloat16 *__restrict__ qt, const int32_t *__restrict__ idx,
                  const __grid_constant__ MlaParams P, __nv_bfloat16 *__restrict__ olat, float *__restrict__ lse,
                  float *__restrict__ opart, float *__restrict__ lpart) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *KV = base;
    float *X = (float *)(KV + NSTAGE * KV_STAGE);     // the peer's partial scores land here
    float *Y = X + NH * BK;                            // this CTA's partial scores, staged for the peer
    uint8_t *kvalid = (uint8_t *)(Y + NH * BK);        // [NSTAGE][BK]
    float *pmax = (float *)(kvalid + NSTAGE * BK);     // [2 tiles][2 halves][NH] row-maximum halves
    float *lsum = pmax + 4 * NH;                       // [2 halves][NH] row-sum halves
    Bars *bar = (Bars *)(lsum + 2 * NH);
    uint32_t *tmem_slot = (uint32_t *)(bar + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    __shared__ int never;
    volatile int *nv = (volatile int *)&never;
    int *err = &g_mla_tc_error;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_rank(), peer = rank ^ 1u;
    const int nslab = rank ? 5 : 4, gslab0 = rank ? 4 : 0;

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
        tc::mbar_init(&bar->q_ready, 8);
        for (int i = 0; i < NSTAGE; ++i) {
            // every gathering thread arrives twice: when its copies land, and to publish the mask bytes
            tc::mbar_init(&bar->kv_full[i], 2 * NPROD * 32);
            tc::mbar_init(&bar->kv_empty[i], 1);
        }
        tc::mbar_init(&bar->s_full, 1);
        tc::mbar_init(&bar->s_empty, 8);
        tc::mbar_init(&bar->p_full, 8);
        tc::mbar_init(&bar->p_empty, 1);
        tc::mbar_init(&bar->xfull, 1);   // armed locally with the 32 KB the peer sends
        tc::mbar_init(&bar->xempty, 8);  // one arrival per peer softmax warp
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

    if ((warp == 0 || warp == 3 || warp >= 12) && n > 0) {
        // ---------------- producers: gather the selected key rows with cp.async ----------------
        // Eight lanes cover one 128-byte segment of a row, so a warp instruction
        // moves four full segments; the 128-byte swizzle of the MMA operand
        // layout is applied to the 16-byte chunk index.
        const int pw = warp == 0 ? 0 : (warp == 3 ? 1 : warp - 10), c = lane & 7, jr = pw * 4 + (lane >> 3);
        const int32_t *row_idx = idx + (int64_t)r * P.k;
        const int last = min(p, S - 1);
        const uint32_t kv_s = tc::smem_u32(KV);
        constexpr int PASSES = BK / (NPROD * 4);
        int rows[PASSES];
        auto fetch = [&](int i) {  // cache rows of this thread's keys of tile i
#pragma unroll
            for (int ps = 0; ps < PASSES; ++ps) {
                const int e = e0 + i * BK + ps * NPROD * 4 + jr;
                const int sidx = e < e1 ? __ldg(row_idx + e) : -1;
                rows[ps] = (sidx >= 0 && sidx <= last) ? sidx : -1;
            }
        };
        fetch(0);
        for (int i = 0; i < n; ++i) {
            const int st = i % NSTAGE;
            if (!tc::mbar_wait(&bar->kv_empty[st], ((i / NSTAGE) & 1) ^ 1, abort_flag, err, 21)) break;
#pragma unroll
            for (int ps = 0; ps < PASSES; ++ps) {
                const int j = ps * NPROD * 4 + jr;
                const int64_t row = kbase + (rows[ps] >= 0 ? rows[ps] : 0);
                const __nv_bfloat16 *lat = kv + row * ld_kv + c * 8;
                const uint32_t dst = kv_s + st * KV_STAGE + j * 128 + ((c ^ (j & 7)) << 4);
                for (int js = 0; js < nslab; ++js) {
                    const int g = gslab0 + js;
                    const __nv_bfloat16 *src = g < 8 ? lat + g * 64 : kpe + row * ld_pe + c * 8;
                    tc::cp_async16(dst + js * SLAB_K, src);
                }
                if (c == 0) kvalid[st * BK + j] = rows[ps] >= 0 ? 1 : 0;
            }
            tc::cp_async_arrive_noinc(&bar->kv_full[st]);  // arrives when this thread's copies have landed
            tc::mbar_arrive(&bar->kv_full[st]);            // releases the mask bytes
            if (i + 1 < n) fetch(i + 1);
        }
        tc::cp_async_wait<0>();  // nothing may still be copying when the CTA exits
    } else if (warp == 1 && lane == 0 && n > 0) {
        // ---------------- MMA issuer ----------------
        bool ok = tc::mbar_wait(&bar->q_ready, 0, abort_flag, err, 24);
        const uint32_t kv0 = tc::smem_u32(KV);
        auto issue_qk = [&](int j) -> bool {
            const int st = j % NSTAGE;
            if (!tc::mbar_wait(&bar->kv_full[st], (j / NSTAGE) & 1, abort_flag, err, 25)) return false;
            // the gathered rows were written by cp.async (generic proxy); the MMA reads them
            // through the async proxy
            tc::fence_proxy_async_smem();
            if (!tc::mbar_wait(&bar->s_empty, (j & 1) ^ 1, abort_flag, err, 26)) return false;
            tc::tc_fence_after();
            for (int js = 0; js < nslab; ++js)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t bd = tc::smem_desc(kv0 + st * KV_STAGE + js * SLAB_K + kk * 32, 16, 1024);
                    tc::mma_f16_ts(tmem + COL_S, tmem + COL_Q + js * 32 + kk * 8, bd, IDESC_QK, (js | kk) != 0);
                }
            tc::mma_commit(&bar->s_full);
            return true;
        };
        if (ok) ok = issue_qk(0);
        for (int i = 0; ok && i < n; ++i) {
            if (i + 1 < n && !(ok = issue_qk(i + 1))) break;
            if (!(ok = tc::mbar_wait(&bar->p_full, i & 1, abort_flag, err, 27))) break;
            tc::tc_fence_after();
            const int st = i % NSTAGE;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                // V: MN-major view of latent slabs 0..3 of the tile (LBO = slab stride, SBO = 8 keys).
                const uint64_t bd = tc::smem_desc(kv0 + st * KV_STAGE + kk * 16 * 128, SLAB_K, 1024);
                tc::mma_f16_ts(tmem + COL_O, tmem + COL_P + kk * 8, bd, IDESC_PV, (i | kk) != 0);
            }
            tc::mma_commit(&bar->kv_empty[st]);
            tc::mma_commit(&bar->p_empty);
        }
        tc::mma_commit(&bar->o_done);
        tc::mbar_wait(&bar->o_done, 0, nv, err, 28);
    } else if (warp >= 4 && warp < 12) {
        // ---------------- softmax: two threads per head (TMEM lane), 32 score columns each ----------------
        const int q = warp & 3, hf = (warp - 4) >> 2, h = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const uint32_t peer_xfull = tc::map_peer(tc::smem_u32(&bar->xfull), peer);
        const uint32_t peer_xempty = tc::map_peer(tc::smem_u32(&bar->xempty), peer);
        float m_used = -INFINITY, l = 0.0f;  // l: this thread's half of the row sum
        bool done_ok = true;
        if (n > 0) {
            // This CTA's slice of the head's q~ row -> tensor memory (A operand of QK^T);
            // the two threads of a row split the 64-column slabs.
            const uint4 *src = (const uint4 *)(qt + ((int64_t)r * NH + h) * QW + gslab0 * 64);
            for (int js = hf * 2; js < (hf ? nslab : 2); ++js) {
                uint32_t qv[32];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint4 t4 = __ldg(src + js * 8 + e);
                    qv[4 * e] = t4.x;
                    qv[4 * e + 1] = t4.y;
                    qv[4 * e + 2] = t4.z;
                    qv[4 * e + 3] = t4.w;
                }
                tc::tmem_st32(tmem + lane_off + COL_Q + js * 32, qv);
            }
            tc::tmem_st_wait();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bar->q_ready);
        }
        const float sl2 = P.scale_log2;
        const uint32_t row_sw = (uint32_t)(h & 7);
        // X / Y are [half][128 rows][32 floats]: a warp's 32 rows of one half are a contiguous 4 KB block.
        uint8_t *xrow = (uint8_t *)X + (hf * NH + h) * 128, *yrow = (uint8_t *)Y + (hf * NH + h) * 128;
        const int wblk = (hf * NH + q * 32) * 128;
        const uint32_t peer_x_warp = tc::map_peer(tc::smem_u32(X) + wblk, peer);
        const uint32_t named = 1 + q;  // the two warps of a lane quarter
        for (int i = 0; i < n; ++i) {
            const int st = i % NSTAGE;
            if (!tc::mbar_wait(&bar->s_full, i & 1, abort_flag, err, 31)) { done_ok = false; break; }
            tc::tc_fence_after();
            float v[32];
            tc::tmem_ld32(tmem + lane_off + COL_S + hf * 32, v);
            tc::tmem_ld_wait();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bar->s_empty);  // the MMA may now compute the next tile's scores
            // --- swap partial scores with the peer: stage locally, one bulk copy per warp ---
            if (threadIdx.x == 4 * 32) tc::mbar_arrive_expect_tx(&bar->xfull, X_BYTES);
            if (i > 0 && lane == 0) tc::bulk_wait_read();  // the previous copy has read Y
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *(float4 *)(yrow + ((c ^ row_sw) << 4)) = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                // the peer has read what the previous copy put in its X
                bool ok = i == 0 || tc::mbar_wait_cluster(&bar->xempty, (i - 1) & 1, abort_flag, err, 32);
                if (ok) tc::bulk_copy_to_peer(peer_x_warp, (const uint8_t *)Y + wblk, 32 * 128, peer_xfull);
            }
            if (!tc::mbar_wait_cluster(&bar->xfull, i & 1, abort_flag, err, 33)) { done_ok = false; break; }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 x = *(const float4 *)(xrow + ((c ^ row_sw) << 4));
                v[4 * c] += x.x;
                v[4 * c + 1] += x.y;
                v[4 * c + 2] += x.z;
                v[4 * c + 3] += x.w;
            }
            // X may be overwritten by the peer's next copy once every warp has read it
            // (the values are already in registers, so no ordering fence is needed).
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_cluster_relaxed(peer_xempty);
            // --- mask: entries that are padding, future or outside the sequence ---
            if (!tc::mbar_wait(&bar->kv_full[st], (i / NSTAGE) & 1, abort_flag, err, 34)) { done_ok = false; break; }
            {
                const uint4 *kv4 = (const uint4 *)(kvalid + st * BK + hf * 32);
                const uint4 m0 = kv4[0], m1 = kv4[1];
                const uint32_t all = m0.x & m0.y & m0.z & m0.w & m1.x & m1.y & m1.z & m1.w;
                if (all != 0x01010101u) {
                    const uint32_t *kvw = (const uint32_t *)(kvalid + st * BK + hf * 32);
#pragma unroll
                    for (int wd = 0; wd < 8; ++wd) {
                        const uint32_t bits = kvw[wd];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            if (!((bits >> (8 * u)) & 0xffu)) v[4 * wd + u] = -INFINITY;
                    }
                }
            }
            float mh = v[0];
#pragma unroll
            for (int j = 1; j < 32; ++j) mh = fmaxf(mh, v[j]);
            // row maximum = max of the two halves (double-buffered by tile parity)
            pmax[(i & 1) * 2 * NH + hf * NH + h] = mh;
            asm volatile("bar.sync %0, 64;" ::"r"(named) : "memory");
            const float mraw = fmaxf(mh, pmax[(i & 1) * 2 * NH + (1 - hf) * NH + h]);
            const float mt = mraw * sl2;  // the scale is positive: max commutes with it
            bool rescale = false;
            float alpha = 1.0f;
            if (mt != -INFINITY) {
                if (m_used == -INFINITY) {
                    m_used = mt;
                } else if (mt > m_used + RESCALE_LOG2) {
                    alpha = tc::ex2_approx(m_used - mt);
                    l *= alpha;
                    m_used = mt;
                    rescale = true;
                }
            }
            const float neg_m = m_used == -INFINITY ? 0.0f : -m_used;
            uint32_t pk[16];
            float psum0 = 0.0f, psum1 = 0.0f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float p0 = tc::ex2_approx(fmaf(v[2 * j], sl2, neg_m));
                const float p1 = tc::ex2_approx(fmaf(v[2 * j + 1], sl2, neg_m));
                const __nv_bfloat162 t2 = __floats2bfloat162_rn(p0, p1);
                psum0 += __low2float(t2);
                psum1 += __high2float(t2);
                pk[j] = *(const uint32_t *)&t2;
            }
            l += psum0 + psum1;
            // the previous PV product must be done before P and O are touched
            if (i > 0 && !tc::mbar_wait(&bar->p_empty, (i - 1) & 1, abort_flag, err, 35)) { done_ok = false; break; }
            tc::tc_fence_after();
            // tcgen05.ld/st are warp-wide: rescale the warp's half of the O columns when any
            // of its rows needs it (rows that do not keep alpha = 1).
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                for (int cc = hf * 4; cc < hf * 4 + 4; ++cc) {
                    float o[32];
                    uint32_t ob[32];
                    tc::tmem_ld32(tmem + lane_off + COL_O + cc * 32, o);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) ob[j] = __float_as_uint(o[j] * alpha);
                    tc::tmem_st32(tmem + lane_off + COL_O + cc * 32, ob);
                }
            }
            tc::tmem_st16(tmem + lane_off + COL_P + hf * 16, pk);  // 32 bf16 probabilities as 16 packed columns
            tc::tmem_st_wait();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bar->p_full);
        }
        if (lane == 0) tc::bulk_wait_all();  // no copy may still read Y when the CTA exits
        // ---------------- epilogue: normalise and store this thread's 128 columns ----------------
        lsum[hf * NH + h] = l;
        asm volatile("bar.sync %0, 64;" ::"r"(named) : "memory");
        const float lrow = l + lsum[(1 - hf) * NH + h];
        const int64_t rh = (int64_t)r * NH + h;
        const bool have = __all_sync(0xffffffffu, n > 0 && done_ok && tc::mbar_wait(&bar->o_done, 0, abort_flag, err, 36));
        const float inv = (have && lrow > 0.0f) ? 1.0f / lrow : 0.0f;
        const float row_lse = (have && lrow > 0.0f) ? (m_used + log2f(lrow)) * LN2 : -INFINITY;
        if (have) tc::tc_fence_after();
        if (P.splits == 1) {
            __nv_bfloat16 *dst = olat + rh * DC + rank * 256;
#pragma unroll 1
            for (int cc = hf * 4; cc < hf * 4 + 4; ++cc) {
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
                uint4 *d4 = (uint4 *)(dst + cc * 32);
#pragma unroll
                for (int e = 0; e < 4; ++e) d4[e] = make_uint4(pw[4 * e], pw[4 * e + 1], pw[4 * e + 2], pw[4 * e + 3]);
            }
            if (rank == 0 && hf == 0 && lse) lse[rh] = row_lse;
        } else {
            const int64_t part = ((int64_t)r * P.splits + split) * NH + h;
            float *dst = opart + part * DC + rank * 256;
#pragma unroll 1
            for (int cc = hf * 4; cc < hf * 4 + 4; ++cc) {
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
            if (rank == 0 && hf == 0) lpart[part] = row_lse;
        }
    }
    __syncthreads();
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
    if (M >= 152) return 1;
    const int want = (152 + M - 1) / M;
    int s = 1;
    while (s < want && s < 8) s *= 2;
    return s;
}

size_t mla_tc_partial_bytes(int M) {
    const int s = mla_tc_splits(M);
    if (s == 1) return 0;
    return (size_t)M * s * NH * DC * sizeof(float) + 256 + (size_t)M * s * NH * sizeof(float);
}

cudaError_t launch_mla_tc(const void *qt, const void *kv, int64_t ld_kv, const void *kpe, int64_t ld_pe,
                          const int32_t *idx, int k, const SeqTab &st, int64_t total_k, int M, float scale,
                          bool prefix_valid, void *olat, float *lse, void *part_ws, cudaStream_t s) {
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
    float *opart = nullptr, *lpart = nullptr;
    if (P.splits > 1) {
        opart = (float *)part_ws;
        lpart = (float *)((char *)part_ws + (((size_t)M * P.splits * NH * DC * sizeof(float) + 255) / 256) * 256);
    }
    cudaError_t e = cudaFuncSetAttribute(mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)M * P.splits * 2;
    mla_tc_kernel<<<grid, NUM_THREADS, SMEM, s>>>((const __nv_bfloat16 *)kv, ld_kv, (const __nv_bfloat16 *)kpe, ld_pe,
                                                   (const __nv_bfloat16 *)qt, idx, P, (__nv_bfloat16 *)olat, lse,
                                                   opart, lpart);
    note_launch(DSA_KERNEL_MLA_TC);
    e = cudaGetLastError();
    if (e != cudaSuccess || P.splits == 1) return e;
    const unsigned cgrid = (unsigned)(((int64_t)M * NH + 7) / 8);
    mla_combine_kernel<<<cgrid, 256, 0, s>>>(opart, lpart, M, P.splits, (__nv_bfloat16 *)olat, lse);
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
