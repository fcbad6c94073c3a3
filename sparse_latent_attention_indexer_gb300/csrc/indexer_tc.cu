// Lightning indexer on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
//   S~^I_{t,s} = 1/(sqrt(H_I) sqrt(D_I)) sum_h w_{t,h} ReLU(q^I_{h,t} . k^I_s) + M_{t,s}
// (DeepSeek-V3.2-Exp atlas page, MoE transformer block, indexer equations;
// H_I = 64 heads of D_I = 128, the released configuration.)
//
// The head dot products are one dense contraction: for a block of 128 keys
// and a group of 4 query tokens, D[128 keys, 4 x 64 (token, head)] =
// K[128 x 128] . Q[256 x 128]^T, one tcgen05.mma chain (M = 128, N = 256,
// K = 128) with the fp32 accumulator in tensor memory.  Keys sit on the MMA's
// M axis, so after the MMA each epilogue thread owns one key (one TMEM lane)
// and reduces that key's 64 head columns in registers: ReLU, the per-head
// weight (with the constant 1/sqrt(H_I D_I) and, for FP8, the q block scale
// folded in), the head sum, the k block scale, and the causal mask.  No
// [T, 64, S] tensor ever reaches memory; only the [T, S] scores are stored.
//
// CTA = one group of 4 query rows (one sequence) x a strided subset of its
// causal key blocks.  Warp roles: warp 0 issues TMA loads (the 4 x 64 query
// rows once, then key blocks through a STAGES-deep ring), warp 1 issues the
// MMAs, warp 2 owns the tensor memory (512 columns = two 256-column
// accumulators, so the epilogue of block i overlaps the MMAs of block i+1),
// warps 4..11 run the epilogue (two warps per TMEM lane quarter, each taking
// two of the four tokens).  Every wait is bounded; a timeout records its
// site in the device error word and the CTA drains and exits.
//
// FP8 variant: q^I and k^I are e4m3 codes with one power-of-two scale per
// 128-value row (ue8m0), MMA kind::f8f6f4.  Because each scale covers a whole
// head row, sum_h w s_q ReLU(s_k cq.ck) = s_k sum_h (w s_q) ReLU(cq.ck) holds
// exactly, so the scales need no block-scaled MMA.
#include <atomic>

#include "tc_common.cuh"
#include "topk_row.cuh"

namespace dsa {

__device__ int g_indexer_tc_error = 0;

namespace {

constexpr int BM = 128;         // keys per block (MMA M)
constexpr int TOK = 4;          // query tokens per group
constexpr int HI = 64;          // indexer heads
constexpr int DI = 128;         // indexer head dim
constexpr int BN = TOK * HI;    // 256 (MMA N)
// Warps 0-3: TMA producer, MMA issuer, tensor-memory owner, idle; then the epilogue warps.  One-shot
// kernel, bf16: 16 of them, one per (TMEM lane quarter, token) pair, four per SM sub-partition; FP8:
// 8, each taking two tokens of its lane quarter (measured faster for the shorter FP8 MMA).  The
// fused kernel (F) has 8 epilogue warps in both precisions, then the selecting warps: 4 for FP8
// (whose epilogue needs the 128 registers a 512-thread CTA leaves), joined there by warps 2 and 3
// once the tensor memory is allocated, and 8 for bf16 (measured: 7.86 against 8.61 ms of indexer +
// top-k on the 32K prefill).
constexpr int EPI_WARP0 = 4;
template <bool FP8, bool F = false> constexpr int num_epi() { return (FP8 || F) ? 8 : 16; }
template <bool FP8> constexpr int sel_warps() { return FP8 ? 4 : 8; }
template <bool FP8> constexpr int sel_spare() { return FP8 ? 2 : 0; }  // warps 2, 3 select too
template <bool FP8> constexpr int sel_threads() { return (sel_warps<FP8>() + sel_spare<FP8>()) * 32; }
template <bool FP8, bool F = false> constexpr int sel_warp0() { return EPI_WARP0 + num_epi<FP8, F>(); }
template <bool FP8, bool F = false> constexpr int num_threads() {
    return (EPI_WARP0 + num_epi<FP8, F>() + (F ? sel_warps<FP8>() : 0)) * 32;
}
constexpr int SPLIT_TAB = 2 * 152;  // launches with fewer query groups split each group's key blocks

template <bool FP8, bool F = false>
struct Cfg {
    static constexpr int ELT = FP8 ? 1 : 2;
    static constexpr int HALVES = FP8 ? 1 : 2;              // 128-byte column slabs per row
    static constexpr int B_BYTES = BN * DI * ELT;           // 64 KB (bf16) / 32 KB (fp8)
    static constexpr int A_BYTES = BM * DI * ELT;           // 32 KB / 16 KB
    static constexpr int B_HALF = BN * 128;                 // bytes of one 128-byte slab of B
    static constexpr int A_HALF = BM * 128;
    // the fused bf16 kernel gives one stage to the selection's candidate list
    static constexpr int STAGES = FP8 ? 6 : (F ? 3 : 4);
    static constexpr int KSTEPS = FP8 ? 4 : 8;              // MMAs per block (K = 32 / 16 each)
    static constexpr int BAR_BYTES = 256;
    // the fused kernel's selection scratch: histogram + warp sums, then the candidate list
    static constexpr int SEL_HEAD = tk::MAX_BINS * 4 + 512;
    static constexpr int CAND_CAP = F ? (FP8 ? 8192 : 6144) : 0;
    static constexpr int SMEM = 1024 /*align slack*/ + B_BYTES + STAGES * A_BYTES + TOK * HI * 4 + BAR_BYTES +
                                (F ? SEL_HEAD + CAND_CAP * 8 : 0);
    static_assert(SMEM <= 232448, "shared memory per CTA");
};

struct IdxParams {
    int B;
    int q_off[DSA_MAX_SEQS + 1];
    int k_base[DSA_MAX_SEQS];
    int k_len[DSA_MAX_SEQS];
    int start_pos[DSA_MAX_SEQS];
    int g_off[DSA_MAX_SEQS + 1];  // cumulative query groups
    int total_groups;
    int splits;                    // CTAs per group (strided key blocks) when every group gets the same
    // Few groups (decode): group g_of[i] gets s_off[i+1] - s_off[i] CTAs, about one per `target`
    // key blocks, and the table lists groups by decreasing blocks per CTA (heaviest CTAs first).
    int balanced;
    int n_tab;
    int s_off[SPLIT_TAB + 1];
    int g_of[SPLIT_TAB];
    int fill_future;
    int dense_k;  // > 0: skip groups whose rows all see at most dense_k keys (they select every causal key)
    int64_t ld;
    long long wait_limit;  // SM cycles a wait may take before the CTA gives up (the drains keep the default)
    float c;
    int topk;  // the fused kernel: k of the selection
};
static_assert(sizeof(IdxParams) + 256 <= 32764, "launch parameters");

// One group: 4 consecutive query rows of one sequence.
struct Group {
    int r0, p0, ntok, S, kbase, nblk;
};

__device__ __forceinline__ Group group_of(const IdxParams &P, int g) {
    int lo = 0, hi = P.B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (P.g_off[mid] <= g) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    Group G;
    const int t0 = (g - P.g_off[b]) * TOK;
    G.ntok = min(TOK, P.q_off[b + 1] - P.q_off[b] - t0);
    G.r0 = P.q_off[b] + t0;
    G.p0 = P.start_pos[b] + t0;
    G.S = P.k_len[b];
    G.kbase = P.k_base[b];
    G.nblk = (G.p0 + G.ntok - 1) / BM + 1;  // blocks holding keys 0 .. last position
    return G;
}

// Shared-memory layout of both indexer kernels: addresses computed from one base pointer.
template <bool FP8, bool F = false>
struct Smem {
    using C = Cfg<FP8, F>;
    uint8_t *base;
    __device__ __forceinline__ explicit Smem(uint8_t *raw)
        : base((uint8_t *)(((uintptr_t)raw + 1023) & ~(uintptr_t)1023)) {}
    __device__ __forceinline__ uint8_t *Bt() const { return base; }
    __device__ __forceinline__ uint8_t *As() const { return base + C::B_BYTES; }
    __device__ __forceinline__ float *wsm() const { return (float *)(base + C::B_BYTES + C::STAGES * C::A_BYTES); }
    __device__ __forceinline__ uint64_t *bars() const { return (uint64_t *)(wsm() + TOK * HI); }
    __device__ __forceinline__ uint64_t *full(int i) const { return bars() + i; }
    __device__ __forceinline__ uint64_t *empty(int i) const { return bars() + C::STAGES + i; }
    __device__ __forceinline__ uint64_t *bfull() const { return bars() + 2 * C::STAGES; }
    __device__ __forceinline__ uint64_t *tfull(int i) const { return bars() + 2 * C::STAGES + 1 + i; }
    __device__ __forceinline__ uint64_t *tempty(int i) const { return bars() + 2 * C::STAGES + 3 + i; }
    __device__ __forceinline__ uint64_t *mmadone() const { return bars() + 2 * C::STAGES + 5; }
    // fused kernel: the query tile is free again / a slot holds a group's scores / a slot was read
    __device__ __forceinline__ uint64_t *bfree() const { return bars() + 2 * C::STAGES + 6; }
    __device__ __forceinline__ uint64_t *slot_full(int i) const { return bars() + 2 * C::STAGES + 7 + i; }
    __device__ __forceinline__ uint64_t *slot_free(int i) const { return bars() + 2 * C::STAGES + 9 + i; }
    __device__ __forceinline__ uint32_t *tmem_slot() const { return (uint32_t *)(bars() + 2 * C::STAGES + 11); }
    __device__ __forceinline__ volatile int *abort_flag() const { return (volatile int *)(tmem_slot() + 1); }
    __device__ __forceinline__ uint8_t *sel() const { return (uint8_t *)bars() + C::BAR_BYTES; }
};

// Barrier phases carried from group to group by a CTA that takes several groups: loads issued
// into the stage ring, accumulators used, query-tile loads and MMA drains.
struct Phases {
    int it = 0, ai = 0, nq = 0, md = 0;
    __device__ __forceinline__ void advance(int mine) {
        it += mine;
        ai += mine;
        nq += mine > 0;
        md += mine > 0;
    }
};

template <bool FP8, bool F = false>
__device__ __forceinline__ void init_barriers(const Smem<FP8, F> &sm) {
    using C = Cfg<FP8, F>;
    static_assert((2 * C::STAGES + 12) * 8 <= C::BAR_BYTES, "barrier area");
    for (int i = 0; i < C::STAGES; ++i) {
        tc::mbar_init(sm.full(i), 1);
        tc::mbar_init(sm.empty(i), 1);
    }
    tc::mbar_init(sm.bfull(), 1);
    for (int i = 0; i < 2; ++i) {
        tc::mbar_init(sm.tfull(i), 1);
        tc::mbar_init(sm.tempty(i), num_epi<FP8, F>());
    }
    tc::mbar_init(sm.mmadone(), 1);
    if (F) {
        tc::mbar_init(sm.bfree(), 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(sm.slot_full(i), num_epi<FP8, F>() * 32);
            tc::mbar_init(sm.slot_free(i), sel_threads<FP8>());
        }
    }
    *sm.abort_flag() = 0;
    tc::fence_mbar_init();
}

// The weights of the group's rows, with the constant 1/sqrt(H_I D_I) and (FP8) the q block scale
// folded in; written by the epilogue threads.
template <bool FP8, bool F = false>
__device__ __forceinline__ void load_weights(const Smem<FP8, F> &sm, const float *__restrict__ w,
                                             const float *__restrict__ q_scale, const IdxParams &P, const Group &G) {
    constexpr int NE = num_epi<FP8, F>() * 32;
    for (int i = threadIdx.x - EPI_WARP0 * 32; i < TOK * HI; i += NE) {
        const int tt = i / HI, h = i % HI;
        float v = 0.0f;
        if (tt < G.ntok) {
            const int64_t qi = (int64_t)(G.r0 + tt) * HI + h;
            v = w[qi] * P.c * (FP8 ? q_scale[qi] : 1.0f);
        }
        sm.wsm()[i] = v;
    }
}

// The epilogue of one key block held in accumulator `acc`: warp (q, first token) reduces its
// tokens for the keys of TMEM lane quarter q (key = this thread's key of the block, keyed from 0
// within the sequence) and writes row tt of the group to out_base + tt * ld.  Releases the
// accumulator to the MMA issuer.
template <bool FP8, bool F>
__device__ __forceinline__ void epilogue_block(const Smem<FP8, F> &sm, uint32_t tmem, int acc, int key,
                                               const Group &G, const float *__restrict__ k_scale, float *out_base,
                                               int64_t ld) {
    constexpr int EPI = num_epi<FP8, F>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, t_first = (warp - EPI_WARP0) >> 2, t_step = EPI / 4;
    const float ks = (FP8 && key < G.S) ? k_scale[G.kbase + key] : 1.0f;
#pragma unroll 1
    for (int tt = t_first; tt < G.ntok; tt += t_step) {
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + acc * BN + tt * HI;
        const float4 *wv = (const float4 *)(sm.wsm() + tt * HI);
        float s0 = 0.0f, s1 = 0.0f;
        if constexpr (EPI == 16) {
            // One token per warp, under the 96 registers a 640-thread CTA leaves: heads 0-31, then
            // 32-63, 32 accumulator values live at a time; the accumulator goes back to the MMA once
            // the second half is loaded.
            {
                float v0[32];
                tc::tmem_ld32(taddr, v0);
                tc::tmem_ld_wait();
#pragma unroll
                for (int h4 = 0; h4 < 8; ++h4) {
                    const float4 a4 = wv[h4];
                    s0 = fmaf(a4.x, fmaxf(v0[4 * h4 + 0], 0.0f), s0);
                    s0 = fmaf(a4.y, fmaxf(v0[4 * h4 + 1], 0.0f), s0);
                    s0 = fmaf(a4.z, fmaxf(v0[4 * h4 + 2], 0.0f), s0);
                    s0 = fmaf(a4.w, fmaxf(v0[4 * h4 + 3], 0.0f), s0);
                }
            }
            float v1[32];
            tc::tmem_ld32(taddr + 32, v1);
            tc::tmem_ld_wait();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(sm.tempty(acc));
#pragma unroll
            for (int h4 = 0; h4 < 8; ++h4) {
                const float4 c4 = wv[8 + h4];
                s1 = fmaf(c4.x, fmaxf(v1[4 * h4 + 0], 0.0f), s1);
                s1 = fmaf(c4.y, fmaxf(v1[4 * h4 + 1], 0.0f), s1);
                s1 = fmaf(c4.z, fmaxf(v1[4 * h4 + 2], 0.0f), s1);
                s1 = fmaf(c4.w, fmaxf(v1[4 * h4 + 3], 0.0f), s1);
            }
        } else {
            // Two tokens per warp, 128 registers: all 64 heads of a token at once.
            float v0[32], v1[32];
            tc::tmem_ld32(taddr, v0);
            tc::tmem_ld32(taddr + 32, v1);
            tc::tmem_ld_wait();
#pragma unroll
            for (int h4 = 0; h4 < 8; ++h4) {
                const float4 a4 = wv[h4], c4 = wv[8 + h4];
                s0 = fmaf(a4.x, fmaxf(v0[4 * h4 + 0], 0.0f), s0);
                s1 = fmaf(c4.x, fmaxf(v1[4 * h4 + 0], 0.0f), s1);
                s0 = fmaf(a4.y, fmaxf(v0[4 * h4 + 1], 0.0f), s0);
                s1 = fmaf(c4.y, fmaxf(v1[4 * h4 + 1], 0.0f), s1);
                s0 = fmaf(a4.z, fmaxf(v0[4 * h4 + 2], 0.0f), s0);
                s1 = fmaf(c4.z, fmaxf(v1[4 * h4 + 2], 0.0f), s1);
                s0 = fmaf(a4.w, fmaxf(v0[4 * h4 + 3], 0.0f), s0);
                s1 = fmaf(c4.w, fmaxf(v1[4 * h4 + 3], 0.0f), s1);
            }
        }
        if (key < G.S) out_base[(int64_t)tt * ld + key] = (key <= G.p0 + tt) ? (s0 + s1) * ks : -INFINITY;
    }
    if (EPI == 8 || t_first >= G.ntok) {
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(sm.tempty(acc));
    }
}

// The scores of `mine` key blocks of group G (blocks split, split + splits, ...): the TMA producer
// (warp 0), the MMA issuer (warp 1) and the epilogue (warps EPI_WARP0..), which writes row tt of the
// group to out_base + tt * P.ld.
template <bool FP8>
__device__ __forceinline__ void group_pipeline(const CUtensorMap *tm_q, const CUtensorMap *tm_k,
                                               const float *__restrict__ k_scale, const IdxParams &P,
                                               const Group &G, int split, int splits, int mine, float *out_base,
                                               const Smem<FP8> &sm, uint32_t tmem, const Phases &ph,
                                               volatile int *never) {
    using C = Cfg<FP8>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int *abort_flag = sm.abort_flag();
    if (mine <= 0) return;
    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        tc::prefetch_tmap(tm_q);
        tc::prefetch_tmap(tm_k);
        tc::mbar_arrive_expect_tx(sm.bfull(), C::B_BYTES);
        for (int h = 0; h < C::HALVES; ++h) tc::tma_load_2d(sm.Bt() + h * C::B_HALF, tm_q, sm.bfull(), h * 64, G.r0 * HI);
        int issued = 0;
        for (int i = 0; i < mine; ++i) {
            const int it = ph.it + i, st = it % C::STAGES;
            if (!tc::mbar_wait(sm.empty(st), ((it / C::STAGES) & 1) ^ 1, abort_flag, &g_indexer_tc_error, 1,
                               P.wait_limit))
                break;
            const int row = G.kbase + (split + i * splits) * BM;
            tc::mbar_arrive_expect_tx(sm.full(st), C::A_BYTES);
            for (int h = 0; h < C::HALVES; ++h)
                tc::tma_load_2d(sm.As() + st * C::A_BYTES + h * C::A_HALF, tm_k, sm.full(st), h * 64, row);
            ++issued;
        }
        // Drain: the last loads of each stage must have landed before the CTA exits.
        tc::mbar_wait(sm.bfull(), ph.nq & 1, never, &g_indexer_tc_error, 2);
        for (int j = max(0, issued - C::STAGES); j < issued; ++j) {
            const int it = ph.it + j;
            tc::mbar_wait(sm.full(it % C::STAGES), (it / C::STAGES) & 1, never, &g_indexer_tc_error, 3);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        bool ok = tc::mbar_wait(sm.bfull(), ph.nq & 1, abort_flag, &g_indexer_tc_error, 4, P.wait_limit);
        // Only the group's valid tokens are multiplied: N = 64 heads x ntok.
        const uint32_t idesc = FP8 ? tc::instr_desc(tc::kFmtE4M3, tc::kFmtE4M3, BM, HI * G.ntok, 0, 0)
                                   : tc::instr_desc(tc::kFmtBF16, tc::kFmtBF16, BM, HI * G.ntok, 0, 0);
        int issued = 0;
        for (int i = 0; ok && i < mine; ++i) {
            const int it = ph.it + i, st = it % C::STAGES, a = ph.ai + i, acc = a & 1;
            if (!tc::mbar_wait(sm.tempty(acc), ((a >> 1) & 1) ^ 1, abort_flag, &g_indexer_tc_error, 5, P.wait_limit))
                break;
            if (!tc::mbar_wait(sm.full(st), (it / C::STAGES) & 1, abort_flag, &g_indexer_tc_error, 6, P.wait_limit))
                break;
            tc::tc_fence_after();
            const uint32_t d = tmem + acc * BN;
            const uint32_t a0 = tc::smem_u32(sm.As() + st * C::A_BYTES), b0 = tc::smem_u32(sm.Bt());
#pragma unroll
            for (int kk = 0; kk < C::KSTEPS; ++kk) {
                // 32 bytes of K per step: 16 bf16 or 32 e4m3 values.
                const int slab = FP8 ? 0 : kk / 4, off = (FP8 ? kk : kk % 4) * 32;
                const uint64_t ad = tc::smem_desc(a0 + slab * C::A_HALF + off, 16, 1024);
                const uint64_t bd = tc::smem_desc(b0 + slab * C::B_HALF + off, 16, 1024);
                if (FP8) tc::mma_f8(d, ad, bd, idesc, kk > 0);
                else tc::mma_f16(d, ad, bd, idesc, kk > 0);
            }
            tc::mma_commit(sm.empty(st));
            tc::mma_commit(sm.tfull(acc));
            ++issued;
        }
        // No MMA may still be running when the tensor memory is released (or the ring reused).
        if (issued > 0) {
            tc::mma_commit(sm.mmadone());
            tc::mbar_wait(sm.mmadone(), ph.md & 1, never, &g_indexer_tc_error, 7);
        }
    } else if (warp >= EPI_WARP0) {
        // ---------------- epilogue ----------------
        // bf16: warp (q, tt) reduces token tt for the keys of lane quarter q.  FP8: the two
        // warps of lane quarter q take tokens hf and hf + 2.  Absent tokens are skipped.
        const int q = warp & 3;
        for (int i = 0; i < mine; ++i) {
            const int a = ph.ai + i, acc = a & 1;
            if (!tc::mbar_wait(sm.tfull(acc), (a >> 1) & 1, abort_flag, &g_indexer_tc_error, 8, P.wait_limit)) break;
            tc::tc_fence_after();
            epilogue_block<FP8, false>(sm, tmem, acc, (split + i * splits) * BM + q * 32 + lane, G, k_scale, out_base,
                                       P.ld);
        }
    }
}

template <bool FP8>
__global__ void __launch_bounds__(num_threads<FP8>(), 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const float *__restrict__ w, const float *__restrict__ q_scale,
                      const float *__restrict__ k_scale, const __grid_constant__ IdxParams P,
                      float *__restrict__ scores) {
    extern __shared__ uint8_t smem_raw[];
    const Smem<FP8> sm(smem_raw);
    __shared__ int never;  // an abort flag nobody raises, for the drain waits

    const int warp = threadIdx.x >> 5;
    // Heavier groups (later tokens of a sequence see more keys) start first.
    int g, split, splits;
    if (P.balanced) {
        int lo = 0, hi = P.n_tab - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (P.s_off[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
        }
        g = P.g_of[lo];
        split = (int)blockIdx.x - P.s_off[lo];
        splits = P.s_off[lo + 1] - P.s_off[lo];
    } else {
        const int lin = P.total_groups * P.splits - 1 - (int)blockIdx.x;
        g = lin / P.splits;
        split = lin % P.splits;
        splits = P.splits;
    }
    const Group G = group_of(P, g);
    // A group whose last row sits at position < dense_k needs no scores: every row of it selects all
    // of its causal keys, and the top-k does not read them.
    const bool dense = P.dense_k > 0 && G.p0 + G.ntok - 1 < P.dense_k;
    const int mine = (split < G.nblk && !dense) ? (G.nblk - split + splits - 1) / splits : 0;

    if (threadIdx.x == 0) {
        init_barriers(sm);
        never = 0;
    }
    if (warp == 2) {
        tc::tmem_alloc(sm.tmem_slot(), 512);
        tc::tmem_relinquish();
    }
    pdl_wait();  // the set-up above overlapped the previous kernel; global memory only from here
    if (warp >= EPI_WARP0) load_weights(sm, w, q_scale, P, G);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *sm.tmem_slot();
    group_pipeline<FP8>(&tm_q, &tm_k, k_scale, P, G, split, splits, mine, scores + (int64_t)G.r0 * P.ld, sm, tmem,
                        Phases(), (volatile int *)&never);
    __syncthreads();
    pdl_trigger();
    // Masked tail: keys past every computed block are future keys of all rows.
    if (P.fill_future && split == 0 && warp >= EPI_WARP0) {
        const int start = G.nblk * BM;
        for (int tt = 0; tt < G.ntok; ++tt)
            for (int s = start + threadIdx.x - EPI_WARP0 * 32; s < G.S; s += num_threads<FP8>() - EPI_WARP0 * 32)
                scores[(int64_t)(G.r0 + tt) * P.ld + s] = -INFINITY;
    }
    if (warp == 2) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// Named barrier ID over N threads that also ANDs `v` over them (so the group takes one decision).
template <int ID, int N>
__device__ __forceinline__ bool bar_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(ID), "n"(N)
        : "memory");
    return r != 0;
}

// Position j of a CTA's walk over the groups, heaviest first: the CTAs take positions in a snake
// order (0 .. G-1, then G-1 .. 0, ...), so each gets a similar mix of heavy and light groups.
__device__ __forceinline__ int walk_group(const IdxParams &P, int j) {
    const int G = (int)gridDim.x;
    const int pos = j * G + ((j & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
    return pos < P.total_groups ? P.total_groups - 1 - pos : -1;
}

// The indexer and the top-k fused.  A persistent CTA per SM walks query groups (walk_group).  The
// producer, the MMA issuer and the epilogue run the indexer of group after group without draining in
// between: the epilogue writes a group's 4 score rows into one of the CTA's two slots (slots:
// [gridDim.x][2][4][P.ld] fp32), and four selecting warps take each filled slot, select every row's
// top-k from it (reading it back from L2) and write the indices to idx [rows, P.topk] -- while the
// tensor cores already compute the next group.  No [rows, S] score buffer exists.  Groups whose rows
// all see at most k keys skip the MMAs; their selection is the dense one (0 .. n-1, then -1).
// Hand-offs: bfree (the MMAs of a group are done, its query tile may be replaced), slot_full (the
// epilogue's rows of a group are in the slot) and slot_free (the selecting warps are done with it).
template <bool FP8>
__global__ void __launch_bounds__(num_threads<FP8, true>(), 1)
    indexer_topk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const float *__restrict__ w, const float *__restrict__ q_scale,
                        const float *__restrict__ k_scale, const __grid_constant__ IdxParams P,
                        float *__restrict__ slots, int32_t *__restrict__ idx) {
    using C = Cfg<FP8, true>;
    constexpr int EPI = num_epi<FP8, true>();
    constexpr int SEL0 = sel_warp0<FP8, true>();
    constexpr int NS = sel_threads<FP8>();  // selecting threads
    extern __shared__ uint8_t smem_raw[];
    const Smem<FP8, true> sm(smem_raw);
    __shared__ int never;
    volatile int *nv = (volatile int *)&never;
    volatile int *abort_flag = sm.abort_flag();
    int *err = &g_indexer_tc_error;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        init_barriers(sm);
        never = 0;
    }
    if (warp == 2) {
        tc::tmem_alloc(sm.tmem_slot(), 512);
        tc::tmem_relinquish();
    }
    pdl_wait();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *sm.tmem_slot();
    float *slot0 = slots + (int64_t)blockIdx.x * 2 * TOK * P.ld;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_k);
        int it = 0, nq = 0;
        bool ok = true;
        for (int j = 0; ok; ++j) {
            const int g = walk_group(P, j);
            if (g < 0) break;
            const Group G = group_of(P, g);
            if (G.p0 + G.ntok - 1 < P.topk) continue;  // dense: no scores
            // the previous group's MMAs must be done reading the query tile
            if (nq > 0 && !(ok = tc::mbar_wait(sm.bfree(), (nq - 1) & 1, abort_flag, err, 41, P.wait_limit))) break;
            tc::mbar_arrive_expect_tx(sm.bfull(), C::B_BYTES);
            for (int h = 0; h < C::HALVES; ++h)
                tc::tma_load_2d(sm.Bt() + h * C::B_HALF, &tm_q, sm.bfull(), h * 64, G.r0 * HI);
            ++nq;
            for (int i = 0; i < G.nblk; ++i, ++it) {
                const int st = it % C::STAGES;
                if (!(ok = tc::mbar_wait(sm.empty(st), ((it / C::STAGES) & 1) ^ 1, abort_flag, err, 42, P.wait_limit)))
                    break;
                tc::mbar_arrive_expect_tx(sm.full(st), C::A_BYTES);
                for (int h = 0; h < C::HALVES; ++h)
                    tc::tma_load_2d(sm.As() + st * C::A_BYTES + h * C::A_HALF, &tm_k, sm.full(st), h * 64,
                                    G.kbase + i * BM);
            }
        }
        // Drain: nothing may still be landing in shared memory when the CTA exits.
        if (nq > 0) tc::mbar_wait(sm.bfull(), (nq - 1) & 1, nv, err, 43);
        for (int i = max(0, it - C::STAGES); i < it; ++i)
            tc::mbar_wait(sm.full(i % C::STAGES), (i / C::STAGES) & 1, nv, err, 44);
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        int it = 0, ai = 0, nq = 0, issued = 0;
        bool ok = true;
        for (int j = 0; ok; ++j) {
            const int g = walk_group(P, j);
            if (g < 0) break;
            const Group G = group_of(P, g);
            if (G.p0 + G.ntok - 1 < P.topk) continue;
            if (!(ok = tc::mbar_wait(sm.bfull(), nq & 1, abort_flag, err, 45, P.wait_limit))) break;
            ++nq;
            const uint32_t idesc = FP8 ? tc::instr_desc(tc::kFmtE4M3, tc::kFmtE4M3, BM, HI * G.ntok, 0, 0)
                                       : tc::instr_desc(tc::kFmtBF16, tc::kFmtBF16, BM, HI * G.ntok, 0, 0);
            for (int i = 0; i < G.nblk; ++i, ++it, ++ai) {
                const int st = it % C::STAGES, acc = ai & 1;
                if (!(ok = tc::mbar_wait(sm.tempty(acc), ((ai >> 1) & 1) ^ 1, abort_flag, err, 46, P.wait_limit)))
                    break;
                if (!(ok = tc::mbar_wait(sm.full(st), (it / C::STAGES) & 1, abort_flag, err, 47, P.wait_limit)))
                    break;
                tc::tc_fence_after();
                const uint32_t d = tmem + acc * BN;
                const uint32_t a0 = tc::smem_u32(sm.As() + st * C::A_BYTES), b0 = tc::smem_u32(sm.Bt());
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS; ++kk) {
                    const int slab = FP8 ? 0 : kk / 4, off = (FP8 ? kk : kk % 4) * 32;
                    const uint64_t ad = tc::smem_desc(a0 + slab * C::A_HALF + off, 16, 1024);
                    const uint64_t bd = tc::smem_desc(b0 + slab * C::B_HALF + off, 16, 1024);
                    if (FP8) tc::mma_f8(d, ad, bd, idesc, kk > 0);
                    else tc::mma_f16(d, ad, bd, idesc, kk > 0);
                }
                tc::mma_commit(sm.empty(st));
                tc::mma_commit(sm.tfull(acc));
                ++issued;
            }
            if (!ok) break;
            tc::mma_commit(sm.bfree());  // arrives once this group's MMAs are done: the query tile is free
        }
        // No MMA may still be running when the tensor memory is released.
        if (issued > 0) {
            tc::mma_commit(sm.mmadone());
            tc::mbar_wait(sm.mmadone(), 0, nv, err, 48);
        }
    } else if (warp >= EPI_WARP0 && warp < SEL0) {
        // ---------------- epilogue: scores into the slots ----------------
        const int q = warp & 3;
        int ai = 0;
        for (int j = 0;; ++j) {
            const int g = walk_group(P, j);
            if (g < 0) break;
            const Group G = group_of(P, g);
            const bool dense = G.p0 + G.ntok - 1 < P.topk;
            const int sb = j & 1;
            // the selecting warps are done with this slot's previous group; all epilogue warps take
            // the same decision (and have finished the previous group, whose weights are replaced next)
            bool ok = j < 2 || tc::mbar_wait(sm.slot_free(sb), ((j >> 1) - 1) & 1, abort_flag, err, 49, P.wait_limit);
            if (!bar_and<1, EPI * 32>(ok)) break;
            if (!dense) {
                load_weights<FP8, true>(sm, w, q_scale, P, G);
                asm volatile("bar.sync 1, %0;" ::"n"(EPI * 32) : "memory");
                float *out = slot0 + (int64_t)sb * TOK * P.ld;
                for (int i = 0; i < G.nblk; ++i, ++ai) {
                    const int acc = ai & 1;
                    if (!(ok = tc::mbar_wait(sm.tfull(acc), (ai >> 1) & 1, abort_flag, err, 50, P.wait_limit))) break;
                    tc::tc_fence_after();
                    epilogue_block<FP8, true>(sm, tmem, acc, i * BM + q * 32 + lane, G, k_scale, out, P.ld);
                }
            }
            tc::mbar_arrive(sm.slot_full(sb));  // releases this thread's score writes
        }
    } else if (warp >= SEL0 || (sel_spare<FP8>() > 0 && (warp == 2 || warp == 3))) {
        // ---------------- selection: the top-k of each filled slot ----------------
        // group-local thread index: warps 2, 3 (when they select) first, then the selecting warps
        const int tid = warp >= SEL0 ? (warp - SEL0 + sel_spare<FP8>()) * 32 + lane : (warp - 2) * 32 + lane;
        uint8_t *sc = sm.sel();
        const tk::FilterSmem fs{(uint32_t *)sc, (int *)(sc + tk::MAX_BINS * 4), (int *)(sc + tk::MAX_BINS * 4 + 128),
                                (int *)(sc + tk::MAX_BINS * 4 + 256), (uint32_t *)(sc + C::SEL_HEAD),
                                (int32_t *)(sc + C::SEL_HEAD + C::CAND_CAP * 4), C::CAND_CAP};
        for (int j = 0;; ++j) {
            const int g = walk_group(P, j);
            if (g < 0) break;
            const Group G = group_of(P, g);
            const int sb = j & 1;
            // one decision for the selecting warps (their selection synchronises on barrier 2)
            if (!bar_and<2, NS>(tc::mbar_wait(sm.slot_full(sb), (j >> 1) & 1, abort_flag, err, 51, P.wait_limit)))
                break;
            const float *slot = slot0 + (int64_t)sb * TOK * P.ld;
            for (int tt = 0; tt < G.ntok; ++tt)
                tk::sampled_row<NS, 2, false>(tid, slot + (int64_t)tt * P.ld, min(G.p0 + tt + 1, G.S), P.topk, true,
                                             idx + (int64_t)(G.r0 + tt) * P.topk, fs);
            tc::mbar_arrive(sm.slot_free(sb));  // the reads of this slot are done
        }
    }
    __syncthreads();
    pdl_trigger();
    if (warp == 2) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool indexer_tc_supported(int dtype, int H_I, int D_I) {
    return (dtype == DSA_BF16 || dtype == DSA_E4M3) && H_I == HI && D_I == DI;
}

int indexer_tc_read_error(int *site) {
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_indexer_tc_error, sizeof(int));
    if (e != cudaSuccess) return fail_cuda(e);
    if (v) {
        e = cudaMemcpyToSymbol(g_indexer_tc_error, &zero, sizeof(int));
        if (e != cudaSuccess) return fail_cuda(e);
        if (site) *site = v;
        return DSA_ERR_TIMEOUT;
    }
    return DSA_OK;
}

namespace {

// The per-launch table of groups.  Returns the number of groups.
unsigned fill_params(IdxParams &P, const SeqTab &st) {
    P.B = st.B;
    P.g_off[0] = 0;
    for (int i = 0; i < st.B; ++i) {
        P.q_off[i] = st.q_off[i];
        P.k_base[i] = st.k_base[i];
        P.k_len[i] = st.k_len[i];
        P.start_pos[i] = st.start_pos[i];
        const int T = st.q_off[i + 1] - st.q_off[i];
        P.g_off[i + 1] = P.g_off[i] + (T + TOK - 1) / TOK;
    }
    P.q_off[st.B] = st.q_off[st.B];
    P.total_groups = P.g_off[st.B];
    P.splits = 1;
    P.balanced = 0;
    P.n_tab = 0;
    P.fill_future = 0;
    P.dense_k = 0;
    P.topk = 0;
    P.wait_limit = wait_limit_cycles();
    P.c = 1.0f / sqrtf((float)(HI * DI));
    return (unsigned)P.total_groups;
}

bool make_maps(CUtensorMap &tq, CUtensorMap &tk, const void *q, const void *k, bool fp8, int total_q,
               int64_t total_k) {
    const CUtensorMapDataType ty = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t row_bytes = (uint64_t)DI * (fp8 ? 1 : 2);
    const uint32_t inner = fp8 ? 128 : 64;
    {
        uint64_t dims[2] = {(uint64_t)DI, (uint64_t)total_q * HI};
        uint64_t strides[1] = {row_bytes};
        uint32_t box[2] = {inner, (uint32_t)BN};
        if (!make_tmap(&tq, ty, 2, q, dims, strides, box)) return false;
    }
    {
        uint64_t dims[2] = {(uint64_t)DI, (uint64_t)std::max<int64_t>(total_k, 1)};
        uint64_t strides[1] = {row_bytes};
        uint32_t box[2] = {inner, (uint32_t)BM};
        if (!make_tmap(&tk, ty, 2, k, dims, strides, box)) return false;
    }
    return true;
}

}  // namespace

cudaError_t launch_indexer_tc(const void *q, const float *q_scale, const void *k, const float *k_scale, int dtype,
                              const float *w, const SeqTab &st, int64_t total_k, float *scores, int64_t ld,
                              bool fill_future, cudaStream_t s, int dense_k) {
    const bool fp8 = dtype == DSA_E4M3;
    static thread_local IdxParams P;  // ~10 KB: keep it off the host stack
    unsigned grid = fill_params(P, st);
    if (grid == 0) return cudaSuccess;
    if (P.total_groups < SPLIT_TAB) {
        // Few groups of (possibly very) different lengths: about SPLIT_TAB CTAs of `target` key
        // blocks each, so that no CTA carries a long row's blocks alone.
        int nblk[SPLIT_TAB], order[SPLIT_TAB];
        int64_t total_blocks = 0;
        for (int b = 0; b < st.B; ++b)
            for (int g = P.g_off[b]; g < P.g_off[b + 1]; ++g) {
                const int t0 = (g - P.g_off[b]) * TOK;
                const int ntok = std::min(TOK, st.q_off[b + 1] - st.q_off[b] - t0);
                nblk[g] = (st.start_pos[b] + t0 + ntok - 1) / BM + 1;
                total_blocks += nblk[g];
            }
        // One CTA per SM at a time: the CTA count must not pass SPLIT_TAB (two full waves), or a
        // third, nearly empty wave of full-size CTAs would follow.  Rounding each group up can
        // overshoot, so the blocks per CTA grow until the count fits.
        int target = (int)std::max<int64_t>(1, (total_blocks + SPLIT_TAB - 1) / SPLIT_TAB);
        int per_cta[SPLIT_TAB], sp[SPLIT_TAB];
        for (;; ++target) {
            int ctas = 0;
            for (int g = 0; g < P.total_groups; ++g) {
                sp[g] = std::max(1, std::min(nblk[g], (nblk[g] + target - 1) / target));
                ctas += sp[g];
            }
            if (ctas <= SPLIT_TAB) break;
        }
        for (int g = 0; g < P.total_groups; ++g) {
            per_cta[g] = (nblk[g] + sp[g] - 1) / sp[g];
            order[g] = g;
        }
        std::stable_sort(order, order + P.total_groups, [&](int a, int b) { return per_cta[a] > per_cta[b]; });
        P.balanced = 1;
        P.n_tab = P.total_groups;
        P.s_off[0] = 0;
        for (int i = 0; i < P.total_groups; ++i) {
            P.g_of[i] = order[i];
            P.s_off[i + 1] = P.s_off[i] + sp[order[i]];
        }
        grid = (unsigned)P.s_off[P.total_groups];
    }
    P.fill_future = fill_future ? 1 : 0;
    P.dense_k = dense_k;
    P.ld = ld;

    CUtensorMap tq, tk;
    if (!make_maps(tq, tk, q, k, fp8, st.q_off[st.B], total_k)) return cudaErrorInvalidValue;
    cudaError_t e;
    if (fp8) {
        e = cudaFuncSetAttribute(indexer_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<true>::SMEM);
        if (e != cudaSuccess) return e;
        e = launch_pdl(indexer_tc_kernel<true>, dim3(grid), dim3(num_threads<true>()), Cfg<true>::SMEM, s, tq, tk, w,
                       q_scale, k_scale, P, scores);
        if (e != cudaSuccess) return e;
        note_launch(DSA_KERNEL_INDEXER_FP8);
    } else {
        e = cudaFuncSetAttribute(indexer_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<false>::SMEM);
        if (e != cudaSuccess) return e;
        e = launch_pdl(indexer_tc_kernel<false>, dim3(grid), dim3(num_threads<false>()), Cfg<false>::SMEM, s, tq, tk,
                       w, (const float *)nullptr, (const float *)nullptr, P, scores);
        if (e != cudaSuccess) return e;
        note_launch(DSA_KERNEL_INDEXER_TC);
    }
    return cudaGetLastError();
}

int indexer_topk_groups(const SeqTab &st) {
    int g = 0;
    for (int b = 0; b < st.B; ++b) g += (st.q_off[b + 1] - st.q_off[b] + TOK - 1) / TOK;
    return g;
}

// -1: automatic (default), 0: never, 1: wherever the fused kernel applies.
std::atomic<int> g_fused_topk{-1};

bool indexer_topk_fused_ok(int dtype, int H_I, int D_I, const SeqTab &st, int k) {
    // Applies with enough groups to fill the GPU (few groups -- decode -- split each group's key
    // blocks over many CTAs instead, and select afterwards) and candidate lists that fit the scratch.
    const int mode = g_fused_topk.load(std::memory_order_relaxed);
    if (mode == 0 || !indexer_tc_supported(dtype, H_I, D_I) || indexer_topk_groups(st) < SPLIT_TAB || k > 8192)
        return false;
    if (mode == 1) return true;
    // Automatic: where it measured faster on the GB300 -- the FP8 indexer over rows that see on
    // average at least 16K keys (the chunked prefill: 24.0 against 25.2 ms of indexer + top-k).  The
    // bf16 variant runs 8 epilogue warps and 3 stages (16 and 4 in the one-shot kernel, which the
    // selection's shared memory and registers leave no room for) and was slower.
    double live = 0.0, rows = 0.0;
    for (int b = 0; b < st.B; ++b) {
        const double T = st.q_off[b + 1] - st.q_off[b], p0 = st.start_pos[b];
        live += T * p0 + T * (T + 1) / 2;
        rows += T;
    }
    return dtype == DSA_E4M3 && rows > 0 && live >= 16384.0 * rows;
}

size_t indexer_topk_slot_bytes(const SeqTab &st, int64_t ld) {
    const int grid = std::min(indexer_topk_groups(st), device_sm_count());
    return (size_t)grid * 2 * TOK * ld * sizeof(float);
}

cudaError_t launch_indexer_topk_tc(const void *q, const float *q_scale, const void *k, const float *k_scale, int dtype,
                                   const float *w, const SeqTab &st, int64_t total_k, float *slots, int64_t ld,
                                   int topk, int32_t *idx, cudaStream_t s) {
    const bool fp8 = dtype == DSA_E4M3;
    static thread_local IdxParams P;
    const unsigned groups = fill_params(P, st);
    if (groups == 0) return cudaSuccess;
    P.ld = ld;
    P.topk = topk;
    P.dense_k = topk;
    const unsigned grid = std::min<unsigned>(groups, (unsigned)device_sm_count());
    CUtensorMap tq, tk;
    if (!make_maps(tq, tk, q, k, fp8, st.q_off[st.B], total_k)) return cudaErrorInvalidValue;
    cudaError_t e;
    if (fp8) {
        e = cudaFuncSetAttribute(indexer_topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<true, true>::SMEM);
        if (e != cudaSuccess) return e;
        e = launch_pdl(indexer_topk_kernel<true>, dim3(grid), dim3(num_threads<true, true>()), Cfg<true, true>::SMEM, s,
                       tq, tk, w, q_scale, k_scale, P, slots, idx);
        if (e != cudaSuccess) return e;
        note_launch(DSA_KERNEL_INDEXER_FP8 | DSA_KERNEL_INDEXER_TOPK);
    } else {
        e = cudaFuncSetAttribute(indexer_topk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<false, true>::SMEM);
        if (e != cudaSuccess) return e;
        e = launch_pdl(indexer_topk_kernel<false>, dim3(grid), dim3(num_threads<false, true>()),
                       Cfg<false, true>::SMEM, s, tq, tk, w, (const float *)nullptr, (const float *)nullptr, P, slots,
                       idx);
        if (e != cudaSuccess) return e;
        note_launch(DSA_KERNEL_INDEXER_TC | DSA_KERNEL_INDEXER_TOPK);
    }
    return cudaGetLastError();
}

}  // namespace dsa

extern "C" int dsa_set_fused_topk(int mode) {
    if (mode < -1 || mode > 1) return DSA_ERR_INVALID_ARG;
    dsa::g_fused_topk.store(mode, std::memory_order_relaxed);
    return DSA_OK;
}
