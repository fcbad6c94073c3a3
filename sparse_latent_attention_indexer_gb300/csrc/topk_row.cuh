// Exact top-k of one row of fp32 scores by a group of NT threads (a radix
// select on order-preserving uint32 keys), shared by the stand-alone top-k
// kernels (topk.cu) and the indexer kernel that selects from the scores it
// has just computed (indexer_tc.cu).  DeepSeek-V3.2-Exp atlas page,
// M^sel_{t,s} = M_{t,s} for s in top_k(S~^I_t).
//
// The group synchronises with __syncthreads() (BAR = 0: the whole CTA) or
// with named barrier BAR over exactly NT threads.  `tid` is the thread's
// index within the group (0 .. NT-1), warp-aligned.
//
// Output of a row: the exact top-k set, written as [keys above the k-th key T,
// in increasing key index][the first keys equal to T, in increasing key
// index], so equal scores resolve to the lower key index.
#pragma once

#include "dsa_common.cuh"

namespace dsa {
namespace tk {

constexpr int MAX_BINS = 2048;
constexpr int SPT = 16;  // consecutive scores per thread per streaming step

template <int NT, int BAR>
__device__ __forceinline__ void group_sync() {
    if constexpr (BAR == 0) {
        __syncthreads();
    } else {
        asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NT) : "memory");
    }
}

// One score: through the read-only path (NC, for rows written before the kernel started) or from
// L2, bypassing L1 (rows the same CTA has just written, after a barrier or an mbarrier wait that
// orders the writes; volatile with a memory clobber, so the compiler keeps them after it).
template <bool NC>
__device__ __forceinline__ float ld_score(const float *p) {
    if constexpr (NC) {
        return __ldg(p);
    } else {
        float v;
        asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
        return v;
    }
}
template <bool NC>
__device__ __forceinline__ float4 ld_score4(const float4 *p) {
    if constexpr (NC) {
        return __ldg(p);
    } else {
        float4 v;
        asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                     : "l"(p)
                     : "memory");
        return v;
    }
}

// Scores s0 .. s0+L-1 of a row (keys of absent positions are 0 and masked by `valid`).
template <bool NC, int L>
__device__ __forceinline__ void load_keys(const float *__restrict__ row, int s0, int n, bool vec,
                                          uint32_t (&u)[L], uint32_t &valid) {
    if (vec && s0 + L <= n) {
        const float4 *p = (const float4 *)(row + s0);
#pragma unroll
        for (int j = 0; j < L / 4; ++j) {
            const float4 f = ld_score4<NC>(p + j);
            u[4 * j] = ordered_key(f.x);
            u[4 * j + 1] = ordered_key(f.y);
            u[4 * j + 2] = ordered_key(f.z);
            u[4 * j + 3] = ordered_key(f.w);
        }
        valid = (1u << L) - 1u;
    } else {
        valid = 0;
#pragma unroll
        for (int j = 0; j < L; ++j) {
            const bool ok = s0 + j < n;
            u[j] = ok ? ordered_key(ld_score<NC>(row + s0 + j)) : 0u;
            valid |= ok ? (1u << j) : 0u;
        }
    }
}

// The bin b of hist[0..nb) (nb a multiple of NT) holding the need-th largest key, counted from the
// top: keys in bins above b number `above` < need <= above + hist[b].  Every thread of the group
// calls it and receives {b, above, above + hist[b]} in res[0..2].  Thread t owns ceil(nb / NT)
// consecutive bins from the top (the last threads fewer or none), so the search is one group-wide scan.
template <int NT, int BAR>
__device__ __forceinline__ void find_bin_from_top(int tid, const uint32_t *hist, int nb, int need, int *res,
                                                  int *warp_sum) {
    constexpr int WARPS = NT / 32;
    const int lane = tid & 31, wid = tid >> 5;
    const int per = (nb + NT - 1) / NT, hi = nb - tid * per, lo = max(hi - per, 0);
    int mine = 0;
    for (int b = hi - 1; b >= lo; --b) mine += (int)hist[b];
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sum[wid] = incl;
    group_sync<NT, BAR>();
    int before = 0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) before += w < wid ? warp_sum[w] : 0;
    const int excl = before + incl - mine;
    if (excl < need && need <= excl + mine) {
        int cum = excl;
        for (int b = hi - 1; b >= lo; --b) {
            const int h = (int)hist[b];
            if (cum + h >= need) {
                res[0] = b;
                res[1] = cum;
                res[2] = cum + h;
                break;
            }
            cum += h;
        }
    }
    group_sync<NT, BAR>();
}

// Exact top-k of n keys (key_at(j), j in index order); idx_at(j) is the row index stored for
// entry j.  Three histogram passes (11 + 11 + 10 bits) find the k-th key T, then one ordered pass
// writes the keys above T and the first keys equal to T.  In the ordered pass each thread takes LO
// consecutive keys per step, so a group of few threads needs fewer barriers.
template <int NT, int BAR, class KeyAt, class IdxAt, int LO = 1>
__device__ __forceinline__ void radix_select_write(int tid, KeyAt key_at, IdxAt idx_at, int n, int k,
                                                   int32_t *__restrict__ out, uint32_t *hist, int *warp_gt,
                                                   int *warp_eq, int *shared3) {
    constexpr int WARPS = NT / 32;
    const int lane = tid & 31, wid = tid >> 5;
    const int &sel_bin = shared3[0], &sel_above = shared3[1];
    uint32_t prefix = 0, pmask = 0;
    int remaining = k;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int width = pass == 2 ? 10 : 11;
        const int nb = 1 << width;
        for (int b = tid; b < nb; b += NT) hist[b] = 0;
        group_sync<NT, BAR>();
        for (int s = tid; s < n; s += NT) {
            const uint32_t u = key_at(s);
            if ((u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & (nb - 1)], 1u);
        }
        group_sync<NT, BAR>();
        find_bin_from_top<NT, BAR>(tid, hist, nb, remaining, shared3, warp_eq);
        remaining -= sel_above;
        prefix |= (uint32_t)sel_bin << shift;
        pmask |= (uint32_t)(nb - 1) << shift;
        group_sync<NT, BAR>();  // sel_* are rewritten by the next pass
    }
    // prefix is now the k-th largest key T; (k - remaining) keys are above it.
    const uint32_t T = prefix;
    const int n_gt = k - remaining;
    int base_gt = 0, base_eq = 0;
    for (int s0 = 0; s0 < n; s0 += NT * LO) {
        if (base_gt >= n_gt && base_eq >= remaining) break;  // group-uniform: every slot is written
        const int s = s0 + tid * LO;
        uint32_t fg = 0, fe = 0;  // bit j: key s + j is above T / equal to T
#pragma unroll
        for (int j = 0; j < LO; ++j)
            if (s + j < n) {
                const uint32_t u = key_at(s + j);
                fg |= (u > T ? 1u : 0u) << j;
                fe |= (u == T ? 1u : 0u) << j;
            }
        const int cg = __popc(fg), ce = __popc(fe);
        int ig = cg, ie = ce;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int vg = __shfl_up_sync(0xffffffffu, ig, o), ve = __shfl_up_sync(0xffffffffu, ie, o);
            if (lane >= o) {
                ig += vg;
                ie += ve;
            }
        }
        if (lane == 31) {
            warp_gt[wid] = ig;
            warp_eq[wid] = ie;
        }
        group_sync<NT, BAR>();
        int off_gt = 0, off_eq = 0, tot_gt = 0, tot_eq = 0;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            off_gt += w < wid ? warp_gt[w] : 0;
            off_eq += w < wid ? warp_eq[w] : 0;
            tot_gt += warp_gt[w];
            tot_eq += warp_eq[w];
        }
        int rg = base_gt + off_gt + ig - cg, re = base_eq + off_eq + ie - ce;
#pragma unroll
        for (int j = 0; j < LO; ++j) {
            if ((fg >> j) & 1u) {
                if (rg < n_gt) out[rg] = idx_at(s + j);
                ++rg;
            }
            if ((fe >> j) & 1u) {
                if (re < remaining) out[n_gt + re] = idx_at(s + j);
                ++re;
            }
        }
        base_gt += tot_gt;
        base_eq += tot_eq;
        group_sync<NT, BAR>();  // warp_gt / warp_eq are rewritten by the next chunk
    }
}

// Shared memory of filter_row: the histogram, per-warp scratch and the candidate list.
struct FilterSmem {
    uint32_t *hist;     // [MAX_BINS]
    int *warp_gt;       // [NT / 32]
    int *warp_eq;       // [NT / 32]
    int *shared3;       // [3]
    uint32_t *cand;     // [cap] keys
    int32_t *cand_idx;  // [cap] row indices
    int cap;
};

// Top-k of the causal prefix row[0 .. n_live) into out[0 .. k): all keys when n_live <= k (then
// -1 padding), else two streaming passes -- an 11-bit histogram of the keys' top bits, then an
// in-order compaction of every key in or above the threshold bin into the candidate list -- and
// the exact radix select on the candidates (on the row itself when they overflow the list).
// L consecutive scores per thread per streaming step (fewer registers for smaller L).
template <int NT, int BAR, bool NC, int L = SPT>
__device__ __forceinline__ void filter_row(int tid, const float *__restrict__ row, int n_live, int k, bool vec,
                                           int32_t *__restrict__ out, const FilterSmem &sm) {
    constexpr int WARPS = NT / 32;
    const int lane = tid & 31, wid = tid >> 5;
    if (n_live <= k) {
        for (int j = tid; j < k; j += NT) out[j] = j < n_live ? j : -1;
        return;
    }
    uint32_t *hist = sm.hist;
    // ---- A: histogram of the top 11 key bits ----
    for (int b = tid; b < MAX_BINS; b += NT) hist[b] = 0;
    group_sync<NT, BAR>();
#pragma unroll 1
    for (int base = 0; base < n_live; base += NT * L) {
        uint32_t u[L], valid;
        load_keys<NC, L>(row, base + tid * L, n_live, vec, u, valid);
#pragma unroll
        for (int j = 0; j < L; ++j)
            if ((valid >> j) & 1u) atomicAdd(&hist[u[j] >> 21], 1u);
    }
    group_sync<NT, BAR>();
    find_bin_from_top<NT, BAR>(tid, hist, MAX_BINS, k, sm.shared3, sm.warp_eq);
    const uint32_t bsel = (uint32_t)sm.shared3[0];
    const int n_cand = sm.shared3[2];  // keys in the threshold bin or above
    group_sync<NT, BAR>();             // shared3 is reused by the select

    if (n_cand <= sm.cap) {
        // ---- B: compact the candidates (top bits >= bsel) in index order ----
        int base = 0;
#pragma unroll 1
        for (int s0 = 0; s0 < n_live; s0 += NT * L) {
            const int first = s0 + tid * L;
            uint32_t u[L], valid = 0;
            if (first < n_live) load_keys<NC, L>(row, first, n_live, vec, u, valid);
            uint32_t take = 0;
#pragma unroll
            for (int j = 0; j < L; ++j) take |= (((valid >> j) & 1u) && (u[j] >> 21) >= bsel) ? (1u << j) : 0u;
            const int c = __popc(take);
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (lane == 31) sm.warp_gt[wid] = incl;
            group_sync<NT, BAR>();
            int before = 0, total = 0;
#pragma unroll
            for (int w = 0; w < WARPS; ++w) {
                before += w < wid ? sm.warp_gt[w] : 0;
                total += sm.warp_gt[w];
            }
            int pos = base + before + incl - c;
#pragma unroll
            for (int j = 0; j < L; ++j)
                if ((take >> j) & 1u) {
                    sm.cand[pos] = u[j];
                    sm.cand_idx[pos] = first + j;
                    ++pos;
                }
            base += total;
            group_sync<NT, BAR>();  // warp_gt is rewritten by the next step
        }
        const uint32_t *cand = sm.cand;
        const int32_t *cidx = sm.cand_idx;
        radix_select_write<NT, BAR>(tid, [&](int j) { return cand[j]; }, [&](int j) { return cidx[j]; }, n_cand, k,
                                    out, hist, sm.warp_gt, sm.warp_eq, sm.shared3);
    } else {
        radix_select_write<NT, BAR>(tid, [&](int j) { return ordered_key(ld_score<NC>(row + j)); },
                                    [&](int j) { return j; }, n_live, k, out, hist, sm.warp_gt, sm.warp_eq,
                                    sm.shared3);
    }
}

// The r-th largest (1-based) of n keys key_at(0 .. n-1), for small n (a sample): four histogram passes
// of 8 bits, each over 256 bins, so clearing and scanning the histogram stays short.
template <int NT, int BAR, class KeyAt>
__device__ __forceinline__ uint32_t kth_largest_key(int tid, KeyAt key_at, int n, int r, uint32_t *hist,
                                                    int *warp_sum, int *shared3) {
    uint32_t prefix = 0, pmask = 0;
    int remaining = r;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int b = tid; b < 256; b += NT) hist[b] = 0;
        group_sync<NT, BAR>();
        for (int s = tid; s < n; s += NT) {
            const uint32_t u = key_at(s);
            if ((u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
        }
        group_sync<NT, BAR>();
        find_bin_from_top<NT, BAR>(tid, hist, 256, remaining, shared3, warp_sum);
        remaining -= shared3[1];
        prefix |= (uint32_t)shared3[0] << shift;
        pmask |= 255u << shift;
        group_sync<NT, BAR>();
    }
    return prefix;
}

// Compacts, in index order, the keys of row[0 .. n_live) whose ordered key is >= thr into the
// candidate list (at most sm.cap of them are stored); returns how many there are.  Each step's loads
// are issued before the previous step is compacted, so their latency hides behind its scan and
// barriers.
template <int NT, int BAR, bool NC, int L>
__device__ __forceinline__ int compact_at_least(int tid, const float *__restrict__ row, int n_live, bool vec,
                                                uint32_t thr, const FilterSmem &sm) {
    constexpr int WARPS = NT / 32;
    const int lane = tid & 31, wid = tid >> 5;
    int base = 0;
    uint32_t u[L], valid = 0;
    if (tid * L < n_live) load_keys<NC, L>(row, tid * L, n_live, vec, u, valid);
#pragma unroll 1
    for (int s0 = 0; s0 < n_live; s0 += NT * L) {
        const int first = s0 + tid * L, next = first + NT * L;
        uint32_t un[L], vn = 0;
        if (next < n_live) load_keys<NC, L>(row, next, n_live, vec, un, vn);
        uint32_t take = 0;
#pragma unroll
        for (int j = 0; j < L; ++j) take |= (((valid >> j) & 1u) && u[j] >= thr) ? (1u << j) : 0u;
        const int c = __popc(take);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) sm.warp_gt[wid] = incl;
        group_sync<NT, BAR>();
        int before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            before += w < wid ? sm.warp_gt[w] : 0;
            total += sm.warp_gt[w];
        }
        int pos = base + before + incl - c;
#pragma unroll
        for (int j = 0; j < L; ++j)
            if ((take >> j) & 1u) {
                if (pos < sm.cap) {
                    sm.cand[pos] = u[j];
                    sm.cand_idx[pos] = first + j;
                }
                ++pos;
            }
        base += total;
        group_sync<NT, BAR>();  // warp_gt is rewritten by the next step
#pragma unroll
        for (int j = 0; j < L; ++j) u[j] = un[j];
        valid = vn;
    }
    return base;
}

// The same output as filter_row, for a group of few threads that selects right after the scores
// were written (the fused indexer): a row that fits the candidate list is copied in whole; a longer
// row gets its threshold from a strided sample of SAMPLE keys -- the r-th largest sample with r a
// few standard deviations above the expected count of sampled keys among the top k -- so that one
// streaming pass (no histogram of the whole row) keeps every key at or above it.  That set holds
// the top k whenever it has at least k keys, and the exact radix select runs on it; otherwise (or
// when it overflows the list) the select runs on the whole row.
template <int NT, int BAR, bool NC, int L = SPT>
__device__ __forceinline__ void sampled_row(int tid, const float *__restrict__ row, int n_live, int k, bool vec,
                                            int32_t *__restrict__ out, const FilterSmem &sm) {
    constexpr int SAMPLE = 1024;
    if (n_live <= k) {
        for (int j = tid; j < k; j += NT) out[j] = j < n_live ? j : -1;
        return;
    }
    uint32_t thr = 0;  // every finite or -inf score maps above 0
    if (n_live > sm.cap) {
        constexpr int PER = (SAMPLE + NT - 1) / NT;
        float v[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) {  // every load in flight before the first is used
            const int j = tid + i * NT;
            v[i] = j < SAMPLE ? ld_score<NC>(row + (int)(((int64_t)j * n_live) / SAMPLE)) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < PER; ++i)
            if (tid + i * NT < SAMPLE) sm.cand[tid + i * NT] = ordered_key(v[i]);
        group_sync<NT, BAR>();
        const float mu = (float)SAMPLE * (float)k / (float)n_live;
        const int r = min(SAMPLE, (int)ceilf(mu + 4.0f * sqrtf(mu) + 8.0f));
        const uint32_t *smp = sm.cand;
        thr = kth_largest_key<NT, BAR>(tid, [&](int j) { return smp[j]; }, SAMPLE, r, sm.hist, sm.warp_eq,
                                       sm.shared3);
    }
    const int n_cand = compact_at_least<NT, BAR, NC, L>(tid, row, n_live, vec, thr, sm);
    if (n_cand >= k && n_cand <= sm.cap) {
        const uint32_t *cand = sm.cand;
        const int32_t *cidx = sm.cand_idx;
        auto key_at = [&](int j) { return cand[j]; };
        auto idx_at = [&](int j) { return cidx[j]; };
        radix_select_write<NT, BAR, decltype(key_at), decltype(idx_at), 8>(tid, key_at, idx_at, n_cand, k, out,
                                                                            sm.hist, sm.warp_gt, sm.warp_eq,
                                                                            sm.shared3);
    } else {
        auto key_at = [&](int j) { return ordered_key(ld_score<NC>(row + j)); };
        auto idx_at = [&](int j) { return j; };
        radix_select_write<NT, BAR, decltype(key_at), decltype(idx_at), 8>(tid, key_at, idx_at, n_live, k, out,
                                                                            sm.hist, sm.warp_gt, sm.warp_eq,
                                                                            sm.shared3);
    }
}

}  // namespace tk
}  // namespace dsa
