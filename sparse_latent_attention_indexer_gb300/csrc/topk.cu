// Exact per-row top-k of the indexer scores (DeepSeek-V3.2-Exp atlas page,
// M^sel_{t,s} = M_{t,s} for s in top_k(S~^I_t)): a radix select on
// order-preserving uint32 keys.
//
// One CTA per query row.  Only the causal keys 0..p are read, once: the first
// pass converts them to keys and keeps them in shared memory when the row fits
// the launch's cache (rows longer than that re-read global memory).  If there
// are at most k causal keys they are all selected.  Otherwise three histogram passes
// over 11 + 11 + 10 key bits (shared-memory histograms, atomics) find the
// exact k-th largest key T and how many keys equal to T are needed; a final
// ordered pass compacts, in increasing key order, every key above T and then
// the first `need` keys equal to T (warp ballots + a block-wide prefix sum),
// so equal scores resolve to the lower key index and the output is
// deterministic.
#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int TK_THREADS = 512;
constexpr int TK_WARPS = TK_THREADS / 32;
constexpr int MAX_BINS = 2048;

__global__ void __launch_bounds__(TK_THREADS) topk_radix_kernel(const float *__restrict__ scores, int64_t ld,
                                                                const __grid_constant__ SeqTab st, int k,
                                                                int32_t *__restrict__ idx, int cache_cap) {
    extern __shared__ uint32_t cache[];
    __shared__ uint32_t hist[MAX_BINS];
    __shared__ int warp_gt[TK_WARPS], warp_eq[TK_WARPS];
    __shared__ int tot_gt, tot_eq;
    __shared__ int sel_bin, sel_above;

    const int r = blockIdx.x;
    const RowInfo ri = row_info(st, r);
    const int n_live = min(ri.p + 1, ri.S);
    const float *row = scores + (int64_t)r * ld;
    int32_t *out = idx + (int64_t)r * k;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

    if (n_live <= k) {
        for (int j = tid; j < k; j += TK_THREADS) out[j] = j < n_live ? j : -1;
        return;
    }

    const bool cached = n_live <= cache_cap;
    auto key_at = [&](int s) -> uint32_t { return cached ? cache[s] : ordered_key(row[s]); };
    uint32_t prefix = 0, pmask = 0;
    int remaining = k;  // keys still to take among those matching the prefix
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int width = pass == 2 ? 10 : 11;
        const int nb = 1 << width;
        for (int b = tid; b < nb; b += TK_THREADS) hist[b] = 0;
        __syncthreads();
        if (pass == 0) {
            for (int s = tid; s < n_live; s += TK_THREADS) {
                const uint32_t u = ordered_key(row[s]);
                if (cached) cache[s] = u;
                atomicAdd(&hist[u >> shift], 1u);
            }
        } else {
            for (int s = tid; s < n_live; s += TK_THREADS) {
                const uint32_t u = key_at(s);
                if ((u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & (nb - 1)], 1u);
            }
        }
        __syncthreads();
        if (wid == 0) {
            // Lane l owns the bins [nb - (l+1)*per, nb - l*per), scanned from the top.
            const int per = nb / 32;
            const int hi = nb - lane * per;
            int mine = 0;
            for (int b = hi - 1; b >= hi - per; --b) mine += (int)hist[b];
            int incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            const int excl = incl - mine;
            if (excl < remaining && remaining <= incl) {
                int cum = excl;
                for (int b = hi - 1; b >= hi - per; --b) {
                    const int h = (int)hist[b];
                    if (cum + h >= remaining) {
                        sel_bin = b;
                        sel_above = cum;
                        break;
                    }
                    cum += h;
                }
            }
        }
        __syncthreads();
        remaining -= sel_above;
        prefix |= (uint32_t)sel_bin << shift;
        pmask |= (uint32_t)(nb - 1) << shift;
        __syncthreads();  // sel_* are rewritten by the next pass
    }

    // prefix is now the k-th largest key T; (k - remaining) keys are above it.
    const uint32_t T = prefix;
    const int n_gt = k - remaining;
    int base_gt = 0, base_eq = 0;
    for (int s0 = 0; s0 < n_live; s0 += TK_THREADS) {
        const int s = s0 + tid;
        const uint32_t u = s < n_live ? key_at(s) : 0u;
        const bool gt = s < n_live && u > T;
        const bool eq = s < n_live && u == T;
        const uint32_t bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
        const uint32_t lt_mask = (1u << lane) - 1u;
        if (lane == 0) {
            warp_gt[wid] = __popc(bg);
            warp_eq[wid] = __popc(be);
        }
        __syncthreads();
        if (wid == 0) {
            int g = lane < TK_WARPS ? warp_gt[lane] : 0, e = lane < TK_WARPS ? warp_eq[lane] : 0;
            int gi = g, ei = e;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int vg = __shfl_up_sync(0xffffffffu, gi, o), ve = __shfl_up_sync(0xffffffffu, ei, o);
                if (lane >= o) { gi += vg; ei += ve; }
            }
            if (lane < TK_WARPS) {
                warp_gt[lane] = gi - g;
                warp_eq[lane] = ei - e;
            }
            if (lane == 31) {
                tot_gt = gi;
                tot_eq = ei;
            }
        }
        __syncthreads();
        if (gt) {
            const int rank = base_gt + warp_gt[wid] + __popc(bg & lt_mask);
            if (rank < n_gt) out[rank] = s;
        }
        if (eq) {
            const int rank = base_eq + warp_eq[wid] + __popc(be & lt_mask);
            if (rank < remaining) out[n_gt + rank] = s;
        }
        base_gt += tot_gt;
        base_eq += tot_eq;
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_topk(const float *scores, int64_t ld, const SeqTab &st, int total_q, int k, int32_t *idx,
                        cudaStream_t s) {
    if (total_q == 0) return cudaSuccess;
    // Shared-memory key cache: the longest causal row of the launch, at most 32768 keys (128 KB).
    int max_live = 0;
    for (int b = 0; b < st.B; ++b) {
        const int T = st.q_off[b + 1] - st.q_off[b];
        if (T > 0) max_live = max(max_live, min(st.start_pos[b] + T, st.k_len[b]));
    }
    const int cap = max_live <= k ? 0 : min(max_live, 32768);
    const size_t smem = (size_t)cap * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(topk_radix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    topk_radix_kernel<<<total_q, TK_THREADS, smem, s>>>(scores, ld, st, k, idx, cap);
    note_launch(DSA_KERNEL_TOPK);
    return cudaGetLastError();
}

}  // namespace dsa
