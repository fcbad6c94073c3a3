// Exact per-row top-k of the indexer scores (DeepSeek-V3.2-Exp atlas page,
// M^sel_{t,s} = M_{t,s} for s in top_k(S~^I_t)): a radix select on
// order-preserving uint32 keys.
//
// Only the causal keys 0..p are read.  If there are at most k causal keys
// they are all selected.  Otherwise three histogram passes over 11 + 11 + 10
// key bits (shared-memory histograms) find the exact k-th largest key T and
// how many keys equal to T are needed; a final ordered pass writes every key
// above T and then the first `need` keys equal to T, each in increasing key
// index, so equal scores resolve to the lower key index and the output is
// deterministic.  Every kernel below writes the same output.
//
// Three kernels for three regimes:
//   * topk_filter_kernel (many rows, e.g. prefill): one CTA per row, two
//     streaming passes (a histogram of the top 11 bits, then a compaction of
//     every key in or above the threshold bin into a shared-memory candidate
//     list); the radix select runs on the candidates.
//   * topk_cluster_kernel (few long rows, e.g. decode): a cluster of eight
//     CTAs per row, each holding a slice of the row's keys in shared memory,
//     histograms merged through distributed shared memory.
//   * topk_radix_wide_kernel (few rows too long for the cluster's shared
//     memory): 1024 threads per row, eight loads in flight per thread in the
//     histogram passes, eight consecutive keys per thread in the ordered pass,
//     the output row assembled in shared memory and written out coalesced.
#include "topk_row.cuh"

namespace dsa {
namespace {

using tk::MAX_BINS;
using tk::SPT;

// ---------------------------------------------------------------------------
// Many rows (prefill): one CTA per row, two streaming passes over the row.
//   A. 16 consecutive scores per thread per step (vector loads), an 11-bit
//      histogram of the keys' top bits (warp-aggregated shared atomics: a
//      row's scores crowd into a few exponent bins).  The bin B holding the
//      k-th largest key follows from a scan from the top.
//   B. every key whose top bits are >= B (all keys of the top k are among
//      them) is compacted, in index order, into a shared-memory candidate
//      list with its index.
// The exact radix select then runs on the candidates only.  A row whose
// candidates overflow the list (massive ties at the threshold) runs it on the
// global row instead.
// ---------------------------------------------------------------------------
constexpr int TF_THREADS = 256;
constexpr int TF_WARPS = TF_THREADS / 32;
constexpr int CAND_CAP = 8192;  // candidates per row kept in shared memory (64 KB)

__global__ void __launch_bounds__(TF_THREADS) topk_filter_kernel(const float *__restrict__ scores, int64_t ld,
                                                                 const __grid_constant__ SeqTab st, int k,
                                                                 int32_t *__restrict__ idx, int vec, int cap) {
    extern __shared__ __align__(16) uint32_t cand[];  // [cap] keys, then [cap] row indices
    __shared__ uint32_t hist[MAX_BINS];
    __shared__ int warp_gt[TF_WARPS], warp_eq[TF_WARPS];
    __shared__ int shared3[3];
    pdl_wait();  // everything below reads or writes global memory

    const int r = blockIdx.x;
    const RowInfo ri = row_info(st, r);
    const int n_live = min(ri.p + 1, ri.S);
    const tk::FilterSmem sm{hist, warp_gt, warp_eq, shared3, cand, (int32_t *)(cand + cap), cap};
    tk::filter_row<TF_THREADS, 0, true>((int)threadIdx.x, scores + (int64_t)r * ld, n_live, k, vec != 0,
                                        idx + (int64_t)r * k, sm);
}

constexpr int KPT = 8;                // consecutive keys per thread in the ordered pass
constexpr int CACHE_MAX = 48 * 1024;  // keys kept in shared memory (192 KB)

constexpr int WIDE_THREADS = 1024;         // threads per row of the wide kernel
constexpr int HB = 8;                 // keys per thread per iteration of a histogram pass

__global__ void __launch_bounds__(WIDE_THREADS, 1) topk_radix_wide_kernel(const float *__restrict__ scores, int64_t ld,
                                                             const __grid_constant__ SeqTab st, int k,
                                                             int32_t *__restrict__ idx, int cache_cap) {
    constexpr int WARPS = WIDE_THREADS / 32;
    extern __shared__ uint32_t cache[];  // [cache_cap] keys, then [k] staged output indices
    __shared__ uint32_t hist[MAX_BINS];
    __shared__ uint32_t warp_tot[2][WARPS];
    __shared__ int sel_bin, sel_above;

    pdl_wait();  // everything below reads or writes global memory
    const int r = blockIdx.x;
    const RowInfo ri = row_info(st, r);
    const int n_live = min(ri.p + 1, ri.S);
    const float *row = scores + (int64_t)r * ld;
    int32_t *out = idx + (int64_t)r * k;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

    if (n_live <= k) {
        for (int j = tid; j < k; j += WIDE_THREADS) out[j] = j < n_live ? j : -1;
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
        const uint32_t nb = 1u << width;
        for (int b = tid; b < (int)nb; b += WIDE_THREADS) hist[b] = 0;
        __syncthreads();
        // HB loads in flight per thread before their atomics: uncached rows read global memory,
        // and one dependent round trip per key would bound the pass by latency.
#pragma unroll 1
        for (int s0 = 0; s0 < n_live; s0 += HB * WIDE_THREADS) {
            uint32_t u[HB];
#pragma unroll
            for (int j = 0; j < HB; ++j) {
                const int s = s0 + j * WIDE_THREADS + tid;
                u[j] = 0;
                if (s < n_live) {
                    if (pass == 0) {
                        u[j] = ordered_key(row[s]);
                        if (cached) cache[s] = u[j];
                    } else {
                        u[j] = key_at(s);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < HB; ++j) {
                const int s = s0 + j * WIDE_THREADS + tid;
                if (s < n_live && (u[j] & pmask) == prefix) atomicAdd(&hist[(u[j] >> shift) & (nb - 1)], 1u);
            }
        }
        __syncthreads();
        if (wid == 0) {
            // Lane l owns the bins [nb - (l+1)*per, nb - l*per), scanned from the top.
            const int per = (int)nb / 32;
            const int hi = (int)nb - lane * per;
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
        pmask |= (nb - 1) << shift;
        __syncthreads();  // sel_* are rewritten by the next pass
    }

    // prefix is now the k-th largest key T; (k - remaining) keys are above it.
    const uint32_t T = prefix;
    const int n_gt = k - remaining;
    // Rows that are not cached stage each chunk of keys in the (unused) cache
    // so that a thread can read 8 consecutive ones.  The output row is
    // assembled in shared memory and written out coalesced at the end.
    uint32_t *stage = cache;
    int32_t *out_s = (int32_t *)(cache + cache_cap);
    int base_gt = 0, base_eq = 0;
#pragma unroll 1
    for (int c = 0, s0 = 0; s0 < n_live; ++c, s0 += KPT * WIDE_THREADS) {
        if (!cached) {
            __syncthreads();  // the previous chunk's reads of the staging area are done
            for (int j = 0; j < KPT; ++j) {
                const int s = s0 + j * WIDE_THREADS + tid;
                stage[j * WIDE_THREADS + tid] = s < n_live ? ordered_key(row[s]) : 0u;
            }
            __syncthreads();
        }
        const int first = s0 + tid * KPT;
        const uint32_t *src = cached ? cache + first : stage + tid * KPT;  // 32-byte aligned
        uint32_t u[KPT];
        if (first + KPT <= n_live) {
            const uint4 a = ((const uint4 *)src)[0], b = ((const uint4 *)src)[1];
            u[0] = a.x, u[1] = a.y, u[2] = a.z, u[3] = a.w, u[4] = b.x, u[5] = b.y, u[6] = b.z, u[7] = b.w;
        } else {
#pragma unroll
            for (int j = 0; j < KPT; ++j) u[j] = first + j < n_live ? src[j] : 0u;
        }
        int g = 0, e = 0;
#pragma unroll
        for (int j = 0; j < KPT; ++j) {
            const bool valid = first + j < n_live;
            g += valid && u[j] > T;
            e += valid && u[j] == T;
        }
        // block-wide exclusive prefix of (g, e), packed as g + e * 2^16
        const uint32_t mine = (uint32_t)g | ((uint32_t)e << 16);
        uint32_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        uint32_t *wt = warp_tot[c & 1];
        if (lane == 31) wt[wid] = incl;
        __syncthreads();
        uint32_t before = 0, total = 0;
        for (int w = 0; w < WARPS; ++w) {
            const uint32_t v = wt[w];
            before += w < wid ? v : 0u;
            total += v;
        }
        const uint32_t excl = before + incl - mine;
        int rg = base_gt + (int)(excl & 0xffffu), re = base_eq + (int)(excl >> 16);
#pragma unroll
        for (int j = 0; j < KPT; ++j) {
            const int s = first + j;
            if (s < n_live && u[j] > T) {
                if (rg < n_gt) out_s[rg] = s;
                ++rg;
            } else if (s < n_live && u[j] == T) {
                if (re < remaining) out_s[n_gt + re] = s;
                ++re;
            }
        }
        base_gt += (int)(total & 0xffffu);
        base_eq += (int)(total >> 16);
        if (base_gt >= n_gt && base_eq >= remaining) break;  // block-uniform: every slot is written
    }
    __syncthreads();
    for (int j = tid; j < k; j += WIDE_THREADS) out[j] = out_s[j];
}

// ---------------------------------------------------------------------------
// Few long rows (decode): a cluster of CL CTAs per row.  CTA c takes the c-th
// contiguous slice of the row's causal keys and keeps its keys in shared
// memory.  Each radix pass builds a per-CTA histogram; after a cluster
// barrier every CTA sums the CL histograms through distributed shared memory
// and makes the same bin decision.  The final pass counts each slice's keys
// above / equal to the threshold, exchanges the counts, and every CTA writes
// its own keys at their ranks in index order: the output is the same as the
// one-CTA kernels'.
// ---------------------------------------------------------------------------
constexpr int CL = 8;              // CTAs per row
constexpr int LONG_ROW = 8192;     // causal keys from which a few rows take the cluster kernel
constexpr int CT = 256;            // threads per CTA
constexpr int CT_WARPS = CT / 32;

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t peer_addr(const void *local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(r)
                 : "r"((uint32_t)__cvta_generic_to_shared(local)), "r"(rank));
    return r;
}
__device__ __forceinline__ uint4 ld_peer_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(CT)
    topk_cluster_kernel(const float *__restrict__ scores, int64_t ld, const __grid_constant__ SeqTab st, int k,
                        int32_t *__restrict__ idx) {
    extern __shared__ __align__(16) uint32_t slice[];  // this CTA's keys
    __shared__ __align__(16) uint32_t hist[2][MAX_BINS];
    __shared__ __align__(16) uint32_t merged[MAX_BINS];
    __shared__ __align__(16) uint32_t counts[4];       // (above, equal) of this slice
    __shared__ uint32_t warp_tot[2][CT_WARPS];
    __shared__ int sel[3], warp_sum[CT_WARPS];

    pdl_wait();  // everything below reads or writes global memory
    const int r = blockIdx.x / CL;
    const uint32_t c = cluster_ctarank();
    const RowInfo ri = row_info(st, r);
    const int n_live = min(ri.p + 1, ri.S);
    const float *row = scores + (int64_t)r * ld;
    int32_t *out = idx + (int64_t)r * k;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid < 4) counts[tid] = 0;  // ordered before the final pass's atomics by the passes' barriers

    if (n_live <= k) {  // the whole cluster takes this branch: no cluster barrier is pending
        if (c == 0)
            for (int j = tid; j < k; j += CT) out[j] = j < n_live ? j : -1;
        return;
    }
    const int s_lo = (int)((int64_t)c * n_live / CL), n = (int)((int64_t)(c + 1) * n_live / CL) - s_lo;

    uint32_t prefix = 0, pmask = 0;
    int remaining = k;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int width = pass == 2 ? 10 : 11;
        const uint32_t nb = 1u << width;
        uint32_t *h = hist[pass & 1];
        for (int b = tid; b < (int)nb; b += CT) h[b] = 0;
        __syncthreads();
        if (pass == 0) {
#pragma unroll 1
            for (int s0 = 0; s0 < n; s0 += 2 * HB * CT) {
                uint32_t u[2 * HB];
#pragma unroll
                for (int j = 0; j < 2 * HB; ++j) {
                    const int s = s0 + j * CT + tid;
                    u[j] = s < n ? ordered_key(row[s_lo + s]) : 0u;
                }
#pragma unroll
                for (int j = 0; j < 2 * HB; ++j) {
                    const int s = s0 + j * CT + tid;
                    if (s < n) {
                        slice[s] = u[j];
                        atomicAdd(&h[u[j] >> shift], 1u);
                    }
                }
            }
        } else {
            for (int s = tid; s < n; s += CT) {
                const uint32_t u = slice[s];
                if ((u & pmask) == prefix) atomicAdd(&h[(u >> shift) & (nb - 1)], 1u);
            }
        }
        // Every CTA's histogram of this pass is complete (and the previous pass's reads of
        // the other buffer are done) once the whole cluster has arrived.
        cluster_barrier();
        for (int q4 = tid; q4 < (int)nb / 4; q4 += CT) {
            uint4 acc = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int cc = 0; cc < CL; ++cc) {
                const uint4 v = ld_peer_v4(peer_addr(h + 4 * q4, (uint32_t)cc));
                acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
            }
            *(uint4 *)(merged + 4 * q4) = acc;
        }
        __syncthreads();
        tk::find_bin_from_top<CT, 0>(tid, merged, (int)nb, remaining, sel, warp_sum);
        remaining -= sel[1];
        prefix |= (uint32_t)sel[0] << shift;
        pmask |= (nb - 1) << shift;
        __syncthreads();  // sel[] and merged[] are rewritten by the next pass
    }

    // prefix is now the k-th largest key T of the row; (k - remaining) keys are above it.
    const uint32_t T = prefix;
    const int n_gt = k - remaining;
    {
        uint32_t g = 0, e = 0;
        for (int s = tid; s < n; s += CT) {
            g += slice[s] > T;
            e += slice[s] == T;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            g += __shfl_xor_sync(0xffffffffu, g, o);
            e += __shfl_xor_sync(0xffffffffu, e, o);
        }
        if (lane == 0) {
            atomicAdd(&counts[0], g);
            atomicAdd(&counts[1], e);
        }
    }
    __syncthreads();
    cluster_barrier();
    // ranks of this slice's first key above / equal to T among the row's keys
    int base_gt = 0, base_eq = 0;
    for (uint32_t cc = 0; cc < c; ++cc) {
        const uint4 v = ld_peer_v4(peer_addr(counts, cc));
        base_gt += (int)v.x;
        base_eq += (int)v.y;
    }
    // No CTA may leave while another can still read its counts.
    cluster_barrier();
#pragma unroll 1
    for (int ch = 0, s0 = 0; s0 < n; ++ch, s0 += KPT * CT) {
        if (base_gt >= n_gt && base_eq >= remaining) break;  // block-uniform: nothing left to place
        const int first = s0 + tid * KPT;
        uint32_t u[KPT];
#pragma unroll
        for (int j = 0; j < KPT; ++j) u[j] = first + j < n ? slice[first + j] : 0u;
        int g = 0, e = 0;
#pragma unroll
        for (int j = 0; j < KPT; ++j) {
            const bool valid = first + j < n;
            g += valid && u[j] > T;
            e += valid && u[j] == T;
        }
        // block-wide exclusive prefix of (g, e), packed as g + e * 2^16
        const uint32_t mine = (uint32_t)g | ((uint32_t)e << 16);
        uint32_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        uint32_t *wt = warp_tot[ch & 1];
        if (lane == 31) wt[wid] = incl;
        __syncthreads();
        uint32_t before = 0, total = 0;
        for (int w = 0; w < CT_WARPS; ++w) {
            const uint32_t v = wt[w];
            before += w < wid ? v : 0u;
            total += v;
        }
        const uint32_t excl = before + incl - mine;
        int rg = base_gt + (int)(excl & 0xffffu), re = base_eq + (int)(excl >> 16);
#pragma unroll
        for (int j = 0; j < KPT; ++j) {
            const int s = first + j;
            if (s < n && u[j] > T) {
                if (rg < n_gt) out[rg] = s_lo + s;
                ++rg;
            } else if (s < n && u[j] == T) {
                if (re < remaining) out[n_gt + re] = s_lo + s;
                ++re;
            }
        }
        base_gt += (int)(total & 0xffffu);
        base_eq += (int)(total >> 16);
    }
}

// The selection of rows that see at most k keys, written without scores: every causal key in
// ascending order, then -1 (what the top-k writes for such rows).  One CTA per row.
__global__ void __launch_bounds__(256) dense_idx_kernel(SeqTab st, int k, int32_t *__restrict__ idx) {
    pdl_wait();
    const int r = blockIdx.x;
    const RowInfo ri = row_info(st, r);
    const int n_live = min(ri.p + 1, ri.S);
    int32_t *out = idx + (int64_t)r * k;
    for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = j < n_live ? j : -1;
}

}  // namespace

cudaError_t launch_dense_idx(const SeqTab &st, int total_q, int k, int32_t *idx, cudaStream_t s) {
    if (total_q == 0) return cudaSuccess;
    cudaError_t e = launch_pdl(dense_idx_kernel, dim3(total_q), dim3(256), 0, s, st, k, idx);
    if (e != cudaSuccess) return e;
    note_launch(DSA_KERNEL_DENSE_IDX);
    return cudaGetLastError();
}

cudaError_t launch_topk(const float *scores, int64_t ld, const SeqTab &st, int total_q, int k, int32_t *idx,
                        cudaStream_t s) {
    if (total_q == 0) return cudaSuccess;
    int max_live = 0;  // the longest causal row of the launch
    for (int b = 0; b < st.B; ++b) {
        const int T = st.q_off[b + 1] - st.q_off[b];
        if (T > 0) max_live = max(max_live, min(st.start_pos[b] + T, st.k_len[b]));
    }
    cudaError_t e;
    // Few long rows (decode): a cluster of CTAs per row when each CTA's slice fits its shared
    // memory; rows too long for that take the wide kernel.  Many rows, or short ones (where a
    // cluster's barriers cost more than they save), take the filter kernel.
    const int slice_cap = (max_live + CL - 1) / CL;
    const bool few_long = total_q < 2 * 152 && max_live >= LONG_ROW && max_live > k;
    if (few_long && slice_cap <= 48 * 1024) {
        const size_t smem = (size_t)slice_cap * sizeof(uint32_t);
        e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) e = launch_pdl(topk_cluster_kernel, dim3(total_q * CL), dim3(CT), smem, s, scores, ld, st, k, idx);
    } else if (few_long) {
        // Few rows longer than the cluster's cache: the wide kernel.  Its dynamic shared memory (200 KB) holds the key cache (at
        // least one chunk: it is also the staging area of the ordered pass for longer rows) and
        // the staged output row.
        constexpr int words = 50 * 1024, chunk = KPT * WIDE_THREADS;
        if (max_live > k && k + chunk > words) return cudaErrorInvalidValue;
        const int cap = max_live <= k ? 0 : max(min(max_live, min(CACHE_MAX, words - k)), chunk);
        const size_t smem = ((size_t)cap + (size_t)k) * sizeof(uint32_t);
        e = cudaFuncSetAttribute(topk_radix_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = launch_pdl(topk_radix_wide_kernel, dim3(total_q), dim3(WIDE_THREADS), smem, s, scores, ld, st, k, idx, cap);
    } else {
        // Many rows: two streaming passes per row and a shared-memory candidate list as long as
        // the longest row (at most CAND_CAP), so that short rows keep more CTAs per SM.
        const int cap = std::max(64, std::min(CAND_CAP, (max_live + 63) / 64 * 64));
        const size_t smem = (size_t)cap * 2 * sizeof(uint32_t);
        const int vec = ((uintptr_t)scores % 16 == 0 && ld % 4 == 0) ? 1 : 0;
        e = cudaFuncSetAttribute(topk_filter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = launch_pdl(topk_filter_kernel, dim3(total_q), dim3(TF_THREADS), smem, s, scores, ld, st, k, idx, vec, cap);
    }
    if (e != cudaSuccess) return e;
    note_launch(DSA_KERNEL_TOPK);
    return cudaGetLastError();
}

}  // namespace dsa
