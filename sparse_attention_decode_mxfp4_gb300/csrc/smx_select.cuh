// smx_select.cuh -- block-wide selection of the k_eff best pages of a row (a4).
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "MXFP4 main KV": the
// selected blocks fill the row's sparse table. Order: larger score first, ties to the lower page
// id, NaN last (score_key); the result is the selected page ids in ascending order.
// Small rows (n <= 2 x threads) rank every page against all others; larger rows use a 4-pass
// 8-bit radix select for the k_eff-th key, then take every page above it and the lowest-id
// pages equal to it. Either way one block-wide scan in page-id order writes the list.
#pragma once

#include "smx_device.cuh"

namespace smx {

constexpr int kRankMax = 512;   // rows up to this many pages select by counting

struct SelectSmem {
    int rank[kRankMax];
    uint32_t hist[256];
    int scan[136];
    uint32_t digit, above, in_bin;
};

// Block-wide exclusive scan of one counter; returns the block total. All threads call.
__device__ __forceinline__ int block_excl_scan(int v, int& total, int* sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += x;
    }
    if (lane == 31) sm[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < nw ? sm[lane] : 0;
        int s = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xFFFFFFFFu, s, o);
            if (lane >= o) s += x;
        }
        if (lane < nw) sm[64 + lane] = s - w;
        if (lane == 31) sm[128] = s;
    }
    __syncthreads();
    const int ex = sm[64 + warp] + inc - v;
    total = sm[128];
    __syncthreads();
    return ex;
}

// keys[0..n) (score_key values in shared memory) -> out[0..k_eff) ascending page ids. out may be
// shared or global memory. Returns k_eff. Every thread of the block must call it.
// An 8-bit radix select walks the key bits from the top: each pass histograms the keys that share
// the bits decided so far, finds the bin holding the k_eff-th key, and stops early once that bin
// is taken whole. Selected = keys above the decided prefix, plus the lowest-id keys equal to it.
static __device__ __forceinline__ int block_select(const uint32_t* keys, int n, int k, int* out, SelectSmem& sm) {
    const int k_eff = min(k, n);
    const int nthr = blockDim.x;
    if (k_eff <= 0) return 0;
    if (k_eff >= n) {
        for (int i = threadIdx.x; i < n; i += nthr) out[i] = i;
        __syncthreads();
        return k_eff;
    }
    if (n <= kRankMax) {
        // small rows: rank of each page = pages with a larger (key, lower id) pair; the comparisons
        // of a page are split in `parts` slices over the threads and added in shared memory
        const int parts = max(1, nthr / n);
        for (int q = threadIdx.x; q < n; q += nthr) sm.rank[q] = 0;
        __syncthreads();
        for (int idx = threadIdx.x; idx < n * parts; idx += nthr) {
            const int i = idx % n, part = idx / n;
            const uint64_t ki = ((uint64_t)keys[i] << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)i);
            const int j0 = part * n / parts, j1 = (part + 1) * n / parts;
            int r = 0;
#pragma unroll 8
            for (int j = j0; j < j1; ++j) {
                const uint64_t kj = ((uint64_t)keys[j] << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)j);
                r += kj > ki;
            }
            if (parts > 1) atomicAdd(&sm.rank[i], r);
            else sm.rank[i] = r;
        }
        __syncthreads();
        // compaction in id order: thread u owns ids [u * per, (u + 1) * per)
        const int per = (n + nthr - 1) / nthr;
        const int i0 = threadIdx.x * per, i1 = min(i0 + per, n);
        int cnt = 0;
        for (int q = i0; q < i1; ++q) cnt += sm.rank[q] < k_eff;
        int total;
        int pos = block_excl_scan(cnt, total, sm.scan);
        for (int q = i0; q < i1; ++q)
            if (sm.rank[q] < k_eff) out[pos++] = q;
        __syncthreads();
        return k_eff;
    }
    uint32_t prefix = 0, mask = 0;
    int k_rem = k_eff;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < 256; i += nthr) sm.hist[i] = 0;
        __syncthreads();
        // warp-aggregated: lanes that fall in the same bin add once (scores crowd a few bins)
        const int n_warp = (n + 31) & ~31;
        for (int i = threadIdx.x; i < n_warp; i += nthr) {
            const uint32_t key = i < n ? keys[i] : 0u;
            const bool in = i < n && (key & mask) == prefix;
            const uint32_t bin = in ? (key >> shift) & 0xFF : 0x100u;
            const unsigned peers = __match_any_sync(0xFFFFFFFFu, bin);
            if (in && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&sm.hist[bin], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            uint32_t c[8], lsum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) { c[i] = sm.hist[255 - 8 * lane - i]; lsum += c[i]; }
            uint32_t incl = lsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += x;
            }
            const uint32_t excl = incl - lsum;
            if (excl < (uint32_t)k_rem && incl >= (uint32_t)k_rem) {
                uint32_t run = excl;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (run + c[i] >= (uint32_t)k_rem) {
                        sm.digit = 255 - 8 * lane - i;
                        sm.above = run;
                        sm.in_bin = c[i];
                        break;
                    }
                    run += c[i];
                }
            }
        }
        __syncthreads();
        prefix |= sm.digit << shift;
        mask |= 0xFFu << shift;
        k_rem -= (int)sm.above;
        const bool whole_bin = (int)sm.in_bin == k_rem;
        __syncthreads();
        if (whole_bin) break;
    }
    // compaction in page-id order: thread u owns up to 32 consecutive ids of a chunk
    int base_sel = 0, base_eq = 0;
    const int chunk = nthr * 32;
    for (int c0 = 0; c0 < n; c0 += chunk) {
        const int per = (min(chunk, n - c0) + nthr - 1) / nthr;
        const int i0 = c0 + threadIdx.x * per;
        const int i1 = min(i0 + per, n);
        uint32_t gt_bits = 0, eq_bits = 0;
        for (int i = i0; i < i1; ++i) {
            const uint32_t key = keys[i] & mask;
            gt_bits |= (uint32_t)(key > prefix) << (i - i0);
            eq_bits |= (uint32_t)(key == prefix) << (i - i0);
        }
        int t_eq;
        const int e_eq = block_excl_scan(__popc(eq_bits), t_eq, sm.scan);
        int taken = 0;
        uint32_t sel_bits = gt_bits;
        for (int i = i0; i < i1; ++i) {
            if ((eq_bits >> (i - i0)) & 1u) {
                if (base_eq + e_eq + taken < k_rem) sel_bits |= 1u << (i - i0);
                ++taken;
            }
        }
        int t_sel;
        int pos = base_sel + block_excl_scan(__popc(sel_bits), t_sel, sm.scan);
        for (int i = i0; i < i1; ++i)
            if ((sel_bits >> (i - i0)) & 1u) out[pos++] = i;
        base_sel += t_sel;
        base_eq += t_eq;
    }
    __syncthreads();
    return k_eff;
}

}  // namespace smx
