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

struct SelectSmem {
    uint32_t hist[256];
    int scan[136];
    uint32_t digit, above;
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

// keys[0..n) (score_key values) -> out[0..k_eff) ascending page ids. out may be shared or
// global memory. Returns k_eff. Every thread of the block must call it.
static __device__ __noinline__ int block_select(const uint32_t* keys, int n, int k, int* out, SelectSmem& sm) {
    const int k_eff = min(k, n);
    const int nthr = blockDim.x;
    if (k_eff <= 0) return 0;
    if (k_eff >= n) {
        for (int i = threadIdx.x; i < n; i += nthr) out[i] = i;
        __syncthreads();
        return k_eff;
    }
    const bool ranks = n <= 2 * nthr;
    uint32_t T = 0;
    int k_rem = 0;
    if (!ranks) {
        uint32_t prefix = 0, mask = 0;
        k_rem = k_eff;
#pragma unroll 1
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            for (int i = threadIdx.x; i < 256; i += nthr) sm.hist[i] = 0;
            __syncthreads();
            for (int i = threadIdx.x; i < n; i += nthr) {
                const uint32_t key = keys[i];
                if ((key & mask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 0xFF], 1u);
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
            __syncthreads();
        }
        T = prefix;
    }
    int base_sel = 0, base_eq = 0;
    for (int start = 0; start < n; start += nthr) {
        const int i = start + threadIdx.x;
        int sel = 0, eq = 0;
        if (i < n) {
            const uint32_t ki = keys[i];
            if (ranks) {
                int rank = 0;
                for (int j = 0; j < n; ++j) {
                    const uint32_t kj = keys[j];
                    rank += (kj > ki) || (kj == ki && j < i);
                }
                sel = rank < k_eff;
            } else {
                sel = ki > T;
                eq = ki == T;
            }
        }
        if (!ranks) {
            int t_eq;
            const int e_eq = block_excl_scan(eq, t_eq, sm.scan);
            sel = sel || (eq && (base_eq + e_eq) < k_rem);
            base_eq += t_eq;
        }
        int t_sel;
        const int e_sel = block_excl_scan(sel, t_sel, sm.scan);
        if (sel) out[base_sel + e_sel] = i;
        base_sel += t_sel;
    }
    __syncthreads();
    return k_eff;
}

}  // namespace smx
