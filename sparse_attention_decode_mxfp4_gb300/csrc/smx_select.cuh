// smx_select.cuh -- block-wide selection of the k_eff best pages of a row (a4).
//
// [ATOM-2812] "Mono decode over the MXFP4 KV and index caches", commit "MXFP4 main KV": the
// selected blocks fill the row's sparse table. Order: larger score first, ties to the lower page
// id, NaN last (score_key); the result is the selected page ids in ascending order.
//
// Rows of at most kSelThreads pages rank every page by counting the pages that beat it. Longer
// rows: radix select over the 32-bit order-preserving keys, for a block of kSelThreads threads:
//  * bits that every key shares are skipped (block-wide AND / OR of the keys);
//  * each pass histograms the next 11 undecided bits of the keys that match the decided prefix
//    (2048 bins, shared-memory atomics), then each thread adds 8 bins and a block scan from the
//    top bin down finds the bin that holds the k_eff-th key; the pass stops early once that bin is
//    taken whole;
//  * warp w owns the contiguous page ids [32 R w, 32 R (w + 1)); a single block scan of the
//    warps' packed (above, equal) counts places every selected id, so the list comes out in
//    ascending id order: all keys above the decided prefix, plus the lowest-id keys equal to it.
#pragma once

#include "smx_device.cuh"

namespace smx {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;

struct SelectSmem {
    __align__(16) uint32_t hist[kSelWarps][256];   // also the (key, ~id) pairs of rows up to 256 pages
    uint32_t wsum[2][kSelWarps];
    uint32_t wred[2][kSelWarps];
    uint32_t digit, above, in_bin;
};

// Inclusive block scan of one value per thread (kSelThreads threads). `slot` picks one of two
// scratch rows so that back-to-back scans need a single barrier each.
__device__ __forceinline__ uint32_t sel_block_incl_scan(uint32_t v, SelectSmem& sm, int slot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += x;
    }
    if (lane == 31) sm.wsum[slot][warp] = inc;
    __syncthreads();
    uint32_t before = 0;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) before += (w < warp) ? sm.wsum[slot][w] : 0u;
    return before + inc;
}

// keys[i] = score_key(row[i]) for i < n (shared memory), every thread of a kSelThreads-thread
// block; up to 8 loads per thread are in flight together (CG: read through L2). No barrier.
template <bool CG>
__device__ __forceinline__ void load_keys(uint32_t* keys, const float* row, int n) {
    for (int base = 0; base < n; base += 8 * kSelThreads) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = base + (int)threadIdx.x + k * kSelThreads;
            v[k] = i < n ? (CG ? ldg_cg_f32(row + i) : row[i]) : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = base + (int)threadIdx.x + k * kSelThreads;
            if (i < n) keys[i] = score_key(v[k]);
        }
    }
}

// keys[0..n) (score_key values, shared memory) -> out[0..k_eff) ascending page ids (shared or
// global memory). Returns k_eff = min(k, n). Every thread of a kSelThreads-thread block calls it;
// keys must be 16-byte aligned.
static __device__ __forceinline__ int block_select(const uint32_t* keys, int n, int k, int* out, SelectSmem& sm) {
    const int k_eff = min(k, n);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (k_eff <= 0) return 0;
    if (k_eff >= n) {
        for (int i = tid; i < n; i += kSelThreads) out[i] = i;
        __syncthreads();
        return k_eff;
    }
    if (n <= kSelThreads) {
        // rank of a page = the pages that beat it (a larger key, or an equal key and a lower id),
        // counted against every page's 64-bit (key, ~id) pair; rows of up to kSelThreads / 2 pages
        // split each page's comparisons over two adjacent threads. The pages of rank < k_eff are
        // written at their id-order position (warp ballots, one barrier).
        uint64_t* k64 = reinterpret_cast<uint64_t*>(&sm.hist[0][0]);   // n <= 256 pairs fit
        if (tid < n) k64[tid] = ((uint64_t)keys[tid] << 32) | (0xFFFFFFFFu - (uint32_t)tid);
        __syncthreads();
        const bool two = n <= kSelThreads / 2;
        const int i = two ? tid >> 1 : tid;                  // this thread's page
        const int j0 = two ? (tid & 1) * (n >> 1) : 0;      // its share of the comparisons
        const int j1 = two ? ((tid & 1) ? n : n >> 1) : n;
        int rank = 0;
        if (i < n) {
            const uint64_t ki = k64[i];
            const ulonglong2* k2 = reinterpret_cast<const ulonglong2*>(k64);
            int j = j0;
            if (j & 1) rank += k64[j++] > ki;
#pragma unroll 4
            for (; j + 1 < j1; j += 2) {
                const ulonglong2 v = k2[j >> 1];
                rank += v.x > ki;
                rank += v.y > ki;
            }
            if (j < j1) rank += k64[j] > ki;
        }
        if (two) rank += __shfl_xor_sync(0xFFFFFFFFu, rank, 1);
        const bool take = i < n && rank < k_eff && (!two || (tid & 1) == 0);
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, take);
        if (lane == 0) sm.wsum[0][warp] = __popc(bal);
        __syncthreads();
        int pos = __popc(bal & ((1u << lane) - 1u));
#pragma unroll
        for (int w = 0; w < kSelWarps; ++w) pos += (w < warp) ? (int)sm.wsum[0][w] : 0;
        if (take) out[pos] = i;
        __syncthreads();
        return k_eff;
    }
    const int R = (n + kSelThreads - 1) / kSelThreads;   // ids per thread

    // bits shared by every key are decided already
    uint32_t k_and = 0xFFFFFFFFu, k_or = 0u;
    for (int i = tid; i < n; i += kSelThreads) {
        const uint32_t key = keys[i];
        k_and &= key;
        k_or |= key;
    }
    k_and = __reduce_and_sync(0xFFFFFFFFu, k_and);
    k_or = __reduce_or_sync(0xFFFFFFFFu, k_or);
    if (lane == 0) {
        sm.wred[0][warp] = k_and;
        sm.wred[1][warp] = k_or;
    }
    __syncthreads();
    k_and = 0xFFFFFFFFu;
    k_or = 0u;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
        k_and &= sm.wred[0][w];
        k_or |= sm.wred[1][w];
    }
    const uint32_t differ = k_and ^ k_or;
    int top = differ ? 31 - __clz(differ) : -1;            // highest undecided bit
    uint32_t mask = top < 0 ? 0xFFFFFFFFu : ~((2u << top) - 1u);   // the bits above it
    uint32_t prefix = k_and & mask;
    int k_rem = k_eff;

    uint32_t* hist = &sm.hist[0][0];   // 2048 bins
#pragma unroll 1
    while (top >= 0) {
        const int shift = max(0, top - 10);
        const uint32_t width_mask = (2u << (top - shift)) - 1u;   // top - shift + 1 <= 11 bits
        // zero the histogram (its last reads came before the previous pass's final barrier)
        for (int i = tid; i < 2048; i += kSelThreads) hist[i] = 0;
        __syncthreads();
        for (int r = 0; r < R; ++r) {
            const int i = r * kSelThreads + tid;   // strided: conflict-free shared loads
            if (i < n) {
                const uint32_t key = keys[i];
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & width_mask], 1u);
            }
        }
        __syncthreads();
        // thread t takes bins 2047 - 8t down to 2040 - 8t, so the inclusive scan counts the keys in
        // bins at or above its lowest bin
        uint32_t cnt[8], sum = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            cnt[q] = hist[2047 - 8 * tid - q];
            sum += cnt[q];
        }
        const uint32_t incl = sel_block_incl_scan(sum, sm, 0);
        uint32_t run = incl - sum;   // keys in bins above this thread's bins
        if (run < (uint32_t)k_rem && incl >= (uint32_t)k_rem) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (run < (uint32_t)k_rem && run + cnt[q] >= (uint32_t)k_rem) {
                    sm.digit = 2047 - 8 * tid - q;
                    sm.above = run;
                    sm.in_bin = cnt[q];
                }
                run += cnt[q];
            }
        }
        __syncthreads();
        const uint32_t digit = sm.digit;
        k_rem -= (int)sm.above;
        const bool whole = (int)sm.in_bin == k_rem;
        prefix |= digit << shift;
        mask |= width_mask << shift;
        top = shift - 1;
        // no barrier here: the next pass rewrites the histogram and sm.digit only after its own
        // first two barriers, which every thread reaches after reading them
        if (whole) break;
    }

    // ids above the decided prefix, plus the lowest-id ids equal to it (k_rem of them). Warp w
    // owns ids [w W, (w + 1) W) with W = 32 R, walked 32 at a time (lane l takes id base + l), so
    // both the shared loads and the output stay in id order and conflict-free.
    const int W = 32 * R, wbase = warp * W;
    uint32_t gt = 0, eq = 0;
    for (int r = 0; r < R; ++r) {
        const int i = wbase + 32 * r + lane;
        const uint32_t key = i < n ? keys[i] & mask : 0u;
        gt += __popc(__ballot_sync(0xFFFFFFFFu, i < n && key > prefix));
        eq += __popc(__ballot_sync(0xFFFFFFFFu, i < n && key == prefix));
    }
    const uint32_t packed = lane == 0 ? (gt << 16) | eq : 0u;   // n <= 65535: the halves never carry
    const uint32_t ex = sel_block_incl_scan(packed, sm, 1) - packed;   // warps before this one (lane 0)
    const uint32_t exw = __shfl_sync(0xFFFFFFFFu, ex, 0);
    int pos = (int)(exw >> 16) + min((int)(exw & 0xFFFFu), k_rem);
    int e = (int)(exw & 0xFFFFu);
    const unsigned lt = (1u << lane) - 1u;
    for (int r = 0; r < R; ++r) {
        const int i = wbase + 32 * r + lane;
        const uint32_t key = i < n ? keys[i] & mask : 0u;
        const unsigned bg = __ballot_sync(0xFFFFFFFFu, i < n && key > prefix);
        const unsigned be = __ballot_sync(0xFFFFFFFFu, i < n && key == prefix);
        // equal keys before this lane (this group and earlier ones) decide whether it is taken
        const int e_here = e + __popc(be & lt);
        const unsigned take = bg | (be & __ballot_sync(0xFFFFFFFFu, (be >> lane & 1u) && e_here < k_rem));
        if ((take >> lane) & 1u) out[pos + __popc(take & lt)] = i;
        pos += __popc(take);
        e += __popc(be);
    }
    __syncthreads();
    return k_eff;
}

}  // namespace smx
