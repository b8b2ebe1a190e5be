// smx_device.cuh -- device helpers shared by the libsmx kernels (sm_103a).
//
// Element formats: E2M1 / E8M0 from the OCP Microscaling Formats v1.0 spec, E4M3 from the
// OCP 8-bit Floating Point spec; conversions use the sm_100-family PTX cvt forms
// (cvt.rn.satfinite.e2m1x2.f32, cvt.rn.f16x2.e2m1x2, cvt.rn.satfinite.e4m3x2.f32,
// cvt.rn.f16x2.e4m3x2). Tensor-core work uses mma.sync m16n8k16 (f16 / bf16, fp32 accum).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/smx.h"

namespace smx {

constexpr int kD = 128;
constexpr int kPage = 128;
constexpr int kMxPageBytes = SMX_MXFP4_PAGE_BYTES;   // 8704
constexpr int kMxScaleOff = 8192;
constexpr int kRsPageBytes = SMX_E4M3RS_PAGE_BYTES;  // 16896
constexpr int kRsScaleOff = 16384;
constexpr int kNvPageBytes = SMX_NVFP4_PAGE_BYTES;   // 9216: 128 x 64 B nibbles, 128 x 8 E4M3 block scales
constexpr int kNvScaleOff = 8192;

__device__ __forceinline__ void flag_status(int32_t* st, int bit) {
    if (st) atomicOr(st, bit);
}

// ---- ordering, bit helpers ---------------------------------------------------------------
// Order-preserving key of an fp32 score for descending selection: larger key = better.
// NaN ranks below every number (key 0); -0 and +0 compare equal.
__device__ __forceinline__ uint32_t score_key(float s) {
    if (s != s) return 0u;
    s = s + 0.0f;  // -0 -> +0
    uint32_t u = __float_as_uint(s);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// 2^e as fp32 for an E8M0 byte: 2^(b-127); b = 0 is the subnormal 2^-127; 0xFF is NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
    if (b == 0xFFu) return __uint_as_float(0x7FC00000u);
    if (b == 0u) return __uint_as_float(0x00400000u);
    return __uint_as_float(b << 23);
}

// ---- quantisation (a1 / a2) ----------------------------------------------------------------
// Two non-negative floats to one byte of E2M1 codes, lo in bits 0..3, hi in bits 4..7
// (round to nearest even, saturating at 6).
__device__ __forceinline__ uint32_t e2m1x2_rn_sat(float lo, float hi) {
    uint16_t r;
    asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n mov.b16 %0, {t, 0};\n}"
        : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r & 0xFFu;
}

// Two non-negative floats (|x| <= 448) to two e4m3 bytes, lo in bits 0..7.
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}

// floor(log2 a) of a finite positive float (exact, subnormals included).
__device__ __forceinline__ int floor_log2_pos(float a) {
    uint32_t u = __float_as_uint(a);
    int e = (int)((u >> 23) & 0xFF);
    if (e != 0) return e - 127;
    return -149 + (31 - __clz(u & 0x7FFFFF));
}

// 2^k as fp32 for k in [-126, 127].
__device__ __forceinline__ float exp2i_normal(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// x * 2^k for any k a float exponent difference can take (two exact power-of-two steps).
__device__ __forceinline__ float mul_exp2(float x, int k) {
    const int k1 = max(-126, min(127, k / 2));
    const int k2 = max(-126, min(127, k - k1));
    return x * exp2i_normal(k1) * exp2i_normal(k2);
}

// q packing rule for two floats: NaN -> 0x7F; otherwise clamp to [-448, 448] and round to nearest
// even; the sign bit is the input's sign. Returns the two e4m3 bytes (lo in bits 0..7).
__device__ __forceinline__ uint32_t pack_q2(float x0, float x1) {
    const uint32_t c = e4m3x2_rn_sat(fminf(fabsf(x0), 448.0f), fminf(fabsf(x1), 448.0f));
    uint32_t b0 = (c & 0xFF) | ((__float_as_uint(x0) >> 24) & 0x80u);
    uint32_t b1 = (c >> 8) | ((__float_as_uint(x1) >> 24) & 0x80u);
    if (x0 != x0) b0 = 0x7F;
    if (x1 != x1) b1 = 0x7F;
    return b0 | (b1 << 8);
}

// Four floats by the same rule (one call of pack_q2 per pair: the standalone packing kernel and
// the fused step share this code).
__device__ __forceinline__ uint32_t pack_q4(float4 x) { return pack_q2(x.x, x.y) | (pack_q2(x.z, x.w) << 16); }

// One 128-element row to MXFP4, warp-cooperative: lane l holds elements 4l..4l+3 (group
// l / 8). Writes 64 nibble bytes at `nib` and 4 scale bytes at `sc`.
__device__ __forceinline__ void quant_row_mxfp4_warp(float4 x, uint8_t* nib, uint8_t* sc, int lane) {
    const float v[4] = {x.x, x.y, x.z, x.w};
    bool nonfinite = false;
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (!isfinite(v[i])) nonfinite = true;
        else amax = fmaxf(amax, fabsf(v[i]));
    }
    const unsigned grp_mask = 0xFFu << (lane & ~7);
    const bool grp_nonfinite = (__ballot_sync(0xFFFFFFFFu, nonfinite) & grp_mask) != 0;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    int se = 0;
    if (amax > 0.0f) {
        se = floor_log2_pos(amax) - 2;
        se = max(-127, min(127, se));
    }
    uint32_t sbyte = grp_nonfinite ? 0xFFu : (uint32_t)(se + 127);
    const float inv = exp2i_normal(-se);  // -se in [-125, 127]
    uint32_t codes = 0;
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
        uint32_t c = e2m1x2_rn_sat(fabsf(v[i]) * inv, fabsf(v[i + 1]) * inv);
        c |= ((__float_as_uint(v[i]) >> 28) & 0x8u) | ((__float_as_uint(v[i + 1]) >> 24) & 0x80u);
        codes |= c << (4 * i);
    }
    if (grp_nonfinite) codes = 0;
    reinterpret_cast<uint16_t*>(nib)[lane] = (uint16_t)codes;
    // lane 0 gathers the four group scale bytes
    uint32_t s0 = __shfl_sync(0xFFFFFFFFu, sbyte, 0), s1 = __shfl_sync(0xFFFFFFFFu, sbyte, 8);
    uint32_t s2 = __shfl_sync(0xFFFFFFFFu, sbyte, 16), s3 = __shfl_sync(0xFFFFFFFFu, sbyte, 24);
    if (lane == 0) *reinterpret_cast<uint32_t*>(sc) = s0 | (s1 << 8) | (s2 << 16) | (s3 << 24);
}

// One 128-element row to e4m3 codes with one fp32 scale s = fl32(amax / 448) (1 if amax = 0;
// NaN and all codes 0x7F if the row holds NaN/Inf), warp-cooperative like above.
__device__ __forceinline__ void quant_row_e4m3rs_warp(float4 x, uint8_t* codes, float* scale, int lane) {
    const float v[4] = {x.x, x.y, x.z, x.w};
    bool nonfinite = false;
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (!isfinite(v[i])) nonfinite = true;
        else amax = fmaxf(amax, fabsf(v[i]));
    }
    const bool any_nf = __any_sync(0xFFFFFFFFu, nonfinite);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
    uint32_t out = 0;
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
        float y0 = fminf(fabsf(__fdiv_rn(v[i], s)), 448.0f);
        float y1 = fminf(fabsf(__fdiv_rn(v[i + 1], s)), 448.0f);
        uint32_t c = e4m3x2_rn_sat(y0, y1);
        c |= ((__float_as_uint(v[i]) >> 24) & 0x80u) | ((__float_as_uint(v[i + 1]) >> 16) & 0x8000u);
        out |= c << (8 * i);
    }
    if (any_nf) out = 0x7F7F7F7Fu;
    reinterpret_cast<uint32_t*>(codes)[lane] = out;
    if (lane == 0) *scale = any_nf ? __uint_as_float(0x7FC00000u) : s;
}

// ---- dequantisation to f16 / bf16 ------------------------------------------------------------
// Four bytes of E2M1 nibbles to four f16x2 (exact values in {0, +-0.5, ..., +-6}); register i
// holds (element 2i in the low half, element 2i+1 in the high half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& h0, uint32_t& h1, uint32_t& h2, uint32_t& h3) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3) : "r"(w));
}

// Two e4m3 bytes (low 16 bits) to f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w16) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)w16));
    return r;
}

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h) {
    __half2 v = *reinterpret_cast<__half2*>(&h);
    return __half22float2(v);
}

// One 128-element row to NVFP4 with the per-tensor decode scale g, warp-cooperative: lane l
// holds elements 4l..4l+3 (block l / 4 of 16). Per block: s = fl32(amax / fl32(6 g)); the E4M3
// scale byte is s rounded to nearest even, saturating at 448; S = fl32(E4M3(byte) x g); each
// code is x / S (fp32, rounded to nearest) rounded to the nearest E2M1 value (ties to even,
// saturating at 6, the sign of x kept). S == 0 gives codes 0; a block holding NaN or an infinity
// gets byte 0x7F (E4M3 NaN) and codes 0. Writes 64 nibble bytes at `nib` and the 8 block scale
// bytes at `sc` (8-byte aligned).
__device__ __forceinline__ void quant_row_nvfp4_warp(float4 x, float g, uint8_t* nib, uint8_t* sc, int lane) {
    const float v[4] = {x.x, x.y, x.z, x.w};
    bool nonfinite = false;
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (!isfinite(v[i])) nonfinite = true;
        else amax = fmaxf(amax, fabsf(v[i]));
    }
    const unsigned blk_mask = 0xFu << (lane & ~3);
    const bool blk_nonfinite = (__ballot_sync(0xFFFFFFFFu, nonfinite) & blk_mask) != 0;
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    const float s = fminf(__fdiv_rn(amax, __fmul_rn(6.0f, g)), 448.0f);
    const uint32_t sbyte = blk_nonfinite ? 0x7Fu : (e4m3x2_rn_sat(s, 0.0f) & 0xFFu);
    const float S = __fmul_rn(f16x2_to_f32x2(e4m3x2_to_f16x2(sbyte)).x, g);
    uint32_t codes = 0;
    if (!blk_nonfinite && S != 0.0f) {
#pragma unroll
        for (int i = 0; i < 4; i += 2) {
            const float y0 = __fdiv_rn(v[i], S), y1 = __fdiv_rn(v[i + 1], S);
            uint32_t c = e2m1x2_rn_sat(fabsf(y0), fabsf(y1));
            c |= ((__float_as_uint(y0) >> 28) & 0x8u) | ((__float_as_uint(y1) >> 24) & 0x80u);
            codes |= c << (4 * i);
        }
    }
    reinterpret_cast<uint16_t*>(nib)[lane] = (uint16_t)codes;
    // lanes 0, 4, ..., 28 hold the eight block bytes; lane 0 gathers them
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        lo |= __shfl_sync(0xFFFFFFFFu, sbyte, 4 * k) << (8 * k);
        hi |= __shfl_sync(0xFFFFFFFFu, sbyte, 16 + 4 * k) << (8 * k);
    }
    if (lane == 0) *reinterpret_cast<uint2*>(sc) = make_uint2(lo, hi);
}


__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}

// ---- tensor cores ---------------------------------------------------------------------------
// Register-only tensor-core ops: not volatile, so the compiler may interleave independent chains.
__device__ __forceinline__ void mma_f16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a) : "memory");
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ldg_cg_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p) : "memory");
    return r;
}

__device__ __forceinline__ uint32_t ldg_cg_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(r) : "l"(p) : "memory");
    return r;
}

__device__ __forceinline__ float ldg_cg_f32(const float* p) {
    float r;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(r) : "l"(p));
    return r;
}

// Programmatic dependent launch: wait for the preceding grid's completion and memory; let the
// next grid in the stream begin launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

// ---- bulk copies (TMA, 1-D) with mbarrier completion -----------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait (about a second at most); false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < (1u << 22); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i > 64) __nanosleep(256);
    }
    return false;
}

// Bounded wait for a pipeline hand-off: polls without sleeping (a sleep would add its wake-up
// latency to every stage of a pipeline), giving up after about two seconds of global time.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t* bar, uint32_t parity) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 0) {
            uint64_t t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            if (i == 0) t0 = t;
            else if (t - t0 > 2000000000ull) return false;
        }
    }
}

// Copy `bytes` (multiple of 16, both addresses 16-byte aligned) global -> shared, completing on bar.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// Order earlier generic-proxy accesses of shared memory before later async-proxy (bulk copy) ones.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Order earlier generic-proxy accesses of global memory (including other threads' writes this
// thread has acquired) before its later async-proxy (bulk copy) reads.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Hint: bring the 128-byte line holding p into L2.
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// The same, with the evict-last priority (kept while streams marked evict-first pass through L2).
__device__ __forceinline__ void prefetch_l2_keep(const void* p) {
    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p));
}

// ---- counters shared by the CTAs of one grid ---------------------------------------------------
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void spin_cycles(long long n) {
    const long long t = clock64();
    while (clock64() - t < n) {
    }
}

// Release: this thread's earlier writes, and those of threads it synchronised with (a barrier
// before the call), are visible before the increment is.
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Default bound of a wait for other CTAs of the step (ns of global time): far above the longest
// step the ABI's largest shapes run (tens of milliseconds), short enough that a stuck step frees
// a shared GPU quickly.
constexpr uint64_t kDefaultWaitNs = 200000000ull;

// One thread waits until *p >= target, then orders its later reads after the writes released
// before the update (a relaxed poll followed by an acquire fence). Between polls it sleeps
// briefly (polling harder floods the counter's L2 slice and slows the updaters); it gives up
// (false) once limit_ns of global time have passed since its first poll, or after 2^24 polls.
__device__ __forceinline__ bool wait_geq_bounded(const uint32_t* p, uint32_t target, uint64_t limit_ns) {
    const uint64_t t0 = global_ns();
    bool ok = false;
    for (uint32_t i = 0; i < (1u << 24); ++i) {
        if (ld_relaxed_u32(p) >= target) {
            ok = true;
            break;
        }
        if (global_ns() - t0 >= limit_ns) break;
        __nanosleep(i < 64 ? 32 : 128);
    }
    fence_acq_rel_gpu();
    return ok;
}

// ---- shape helpers -----------------------------------------------------------------------------
__device__ __forceinline__ int clamp_ctx(int ctx, int Q, int max_pages, int32_t* st) {
    const int cap = max_pages * kPage;
    if (ctx < Q || ctx > cap) {
        flag_status(st, SMX_DEV_BAD_CTX);
        ctx = max(0, min(ctx, cap));
    }
    return ctx;
}

}  // namespace smx
