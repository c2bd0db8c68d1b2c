// common.cuh -- device utilities shared by the libdspark kernels (GPU side only).
//
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC 2011), the (0,1) mapping, bf16
// loads, warp reductions and a bounded grid-wide wait.  Nothing here is shared
// with the CPU oracle.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

// ---------------------------------------------------------------- workspace
// Every workspace starts with a 256-byte header: the device status word and
// the grid-wait arrival counter, on separate 128-byte lines.
struct WsHeader {
    int32_t status;
    int32_t pad0[31];
    uint32_t arrivals;
    uint32_t pad1[31];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");
constexpr size_t kHeaderBytes = 256;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__device__ __forceinline__ void record_status(int32_t* st, int code) { atomicCAS(st, 0, code); }

// ---------------------------------------------------------------- PTX helpers
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
__device__ __forceinline__ int32_t ld_relaxed_s32(const int32_t* p) {
    int32_t v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Hardware base-2 exponential / logarithm (PTX ex2.approx / lg2.approx, max rel. error ~2^-22).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- loads
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T>
__device__ __forceinline__ float load_logit(const T* p, size_t idx);
template <>
__device__ __forceinline__ float load_logit<float>(const float* p, size_t idx) {
    return __ldg(p + idx);
}
template <>
__device__ __forceinline__ float load_logit<__nv_bfloat16>(const __nv_bfloat16* p, size_t idx) {
    return bf16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short*>(p) + idx));
}

// Eight consecutive logits starting at an index that is a multiple of 8 (16-byte aligned for
// bf16, 32-byte aligned for fp32).  `streaming` marks data read once (evict-first).
template <typename T>
__device__ __forceinline__ void load8(const T* p, size_t idx, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, size_t idx, float (&v)[8]) {
    uint4 w = __ldg(reinterpret_cast<const uint4*>(p + idx));
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, size_t idx, float (&v)[8]) {
    float4 a = __ldg(reinterpret_cast<const float4*>(p + idx));
    float4 b = __ldg(reinterpret_cast<const float4*>(p + idx) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Eight bf16 values (one 16-byte word) as floats, in memory order.
__device__ __forceinline__ void unpack_bf16x8(const uint4 w, float (&x)[8]) {
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
}

// Packed fp32x2 arithmetic (two lanes per instruction, each rounded as the scalar op).
__device__ __forceinline__ uint64_t pk2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 up2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// ---------------------------------------------------------------- 32 bf16 values per thread
// A thread's 32 values of a row chunk, as 16 packed bf16 pairs: four 16-byte groups at
// my0 + g GRP (each a conflict-free 16-byte read across a warp whose lanes take consecutive
// my0).  Word k holds elements (k / 4) GRP + my0 + 2 (k % 4) + {0, 1} in its low and high halves,
// so the elements ascend with (k, half).
template <int GRP>
__device__ __forceinline__ void load32w(const uint16_t* arr, int my0, uint32_t (&w)[16]) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint4 v = *reinterpret_cast<const uint4*>(arr + g * GRP + my0);
        w[4 * g] = v.x;
        w[4 * g + 1] = v.y;
        w[4 * g + 2] = v.z;
        w[4 * g + 3] = v.w;
    }
}

// Elements at or past `tail` (the ragged last chunk of a row) read as bf16 -inf: no mass, no max.
// Row lengths are multiples of 8, so a 16-byte group is wholly inside or outside.
template <int GRP>
__device__ __forceinline__ void mask_tail32(uint32_t (&w)[16], int my0, int tail) {
#pragma unroll
    for (int g = 0; g < 4; ++g)
        if (g * GRP + my0 >= tail) {
#pragma unroll
            for (int k = 0; k < 4; ++k) w[4 * g + k] = 0xFF80FF80u;
        }
}

// x - c for the low or high bf16 half of a packed word, in fp32 with one rounding (a mixed-precision
// subtract: the half is taken as it is, no unpacking).
__device__ __forceinline__ float sub_bf16_lo(uint32_t w, float c) {
    float r;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; sub.rn.f32.bf16 %0, l, %2; }" : "=f"(r) : "r"(w), "f"(c));
    return r;
}
__device__ __forceinline__ float sub_bf16_hi(uint32_t w, float c) {
    float r;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; sub.rn.f32.bf16 %0, h, %2; }" : "=f"(r) : "r"(w), "f"(c));
    return r;
}

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Sum over the 32 values of 2^(c (x - mu)) (c2 = c in both lanes; mu = m / c for the terms
// 2^(x c - m)), four packed accumulators: one mixed-precision subtract per value, one packed
// multiply per pair.
__device__ __forceinline__ float exp_sum32(const uint32_t (&w)[16], uint64_t c2, float mu) {
    uint64_t acc[4];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float2 y = up2(mul2(pk2(sub_bf16_lo(w[k], mu), sub_bf16_hi(w[k], mu)), c2));
        const uint64_t e = pk2(ex2(y.x), ex2(y.y));
        acc[k & 3] = k < 4 ? e : add2(acc[k & 3], e);
    }
    const float2 r = up2(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])));
    return r.x + r.y;
}

// One group of the online (max m, sum s of 2^(x scale - m)) statistics (scale > 0, inv = 1 / scale,
// c2 = scale in both lanes; m and s in the log2 domain).  The terms are taken against the running maximum as it
// stands; only when their sum reaches 2^64 (a row's first group, where m = -inf makes it inf or
// NaN, or a maximum that jumped far) is the group's maximum taken (packed bf16 maxima of the words:
// the maximum of the values exactly) and the sum rescaled.  While every value so far is -inf the
// pair stays (-inf, 0).
__device__ __forceinline__ void lse_step32w(const uint32_t (&w)[16], float scale, float inv, uint64_t c2, float& m,
                                            float& s) {
    float g = exp_sum32(w, c2, m * inv);  // (m = -inf: every term inf or NaN, so the exact path below)
    if (!(g < 0x1p64f)) {
        uint32_t mw[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mw[k] = bmax2(w[k], w[8 + k]);
        const uint32_t x = bmax2(bmax2(bmax2(mw[0], mw[1]), bmax2(mw[2], mw[3])),
                                 bmax2(bmax2(mw[4], mw[5]), bmax2(mw[6], mw[7])));
        const float gm = fmaxf(bf16_lo(x), bf16_hi(x)) * scale;
        const float mn = fmaxf(m, gm);
        const bool none = mn == -CUDART_INF_F;
        const float sc = none ? 0.f : ex2(m - mn);  // m = -inf, mn finite: 0
        const float mo = none ? 0.f : mn;           // x = -inf then gives 2^-inf = 0, never NaN
        g = exp_sum32(w, c2, mo * inv);
        s *= sc;
        m = mn;
    }
    s += g;
}

// ---------------------------------------------------------------- Philox4x32-10
// Ten rounds; each multiplies counter words 0 and 2 by two fixed odd constants, xors the
// high halves with the other counter words and the round key, and the key is advanced by
// two Weyl increments between rounds.
__device__ __forceinline__ uint4 philox10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t lo_a = 0xD2511F53u * c.x, hi_a = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo_b = 0xCD9E8D57u * c.z, hi_b = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi_b ^ c.y ^ k0, lo_b, hi_a ^ c.w ^ k1, lo_a);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}
__device__ __forceinline__ uint32_t philox_word(uint64_t seed, uint32_t j, uint32_t i, uint32_t purpose,
                                                uint32_t n) {
    const uint4 o = philox10(make_uint4(n >> 2, i, j, purpose), (uint32_t)seed, (uint32_t)(seed >> 32));
    const uint32_t s = n & 3u;
    return s == 0 ? o.x : (s == 1 ? o.y : (s == 2 ? o.z : o.w));
}
// (floor(x / 2^9) + 1/2) * 2^-23: exact in fp32, in [2^-24, 1 - 2^-24].
__device__ __forceinline__ float u01(uint32_t x) { return ((float)(x >> 9) + 0.5f) * (1.0f / 8388608.0f); }
__device__ __forceinline__ float uniform(uint64_t seed, uint32_t j, uint32_t i, uint32_t purpose, uint32_t n) {
    return u01(philox_word(seed, j, i, purpose, n));
}
// ln E with E = -ln u, for the exponential variates of the Gumbel races (absolute error a few
// 1e-7, far inside the decision margin).  u < 1/2: E = -log2(u) ln 2 by the hardware log2.
// u >= 1/2 (E small, where a variate is most likely to win): t = u - 1 is exact and
// E = -log1p(t) = -2 atanh(s), s = t / (2 + t) in [-1/3, 0), summed as the odd series
// 2 (s + s^3/3 + s^5/5 + ...) to s^19 (truncation below 2e-10 relative at |s| = 1/3), so E keeps
// its relative precision down to E ~ 2^-24.  Then ln E = log2(E) ln 2 by the hardware log2.
__device__ __forceinline__ float log_neg_log_u(float u) {
    float e;
    if (u < 0.5f) {
        e = -lg2(u) * 0.69314718055994531f;
    } else {
        const float t = u - 1.0f;
        const float sv = __fdividef(t, 2.0f + t);
        const float s2 = sv * sv;
        float q = 1.0f / 19.0f;
        q = fmaf(q, s2, 1.0f / 17.0f);
        q = fmaf(q, s2, 1.0f / 15.0f);
        q = fmaf(q, s2, 1.0f / 13.0f);
        q = fmaf(q, s2, 1.0f / 11.0f);
        q = fmaf(q, s2, 1.0f / 9.0f);
        q = fmaf(q, s2, 1.0f / 7.0f);
        q = fmaf(q, s2, 1.0f / 5.0f);
        q = fmaf(q, s2, 1.0f / 3.0f);
        q = fmaf(q, s2, 1.0f);
        e = -2.0f * sv * q;
    }
    return lg2(e) * 0.69314718055994531f;
}

// ln E, E = -ln u, with two hardware logarithms and no divide.  u < 1/2: E = -log2(u) ln 2 as
// above.  u >= 1/2: t = 1 - u is exact and ln E = ln t + G(t), G(t) = ln(-ln(1 - t) / t), a smooth
// function on [0, 1/2] (G(0) = 0, G'(0) = 1/2) evaluated as t Q(t), Q of degree 7 fitted by least
// squares in double precision on Chebyshev nodes of [0, 1/2] (largest error 5e-8 evaluated in
// single precision), so ln E keeps its absolute precision as E -> 0.
__device__ __forceinline__ float log_neg_log_u_2(float u) {
    const float t = 1.0f - u;
    const float lu = lg2(u);
    const bool lo = u < 0.5f;
    const float l = lg2(lo ? -lu * 0.69314718055994531f : t) * 0.69314718055994531f;
    float q = 4.252784252e-01f;
    q = fmaf(q, t, -4.789235294e-01f);
    q = fmaf(q, t, 3.674743176e-01f);
    q = fmaf(q, t, -3.672786430e-02f);
    q = fmaf(q, t, 1.060034558e-01f);
    q = fmaf(q, t, 1.231230795e-01f);
    q = fmaf(q, t, 2.084227204e-01f);
    q = fmaf(q, t, 4.999985397e-01f);
    return lo ? l : fmaf(q, t, l);
}

// 0xffffffff when a <= b, else 0 (one compare-and-set)
__device__ __forceinline__ uint32_t le_mask(float a, float b) {
    uint32_t r;
    asm("set.le.u32.f32 %0, %1, %2;" : "=r"(r) : "f"(a), "f"(b));
    return r;
}

// max of three (one instruction on this architecture)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// max of 32 values as a tree of three-input maxima (depth 4)
__device__ __forceinline__ float max32(const float (&z)[32]) {
    float a[11];
#pragma unroll
    for (int k = 0; k < 10; ++k) a[k] = fmax3(z[3 * k], z[3 * k + 1], z[3 * k + 2]);
    a[10] = fmaxf(z[30], z[31]);
    const float b0 = fmax3(a[0], a[1], a[2]), b1 = fmax3(a[3], a[4], a[5]), b2 = fmax3(a[6], a[7], a[8]);
    const float b3 = fmaxf(a[9], a[10]);
    return fmaxf(fmax3(b0, b1, b2), b3);
}

// ---------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_incl_scan(float v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}
// Argmax over a warp: larger value wins, lower index on equal values.
__device__ __forceinline__ void warp_argmax(float& v, int& idx) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
        if (ov > v || (ov == v && oi < idx)) {
            v = ov;
            idx = oi;
        }
    }
}

// ---------------------------------------------------------------- mbarrier + bulk copy
// Shared-memory mbarriers and the 1-D bulk copy engine (cp.async.bulk): a copy of `bytes`
// (multiple of 16, both addresses 16-byte aligned) from global to this block's shared memory
// signals completion on an mbarrier through its transaction count.
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}
// L2 eviction-priority policies (createpolicy): data read once goes first, data read again stays.
__device__ __forceinline__ void red_max_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Order-preserving 32-bit image of a float (-0 taken as +0) above the complemented id.
__device__ __forceinline__ unsigned long long pack_key(float key, int cand) {
    const uint32_t b = __float_as_uint(__fadd_rn(key, 0.f));
    const uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)o << 32) | (uint32_t)(~cand);
}
__device__ __forceinline__ float unpack_key(unsigned long long w) {
    const uint32_t o = (uint32_t)(w >> 32);
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// L2 prefetch of a contiguous byte range (16-byte aligned, multiple of 16 bytes).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// bulk_g2s with an L2 eviction policy for the source lines.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ void mbar_arrive_local(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// try_wait with a suspend-time hint: the thread sleeps in hardware until the phase completes or
// about `ns` nanoseconds pass, so a waiting warp issues almost nothing.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
        : "memory");
    return done != 0;
}

// Bounded wait that also gives up at once when `*abort` is set; records DSPARK_ERR_TIMEOUT
// and sets *abort on its own timeout.  cluster = acquire at cluster scope.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* status,
                                                   uint64_t limit_ns, bool cluster) {
    auto test = [&]() { return cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (test()) return true;
    const uint64_t t0 = global_ns();
    while (!test()) {
        if (*abort) return false;
        if (global_ns() - t0 > limit_ns) {
            record_status(status, DSPARK_ERR_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
    return true;
}

// mbar_wait_or_abort for a CTA-local barrier with suspended waits (bounded the same way).
__device__ __forceinline__ bool mbar_wait_hint_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                        int32_t* status, uint64_t limit_ns) {
    if (mbar_try_wait_hint(bar, parity, 100000u)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait_hint(bar, parity, 100000u)) {
        if (*abort) return false;
        if (global_ns() - t0 > limit_ns) {
            record_status(status, DSPARK_ERR_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
    return true;
}
// Named barrier over `count` threads (a multiple of 32) with id `id` (1..15).
__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Bounded wait for the phase with the given parity; false (and DSPARK_ERR_TIMEOUT recorded)
// if it did not complete within limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int32_t* status, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) {
            record_status(status, DSPARK_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// ---------------------------------------------------------------- grid-wide wait
// All blocks of a co-resident (cooperative) grid meet here.  `target` is the total number of
// arrivals expected so far (a monotonically growing counter, zeroed before the launch).
// The wait is bounded: past `limit_ns` it records DSPARK_ERR_TIMEOUT (first error wins) and
// returns false, as it does once another block has recorded a timeout; the caller must return.
// Split phase: grid_arrive() then independent work then grid_wait_arrived().
__device__ __forceinline__ void grid_arrive(WsHeader* h) {
    __syncthreads();
    if (threadIdx.x == 0)  // release: this block's writes are visible to whoever sees the arrival
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&h->arrivals) : "memory");
}

__device__ __forceinline__ bool grid_wait_arrived(WsHeader* h, uint32_t target, uint64_t limit_ns) {
    __shared__ int s_ok;
    if (threadIdx.x == 0) {
        int ok = 1;
        const uint64_t t0 = global_ns();
        while (ld_acquire_u32(&h->arrivals) < target) {
            if (ld_relaxed_s32(&h->status) == DSPARK_ERR_TIMEOUT) {  // another block gave up
                ok = 0;
                break;
            }
            if (global_ns() - t0 > limit_ns) {
                record_status(&h->status, DSPARK_ERR_TIMEOUT);
                ok = 0;
                break;
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

__device__ __forceinline__ bool grid_wait(WsHeader* h, uint32_t target, uint64_t limit_ns) {
    grid_arrive(h);
    return grid_wait_arrived(h, target, limit_ns);
}

}  // namespace dspark
