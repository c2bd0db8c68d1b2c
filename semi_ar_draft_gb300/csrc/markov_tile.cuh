// markov_tile.cuh -- per-tile building blocks shared by the sampling and verify kernels.
//
// A "tile" is DSPARK_TILE consecutive vocabulary ids, a "chunk" DSPARK_CHUNK consecutive ids
// of a tile, a "row block" 16 rows (requests).  The producer computes, for a row block over
// one tile, z = base + W2 . W1[prev] in registers (tensor-core mma.sync bf16 with the
// accumulator initialised from the base logits, or a CUDA-core GEMV), turns it into the row's
// log2-weights (draft sampling, residual or bonus draw) and reduces every chunk to
//   {max log2-weight m_c, sum 2^(l - m_c)}
// (greedy: {max value, lowest argmax}); the values go to a shared-memory row buffer.
// finalize_tile_cg() turns a row's 32 chunk statistics into the tile record of the chunk-Gumbel
// contract (dspark.h): the best chunk key of the tile, the tile's log-mass, and the in-chunk
// inverse-CDF candidate of the winning chunk -- before the winning tile is known.
#pragma once

#include "common.cuh"

namespace dspark {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kTS = DSPARK_TILE;
constexpr int kCS = DSPARK_CHUNK;
constexpr int kChunks = kTS / kCS;
constexpr int kRows = 16;
constexpr int kChunksPerWarp = kChunks / kWarps;
static_assert(kChunks == 32, "one warp lane per chunk in finalize_chunks");
static_assert(kCS == 32, "a lane quad holds one chunk: 4 lanes x 8 ids");
constexpr int kXRow = kTS + 4;  // padded row stride (floats) of the value buffer: conflict-free 16-byte stores

enum RowMode { ROW_OFF = 0, ROW_SAMPLE = 1, ROW_RESID = 2, ROW_BONUS = 3 };

// Final-logit softcap of the draft model (page "03 · DSpark 建模：Markov 与 Confidence", section
// 3.12: compute_logits returns s tanh(logits / s)): applied to base logits as they are loaded,
// before the Markov bias; ids past V keep the -inf of their padding.  s = 0: none.
// tanh from its definition, without branches.  For |x| >= 1/8: tanh|x| = (1 - e) / (1 + e) with
// e = exp(-2|x|) in (0, 0.78], so the numerator loses at most a factor 4.6 of e's relative error
// (about 1e-6 in all); |x| = inf gives e = 0 and 1.  For |x| < 1/8: the odd Taylor series
// x - x^3/3 + 2x^5/15 - 17x^7/315, whose next term (62/2835) x^9 is below 2e-9 of x there.  NaN
// stays NaN.
__device__ __forceinline__ float tanh_def(float x) {
    const float a = fabsf(x), x2 = x * x;
    const float series = x * fmaf(x2, fmaf(x2, fmaf(x2, -17.f / 315.f, 2.f / 15.f), -1.f / 3.f), 1.f);
    const float e = ex2(-2.f * kLog2e * a);
    const float t = copysignf(__fdividef(1.f - e, 1.f + e), x);
    return a < 0.125f ? series : t;
}

__device__ __forceinline__ void softcap8(float (&x)[8], int id0, int V, float s, float inv_s) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = id0 + e < V ? s * tanh_def(x[e] * inv_s) : -CUDART_INF_F;
}

// Per-row inputs of a row block, staged in shared memory by the caller.
struct RowBlock {
    int prev[kRows];         // W1 row (previous token)
    int mode[kRows];         // RowMode
    long long brow[kRows];   // element offset of the base-logit row (-1: z not needed)
    long long trow[kRows];   // element offset of the target-logit row (-1: none)
    float u1[kRows];         // chunk-level uniform
    float u2[kRows];         // id-level uniform
    float lnE[kRows];        // ln of the tile's exponential variate
    float lse2[kRows];       // residual: log2-sum-exp of the target row (t * scale2)
    float dl2[kRows];        // residual: draft LSE in log2 units
};

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t a0, const uint32_t a1, const uint32_t a2,
                                         const uint32_t a3, const uint32_t b0, const uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}


// --------------------------------------------------------------------------------------------
// Tensor-core bias: mma.sync m16n8k16, rows = 16 requests (A = W1[prev]), columns = 8 ids
// (B = W2 rows), K = r = 16*KS.
// K permutation: in k-step s, quad lane tq feeds MMA slots {2tq, 2tq+1, 2tq+8, 2tq+9} with
// k = tq*r/4 + 4s + {0,1,2,3}.  Any bijection is valid if A and B use the same one; this one
// lets each lane read r/4 contiguous weights of a row.
// Column permutation: in n-tile nt of a 32-id chunk, MMA column n is id 8*(n/2) + 2*nt + n%2,
// so the accumulator of lane (g, tq) holds ids 8*tq .. 8*tq+7 of the chunk, rows g and g+8.
// --------------------------------------------------------------------------------------------
template <int KS>
struct Frag {
    uint32_t w[KS > 0 ? 2 * KS : 1];  // the lane's r/4 weights of one row, as bf16 pairs
};

template <int KS>
__device__ __forceinline__ void frag_zero(Frag<KS>& f) {
#pragma unroll
    for (int w = 0; w < 2 * KS; ++w) f.w[w] = 0u;
}

template <int KS>
__device__ __forceinline__ void load_frag_global(const uint16_t* W, int row, int tq, Frag<KS>& f) {
    constexpr int r = 16 * KS;
    const uint16_t* p = W + (size_t)row * r + tq * (r / 4);
    if constexpr (KS == 1) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        f.w[0] = u.x;
        f.w[1] = u.y;
    } else {
#pragma unroll
        for (int q = 0; q < KS / 2; ++q) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(p) + q);
            f.w[4 * q + 0] = u.x;
            f.w[4 * q + 1] = u.y;
            f.w[4 * q + 2] = u.z;
            f.w[4 * q + 3] = u.w;
        }
    }
}

// Shared-memory W2 tile: row vl holds r bf16 as 16-byte units; unit u is stored at position
// u ^ (vl & mask), mask = min(units, 8) - 1, so the 8 lanes of a quarter-warp (rows vl, vl+1)
// hit 8 distinct bank groups.
template <int KS>
__host__ __device__ constexpr int w2_units() {
    return (16 * KS) / 8;
}
template <int KS>
__host__ __device__ constexpr int w2_mask() {
    return (w2_units<KS>() >= 8 ? 8 : w2_units<KS>()) - 1;
}

template <int KS>
__device__ __forceinline__ void load_frag_smem(const uint4* w2s, int vl, int tq, Frag<KS>& f) {
    constexpr int units = w2_units<KS>();
    constexpr int mask = w2_mask<KS>();
    const uint4* row = w2s + (size_t)vl * units;
    if constexpr (KS == 1) {
        const int u = tq >> 1, half = tq & 1;  // r = 16: the lane reads 8 bytes (half a unit)
        const uint2 v = reinterpret_cast<const uint2*>(row + (u ^ (vl & mask)))[half];
        f.w[0] = v.x;
        f.w[1] = v.y;
    } else {
#pragma unroll
        for (int q = 0; q < KS / 2; ++q) {
            const int u = tq * (KS / 2) + q;
            const uint4 v = row[u ^ (vl & mask)];
            f.w[4 * q + 0] = v.x;
            f.w[4 * q + 1] = v.y;
            f.w[4 * q + 2] = v.z;
            f.w[4 * q + 3] = v.w;
        }
    }
}

// Stage W2 rows [tile0, tile0 + kTS) into shared memory (swizzled; threads 0 .. nthreads-1
// take part); rows past V are zero.
template <int KS>
__device__ void stage_w2_tile(const uint16_t* W2, int tile0, int V, uint4* dst, int nthreads) {
    constexpr int units = w2_units<KS>();
    constexpr int mask = w2_mask<KS>();
    for (int idx = threadIdx.x; idx < kTS * units; idx += nthreads) {
        const int vl = idx / units, u = idx % units;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (tile0 + vl < V) v = __ldg(reinterpret_cast<const uint4*>(W2 + (size_t)(tile0 + vl) * (16 * KS)) + u);
        dst[vl * units + (u ^ (vl & mask))] = v;
    }
}

// The same staging with every 16-byte copy in flight at once (cp.async, L2 -> shared memory,
// no register round trip); the caller waits with cp_async_wait_all() and a barrier.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n cp.async.wait_group 0;" ::: "memory");
}
template <int KS>
__device__ void stage_w2_tile_async(const uint16_t* W2, int tile0, int V, uint4* dst, int nthreads) {
    constexpr int units = w2_units<KS>();
    constexpr int mask = w2_mask<KS>();
    for (int idx = threadIdx.x; idx < kTS * units; idx += nthreads) {
        const int vl = idx / units, u = idx % units;
        uint4* d = dst + vl * units + (u ^ (vl & mask));
        if (tile0 + vl < V) cp_async16(d, reinterpret_cast<const uint4*>(W2 + (size_t)(tile0 + vl) * (16 * KS)) + u);
        else *d = make_uint4(0u, 0u, 0u, 0u);
    }
}

// --------------------------------------------------------------------------------------------
// Eight consecutive logits kept as raw words until needed (so many loads can be in flight).
// --------------------------------------------------------------------------------------------
template <typename TL>
struct Raw8 {
    static constexpr int kWords = sizeof(TL) * 2;  // bf16: 4 words, fp32: 8 words
    uint32_t w[kWords];
};

template <typename TL>
__device__ __forceinline__ void load_raw8(const TL* row, int v0, int V, bool vec, Raw8<TL>& r) {
    if (vec && v0 + 8 <= V) {
        const uint4* p = reinterpret_cast<const uint4*>(row + v0);
#pragma unroll
        for (int q = 0; q < Raw8<TL>::kWords / 4; ++q) {
            const uint4 u = __ldg(p + q);
            r.w[4 * q] = u.x;
            r.w[4 * q + 1] = u.y;
            r.w[4 * q + 2] = u.z;
            r.w[4 * q + 3] = u.w;
        }
    } else if constexpr (sizeof(TL) == 2) {
        const unsigned short* p = reinterpret_cast<const unsigned short*>(row);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const uint32_t lo = (v0 + e < V) ? __ldg(p + v0 + e) : 0xFF80u;  // bf16 -inf past V
            const uint32_t hi = (v0 + e + 1 < V) ? __ldg(p + v0 + e + 1) : 0xFF80u;
            r.w[e / 2] = lo | (hi << 16);
        }
    } else {
        const float* p = reinterpret_cast<const float*>(row);
#pragma unroll
        for (int e = 0; e < 8; ++e) r.w[e] = (v0 + e < V) ? __float_as_uint(__ldg(p + v0 + e)) : 0xFF800000u;
    }
}

template <typename TL>
__device__ __forceinline__ void unpack8(const Raw8<TL>& r, float (&x)[8]) {
    if constexpr (sizeof(TL) == 2) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            x[2 * q] = bf16_lo(r.w[q]);
            x[2 * q + 1] = bf16_hi(r.w[q]);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(r.w[e]);
    }
}

// --------------------------------------------------------------------------------------------
// Chunk statistics from one lane quad (lane tq holds ids id0 .. id0+7 = chunk base + 8 tq):
// T > 0: (max m_c of the log2-weights, sum 2^(l - m_c)); greedy: (max value, lowest argmax).
// Every lane runs every shuffle (full-warp masks); nothing returns early.
// --------------------------------------------------------------------------------------------
__device__ __forceinline__ float2 chunk_stats(const float (&l)[8], int id0, int greedy) {
    if (greedy) {
        float m = l[0];
        int idx = id0;
#pragma unroll
        for (int e = 1; e < 8; ++e)
            if (l[e] > m) {
                m = l[e];
                idx = id0 + e;
            }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            const float om = __shfl_xor_sync(0xffffffffu, m, o);
            const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
            if (om > m || (om == m && oi < idx)) {
                m = om;
                idx = oi;
            }
        }
        return make_float2(m, __int_as_float(idx));
    }
    float m = l[0];
#pragma unroll
    for (int e = 1; e < 8; ++e) m = fmaxf(m, l[e]);
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const float mref = (m == -CUDART_INF_F) ? 0.f : m;  // an empty quad sums to 0
    float sum = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) sum += ex2(l[e] - mref);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    return make_float2(m, sum);
}

__device__ __forceinline__ float2 empty_stats(int greedy) {
    return greedy ? make_float2(-CUDART_INF_F, __int_as_float(0x7fffffff)) : make_float2(-CUDART_INF_F, 0.f);
}

// --------------------------------------------------------------------------------------------
// Producer: for a row block over one tile, the buffered values xbuf[16][kXRow] (z for draft
// rows, the log2-weight for residual / bonus rows) and the chunk statistics cstat[16][32].
// --------------------------------------------------------------------------------------------
struct ProdArgs {
    const void* base;
    const void* target;
    const void* W1;
    const void* W2;
    const uint4* w2s;   // W2 tile in shared memory (tensor-core path) or null
    const float* w1s;   // W1 rows of the row block as fp32 [16][r] (CUDA-core path)
    int V, r;
    int greedy;
    float scale2;       // log2(e) / T
    int vec_b, vec_t;   // 16-byte aligned rows: 8-wide loads allowed
    float softcap, inv_softcap;  // draft softcap of the base logits (0: none)
};

// HAS_T: rows may read target logits (residual / bonus draws of the verify pass).
template <typename TL, int KS, typename TW, bool HAS_T>
__device__ __forceinline__ void produce_chunks(const ProdArgs& pa, int tile, const RowBlock& rb, float* xbuf,
                                               float2* cstat) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int ma = rb.mode[g], mb = rb.mode[g + 8];
    const bool za = ma == ROW_SAMPLE || ma == ROW_RESID, zb = mb == ROW_SAMPLE || mb == ROW_RESID;
    const bool ta = HAS_T && (ma == ROW_RESID || ma == ROW_BONUS);
    const bool tb = HAS_T && (mb == ROW_RESID || mb == ROW_BONUS);
    const bool need_z = __any_sync(0xffffffffu, za || zb);
    const bool need_t = HAS_T && __any_sync(0xffffffffu, ta || tb);
    const TL* base = reinterpret_cast<const TL*>(pa.base);
    const TL* tgt = reinterpret_cast<const TL*>(pa.target);
    const TL* browA = base + (za ? rb.brow[g] : 0);
    const TL* browB = base + (zb ? rb.brow[g + 8] : 0);
    const TL* trowA = tgt + (ta ? rb.trow[g] : 0);
    const TL* trowB = tgt + (tb ? rb.trow[g + 8] : 0);
    const int tile0 = tile * kTS;

    // all of this warp's loads first: kChunksPerWarp chunks x 2 rows (x 2 tensors)
    Raw8<TL> xb_[kChunksPerWarp][2];
    Raw8<TL> xt_[HAS_T ? kChunksPerWarp : 1][2];
#pragma unroll
    for (int k = 0; k < kChunksPerWarp; ++k) {
        const int v0 = tile0 + kCS * (warp + kWarps * k) + 8 * tq;
        if (need_z) {
            if (za) load_raw8<TL>(browA, v0, pa.V, pa.vec_b, xb_[k][0]);
            if (zb) load_raw8<TL>(browB, v0, pa.V, pa.vec_b, xb_[k][1]);
        }
        if constexpr (HAS_T) {
            if (need_t) {
                if (ta) load_raw8<TL>(trowA, v0, pa.V, pa.vec_t, xt_[k][0]);
                if (tb) load_raw8<TL>(trowB, v0, pa.V, pa.vec_t, xt_[k][1]);
            }
        }
    }
    Frag<KS> fa, fb;
    if constexpr (KS > 0) {
        const uint16_t* W1 = reinterpret_cast<const uint16_t*>(pa.W1);
        if (za) load_frag_global<KS>(W1, rb.prev[g], tq, fa);
        else frag_zero<KS>(fa);
        if (zb) load_frag_global<KS>(W1, rb.prev[g + 8], tq, fb);
        else frag_zero<KS>(fb);
    }
#pragma unroll
    for (int k = 0; k < kChunksPerWarp; ++k) {
        const int c = warp + kWarps * k;
        const int cb = tile0 + kCS * c;
        if (cb >= pa.V) {
            if (tq == 0) {
                cstat[g * kChunks + c] = empty_stats(pa.greedy);
                cstat[(g + 8) * kChunks + c] = empty_stats(pa.greedy);
            }
            continue;
        }
        const int id0 = cb + 8 * tq;
        float xa[8], xb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) xa[e] = xb[e] = 0.f;
        if (need_z) {
            if (za) unpack8<TL>(xb_[k][0], xa);
            if (zb) unpack8<TL>(xb_[k][1], xb);
            if (pa.softcap > 0.f) {
                softcap8(xa, id0, pa.V, pa.softcap, pa.inv_softcap);
                softcap8(xb, id0, pa.V, pa.softcap, pa.inv_softcap);
            }
            if constexpr (KS > 0) {
                const uint16_t* W2 = reinterpret_cast<const uint16_t*>(pa.W2);
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    float d[4] = {xa[2 * nt], xa[2 * nt + 1], xb[2 * nt], xb[2 * nt + 1]};
                    const int vcol = cb + 8 * (g >> 1) + 2 * nt + (g & 1);  // id this lane feeds as column g
                    Frag<KS> fw;
                    if (vcol < pa.V) {
                        if (pa.w2s) load_frag_smem<KS>(pa.w2s, vcol - tile0, tq, fw);
                        else load_frag_global<KS>(W2, vcol, tq, fw);
                    } else {
                        frag_zero<KS>(fw);
                    }
#pragma unroll
                    for (int s = 0; s < KS; ++s)
                        mma_bf16(d, fa.w[2 * s], fb.w[2 * s], fa.w[2 * s + 1], fb.w[2 * s + 1], fw.w[2 * s],
                                 fw.w[2 * s + 1]);
                    xa[2 * nt] = d[0];
                    xa[2 * nt + 1] = d[1];
                    xb[2 * nt] = d[2];
                    xb[2 * nt + 1] = d[3];
                }
            } else if (pa.r > 0) {
                const TW* W2 = reinterpret_cast<const TW*>(pa.W2);
                const float* w1a = pa.w1s + g * pa.r;
                const float* w1b = pa.w1s + (g + 8) * pa.r;
                for (int kk = 0; kk < pa.r; ++kk) {
                    const float wa = w1a[kk], wb = w1b[kk];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float w2 = (id0 + e < pa.V) ? load_logit<TW>(W2, (size_t)(id0 + e) * pa.r + kk) : 0.f;
                        xa[e] = fmaf(wa, w2, xa[e]);
                        xb[e] = fmaf(wb, w2, xb[e]);
                    }
                }
            }
        }
        // per-row log2-weights (greedy: the values themselves); buffered: z for draft rows, the
        // log2-weight (greedy: the value) for residual / bonus rows
        float la[8], lb[8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int mode = h ? mb : ma;
            float(&x)[8] = h ? xb : xa;
            float(&l)[8] = h ? lb : la;
            const int row = h ? g + 8 : g;
            if (mode == ROW_SAMPLE) {
#pragma unroll
                for (int e = 0; e < 8; ++e) l[e] = pa.greedy ? x[e] : x[e] * pa.scale2;
            } else if (HAS_T && (mode == ROW_BONUS || mode == ROW_RESID)) {
                float t[8];
                unpack8<TL>(xt_[HAS_T ? k : 0][h], t);
                if (mode == ROW_BONUS) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) l[e] = pa.greedy ? t[e] : t[e] * pa.scale2;
                } else {
                    const float lse2 = rb.lse2[row], dl2 = rb.dl2[row];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float w = ex2(fmaf(t[e], pa.scale2, -lse2)) - ex2(fmaf(x[e], pa.scale2, -dl2));
                        l[e] = w > 0.f ? lg2(w) : -CUDART_INF_F;
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = l[e];
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) l[e] = x[e] = -CUDART_INF_F;
            }
            float4* dst = reinterpret_cast<float4*>(xbuf + row * kXRow + kCS * c + 8 * tq);
            dst[0] = make_float4(x[0], x[1], x[2], x[3]);
            dst[1] = make_float4(x[4], x[5], x[6], x[7]);
        }
        const float2 sa = chunk_stats(la, id0, pa.greedy);
        const float2 sb = chunk_stats(lb, id0, pa.greedy);
        if (tq == 0) {
            cstat[g * kChunks + c] = sa;
            cstat[(g + 8) * kChunks + c] = sb;
        }
    }
}

// --------------------------------------------------------------------------------------------
// Draft-sampling producer (tensor-core path): every row is a draft row (rows past B read row
// brow[0] and are never finalised), so there is no per-lane mode logic; greedy, the W2 source
// and "tile fully inside the vocabulary" are compile-time.  Writes z to xbuf and the chunk
// statistics of z * scale2 (greedy: of z) to cstat.
// --------------------------------------------------------------------------------------------
__device__ __forceinline__ void mma4(float& d0, float& d1, float& d2, float& d3, const uint32_t a0, const uint32_t a1,
                                     const uint32_t a2, const uint32_t a3, const uint32_t b0, const uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <typename TL, int KS, bool GREEDY, bool W2SMEM, bool FULL>
__device__ __forceinline__ void produce_sample(const TL* base, const uint16_t* W1, const uint16_t* W2, const uint4* w2s,
                                               int V, bool vec, int tile, const RowBlock& rb, float* xbuf,
                                               float2* cstat, float scale2, float softcap, float inv_softcap) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    const long long oA = rb.brow[g] >= 0 ? rb.brow[g] : rb.brow[0];
    const long long oB = rb.brow[g + 8] >= 0 ? rb.brow[g + 8] : rb.brow[0];
    const TL* rowA = base + oA;
    const TL* rowB = base + oB;
    const int tile0 = tile * kTS;
    Raw8<TL> ra[kChunksPerWarp], rbv[kChunksPerWarp];
#pragma unroll
    for (int k = 0; k < kChunksPerWarp; ++k) {
        const int v0 = tile0 + kCS * (warp + kWarps * k) + 8 * tq;
        load_raw8<TL>(rowA, v0, V, FULL || vec, ra[k]);
        load_raw8<TL>(rowB, v0, V, FULL || vec, rbv[k]);
    }
    Frag<KS> fa, fb;
    load_frag_global<KS>(W1, rb.prev[g], tq, fa);
    load_frag_global<KS>(W1, rb.prev[g + 8], tq, fb);
#pragma unroll
    for (int k = 0; k < kChunksPerWarp; ++k) {
        const int c = warp + kWarps * k;
        const int cb = tile0 + kCS * c;
        if (!FULL && cb >= V) {
            if (tq == 0) {
                cstat[g * kChunks + c] = empty_stats(GREEDY);
                cstat[(g + 8) * kChunks + c] = empty_stats(GREEDY);
            }
            continue;
        }
        float xa[8], xb[8];
        unpack8<TL>(ra[k], xa);
        unpack8<TL>(rbv[k], xb);
        if (softcap > 0.f) {
            softcap8(xa, cb + 8 * tq, V, softcap, inv_softcap);
            softcap8(xb, cb + 8 * tq, V, softcap, inv_softcap);
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int vl = kCS * c + 8 * (g >> 1) + 2 * nt + (g & 1);  // id (in tile) this lane feeds as column g
            Frag<KS> fw;
            if (FULL || tile0 + vl < V) {
                if constexpr (W2SMEM) load_frag_smem<KS>(w2s, vl, tq, fw);
                else load_frag_global<KS>(W2, tile0 + vl, tq, fw);
            } else {
                frag_zero<KS>(fw);
            }
#pragma unroll
            for (int s = 0; s < KS; ++s)
                mma4(xa[2 * nt], xa[2 * nt + 1], xb[2 * nt], xb[2 * nt + 1], fa.w[2 * s], fb.w[2 * s], fa.w[2 * s + 1],
                     fb.w[2 * s + 1], fw.w[2 * s], fw.w[2 * s + 1]);
        }
        float4* dA = reinterpret_cast<float4*>(xbuf + g * kXRow + kCS * c + 8 * tq);
        float4* dB = reinterpret_cast<float4*>(xbuf + (g + 8) * kXRow + kCS * c + 8 * tq);
        dA[0] = make_float4(xa[0], xa[1], xa[2], xa[3]);
        dA[1] = make_float4(xa[4], xa[5], xa[6], xa[7]);
        dB[0] = make_float4(xb[0], xb[1], xb[2], xb[3]);
        dB[1] = make_float4(xb[4], xb[5], xb[6], xb[7]);
        if constexpr (!GREEDY) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                xa[e] *= scale2;
                xb[e] *= scale2;
            }
        }
        const float2 sa = chunk_stats(xa, cb + 8 * tq, GREEDY);
        const float2 sb = chunk_stats(xb, cb + 8 * tq, GREEDY);
        if (tq == 0) {
            cstat[g * kChunks + c] = sa;
            cstat[(g + 8) * kChunks + c] = sb;
        }
    }
}

// --------------------------------------------------------------------------------------------
// Staged draft sampling (bf16 logits, tensor-core path).  The base logits of a row block over
// the block's tile are copied into shared memory by the bulk-copy engine one row block ahead;
// rows are padded to kStageRow ids so the 16-byte reads of a quarter-warp (rows g, g+1, four
// 8-id groups each) fall on distinct bank groups.  The producer forms every chunk's record of
// the chunk-Gumbel contract in the registers that hold its z (produce_cg below); z is never
// stored.
// --------------------------------------------------------------------------------------------
constexpr int kStageRow = kTS + 32;  // ids per staged row (2112 bytes)

// Row-block W1 fragments in shared memory, interleaved so that one 16-byte load is a whole A
// fragment: unit (s, g, tq) [s = k-step, g = 0..7, tq = 0..3] holds the four 32-bit words
// {W1 row g, row g + 8} x {k0 .. k0 + 1, k0 + 2 .. k0 + 3}, k0 = tq r/4 + 4 s, in MMA order
// (a0 a1 a2 a3); a quarter-warp reads 8 consecutive units.  unit index = (s * 8 + g) * 4 + tq.
template <int KS>
__host__ __device__ constexpr int w1_units() {
    return KS * 32;
}

// z of one chunk for rows g and g + 8 in MMA accumulator layout: acc[nt] = {row g: ids
// 8 tq + 2 nt, +1; row g + 8: the same ids}; acc holds the base values on entry.
template <int KS, bool W2SMEM, bool FULL>
__device__ __forceinline__ void mma_chunk_frag(float (&acc)[4][4], const uint4* w1i, const uint16_t* W2,
                                               const uint4* w2s, int tile0, int c, int V, int g, int tq) {
    constexpr int r = 16 * KS;
    constexpr int units = w2_units<KS>();
    constexpr int mask = w2_mask<KS>();
#pragma unroll
    for (int s = 0; s < KS; s += 2) {  // k-steps s and s + 1 share a 16-byte unit of W2
        const uint4 ua = w1i[(s * 8 + g) * 4 + tq];
        uint4 ub = make_uint4(0u, 0u, 0u, 0u);
        if (s + 1 < KS) ub = w1i[((s + 1) * 8 + g) * 4 + tq];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int vl = kCS * c + 8 * (g >> 1) + 2 * nt + (g & 1);
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if (FULL || tile0 + vl < V) {
                if constexpr (KS == 1) {
                    const int u = tq >> 1, half = tq & 1;
                    uint2 v;
                    if constexpr (W2SMEM) v = reinterpret_cast<const uint2*>(w2s + (size_t)vl * units + (u ^ (vl & mask)))[half];
                    else v = __ldg(reinterpret_cast<const uint2*>(W2 + (size_t)(tile0 + vl) * r + tq * (r / 4)));
                    w.x = v.x;
                    w.y = v.y;
                } else {
                    const int u = tq * (KS / 2) + s / 2;
                    if constexpr (W2SMEM) w = w2s[(size_t)vl * units + (u ^ (vl & mask))];
                    else w = __ldg(reinterpret_cast<const uint4*>(W2 + (size_t)(tile0 + vl) * r + tq * (r / 4)) + s / 2);
                }
            }
            mma4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3], ua.x, ua.y, ua.z, ua.w, w.x, w.y);
            if (s + 1 < KS) mma4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3], ub.x, ub.y, ub.z, ub.w, w.z, w.w);
        }
    }
}

// --------------------------------------------------------------------------------------------
// Chunk-Gumbel draft sampling (dspark.h): every chunk's record is formed where its z values sit,
// in the lane quad that holds them (lane tq: ids 8 tq .. 8 tq + 7 of the chunk):
//   T > 0: {key = LSE_c - ln E_c, LSE_c, candidate by the in-chunk inverse CDF of u, z at it}
//          (natural-log units; a chunk without mass: {-inf, -inf, -1, 0});
//   greedy: {max z, NaN, lowest argmax, max z}.
// --------------------------------------------------------------------------------------------
__device__ __forceinline__ float4 chunk_record_cg(const float (&z)[8], int id0, float scale2, float lnE, float u) {
    const int lane = threadIdx.x & 31, tq = lane & 3;
    float m = z[0];
#pragma unroll
    for (int e = 1; e < 8; ++e) m = fmaxf(m, z[e]);
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const float m2 = m * scale2;
    const float mref = (m2 == -CUDART_INF_F) ? 0.f : m2;
    float cum[8];
    float run = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        run += ex2(fmaf(z[e], scale2, -mref));
        cum[e] = run;
    }
    // in-order prefix over the quad, summed left to right so that a lane's end is exactly the
    // next lane's start (the crossing lane is then unique)
    const float r0 = __shfl_sync(0xffffffffu, run, 0, 4);
    const float r1 = __shfl_sync(0xffffffffu, run, 1, 4);
    const float r2 = __shfl_sync(0xffffffffu, run, 2, 4);
    const float r3 = __shfl_sync(0xffffffffu, run, 3, 4);
    const float b2 = r0 + r1, b3 = b2 + r2, S = b3 + r3;
    const float before = tq == 0 ? 0.f : (tq == 1 ? r0 : (tq == 2 ? b2 : b3));
    const float target = u * S;
    // the lane holding the first crossing: cumulative mass reaches past target inside it
    const bool mine = before <= target && before + run > target;  // before + run == next lane's start
    // first id of this lane whose cumulative mass passes target (the last one when rounding
    // leaves none), and its z
    const float tl = target - before;
    int e_star = 7;
    float z_star = z[7];
#pragma unroll
    for (int e = 6; e >= 0; --e) {  // selects, not branches
        const bool past = cum[e] > tl;
        e_star = past ? e : e_star;
        z_star = past ? z[e] : z_star;
    }
    const unsigned quad = (unsigned)(lane & ~3);
    const unsigned bal = (__ballot_sync(0xffffffffu, mine) >> quad) & 0xFu;
    int src = bal ? (__ffs(bal) - 1) : 0;
    int my_e = e_star;
    float zsel = z_star;
    if (__any_sync(0xffffffffu, bal == 0u && S > 0.f)) {
        // rounding left no crossing in some quad: there, the last id with mass
        int lz = -1;
        float zl = z[0];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const bool has_e = ex2(fmaf(z[e], scale2, -mref)) > 0.f;
            lz = has_e ? e : lz;
            zl = has_e ? z[e] : zl;
        }
        const unsigned nzb = (__ballot_sync(0xffffffffu, lz >= 0) >> quad) & 0xFu;
        if (!bal) {
            src = nzb ? 31 - __clz(nzb) : 0;
            my_e = max(lz, 0);
            zsel = zl;
        }
    }
    const int e_src = __shfl_sync(0xffffffffu, my_e, src, 4);
    const float z_src = __shfl_sync(0xffffffffu, zsel, src, 4);
    const bool has = S > 0.f;  // a chunk without mass: {-inf, -inf, -1, 0}
    const float lmass = has ? (m2 + lg2(S)) * kLn2 : -CUDART_INF_F;
    return make_float4(lmass - lnE, lmass, __int_as_float(has ? id0 - 8 * tq + 8 * src + e_src : -1), has ? z_src : 0.f);
}

// Two records of one request merged: the higher key wins (the first on ties: callers pass the
// lower ids first); T > 0 also the log-sum of the log-masses (natural units).
__device__ __forceinline__ float log_add(float a, float b) {
    const float m = fmaxf(a, b);
    if (m == -CUDART_INF_F) return m;
    return m + lg2(1.0f + ex2((fminf(a, b) - m) * kLog2e)) * kLn2;
}
__device__ __forceinline__ float4 merge_rec(const float4 lo, const float4 hi, bool greedy) {
    const bool take = hi.x > lo.x;
    float4 r = take ? hi : lo;
    if (!greedy) r.y = log_add(lo.y, hi.y);
    return r;
}

template <int KS, bool GREEDY, bool W2SMEM, bool FULL>
__device__ __forceinline__ void produce_cg(const uint16_t* stage, const uint4* w1i, const uint16_t* W2,
                                           const uint4* w2s, int V, int tile, float4* crec, float scale2,
                                           const float* lnEt, int ld, const float* urow, int nv, float softcap,
                                           float inv_softcap) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int tile0 = tile * kTS;
    const uint16_t* srowA = stage + g * kStageRow;
    const uint16_t* srowB = stage + (g + 8) * kStageRow;
    // rows past the valid ones compute on stale data and are never reduced: clamp their table reads
    const int ga = min(g, nv - 1), gb = min(g + 8, nv - 1);
    float uA = 0.f, uB = 0.f;
    if constexpr (!GREEDY) {
        uA = urow[ga];
        uB = urow[gb];
    }
    const float4 empty = GREEDY ? make_float4(-CUDART_INF_F, CUDART_NAN_F, __int_as_float(0x7fffffff), -CUDART_INF_F)
                                : make_float4(-CUDART_INF_F, -CUDART_INF_F, __int_as_float(-1), 0.f);
    float4 accA = empty, accB = empty;  // this warp's chunks merged, rows g and g + 8
#pragma unroll 1
    for (int k = 0; k < kChunksPerWarp; ++k) {
        const int c = warp + kWarps * k;
        const int cb = tile0 + kCS * c;
        if (!FULL && cb >= V) continue;
        float acc[4][4];
        {
            const uint4 wa = *reinterpret_cast<const uint4*>(srowA + kCS * c + 8 * tq);
            const uint4 wb = *reinterpret_cast<const uint4*>(srowB + kCS * c + 8 * tq);
            const uint32_t pa[4] = {wa.x, wa.y, wa.z, wa.w}, pb[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                acc[nt][0] = bf16_lo(pa[nt]);
                acc[nt][1] = bf16_hi(pa[nt]);
                acc[nt][2] = bf16_lo(pb[nt]);
                acc[nt][3] = bf16_hi(pb[nt]);
            }
            if (softcap > 0.f) {  // (ids past V are set to -inf just below)
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int h = 0; h < 4; ++h) acc[nt][h] = softcap * tanh_def(acc[nt][h] * inv_softcap);
            }
            if (!FULL) {  // ids past V take no part
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        if (cb + 8 * tq + 2 * nt + h >= V) {
                            acc[nt][h] = -CUDART_INF_F;
                            acc[nt][2 + h] = -CUDART_INF_F;
                        }
            }
        }
        mma_chunk_frag<KS, W2SMEM, FULL>(acc, w1i, W2, w2s, tile0, c, V, g, tq);
        float xa[8], xb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            xa[e] = acc[e >> 1][e & 1];
            xb[e] = acc[e >> 1][2 + (e & 1)];
        }
        float4 ra, rbk;
        if constexpr (GREEDY) {
            const float2 sa = chunk_stats(xa, cb + 8 * tq, 1);
            const float2 sb = chunk_stats(xb, cb + 8 * tq, 1);
            ra = make_float4(sa.x, CUDART_NAN_F, sa.y, sa.x);
            rbk = make_float4(sb.x, CUDART_NAN_F, sb.y, sb.x);
        } else {
            ra = chunk_record_cg(xa, cb + 8 * tq, scale2, lnEt[c * ld + ga], uA);
            rbk = chunk_record_cg(xb, cb + 8 * tq, scale2, lnEt[c * ld + gb], uB);
        }
        accA = merge_rec(accA, ra, GREEDY);  // chunks in increasing order: ties keep the lower id
        accB = merge_rec(accB, rbk, GREEDY);
    }
    if (tq == 0) {
        crec[g * kWarps + warp] = accA;
        crec[(g + 8) * kWarps + warp] = accB;
    }
}

// A row's tile record from its per-warp records crow[0 .. kWarps) (one warp; lanes 16 .. 31
// mirror lanes 0 .. 15): the arg-max (the lower warp, i.e. the lower ids, on ties) and the
// maximum log-mass share one shuffle tree, then the sum of the log-masses' exponentials.
__device__ __forceinline__ float4 reduce_row_chunks(const float4* crow, bool greedy) {
    static_assert(kWarps == 16, "one lane per producing warp in a half-warp");
    const int lane = threadIdx.x & 31;
    const float4 q = crow[lane & 15];
    float key = q.x, ym = q.y;
    int who = lane & 15;
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, key, o);
        const int ow = __shfl_xor_sync(0xffffffffu, who, o);
        const bool take = ok > key || (ok == key && ow < who);
        key = take ? ok : key;
        who = take ? ow : who;
        if (!greedy) ym = fmaxf(ym, __shfl_xor_sync(0xffffffffu, ym, o));
    }
    const float4 w = crow[who];
    if (greedy) return make_float4(key, CUDART_NAN_F, w.z, w.w);
    float sum = (q.y == -CUDART_INF_F) ? 0.f : ex2((q.y - ym) * kLog2e);
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float lm = (ym == -CUDART_INF_F) ? -CUDART_INF_F : ym + lg2(sum) * kLn2;
    return make_float4(key, lm, w.z, w.w);
}

// --------------------------------------------------------------------------------------------
// Tile record of one row under the chunk-Gumbel contract (one warp, lane = chunk) from its 32
// chunk statistics and its buffered z values xrow (weights 2^(x * lscale)):
// {max over chunks of LSE_c - ln E_c, the tile's log-mass, the candidate of the winning chunk by
// the in-chunk inverse CDF of u, z at it}; greedy: {max, NaN, argmax id, max}.  The chunk
// variates are drawn here (one Philox call per lane, draw n = global chunk index, purpose p_chunk:
// the draft draw's or a verify correction's).
// --------------------------------------------------------------------------------------------
__device__ __forceinline__ float4 finalize_tile_cg(const float* xrow, float2 cs, int tile, int V, int greedy,
                                                   float lscale, float u, uint64_t seed, uint32_t j, uint32_t i,
                                                   uint32_t p_chunk) {
    const int lane = threadIdx.x & 31;
    const int tile0 = tile * kTS;
    const bool valid = tile0 + kCS * lane < V;
    if (greedy) {
        float m = valid ? cs.x : -CUDART_INF_F;
        int idx = valid ? __float_as_int(cs.y) : 0x7fffffff;
        warp_argmax(m, idx);
        return make_float4(m, CUDART_NAN_F, __int_as_float(idx), m);
    }
    const float mc = valid ? cs.x : -CUDART_INF_F;
    const float sc = valid ? cs.y : 0.f;
    const float lnE = log_neg_log_u(uniform(seed, j, i, p_chunk, (uint32_t)(tile * kChunks + lane)));
    float key = (sc > 0.f) ? (mc + lg2(sc)) * kLn2 - lnE : -CUDART_INF_F;
    int who = lane;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, key, o);
        const int ow = __shfl_xor_sync(0xffffffffu, who, o);
        if (ok > key || (ok == key && ow < who)) {
            key = ok;
            who = ow;
        }
    }
    const float mt = warp_max(mc);
    if (mt == -CUDART_INF_F || key == -CUDART_INF_F)
        return make_float4(-CUDART_INF_F, -CUDART_INF_F, __int_as_float(-1), 0.f);
    const float St = warp_sum((sc > 0.f) ? sc * ex2(mc - mt) : 0.f);
    const float lmass = (mt + lg2(St)) * kLn2;
    // id by u inside chunk `who` (masses relative to its own maximum)
    const float mcs = __shfl_sync(0xffffffffu, mc, who);
    const int vl = kCS * who + lane;
    const float xv = xrow[vl];
    const float e = (tile0 + vl < V) ? ex2(xv * lscale - mcs) : 0.f;
    const float Q = warp_incl_scan(e);
    const float Sc = __shfl_sync(0xffffffffu, Q, 31);
    const unsigned hit = __ballot_sync(0xffffffffu, Q > u * Sc);
    int xl;
    if (hit) {
        xl = __ffs(hit) - 1;
    } else {
        const unsigned nz = __ballot_sync(0xffffffffu, e > 0.f);
        xl = nz ? 31 - __clz(nz) : 0;
    }
    const float zv = __shfl_sync(0xffffffffu, xv, xl);
    return make_float4(key, lmass, __int_as_float(tile0 + kCS * who + xl), zv);
}

// Running reduction of tile records: the highest key wins (lowest tile on ties); the tiles'
// log-masses are merged into a log-sum-exp on the fly.
struct TileAcc {
    float key, val, m, s;
    int tile, cand;
};
__device__ __forceinline__ TileAcc tile_acc_init() {
    return TileAcc{-CUDART_INF_F, 0.f, -CUDART_INF_F, 0.f, 0x7fffffff, -1};
}
// Merge over `width` consecutive lanes (a power of two <= 32); every lane of the warp calls it.
__device__ __forceinline__ void tile_acc_shfl_merge(TileAcc& a, int width, bool want_lse) {
    for (int o = 1; o < width; o <<= 1) {
        TileAcc b;
        b.key = __shfl_xor_sync(0xffffffffu, a.key, o);
        b.tile = __shfl_xor_sync(0xffffffffu, a.tile, o);
        b.cand = __shfl_xor_sync(0xffffffffu, a.cand, o);
        b.val = __shfl_xor_sync(0xffffffffu, a.val, o);
        b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
        b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
        if (b.tile != 0x7fffffff && (a.tile == 0x7fffffff || b.key > a.key || (b.key == a.key && b.tile < a.tile))) {
            a.key = b.key;
            a.tile = b.tile;
            a.cand = b.cand;
            a.val = b.val;
        }
        if (want_lse) {
            const float M = fmaxf(a.m, b.m);
            a.s = (M == -CUDART_INF_F) ? 0.f
                                       : (a.m == -CUDART_INF_F ? 0.f : a.s * ex2(a.m - M)) +
                                             (b.m == -CUDART_INF_F ? 0.f : b.s * ex2(b.m - M));
            a.m = M;
        }
    }
}
// ln of the merged log-sum-exp (natural units).
__device__ __forceinline__ float tile_acc_lse(const TileAcc& a) {
    return a.m == -CUDART_INF_F ? -CUDART_INF_F : (a.m + lg2(a.s)) * kLn2;
}

// Reduction of one request's tile records rec[0..nt) by `width` consecutive lanes starting at a
// multiple of `width` (sub = lane index within the group); records are loaded in batches of 8
// per lane before they are used, so a batch costs one memory round trip.
template <int kBatch = 8>
__device__ __forceinline__ TileAcc reduce_tiles_group(const float4* rec, int nt, int sub, int width, bool want_lse) {
    TileAcc acc = tile_acc_init();
    for (int t0 = sub; t0 < nt; t0 += width * kBatch) {
        float4 q[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int t = t0 + width * k;
            q[k] = t < nt ? __ldcg(rec + t) : make_float4(-CUDART_INF_F, -CUDART_INF_F, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int t = t0 + width * k;  // ascending: equal keys keep the lower tile
            if (t < nt && (acc.tile == 0x7fffffff || q[k].x > acc.key)) {
                acc.key = q[k].x;
                acc.tile = t;
                acc.cand = __float_as_int(q[k].z);
                acc.val = q[k].w;
            }
        }
        if (want_lse) {
            float bm = -CUDART_INF_F;
#pragma unroll
            for (int k = 0; k < kBatch; ++k) bm = fmaxf(bm, q[k].y);  // padding is -inf
            if (bm != -CUDART_INF_F) {
                const float bm2 = bm * kLog2e;
                float bs = 0.f;
#pragma unroll
                for (int k = 0; k < kBatch; ++k) bs += ex2(fmaf(q[k].y, kLog2e, -bm2));
                const float M = fmaxf(acc.m, bm2);
                acc.s = (acc.m == -CUDART_INF_F ? 0.f : acc.s * ex2(acc.m - M)) + bs * ex2(bm2 - M);
                acc.m = M;
            }
        }
    }
    tile_acc_shfl_merge(acc, width, want_lse);
    return acc;
}

}  // namespace dspark
