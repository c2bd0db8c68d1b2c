// markov_tile.cuh -- the per-tile building blocks shared by the sampling and verify kernels.
//
// A "tile" is DSPARK_TILE consecutive vocabulary ids; a "row block" is 16 rows (requests).
// Producers compute z = base + W2 . W1[prev] for a row block over one tile into a shared
// memory buffer (fp32, padded stride) and, optionally, per-32-id chunk statistics.
// finalize_tile() turns a row's chunk statistics and buffered values into the tile's record
// of the tile-Gumbel contract (dspark.h): log-mass, Gumbel key, and the in-tile inverse-CDF
// candidate, drawn speculatively before the winning tile is known.
#pragma once

#include "common.cuh"

namespace dspark {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTS = DSPARK_TILE;
constexpr int kChunks = kTS / 32;
constexpr int kRows = 16;
constexpr int kSRow = kTS + 4;  // padded row stride (floats): the 16-byte stores of a quarter-warp are conflict-free
static_assert(kChunks == 32, "one warp lane per chunk");

// Per-row inputs of a row block, staged in shared memory by the caller.
struct RowBlock {
    int prev[kRows];      // W1 row (previous token) of each row
    long long brow[kRows];  // element offset of the row's base logits (-1: row not computed)
};

__device__ __forceinline__ float2 empty_stat(int greedy) {
    return greedy ? make_float2(-CUDART_INF_F, __int_as_float(0x7fffffff)) : make_float2(-CUDART_INF_F, 0.f);
}

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
    uint32_t w[2 * KS];  // the lane's r/4 weights of one row, as bf16 pairs
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

// Stage W2 rows [tile0, tile0 + kTS) into shared memory (swizzled); rows past V are zero.
template <int KS>
__device__ void stage_w2_tile(const uint16_t* W2, int tile0, int V, uint4* dst) {
    constexpr int units = w2_units<KS>();
    constexpr int mask = w2_mask<KS>();
    for (int idx = threadIdx.x; idx < kTS * units; idx += blockDim.x) {
        const int vl = idx / units, u = idx % units;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (tile0 + vl < V) v = __ldg(reinterpret_cast<const uint4*>(W2 + (size_t)(tile0 + vl) * (16 * KS)) + u);
        dst[vl * units + (u ^ (vl & mask))] = v;
    }
}

template <typename TL>
__device__ __forceinline__ void load_vals8(const TL* row, int v0, int V, bool vec, float (&x)[8]) {
    if (vec && v0 + 8 <= V) {
        load8<TL>(row, (size_t)v0, x);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = (v0 + e < V) ? load_logit<TL>(row, (size_t)(v0 + e)) : -CUDART_INF_F;
    }
}

// Chunk statistics of 8 values per lane, combined over the lane quad (tq = 0..3 hold ids
// 8*tq.. of the chunk).  T > 0: (max s2, sum 2^(s2 - max)) with s2 = x * scale2;
// greedy: (max x, lowest argmax id).
__device__ __forceinline__ float2 quad_stats(const float (&z)[8], int id0, int greedy, float scale2) {
    if (greedy) {
        float m = z[0];
        int idx = id0;
#pragma unroll
        for (int e = 1; e < 8; ++e)
            if (z[e] > m) {
                m = z[e];
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
    float s[8];
    float m = -CUDART_INF_F;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        s[e] = z[e] * scale2;
        m = fmaxf(m, s[e]);
    }
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    float acc = 0.f;
    if (m != -CUDART_INF_F) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc += ex2(s[e] - m);
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    return make_float2(m, acc);
}

// z = base + bias for the row block over one tile, tensor-core path.  Writes zbuf[16][kSRow]
// and, when `stats`, cstat[16][kChunks].  Rows with brow < 0 get A = 0 and base = 0.
template <typename TL, int KS>
__device__ inline void produce_z_mma(const TL* base, const uint16_t* W1, const uint16_t* W2, const uint4* w2s, int V,
                              bool vec_ok, int tile, const RowBlock& rb, float* zbuf, float2* cstat, bool stats,
                              int greedy, float scale2) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    const bool okA = rb.brow[g] >= 0, okB = rb.brow[g + 8] >= 0;
    Frag<KS> fa, fb;
    if (okA) load_frag_global<KS>(W1, rb.prev[g], tq, fa);
    else frag_zero<KS>(fa);
    if (okB) load_frag_global<KS>(W1, rb.prev[g + 8], tq, fb);
    else frag_zero<KS>(fb);
    const TL* rowA = base + (okA ? rb.brow[g] : 0);
    const TL* rowB = base + (okB ? rb.brow[g + 8] : 0);
    const int tile0 = tile * kTS;
    for (int c = warp; c < kChunks; c += kWarps) {
        const int cb = tile0 + 32 * c;
        if (cb >= V) {
            if (stats && tq == 0) {
                cstat[g * kChunks + c] = empty_stat(greedy);
                cstat[(g + 8) * kChunks + c] = empty_stat(greedy);
            }
            continue;
        }
        float xa[8], xb[8];
        if (okA) load_vals8<TL>(rowA, cb + 8 * tq, V, vec_ok, xa);
        else
#pragma unroll
            for (int e = 0; e < 8; ++e) xa[e] = 0.f;
        if (okB) load_vals8<TL>(rowB, cb + 8 * tq, V, vec_ok, xb);
        else
#pragma unroll
            for (int e = 0; e < 8; ++e) xb[e] = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            float d[4] = {xa[2 * nt], xa[2 * nt + 1], xb[2 * nt], xb[2 * nt + 1]};
            const int vcol = cb + 8 * (g >> 1) + 2 * nt + (g & 1);  // id this lane feeds as MMA column g
            Frag<KS> fw;
            if (vcol < V) {
                if (w2s) load_frag_smem<KS>(w2s, vcol - tile0, tq, fw);
                else load_frag_global<KS>(W2, vcol, tq, fw);
            } else {
                frag_zero<KS>(fw);
            }
#pragma unroll
            for (int s = 0; s < KS; ++s)
                mma_bf16(d, fa.w[2 * s], fb.w[2 * s], fa.w[2 * s + 1], fb.w[2 * s + 1], fw.w[2 * s], fw.w[2 * s + 1]);
            xa[2 * nt] = d[0];
            xa[2 * nt + 1] = d[1];
            xb[2 * nt] = d[2];
            xb[2 * nt + 1] = d[3];
        }
        float4* zA = reinterpret_cast<float4*>(zbuf + g * kSRow + 32 * c + 8 * tq);
        float4* zB = reinterpret_cast<float4*>(zbuf + (g + 8) * kSRow + 32 * c + 8 * tq);
        zA[0] = make_float4(xa[0], xa[1], xa[2], xa[3]);
        zA[1] = make_float4(xa[4], xa[5], xa[6], xa[7]);
        zB[0] = make_float4(xb[0], xb[1], xb[2], xb[3]);
        zB[1] = make_float4(xb[4], xb[5], xb[6], xb[7]);
        if (stats) {
            const float2 sA = quad_stats(xa, cb + 8 * tq, greedy, scale2);
            const float2 sB = quad_stats(xb, cb + 8 * tq, greedy, scale2);
            if (tq == 0) {
                cstat[g * kChunks + c] = sA;
                cstat[(g + 8) * kChunks + c] = sB;
            }
        }
    }
}

// CUDA-core path (fp32 weights, ranks not in {16,...,256}, r = 0).  Lane = id; the W1 rows of
// the row block are staged as fp32 in w1s[16][r] by the caller.
template <typename TL, typename TW>
__device__ void produce_z_gemv(const TL* base, const TW* W2, const float* w1s, int r, int V, int tile,
                               const RowBlock& rb, float* zbuf, float2* cstat, bool stats, int greedy,
                               float scale2) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile0 = tile * kTS;
    for (int c = warp; c < kChunks; c += kWarps) {
        const int cb = tile0 + 32 * c;
        if (cb >= V) {
            if (stats && lane < kRows) cstat[lane * kChunks + c] = empty_stat(greedy);
            continue;
        }
        const int v = cb + lane;
        const bool vok = v < V;
        float acc[kRows];
#pragma unroll
        for (int q = 0; q < kRows; ++q) acc[q] = 0.f;
        for (int k0 = 0; k0 < r; k0 += 8) {
            float w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = (vok && k0 + e < r) ? load_logit<TW>(W2, (size_t)v * r + k0 + e) : 0.f;
#pragma unroll
            for (int q = 0; q < kRows; ++q) {
                const float* w1 = w1s + q * r + k0;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (k0 + e < r) acc[q] = fmaf(w1[e], w[e], acc[q]);
            }
        }
#pragma unroll 1
        for (int q = 0; q < kRows; ++q) {
            float z = -CUDART_INF_F;
            if (vok && rb.brow[q] >= 0) z = load_logit<TL>(base, (size_t)rb.brow[q] + v) + acc[q];
            zbuf[q * kSRow + 32 * c + lane] = z;
            if (stats) {
                float2 st;
                if (greedy) {
                    float m = z;
                    int idx = vok ? v : 0x7fffffff;
                    warp_argmax(m, idx);
                    st = make_float2(m, __int_as_float(idx));
                } else {
                    const float s2 = z * scale2;
                    const float m = warp_max(s2);
                    const float e = (m == -CUDART_INF_F) ? 0.f : ex2(s2 - m);
                    st = make_float2(m, warp_sum(e));
                }
                if (lane == 0) cstat[q * kChunks + c] = st;
            }
        }
    }
}

// --------------------------------------------------------------------------------------------
// Tile record of one row (one warp, lane = chunk).  The buffered value x_v of id v has weight
// 2^(x_v * lscale - m) (lscale = log2(e)/T when the buffer holds z, 1 when it holds log2-weights).
// T > 0 record: {key = ln(mass_t) - ln E_t, ln(mass_t), candidate id, buffered value at it};
// greedy record: {max, NaN, argmax id, max}.  Only lane 0's return value is meaningful.
// --------------------------------------------------------------------------------------------
__device__ inline float4 finalize_tile(const float* xrow, float2 cs, int tile, int V, int greedy, float lscale,
                                uint64_t seed, uint32_t j, uint32_t i, uint32_t p_tile, uint32_t p_intile) {
    const int lane = threadIdx.x & 31;
    const int tile0 = tile * kTS;
    const bool valid = tile0 + 32 * lane < V;
    if (greedy) {
        float m = valid ? cs.x : -CUDART_INF_F;
        int idx = valid ? __float_as_int(cs.y) : 0x7fffffff;
        warp_argmax(m, idx);
        return make_float4(m, CUDART_NAN_F, __int_as_float(idx), m);
    }
    const float mc = valid ? cs.x : -CUDART_INF_F;
    const float sc = valid ? cs.y : 0.f;
    const float mt = warp_max(mc);
    const float w = (sc > 0.f) ? sc * ex2(mc - mt) : 0.f;
    const float P = warp_incl_scan(w);
    const float St = __shfl_sync(0xffffffffu, P, 31);
    if (!(St > 0.f)) {  // no mass in this tile: it can never win
        return make_float4(-CUDART_INF_F, -CUDART_INF_F, __int_as_float(-1), 0.f);
    }
    const float lmass = (mt + lg2(St)) * kLn2;
    float key = 0.f, up = 0.f;
    if (lane == 0) {
        key = lmass - log_neg_log_u(uniform(seed, j, i, p_tile, (uint32_t)tile));
        up = uniform(seed, j, i, p_intile, 0u);
    }
    up = __shfl_sync(0xffffffffu, up, 0);
    const float target = up * St;
    const unsigned hit = __ballot_sync(0xffffffffu, P > target);
    int cstar;
    if (hit) {
        cstar = __ffs(hit) - 1;
    } else {
        const unsigned nz = __ballot_sync(0xffffffffu, w > 0.f);
        cstar = nz ? 31 - __clz(nz) : 0;
    }
    const float before = __shfl_sync(0xffffffffu, P - w, cstar);
    const int vl = 32 * cstar + lane;
    const float xv = xrow[vl];
    const float e = (tile0 + vl < V) ? ex2(xv * lscale - mt) : 0.f;
    const float Q = warp_incl_scan(e) + before;
    const unsigned hit2 = __ballot_sync(0xffffffffu, Q > target);
    int xl;
    if (hit2) {
        xl = __ffs(hit2) - 1;
    } else {
        const unsigned nz = __ballot_sync(0xffffffffu, e > 0.f);
        xl = nz ? 31 - __clz(nz) : 0;
    }
    const float xc = __shfl_sync(0xffffffffu, xv, xl);
    return make_float4(key, lmass, __int_as_float(tile0 + 32 * cstar + xl), xc);
}

// Reduction of a request's tile records (one warp): the highest key wins, lowest tile on ties.
// Returns (candidate, value at it) in lane 0 and, optionally, the log-sum of the tiles' masses.
struct TileWinner {
    int cand;
    float val;
    float key;
    float lse;
};
__device__ inline TileWinner reduce_tiles(const float4* rec, int nt, bool want_lse) {
    const int lane = threadIdx.x & 31;
    float bk = -CUDART_INF_F, bz = 0.f, lmax = -CUDART_INF_F;
    int bt = 0x7fffffff, bc = -1;
    for (int t = lane; t < nt; t += 32) {
        const float4 q = __ldcg(rec + t);
        if (bt == 0x7fffffff || q.x > bk) {  // t ascends: equal keys keep the lower tile
            bk = q.x;
            bt = t;
            bc = __float_as_int(q.z);
            bz = q.w;
        }
        lmax = fmaxf(lmax, q.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
        const int ot = __shfl_xor_sync(0xffffffffu, bt, o);
        const int oc = __shfl_xor_sync(0xffffffffu, bc, o);
        const float oz = __shfl_xor_sync(0xffffffffu, bz, o);
        const bool take = (ot != 0x7fffffff) && (bt == 0x7fffffff || ok > bk || (ok == bk && ot < bt));
        if (take) {
            bk = ok;
            bt = ot;
            bc = oc;
            bz = oz;
        }
    }
    TileWinner wv{bc, bz, bk, CUDART_NAN_F};
    if (want_lse) {
        const float M = warp_max(lmax);
        float s = 0.f;
        if (M != -CUDART_INF_F)
            for (int t = lane; t < nt; t += 32) s += ex2((__ldcg(&rec[t].y) - M) * kLog2e);
        s = warp_sum(s);
        wv.lse = (M == -CUDART_INF_F) ? -CUDART_INF_F : M + logf(s);
    }
    return wv;
}

}  // namespace dspark
