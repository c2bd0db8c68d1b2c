// tv.cu -- dspark_accept_rate_tv: accept-rate targets, eval_mask and tau.
//
// Method (P1 "03 · DSpark 建模：Markov 与 Confidence" section 3.9 "Accept rate 3D" and
// P2 "从 DFlash 到 dLLM Self-Spec（三）" section 3.5): accept = 1 - 0.5 * sum|softmax(d) -
// softmax(t)| clamped to [0,1], computed here as sum_v min(p_v, q_v) (the same quantity with
// no cancellation); min(p, q) = 2^min(d2 - Ld2, t2 - Lt2) needs one exponential per id.
// eval_mask = cumprod of (keep && pos_valid) (P1 section 3.6), tau = 1 + sum_i prod_{k<=i}
// acc_k * mask_k (P1 section 3.10).
//
// Two kernels: tv_rows_kernel (bf16 rows on 16-byte boundaries: a block streams whole rows twice
// through a shared-memory ring fed by the bulk-copy engine, pass 1 from HBM and pass 2 from L2)
// and tv_kernel (any other case: a thread-block cluster shares a row, each block takes a 1/cs
// segment, the blocks exchange (max, sum) through distributed shared memory, and the second
// pass re-reads the segment, an L2 hit).  tau_kernel follows them; tv_l1_kernel is the separate
// training-side L1 term (dspark_tv_l1_loss, P1 section 3.9) on the accept rates.
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "host_util.h"

namespace cg = cooperative_groups;

namespace dspark {
namespace {

constexpr int kTVThreads = 512;
constexpr int kTVWarps = kTVThreads / 32;
constexpr int kUnroll = 4;  // 8-id groups per thread in flight

struct TVArgs {
    long long rows;  // S * A * gamma
    int V, gamma, segsz, nclusters, cs;
    const void* d;
    const void* t;
    const uint8_t* keep;
    const uint8_t* posv;
    float* acc;
    float* mask;
    int vec_ok;
};

template <typename TL>
__device__ __forceinline__ void tv_load8(const TL* row, int v0, int vhi, bool vec, float (&x)[8]) {
    if (vec && v0 + 8 <= vhi) {
        load8<TL>(row, (size_t)v0, x);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = (v0 + e < vhi) ? load_logit<TL>(row, (size_t)(v0 + e)) : -CUDART_INF_F;
    }
}

// (max, sum 2^(x*log2e - max)) of 8 values merged into a running pair (log2 units).
__device__ __forceinline__ void lse_merge8(const float (&x)[8], float& m, float& s) {
    float gm = x[0];
#pragma unroll
    for (int e = 1; e < 8; ++e) gm = fmaxf(gm, x[e]);
    const float mn = fmaxf(m, gm * kLog2e);
    if (mn == -CUDART_INF_F) return;
    s = (m == -CUDART_INF_F) ? 0.f : s * ex2(m - mn);
#pragma unroll
    for (int e = 0; e < 8; ++e) s += ex2(fmaf(x[e], kLog2e, -mn));
    m = mn;
}

__device__ __forceinline__ float2 merge_pair(float2 a, float2 b) {
    const float m = fmaxf(a.x, b.x);
    if (m == -CUDART_INF_F) return make_float2(m, 0.f);
    return make_float2(m, a.y * ex2(a.x - m) + b.y * ex2(b.x - m));
}

template <typename TL>
__global__ void __launch_bounds__(kTVThreads, 1) tv_kernel(TVArgs a) {
    cg::cluster_group cluster = cg::this_cluster();
    const int crank = (int)cluster.block_rank();
    const int cid = blockIdx.x / a.cs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __shared__ float4 xch[2];      // per row parity: (m_d, S_d, m_t, S_t) of this block's segment
    __shared__ float xsum[2];      // per row parity: this block's sum of minima
    __shared__ float4 red4[kTVWarps];
    __shared__ float red1[kTVWarps];
    __shared__ float2 s_norm;      // (Ld2, Lt2) of the row
    const TL* D = reinterpret_cast<const TL*>(a.d);
    const TL* T = reinterpret_cast<const TL*>(a.t);
    const int v_lo = crank * a.segsz, v_hi = min(a.V, v_lo + a.segsz);
    int it = 0;
    for (long long row = cid; row < a.rows; row += a.nclusters, ++it) {
        const int par = it & 1;
        const TL* drow = D + row * (long long)a.V;
        const TL* trow = T + row * (long long)a.V;
        // ---- pass 1: softmax statistics of both rows over the segment
        float md = -CUDART_INF_F, sd = 0.f, mt = -CUDART_INF_F, st = 0.f;
        for (int v0 = v_lo + 8 * tid; v0 < v_hi; v0 += 8 * kTVThreads * kUnroll) {
            float xd[kUnroll][8], xt[kUnroll][8];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int vv = v0 + u * 8 * kTVThreads;
                if (vv < v_hi) {
                    tv_load8<TL>(drow, vv, v_hi, a.vec_ok != 0, xd[u]);
                    tv_load8<TL>(trow, vv, v_hi, a.vec_ok != 0, xt[u]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) xd[u][e] = xt[u][e] = -CUDART_INF_F;
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                lse_merge8(xd[u], md, sd);
                lse_merge8(xt[u], mt, st);
            }
        }
        {
            float2 pd = make_float2(md, sd), pt = make_float2(mt, st);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                pd = merge_pair(pd, make_float2(__shfl_xor_sync(0xffffffffu, pd.x, o), __shfl_xor_sync(0xffffffffu, pd.y, o)));
                pt = merge_pair(pt, make_float2(__shfl_xor_sync(0xffffffffu, pt.x, o), __shfl_xor_sync(0xffffffffu, pt.y, o)));
            }
            if (lane == 0) red4[warp] = make_float4(pd.x, pd.y, pt.x, pt.y);
            __syncthreads();
            if (warp == 0) {
                float4 q = lane < kTVWarps ? red4[lane] : make_float4(-CUDART_INF_F, 0.f, -CUDART_INF_F, 0.f);
                float2 qd = make_float2(q.x, q.y), qt = make_float2(q.z, q.w);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    qd = merge_pair(qd, make_float2(__shfl_xor_sync(0xffffffffu, qd.x, o), __shfl_xor_sync(0xffffffffu, qd.y, o)));
                    qt = merge_pair(qt, make_float2(__shfl_xor_sync(0xffffffffu, qt.x, o), __shfl_xor_sync(0xffffffffu, qt.y, o)));
                }
                if (lane == 0) xch[par] = make_float4(qd.x, qd.y, qt.x, qt.y);
            }
        }
        cluster.sync();  // every block's statistics are visible cluster-wide
        if (tid == 0) {
            float2 gd = make_float2(-CUDART_INF_F, 0.f), gt = make_float2(-CUDART_INF_F, 0.f);
            for (int rnk = 0; rnk < a.cs; ++rnk) {
                const float4 q = cluster.map_shared_rank(&xch[par], rnk)[0];
                gd = merge_pair(gd, make_float2(q.x, q.y));
                gt = merge_pair(gt, make_float2(q.z, q.w));
            }
            s_norm = make_float2(gd.x + lg2(gd.y), gt.x + lg2(gt.y));
        }
        __syncthreads();
        const float Ld2 = s_norm.x, Lt2 = s_norm.y;
        // ---- pass 2: sum of min(p, q) over the segment
        float acc = 0.f;
        for (int v0 = v_lo + 8 * tid; v0 < v_hi; v0 += 8 * kTVThreads * kUnroll) {
            float xd[kUnroll][8], xt[kUnroll][8];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int vv = v0 + u * 8 * kTVThreads;
                if (vv < v_hi) {
                    tv_load8<TL>(drow, vv, v_hi, a.vec_ok != 0, xd[u]);
                    tv_load8<TL>(trow, vv, v_hi, a.vec_ok != 0, xt[u]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) xd[u][e] = xt[u][e] = -CUDART_INF_F;
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc += ex2(fminf(fmaf(xd[u][e], kLog2e, -Ld2), fmaf(xt[u][e], kLog2e, -Lt2)));
        }
        acc = warp_sum(acc);
        if (lane == 0) red1[warp] = acc;
        __syncthreads();
        if (warp == 0) {
            float q = lane < kTVWarps ? red1[lane] : 0.f;
            q = warp_sum(q);
            if (lane == 0) xsum[par] = q;
        }
        cluster.sync();  // partial sums visible
        if (crank == 0 && tid == 0) {
            float tot = 0.f;
            for (int rnk = 0; rnk < a.cs; ++rnk) tot += cluster.map_shared_rank(&xsum[par], rnk)[0];
            a.acc[row] = fminf(fmaxf(tot, 0.f), 1.f);
            const long long blk = row / a.gamma;
            const int i = (int)(row % a.gamma);
            float mval = a.keep[blk] ? 1.f : 0.f;
            if (a.posv)
                for (int k = 0; k <= i; ++k) mval = a.posv[blk * a.gamma + k] ? mval : 0.f;
            a.mask[row] = mval;
        }
    }
    cluster.sync();  // no block leaves while a peer may still read its shared memory
}

// ------------------------------------------------------------------------------------------
// bf16 fast path: one block per row at a time (persistent over rows, no cluster), warp-specialised.
// A producer warp streams every row twice through a ring of kNS shared-memory slots (kCE ids of
// d and t per slot, 32 per consumer thread) with the bulk-copy engine: pass 1 from HBM with an
// L2 evict-last policy, so that pass 2, which follows right after, reads the same bytes from L2
// (evict-first); a slot is refilled once all 16 consumer warps have released it.  The consumer
// warps take the softmax statistics of d and t in pass 1, combine them across the block, then form
// sum_v min(p_v, q_v) = sum_v 2^min(d_v log2e - Ld, t_v log2e - Lt) in pass 2.  Both passes read
// the bf16 values straight from their packed words (mixed-precision subtracts, no unpacking).
// Every wait is bounded; after a timeout the block-wide abort flag makes the consumers skip the
// data while keeping the same sequence of named barriers, and in-flight copies are awaited.
// ------------------------------------------------------------------------------------------
constexpr int kCE = 16384;                // ids per array per slot
constexpr int kNS = 3;                    // ring slots (3 x 64 KB)
constexpr int kWSCons = 512;              // consumer threads (16 warps)
constexpr int kWSWarps = kWSCons / 32;
constexpr int kWSThreads = kWSCons + 32;  // + one producer warp
constexpr int kGrp = kCE / 4;             // ids between a thread's 16-byte groups
static_assert(kCE == 32 * kWSCons, "four 16-byte groups of each array per consumer thread per slot");

struct TVRSmem {
    uint16_t slots[kNS][2][kCE];
    uint64_t full[kNS];
    uint64_t empty[kNS];
    float4 red4[kWSWarps];
    float red1[kWSWarps];
    int abort;
};
constexpr size_t kRowSmem = sizeof(TVRSmem);

struct TVRArgs {
    int rows, V, gamma, nch;
    const __nv_bfloat16* d;
    const __nv_bfloat16* t;
    const uint8_t* keep;
    const uint8_t* posv;
    float* acc;
    float* mask;
    WsHeader* hdr;
    uint64_t limit_ns;
};


// Sum over the 32 ids of 2^min(d log2e - Ld2, t log2e - Lt2), as 2^(log2e min(d - ld, t - lt))
// with ld = Ld2 / log2e, lt = Lt2 / log2e: each difference is one mixed-precision subtract (bf16
// operand taken from its half of the word, fp32 result), the scale one packed multiply per pair.
__device__ __forceinline__ float minsum32w(const uint32_t (&wd)[16], const uint32_t (&wt)[16], uint64_t c2, float ld,
                                           float lt) {
    uint64_t acc[4];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float m0 = fminf(sub_bf16_lo(wd[k], ld), sub_bf16_lo(wt[k], lt));
        const float m1 = fminf(sub_bf16_hi(wd[k], ld), sub_bf16_hi(wt[k], lt));
        const float2 y = up2(mul2(pk2(m0, m1), c2));
        const uint64_t e = pk2(ex2(y.x), ex2(y.y));
        acc[k & 3] = k < 4 ? e : add2(acc[k & 3], e);
    }
    const float2 r = up2(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])));
    return r.x + r.y;
}

// Warp-wide combine of (max, sum 2^(x - max)) pairs: the max first, then one rescale per lane.
__device__ __forceinline__ float2 warp_lse_pair(float m, float s) {
    const float M = warp_max(m);
    const float sc = (m == -CUDART_INF_F) ? 0.f : s * ex2(m - M);
    return make_float2(M, warp_sum(sc));
}

__global__ void __launch_bounds__(kWSThreads, 1) tv_rows_kernel(TVRArgs a) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    TVRSmem& S = *reinterpret_cast<TVRSmem*>(smem_raw);
    volatile int* abort = &S.abort;
    const int nch = a.nch;
    const int nrows = (a.rows - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;  // rows of this block
    const int Q = nrows * 2 * nch;  // chunks: per row, pass 1 then pass 2
    if (tid == 0) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], kWSWarps);
        }
        S.abort = 0;
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == kWSWarps) {
        // ---------------- producer warp
        if (lane == 0) {
            const uint64_t keep_pol = l2_policy_evict_last(), drop_pol = l2_policy_evict_first();
            for (int q = 0; q < Q; ++q) {
                const int slot = q % kNS;
                // the (q / kNS)-th use of the slot waits for the release of its previous use
                if (q >= kNS && !mbar_wait_or_abort(&S.empty[slot], (uint32_t)((q / kNS - 1) & 1), abort,
                                                    &a.hdr->status, a.limit_ns, false))
                    break;
                const int rl = q / (2 * nch), pass = (q / nch) & 1, k = q % nch;
                const int len = min(kCE, a.V - k * kCE);
                const size_t off = (size_t)((int)blockIdx.x + rl * (int)gridDim.x) * a.V + (size_t)k * kCE;
                const uint64_t pol = pass ? drop_pol : keep_pol;
                mbar_arrive_expect_tx(&S.full[slot], (uint32_t)(4 * len));
                bulk_g2s_hint(&S.slots[slot][0][0], a.d + off, (uint32_t)(2 * len), &S.full[slot], pol);
                bulk_g2s_hint(&S.slots[slot][1][0], a.t + off, (uint32_t)(2 * len), &S.full[slot], pol);
            }
        }
        __syncwarp();
    } else {
        // ---------------- 16 consumer warps
        const int my0 = 8 * tid;
        const int tail = a.V - (nch - 1) * kCE;  // ids in the last chunk of a row
        int slot = 0;
        uint32_t phase = 0;
        // After an abort the waits return at once and the slots hold stale data: the arithmetic
        // runs on it (shared-memory reads cannot fault) and the result is never stored.
        auto take = [&](uint32_t (&wd)[16], uint32_t (&wt)[16]) {
            mbar_wait_hint_or_abort(&S.full[slot], phase, abort, &a.hdr->status, a.limit_ns);
            load32w<kGrp>(&S.slots[slot][0][0], my0, wd);
            load32w<kGrp>(&S.slots[slot][1][0], my0, wt);
            __syncwarp();
            if (lane == 0) mbar_arrive_local(&S.empty[slot]);
            if (++slot == kNS) {
                slot = 0;
                phase ^= 1u;
            }
        };
        const uint64_t c2 = pk2(kLog2e, kLog2e);
        for (int rl = 0; rl < nrows; ++rl) {
            // ---- pass 1: softmax statistics of d and t (log2 domain)
            float md = -CUDART_INF_F, sd = 0.f, mt = -CUDART_INF_F, st = 0.f;
            for (int k = 0; k < nch - 1; ++k) {
                uint32_t wd[16], wt[16];
                take(wd, wt);
                lse_step32w(wd, kLog2e, kLn2, c2, md, sd);
                lse_step32w(wt, kLog2e, kLn2, c2, mt, st);
            }
            {
                uint32_t wd[16], wt[16];
                take(wd, wt);
                mask_tail32<kGrp>(wd, my0, tail);
                mask_tail32<kGrp>(wt, my0, tail);
                lse_step32w(wd, kLog2e, kLn2, c2, md, sd);
                lse_step32w(wt, kLog2e, kLn2, c2, mt, st);
            }
            {
                const float2 wdp = warp_lse_pair(md, sd);
                const float2 wtp = warp_lse_pair(mt, st);
                if (lane == 0) S.red4[warp] = make_float4(wdp.x, wdp.y, wtp.x, wtp.y);
            }
            named_barrier(1, kWSCons);
            float Ld2, Lt2;
            {
                const float4 v = lane < kWSWarps ? S.red4[lane] : make_float4(-CUDART_INF_F, 0.f, -CUDART_INF_F, 0.f);
                const float2 cd = warp_lse_pair(v.x, v.y);
                const float2 ct = warp_lse_pair(v.z, v.w);
                Ld2 = cd.x + lg2(cd.y);
                Lt2 = ct.x + lg2(ct.y);
            }
            // ---- pass 2: sum of min(p, q) = 2^min(d log2e - Ld2, t log2e - Lt2)
            const float ld = Ld2 * kLn2, lt = Lt2 * kLn2;  // the normalisers in the logits' units
            float acc = 0.f;
            for (int k = 0; k < nch - 1; ++k) {
                uint32_t wd[16], wt[16];
                take(wd, wt);
                acc += minsum32w(wd, wt, c2, ld, lt);
            }
            {
                uint32_t wd[16], wt[16];
                take(wd, wt);
                mask_tail32<kGrp>(wd, my0, tail);
                mask_tail32<kGrp>(wt, my0, tail);
                acc += minsum32w(wd, wt, c2, ld, lt);
            }
            const float w = warp_sum(acc);
            if (lane == 0) S.red1[warp] = w;
            named_barrier(2, kWSCons);
            if (warp == 0) {
                const float v = warp_sum(lane < kWSWarps ? S.red1[lane] : 0.f);
                if (lane == 0 && !*abort) {
                    const int row = (int)blockIdx.x + rl * (int)gridDim.x;
                    a.acc[row] = fminf(fmaxf(v, 0.f), 1.f);
                    const int blk = row / a.gamma, i = row % a.gamma;
                    float mval = a.keep[blk] ? 1.f : 0.f;
                    if (a.posv)
                        for (int kk = 0; kk <= i; ++kk) mval = a.posv[(size_t)blk * a.gamma + kk] ? mval : 0.f;
                    a.mask[row] = mval;
                }
            }
        }
    }
    __syncthreads();
    // copies still in flight after an abort: wait for them (bounded) before the block leaves
    if (tid == 0 && *abort) {
        const uint64_t t0 = global_ns();
        for (int qq = max(0, Q - kNS); qq < Q; ++qq) {
            const int sl = qq % kNS;
            while (!mbar_try_wait(&S.full[sl], (uint32_t)((qq / kNS) & 1)) && global_ns() - t0 < a.limit_ns) {
            }
        }
    }
}

// tau[s,a] = 1 + sum_i prod_{k<=i} acc * mask (one thread per block of gamma positions).
__global__ void tau_kernel(long long nblk, int gamma, const float* acc, const float* mask, float* tau) {
    const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblk) return;
    float prod = 1.f, expected = 0.f;
    for (int i = 0; i < gamma; ++i) {
        prod *= acc[b * gamma + i] * mask[b * gamma + i];
        expected += prod;
    }
    tau[b] = 1.f + expected;
}

// Training-side L1 term over the accept rates of a batch: l1 = sum_v |p - q| = 2 (1 - accept) per
// position (accept = sum_v min(p, q)), position weights w_k = exp(-(k-1)/decay) for k = 1..gamma,
// numerator sum w mask l1 and denominator sum w mask.  One block; every thread adds its elements in
// index order in fp64 and the block adds the threads in a fixed tree, so the sums are deterministic.
constexpr int kL1Threads = 512;
constexpr int kL1MaxGamma = 1024;  // positions per block (the sampling calls accept gamma <= 1024 too)
__global__ void __launch_bounds__(kL1Threads) tv_l1_kernel(long long n, int gamma, const float* __restrict__ acc,
                                                           const float* __restrict__ mask, double decay,
                                                           float* __restrict__ l1, double* __restrict__ sums) {
    __shared__ double red[2][kL1Threads / 32];
    __shared__ double wtab[kL1MaxGamma];  // w_k = exp(-(k - 1) / decay), one per position
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int k = tid; k < gamma; k += kL1Threads) wtab[k] = exp(-(double)k / decay);
    __syncthreads();
    double num = 0.0, den = 0.0;
    for (long long e = tid; e < n; e += kL1Threads) {
        const int k = (int)(e % gamma);  // position k + 1
        const float d = 2.f * (1.f - acc[e]);
        if (l1) l1[e] = d;
        const double w = wtab[k] * (double)mask[e];
        num += w * (double)d;
        den += w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        num += __shfl_xor_sync(0xffffffffu, num, o);
        den += __shfl_xor_sync(0xffffffffu, den, o);
    }
    if (lane == 0) {
        red[0][warp] = num;
        red[1][warp] = den;
    }
    __syncthreads();
    if (warp == 0) {
        num = lane < kL1Threads / 32 ? red[0][lane] : 0.0;
        den = lane < kL1Threads / 32 ? red[1][lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            num += __shfl_xor_sync(0xffffffffu, num, o);
            den += __shfl_xor_sync(0xffffffffu, den, o);
        }
        if (lane == 0) {
            sums[0] = num;
            sums[1] = den;
        }
    }
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_accept_rate_tv_workspace_size(int S, int A, int gamma, int V, int dtype) {
    (void)S; (void)A; (void)gamma; (void)V; (void)dtype;
    return kHeaderBytes;  // the status word
}

extern "C" dspark_status dspark_accept_rate_tv(int S, int A, int gamma, int V, int dtype, const void* draft_logits,
                                               const void* target_logits, const uint8_t* block_keep,
                                               const uint8_t* pos_valid, float* accept_rate, float* eval_mask,
                                               float* tau, void* workspace, size_t ws_bytes, dspark_stream_t stream) {
    if (S < 1 || A < 1 || gamma < 1 || V < 1) return DSPARK_ERR_INVALID_ARG;
    if (dtype != DSPARK_F32 && dtype != DSPARK_BF16) return DSPARK_ERR_INVALID_ARG;
    if (!draft_logits || !target_logits || !block_keep || !accept_rate || !eval_mask) return DSPARK_ERR_INVALID_ARG;
    if (!workspace || ((uintptr_t)workspace & 255u) || ws_bytes < kHeaderBytes) return DSPARK_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, kHeaderBytes, s) != cudaSuccess) return DSPARK_ERR_CUDA;

    const long long rows = (long long)S * A * gamma;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    cfg.blockDim = dim3(kTVThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool tma = dtype == DSPARK_BF16 && V % 8 == 0 && (uintptr_t)draft_logits % 16 == 0 &&
                     (uintptr_t)target_logits % 16 == 0 && V >= 16;
    int per_sm = 0;
    if (tma && prepare_kernel((const void*)tv_rows_kernel, kRowSmem, kWSThreads, &per_sm) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    if (tma && per_sm > 0 && rows <= (long long)INT32_MAX / 2) {
        int sms = 0;
        if (device_sm_count(&sms) != cudaSuccess) return DSPARK_ERR_CUDA;
        const long long G = std::min<long long>(rows, (long long)sms * per_sm);
        TVRArgs a;
        a.rows = (int)rows;
        a.V = V;
        a.gamma = gamma;
        a.nch = (V + kCE - 1) / kCE;
        a.d = static_cast<const __nv_bfloat16*>(draft_logits);
        a.t = static_cast<const __nv_bfloat16*>(target_logits);
        a.keep = block_keep;
        a.posv = pos_valid;
        a.acc = accept_rate;
        a.mask = eval_mask;
        a.hdr = static_cast<WsHeader*>(workspace);
        a.limit_ns = wait_limit_ns();
        tv_rows_kernel<<<(unsigned)G, kWSThreads, kRowSmem, s>>>(a);
        if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
        note_launch();
    } else {
        void (*fn)(TVArgs) = dtype == DSPARK_BF16 ? tv_kernel<__nv_bfloat16> : tv_kernel<float>;
        cfg.blockDim = dim3(kTVThreads);
        cfg.dynamicSmemBytes = 0;
        int cs = 4;
        int nclusters = 0;
        for (; cs >= 1; cs >>= 1) {
            if (max_active_clusters((const void*)fn, cs, kTVThreads, 0, &nclusters) != cudaSuccess) return DSPARK_ERR_CUDA;
            if (nclusters > 0) break;
        }
        if (cs < 1 || nclusters < 1) return DSPARK_ERR_CUDA;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        if ((long long)nclusters > rows) nclusters = (int)rows;
        TVArgs a;
        a.rows = rows;
        a.V = V;
        a.gamma = gamma;
        a.segsz = (int)align_up((size_t)((V + cs - 1) / cs), 8);
        a.nclusters = nclusters;
        a.cs = cs;
        a.d = draft_logits;
        a.t = target_logits;
        a.keep = block_keep;
        a.posv = pos_valid;
        a.acc = accept_rate;
        a.mask = eval_mask;
        const size_t esz = dtype == DSPARK_BF16 ? 2 : 4;
        a.vec_ok = ((size_t)V * esz) % 16 == 0 && (uintptr_t)draft_logits % 16 == 0 && (uintptr_t)target_logits % 16 == 0;
        cfg.gridDim = dim3(nclusters * cs);
        if (cudaLaunchKernelEx(&cfg, fn, a) != cudaSuccess) return DSPARK_ERR_CUDA;
        note_launch();
    }
    if (tau) {
        const long long nblk = (long long)S * A;
        tau_kernel<<<(unsigned)((nblk + 255) / 256), 256, 0, s>>>(nblk, gamma, accept_rate, eval_mask, tau);
        if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
        note_launch();
    }
    return DSPARK_OK;
}

extern "C" dspark_status dspark_tv_l1_loss(int S, int A, int gamma, const float* accept_rate, const float* eval_mask,
                                           float decay_gamma, float* l1, double* sums, dspark_stream_t stream) {
    if (S < 1 || A < 1 || gamma < 1 || !accept_rate || !eval_mask || !sums) return DSPARK_ERR_INVALID_ARG;
    if (!(decay_gamma > 0.f)) return DSPARK_ERR_INVALID_ARG;
    if (gamma > kL1MaxGamma) return DSPARK_ERR_UNSUPPORTED;
    const long long n = (long long)S * A * gamma;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    tv_l1_kernel<<<1, kL1Threads, 0, s>>>(n, gamma, accept_rate, eval_mask, (double)decay_gamma, l1, sums);
    if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
    note_launch();
    return DSPARK_OK;
}
