// tv.cu -- dspark_accept_rate_tv: accept-rate targets, eval_mask and tau.
//
// Method (P1 "03 · DSpark 建模：Markov 与 Confidence" section 3.9 "Accept rate 3D" and
// P2 "从 DFlash 到 dLLM Self-Spec（三）" section 3.5): accept = 1 - 0.5 * sum|softmax(d) -
// softmax(t)| clamped to [0,1], computed here as sum_v min(p_v, q_v) (the same quantity with
// no cancellation); min(p, q) = 2^min(d2 - Ld2, t2 - Lt2) needs one exponential per id.
// eval_mask = cumprod of (keep && pos_valid) (P1 section 3.6), tau = 1 + sum_i prod_{k<=i}
// acc_k * mask_k (P1 section 3.10).
//
// Design: a thread-block cluster of kCS blocks owns one row at a time (persistent over rows);
// each block streams its 1/kCS segment of d and t once to get (max, sum) of both softmaxes,
// the blocks exchange those through distributed shared memory, then each block re-reads its
// segment (an L2 hit: the rows in flight stay far below the L2 size) for the sum of minima,
// and block 0 of the cluster sums the partial results and writes acc and eval_mask.
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
// bf16 fast path: the block's segment of each row streams through a ring of shared-memory
// slots filled by the bulk-copy engine (one slot = kCE ids of d and of t), so both passes read
// shared memory and the copies of the next rows proceed while a row is being finished.
// Chunk q of this block (row iteration q / nch, chunk q % nch) lives in slot q % kNS; slot
// reuse is ordered by a block barrier after the slot's second pass.  Every wait is bounded;
// after a timeout the block keeps pace with its cluster (the cluster barriers have no
// timeout) but stops waiting on copies.
// ------------------------------------------------------------------------------------------
constexpr int kCE = 4096;  // ids per array per slot
constexpr int kNS = 13;    // slots: 13 x 16 KB
constexpr size_t kTmaSmem = (size_t)kNS * 2 * kCE * 2 + kNS * sizeof(uint64_t);

struct TVTArgs {
    long long rows;
    int V, gamma, segsz, nch, nclusters, cs;
    const __nv_bfloat16* d;
    const __nv_bfloat16* t;
    const uint8_t* keep;
    const uint8_t* posv;
    float* acc;
    float* mask;
    WsHeader* hdr;
    uint64_t limit_ns;
};

__global__ void __launch_bounds__(kTVThreads, 1) tv_tma_kernel(TVTArgs a) {
    cg::cluster_group cluster = cg::this_cluster();
    const int crank = (int)cluster.block_rank();
    const int cid = blockIdx.x / a.cs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    uint16_t* slots = reinterpret_cast<uint16_t*>(smem_raw);  // [kNS][2][kCE]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + (size_t)kNS * 2 * kCE * 2);
    __shared__ float4 xch[2];
    __shared__ float xsum[2];
    __shared__ float4 red4[kTVWarps];
    __shared__ float red1[kTVWarps];
    __shared__ float2 s_norm;
    __shared__ int s_ok;
    const int seg_lo = crank * a.segsz;
    const int seg_len = max(0, min(a.V - seg_lo, a.segsz));
    const long long niters = (a.rows - cid + a.nclusters - 1) / a.nclusters;
    const long long Q = niters * a.nch;
    auto chunk_len = [&](int k) { return max(0, min(kCE, seg_len - k * kCE)); };
    auto issue = [&](long long q) {  // thread 0 only
        const int slot = (int)(q % kNS);
        const long long it = q / a.nch;
        const int k = (int)(q % a.nch);
        const int len = chunk_len(k);
        const long long row = cid + it * a.nclusters;
        uint16_t* dst = slots + (size_t)slot * 2 * kCE;
        if (len == 0) {  // keep the phase sequence: an arrival without bytes
            mbar_arrive_expect_tx(&bars[slot], 0);
            return;
        }
        mbar_arrive_expect_tx(&bars[slot], (uint32_t)(2 * len * 2));
        const size_t off = (size_t)row * a.V + seg_lo + (size_t)k * kCE;
        bulk_g2s(dst, a.d + off, (uint32_t)(len * 2), &bars[slot]);
        bulk_g2s(dst + kCE, a.t + off, (uint32_t)(len * 2), &bars[slot]);
    };
    if (tid == 0) {
        for (int i = 0; i < kNS; ++i) mbar_init(&bars[i], 1);
        mbar_init_fence();
        s_ok = 1;
    }
    __syncthreads();
    if (tid == 0)
        for (long long q = 0; q < min(Q, (long long)kNS); ++q) issue(q);

    for (long long it = 0; it < niters; ++it) {
        const int par = (int)(it & 1);
        const long long row = cid + it * a.nclusters;
        // ---- pass 1: softmax statistics of the segment of d and t
        float md = -CUDART_INF_F, sd = 0.f, mt = -CUDART_INF_F, st = 0.f;
        for (int k = 0; k < a.nch; ++k) {
            const long long q = it * a.nch + k;
            const int slot = (int)(q % kNS);
            if (tid == 0 && s_ok) s_ok = mbar_wait_bounded(&bars[slot], (uint32_t)((q / kNS) & 1), &a.hdr->status, a.limit_ns);
            __syncthreads();
            if (s_ok) mbar_try_wait(&bars[slot], (uint32_t)((q / kNS) & 1));  // completed: acquire for this thread
            const int len = chunk_len(k);
            if (s_ok && 8 * tid < len) {
                const uint16_t* sd_ = slots + (size_t)slot * 2 * kCE + 8 * tid;
                const uint4 wd = *reinterpret_cast<const uint4*>(sd_);
                const uint4 wt = *reinterpret_cast<const uint4*>(sd_ + kCE);
                float xd[8], xt[8];
                xd[0] = bf16_lo(wd.x); xd[1] = bf16_hi(wd.x); xd[2] = bf16_lo(wd.y); xd[3] = bf16_hi(wd.y);
                xd[4] = bf16_lo(wd.z); xd[5] = bf16_hi(wd.z); xd[6] = bf16_lo(wd.w); xd[7] = bf16_hi(wd.w);
                xt[0] = bf16_lo(wt.x); xt[1] = bf16_hi(wt.x); xt[2] = bf16_lo(wt.y); xt[3] = bf16_hi(wt.y);
                xt[4] = bf16_lo(wt.z); xt[5] = bf16_hi(wt.z); xt[6] = bf16_lo(wt.w); xt[7] = bf16_hi(wt.w);
                lse_merge8(xd, md, sd);
                lse_merge8(xt, mt, st);
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
        cluster.sync();
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
        // ---- pass 2: sum of min(p, q) over the segment, then the slot is refilled
        float acc = 0.f;
        for (int k = 0; k < a.nch; ++k) {
            const long long q = it * a.nch + k;
            const int slot = (int)(q % kNS);
            const int len = chunk_len(k);
            if (s_ok && 8 * tid < len) {
                const uint16_t* sd_ = slots + (size_t)slot * 2 * kCE + 8 * tid;
                const uint4 wd = *reinterpret_cast<const uint4*>(sd_);
                const uint4 wt = *reinterpret_cast<const uint4*>(sd_ + kCE);
                const uint32_t dw[4] = {wd.x, wd.y, wd.z, wd.w}, tw[4] = {wt.x, wt.y, wt.z, wt.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    acc += ex2(fminf(fmaf(bf16_lo(dw[h]), kLog2e, -Ld2), fmaf(bf16_lo(tw[h]), kLog2e, -Lt2)));
                    acc += ex2(fminf(fmaf(bf16_hi(dw[h]), kLog2e, -Ld2), fmaf(bf16_hi(tw[h]), kLog2e, -Lt2)));
                }
            }
            __syncthreads();  // every thread has read the slot: the copy engine may overwrite it
            if (tid == 0 && q + kNS < Q) issue(q + kNS);
        }
        acc = warp_sum(acc);
        if (lane == 0) red1[warp] = acc;
        __syncthreads();
        if (warp == 0) {
            float q = lane < kTVWarps ? red1[lane] : 0.f;
            q = warp_sum(q);
            if (lane == 0) xsum[par] = q;
        }
        cluster.sync();
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
    // after a timeout, copies may still be in flight: wait for them (bounded) before leaving
    if (tid == 0 && !s_ok) {
        for (long long q = max(0LL, Q - kNS); q < Q; ++q) {
            const int slot = (int)(q % kNS);
            mbar_wait_bounded(&bars[slot], (uint32_t)((q / kNS) & 1), &a.hdr->status, a.limit_ns);
        }
    }
    cluster.sync();
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
                     (uintptr_t)target_logits % 16 == 0 && V >= 4 * 8;
    if (tma) {
        // cluster of 4 (8 when it packs the SMs as well): each block owns a quarter (eighth) row
        static bool attr_set = false;
        if (!attr_set) {
            if (cudaFuncSetAttribute((const void*)tv_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kTmaSmem) != cudaSuccess)
                return DSPARK_ERR_CUDA;
            cudaFuncSetAttribute((const void*)tv_tma_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            attr_set = true;
        }
        cfg.dynamicSmemBytes = kTmaSmem;
        int cs = 4, nclusters = 0;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(cs);
        if (cudaOccupancyMaxActiveClusters(&nclusters, (const void*)tv_tma_kernel, &cfg) != cudaSuccess ||
            nclusters < 1)
            return DSPARK_ERR_CUDA;
        if ((long long)nclusters > rows) nclusters = (int)rows;
        TVTArgs a;
        a.rows = rows;
        a.V = V;
        a.gamma = gamma;
        a.segsz = (int)align_up((size_t)((V + cs - 1) / cs), 8);
        a.nch = (a.segsz + kCE - 1) / kCE;
        a.nclusters = nclusters;
        a.cs = cs;
        a.d = static_cast<const __nv_bfloat16*>(draft_logits);
        a.t = static_cast<const __nv_bfloat16*>(target_logits);
        a.keep = block_keep;
        a.posv = pos_valid;
        a.acc = accept_rate;
        a.mask = eval_mask;
        a.hdr = static_cast<WsHeader*>(workspace);
        a.limit_ns = wait_limit_ns();
        cfg.gridDim = dim3(nclusters * cs);
        if (cudaLaunchKernelEx(&cfg, tv_tma_kernel, a) != cudaSuccess) return DSPARK_ERR_CUDA;
    } else {
        void (*fn)(TVArgs) = dtype == DSPARK_BF16 ? tv_kernel<__nv_bfloat16> : tv_kernel<float>;
        cfg.dynamicSmemBytes = 0;
        int cs = 4;
        int nclusters = 0;
        for (; cs >= 1; cs >>= 1) {
            attr[0].val.clusterDim.x = cs;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(cs);
            if (cudaOccupancyMaxActiveClusters(&nclusters, (const void*)fn, &cfg) == cudaSuccess && nclusters > 0) break;
            cudaGetLastError();
        }
        if (cs < 1 || nclusters < 1) return DSPARK_ERR_CUDA;
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
    }
    if (tau) {
        const long long nblk = (long long)S * A;
        tau_kernel<<<(unsigned)((nblk + 255) / 256), 256, 0, s>>>(nblk, gamma, accept_rate, eval_mask, tau);
        if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
    }
    return DSPARK_OK;
}
