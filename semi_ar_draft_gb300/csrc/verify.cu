// verify.cu -- dspark_verify: lossless rejection-sampling verification.
//
// Method (P3 "如何评价 DeepSeek 发布 DSpark？" section "Speculative Decoding": the target scores
// the drafted positions in one parallel pass, accepts left to right by rejection sampling,
// truncates at the first failure and resamples from the target, so the output law equals the
// target's; the verify tokens of all requests form one flattened list, P2 section 3.7.2).
// Contract in dspark.h.
//
// Two stages, no grid-wide waits:
//   1. rows: the target rows' (max, sum 2^(s2 - max)) (T > 0) or (max, argmax) (T = 0).  For bf16
//      rows on 16-byte boundaries a persistent block per SM streams whole rows through a
//      shared-memory ring (verify_rows_ws_kernel); otherwise one block per (vocabulary segment,
//      position, request).  The block completing a request (arrival counter) walks the accept
//      tests left to right, writing n_accepted and, when needed, a job: RESID at the rejecting
//      position or BONUS from target row L+1.
//   2. draws (the chunk-Gumbel contract of dspark.h, with the correction purposes):
//      - bf16 logits and weights of rank 64, at least 64 requests, dense target rows, vanilla head:
//        the tensor-core kernel of sample_tc.cu (z and the target rows in tensor memory, one CTA
//        per tile over row blocks of 128 jobs), then verify_fallback_kernel for residuals that
//        had no mass anywhere (a whole-row draw from p);
//      - otherwise verify_jobs_kernel, one block per (tile, 16 requests): z = base + bias for
//        RESID rows (the sampler's producer, or the head vectors), per-id weights max(0, p - q)
//        (RESID) or the target softmax (BONUS), the tile's best chunk key; the last block of a row
//        block reduces the tiles to the correction token, and draws from p where a residual had no
//        mass.
#include <algorithm>

#include "host_util.h"
#include "markov_tile.cuh"

namespace dspark {
namespace {

enum { JOB_NONE = 0, JOB_RESID = 1, JOB_BONUS = 2 };

struct VerifyArgs {
    int B, gamma, V, r, nt, nseg, segsz, gamma_t, nrb;
    int greedy;
    float scale2;  // log2(e) / T
    float invT;
    uint64_t seed;
    const void* base;
    const void* W1;
    const void* W2;
    const int32_t* anchor;
    const int32_t* tokens;
    uint64_t limit_ns;  // bound of every wait of the persistent rows kernel
    const float* dlse;
    const float* zat;
    const void* target;
    const int32_t* vlen;
    const int32_t* toff;
    int32_t* nacc;
    int32_t* corr;
    WsHeader* hdr;
    uint32_t* cnt_req;  // [B]
    uint32_t* cnt_rb;   // [nrb]
    float2* rowpart;    // [B][gamma][nseg]
    int4* job;          // [B] {type, position (1-based), prev token, lse2 bits of the target row}
    float4* jobpart;    // [B][nt]
    int vec_b, vec_t;
    float softcap;  // draft softcap of the base logits (0: none)
    const float* head_vec;  // [B][gamma][r] head vectors of a Gated / RNN head, or null (W1[prev])
};

__device__ __forceinline__ int req_len(const VerifyArgs& a, int j) { return a.vlen ? a.vlen[j] : a.gamma; }
__device__ __forceinline__ int req_rows(const VerifyArgs& a, int j) {
    return a.toff ? a.toff[j + 1] - a.toff[j] : a.gamma_t;
}
__device__ __forceinline__ long long trow_off(const VerifyArgs& a, int j, int i) {
    return a.toff ? ((long long)a.toff[j] + i - 1) * a.V : ((long long)j * a.gamma_t + i - 1) * a.V;
}

// Block-wide combine of per-thread (max, sum 2^(x - max)) pairs; result valid in thread 0.
__device__ float2 block_lse_pair(float m, float s, float2* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    float wm = warp_max(m);
    float ws = warp_sum(m == -CUDART_INF_F ? 0.f : s * ex2(m - wm));
    if (lane == 0) red[warp] = make_float2(wm, ws);
    __syncthreads();
    float2 out = make_float2(-CUDART_INF_F, 0.f);
    if (warp == 0) {
        const float2 v = lane < nw ? red[lane] : make_float2(-CUDART_INF_F, 0.f);
        const float M = warp_max(v.x);
        const float S = warp_sum(v.x == -CUDART_INF_F ? 0.f : v.y * ex2(v.x - M));
        out = make_float2(M, S);
    }
    __syncthreads();
    return out;
}

__device__ float2 block_argmax_pair(float m, int idx, float2* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    warp_argmax(m, idx);
    if (lane == 0) red[warp] = make_float2(m, __int_as_float(idx));
    __syncthreads();
    float2 out = make_float2(-CUDART_INF_F, __int_as_float(0x7fffffff));
    if (warp == 0) {
        float2 v = lane < nw ? red[lane] : make_float2(-CUDART_INF_F, __int_as_float(0x7fffffff));
        float vm = v.x;
        int vi = __float_as_int(v.y);
        warp_argmax(vm, vi);
        out = make_float2(vm, __int_as_float(vi));
    }
    __syncthreads();
    return out;
}

// ------------------------------------------------------------------------------- launch 1
// The accept walk of request j by one warp (lane = segment of the rows' partial results, nseg of
// them): the accept test at every position left to right, n_accepted, the greedy correction,
// or the job (residual at the rejecting position, or the bonus row) for the second launch.
template <typename TL>
__device__ void accept_walk(const VerifyArgs& a, int j, int L, int lane) {
    int n = L, corr = -1, jtype = JOB_NONE, jpos = 0, jprev = 0;
    float jlse2 = 0.f;
    const TL* tgt = reinterpret_cast<const TL*>(a.target);
    for (int ii = 1; ii <= L; ++ii) {
        const float2 p = lane < a.nseg ? __ldcg(&a.rowpart[((size_t)j * a.gamma + (ii - 1)) * a.nseg + lane])
                                       : (a.greedy ? make_float2(-CUDART_INF_F, __int_as_float(0x7fffffff))
                                                   : make_float2(-CUDART_INF_F, 0.f));
        const int x = a.tokens[(size_t)j * a.gamma + ii - 1];
        const bool xok = x >= 0 && x < a.V;
        int accept;
        int am = 0;
        float lse2 = 0.f;
        if (a.greedy) {
            float m = p.x;
            int idx = __float_as_int(p.y);
            warp_argmax(m, idx);
            am = idx;
            accept = xok && (am == x);
        } else {
            const float M = warp_max(p.x);
            const float S = warp_sum(p.x == -CUDART_INF_F ? 0.f : p.y * ex2(p.x - M));
            lse2 = M + lg2(S);
            accept = 0;
            if (lane == 0 && xok) {
                const float tx = load_logit<TL>(tgt, (size_t)(trow_off(a, j, ii) + x));
                const float lnp = (tx * a.scale2 - lse2) * kLn2;
                const float lnq = a.zat[(size_t)j * a.gamma + ii - 1] * a.invT - a.dlse[(size_t)j * a.gamma + ii - 1];
                const float lnu = logf(uniform(a.seed, (uint32_t)j, (uint32_t)ii, DSPARK_P_ACCEPT, 0u));
                accept = lnu < lnp - lnq;
            }
            accept = __shfl_sync(0xffffffffu, accept, 0);
        }
        if (!xok && lane == 0) record_status(&a.hdr->status, DSPARK_ERR_TOKEN_RANGE);
        if (!accept) {
            n = ii - 1;
            if (!xok) break;
            if (a.greedy) {
                corr = am;
            } else {
                jtype = JOB_RESID;
                jpos = ii;
                jlse2 = lse2;
                jprev = (ii == 1) ? a.anchor[j] : a.tokens[(size_t)j * a.gamma + ii - 2];
                if (jprev < 0 || jprev >= a.V) {
                    if (lane == 0) record_status(&a.hdr->status, DSPARK_ERR_TOKEN_RANGE);
                    jtype = JOB_NONE;
                }
            }
            break;
        }
    }
    if (n == L && req_rows(a, j) > L) {
        jtype = JOB_BONUS;
        jpos = L + 1;
    }
    if (lane == 0) {
        a.nacc[j] = n;
        a.corr[j] = corr;
        a.job[j] = make_int4(jtype, jpos, jprev, __float_as_int(jlse2));
    }
}

template <typename TL>
__global__ void __launch_bounds__(kThreads) verify_rows_kernel(VerifyArgs a) {
    __shared__ float2 red[kWarps];
    __shared__ int s_last;
    const int seg = blockIdx.x, i = blockIdx.y + 1, j = blockIdx.z;
    const int tid = threadIdx.x;
    const int L = req_len(a, j);
    const bool ok = L >= 1 && L <= a.gamma && req_rows(a, j) >= L;
    if (!ok) {
        if (i == 1 && seg == 0 && tid == 0) {
            record_status(&a.hdr->status, DSPARK_ERR_TOKEN_RANGE);
            a.nacc[j] = 0;
            a.corr[j] = -1;
            a.job[j] = make_int4(JOB_NONE, 0, 0, 0);
        }
        return;
    }
    if (i > L) return;
    const TL* row = reinterpret_cast<const TL*>(a.target) + trow_off(a, j, i);
    const int v_lo = seg * a.segsz, v_hi = min(a.V, v_lo + a.segsz);
    float2 res;
    constexpr int U = 4;  // 8-id groups per thread in flight
    if (a.greedy) {
        float m = -CUDART_INF_F;
        int idx = 0x7fffffff;
        for (int v0 = v_lo + 8 * tid; v0 < v_hi; v0 += 8 * kThreads * U) {
            Raw8<TL> raw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int vv = v0 + 8 * kThreads * u;
                if (vv < v_hi) load_raw8<TL>(row, vv, a.V, a.vec_t != 0, raw[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int vv = v0 + 8 * kThreads * u;
                if (vv >= v_hi) break;
                float x[8];
                unpack8<TL>(raw[u], x);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (x[e] > m) {
                        m = x[e];
                        idx = vv + e;
                    }
            }
        }
        res = block_argmax_pair(m, idx, red);
    } else {
        float m = -CUDART_INF_F, s = 0.f;
        for (int v0 = v_lo + 8 * tid; v0 < v_hi; v0 += 8 * kThreads * U) {
            Raw8<TL> raw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int vv = v0 + 8 * kThreads * u;
                if (vv < v_hi) load_raw8<TL>(row, vv, a.V, a.vec_t != 0, raw[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int vv = v0 + 8 * kThreads * u;
                if (vv >= v_hi) break;
                float x[8];
                unpack8<TL>(raw[u], x);
                float gm = x[0];
#pragma unroll
                for (int e = 1; e < 8; ++e) gm = fmaxf(gm, x[e]);
                const float mn = fmaxf(m, gm * a.scale2);
                if (mn != -CUDART_INF_F) {
                    s = (m == -CUDART_INF_F) ? 0.f : s * ex2(m - mn);
#pragma unroll
                    for (int e = 0; e < 8; ++e) s += ex2(fmaf(x[e], a.scale2, -mn));
                    m = mn;
                }
            }
        }
        res = block_lse_pair(m, s, red);
    }
    if (tid == 0) {
        a.rowpart[((size_t)j * a.gamma + (i - 1)) * a.nseg + seg] = res;
        __threadfence();
        const uint32_t old = atomicAdd(&a.cnt_req[j], 1u);
        s_last = (old == (uint32_t)(a.nseg * L - 1));
    }
    __syncthreads();
    if (!s_last || tid >= 32) return;
    __threadfence();

    accept_walk<TL>(a, j, L, tid);
}

// The accept walk when every row has one segment: lane q takes position q + 1 (32 at a time),
// so the rows' partials, the tokens, the target logits at the tokens and the draft terms are
// all read at once; the first rejection is the lowest lane whose test fails.  Same decisions
// and outputs as accept_walk.
template <typename TL>
__device__ void accept_walk_lanes(const VerifyArgs& a, int j, int L, int lane) {
    const TL* tgt = reinterpret_cast<const TL*>(a.target);
    int n = L, corr = -1, jtype = JOB_NONE, jpos = 0, jprev = 0;
    float jlse2 = 0.f;
    for (int base = 0; base < L; base += 32) {
        const int ii = base + lane + 1;  // this lane's position
        const bool act = ii <= L;
        int accept = 1, xok = 1, am = 0;
        float lse2 = 0.f;
        if (act) {
            const float2 p = __ldcg(&a.rowpart[(size_t)j * a.gamma + (ii - 1)]);
            const int x = a.tokens[(size_t)j * a.gamma + ii - 1];
            xok = x >= 0 && x < a.V;
            if (a.greedy) {
                am = __float_as_int(p.y);
                accept = xok && (am == x);
            } else {
                lse2 = p.x + lg2(p.y);
                accept = 0;
                if (xok) {
                    const float tx = load_logit<TL>(tgt, (size_t)(trow_off(a, j, ii) + x));
                    const float lnp = (tx * a.scale2 - lse2) * kLn2;
                    const float lnq = a.zat[(size_t)j * a.gamma + ii - 1] * a.invT - a.dlse[(size_t)j * a.gamma + ii - 1];
                    const float lnu = logf(uniform(a.seed, (uint32_t)j, (uint32_t)ii, DSPARK_P_ACCEPT, 0u));
                    accept = lnu < lnp - lnq;
                }
            }
        }
        const unsigned rej = __ballot_sync(0xffffffffu, act && !accept);
        if (!rej) continue;
        const int f = __ffs(rej) - 1;  // the first rejecting position of this group: base + f + 1
        const int fx = __shfl_sync(0xffffffffu, xok, f);
        const int fam = __shfl_sync(0xffffffffu, am, f);
        const float flse2 = __shfl_sync(0xffffffffu, lse2, f);
        const int fi = base + f + 1;
        if (lane == 0 && !fx) record_status(&a.hdr->status, DSPARK_ERR_TOKEN_RANGE);
        n = fi - 1;
        if (fx) {
            if (a.greedy) {
                corr = fam;
            } else {
                jtype = JOB_RESID;
                jpos = fi;
                jlse2 = flse2;
                jprev = (fi == 1) ? a.anchor[j] : a.tokens[(size_t)j * a.gamma + fi - 2];
                if (jprev < 0 || jprev >= a.V) {
                    if (lane == 0) record_status(&a.hdr->status, DSPARK_ERR_TOKEN_RANGE);
                    jtype = JOB_NONE;
                }
            }
        }
        break;
    }
    if (n == L && req_rows(a, j) > L) {
        jtype = JOB_BONUS;
        jpos = L + 1;
    }
    if (lane == 0) {
        a.nacc[j] = n;
        a.corr[j] = corr;
        a.job[j] = make_int4(jtype, jpos, jprev, __float_as_int(jlse2));
    }
}

// ------------------------------------------------------------------------------- launch 1, bf16
// Persistent variant for bf16 target rows on 16-byte boundaries: one block per SM walks the
// verified rows, numbered v = 0 .. sum_j L_j - 1 in request order (v = blockIdx.x, blockIdx.x + G,
// ...), so every block gets the same number of rows whatever the lengths; each block finds the
// request of row v by binary search in the prefix sums of L_j it forms first in shared memory.
// A producer warp streams each row through a ring of kVNS shared-memory slots with the bulk-copy
// engine; 16 consumer warps reduce it to (max, sum 2^(t * scale2 - max)) (T > 0) or (max, lowest
// argmax) (T = 0).  The block that completes a request's last row runs the accept walk (rows then
// have one segment).
constexpr int kVCE = 16384;        // target ids per slot (32 per consumer thread)
constexpr int kVNS = 6;            // ring slots (6 x 32 KB)
constexpr int kVGrp = kVCE / 4;    // ids between a consumer thread's 16-byte groups
constexpr int kVThreads = kThreads + 32;
constexpr int kVMaxB = 4096;  // requests (the prefix of their lengths is kept in shared memory)

struct VRSmem {
    uint16_t slots[kVNS][kVCE];
    uint64_t full[kVNS];
    uint64_t empty[kVNS];
    float2 red[2][kWarps];
    int s_last;
    int abort;
    int issued;  // chunks the producer has issued
    int nver;    // verified rows of the call
    int voff[kVMaxB + 1];  // exclusive prefix of the valid L_j (0 for a request with an invalid length)
};

__device__ __forceinline__ int valid_len(const VerifyArgs& a, int j) {
    const int L = req_len(a, j);
    return (L >= 1 && L <= a.gamma && req_rows(a, j) >= L) ? L : 0;
}

// Verified row v -> request j, position i (1-based) and that request's length L.
__device__ __forceinline__ void verified_row(const VerifyArgs& a, const int* voff, int v, int& j, int& i, int& L) {
    int lo = 0, hi = a.B - 1;  // the last j with voff[j] <= v
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (voff[mid] <= v) lo = mid;
        else hi = mid - 1;
    }
    j = lo;
    i = v - voff[j] + 1;
    L = voff[j + 1] - voff[j];
}

// Exclusive prefix of the valid lengths into S.voff (all threads of the block take part).
__device__ void length_prefix(const VerifyArgs& a, VRSmem& S) {
    const int tid = threadIdx.x, nth = blockDim.x;
    const int per = (a.B + nth - 1) / nth;  // consecutive requests per thread
    const int j0 = tid * per;
    int sum = 0;
    for (int j = j0; j < min(a.B, j0 + per); ++j) sum += valid_len(a, j);
    // block-wide exclusive scan of the per-thread sums (warp scans, then the warp totals)
    const int lane = tid & 31, warp = tid >> 5, nw = nth >> 5;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    __shared__ int wsum[32];
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        wsum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    int run = incl - sum + (warp > 0 ? wsum[warp - 1] : 0);
    for (int j = j0; j < min(a.B, j0 + per); ++j) {
        S.voff[j] = run;
        run += valid_len(a, j);
    }
    if (tid == nth - 1) {
        S.voff[a.B] = run;
        S.nver = run;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kVThreads, 1) verify_rows_ws_kernel(VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    VRSmem& S = *reinterpret_cast<VRSmem*>(smem_raw);
    volatile int* abort = &S.abort;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nch = (a.V + kVCE - 1) / kVCE;
    length_prefix(a, S);
    const int nver = S.nver;
    if (tid == 0) {
        for (int k = 0; k < kVNS; ++k) {
            mbar_init(&S.full[k], 1);
            mbar_init(&S.empty[k], kWarps);
        }
        S.abort = 0;
        S.issued = 0;
        mbar_init_fence();
        for (int j = blockIdx.x; j < a.B; j += gridDim.x) {  // requests without a valid length: no walk
            const int L = req_len(a, j);
            if (!(L >= 1 && L <= a.gamma && req_rows(a, j) >= L)) {
                record_status(&a.hdr->status, DSPARK_ERR_TOKEN_RANGE);
                a.nacc[j] = 0;
                a.corr[j] = -1;
                a.job[j] = make_int4(JOB_NONE, 0, 0, 0);
            }
        }
    }
    __syncthreads();
    const __nv_bfloat16* tgt = reinterpret_cast<const __nv_bfloat16*>(a.target);
    int q = 0;
    if (warp == kWarps) {
        // ---------------- producer warp
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            for (int v = blockIdx.x; v < nver; v += gridDim.x) {
                int j, i, L;
                verified_row(a, S.voff, v, j, i, L);
                const __nv_bfloat16* row = tgt + trow_off(a, j, i);
                for (int k = 0; k < nch; ++k, ++q) {
                    const int slot = q % kVNS;
                    if (q >= kVNS && !mbar_wait_or_abort(&S.empty[slot], (uint32_t)((q / kVNS - 1) & 1), abort,
                                                        &a.hdr->status, a.limit_ns, false))
                        break;
                    const int len = min(kVCE, a.V - k * kVCE);
                    mbar_arrive_expect_tx(&S.full[slot], (uint32_t)(2 * len));
                    bulk_g2s_hint(&S.slots[slot][0], row + (size_t)k * kVCE, (uint32_t)(2 * len), &S.full[slot], pol);
                    S.issued = q + 1;
                }
                if (*abort) break;
            }
        }
        __syncwarp();
    } else {
        // ---------------- 16 consumer warps; thread t takes ids g kVGrp + 8t .. g kVGrp + 8t + 7, g < 4
        // After an abort the waits return at once and the slots hold stale data: the arithmetic runs
        // on it (shared-memory reads cannot fault) and nothing is stored.
        static_assert(kVCE == 32 * kThreads, "four 16-byte groups per consumer thread per slot");
        const int my0 = 8 * tid;
        const int tail = a.V - (nch - 1) * kVCE;  // ids in the last chunk of a row
        const uint64_t c2 = pk2(a.scale2, a.scale2);
        const float inv2 = 1.f / a.scale2;
        int par = 0, slot = 0;
        uint32_t phase = 0;
        for (int v = blockIdx.x; v < nver; v += gridDim.x) {
            int j, i, L;
            verified_row(a, S.voff, v, j, i, L);
            float m = -CUDART_INF_F, sacc = 0.f;
            int idx = 0x7fffffff;
            auto chunk = [&](int k, bool last) {
                mbar_wait_hint_or_abort(&S.full[slot], phase, abort, &a.hdr->status, a.limit_ns);
                uint32_t w[16];
                load32w<kVGrp>(&S.slots[slot][0], my0, w);
                __syncwarp();
                if (lane == 0) mbar_arrive_local(&S.empty[slot]);
                if (++slot == kVNS) {
                    slot = 0;
                    phase ^= 1u;
                }
                if (last) mask_tail32<kVGrp>(w, my0, tail);
                if (a.greedy) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {  // ids ascend with (e, half): the first maximum is kept
                        const int id = k * kVCE + (e >> 2) * kVGrp + my0 + 2 * (e & 3);
                        const float lo = bf16_lo(w[e]), hi = bf16_hi(w[e]);
                        if (lo > m) {
                            m = lo;
                            idx = id;
                        }
                        if (hi > m) {
                            m = hi;
                            idx = id + 1;
                        }
                    }
                } else {
                    lse_step32w(w, a.scale2, inv2, c2, m, sacc);
                }
            };
            for (int k = 0; k < nch - 1; ++k) chunk(k, false);
            chunk(nch - 1, true);
            q += nch;
            // block combine -> the row's partial, then the request's counter
            if (a.greedy) {
                warp_argmax(m, idx);
                if (lane == 0) S.red[par][warp] = make_float2(m, __int_as_float(idx));
            } else {
                const float M = warp_max(m);
                const float Sm = warp_sum(m == -CUDART_INF_F ? 0.f : sacc * ex2(m - M));
                if (lane == 0) S.red[par][warp] = make_float2(M, Sm);
            }
            named_barrier(1, kThreads);
            if (warp == 0) {
                float2 v = lane < kWarps ? S.red[par][lane]
                                         : (a.greedy ? make_float2(-CUDART_INF_F, __int_as_float(0x7fffffff))
                                                     : make_float2(-CUDART_INF_F, 0.f));
                float2 res;
                if (a.greedy) {
                    int id = __float_as_int(v.y);
                    warp_argmax(v.x, id);
                    res = make_float2(v.x, __int_as_float(id));
                } else {
                    const float M = warp_max(v.x);
                    const float Sm = warp_sum(v.x == -CUDART_INF_F ? 0.f : v.y * ex2(v.x - M));
                    res = make_float2(M, Sm);
                }
                if (lane == 0) {
                    if (!*abort) a.rowpart[(size_t)j * a.gamma + (i - 1)] = res;  // one segment per row
                    __threadfence();
                    const uint32_t old = atomicAdd(&a.cnt_req[j], 1u);
                    S.s_last = (old == (uint32_t)(L - 1)) && !*abort;
                }
                __syncwarp();
                if (S.s_last) {  // warp-uniform: every row of request j is in
                    __threadfence();
                    accept_walk_lanes<__nv_bfloat16>(a, j, L, lane);
                }
            }
            par ^= 1;
        }
    }
    __syncthreads();
    // copies still in flight after an abort: wait for them (bounded) before the block leaves
    if (tid == 0 && *abort) {
        const int nq = S.issued;
        const uint64_t t0 = global_ns();
        for (int qq = max(0, nq - kVNS); qq < nq; ++qq) {
            const int sl = qq % kVNS;
            while (!mbar_try_wait(&S.full[sl], (uint32_t)((qq / kVNS) & 1)) && global_ns() - t0 < a.limit_ns) {
            }
        }
    }
    (void)q;
}

// ------------------------------------------------------------------------------- launch 2
// Whole-block draw from softmax(target row / T) with the RESID purposes and the chunk-Gumbel
// contract (a warp per chunk: lane = id; the chunk's key LSE_c - ln E_c, its in-chunk inverse-CDF
// candidate; the best key over the block, the lowest chunk on ties): the fallback when a residual
// max(0, p - q) has no mass at all.  sh: 64 floats of shared scratch.
template <typename TL>
__device__ int block_sample_row(const VerifyArgs& a, const TL* row, int j, int pos, float* sh) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float u = uniform(a.seed, (uint32_t)j, (uint32_t)pos, DSPARK_P_RESID_INCHUNK, 0u);
    const int nc = (a.V + kCS - 1) / kCS;
    float bkey = -CUDART_INF_F;
    int bcand = 0x7fffffff;
    for (int c = warp; c < nc; c += kWarps) {  // ascending chunks per warp: ties keep the lower one
        const int v = kCS * c + lane;
        const float x = v < a.V ? load_logit<TL>(row, (size_t)v) * a.scale2 : -CUDART_INF_F;
        const float m = warp_max(x);
        if (m == -CUDART_INF_F) continue;  // (warp-uniform) a chunk without mass never wins
        const float e = v < a.V ? ex2(x - m) : 0.f;
        const float Q = warp_incl_scan(e);
        const float S = __shfl_sync(0xffffffffu, Q, 31);
        const float key = (m + lg2(S)) * kLn2 - log_neg_log_u(uniform(a.seed, (uint32_t)j, (uint32_t)pos,
                                                                         DSPARK_P_RESID_CHUNK, (uint32_t)c));
        const unsigned hit = __ballot_sync(0xffffffffu, Q > u * S);
        const unsigned nz = __ballot_sync(0xffffffffu, e > 0.f);
        const int k = hit ? __ffs(hit) - 1 : (nz ? 31 - __clz(nz) : 0);
        if (key > bkey) {
            bkey = key;
            bcand = kCS * c + k;
        }
    }
    if (lane == 0) {
        sh[warp] = bkey;
        sh[16 + warp] = __int_as_float(bcand);
    }
    __syncthreads();
    if (warp == 0) {
        float k = lane < kWarps ? sh[lane] : -CUDART_INF_F;
        int x = lane < kWarps ? __float_as_int(sh[16 + lane]) : 0x7fffffff;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float ok = __shfl_xor_sync(0xffffffffu, k, o);
            const int ox = __shfl_xor_sync(0xffffffffu, x, o);
            if (ok > k || (ok == k && ox < x)) {
                k = ok;
                x = ox;
            }
        }
        if (lane == 0) sh[32] = __int_as_float(x == 0x7fffffff ? -1 : x);
    }
    __syncthreads();
    const int x = __float_as_int(sh[32]);
    __syncthreads();
    return x;
}

// After the tensor-core jobs kernel: the whole-row draw from p for the residuals it found without
// mass (one block per request; the others return at once).
template <typename TL>
__global__ void __launch_bounds__(kThreads) verify_fallback_kernel(VerifyArgs a, const int32_t* fb) {
    const int j = blockIdx.x;
    if (!fb[j]) return;  // (uniform per block)
    __shared__ float sh[64];
    const int4 q = a.job[j];
    const int x = block_sample_row<TL>(a, reinterpret_cast<const TL*>(a.target) + trow_off(a, j, q.y), j, q.y, sh);
    if (threadIdx.x == 0) a.corr[j] = x;
}

template <typename TL, int KS, typename TW>
__global__ void __launch_bounds__(kThreads, 1) verify_jobs_kernel(VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* xbuf = reinterpret_cast<float*>(smem_raw);                 // [kRows][kXRow]: log2-weights
    float2* cstat = reinterpret_cast<float2*>(xbuf + kRows * kXRow);  // [kRows][kChunks]
    RowBlock* rb = reinterpret_cast<RowBlock*>(cstat + kRows * kChunks);
    int4* jb = reinterpret_cast<int4*>(reinterpret_cast<unsigned char*>(rb) + align_up(sizeof(RowBlock), 16));
    float* scratch = reinterpret_cast<float*>(jb + kRows);  // fallback scratch [64]
    float* w1s = scratch + 64;                              // CUDA-core path: [kRows][r]
    __shared__ int s_any, s_last, s_fallback[kRows];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, row0 = blockIdx.y * kRows;
    if (tid == 0) s_any = 0;
    __syncthreads();
    if (tid < kRows) {
        const int j = row0 + tid;
        int4 q = make_int4(JOB_NONE, 0, 0, 0);
        if (j < a.B) q = a.job[j];
        jb[tid] = q;
        const bool resid = q.x == JOB_RESID, bonus = q.x == JOB_BONUS;
        rb->mode[tid] = resid ? ROW_RESID : (bonus ? ROW_BONUS : ROW_OFF);
        rb->prev[tid] = resid ? q.z : 0;
        rb->brow[tid] = resid ? ((long long)j * a.gamma + q.y - 1) * (long long)a.V : -1;
        rb->trow[tid] = (resid || bonus) ? trow_off(a, j, q.y) : -1;
        float u = 0.f, dl2 = 0.f;
        if (resid || bonus) {  // the in-chunk uniform of the correction's chunk-Gumbel draw
            u = uniform(a.seed, (uint32_t)j, (uint32_t)q.y, resid ? DSPARK_P_RESID_INCHUNK : DSPARK_P_BONUS_INCHUNK,
                        0u);
            if (resid) dl2 = a.dlse[(size_t)j * a.gamma + q.y - 1] * kLog2e;
            atomicOr(&s_any, 1);
        }
        rb->u1[tid] = 0.f;
        rb->u2[tid] = u;
        rb->lnE[tid] = 0.f;
        rb->lse2[tid] = __int_as_float(q.w);
        rb->dl2[tid] = dl2;
    }
    __syncthreads();
    if (!s_any) return;  // uniform over the row block's tiles: no arrival is expected from them either
    ProdArgs pa;
    pa.base = a.base;
    pa.target = a.target;
    pa.W1 = a.W1;
    pa.W2 = a.W2;
    pa.w2s = nullptr;
    pa.w1s = w1s;
    pa.V = a.V;
    pa.r = a.r;
    pa.greedy = a.greedy;
    pa.scale2 = a.scale2;
    pa.vec_b = a.vec_b;
    pa.vec_t = a.vec_t;
    pa.softcap = a.softcap;
    pa.inv_softcap = a.softcap > 0.f ? 1.f / a.softcap : 0.f;
    if constexpr (KS == 0) {
        const TW* W1 = reinterpret_cast<const TW*>(a.W1);
        for (int idx = tid; idx < kRows * a.r; idx += kThreads) {
            const int q = idx / a.r, k = idx % a.r;
            w1s[idx] = rb->brow[q] < 0 ? 0.f
                       : a.head_vec ? a.head_vec[((size_t)(row0 + q) * a.gamma + jb[q].y - 1) * a.r + k]
                                    : load_logit<TW>(W1, (size_t)rb->prev[q] * a.r + k);
        }
        __syncthreads();
    }
    produce_chunks<TL, KS, TW, true>(pa, tile, *rb, xbuf, cstat);
    __syncthreads();
    for (int q = warp; q < kRows; q += kWarps) {
        if (rb->mode[q] == ROW_OFF) continue;
        const int j = row0 + q;
        const float4 rec = finalize_tile_cg(xbuf + q * kXRow, cstat[q * kChunks + lane], tile, a.V, a.greedy, 1.f,
                                            rb->u2[q], a.seed, (uint32_t)j, (uint32_t)jb[q].y,
                                            rb->mode[q] == ROW_RESID ? DSPARK_P_RESID_CHUNK : DSPARK_P_BONUS_CHUNK);
        if (lane == 0) a.jobpart[(size_t)j * a.nt + tile] = rec;
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t old = atomicAdd(&a.cnt_rb[blockIdx.y], 1u);
        s_last = (old == (uint32_t)(a.nt - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int q = warp; q < kRows; q += kWarps) {
        const int4 job = jb[q];
        if (job.x == JOB_NONE) continue;
        const int j = row0 + q;
        const TileAcc w = reduce_tiles_group(a.jobpart + (size_t)j * a.nt, a.nt, lane, 32, false);
        if (lane == 0) {
            s_fallback[q] = (w.cand < 0);
            if (w.cand >= 0) a.corr[j] = w.cand;
        }
    }
    __syncthreads();
    for (int q = 0; q < kRows; ++q) {
        const int4 job = jb[q];
        if (job.x != JOB_RESID || !s_fallback[q]) continue;
        const int j = row0 + q;
        const int x = block_sample_row<TL>(a, reinterpret_cast<const TL*>(a.target) + trow_off(a, j, job.y), j,
                                           job.y, scratch);
        if (tid == 0) a.corr[j] = x;
    }
}

using RowsFn = void (*)(VerifyArgs);

template <typename TL>
RowsFn pick_jobs_mma(int r) {
    switch (r) {
        case 16: return verify_jobs_kernel<TL, 1, uint16_t>;
        case 32: return verify_jobs_kernel<TL, 2, uint16_t>;
        case 64: return verify_jobs_kernel<TL, 4, uint16_t>;
        case 128: return verify_jobs_kernel<TL, 8, uint16_t>;
        case 256: return verify_jobs_kernel<TL, 16, uint16_t>;
        default: return nullptr;
    }
}

RowsFn pick_jobs(const dspark_sample_params* p, bool mma) {
    const bool lb = p->logits_dtype == DSPARK_BF16;
    if (mma) return lb ? pick_jobs_mma<__nv_bfloat16>(p->r) : pick_jobs_mma<float>(p->r);
    const bool wb = p->w_dtype == DSPARK_BF16;
    if (lb) return wb ? verify_jobs_kernel<__nv_bfloat16, 0, __nv_bfloat16> : verify_jobs_kernel<__nv_bfloat16, 0, float>;
    return wb ? verify_jobs_kernel<float, 0, __nv_bfloat16> : verify_jobs_kernel<float, 0, float>;
}

struct Layout {
    int nt, nseg, segsz, nrb;
    size_t off_cnt_req, off_cnt_rb, off_tc_words, off_tc_count, off_fb, zero_bytes, off_rowpart, off_job, off_jobpart,
        total;
};

Layout layout(const dspark_sample_params* p) {
    Layout L;
    L.nt = (p->V + kTS - 1) / kTS;
    int nseg = (p->V + 16383) / 16384;
    nseg = std::max(1, std::min(32, nseg));
    L.segsz = (int)align_up((size_t)((p->V + nseg - 1) / nseg), 8);
    L.nseg = (p->V + L.segsz - 1) / L.segsz;
    L.nrb = (p->B + kRows - 1) / kRows;
    L.off_cnt_req = kHeaderBytes;
    L.off_cnt_rb = L.off_cnt_req + sizeof(uint32_t) * (size_t)p->B;
    // the tensor-core jobs kernel: a packed word per job and an arrival counter per 128 jobs, one
    // 128-byte line each, and the fallback flags
    L.off_tc_words = align_up(L.off_cnt_rb + sizeof(uint32_t) * (size_t)L.nrb, 256);
    L.off_tc_count = L.off_tc_words + kVtcLine * (size_t)p->B;
    L.off_fb = L.off_tc_count + kVtcLine * (size_t)((p->B + 127) / 128);
    L.zero_bytes = align_up(L.off_fb + sizeof(int32_t) * (size_t)p->B, 256);
    L.off_rowpart = L.zero_bytes;
    L.off_job = L.off_rowpart + align_up(sizeof(float2) * (size_t)p->B * p->gamma * L.nseg, 256);
    L.off_jobpart = L.off_job + align_up(sizeof(int4) * (size_t)p->B, 256);
    L.total = L.off_jobpart + align_up(sizeof(float4) * (size_t)p->B * L.nt, 256);
    return L;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_verify_workspace_size(const dspark_sample_params* p, int gamma_t) {
    (void)gamma_t;
    if (validate_sample_params(p) != DSPARK_OK) return 0;
    return layout(p).total;
}

namespace {

// Shared by dspark_verify and dspark_verify_head (head_vec non-null: the CUDA-core bias path
// reads the head vectors instead of W1 rows).
dspark_status verify_impl(const dspark_sample_params* p, const void* base_logits, const void* W1,
                          const float* head_vec, const void* W2, const int32_t* anchor, const int32_t* tokens,
                          const float* draft_lse, const float* draft_logit_at_tok, const void* target_logits,
                          int gamma_t, const int32_t* verify_len, const int32_t* target_row_offsets,
                          int32_t* n_accepted, int32_t* correction_token, void* workspace, size_t ws_bytes,
                          dspark_stream_t stream) {
    dspark_status st = validate_sample_params(p);
    if (st != DSPARK_OK) return st;
    if (!base_logits || !anchor || !tokens || !draft_lse || !draft_logit_at_tok || !target_logits || !n_accepted ||
        !correction_token)
        return DSPARK_ERR_INVALID_ARG;
    if (p->r > 0 && ((!W1 && !head_vec) || !W2)) return DSPARK_ERR_INVALID_ARG;
    if (!target_row_offsets && gamma_t < 1) return DSPARK_ERR_INVALID_ARG;
    const Layout L = layout(p);
    if (!workspace || ((uintptr_t)workspace & 255u) || ws_bytes < L.total) return DSPARK_ERR_WORKSPACE;
    const bool mma = !head_vec && markov_use_mma(p);

    VerifyArgs a;
    a.B = p->B;
    a.gamma = p->gamma;
    a.V = p->V;
    a.r = p->r;
    a.nt = L.nt;
    a.nseg = L.nseg;
    a.segsz = L.segsz;
    a.gamma_t = target_row_offsets ? 0 : gamma_t;
    a.nrb = L.nrb;
    a.greedy = p->temperature == 0.f;
    a.scale2 = a.greedy ? 1.f : kLog2e / p->temperature;
    a.invT = a.greedy ? 0.f : 1.f / p->temperature;
    a.seed = p->seed;
    a.base = base_logits;
    a.W1 = W1;
    a.W2 = W2;
    a.anchor = anchor;
    a.tokens = tokens;
    a.limit_ns = wait_limit_ns();
    a.dlse = draft_lse;
    a.zat = draft_logit_at_tok;
    a.target = target_logits;
    a.vlen = verify_len;
    a.toff = target_row_offsets;
    a.nacc = n_accepted;
    a.corr = correction_token;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    a.hdr = reinterpret_cast<WsHeader*>(ws);
    a.cnt_req = reinterpret_cast<uint32_t*>(ws + L.off_cnt_req);
    a.cnt_rb = reinterpret_cast<uint32_t*>(ws + L.off_cnt_rb);
    a.rowpart = reinterpret_cast<float2*>(ws + L.off_rowpart);
    a.job = reinterpret_cast<int4*>(ws + L.off_job);
    a.jobpart = reinterpret_cast<float4*>(ws + L.off_jobpart);
    const size_t esz = p->logits_dtype == DSPARK_BF16 ? 2 : 4;
    const bool rows16 = ((size_t)p->V * esz) % 16 == 0;
    a.vec_b = rows16 && ((uintptr_t)base_logits % 16 == 0);
    a.vec_t = rows16 && ((uintptr_t)target_logits % 16 == 0);
    a.softcap = p->softcap;
    a.head_vec = head_vec;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, L.zero_bytes, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    void* args[] = {&a};
    const bool ws_rows = p->logits_dtype == DSPARK_BF16 && a.vec_t && p->B <= kVMaxB;
    if (ws_rows) {  // persistent streaming kernel: rows have one segment
        int per_sm = 0, sms = 0;
        if (prepare_kernel((const void*)verify_rows_ws_kernel, sizeof(VRSmem), kVThreads, &per_sm) != cudaSuccess ||
            per_sm < 1 || device_sm_count(&sms) != cudaSuccess)
            return DSPARK_ERR_CUDA;
        a.nseg = 1;
        const int G = std::max(1, std::min(p->B * p->gamma, sms * per_sm));
        if (cudaLaunchKernel((const void*)verify_rows_ws_kernel, dim3(G), dim3(kVThreads), args, sizeof(VRSmem), s) !=
            cudaSuccess)
            return DSPARK_ERR_CUDA;
        note_launch();
    } else {
        RowsFn rows = p->logits_dtype == DSPARK_BF16 ? verify_rows_kernel<__nv_bfloat16> : verify_rows_kernel<float>;
        if (cudaLaunchKernel((const void*)rows, dim3(L.nseg, p->gamma, p->B), dim3(kThreads), args, 0, s) !=
            cudaSuccess)
            return DSPARK_ERR_CUDA;
        note_launch();
    }
    // the tensor-core draws: dense target rows (the CSR layout's row count is not known on the host)
    if (!head_vec && ws_rows && !target_row_offsets && verify_tc_eligible(p, base_logits, target_logits, W1, W2)) {
        VerifyTcArgs t;
        t.B = p->B;
        t.gamma = p->gamma;
        t.V = p->V;
        t.nt = L.nt;
        t.nrb = (p->B + 127) / 128;
        t.greedy = a.greedy;
        t.scale2 = a.scale2;
        t.seed = p->seed;
        t.base = base_logits;
        t.target = target_logits;
        t.gamma_t = gamma_t;
        t.toff = nullptr;
        t.target_rows = (long long)p->B * gamma_t;
        t.W1 = W1;
        t.W2 = W2;
        t.job = a.job;
        t.dlse = draft_lse;
        t.corr = correction_token;
        t.fb = reinterpret_cast<int32_t*>(ws + L.off_fb);
        t.words = reinterpret_cast<unsigned long long*>(ws + L.off_tc_words);
        t.rb_count = reinterpret_cast<unsigned*>(ws + L.off_tc_count);
        t.hdr = a.hdr;
        t.limit_ns = a.limit_ns;
        if (t.target_rows >= 1) {
            st = launch_verify_tc(t, s);
            if (st != DSPARK_OK) return st;
            verify_fallback_kernel<__nv_bfloat16><<<p->B, kThreads, 0, s>>>(a, t.fb);
            if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
            note_launch();
            return DSPARK_OK;
        }
    }
    RowsFn jobs = pick_jobs(p, mma);
    size_t smem = sizeof(float) * kRows * kXRow + sizeof(float2) * kRows * kChunks + align_up(sizeof(RowBlock), 16) +
                  sizeof(int4) * kRows + sizeof(float) * 64 + (mma ? 0 : sizeof(float) * kRows * (size_t)p->r);
    if (smem > kMaxSmem) return DSPARK_ERR_UNSUPPORTED;
    int per_sm = 0;
    if (prepare_kernel((const void*)jobs, smem, kThreads, &per_sm) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (cudaLaunchKernel((const void*)jobs, dim3(L.nt, L.nrb), dim3(kThreads), args, smem, s) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    note_launch();
    return DSPARK_OK;
}

}  // namespace

extern "C" dspark_status dspark_verify(const dspark_sample_params* p, const void* base_logits, const void* W1,
                                       const void* W2, const int32_t* anchor, const int32_t* tokens,
                                       const float* draft_lse, const float* draft_logit_at_tok,
                                       const void* target_logits, int gamma_t, const int32_t* verify_len,
                                       const int32_t* target_row_offsets, int32_t* n_accepted,
                                       int32_t* correction_token, void* workspace, size_t ws_bytes,
                                       dspark_stream_t stream) {
    return verify_impl(p, base_logits, W1, nullptr, W2, anchor, tokens, draft_lse, draft_logit_at_tok,
                       target_logits, gamma_t, verify_len, target_row_offsets, n_accepted, correction_token,
                       workspace, ws_bytes, stream);
}

extern "C" dspark_status dspark_verify_head(const dspark_sample_params* p, const void* base_logits,
                                            const float* head_vec, const void* W2, const int32_t* anchor,
                                            const int32_t* tokens, const float* draft_lse,
                                            const float* draft_logit_at_tok, const void* target_logits, int gamma_t,
                                            const int32_t* verify_len, const int32_t* target_row_offsets,
                                            int32_t* n_accepted, int32_t* correction_token, void* workspace,
                                            size_t ws_bytes, dspark_stream_t stream) {
    if (!p || p->r < 1 || !head_vec) return DSPARK_ERR_INVALID_ARG;
    return verify_impl(p, base_logits, nullptr, head_vec, W2, anchor, tokens, draft_lse, draft_logit_at_tok,
                       target_logits, gamma_t, verify_len, target_row_offsets, n_accepted, correction_token,
                       workspace, ws_bytes, stream);
}
