// schedule.cu -- dspark_schedule_verify_len: confidence-scheduled verify lengths.
//
// Method (P3 "如何评价 DeepSeek 发布 DSpark？" section "置信度调度与验证截断": choose L_j in
// [1, K] to maximise sum_j sum_{i<=L_j} c~^(j)_{t+i} under the SLA; survival is the product
// of conditional confidences, P2 section 3.8.3).  The SLA is read as a verify-token budget.
// Contract in dspark.h: a = left-to-right fp32 product of clamped c; every request verifies
// one token; the other budget - B slots go to the largest a_{j,i}, i >= 2, ordered by
// (a desc, j asc, i asc).
//
// One block: the survival values (fp32 bit patterns, order-preserving for a >= 0) are selected
// with an 8-bit-digit radix select for the K-th largest, ties at the threshold are taken in
// index order with a block-wide prefix count, and L_j / offsets / objective follow from
// block scans.  All decisions are integer or exact fp32, so the result is bit-identical to a
// sequential implementation of the same definition.  When the budget covers every position the
// selection is skipped (L_j = gamma).
//
// The file also holds dspark_theta_schedule, the throughput-aware prefix choice with a causal
// stop (P4 "DSpark 深度解读：DeepSeek-V4 如何用「半自回归」把推理速度提升 85%" section 5.1):
// one request per thread, decisions in IEEE single precision.
#include "common.cuh"
#include "host_util.h"

namespace dspark {
namespace {

constexpr int kSchedThreads = 1024;
constexpr int kSchedWarps = kSchedThreads / 32;
constexpr int kMaxCells = 16384;

// Exclusive block scan of one int per thread (thread order); returns the block total too.
__device__ int block_excl_scan(int v, int* tot, int* sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += t;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kSchedWarps ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        sh[32 + lane] = w;  // inclusive prefix of warp totals
    }
    __syncthreads();
    const int before = (warp > 0 ? sh[32 + warp - 1] : 0) + x - v;
    *tot = sh[32 + kSchedWarps - 1];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(kSchedThreads, 1)
    schedule_kernel(int B, int gamma, const float* __restrict__ conf, int budget, int32_t* __restrict__ L_out,
                    int32_t* __restrict__ off_out, float* __restrict__ obj_out, int32_t* __restrict__ status) {
    extern __shared__ uint32_t a_bits[];  // [B * gamma]
    __shared__ int hist[256];
    __shared__ int scan_sh[64];
    __shared__ uint32_t s_prefix, s_mask;
    __shared__ int s_rem;
    __shared__ double red_d[kSchedWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) *status = DSPARK_OK;  // one block and no device-side error: the status word is just reset

    // survival a_{j,i}: left-to-right fp32 products of clamped confidences
    for (int j = tid; j < B; j += kSchedThreads) {
        float run = 1.f;
        for (int i = 0; i < gamma; ++i) {
            float c = conf[(size_t)j * gamma + i];
            if (!(c >= 0.f)) c = 0.f;
            if (c > 1.f) c = 1.f;
            run = __fmul_rn(run, c);
            a_bits[j * gamma + i] = __float_as_uint(run);
        }
    }
    const int K = budget - B;                  // extra slots
    const int ncand = B * (gamma - 1);         // candidates: positions i >= 2
    if (K >= ncand) {  // the budget covers every position: L_j = gamma, no selection
        // the same contiguous rows per thread and summation order as the general path below
        __syncthreads();
        const int rpt = (B + kSchedThreads - 1) / kSchedThreads;
        const int r0 = min(B, tid * rpt), r1 = min(B, r0 + rpt);
        double obj = 0.0;
        for (int j = r0; j < r1; ++j) {
            for (int i = 0; i < gamma; ++i) obj += (double)__uint_as_float(a_bits[j * gamma + i]);
            L_out[j] = gamma;
            off_out[j] = j * gamma;
        }
        if (tid == 0) off_out[B] = B * gamma;
        if (obj_out) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) obj += __shfl_xor_sync(0xffffffffu, obj, o);
            if (lane == 0) red_d[warp] = obj;
            __syncthreads();
            if (warp == 0) {
                double q = lane < kSchedWarps ? red_d[lane] : 0.0;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
                if (lane == 0) obj_out[0] = (float)q;
            }
        }
        return;
    }
    if (tid == 0) {
        s_prefix = 0u;
        s_mask = 0u;
        s_rem = K;
    }
    __syncthreads();
    const bool all_full = K >= ncand, none = K <= 0;
    if (!all_full && !none) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            if (tid < 256) hist[tid] = 0;
            __syncthreads();
            const uint32_t pre = s_prefix, msk = s_mask;
            for (int q = tid; q < ncand; q += kSchedThreads) {
                const int j = q / (gamma - 1), i = q % (gamma - 1) + 1;
                const uint32_t b = a_bits[j * gamma + i];
                if ((b & msk) == pre) atomicAdd(&hist[(b >> shift) & 255u], 1);
            }
            __syncthreads();
            if (tid == 0) {  // largest digit whose cumulative count from the top reaches rem
                int rem = s_rem, cum = 0, d = 255;
                for (; d > 0; --d) {
                    if (cum + hist[d] >= rem) break;
                    cum += hist[d];
                }
                s_rem = rem - cum;
                s_prefix = pre | ((uint32_t)d << shift);
                s_mask = msk | (255u << shift);
            }
            __syncthreads();
        }
    }
    const uint32_t theta = s_prefix;  // the K-th largest survival (bit pattern)
    const int need_eq = s_rem;        // how many values equal to theta are taken, in index order

    // per-thread contiguous row ranges
    const int rpt = (B + kSchedThreads - 1) / kSchedThreads;
    const int r0 = min(B, tid * rpt), r1 = min(B, r0 + rpt);
    int eq_cnt = 0;
    if (!all_full && !none)
        for (int j = r0; j < r1; ++j)
            for (int i = 1; i < gamma; ++i) eq_cnt += (a_bits[j * gamma + i] == theta);
    int eq_tot;
    int eq_before = block_excl_scan(eq_cnt, &eq_tot, scan_sh);
    int lsum = 0;
    double obj = 0.0;
    int Lr[64];  // rows per thread <= kMaxCells / kSchedThreads
    for (int j = r0; j < r1; ++j) {
        int Lj;
        if (all_full) {
            Lj = gamma;
        } else if (none) {
            Lj = 1;
        } else {
            int gt = 0, eq = 0;
            for (int i = 1; i < gamma; ++i) {
                const uint32_t b = a_bits[j * gamma + i];
                gt += (b > theta);
                eq += (b == theta);
            }
            const int take = max(0, min(eq, need_eq - eq_before));
            eq_before += eq;
            Lj = 1 + gt + take;
        }
        Lr[j - r0] = Lj;
        lsum += Lj;
        for (int i = 0; i < Lj; ++i) obj += (double)__uint_as_float(a_bits[j * gamma + i]);
    }
    int ltot;
    int lbefore = block_excl_scan(lsum, &ltot, scan_sh);
    for (int j = r0; j < r1; ++j) {
        L_out[j] = Lr[j - r0];
        off_out[j] = lbefore;
        lbefore += Lr[j - r0];
    }
    if (tid == 0) off_out[B] = ltot;
    if (obj_out) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) obj += __shfl_xor_sync(0xffffffffu, obj, o);
        if (lane == 0) red_d[warp] = obj;
        __syncthreads();
        if (warp == 0) {
            double q = lane < kSchedWarps ? red_d[lane] : 0.0;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
            if (lane == 0) obj_out[0] = (float)q;
        }
    }
}

// Throughput-aware prefix choice, one request per thread, in IEEE single precision with explicit
// round-to-nearest operations (no contraction), in the order of the definition.
__global__ void theta_kernel(int B, int gamma, const float* __restrict__ conf, const float* __restrict__ sps,
                             int32_t* __restrict__ ell, float* __restrict__ theta) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= B) return;
    float a = 1.f, acc = 0.f, prev = -CUDART_INF_F;
    int out = gamma;
    bool stopped = false;
    for (int l = 0; l <= gamma; ++l) {
        float th = CUDART_NAN_F;
        if (!stopped) {
            if (l > 0) {
                a = __fmul_rn(a, conf[(size_t)j * gamma + l - 1]);
                acc = __fadd_rn(acc, a);
            }
            th = __fmul_rn(__fadd_rn(1.f, acc), sps[l]);
            if (l > 0 && th < prev) {
                out = l - 1;
                stopped = true;
            }
            prev = th;
        }
        if (theta) theta[(size_t)j * (gamma + 1) + l] = th;
    }
    ell[j] = out;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_schedule_workspace_size(int B, int gamma) {
    (void)B;
    (void)gamma;
    return kHeaderBytes;
}

extern "C" dspark_status dspark_schedule_verify_len(int B, int gamma, const float* conf, int budget,
                                                    int32_t* verify_len, int32_t* offsets, float* objective,
                                                    void* workspace, size_t ws_bytes, dspark_stream_t stream) {
    if (B < 1 || gamma < 1 || !conf || !verify_len || !offsets) return DSPARK_ERR_INVALID_ARG;
    if ((long long)B * gamma > kMaxCells) return DSPARK_ERR_UNSUPPORTED;
    if (budget < B) return DSPARK_ERR_BUDGET;
    if (!workspace || ((uintptr_t)workspace & 255u) || ws_bytes < kHeaderBytes) return DSPARK_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const long long bg = (long long)B * gamma;
    const int budget_c = (long long)budget > bg ? (int)bg : budget;
    const size_t smem = sizeof(uint32_t) * (size_t)bg;
    int per_sm = 0;
    if (prepare_kernel((const void*)schedule_kernel, smem, kSchedThreads, &per_sm) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    schedule_kernel<<<1, kSchedThreads, smem, s>>>(B, gamma, conf, budget_c, verify_len, offsets, objective,
                                                   &static_cast<WsHeader*>(workspace)->status);
    if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
    note_launch();
    return DSPARK_OK;
}

extern "C" dspark_status dspark_theta_schedule(int B, int gamma, const float* conf, const float* sps, int32_t* ell,
                                               float* theta, dspark_stream_t stream) {
    if (B < 1 || gamma < 1 || !conf || !sps || !ell) return DSPARK_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    theta_kernel<<<(unsigned)((B + 127) / 128), 128, 0, s>>>(B, gamma, conf, sps, ell, theta);
    if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
    note_launch();
    return DSPARK_OK;
}
