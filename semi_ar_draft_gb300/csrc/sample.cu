// sample.cu -- dspark_markov_sample_block: Markov-head block sampling.
//
// Method (P2 "从 DFlash 到 dLLM Self-Spec（三）" section 3.4, VanillaMarkov and the
// sample_block_tokens loop; P1 "03 · DSpark 建模：Markov 与 Confidence" section 3.7):
// for i = 1..gamma, z = base_i + W2 . W1[prev]; sample; prev = sampled.  The sampling
// contract is the tile-Gumbel draw stated in dspark.h.
//
// One persistent cooperative kernel runs all gamma steps:
//   - vocabulary split: block b owns tiles t = b, b + G, ... (G <= number of SMs);
//   - per step and tile, rows go in blocks of 16 requests: the producer writes z = base + bias
//     for 16 rows x 1024 ids to shared memory with per-32-id chunk statistics (tensor-core
//     mma.sync bias with the accumulator initialised from the base logits, or a CUDA-core GEMV
//     for fp32 weights); a warp per row turns them into the tile's record {Gumbel key, log-mass,
//     in-tile candidate, z at it} in global scratch;
//   - bounded grid-wide wait; block b reduces the records of requests b, b + G, ... to the
//     step's token, LSE(z/T) and z at the token; bounded grid-wide wait; next step.
// When each block owns a single tile and the W2 rows of it fit, they are staged in shared
// memory once for all gamma steps.
#include <algorithm>
#include <atomic>
#include <cmath>

#include "host_util.h"
#include "markov_tile.cuh"

namespace dspark {
namespace {

struct SampleArgs {
    int B, gamma, V, r, nt, G;
    int greedy;
    float scale2;  // log2(e) / T
    uint64_t seed;
    const void* base;
    const void* W1;
    const void* W2;
    const int32_t* anchor;
    int32_t* tokens;
    float* draft_lse;
    float* zat;
    WsHeader* hdr;
    int32_t* cur_tok;
    float4* part;  // [2][B][nt] tile records, by step parity
    uint64_t limit_ns;
    int redundant;  // every block reduces every request (one grid-wide wait per step)
    int w2_smem;
    int vec_ok;  // base rows start on 16-byte boundaries: 8-wide loads and L2 prefetch allowed
};

size_t sample_smem_bytes(int B, int r, bool mma, bool w2_smem) {
    size_t b = sizeof(float) * kRows * kXRow + sizeof(float2) * kRows * kChunks + align_up(sizeof(RowBlock), 16) +
               align_up(sizeof(int) * (size_t)B, 16) + sizeof(float4) * (size_t)B;
    if (mma) {
        if (w2_smem) b += (size_t)kTS * r * 2;
    } else {
        b += sizeof(float) * kRows * (size_t)r;
    }
    return b;
}

// The step's random draws of every request that do not depend on the drafted tokens:
// (u1, u2) of SAMPLE_INTILE (one Philox call, words 0 and 1) and ln E of this block's first tile.
__device__ void step_randoms(const SampleArgs& a, int step, float4* rnd) {
    const uint32_t i = (uint32_t)step + 1u;
    for (int j = threadIdx.x; j < a.B; j += kThreads) {
        const uint4 w = philox10(make_uint4(0u, i, (uint32_t)j, DSPARK_P_SAMPLE_INTILE), (uint32_t)a.seed,
                                 (uint32_t)(a.seed >> 32));
        const float lnE = log_neg_log_u(uniform(a.seed, (uint32_t)j, i, DSPARK_P_SAMPLE_TILE, blockIdx.x));
        rnd[j] = make_float4(u01(w.x), u01(w.y), lnE, 0.f);
    }
}

// L2 prefetch of the base rows of row block [row0, row0 + 16) at `step` over this block's tile.
template <typename TL>
__device__ void prefetch_rows(const SampleArgs& a, int tile, int row0, int step) {
    const int q = threadIdx.x;
    if (!a.vec_ok || q >= kRows || row0 + q >= a.B || step >= a.gamma || tile >= a.nt) return;
    const int tile0 = tile * kTS;
    const int n = min(kTS, a.V - tile0);
    const TL* p = reinterpret_cast<const TL*>(a.base) + ((size_t)(row0 + q) * a.gamma + step) * (size_t)a.V + tile0;
    prefetch_l2(p, (uint32_t)(n * sizeof(TL)));
}

template <typename TL, int KS, typename TW, bool GREEDY>
__global__ void __launch_bounds__(kThreads, 1) sample_kernel(SampleArgs a) {
    constexpr bool kMMA = KS > 0;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* xbuf = reinterpret_cast<float*>(smem_raw);                  // [kRows][kXRow]: z
    float2* cstat = reinterpret_cast<float2*>(xbuf + kRows * kXRow);   // [kRows][kChunks]
    RowBlock* rb = reinterpret_cast<RowBlock*>(cstat + kRows * kChunks);
    int* prev = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(rb) + align_up(sizeof(RowBlock), 16));
    float4* rnd = reinterpret_cast<float4*>(reinterpret_cast<unsigned char*>(prev) + align_up(sizeof(int) * (size_t)a.B, 16));
    unsigned char* wreg = reinterpret_cast<unsigned char*>(rnd + a.B);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    ProdArgs pa;
    pa.base = a.base;
    pa.target = nullptr;
    pa.W1 = a.W1;
    pa.W2 = a.W2;
    pa.w2s = nullptr;
    pa.w1s = reinterpret_cast<const float*>(wreg);
    pa.V = a.V;
    pa.r = a.r;
    pa.greedy = a.greedy;
    pa.scale2 = a.scale2;
    pa.vec_b = a.vec_ok;
    pa.vec_t = 0;
    if constexpr (kMMA) {
        if (a.w2_smem) {
            stage_w2_tile<KS>(reinterpret_cast<const uint16_t*>(a.W2), blockIdx.x * kTS, a.V,
                              reinterpret_cast<uint4*>(wreg));
            pa.w2s = reinterpret_cast<const uint4*>(wreg);
        }
    }
    prefetch_rows<TL>(a, blockIdx.x, 0, 0);
    if (!a.greedy) step_randoms(a, 0, rnd);

    uint32_t target = 0;
    const size_t part_stride = (size_t)a.B * a.nt;
    for (int step = 0; step < a.gamma; ++step) {
        float4* part = a.part + (size_t)(step & 1) * part_stride;
        if (step == 0 || !a.redundant) {
            for (int j = tid; j < a.B; j += kThreads) {
                int p = step == 0 ? a.anchor[j] : __ldcg(a.cur_tok + j);
                if (p < 0 || p >= a.V) {  // a bad anchor, or a row whose tiles all had no mass
                    record_status(&a.hdr->status, DSPARK_ERR_TOKEN_RANGE);
                    p = min(max(p, 0), a.V - 1);
                }
                prev[j] = p;
            }
        }
        __syncthreads();
        for (int tile = blockIdx.x; tile < a.nt; tile += a.G) {
            for (int row0 = 0; row0 < a.B; row0 += kRows) {
                if (tid < kRows) {
                    const int j = row0 + tid;
                    const bool ok = j < a.B;
                    rb->prev[tid] = ok ? prev[j] : 0;
                    rb->mode[tid] = ok ? ROW_SAMPLE : ROW_OFF;
                    rb->brow[tid] = ok ? ((long long)j * a.gamma + step) * (long long)a.V : -1;
                    rb->trow[tid] = -1;
                    float4 q = ok && !a.greedy ? rnd[j] : make_float4(0.f, 0.f, 0.f, 0.f);
                    if (ok && !a.greedy && tile != blockIdx.x)  // blocks owning several tiles: per-tile variate
                        q.z = log_neg_log_u(uniform(a.seed, (uint32_t)j, (uint32_t)step + 1u, DSPARK_P_SAMPLE_TILE,
                                                    (uint32_t)tile));
                    rb->u1[tid] = q.x;
                    rb->u2[tid] = q.y;
                    rb->lnE[tid] = q.z;
                }
                // the next row block of this step (the first of the next step is prefetched at the wait)
                if (row0 + kRows < a.B) prefetch_rows<TL>(a, tile, row0 + kRows, step);
                if constexpr (!kMMA) {
                    __syncthreads();
                    float* w1s = reinterpret_cast<float*>(wreg);
                    const TW* W1 = reinterpret_cast<const TW*>(a.W1);
                    for (int idx = tid; idx < kRows * a.r; idx += kThreads) {
                        const int q = idx / a.r, k = idx % a.r;
                        w1s[idx] = (rb->brow[q] >= 0) ? load_logit<TW>(W1, (size_t)rb->prev[q] * a.r + k) : 0.f;
                    }
                }
                __syncthreads();
                if constexpr (kMMA) {
                    const TL* base = reinterpret_cast<const TL*>(a.base);
                    const uint16_t* W1 = reinterpret_cast<const uint16_t*>(a.W1);
                    const uint16_t* W2 = reinterpret_cast<const uint16_t*>(a.W2);
                    const bool full = (tile + 1) * kTS <= a.V && a.vec_ok;
                    if (pa.w2s) {
                        if (full) produce_sample<TL, KS, GREEDY, true, true>(base, W1, W2, pa.w2s, a.V, true, tile, *rb, xbuf, cstat, a.scale2);
                        else produce_sample<TL, KS, GREEDY, true, false>(base, W1, W2, pa.w2s, a.V, a.vec_ok, tile, *rb, xbuf, cstat, a.scale2);
                    } else {
                        if (full) produce_sample<TL, KS, GREEDY, false, true>(base, W1, W2, nullptr, a.V, true, tile, *rb, xbuf, cstat, a.scale2);
                        else produce_sample<TL, KS, GREEDY, false, false>(base, W1, W2, nullptr, a.V, a.vec_ok, tile, *rb, xbuf, cstat, a.scale2);
                    }
                } else {
                    produce_chunks<TL, KS, TW, false>(pa, tile, *rb, xbuf, cstat);
                }
                __syncthreads();
                for (int rl = warp; rl < kRows; rl += kWarps) {
                    const int j = row0 + rl;
                    if (j >= a.B) continue;
                    const float4 rec = finalize_tile(xbuf + rl * kXRow, cstat[rl * kChunks + lane], tile, a.V,
                                                     GREEDY, a.scale2, rb->u1[rl], rb->u2[rl], rb->lnE[rl]);
                    if (lane == 0) part[(size_t)j * a.nt + tile] = rec;
                }
                __syncthreads();
            }
        }
        // Everything of the next step that does not depend on its tokens happens while the
        // last blocks arrive: its random draws and the L2 prefetch of its first row block.
        target += (uint32_t)a.G;
        grid_arrive(a.hdr);
        if (step + 1 < a.gamma) {
            prefetch_rows<TL>(a, blockIdx.x, 0, step + 1);
            if (!a.greedy) step_randoms(a, step + 1, rnd);
        }
        if (!grid_wait_arrived(a.hdr, target, a.limit_ns)) return;
        if (a.redundant) {
            // every block reduces every request: width = threads per request (power of two)
            int width = kThreads / a.B;
            width = width >= 32 ? 32 : (width >= 16 ? 16 : (width >= 8 ? 8 : (width >= 4 ? 4 : (width >= 2 ? 2 : 1))));
            const int per_pass = kThreads / width;
            for (int jb = 0; jb < a.B; jb += per_pass) {  // uniform trip count: every lane reaches the shuffles
                const int j = jb + tid / width, sub = tid % width;
                const TileAcc w = reduce_tiles_group(part + (size_t)min(j, a.B - 1) * a.nt, a.nt, sub, width, !GREEDY);
                if (sub == 0 && j < a.B) {
                    prev[j] = w.cand;
                    if ((int)blockIdx.x == j % a.G) {
                        const size_t o = (size_t)j * a.gamma + step;
                        a.tokens[o] = w.cand;
                        a.draft_lse[o] = a.greedy ? CUDART_NAN_F : tile_acc_lse(w);
                        a.zat[o] = w.val;
                    }
                }
            }
            __syncthreads();
            for (int j = tid; j < a.B; j += kThreads)
                if (prev[j] < 0 || prev[j] >= a.V) {  // only when every tile of a row had no mass
                    record_status(&a.hdr->status, DSPARK_ERR_TOKEN_RANGE);
                    prev[j] = min(max(prev[j], 0), a.V - 1);
                }
        } else {
            for (int j = blockIdx.x + a.G * warp; j < a.B; j += a.G * kWarps) {
                const TileAcc w = reduce_tiles_group(part + (size_t)j * a.nt, a.nt, lane, 32, !GREEDY);
                if (lane == 0) {
                    a.cur_tok[j] = w.cand;
                    const size_t o = (size_t)j * a.gamma + step;
                    a.tokens[o] = w.cand;
                    a.draft_lse[o] = a.greedy ? CUDART_NAN_F : tile_acc_lse(w);
                    a.zat[o] = w.val;
                }
            }
            if (step + 1 < a.gamma) {
                target += (uint32_t)a.G;
                if (!grid_wait(a.hdr, target, a.limit_ns)) return;
            }
        }
    }
}

using KernelFn = void (*)(SampleArgs);

template <typename TL, bool G>
KernelFn pick_mma(int r) {
    switch (r) {
        case 16: return sample_kernel<TL, 1, uint16_t, G>;
        case 32: return sample_kernel<TL, 2, uint16_t, G>;
        case 64: return sample_kernel<TL, 4, uint16_t, G>;
        case 128: return sample_kernel<TL, 8, uint16_t, G>;
        case 256: return sample_kernel<TL, 16, uint16_t, G>;
        default: return nullptr;
    }
}

template <bool G>
KernelFn pick_kernel_g(const dspark_sample_params* p, bool mma) {
    const bool lb = p->logits_dtype == DSPARK_BF16;
    if (mma) return lb ? pick_mma<__nv_bfloat16, G>(p->r) : pick_mma<float, G>(p->r);
    const bool wb = p->w_dtype == DSPARK_BF16;
    if (lb) return wb ? sample_kernel<__nv_bfloat16, 0, __nv_bfloat16, G> : sample_kernel<__nv_bfloat16, 0, float, G>;
    return wb ? sample_kernel<float, 0, __nv_bfloat16, G> : sample_kernel<float, 0, float, G>;
}

KernelFn pick_kernel(const dspark_sample_params* p, bool mma) {
    return p->temperature == 0.f ? pick_kernel_g<true>(p, mma) : pick_kernel_g<false>(p, mma);
}

}  // namespace

bool markov_use_mma(const dspark_sample_params* p) {
    return p->r > 0 && p->w_dtype == DSPARK_BF16 &&
           (p->r == 16 || p->r == 32 || p->r == 64 || p->r == 128 || p->r == 256);
}

dspark_status validate_sample_params(const dspark_sample_params* p) {
    if (!p) return DSPARK_ERR_INVALID_ARG;
    if (p->B < 1 || p->gamma < 1 || p->V < 1 || p->r < 0) return DSPARK_ERR_INVALID_ARG;
    if (!(p->temperature >= 0.f) || std::isinf(p->temperature)) return DSPARK_ERR_INVALID_ARG;
    if (p->logits_dtype != DSPARK_F32 && p->logits_dtype != DSPARK_BF16) return DSPARK_ERR_INVALID_ARG;
    if (p->r > 0 && p->w_dtype != DSPARK_F32 && p->w_dtype != DSPARK_BF16) return DSPARK_ERR_INVALID_ARG;
    if (p->B > 4096 || p->r > 1024 || p->gamma > 1024) return DSPARK_ERR_UNSUPPORTED;
    return DSPARK_OK;
}

size_t sample_workspace_bytes(const dspark_sample_params* p) {
    const size_t nt = (size_t)(p->V + kTS - 1) / kTS;
    return kHeaderBytes + align_up(sizeof(int32_t) * (size_t)p->B, 256) +
           align_up(2 * sizeof(float4) * (size_t)p->B * nt, 256);
}

}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_sample_workspace_size(const dspark_sample_params* p) {
    if (validate_sample_params(p) != DSPARK_OK) return 0;
    return sample_workspace_bytes(p);
}

extern "C" dspark_status dspark_markov_sample_block(const dspark_sample_params* p, const void* base_logits,
                                                    const void* W1, const void* W2, const int32_t* anchor,
                                                    int32_t* tokens, float* draft_lse, float* draft_logit_at_tok,
                                                    void* workspace, size_t ws_bytes, dspark_stream_t stream) {
    dspark_status st = validate_sample_params(p);
    if (st != DSPARK_OK) return st;
    if (!base_logits || !anchor || !tokens || !draft_lse || !draft_logit_at_tok) return DSPARK_ERR_INVALID_ARG;
    if (p->r > 0 && (!W1 || !W2)) return DSPARK_ERR_INVALID_ARG;
    if (!workspace || ((uintptr_t)workspace & 255u) || ws_bytes < sample_workspace_bytes(p))
        return DSPARK_ERR_WORKSPACE;

    const bool mma = markov_use_mma(p);
    const int nt = (p->V + kTS - 1) / kTS;
    int sms = 0;
    if (device_sm_count(&sms) != cudaSuccess) return DSPARK_ERR_CUDA;
    KernelFn fn = pick_kernel(p, mma);
    bool w2_smem = mma && (size_t)kTS * p->r * 2 <= 128 * 1024 && nt <= sms;
    size_t smem = sample_smem_bytes(p->B, p->r, mma, w2_smem);
    if (smem > kMaxSmem && w2_smem) {
        w2_smem = false;
        smem = sample_smem_bytes(p->B, p->r, mma, false);
    }
    if (smem > kMaxSmem) return DSPARK_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, (const void*)fn, kThreads, smem) != cudaSuccess ||
        per_sm < 1)
        return DSPARK_ERR_CUDA;
    const int G = std::min(nt, sms * per_sm);
    if (G < nt) w2_smem = false;  // a block owning several tiles cannot keep one tile's W2

    SampleArgs a;
    a.B = p->B;
    a.gamma = p->gamma;
    a.V = p->V;
    a.r = p->r;
    a.nt = nt;
    a.G = G;
    a.greedy = p->temperature == 0.f;
    a.scale2 = a.greedy ? 1.f : kLog2e / p->temperature;
    a.seed = p->seed;
    a.base = base_logits;
    a.W1 = W1;
    a.W2 = W2;
    a.anchor = anchor;
    a.tokens = tokens;
    a.draft_lse = draft_lse;
    a.zat = draft_logit_at_tok;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    a.hdr = reinterpret_cast<WsHeader*>(ws);
    a.cur_tok = reinterpret_cast<int32_t*>(ws + kHeaderBytes);
    a.part = reinterpret_cast<float4*>(ws + kHeaderBytes + align_up(sizeof(int32_t) * (size_t)p->B, 256));
    a.limit_ns = wait_limit_ns();
    a.redundant = (size_t)p->B * nt <= 8192 && p->B <= kThreads;
    a.w2_smem = w2_smem;
    const size_t esz = p->logits_dtype == DSPARK_BF16 ? 2 : 4;
    a.vec_ok = ((uintptr_t)base_logits % 16 == 0) && (((size_t)p->V * esz) % 16 == 0);

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, kHeaderBytes, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    void* args[] = {&a};
    if (cudaLaunchCooperativeKernel((const void*)fn, dim3(G), dim3(kThreads), args, smem, s) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    return DSPARK_OK;
}

// ------------------------------------------------------------------------------------------
// No-allocation variant: the scratch of dspark_markov_sample_block lives in this file-scope
// device array.  Host code must not use the array's name as an address (it names a host-side
// stand-in); the device address is looked up once per device with cudaGetSymbolAddress.
// ------------------------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[DSPARK_NOALLOC_SCRATCH_BYTES];
static std::atomic<void*> g_noalloc_addr[64];

extern "C" dspark_status dspark_markov_sample_block_noalloc(const dspark_sample_params* p, const void* base_logits,
                                                           const void* W1, const void* W2, const int32_t* anchor,
                                                           int32_t* tokens, float* draft_lse,
                                                           float* draft_logit_at_tok, dspark_stream_t stream) {
    const dspark_status st = validate_sample_params(p);
    if (st != DSPARK_OK) return st;
    const size_t need = sample_workspace_bytes(p);
    if (need > DSPARK_NOALLOC_SCRATCH_BYTES) return DSPARK_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DSPARK_ERR_CUDA;
    void* scratch = g_noalloc_addr[dev].load();
    if (!scratch) {  // first call on this device: this device is current
        if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || !scratch) return DSPARK_ERR_CUDA;
        g_noalloc_addr[dev].store(scratch);
    }
    // Same kernel and launch as the workspace entry point; it zeroes the scratch header
    // (status word and grid-wait counter) before the launch.
    return dspark_markov_sample_block(p, base_logits, W1, W2, anchor, tokens, draft_lse, draft_logit_at_tok, scratch,
                                      DSPARK_NOALLOC_SCRATCH_BYTES, stream);
}
