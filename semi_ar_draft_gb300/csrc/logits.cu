// logits.cu -- dspark_markov_block_logits: teacher-forced block logits of the Markov head.
//
// Method (P1 "03 · DSpark 建模：Markov 与 Confidence", section on build_markov_head /
// VanillaMarkov, Eq. 5): at training time every position's bias comes from its true previous
// token, all positions at once,
//     z_{j,i} = base_{j,i} + W2 W1[prev_{j,i}],  prev_{j,1} = anchor_j,  prev_{j,i} = x_{j,i-1},
// the sampling path's a1 + a2 without the draw.  One block per (1024-id tile, 16 flattened
// (request, position) rows) runs the sampler's producer (tensor-core bias when the weights are
// bf16 and r is in {16..256}, CUDA cores otherwise), which leaves z in shared memory, and writes
// the tile of z out row by row.
#include "common.cuh"
#include "host_util.h"
#include "markov_tile.cuh"

namespace dspark {
namespace {

struct BLArgs {
    int B, gamma, V, r;
    const void* base;
    const void* W1;
    const void* W2;
    const int32_t* anchor;
    const int32_t* tokens;
    float* z;
    int vec_b;
    float softcap;  // draft softcap of the base logits (0: none)
    WsHeader* hdr;
};

template <typename TL, int KS, typename TW>
__global__ void __launch_bounds__(kThreads, 1) block_logits_kernel(BLArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* xbuf = reinterpret_cast<float*>(smem_raw);                 // [kRows][kXRow]: z of the tile
    float2* cstat = reinterpret_cast<float2*>(xbuf + kRows * kXRow);  // [kRows][kChunks] (not used here)
    RowBlock* rb = reinterpret_cast<RowBlock*>(cstat + kRows * kChunks);
    float* w1s = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(rb) + align_up(sizeof(RowBlock), 16));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, tile0 = tile * kTS;
    const long long row0 = (long long)blockIdx.y * kRows, nrows = (long long)a.B * a.gamma;
    if (tid < kRows) {
        const long long rr = row0 + tid;
        int prev = 0, mode = ROW_OFF;
        long long brow = -1;
        if (rr < nrows) {
            const int j = (int)(rr / a.gamma), i = (int)(rr % a.gamma);
            prev = i == 0 ? a.anchor[j] : a.tokens[(size_t)j * a.gamma + i - 1];
            if (prev < 0 || prev >= a.V) {
                record_status(&a.hdr->status, DSPARK_ERR_TOKEN_RANGE);
                prev = min(max(prev, 0), a.V - 1);
            }
            mode = ROW_SAMPLE;
            brow = rr * a.V;
        }
        rb->prev[tid] = prev;
        rb->mode[tid] = mode;
        rb->brow[tid] = brow;
        rb->trow[tid] = -1;
        rb->u1[tid] = rb->u2[tid] = rb->lnE[tid] = rb->lse2[tid] = rb->dl2[tid] = 0.f;
    }
    __syncthreads();
    if constexpr (KS == 0) {
        const TW* W1 = reinterpret_cast<const TW*>(a.W1);
        for (int idx = tid; idx < kRows * a.r; idx += kThreads) {
            const int q = idx / a.r, k = idx % a.r;
            w1s[idx] = (rb->brow[q] >= 0) ? load_logit<TW>(W1, (size_t)rb->prev[q] * a.r + k) : 0.f;
        }
        __syncthreads();
    }
    ProdArgs pa;
    pa.base = a.base;
    pa.target = nullptr;
    pa.W1 = a.W1;
    pa.W2 = a.W2;
    pa.w2s = nullptr;
    pa.w1s = w1s;
    pa.V = a.V;
    pa.r = a.r;
    pa.greedy = 1;  // sampling rows keep z itself in the buffer
    pa.scale2 = 1.f;
    pa.vec_b = a.vec_b;
    pa.vec_t = 0;
    pa.softcap = a.softcap;
    pa.inv_softcap = a.softcap > 0.f ? 1.f / a.softcap : 0.f;
    produce_chunks<TL, KS, TW, false>(pa, tile, *rb, xbuf, cstat);
    __syncthreads();
    const int n = min(kTS, a.V - tile0);
    for (int q = warp; q < kRows; q += kWarps) {
        if (rb->mode[q] == ROW_OFF) continue;
        float* dst = a.z + (size_t)(row0 + q) * a.V + tile0;
        const float* src = xbuf + q * kXRow;
        for (int c = lane; c < n; c += 32) dst[c] = src[c];
    }
}

using BLFn = void (*)(BLArgs);

template <typename TL>
BLFn pick_mma(int r) {
    switch (r) {
        case 16: return block_logits_kernel<TL, 1, uint16_t>;
        case 32: return block_logits_kernel<TL, 2, uint16_t>;
        case 64: return block_logits_kernel<TL, 4, uint16_t>;
        case 128: return block_logits_kernel<TL, 8, uint16_t>;
        case 256: return block_logits_kernel<TL, 16, uint16_t>;
        default: return nullptr;
    }
}

BLFn pick(const dspark_sample_params* p, bool mma) {
    const bool lb = p->logits_dtype == DSPARK_BF16;
    if (mma) return lb ? pick_mma<__nv_bfloat16>(p->r) : pick_mma<float>(p->r);
    const bool wb = p->w_dtype == DSPARK_BF16;
    if (lb) return wb ? block_logits_kernel<__nv_bfloat16, 0, __nv_bfloat16> : block_logits_kernel<__nv_bfloat16, 0, float>;
    return wb ? block_logits_kernel<float, 0, __nv_bfloat16> : block_logits_kernel<float, 0, float>;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_markov_block_logits_workspace_size(const dspark_sample_params* p) {
    if (validate_sample_params(p) != DSPARK_OK) return 0;
    return kHeaderBytes;
}

extern "C" dspark_status dspark_markov_block_logits(const dspark_sample_params* p, const void* base_logits,
                                                    const void* W1, const void* W2, const int32_t* anchor,
                                                    const int32_t* tokens, float* z_out, void* workspace,
                                                    size_t ws_bytes, dspark_stream_t stream) {
    dspark_status st = validate_sample_params(p);
    if (st != DSPARK_OK) return st;
    if (!base_logits || !anchor || !z_out || (p->gamma > 1 && !tokens)) return DSPARK_ERR_INVALID_ARG;
    if (p->r > 0 && (!W1 || !W2)) return DSPARK_ERR_INVALID_ARG;
    if (!workspace || ((uintptr_t)workspace & 255u) || ws_bytes < kHeaderBytes) return DSPARK_ERR_WORKSPACE;
    const bool mma = markov_use_mma(p);
    BLFn fn = pick(p, mma);
    if (!fn) return DSPARK_ERR_UNSUPPORTED;
    BLArgs a;
    a.B = p->B;
    a.gamma = p->gamma;
    a.V = p->V;
    a.r = p->r;
    a.base = base_logits;
    a.W1 = W1;
    a.W2 = W2;
    a.anchor = anchor;
    a.tokens = tokens;
    a.z = z_out;
    const size_t esz = p->logits_dtype == DSPARK_BF16 ? 2 : 4;
    a.vec_b = ((size_t)p->V * esz) % 16 == 0 && (uintptr_t)base_logits % 16 == 0;
    a.softcap = p->softcap;
    a.hdr = static_cast<WsHeader*>(workspace);
    const size_t smem = sizeof(float) * kRows * kXRow + sizeof(float2) * kRows * kChunks +
                        align_up(sizeof(RowBlock), 16) + (mma ? 0 : sizeof(float) * kRows * (size_t)p->r);
    if (smem > kMaxSmem) return DSPARK_ERR_UNSUPPORTED;
    int per_sm = 0;
    if (prepare_kernel((const void*)fn, smem, kThreads, &per_sm) != cudaSuccess) return DSPARK_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, kHeaderBytes, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    const long long nrb = ((long long)p->B * p->gamma + kRows - 1) / kRows;
    const int nt = (p->V + kTS - 1) / kTS;
    if (nrb > 65535) return DSPARK_ERR_UNSUPPORTED;
    void* args[] = {&a};
    if (cudaLaunchKernel((const void*)fn, dim3(nt, (unsigned)nrb), dim3(kThreads), args, smem, s) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    note_launch();
    return DSPARK_OK;
}
