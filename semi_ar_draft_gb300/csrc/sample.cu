// sample.cu -- dspark_markov_sample_block: Markov-head block sampling.
//
// Method (P2 "从 DFlash 到 dLLM Self-Spec（三）" section 3.4, VanillaMarkov and the
// sample_block_tokens loop; P1 "03 · DSpark 建模：Markov 与 Confidence" section 3.7):
// for i = 1..gamma, z = base_i + W2 . W1[prev]; sample; prev = sampled.  The sampling
// contract is the chunk-Gumbel draw stated in dspark.h.
//
// One persistent cooperative kernel runs all gamma steps:
//   - vocabulary split: block b owns tiles t = b, b + G, ... (G <= number of SMs);
//   - per step and tile, rows go in blocks of 16 requests: the producer writes z = base + bias
//     for 16 rows x 1024 ids to shared memory with per-32-id chunk statistics (tensor-core
//     mma.sync bias with the accumulator initialised from the base logits, or a CUDA-core GEMV
//     for fp32 weights); a warp per row turns them into the tile's record {its best chunk key,
//     log-mass, that chunk's candidate, z at it} in global scratch;
//   - bounded grid-wide wait; block b reduces the records of requests b, b + G, ... to the
//     step's token, LSE(z/T) and z at the token; bounded grid-wide wait; next step.
// When each block owns a single tile and the W2 rows of it fit, they are staged in shared
// memory once for all gamma steps.
// Two kernels implement this: sample_staged_kernel (bf16 logits, tensor-core bias, one tile
// per block: base and W1 rows staged by the bulk-copy engine, tile winners exchanged through
// one packed atomic max per request and step, one grid-wide wait per step) and sample_kernel
// (every other case: fp32 logits, CUDA-core GEMV bias, vocabularies with more tiles than
// co-resident blocks; records reduced redundantly or by owner blocks).
#include <algorithm>
#include <atomic>
#include <cmath>

#include "host_util.h"
#include "markov_tile.cuh"

namespace dspark {
namespace {

constexpr int kMaxStagedTiles = 160;
constexpr int kSlotStride = 16;   // 64-bit words between two requests' maxima
constexpr int kCountStride = 32;  // 32-bit words between two row blocks' arrival counters

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
    float4* part;  // [3][B][nt] tile records, by step mod 2 (general kernel) or mod 3 (staged kernel)
    unsigned long long* slots;  // [gamma][B] packed (key, id) maxima of the staged kernel, kSlotStride words
                                // apart (one 128-byte line each, so the atomics spread over L2); zeroed per call
    unsigned* rb_count;         // [nrb] grid-wide arrival counters per row block (staged kernel), kCountStride apart
    uint64_t limit_ns;
    int redundant;  // every block reduces every request (one grid-wide wait per step)
    int w2_smem;
    int vec_ok;  // base rows start on 16-byte boundaries: 8-wide loads and L2 prefetch allowed
    float softcap, inv_softcap;  // draft softcap of the base logits (0: none)
    // Gated / RNN heads (general kernel): the vector u that W2 multiplies replaces W1[prev]
    int head;              // DSPARK_HEAD_*
    int hd;                // backbone hidden size d
    const float* hpre;     // [B][gamma][m r] hidden-state parts of the pre-activations (m = 1 gated, 3 rnn)
    const void* Wg;
    const void* Wc;
    const void* Wo;        // head weights (w_dtype): gated [r][d + r]; rnn [r][2r + d] each
    float* head_out;       // [B][gamma][r] the head vectors, or null
};

// Shared memory of the general kernel; a Gated / RNN head adds u [B][r] and, for the RNN head,
// two state buffers [2][B][r] (fp32).
size_t sample_smem_bytes(int B, int r, bool mma, bool w2_smem, int head = DSPARK_HEAD_VANILLA) {
    size_t b = sizeof(float) * kRows * kXRow + sizeof(float2) * kRows * kChunks + align_up(sizeof(RowBlock), 16) +
               align_up(sizeof(int) * (size_t)B, 16) + sizeof(float4) * (size_t)B;
    if (mma) {
        if (w2_smem) b += (size_t)kTS * r * 2;
    } else {
        b += sizeof(float) * kRows * (size_t)r;
    }
    if (head != DSPARK_HEAD_VANILLA) b += sizeof(float) * (size_t)B * r * (head == DSPARK_HEAD_RNN ? 3 : 1);
    return b;
}

// Head vectors of every request for `step` (all threads of the block; every block computes the
// same values in the same order, so all tiles use identical u):
//   gated: u_i = sigmoid(hpre_i + sum_c Wg[i][d + c] e_c) e_i,  e = W1[prev]
//   rnn:   a_t = hpre_t + sum_c Wt[i][c] s_c + sum_c Wt[i][r + c] e_c  (t = g, c, o),
//          s'_i = sigmoid(a_g) s_i + (1 - sigmoid(a_g)) tanh(a_c),  u_i = tanh(a_o)
// (page "03 · DSpark 建模：Markov 与 Confidence", section 3.7; z = [s; W1[x]; h], the h part in hpre).
template <typename TW>
__device__ void head_vectors(const SampleArgs& a, int step, const int* prev, float* hu, const float* hs_cur,
                             float* hs_next) {
    const int r = a.r, d = a.hd;
    const TW* W1 = reinterpret_cast<const TW*>(a.W1);
    const int m = a.head == DSPARK_HEAD_RNN ? 3 : 1;
    for (int idx = threadIdx.x; idx < a.B * r; idx += kThreads) {
        const int j = idx / r, i = idx % r;
        const TW* e = W1 + (size_t)prev[j] * r;
        const float* hp = a.hpre + ((size_t)j * a.gamma + step) * (size_t)(m * r);
        float u;
        if (a.head == DSPARK_HEAD_GATED) {
            const TW* wr = reinterpret_cast<const TW*>(a.Wg) + (size_t)i * (d + r) + d;
            float acc = hp[i];
            for (int c = 0; c < r; ++c) acc = fmaf(load_logit<TW>(wr, c), load_logit<TW>(e, c), acc);
            u = load_logit<TW>(e, i) / (1.f + expf(-acc));
        } else {
            const int w = 2 * r + d;
            const TW* wg = reinterpret_cast<const TW*>(a.Wg) + (size_t)i * w;
            const TW* wc = reinterpret_cast<const TW*>(a.Wc) + (size_t)i * w;
            const TW* wo = reinterpret_cast<const TW*>(a.Wo) + (size_t)i * w;
            const float* sj = hs_cur + (size_t)j * r;
            float ag = hp[i], ac = hp[r + i], ao = hp[2 * r + i];
            for (int c = 0; c < r; ++c) {
                const float sc = sj[c];
                ag = fmaf(load_logit<TW>(wg, c), sc, ag);
                ac = fmaf(load_logit<TW>(wc, c), sc, ac);
                ao = fmaf(load_logit<TW>(wo, c), sc, ao);
            }
            for (int c = 0; c < r; ++c) {
                const float ec = load_logit<TW>(e, c);
                ag = fmaf(load_logit<TW>(wg, r + c), ec, ag);
                ac = fmaf(load_logit<TW>(wc, r + c), ec, ac);
                ao = fmaf(load_logit<TW>(wo, r + c), ec, ao);
            }
            const float g = 1.f / (1.f + expf(-ag));
            hs_next[(size_t)j * r + i] = g * sj[i] + (1.f - g) * tanhf(ac);
            u = tanhf(ao);
        }
        hu[(size_t)j * r + i] = u;
        if (a.head_out && j % a.G == (int)blockIdx.x) a.head_out[((size_t)j * a.gamma + step) * r + i] = u;
    }
}

// The hidden-state parts of the head pre-activations, for every (request, position): one block
// per (j, i), a warp per output, the d products split over the lanes.
//   gated: out[i] = sum_c Wg[i][c] h_c;  rnn: out[t r + i] = sum_c Wt[i][2r + c] h_c (t = g, c, o).
template <typename TW>
__global__ void __launch_bounds__(256) head_hidden_kernel(int r, int d, int head, const TW* __restrict__ hidden,
                                                          const TW* __restrict__ Wg, const TW* __restrict__ Wc,
                                                          const TW* __restrict__ Wo, float* __restrict__ out) {
    const int row = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m = head == DSPARK_HEAD_RNN ? 3 : 1;
    const TW* h = hidden + (size_t)row * d;
    const int stride = head == DSPARK_HEAD_RNN ? 2 * r + d : d + r;
    const int off = head == DSPARK_HEAD_RNN ? 2 * r : 0;
    for (int t = warp; t < m * r; t += 8) {
        const TW* W = (t < r) ? Wg : (t < 2 * r ? Wc : Wo);
        const TW* wr = W + (size_t)(t % r) * stride + off;
        float acc = 0.f;
        for (int c = lane; c < d; c += 32) acc = fmaf(load_logit<TW>(wr, c), load_logit<TW>(h, c), acc);
        acc = warp_sum(acc);
        if (lane == 0) out[(size_t)row * (m * r) + t] = acc;
    }
}

// The step's in-chunk uniform of every request (SAMPLE_INCHUNK, draw 0), in .y; the chunk
// variates are drawn in the finalize.
__device__ void step_randoms(const SampleArgs& a, int step, float4* rnd) {
    const uint32_t i = (uint32_t)step + 1u;
    for (int j = threadIdx.x; j < a.B; j += kThreads)
        rnd[j] = make_float4(0.f, uniform(a.seed, (uint32_t)j, i, DSPARK_P_SAMPLE_INCHUNK, 0u), 0.f, 0.f);
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
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* xbuf = reinterpret_cast<float*>(smem_raw);                  // [kRows][kXRow]: z
    float2* cstat = reinterpret_cast<float2*>(xbuf + kRows * kXRow);   // [kRows][kChunks]
    RowBlock* rb = reinterpret_cast<RowBlock*>(cstat + kRows * kChunks);
    int* prev = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(rb) + align_up(sizeof(RowBlock), 16));
    float4* rnd = reinterpret_cast<float4*>(reinterpret_cast<unsigned char*>(prev) + align_up(sizeof(int) * (size_t)a.B, 16));
    unsigned char* wreg = reinterpret_cast<unsigned char*>(rnd + a.B);
    // after the W1-row staging of the CUDA-core path: the head vectors and the RNN state
    float* hu = reinterpret_cast<float*>(wreg + sizeof(float) * kRows * (size_t)a.r);
    float* hs = hu + (size_t)a.B * a.r;  // [2][B][r]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if constexpr (!kMMA) {
        if (a.head == DSPARK_HEAD_RNN)
            for (int idx = tid; idx < a.B * a.r; idx += kThreads) hs[idx] = 0.f;  // s_0 = 0
    }

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
    pa.softcap = a.softcap;
    pa.inv_softcap = a.inv_softcap;
    if constexpr (kMMA) {
        if (a.w2_smem) {
            stage_w2_tile<KS>(reinterpret_cast<const uint16_t*>(a.W2), blockIdx.x * kTS, a.V,
                              reinterpret_cast<uint4*>(wreg), kThreads);
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
        if constexpr (!kMMA) {
            if (a.head != DSPARK_HEAD_VANILLA) {
                float* s_cur = hs + (size_t)(step & 1) * a.B * a.r;
                float* s_nxt = hs + (size_t)((step + 1) & 1) * a.B * a.r;
                head_vectors<TW>(a, step, prev, hu, s_cur, s_nxt);
                __syncthreads();
            }
        }
        for (int tile = blockIdx.x; tile < a.nt; tile += a.G) {
            for (int row0 = 0; row0 < a.B; row0 += kRows) {
                if (tid < kRows) {
                    const int j = row0 + tid;
                    const bool ok = j < a.B;
                    rb->prev[tid] = ok ? prev[j] : 0;
                    rb->mode[tid] = ok ? ROW_SAMPLE : ROW_OFF;
                    rb->brow[tid] = ok ? ((long long)j * a.gamma + step) * (long long)a.V : -1;
                    rb->trow[tid] = -1;
                    const float4 q = ok && !a.greedy ? rnd[j] : make_float4(0.f, 0.f, 0.f, 0.f);
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
                        w1s[idx] = (rb->brow[q] >= 0)
                                       ? (a.head != DSPARK_HEAD_VANILLA ? hu[(size_t)(row0 + q) * a.r + k]
                                                                        : load_logit<TW>(W1, (size_t)rb->prev[q] * a.r + k))
                                       : 0.f;
                    }
                }
                __syncthreads();
                if constexpr (kMMA) {
                    const TL* base = reinterpret_cast<const TL*>(a.base);
                    const uint16_t* W1 = reinterpret_cast<const uint16_t*>(a.W1);
                    const uint16_t* W2 = reinterpret_cast<const uint16_t*>(a.W2);
                    const bool full = (tile + 1) * kTS <= a.V && a.vec_ok;
                    if (pa.w2s) {
                        if (full) produce_sample<TL, KS, GREEDY, true, true>(base, W1, W2, pa.w2s, a.V, true, tile, *rb, xbuf, cstat, a.scale2, a.softcap, a.inv_softcap);
                        else produce_sample<TL, KS, GREEDY, true, false>(base, W1, W2, pa.w2s, a.V, a.vec_ok, tile, *rb, xbuf, cstat, a.scale2, a.softcap, a.inv_softcap);
                    } else {
                        if (full) produce_sample<TL, KS, GREEDY, false, true>(base, W1, W2, nullptr, a.V, true, tile, *rb, xbuf, cstat, a.scale2, a.softcap, a.inv_softcap);
                        else produce_sample<TL, KS, GREEDY, false, false>(base, W1, W2, nullptr, a.V, a.vec_ok, tile, *rb, xbuf, cstat, a.scale2, a.softcap, a.inv_softcap);
                    }
                } else {
                    produce_chunks<TL, KS, TW, false>(pa, tile, *rb, xbuf, cstat);
                }
                __syncthreads();
                for (int rl = warp; rl < kRows; rl += kWarps) {
                    const int j = row0 + rl;
                    if (j >= a.B) continue;
                    const float4 rec = finalize_tile_cg(xbuf + rl * kXRow, cstat[rl * kChunks + lane], tile, a.V,
                                                        GREEDY, a.scale2, rb->u2[rl], a.seed, (uint32_t)j,
                                                        (uint32_t)step + 1u, DSPARK_P_SAMPLE_CHUNK);
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

using KernelFnS = void (*)(SampleArgs);
// ------------------------------------------------------------------------------------------
// Staged variant (bf16 logits, tensor-core bias, one tile per block).
//   - The base rows of each row block and the W1 rows of its previous tokens are copied into
//     shared memory by the bulk-copy engine one row block ahead (double buffer; the base rows of
//     a step's first row block are requested while the previous step finishes, its W1 rows as
//     soon as the tokens are known).  z is never stored: the finalize recomputes the one chunk
//     the draw selects with the producer's MMA sequence.
//   - Exchange: each tile's record is folded into one 64-bit word per request and step with an
//     atomic max (order-preserving key bits above the complemented candidate id: the highest
//     key wins, the lowest id on ties); after the grid-wide wait every block reads the B words.
//     The owner of request j (block j mod G) writes the token, and later, while it waits at
//     the next step's grid barrier, LSE(z/T) over the tiles' log-masses and z at the token
//     (records in three rotating buffers, so none is rewritten before its owner read it).
// ------------------------------------------------------------------------------------------
struct StagedLayout {
    size_t stage, w1s, crec, prev, urow, lnEt, bars, w2s, total;
    int lnE_rows;  // rows of the chunk-variate table: B (filled once per step) or 16 (per row block)
};

constexpr int kStepTableRows = 64;             // up to this many requests the per-step variate table is kept
constexpr int kHelperWarps = 4;                         // copy issuer, arriver, two exchangers
constexpr int kStagedThreads = kThreads + 32 * kHelperWarps;

__host__ __device__ inline StagedLayout staged_layout(int B, int r, bool w2_smem) {
    StagedLayout L;
    size_t o = 0;
    L.stage = o;
    o += sizeof(uint16_t) * 2 * kRows * kStageRow;
    L.w1s = o;
    o += 2 * sizeof(uint4) * (size_t)(2 * r);  // [2] x (r / 16 k-steps x 32 fragment units)
    L.crec = o;
    o += sizeof(float4) * 2 * kRows * kWarps;
    L.prev = o;
    o += align_up(sizeof(int) * 2 * (size_t)B, 16);
    L.lnE_rows = B <= kStepTableRows ? B : kRows;
    L.urow = o;
    o += align_up(sizeof(float) * (size_t)B, 16);
    L.lnEt = o;
    o += sizeof(float) * kChunks * (size_t)L.lnE_rows;
    L.bars = o;
    o += 64;  // full[2], empty[2], reduced barrier; flags: abort, ok, reduced count, bases issued, W1 rows done [2]
    L.w2s = o;
    if (w2_smem) o += (size_t)kTS * r * 2;
    L.total = o;
    return L;
}

// Base rows of row block `cnt` (step cnt / nrb) over this block's tile (one warp): one of the two
// arrivals of the buffer's full barrier, with the bytes; load_w1_rows() gives the other.
__device__ __forceinline__ void issue_base(const SampleArgs& a, int cnt, int nrb, uint16_t* dst, uint64_t* bar) {
    const int lane = threadIdx.x & 31;
    const int step = cnt / nrb, row0 = (cnt % nrb) * kRows;
    const int tile0 = blockIdx.x * kTS;
    const int nvalid = min(kTS, a.V - tile0);
    const int nrows = min(kRows, a.B - row0);
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(nrows * nvalid * 2));
    __syncwarp();
    if (lane < nrows) {
        const __nv_bfloat16* src =
            reinterpret_cast<const __nv_bfloat16*>(a.base) + ((size_t)(row0 + lane) * a.gamma + step) * (size_t)a.V + tile0;
        bulk_g2s_hint(dst + (size_t)lane * kStageRow, src, (uint32_t)(nvalid * 2), bar, l2_policy_evict_first());
    }
}

// W1 rows of the previous tokens of row block `cnt` (rows past B repeat its first row) into its
// stage buffer as interleaved A fragments (see w1_units), with plain loads by one warp: a batch
// of loads is in flight before its shared-memory stores.
template <int KS>
__device__ void load_w1_rows(const SampleArgs& a, int cnt, int nrb, const int* toks, uint4* w1s) {
    constexpr int r = 16 * KS, nunits = w1_units<KS>(), kBatch = 8;
    const int lane = threadIdx.x & 31;
    const uint2* W1 = reinterpret_cast<const uint2*>(a.W1);  // 4 bf16 per uint2
    const int row0 = (cnt % nrb) * kRows;
    uint4* dst = w1s + (size_t)(cnt & 1) * nunits;
    for (int b0 = 0; b0 < nunits; b0 += 32 * kBatch) {
        uint2 va[kBatch], vb[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int idx = b0 + k * 32 + lane;
            if (idx < nunits) {
                const int sk = idx >> 5, g = (idx >> 2) & 7, tq = idx & 3;
                const int k4 = (tq * (r / 4) + 4 * sk) / 4;  // uint2 index inside a row
                const int ja = row0 + g, jb = row0 + g + 8;
                va[k] = __ldg(W1 + (size_t)toks[ja < a.B ? ja : row0] * (r / 4) + k4);
                vb[k] = __ldg(W1 + (size_t)toks[jb < a.B ? jb : row0] * (r / 4) + k4);
            }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int idx = b0 + k * 32 + lane;
            if (idx < nunits) dst[idx] = make_uint4(va[k].x, vb[k].x, va[k].y, vb[k].y);
        }
    }
}

__device__ __forceinline__ void st_release_cta(volatile int* p, int v) {
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_addr((const void*)p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(volatile int* p) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr((const void*)p)) : "memory");
    return v;
}

// In-chunk uniforms of every request for `step` (SAMPLE_INCHUNK, draw 0).
__device__ void step_uniforms(const SampleArgs& a, int step, float* urow, int nthreads, int t0) {
    for (int j = t0; j < a.B; j += nthreads)
        urow[j] = uniform(a.seed, (uint32_t)j, (uint32_t)step + 1u, DSPARK_P_SAMPLE_INCHUNK, 0u);
}

// ln E_c of this block's 32 chunks for requests row0 .. row0 + nrows - 1 at `step`: one Philox
// call gives the four chunks 4q .. 4q + 3 (draws n = global chunk index).  The table is
// chunk-major, table[c * ld + row - row0], so the producer's reads of one chunk for eight rows
// fall on consecutive banks.
__device__ void chunk_variates(const SampleArgs& a, int step, int row0, int nrows, float* table, int ld,
                               int nthreads, int t0) {
    const uint32_t i = (uint32_t)step + 1u;
    for (int idx = t0; idx < nrows * (kChunks / 4); idx += nthreads) {
        const int rl = idx % nrows, q = idx / nrows;
        const uint32_t j = (uint32_t)(row0 + rl);
        const uint4 w = philox10(make_uint4(blockIdx.x * (kChunks / 4) + (uint32_t)q, i, j, DSPARK_P_SAMPLE_CHUNK),
                                 (uint32_t)a.seed, (uint32_t)(a.seed >> 32));
        table[(size_t)(4 * q + 0) * ld + rl] = log_neg_log_u(u01(w.x));
        table[(size_t)(4 * q + 1) * ld + rl] = log_neg_log_u(u01(w.y));
        table[(size_t)(4 * q + 2) * ld + rl] = log_neg_log_u(u01(w.z));
        table[(size_t)(4 * q + 3) * ld + rl] = log_neg_log_u(u01(w.w));
    }
}

// Helper warps of the staged kernel.  Waits are bounded (a.limit_ns without progress) and
// give up once the block's abort flag is raised; lane 0 decides, the warp follows.
__device__ __forceinline__ bool helper_should_stop(volatile int* abort, uint64_t t0, const SampleArgs& a) {
    int stop = 0;
    if ((threadIdx.x & 31) == 0) {
        if (*abort) {
            stop = 1;
        } else if (global_ns() - t0 > a.limit_ns) {
            record_status(&a.hdr->status, DSPARK_ERR_TIMEOUT);
            *abort = 1;
            stop = 1;
        }
    }
    return __shfl_sync(0xffffffffu, stop, 0) != 0;
}

// Copy issuer: the base rows of every row block as soon as its stage buffer is released (two row
// blocks ahead of the compute warps).
template <int KS>
__device__ void copy_issuer(const SampleArgs& a, uint16_t* stage, uint64_t* full, uint64_t* empty,
                            volatile int* abort, volatile int* nb_out) {
    const int lane = threadIdx.x & 31;
    const int nrb = (a.B + kRows - 1) / kRows, total = a.gamma * nrb;
    for (int nb = 0; nb < total; ++nb) {
        if (nb >= 2) {
            const uint64_t t0 = global_ns();
            bool ok = false;
            while (true) {
                int done = lane == 0 ? (int)mbar_try_wait(&empty[nb & 1], (uint32_t)(((nb - 2) >> 1) & 1)) : 0;
                if (__shfl_sync(0xffffffffu, done, 0)) {
                    ok = true;
                    break;
                }
                if (helper_should_stop(abort, t0, a)) break;
            }
            if (!ok) return;
        }
        issue_base(a, nb, nrb, stage + (size_t)(nb & 1) * kRows * kStageRow, &full[nb & 1]);
        if (lane == 0) *nb_out = nb + 1;
        __syncwarp();
    }
}

// Arriver: once the compute warps have issued a row block's maxima, one release-arrival on that
// row block's grid-wide counter (the release waits for the maxima to be performed in L2: that
// wait happens here, not in the compute warps).
__device__ void arriver(const SampleArgs& a, volatile int* reduced, uint64_t* redbar, volatile int* abort) {
    const int lane = threadIdx.x & 31;
    const int nrb = (a.B + kRows - 1) / kRows, total = a.gamma * nrb;
    for (int cnt = 0; cnt < total; ++cnt) {
        const uint64_t t0 = global_ns();
        bool ok = false;
        while (true) {
            // the count decides; the barrier (one phase per row block) only wakes this warp, so a
            // phase that went by unseen costs one suspended wait, never a wrong count
            int done = 0;
            if (lane == 0) {
                done = ld_acquire_cta(reduced) > cnt ? 1 : 0;
                if (!done) mbar_try_wait_hint(redbar, (uint32_t)(cnt & 1), 4000u);
            }
            if (__shfl_sync(0xffffffffu, done, 0)) {
                ok = true;
                break;
            }
            if (helper_should_stop(abort, t0, a)) break;
        }
        if (!ok) return;
        if (lane == 0)
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.rb_count + (size_t)(cnt % nrb) * kCountStride)
                         : "memory");
        __syncwarp();
    }
}

// Exchanger `par` (0 or 1) serves the row blocks whose index has that parity: for each of their
// row blocks of step st >= 1 it waits until every block has arrived for (st - 1, row block),
// turns the packed maxima into the tokens (the owner writes them out), then loads the W1 rows
// of those tokens into the row block's stage buffer and gives its second arrival.  After the
// last step it collects that step's tokens too.
// The LSE(z/T) and z at the token of step s for the requests of row block rbi this block owns
// (one warp; T > 0).  Runs once every block has arrived for (s, rbi): the records are complete.
__device__ void owner_lse_rb(const SampleArgs& a, int s, int rbi, const int* toks) {
    const int lane = threadIdx.x & 31;
    const float4* part = a.part + (size_t)(s % 3) * a.B * a.nt;
    const int row0 = rbi * kRows, row1 = min(a.B, row0 + kRows);
    int j = row0 + (((int)blockIdx.x - row0) % a.G + a.G) % a.G;  // first row >= row0 owned here
    for (; j < row1; j += a.G) {
        const float4* rec = part + (size_t)j * a.nt;
        float y[kMaxStagedTiles / 32];
        float m = -CUDART_INF_F;
#pragma unroll
        for (int i = 0; i < kMaxStagedTiles / 32; ++i) {
            const int t = lane + 32 * i;
            y[i] = t < a.nt ? __ldcg(&rec[t].y) : -CUDART_INF_F;
            m = fmaxf(m, y[i]);
        }
        m = warp_max(m);
        float lse = -CUDART_INF_F;
        if (m != -CUDART_INF_F) {
            const float m2 = m * kLog2e;
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < kMaxStagedTiles / 32; ++i) sum += ex2(fmaf(y[i], kLog2e, -m2));
            sum = warp_sum(sum);
            lse = (m2 + lg2(sum)) * kLn2;
        }
        if (lane == 0) {
            const size_t o = (size_t)j * a.gamma + s;
            a.draft_lse[o] = lse;
            a.zat[o] = __ldcg(&rec[toks[j] / kTS].w);
        }
    }
}

template <int KS>
__device__ void exchanger(const SampleArgs& a, int par, int* prev, uint4* w1s, uint64_t* full, uint64_t* empty,
                          volatile int* abort, volatile int* w1_upto) {
    const int lane = threadIdx.x & 31;
    const int nrb = (a.B + kRows - 1) / kRows, total = a.gamma * nrb;
    auto collect = [&](int rbi, int st) -> bool {  // tokens of step st - 1, row block rbi
        const uint64_t t0 = global_ns();
        const unsigned* cnt_p = a.rb_count + (size_t)rbi * kCountStride;
        while (true) {
            int st_ok = 0;
            if (lane == 0) {
                st_ok = ld_acquire_u32(cnt_p) >= (uint32_t)a.G * (uint32_t)st ? 1 : 0;
                if (!st_ok && ld_relaxed_s32(&a.hdr->status) == DSPARK_ERR_TIMEOUT) {
                    *abort = 1;
                    st_ok = -1;
                }
            }
            st_ok = __shfl_sync(0xffffffffu, st_ok, 0);
            if (st_ok > 0) break;
            __nanosleep(128);
            if (st_ok < 0 || helper_should_stop(abort, t0, a)) return false;
        }
        __syncwarp();
        const int row0 = rbi * kRows, nv = min(kRows, a.B - row0);
        const unsigned long long* slot = a.slots + (size_t)(st - 1) * a.B * kSlotStride;
        int* nxt = prev + (size_t)(st & 1) * a.B;
        if (lane < nv) {
            const int j = row0 + lane;
            const unsigned long long w = __ldcg(slot + (size_t)j * kSlotStride);
            const int cand = ~(int)(uint32_t)w;
            int p = cand;
            if (p < 0 || p >= a.V) {  // a row whose chunks all had no mass
                record_status(&a.hdr->status, DSPARK_ERR_TOKEN_RANGE);
                p = min(max(p, 0), a.V - 1);
            }
            nxt[j] = p;
            if (j % a.G == (int)blockIdx.x) {
                const size_t o = (size_t)j * a.gamma + (st - 1);
                a.tokens[o] = cand;
                if (a.greedy) {
                    a.draft_lse[o] = CUDART_NAN_F;
                    a.zat[o] = unpack_key(w);
                }
            }
        }
        __syncwarp();
        return true;
    };
    for (int cnt = 0; cnt < total; ++cnt) {
        const int rbi = cnt % nrb, st = cnt / nrb;
        if ((rbi & 1) != par) continue;
        if (st > 0 && !collect(rbi, st)) return;
        if (cnt >= 2) {  // the stage buffer's W1 rows were read by row block cnt - 2
            const uint64_t t0 = global_ns();
            bool ok = false;
            while (true) {
                int done = lane == 0 ? (int)mbar_try_wait(&empty[cnt & 1], (uint32_t)(((cnt - 2) >> 1) & 1)) : 0;
                if (__shfl_sync(0xffffffffu, done, 0)) {
                    ok = true;
                    break;
                }
                if (helper_should_stop(abort, t0, a)) break;
            }
            if (!ok) return;
        }
        load_w1_rows<KS>(a, cnt, nrb, prev + (size_t)(st & 1) * a.B, w1s);
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_local(&full[cnt & 1]);  // release: the W1 rows above are visible to its waiters
            *w1_upto = cnt + 1;
        }
        __syncwarp();
        if (!a.greedy && st > 0) owner_lse_rb(a, st - 1, rbi, prev + (size_t)(st & 1) * a.B);
    }
    for (int rbi = par; rbi < nrb; rbi += 2) {
        if (!collect(rbi, a.gamma)) return;
        if (!a.greedy) owner_lse_rb(a, a.gamma - 1, rbi, prev + (size_t)(a.gamma & 1) * a.B);
    }
}

template <int KS, bool GREEDY>
__global__ void __launch_bounds__(kStagedThreads, 1) sample_staged_kernel(SampleArgs a) {
    constexpr int r = 16 * KS;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const StagedLayout L = staged_layout(a.B, r, a.w2_smem);
    uint16_t* stage = reinterpret_cast<uint16_t*>(smem_raw + L.stage);  // [2][kRows][kStageRow] bf16 bits
    uint4* w1s = reinterpret_cast<uint4*>(smem_raw + L.w1s);            // [2][w1_units] A fragments
    float4* crec = reinterpret_cast<float4*>(smem_raw + L.crec);        // [2][kRows][kWarps] per-warp records
    int* prev = reinterpret_cast<int*>(smem_raw + L.prev);              // [2][B]: tokens feeding step s at s & 1
    float* urow = reinterpret_cast<float*>(smem_raw + L.urow);          // [B] in-chunk uniforms
    float* lnEt = reinterpret_cast<float*>(smem_raw + L.lnEt);          // [kChunks][lnE_rows]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + L.bars);    // [2] stage buffer filled (2 arrivals)
    uint64_t* empty = full + 2;                                         // [2] stage buffer released
    uint64_t* redbar = full + 4;                                        // a phase per row block reduced
    volatile int* flags = reinterpret_cast<volatile int*>(full + 5);
    volatile int* abort = flags + 0;
    volatile int* s_ok = flags + 1;
    volatile int* reduced = flags + 2;  // row blocks whose maxima the compute warps have issued
    volatile int* nb_issued = flags + 3;
    volatile int* w1_upto = flags + 4;  // [2]: per exchanger, row blocks whose W1 rows are in
    uint4* w2s = reinterpret_cast<uint4*>(smem_raw + L.w2s);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, tile0 = tile * kTS;
    const bool full_tile = tile0 + kTS <= a.V;
    const int nrb = (a.B + kRows - 1) / kRows, total = a.gamma * nrb;
    const bool step_table = L.lnE_rows == a.B;
    const uint16_t* W2 = reinterpret_cast<const uint16_t*>(a.W2);
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&full[b], 2);
            mbar_init(&empty[b], 1);
        }
        mbar_init(redbar, 1);
        for (int f = 0; f < 6; ++f) flags[f] = 0;
        mbar_init_fence();
    }
    for (int j = tid; j < a.B; j += kStagedThreads) {
        int p = a.anchor[j];
        if (p < 0 || p >= a.V) {
            record_status(&a.hdr->status, DSPARK_ERR_TOKEN_RANGE);
            p = min(max(p, 0), a.V - 1);
        }
        prev[j] = p;
    }
    __syncthreads();
    if (warp == kWarps) {
        copy_issuer<KS>(a, stage, full, empty, abort, nb_issued);
    } else if (warp == kWarps + 1) {
        arriver(a, reduced, redbar, abort);
    } else if (warp >= kWarps + 2) {
        exchanger<KS>(a, warp - kWarps - 2, prev, w1s, full, empty, abort, w1_upto + (warp - kWarps - 2));
    } else {
        if (a.w2_smem) stage_w2_tile_async<KS>(W2, tile0, a.V, w2s, kThreads);
        if (!GREEDY && step_table) {  // step 0's draws for every request
            step_uniforms(a, 0, urow, kThreads, tid);
            chunk_variates(a, 0, 0, a.B, lnEt, a.B, kThreads, tid);
        }
        if (a.w2_smem) cp_async_wait_all();
        named_barrier(1, kThreads);
        int cnt = 0;
        bool live = true;
        for (int step = 0; step < a.gamma && live; ++step) {
            float4* part = a.part + (size_t)(step % 3) * a.B * a.nt;
            unsigned long long* slot = a.slots + (size_t)step * a.B * kSlotStride;
            for (int rbi = 0; rbi < nrb; ++rbi, ++cnt) {
                const int buf = cnt & 1, row0 = rbi * kRows;
                const uint32_t par = (uint32_t)((cnt >> 1) & 1);
                const int nv = min(kRows, a.B - row0);
                if (!GREEDY && !step_table) {  // the row block's draws
                    if (rbi == 0) step_uniforms(a, step, urow, kThreads, tid);
                    chunk_variates(a, step, row0, nv, lnEt, kRows, kThreads, tid);
                }
                if (tid == 0) *s_ok = mbar_wait_or_abort(&full[buf], par, abort, &a.hdr->status, a.limit_ns, false);
                named_barrier(1, kThreads);
                if (!*s_ok) {
                    live = false;
                    break;
                }
                mbar_try_wait(&full[buf], par);  // completed: acquire for this thread
                const uint16_t* sbuf = stage + (size_t)buf * kRows * kStageRow;
                const uint4* wbuf = w1s + (size_t)buf * w1_units<KS>();
                float4* cr = crec + (size_t)buf * kRows * kWarps;
                const float* lt = lnEt + (step_table ? (size_t)row0 : 0);  // chunk-major, leading dimension ld
                const int ld = step_table ? a.B : kRows;
                const float* ut = urow + row0;
                if (a.w2_smem) {
                    if (full_tile) produce_cg<KS, GREEDY, true, true>(sbuf, wbuf, W2, w2s, a.V, tile, cr, a.scale2, lt, ld, ut, nv, a.softcap, a.inv_softcap);
                    else produce_cg<KS, GREEDY, true, false>(sbuf, wbuf, W2, w2s, a.V, tile, cr, a.scale2, lt, ld, ut, nv, a.softcap, a.inv_softcap);
                } else {
                    if (full_tile) produce_cg<KS, GREEDY, false, true>(sbuf, wbuf, W2, nullptr, a.V, tile, cr, a.scale2, lt, ld, ut, nv, a.softcap, a.inv_softcap);
                    else produce_cg<KS, GREEDY, false, false>(sbuf, wbuf, W2, nullptr, a.V, tile, cr, a.scale2, lt, ld, ut, nv, a.softcap, a.inv_softcap);
                }
                named_barrier(1, kThreads);
                if (tid == 0) mbar_arrive_local(&empty[buf]);  // stage and W1 buffer free for row block cnt + 2
                if (warp < nv) {  // one request per warp
                    const int j = row0 + warp;
                    const float4 rec = reduce_row_chunks(cr + warp * kWarps, GREEDY);
                    if (lane == 0) {
                        if (!GREEDY) part[(size_t)j * a.nt + tile] = rec;
                        red_max_u64(slot + (size_t)j * kSlotStride, pack_key(rec.x, __float_as_int(rec.z)));
                    }
                }
                named_barrier(1, kThreads);
                if (tid == 0) {  // the arriver publishes this row block
                    st_release_cta(reduced, cnt + 1);
                    mbar_arrive_local(redbar);
                }
            }
            if (!live) break;
            if (!GREEDY && step_table && step + 1 < a.gamma) {  // the next step's draws (this step's are read)
                step_uniforms(a, step + 1, urow, kThreads, tid);
                chunk_variates(a, step + 1, 0, a.B, lnEt, a.B, kThreads, tid);
                named_barrier(1, kThreads);
            }
        }
    }
    __syncthreads();
    if (tid == 0 && *abort) {  // the (at most two) newest row blocks' copies may still be in flight
        const int nb = *nb_issued;
        for (int c = max(0, nb - 2); c < nb; ++c) {
            const int ex = (c % nrb) & 1;
            if (w1_upto[ex] <= c) mbar_arrive_local(&full[c & 1]);  // its W1 arrival never came
            mbar_wait_bounded(&full[c & 1], (uint32_t)((c >> 1) & 1), &a.hdr->status, a.limit_ns);
        }
    }
    (void)total;
}

template <bool G>
KernelFnS pick_staged(int r) {
    switch (r) {
        case 16: return sample_staged_kernel<1, G>;
        case 32: return sample_staged_kernel<2, G>;
        case 64: return sample_staged_kernel<4, G>;
        case 128: return sample_staged_kernel<8, G>;
        case 256: return sample_staged_kernel<16, G>;
        default: return nullptr;
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
    if (!(p->softcap >= 0.f) || std::isinf(p->softcap)) return DSPARK_ERR_INVALID_ARG;
    if (p->logits_dtype != DSPARK_F32 && p->logits_dtype != DSPARK_BF16) return DSPARK_ERR_INVALID_ARG;
    if (p->r > 0 && p->w_dtype != DSPARK_F32 && p->w_dtype != DSPARK_BF16) return DSPARK_ERR_INVALID_ARG;
    if (p->B > 4096 || p->r > 1024 || p->gamma > 1024) return DSPARK_ERR_UNSUPPORTED;
    return DSPARK_OK;
}

size_t sample_slot_bytes(const dspark_sample_params* p) {  // maxima and per-row-block counters
    const size_t nrb = (size_t)(p->B + kRows - 1) / kRows;
    return align_up((size_t)kSlotStride * sizeof(unsigned long long) * (size_t)p->B * p->gamma, 256) +
           align_up((size_t)kCountStride * sizeof(unsigned) * nrb, 256);
}

size_t sample_workspace_bytes(const dspark_sample_params* p) {
    const size_t nt = (size_t)(p->V + kTS - 1) / kTS;
    return kHeaderBytes + sample_slot_bytes(p) + align_up(sizeof(int32_t) * (size_t)p->B, 256) +
           align_up(3 * sizeof(float4) * (size_t)p->B * nt, 256);
}

SampleWsLayout sample_ws_layout(const dspark_sample_params* p) {
    SampleWsLayout L;
    L.slots = kHeaderBytes;
    L.counts = kHeaderBytes + align_up((size_t)kSlotStride * sizeof(unsigned long long) * (size_t)p->B * p->gamma, 256);
    L.zeroed = kHeaderBytes + sample_slot_bytes(p);
    L.part = L.zeroed + align_up(sizeof(int32_t) * (size_t)p->B, 256);
    return L;
}

}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_sample_workspace_size(const dspark_sample_params* p) {
    if (validate_sample_params(p) != DSPARK_OK) return 0;
    return sample_workspace_bytes(p);
}

namespace {

// The launch shared by the vanilla and the head entry points (arguments already validated).
// head: null for the vanilla head; hpre: the head's precomputed hidden-state parts.
dspark_status sample_block_launch(const dspark_sample_params* p, const dspark_head* head, const float* hpre,
                                  float* head_vec, const void* base_logits, const void* W1, const void* W2,
                                  const int32_t* anchor, int32_t* tokens, float* draft_lse,
                                  float* draft_logit_at_tok, void* workspace, dspark_stream_t stream) {
    const int hk = head ? head->kind : DSPARK_HEAD_VANILLA;
    const bool mma = hk == DSPARK_HEAD_VANILLA && markov_use_mma(p);
    const int nt = (p->V + kTS - 1) / kTS;
    int sms = 0;
    if (device_sm_count(&sms) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (hk == DSPARK_HEAD_VANILLA && sample_tc_eligible(p, base_logits, W1, W2, sms))
        return launch_sample_tc(p, base_logits, W1, W2, anchor, tokens, draft_lse, draft_logit_at_tok,
                                sample_ws_layout(p), workspace, reinterpret_cast<cudaStream_t>(stream));
    const size_t esz = p->logits_dtype == DSPARK_BF16 ? 2 : 4;
    const bool vec_ok = ((uintptr_t)base_logits % 16 == 0) && (((size_t)p->V * esz) % 16 == 0);
    // staged path: bf16 logits, tensor-core bias, one tile per block (one block per SM)
    bool staged = mma && hk == DSPARK_HEAD_VANILLA && p->logits_dtype == DSPARK_BF16 && vec_ok && ((uintptr_t)W1 % 16 == 0) &&
                  ((uintptr_t)W2 % 16 == 0) && nt <= sms &&
                  nt <= kMaxStagedTiles;
    bool w2_staged = (size_t)kTS * p->r * 2 <= 128 * 1024;
    if (staged && staged_layout(p->B, p->r, w2_staged).total > kMaxSmem) w2_staged = false;
    if (staged && staged_layout(p->B, p->r, false).total > kMaxSmem) staged = false;
    KernelFn fn = staged ? (p->temperature == 0.f ? pick_staged<true>(p->r) : pick_staged<false>(p->r))
                         : pick_kernel(p, mma);
    bool w2_smem = mma && (size_t)kTS * p->r * 2 <= 128 * 1024 && nt <= sms;
    size_t smem = sample_smem_bytes(p->B, p->r, mma, w2_smem, hk);
    if (smem > kMaxSmem && w2_smem) {
        w2_smem = false;
        smem = sample_smem_bytes(p->B, p->r, mma, false, hk);
    }
    if (staged) {
        w2_smem = w2_staged;
        smem = staged_layout(p->B, p->r, w2_smem).total;
    }
    if (smem > kMaxSmem) return DSPARK_ERR_UNSUPPORTED;
    const int threads = staged ? kStagedThreads : kThreads;
    int per_sm = 0;
    if (prepare_kernel((const void*)fn, smem, threads, &per_sm) != cudaSuccess || per_sm < 1) return DSPARK_ERR_CUDA;
    const int G = std::min(nt, sms * per_sm);
    if (G < nt) w2_smem = false;  // a block owning several tiles cannot keep one tile's W2
    if (staged && G < nt) return DSPARK_ERR_CUDA;  // (cannot happen: nt <= SMs and one block per SM)

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
    const SampleWsLayout WL = sample_ws_layout(p);
    a.hdr = reinterpret_cast<WsHeader*>(ws);
    a.slots = reinterpret_cast<unsigned long long*>(ws + WL.slots);
    a.rb_count = reinterpret_cast<unsigned*>(ws + WL.counts);
    a.cur_tok = reinterpret_cast<int32_t*>(ws + WL.zeroed);
    a.part = reinterpret_cast<float4*>(ws + WL.part);
    a.limit_ns = wait_limit_ns();
    a.redundant = (size_t)p->B * nt <= 8192 && p->B <= kThreads;
    a.w2_smem = w2_smem;
    a.vec_ok = vec_ok;
    a.softcap = p->softcap;
    a.inv_softcap = p->softcap > 0.f ? 1.f / p->softcap : 0.f;
    a.head = hk;
    a.hd = head ? head->d : 0;
    a.hpre = hpre;
    a.Wg = head ? head->Wg : nullptr;
    a.Wc = head ? head->Wc : nullptr;
    a.Wo = head ? head->Wo : nullptr;
    a.head_out = head_vec;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, kHeaderBytes + (staged ? sample_slot_bytes(p) : 0), s) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    void* args[] = {&a};
    if (cudaLaunchCooperativeKernel((const void*)fn, dim3(G), dim3(threads), args, smem, s) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    note_launch();
    return DSPARK_OK;
}

dspark_status validate_head(const dspark_sample_params* p, const dspark_head* h) {
    if (!h || p->r < 1 || h->d < 1 || !h->hidden || !h->Wg) return DSPARK_ERR_INVALID_ARG;
    if (h->kind == DSPARK_HEAD_RNN) {
        if (!h->Wc || !h->Wo) return DSPARK_ERR_INVALID_ARG;
    } else if (h->kind != DSPARK_HEAD_GATED) {
        return DSPARK_ERR_INVALID_ARG;
    }
    if (h->d > (1 << 20)) return DSPARK_ERR_UNSUPPORTED;
    return DSPARK_OK;
}

size_t head_hpre_bytes(const dspark_sample_params* p, const dspark_head* h) {
    const size_t m = h->kind == DSPARK_HEAD_RNN ? 3 : 1;
    return align_up(sizeof(float) * (size_t)p->B * p->gamma * m * p->r, 256);
}

}  // namespace

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
    return sample_block_launch(p, nullptr, nullptr, nullptr, base_logits, W1, W2, anchor, tokens, draft_lse,
                               draft_logit_at_tok, workspace, stream);
}

extern "C" size_t dspark_sample_head_workspace_size(const dspark_sample_params* p, const dspark_head* head) {
    if (validate_sample_params(p) != DSPARK_OK || validate_head(p, head) != DSPARK_OK) return 0;
    return sample_workspace_bytes(p) + head_hpre_bytes(p, head);
}

extern "C" dspark_status dspark_markov_sample_block_head(const dspark_sample_params* p, const dspark_head* head,
                                                         const void* base_logits, const void* W1, const void* W2,
                                                         const int32_t* anchor, int32_t* tokens, float* draft_lse,
                                                         float* draft_logit_at_tok, float* head_vec, void* workspace,
                                                         size_t ws_bytes, dspark_stream_t stream) {
    dspark_status st = validate_sample_params(p);
    if (st != DSPARK_OK) return st;
    if ((st = validate_head(p, head)) != DSPARK_OK) return st;
    if (!base_logits || !anchor || !tokens || !draft_lse || !draft_logit_at_tok || !W1 || !W2)
        return DSPARK_ERR_INVALID_ARG;
    const size_t base_ws = sample_workspace_bytes(p);
    if (!workspace || ((uintptr_t)workspace & 255u) || ws_bytes < base_ws + head_hpre_bytes(p, head))
        return DSPARK_ERR_WORKSPACE;
    if (sample_smem_bytes(p->B, p->r, false, false, head->kind) > kMaxSmem) return DSPARK_ERR_UNSUPPORTED;
    float* hpre = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + base_ws);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const unsigned rows = (unsigned)((size_t)p->B * p->gamma);
    if (p->w_dtype == DSPARK_BF16) {
        head_hidden_kernel<__nv_bfloat16><<<rows, 256, 0, s>>>(
            p->r, head->d, head->kind, static_cast<const __nv_bfloat16*>(head->hidden),
            static_cast<const __nv_bfloat16*>(head->Wg), static_cast<const __nv_bfloat16*>(head->Wc),
            static_cast<const __nv_bfloat16*>(head->Wo), hpre);
    } else {
        head_hidden_kernel<float><<<rows, 256, 0, s>>>(p->r, head->d, head->kind,
                                                       static_cast<const float*>(head->hidden),
                                                       static_cast<const float*>(head->Wg),
                                                       static_cast<const float*>(head->Wc),
                                                       static_cast<const float*>(head->Wo), hpre);
    }
    if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
    note_launch();
    return sample_block_launch(p, head, hpre, head_vec, base_logits, W1, W2, anchor, tokens, draft_lse,
                               draft_logit_at_tok, workspace, stream);
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
