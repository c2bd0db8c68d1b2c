// sample_tc.cu -- Markov-head block sampling on the fifth-generation tensor cores (tcgen05), for
// batches of many requests with bf16 logits and weights of rank 64, 128 or 256.
//
// Method (P2 "从 DFlash 到 dLLM Self-Spec（三）" section 3.4, VanillaMarkov and the
// sample_block_tokens loop; P1 "03 · DSpark 建模：Markov 与 Confidence" section 3.7): for
// i = 1..gamma, z = base_i + W2 . W1[prev]; draw x_i from softmax(z / T) by the chunk-Gumbel
// contract of dspark.h; prev = x_i.
//
// One persistent cooperative kernel; CTA b owns vocabulary tile b (1024 ids) for all gamma steps.
// Requests go in row blocks of 128 (one TMEM lane each); a unit is one (step, row block).
//   - z of a unit, D[128 requests x 1024 ids], is computed entirely on the tensor cores, as eight
//     accumulators of 128 ids in fp32 TMEM columns (four rotating slots of 128 columns at rank 64;
//     three at ranks 128 and 256, where the A operand takes the remaining columns):
//       bias: D = W1[prev] . W2_rows^T, kind::f16 MMAs of M = 128, N = 128, K = 16 over the rank,
//             with A = the 128 W1 rows of the previous tokens (written by the exchange warps into
//             shared memory, swizzled, at rank 64, or into tensor memory at ranks 128 and 256) and
//             B = the accumulator's W2 rows (R / 64 swizzled K-chunks);
//       base: D += base . I, the accumulator's base logits (bf16, two 3-D copies of 64 ids x 128
//             requests) as the A operand and a 16 x 16 identity as B: four MMAs of N = 16, K = 16
//             per copy, each adding 16 ids' base values in fp32.
//     The operands of each accumulator (its W2 rows, re-read from L2 where W2 is kept with an
//     evict-last policy, and its base copies, evict-first) arrive by tiled tensor copies (128-byte
//     swizzle, the K-major MMA layout) in one stage of a ring, one accumulator per stage (rank 64:
//     four stages of 48 KB; rank 128: three of 64 KB; rank 256: two of 96 KB).  With the TMEM
//     accumulators the copies of the next units (they do not depend on the tokens) run ahead of
//     the epilogue.
//   - Epilogue: two warpgroups, one per parity of accumulator.  Thread = request: it reads its
//     lane's 32 columns of a chunk from TMEM (the next chunk's load in flight meanwhile) and forms
//     the chunk record of the contract with no shuffles: max, the weights 2^(z s - max), their
//     prefix sums in four blocks of eight, the in-chunk inverse-CDF candidate (the count of prefix
//     values not above u times the sum), and the key LSE_c - ln E_c (E_c from Philox: one call per
//     accumulator gives its four chunks).  Each warpgroup keeps the best key and the log-mass of
//     its half of the tile and, at the end of a unit, folds the key into the request's 64-bit word
//     with one atomic max (key bits above the complemented id: highest key, then lowest id, wins)
//     and stores the log-mass.
//   - An arriver warp then performs one release-add on the row block's arrival counter.  The
//     exchange warps of every CTA wait for all G arrivals of (step - 1, row block), read the
//     words (the token), write the W1 rows of the tokens as the next A operand, and the owner of
//     request j (CTA j mod G) writes the token, LSE(z/T) over the log-masses and z at the token.
// Every wait is bounded (DSPARK_ERR_TIMEOUT in the status word); on a timeout the kernel drains
// its copies and MMAs in flight, frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "host_util.h"
#include "tc05.cuh"

namespace dspark {
namespace {

constexpr int kTcTile = 1024;                 // ids per CTA (one vocabulary tile)
constexpr int kTcRows = 128;                  // requests per row block = MMA M = TMEM lanes
constexpr int kTcN = 128;                     // ids per accumulator = MMA N of the bias
constexpr int kTcAccs = kTcTile / kTcN;       // accumulators per unit
constexpr int kTcBox = 64;                    // ids per base copy (128 bytes: one swizzle span)
constexpr int kTcThreads = 512;
constexpr int kTcMaxTiles = 160;              // vocabulary tiles (CTAs) at most
constexpr int kTcEpiGroups = 2;               // epilogue warpgroups (one partial record each per tile and request)
constexpr int kTcSlotStride = 16;             // 64-bit words between two requests' maxima (one 128-byte line)
constexpr int kTcCountStride = 32;            // 32-bit words between two row blocks' arrival counters
constexpr uint32_t kIdBytes = 16 * 128;                    // 16 x 16 identity, rows of a 128-byte swizzled tile

// Layout for rank R.  Operands are split in K-chunks of 64 (128 bytes per row: one swizzle span).
// One ring stage holds everything one accumulator (128 ids) needs: its W2 rows as R / 64 tiles of
// 128 ids x one K-chunk (four MMAs of N = 128, K = 16 each) and its base logits as two copies of
// 64 ids x 128 requests (four identity MMAs of N = 16 each).  One wait and one release per
// accumulator keep the MMA thread's own instruction stream short: it shares its scheduler with
// the epilogue warps, so every instruction it issues costs it several cycles.
// Shared-memory offsets are from the 1024-byte aligned base.
template <int R>
struct TcCfg {
    static_assert(R == 64 || R == 128 || R == 256, "ranks of the tensor-core sampler");
    static constexpr int kKChunks = R / 64;
    static constexpr uint32_t kTileBytes = 16384;                // one tiled copy: 128 rows x 128 bytes
    static constexpr uint32_t kStageBytes = (kKChunks + 2) * kTileBytes;
    // A (the W1 rows) sits in shared memory at rank 64; at ranks 128 and 256 it sits in tensor memory
    // (written by the exchange threads, lane = request), which leaves shared memory to the ring, and
    // the accumulators keep three 128-column slots.
    static constexpr bool kATmem = R >= 128;
    static constexpr int kSlots = kATmem ? 3 : 4;                // accumulator slots of 128 TMEM columns
    static constexpr uint32_t kACol = kSlots * kTcN;              // first TMEM column of A (tensor-memory A)
    static constexpr uint32_t kACols = R / 2;                     // columns of one A operand (two bf16 each)
    static constexpr uint32_t kAChunkBytes = kTcRows * 128;      // one K-chunk of a shared-memory A: 16 KB
    static constexpr uint32_t kABytes = kATmem ? 0 : kAChunkBytes * kKChunks;
    static constexpr int kABufs = R == 256 ? 1 : 2;              // A operands in flight
    static_assert(!kATmem || kACol + kABufs * kACols <= 512, "tensor memory of the A operands");
    static constexpr int kStages = R == 64 ? 4 : (R == 128 ? 3 : 2);
    static constexpr uint32_t kSmRing = 0;                       // [kStages] {W2 K-chunks, base copy 0, 1}
    static constexpr uint32_t kSmA = kSmRing + kStages * kStageBytes;  // [kABufs] {A K-chunks}
    static constexpr uint32_t kSmId = kSmA + kABufs * kABytes;
    static constexpr uint32_t kSmBars = kSmId + kIdBytes;
    static constexpr int kNumBars = 2 * kABufs + 2 * kStages + 2 * kSlots + 2;
    static constexpr uint32_t kSmFlags = kSmBars + 8 * kNumBars;
    static constexpr size_t kSmemBytes = kSmFlags + 64;  // the dynamic base is 1024-byte aligned (checked at entry)
    static_assert(kSmA % 1024 == 0, "operand tiles are 1024-byte aligned");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory of the tensor-core sampler");
};

struct TcArgs {
    int B, gamma, V, nt, nrb, G;
    int part_ld;          // floats per request row of the log-mass records (kTcEpiGroups per tile)
    float scale2;         // log2(e) / T (1 when greedy)
    uint64_t seed;
    const uint16_t* base;  // bf16 bits [B, gamma, V]
    const uint16_t* W1;    // bf16 bits [V, R]
    const uint16_t* W2;    // bf16 bits [V, R]
    const int32_t* anchor;
    int32_t* tokens;
    float* draft_lse;
    float* zat;
    WsHeader* hdr;
    unsigned long long* slots;  // [gamma][B] packed maxima, kTcSlotStride words apart (zeroed per call)
    unsigned* rb_count;         // [nrb] arrival counters, kTcCountStride apart (zeroed per call)
    float* part;                // [3][B][part_ld] partial log-masses (natural log), one per tile and warpgroup
    uint64_t limit_ns;
};

__device__ __forceinline__ bool bar_red_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ int ld_acq_cta(const int* p) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}
__device__ __forceinline__ void add_rel_cta(int* p, int v) {
    asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

// One lane waits (bounded, abort-aware), the warp follows; every lane then takes its own acquire.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, const TcArgs& a) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_hint_or_abort(bar, parity, abort, &a.hdr->status, a.limit_ns) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait(bar, parity);
    return ok != 0;
}

// Running state of one request over the chunks of a half tile.
struct ChunkState {
    float bkey;  // best key so far (T > 0: LSE_c - ln E_c; greedy: max z)
    int bcand;   // its candidate id
    float mt, st;  // mass of the chunks seen = 2^mt * st; mt = the largest scaled chunk maximum so far
};

// Chunk record of one request over 32 ids in registers (T > 0), folded into the state.  Chunks
// arrive in increasing id order, so a strictly greater key is needed to replace the best (ties
// keep the lower chunk).  ids past V (MASK) are -inf.  The weights are taken relative to the
// running maximum mt (not the chunk's own), which folds the chunk into the mass with one
// exponential; a chunk more than 2^126 below the running maximum then has no weight, and it
// cannot win the race (its key is ~87 nats below the leader's, beyond any Gumbel variate).
// The inverse CDF runs on prefix sums in four blocks of eight ids, kept as two packed pairs of
// blocks (0, 1) and (2, 3).  No early exit and one warp vote: every lane of the warp runs this
// in step.
template <bool MASK>
__device__ __forceinline__ void chunk_sample(const uint32_t (&v)[32], int id0, int V, float scale2, float u, float lnE,
                                             ChunkState& cs) {
    float z[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) z[e] = (MASK && id0 + e >= V) ? -CUDART_INF_F : __uint_as_float(v[e]);
    const float nm = fmaxf(cs.mt, max32(z) * scale2);
    const float ref = nm == -CUDART_INF_F ? 0.f : nm;  // no ids at all: weights 2^-inf = 0, never NaN
    const uint64_t s2 = pk2(scale2, scale2), nr = pk2(-ref, -ref);
    uint64_t q[8], r[8];  // q[k] = ids (k, 8 + k), r[k] = ids (16 + k, 24 + k)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float2 x = up2(fma2(pk2(z[k], z[8 + k]), s2, nr));
        const float2 y = up2(fma2(pk2(z[16 + k], z[24 + k]), s2, nr));
        q[k] = pk2(ex2(x.x), ex2(x.y));
        r[k] = pk2(ex2(y.x), ex2(y.y));
    }
#pragma unroll
    for (int k = 1; k < 8; ++k) {  // inclusive prefix inside each block of eight
        q[k] = add2(q[k], q[k - 1]);
        r[k] = add2(r[k], r[k - 1]);
    }
    const float2 qe = up2(q[7]), re = up2(r[7]);
    const float o1 = qe.x, o2 = o1 + qe.y, o3 = o2 + re.x;
    const float S = o3 + re.y;
    const float t = u * S, t1 = t - o1, t2 = t - o2, t3 = t - o3;
    uint32_t neg = 0;  // minus the number of prefix values not above the target: the crossing index
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float2 a = up2(q[k]), b = up2(r[k]);
        neg += le_mask(a.x, t) + le_mask(a.y, t1) + le_mask(b.x, t2) + le_mask(b.y, t3);
    }
    int cnt = -(int)neg;
    if (__any_sync(0xffffffffu, cnt == 32)) {  // rounding left no crossing: the last id with weight
        if (cnt == 32) {
            int last = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float2 a = up2(q[k]), b = up2(r[k]);
                const float2 pa = k ? up2(q[k - 1]) : make_float2(0.f, 0.f);
                const float2 pb = k ? up2(r[k - 1]) : make_float2(0.f, 0.f);
                last = a.x > pa.x ? max(last, k) : last;
                last = a.y > pa.y ? max(last, 8 + k) : last;
                last = b.x > pb.x ? max(last, 16 + k) : last;
                last = b.y > pb.y ? max(last, 24 + k) : last;
            }
            cnt = last;
        }
    }
    if (S > 0.f) {
        const float key = (ref + lg2(S)) * kLn2 - lnE;
        if (key > cs.bkey) {
            cs.bkey = key;
            cs.bcand = id0 + cnt;
        }
    }
    cs.st = cs.st * ex2(cs.mt - ref) + S;  // (st = 0 while mt = -inf: 0 * 0)
    cs.mt = nm == -CUDART_INF_F ? cs.mt : nm;
}

// Greedy: the chunk's maximum and its lowest argmax.
template <bool MASK>
__device__ __forceinline__ void chunk_greedy(const uint32_t (&v)[32], int id0, int V, ChunkState& cs) {
    float z[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) z[e] = (MASK && id0 + e >= V) ? -CUDART_INF_F : __uint_as_float(v[e]);
    const float m = max32(z);
    int x = 31;
#pragma unroll
    for (int e = 31; e >= 0; --e) x = z[e] == m ? e : x;
    if (m > cs.bkey) {
        cs.bkey = m;
        cs.bcand = id0 + x;
    }
}

// The four chunks of one accumulator for this thread's request: TMEM loads double-buffered, the
// next chunk's in flight while the current one is reduced.  With ROLL the loop runs over pairs of
// chunks and is not unrolled: two copies of the chunk code rather than four.  That keeps the
// larger kernels of ranks 128 and 256 in the instruction cache (b128_r256: 0.33 ms against 0.38 ms);
// at rank 64 the unrolled loop is faster (0.65 ms against 0.76 ms at b512).
template <bool GREEDY, bool MASK, bool ROLL>
__device__ __forceinline__ void accumulator_chunks(uint32_t taddr, int id0, int V, float scale2, float u,
                                                   const float (&lnE)[4], ChunkState& cs) {
    uint32_t va[32], vb[32];
    tmem_ld32(taddr, va);
    tmem_wait_ld(va);
    if constexpr (ROLL) {
#pragma unroll 1
        for (int p = 0; p < 2; ++p) {
            const int c0 = 2 * p, c1 = c0 + 1;
            tmem_ld32(taddr + 32u * (uint32_t)c1, vb);  // chunk c1 in flight while c0 is reduced
            if (!MASK || id0 + 32 * c0 < V) {           // (uniform) a chunk wholly past V has no ids
                if (GREEDY) chunk_greedy<MASK>(va, id0 + 32 * c0, V, cs);
                else chunk_sample<MASK>(va, id0 + 32 * c0, V, scale2, u, p ? lnE[2] : lnE[0], cs);
            }
            tmem_wait_ld(vb);
            if (p == 0) tmem_ld32(taddr + 32u * (uint32_t)(c1 + 1), va);  // chunk 2 in flight while 1 is reduced
            if (!MASK || id0 + 32 * c1 < V) {
                if (GREEDY) chunk_greedy<MASK>(vb, id0 + 32 * c1, V, cs);
                else chunk_sample<MASK>(vb, id0 + 32 * c1, V, scale2, u, p ? lnE[3] : lnE[1], cs);
            }
            if (p == 0) tmem_wait_ld(va);
        }
    } else {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t(&cur)[32] = (cc & 1) ? vb : va;
            uint32_t(&nxt)[32] = (cc & 1) ? va : vb;
            if (cc < 3) tmem_ld32(taddr + 32u * (uint32_t)(cc + 1), nxt);
            if (!MASK || id0 + 32 * cc < V) {  // (uniform) a chunk wholly past V has no ids
                if (GREEDY) chunk_greedy<MASK>(cur, id0 + 32 * cc, V, cs);
                else chunk_sample<MASK>(cur, id0 + 32 * cc, V, scale2, u, lnE[cc], cs);
            }
            if (cc < 3) tmem_wait_ld(nxt);
        }
    }
}

// ln E_c of four consecutive chunks 4q .. 4q + 3 (one Philox call, draws n = global chunk index).
__device__ __forceinline__ void chunk_variates4(uint64_t seed, uint32_t j, uint32_t i, uint32_t q, float (&lnE)[4],
                                                uint32_t purpose = DSPARK_P_SAMPLE_CHUNK) {
    const uint4 w = philox10(make_uint4(q, i, j, purpose), (uint32_t)seed, (uint32_t)(seed >> 32));
    lnE[0] = log_neg_log_u_2(u01(w.x));
    lnE[1] = log_neg_log_u_2(u01(w.y));
    lnE[2] = log_neg_log_u_2(u01(w.z));
    lnE[3] = log_neg_log_u_2(u01(w.w));
}

template <int R, bool GREEDY>
__global__ void __launch_bounds__(kTcThreads, 1)
    sample_tc_kernel(const __grid_constant__ CUtensorMap tm_base, const __grid_constant__ CUtensorMap tm_w2,
                     const TcArgs a) {
    using C = TcCfg<R>;
    constexpr int kStages = C::kStages, kABufs = C::kABufs;
    constexpr uint32_t kSmRing = C::kSmRing, kSmA = C::kSmA, kSmId = C::kSmId, kSmBars = C::kSmBars,
                       kSmFlags = C::kSmFlags, kStageBytes = C::kStageBytes, kABytes = C::kABytes;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    if (smem_addr(smem_raw) & 1023u) {  // the swizzled tiles need 1024-byte alignment (uniform exit)
        if (threadIdx.x == 0) record_status(&a.hdr->status, DSPARK_ERR_UNSUPPORTED);
        return;
    }
    unsigned char* sm = smem_raw;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kSmBars);
    uint64_t* a_full = bars;                           // [kABufs]
    uint64_t* a_empty = bars + kABufs;                 // [kABufs]
    uint64_t* b_full = bars + 2 * kABufs;              // [kStages]
    uint64_t* b_empty = b_full + kStages;              // [kStages]
    constexpr int kSlots = C::kSlots;
    uint64_t* t_full = b_empty + kStages;              // [kSlots]
    uint64_t* t_empty = t_full + kSlots;               // [kSlots]
    uint64_t* done_bar = t_empty + kSlots;
    uint64_t* drain_bar = done_bar + 1;
    int* flags = reinterpret_cast<int*>(sm + kSmFlags);
    volatile int* abort = flags;
    int* wg_done = flags + 1;          // warpgroup-units finished (two per unit)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(flags + 2);
    volatile int* nb_issued = flags + 3;
    volatile int* n_mma = flags + 4;   // MMAs issued (drained before the tensor memory is freed)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, tile0 = tile * kTcTile;
    const int total = a.gamma * a.nrb;

    if (tid == 0) {
        for (int b = 0; b < kABufs; ++b) {
            mbar_init(&a_full[b], 4);
            mbar_init(&a_empty[b], 1);
        }
        for (int b = 0; b < kStages; ++b) {
            mbar_init(&b_full[b], 1);
            mbar_init(&b_empty[b], 1);
        }
        for (int b = 0; b < kSlots; ++b) {
            mbar_init(&t_full[b], 1);
            mbar_init(&t_empty[b], 4);
        }
        mbar_init(done_bar, 1);
        mbar_init(drain_bar, 1);
        for (int f = 0; f < 16; ++f) flags[f] = 0;
        mbar_init_fence();
    }
    if (tid < 128) {  // the identity B operand: row n holds 1.0 at k = n (units 0 and 1 of its row)
        const int n = tid >> 3, u = tid & 7;
        const int k = n & 7;  // bf16 1.0 = 0x3F80 at element k of unit n / 8
        const uint32_t one = (u < 2 && (n >> 3) == u) ? ((k & 1) ? 0x3F800000u : 0x00003F80u) : 0u;
        const int wd = k >> 1;
        *reinterpret_cast<uint4*>(sm + kSmId + sw128_offset(n, u)) =
            make_uint4(wd == 0 ? one : 0u, wd == 1 ? one : 0u, wd == 2 ? one : 0u, wd == 3 ? one : 0u);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------------- tensor copies
        if (lane == 0) {
            tma_prefetch_desc(&tm_base);
            tma_prefetch_desc(&tm_w2);
            const uint64_t keep = l2_policy_evict_last(), stream = l2_policy_evict_first();
            const int nstage = total * kTcAccs;
            for (int gs = 0; gs < nstage; ++gs) {  // one stage per accumulator: its W2 rows and base copies
                const int st = gs % kStages, use = gs / kStages;
                if (use > 0 && !mbar_wait_hint_or_abort(&b_empty[st], (uint32_t)((use - 1) & 1), abort,
                                                        &a.hdr->status, a.limit_ns))
                    break;
                const int u = gs / kTcAccs, acc = gs % kTcAccs;
                const int s = u / a.nrb, rb = u % a.nrb;
                const int id0 = tile0 + kTcN * acc;
                unsigned char* dst = sm + kSmRing + st * kStageBytes;
                mbar_arrive_expect_tx(&b_full[st], kStageBytes);
#pragma unroll
                for (int kc = 0; kc < C::kKChunks; ++kc)  // W2 stays in L2
                    tma_load_2d(dst + kc * C::kTileBytes, &tm_w2, 64 * kc, id0, &b_full[st], keep);
#pragma unroll
                for (int bx = 0; bx < 2; ++bx)
                    tma_load_3d(dst + (C::kKChunks + bx) * C::kTileBytes, &tm_base, id0 + kTcBox * bx, s, rb * kTcRows,
                                &b_full[st], stream);
                *nb_issued = gs + 1;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc_bias = umma_idesc_bf16(kTcRows, kTcN);
            constexpr uint32_t idesc_base = umma_idesc_bf16(kTcRows, 16);
            // descriptors advance by address / 16 in their low bits: 1024 per 16 KB stage, 2 per K-step
            const uint64_t id_desc = umma_desc_sw128(smem_addr(sm + kSmId), 1024);
            const uint64_t ring_desc = umma_desc_sw128(smem_addr(sm + kSmRing), 1024);
            const uint64_t a_desc = umma_desc_sw128(smem_addr(sm + kSmA), 1024);
            bool ok = true;
            for (int u = 0; u < total && ok; ++u) {
                const int ab = u % kABufs;
                if (!mbar_wait_hint_or_abort(&a_full[ab], (uint32_t)((u / kABufs) & 1), abort, &a.hdr->status,
                                             a.limit_ns))
                    break;
                for (int acc = 0; acc < kTcAccs && ok; ++acc) {
                    const int ga = u * kTcAccs + acc, sl = ga % kSlots, use = ga / kSlots;
                    if (use > 0 && !mbar_wait_hint_or_abort(&t_empty[sl], (uint32_t)((use - 1) & 1), abort,
                                                            &a.hdr->status, a.limit_ns)) {
                        ok = false;
                        break;
                    }
                    const int st = ga % kStages;
                    if (!mbar_wait_hint_or_abort(&b_full[st], (uint32_t)((ga / kStages) & 1), abort, &a.hdr->status,
                                                 a.limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)(sl * kTcN);
                    const uint64_t sd = ring_desc + (uint64_t)(st * (int)(kStageBytes >> 4));
#pragma unroll
                    for (int kc = 0; kc < C::kKChunks; ++kc)
#pragma unroll
                        for (int k = 0; k < 4; ++k) {  // D = W1[prev] . W2_rows^T
                            const uint64_t bd = sd + (uint64_t)(kc * (int)(C::kTileBytes >> 4) + 2 * k);
                            if constexpr (C::kATmem)
                                umma_bf16_ts(d, tmem + C::kACol + (uint32_t)ab * C::kACols + 32u * kc + 8u * k, bd,
                                             idesc_bias, (kc | k) > 0 ? 1u : 0u);
                            else
                                umma_bf16(d,
                                          a_desc + (uint64_t)(ab * (int)(C::kABytes >> 4) +
                                                              kc * (int)(C::kAChunkBytes >> 4) + 2 * k),
                                          bd, idesc_bias, (kc | k) > 0 ? 1u : 0u);
                        }
                    *n_mma = 1;
#pragma unroll
                    for (int bx = 0; bx < 2; ++bx)
#pragma unroll
                        for (int i = 0; i < kTcBox / 16; ++i)  // D[:, 64 bx + 16 i ..] += base[:, 16 i ..] . I
                            umma_bf16(d + (uint32_t)(kTcBox * bx + 16 * i),
                                      sd + (uint64_t)((C::kKChunks + bx) * (int)(C::kTileBytes >> 4) + 2 * i), id_desc,
                                      idesc_base, 1u);
                    umma_commit(&b_empty[st]);  // the stage is free once these have read it
                    umma_commit(&t_full[sl]);
                }
                if (ok) umma_commit(&a_empty[ab]);
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ---------------------------------------------------------------- arriver
        if (lane == 0) {
            for (int u = 0; u < total; ++u) {
                const uint64_t t0 = global_ns();
                bool ok = true;
                int c;
                while ((c = ld_acq_cta(wg_done)) < kTcEpiGroups * (u + 1)) {
                    // one arrival per finished warpgroup-unit, so phase c completes at the next one;
                    // the count decides, the barrier only wakes this thread
                    mbar_try_wait_hint(done_bar, (uint32_t)(c & 1), 20000u);
                    if (*abort) {
                        ok = false;
                        break;
                    }
                    if (global_ns() - t0 > a.limit_ns) {
                        record_status(&a.hdr->status, DSPARK_ERR_TIMEOUT);
                        *abort = 1;
                        ok = false;
                        break;
                    }
                }
                if (!ok) break;
                asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.rb_count + (size_t)(u % a.nrb) *
                                                                                             kTcCountStride)
                             : "memory");
            }
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // ---------------------------------------------------------------- exchange
        const int row = tid - 128;
        bool live = true;
        auto collect = [&](int s, int rb, int& tok) -> bool {  // the token drawn at step s - 1 (s >= 1)
            int ok = 1;
            if (row == 0) {
                const unsigned* cp = a.rb_count + (size_t)rb * kTcCountStride;
                const uint64_t t0 = global_ns();
                while (ld_acquire_u32(cp) < (uint32_t)a.G * (uint32_t)s) {
                    if (*abort || ld_relaxed_s32(&a.hdr->status) == DSPARK_ERR_TIMEOUT) {
                        *abort = 1;
                        ok = 0;
                        break;
                    }
                    if (global_ns() - t0 > a.limit_ns) {
                        record_status(&a.hdr->status, DSPARK_ERR_TIMEOUT);
                        *abort = 1;
                        ok = 0;
                        break;
                    }
                    __nanosleep(64);
                }
            }
            if (bar_red_or(3, 128, ok == 0)) return false;
            const int j = rb * kTcRows + row;
            tok = 0;
            if (j < a.B) {
                const unsigned long long w = __ldcg(a.slots + ((size_t)(s - 1) * a.B + j) * kTcSlotStride);
                const int cand = ~(int)(uint32_t)w;
                tok = cand;
                if (tok < 0 || tok >= a.V) {  // a request whose chunks all had no mass
                    record_status(&a.hdr->status, DSPARK_ERR_TOKEN_RANGE);
                    tok = min(max(tok, 0), a.V - 1);
                }
                if (j % a.G == (int)blockIdx.x) {
                    const size_t o = (size_t)j * a.gamma + (s - 1);
                    a.tokens[o] = cand;
                    if (GREEDY) {
                        a.draft_lse[o] = CUDART_NAN_F;
                        a.zat[o] = unpack_key(w);
                    }
                }
            }
            return true;
        };
        // LSE(z/T) over the half-tile log-masses and z at the token of the rows this CTA owns
        // (T > 0), a warp per owned row: one load of all records, warp reductions, and the
        // 64-term dot product of z at the token split over the lanes.
        auto owner_stats = [&](int s, int rb, int tok) {
            if (GREEDY) return;
            const int j = rb * kTcRows + row;
            unsigned own = __ballot_sync(0xffffffffu, j < a.B && j % a.G == (int)blockIdx.x);
            const int n = kTcEpiGroups * a.nt;
            while (own) {
                const int src = __ffs(own) - 1;
                own &= own - 1;
                const int jj = j - lane + src;
                const int tk = __shfl_sync(0xffffffffu, tok, src);
                const float* rec = a.part + ((size_t)(s % 3) * a.B + jj) * a.part_ld;
                float y[kTcMaxTiles * kTcEpiGroups / 32];
                float m = -CUDART_INF_F;
#pragma unroll
                for (int q = 0; q < kTcMaxTiles * kTcEpiGroups / 32; ++q) {
                    const int idx = lane + 32 * q;
                    y[q] = idx < n ? __ldcg(rec + idx) * kLog2e : -CUDART_INF_F;
                    m = fmaxf(m, y[q]);
                }
                m = warp_max(m);
                float sum = 0.f;
                if (m != -CUDART_INF_F) {
#pragma unroll
                    for (int q = 0; q < kTcMaxTiles * kTcEpiGroups / 32; ++q) sum += ex2(y[q] - m);
                }
                sum = warp_sum(sum);
                // z at the token: base + W2[tok] . W1[prev], prev = the token before step s
                const size_t o = (size_t)jj * a.gamma + s;
                int prev = s == 0 ? a.anchor[jj] : a.tokens[o - 1];
                prev = min(max(prev, 0), a.V - 1);
                const uint32_t* w1r = reinterpret_cast<const uint32_t*>(a.W1 + (size_t)prev * R);
                const uint32_t* w2r = reinterpret_cast<const uint32_t*>(a.W2 + (size_t)tk * R);
                float bias = 0.f;
#pragma unroll
                for (int q = 0; q < R / 64; ++q) {
                    const uint32_t w1 = __ldg(w1r + lane + 32 * q), w2 = __ldg(w2r + lane + 32 * q);
                    bias = fmaf(bf16_lo(w1), bf16_lo(w2), fmaf(bf16_hi(w1), bf16_hi(w2), bias));
                }
                bias = warp_sum(bias);
                if (lane == 0) {
                    a.draft_lse[o] = m == -CUDART_INF_F ? -CUDART_INF_F : (m + lg2(sum)) * kLn2;
                    a.zat[o] = bf16_bits_to_f32(__ldg(a.base + o * (size_t)a.V + tk)) + bias;
                }
            }
        };
        for (int u = 0; u < total && live; ++u) {
            const int s = u / a.nrb, rb = u % a.nrb;
            const int j = rb * kTcRows + row;
            int tok = 0;
            if (s == 0) {
                if (j < a.B) {
                    tok = a.anchor[j];
                    if (tok < 0 || tok >= a.V) {
                        record_status(&a.hdr->status, DSPARK_ERR_TOKEN_RANGE);
                        tok = min(max(tok, 0), a.V - 1);
                    }
                }
            } else if (!collect(s, rb, tok)) {
                live = false;
                break;
            }
            // the W1 row (R / 8 units of 16 bytes) in batches of at most 16 units; the first batch is
            // loaded before the A buffer is free
            constexpr int kQ = R / 8, kQB = kQ < 16 ? kQ : 16;
            const uint4* src = reinterpret_cast<const uint4*>(a.W1 + (size_t)tok * R);
            uint4 w[kQB];
#pragma unroll
            for (int q = 0; q < kQB; ++q) w[q] = j < a.B ? __ldg(src + q) : make_uint4(0u, 0u, 0u, 0u);
            // the A buffer was last read by the MMAs of unit u - kABufs
            if (u >= kABufs && !warp_wait(&a_empty[u % kABufs], (uint32_t)(((u / kABufs) - 1) & 1), abort, a))
                live = false;
            if (live && C::kATmem) {  // this thread's TMEM lane, 8 columns per unit of 16 bytes
                tc_fence_after();
                const uint32_t ta = tmem + ((uint32_t)(row & ~31) << 16) + C::kACol + (uint32_t)(u % kABufs) * C::kACols;
#pragma unroll
                for (int b0 = 0; b0 < kQ; b0 += kQB) {
                    if (b0 > 0) {
#pragma unroll
                        for (int q = 0; q < kQB; ++q)
                            w[q] = j < a.B ? __ldg(src + b0 + q) : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                    for (int h8 = 0; h8 < kQB / 8; ++h8) {  // 32 columns at a time
                        uint32_t v[32];
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            v[4 * q] = w[8 * h8 + q].x;
                            v[4 * q + 1] = w[8 * h8 + q].y;
                            v[4 * q + 2] = w[8 * h8 + q].z;
                            v[4 * q + 3] = w[8 * h8 + q].w;
                        }
                        tmem_st32(ta + 4u * (uint32_t)(b0 + 8 * h8), v);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_local(&a_full[u % kABufs]);
            } else if (live) {
                unsigned char* ad = sm + kSmA + (u % kABufs) * kABytes;
#pragma unroll
                for (int b0 = 0; b0 < kQ; b0 += kQB) {
                    if (b0 > 0) {
#pragma unroll
                        for (int q = 0; q < kQB; ++q)
                            w[q] = j < a.B ? __ldg(src + b0 + q) : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                    for (int q = 0; q < kQB; ++q) {  // unit q of the row: K-chunk q / 8, unit q % 8 of it
                        const int qq = b0 + q;
                        *reinterpret_cast<uint4*>(ad + (qq >> 3) * C::kAChunkBytes + sw128_offset(row, qq & 7)) = w[q];
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive_local(&a_full[u % kABufs]);
            }
            if (bar_red_or(3, 128, !live)) break;
            if (s > 0) owner_stats(s - 1, rb, tok);
        }
        // the last step's tokens
        for (int rb = 0; rb < a.nrb && live; ++rb) {
            int tok = 0;
            if (!collect(a.gamma, rb, tok)) break;
            owner_stats(a.gamma - 1, rb, tok);
        }
    } else if (warp >= 8) {
        // ---------------------------------------------------------------- epilogue
        const int h = (warp - 8) >> 2;                 // accumulators of parity h
        const int row = (warp & 3) * 32 + lane;        // TMEM lane = request within the row block
        const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const bool full_tile = tile0 + kTcTile <= a.V;
        bool live = true;
        for (int u = 0; u < total && live; ++u) {
            const int s = u / a.nrb, rb = u % a.nrb;
            const int j = rb * kTcRows + row;
            const bool valid = j < a.B;
            const uint32_t i = (uint32_t)s + 1u;
            const float uin = (!GREEDY && valid) ? uniform(a.seed, (uint32_t)j, i, DSPARK_P_SAMPLE_INCHUNK, 0u) : 0.f;
            ChunkState cs{-CUDART_INF_F, -1, -CUDART_INF_F, 0.f};
            bool ok = true;
            for (int ah = 0; ah < kTcAccs / 2; ++ah) {
                const int acc = 2 * ah + h;
                const int ga = u * kTcAccs + acc, sl = ga % kSlots;
                float lnE[4] = {0.f, 0.f, 0.f, 0.f};
                if (!GREEDY) chunk_variates4(a.seed, (uint32_t)j, i, (uint32_t)(tile * (kTcTile / 128) + acc), lnE);
                if (!warp_wait(&t_full[sl], (uint32_t)((ga / kSlots) & 1), abort, a)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tl + (uint32_t)(sl * kTcN);
                const int id0 = tile0 + kTcN * acc;
                if (full_tile) accumulator_chunks<GREEDY, false, (R >= 128)>(taddr, id0, a.V, a.scale2, uin, lnE, cs);
                else accumulator_chunks<GREEDY, true, (R >= 128)>(taddr, id0, a.V, a.scale2, uin, lnE, cs);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_local(&t_empty[sl]);
            }
            if (ok && valid) {
                if (!GREEDY) a.part[((size_t)(s % 3) * a.B + j) * a.part_ld + kTcEpiGroups * tile + h] =
                    (cs.mt == -CUDART_INF_F) ? -CUDART_INF_F : (cs.mt + lg2(cs.st)) * kLn2;
                red_max_u64(a.slots + ((size_t)s * a.B + j) * kTcSlotStride, pack_key(cs.bkey, cs.bcand));
            }
            if (bar_red_or(1 + h, 128, !ok)) {
                live = false;
                break;
            }
            if (row == 0) {  // this warpgroup's maxima are issued: the arriver publishes the unit
                add_rel_cta(wg_done, 1);
                mbar_arrive_local(done_bar);
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *abort) {  // copies in flight land before the shared memory goes away
        const int nb = *nb_issued;
        for (int g = max(0, nb - kStages); g < nb; ++g)
            mbar_wait_bounded(&b_full[g % kStages], (uint32_t)((g / kStages) & 1), &a.hdr->status, a.limit_ns);
    }
    if (warp == 1) {
        if (lane == 0 && *n_mma) {  // every MMA issued has completed
            umma_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, &a.hdr->status, a.limit_ns);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

bool sample_tc_eligible(const dspark_sample_params* p, const void* base, const void* W1, const void* W2, int sms) {
    const int nt = (p->V + kTcTile - 1) / kTcTile;
    // (the base logits are added on the tensor cores: a softcap of them needs the other samplers)
    return p->logits_dtype == DSPARK_BF16 && p->w_dtype == DSPARK_BF16 &&
           (p->r == 64 || p->r == 128 || p->r == 256) && p->B >= kTcMinBatch &&
           p->softcap == 0.f &&
           p->V % 8 == 0 && ((uintptr_t)base % 16) == 0 && ((uintptr_t)W1 % 16) == 0 && ((uintptr_t)W2 % 16) == 0 &&
           nt <= sms && nt <= kTcMaxTiles && tensor_map_encoder() != nullptr;
}

dspark_status launch_sample_tc(const dspark_sample_params* p, const void* base_logits, const void* W1, const void* W2,
                               const int32_t* anchor, int32_t* tokens, float* draft_lse, float* draft_logit_at_tok,
                               const SampleWsLayout& L, void* workspace, cudaStream_t s) {
    auto enc = tensor_map_encoder();
    if (!enc) return DSPARK_ERR_UNSUPPORTED;
    const int nt = (p->V + kTcTile - 1) / kTcTile;
    CUtensorMap m_base, m_w2;
    {
        cuuint64_t dims[3] = {(cuuint64_t)p->V, (cuuint64_t)p->gamma, (cuuint64_t)p->B};
        cuuint64_t strides[2] = {(cuuint64_t)p->V * 2, (cuuint64_t)p->gamma * p->V * 2};
        cuuint32_t box[3] = {kTcBox, 1, kTcRows};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(&m_base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base_logits), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DSPARK_ERR_UNSUPPORTED;
    }
    {
        // W2 [V, r]: boxes of one K-chunk (64) x the 128 ids of an accumulator
        cuuint64_t dims[2] = {(cuuint64_t)p->r, (cuuint64_t)p->V};
        cuuint64_t strides[1] = {(cuuint64_t)p->r * 2};
        cuuint32_t box[2] = {64, kTcN};
        cuuint32_t es[2] = {1, 1};
        if (enc(&m_w2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W2), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DSPARK_ERR_UNSUPPORTED;
    }
    const bool greedy = p->temperature == 0.f;
    const void* fn = nullptr;
    size_t smem = 0;
    switch (p->r) {
        case 64:
            fn = greedy ? (const void*)sample_tc_kernel<64, true> : (const void*)sample_tc_kernel<64, false>;
            smem = TcCfg<64>::kSmemBytes;
            break;
        case 128:
            fn = greedy ? (const void*)sample_tc_kernel<128, true> : (const void*)sample_tc_kernel<128, false>;
            smem = TcCfg<128>::kSmemBytes;
            break;
        case 256:
            fn = greedy ? (const void*)sample_tc_kernel<256, true> : (const void*)sample_tc_kernel<256, false>;
            smem = TcCfg<256>::kSmemBytes;
            break;
        default: return DSPARK_ERR_UNSUPPORTED;
    }
    int per_sm = 0;
    if (prepare_kernel(fn, smem, kTcThreads, &per_sm) != cudaSuccess || per_sm < 1) return DSPARK_ERR_CUDA;

    TcArgs a;
    a.B = p->B;
    a.gamma = p->gamma;
    a.V = p->V;
    a.nt = nt;
    a.nrb = (p->B + kTcRows - 1) / kTcRows;
    a.G = nt;
    a.part_ld = kTcEpiGroups * nt;
    a.scale2 = greedy ? 1.f : kLog2e / p->temperature;
    a.seed = p->seed;
    a.base = static_cast<const uint16_t*>(base_logits);
    a.W1 = static_cast<const uint16_t*>(W1);
    a.W2 = static_cast<const uint16_t*>(W2);
    a.anchor = anchor;
    a.tokens = tokens;
    a.draft_lse = draft_lse;
    a.zat = draft_logit_at_tok;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    a.hdr = reinterpret_cast<WsHeader*>(ws);
    a.slots = reinterpret_cast<unsigned long long*>(ws + L.slots);
    a.rb_count = reinterpret_cast<unsigned*>(ws + L.counts);
    a.part = reinterpret_cast<float*>(ws + L.part);
    a.limit_ns = wait_limit_ns();
    if (cudaMemsetAsync(workspace, 0, L.zeroed, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    void* args[] = {(void*)&m_base, (void*)&m_w2, (void*)&a};
    if (cudaLaunchCooperativeKernel(fn, dim3(nt), dim3(kTcThreads), args, smem, s) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    note_launch();
    return DSPARK_OK;
}

// ==========================================================================================
// Verify's residual and bonus draws on the tensor cores (dspark_verify, the correction draw of
// the chunk-Gumbel contract).  Method (P3 "Speculative Decoding"; P2 section 3.4): at the first
// rejection k of request j the correction is drawn from norm(max(0, p - q)), p = softmax(t/T) of
// target row k and q = softmax(z/T) with z = base[j, k-1] + W2 . W1[prev] rebuilt here; after a
// fully accepted block the bonus token is drawn from softmax(t/T) of row L_j + 1.
//
// One CTA per vocabulary tile (1024 ids) walks row blocks of 128 jobs (one TMEM lane each); the
// row blocks are independent.  Per accumulator of 128 ids one ring stage holds its W2 rows (one
// tiled copy) and each job's base and target rows (every job sits at its own position), copied
// by four warps in 16-byte pieces straight into the swizzled layout (tensor-copy gathers of four
// rows per instruction stream at 1.8 TB/s on this part: no faster).  z = base + W1[prev] . W2_rows^T is
// formed on the tensor cores exactly as in the sampler, and the target rows are moved into the
// neighbouring TMEM columns by the same identity MMAs, so a stage is free as soon as its MMAs have
// read it; the epilogue (thread = job) reads z and t from TMEM, forms the weights (residual: max(0, 2^(t s - lse2) - 2^(z s - dl2));
// bonus: 2^(t s - max of the chunk)) and the chunk records, and folds the best into the job's
// 64-bit word with one atomic max.  The last CTA to finish a row block writes the corrections;
// a residual with no mass at all is flagged for the whole-row fallback draw from p.
// ==========================================================================================
namespace {

enum { VJOB_NONE = 0, VJOB_RESID = 1, VJOB_BONUS = 2 };  // the job types the rows kernel emits
constexpr uint32_t kVtTile = 16384;                        // 128 rows x 128 bytes
constexpr uint32_t kVtStageBytes = 5 * kVtTile;            // {W2 rows, base box 0, 1, target box 0, 1}
constexpr int kVtStages = 2;
constexpr int kVtSlots = 2;  // accumulator pairs {z, t}: 2 x 256 TMEM columns
constexpr uint32_t kVtSmA = kVtStages * kVtStageBytes;     // [2] A operands (W1 rows of the prevs)
constexpr uint32_t kVtSmId = kVtSmA + 2 * kVtTile;
constexpr uint32_t kVtSmBars = kVtSmId + kIdBytes;
constexpr int kVtNumBars = 4 + 2 * kVtStages + 2 * kVtSlots + 3;
constexpr uint32_t kVtSmFlags = kVtSmBars + 8 * kVtNumBars;
constexpr uint32_t kVtSmRows = kVtSmFlags + 64;            // [2][128] the unit's base and target rows (-1: none)
constexpr size_t kVtSmemBytes = kVtSmRows + 2 * kTcRows * 4;
static_assert(kVtSmemBytes <= 227 * 1024, "shared memory of the tensor-core verify kernel");
constexpr int kVtLineWords = (int)(kVtcLine / 8);
constexpr int kVtLineInts = (int)(kVtcLine / 4);

__device__ __forceinline__ long long vt_target_row(const VerifyTcArgs& a, int j, int i) {  // i 1-based
    return a.toff ? (long long)a.toff[j] + i - 1 : (long long)j * a.gamma_t + i - 1;
}

// The chunk record of one job over 32 ids (t: target values, z: TMEM bits of z; mode: the job's
// type).  Every lane of the warp calls it for the same chunk (its one vote stays warp-uniform).
template <bool GREEDY, bool MASK>
__device__ __forceinline__ void chunk_job(const float (&t)[32], const uint32_t (&zv)[32], int mode, int id0, int V,
                                          float scale2, float lse2, float dl2, float u, float lnE, float& bkey,
                                          int& bcand) {
    if (GREEDY) {  // bonus jobs only: the argmax of the target row, lowest id on ties
        float m = -CUDART_INF_F;
        int x = 0;
#pragma unroll
        for (int e = 31; e >= 0; --e) {
            const float v = (MASK && id0 + e >= V) ? -CUDART_INF_F : t[e];
            if (v >= m) {
                m = v;
                x = e;
            }
        }
        if (mode == VJOB_BONUS && m > bkey) {
            bkey = m;
            bcand = id0 + x;
        }
        return;
    }
    uint64_t q[8], r[8];  // weights: q[k] = ids (k, 8 + k), r[k] = ids (16 + k, 24 + k)
    float ref = 0.f;
    if (mode == VJOB_RESID) {
        const uint64_t s2 = pk2(scale2, scale2), nl = pk2(-lse2, -lse2), nd = pk2(-dl2, -dl2);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float2 pa = up2(fma2(pk2(t[k], t[8 + k]), s2, nl));
            const float2 qa = up2(fma2(pk2(__uint_as_float(zv[k]), __uint_as_float(zv[8 + k])), s2, nd));
            const float2 pb = up2(fma2(pk2(t[16 + k], t[24 + k]), s2, nl));
            const float2 qb = up2(fma2(pk2(__uint_as_float(zv[16 + k]), __uint_as_float(zv[24 + k])), s2, nd));
            float w0 = fmaxf(ex2(pa.x) - ex2(qa.x), 0.f), w1 = fmaxf(ex2(pa.y) - ex2(qa.y), 0.f);
            float w2 = fmaxf(ex2(pb.x) - ex2(qb.x), 0.f), w3 = fmaxf(ex2(pb.y) - ex2(qb.y), 0.f);
            if (MASK) {
                w0 = id0 + k < V ? w0 : 0.f;
                w1 = id0 + 8 + k < V ? w1 : 0.f;
                w2 = id0 + 16 + k < V ? w2 : 0.f;
                w3 = id0 + 24 + k < V ? w3 : 0.f;
            }
            q[k] = pk2(w0, w1);
            r[k] = pk2(w2, w3);
        }
    } else if (mode == VJOB_BONUS) {
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = (MASK && id0 + e >= V) ? -CUDART_INF_F : t[e];
        const float m = max32(x) * scale2;
        ref = m == -CUDART_INF_F ? 0.f : m;
        const uint64_t s2 = pk2(scale2, scale2), nr = pk2(-ref, -ref);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float2 xa = up2(fma2(pk2(x[k], x[8 + k]), s2, nr));
            const float2 xb = up2(fma2(pk2(x[16 + k], x[24 + k]), s2, nr));
            q[k] = pk2(ex2(xa.x), ex2(xa.y));
            r[k] = pk2(ex2(xb.x), ex2(xb.y));
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = r[k] = pk2(0.f, 0.f);
    }
#pragma unroll
    for (int k = 1; k < 8; ++k) {  // inclusive prefix inside each block of eight
        q[k] = add2(q[k], q[k - 1]);
        r[k] = add2(r[k], r[k - 1]);
    }
    const float2 qe = up2(q[7]), re = up2(r[7]);
    const float o1 = qe.x, o2 = o1 + qe.y, o3 = o2 + re.x;
    const float S = o3 + re.y;
    const float tt = u * S, t1 = tt - o1, t2 = tt - o2, t3 = tt - o3;
    uint32_t neg = 0;  // minus the number of prefix values not above the target: the crossing index
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float2 qa = up2(q[k]), rb = up2(r[k]);
        neg += le_mask(qa.x, tt) + le_mask(qa.y, t1) + le_mask(rb.x, t2) + le_mask(rb.y, t3);
    }
    int cnt = -(int)neg;
    if (__any_sync(0xffffffffu, cnt == 32)) {  // rounding left no crossing: the last id with weight
        if (cnt == 32) {
            int last = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float2 qa = up2(q[k]), rb = up2(r[k]);
                const float2 pa = k ? up2(q[k - 1]) : make_float2(0.f, 0.f);
                const float2 pb = k ? up2(r[k - 1]) : make_float2(0.f, 0.f);
                last = qa.x > pa.x ? max(last, k) : last;
                last = qa.y > pa.y ? max(last, 8 + k) : last;
                last = rb.x > pb.x ? max(last, 16 + k) : last;
                last = rb.y > pb.y ? max(last, 24 + k) : last;
            }
            cnt = last;
        }
    }
    if (S > 0.f) {
        const float key = (ref + lg2(S)) * kLn2 - lnE;
        if (key > bkey) {
            bkey = key;
            bcand = id0 + cnt;
        }
    }
}

template <bool GREEDY>
__global__ void __launch_bounds__(kTcThreads, 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap tm_w2, const VerifyTcArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.hdr);
    if (smem_addr(smem_raw) & 1023u) {  // the swizzled tiles need 1024-byte alignment (uniform exit)
        if (threadIdx.x == 0) record_status(&hdr->status, DSPARK_ERR_UNSUPPORTED);
        return;
    }
    unsigned char* sm = smem_raw;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kVtSmBars);
    uint64_t* a_full = bars;                    // [2]
    uint64_t* a_empty = bars + 2;               // [2]
    uint64_t* b_full = bars + 4;                // [kVtStages]
    uint64_t* b_empty = b_full + kVtStages;     // [kVtStages]
    uint64_t* t_full = b_empty + kVtStages;     // [kVtSlots]
    uint64_t* t_empty = t_full + kVtSlots;      // [kVtSlots]
    uint64_t* done_bar = t_empty + kVtSlots;
    uint64_t* drain_bar = done_bar + 1;
    uint64_t* drain_t = drain_bar + 1;  // the target mover's MMAs
    int* flags = reinterpret_cast<int*>(sm + kVtSmFlags);
    volatile int* abort = flags;
    int* wg_done = flags + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(flags + 2);
    volatile int* nb_issued = flags + 3;
    volatile int* n_mma = flags + 4;
    volatile int* n_mma_t = flags + 5;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, tile0 = tile * kTcTile;
    const int total = a.nrb;
    const uint64_t lim = a.limit_ns;

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&a_full[b], 4);
            mbar_init(&a_empty[b], 1);
        }
        for (int b = 0; b < kVtStages; ++b) {
            mbar_init(&b_full[b], 5);   // the W2 copy's arrival with its bytes + one per copying warp
            mbar_init(&b_empty[b], 2);  // both MMA issuers have read the stage
        }
        for (int b = 0; b < kVtSlots; ++b) {
            mbar_init(&t_full[b], 2);  // z and t are in: both MMA issuers' commits
            mbar_init(&t_empty[b], 4);
        }
        mbar_init(done_bar, 1);
        mbar_init(drain_bar, 1);
        mbar_init(drain_t, 1);
        for (int f = 0; f < 16; ++f) flags[f] = 0;
        mbar_init_fence();
    }
    if (tid < 128) {  // the identity B operand: row n holds 1.0 at k = n (units 0 and 1 of its row)
        const int n = tid >> 3, u = tid & 7;
        const int k = n & 7;
        const uint32_t one = (u < 2 && (n >> 3) == u) ? ((k & 1) ? 0x3F800000u : 0x00003F80u) : 0u;
        const int wd = k >> 1;
        *reinterpret_cast<uint4*>(sm + kVtSmId + sw128_offset(n, u)) =
            make_uint4(wd == 0 ? one : 0u, wd == 1 ? one : 0u, wd == 2 ? one : 0u, wd == 3 ? one : 0u);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------------- W2 copies
        if (lane == 0) {
            tma_prefetch_desc(&tm_w2);
            const uint64_t keep = l2_policy_evict_last();
            const int nacc = total * kTcAccs;
            for (int ga = 0; ga < nacc; ++ga) {
                const int st = ga % kVtStages, use = ga / kVtStages;
                if (use > 0 &&
                    !mbar_wait_hint_or_abort(&b_empty[st], (uint32_t)((use - 1) & 1), abort, &hdr->status, lim))
                    break;
                mbar_arrive_expect_tx(&b_full[st], kVtTile);
                tma_load_2d(sm + st * kVtStageBytes, &tm_w2, 0, tile0 + kTcN * (ga % kTcAccs), &b_full[st], keep);
                *nb_issued = ga + 1;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc_bias = umma_idesc_bf16(kTcRows, kTcN);
            constexpr uint32_t idesc_base = umma_idesc_bf16(kTcRows, 16);
            const uint64_t id_desc = umma_desc_sw128(smem_addr(sm + kVtSmId), 1024);
            const uint64_t ring_desc = umma_desc_sw128(smem_addr(sm), 1024);
            const uint64_t a_desc = umma_desc_sw128(smem_addr(sm + kVtSmA), 1024);
            bool ok = true;
            for (int u = 0; u < total && ok; ++u) {
                const int ab = u & 1;
                if (!mbar_wait_hint_or_abort(&a_full[ab], (uint32_t)((u >> 1) & 1), abort, &hdr->status, lim)) break;
                for (int acc = 0; acc < kTcAccs && ok; ++acc) {
                    const int ga = u * kTcAccs + acc, sl = ga % kVtSlots, use = ga / kVtSlots, st = ga % kVtStages;
                    if ((use > 0 && !mbar_wait_hint_or_abort(&t_empty[sl], (uint32_t)((use - 1) & 1), abort,
                                                             &hdr->status, lim)) ||
                        !mbar_wait_hint_or_abort(&b_full[st], (uint32_t)((ga / kVtStages) & 1), abort, &hdr->status,
                                                 lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)(sl * 2 * kTcN);
                    const uint64_t sd = ring_desc + (uint64_t)(st * (int)(kVtStageBytes >> 4));
#pragma unroll
                    for (int k = 0; k < 4; ++k)  // D = W1[prev] . W2_rows^T
                        umma_bf16(d, a_desc + (uint64_t)(ab * (int)(kVtTile >> 4) + 2 * k), sd + 2 * k, idesc_bias,
                                  k > 0 ? 1u : 0u);
                    *n_mma = 1;
#pragma unroll
                    for (int bx = 0; bx < 2; ++bx)
#pragma unroll
                        for (int i = 0; i < kTcBox / 16; ++i)  // D[:, 64 bx + 16 i ..] += base[:, 16 i ..] . I
                            umma_bf16(d + (uint32_t)(kTcBox * bx + 16 * i),
                                      sd + (uint64_t)((1 + bx) * (int)(kVtTile >> 4) + 2 * i), id_desc, idesc_base, 1u);
                    umma_commit(&b_empty[st]);  // the stage is free once these (and the target mover's) have read it
                    umma_commit(&t_full[sl]);
                }
                if (ok) umma_commit(&a_empty[ab]);
            }
        }
        __syncwarp();
    } else if (warp == 3) {
        // ---------------------------------------------------------------- target mover
        // A second MMA issuer: the eight identity MMAs per accumulator that move the jobs' target rows
        // into the neighbouring TMEM columns (their own columns, so no order against warp 1's MMAs is
        // needed); the stage and the slot each wait for both issuers' commits.
        if (lane == 0) {
            constexpr uint32_t idesc_base = umma_idesc_bf16(kTcRows, 16);
            const uint64_t id_desc = umma_desc_sw128(smem_addr(sm + kVtSmId), 1024);
            const uint64_t ring_desc = umma_desc_sw128(smem_addr(sm), 1024);
            const int nacc = total * kTcAccs;
            for (int ga = 0; ga < nacc; ++ga) {
                const int sl = ga % kVtSlots, use = ga / kVtSlots, st = ga % kVtStages;
                if ((use > 0 && !mbar_wait_hint_or_abort(&t_empty[sl], (uint32_t)((use - 1) & 1), abort, &hdr->status,
                                                         lim)) ||
                    !mbar_wait_hint_or_abort(&b_full[st], (uint32_t)((ga / kVtStages) & 1), abort, &hdr->status, lim))
                    break;
                tc_fence_after();
                const uint32_t dt = tmem + (uint32_t)(sl * 2 * kTcN) + (uint32_t)kTcN;
                const uint64_t sd = ring_desc + (uint64_t)(st * (int)(kVtStageBytes >> 4));
                *n_mma_t = 1;
#pragma unroll
                for (int bx = 0; bx < 2; ++bx)
#pragma unroll
                    for (int i = 0; i < kTcBox / 16; ++i)  // T[:, 64 bx + 16 i ..] = target[:, 16 i ..] . I
                        umma_bf16(dt + (uint32_t)(kTcBox * bx + 16 * i),
                                  sd + (uint64_t)((3 + bx) * (int)(kVtTile >> 4) + 2 * i), id_desc, idesc_base, 0u);
                umma_commit(&b_empty[st]);
                umma_commit(&t_full[sl]);
            }
            if (*n_mma_t) {  // every MMA of this thread has completed before the tensor memory is freed
                umma_commit(drain_t);
                mbar_wait_bounded(drain_t, 0, &hdr->status, lim);
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ---------------------------------------------------------------- finisher
        for (int u = 0; u < total; ++u) {
            int ok = 1, last = 0;
            if (lane == 0) {
                const uint64_t t0 = global_ns();
                int c;
                while ((c = ld_acq_cta(wg_done)) < kTcEpiGroups * (u + 1)) {
                    mbar_try_wait_hint(done_bar, (uint32_t)(c & 1), 20000u);
                    if (*abort) {
                        ok = 0;
                        break;
                    }
                    if (global_ns() - t0 > lim) {
                        record_status(&hdr->status, DSPARK_ERR_TIMEOUT);
                        *abort = 1;
                        ok = 0;
                        break;
                    }
                }
                if (ok) {  // this tile's maxima of row block u are in: count it; the last tile finishes
                    unsigned old;
                    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                                 : "=r"(old)
                                 : "l"(a.rb_count + (size_t)u * kVtLineInts)
                                 : "memory");
                    last = old == (unsigned)(a.nt - 1);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            last = __shfl_sync(0xffffffffu, last, 0);
            if (!ok) break;
            if (last) {
                __syncwarp();  // lane 0's acquire above orders the other CTAs' maxima before these reads
                __threadfence();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int j = u * kTcRows + 4 * lane + k;
                    if (j >= a.B) continue;
                    const int4 q = a.job[j];
                    if (q.x != VJOB_RESID && q.x != VJOB_BONUS) continue;
                    const unsigned long long w = __ldcg(a.words + (size_t)j * kVtLineWords);
                    const int cand = ~(int)(uint32_t)w;
                    if (cand >= 0 && cand < a.V) a.corr[j] = cand;
                    else if (q.x == VJOB_RESID) a.fb[j] = 1;  // no residual mass anywhere: draw from p instead
                }
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------------------------------------------------------- job rows and A operands
        // Per unit: the table of the jobs' base and target rows, then the A operand (thread = job).
        // Per accumulator: warp w copies rows 32 w .. 32 w + 31 of both arrays, 16 lanes per row
        // (one 256-byte segment, 16-byte pieces into the swizzled slots); the copies of the next
        // accumulator are in flight while the previous ones complete and are handed over.
        const int row = tid - 128, cw = warp - 4;
        int* s_br = reinterpret_cast<int*>(sm + kVtSmRows);
        int* s_tr = s_br + kTcRows;
        const uint16_t* basep = static_cast<const uint16_t*>(a.base);
        const uint16_t* tgtp = static_cast<const uint16_t*>(a.target);
        // A warp whose bounded wait gave up stays in the loop without doing work until the four warps
        // agree, at the next unit start (a barrier reduction), to leave together: the named barriers
        // are never left with a warp missing.
        int pend = -1;  // stage whose copies are in flight and not yet handed over
        bool live = true;
        const int nacc = total * kTcAccs;
        for (int ga = 0; ga < nacc; ++ga) {
            const int u = ga / kTcAccs, acc = ga % kTcAccs, st = ga % kVtStages, use = ga / kVtStages;
            if (acc == 0) {
                // every copier has issued the previous unit's copies (its table reads); all alive?
                if (bar_red_or(4, 128, !live)) break;
                const int j = u * kTcRows + row;
                const int4 q = j < a.B ? a.job[j] : make_int4(VJOB_NONE, 0, 0, 0);
                const bool resid = q.x == VJOB_RESID, bonus = q.x == VJOB_BONUS;
                const long long t = (resid || bonus) && q.y >= 1 ? vt_target_row(a, j, q.y) : -1;
                s_br[row] = resid && q.y >= 1 && q.y <= a.gamma ? j * a.gamma + q.y - 1 : -1;
                s_tr[row] = (t >= 0 && t < a.target_rows) ? (int)t : -1;
                // the A operand of the unit: the W1 row of the job's previous token
                const int prev = resid ? min(max(q.z, 0), a.V - 1) : 0;
                uint4 w[8];
                const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.W1) + (size_t)prev * 64);
#pragma unroll
                for (int k = 0; k < 8; ++k) w[k] = __ldg(src + k);
                int ok = 1;
                if (u >= 2 && lane == 0)
                    ok = mbar_wait_hint_or_abort(&a_empty[u & 1], (uint32_t)(((u >> 1) - 1) & 1), abort, &hdr->status,
                                                 lim) ? 1 : 0;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (ok) {
                    if (u >= 2) mbar_try_wait(&a_empty[u & 1], (uint32_t)(((u >> 1) - 1) & 1));  // (this lane's acquire)
                    unsigned char* ad = sm + kVtSmA + (u & 1) * kVtTile;
#pragma unroll
                    for (int k = 0; k < 8; ++k) *reinterpret_cast<uint4*>(ad + sw128_offset(row, k)) = w[k];
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                if (bar_red_or(4, 128, !ok)) {  // the table is complete (or the kernel is giving up)
                    live = false;
                    break;
                }
                if (lane == 0) mbar_arrive_local(&a_full[u & 1]);
            }
            if (!live) continue;
            int ok = 1;
            if (use > 0 && lane == 0)
                ok = mbar_wait_hint_or_abort(&b_empty[st], (uint32_t)((use - 1) & 1), abort, &hdr->status, lim) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                live = false;
                continue;
            }
            if (use > 0) mbar_try_wait(&b_empty[st], (uint32_t)((use - 1) & 1));  // (this lane's acquire)
            const int id0 = tile0 + kTcN * acc;
            const int unit = lane & 15, box = unit >> 3;
            if (id0 + kTcBox * box < a.V) {  // (V % 64 == 0: a box is wholly inside or outside)
                unsigned char* stg = sm + st * kVtStageBytes;
#pragma unroll 4
                for (int i = 0; i < 16; ++i) {
                    const int rr = 32 * cw + 2 * i + (lane >> 4);
                    const uint32_t off = sw128_offset(rr, unit & 7);
                    const int br = s_br[rr], tr = s_tr[rr];
                    if (br >= 0)
                        cp_async_16(stg + (1 + box) * kVtTile + off, basep + (size_t)br * a.V + id0 + 8 * unit);
                    if (tr >= 0)
                        cp_async_16(stg + (3 + box) * kVtTile + off, tgtp + (size_t)tr * a.V + id0 + 8 * unit);
                }
            }
            cp_async_commit();
            if (pend >= 0) {  // the previous accumulator's rows have landed: hand its stage over
                cp_async_wait_group<1>();
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive_local(&b_full[pend]);
            }
            pend = st;
        }
        cp_async_wait_group<0>();  // nothing of this thread's lands after the block leaves
        if (pend >= 0 && live) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive_local(&b_full[pend]);
        }
    } else if (warp >= 8) {
        // ---------------------------------------------------------------- epilogue (thread = job)
        const int h = (warp - 8) >> 2;
        const int row = (warp & 3) * 32 + lane;
        const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const bool full_tile = tile0 + kTcTile <= a.V;
        bool live = true;
        for (int u = 0; u < total && live; ++u) {
            const int j = u * kTcRows + row;
            const int4 q = j < a.B ? a.job[j] : make_int4(VJOB_NONE, 0, 0, 0);
            const int mode = (q.x == VJOB_RESID || q.x == VJOB_BONUS) ? q.x : VJOB_NONE;
            const uint32_t pos = (uint32_t)q.y;
            const uint32_t p_chunk = mode == VJOB_RESID ? DSPARK_P_RESID_CHUNK : DSPARK_P_BONUS_CHUNK;
            const float uin = (!GREEDY && mode != VJOB_NONE)
                                  ? uniform(a.seed, (uint32_t)j, pos,
                                            mode == VJOB_RESID ? DSPARK_P_RESID_INCHUNK : DSPARK_P_BONUS_INCHUNK, 0u)
                                  : 0.f;
            const float lse2 = __int_as_float(q.w);
            const float dl2 = mode == VJOB_RESID ? a.dlse[(size_t)j * a.gamma + q.y - 1] * kLog2e : 0.f;
            float bkey = -CUDART_INF_F;
            int bcand = -1;
            bool ok = true;
            for (int ah = 0; ah < kTcAccs / 2; ++ah) {
                const int acc = 2 * ah + h;
                const int ga = u * kTcAccs + acc, sl = ga % kVtSlots;
                float lnE[4] = {0.f, 0.f, 0.f, 0.f};
                if (!GREEDY && mode != VJOB_NONE)
                    chunk_variates4(a.seed, (uint32_t)j, pos, (uint32_t)(tile * (kTcTile / 128) + acc), lnE, p_chunk);
                int okw = 1;
                if (lane == 0)
                    okw = mbar_wait_hint_or_abort(&t_full[sl], (uint32_t)((ga / kVtSlots) & 1), abort, &hdr->status, lim)
                              ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, okw, 0)) {
                    ok = false;
                    break;
                }
                mbar_try_wait(&t_full[sl], (uint32_t)((ga / kVtSlots) & 1));  // (this lane's acquire)
                tc_fence_after();
                const uint32_t taddr = tl + (uint32_t)(sl * 2 * kTcN);  // z; t in the next 128 columns
                const int id0 = tile0 + kTcN * acc;
                // one copy of the chunk code, not four (the variants of chunk_job are large): the
                // instruction cache, not the arithmetic, held this loop back when it was unrolled
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    const float le = cc == 0 ? lnE[0] : (cc == 1 ? lnE[1] : (cc == 2 ? lnE[2] : lnE[3]));
                    uint32_t zv[32], tv[32];
                    tmem_ld32(taddr + 32u * (uint32_t)cc, zv);
                    tmem_ld32(taddr + (uint32_t)kTcN + 32u * (uint32_t)cc, tv);
                    tmem_wait_ld(zv);
                    tmem_wait_ld(tv);
                    float t[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) t[e] = __uint_as_float(tv[e]);
                    const int idc = id0 + 32 * cc;
                    if (full_tile)
                        chunk_job<GREEDY, false>(t, zv, mode, idc, a.V, a.scale2, lse2, dl2, uin, le, bkey, bcand);
                    else if (idc < a.V)  // (uniform) a chunk wholly past V has no ids
                        chunk_job<GREEDY, true>(t, zv, mode, idc, a.V, a.scale2, lse2, dl2, uin, le, bkey, bcand);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_local(&t_empty[sl]);
            }
            if (ok && mode != VJOB_NONE && bcand >= 0)
                red_max_u64(a.words + (size_t)j * kVtLineWords, pack_key(bkey, bcand));
            if (bar_red_or(1 + h, 128, !ok)) {
                live = false;
                break;
            }
            if (row == 0) {
                add_rel_cta(wg_done, 1);
                mbar_arrive_local(done_bar);
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *abort) {  // copies in flight land before the shared memory goes away
        const int nb = *nb_issued;
        for (int g = max(0, nb - kVtStages); g < nb; ++g)
            mbar_wait_bounded(&b_full[g % kVtStages], (uint32_t)((g / kVtStages) & 1), &hdr->status, lim);
    }
    if (warp == 1) {
        if (lane == 0 && *n_mma) {
            umma_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, &hdr->status, lim);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool verify_tc_eligible(const dspark_sample_params* p, const void* base, const void* target, const void* W1,
                        const void* W2) {
    return p->logits_dtype == DSPARK_BF16 && p->w_dtype == DSPARK_BF16 && p->r == 64 && p->B >= kTcMinBatch &&
           p->softcap == 0.f && p->V % 64 == 0 && ((uintptr_t)base % 16) == 0 && ((uintptr_t)target % 16) == 0 &&
           ((uintptr_t)W1 % 16) == 0 && ((uintptr_t)W2 % 16) == 0 && tensor_map_encoder() != nullptr;
}

dspark_status launch_verify_tc(const VerifyTcArgs& a, cudaStream_t s) {
    auto enc = tensor_map_encoder();
    if (!enc) return DSPARK_ERR_UNSUPPORTED;
    CUtensorMap m_w2;
    {
        cuuint64_t dims[2] = {64, (cuuint64_t)a.V};
        cuuint64_t strides[1] = {64 * 2};
        cuuint32_t box[2] = {64, kTcN};
        cuuint32_t es[2] = {1, 1};
        if (enc(&m_w2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.W2), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DSPARK_ERR_UNSUPPORTED;
    }
    if (a.target_rows < 1 || a.target_rows > (long long)INT32_MAX || (long long)a.B * a.gamma > (long long)INT32_MAX)
        return DSPARK_ERR_UNSUPPORTED;
    const void* fn = a.greedy ? (const void*)verify_tc_kernel<true> : (const void*)verify_tc_kernel<false>;
    int per_sm = 0;
    if (prepare_kernel(fn, kVtSmemBytes, kTcThreads, &per_sm) != cudaSuccess || per_sm < 1) return DSPARK_ERR_CUDA;
    void* args[] = {(void*)&m_w2, (void*)&a};
    if (cudaLaunchKernel(fn, dim3(a.nt), dim3(kTcThreads), args, kVtSmemBytes, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    note_launch();
    return DSPARK_OK;
}

}  // namespace dspark
