// host_util.h -- host-side helpers shared by the libdspark translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

constexpr size_t kMaxSmem = 227 * 1024;  // opt-in dynamic shared memory per block on sm_103a

cudaError_t device_sm_count(int* sms);  // multiprocessors of the current device (cached)
// Raises the kernel's dynamic shared-memory limit to `smem` (once per device and kernel) and
// returns its co-resident blocks per SM at (threads, smem); both cached per device.
cudaError_t prepare_kernel(const void* fn, size_t smem, int threads, int* per_sm);
// Co-resident clusters of `cs` blocks of (threads, smem) for `fn` (its shared-memory limit must
// already be raised); cached per device.  *n = 0 when the shape cannot launch.
cudaError_t max_active_clusters(const void* fn, int cs, int threads, size_t smem, int* n);
uint64_t wait_limit_ns();               // bound of every grid-wide wait

dspark_status validate_sample_params(const dspark_sample_params* p);
size_t sample_workspace_bytes(const dspark_sample_params* p);
bool markov_use_mma(const dspark_sample_params* p);

// Byte offsets inside the draft-sampling workspace (dspark_sample_workspace_size bytes):
// packed maxima [gamma][B] (one 128-byte line each), per-row-block arrival counters, and the
// per-tile records; the first `zeroed` bytes (header, maxima, counters) are cleared per call.
struct SampleWsLayout {
    size_t slots, counts, part, zeroed;
};
SampleWsLayout sample_ws_layout(const dspark_sample_params* p);

// Tensor-core draft sampler (sample_tc.cu): bf16 logits and weights of rank 64, 128 or 256, at least
// kTcMinBatch requests, V % 8 == 0, 16-byte aligned tensors, one vocabulary tile per SM.
constexpr int kTcMinBatch = 64;
bool sample_tc_eligible(const dspark_sample_params* p, const void* base, const void* W1, const void* W2, int sms);
dspark_status launch_sample_tc(const dspark_sample_params* p, const void* base_logits, const void* W1, const void* W2,
                               const int32_t* anchor, int32_t* tokens, float* draft_lse, float* draft_logit_at_tok,
                               const SampleWsLayout& L, void* workspace, cudaStream_t s);

// Counts the kernels the library enqueues (dspark_kernel_launches reads the total).
void note_launch(int n = 1);

// Tensor-core residual / bonus draws of verify (sample_tc.cu): bf16 logits and weights of rank 64,
// V % 64 == 0, at least kTcMinBatch requests, 16-byte aligned tensors, no softcap, vanilla head.
// One CTA per vocabulary tile walks row blocks of 128 jobs; each job's base and target rows are
// gathered four at a time by tensor copies.
constexpr size_t kVtcLine = 128;  // bytes between two jobs' packed words / two row blocks' counters
struct VerifyTcArgs {
    int B, gamma, V, nt, nrb, greedy;
    float scale2;                 // log2(e) / T (1 when greedy)
    uint64_t seed;
    const void* base;             // bf16 [B, gamma, V]
    const void* target;           // bf16 target rows: dense [B, gamma_t, V] or CSR [target_rows, V]
    long long target_rows;
    int gamma_t;                  // dense layout: rows per request (0 with offsets)
    const int32_t* toff;          // CSR row offsets [B + 1] or null
    const void* W1;               // bf16 [V, 64]
    const void* W2;               // bf16 [V, 64]
    const int4* job;              // [B] {type, 1-based position, prev token, log2-sum-exp bits of the target row}
    const float* dlse;            // [B, gamma] draft LSE (natural)
    int32_t* corr;                // [B] corrections (written for RESID / BONUS jobs)
    int32_t* fb;                  // [B] set where a residual has no mass (zeroed per call)
    unsigned long long* words;    // [B] packed maxima, kVtcLine apart (zeroed per call)
    unsigned* rb_count;           // [nrb] arrival counters, kVtcLine apart (zeroed per call)
    void* hdr;                    // the workspace header (status word)
    uint64_t limit_ns;
};
bool verify_tc_eligible(const dspark_sample_params* p, const void* base, const void* target, const void* W1,
                        const void* W2);
dspark_status launch_verify_tc(const VerifyTcArgs& a, cudaStream_t s);

}  // namespace dspark
