/*
 * dspark.h -- C ABI of libdspark, the GB300 (sm_103a) hot path of DSpark
 * semi-autoregressive speculative decoding.
 *
 * The operations follow four web pages about DSpark, cited by title and section:
 *   P1 "03 · DSpark 建模：Markov 与 Confidence"
 *   P2 "从 DFlash 到 dLLM Self-Spec（三）：DSpark 的半自回归 Draft 与负载感知 Verify"
 *   P3 "如何评价 DeepSeek 发布 DSpark？哪些亮点值得关注？" (reading notes)
 *   P4 "DSpark 深度解读：DeepSeek-V4 如何用「半自回归」把推理速度提升 85%"
 *
 * Conventions for every entry point
 *   - Pointers to tensors are DEVICE pointers (cudaMalloc / torch CUDA memory) unless
 *     stated otherwise; all tensors are dense, row-major, C-contiguous.
 *   - The caller owns every buffer.  The library allocates no device memory: scratch
 *     comes from a caller-provided workspace of at least dspark_*_workspace_size()
 *     bytes, 256-byte aligned.  A workspace may be reused by later calls on the same
 *     stream but must not be shared by calls that can run concurrently.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous: they validate arguments on the host, enqueue kernels and return.
 *     Host-detected errors return a status and enqueue nothing.  Errors detected on
 *     the device (out-of-range token ids, a device wait that gave up) are written to
 *     a status word at the start of the workspace; read it with
 *     dspark_get_device_status(), which synchronises the stream.
 *   - Token ids are int32 in [0, V).  Logits are fp32 or bf16 (DSPARK_F32 /
 *     DSPARK_BF16); arithmetic is fp32 with fp32 accumulation.
 *   - Randomness is counter-based (Philox4x32-10; Salmon et al., SC 2011), so every
 *     call is reproducible from its arguments: key = (low 32 bits of seed, high 32
 *     bits), counter = (n / 4, i, j, purpose), output word n mod 4, mapped to
 *     (0,1) as (floor(word / 2^9) + 1/2) * 2^-23.  j = request index within the call,
 *     i = 1-based block position, purpose = one of DSPARK_P_*, n = draw index.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* dspark_stream_t;

typedef enum {
    DSPARK_OK = 0,
    DSPARK_ERR_INVALID_ARG = 1, /* bad pointer, size, dtype or value */
    DSPARK_ERR_UNSUPPORTED = 2, /* valid but outside what this build handles */
    DSPARK_ERR_CUDA = 3,        /* a CUDA runtime call failed */
    DSPARK_ERR_TIMEOUT = 4,     /* device: a grid-wide wait gave up (status word only) */
    DSPARK_ERR_BUDGET = 5,      /* scheduler: budget < B */
    DSPARK_ERR_WORKSPACE = 6,   /* workspace NULL, misaligned or too small */
    DSPARK_ERR_TOKEN_RANGE = 7  /* device: a token/anchor id outside [0, V) or a bad row count (status word only) */
} dspark_status;

enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 };

/* Random-draw purposes (the fourth Philox counter word). */
enum {
    DSPARK_P_SAMPLE_CHUNK = 1,   /* draft sampling: one uniform per vocabulary chunk (n = chunk index) */
    DSPARK_P_SAMPLE_INCHUNK = 2, /* draft sampling: the in-chunk inverse-CDF uniform (n = 0) */
    DSPARK_P_ACCEPT = 3,        /* verify: the acceptance uniform u_i */
    DSPARK_P_RESID_CHUNK = 4,   /* verify: residual draw, one uniform per vocabulary chunk (n = chunk index) */
    DSPARK_P_RESID_INCHUNK = 5, /* verify: residual draw, the in-chunk inverse-CDF uniform (n = 0) */
    DSPARK_P_BONUS_CHUNK = 6,   /* verify: bonus draw from the next target row, per chunk */
    DSPARK_P_BONUS_INCHUNK = 7  /* verify: bonus draw, in chunk */
};

/* The chunk of the sampling contract below; the kernels split the vocabulary into tiles of
 * DSPARK_TILE ids (a whole number of chunks), which does not change the draw. */
#define DSPARK_TILE 1024
#define DSPARK_CHUNK 32

/*
 * Sampling contract (the pages never show the body of sample_tokens, P2 section 3.4; any exact
 * categorical draw is lossless, bit-parity needs one fixed definition).  Every draw of the library
 * -- the draft tokens and verify's residual and bonus corrections -- is the same chunk-Gumbel draw
 * with its own pair of purposes (CHUNK, INCHUNK):
 *   T == 0: x = argmax_v z_v, lowest index on ties.
 *   T > 0, over log-weights s_v (draft: z / T; residual: log max(0, p - q); bonus: t / T):
 *     chunks of DSPARK_CHUNK consecutive ids over the whole vocabulary (the last may be short);
 *     LSE_c = log sum_{v in c} e^{s_v};
 *       c* = argmax_c (LSE_c - ln E_c), E_c = -ln U(seed, j, i, CHUNK, c), lowest c on ties
 *            (chunks without mass never win);
 *       x  = smallest id v of c* with sum_{w in c*, w <= v} e^{s_w - LSE_c*} > U(.., INCHUNK, 0),
 *            or, where rounding leaves no crossing, the last id of c* with nonzero mass.
 *     Gumbel-max over chunks picks c with probability proportional to e^{LSE_c}; the in-chunk
 *     uniform is independent of the race, so v follows e^{s_v} inside c: the draw is softmax(s).
 */

typedef struct {
    int B;             /* requests in the call */
    int gamma;         /* block length: draft positions per request */
    int V;             /* vocabulary size */
    int r;             /* Markov rank (0 = no Markov head: the DFlash configuration, P1 section 3.13) */
    float temperature; /* 0 = greedy; > 0 = sample softmax(z / T) */
    uint64_t seed;     /* Philox key */
    int logits_dtype;  /* dtype of base (and target) logits: DSPARK_F32 or DSPARK_BF16 */
    int w_dtype;       /* dtype of W1 and W2 */
    float softcap;     /* final-logit softcap s of the draft model (P1 section 3.12, compute_logits:
                          s tanh(logits / s)): every base logit b is replaced by s tanh(b / s) before
                          the Markov bias is added (+-inf -> +-s); 0 = none.  Target logits are taken
                          as given (the target model applies its own cap). */
} dspark_sample_params;

/*
 * Markov-head block sampling (P2 section 3.4, VanillaMarkov and sample_block_tokens;
 * P1 section 3.7; P4 section 3.3):
 *   prev_1 = anchor[j];  for i = 1..gamma:
 *     z_{j,i} = cap(base[j, i-1, :]) + W2 . W1[prev_i]  (bias_v = sum_k W1[prev_i, k] W2[v, k];
 *                                                        cap = the softcap of p, or the identity)
 *     x_{j,i} ~ draft sampling contract on z_{j,i} / T;  prev_{i+1} = x_{j,i}
 * Arguments
 *   base_logits [B, gamma, V] (logits_dtype); W1 [V, r], W2 [V, r] (w_dtype; W2 is the
 *   nn.Linear(r, V).weight layout, i.e. the page's r x V matrix transposed in memory;
 *   both may be NULL when r == 0); anchor [B] int32 (the token before the block).
 * Outputs
 *   tokens [B, gamma] int32; draft_lse [B, gamma] float = LSE_v(z/T) (NaN when T == 0);
 *   draft_logit_at_tok [B, gamma] float = z at the drafted token.
 * The gamma steps run inside one persistent kernel (a grid-wide wait per step).
 * Device status: DSPARK_ERR_TOKEN_RANGE for an anchor outside [0, V) (it is clamped and
 * the outputs are then undefined), DSPARK_ERR_TIMEOUT if a grid-wide wait gave up.
 */
size_t dspark_sample_workspace_size(const dspark_sample_params* p);
dspark_status dspark_markov_sample_block(const dspark_sample_params* p, const void* base_logits, const void* W1,
                                         const void* W2, const int32_t* anchor, int32_t* tokens, float* draft_lse,
                                         float* draft_logit_at_tok, void* workspace, size_t ws_bytes,
                                         dspark_stream_t stream);

/*
 * Gated and RNN Markov heads (P1 section 3.7; P4 section 3.3, the table of the three heads).
 * Both replace the vector that W2 multiplies: the vanilla head uses e = W1[prev]; with the
 * backbone's hidden state h_{j,i} [d] of position i these use
 *   DSPARK_HEAD_GATED: u = sigmoid(Wg [h; e]) * e              Wg [r, d + r], columns [h | e]
 *   DSPARK_HEAD_RNN:   z = [s; e; h]  (s_{j,0} = 0 per request, one state per request)
 *                      g = sigmoid(Wg z),  s <- g * s + (1 - g) * tanh(Wc z),  u = tanh(Wo z)
 *                                                              Wg, Wc, Wo [r, 2r + d], columns [s | e | h]
 * and z_{j,i} = cap(base[j, i-1, :]) + W2 u.  The RNN step forms u from the state before the update.
 * The gate is a logistic sigmoid and the state starts at zero (the pages show neither).
 */
enum { DSPARK_HEAD_VANILLA = 0, DSPARK_HEAD_GATED = 1, DSPARK_HEAD_RNN = 2 };
typedef struct {
    int kind;           /* DSPARK_HEAD_GATED or DSPARK_HEAD_RNN */
    int d;              /* hidden size (>= 1) */
    const void* hidden; /* [B, gamma, d] (w_dtype): the hidden state feeding position i (row i-1) */
    const void* Wg;     /* gated: [r, d + r]; rnn: [r, 2r + d]  (w_dtype) */
    const void* Wc;     /* rnn only: [r, 2r + d] (w_dtype); NULL for gated */
    const void* Wo;     /* rnn only: [r, 2r + d] (w_dtype); NULL for gated */
} dspark_head;

/*
 * dspark_markov_sample_block with a Gated or RNN head: the same draw, contracts and outputs,
 * with W2 u in place of W2 W1[prev].  Needs r >= 1.  head_vec [B, gamma, r] float (or NULL)
 * receives the u of every position, for dspark_verify_head.  The head vectors of a step are
 * computed in fp32 on CUDA cores inside the persistent kernel (B r (r + d) multiply-adds per step
 * for the gated head, 3 B r (2r + d) for the RNN head).
 * Host errors: as dspark_markov_sample_block, plus DSPARK_ERR_INVALID_ARG for a bad kind, d < 1,
 * r < 1 or a NULL hidden / weight, and DSPARK_ERR_UNSUPPORTED when the per-request head state
 * does not fit one block's shared memory (B r (1 gated, 3 rnn) floats next to the sampler's own).
 * Workspace: dspark_sample_head_workspace_size(p, head) bytes.
 */
size_t dspark_sample_head_workspace_size(const dspark_sample_params* p, const dspark_head* head);
dspark_status dspark_markov_sample_block_head(const dspark_sample_params* p, const dspark_head* head,
                                              const void* base_logits, const void* W1, const void* W2,
                                              const int32_t* anchor, int32_t* tokens, float* draft_lse,
                                              float* draft_logit_at_tok, float* head_vec, void* workspace,
                                              size_t ws_bytes, dspark_stream_t stream);

/*
 * Lossless verification by rejection sampling (P3 "Speculative Decoding": the target checks
 * the drafted positions in parallel, accepts left to right, truncates at the first failure
 * and resamples from the target, so the output law is the target's; the verify tokens of all
 * requests are one flattened list, P2 section 3.7.2):
 *   for i = 1..L_j:  p = softmax(t_{j,i} / T),  q(x) = exp(z_x / T - draft_lse)
 *     accept x_{j,i} iff ln U(seed, j, i, ACCEPT, 0) < ln p(x) - ln q(x)   (u < p/q)
 *   first rejection at k:  correction ~ norm(max(0, p_k - q_k)) (RESID purposes), where q_k over
 *     the vocabulary is rebuilt from base, W1, W2 and prev = x_{k-1} (anchor for k = 1) and
 *     normalised by draft_lse; if that residual has no mass, correction ~ p_k instead.
 *   all L_j accepted:  correction ~ p_{L_j+1} (BONUS purposes) if target row L_j+1 exists,
 *     else -1.
 *   T == 0: accept iff argmax t_{j,i} == x_{j,i}; the correction is the argmax of the
 *     rejecting (or bonus) target row.
 * Arguments
 *   p: the same parameters as the sampling call (B, gamma, V, r, T, seed, dtypes).
 *   base_logits, W1, W2, anchor: as for dspark_markov_sample_block.
 *   tokens, draft_lse, draft_logit_at_tok [B, gamma]: the sampling call's outputs.
 *   target_logits: target row i (1-based) of request j is
 *     dense  (target_row_offsets == NULL): target_logits[j, i-1, :] of a [B, gamma_t, V] tensor;
 *     flattened (target_row_offsets != NULL, [B+1] int32 CSR): row target_row_offsets[j] + i - 1
 *       of a [target_row_offsets[B], V] tensor; request j owns target_row_offsets[j+1] -
 *       target_row_offsets[j] rows (gamma_t is then ignored and may be 0).
 *   verify_len [B] int32 in [1, gamma] (NULL = gamma for every request): L_j.  Request j must own
 *     at least L_j target rows; a row L_j+1, when present, is the bonus row.
 * Outputs
 *   n_accepted [B] int32; correction_token [B] int32 (-1 = none).
 * Device status: DSPARK_ERR_TOKEN_RANGE for a token outside [0, V) or a request with fewer
 * than L_j target rows.
 */
size_t dspark_verify_workspace_size(const dspark_sample_params* p, int gamma_t);
dspark_status dspark_verify(const dspark_sample_params* p, const void* base_logits, const void* W1, const void* W2,
                            const int32_t* anchor, const int32_t* tokens, const float* draft_lse,
                            const float* draft_logit_at_tok, const void* target_logits, int gamma_t,
                            const int32_t* verify_len, const int32_t* target_row_offsets, int32_t* n_accepted,
                            int32_t* correction_token, void* workspace, size_t ws_bytes, dspark_stream_t stream);

/*
 * dspark_verify for drafts of a Gated or RNN head: the residual's q_k is rebuilt from
 * head_vec [B, gamma, r] float (dspark_markov_sample_block_head's output) as
 * cap(base) + W2 head_vec[j, k-1] instead of W1[prev].  W1 is not read and may be NULL; every
 * other argument, output and error is that of dspark_verify.  Workspace: dspark_verify_workspace_size.
 */
dspark_status dspark_verify_head(const dspark_sample_params* p, const void* base_logits, const float* head_vec,
                                 const void* W2, const int32_t* anchor, const int32_t* tokens, const float* draft_lse,
                                 const float* draft_logit_at_tok, const void* target_logits, int gamma_t,
                                 const int32_t* verify_len, const int32_t* target_row_offsets, int32_t* n_accepted,
                                 int32_t* correction_token, void* workspace, size_t ws_bytes, dspark_stream_t stream);

/*
 * Training-side accept-rate targets (P1 section 3.9 "Accept rate 3D", P2 section 3.5) and the
 * prefix-validity mask (P1 sections 3.6 and 3.10):
 *   acc[s,a,i] = clamp(1 - 0.5 sum_v |softmax(d)_v - softmax(t)_v|, 0, 1) = clamp(sum_v min(p_v, q_v))
 *     with softmax over fp32 logits and no temperature;
 *   eval_mask[s,a,i] = prod_{k<=i} (block_keep[s,a] != 0 && pos_valid[s,a,k] != 0)   (cumprod)
 *   tau[s,a] = 1 + sum_i prod_{k<=i} acc[s,a,k] * eval_mask[s,a,k]   (optional)
 * Arguments
 *   draft_logits, target_logits [S, A, gamma, V] (dtype); block_keep [S, A] uint8;
 *   pos_valid [S, A, gamma] uint8 or NULL (all valid).
 * Outputs
 *   accept_rate, eval_mask [S, A, gamma] float; tau [S, A] float or NULL.
 */
size_t dspark_accept_rate_tv_workspace_size(int S, int A, int gamma, int V, int dtype);
dspark_status dspark_accept_rate_tv(int S, int A, int gamma, int V, int dtype, const void* draft_logits,
                                    const void* target_logits, const uint8_t* block_keep, const uint8_t* pos_valid,
                                    float* accept_rate, float* eval_mask, float* tau, void* workspace,
                                    size_t ws_bytes, dspark_stream_t stream);

/*
 * Confidence-scheduled verify length (P3 section "置信度调度与验证截断":
 *   max_{L} sum_j sum_{i<=L_j} c~_{t+i}^{(j)},  1 <= L_j <= gamma, under a latency SLA;
 * survival a_k = prod_{i<=k} c_i, P2 section 3.8.3).  The SLA is a total verify-token budget:
 *   sum_j L_j <= budget.
 *   c is clamped to [0, 1] (NaN -> 0); a_{j,i} = prod_{k<=i} c_{j,k}, formed left to right in fp32.
 *   Each request verifies one token; the remaining budget - B slots go to the largest a_{j,i}
 *   with i >= 2, ordered by (a desc, j asc, i asc).  Since a is non-increasing along i the choice
 *   is prefix-closed and optimal.
 * Arguments
 *   conf [B, gamma] float: conditional confidences c_{j,i}; budget: total verify tokens.
 * Outputs
 *   verify_len [B] int32; offsets [B+1] int32 = exclusive prefix sum of verify_len (CSR of the
 *   flattened verify-token list); objective [1] float (sum of the chosen a) or NULL.
 * Host errors: DSPARK_ERR_BUDGET when budget < B; DSPARK_ERR_UNSUPPORTED when B * gamma > 16384.
 */
size_t dspark_schedule_workspace_size(int B, int gamma);
dspark_status dspark_schedule_verify_len(int B, int gamma, const float* conf, int budget, int32_t* verify_len,
                                         int32_t* offsets, float* objective, void* workspace, size_t ws_bytes,
                                         dspark_stream_t stream);

/*
 * Training-side L1 term on the accept rates (page "03 · DSpark 建模：Markov 与 Confidence",
 * section 3.9, the three weighted loss terms; the L1 / TV loss l1_dist = sum_v |softmax(d) -
 * softmax(t)|, with the position weights w_k = exp(-(k-1)/loss_decay_gamma)).  Per position
 * (s, a, k), k = 1..gamma:
 *   l1 = 2 (1 - accept_rate)          (sum |p - q| = 2 (1 - sum min(p, q)))
 *   sums[0] = sum w_k eval_mask l1,   sums[1] = sum w_k eval_mask
 * The two sums are returned apart so that ranks can add them before dividing.  Another page writes
 * the weight as e^(-k/gamma); the page that cites the loss code writes k-1, which is used here.
 * Arguments (device memory): accept_rate, eval_mask [S, A, gamma] float (dspark_accept_rate_tv's
 * outputs); decay_gamma > 0 (the pages use 4).
 * Outputs (device memory): l1 [S, A, gamma] float or NULL; sums [2] double.
 * Host errors: DSPARK_ERR_INVALID_ARG (sizes < 1, NULL accept_rate / eval_mask / sums,
 * decay_gamma <= 0), DSPARK_ERR_UNSUPPORTED when gamma > 1024.
 * The sums are added in a fixed order: the same inputs give the same bits.
 * Precision: l1 is formed from the fp32 accept rate, so its absolute error is twice the accept
 * rate's (at most 2 (1e-5 accept + 2^-24) against an exact sum |p - q|); as the accept rate tends
 * to 1 that error is a growing fraction of the small l1 itself.
 */
dspark_status dspark_tv_l1_loss(int S, int A, int gamma, const float* accept_rate, const float* eval_mask,
                                float decay_gamma, float* l1, double* sums, dspark_stream_t stream);

/*
 * Teacher-forced block logits of the Markov head (page "03 · DSpark 建模：Markov 与 Confidence",
 * build_markov_head / VanillaMarkov, Eq. 5; apply_block_logits): at training time every position's
 * bias comes from its true previous token, all positions at once:
 *   z[j, i, :] = base[j, i, :] + W2 W1[prev_{j,i}],  prev_{j,0} = anchor[j],  prev_{j,i} = tokens[j, i-1].
 * The same bias and add as dspark_markov_sample_block (params p: B, gamma, V, r, dtypes; T and
 * seed are not used), without the draw.
 * Arguments (device memory): base_logits [B, gamma, V] (logits_dtype); W1 [V, r], W2 [V, r]
 * (w_dtype); anchor [B] int32; tokens [B, gamma] int32 (the true tokens; column gamma-1 is not read).
 * Output: z_out [B, gamma, V] float32 (caller-owned).
 * Workspace: dspark_markov_block_logits_workspace_size(p) bytes, 256-byte aligned.  A previous token
 * outside [0, V) is clamped and recorded as DSPARK_ERR_TOKEN_RANGE in the workspace status.
 */
size_t dspark_markov_block_logits_workspace_size(const dspark_sample_params* p);
dspark_status dspark_markov_block_logits(const dspark_sample_params* p, const void* base_logits, const void* W1,
                                         const void* W2, const int32_t* anchor, const int32_t* tokens, float* z_out,
                                         void* workspace, size_t ws_bytes, dspark_stream_t stream);

/*
 * Throughput-aware prefix choice with a causal stop (page "DSpark 深度解读：DeepSeek-V4 如何用
 * 「半自回归」把推理速度提升 85%", section 5.1, 调度核心: 应该验证多少 token?), per request j:
 *   a_k = prod_{i<=k} c_{j,i},   Theta_l = (1 + sum_{k<=l} a_k) * SPS(l + 1),   l = 0 .. gamma,
 * searched from l = 0 upwards; the search stops at the first l with Theta_l < Theta_{l-1} and
 * chooses l - 1 (gamma when it never stops).  The page's worked example prints conditional
 * confidences as a_1, a_2; its Theta_2 holds only with a_2 = c_1 c_2, so a_k is the running
 * product.  Everything is computed in IEEE single precision, one rounding per multiply and per
 * add in the order above (no fused operations), so the choice is reproducible bit for bit.
 * Arguments (device memory)
 *   conf [B, gamma] float: conditional confidences, used as given (no clamping);
 *   sps [gamma + 1] float: SPS(1) .. SPS(gamma + 1), the throughput profile for a verify of
 *   l + 1 tokens, shared by the batch.
 * Outputs (device memory)
 *   ell [B] int32 in [0, gamma]; theta [B, gamma + 1] float or NULL: Theta_0 .. Theta_l as far as
 *   the search evaluated them, NaN after.
 * Host errors: DSPARK_ERR_INVALID_ARG for B < 1, gamma < 1 or a NULL conf / sps / ell.
 * No workspace and no device-side errors.
 */
dspark_status dspark_theta_schedule(int B, int gamma, const float* conf, const float* sps, int32_t* ell,
                                    float* theta, dspark_stream_t stream);

/*
 * Draft sampling without any allocation by the caller.  (No counterpart on the pages: this is a
 * convenience of this library.)  Some callers cannot call cudaMalloc at all -- for instance a
 * plug-in running inside a serving process whose device memory is owned by someone else's
 * pool, or a loop that must not allocate after start-up because an allocation can synchronise
 * the device -- and so cannot provide the workspace that dspark_markov_sample_block needs.
 * This variant runs the same kernel with its scratch in a fixed array that the library keeps
 * in device memory (a file-scope __device__ array of DSPARK_NOALLOC_SCRATCH_BYTES, present on
 * every GPU that loads the library until the process exits).  The caller still passes every
 * input and output, exactly as for dspark_markov_sample_block.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current; make that first call before any stream capture.  The address
 *     is kept for the life of the process: after cudaDeviceReset (or anything else that unloads
 *     the library's module from the device) it is stale, so reload the library before calling
 *     this entry point again.
 *   - A call whose scratch would exceed the array (dspark_sample_workspace_size(p) >
 *     DSPARK_NOALLOC_SCRATCH_BYTES) returns DSPARK_ERR_UNSUPPORTED and enqueues nothing.
 *   - All calls share the one array and it keeps the last call's contents; each call clears
 *     the part that must start at zero.  Calls that can overlap on the GPU (other streams,
 *     other host threads) race on the array: serialise them.
 *   - Device-side errors land in the shared array's status word, which is not exposed; use
 *     dspark_markov_sample_block when the device status is needed.
 */
#define DSPARK_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
dspark_status dspark_markov_sample_block_noalloc(const dspark_sample_params* p, const void* base_logits,
                                                 const void* W1, const void* W2, const int32_t* anchor,
                                                 int32_t* tokens, float* draft_lse, float* draft_logit_at_tok,
                                                 dspark_stream_t stream);

/* Reads the device status word of `workspace` after synchronising `stream`
 * (DSPARK_OK when no device-side error was recorded).  `workspace` is a device pointer;
 * `out` is a host pointer. */
dspark_status dspark_get_device_status(const void* workspace, dspark_stream_t stream, int32_t* out);

/* Upper bound, in nanoseconds, on every grid-wide wait inside the kernels (default 2e9).
 * A wait that exceeds it records DSPARK_ERR_TIMEOUT and its kernel returns early.
 * Process-wide; affects launches made after the call. */
void dspark_set_wait_limit_ns(uint64_t ns);

/* Test support: launches `nblocks` co-resident blocks that meet at one grid-wide wait which
 * expects `nblocks + missing` arrivals.  With missing > 0 the wait cannot complete and must
 * give up after the wait limit, recording DSPARK_ERR_TIMEOUT in the workspace status word.
 * Needs a workspace of dspark_sample_workspace_size-style header size (256 bytes). */
dspark_status dspark_selftest_grid_wait(int nblocks, int missing, void* workspace, size_t ws_bytes,
                                        dspark_stream_t stream);

const char* dspark_status_string(dspark_status s);

/* Number of kernels the library has enqueued in this process so far (all devices and streams;
 * an entry point that returns an error may have enqueued some).  For counting launches around a
 * region: read it before and after. */
uint64_t dspark_kernel_launches(void);

#ifdef __cplusplus
}
#endif
#endif /* DSPARK_H */
