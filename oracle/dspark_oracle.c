/*
 * dspark_oracle.c -- plain, slow, single-threaded CPU oracle for the DSpark
 * vocabulary-wide hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file.  The product path (the CUDA
 * library) never calls it, shares no code, header, table or helper with it, and
 * must fail loudly when its own extension is missing.
 *
 * Every quantity is computed in IEEE double from inputs converted exactly from
 * their stored type (fp32 or bf16), in the order the method states, with no
 * blocking, fusion or reordering.  The one exception is the verify-length
 * scheduler, whose survival products are formed in fp32 on purpose: there the
 * floating-point value decides an integer (which prefix tokens are selected),
 * and both sides take that decision in the kernel's precision.
 *
 * Sources (web pages about DSpark; "P1".."P4" below):
 *   P1  "03 · DSpark 建模：Markov 与 Confidence"
 *   P2  "从 DFlash 到 dLLM Self-Spec（三）：DSpark 的半自回归 Draft 与负载感知 Verify"
 *   P3  "如何评价 DeepSeek 发布 DSpark？哪些亮点值得关注？" (reading notes)
 *   P4  "DSpark 深度解读：DeepSeek-V4 如何用「半自回归」把推理速度提升 85%"
 * Random numbers: Philox4x32-10 from its published definition (Salmon, Moraes,
 * Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011).
 *
 * Pins (checked by the CPU test-suite): Philox known-answer vectors, closed
 * forms (sum-min = 1 - TV, residual + accepted mass = target), direct checks of
 * the tile / chunk / id inverse CDFs, chi-square of every sampler on V=8, brute force for the scheduler, exact enumeration of the
 * accepted-length law, and the worked example of the throughput-aware Theta
 * scheduler (P4 section 5.1).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1

/* Purposes: the fourth Philox counter word.  Which random draw is which. */
#define OR_P_SAMPLE_CHUNK 1
#define OR_P_SAMPLE_INCHUNK 2
#define OR_P_ACCEPT 3
#define OR_P_RESID_CHUNK 4
#define OR_P_RESID_INCHUNK 5
#define OR_P_BONUS_CHUNK 6
#define OR_P_BONUS_INCHUNK 7
#define OR_P_ELEM_GUMBEL 8

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (SC'11, section 4.2): ten rounds of two 32x32->64     */
/* multiplies whose halves are xored with the other counter words and  */
/* the key; the key is bumped by two Weyl constants between rounds.    */
/* ------------------------------------------------------------------ */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u; /* golden ratio */
            k1 += 0xBB67AE85u; /* sqrt(3) - 1 */
        }
        uint64_t prod_a = (uint64_t)0xD2511F53u * (uint64_t)x0;
        uint64_t prod_b = (uint64_t)0xCD9E8D57u * (uint64_t)x2;
        uint32_t hi_a = (uint32_t)(prod_a >> 32), lo_a = (uint32_t)prod_a;
        uint32_t hi_b = (uint32_t)(prod_b >> 32), lo_b = (uint32_t)prod_b;
        uint32_t y0 = hi_b ^ x1 ^ k0;
        uint32_t y1 = lo_b;
        uint32_t y2 = hi_a ^ x3 ^ k1;
        uint32_t y3 = lo_a;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* The shared randomness contract.  key = (lo32 seed, hi32 seed), counter =
 * (n / 4, i, j, purpose), output word n mod 4, mapped to the open interval
 * (0,1) as (floor(x / 2^9) + 1/2) * 2^-23: 2^23 equally spaced values that are
 * exact in fp32, never 0 and never 1. */
uint32_t oracle_philox_word(uint64_t seed, uint32_t j, uint32_t i, uint32_t purpose, uint32_t n) {
    uint32_t ctr[4] = {n >> 2, i, j, purpose};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return out[n & 3u];
}

double oracle_uniform(uint64_t seed, uint32_t j, uint32_t i, uint32_t purpose, uint32_t n) {
    uint32_t x = oracle_philox_word(seed, j, i, purpose, n);
    return ((double)(x >> 9) + 0.5) * (1.0 / 8388608.0);
}

/* ------------------------------------------------------------------ */
/* Input access                                                        */
/* ------------------------------------------------------------------ */
static double load_val(const void* p, int dtype, size_t idx) {
    if (dtype == OR_F32) return (double)((const float*)p)[idx];
    uint32_t bits = ((uint32_t)((const uint16_t*)p)[idx]) << 16; /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* Markov head (P1 section 3.7 VanillaMarkov; P2 section 3.4):         */
/*   bias = W2(W1[prev]),  W1 = Embedding(V, r), W2 = Linear(r, V)     */
/* W1 and W2 are both stored [V, r] row-major (W2 is nn.Linear.weight).*/
/*   z_v = base_v + sum_k W1[prev, k] * W2[v, k]                       */
/* r = 0 is the DFlash degenerate configuration (P1 section 3.13): no   */
/* bias.                                                                */
/* ------------------------------------------------------------------ */
void oracle_markov_logits(int V, int r, int logits_dtype, int w_dtype, const void* base_row,
                          const void* W1, const void* W2, int prev, double softcap, double* z_out) {
    for (int v = 0; v < V; ++v) {
        double bias = 0.0;
        for (int k = 0; k < r; ++k)
            bias += load_val(W1, w_dtype, (size_t)prev * r + k) * load_val(W2, w_dtype, (size_t)v * r + k);
        double b = load_val(base_row, logits_dtype, (size_t)v);
        /* final-logit softcap of the draft model's logits (P1 section 3.12): s tanh(b / s), before
         * the Markov bias is added; softcap = 0: none */
        if (softcap > 0.0) b = softcap * tanh(b / softcap);
        z_out[v] = b + bias;
    }
}

/* Greedy (temperature 0): argmax, lowest index on ties.  Margin = gap between
 * the winner and the best other index. */
int oracle_argmax(const double* z, int V, double* margin) {
    int best = 0;
    for (int v = 1; v < V; ++v)
        if (z[v] > z[best]) best = v;
    double second = -INFINITY;
    for (int v = 0; v < V; ++v)
        if (v != best && z[v] > second) second = z[v];
    if (margin) *margin = (V > 1) ? z[best] - second : INFINITY;
    return best;
}

static double logsumexp(const double* lw, int n) {
    double m = -INFINITY;
    for (int v = 0; v < n; ++v)
        if (lw[v] > m) m = lw[v];
    if (m == -INFINITY) return -INFINITY;
    double s = 0.0;
    for (int v = 0; v < n; ++v) s += exp(lw[v] - m);
    return m + log(s);
}

/* Exponential variate E = -ln U for the race between chunks. */
static double neg_log_u(double u) { return -log(u); }

/* In-order inverse CDF of u over n log-weights normalised by lse: the smallest k whose cumulative
 * mass exceeds u; where rounding leaves no crossing, the last k with mass.  *margin = distance of u
 * to the CDF boundaries around k. */
static int inverse_cdf(const double* lw, int n, double lse, double u, double* margin) {
    double cum = 0.0, prev_cum = 0.0;
    int last_nz = -1;
    for (int k = 0; k < n; ++k) {
        double w = exp(lw[k] - lse);
        if (w > 0.0) last_nz = k;
        prev_cum = cum;
        cum += w;
        if (cum > u) {
            double a = u - prev_cum, b = cum - u;
            *margin = a < b ? a : b;
            return k;
        }
    }
    *margin = 0.0; /* rounding left the total below u */
    return last_nz;
}

/* ------------------------------------------------------------------ */
/* Chunk-Gumbel categorical sampler over log-weights lw[0..V): the     */
/* contract of every draw, the draft sampler's and verify's residual   */
/* and bonus corrections (the body of sample_tokens is not shown, P2   */
/* section 3.4; any exact categorical draw is lossless).               */
/*   chunks of CS consecutive ids over the whole vocabulary (the last  */
/*   one may be short); LSE_c = log sum_{v in c} e^lw_v;               */
/*   c* = argmax_c LSE_c - ln E_c, E_c = -ln U(.., p_chunk, c), lowest */
/*   c on ties; chunks without mass never win;                         */
/*   x  = smallest id of c* whose in-order cumulative mass             */
/*   sum_{w<=v} e^(lw_w - LSE_c*) exceeds u = U(.., p_inchunk, 0);     */
/*   where rounding leaves no crossing, the last id with mass.         */
/* Gumbel-max over chunks gives P(c) proportional to e^LSE_c; u is     */
/* independent of the race, so P(v | c) is proportional to e^lw_v and  */
/* the product is softmax(lw).  Returns x (-1 when nothing has mass);  */
/* *lse_all = log-sum-exp of all lw; *margin = min(chunk-key gap,      */
/* distance of u to the id CDF boundaries around x).                   */
/* ------------------------------------------------------------------ */
int oracle_chunk_gumbel(const double* lw, int V, int CS, uint64_t seed, int j, int i, int p_chunk, int p_inchunk,
                        double* margin, double* lse_all) {
    int nc = (V + CS - 1) / CS;
    double* lse_c = (double*)malloc(sizeof(double) * (size_t)nc);
    for (int c = 0; c < nc; ++c) {
        int lo = c * CS, n = (lo + CS <= V) ? CS : V - lo;
        lse_c[c] = logsumexp(lw + lo, n);
    }
    if (lse_all) *lse_all = logsumexp(lse_c, nc);
    int best = -1;
    double best_key = -INFINITY, second_key = -INFINITY;
    for (int c = 0; c < nc; ++c) {
        if (lse_c[c] == -INFINITY) continue;
        double key = lse_c[c] - log(neg_log_u(oracle_uniform(seed, (uint32_t)j, (uint32_t)i, (uint32_t)p_chunk, (uint32_t)c)));
        if (best < 0 || key > best_key) {
            if (best >= 0) second_key = best_key;
            best_key = key;
            best = c;
        } else if (key > second_key) {
            second_key = key;
        }
    }
    if (best < 0) {
        free(lse_c);
        if (margin) *margin = 0.0;
        return -1;
    }
    double u = oracle_uniform(seed, (uint32_t)j, (uint32_t)i, (uint32_t)p_inchunk, 0u);
    int lo = best * CS, n = (lo + CS <= V) ? CS : V - lo;
    double m_id;
    int k = inverse_cdf(lw + lo, n, lse_c[best], u, &m_id);
    if (margin) {
        double m_chunk = best_key - second_key; /* +inf when a single chunk has mass */
        *margin = m_chunk < m_id ? m_chunk : m_id;
    }
    free(lse_c);
    return lo + k;
}

/* Second sampler (reference for the chi-square test): per-element Gumbel-max,
 * x = argmax_v lw_v - ln E_v with E_v = -ln U(.., p_elem, v). */
int oracle_gumbel_elem(const double* lw, int V, uint64_t seed, int j, int i, double* margin) {
    int best = -1;
    double bk = -INFINITY, sk = -INFINITY;
    for (int v = 0; v < V; ++v) {
        if (lw[v] == -INFINITY) continue;
        double key = lw[v] - log(neg_log_u(oracle_uniform(seed, (uint32_t)j, (uint32_t)i, OR_P_ELEM_GUMBEL, (uint32_t)v)));
        if (best < 0 || key > bk) {
            if (best >= 0) sk = bk;
            bk = key;
            best = v;
        } else if (key > sk) {
            sk = key;
        }
    }
    if (margin) *margin = bk - sk;
    return best;
}

/* ------------------------------------------------------------------ */
/* Block sampling for one request (P2 section 3.4, sample_block_tokens: */
/* prev = anchor; for each step: logits = base[step] + bias(prev);      */
/* sample; prev = sampled).  Temperature: T = 0 is greedy, T > 0 draws  */
/* from softmax(z / T).  Outputs per step: token, LSE(z/T) (NaN when    */
/* T = 0), z at the token, decision margin.                             */
/*   base_req: this request's [gamma, V] block of base logits;          */
/*   W1, W2: [V, r]; j: request index (selects the random stream).      */
/* ------------------------------------------------------------------ */
void oracle_sample_request(int V, int r, int gamma, int TS, int CS, double T, uint64_t seed, int logits_dtype,
                           int w_dtype, const void* base_req, const void* W1, const void* W2, int anchor, int j,
                           int32_t* tokens, double* draft_lse, double* z_at_tok, double* margin, double softcap) {
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    double* s = (double*)malloc(sizeof(double) * (size_t)V);
    size_t esz = (logits_dtype == OR_F32) ? 4 : 2;
    int prev = anchor;
    for (int step = 0; step < gamma; ++step) {
        int i = step + 1; /* 1-based block position */
        const char* row = (const char*)base_req + (size_t)step * (size_t)V * esz;
        oracle_markov_logits(V, r, logits_dtype, w_dtype, row, W1, W2, prev, softcap, z);
        int x;
        double mg, lse;
        if (T == 0.0) {
            x = oracle_argmax(z, V, &mg);
            lse = NAN;
        } else {
            for (int v = 0; v < V; ++v) s[v] = z[v] / T;
            x = oracle_chunk_gumbel(s, V, CS, seed, j, i, OR_P_SAMPLE_CHUNK, OR_P_SAMPLE_INCHUNK, &mg, &lse);
        }
        tokens[step] = x;
        draft_lse[step] = lse;
        z_at_tok[step] = z[x];
        margin[step] = mg;
        prev = x;
    }
    free(z);
    free(s);
}

/* ------------------------------------------------------------------ */
/* Lossless verification of one request (P3 "Speculative Decoding":    */
/* the target checks the K positions in parallel, accepts left to       */
/* right by rejection sampling, truncates at the first failure and      */
/* resamples from the target; the output law equals the target's).     */
/*   accept x_i iff u_i < p(x_i) / q(x_i), tested in the log domain:    */
/*   ln u_i < (t_x/T - LSE(t_i/T)) - (z_x/T - draft_lse_i)              */
/*   at the first rejection k: sample from norm(max(0, p_k - q_k));     */
/*   if every one of the L verified tokens is accepted and a target row */
/*   L+1 exists, the bonus token is drawn from p_{L+1}; else none (-1). */
/* T = 0: p and q are one-hot; accept iff argmax t_i == x_i; the        */
/* correction is argmax of the rejecting (or bonus) target row.         */
/* q over the whole vocabulary at the rejecting position is rebuilt     */
/* from base + bias(prev) and normalised by the given draft_lse; q at   */
/* the drafted token uses the given z_at_tok.                           */
/*   base_req: this request's [gamma, V] base block; target_req: its    */
/*   [gamma_t, V] target block; tokens, draft_lse, z_at_tok: its gamma  */
/*   entries; j selects the random stream.  Returns n accepted;          */
/*   *correction;                                                        */
/*   *min_margin over all decisions; *resid_fallback = 1 when the       */
/*   residual had no mass and p was used instead.                       */
/* ------------------------------------------------------------------ */
/* Gated and RNN Markov heads (P1 section 3.7, 三种 Markov head; P4    */
/* section 3.3): the vector u_k that W2 multiplies at draft step k,    */
/* from e = W1[x_{k-1}] (r), the backbone hidden state h_k (d) and,    */
/* for the RNN head, the state s_{k-1} (r, updated in place to s_k).   */
/*   gated: gate = sigmoid(Wg [h; e]),  u = gate * e                   */
/*          (Wg: r x (d + r), columns h then e)                        */
/*   rnn:   z = [s; e; h] (2r + d),  g = sigmoid(Wg z),                */
/*          s <- g * s + (1 - g) * tanh(Wc z),  u = tanh(Wo z)         */
/*          (Wg, Wc, Wo: r x (2r + d)); the bias uses z_k, which holds */
/*          s_{k-1}.  The initial state is zero (the pages give none). */
/* sigmoid(a) = 1 / (1 + exp(-a)).                                     */
/* ------------------------------------------------------------------ */
enum { OR_HEAD_VANILLA = 0, OR_HEAD_GATED = 1, OR_HEAD_RNN = 2 };

static double sigmoid(double a) { return 1.0 / (1.0 + exp(-a)); }

void oracle_head_vector(int kind, int r, int d, int dtype, const void* Wg, const void* Wc, const void* Wo,
                        const double* e, const void* h_row, double* s, double* u) {
    if (kind == OR_HEAD_GATED) {
        for (int i = 0; i < r; ++i) {
            double a = 0.0;
            for (int c = 0; c < d; ++c) a += load_val(Wg, dtype, (size_t)i * (d + r) + c) * load_val(h_row, dtype, c);
            for (int c = 0; c < r; ++c) a += load_val(Wg, dtype, (size_t)i * (d + r) + d + c) * e[c];
            u[i] = sigmoid(a) * e[i];
        }
        return;
    }
    if (kind == OR_HEAD_RNN) {
        const int w = 2 * r + d;
        double* z = (double*)malloc(sizeof(double) * (size_t)w);
        double* s_new = (double*)malloc(sizeof(double) * (size_t)r);
        for (int c = 0; c < r; ++c) z[c] = s[c];
        for (int c = 0; c < r; ++c) z[r + c] = e[c];
        for (int c = 0; c < d; ++c) z[2 * r + c] = load_val(h_row, dtype, c);
        for (int i = 0; i < r; ++i) {
            double ag = 0.0, ac = 0.0, ao = 0.0;
            for (int c = 0; c < w; ++c) {
                ag += load_val(Wg, dtype, (size_t)i * w + c) * z[c];
                ac += load_val(Wc, dtype, (size_t)i * w + c) * z[c];
                ao += load_val(Wo, dtype, (size_t)i * w + c) * z[c];
            }
            const double g = sigmoid(ag);
            s_new[i] = g * s[i] + (1.0 - g) * tanh(ac);
            u[i] = tanh(ao);
        }
        for (int i = 0; i < r; ++i) s[i] = s_new[i];
        free(z);
        free(s_new);
        return;
    }
    for (int i = 0; i < r; ++i) u[i] = e[i]; /* vanilla: u = W1[x] */
}

/* z_v = cap(base_v) + sum_i W2[v, i] u_i (the Markov logits with an explicit head vector). */
void oracle_head_logits(int V, int r, int logits_dtype, int w_dtype, const void* base_row, const double* u,
                        const void* W2, double softcap, double* z_out) {
    for (int v = 0; v < V; ++v) {
        double bias = 0.0;
        for (int k = 0; k < r; ++k) bias += load_val(W2, w_dtype, (size_t)v * r + k) * u[k];
        double b = load_val(base_row, logits_dtype, (size_t)v);
        if (softcap > 0.0) b = softcap * tanh(b / softcap);
        z_out[v] = b + bias;
    }
}

/* One request of the head sampler: as oracle_sample_request with the bias W2 u_k of the head
 * (hidden_req [gamma, d] in the head dtype); u_out [gamma, r] receives the head vectors. */
void oracle_sample_request_head(int V, int r, int gamma, int TS, int CS, double T, uint64_t seed, int logits_dtype,
                                int w_dtype, const void* base_req, const void* W1, const void* W2, int anchor, int j,
                                int kind, int d, const void* hidden_req, const void* Wg, const void* Wc,
                                const void* Wo, int32_t* tokens, double* draft_lse, double* z_at_tok, double* margin,
                                double* u_out, double softcap) {
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    double* sv = (double*)malloc(sizeof(double) * (size_t)V);
    double* e = (double*)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
    double* st = (double*)calloc((size_t)(r > 0 ? r : 1), sizeof(double));
    size_t esz = (logits_dtype == OR_F32) ? 4 : 2, hsz = (w_dtype == OR_F32) ? 4 : 2;
    int prev = anchor;
    for (int step = 0; step < gamma; ++step) {
        int i = step + 1;
        for (int c = 0; c < r; ++c) e[c] = load_val(W1, w_dtype, (size_t)prev * r + c);
        const char* hrow = (const char*)hidden_req + (size_t)step * (size_t)d * hsz;
        double* u = u_out + (size_t)step * r;
        oracle_head_vector(kind, r, d, w_dtype, Wg, Wc, Wo, e, hrow, st, u);
        const char* row = (const char*)base_req + (size_t)step * (size_t)V * esz;
        oracle_head_logits(V, r, logits_dtype, w_dtype, row, u, W2, softcap, z);
        int x;
        double mg, lse;
        if (T == 0.0) {
            x = oracle_argmax(z, V, &mg);
            lse = NAN;
        } else {
            for (int v = 0; v < V; ++v) sv[v] = z[v] / T;
            x = oracle_chunk_gumbel(sv, V, CS, seed, j, i, OR_P_SAMPLE_CHUNK, OR_P_SAMPLE_INCHUNK, &mg, &lse);
        }
        tokens[step] = x;
        draft_lse[step] = lse;
        z_at_tok[step] = z[x];
        margin[step] = mg;
        prev = x;
    }
    free(z);
    free(sv);
    free(e);
    free(st);
}

/* ------------------------------------------------------------------ */
int oracle_verify_request(int V, int r, int gamma, int gamma_t, int TS, int CS, double T, uint64_t seed,
                          int logits_dtype, int w_dtype, int target_dtype, const void* base_req, const void* W1,
                          const void* W2, int anchor, int j, const int32_t* tokens, const float* draft_lse,
                          const float* z_at_tok, const void* target_req, int L, int32_t* correction,
                          double* min_margin, int* resid_fallback, double softcap, const double* head_vec) {
    size_t tsz = (target_dtype == OR_F32) ? 4 : 2;
    size_t bsz = (logits_dtype == OR_F32) ? 4 : 2;
    (void)gamma; /* the per-request blocks are already sliced */
    double* tl = (double*)malloc(sizeof(double) * (size_t)V);
    double* lw = (double*)malloc(sizeof(double) * (size_t)V);
    double mm = INFINITY;
    int n = L;
    *correction = -1;
    if (resid_fallback) *resid_fallback = 0;
    for (int step = 0; step < L; ++step) {
        int i = step + 1;
        const char* trow = (const char*)target_req + (size_t)step * (size_t)V * tsz;
        for (int v = 0; v < V; ++v) tl[v] = load_val(trow, target_dtype, (size_t)v);
        int x = tokens[step];
        int accept;
        if (T == 0.0) {
            double mg;
            int am = oracle_argmax(tl, V, &mg);
            accept = (am == x);
            if (mg < mm) mm = mg;
        } else {
            for (int v = 0; v < V; ++v) lw[v] = tl[v] / T;
            double lse_t = logsumexp(lw, V);
            double lnp = tl[x] / T - lse_t;
            double lnq = (double)z_at_tok[step] / T - (double)draft_lse[step];
            double lnu = log(oracle_uniform(seed, (uint32_t)j, (uint32_t)i, OR_P_ACCEPT, 0u));
            double d = lnu - (lnp - lnq);
            accept = d < 0.0;
            if (fabs(d) < mm) mm = fabs(d);
        }
        if (!accept) {
            n = step;
            if (T == 0.0) {
                *correction = oracle_argmax(tl, V, NULL);
            } else {
                /* residual norm(max(0, p - q)) at position i */
                int prev = (step == 0) ? anchor : tokens[step - 1];
                const char* brow = (const char*)base_req + (size_t)step * (size_t)V * bsz;
                double* z = (double*)malloc(sizeof(double) * (size_t)V);
                if (head_vec) /* a Gated / RNN head: the draft's own head vector of this position */
                    oracle_head_logits(V, r, logits_dtype, w_dtype, brow, head_vec + (size_t)step * r, W2, softcap, z);
                else
                    oracle_markov_logits(V, r, logits_dtype, w_dtype, brow, W1, W2, prev, softcap, z);
                double lse_t = logsumexp(lw, V); /* lw still holds t/T of this row */
                int any = 0;
                for (int v = 0; v < V; ++v) {
                    double p = exp(lw[v] - lse_t);
                    double q = exp(z[v] / T - (double)draft_lse[step]);
                    double rv = p - q;
                    z[v] = rv > 0.0 ? log(rv) : -INFINITY; /* reuse z as residual log-weights */
                    if (rv > 0.0) any = 1;
                }
                double mg;
                if (any) {
                    *correction = oracle_chunk_gumbel(z, V, CS, seed, j, i, OR_P_RESID_CHUNK, OR_P_RESID_INCHUNK, &mg, NULL);
                } else { /* p == q everywhere yet a float rejection: fall back to p */
                    if (resid_fallback) *resid_fallback = 1;
                    *correction = oracle_chunk_gumbel(lw, V, CS, seed, j, i, OR_P_RESID_CHUNK, OR_P_RESID_INCHUNK, &mg, NULL);
                }
                if (mg < mm) mm = mg;
                free(z);
            }
            break;
        }
    }
    if (n == L && gamma_t > L) { /* bonus token from target row L+1 */
        int i = L + 1;
        const char* trow = (const char*)target_req + (size_t)L * (size_t)V * tsz;
        for (int v = 0; v < V; ++v) tl[v] = load_val(trow, target_dtype, (size_t)v);
        double mg;
        if (T == 0.0) {
            *correction = oracle_argmax(tl, V, &mg);
        } else {
            for (int v = 0; v < V; ++v) lw[v] = tl[v] / T;
            *correction = oracle_chunk_gumbel(lw, V, CS, seed, j, i, OR_P_BONUS_CHUNK, OR_P_BONUS_INCHUNK, &mg, NULL);
        }
        if (mg < mm) mm = mg;
    }
    if (min_margin) *min_margin = mm;
    free(tl);
    free(lw);
    return n;
}

/* ------------------------------------------------------------------ */
/* Accept-rate target (P1 section 3.9 "Accept rate 3D"; P2 section 3.5):*/
/*   p = softmax(target), q = softmax(draft), no temperature,           */
/*   acc = clamp(1 - 0.5 * sum|p - q|, 0, 1) = clamp(sum min(p, q)).    */
/* Returns sum-min (no cancellation); *one_minus_tv = 1 - 0.5 sum|p-q|. */
/* ------------------------------------------------------------------ */
double oracle_tv_row(int V, int dtype, const void* d_row, const void* t_row, double* one_minus_tv) {
    double* a = (double*)malloc(sizeof(double) * (size_t)V);
    double* b = (double*)malloc(sizeof(double) * (size_t)V);
    for (int v = 0; v < V; ++v) {
        a[v] = load_val(d_row, dtype, (size_t)v);
        b[v] = load_val(t_row, dtype, (size_t)v);
    }
    double la = logsumexp(a, V), lb = logsumexp(b, V);
    double smin = 0.0, sabs = 0.0;
    for (int v = 0; v < V; ++v) {
        double q = exp(a[v] - la), p = exp(b[v] - lb);
        smin += (p < q) ? p : q;
        sabs += fabs(p - q);
    }
    if (one_minus_tv) *one_minus_tv = 1.0 - 0.5 * sabs;
    free(a);
    free(b);
    if (smin < 0.0) smin = 0.0;
    if (smin > 1.0) smin = 1.0;
    return smin;
}

/* eval_mask and tau for one block (P1 sections 3.6 and 3.10):
 *   valid_i = keep && pos_valid_i (pos_valid NULL = all valid)
 *   mask_i = prod_{k<=i} valid_k      (cumprod: zero after the first zero)
 *   tau = 1 + sum_i prod_{k<=i} acc_k * mask_k */
double oracle_eval_mask_tau(int gamma, int keep, const uint8_t* pos_valid, const double* acc, double* mask) {
    double run = 1.0, prod = 1.0, expected = 0.0;
    for (int i = 0; i < gamma; ++i) {
        double valid = (keep && (pos_valid == NULL || pos_valid[i])) ? 1.0 : 0.0;
        run *= valid;
        mask[i] = run;
        prod *= acc[i] * mask[i];
        expected += prod;
    }
    return 1.0 + expected;
}

/* ------------------------------------------------------------------ */
/* Verify-length selection under a token budget (P3 section             */
/* "置信度调度与验证截断": max sum_j sum_{i<=L_j} c~_{t+i}^(j), 1 <= L_j */
/* <= K; the SLA constraint is read as sum_j L_j <= budget; survival is */
/* a product of conditional confidences, P2 section 3.8.3).             */
/*   c is clamped to [0,1] (NaN -> 0); a_{j,i} = prod_{k<=i} c_{j,k}     */
/*   formed left to right in double.  Every request verifies one token; */
/*   the remaining budget - B slots go to the largest a_{j,i}, i >= 2,  */
/*   ordered by (a desc, j asc, i asc).  Because c <= 1, a is           */
/*   non-increasing along i, so the chosen set is prefix-closed and the */
/*   greedy choice is optimal (concave gains).  budget < B: returns -1. */
/*   *margin = a of the last taken key minus a of the first key left    */
/*   out (infinite when nothing is left out or nothing is taken).       */
/* ------------------------------------------------------------------ */
typedef struct {
    double a;
    long idx; /* j * gamma + i */
} sched_key;

static int cmp_sched_key(const void* pa, const void* pb) {
    const sched_key* x = (const sched_key*)pa;
    const sched_key* y = (const sched_key*)pb;
    if (x->a > y->a) return -1;
    if (x->a < y->a) return 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

int oracle_schedule(int B, int gamma, const float* conf, int budget, int32_t* L, int32_t* offsets,
                    double* objective, double* margin) {
    if (budget < B) return -1;
    double* a = (double*)malloc(sizeof(double) * (size_t)B * gamma);
    for (int j = 0; j < B; ++j) {
        double run = 1.0;
        for (int i = 0; i < gamma; ++i) {
            double c = (double)conf[(size_t)j * gamma + i];
            if (!(c >= 0.0)) c = 0.0; /* also NaN */
            if (c > 1.0) c = 1.0;
            run = run * c;
            a[(size_t)j * gamma + i] = run;
        }
    }
    long extra = (long)budget - B;
    long cand = (long)B * (gamma - 1);
    if (extra > cand) extra = cand;
    sched_key* keys = (sched_key*)malloc(sizeof(sched_key) * (size_t)(cand > 0 ? cand : 1));
    long nk = 0;
    for (int j = 0; j < B; ++j)
        for (int i = 1; i < gamma; ++i) {
            keys[nk].a = a[(size_t)j * gamma + i];
            keys[nk].idx = (long)j * gamma + i;
            ++nk;
        }
    qsort(keys, (size_t)nk, sizeof(sched_key), cmp_sched_key);
    for (int j = 0; j < B; ++j) L[j] = 1;
    for (long k = 0; k < extra; ++k) L[keys[k].idx / gamma] += 1;
    if (margin) *margin = (extra > 0 && extra < nk) ? keys[extra - 1].a - keys[extra].a : INFINITY;
    double obj = 0.0;
    offsets[0] = 0;
    for (int j = 0; j < B; ++j) {
        for (int i = 0; i < L[j]; ++i) obj += a[(size_t)j * gamma + i];
        offsets[j + 1] = offsets[j] + L[j];
    }
    if (objective) *objective = obj;
    free(a);
    free(keys);
    return 0;
}

/* Throughput-aware prefix choice (P4 section 5.1):
 *   Theta_l = (1 + sum_{k<=l} a_k) * SPS(l + 1),  a_k = prod_{i<=k} c_i,
 * searched causally from l = 0, stopping at the first l with
 * Theta_l < Theta_{l-1}; returns that l - 1 (or gamma when it never stops).
 * theta_out receives Theta_0..Theta_gamma as far as they were evaluated (NaN
 * after).  Computed in double.  *margin = the smallest relative gap
 * |Theta_l - Theta_{l-1}| / max(|Theta_l|, |Theta_{l-1}|) over the
 * comparisons the search made (infinite when gamma = 0): a comparison whose
 * gap is below rounding could go either way in a lower precision. */
int oracle_theta_schedule(int gamma, const double* c, const double* sps, double* theta_out, double* margin) {
    double a = 1.0, acc = 0.0, prev = -INFINITY, mg = INFINITY;
    for (int l = 0; l <= gamma; ++l) theta_out[l] = NAN;
    for (int l = 0; l <= gamma; ++l) {
        if (l > 0) {
            a = a * c[l - 1];
            acc = acc + a;
        }
        const double th = (1.0 + acc) * sps[l];
        theta_out[l] = th;
        if (l > 0) {
            const double den = fmax(fabs(th), fabs(prev));
            const double gap = den > 0.0 ? fabs(th - prev) / den : 0.0;
            if (gap < mg) mg = gap;
            if (th < prev) {
                if (margin) *margin = mg;
                return l - 1;
            }
        }
        prev = th;
    }
    if (margin) *margin = mg;
    return gamma;
}

/* ------------------------------------------------------------------ */
/* Trial loops for the chi-square pins (thin drivers of the above).    */
/* ------------------------------------------------------------------ */
/* variant 0: chunk-Gumbel with chunk size CS and the residual purposes (verify's corrections);
 * 1: per-element Gumbel-max; 2: chunk-Gumbel with chunk size CS and the sampling purposes (the
 * draft sampler).  Trial n uses request index j = n, position i = 1. */
void oracle_trials_sampler(int V, int CS, const double* lw, uint64_t seed, long ntrials, int variant,
                           int64_t* counts) {
    for (int v = 0; v < V; ++v) counts[v] = 0;
    for (long n = 0; n < ntrials; ++n) {
        int x = variant == 0   ? oracle_chunk_gumbel(lw, V, CS, seed, (int)n, 1, OR_P_RESID_CHUNK, OR_P_RESID_INCHUNK, NULL, NULL)
                : variant == 1 ? oracle_gumbel_elem(lw, V, seed, (int)n, 1, NULL)
                               : oracle_chunk_gumbel(lw, V, CS, seed, (int)n, 1, OR_P_SAMPLE_CHUNK, OR_P_SAMPLE_INCHUNK, NULL, NULL);
        counts[x] += 1;
    }
}

/* One speculative position per trial on V-sized fp32 logits (r = 0, one
 * position, no bonus row): draft x ~ softmax(zd/T) by the chunk sampler, verify
 * against softmax(zt/T); counts the emitted token (x if accepted, else the
 * residual draw) and the number of acceptances. */
void oracle_trials_spec_one(int V, int TS, int CS, double T, const float* zd, const float* zt, uint64_t seed, long ntrials,
                            int64_t* emitted, int64_t* n_accept) {
    double* s = (double*)malloc(sizeof(double) * (size_t)V);
    for (int v = 0; v < V; ++v) s[v] = (double)zd[v] / T;
    double lse_d = logsumexp(s, V);
    *n_accept = 0;
    for (int v = 0; v < V; ++v) emitted[v] = 0;
    for (long n = 0; n < ntrials; ++n) {
        int32_t x = oracle_chunk_gumbel(s, V, CS, seed, (int)n, 1, OR_P_SAMPLE_CHUNK, OR_P_SAMPLE_INCHUNK, NULL, NULL);
        float lse_f = (float)lse_d, zx_f = zd[x];
        int32_t corr;
        int nacc = oracle_verify_request(V, 0, 1, 1, TS, CS, T, seed, OR_F32, OR_F32, OR_F32, zd, NULL, NULL, 0, (int)n,
                                         &x, &lse_f, &zx_f, zt, 1, &corr, NULL, NULL, 0.0, NULL);
        if (nacc == 1) {
            emitted[x] += 1;
            *n_accept += 1;
        } else {
            emitted[corr] += 1;
        }
    }
    free(s);
}

/* One whole draft block + verification per trial (fp32 data, one request's
 * block base_req [gamma, V], target_req [gamma, V], W1/W2 [V, r] fp32):
 * trial n draws with request id n.  hist[k] counts trials with k accepted
 * tokens (k = 0..gamma). */
void oracle_trials_spec_block(int V, int r, int gamma, int TS, int CS, double T, const float* base_req, const float* W1,
                              const float* W2, int anchor, const float* target_req, uint64_t seed, long ntrials,
                              int64_t* hist) {
    int32_t* tok = (int32_t*)malloc(sizeof(int32_t) * (size_t)gamma);
    double* lse = (double*)malloc(sizeof(double) * (size_t)gamma);
    double* zx = (double*)malloc(sizeof(double) * (size_t)gamma);
    double* mg = (double*)malloc(sizeof(double) * (size_t)gamma);
    float* lse_f = (float*)malloc(sizeof(float) * (size_t)gamma);
    float* zx_f = (float*)malloc(sizeof(float) * (size_t)gamma);
    for (int k = 0; k <= gamma; ++k) hist[k] = 0;
    for (long n = 0; n < ntrials; ++n) {
        oracle_sample_request(V, r, gamma, TS, CS, T, seed, OR_F32, OR_F32, base_req, W1, W2, anchor, (int)n, tok, lse, zx, mg, 0.0);
        for (int i = 0; i < gamma; ++i) {
            lse_f[i] = (float)lse[i];
            zx_f[i] = (float)zx[i];
        }
        int32_t corr;
        int nacc = oracle_verify_request(V, r, gamma, gamma, TS, CS, T, seed, OR_F32, OR_F32, OR_F32, base_req, W1, W2,
                                         anchor, (int)n, tok, lse_f, zx_f, target_req, gamma, &corr, NULL, NULL, 0.0, NULL);
        hist[nacc] += 1;
    }
    free(tok); free(lse); free(zx); free(mg); free(lse_f); free(zx_f);
}
