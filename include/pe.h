/*
 * pe.h — C ABI of libpe.so: P-EAGLE parallel drafting and greedy
 * verify / batch-metadata rebuild on one GB300 (sm_103a).
 *
 * The method (cited by page title and section):
 *  - "在 Amazon SageMaker AI 上使用 P-EAGLE 并行化推测解码" (Chinese translation
 *    of the AWS post), section "解决方案概述" (Solution overview):
 *    "P-EAGLE 如何打破这个链" — learned placeholders emb_mask and h_shared;
 *    "逐步草稿过程" — Step 1: target hidden states of layers 2, L/2, L-1
 *    concatenated to 3d; Step 2: position 1 = real token embedding + target
 *    hidden, positions 2..K = emb_mask + h_shared, all K positions through
 *    the 4 drafter layers and the LM head in one pass, K drafts at once; the
 *    target then verifies all K in one pass with the standard acceptance rule.
 *  - "Amazon SageMaker AIにおけるP-EAGLEによる推論高速化": a fused kernel
 *    rebuilds the batch metadata after verification.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller unless stated
 *    otherwise; the library never frees them. Matrices are row-major,
 *    weight matrices are stored [out, in].
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *    asynchronous on that stream; outputs are valid once it reaches them.
 *  - The return value is PE_OK or a negative PE_ERR_* code; on error
 *    pe_last_error() (thread-local) describes it and nothing was enqueued.
 *  - Problems found on the device for one request (bad page index, cache
 *    capacity) are reported per request in `status[b]` (PE_REQ_*); other
 *    requests are unaffected. No kernel traps; every device-side wait is
 *    bounded and a wait that gives up sets a flag read by pe_device_errors().
 */
#ifndef PE_H
#define PE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PE_ABI_VERSION 1

/* return codes */
#define PE_OK               0
#define PE_ERR_ARG         -1   /* null pointer, size out of range, misaligned pointer */
#define PE_ERR_UNSUPPORTED -2   /* shape the kernels do not implement */
#define PE_ERR_CUDA        -3   /* a CUDA runtime / driver call failed */
#define PE_ERR_NOMEM       -4   /* workspace allocation failed */

/* per-request status written by pe_draft and pe_verify_rebuild */
#define PE_REQ_OK          0
#define PE_REQ_CAPACITY    1    /* entries needed exceed max_pages * page_size */
#define PE_REQ_BAD_PAGE    2    /* a needed page-table entry is outside [0, num_pages) */
#define PE_REQ_BAD_INPUT   3    /* token id outside [0, V), negative length */

/* bits of the device error word (pe_device_errors) */
#define PE_DEVERR_GEMM_TIMEOUT  1u
#define PE_DEVERR_ATTN_TIMEOUT  2u
#define PE_DEVERR_CHAIN_TIMEOUT 4u   /* the persistent layer-chain kernel */

#define PE_DTYPE_BF16 0         /* bf16 weights/activations/KV, fp32 accumulate */
#define PE_DTYPE_FP32 1         /* fp32 everything; GEMMs run as tf32 */
#define PE_DTYPE_FP8W 2         /* FP8 (E4M3) GEMM weights with one fp32 scale per output row;
                                   bf16 activations, embeddings, norm gains and KV cache
                                   (pe_init_drafter_fp8) */

/* Drafter shape. n_layers must be 4, page_size 16, head_dim 64 or 128,
 * n_kv_heads must divide n_q_heads, n_q_heads*head_dim and
 * n_kv_heads*head_dim must be multiples of 128, hidden and ffn multiples
 * of 64. k_max (1..16) is the largest K any call will pass. */
typedef struct pe_config {
    int32_t hidden;       /* H */
    int32_t n_layers;     /* 4 */
    int32_t n_q_heads;    /* nq */
    int32_t n_kv_heads;   /* nkv */
    int32_t head_dim;     /* hd */
    int32_t ffn;          /* F (SwiGLU width) */
    int32_t vocab;        /* V */
    float   rms_eps;      /* RMSNorm epsilon */
    float   rope_theta;   /* RoPE base */
    int32_t page_size;    /* 16 */
    int32_t k_max;        /* largest K a call may pass */
    int32_t dtype;        /* PE_DTYPE_* for weights, activations and KV cache */
} pe_config;

/* Per-layer weights, all of the config dtype, device pointers, 16-byte aligned. */
typedef struct pe_layer_weights {
    const void* norm_e;     /* [H]  layer 0 only: gain of RMSNorm on the token embedding half */
    const void* norm_h;     /* [H]  layer 0 only: gain of RMSNorm on the hidden half */
    const void* attn_norm;  /* [H]  layers 1..3: pre-attention RMSNorm gain (NULL for layer 0) */
    const void* w_qkv;      /* [(nq+2nkv)*hd, in], in = 2H for layer 0, H otherwise; rows q | k | v */
    const void* w_o;        /* [H, nq*hd] */
    const void* mlp_norm;   /* [H]  pre-MLP RMSNorm gain */
    const void* w_gate;     /* [F, H] */
    const void* w_up;       /* [F, H] */
    const void* w_down;     /* [H, F] */
} pe_layer_weights;

typedef struct pe_weights {
    const void* fc;          /* [H, 3H]: fuses [h_lo; h_mid; h_hi] into H */
    const void* embed;       /* [V, H] token embedding */
    const void* emb_mask;    /* [H] learned mask-token embedding (positions 2..K) */
    const void* h_shared;    /* [H] learned shared hidden state (positions 2..K) */
    const void* final_norm;  /* [H] */
    const void* lm_head;     /* [V, H] (not tied to embed) */
    pe_layer_weights layer[4];
} pe_weights;

/* FP8 drafter weights. The pages run their benchmarks in FP8 ("在 Amazon
 * SageMaker AI 上使用 P-EAGLE 并行化推测解码", section "基准测试"); here every
 * GEMM weight matrix (FC, QKV, O, gate, up, down, LM head) may be given as
 * E4M3 codes q[m, k] (uint8, the same [out, in] layout, rows a multiple of 16
 * bytes) standing for W[m, k] = q[m, k] * scale[m]. The codes are widened to
 * bf16 in shared memory (exactly: every E4M3 value is a bf16 value), the
 * tensor cores multiply bf16 by bf16 with fp32 accumulation, and the epilogue
 * applies scale[m]. Each array below is fp32 [rows of that matrix]. Codes
 * must be finite: the NaN codes 0x7F / 0xFF are not decoded as NaN. */
typedef struct pe_layer_scales {
    const float* w_qkv;     /* [(nq+2nkv)*hd] */
    const float* w_o;       /* [H] */
    const float* w_gate;    /* [F] */
    const float* w_up;      /* [F] */
    const float* w_down;    /* [H] */
} pe_layer_scales;

typedef struct pe_weight_scales {
    const float* fc;        /* [H] */
    const float* lm_head;   /* [V] */
    pe_layer_scales layer[4];
} pe_weight_scales;

typedef struct pe_handle pe_handle;

/* Create a drafter on `device` (the device must be current or will be made
 * current). Records the weight pointers (caller keeps them alive until
 * pe_destroy), allocates the workspaces for up to max_batch requests of up to
 * cfg->k_max rows and builds TMA descriptors for the weights. Synchronous. */
int pe_init_drafter(const pe_config* cfg, const pe_weights* weights,
                    int32_t max_batch, int32_t device, pe_handle** out);

/* The same for FP8 weights: cfg->dtype must be PE_DTYPE_FP8W; the GEMM
 * matrices of `weights` point at E4M3 codes, the other entries (embed,
 * emb_mask, h_shared, norm gains) at bf16; `scales` gives the per-row scales
 * (device fp32, caller-owned like the weights). Every other entry point works
 * unchanged on the handle, with bf16 target hidden states and KV cache. The
 * persistent layer chain (PE_LAYER_CHAIN) is not used with FP8 weights. */
int pe_init_drafter_fp8(const pe_config* cfg, const pe_weights* weights, const pe_weight_scales* scales,
                        int32_t max_batch, int32_t device, pe_handle** out);

/* One parallel draft pass (pages' Step 2) for B requests, K drafts each.
 *
 *  last_token    [B] int32     last accepted token of each request (row 0 input)
 *  target_hidden [B, 3H]       config dtype; [h_lo | h_mid | h_hi] of that token
 *  positions     [B] int32     Q_b: RoPE position of row 0; row j uses Q_b + j
 *  seq_lens      [B] int32     S_b: committed drafter-cache entries; row j is
 *                              written to and attends through entry S_b + j
 *  page_table    [B, max_pages] int32  physical page of each 16-entry block
 *  num_pages     pages in each layer of the caches
 *  k_cache, v_cache  [4][num_pages][nkv][16][hd] config dtype; read for
 *                entries < S_b, written at entries S_b..S_b+K-1
 *  drafts        [B, K] int32  OUT: argmax of the LM head per row
 *  logits_dbg    [B, K, V] fp32 OUT or NULL: full logits (testing only)
 *  status        [B] int32     OUT: PE_REQ_*; a request that is not OK gets
 *                drafts -1 and no cache writes
 * Requires 1 <= B <= max_batch, 1 <= K <= k_max, target_hidden 16-byte aligned. */
int pe_draft(pe_handle* h, int32_t B, int32_t K,
             const int32_t* last_token, const void* target_hidden,
             const int32_t* positions, const int32_t* seq_lens,
             const int32_t* page_table, int32_t max_pages, int32_t num_pages,
             void* k_cache, void* v_cache,
             int32_t* drafts, float* logits_dbg, int32_t* status, void* stream);

/* Sequential (EAGLE-style) drafting on the same kernels: the chain that
 * P-EAGLE breaks ("在 Amazon SageMaker AI 上使用 P-EAGLE 并行化推测解码",
 * "P-EAGLE 如何打破这个链": each draft needs the embedding of the token drafted
 * just before it and the hidden state that produced it). K passes of one row
 * per request, each a full drafter forward:
 *  - pass 0 is the parallel pass's row 0 (embedding of last_token, FC-fused
 *    target hidden state);
 *  - pass j > 0 takes the embedding of draft j-1 and, as its hidden input and
 *    residual start, the drafter's own final residual stream of pass j-1
 *    (the hidden state before the final RMSNorm);
 *  - pass j sits at RoPE position Q_b + j and cache entry S_b + j and writes
 *    its k/v rows there before pass j+1 attends over them.
 * Same arguments, layouts, outputs and errors as pe_draft (drafts[b, j] is
 * pass j's argmax; logits_dbg row (b, j) its logits); every entry
 * S_b .. S_b+K-1 the step writes is validated by pass 0. The launch count
 * grows linearly in K (K forward passes), where pe_draft's does not. */
int pe_draft_sequential(pe_handle* h, int32_t B, int32_t K,
                        const int32_t* last_token, const void* target_hidden,
                        const int32_t* positions, const int32_t* seq_lens,
                        const int32_t* page_table, int32_t max_pages, int32_t num_pages,
                        void* k_cache, void* v_cache,
                        int32_t* drafts, float* logits_dbg, int32_t* status, void* stream);

/* The parallel draft pass with the tokens of the last verify re-fed as real
 * rows (the alternative to the single-real-row bookkeeping; the pages leave
 * the drafter's cache bookkeeping open). Request b brings n_b = n_real[b]
 * real rows - tokens[b, i] with their target hidden states target_hidden[b, i]
 * (each row: token embedding and FC-fused hidden state, the pages'
 * position-1 input) - ahead of the K-1 placeholder rows. Real row i sits at
 * position Q_b + i and entry S_b + i; placeholder j (1..K-1) at position
 * Q_b + n_b - 1 + j and entry S_b + n_b - 1 + j; every row attends causally.
 * drafts[b, 0] is the argmax of the last real row, drafts[b, j] that of
 * placeholder j.
 *  tokens        [B, n_max] int32 (entries past n_b unused), n_real [B] int32 in 1..n_max
 *  target_hidden [B, n_max, 3H] bf16 (rows past n_b unused)
 *  1 <= n_max <= k_max. Other arguments, outputs and errors as for pe_draft;
 *  every entry S_b .. S_b+n_max+K-2 is validated (PE_REQ_BAD_INPUT also for
 *  n_b out of range or a bad token).
 * Runs as two passes: the layers over real rows 0..n_b-2 (which writes their
 * cache rows; padded to n_max-1 rows, the padding writes nothing), then the
 * parallel pass whose row 0 is the last real row. The result is that of one
 * joint pass, because attention is the only place where rows meet. */
int pe_draft_refeed(pe_handle* h, int32_t B, int32_t K, int32_t n_max, const int32_t* tokens,
                    const int32_t* n_real, const void* target_hidden, const int32_t* positions,
                    const int32_t* seq_lens, const int32_t* page_table, int32_t max_pages, int32_t num_pages,
                    void* k_cache, void* v_cache, int32_t* drafts, float* logits_dbg, int32_t* status,
                    void* stream);

/* Greedy verification + batch-metadata rebuild + KV rollback (one kernel).
 * h may be NULL (the kernel needs no drafter state).
 *
 *  drafts        [B, K] int32     the step's drafts d
 *  target_tokens [B, K+1] int32   target argmax tokens g for the K+1 positions
 *  page_table    [B, max_pages] int32, num_pages as for pe_draft
 *  positions, seq_lens  [B] int32 in: Q_b, S_b of the step just drafted
 *  positions_out, seq_lens_out [B] int32 OUT (may alias the inputs):
 *                 Q_b' = Q_b + a_b + 1, S_b' = S_b + min(a_b, K-1) + 1
 *  accepted      [B] int32 OUT  a_b = longest prefix with d == g, 0..K
 *  bonus         [B] int32 OUT  g[b, a_b]
 *  emitted       [B, K+1] int32 OUT or NULL: d[b, :a_b], bonus, then -1
 *  slot_mapping  [B, K] int32 OUT  physical slot (page*16 + offset) of entries
 *                 S_b' .. S_b'+K-1 (where the next draft pass writes)
 *  rollback_slots [B, K] int32 OUT  slots of rejected entries S_b' .. S_b+K-1,
 *                 then -1 padding
 *  status        [B] int32 OUT  PE_REQ_*; when not OK, positions/seq_lens are
 *                 passed through unchanged and slot/rollback rows are -1.
 * Requires 1 <= K <= 31. */
int pe_verify_rebuild(pe_handle* h, int32_t B, int32_t K,
                      const int32_t* drafts, const int32_t* target_tokens,
                      const int32_t* page_table, int32_t max_pages, int32_t num_pages,
                      const int32_t* positions, const int32_t* seq_lens,
                      int32_t* positions_out, int32_t* seq_lens_out,
                      int32_t* accepted, int32_t* bonus, int32_t* emitted,
                      int32_t* slot_mapping, int32_t* rollback_slots,
                      int32_t* status, void* stream);

/* Verify + rebuild after a pe_draft_refeed pass: the same greedy acceptance,
 * bonus and emitted tokens; the n_b real rows stay committed and the K-1
 * placeholder rows are rolled back:
 *  n_real, positions, seq_lens [B] in; n_real_out = a_b + 1,
 *  positions_out = Q_b + n_b, seq_lens_out = S_b + n_b (may alias the inputs)
 *  slot_mapping  [B, 2K] OUT  slots of the next pass's entries
 *                 S_b' .. S_b'+n_b'+K-2, then -1
 *  rollback_slots [B, K] OUT  slots of entries S_b+n_b .. S_b+n_b+K-2, then -1
 *  status: as pe_verify_rebuild (PE_REQ_BAD_INPUT also for n_b outside
 *  1..K+1); a failed request keeps its metadata and n_real.
 * The next step re-feeds emitted[b, 0..a_b] with their target hidden states.
 * Requires 1 <= K <= 16. */
int pe_verify_rebuild_refeed(pe_handle* h, int32_t B, int32_t K, const int32_t* drafts,
                             const int32_t* target_tokens, const int32_t* page_table, int32_t max_pages,
                             int32_t num_pages, const int32_t* n_real, const int32_t* positions,
                             const int32_t* seq_lens, int32_t* n_real_out, int32_t* positions_out,
                             int32_t* seq_lens_out, int32_t* accepted, int32_t* bonus, int32_t* emitted,
                             int32_t* slot_mapping, int32_t* rollback_slots, int32_t* status, void* stream);

/* Sampled drafting and stochastic acceptance (the pages' "standard
 * acceptance criterion" when decoding samples, as their deployment does at
 * temperature 0.3: "在 Amazon SageMaker AI 上使用 P-EAGLE 并行化推测解码",
 * "逐步草稿过程"). With q_j = softmax(draft logits of row j / T) and
 * p_j = softmax(target logits of position j / T), speculative sampling
 * accepts draft d_j while u_j < p_j(d_j) / q_j(d_j), and emits at the first
 * rejection a token drawn from max(0, p_j - q_j) (normalised), or after K
 * acceptances a bonus token drawn from p_K; the emitted tokens are then
 * distributed as sampling the target alone. Every draw is inverse-CDF
 * sampling with a caller-supplied uniform u in [0, 1): the smallest index
 * whose running weight, summed in index order, exceeds u times the total.
 *
 * pe_sample_drafts: drafts[b, j] ~ q_j from logits [B, K, V] fp32 (the
 *  logits output of pe_draft / pe_draft_refeed; P-EAGLE's rows come from one
 *  pass, so each row is drawn independently), u [B, K] fp32; status [B]
 *  (nullable: requests not PE_REQ_OK get -1).
 * pe_verify_stochastic: draft_logits [B, K, V], target_logits [B, K+1, V]
 *  fp32, u_accept [B, K], u_final [B] fp32; accepted [B] OUT a_b,
 *  final_token [B] OUT the drawn token (it takes the place of the greedy
 *  bonus); emitted, the metadata rebuild, rollback and status exactly as
 *  pe_verify_rebuild given a_b. Uses the handle's workspace (h required;
 *  B <= max_batch, K <= k_max). temperature > 0. */
int pe_sample_drafts(pe_handle* h, int32_t B, int32_t K, const float* logits, float temperature, const float* u,
                     const int32_t* status, int32_t* drafts, void* stream);
int pe_verify_stochastic(pe_handle* h, int32_t B, int32_t K, const int32_t* drafts, const float* draft_logits,
                         const float* target_logits, float temperature, const float* u_accept, const float* u_final,
                         const int32_t* page_table, int32_t max_pages, int32_t num_pages, const int32_t* positions,
                         const int32_t* seq_lens, int32_t* positions_out, int32_t* seq_lens_out, int32_t* accepted,
                         int32_t* final_token, int32_t* emitted, int32_t* slot_mapping, int32_t* rollback_slots,
                         int32_t* status, void* stream);

/* The draft pass's tcgen05 GEMM engine on its own (plain store epilogue):
 *   y[n, m] = sum_k w[m, k] * x[n, k]
 *  w  [M, Kd] config-dtype weights, x [N, Kd] activations (same dtype),
 *  y  [N, M] fp32 OUT. w and x 16-byte aligned, Kd a multiple of 8.
 *  ws       fp32 split-K scratch of at least *ws_floats elements (may be NULL
 *           when *ws_floats is 0), tickets int32 [*n_tickets] that must be
 *           zero before the first call; the kernel leaves them zero again.
 * pe_linear_scratch reports the sizes for a shape on the current device. */
int pe_linear_scratch(int32_t dtype, int32_t M, int32_t N, int32_t Kd, int64_t* ws_floats, int32_t* n_tickets);
int pe_linear(int32_t dtype, int32_t M, int32_t N, int32_t Kd, const void* w, const void* x, float* y,
              float* ws, int32_t* tickets, void* stream);
/* The FP8-weight GEMM engine on its own: y[n, m] = scale[m] * sum_k q[m, k] * x[n, k]
 *  w  [M, Kd] E4M3 codes (uint8), w_scale [M] fp32, x [N, Kd] bf16, y [N, M]
 *  fp32 OUT; Kd a multiple of 16, w and x 16-byte aligned. ws / tickets as
 *  for pe_linear, sized by pe_linear_scratch(PE_DTYPE_FP8W, ...). */
int pe_linear_fp8(int32_t M, int32_t N, int32_t Kd, const void* w, const float* w_scale, const void* x, float* y,
                  float* ws, int32_t* tickets, void* stream);

/* pe_linear for callers that cannot allocate device memory (this entry point
 * has no counterpart in the method's description). Some callers may not call cudaMalloc
 * where they run a GEMM: code running while another thread captures a CUDA
 * graph in global capture mode, where cudaMalloc is prohibited, or runtimes
 * whose device memory is fully reserved by their own allocator. This variant
 * computes the same y[n, m] = sum_k w[m, k] * x[n, k] as pe_linear (same
 * arguments minus ws / tickets) but keeps its split-K scratch in fixed arrays
 * inside the library: 8 MiB of partials and 4096 tickets per device, held
 * until the process exits. It allocates nothing.
 *  - Shapes whose plan needs more scratch than that (pe_linear_scratch
 *    reports the need: more than 2 Mi floats, or more than 4096 tickets
 *    when it needs tickets at all) return PE_ERR_ARG with a message giving
 *    the need and the maximum, before any launch (pe_linear has no limit).
 *  - The first call on each device looks up the arrays' device addresses
 *    (cudaGetSymbolAddress) with that device current and loads the kernel
 *    of both dtypes; make that first call (in either dtype) before any
 *    stream capture that should contain later calls, or that runs while
 *    later calls are made. After cudaDeviceReset the cached addresses are
 *    stale: do not call it on that device again in the same process.
 *  - Every call on a device shares the same arrays: calls that can overlap
 *    on the GPU (several streams or host threads) race and must be serialised
 *    by the caller. Each call clears the tickets it uses on its stream. */
int pe_linear_noalloc(int32_t dtype, int32_t M, int32_t N, int32_t Kd, const void* w, const void* x, float* y,
                      void* stream);

/* One whole step (pe_draft, then pe_verify_rebuild on its drafts) captured
 * once into a CUDA graph and replayed with a single launch. The arguments are
 * those of pe_draft and pe_verify_rebuild (drafts are shared; draft_status and
 * verify_status are the two status arrays); every pointer is baked into the
 * graph, so callers update buffer CONTENTS between launches, not addresses.
 * When positions_out/seq_lens_out alias positions/seq_lens, each replay
 * advances the batch metadata in place. Creation synchronises nothing and
 * enqueues nothing; launches are asynchronous on `stream`. */
typedef struct pe_step_graph pe_step_graph;
int pe_step_graph_create(pe_handle* h, int32_t B, int32_t K, const int32_t* last_token, const void* target_hidden,
                         const int32_t* positions, const int32_t* seq_lens, const int32_t* page_table,
                         int32_t max_pages, int32_t num_pages, void* k_cache, void* v_cache, int32_t* drafts,
                         int32_t* draft_status, const int32_t* target_tokens, int32_t* positions_out,
                         int32_t* seq_lens_out, int32_t* accepted, int32_t* bonus, int32_t* emitted,
                         int32_t* slot_mapping, int32_t* rollback_slots, int32_t* verify_status,
                         pe_step_graph** out);
/* The same with the draft half chosen by draft_mode: PE_DRAFT_PARALLEL
 * (pe_draft, what pe_step_graph_create captures) or PE_DRAFT_SEQUENTIAL
 * (pe_draft_sequential). */
#define PE_DRAFT_PARALLEL   0
#define PE_DRAFT_SEQUENTIAL 1
int pe_step_graph_create_ex(pe_handle* h, int32_t draft_mode, int32_t B, int32_t K, const int32_t* last_token,
                            const void* target_hidden, const int32_t* positions, const int32_t* seq_lens,
                            const int32_t* page_table, int32_t max_pages, int32_t num_pages, void* k_cache,
                            void* v_cache, int32_t* drafts, int32_t* draft_status, const int32_t* target_tokens,
                            int32_t* positions_out, int32_t* seq_lens_out, int32_t* accepted, int32_t* bonus,
                            int32_t* emitted, int32_t* slot_mapping, int32_t* rollback_slots,
                            int32_t* verify_status, pe_step_graph** out);
int pe_step_graph_launch(pe_step_graph* g, void* stream);
/* kernels one replay launches */
int pe_step_graph_launch_count(const pe_step_graph* g);
void pe_step_graph_destroy(pe_step_graph* g);

/* Synchronise `stream` and return (then clear) the device error word of h
 * (PE_DEVERR_* bits; 0 = no device-side wait gave up). */
int pe_device_errors(pe_handle* h, void* stream, uint32_t* out_bits);

/* Test support for the bounded-wait give-up path (no counterpart in the
 * method's description; host-side fault injection, nothing on the device is made to fault).
 * Enqueues on `stream` a write that primes the arrival tickets of the first
 * phase of the handle's persistent layer chain so that its shared tiles never
 * complete. The next pe_draft's chain launches then wait for a phase that
 * never finishes: each such wait gives up after its time limit (1 s), sets
 * PE_DEVERR_CHAIN_TIMEOUT, and the kernel returns; its outputs for that call
 * are meaningless. The chain resets its tickets and counters on the way out,
 * so the handle is usable again once pe_device_errors has read and cleared
 * the error word. Returns PE_ERR_UNSUPPORTED when the handle runs no chain
 * (it runs one when created with PE_LAYER_CHAIN=1 in the environment, bf16,
 * for draft passes of at most 64 rows). */
int pe_test_stall_chain(pe_handle* h, void* stream);

/* Kernel kinds of the draft pass, for launch accounting and profiling. */
#define PE_KERNEL_FC         0
#define PE_KERNEL_ROW_BUILD  1
#define PE_KERNEL_RMSNORM    2   /* reserved: RMSNorm is folded into the GEMM epilogues and never launched */
#define PE_KERNEL_QKV        3
#define PE_KERNEL_ATTENTION  4   /* with length-aware pieces also the merge kernel that follows it */
#define PE_KERNEL_O_PROJ     5
#define PE_KERNEL_GATE_UP    6
#define PE_KERNEL_DOWN       7
#define PE_KERNEL_LM_HEAD    8
#define PE_KERNEL_ARGMAX     9
#define PE_KERNEL_LAYER_CHAIN 10  /* O, gate/up, down and the next QKV (or the LM head) in one persistent launch */
#define PE_KERNEL_COUNT      11

/* Measurement hook: after pe_profile_start, every launch of `kernel_kind`
 * made by pe_draft (up to max_launches of them) is bracketed by CUDA events
 * recorded on the launch stream; an attention that runs as length-aware
 * pieces is bracketed together with its merge kernel (one interval per
 * layer). pe_profile_stop waits for those events and returns the summed
 * device time (ms) and the number of intervals timed. */
int pe_profile_start(pe_handle* h, int32_t kernel_kind, int32_t max_launches);
int pe_profile_stop(pe_handle* h, float* total_ms, int32_t* launches);
const char* pe_kernel_name(int32_t kind);

/* Number of kernels the last pe_draft call enqueued (for launch accounting;
 * merge kernels included). */
int pe_last_launch_count(const pe_handle* h);

void pe_destroy(pe_handle* h);

/* Thread-local description of the last error (never NULL). */
const char* pe_last_error(void);

int pe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PE_H */
