// Internal declarations shared by the libpe.so translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <string>
#include <utility>

#include "pe.h"

namespace pe {

// ---------------------------------------------------------------- errors

void set_error(const std::string& msg);
#define PE_CUDA_TRY(expr)                                                                   \
    do {                                                                                    \
        cudaError_t e_ = (expr);                                                            \
        if (e_ != cudaSuccess) {                                                            \
            ::pe::set_error(std::string(#expr) + ": " + cudaGetErrorString(e_));            \
            return PE_ERR_CUDA;                                                             \
        }                                                                                   \
    } while (0)

int encode_tmap_2d(CUtensorMap* map, const void* base, int dtype, uint64_t inner, uint64_t rows,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows);
// the same over one-byte elements (FP8 weight codes)
int encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows);

// ---------------------------------------------------------------- GEMM

enum Epi : int { EPI_STORE = 0, EPI_QKV = 1, EPI_RESID = 2, EPI_SWIGLU = 3, EPI_ARGMAX = 4 };

// One tcgen05 GEMM  D[m, n] = sum_k W[m, k] * X[n, k]  (weights W fill the
// 128-row M side, token rows X the N side), followed by a fused epilogue.
struct GemmParams {
    int M;              // output features (for SWIGLU: F, each tile = 64 gate + 64 up rows)
    int N;              // token rows
    int Kd;             // reduction length
    int m_tiles, n_tiles, splits, kb_total, kb_per_split, bn, stages;
    int cstages;        // FP8 weights: bf16 copies of half weight stages in shared memory
    // STORE / RESID: fp32 [N, ld_out]
    float* out_f32;
    int ld_out;
    // QKV: q out (T) [N, ld_act]; SWIGLU: act out (T) [N, ld_act]
    void* out_act;
    int ld_act;
    // QKV extras
    void* k_cache;      // this layer's [num_pages][nkv][16][hd]
    void* v_cache;
    int nq_hd, nkv, hd;
    const int* row_slot;        // [N] physical cache slot of row n, -1 = skip
    const float2* rope_cs;      // [N][hd/2] (cos, sin)
    // ARGMAX
    unsigned long long* amax;   // [N]
    float* logits;              // [N, ld_logits] or null
    int ld_logits;
    // Folded RMSNorm, producer side (RESID): besides the residual, write
    // xg[n, m] = gain[m] * r[n, m] in the activation dtype [N, ld_xg] and this
    // m tile's partial sum of r[n, :]^2 to ss_out[n * ss_ld + m_tile].
    void* xg;
    const void* xg_gain;
    int ld_xg;
    float* ss_out;
    // Folded RMSNorm, consumer side: the B operand is xg; column n of the
    // accumulator is scaled by rsqrt(sum_q ss_in[n * ss_ld + q] * ss_scale + ss_eps)
    // (q in order; ss_ld a multiple of 4 and the entries past the producer's
    // m tiles zero) before the epilogue.
    const float* ss_in;
    int ss_parts;
    int ss_ld;
    float ss_scale;
    float ss_eps;
    // split-K: cluster != 0 reduces through distributed shared memory;
    // otherwise partials go through ws and the tile's ticket
    int cluster;
    int persistent;     // walk units with stride gridDim.x, double-buffered accumulator
    float* ws;
    int* tickets;
    unsigned* err;
    // weight tiles m_tile < keep_tiles are loaded evict-last (they stay in L2
    // across steps); the rest evict-first
    int keep_tiles;
    // FP8 weights (the kernel's W8 instance): accumulator row m is multiplied
    // by w_scale[m] before the epilogue (SWIGLU: gate row f by w_scale[f], up
    // row f by w_scale2[f])
    const float* w_scale;
    const float* w_scale2;
};

struct GemmPlan {
    bool w8;            // FP8 (E4M3) weights widened to bf16 in shared memory; 128 k per stage
    int cstages;        // W8: bf16 copies of half weight stages (double-buffered)
    int bn, n_tiles, m_tiles, splits, kb_total, kb_per_split, stages;
    int units;
    size_t smem_bytes;
    size_t ws_floats;   // global split-K scratch needed (0 if splits == 1 or cluster)
    int tiles;          // tickets needed
    bool cluster;       // splits of a tile form one thread-block cluster
    bool persistent;    // grid < units: CTAs loop over tiles
    int grid;           // CTAs launched
    int epi_groups;     // groups of four epilogue warps (2: 320 threads, one CTA per SM)
    bool w8_one;        // FP8 weights: the kernel compiled for one CTA per SM
};

GemmPlan plan_gemm(int M, int N, int Kd, int epi, int elem_bytes, int num_sms, bool cluster, bool w8 = false);
int launch_gemm(int dtype, int epi, const CUtensorMap& A, const CUtensorMap& A2, const CUtensorMap& B,
                const GemmPlan& plan, GemmParams p, cudaStream_t stream, bool pdl);
// Loads the plain-store GEMM kernels of both dtypes on the current device
// (module loading is lazy; this makes the first launch of either load nothing)
int gemm_store_kernels_load();

// ---------------------------------------------------------------- persistent layer chain

// Several weight-streaming GEMMs of one draft pass (O, gate/up, down and the
// next layer's QKV, or the LM head) in one cooperative launch with one CTA per
// SM. Each phase's k-blocks are split evenly over the CTAs (a tile shared by
// several CTAs is summed in CTA order by the last to arrive); the weight ring
// runs ahead across phases, and a phase's activations are loaded once the
// previous phase's per-tile completion counter is full.
constexpr int kMaxChainPhases = 4;
constexpr int kMaxChainBn = 64;

struct ChainPhase {
    CUtensorMap tmA;     // weights; SWIGLU: gate rows (64-row boxes)
    CUtensorMap tmA2;    // SWIGLU: up rows
    CUtensorMap tmB;     // activations [N, Kd], box rows = bn
    GemmParams gp;       // epilogue parameters (M, N, Kd, outputs, folded norm)
    int epi;
    int m_tiles;         // weight tiles (128 rows; SWIGLU: 64 gate + 64 up)
    int kb_total;        // 64-element k-blocks per tile
    int max_segs;        // most CTAs sharing one tile (stride of the partial buffer)
    long long ws_off;    // this phase's region of the partial buffer (floats)
    int ticket_off;      // this phase's tickets
};

struct ChainParams {
    ChainPhase ph[kMaxChainPhases];
    int nphases;
    int bn, stages;
    unsigned* counters;  // [kMaxChainPhases + 1]: tiles finished per phase, then CTAs finished; zero between launches
    float* ws;           // partial tiles of shared tiles
    int* tickets;        // per-tile arrival counts, zero between launches
    unsigned* err;
};

struct ChainPlan {
    int bn, stages, grid;
    size_t smem_bytes;
    size_t ws_floats;    // partial buffer of all phases given to chain_plan (one region each)
    int tickets;         // tickets of all phases (one run each)
};

// Plan for token rows N and the phases' (m_tiles, kb_total); ok = false when
// the chain does not apply (N > kMaxChainBn or no co-resident CTA per SM).
ChainPlan chain_plan(int N, const int* m_tiles, const int* kb_total, int nphases, int num_sms, bool* ok);
int chain_max_segs(int m_tiles, int kb_total, int grid);
int launch_chain(const ChainParams& p, const ChainPlan& plan, cudaStream_t s, bool pdl);
bool chain_supported(int device);

// ---------------------------------------------------------------- small kernels

struct RowBuildParams {
    int B, K, H, V, hd, max_pages, num_pages, page_size;
    const int32_t* last_token; // row-0 token of request b: last_token[b * tok_stride]
    int tok_stride;
    const int32_t* positions;
    const int32_t* seq_lens;
    const int32_t* page_table;
    const float* h;            // row-0 hidden of request b: h[b * hid_stride .. + H) (FC output, or a residual row)
    int hid_stride;
    // This pass's rows sit j0 entries (and positions) past S_b / Q_b: row j
    // at entry S_b + j0 + j, RoPE position Q_b + j0 + j (0 for the parallel
    // pass; the pass index for sequential drafting). k_check: entries past
    // S_b that the whole step writes, validated against the page table.
    int j0, k_check;
    int status_in;             // 1: status[b] was set by an earlier pass; read it, write nothing
    int32_t* seq_eff;          // OUT [B] or null: S_b + j0_b (the attention's committed-entry count)
    // Rows with their own inputs and per-request offsets (re-fed real rows).
    // Rows j < n_lead take token last_token[b * tok_stride + (o_b + j) * tok_jstride]
    // and hidden h[b * hid_bstride + (o_b + j) * hid_stride], o_b = row_off[b] + off_add
    // (0 without row_off); rows past them are placeholders. The pass's rows
    // sit at entry S_b + j0 + o_b + j. Rows j >= row_lim[b] + lim_add (when
    // row_lim is set) are padding: no cache write, outputs unused.
    int n_lead;
    int tok_jstride, hid_bstride;
    const int32_t* row_off;
    int off_add;
    const int32_t* row_lim;
    int lim_add;
    // re-fed real rows: status also checks n_real[b] in [1, n_max] and the
    // tokens last_token[b * tok_stride + i], i < n_real[b]
    const int32_t* n_real;
    int n_max;
    const void* embed;         // [V, H]
    const void* emb_mask;      // [H]
    const void* h_shared;      // [H]
    const void* norm_e;        // [H]
    const void* norm_h;        // [H]
    float eps;
    void* u;                   // OUT [R, 2H] T
    float* resid;              // OUT [R, H]
    int* row_slot;             // OUT [R]
    float2* rope_cs;           // OUT [R, hd/2]
    const double* inv_freq;    // [hd/2]
    unsigned long long* amax;  // OUT [R] zeroed
    int32_t* status;           // OUT [B]
    int32_t* order;            // OUT [B] or null: requests by decreasing seq_len (ties by index)
    // Length-aware attention pieces (null: none). Block 0 cuts every
    // request's S + K cache entries into n_b pieces of about the same tile
    // count (total tiles / piece_slots, at least piece_min_tiles; with
    // piece_wave > 0 the smallest count from total tiles / piece_wave up
    // whose pieces still number at most piece_wave) and writes
    // one item {b, kv head, first entry, end entry} per (piece, kv head),
    // longest requests first; item (nkv * (off_b + i) + kv head) is piece i
    // of request b. attn_plan: [0] item count, [1 + b] n_b, [1 + B + b] off_b.
    int4* attn_items;
    int* attn_plan;
    int nkv, piece_slots, piece_min_tiles, piece_wave;
};
int launch_row_build(int dtype, const RowBuildParams& p, cudaStream_t s, bool pdl);

// logits[n, :V] *= 1/rms of token row n, from the folded norm's partial sums
// of squares ss[n * ss_ld + q] (the LM head's optional logits output)
int launch_logits_rms_scale(float* logits, int rows, int V, int ld, const float* ss, int ss_ld, float scale,
                            float eps, cudaStream_t s, bool pdl);

// drafts[b * out_stride + j] = decoded record of row b * K + j (-1 when the
// request is not OK)
int launch_argmax_finalize(const unsigned long long* amax, const int32_t* status, int B, int K, int32_t* drafts,
                           int out_stride, cudaStream_t s, bool pdl);

// ---------------------------------------------------------------- attention

struct AttnParams {
    int B, K, nq, nkv, hd, max_pages, num_pages, page_size;
    int chunk;        // cache entries per split
    int max_splits;   // grid.y
    int layer_page0;  // layer * num_pages: first page of this layer in the 4-D KV tensor map
    const void* q;            // [R, nq*hd] T (rotated)
    const void* k_cache;      // this layer
    const void* v_cache;
    const int32_t* page_table;
    const int32_t* seq_lens;
    const int32_t* status;
    const int32_t* order;     // [B] or null: CTA pair i serves request order[i / nkv] (longest first)
    void* out;                // [R, nq*hd] T
    float* ws;                // split partials
    int* tickets;             // [B*nkv]
    unsigned* err;
    // length-aware pieces (tcgen05 kernel; null: one cluster of max_splits
    // CTAs per (request, kv head)): CTA i serves items[i] while i < plan[0];
    // a piece of a request with several writes its partial (O, running max,
    // sum) to ws[i] and k_attn_merge combines them
    const int4* items;
    const int* plan;
    int grid;                 // CTAs launched (>= the item count)
    int l2_prefetch;          // CTAs warm L2 with their first K/V pages before the dependency wait
};
struct AttnPlan {
    int chunk, max_splits;
    size_t ws_floats;
    int tickets;
    bool pieces;              // length-aware pieces + merge kernel
    int piece_slots;          // CTAs resident at once (SMs x CTAs per SM)
    int piece_min_tiles;
    int piece_wave;           // > 0: the pieces fit one wave of this many CTAs
    int grid;                 // piece_slots + B * nkv
    bool one_wave;            // every CTA of the launch is resident at once
};
AttnPlan plan_attention(int B, int K, int nq, int nkv, int hd, int max_pages, int page_size, int num_sms);
int launch_attention(int dtype, const AttnParams& p, cudaStream_t s, bool pdl);
// tk / tv are 4-D maps {hd, 16, nkv, 4 * num_pages} over the paged caches
int encode_tmap_kv(CUtensorMap* map, const void* cache, int hd, int nkv, int num_pages);
// bf16 tcgen05 attention; tq is a 3-D map {hd, nq, rows} over q with box {64, nq/nkv, K}
AttnPlan plan_attention_umma(int B, int K, int nq, int nkv, int hd, int max_pages, int page_size, int num_sms);
int launch_attention_umma(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                          cudaStream_t s, bool pdl);
// combines the pieces of every (request, kv head) with more than one
int launch_attention_merge(const AttnParams& p, cudaStream_t s, bool pdl);
// floats of one piece partial in the attention scratch: O [Rq][hd], then the
// running max [Rq] and sum [Rq], each block a multiple of 16 bytes
__host__ __device__ inline size_t attn_piece_floats(int Rq, int hd) {
    return static_cast<size_t>(Rq) * hd + 2 * static_cast<size_t>((Rq + 3) & ~3);
}
int encode_tmap_q(CUtensorMap* map, const void* q, int hd, int nq, int rows, int G, int K);

// ---------------------------------------------------------------- verify

int launch_verify_rebuild(int B, int K, const int32_t* drafts, const int32_t* target, const int32_t* page_table,
                          int max_pages, int num_pages, int page_size, const int32_t* positions,
                          const int32_t* seq_lens, int32_t* positions_out, int32_t* seq_lens_out,
                          int32_t* accepted, int32_t* bonus, int32_t* emitted, int32_t* slot_mapping,
                          int32_t* rollback, int32_t* status, cudaStream_t s);

// metadata rebuild for an acceptance decided elsewhere: accepted [B] and the
// final token [B] are inputs (emitted, slots, rollback, status as above)
int launch_rebuild_given_acceptance(int B, int K, const int32_t* drafts, const int32_t* page_table, int max_pages,
                                    int num_pages, int page_size, const int32_t* positions, const int32_t* seq_lens,
                                    int32_t* positions_out, int32_t* seq_lens_out, const int32_t* accepted,
                                    const int32_t* final_tok, int32_t* emitted, int32_t* slot_mapping,
                                    int32_t* rollback, int32_t* status, cudaStream_t s);

// ---------------------------------------------------------------- sampling (stochastic acceptance)

// drafts[r] ~ softmax(logits[r] / T) by inverse CDF with u[r], rows r = b * K + j
// (status[b] not OK: -1); one CTA per row
int launch_sample_rows(const float* logits, int rows, int V, float temperature, const float* u,
                       const int32_t* status, int K, int32_t* drafts, cudaStream_t s);
// speculative-sampling acceptance: per-row softmax statistics into `stats`
// ([B*K + B*(K+1)] float2), then per request the accepted length and the
// final token (residual draw or bonus)
int launch_stochastic_accept(int B, int K, int V, float temperature, const int32_t* drafts, const float* dlogits,
                             const float* tlogits, const float* u_accept, const float* u_final, float2* stats,
                             int32_t* accepted, int32_t* final_tok, cudaStream_t s);

// the same for re-fed real rows: n_real in/out, slot_mapping [B, 2K], rollback [B, K]
int launch_verify_rebuild_refeed(int B, int K, const int32_t* drafts, const int32_t* target,
                                 const int32_t* page_table, int max_pages, int num_pages, int page_size,
                                 const int32_t* n_real, const int32_t* positions, const int32_t* seq_lens,
                                 int32_t* n_real_out, int32_t* positions_out, int32_t* seq_lens_out,
                                 int32_t* accepted, int32_t* bonus, int32_t* emitted, int32_t* slot_mapping,
                                 int32_t* rollback, int32_t* status, cudaStream_t s);

// Launch helper: every kernel goes through cudaLaunchKernelEx so that the
// programmatic-dependent-launch attribute can be set uniformly.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                      Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pe
