// C ABI of libpe.so: drafter handle, workspaces, TMA descriptors and the
// per-step orchestration of the draft pass (see include/pe.h).
//
// One draft pass enqueues, on the caller's stream:
//   FC GEMM (3H -> H, rows = B)                          [a1]
//   row build (rows, slots, RoPE table, status)          [a2]
//   4 x { [RMSNorm] QKV GEMM + RoPE + paged KV write,    [a3]
//         paged attention,                               [a4]
//         O GEMM + residual,                             [a5]
//         RMSNorm, gate/up GEMM + SwiGLU,                [a6]
//         down GEMM + residual }
//   final RMSNorm, LM-head GEMM + fused argmax,          [a7]
//   argmax finalisation -> drafts.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

struct pe_handle {
    pe_config cfg;                // dtype is the activation dtype (bf16 for an FP8-weight drafter)
    pe_weights w;
    bool w8 = false;              // GEMM weights are E4M3 codes with per-row scales
    pe_weight_scales sc{};
    int device = 0;
    int max_batch = 0;
    int max_rows = 0;
    int num_sms = 0;
    size_t elem = 2;
    bool pdl = false;
    // workspaces (device)
    float* h = nullptr;           // [max_rows, H] FC outputs (one row per request, or per re-fed real row)
    float* resid = nullptr;       // [max_rows, H]
    void* u = nullptr;            // [max_rows, 2H]
    void* xn = nullptr;           // [max_rows, H] gain * residual (folded RMSNorm input)
    float* ss = nullptr;          // [max_rows, ss_ld] per-128-feature partial sums of squares of the residual
    int ss_ld = 0;                // ceil(H/128) rounded up to a multiple of 4 (the padding stays zero)
    void* q = nullptr;            // [max_rows, nq*hd]
    void* attn = nullptr;         // [max_rows, nq*hd]
    void* act = nullptr;          // [max_rows, F]
    unsigned long long* amax = nullptr;
    int* row_slot = nullptr;
    int32_t* attn_order = nullptr;   // [max_batch] requests by decreasing seq_len
    int32_t* seq_eff = nullptr;      // [max_batch] S_b + j0 of the current sequential pass
    float2* samp_stats = nullptr;    // [max_batch * (2 k_max + 1)] softmax (max, sum) per logit row
    float2* rope_cs = nullptr;
    double* inv_freq = nullptr;
    float* gemm_ws = nullptr;
    size_t gemm_ws_floats = 0;
    int* gemm_tickets = nullptr;
    int gemm_tickets_n = 0;
    float* attn_ws = nullptr;
    size_t attn_ws_floats = 0;
    int* attn_tickets = nullptr;
    int attn_tickets_n = 0;
    int4* attn_items = nullptr;      // [attn_items_n] length-aware attention pieces
    int attn_items_n = 0;
    int* attn_plan = nullptr;        // [1 + 2 * max_batch] piece count, pieces and first piece per request
    unsigned* err = nullptr;
    // persistent layer chain (bf16, up to kMaxChainBn token rows)
    bool chain = false;
    unsigned* chain_ctr = nullptr;   // [kMaxChainPhases + 1]
    float* chain_ws = nullptr;
    size_t chain_ws_floats = 0;
    int* chain_tickets = nullptr;
    int chain_tickets_n = 0;
    // weight tensor maps
    CUtensorMap tm_fc, tm_lm;
    CUtensorMap tm_qkv[4], tm_o[4], tm_gate[4], tm_up[4], tm_down[4];
    int last_launches = 0;
    // profiling hook (pe_profile_start / pe_profile_stop)
    int prof_kind = -1;
    int prof_used = 0;
    std::vector<cudaEvent_t> prof_events;
};

namespace pe {

static thread_local std::string g_last_error = "no error";
void set_error(const std::string& msg) { g_last_error = msg; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

int encode_tmap_2d(CUtensorMap* map, const void* base, int dtype, uint64_t inner, uint64_t rows,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows) {
    EncodeTiledFn fn = get_encode_fn();
    if (fn == nullptr) {
        set_error("cuTensorMapEncodeTiled entry point not available");
        return PE_ERR_CUDA;
    }
    if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || (row_stride_bytes & 15u) != 0) {
        set_error("TMA operand must be 16-byte aligned with a 16-byte multiple row stride");
        return PE_ERR_ARG;
    }
    cuuint64_t dims[2] = {inner, rows < 1 ? 1 : rows};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        dtype == PE_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed with code " + std::to_string(static_cast<int>(r)));
        return PE_ERR_CUDA;
    }
    return PE_OK;
}

int encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn fn = get_encode_fn();
    if (fn == nullptr) {
        set_error("cuTensorMapEncodeTiled entry point not available");
        return PE_ERR_CUDA;
    }
    if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || (inner & 15u) != 0) {
        set_error("FP8 weights must be 16-byte aligned with rows a multiple of 16 bytes");
        return PE_ERR_ARG;
    }
    cuuint64_t dims[2] = {inner, rows < 1 ? 1 : rows};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled (u8) failed with code " + std::to_string(static_cast<int>(r)));
        return PE_ERR_CUDA;
    }
    return PE_OK;
}

// bf16 paged KV cache [4][num_pages][nkv][16][hd] as a 4-D tensor
// {hd, 16 slots, nkv, 4 * num_pages}; box = one page of one kv head, 64 dims
// (128 bytes) wide, 128-byte swizzle.
int encode_tmap_kv(CUtensorMap* map, const void* cache, int hd, int nkv, int num_pages) {
    EncodeTiledFn fn = get_encode_fn();
    if (fn == nullptr) {
        set_error("cuTensorMapEncodeTiled entry point not available");
        return PE_ERR_CUDA;
    }
    if ((reinterpret_cast<uintptr_t>(cache) & 15u) != 0) {
        set_error("KV cache must be 16-byte aligned");
        return PE_ERR_ARG;
    }
    const uint64_t e = 2;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(hd), 16, static_cast<cuuint64_t>(nkv),
                          4ull * static_cast<cuuint64_t>(num_pages)};
    cuuint64_t strides[3] = {hd * e, 16ull * hd * e, static_cast<cuuint64_t>(nkv) * 16ull * hd * e};
    cuuint32_t box[4] = {64, 16, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(cache), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled (KV) failed with code " + std::to_string(static_cast<int>(r)));
        return PE_ERR_CUDA;
    }
    return PE_OK;
}

// bf16 query rows q [rows][nq][hd] as a 3-D tensor {hd, nq, rows}; box = the
// nq/nkv heads of one kv head for the K rows of one request, 64 dims wide.
int encode_tmap_q(CUtensorMap* map, const void* q, int hd, int nq, int rows, int G, int K) {
    EncodeTiledFn fn = get_encode_fn();
    if (fn == nullptr) {
        set_error("cuTensorMapEncodeTiled entry point not available");
        return PE_ERR_CUDA;
    }
    const uint64_t e = 2;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(hd), static_cast<cuuint64_t>(nq), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {hd * e, static_cast<cuuint64_t>(nq) * hd * e};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(K)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled (q) failed with code " + std::to_string(static_cast<int>(r)));
        return PE_ERR_CUDA;
    }
    return PE_OK;
}

}  // namespace pe

using namespace pe;

namespace {

constexpr int kBoxBytes = 128;   // inner TMA box = one 128-byte swizzle row

int box_inner(const pe_handle* h) { return kBoxBytes / static_cast<int>(h->elem); }

// weight [rows, cols] row-major; box rows 128 (64 for gate/up halves); FP8
// codes as one-byte elements, 128 per box row
int weight_map(pe_handle* h, CUtensorMap* m, const void* w, int rows, int cols, int box_rows) {
    if (h->w8) return encode_tmap_2d_u8(m, w, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows), box_rows);
    return encode_tmap_2d(m, w, h->cfg.dtype, cols, rows, static_cast<uint64_t>(cols) * h->elem, box_inner(h),
                          box_rows);
}

// activation [rows, cols]; box rows = bn of the GEMM consuming it
int act_map(const pe_handle* h, CUtensorMap* m, const void* x, int rows, int cols, int bn) {
    return encode_tmap_2d(m, x, h->cfg.dtype, cols, rows, static_cast<uint64_t>(cols) * h->elem,
                          kBoxBytes / static_cast<int>(h->elem), bn);
}

void free_handle(pe_handle* h) {
    if (h == nullptr) return;
    for (cudaEvent_t e : h->prof_events) cudaEventDestroy(e);
    void* ptrs[] = {h->h,    h->resid,    h->u,        h->xn,         h->ss,      h->q,            h->attn,      h->act,
                    h->amax, h->row_slot, h->attn_order, h->rope_cs, h->inv_freq, h->gemm_ws, h->gemm_tickets, h->attn_ws,
                    h->attn_tickets, h->err, h->chain_ctr, h->chain_ws, h->chain_tickets, h->attn_items,
                    h->attn_plan, h->seq_eff, h->samp_stats};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    delete h;
}

int check_config(const pe_config& c) {
    if (c.n_layers != 4) { set_error("n_layers must be 4"); return PE_ERR_UNSUPPORTED; }
    if (c.page_size != 16) { set_error("page_size must be 16"); return PE_ERR_UNSUPPORTED; }
    if (c.head_dim != 64 && c.head_dim != 128) { set_error("head_dim must be 64 or 128"); return PE_ERR_UNSUPPORTED; }
    if (c.n_kv_heads <= 0 || c.n_q_heads % c.n_kv_heads != 0) {
        set_error("n_kv_heads must divide n_q_heads");
        return PE_ERR_UNSUPPORTED;
    }
    if ((c.n_q_heads * c.head_dim) % 128 != 0 || (c.n_kv_heads * c.head_dim) % 128 != 0) {
        set_error("n_q_heads*head_dim and n_kv_heads*head_dim must be multiples of 128");
        return PE_ERR_UNSUPPORTED;
    }
    if (c.hidden % 64 != 0 || c.ffn % 64 != 0 || c.hidden <= 0 || c.ffn <= 0 || c.hidden > 8192) {
        set_error("hidden and ffn must be positive multiples of 64, hidden <= 8192");
        return PE_ERR_UNSUPPORTED;
    }
    if (c.vocab <= 0) { set_error("vocab must be positive"); return PE_ERR_ARG; }
    if (c.k_max < 1 || c.k_max > 16) { set_error("k_max must be in 1..16"); return PE_ERR_UNSUPPORTED; }
    if (c.k_max * (c.n_q_heads / c.n_kv_heads) > 128) {
        set_error("k_max * (n_q_heads / n_kv_heads) must be <= 128");
        return PE_ERR_UNSUPPORTED;
    }
    if (c.dtype != PE_DTYPE_BF16 && c.dtype != PE_DTYPE_FP32 && c.dtype != PE_DTYPE_FP8W) {
        set_error("unknown dtype");
        return PE_ERR_ARG;
    }
    if (!(c.rms_eps > 0.f) || !(c.rope_theta > 0.f)) { set_error("rms_eps and rope_theta must be > 0"); return PE_ERR_ARG; }
    return PE_OK;
}

template <typename P>
int dev_alloc(P** p, size_t bytes) {
    if (bytes == 0) bytes = 16;
    if (cudaMalloc(reinterpret_cast<void**>(p), bytes) != cudaSuccess) {
        set_error("cudaMalloc of " + std::to_string(bytes) + " bytes failed");
        return PE_ERR_NOMEM;
    }
    return PE_OK;
}

}  // namespace

extern "C" {

int pe_abi_version(void) { return PE_ABI_VERSION; }

const char* pe_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"

namespace {

int init_drafter(const pe_config* cfg, const pe_weights* weights, const pe_weight_scales* scales, int32_t max_batch,
                 int32_t device, pe_handle** out) {
    if (cfg == nullptr || weights == nullptr || out == nullptr) { set_error("null argument"); return PE_ERR_ARG; }
    *out = nullptr;
    int rc = check_config(*cfg);
    if (rc != PE_OK) return rc;
    const bool w8 = cfg->dtype == PE_DTYPE_FP8W;
    if (w8 != (scales != nullptr)) {
        set_error(w8 ? "FP8 weights need pe_init_drafter_fp8 and its scales"
                     : "weight scales are only taken with dtype PE_DTYPE_FP8W");
        return PE_ERR_ARG;
    }
    if (w8) {
        const void* sp[] = {scales->fc, scales->lm_head};
        for (const void* p : sp)
            if (p == nullptr) { set_error("null weight scale pointer"); return PE_ERR_ARG; }
        for (int l = 0; l < 4; ++l) {
            const pe_layer_scales& L = scales->layer[l];
            const void* lp[] = {L.w_qkv, L.w_o, L.w_gate, L.w_up, L.w_down};
            for (const void* p : lp)
                if (p == nullptr) { set_error("null layer weight scale pointer"); return PE_ERR_ARG; }
        }
    }
    if (max_batch < 1) { set_error("max_batch must be >= 1"); return PE_ERR_ARG; }
    const pe_weights& w = *weights;
    const void* req[] = {w.fc, w.embed, w.emb_mask, w.h_shared, w.final_norm, w.lm_head};
    for (const void* p : req)
        if (p == nullptr) { set_error("null weight pointer"); return PE_ERR_ARG; }
    for (int l = 0; l < 4; ++l) {
        const pe_layer_weights& L = w.layer[l];
        const void* lp[] = {L.w_qkv, L.w_o, L.mlp_norm, L.w_gate, L.w_up, L.w_down};
        for (const void* p : lp)
            if (p == nullptr) { set_error("null layer weight pointer"); return PE_ERR_ARG; }
        if (l == 0 && (L.norm_e == nullptr || L.norm_h == nullptr)) { set_error("layer 0 needs norm_e and norm_h"); return PE_ERR_ARG; }
        if (l > 0 && L.attn_norm == nullptr) { set_error("layers 1..3 need attn_norm"); return PE_ERR_ARG; }
    }
    PE_CUDA_TRY(cudaSetDevice(device));
    int cc_major = 0, cc_minor = 0;
    PE_CUDA_TRY(cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, device));
    PE_CUDA_TRY(cudaDeviceGetAttribute(&cc_minor, cudaDevAttrComputeCapabilityMinor, device));
    if (cc_major != 10 || cc_minor != 3) {
        set_error("libpe.so is built for sm_103a; device compute capability is " + std::to_string(cc_major) + "." +
                  std::to_string(cc_minor));
        return PE_ERR_UNSUPPORTED;
    }

    pe_handle* h = new pe_handle();
    h->cfg = *cfg;
    h->w8 = w8;
    if (w8) {
        h->sc = *scales;
        h->cfg.dtype = PE_DTYPE_BF16;   // activations, embeddings, norms and KV cache
    }
    h->w = w;
    h->device = device;
    h->max_batch = max_batch;
    h->max_rows = max_batch * cfg->k_max;
    h->elem = h->cfg.dtype == PE_DTYPE_BF16 ? 2 : 4;
    const char* pdl_env = std::getenv("PE_PDL");
    h->pdl = !(pdl_env != nullptr && pdl_env[0] == '0');
    if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        free_handle(h);
        set_error("cudaDeviceGetAttribute failed");
        return PE_ERR_CUDA;
    }

    const int H = cfg->hidden, F = cfg->ffn, V = cfg->vocab, hd = cfg->head_dim;
    const int nq = cfg->n_q_heads, nkv = cfg->n_kv_heads;
    const int qd = nq * hd, qkv_rows = (nq + 2 * nkv) * hd;
    const size_t R = static_cast<size_t>(h->max_rows), E = h->elem;

    // split-K scratch: the largest plan over every row count this handle accepts
    size_t ws = 0;
    int tiles = 1;
    const int elem_bytes = static_cast<int>(E);
    struct Shape { int M, Kd, epi; };
    const Shape shapes[] = {{H, 3 * H, EPI_STORE}, {qkv_rows, 2 * H, EPI_QKV}, {qkv_rows, H, EPI_QKV},
                            {H, qd, EPI_RESID},    {F, H, EPI_SWIGLU},        {H, F, EPI_RESID},
                            {V, H, EPI_ARGMAX}};
    for (const Shape& s : shapes) {
        for (int n = 1; n <= h->max_rows; ++n) {
            GemmPlan g = plan_gemm(s.M, n, s.Kd, s.epi, elem_bytes, h->num_sms, true, h->w8);
            ws = ws > g.ws_floats ? ws : g.ws_floats;
            tiles = tiles > g.tiles ? tiles : g.tiles;
        }
    }
    h->gemm_ws_floats = ws;
    h->gemm_tickets_n = tiles;
    // attention split scratch: bounded by ~2 CTAs per SM plus one partial split per pair
    const int G = nq / nkv;
    const size_t pairs_max = static_cast<size_t>(max_batch) * nkv;
    h->attn_ws_floats = (2 * static_cast<size_t>(h->num_sms) + 2 * pairs_max) * (cfg->k_max * G) * (hd + 2);
    h->attn_tickets_n = static_cast<int>(pairs_max);
    h->attn_items_n = 2 * h->num_sms + static_cast<int>(pairs_max);
    // persistent layer chain: the partial buffer of its two phase lists
    // (O, gate/up, down, QKV and O, gate/up, down, LM head) at the widest
    // token tile it serves
    const char* chain_env = std::getenv("PE_LAYER_CHAIN");
    h->chain = cfg->dtype == PE_DTYPE_BF16 && !h->w8 && chain_env != nullptr && chain_env[0] == '1' &&
               chain_supported(device);
    if (h->chain) {
        const int n_top = h->max_rows < kMaxChainBn ? h->max_rows : kMaxChainBn;
        const int mt_mid[4] = {(H + 127) / 128, F / 64, (H + 127) / 128, qkv_rows / 128};
        const int mt_last[4] = {(H + 127) / 128, F / 64, (H + 127) / 128, (V + 127) / 128};
        const int kb[4] = {qd / 64, H / 64, F / 64, H / 64};
        bool ok1 = false, ok2 = false;
        const ChainPlan c1 = chain_plan(n_top, mt_mid, kb, 4, h->num_sms, &ok1);
        const ChainPlan c2 = chain_plan(n_top, mt_last, kb, 4, h->num_sms, &ok2);
        h->chain = ok1 && ok2;
        h->chain_ws_floats = c1.ws_floats > c2.ws_floats ? c1.ws_floats : c2.ws_floats;
        h->chain_tickets_n = c1.tickets > c2.tickets ? c1.tickets : c2.tickets;
    }

    int a = PE_OK;
    if (a == PE_OK) a = dev_alloc(&h->h, R * H * 4);
    if (a == PE_OK) a = dev_alloc(&h->resid, R * H * 4);
    if (a == PE_OK) a = dev_alloc(&h->u, R * 2 * H * E);
    if (a == PE_OK) a = dev_alloc(&h->xn, R * H * E);
    h->ss_ld = (((H + 127) / 128) + 3) / 4 * 4;
    if (a == PE_OK) a = dev_alloc(&h->ss, static_cast<size_t>(h->ss_ld) * R * 4);
    if (a == PE_OK) a = dev_alloc(&h->q, R * qd * E);
    if (a == PE_OK) a = dev_alloc(&h->attn, R * qd * E);
    if (a == PE_OK) a = dev_alloc(&h->act, R * F * E);
    if (a == PE_OK) a = dev_alloc(&h->amax, R * 8);
    if (a == PE_OK) a = dev_alloc(&h->row_slot, R * 4);
    if (a == PE_OK) a = dev_alloc(&h->attn_order, static_cast<size_t>(max_batch) * 4);
    if (a == PE_OK) a = dev_alloc(&h->seq_eff, static_cast<size_t>(max_batch) * 4);
    if (a == PE_OK)
        a = dev_alloc(&h->samp_stats, static_cast<size_t>(max_batch) * (2 * cfg->k_max + 1) * sizeof(float2));
    if (a == PE_OK) a = dev_alloc(&h->rope_cs, R * (hd / 2) * sizeof(float2));
    if (a == PE_OK) a = dev_alloc(&h->inv_freq, (hd / 2) * sizeof(double));
    if (a == PE_OK) a = dev_alloc(&h->gemm_ws, h->gemm_ws_floats * 4);
    if (a == PE_OK) a = dev_alloc(&h->gemm_tickets, static_cast<size_t>(h->gemm_tickets_n) * 4);
    if (a == PE_OK) a = dev_alloc(&h->attn_ws, h->attn_ws_floats * 4);
    if (a == PE_OK) a = dev_alloc(&h->attn_tickets, static_cast<size_t>(h->attn_tickets_n) * 4);
    if (a == PE_OK) a = dev_alloc(&h->attn_items, static_cast<size_t>(h->attn_items_n) * sizeof(int4));
    if (a == PE_OK) a = dev_alloc(&h->attn_plan, (1 + 2 * static_cast<size_t>(max_batch)) * 4);
    if (a == PE_OK) a = dev_alloc(&h->err, 16);
    if (h->chain) {
        if (a == PE_OK) a = dev_alloc(&h->chain_ctr, (kMaxChainPhases + 1) * sizeof(unsigned));
        if (a == PE_OK) a = dev_alloc(&h->chain_ws, h->chain_ws_floats * 4);
        if (a == PE_OK) a = dev_alloc(&h->chain_tickets, static_cast<size_t>(h->chain_tickets_n) * 4);
    }
    if (a != PE_OK) {
        free_handle(h);
        return a;
    }
    // zero what must start at zero: tickets, error word, and the activation
    // buffers (TMA reads only rows < N, but keep them defined)
    bool zok = cudaMemset(h->gemm_tickets, 0, static_cast<size_t>(h->gemm_tickets_n) * 4) == cudaSuccess &&
               cudaMemset(h->attn_tickets, 0, static_cast<size_t>(h->attn_tickets_n) * 4) == cudaSuccess &&
               cudaMemset(h->err, 0, 16) == cudaSuccess && cudaMemset(h->u, 0, R * 2 * H * E) == cudaSuccess &&
               cudaMemset(h->xn, 0, R * H * E) == cudaSuccess && cudaMemset(h->attn, 0, R * qd * E) == cudaSuccess &&
               cudaMemset(h->act, 0, R * F * E) == cudaSuccess &&
               cudaMemset(h->ss, 0, static_cast<size_t>(h->ss_ld) * R * 4) == cudaSuccess &&
               (!h->chain ||
                (cudaMemset(h->chain_ctr, 0, (kMaxChainPhases + 1) * sizeof(unsigned)) == cudaSuccess &&
                 cudaMemset(h->chain_tickets, 0, static_cast<size_t>(h->chain_tickets_n) * 4) == cudaSuccess));
    std::vector<double> inv(hd / 2);
    for (int i = 0; i < hd / 2; ++i) inv[i] = std::pow(static_cast<double>(cfg->rope_theta), -2.0 * i / hd);
    zok = zok && cudaMemcpy(h->inv_freq, inv.data(), inv.size() * sizeof(double), cudaMemcpyHostToDevice) == cudaSuccess;
    zok = zok && cudaDeviceSynchronize() == cudaSuccess;
    if (!zok) {
        free_handle(h);
        set_error("workspace initialisation failed");
        return PE_ERR_CUDA;
    }

    rc = weight_map(h, &h->tm_fc, w.fc, H, 3 * H, 128);
    if (rc == PE_OK) rc = weight_map(h, &h->tm_lm, w.lm_head, V, H, 128);
    for (int l = 0; l < 4 && rc == PE_OK; ++l) {
        const pe_layer_weights& L = w.layer[l];
        rc = weight_map(h, &h->tm_qkv[l], L.w_qkv, qkv_rows, l == 0 ? 2 * H : H, 128);
        if (rc == PE_OK) rc = weight_map(h, &h->tm_o[l], L.w_o, H, qd, 128);
        if (rc == PE_OK) rc = weight_map(h, &h->tm_gate[l], L.w_gate, F, H, 64);
        if (rc == PE_OK) rc = weight_map(h, &h->tm_up[l], L.w_up, F, H, 64);
        if (rc == PE_OK) rc = weight_map(h, &h->tm_down[l], L.w_down, H, F, 128);
    }
    if (rc != PE_OK) {
        free_handle(h);
        return rc;
    }
    *out = h;
    return PE_OK;
}

}  // namespace

extern "C" {

int pe_init_drafter(const pe_config* cfg, const pe_weights* weights, int32_t max_batch, int32_t device,
                    pe_handle** out) {
    return init_drafter(cfg, weights, nullptr, max_batch, device, out);
}

int pe_init_drafter_fp8(const pe_config* cfg, const pe_weights* weights, const pe_weight_scales* scales,
                        int32_t max_batch, int32_t device, pe_handle** out) {
    if (scales == nullptr) { set_error("null weight scales"); return PE_ERR_ARG; }
    if (cfg != nullptr && cfg->dtype != PE_DTYPE_FP8W) { set_error("pe_init_drafter_fp8 needs dtype PE_DTYPE_FP8W"); return PE_ERR_ARG; }
    return init_drafter(cfg, weights, scales, max_batch, device, out);
}

void pe_destroy(pe_handle* h) {
    if (h == nullptr) return;
    cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    free_handle(h);
}

int pe_last_launch_count(const pe_handle* h) { return h ? h->last_launches : 0; }

int pe_test_stall_chain(pe_handle* h, void* stream) {
    if (h == nullptr) { set_error("null handle"); return PE_ERR_ARG; }
    if (!h->chain) {
        set_error("the handle runs no layer chain (create it with PE_LAYER_CHAIN=1, bf16)");
        return PE_ERR_UNSUPPORTED;
    }
    // Phase 0 (the O projection) owns the first ceil(H/128) tickets. Bytes of
    // 0x01 make each ticket 0x01010101: no segment of a shared tile then sees
    // the arrival count that makes it the last, so phase 0 never completes.
    const size_t n = static_cast<size_t>((h->cfg.hidden + 127) / 128);
    PE_CUDA_TRY(cudaMemsetAsync(h->chain_tickets, 0x01, n * sizeof(int), static_cast<cudaStream_t>(stream)));
    return PE_OK;
}

int pe_device_errors(pe_handle* h, void* stream, uint32_t* out_bits) {
    if (h == nullptr || out_bits == nullptr) { set_error("null argument"); return PE_ERR_ARG; }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned bits = 0;
    PE_CUDA_TRY(cudaMemcpyAsync(&bits, h->err, sizeof(unsigned), cudaMemcpyDeviceToHost, s));
    PE_CUDA_TRY(cudaStreamSynchronize(s));
    PE_CUDA_TRY(cudaMemsetAsync(h->err, 0, sizeof(unsigned), s));
    PE_CUDA_TRY(cudaStreamSynchronize(s));
    *out_bits = bits;
    return PE_OK;
}

}  // extern "C"

namespace {

// One draft pass over B requests of ps.Kp rows each (all K rows of the
// parallel pass, or one row of a sequential pass).
struct PassSpec {
    int B = 0, Kp = 0;
    int j0 = 0;                    // entry / position offset of the pass's rows
    int k_check = 0;               // entries past S_b the step writes (validated by the first pass)
    bool run_fc = true;            // compute h = W_fc [h_lo; h_mid; h_hi] first
    const int32_t* tok = nullptr;  // row-0 token of request b: tok[b * tok_stride]
    int tok_stride = 1;
    const float* hid = nullptr;    // row-0 hidden of request b (null: the FC output)
    int hid_stride = 0;
    bool status_in = false;        // status was written by an earlier pass of the step
    bool seq_eff_out = false;      // the attention reads S_b + j0 from the workspace
    int32_t* drafts = nullptr;     // drafts[b * drafts_stride + j]
    int drafts_stride = 0;
    float* logits = nullptr;       // optional: pass row n (= b * Kp + j) at logits + n * logits_ld
    int logits_ld = 0;
    // re-fed real rows (see RowBuildParams): rows j < n_lead take their own
    // token and FC output, at a per-request row offset; padding rows
    int n_lead = 1;
    int tok_jstride = 0;
    int fc_rows = 1;               // FC rows per request (hidden rows read at b * fc_rows + o_b + j)
    const int32_t* row_off = nullptr;
    int off_add = 0;
    const int32_t* row_lim = nullptr;
    int lim_add = 0;
    const int32_t* n_real = nullptr;
    int n_max = 0;
    bool head = true;              // run the LM head and the argmax (off: the rows only feed the cache)
};

int enqueue_pass(pe_handle* h, const PassSpec& ps, const void* target_hidden, const int32_t* positions,
                 const int32_t* seq_lens, const int32_t* page_table, int32_t max_pages, int32_t num_pages,
                 void* k_cache, void* v_cache, int32_t* status, cudaStream_t s, int& launches) {
    const pe_config& c = h->cfg;
    const int H = c.hidden, F = c.ffn, V = c.vocab, hd = c.head_dim, nq = c.n_q_heads, nkv = c.n_kv_heads;
    const int qd = nq * hd, qkv_rows = (nq + 2 * nkv) * hd;
    const int B = ps.B, K = ps.Kp;
    const int R = B * K;
    const int eb = static_cast<int>(h->elem);
    const int dt = c.dtype;
    const bool pdl = h->pdl;
    int rc;

    // GEMM plans (bn depends only on the row count)
    const int fc_n = B * ps.fc_rows;
    const GemmPlan p_fc = plan_gemm(H, fc_n, 3 * H, EPI_STORE, eb, h->num_sms, true, h->w8);
    const GemmPlan p_qkv0 = plan_gemm(qkv_rows, R, 2 * H, EPI_QKV, eb, h->num_sms, true, h->w8);
    const GemmPlan p_qkv = plan_gemm(qkv_rows, R, H, EPI_QKV, eb, h->num_sms, true, h->w8);
    const GemmPlan p_o = plan_gemm(H, R, qd, EPI_RESID, eb, h->num_sms, true, h->w8);
    const GemmPlan p_gu = plan_gemm(F, R, H, EPI_SWIGLU, eb, h->num_sms, true, h->w8);
    const GemmPlan p_down = plan_gemm(H, R, F, EPI_RESID, eb, h->num_sms, true, h->w8);
    const GemmPlan p_lm = plan_gemm(V, R, H, EPI_ARGMAX, eb, h->num_sms, true, h->w8);
    const bool attn_umma = dt == PE_DTYPE_BF16;
    const AttnPlan p_at = attn_umma ? plan_attention_umma(B, K, nq, nkv, hd, max_pages, c.page_size, h->num_sms)
                                  : plan_attention(B, K, nq, nkv, hd, max_pages, c.page_size, h->num_sms);
    if (p_at.ws_floats > h->attn_ws_floats) { set_error("attention scratch too small for this max_pages"); return PE_ERR_ARG; }
    if (p_at.pieces && (p_at.grid > h->attn_items_n ||
                        static_cast<size_t>(p_at.grid) * attn_piece_floats(K * (nq / nkv), hd) > h->attn_ws_floats)) {
        set_error("attention piece scratch too small");
        return PE_ERR_ARG;
    }

    // B-operand maps: the box height is the token tile of the GEMM that reads
    // the map (QKV, O and down may take narrower tiles than gate/up and the LM head)
    CUtensorMap tm_th, tm_u, tm_xq, tm_xn, tm_xn_lm, tm_attn, tm_act;
    if (p_qkv0.bn != p_qkv.bn) { set_error("GEMM token tiles disagree"); return PE_ERR_UNSUPPORTED; }
    if (ps.run_fc && (rc = act_map(h, &tm_th, target_hidden, fc_n, 3 * H, p_fc.bn)) != PE_OK) return rc;
    if ((rc = act_map(h, &tm_u, h->u, R, 2 * H, p_qkv.bn)) != PE_OK) return rc;      // layer 0's QKV
    if ((rc = act_map(h, &tm_xq, h->xn, R, H, p_qkv.bn)) != PE_OK) return rc;       // QKV of layers 1-3
    if ((rc = act_map(h, &tm_xn, h->xn, R, H, p_gu.bn)) != PE_OK) return rc;        // gate/up
    if ((rc = act_map(h, &tm_xn_lm, h->xn, R, H, p_lm.bn)) != PE_OK) return rc;     // LM head (its own token tile)
    if ((rc = act_map(h, &tm_attn, h->attn, R, qd, p_o.bn)) != PE_OK) return rc;       // B operand of O
    if ((rc = act_map(h, &tm_act, h->act, R, F, p_down.bn)) != PE_OK) return rc;       // B operand of down
    CUtensorMap tm_kc, tm_vc, tm_q;
    if (attn_umma) {
        if ((rc = encode_tmap_kv(&tm_kc, k_cache, hd, nkv, num_pages)) != PE_OK) return rc;
        if ((rc = encode_tmap_kv(&tm_vc, v_cache, hd, nkv, num_pages)) != PE_OK) return rc;
        if ((rc = encode_tmap_q(&tm_q, h->q, hd, nq, R, nq / nkv, K)) != PE_OK) return rc;
    }

    GemmParams base{};
    base.N = R;
    base.ws = h->gemm_ws;
    base.tickets = h->gemm_tickets;
    base.err = h->err;

    // RMSNorm folded into the GEMMs around it: the residual-producing GEMM
    // (O, down) also writes gain * r and per-tile sums of r^2; the consuming
    // GEMM (QKV of the next layer, gate/up, LM head) reads gain * r as its B
    // operand and scales accumulator column n by 1/rms(r[n]), which is the
    // same product because the GEMM is linear in each token row.
    auto fold_norm_out = [&](GemmParams& p, const void* gain) {
        p.xg = h->xn; p.xg_gain = gain; p.ld_xg = H; p.ss_out = h->ss; p.ss_ld = h->ss_ld;
    };
    auto fold_norm_in = [&](GemmParams& p) {
        p.ss_in = h->ss; p.ss_parts = (H + 127) / 128; p.ss_ld = h->ss_ld;
        p.ss_scale = 1.0f / static_cast<float>(H); p.ss_eps = c.rms_eps;
    };

    // Every launch goes through `run`, which counts it and, when the kernel
    // kind is being profiled, brackets it with CUDA events on stream s.
    // `kernels`: launches fn makes (one profiled interval for all of them)
    auto run = [&](int kind, auto&& fn, int kernels = 1) -> int {
        const bool prof = h->prof_kind == kind && h->prof_used + 2 <= static_cast<int>(h->prof_events.size());
        if (prof) cudaEventRecord(h->prof_events[h->prof_used], s);
        const int r = fn();
        if (r == PE_OK) launches += kernels;
        if (prof) {
            cudaEventRecord(h->prof_events[h->prof_used + 1], s);
            h->prof_used += 2;
        }
        return r;
    };

    // a1: h = W_fc [h_lo; h_mid; h_hi] (the first pass of a step)
    if (ps.run_fc) {
        GemmParams p = base;
        p.M = H; p.N = fc_n; p.Kd = 3 * H;
        p.out_f32 = h->h; p.ld_out = H;
        p.w_scale = h->sc.fc;
        rc = run(PE_KERNEL_FC, [&] { return launch_gemm(dt, EPI_STORE, h->tm_fc, h->tm_fc, tm_th, p_fc, p, s, pdl); });
        if (rc != PE_OK) return rc;
    }
    // a2: rows, slots, RoPE table, status, argmax reset
    {
        RowBuildParams rp{};
        rp.B = B; rp.K = K; rp.H = H; rp.V = V; rp.hd = hd;
        rp.max_pages = max_pages; rp.num_pages = num_pages; rp.page_size = c.page_size;
        rp.last_token = ps.tok; rp.tok_stride = ps.tok_stride;
        rp.positions = positions; rp.seq_lens = seq_lens; rp.page_table = page_table;
        rp.h = ps.hid != nullptr ? ps.hid : h->h;
        rp.hid_stride = H;
        rp.hid_bstride = ps.hid != nullptr ? ps.hid_stride : ps.fc_rows * H;
        rp.n_lead = ps.n_lead; rp.tok_jstride = ps.tok_jstride;
        rp.row_off = ps.row_off; rp.off_add = ps.off_add; rp.row_lim = ps.row_lim; rp.lim_add = ps.lim_add;
        rp.n_real = ps.n_real; rp.n_max = ps.n_max;
        rp.j0 = ps.j0; rp.k_check = ps.k_check; rp.status_in = ps.status_in ? 1 : 0;
        rp.seq_eff = ps.j0 > 0 || ps.seq_eff_out || ps.row_off != nullptr ? h->seq_eff : nullptr;
        rp.embed = h->w.embed; rp.emb_mask = h->w.emb_mask; rp.h_shared = h->w.h_shared;
        rp.norm_e = h->w.layer[0].norm_e; rp.norm_h = h->w.layer[0].norm_h; rp.eps = c.rms_eps;
        rp.u = h->u; rp.resid = h->resid; rp.row_slot = h->row_slot; rp.rope_cs = h->rope_cs;
        rp.inv_freq = h->inv_freq; rp.amax = h->amax; rp.status = status;
        rp.order = attn_umma && B <= 1024 && !p_at.pieces ? h->attn_order : nullptr;
        rp.attn_items = p_at.pieces ? h->attn_items : nullptr;
        rp.attn_plan = h->attn_plan;
        rp.nkv = nkv;
        rp.piece_slots = p_at.piece_slots;
        rp.piece_min_tiles = p_at.piece_min_tiles;
        rp.piece_wave = p_at.piece_wave;
        if ((rc = run(PE_KERNEL_ROW_BUILD, [&] { return launch_row_build(dt, rp, s, pdl); })) != PE_OK) return rc;
    }
    const int32_t* rp_seq = ps.j0 > 0 || ps.seq_eff_out || ps.row_off != nullptr ? h->seq_eff : seq_lens;
    const size_t layer_elems = static_cast<size_t>(num_pages) * nkv * c.page_size * hd;
    auto kcache = [&](int l) { return static_cast<char*>(k_cache) + l * layer_elems * h->elem; };
    auto vcache = [&](int l) { return static_cast<char*>(v_cache) + l * layer_elems * h->elem; };
    // epilogue parameters of each GEMM of the pass
    auto gp_qkv = [&](int l) {
        GemmParams p = base;
        p.M = qkv_rows; p.Kd = l == 0 ? 2 * H : H;
        p.out_act = h->q; p.ld_act = qd;
        p.k_cache = kcache(l); p.v_cache = vcache(l); p.nq_hd = qd; p.nkv = nkv; p.hd = hd;
        p.row_slot = h->row_slot; p.rope_cs = h->rope_cs;
        p.w_scale = h->sc.layer[l].w_qkv;
        if (l > 0) fold_norm_in(p);   // attention RMSNorm of layer l
        return p;
    };
    auto gp_o = [&](int l) {      // a5: O projection + residual
        GemmParams p = base;
        p.M = H; p.Kd = qd; p.out_f32 = h->resid; p.ld_out = H;
        p.w_scale = h->sc.layer[l].w_o;
        fold_norm_out(p, h->w.layer[l].mlp_norm);
        return p;
    };
    auto gp_gu = [&](int l) {     // a6: gate/up + SwiGLU
        GemmParams p = base;
        p.M = F; p.Kd = H; p.out_act = h->act; p.ld_act = F;
        p.w_scale = h->sc.layer[l].w_gate; p.w_scale2 = h->sc.layer[l].w_up;
        fold_norm_in(p);   // MLP RMSNorm
        return p;
    };
    auto gp_down = [&](int l) {   // a6: down + residual
        GemmParams p = base;
        p.M = H; p.Kd = F; p.out_f32 = h->resid; p.ld_out = H;
        p.w_scale = h->sc.layer[l].w_down;
        fold_norm_out(p, l < 3 ? h->w.layer[l + 1].attn_norm : h->w.final_norm);
        return p;
    };
    auto gp_lm = [&]() {          // a7: LM head + fused argmax on W_lm (g * r): 1/rms(r) > 0 does not move it
        GemmParams p = base;
        p.M = V; p.Kd = H; p.amax = h->amax; p.logits = ps.logits; p.ld_logits = ps.logits_ld;
        // the LM head's first ~40 MB of weights stay in L2 between steps
        // (measured: 40 MB faster, 80 and 100 MB slower than none at B=1, B=4)
        p.keep_tiles = static_cast<int>((40LL << 20) / (128LL * H * (h->w8 ? 1LL : static_cast<long long>(h->elem))));
        p.w_scale = h->sc.lm_head;
        return p;
    };
    // O, gate/up, down of layer l and then the next layer's QKV (or the LM
    // head) as one persistent launch
    const bool use_chain = h->chain && R <= kMaxChainBn && ps.head;
    auto launch_layer_chain = [&](int l) -> int {
        ChainParams cp{};
        cp.nphases = 4;
        const CUtensorMap* a1[4] = {&h->tm_o[l], &h->tm_gate[l], &h->tm_down[l], l < 3 ? &h->tm_qkv[l + 1] : &h->tm_lm};
        const CUtensorMap* a2[4] = {&h->tm_o[l], &h->tm_up[l], &h->tm_down[l], l < 3 ? &h->tm_qkv[l + 1] : &h->tm_lm};
        const CUtensorMap* bm[4] = {&tm_attn, &tm_xn, &tm_act, l < 3 ? &tm_xn : &tm_xn_lm};
        const GemmParams gps[4] = {gp_o(l), gp_gu(l), gp_down(l), l < 3 ? gp_qkv(l + 1) : gp_lm()};
        const int epis[4] = {EPI_RESID, EPI_SWIGLU, EPI_RESID, l < 3 ? EPI_QKV : EPI_ARGMAX};
        const int mt[4] = {(H + 127) / 128, F / 64, (H + 127) / 128, l < 3 ? qkv_rows / 128 : (V + 127) / 128};
        const int kb[4] = {qd / 64, H / 64, F / 64, H / 64};
        bool ok = false;
        const ChainPlan plan = chain_plan(R, mt, kb, 4, h->num_sms, &ok);
        if (!ok || plan.ws_floats > h->chain_ws_floats || plan.tickets > h->chain_tickets_n) {
            set_error("layer chain: plan exceeds the handle's scratch");
            return PE_ERR_ARG;
        }
        long long ws_off = 0;
        int ticket_off = 0;
        for (int i = 0; i < 4; ++i) {
            ChainPhase& ph = cp.ph[i];
            ph.tmA = *a1[i];
            ph.tmA2 = *a2[i];
            ph.tmB = *bm[i];
            ph.gp = gps[i];
            ph.gp.bn = plan.bn;
            ph.epi = epis[i];
            ph.m_tiles = mt[i];
            ph.kb_total = kb[i];
            ph.max_segs = chain_max_segs(mt[i], kb[i], plan.grid);
            ph.ws_off = ws_off;
            ph.ticket_off = ticket_off;
            ws_off += static_cast<long long>(mt[i]) * ph.max_segs * plan.bn * 128;
            ticket_off += mt[i];
        }
        cp.bn = plan.bn;
        cp.stages = plan.stages;
        cp.counters = h->chain_ctr;
        cp.ws = h->chain_ws;
        cp.tickets = h->chain_tickets;
        cp.err = h->err;
        return run(PE_KERNEL_LAYER_CHAIN, [&] { return launch_chain(cp, plan, s, pdl); });
    };

    for (int l = 0; l < 4; ++l) {
        char* kc = kcache(l);
        char* vc = vcache(l);
        if (!use_chain || l == 0) {   // a3: QKV + RoPE + paged KV write
            GemmParams p = gp_qkv(l);
            rc = run(PE_KERNEL_QKV, [&] {
                return launch_gemm(dt, EPI_QKV, h->tm_qkv[l], h->tm_qkv[l], l == 0 ? tm_u : tm_xq,
                                   l == 0 ? p_qkv0 : p_qkv, p, s, pdl);
            });
            if (rc != PE_OK) return rc;
        }
        {   // a4: paged attention
            AttnParams ap{};
            ap.B = B; ap.K = K; ap.nq = nq; ap.nkv = nkv; ap.hd = hd;
            ap.max_pages = max_pages; ap.num_pages = num_pages; ap.page_size = c.page_size;
            ap.chunk = p_at.chunk; ap.max_splits = p_at.max_splits;
            ap.q = h->q; ap.k_cache = kc; ap.v_cache = vc; ap.page_table = page_table;
            ap.seq_lens = rp_seq;   // S_b + j0: the entries committed before this pass's rows
            ap.status = status; ap.out = h->attn;
            ap.order = attn_umma && B <= 1024 ? h->attn_order : nullptr; ap.ws = h->attn_ws; ap.tickets = h->attn_tickets; ap.err = h->err;
            ap.layer_page0 = l * num_pages;
            ap.items = p_at.pieces ? h->attn_items : nullptr;
            ap.plan = h->attn_plan;
            ap.grid = p_at.grid;
            ap.l2_prefetch = p_at.one_wave ? 1 : 0;   // with a second wave, early prefetches only compete
            // with length-aware pieces the merge kernel follows in the same
            // profiled interval (one attention per layer)
            rc = run(
                PE_KERNEL_ATTENTION,
                [&] {
                    if (!attn_umma) return launch_attention(dt, ap, s, pdl);
                    const int r = launch_attention_umma(tm_q, tm_kc, tm_vc, ap, s, pdl);
                    return (r == PE_OK && p_at.pieces) ? launch_attention_merge(ap, s, pdl) : r;
                },
                p_at.pieces ? 2 : 1);
            if (rc != PE_OK) return rc;
        }
        if (use_chain) {
            if ((rc = launch_layer_chain(l)) != PE_OK) return rc;
            continue;
        }
        {
            GemmParams p = gp_o(l);
            rc = run(PE_KERNEL_O_PROJ,
                     [&] { return launch_gemm(dt, EPI_RESID, h->tm_o[l], h->tm_o[l], tm_attn, p_o, p, s, pdl); });
            if (rc != PE_OK) return rc;
        }
        {
            GemmParams p = gp_gu(l);
            rc = run(PE_KERNEL_GATE_UP,
                     [&] { return launch_gemm(dt, EPI_SWIGLU, h->tm_gate[l], h->tm_up[l], tm_xn, p_gu, p, s, pdl); });
            if (rc != PE_OK) return rc;
            GemmParams d = gp_down(l);
            rc = run(PE_KERNEL_DOWN,
                     [&] { return launch_gemm(dt, EPI_RESID, h->tm_down[l], h->tm_down[l], tm_act, p_down, d, s, pdl); });
            if (rc != PE_OK) return rc;
        }
    }
    if (!ps.head) return PE_OK;
    // a7: final norm (folded), LM head + fused argmax (inside the last chain launch when chained)
    if (!use_chain) {
        GemmParams p = gp_lm();
        rc = run(PE_KERNEL_LM_HEAD,
                 [&] { return launch_gemm(dt, EPI_ARGMAX, h->tm_lm, h->tm_lm, tm_xn_lm, p_lm, p, s, pdl); });
        if (rc != PE_OK) return rc;
    }
    if (ps.logits != nullptr) {
        rc = run(PE_KERNEL_LM_HEAD, [&] {
            return launch_logits_rms_scale(ps.logits, R, V, ps.logits_ld, h->ss, h->ss_ld,
                                           1.0f / static_cast<float>(H), c.rms_eps, s, pdl);
        });
        if (rc != PE_OK) return rc;
    }
    rc = run(PE_KERNEL_ARGMAX,
             [&] { return launch_argmax_finalize(h->amax, status, B, K, ps.drafts, ps.drafts_stride, s, pdl); });
    if (rc != PE_OK) return rc;
    return PE_OK;
}


int check_draft_args(pe_handle* h, int32_t B, int32_t K, const int32_t* last_token, const void* target_hidden,
                     const int32_t* positions, const int32_t* seq_lens, const int32_t* page_table, int32_t max_pages,
                     int32_t num_pages, void* k_cache, void* v_cache, int32_t* drafts, int32_t* status) {
    if (h == nullptr) { set_error("null handle"); return PE_ERR_ARG; }
    if (B < 1 || B > h->max_batch) { set_error("B out of range 1..max_batch"); return PE_ERR_ARG; }
    if (K < 1 || K > h->cfg.k_max) { set_error("K out of range 1..k_max"); return PE_ERR_ARG; }
    if (!last_token || !target_hidden || !positions || !seq_lens || !page_table || !k_cache || !v_cache || !drafts ||
        !status) {
        set_error("null tensor argument");
        return PE_ERR_ARG;
    }
    if (max_pages < 1 || num_pages < 1) { set_error("max_pages and num_pages must be >= 1"); return PE_ERR_ARG; }
    return PE_OK;
}

}  // namespace

extern "C" {

int pe_draft(pe_handle* h, int32_t B, int32_t K, const int32_t* last_token, const void* target_hidden,
             const int32_t* positions, const int32_t* seq_lens, const int32_t* page_table, int32_t max_pages,
             int32_t num_pages, void* k_cache, void* v_cache, int32_t* drafts, float* logits_dbg, int32_t* status,
             void* stream) {
    int rc = check_draft_args(h, B, K, last_token, target_hidden, positions, seq_lens, page_table, max_pages,
                              num_pages, k_cache, v_cache, drafts, status);
    if (rc != PE_OK) return rc;
    PassSpec ps;
    ps.B = B; ps.Kp = K; ps.j0 = 0; ps.k_check = K; ps.run_fc = true;
    ps.tok = last_token; ps.tok_stride = 1;
    ps.drafts = drafts; ps.drafts_stride = K;
    ps.logits = logits_dbg; ps.logits_ld = h->cfg.vocab;
    int launches = 0;
    rc = enqueue_pass(h, ps, target_hidden, positions, seq_lens, page_table, max_pages, num_pages, k_cache, v_cache,
                      status, static_cast<cudaStream_t>(stream), launches);
    if (rc != PE_OK) return rc;
    h->last_launches = launches;
    return PE_OK;
}

int pe_draft_sequential(pe_handle* h, int32_t B, int32_t K, const int32_t* last_token, const void* target_hidden,
                        const int32_t* positions, const int32_t* seq_lens, const int32_t* page_table,
                        int32_t max_pages, int32_t num_pages, void* k_cache, void* v_cache, int32_t* drafts,
                        float* logits_dbg, int32_t* status, void* stream) {
    int rc = check_draft_args(h, B, K, last_token, target_hidden, positions, seq_lens, page_table, max_pages,
                              num_pages, k_cache, v_cache, drafts, status);
    if (rc != PE_OK) return rc;
    const int H = h->cfg.hidden, V = h->cfg.vocab;
    int launches = 0;
    for (int j = 0; j < K; ++j) {
        PassSpec ps;
        ps.B = B; ps.Kp = 1; ps.j0 = j; ps.k_check = K;
        ps.run_fc = j == 0;
        // pass 0: the last accepted token and the fused target hidden state;
        // pass j: draft j-1 and the drafter's own final residual of pass j-1
        ps.tok = j == 0 ? last_token : drafts + (j - 1);
        ps.tok_stride = j == 0 ? 1 : K;
        ps.hid = j == 0 ? nullptr : h->resid;
        ps.hid_stride = H;
        ps.status_in = j > 0;
        ps.seq_eff_out = true;
        ps.drafts = drafts + j; ps.drafts_stride = K;
        ps.logits = logits_dbg != nullptr ? logits_dbg + static_cast<size_t>(j) * V : nullptr;
        ps.logits_ld = K * V;
        rc = enqueue_pass(h, ps, target_hidden, positions, seq_lens, page_table, max_pages, num_pages, k_cache,
                          v_cache, status, static_cast<cudaStream_t>(stream), launches);
        if (rc != PE_OK) return rc;
    }
    h->last_launches = launches;
    return PE_OK;
}

int pe_draft_refeed(pe_handle* h, int32_t B, int32_t K, int32_t n_max, const int32_t* tokens,
                    const int32_t* n_real, const void* target_hidden, const int32_t* positions,
                    const int32_t* seq_lens, const int32_t* page_table, int32_t max_pages, int32_t num_pages,
                    void* k_cache, void* v_cache, int32_t* drafts, float* logits_dbg, int32_t* status,
                    void* stream) {
    int rc = check_draft_args(h, B, K, tokens, target_hidden, positions, seq_lens, page_table, max_pages, num_pages,
                              k_cache, v_cache, drafts, status);
    if (rc != PE_OK) return rc;
    if (n_real == nullptr) { set_error("null n_real"); return PE_ERR_ARG; }
    if (n_max < 1 || n_max > h->cfg.k_max) { set_error("n_max out of range 1..k_max"); return PE_ERR_ARG; }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    // Pass A: real rows 0 .. n_b-2 of every request (right-padded to n_max-1
    // rows) through the layers, which writes their cache rows; no LM head.
    // The FC runs here for all n_max hidden rows of every request.
    // Pass B: the parallel pass with the last real row as row 0 and the K-1
    // placeholders, at entry offset n_b - 1; it attends over pass A's rows.
    PassSpec a;
    a.B = B; a.Kp = n_max - 1; a.j0 = 0; a.k_check = n_max + K - 1;
    a.run_fc = true; a.fc_rows = n_max;
    a.tok = tokens; a.tok_stride = n_max; a.tok_jstride = 1;
    a.n_lead = n_max - 1;
    a.row_lim = n_real; a.lim_add = -1;
    a.n_real = n_real; a.n_max = n_max;
    a.seq_eff_out = true;
    a.head = false;
    if (n_max > 1) {
        rc = enqueue_pass(h, a, target_hidden, positions, seq_lens, page_table, max_pages, num_pages, k_cache,
                          v_cache, status, s, launches);
        if (rc != PE_OK) return rc;
    }
    PassSpec b;
    b.B = B; b.Kp = K; b.j0 = 0; b.k_check = n_max + K - 1;
    b.run_fc = n_max == 1; b.fc_rows = n_max;
    b.tok = tokens; b.tok_stride = n_max; b.tok_jstride = 1;
    b.n_lead = 1;
    b.row_off = n_real; b.off_add = -1;
    b.n_real = n_real; b.n_max = n_max;
    b.status_in = n_max > 1;
    b.seq_eff_out = true;
    b.drafts = drafts; b.drafts_stride = K;
    b.logits = logits_dbg; b.logits_ld = h->cfg.vocab;
    rc = enqueue_pass(h, b, target_hidden, positions, seq_lens, page_table, max_pages, num_pages, k_cache, v_cache,
                      status, s, launches);
    if (rc != PE_OK) return rc;
    h->last_launches = launches;
    return PE_OK;
}

int pe_profile_start(pe_handle* h, int32_t kernel_kind, int32_t max_launches) {
    if (h == nullptr || kernel_kind < 0 || kernel_kind >= PE_KERNEL_COUNT || max_launches < 1) {
        set_error("bad profiling arguments");
        return PE_ERR_ARG;
    }
    for (cudaEvent_t e : h->prof_events) cudaEventDestroy(e);
    h->prof_events.assign(2 * static_cast<size_t>(max_launches), nullptr);
    for (auto& e : h->prof_events) PE_CUDA_TRY(cudaEventCreate(&e));
    h->prof_used = 0;
    h->prof_kind = kernel_kind;
    return PE_OK;
}

int pe_profile_stop(pe_handle* h, float* total_ms, int32_t* launches) {
    if (h == nullptr || total_ms == nullptr || launches == nullptr) { set_error("null argument"); return PE_ERR_ARG; }
    double total = 0.0;
    int n = 0;
    for (int i = 0; i + 1 < h->prof_used; i += 2) {
        PE_CUDA_TRY(cudaEventSynchronize(h->prof_events[i + 1]));
        float ms = 0.f;
        PE_CUDA_TRY(cudaEventElapsedTime(&ms, h->prof_events[i], h->prof_events[i + 1]));
        total += ms;
        ++n;
    }
    for (cudaEvent_t e : h->prof_events) cudaEventDestroy(e);
    h->prof_events.clear();
    h->prof_used = 0;
    h->prof_kind = -1;
    *total_ms = static_cast<float>(total);
    *launches = n;
    return PE_OK;
}

const char* pe_kernel_name(int32_t kind) {
    static const char* names[PE_KERNEL_COUNT] = {"fc_gemm", "row_build", "rmsnorm", "qkv_rope_kv_gemm",
                                                 "paged_attention", "o_proj_resid_gemm", "gate_up_swiglu_gemm",
                                                 "down_resid_gemm", "lm_head_argmax_gemm", "argmax_finalize",
                                                 "layer_chain"};
    return (kind >= 0 && kind < PE_KERNEL_COUNT) ? names[kind] : "unknown";
}

int pe_verify_rebuild(pe_handle* h, int32_t B, int32_t K, const int32_t* drafts, const int32_t* target_tokens,
                      const int32_t* page_table, int32_t max_pages, int32_t num_pages, const int32_t* positions,
                      const int32_t* seq_lens, int32_t* positions_out, int32_t* seq_lens_out, int32_t* accepted,
                      int32_t* bonus, int32_t* emitted, int32_t* slot_mapping, int32_t* rollback_slots,
                      int32_t* status, void* stream) {
    (void)h;
    if (B < 1) { set_error("B must be >= 1"); return PE_ERR_ARG; }
    if (K < 1 || K > 31) { set_error("K must be in 1..31"); return PE_ERR_ARG; }
    if (max_pages < 1 || num_pages < 1) { set_error("max_pages and num_pages must be >= 1"); return PE_ERR_ARG; }
    if (!drafts || !target_tokens || !page_table || !positions || !seq_lens || !positions_out || !seq_lens_out ||
        !accepted || !bonus || !slot_mapping || !rollback_slots || !status) {
        set_error("null tensor argument");
        return PE_ERR_ARG;
    }
    return launch_verify_rebuild(B, K, drafts, target_tokens, page_table, max_pages, num_pages, 16, positions,
                                 seq_lens, positions_out, seq_lens_out, accepted, bonus, emitted, slot_mapping,
                                 rollback_slots, status, static_cast<cudaStream_t>(stream));
}

int pe_verify_rebuild_refeed(pe_handle* h, int32_t B, int32_t K, const int32_t* drafts,
                             const int32_t* target_tokens, const int32_t* page_table, int32_t max_pages,
                             int32_t num_pages, const int32_t* n_real, const int32_t* positions,
                             const int32_t* seq_lens, int32_t* n_real_out, int32_t* positions_out,
                             int32_t* seq_lens_out, int32_t* accepted, int32_t* bonus, int32_t* emitted,
                             int32_t* slot_mapping, int32_t* rollback_slots, int32_t* status, void* stream) {
    (void)h;
    if (B < 1) { set_error("B must be >= 1"); return PE_ERR_ARG; }
    if (K < 1 || K > 16) { set_error("K must be in 1..16"); return PE_ERR_ARG; }
    if (max_pages < 1 || num_pages < 1) { set_error("max_pages and num_pages must be >= 1"); return PE_ERR_ARG; }
    if (!drafts || !target_tokens || !page_table || !n_real || !positions || !seq_lens || !n_real_out ||
        !positions_out || !seq_lens_out || !accepted || !bonus || !slot_mapping || !rollback_slots || !status) {
        set_error("null tensor argument");
        return PE_ERR_ARG;
    }
    return launch_verify_rebuild_refeed(B, K, drafts, target_tokens, page_table, max_pages, num_pages, 16, n_real,
                                        positions, seq_lens, n_real_out, positions_out, seq_lens_out, accepted, bonus,
                                        emitted, slot_mapping, rollback_slots, status,
                                        static_cast<cudaStream_t>(stream));
}

int pe_sample_drafts(pe_handle* h, int32_t B, int32_t K, const float* logits, float temperature, const float* u,
                     const int32_t* status, int32_t* drafts, void* stream) {
    if (h == nullptr) { set_error("null handle"); return PE_ERR_ARG; }
    if (B < 1 || B > h->max_batch || K < 1 || K > h->cfg.k_max) { set_error("B or K out of range"); return PE_ERR_ARG; }
    if (!logits || !u || !drafts) { set_error("null tensor argument"); return PE_ERR_ARG; }
    if (!(temperature > 0.f)) { set_error("temperature must be > 0"); return PE_ERR_ARG; }
    return launch_sample_rows(logits, B * K, h->cfg.vocab, temperature, u, status, K, drafts,
                              static_cast<cudaStream_t>(stream));
}

int pe_verify_stochastic(pe_handle* h, int32_t B, int32_t K, const int32_t* drafts, const float* draft_logits,
                         const float* target_logits, float temperature, const float* u_accept, const float* u_final,
                         const int32_t* page_table, int32_t max_pages, int32_t num_pages, const int32_t* positions,
                         const int32_t* seq_lens, int32_t* positions_out, int32_t* seq_lens_out, int32_t* accepted,
                         int32_t* final_token, int32_t* emitted, int32_t* slot_mapping, int32_t* rollback_slots,
                         int32_t* status, void* stream) {
    if (h == nullptr) { set_error("null handle"); return PE_ERR_ARG; }
    if (B < 1 || B > h->max_batch || K < 1 || K > h->cfg.k_max) { set_error("B or K out of range"); return PE_ERR_ARG; }
    if (!(temperature > 0.f)) { set_error("temperature must be > 0"); return PE_ERR_ARG; }
    if (max_pages < 1 || num_pages < 1) { set_error("max_pages and num_pages must be >= 1"); return PE_ERR_ARG; }
    if (!drafts || !draft_logits || !target_logits || !u_accept || !u_final || !page_table || !positions ||
        !seq_lens || !positions_out || !seq_lens_out || !accepted || !final_token || !slot_mapping ||
        !rollback_slots || !status) {
        set_error("null tensor argument");
        return PE_ERR_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = launch_stochastic_accept(B, K, h->cfg.vocab, temperature, drafts, draft_logits, target_logits, u_accept,
                                      u_final, h->samp_stats, accepted, final_token, s);
    if (rc != PE_OK) return rc;
    return launch_rebuild_given_acceptance(B, K, drafts, page_table, max_pages, num_pages, 16, positions, seq_lens,
                                           positions_out, seq_lens_out, accepted, final_token, emitted, slot_mapping,
                                           rollback_slots, status, s);
}

int pe_linear_scratch(int32_t dtype, int32_t M, int32_t N, int32_t Kd, int64_t* ws_floats, int32_t* n_tickets) {
    if (ws_floats == nullptr || n_tickets == nullptr) { set_error("null argument"); return PE_ERR_ARG; }
    if (dtype != PE_DTYPE_BF16 && dtype != PE_DTYPE_FP32 && dtype != PE_DTYPE_FP8W) {
        set_error("unknown dtype");
        return PE_ERR_ARG;
    }
    if (M < 1 || N < 1 || Kd < 1) { set_error("M, N, Kd must be >= 1"); return PE_ERR_ARG; }
    int dev = 0, sms = 0;
    PE_CUDA_TRY(cudaGetDevice(&dev));
    PE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const GemmPlan g = plan_gemm(M, N, Kd, EPI_STORE, dtype == PE_DTYPE_FP32 ? 4 : 2, sms, false,
                                 dtype == PE_DTYPE_FP8W);
    *ws_floats = static_cast<int64_t>(g.ws_floats);
    *n_tickets = g.tiles;
    return PE_OK;
}

int pe_linear(int32_t dtype, int32_t M, int32_t N, int32_t Kd, const void* w, const void* x, float* y, float* ws,
              int32_t* tickets, void* stream) {
    if (!w || !x || !y || !tickets) { set_error("null tensor argument"); return PE_ERR_ARG; }
    if (dtype != PE_DTYPE_BF16 && dtype != PE_DTYPE_FP32) { set_error("unknown dtype"); return PE_ERR_ARG; }
    if (M < 1 || N < 1 || Kd < 1 || Kd % 8 != 0) { set_error("need M, N >= 1 and Kd a positive multiple of 8"); return PE_ERR_ARG; }
    int dev = 0, sms = 0;
    PE_CUDA_TRY(cudaGetDevice(&dev));
    PE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const int eb = dtype == PE_DTYPE_BF16 ? 2 : 4;
    const GemmPlan g = plan_gemm(M, N, Kd, EPI_STORE, eb, sms, false);
    if (g.ws_floats > 0 && ws == nullptr) { set_error("this shape needs split-K scratch"); return PE_ERR_ARG; }
    CUtensorMap ta, tb;
    int rc = encode_tmap_2d(&ta, w, dtype, Kd, M, static_cast<uint64_t>(Kd) * eb, 128 / eb, 128);
    if (rc == PE_OK) rc = encode_tmap_2d(&tb, x, dtype, Kd, N, static_cast<uint64_t>(Kd) * eb, 128 / eb, g.bn);
    if (rc != PE_OK) return rc;
    GemmParams p{};
    p.M = M; p.N = N; p.Kd = Kd; p.out_f32 = y; p.ld_out = M; p.ws = ws; p.tickets = tickets; p.err = nullptr;
    return launch_gemm(dtype, EPI_STORE, ta, ta, tb, g, p, static_cast<cudaStream_t>(stream), false);
}

int pe_linear_fp8(int32_t M, int32_t N, int32_t Kd, const void* w, const float* w_scale, const void* x, float* y,
                  float* ws, int32_t* tickets, void* stream) {
    if (!w || !w_scale || !x || !y || !tickets) { set_error("null tensor argument"); return PE_ERR_ARG; }
    if (M < 1 || N < 1 || Kd < 16 || Kd % 16 != 0) {
        set_error("need M, N >= 1 and Kd a positive multiple of 16");
        return PE_ERR_ARG;
    }
    int dev = 0, sms = 0;
    PE_CUDA_TRY(cudaGetDevice(&dev));
    PE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const GemmPlan g = plan_gemm(M, N, Kd, EPI_STORE, 2, sms, false, true);
    if (g.ws_floats > 0 && ws == nullptr) { set_error("this shape needs split-K scratch"); return PE_ERR_ARG; }
    CUtensorMap ta, tb;
    int rc = encode_tmap_2d_u8(&ta, w, static_cast<uint64_t>(Kd), static_cast<uint64_t>(M), 128);
    if (rc == PE_OK) rc = encode_tmap_2d(&tb, x, PE_DTYPE_BF16, Kd, N, static_cast<uint64_t>(Kd) * 2, 64, g.bn);
    if (rc != PE_OK) return rc;
    GemmParams p{};
    p.M = M; p.N = N; p.Kd = Kd; p.out_f32 = y; p.ld_out = M; p.ws = ws; p.tickets = tickets; p.err = nullptr;
    p.w_scale = w_scale;
    return launch_gemm(PE_DTYPE_BF16, EPI_STORE, ta, ta, tb, g, p, static_cast<cudaStream_t>(stream), false);
}

struct pe_step_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int launches = 0;
};

int pe_step_graph_create_ex(pe_handle* h, int32_t draft_mode, int32_t B, int32_t K, const int32_t* last_token,
                            const void* target_hidden, const int32_t* positions, const int32_t* seq_lens,
                            const int32_t* page_table, int32_t max_pages, int32_t num_pages, void* k_cache,
                            void* v_cache, int32_t* drafts, int32_t* draft_status, const int32_t* target_tokens,
                            int32_t* positions_out, int32_t* seq_lens_out, int32_t* accepted, int32_t* bonus,
                            int32_t* emitted, int32_t* slot_mapping, int32_t* rollback_slots,
                            int32_t* verify_status, pe_step_graph** out) {
    if (h == nullptr || out == nullptr) { set_error("null argument"); return PE_ERR_ARG; }
    if (draft_mode != PE_DRAFT_PARALLEL && draft_mode != PE_DRAFT_SEQUENTIAL) {
        set_error("unknown draft mode");
        return PE_ERR_ARG;
    }
    *out = nullptr;
    PE_CUDA_TRY(cudaSetDevice(h->device));
    cudaStream_t cs = nullptr;
    PE_CUDA_TRY(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
    const int saved_prof = h->prof_kind;
    h->prof_kind = -1;   // no profiling events inside a graph
    cudaError_t ce = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
    int rc = ce == cudaSuccess ? PE_OK : PE_ERR_CUDA;
    if (rc == PE_OK) {
        auto draft = draft_mode == PE_DRAFT_PARALLEL ? pe_draft : pe_draft_sequential;
        rc = draft(h, B, K, last_token, target_hidden, positions, seq_lens, page_table, max_pages, num_pages,
                   k_cache, v_cache, drafts, nullptr, draft_status, cs);
    }
    const int n_draft = h->last_launches;
    if (rc == PE_OK)
        rc = pe_verify_rebuild(h, B, K, drafts, target_tokens, page_table, max_pages, num_pages, positions, seq_lens,
                               positions_out, seq_lens_out, accepted, bonus, emitted, slot_mapping, rollback_slots,
                               verify_status, cs);
    cudaGraph_t graph = nullptr;
    const cudaError_t ee = cudaStreamEndCapture(cs, &graph);
    h->prof_kind = saved_prof;
    cudaStreamDestroy(cs);
    if (rc != PE_OK || ee != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        if (rc == PE_OK) set_error(std::string("graph capture failed: ") + cudaGetErrorString(ee));
        return rc == PE_OK ? PE_ERR_CUDA : rc;
    }
    cudaGraphExec_t exec = nullptr;
    const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
    if (ie != cudaSuccess) {
        cudaGraphDestroy(graph);
        set_error(std::string("cudaGraphInstantiate: ") + cudaGetErrorString(ie));
        return PE_ERR_CUDA;
    }
    pe_step_graph* g = new pe_step_graph();
    g->graph = graph;
    g->exec = exec;
    g->launches = n_draft + 1;
    *out = g;
    return PE_OK;
}

int pe_step_graph_create(pe_handle* h, int32_t B, int32_t K, const int32_t* last_token, const void* target_hidden,
                         const int32_t* positions, const int32_t* seq_lens, const int32_t* page_table,
                         int32_t max_pages, int32_t num_pages, void* k_cache, void* v_cache, int32_t* drafts,
                         int32_t* draft_status, const int32_t* target_tokens, int32_t* positions_out,
                         int32_t* seq_lens_out, int32_t* accepted, int32_t* bonus, int32_t* emitted,
                         int32_t* slot_mapping, int32_t* rollback_slots, int32_t* verify_status,
                         pe_step_graph** out) {
    return pe_step_graph_create_ex(h, PE_DRAFT_PARALLEL, B, K, last_token, target_hidden, positions, seq_lens,
                                   page_table, max_pages, num_pages, k_cache, v_cache, drafts, draft_status,
                                   target_tokens, positions_out, seq_lens_out, accepted, bonus, emitted, slot_mapping,
                                   rollback_slots, verify_status, out);
}

int pe_step_graph_launch(pe_step_graph* g, void* stream) {
    if (g == nullptr) { set_error("null graph"); return PE_ERR_ARG; }
    PE_CUDA_TRY(cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream)));
    return PE_OK;
}

int pe_step_graph_launch_count(const pe_step_graph* g) { return g ? g->launches : 0; }

void pe_step_graph_destroy(pe_step_graph* g) {
    if (g == nullptr) return;
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
}

}  // extern "C"
