// Row construction and argmax finalisation.
//
// k_row_build builds the K input rows of every request (P-EAGLE post,
// "Solution overview / step-by-step drafting", Step 2): row 0 from the real
// token embedding and the FC-fused target hidden state, rows 1..K-1 from the
// learned mask embedding emb_mask and the shared hidden state h_shared. Layer
// 0 attends over the 2H concat [RMSNorm_e(emb); RMSNorm_h(hid)] and its
// residual stream starts at `hid`. The same kernel validates each request,
// computes each row's cache slot (entry S_b + j) and RoPE cos/sin (position
// Q_b + j), and clears the packed argmax records for this step.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace pe {
namespace {

constexpr int kRowThreads = 256;
constexpr int kMaxPieceB = 256;   // requests the attention piece list serves (= kPieceMaxBatch of
                                  // attn_umma.cu, whose planner uses pieces only up to it)
constexpr int kPieceTile = 64;    // cache entries per attention tile

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += red[w];
    return t;
}

// 4-element vector load / store of the config dtype as float4.
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ float dot4(float4 a) { return a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w; }
__device__ __forceinline__ float4 scale4(float4 a, float s, float4 g) {
    return make_float4(a.x * s * g.x, a.y * s * g.y, a.z * s * g.z, a.w * s * g.w);
}

constexpr int kMaxG = 8;   // 4-element groups per thread: H <= 4 * 8 * 256

// Status of request b: inputs, capacity, page indices of entries
// 0..S+k_check-1 (every entry the step writes).
__device__ int request_status(const RowBuildParams& p, int b) {
    const int S = p.seq_lens[b];
    const int Q = p.positions[b];
    int n_tok = 1;
    if (p.n_real != nullptr) {
        n_tok = p.n_real[b];
        if (n_tok < 1 || n_tok > p.n_max) return PE_REQ_BAD_INPUT;
    }
    if (S < 0 || Q < 0) return PE_REQ_BAD_INPUT;
    int bad_tok = 0;
    for (int i = threadIdx.x; i < n_tok; i += blockDim.x) {
        const int tok = p.last_token[static_cast<size_t>(b) * p.tok_stride + static_cast<size_t>(i) * p.tok_jstride];
        if (tok < 0 || tok >= p.V) bad_tok = 1;
    }
    if (__syncthreads_or(bad_tok)) return PE_REQ_BAD_INPUT;
    if (static_cast<long long>(S) + p.k_check > static_cast<long long>(p.max_pages) * p.page_size)
        return PE_REQ_CAPACITY;
    const int n_pages = (S + p.k_check + p.page_size - 1) / p.page_size;
    int bad = 0;
    for (int i = threadIdx.x; i < n_pages; i += blockDim.x) {
        const int pg = p.page_table[static_cast<size_t>(b) * p.max_pages + i];
        if (pg < 0 || pg >= p.num_pages) bad = 1;
    }
    bad = __syncthreads_or(bad);
    return bad ? PE_REQ_BAD_PAGE : PE_REQ_OK;
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) k_row_build(const RowBuildParams p) {
    __shared__ float red[32];
    const int r = blockIdx.x;
    const int b = r / p.K;
    const int j = r - b * p.K;
    const int H = p.H;
    const int ng = H / 4;
    const int tid = threadIdx.x;
    // weights (independent of earlier kernels) are read before the dependency wait
    float4 ge[kMaxG], gh[kMaxG], ev[kMaxG], hv[kMaxG];
#pragma unroll
    for (int i = 0; i < kMaxG; ++i) {
        const int g = tid + i * kRowThreads;
        if (g < ng) {
            ge[i] = load4(static_cast<const T*>(p.norm_e) + 4 * g);
            gh[i] = load4(static_cast<const T*>(p.norm_h) + 4 * g);
            if (j >= p.n_lead || p.row_lim != nullptr) {   // placeholder (or a padding row's stand-in)
                ev[i] = load4(static_cast<const T*>(p.emb_mask) + 4 * g);
                hv[i] = load4(static_cast<const T*>(p.h_shared) + 4 * g);
            }
        }
    }
    pdl_launch_dependents();
    pdl_wait();
    const int st = p.status_in ? p.status[b] : request_status(p, b);
    const bool ok = st == PE_REQ_OK;
    // per-request row offset (re-fed rows), only for a request that passed
    // the checks (its n_real is in range)
    auto off_of = [&](int q) { return p.row_off != nullptr ? p.row_off[q] + p.off_add : 0; };
    const int o_b = ok ? off_of(b) : 0;
    const bool pad = ok && p.row_lim != nullptr && j >= p.row_lim[b] + p.lim_add;
    if (j == 0 && tid == 0 && !p.status_in) p.status[b] = st;
    if (j == 0 && tid == 0 && p.seq_eff != nullptr) p.seq_eff[b] = p.seq_lens[b] + p.j0 + o_b;
    if (tid == 0) p.amax[r] = 0ull;
    if (r == 0 && p.order != nullptr) {
        // requests by decreasing length (ties by index, so a permutation):
        // the attention issues its longest (request, kv head) CTAs first
        // (every pass of a step adds the same j0, so S_b orders them)
        for (int q = tid; q < p.B; q += blockDim.x) {
            const int sq = p.seq_lens[q];
            int rank = 0;
            for (int o = 0; o < p.B; ++o) {
                const int so = p.seq_lens[o];
                rank += (so > sq || (so == sq && o < q)) ? 1 : 0;
            }
            p.order[rank] = q;
        }
    }
    if (r == 0 && p.attn_items != nullptr) {
        // Length-aware attention pieces. tiles_b = ceil((S_b + K) / 64) for a
        // request whose entries fit its page table (none otherwise); a piece
        // holds about tc = total tiles / piece_slots of them; pieces are
        // listed largest first (requests ranked by piece size, ties by index),
        // so the CTAs dispatched first carry the most work.
        __shared__ int s_t[kMaxPieceB], s_sz[kMaxPieceB], s_req[kMaxPieceB], s_off[kMaxPieceB + 1];
        __shared__ int s_total;
        if (tid == 0) s_total = 0;
        __syncthreads();
        const long long cap = static_cast<long long>(p.max_pages) * p.page_size;
        for (int q = tid; q < p.B; q += blockDim.x) {
            const int oq = p.row_off != nullptr ? max(0, min(p.n_max, off_of(q))) : 0;
            const int sq = p.seq_lens[q] + p.j0 + oq;
            const bool fits = sq >= p.j0 + oq && static_cast<long long>(sq) + p.K <= cap;
            const int tiles = fits ? (sq + p.K + kPieceTile - 1) / kPieceTile : 0;
            s_t[q] = tiles;
            atomicAdd(&s_total, tiles);
        }
        __syncthreads();
        const long long all = static_cast<long long>(s_total) * p.nkv;
        int tc = static_cast<int>((all + p.piece_slots - 1) / p.piece_slots);
        tc = tc < p.piece_min_tiles ? p.piece_min_tiles : tc;
        if (p.piece_wave > 0) {
            // piece_slots leaves one slot per (request, kv head) for the
            // rounding up of every request's piece count; smaller pieces
            // often still fit the wave: take the smallest size from the
            // even share up whose count does
            __shared__ int s_cnt;
            int lo = static_cast<int>((all + p.piece_wave - 1) / p.piece_wave);
            lo = lo < p.piece_min_tiles ? p.piece_min_tiles : lo;
            for (int c = lo; c < tc; ++c) {
                if (tid == 0) s_cnt = 0;
                __syncthreads();
                int part = 0;
                for (int q = tid; q < p.B; q += blockDim.x) part += s_t[q] > 0 ? (s_t[q] + c - 1) / c : 1;
                if (part > 0) atomicAdd(&s_cnt, part);
                __syncthreads();
                const bool fits = static_cast<long long>(s_cnt) * p.nkv <= p.piece_wave;
                __syncthreads();
                if (fits) {
                    tc = c;
                    break;
                }
            }
        }
        auto pieces_of = [&](int t) { return t > 0 ? (t + tc - 1) / tc : 1; };
        for (int q = tid; q < p.B; q += blockDim.x) {
            const int t = s_t[q];
            s_sz[q] = t > 0 ? (t + pieces_of(t) - 1) / pieces_of(t) : 0;
        }
        __syncthreads();
        for (int q = tid; q < p.B; q += blockDim.x) {
            const int sq = s_sz[q];
            int rank = 0;
            for (int o = 0; o < p.B; ++o) {
                const int so = s_sz[o];
                rank += (so > sq || (so == sq && o < q)) ? 1 : 0;
            }
            s_req[rank] = q;
        }
        __syncthreads();
        const int warp = tid >> 5, lane = tid & 31;
        if (warp == 0) {
            // exclusive prefix of the piece counts in rank order: each lane a
            // contiguous run of ranks, then a warp scan of the run sums
            const int per = (p.B + 31) / 32;
            const int k0 = lane * per, k1 = min(p.B, k0 + per);
            int sum = 0;
            for (int k = k0; k < k1; ++k) sum += pieces_of(s_t[s_req[k]]);
            int incl = sum;
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            int run = incl - sum;
            for (int k = k0; k < k1; ++k) {
                s_off[k] = run;
                run += pieces_of(s_t[s_req[k]]);
            }
            if (lane == 31) s_off[p.B] = incl;
        }
        __syncthreads();
        const int max_items = p.piece_slots + p.B * p.nkv;
        if (tid == 0) p.attn_plan[0] = min(s_off[p.B] * p.nkv, max_items);
        for (int k = tid; k < p.B; k += blockDim.x) {
            const int q = s_req[k];
            const int t = s_t[q];
            const int n = pieces_of(t);
            const int per_piece = s_sz[q];
            const int oq = p.row_off != nullptr ? max(0, min(p.n_max, off_of(q))) : 0;
            const int len = t > 0 ? p.seq_lens[q] + p.j0 + oq + p.K : 0;
            p.attn_plan[1 + q] = n;
            p.attn_plan[1 + p.B + q] = s_off[k];
            for (int i = 0; i < n; ++i) {
                const int e0 = i * per_piece * kPieceTile;
                const int e1 = min(len, (i + 1) * per_piece * kPieceTile);
                for (int hh = 0; hh < p.nkv; ++hh) {
                    const int idx = p.nkv * (s_off[k] + i) + hh;
                    if (idx < max_items) p.attn_items[idx] = make_int4(q, hh, e0, e1);
                }
            }
        }
    }
    if (j < p.n_lead && !pad) {
        const size_t r_src = static_cast<size_t>(o_b + j);
        const T* emb = static_cast<const T*>(p.embed) +
                       static_cast<size_t>(ok ? p.last_token[static_cast<size_t>(b) * p.tok_stride + r_src * p.tok_jstride]
                                              : 0) * H;
        const float* h0 = p.h + static_cast<size_t>(b) * p.hid_bstride + r_src * p.hid_stride;
#pragma unroll
        for (int i = 0; i < kMaxG; ++i) {
            const int g = tid + i * kRowThreads;
            if (g < ng) {
                ev[i] = load4(emb + 4 * g);
                hv[i] = load4(h0 + 4 * g);
            }
        }
    }
    float ss_e = 0.f, ss_h = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxG; ++i) {
        if (tid + i * kRowThreads < ng) {
            ss_e += dot4(ev[i]);
            ss_h += dot4(hv[i]);
        }
    }
    const float inv_e = ok ? rsqrtf(block_sum(ss_e, red) / H + p.eps) : 0.f;
    const float inv_h = ok ? rsqrtf(block_sum(ss_h, red) / H + p.eps) : 0.f;
    T* u = static_cast<T*>(p.u) + static_cast<size_t>(r) * 2 * H;
    float* resid = p.resid + static_cast<size_t>(r) * H;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kMaxG; ++i) {
        const int g = tid + i * kRowThreads;
        if (g < ng) {
            store4(u + 4 * g, scale4(ev[i], inv_e, ge[i]));
            store4(u + H + 4 * g, scale4(hv[i], inv_h, gh[i]));
            store4(resid + 4 * g, ok ? hv[i] : zero);
        }
    }

    if (tid == 0) {
        int slot = -1;
        if (ok && !pad) {
            const int e = p.seq_lens[b] + p.j0 + o_b + j;
            const int pg = p.page_table[static_cast<size_t>(b) * p.max_pages + e / p.page_size];
            slot = pg * p.page_size + e % p.page_size;
        }
        p.row_slot[r] = slot;
    }
    // RoPE table for this row: angle = (Q_b + j) * inv_freq_i in double,
    // reduced to [-pi, pi] in double, then sin/cos in float.
    const int half = p.hd / 2;
    const double pos = static_cast<double>(ok ? p.positions[b] + p.j0 + o_b + j : 0);
    for (int i = tid; i < half; i += blockDim.x) {
        const double a = pos * p.inv_freq[i];
        const double two_pi = 6.283185307179586476925286766559;
        const double red_a = a - two_pi * rint(a / two_pi);
        float sn, cs;
        sincosf(static_cast<float>(red_a), &sn, &cs);
        p.rope_cs[static_cast<size_t>(r) * half + i] = make_float2(cs, sn);
    }
}

// Debug logits of the LM head (written from the un-normalised operand g * r)
// scaled to the final RMSNorm: row n times 1/rms(r[n]), the partial sums of
// squares added in partial order as the folding GEMMs do.
__global__ void k_logits_rms_scale(float* __restrict__ logits, int V, int ld, const float* __restrict__ ss, int ss_ld,
                                   float scale, float eps) {
    pdl_launch_dependents();
    pdl_wait();
    const int n = blockIdx.y;
    float sum = 0.f;
    for (int q = 0; q < ss_ld; ++q) sum += ss[static_cast<size_t>(n) * ss_ld + q];
    const float inv = rsqrtf(sum * scale + eps);
    float* row = logits + static_cast<size_t>(n) * ld;
    for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < V; v += gridDim.x * blockDim.x) row[v] *= inv;
}

__global__ void k_argmax_finalize(const unsigned long long* __restrict__ amax, const int32_t* __restrict__ status,
                                  int B, int K, int32_t* __restrict__ drafts, int out_stride) {
    pdl_launch_dependents();
    pdl_wait();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= B * K) return;
    const int b = r / K;
    const unsigned long long key = amax[r];
    drafts[static_cast<size_t>(b) * out_stride + (r - b * K)] =
        (status[b] == PE_REQ_OK && key != 0ull) ? static_cast<int32_t>(argmax_key_index(key)) : -1;
}

}  // namespace

int launch_row_build(int dtype, const RowBuildParams& p, cudaStream_t s, bool pdl) {
    const dim3 grid(p.B * p.K), block(kRowThreads);
    if (dtype == PE_DTYPE_BF16) PE_CUDA_TRY(launch_ex(k_row_build<__nv_bfloat16>, grid, block, 0, s, pdl, p));
    else PE_CUDA_TRY(launch_ex(k_row_build<float>, grid, block, 0, s, pdl, p));
    return PE_OK;
}

int launch_logits_rms_scale(float* logits, int rows, int V, int ld, const float* ss, int ss_ld, float scale,
                            float eps, cudaStream_t s, bool pdl) {
    PE_CUDA_TRY(launch_ex(k_logits_rms_scale, dim3(16, rows), dim3(256), 0, s, pdl, logits, V, ld, ss, ss_ld, scale,
                          eps));
    return PE_OK;
}

int launch_argmax_finalize(const unsigned long long* amax, const int32_t* status, int B, int K, int32_t* drafts,
                           int out_stride, cudaStream_t s, bool pdl) {
    const int R = B * K;
    PE_CUDA_TRY(launch_ex(k_argmax_finalize, dim3((R + 127) / 128), dim3(128), 0, s, pdl, amax, status, B, K, drafts,
                          out_stride));
    return PE_OK;
}

}  // namespace pe
