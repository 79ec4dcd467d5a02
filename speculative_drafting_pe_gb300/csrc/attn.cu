// Decode-style paged GQA attention over the drafter KV cache.
//
// Row j of request b (query heads of kv head kvh) attends to cache entries
// 0 .. S_b + j: the S_b committed entries and this pass's rows 0..j, which
// the QKV epilogue has just written at entries S_b .. S_b + K - 1. Query head
// h reads kv head h / (nq / nkv); scores are scaled by 1/sqrt(hd); softmax
// is computed online in fp32.
//
// One CTA per (request, kv head, entry split). All K * (nq/nkv) query rows of
// a kv head share each KV tile, so every cache entry is read once per pass.
// Splits of one (request, kv head) are combined by the last CTA to arrive, in
// split order, from fp32 partials (unnormalised output, running max, sum).
#include <cfloat>

#include "common.cuh"
#include "internal.h"

namespace pe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 32;            // cache entries per smem tile
constexpr int kMaxRowsPerWarp = 16;  // K * nq/nkv <= 128

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

template <typename T, int HD>
__global__ void __launch_bounds__(kThreads) k_attn(const AttnParams p) {
    constexpr int kDpl = HD / 32;       // dims per lane
    constexpr int kPitch = HD + 1;
    extern __shared__ float sm[];
    __shared__ int s_last;
    pdl_launch_dependents();
    pdl_wait();

    const int pair = blockIdx.x;
    const int b = pair / p.nkv;
    const int kvh = pair - b * p.nkv;
    const int split = blockIdx.y;
    const int G = p.nq / p.nkv;
    const int K = p.K;
    const int Rq = K * G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const T* q = static_cast<const T*>(p.q);
    T* out = static_cast<T*>(p.out);
    const size_t row_stride = static_cast<size_t>(p.nq) * HD;

    if (p.status[b] != PE_REQ_OK) {
        if (split == 0) {
            for (int idx = tid; idx < Rq * HD; idx += kThreads) {
                const int qr = idx / HD, d = idx - (idx / HD) * HD;
                const int j = qr / G, g = qr - j * G;
                out[static_cast<size_t>(b * K + j) * row_stride + static_cast<size_t>(kvh * G + g) * HD + d] =
                    Elem<T>::from_f(0.f);
            }
        }
        return;
    }
    const int S = p.seq_lens[b];
    const int total = S + K;
    const int nsplit = (total + p.chunk - 1) / p.chunk;
    if (split >= nsplit) return;
    const int e0 = split * p.chunk;
    const int e1 = min(total, e0 + p.chunk);

    float* sq = sm;                          // [Rq][HD], pre-scaled
    float* sk = sq + Rq * HD;                // [kTile][HD+1]
    float* sv = sk + kTile * kPitch;
    const float scale = rsqrtf(static_cast<float>(HD));
    for (int idx = tid; idx < Rq * HD; idx += kThreads) {
        const int qr = idx / HD, d = idx - (idx / HD) * HD;
        const int j = qr / G, g = qr - j * G;
        sq[idx] = Elem<T>::to_f(q[static_cast<size_t>(b * K + j) * row_stride + static_cast<size_t>(kvh * G + g) * HD + d]) *
                  scale;
    }

    float o[kMaxRowsPerWarp][kDpl];
    float mrow[kMaxRowsPerWarp], lrow[kMaxRowsPerWarp];
#pragma unroll
    for (int ri = 0; ri < kMaxRowsPerWarp; ++ri) {
        mrow[ri] = -FLT_MAX;
        lrow[ri] = 0.f;
#pragma unroll
        for (int i = 0; i < kDpl; ++i) o[ri][i] = 0.f;
    }

    const T* kc = static_cast<const T*>(p.k_cache);
    const T* vc = static_cast<const T*>(p.v_cache);
    const int32_t* pt = p.page_table + static_cast<size_t>(b) * p.max_pages;

    for (int t0 = e0; t0 < e1; t0 += kTile) {
        __syncthreads();
        for (int idx = tid; idx < kTile * HD; idx += kThreads) {
            const int t = idx / HD, d = idx - (idx / HD) * HD;
            const int e = t0 + t;
            float kv = 0.f, vv = 0.f;
            if (e < e1) {
                const int page = pt[e >> 4];
                const size_t off = ((static_cast<size_t>(page) * p.nkv + kvh) * 16 + (e & 15)) * HD + d;
                kv = Elem<T>::to_f(kc[off]);
                vv = Elem<T>::to_f(vc[off]);
            }
            sk[t * kPitch + d] = kv;
            sv[t * kPitch + d] = vv;
        }
        __syncthreads();
        const int e = t0 + lane;
#pragma unroll
        for (int ri = 0; ri < kMaxRowsPerWarp; ++ri) {
            const int qr = warp + ri * kWarps;
            if (qr < Rq) {
                const int j = qr / G;
                const bool valid = e < e1 && e <= S + j;
                float sc = -FLT_MAX;
                if (valid) {
                    float acc = 0.f;
                    const float* qrow = sq + qr * HD;
                    const float* krow = sk + lane * kPitch;
#pragma unroll 8
                    for (int d = 0; d < HD; ++d) acc = fmaf(qrow[d], krow[d], acc);
                    sc = acc;
                }
                const float tmax = warp_max(sc);
                if (tmax > -FLT_MAX) {
                    const float mnew = fmaxf(mrow[ri], tmax);
                    const float corr = __expf(mrow[ri] - mnew);
                    const float pj = valid ? __expf(sc - mnew) : 0.f;
                    lrow[ri] = lrow[ri] * corr + warp_sum(pj);
#pragma unroll
                    for (int i = 0; i < kDpl; ++i) o[ri][i] *= corr;
                    for (int t = 0; t < kTile; ++t) {
                        const float pt_ = __shfl_sync(0xffffffffu, pj, t);
#pragma unroll
                        for (int i = 0; i < kDpl; ++i) o[ri][i] = fmaf(pt_, sv[t * kPitch + lane + 32 * i], o[ri][i]);
                    }
                    mrow[ri] = mnew;
                }
            }
        }
    }

    if (nsplit == 1) {
#pragma unroll
        for (int ri = 0; ri < kMaxRowsPerWarp; ++ri) {
            const int qr = warp + ri * kWarps;
            if (qr < Rq) {
                const int j = qr / G, g = qr - j * G;
                const float inv = lrow[ri] > 0.f ? 1.f / lrow[ri] : 0.f;
                T* dst = out + static_cast<size_t>(b * K + j) * row_stride + static_cast<size_t>(kvh * G + g) * HD;
#pragma unroll
                for (int i = 0; i < kDpl; ++i) dst[lane + 32 * i] = Elem<T>::from_f(o[ri][i] * inv);
            }
        }
        return;
    }

    // split partials: [pair][split][Rq][HD + 2] (o..., m, l)
    const int rec = HD + 2;
    float* mine = p.ws + (static_cast<size_t>(pair) * p.max_splits + split) * Rq * rec;
#pragma unroll
    for (int ri = 0; ri < kMaxRowsPerWarp; ++ri) {
        const int qr = warp + ri * kWarps;
        if (qr < Rq) {
#pragma unroll
            for (int i = 0; i < kDpl; ++i) __stcg(mine + qr * rec + lane + 32 * i, o[ri][i]);
            if (lane == 0) {
                __stcg(mine + qr * rec + HD, mrow[ri]);
                __stcg(mine + qr * rec + HD + 1, lrow[ri]);
            }
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int old = atomicAdd(p.tickets + pair, 1);
        s_last = (old == nsplit - 1) ? 1 : 0;
        if (s_last) atomicExch(p.tickets + pair, 0);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const float* base = p.ws + static_cast<size_t>(pair) * p.max_splits * Rq * rec;
    for (int qr = warp; qr < Rq; qr += kWarps) {
        float M = -FLT_MAX;
        for (int s = 0; s < nsplit; ++s) M = fmaxf(M, __ldcg(base + (static_cast<size_t>(s) * Rq + qr) * rec + HD));
        float den = 0.f;
        float num[kDpl];
#pragma unroll
        for (int i = 0; i < kDpl; ++i) num[i] = 0.f;
        for (int s = 0; s < nsplit; ++s) {
            const float* r = base + (static_cast<size_t>(s) * Rq + qr) * rec;
            const float ms = __ldcg(r + HD);
            const float ls = __ldcg(r + HD + 1);
            if (ls <= 0.f) continue;                    // no visible entry in this split
            const float w = __expf(ms - M);
            den = fmaf(ls, w, den);
#pragma unroll
            for (int i = 0; i < kDpl; ++i) num[i] = fmaf(w, __ldcg(r + lane + 32 * i), num[i]);
        }
        const int j = qr / G, g = qr - j * G;
        const float inv = den > 0.f ? 1.f / den : 0.f;
        T* dst = out + static_cast<size_t>(b * K + j) * row_stride + static_cast<size_t>(kvh * G + g) * HD;
#pragma unroll
        for (int i = 0; i < kDpl; ++i) dst[lane + 32 * i] = Elem<T>::from_f(num[i] * inv);
    }
}

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

template <typename T, int HD>
int launch_hd(const AttnParams& p, cudaStream_t s, bool pdl) {
    const int Rq = p.K * (p.nq / p.nkv);
    const size_t smem = (static_cast<size_t>(Rq) * HD + 2 * kTile * (HD + 1)) * sizeof(float);
    auto kern = k_attn<T, HD>;
    PE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
    PE_CUDA_TRY(launch_ex(kern, dim3(p.B * p.nkv, p.max_splits), dim3(kThreads), smem, s, pdl, p));
    return PE_OK;
}

}  // namespace

AttnPlan plan_attention(int B, int K, int nq, int nkv, int hd, int max_pages, int page_size, int num_sms) {
    AttnPlan a{};
    const int max_entries = max_pages * page_size;
    const int pairs = B * nkv;
    const int want = ceil_div(2 * num_sms, pairs);
    int chunk = ceil_div(ceil_div(max_entries, want), 64) * 64;
    if (chunk < 64) chunk = 64;
    a.chunk = chunk;
    a.max_splits = ceil_div(max_entries, chunk);
    const int Rq = K * (nq / nkv);
    a.ws_floats = a.max_splits > 1 ? static_cast<size_t>(pairs) * a.max_splits * Rq * (hd + 2) : 0;
    a.tickets = pairs;
    return a;
}

int launch_attention(int dtype, const AttnParams& p, cudaStream_t s, bool pdl) {
    if (dtype == PE_DTYPE_BF16) {
        if (p.hd == 128) return launch_hd<__nv_bfloat16, 128>(p, s, pdl);
        if (p.hd == 64) return launch_hd<__nv_bfloat16, 64>(p, s, pdl);
    } else {
        if (p.hd == 128) return launch_hd<float, 128>(p, s, pdl);
        if (p.hd == 64) return launch_hd<float, 64>(p, s, pdl);
    }
    set_error("attention: head_dim must be 64 or 128");
    return PE_ERR_UNSUPPORTED;
}

}  // namespace pe
