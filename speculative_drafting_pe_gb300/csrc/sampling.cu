// Sampled drafting and stochastic (speculative-sampling) acceptance.
//
// The P-EAGLE post ("在 Amazon SageMaker AI 上使用 P-EAGLE 并行化推测解码",
// "逐步草稿过程") has the target verify the K drafts with the standard
// acceptance rule, with no loss of output quality; its deployment samples at
// temperature 0.3. With sampling that rule is speculative sampling:
//   q_j = softmax(l_j / T) (drafter row j), p_j = softmax(g_j / T) (target);
//   draft d_j is accepted while u_j < p_j(d_j) / q_j(d_j); at the first
//   rejection a token is drawn from max(0, p_j - q_j) (normalised), and
//   after K acceptances a bonus token from p_K.
// Every draw is inverse-CDF sampling with a caller-supplied uniform u: the
// smallest index whose running weight exceeds u * total, the running sum
// taken in index order.
//
// Layout of one row's ordered reduction (k_sample_rows, k_accept_and_draw):
// warp w owns the contiguous segment [w * seg, (w + 1) * seg) of the row and
// walks it 32 elements at a time (coalesced loads, an in-order warp scan per
// group); the warps' segment totals are scanned in warp order, and the one
// warp whose segment holds u * total walks it again to find the index.
#include <cfloat>

#include "common.cuh"
#include "internal.h"

namespace pe {
namespace {

constexpr int kSampThreads = 512;
constexpr int kSampWarps = kSampThreads / 32;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Block maximum of a row (every thread returns it).
__device__ float block_row_max(const float* row, int V, float* red) {
    float m = -FLT_MAX;
    for (int i = threadIdx.x; i < V; i += blockDim.x) m = fmaxf(m, row[i]);
    m = warp_max(m);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[w] = m;
    __syncthreads();
    float r = red[0];
    for (int i = 1; i < kSampWarps; ++i) r = fmaxf(r, red[i]);
    return r;
}

// Inclusive in-order scan over the warp's 32 lanes.
__device__ __forceinline__ float warp_incl_scan(float v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Ordered inverse-CDF draw over weights weight(i), i < V, where `weight` is
// a device functor. Returns the drawn index (all threads).
template <typename Wt>
__device__ int ordered_draw(const Wt& weight, int V, float u, float* s_tot, int* s_pick) {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = (V + kSampWarps - 1) / kSampWarps;
    const int lo = w * seg, hi = min(V, lo + seg);
    // segment totals, each summed group by group in index order
    float run = 0.f;
    for (int g = lo; g < hi; g += 32) {
        const int i = g + lane;
        const float x = i < hi ? weight(i) : 0.f;
        run += __shfl_sync(0xffffffffu, warp_incl_scan(x), 31);
    }
    __syncthreads();
    if (lane == 0) s_tot[w] = run;
    if (threadIdx.x == 0) *s_pick = -1;
    __syncthreads();
    float before = 0.f, total = 0.f;
    for (int i = 0; i < kSampWarps; ++i) {
        if (i < w) before += s_tot[i];
        total += s_tot[i];
    }
    const float target = u * total;
    // the warp whose segment holds the target walks it again
    if (target >= before && target < before + s_tot[w] && s_tot[w] > 0.f) {
        float acc = before;
        int last_pos = -1;     // the segment's last index of positive weight seen so far
        bool found = false;
        for (int g = lo; g < hi; g += 32) {
            const int i = g + lane;
            const float x = i < hi ? weight(i) : 0.f;
            const float incl = acc + warp_incl_scan(x);
            const unsigned hit = __ballot_sync(0xffffffffu, i < hi && x > 0.f && incl > target);
            if (hit) {
                if (lane == 0) *s_pick = g + __ffs(hit) - 1;
                found = true;
                break;
            }
            const unsigned pos = __ballot_sync(0xffffffffu, i < hi && x > 0.f);
            if (pos) last_pos = g + 31 - __clz(pos);
            acc = __shfl_sync(0xffffffffu, incl, 31);
        }
        // the walk's running sum rounded a little below the first pass's
        // total: the target lies at the segment's end
        if (!found && lane == 0) *s_pick = last_pos;
    }
    __syncthreads();
    int pick = *s_pick;
    if (pick < 0) {
        // target at the very end (u * total rounded up to total): the last
        // index of positive weight
        __shared__ int s_last;
        if (threadIdx.x == 0) s_last = -1;
        __syncthreads();
        for (int i = threadIdx.x; i < V; i += blockDim.x)
            if (weight(i) > 0.f) atomicMax(&s_last, i);
        __syncthreads();
        pick = s_last < 0 ? 0 : s_last;
    }
    return pick;
}

// Drafts d[r] ~ softmax(logits[r] / T) for every row r = b * K + j.
__global__ void __launch_bounds__(kSampThreads) k_sample_rows(const float* __restrict__ logits, int V, float inv_t,
                                                                const float* __restrict__ u,
                                                                const int32_t* __restrict__ status, int K,
                                                                int32_t* __restrict__ drafts) {
    __shared__ float red[kSampWarps];
    __shared__ float s_tot[kSampWarps];
    __shared__ int s_pick;
    pdl_launch_dependents();
    pdl_wait();
    const int r = blockIdx.x;
    const int b = r / K;
    if (status != nullptr && status[b] != PE_REQ_OK) {
        if (threadIdx.x == 0) drafts[r] = -1;
        return;
    }
    const float* row = logits + static_cast<size_t>(r) * V;
    const float m = block_row_max(row, V, red);
    auto weight = [&](int i) { return expf((row[i] - m) * inv_t); };
    const int pick = ordered_draw(weight, V, u[r], s_tot, &s_pick);
    if (threadIdx.x == 0) drafts[r] = pick;
}

// Row statistics: max and sum of exp((x - max) / T) of every row.
__global__ void __launch_bounds__(kSampThreads) k_row_softmax_stats(const float* __restrict__ logits, int V,
                                                                      float inv_t, float2* __restrict__ stats) {
    __shared__ float red[kSampWarps];
    pdl_launch_dependents();
    pdl_wait();
    const float* row = logits + static_cast<size_t>(blockIdx.x) * V;
    const float m = block_row_max(row, V, red);
    float z = 0.f;
    for (int i = threadIdx.x; i < V; i += blockDim.x) z += expf((row[i] - m) * inv_t);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[w] = z;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < kSampWarps; ++i) t += red[i];
        stats[blockIdx.x] = make_float2(m, t);
    }
}

// One request per CTA: the acceptance tests in position order, then the
// final draw (residual max(0, p_a - q_a) or p_K).
__global__ void __launch_bounds__(kSampThreads)
    k_accept_and_draw(int K, int V, float inv_t, const int32_t* __restrict__ drafts,
                      const float* __restrict__ dlogits, const float* __restrict__ tlogits,
                      const float2* __restrict__ dstats, const float2* __restrict__ tstats,
                      const float* __restrict__ u_accept, const float* __restrict__ u_final,
                      int32_t* __restrict__ accepted, int32_t* __restrict__ final_tok) {
    __shared__ float s_tot[kSampWarps];
    __shared__ int s_pick;
    __shared__ int s_a;
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.x;
    if (threadIdx.x == 0) {
        int a = 0;
        while (a < K) {
            const int r = b * K + a;
            const int d = drafts[r];
            if (d < 0 || d >= V) break;
            const float2 ds = dstats[r];
            const float2 ts = tstats[b * (K + 1) + a];
            const float q = expf((dlogits[static_cast<size_t>(r) * V + d] - ds.x) * inv_t) / ds.y;
            const float p = expf((tlogits[static_cast<size_t>(b * (K + 1) + a) * V + d] - ts.x) * inv_t) / ts.y;
            if (u_accept[r] < p / q) ++a;
            else break;
        }
        s_a = a;
    }
    __syncthreads();
    const int a = s_a;
    const float* trow = tlogits + static_cast<size_t>(b * (K + 1) + a) * V;
    const float2 ts = tstats[b * (K + 1) + a];
    int pick;
    if (a < K) {
        const float* drow = dlogits + static_cast<size_t>(b * K + a) * V;
        const float2 ds = dstats[b * K + a];
        auto weight = [&](int i) {
            const float p = expf((trow[i] - ts.x) * inv_t) / ts.y;
            const float q = expf((drow[i] - ds.x) * inv_t) / ds.y;
            return fmaxf(p - q, 0.f);
        };
        pick = ordered_draw(weight, V, u_final[b], s_tot, &s_pick);
    } else {
        auto weight = [&](int i) { return expf((trow[i] - ts.x) * inv_t); };
        pick = ordered_draw(weight, V, u_final[b], s_tot, &s_pick);
    }
    if (threadIdx.x == 0) {
        accepted[b] = a;
        final_tok[b] = pick;
    }
}

}  // namespace

int launch_sample_rows(const float* logits, int rows, int V, float temperature, const float* u,
                       const int32_t* status, int K, int32_t* drafts, cudaStream_t s) {
    PE_CUDA_TRY(launch_ex(k_sample_rows, dim3(rows), dim3(kSampThreads), 0, s, false, logits, V,
                          1.0f / temperature, u, status, K, drafts));
    return PE_OK;
}

int launch_stochastic_accept(int B, int K, int V, float temperature, const int32_t* drafts, const float* dlogits,
                             const float* tlogits, const float* u_accept, const float* u_final, float2* stats,
                             int32_t* accepted, int32_t* final_tok, cudaStream_t s) {
    const float inv_t = 1.0f / temperature;
    float2* dstats = stats;
    float2* tstats = stats + static_cast<size_t>(B) * K;
    PE_CUDA_TRY(launch_ex(k_row_softmax_stats, dim3(B * K), dim3(kSampThreads), 0, s, false, dlogits, V, inv_t,
                          dstats));
    PE_CUDA_TRY(launch_ex(k_row_softmax_stats, dim3(B * (K + 1)), dim3(kSampThreads), 0, s, false, tlogits, V,
                          inv_t, tstats));
    PE_CUDA_TRY(launch_ex(k_accept_and_draw, dim3(B), dim3(kSampThreads), 0, s, false, K, V, inv_t, drafts, dlogits,
                          tlogits, static_cast<const float2*>(dstats), static_cast<const float2*>(tstats), u_accept,
                          u_final, accepted, final_tok));
    return PE_OK;
}

}  // namespace pe
