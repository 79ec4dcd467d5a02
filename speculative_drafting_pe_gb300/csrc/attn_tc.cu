// Tensor-core decode-style paged GQA attention (bf16 KV cache).
//
// Row j of request b (all nq/nkv query heads of one kv head packed as
// rows j*G + g) attends to cache entries 0 .. S_b + j; scores are scaled by
// 1/sqrt(hd); softmax is online in fp32 (base-2 exponent).
//
// One CTA per (request, kv head, entry split). KV pages are TMA-staged into
// shared memory: a tile is 64 cache entries = 4 pages; each page of one kv
// head is loaded as 128-byte-swizzled boxes [16 entries x 64 dims] (two per
// page at hd = 128). QK^T and PV run on mma.sync m16n8k16 (bf16 in, fp32
// accumulate), one 16-row query tile per warp, K fragments read with
// ldmatrix and V fragments with ldmatrix.trans from the swizzled tiles.
// The entry splits of one (request, kv head) form one thread-block cluster:
// each CTA leaves its fp32 partial (unnormalised output, running max, sum) in
// its own shared memory, and after a cluster barrier every CTA combines a
// slice of the rows by reading its peers' partials through distributed shared
// memory, in split order. No global scratch is used.
#include <cfloat>

#include "common.cuh"
#include "internal.h"

namespace pe {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;          // cache entries per tile (4 pages)
constexpr int kStages = 3;
constexpr int kBoxBytes = 16 * 128;
constexpr int kMaxRq = 128;        // K * nq/nkv query rows per kv head
constexpr int kMaxCluster = 16;    // non-portable cluster size limit

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of (entry e, 8-element chunk c) inside a [64 x HD] tile made of
// HD/64 sub-tiles [64 entries x 128 B] with the 128-byte swizzle.
template <int HD>
__device__ __forceinline__ uint32_t tile_off(int e, int c) {
    const int sub = c >> 3;
    const int cw = c & 7;
    return static_cast<uint32_t>(sub * (kTile * 128) + e * 128 + ((cw ^ (e & 7)) << 4));
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    constexpr int kTileBytes = kTile * HD * 2;     // one of K or V
    constexpr int kSub = HD / 64;                  // 128-byte sub-tiles per entry row
    constexpr int kNT = HD / 8;                    // n-tiles of the output
    constexpr int kKS = HD / 16;                   // k-steps of QK^T
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = smem;
    uint8_t* sV = smem + kStages * kTileBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(sV + kStages * kTileBytes);
    int* s_pages = reinterpret_cast<int*>(full + kStages);   // page coordinates of this CTA's entry range
    __shared__ float s_m[kMaxRq], s_l[kMaxRq];   // per-row running max (log2) and sum of this split

    const int pair = blockIdx.x;
    const int b = pair / p.nkv;
    const int kvh = pair - b * p.nkv;
    const int split = blockIdx.y;
    const int G = p.nq / p.nkv;
    const int K = p.K;
    const int Rq = K * G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    const size_t row_stride = static_cast<size_t>(p.nq) * HD;

    pdl_launch_dependents();
    pdl_wait();

    // Every CTA of a cluster runs to the end (cluster barriers); CTAs without
    // work simply contribute an empty partial.
    const int C = gridDim.y;                 // cluster size = entry splits per (request, kv head)
    const bool req_ok = p.status[b] == PE_REQ_OK;
    const int S = req_ok ? p.seq_lens[b] : 0;
    const int total = S + K;
    const int e0 = split * p.chunk;
    const int e1 = req_ok ? min(total, e0 + p.chunk) : e0;
    const int n_tiles = e1 > e0 ? (e1 - e0 + kTile - 1) / kTile : 0;
    const int32_t* pt = p.page_table + static_cast<size_t>(b) * p.max_pages;
    const int last_page = (total - 1) >> 4;       // last page index holding a valid entry

    if (tid == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    // page coordinates of every tile of this CTA, read once; pages past the
    // request's last entry get a negative (out-of-range, zero-filled) coordinate
    const int n_pg = n_tiles * (kTile / 16);
    const int pg0 = e0 >> 4;
    for (int i = tid; i < n_pg; i += kThreads) {
        const int pi = pg0 + i;
        s_pages[i] = pi <= last_page ? pt[pi] + p.layer_page0 : -1;
    }
    __syncthreads();

    const uint64_t pol = l2_policy_evict_first();
    auto issue = [&](int t) {   // thread 0 only
        const int st = t % kStages;
        mbar_arrive_expect_tx(&full[st], 2u * kTileBytes);
        for (int pg = 0; pg < kTile / 16; ++pg) {
            const int pc = s_pages[t * (kTile / 16) + pg];
            for (int sb = 0; sb < kSub; ++sb) {
                const uint32_t off = static_cast<uint32_t>(sb * (kTile * 128) + pg * kBoxBytes);
                tma_load_4d(sK + st * kTileBytes + off, &tmK, &full[st], sb * 64, 0, kvh, pc, pol);
                tma_load_4d(sV + st * kTileBytes + off, &tmV, &full[st], sb * 64, 0, kvh, pc, pol);
            }
        }
    };
    if (tid == 0)
        for (int t = 0; t < min(kStages, n_tiles); ++t) issue(t);

    // this warp's 16 query rows (packed j*G + g); rows >= Rq are padding
    const int n_mt = (Rq + 15) >> 4;
    const bool active = warp < n_mt;
    const int r_lo = warp * 16 + gid;
    const int r_hi = r_lo + 8;
    const int j_lo = r_lo / G, j_hi = r_hi / G;
    uint32_t qa[kKS][4];
    if (active && n_tiles > 0) {
#pragma unroll
        for (int kk = 0; kk < kKS; ++kk) {
#pragma unroll
            for (int hv = 0; hv < 2; ++hv) {           // hv = 0: k lo half, 1: k hi half
                const int d = kk * 16 + hv * 8 + tig * 2;
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {       // rr = 0: row g, 1: row g + 8
                    const int r = rr ? r_hi : r_lo;
                    uint32_t v = 0u;
                    if (r < Rq) {
                        const int j = r / G, g = r - (r / G) * G;
                        v = *reinterpret_cast<const uint32_t*>(
                            q + static_cast<size_t>(b * K + j) * row_stride + static_cast<size_t>(kvh * G + g) * HD + d);
                    }
                    qa[kk][hv * 2 + rr] = v;
                }
            }
        }
    }

    float o[kNT][4];
#pragma unroll
    for (int i = 0; i < kNT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
    const float sl2 = rsqrtf(static_cast<float>(HD)) * 1.4426950408889634f;
    const int lim_lo = S + j_lo, lim_hi = S + j_hi;   // last visible entry per row

    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
        const int st = t % kStages;
        if (!mbar_wait(&full[st], static_cast<uint32_t>((t / kStages) & 1), p.err, PE_DEVERR_ATTN_TIMEOUT)) ok = false;
        const int tbase = e0 + t * kTile;
        if (active && ok) {
            const uint32_t kb = smem_u32(sK + st * kTileBytes);
            const uint32_t vb = smem_u32(sV + st * kTileBytes);
            float s[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
            const int mi = lane >> 3, rr8 = lane & 7;
#pragma unroll
            for (int kk = 0; kk < kKS; ++kk) {
#pragma unroll
                for (int nt = 0; nt < 8; nt += 2) {
                    const int e = nt * 8 + (mi >> 1) * 8 + rr8;
                    const int c = kk * 2 + (mi & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kb + tile_off<HD>(e, c), b0, b1, b2, b3);
                    mma_bf16(s[nt], qa[kk], b0, b1);
                    mma_bf16(s[nt + 1], qa[kk], b2, b3);
                }
            }
            // mask + online softmax (log2 domain)
            float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int e = tbase + nt * 8 + tig * 2 + c;
                    const bool in = e < e1;
                    s[nt][c] = (in && e <= lim_lo) ? s[nt][c] * sl2 : -INFINITY;
                    s[nt][2 + c] = (in && e <= lim_hi) ? s[nt][2 + c] * sl2 : -INFINITY;
                    mx_lo = fmaxf(mx_lo, s[nt][c]);
                    mx_hi = fmaxf(mx_hi, s[nt][2 + c]);
                }
            }
            mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
            mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
            mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
            mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
            const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
            const float base_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
            const float base_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
            const float corr_lo = exp2f(m_lo - base_lo), corr_hi = exp2f(m_hi - base_hi);
            m_lo = mn_lo;
            m_hi = mn_hi;
            float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                s[nt][0] = exp2f(s[nt][0] - base_lo);
                s[nt][1] = exp2f(s[nt][1] - base_lo);
                s[nt][2] = exp2f(s[nt][2] - base_hi);
                s[nt][3] = exp2f(s[nt][3] - base_hi);
                sum_lo += s[nt][0] + s[nt][1];
                sum_hi += s[nt][2] + s[nt][3];
            }
            l_lo = l_lo * corr_lo + sum_lo;
            l_hi = l_hi * corr_hi + sum_hi;
#pragma unroll
            for (int i = 0; i < kNT; ++i) {
                o[i][0] *= corr_lo;
                o[i][1] *= corr_lo;
                o[i][2] *= corr_hi;
                o[i][3] *= corr_hi;
            }
            // O += P V
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t pa[4];
                pa[0] = pack_bf16(s[2 * ks][0], s[2 * ks][1]);
                pa[1] = pack_bf16(s[2 * ks][2], s[2 * ks][3]);
                pa[2] = pack_bf16(s[2 * ks + 1][0], s[2 * ks + 1][1]);
                pa[3] = pack_bf16(s[2 * ks + 1][2], s[2 * ks + 1][3]);
#pragma unroll
                for (int np = 0; np < kNT; np += 2) {
                    const int e = ks * 16 + (mi & 1) * 8 + rr8;
                    const int c = np + (mi >> 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vb + tile_off<HD>(e, c), b0, b1, b2, b3);
                    mma_bf16(o[np], pa, b0, b1);
                    mma_bf16(o[np + 1], pa, b2, b3);
                }
            }
        }
        // all threads agree on whether every wait succeeded before reusing a stage
        if (!__syncthreads_and(ok ? 1 : 0)) {
            ok = false;
            break;
        }
        if (tid == 0 && t + kStages < n_tiles) issue(t + kStages);
    }
    if (!ok) __nanosleep(100000);    // a wait gave up: let copies still in flight land

    // full row sums across the quad
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    if (!ok) l_lo = l_hi = 0.f;

    if (C == 1) {
        if (active) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = rr ? r_hi : r_lo;
                if (r < Rq) {
                    const float l = rr ? l_hi : l_lo;
                    const float inv = (req_ok && l > 0.f) ? 1.f / l : 0.f;
                    const int j = r / G, g = r - (r / G) * G;
                    __nv_bfloat16* dst = out + static_cast<size_t>(b * K + j) * row_stride + static_cast<size_t>(kvh * G + g) * HD;
#pragma unroll
                    for (int nt = 0; nt < kNT; ++nt) {
                        const int d = nt * 8 + tig * 2;
                        *reinterpret_cast<__nv_bfloat162*>(dst + d) =
                            __floats2bfloat162_rn(o[nt][rr * 2] * inv, o[nt][rr * 2 + 1] * inv);
                    }
                }
            }
        }
        return;
    }

    // Split partial into this CTA's shared memory. The KV stage buffers are
    // free again (every tile was consumed before the last block barrier).
    float* s_o = reinterpret_cast<float*>(smem);      // [Rq][HD]
    if (active) {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int r = rr ? r_hi : r_lo;
            if (r < Rq) {
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt) {
                    const int d = nt * 8 + tig * 2;
                    *reinterpret_cast<float2*>(s_o + r * HD + d) = make_float2(o[nt][rr * 2], o[nt][rr * 2 + 1]);
                }
                if (tig == 0) {
                    s_m[r] = rr ? m_hi : m_lo;
                    s_l[r] = rr ? l_hi : l_lo;
                }
            }
        }
    }
    cluster_sync_all();

    // CTA `rank` combines rows rank, rank + C, ... from all C partials, in split order.
    const uint32_t rank = cluster_ctarank();
    const uint32_t o_base = smem_u32(s_o), m_base = smem_u32(s_m), l_base = smem_u32(s_l);
    const int my_rows = (Rq - static_cast<int>(rank) + C - 1) / C;
    for (int item = tid; item < my_rows * (HD / 2); item += kThreads) {
        const int r = static_cast<int>(rank) + (item / (HD / 2)) * C;
        const int d = (item - (item / (HD / 2)) * (HD / 2)) * 2;
        float M = -INFINITY;
        for (int sp = 0; sp < C; ++sp) M = fmaxf(M, dsmem_ld(dsmem_addr(m_base + 4u * r, sp)));
        float den = 0.f, n0 = 0.f, n1 = 0.f;
        for (int sp = 0; sp < C; ++sp) {
            const float ls = dsmem_ld(dsmem_addr(l_base + 4u * r, sp));
            if (ls <= 0.f) continue;
            const float w = exp2f(dsmem_ld(dsmem_addr(m_base + 4u * r, sp)) - M);
            const float2 ov = dsmem_ld2(dsmem_addr(o_base + 4u * (r * HD + d), sp));
            den = fmaf(ls, w, den);
            n0 = fmaf(w, ov.x, n0);
            n1 = fmaf(w, ov.y, n1);
        }
        const float inv = (req_ok && den > 0.f) ? 1.f / den : 0.f;
        const int j = r / G, g = r - (r / G) * G;
        __nv_bfloat16* dst = out + static_cast<size_t>(b * K + j) * row_stride + static_cast<size_t>(kvh * G + g) * HD + d;
        *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(n0 * inv, n1 * inv);
    }
    // peers may still be reading this CTA's partial
    cluster_sync_all();
}

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

size_t attn_smem_bytes(int hd, int chunk) {
    return 2 * kStages * static_cast<size_t>(kTile) * hd * 2 + kStages * 8 +
           (static_cast<size_t>(chunk) / 16 + 4) * sizeof(int) + 1024;
}

template <int HD>
int launch_hd(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, cudaStream_t s, bool pdl) {
    const size_t smem = attn_smem_bytes(HD, p.chunk);
    auto kern = k_attn_tc<HD>;
    static size_t smem_set[64] = {};
    int dev = 0;
    PE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64 || smem > smem_set[dev]) {
        PE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
        PE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
        if (dev >= 0 && dev < 64) smem_set[dev] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.B * p.nkv, p.max_splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = static_cast<unsigned>(p.max_splits);
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    PE_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, tk, tv, p));
    return PE_OK;
}

}  // namespace

// Largest cluster size (<= 16) for which every (request, kv head) cluster is
// resident in one wave, from the occupancy calculator (cached per size).
static int max_active_clusters(int hd, int C, size_t smem) {
    static int cache[2][17] = {};
    int& c = cache[hd == 128 ? 1 : 0][C];
    if (c != 0) return c;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, C);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = static_cast<unsigned>(C);
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e;
    if (hd == 128) {
        cudaFuncSetAttribute(k_attn_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        cudaFuncSetAttribute(k_attn_tc<128>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        e = cudaOccupancyMaxActiveClusters(&n, k_attn_tc<128>, &cfg);
    } else {
        cudaFuncSetAttribute(k_attn_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        cudaFuncSetAttribute(k_attn_tc<64>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        e = cudaOccupancyMaxActiveClusters(&n, k_attn_tc<64>, &cfg);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        n = -1;   // size not launchable
    }
    c = n == 0 ? -1 : n;
    return c;
}

AttnPlan plan_attention_tc(int B, int K, int nq, int nkv, int hd, int max_pages, int page_size, int num_sms) {
    AttnPlan a{};
    const int max_entries = max_pages * page_size;
    const int pairs = B * nkv;
    int want = ceil_div(num_sms, pairs);                 // about one wave of CTAs
    if (want > kMaxCluster) want = kMaxCluster;
    if (want < 1) want = 1;
    int C = 1, chunk = ceil_div(max_entries, kTile) * kTile;
    for (int c = want; c >= 2; --c) {
        const int ch = ceil_div(ceil_div(max_entries, c), kTile) * kTile;
        const int n = max_active_clusters(hd, c, attn_smem_bytes(hd, ch));
        if (n > 0 && n >= pairs) {                       // every cluster resident at once
            C = c;
            chunk = ch;
            break;
        }
    }
    C = ceil_div(max_entries, chunk);                    // splits actually needed
    a.chunk = chunk;
    a.max_splits = C;                                    // one cluster of C CTAs per (request, kv head)
    a.ws_floats = 0;
    a.tickets = 0;
    (void)K; (void)nq;
    return a;
}

int launch_attention_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, cudaStream_t s,
                        bool pdl) {
    if (p.hd == 128) return launch_hd<128>(tk, tv, p, s, pdl);
    if (p.hd == 64) return launch_hd<64>(tk, tv, p, s, pdl);
    set_error("attention: head_dim must be 64 or 128");
    return PE_ERR_UNSUPPORTED;
}

}  // namespace pe
