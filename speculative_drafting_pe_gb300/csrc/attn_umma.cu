// Tensor-core (tcgen05 / TMEM) decode-style paged GQA attention, bf16 KV cache.
//
// Row j of request b (all nq/nkv query heads of one kv head packed as
// rows j*G + g, zero-padded to the MMA's 128 rows) attends to cache entries
// 0 .. S_b + j; scores are scaled by 1/sqrt(hd); softmax is online in fp32
// (base-2 exponent).
//
// Work layouts (chosen by plan_attention_umma from the (request, kv head)
// pair count): clusters - one CTA per (request, kv head, entry split),
// requests issued longest first (an order the row build computes), the
// splits of a pair combined through distributed shared memory; or
// length-aware pieces - one CTA per item of the row build's piece list, no
// cluster, a request with several pieces combined by k_attn_merge. A tile
// is 64 cache entries (4 pages). Roles (192 threads):
//   warp 4   TMA: the packed query rows once (3-D map over q), then K and V
//            pages of every tile (4-D map over the paged cache) into a
//            4-stage ring, 128-byte swizzle. A stage is refilled once the
//            P.V of its tile has completed.
//   warp 5   TMEM allocation; lane 0 issues  S_t = Q K_t^T  (M=128, N=64,
//            K=hd, both operands K-major) into one of two TMEM score
//            buffers, and  O += P_t V_t  (M=128, N=hd, K=64) into the TMEM
//            output accumulator, with P_t read from TMEM as the A operand.
//            V_t is read where TMA put it, as an MN-major operand (entries
//            are the reduction dimension, the 64-dim rows the N dimension),
//            so it is never transposed.
//   warps 0-3  one thread per query row (= TMEM lane): read the row of S_t
//            from TMEM, mask, keep the running max, write P_t = exp2(S - m)
//            as bf16 pairs over the columns of S_t it has just read (the
//            next S MMA into that buffer is issued after this tile's P.V,
//            and a CTA's MMAs run in issue order), and rescale the TMEM
//            output row only when the running max grows by more than 2^8.
// In the cluster layout the entry splits of one (request, kv head) form one
// thread-block cluster and are combined through distributed shared memory in
// split order; a piece of a request with several writes its partial (O,
// running max, sum) to scratch for k_attn_merge.
#include <cfloat>

#include "common.cuh"
#include "internal.h"

namespace pe {
namespace {

constexpr int kThreads = 192;      // warps 0-3 softmax, 4 TMA, 5 MMA
constexpr int kTile = 64;           // cache entries per tile
constexpr int kStages = 4;
constexpr int kRows = 128;          // MMA M (query rows, zero padded)
constexpr int kBoxBytes = 16 * 128; // one page of one kv head, 64 dims
constexpr float kRescaleLog2 = 8.f;
constexpr int kMaxCluster = 16;
constexpr int kPiecePairs = 16;      // (request, kv head) pairs from which length-aware pieces are used
constexpr int kPieceMaxBatch = 256;  // requests the row build's piece list serves (= kMaxPieceB of
                                     // rows.cu, the size of its shared arrays)
constexpr int kPieceMinTiles = 4;


template <int HD>
struct Layout {
    static constexpr int kSub = HD / 64;                    // 128-byte sub-tiles per row
    static constexpr int kQBytes = kSub * kRows * 128;      // Q: kSub x [128 rows x 128 B]
    static constexpr int kKVBytes = kSub * kTile * 128;     // K or V tile: kSub x [64 entries x 128 B]
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kQBytes;
    static constexpr int kV = kK + kStages * kKVBytes;
    static constexpr int kBar = kV + kStages * kKVBytes;
    static constexpr int kNumBars = 1 + 2 * kStages + 6;   // q_full, kv_full[], kv_empty[], s_full[2], p_full[2], o_done[2]
    static constexpr int kTmem = kBar + kNumBars * 8;
    static constexpr int kPages = kTmem + 16;
};

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
// 2^x with the hardware approximation (ex2.approx.ftz.f32): 2^-inf = 0.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_umma(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using L = Layout<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
    uint64_t* q_full = bars;
    uint64_t* kv_full = bars + 1;
    uint64_t* kv_empty = kv_full + kStages;
    uint64_t* s_full = kv_empty + kStages;
    uint64_t* p_full = s_full + 2;
    uint64_t* o_done = p_full + 2;         // [2]: P.V of tiles with this parity complete
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kTmem);
    int* s_pages = reinterpret_cast<int*>(sm + L::kPages);
    // Cluster combine: the running max (log2) and sum of row r from split sp,
    // held by the CTA that combines row r (rank r mod C) at (r / C) * C + sp
    __shared__ float2 s_ml[kRows + kMaxCluster];

    const int C = gridDim.y;                   // cluster size = entry splits per (request, kv head)
    const int G = p.nq / p.nkv;
    const int K = p.K;
    const int Rq = K * G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    const size_t row_stride = static_cast<size_t>(p.nq) * HD;

    pdl_launch_dependents();
    // Before the dependency wait: set-up that reads nothing an earlier kernel
    // writes (barriers, the query tile's zero padding), and an L2
    // prefetch of this CTA's first K/V pages. The prefetch reads the order
    // list, lengths and page table as they are now - possibly still being
    // written by earlier kernels of the stream - which is harmless: a wrong
    // guess only warms the wrong lines; everything used below is read again
    // after the wait.
    if (tid == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        mbar_init(q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&kv_full[s], 1);
            // free once the P.V of the stage's tile has completed (one MMA
            // commit; it is issued after the S that read K)
            mbar_init(&kv_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&p_full[s], 128);
        }
        mbar_init(&o_done[0], 1);
        mbar_init(&o_done[1], 1);
        fence_mbar_init();
    }
    {
        // zero the padding query rows Rq..127 (the TMA box fills rows < Rq)
        const int Rq0 = p.K * (p.nq / p.nkv);
        for (int idx = tid; idx < (kRows - Rq0) * 8 * L::kSub; idx += kThreads) {
            const int sub = idx / ((kRows - Rq0) * 8);
            const int rem = idx - sub * (kRows - Rq0) * 8;
            const int r = Rq0 + rem / 8, c = rem % 8;
            sts128(smem_u32(sm + L::kQ + sub * kRows * 128 + r * 128 + c * 16), 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
    }
    if (tid == 4 * 32 && p.items == nullptr && p.l2_prefetch) {
        const int pair = blockIdx.x;
        const int kv_g = pair % p.nkv;
        int b_g = p.order != nullptr ? p.order[pair / p.nkv] : pair / p.nkv;
        b_g = b_g < 0 || b_g >= p.B ? 0 : b_g;
        const int S_g = max(0, p.seq_lens[b_g]);
        const int ea = static_cast<int>(blockIdx.y) * p.chunk;
        const int eb = min(S_g + p.K, ea + p.chunk);
        const int n_pf = min(kStages * (kTile / 16), eb > ea ? (eb - ea + 15) / 16 : 0);
        const int32_t* pt_g = p.page_table + static_cast<size_t>(b_g) * p.max_pages;
        for (int i = 0; i < n_pf; ++i) {
            const int pi = (ea >> 4) + i;
            const int pg = pi < p.max_pages ? pt_g[pi] : -1;
            if (pg < 0 || pg >= p.num_pages) continue;
            for (int sb = 0; sb < L::kSub; ++sb) {
                tma_prefetch_l2_4d(&tmK, sb * 64, 0, kv_g, pg + p.layer_page0);
                tma_prefetch_l2_4d(&tmV, sb * 64, 0, kv_g, pg + p.layer_page0);
            }
        }
    }
    pdl_wait();
    int b, kvh, e0, e_end;
    bool single;                               // this CTA alone covers its (request, kv head)
    if (p.items != nullptr) {
        // length-aware piece; CTAs past the item count have none
        if (static_cast<int>(blockIdx.x) >= p.plan[0]) return;
        const int4 it = p.items[blockIdx.x];
        b = it.x;
        kvh = it.y;
        e0 = it.z;
        e_end = it.w;
        single = p.plan[1 + b] <= 1;
    } else {
        // the request of this CTA: longest first when an order is given
        const int pair = blockIdx.x;
        kvh = pair % p.nkv;
        b = p.order != nullptr ? p.order[pair / p.nkv] : pair / p.nkv;
        e0 = static_cast<int>(blockIdx.y) * p.chunk;
        e_end = e0 + p.chunk;
        single = C == 1;
    }

    // Every CTA of a cluster runs to the end (cluster barriers); CTAs without
    // work contribute an empty partial.
    const bool req_ok = p.status[b] == PE_REQ_OK;
    const int S = req_ok ? p.seq_lens[b] : 0;
    const int total = S + K;
    const int e1 = req_ok ? min(total, e_end) : e0;
    const int n_tiles = e1 > e0 ? (e1 - e0 + kTile - 1) / kTile : 0;
    const int32_t* pt = p.page_table + static_cast<size_t>(b) * p.max_pages;
    const int last_page = (total - 1) >> 4;

    // page coordinates of this CTA's tiles; pages past the request's last
    // entry get a negative (out-of-range, zero-filled) coordinate
    for (int i = tid; i < n_tiles * (kTile / 16); i += kThreads) {
        const int pi = (e0 >> 4) + i;
        s_pages[i] = pi <= last_page ? pt[pi] + p.layer_page0 : -1;
    }
    // TMEM after the early return of CTAs without a piece (a CTA must free
    // what it allocates)
    if (warp == 5) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_o = tmem + 128;             // output accumulator: columns 128 .. 128+hd
    bool ok = true;

    if (warp == 4) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && n_tiles > 0) {
            const uint64_t pol_kv = l2_policy_evict_first();
            const uint64_t pol_q = l2_policy_evict_last();
            mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(L::kSub * 128 * Rq));
            for (int sb = 0; sb < L::kSub; ++sb)
                tma_load_3d(sm + L::kQ + sb * kRows * 128, &tmQ, q_full, sb * 64, kvh * G, b * K, pol_q);
            for (int t = 0; t < n_tiles; ++t) {
                const int st = t % kStages;
                if (t >= kStages &&
                    !mbar_wait(&kv_empty[st], static_cast<uint32_t>((t / kStages) & 1) ^ 1u, p.err,
                               PE_DEVERR_ATTN_TIMEOUT)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&kv_full[st], 2u * L::kKVBytes);
                for (int pg = 0; pg < kTile / 16; ++pg) {
                    const int pc = s_pages[t * (kTile / 16) + pg];
                    for (int sb = 0; sb < L::kSub; ++sb) {
                        const int off = st * L::kKVBytes + sb * kTile * 128 + pg * kBoxBytes;
                        tma_load_4d(sm + L::kK + off, &tmK, &kv_full[st], sb * 64, 0, kvh, pc, pol_kv);
                        tma_load_4d(sm + L::kV + off, &tmV, &kv_full[st], sb * 64, 0, kvh, pc, pol_kv);
                    }
                }
            }
        }
        __syncwarp();   // reconverge before the CTA-wide barriers below
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0 && n_tiles > 0) {
            const uint32_t idesc_s = umma_idesc(1, kRows, kTile);
            const uint32_t idesc_o = umma_idesc(1, kRows, HD) | kIdescBMnMajor;
            const uint32_t q_addr = smem_u32(sm + L::kQ);
            auto issue_s = [&](int t) {
                const uint32_t k_addr = smem_u32(sm + L::kK + (t % kStages) * L::kKVBytes);
                const uint32_t d = tmem + static_cast<uint32_t>((t & 1) * kTile);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t sub = static_cast<uint32_t>(kk >> 2), within = static_cast<uint32_t>((kk & 3) * 32);
                    UmmaKind<__nv_bfloat16>::mma(d, umma_desc_sw128(q_addr + sub * kRows * 128 + within),
                                                 umma_desc_sw128(k_addr + sub * kTile * 128 + within), idesc_s,
                                                 kk > 0 ? 1u : 0u);
                }
                umma_commit(&s_full[t & 1]);
            };
            if (!mbar_wait(q_full, 0, p.err, PE_DEVERR_ATTN_TIMEOUT) ||
                !mbar_wait(&kv_full[0], 0, p.err, PE_DEVERR_ATTN_TIMEOUT)) {
                ok = false;
            } else {
                tc_fence_after_sync();
                issue_s(0);
            }
            for (int t = 0; t < n_tiles && ok; ++t) {
                if (t + 1 < n_tiles) {
                    if (!mbar_wait(&kv_full[(t + 1) % kStages], static_cast<uint32_t>(((t + 1) / kStages) & 1), p.err,
                                   PE_DEVERR_ATTN_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    issue_s(t + 1);
                }
                if (!mbar_wait(&p_full[t & 1], static_cast<uint32_t>((t >> 1) & 1), p.err, PE_DEVERR_ATTN_TIMEOUT)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                // P_t in TMEM over the columns of S_t (bf16 pairs, 8 columns
                // per 16 entries)
                const uint32_t p_tmem = tmem + static_cast<uint32_t>((t & 1) * kTile);
                const uint32_t v_addr = smem_u32(sm + L::kV + (t % kStages) * L::kKVBytes);
                // V_t as the MN-major B operand: 16 entries (two 8-row swizzle
                // atoms, 1024 B apart) per MMA, 64-dim blocks kTile*128 B apart
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                    umma_bf16_a_tmem(t_o, p_tmem + static_cast<uint32_t>(kk * 8),
                                     umma_desc_sw128_mn(v_addr + kk * 16 * 128, kTile * 128), idesc_o,
                                     (t > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&o_done[t & 1]);
                umma_commit(&kv_empty[t % kStages]);   // K and V of this stage are read
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax warps: thread = query row = TMEM lane
        const int row = tid;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const bool row_ok = row < Rq;
        const int lim = S + row / G;          // last visible entry of this row
        const float sl2 = rsqrtf(static_cast<float>(HD)) * 1.4426950408889634f;
        float m_used = -INFINITY, l = 0.f;    // m_used: running max of the scaled (log2) scores
        for (int t = 0; t < n_tiles; ++t) {
            // the P buffer (t & 1) was last read by the P.V of tile t-2
            if (t >= 2 && !mbar_wait(&o_done[t & 1], static_cast<uint32_t>(((t >> 1) - 1) & 1), p.err,
                                     PE_DEVERR_ATTN_TIMEOUT))
                ok = false;
            if (ok && !mbar_wait(&s_full[t & 1], static_cast<uint32_t>((t >> 1) & 1), p.err, PE_DEVERR_ATTN_TIMEOUT))
                ok = false;
            ok = __all_sync(0xffffffffu, ok);   // keep the warp converged for the .aligned instructions
            if (!ok) break;
            tc_fence_after_sync();
            float sv[kTile];
#pragma unroll
            for (int c = 0; c < kTile / 16; ++c) {
                float v16[16];
                tmem_ld16(tmem + lane_off + static_cast<uint32_t>((t & 1) * kTile + c * 16), v16);
#pragma unroll
                for (int i = 0; i < 16; ++i) sv[c * 16 + i] = v16[i];
            }
            const int tbase = e0 + t * kTile;
            // interior tile: every entry is visible to every row (CTA-uniform)
            const bool interior = tbase + kTile <= e1 && tbase + kTile <= S + 1;
            float tmax = -INFINITY;
            if (interior) {
#pragma unroll
                for (int i = 0; i < kTile; ++i) tmax = fmaxf(tmax, sv[i]);
            } else {
#pragma unroll
                for (int i = 0; i < kTile; ++i) {
                    const int e = tbase + i;
                    if (!(row_ok && e < e1 && e <= lim)) sv[i] = -INFINITY;
                    tmax = fmaxf(tmax, sv[i]);
                }
            }
            tmax *= sl2;
            const bool need = tmax > -INFINITY && (m_used == -INFINITY || tmax > m_used + kRescaleLog2);
            float f = 1.f;
            if (need) {
                f = m_used == -INFINITY ? 0.f : ex2_approx(m_used - tmax);
                l *= f;
                m_used = tmax;
            }
            if (t > 0 && __any_sync(0xffffffffu, need)) {
                // scale the rows of O in TMEM once the P.V of tile t-1 is
                // complete, the whole warp together (rows that need none use f = 1)
                bool w_ok = mbar_wait(&o_done[(t - 1) & 1], static_cast<uint32_t>(((t - 1) >> 1) & 1), p.err,
                                      PE_DEVERR_ATTN_TIMEOUT);
                w_ok = __all_sync(0xffffffffu, w_ok);
                if (!w_ok) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
#pragma unroll
                for (int c = 0; c < HD / 16; ++c) {
                    float o16[16];
                    tmem_ld16(t_o + lane_off + static_cast<uint32_t>(c * 16), o16);
#pragma unroll
                    for (int i = 0; i < 16; ++i) o16[i] *= f;
                    tmem_st16(t_o + lane_off + static_cast<uint32_t>(c * 16), o16);
                }
            }
            // P_t row (bf16 pairs) into TMEM over S_t, which this thread has
            // read: p = 2^(s * scale - m)
            const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
            float psum = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float p0 = ex2_approx(fmaf(sv[h * 32 + 2 * i], sl2, neg_m));
                    const float p1 = ex2_approx(fmaf(sv[h * 32 + 2 * i + 1], sl2, neg_m));
                    psum += p0;
                    psum += p1;
                    pk[i] = __uint_as_float(pack_bf16(p0, p1));
                }
                tmem_st16(tmem + lane_off + static_cast<uint32_t>((t & 1) * kTile + h * 16), pk);
            }
            l += psum;
            tc_fence_before_sync();
            mbar_arrive(&p_full[t & 1]);
        }
        if (ok && n_tiles > 0 &&
            !mbar_wait(&o_done[(n_tiles - 1) & 1], static_cast<uint32_t>(((n_tiles - 1) >> 1) & 1), p.err,
                       PE_DEVERR_ATTN_TIMEOUT))
            ok = false;
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after_sync();
        if (!ok) l = 0.f;
        const bool have_o = ok && n_tiles > 0;   // warp-uniform

        if (single) {
            const int j = row / G, g = row - (row / G) * G;
            __nv_bfloat16* dst = out + static_cast<size_t>(b * K + j) * row_stride + static_cast<size_t>(kvh * G + g) * HD;
            const float inv = (req_ok && have_o && l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
            for (int c = 0; c < HD / 64; ++c) {
                float o64[64];
#pragma unroll
                for (int i = 0; i < 64; ++i) o64[i] = 0.f;
                if (have_o) tmem_ld64(t_o + lane_off + static_cast<uint32_t>(c * 64), o64);
                if (row_ok) {
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        const float* o8 = o64 + h * 8;
                        uint4 w;
                        w.x = pack_bf16(o8[0] * inv, o8[1] * inv);
                        w.y = pack_bf16(o8[2] * inv, o8[3] * inv);
                        w.z = pack_bf16(o8[4] * inv, o8[5] * inv);
                        w.w = pack_bf16(o8[6] * inv, o8[7] * inv);
                        *reinterpret_cast<uint4*>(dst + c * 64 + h * 8) = w;
                    }
                }
            }
        } else if (p.items != nullptr) {
            // piece partial to global scratch: O [Rq][hd], then the running
            // max (log2) and sum of each row, for k_attn_merge
            float* w = p.ws + static_cast<size_t>(blockIdx.x) * attn_piece_floats(Rq, HD);
#pragma unroll
            for (int c = 0; c < HD / 64; ++c) {
                float o64[64];
#pragma unroll
                for (int i = 0; i < 64; ++i) o64[i] = 0.f;
                if (have_o) tmem_ld64(t_o + lane_off + static_cast<uint32_t>(c * 64), o64);
                if (row_ok) {
#pragma unroll
                    for (int i = 0; i < 64; i += 4)
                        *reinterpret_cast<float4*>(w + row * HD + c * 64 + i) =
                            make_float4(o64[i], o64[i + 1], o64[i + 2], o64[i + 3]);
                }
            }
            if (row_ok) {
                w[Rq * HD + row] = m_used;
                w[Rq * HD + ((Rq + 3) & ~3) + row] = l;
            }
        } else {
            // split partial into this CTA's shared memory (the K stage ring is
            // free): row r's 16-byte chunk q at chunk q ^ (r & 7), so that the
            // eight rows of a quarter warp store to distinct banks
            float* s_o = reinterpret_cast<float*>(sm + L::kK);   // [Rq][hd] fp32
#pragma unroll
            for (int c = 0; c < HD / 64; ++c) {
                float o64[64];
#pragma unroll
                for (int i = 0; i < 64; ++i) o64[i] = 0.f;
                if (have_o) tmem_ld64(t_o + lane_off + static_cast<uint32_t>(c * 64), o64);
                if (row_ok) {
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int qs = (c * 16 + q) ^ (row & 7);
                        *reinterpret_cast<float4*>(s_o + row * HD + qs * 4) =
                            make_float4(o64[4 * q], o64[4 * q + 1], o64[4 * q + 2], o64[4 * q + 3]);
                    }
                }
            }
            if (row_ok) {
                // this split's max and sum of the row, straight into the table
                // of the CTA that combines it (published by the cluster barrier)
                const uint32_t at = smem_u32(&s_ml[(row / C) * C + static_cast<int>(cluster_ctarank())]);
                dsmem_st2(dsmem_addr(at, static_cast<uint32_t>(row % C)), m_used, l);
            }
        }
    }

    if (!ok) __nanosleep(100000);    // a wait gave up: let copies still in flight land
    if (C > 1) {
        __syncthreads();
        cluster_sync_all();
        // CTA `rank` combines rows rank, rank + C, ... from all C partials, in split order
        const uint32_t rank = cluster_ctarank();
        const uint32_t o_base = smem_u32(sm + L::kK);
        const int my_rows = (Rq - static_cast<int>(rank) + C - 1) / C;
        // Per row, once: the weight 2^(m_sp - M) of every split with a
        // positive sum (M the largest running max), and 1 / sum_sp l_sp w_sp;
        // kept in this CTA's query tile, which no MMA or peer reads any more
        float* s_w = reinterpret_cast<float*>(sm + L::kQ);                  // [row][kMaxCluster]
        float* s_rinv = s_w + kRows * kMaxCluster;                           // [row]
        uint32_t* s_mask = reinterpret_cast<uint32_t*>(s_rinv + kRows);     // [row] splits with l > 0
        if (tid < my_rows) {
            float mv[kMaxCluster], lv[kMaxCluster];
#pragma unroll
            for (int sp = 0; sp < kMaxCluster; ++sp) {
                if (sp < C) {
                    const float2 ml = s_ml[tid * C + sp];
                    mv[sp] = ml.x;
                    lv[sp] = ml.y;
                }
            }
            float M = -INFINITY;
#pragma unroll
            for (int sp = 0; sp < kMaxCluster; ++sp)
                if (sp < C) M = fmaxf(M, mv[sp]);
            float den = 0.f;
            uint32_t mask = 0u;
#pragma unroll
            for (int sp = 0; sp < kMaxCluster; ++sp) {
                if (sp < C && lv[sp] > 0.f) {
                    const float w = exp2f(mv[sp] - M);
                    den = fmaf(lv[sp], w, den);
                    s_w[tid * kMaxCluster + sp] = w;
                    mask |= 1u << sp;
                }
            }
            s_rinv[tid] = (req_ok && den > 0.f) ? 1.f / den : 0.f;
            s_mask[tid] = mask;
        }
        __syncthreads();
        for (int item = tid; item < my_rows * (HD / 2); item += kThreads) {
            const int rl = item / (HD / 2);
            const int r = static_cast<int>(rank) + rl * C;
            const int d = (item - rl * (HD / 2)) * 2;
            const uint32_t mask = s_mask[rl];
            // the pair's float index in the partial (its 16-byte chunk swizzled by the row)
            const int oi = r * HD + ((((d >> 2) ^ (r & 7)) << 2) | (d & 3));
            // every weighted split's output pair in flight at once, then
            // combined in split order
            float2 ov[kMaxCluster];
#pragma unroll
            for (int sp = 0; sp < kMaxCluster; ++sp)
                if (sp < C && ((mask >> sp) & 1u))
                    ov[sp] = dsmem_ld2(dsmem_addr(o_base + 4u * oi, static_cast<uint32_t>(sp)));
            float n0 = 0.f, n1 = 0.f;
#pragma unroll
            for (int sp = 0; sp < kMaxCluster; ++sp) {
                if (sp < C && ((mask >> sp) & 1u)) {
                    const float w = s_w[rl * kMaxCluster + sp];
                    n0 = fmaf(w, ov[sp].x, n0);
                    n1 = fmaf(w, ov[sp].y, n1);
                }
            }
            const float inv = s_rinv[rl];
            const int j = r / G, g = r - (r / G) * G;
            __nv_bfloat16* dst = out + static_cast<size_t>(b * K + j) * row_stride + static_cast<size_t>(kvh * G + g) * HD + d;
            *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(n0 * inv, n1 * inv);
        }
        cluster_sync_all();           // peers may still be reading this CTA's partial
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 256);
    }
}

// Combines the pieces of each (request, kv head) that has more than one:
// with M the largest running max of the pieces, a row's output is
// sum_i 2^(m_i - M) O_i / sum_i 2^(m_i - M) l_i. One thread per (query row,
// pair of dims); the pieces are read eight at a time (all loads of a batch in
// flight) and folded in piece order with a running max.
constexpr int kMergeThreads = 256;
constexpr int kMergeBatch = 8;

template <int HD>
__global__ void __launch_bounds__(kMergeThreads) k_attn_merge(const AttnParams p) {
    pdl_launch_dependents();
    pdl_wait();
    const int b = static_cast<int>(blockIdx.x) / p.nkv;
    const int kvh = static_cast<int>(blockIdx.x) - b * p.nkv;
    const int n = p.plan[1 + b];
    if (n <= 1) return;                        // written by its only piece
    const int G = p.nq / p.nkv;
    const int K = p.K;
    const int Rq = K * G;
    const int item = static_cast<int>(blockIdx.y) * kMergeThreads + static_cast<int>(threadIdx.x);
    const int r = item / (HD / 2);
    if (r >= Rq) return;
    const int d = (item - r * (HD / 2)) * 2;
    const int off = p.plan[1 + p.B + b];
    const int Rq4 = (Rq + 3) & ~3;
    const size_t pf = attn_piece_floats(Rq, HD);
    float M = -INFINITY, den = 0.f, n0 = 0.f, n1 = 0.f;
    for (int i0 = 0; i0 < n; i0 += kMergeBatch) {
        float mv[kMergeBatch], lv[kMergeBatch];
        float2 ov[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            mv[u] = -INFINITY;
            lv[u] = 0.f;
            ov[u] = make_float2(0.f, 0.f);
            const int slot = p.nkv * (off + i0 + u) + kvh;
            if (i0 + u < n && slot < p.grid) {
                const float* w = p.ws + static_cast<size_t>(slot) * pf;
                mv[u] = w[Rq * HD + r];
                lv[u] = w[Rq * HD + Rq4 + r];
                ov[u] = *reinterpret_cast<const float2*>(w + r * HD + d);
            }
        }
        float bm = M;
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u)
            if (lv[u] > 0.f) bm = fmaxf(bm, mv[u]);
        if (bm > M) {
            // earlier sums are relative to M: bring them to the new maximum
            const float f = exp2f(M - bm);     // 0 while nothing has been added
            den *= f;
            n0 *= f;
            n1 *= f;
            M = bm;
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            if (lv[u] > 0.f) {
                const float f = exp2f(mv[u] - M);
                den = fmaf(lv[u], f, den);
                n0 = fmaf(f, ov[u].x, n0);
                n1 = fmaf(f, ov[u].y, n1);
            }
        }
    }
    const bool req_ok = p.status[b] == PE_REQ_OK;
    const float inv = (req_ok && den > 0.f) ? 1.f / den : 0.f;
    const int j = r / G, g = r - (r / G) * G;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(b * K + j) * p.nq * HD +
                         static_cast<size_t>(kvh * G + g) * HD + d;
    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(n0 * inv, n1 * inv);
}

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

size_t umma_smem_bytes(int hd, int chunk) {
    const size_t pages = (static_cast<size_t>(chunk) / 16 + 4) * sizeof(int);
    const size_t base = hd == 128 ? static_cast<size_t>(Layout<128>::kPages) : static_cast<size_t>(Layout<64>::kPages);
    return base + pages + 1024;
}

// The dynamic shared-memory limit currently set on k_attn_umma<HD> per
// device: the occupancy queries below change it too, so every launch sets it
// again whenever it differs.
template <int HD>
size_t& smem_attr(int dev) {
    static size_t now[64] = {};
    return now[dev >= 0 && dev < 64 ? dev : 0];
}

template <int HD>
cudaError_t set_smem_attr(size_t smem) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (smem_attr<HD>(dev) == smem) return cudaSuccess;
    e = cudaFuncSetAttribute(k_attn_umma<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) smem_attr<HD>(dev) = smem;
    return e;
}

template <int HD>
int max_active(int C, size_t smem) {
    static int cache[kMaxCluster + 1] = {};
    if (cache[C] != 0) return cache[C];
    set_smem_attr<HD>(smem);
    cudaFuncSetAttribute(k_attn_umma<HD>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
    if (cudaOccupancyMaxActiveClusters(&n, k_attn_umma<HD>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = -1;
    }
    cache[C] = n == 0 ? -1 : n;
    return cache[C];
}

template <int HD>
int launch_hd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
              cudaStream_t s, bool pdl) {
    const size_t smem = umma_smem_bytes(HD, p.chunk);
    auto kern = k_attn_umma<HD>;
    PE_CUDA_TRY(set_smem_attr<HD>(smem));
    PE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = p.items != nullptr ? dim3(p.grid, 1) : dim3(p.B * p.nkv, p.max_splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = p.items != nullptr ? 1u : static_cast<unsigned>(p.max_splits);
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    PE_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p));
    return PE_OK;
}

}  // namespace

AttnPlan plan_attention_umma(int B, int K, int nq, int nkv, int hd, int max_pages, int page_size, int num_sms) {
    AttnPlan a{};
    const int max_entries = max_pages * page_size;
    const int pairs = B * nkv;
    if (pairs >= kPiecePairs && B <= kPieceMaxBatch) {
        // length-aware pieces while the pairs are fewer than one wave:
        // about total tiles / slots tiles each, where slots = the CTAs
        // resident at once, less one per pair when that keeps the pieces to
        // one wave
        const int chunk = ceil_div(max_entries, kTile) * kTile;
        const size_t smem = umma_smem_bytes(hd, chunk);
        static size_t q_smem[2] = {0, 0};
        static int q_per_sm[2] = {0, 0};
        const int hi = hd == 128 ? 1 : 0;
        if (q_smem[hi] != smem) {
            int n = 0;
            cudaError_t e;
            if (hd == 128) {
                set_smem_attr<128>(smem);
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_attn_umma<128>, kThreads, smem);
            } else {
                set_smem_attr<64>(smem);
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_attn_umma<64>, kThreads, smem);
            }
            if (e != cudaSuccess) {
                cudaGetLastError();
                n = 1;
            }
            q_smem[hi] = smem;
            q_per_sm[hi] = n;
        }
        const int per_sm = q_per_sm[hi];
        const int slots = num_sms * (per_sm > 0 ? per_sm : 1);
        if (pairs < slots) {
            a.pieces = true;
            a.piece_slots = pairs <= slots / 2 ? slots - pairs : slots;
            a.piece_wave = pairs <= slots / 2 ? slots : 0;
            a.piece_min_tiles = kPieceMinTiles;
            a.grid = a.piece_slots + pairs;
            a.chunk = chunk;
            a.max_splits = 1;
            (void)K;
            (void)nq;
            return a;
        }
        // a wave or more of (request, kv head) CTAs: issuing the longest
        // first already balances them
    }
    int want = ceil_div(num_sms, pairs);                 // about one wave of CTAs
    if (want > kMaxCluster) want = kMaxCluster;
    if (want < 1) want = 1;
    int chunk = ceil_div(max_entries, kTile) * kTile;
    for (int c = want; c >= 2; --c) {
        const int ch = ceil_div(ceil_div(max_entries, c), kTile) * kTile;
        const size_t smem = umma_smem_bytes(hd, ch);
        const int n = hd == 128 ? max_active<128>(c, smem) : max_active<64>(c, smem);
        if (n > 0 && n >= pairs) {                       // every cluster resident at once
            chunk = ch;
            break;
        }
    }
    a.chunk = chunk;
    a.max_splits = ceil_div(max_entries, chunk);         // one cluster of this many CTAs per (request, kv head)
    a.one_wave = static_cast<long long>(pairs) * a.max_splits <= num_sms;
    a.ws_floats = 0;
    a.tickets = 0;
    (void)K;
    (void)nq;
    return a;
}

int launch_attention_umma(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                          cudaStream_t s, bool pdl) {
    if (p.hd == 128) return launch_hd<128>(tq, tk, tv, p, s, pdl);
    if (p.hd == 64) return launch_hd<64>(tq, tk, tv, p, s, pdl);
    set_error("attention: head_dim must be 64 or 128");
    return PE_ERR_UNSUPPORTED;
}

int launch_attention_merge(const AttnParams& p, cudaStream_t s, bool pdl) {
    if (p.items == nullptr) return PE_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.B * p.nkv, ceil_div(p.K * (p.nq / p.nkv) * (p.hd / 2), kMergeThreads));
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.hd == 128) PE_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_attn_merge<128>, p));
    else PE_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_attn_merge<64>, p));
    return PE_OK;
}

}  // namespace pe
