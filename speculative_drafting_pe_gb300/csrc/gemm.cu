// tcgen05 weight-streaming GEMM with fused epilogues.
//
// D[m, n] = sum_k W[m, k] * X[n, k] with the weight rows on the 128-row M
// side of the MMA and the B*K token rows on the N side (16..256 per tile), so
// that at small batch the kernel streams each weight byte from HBM once.
//
// Roles (192 threads, one work unit per CTA):
//   warp 0      TMA producer: weight tile [128 x 128 B] + token tile
//               [bn x 128 B] per stage, 128-byte swizzle, into a smem ring.
//   warp 1      TMEM allocation; lane 0 issues tcgen05.mma (M=128, N=bn)
//               into an fp32 TMEM accumulator and commits stages back.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one TMEM lane per
//               thread), optional split-K reduction, fused epilogue.
//
// Split-K: every split writes its fp32 partial tile to scratch; the last
// split to arrive at the tile's ticket sums the partials in split order
// (0, 1, ..., S-1), so the result does not depend on arrival order, then
// applies the epilogue and resets the ticket for the next launch.
#include <type_traits>

#include "gemm_epi.cuh"

namespace pe {
namespace {

constexpr int kThreads = 192;
constexpr int kConvThreads = 128;            // warps 6..9: FP8 -> bf16 weight converters
constexpr int kThreadsW8 = kThreads + kConvThreads;
constexpr int kMaxClusterSplits = 8;         // cluster split-K: at most 8 CTAs per tile
constexpr int kConvStages = 2;               // W8: bf16 copies of half a weight stage, double-buffered
constexpr uint32_t kConvBytes = kABytes;     // 128 rows x 64 k: one SW128 bf16 tile

__host__ __device__ inline size_t gemm_smem_bytes(int stages, int bn, int inv_floats, bool w8, int cstages,
                                                  int egroups = 1) {
    const size_t b_stage = static_cast<size_t>(bn) * kRowBytes * (w8 ? 2 : 1);
    size_t off = static_cast<size_t>(stages) * (kABytes + b_stage);
    if (w8) off += static_cast<size_t>(cstages) * kConvBytes;
    off += static_cast<size_t>(2 * stages + 4 + 2 * kConvStages) * 8;   // mbarriers
    off += 16;                                        // TMEM base + flags
    off = (off + 15) & ~static_cast<size_t>(15);
    off += static_cast<size_t>(kChunk) * kPitch * 4 * egroups;  // epilogue staging tile per warp group
    off += static_cast<size_t>(inv_floats) * 4;       // folded-norm column scales
    return off + 1024;                                // base alignment slack
}

// FP8 weights: the scale of this thread's accumulator row (TMEM lane ml of
// weight tile m_tile).
template <int EPI>
__device__ __forceinline__ float w8_row_scale(const GemmParams& p, int m_tile, int ml) {
    if constexpr (EPI == EPI_SWIGLU) {
        const int f = m_tile * 64 + (ml & 63);
        if (f >= p.M) return 0.f;
        return ml < 64 ? p.w_scale[f] : p.w_scale2[f];
    } else {
        const int m = m_tile * kBM + ml;
        return m < p.M ? p.w_scale[m] : 0.f;
    }
}

template <bool W8>
__device__ __forceinline__ void scale_row(float (&v)[kChunk], float s) {
    if constexpr (W8) {
#pragma unroll
        for (int i = 0; i < kChunk; ++i) v[i] *= s;
    }
}

// Two E4M3 codes (bytes `lo_sel`/`hi_sel` of w) widened to a bf16 pair with
// integer operations only: PRMT places each code in the low byte of a 16-bit
// lane and replicates its sign bit into the high byte; shifted left by 4, the
// code's exponent and mantissa land in bf16's exponent and mantissa fields
// and a copy of the sign in bit 15, so the masked lane is the bf16 of
// value * 2^-120 (an E4M3 subnormal lands on a bf16 subnormal, zero on
// zero). One exact bf16 multiply by 2^120 restores the value. The NaN codes
// (S.1111.111) are not decoded as NaN: weights must be finite.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t w, uint32_t sel) {
    uint32_t t;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(t) : "r"(w), "r"(sel));
    const uint32_t v = (t << 4) & 0x87F087F0u;
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v);
    const uint32_t k = 0x7B807B80u;   // bf16 pair (2^120, 2^120)
    b = __hmul2(b, *reinterpret_cast<const __nv_bfloat162*>(&k));
    return *reinterpret_cast<const uint32_t*>(&b);
}

// Half `half` of one row of an FP8 weight stage (128 rows x 128 E4M3 codes,
// 128-byte swizzle) widened to bf16: codes k = 64 * half .. + 63 (chunks
// c = 4 * half .. + 3) become one 64-k tile in the same swizzle (the 16-byte
// chunk c of row r sits at r*128 + ((c ^ (r & 7)) << 4) in both tiles).
// E4M3 -> bf16 is exact (every finite E4M3 value is a bf16 value).
__device__ __forceinline__ void widen_fp8_row_half(const uint8_t* raw, uint8_t* conv, int r, int half) {
    const int sw = r & 7;
    const uint8_t* src = raw + r * kRowBytes;
#pragma unroll
    for (int c = 4 * half; c < 4 * half + 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + ((c ^ sw) << 4));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o[2 * i] = e4m3x2_to_bf16x2(w[i], 0x9180u);       // bytes 0, 1
            o[2 * i + 1] = e4m3x2_to_bf16x2(w[i], 0xB3A2u);   // bytes 2, 3
        }
        uint8_t* dst = conv + r * kRowBytes;
        const int j0 = 2 * (c & 3);
        *reinterpret_cast<uint4*>(dst + ((j0 ^ sw) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(dst + (((j0 + 1) ^ sw) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// With `ngrp` groups of epilogue warps (barrier `bar`, staging tile `stile`
// of their own), group `grp` takes the tile's 16-column chunks grp, grp +
// ngrp, ...; the scratch split-K path runs with one group only.
template <typename T, int EPI, bool W8>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, uint32_t t_acc, float* stile, int* sflag,
                                              float* part, const float* inv, float xg_g, float wsc, int m_tile,
                                              int n_tile, int split, int warp, int lane, int grp = 0,
                                              int ngrp = 1, int bar = 1) {
    const int quad = warp & 3;               // TMEM lane quadrant this warp may read
    const int ml = quad * 32 + lane;         // tile row = TMEM lane
    const uint32_t t_row = t_acc + (static_cast<uint32_t>(quad * 32) << 16);
    const int bn = p.bn;
    const int n_base = n_tile * bn;
    if (p.splits > 1 && p.cluster) {
        // cluster split-K: leave this split's partial tile in shared memory
        // (the stage ring is free once the accumulator is complete)
        for (int c0 = grp * kChunk; c0 < bn; c0 += ngrp * kChunk) {
            float v[kChunk];
            tmem_ld16(t_row + c0, v);
#pragma unroll
            for (int i = 0; i < kChunk; ++i) part[(c0 + i) * kBM + ml] = v[i];
        }
    } else if (p.splits > 1) {
        const int tile = m_tile * p.n_tiles + n_tile;
        float* mine = p.ws + (static_cast<size_t>(tile) * p.splits + split) * bn * kBM;
        for (int c0 = 0; c0 < bn; c0 += kChunk) {
            float v[kChunk];
            tmem_ld16(t_row + c0, v);
#pragma unroll
            for (int i = 0; i < kChunk; ++i) __stcg(mine + static_cast<size_t>(c0 + i) * kBM + ml, v[i]);
        }
        __threadfence();
        named_bar_sync(1, 128);
        if (ml == 0) {
            const int old = atomicAdd(p.tickets + tile, 1);
            const int last = (old == p.splits - 1) ? 1 : 0;
            if (last) atomicExch(p.tickets + tile, 0);
            sflag[1] = last;
        }
        named_bar_sync(1, 128);
        if (!sflag[1]) return;
        __threadfence();
        const float* base = p.ws + static_cast<size_t>(tile) * p.splits * bn * kBM;
        for (int c0 = 0; c0 < bn; c0 += kChunk) {
            float v[kChunk];
#pragma unroll
            for (int i = 0; i < kChunk; ++i) v[i] = 0.f;
            // issue the loads of up to kGroup splits at once, then add them
            // in split order (the sum does not depend on arrival order)
            constexpr int kGroup = 4;
            for (int s0 = 0; s0 < p.splits; s0 += kGroup) {
                float t[kGroup][kChunk];
#pragma unroll
                for (int u = 0; u < kGroup; ++u) {
                    if (s0 + u < p.splits) {
                        const float* src = base + (static_cast<size_t>(s0 + u) * bn + c0) * kBM + ml;
#pragma unroll
                        for (int i = 0; i < kChunk; ++i) t[u][i] = __ldcg(src + static_cast<size_t>(i) * kBM);
                    }
                }
#pragma unroll
                for (int u = 0; u < kGroup; ++u) {
                    if (s0 + u < p.splits) {
#pragma unroll
                        for (int i = 0; i < kChunk; ++i) v[i] += t[u][i];
                    }
                }
            }
            scale_row<W8>(v, wsc);
            scale_cols(v, inv, c0, 1, kChunk);
            apply_chunk<T, EPI>(p, v, ml, m_tile, ColMap{n_base + c0, 1, kChunk, c0}, stile, xg_g);
        }
        finish_norm_partials<EPI>(p, stile, m_tile, n_base, 1, bn, ml);
    } else {
        for (int c0 = grp * kChunk; c0 < bn; c0 += ngrp * kChunk) {
            float v[kChunk];
            tmem_ld16(t_row + c0, v);
            scale_row<W8>(v, wsc);
            scale_cols(v, inv, c0, 1, kChunk);
            apply_chunk<T, EPI>(p, v, ml, m_tile, ColMap{n_base + c0, 1, kChunk, c0}, stile, xg_g, bar);
        }
        finish_norm_partials<EPI>(p, stile, m_tile, n_base, 1, bn, ml, bar, grp, ngrp);
    }
}

// Cluster split-K, second half: after a cluster barrier, CTA `rank` sums the
// columns c = rank + j * splits over all peers' partial tiles (read through
// distributed shared memory, in split order) and applies the epilogue to
// them, 16 of its own columns per chunk.
template <typename T, int EPI, bool W8>
__device__ __forceinline__ void cluster_reduce(const GemmParams& p, float* stile, const float* part,
                                               const float* inv, float xg_g, float wsc, int m_tile, int n_tile,
                                               int warp, int lane, int grp = 0, int ngrp = 1, int bar = 1) {
    const int ml = (warp & 3) * 32 + lane;
    const int bn = p.bn;
    const int C = p.splits;
    const uint32_t rank = cluster_ctarank();
    const uint32_t base = smem_u32(part);
    const int first = static_cast<int>(rank);
    const int owned = first < bn ? (bn - first + C - 1) / C : 0;
    for (int j0 = grp * kChunk; j0 < owned; j0 += ngrp * kChunk) {
        const int cnt = min(kChunk, owned - j0);
        const int c0 = first + j0 * C;     // tile column of chunk column 0
        float v[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) v[i] = 0.f;
        // four columns at a time: all their peers' values in flight together,
        // then added in split order
#pragma unroll
        for (int i0 = 0; i0 < kChunk; i0 += 4) {
            if (i0 < cnt) {
                float t[4][kMaxClusterSplits];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t a = base + 4u * static_cast<uint32_t>((c0 + (i0 + u) * C) * kBM + ml);
#pragma unroll
                    for (int sp = 0; sp < kMaxClusterSplits; ++sp)
                        if (i0 + u < cnt && sp < C) t[u][sp] = dsmem_ld(dsmem_addr(a, static_cast<uint32_t>(sp)));
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
#pragma unroll
                    for (int sp = 0; sp < kMaxClusterSplits; ++sp)
                        if (i0 + u < cnt && sp < C) v[i0 + u] += t[u][sp];
                }
            }
        }
        scale_row<W8>(v, wsc);
        scale_cols(v, inv, c0, C, cnt);
        apply_chunk<T, EPI>(p, v, ml, m_tile, ColMap{n_tile * bn + c0, C, cnt, j0}, stile, xg_g, bar);
    }
    finish_norm_partials<EPI>(p, stile, m_tile, n_tile * bn + first, C, owned, ml, bar, grp, ngrp);
}

// ------------------------------------------------------------ kernel
//
// W8 (FP8 weights, bf16 activations): a stage holds 128 k of E4M3 weight
// codes (one 16 KB TMA box) and the matching two 64-k bf16 token tiles; the
// converter warps 6..9 widen each half stage (64 k) into one of two bf16
// tiles, alternately, so that one half converts while the MMA reads the
// other (the tensor cores see a bf16 x bf16 product: A and B of one
// kind::f16 MMA share a type).

// EG = 2 (bf16 weights, one CTA per SM): a second group of epilogue warps
// 6..9; the two groups take a tile's 16-column chunks in turn. ONE (FP8
// weights): compiled for one CTA per SM, which gives the 320 threads up to
// 168 registers instead of 96 (no split-K epilogue in local memory).
template <typename T, int EPI, bool W8, int EG, bool ONE = false>
__global__ void __launch_bounds__(W8 || EG == 2 ? kThreadsW8 : kThreads, EG == 2 || ONE ? 1 : 2)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
           const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stages = p.stages;
    const int bn = p.bn;
    const uint32_t b_box = static_cast<uint32_t>(bn) * kRowBytes;     // one 128-byte-wide token tile
    const uint32_t b_bytes = W8 ? 2 * b_box : b_box;                  // token bytes per stage
    uint8_t* sA = smem;
    uint8_t* sB = smem + static_cast<size_t>(stages) * kABytes;
    uint8_t* sC = sB + static_cast<size_t>(stages) * b_bytes;         // W8: bf16 copies of half stages
    const int cstages = W8 ? kConvStages : 0;
    uint64_t* full = reinterpret_cast<uint64_t*>(sC + static_cast<size_t>(cstages) * kConvBytes);
    uint64_t* empty = full + stages;
    uint64_t* tfull = empty + stages;      // [2] accumulator ready
    uint64_t* tempty = tfull + 2;          // [2] accumulator drained by the epilogue
    uint64_t* cfull = tempty + 2;          // [kConvStages] W8: bf16 copy written
    uint64_t* cempty = cfull + kConvStages;   // [kConvStages] W8: bf16 copy consumed by the MMA
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cempty + kConvStages);
    int* sflag = reinterpret_cast<int*>(tmem_slot + 1);
    float* stile = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(sflag + 3) + 15) & ~uintptr_t(15));
    float* s_inv = stile + kChunk * kPitch * EG;   // [inv_slots(N)] in the QKV and gate/up GEMMs

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Work units u = blockIdx.x, blockIdx.x + gridDim.x, ... (one unit per CTA
    // unless the launch is persistent). The splits of one tile are adjacent
    // (one cluster in cluster split-K mode), then n tiles, then m tiles.
    const int units = p.m_tiles * p.n_tiles * p.splits;
    auto decode = [&](int u, int& m_tile, int& n_tile, int& split, int& kb0, int& kb1) {
        split = u % p.splits;
        const int rest = u / p.splits;
        n_tile = rest % p.n_tiles;
        m_tile = rest / p.n_tiles;
        kb0 = split * p.kb_per_split;
        kb1 = min(p.kb_total, kb0 + p.kb_per_split);
    };
    const int nacc = p.persistent ? 2 : 1;           // double-buffered accumulator when persistent
    const bool inv_all = norm_scaled<EPI>(p) && p.N <= kMaxInvAll;
    float xg_g = 0.f;                                // folded RMSNorm gain of this epilogue thread's row
    float wsc = 1.f;                                 // W8: scale of this epilogue thread's row
    const uint32_t acc_cols = tmem_cols_for(bn);
    const uint32_t tmem_cols = acc_cols * static_cast<uint32_t>(nacc);

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        if constexpr (EPI == EPI_SWIGLU) tma_prefetch_desc(&tmA2);
        tma_prefetch_desc(&tmB);
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128 * EG);
        }
        if constexpr (W8) {
            for (int c = 0; c < cstages; ++c) {
                mbar_init(&cfull[c], kConvThreads);
                mbar_init(&cempty[c], 1);
            }
        }
        sflag[0] = 0;
        sflag[1] = 0;
        sflag[2] = 0;   // set when any wait of this CTA gives up
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    pdl_launch_dependents();
    // Everything but the producer and the converters waits here for the
    // previous kernel in the stream (a no-op without programmatic dependent
    // launch); the converters only touch weights. Warps 6..9 of the EG = 2
    // kernel are epilogue warps: they read the previous kernel's outputs.
    if (warp != 0 && (warp < 6 || EG == 2)) pdl_wait();

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_keep = l2_policy_evict_last();   // weight tiles kept in L2 across steps
            const uint64_t pol_x = l2_policy_evict_last();
            // k elements per stage: one 128-byte swizzle row of weights
            constexpr int kBK = W8 ? kRowBytes : kRowBytes / static_cast<int>(sizeof(T));
            int s = 0;
            uint32_t ph = 0;
            bool first = true, ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                int m_tile, n_tile, split, kb0, kb1;
                decode(u, m_tile, n_tile, split, kb0, kb1);
                auto load_a = [&](int st, int kb) {
                    uint8_t* a_dst = sA + static_cast<size_t>(st) * kABytes;
                    if constexpr (EPI == EPI_SWIGLU) {
                        tma_load_2d(a_dst, &tmA, &full[st], kb * kBK, m_tile * 64, pol_w);
                        tma_load_2d(a_dst + kABytes / 2, &tmA2, &full[st], kb * kBK, m_tile * 64, pol_w);
                    } else {
                        tma_load_2d(a_dst, &tmA, &full[st], kb * kBK, m_tile * kBM,
                                    m_tile < p.keep_tiles ? pol_keep : pol_w);
                    }
                };
                auto load_b = [&](int st, int kb) {
                    uint8_t* b_dst = sB + static_cast<size_t>(st) * b_bytes;
                    if constexpr (W8) {
                        // the stage's 128 k as two 64-element bf16 token tiles
                        tma_load_2d(b_dst, &tmB, &full[st], kb * kBK, n_tile * bn, pol_x);
                        tma_load_2d(b_dst + b_box, &tmB, &full[st], kb * kBK + kBK / 2, n_tile * bn, pol_x);
                    } else {
                        tma_load_2d(b_dst, &tmB, &full[st], kb * kBK, n_tile * bn, pol_x);
                    }
                };
                int kb = kb0;
                if (first) {
                    // Weights do not depend on earlier kernels: start streaming
                    // the first stages' weight tiles before the dependency
                    // wait, then add the token tiles of those stages.
                    const int pre = min(stages, kb1 - kb0);
                    for (int i = 0; i < pre; ++i) {
                        mbar_arrive_expect_tx(&full[i], kABytes + b_bytes);
                        load_a(i, kb0 + i);
                    }
                    pdl_wait();
                    for (int i = 0; i < pre; ++i) load_b(i, kb0 + i);
                    s = pre % stages;
                    ph = (pre == stages) ? 1u : 0u;
                    kb = kb0 + pre;
                    first = false;
                }
                for (; kb < kb1; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, p.err, PE_DEVERR_GEMM_TIMEOUT)) {
                        ok = false;
                        sflag[2] = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], kABytes + b_bytes);
                    load_a(s, kb);
                    load_b(s, kb);
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (first) pdl_wait();
        }
        __syncwarp();   // reconverge before the CTA-wide barriers of the teardown
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = umma_idesc(UmmaKind<T>::kFmt, kBM, bn);
            int s = 0;
            uint32_t ph = 0;
            int c = 0;
            uint32_t cph = 0;
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++it) {
                int m_tile, n_tile, split, kb0, kb1;
                decode(u, m_tile, n_tile, split, kb0, kb1);
                const int acc = it % nacc;
                const int use = it / nacc;
                // wait until the epilogue has drained this accumulator's previous use
                if (!mbar_wait(&tempty[acc], static_cast<uint32_t>(use & 1) ^ 1u, p.err, PE_DEVERR_GEMM_TIMEOUT)) {
                    ok = false;
                    sflag[2] = 1;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * acc_cols;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full[s], ph, p.err, PE_DEVERR_GEMM_TIMEOUT)) {
                        ok = false;
                        sflag[2] = 1;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t b_addr = smem_u32(sB + static_cast<size_t>(s) * b_bytes);
                    if constexpr (W8) {
                        // each half stage as soon as its bf16 copy is ready
                        for (int half = 0; half < 2 && ok; ++half) {
                            if (!mbar_wait(&cfull[c], cph, p.err, PE_DEVERR_GEMM_TIMEOUT)) {
                                ok = false;
                        sflag[2] = 1;
                                break;
                            }
                            tc_fence_after_sync();
                            const uint32_t a_addr = smem_u32(sC + static_cast<size_t>(c) * kConvBytes);
#pragma unroll
                            for (int kk = 0; kk < kRowBytes / 32; ++kk) {
                                UmmaKind<T>::mma(d_tmem, umma_desc_sw128(a_addr + kk * 32),
                                                 umma_desc_sw128(b_addr + half * b_box + kk * 32), idesc,
                                                 (kb > kb0 || half > 0 || kk > 0) ? 1u : 0u);
                            }
                            umma_commit(&cempty[c]);
                            if (++c == cstages) {
                                c = 0;
                                cph ^= 1u;
                            }
                        }
                        if (!ok) break;
                    } else {
                        const uint32_t a_addr = smem_u32(sA + static_cast<size_t>(s) * kABytes);
#pragma unroll
                        for (int kk = 0; kk < kRowBytes / 32; ++kk) {
                            UmmaKind<T>::mma(d_tmem, umma_desc_sw128(a_addr + kk * 32),
                                             umma_desc_sw128(b_addr + kk * 32), idesc,
                                             (kb > kb0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    umma_commit(&empty[s]);
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                umma_commit(&tfull[acc]);
            }
        }
        __syncwarp();
    } else if (W8 && warp >= 6) {   // warps 6..9
        // converters: widen each weight stage into the next bf16 copy, in the
        // MMA's order; the MMA releases the raw stage, so the codes stay put
        // until the copy is complete
        if constexpr (W8) {
            const int t = static_cast<int>(threadIdx.x) - 192;
            int s = 0;
            uint32_t ph = 0;
            int c = 0;
            uint32_t cph = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                int m_tile, n_tile, split, kb0, kb1;
                decode(u, m_tile, n_tile, split, kb0, kb1);
                for (int kb = kb0; kb < kb1 && ok; ++kb) {
                    if (!mbar_wait(&full[s], ph, p.err, PE_DEVERR_GEMM_TIMEOUT)) {
                        ok = false;
                        sflag[2] = 1;
                        break;
                    }
                    for (int half = 0; half < 2; ++half) {
                        if (!mbar_wait(&cempty[c], cph ^ 1u, p.err, PE_DEVERR_GEMM_TIMEOUT)) {
                            ok = false;
                        sflag[2] = 1;
                            break;
                        }
                        for (int r = t; r < kBM; r += kConvThreads)
                            widen_fp8_row_half(sA + static_cast<size_t>(s) * kABytes,
                                               sC + static_cast<size_t>(c) * kConvBytes, r, half);
                        fence_proxy_async_smem();   // the MMA (async proxy) reads what these threads wrote
                        mbar_arrive(&cfull[c]);
                        if (++c == cstages) {
                            c = 0;
                            cph ^= 1u;
                        }
                    }
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else {
        // Folded RMSNorm: the scales of every token row, computed once while
        // the first mainloop runs (published by the barrier after the first
        // accumulator wait), unless there are too many rows for shared memory.
        const int grp = (EG == 2 && warp >= 6) ? 1 : 0;     // epilogue warp group
        const int bar = 1 + grp;                             // its named barrier (128 threads)
        float* stile_g = stile + grp * kChunk * kPitch;      // its staging tile
        if constexpr (epi_norm_scaled<EPI>()) {
            if (inv_all) fold_norm_scales(p, s_inv, 0, p.N, threadIdx.x - 64, 128 * EG);
        }
        int it = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++it) {
            int m_tile, n_tile, split, kb0, kb1;
            decode(u, m_tile, n_tile, split, kb0, kb1);
            const int acc = it % nacc;
            const int use = it / nacc;
            const float* inv = nullptr;
            if (inv_all) {
                inv = s_inv + n_tile * bn;
            } else if (norm_scaled<EPI>(p)) {
                if constexpr (epi_norm_scaled<EPI>()) {
                    // double-buffered: the previous tile's epilogue may still read the other half
                    float* buf = s_inv + (it & 1) * kMaxBn;
                    fold_norm_scales(p, buf, n_tile * bn, bn, threadIdx.x - 64);   // (one warp group)
                    inv = buf;
                }
            }
            if constexpr (EPI == EPI_RESID) {
                // gain of this thread's output row for the folded RMSNorm
                const int m = m_tile * kBM + (warp & 3) * 32 + lane;
                xg_g = (p.xg != nullptr && m < p.M) ? Elem<T>::to_f(static_cast<const T*>(p.xg_gain)[m]) : 0.f;
            }
            if constexpr (W8) wsc = w8_row_scale<EPI>(p, m_tile, (warp & 3) * 32 + lane);
            const bool ok = mbar_wait(&tfull[acc], static_cast<uint32_t>(use & 1), p.err, PE_DEVERR_GEMM_TIMEOUT);
            tc_fence_after_sync();
            if (!ok) {
                sflag[0] = 1;
                sflag[2] = 1;
            }
            // both groups: the scales and sflag written before it are published
            named_bar_sync(EG == 2 ? 3 : 1, 128 * EG);
            if (sflag[0]) break;
            epilogue_tile<T, EPI, W8>(p, tmem_base + static_cast<uint32_t>(acc) * acc_cols, stile_g, sflag,
                                      reinterpret_cast<float*>(smem), inv, xg_g, wsc, m_tile, n_tile, split, warp,
                                      lane, grp, EG, bar);
            tc_fence_before_sync();
            mbar_arrive(&tempty[acc]);
        }
    }
    if (p.splits > 1 && p.cluster) {
        // cluster split-K (one unit per CTA): reduce through distributed shared memory
        int m_tile, n_tile, split, kb0, kb1;
        decode(blockIdx.x, m_tile, n_tile, split, kb0, kb1);
        __syncthreads();              // this CTA's partial is in shared memory
        cluster_sync_all();           // ... and so are the peers'
        if (warp >= 2 && warp < (EG == 2 ? 10 : 6) && !sflag[0]) {
            const int grp = (EG == 2 && warp >= 6) ? 1 : 0;
            const float* inv = inv_all ? s_inv + n_tile * bn : (norm_scaled<EPI>(p) ? s_inv : nullptr);
            cluster_reduce<T, EPI, W8>(p, stile + grp * kChunk * kPitch, reinterpret_cast<const float*>(smem), inv,
                                       xg_g, wsc, m_tile, n_tile, warp, lane, grp, EG, 1 + grp);
        }
        cluster_sync_all();           // peers are done reading this CTA's partial
    }

    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && *reinterpret_cast<volatile int*>(&sflag[2])) {
        // A wait of this CTA gave up: let any bulk copy still in flight land
        // before its shared memory is released.
        __nanosleep(100000);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, tmem_cols);
    }
}

template <typename T, int EPI, bool W8, int EG, bool ONE = false>
int launch_typed(const CUtensorMap& A, const CUtensorMap& A2, const CUtensorMap& B, const GemmPlan& plan,
                 const GemmParams& p, cudaStream_t stream, bool pdl) {
    auto kern = k_gemm<T, EPI, W8, EG, ONE>;
    static size_t smem_set[64] = {};
    int dev = 0;
    PE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64 || plan.smem_bytes > smem_set[dev]) {
        PE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(plan.smem_bytes)));
        PE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
        if (dev >= 0 && dev < 64) smem_set[dev] = plan.smem_bytes;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(W8 || EG == 2 ? kThreadsW8 : kThreads);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    int na = 1;
    if (p.cluster && plan.splits > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(plan.splits);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    PE_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, A, A2, B, p));
    return PE_OK;
}

template <typename T, bool W8>
int launch_dispatch(int epi, const CUtensorMap& A, const CUtensorMap& A2, const CUtensorMap& B,
                    const GemmPlan& plan, const GemmParams& p, cudaStream_t stream, bool pdl) {
    if constexpr (!W8 && std::is_same<T, __nv_bfloat16>::value) {
        if (plan.epi_groups == 2) {
            switch (epi) {
                case EPI_STORE: return launch_typed<T, EPI_STORE, W8, 2>(A, A2, B, plan, p, stream, pdl);
                case EPI_QKV: return launch_typed<T, EPI_QKV, W8, 2>(A, A2, B, plan, p, stream, pdl);
                case EPI_RESID: return launch_typed<T, EPI_RESID, W8, 2>(A, A2, B, plan, p, stream, pdl);
                case EPI_SWIGLU: return launch_typed<T, EPI_SWIGLU, W8, 2>(A, A2, B, plan, p, stream, pdl);
                default: set_error("GEMM epilogue without a second epilogue warp group"); return PE_ERR_ARG;
            }
        }
    }
    if (plan.epi_groups != 1) {
        set_error("GEMM plan with two epilogue warp groups for FP8 or fp32 weights");
        return PE_ERR_ARG;
    }
    if constexpr (W8) {
        if (plan.w8_one) {
            switch (epi) {
                case EPI_QKV: return launch_typed<T, EPI_QKV, W8, 1, true>(A, A2, B, plan, p, stream, pdl);
                case EPI_RESID: return launch_typed<T, EPI_RESID, W8, 1, true>(A, A2, B, plan, p, stream, pdl);
                case EPI_SWIGLU: return launch_typed<T, EPI_SWIGLU, W8, 1, true>(A, A2, B, plan, p, stream, pdl);
                default: set_error("GEMM epilogue without a one-CTA-per-SM FP8 kernel"); return PE_ERR_ARG;
            }
        }
    }
    switch (epi) {
        case EPI_STORE: return launch_typed<T, EPI_STORE, W8, 1>(A, A2, B, plan, p, stream, pdl);
        case EPI_QKV: return launch_typed<T, EPI_QKV, W8, 1>(A, A2, B, plan, p, stream, pdl);
        case EPI_RESID: return launch_typed<T, EPI_RESID, W8, 1>(A, A2, B, plan, p, stream, pdl);
        case EPI_SWIGLU: return launch_typed<T, EPI_SWIGLU, W8, 1>(A, A2, B, plan, p, stream, pdl);
        case EPI_ARGMAX: return launch_typed<T, EPI_ARGMAX, W8, 1>(A, A2, B, plan, p, stream, pdl);
        default: set_error("unknown GEMM epilogue"); return PE_ERR_ARG;
    }
}

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline int round_up(int a, int b) { return ceil_div(a, b) * b; }

}  // namespace

GemmPlan plan_gemm(int M, int N, int Kd, int epi, int elem_bytes, int num_sms, bool cluster, bool w8) {
    GemmPlan g{};
    g.w8 = w8;
    // k elements per stage: one 128-byte swizzle row of weights (128 FP8 codes)
    const int bk = w8 ? kRowBytes : kRowBytes / elem_bytes;
    g.kb_total = ceil_div(Kd, bk);
    // token tile: up to 256 rows (128 with FP8 weights, whose stages carry
    // two token tiles each next to the bf16 weight copies)
    const int bn_max = w8 ? 128 : 256;
    if (N <= bn_max) {
        g.n_tiles = 1;
        g.bn = round_up(N < 1 ? 1 : N, 16);
    } else {
        g.n_tiles = ceil_div(N, bn_max);
        g.bn = round_up(ceil_div(N, g.n_tiles), 16);
    }
    const int rows_per_tile = epi == EPI_SWIGLU ? 64 : kBM;
    g.m_tiles = ceil_div(M, rows_per_tile);
    if (epi == EPI_RESID && cluster && N > 256 && !w8) {
        // O and down have few weight tiles (16 at the Qwen shape): narrower
        // token tiles, down to 128 rows, when that lets the tiles fill one
        // wave of SMs
        const int n_fill = num_sms / g.m_tiles;
        if (n_fill > g.n_tiles) {
            const int bn2 = round_up(ceil_div(N, n_fill), 16);
            if (bn2 >= 128) {
                g.bn = bn2;
                g.n_tiles = ceil_div(N, bn2);
            }
        }
    }
    if (epi == EPI_RESID && cluster && N > 128 && N <= 256 && !w8) {
        // one token tile of 129-256 rows takes the large ring (one CTA per
        // SM); two tiles of <= 128 rows measured faster (224 rows: O 140 ->
        // 88 us, down 150 -> 98 us per step)
        g.n_tiles = 2;
        g.bn = round_up(ceil_div(N, 2), 16);
    }
    if ((epi == EPI_SWIGLU || epi == EPI_ARGMAX) && cluster && N > 128 && N <= 512 && !w8) {
        // gate/up and the LM head (equal token tiles: they share the
        // activation tile shape) up to 512 rows: tiles of <= 128 rows
        // (352 and 384 rows: gate/up 156 -> 117 us and LM head 184 -> 175 us
        // per step against 176/192-row tiles; at 896 rows 128-row tiles were
        // slower)
        g.n_tiles = ceil_div(N, 128);
        g.bn = round_up(ceil_div(N, g.n_tiles), 16);
    }
    if (epi == EPI_QKV && cluster && N > 128 && !w8) {
        // QKV (40 weight tiles at the Qwen shape): the token tile that
        // minimises ceil(tiles / SMs) * tile width, the busiest SM's share of
        // the work (ties to the narrower tile). Measured: at 1408 rows 96-row
        // tiles (600 tiles, two CTAs per SM) 263 -> 203 us per step against
        // 240-row tiles; at 224 rows 80-row tiles 155 -> 118 us against one
        // 224-row tile; at 352 rows it picks 128 (3 tiles of 128, as tuned).
        int best_bn = g.bn, best_nt = g.n_tiles;
        long long best = static_cast<long long>(ceil_div(g.m_tiles * g.n_tiles, num_sms)) * g.bn;
        for (int cand = 96; cand < g.bn; cand += 16) {
            const int nt = ceil_div(N, cand);
            const int bn2 = round_up(ceil_div(N, nt), 16);
            const long long cost = static_cast<long long>(ceil_div(g.m_tiles * nt, num_sms)) * bn2;
            if (cost < best || (cost == best && bn2 < best_bn)) {
                best = cost;
                best_bn = bn2;
                best_nt = nt;
            }
        }
        g.bn = best_bn;
        g.n_tiles = best_nt;
    }
    g.tiles = g.m_tiles * g.n_tiles;
    // shared-memory ring: ~100 KB (two CTAs per SM, so the next kernel's CTAs
    // can start their weight loads beside this one) for token tiles up to
    // 128 rows; ~190 KB above that (at 96 rows the small ring measured 17%
    // faster per step, at 176 rows its two stages were much slower)
    const size_t stage = kABytes + static_cast<size_t>(g.bn) * kRowBytes * (w8 ? 2 : 1);
    const int inv_floats = (epi == EPI_QKV || epi == EPI_SWIGLU) ? inv_slots(N) : 0;
    // FP8 weights: two 16 KB bf16 copies of half stages; up to 64 token rows
    // the ring keeps the CTA within ~112 KB (two CTAs per SM, so the next
    // kernel's CTAs can start streaming beside it, as in the bf16 path);
    // wider token tiles take one CTA per SM (~215 KB)
    g.cstages = w8 ? kConvStages : 0;
    const size_t fixed = static_cast<size_t>(g.cstages) * kConvBytes + static_cast<size_t>(kChunk) * kPitch * 4 +
                         static_cast<size_t>(inv_floats) * 4 + 2048;
    // The ~190 KB ring (one CTA per SM, which brings the second epilogue
    // group) for bf16 tiles of up to 128 rows too where it measured faster:
    // QKV from 65 rows while its tiles fit one wave (B=32, K=11: 133 -> 108
    // us per step; 600 tiles at 1408 rows were slower), gate/up from 49 to
    // 128 rows (one token tile: 88 rows 100 -> 84 us; slower below 48 and at
    // two or three tiles), O and down at 129-256 rows (their two tiles:
    // 224 rows O 89 -> 77, down 100 -> 85 us)
    bool big = false;
    if (cluster && !w8 && elem_bytes == 2 && g.bn <= 128) {
        if (epi == EPI_QKV) big = N > 64 && g.tiles <= num_sms;
        else if (epi == EPI_SWIGLU) big = N > 48 && N <= 128;
        else if (epi == EPI_RESID) big = N > 128 && N <= 256;
    }
    // FP8 weights, one CTA per SM (compiled for up to 168 registers): gate/up
    // always, QKV and O/down above 128 token rows; with fewer rows QKV and
    // O/down measured faster at two CTAs per SM (96 registers), where they
    // start streaming their weights beside the attention's CTAs
    // (B=1, K=7: O and down 72/76 -> 98/108 us per step at one CTA per SM;
    // B=128, K=11: O, down and QKV 394/463/402 -> 282/381/299)
    g.w8_one = w8 && (epi == EPI_SWIGLU || ((epi == EPI_QKV || epi == EPI_RESID) && N > 128));
    const size_t budget = w8 ? ((g.bn <= 64 && !g.w8_one) ? 112 * 1024 : 215 * 1024) - fixed
                             : ((g.bn <= 128 && !big) ? 100 * 1024 : 190 * 1024);
    int st = static_cast<int>(budget / stage);
    g.stages = st < 2 ? 2 : (st > 8 ? 8 : st);
    g.smem_bytes = gemm_smem_bytes(g.stages, g.bn, inv_floats, w8, g.cstages);
    const int ctas_per_sm = g.w8_one ? 1 : (g.smem_bytes <= 113 * 1024 ? 2 : 1);
    int splits = 1;
    if (epi != EPI_ARGMAX) {
        if (cluster) {
            // the splits of a tile form one cluster of <= 8 CTAs; aim at about
            // one CTA per SM, which leaves room on each SM for the next
            // kernel's CTAs to start streaming their weights early
            // (programmatic dependent launch). The QKV GEMM (RoPE and cache
            // scatter in its epilogue) measured faster with ~1.5 per SM.
            const int target = (epi == EPI_QKV && ctas_per_sm == 2) ? (num_sms * 3) / 2 : num_sms;
            const int max_c = kMaxClusterSplits;
            splits = target / g.tiles;
            splits = splits > max_c ? max_c : splits;
            const int cap = g.kb_total / 2 > 1 ? g.kb_total / 2 : 1;   // >= 2 k-blocks per split
            splits = splits < cap ? splits : cap;
            splits = splits < 1 ? 1 : splits;
        } else if (g.tiles < 2 * num_sms) {
            splits = ceil_div(2 * num_sms, g.tiles);
            const int cap = g.kb_total / 4 > 1 ? g.kb_total / 4 : 1;   // >= 4 k-blocks per split
            splits = splits < cap ? splits : cap;
        }
    }
    g.kb_per_split = ceil_div(g.kb_total, splits);
    g.splits = ceil_div(g.kb_total, g.kb_per_split);
    g.cluster = cluster && g.splits > 1;
    if (g.cluster && static_cast<size_t>(g.stages) * stage < static_cast<size_t>(g.bn) * kBM * 4) {
        // the partial tile must fit in the freed stage ring
        g.kb_per_split = g.kb_total;
        g.splits = 1;
        g.cluster = false;
    }
    g.units = g.tiles * g.splits;
    // Without split-K the kernel is persistent: one CTA per resident slot
    // walks the tiles with a double-buffered TMEM accumulator, so the
    // epilogue of one tile overlaps the mainloop of the next.
    g.persistent = g.splits == 1 && g.units > 1;
    g.grid = g.persistent ? (g.units < num_sms * ctas_per_sm ? g.units : num_sms * ctas_per_sm) : g.units;
    g.ws_floats = (g.splits > 1 && !g.cluster) ? static_cast<size_t>(g.tiles) * g.splits * g.bn * kBM : 0;
    // One CTA per SM (token tiles over 128 rows) leaves room for a second
    // group of epilogue warps, whose share of each tile's 16-column chunks
    // halves the epilogue after the last MMA (bf16 weights; the norm scales
    // of every token row must fit in shared memory; not the LM head)
    g.epi_groups = 1;
    if (cluster && !w8 && elem_bytes == 2 && ctas_per_sm == 1 && epi != EPI_ARGMAX && N <= kMaxInvAll &&
        (g.splits == 1 || g.cluster)) {
        g.epi_groups = 2;
        g.smem_bytes = gemm_smem_bytes(g.stages, g.bn, inv_floats, w8, g.cstages, 2);
    }
    return g;
}

int gemm_store_kernels_load() {
    cudaFuncAttributes fa;
    PE_CUDA_TRY(cudaFuncGetAttributes(&fa, k_gemm<__nv_bfloat16, EPI_STORE, false, 1>));
    PE_CUDA_TRY(cudaFuncGetAttributes(&fa, k_gemm<float, EPI_STORE, false, 1>));
    return PE_OK;
}

int launch_gemm(int dtype, int epi, const CUtensorMap& A, const CUtensorMap& A2, const CUtensorMap& B,
                const GemmPlan& plan, GemmParams p, cudaStream_t stream, bool pdl) {
    p.m_tiles = plan.m_tiles;
    p.n_tiles = plan.n_tiles;
    p.splits = plan.splits;
    p.kb_total = plan.kb_total;
    p.kb_per_split = plan.kb_per_split;
    p.bn = plan.bn;
    p.stages = plan.stages;
    p.cstages = plan.cstages;
    p.cluster = plan.cluster ? 1 : 0;
    p.persistent = plan.persistent ? 1 : 0;
    if (plan.w8) {
        if (dtype != PE_DTYPE_BF16 || p.w_scale == nullptr || (epi == EPI_SWIGLU && p.w_scale2 == nullptr)) {
            set_error("FP8 weights need bf16 activations and per-row weight scales");
            return PE_ERR_ARG;
        }
        return launch_dispatch<__nv_bfloat16, true>(epi, A, A2, B, plan, p, stream, pdl);
    }
    if (dtype == PE_DTYPE_BF16) return launch_dispatch<__nv_bfloat16, false>(epi, A, A2, B, plan, p, stream, pdl);
    return launch_dispatch<float, false>(epi, A, A2, B, plan, p, stream, pdl);
}

}  // namespace pe
