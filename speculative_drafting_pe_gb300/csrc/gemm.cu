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
#include "gemm_epi.cuh"

namespace pe {
namespace {

constexpr int kThreads = 192;
constexpr int kMaxClusterSplits = 8;         // cluster split-K: at most 8 CTAs per tile

__host__ __device__ inline size_t gemm_smem_bytes(int stages, int bn, int inv_floats) {
    size_t off = static_cast<size_t>(stages) * (kABytes + static_cast<size_t>(bn) * kRowBytes);
    off += static_cast<size_t>(2 * stages + 4) * 8;   // mbarriers
    off += 16;                                        // TMEM base + flags
    off = (off + 15) & ~static_cast<size_t>(15);
    off += static_cast<size_t>(kChunk) * kPitch * 4;  // epilogue staging tile
    off += static_cast<size_t>(inv_floats) * 4;       // folded-norm column scales
    return off + 1024;                                // base alignment slack
}

template <typename T, int EPI>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, uint32_t t_acc, float* stile, int* sflag,
                                              float* part, const float* inv, float xg_g, int m_tile, int n_tile,
                                              int split, int warp, int lane) {
    const int quad = warp & 3;               // TMEM lane quadrant this warp may read
    const int ml = quad * 32 + lane;         // tile row = TMEM lane
    const uint32_t t_row = t_acc + (static_cast<uint32_t>(quad * 32) << 16);
    const int bn = p.bn;
    const int n_base = n_tile * bn;
    if (p.splits > 1 && p.cluster) {
        // cluster split-K: leave this split's partial tile in shared memory
        // (the stage ring is free once the accumulator is complete)
        for (int c0 = 0; c0 < bn; c0 += kChunk) {
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
            scale_cols(v, inv, c0, 1, kChunk);
            apply_chunk<T, EPI>(p, v, ml, m_tile, ColMap{n_base + c0, 1, kChunk, c0}, stile, xg_g);
        }
        finish_norm_partials<EPI>(p, stile, m_tile, n_base, 1, bn, ml);
    } else {
        for (int c0 = 0; c0 < bn; c0 += kChunk) {
            float v[kChunk];
            tmem_ld16(t_row + c0, v);
            scale_cols(v, inv, c0, 1, kChunk);
            apply_chunk<T, EPI>(p, v, ml, m_tile, ColMap{n_base + c0, 1, kChunk, c0}, stile, xg_g);
        }
        finish_norm_partials<EPI>(p, stile, m_tile, n_base, 1, bn, ml);
    }
}

// Cluster split-K, second half: after a cluster barrier, CTA `rank` sums the
// columns c = rank + j * splits over all peers' partial tiles (read through
// distributed shared memory, in split order) and applies the epilogue to
// them, 16 of its own columns per chunk.
template <typename T, int EPI>
__device__ __forceinline__ void cluster_reduce(const GemmParams& p, float* stile, const float* part,
                                               const float* inv, float xg_g, int m_tile, int n_tile, int warp,
                                               int lane) {
    const int ml = (warp & 3) * 32 + lane;
    const int bn = p.bn;
    const int C = p.splits;
    const uint32_t rank = cluster_ctarank();
    const uint32_t base = smem_u32(part);
    const int first = static_cast<int>(rank);
    const int owned = first < bn ? (bn - first + C - 1) / C : 0;
    for (int j0 = 0; j0 < owned; j0 += kChunk) {
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
        scale_cols(v, inv, c0, C, cnt);
        apply_chunk<T, EPI>(p, v, ml, m_tile, ColMap{n_tile * bn + c0, C, cnt, j0}, stile, xg_g);
    }
    finish_norm_partials<EPI>(p, stile, m_tile, n_tile * bn + first, C, owned, ml);
}

// ------------------------------------------------------------ kernel

template <typename T, int EPI>
__global__ void __launch_bounds__(kThreads, 2)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
           const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stages = p.stages;
    const int bn = p.bn;
    const uint32_t b_bytes = static_cast<uint32_t>(bn) * kRowBytes;
    uint8_t* sA = smem;
    uint8_t* sB = smem + static_cast<size_t>(stages) * kABytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + static_cast<size_t>(stages) * b_bytes);
    uint64_t* empty = full + stages;
    uint64_t* tfull = empty + stages;      // [2] accumulator ready
    uint64_t* tempty = tfull + 2;          // [2] accumulator drained by the epilogue
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
    int* sflag = reinterpret_cast<int*>(tmem_slot + 1);
    float* stile = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(sflag + 3) + 15) & ~uintptr_t(15));
    float* s_inv = stile + kChunk * kPitch;   // [inv_slots(N)] in the QKV and gate/up GEMMs

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
            mbar_init(&tempty[a], 128);
        }
        sflag[0] = 0;
        sflag[1] = 0;
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
    // Everything but the producer waits here for the previous kernel in the
    // stream (a no-op without programmatic dependent launch).
    if (warp != 0) pdl_wait();

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_keep = l2_policy_evict_last();   // weight tiles kept in L2 across steps
            const uint64_t pol_x = l2_policy_evict_last();
            constexpr int kBK = kRowBytes / static_cast<int>(sizeof(T));
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
                    tma_load_2d(sB + static_cast<size_t>(st) * b_bytes, &tmB, &full[st], kb * kBK, n_tile * bn,
                                pol_x);
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
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * acc_cols;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full[s], ph, p.err, PE_DEVERR_GEMM_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_addr = smem_u32(sA + static_cast<size_t>(s) * kABytes);
                    const uint32_t b_addr = smem_u32(sB + static_cast<size_t>(s) * b_bytes);
#pragma unroll
                    for (int kk = 0; kk < kRowBytes / 32; ++kk) {
                        UmmaKind<T>::mma(d_tmem, umma_desc_sw128(a_addr + kk * 32), umma_desc_sw128(b_addr + kk * 32),
                                         idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
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
    } else {
        // Folded RMSNorm: the scales of every token row, computed once while
        // the first mainloop runs (published by the barrier after the first
        // accumulator wait), unless there are too many rows for shared memory.
        if constexpr (epi_norm_scaled<EPI>()) {
            if (inv_all) fold_norm_scales(p, s_inv, 0, p.N, threadIdx.x - 64);
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
                    fold_norm_scales(p, buf, n_tile * bn, bn, threadIdx.x - 64);
                    inv = buf;
                }
            }
            if constexpr (EPI == EPI_RESID) {
                // gain of this thread's output row for the folded RMSNorm
                const int m = m_tile * kBM + (warp & 3) * 32 + lane;
                xg_g = (p.xg != nullptr && m < p.M) ? Elem<T>::to_f(static_cast<const T*>(p.xg_gain)[m]) : 0.f;
            }
            const bool ok = mbar_wait(&tfull[acc], static_cast<uint32_t>(use & 1), p.err, PE_DEVERR_GEMM_TIMEOUT);
            tc_fence_after_sync();
            if (!ok) sflag[0] = 1;
            named_bar_sync(1, 128);
            if (sflag[0]) break;
            epilogue_tile<T, EPI>(p, tmem_base + static_cast<uint32_t>(acc) * acc_cols, stile, sflag,
                                  reinterpret_cast<float*>(smem), inv, xg_g, m_tile, n_tile, split, warp, lane);
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
        if (warp >= 2 && !sflag[0]) {
            const float* inv = inv_all ? s_inv + n_tile * bn : (norm_scaled<EPI>(p) ? s_inv : nullptr);
            cluster_reduce<T, EPI>(p, stile, reinterpret_cast<const float*>(smem), inv, xg_g, m_tile, n_tile, warp,
                                   lane);
        }
        cluster_sync_all();           // peers are done reading this CTA's partial
    }

    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && p.err != nullptr && (*reinterpret_cast<volatile unsigned*>(p.err) & PE_DEVERR_GEMM_TIMEOUT)) {
        // A wait gave up: let any bulk copy still in flight land before this
        // CTA's shared memory is released.
        __nanosleep(100000);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, tmem_cols);
    }
}

template <typename T, int EPI>
int launch_typed(const CUtensorMap& A, const CUtensorMap& A2, const CUtensorMap& B, const GemmPlan& plan,
                 const GemmParams& p, cudaStream_t stream, bool pdl) {
    auto kern = k_gemm<T, EPI>;
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
    cfg.blockDim = dim3(kThreads);
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

template <typename T>
int launch_dispatch(int epi, const CUtensorMap& A, const CUtensorMap& A2, const CUtensorMap& B,
                    const GemmPlan& plan, const GemmParams& p, cudaStream_t stream, bool pdl) {
    switch (epi) {
        case EPI_STORE: return launch_typed<T, EPI_STORE>(A, A2, B, plan, p, stream, pdl);
        case EPI_QKV: return launch_typed<T, EPI_QKV>(A, A2, B, plan, p, stream, pdl);
        case EPI_RESID: return launch_typed<T, EPI_RESID>(A, A2, B, plan, p, stream, pdl);
        case EPI_SWIGLU: return launch_typed<T, EPI_SWIGLU>(A, A2, B, plan, p, stream, pdl);
        case EPI_ARGMAX: return launch_typed<T, EPI_ARGMAX>(A, A2, B, plan, p, stream, pdl);
        default: set_error("unknown GEMM epilogue"); return PE_ERR_ARG;
    }
}

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline int round_up(int a, int b) { return ceil_div(a, b) * b; }

}  // namespace

GemmPlan plan_gemm(int M, int N, int Kd, int epi, int elem_bytes, int num_sms, bool cluster) {
    GemmPlan g{};
    const int bk = kRowBytes / elem_bytes;
    g.kb_total = ceil_div(Kd, bk);
    if (N <= 256) {
        g.n_tiles = 1;
        g.bn = round_up(N < 1 ? 1 : N, 16);
    } else {
        g.n_tiles = ceil_div(N, 256);
        g.bn = round_up(ceil_div(N, g.n_tiles), 16);
    }
    const int rows_per_tile = epi == EPI_SWIGLU ? 64 : kBM;
    g.m_tiles = ceil_div(M, rows_per_tile);
    if ((epi == EPI_RESID || epi == EPI_QKV) && cluster && N > 256) {
        // O, down and QKV have few weight tiles (16 and 40 at the Qwen
        // shape): narrower token tiles, down to 128 rows, when that lets the
        // tiles fill one wave of SMs
        const int n_fill = num_sms / g.m_tiles;
        if (n_fill > g.n_tiles) {
            const int bn2 = round_up(ceil_div(N, n_fill), 16);
            if (bn2 >= 128) {
                g.bn = bn2;
                g.n_tiles = ceil_div(N, bn2);
            }
        }
    }
    g.tiles = g.m_tiles * g.n_tiles;
    // shared-memory ring: ~100 KB (two CTAs per SM, so the next kernel's CTAs
    // can start their weight loads beside this one) for token tiles up to
    // 128 rows; ~190 KB above that (at 96 rows the small ring measured 17%
    // faster per step, at 176 rows its two stages were much slower)
    const size_t stage = kABytes + static_cast<size_t>(g.bn) * kRowBytes;
    const size_t budget = g.bn <= 128 ? 100 * 1024 : 190 * 1024;
    int st = static_cast<int>(budget / stage);
    g.stages = st < 2 ? 2 : (st > 8 ? 8 : st);
    g.smem_bytes = gemm_smem_bytes(g.stages, g.bn, (epi == EPI_QKV || epi == EPI_SWIGLU) ? inv_slots(N) : 0);
    const int ctas_per_sm = g.smem_bytes <= 113 * 1024 ? 2 : 1;
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
    return g;
}

int gemm_store_kernels_load() {
    cudaFuncAttributes fa;
    PE_CUDA_TRY(cudaFuncGetAttributes(&fa, k_gemm<__nv_bfloat16, EPI_STORE>));
    PE_CUDA_TRY(cudaFuncGetAttributes(&fa, k_gemm<float, EPI_STORE>));
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
    p.cluster = plan.cluster ? 1 : 0;
    p.persistent = plan.persistent ? 1 : 0;
    if (dtype == PE_DTYPE_BF16) return launch_dispatch<__nv_bfloat16>(epi, A, A2, B, plan, p, stream, pdl);
    return launch_dispatch<float>(epi, A, A2, B, plan, p, stream, pdl);
}

}  // namespace pe
