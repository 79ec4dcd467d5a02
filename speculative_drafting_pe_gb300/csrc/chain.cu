// Persistent layer chain: the O projection, gate/up, down and the next
// layer's QKV (or the LM head) of one draft pass in ONE cooperative launch.
//
// At a handful of token rows every one of these GEMMs streams its weights
// from HBM once and does little else, so launched one by one each pays a
// ramp-up and a drain in which HBM idles. Here one CTA per SM walks all the
// phases: a producer warp streams the weight k-blocks of every phase back to
// back into a deep shared-memory ring (weights depend on nothing), while a
// second producer loads a phase's activations once the previous phase is
// complete. The ring's depth of the next phase's weights streams from HBM
// while a phase finishes.
//
// Work split: the k-block units (tile-major) of a phase are divided evenly
// over the CTAs, so every CTA streams the same number of weight bytes. A tile
// whose k-blocks fall to several CTAs is summed by the last of them to
// arrive, in CTA order (the result does not depend on arrival order). The CTA that
// finishes a tile applies the fused epilogue (QKV + RoPE + paged KV write,
// residual + folded RMSNorm outputs, SwiGLU, argmax) and counts the tile on
// the phase's completion counter, which the next phase waits for.
//
// Roles (224 threads): warp 0 weight producer, warp 1 TMEM allocation and
// tcgen05.mma issue (two accumulators, so a tile's epilogue overlaps the next
// tile's k-loop), warps 2..5 epilogue, warp 6 activation producer.
//
// All CTAs must be resident at once (phases wait for other CTAs), hence the
// cooperative launch. Every wait is bounded: a wait that gives up sets
// PE_DEVERR_CHAIN_TIMEOUT, and the other CTAs see that bit and stop.
#include "gemm_epi.cuh"

namespace pe {
namespace {

constexpr int kChainThreads = 224;
constexpr int kWarpA = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpB = 6;

__host__ __device__ inline size_t chain_smem_bytes(int stages, int bn) {
    size_t off = static_cast<size_t>(stages) * (kABytes + static_cast<size_t>(bn) * kRowBytes);
    off += static_cast<size_t>(2 * stages + 4) * 8;   // full, empty, tfull[2], tempty[2]
    off += 16;                                        // TMEM base, abort flag, last-arriver flag
    off = (off + 15) & ~static_cast<size_t>(15);
    off += static_cast<size_t>(kChunk) * kPitch * 4;  // epilogue staging / folded-norm partial slots
    off += static_cast<size_t>(2) * kMaxChainBn * 4;  // folded-norm column scales
    return off + 1024;                                // base alignment slack
}

// The CTA whose share of the phase's U units holds unit x (shares are
// [c * U / G, (c + 1) * U / G)).
__host__ __device__ inline int chain_owner(long long x, int grid, long long units) {
    return static_cast<int>(((x + 1) * grid - 1) / units);
}

// Segments of the tile whose units are [t0, t0 + kb_total): maximal runs of
// units with one owner, in unit order (CTAs whose share is empty own none, so
// the count is not simply the owners' index range). Returns the number of
// segments and, in *ordinal, the index of the segment that starts at unit x0.
__host__ __device__ inline int tile_segments(long long t0, int kb_total, int grid, long long units, long long x0,
                                             int* ordinal) {
    int n = 0;
    const long long end = t0 + kb_total;
    for (long long x = t0; x < end;) {
        const int c = chain_owner(x, grid, units);
        const long long hi_c = (static_cast<long long>(c) + 1) * units / grid;
        if (x == x0 && ordinal != nullptr) *ordinal = n;
        ++n;
        x = hi_c < end ? hi_c : end;
    }
    return n;
}

// Named barrier over the 128 epilogue threads that also ORs a predicate.
__device__ __forceinline__ bool epi_bar_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u)
        : "memory");
    return r != 0;
}

// Bounded wait until *ctr >= target (acquire). Gives up when this CTA or any
// other CTA of the chain already gave up.
__device__ bool wait_counter(const unsigned* ctr, unsigned target, unsigned* err, volatile int* abort) {
    if (ld_acquire_gpu(ctr) >= target) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        __nanosleep(64);
        if (ld_acquire_gpu(ctr) >= target) return true;
        if (*abort) return false;
        if (err != nullptr && (*reinterpret_cast<volatile unsigned*>(err) & PE_DEVERR_CHAIN_TIMEOUT)) {
            *abort = 1;
            return false;
        }
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            if (err != nullptr) atomicOr(err, PE_DEVERR_CHAIN_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
}

// Epilogue of one tile segment. Returns true when this CTA finished the tile
// (it was the tile's only segment, or the last one to arrive).
template <typename T, int EPI>
__device__ bool chain_tile(const ChainParams& P, const ChainPhase& Q, uint32_t t_acc, uint64_t* tempty_acc,
                           float* stile, int* sflag, const float* inv, float xg_g, int tile, int seg, int nseg,
                           int ml, int quad) {
    const GemmParams& gp = Q.gp;
    const int bn = P.bn;
    const uint32_t t_row = t_acc + (static_cast<uint32_t>(quad * 32) << 16);
    if (nseg == 1) {
        for (int c0 = 0; c0 < bn; c0 += kChunk) {
            float v[kChunk];
            tmem_ld16(t_row + c0, v);
            if constexpr (epi_norm_scaled<EPI>()) scale_cols(v, inv, c0, 1, kChunk);
            apply_chunk<T, EPI>(gp, v, ml, tile, ColMap{c0, 1, kChunk, c0}, stile, xg_g);
        }
        tc_fence_before_sync();
        mbar_arrive(tempty_acc);
        finish_norm_partials<EPI>(gp, stile, tile, 0, 1, bn, ml);
        return true;
    }
    // shared tile: park this segment's partial, count the arrival
    // partial tile row-major [128 rows][bn]: each thread's 16 columns are 64 contiguous bytes
    float* mine = P.ws + Q.ws_off + (static_cast<size_t>(tile) * Q.max_segs + seg) * bn * kBM;
    for (int c0 = 0; c0 < bn; c0 += kChunk) {
        float v[kChunk];
        tmem_ld16(t_row + c0, v);
        float4* dst = reinterpret_cast<float4*>(mine + static_cast<size_t>(ml) * bn + c0);
#pragma unroll
        for (int j = 0; j < kChunk / 4; ++j)
            __stcg(dst + j, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
    }
    tc_fence_before_sync();
    mbar_arrive(tempty_acc);   // the accumulator is free for the next segment
    __threadfence();
    named_bar_sync(1, 128);
    if (ml == 0) {
        int* ticket = P.tickets + Q.ticket_off + tile;
        const int old = atomicAdd(ticket, 1);
        const int last = (old == nseg - 1) ? 1 : 0;
        if (last) atomicExch(ticket, 0);
        sflag[0] = last;
    }
    named_bar_sync(1, 128);
    if (!sflag[0]) return false;
    __threadfence();
    const float* base = P.ws + Q.ws_off + static_cast<size_t>(tile) * Q.max_segs * bn * kBM;
    for (int c0 = 0; c0 < bn; c0 += kChunk) {
        float v[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) v[i] = 0.f;
        // loads of up to kGroup segments in flight, added in segment order
        constexpr int kGroup = 2;
        for (int s0 = 0; s0 < nseg; s0 += kGroup) {
            float4 t[kGroup][kChunk / 4];
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                if (s0 + u < nseg) {
                    const float4* src = reinterpret_cast<const float4*>(
                        base + static_cast<size_t>(s0 + u) * bn * kBM + static_cast<size_t>(ml) * bn + c0);
#pragma unroll
                    for (int j = 0; j < kChunk / 4; ++j) t[u][j] = __ldcg(src + j);
                }
            }
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                if (s0 + u < nseg) {
#pragma unroll
                    for (int j = 0; j < kChunk / 4; ++j) {
                        v[4 * j] += t[u][j].x;
                        v[4 * j + 1] += t[u][j].y;
                        v[4 * j + 2] += t[u][j].z;
                        v[4 * j + 3] += t[u][j].w;
                    }
                }
            }
        }
        if constexpr (epi_norm_scaled<EPI>()) scale_cols(v, inv, c0, 1, kChunk);
        apply_chunk<T, EPI>(gp, v, ml, tile, ColMap{c0, 1, kChunk, c0}, stile, xg_g);
    }
    finish_norm_partials<EPI>(gp, stile, tile, 0, 1, bn, ml);
    return true;
}

template <typename T>
__global__ void __launch_bounds__(kChainThreads, 1) k_chain(const __grid_constant__ ChainParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stages = P.stages;
    const int bn = P.bn;
    const uint32_t b_bytes = static_cast<uint32_t>(bn) * kRowBytes;
    uint8_t* sA = smem;
    uint8_t* sB = smem + static_cast<size_t>(stages) * kABytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + static_cast<size_t>(stages) * b_bytes);
    uint64_t* empty = full + stages;
    uint64_t* tfull = empty + stages;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* sflag = reinterpret_cast<int*>(tmem_slot + 2);
    float* stile = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(tmem_slot + 4) + 15) & ~uintptr_t(15));
    float* s_inv = stile + kChunk * kPitch;   // [2][kMaxChainBn]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = static_cast<int>(gridDim.x);
    const int cta = static_cast<int>(blockIdx.x);
    const uint32_t acc_cols = tmem_cols_for(bn);
    const uint32_t tmem_cols = 2 * acc_cols;
    constexpr int kBK = kRowBytes / static_cast<int>(sizeof(T));

    if (warp == kWarpA && lane == 0) {
        for (int p = 0; p < P.nphases; ++p) {
            tma_prefetch_desc(&P.ph[p].tmA);
            if (P.ph[p].epi == EPI_SWIGLU) tma_prefetch_desc(&P.ph[p].tmA2);
            tma_prefetch_desc(&P.ph[p].tmB);
        }
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 2);    // weight producer + activation producer
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        *abort = 0;
        sflag[0] = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    pdl_launch_dependents();

    // This CTA's k-block units of phase p: [lo, hi) of m_tiles * kb_total.
    auto share = [&](int p, long long& lo, long long& hi, long long& U) {
        U = static_cast<long long>(P.ph[p].m_tiles) * P.ph[p].kb_total;
        lo = static_cast<long long>(cta) * U / G;
        hi = static_cast<long long>(cta + 1) * U / G;
    };

    if (warp == kWarpA) {
        // ---- weight producer: every phase's weight k-blocks, back to back
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int p = 0; p < P.nphases && ok; ++p) {
                const ChainPhase& Q = P.ph[p];
                long long lo, hi, U;
                share(p, lo, hi, U);
                for (long long x = lo; x < hi; ++x) {
                    const int tile = static_cast<int>(x / Q.kb_total);
                    const int kb = static_cast<int>(x - static_cast<long long>(tile) * Q.kb_total);
                    if (!mbar_wait_ab(&empty[s], ph ^ 1u, P.err, PE_DEVERR_CHAIN_TIMEOUT, abort)) {
                        *abort = 1;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], kABytes);
                    uint8_t* a_dst = sA + static_cast<size_t>(s) * kABytes;
                    if (Q.epi == EPI_SWIGLU) {
                        tma_load_2d(a_dst, &Q.tmA, &full[s], kb * kBK, tile * 64, pol_w);
                        tma_load_2d(a_dst + kABytes / 2, &Q.tmA2, &full[s], kb * kBK, tile * 64, pol_w);
                    } else {
                        tma_load_2d(a_dst, &Q.tmA, &full[s], kb * kBK, tile * kBM, pol_w);
                    }
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
        __syncwarp();   // reconverge before the CTA-wide barriers below
    } else if (warp == kWarpB) {
        // ---- activation producer: a phase's token tiles once its input is complete
        if (lane == 0) {
            pdl_wait();
            const uint64_t pol_x = l2_policy_evict_last();
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int p = 0; p < P.nphases && ok; ++p) {
                const ChainPhase& Q = P.ph[p];
                long long lo, hi, U;
                share(p, lo, hi, U);
                if (lo >= hi) continue;
                if (p > 0 && !wait_counter(&P.counters[p - 1], static_cast<unsigned>(P.ph[p - 1].m_tiles), P.err, abort)) {
                    ok = false;
                    break;
                }
                fence_proxy_async_global();   // TMA reads below see the generic-proxy writes acquired above
                for (long long x = lo; x < hi; ++x) {
                    const int tile = static_cast<int>(x / Q.kb_total);
                    const int kb = static_cast<int>(x - static_cast<long long>(tile) * Q.kb_total);
                    if (!mbar_wait_ab(&empty[s], ph ^ 1u, P.err, PE_DEVERR_CHAIN_TIMEOUT, abort)) {
                        *abort = 1;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], b_bytes);
                    tma_load_2d(sB + static_cast<size_t>(s) * b_bytes, &Q.tmB, &full[s], kb * kBK, 0, pol_x);
                    if (++s == stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ---- MMA issue: one accumulator per tile segment, alternating
        if (lane == 0) {
            const uint32_t idesc = umma_idesc(UmmaKind<T>::kFmt, kBM, bn);
            int s = 0;
            uint32_t ph = 0;
            int nseg_done = 0;
            bool ok = true;
            for (int p = 0; p < P.nphases && ok; ++p) {
                const ChainPhase& Q = P.ph[p];
                long long lo, hi, U;
                share(p, lo, hi, U);
                for (long long x = lo; x < hi && ok;) {
                    const int tile = static_cast<int>(x / Q.kb_total);
                    const long long tile0 = static_cast<long long>(tile) * Q.kb_total;
                    const long long end = min(hi, tile0 + Q.kb_total);
                    const int acc = nseg_done & 1;
                    const uint32_t use = static_cast<uint32_t>(nseg_done >> 1);
                    if (!mbar_wait_ab(&tempty[acc], (use & 1u) ^ 1u, P.err, PE_DEVERR_CHAIN_TIMEOUT, abort)) {
                        *abort = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * acc_cols;
                    for (long long k = x; k < end; ++k) {
                        if (!mbar_wait_ab(&full[s], ph, P.err, PE_DEVERR_CHAIN_TIMEOUT, abort)) {
                            *abort = 1;
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t a_addr = smem_u32(sA + static_cast<size_t>(s) * kABytes);
                        const uint32_t b_addr = smem_u32(sB + static_cast<size_t>(s) * b_bytes);
#pragma unroll
                        for (int kk = 0; kk < kRowBytes / 32; ++kk) {
                            UmmaKind<T>::mma(d_tmem, umma_desc_sw128(a_addr + kk * 32),
                                             umma_desc_sw128(b_addr + kk * 32), idesc,
                                             (k > x || kk > 0) ? 1u : 0u);
                        }
                        umma_commit(&empty[s]);
                        if (++s == stages) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit(&tfull[acc]);
                    ++nseg_done;
                    x = end;
                }
            }
        }
        __syncwarp();
    } else {
        // ---- epilogue warps 2..5: TMEM lane quadrant warp % 4
        const int quad = warp & 3;
        const int ml = quad * 32 + lane;
        pdl_wait();
        int nseg_done = 0;
        bool stop = false;
        for (int p = 0; p < P.nphases && !stop; ++p) {
            const ChainPhase& Q = P.ph[p];
            long long lo, hi, U;
            share(p, lo, hi, U);
            if (lo >= hi) continue;
            if (p > 0) {
                // everything earlier phases wrote (residual, folded-norm sums) is complete
                bool ok = true;
                if (ml == 0)
                    ok = wait_counter(&P.counters[p - 1], static_cast<unsigned>(P.ph[p - 1].m_tiles), P.err, abort);
                if (epi_bar_or(!ok)) {
                    *abort = 1;
                    break;
                }
                (void)ld_acquire_gpu(&P.counters[p - 1]);
            }
            float* inv = nullptr;
            if (Q.epi == EPI_QKV || Q.epi == EPI_SWIGLU) {
                if (Q.gp.ss_in != nullptr) {
                    inv = s_inv + (p & 1) * kMaxChainBn;
                    fold_norm_scales(Q.gp, inv, 0, Q.gp.N, ml);   // published by the barrier below
                }
            }
            for (long long x = lo; x < hi;) {
                const int tile = static_cast<int>(x / Q.kb_total);
                const long long tile0 = static_cast<long long>(tile) * Q.kb_total;
                const long long end = min(hi, tile0 + Q.kb_total);
                int seg = 0;
                const int nseg = tile_segments(tile0, Q.kb_total, G, U, x, &seg);
                float xg_g = 0.f;
                if (Q.epi == EPI_RESID && Q.gp.xg != nullptr) {
                    const int m = tile * kBM + ml;
                    xg_g = m < Q.gp.M ? Elem<T>::to_f(static_cast<const T*>(Q.gp.xg_gain)[m]) : 0.f;
                }
                const int acc = nseg_done & 1;
                const uint32_t use = static_cast<uint32_t>(nseg_done >> 1);
                const bool ok = mbar_wait_ab(&tfull[acc], use & 1u, P.err, PE_DEVERR_CHAIN_TIMEOUT, abort);
                tc_fence_after_sync();
                if (epi_bar_or(!ok || *abort != 0)) {
                    *abort = 1;
                    stop = true;
                    break;
                }
                const uint32_t t_acc = tmem_base + static_cast<uint32_t>(acc) * acc_cols;
                bool fin = false;
                switch (Q.epi) {
                    case EPI_QKV:
                        fin = chain_tile<T, EPI_QKV>(P, Q, t_acc, &tempty[acc], stile, sflag, inv, xg_g, tile, seg,
                                                     nseg, ml, quad);
                        break;
                    case EPI_RESID:
                        fin = chain_tile<T, EPI_RESID>(P, Q, t_acc, &tempty[acc], stile, sflag, inv, xg_g, tile, seg,
                                                       nseg, ml, quad);
                        break;
                    case EPI_SWIGLU:
                        fin = chain_tile<T, EPI_SWIGLU>(P, Q, t_acc, &tempty[acc], stile, sflag, inv, xg_g, tile,
                                                        seg, nseg, ml, quad);
                        break;
                    default:
                        fin = chain_tile<T, EPI_ARGMAX>(P, Q, t_acc, &tempty[acc], stile, sflag, inv, xg_g, tile,
                                                        seg, nseg, ml, quad);
                        break;
                }
                if (fin) {
                    // publish the tile: every thread's stores, then one count
                    __threadfence();
                    named_bar_sync(1, 128);
                    if (ml == 0) {
                        fence_proxy_async_global();
                        red_release_gpu_add(&P.counters[p], 1u);
                    }
                }
                ++nseg_done;
                x = end;
            }
        }
    }

    // ---- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && *abort) {
        // a wait gave up: let bulk copies still in flight land before this
        // CTA's shared memory and TMEM are released
        __nanosleep(100000);
    }
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, tmem_cols);
    }
    if (threadIdx.x == 0) {
        // the last CTA to finish zeroes the counters (and, after a failure,
        // the tickets) for the next launch
        __threadfence();
        const unsigned old = atomicAdd(&P.counters[kMaxChainPhases], 1u);
        if (old == static_cast<unsigned>(G - 1)) {
            for (int p = 0; p < P.nphases; ++p) atomicExch(&P.counters[p], 0u);
            if (P.err != nullptr && (*reinterpret_cast<volatile unsigned*>(P.err) & PE_DEVERR_CHAIN_TIMEOUT)) {
                for (int p = 0; p < P.nphases; ++p)
                    for (int t = 0; t < P.ph[p].m_tiles; ++t) atomicExch(P.tickets + P.ph[p].ticket_off + t, 0);
            }
            __threadfence();
            atomicExch(&P.counters[kMaxChainPhases], 0u);
        }
    }
}

}  // namespace

int chain_max_segs(int m_tiles, int kb_total, int grid) {
    const long long U = static_cast<long long>(m_tiles) * kb_total;
    int best = 1;
    for (int t = 0; t < m_tiles; ++t) {
        const int n = tile_segments(static_cast<long long>(t) * kb_total, kb_total, grid, U, -1, nullptr);
        best = n > best ? n : best;
    }
    return best;
}

ChainPlan chain_plan(int N, const int* m_tiles, const int* kb_total, int nphases, int num_sms, bool* ok) {
    ChainPlan c{};
    *ok = N >= 1 && N <= kMaxChainBn && nphases >= 1 && nphases <= kMaxChainPhases && num_sms >= 1;
    if (!*ok) return c;
    c.bn = (N + 15) / 16 * 16;
    const size_t stage = kABytes + static_cast<size_t>(c.bn) * kRowBytes;
    const size_t ring_budget = 212 * 1024;
    int st = static_cast<int>(ring_budget / stage);
    c.stages = st < 2 ? 2 : (st > 16 ? 16 : st);
    c.smem_bytes = chain_smem_bytes(c.stages, c.bn);
    c.grid = num_sms;
    c.ws_floats = 0;
    c.tickets = 0;
    for (int p = 0; p < nphases; ++p) {
        c.ws_floats += static_cast<size_t>(m_tiles[p]) * chain_max_segs(m_tiles[p], kb_total[p], c.grid) * c.bn * kBM;
        c.tickets += m_tiles[p];
    }
    return c;
}

bool chain_supported(int device) {
    int coop = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device) != cudaSuccess || !coop) return false;
    // the largest plan: the narrowest token tile has the most ring stages
    size_t smem = 0;
    for (int bn = 16; bn <= kMaxChainBn; bn += 16) {
        const int st = static_cast<int>((212 * 1024) / (kABytes + static_cast<size_t>(bn) * kRowBytes));
        const size_t b = chain_smem_bytes(st < 2 ? 2 : (st > 16 ? 16 : st), bn);
        smem = b > smem ? b : smem;
    }
    if (cudaFuncSetAttribute(k_chain<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return false;
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_chain<__nv_bfloat16>, kChainThreads, smem) !=
        cudaSuccess)
        return false;
    return blocks >= 1;
}

int launch_chain(const ChainParams& p, const ChainPlan& plan, cudaStream_t stream, bool pdl) {
    auto kern = k_chain<__nv_bfloat16>;
    PE_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(plan.smem_bytes)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kChainThreads);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    PE_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, p));
    return PE_OK;
}

}  // namespace pe
