// Shared epilogue pieces of the tcgen05 weight-streaming GEMMs (the
// per-GEMM kernel and the persistent layer chain): tile geometry, the fused
// epilogues (store, QKV + RoPE + paged KV write, residual with the folded
// RMSNorm's outputs, SwiGLU, argmax) and the folded-norm helpers.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace pe {
namespace {

constexpr int kBM = 128;
constexpr int kRowBytes = 128;               // one 128-byte swizzle row per tile row
constexpr int kABytes = kBM * kRowBytes;     // 16 KB weight tile per stage
constexpr int kChunk = 16;                   // accumulator columns per tcgen05.ld
constexpr int kPitch = kBM + 4;              // epilogue staging row pitch (floats)
constexpr int kMaxBn = 256;                  // widest token tile
constexpr int kMaxInvAll = 4096;             // folded-norm scales of up to this many token rows stay in smem

// Folded-norm scale slots: every token row of the launch when there are at
// most kMaxInvAll of them, else two tiles' worth (double-buffered per tile).
__host__ __device__ inline int inv_slots(int N) { return N <= kMaxInvAll ? ((N + 3) & ~3) : 2 * kMaxBn; }

__host__ __device__ inline uint32_t tmem_cols_for(int bn) {
    return bn <= 32 ? 32u : (bn <= 64 ? 64u : (bn <= 128 ? 128u : 256u));
}

// ------------------------------------------------------------ epilogues

// The 16 columns of an epilogue chunk: column i is token row n0 + i * cs,
// valid when i < cnt and the row exists. `slot0` numbers the chunk's columns
// within the tile's epilogue (the folded-norm partials are kept per slot).
struct ColMap {
    int n0, cs, cnt, slot0;
    __device__ __forceinline__ int col(int i) const { return n0 + i * cs; }
};

// `bar`: the named barrier (128 threads) of the epilogue warps applying it.
template <typename T, int EPI>
__device__ __forceinline__ void apply_chunk(const GemmParams& p, const float (&v)[kChunk], int ml, int m_tile,
                                            const ColMap& cm, float* stile, float xg_g, int bar = 1) {
    auto col_ok = [&](int i) { return i < cm.cnt && cm.col(i) < p.N; };
    if constexpr (EPI == EPI_STORE || EPI == EPI_RESID) {
        // all loads of the chunk first, then all stores (the destinations of
        // different columns never alias, but the compiler cannot know that)
        const int m = m_tile * kBM + ml;
        float r[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) r[i] = 0.f;
        if (m < p.M) {
            float* __restrict__ base = p.out_f32 + m;
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                if constexpr (EPI == EPI_RESID) {
                    if (col_ok(i)) r[i] = base[static_cast<size_t>(cm.col(i)) * p.ld_out];
                }
            }
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                r[i] += v[i];
                if (col_ok(i)) base[static_cast<size_t>(cm.col(i)) * p.ld_out] = r[i];
            }
        }
        if constexpr (EPI == EPI_RESID) {
            if (p.xg != nullptr) {
                // The next RMSNorm, folded: its consumer reads g * r and
                // scales by 1/rms after the GEMM, so only the per-row sums of
                // squares are needed here (this tile's 128 features).
                const bool mv = m < p.M;
                T* __restrict__ xg = static_cast<T*>(p.xg) + m;
                float q[kChunk];
#pragma unroll
                for (int i = 0; i < kChunk; ++i) {
                    const bool ok = mv && col_ok(i);
                    if (ok) xg[static_cast<size_t>(cm.col(i)) * p.ld_xg] = Elem<T>::from_f(xg_g * r[i]);
                    q[i] = ok ? r[i] * r[i] : 0.f;
                }
                // transpose-reduce over the warp's 32 rows (fixed order), as
                // in the argmax epilogue: lanes 2c, 2c+1 end with column c
                const int lane = ml & 31;
#pragma unroll
                for (int rd = 0; rd < 4; ++rd) {
                    const int half = 8 >> rd;
                    const int bit = 16 >> rd;
                    const bool upper = (lane & bit) != 0;
#pragma unroll
                    for (int j = 0; j < half; ++j) {
                        const float send = upper ? q[j] : q[j + half];
                        const float keep = upper ? q[j + half] : q[j];
                        q[j] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
                    }
                }
                q[0] += __shfl_xor_sync(0xffffffffu, q[0], 1);
                // this warp's partial for chunk column c, in a slot of its own
                // (the four warps' slots are added by finish_norm_partials)
                if ((lane & 1) == 0) stile[(ml >> 5) * kMaxBn + cm.slot0 + ((lane >> 1) & 15)] = q[0];
            }
        }
    } else if constexpr (EPI == EPI_ARGMAX) {
        const int m = m_tile * kBM + ml;
        const bool valid = m < p.M;
        unsigned long long k[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            if (p.logits != nullptr && valid && col_ok(i)) p.logits[static_cast<size_t>(cm.col(i)) * p.ld_logits + m] = v[i];
            k[i] = valid ? argmax_key(v[i], static_cast<uint32_t>(m)) : 0ull;
        }
        // Transpose-reduce over the warp's 32 rows: each round halves the
        // columns a lane keeps and doubles the rows each kept key covers.
        // Afterwards lanes 2c and 2c+1 hold column c's maximum.
        const int lane = ml & 31;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int half = 8 >> r;
            const int bit = 16 >> r;
            const bool upper = (lane & bit) != 0;
#pragma unroll
            for (int j = 0; j < half; ++j) {
                const unsigned long long send = upper ? k[j] : k[j + half];
                const unsigned long long keep = upper ? k[j + half] : k[j];
                const unsigned long long recv = __shfl_xor_sync(0xffffffffu, send, bit);
                k[j] = keep > recv ? keep : recv;
            }
        }
        {
            const unsigned long long recv = __shfl_xor_sync(0xffffffffu, k[0], 1);
            k[0] = k[0] > recv ? k[0] : recv;
        }
        const int c = (lane >> 1) & 15;
        if ((lane & 1) == 0 && col_ok(c) && k[0] != 0ull) atomicMax(p.amax + cm.col(c), k[0]);
    } else if constexpr (EPI == EPI_SWIGLU) {
        // rows 0..63 of the tile are gate rows, 64..127 the matching up rows
        named_bar_sync(bar, 128);
#pragma unroll
        for (int i = 0; i < kChunk; ++i) stile[i * kPitch + ml] = v[i];
        named_bar_sync(bar, 128);
        const int fl = ml & 63;
        const int f = m_tile * 64 + fl;
        const int ibeg = (ml >> 6) * (kChunk / 2);
        float g[kChunk / 2], u[kChunk / 2];
#pragma unroll
        for (int i = 0; i < kChunk / 2; ++i) {
            g[i] = stile[(ibeg + i) * kPitch + fl];
            u[i] = stile[(ibeg + i) * kPitch + fl + 64];
        }
        if (f < p.M) {
            T* __restrict__ out = static_cast<T*>(p.out_act) + f;
#pragma unroll
            for (int i = 0; i < kChunk / 2; ++i)
                if (col_ok(ibeg + i))
                    out[static_cast<size_t>(cm.col(ibeg + i)) * p.ld_act] = Elem<T>::from_f(silu_f(g[i]) * u[i]);
        }
    } else if constexpr (EPI == EPI_QKV) {
        // A 128-row tile holds whole heads of exactly one of q, k, v.
        const int m0 = m_tile * kBM;
        const int m = m0 + ml;
        const int hd = p.hd;
        const int half = hd >> 1;
        const int region = m0 < p.nq_hd ? 0 : (m0 < p.nq_hd + p.nkv * hd ? 1 : 2);
        // loads first: slots of the chunk's rows, RoPE factors, partner values
        int slot[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) slot[i] = (region > 0 && col_ok(i)) ? p.row_slot[cm.col(i)] : -1;
        float outv[kChunk];
        if (region < 2) {
            const int d = ml % hd;
            const bool lo = d < half;
            const int partner = lo ? ml + half : ml - half;
            const int fi = lo ? d : d - half;
            float2 cs[kChunk];
#pragma unroll
            for (int i = 0; i < kChunk; ++i)
                cs[i] = col_ok(i) ? p.rope_cs[static_cast<size_t>(cm.col(i)) * half + fi] : make_float2(1.f, 0.f);
            named_bar_sync(bar, 128);
#pragma unroll
            for (int i = 0; i < kChunk; ++i) stile[i * kPitch + ml] = v[i];
            named_bar_sync(bar, 128);
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                const float y = stile[i * kPitch + partner];
                outv[i] = lo ? (v[i] * cs[i].x - y * cs[i].y) : (v[i] * cs[i].x + y * cs[i].y);
            }
        } else {
#pragma unroll
            for (int i = 0; i < kChunk; ++i) outv[i] = v[i];
        }
        if (m < p.M) {
            if (region == 0) {
                T* __restrict__ q = static_cast<T*>(p.out_act) + m;
#pragma unroll
                for (int i = 0; i < kChunk; ++i)
                    if (col_ok(i)) q[static_cast<size_t>(cm.col(i)) * p.ld_act] = Elem<T>::from_f(outv[i]);
            } else {
                const int r = m - p.nq_hd - (region == 2 ? p.nkv * hd : 0);
                const int kvh = r / hd;
                const int d = r - kvh * hd;
                T* __restrict__ cache = static_cast<T*>(region == 1 ? p.k_cache : p.v_cache);
#pragma unroll
                for (int i = 0; i < kChunk; ++i) {
                    if (slot[i] >= 0) {
                        const size_t page = static_cast<size_t>(slot[i] >> 4);
                        const int off = slot[i] & 15;
                        cache[((page * p.nkv + kvh) * 16 + off) * hd + d] = Elem<T>::from_f(outv[i]);
                    }
                }
            }
        }
    }
}

// Folded RMSNorm, consumer side: inv[j] = 1/rms of token row n0 + j for
// j < count, from the producer's partial sums of squares (row n's partials
// are contiguous, zero-padded to a multiple of 4). Thread t of the nthr
// epilogue threads takes j = t, t + nthr, ...; the loads of four such rows
// are in flight together, and each sum runs in partial order.
__device__ __forceinline__ void fold_norm_scales(const GemmParams& p, float* inv, int n0, int count, int t,
                                                 int nthr = 128) {
    constexpr int kCols = 4;
    constexpr int kVec = 4;   // float4 loads per row per round
    const int nvec = p.ss_ld >> 2;
    for (int j0 = t; j0 < count; j0 += nthr * kCols) {
        float ss[kCols];
#pragma unroll
        for (int c = 0; c < kCols; ++c) ss[c] = 0.f;
        for (int v0 = 0; v0 < nvec; v0 += kVec) {
            float4 x[kCols][kVec];
#pragma unroll
            for (int c = 0; c < kCols; ++c) {
                const int j = j0 + c * nthr;
                const bool ok = j < count && n0 + j < p.N;
                const float4* src = reinterpret_cast<const float4*>(p.ss_in + static_cast<size_t>(n0 + j) * p.ss_ld);
#pragma unroll
                for (int u = 0; u < kVec; ++u)
                    x[c][u] = (ok && v0 + u < nvec) ? __ldcg(src + v0 + u) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int c = 0; c < kCols; ++c) {
#pragma unroll
                for (int u = 0; u < kVec; ++u) {
                    ss[c] += x[c][u].x;
                    ss[c] += x[c][u].y;
                    ss[c] += x[c][u].z;
                    ss[c] += x[c][u].w;
                }
            }
        }
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
            const int j = j0 + c * nthr;
            if (j < count) inv[j] = n0 + j < p.N ? rsqrtf(ss[c] * p.ss_scale + p.ss_eps) : 1.f;
        }
    }
}

// Whether the epilogue scales accumulator columns by the folded norm's
// 1/rms: only QKV and gate/up, whose epilogues are not linear in a column.
// The residual GEMMs produce the norm's inputs and never consume them. The
// LM head's argmax needs no scaling, because 1/rms of a token row is positive
// and so cannot change which vocabulary entry is largest in that row (its
// optional logits output is scaled by a separate kernel).
template <int EPI>
constexpr bool epi_norm_scaled() { return EPI == EPI_QKV || EPI == EPI_SWIGLU; }
template <int EPI>
__device__ __forceinline__ bool norm_scaled(const GemmParams& p) {
    if constexpr (epi_norm_scaled<EPI>()) return p.ss_in != nullptr;
    else return false;
}

// Folded RMSNorm of the B operand: chunk column i (tile column c0 + i * cs,
// valid for i < cnt) times inv[c0 + i * cs].
__device__ __forceinline__ void scale_cols(float (&v)[kChunk], const float* inv, int c0, int cs, int cnt) {
    if (inv == nullptr) return;
#pragma unroll
    for (int i = 0; i < kChunk; ++i)
        if (i < cnt) v[i] *= inv[c0 + i * cs];
}

// Folded RMSNorm, producer side, after all chunks of a tile: the partial sum
// of squares of each of the tile's `count` columns (token row n0 + j * cs) is
// the four warps' slot values added in warp order. With `ngrp` groups of
// epilogue warps taking the 16-column chunks in turn, group `grp` (barrier
// `bar`, its own slots in `stile`) writes the columns of its chunks.
template <int EPI>
__device__ __forceinline__ void finish_norm_partials(const GemmParams& p, const float* stile, int m_tile, int n0,
                                                     int cs, int count, int ml, int bar = 1, int grp = 0,
                                                     int ngrp = 1) {
    if constexpr (EPI == EPI_RESID) {
        if (p.xg == nullptr) return;
        named_bar_sync(bar, 128);
        for (int j = ml; j < count; j += 128) {
            const int n = n0 + j * cs;
            if (n < p.N && (j / kChunk) % ngrp == grp)
                p.ss_out[static_cast<size_t>(n) * p.ss_ld + m_tile] =
                    ((stile[j] + stile[kMaxBn + j]) + stile[2 * kMaxBn + j]) + stile[3 * kMaxBn + j];
        }
    }
}

}  // namespace
}  // namespace pe
