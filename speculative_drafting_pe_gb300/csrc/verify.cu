// Fused greedy verification + batch-metadata rebuild + KV rollback.
//
// One warp per request. With the target's argmax tokens g for the K+1
// verified positions (P-EAGLE post, "Solution overview": the target checks
// all K drafts in one pass; greedy decoding keeps the output identical to the
// target's own), the kernel computes in one pass:
//   a     = length of the longest prefix with d == g          (warp ballot)
//   bonus = g[a]
//   kept  = min(a, K-1) + 1 drafter-cache rows stay committed
//   S'    = S + kept,  Q' = Q + a + 1
//   slot_mapping[j] = page_table[(S'+j)/16]*16 + (S'+j)%16,  j < K
//   rollback: slots of entries S' .. S+K-1, then -1
// A request whose length or position is negative or too close to 2^31 - 1,
// whose next K entries exceed its page table, or whose page index is out of
// range gets a per-request status and pass-through metadata.
#include "common.cuh"
#include "internal.h"

namespace pe {
namespace {

constexpr int kWarpsPerBlock = 8;

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    k_verify_rebuild(int B, int K, const int32_t* __restrict__ drafts, const int32_t* __restrict__ target,
                     const int32_t* __restrict__ page_table, int max_pages, int num_pages, int page_size,
                     const int32_t* positions, const int32_t* seq_lens, int32_t* positions_out,
                     int32_t* seq_lens_out, int32_t* __restrict__ accepted, int32_t* __restrict__ bonus,
                     int32_t* __restrict__ emitted, int32_t* __restrict__ slot_mapping,
                     int32_t* __restrict__ rollback, int32_t* __restrict__ status, const int32_t* acc_in,
                     const int32_t* bonus_in) {
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (b >= B) return;
    const unsigned full = 0xffffffffu;

    const int dj = lane < K ? drafts[static_cast<size_t>(b) * K + lane] : 0;
    int a, bon;
    if (acc_in != nullptr) {
        // acceptance decided elsewhere (stochastic acceptance): a and the
        // final token are given
        a = min(max(acc_in[b], 0), K);
        bon = bonus_in[b];
    } else {
        const int gj = lane <= K ? target[static_cast<size_t>(b) * (K + 1) + lane] : 0;
        const unsigned mism = __ballot_sync(full, lane < K && dj != gj);
        a = mism ? (__ffs(mism) - 1) : K;
        bon = __shfl_sync(full, gj, a);
    }

    const int S = seq_lens[b];
    const int Q = positions[b];
    __syncwarp();
    // Lengths and positions must leave room for the next step's K entries and
    // positions in a signed 32-bit integer; with S, Q <= 2^31 - 1 - 2K the
    // sums below cannot overflow.
    const int lim = 0x7FFFFFFF - 2 * K;
    const bool in_range = S >= 0 && Q >= 0 && S <= lim && Q <= lim;
    const int kept = min(a, K - 1) + 1;
    const int S2 = in_range ? S + kept : 0;
    const int Q2 = in_range ? Q + a + 1 : 0;

    int st = PE_REQ_OK;
    if (!in_range) st = PE_REQ_BAD_INPUT;
    else if (static_cast<long long>(S2) + K > static_cast<long long>(max_pages) * page_size) st = PE_REQ_CAPACITY;
    int slot = -1;
    int bad = 0;
    if (st == PE_REQ_OK && lane < K) {
        const int e = S2 + lane;
        const int page = page_table[static_cast<size_t>(b) * max_pages + e / page_size];
        if (page < 0 || page >= num_pages) bad = 1;
        else slot = page * page_size + e % page_size;
    }
    if (__any_sync(full, bad) && st == PE_REQ_OK) st = PE_REQ_BAD_PAGE;
    const bool ok = st == PE_REQ_OK;

    if (lane < K) {
        slot_mapping[static_cast<size_t>(b) * K + lane] = ok ? slot : -1;
        rollback[static_cast<size_t>(b) * K + lane] = (ok && lane < K - kept) ? slot : -1;
    }
    if (emitted != nullptr && lane <= K)
        emitted[static_cast<size_t>(b) * (K + 1) + lane] = lane < a ? dj : (lane == a ? bon : -1);
    if (lane == 0) {
        if (acc_in == nullptr) {
            accepted[b] = a;
            bonus[b] = bon;
        }
        status[b] = st;
        seq_lens_out[b] = ok ? S2 : S;
        positions_out[b] = ok ? Q2 : Q;
    }
}

// The same acceptance with re-fed real rows: the pass just verified wrote
// n_b real rows at entries S..S+n_b-1 and K-1 placeholder rows after them.
// The real rows stay: S' = S + n_b, Q' = Q + n_b, and the next pass re-feeds
// n_b' = a + 1 tokens (the accepted drafts and the bonus). Lane j < n_b'+K-1
// computes the slot of the next pass's entry S'+j (at most 2K of them); lane
// j < K-1 rolls back placeholder entry S+n_b+j.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    k_verify_rebuild_refeed(int B, int K, const int32_t* __restrict__ drafts, const int32_t* __restrict__ target,
                            const int32_t* __restrict__ page_table, int max_pages, int num_pages, int page_size,
                            const int32_t* n_real, const int32_t* positions, const int32_t* seq_lens,
                            int32_t* n_real_out, int32_t* positions_out, int32_t* seq_lens_out,
                            int32_t* __restrict__ accepted, int32_t* __restrict__ bonus,
                            int32_t* __restrict__ emitted, int32_t* __restrict__ slot_mapping,
                            int32_t* __restrict__ rollback, int32_t* __restrict__ status) {
    pdl_launch_dependents();
    pdl_wait();
    const int b = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (b >= B) return;
    const unsigned full = 0xffffffffu;

    const int dj = lane < K ? drafts[static_cast<size_t>(b) * K + lane] : 0;
    const int gj = lane <= K ? target[static_cast<size_t>(b) * (K + 1) + lane] : 0;
    const unsigned mism = __ballot_sync(full, lane < K && dj != gj);
    const int a = mism ? (__ffs(mism) - 1) : K;
    const int bon = __shfl_sync(full, gj, a);

    const int S = seq_lens[b];
    const int Q = positions[b];
    const int n = n_real[b];
    __syncwarp();
    const int lim = 0x7FFFFFFF - 4 * K;
    const bool in_range = S >= 0 && Q >= 0 && S <= lim && Q <= lim && n >= 1 && n <= K + 1;
    const int S2 = in_range ? S + n : 0;
    const int Q2 = in_range ? Q + n : 0;
    const int n2 = a + 1;
    const int rows_next = n2 + K - 1;

    int st = PE_REQ_OK;
    if (!in_range) st = PE_REQ_BAD_INPUT;
    else if (static_cast<long long>(S2) + rows_next > static_cast<long long>(max_pages) * page_size)
        st = PE_REQ_CAPACITY;
    int slot = -1, rb = -1;
    int bad = 0;
    if (st == PE_REQ_OK) {
        if (lane < rows_next) {
            const int e = S2 + lane;
            const int page = page_table[static_cast<size_t>(b) * max_pages + e / page_size];
            if (page < 0 || page >= num_pages) bad = 1;
            else slot = page * page_size + e % page_size;
        }
        if (lane < K - 1) {
            const int e = S + n + lane;
            const int page = page_table[static_cast<size_t>(b) * max_pages + e / page_size];
            if (page < 0 || page >= num_pages) bad = 1;
            else rb = page * page_size + e % page_size;
        }
    }
    if (__any_sync(full, bad) && st == PE_REQ_OK) st = PE_REQ_BAD_PAGE;
    const bool ok = st == PE_REQ_OK;

    if (lane < 2 * K) slot_mapping[static_cast<size_t>(b) * 2 * K + lane] = (ok && lane < rows_next) ? slot : -1;
    if (lane < K) rollback[static_cast<size_t>(b) * K + lane] = (ok && lane < K - 1) ? rb : -1;
    if (emitted != nullptr && lane <= K)
        emitted[static_cast<size_t>(b) * (K + 1) + lane] = lane < a ? dj : (lane == a ? bon : -1);
    if (lane == 0) {
        accepted[b] = a;
        bonus[b] = bon;
        status[b] = st;
        seq_lens_out[b] = ok ? S2 : S;
        positions_out[b] = ok ? Q2 : Q;
        n_real_out[b] = ok ? n2 : n;
    }
}

}  // namespace

int launch_verify_rebuild_refeed(int B, int K, const int32_t* drafts, const int32_t* target,
                                 const int32_t* page_table, int max_pages, int num_pages, int page_size,
                                 const int32_t* n_real, const int32_t* positions, const int32_t* seq_lens,
                                 int32_t* n_real_out, int32_t* positions_out, int32_t* seq_lens_out,
                                 int32_t* accepted, int32_t* bonus, int32_t* emitted, int32_t* slot_mapping,
                                 int32_t* rollback, int32_t* status, cudaStream_t s) {
    const dim3 grid((B + kWarpsPerBlock - 1) / kWarpsPerBlock), block(kWarpsPerBlock * 32);
    PE_CUDA_TRY(launch_ex(k_verify_rebuild_refeed, grid, block, 0, s, false, B, K, drafts, target, page_table,
                          max_pages, num_pages, page_size, n_real, positions, seq_lens, n_real_out, positions_out,
                          seq_lens_out, accepted, bonus, emitted, slot_mapping, rollback, status));
    return PE_OK;
}

int launch_verify_rebuild(int B, int K, const int32_t* drafts, const int32_t* target, const int32_t* page_table,
                          int max_pages, int num_pages, int page_size, const int32_t* positions,
                          const int32_t* seq_lens, int32_t* positions_out, int32_t* seq_lens_out,
                          int32_t* accepted, int32_t* bonus, int32_t* emitted, int32_t* slot_mapping,
                          int32_t* rollback, int32_t* status, cudaStream_t s) {
    const dim3 grid((B + kWarpsPerBlock - 1) / kWarpsPerBlock), block(kWarpsPerBlock * 32);
    PE_CUDA_TRY(launch_ex(k_verify_rebuild, grid, block, 0, s, false, B, K, drafts, target, page_table, max_pages,
                          num_pages, page_size, positions, seq_lens, positions_out, seq_lens_out, accepted, bonus,
                          emitted, slot_mapping, rollback, status, static_cast<const int32_t*>(nullptr),
                          static_cast<const int32_t*>(nullptr)));
    return PE_OK;
}

int launch_rebuild_given_acceptance(int B, int K, const int32_t* drafts, const int32_t* page_table, int max_pages,
                                    int num_pages, int page_size, const int32_t* positions, const int32_t* seq_lens,
                                    int32_t* positions_out, int32_t* seq_lens_out, const int32_t* accepted,
                                    const int32_t* final_tok, int32_t* emitted, int32_t* slot_mapping,
                                    int32_t* rollback, int32_t* status, cudaStream_t s) {
    const dim3 grid((B + kWarpsPerBlock - 1) / kWarpsPerBlock), block(kWarpsPerBlock * 32);
    PE_CUDA_TRY(launch_ex(k_verify_rebuild, grid, block, 0, s, false, B, K, drafts,
                          static_cast<const int32_t*>(nullptr), page_table, max_pages, num_pages, page_size,
                          positions, seq_lens, positions_out, seq_lens_out, static_cast<int32_t*>(nullptr),
                          static_cast<int32_t*>(nullptr), emitted, slot_mapping, rollback, status, accepted,
                          final_tok));
    return PE_OK;
}

}  // namespace pe
