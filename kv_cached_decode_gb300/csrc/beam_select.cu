// beam_select.cu -- logit filters and the beam-search selection step.
//
// "Whisper のデコーダー内部" of readoss.com:
//  * "LogitFilter チェーン": SuppressBlank masks the blank ids and EOT at the first
//    sampling position only; SuppressTokens masks a list of ids at every position
//    (masked logits become -inf before the decoder sees them).
//  * "Inference 抽象と KV キャッシュ" (BeamSearchDecoder.update), per window of `beam`
//    rows: the beam+1 most probable tokens of each row (log-softmax of the filtered
//    logits); every continuation scores cum[row] + logprob; from the best score down,
//    EOT continuations are collected as finished and the others kept until `beam` are
//    kept; the kept continuations' rows are the parents the caches are reordered by.
//
// Design: one thread-block cluster per window. The window's rows are cut into `parts`
// pieces each (beam x parts <= 16 CTAs); a CTA stages its piece of fp32 logits into
// shared memory with one bulk asynchronous copy (plain loads for the few elements
// before the first 16-byte boundary and after the last), writes -inf over the masked
// ids it holds (the id lists are read while the copy is in flight), and reduces the
// piece in two passes of 8-element batches (independent shared-memory loads) to
//   - an online-softmax pair (max, sum of exp(x - max)), and
//   - its beam+1 best (logit, id) pairs: the (beam+1)-th largest per-thread maximum of
//     some warp bounds the answer from below, so only elements at or above the largest
//     such bound are collected and ranked (a handful on real logits); if too many tie
//     at the bound, K rounds of a block-wide "next best" reduction are used instead.
// Ranking uses an order-preserving 32-bit key of the logit, ties to the lower id. The
// CTA's record (20 words) goes to the cluster's first CTA through distributed shared
// memory (st.async completing on its mbarrier, which that CTA waits on with a bound);
// that CTA merges each row's pieces,
// forms the scores and ranks all beam x (beam+1) continuations at once, then selects
// with one prefix count over the ranked EOT flags. Every id and parent is decided by
// exact comparisons of fp32 values. Nothing goes through global memory but the inputs
// and the outputs: no workspace, no ticket.
#include <algorithm>
#include <mutex>

#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelMaxK = KVD_MAX_BEAM + 1;
constexpr int kSelMaxCluster = 16;
constexpr int kSelMinPart = 2048;          // a row is not cut into pieces shorter than this
constexpr int kSelSmemBudget = 200 * 1024;  // dynamic shared memory of one CTA
constexpr int kSelCandCap = kSelThreads;   // candidates ranked in one step
constexpr int kRec = 20;                   // record words: max, sum, 9 keys, 9 ids
constexpr uint32_t kNone = 0xffffffffu;    // id of an empty item (its key is 0)

struct SelectParams {
    const float* logits;
    const float* cum;
    const int32_t* suppress;
    const int32_t* blank;
    int32_t* row_token;
    float* row_logprob;
    int32_t* parent;
    int32_t* token;
    float* new_cum;
    int32_t* n_fin;
    int32_t* fin_parent;
    float* fin_score;
    int32_t* dev_err;
    int32_t beam, vocab, parts, cluster, part_len, stage_len, n_suppress, n_blank, eot,
        first_step;
    uint32_t rec_off, bar_off;  // dynamic shared memory offsets (bytes)
};

// Order-preserving map of a non-NaN float onto uint32 (larger float -> larger key).
// -inf maps to 0x007fffff, so key 0 is below every real element and marks an empty one.
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// (ka, ia) ranks before (kb, ib): larger key, or equal key and lower id
__device__ __forceinline__ bool ranks_before(uint32_t ka, uint32_t ia, uint32_t kb,
                                             uint32_t ib) {
    return ka > kb || (ka == kb && ia < ib);
}

// Online-softmax pair (m, l = sum exp(x - m)); m = -inf means "nothing yet".
__device__ __forceinline__ void ml_combine(float& m, float& l, float m2, float l2) {
    const float M = fmaxf(m, m2);
    if (M == -INFINITY) return;
    l = (m == -INFINITY ? 0.f : l * exp2f((m - M) * kLog2e)) +
        (m2 == -INFINITY ? 0.f : l2 * exp2f((m2 - M) * kLog2e));
    m = M;
}
struct SelectShared {
    uint32_t cand_k[kSelCandCap], cand_i[kSelCandCap];
    uint32_t run_k[kSelMaxK], run_i[kSelMaxK];      // the CTA's best so far
    uint32_t stage_k[kSelMaxK], stage_i[kSelMaxK];  // the current stage's best
    uint32_t warp_k[kSelWarps], warp_i[kSelWarps];
    float warp_l[kSelWarps];
    uint32_t row_k[KVD_MAX_BEAM][kSelMaxK], row_i[KVD_MAX_BEAM][kSelMaxK];
    float score[KVD_MAX_BEAM * kSelMaxK];
    int32_t tok[KVD_MAX_BEAM * kSelMaxK];
    uint8_t order[KVD_MAX_BEAM * kSelMaxK];
    float cum[KVD_MAX_BEAM];
    float run_m, run_l;  // the CTA's online-softmax pair so far
    uint32_t thresh, smax;
    int n_cand;
};

constexpr int kBatch = 8;  // shared-memory elements a thread loads before using any

// The K best (key, id) of the stage's n filtered values buf[shift + e] (ids a + e),
// into S.stage_k/i, best first, when the candidates at or above S.thresh number nc.
// All threads; ends synchronised.
__device__ void rank_candidates(SelectShared& S, const float* buf, int shift, int n, int a,
                                int K, int nc) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (nc <= kSelCandCap) {
        // every candidate counts the candidates ranked before it
        if (tid < nc) {
            const uint32_t mk = S.cand_k[tid], mi = S.cand_i[tid];
            int rk = 0;
#pragma unroll 4
            for (int u = 0; u < nc; ++u) rk += ranks_before(S.cand_k[u], S.cand_i[u], mk, mi);
            if (rk < K) {
                S.stage_k[rk] = mk;
                S.stage_i[rk] = mi;
            }
        }
        __syncthreads();
        return;
    }
    // Many elements tie at the bound: K rounds of "the best element ranked after the
    // last one taken", reduced over the block.
    uint32_t lk = 0xffffffffu, li = 0;
    for (int r = 0; r < K; ++r) {
        uint32_t bk = 0, bi = kNone;
        for (int e = tid; e < n; e += kSelThreads) {
            const uint32_t k = order_key(buf[shift + e]), id = (uint32_t)(a + e);
            if (ranks_before(lk, li, k, id) && ranks_before(k, id, bk, bi)) {
                bk = k;
                bi = id;
            }
        }
        uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
        uint32_t imin = __reduce_min_sync(0xffffffffu, bk == kmax ? bi : kNone);
        if (lane == 0) {
            S.warp_k[warp] = kmax;
            S.warp_i[warp] = imin;
        }
        __syncthreads();
        if (warp == 0) {
            const uint32_t xk = lane < kSelWarps ? S.warp_k[lane] : 0u;
            const uint32_t xi = lane < kSelWarps ? S.warp_i[lane] : kNone;
            kmax = __reduce_max_sync(0xffffffffu, xk);
            imin = __reduce_min_sync(0xffffffffu, xk == kmax ? xi : kNone);
            if (lane == 0) {
                S.stage_k[r] = kmax;
                S.stage_i[r] = imin;
            }
        }
        __syncthreads();
        lk = S.stage_k[r];
        li = S.stage_i[r];
    }
}

__global__ void __launch_bounds__(kSelThreads, 2)
    beam_select_kernel(const __grid_constant__ SelectParams p) {
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ SelectShared S;
    float* buf = reinterpret_cast<float*>(sm);
    float* rec = reinterpret_cast<float*>(sm + p.rec_off);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + p.bar_off);  // [0] load, [1] merge
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = (int)(blockIdx.x % (unsigned)p.cluster);
    const int w = (int)(blockIdx.x / (unsigned)p.cluster);
    const int K = p.beam + 1;
    const int j = rank / p.parts, part = rank % p.parts;
    const int row = w * p.beam + j;
    const int lo = part * p.part_len, hi = min(p.vocab, lo + p.part_len);
    const uint32_t load_bar = smem_u32(&bars[0]), merge_bar = smem_u32(&bars[1]);

    if (tid == 0) {
        mbar_init(load_bar, 1);
        if (rank == 0 && p.cluster > 1) {
            mbar_init(merge_bar, 1);
            // the one arrival; the other CTAs' record bytes complete the phase
            mbar_expect_tx(merge_bar, (uint32_t)((p.cluster - 1) * kRec * 4));
        }
        fence_barrier_init();
        S.thresh = 0;
        S.smax = 0;
        S.n_cand = 0;
        S.run_m = -INFINITY;
        S.run_l = 0.f;
    }
    if (tid < kSelMaxK) {
        S.run_k[tid] = 0;
        S.run_i[tid] = kNone;
    }
    __syncthreads();
    // Cluster instructions only run in a real cluster launch (more than one CTA). The
    // first CTA writes its own record with plain stores.
    if (p.cluster > 1) cluster_arrive_relaxed();  // the first CTA's merge barrier is ready
    pdl_wait();
    if (rank == 0 && tid < p.beam) S.cum[tid] = p.cum ? p.cum[w * p.beam + tid] : 0.f;

    const int n_ids = p.n_suppress + (p.first_step ? p.n_blank + 1 : 0);
    bool saw_nan = false, bad = false, failed = false;
    uint32_t phase = 0;
    for (int a = lo; a < hi; a += p.stage_len) {
        const int n = min(p.stage_len, hi - a);
        const float* src = p.logits + (int64_t)row * p.vocab + a;
        // elements before the first 16-byte boundary, the bulk body, the tail
        const int hd = min(n, (int)(((16u - (reinterpret_cast<uintptr_t>(src) & 15u)) & 15u) >> 2));
        const int body = (n - hd) & ~3;
        const int shift = (4 - hd) & 3;  // buf[shift + hd] is 16-byte aligned
        if (tid == 0 && body > 0) {
            mbar_expect_tx(load_bar, (uint32_t)body * 4);
            bulk_load(smem_u32(buf + shift + hd), src + hd, (uint32_t)body * 4, load_bar);
        }
        if (tid < hd) buf[shift + tid] = __ldcs(src + tid);
        const int tl = n - hd - body;
        if (tid >= 32 && tid < 32 + tl) {
            const int e = hd + body + tid - 32;
            buf[shift + e] = __ldcs(src + e);
        }
        // the masked ids (suppressed always; blank ids and EOT at the first sampling
        // position) are read while the copy is in flight and applied once it has landed
        int mid = -1;
        if (tid < n_ids) {
            mid = tid < p.n_suppress              ? p.suppress[tid]
                  : tid < p.n_suppress + p.n_blank ? p.blank[tid - p.n_suppress]
                                                   : p.eot;
            bad |= mid < 0 || mid >= p.vocab;
        }
        bool ok = true;
        if (body > 0) {
            ok = mbar_wait_bounded(load_bar, phase);
            phase ^= 1;
        }
        if (__syncthreads_or(!ok)) {
            if (tid == 0) flag_error(p.dev_err, KVD_ERR_TIMEOUT);
            if (body > 0) mbar_wait_bounded(load_bar, phase ^ 1);  // copies still in flight
            failed = true;
            break;
        }
        if (mid >= a && mid < a + n) buf[shift + mid - a] = -INFINITY;
        // -inf past the stage's end up to a whole number of batches: the passes below
        // need no bounds checks
        const int npad = (n + kBatch * kSelThreads - 1) / (kBatch * kSelThreads) * (kBatch * kSelThreads);
        for (int e = n + tid; e < npad; e += kSelThreads) buf[shift + e] = -INFINITY;
        for (int i = tid + kSelThreads; i < n_ids; i += kSelThreads) {  // long lists
            const int t = i < p.n_suppress              ? p.suppress[i]
                          : i < p.n_suppress + p.n_blank ? p.blank[i - p.n_suppress]
                                                         : p.eot;
            bad |= t < 0 || t >= p.vocab;
            if (t >= a && t < a + n) buf[shift + t - a] = -INFINITY;
        }
        __syncthreads();
        // pass 1: this thread's largest value (fmaxf skips NaNs; they are noted)
        float tmax = -INFINITY;
        bool stage_nan = false;
        for (int e0 = tid; e0 < npad; e0 += kBatch * kSelThreads) {
            float f[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) f[u] = buf[shift + e0 + u * kSelThreads];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                stage_nan |= f[u] != f[u];
                tmax = fmaxf(tmax, f[u]);
            }
        }
        const uint32_t tk = order_key(tmax);
        // the stage maximum, and the K-th largest of the warp's per-thread maxima
        // (counted with multiplicity): the warp has at least K elements at or above it,
        // so the stage's K best are too. Padding and masked entries are -inf, the lowest
        // key of a real element, so a bound they set (-inf) admits every element.
        uint32_t v = tk, tw = 0, wmax = 0;
        int acc = 0;
        for (int r = 0; r < K; ++r) {
            const uint32_t kmax = __reduce_max_sync(0xffffffffu, v);
            if (r == 0) wmax = kmax;
            acc += __popc(__ballot_sync(0xffffffffu, v == kmax));
            tw = kmax;
            if (acc >= K || kmax == 0) break;
            if (v == kmax) v = 0;
        }
        if (lane == 0) {
            atomicMax(&S.thresh, tw);
            atomicMax(&S.smax, wmax);
        }
        if (tid < kSelMaxK) {
            S.stage_k[tid] = 0;
            S.stage_i[tid] = kNone;
        }
        if (__syncthreads_or(stage_nan)) {  // rare: NaN -> -inf before the next pass
            saw_nan = true;
            for (int e = tid; e < n; e += kSelThreads)
                if (isnan(buf[shift + e])) buf[shift + e] = -INFINITY;
            __syncthreads();
        }
        // pass 2: sum of exp(x - stage max); mark the candidates at or above the bound
        // (a bit per batch element), then collect the few marked ones
        const uint32_t T = S.thresh;
        const float Tf = T > 0x007fffffu ? key_value(T) : -INFINITY;
        const float M = key_value(S.smax);
        const float Mr = M == -INFINITY ? 0.f : M;  // all -inf: nothing to sum
        float l = 0.f;
        for (int e0 = tid; e0 < npad; e0 += kBatch * kSelThreads) {
            float f[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) f[u] = buf[shift + e0 + u * kSelThreads];
            uint32_t marks = 0;
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                l += __expf(f[u] - Mr);  // x - max first: exact near the max
                marks |= f[u] >= Tf ? 1u << u : 0u;
            }
            while (marks) {  // a handful per CTA
                const int u = __ffs(marks) - 1;
                marks &= marks - 1;
                const int e = e0 + u * kSelThreads;
                if (e < n) {
                    const uint32_t k = order_key(buf[shift + e]);
                    if (k >= T) {
                        const int slot = atomicAdd(&S.n_cand, 1);
                        if (slot < kSelCandCap) {
                            S.cand_k[slot] = k;
                            S.cand_i[slot] = (uint32_t)(a + e);
                        }
                    }
                }
            }
        }
        if (M == -INFINITY) l = 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane == 0) S.warp_l[warp] = l;
        __syncthreads();
        if (tid == 0) {
            // fold the stage's (max, sum) into the CTA's
            float L = 0.f;
            for (int i = 0; i < kSelWarps; ++i) L += S.warp_l[i];
            float m = S.run_m, rl = S.run_l;
            ml_combine(m, rl, M, L);
            S.run_m = m;
            S.run_l = rl;
        }
        rank_candidates(S, buf, shift, n, a, K, S.n_cand);
        if (p.stage_len >= p.part_len) {
            if (tid < K) {
                S.run_k[tid] = S.stage_k[tid];
                S.run_i[tid] = S.stage_i[tid];
            }
        } else {
            // merge two sorted lists: each item's place is its index plus the number of
            // items of the other list ranked before it
            int place = kSelMaxK;
            uint32_t ik = 0, ii = kNone;
            if (tid < K || (tid >= 32 && tid < 32 + K)) {
                const bool st = tid < K;
                const int x = st ? tid : tid - 32;
                ik = st ? S.stage_k[x] : S.run_k[x];
                ii = st ? S.stage_i[x] : S.run_i[x];
                place = x;
                for (int y = 0; y < K; ++y) {
                    const uint32_t ok2 = st ? S.run_k[y] : S.stage_k[y];
                    const uint32_t oi2 = st ? S.run_i[y] : S.stage_i[y];
                    place += ranks_before(ok2, oi2, ik, ii);
                }
            }
            __syncthreads();
            if (place < K) {
                S.cand_k[place] = ik;
                S.cand_i[place] = ii;
            }
            __syncthreads();
            if (tid < K) {
                S.run_k[tid] = S.cand_k[tid];
                S.run_i[tid] = S.cand_i[tid];
            }
        }
        if (tid == 0) {
            S.thresh = 0;
            S.smax = 0;
            S.n_cand = 0;
            fence_proxy_async();  // generic accesses to buf before the next bulk copy
        }
        __syncthreads();
    }
    if (__syncthreads_or(saw_nan) && tid == 0) flag_error(p.dev_err, KVD_ERR_NAN);
    if (__syncthreads_or(bad && blockIdx.x == 0) && tid == 0)
        flag_error(p.dev_err, KVD_ERR_BAD_TOKEN);

    // ---- the CTA's record to the cluster's first CTA ----
    if (p.cluster > 1) cluster_wait();  // the first CTA's merge barrier is initialised
    if (!failed && tid < kRec / 4) {
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int x = 4 * tid + q;  // word x of the record
            v[q] = x == 0 ? S.run_m
                   : x == 1 ? S.run_l
                   : x < 2 + kSelMaxK ? __uint_as_float(x - 2 < K ? S.run_k[x - 2] : 0u)
                                      : __uint_as_float(x - 11 < K ? S.run_i[x - 11] : kNone);
        }
        if (rank != 0) {
            const uint32_t dst = map_shared(smem_u32(rec + rank * kRec + 4 * tid), 0);
            st_async_v4(dst, make_float4(v[0], v[1], v[2], v[3]), map_shared(merge_bar, 0));
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) rec[4 * tid + q] = v[q];
        }
    }
    pdl_trigger();
    if (rank != 0) return;

    // ---- the first CTA: merge each row's pieces, score, rank, select ----
    const bool ok = tid >= 32 || p.cluster == 1 || mbar_wait_bounded_cluster(merge_bar, 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) flag_error(p.dev_err, KVD_ERR_TIMEOUT);
        return;
    }
    if (failed) return;
    if (warp < p.beam) {
        const int rj = warp, r = w * p.beam + rj, n_it = p.parts * K;
        const float* rr = rec + rj * p.parts * kRec;  // the row's pieces
        // log-sum-exp over the pieces: the largest max, then the rescaled sums
        const float pm = lane < p.parts ? rr[lane * kRec] : -INFINITY;
        const float pl = lane < p.parts ? rr[lane * kRec + 1] : 0.f;
        const float Mx = key_value(__reduce_max_sync(0xffffffffu, order_key(pm)));
        float L = pm == -INFINITY ? 0.f : pl * exp2f((pm - Mx) * kLog2e);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        const int ps = lane / K, pk = lane % K;
        const uint32_t ik = lane < n_it ? __float_as_uint(rr[ps * kRec + 2 + pk]) : 0u;
        const uint32_t ii = lane < n_it ? __float_as_uint(rr[ps * kRec + 11 + pk]) : kNone;
        int rk = 0;
#pragma unroll 4
        for (int u = 0; u < n_it; ++u)
            rk += ranks_before(__shfl_sync(0xffffffffu, ik, u), __shfl_sync(0xffffffffu, ii, u),
                               ik, ii);
        if (lane < n_it && rk < K) {
            S.row_k[rj][rk] = ik;
            S.row_i[rj][rk] = ii;
        }
        __syncwarp();
        if (lane < K) {
            const uint32_t kk = S.row_k[rj][lane], id = S.row_i[rj][lane];
            const float lp = Mx == -INFINITY ? -INFINITY : key_value(kk) - (Mx + logf(L));
            float c = S.cum[rj];
            if (isnan(c)) {
                flag_error(p.dev_err, KVD_ERR_NAN);
                c = -INFINITY;
            }
            if (p.row_token) p.row_token[(int64_t)r * K + lane] = (int32_t)id;
            if (p.row_logprob) p.row_logprob[(int64_t)r * K + lane] = lp;
            S.score[rj * K + lane] = c + lp;
            S.tok[rj * K + lane] = (int32_t)id;
        }
    }
    __syncthreads();
    if (!p.parent || warp != 0) return;
    // rank the beam x K continuations: higher score first, then lower index (row, rank)
    const int n = p.beam * K;
    int pos[3];
    float sc[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        pos[i] = 0;
        sc[i] = lane + 32 * i < n ? S.score[lane + 32 * i] : 0.f;
    }
#pragma unroll 8
    for (int u = 0; u < n; ++u) {
        const float su = S.score[u];
#pragma unroll
        for (int i = 0; i < 3; ++i) pos[i] += su > sc[i] || (su == sc[i] && u < lane + 32 * i);
    }
#pragma unroll
    for (int i = 0; i < 3; ++i)
        if (lane + 32 * i < n) S.order[pos[i]] = (uint8_t)(lane + 32 * i);
    __syncwarp();
    // walk the ranked list: position q is kept (non-EOT) or finished (EOT) while fewer
    // than `beam` non-EOT continuations rank before it
    const int out0 = w * p.beam;
    int live_before = 0, n_fin = 0;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const int q = lane + 32 * i;
        const bool valid = q < n;
        const int c = valid ? S.order[q] : 0;
        const bool live = valid && S.tok[c] != p.eot;
        const uint32_t bal = __ballot_sync(0xffffffffu, live);
        const int before = live_before + __popc(bal & ((1u << lane) - 1u));
        const bool take = valid && before < p.beam;
        if (take && live) {
            p.parent[out0 + before] = out0 + c / K;
            p.token[out0 + before] = S.tok[c];
            p.new_cum[out0 + before] = S.score[c];
        } else if (take) {
            p.fin_parent[out0 + q - before] = out0 + c / K;
            p.fin_score[out0 + q - before] = S.score[c];
        }
        n_fin += __popc(__ballot_sync(0xffffffffu, take && !live));
        live_before += __popc(bal);
    }
    if (lane == 0) p.n_fin[w] = n_fin;
    if (lane >= n_fin && lane < p.beam) {
        p.fin_parent[out0 + lane] = -1;
        p.fin_score[out0 + lane] = -INFINITY;
    }
}

struct SelectPlan {
    int parts, cluster, part_len, stage_len;
    uint32_t rec_off, bar_off, smem;
};

SelectPlan plan_for_parts(int beam, int vocab, int parts) {
    SelectPlan P;
    P.parts = parts;
    P.cluster = beam * parts;
    P.part_len = ((vocab + parts - 1) / parts + 3) & ~3;
    const uint32_t rec_bytes = (uint32_t)(P.cluster * kRec * 4);
    // buf: the stage, 4 floats of alignment slack, up to one batch round of padding
    const int pad = kBatch * kSelThreads;
    const int stage_cap = ((kSelSmemBudget - (int)rec_bytes - 16) / 4 - 4 - pad) & ~3;
    P.stage_len = std::min(P.part_len, stage_cap);
    P.rec_off = (uint32_t)(((P.stage_len + 4 + pad) * 4 + 15) & ~15);
    P.bar_off = P.rec_off + rec_bytes;
    P.smem = P.bar_off + 16;
    return P;
}

// The kernel's attributes, set once per device: dynamic shared memory up to the budget
// and clusters of up to 16 CTAs. False if the device refuses them.
bool prepare_select(int dev) {
    static std::mutex mu;
    static int state[64];  // 0 unknown, 1 ready, 2 refused
    if (dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> g(mu);
    if (state[dev] == 0) {
        const bool a = cudaFuncSetAttribute(beam_select_kernel,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            kSelSmemBudget + 1024) == cudaSuccess;
        const bool b = cudaFuncSetAttribute(beam_select_kernel,
                                            cudaFuncAttributeNonPortableClusterSizeAllowed,
                                            1) == cudaSuccess;
        cudaGetLastError();
        state[dev] = a && b ? 1 : 2;
    }
    return state[dev] == 1;
}

// The most pieces per row (at most 16 / beam, none shorter than kSelMinPart) whose
// cluster the device can hold; cached per (device, beam, vocab).
bool choose_select_plan(int dev, int beam, int vocab, SelectPlan& out) {
    static std::mutex mu;
    struct Entry {
        int dev, beam, vocab;
        SelectPlan plan;
    };
    static Entry cache[64];
    static int n_cache = 0;
    {
        std::lock_guard<std::mutex> g(mu);
        for (int i = 0; i < n_cache; ++i)
            if (cache[i].dev == dev && cache[i].beam == beam && cache[i].vocab == vocab) {
                out = cache[i].plan;
                return true;
            }
    }
    int parts = std::max(1, std::min(kSelMaxCluster / beam, (vocab + kSelMinPart - 1) / kSelMinPart));
    for (; parts >= 1; --parts) {
        const SelectPlan P = plan_for_parts(beam, vocab, parts);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)P.cluster);
        cfg.blockDim = dim3(kSelThreads);
        cfg.dynamicSmemBytes = P.smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = (unsigned)P.cluster;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, beam_select_kernel, &cfg) != cudaSuccess) n = 0;
        cudaGetLastError();
        if (n > 0) {
            out = P;
            std::lock_guard<std::mutex> g(mu);
            if (n_cache < 64) cache[n_cache++] = {dev, beam, vocab, P};
            return true;
        }
    }
    return false;
}

}  // namespace
}  // namespace kvd

using namespace kvd;

extern "C" kvd_status kvd_beam_select(const float* logits, int32_t windows, int32_t beam,
                                      int32_t vocab, const float* cum,
                                      const int32_t* suppress, int32_t n_suppress,
                                      const int32_t* blank, int32_t n_blank, int32_t eot,
                                      int32_t first_step, int32_t* row_token,
                                      float* row_logprob, int32_t* parent, int32_t* token,
                                      float* new_cum, int32_t* n_finished,
                                      int32_t* fin_parent, float* fin_score, uint32_t flags,
                                      int32_t* dev_err, kvd_stream_t stream) {
    if (windows < 0 || n_suppress < 0 || n_blank < 0) return KVD_ERR_INVALID_ARG;
    if (windows == 0) return KVD_OK;
    if (beam < 1 || beam > KVD_MAX_BEAM) return KVD_ERR_UNSUPPORTED;
    if (vocab <= beam || eot < 0 || eot >= vocab) return KVD_ERR_INVALID_ARG;
    if (vocab > KVD_MAX_VOCAB || windows > (1 << 24)) return KVD_ERR_UNSUPPORTED;
    if (!logits || (reinterpret_cast<uintptr_t>(logits) & 3) || (n_suppress && !suppress) ||
        (first_step && n_blank && !blank))
        return KVD_ERR_INVALID_ARG;
    const bool walk = parent != nullptr;
    if (walk && (!token || !new_cum || !n_finished || !fin_parent || !fin_score))
        return KVD_ERR_INVALID_ARG;
    if (!walk && !row_token && !row_logprob) return KVD_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || !prepare_select(dev)) return KVD_ERR_CUDA;
    SelectPlan P;
    if (!choose_select_plan(dev, beam, vocab, P)) return KVD_ERR_UNSUPPORTED;
    SelectParams p;
    p.logits = logits;
    p.cum = cum;
    p.suppress = suppress;
    p.blank = blank;
    p.row_token = row_token;
    p.row_logprob = row_logprob;
    p.parent = parent;
    p.token = token;
    p.new_cum = new_cum;
    p.n_fin = n_finished;
    p.fin_parent = fin_parent;
    p.fin_score = fin_score;
    p.dev_err = dev_err;
    p.beam = beam;
    p.vocab = vocab;
    p.parts = P.parts;
    p.cluster = P.cluster;
    p.part_len = P.part_len;
    p.stage_len = P.stage_len;
    p.n_suppress = n_suppress;
    p.n_blank = first_step ? n_blank : 0;
    p.eot = eot;
    p.first_step = first_step ? 1 : 0;
    p.rec_off = P.rec_off;
    p.bar_off = P.bar_off;
    return launch_ex(beam_select_kernel, dim3((unsigned)(windows * P.cluster)), dim3(kSelThreads),
                     P.smem, reinterpret_cast<cudaStream_t>(stream), (flags & KVD_FLAG_PDL) != 0,
                     (unsigned)P.cluster, p);
}
