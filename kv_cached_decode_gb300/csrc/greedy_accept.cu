// greedy_accept.cu -- greedy verification of k draft tokens.
//
// "추측 디코딩이란?" of "추측 디코딩으로 Whisper 추론 속도 2배 향상" and the aitime.ge
// speculative-decoding article: the main model's token at every candidate position is
// compared with the candidate; candidates are kept up to the first mismatch, the
// mismatch is replaced by the main model's token and the rest are dropped. At
// temperature 0 the main model's token is the argmax of its logits (GreedyDecoder in
// "Inference 抽象と KV キャッシュ" of "Whisper のデコーダー内部"). "배치 크기 고려사항":
// rows of a batch advance together only as far as every row matched -> n_min.
//
// Design: the [batch, k+1, vocab] fp32 logits (1.24 MB at k=5, vocab 51865) are read
// once by enough thread blocks to cover the GPU. Each block reduces one segment of one
// row with the rule "NaN first (lowest index among NaNs), then larger value, then lower
// index". That rule is an unsigned order on a 64-bit key -- an order-preserving image of
// the value (NaN above every number, -0 as +0) in the high word, the bitwise complement
// of the index in the low word -- so a block publishes its segment's best as one atomic
// max on its row's key word, then takes a ticket (release); the last block of a batch
// row (acquire) reads the k+1 words and applies the accept rule, and the last batch row
// to finish writes the batch minimum. The max is order-independent, so the integer
// outputs are exact and independent of scheduling. (Batches whose key words do not fit
// in the workspace's counter region reduce per-segment pairs in a second pass instead.)
#include <algorithm>

#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {

struct AcceptParams {
    const float* logits;
    const int32_t* draft;
    int32_t* n_acc;
    int32_t* next;
    int32_t* n_min;
    int32_t* amax;
    float* ws_val;
    int32_t* ws_idx;
    int32_t* ws_n;
    int32_t* cnt;  // [batch] per-row tickets, [batch] = global ticket
    unsigned long long* key;  // [batch, k+1] best keys (zero at rest), or NULL: two passes
    int32_t* dev_err;
    int32_t batch, k, vocab, seg, seg_len;
};

// The 64-bit key of (value v, index i): larger key = preferred by the argmax rule.
__device__ __forceinline__ unsigned long long argmax_key(float v, int i) {
    uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);  // -0 ties with +0
    const uint32_t ord = isnan(v) ? 0xFFFFFFFFu : (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (uint32_t)~(uint32_t)i;
}
__device__ __forceinline__ int key_index(unsigned long long k) {
    return (int)~(uint32_t)(k & 0xFFFFFFFFull);
}
// Warp-wide maximum of a 64-bit key: the high words first, then the low words of the
// lanes that hold the highest one.
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long k) {
    const uint32_t hi = (uint32_t)(k >> 32);
    const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? (uint32_t)k : 0u);
    return ((unsigned long long)mhi << 32) | mlo;
}
__device__ __forceinline__ void red_max_u64(unsigned long long* a, unsigned long long v) {
    asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(a), "l"(v) : "memory");
}
// Ticket with release semantics: this thread's earlier writes (the key) are visible to
// whoever acquires the ticket's later value.
__device__ __forceinline__ int ticket_release(int32_t* a) {
    int old;
    asm volatile("atom.add.release.gpu.global.s32 %0, [%1], 1;" : "=r"(old) : "l"(a) : "memory");
    return old;
}
__device__ __forceinline__ void fence_acquire() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* a) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
    return v;
}

struct Cand {
    float v;
    int i;  // -1 = empty
};

__device__ __forceinline__ bool beats(const Cand& a, const Cand& b) {
    if (a.i < 0) return false;
    if (b.i < 0) return true;
    const bool an = isnan(a.v), bn = isnan(b.v);
    if (an != bn) return an;
    if (!an && a.v != b.v) return a.v > b.v;
    return a.i < b.i;
}

__device__ __forceinline__ Cand warp_best(Cand c) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Cand o;
        o.v = __shfl_xor_sync(0xffffffffu, c.v, off);
        o.i = __shfl_xor_sync(0xffffffffu, c.i, off);
        if (beats(o, c)) c = o;
    }
    return c;
}

constexpr int kAcceptThreads = 256;
constexpr int kAcceptLoads = 8;  // per thread and pass: a 2048-logit segment in one pass

__global__ void __launch_bounds__(kAcceptThreads) greedy_accept_kernel(const AcceptParams p) {
    __shared__ Cand s_warp[kAcceptThreads / 32];
    __shared__ int s_amax[KVD_MAX_QLEN + 1];
    __shared__ int s_flag;
    __shared__ int s_draft[KVD_MAX_QLEN];
    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = blockIdx.x, row = blockIdx.y, b = blockIdx.z;
    const int k1 = p.k + 1;
    // The block that finishes last applies the rule; every block fetches the drafts now,
    // so that block does not wait for them at the end.
    if (warp == kAcceptThreads / 32 - 1 && lane < p.k)
        s_draft[lane] = p.draft[(int64_t)b * p.k + lane];
    const float* x = p.logits + ((int64_t)b * k1 + row) * p.vocab;
    const int lo = s * p.seg_len, hi = min(p.vocab, lo + p.seg_len);

    if (p.key) {
        // ---- one pass: the block's best key goes to its row's word by an atomic max ----
        __shared__ unsigned long long s_key[kAcceptThreads / 32];
        unsigned long long best = 0ull;  // below every real key
        for (int base = lo; base < hi; base += kAcceptLoads * kAcceptThreads) {
            float v[kAcceptLoads];
#pragma unroll
            for (int u = 0; u < kAcceptLoads; ++u)
                v[u] = __ldcs(x + min(base + u * kAcceptThreads + tid, hi - 1));
#pragma unroll
            for (int u = 0; u < kAcceptLoads; ++u) {
                const int i = base + u * kAcceptThreads + tid;
                const unsigned long long kk = argmax_key(v[u], i);
                if (i < hi && kk > best) best = kk;
            }
        }
        best = warp_max_key(best);
        if (lane == 0) s_key[warp] = best;
        __syncthreads();
        pdl_trigger();
        if (warp != 0) return;
        best = warp_max_key(lane < kAcceptThreads / 32 ? s_key[lane] : 0ull);
        int last = 0;
        if (lane == 0) {
            if ((uint32_t)(best >> 32) == 0xFFFFFFFFu) flag_error(p.dev_err, KVD_ERR_NAN);
            red_max_u64(p.key + (int64_t)b * k1 + row, best);
            last = ticket_release(&p.cnt[b]) == k1 * p.seg - 1;
            if (last) fence_acquire();  // with the ticket read: every block's key is seen
        }
        if (!__shfl_sync(0xffffffffu, last, 0)) return;
        __syncwarp();  // orders lane 0's acquire before the other lanes' reads
        // ---- the last block of batch row b: the k+1 argmaxes and the accept rule ----
        int am = 0;
        if (lane < k1) {
            unsigned long long* w = p.key + (int64_t)b * k1 + lane;
            am = key_index(ld_relaxed_u64(w));
            *w = 0ull;  // back to rest for the next call
        }
        int n = p.k;
        bool bad_token = false;
        for (int i = 0; i < p.k; ++i) {
            const int d = s_draft[i];
            const int a = __shfl_sync(0xffffffffu, am, i);
            const bool oob = d < 0 || d >= p.vocab;
            bad_token |= oob;
            if (n == p.k && (oob || d != a)) n = i;
        }
        const int nx = __shfl_sync(0xffffffffu, am, n);
        if (p.amax && lane < k1) p.amax[(int64_t)b * k1 + lane] = am;
        if (lane != 0) return;
        if (bad_token) flag_error(p.dev_err, KVD_ERR_BAD_TOKEN);
        p.n_acc[b] = n;
        p.next[b] = nx;
        p.cnt[b] = 0;
        if (!p.n_min) return;
        p.ws_n[b] = n;
        if (ticket_release(&p.cnt[p.batch]) != p.batch - 1) return;
        fence_acquire();
        int mn = p.k;
        for (int i = 0; i < p.batch; ++i) mn = min(mn, __ldcg(p.ws_n + i));
        *p.n_min = mn;
        p.cnt[p.batch] = 0;
        return;
    }

    // ---- two passes: per-segment pairs in the workspace, reduced by the last block ----
    Cand best = {0.f, -1};
    bool saw_nan = false;
    // All loads of a pass are unconditional (clamped into the segment) and issued before
    // the first compare, so a segment streams in one memory round trip.
    for (int base = lo; base < hi; base += kAcceptLoads * kAcceptThreads) {
        float v[kAcceptLoads];
#pragma unroll
        for (int u = 0; u < kAcceptLoads; ++u)
            v[u] = __ldcs(x + min(base + u * kAcceptThreads + tid, hi - 1));
#pragma unroll
        for (int u = 0; u < kAcceptLoads; ++u) {
            const int i = base + u * kAcceptThreads + tid;
            if (i < hi) {
                saw_nan |= isnan(v[u]);
                const Cand c = {v[u], i};
                if (beats(c, best)) best = c;
            }
        }
    }
    best = warp_best(best);
    if (lane == 0) s_warp[warp] = best;
    if (__syncthreads_or(saw_nan) && tid == 0) flag_error(p.dev_err, KVD_ERR_NAN);
    if (warp == 0) {
        Cand c = lane < kAcceptThreads / 32 ? s_warp[lane] : Cand{0.f, -1};
        c = warp_best(c);
        if (lane == 0) {
            const int64_t slot = ((int64_t)b * k1 + row) * p.seg + s;
            p.ws_val[slot] = c.v;
            p.ws_idx[slot] = c.i;
        }
    }
    pdl_trigger();

    // ---- the last block of batch row b reduces the segments and applies the rule ----
    __threadfence();
    __syncthreads();
    if (tid == 0) s_flag = atomicAdd(&p.cnt[b], 1) == k1 * p.seg - 1;
    __syncthreads();
    if (!s_flag) return;
    __threadfence();
    for (int r = warp; r < k1; r += kAcceptThreads / 32) {
        Cand c = {0.f, -1};
        const int64_t base = ((int64_t)b * k1 + r) * p.seg;
        for (int j = lane; j < p.seg; j += 32) {
            const Cand o = {__ldcg(p.ws_val + base + j), __ldcg(p.ws_idx + base + j)};
            if (beats(o, c)) c = o;
        }
        c = warp_best(c);
        if (lane == 0) s_amax[r] = c.i;
    }
    __syncthreads();
    if (tid != 0) return;
    int n = p.k;
    bool bad_token = false;
    for (int i = 0; i < p.k; ++i) {
        const int d = s_draft[i];
        const bool oob = d < 0 || d >= p.vocab;
        bad_token |= oob;
        if (n == p.k && (oob || d != s_amax[i])) n = i;
    }
    if (bad_token) flag_error(p.dev_err, KVD_ERR_BAD_TOKEN);
    p.n_acc[b] = n;
    p.next[b] = s_amax[n];
    if (p.amax)
        for (int i = 0; i < k1; ++i) p.amax[(int64_t)b * k1 + i] = s_amax[i];
    p.cnt[b] = 0;
    if (!p.n_min) return;
    p.ws_n[b] = n;
    __threadfence();
    if (atomicAdd(&p.cnt[p.batch], 1) != p.batch - 1) return;
    __threadfence();
    int mn = p.k;
    for (int i = 0; i < p.batch; ++i) mn = min(mn, __ldcg(p.ws_n + i));
    *p.n_min = mn;
    p.cnt[p.batch] = 0;
}

namespace {
struct AcceptPlan {
    int seg, seg_len;
    size_t key_off;  // offset of the [batch, k+1] key words in the counter region, 0: none
    size_t val_off, idx_off, n_off, bytes;
};
AcceptPlan plan_accept(int batch, int k, int vocab, int target) {
    AcceptPlan P;
    const int rows = batch * (k + 1);
    const int max_seg = std::max(1, (vocab + 2047) / 2048);
    const int want = std::max(1, (target + rows - 1) / rows);
    int seg = std::min(max_seg, want);
    P.seg_len = ((vocab + seg - 1) / seg + 31) / 32 * 32;
    P.seg = (vocab + P.seg_len - 1) / P.seg_len;
    // The key words sit after the tickets in the counter region (zero at rest) when they
    // fit there.
    const size_t key_off = ((size_t)(batch + 1) * 4 + 7) / 8 * 8;
    P.key_off = key_off + (size_t)rows * 8 <= KVD_WS_COUNTER_BYTES ? key_off : 0;
    const size_t slots = (size_t)rows * P.seg;
    P.val_off = KVD_WS_COUNTER_BYTES;
    P.idx_off = P.val_off + (slots * 4 + 255) / 256 * 256;
    P.n_off = P.idx_off + (slots * 4 + 255) / 256 * 256;
    P.bytes = P.n_off + ((size_t)batch * 4 + 255) / 256 * 256;
    return P;
}
}  // namespace

size_t accept_workspace_bytes(int batch, int k, int vocab, int target) {
    return plan_accept(batch, k, vocab, target).bytes;
}

}  // namespace kvd

using namespace kvd;

extern "C" kvd_status kvd_greedy_accept(const float* logits, int32_t batch, int32_t k,
                                        int32_t vocab, const int32_t* draft,
                                        int32_t* n_accepted, int32_t* next_token,
                                        int32_t* n_min, int32_t* argmax, void* workspace,
                                        size_t workspace_bytes, uint32_t flags,
                                        int32_t* dev_err, kvd_stream_t stream) {
    if (batch < 0 || vocab <= 0) return KVD_ERR_INVALID_ARG;
    if (k < 1 || k > KVD_MAX_QLEN) return KVD_ERR_UNSUPPORTED;
    if (batch == 0) return KVD_OK;
    if (!logits || !draft || !n_accepted || !next_token) return KVD_ERR_INVALID_ARG;
    if ((size_t)(batch + 1) * sizeof(int32_t) > KVD_WS_COUNTER_BYTES || batch > 65535)
        return KVD_ERR_UNSUPPORTED;
    const int nsm = sm_count();
    if (nsm <= 0) return KVD_ERR_CUDA;
    const AcceptPlan P = plan_accept(batch, k, vocab, 4 * nsm);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) || workspace_bytes < P.bytes)
        return KVD_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    AcceptParams p;
    p.logits = logits;
    p.draft = draft;
    p.n_acc = n_accepted;
    p.next = next_token;
    p.n_min = n_min;
    p.amax = argmax;
    p.ws_val = reinterpret_cast<float*>(ws + P.val_off);
    p.ws_idx = reinterpret_cast<int32_t*>(ws + P.idx_off);
    p.ws_n = reinterpret_cast<int32_t*>(ws + P.n_off);
    p.cnt = reinterpret_cast<int32_t*>(ws);
    p.key = P.key_off ? reinterpret_cast<unsigned long long*>(ws + P.key_off) : nullptr;
    p.dev_err = dev_err;
    p.batch = batch;
    p.k = k;
    p.vocab = vocab;
    p.seg = P.seg;
    p.seg_len = P.seg_len;
    return launch(greedy_accept_kernel, dim3(P.seg, k + 1, batch), dim3(kAcceptThreads), 0,
                  reinterpret_cast<cudaStream_t>(stream), (flags & KVD_FLAG_PDL) != 0, p);
}
