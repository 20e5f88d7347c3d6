// sample_accept.cu -- temperature sampling and stochastic speculative acceptance.
//
// "Inference 抽象と KV キャッシュ" of "Whisper のデコーダー内部": above temperature 0 the
// decoder samples from Categorical(logits / T). "추측 디코딩이란?" of "추측 디코딩으로
// Whisper 추론 속도 2배 향상" names Leviathan et al.'s speculative decoding; its sampling
// form accepts drafted token x_i with probability min(1, p_i(x_i) / q_i(x_i)) (p: the main
// model's distribution, q: the draft's), and at the first rejection n draws the next
// token from max(0, p_n - q_n) normalised; if all k drafts pass, from p_k.
//
//   accept x_i  <=>  r_i * q_i(x_i) < p_i(x_i)          (r_i, u: the caller's uniforms)
//   next        =  the smallest id whose running sum of w exceeds u * sum(w), in id order
//   w = max(0, p_n - q_n) (p_n if that sums to 0), or p_k when n = k
//
// Design: two launches.
//  A. The 2k + 1 rows (k + 1 main-model rows, k draft rows) are cut into 2048-id
//     segments, one 256-thread block each over the whole GPU; a block reduces its
//     segment to (max, sum of 2^(y - max)), y = x * log2(e) / T, into the workspace.
//  B. One thread-block cluster per batch row; CTA c owns the id slice
//     [c * slice, (c + 1) * slice). Every CTA reduces the segment pairs to each row's
//     log-sum-exp (a warp per row) and takes the same acceptance decision (the drafted
//     ids' logits are fetched by one thread each).
//     Then each CTA sums the draw's weights over its slice and stores the sums into every
//     CTA; cluster barrier (after it nothing is read remotely, so CTAs may exit); the
//     prefix over the CTAs names the CTA whose slice holds u * sum(w); that CTA scans its slice
//     (contiguous chunks per thread, a block-wide exclusive scan of the chunk sums) and
//     writes the result.
// fp32 throughout; the random numbers are inputs, so repeated calls give the same bits.
#include <algorithm>
#include <mutex>

#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {
namespace {

constexpr int kSaThreads = 512;
constexpr int kSaWarps = kSaThreads / 32;
constexpr int kSaMaxK = 7;
constexpr int kSaMaxRows = 2 * kSaMaxK + 1;
constexpr int kSaMaxCluster = 16;
constexpr int kSaMinSlice = 2048;  // ids per CTA below which the cluster is not widened

struct SampleParams {
    const float* target;  // [batch, k+1, vocab]
    const float* draft;   // [batch, k, vocab]
    const int32_t* drafts;
    const float* r;
    const float* u;
    int32_t* n_acc;
    int32_t* next;
    int32_t* dev_err;
    float2* ws_ml;        // [batch, 2k+1, segs] (max, sum) per 2048-id segment
    int32_t k, vocab, cluster, slice, segs;
    float c2;  // log2(e) / T
};

struct SampleShared {
    float row_m[kSaMaxRows], row_l[kSaMaxRows];  // each row's, over the whole vocabulary
    float warp_s[kSaWarps][2];
    float all_s[kSaMaxCluster][2];  // every CTA's sums of the draw weights: [0] w, [1]
                                    // the fallback p_n (each CTA writes its pair into all)
    float chunk_pre[kSaWarps];
    int n, use_p, owner, token, last_pos;
    int acc[kSaMaxK], bad[kSaMaxK];
    float t_local;
};

__device__ __forceinline__ void st_cluster_f32(float* local, int rank, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(map_shared(smem_u32(local), (uint32_t)rank)),
                 "f"(v)
                 : "memory");
}
// All threads of all CTAs of the cluster: writes before are visible to reads after.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- kernel A: each row's (max, sum) per 2048-id segment, over the whole GPU ----
constexpr int kStThreads = 256;
constexpr int kStLoads = 8;
constexpr int kSeg = kStThreads * kStLoads;

__device__ __forceinline__ float exp2_or0(float a, float m) {
    return a == -INFINITY ? 0.f : exp2f(a - m);  // 2^(a - m), 0 for an empty term
}
// (m, l) = (m1, l1) + (m2, l2), branch-free (an empty pair has m = -inf, l = 0)
__device__ __forceinline__ void pair_add(float& m, float& l, float m2, float l2) {
    const float M = fmaxf(m, m2);
    l = l * exp2_or0(m, M) + l2 * exp2_or0(m2, M);
    m = M;
}

__global__ void __launch_bounds__(kStThreads) sample_stats_kernel(const SampleParams p) {
    __shared__ float s_m[kStThreads / 32], s_l[kStThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int seg = blockIdx.x, r = blockIdx.y, b = blockIdx.z;
    const int k = p.k;
    pdl_wait();
    const float* row = r <= k ? p.target + ((int64_t)b * (k + 1) + r) * p.vocab
                              : p.draft + ((int64_t)b * k + (r - k - 1)) * p.vocab;
    const int lo = seg * kSeg, hi = min(p.vocab, lo + kSeg);
    float y[kStLoads];
    bool nan = false;
#pragma unroll
    for (int a = 0; a < kStLoads; ++a) {
        const int e = lo + a * kStThreads + tid;
        const float x = __ldcs(row + min(e, hi - 1));
        nan |= e < hi && isnan(x);
        y[a] = (e < hi && !isnan(x)) ? x * p.c2 : -INFINITY;
    }
    float m = y[0];
#pragma unroll
    for (int a = 1; a < kStLoads; ++a) m = fmaxf(m, y[a]);
    float l = 0.f;
#pragma unroll
    for (int a = 0; a < kStLoads; ++a) l += exp2_or0(y[a], m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        pair_add(m, l, __shfl_xor_sync(0xffffffffu, m, off), __shfl_xor_sync(0xffffffffu, l, off));
    if (lane == 0) {
        s_m[warp] = m;
        s_l[warp] = l;
    }
    if (__syncthreads_or(nan) && tid == 0) flag_error(p.dev_err, KVD_ERR_NAN);
    pdl_trigger();
    if (warp == 0) {
        m = lane < kStThreads / 32 ? s_m[lane] : -INFINITY;
        l = lane < kStThreads / 32 ? s_l[lane] : 0.f;
#pragma unroll
        for (int off = 4; off > 0; off >>= 1)
            pair_add(m, l, __shfl_xor_sync(0xffffffffu, m, off), __shfl_xor_sync(0xffffffffu, l, off));
        if (lane == 0) {
            const int64_t slot = ((int64_t)b * (2 * k + 1) + r) * p.segs + seg;
            p.ws_ml[slot] = make_float2(m, l);
        }
    }
}

// ---- kernel B: the decision and the draw, one cluster per batch row ----
template <int R>
__global__ void __launch_bounds__(kSaThreads, 1) sample_accept_kernel(const SampleParams p) {
    __shared__ SampleShared S;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = (int)(blockIdx.x % (unsigned)p.cluster);
    const int b = (int)(blockIdx.x / (unsigned)p.cluster);
    const int k = p.k;
    const int lo = rank * p.slice, hi = min(p.vocab, lo + p.slice);
    auto row_ptr = [&](int r) -> const float* {
        return r <= k ? p.target + ((int64_t)b * (k + 1) + r) * p.vocab
                      : p.draft + ((int64_t)b * k + (r - k - 1)) * p.vocab;
    };
    pdl_wait();

    // ---- every row's log-sum-exp (log2 domain) from kernel A's segment pairs: one warp
    // per row ----
    if (warp < R) {
        const float2* ml = p.ws_ml + ((int64_t)b * R + warp) * p.segs;
        float m = -INFINITY, l = 0.f;
        for (int sg = lane; sg < p.segs; sg += 32) {
            const float2 v = __ldcg(ml + sg);
            pair_add(m, l, v.x, v.y);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            pair_add(m, l, __shfl_xor_sync(0xffffffffu, m, off), __shfl_xor_sync(0xffffffffu, l, off));
        if (lane == 0) {
            S.row_m[warp] = m;
            S.row_l[warp] = l;
        }
    }
    __syncthreads();
    // the drafted ids' probabilities, all fetched at once (thread i: draft i)
    if (tid < k) {
        const int x = p.drafts[b * k + tid];
        const bool ok = x >= 0 && x < p.vocab;
        float pt = 0.f, qd = 0.f;
        if (ok) {
            const float xt = row_ptr(tid)[x], xd = row_ptr(k + 1 + tid)[x];
            const float yt = isnan(xt) ? -INFINITY : xt * p.c2;
            const float yd = isnan(xd) ? -INFINITY : xd * p.c2;
            const int rd = k + 1 + tid;
            pt = S.row_l[tid] > 0.f ? exp2f(yt - S.row_m[tid]) / S.row_l[tid] : 0.f;
            qd = S.row_l[rd] > 0.f ? exp2f(yd - S.row_m[rd]) / S.row_l[rd] : 0.f;
        }
        // accepted iff the id is valid and r * q < p
        S.acc[tid] = ok && p.r[b * k + tid] * qd < pt;
        S.bad[tid] = !ok;
    }
    __syncthreads();
    if (tid == 0) {
        int n = k;
        for (int i = 0; i < k; ++i)
            if (!S.acc[i]) {
                n = i;
                break;
            }
        if (n < k && S.bad[n] && rank == 0) flag_error(p.dev_err, KVD_ERR_BAD_TOKEN);
        S.n = n;
    }
    __syncthreads();

    // ---- 3. the draw: weights w (residual of row n, or p_k) and the fallback p_n ----
    const int n = S.n;
    const bool resid = n < k;
    const float* pt_row = row_ptr(n);
    const float* pd_row = resid ? row_ptr(k + 1 + n) : pt_row;
    const float mt = S.row_m[n], lt = S.row_l[n];
    const float md = resid ? S.row_m[k + 1 + n] : mt, ld = resid ? S.row_l[k + 1 + n] : lt;
    auto wp = [&](float xt, float xd, float& w, float& pw) {
        const float pv = lt > 0.f && !isnan(xt) ? exp2f(xt * p.c2 - mt) / lt : 0.f;
        const float qv = resid && ld > 0.f && !isnan(xd) ? exp2f(xd * p.c2 - md) / ld : 0.f;
        pw = pv;
        w = resid ? fmaxf(pv - qv, 0.f) : pv;
    };
    // contiguous chunks, so a thread's ids are consecutive for the scan below; the
    // chunk is read in groups of G with all loads of a group issued first
    constexpr int G = 8;
    const int len = max(0, hi - lo);
    const int per = (len + kSaThreads - 1) / kSaThreads;
    const int c0 = lo + min(len, tid * per), c1 = lo + min(len, (tid + 1) * per);
    auto load_group = [&](int e0, float (&xt)[G], float (&xd)[G]) {
#pragma unroll
        for (int a = 0; a < G; ++a) {
            const int e = min(e0 + a, c1 - 1);
            xt[a] = pt_row[e];
            xd[a] = resid ? pd_row[e] : 0.f;
        }
    };
    float sw = 0.f, sp = 0.f;
    int lw = -1, lp = -1;  // the chunk's last ids with a positive weight
    auto chunk_pass = [&]() {
        for (int e0 = c0; e0 < c1; e0 += G) {
            float xt[G], xd[G];
            load_group(e0, xt, xd);
#pragma unroll
            for (int a = 0; a < G; ++a) {
                if (e0 + a < c1) {
                    float w, pw;
                    wp(xt[a], xd[a], w, pw);
                    sw += w;
                    sp += pw;
                    if (w > 0.f) lw = e0 + a;
                    if (pw > 0.f) lp = e0 + a;
                }
            }
        }
    };
    if (!resid) {
        // The draw is from p (of row n = k): each slice's sum follows from kernel A's
        // segment pairs (slices are whole segments), so every CTA finds the owner itself:
        // no pass over the logits and no exchange; only the owner reads its slice.
        if (tid < p.cluster) {
            const float2* ml = p.ws_ml + ((int64_t)b * R + n) * p.segs;
            const int s_lo = tid * (p.slice / kSeg);
            const int s_hi = min(p.segs, s_lo + p.slice / kSeg);
            float a = 0.f;
            for (int sg = s_lo; sg < s_hi; ++sg) {
                const float2 v = __ldcg(ml + sg);
                a += v.x == -INFINITY || !(lt > 0.f) ? 0.f : v.y * exp2f(v.x - mt) / lt;
            }
            S.all_s[tid][0] = a;
            S.all_s[tid][1] = a;
        }
        __syncthreads();
    } else {
        chunk_pass();
        float rw = sw, rp = sp;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            rw += __shfl_xor_sync(0xffffffffu, rw, off);
            rp += __shfl_xor_sync(0xffffffffu, rp, off);
        }
        if (lane == 0) {
            S.warp_s[warp][0] = rw;
            S.warp_s[warp][1] = rp;
        }
        __syncthreads();
        if (tid < p.cluster) {
            // this CTA's pair into every CTA (so that no shared memory is read remotely after
            // the barrier, and a CTA may exit as soon as it is done)
            float a = 0.f, c = 0.f;
            for (int w = 0; w < kSaWarps; ++w) {
                a += S.warp_s[w][0];
                c += S.warp_s[w][1];
            }
            if (p.cluster > 1) {
                st_cluster_f32(&S.all_s[rank][0], tid, a);
                st_cluster_f32(&S.all_s[rank][1], tid, c);
            } else {
                S.all_s[0][0] = a;
                S.all_s[0][1] = c;
            }
        }
        if (p.cluster > 1) cluster_sync_all();
        else __syncthreads();
    }
    if (tid == 0) {
        // the CTA whose slice holds u * sum(w): the first whose running sum exceeds it,
        // else the last with a positive sum (rounding), else CTA 0 (no weight at all)
        float tot_w = 0.f;
        for (int c = 0; c < p.cluster; ++c) tot_w += S.all_s[c][0];
        const int use_p = resid && !(tot_w > 0.f);
        float total = 0.f;
        for (int c = 0; c < p.cluster; ++c) total += S.all_s[c][use_p];
        const float t = p.u[b] * total;
        float run = 0.f;
        int owner = -1, last = 0;
        float before = 0.f, before_last = 0.f;
        for (int c = 0; c < p.cluster; ++c) {
            const float s = S.all_s[c][use_p];
            if (s > 0.f) {
                last = c;
                before_last = run;
            }
            if (owner < 0 && run + s > t) {
                owner = c;
                before = run;
            }
            run += s;
        }
        if (owner < 0) {
            owner = last;
            before = before_last;
        }
        S.use_p = use_p;
        S.owner = owner;
        S.t_local = t - before;
        S.token = INT_MAX;
        S.last_pos = -1;
    }
    __syncthreads();
    if (S.owner != rank) return;
    if (!resid) chunk_pass();  // the owner's slice, read now

    // ---- this CTA holds the draw: exclusive scan of the chunk sums, then one chunk ----
    const bool use_p = S.use_p != 0;
    const float mine = use_p ? sp : sw;
    float incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) S.chunk_pre[warp] = incl;
    __syncthreads();
    float base = 0.f;
    for (int w = 0; w < warp; ++w) base += S.chunk_pre[w];
    const float excl = base + incl - mine;
    const float t = S.t_local;
    const int mine_last = use_p ? lp : lw;
    if (excl <= t && t < excl + mine) {
        float run = excl;
        int tok = -1;
        for (int e0 = c0; e0 < c1 && tok < 0; e0 += G) {
            float xt[G], xd[G];
            load_group(e0, xt, xd);
#pragma unroll
            for (int a = 0; a < G; ++a) {
                if (tok < 0 && e0 + a < c1) {
                    float w, pw;
                    wp(xt[a], xd[a], w, pw);
                    run += use_p ? pw : w;
                    if (run > t) tok = e0 + a;
                }
            }
        }
        atomicMin(&S.token, tok >= 0 ? tok : (mine_last >= 0 ? mine_last : INT_MAX));
    }
    // the slice's last id with a positive weight, for a draw lost to rounding
    if (mine_last >= 0) atomicMax(&S.last_pos, mine_last);
    __syncthreads();
    if (tid == 0) {
        const int tok = S.token != INT_MAX ? S.token : (S.last_pos >= 0 ? S.last_pos : lo);
        p.next[b] = tok;
        p.n_acc[b] = n;
    }
}

template <int R>
kvd_status launch_sample(int batch, cudaStream_t st, bool pdl, const SampleParams& p) {
    static std::mutex mu;
    static bool ready[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVD_ERR_CUDA;
    {
        std::lock_guard<std::mutex> g(mu);
        if (!ready[dev]) {
            if (cudaFuncSetAttribute(sample_accept_kernel<R>,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed,
                                     1) != cudaSuccess) {
                cudaGetLastError();
                return KVD_ERR_CUDA;
            }
            ready[dev] = true;
        }
    }
    // the widest cluster (at most the requested one) the device can hold
    SampleParams q = p;
    for (; q.cluster > 1; --q.cluster) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)q.cluster);
        cfg.blockDim = dim3(kSaThreads);
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = (unsigned)q.cluster;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, sample_accept_kernel<R>, &cfg) != cudaSuccess) n = 0;
        cudaGetLastError();
        if (n > 0) break;
    }
    q.slice = ((q.vocab + q.cluster - 1) / q.cluster + kSeg - 1) / kSeg * kSeg;  // whole segments
    q.cluster = (q.vocab + q.slice - 1) / q.slice;
    // A: the rows' segment pairs, over the whole GPU; B: the decision and the draw (a
    // dependent launch when PDL is requested: B waits for A either way)
    if (kvd_status s = launch(sample_stats_kernel, dim3((unsigned)q.segs, (unsigned)R,
                                                        (unsigned)batch),
                              dim3(kStThreads), 0, st, pdl, q))
        return s;
    return launch_ex(sample_accept_kernel<R>, dim3((unsigned)(batch * q.cluster)),
                     dim3(kSaThreads), 0, st, pdl, (unsigned)q.cluster, q);
}

}  // namespace

size_t sample_workspace_bytes(int batch, int k, int vocab) {
    const size_t segs = ((size_t)vocab + kSeg - 1) / kSeg;
    return KVD_WS_COUNTER_BYTES + ((size_t)batch * (2 * k + 1) * segs * 8 + 255) / 256 * 256;
}

}  // namespace kvd

using namespace kvd;

extern "C" kvd_status kvd_sample_accept(const float* target, const float* draft,
                                        const int32_t* drafts, int32_t batch, int32_t k,
                                        int32_t vocab, float temperature, const float* r,
                                        const float* u, int32_t* n_accepted,
                                        int32_t* next_token, void* workspace,
                                        size_t workspace_bytes, uint32_t flags,
                                        int32_t* dev_err, kvd_stream_t stream) {
    if (batch < 0 || vocab <= 0 || k < 0) return KVD_ERR_INVALID_ARG;
    if (k > kSaMaxK) return KVD_ERR_UNSUPPORTED;
    if (!(temperature > 0.f) || !(temperature < INFINITY)) return KVD_ERR_INVALID_ARG;
    if (batch == 0) return KVD_OK;
    if (!target || !u || !n_accepted || !next_token) return KVD_ERR_INVALID_ARG;
    if (k > 0 && (!draft || !drafts || !r)) return KVD_ERR_INVALID_ARG;
    if ((int64_t)batch * kSaMaxCluster > 0x7fffffff || batch > 65535) return KVD_ERR_UNSUPPORTED;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) ||
        workspace_bytes < sample_workspace_bytes(batch, k, vocab))
        return KVD_ERR_WORKSPACE;
    SampleParams p;
    p.ws_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + KVD_WS_COUNTER_BYTES);
    p.segs = (vocab + kSeg - 1) / kSeg;
    p.target = target;
    p.draft = draft;
    p.drafts = drafts;
    p.r = r;
    p.u = u;
    p.n_acc = n_accepted;
    p.next = next_token;
    p.dev_err = dev_err;
    p.k = k;
    p.vocab = vocab;
    p.cluster = std::max(1, std::min(kSaMaxCluster, (vocab + kSaMinSlice - 1) / kSaMinSlice));
    p.slice = ((vocab + p.cluster - 1) / p.cluster + kSeg - 1) / kSeg * kSeg;  // whole segments
    p.cluster = (vocab + p.slice - 1) / p.slice;
    p.c2 = 1.4426950408889634f / temperature;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const bool pdl = (flags & KVD_FLAG_PDL) != 0;
    switch (2 * k + 1) {
    case 1: return launch_sample<1>(batch, st, pdl, p);
    case 3: return launch_sample<3>(batch, st, pdl, p);
    case 5: return launch_sample<5>(batch, st, pdl, p);
    case 7: return launch_sample<7>(batch, st, pdl, p);
    case 9: return launch_sample<9>(batch, st, pdl, p);
    case 11: return launch_sample<11>(batch, st, pdl, p);
    case 13: return launch_sample<13>(batch, st, pdl, p);
    default: return launch_sample<15>(batch, st, pdl, p);
    }
}
