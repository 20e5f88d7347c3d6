// attention.cu -- decode attention (A2/A3), verify-block attention (A5) and the split
// merge (A4) for sm_103a.
//
// What is computed ("KV キャッシュが推論を最適化する方法" step 4 of "nanoVLM における KV
// キャッシュ実装"; "Inference 抽象と KV キャッシュ" of "Whisper のデコーダー内部"; "추측
// 디코딩이란?" of "추측 디코딩으로 Whisper 추론 속도 2배 향상"):
//   out[r,hq,i,:] = sum_{t < limit_i} softmax_t(scale * q[r,hq,i] . K[b,h,t]) V[b,h,t]
// with b = r / rows_per_kv, h = hq / group, limit_i = len (decode, cross) or
// len - qlen + 1 + i (causal verify block whose K/V are already appended).
//
// How (GB300 design):
//  * One thread block handles one (cache row b, KV head h, chunk of positions) and ALL
//    query vectors that read that KV head -- rows_per_kv beam rows x group query heads x
//    qlen tokens -- so every K/V byte is fetched from HBM once per step.
//  * K/V tiles of 64 positions x 64 dims (8 KiB each) are staged into shared memory by
//    TMA (cp.async.bulk.tensor, 128-byte swizzle) through a ring of up to 4 stages whose
//    full-barriers are mbarriers with transaction counts; one thread issues the copies.
//  * Decode (one query token): CUDA cores. Eight lanes share a cache position, each
//    holding 16 bytes (8 dims) of K and V; dot products are finished with three xor
//    shuffles and folded into an online softmax in the exp2 domain.
//  * Verify (a block of up to 16 query vectors): tensor cores. S = Q.K^T and O = P.V
//    run as mma.sync m16n8k16 (fp16/bf16 in, fp32 accumulate) with operands read from
//    the swizzled tiles by ldmatrix (K) and ldmatrix.trans (V).
//  * Long ranges are split over thread blocks; each writes its partial (max, sum, o)
//    to the workspace and the last block to arrive (atomic ticket) merges the splits in
//    fixed order with log-sum-exp weights, so results do not depend on timing.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {

struct AttnParams {
    const void* q;
    void* out;
    const int32_t* lens;
    int32_t fixed_len;
    int32_t capacity;
    int32_t n_q_heads;
    int32_t group;
    int32_t rows_per_kv;
    int32_t qlen;
    int32_t causal;
    int32_t M;
    int32_t msub;
    int32_t nsub;
    int32_t splits;
    int32_t tiles_per_split;
    int32_t stages;
    int32_t box_rows;
    int32_t early;
    int32_t cluster;  // 1: the splits of a unit form one thread-block cluster
    float scale_log2;
    float* ws_part;
    float2* ws_ml;
    int32_t* ws_cnt;
    int32_t* dev_err;
};

// Shared memory: [stages x (K tile, V tile)] [stage barriers] [warp partials]
// [block partial, read by the other CTAs of the cluster] [flag]
struct SmemLayout {
    uint32_t bar_off, red_off, fin_off, misc_off, total;
};
__host__ __device__ inline SmemLayout smem_layout(int stages, int rmax) {
    SmemLayout L;
    L.bar_off = stages * 2 * kTileBytes;
    L.red_off = (L.bar_off + stages * 8 + 15) & ~15u;
    L.fin_off = L.red_off + 4 * rmax * (kHeadDim + 2) * 4;
    L.misc_off = L.fin_off + rmax * (kHeadDim + 2) * 4;
    L.total = L.misc_off + 16 + 1024;  // + slack to align the base to 1024 B
    return L;
}

struct CtaCtx {
    int bk, h, sub, s, m0, mcount, len, t_begin, t_end, n_tiles, unit;
    bool bad;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void setup_ctx(const AttnParams& p, CtaCtx& c) {
    c.s = blockIdx.x;
    c.h = blockIdx.y / p.nsub;
    c.sub = blockIdx.y % p.nsub;
    c.bk = blockIdx.z;
    c.unit = (c.bk * (gridDim.y / p.nsub) + c.h) * p.nsub + c.sub;
    c.m0 = c.sub * p.msub;
    c.mcount = min(p.msub, p.M - c.m0);
    c.len = p.lens ? p.lens[c.bk] : p.fixed_len;
    c.bad = c.len < 0 || c.len > p.capacity;
    c.t_begin = c.s * p.tiles_per_split * kTile;
    c.t_end = c.bad ? c.t_begin : min(c.len, c.t_begin + p.tiles_per_split * kTile);
    c.n_tiles = c.t_end > c.t_begin ? (c.t_end - c.t_begin + kTile - 1) / kTile : 0;
}

// Element offset of query vector m (0 <= m < M) of unit (bk, h) in q / out.
__device__ __forceinline__ int64_t qrow(const AttnParams& p, int bk, int h, int m) {
    const int i = m % p.qlen;
    const int t2 = m / p.qlen;
    const int r = bk * p.rows_per_kv + t2 / p.group;
    const int hq = h * p.group + t2 % p.group;
    return ((int64_t)(r * p.n_q_heads + hq) * p.qlen + i) * kHeadDim;
}

__device__ __forceinline__ void issue_tile(const CUtensorMap* tmk, const CUtensorMap* tmv,
                                           uint8_t* smem, uint64_t* bars, int stage, int pos,
                                           int h, int bk, uint32_t tx) {
    const uint32_t bar = smem_u32(&bars[stage]);
    mbar_expect_tx(bar, tx);
    const uint32_t dk = smem_u32(smem + stage * 2 * kTileBytes);
    tma_load_4d(dk, tmk, bar, 0, pos, h, bk);
    tma_load_4d(dk + kTileBytes, tmv, bar, 0, pos, h, bk);
}

template <typename T>
__device__ __forceinline__ void store_out(const AttnParams& p, const CtaCtx& c, int m, int d,
                                          float v) {
    T* o = static_cast<T*>(p.out) + qrow(p, c.bk, c.h, c.m0 + m) + d;
    *o = Half16<T>::from_f(v);
}

// Combine the four warps' partial states, then
//  * one split: write the output;
//  * splits forming a cluster: publish the block's (max, sum, o) in shared memory and
//    merge through distributed shared memory, the work spread over the cluster's CTAs;
//  * more splits than a cluster holds: publish to the workspace; the last block to
//    arrive (atomic ticket) merges all splits, loading them in parallel.
// Merges run over the splits in index order, so results do not depend on timing.
// red: o [4][RMAX][64], m [4][RMAX], l [4][RMAX]; fin: o [RMAX][64], m [RMAX], l [RMAX].
template <typename T, int RMAX>
__device__ void finish_cta(const AttnParams& p, const CtaCtx& c, float* red, float* fin,
                           int* misc, uint8_t* stage_mem) {
    const float* red_o = red;
    const float* red_m = red + 4 * RMAX * kHeadDim;
    const float* red_l = red_m + 4 * RMAX;
    float* fin_o = fin;
    float* fin_m = fin + RMAX * kHeadDim;
    float* fin_l = fin_m + RMAX;
    const int tid = threadIdx.x;
    const int S = p.splits;
    const size_t base = (size_t)c.unit * S * p.msub;
    const size_t slot0 = base + (size_t)c.s * p.msub;
    for (int idx = tid; idx < c.mcount * kHeadDim; idx += blockDim.x) {
        const int m = idx >> 6, d = idx & 63;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) mx = fmaxf(mx, red_m[w * RMAX + m]);
        const float ref = mx == -INFINITY ? 0.f : mx;
        float l = 0.f, o = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float a = exp2f(red_m[w * RMAX + m] - ref);
            l = fmaf(red_l[w * RMAX + m], a, l);
            o = fmaf(red_o[(w * RMAX + m) * kHeadDim + d], a, o);
        }
        if (S == 1) {
            store_out<T>(p, c, m, d, l > 0.f ? o / l : 0.f);
        } else if (p.cluster) {
            fin_o[m * kHeadDim + d] = o;
            if (d == 0) {
                fin_m[m] = mx;
                fin_l[m] = l;
            }
        } else {
            p.ws_part[(slot0 + m) * kHeadDim + d] = o;
            if (d == 0) p.ws_ml[slot0 + m] = make_float2(mx, l);
        }
    }
    if (S == 1) return;

    if (p.cluster) {
        cluster_sync();  // every split's partial is now visible cluster-wide
        const uint32_t fo = smem_u32(fin_o), fm = smem_u32(fin_m), fl = smem_u32(fin_l);
        for (int it = c.s * blockDim.x + tid; it < c.mcount * kHeadDim; it += S * blockDim.x) {
            const int m = it >> 6, d = it & 63;
            float ms[kMaxClusterSplits];
            float mx = -INFINITY;
#pragma unroll
            for (int r = 0; r < kMaxClusterSplits; ++r) {
                ms[r] = r < S ? ld_dsmem(map_shared(fm + m * 4, r)) : -INFINITY;
                mx = fmaxf(mx, ms[r]);
            }
            const float ref = mx == -INFINITY ? 0.f : mx;
            float l = 0.f, o = 0.f;
#pragma unroll
            for (int r = 0; r < kMaxClusterSplits; ++r) {
                if (r < S) {
                    const float a = exp2f(ms[r] - ref);
                    l = fmaf(ld_dsmem(map_shared(fl + m * 4, r)), a, l);
                    o = fmaf(ld_dsmem(map_shared(fo + (m * kHeadDim + d) * 4, r)), a, o);
                }
            }
            store_out<T>(p, c, m, d, l > 0.f ? o / l : 0.f);
        }
        cluster_sync();  // no CTA leaves while another may still read its shared memory
        return;
    }

    __threadfence();
    __syncthreads();
    if (tid == 0) misc[0] = (atomicAdd(&p.ws_cnt[c.unit], 1) == S - 1) ? 1 : 0;
    __syncthreads();
    if (!misc[0]) return;
    __threadfence();
    // (a) all (max, sum) pairs at once -> normalised weights in shared memory
    // 2 * S * mcount <= 2 * kMaxSplits * RMAX floats fit in the warp-partial area; each
    // query's thread then overwrites its pairs' first field with the normalised weight.
    float2* ml = reinterpret_cast<float2*>(red);
    for (int i = tid; i < S * c.mcount; i += blockDim.x)
        ml[i] = __ldcg(&p.ws_ml[base + (size_t)(i / c.mcount) * p.msub + i % c.mcount]);
    __syncthreads();
    for (int m = tid; m < c.mcount; m += blockDim.x) {
        float mx = -INFINITY;
        for (int s2 = 0; s2 < S; ++s2) mx = fmaxf(mx, ml[s2 * c.mcount + m].x);
        const float ref = mx == -INFINITY ? 0.f : mx;
        float l = 0.f;
        for (int s2 = 0; s2 < S; ++s2)
            l = fmaf(ml[s2 * c.mcount + m].y, exp2f(ml[s2 * c.mcount + m].x - ref), l);
        const float inv = l > 0.f ? 1.f / l : 0.f;
        for (int s2 = 0; s2 < S; ++s2)
            ml[s2 * c.mcount + m].x = exp2f(ml[s2 * c.mcount + m].x - ref) * inv;
    }
    __syncthreads();
    // (b) weighted sum of the partial outputs: float4 items x split groups, all loads
    //     of a thread independent; split groups are combined in a fixed order.
    const int nq4 = c.mcount * (kHeadDim / 4);
    const int groups = max(1, (int)blockDim.x / nq4);
    // groups * nq4 <= max(blockDim.x, nq4) float4s (at most 4 KiB) go to the stage
    // buffers, whose copies have all completed.
    float4* tmp = reinterpret_cast<float4*>(stage_mem);
    for (int item = tid; item < nq4 * groups; item += blockDim.x) {
        const int q4 = item % nq4, g = item / nq4;
        const int m = q4 / (kHeadDim / 4), d4 = q4 % (kHeadDim / 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int s2 = g; s2 < S; s2 += groups) {
            const float ww = ml[s2 * c.mcount + m].x;
            const float4 v = __ldcg(reinterpret_cast<const float4*>(
                p.ws_part + (base + (size_t)s2 * p.msub + m) * kHeadDim) + d4);
            acc.x = fmaf(ww, v.x, acc.x);
            acc.y = fmaf(ww, v.y, acc.y);
            acc.z = fmaf(ww, v.z, acc.z);
            acc.w = fmaf(ww, v.w, acc.w);
        }
        tmp[g * nq4 + q4] = acc;
    }
    __syncthreads();
    for (int q4 = tid; q4 < nq4; q4 += blockDim.x) {
        float4 acc = tmp[q4];
        for (int g = 1; g < groups; ++g) {
            const float4 v = tmp[g * nq4 + q4];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const int m = q4 / (kHeadDim / 4), d = (q4 % (kHeadDim / 4)) * 4;
        store_out<T>(p, c, m, d + 0, acc.x);
        store_out<T>(p, c, m, d + 1, acc.y);
        store_out<T>(p, c, m, d + 2, acc.z);
        store_out<T>(p, c, m, d + 3, acc.w);
    }
    if (tid == 0) p.ws_cnt[c.unit] = 0;
}

// After a timeout the block still has to meet its cluster peers at both merge barriers.
__device__ __forceinline__ void abort_block(const AttnParams& p) {
    if (p.cluster && p.splits > 1) {
        cluster_sync();
        cluster_sync();
    }
}

// Shared prologue: barrier init, first copies, PDL wait. Returns false if the block
// has nothing to do (a bad length: flagged, nothing written).
__device__ __forceinline__ bool prologue(const AttnParams& p, CtaCtx& c, uint8_t* smem,
                                         uint64_t* bars, const CUtensorMap* tmk,
                                         const CUtensorMap* tmv) {
    const int tid = threadIdx.x;
    if (!p.early) pdl_wait();
    setup_ctx(p, c);
    if (c.bad) {
        if (p.early) pdl_wait();
        if (tid == 0 && c.s == 0 && c.h == 0 && c.sub == 0)
            flag_error(p.dev_err, KVD_ERR_LEN_OVERFLOW);
        return false;
    }
    if (tid == 0) {
        for (int j = 0; j < p.stages; ++j) mbar_init(smem_u32(&bars[j]), 1);
        fence_barrier_init();
        prefetch_tensormap(tmk);
        prefetch_tensormap(tmv);
    }
    __syncthreads();
    if (tid == 0) {
        const uint32_t tx = 2u * p.box_rows * kRowBytes;
        const int first = min(p.stages, c.n_tiles);
        for (int j = 0; j < first; ++j)
            issue_tile(tmk, tmv, smem, bars, j, c.t_begin + j * kTile, c.h, c.bk, tx);
    }
    if (p.early) pdl_wait();
    return true;
}

// Wait (bounded) for the copies of stages whose tiles were issued but never consumed,
// so that no copy is still writing shared memory when the block exits after a timeout.
__device__ void drain_after_timeout(const AttnParams& p, const CtaCtx& c, uint64_t* bars,
                                    int next_tile) {
    if (threadIdx.x != 0) return;
    flag_error(p.dev_err, KVD_ERR_TIMEOUT);
    const int last = min(c.n_tiles, next_tile + p.stages);
    for (int j = next_tile; j < last; ++j)
        mbar_wait_bounded(smem_u32(&bars[j % p.stages]), (j / p.stages) & 1);
}

// ---------------------------------------------------------------- decode (SIMT) ----
template <typename T, int MS>
__global__ void __launch_bounds__(128)
    decode_attn_kernel(const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    const SmemLayout L = smem_layout(p.stages, MS);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);
    float* red = reinterpret_cast<float*>(smem + L.red_off);
    float* fin = reinterpret_cast<float*>(smem + L.fin_off);
    int* misc = reinterpret_cast<int*>(smem + L.misc_off);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = lane >> 3, c8 = lane & 7;

    CtaCtx c;
    if (!prologue(p, c, smem, bars, &tmk, &tmv)) return;

    float qf[MS][8];
#pragma unroll
    for (int m = 0; m < MS; ++m) {
        if (m < c.mcount) {
            const uint4 u = *reinterpret_cast<const uint4*>(
                static_cast<const T*>(p.q) + qrow(p, c.bk, c.h, c.m0 + m) + c8 * 8);
            unpack8<T>(u, qf[m]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[m][e] = 0.f;
        }
    }
    float mrun[MS], lrun[MS], acc[MS][8];
#pragma unroll
    for (int m = 0; m < MS; ++m) {
        mrun[m] = -INFINITY;
        lrun[m] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[m][e] = 0.f;
    }

    const uint32_t tx = 2u * p.box_rows * kRowBytes;
    for (int j = 0; j < c.n_tiles; ++j) {
        const int st = j % p.stages;
        const bool ok = mbar_wait_bounded(smem_u32(&bars[st]), (j / p.stages) & 1);
        if (ok) {
            const uint8_t* sK = smem + st * 2 * kTileBytes;
            const uint8_t* sV = sK + kTileBytes;
            const int tile0 = c.t_begin + j * kTile;
            float sc[4][MS];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int row = warp * 16 + grp * 4 + jj;
                const bool valid = tile0 + row < c.t_end;
                const uint4 kr = *reinterpret_cast<const uint4*>(sK + swz(row, c8));
                float kf[8];
                unpack8<T>(kr, kf);
#pragma unroll
                for (int m = 0; m < MS; ++m) {
                    float d = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) d = fmaf(qf[m][e], kf[e], d);
                    d += __shfl_xor_sync(0xffffffffu, d, 1);
                    d += __shfl_xor_sync(0xffffffffu, d, 2);
                    d += __shfl_xor_sync(0xffffffffu, d, 4);
                    sc[jj][m] = valid ? d * p.scale_log2 : -INFINITY;
                }
            }
#pragma unroll
            for (int m = 0; m < MS; ++m) {
                const float mt = fmaxf(fmaxf(sc[0][m], sc[1][m]), fmaxf(sc[2][m], sc[3][m]));
                const float mn = fmaxf(mrun[m], mt);
                const float ref = mn == -INFINITY ? 0.f : mn;
                const float alpha = exp2f(mrun[m] - ref);
                float ls = 0.f;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    sc[jj][m] = exp2f(sc[jj][m] - ref);
                    ls += sc[jj][m];
                }
                lrun[m] = fmaf(lrun[m], alpha, ls);
                mrun[m] = mn;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[m][e] *= alpha;
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int row = warp * 16 + grp * 4 + jj;
                const bool valid = tile0 + row < c.t_end;
                const uint4 vr = *reinterpret_cast<const uint4*>(sV + swz(row, c8));
                float vf[8];
                unpack8<T>(vr, vf);
#pragma unroll
                for (int e = 0; e < 8; ++e) vf[e] = valid ? vf[e] : 0.f;
#pragma unroll
                for (int m = 0; m < MS; ++m)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[m][e] = fmaf(sc[jj][m], vf[e], acc[m][e]);
            }
        }
        if (__syncthreads_or(!ok)) {
            drain_after_timeout(p, c, bars, j);
            abort_block(p);
            return;
        }
        if (tid == 0 && j + p.stages < c.n_tiles) {
            fence_proxy_async();
            issue_tile(&tmk, &tmv, smem, bars, st, c.t_begin + (j + p.stages) * kTile, c.h,
                       c.bk, tx);
        }
    }
    pdl_trigger();

    // Merge the four 8-lane groups of each warp (they saw different positions).
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
        for (int m = 0; m < MS; ++m) {
            const float mo = __shfl_xor_sync(0xffffffffu, mrun[m], off);
            const float lo = __shfl_xor_sync(0xffffffffu, lrun[m], off);
            const float mn = fmaxf(mrun[m], mo);
            const float ref = mn == -INFINITY ? 0.f : mn;
            const float a = exp2f(mrun[m] - ref), b = exp2f(mo - ref);
            lrun[m] = lrun[m] * a + lo * b;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[m][e] = acc[m][e] * a + __shfl_xor_sync(0xffffffffu, acc[m][e], off) * b;
            mrun[m] = mn;
        }
    }
    if (grp == 0) {
        float* red_o = red;
        float* red_m = red + 4 * MS * kHeadDim;
        float* red_l = red_m + 4 * MS;
#pragma unroll
        for (int m = 0; m < MS; ++m) {
#pragma unroll
            for (int e = 0; e < 8; ++e) red_o[(warp * MS + m) * kHeadDim + c8 * 8 + e] = acc[m][e];
            if (c8 == 0) {
                red_m[warp * MS + m] = mrun[m];
                red_l[warp * MS + m] = lrun[m];
            }
        }
    }
    __syncthreads();
    finish_cta<T, MS>(p, c, red, fin, misc, smem);
}

// ---------------------------------------------------------------- verify (MMA) -----
template <typename T>
__global__ void __launch_bounds__(128)
    verify_attn_kernel(const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const AttnParams p) {
    constexpr int RM = 16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    const SmemLayout L = smem_layout(p.stages, RM);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);
    float* red = reinterpret_cast<float*>(smem + L.red_off);
    float* fin = reinterpret_cast<float*>(smem + L.fin_off);
    int* misc = reinterpret_cast<int*>(smem + L.misc_off);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int qr = lane >> 2, qc = (lane & 3) * 2;  // fragment row / column pair
    const int jm = lane >> 3, rr = lane & 7;         // ldmatrix matrix / row

    CtaCtx c;
    if (!prologue(p, c, smem, bars, &tmk, &tmv)) return;

    // Q as m16n8k16 A fragments for the four 16-dim k-steps (rows >= mcount are 0).
    uint32_t qa[4][4];
    const T* qbase = static_cast<const T*>(p.q);
    const bool rowA = qr < c.mcount, rowB = qr + 8 < c.mcount;
    const int64_t offA = rowA ? qrow(p, c.bk, c.h, c.m0 + qr) : 0;
    const int64_t offB = rowB ? qrow(p, c.bk, c.h, c.m0 + qr + 8) : 0;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int d0 = kk * 16 + qc;
        qa[kk][0] = rowA ? *reinterpret_cast<const uint32_t*>(qbase + offA + d0) : 0u;
        qa[kk][1] = rowB ? *reinterpret_cast<const uint32_t*>(qbase + offB + d0) : 0u;
        qa[kk][2] = rowA ? *reinterpret_cast<const uint32_t*>(qbase + offA + d0 + 8) : 0u;
        qa[kk][3] = rowB ? *reinterpret_cast<const uint32_t*>(qbase + offB + d0 + 8) : 0u;
    }
    auto limit_of = [&](int r, bool live) -> int {
        if (!live) return 0;
        const int lim = p.causal ? c.len - p.qlen + 1 + (c.m0 + r) % p.qlen : c.len;
        return min(lim, c.t_end);
    };
    const int limA = limit_of(qr, rowA), limB = limit_of(qr + 8, rowB);

    float oacc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[n][e] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

    const uint32_t tx = 2u * p.box_rows * kRowBytes;
    for (int j = 0; j < c.n_tiles; ++j) {
        const int st = j % p.stages;
        const bool ok = mbar_wait_bounded(smem_u32(&bars[st]), (j / p.stages) & 1);
        const int tile0 = c.t_begin + j * kTile;
        const int nvalid = min(16, max(0, c.t_end - tile0 - warp * 16));
        if (ok && nvalid > 0) {
            uint8_t* sK = smem + st * 2 * kTileBytes;
            uint8_t* sV = sK + kTileBytes;
            if (nvalid < 16) {
                // Rows past the end hold stale or fill data; P is 0 there but 0 * NaN
                // would still poison the product, so clear them before P.V.
                for (int x = lane; x < (16 - nvalid) * 8; x += 32) {
                    const int row = warp * 16 + nvalid + (x >> 3);
                    *reinterpret_cast<uint4*>(sV + swz(row, x & 7)) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async();
                __syncwarp();
            }
            const uint32_t kb = smem_u32(sK), vb = smem_u32(sV);
            float sacc[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[n][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int krow = warp * 16 + (jm >> 1) * 8 + rr;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kb + swz(krow, kk * 2 + (jm & 1)), b0, b1, b2, b3);
                Mma<T>::run(sacc[0], qa[kk], b0, b1);
                Mma<T>::run(sacc[1], qa[kk], b2, b3);
            }
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = tile0 + warp * 16 + n * 8 + qc + (e & 1);
                    const int lim = e < 2 ? limA : limB;
                    sacc[n][e] = key < lim ? sacc[n][e] * p.scale_log2 : -INFINITY;
                }
            float tA = fmaxf(fmaxf(sacc[0][0], sacc[0][1]), fmaxf(sacc[1][0], sacc[1][1]));
            float tB = fmaxf(fmaxf(sacc[0][2], sacc[0][3]), fmaxf(sacc[1][2], sacc[1][3]));
            tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, 1));
            tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, 2));
            tB = fmaxf(tB, __shfl_xor_sync(0xffffffffu, tB, 1));
            tB = fmaxf(tB, __shfl_xor_sync(0xffffffffu, tB, 2));
            const float nA = fmaxf(mA, tA), nB = fmaxf(mB, tB);
            const float refA = nA == -INFINITY ? 0.f : nA, refB = nB == -INFINITY ? 0.f : nB;
            const float aA = exp2f(mA - refA), aB = exp2f(mB - refB);
            mA = nA;
            mB = nB;
            uint32_t pa[4];
            pa[0] = Half16<T>::from_f2(exp2f(sacc[0][0] - refA), exp2f(sacc[0][1] - refA));
            pa[1] = Half16<T>::from_f2(exp2f(sacc[0][2] - refB), exp2f(sacc[0][3] - refB));
            pa[2] = Half16<T>::from_f2(exp2f(sacc[1][0] - refA), exp2f(sacc[1][1] - refA));
            pa[3] = Half16<T>::from_f2(exp2f(sacc[1][2] - refB), exp2f(sacc[1][3] - refB));
            // The normaliser sums the rounded weights that actually multiply V.
            const float2 r0 = Half16<T>::to_f2(pa[0]), r1 = Half16<T>::to_f2(pa[1]);
            const float2 r2 = Half16<T>::to_f2(pa[2]), r3 = Half16<T>::to_f2(pa[3]);
            lA = fmaf(lA, aA, (r0.x + r0.y) + (r2.x + r2.y));
            lB = fmaf(lB, aB, (r1.x + r1.y) + (r3.x + r3.y));
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                oacc[n][0] *= aA;
                oacc[n][1] *= aA;
                oacc[n][2] *= aB;
                oacc[n][3] *= aB;
            }
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                const int vrow = warp * 16 + (jm & 1) * 8 + rr;
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(vb + swz(vrow, 2 * np + (jm >> 1)), v0, v1, v2, v3);
                Mma<T>::run(oacc[2 * np], pa, v0, v1);
                Mma<T>::run(oacc[2 * np + 1], pa, v2, v3);
            }
        }
        if (__syncthreads_or(!ok)) {
            drain_after_timeout(p, c, bars, j);
            abort_block(p);
            return;
        }
        if (tid == 0 && j + p.stages < c.n_tiles) {
            fence_proxy_async();
            issue_tile(&tmk, &tmv, smem, bars, st, c.t_begin + (j + p.stages) * kTile, c.h,
                       c.bk, tx);
        }
    }
    pdl_trigger();

    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    {
        float* red_o = red;
        float* red_m = red + 4 * RM * kHeadDim;
        float* red_l = red_m + 4 * RM;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            float* oa = red_o + (warp * RM + qr) * kHeadDim + n * 8 + qc;
            float* ob = red_o + (warp * RM + qr + 8) * kHeadDim + n * 8 + qc;
            oa[0] = oacc[n][0];
            oa[1] = oacc[n][1];
            ob[0] = oacc[n][2];
            ob[1] = oacc[n][3];
        }
        if ((lane & 3) == 0) {
            red_m[warp * RM + qr] = mA;
            red_m[warp * RM + qr + 8] = mB;
            red_l[warp * RM + qr] = lA;
            red_l[warp * RM + qr + 8] = lB;
        }
    }
    __syncthreads();
    finish_cta<T, RM>(p, c, red, fin, misc, smem);
}

// ---------------------------------------------------------------- host side --------
namespace {

constexpr int kDecodeMmax = 8;
constexpr int kVerifyMmax = 16;
constexpr int kMaxDev = 64;

// Once per kernel and device: allow more than 48 KiB of dynamic shared memory and
// clusters of up to 16 CTAs. Returns the largest usable cluster (16, else 8), 0 on error.
template <auto Kern>
int prepare_kernel(size_t smem_bytes) {
    static std::once_flag once[kMaxDev];
    static int result[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    std::call_once(once[dev], [&] {
        if (cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_bytes) != cudaSuccess) {
            result[dev] = 0;
            return;
        }
        const bool big = cudaFuncSetAttribute(Kern, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                              1) == cudaSuccess;
        cudaGetLastError();
        result[dev] = big ? kMaxClusterSplits : 8;
    });
    return result[dev];
}

template <typename T, int MS>
int prepare_decode_ms() {
    return prepare_kernel<decode_attn_kernel<T, MS>>(smem_layout(kMaxStages, MS).total);
}

template <typename T>
int prepare_decode(int ms) {
    switch (ms) {
    case 1: return prepare_decode_ms<T, 1>();
    case 2: return prepare_decode_ms<T, 2>();
    case 3: return prepare_decode_ms<T, 3>();
    case 4: return prepare_decode_ms<T, 4>();
    case 5: return prepare_decode_ms<T, 5>();
    case 6: return prepare_decode_ms<T, 6>();
    case 7: return prepare_decode_ms<T, 7>();
    case 8: return prepare_decode_ms<T, 8>();
    }
    return 0;
}

template <typename T>
int prepare_verify() {
    return prepare_kernel<verify_attn_kernel<T>>(smem_layout(kMaxStages, 16).total);
}

template <typename T, int MS>
kvd_status launch_decode_ms(dim3 grid, cudaStream_t st, bool pdl, unsigned cl,
                            const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p) {
    return launch_ex(decode_attn_kernel<T, MS>, grid, dim3(128), smem_layout(p.stages, MS).total,
                     st, pdl, cl, mk, mv, p);
}

template <typename T>
kvd_status launch_decode(int ms, dim3 grid, cudaStream_t st, bool pdl, unsigned cl,
                         const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p) {
    switch (ms) {
    case 1: return launch_decode_ms<T, 1>(grid, st, pdl, cl, mk, mv, p);
    case 2: return launch_decode_ms<T, 2>(grid, st, pdl, cl, mk, mv, p);
    case 3: return launch_decode_ms<T, 3>(grid, st, pdl, cl, mk, mv, p);
    case 4: return launch_decode_ms<T, 4>(grid, st, pdl, cl, mk, mv, p);
    case 5: return launch_decode_ms<T, 5>(grid, st, pdl, cl, mk, mv, p);
    case 6: return launch_decode_ms<T, 6>(grid, st, pdl, cl, mk, mv, p);
    case 7: return launch_decode_ms<T, 7>(grid, st, pdl, cl, mk, mv, p);
    case 8: return launch_decode_ms<T, 8>(grid, st, pdl, cl, mk, mv, p);
    }
    return KVD_ERR_UNSUPPORTED;
}

template <typename T>
kvd_status launch_verify(dim3 grid, cudaStream_t st, bool pdl, unsigned cl,
                         const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p) {
    return launch_ex(verify_attn_kernel<T>, grid, dim3(128), smem_layout(p.stages, 16).total, st,
                     pdl, cl, mk, mv, p);
}

kvd_status attention(bool verify, kvd_dtype dtype, int32_t batch, int32_t n_q_heads,
                     int32_t qlen, const void* q, const kvd_cache* kv, const int32_t* lens,
                     int32_t fixed_len, int32_t rows_per_kv, int32_t causal, float scale,
                     void* out, void* ws, size_t ws_bytes, uint32_t flags, int32_t* dev_err,
                     cudaStream_t stream) {
    if (dtype != KVD_F16 && dtype != KVD_BF16) return KVD_ERR_INVALID_ARG;
    if (kvd_status s = validate_cache(kv)) return s;
    if (batch < 0 || n_q_heads <= 0 || rows_per_kv <= 0) return KVD_ERR_INVALID_ARG;
    if (qlen < 1 || qlen > KVD_MAX_QLEN) return KVD_ERR_UNSUPPORTED;
    if (n_q_heads % kv->n_kv_heads || batch % rows_per_kv) return KVD_ERR_INVALID_ARG;
    if (batch == 0) return KVD_OK;
    if (!q || !out || !aligned16(q) || !aligned16(out)) return KVD_ERR_INVALID_ARG;
    if (batch / rows_per_kv > kv->batch || batch / rows_per_kv > 65535) return KVD_ERR_INVALID_ARG;
    if (!lens && (fixed_len < 0 || fixed_len > kv->capacity)) return KVD_ERR_INVALID_ARG;
    if (!(scale == scale)) return KVD_ERR_INVALID_ARG;
    const int nsm = sm_count();
    if (nsm <= 0) return KVD_ERR_CUDA;
    const int len_bound = lens ? kv->capacity : fixed_len;
    const bool bf = dtype == KVD_BF16;
    const int mmax = verify ? kVerifyMmax : kDecodeMmax;
    // the query block size per thread block depends only on the shape
    const AttnPlan P0 = plan_attention(batch, n_q_heads, kv->n_kv_heads, rows_per_kv, qlen,
                                       len_bound, mmax, 4 * nsm, 1);
    const int max_cluster = verify ? (bf ? prepare_verify<__nv_bfloat16>() : prepare_verify<__half>())
                                   : (bf ? prepare_decode<__nv_bfloat16>(P0.msub)
                                         : prepare_decode<__half>(P0.msub));
    if (max_cluster <= 0) return KVD_ERR_CUDA;
    const AttnPlan P = plan_attention(batch, n_q_heads, kv->n_kv_heads, rows_per_kv, qlen,
                                      len_bound, mmax, 4 * nsm, max_cluster);
    if ((int64_t)kv->n_kv_heads * P.nsub > 65535) return KVD_ERR_UNSUPPORTED;
    if (P.splits > 1 && !P.cluster) {
        if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < P.ws_bytes)
            return KVD_ERR_WORKSPACE;
        if ((size_t)P.units * sizeof(int32_t) > KVD_WS_COUNTER_BYTES) return KVD_ERR_UNSUPPORTED;
    }
    CUtensorMap mk, mv;
    if (kvd_status s = encode_cache_map(&mk, dtype, kv->k, kv)) return s;
    if (kvd_status s = encode_cache_map(&mv, dtype, kv->v, kv)) return s;

    AttnParams p = {};
    p.q = q;
    p.out = out;
    p.lens = lens;
    p.fixed_len = fixed_len;
    p.capacity = kv->capacity;
    p.n_q_heads = n_q_heads;
    p.group = P.group;
    p.rows_per_kv = rows_per_kv;
    p.qlen = qlen;
    p.causal = verify ? (causal != 0) : 0;
    p.M = P.M;
    p.msub = P.msub;
    p.nsub = P.nsub;
    p.splits = P.splits;
    p.tiles_per_split = P.tiles_per_split;
    p.stages = std::max(1, P.stages);
    p.box_rows = std::min(64, kv->capacity);
    p.early = (flags & KVD_FLAG_EARLY_KV) ? 1 : 0;
    p.cluster = P.cluster ? 1 : 0;
    p.scale_log2 = scale * kLog2e;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    p.ws_cnt = reinterpret_cast<int32_t*>(wsb);
    p.ws_part = wsb ? reinterpret_cast<float*>(wsb + P.part_offset) : nullptr;
    p.ws_ml = wsb ? reinterpret_cast<float2*>(wsb + P.ml_offset) : nullptr;
    p.dev_err = dev_err;

    const bool pdl = (flags & (KVD_FLAG_PDL | KVD_FLAG_EARLY_KV)) != 0;
    const dim3 grid(P.splits, kv->n_kv_heads * P.nsub, P.bkv);
    const unsigned cl = P.cluster ? (unsigned)P.splits : 1u;
    if (verify)
        return bf ? launch_verify<__nv_bfloat16>(grid, stream, pdl, cl, mk, mv, p)
                  : launch_verify<__half>(grid, stream, pdl, cl, mk, mv, p);
    return bf ? launch_decode<__nv_bfloat16>(P.msub, grid, stream, pdl, cl, mk, mv, p)
              : launch_decode<__half>(P.msub, grid, stream, pdl, cl, mk, mv, p);
}

}  // namespace
}  // namespace kvd

extern "C" kvd_status kvd_decode_attn(kvd_dtype dtype, int32_t batch, int32_t n_q_heads,
                                      const void* q, const kvd_cache* kv, const int32_t* lens,
                                      int32_t fixed_len, int32_t rows_per_kv, float scale,
                                      void* out, void* workspace, size_t workspace_bytes,
                                      uint32_t flags, int32_t* dev_err, kvd_stream_t stream) {
    return kvd::attention(false, dtype, batch, n_q_heads, 1, q, kv, lens, fixed_len, rows_per_kv,
                          0, scale, out, workspace, workspace_bytes, flags, dev_err,
                          reinterpret_cast<cudaStream_t>(stream));
}

extern "C" kvd_status kvd_verify_attn(kvd_dtype dtype, int32_t batch, int32_t n_q_heads,
                                      int32_t qlen, const void* q, const kvd_cache* kv,
                                      const int32_t* lens, int32_t fixed_len,
                                      int32_t rows_per_kv, int32_t causal, float scale,
                                      void* out, void* workspace, size_t workspace_bytes,
                                      uint32_t flags, int32_t* dev_err, kvd_stream_t stream) {
    return kvd::attention(true, dtype, batch, n_q_heads, qlen, q, kv, lens, fixed_len,
                          rows_per_kv, causal, scale, out, workspace, workspace_bytes, flags,
                          dev_err, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- no-allocation entry
// kvd_decode_attn_noalloc: the decode kernel with its split-merge scratch in a buffer
// compiled into the library, for callers that cannot allocate a workspace (see
// kvdecode.h). Host code must never pass `g_noalloc_scratch` itself to a kernel: on the
// host that name is only a stand-in for the device symbol. The device address is looked
// up once per device with cudaGetSymbolAddress while that device is current.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KVD_NOALLOC_SCRATCH_BYTES];

namespace kvd {
namespace {
std::once_flag g_noalloc_once[kMaxDev];
void* g_noalloc_ptr[kMaxDev];
cudaError_t g_noalloc_err[kMaxDev];

kvd_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return KVD_ERR_CUDA;
    std::call_once(g_noalloc_once[dev], [dev] {
        g_noalloc_err[dev] = cudaGetSymbolAddress(&g_noalloc_ptr[dev], g_noalloc_scratch);
    });
    if (g_noalloc_err[dev] != cudaSuccess || !g_noalloc_ptr[dev]) return KVD_ERR_CUDA;
    *out = g_noalloc_ptr[dev];
    return KVD_OK;
}
}  // namespace
}  // namespace kvd

extern "C" kvd_status kvd_decode_attn_noalloc(kvd_dtype dtype, int32_t batch, int32_t n_q_heads,
                                              const void* q, const kvd_cache* kv,
                                              const int32_t* lens, int32_t fixed_len,
                                              int32_t rows_per_kv, float scale, void* out,
                                              uint32_t flags, int32_t* dev_err,
                                              kvd_stream_t stream) {
    void* scratch = nullptr;
    if (kvd_status s = kvd::noalloc_scratch(&scratch)) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // The buffer keeps whatever the previous call left; its arrival counters must start
    // at zero, so clear them (a call that stopped early could have left them non-zero).
    if (cudaMemsetAsync(scratch, 0, KVD_WS_COUNTER_BYTES, st) != cudaSuccess) return KVD_ERR_CUDA;
    return kvd::attention(false, dtype, batch, n_q_heads, 1, q, kv, lens, fixed_len, rows_per_kv,
                          0, scale, out, scratch, KVD_NOALLOC_SCRATCH_BYTES, flags, dev_err, st);
}
