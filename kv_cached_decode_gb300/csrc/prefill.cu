// prefill.cu -- prefill: the first forward pass over a prompt.
//
// "KV キャッシュが推論を最適化する方法" of "nanoVLM における KV キャッシュ実装": the
// prefill runs the whole prompt through the model once and fills the cache with every
// prompt token's K/V; decoding then adds one token per step. "Inference 抽象と KV
// キャッシュ" of "Whisper のデコーダー内部": the first forward pass covers the initial
// tokens, later ones only the newest. Per head, prompt token j (stored at position
// lens_in + j) attends causally to every cached position t <= lens_in + j:
//   out[b,hq,j,:] = sum_{t <= lens_in[b]+j} softmax_t(scale * q[b,hq,j] . K[b,h,t]) V[b,h,t]
// for j < plens[b] (rows past a row's prompt length are written as zeros).
//
// Design: the prompt's K/V are first written into the cache by the append kernel (with a
// per-row count), then one block handles 64 query positions of one query head: four
// warps of 16 rows each, with Q as m16n8k16 A fragments in registers. K/V tiles of 64
// positions arrive by TMA (128-byte swizzle) through a 3-stage ring and are shared by
// the four warps: S = Q.K^T and O = P.V run on the tensor cores (mma.sync, fp32
// accumulate) with an online softmax in exp2 form; only the tiles a block's rows can see
// are read (causal), and blocks with the most tiles start first.
#include <algorithm>
#include <mutex>

#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {
namespace {

constexpr int kPfWarps = 4;
constexpr int kPfThreads = kPfWarps * 32;
constexpr int kPfRows = kPfWarps * 16;  // query positions per block
constexpr int kPfStages = 3;
constexpr uint32_t kPfSmem = kPfStages * 2 * kTileBytes + kPfStages * 8 + 1024;

struct PrefillParams {
    const void* q;            // [batch, n_q_heads, max_len, 64]
    void* out;                // same layout
    const int32_t* lens_in;   // [batch] positions cached before the prompt, or NULL (0)
    const int32_t* plens;     // [batch] prompt lengths, <= max_len
    int32_t* dev_err;
    int32_t max_len, n_q_heads, group, capacity, q_tiles, box_rows;
    float scale_log2;
    float rope_log2_base;     // > 0 sets the rotary variant's base (log2)
};

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <typename T, bool ROPE>
__global__ void __launch_bounds__(kPfThreads)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPfStages * 2 * kTileBytes);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int qt = p.q_tiles - 1 - (int)blockIdx.x;  // the blocks with most tiles first
    const int hq = blockIdx.y, b = blockIdx.z, hk = hq / p.group;
    pdl_wait();
    const int s0 = p.lens_in ? p.lens_in[b] : 0;
    const int plen = p.plens[b];
    const int q0 = qt * kPfRows;
    const int64_t head_off = ((int64_t)b * p.n_q_heads + hq) * p.max_len * kHeadDim;
    T* outp = static_cast<T*>(p.out) + head_off;
    // a row the append rejected (length out of range) gets zeros, like padding rows
    const bool bad = s0 < 0 || plen < 0 || plen > p.max_len || (int64_t)s0 + plen > p.capacity;
    const int rows_live = bad ? 0 : max(0, min(kPfRows, plen - q0));
    if (rows_live == 0) {
        for (int x = tid; x < kPfRows * 8; x += kPfThreads) {
            const int r = q0 + (x >> 3);
            if (r < p.max_len)
                *reinterpret_cast<uint4*>(outp + (int64_t)r * kHeadDim + (x & 7) * 8) =
                    make_uint4(0u, 0u, 0u, 0u);
        }
        pdl_trigger();
        return;
    }
    const int kv_end = s0 + q0 + rows_live;  // exclusive: the last live row's limit
    const int n_tiles = (kv_end + kTile - 1) / kTile;
    const uint32_t tx = 2u * p.box_rows * kRowBytes;
    auto issue = [&](int j) {
        const int st = j % kPfStages;
        const uint32_t bar = smem_u32(&bars[st]);
        mbar_expect_tx(bar, tx);
        const uint32_t dk = smem_u32(smem + st * 2 * kTileBytes);
        tma_load_4d(dk, &tmk, bar, 0, j * kTile, hk, b);
        tma_load_4d(dk + kTileBytes, &tmv, bar, 0, j * kTile, hk, b);
    };
    if (tid == 0) {
        for (int j = 0; j < kPfStages; ++j) mbar_init(smem_u32(&bars[j]), 1);
        fence_barrier_init();
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        for (int j = 0; j < min(kPfStages, n_tiles); ++j) issue(j);
    }
    __syncthreads();
    pdl_trigger();

    // This warp's 16 query rows as m16n8k16 A fragments (rows past the prompt are 0).
    const int qr = lane >> 2, qc = (lane & 3) * 2;  // fragment row / column pair
    const int jm = lane >> 3, rr = lane & 7;         // ldmatrix matrix / row
    const int rowA = q0 + warp * 16 + qr, rowB = rowA + 8;
    const bool liveA = rowA < plen, liveB = rowB < plen;
    const T* qbase = static_cast<const T*>(p.q) + head_off;
    uint32_t qa[4][4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int d0 = kk * 16 + qc;
        const T* a = qbase + (int64_t)rowA * kHeadDim + d0;
        const T* bq = qbase + (int64_t)rowB * kHeadDim + d0;
        qa[kk][0] = liveA ? *reinterpret_cast<const uint32_t*>(a) : 0u;
        qa[kk][1] = liveB ? *reinterpret_cast<const uint32_t*>(bq) : 0u;
        qa[kk][2] = liveA ? *reinterpret_cast<const uint32_t*>(a + 8) : 0u;
        qa[kk][3] = liveB ? *reinterpret_cast<const uint32_t*>(bq + 8) : 0u;
    }
    if (ROPE) {
        // prompt row r sits at position s0 + r; k-steps kk and kk + 2 hold the two halves
        // of the same rotation pairs in this lane
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = kk * 16 + qc + (e >= 2 ? 8 : 0);
                const int pos = s0 + ((e & 1) ? rowB : rowA);
                float2 lo = Half16<T>::to_f2(qa[kk][e]), hi = Half16<T>::to_f2(qa[kk + 2][e]);
                rope_rotate(lo.x, hi.x, rope_cos_sin(pos, i, p.rope_log2_base));
                rope_rotate(lo.y, hi.y, rope_cos_sin(pos, i + 1, p.rope_log2_base));
                qa[kk][e] = Half16<T>::from_f2(lo.x, lo.y);
                qa[kk + 2][e] = Half16<T>::from_f2(hi.x, hi.y);
            }
    }
    // keys t < lim are visible; rows past the prompt are clamped to the live rows' keys
    // (positions beyond hold other data) and written as zeros
    const int limA = min(s0 + rowA + 1, kv_end), limB = min(s0 + rowB + 1, kv_end);

    float oacc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[n][e] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

    for (int j = 0; j < n_tiles; ++j) {
        const int st = j % kPfStages;
        const bool ok = mbar_wait_bounded(smem_u32(&bars[st]), (j / kPfStages) & 1);
        if (__syncthreads_or(!ok)) {
            // let the copies still in flight land, then leave; the outputs stay unwritten
            if (tid == 0) {
                flag_error(p.dev_err, KVD_ERR_TIMEOUT);
                for (int jj = j; jj < min(n_tiles, j + kPfStages); ++jj)
                    mbar_wait_bounded(smem_u32(&bars[jj % kPfStages]), (jj / kPfStages) & 1);
            }
            return;
        }
        uint8_t* sK = smem + st * 2 * kTileBytes;
        uint8_t* sV = sK + kTileBytes;
        const int t0 = j * kTile;
        if (t0 + kTile > kv_end) {
            // Positions past the last visible key hold other data (or nothing): P is 0
            // there, but 0 * NaN would still poison P.V, so clear those V rows first.
            const int first = kv_end - t0;
            for (int x = tid; x < (kTile - first) * 8; x += kPfThreads)
                *reinterpret_cast<uint4*>(sV + swz(first + (x >> 3), x & 7)) =
                    make_uint4(0u, 0u, 0u, 0u);
            __syncthreads();
        }
        const uint32_t kb = smem_u32(sK), vb = smem_u32(sV);
        // S = Q . K^T over the 64 keys of the tile: 8 key blocks of 8
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kb + swz(np * 16 + (jm >> 1) * 8 + rr, kk * 2 + (jm & 1)), b0, b1, b2, b3);
                Mma<T>::run(s[2 * np], qa[kk], b0, b1);
                Mma<T>::run(s[2 * np + 1], qa[kk], b2, b3);
            }
        }
        float tA = -INFINITY, tB = -INFINITY;
        if (__all_sync(0xffffffffu, t0 + kTile <= min(limA, limB))) {
            // the whole tile is visible to every row of the warp: no mask
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    s[n][e] *= p.scale_log2;
                    if (e < 2) tA = fmaxf(tA, s[n][e]);
                    else tB = fmaxf(tB, s[n][e]);
                }
        } else {
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = t0 + n * 8 + qc + (e & 1);
                    const bool vis = key < (e < 2 ? limA : limB);
                    s[n][e] = vis ? s[n][e] * p.scale_log2 : -INFINITY;
                    if (e < 2) tA = fmaxf(tA, s[n][e]);
                    else tB = fmaxf(tB, s[n][e]);
                }
        }
        tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, 1));
        tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, 2));
        tB = fmaxf(tB, __shfl_xor_sync(0xffffffffu, tB, 1));
        tB = fmaxf(tB, __shfl_xor_sync(0xffffffffu, tB, 2));
        const float nA = fmaxf(mA, tA), nB = fmaxf(mB, tB);
        const float refA = nA == -INFINITY ? 0.f : nA, refB = nB == -INFINITY ? 0.f : nB;
        const float aA = exp2f(mA - refA), aB = exp2f(mB - refB);
        mA = nA;
        mB = nB;
        // P, rounded to the input type, as A fragments of the four 16-key steps; the
        // normaliser sums the rounded weights that multiply V
        uint32_t pa[4][4];
        float sumA = 0.f, sumB = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            pa[ks][0] = Half16<T>::from_f2(exp2f(s[2 * ks][0] - refA), exp2f(s[2 * ks][1] - refA));
            pa[ks][1] = Half16<T>::from_f2(exp2f(s[2 * ks][2] - refB), exp2f(s[2 * ks][3] - refB));
            pa[ks][2] =
                Half16<T>::from_f2(exp2f(s[2 * ks + 1][0] - refA), exp2f(s[2 * ks + 1][1] - refA));
            pa[ks][3] =
                Half16<T>::from_f2(exp2f(s[2 * ks + 1][2] - refB), exp2f(s[2 * ks + 1][3] - refB));
            const float2 r0 = Half16<T>::to_f2(pa[ks][0]), r1 = Half16<T>::to_f2(pa[ks][1]);
            const float2 r2 = Half16<T>::to_f2(pa[ks][2]), r3 = Half16<T>::to_f2(pa[ks][3]);
            sumA += (r0.x + r0.y) + (r2.x + r2.y);
            sumB += (r1.x + r1.y) + (r3.x + r3.y);
        }
        lA = fmaf(lA, aA, sumA);
        lB = fmaf(lB, aB, sumB);
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            oacc[n][0] *= aA;
            oacc[n][1] *= aA;
            oacc[n][2] *= aB;
            oacc[n][3] *= aB;
        }
        // O += P . V: four 16-key steps x 8 blocks of 8 dims
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(vb + swz(ks * 16 + (jm & 1) * 8 + rr, 2 * np + (jm >> 1)), v0, v1, v2, v3);
                Mma<T>::run(oacc[2 * np], pa[ks], v0, v1);
                Mma<T>::run(oacc[2 * np + 1], pa[ks], v2, v3);
            }
        }
        __syncthreads();  // every warp is done with this stage
        if (tid == 0 && j + kPfStages < n_tiles) {
            fence_proxy_async();  // generic writes (cleared rows) before the refill
            issue(j + kPfStages);
        }
    }

    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    const float invA = liveA && lA > 0.f ? 1.f / lA : 0.f;
    const float invB = liveB && lB > 0.f ? 1.f / lB : 0.f;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
        if (rowA < p.max_len)
            *reinterpret_cast<uint32_t*>(outp + (int64_t)rowA * kHeadDim + n * 8 + qc) =
                liveA ? Half16<T>::from_f2(oacc[n][0] * invA, oacc[n][1] * invA) : 0u;
        if (rowB < p.max_len)
            *reinterpret_cast<uint32_t*>(outp + (int64_t)rowB * kHeadDim + n * 8 + qc) =
                liveB ? Half16<T>::from_f2(oacc[n][2] * invB, oacc[n][3] * invB) : 0u;
    }
}

constexpr int kMaxDev = 64;

template <typename T, bool ROPE>
bool prepare_prefill() {
    static std::once_flag once[kMaxDev];
    static bool ok[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
    std::call_once(once[dev], [dev] {
        ok[dev] = cudaFuncSetAttribute(prefill_attn_kernel<T, ROPE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kPfSmem) == cudaSuccess;
        cudaGetLastError();
    });
    return ok[dev];
}

template <typename T, bool ROPE>
kvd_status launch_prefill(dim3 grid, cudaStream_t st, bool pdl, const CUtensorMap& mk,
                          const CUtensorMap& mv, const PrefillParams& p) {
    if (!prepare_prefill<T, ROPE>()) return KVD_ERR_CUDA;
    return launch(prefill_attn_kernel<T, ROPE>, grid, dim3(kPfThreads), kPfSmem, st, pdl, mk,
                  mv, p);
}

}  // namespace
}  // namespace kvd

using namespace kvd;

extern "C" kvd_status kvd_prefill_attn(kvd_dtype dtype, int32_t batch, int32_t n_q_heads,
                                       int32_t max_len, const void* q, const kvd_cache* kv,
                                       const void* k_new, const void* v_new,
                                       const int32_t* lens_in, const int32_t* plens,
                                       int32_t* lens_out, float scale, float rope_base,
                                       void* out, uint32_t flags, int32_t* dev_err,
                                       kvd_stream_t stream) {
    if (dtype != KVD_F16 && dtype != KVD_BF16) return KVD_ERR_INVALID_ARG;
    if (kvd_status s = validate_cache(kv)) return s;
    if (batch < 0 || n_q_heads <= 0 || max_len < 0 || batch > kv->batch)
        return KVD_ERR_INVALID_ARG;
    if (n_q_heads % kv->n_kv_heads) return KVD_ERR_INVALID_ARG;
    if (batch == 0 || max_len == 0) return KVD_OK;
    if (!q || !out || !k_new || !v_new || !plens) return KVD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(k_new) || !aligned16(v_new))
        return KVD_ERR_INVALID_ARG;
    if (lens_out && lens_out == lens_in) return KVD_ERR_INVALID_ARG;
    if (!(scale == scale)) return KVD_ERR_INVALID_ARG;
    if (!(rope_base >= 0.f) || !(rope_base < INFINITY)) return KVD_ERR_INVALID_ARG;
    const int64_t q_tiles = ((int64_t)max_len + kPfRows - 1) / kPfRows;
    if (q_tiles > 0x7fffffff || n_q_heads > 65535 || batch > 65535) return KVD_ERR_UNSUPPORTED;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // 1: the prompt's K/V into the cache (rows j < plens[b] at lens_in[b] + j)
    if (kvd_status s = launch_append(kv, batch, max_len, k_new, v_new, lens_in, plens, lens_out,
                                     dtype, rope_base, flags, dev_err, st))
        return s;
    // 2: causal attention of the prompt over the cache
    CUtensorMap mk, mv;
    if (kvd_status s = encode_cache_map(&mk, dtype, kv->k, kv)) return s;
    if (kvd_status s = encode_cache_map(&mv, dtype, kv->v, kv)) return s;
    PrefillParams p;
    p.q = q;
    p.out = out;
    p.lens_in = lens_in;
    p.plens = plens;
    p.dev_err = dev_err;
    p.max_len = max_len;
    p.n_q_heads = n_q_heads;
    p.group = n_q_heads / kv->n_kv_heads;
    p.capacity = kv->capacity;
    p.q_tiles = (int)q_tiles;
    p.box_rows = std::min(64, kv->capacity);
    p.scale_log2 = scale * 1.4426950408889634f;
    const dim3 grid((unsigned)q_tiles, (unsigned)n_q_heads, (unsigned)batch);
    // The attention waits for the append (a dependent launch when PDL is requested).
    const bool pdl = (flags & (KVD_FLAG_PDL | KVD_FLAG_EARLY_KV)) != 0;
    const bool rope = rope_base > 0.f;
    p.rope_log2_base = rope ? log2f(rope_base) : 0.f;
    if (dtype == KVD_BF16)
        return rope ? launch_prefill<__nv_bfloat16, true>(grid, st, pdl, mk, mv, p)
                    : launch_prefill<__nv_bfloat16, false>(grid, st, pdl, mk, mv, p);
    return rope ? launch_prefill<__half, true>(grid, st, pdl, mk, mv, p)
                : launch_prefill<__half, false>(grid, st, pdl, mk, mv, p);
}
