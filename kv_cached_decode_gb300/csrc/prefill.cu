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
// per-row count); then the attention kernel runs on the fifth-generation tensor cores.
// A block takes 128 query positions of one query head: four softmax warps own the rows
// (thread t: row t, tensor-memory lane t) and one producer warp issues every TMA copy
// and every tcgen05.mma. The rows, rotated if asked, are staged once into shared memory
// in the 128-byte-swizzled layout; K/V tiles of 64 positions arrive by TMA (the same
// swizzle) through 5 slots of K/V pairs.
//   S = Q . K^T   M 128, N 64, K 64 (Q and K K-major, shared memory) -> tensor memory
//   O += P . V    M 128, N 64, K 64 (P in tensor memory, V MN-major)  -> tensor memory
// Each row reads its S with tcgen05.ld, applies the causal mask where the tile is not
// wholly visible to its warp, forms the weights exp2(s * scale * log2 e - m) rounded to
// the input type in registers, sums them, and stores them into its lane of the P
// operand (two buffers) with tcgen05.st. A row's reference m moves
// only when its maximum grows by more than 2^8; the rows then rescale their O in tensor
// memory. Hand-offs run through mbarriers, every wait bounded. Only the tiles a block's
// rows can see are read, and the blocks with the most tiles start first.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "kvd_common.cuh"
#include "kvd_internal.h"
#include "kvd_tc.cuh"

namespace kvd {
namespace {

constexpr int kPfSoftWarps = 4;                        // softmax warps: thread t owns row t
constexpr int kPfThreads = (kPfSoftWarps + 1) * 32;    // + the producer warp
constexpr int kPfRows = kPfSoftWarps * 32;             // query positions per block (MMA M)
constexpr int kPfSlots = 5;    // K/V tile pairs in flight (one barrier per pair)
constexpr int kPfSBufs = 2;    // S buffers in tensor memory: S is issued two tiles ahead
constexpr int kPfPBufs = 2;    // P buffers in tensor memory
// The hand-offs, per tile j (one producer iteration per tile):
//  * the rows wait for S_j, write P_j into P buffer j % 2 and signal P_j;
//  * the producer waits for that signal, issues P_j . V_j and then S_{j+2} into S buffer
//    j % 2 (the rows have read S_j), and refills the slot of tile j - 2 with tile
//    j - 2 + kPfSlots.
// A commit tracks every MMA its thread issued before it, and P_{j-2} . V_{j-2} is issued
// before S_j. So a row that sees S_j complete may overwrite P buffer j % 2 without a wait
// of its own, and the signal of P_j, sent after the rows saw S_j, tells the producer that
// the slot of tile j - 2 is free (no wait on P_{j-2} . V_{j-2}). The refilled pair is
// needed by S_{j-2+kPfSlots}, issued kPfSlots - 4 iterations later.
static_assert(kPfSBufs == 2 && kPfPBufs == 2 && kPfSlots >= 5, "the hand-offs above");
constexpr int kPfMinBlocks = 2;  // blocks per SM the sizes below are chosen for
// tensor memory: S buffers (64 fp32 columns each), O (64), then P buffers (32 columns
// each: a row's 64 weights, two 16-bit values per column)
constexpr uint32_t kPfColsO = kPfSBufs * kTile;
constexpr uint32_t kPfColsP = kPfColsO + kHeadDim;
constexpr uint32_t kPfCols = 256;  // allocated (a power of two)
static_assert(kPfCols >= kPfColsP + kPfPBufs * (kTile / 2), "tensor memory columns");
static_assert(kPfMinBlocks * kPfCols <= 512, "the resident blocks' tensor memory");
constexpr uint32_t kPfRowsBytes = kPfRows * kRowBytes;  // 16 KiB: the Q block
// shared memory: K slots | V slots | Q | barriers
constexpr uint32_t kPfSmem = 2 * kPfSlots * kTileBytes + kPfRowsBytes + 256 + 1024;
// The softmax reference of a row moves only when its maximum grows by more than this
// (log2 units): the weights then stay below 2^8 and the output is rescaled rarely.
constexpr float kRescaleLog2 = 8.f;

struct PrefillParams {
    const void* q;            // [batch, n_q_heads, max_len, 64]
    void* out;                // same layout
    const int32_t* lens_in;   // [batch] positions cached before the prompt, or NULL (0)
    const int32_t* plens;     // [batch] prompt lengths, <= max_len
    int32_t* dev_err;
    int32_t max_len, n_q_heads, group, capacity, q_tiles, box_rows;
    float scale_log2;
    float rope_log2_base;     // > 0 sets the rotary variant's base (log2)
    int32_t test_stall;       // KVD_FLAG_TEST_STALL: the first K copy is never issued
};

// Three-input maximum and two-lane fp32 arithmetic of this architecture: one instruction
// for what takes two otherwise; each lane rounds as the scalar instruction does.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// (a.x * b.x + c.x, a.y * b.y + c.y), each fused and rounded to nearest
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 a, b, c, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
// (a.x + b.x, a.y + b.y), each rounded to nearest
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Barrier indices inside the block's barrier array.
enum PfBar {
    kBarKV = 0,                          // K and V of slot s landed (TMA bytes)
    kBarS = kBarKV + kPfSlots,           // S buffer b written (MMA commit)
    kBarPFull = kBarS + kPfSBufs,        // P buffer b written by every row (128 arrivals)
    kBarO = kBarPFull + kPfPBufs,        // P.V from P buffer b done (MMA commit)
    kBarDrain = kBarO + kPfPBufs,        // every MMA issued so far done (after a failure)
    kBarCount = kBarDrain + 1
};

template <typename T, bool ROPE>
__global__ void __launch_bounds__(kPfThreads, kPfMinBlocks)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv,
                        const __grid_constant__ CUtensorMap tmo, const PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    uint8_t* sK = smem;                        // kPfSlots x 8 KiB
    uint8_t* sV = sK + kPfSlots * kTileBytes;   // kPfSlots x 8 KiB
    uint8_t* sQ = sV + kPfSlots * kTileBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sQ + kPfRowsBytes);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kBarCount);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int tid = threadIdx.x, warp = tid >> 5;
    const bool producer = warp == kPfSoftWarps;
    // Blocks are dispatched in linear order; the linear index runs over the query tiles
    // last to first, then over (head, row), so the blocks with the most K/V tiles of
    // every row start first and the short ones fill in behind them.
    const int64_t lin =
        blockIdx.x + (int64_t)gridDim.x * (blockIdx.y + (int64_t)gridDim.y * blockIdx.z);
    const int64_t per_tile = (int64_t)gridDim.y * gridDim.z;
    const int qt = p.q_tiles - 1 - (int)(lin / per_tile);
    const int hq = (int)(lin % per_tile % gridDim.y), b = (int)(lin % per_tile / gridDim.y);
    const int hk = hq / p.group;
    pdl_wait();
    const int s0 = p.lens_in ? p.lens_in[b] : 0;
    const int plen = p.plens[b];
    const int q0 = qt * kPfRows;
    const int row = q0 + tid;  // meaningful for the softmax threads
    const int64_t head_off = ((int64_t)b * p.n_q_heads + hq) * p.max_len * kHeadDim;
    // a row the append rejected (length out of range) gets zeros, like padding rows
    const bool bad = s0 < 0 || plen < 0 || plen > p.max_len || (int64_t)s0 + plen > p.capacity;
    const int rows_live = bad ? 0 : max(0, min(kPfRows, plen - q0));
    // The block's 128 output rows leave through the Q tile's shared memory (free once every
    // S has completed) and one tensor store; rows past max_len fall outside the tensor.
    auto store_rows = [&]() {
        fence_proxy_async();  // the rows' generic writes, read by the tensor store
        asm volatile("bar.sync 1, %0;" ::"n"(kPfRows) : "memory");
        if (tid == 0 && tslot[1] == 0) {
            tma_store_4d(&tmo, smem_u32(sQ), 0, q0, hq, b);
            bulk_commit();
            bulk_wait_read();
        }
    };
    if (rows_live == 0) {
        // no live row: the tile's rows below max_len get zeros, by plain stores
        const int nrows = min(kPfRows, p.max_len - q0);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + head_off +
                                              (int64_t)q0 * kHeadDim);
        for (int x = tid; x < nrows * 8; x += kPfThreads) dst[x] = make_uint4(0u, 0u, 0u, 0u);
        pdl_trigger();
        return;
    }
    const int kv_end = s0 + q0 + rows_live;  // exclusive: the last live row's limit
    const int n_tiles = (kv_end + kTile - 1) / kTile;
    const uint32_t tx = p.box_rows * kRowBytes;  // bytes of one K or V tile copy
    // K_j and V_j into slot j % kPfSlots, both completing on the slot's barrier
    auto load_kv = [&](int j) {
        const int s = j % kPfSlots;
        mbar_expect_tx(bar(kBarKV + s), 2 * tx);
        tma_load_4d(smem_u32(sK + s * kTileBytes), &tmk, bar(kBarKV + s), 0, j * kTile, hk, b);
        tma_load_4d(smem_u32(sV + s * kTileBytes), &tmv, bar(kBarKV + s), 0, j * kTile, hk, b);
    };
    if (producer && (tid & 31) == 0) {
        for (int i = 0; i < kBarCount; ++i)
            mbar_init(bar(i), (i >= kBarPFull && i < kBarPFull + kPfPBufs) ? kPfRows : 1);
        fence_barrier_init();
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
        for (int j = p.test_stall ? 1 : 0; j < min(kPfSlots, n_tiles); ++j) load_kv(j);
    }
    if (warp == 0) {
        tc_alloc(smem_u32(tslot), kPfCols);
        tc_relinquish();
    }
    if (tid == kPfRows - 1) tslot[1] = 0;  // set when a row could not produce its output
    const bool live = !producer && row < plen;
    if (!producer) {
        // this thread's query row (zeros past the prompt), rotated at position s0 + row,
        // into the swizzled A operand
        uint4 qv[8];
        const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + head_off +
                                                           (int64_t)row * kHeadDim);
#pragma unroll
        for (int c = 0; c < 8; ++c) qv[c] = live ? qrow[c] : make_uint4(0u, 0u, 0u, 0u);
        if (ROPE && live) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
                rope_rotate8_at<T>(qv[c], qv[c + 4], s0 + row, 8 * c, p.rope_log2_base);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(sQ + swz(tid, c)) = qv[c];
        fence_proxy_async();  // generic writes, read by the tensor cores
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    pdl_trigger();

    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kIdS = tc_idesc_f16(kBf16, kPfRows, kTile, false);
    constexpr uint32_t kIdO = tc_idesc_f16(kBf16, kPfRows, kHeadDim, true);
    const uint32_t t_o = tmem + kPfColsO;  // the output accumulator
    bool ok = true;

    if (producer) {
        // ---- producer warp: the whole warp runs the loop, so its control flow and the
        // operand descriptors stay warp-uniform; one elected lane (the same one every
        // time, so its commits track its own MMAs) issues each copy, MMA and commit ----
        const uint32_t qaddr = smem_u32(sQ);
        int kv_issued = min(kPfSlots, n_tiles);
        auto wait_all = [&](int i, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar(i), parity));
        };
        // S_j = Q . K_j^T into S buffer j % 2 once tile j has landed
        auto issue_s = [&](int j) -> bool {
            const int s = j % kPfSlots, sb = j % kPfSBufs;
            if (!wait_all(kBarKV + s, (j / kPfSlots) & 1)) return false;
            tc_fence_after();
            const uint32_t kaddr = smem_u32(sK + s * kTileBytes);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_f16(tmem + sb * kTile, tc_desc_sw128(qaddr + kk * 32),
                               tc_desc_sw128(kaddr + kk * 32), kIdS, kk);
                tc_commit(bar(kBarS + sb));
            }
            __syncwarp();
            return true;
        };
        for (int j = 0; ok && j < min(kPfSBufs, n_tiles); ++j) ok = issue_s(j);
        for (int j = 0; ok && j < n_tiles; ++j) {
            // P_j . V_j once the rows have written P_j (V_j landed before S_j was issued)
            const int pb = j % kPfPBufs;
            if (!(ok = wait_all(kBarPFull + pb, (j / kPfPBufs) & 1))) break;
            tc_fence_after();
            const uint32_t t_p = tmem + kPfColsP + pb * (kTile / 2);
            const uint32_t vaddr = smem_u32(sV + (j % kPfSlots) * kTileBytes);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_f16_tmem_a(t_o, t_p + kk * 8,
                                      tc_desc_sw128(vaddr + kk * 16 * kRowBytes), kIdO,
                                      j > 0 || kk > 0);
                tc_commit(bar(kBarO + pb));
            }
            __syncwarp();
            // S_{j+2} into the S buffer the rows have read S_j from
            if (j + kPfSBufs < n_tiles && !(ok = issue_s(j + kPfSBufs))) break;
            // the rows saw S_j complete before they signalled P_j, and P_{j-2} . V_{j-2}
            // (the last reader of the slot of tile j - 2) was issued before S_j: that
            // slot takes tile j - 2 + kPfSlots
            if (j >= 2 && j - 2 + kPfSlots < n_tiles) {
                if (elect_one()) load_kv(j - 2 + kPfSlots);
                __syncwarp();
                kv_issued = j - 1 + kPfSlots;
            }
        }
        if (!ok && elect_one()) {
            // let the MMAs and copies in flight finish before the block leaves
            flag_error(p.dev_err, KVD_ERR_TIMEOUT);
            tc_commit(bar(kBarDrain));
            mbar_wait_bounded(bar(kBarDrain), 0);
            for (int jj = max(p.test_stall ? 1 : 0, kv_issued - kPfSlots); jj < kv_issued; ++jj)
                mbar_wait_bounded(bar(kBarKV + jj % kPfSlots), (jj / kPfSlots) & 1);
        }
        __syncwarp();
    } else {
        // ---- the rows: S_j into P_j, one row per thread ----
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;  // this warp's 32 lanes
        // With a positive scale the maximum is taken over the raw scores and the scale is
        // folded into the exponent, one FFMA per weight.
        const bool pos_scale = p.scale_log2 > 0.f;
        const float cs = pos_scale ? p.scale_log2 : 1.f;
        // keys t < lim are visible; rows past the prompt are clamped to the live rows'
        // keys (positions beyond hold other data) and written as zeros. Rows ascend with
        // the lane, so lane 0 holds the warp's smallest limit.
        const int lim = min(s0 + row + 1, kv_end);
        const int lim_warp = __shfl_sync(0xffffffffu, lim, 0);
        float m = -INFINITY, l = 0.f;  // the row's reference (log2 units) and normaliser
        for (int j = 0; j < n_tiles; ++j) {
            const int sb = j % kPfSBufs, pb = j % kPfPBufs;
            const int t0 = j * kTile;
            if (!__all_sync(0xffffffffu,
                            mbar_wait_bounded(bar(kBarS + sb), (j / kPfSBufs) & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[kTile];
            tc_ld32(tmem + lane_off + sb * kTile, s);
            tc_ld32(tmem + lane_off + sb * kTile + 32, s + 32);
            if (!pos_scale) {
#pragma unroll
                for (int i = 0; i < kTile; ++i) s[i] *= p.scale_log2;
            }
            if (t0 + kTile > lim_warp) {
                // the tile is not wholly visible to every row of the warp: mask it
#pragma unroll
                for (int i = 0; i < kTile; ++i) s[i] = t0 + i < lim ? s[i] : -INFINITY;
            }
            // (eight independent partial maxima over eight scores each: short chains)
            float pm[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float a = fmax3(s[e], s[e + 8], s[e + 16]);
                a = fmax3(a, s[e + 24], s[e + 32]);
                a = fmax3(a, s[e + 40], s[e + 48]);
                pm[e] = fmaxf(a, s[e + 56]);
            }
            const float tmax =
                fmaxf(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], fmaxf(pm[5],
                      fmaxf(pm[6], pm[7])))) * cs;
            const float mc = fmaxf(m, tmax);
            const bool grow = mc > m + kRescaleLog2;
            float factor = 1.f;
            if (grow) {
                factor = exp2f(m - mc);  // 0 on the first tile
                m = mc;
            }
            l *= factor;
            if (j >= 1 && __any_sync(0xffffffffu, grow)) {
                // O is rescaled once P_{j-1} . V_{j-1} is done
                if (!__all_sync(0xffffffffu,
                                mbar_wait_bounded(bar(kBarO + (j - 1) % kPfPBufs),
                                                  ((j - 1) / kPfPBufs) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float ov[32];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    tc_ld32(t_o + lane_off + h * 32, ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] *= factor;
                    tc_st32(t_o + lane_off + h * 32, ov);
                }
            }
            // The weights, rounded to the input type; the normaliser sums the unrounded
            // weights (rounding to nearest leaves no bias).
            const float nref = m == -INFINITY ? 0.f : -m;
            // eight partial sums, as four lane pairs
            float2 ps[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) ps[e] = make_float2(0.f, 0.f);
            uint32_t w[kTile / 2];
#pragma unroll
            for (int i = 0; i < kTile / 2; ++i) {
                const float2 x = ffma2(make_float2(s[2 * i], s[2 * i + 1]), make_float2(cs, cs),
                                       make_float2(nref, nref));
                const float2 pw = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                ps[i & 3] = fadd2(ps[i & 3], pw);
                w[i] = Half16<T>::from_f2(pw.x, pw.y);
            }
            l += ((ps[0].x + ps[0].y) + (ps[1].x + ps[1].y)) +
                 ((ps[2].x + ps[2].y) + (ps[3].x + ps[3].y));
            // this row of the A operand, in this thread's lane of tensor memory (its last
            // reader, P_{j-2} . V_{j-2}, completed before S_j did)
            tc_st32_u(tmem + lane_off + kPfColsP + pb * (kTile / 2), w);
            if (t0 + kTile > kv_end) {
                // Positions past the last visible key hold other data (or nothing): P is
                // 0 there, but 0 * NaN would still poison P.V, so clear those V rows once
                // the tile's copy has landed.
                const int vs = j % kPfSlots;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarKV + vs),
                                                                (j / kPfSlots) & 1))) {
                    ok = false;
                    break;
                }
                uint8_t* vt = sV + vs * kTileBytes;
                const int first = kv_end - t0;
                for (int x = tid; x < (kTile - first) * 8; x += kPfRows)
                    *reinterpret_cast<uint4*>(vt + swz(first + (x >> 3), x & 7)) =
                        make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async();  // the cleared rows are read by the tensor cores
            }
            tc_fence_before();
            mbar_arrive(bar(kBarPFull + pb));
        }
        bool wrote = false;
        if (!ok) {
            if ((tid & 31) == 0) flag_error(p.dev_err, KVD_ERR_TIMEOUT);
        } else {
            const int jl = n_tiles - 1;
            const bool done =
                __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarO + jl % kPfPBufs),
                                                          (jl / kPfPBufs) & 1));
            tc_fence_after();
            float o[kHeadDim];
            tc_ld32(t_o + lane_off, o);
            tc_ld32(t_o + lane_off + 32, o + 32);
            if (!done) {
                if ((tid & 31) == 0) flag_error(p.dev_err, KVD_ERR_TIMEOUT);
            } else {
                // every MMA has completed, so this row of the Q tile is free
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);  // rows past the prompt: +0
                    if (live) {
                        w.x = Half16<T>::from_f2(o[8 * c] * inv, o[8 * c + 1] * inv);
                        w.y = Half16<T>::from_f2(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
                        w.z = Half16<T>::from_f2(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
                        w.w = Half16<T>::from_f2(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
                    }
                    *reinterpret_cast<uint4*>(sQ + swz(tid, c)) = w;
                }
                wrote = true;
            }
        }
        // a warp that gave up leaves the whole tile unwritten
        if ((tid & 31) == 0 && !wrote) atomicOr(reinterpret_cast<int*>(&tslot[1]), 1);
        store_rows();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tc_dealloc(tmem, kPfCols);
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
                          const CUtensorMap& mv, const CUtensorMap& mo, const PrefillParams& p) {
    if (!prepare_prefill<T, ROPE>()) return KVD_ERR_CUDA;
    return launch(prefill_attn_kernel<T, ROPE>, grid, dim3(kPfThreads), kPfSmem, st, pdl, mk,
                  mv, mo, p);
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
    CUtensorMap mk, mv, mo;
    if (kvd_status s = encode_cache_map(&mk, dtype, kv->k, kv)) return s;
    if (kvd_status s = encode_cache_map(&mv, dtype, kv->v, kv)) return s;
    if (kvd_status s = encode_rows_map(&mo, dtype, out, max_len, n_q_heads, batch,
                                       std::min(kPfRows, max_len)))
        return s;
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
    p.test_stall = (flags & KVD_FLAG_TEST_STALL) ? 1 : 0;
    const dim3 grid((unsigned)q_tiles, (unsigned)n_q_heads, (unsigned)batch);
    // The attention waits for the append (a dependent launch when PDL is requested).
    const bool pdl = (flags & (KVD_FLAG_PDL | KVD_FLAG_EARLY_KV)) != 0;
    const bool rope = rope_base > 0.f;
    p.rope_log2_base = rope ? log2f(rope_base) : 0.f;
    if (dtype == KVD_BF16)
        return rope ? launch_prefill<__nv_bfloat16, true>(grid, st, pdl, mk, mv, mo, p)
                    : launch_prefill<__nv_bfloat16, false>(grid, st, pdl, mk, mv, mo, p);
    return rope ? launch_prefill<__half, true>(grid, st, pdl, mk, mv, mo, p)
                : launch_prefill<__half, false>(grid, st, pdl, mk, mv, mo, p);
}
