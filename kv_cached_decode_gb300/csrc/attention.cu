// attention.cu -- decode attention (self and cross), verify-block attention, the split
// merge and the optional fused append of the new tokens, for sm_103a.
//
// What is computed ("KV キャッシュが推論を最適化する方法" steps 2-4 of "nanoVLM における KV
// キャッシュ実装"; "Inference 抽象と KV キャッシュ" of "Whisper のデコーダー内部"; "추측
// 디코딩이란?" of "추측 디코딩으로 Whisper 추론 속도 2배 향상"):
//   out[r,hq,i,:] = sum_{t < limit_i} softmax_t(scale * q[r,hq,i] . K[b,h,t]) V[b,h,t]
// with b = r / rows_per_kv, h = hq / group, limit_i = len (decode, cross) or
// len - qlen + 1 + i (causal verify block whose K/V are appended).
//
// How (GB300 design):
//  * One thread block handles one (cache row b, KV head h, chunk of positions) and ALL
//    query vectors that read that KV head -- rows_per_kv beam rows x group query heads x
//    qlen tokens -- so every K/V byte is fetched from HBM once per call.
//  * K/V tiles of 64 positions x 64 dims (8 KiB each) are staged into shared memory by
//    TMA (cp.async.bulk.tensor, 128-byte swizzle) through a ring of 2 or 4 stages whose
//    full-barriers are mbarriers with transaction counts; one thread issues the copies.
//    Eight warps work on two tiles at a time, each warp on its own 16-position slab, so
//    a warp waits only for its own tile and no block barrier is needed except before a
//    stage is refilled.
//  * One query vector per KV head (plain multi-head decode) runs on CUDA cores: eight
//    lanes share a cache position, each holding 16 bytes (8 dims) of K and V; the dot
//    product finishes with three xor shuffles and feeds an online softmax in exp2 form.
//  * Two to sixteen query vectors per KV head (grouped-query heads, beam rows sharing a
//    window, a verify block) form a small GEMM and run on the tensor cores: S = Q.K^T
//    and O = P.V as mma.sync m16n8k16 (fp16/bf16 in, fp32 accumulate), operands read
//    from the swizzled tiles by ldmatrix (K) and ldmatrix.trans (V).
//  * Fused append: when the new tokens' K/V are passed, the warp whose slab holds their
//    positions writes them into the cache and into its staged tile, so attention sees
//    them without a separate launch.
//  * Long ranges are split over thread blocks. Splits of one unit that fit in a cluster
//    (<= 16 CTAs) send their (max, sum, o) partials straight into the shared memory of
//    the cluster's first CTA with asynchronous stores (st.async) that count their bytes
//    on its mbarrier; that CTA merges them locally while the others exit. The split
//    count is the largest whose clusters are all resident at once (occupancy
//    calculator), so a launch never runs a second, partial wave. Only a handful of
//    units over a long range split further: each unit then spans several clusters,
//    whose first CTAs' merged partials go through the workspace (or, with few enough
//    splits, every block's partial does), and the last block to arrive (atomic
//    ticket) merges them. Merges run in fixed split order, so results are repeatable.
//  * Programmatic dependent launch: every block lets the next kernel on the stream
//    start as soon as its own copies are issued; with KVD_FLAG_EARLY_KV it also issues
//    those copies before waiting for the previous kernel.
#include <algorithm>
#include <atomic>
#include <climits>
#include <mutex>
#include <unordered_map>

#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSlot = kHeadDim + 4;   // floats per merge slot: o[64], max, sum, 2 pad
constexpr int kSlotQuads = kSlot / 4;  // 17 float4 per slot
// Row stride (floats) of the warp partials o[warp][row][.]: with 16 rows per warp the
// fragment layout writes 8 rows at once, and a stride of 72 (8 banks apart) keeps
// those float2 stores free of bank conflicts.
__host__ __device__ constexpr int red_stride(int rmax) { return rmax > 1 ? kHeadDim + 8 : kHeadDim; }

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
    int32_t cluster;   // 1: the splits of a unit form thread-block clusters
    int32_t cgroups;   // clusters per unit; > 1: their first CTAs merge through the workspace
    int32_t csize;     // CTAs per cluster (splits / cgroups)
    int32_t test_stall;  // test only: the last split of every unit never sees its first stage
    unsigned long long merge_wait_ns;  // the first CTA's bound on its wait for the partials
    int32_t append;    // 1: k_new/v_new are written at positions lens[b] .. lens[b]+qlen-1
    int32_t rope;      // 1: rotary encoding of the queries and the appended keys
    float rope_log2_base;
    const uint8_t* k_new;
    const uint8_t* v_new;
    int32_t* lens_out;
    uint8_t* kc;       // cache bases and byte strides, for the appended rows
    uint8_t* vc;
    int64_t sb, sh, st;
    int32_t n_kv_heads;
    float scale_log2;
    float* ws_part;
    float2* ws_ml;
    int32_t* ws_cnt;
    int32_t* dev_err;
};

// Shared memory: [stages x (K tile, V tile); after the tile loop the same bytes hold the
// warp partials] [stage barriers, merge barrier] [split partials of the cluster, used in
// its first CTA] [flag] [q/out row offsets]. The last 4 KiB of the stage area are scratch
// for the workspace merge.
struct SmemLayout {
    uint32_t bar_off, red_off, mrg_off, misc_off, qoff_off, app_off, total;
};
// app_rows: 256-byte units staged for the fused append: qlen (the K and V rows), plus
// with rotary encoding qlen more (the cos/sin table, 32 float2 per token) and the
// rotated query rows of the block, else 0.
__host__ __device__ inline SmemLayout smem_layout(int stages, int rmax, int merge_slots,
                                                  int app_rows) {
    SmemLayout L;
    const uint32_t tiles = stages * 2 * kTileBytes;
    const uint32_t red = kWarps * rmax * (red_stride(rmax) + 2) * 4;
    L.red_off = 0;
    L.bar_off = ((tiles > red ? tiles : red) + 1023) & ~1023u;
    L.mrg_off = (L.bar_off + (stages + 1) * 8 + 15) & ~15u;
    L.misc_off = L.mrg_off + merge_slots * kSlot * 4;
    L.qoff_off = L.misc_off + 16;  // element offsets of the block's query rows in q / out
    L.app_off = L.qoff_off + kMmaQueryBlock * 8;  // appended rows: K [qlen][128 B], V, table
    L.total = L.app_off + app_rows * 2 * kRowBytes + 1024;  // + slack to align the base
    return L;
}
__host__ __device__ inline int merge_slots(int cluster, int splits, int msub) {
    return cluster ? splits * msub : 0;
}
// The rotated query rows of a tensor-core block (16 rows, 144-byte stride so that the
// ldmatrix rows fall in distinct banks): 2304 bytes = 9 units.
constexpr int kQsStride = 144;
constexpr int kQsUnits = 9;
__host__ __device__ inline int app_units(int append, int rope, int qlen) {
    return append ? qlen * (rope ? 2 : 1) + (rope ? kQsUnits : 0) : 0;
}
__host__ __device__ inline int app_units(const AttnParams& p) {
    return app_units(p.append, p.rope, p.qlen);
}
// The rotary cos/sin table of the call's new tokens: [qlen][32] float2, token j at
// position len - qlen + j (its absolute position), after the appended rows.
__device__ __forceinline__ const float2* rope_table(const AttnParams& p, const uint8_t* app) {
    return reinterpret_cast<const float2*>(app + p.qlen * 2 * kRowBytes);
}

struct CtaCtx {
    // s: split of the unit; rank / grp: place in its cluster / the cluster's index
    int bk, h, sub, s, rank, grp, m0, mcount, len, new0, t_begin, t_end, n_tiles, unit;
    bool bad;
};

// Give-up points of the block's waits. Every wait is bounded relative to its own start
// (kWaitNs, 1 s, in the mbarrier helpers; the timer is read only once a wait turns
// slow), and they are ordered so that a first CTA that receives its cluster peers'
// partials never exits while a peer can still send:
//  * a thread's tile waits: at most one per round, each within 1 s, and none after the
//    first that runs out -- at most `rounds` seconds in all;
//  * a block that gave up drains its copies in flight (at most one wait per stage, each
//    within 1 s) and sends nothing;
//  * so every peer that sends has sent within `rounds` seconds of passing the
//    dependency wait, and the first CTA waits for the partials (rounds + stages + 1)
//    seconds after it starts waiting, which is after it passed that wait too: it is
//    still waiting when the last partial lands, and a unit with a peer that gave up
//    ends in the first CTA's timeout (no output). All CTAs of a cluster are resident
//    together and pass the dependency wait within microseconds of one another, far
//    inside the 1 s margin.
// (rounds + stages + 1) seconds, computed on the host into AttnParams::merge_wait_ns.
inline unsigned long long merge_wait_budget(int tiles_per_split, int stages) {
    return (unsigned long long)((tiles_per_split + 1) / 2 + stages + 1) * kWaitNs;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void setup_ctx(const AttnParams& p, CtaCtx& c) {
    c.s = blockIdx.x;
    c.grp = p.cgroups > 1 ? c.s / p.csize : 0;
    c.rank = c.s - c.grp * p.csize;
    c.h = blockIdx.y / p.nsub;
    c.sub = blockIdx.y % p.nsub;
    c.bk = blockIdx.z;
    c.unit = (c.bk * p.n_kv_heads + c.h) * p.nsub + c.sub;
    c.m0 = c.sub * p.msub;
    c.mcount = min(p.msub, p.M - c.m0);
    const int len0 = p.lens ? p.lens[c.bk] : p.fixed_len;
    c.len = p.append ? len0 + p.qlen : len0;
    c.new0 = p.append ? len0 : INT_MAX;
    c.bad = len0 < 0 || c.len > p.capacity;
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

// Bytes every non-first CTA of a cluster sends into the first CTA's merge slots.
__device__ __forceinline__ uint32_t merge_bytes_per_cta(int mcount) {
    return (uint32_t)(kSlotQuads * mcount * 16);
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

// qoff[m]: element offset of the block's query vector m in q and out (computed once in
// the prologue: the index arithmetic has runtime divisions).
template <typename T>
__device__ __forceinline__ void store_out(const AttnParams& p, const int64_t* qoff, int m, int d,
                                          float v) {
    T* o = static_cast<T*>(p.out) + qoff[m] + d;
    *o = Half16<T>::from_f(v);
}

// Shared prologue. Reads the length, initialises the stage barriers (and, in the first
// CTA of a cluster, the merge barrier), issues the first copies, lets the next kernel
// start, and waits for the previous one (before all of this unless the call was made
// with KVD_FLAG_EARLY_KV). Returns false if the length is out of range: flagged,
// nothing written.
template <bool ROPE>
__device__ __forceinline__ bool prologue(const AttnParams& p, CtaCtx& c, uint8_t* smem,
                                         uint64_t* bars, int64_t* qoff, uint8_t* app,
                                         const CUtensorMap* tmk, const CUtensorMap* tmv) {
    const int tid = threadIdx.x;
    if (!p.early) pdl_wait();
    setup_ctx(p, c);
    if (c.bad) {
        if (p.early) pdl_wait();
        if (tid == 0 && c.s == 0 && c.h == 0 && c.sub == 0) {
            flag_error(p.dev_err, KVD_ERR_LEN_OVERFLOW);
            if (p.append && p.lens_out) p.lens_out[c.bk] = p.lens[c.bk];
        }
        return false;
    }
    if (tid == 0) {
        for (int j = 0; j < p.stages; ++j) mbar_init(smem_u32(&bars[j]), 1);
        if (p.cluster && c.rank == 0) mbar_init(smem_u32(&bars[p.stages]), 1);
        fence_barrier_init();
        if (p.cluster && c.rank == 0)  // the one arrival; the others' bytes complete the phase
            mbar_expect_tx(smem_u32(&bars[p.stages]),
                           (p.csize - 1) * merge_bytes_per_cta(c.mcount));
        prefetch_tensormap(tmk);
        prefetch_tensormap(tmv);
        const uint32_t tx = 2u * p.box_rows * kRowBytes;
        const int first = min(p.stages, c.n_tiles);
        // test only: the last split's first stage expects 16 bytes more than its copies
        // bring (set before they are issued), so that phase never completes and every wait
        // on it runs out; the copies themselves all land
        if (p.test_stall && c.s == p.splits - 1 && first > 0)
            mbar_expect_tx_only(smem_u32(&bars[0]), 16);
        for (int j = 0; j < first; ++j)
            issue_tile(tmk, tmv, smem, bars, j, c.t_begin + j * kTile, c.h, c.bk, tx);
    }
    // the last warp, clear of thread 0's copies
    const int qi = tid - (kThreads - kMmaQueryBlock);
    if (qi >= 0 && qi < c.mcount) {
        const int64_t off = qrow(p, c.bk, c.h, c.m0 + qi);
        qoff[qi] = off;
        if (p.early)  // bring the query rows into L2 while waiting
            prefetch_l2(static_cast<const uint8_t*>(p.q) + off * 2);
    }
    // Blocks that inject appended rows bring those rows of k_new / v_new into L2 too
    // (one 128-byte line per row and tensor).
    if (p.early && p.append && c.new0 < c.t_end && c.len > c.t_begin) {
        const int ai = tid - (kThreads - 2 * kMmaQueryBlock);
        if (ai >= 0 && ai < 2 * p.qlen) {
            const int j = ai >> 1;
            const int64_t row = ((int64_t)c.bk * p.n_kv_heads + c.h) * p.qlen + j;
            prefetch_l2((ai & 1 ? p.v_new : p.k_new) + row * kRowBytes);
        }
    }
    // The rotary table of the new tokens' positions (with KVD_FLAG_EARLY_KV, before the
    // wait: it depends only on the length).
    if (ROPE) {
        float2* tab = const_cast<float2*>(rope_table(p, app));
        const int pos0 = c.len - p.qlen;
        for (int x = tid; x < p.qlen * 32; x += kThreads)
            tab[x] = rope_cos_sin(pos0 + (x >> 5), x & 31, p.rope_log2_base);
    }
    __syncthreads();
    // Every CTA of a cluster arrives here, before any wait of its own: the cluster
    // barrier waits below (merge, abort) therefore always complete.
    if (p.cluster) cluster_arrive_relaxed();  // the first CTA's merge barrier is ready
    pdl_trigger();
    if (p.early) pdl_wait();
    if (p.append && p.lens_out && tid == 0 && c.s == 0 && c.h == 0 && c.sub == 0)
        p.lens_out[c.bk] = c.len;
    return true;
}

// Fused append, per warp: the rows of this warp's 16-position slab that hold new tokens
// come from k_new/v_new, not from the copy (which saw the cache before the append).
// The warp stages those rows into shared memory with cp.async right after the dependency
// wait (stage_appended), so their load latency overlaps the rest of the prologue; here
// it copies them into its staged tile (the warp reads only its own slab) and, by the
// first query sub-block, into the cache. app: K rows [qlen][128 B], then V rows.
__device__ __forceinline__ void for_appended_chunks(const AttnParams& p, const CtaCtx& c,
                                                    int tile0, int slab0, int& r0, int& n2) {
    r0 = max(tile0 + slab0, c.new0);
    const int r1 = min(tile0 + slab0 + 16, c.len);
    n2 = r0 < r1 ? 2 * (r1 - r0) * 8 : 0;  // 16-byte chunks of K and V
}
__device__ __forceinline__ void stage_appended(const AttnParams& p, const CtaCtx& c,
                                               uint8_t* app, int tile0, int slab0) {
    int r0, n2;
    for_appended_chunks(p, c, tile0, slab0, r0, n2);
    const int lane = threadIdx.x & 31;
    for (int x = lane; x < n2; x += 32) {
        const bool is_v = x >= n2 / 2;
        const int y = is_v ? x - n2 / 2 : x;
        const int j = r0 + (y >> 3) - c.new0, ch = y & 7;
        const int64_t src =
            (((int64_t)c.bk * p.n_kv_heads + c.h) * p.qlen + j) * kRowBytes + ch * 16;
        cp_async16(smem_u32(app + (is_v ? p.qlen * kRowBytes : 0) + j * kRowBytes + ch * 16),
                   (is_v ? p.v_new : p.k_new) + src);
    }
}
template <typename T, bool ROPE>
__device__ __forceinline__ void inject_slab(const AttnParams& p, const CtaCtx& c, uint8_t* sK,
                                            uint8_t* sV, const uint8_t* app, int tile0,
                                            int slab0) {
    int r0, n2;
    for_appended_chunks(p, c, tile0, slab0, r0, n2);
    if (n2 == 0) return;
    cp_async_wait_all();
    __syncwarp();
    const int lane = threadIdx.x & 31;
    auto put = [&](bool is_v, int t, int ch, const uint4& val) {
        *reinterpret_cast<uint4*>((is_v ? sV : sK) + swz(t - tile0, ch)) = val;
        if (c.sub == 0)
            *reinterpret_cast<uint4*>((is_v ? p.vc : p.kc) + c.bk * p.sb + c.h * p.sh +
                                      (int64_t)t * p.st + ch * 16) = val;
    };
    if (ROPE) {
        // per row: 4 K chunk pairs (ch, ch + 4), rotated at the token's position, then
        // the 8 V chunks as they are
        const float2* tab = rope_table(p, app);
        const int rows = n2 / 16;
        for (int x = lane; x < rows * 12; x += 32) {
            const int t = r0 + x / 12, y = x % 12, j = t - c.new0;
            if (y < 4) {
                const uint8_t* kr = app + j * kRowBytes;
                uint4 lo = *reinterpret_cast<const uint4*>(kr + y * 16);
                uint4 hi = *reinterpret_cast<const uint4*>(kr + (y + 4) * 16);
                rope_rotate8<T>(lo, hi, tab + j * 32, y * 8);
                put(false, t, y, lo);
                put(false, t, y + 4, hi);
            } else {
                const int ch = y - 4;
                put(true, t, ch,
                    *reinterpret_cast<const uint4*>(app + p.qlen * kRowBytes + j * kRowBytes +
                                                    ch * 16));
            }
        }
    } else {
        for (int x = lane; x < n2; x += 32) {
            const bool is_v = x >= n2 / 2;
            const int y = is_v ? x - n2 / 2 : x;
            const int t = r0 + (y >> 3), ch = y & 7;
            put(is_v, t, ch,
                *reinterpret_cast<const uint4*>(app + (is_v ? p.qlen * kRowBytes : 0) +
                                                (t - c.new0) * kRowBytes + ch * 16));
        }
    }
    fence_proxy_async();  // the stage is refilled by TMA later
    __syncwarp();
}

// After a timed-out wait: wait (each within 1 s) for the latest copy issued into every
// stage, so that none is still writing shared memory when the block exits. A non-first
// CTA of a cluster then sends nothing: the first CTA's wait for the partials runs out,
// so it flags the timeout and writes no output for the unit. A first CTA that gave up
// still waits (merge_wait_ns) for the others' partials, since they land in its shared
// memory, before it exits.
//
// Every wait on this path ends: the drain waits and the first CTA's wait are bounded;
// __syncthreads is reached by all threads (the caller's __syncthreads_or is
// block-uniform); the cluster barrier wait completes because every CTA of the cluster
// arrived on it in the prologue, before any wait.
__device__ void abort_after_timeout(const AttnParams& p, const CtaCtx& c, uint64_t* bars,
                                    float* mrg, int issued) {
    const int tid = threadIdx.x;
    if (tid == 0) {
        flag_error(p.dev_err, KVD_ERR_TIMEOUT);
        for (int j = max(0, issued - p.stages); j < issued; ++j)
            mbar_wait_bounded(smem_u32(&bars[j % p.stages]), (j / p.stages) & 1);
    }
    __syncthreads();
    if (p.cluster) {
        cluster_wait();
        if (c.rank == 0 && tid == 0)
            mbar_wait_bounded_cluster(smem_u32(&bars[p.stages]), 0, p.merge_wait_ns);
    }
}

// The tile loop shared by both kernels. Tiles are taken two at a time (a round); warp w
// works on tile 2r + w/4, positions (w%4)*16 .. +15, through slab(sK, sV, tile0, slab0).
// Returns false after a timeout (already handled: the caller just returns).
template <typename T, bool ROPE, typename Slab>
__device__ __forceinline__ bool run_tiles(const AttnParams& p, const CtaCtx& c, uint8_t* smem,
                                          uint64_t* bars, float* mrg, uint8_t* app,
                                          const CUtensorMap* tmk, const CUtensorMap* tmv,
                                          Slab&& slab) {
    const int tid = threadIdx.x, warp = tid >> 5;
    const int half = warp >> 2, slab0 = (warp & 3) * 16;
    const uint32_t tx = 2u * p.box_rows * kRowBytes;
    bool all_ok = true;
    int issued = min(p.stages, c.n_tiles);
    const int rounds = (c.n_tiles + 1) / 2;
    if (p.append && c.new0 < c.t_end) {
        for (int r = 0; r < rounds; ++r)
            if (2 * r + half < c.n_tiles)
                stage_appended(p, c, app, c.t_begin + (2 * r + half) * kTile, slab0);
        cp_async_commit();
    }
    for (int r = 0; r < rounds; ++r) {
        const int j = 2 * r + half;
        if (j < c.n_tiles) {
            const int st = j % p.stages;
            // after a failed wait this thread does not wait again; the block aborts at the
            // next block barrier
            const bool ok = all_ok && mbar_wait_bounded(smem_u32(&bars[st]), (j / p.stages) & 1);
            all_ok = ok;
            if (ok) {
                uint8_t* sK = smem + st * 2 * kTileBytes;
                uint8_t* sV = sK + kTileBytes;
                const int tile0 = c.t_begin + j * kTile;
                if (p.append) inject_slab<T, ROPE>(p, c, sK, sV, app, tile0, slab0);
                slab(sK, sV, tile0, slab0);
            }
        }
        if (2 * r + p.stages < c.n_tiles) {  // this round's stages are refilled
            if (__syncthreads_or(!all_ok)) {
                abort_after_timeout(p, c, bars, mrg, issued);
                return false;
            }
            if (tid == 0) {
                fence_proxy_async();
                for (int k = 0; k < 2 && 2 * r + p.stages + k < c.n_tiles; ++k) {
                    const int jn = 2 * r + p.stages + k;
                    issue_tile(tmk, tmv, smem, bars, jn % p.stages, c.t_begin + jn * kTile, c.h,
                               c.bk, tx);
                }
            }
            issued = min(c.n_tiles, issued + 2);
        }
    }
    if (__syncthreads_or(!all_ok)) {
        abort_after_timeout(p, c, bars, mrg, issued);
        return false;
    }
    return true;
}

// The partials of a unit in the workspace (n of them, slots unit * n * msub + i * msub +
// m): the block that arrives last (atomic ticket) merges them in slot order, loading them
// in parallel, and writes the output.
template <typename T>
__device__ void ws_merge_last(const AttnParams& p, const CtaCtx& c, float* red, int* misc,
                              const int64_t* qoff, uint8_t* scratch4k, int n) {
    const int tid = threadIdx.x;
    const int S = n;
    const size_t base = (size_t)c.unit * S * p.msub;
    __threadfence();
    __syncthreads();
    if (tid == 0) misc[0] = (atomicAdd(&p.ws_cnt[c.unit], 1) == S - 1) ? 1 : 0;
    __syncthreads();
    if (!misc[0]) return;
    __threadfence();
    // (a) all (max, sum) pairs at once -> normalised weights in shared memory.
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
    // groups * nq4 <= max(blockDim.x, nq4) float4s (at most 4 KiB), at the end of the
    // stage area, clear of the weights above
    float4* tmp = reinterpret_cast<float4*>(scratch4k);
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
        uint2 packed;
        packed.x = Half16<T>::from_f2(acc.x, acc.y);
        packed.y = Half16<T>::from_f2(acc.z, acc.w);
        *reinterpret_cast<uint2*>(static_cast<T*>(p.out) + qoff[m] + d) = packed;
    }
    if (tid == 0) p.ws_cnt[c.unit] = 0;
}

// A cluster's merge of float4 q4 of one query vector's output: the vector's slots in
// the cluster's CS splits (at sl0 + r * stride: o[64], max, sum) combined in split order
// into (max, sum, o), o unnormalised. Loads are unconditional (a split past CS re-reads the last slot and gets
// weight 0) and go in batches of four, so they overlap.
__device__ __forceinline__ void merge_cluster_quad(const float* sl0, int stride, int CS, int q4,
                                                   float& mx, float& l, float4& o) {
    mx = -INFINITY;
#pragma unroll
    for (int r = 0; r < kMaxClusterSplits; ++r)
        mx = fmaxf(mx, sl0[min(r, CS - 1) * stride + kHeadDim]);
    const float ref = mx == -INFINITY ? 0.f : mx;
    l = 0.f;
    o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int r0 = 0; r0 < CS; r0 += 4) {
        float4 v[4];
        float mv[4], lv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float* sl = sl0 + min(r0 + j, CS - 1) * stride;
            v[j] = *reinterpret_cast<const float4*>(sl + 4 * q4);
            mv[j] = sl[kHeadDim];
            lv[j] = sl[kHeadDim + 1];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = r0 + j < CS ? exp2f(mv[j] - ref) : 0.f;
            l = fmaf(lv[j], a, l);
            o.x = fmaf(v[j].x, a, o.x);
            o.y = fmaf(v[j].y, a, o.y);
            o.z = fmaf(v[j].z, a, o.z);
            o.w = fmaf(v[j].w, a, o.w);
        }
    }
}

// Combine the eight warps' partial states, then
//  * one split: write the output;
//  * splits forming clusters: store the block's (max, sum, o) into the merge slots of its
//    cluster's first CTA (one float4 per thread, asynchronous stores counted on that
//    CTA's barrier); the first CTA waits for all of them and merges locally. With one
//    cluster per unit it writes the output; with several, each first CTA publishes its
//    cluster's (max, sum, o) to the workspace and the last to arrive merges those;
//  * more splits than a cluster holds, without clusters: publish to the workspace; the
//    last block to arrive (atomic ticket) merges all splits, loading them in parallel.
// Merges run over the splits in index order, so results do not depend on timing. The
// merge across clusters is compiled only into the GROUPED builds, which run the launches
// whose plan has several clusters per unit: kept out of the other builds, the code after
// the cluster merge stays as short as the chain of every single-cluster launch needs.
// red: o [8][RMAX][red_stride], m [8][RMAX], l [8][RMAX]; mrg: [splits][msub][kSlot].
template <typename T, int RMAX, bool GROUPED>
__device__ void finish_cta(const AttnParams& p, const CtaCtx& c, float* red, float* mrg,
                           uint64_t* merge_bar, int* misc, const int64_t* qoff,
                           uint8_t* scratch4k) {
    constexpr int RS = red_stride(RMAX);
    const float* red_o = red;
    const float* red_m = red + kWarps * RMAX * RS;
    const float* red_l = red_m + kWarps * RMAX;
    const int tid = threadIdx.x;
    const int S = p.splits;
    const size_t base = (size_t)c.unit * S * p.msub;

    if (S > 1 && p.cluster) {
        const int CS = p.csize;  // splits of this cluster
        cluster_wait();  // the first CTA's merge barrier is initialised
        const bool leader = c.rank == 0;
        const uint32_t dst = leader ? 0u : map_shared(smem_u32(mrg), 0);
        const uint32_t rbar = leader ? 0u : map_shared(smem_u32(merge_bar), 0);
        // One thread per float4 of a slot: 16 of o, then (max, sum). Loads are
        // unconditional (the (max, sum) thread reads an o quad it ignores) and go in
        // batches of four warps.
        for (int it = tid; it < kSlotQuads * c.mcount; it += blockDim.x) {
            const int m = it / kSlotQuads, k = it % kSlotQuads;
            const int kk = min(k, kHeadDim / 4 - 1);
            float mx = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, red_m[w * RMAX + m]);
            const float ref = mx == -INFINITY ? 0.f : mx;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            float l = 0.f;
#pragma unroll
            for (int w0 = 0; w0 < kWarps; w0 += 4) {
                float4 o[4];
                float mw[4], lw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int w = w0 + j;
                    o[j] = *reinterpret_cast<const float4*>(red_o + (w * RMAX + m) * RS + 4 * kk);
                    mw[j] = red_m[w * RMAX + m];
                    lw[j] = red_l[w * RMAX + m];
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float a = exp2f(mw[j] - ref);
                    l = fmaf(lw[j], a, l);
                    v.x = fmaf(o[j].x, a, v.x);
                    v.y = fmaf(o[j].y, a, v.y);
                    v.z = fmaf(o[j].z, a, v.z);
                    v.w = fmaf(o[j].w, a, v.w);
                }
            }
            if (k == kHeadDim / 4) v = make_float4(mx, l, 0.f, 0.f);
            const int slot = (c.rank * p.msub + m) * kSlot + 4 * k;
            if (leader)
                *reinterpret_cast<float4*>(mrg + slot) = v;
            else
                st_async_v4(dst + slot * 4, v, rbar);
        }
        if (!leader) return;
        // One warp waits for the other CTAs' bytes (merge_wait_ns: longer than any peer
        // can take to send); the block barrier then orders those bytes, and the slots
        // this CTA's own threads wrote, before every thread's reads.
        const bool ok =
            tid >= 32 || mbar_wait_bounded_cluster(smem_u32(merge_bar), 0, p.merge_wait_ns);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) flag_error(p.dev_err, KVD_ERR_TIMEOUT);
            return;
        }
        if (GROUPED && p.cgroups > 1) {
            // this cluster's (max, sum, o), unnormalised, for the merge across clusters
            for (int it = tid; it < c.mcount * (kHeadDim / 4); it += blockDim.x) {
                const int m = it >> 4, q4 = it & 15;
                float mx, l;
                float4 o;
                merge_cluster_quad(mrg + m * kSlot, p.msub * kSlot, CS, q4, mx, l, o);
                const size_t slot = ((size_t)c.unit * p.cgroups + c.grp) * p.msub + m;
                *reinterpret_cast<float4*>(p.ws_part + slot * kHeadDim + 4 * q4) = o;
                if (q4 == 0) p.ws_ml[slot] = make_float2(mx, l);
            }
            ws_merge_last<T>(p, c, red, misc, qoff, scratch4k, p.cgroups);
            return;
        }
        // One thread per (query vector, 4 dims).
        for (int it = tid; it < c.mcount * (kHeadDim / 4); it += blockDim.x) {
            const int m = it >> 4, q4 = it & 15;
            float mx, l;
            float4 o;
            merge_cluster_quad(mrg + m * kSlot, p.msub * kSlot, CS, q4, mx, l, o);
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint2 packed;
            packed.x = Half16<T>::from_f2(o.x * inv, o.y * inv);
            packed.y = Half16<T>::from_f2(o.z * inv, o.w * inv);
            *reinterpret_cast<uint2*>(static_cast<T*>(p.out) + qoff[m] + 4 * q4) = packed;
        }
        return;
    }

    const size_t slot0 = base + (size_t)c.s * p.msub;
    for (int idx = tid; idx < c.mcount * kHeadDim; idx += blockDim.x) {
        const int m = idx >> 6, d = idx & 63;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, red_m[w * RMAX + m]);
        const float ref = mx == -INFINITY ? 0.f : mx;
        float l = 0.f, o = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float a = exp2f(red_m[w * RMAX + m] - ref);
            l = fmaf(red_l[w * RMAX + m], a, l);
            o = fmaf(red_o[(w * RMAX + m) * RS + d], a, o);
        }
        if (S == 1) {
            store_out<T>(p, qoff, m, d, l > 0.f ? o / l : 0.f);
        } else {
            p.ws_part[(slot0 + m) * kHeadDim + d] = o;
            if (d == 0) p.ws_ml[slot0 + m] = make_float2(mx, l);
        }
    }
    if (S == 1) return;
    ws_merge_last<T>(p, c, red, misc, qoff, scratch4k, S);
}

// ------------------------------------------------- one query vector per KV head (SIMT) --
template <typename T, bool ROPE, bool GROUPED = false>
__global__ void __launch_bounds__(kThreads, 4)  // <= 64 registers: 4 blocks per SM
    decode_attn_kernel(const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const AttnParams p) {
    constexpr int RM = 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    const SmemLayout L = smem_layout(p.stages, RM,
                                     merge_slots(p.cluster, p.csize, p.msub),
                                     app_units(p));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);
    float* red = reinterpret_cast<float*>(smem + L.red_off);
    float* mrg = reinterpret_cast<float*>(smem + L.mrg_off);
    int* misc = reinterpret_cast<int*>(smem + L.misc_off);
    int64_t* qoff = reinterpret_cast<int64_t*>(smem + L.qoff_off);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = lane >> 3, c8 = lane & 7;

    CtaCtx c;
    if (!prologue<ROPE>(p, c, smem, bars, qoff, smem + L.app_off, &tmk, &tmv)) return;

    float qf[8];
    {
        const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + qoff[0] +
                                                        c8 * 8);
        unpack8<T>(u, qf);
    }
    if (ROPE) {
        // the one query token sits at position len - 1; lane c8 ^ 4 holds the other half
        // of its rotation pairs
        const float2* tab = rope_table(p, smem + L.app_off);
        const bool hi = c8 >= 4;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            float y[2];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const float other = __shfl_xor_sync(0xffffffffu, qf[e + t], 4);
                float x0 = hi ? other : qf[e + t], x1 = hi ? qf[e + t] : other;
                rope_rotate(x0, x1, tab[(c8 & 3) * 8 + e + t]);
                y[t] = hi ? x1 : x0;
            }
            const float2 r = Half16<T>::to_f2(Half16<T>::from_f2(y[0], y[1]));
            qf[e] = r.x;
            qf[e + 1] = r.y;
        }
    }
    float mrun = -INFINITY, lrun = 0.f, acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;

    auto slab = [&](const uint8_t* sK, const uint8_t* sV, int tile0, int slab0) {
        float sc[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int row = slab0 + grp * 4 + jj;
            const bool valid = tile0 + row < c.t_end;
            const uint4 kr = *reinterpret_cast<const uint4*>(sK + swz(row, c8));
            float kf[8];
            unpack8<T>(kr, kf);
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) d = fmaf(qf[e], kf[e], d);
            d += __shfl_xor_sync(0xffffffffu, d, 1);
            d += __shfl_xor_sync(0xffffffffu, d, 2);
            d += __shfl_xor_sync(0xffffffffu, d, 4);
            sc[jj] = valid ? d * p.scale_log2 : -INFINITY;
        }
        const float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        const float mn = fmaxf(mrun, mt);
        const float ref = mn == -INFINITY ? 0.f : mn;
        const float alpha = exp2f(mrun - ref);
        float ls = 0.f;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            sc[jj] = exp2f(sc[jj] - ref);
            ls += sc[jj];
        }
        lrun = fmaf(lrun, alpha, ls);
        mrun = mn;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] *= alpha;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int row = slab0 + grp * 4 + jj;
            const bool valid = tile0 + row < c.t_end;
            const uint4 vr = *reinterpret_cast<const uint4*>(sV + swz(row, c8));
            float vf[8];
            unpack8<T>(vr, vf);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(sc[jj], valid ? vf[e] : 0.f, acc[e]);
        }
    };
    if (!run_tiles<T, ROPE>(p, c, smem, bars, mrg, smem + L.app_off, &tmk, &tmv, slab)) return;

    // Merge the four 8-lane groups of each warp (they saw different positions).
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, mrun, off);
        const float lo = __shfl_xor_sync(0xffffffffu, lrun, off);
        const float mn = fmaxf(mrun, mo);
        const float ref = mn == -INFINITY ? 0.f : mn;
        const float a = exp2f(mrun - ref), b = exp2f(mo - ref);
        lrun = lrun * a + lo * b;
#pragma unroll
        for (int e = 0; e < 8; ++e)
            acc[e] = acc[e] * a + __shfl_xor_sync(0xffffffffu, acc[e], off) * b;
        mrun = mn;
    }
    if (grp == 0) {
        float* red_o = red;
        float* red_m = red + kWarps * RM * red_stride(RM);
        float* red_l = red_m + kWarps * RM;
#pragma unroll
        for (int e = 0; e < 8; ++e) red_o[warp * red_stride(RM) + c8 * 8 + e] = acc[e];
        if (c8 == 0) {
            red_m[warp] = mrun;
            red_l[warp] = lrun;
        }
    }
    __syncthreads();
    finish_cta<T, RM, GROUPED>(p, c, red, mrg, &bars[p.stages], misc, qoff,
                               smem + L.bar_off - 4096);
}

// ------------------------------------ 2..16 query vectors per KV head (tensor cores) ----
// MINB: blocks per SM the register budget is cut for. 2 (no cut) is the default; 3 gives
// more resident blocks, hence more splits, when a launch is limited by residency, at the
// price of a few spilled registers.
// RM: query vectors a block holds, 16 or 8. With at most 8 (decode of one token, a
// verify block of up to 8, grouped heads of up to 8, up to 8 beam rows on one window)
// rows 8..15 of every m16n8k16 product are zero: the A fragments of those rows are the
// constant 0, their S and O accumulators are not kept, and the block needs about 30
// fewer registers -- three blocks per SM without spilling, so that more of the next
// launch's blocks (and its thread-block clusters) fit beside a running launch.
template <typename T, int MINB, bool ROPE, int RM = 16, bool GROUPED = false>
__global__ void __launch_bounds__(kThreads, MINB)
    block_attn_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const AttnParams p) {
    static_assert(RM == 16 || (RM == 8 && !ROPE), "the 8-row build has no rotation");
    constexpr bool kFull = RM == 16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    const SmemLayout L = smem_layout(p.stages, RM,
                                     merge_slots(p.cluster, p.csize, p.msub),
                                     app_units(p));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);
    float* red = reinterpret_cast<float*>(smem + L.red_off);
    float* mrg = reinterpret_cast<float*>(smem + L.mrg_off);
    int* misc = reinterpret_cast<int*>(smem + L.misc_off);
    int64_t* qoff = reinterpret_cast<int64_t*>(smem + L.qoff_off);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int qr = lane >> 2, qc = (lane & 3) * 2;  // fragment row / column pair
    const int jm = lane >> 3, rr = lane & 7;         // ldmatrix matrix / row

    CtaCtx c;
    if (!prologue<ROPE>(p, c, smem, bars, qoff, smem + L.app_off, &tmk, &tmv)) return;

    // Q as m16n8k16 A fragments for the four 16-dim k-steps (rows >= mcount are 0).
    uint32_t qa[4][4];
    const T* qbase = static_cast<const T*>(p.q);
    const bool rowA = qr < c.mcount, rowB = kFull && qr + 8 < c.mcount;
    if (ROPE) {
        // The block's query rows are rotated once, into shared memory (16 threads per
        // row, 2 rotation pairs each; query m is token m % qlen of the new tokens), and
        // every warp then loads its fragments from there with ldmatrix.
        uint8_t* qs = smem + L.app_off + p.qlen * 4 * kRowBytes;
        const float2* tab = rope_table(p, smem + L.app_off);
        const int m = tid >> 4, g = tid & 15;
        uint32_t lo = 0u, hi = 0u;  // dims (2g, 2g + 1) and (2g + 32, 2g + 33)
        if (m < c.mcount) {
            const T* row = qbase + qoff[m];
            lo = *reinterpret_cast<const uint32_t*>(row + 2 * g);
            hi = *reinterpret_cast<const uint32_t*>(row + 32 + 2 * g);
            const float2* tr = tab + ((c.m0 + m) % p.qlen) * 32;
            float2 x0 = Half16<T>::to_f2(lo), x1 = Half16<T>::to_f2(hi);
            rope_rotate(x0.x, x1.x, tr[2 * g]);
            rope_rotate(x0.y, x1.y, tr[2 * g + 1]);
            lo = Half16<T>::from_f2(x0.x, x0.y);
            hi = Half16<T>::from_f2(x1.x, x1.y);
        }
        *reinterpret_cast<uint32_t*>(qs + m * kQsStride + 4 * g) = lo;
        *reinterpret_cast<uint32_t*>(qs + m * kQsStride + 64 + 4 * g) = hi;
        __syncthreads();
        const uint32_t qb = smem_u32(qs) + (uint32_t)(((lane & 7) + ((lane >> 3) & 1) * 8) * kQsStride +
                                                      (lane >> 4) * 16);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            ldsm_x4(qb + kk * 32, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    } else {
        const int64_t offA = rowA ? qoff[qr] : 0;
        const int64_t offB = rowB ? qoff[qr + 8] : 0;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int d0 = kk * 16 + qc;
            qa[kk][0] = rowA ? *reinterpret_cast<const uint32_t*>(qbase + offA + d0) : 0u;
            qa[kk][1] = rowB ? *reinterpret_cast<const uint32_t*>(qbase + offB + d0) : 0u;
            qa[kk][2] = rowA ? *reinterpret_cast<const uint32_t*>(qbase + offA + d0 + 8) : 0u;
            qa[kk][3] = rowB ? *reinterpret_cast<const uint32_t*>(qbase + offB + d0 + 8) : 0u;
        }
    }
    // One product: the full m16n8k16, or with RM == 8 the rows 0..7 only (rows 8..15 of
    // A are zero and their accumulators are not kept).
    auto mma = [&](float* acc, const uint32_t* a, uint32_t b0, uint32_t b1) {
        if (kFull) Mma<T>::run(acc, a, b0, b1);
        else Mma<T>::run_top(acc, a[0], a[2], b0, b1);
    };
    auto limit_of = [&](int r, bool live) -> int {
        if (!live) return 0;
        const int lim = p.causal ? c.len - p.qlen + 1 + (c.m0 + r) % p.qlen : c.len;
        return min(lim, c.t_end);
    };
    const int limA = limit_of(qr, rowA), limB = limit_of(qr + 8, rowB);

    constexpr int kAcc = kFull ? 4 : 2;  // accumulator elements kept per n8 block
    float oacc[8][kAcc];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < kAcc; ++e) oacc[n][e] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

    auto slab = [&](uint8_t* sK, uint8_t* sV, int tile0, int slab0) {
        const int nvalid = min(16, max(0, c.t_end - tile0 - slab0));
        if (nvalid == 0) return;
        if (nvalid < 16) {
            // Rows past the end hold stale or fill data; P is 0 there but 0 * NaN would
            // still poison the product, so clear them before P.V.
            for (int x = lane; x < (16 - nvalid) * 8; x += 32) {
                const int row = slab0 + nvalid + (x >> 3);
                *reinterpret_cast<uint4*>(sV + swz(row, x & 7)) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async();
            __syncwarp();
        }
        const uint32_t kb = smem_u32(sK), vb = smem_u32(sV);
        float sacc[2][kAcc];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < kAcc; ++e) sacc[n][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int krow = slab0 + (jm >> 1) * 8 + rr;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kb + swz(krow, kk * 2 + (jm & 1)), b0, b1, b2, b3);
            mma(sacc[0], qa[kk], b0, b1);
            mma(sacc[1], qa[kk], b2, b3);
        }
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < kAcc; ++e) {
                const int key = tile0 + slab0 + n * 8 + qc + (e & 1);
                const int lim = e < 2 ? limA : limB;
                sacc[n][e] = key < lim ? sacc[n][e] * p.scale_log2 : -INFINITY;
            }
        uint32_t pa[4];
        if constexpr (kFull) {
            // rows 0..7 (A) and 8..15 (B): two independent chains, interleaved
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
                oacc[n][kAcc - 2] *= aB;
                oacc[n][kAcc - 1] *= aB;
            }
        } else {
            float tA = fmaxf(fmaxf(sacc[0][0], sacc[0][1]), fmaxf(sacc[1][0], sacc[1][1]));
            tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, 1));
            tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, 2));
            const float nA = fmaxf(mA, tA);
            const float refA = nA == -INFINITY ? 0.f : nA;
            const float aA = exp2f(mA - refA);
            mA = nA;
            pa[0] = Half16<T>::from_f2(exp2f(sacc[0][0] - refA), exp2f(sacc[0][1] - refA));
            pa[2] = Half16<T>::from_f2(exp2f(sacc[1][0] - refA), exp2f(sacc[1][1] - refA));
            pa[1] = pa[3] = 0u;
            const float2 r0 = Half16<T>::to_f2(pa[0]), r2 = Half16<T>::to_f2(pa[2]);
            lA = fmaf(lA, aA, (r0.x + r0.y) + (r2.x + r2.y));
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                oacc[n][0] *= aA;
                oacc[n][1] *= aA;
            }
        }
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            const int vrow = slab0 + (jm & 1) * 8 + rr;
            uint32_t v0, v1, v2, v3;
            ldsm_x4_t(vb + swz(vrow, 2 * np + (jm >> 1)), v0, v1, v2, v3);
            mma(oacc[2 * np], pa, v0, v1);
            mma(oacc[2 * np + 1], pa, v2, v3);
        }
    };
    if (!run_tiles<T, ROPE>(p, c, smem, bars, mrg, smem + L.app_off, &tmk, &tmv, slab)) return;

    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    if (kFull) {
        lB += __shfl_xor_sync(0xffffffffu, lB, 1);
        lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    }
    {
        constexpr int RS = red_stride(RM);
        float* red_o = red;
        float* red_m = red + kWarps * RM * RS;
        float* red_l = red_m + kWarps * RM;
        // only the rows that hold query vectors are read back
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            if (rowA)
                *reinterpret_cast<float2*>(red_o + (warp * RM + qr) * RS + n * 8 + qc) =
                    make_float2(oacc[n][0], oacc[n][1]);
            if (rowB)
                *reinterpret_cast<float2*>(red_o + (warp * RM + qr + 8) * RS + n * 8 + qc) =
                    make_float2(oacc[n][kAcc - 2], oacc[n][kAcc - 1]);
        }
        if ((lane & 3) == 0) {
            red_m[warp * RM + qr] = mA;
            red_l[warp * RM + qr] = lA;
            if (kFull) {
                red_m[warp * RM + qr + 8] = mB;
                red_l[warp * RM + qr + 8] = lB;
            }
        }
    }
    __syncthreads();
    finish_cta<T, RM, GROUPED>(p, c, red, mrg, &bars[p.stages], misc, qoff,
                               smem + L.bar_off - 4096);
}

// ---------------------------------------------------------------- no-allocation scratch
// kvd_decode_attn_noalloc merges split results in this buffer compiled into the library
// instead of a caller's workspace (see kvdecode.h). Host code must never pass
// `g_noalloc_scratch` itself to a kernel: on the host that name is only a stand-in for
// the device symbol. The device address is looked up once per device with
// cudaGetSymbolAddress while that device is current.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KVD_NOALLOC_SCRATCH_BYTES];

namespace {
std::once_flag g_noalloc_once[64];
void* g_noalloc_ptr[64];
cudaError_t g_noalloc_err[64];

kvd_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return KVD_ERR_CUDA;
    std::call_once(g_noalloc_once[dev], [dev] {
        g_noalloc_err[dev] = cudaGetSymbolAddress(&g_noalloc_ptr[dev], g_noalloc_scratch);
    });
    if (g_noalloc_err[dev] != cudaSuccess || !g_noalloc_ptr[dev]) return KVD_ERR_CUDA;
    *out = g_noalloc_ptr[dev];
    return KVD_OK;
}
}  // namespace

// ---------------------------------------------------------------- host side --------
namespace {

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

// Kernel variants: the CUDA-core kernel; the tensor-core kernel built for 2 or 3
// resident blocks per SM; its build for blocks of at most 8 query vectors (3 per SM);
// the first two also with the rotary encoding compiled in (the rotation code is kept out
// of the other builds, whose register budgets it would raise).
enum Variant {
    kSimt = 1, kMma = 2, kMma3 = 3, kSimtRope = 4, kMmaRope = 5, kMma8 = 6,
    kSimtG = 7, kMmaG = 8  // kSimt / kMma with the merge across clusters of a unit
};

// Rows of the warp partials (the red area) of a variant: 16 for the tensor-core builds,
// 8 for the 8-vector build, 1 for the CUDA-core kernel.
constexpr int variant_rmax(int var) {
    return (var == kSimt || var == kSimtRope || var == kSimtG) ? 1 : var == kMma8 ? 8 : 16;
}

template <typename T>
int prepare(int var) {
    const int rmax = variant_rmax(var);
    const uint32_t smem = smem_layout(kMaxStages, rmax, kMaxClusterSplits * std::min(rmax, 16),
                                      2 * KVD_MAX_QLEN + kQsUnits).total;
    switch (var) {
    case kMma: return prepare_kernel<block_attn_kernel<T, 2, false>>(smem);
    case kMma3: return prepare_kernel<block_attn_kernel<T, 3, false>>(smem);
    case kMmaRope: return prepare_kernel<block_attn_kernel<T, 2, true>>(smem);
    case kMma8: return prepare_kernel<block_attn_kernel<T, 3, false, 8>>(smem);
    case kSimtRope: return prepare_kernel<decode_attn_kernel<T, true>>(smem);
    case kMmaG: return prepare_kernel<block_attn_kernel<T, 2, false, 16, true>>(smem);
    case kSimtG: return prepare_kernel<decode_attn_kernel<T, false, true>>(smem);
    default: return prepare_kernel<decode_attn_kernel<T, false>>(smem);
    }
}

template <typename T>
const void* kernel_of(int var) {
    switch (var) {
    case kMma: return reinterpret_cast<const void*>(block_attn_kernel<T, 2, false>);
    case kMma3: return reinterpret_cast<const void*>(block_attn_kernel<T, 3, false>);
    case kMmaRope: return reinterpret_cast<const void*>(block_attn_kernel<T, 2, true>);
    case kMma8: return reinterpret_cast<const void*>(block_attn_kernel<T, 3, false, 8>);
    case kSimtRope: return reinterpret_cast<const void*>(decode_attn_kernel<T, true>);
    case kMmaG: return reinterpret_cast<const void*>(block_attn_kernel<T, 2, false, 16, true>);
    case kSimtG: return reinterpret_cast<const void*>(decode_attn_kernel<T, false, true>);
    default: return reinterpret_cast<const void*>(decode_attn_kernel<T, false>);
    }
}

template <typename T>
kvd_status launch_attn(int var, dim3 grid, cudaStream_t st, bool pdl, unsigned cl,
                       const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p) {
    const int slots = merge_slots(p.cluster, p.csize, p.msub);
    const int app_rows = app_units(p);
    const uint32_t mma_smem = smem_layout(p.stages, 16, slots, app_rows).total;
    const uint32_t simt_smem = smem_layout(p.stages, 1, slots, app_rows).total;
    switch (var) {
    case kMma8:
        return launch_ex(block_attn_kernel<T, 3, false, 8>, grid, dim3(kThreads),
                         smem_layout(p.stages, 8, slots, app_rows).total, st, pdl, cl, mk, mv, p);
    case kMma:
        return launch_ex(block_attn_kernel<T, 2, false>, grid, dim3(kThreads), mma_smem, st, pdl,
                         cl, mk, mv, p);
    case kMma3:
        return launch_ex(block_attn_kernel<T, 3, false>, grid, dim3(kThreads), mma_smem, st, pdl,
                         cl, mk, mv, p);
    case kMmaRope:
        return launch_ex(block_attn_kernel<T, 2, true>, grid, dim3(kThreads), mma_smem, st, pdl,
                         cl, mk, mv, p);
    case kSimtRope:
        return launch_ex(decode_attn_kernel<T, true>, grid, dim3(kThreads), simt_smem, st, pdl,
                         cl, mk, mv, p);
    case kMmaG:
        return launch_ex(block_attn_kernel<T, 2, false, 16, true>, grid, dim3(kThreads), mma_smem,
                         st, pdl, cl, mk, mv, p);
    case kSimtG:
        return launch_ex(decode_attn_kernel<T, false, true>, grid, dim3(kThreads), simt_smem, st,
                         pdl, cl, mk, mv, p);
    default:
        return launch_ex(decode_attn_kernel<T, false>, grid, dim3(kThreads), simt_smem, st, pdl,
                         cl, mk, mv, p);
    }
}

size_t plan_smem(const AttnPlan& P, int var, int app_rows) {
    return smem_layout(P.stages, variant_rmax(var),
                       merge_slots(P.cluster, P.splits / P.cgroups, P.msub), app_rows)
        .total;
}

// How many thread blocks (cluster == 1, whole GPU) or clusters of `cluster` blocks can
// be resident at once, from the CUDA occupancy calculator; cached per device, kernel,
// shared-memory size and cluster size. 0 if the query fails.
int resident(const void* kern, int kid, size_t smem, int cluster, int nsm) {
    static std::mutex mu;
    static std::unordered_map<uint64_t, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const uint64_t key = ((uint64_t)dev << 48) | ((uint64_t)kid << 40) |
                         ((uint64_t)cluster << 32) | (uint64_t)smem;
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int n = 0;
    if (cluster <= 1) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem) != cudaSuccess)
            n = 0;
        n *= nsm;
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cluster, 1, 1);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = cluster;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        cfg.attrs = a;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    std::lock_guard<std::mutex> g(mu);
    cache[key] = n;
    return n;
}

// Split choice. Blocks of one launch should all be resident at once: a second, partial
// wave costs as much as the first. So, for few long units, take the most splits whose
// clusters (one per unit) are all resident together; fall back to one block per unit
// when none fits (many units fill the GPU by themselves). For a handful of units over a
// range longer than one cluster takes in a round per block, give each unit several
// clusters, merged through the workspace after each has merged on chip, as long as all
// of them are resident at once and each block's tiles at least halve. Failing that, and
// only where even 16-block clusters leave each block streaming many tiles, split
// further without clusters and merge through the workspace.
// kern_g / kid_g: the variant's build with the merge across clusters (null: none).
AttnPlan choose_plan(const void* kern, int kid, int var, int nsm, int batch, int n_q_heads,
                     int n_kv_heads, int rows_per_kv, int qlen, int len_bound, int max_cluster,
                     int app_rows, const void* kern_g, int kid_g) {
    const int mmax = variant_rmax(var) > 1 ? kMmaQueryBlock : 1;
    const AttnPlan P1 = plan_attention(batch, n_q_heads, n_kv_heads, rows_per_kv, qlen, len_bound,
                                       mmax, 1, max_cluster);
    if (P1.rounds <= 1) return P1;
    if (workspace_merge_pays(P1.units, P1.rounds)) {
        AttnPlan W = plan_attention(batch, n_q_heads, n_kv_heads, rows_per_kv, qlen, len_bound,
                                    mmax, kMaxSplits, 1);
        const int blocks = resident(kern, kid, plan_smem(W, var, app_rows), 1, nsm);
        W = plan_attention(batch, n_q_heads, n_kv_heads, rows_per_kv, qlen, len_bound, mmax,
                           std::max(1, blocks / P1.units), max_cluster);
        // Several clusters per unit, each merging on chip, leave the workspace only their
        // first CTAs' partials. Where the plain merge would gather many partials that pays
        // even with more tiles per block (measured: 1 row x 4 KV heads over 32768
        // positions, 64 plain splits 17.1 us, 3 clusters of 16 per head 14.1 us; with 37
        // plain splits, 2 clusters per head lost, 18.9 -> 20.1 us): taken with the most
        // clusters per unit that are all resident at once.
        if (kern_g && W.splits >= kGroupedMinSplits && max_cluster >= 2) {
            const int most = std::min(kMaxGroups, (P1.rounds + max_cluster - 1) / max_cluster);
            for (int g = most; g >= 2; --g) {
                const AttnPlan G = plan_grouped(batch, n_q_heads, n_kv_heads, rows_per_kv,
                                                qlen, len_bound, mmax, g, max_cluster);
                const int cs = G.splits / G.cgroups;
                if (cs >= 2 &&
                    resident(kern_g, kid_g, plan_smem(G, var, app_rows), cs, nsm) >= G.units * g)
                    return G;
            }
        }
        return W;
    }
    int last = 0;
    for (int s = std::min(P1.rounds, max_cluster); s >= 2; --s) {
        const AttnPlan P = plan_attention(batch, n_q_heads, n_kv_heads, rows_per_kv, qlen,
                                          len_bound, mmax, s, max_cluster);
        if (P.splits == last) continue;
        last = P.splits;
        if (P.splits < 2) break;
        if (P.cluster && resident(kern, kid, plan_smem(P, var, app_rows), P.splits, nsm) >= P.units)
            return P;
    }
    return P1;
}

kvd_status attention(bool verify, kvd_dtype dtype, int32_t batch, int32_t n_q_heads,
                     int32_t qlen, const void* q, const kvd_cache* kv, const int32_t* lens,
                     int32_t fixed_len, const kvd_new_tokens* app, int32_t rows_per_kv,
                     int32_t causal, float scale, void* out, void* ws, size_t ws_bytes,
                     uint32_t flags, int32_t* dev_err, cudaStream_t stream,
                     bool noalloc = false) {
    if (dtype != KVD_F16 && dtype != KVD_BF16) return KVD_ERR_INVALID_ARG;
    if (kvd_status s = validate_cache(kv)) return s;
    if (batch < 0 || n_q_heads <= 0 || rows_per_kv <= 0) return KVD_ERR_INVALID_ARG;
    if (qlen < 1 || qlen > KVD_MAX_QLEN) return KVD_ERR_UNSUPPORTED;
    if (n_q_heads % kv->n_kv_heads || batch % rows_per_kv) return KVD_ERR_INVALID_ARG;
    if (batch == 0) return KVD_OK;
    if (!q || !out || !aligned16(q) || !aligned16(out)) return KVD_ERR_INVALID_ARG;
    if (batch / rows_per_kv > kv->batch || batch / rows_per_kv > 65535) return KVD_ERR_INVALID_ARG;
    if (!lens && (fixed_len < 0 || fixed_len > kv->capacity)) return KVD_ERR_INVALID_ARG;
    if (app) {
        if (!lens || !app->k_new || !app->v_new || !aligned16(app->k_new) ||
            !aligned16(app->v_new) || app->lens_out == lens)
            return KVD_ERR_INVALID_ARG;
        if (!(app->rope_base >= 0.f) || !(app->rope_base < INFINITY)) return KVD_ERR_INVALID_ARG;
    }
    const bool rope = app && app->rope_base > 0.f;
    if (!(scale == scale)) return KVD_ERR_INVALID_ARG;
    const int nsm = sm_count();
    if (nsm <= 0) return KVD_ERR_CUDA;
    if (noalloc) {  // the built-in scratch stands in for the workspace
        if (kvd_status s = noalloc_scratch(&ws)) return s;
        ws_bytes = KVD_NOALLOC_SCRATCH_BYTES;
    }
    const int len_bound = lens ? kv->capacity : fixed_len;
    const bool bf = dtype == KVD_BF16;
    const int group = n_q_heads / kv->n_kv_heads;
    const int app_rows = app_units(app ? 1 : 0, rope ? 1 : 0, qlen);
    // Plan for one kernel variant; false if it cannot be prepared.
    auto plan_for = [&](int var, AttnPlan& out) -> bool {
        const int mc = bf ? prepare<__nv_bfloat16>(var) : prepare<__half>(var);
        if (mc <= 0) return false;
        const void* kern = bf ? kernel_of<__nv_bfloat16>(var) : kernel_of<__half>(var);
        // the build with the merge across clusters, for the variants that have one
        const int gvar = var == kSimt ? kSimtG : var == kMma ? kMmaG : 0;
        const void* kern_g = nullptr;
        if (gvar && (bf ? prepare<__nv_bfloat16>(gvar) : prepare<__half>(gvar)) == mc)
            kern_g = bf ? kernel_of<__nv_bfloat16>(gvar) : kernel_of<__half>(gvar);
        out = choose_plan(kern, var * 2 + (bf ? 1 : 0), var, nsm, batch, n_q_heads,
                          kv->n_kv_heads, rows_per_kv, qlen, len_bound, mc, app_rows, kern_g,
                          gvar * 2 + (bf ? 1 : 0));
        return true;
    };
    // Whether a tensor-core plan keeps all its blocks resident at once.
    auto one_wave = [&](int var, const AttnPlan& Q) -> bool {
        if (Q.cluster) return true;  // choose_plan checked the clusters' residency
        if (Q.splits != 1) return false;
        const void* kern = bf ? kernel_of<__nv_bfloat16>(var) : kernel_of<__half>(var);
        return (int64_t)Q.units <=
               resident(kern, var * 2 + (bf ? 1 : 0), plan_smem(Q, var, app_rows), 1, nsm);
    };
    // the builds with the rotation compiled in stand for kSimt and kMma when it is on
    const int simt = rope ? kSimtRope : kSimt, mma = rope ? kMmaRope : kMma;
    int var = (verify || (int64_t)rows_per_kv * group * qlen >= 2) ? mma : simt;
    AttnPlan P;
    if (!plan_for(var, P)) return KVD_ERR_CUDA;
    if (var == simt && P.tiles_per_split <= 2) {
        // Each block has a single round of tiles: then the time is the chain after the
        // dependency wait, and the tensor-core kernel's per-tile chain (ldmatrix + mma,
        // two shuffles) is shorter than the CUDA-core one (a shuffle tree per position).
        // Measured for 20 heads: 3.70 vs 4.47 us over 1500 frames, 3.02 vs 3.31 us at 448
        // positions with the append. It has half the resident blocks per SM, so it is
        // taken only while its launch still fits in one wave.
        AttnPlan P2;
        if (plan_for(mma, P2) && one_wave(mma, P2) && P2.tiles_per_split <= 2) {
            var = mma;
            P = P2;
        }
    }
    if (var == kMma && P.tiles_per_split >= 8) {
        // Residency limits the split count and blocks stream 4 or more rounds: a build
        // with 3 blocks per SM allows more splits. For blocks of at most 8 query vectors
        // that is the 8-vector build (no spill); otherwise the full build cut to 80
        // registers, whose rounds are slower (spills). Either is taken only when it at
        // least halves every block's tiles. Measured: beam cross attention (160 units over
        // 1500 frames) 16.0 -> 13.2 us with the cut full build, and the beam step 1211 ->
        // 1159 us with the 8-vector build instead; with a smaller cut (GQA-LM: 8 -> 6
        // tiles per block) it lost, 6.9 -> 8.1 us per layer. Three blocks per SM do not
        // pay for launches that are latency chains: packed more densely, the blocks of
        // one launch slow one another (Whisper step 0.441 -> 0.492 ms with the 8-vector
        // build used for every launch of at most 8 vectors).
        const int v3 = (int64_t)P.msub <= 8 ? kMma8 : kMma3;
        AttnPlan P3;
        if (plan_for(v3, P3) && one_wave(v3, P3) && 2 * P3.tiles_per_split <= P.tiles_per_split) {
            var = v3;
            P = P3;
        }
    }
    // several clusters per unit run on the build with the merge across clusters (only
    // kSimt and kMma plans have them)
    if (P.cgroups > 1) var = var == kSimt ? kSimtG : kMmaG;
    // Few blocks, each streaming more tiles than the ring holds: when every block can
    // have an SM of its own, a ring as deep as the block's tiles stages all of them
    // before the dependency wait (kept only if the clusters all stay resident).
    if (P.cluster && P.cgroups == 1 && P.tiles_per_split > P.stages &&
        P.tiles_per_split <= kMaxStages && (int64_t)P.units * P.splits <= nsm) {
        AttnPlan D = P;
        D.stages = P.tiles_per_split;
        const void* kern = bf ? kernel_of<__nv_bfloat16>(var) : kernel_of<__half>(var);
        if (resident(kern, var * 2 + (bf ? 1 : 0), plan_smem(D, var, app_rows), D.splits, nsm) >=
            D.units)
            P = D;
    }
    if ((int64_t)kv->n_kv_heads * P.nsub > 65535) return KVD_ERR_UNSUPPORTED;
    const bool ws_merge = (P.splits > 1 && !P.cluster) || P.cgroups > 1;
    if (ws_merge) {
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
    p.cgroups = P.cgroups;
    p.csize = P.splits / P.cgroups;
    p.test_stall = (flags & KVD_FLAG_TEST_STALL) ? 1 : 0;
    p.merge_wait_ns = merge_wait_budget(P.tiles_per_split, p.stages);
    p.append = app ? 1 : 0;
    p.rope = rope ? 1 : 0;
    p.rope_log2_base = rope ? log2f(app->rope_base) : 0.f;
    p.k_new = app ? static_cast<const uint8_t*>(app->k_new) : nullptr;
    p.v_new = app ? static_cast<const uint8_t*>(app->v_new) : nullptr;
    p.lens_out = app ? app->lens_out : nullptr;
    p.kc = static_cast<uint8_t*>(kv->k);
    p.vc = static_cast<uint8_t*>(kv->v);
    p.sb = kv->stride_b * 2;
    p.sh = kv->stride_h * 2;
    p.st = kv->stride_t * 2;
    p.n_kv_heads = kv->n_kv_heads;
    p.scale_log2 = scale * kLog2e;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    p.ws_cnt = reinterpret_cast<int32_t*>(wsb);
    p.ws_part = wsb ? reinterpret_cast<float*>(wsb + P.part_offset) : nullptr;
    p.ws_ml = wsb ? reinterpret_cast<float2*>(wsb + P.ml_offset) : nullptr;
    p.dev_err = dev_err;

    // The built-in scratch keeps whatever the previous call left; a plan that merges
    // through it needs its units' arrival counters at zero (a call that stopped early
    // could have left them non-zero). Cleared here, after every check has passed.
    if (noalloc && ws_merge &&
        cudaMemsetAsync(ws, 0, (size_t)P.units * sizeof(int32_t), stream) != cudaSuccess)
        return KVD_ERR_CUDA;
    const bool pdl = (flags & (KVD_FLAG_PDL | KVD_FLAG_EARLY_KV)) != 0;
    const dim3 grid(P.splits, kv->n_kv_heads * P.nsub, P.bkv);
    const unsigned cl = P.cluster ? (unsigned)(P.splits / P.cgroups) : 1u;
    return bf ? launch_attn<__nv_bfloat16>(var, grid, stream, pdl, cl, mk, mv, p)
              : launch_attn<__half>(var, grid, stream, pdl, cl, mk, mv, p);
}

}  // namespace
}  // namespace kvd

extern "C" kvd_status kvd_decode_attn(kvd_dtype dtype, int32_t batch, int32_t n_q_heads,
                                      const void* q, const kvd_cache* kv, const int32_t* lens,
                                      int32_t fixed_len, const kvd_new_tokens* append,
                                      int32_t rows_per_kv, float scale, void* out,
                                      void* workspace, size_t workspace_bytes, uint32_t flags,
                                      int32_t* dev_err, kvd_stream_t stream) {
    return kvd::attention(false, dtype, batch, n_q_heads, 1, q, kv, lens, fixed_len, append,
                          rows_per_kv, 0, scale, out, workspace, workspace_bytes, flags, dev_err,
                          reinterpret_cast<cudaStream_t>(stream));
}

extern "C" kvd_status kvd_verify_attn(kvd_dtype dtype, int32_t batch, int32_t n_q_heads,
                                      int32_t qlen, const void* q, const kvd_cache* kv,
                                      const int32_t* lens, int32_t fixed_len,
                                      const kvd_new_tokens* append, int32_t rows_per_kv,
                                      int32_t causal, float scale, void* out, void* workspace,
                                      size_t workspace_bytes, uint32_t flags, int32_t* dev_err,
                                      kvd_stream_t stream) {
    return kvd::attention(true, dtype, batch, n_q_heads, qlen, q, kv, lens, fixed_len, append,
                          rows_per_kv, causal, scale, out, workspace, workspace_bytes, flags,
                          dev_err, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- no-allocation entry
// kvd_decode_attn_noalloc: the decode kernels with their split-merge scratch in the
// buffer compiled into the library, for callers that cannot allocate a workspace (see
// kvdecode.h). Every host check and the plan come first; the scratch's arrival counters
// are cleared only for a plan that merges through them, right before the launch.
extern "C" kvd_status kvd_decode_attn_noalloc(kvd_dtype dtype, int32_t batch, int32_t n_q_heads,
                                              const void* q, const kvd_cache* kv,
                                              const int32_t* lens, int32_t fixed_len,
                                              const kvd_new_tokens* append, int32_t rows_per_kv,
                                              float scale, void* out, uint32_t flags,
                                              int32_t* dev_err, kvd_stream_t stream) {
    return kvd::attention(false, dtype, batch, n_q_heads, 1, q, kv, lens, fixed_len, append,
                          rows_per_kv, 0, scale, out, nullptr, 0, flags, dev_err,
                          reinterpret_cast<cudaStream_t>(stream), /*noalloc=*/true);
}

// Test support: overwrite the built-in scratch's arrival counters on `stream`, as a call
// that stopped early (a timed-out wait) could leave them.
extern "C" kvd_status kvd_noalloc_test_fill_counters(uint8_t byte_value, kvd_stream_t stream) {
    void* scratch = nullptr;
    if (kvd_status s = kvd::noalloc_scratch(&scratch)) return s;
    return cudaMemsetAsync(scratch, byte_value, KVD_WS_COUNTER_BYTES,
                           reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KVD_OK
               : KVD_ERR_CUDA;
}
