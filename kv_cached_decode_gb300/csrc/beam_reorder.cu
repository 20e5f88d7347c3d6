// beam_reorder.cu -- reorder every layer's self-attention K/V by beam parent.
//
// BeamSearchDecoder.update and rearrange_kv_cache in "Inference 抽象と KV キャッシュ" of
// "Whisper のデコーダー内部：Beam Search、Logit フィルター、KV キャッシュ": once the beams are
// re-ranked, the cached key/value tensors are put in the new beam order so that no
// beam continues another beam's cache.
//
// Design: one launch covers all layers, K and V. A thread block owns one (layer, K or
// V, window, head, tile of 64 positions) and every thread owns fixed 16-byte chunks of
// that tile; it first loads the chunk of every row that is a parent of a moving row,
// then writes the moving rows. Reads of one window/tile never race with writes of
// another block, and each chunk is read before it is overwritten by the same thread,
// so the reorder is done in place without scratch memory even when a beam has several
// children or parents form cycles. Rows that keep their own cache are never touched;
// a source is read once however many children it has.
#include <algorithm>
#include <mutex>

#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {

struct BeamLayer {
    uint8_t* k;
    uint8_t* v;
    int64_t sb, sh, st;  // bytes
    int32_t capacity;
    int32_t pad;
};

struct BeamParams {
    BeamLayer layer[KVD_MAX_LAYERS_PER_CALL];
    const int32_t* parent;
    const int32_t* lens;
    int32_t* dev_err;
    int32_t n_layers, beam, windows, heads, pos_tiles, fixed_len;
};

constexpr int kBeamThreads = 256;
constexpr int kChunksPerTile = kTile * 8;  // 64 positions x 8 chunks of 16 bytes

// One block's share: (layer, K or V, window, head, 64-position tile), decoded from the
// block index, and the window's parents. moved: rows that take another row's cache;
// needed: rows that are read as parents; len_max: longest moved row. Bad parents and
// lengths are flagged (once per launch) and leave their row untouched.
struct BeamItem {
    int pt, h, w, is_v, l, row0, len_max;
    unsigned moved, needed;
    int par[KVD_MAX_BEAM], len[KVD_MAX_BEAM];
};

// tiles: position tiles per block index (1 when a block walks all tiles itself).
__device__ __forceinline__ void beam_item(const BeamParams& p, int tiles, BeamItem& it) {
    int64_t item = blockIdx.x;
    it.pt = (int)(item % tiles);
    item /= tiles;
    it.h = (int)(item % p.heads);
    item /= p.heads;
    it.w = (int)(item % p.windows);
    item /= p.windows;
    it.is_v = (int)(item & 1);
    it.l = (int)(item >> 1);
    const BeamLayer& L = p.layer[it.l];
    const bool reporter = it.pt == 0 && it.h == 0 && it.is_v == 0 && it.l == 0 && threadIdx.x == 0;
    it.moved = it.needed = 0;
    it.len_max = 0;
    it.row0 = it.w * p.beam;
#pragma unroll
    for (int j = 0; j < KVD_MAX_BEAM; ++j) {
        it.par[j] = j;
        it.len[j] = 0;
        if (j < p.beam) {
            const int pr = p.parent[it.row0 + j] - it.row0;
            const int ln = p.lens ? p.lens[it.row0 + j] : p.fixed_len;
            const bool ok_p = pr >= 0 && pr < p.beam;
            const bool ok_l = ln >= 0 && ln <= L.capacity;
            if (!ok_p && reporter) flag_error(p.dev_err, KVD_ERR_BAD_INDEX);
            if (!ok_l && reporter) flag_error(p.dev_err, KVD_ERR_LEN_OVERFLOW);
            if (ok_p && ok_l && pr != j) {
                it.par[j] = pr;
                it.len[j] = ln;
                it.moved |= 1u << j;
                it.needed |= 1u << pr;
                it.len_max = max(it.len_max, ln);
            }
        }
    }
}

__global__ void __launch_bounds__(kBeamThreads)
    beam_reorder_kernel(const __grid_constant__ BeamParams p) {
    pdl_wait();
    BeamItem it;
    beam_item(p, p.pos_tiles, it);
    const BeamLayer& L = p.layer[it.l];
    const int pt = it.pt, h = it.h, is_v = it.is_v, row0 = it.row0, len_max = it.len_max;
    const unsigned moved = it.moved, needed = it.needed;
    const int* par = it.par;
    const int* len = it.len;
    const int t0 = pt * kTile;
    if (moved && t0 < len_max) {
        uint8_t* base = (is_v ? L.v : L.k) + h * L.sh;
        for (int x = threadIdx.x; x < kChunksPerTile; x += kBeamThreads) {
            const int t = t0 + (x >> 3);
            if (t >= len_max) break;
            const int64_t off = (int64_t)t * L.st + (x & 7) * 16;
            uint4 val[KVD_MAX_BEAM];
#pragma unroll
            for (int j = 0; j < KVD_MAX_BEAM; ++j)
                if (needed >> j & 1)
                    val[j] = *reinterpret_cast<const uint4*>(base + (row0 + j) * L.sb + off);
#pragma unroll
            for (int j = 0; j < KVD_MAX_BEAM; ++j) {
                if ((moved >> j & 1) && t < len[j]) {
                    uint4 v = val[0];
#pragma unroll
                    for (int s = 1; s < KVD_MAX_BEAM; ++s)
                        if (par[j] == s) v = val[s];
                    *reinterpret_cast<uint4*>(base + (row0 + j) * L.sb + off) = v;
                }
            }
        }
    }
    pdl_trigger();
}

// ---- bulk-copy path, for caches whose positions are contiguous 128-byte rows ----------
// The (window, head) region of every row is then one contiguous span per 64-position
// tile, so a single thread moves it with bulk asynchronous copies. A block owns (layer,
// K or V, window, head) and walks the tiles up to the longest moving row: every needed
// parent span of a tile is copied into shared memory (completing on one mbarrier), and
// once all have arrived each moving row's span is copied back out from its parent's
// copy. Loads of a tile finish before any of its stores, as in the per-thread path, so
// the reorder stays in place; tiles of one block touch disjoint rows' spans.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(src), "r"(bytes)
                 : "memory");
}
// the stores are complete
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

constexpr int kBulkThreads = 32;
constexpr int kBulkSmem = KVD_MAX_BEAM * kTileBytes + 16;  // parent spans, mbarrier

__global__ void __launch_bounds__(kBulkThreads)
    beam_reorder_bulk_kernel(const __grid_constant__ BeamParams p) {
    extern __shared__ __align__(128) uint8_t sm[];
    pdl_wait();
    BeamItem it;
    beam_item(p, 1, it);
    if (threadIdx.x == 0 && it.moved) {
        const BeamLayer& L = p.layer[it.l];
        uint8_t* head = (it.is_v ? L.v : L.k) + it.h * L.sh;
        const uint32_t bar = smem_u32(sm + KVD_MAX_BEAM * kTileBytes);
        mbar_init(bar, 1);
        fence_barrier_init();
        const int n_needed = __popc(it.needed);
        for (int t0 = 0, phase = 0; t0 < it.len_max; t0 += kTile, phase ^= 1) {
            uint8_t* base = head + (int64_t)t0 * kRowBytes;
            const uint32_t bytes = (uint32_t)(min(it.len_max, t0 + kTile) - t0) * kRowBytes;
            mbar_expect_tx(bar, bytes * n_needed);
            for (int j = 0; j < p.beam; ++j)
                if (it.needed >> j & 1)
                    bulk_load(smem_u32(sm + j * kTileBytes), base + (it.row0 + j) * L.sb,
                              bytes, bar);
            if (!mbar_wait_bounded(bar, phase)) {
                flag_error(p.dev_err, KVD_ERR_TIMEOUT);
                // Let copies in flight land before the block exits, for at most another
                // second. If that wait runs out too, the block still exits (the error is
                // already flagged): a copy that has not landed in two seconds is not
                // waited for without bound, and could then write into shared memory the
                // next block on this SM receives.
                const bool drained = mbar_wait_bounded(bar, phase);
                (void)drained;
                break;
            }
            fence_proxy_async();
            for (int j = 0; j < p.beam; ++j) {
                const int rows = min(it.len[j], t0 + kTile) - t0;
                if ((it.moved >> j & 1) && rows > 0)
                    bulk_store(base + (it.row0 + j) * L.sb,
                               smem_u32(sm + it.par[j] * kTileBytes), (uint32_t)rows * kRowBytes);
            }
            bulk_commit();
            bulk_wait_read();  // before the next tile refills shared memory
        }
        bulk_wait_all();
    }
    pdl_trigger();
}

}  // namespace kvd

using namespace kvd;

namespace {
constexpr int kMaxDev = 64;
}

extern "C" kvd_status kvd_beam_reorder_kv(kvd_dtype dtype, const kvd_cache* layers,
                                          int32_t n_layers, int32_t rows, int32_t beam,
                                          const int32_t* parent, const int32_t* lens,
                                          int32_t fixed_len, uint32_t flags, int32_t* dev_err,
                                          kvd_stream_t stream) {
    if (dtype != KVD_F16 && dtype != KVD_BF16) return KVD_ERR_INVALID_ARG;
    if (n_layers < 0 || rows < 0 || beam <= 0) return KVD_ERR_INVALID_ARG;
    if (n_layers > KVD_MAX_LAYERS_PER_CALL || beam > KVD_MAX_BEAM) return KVD_ERR_UNSUPPORTED;
    if (rows % beam) return KVD_ERR_INVALID_ARG;
    if (n_layers == 0 || rows == 0) return KVD_OK;
    if (!layers || !parent) return KVD_ERR_INVALID_ARG;
    BeamParams p;
    int cap_max = 0;
    bool rows_contiguous = true;  // every layer's positions are adjacent 128-byte rows
    for (int l = 0; l < n_layers; ++l) {
        const kvd_cache* c = &layers[l];
        if (kvd_status s = validate_cache(c)) return s;
        if (c->batch < rows || c->n_kv_heads != layers[0].n_kv_heads) return KVD_ERR_INVALID_ARG;
        p.layer[l].k = static_cast<uint8_t*>(c->k);
        p.layer[l].v = static_cast<uint8_t*>(c->v);
        p.layer[l].sb = c->stride_b * 2;
        p.layer[l].sh = c->stride_h * 2;
        p.layer[l].st = c->stride_t * 2;
        p.layer[l].capacity = c->capacity;
        rows_contiguous = rows_contiguous && c->stride_t == KVD_HEAD_DIM;
        p.layer[l].pad = 0;
        cap_max = std::max(cap_max, c->capacity);
    }
    if (!lens && fixed_len < 0) return KVD_ERR_INVALID_ARG;
    const int bound = lens ? cap_max : std::min(fixed_len, cap_max);
    p.parent = parent;
    p.lens = lens;
    p.dev_err = dev_err;
    p.n_layers = n_layers;
    p.beam = beam;
    p.windows = rows / beam;
    p.heads = layers[0].n_kv_heads;
    p.pos_tiles = std::max(1, (bound + kTile - 1) / kTile);
    p.fixed_len = fixed_len;
    const int64_t blocks = (int64_t)n_layers * 2 * p.windows * p.heads * p.pos_tiles;
    if (blocks > 0x7fffffff) return KVD_ERR_UNSUPPORTED;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const bool pdl = (flags & KVD_FLAG_PDL) != 0;
    if (rows_contiguous) {
        static std::once_flag once[kMaxDev];
        static bool ok[kMaxDev];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return KVD_ERR_CUDA;
        std::call_once(once[dev], [dev] {
            ok[dev] = cudaFuncSetAttribute(beam_reorder_bulk_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kBulkSmem) == cudaSuccess;
            cudaGetLastError();
        });
        if (!ok[dev]) return KVD_ERR_CUDA;
        return launch(beam_reorder_bulk_kernel, dim3((unsigned)(blocks / p.pos_tiles)),
                      dim3(kBulkThreads), kBulkSmem, st, pdl, p);
    }
    return launch(beam_reorder_kernel, dim3((unsigned)blocks), dim3(kBeamThreads), 0, st, pdl,
                  p);
}
