// beam_reorder.cu -- A7: reorder every layer's self-attention K/V by beam parent.
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

__global__ void __launch_bounds__(kBeamThreads)
    beam_reorder_kernel(const __grid_constant__ BeamParams p) {
    pdl_wait();
    int64_t item = blockIdx.x;
    const int pt = (int)(item % p.pos_tiles);
    item /= p.pos_tiles;
    const int h = (int)(item % p.heads);
    item /= p.heads;
    const int w = (int)(item % p.windows);
    item /= p.windows;
    const int is_v = (int)(item & 1);
    const int l = (int)(item >> 1);
    const BeamLayer& L = p.layer[l];
    const bool reporter = pt == 0 && h == 0 && is_v == 0 && l == 0 && threadIdx.x == 0;

    // Parents and lengths of this window's rows.
    int par[KVD_MAX_BEAM], len[KVD_MAX_BEAM];
    unsigned moved = 0, needed = 0;
    int len_max = 0;
    const int row0 = w * p.beam;
#pragma unroll
    for (int j = 0; j < KVD_MAX_BEAM; ++j) {
        par[j] = j;
        len[j] = 0;
        if (j < p.beam) {
            const int pr = p.parent[row0 + j] - row0;
            const int ln = p.lens ? p.lens[row0 + j] : p.fixed_len;
            const bool ok_p = pr >= 0 && pr < p.beam;
            const bool ok_l = ln >= 0 && ln <= L.capacity;
            if (!ok_p && reporter) flag_error(p.dev_err, KVD_ERR_BAD_INDEX);
            if (!ok_l && reporter) flag_error(p.dev_err, KVD_ERR_LEN_OVERFLOW);
            if (ok_p && ok_l && pr != j) {
                par[j] = pr;
                len[j] = ln;
                moved |= 1u << j;
                needed |= 1u << pr;
                len_max = max(len_max, ln);
            }
        }
    }
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

}  // namespace kvd

using namespace kvd;

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
    return launch(beam_reorder_kernel, dim3((unsigned)blocks), dim3(kBeamThreads), 0,
                  reinterpret_cast<cudaStream_t>(stream), (flags & KVD_FLAG_PDL) != 0, p);
}
