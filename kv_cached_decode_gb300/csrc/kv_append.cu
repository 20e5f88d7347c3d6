// kv_append.cu -- write the new tokens' K/V into the preallocated cache.
//
// "KV キャッシュが推論を最適化する方法" (steps 2-3) of "nanoVLM における KV キャッシュ実装":
// only the newest token's K/V are computed and added to the stored cache; "Inference 抽象
// と KV キャッシュ" of "Whisper のデコーダー内部": they are concatenated along the sequence
// axis. With a preallocated [batch, heads, capacity, 64] cache this is an O(q) write of
// 16-byte chunks; nothing already cached moves.
#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {

struct AppendParams {
    uint8_t* k;
    uint8_t* v;
    int64_t sb, sh, st;  // bytes
    const uint8_t* k_new;
    const uint8_t* v_new;
    const int32_t* lens_in;   // NULL: every row starts empty
    const int32_t* counts;    // NULL: q rows for every batch row; else rows for row b
    int32_t* lens_out;
    int32_t* dev_err;
    int32_t capacity, heads, q;
    int64_t chunks;  // 16-byte chunks per tensor: batch * heads * q * 8
    float rope_log2_base;  // the rotary variant only
};

__global__ void __launch_bounds__(256) kv_append_kernel(const AppendParams p) {
    pdl_wait();
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx < 2 * p.chunks) {
        const bool is_v = idx >= p.chunks;
        const int64_t rem = is_v ? idx - p.chunks : idx;
        const int c = (int)(rem & 7);
        const int64_t row = rem >> 3;  // (b, h, j)
        const int j = (int)(row % p.q);
        const int64_t bh = row / p.q;
        const int h = (int)(bh % p.heads);
        const int b = (int)(bh / p.heads);
        const int len = p.lens_in ? p.lens_in[b] : 0;
        const int n = p.counts ? p.counts[b] : p.q;
        const bool first = !is_v && h == 0 && j == 0 && c == 0;
        if (len < 0 || n < 0 || n > p.q || (int64_t)len + n > p.capacity) {
            if (first) {
                flag_error(p.dev_err, KVD_ERR_LEN_OVERFLOW);
                if (p.lens_out) p.lens_out[b] = len;
            }
        } else if (j < n) {
            const uint4 val = *reinterpret_cast<const uint4*>((is_v ? p.v_new : p.k_new) + rem * 16);
            uint8_t* dst = (is_v ? p.v : p.k) + b * p.sb + h * p.sh + (int64_t)(len + j) * p.st + c * 16;
            *reinterpret_cast<uint4*>(dst) = val;
            if (first && p.lens_out) p.lens_out[b] = len + n;
        } else if (first && p.lens_out) {
            p.lens_out[b] = len;  // n == 0
        }
    }
    pdl_trigger();
}

// With rotary encoding of the keys ("nanoVLM における KV キャッシュ実装": the new tokens
// are encoded at their absolute positions, start_pos = the cached length): a K item is a
// pair of chunks (c, c + 4), i.e. the two halves of 8 rotation pairs of row j, rotated
// at position len + j; V chunks are copied as they are.
template <typename T>
__global__ void __launch_bounds__(256) kv_append_rope_kernel(const AppendParams p) {
    pdl_wait();
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t k_items = p.chunks / 2;
    if (idx < k_items + p.chunks) {
        const bool is_v = idx >= k_items;
        const int64_t rem = is_v ? idx - k_items : idx;
        const int c = is_v ? (int)(rem & 7) : (int)(rem & 3);
        const int64_t row = is_v ? rem >> 3 : rem >> 2;  // (b, h, j)
        const int j = (int)(row % p.q);
        const int64_t bh = row / p.q;
        const int h = (int)(bh % p.heads);
        const int b = (int)(bh / p.heads);
        const int len = p.lens_in ? p.lens_in[b] : 0;
        const int n = p.counts ? p.counts[b] : p.q;
        const bool first = !is_v && h == 0 && j == 0 && c == 0;
        if (len < 0 || n < 0 || n > p.q || (int64_t)len + n > p.capacity) {
            if (first) {
                flag_error(p.dev_err, KVD_ERR_LEN_OVERFLOW);
                if (p.lens_out) p.lens_out[b] = len;
            }
        } else if (j < n) {
            uint8_t* dst = (is_v ? p.v : p.k) + b * p.sb + h * p.sh + (int64_t)(len + j) * p.st;
            if (is_v) {
                *reinterpret_cast<uint4*>(dst + c * 16) =
                    *reinterpret_cast<const uint4*>(p.v_new + rem * 16);
            } else {
                const uint8_t* src = p.k_new + row * kRowBytes;
                uint4 lo = *reinterpret_cast<const uint4*>(src + c * 16);
                uint4 hi = *reinterpret_cast<const uint4*>(src + (c + 4) * 16);
                rope_rotate8_at<T>(lo, hi, len + j, c * 8, p.rope_log2_base);
                *reinterpret_cast<uint4*>(dst + c * 16) = lo;
                *reinterpret_cast<uint4*>(dst + (c + 4) * 16) = hi;
            }
            if (first && p.lens_out) p.lens_out[b] = len + n;
        } else if (first && p.lens_out) {
            p.lens_out[b] = len;  // n == 0
        }
    }
    pdl_trigger();
}

}  // namespace kvd

using namespace kvd;

namespace kvd {
// Shared by kvd_kv_append(_rope) and the prefill: arguments already validated.
kvd_status launch_append(const kvd_cache* cache, int32_t batch, int32_t q, const void* k_new,
                         const void* v_new, const int32_t* lens_in, const int32_t* counts,
                         int32_t* lens_out, kvd_dtype dtype, float rope_base, uint32_t flags,
                         int32_t* dev_err, cudaStream_t stream) {
    AppendParams p;
    p.k = static_cast<uint8_t*>(cache->k);
    p.v = static_cast<uint8_t*>(cache->v);
    p.sb = cache->stride_b * 2;
    p.sh = cache->stride_h * 2;
    p.st = cache->stride_t * 2;
    p.k_new = static_cast<const uint8_t*>(k_new);
    p.v_new = static_cast<const uint8_t*>(v_new);
    p.lens_in = lens_in;
    p.counts = counts;
    p.lens_out = lens_out;
    p.dev_err = dev_err;
    p.capacity = cache->capacity;
    p.heads = cache->n_kv_heads;
    p.q = q;
    p.chunks = (int64_t)batch * cache->n_kv_heads * q * 8;
    const bool pdl = (flags & KVD_FLAG_PDL) != 0;
    if (rope_base > 0.f) {
        p.rope_log2_base = log2f(rope_base);
        const int64_t blocks = (p.chunks / 2 + p.chunks + 255) / 256;
        if (blocks > 0x7fffffff) return KVD_ERR_UNSUPPORTED;
        if (dtype == KVD_BF16)
            return launch(kv_append_rope_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256),
                          0, stream, pdl, p);
        return launch(kv_append_rope_kernel<__half>, dim3((unsigned)blocks), dim3(256), 0,
                      stream, pdl, p);
    }
    p.rope_log2_base = 0.f;
    const int64_t blocks = (2 * p.chunks + 255) / 256;
    if (blocks > 0x7fffffff) return KVD_ERR_UNSUPPORTED;
    return launch(kv_append_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, pdl, p);
}
}  // namespace kvd

namespace {
kvd_status append_entry(kvd_dtype dtype, const kvd_cache* cache, int32_t batch, int32_t q,
                        const void* k_new, const void* v_new, const int32_t* lens_in,
                        int32_t* lens_out, float rope_base, uint32_t flags, int32_t* dev_err,
                        kvd_stream_t stream) {
    if (dtype != KVD_F16 && dtype != KVD_BF16) return KVD_ERR_INVALID_ARG;
    if (kvd_status s = validate_cache(cache)) return s;
    if (batch < 0 || q < 0 || batch > cache->batch) return KVD_ERR_INVALID_ARG;
    if (!(rope_base >= 0.f) || !(rope_base < INFINITY)) return KVD_ERR_INVALID_ARG;
    if (batch == 0 || q == 0) return KVD_OK;
    if (!k_new || !v_new || !lens_in || !aligned16(k_new) || !aligned16(v_new))
        return KVD_ERR_INVALID_ARG;
    if (lens_out && lens_out == lens_in) return KVD_ERR_INVALID_ARG;
    return launch_append(cache, batch, q, k_new, v_new, lens_in, nullptr, lens_out, dtype,
                         rope_base, flags, dev_err, reinterpret_cast<cudaStream_t>(stream));
}
}  // namespace

extern "C" kvd_status kvd_kv_append(kvd_dtype dtype, const kvd_cache* cache, int32_t batch,
                                    int32_t q, const void* k_new, const void* v_new,
                                    const int32_t* lens_in, int32_t* lens_out, uint32_t flags,
                                    int32_t* dev_err, kvd_stream_t stream) {
    return append_entry(dtype, cache, batch, q, k_new, v_new, lens_in, lens_out, 0.f, flags,
                        dev_err, stream);
}

extern "C" kvd_status kvd_kv_append_rope(kvd_dtype dtype, const kvd_cache* cache, int32_t batch,
                                         int32_t q, const void* k_new, const void* v_new,
                                         const int32_t* lens_in, int32_t* lens_out,
                                         float rope_base, uint32_t flags, int32_t* dev_err,
                                         kvd_stream_t stream) {
    if (!(rope_base > 0.f)) return KVD_ERR_INVALID_ARG;
    return append_entry(dtype, cache, batch, q, k_new, v_new, lens_in, lens_out, rope_base,
                        flags, dev_err, stream);
}
