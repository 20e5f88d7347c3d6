// rope.cu -- rotary position encoding at absolute positions.
//
// "nanoVLM における KV キャッシュ実装" (the LanguageModel passes start_pos so that the
// rotary encoding of the new tokens matches their absolute positions). Rotate-half form:
// for i < 32, theta_i = base^(-i/32), a = pos * theta_i,
//   y[i] = x[i] cos a - x[i+32] sin a,   y[i+32] = x[i+32] cos a + x[i] sin a,
// with token j of row b at pos0[b] + j. Applied in place to the queries and the new
// keys of a step before they reach kv_append / decode_attn / verify_attn / prefill.
//
// Design: one thread per 8 rotation pairs (16-byte loads of x[i..i+7] and
// x[i+32..i+39]); both tensors in one launch. The rotation itself (rope_cos_sin,
// rope_rotate) is shared with the attention kernel, which can apply it to the queries
// and the appended keys of a call instead of this launch, with the same bits: angle in
// fp32, sin/cos from sincosf (full argument reduction, accurate for positions in the
// thousands), the result rounded to the storage type.
#include <algorithm>

#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {
namespace {

struct RopeParams {
    uint8_t* x[2];       // q, k (either may be null)
    int32_t heads[2];
    const int32_t* pos0;  // [batch] or null
    int32_t batch, n;
    float log2_base;
    int64_t items[2];    // 16-byte items per tensor: batch * heads * n * 4
};

template <typename T>
__global__ void __launch_bounds__(256) rope_kernel(const RopeParams p) {
    pdl_wait();
    int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int which = idx < p.items[0] ? 0 : 1;
    if (which == 1) idx -= p.items[0];
    if (idx < p.items[which]) {
        const int g = (int)(idx & 3);  // pairs 8g .. 8g+7
        const int64_t row = idx >> 2;  // (b, h, j)
        const int j = (int)(row % p.n);
        const int b = (int)(row / p.n / p.heads[which]);
        const int pos = (p.pos0 ? p.pos0[b] : 0) + j;
        uint8_t* base = p.x[which] + row * kRowBytes;
        uint4* lo = reinterpret_cast<uint4*>(base + g * 16);
        uint4* hi = reinterpret_cast<uint4*>(base + 64 + g * 16);
        const uint4 ul = *lo, uh = *hi;
        const uint32_t* wl = reinterpret_cast<const uint32_t*>(&ul);
        const uint32_t* wh = reinterpret_cast<const uint32_t*>(&uh);
        uint32_t ol[4], oh[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float2 x0 = Half16<T>::to_f2(wl[e]), x1 = Half16<T>::to_f2(wh[e]);
            const int i = 8 * g + 2 * e;
            rope_rotate(x0.x, x1.x, rope_cos_sin(pos, i, p.log2_base));
            rope_rotate(x0.y, x1.y, rope_cos_sin(pos, i + 1, p.log2_base));
            ol[e] = Half16<T>::from_f2(x0.x, x0.y);
            oh[e] = Half16<T>::from_f2(x1.x, x1.y);
        }
        *lo = make_uint4(ol[0], ol[1], ol[2], ol[3]);
        *hi = make_uint4(oh[0], oh[1], oh[2], oh[3]);
    }
    pdl_trigger();
}

}  // namespace
}  // namespace kvd

using namespace kvd;

extern "C" kvd_status kvd_rope(kvd_dtype dtype, int32_t batch, int32_t n, void* q,
                               int32_t n_q_heads, void* k, int32_t n_k_heads,
                               const int32_t* pos0, float base, uint32_t flags,
                               int32_t* dev_err, kvd_stream_t stream) {
    (void)dev_err;
    if (dtype != KVD_F16 && dtype != KVD_BF16) return KVD_ERR_INVALID_ARG;
    if (batch < 0 || n < 0 || !(base > 0.f) || !(base < INFINITY)) return KVD_ERR_INVALID_ARG;
    if ((q && (n_q_heads <= 0 || !aligned16(q))) || (k && (n_k_heads <= 0 || !aligned16(k))))
        return KVD_ERR_INVALID_ARG;
    RopeParams p;
    p.x[0] = static_cast<uint8_t*>(q);
    p.x[1] = static_cast<uint8_t*>(k);
    p.heads[0] = q ? n_q_heads : 1;
    p.heads[1] = k ? n_k_heads : 1;
    p.items[0] = q ? (int64_t)batch * n_q_heads * n * 4 : 0;
    p.items[1] = k ? (int64_t)batch * n_k_heads * n * 4 : 0;
    p.pos0 = pos0;
    p.batch = batch;
    p.n = n;
    p.log2_base = log2f(base);
    const int64_t total = p.items[0] + p.items[1];
    if (total == 0) return KVD_OK;
    const int64_t blocks = (total + 255) / 256;
    if (blocks > 0x7fffffff) return KVD_ERR_UNSUPPORTED;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const bool pdl = (flags & KVD_FLAG_PDL) != 0;
    if (dtype == KVD_BF16)
        return launch(rope_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256), 0, st, pdl,
                      p);
    return launch(rope_kernel<__half>, dim3((unsigned)blocks), dim3(256), 0, st, pdl, p);
}
