// api.cu -- status strings, version, workspace sizing and shared host helpers.
#include <algorithm>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "kvd_internal.h"

namespace kvd {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
}  // namespace

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

kvd_status encode_cache_map(CUtensorMap* map, kvd_dtype dtype, void* base, const kvd_cache* c) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return KVD_ERR_CUDA;
    const cuuint64_t dims[4] = {(cuuint64_t)c->head_dim, (cuuint64_t)c->capacity,
                                (cuuint64_t)c->n_kv_heads, (cuuint64_t)c->batch};
    const cuuint64_t strides[3] = {(cuuint64_t)c->stride_t * 2, (cuuint64_t)c->stride_h * 2,
                                   (cuuint64_t)c->stride_b * 2};
    const cuuint32_t box[4] = {(cuuint32_t)KVD_HEAD_DIM, (cuuint32_t)std::min(64, c->capacity),
                               1, 1};
    const cuuint32_t elem[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map,
                          dtype == KVD_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          4, base, dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KVD_OK : KVD_ERR_INVALID_ARG;
}

kvd_status encode_rows_map(CUtensorMap* map, kvd_dtype dtype, void* base, int rows, int heads,
                           int batch, int box_rows) {
    kvd_cache c = {};
    c.head_dim = KVD_HEAD_DIM;
    c.capacity = rows;
    c.n_kv_heads = heads;
    c.batch = batch;
    c.stride_t = KVD_HEAD_DIM;
    c.stride_h = (int64_t)rows * KVD_HEAD_DIM;
    c.stride_b = (int64_t)heads * rows * KVD_HEAD_DIM;
    if (kvd_status s = encode_cache_map(map, dtype, base, &c)) return s;
    if (box_rows == std::min(64, rows)) return KVD_OK;
    // the same map with a taller box
    const cuuint64_t dims[4] = {(cuuint64_t)KVD_HEAD_DIM, (cuuint64_t)rows, (cuuint64_t)heads,
                                (cuuint64_t)batch};
    const cuuint64_t strides[3] = {(cuuint64_t)c.stride_t * 2, (cuuint64_t)c.stride_h * 2,
                                   (cuuint64_t)c.stride_b * 2};
    const cuuint32_t box[4] = {(cuuint32_t)KVD_HEAD_DIM, (cuuint32_t)box_rows, 1, 1};
    const cuuint32_t elem[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map,
                          dtype == KVD_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          4, base, dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KVD_OK : KVD_ERR_INVALID_ARG;
}

kvd_status validate_cache(const kvd_cache* c) {
    if (!c || !c->k || !c->v) return KVD_ERR_INVALID_ARG;
    if (c->head_dim != KVD_HEAD_DIM) return KVD_ERR_UNSUPPORTED;
    if (c->batch <= 0 || c->n_kv_heads <= 0 || c->capacity <= 0) return KVD_ERR_INVALID_ARG;
    if (c->stride_t < KVD_HEAD_DIM || c->stride_h <= 0 || c->stride_b <= 0)
        return KVD_ERR_INVALID_ARG;
    if ((c->stride_t | c->stride_h | c->stride_b) & 7) return KVD_ERR_INVALID_ARG;
    if (!aligned16(c->k) || !aligned16(c->v)) return KVD_ERR_INVALID_ARG;
    return KVD_OK;
}

AttnPlan plan_attention(int batch, int n_q_heads, int n_kv_heads, int rows_per_kv, int qlen,
                        int len_bound, int mmax, int s, int max_cluster) {
    AttnPlan P = {};
    P.bkv = batch / rows_per_kv;
    P.group = n_q_heads / n_kv_heads;
    P.M = rows_per_kv * P.group * qlen;
    P.nsub = (P.M + mmax - 1) / mmax;
    P.msub = (P.M + P.nsub - 1) / P.nsub;
    P.units = P.bkv * n_kv_heads * P.nsub;
    P.tiles_total = (std::max(len_bound, 0) + 63) / 64;
    // Work is handed out in rounds of two 64-position tiles (the eight warps of a block
    // work on two tiles at once).
    P.rounds = (P.tiles_total + 1) / 2;
    s = std::max(1, std::min({s, P.rounds, kMaxSplits}));
    P.tiles_per_split = 2 * std::max(1, (P.rounds + s - 1) / s);
    P.splits = P.tiles_total > 0 ? (P.tiles_total + P.tiles_per_split - 1) / P.tiles_per_split : 1;
    P.cluster = P.splits > 1 && P.splits <= max_cluster;
    P.cgroups = 1;
    P.stages = P.tiles_per_split >= 4 ? 4 : 2;
    P.part_offset = KVD_WS_COUNTER_BYTES;
    const size_t slots = (size_t)P.units * P.splits * P.msub;
    P.ml_offset = align_up(P.part_offset + slots * 64 * sizeof(float), 256);
    P.ws_bytes = (P.splits > 1 && !P.cluster) ? P.ml_offset + slots * 2 * sizeof(float) : 0;
    return P;
}

AttnPlan plan_grouped(int batch, int n_q_heads, int n_kv_heads, int rows_per_kv, int qlen,
                      int len_bound, int mmax, int groups, int csize) {
    AttnPlan P = plan_attention(batch, n_q_heads, n_kv_heads, rows_per_kv, qlen, len_bound, mmax,
                                groups * csize, 1);
    const int cs = (P.splits + groups - 1) / groups;
    P.cgroups = groups;
    P.splits = cs * groups;
    P.cluster = true;
    const size_t slots = (size_t)P.units * groups * P.msub;
    P.ml_offset = align_up(P.part_offset + slots * 64 * sizeof(float), 256);
    P.ws_bytes = P.ml_offset + slots * 2 * sizeof(float);
    return P;
}

bool workspace_merge_pays(int units, int rounds) {
    if (units > kWsMaxUnits || rounds <= kMaxClusterSplits) return false;
    const int tps_cluster = 2 * ((rounds + kMaxClusterSplits - 1) / kMaxClusterSplits);
    const int s = std::min(rounds, kMaxSplits);
    const int tps_ws = 2 * ((rounds + s - 1) / s);
    return tps_cluster - tps_ws > kWsMergeTiles;
}

}  // namespace kvd

using namespace kvd;

extern "C" size_t kvd_workspace_size(kvd_op op, int32_t batch, int32_t n_q_heads,
                                     int32_t n_kv_heads, int32_t rows_per_kv, int32_t qlen,
                                     int32_t max_len, int32_t vocab) {
    switch (op) {
    case KVD_OP_DECODE_ATTN:
    case KVD_OP_VERIFY_ATTN: {
        const int q = op == KVD_OP_DECODE_ATTN ? 1 : qlen;
        if (batch <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || rows_per_kv <= 0 ||
            n_q_heads % n_kv_heads || batch % rows_per_kv || q < 1 || q > KVD_MAX_QLEN ||
            max_len < 0)
            return 0;
        // one query vector per KV head runs alone; two or more go in blocks of 16
        const int64_t M = (int64_t)rows_per_kv * (n_q_heads / n_kv_heads) * q;
        const int mmax = M >= 2 ? kMmaQueryBlock : 1;
        const AttnPlan P1 = plan_attention(batch, n_q_heads, n_kv_heads, rows_per_kv, q, max_len,
                                           mmax, 1, 1);
        if (!workspace_merge_pays(P1.units, P1.rounds)) return KVD_WS_COUNTER_BYTES;
        // The most splits a launch can use bounds every workspace plan (a grouped plan
        // keeps kMaxGroups <= kMaxSplits partials per unit).
        const AttnPlan P = plan_attention(batch, n_q_heads, n_kv_heads, rows_per_kv, q, max_len,
                                          mmax, kMaxSplits, 1);
        return std::max<size_t>(P.ws_bytes, KVD_WS_COUNTER_BYTES);
    }
    case KVD_OP_GREEDY_ACCEPT: {
        if (batch <= 0 || qlen < 1 || qlen > KVD_MAX_QLEN || vocab <= 0) return 0;
        return accept_workspace_bytes(batch, qlen, vocab, kWsTargetBound);
    }
    case KVD_OP_SAMPLE_ACCEPT: {
        if (batch <= 0 || qlen < 0 || qlen > 7 || vocab <= 0) return 0;
        return sample_workspace_bytes(batch, qlen, vocab);
    }
    }
    return 0;
}

extern "C" const char* kvd_status_string(kvd_status s) {
    switch (s) {
    case KVD_OK: return "KVD_OK";
    case KVD_ERR_INVALID_ARG: return "KVD_ERR_INVALID_ARG: invalid argument";
    case KVD_ERR_UNSUPPORTED: return "KVD_ERR_UNSUPPORTED: unsupported shape or option";
    case KVD_ERR_WORKSPACE: return "KVD_ERR_WORKSPACE: workspace missing or too small";
    case KVD_ERR_CUDA: return "KVD_ERR_CUDA: CUDA call failed";
    case KVD_ERR_LEN_OVERFLOW: return "KVD_ERR_LEN_OVERFLOW: length outside [0, capacity]";
    case KVD_ERR_BAD_INDEX: return "KVD_ERR_BAD_INDEX: beam parent outside its window";
    case KVD_ERR_BAD_TOKEN: return "KVD_ERR_BAD_TOKEN: draft id outside the vocabulary";
    case KVD_ERR_NAN: return "KVD_ERR_NAN: NaN in the logits";
    case KVD_ERR_TIMEOUT: return "KVD_ERR_TIMEOUT: a bounded device wait gave up";
    }
    return "unknown kvd_status";
}

extern "C" int32_t kvd_version(void) { return 100; }
