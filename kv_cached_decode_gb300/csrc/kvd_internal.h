// kvd_internal.h -- host-side helpers shared by the launchers (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kvdecode.h"

namespace kvd {

// Number of SMs of the current device (cached per device).
int sm_count();

// 4-D TMA descriptor over one layer's K or V cache: dims (64, capacity, heads, batch),
// box (64 dims, min(64, capacity) positions, 1, 1), 128-byte swizzle, zero fill out of
// range.
kvd_status encode_cache_map(CUtensorMap* map, kvd_dtype dtype, void* base, const kvd_cache* c);

// 4-D TMA descriptor over dense rows of 64 16-bit values [batch, heads, rows, 64]: dims
// (64, rows, heads, batch), box (64, box_rows, 1, 1), 128-byte swizzle.
kvd_status encode_rows_map(CUtensorMap* map, kvd_dtype dtype, void* base, int rows, int heads,
                           int batch, int box_rows);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvd_status validate_cache(const kvd_cache* c);

// Launch with an optional programmatic-dependent-launch attribute; maps errors.
// Launch with an optional programmatic-dependent-launch attribute and an optional
// cluster shape (cluster_x CTAs along x); maps errors.
template <typename Kernel, typename... Args>
kvd_status launch_ex(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     bool pdl, unsigned cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

template <typename Kernel, typename... Args>
kvd_status launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                  bool pdl, Args... args) {
    return launch_ex(kernel, grid, block, smem, stream, pdl, 1u, args...);
}


// ---- attention work plan ------------------------------------------------------------
// The query vectors of one (cache row, KV head) -- rows_per_kv rows x group query
// heads x qlen tokens -- are processed together so every K/V tile is read once for
// all of them; they are cut into `nsub` blocks of at most `mmax`. A (row, KV head,
// block) triple is a "unit". The attended range of a unit is cut into `splits` chunks
// of `tiles_per_split` 64-position tiles, one thread block each. Splits of one unit
// that fit in one thread-block cluster merge through distributed shared memory (no
// workspace). A unit may also span `cgroups` clusters: each merges on chip, then their
// first CTAs merge through the workspace. Without clusters, more splits than one cluster
// holds merge through the workspace.
struct AttnPlan {
    int bkv, group, M, msub, nsub, units, tiles_total, rounds, splits, tiles_per_split, stages;
    int cgroups;  // clusters per unit (1: one cluster, or no cluster)
    bool cluster;
    size_t part_offset, ml_offset, ws_bytes;
};

constexpr int kMaxStages = 8;  // deepest K/V ring of an attention block
constexpr int kMmaQueryBlock = 16;     // query vectors per block on the tensor-core path
constexpr int kMaxSplits = 128;        // splits per unit (merge scratch is sized for this)
constexpr int kMaxClusterSplits = 16;  // largest cluster used for a merge
// A workspace merge (more splits than a cluster holds) is only considered for at most
// this many units: more units already fill the GPU with cluster-sized splits.
constexpr int kWsMaxUnits = 8;
// Most clusters per unit (kMaxGroups * kMaxClusterSplits <= kMaxSplits).
constexpr int kMaxGroups = 8;
// Least plain splits per unit for which several clusters per unit replace them.
constexpr int kGroupedMinSplits = 48;
// What the workspace merge costs (a global ticket, partials written and read back by
// the last block), in 64-position tiles of per-block streaming time.
constexpr int kWsMergeTiles = 12;

// The plan for a requested split count `s` (clamped to [1, min(rounds, kMaxSplits)];
// work is handed out in rounds of two tiles, so several s give the same plan).
// max_cluster: largest usable cluster (1 = never merge through a cluster).
AttnPlan plan_attention(int batch, int n_q_heads, int n_kv_heads, int rows_per_kv, int qlen,
                        int len_bound, int mmax, int s, int max_cluster);

// Whether splitting a unit beyond one cluster (merging through the workspace) can pay
// off: the tiles a block streams must drop by more than the merge costs. Depends only
// on the shape, so workspace sizing and the launcher agree.
bool workspace_merge_pays(int units, int rounds);

// The plan with `groups` clusters of at most `csize` splits per unit (the splits of the
// plan for groups * csize blocks, padded to a multiple of `groups`: padding blocks have no
// tiles). Their first CTAs merge through the workspace. It is considered only where
// workspace_merge_pays, and needs no more workspace than the plain workspace merge.
AttnPlan plan_grouped(int batch, int n_q_heads, int n_kv_heads, int rows_per_kv, int qlen,
                      int len_bound, int mmax, int groups, int csize);


// Workspace bytes of greedy_accept for a given target block count (greedy_accept.cu);
// sized with kWsTargetBound, an upper bound of the block count any launch targets.
constexpr int kWsTargetBound = 4096;
size_t accept_workspace_bytes(int batch, int k, int vocab, int target_ctas);

// Workspace bytes of kvd_sample_accept (sample_accept.cu).
size_t sample_workspace_bytes(int batch, int k, int vocab);

// The append kernel's launcher (kv_append.cu), arguments already validated. counts:
// NULL (q rows for every batch row) or device int32 [batch] rows per batch row (<= q).
// lens_in NULL means every row starts empty. rope_base > 0: the keys are written with
// rotary encoding at their absolute positions (dtype selects the element type).
kvd_status launch_append(const kvd_cache* cache, int32_t batch, int32_t q, const void* k_new,
                         const void* v_new, const int32_t* lens_in, const int32_t* counts,
                         int32_t* lens_out, kvd_dtype dtype, float rope_base, uint32_t flags,
                         int32_t* dev_err, cudaStream_t stream);

}  // namespace kvd
