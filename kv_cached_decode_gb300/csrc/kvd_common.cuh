// kvd_common.cuh -- device-side building blocks shared by the sm_103a kernels.
//
// Inline-PTX wrappers written from the PTX ISA: mbarrier, TMA tensor loads
// (cp.async.bulk.tensor), proxy fences, programmatic dependent launch
// (griddepcontrol), ldmatrix and the m16n8k16 tensor-core MMA. Every wait on an
// mbarrier is bounded by the global nanosecond timer; on timeout the kernel records
// KVD_ERR_TIMEOUT and gives up instead of spinning.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <stdint.h>

#include "kvdecode.h"

namespace kvd {

constexpr int kHeadDim = 64;
constexpr int kTile = 64;                          // cache positions per TMA box
constexpr int kRowBytes = kHeadDim * 2;            // 128 B per position (16-bit types)
constexpr int kTileBytes = kTile * kRowBytes;      // 8 KiB per K (or V) tile
constexpr unsigned long long kWaitNs = 1000000000ull;  // 1 s bound on any wait
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- error flag -------
__device__ __forceinline__ void flag_error(int32_t* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------- 16-bit types ------
template <typename T> struct Half16;
template <> struct Half16<__half> {
    static __device__ __forceinline__ float2 to_f2(uint32_t w) {
        return __half22float2(*reinterpret_cast<const __half2*>(&w));
    }
    static __device__ __forceinline__ uint32_t from_f2(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    static __device__ __forceinline__ __half from_f(float a) { return __float2half_rn(a); }
};
template <> struct Half16<__nv_bfloat16> {
    static __device__ __forceinline__ float2 to_f2(uint32_t w) {
        // bfloat16 is the upper half of an fp32 pattern: widening is exact.
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    }
    static __device__ __forceinline__ uint32_t from_f2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float a) {
        return __float2bfloat16_rn(a);
    }
};

template <typename T>
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
    float2 a = Half16<T>::to_f2(u.x), b = Half16<T>::to_f2(u.y);
    float2 c = Half16<T>::to_f2(u.z), d = Half16<T>::to_f2(u.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

// ---------------------------------------------------------------- rotary encoding --
// Rotate-half rotary encoding of 64-dim vectors: dims i and i + 32 form a pair rotated
// by pos * theta_i, theta_i = base^(-i/32). One definition for every kernel that
// rotates, so a rotation fused into another kernel gives the same bits as the stand-
// alone one: the angle is formed in fp32 and sin/cos come from sincosf; the products are
// rounded explicitly (no contraction choices left to the compiler).
__device__ __forceinline__ float2 rope_cos_sin(int pos, int i, float log2_base) {
    const float a = (float)pos * exp2f(-(float)i / 32.f * log2_base);
    float sn, cs;
    sincosf(a, &sn, &cs);
    return make_float2(cs, sn);
}
// (x0, x1) = (x[i], x[i+32]) -> (x0 cos - x1 sin, x1 cos + x0 sin)
__device__ __forceinline__ void rope_rotate(float& x0, float& x1, float2 cs) {
    const float y0 = __fmaf_rn(x0, cs.x, -__fmul_rn(x1, cs.y));
    const float y1 = __fmaf_rn(x1, cs.x, __fmul_rn(x0, cs.y));
    x0 = y0;
    x1 = y1;
}

// Rotary encoding of 8 pairs: dims i0..i0+7 in lo, i0+32..i0+39 in hi, rounded back to
// the storage type (the same bits as the stand-alone rotation).
template <typename T>
__device__ __forceinline__ void rope_rotate8(uint4& lo, uint4& hi, const float2* tr, int i0) {
    uint32_t* a = reinterpret_cast<uint32_t*>(&lo);
    uint32_t* b = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        float2 x = Half16<T>::to_f2(a[w]), y = Half16<T>::to_f2(b[w]);
        rope_rotate(x.x, y.x, tr[i0 + 2 * w]);
        rope_rotate(x.y, y.y, tr[i0 + 2 * w + 1]);
        a[w] = Half16<T>::from_f2(x.x, x.y);
        b[w] = Half16<T>::from_f2(y.x, y.y);
    }
}
// As rope_rotate8, with the cos/sin of position pos computed here.
template <typename T>
__device__ __forceinline__ void rope_rotate8_at(uint4& lo, uint4& hi, int pos, int i0,
                                                float log2_base) {
    uint32_t* a = reinterpret_cast<uint32_t*>(&lo);
    uint32_t* b = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        float2 x = Half16<T>::to_f2(a[w]), y = Half16<T>::to_f2(b[w]);
        rope_rotate(x.x, y.x, rope_cos_sin(pos, i0 + 2 * w, log2_base));
        rope_rotate(x.y, y.y, rope_cos_sin(pos, i0 + 2 * w + 1, log2_base));
        a[w] = Half16<T>::from_f2(x.x, x.y);
        b[w] = Half16<T>::from_f2(y.x, y.y);
    }
}

// 2^x by the hardware approximation (ex2.approx.ftz: relative error near 2^-22, -inf
// gives +0); for softmax weights that are rounded to 16 bits afterwards.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- shared memory ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of 16-byte chunk `c` of row `r` inside a tile written by TMA with the
// 128-byte swizzle: the chunk index is XORed with the row index modulo 8.
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>(r * kRowBytes + ((c ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------- mbarrier ---------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}
// Raise the transaction count of the current phase by `bytes`, without an arrival.
__device__ __forceinline__ void mbar_expect_tx_only(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// One arrival (release) on the barrier.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// As mbar_wait_bounded, for a barrier that other CTAs of the cluster arrive on (the
// acquire covers their writes to this CTA's shared memory), with a bound of `budget_ns`.
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                          unsigned long long budget_ns = kWaitNs) {
    // the clock is read every 64 polls only: polling threads then stay cheap
    unsigned long long t0 = 0;
    for (unsigned n = 1; !mbar_try_wait_cluster(bar, parity); ++n) {
        if (n % 64 == 0) {
            if (t0 == 0) t0 = global_ns();
            else if (global_ns() - t0 > budget_ns) return false;
        }
    }
    return true;
}
// Wait for phase `parity` of the barrier; false if it did not complete within about 1 s.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    unsigned long long t0 = 0;
    for (unsigned n = 1; !mbar_try_wait(bar, parity); ++n) {
        if (n % 64 == 0) {
            if (t0 == 0) t0 = global_ns();
            else if (global_ns() - t0 > kWaitNs) return false;
        }
    }
    return true;
}

// ---------------------------------------------------------------- cp.async ---------
// 16-byte asynchronous global -> shared copy (L2 only), and the wait for all of this
// thread's copies.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------- bulk copies ------
// Untiled bulk copy global -> shared completing on `bar` (both addresses 16-byte
// aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// ---------------------------------------------------------------- TMA --------------
// 4-D tiled tensor load (coordinates innermost first) completing on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}
// Tiled shared -> global copy of one box at (c0, c1, c2, c3) (every coordinate >= 0; the
// part of the box outside the tensor is not written), tracked in this thread's bulk group.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];"
        ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until this thread's committed bulk copies have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- PDL --------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- clusters ---------
// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_shared(uint32_t addr, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
    return out;
}
// Asynchronous 16-byte store into another CTA's shared memory; completion is counted
// in bytes on that CTA's mbarrier (complete_tx), so no fence or arrive is needed.
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, float4 v, uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, "
        "[%5];" ::"r"(remote_addr),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
        : "memory");
}
// Split cluster barrier: arrive early, wait (acquire) later. The arrive is relaxed: what
// it publishes (mbarrier initialisation) is ordered by fence.mbarrier_init.release.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---------------------------------------------------------------- tensor cores -----
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

template <typename T> struct Mma;
template <> struct Mma<__half> {
    static __device__ __forceinline__ void run(float* c, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // Rows 0..7 only: A rows 8..15 are zero (a1 = a3 = 0), the accumulator of rows
    // 0..7 is c[0..1]; rows 8..15 start from 0 and their results are discarded.
    static __device__ __forceinline__ void run_top(float* c, uint32_t a0, uint32_t a2,
                                                   uint32_t b0, uint32_t b1) {
        float d2, d3;
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %10, %10};"
            : "+f"(c[0]), "+f"(c[1]), "=f"(d2), "=f"(d3)
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.f));
    }
};
template <> struct Mma<__nv_bfloat16> {
    static __device__ __forceinline__ void run(float* c, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // Rows 0..7 only: A rows 8..15 are zero (a1 = a3 = 0), the accumulator of rows
    // 0..7 is c[0..1]; rows 8..15 start from 0 and their results are discarded.
    static __device__ __forceinline__ void run_top(float* c, uint32_t a0, uint32_t a2,
                                                   uint32_t b0, uint32_t b1) {
        float d2, d3;
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %10, %10};"
            : "+f"(c[0]), "+f"(c[1]), "=f"(d2), "=f"(d3)
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.f));
    }
};

}  // namespace kvd
