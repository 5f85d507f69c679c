// pa_common.cuh -- device helpers shared by the kernels: element types,
// mbarrier / bulk-copy / cluster PTX wrappers, the exp2 instruction and the
// device error word.  Written for sm_103a (GB300).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// ---- device error word (sticky; read and cleared by pa_device_error) ------
// Kernels receive its address as a parameter (it lives in one translation
// unit; the library is built without relocatable device code).
__device__ __forceinline__ void set_error(unsigned int *err, unsigned int bits) {
    atomicOr(err, bits);
}

constexpr unsigned ERR_BLOCK_ID = 0x1u;
constexpr unsigned ERR_SEQ_LEN = 0x2u;
constexpr unsigned ERR_SLOT = 0x4u;
constexpr unsigned ERR_TIMEOUT = 0x8u;

// Wall-clock limit of any wait on an asynchronous copy (ns).
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;

// ---- element types --------------------------------------------------------
// Each 16-byte chunk holds E elements; to_f32 widens them exactly.
template <typename T> struct Elem;

template <> struct Elem<float> {
    static constexpr int E = 4;
    __device__ __forceinline__ static void to_f32(const uint4 &c, float *f) {
        f[0] = __uint_as_float(c.x); f[1] = __uint_as_float(c.y);
        f[2] = __uint_as_float(c.z); f[3] = __uint_as_float(c.w);
    }
    __device__ __forceinline__ static float load1(const float *p) { return *p; }
    __device__ __forceinline__ static void store1(float *p, float v) { *p = v; }
};

template <> struct Elem<__nv_bfloat16> {
    static constexpr int E = 8;
    // bf16 is the top half of a binary32: widening is a shift / mask.
    __device__ __forceinline__ static void pair(uint32_t w, float &lo, float &hi) {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xffff0000u);
    }
    __device__ __forceinline__ static void to_f32(const uint4 &c, float *f) {
        pair(c.x, f[0], f[1]); pair(c.y, f[2], f[3]);
        pair(c.z, f[4], f[5]); pair(c.w, f[6], f[7]);
    }
    __device__ __forceinline__ static float load1(const __nv_bfloat16 *p) {
        return __bfloat162float(*p);
    }
    __device__ __forceinline__ static void store1(__nv_bfloat16 *p, float v) {
        *p = __float2bfloat16_rn(v);
    }
};

template <> struct Elem<__half> {
    static constexpr int E = 8;
    __device__ __forceinline__ static void pair(uint32_t w, float &lo, float &hi) {
        __half2 h = *reinterpret_cast<__half2 *>(&w);
        float2 f = __half22float2(h);
        lo = f.x; hi = f.y;
    }
    __device__ __forceinline__ static void to_f32(const uint4 &c, float *f) {
        pair(c.x, f[0], f[1]); pair(c.y, f[2], f[3]);
        pair(c.z, f[4], f[5]); pair(c.w, f[6], f[7]);
    }
    __device__ __forceinline__ static float load1(const __half *p) {
        return __half2float(*p);
    }
    __device__ __forceinline__ static void store1(__half *p, float v) {
        *p = __float2half_rn(v);
    }
};

// ---- math -----------------------------------------------------------------
// 2^x with the hardware approximation instruction (MUFU.EX2): relative error
// about 2^-22, ex2(-inf) = 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction (three-input max.f32 of sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Two fp32 lanes at once (the packed f32x2 arithmetic of sm_100 and later):
// d = a * b + c and d = a + b, each lane rounded to nearest like its scalar
// counterpart.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

constexpr float LOG2E = 1.4426950408889634f;   // log2(e)
constexpr float LN2 = 0.6931471805599453f;     // ln(2)

// ---- time -----------------------------------------------------------------
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- shared-memory addresses and mbarriers --------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

// make barrier initialisation visible to the async proxy and the cluster
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// order this thread's prior generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile(
        "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
        :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, for at most WAIT_LIMIT_NS.
// Returns false (and sets ERR_TIMEOUT) if the limit was reached.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  unsigned int *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > WAIT_LIMIT_NS) {
            set_error(err, ERR_TIMEOUT);
            return false;
        }
    }
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes`
// transaction bytes on `bar`.  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Tensor-map bulk copy of one 3-D box (coordinates x, y, z in elements) to
// this CTA's shared memory, completing on `bar`.  x * element size must be a
// multiple of 16 bytes; dst must be 1024-byte aligned for the 128-byte swizzle.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, int x, int y, int z,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;"
        :: "r"(smem_u32(dst)), "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)),
           "l"(policy)
        : "memory");
}

// Bring a tensor-map descriptor (kernel parameter) into the TMA unit's cache.
__device__ __forceinline__ void prefetch_tensormap(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(tmap) : "memory");
}

// L2 policy for data read once per call (the streamed K/V tiles).
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// L2 policy for data several blocks read in turn (K/V of a long query run).
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- clusters -------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Programmatic dependent launch.  A kernel launched with programmatic
// stream serialization may start while the kernel before it in the stream
// is still running once every block of that kernel has called
// launch_dependents(); grid_dependency_wait() then blocks until that kernel
// has completed and its writes are visible (it returns at once when there is
// no such kernel).
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The two halves of cluster_sync(), for work in between: arrive (release)
// once, and wait (acquire) before the first access to a peer's shared memory.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bring the 128-byte lines of [base, base + bytes) into L2, spread over every
// thread of the grid (a hint: no data moves into the SM).
__device__ __forceinline__ void prefetch_l2_range(const void *base, size_t bytes) {
    const char *b = reinterpret_cast<const char *>(base);
    const size_t stride = (size_t)gridDim.x * blockDim.x * 128;
    for (size_t off = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 128; off < bytes; off += stride)
        asm volatile("prefetch.global.L2 [%0];" :: "l"(b + off));
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// address of the same shared-memory variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_to_rank(const void *p, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
    return out;
}

__device__ __forceinline__ float4 ld_dsmem_f32x4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ int ld_acquire_dsmem_s32(uint32_t addr) {
    int v;
    asm volatile("ld.acquire.cluster.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_dsmem_s32(uint32_t addr, int v) {
    asm volatile("st.release.cluster.shared::cluster.s32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}

// monotonic publish: *addr = max(*addr, v), release at cluster scope
__device__ __forceinline__ void red_max_release_dsmem(uint32_t addr, int v) {
    asm volatile("red.release.cluster.shared::cluster.max.s32 [%0], %1;" :: "r"(addr), "r"(v)
                 : "memory");
}

__device__ __forceinline__ void st_dsmem_s32(uint32_t addr, int v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}

// atomic add on a cluster-shared int with acquire-release ordering at
// cluster scope; returns the old value
__device__ __forceinline__ int atom_add_acq_rel_dsmem(uint32_t addr, int v) {
    int old;
    asm volatile("atom.acq_rel.cluster.shared::cluster.add.s32 %0, [%1], %2;"
                 : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void fence_acq_rel_cluster() {
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Ascending sort of 32*EPT keys (distinct values; `in` padded with
// 0xffffffff) by one warp, EPT keys per lane in registers: a bitonic network
// whose strides inside a lane are register swaps and whose longer strides
// are shuffles, so no step waits on shared memory or a block barrier.
template <int EPT>
__device__ __forceinline__ void warp_bitonic_sort(const uint32_t *in, uint32_t *out) {
    constexpr int N = 32 * EPT;
    const int lane = threadIdx.x & 31;
    uint32_t v[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) v[e] = in[lane * EPT + e];
#pragma unroll
    for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j < EPT) {
#pragma unroll
                for (int e = 0; e < EPT; ++e) {
                    const int e2 = e ^ j;
                    if (e2 > e) {
                        const bool up = ((lane * EPT + e) & k) == 0;
                        const uint32_t x = v[e], y = v[e2];
                        const bool swap = (x > y) == up;
                        v[e] = swap ? y : x;
                        v[e2] = swap ? x : y;
                    }
                }
            } else {
                const int m = j / EPT;                 // partner lane offset
                const bool lower = (lane & m) == 0;
#pragma unroll
                for (int e = 0; e < EPT; ++e) {
                    const bool up = ((lane * EPT + e) & k) == 0;
                    const uint32_t y = __shfl_xor_sync(0xffffffffu, v[e], m);
                    v[e] = (lower == up) ? min(v[e], y) : max(v[e], y);
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) out[lane * EPT + e] = v[e];
}

}  // namespace pa
