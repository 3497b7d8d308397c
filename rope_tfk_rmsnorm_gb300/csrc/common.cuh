// common.cuh - device helpers shared by the libtfk kernels (sm_103a).
//
// 128-bit global accesses of 8 bf16 values, bf16 <-> fp32 conversion,
// cp.async staging into shared memory and warp reductions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"  // TFK_PDL

namespace tfk {

// Programmatic dependent launch (sm_90 and later): wait until every earlier
// grid on the stream has completed and its memory operations are visible to
// this grid.  A no-op for a launch without the programmatic attribute.  Every
// kernel calls it before its first global memory access.
__device__ __forceinline__ void grid_dep_wait() {
#if TFK_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

// Eight bf16 values in one 16-byte vector.
struct alignas(16) Vec8 {
    uint32_t w[4];
};

// Read-only 16-byte load through the non-coherent path (inputs never written
// by the kernel).
__device__ __forceinline__ Vec8 ld_ro(const void* p) {
    Vec8 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_vec(void* p, const Vec8& v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3])
                 : "memory");
}

__device__ __forceinline__ float4 ld_f4(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}

// bf16 widening is exact: the bf16 bits are the top half of the fp32 bits.
__device__ __forceinline__ void unpack8(const Vec8& v, float f[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(v.w[i] << 16);
        f[2 * i + 1] = __uint_as_float(v.w[i] & 0xFFFF0000u);
    }
}

// Two fp32 -> one bf16x2 word, round to nearest even (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ Vec8 pack8(const float f[8]) {
    Vec8 v;
#pragma unroll
    for (int i = 0; i < 4; ++i) v.w[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
    return v;
}

// ---- packed fp32x2 arithmetic (sm_100+) ------------------------------------
// Two fp32 values in one 64-bit register pair: lane 0 = the lower-addressed
// element.  mul/fma .rn round each lane exactly like the scalar instruction,
// at half the instruction count.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_make(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_split(f32x2 v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// One bf16x2 word (element 2i in the low half) -> exact fp32x2.
__device__ __forceinline__ f32x2 bf2_to_f2(uint32_t w) {
    return f2_make(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// fp32x2 -> one bf16x2 word, round to nearest even.
__device__ __forceinline__ uint32_t f2_to_bf2(f32x2 v) {
    float lo, hi;
    f2_split(v, lo, hi);
    return pack_bf16x2(lo, hi);
}

// ---- cp.async staging (16 bytes per thread, bypassing L1) -----------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"(smem_addr(smem_dst)), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

// Same wait with a run-time depth (a ring of `stages` buffers keeps
// stages-1 groups in flight); the branch is uniform over the CTA.
__device__ __forceinline__ void cp_async_wait_dyn(int pending) {
    switch (pending) {
        case 0: cp_async_wait<0>(); break;
        case 1: cp_async_wait<1>(); break;
        case 2: cp_async_wait<2>(); break;
        case 3: cp_async_wait<3>(); break;
        case 4: cp_async_wait<4>(); break;
        case 5: cp_async_wait<5>(); break;
        case 6: cp_async_wait<6>(); break;
        case 7: cp_async_wait<7>(); break;
        case 8: cp_async_wait<8>(); break;
        case 9: cp_async_wait<9>(); break;
        case 10: cp_async_wait<10>(); break;
        case 11: cp_async_wait<11>(); break;
        case 12: cp_async_wait<12>(); break;
        case 13: cp_async_wait<13>(); break;
        case 14: cp_async_wait<14>(); break;
        default: cp_async_wait<15>(); break;
    }
}

__device__ __forceinline__ Vec8 ld_smem_vec(const void* p) {
    Vec8 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "r"(smem_addr(p)));
    return v;
}

// ---- thread-block clusters ---------------------------------------------------

// Rank of this CTA in its cluster.
__device__ __forceinline__ unsigned cluster_ctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives and waits (a hardware
// barrier, like __syncthreads for the cluster); shared-memory writes made
// before it, to this CTA or to another CTA of the cluster, are visible after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store v to the same shared-memory variable as `local` in CTA `peer` of the cluster.
__device__ __forceinline__ void st_peer_f32(const void* local, unsigned peer, float v) {
    unsigned remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(peer));
    asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(remote), "f"(v) : "memory");
}

// ---- reductions -------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

}  // namespace tfk
