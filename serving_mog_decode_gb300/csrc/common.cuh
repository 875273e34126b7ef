// common.cuh -- device helpers shared by libmog's kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MOG_D 128          // head dimension supported by the kernels
#define MOG_MAX_G 16       // query heads per KV head (one mma M tile)
#define MOG_MAX_L 32       // subclusters per cluster (one warp of lanes)
#define MOG_MAX_UNION 256  // top_c * G: distinct selected clusters per unit

namespace mog {

// ---------------------------------------------------------------------------------- bf16

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf1(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// round-to-nearest-even float -> bf16 bits (finite inputs)
__device__ __forceinline__ uint32_t f2bf(float f) {
    uint32_t u = __float_as_uint(f);
    u += 0x7fffu + ((u >> 16) & 1u);
    return u >> 16;
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    return f2bf(lo) | (f2bf(hi) << 16);
}
// the same with one conversion instruction (round to nearest even, both halves)
__device__ __forceinline__ uint32_t cvt_bf2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// float -> fp8 e4m3 bits, nearest with ties to even, saturating at +-448
__device__ __forceinline__ uint32_t f2e4m3(float f) {
    uint16_t r;
    asm("{\n.reg .b16 t;\ncvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\nmov.b16 %0, t;\n}" : "=h"(r) : "f"(0.f), "f"(f));
    return r & 0xffu;
}
// four fp8 e4m3 values (bytes of w, lowest first) -> floats (exact)
__device__ __forceinline__ float4 e4m3x4_to_float4(uint32_t w) {
    uint32_t lo, hi;
    asm("{\n.reg .b16 a, b;\nmov.b32 {a, b}, %2;\ncvt.rn.f16x2.e4m3x2 %0, a;\ncvt.rn.f16x2.e4m3x2 %1, b;\n}"
        : "=r"(lo), "=r"(hi) : "r"(w));
    const __half2 h0 = *reinterpret_cast<const __half2 *>(&lo), h1 = *reinterpret_cast<const __half2 *>(&hi);
    return make_float4(__low2float(h0), __high2float(h0), __low2float(h1), __high2float(h1));
}
// the float value of an e4m3 byte (exact)
__device__ __forceinline__ float e4m3_to_float(uint32_t b) { return e4m3x4_to_float4(b & 0xffu).x; }
// x rounded to the nearest e4m3 value (ties to even, saturating), as a float
__device__ __forceinline__ float e4m3_round(float x) { return e4m3_to_float(f2e4m3(x)); }

// 2^x by the hardware approximation (flush-to-zero; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// min(a, b, c) in one three-input instruction (the minimum of three floats; NaN inputs
// are ignored as by fminf)
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// ------------------------------------------------------------------------------ warp ops

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ int warp_isum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// (score desc, index asc) ordering: true if (a, ia) ranks before (b, ib)
__device__ __forceinline__ bool ranks_before(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

// ---------------------------------------------------------------------- Kahan summation

struct Kahan {
    float s, c;
    __device__ __forceinline__ void init() { s = 0.f; c = 0.f; }
    __device__ __forceinline__ void add(float x) {
        float y = __fsub_rn(x, c);
        float t = __fadd_rn(s, y);
        c = __fsub_rn(__fsub_rn(t, s), y);
        s = t;
    }
};

// ------------------------------------------------------------------------- async copies

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
// 16-byte global->shared copy; src_bytes = 0 zero-fills the destination
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// wait until at most n (runtime, 0..5) cp.async groups are pending
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
    switch (n <= 0 ? 0 : n) {
        case 0: cp_async_wait<0>(); break;
        case 1: cp_async_wait<1>(); break;
        case 2: cp_async_wait<2>(); break;
        case 3: cp_async_wait<3>(); break;
        case 4: cp_async_wait<4>(); break;
        default: cp_async_wait<5>(); break;
    }
}

// read-only 16-byte global load, not kept in L1
__device__ __forceinline__ uint4 ldg_nc16(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// --------------------------------------------------------------------- tensor-core mma

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// transpose of an 8 x 8 matrix of 16-bit elements held one row pair per lane (mma layout)
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
    return d;
}
// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------ thread-block clusters

// Split cluster barrier: arrive (relaxed: orders nothing) and wait.  Every thread of every
// CTA of the cluster executes both, arrive first.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
// Request the 128-byte line holding p into L2 (no register result, no fault on the line)
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---------------------------------------------------------- programmatic dependent launch

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------- misc

__host__ __device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) {
    return (a + b - 1) / b;
}

// Device status word bits (arena status[0])
enum : int { ST_OK = 0, ST_BAD_INDEX = 1, ST_BAD_SIZE = 2, ST_TIMEOUT = 3 };

__device__ __forceinline__ void flag_error(int *status, int code) {
    if (status) atomicOr(status, 1 << code);
}

}  // namespace mog
