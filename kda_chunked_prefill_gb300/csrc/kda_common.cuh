// Device helpers shared by the KDA kernels: warp-level MMA and ldmatrix
// wrappers, async copies, base-2 exponent, bf16 packing.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr int BT = 64;   // chunk length (tokens)
constexpr int SB = 16;   // sub-block length (tokens)
constexpr int DK = 128;  // key head dim
constexpr int DV = 128;  // value head dim
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 2^x on the special-function unit (flushes subnormal results to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 p = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

__device__ __forceinline__ float2 unpack_f16(uint32_t u) {
    __half2 p = *reinterpret_cast<__half2 *>(&u);
    return __half22float2(p);
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi): about 16 significant bits
// in two bf16 operands, with bf16's exponent range.
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
    const float r0 = x0 - __bfloat162float(h0), r1 = x1 - __bfloat162float(h1);
    __nv_bfloat162 h;
    h.x = h0;
    h.y = h1;
    hi = *reinterpret_cast<uint32_t *>(&h);
    lo = pack_bf16(r0, r1);
}

// Largest magnitude kept below fp16's finite limit (65504) with margin.
constexpr float F16_SAFE = 60000.f;

__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    __nv_bfloat162 p = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(p);
}

// 16-byte global -> shared copy; src_bytes = 0 zero-fills the destination.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// ldmatrix: four 8x8 b16 matrices; lane l supplies the row address of
// matrix l/8, row l%8.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A(16x16, row) * B(16x8, col), fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Fragment addressing (lane = threadIdx.x % 32) for a 16x16 tile at (row0,col0)
// of a row-major bf16 matrix with row stride `ld` elements.
//  A operand, stored [m][k]:                 ldsm_x4  at  a_addr
//  A operand, stored transposed [k][m]:      ldsm_x4_t at at_addr
//  B operand (two n8 tiles), stored [n][k]:  ldsm_x4  at  bn_addr
//  B operand (two n8 tiles), stored [k][n]:  ldsm_x4_t at bk_addr
__device__ __forceinline__ int a_off(int lane, int row0, int col0, int ld) {
    return (row0 + (lane & 15)) * ld + col0 + ((lane >> 4) << 3);
}
__device__ __forceinline__ int at_off(int lane, int m0, int k0, int ld) {
    const int mi = lane >> 3, r = lane & 7;
    return (k0 + ((mi >> 1) << 3) + r) * ld + m0 + ((mi & 1) << 3);
}
__device__ __forceinline__ int bn_off(int lane, int n0, int k0, int ld) {
    const int mi = lane >> 3, r = lane & 7;
    return (n0 + ((mi >> 1) << 3) + r) * ld + k0 + ((mi & 1) << 3);
}
__device__ __forceinline__ int bk_off(int lane, int k0, int n0, int ld) {
    const int mi = lane >> 3, r = lane & 7;
    return (k0 + ((mi & 1) << 3) + r) * ld + n0 + ((mi >> 1) << 3);
}

__device__ __forceinline__ void set_status(int32_t *status, int32_t code) {
    if (status) atomicCAS(status, 0, code);
}

}  // namespace kda
