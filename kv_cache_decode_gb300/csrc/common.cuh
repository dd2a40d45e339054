// Small device helpers: inline PTX for the sm_103a paths used by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace kvd {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy through L2 only. src_bytes = 0 copies nothing
// and fills the 16 bytes with zeros (used for rows past a sequence's end).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n" ::"r"(dst),
        "l"(src), "r"(src_bytes), "l"(policy));
}
// 4-byte global -> shared copy (through L1); src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// L2 policy: the KV cache is streamed once per step, so let it go first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
    return p;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D[16x8] += A[16x16] * B[16x8], bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same with fp16 inputs.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <bool F16>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (F16)
        mma_f16_16816(d, a, b0, b1);
    else
        mma_bf16_16816(d, a, b0, b1);
}

// Four 8x8 b16 matrices to shared memory; thread t supplies the address of row
// t % 8 of matrix t / 8 and holds, in r[i], row t / 4, columns 2(t % 4) + 0..1
// of matrix i.
__device__ __forceinline__ void stmatrix_x4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(r0), "r"(r1),
                 "r"(r2), "r"(r3)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float f16_lo(uint32_t v) { return __low2float(*reinterpret_cast<__half2*>(&v)); }
__device__ __forceinline__ float f16_hi(uint32_t v) { return __high2float(*reinterpret_cast<__half2*>(&v)); }
// bf16x2 -> f16x2 (exact for values in f16's normal range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) { return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u)); }
// Four int8 codes (one 32-bit word, byte i = code of column i) as two f16x2
// values, exactly: each byte is biased to 0..255, placed in the low mantissa
// bits of 1024.0h (0x6400 | u = 1024 + u), and 1024 + 128 is subtracted.
__device__ __forceinline__ void i8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
    lo = *reinterpret_cast<uint32_t*>(&ha);
    hi = *reinterpret_cast<uint32_t*>(&hb);
}
// Four fp8 E4M3 codes (byte i = column i) as two f16x2 values equal to the
// codes' values divided by 256, exactly. E4M3 (sign, 4 exponent bits with bias
// 7, 3 mantissa bits) and f16 (bias 15) differ by 8 in the exponent bias, so
// placing a code's exponent and mantissa bits at the top of an f16's exponent
// and mantissa fields (and its sign on the sign bit) reads as value * 2^-8,
// subnormals included. Each byte goes to bits 15..8 of a 16-bit lane (byte
// permute), the exponent and mantissa bits move down by one, the sign stays.
__device__ __forceinline__ void e4m3x4_to_f16x2x2_div256(uint32_t w, uint32_t& lo, uint32_t& hi) {
    uint32_t a, b;
    asm("prmt.b32 %0, %1, 0, 0x1404;" : "=r"(a) : "r"(w));  // byte 0 -> bits 15..8, byte 1 -> bits 31..24
    asm("prmt.b32 %0, %1, 0, 0x3424;" : "=r"(b) : "r"(w));  // bytes 2, 3 likewise
    lo = (a & 0x80008000u) | ((a >> 1) & 0x3f803f80u);
    hi = (b & 0x80008000u) | ((b >> 1) & 0x3f803f80u);
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Programmatic dependent launch: wait for the preceding grid's results /
// allow the following grid to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::);
}

}  // namespace kvd
