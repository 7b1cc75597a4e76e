// common.cuh -- small device helpers (inline PTX wrappers) shared by the
// attention kernels of libattn.  sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>

#include "internal.h"

namespace attn {

// ------------------------------------------------------------ type helpers

template <int KIND> struct Elem;            // storage type by dtype code
template <> struct Elem<DT_BF16> { using T = __nv_bfloat16; static constexpr int bytes = 2; };
template <> struct Elem<DT_FP16> { using T = __half;        static constexpr int bytes = 2; };
template <> struct Elem<DT_E4M3> { using T = uint8_t;       static constexpr int bytes = 1; };
template <> struct Elem<DT_FP32> { using T = float;         static constexpr int bytes = 4; };

__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_float(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_float(float x) { return x; }

// pack two floats into one 32-bit register of the MMA operand type
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
}

// Four e4m3 values (the bytes of w, lowest first) as the fp16 bit patterns
// of value * 2^-8, two per register (lo: bytes 0, 1; hi: bytes 2, 3).  The
// e4m3 sign, exponent and mantissa fields drop into the fp16 fields
// unchanged -- only the exponent bias differs (7 against 15), hence the
// factor 2^-8, which callers fold into their scales -- and e4m3 subnormals
// land on fp16 subnormals exactly.  Each byte is sign-extended to 16 bits
// (prmt with the sign-replicate selector bit), shifted into place, and
// masked to sign | low 7 bits.  The e4m3 NaN pattern S.1111.111 is not
// special-cased: it reads as +-480 * 2^-8.
__device__ __forceinline__ void e4m3x4_to_h2x2_lo8(uint32_t w, uint32_t &lo, uint32_t &hi) {
    uint32_t a, b;
    asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(a) : "r"(w));
    asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(b) : "r"(w));
    lo = (a << 7) & 0xBF80BF80u;
    hi = (b << 7) & 0xBF80BF80u;
}
// 2^8: the factor e4m3x4_to_h2x2_lo8 leaves out
constexpr float kE4m3Lo8Scale = 256.f;

// Byte I of x and byte I of y (two e4m3 values) as one fp16x2 register of
// value * 2^-8 (x's value in the low half): the same field placement as
// e4m3x4_to_h2x2_lo8, with prmt taking one byte from each register
template <int I>
__device__ __forceinline__ uint32_t e4m3_pair_to_h2_lo8(uint32_t x, uint32_t y) {
    static_assert(I >= 0 && I < 4, "byte index");
    constexpr uint32_t sel = (uint32_t)I | ((8u | I) << 4) | ((4u + I) << 8) | ((12u + I) << 12);
    uint32_t a;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(a) : "r"(x), "r"(y), "n"(sel));
    return (a << 7) & 0xBF80BF80u;
}

// ------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared async copy; src_bytes = 0 zero-fills the chunk
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// D = A * B + D, m16n8k16, fp32 accumulate; BF16 selects bf16 vs f16 inputs
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// D += A * B with e4m3 operands (m16n8k32, fp32 accumulators): a thread
// holds four A bytes per register (rows g and g + 8, k offsets 4t and
// 16 + 4t) and four B bytes per register (k offsets 4t and 16 + 4t of
// column g), g = lane / 4, t = lane % 4
__device__ __forceinline__ void mma16832_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ int4 ldg_nc16(const void *p) {
    int4 v;
    asm volatile("ld.global.nc.v4.s32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// raise bits of the device error word (first writer wins nothing; OR only)
// tanh(y) = 1 - 2 / (1 + e^(2y)), e^(2y) = 2^(2 y log2 e) by ex2; the
// exponent is clamped to +-60, where the result is +-1 in fp32 anyway.
// Absolute error about 1e-7 (the soft cap multiplies it by the cap).
__device__ __forceinline__ float tanh_ex2(float y) {
    const float t = fminf(fmaxf(2.8853900817779268f * y, -60.f), 60.f);
    return 1.f - __fdividef(2.f, 1.f + ex2(t));
}

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialisation, so it may be scheduled while the
// previous kernel in the stream drains.  pdl_wait() blocks until that
// kernel has completed and its writes are visible (it returns at once when
// there is none); every thread calls it before its first global-memory
// access and before any exit, so a kernel never completes ahead of its
// predecessor.  pdl_trigger() lets the next kernel be scheduled once every
// CTA of this one has triggered or exited.
// named barrier ID (1..15; 0 is __syncthreads) of COUNT threads, whole
// warps; a constant id lets the compiler reserve only the barriers in use
template <int ID, int COUNT>
__device__ __forceinline__ void named_bar_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(COUNT) : "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void raise_error(unsigned *err, unsigned bits) {
    if (err) atomicOr(err, bits);
}

// byte offset of 16-byte chunk c of row r in a tile whose rows are
// row_bytes long (a multiple of 128): chunks are XOR-swizzled by r & 7 so
// that eight consecutive rows' chunk c land in eight different bank groups
__device__ __forceinline__ uint32_t swz(int r, int c, int row_bytes) {
    return (uint32_t)(r * row_bytes + ((c ^ (r & 7)) << 4));
}

}  // namespace attn
