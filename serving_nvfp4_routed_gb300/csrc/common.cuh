// common.cuh -- device helpers and host bookkeeping shared by the kernels of
// libnvfp4moe.  Nothing here is shared with the CPU oracle.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "nvfp4moe.h"

namespace nvfp4 {

// ---------------------------------------------------------------------------
// host: launch accounting and optional per-kernel event timing
// ---------------------------------------------------------------------------
void launch_begin(const char* name, cudaStream_t s);
void launch_end(const char* name, cudaStream_t s);
int num_sms();
int device_cc_major();
// nvfp4_set_kernel_choice: 0 by shape, 1 decode-shaped, 2 prompt-shaped,
// 3 decode-shaped as two launches, 4 decode-shaped as one persistent launch.
int kernel_choice();

#define NVFP4_LAUNCH(name, stream, ...)            \
    do {                                           \
        ::nvfp4::launch_begin(name, stream);       \
        __VA_ARGS__;                               \
        ::nvfp4::launch_end(name, stream);         \
    } while (0)

// Programmatic dependent launch: a kernel may be scheduled while its
// predecessor on the stream drains; every kernel of the library waits for
// its predecessor's completion (and memory) before touching global memory.
bool pdl_enabled();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

inline nvfp4_status last_launch_status() {
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Carves consecutive 256-byte-aligned regions out of a workspace.
struct Carver {
    char* base;
    size_t off = 0;
    explicit Carver(void* b) : base(static_cast<char*>(b)) {}
    template <class T>
    T* take(size_t count) {
        off = align_up(off, 256);
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
};

// ---------------------------------------------------------------------------
// device: number formats (inline PTX conversions of sm_100-family)
// ---------------------------------------------------------------------------

// fp32 -> e4m3 byte, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return r & 0xFFu;
}

// Two e4m3 bytes (low byte first) -> f16x2 (exact: every e4m3 value is an f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
    uint32_t r;
    uint16_t in = static_cast<uint16_t>(two_bytes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(in));
    return r;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    uint32_t h2 = e4m3x2_to_f16x2(b & 0xFFu);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Eight fp32 -> eight e2m1 codes (round to nearest even, saturating to +-6),
// element i in bits [4i, 4i+4).  The conversion keeps the sign of an input
// that rounds to zero (-0.1 and -0.0 give code 8, -0), as the format's
// definition does: checked on sm_103a for -0.0, -1e-30, -0.1 and -0.25.
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float v[8]) {
    uint32_t r;
    asm("{\n"
        ".reg .b8 b0, b1, b2, b3;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
        "mov.b32 %0, {b0, b1, b2, b3};\n"
        "}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// A quotient fl(v / d) for the e2m1 rounding that follows, given r = fl(1/d).
// v * r (two roundings) is within 3 ulp of fl(v / d), so both give the same
// e2m1 code unless the quotient lies within a few ulp of a number whose
// significand is 1, 1.25, 1.5 or 1.75: a superset of the e2m1 rounding
// boundaries (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5).  Only there (and for
// inf / NaN, whose low significand bits are zero) is the correctly rounded
// division taken, so the code is always that of fl(v / d).
__device__ __forceinline__ bool e2m1_quotient_near(float q) {
    return ((__float_as_uint(q) + 4u) & 0x1FFFFFu) <= 8u;
}
__device__ __forceinline__ float e2m1_quotient(float v, float d, float r) {
    const float q = __fmul_rn(v, r);
    if (e2m1_quotient_near(q)) return __fdiv_rn(v, d);
    return q;
}

// Eight e2m1 codes (one 32-bit word, element 0 in the low nibble) -> four
// f16x2 words, out[i] = (element 2i in the low half, element 2i+1 high).
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t out[4]) {
    asm("{\n"
        ".reg .b8 b0, b1, b2, b3;\n"
        "mov.b32 {b0, b1, b2, b3}, %4;\n"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n"
        "}"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
        : "r"(w));
}

// e2m1 codes of two values as one byte (lo in the low nibble).
__device__ __forceinline__ uint32_t e2m1x2_byte(float lo, float hi) {
    uint32_t r;
    asm("{\n.reg .b8 b;\ncvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\nmov.b32 %0, {b, b, b, b};\n}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r & 0xFFu;  // (the sign of a zero is kept, as in f32x8_to_e2m1x8)
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}

// Broadcast the f16 in the low (hi=0) or high (hi=1) half to both halves.
__device__ __forceinline__ uint32_t f16x2_bcast(uint32_t v, int hi) {
    return __byte_perm(v, 0u, hi ? 0x3232u : 0x1010u);  // one byte permute
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t*>(&b);
}

__device__ __forceinline__ float round_bf16(float v) { return bf16_bits_to_f32(f32_to_bf16_bits(v)); }

// 2^e as an fp32 (e in [-126, 127]).
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// Power-of-two exponent s for a row with max |x| = amax such that
// amax * 2^-s lies in [2^14, 2^15): the row then fits f16 with its largest
// element near the top of the f16 range.
__device__ __forceinline__ int row_exponent(float amax) {
    if (!(amax > 0.0f)) return 0;
    int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127;
    if (e < -126) e = -126;  // subnormal amax
    int s = e - 14;
    return s < -100 ? -100 : (s > 100 ? 100 : s);
}

// Warp-level mma: D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col).
__device__ __forceinline__ void mma_16816(float c[4], const uint32_t a[4], const uint32_t b[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Fire-and-forget fp32x4 add to global memory (no return value).
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Non-negative float atomic max through its bit pattern (monotone for >= 0).
__device__ __forceinline__ void atomic_max_nonneg(float* addr, float v) {
    atomicMax(reinterpret_cast<unsigned int*>(addr), __float_as_uint(v));
}

}  // namespace nvfp4
