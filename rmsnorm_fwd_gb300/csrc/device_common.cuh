// device_common.cuh -- element traits, vector memory access and reductions
// shared by the RMSNorm kernels (sm_103a).
//
// Vector width: every thread moves 16-byte (8 x bf16/f16, 4 x f32) or, on
// Blackwell, 32-byte vectors per instruction ("CuTeDSL at Perplexity",
// sections "Prefill and decode specialization" and "Blackwell support").
// Squares are accumulated in fp32 and the output is cast back to the element
// type with round-to-nearest-even (same page, section "QK Norm").
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace rmsnorm {

// ---------------------------------------------------------------- elements

// Two packed 16-bit elements (or one f32) per 32-bit word.
template <int DT> struct Elem;

template <> struct Elem<RMSNORM_F32> {
    static constexpr int kSize = 4;
    static constexpr int kPerWord = 1;
    __device__ static inline void widen(uint32_t u, float &a, float & /*b*/) { a = __uint_as_float(u); }
    __device__ static inline uint32_t narrow(float a, float /*b*/) { return __float_as_uint(a); }
    __device__ static inline float widen1(const void *p, int64_t i) { return static_cast<const float *>(p)[i]; }
    __device__ static inline void store1(void *p, int64_t i, float v) { static_cast<float *>(p)[i] = v; }
};

template <> struct Elem<RMSNORM_BF16> {
    static constexpr int kSize = 2;
    static constexpr int kPerWord = 2;
    // bf16 -> f32 is exact: the bf16 bits are the top half of the f32 bits.
    __device__ static inline void widen(uint32_t u, float &a, float &b)
    {
        a = __uint_as_float(u << 16);
        b = __uint_as_float(u & 0xFFFF0000u);
    }
    __device__ static inline uint32_t narrow(float a, float b)
    {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b); // .x = a (low half), .y = b
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ static inline float widen1(const void *p, int64_t i)
    {
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
    }
    __device__ static inline void store1(void *p, int64_t i, float v)
    {
        static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
    }
};

template <> struct Elem<RMSNORM_F16> {
    static constexpr int kSize = 2;
    static constexpr int kPerWord = 2;
    __device__ static inline void widen(uint32_t u, float &a, float &b)
    {
        __half2 h = *reinterpret_cast<__half2 *>(&u);
        float2 f = __half22float2(h);
        a = f.x;
        b = f.y;
    }
    __device__ static inline uint32_t narrow(float a, float b)
    {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ static inline float widen1(const void *p, int64_t i)
    {
        return __half2float(static_cast<const __half *>(p)[i]);
    }
    __device__ static inline void store1(void *p, int64_t i, float v)
    {
        static_cast<__half *>(p)[i] = __float2half_rn(v);
    }
};

// ---------------------------------------------------------------- vectors

template <int VB> struct alignas(VB) Vec {
    static constexpr int kWords = VB / 4;
    uint32_t w[kWords];
};

// Streaming load of x.  No .nc: x may be the output too (in-place), so the
// read-only path is not used.  Cache policy CP:
//   0: not kept in L1 (each byte is read once);
//   1: as 0, plus a 256-byte L2 prefetch hint (whole DRAM bursts);
//   2: .cs (streaming, evict-first in L1 and L2).
template <int CP>
__device__ inline void ld_stream(Vec<16> &v, const void *p)
{
    if (CP == 1)
        asm volatile("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                     : "l"(p));
    else if (CP == 2)
        asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                     : "l"(p));
    else
        asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                     : "l"(p));
}
template <int CP>
__device__ inline void ld_stream(Vec<32> &v, const void *p)
{
    if (CP == 1)
        asm volatile("ld.global.L1::no_allocate.L2::256B.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]),
                       "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                     : "l"(p));
    else if (CP == 2)
        asm volatile("ld.global.cs.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]),
                       "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                     : "l"(p));
    else
        asm volatile("ld.global.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]),
                       "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                     : "l"(p));
}

// Weight load: read-only for the whole kernel (y never overlaps it), reused
// by every row, so it goes through the non-coherent cached path.
__device__ inline void ld_weight(Vec<16> &v, const void *p)
{
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
}
__device__ inline void ld_weight(Vec<32> &v, const void *p)
{
    asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]),
                   "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
}

// Output store: written once, not re-read by this kernel.  CP as for loads
// (2 = .cs streaming store, otherwise not allocated in L1).
template <int CP>
__device__ inline void st_stream(void *p, const Vec<16> &v)
{
    if (CP == 2)
        asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                     ::"l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3])
                     : "memory");
    else
        asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};"
                     ::"l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3])
                     : "memory");
}
template <int CP>
__device__ inline void st_stream(void *p, const Vec<32> &v)
{
    if (CP == 2)
        asm volatile("st.global.cs.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                     ::"l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]),
                       "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                     : "memory");
    else
        asm volatile("st.global.L1::no_allocate.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                     ::"l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]),
                       "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                     : "memory");
}

// Hides the vector's words from the compiler's value numbering, so the fp32
// unpacked copies made for the sum of squares are not kept alive until the
// scale pass (the scale pass unpacks the words again; that costs one integer
// op per element and saves two registers per packed word).
template <int VB>
__device__ inline void reuse_barrier(Vec<VB> &v)
{
#pragma unroll
    for (int k = 0; k < Vec<VB>::kWords; ++k)
        asm("mov.b32 %0, %0;" : "+r"(v.w[k]));
}

// Sum of squares of one vector, accumulated into s (fp32).
template <int DT, int VB>
__device__ inline float sumsq(const Vec<VB> &v, float s)
{
#pragma unroll
    for (int k = 0; k < Vec<VB>::kWords; ++k) {
        float a, b = 0.f;
        Elem<DT>::widen(v.w[k], a, b);
        s = fmaf(a, a, s);
        if (Elem<DT>::kPerWord == 2)
            s = fmaf(b, b, s);
    }
    return s;
}

// out = (x * r) * w per element, rounded to the element type.
template <int DT, int VB>
__device__ inline void scale(Vec<VB> &out, const Vec<VB> &xv, const Vec<VB> &wv, float r)
{
#pragma unroll
    for (int k = 0; k < Vec<VB>::kWords; ++k) {
        float xa, xb = 0.f, wa, wb = 0.f;
        Elem<DT>::widen(xv.w[k], xa, xb);
        Elem<DT>::widen(wv.w[k], wa, wb);
        out.w[k] = Elem<DT>::narrow((xa * r) * wa, (xb * r) * wb);
    }
}

// ---------------------------------------------------------------- range guard
//
// The squares are summed in fp32 ("CuTeDSL at Perplexity", section "QK
// Norm"), but bf16 and f32 elements span fp32's whole exponent range: the sum
// S overflows to +inf once |x| reaches about 2^64, and squares below 2^-126
// lose bits (below 2^-150 all of them).  Either way the plain factor is
// wrong where the definition (mean of the squares, plus eps, reciprocal
// square root, in exact arithmetic) is not.  f16 elements cannot get there
// (their squares lie in [2^-48, 2^32]), so only bf16 and f32 bodies carry
// the guard.
//
// The guard is one compare per row.  S is trusted when it is finite and
// either at least 2^-100 (the squares lost to underflow are then at most
// hidden * 2^-150 <= 2^-124, below one part in 2^24 of S for rows up to 2^26
// elements) or eps >= 2^-120 (eps then outweighs what underflow lost by 2^29
// or more).  Otherwise the row's sum is formed again from k * x, a power of
// two: k = 2^-80 after an overflow (the rescaled squares stay below 2^96 and
// their sum below 2^122; squares that now underflow are below 2^10 against
// S >= 2^128), k = 2^100 after an underflow (every nonzero square of a bf16 or f32
// value becomes at least 2^-98, and a sum below 2^-100 becomes one below
// 2^100).  k * x is exact for every element that can matter.  A row holding
// an Inf or a NaN keeps its +inf or NaN sum: the plain factor is then what
// IEEE arithmetic gives (0 for +inf), as in the definition.
template <int DT>
constexpr bool kRangeGuard = DT != RMSNORM_F16;

__device__ inline bool sum_needs_rescale(float S, float eps)
{
    return S > 0x1.fffffep127f || (S < 0x1p-100f && eps < 0x1p-120f);
}

// The power of two the redo scales x by.
__device__ inline float rescale_k(float S)
{
    return S > 0x1.fffffep127f ? 0x1p-80f : 0x1p100f;
}

// Sum of the squares of k * x over one vector, accumulated into s.
template <int DT, int VB>
__device__ inline float sumsq_k(const Vec<VB> &v, float k, float s)
{
#pragma unroll
    for (int i = 0; i < Vec<VB>::kWords; ++i) {
        float a, b = 0.f;
        Elem<DT>::widen(v.w[i], a, b);
        a *= k;
        s = fmaf(a, a, s);
        if (Elem<DT>::kPerWord == 2) {
            b *= k;
            s = fmaf(b, b, s);
        }
    }
    return s;
}

// x <- 2^100 * x for one vector, exact (used only on rows whose elements
// are all below 2^-100 in magnitude, so nothing overflows).
template <int DT, int VB>
__device__ inline void scale_up(Vec<VB> &v)
{
#pragma unroll
    for (int i = 0; i < Vec<VB>::kWords; ++i) {
        float a, b = 0.f;
        Elem<DT>::widen(v.w[i], a, b);
        v.w[i] = Elem<DT>::narrow(a * 0x1p100f, b * 0x1p100f);
    }
}

// The factor from the rescaled sum Sk = sum (k x)^2:
//   r = 1 / sqrt(Sk / (k^2 n) + eps) = k * rsqrt(Sk / n + (eps * k) * k),
// with (eps * k) * k exact where it matters (on the 2^100 side eps < 2^-120,
// so it stays below 2^80; on the 2^-80 side it is exact unless it falls
// below 2^-126, where it is negligible against Sk / n >= 2^-58).
// k * rho is exact while it is a normal float.  It would overflow only on the
// 2^100 side with rho >= 2^27, i.e. a row whose RMS with eps is below 2^-127
// (eps = 0 and every element tiny); then `up` is set, r = rho, and the caller
// multiplies x by 2^100 before scaling (scale_up; exact there), so that
// (x * 2^100) * rho = x * r without leaving the float range.  An all-zero
// row with eps = 0 gives rho = inf, up, and 0 * inf = NaN, as the definition.
struct Factor {
    float r;
    bool up;
};
__device__ inline Factor rescaled_factor(float Sk, float k, float n, float eps)
{
    const float rho = rsqrtf(Sk / n + (eps * k) * k);
    Factor f;
    f.up = k > 1.f && !(rho < 0x1p27f);
    f.r = f.up ? rho : k * rho;
    return f;
}

// For bodies whose row total is combined from several partial sums held in
// binary64 (thread-block clusters, the grid variant): the total's (Sk, k)
// form for rescaled_factor -- k = 1 when it fits fp32's trusted range, else
// the power of two sum_needs_rescale would have chosen.  D * k^2 is exact.
__device__ inline void wide_total(double D, float eps, float &Sk, float &k)
{
    if (D > 0x1.fffffep127) {
        k = 0x1p-80f;
        Sk = static_cast<float>(D * 0x1p-160);
    } else if (D < 0x1p-100 && eps < 0x1p-120f) {
        k = 0x1p100f;
        Sk = static_cast<float>(D * 0x1p200);
    } else {
        k = 1.f;
        Sk = static_cast<float>(D);
    }
}

// ---------------------------------------------------------------- epilogues

// out = (x * r) * (w + bias) per element -- the weight offset WEIGHT_BIAS of
// "CuTeDSL at Perplexity", section "QK Norm" -- rounded to the element type.
template <int DT, int VB>
__device__ inline void scale_bias(Vec<VB> &out, const Vec<VB> &xv, const Vec<VB> &wv, float r,
                                  float bias)
{
#pragma unroll
    for (int k = 0; k < Vec<VB>::kWords; ++k) {
        float xa, xb = 0.f, wa, wb = 0.f;
        Elem<DT>::widen(xv.w[k], xa, xb);
        Elem<DT>::widen(wv.w[k], wa, wb);
        out.w[k] = Elem<DT>::narrow((xa * r) * (wa + bias), (xb * r) * (wb + bias));
    }
}

// Block-scaled output formats ("CuTeDSL at Perplexity", section "Blackwell
// support": MXFP8, MXFP4 and NVFP4, absolute maxima over blocks of 32 or 16
// elements).  MX formats (OCP Microscaling v1.0): 32-element blocks, E8M0
// power-of-two scale 2^(floor(log2 max) - kEmax), kEmax the element format's
// largest exponent.  NVFP4 (NVIDIA's description): 16-element blocks, E4M3
// scale E4M3(max / (6 g)) times a per-tensor fp32 scale g.
enum { kQMxfp8 = 0, kQMxfp4 = 1, kQNvfp4 = 2 };
template <int Q> struct QFmt;
template <> struct QFmt<kQMxfp8> {
    static constexpr int kBlock = 32, kBits = 8, kEmax = 8;
};
template <> struct QFmt<kQMxfp4> {
    static constexpr int kBlock = 32, kBits = 4, kEmax = 2;
};
template <> struct QFmt<kQNvfp4> {
    static constexpr int kBlock = 16, kBits = 4, kEmax = 0;
};

// Geometry of one vector's output: its kElems elements become kCodeBytes
// code bytes, and one scale block spans kLanes consecutive vectors (held by
// kLanes consecutive lanes).
template <int DT, int VB, int Q> struct QGeo {
    static constexpr int kElems = VB / Elem<DT>::kSize;
    static constexpr int kLanes = QFmt<Q>::kBlock / kElems;
    static constexpr int kCodeBytes = kElems * QFmt<Q>::kBits / 8;
    static_assert(kLanes >= 1, "a vector must not straddle two scale blocks");
};

// Four fp32 values to four E4M3 codes, value i in byte i.  The conversion
// instruction rounds to nearest-even and saturates finite overflow to +-448
// (.satfinite); a NaN stays NaN.  The instruction puts its first source in
// the upper byte of each 16-bit pair.
__device__ inline uint32_t e4m3x4(float a0, float a1, float a2, float a3)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
    return r;
}

// Eight fp32 values to eight E2M1 codes packed in a word, value i in
// nibble i (the even element of each byte in its low nibble).  Nearest-even,
// saturating at +-6 (.satfinite).  The instruction puts its first source in
// the upper nibble of its byte.
__device__ inline uint32_t e2m1x8(const float (&f)[8])
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]),
          "f"(f[7]));
    return r;
}

// Four fp32 values to four E2M1 codes in the low 16 bits.
__device__ inline uint32_t e2m1x4(const float (&f)[4])
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1;\n\t.reg .b16 h;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "mov.b16 h, {b0, b1};\n\t"
        "cvt.u32.u16 %0, h;\n\t}"
        : "=r"(r)
        : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]));
    return r;
}

// The E4M3 code of a non-negative value (nearest-even, saturating at 448, a
// NaN giving 0x7F) and the value that code stands for.
__device__ inline uint32_t e4m3_code(float t)
{
    uint16_t h;
    asm("{\n\t.reg .b16 c;\n\tcvt.rn.satfinite.e4m3x2.f32 c, %1, %2;\n\tmov.b16 %0, c;\n\t}"
        : "=h"(h)
        : "f"(0.f), "f"(t));
    return h & 0xFFu;
}
__device__ inline float e4m3_value(uint32_t code)
{
    uint32_t hh;
    asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
        : "=r"(hh)
        : "r"(code));
    return __half2float(__ushort_as_half(static_cast<unsigned short>(hh & 0xFFFFu)));
}

// Stores NB = 2, 4, 8 or 16 code bytes (not allocated in L1).
template <int NB>
__device__ inline void st_codes(void *p, const uint32_t (&w)[(NB + 3) / 4])
{
    if constexpr (NB == 2)
        asm volatile("st.global.L1::no_allocate.u16 [%0], %1;" ::"l"(p),
                     "h"(static_cast<unsigned short>(w[0]))
                     : "memory");
    else if constexpr (NB == 4)
        asm volatile("st.global.L1::no_allocate.u32 [%0], %1;" ::"l"(p), "r"(w[0]) : "memory");
    else if constexpr (NB == 8)
        asm volatile("st.global.L1::no_allocate.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(w[0]),
                     "r"(w[1])
                     : "memory");
    else
        asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p),
                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
}

// Two fp32 lanes in one 64-bit register for the sm_100-family packed
// arithmetic (add / mul .rn.f32x2: one instruction for two IEEE operations,
// each rounded exactly as its scalar form).
__device__ inline uint64_t f2(float a, float b)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ inline void f2split(uint64_t v, float &a, float &b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ inline uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ inline uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Element pair p of a vector (elements 2p and 2p + 1) widened to fp32.
template <int DT, int VB>
__device__ inline uint64_t widen_pair(const Vec<VB> &v, int p)
{
    float a, b = 0.f;
    if (Elem<DT>::kPerWord == 2) {
        Elem<DT>::widen(v.w[p], a, b);
    } else {
        float u;
        Elem<DT>::widen(v.w[2 * p], a, u);
        Elem<DT>::widen(v.w[2 * p + 1], b, u);
    }
    return f2(a, b);
}

// scale() with two elements per packed fp32x2 instruction: the same IEEE
// products in the same order, so the same result.  Fewer instructions but a
// register or two more; the block-per-row bodies use it.
template <int DT, int VB>
__device__ inline void scale_packed(Vec<VB> &out, const Vec<VB> &xv, const Vec<VB> &wv, float r)
{
    constexpr int P = VB / Elem<DT>::kSize / 2;
    const uint64_t r2 = f2(r, r);
    float f[2 * P];
#pragma unroll
    for (int p = 0; p < P; ++p)
        f2split(mul2(mul2(widen_pair<DT, VB>(xv, p), r2), widen_pair<DT, VB>(wv, p)), f[2 * p],
                f[2 * p + 1]);
#pragma unroll
    for (int k = 0; k < Vec<VB>::kWords; ++k)
        out.w[k] = Elem<DT>::kPerWord == 2 ? Elem<DT>::narrow(f[2 * k], f[2 * k + 1])
                                           : Elem<DT>::narrow(f[k], 0.f);
}

// scale_bias() in the packed form: (x * r) * (w + bias), each operation an
// IEEE fp32 one in the scalar order, so the same result.
template <int DT, int VB>
__device__ inline void scale_bias_packed(Vec<VB> &out, const Vec<VB> &xv, const Vec<VB> &wv,
                                         float r, float bias)
{
    constexpr int P = VB / Elem<DT>::kSize / 2;
    const uint64_t r2 = f2(r, r), b2 = f2(bias, bias);
    float f[2 * P];
#pragma unroll
    for (int p = 0; p < P; ++p)
        f2split(mul2(mul2(widen_pair<DT, VB>(xv, p), r2), add2(widen_pair<DT, VB>(wv, p), b2)),
                f[2 * p], f[2 * p + 1]);
#pragma unroll
    for (int k = 0; k < Vec<VB>::kWords; ++k)
        out.w[k] = Elem<DT>::kPerWord == 2 ? Elem<DT>::narrow(f[2 * k], f[2 * k + 1])
                                           : Elem<DT>::narrow(f[k], 0.f);
}

// Sum of squares of one vector, element by element in the order sumsq()
// uses, so the total is bit-identical to it.  16-bit elements go straight
// into the mixed-precision fma (bf16 / f16 operands, fp32 accumulator): the
// product of two 16-bit values is exact in fp32 and the fma rounds once, as
// the fp32 fma on the widened values does, without the widening.
template <int DT, int VB>
__device__ inline float sumsq_mixed(const Vec<VB> &v, float s)
{
    if constexpr (DT == RMSNORM_F32) {
        return sumsq<DT, VB>(v, s);
    } else {
#pragma unroll
        for (int k = 0; k < Vec<VB>::kWords; ++k) {
            if constexpr (DT == RMSNORM_BF16)
                asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
                    "fma.rn.f32.bf16 %0, lo, lo, %0;\n\tfma.rn.f32.bf16 %0, hi, hi, %0;\n\t}"
                    : "+f"(s)
                    : "r"(v.w[k]));
            else
                asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
                    "fma.rn.f32.f16 %0, lo, lo, %0;\n\tfma.rn.f32.f16 %0, hi, hi, %0;\n\t}"
                    : "+f"(s)
                    : "r"(v.w[k]));
        }
        return s;
    }
}

// max(|a|, |b|, m), a NaN in any giving NaN (three-input max.NaN).
__device__ inline float absmax3_nan(float a, float b, float m)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(fabsf(a)), "f"(fabsf(b)), "f"(m));
    return r;
}

// max(a, m), a NaN in either giving NaN.
__device__ inline float max_nan(float a, float m)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(m));
    return r;
}

// 1 / a by the hardware reciprocal (within one unit in the last place;
// subnormal inputs kept).  The NVFP4 scale and element decisions it feeds
// are checked against the exact quotients with a 1e-5 relative band.
__device__ inline float rcp_approx(float a)
{
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

// 1 / a by the hardware reciprocal with subnormal inputs and results
// flushed to zero: for an `a` and a 1 / a that are both normal floats.
__device__ inline float rcp_approx_ftz(float a)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

// The exact products x * w of element pair p of two 16-bit vectors, in fp32:
// the mixed-precision fma with a -0 addend (the product of two bf16 or two
// f16 values has at most 16 or 22 significant bits, so it is exact in fp32
// unless it leaves fp32's normal range, and x * w + (-0) is x * w with its
// sign, zeros included).
template <int DT>
__device__ inline void exact_products(uint32_t xw, uint32_t ww, float &a, float &b)
{
    static_assert(DT != RMSNORM_F32, "16-bit elements only");
    if constexpr (DT == RMSNORM_BF16)
        asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\tmov.b32 {xl, xh}, %2;\n\tmov.b32 {wl, wh}, %3;\n\t"
            "fma.rn.f32.bf16 %0, xl, wl, 0f80000000;\n\tfma.rn.f32.bf16 %1, xh, wh, 0f80000000;\n\t}"
            : "=f"(a), "=f"(b)
            : "r"(xw), "r"(ww));
    else
        asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\tmov.b32 {xl, xh}, %2;\n\tmov.b32 {wl, wh}, %3;\n\t"
            "fma.rn.f32.f16 %0, xl, wl, 0f80000000;\n\tfma.rn.f32.f16 %1, xh, wh, 0f80000000;\n\t}"
            : "=f"(a), "=f"(b)
            : "r"(xw), "r"(ww));
}

// Per-launch constants of a block-scaled epilogue.
struct QParams {
    float bias; // weight offset
    float g;    // NVFP4 per-tensor scale
};
__device__ inline QParams q_params(float bias, float g)
{
    QParams p;
    p.bias = bias;
    p.g = g;
    return p;
}

// v = (x * r) * (w + bias) of one vector, two elements per packed
// instruction, and max |v| of this lane (NaN-propagating).
template <int DT, int VB>
__device__ inline float q_values(const Vec<VB> &xv, const Vec<VB> &wv, float r, float bias,
                                 uint64_t (&v)[VB / Elem<DT>::kSize / 2])
{
    constexpr int P = VB / Elem<DT>::kSize / 2;
    const uint64_t r2 = f2(r, r), b2 = f2(bias, bias);
    float m = 0.f;
#pragma unroll
    for (int p = 0; p < P; ++p) {
        v[p] = mul2(mul2(widen_pair<DT, VB>(xv, p), r2), add2(widen_pair<DT, VB>(wv, p), b2));
        float a, b;
        f2split(v[p], a, b);
        m = absmax3_nan(a, b, m);
    }
    return m;
}

// NaN-propagating maximum over the kLanes lanes of a scale block.
template <int LPB>
__device__ inline float block_max(float m)
{
#pragma unroll
    for (int off = 1; off < LPB; off <<= 1)
        m = max_nan(__shfl_xor_sync(0xFFFFFFFFu, m, off, 32), m);
    return m;
}

// One vector of a block-scaled epilogue (QFmt above).
//
// The values are v = (x * r) * (w + bias) in fp32.  The block maximum of |v|
// is a NaN-propagating max (a NaN or an Inf in the block must reach the
// scale; fmaxf would drop a NaN), reduced over the block's kLanes lanes with
// butterfly shuffles.  MX formats: the biased exponent e of the maximum gives
// the shared exponent floor(log2 max) - kEmax = e - 127 - kEmax, clamped at
// -127: E8M0 code max(e - kEmax, 0), or 0xFF when e = 255 (Inf / NaN);
// scaling by 2^(127 - code) is exact.  NVFP4: the scale code is
// E4M3(max * (1 / (6 g))) and the values are multiplied by
// 1 / (value(code) * g) (by 0 when the scale is 0), both reciprocals from
// rcp.approx.  The conversions round each scaled value to the element format.
//
// With XW (16-bit elements, weight offset -0 and, for NVFP4, a per-tensor
// scale g in [2^-117, 2^100], so that every value(code) * g and its
// reciprocal are normal floats and the flush-to-zero reciprocal serves; the
// launch picks this instantiation) the values are formed the other way round,
// as the exact products u = x * w (one mixed-precision fma per element, no
// widening), the block maximum as max |u| * r and the scaled values as
// u * (r * mul): the same quantities up to one or two fp32 roundings (the
// decisions they feed are checked against the exact values with a 1e-5
// relative band).  That holds while the products and the block maximum are
// normal fp32 numbers well away from overflow.  The return value says that
// this lane's block is outside that range -- max |u| or max |u| * r outside
// [2^-100, 2^100): zero blocks, NaN, Inf, extreme ranges -- and that what it
// stored there must be replaced: the caller then writes the vectors of the
// whole warp again in the order above, from x and w read again (a rare,
// warp-uniform branch after the warp's last vector, so the common path holds
// no registers for it; neither the codes nor the scales may overlap x or w).
// An element below 2^-119 of its block's maximum is below half the smallest
// nonzero code of every format, so at 2^-100 nothing that can reach a code
// is subnormal.  Without XW the return value is false.
//
// Every lane of the warp must call this (the shuffles span the full warp);
// `live` says whether this lane's vector is part of the row.  The lane
// holding the first vector of a block (`leader`) stores the scale byte.
template <int DT, int VB, int Q, bool XW>
__device__ inline bool q_emit(const Vec<VB> &xv, const Vec<VB> &wv, float r, const QParams &qp,
                              bool live, bool leader, void *q, uint8_t *scale)
{
    static_assert(!XW || DT != RMSNORM_F32, "exact products: 16-bit elements only");
    using G = QGeo<DT, VB, Q>;
    constexpr int NE = G::kElems;
    constexpr int LPB = G::kLanes;
    constexpr int P = NE / 2;
    uint64_t v[P];
    float m, fac;
    bool bad = false;
    if constexpr (XW) {
        m = 0.f;
#pragma unroll
        for (int p = 0; p < P; ++p) {
            float a, b;
            exact_products<DT>(xv.w[p], wv.w[p], a, b);
            v[p] = f2(a, b);
            m = absmax3_nan(a, b, m);
        }
        m = block_max<LPB>(m);
        const float mr = m * r;
        bad = !(m >= 0x1p-100f && m < 0x1p100f && mr >= 0x1p-100f && mr < 0x1p100f);
        m = mr;
        fac = r;
    } else {
        m = block_max<LPB>(q_values<DT, VB>(xv, wv, r, qp.bias, v));
        fac = 1.f;
    }
    uint32_t code;
    float f;
    if constexpr (Q == kQNvfp4) {
        code = e4m3_code(m * rcp_approx(6.f * qp.g));
        const float d = e4m3_value(code);
        const float dg = d * qp.g;
        f = (d == 0.f ? 0.f : (XW ? rcp_approx_ftz(dg) : rcp_approx(dg))) * fac;
    } else if constexpr (XW) {
        // A block in the trusted range has 2^-100 <= max |u| * r < 2^100, so
        // its biased exponent e lies in [27, 227): the code is e - kEmax, and
        // r * 2^(127 - code) -- a normal float, the scaled block maximum being
        // in [2^kEmax, 2^(kEmax + 1)) -- is r with 127 - code added to its
        // exponent field.  Blocks outside the range are written again (above).
        constexpr uint32_t EM = QFmt<Q>::kEmax;
        const uint32_t eb = __float_as_uint(m) & 0x7F800000u; // m >= 0 or NaN
        code = (eb >> 23) - EM;
        f = __uint_as_float(__float_as_uint(r) + ((127u + EM) << 23) - eb);
    } else {
        constexpr uint32_t EM = QFmt<Q>::kEmax;
        const uint32_t e = __float_as_uint(m) >> 23;
        code = e == 255u ? 255u : (e > EM ? e - EM : 0u);
        f = __uint_as_float(code == 255u ? 0x3F800000u : (254u - code) << 23) * fac;
    }
    const uint64_t mul2v = f2(f, f);
    float sv[NE];
#pragma unroll
    for (int p = 0; p < P; ++p)
        f2split(mul2(v[p], mul2v), sv[2 * p], sv[2 * p + 1]);
    constexpr int NB = G::kCodeBytes;
    uint32_t words[(NB + 3) / 4];
    if constexpr (QFmt<Q>::kBits == 8) {
#pragma unroll
        for (int j = 0; j < NE / 4; ++j)
            words[j] = e4m3x4(sv[4 * j], sv[4 * j + 1], sv[4 * j + 2], sv[4 * j + 3]);
    } else if constexpr (NE == 4) {
        const float f4[4] = {sv[0], sv[1], sv[2], sv[3]};
        words[0] = e2m1x4(f4);
    } else {
#pragma unroll
        for (int j = 0; j < NE / 8; ++j) {
            const float f8[8] = {sv[8 * j], sv[8 * j + 1], sv[8 * j + 2], sv[8 * j + 3],
                                 sv[8 * j + 4], sv[8 * j + 5], sv[8 * j + 6], sv[8 * j + 7]};
            words[j] = e2m1x8(f8);
        }
    }
    if (live) {
        st_codes<NB>(q, words);
        if (leader)
            *scale = static_cast<uint8_t>(code);
    }
    return bad;
}

// ---------------------------------------------------------------- launch order

// Programmatic dependent launch.  Every kernel calls pdl_begin() before its
// first global-memory access: the wait returns once the grid this launch
// depends on has completed and its writes are visible (immediately when the
// launch carries no programmatic dependency), and the trigger lets the next
// dependent launch be scheduled as soon as every block of this grid has
// started, so its blocks take SM slots while this grid's last blocks finish.
__device__ inline void pdl_begin()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- reductions

// Butterfly sum over aligned groups of WIDTH lanes (WIDTH a power of two
// <= 32); every lane of the group ends with the group's total.
template <int WIDTH>
__device__ inline float group_allreduce(float s)
{
#pragma unroll
    for (int off = WIDTH / 2; off > 0; off >>= 1)
        s += __shfl_xor_sync(0xFFFFFFFFu, s, off, 32);
    return s;
}

// The row factor, in the order the steps are listed for RMSNorm in "Build a
// GPU compiler from scratch ... (Emmy)", section "Tensor IR": divide the sum
// of squares by the count, add epsilon, reciprocal square root.
__device__ inline float row_factor(float S, float n, float eps)
{
    return rsqrtf(S / n + eps);
}

// The count n of a row and what the division by it needs: when n is a power
// of two, S / n is S * (1 / n) exactly (a product by a power of two rounds
// as the quotient does, subnormal results included), which the block-scaled
// bodies take instead of the division (the plain ones keep the division:
// their register caps leave no room for the flag).
struct RowCount {
    float n, inv;
    bool pow2;
};
__device__ inline RowCount row_count(int32_t hidden)
{
    RowCount c;
    c.n = static_cast<float>(hidden);
    c.pow2 = (hidden & (hidden - 1)) == 0;
    c.inv = c.pow2 ? __uint_as_float(static_cast<uint32_t>(127 - __ffs(hidden) + 1) << 23) : 0.f;
    return c;
}
__device__ inline float row_factor(float S, const RowCount &c, float eps)
{
    return rsqrtf((c.pow2 ? S * c.inv : S / c.n) + eps);
}

} // namespace rmsnorm
