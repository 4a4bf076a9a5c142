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

} // namespace rmsnorm
