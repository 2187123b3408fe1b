// Device helpers shared by the kernel translation units (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mkv_internal.h"

namespace mkv {
namespace dev {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// 16-byte non-coherent load that stays in L1 (for rows read twice in a row).
__device__ __forceinline__ uint4 ld_nc(const void *p)
{
    uint4 r;
    asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v)
{
    *reinterpret_cast<uint4 *>(p) = v;
}

// Streaming 16-byte store (evict-first: the compacted cache is not re-read
// by this path).
__device__ __forceinline__ void st_stream(void *p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Eight bf16 values of a 16-byte chunk, widened exactly to fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float f[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Eight E4M3 codes (OCP 8-bit floating point, E4M3: sign, 4 exponent bits
// with bias 7, 3 mantissa bits, subnormals at exponent field 0), widened
// exactly to fp32: the conversion instruction takes two codes to two fp16
// (every finite E4M3 value, 2^-9 .. 448, is an fp16 value), and fp16 ->
// fp32 is exact. Element order is kept: the code in the lower byte becomes
// the lower half. The NaN codes are outside the contract.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint16_t codes)
{
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(codes));
    float lo, hi;
    asm("{ .reg .f16 a, b; mov.b32 {a, b}, %2; cvt.f32.f16 %0, a; cvt.f32.f16 %1, b; }"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
    return make_float2(lo, hi);
}

__device__ __forceinline__ void e4m3x8_to_f32(const uint2 v, float f[8])
{
    const uint32_t w[2] = {v.x, v.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float2 a = e4m3x2_to_f32((uint16_t)(w[i] & 0xFFFFu));
        const float2 b = e4m3x2_to_f32((uint16_t)(w[i] >> 16));
        f[4 * i + 0] = a.x;
        f[4 * i + 1] = a.y;
        f[4 * i + 2] = b.x;
        f[4 * i + 3] = b.y;
    }
}

// Two E4M3 codes to two fp16 values (exact), lower byte to lower half.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t codes)
{
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)codes));
    return h;
}

// a0 += lower half of h, a1 += upper half, each in fp32 with one rounding:
// the mixed-precision add widens its fp16 operand exactly, so the bits are
// those of widening first and adding in fp32.
__device__ __forceinline__ void add_f16x2(uint32_t h, float &a0, float &a1)
{
    asm("{ .reg .f16 lo, hi; mov.b32 {lo, hi}, %2; add.rn.f32.f16 %0, lo, %0; add.rn.f32.f16 %1, hi, %1; }"
        : "+f"(a0), "+f"(a1)
        : "r"(h));
}

// d0 = (lower half of h) - c0, d1 = (upper half) - c1, in fp32 with one
// rounding each (the fp16 operand is widened exactly).
__device__ __forceinline__ void sub_f16x2(uint32_t h, float c0, float c1, float &d0, float &d1)
{
    asm("{ .reg .f16 lo, hi; mov.b32 {lo, hi}, %4; sub.rn.f32.f16 %0, lo, %2; sub.rn.f32.f16 %1, hi, %3; }"
        : "=f"(d0), "=f"(d1)
        : "f"(c0), "f"(c1), "r"(h));
}

__device__ __forceinline__ uint2 ld_stream8(const void *p)
{
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

// A cache row split into chunks of 8 consecutive elements: 16 bytes of bf16
// (ES = 2) or 8 bytes of E4M3 (ES = 1). Lane q of a row's 8 lanes takes the
// chunks at elements 64k + 8q, k < d / 64, whatever the element type.
template <int ES>
struct Chunk;

__device__ __forceinline__ uint2 ld_nc8(const void *p)
{
    uint2 r;
    asm("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

template <>
struct Chunk<2> {
    using raw = uint4;
    static __device__ __forceinline__ raw load(const void *p) { return ld_stream(p); }
    static __device__ __forceinline__ raw load_l1(const void *p) { return ld_nc(p); }
    static __device__ __forceinline__ void to_f32(const raw &v, float f[8]) { bf16x8_to_f32(v, f); }
    // acc[i] += element i (fp32)
    static __device__ __forceinline__ void add_to(const raw &v, float acc[8])
    {
        float f[8];
        bf16x8_to_f32(v, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += f[i];
    }
    // d[i] = element i - c[i] (fp32)
    static __device__ __forceinline__ void sub_from(const raw &v, const float c[8], float d[8])
    {
        float f[8];
        bf16x8_to_f32(v, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) d[i] = f[i] - c[i];
    }
};

template <>
struct Chunk<1> {
    using raw = uint2;
    static __device__ __forceinline__ raw load(const void *p) { return ld_stream8(p); }
    static __device__ __forceinline__ raw load_l1(const void *p) { return ld_nc8(p); }
    static __device__ __forceinline__ void to_f32(const raw &v, float f[8]) { e4m3x8_to_f32(v, f); }
    // The same results as to_f32 followed by fp32 adds / subtractions, with
    // the fp16 -> fp32 widening folded into mixed-precision instructions.
    static __device__ __forceinline__ void add_to(const raw &v, float acc[8])
    {
        const uint32_t w[2] = {v.x, v.y};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            add_f16x2(e4m3x2_to_f16x2(w[i] & 0xFFFFu), acc[4 * i + 0], acc[4 * i + 1]);
            add_f16x2(e4m3x2_to_f16x2(w[i] >> 16), acc[4 * i + 2], acc[4 * i + 3]);
        }
    }
    static __device__ __forceinline__ void sub_from(const raw &v, const float c[8], float d[8])
    {
        const uint32_t w[2] = {v.x, v.y};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            sub_f16x2(e4m3x2_to_f16x2(w[i] & 0xFFFFu), c[4 * i + 0], c[4 * i + 1], d[4 * i + 0], d[4 * i + 1]);
            sub_f16x2(e4m3x2_to_f16x2(w[i] >> 16), c[4 * i + 2], c[4 * i + 3], d[4 * i + 2], d[4 * i + 3]);
        }
    }
};

// Sum over the 16 lanes of a half-warp (all 32 lanes must call it).
__device__ __forceinline__ float half_warp_sum(float v)
{
    v += __shfl_xor_sync(kFull, v, 8);
    v += __shfl_xor_sync(kFull, v, 4);
    v += __shfl_xor_sync(kFull, v, 2);
    v += __shfl_xor_sync(kFull, v, 1);
    return v;
}

// Order-preserving map of fp32 bits to uint32 (larger score -> larger key).
__device__ __forceinline__ uint32_t score_key(float s)
{
    const uint32_t b = __float_as_uint(s);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Tokens of head `head`; a length outside [0, t_max] is reported and the
// head treated as empty.
__device__ __forceinline__ int head_len(const int32_t *seq_lens, int64_t head, int heads, int t_max,
                                        uint32_t *status, bool report)
{
    if (!seq_lens) return t_max;
    const int T = seq_lens[head / heads];
    if (T < 0 || T > t_max) {
        if (report) atomicOr(status, MKV_DEV_BAD_SEQ_LEN);
        return 0;
    }
    return T;
}

__device__ __forceinline__ int window_len(int T, int window)
{
    return (window <= 0 || window >= T) ? T : window;
}

// floor(T*(1-ratio) + 0.5) clamped to [0, T], each operation rounded once
// (no contraction into an FMA), matching the host helper bit for bit.
__device__ __forceinline__ int num_keep_dev(int T, double ratio)
{
    if (T <= 0) return 0;
    const double x = floor(__dadd_rn(__dmul_rn((double)T, __dsub_rn(1.0, ratio)), 0.5));
    if (x < 0.0) return 0;
    if (x > (double)T) return T;
    return (int)x;
}

// Exclusive prefix sum over the CTA in thread order; *total gets the sum.
// Every thread of the CTA must call it; `scratch` holds one word per warp.
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *scratch, uint32_t *total)
{
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < NW ? scratch[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NW) scratch[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    const uint32_t before_warp = warp ? scratch[warp - 1] : 0u;
    if (total) *total = scratch[NW - 1];
    __syncthreads();  // scratch may be reused right after
    return before_warp + x - v;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel on the stream drains;
// it must wait here before it reads that kernel's outputs (a no-op for an
// ordinary launch). The previous kernel allows the early launch with
// pdl_trigger(); persistent kernels call it when a CTA starts its last item,
// since dependent CTAs that wait through many rounds slow those rounds down.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Nanoseconds since an arbitrary origin (the GPU's global timer); bounds
// every wait in the kernels.
__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace dev
}  // namespace mkv
