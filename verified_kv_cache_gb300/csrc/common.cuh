// Device helpers shared by the compress and decode kernels of libverkv.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace verkv {

constexpr int kHeadDim = 128;
constexpr float kTauFloor = 0x1p-38f;  // smallest importance score; tau * 2^61 is then an integer

// ---------------------------------------------------------------------------------------------
// Element access for the two K/V storage types.
// ---------------------------------------------------------------------------------------------
template <typename T> struct Elt;
template <> struct Elt<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }
};
template <> struct Elt<float> {
    static __device__ __forceinline__ float load(const float* p, int64_t i) { return p[i]; }
};

// ---------------------------------------------------------------------------------------------
// Float-float ("double-fp32") arithmetic: a value is hi + lo with |lo| <= ulp(hi)/2.  Used
// wherever a decision (an order, a threshold) needs more than fp32 precision: the sketch and exact
// logits, the certificate sums and the k* scan.  Error-free transformations (Knuth's two-sum,
// Dekker's fast-two-sum, the FMA two-product); the __f*_rn intrinsics keep the compiler from
// contracting or reassociating them.
// ---------------------------------------------------------------------------------------------
struct ff {
    float hi, lo;
};

__device__ __forceinline__ ff two_sum(float a, float b)
{
    float s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, err};
}

__device__ __forceinline__ ff fast_two_sum(float a, float b)
{
    float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ ff two_prod(float a, float b)
{
    float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ ff ff_add(ff x, ff y)
{
    ff s = two_sum(x.hi, y.hi);
    float lo = __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo));
    return fast_two_sum(s.hi, lo);
}

__device__ __forceinline__ ff ff_add_f(ff x, float y)
{
    ff s = two_sum(x.hi, y);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, x.lo));
}

__device__ __forceinline__ ff ff_mul_f(ff x, float y)
{
    ff p = two_prod(x.hi, y);
    return fast_two_sum(p.hi, __fmaf_rn(x.lo, y, p.lo));
}

__device__ __forceinline__ ff ff_mul(ff x, ff y)
{
    ff p = two_prod(x.hi, y.hi);
    float lo = __fmaf_rn(x.hi, y.lo, __fmaf_rn(x.lo, y.hi, p.lo));
    return fast_two_sum(p.hi, lo);
}

__device__ __forceinline__ ff ff_neg(ff x) { return {-x.hi, -x.lo}; }

__device__ __forceinline__ ff ff_sub(ff x, ff y) { return ff_add(x, ff_neg(y)); }

// x / y: the fp32 quotient corrected by one step on the float-float remainder (~2^-46 relative).
__device__ __forceinline__ ff ff_div(ff x, ff y)
{
    if (x.hi == 0.f) return {0.f, 0.f};   // also keeps zero numerators off the division's slow path
    const float q1 = __fdiv_rn(x.hi, y.hi);
    const ff r = ff_sub(x, ff_mul_f(y, q1));
    return fast_two_sum(q1, __fdiv_rn(r.hi, y.hi));
}

// sqrt(x) for x >= 0: the fp32 root corrected by one Newton step on the float-float residual.
__device__ __forceinline__ ff ff_sqrt(ff x)
{
    if (!(x.hi > 0.f)) return {0.f, 0.f};
    const float s = __fsqrt_rn(x.hi);
    const ff e = ff_sub(x, two_prod(s, s));
    return fast_two_sum(s, __fdiv_rn(e.hi, __fmul_rn(2.0f, s)));
}

// Comparisons of normalised float-float values (|lo| <= ulp(hi)/2).
__device__ __forceinline__ bool ff_lt(ff x, ff y) { return x.hi < y.hi || (x.hi == y.hi && x.lo < y.lo); }
__device__ __forceinline__ bool ff_eq(ff x, ff y) { return x.hi == y.hi && x.lo == y.lo; }
__device__ __forceinline__ ff ff_min(ff x, ff y) { return ff_lt(y, x) ? y : x; }
__device__ __forceinline__ ff ff_max(ff x, ff y) { return ff_lt(x, y) ? y : x; }

// The binary64 value of a binary32 one, assembled from its bit fields (sign, exponent rebiased from
// 127 to 1023, fraction widened by 29 bits; subnormals normalised): exact, and free of the
// conversion instructions, which are slow on parts with few FP64 units.
__device__ __forceinline__ double f32_to_f64_bits(float x)
{
    const unsigned u = __float_as_uint(x);
    const unsigned long long sign = (unsigned long long)(u >> 31) << 63;
    const unsigned e = (u >> 23) & 0xffu;
    unsigned long long frac = u & 0x7fffffu;
    unsigned long long bits;
    if (e == 0xffu) {
        bits = sign | (0x7ffull << 52) | (frac << 29);
    } else if (e != 0u) {
        bits = sign | ((unsigned long long)(e + 896u) << 52) | (frac << 29);
    } else if (frac == 0ull) {
        bits = sign;
    } else {
        // value = frac * 2^-149 with the top set bit at position p (0..22)
        const int p = 31 - __clz((unsigned)frac);
        bits = sign | ((unsigned long long)(p + 874) << 52) | ((frac << (52 - p)) & ((1ull << 52) - 1ull));
    }
    return __longlong_as_double((long long)bits);
}

__device__ __forceinline__ double ff_to_f64(ff x) { return f32_to_f64_bits(x.hi) + f32_to_f64_bits(x.lo); }

__device__ __forceinline__ double ff_to_double(ff x) { return (double)x.hi + (double)x.lo; }

__device__ __forceinline__ ff ff_from_double(double v)
{
    float hi = __double2float_rn(v);
    float lo = __double2float_rn(v - (double)hi);
    return {hi, lo};
}

// exp(x.hi + x.lo) with ~2 ulp relative error: expf(hi) * (1 + lo).
__device__ __forceinline__ float ff_exp(ff x)
{
    float e = expf(x.hi);
    return __fmaf_rn(e, x.lo, e);
}

__device__ __forceinline__ ff shfl_xor_ff(ff v, int mask)
{
    return {__shfl_xor_sync(0xffffffffu, v.hi, mask), __shfl_xor_sync(0xffffffffu, v.lo, mask)};
}

__device__ __forceinline__ ff warp_sum_ff(ff v)
{
    for (int o = 16; o > 0; o >>= 1) v = ff_add(v, shfl_xor_ff(v, o));
    return v;
}

// Block-wide float-float sum; every thread gets the total.  `scratch` holds >= 32 ff.
__device__ __forceinline__ ff block_sum_ff(ff v, ff* scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v = warp_sum_ff(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    ff t = lane < nw ? scratch[lane] : ff{0.f, 0.f};
    t = warp_sum_ff(t);
    return t;
}

__device__ __forceinline__ float warp_max(float v)
{
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float block_max(float v, float* scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v = warp_max(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float t = lane < nw ? scratch[lane] : -INFINITY;
    return warp_max(t);
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v)
{
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T>
__device__ __forceinline__ T block_sum(T v, T* scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    T t = lane < nw ? scratch[lane] : T(0);
    return warp_sum(t);
}

// Exclusive block scan of ints (block size a multiple of 32, <= 1024).  Returns the exclusive
// prefix of this thread; *total gets the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = lane < nw ? scratch[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < nw) scratch[lane] = s;
    }
    __syncthreads();
    int before = warp > 0 ? scratch[warp - 1] : 0;
    *total = scratch[nw - 1];
    return before + x - v;
}

// Order-preserving map float -> int for atomicMax on floats.
__device__ __forceinline__ int float_to_ordered(float f)
{
    int i = __float_as_int(f);
    return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float ordered_to_float(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff); }

// A running maximum tagged with a generation: values of an older generation compare smaller, so the
// slot needs no reset between calls.  atomicMax on the 64-bit word keeps the largest float of the
// newest generation.
__device__ __forceinline__ unsigned long long tag_max(unsigned gen, float f)
{
    return ((unsigned long long)gen << 32) | (unsigned)(float_to_ordered(f) ^ 0x80000000);
}
__device__ __forceinline__ float untag_max(unsigned long long t, unsigned gen)
{
    if ((unsigned)(t >> 32) != gen) return -INFINITY;
    return ordered_to_float((int)((unsigned)t ^ 0x80000000u));
}

// ---------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC'11): ten rounds of two 32x32 -> 64-bit products, key bumped by
// the Weyl constants between rounds.  The Poisson draw of a token uses word 0 of the block at
// counter (token, kv_head, layer, seq); u = (x >> 8) * 2^-24 is exact in fp32.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 ctr, uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        const uint32_t lo0 = 0xD2511F53u * ctr.x, hi0 = __umulhi(0xD2511F53u, ctr.x);
        const uint32_t lo1 = 0xCD9E8D57u * ctr.z, hi1 = __umulhi(0xCD9E8D57u, ctr.z);
        ctr = make_uint4(hi1 ^ ctr.y ^ k0, lo1, hi0 ^ ctr.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return ctr;
}

__device__ __forceinline__ float poisson_uniform(uint64_t seed, uint32_t token, uint32_t kv_head, uint32_t layer,
                                                 uint32_t seq)
{
    uint4 x = philox4x32_10(make_uint4(token, kv_head, layer, seq), (uint32_t)seed, (uint32_t)(seed >> 32));
    return (float)(x.x >> 8) * 0x1p-24f;
}

// Correctly rounded (to nearest even) conversion of an unsigned 128-bit integer to double.
__device__ __forceinline__ double u128_to_double_rn(uint64_t hi, uint64_t lo)
{
    if (hi == 0) return __ull2double_rn(lo);
    const int bits_hi = 64 - __clzll(hi);             // 1..64
    // top 64 bits of the value, with a sticky bit for everything shifted out
    uint64_t top = (hi << (64 - bits_hi)) | (bits_hi == 64 ? 0 : (lo >> bits_hi));
    const uint64_t rest = bits_hi == 64 ? lo : (lo << (64 - bits_hi));
    if (rest != 0) top |= 1ull;
    return ldexp(__ull2double_rn(top), bits_hi);
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float tau_clamp(float t)
{
    return t > kTauFloor ? (t < 1.0f ? t : 1.0f) : kTauFloor;
}

}  // namespace verkv
