// quantize.cu -- activation quantize kernels (per-row, tensorwise, ConvRot-rotated)
// and the int8 -> bf16 widening of tensor-core operands.  All are HBM-bandwidth bound:
// 16-byte vector loads straight into registers, warp-shuffle reductions.
//
// What they compute (comfy-kitchen issue #278, quantize_int8_rowwise, and issue #280,
// tensor-wide scales):
//   x_scale = max|v| / 127 (fp32),  q = clamp(rint(v / x_scale), -127, 127)
// with v = x, or v = x @ H for ConvRot (issue #278, "Suggested fix").
//
// Division.  rint(v / x_scale) must see the correctly rounded fp32 quotient.  When v
// is a bf16 value (per-row and tensorwise modes) the row maximum is a bf16 value too,
// and the quotient is formed from the correctly rounded reciprocal r = 1/s with one
// FMA correction (Markstein, IBM J. Res. Dev. 34(1), 1990):
//   t = v * r;  e = fma(-t, s, v)  (exact remainder);  t = fma(e, r, t)
// which equals the IEEE quotient; this was checked exhaustively on the CPU for every
// pair of bf16 significands (numerator <= maximum) over the full exponent range that
// can reach rint's decision, with zero mismatches.  ConvRot values are fp32: there the
// product v * r decides the code wherever a rigorous error bound shows it must agree
// with the IEEE quotient, and the IEEE division settles the rest (see Coder).  Scales
// below 2^-100 use the IEEE division throughout.  x_scale itself is fl(amax / 127) by a
// correction sequence checked exhaustively (div127), and the rounding to an integer is an
// fp32 add (kRoundMagic): no step needs the quarter-rate conversion instructions.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <unistd.h>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ck_device.cuh"
#include "ck_internal.h"

namespace ck {
namespace quant {

constexpr int ROWS_PER_BLOCK = 8;  // one warp per row
constexpr int THREADS = 32 * ROWS_PER_BLOCK;
constexpr int UNROLL = 4;          // independent 16-byte loads in flight per thread in grid-stride loops

__device__ __forceinline__ uint4 ld_stream(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// max |x| over the 8 bf16 values of a vector, on packed pairs (exact)
__device__ __forceinline__ __nv_bfloat162 absmax8(__nv_bfloat162 m, const uint4& v)
{
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        m = __hmax2(m, __habs2(p[i]));
    return m;
}

// Rounding without the conversion pipe.  For |t| < 2^22, t + 1.5 * 2^23 lands in
// [2^23, 2^24), where the fp32 spacing is 1, so the add rounds t to an integer (half to
// even) and leaves it in the low mantissa bits: the low byte of the sum's bits is that
// integer's int8 two's-complement byte, and subtracting 1.5 * 2^23 again gives it back as
// an exact float.  A bf16 value of an integer |q| <= 127 (at most 7 significant bits) is
// the upper half of q's fp32 bits, without rounding.  This keeps the quantize off the
// quarter-rate conversion instructions, which at HBM speed would be its bottleneck.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23

// Two fp32 values per instruction (the packed helpers of ck_device.cuh): each lane
// rounds exactly like the scalar instruction and nothing is contracted, so a packed step
// is the same IEEE operation on both values at half the issue cost.  a - b is formed as
// fma(b, -1, a): the product by -1 is exact, so it is a - b rounded once.
__device__ __forceinline__ float2 dup2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return f2_add_rn(a, b); }
__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return f2_fma_rn(b, dup2(-1.0f), a); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return f2_mul_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return f2_fma_rn(a, b, c); }

// x_scale = fl(amax / 127) for amax >= 0 finite, without a division: q1 = fl(amax * c)
// with c = fl(1/127), then one FMA correction of the remainder (Markstein, IBM J. Res.
// Dev. 34(1), 1990).  The result equals the correctly rounded quotient for every
// non-negative finite fp32 amax: checked exhaustively on the CPU (all 2^31 - 2^23 of
// them, against the exact remainder amax - 127 * s), and on the GPU for every bf16 amax.
__device__ __forceinline__ float div127(float amax)
{
    const float c = 0x1.020408p-7f;  // fl(1/127), bits 0x3C010204
    const float q1 = __fmul_rn(amax, c);
    const float e = __fmaf_rn(-q1, 127.0f, amax);
    return __fmaf_rn(e, c, q1);
}

// One code, as the magic sum (t rounded + kRoundMagic), by the scale's rule:
//   kind 1 (bf16 v, scale >= 2^-100): the reciprocal and Markstein correction give the
//     IEEE quotient; with s = fl(amax / 127) normal, |v / s| <= 127 (1 + 2^-23), whose rint
//     is 127, so no clamp is needed;
//   kind 3 (fp32 v of ConvRot, scale >= 2^-100): t = v * fl(1/s) is within 2^-16 of v / s
//     (two roundings of a quotient below 128) and the IEEE quotient within 2^-18 of it,
//     so where t is more than 2^-14 away from a half-integer both round to the same
//     integer; nearer than that (about 1 value in 16000) the IEEE quotient is formed;
//   kind 2 (scales below 2^-100): the IEEE quotient, clamped;  kind 0: code 0.
struct Coder {
    float s, r;
    int kind;
    __device__ __forceinline__ Coder(float s_, bool fp32_values)
    {
        s = s_;
        r = 0.0f;
        if (s_ == 0.0f) {
            kind = 0;
        } else if (s_ >= 0x1p-100f) {
            kind = fp32_values ? 3 : 1;
            r = __frcp_rn(s_);  // correctly rounded 1 / s
        } else {
            kind = 2;
        }
    }
    __device__ __forceinline__ float slow(float v) const
    {
        return __fadd_rn(fminf(fmaxf(rintf(__fdiv_rn(v, s)), -127.0f), 127.0f), kRoundMagic);
    }
    __device__ __forceinline__ float magic1(float v) const
    {
        float t = __fmul_rn(v, r);
        const float e = __fmaf_rn(-t, s, v);
        t = __fmaf_rn(e, r, t);
        return __fadd_rn(t, kRoundMagic);
    }
    __device__ __forceinline__ float magic3(float v) const
    {
        const float t = __fmul_rn(v, r);
        const float m = __fadd_rn(t, kRoundMagic);
        const float d = __fsub_rn(t, __fsub_rn(m, kRoundMagic));
        return fabsf(__fsub_rn(fabsf(d), 0.5f)) <= 0x1p-14f ? slow(v) : m;
    }
    __device__ __forceinline__ float magic(float v) const
    {
        if (kind == 1)
            return magic1(v);
        if (kind == 3)
            return magic3(v);
        if (kind == 2)
            return slow(v);
        return kRoundMagic;
    }
    // kind 1 on two values: magic1's steps, packed
    __device__ __forceinline__ float2 magic1x2(float2 v) const
    {
        float2 t = mul2(v, dup2(r));
        const float2 e = fma2(t, dup2(-s), v);  // t * (-s) is -(t * s) exactly
        t = fma2(e, dup2(r), t);
        return add2(t, dup2(kRoundMagic));
    }
    // kind 3 on two values, without the near-tie test: the magic sum of t = v * r, and
    // d = t - rint(t) (exact: Fast2Sum against kRoundMagic, then Sterbenz).  |d| <= 1/2,
    // and magic3's test |(|d| - 1/2)| <= 2^-14 is |d| >= 1/2 - 2^-14 (the subtraction is
    // exact for |d| >= 1/4); a caller that finds such a d redoes those values by magic3.
    // Should the compiler fuse the product into the magic add (it has fused a packed add
    // with a packed product of single use), the sum rounds v * r exactly instead of t; the
    // two differ only if t lies within half an ulp (<= 2^-18) of a half-integer, and then
    // d is at least 1/2 away from the integer taken, so those values take magic3 as well.
    __device__ __forceinline__ float2 magic3x2(float2 v, float& dmax) const
    {
        const float2 t = mul2(v, dup2(r));
        const float2 m = add2(t, dup2(kRoundMagic));
        const float2 d = sub2(t, add2(m, dup2(-kRoundMagic)));
        dmax = fmaxf(dmax, fmaxf(fabsf(d.x), fabsf(d.y)));
        return m;
    }
};
constexpr float kNearTie = 0.5f - 0x1p-14f;  // magic3's near-tie bound on |t - rint(t)|

// Eight codes from eight magic sums: int8 bytes, or bf16 codes.
template <bool OUT8>
__device__ __forceinline__ void store_magic8(const float (&m)[8], int8_t* q8, __nv_bfloat16* q16, int64_t off)
{
    if (OUT8) {
        uint32_t u[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            u[i] = __float_as_uint(m[i]);
        const uint32_t lo = __byte_perm(__byte_perm(u[0], u[1], 0x0040), __byte_perm(u[2], u[3], 0x0040), 0x5410);
        const uint32_t hi = __byte_perm(__byte_perm(u[4], u[5], 0x0040), __byte_perm(u[6], u[7], 0x0040), 0x5410);
        *reinterpret_cast<uint2*>(q8 + off) = make_uint2(lo, hi);
    } else {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 n = add2(make_float2(m[2 * i], m[2 * i + 1]), dup2(-kRoundMagic));
            w[i] = __byte_perm(__float_as_uint(n.x), __float_as_uint(n.y), 0x7632);
        }
        *reinterpret_cast<uint4*>(q16 + off) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// The codes of one vector (8 values) by the rule of `cd` (branching once per vector:
// the rule is uniform over a row, or over the tensor), stored as int8 codes and/or bf16
// codes at element offset `off`.
template <bool OUT8, bool OUT16>
__device__ __forceinline__ void code_store8(const Coder& cd, const float (&f)[8], int8_t* q8, __nv_bfloat16* q16,
                                            int64_t off)
{
    float m[8];
    bool done = false;
    if (cd.kind == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 mm = cd.magic1x2(make_float2(f[2 * i], f[2 * i + 1]));
            m[2 * i] = mm.x;
            m[2 * i + 1] = mm.y;
        }
        done = true;
    } else if (cd.kind == 3) {
        float dmax = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 mm = cd.magic3x2(make_float2(f[2 * i], f[2 * i + 1]), dmax);
            m[2 * i] = mm.x;
            m[2 * i + 1] = mm.y;
        }
        done = dmax < kNearTie;
    }
    if (!done) {
        for (int e = 0; e < 8; ++e)
            m[e] = cd.magic(f[e]);
    }
    if (OUT8)
        store_magic8<true>(m, q8, nullptr, off);
    if (OUT16)
        store_magic8<false>(m, nullptr, q16, off);
}

// bf16 bits -> fp32 (exact), two per 32-bit word, without conversion instructions.
__device__ __forceinline__ void unpack8_bits(const uint4& v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// 8 int8 weight codes (given as the two 32-bit halves of 8 bytes) -> 8 bf16 codes: byte
// b ^ 0x80 is b + 128 as an unsigned byte; placed in the low mantissa of 2^23 and reduced
// by 2^23 + 128 it is b as an exact float, whose upper half is its bf16.
__device__ __forceinline__ uint4 widen8_bits(uint32_t lo, uint32_t hi)
{
    const uint32_t w[2] = {lo ^ 0x80808080u, hi ^ 0x80808080u};
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const uint32_t word = w[h >> 1];
        const float a = __fsub_rn(__uint_as_float(0x4B000000u | ((word >> (16 * (h & 1))) & 0xFFu)), 8388736.0f);
        const float b = __fsub_rn(__uint_as_float(0x4B000000u | ((word >> (16 * (h & 1) + 8)) & 0xFFu)), 8388736.0f);
        o[h] = __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x7632);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// ConvRot block transform of the 8 values a lane holds for one vector slot.  A
// 128-block spans 16 lanes: element i = 8*(lane % 16) + e.  Spans 1, 2, 4 pair values
// inside the thread, spans 8..64 pair lanes lane ^ 1..8.  (lo, hi) -> (lo + hi, lo - hi),
// in ascending span order, then a multiply by fp32(1/sqrt(128)).
__device__ __forceinline__ void fwht_slot(float (&v)[8], int lane)
{
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if ((e & h) == 0) {
                const float lo = v[e], hi = v[e + h];
                v[e] = __fadd_rn(lo, hi);
                v[e + h] = __fsub_rn(lo, hi);
            }
        }
    }
    // across lanes: the lower lane of a pair keeps v + p, the upper one p - v; both are
    // one correctly rounded fma(+-1, v, p) (the product by +-1 is exact)
#pragma unroll
    for (int hl = 1; hl < 16; hl <<= 1) {
        const float sgn = (lane & hl) ? -1.0f : 1.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float p = __shfl_xor_sync(0xffffffffu, v[e], hl);
            v[e] = __fmaf_rn(sgn, v[e], p);
        }
    }
    const float c128 = 0.088388346f;  // fp32(1/sqrt(128)) = 0x3DB504F3
#pragma unroll
    for (int e = 0; e < 8; ++e)
        v[e] = __fmul_rn(v[e], c128);
}

// The same transform on two vector slots of a lane at once: element e of slot a in
// v[e].x, of slot b in v[e].y.  Every butterfly is the scalar one, two values per packed
// instruction (a - b as fma(b, -1, a), exact product), in the same span order.
__device__ __forceinline__ void fwht_pair(float2 (&v)[8], int lane)
{
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if ((e & h) == 0) {
                const float2 lo = v[e], hi = v[e + h];
                v[e] = add2(lo, hi);
                v[e + h] = sub2(lo, hi);
            }
        }
    }
#pragma unroll
    for (int hl = 1; hl < 16; hl <<= 1) {
        const float2 sgn = dup2((lane & hl) ? -1.0f : 1.0f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float2 p = make_float2(__shfl_xor_sync(0xffffffffu, v[e].x, hl),
                                         __shfl_xor_sync(0xffffffffu, v[e].y, hl));
            v[e] = fma2(sgn, v[e], p);
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e)
        v[e] = mul2(v[e], dup2(0.088388346f));  // fp32(1/sqrt(128)), as in fwht_slot
}

// The codes of two slots (element e of slot a in v[e].x, of slot b in v[e].y) by the rule
// of `cd`, stored at element offsets off_a / off_b where st_a / st_b hold.  The scale's
// rule is the same for both (one row).
template <bool OUT8, bool OUT16>
__device__ __forceinline__ void code_store_pair(const Coder& cd, const float2 (&v)[8], int8_t* q8,
                                                __nv_bfloat16* q16, int64_t off_a, bool st_a, int64_t off_b,
                                                bool st_b)
{
    float2 m[8];
    bool done = false;
    if (cd.kind == 3) {
        float dmax = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e)
            m[e] = cd.magic3x2(v[e], dmax);
        done = dmax < kNearTie;
    } else if (cd.kind == 1) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            m[e] = cd.magic1x2(v[e]);
        done = true;
    }
    if (!done) {
        for (int e = 0; e < 8; ++e)
            m[e] = make_float2(cd.magic(v[e].x), cd.magic(v[e].y));
    }
    if (OUT8) {
        float ma[8], mb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            ma[e] = m[e].x;
            mb[e] = m[e].y;
        }
        if (st_a)
            store_magic8<true>(ma, q8, nullptr, off_a);
        if (st_b)
            store_magic8<true>(mb, q8, nullptr, off_b);
    }
    if (OUT16) {
        uint32_t wa[4], wb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 n0 = add2(m[2 * i], dup2(-kRoundMagic));
            const float2 n1 = add2(m[2 * i + 1], dup2(-kRoundMagic));
            wa[i] = __byte_perm(__float_as_uint(n0.x), __float_as_uint(n1.x), 0x7632);
            wb[i] = __byte_perm(__float_as_uint(n0.y), __float_as_uint(n1.y), 0x7632);
        }
        if (st_a)
            *reinterpret_cast<uint4*>(q16 + off_a) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
        if (st_b)
            *reinterpret_cast<uint4*>(q16 + off_b) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
    }
}

// int8 -> bf16 (exact), 16 values per thread and vector.
__device__ __forceinline__ void widen16(const uint4& v, uint4& lo, uint4& hi)
{
    lo = widen8_bits(v.x, v.y);
    hi = widen8_bits(v.z, v.w);
}

// This block's share of an int8 -> bf16 widening, called by every thread of the block.
// A warp takes 32 consecutive 16-byte input vectors at a time; the lanes exchange their
// converted halves (shuffles) so that each of the warp's two stores covers 512
// contiguous bytes of the output (per-lane 32-byte outputs at a 32-byte stride left
// every store half a line and ran ~30% slower).
__device__ __forceinline__ void widen_share(const uint4* __restrict__ src, int64_t n16, uint4* __restrict__ dst)
{
    if (src == nullptr)
        return;
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    for (int64_t base = wid * 32 * UNROLL; base < n16; base += warps * 32 * UNROLL) {  // warp-uniform
        uint4 v[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t i = base + u * 32 + lane;
            v[u] = i < n16 ? ld_stream(src + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            uint4 lo, hi;
            widen16(v[u], lo, hi);
            // output vector 2j is lo of input j, 2j + 1 its hi: lane l writes output l
            // (from lane l / 2) and output 32 + l (from lane 16 + l / 2)
            const int64_t i0 = base + u * 32;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const int srcl = 16 * part + (lane >> 1);
                uint4 a, b;
                a.x = __shfl_sync(0xffffffffu, lo.x, srcl);
                a.y = __shfl_sync(0xffffffffu, lo.y, srcl);
                a.z = __shfl_sync(0xffffffffu, lo.z, srcl);
                a.w = __shfl_sync(0xffffffffu, lo.w, srcl);
                b.x = __shfl_sync(0xffffffffu, hi.x, srcl);
                b.y = __shfl_sync(0xffffffffu, hi.y, srcl);
                b.z = __shfl_sync(0xffffffffu, hi.z, srcl);
                b.w = __shfl_sync(0xffffffffu, hi.w, srcl);
                if (i0 + srcl < n16)
                    dst[2 * i0 + 32 * part + lane] = (lane & 1) ? b : a;
            }
        }
    }
}

// Per-row quantize with the row held in registers: TPR threads per row (one to eight
// warps), VPT 16-byte vectors per thread, K <= 8 * TPR * VPT.  Vector j of thread t is
// row vector t + TPR*j, so a warp's 32 lanes hold 32 consecutive vectors (two ConvRot
// blocks) in every slot.  The row maximum is reduced by shuffles, then across the
// row's warps through shared memory.
// With w8 != null the launch also widens the weight (each block takes a share after
// its rows), so the layer's two bandwidth-bound passes share one launch.
template <int TPR, int VPT, bool ROT, bool OUT8, bool OUT16>
__global__ void __launch_bounds__(THREADS) rows_kernel(const uint4* __restrict__ x, int64_t M, int64_t K,
                                                       int8_t* __restrict__ q8, __nv_bfloat16* __restrict__ q16,
                                                       float* __restrict__ xs, const uint4* __restrict__ w8,
                                                       int64_t w_n16, uint4* __restrict__ w16)
{
    griddep_wait();
    griddep_launch_dependents();
    constexpr int RPB = THREADS / TPR;  // rows per block
    constexpr int WPR = TPR / 32;       // warps per row
    __shared__ float red[THREADS / 32];
    const int lane = threadIdx.x & 31;
    const int t = threadIdx.x % TPR;
    const int g = threadIdx.x / TPR;
    const int64_t row = (int64_t)blockIdx.x * RPB + g;
    const bool live = row < M;
    const int64_t nvec = K >> 3;
    const uint4* xr = x + (live ? row : 0) * nvec;
    const int64_t warp_first = t - lane;  // first vector of this warp in slot 0

    // ConvRot: slots 2i and 2i + 1 are transformed together (packed pairs); an odd
    // VPT leaves the last slot to the scalar transform
    constexpr int NP = ROT ? VPT / 2 : 0;
    constexpr int NS = ROT ? VPT % 2 : 0;
    float2 vp[NP > 0 ? NP : 1][8];
    float vs[8];
    uint4 raw[VPT];
    float amax = 0.0f;
    __nv_bfloat162 m2 = __float2bfloat162_rn(0.0f);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t idx = t + (int64_t)TPR * j;
        raw[j] = (live && idx < nvec) ? ld_stream(xr + idx) : make_uint4(0, 0, 0, 0);
        if (!ROT)
            m2 = absmax8(m2, raw[j]);
    }
    if (ROT) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            // slot 2i + 1 of the warp may lie past the row while slot 2i does not: its
            // values are zeros then, which leave the maximum alone
            if (warp_first + (int64_t)TPR * (2 * i) < nvec) {  // warp-uniform
                float fa[8], fb[8];
                unpack8_bits(raw[2 * i], fa);
                unpack8_bits(raw[2 * i + 1], fb);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    vp[i][e] = make_float2(fa[e], fb[e]);
                fwht_pair(vp[i], lane);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    amax = fmaxf(amax, fmaxf(fabsf(vp[i][e].x), fabsf(vp[i][e].y)));
            }
        }
        if (NS) {
            unpack8_bits(raw[VPT - 1], vs);
            if (warp_first + (int64_t)TPR * (VPT - 1) < nvec) {  // warp-uniform
                fwht_slot(vs, lane);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    amax = fmaxf(amax, fabsf(vs[e]));
            }
        }
    } else {
        amax = fmaxf(__low2float(m2), __high2float(m2));
    }
    amax = warp_max(amax);
    if (WPR > 1) {
        if (lane == 0)
            red[threadIdx.x >> 5] = amax;
        __syncthreads();
#pragma unroll
        for (int i = 0; i < WPR; ++i)
            amax = fmaxf(amax, red[g * WPR + i]);
    }
    if (live) {
        const float s = div127(amax);
        if (t == 0)
            xs[row] = s;
        const Coder cd(s, ROT);
        if (ROT) {
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                const int64_t ia = t + (int64_t)TPR * (2 * i), ib = ia + TPR;
                if (ia < nvec)
                    code_store_pair<OUT8, OUT16>(cd, vp[i], q8, q16, row * K + ia * 8, true, row * K + ib * 8,
                                                 ib < nvec);
            }
            if (NS) {
                const int64_t idx = t + (int64_t)TPR * (VPT - 1);
                if (idx < nvec)
                    code_store8<OUT8, OUT16>(cd, vs, q8, q16, row * K + idx * 8);
            }
        } else {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int64_t idx = t + (int64_t)TPR * j;
                if (idx < nvec) {
                    float f[8];
                    unpack8_bits(raw[j], f);
                    code_store8<OUT8, OUT16>(cd, f, q8, q16, row * K + idx * 8);
                }
            }
        }
    }
    widen_share(w8, w_n16, w16);
}

// One row of rows_stream_kernel (one warp): pass 1 finds the maximum, pass 2 re-reads
// (from L2) and quantizes.
template <bool ROT, bool OUT8, bool OUT16>
__device__ __forceinline__ void stream_row(const uint4* __restrict__ x, int64_t row, int64_t K, int lane,
                                           int8_t* __restrict__ q8, __nv_bfloat16* __restrict__ q16,
                                           float* __restrict__ xs)
{
    const int64_t nvec = K >> 3;
    const uint4* xr = x + row * nvec;
    float amax = 0.0f;
    for (int64_t base = 0; base < nvec; base += 32) {
        const int64_t idx = base + lane;
        const uint4 r = (idx < nvec) ? xr[idx] : make_uint4(0, 0, 0, 0);
        float f[8];
        unpack8_bits(r, f);
        if (ROT)
            fwht_slot(f, lane);
        if (idx < nvec) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                amax = fmaxf(amax, fabsf(f[e]));
        }
    }
    amax = warp_max(amax);
    const float s = div127(amax);
    if (lane == 0)
        xs[row] = s;
    const Coder cd(s, ROT);
    for (int64_t base = 0; base < nvec; base += 32) {
        const int64_t idx = base + lane;
        const uint4 r = (idx < nvec) ? ld_stream(xr + idx) : make_uint4(0, 0, 0, 0);
        float f[8];
        unpack8_bits(r, f);
        if (ROT)
            fwht_slot(f, lane);
        if (idx < nvec)
            code_store8<OUT8, OUT16>(cd, f, q8, q16, row * K + idx * 8);
    }
}

// Per-row quantize for rows too long to keep in registers, one warp per row.
template <bool ROT, bool OUT8, bool OUT16>
__global__ void __launch_bounds__(THREADS) rows_stream_kernel(const uint4* __restrict__ x, int64_t M, int64_t K,
                                                              int8_t* __restrict__ q8, __nv_bfloat16* __restrict__ q16,
                                                              float* __restrict__ xs, const uint4* __restrict__ w8,
                                                              int64_t w_n16, uint4* __restrict__ w16)
{
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * ROWS_PER_BLOCK + (threadIdx.x >> 5);
    if (row < M)
        stream_row<ROT, OUT8, OUT16>(x, row, K, lane, q8, q16, xs);
    widen_share(w8, w_n16, w16);
}

// ConvRot weight preparation (issue #278, "Suggested fix": the stored weight is
// W_rot = W @ H^T, quantized per output row).  H is symmetric, so row n of W @ H^T is row
// n of W times H: the block transform of the activations, applied to fp32 rows.  Then
// w_scale[n] = max|W_rot[n]| / 127 and w = clamp(rint(W_rot / w_scale), -127, 127), with
// the IEEE division (fp32 input).  A vector slot here is 8 fp32 values (two 16-byte loads).
__device__ __forceinline__ void load8_f32(const float4* __restrict__ p, int64_t idx, bool valid, float (&f)[8])
{
    if (valid) {
        const float4 a = __ldg(p + 2 * idx), b = __ldg(p + 2 * idx + 1);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            f[i] = 0.0f;
    }
}

template <int TPR, int VPT>
__global__ void __launch_bounds__(THREADS) weight_rot_kernel(const float4* __restrict__ W, int64_t N, int64_t K,
                                                             int8_t* __restrict__ w, float* __restrict__ ws)
{
    griddep_wait();
    griddep_launch_dependents();
    constexpr int RPB = THREADS / TPR;
    constexpr int WPR = TPR / 32;
    __shared__ float red[THREADS / 32];
    const int lane = threadIdx.x & 31;
    const int t = threadIdx.x % TPR;
    const int g = threadIdx.x / TPR;
    const int64_t row = (int64_t)blockIdx.x * RPB + g;
    const bool live = row < N;
    const int64_t nvec = K >> 3;
    const float4* wr = W + (live ? row : 0) * (nvec * 2);
    const int64_t warp_first = t - lane;
    float v[VPT][8];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t idx = t + (int64_t)TPR * j;
        load8_f32(wr, idx, live && idx < nvec, v[j]);
        if (warp_first + (int64_t)TPR * j < nvec) {  // warp-uniform
            fwht_slot(v[j], lane);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                amax = fmaxf(amax, fabsf(v[j][e]));
        }
    }
    amax = warp_max(amax);
    if (WPR > 1) {
        if (lane == 0)
            red[threadIdx.x >> 5] = amax;
        __syncthreads();
#pragma unroll
        for (int i = 0; i < WPR; ++i)
            amax = fmaxf(amax, red[g * WPR + i]);
    }
    if (!live)
        return;
    const float s = div127(amax);
    if (t == 0)
        ws[row] = s;
    const Coder cd(s, true);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int64_t idx = t + (int64_t)TPR * j;
        if (idx < nvec)
            code_store8<true, false>(cd, v[j], w, nullptr, row * K + idx * 8);
    }
}

// The same for rows longer than 16384 values: one warp per row, two passes.
__global__ void __launch_bounds__(THREADS) weight_rot_stream_kernel(const float4* __restrict__ W, int64_t N,
                                                                    int64_t K, int8_t* __restrict__ w,
                                                                    float* __restrict__ ws)
{
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * ROWS_PER_BLOCK + (threadIdx.x >> 5);
    if (row >= N)
        return;  // the whole warp leaves together
    const int64_t nvec = K >> 3;
    const float4* wr = W + row * (nvec * 2);
    float amax = 0.0f;
    for (int64_t base = 0; base < nvec; base += 32) {
        const int64_t idx = base + lane;
        float f[8];
        load8_f32(wr, idx, idx < nvec, f);
        fwht_slot(f, lane);
        if (idx < nvec) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                amax = fmaxf(amax, fabsf(f[e]));
        }
    }
    amax = warp_max(amax);
    const float s = div127(amax);
    if (lane == 0)
        ws[row] = s;
    const Coder cd(s, true);
    for (int64_t base = 0; base < nvec; base += 32) {
        const int64_t idx = base + lane;
        float f[8];
        load8_f32(wr, idx, idx < nvec, f);
        fwht_slot(f, lane);
        if (idx < nvec)
            code_store8<true, false>(cd, f, w, nullptr, row * K + idx * 8);
    }
}

// Tensorwise pass 1: per-block maximum of |x| over a grid-stride slice.
__global__ void __launch_bounds__(256) amax_partials_kernel(const uint4* __restrict__ x, int64_t nvec,
                                                            float* __restrict__ partials,
                                                            const uint4* __restrict__ w8 = nullptr,
                                                            int64_t w_n16 = 0, uint4* __restrict__ w16 = nullptr)
{
    griddep_wait();
    griddep_launch_dependents();
    __shared__ float red[8];
    __nv_bfloat162 m2 = __float2bfloat162_rn(0.0f);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; base < nvec; base += UNROLL * stride) {
        uint4 v[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t i = base + u * stride;
            v[u] = i < nvec ? ld_stream(x + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
            m2 = absmax8(m2, v[u]);
    }
    float m = warp_max(fmaxf(__low2float(m2), __high2float(m2)));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
        m = warp_max(m);
        if (threadIdx.x == 0)
            partials[blockIdx.x] = m;
    }
    widen_share(w8, w_n16, w16);  // a weight widening may share the launch
}

// Tensorwise pass 2: every block reduces the partial maxima (a few KB, L2 resident),
// forms the one scale, and quantizes its grid-stride slice.
template <bool OUT8, bool OUT16>
__global__ void __launch_bounds__(256) quant_flat_kernel(const uint4* __restrict__ x, int64_t nvec,
                                                         const float* __restrict__ partials, int nparts,
                                                         int8_t* __restrict__ q8, __nv_bfloat16* __restrict__ q16,
                                                         float* __restrict__ xs)
{
    griddep_wait();
    griddep_launch_dependents();
    __shared__ float red[8];
    __shared__ float s_amax;
    float m = 0.0f;
    for (int i = threadIdx.x; i < nparts; i += blockDim.x)
        m = fmaxf(m, partials[i]);
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
        m = warp_max(m);
        if (threadIdx.x == 0)
            s_amax = m;
    }
    __syncthreads();
    const float s = div127(s_amax);
    if (blockIdx.x == 0 && threadIdx.x == 0)
        xs[0] = s;
    const Coder cd(s, false);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; base < nvec; base += UNROLL * stride) {
        uint4 v[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t i = base + u * stride;
            v[u] = i < nvec ? ld_stream(x + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t i = base + u * stride;
            if (i < nvec) {
                float f[8];
                unpack8_bits(v[u], f);
                code_store8<OUT8, OUT16>(cd, f, q8, q16, i * 8);
            }
        }
    }
}

// The tensorwise layer's whole preparation in one launch: each block takes the maximum
// of |x| over its grid-stride slice and publishes it, widens its share of the weight
// while the other blocks finish, learns the global maximum, and quantizes its slice
// (re-read from L2) into bf16 codes.
// Hand-off without atomics or resets: block b writes its maximum into slot b of the
// caller's workspace and then, with release semantics, this launch's 64-bit epoch next
// to it; every block then polls all slots (relaxed loads, one acquire fence once every
// slot carries the epoch) and reduces the maxima itself, so the maximum is known one
// round trip after the last block published.  Values left by any earlier launch carry
// another epoch and are never taken.  The grid never exceeds the number of co-resident
// blocks (nor kMaxSlotsPerThread * 256), so every block gets to publish; the waits are
// bounded all the same.
// A block whose wait gives up sets kErrWaitGrid in `err` and makes x_scale NaN, so that
// every output of the layer is NaN instead of plausible: it first tags the `poison` word
// with this launch's epoch, then (after an SC fence) stores NaN into x_scale.  Block 0
// stores the real scale, and at its end (after an SC fence) reads the poison word and
// stores NaN if it carries this epoch.  Of two SC fences one comes first, so either block
// 0 sees the tag or its store precedes the NaN store: x_scale ends NaN either way.
struct alignas(16) EpochSlot {
    unsigned long long epoch;
    float value;
    float pad;
};
constexpr int kMaxSlotsPerThread = 4;  // slots one thread of the block watches

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_gpu()
{
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ void fence_sc_gpu()
{
    asm volatile("fence.sc.gpu;" ::: "memory");
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_f32(float* p, float v)
{
    asm volatile("st.relaxed.gpu.global.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// The first `staged` vectors a thread loads in step 1 are also kept in dynamic shared
// memory (slot j of thread t at [j][t]: conflict-free, only the thread itself reads it
// back), so step 4 reads them from there instead of from L2 / HBM.
constexpr int kMaxStagedVectors = 13;  // 13 vectors per thread: 208 KiB of the SM
constexpr int kPrepThreads = 256;      // threads per block
template <int TPB>
__global__ void __launch_bounds__(TPB) tensorwise_prep_kernel(
    const uint4* __restrict__ x, int64_t nvec, EpochSlot* slots, unsigned long long* poison,
    unsigned long long epoch, __nv_bfloat16* __restrict__ q16, float* xs, const uint4* __restrict__ w8,
    int64_t w_n16, uint4* __restrict__ w16, uint64_t timeout_ns, unsigned int* err, int staged)
{
    extern __shared__ uint4 x_stage[];
    griddep_wait();
    griddep_launch_dependents();
    __shared__ float red[TPB / 32];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int G = (int)gridDim.x;
    // 1. this block's maximum, published
    __nv_bfloat162 m2 = __float2bfloat162_rn(0.0f);
    int slot = 0;  // vectors this thread has loaded so far
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; base < nvec;
         base += UNROLL * stride, slot += UNROLL) {
        uint4 v[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t i = base + u * stride;
            v[u] = i < nvec ? ld_stream(x + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            m2 = absmax8(m2, v[u]);
            if (slot + u < staged)
                x_stage[(slot + u) * TPB + threadIdx.x] = v[u];
        }
    }
    float m = warp_max(fmaxf(__low2float(m2), __high2float(m2)));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float bm = 0.0f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i)
            bm = fmaxf(bm, red[i]);
        slots[blockIdx.x].value = bm;
        st_release_u64(&slots[blockIdx.x].epoch, epoch);
    }
    // 2. the weight widening hides the wait for the slowest block
    widen_share(w8, w_n16, w16);
    // 3. the global maximum: every slot carries this launch's epoch
    uint32_t seen = 0;
#pragma unroll
    for (int j = 0; j < kMaxSlotsPerThread; ++j)
        if ((int)threadIdx.x + TPB * j >= G)
            seen |= 1u << j;
    const uint64_t t0 = globaltimer_ns();
    bool gave_up = false;  // block-uniform
    for (uint32_t round = 1;; ++round) {
#pragma unroll
        for (int j = 0; j < kMaxSlotsPerThread; ++j)
            if (!(seen & (1u << j)) && ld_relaxed_u64(&slots[threadIdx.x + TPB * j].epoch) == epoch)
                seen |= 1u << j;
        int give_up = 0;
        if ((round & 15u) == 0 && threadIdx.x == 0 && globaltimer_ns() - t0 > timeout_ns)
            give_up = 1;
        if (__syncthreads_or(give_up)) {
            if (threadIdx.x == 0)
                atomicOr(err, kErrWaitGrid);
            gave_up = true;
            break;
        }
        if (__syncthreads_and(seen == (1u << kMaxSlotsPerThread) - 1u))
            break;
    }
    fence_acq_rel_gpu();  // with the relaxed epoch loads: acquire of every block's release
    m = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxSlotsPerThread; ++j)
        if ((int)threadIdx.x + TPB * j < G)
            m = fmaxf(m, __ldcg(&slots[threadIdx.x + TPB * j].value));
    m = warp_max(m);
    __syncthreads();  // every warp is done with red[] from step 1
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = m;
    __syncthreads();
    float g = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i)
        g = fmaxf(g, red[i]);
    const float sc = gave_up ? __int_as_float(0x7FFFFFFF) : div127(g);
    if (threadIdx.x == 0) {
        if (gave_up) {
            st_relaxed_u64(poison, epoch);
            fence_sc_gpu();
            st_relaxed_f32(xs, sc);
        } else if (blockIdx.x == 0) {
            st_relaxed_f32(xs, sc);
        }
    }
    // 4. quantize this block's slice
    const Coder cd(sc, false);
    slot = 0;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; base < nvec;
         base += UNROLL * stride, slot += UNROLL) {
        uint4 v[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t i = base + u * stride;
            if (slot + u < staged)
                v[u] = x_stage[(slot + u) * TPB + threadIdx.x];
            else
                v[u] = i < nvec ? ld_stream(x + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t i = base + u * stride;
            if (i < nvec) {
                float f[8];
                unpack8_bits(v[u], f);
                code_store8<false, true>(cd, f, nullptr, q16, i * 8);
            }
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && !gave_up) {
        fence_sc_gpu();
        if (ld_relaxed_u64(poison) == epoch)
            st_relaxed_f32(xs, __int_as_float(0x7FFFFFFF));
    }
}

// The 16-bit-activation ConvRot operand: x @ H (the same fp32 block transform as the
// quantizing path), rounded once to bf16.  The 128-blocks of the flattened x are
// independent (K % 128 == 0, so no block spans two rows): a warp takes 32 consecutive
// 16-byte vectors, two blocks, at a time.  The launch also widens the weight.
__global__ void __launch_bounds__(256) rotate_bf16_kernel(const uint4* __restrict__ x, int64_t nvec,
                                                          uint4* __restrict__ out, const uint4* __restrict__ w8,
                                                          int64_t w_n16, uint4* __restrict__ w16)
{
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t base = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 32; base < nvec;
         base += warps * 32) {
        const int64_t i = base + lane;
        // a warp's 32 vectors are two whole blocks or, at the very end, the last block
        // (lanes 16-31 then idle: their shuffle partners stay within lanes 16-31)
        const uint4 raw = i < nvec ? ld_stream(x + i) : make_uint4(0, 0, 0, 0);
        float v[8];
        unpack8_bits(raw, v);
        fwht_slot(v, lane);
        if (i < nvec) {
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                o[e] = *reinterpret_cast<uint32_t*>(&b);
            }
            out[i] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    widen_share(w8, w_n16, w16);
}

// Two int8 -> bf16 widenings in one launch (operands of the pre-quantized GEMM entries).
__global__ void __launch_bounds__(256) widen2_kernel(const uint4* __restrict__ a8, int64_t a_n16,
                                                     uint4* __restrict__ a16, const uint4* __restrict__ b8,
                                                     int64_t b_n16, uint4* __restrict__ b16)
{
    griddep_wait();
    griddep_launch_dependents();
    widen_share(a8, a_n16, a16);
    widen_share(b8, b_n16, b16);
}

__global__ void __launch_bounds__(256) widen_kernel(const uint4* __restrict__ src, int64_t n16,
                                                    uint4* __restrict__ dst)
{
    griddep_wait();
    griddep_launch_dependents();
    widen_share(src, n16, dst);
}

}  // namespace quant

namespace {

template <bool OUT8, bool OUT16>
cudaError_t rows_dispatch(const void* x, int64_t M, int64_t K, bool rotate, int8_t* q8, void* q16, float* xs,
                          const int8_t* w8_, int64_t w_n, void* w16_, cudaStream_t s)
{
    using namespace quant;
    const uint4* xv = static_cast<const uint4*>(x);
    const uint4* w8 = reinterpret_cast<const uint4*>(w8_);
    uint4* w16 = static_cast<uint4*>(w16_);
    const int64_t w_n16 = w8 ? (w_n >> 4) : 0;
    __nv_bfloat16* q16b = static_cast<__nv_bfloat16*>(q16);
    const int64_t nvec = K / 8;
    // threads per row (32..256) and vectors per thread (at most 8: rows up to K = 16384
    // stay in registers), chosen so that few of the tpr * vpt vector slots stay empty:
    // idle slots cost bandwidth (K = 5376, 672 vectors, in 256 x 4 slots ran at 81% of
    // HBM, in 128 x 6 at 98%).  The stand-alone quantize of plain rows takes as many
    // vectors per thread as fill (the loads a thread has in flight are what keeps HBM
    // busy: K = 4096 as 64 x 8 instead of 128 x 4 went 0.91 -> 1.00 of HBM on 25900 rows,
    // K = 2048 as 32 x 8 instead of 64 x 4 0.73 -> 0.87 on 16384).  The layer's
    // preparation keeps the shallower shapes: each of its blocks also widens a share of
    // the weight, and with half the blocks the deep shapes gave no faster large-shape
    // steps and slower small ones (1024x4096x4096 39.8 -> 45.3 us, the preparation no
    // longer overlapping the GEMM's start).  ConvRot rows, whose transform makes them
    // issue-bound, keep more threads per row (64 x 6 / 64 x 8 / 128 x 4 measured slower).
    int tpr = 0, vpt = 0;
    if (rotate || !OUT8) {
        if (nvec <= 64) { tpr = 32; vpt = 2; }
        else if (nvec <= 128) { tpr = 32; vpt = 4; }
        else if (nvec <= 256) { tpr = 64; vpt = 4; }
        else if (nvec <= 384) { tpr = 128; vpt = 3; }
        else if (nvec <= 512) { tpr = 128; vpt = 4; }
        else if (nvec <= 768) { tpr = 128; vpt = 6; }
        else if (nvec <= 1024) { tpr = 256; vpt = 4; }
        else if (nvec <= 1536) { tpr = 256; vpt = 6; }
        else if (nvec <= 2048) { tpr = 256; vpt = 8; }
    } else {
        if (nvec <= 64) { tpr = 32; vpt = 2; }
        else if (nvec <= 128) { tpr = 32; vpt = 4; }
        else if (nvec <= 256) { tpr = 32; vpt = 8; }
        else if (nvec <= 384) { tpr = 64; vpt = 6; }
        else if (nvec <= 512) { tpr = 64; vpt = 8; }
        else if (nvec <= 768) { tpr = 128; vpt = 6; }
        else if (nvec <= 1024) { tpr = 128; vpt = 8; }
        else if (nvec <= 1536) { tpr = 256; vpt = 6; }
        else if (nvec <= 2048) { tpr = 256; vpt = 8; }
    }
    if (tpr == 0) {
        const int64_t blocks = (M + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK;
        if (blocks > 0x7FFFFFFF)
            return cudaErrorInvalidValue;
        if (rotate)
            return launch_pdl(rows_stream_kernel<true, OUT8, OUT16>, (unsigned)blocks, THREADS, 0, s, xv, M, K, q8,
                              q16b, xs, w8, w_n16, w16);
        return launch_pdl(rows_stream_kernel<false, OUT8, OUT16>, (unsigned)blocks, THREADS, 0, s, xv, M, K, q8,
                          q16b, xs, w8, w_n16, w16);
    }
    const int64_t rpb = THREADS / tpr;
    const int64_t blocks = (M + rpb - 1) / rpb;
    if (blocks > 0x7FFFFFFF)
        return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)blocks;
#define CK_ROWS(T, V, R) \
    launch_pdl(rows_kernel<T, V, R, OUT8, OUT16>, grid, THREADS, 0, s, xv, M, K, q8, q16b, xs, w8, w_n16, w16)
#define CK_SHALLOW(R)                                  \
    switch (tpr * 16 + vpt) {                          \
    case 32 * 16 + 2: return CK_ROWS(32, 2, R);        \
    case 32 * 16 + 4: return CK_ROWS(32, 4, R);        \
    case 64 * 16 + 4: return CK_ROWS(64, 4, R);        \
    case 128 * 16 + 3: return CK_ROWS(128, 3, R);      \
    case 128 * 16 + 4: return CK_ROWS(128, 4, R);      \
    case 128 * 16 + 6: return CK_ROWS(128, 6, R);      \
    case 256 * 16 + 4: return CK_ROWS(256, 4, R);      \
    case 256 * 16 + 6: return CK_ROWS(256, 6, R);      \
    default: return CK_ROWS(256, 8, R);                \
    }
    if (rotate) {
        CK_SHALLOW(true)
    }
    if constexpr (!OUT8) {
        CK_SHALLOW(false)
    } else {
        switch (tpr * 16 + vpt) {
        case 32 * 16 + 2: return CK_ROWS(32, 2, false);
        case 32 * 16 + 4: return CK_ROWS(32, 4, false);
        case 32 * 16 + 8: return CK_ROWS(32, 8, false);
        case 64 * 16 + 6: return CK_ROWS(64, 6, false);
        case 64 * 16 + 8: return CK_ROWS(64, 8, false);
        case 128 * 16 + 6: return CK_ROWS(128, 6, false);
        case 128 * 16 + 8: return CK_ROWS(128, 8, false);
        case 256 * 16 + 6: return CK_ROWS(256, 6, false);
        default: return CK_ROWS(256, 8, false);
        }
    }
#undef CK_SHALLOW
#undef CK_ROWS
}

}  // namespace

cudaError_t launch_quantize_rows(const void* x, int64_t M, int64_t K, bool rotate, int8_t* q8, void* q16,
                                 float* x_scale, const DeviceInfo& dev, cudaStream_t s)
{
    (void)dev;
    if (M == 0)
        return cudaSuccess;
    if (q8)
        return rows_dispatch<true, false>(x, M, K, rotate, q8, q16, x_scale, nullptr, 0, nullptr, s);
    return rows_dispatch<false, true>(x, M, K, rotate, q8, q16, x_scale, nullptr, 0, nullptr, s);
}

int tensorwise_partials(const DeviceInfo& dev)
{
    int n = 4 * dev.sm_count;
    return n < 1 ? 1 : (n > 1024 ? 1024 : n);
}

cudaError_t launch_quantize_tensorwise(const void* x, int64_t M, int64_t K, int8_t* q8, void* q16, float* x_scale,
                                       float* partials, const DeviceInfo& dev, cudaStream_t s)
{
    using namespace quant;
    const int64_t nvec = (M * K) >> 3;
    const int nparts = tensorwise_partials(dev);
    const uint4* xv = static_cast<const uint4*>(x);
    __nv_bfloat16* q16b = static_cast<__nv_bfloat16*>(q16);
    cudaError_t e = launch_pdl(amax_partials_kernel, nparts, 256, 0, s, xv, nvec, partials, (const uint4*)nullptr,
                               (int64_t)0, (uint4*)nullptr);
    if (e != cudaSuccess)
        return e;
    const int grid = 4 * dev.sm_count;
    if (q8 && q16)
        e = launch_pdl(quant_flat_kernel<true, true>, grid, 256, 0, s, xv, nvec, partials, nparts, q8, q16b, x_scale);
    else if (q8)
        e = launch_pdl(quant_flat_kernel<true, false>, grid, 256, 0, s, xv, nvec, partials, nparts, q8, q16b, x_scale);
    else
        e = launch_pdl(quant_flat_kernel<false, true>, grid, 256, 0, s, xv, nvec, partials, nparts, q8, q16b, x_scale);
    return e;
}

cudaError_t launch_quantize_tensorwise_parts(const void* x, int64_t M, int64_t K, int8_t* q8, void* q16,
                                             float* x_scale, float* partials, int nparts, const DeviceInfo& dev,
                                             cudaStream_t s)
{
    using namespace quant;
    const int64_t nvec = (M * K) >> 3;
    const uint4* xv = static_cast<const uint4*>(x);
    __nv_bfloat16* q16b = static_cast<__nv_bfloat16*>(q16);
    cudaError_t e = launch_pdl(amax_partials_kernel, nparts, 256, 0, s, xv, nvec, partials, (const uint4*)nullptr,
                               (int64_t)0, (uint4*)nullptr);
    if (e != cudaSuccess)
        return e;
    const int grid = 4 * dev.sm_count;
    if (q8 && q16)
        e = launch_pdl(quant_flat_kernel<true, true>, grid, 256, 0, s, xv, nvec, partials, nparts, q8, q16b, x_scale);
    else if (q8)
        e = launch_pdl(quant_flat_kernel<true, false>, grid, 256, 0, s, xv, nvec, partials, nparts, q8, q16b, x_scale);
    else
        e = launch_pdl(quant_flat_kernel<false, true>, grid, 256, 0, s, xv, nvec, partials, nparts, q8, q16b, x_scale);
    return e;
}

cudaError_t launch_widen_int8(const int8_t* src, void* dst, int64_t n, const DeviceInfo& dev, cudaStream_t s)
{
    const int64_t n16 = n >> 4;
    if (n16 == 0)
        return cudaSuccess;
    int64_t want = (n16 + 255) / 256;
    const int64_t cap = (int64_t)8 * dev.sm_count;
    const int grid = (int)(want < cap ? want : cap);
    return launch_pdl(quant::widen_kernel, grid, 256, 0, s, reinterpret_cast<const uint4*>(src), n16,
                      static_cast<uint4*>(dst));
}

cudaError_t launch_prep_rows(const void* x, int64_t M, int64_t K, bool rotate, void* q16, float* x_scale,
                             const int8_t* w8, int64_t w_n, void* w16, const DeviceInfo& dev, cudaStream_t s)
{
    if (M == 0)
        return launch_widen_int8(w8, w16, w_n, dev, s);
    return rows_dispatch<false, true>(x, M, K, rotate, nullptr, q16, x_scale, w8, w_n, w16, s);
}

namespace {

// Blocks of tensorwise_prep_kernel that are resident at once on the whole device (the
// shared-memory attribute it needs is set once per context).
int prep_capacity(const DeviceInfo& dev)
{
    static ContextCache<int> cache;
    int per_sm = 0;
    const cudaError_t e = cache.get(&per_sm, [](int* n) {
        constexpr int TPB = quant::kPrepThreads;
        const size_t smem = (size_t)quant::kMaxStagedVectors * TPB * sizeof(uint4);
        cudaError_t r = cudaFuncSetAttribute(quant::tensorwise_prep_kernel<TPB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (r == cudaSuccess)
            r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, quant::tensorwise_prep_kernel<TPB>, TPB, smem);
        return r;
    });
    if (e != cudaSuccess || per_sm <= 0)
        per_sm = 1;
    return per_sm * dev.sm_count;
}

// A 64-bit value no earlier launch of this process used (high-entropy start, so values
// left in recycled memory by another process do not match either).
unsigned long long next_prep_epoch()
{
    static std::atomic<unsigned long long> counter([] {
        unsigned long long z = (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() ^
                               ((unsigned long long)getpid() << 29) ^ 0x9E3779B97F4A7C15ull;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;  // splitmix64 finaliser
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        return z ^ (z >> 31);
    }());
    unsigned long long e;
    do {
        e = counter.fetch_add(1, std::memory_order_relaxed);
    } while (e == 0);
    return e;
}

}  // namespace

size_t prep_tensorwise_scratch_bytes(int max_blocks)
{
    // one slot per block, then the poison word of a wait that gave up
    return sizeof(quant::EpochSlot) * ((size_t)max_blocks + 1);
}

cudaError_t launch_prep_tensorwise(const void* x, int64_t M, int64_t K, void* q16, float* x_scale, void* scratch,
                                   int max_blocks, const int8_t* w8, int64_t w_n, void* w16, const DeviceInfo& dev,
                                   cudaStream_t s)
{
    const int64_t nvec = (M * K) >> 3;
    constexpr int TPB = quant::kPrepThreads;
    const int64_t want = std::max<int64_t>(1, (nvec + TPB - 1) / TPB);
    const int64_t cap = std::min<int64_t>(prep_capacity(dev), (int64_t)quant::kMaxSlotsPerThread * TPB);
    const int grid = (int)std::min<int64_t>(std::min<int64_t>(want, cap), max_blocks);
    // vectors per thread, and how many of them step 1 keeps on chip for step 4
    const int64_t per_thread = (nvec + (int64_t)grid * TPB - 1) / ((int64_t)grid * TPB);
    const int staged = (int)std::min<int64_t>(per_thread, quant::kMaxStagedVectors);
    unsigned int* err = nullptr;
    cudaError_t e = device_error_ptr(&err);
    if (e != cudaSuccess)
        return e;
    // The blocks wait for each other's maxima, so all of them must be resident at once: the
    // grid is at most what fits on the device, and the launch is cooperative, which the
    // runtime starts only when every block can be placed (another stream's kernels may
    // hold part of the GPU).  Programmatic serialization keeps the launch overlapping the
    // previous kernel's tail.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(TPB);
    cfg.dynamicSmemBytes = (size_t)staged * TPB * sizeof(uint4);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    quant::EpochSlot* slots = static_cast<quant::EpochSlot*>(scratch);
    return cudaLaunchKernelEx(&cfg, quant::tensorwise_prep_kernel<TPB>, static_cast<const uint4*>(x), nvec, slots,
                              &slots[max_blocks].epoch, next_prep_epoch(),
                              static_cast<__nv_bfloat16*>(q16), x_scale, reinterpret_cast<const uint4*>(w8),
                              w_n >> 4, static_cast<uint4*>(w16), (uint64_t)2000000000ull, err, staged);
}

cudaError_t launch_rotate_bf16(const void* x, int64_t M, int64_t K, void* a16, const int8_t* w8, int64_t w_n,
                               void* w16, const DeviceInfo& dev, cudaStream_t s)
{
    const int64_t nvec = (M * K) >> 3;
    const int64_t want = std::max<int64_t>(1, (nvec + 255) / 256);  // 8 warps x 32 vectors per block
    const int grid = (int)std::min<int64_t>(want, (int64_t)8 * dev.sm_count);
    return launch_pdl(quant::rotate_bf16_kernel, grid, 256, 0, s, static_cast<const uint4*>(x), nvec,
                      static_cast<uint4*>(a16), reinterpret_cast<const uint4*>(w8), w_n >> 4,
                      static_cast<uint4*>(w16));
}

cudaError_t launch_widen2(const int8_t* a8, int64_t a_n, void* a16, const int8_t* b8, int64_t b_n, void* b16,
                          const DeviceInfo& dev, cudaStream_t s)
{
    const int64_t n16 = (a_n >> 4) + (b_n >> 4);
    const int64_t want = std::max<int64_t>(1, (n16 + 1023) / 1024);
    const int grid = (int)std::min<int64_t>(want, (int64_t)8 * dev.sm_count);
    return launch_pdl(quant::widen2_kernel, grid, 256, 0, s, reinterpret_cast<const uint4*>(a8), a_n >> 4,
                      static_cast<uint4*>(a16), reinterpret_cast<const uint4*>(b8), b_n >> 4,
                      static_cast<uint4*>(b16));
}

cudaError_t launch_convrot_weight(const float* W, int64_t N, int64_t K, int8_t* w, float* w_scale,
                                  const DeviceInfo& dev, cudaStream_t s)
{
    (void)dev;
    using namespace quant;
    if (N == 0)
        return cudaSuccess;
    const float4* Wv = reinterpret_cast<const float4*>(W);
    const int64_t nvec = K / 8;
    int tpr, vpt;
    if (nvec <= 128) { tpr = 32; vpt = 4; }
    else if (nvec <= 256) { tpr = 64; vpt = 4; }
    else if (nvec <= 512) { tpr = 128; vpt = 4; }
    else if (nvec <= 1024) { tpr = 256; vpt = 4; }
    else if (nvec <= 2048) { tpr = 256; vpt = 8; }
    else { tpr = 0; vpt = 0; }
    if (tpr == 0) {
        const int64_t blocks = (N + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK;
        if (blocks > 0x7FFFFFFF)
            return cudaErrorInvalidValue;
        return launch_pdl(weight_rot_stream_kernel, (unsigned)blocks, THREADS, 0, s, Wv, N, K, w, w_scale);
    }
    const int64_t blocks = (N + THREADS / tpr - 1) / (THREADS / tpr);
    if (blocks > 0x7FFFFFFF)
        return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)blocks;
    switch (tpr * 16 + vpt) {
    case 32 * 16 + 4: return launch_pdl(weight_rot_kernel<32, 4>, grid, THREADS, 0, s, Wv, N, K, w, w_scale);
    case 64 * 16 + 4: return launch_pdl(weight_rot_kernel<64, 4>, grid, THREADS, 0, s, Wv, N, K, w, w_scale);
    case 128 * 16 + 4: return launch_pdl(weight_rot_kernel<128, 4>, grid, THREADS, 0, s, Wv, N, K, w, w_scale);
    case 256 * 16 + 4: return launch_pdl(weight_rot_kernel<256, 4>, grid, THREADS, 0, s, Wv, N, K, w, w_scale);
    default: return launch_pdl(weight_rot_kernel<256, 8>, grid, THREADS, 0, s, Wv, N, K, w, w_scale);
    }
}

}  // namespace ck
