// Device helpers shared by the routing kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace mr {

constexpr unsigned kFull = 0xffffffffu;

// 16-byte streaming load of data read once per launch (the gate weight):
// read-only path, no L1 allocation.  volatile: the load is issued where it
// is written, so loads of parameters placed before the programmatic-
// dependent-launch wait are in flight while the kernel waits (a plain asm
// without memory operands may be sunk to its first use, after the wait).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16-byte read-only load that may be served from L1 (activations reused by
// the warps of one CTA).
__device__ __forceinline__ uint4 ld_ro_v4(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// D += A * B for one m16n8k16 bf16 tile with fp32 accumulation (no side
// effects beyond its outputs, so the compiler may interleave independent ones).
__device__ __forceinline__ void mma_bf16_m16n8k16(float (&c)[4], uint32_t a0, uint32_t a1,
                                                  uint32_t a2, uint32_t a3, uint32_t b0,
                                                  uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A * B for one m16n8k16 f16 tile with fp32 accumulation.
__device__ __forceinline__ void mma_f16_m16n8k16(float (&c)[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0,
                                                 uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two bf16 (one 32-bit pair) -> two f16.  *exact is cleared unless both
// convert exactly: zero, or a biased exponent in [110, 142] (2^-17 <= |v| <
// 2^16: f16 covers that bf16 range to the last bit, its subnormal spacing
// 2^-24 down to 2^-17; larger values overflow and smaller ones lose bits).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t two, bool* exact) {
    const uint32_t e_lo = (two >> 7) & 0xFFu, e_hi = (two >> 23) & 0xFFu;
    const bool ok_lo = (two & 0x7FFFu) == 0u || (e_lo >= 110u && e_lo <= 142u);
    const bool ok_hi = (two & 0x7FFF0000u) == 0u || (e_hi >= 110u && e_hi <= 142u);
    if (!(ok_lo && ok_hi)) *exact = false;
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__uint_as_float(two & 0xFFFF0000u)), "f"(__uint_as_float(two << 16)));
    return r;
}

// Two E4M3 codes (the low 16 bits) -> two f16 (exact: every E4M3 value is an f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    return (uint32_t)hr.x | ((uint32_t)hr.y << 16);
}

// Router input on the norm's scale: two bf16 residual values (one 32-bit
// pair) -> bf16((x * rstd) * s) with s = g or, for a Gemma RMSNorm, 1 + g;
// each fp32 step rounds to nearest even (no contraction), and the bf16
// store rounds to nearest even.  Subnormals are kept (no -ftz).
__device__ __forceinline__ uint32_t norm_pair(uint32_t xp, uint32_t gp, float rstd, bool gemma) {
    const float x0 = __uint_as_float(xp << 16), x1 = __uint_as_float(xp & 0xffff0000u);
    float s0 = __uint_as_float(gp << 16), s1 = __uint_as_float(gp & 0xffff0000u);
    if (gemma) {
        s0 = __fadd_rn(1.0f, s0);
        s1 = __fadd_rn(1.0f, s1);
    }
    const float p0 = __fmul_rn(__fmul_rn(x0, rstd), s0);
    const float p1 = __fmul_rn(__fmul_rn(x1, rstd), s1);
    uint32_t d;  // upper half from the first source operand
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(p1), "f"(p0));
    return d;
}

// Eight consecutive elements of a row (one 16-byte chunk) through norm_pair.
__device__ __forceinline__ uint4 norm_chunk(uint4 x, uint4 g, float rstd, bool gemma) {
    return make_uint4(norm_pair(x.x, g.x, rstd, gemma), norm_pair(x.y, g.y, rstd, gemma),
                      norm_pair(x.z, g.z, rstd, gemma), norm_pair(x.w, g.w, rstd, gemma));
}

// Programmatic dependent launch.  pdl_wait() blocks until the kernel
// launched before this one on the stream has completed and its writes are
// visible (a no-op when the launch did not allow overlap); pdl_trigger()
// lets the next kernel on the stream start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Last-arriver ticket: returns the counter value before this CTA's increment.
// The whole CTA calls it after writing what it publishes.  The barrier
// orders every thread's writes before thread 0's fence and acq_rel atomic,
// which publish them at gpu scope (release is cumulative: one thread's
// fence covers what the barrier ordered before it) and, in the CTA that
// draws the last ticket, acquire every other CTA's; the second barrier
// passes that on to the CTA's threads, which then read the published data
// through L2 (ld.cg).  (A fence in every thread measured slower.)
__device__ __forceinline__ unsigned cta_ticket(unsigned* counter, unsigned* s_slot) {
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned old;
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
        *s_slot = old;
    }
    __syncthreads();
    return *s_slot;
}

// Optional phase stamps (compile with -DMR_TRACE), 512 u64 per CTA at
// trace + (blockIdx.y * gridDim.x + blockIdx.x) * 512.  %globaltimer (ns):
// MR_TRACE_STAMP: thread 0 writes slot (< 32), and %clock64 (SM cycles) at
// slot 288 + slot; MR_TRACE_WARP: lane 0 of every warp writes slot
// 32 + 16 * phase + warp (phase < 14, 16 warps at most).
// MR_TRACE_CLK: thread 0 writes %clock64 at slot 256 + slot (< 32).
#ifdef MR_TRACE
#define MR_TRACE_AT(trace, slot)                                                     \
    do {                                                                             \
        unsigned long long t_;                                                       \
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                       \
        (trace)[(blockIdx.y * gridDim.x + blockIdx.x) * 512 + (slot)] = t_;          \
    } while (0)
#define MR_TRACE_STAMP(trace, slot)                                                  \
    do {                                                                             \
        if (threadIdx.x == 0 && (trace) != nullptr) {                                \
            MR_TRACE_AT(trace, slot);                                                \
            (trace)[(blockIdx.y * gridDim.x + blockIdx.x) * 512 + 288 + (slot)] = clock64(); \
        }                                                                            \
    } while (0)
#define MR_TRACE_WARP(trace, phase)                                                  \
    do {                                                                             \
        if ((threadIdx.x & 31) == 0 && (trace) != nullptr)                           \
            MR_TRACE_AT(trace, 32 + 16 * (phase) + (threadIdx.x >> 5));              \
    } while (0)
#define MR_TRACE_CLK(trace, slot)                                                    \
    do {                                                                             \
        if (threadIdx.x == 0 && (trace) != nullptr)                                  \
            (trace)[(blockIdx.y * gridDim.x + blockIdx.x) * 512 + 256 + (slot)] = clock64(); \
    } while (0)
#else
#define MR_TRACE_CLK(trace, slot) \
    do {                          \
    } while (0)
#define MR_TRACE_STAMP(trace, slot) \
    do {                            \
    } while (0)
#define MR_TRACE_WARP(trace, phase) \
    do {                            \
    } while (0)
#endif

// Orderable image of an fp32 key: larger float -> larger unsigned.  The key
// is first canonicalised (-0 -> +0) so that the two zeros tie.
__device__ __forceinline__ unsigned ordered_key(float v) {
    unsigned u = __float_as_uint(__fadd_rn(v, 0.0f));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_sum_fixed(float v) {
    // butterfly: same tree on every call, so the sum is deterministic
    v = __fadd_rn(v, __shfl_xor_sync(kFull, v, 16));
    v = __fadd_rn(v, __shfl_xor_sync(kFull, v, 8));
    v = __fadd_rn(v, __shfl_xor_sync(kFull, v, 4));
    v = __fadd_rn(v, __shfl_xor_sync(kFull, v, 2));
    v = __fadd_rn(v, __shfl_xor_sync(kFull, v, 1));
    return v;
}

// ---------------------------------------------------------------- MXFP8

// E8M0 exponent X of a 32-block from the largest |x| as a bf16 magnitude
// pattern (sign cleared): X = floor(log2(amax)) - emax (8 for E4M3, 2 for
// E2M1), clamped to [-127, 127]; amax == 0 gives -127.  For a normal bf16
// floor(log2(amax)) is its exponent field e minus 127; a subnormal or zero
// amax (e = 0) has floor(log2) <= -127, so X <= -129 clamps to -127, as
// e - 127 - emax does; e <= 255 keeps X <= 128 - emax < 127.  So X is
// max(e - 127 - emax, -127) for every pattern.
__device__ __forceinline__ int mx_scale_exponent(unsigned amax16, int emax) {
    return max((int)(amax16 >> 7) - 127 - emax, -127);
}

// Largest |x| of a 32-block as a bf16 magnitude pattern: the 8 values of v
// (this lane) and those of the other 3 lanes of its quad.  Non-negative bf16
// patterns order like their values, so the maximum runs on packed 16-bit
// integers (sign bits cleared).
__device__ __forceinline__ unsigned vmax_u16x2(unsigned a, unsigned b) {
    unsigned d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ unsigned quad_amax16(uint4 v) {
    unsigned m = vmax_u16x2(vmax_u16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                            vmax_u16x2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
    m = vmax_u16x2(m, __shfl_xor_sync(kFull, m, 1));
    m = vmax_u16x2(m, __shfl_xor_sync(kFull, m, 2));
    return max(m & 0xFFFFu, m >> 16);
}

// Quantise the 8 consecutive bf16 values of v (k = 8t .. 8t+7 of a 32-block
// spread over the 4 lanes t = lane & 3 of a lane quad).  All 32 lanes of the
// warp must call it together.  Returns the 8 e4m3 codes (lowest k in the
// lowest byte) and writes the block's E8M0 byte to *scale_byte.
__device__ __forceinline__ uint2 mx_quant_quad(uint4 v, unsigned* scale_byte) {
    int X = mx_scale_exponent(quad_amax16(v), 8);
    *scale_byte = (unsigned)(X + 127);
    // 2^-X is a normal fp32 for every X reachable from bf16 input (X <= 119).
    float inv = __uint_as_float((unsigned)(127 - X) << 23);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float lo = __fmul_rn(__uint_as_float(w[i] << 16), inv);
        float hi = __fmul_rn(__uint_as_float(w[i] & 0xFFFF0000u), inv);
        __nv_fp8x2_storage_t p = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
        if (i & 1)
            out[i >> 1] |= (uint32_t)p << 16;
        else
            out[i >> 1] = (uint32_t)p;
    }
    return make_uint2(out[0], out[1]);
}

// Two E4M3 codes (lower k in the low byte) -> two bf16 values (lower k in
// the low half), exactly: every E4M3 value is a normal f16 or zero (the
// conversion to f16 is exact), and its three mantissa bits sit at the top of
// the f16 mantissa, so the bf16 code is the f16 magnitude shifted right by 3
// with the exponent rebiased by 127 - 15 = 112; zeros stay zero.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    const uint32_t h = (uint32_t)hr.x | ((uint32_t)hr.y << 16);
    const uint32_t mag = h & 0x7FFF7FFFu;
    uint32_t nz;  // 1 in each half whose magnitude is nonzero
    asm("min.u16x2 %0, %1, %2;" : "=r"(nz) : "r"(mag), "r"(0x00010001u));
    return (h & 0x80008000u) | (((mag >> 3) & 0x0FFF0FFFu) + nz * 0x3800u);
}

// 2^(byte - 127) as fp32 for an E8M0 scale byte < 255 (byte 0: the subnormal 2^-127).
__device__ __forceinline__ float e8m0_value(unsigned byte) {
    return byte != 0u ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}

// ---------------------------------------------------------------- MXFP4

// Eight fp32 values -> eight E2M1 codes (round to nearest even, saturating
// to +-6, sign kept), element i in bits 4i .. 4i + 3.  The conversion puts
// its first source operand in the high nibble of each byte.
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
    uint32_t d;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(d)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return d;
}

// MXFP4 of the 8 consecutive bf16 values of v (one lane of the lane quad
// that holds a 32-block, as mx_quant_quad).  Returns the 8 packed E2M1 codes
// (element i in nibble i: 4 bytes of the [M, K/2] output) and writes the
// block's E8M0 byte X + 127, X = floor(log2(amax)) - 2.
__device__ __forceinline__ uint32_t mx4_quant_quad(uint4 v, unsigned* scale_byte) {
    int X = mx_scale_exponent(quad_amax16(v), 2);
    *scale_byte = (unsigned)(X + 127);
    // X in [-127, 125] for bf16 input: 2^-X is a normal fp32, and x * 2^-X
    // is exact wherever it can round to a nonzero code
    float inv = __uint_as_float((unsigned)(127 - X) << 23);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __fmul_rn(__uint_as_float(w[i] << 16), inv);
        f[2 * i + 1] = __fmul_rn(__uint_as_float(w[i] & 0xFFFF0000u), inv);
    }
    return e2m1x8(f);
}

// ---------------------------------------------------------------- sigmoid
//
// The sigmoid gate (sglang #46652, Modifications: fp32 sigmoid scores plus a
// per-expert selection bias) scores expert n by s = sigma(l) = 1 / (1 + e^-l)
// of its fp32 logit, rounded once to the nearest fp32 value (the correctly
// rounded sigmoid), and selects by the fp32 sum s + bias.  Evaluating that
// exactly for every expert would need fp64 throughout, which runs at a small
// fraction of the fp32 rate here, so the gate works in two steps:
//   1. sigmoid_approx (fp32, a few ulps) for every expert: selection keys good
//      to well within kSigmoidKeyMargin, used only to find candidates;
//   2. sigmoid_exact for the few candidates whose approximate key lies within
//      the margin of the k-th largest: the correctly rounded score, from which
//      the exact keys, the ranking and the weights are formed.

// fp32 sigmoid good to a few ulps (every step rounded to nearest, no
// contraction): y = clamp(-l, -87, 88); n = rint(y log2 e); Cody and Waite's
// reduction r = y - n ln2 with a two-part ln 2; e^r by its degree-7 Taylor
// polynomial in Horner form (truncation below 2^-27 on |r| <= ln2 / 2);
// s = 1 / (1 + p 2^n).  Its absolute error is below 2^-21 for every l (below
// 2^-37 once the clamp acts), so selection keys s + bias from it lie within
// 2^-20 of the exact keys.
__device__ __forceinline__ float sigmoid_approx(float l) {
    float y = -l;
    y = y < -87.0f ? -87.0f : y;
    y = y > 88.0f ? 88.0f : y;
    float n = rintf(__fmul_rn(y, 0x1.715476p+0f));
    float r = __fmaf_rn(-n, 0x1.62e430p-1f, y);
    r = __fmaf_rn(-n, -0x1.05c610p-29f, r);
    float p = 0x1.a01a02p-13f;
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
    p = __fmaf_rn(p, r, 0x1.111112p-7f);
    p = __fmaf_rn(p, r, 0x1.555556p-5f);
    p = __fmaf_rn(p, r, 0x1.555556p-3f);
    p = __fmaf_rn(p, r, 0x1p-1f);
    p = __fmaf_rn(p, r, 0x1p+0f);
    p = __fmaf_rn(p, r, 0x1p+0f);
    float two_n = __uint_as_float((unsigned)((int)n + 127) << 23);
    float e = __fmul_rn(p, two_n);
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
}

// Keys within this distance below the k-th largest approximate key are
// re-scored exactly (four times the worst gap between approximate and exact
// keys, so that every expert of the exact top-k is a candidate).
constexpr float kSigmoidKeyMargin = 0x1p-18f;

// Double-double arithmetic (a value is hi + lo, |lo| <= ulp(hi) / 2): the
// error-free sum of Knuth and product via fma of Dekker, and the accurate
// addition and division of Hida, Li and Bailey's double-double library
// ("Algorithms for quad-double precision floating point arithmetic", 2001).
// Every operation is an explicit round-to-nearest intrinsic (no contraction).
struct ddouble {
    double hi, lo;
};
__device__ __forceinline__ ddouble dd_two_sum(double a, double b) {
    const double s = __dadd_rn(a, b), bb = __dsub_rn(s, a);
    return {s, __dadd_rn(__dsub_rn(a, __dsub_rn(s, bb)), __dsub_rn(b, bb))};
}
__device__ __forceinline__ ddouble dd_quick_two_sum(double a, double b) {  // |a| >= |b|
    const double s = __dadd_rn(a, b);
    return {s, __dsub_rn(b, __dsub_rn(s, a))};
}
__device__ __forceinline__ ddouble dd_two_prod(double a, double b) {
    const double p = __dmul_rn(a, b);
    return {p, __fma_rn(a, b, -p)};
}
__device__ __forceinline__ ddouble dd_add(ddouble a, ddouble b) {
    ddouble s = dd_two_sum(a.hi, b.hi);
    const ddouble t = dd_two_sum(a.lo, b.lo);
    s.lo = __dadd_rn(s.lo, t.hi);
    s = dd_quick_two_sum(s.hi, s.lo);
    s.lo = __dadd_rn(s.lo, t.lo);
    return dd_quick_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ ddouble dd_mul(ddouble a, ddouble b) {
    ddouble p = dd_two_prod(a.hi, b.hi);
    p.lo = __dadd_rn(p.lo, __dadd_rn(__dmul_rn(a.hi, b.lo), __dmul_rn(a.lo, b.hi)));
    return dd_quick_two_sum(p.hi, p.lo);
}
__device__ __forceinline__ ddouble dd_mul_d(ddouble a, double b) {
    ddouble p = dd_two_prod(a.hi, b);
    p.lo = __fma_rn(a.lo, b, p.lo);
    return dd_quick_two_sum(p.hi, p.lo);
}
__device__ __forceinline__ ddouble dd_div(ddouble a, ddouble b) {
    // three quotient digits, each from the remainder of the previous ones
    const double q1 = __ddiv_rn(a.hi, b.hi);
    ddouble r = dd_add(a, dd_mul_d(b, -q1));
    const double q2 = __ddiv_rn(r.hi, b.hi);
    r = dd_add(r, dd_mul_d(b, -q2));
    const double q3 = __ddiv_rn(r.hi, b.hi);
    ddouble q = dd_quick_two_sum(q1, q2);
    return dd_add(q, ddouble{q3, 0.0});
}

// The fp64 level with its rounding test, then double-double (see
// sigmoid_exact): out of line, since the float-float level decides almost
// every call.
static __device__ __noinline__ float sigmoid_exact_wide(float l, bool slow);

// sigma(l) correctly rounded to fp32, evaluated in double-double (relative
// error far below 2^-90): ln 2 as three doubles (its value to 2^-160), n =
// rint(y / ln2), r = y - n ln 2 (|r| <= ln2 / 2), e^r by its Taylor series to
// degree 24 (truncation below 2^-115) in the nested form
// 1 + r (1 + r/2 (1 + r/3 (...))), E = 2^n e^r, S = 1 / (1 + E); then the
// one rounding of hi + lo to fp32.  Outside y = -l in (-20, 104) the result
// is decided without evaluation: sigma < e^-104 < 2^-150 rounds to 0, and
// 1 - sigma < e^-20 < 2^-25 rounds to 1.
static __device__ __noinline__ float sigmoid_dd(float l) {
    const double y = -(double)l;
    if (y >= 104.0) return 0.0f;
    if (y <= -20.0) return 1.0f;
    constexpr double ln2_1 = 0x1.62e42fefa39efp-1, ln2_2 = 0x1.abc9e3b39803fp-56, ln2_3 = 0x1.7b57a079a1934p-111;
    const double n = rint(__dmul_rn(y, 0x1.71547652b82fep+0));
    const ddouble p1 = dd_two_prod(-n, ln2_1);  // -n ln2_1 exactly
    ddouble r = dd_add(ddouble{y, 0.0}, p1);
    r = dd_add(r, dd_two_prod(-n, ln2_2));
    r = dd_add(r, ddouble{__dmul_rn(-n, ln2_3), 0.0});
    ddouble p = {1.0, 0.0};
    for (int j = 24; j >= 1; --j) {
        const ddouble rj = dd_div(r, ddouble{(double)j, 0.0});
        p = dd_add(ddouble{1.0, 0.0}, dd_mul(rj, p));
    }
    const double two_n = __longlong_as_double((long long)((int)n + 1023) << 52);  // n in [-29, 151]
    const ddouble E = {__dmul_rn(p.hi, two_n), __dmul_rn(p.lo, two_n)};
    const ddouble S = dd_div(ddouble{1.0, 0.0}, dd_add(ddouble{1.0, 0.0}, E));
    // the fp32 value nearest to S.hi + S.lo: that of S.hi unless S.hi is
    // exactly the midpoint between two fp32 values, where S.lo decides
    const float c = __double2float_rn(S.hi);
    const double cd = (double)c;
    if (cd == S.hi) return c;
    const float nb = S.hi > cd ? __uint_as_float(__float_as_uint(c) + 1u) : __uint_as_float(__float_as_uint(c) - 1u);
    const double mid = __dmul_rn(0.5, __dadd_rn(cd, (double)nb));  // exact: a midpoint of fp32 values
    if (S.hi != mid) return c;
    return ((S.lo > 0.0) == (nb > c)) ? nb : c;
}

static __device__ __noinline__ float sigmoid_exact_wide(float l, bool slow) {
    const double e = exp(-(double)l);
    const double s = __ddiv_rn(1.0, __dadd_rn(1.0, e));
    const double m = __dmul_rn(s, 0x1p-48);
    const float lo = __double2float_rn(__dsub_rn(s, m)), hi = __double2float_rn(__dadd_rn(s, m));
    if (lo == hi && !slow) return lo;
    return sigmoid_dd(l);
}

// Float-float arithmetic (a value is hi + lo in fp32, |lo| <= ulp(hi) / 2):
// the same error-free transformations and accurate addition and division as
// the double-double ones above, on fp32 FMA pipes (which run at many times
// the fp64 rate here); relative error of an operation a few 2^-48.
struct ffloat {
    float hi, lo;
};
__device__ __forceinline__ ffloat ff_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b), bb = __fsub_rn(s, a);
    return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ ffloat ff_quick_two_sum(float a, float b) {  // |a| >= |b|
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ ffloat ff_two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ ffloat ff_add(ffloat a, ffloat b) {
    ffloat s = ff_two_sum(a.hi, b.hi);
    const ffloat t = ff_two_sum(a.lo, b.lo);
    s.lo = __fadd_rn(s.lo, t.hi);
    s = ff_quick_two_sum(s.hi, s.lo);
    s.lo = __fadd_rn(s.lo, t.lo);
    return ff_quick_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ ffloat ff_mul(ffloat a, ffloat b) {
    ffloat p = ff_two_prod(a.hi, b.hi);
    p.lo = __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, p.lo));
    return ff_quick_two_sum(p.hi, p.lo);
}
__device__ __forceinline__ ffloat ff_div(ffloat a, ffloat b) {
    const float q1 = __fdiv_rn(a.hi, b.hi);
    ffloat r = ff_add(a, ff_mul(b, ffloat{-q1, 0.0f}));
    const float q2 = __fdiv_rn(r.hi, b.hi);
    r = ff_add(r, ff_mul(b, ffloat{-q2, 0.0f}));
    const float q3 = __fdiv_rn(r.hi, b.hi);
    return ff_add(ff_quick_two_sum(q1, q2), ffloat{q3, 0.0f});
}

// sigma(l) in float-float for |l| <= 69, with Ziv's rounding test: *done
// is set when the fp32 value returned is sigma correctly rounded.  With
// a = |l| and z = e^-a = 2^-n e^u, n = rint(a log2 e), u = n ln2 - a in
// [-ln2/2, ln2/2] (ln 2 as three floats, good to 2^-72): e^u by its Taylor
// series to degree 11 (truncation below 2^-47), degrees 7-11 in fp32 on
// u.hi (below 2^-47 of the sum), degrees 6..0 as float-float Horner steps;
// sigma = 1 / (1 + z) for l >= 0, z / (1 + z) for l < 0 (no overflow, and z
// >= e^-69 stays a normal fp32).  The evaluation's relative error is below
// 2^-42; sigma rounds to s.hi when both s (1 -+ 2^-39) lie inside s.hi's
// rounding interval (the margin also covers the rounding of the test).
__device__ __forceinline__ float sigmoid_ff(float l, bool* done) {
    const float a = fabsf(l);
    *done = false;
    if (!(a <= 69.0f)) return 0.0f;
    const float n = rintf(__fmul_rn(a, 0x1.715476p+0f));
    ffloat u = ff_add(ff_two_prod(n, 0x1.62e430p-1f), ffloat{-a, 0.0f});
    u = ff_add(u, ff_two_prod(n, -0x1.05c610p-29f));
    u = ff_add(u, ffloat{__fmul_rn(n, -0x1.950d88p-54f), 0.0f});
    float t = 0x1.ae6456p-26f;  // 1/11!, then 1/10! .. 1/7!
    t = __fmaf_rn(t, u.hi, 0x1.27e4fcp-22f);
    t = __fmaf_rn(t, u.hi, 0x1.71de3ap-19f);
    t = __fmaf_rn(t, u.hi, 0x1.a01a02p-16f);
    t = __fmaf_rn(t, u.hi, 0x1.a01a02p-13f);
    ffloat p = {t, 0.0f};
    p = ff_add(ffloat{0x1.6c16c2p-10f, -0x1.27d27ep-35f}, ff_mul(u, p));  // 1/6!
    p = ff_add(ffloat{0x1.111112p-7f, -0x1.dddddep-32f}, ff_mul(u, p));   // 1/5!
    p = ff_add(ffloat{0x1.555556p-5f, -0x1.555556p-30f}, ff_mul(u, p));   // 1/4!
    p = ff_add(ffloat{0x1.555556p-3f, -0x1.555556p-28f}, ff_mul(u, p));   // 1/3!
    p = ff_add(ffloat{0x1p-1f, 0.0f}, ff_mul(u, p));
    p = ff_add(ffloat{1.0f, 0.0f}, ff_mul(u, p));
    p = ff_add(ffloat{1.0f, 0.0f}, ff_mul(u, p));
    const float two_mn = __uint_as_float((unsigned)(127 - (int)n) << 23);  // n in [0, 100]
    const ffloat z = {__fmul_rn(p.hi, two_mn), __fmul_rn(p.lo, two_mn)};
    const ffloat s = ff_div(l >= 0.0f ? ffloat{1.0f, 0.0f} : z, ff_add(ffloat{1.0f, 0.0f}, z));
    const float c = s.hi;  // in [e^-69 / 2, 1]: normal, positive
    const float up = __fsub_rn(__uint_as_float(__float_as_uint(c) + 1u), c);
    const float dn = __fsub_rn(c, __uint_as_float(__float_as_uint(c) - 1u));
    const float m = __fmul_rn(c, 0x1p-39f);
    *done = __fadd_rn(s.lo, m) < __fmul_rn(0.5f, up) && __fsub_rn(s.lo, m) > -__fmul_rn(0.5f, dn);
    return c;
}

// sigma(l) correctly rounded to fp32.  First the float-float evaluation with
// its rounding test (decides all but about one logit in 10^4).  Then fp64:
// the CUDA Math API documents exp (double) to within 1 ulp, and the addition
// and the division each round once, so s = sigma (1 + d) with |d| <= 2^-51;
// rounding is monotone, so if s (1 - 2^-48) and s (1 + 2^-48) round to the
// same fp32 value, so does sigma (Ziv's rounding test, "Fast evaluation of
// elementary mathematical functions with correctly rounded last bit", 1991).
// Otherwise (about one logit in 10^7, or every call when slow is set, a
// test hook) the double-double evaluation decides.  Non-negative result; +0
// when sigma is below half the smallest fp32 subnormal.
__device__ __forceinline__ float sigmoid_exact(float l, bool slow) {
    if (!slow) {
        bool done;
        const float r = sigmoid_ff(l, &done);
        if (done) return r;
    }
    return sigmoid_exact_wide(l, slow);
}

// The same, out of line, for the standalone gate: it calls it for the few
// candidates only, and inlined at its call sites (one per unrolled key) it
// made the kernel's code several times larger.  (The route kernel's one
// call site stays inline: out of line measured 0.2-0.3 us slower there.)
static __device__ __noinline__ float sigmoid_exact_call(float l, bool slow) { return sigmoid_exact(l, slow); }

// Inverse of ordered_key (the canonical fp32 value of a key).
__device__ __forceinline__ float key_value(unsigned key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// The lowest approximate key that can still belong to the exact top-k, given
// the k-th largest approximate key kth (an ordered key).
__device__ __forceinline__ unsigned sigmoid_candidate_floor(unsigned kth) {
    return ordered_key(__fsub_rn(key_value(kth), kSigmoidKeyMargin));
}

}  // namespace mr
