// dsa_decode.cuh -- the fused decode-step kernel of diagonal-aware sparse
// attention ("Understanding and Exploiting Diagonal Attention Sparsity in
// Autoregressive Image Generation", section 4, Algorithm 1 and Fig. 12;
// section 5.1 for Diagonal+sink4 and the fused-kernel description).
//
// One launch is a persistent grid whose warps each take work items
// (stream, split) in turn; a stream is one sequence-head of one layer.  Per
// item, one warp performs:
//   a2  append: the current token, read into registers, is stored to ring
//       slot t' mod R (the slot of the entry evicted at this step) or,
//       during the sink fill, to prefix row L_p + t (in the fused layer step
//       the projection has stored it there already, and the kernel reads it
//       from that slot);
//   a4  index set: the attended relative offsets r in [0, min(t'+1, R)) whose
//       skip bit is clear, listed by a warp scan over the mask words;
//   a5  gather + logits: the prompt rows (bulk copies) and the attended ring
//       rows (TMA tile::gather4, four rows per instruction, or contiguous
//       bulk runs when nothing can be skipped) stream through the warp's
//       shared-memory stages; fp32 logits q.k with 8 lanes per row;
//   a6  online softmax and P.V, combined over the warp's row groups with
//       shuffles;
//   a7  split combine: when a stream is split into 2 or 4 pieces, they are
//       warps of one CTA and the piece-0 warp combines them through shared
//       memory; otherwise split items write (m, l, acc, argmin) partials
//       that merge_kernel, launched right after, combines;
//   a8  fused argmin over the attended decode logits on selection steps; the
//       warp (the piece-0 warp, or merge_kernel, for split streams) sets bit
//       r* of the stream's relative-offset skip mask.
// The diagonal shift (+1 per step) costs nothing: skipped entries are kept as
// relative offsets r = t' - position, which the shift leaves unchanged, and
// the slot of offset r is (t' - r) mod R.  Many independent warps per SM each
// keep their own copies in flight, so no single warp's issue rate or latency
// bounds the HBM stream.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "dsa_ptx.cuh"

namespace dsa {

enum : int { ST_TIMEOUT = 1, ST_CHECK = 2 };

// Time cap of every bounded wait, in nanoseconds of the global timer.
constexpr uint64_t kWaitNs = 1000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the barrier phase: each poll sleeps until the phase completes
// or kPollNs pass; gives up after `limit` polls or after kWaitNs in total.
// limit == 0 gives up without polling (the test knob).
constexpr uint32_t kPollNs = 20000;

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, uint32_t limit)
{
    if (limit == 0) return false;
    if (mbar_try_wait_sleep(bar, parity, kPollNs)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1; i < limit; ++i) {
        if (globaltimer_ns() - t0 > kWaitNs) return false;
        if (mbar_try_wait_sleep(bar, parity, kPollNs)) return true;
    }
    return false;
}

// Waits (time-capped) for copies already issued.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, parity, kPollNs))
        if (globaltimer_ns() - t0 > kWaitNs) return;
}

struct DecodeParams {
    const void *q;        // [S, D]
    const void *knew;     // [S, D]
    const void *vnew;     // [S, D]
    void *out;            // [S, D]
    void *prefix;         // [S, Lcap, 2, D]  (K row then V row)
    void *ring;           // [S, R, 2, D]
    uint32_t *mask;       // [S, MW]   bit r: relative offset r skipped
    int32_t *last_sel;    // [S]
    float *part_acc;      // [S, pstride, D]
    float2 *part_ml;      // [S, pstride]  (m, l)
    float2 *part_min;     // [S, pstride]  (min logit, r as int bits)
    int *status;          // sticky device status bits
    int S;
    int Lcap;             // prefix rows per stream (L_p + sink)
    int P;                // prefix rows attended at this step
    int sinkmode;         // 1: the new token goes to prefix row P
    int R;                // ring slots (N_r - sink)
    int tin;              // inner step t' = t - sink (-1 in sink mode)
    int tin_mod;          // t' mod R: ring slot of the current token (0 in sink mode)
    int wlen;             // live window length min(t' + 1, R) (1 in sink mode)
    int a;                // attended decode rows (host count)
    int n;                // P + a
    int nsplit;           // work items per stream
    int nbuf;             // shared-memory stages per warp (2 .. kMaxNbuf)
    int chunk;            // rows per work item (multiple of the stage rows)
    int nitems;           // S * nsplit
    int pstride;          // partial slots per stream
    int select;           // 1: selection step (fused argmin)
    int noskip;           // 1: N_att == N_r, no offset is ever skipped
    int MW;               // mask words per stream
    int *step_dev;        // graph mode: [0] the decode step t on the device, [1] CTAs finished (NULL: host values)
    int sink;             // t - t' (graph mode derives t' mod R from [0])
    int early;            // 1: the previous grid in the stream does not write this state, so
                          // the mask, prefix and ring may be read before the grid dependency wait
    uint16_t *glist;      // [S, LS] attended relative offsets, ascending (steady state), or NULL
    int LS;               // entries per stream of glist (even)
    int list_mode;        // 0: list from the mask; 1: list from the mask and store it to glist;
                          // 2: read the list from glist (the mask no longer changes)
    int appended;         // 1: the current token is already stored in its slot (read there, no append)
    int cta_merge;        // 1 (nsplit 2 or 4): the pieces of a stream are warps of one CTA, and the
                          // piece-0 warp combines them through shared memory (no partials, no merge launch)
    float qscale;         // log2(e) / sqrt(D), applied to q.k
    const float *kscale;  // [S] FP8 storage: K scale, V scale and their fp32 inverses
    const float *vscale;  //     (NULL for bf16 / fp32 storage)
    const float *kinv;
    const float *vinv;
    uint32_t wait_limit;
};

// Packed fp32 FMA on two lanes of a register pair: (d0, d1) += (a0, a1) * (b0, b1).
__device__ __forceinline__ void fma_f32x2(float &d0, float &d1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 A, B, C;\n\t"
        "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\tmov.b64 C, {%0, %1};\n\t"
        "fma.rn.f32x2 C, A, B, C;\n\tmov.b64 {%0, %1}, C;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// 2^x on the special-function unit.
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A stored vector (16 or 8 bytes) held in, and taken back from, a uint4.
__device__ __forceinline__ uint4 to_u4(const uint4 &v) { return v; }
__device__ __forceinline__ uint4 to_u4(const uint2 &v) { return make_uint4(v.x, v.y, 0u, 0u); }
template <typename V>
__device__ __forceinline__ V from_u4(const uint4 &x);
template <>
__device__ __forceinline__ uint4 from_u4<uint4>(const uint4 &x) { return x; }
template <>
__device__ __forceinline__ uint2 from_u4<uint2>(const uint4 &x) { return make_uint2(x.x, x.y); }

// Per element type: the query fragment a lane keeps, the q.k partial dot
// product of one 16-byte vector, and acc += p * v for one 16-byte vector.
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    using IO = float;                   // type of q, k_new, v_new, prompt K / V and out
    using Vec = uint4;                  // one stored vector of a K or V row
    static constexpr bool SCALED = false;
    static constexpr int VEC = 4;       // elements per Vec
    struct Q { float x[4]; };
    static __device__ __forceinline__ Q load_q(const uint4 &v)
    {
        return Q{{__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w)}};
    }
    // returns two partial sums (even / odd elements)
    static __device__ __forceinline__ void dot(const Q &q, const uint4 &k, float &s0, float &s1)
    {
        fma_f32x2(s0, s1, q.x[0], q.x[1], __uint_as_float(k.x), __uint_as_float(k.y));
        fma_f32x2(s0, s1, q.x[2], q.x[3], __uint_as_float(k.z), __uint_as_float(k.w));
    }
    static __device__ __forceinline__ void axpy(float p, const uint4 &v, float *acc)
    {
        fma_f32x2(acc[0], acc[1], p, p, __uint_as_float(v.x), __uint_as_float(v.y));
        fma_f32x2(acc[2], acc[3], p, p, __uint_as_float(v.z), __uint_as_float(v.w));
    }
    static __device__ __forceinline__ float narrow(float x) { return x; }
    static __device__ __forceinline__ uint4 pack(const float *a, float scale)
    {
        return make_uint4(__float_as_uint(a[0] * scale), __float_as_uint(a[1] * scale), __float_as_uint(a[2] * scale),
                          __float_as_uint(a[3] * scale));
    }
    // Stored form of 16 loaded bytes of an input row (unchanged), and of
    // vector `vec` of an input row.
    static __device__ __forceinline__ Vec from_raw(const uint4 &x, float) { return x; }
    static __device__ __forceinline__ Vec load_kv(const IO *row, int vec, float)
    {
        return __ldg(reinterpret_cast<const Vec *>(row) + vec);
    }
};

template <>
struct Elem<__nv_bfloat16> {
    using IO = __nv_bfloat16;
    using Vec = uint4;
    static constexpr bool SCALED = false;
    static constexpr int VEC = 8;
    struct Q { uint4 raw; };  // q stays packed bf16: the dot uses mixed-precision FMAs
    static __device__ __forceinline__ Q load_q(const uint4 &v) { return Q{v}; }
    // bf16 x bf16 products accumulate in fp32 (exact products, fp32 sums).
    static __device__ __forceinline__ void dot(const Q &q, const uint4 &k, float &s0, float &s1)
    {
        asm("{\n\t.reg .b16 k0, k1, k2, k3, k4, k5, k6, k7, q0, q1, q2, q3, q4, q5, q6, q7;\n\t"
            "mov.b32 {k0, k1}, %2;\n\tmov.b32 {k2, k3}, %3;\n\tmov.b32 {k4, k5}, %4;\n\tmov.b32 {k6, k7}, %5;\n\t"
            "mov.b32 {q0, q1}, %6;\n\tmov.b32 {q2, q3}, %7;\n\tmov.b32 {q4, q5}, %8;\n\tmov.b32 {q6, q7}, %9;\n\t"
            "fma.rn.f32.bf16 %0, k0, q0, %0;\n\tfma.rn.f32.bf16 %1, k1, q1, %1;\n\t"
            "fma.rn.f32.bf16 %0, k2, q2, %0;\n\tfma.rn.f32.bf16 %1, k3, q3, %1;\n\t"
            "fma.rn.f32.bf16 %0, k4, q4, %0;\n\tfma.rn.f32.bf16 %1, k5, q5, %1;\n\t"
            "fma.rn.f32.bf16 %0, k6, q6, %0;\n\tfma.rn.f32.bf16 %1, k7, q7, %1;\n\t}"
            : "+f"(s0), "+f"(s1)
            : "r"(k.x), "r"(k.y), "r"(k.z), "r"(k.w), "r"(q.raw.x), "r"(q.raw.y), "r"(q.raw.z), "r"(q.raw.w));
    }
    static __device__ __forceinline__ void axpy(float p, const uint4 &v, float *acc)
    {
        fma_f32x2(acc[0], acc[1], p, p, __uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
        fma_f32x2(acc[2], acc[3], p, p, __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
        fma_f32x2(acc[4], acc[5], p, p, __uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u));
        fma_f32x2(acc[6], acc[7], p, p, __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
    }
    static __device__ __forceinline__ __nv_bfloat16 narrow(float x) { return __float2bfloat16_rn(x); }
    static __device__ __forceinline__ uint4 pack(const float *a, float scale)
    {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(a[2 * i] * scale, a[2 * i + 1] * scale);
            w[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    static __device__ __forceinline__ Vec from_raw(const uint4 &x, float) { return x; }
    static __device__ __forceinline__ Vec load_kv(const IO *row, int vec, float)
    {
        return __ldg(reinterpret_cast<const Vec *>(row) + vec);
    }
};

// FP8 E4M3 storage of K and V with one scale per stream for each; q, k_new,
// v_new, the prompt K / V and out are bf16.  A stored code is the E4M3 value
// nearest to fp32(x) * fp32(1 / scale) (satfinite); its value is code *
// scale.  The kernel keeps the scales out of the inner loops: logits are
// q . code (times the K scale, applied once per logit with the softmax
// scale) and P.V accumulates p * code (times the V scale at the end).
// q is rounded to f16 once per item (exact: every bf16 value in the f16
// range is an f16 value), each pair of codes widens exactly to an f16 pair
// with one conversion instruction (every E4M3 value is an f16 value), and
// products accumulate in fp32 (mixed-precision FMA: f16 x f16 products are
// exact in fp32).  Stored codes are finite (satfinite), so no NaN code is
// ever widened.
__device__ __forceinline__ uint32_t f16x2_bits(__half2 h) { return *reinterpret_cast<const uint32_t *>(&h); }

// The four E4M3 codes of w as two f16 pairs: codes 0, 1 in lo and 2, 3 in
// hi (the lower code in the low half of each).  The word is split into its
// 16-bit halves as operands of the two conversions (no shift).
__device__ __forceinline__ void e4m3x4_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// acc0 += lo(a) * lo(b), acc1 += hi(a) * hi(b) for f16x2 a, b in fp32.
__device__ __forceinline__ void fma2_f16_f32(float &acc0, float &acc1, uint32_t a, uint32_t b)
{
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\tfma.rn.f32.f16 %1, a1, b1, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(a), "r"(b));
}

// E4M3 codes of 8 bf16 elements (x holds them as pairs, element 0 in the low
// half of x.x): each is the code nearest to fp32(element) * inv, satfinite.
__device__ __forceinline__ uint2 e4m3_codes(const uint4 &x, float inv)
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = make_float2(__uint_as_float(w[i] << 16) * inv, __uint_as_float(w[i] & 0xffff0000u) * inv);
        c[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
    }
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

template <>
struct Elem<__nv_fp8_e4m3> {
    using IO = __nv_bfloat16;
    using Vec = uint2;                  // 8 codes
    static constexpr bool SCALED = true;
    static constexpr int VEC = 8;
    struct Q { uint32_t h[4]; };          // 8 q elements as f16 pairs (0, 1), (2, 3), (4, 5), (6, 7)
    static __device__ __forceinline__ Q load_q(const uint4 &v)  // 8 bf16
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        Q q;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            q.h[i] = f16x2_bits(__floats2half2_rn(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u)));
        return q;
    }
    // q . code (partial sums)
    static __device__ __forceinline__ void dot(const Q &q, const uint2 &k, float &s0, float &s1)
    {
        uint32_t c01, c23, c45, c67;
        e4m3x4_f16x4(k.x, c01, c23);
        e4m3x4_f16x4(k.y, c45, c67);
        fma2_f16_f32(s0, s1, c01, q.h[0]);
        fma2_f16_f32(s0, s1, c23, q.h[1]);
        fma2_f16_f32(s0, s1, c45, q.h[2]);
        fma2_f16_f32(s0, s1, c67, q.h[3]);
    }
    // acc[0..7] += p * code (p rounded to f16, products in fp32)
    static __device__ __forceinline__ void axpy(float p, const uint2 &v, float *acc)
    {
        const uint32_t pp = f16x2_bits(__float2half2_rn(p));
        uint32_t c01, c23, c45, c67;
        e4m3x4_f16x4(v.x, c01, c23);
        e4m3x4_f16x4(v.y, c45, c67);
        fma2_f16_f32(acc[0], acc[1], c01, pp);
        fma2_f16_f32(acc[2], acc[3], c23, pp);
        fma2_f16_f32(acc[4], acc[5], c45, pp);
        fma2_f16_f32(acc[6], acc[7], c67, pp);
    }
    static __device__ __forceinline__ __nv_bfloat16 narrow(float x) { return __float2bfloat16_rn(x); }
    static __device__ __forceinline__ uint4 pack(const float *a, float scale)
    {
        return Elem<__nv_bfloat16>::pack(a, scale);
    }
    // Codes of the 8 bf16 elements of vector `vec` of an input row.
    static __device__ __forceinline__ Vec from_raw(const uint4 &x, float inv) { return e4m3_codes(x, inv); }
    static __device__ __forceinline__ Vec load_kv(const IO *row, int vec, float inv)
    {
        return e4m3_codes(__ldg(reinterpret_cast<const uint4 *>(row) + vec), inv);
    }
};

// Stage shapes (compile-time): warps per CTA, the size of a shared-memory
// stage and the decode rows one work item may list.  With two stages per
// warp, shape 0 (8 KB stages, 512-row items, three CTAs of 4 warps per SM)
// keeps the most bytes in flight per warp and shape 1 (6 KB stages, 256-row
// items, four CTAs per SM) has a third more warps, so more streams (or
// pieces of streams) run in one round; both hold about the same bytes in
// flight per SM.  The number of stages per warp (2 or 3; three leave two
// CTAs per SM) is a launch parameter; the host picks shape and stage count
// per launch.
#ifndef DSA_WARPS
#define DSA_WARPS 4
#endif

constexpr int kPipes = 2;      // stage shapes
constexpr int kMaskRegs = 8;   // mask words (or stored-list pairs) per lane kept in registers
// Longest slice of the stored offset list one item may read, counted from
// its first rank rounded down to even: 32 lanes x kMaskRegs pairs.
constexpr int kListSliceMax = 2 * 32 * kMaskRegs;
constexpr int kMaxNbuf = 3;    // stages per warp: 2 or 3, per launch (DecodeParams::nbuf)
// Launch pipelines: shape pi & 1 with 2 + (pi >> 1) stages per warp.
constexpr int kPipelines = kPipes * (kMaxNbuf - 1);

template <int SH>
struct Pipe;
template <>
struct Pipe<0> {
    static constexpr int STAGE_BYTES = 8192;
    static constexpr int CHUNK_MAX = 512;
};
template <>
struct Pipe<1> {
    static constexpr int STAGE_BYTES = 6144;
    static constexpr int CHUNK_MAX = 256;
};

template <typename T, int D, int SH>
struct KCfg {
    static constexpr int E = sizeof(T);        // bytes of a stored element
    static constexpr int VEC = Elem<T>::VEC;   // elements per stored vector (16 bytes; 8 for FP8)
    static constexpr int LPR = D / (2 * VEC);  // lanes per row: each lane reads 2 vectors of K and of V
    static constexpr int RPW = 32 / LPR;       // rows per warp instruction
    static constexpr int KROW = D * E;         // bytes of a K (or V) row
    static constexpr int ROW = 2 * KROW;       // bytes of a K|V entry
    static constexpr int WARPS = DSA_WARPS;
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int STAGE_BYTES = Pipe<SH>::STAGE_BYTES;
    static constexpr int SROWS = STAGE_BYTES / ROW;  // entries per stage
    static constexpr int NIT = SROWS / RPW;          // warp instructions per stage
    static constexpr int CHUNK_MAX = Pipe<SH>::CHUNK_MAX;  // decode ranks per work item
    static constexpr int MAXW = kMaskRegs;           // mask words per lane kept in registers
    // Shared memory of one warp with nbuf stages: the stages, their barriers
    // (room for kMaxNbuf) and the two item lists; 128-byte aligned.
    static constexpr __host__ __device__ int off_bar(int nbuf) { return nbuf * STAGE_BYTES; }
    static constexpr __host__ __device__ int off_list(int nbuf) { return off_bar(nbuf) + kMaxNbuf * 8; }
    static constexpr __host__ __device__ int warp_smem(int nbuf) { return (off_list(nbuf) + 2 * CHUNK_MAX * 2 + 127) / 128 * 128; }
    static constexpr __host__ __device__ int smem(int nbuf) { return WARPS * warp_smem(nbuf); }
    // CTA merge (DecodeParams::cta_merge), after the warps' areas: two
    // barriers per stream group (pieces done, pieces read) and one slot per
    // warp for its piece (acc[D], m, l, min logit, min offset).
    static constexpr int XSLOT = D + 4;  // floats
    static constexpr __host__ __device__ int xm_bytes() { return 32 + WARPS * XSLOT * 4; }
    static_assert(LPR >= 2 && LPR <= 16 && 32 % LPR == 0, "row must span a power-of-two lane group");
    static_assert(SROWS % RPW == 0 && NIT >= 1, "stage rows must fill whole warp instructions");
    static_assert(ROW % 128 == 0 || ROW == 256, "gather destinations must stay 128-byte aligned");
    static_assert(STAGE_BYTES % 128 == 0 && CHUNK_MAX <= 65536, "stage buffers stay 128-byte aligned");
};

// Bits of mask word w that are attended window offsets (clear and < wlen);
// w must satisfy 32 * w < wlen.
__device__ __forceinline__ uint32_t attended_bits(uint32_t word, int w, int wlen)
{
    const int base = w * 32;
    const uint32_t valid = (base + 32 <= wlen) ? 0xffffffffu : ((1u << (wlen - base)) - 1u);
    return ~word & valid;
}

__device__ __forceinline__ bool better(float v, int r, float bv, int br)
{
    return v < bv || (v == bv && r > br);  // lower logit; on a tie the older entry (larger r)
}

// Warp-per-item decode kernel: a persistent grid whose warps take work items
// (stream, split) in turn.  A warp lists the item's attended offsets (warp
// scan over the stream's mask words, prefetched one item ahead), streams the
// prompt rows (bulk copies) and the attended ring rows (TMA tile::gather4
// through `tmap`, or contiguous bulk runs when nothing can be skipped)
// through its own nbuf shared-memory stages (stage shape SH), reads q and the current token
// straight into registers, and ends with a warp-shuffle combine.
template <typename T, int D, int SH>
__global__ void __launch_bounds__(KCfg<T, D, SH>::THREADS, SH == 0 ? 3 : 4) decode_kernel(const DecodeParams p,
                                                                          const __grid_constant__ CUtensorMap tmap)
{
    using C = KCfg<T, D, SH>;
    using EL = Elem<T>;
    using IO = typename EL::IO;
    using Vec = typename EL::Vec;
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nbuf = p.nbuf;
    unsigned char *ws = smem + warp * C::warp_smem(nbuf);
    uint64_t *bars = reinterpret_cast<uint64_t *>(ws + C::off_bar(nbuf));
    uint16_t *list = reinterpret_cast<uint16_t *>(ws + C::off_list(nbuf));
    if (lane == 0) {
        for (int b = 0; b < nbuf; ++b) mbar_init(smem_u32(&bars[b]), 1);
        fence_barrier_init();
    }
    __syncwarp();
    // CTA merge: the pieces of a stream are warps [nsplit k, nsplit k + nsplit)
    // of the CTA (items are dealt to the grid's warps in order and nsplit
    // divides the CTA's warps); group k's barriers: pieces 1.. written (every
    // lane of those warps arrives), piece 0 done reading (its every lane).
    unsigned char *const xm = smem + C::smem(nbuf);
    if (p.cta_merge) {
        if (threadIdx.x == 0) {
            for (int k = 0; k < C::WARPS / p.nsplit; ++k) {
                mbar_init(smem_u32(xm) + 16 * k, 32 * (p.nsplit - 1));
                mbar_init(smem_u32(xm) + 16 * k + 8, 32);
            }
            fence_barrier_init();
        }
        __syncthreads();
    }
    const uint32_t bar0 = smem_u32(&bars[0]);
    const uint32_t buf0 = smem_u32(ws);

    const int g = lane / C::LPR;   // row group of the lane within a warp instruction
    const int cl = lane % C::LPR;  // the lane handles vectors cl and cl + LPR of every row
    const uint64_t pol = policy_evict_first();
    const int nwords = p.noskip ? 0 : (p.wlen + 31) >> 5;
    const int wpl = (nwords + 31) >> 5;  // contiguous mask words per lane
    const bool inreg = wpl <= C::MAXW;
    const int GW = gridDim.x * C::WARPS;
    const int first_item = blockIdx.x * C::WARPS + warp;

    // The next item's mask words or, when the list is read (list_mode 2),
    // its slice of the stored list as pairs of offsets: word i of a lane
    // holds entries (klo & ~1) + 2 (lane + 32 i) + {0, 1} (the host keeps
    // every slice within 2 * 32 * MAXW entries).
    uint32_t words[C::MAXW];
    uint32_t w0n = 0;  // list_mode 2: the next item's mask word 0 (bit 0: its current token is skipped)
    auto load_words = [&](int item) {
        const int s = item / p.nsplit;
        if (p.list_mode == 2) {
            const int lo = (item - s * p.nsplit) * p.chunk;
            const int klo = max(lo, p.P) - p.P;
            const int khi = max(min(lo + p.chunk, p.n), p.P) - p.P;
            const uint32_t *src = reinterpret_cast<const uint32_t *>(p.glist + (size_t)s * p.LS);
            const int e0 = klo & ~1;
#pragma unroll
            for (int i = 0; i < C::MAXW; ++i) {
                const int e = e0 + 2 * (lane + 32 * i);
                words[i] = e < khi ? __ldcg(src + (e >> 1)) : 0u;
            }
            w0n = __ldcg(p.mask + (size_t)s * p.MW);
            return;
        }
        const uint32_t *row = p.mask + (size_t)s * p.MW;
#pragma unroll
        for (int i = 0; i < C::MAXW; ++i) {
            const int w = lane * wpl + i;
            words[i] = (i < wpl && w < nwords) ? __ldcg(row + w) : 0u;
        }
    };
    uint4 qn0 = make_uint4(0, 0, 0, 0), qn1 = qn0;  // q vectors of the next item
    auto load_q = [&](int item) {
        const uint4 *qr = reinterpret_cast<const uint4 *>(reinterpret_cast<const IO *>(p.q) + (size_t)(item / p.nsplit) * D);
        qn0 = __ldg(qr + cl);
        qn1 = __ldg(qr + cl + C::LPR);
    };
    // Programmatic dependent launch.  Before the grid dependency wait this
    // grid only reads its own state (mask, prompt prefix, ring), and only when
    // the previous grid in the stream is not a step of the same state
    // (p.early); q, k_new, v_new and every write come after the wait.  Each
    // CTA lets the next grid start only after its own wait, so the next
    // grid's early reads happen after the grid before this one completed.
    if (!p.early) {
        pdl_wait();
        pdl_launch_dependents();
    }
    // Graph mode: the step comes from device memory (advanced by the last CTA
    // of the previous launch of this state, which has completed here).
    const int tin_mod = p.step_dev ? (__ldcg(p.step_dev) - p.sink) % p.R : p.tin_mod;
    const bool prefetch = p.list_mode == 2 || (inreg && nwords > 0);  // load_words serves the listing
    if (first_item < p.nitems && prefetch) load_words(first_item);

    bool aborted = false;
    int issued = 0, consumed = 0;  // stages issued / consumed by this warp over all its items
    int ib = 0;                    // buffer of the next issued stage
    int cb = 0, cpar = 0;          // buffer and phase parity of the next consumed stage

    // ---- issuer: a cursor over the stages of this warp's items.  Each freed
    // buffer is refilled at once, with a stage of the next item once the
    // current item is fully issued, so the warp's copies stay in flight
    // across item boundaries.  Items are numbered by seq (0, 1, ... for
    // this warp); item seq's offsets are listed in list buffer seq & 1, so
    // the issuer may run at most one item ahead of the consumer.
    // An item's prompt-only stages need no offsets: they are issued first
    // (iss_state 1), and the offsets are listed (iss_state 2) when the first
    // stage with ring rows is due or the consumer reaches the item, so the
    // listing overlaps the first copies.
    int iss_item = first_item, iss_seq = 0, iss_j = 0;
    int iss_state = 0;  // 0: not set up; 1: prompt stages may be issued; 2: offsets listed
    int I_s = 0, I_lo = 0, I_npre = 0, I_kr0 = 0, I_klo = 0, I_khi = 0, I_nrows = 0, I_nst = 0;
    uint32_t self_skip_bits = 0;  // bit (seq & 1): the item's current token is itself skipped

    auto setup_basic = [&]() {
        const int s = iss_item / p.nsplit;
        const int lo = (iss_item - s * p.nsplit) * p.chunk;
        const int hi = min(lo + p.chunk, p.n);
        I_s = s;
        I_lo = lo;
        I_klo = max(lo, p.P) - p.P;
        I_khi = max(hi, p.P) - p.P;
        I_npre = max(min(hi, p.P) - lo, 0);
        I_nrows = I_npre;  // until the offsets are listed
        iss_state = 1;
    };

    // a4: list the attended offsets of ranks [klo, khi) of the issuer's item
    auto setup_list = [&]() {
        const int item = iss_item;
        const int s = I_s;
        const int klo = I_klo;
        const int khi = I_khi;
        uint16_t *lst = list + (iss_seq & 1) * C::CHUNK_MAX;
        const uint32_t *mrow = p.mask + (size_t)s * p.MW;
        bool self_skip = false;
        if (p.list_mode == 2) {
            // the stored list: entries e of the prefetched pairs within [klo, khi)
            const int e0 = klo & ~1;
#pragma unroll
            for (int i = 0; i < C::MAXW; ++i) {
                const int e = e0 + 2 * (lane + 32 * i);
                if (e >= klo && e < khi) lst[e - klo] = (uint16_t)(words[i] & 0xffffu);
                if (e + 1 >= klo && e + 1 < khi) lst[e + 1 - klo] = (uint16_t)(words[i] >> 16);
            }
            self_skip = (w0n & 1u) != 0;
            if (item + GW < p.nitems) load_words(item + GW);  // prefetch for the next item
        } else if (nwords > 0) {
            int mine = 0;
            if (inreg) {
#pragma unroll
                for (int i = 0; i < C::MAXW; ++i) {
                    const int w = lane * wpl + i;
                    if (i < wpl && w < nwords) mine += __popc(attended_bits(words[i], w, p.wlen));
                }
            } else {
                for (int i = 0; i < wpl; ++i) {
                    const int w = lane * wpl + i;
                    if (w < nwords) mine += __popc(attended_bits(__ldcg(mrow + w), w, p.wlen));
                }
            }
            int incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int total = __shfl_sync(0xffffffffu, incl, 31);
            if (total != p.a) {
                // The skip mask disagrees with the host's count: record it and
                // keep every listed offset in range.
                if (lane == 0) atomicOr(p.status, ST_CHECK);
                for (int i = lane; i < khi - klo; i += 32) lst[i] = 0;
                __syncwarp();
            }
            int rank = incl - mine;
            for (int i = 0; i < wpl && rank < khi; ++i) {
                const int w = lane * wpl + i;
                if (w >= nwords) break;
                uint32_t word;
                if (inreg) {
                    word = 0;
#pragma unroll
                    for (int k = 0; k < C::MAXW; ++k) word = (k == i) ? words[k] : word;
                } else {
                    word = __ldcg(mrow + w);
                }
                uint32_t bits = attended_bits(word, w, p.wlen);
                const int cnt = __popc(bits);
                if (rank + cnt <= klo) {
                    rank += cnt;
                    continue;
                }
                while (bits) {
                    const int bt = __ffs(bits) - 1;
                    if (rank >= klo && rank < khi) lst[rank - klo] = (uint16_t)(w * 32 + bt);
                    ++rank;
                    bits &= bits - 1;
                }
            }
            const uint32_t w0 = inreg ? words[0] : __ldcg(mrow);
            self_skip = (__shfl_sync(0xffffffffu, w0, 0) & 1u) != 0;
            if (inreg && item + GW < p.nitems) load_words(item + GW);  // prefetch for the next item
        }
        __syncwarp();
        const bool has_cur = (klo == 0 && khi > 0 && !self_skip);
        self_skip_bits = (self_skip_bits & ~(1u << (iss_seq & 1))) | ((self_skip ? 1u : 0u) << (iss_seq & 1));
        I_kr0 = has_cur ? klo + 1 : klo;
        I_nrows = I_npre + max(khi - I_kr0, 0);
        I_nst = (I_nrows + C::SROWS - 1) / C::SROWS;
        iss_state = 2;
    };

    // a5: issue stage iss_j of the issuer's item into buffer ib (= issued mod nbuf)
    auto issue_stage = [&]() {
        const int b = ib;
        ib = ib + 1 == nbuf ? 0 : ib + 1;
        const uint32_t fb = bar0 + 8 * b;
        const uint32_t dst = buf0 + b * C::STAGE_BYTES;
        const int u0 = iss_j * C::SROWS;
        const int u1 = min(u0 + C::SROWS, I_nrows);
        const unsigned char *pre = reinterpret_cast<const unsigned char *>(p.prefix) + ((size_t)I_s * p.Lcap + I_lo) * C::ROW;
        const unsigned char *rng = reinterpret_cast<const unsigned char *>(p.ring) + (size_t)I_s * p.R * C::ROW;
        if (lane == 0) {
            fence_proxy_async_smem();  // this warp's reads of the buffer precede the new fill
            mbar_arrive_expect_tx(fb, (uint32_t)(u1 - u0) * C::ROW);
            const int pb = min(u1, I_npre);
            if (pb > u0) bulk_g2s_hint(dst, pre + (size_t)u0 * C::ROW, (pb - u0) * C::ROW, fb, pol);
        }
        const int ua = max(u0, I_npre);
        const int nr = u1 - ua;  // ring entries of the stage
        if (nr > 0) {
            const int k0 = I_kr0 + (ua - I_npre);
            const uint32_t rd = dst + (ua - u0) * C::ROW;
            if (p.noskip) {
                // offset r = rank: descending slots, at most two contiguous runs
                if (lane == 0) {
                    const int kA = min(k0 + nr, tin_mod + 1);
                    const int nA = max(kA - k0, 0);
                    if (nA > 0) bulk_g2s_hint(rd, rng + (size_t)(tin_mod - (kA - 1)) * C::ROW, nA * C::ROW, fb, pol);
                    if (nr > nA)
                        bulk_g2s_hint(rd + nA * C::ROW, rng + (size_t)(tin_mod - (k0 + nr - 1) + p.R) * C::ROW,
                                      (nr - nA) * C::ROW, fb, pol);
                }
            } else {
                const uint16_t *lst = list + (iss_seq & 1) * C::CHUNK_MAX;
                const int ybase = I_s * p.R;
                const int ngrp = nr >> 2;
                for (int g4 = lane; g4 < ngrp; g4 += 32) {
                    const int k = k0 + 4 * g4 - I_klo;
                    int y[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int sl = tin_mod - (int)lst[k + m];
                        y[m] = ybase + (sl < 0 ? sl + p.R : sl);
                    }
                    tma_gather4(rd + 4 * g4 * C::ROW, &tmap, 0, y[0], y[1], y[2], y[3], fb);
                }
                const int tail = nr - 4 * ngrp;
                if (lane < tail) {
                    int sl = tin_mod - (int)lst[k0 + 4 * ngrp + lane - I_klo];
                    sl = sl < 0 ? sl + p.R : sl;
                    bulk_g2s_hint(rd + (4 * ngrp + lane) * C::ROW, rng + (size_t)sl * C::ROW, C::ROW, fb, pol);
                }
            }
        }
        ++issued;
        ++iss_j;
    };

    // Issues the next stage in the warp's stream, if any (at most one item
    // ahead of the consumer's item con_seq).
    auto issue_next = [&](int con_seq) {
        while (iss_item < p.nitems) {
            if (iss_state == 0) {
                if (iss_seq > con_seq + 1) return;
                setup_basic();
            }
            if (iss_state == 1 && (iss_j + 1) * C::SROWS > I_npre) setup_list();  // the stage needs offsets
            if (iss_state == 1 || iss_j < I_nst) {
                issue_stage();
                return;
            }
            iss_item += GW;
            ++iss_seq;
            iss_j = 0;
            iss_state = 0;
        }
    };

    // Keeps nbuf stages of the warp's stream in flight (fewer at its end).
    auto top_up = [&](int con_seq) {
        while (issued - consumed < nbuf) {
            const int before = issued;
            issue_next(con_seq);
            if (issued == before) return;
        }
    };
    top_up(0);
    if (p.early) {
        pdl_wait();
        pdl_launch_dependents();
    }
    if (first_item < p.nitems) load_q(first_item);

    // ---- consumer: the items in order
    int con_seq = 0;
    for (int item = first_item; item < p.nitems; item += GW, ++con_seq) {
        // The issuer set up every earlier item; bring it to this one if items
        // without staged rows left it behind, and list this item if needed.
        while (iss_seq < con_seq) {
            iss_item += GW;
            ++iss_seq;
            iss_j = 0;
            iss_state = 0;
        }
        if (iss_seq == con_seq && iss_state < 2) {
            if (iss_state == 0) setup_basic();
            setup_list();
        }
        top_up(con_seq);
        const int s = item / p.nsplit;
        const int c = item - s * p.nsplit;
        const int lo = c * p.chunk;
        const int hi = min(lo + p.chunk, p.n);
        const int klo = max(lo, p.P) - p.P;
        const int khi = max(hi, p.P) - p.P;
        const bool self_skip = (self_skip_bits >> (con_seq & 1)) & 1u;
        const uint16_t *lst = list + (con_seq & 1) * C::CHUNK_MAX;
        if (p.list_mode == 1) {  // the last step before the steady state: store the list
            uint16_t *dst = p.glist + (size_t)s * p.LS + klo;
            for (int i = lane; i < khi - klo; i += 32) dst[i] = lst[i];
        }
        // rank 0 is the current token (offset 0) unless it is itself skipped
        const bool has_cur = (klo == 0 && khi > 0 && !self_skip);
        T *const cur_dst = p.sinkmode ? reinterpret_cast<T *>(p.prefix) + ((size_t)s * p.Lcap + p.P) * 2 * D
                                      : reinterpret_cast<T *>(p.ring) + ((size_t)s * p.R + tin_mod) * 2 * D;
        // FP8 storage: per-stream scales (1 otherwise)
        const float kinv = EL::SCALED ? __ldg(p.kinv + s) : 1.f;
        const float vinv = EL::SCALED ? __ldg(p.vinv + s) : 1.f;
        const float xs = EL::SCALED ? p.qscale * __ldg(p.kscale + s) : p.qscale;
        const IO *kio = reinterpret_cast<const IO *>(p.knew) + (size_t)s * D;
        const IO *vio = reinterpret_cast<const IO *>(p.vnew) + (size_t)s * D;
        // The current token goes straight to registers: its k_new / v_new
        // vectors (or, already stored in its slot by the fused step, its
        // stored vectors) are loaded here and turned into the stored form
        // after the stage loop, so the loads overlap the wait for q and the
        // stages.
        uint4 kn0 = make_uint4(0, 0, 0, 0), kn1 = kn0, vn0 = kn0, vn1 = kn0;
        if (has_cur && p.appended) {
            const Vec *cur = reinterpret_cast<const Vec *>(cur_dst);
            kn0 = to_u4(cur[cl]);
            kn1 = to_u4(cur[cl + C::LPR]);
            vn0 = to_u4(cur[2 * C::LPR + cl]);
            vn1 = to_u4(cur[3 * C::LPR + cl]);
        } else if (has_cur) {
            const uint4 *k4 = reinterpret_cast<const uint4 *>(kio), *v4 = reinterpret_cast<const uint4 *>(vio);
            kn0 = __ldg(k4 + cl);
            kn1 = __ldg(k4 + cl + C::LPR);
            vn0 = __ldg(v4 + cl);
            vn1 = __ldg(v4 + cl + C::LPR);
        } else if (self_skip && c == 0 && !p.appended) {
            // a2 for a token that is not attended: it is in no stage; store it.
            constexpr int NV = D / C::VEC;
            Vec *dst = reinterpret_cast<Vec *>(cur_dst);
            for (int i = lane; i < 2 * NV; i += 32)
                dst[i] = (i < NV) ? EL::load_kv(kio, i, kinv) : EL::load_kv(vio, i - NV, vinv);
        }
        const typename EL::Q q0 = EL::load_q(qn0), q1 = EL::load_q(qn1);
        if (item + GW < p.nitems) load_q(item + GW);  // prefetch the next item's q
        const int npre = max(min(hi, p.P) - lo, 0);
        const int kr0 = has_cur ? klo + 1 : klo;
        const int nrows = npre + max(khi - kr0, 0);
        const int nst = (nrows + C::SROWS - 1) / C::SROWS;

        float acc[2 * C::VEC];
#pragma unroll
        for (int e = 0; e < 2 * C::VEC; ++e) acc[e] = 0.f;
        float m = -INFINITY, l = 0.f, minv = INFINITY;
        int minr = -1;

        for (int j = 0; j < nst; ++j) {
            const int b = cb;
            const bool ok = wait_phase(bar0 + 8 * b, (uint32_t)cpar, p.wait_limit);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) atomicOr(p.status, ST_TIMEOUT);
                aborted = true;
                break;
            }
            ++consumed;
            if (++cb == nbuf) {
                cb = 0;
                cpar ^= 1;
            }
            const unsigned char *st = ws + b * C::STAGE_BYTES;
            const int u0 = j * C::SROWS;
            const int nv = min(C::SROWS, nrows - u0);  // valid rows of the stage (>= 1)
            // Rows past nv (only in an item's last stage) read row 0 of the
            // stage instead, so every row read holds loaded data; their logit
            // is -inf and their softmax weight 0.  No branch per row.
            float sc[C::NIT];
#pragma unroll
            for (int it = 0; it < C::NIT; ++it) {
                const int row = it * C::RPW + g;
                const bool valid = row < nv;
                const Vec *kr = reinterpret_cast<const Vec *>(st + (valid ? row : 0) * C::ROW);
                float s0 = 0.f, s1 = 0.f;
                EL::dot(q0, kr[cl], s0, s1);
                EL::dot(q1, kr[cl + C::LPR], s0, s1);
                float x = s0 + s1;
#pragma unroll
                for (int o = C::LPR / 2; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                sc[it] = valid ? x * xs : -INFINITY;
            }
            if (p.select) {  // a8: argmin over the stage's attended decode rows
#pragma unroll
                for (int it = 0; it < C::NIT; ++it) {
                    const int row = it * C::RPW + g;
                    if (row < nv && u0 + row >= npre) {
                        const int r = lst[kr0 + (u0 + row - npre) - klo];
                        if (better(sc[it], r, minv, minr)) {
                            minv = sc[it];
                            minr = r;
                        }
                    }
                }
            }
            float mx = sc[0];
#pragma unroll
            for (int it = 1; it < C::NIT; ++it) mx = fmaxf(mx, sc[it]);
#pragma unroll
            for (int o = C::LPR; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (mx > m) {  // warp-uniform; rescale only when the running max grows
                const float alpha = ex2(m - mx);
                l *= alpha;
#pragma unroll
                for (int e = 0; e < 2 * C::VEC; ++e) acc[e] *= alpha;
                m = mx;
            }
#pragma unroll
            for (int it = 0; it < C::NIT; ++it) {
                const int row = it * C::RPW + g;
                const float pj = ex2(sc[it] - m);  // 0 for rows past nv
                l += pj;
                const Vec *vr = reinterpret_cast<const Vec *>(st + (row < nv ? row : 0) * C::ROW + C::KROW);
                EL::axpy(pj, vr[cl], acc);
                EL::axpy(pj, vr[cl + C::LPR], acc + C::VEC);
            }
            __syncwarp();
            top_up(con_seq);  // refill the freed buffer
        }
        if (aborted) break;

        // ---- the current token (a2 append, logit, softmax.V), from registers
        if (has_cur) {
            Vec kc0, kc1, vc0, vc1;
            if (p.appended) {
                kc0 = from_u4<Vec>(kn0);
                kc1 = from_u4<Vec>(kn1);
                vc0 = from_u4<Vec>(vn0);
                vc1 = from_u4<Vec>(vn1);
            } else {
                kc0 = EL::from_raw(kn0, kinv);
                kc1 = EL::from_raw(kn1, kinv);
                vc0 = EL::from_raw(vn0, vinv);
                vc1 = EL::from_raw(vn1, vinv);
            }
            float s0 = 0.f, s1 = 0.f;
            EL::dot(q0, kc0, s0, s1);
            EL::dot(q1, kc1, s0, s1);
            float x = s0 + s1;
#pragma unroll
            for (int o = C::LPR / 2; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            x *= xs;  // identical in every row group
            if (p.select && better(x, 0, minv, minr)) {
                minv = x;
                minr = 0;
            }
            if (x > m) {
                const float alpha = ex2(m - x);
                l *= alpha;
#pragma unroll
                for (int e = 0; e < 2 * C::VEC; ++e) acc[e] *= alpha;
                m = x;
            }
            if (g == 0) {
                const float pj = ex2(x - m);
                l += pj;
                EL::axpy(pj, vc0, acc);
                EL::axpy(pj, vc1, acc + C::VEC);
                if (!p.appended) {
                    Vec *dst = reinterpret_cast<Vec *>(cur_dst);
                    dst[cl] = kc0;
                    dst[cl + C::LPR] = kc1;
                    dst[2 * C::LPR + cl] = vc0;
                    dst[3 * C::LPR + cl] = vc1;
                }
            }
        }

        // ---- a6: combine the row groups of the warp (shuffles)
#pragma unroll
        for (int o = C::LPR; o < 32; o <<= 1) {
            l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
            for (int e = 0; e < 2 * C::VEC; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
            const float ov = __shfl_xor_sync(0xffffffffu, minv, o);
            const int orr = __shfl_xor_sync(0xffffffffu, minr, o);
            if (better(ov, orr, minv, minr)) {
                minv = ov;
                minr = orr;
            }
        }
        if (p.nsplit == 1) {
            if (g == 0) {
                const float inv = (EL::SCALED ? __ldg(p.vscale + s) : 1.f) / l;
                uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<IO *>(p.out) + (size_t)s * D);
                o[cl] = EL::pack(acc, inv);
                o[cl + C::LPR] = EL::pack(acc + C::VEC, inv);
            }
            if (lane == 0 && p.select && minr >= 0) {
                p.last_sel[s] = minr;
                p.mask[(size_t)s * p.MW + (minr >> 5)] |= 1u << (minr & 31);
            }
        } else if (p.cta_merge) {
            // ---- a7 inside the CTA: pieces 1.. leave (acc, m, l, argmin) in
            // their slots; piece 0 combines the pieces in split order with the
            // arithmetic of merge_kernel (so the two paths agree bit for bit),
            // writes out and the skip bit, and frees the slots.
            float *const xs = reinterpret_cast<float *>(xm + 32);
            const uint32_t xfull = smem_u32(xm) + 16 * (warp / p.nsplit), xfree = xfull + 8;
            const uint32_t xpar = (uint32_t)(con_seq & 1);
            bool ok;
            if (c != 0) {
                float *slot = xs + warp * C::XSLOT;
                if (g == 0) {
                    float4 *s4 = reinterpret_cast<float4 *>(slot);
#pragma unroll
                    for (int e = 0; e < C::VEC / 4; ++e) {
                        s4[cl * (C::VEC / 4) + e] = make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2], acc[4 * e + 3]);
                        s4[(cl + C::LPR) * (C::VEC / 4) + e] = make_float4(acc[C::VEC + 4 * e], acc[C::VEC + 4 * e + 1],
                                                                           acc[C::VEC + 4 * e + 2], acc[C::VEC + 4 * e + 3]);
                    }
                }
                if (lane == 0) {
                    slot[D] = m;
                    slot[D + 1] = l;
                    slot[D + 2] = minv;
                    slot[D + 3] = __int_as_float(minr);
                }
                mbar_arrive(xfull);
                ok = wait_phase(xfree, xpar, p.wait_limit);  // piece 0 has read the slot
            } else {
                ok = wait_phase(xfull, xpar, p.wait_limit);
                if (__all_sync(0xffffffffu, ok)) {
                    float Mx = m;
                    for (int i = 1; i < p.nsplit; ++i) Mx = fmaxf(Mx, xs[(warp + i) * C::XSLOT + D]);
                    float O[2 * C::VEC];
#pragma unroll
                    for (int e = 0; e < 2 * C::VEC; ++e) O[e] = 0.f;
                    float Lx = 0.f;
                    float bv = minv;
                    int br = minr;
                    for (int i = 0; i < p.nsplit; ++i) {
                        const float *sl = xs + (warp + i) * C::XSLOT;
                        const float mi = i == 0 ? m : sl[D];
                        const float li = i == 0 ? l : sl[D + 1];
                        if (mi != -INFINITY) {
                            const float f = ex2(mi - Mx);
                            Lx = fmaf(li, f, Lx);
#pragma unroll
                            for (int e = 0; e < C::VEC; ++e) {
                                O[e] = fmaf(i == 0 ? acc[e] : sl[cl * C::VEC + e], f, O[e]);
                                O[C::VEC + e] = fmaf(i == 0 ? acc[C::VEC + e] : sl[(cl + C::LPR) * C::VEC + e], f, O[C::VEC + e]);
                            }
                        }
                        if (i > 0 && better(sl[D + 2], __float_as_int(sl[D + 3]), bv, br)) {
                            bv = sl[D + 2];
                            br = __float_as_int(sl[D + 3]);
                        }
                    }
                    if (g == 0) {
                        const float inv = (EL::SCALED ? __ldg(p.vscale + s) : 1.f) / Lx;
                        uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<IO *>(p.out) + (size_t)s * D);
                        o[cl] = EL::pack(O, inv);
                        o[cl + C::LPR] = EL::pack(O + C::VEC, inv);
                    }
                    if (lane == 0 && p.select && br >= 0) {
                        p.last_sel[s] = br;
                        p.mask[(size_t)s * p.MW + (br >> 5)] |= 1u << (br & 31);
                    }
                }
                mbar_arrive(xfree);
            }
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) atomicOr(p.status, ST_TIMEOUT);
                aborted = true;
                break;
            }
        } else {
            // ---- a7: partial (m, l, acc, argmin) of this split; merge_kernel,
            // launched right after this kernel, combines the splits
            const size_t slot = (size_t)s * p.pstride + c;
            if (g == 0) {
                float4 *pa = reinterpret_cast<float4 *>(p.part_acc + slot * D);
#pragma unroll
                for (int e = 0; e < C::VEC / 4; ++e) {
                    pa[cl * (C::VEC / 4) + e] = make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2], acc[4 * e + 3]);
                    pa[(cl + C::LPR) * (C::VEC / 4) + e] =
                        make_float4(acc[C::VEC + 4 * e], acc[C::VEC + 4 * e + 1], acc[C::VEC + 4 * e + 2], acc[C::VEC + 4 * e + 3]);
                }
            }
            if (lane == 0) {
                p.part_ml[slot] = make_float2(m, l);
                p.part_min[slot] = make_float2(minv, __int_as_float(minr));
            }
        }
    }
    // A warp that gave up lets its own copies in flight land before exit.
    if (aborted && lane == 0) {
        for (int q = consumed; q < issued; ++q) drain_phase(bar0 + 8 * (q % nbuf), (q / nbuf) & 1);
    }
    __syncwarp();
    if (p.step_dev) {
        // Graph mode: the last CTA to finish advances the device step (every
        // CTA of this launch has read it by then).
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            if (atomicAdd(p.step_dev + 1, 1) == (int)gridDim.x - 1) {
                p.step_dev[1] = 0;
                atomicAdd(p.step_dev, 1);
            }
        }
    }
}

// a7: merges the per-split partials of every stream after a decode launch
// whose streams were split: out = sum_i e^(m_i - M) acc_i / sum_i e^(m_i - M) l_i,
// and on selection steps the argmin over the splits' (logit, offset) pairs
// sets the stream's skip bit.  One warp per stream.
constexpr int kMergeWarps = 4;

template <typename T, int D>
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(const DecodeParams p)
{
    using EL = Elem<T>;
    pdl_wait();  // the decode kernel's partials
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int s = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    if (s >= p.S) return;
    const size_t base = (size_t)s * p.pstride;
    float Mx = -INFINITY;
    for (int i = lane; i < p.nsplit; i += 32) Mx = fmaxf(Mx, __ldcg(&p.part_ml[base + i].x));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, o));
    constexpr int DPL = D / 32;  // output elements per lane
    float O[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) O[e] = 0.f;
    float Lx = 0.f;
    for (int i = 0; i < p.nsplit; ++i) {
        const float2 ml = __ldcg(&p.part_ml[base + i]);
        if (ml.x != -INFINITY) {
            const float f = ex2(ml.x - Mx);
            Lx = fmaf(ml.y, f, Lx);
#pragma unroll
            for (int e = 0; e < DPL; ++e) O[e] = fmaf(__ldcg(&p.part_acc[(base + i) * D + lane * DPL + e]), f, O[e]);
        }
    }
    typename EL::IO *o = reinterpret_cast<typename EL::IO *>(p.out) + (size_t)s * D + lane * DPL;
    const float inv = (EL::SCALED ? __ldg(p.vscale + s) : 1.f) / Lx;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] = EL::narrow(O[e] * inv);
    if (p.select) {
        float bv = INFINITY;
        int br = -1;
        for (int i = lane; i < p.nsplit; i += 32) {
            const float2 x = __ldcg(&p.part_min[base + i]);
            if (better(x.x, __float_as_int(x.y), bv, br)) {
                bv = x.x;
                br = __float_as_int(x.y);
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int orr = __shfl_xor_sync(0xffffffffu, br, off);
            if (better(ov, orr, bv, br)) {
                bv = ov;
                br = orr;
            }
        }
        if (lane == 0 && br >= 0 && *reinterpret_cast<volatile int *>(p.status) == 0) {
            p.last_sel[s] = br;
            p.mask[(size_t)s * p.MW + (br >> 5)] |= 1u << (br & 31);
        }
    }
}

// a1: prompt K, V [S, L_p, D] -> prefix [S, Lcap, 2, D] in the stored form
// (FP8 storage: codes with the per-stream inverse scales kinv, vinv).
template <typename T, int D>
__global__ void prefill_kernel(const typename Elem<T>::IO *__restrict__ K, const typename Elem<T>::IO *__restrict__ V,
                               T *__restrict__ prefix, const float *kinv, const float *vinv, int S, int L_p, int Lcap)
{
    using EL = Elem<T>;
    constexpr int NV = D / EL::VEC;  // stored vectors per K (or V) row
    const size_t total = (size_t)S * L_p * 2 * NV;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int vec = (int)(i % NV);
        size_t rest = i / NV;
        const int kv = (int)(rest & 1);
        rest >>= 1;
        const int row = (int)(rest % L_p);
        const size_t s = rest / L_p;
        const float inv = EL::SCALED ? __ldg((kv ? vinv : kinv) + s) : 1.f;
        typename EL::Vec *dst = reinterpret_cast<typename EL::Vec *>(prefix + ((s * Lcap + row) * 2 + kv) * D) + vec;
        *dst = EL::load_kv((kv ? V : K) + (s * L_p + row) * D, vec, inv);
    }
}

}  // namespace dsa
