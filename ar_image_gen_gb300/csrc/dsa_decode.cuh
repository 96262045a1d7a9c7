// dsa_decode.cuh -- the fused decode-step kernel of diagonal-aware sparse
// attention ("Understanding and Exploiting Diagonal Attention Sparsity in
// Autoregressive Image Generation", section 4, Algorithm 1 and Fig. 12;
// section 5.1 for Diagonal+sink4 and the fused-kernel description).
//
// One launch performs, for every stream s (a sequence-head of one layer):
//   a2  append: k_new, v_new -> ring slot t' mod R (the slot of the entry
//       evicted at this step) or, during the sink fill, prefix row L_p + t;
//   a4  index set: the attended relative offsets r in [0, min(t'+1, R)) whose
//       skip bit is clear, compacted in shared memory with a block scan;
//   a5  gather + logits: prompt rows (one contiguous bulk copy per stage)
//       and attended ring rows (one bulk copy per row) staged into a
//       4-stage shared-memory ring by a producer warp; fp32 logits q.k;
//   a6  online softmax and P.V per consumer warp, then across warps;
//   a7  split combine: the last CTA of a stream (atomic ticket) merges the
//       per-split (m, l, acc) partials;
//   a8  fused argmin over the attended decode logits on selection steps; the
//       finishing CTA sets bit r* of the stream's relative-offset skip mask.
// The diagonal shift (+1 per step) costs nothing: skipped entries are kept as
// relative offsets r = t' - position, which the shift leaves unchanged, and
// the slot of offset r is (t' - r) mod R.
#pragma once

#include <cuda_bf16.h>

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

// Polls the barrier phase at most `limit` times and for at most kWaitNs.
// limit == 0 gives up without polling (the test knob).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, uint32_t limit)
{
    if (limit == 0) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitNs) return false;
    }
    return false;
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
    int *ticket;          // [S]
    int *status;          // sticky device status bits
    int S;
    int Lcap;             // prefix rows per stream (L_p + sink)
    int P;                // prefix rows attended at this step
    int sinkmode;         // 1: the new token goes to prefix row P
    int R;                // ring slots (N_r - sink)
    int tin;              // inner step t' = t - sink (-1 in sink mode)
    int wlen;             // live window length min(t' + 1, R) (1 in sink mode)
    int a;                // attended decode rows (host count)
    int n;                // P + a
    int nsplit;           // CTAs per stream
    int chunk;            // rows per CTA (multiple of the stage rows)
    int pstride;          // partial slots per stream
    int select;           // 1: selection step (fused argmin)
    int MW;               // mask words per stream
    float qscale;         // log2(e) / sqrt(D)
    uint32_t wait_limit;
};

template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int VEC = 4;
    static __device__ __forceinline__ void widen(const uint4 &v, float *f)
    {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    static __device__ __forceinline__ float narrow(float x) { return x; }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int VEC = 8;
    static __device__ __forceinline__ void widen(const uint4 &v, float *f)
    {
        f[0] = __uint_as_float(v.x << 16);
        f[1] = __uint_as_float(v.x & 0xffff0000u);
        f[2] = __uint_as_float(v.y << 16);
        f[3] = __uint_as_float(v.y & 0xffff0000u);
        f[4] = __uint_as_float(v.z << 16);
        f[5] = __uint_as_float(v.z & 0xffff0000u);
        f[6] = __uint_as_float(v.w << 16);
        f[7] = __uint_as_float(v.w & 0xffff0000u);
    }
    static __device__ __forceinline__ __nv_bfloat16 narrow(float x) { return __float2bfloat16_rn(x); }
};

template <typename T, int D>
struct KCfg {
    static constexpr int E = sizeof(T);
    static constexpr int VEC = Elem<T>::VEC;   // elements per 16-byte vector
    static constexpr int LPR = D / VEC;        // lanes per row
    static constexpr int RPW = 32 / LPR;       // rows per warp instruction
    static constexpr int KROW = D * E;         // bytes of a K (or V) row
    static constexpr int ROW = 2 * KROW;       // bytes of a K|V entry
    static constexpr int NCW = 4;              // consumer warps
    static constexpr int THREADS = 32 * (NCW + 1);
    static constexpr int STAGE_BYTES = 16384;
    static constexpr int ROWS = STAGE_BYTES / ROW;  // entries per stage
    static constexpr int RPC = ROWS / NCW;          // entries per consumer warp per stage
    static constexpr int NIT = RPC / RPW;
    static constexpr int NSTAGE = 4;
    static constexpr int CHUNK_MAX = 2048;          // decode entries listed per CTA
    static constexpr int OFF_BAR = NSTAGE * STAGE_BYTES;
    static constexpr int OFF_LIST = OFF_BAR + 2 * NSTAGE * 8;
    static constexpr int OFF_CNT = OFF_LIST + CHUNK_MAX * 2;
    static constexpr int OFF_COMB = OFF_CNT + 32 * 4;
    static constexpr int OFF_CML = OFF_COMB + NCW * D * 4;
    static constexpr int OFF_FLAG = OFF_CML + NCW * 16;
    static constexpr int SMEM = OFF_FLAG + 16;
    static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "row must span a power-of-two lane group");
    static_assert(RPC % RPW == 0 && NIT >= 1, "stage rows must split evenly over consumer warps");
    static_assert(ROW % 16 == 0 && OFF_COMB % 16 == 0, "alignment");
};

// Bits of mask word w that are attended window offsets (clear and < wlen).
__device__ __forceinline__ uint32_t attended_bits(uint32_t word, int w, int wlen)
{
    const int base = w * 32;
    const uint32_t valid = (base + 32 <= wlen) ? 0xffffffffu : ((1u << (wlen - base)) - 1u);
    return ~word & valid;
}

template <typename T, int D>
__global__ void __launch_bounds__(KCfg<T, D>::THREADS) decode_kernel(const DecodeParams p)
{
    using C = KCfg<T, D>;
    using EL = Elem<T>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint16_t *list = reinterpret_cast<uint16_t *>(smem + C::OFF_LIST);
    int *wsum = reinterpret_cast<int *>(smem + C::OFF_CNT);
    float *comb = reinterpret_cast<float *>(smem + C::OFF_COMB);
    float4 *cml = reinterpret_cast<float4 *>(smem + C::OFF_CML);
    volatile int *flag = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int s = blockIdx.x / p.nsplit;
    const int c = blockIdx.x - s * p.nsplit;
    const int lo = c * p.chunk;
    const int hi = min(lo + p.chunk, p.n);
    const int nst = (hi - lo + C::ROWS - 1) / C::ROWS;
    const int klo = max(lo, p.P) - p.P;  // decode ranks of this CTA: [klo, khi)
    const int khi = max(hi, p.P) - p.P;

    if (tid == 0) {
        for (int b = 0; b < C::NSTAGE; ++b) {
            mbar_init(smem_u32(&bars[b]), 1);
            mbar_init(smem_u32(&bars[C::NSTAGE + b]), C::NCW);
        }
        flag[0] = 0;
        flag[1] = 0;
        fence_barrier_init();
    }

    // a4: rank -> relative offset of the attended decode entries of this CTA.
    const uint32_t *mrow = p.mask + (size_t)s * p.MW;
    const int nwords = (p.wlen + 31) >> 5;
    const int wpt = (nwords + C::THREADS - 1) / C::THREADS;
    const int w0 = min(tid * wpt, nwords);
    const int w1 = min(w0 + wpt, nwords);
    int mine = 0;
    for (int w = w0; w < w1; ++w) mine += __popc(attended_bits(__ldg(mrow + w), w, p.wlen));
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int rank = incl - mine;
    int total = 0;
    for (int wi = 0; wi < C::NCW + 1; ++wi) {
        const int x = wsum[wi];
        rank += (wi < warp) ? x : 0;
        total += x;
    }
    if (total != p.a) {
        // The skip mask disagrees with the host's count: record it and keep
        // every listed offset in range (missing entries read as offset 0).
        if (tid == 0) atomicOr(p.status, ST_CHECK);
        for (int i = tid; i < khi - klo; i += C::THREADS) list[i] = 0;
        __syncthreads();
    }
    if (rank < khi) {
        for (int w = w0; w < w1 && rank < khi; ++w) {
            uint32_t bits = attended_bits(__ldg(mrow + w), w, p.wlen);
            const int cnt = __popc(bits);
            if (rank + cnt <= klo) {
                rank += cnt;
                continue;
            }
            while (bits) {
                const int b = __ffs(bits) - 1;
                if (rank >= klo && rank < khi) list[rank - klo] = (uint16_t)(w * 32 + b);
                ++rank;
                bits &= bits - 1;
            }
        }
    }

    // a2: append the new entry (split 0 of each stream).
    if (c == 0 && warp < C::NCW) {
        constexpr int NV = C::KROW / 16;
        T *dst = p.sinkmode ? reinterpret_cast<T *>(p.prefix) + ((size_t)s * p.Lcap + p.P) * 2 * D
                            : reinterpret_cast<T *>(p.ring) + ((size_t)s * p.R + (p.tin % p.R)) * 2 * D;
        const uint4 *ks = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.knew) + (size_t)s * D);
        const uint4 *vs = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.vnew) + (size_t)s * D);
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
        for (int i = tid; i < 2 * NV; i += 32 * C::NCW) d4[i] = (i < NV) ? __ldg(ks + i) : __ldg(vs + i - NV);
    }
    __syncthreads();

    const uint32_t full0 = smem_u32(&bars[0]);
    const uint32_t empty0 = smem_u32(&bars[C::NSTAGE]);
    int lastj[C::NSTAGE];  // producer: last stage issued into each buffer
#pragma unroll
    for (int b = 0; b < C::NSTAGE; ++b) lastj[b] = -1;

    if (warp == C::NCW) {
        // ---------------- producer warp: a5 gather via the bulk-copy engine
        const unsigned char *pre =
            reinterpret_cast<const unsigned char *>(p.prefix) + (size_t)s * p.Lcap * C::ROW;
        const unsigned char *rng = reinterpret_cast<const unsigned char *>(p.ring) + (size_t)s * p.R * C::ROW;
        const unsigned char *kn = reinterpret_cast<const unsigned char *>(p.knew) + (size_t)s * C::KROW;
        const unsigned char *vn = reinterpret_cast<const unsigned char *>(p.vnew) + (size_t)s * C::KROW;
        const uint64_t pol = policy_evict_first();
        for (int j = 0; j < nst; ++j) {
            const int b = j % C::NSTAGE;
            if (j >= C::NSTAGE) {
                bool ok = true;
                if (lane == 0) ok = wait_phase(empty0 + 8 * b, ((j / C::NSTAGE) - 1) & 1, p.wait_limit);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0) {
                        flag[0] = 1;
                        atomicOr(p.status, ST_TIMEOUT);
                    }
                    break;
                }
                if (flag[0]) break;
            }
            const int v0 = lo + j * C::ROWS;
            const int v1 = min(v0 + C::ROWS, hi);
            const uint32_t dst = smem_u32(smem + b * C::STAGE_BYTES);
            const uint32_t fb = full0 + 8 * b;
            if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)(v1 - v0) * C::ROW);
            __syncwarp();
            const int pe = min(v1, p.P);
            if (lane == 0 && pe > v0) bulk_g2s_hint(dst, pre + (size_t)v0 * C::ROW, (pe - v0) * C::ROW, fb, pol);
            for (int i = max(v0, p.P) + lane; i < v1; i += 32) {
                const int r = list[i - p.P - klo];
                const uint32_t sd = dst + (i - v0) * C::ROW;
                if (r == 0) {
                    bulk_g2s(sd, kn, C::KROW, fb);
                    bulk_g2s(sd + C::KROW, vn, C::KROW, fb);
                } else {
                    const int slot = (p.tin - r) % p.R;
                    bulk_g2s_hint(sd, rng + (size_t)slot * C::ROW, C::ROW, fb, pol);
                }
            }
            lastj[b] = j;
        }
        __syncwarp();
    } else {
        // ---------------- consumer warps: a5 logits, a6 softmax.V, a8 argmin
        const int g = lane / C::LPR;
        const int cl = lane % C::LPR;
        float qf[C::VEC];
        {
            const uint4 qv = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.q) + (size_t)s * D) + cl);
            EL::widen(qv, qf);
#pragma unroll
            for (int e = 0; e < C::VEC; ++e) qf[e] *= p.qscale;
        }
        float acc[C::VEC];
#pragma unroll
        for (int e = 0; e < C::VEC; ++e) acc[e] = 0.f;
        float m = -INFINITY, l = 0.f;
        float minv = INFINITY;
        int minr = -1;
        for (int j = 0; j < nst; ++j) {
            const int b = j % C::NSTAGE;
            const bool ok = wait_phase(full0 + 8 * b, (j / C::NSTAGE) & 1, p.wait_limit);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) {
                    flag[0] = 1;
                    atomicOr(p.status, ST_TIMEOUT);
                }
                break;
            }
            const int v0 = lo + j * C::ROWS;
            const int nr = min(C::ROWS, hi - v0);
            const unsigned char *st = smem + b * C::STAGE_BYTES;
            float sc[C::NIT];
#pragma unroll
            for (int it = 0; it < C::NIT; ++it) {
                const int row = warp * C::RPC + it * C::RPW + g;
                const bool valid = row < nr;
                float x = 0.f;
                if (valid) {
                    float kf[C::VEC];
                    EL::widen(*reinterpret_cast<const uint4 *>(st + row * C::ROW + cl * 16), kf);
#pragma unroll
                    for (int e = 0; e < C::VEC; ++e) x = fmaf(qf[e], kf[e], x);
                }
#pragma unroll
                for (int o = C::LPR / 2; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                sc[it] = valid ? x : -INFINITY;
                if (p.select && valid && v0 + row >= p.P) {
                    const int r = list[v0 + row - p.P - klo];
                    if (x < minv || (x == minv && r > minr)) {
                        minv = x;
                        minr = r;
                    }
                }
            }
            float mx = sc[0];
#pragma unroll
            for (int it = 1; it < C::NIT; ++it) mx = fmaxf(mx, sc[it]);
#pragma unroll
            for (int o = C::LPR; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float mn = fmaxf(m, mx);
            if (mn != -INFINITY) {
                const float alpha = exp2f(m - mn);
                l *= alpha;
#pragma unroll
                for (int e = 0; e < C::VEC; ++e) acc[e] *= alpha;
#pragma unroll
                for (int it = 0; it < C::NIT; ++it) {
                    const int row = warp * C::RPC + it * C::RPW + g;
                    if (row < nr) {
                        const float pj = exp2f(sc[it] - mn);
                        l += pj;
                        float vf[C::VEC];
                        EL::widen(*reinterpret_cast<const uint4 *>(st + row * C::ROW + C::KROW + cl * 16), vf);
#pragma unroll
                        for (int e = 0; e < C::VEC; ++e) acc[e] = fmaf(pj, vf[e], acc[e]);
                    }
                }
                m = mn;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * b);
        }
        // merge the row groups of the warp (m is warp-uniform)
#pragma unroll
        for (int o = C::LPR; o < 32; o <<= 1) {
            l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
            for (int e = 0; e < C::VEC; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
            const float ov = __shfl_xor_sync(0xffffffffu, minv, o);
            const int orr = __shfl_xor_sync(0xffffffffu, minr, o);
            if (ov < minv || (ov == minv && orr > minr)) {
                minv = ov;
                minr = orr;
            }
        }
        if (lane < C::LPR) {
#pragma unroll
            for (int e = 0; e < C::VEC; ++e) comb[warp * D + cl * C::VEC + e] = acc[e];
        }
        if (lane == 0) cml[warp] = make_float4(m, l, minv, __int_as_float(minr));
    }
    __syncthreads();
    // If any warp gave up, every copy still in flight must land (bounded
    // wait) before the CTA's shared memory is released.  The flag is read
    // after the barrier, so a late abort by a consumer is seen here.
    if (flag[0]) {
        if (warp == C::NCW && lane == 0) {
#pragma unroll
            for (int b = 0; b < C::NSTAGE; ++b)
                if (lastj[b] >= 0) wait_phase(full0 + 8 * b, (lastj[b] / C::NSTAGE) & 1, 0xffffffffu);
        }
        __syncthreads();
    }

    // a6/a7: merge the consumer warps of this CTA.
    float2 best = make_float2(INFINITY, __int_as_float(-1));
    if (tid == 0 && p.select) {
        for (int w = 0; w < C::NCW; ++w) {
            const float4 x = cml[w];
            const int rx = __float_as_int(x.w), rb = __float_as_int(best.y);
            if (x.z < best.x || (x.z == best.x && rx > rb)) best = make_float2(x.z, x.w);
        }
    }
    float O = 0.f, M = -INFINITY, L = 0.f;
    if (tid < D) {
        for (int w = 0; w < C::NCW; ++w) M = fmaxf(M, cml[w].x);
        for (int w = 0; w < C::NCW; ++w) {
            const float4 x = cml[w];
            if (x.x != -INFINITY) {
                const float f = exp2f(x.x - M);
                O = fmaf(comb[w * D + tid], f, O);
                L = fmaf(x.y, f, L);
            }
        }
    }
    const size_t slot = (size_t)s * p.pstride + c;
    if (p.nsplit == 1) {
        if (tid < D) reinterpret_cast<T *>(p.out)[(size_t)s * D + tid] = EL::narrow(O / L);
        if (tid == 0 && p.select && !flag[0] && __float_as_int(best.y) >= 0) {
            const int r = __float_as_int(best.y);
            p.last_sel[s] = r;
            p.mask[(size_t)s * p.MW + (r >> 5)] |= 1u << (r & 31);
        }
        return;
    }
    if (tid < D) p.part_acc[slot * D + tid] = O;
    if (tid == 0) {
        p.part_ml[slot] = make_float2(M, L);
        p.part_min[slot] = best;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) flag[1] = (atomicAdd(p.ticket + s, 1) == p.nsplit - 1);
    __syncthreads();
    if (!flag[1]) return;
    __threadfence();
    const size_t base = (size_t)s * p.pstride;
    if (tid < D) {
        float Mx = -INFINITY;
        for (int i = 0; i < p.nsplit; ++i) Mx = fmaxf(Mx, __ldcg(&p.part_ml[base + i].x));
        float Ox = 0.f, Lx = 0.f;
        for (int i = 0; i < p.nsplit; ++i) {
            const float2 ml = __ldcg(&p.part_ml[base + i]);
            if (ml.x != -INFINITY) {
                const float f = exp2f(ml.x - Mx);
                Ox = fmaf(__ldcg(&p.part_acc[(base + i) * D + tid]), f, Ox);
                Lx = fmaf(ml.y, f, Lx);
            }
        }
        reinterpret_cast<T *>(p.out)[(size_t)s * D + tid] = EL::narrow(Ox / Lx);
    }
    if (tid == 0) {
        p.ticket[s] = 0;
        if (p.select && *reinterpret_cast<volatile int *>(p.status) == 0) {
            float bv = INFINITY;
            int br = -1;
            for (int i = 0; i < p.nsplit; ++i) {
                const float2 x = __ldcg(&p.part_min[base + i]);
                const int rx = __float_as_int(x.y);
                if (x.x < bv || (x.x == bv && rx > br)) {
                    bv = x.x;
                    br = rx;
                }
            }
            if (br >= 0) {
                p.last_sel[s] = br;
                p.mask[(size_t)s * p.MW + (br >> 5)] |= 1u << (br & 31);
            }
        }
    }
}

// a1: prompt K, V [S, L_p, D] -> prefix [S, Lcap, 2, D].
template <typename T, int D>
__global__ void prefill_kernel(const T *__restrict__ K, const T *__restrict__ V, T *__restrict__ prefix, int S,
                               int L_p, int Lcap)
{
    constexpr int VPR = D * (int)sizeof(T) / 16;
    const size_t total = (size_t)S * L_p * 2 * VPR;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int vec = (int)(i % VPR);
        size_t rest = i / VPR;
        const int kv = (int)(rest & 1);
        rest >>= 1;
        const int row = (int)(rest % L_p);
        const size_t s = rest / L_p;
        const uint4 *src = reinterpret_cast<const uint4 *>((kv ? V : K) + (s * L_p + row) * D) + vec;
        uint4 *dst = reinterpret_cast<uint4 *>(prefix + ((s * Lcap + row) * 2 + kv) * D) + vec;
        *dst = __ldg(src);
    }
}

}  // namespace dsa
