// dsa_policy.cu -- score-based KV eviction baselines (TOVA, H2O) for the
// comparison in "Understanding and Exploiting Diagonal Attention Sparsity in
// Autoregressive Image Generation", section 2 (Fig. 2, "KV cache sparsity
// techniques") and section 5.1 ("Sparse KV baselines").  C ABI in
// include/dsa_policy.h, readings there.
//
// State per stream: the prompt prefix and N_att slots of K|V entries (512 B
// each at bf16, head_dim 128), the position each slot holds, the slot the
// next token goes to, and for H2O each slot's accumulated weight.  At step
// t the attended decode entries are the occupied slots other than the
// current token's slot (one or two contiguous runs) plus the current token.
//
// policy_kernel: a persistent grid whose warps take whole streams (striped
// over the CTAs, so that every CTA gets as many streams as the others give
// or take one).  A warp streams the stream's prompt rows and slot runs
// through its own shared-memory stages (bulk copies, nbuf in flight,
// continuing into the next stream), computes the logits with 8 lanes per row and an online softmax
// with P.V, holds the current token in registers (and stores it to its
// slot), combines its row groups with shuffles, writes the output and
// applies the eviction: TOVA's argmin of (logit, position) is tracked in the
// same pass; H2O keeps the decode logits in shared memory, adds each
// entry's normalised weight to its slot's accumulated weight once the
// softmax is complete, and takes the argmin of (accumulated weight,
// position) outside the recent window.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <new>

#include "../../include/dsa.h"
#include "../../include/dsa_policy.h"
#include "dsa_decode.cuh"
#include "dsa_internal.h"

namespace dsa_pol_k {

using namespace dsa;

constexpr int kWarps = 4;
constexpr int kMaxNbuf = 4;
// Stage sizes 8 KB or 6 KB, and 2 to 4 stages per warp: the host picks per
// handle the pair whose resident warps take the streams in the fewest
// rounds, and among those the deepest pipeline per warp (with fewer streams
// than warp slots, the idle warps' shared memory goes to the busy ones).
constexpr int kStages[2] = {8192, 6144};
constexpr uint32_t kNoWaitLimit = 0xffffffffu;

struct PolParams {
    const void *q, *knew, *vnew;
    void *out;
    const void *prefix;  // [S, L_p, 2, D]
    void *slots;         // [S, R, 2, D]
    int32_t *slot_pos;   // [S, R]
    int32_t *free_slot;  // [S]
    float *acc;          // [S, R] (H2O)
    int32_t *last_evict; // [S]
    int *status;
    int S, L_p, R, t;
    int nos;             // occupied slots before this step's token: min(t, R)
    int full;            // 1: this step attends N_att decode entries and evicts one
    int n_recent;        // H2O: newest entries never evicted
    float qscale;        // log2(e) / sqrt(D)
    uint32_t wait_limit;
    int warp_smem;       // bytes of shared memory per warp
    int nbuf;            // stages per warp (2 .. kMaxNbuf)
    int early;           // 1: the previous grid in the stream is not one of this handle's, so
                         // the handle's own state may be read before the grid dependency wait
};

template <typename T, int D, int STAGE>
struct PCfg {
    static constexpr int VEC = Elem<T>::VEC;
    static constexpr int LPR = D / (2 * VEC);
    static constexpr int RPW = 32 / LPR;
    static constexpr int KROW = D * (int)sizeof(T);
    static constexpr int ROW = 2 * KROW;
    static constexpr int SR = STAGE / ROW;  // rows per stage
    static constexpr int NIT = SR / RPW;
    static_assert(SR % RPW == 0, "stage rows fill whole warp instructions");
};

__device__ __forceinline__ bool lower(float v, int pos, float bv, int bpos)
{
    return v < bv || (v == bv && pos < bpos);  // lower score; on a tie the older entry
}

// Rows of stream s at this step: prompt rows, then slot run A = [0, nA),
// then slot run B = [fs + 1, fs + 1 + nB).
struct Rows {
    int fs, nA, nB, n;
};

__device__ __forceinline__ Rows stream_rows(const PolParams &p, int s)
{
    Rows r;
    r.fs = __ldcg(p.free_slot + s);
    if (r.fs < 0 || r.fs >= p.R) {  // never happens on a consistent state; keeps every access in range
        if ((threadIdx.x & 31) == 0) atomicOr(p.status, ST_CHECK);
        r.fs = p.R - 1;
    }
    r.nA = min(r.fs, p.nos);
    r.nB = max(p.nos - r.fs - 1, 0);
    r.n = p.L_p + r.nA + r.nB;
    return r;
}

template <typename T, int D, int POL, int STAGE>
__global__ void __launch_bounds__(32 * kWarps) policy_kernel(const PolParams p)
{
    using C = PCfg<T, D, STAGE>;
    constexpr int kStage = STAGE;
    using EL = Elem<T>;
    using IO = typename EL::IO;
    using Vec = typename EL::Vec;
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbuf = p.nbuf;
    unsigned char *ws = smem + warp * p.warp_smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(ws + nbuf * kStage);
    float *xs = reinterpret_cast<float *>(ws + nbuf * kStage + 8 * kMaxNbuf);  // decode logits of the stream
    if (lane == 0) {
        for (int b = 0; b < nbuf; ++b) mbar_init(smem_u32(&bars[b]), 1);
        fence_barrier_init();
    }
    __syncwarp();
    const uint32_t bar0 = smem_u32(&bars[0]);
    const uint32_t buf0 = smem_u32(ws);
    const int g = lane / C::LPR, cl = lane % C::LPR;
    const uint64_t pol = policy_evict_first();
    const int GW = gridDim.x * kWarps;
    const int first = warp * gridDim.x + blockIdx.x;

    int issued = 0, consumed = 0;
    int ib = 0;            // buffer of the next issued stage
    int cb = 0, cpar = 0;  // buffer and phase parity of the next consumed stage
    bool aborted = false;
    // issuer cursor over (stream, stage) of this warp's streams
    int is = first, ij = 0;
    Rows ir{};
    bool iset = false;
    auto issue_one = [&]() -> bool {
        while (is < p.S) {
            if (!iset) {
                ir = stream_rows(p, is);
                iset = true;
            }
            if (ij * C::SR < ir.n) {
                const int b = ib;
                ib = ib + 1 == nbuf ? 0 : ib + 1;
                const uint32_t fb = bar0 + 8 * b;
                const uint32_t dst = buf0 + b * kStage;
                const int u0 = ij * C::SR, u1 = min(u0 + C::SR, ir.n);
                if (lane == 0) {
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(fb, (uint32_t)(u1 - u0) * C::ROW);
                    const unsigned char *pre = reinterpret_cast<const unsigned char *>(p.prefix) + (size_t)is * p.L_p * C::ROW;
                    const unsigned char *sl = reinterpret_cast<const unsigned char *>(p.slots) + (size_t)is * p.R * C::ROW;
                    // prompt part
                    int a = u0, e = min(u1, p.L_p);
                    if (e > a) bulk_g2s_hint(dst, pre + (size_t)a * C::ROW, (e - a) * C::ROW, fb, pol);
                    // run A: rows L_p .. L_p + nA -> slots 0 .. nA
                    a = max(u0, p.L_p);
                    e = min(u1, p.L_p + ir.nA);
                    if (e > a) bulk_g2s_hint(dst + (a - u0) * C::ROW, sl + (size_t)(a - p.L_p) * C::ROW, (e - a) * C::ROW, fb, pol);
                    // run B: rows L_p + nA .. n -> slots fs + 1 ..
                    a = max(u0, p.L_p + ir.nA);
                    e = u1;
                    if (e > a)
                        bulk_g2s_hint(dst + (a - u0) * C::ROW, sl + (size_t)(a - p.L_p - ir.nA + ir.fs + 1) * C::ROW,
                                      (e - a) * C::ROW, fb, pol);
                }
                ++issued;
                ++ij;
                return true;
            }
            is += GW;
            ij = 0;
            iset = false;
        }
        return false;
    };
    auto top_up = [&]() {
        while (issued - consumed < nbuf && issue_one()) {
        }
    };
    // Programmatic dependent launch.  The previous grid in the stream may have
    // written q, k_new and v_new, and, if it was this handle's own step or
    // prefill, the handle's state.  Otherwise that state is final here (the
    // previous grid let this one start only after its own wait, which
    // followed this handle's last kernel), so the first stages are issued
    // before the wait; q, k_new, v_new and every write come after it.
    if (p.early) top_up();
    pdl_wait();
    pdl_launch_dependents();
    top_up();

    for (int s = first; s < p.S && !aborted; s += GW) {
        const Rows rw = stream_rows(p, s);
        const int nst = (rw.n + C::SR - 1) / C::SR;
        const uint4 *qr = reinterpret_cast<const uint4 *>(reinterpret_cast<const IO *>(p.q) + (size_t)s * D);
        const typename EL::Q q0 = EL::load_q(__ldg(qr + cl)), q1 = EL::load_q(__ldg(qr + cl + C::LPR));
        const IO *kio = reinterpret_cast<const IO *>(p.knew) + (size_t)s * D;
        const IO *vio = reinterpret_cast<const IO *>(p.vnew) + (size_t)s * D;
        const Vec kc0 = EL::load_kv(kio, cl, 1.f), kc1 = EL::load_kv(kio, cl + C::LPR, 1.f);
        const Vec vc0 = EL::load_kv(vio, cl, 1.f), vc1 = EL::load_kv(vio, cl + C::LPR, 1.f);
        const int32_t *spos = p.slot_pos + (size_t)s * p.R;

        float acc[2 * C::VEC];
#pragma unroll
        for (int e = 0; e < 2 * C::VEC; ++e) acc[e] = 0.f;
        float m = -INFINITY, l = 0.f;

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
            const unsigned char *st = ws + b * kStage;
            const int u0 = j * C::SR;
            const int nv = min(C::SR, rw.n - u0);
            float sc[C::NIT];
#pragma unroll
            for (int it = 0; it < C::NIT; ++it) {
                const int row = it * C::RPW + g;
                const bool valid = row < nv;
                float s0 = 0.f, s1 = 0.f;
                if (valid) {
                    const Vec *kr = reinterpret_cast<const Vec *>(st + row * C::ROW);
                    EL::dot(q0, kr[cl], s0, s1);
                    EL::dot(q1, kr[cl + C::LPR], s0, s1);
                }
                float x = s0 + s1;
#pragma unroll
                for (int o = C::LPR / 2; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                x *= p.qscale;
                sc[it] = valid ? x : -INFINITY;
                const int k = u0 + row - p.L_p;  // decode rank of the row (< 0: prompt)
                if (valid && k >= 0 && cl == 0) xs[k] = x;  // for the eviction, after the pass
            }
            float mx = sc[0];
#pragma unroll
            for (int it = 1; it < C::NIT; ++it) mx = fmaxf(mx, sc[it]);
#pragma unroll
            for (int o = C::LPR; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (mx > m) {
                const float alpha = ex2(m - mx);
                l *= alpha;
#pragma unroll
                for (int e = 0; e < 2 * C::VEC; ++e) acc[e] *= alpha;
                m = mx;
            }
#pragma unroll
            for (int it = 0; it < C::NIT; ++it) {
                const int row = it * C::RPW + g;
                if (row < nv) {
                    const float pj = ex2(sc[it] - m);
                    l += pj;
                    const Vec *vr = reinterpret_cast<const Vec *>(st + row * C::ROW + C::KROW);
                    EL::axpy(pj, vr[cl], acc);
                    EL::axpy(pj, vr[cl + C::LPR], acc + C::VEC);
                }
            }
            __syncwarp();
            top_up();
        }
        if (aborted) break;

        // the current token, from registers; stored to its slot
        float xc;
        {
            float s0 = 0.f, s1 = 0.f;
            EL::dot(q0, kc0, s0, s1);
            EL::dot(q1, kc1, s0, s1);
            xc = s0 + s1;
#pragma unroll
            for (int o = C::LPR / 2; o >= 1; o >>= 1) xc += __shfl_xor_sync(0xffffffffu, xc, o);
            xc *= p.qscale;
        }
        if (xc > m) {
            const float alpha = ex2(m - xc);
            l *= alpha;
#pragma unroll
            for (int e = 0; e < 2 * C::VEC; ++e) acc[e] *= alpha;
            m = xc;
        }
        if (g == 0) {
            const float pj = ex2(xc - m);
            l += pj;
            EL::axpy(pj, vc0, acc);
            EL::axpy(pj, vc1, acc + C::VEC);
            Vec *dst = reinterpret_cast<Vec *>(reinterpret_cast<T *>(p.slots) + ((size_t)s * p.R + rw.fs) * 2 * D);
            dst[cl] = kc0;
            dst[cl + C::LPR] = kc1;
            dst[2 * C::LPR + cl] = vc0;
            dst[3 * C::LPR + cl] = vc1;
        }
        // combine the row groups
#pragma unroll
        for (int o = C::LPR; o < 32; o <<= 1) {
            l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
            for (int e = 0; e < 2 * C::VEC; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
        }
        if (g == 0) {
            const float inv = 1.f / l;
            uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<IO *>(p.out) + (size_t)s * D);
            o[cl] = EL::pack(acc, inv);
            o[cl + C::LPR] = EL::pack(acc + C::VEC, inv);
        }
        // The eviction.  TOVA: the lowest logit among the attended decode
        // entries and the current token.  H2O: every attended decode entry
        // adds its normalised weight to its slot's total; the lowest total
        // outside the recent window goes.  Ties go to the older position.
        float minv = INFINITY;
        int minpos = INT_MAX, minslot = -1;
        if (POL == DSA_POLICY_H2O || p.full) {
            __syncwarp();
            float *accw = p.acc + (size_t)s * p.R;
            const float inv = 1.f / l;
            const int nold = rw.nA + rw.nB;
            const int oldest_recent = POL == DSA_POLICY_H2O ? p.t - p.n_recent + 1 : INT_MAX;  // positions >= this are kept
            for (int k = lane; k < nold; k += 32) {
                const int slot = k < rw.nA ? k : k + 1;
                float a = xs[k];
                if (POL == DSA_POLICY_H2O) {
                    a = __ldcg(accw + slot) + ex2(a - m) * inv;
                    accw[slot] = a;
                }
                const int pos = __ldg(spos + slot);
                if (p.full && pos < oldest_recent && lower(a, pos, minv, minpos)) {
                    minv = a;
                    minpos = pos;
                    minslot = slot;
                }
            }
            float ac = xc;
            if (POL == DSA_POLICY_H2O) ac = ex2(xc - m) * inv;
            if (lane == 0) {
                if (POL == DSA_POLICY_H2O) accw[rw.fs] = ac;
                if (p.full && p.t < oldest_recent && lower(ac, p.t, minv, minpos)) {
                    minv = ac;
                    minpos = p.t;
                    minslot = rw.fs;
                }
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, minv, o);
                const int op = __shfl_xor_sync(0xffffffffu, minpos, o);
                const int osl = __shfl_xor_sync(0xffffffffu, minslot, o);
                if (lower(ov, op, minv, minpos)) {
                    minv = ov;
                    minpos = op;
                    minslot = osl;
                }
            }
        }
        if (lane == 0) {
            p.slot_pos[(size_t)s * p.R + rw.fs] = p.t;
            if (p.full && minslot >= 0) {
                p.slot_pos[(size_t)s * p.R + minslot] = -1;
                p.free_slot[s] = minslot;
                p.last_evict[s] = minpos;
            } else {
                // filling: the next slot (a full step always finds a victim
                // unless its scores are NaN; then the current slot is reused)
                p.free_slot[s] = p.full ? rw.fs : rw.fs + 1;
                p.last_evict[s] = -1;
            }
        }
        __syncwarp();
    }
    // A warp that gave up lets its own copies in flight land before exit.
    if (aborted && lane == 0) {
        for (int q = consumed; q < issued; ++q) drain_phase(bar0 + 8 * (q % nbuf), (q / nbuf) & 1);
    }
    __syncwarp();
}

}  // namespace dsa_pol_k

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
using dsa_detail::cuda_fail;
using dsa_detail::dev_alloc;
using dsa_detail::fail;

namespace {

constexpr uint32_t kPolMagic = 0x44535054u;  // "DSPT"

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
int row_bytes(int dtype, int D) { return 2 * D * (dtype == DSA_F32 ? 4 : 2); }

}  // namespace

struct dsa_pol_ctx {
    uint32_t magic;
    int S, D, L_p, R, policy, dtype;
    int t, prefilled, evicted_last;
    int sms, grid, warp_smem, smem, shape, nbuf;
    uint32_t wait_limit;
    void *prefix, *slots;
    int32_t *slot_pos, *free_slot, *last_evict;
    float *acc;
    int *status;
};

namespace {

bool valid(const dsa_pol_ctx *h) { return h != nullptr && h->magic == kPolMagic; }

void free_pol(dsa_pol_ctx *h)
{
    if (!h) return;
    cudaFree(h->prefix);
    cudaFree(h->slots);
    cudaFree(h->slot_pos);
    cudaFree(h->free_slot);
    cudaFree(h->last_evict);
    cudaFree(h->acc);
    cudaFree(h->status);
    h->magic = 0;
    dsa_detail::forget_handle(h);
    delete h;
}

template <typename T, int D, int POL, int STAGE>
cudaError_t pol_occupancy(int smem, int *ctas)
{
    cudaError_t e = cudaFuncSetAttribute(dsa_pol_k::policy_kernel<T, D, POL, STAGE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, dsa_pol_k::policy_kernel<T, D, POL, STAGE>,
                                                         32 * dsa_pol_k::kWarps, smem);
}

template <typename T, int D, int POL>
cudaError_t pol_occupancy_s(int shape, int smem, int *ctas)
{
    return shape == 0 ? pol_occupancy<T, D, POL, dsa_pol_k::kStages[0]>(smem, ctas)
                      : pol_occupancy<T, D, POL, dsa_pol_k::kStages[1]>(smem, ctas);
}

template <typename T, int D>
cudaError_t pol_occupancy_d(int policy, int shape, int smem, int *ctas)
{
    return policy == DSA_POLICY_H2O ? pol_occupancy_s<T, D, DSA_POLICY_H2O>(shape, smem, ctas)
                                    : pol_occupancy_s<T, D, DSA_POLICY_TOVA>(shape, smem, ctas);
}

cudaError_t pol_occupancy_any(int dtype, int D, int policy, int shape, int smem, int *ctas)
{
    if (dtype == DSA_BF16)
        return D == 64 ? pol_occupancy_d<__nv_bfloat16, 64>(policy, shape, smem, ctas)
                       : pol_occupancy_d<__nv_bfloat16, 128>(policy, shape, smem, ctas);
    return D == 64 ? pol_occupancy_d<float, 64>(policy, shape, smem, ctas)
                   : pol_occupancy_d<float, 128>(policy, shape, smem, ctas);
}

// Shared memory per warp for `nbuf` stages of stage size sh.
int warp_bytes(const dsa_pol_ctx *h, int sh, int nbuf)
{
    return (nbuf * dsa_pol_k::kStages[sh] + 8 * dsa_pol_k::kMaxNbuf + 4 * h->R + 127) / 128 * 128;
}

// Resident CTAs per SM of the launch shape (stage size sh, nbuf stages per
// warp); 0 if it cannot launch.
int shape_ctas(const dsa_pol_ctx *h, int sh, int nbuf)
{
    int ctas = 0;
    const cudaError_t e = pol_occupancy_any(h->dtype, h->D, h->policy, sh, dsa_pol_k::kWarps * warp_bytes(h, sh, nbuf), &ctas);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return ctas;
}

void apply_shape(dsa_pol_ctx *h, int sh, int nbuf, int ctas)
{
    h->shape = sh;
    h->nbuf = nbuf;
    h->warp_smem = warp_bytes(h, sh, nbuf);
    h->smem = dsa_pol_k::kWarps * h->warp_smem;
    const long long cap = (long long)h->sms * ctas;
    h->grid = (int)(h->S < cap ? h->S : cap);  // streams are striped over the CTAs: none is left empty
}

// The automatic launch shape: the fewest rounds of resident warps over the
// streams, then the most stage bytes per warp, then 8 KB stages.  Returns
// false if no shape can launch.
bool auto_shape(dsa_pol_ctx *h)
{
    long long best_rounds = LLONG_MAX;
    int best_depth = 0, best_sh = -1, best_nb = 0, best_ctas = 0;
    for (int sh = 0; sh < 2; ++sh)
        for (int nb = 2; nb <= dsa_pol_k::kMaxNbuf; ++nb) {
            const int ctas = shape_ctas(h, sh, nb);
            if (ctas < 1) continue;
            const long long warps = (long long)h->sms * ctas * dsa_pol_k::kWarps;
            const long long rounds = (h->S + warps - 1) / warps;
            const int depth = nb * dsa_pol_k::kStages[sh];
            if (rounds < best_rounds || (rounds == best_rounds && depth > best_depth)) {
                best_rounds = rounds;
                best_depth = depth;
                best_sh = sh;
                best_nb = nb;
                best_ctas = ctas;
            }
        }
    if (best_sh < 0) return false;
    apply_shape(h, best_sh, best_nb, best_ctas);
    return true;
}

template <typename T, int D, int POL, int STAGE>
cudaError_t pol_launch(const dsa_pol_k::PolParams &p, int grid, int smem, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * dsa_pol_k::kWarps);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dsa_pol_k::policy_kernel<T, D, POL, STAGE>, p);
}

template <typename T, int D, int POL>
cudaError_t pol_launch_s(int shape, const dsa_pol_k::PolParams &p, int grid, int smem, cudaStream_t st)
{
    return shape == 0 ? pol_launch<T, D, POL, dsa_pol_k::kStages[0]>(p, grid, smem, st)
                      : pol_launch<T, D, POL, dsa_pol_k::kStages[1]>(p, grid, smem, st);
}

template <typename T, int D>
cudaError_t pol_launch_d(int policy, int shape, const dsa_pol_k::PolParams &p, int grid, int smem, cudaStream_t st)
{
    return policy == DSA_POLICY_H2O ? pol_launch_s<T, D, DSA_POLICY_H2O>(shape, p, grid, smem, st)
                                    : pol_launch_s<T, D, DSA_POLICY_TOVA>(shape, p, grid, smem, st);
}

template <typename T, int D>
cudaError_t pol_prefill(const void *K, const void *V, void *prefix, int S, int L_p, cudaStream_t st)
{
    using IO = typename dsa::Elem<T>::IO;
    const size_t total = (size_t)S * L_p * 2 * (D / dsa::Elem<T>::VEC);
    if (total == 0) return cudaSuccess;
    size_t blocks = (total + 255) / 256;
    if (blocks > 65535 * 8) blocks = 65535 * 8;
    dsa::prefill_kernel<T, D><<<(unsigned)blocks, 256, 0, st>>>((const IO *)K, (const IO *)V, (T *)prefix, nullptr,
                                                                nullptr, S, L_p, L_p);
    return cudaGetLastError();
}

int copy_back(const void *src, void *host, size_t bytes, cudaStream_t st, const char *what)
{
    cudaError_t e = cudaMemcpyAsync(host, src, bytes, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, what);
}

}  // namespace

extern "C" {

int dsa_pol_create(int heads, int head_dim, int L_p, int N_att, int policy, int dtype, dsa_pol *out)
{
    if (!out) return fail(DSA_ERR_ARG, "out is NULL");
    *out = nullptr;
    if (heads < 1) return fail(DSA_ERR_ARG, "heads must be >= 1 (got %d)", heads);
    if (head_dim != 64 && head_dim != 128) return fail(DSA_ERR_ARG, "head_dim must be 64 or 128 (got %d)", head_dim);
    if (L_p < 0) return fail(DSA_ERR_ARG, "L_p must be >= 0 (got %d)", L_p);
    if (N_att < 1 || N_att > 65536) return fail(DSA_ERR_ARG, "N_att must be in [1, 65536] (got %d)", N_att);
    if (policy != DSA_POLICY_TOVA && policy != DSA_POLICY_H2O)
        return fail(DSA_ERR_ARG, "policy must be DSA_POLICY_TOVA or DSA_POLICY_H2O (got %d)", policy);
    if (dtype != DSA_BF16 && dtype != DSA_F32) return fail(DSA_ERR_ARG, "dtype must be DSA_BF16 or DSA_F32 (got %d)", dtype);
    if ((long long)heads * N_att > INT_MAX || (long long)L_p * heads > INT_MAX / 4)
        return fail(DSA_ERR_ARG, "heads x N_att or heads x L_p too large");

    dsa_pol_ctx *h = new (std::nothrow) dsa_pol_ctx();
    if (!h) return fail(DSA_ERR_OOM, "host allocation failed");
    h->magic = kPolMagic;
    h->S = heads;
    h->D = head_dim;
    h->L_p = L_p;
    h->R = N_att;
    h->policy = policy;
    h->dtype = dtype;
    h->wait_limit = dsa_pol_k::kNoWaitLimit;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        free_pol(h);
        return cuda_fail(e, "device query");
    }
    if (!auto_shape(h)) {
        free_pol(h);
        return fail(DSA_ERR_CUDA, "policy kernel setup failed (is this an sm_103 device, and N_att within shared memory?)");
    }

    const size_t S = (size_t)heads, row = (size_t)row_bytes(dtype, head_dim);
    int rc = dev_alloc(&h->prefix, S * L_p * row, "policy prompt prefix");
    if (rc == DSA_OK) rc = dev_alloc(&h->slots, S * N_att * row, "policy slots");
    if (rc == DSA_OK) rc = dev_alloc((void **)&h->slot_pos, S * N_att * 4, "slot positions");
    if (rc == DSA_OK) rc = dev_alloc((void **)&h->free_slot, S * 4, "free slots");
    if (rc == DSA_OK) rc = dev_alloc((void **)&h->last_evict, S * 4, "last evictions");
    if (rc == DSA_OK && policy == DSA_POLICY_H2O) rc = dev_alloc((void **)&h->acc, S * N_att * 4, "accumulated weights");
    if (rc == DSA_OK) rc = dev_alloc((void **)&h->status, 16, "status word");
    if (rc != DSA_OK) {
        free_pol(h);
        return rc;
    }
    if ((e = cudaMemset(h->status, 0, 16)) != cudaSuccess) {
        free_pol(h);
        return cuda_fail(e, "cudaMemset");
    }
    *out = h;
    return DSA_OK;
}

int dsa_pol_destroy(dsa_pol h)
{
    if (!h) return DSA_OK;
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid policy handle");
    cudaDeviceSynchronize();
    free_pol(h);
    return DSA_OK;
}

int dsa_pol_prefill(dsa_pol h, const void *K, const void *V, void *stream)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid policy handle");
    if (h->L_p > 0 && (!K || !V)) return fail(DSA_ERR_ARG, "K and V must be non-NULL when L_p > 0");
    if (h->L_p > 0 && (!aligned16(K) || !aligned16(V))) return fail(DSA_ERR_ARG, "K and V must be 16-byte aligned");
    cudaStream_t st = (cudaStream_t)stream;
    const size_t S = (size_t)h->S;
    cudaError_t e;
    if ((e = cudaMemsetAsync(h->slot_pos, 0xff, S * h->R * 4, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(h->free_slot, 0, S * 4, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(h->last_evict, 0xff, S * 4, st)) != cudaSuccess ||
        (h->acc && (e = cudaMemsetAsync(h->acc, 0, S * h->R * 4, st)) != cudaSuccess) ||
        (e = cudaMemsetAsync(h->status, 0, 16, st)) != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync");
    if (h->dtype == DSA_BF16)
        e = h->D == 64 ? pol_prefill<__nv_bfloat16, 64>(K, V, h->prefix, h->S, h->L_p, st)
                       : pol_prefill<__nv_bfloat16, 128>(K, V, h->prefix, h->S, h->L_p, st);
    else
        e = h->D == 64 ? pol_prefill<float, 64>(K, V, h->prefix, h->S, h->L_p, st)
                       : pol_prefill<float, 128>(K, V, h->prefix, h->S, h->L_p, st);
    if (e != cudaSuccess) return cuda_fail(e, "policy prefill launch");
    dsa_detail::note_launch(st, h);  // the next step waits for the prefill before reading the state
    h->t = 0;
    h->prefilled = 1;
    h->evicted_last = 0;
    return DSA_OK;
}

int dsa_pol_decode_step(dsa_pol h, const void *q, const void *k_new, const void *v_new, void *out, void *stream)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid policy handle");
    if (!h->prefilled) return fail(DSA_ERR_STATE, "dsa_pol_decode_step before dsa_pol_prefill");
    if (!q || !k_new || !v_new || !out) return fail(DSA_ERR_ARG, "q, k_new, v_new and out must be non-NULL");
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out))
        return fail(DSA_ERR_ARG, "q, k_new, v_new and out must be 16-byte aligned");
    if (h->t == INT_MAX) return fail(DSA_ERR_STATE, "decode step counter exhausted");
    dsa_pol_k::PolParams p;
    p.q = q;
    p.knew = k_new;
    p.vnew = v_new;
    p.out = out;
    p.prefix = h->prefix;
    p.slots = h->slots;
    p.slot_pos = h->slot_pos;
    p.free_slot = h->free_slot;
    p.acc = h->acc;
    p.last_evict = h->last_evict;
    p.status = h->status;
    p.S = h->S;
    p.L_p = h->L_p;
    p.R = h->R;
    p.t = h->t;
    p.nos = h->t < h->R ? h->t : h->R;
    p.full = (h->t + 1 >= h->R) ? 1 : 0;
    p.n_recent = (h->R + 1) / 2 < h->R - 1 ? (h->R + 1) / 2 : h->R - 1;
    p.qscale = (float)(1.4426950408889634 / std::sqrt((double)h->D));
    p.wait_limit = h->wait_limit;
    p.warp_smem = h->warp_smem;
    p.nbuf = h->nbuf;
    cudaStream_t st = (cudaStream_t)stream;
    p.early = dsa_detail::note_launch(st, h) ? 1 : 0;
    cudaError_t e;
    if (h->dtype == DSA_BF16)
        e = h->D == 64 ? pol_launch_d<__nv_bfloat16, 64>(h->policy, h->shape, p, h->grid, h->smem, st)
                       : pol_launch_d<__nv_bfloat16, 128>(h->policy, h->shape, p, h->grid, h->smem, st);
    else
        e = h->D == 64 ? pol_launch_d<float, 64>(h->policy, h->shape, p, h->grid, h->smem, st)
                       : pol_launch_d<float, 128>(h->policy, h->shape, p, h->grid, h->smem, st);
    if (e != cudaSuccess) return cuda_fail(e, "policy decode launch");
    h->evicted_last = p.full;
    h->t += 1;
    return DSA_OK;
}

int dsa_pol_get_positions(dsa_pol h, int32_t *host_dst, void *stream)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid policy handle");
    if (!host_dst) return fail(DSA_ERR_ARG, "host_dst is NULL");
    return copy_back(h->slot_pos, host_dst, (size_t)h->S * h->R * 4, (cudaStream_t)stream, "slot position copy");
}

int dsa_pol_get_last_eviction(dsa_pol h, int32_t *host_dst, void *stream)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid policy handle");
    if (!host_dst) return fail(DSA_ERR_ARG, "host_dst is NULL");
    if (!h->evicted_last) {
        for (int i = 0; i < h->S; ++i) host_dst[i] = -1;
        return DSA_OK;
    }
    return copy_back(h->last_evict, host_dst, (size_t)h->S * 4, (cudaStream_t)stream, "last eviction copy");
}

int dsa_pol_sync_status(dsa_pol h, void *stream)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid policy handle");
    int word = 0;
    int rc = copy_back(h->status, &word, 4, (cudaStream_t)stream, "status copy");
    if (rc != DSA_OK) return rc;
    if (word & dsa::ST_TIMEOUT) return fail(DSA_ERR_TIMEOUT, "a bounded wait in the policy kernel gave up");
    if (word & dsa::ST_CHECK) return fail(DSA_ERR_DEVICE_CHECK, "policy state inconsistent (free slot out of range)");
    return DSA_OK;
}

int dsa_pol_set_shape(dsa_pol h, int shape)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid policy handle");
    const int nshapes = 2 * (dsa_pol_k::kMaxNbuf - 1);
    if (shape < 0 || shape > nshapes)
        return fail(DSA_ERR_ARG, "shape must be 0 (automatic) or 1 .. %d (got %d)", nshapes, shape);
    if (shape == 0) {
        if (!auto_shape(h)) return fail(DSA_ERR_CUDA, "no launch shape for this handle");
        return DSA_OK;
    }
    const int sh = (shape - 1) % 2, nb = 2 + (shape - 1) / 2;
    const int ctas = shape_ctas(h, sh, nb);
    if (ctas < 1) return fail(DSA_ERR_ARG, "launch shape %d cannot be launched for this handle", shape);
    apply_shape(h, sh, nb, ctas);
    return DSA_OK;
}

int dsa_pol_set_wait_limit(dsa_pol h, uint32_t limit)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid policy handle");
    h->wait_limit = limit;
    return DSA_OK;
}

}  // extern "C"
