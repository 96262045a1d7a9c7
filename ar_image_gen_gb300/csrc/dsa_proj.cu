// dsa_proj.cu -- QKV projection with rotary position embedding on the
// tensor cores, feeding a decode step ("Understanding and Exploiting Diagonal
// Attention Sparsity in Autoregressive Image Generation", section 2,
// "LLM-aligned decoding behavior", and section 5.3, Fig. 16(b)).  C ABI in
// include/dsa_proj.h.
//
// One launch computes Y^T = W x^T for one decode step: the 3 H d output
// features are the MMA's M dimension (tiles of 128, each one head's q, k or v
// at head_dim 128, two heads at 64) and the batch is its N dimension (padded
// to a multiple of 16), so a batch of a few dozen tokens still fills the
// 128-row tensor-core tile.  At decode batch sizes the launch streams W once
// from HBM (2 bytes per weight against 2 B flops), so it is bound by HBM,
// not by the tensor cores; what matters is keeping every SM's copies in
// flight.  The work (tiles x k-blocks of 64) is divided evenly over a
// persistent grid of one CTA per SM (stream-K): a CTA takes a contiguous run
// of k-blocks, which may end inside one tile and begin inside another.  A
// tile finished by one CTA is written directly; a tile shared by several
// CTAs is summed by the CTA that holds the tile's first k-block (for which
// it is the last piece of its run): the others write fp32 partials and
// count themselves done on the tile's counter, and that CTA waits for the
// count, adds the partials in k order (deterministic) and writes the tile.
//
// CTA of 10 warps: warp 0 issues the TMA loads of W and x tiles (128-byte
// swizzle) into a ring of shared-memory stages, warp 1 issues tcgen05.mma
// (M 128, N = padded batch, K 16; fp32 accumulator in tensor memory), warps
// 2-9 drain the accumulator with tcgen05.ld (warp w reads TMEM lanes
// 32 (w % 4) ..; two warps per lane quarter split the batch columns),
// apply RoPE (a head's halves meet through a warp shuffle) and store bf16.  Every mbarrier wait is bounded; a wait that gives
// up sets a status bit and the CTA drains its copies and MMAs and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include "../../include/dsa.h"
#include "../../include/dsa_proj.h"
#include "dsa_decode.cuh"
#include "dsa_internal.h"
#include "dsa_tc.cuh"

namespace dsa_proj_k {

using namespace dsa;

constexpr int kThreads = 320;  // producer warp, MMA warp, 8 epilogue warps
constexpr int kBM = 128;       // output features per tile
constexpr int kBK = 64;        // hidden elements per k-block (one 128-byte swizzled row)
constexpr int kUK = 16;        // K of one tcgen05.mma kind::f16
constexpr int kATile = kBM * kBK * 2;
constexpr int kMaxBatch = 256;
constexpr int kEpiThreads = 256;   // the epilogue warps
constexpr int kGroupThreads = 128; // one column group of epilogue warps (one warp per TMEM lane quarter)
constexpr int kXchBytes = 2 * 32 * kBM * 2;  // per group: 32 columns x 128 features of bf16
constexpr uint32_t kEpiBar = 1;    // all epilogue warps
constexpr uint32_t kGroupBar0 = 2; // column groups 0 and 1: barriers 2 and 3
constexpr int kExtraBars = 4;            // acc_full, acc_empty, drain, red_full
constexpr uint32_t kBulkPiece = 32768;  // bytes per bulk copy of a partial

struct ProjParams {
    // Row of stream s = b * H + h of q, k, v: q + s * D, k + s * kstride,
    // v + s * vstride elements (a stride of D: [B, HD] tensors; the fused
    // decode step points k and v at the decode state's slot of the newest
    // token instead).  With kinv / vinv set, k and v are stored as E4M3 codes
    // (one byte each) of fp32(value) * inv[s] instead of bf16.
    __nv_bfloat16 *q, *k, *v;
    int kstride, vstride;
    const float *kinv, *vinv;
    float *part;               // [grid][npad / 16][4][128] float4 partials of shared tiles
    int *counters;             // [tiles] published pieces per shared tile
    int *status;
    int B, H, npad, HD, D, tiles, kblocks, stages, tmem_cols;
    int pos;
    uint32_t wait_limit;
    double inv_freq[64];       // 10000^(-2j/D), j < D/2
};

// Work units (tile, k-block) are numbered u = tile * kblocks + kb.  CTA c of
// the G in the grid takes the run of units [start(c), start(c + 1)) with
// start(c) = c U / G (the host keeps U * G below 2^31).
__device__ __forceinline__ int run_start(int c, int U, int G) { return (int)((unsigned)c * (unsigned)U / (unsigned)G); }

// The CTA whose run holds unit u: the largest c with start(c) <= u.
__device__ __forceinline__ int owner(int u, int U, int G) { return (int)(((unsigned)(u + 1) * G + U - 1) / U) - 1; }

// One piece of a CTA's run: k-blocks [kb0, kb1) of `tile`, and the CTAs
// whose runs share the tile (first, count; `first` holds k-block 0, the
// others follow in k order).  A run's pieces after its first start at a tile
// boundary, so a shared tile consists of a head (k-block 0), which is the
// LAST piece of its CTA's run, and pieces that are each the FIRST piece of a
// later CTA's run: every CTA publishes at most one partial (slot c), and the
// head's CTA, which reaches the tile at the end of its run, sums them.
struct Seg {
    int tile, kb0, kb1;
    int first, nseg;
};

__device__ __forceinline__ Seg make_seg(int u, int u1, int kblocks, int U, int G)
{
    Seg s;
    s.tile = u / kblocks;
    s.kb0 = u - s.tile * kblocks;
    const int tile_end = (s.tile + 1) * kblocks;
    s.kb1 = (u1 < tile_end ? u1 : tile_end) - s.tile * kblocks;
    s.first = owner(s.tile * kblocks, U, G);
    s.nseg = owner(tile_end - 1, U, G) - s.first + 1;
    return s;
}

__device__ __forceinline__ void set_status(int *status, int bit) { atomicOr(status, bit); }

__device__ __forceinline__ int ld_acquire(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Orders this thread's earlier generic-proxy view of global memory (the
// acquire above) before its later bulk copies read global memory.
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

// Two floats rounded to bf16 (nearest even), low half first.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// y[4i .. 4i + 3] += v
__device__ __forceinline__ void add4(float (&y)[32], int i, const float4 &v)
{
    y[4 * i] += v.x;
    y[4 * i + 1] += v.y;
    y[4 * i + 2] += v.z;
    y[4 * i + 3] += v.w;
}

// Bounded wait for a barrier phase by polling (no suspend hint): the
// producer and MMA threads are alone on their warps and each hand-off sits
// on the launch's critical path.  Gives up after `limit` polls or about one
// second (limit 0: at once).
__device__ __forceinline__ bool wait_spin(uint32_t bar, uint32_t parity, uint32_t limit)
{
    if (limit == 0) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1; i < limit; ++i) {
        if ((i & 255u) == 0 && globaltimer_ns() - t0 > kWaitNs) return false;
        if (mbar_try_wait(bar, parity)) return true;
    }
    return false;
}

// Bounded wait until the counter reaches `want` (the other pieces of a
// shared tile have published their partials).
__device__ __forceinline__ bool wait_count(const int *ctr, int want, uint32_t limit)
{
    if (limit == 0) return false;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < limit; ++i) {
        if (ld_acquire(ctr) >= want) return true;
        if ((i & 63u) == 63u && globaltimer_ns() - t0 > kWaitNs) return false;
        __nanosleep(64);
    }
    return false;
}

// cos and sin of pos * inv_freq: the angle in fp64, reduced by 2 pi in two
// parts (Cody and Waite), then the fp32 functions on |r| <= pi.
__device__ __forceinline__ void rope_cs(int pos, double inv_freq, float &c, float &s)
{
    const double two_pi_hi = 6.283185307179586;      // nearest double to 2 pi
    const double two_pi_lo = 2.4492935982947064e-16;  // 2 pi - two_pi_hi
    const double a = (double)pos * inv_freq;
    const double n = rint(a * (1.0 / two_pi_hi));
    double r = fma(-n, two_pi_hi, a);
    r = fma(-n, two_pi_lo, r);
    sincosf((float)r, &s, &c);
}

// RoPE (q and k tiles) and bf16 store of `ncol` (16 or 32) accumulator
// columns c0 .. c0 + ncol - 1 (batch rows) of the tile; y[j] is this
// thread's value for feature f of the tile and column c0 + j.  A feature's
// RoPE partner (f +- D/2) sits 8 lanes away in the same warp (the W rows
// reach the tile interleaved, see the W tensor map), so the rotation needs
// one shuffle per value.  Through the group's `xch` ([32][128] bf16) the
// tile is then turned so that each thread stores 8 consecutive features of
// one row as one 16-byte vector.  The 128 threads of one epilogue group
// (gt = 0..127, named barrier `bar`) call it together.
__device__ __forceinline__ void finish_cols(float (&y)[32], int ncol, int c0, int f, int gt, uint32_t bar, bool rope,
                                            bool upper, float cs, float sn, __nv_bfloat16 *xch, __nv_bfloat16 *base,
                                            int stride, int f0, const float *inv, const ProjParams &p)
{
    if (rope) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j < ncol) {
                const float o = __shfl_xor_sync(0xffffffffu, y[j], 8);
                y[j] = upper ? fmaf(o, sn, y[j] * cs) : fmaf(-o, sn, y[j] * cs);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (j < ncol) xch[j * kBM + f] = __float2bfloat16_rn(y[j]);
    named_bar_sync(bar, kGroupThreads);
    const int g = gt & 15, r = gt >> 4;  // 8 features [8 g, 8 g + 8) of rows r, r + 8, ...
    const int fe = f0 + 8 * g;            // feature fe of token b: element fe % D of stream b * H + fe / D
    const size_t off = (size_t)(fe / p.D) * stride + fe % p.D;
    for (int j = r; j < ncol; j += 8) {
        const int b = c0 + j;
        if (b >= p.B) continue;
        const uint4 x = *reinterpret_cast<const uint4 *>(xch + j * kBM + 8 * g);
        if (inv) {  // E4M3 codes of the bf16 values, as the decode state stores them
            const size_t sidx = (size_t)b * p.H + fe / p.D;
            *reinterpret_cast<uint2 *>(reinterpret_cast<unsigned char *>(base) + (size_t)b * p.H * stride + off) =
                e4m3_codes(x, __ldg(inv + sidx));
        } else {
            *reinterpret_cast<uint4 *>(base + (size_t)b * p.H * stride + off) = x;
        }
    }
    named_bar_sync(bar, kGroupThreads);  // xch is rewritten by the next call
}

// Drains columns [cb, ce) of this thread's accumulator lane, 32 columns at a
// time (16 for an odd last chunk): fn(y, ncol, c0, last) with y[0 .. ncol)
// the fp32 values of columns c0 .. c0 + ncol - 1; `last` marks the final
// chunk, whose load is this thread's last use of the accumulator.  cb and ce
// are multiples of 16; an empty range calls nothing.
template <typename Fn>
__device__ __forceinline__ void drain_lane(uint32_t trow, int cb, int ce, Fn &&fn)
{
    for (int c0 = cb; c0 < ce; c0 += 32) {
        const int ncol = ce - c0 >= 32 ? 32 : 16;
        float y[32];
        if (ncol == 32)
            tmem_ld32(trow + (uint32_t)c0, y);
        else
            tmem_ld16(trow + (uint32_t)c0, *reinterpret_cast<float(*)[16]>(&y[0]));
        fn(y, ncol, c0, c0 + ncol >= ce);
    }
}

// The eight epilogue warps (threads 64..319), two per TMEM lane quarter: the
// warps of group 0 (2..5) take the first half of the batch columns, those of
// group 1 (6..9) the rest.  Per piece of the CTA's run: drain the
// accumulator from tensor memory and write the output tile; for a tile
// shared by several CTAs, every piece but the head (k-block 0) publishes an
// fp32 partial, and the head's CTA, for which the head is the last piece of
// its run (so its stage memory is idle), waits until the others are out,
// fetches them with bulk copies and adds all pieces in k order, its own
// straight from tensor memory.  Every branch below is uniform over the 256
// threads (decisions go through shared flags and the all-epilogue barrier).
__device__ __forceinline__ void epilogue(const ProjParams &p, int c, int U, int G, int u0, int u1, uint32_t tmem,
                                         uint32_t acc_full, uint32_t acc_empty, uint32_t red_full,
                                         const unsigned char *smem, uint32_t sbase, uint32_t stage_bytes, int *flags,
                                         __nv_bfloat16 *xch_base)
{
    const int et = threadIdx.x - 64;  // 0..255
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qw = warp & 3;          // the TMEM lane quarter this warp may read
    const int grp = et >> 7;          // column group
    const int gt = et & 127;          // thread within the group
    const uint32_t gbar = kGroupBar0 + grp;
    __nv_bfloat16 *xch = xch_base + grp * 32 * kBM;
    const int L = qw * 32 + lane;     // accumulator row = TMEM lane
    const int rem = L % p.D;
    const bool upper = (rem >> 3) & 1;                   // lane L holds the upper half of its head
    const int jr = (rem >> 4) * 8 + (L & 7);             // rotation index within the half
    const int f = L - rem + (upper ? p.D / 2 : 0) + jr;  // feature within the tile
    const uint32_t trow = tmem + ((uint32_t)(qw * 32) << 16);
    const int split = ((p.npad / 16 + 1) / 2) * 16;      // group 0: columns [0, split), group 1: [split, npad)
    const int cb = grp == 0 ? 0 : split, ce = grp == 0 ? split : p.npad;
    const uint32_t pbytes = (uint32_t)p.npad * kBM * 4;   // one partial
    const size_t pslot = (size_t)(p.npad / 16) * 4 * kBM;  // float4s per partial slot
    float4 *const part4 = reinterpret_cast<float4 *>(p.part);
    uint32_t aph = 0;
    bool red_armed = false;
    int nseen = 0;
    for (int u = u0; u < u1; ++nseen) {
        const Seg sg = make_seg(u, u1, p.kblocks, U, G);
        u += sg.kb1 - sg.kb0;
        const int part = sg.tile * kBM / p.HD;
        const int f0 = sg.tile * kBM - part * p.HD;
        const bool rope = part < 2;
        __nv_bfloat16 *const dbase = part == 0 ? p.q : (part == 1 ? p.k : p.v);
        const int dstride = part == 0 ? p.D : (part == 1 ? p.kstride : p.vstride);
        const float *dinv = part == 0 ? nullptr : (part == 1 ? p.kinv : p.vinv);
        float cs = 1.f, sn = 0.f;
        if (rope) rope_cs(p.pos, p.inv_freq[jr], cs, sn);
        // One thread waits; the others learn the outcome at the barrier.
        if (et == 0) flags[nseen & 1] = wait_spin(acc_full, aph, p.wait_limit) ? 1 : 0;
        named_bar_sync(kEpiBar, kEpiThreads);
        if (!flags[nseen & 1]) {
            if (et == 0) set_status(p.status, ST_TIMEOUT);
            break;
        }
        tc_fence_after();
        aph ^= 1u;
        if (cb >= ce) {  // a group without columns (batch <= 16) is done with the accumulator at once
            tc_fence_before();
            mbar_arrive(acc_empty);
        }
        if (sg.nseg > 1 && sg.kb0 > 0) {
            // Not the head (so the first piece of this run): publish the
            // partial in slot c, laid out [16-column chunk][4][128 lanes] of
            // float4 so that stores and the head's reads are contiguous per warp.
            float4 *out4 = part4 + (size_t)c * pslot + L;
            drain_lane(trow, cb, ce, [&](float(&y)[32], int ncol, int c0, bool last) {
                if (last) {
                    tc_fence_before();
                    mbar_arrive(acc_empty);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (4 * i < ncol)
                        __stcg(out4 + (size_t)(c0 / 4 + i) * kBM,
                               make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]));
            });
            named_bar_sync(kEpiBar, kEpiThreads);  // every store of the partial issued
            if (et == 0) {
                __threadfence();
                atomicAdd(p.counters + sg.tile, 1);
            }
            continue;
        }
        const int nother = sg.nseg - 1;  // published pieces to add (0: an unshared tile)
        const bool bulk = nother > 0 && (uint64_t)nother * pbytes <= (uint64_t)p.stages * stage_bytes;
        if (nother > 0) {
            if (et == 0) {
                int ok = wait_count(p.counters + sg.tile, nother, p.wait_limit) ? 1 : 0;
                if (ok && bulk) {
                    // The head is the last piece of this run: every MMA of the
                    // run is done and the stage memory is idle.
                    fence_proxy_async_all();
                    mbar_arrive_expect_tx(red_full, (uint32_t)nother * pbytes);
                    for (int jj = 0; jj < nother; ++jj) {
                        const unsigned char *src =
                            reinterpret_cast<const unsigned char *>(part4 + (size_t)(sg.first + 1 + jj) * pslot);
                        for (uint32_t off = 0; off < pbytes; off += kBulkPiece) {
                            const uint32_t n = pbytes - off < kBulkPiece ? pbytes - off : kBulkPiece;
                            bulk_g2s(sbase + (uint32_t)jj * pbytes + off, src + off, n, red_full);
                        }
                    }
                    red_armed = true;
                    ok = wait_spin(red_full, 0, p.wait_limit) ? 1 : 0;
                }
                flags[2] = ok;
            }
            named_bar_sync(kEpiBar, kEpiThreads);
            if (!flags[2]) {
                if (et == 0) set_status(p.status, ST_TIMEOUT);
                break;
            }
            if (bulk) (void)mbar_try_wait(red_full, 0);  // completed: makes the copied bytes visible here too
        }
        drain_lane(trow, cb, ce, [&](float(&y)[32], int ncol, int c0, bool last) {
            if (last) {
                tc_fence_before();
                mbar_arrive(acc_empty);
            }
            for (int jj = 0; jj < nother; ++jj) {  // the other pieces, in k order after the head
                float4 v[8];
                if (bulk) {
                    const float4 *src =
                        reinterpret_cast<const float4 *>(smem + (size_t)jj * pbytes) + (size_t)(c0 / 4) * kBM + L;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (4 * i < ncol) v[i] = src[i * kBM];
                } else {
                    const float4 *src = part4 + (size_t)(sg.first + 1 + jj) * pslot + (size_t)(c0 / 4) * kBM + L;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (4 * i < ncol) v[i] = __ldcg(src + i * kBM);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (4 * i < ncol) add4(y, i, v[i]);
            }
            finish_cols(y, ncol, c0, f, gt, gbar, rope, upper, cs, sn, xch, dbase, dstride, f0, dinv, p);
        });
        named_bar_sync(kEpiBar, kEpiThreads);  // both groups are done with this piece
        if (nother > 0 && et == 0) atomicExch(p.counters + sg.tile, 0);
    }
    if (red_armed) drain_phase(red_full, 0);  // (et == 0 only) the copies have landed before exit
}

__global__ void __launch_bounds__(kThreads, 1)
    qkv_rope_kernel(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapX,
                    const ProjParams p)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;  // 128-byte swizzled tiles need 1024-byte alignment
    unsigned char *smem = smem_raw + (sbase - raw);
    const uint32_t stage_bytes = kATile + (uint32_t)p.npad * kBK * 2;
    const uint32_t off_bar = (uint32_t)p.stages * stage_bytes;
    const uint32_t bar0 = sbase + off_bar;           // full[s] at bar0 + 8 s, empty[s] at bar0 + 8 (stages + s)
    const uint32_t acc_full = bar0 + 16u * p.stages;
    const uint32_t acc_empty = acc_full + 8u;
    const uint32_t drain = acc_full + 16u;
    const uint32_t red_full = acc_full + 24u;       // partials of a shared tile landed in the stage memory
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + off_bar + 8u * (2 * p.stages + kExtraBars));
    // flags[0], [1]: accumulator ready (alternating); [2]: partials published; [3]: partials landed
    int *flags = reinterpret_cast<int *>(tmem_slot + 1);
    __nv_bfloat16 *xch = reinterpret_cast<__nv_bfloat16 *>(smem + ((off_bar + 8u * (2 * p.stages + kExtraBars) + 32u + 15u) & ~15u));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int U = p.tiles * p.kblocks;
    const int u0 = run_start(c, U, G), u1 = run_start(c + 1, U, G);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(bar0 + 8u * s, 1);                // one expect_tx arrival + the TMA bytes
            mbar_init(bar0 + 8u * (p.stages + s), 1);   // one MMA commit
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kEpiThreads);
        mbar_init(drain, 1);
        mbar_init(red_full, 1);
        fence_barrier_init();
        prefetch_tmap(&mapW);
        prefetch_tmap(&mapX);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int issued = 0;  // k-blocks whose copies warp 0 issued

    // Programmatic dependent launch: this grid may start while the previous
    // kernel in the stream finishes.  W is never written by the kernels
    // around it, so warp 0 starts streaming it at once; x, the outputs, the
    // partials and the counters are touched only after the wait (every
    // thread waits for itself), and then the next grid may start its CTAs.
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();  // W is read once per launch
            const int total = u1 - u0;
            const int pre = total < p.stages ? total : p.stages;
            for (int i = 0; i < pre; ++i) {  // first use of stages 0 .. pre - 1: nothing to wait for
                const int u = u0 + i, tile = u / p.kblocks, kb = u - tile * p.kblocks;
                mbar_arrive_expect_tx(bar0 + 8u * i, stage_bytes);
                tma_load_5d_hint(sbase + (uint32_t)i * stage_bytes, &mapW, kb * kBK, 0, 0, 0, tile * (kBM / p.D), bar0 + 8u * i, pol);
            }
            pdl_wait();
            pdl_launch_dependents();
            for (int i = 0; i < pre; ++i) {
                const int kb = (u0 + i) % p.kblocks;
                tma_load_2d(sbase + (uint32_t)i * stage_bytes + kATile, &mapX, kb * kBK, 0, bar0 + 8u * i);
            }
            issued = pre;
            for (int i = pre; i < total; ++i) {
                const uint32_t s = (uint32_t)(i % p.stages), ph = (uint32_t)((i / p.stages) & 1);
                if (!wait_spin(bar0 + 8u * (p.stages + s), ph ^ 1u, p.wait_limit)) {
                    set_status(p.status, ST_TIMEOUT);
                    break;
                }
                const int u = u0 + i, tile = u / p.kblocks, kb = u - tile * p.kblocks;
                const uint32_t a = sbase + s * stage_bytes;
                mbar_arrive_expect_tx(bar0 + 8u * s, stage_bytes);
                tma_load_5d_hint(a, &mapW, kb * kBK, 0, 0, 0, tile * (kBM / p.D), bar0 + 8u * s, pol);
                tma_load_2d(a + kATile, &mapX, kb * kBK, 0, bar0 + 8u * s);
                ++issued;
            }
        } else {
            pdl_wait();
            pdl_launch_dependents();
        }
        __syncwarp();
    } else if (warp == 1) {
        pdl_wait();
        pdl_launch_dependents();
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kBM, p.npad);
            uint32_t s = 0, ph = 0, aph = 0;
            bool ok = true;
            for (int u = u0; u < u1 && ok;) {
                const Seg sg = make_seg(u, u1, p.kblocks, U, G);
                if (!wait_spin(acc_empty, aph ^ 1u, p.wait_limit)) {
                    set_status(p.status, ST_TIMEOUT);
                    break;
                }
                tc_fence_after();
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!wait_spin(bar0 + 8u * s, ph, p.wait_limit)) {
                        set_status(p.status, ST_TIMEOUT);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = sbase + s * stage_bytes;
                    const uint64_t ad = sw128_kmajor_desc(a), bd = sw128_kmajor_desc(a + kATile);
#pragma unroll
                    for (int k = 0; k < kBK / kUK; ++k)
                        umma_bf16(tmem, ad + 2u * k, bd + 2u * k, idesc, (kb > sg.kb0 || k > 0) ? 1u : 0u);
                    umma_commit(bar0 + 8u * (p.stages + s));  // stage s free once these MMAs are done
                    if (++s == (uint32_t)p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(acc_full);
                aph ^= 1u;
                u += sg.kb1 - sg.kb0;
            }
        }
        __syncwarp();
    } else {
        pdl_wait();
        pdl_launch_dependents();
        epilogue(p, c, U, G, u0, u1, tmem, acc_full, acc_empty, red_full, smem, sbase, stage_bytes, flags, xch);
    }

    __syncthreads();
    if (warp == 0 && lane == 0) {
        // Every copy issued has landed before the CTA's shared memory goes.
        for (int s = 0; s < p.stages && s < issued; ++s) {
            const int armed = (issued - 1 - s) / p.stages + 1;
            drain_phase(bar0 + 8u * s, (uint32_t)((armed - 1) & 1));
        }
    }
    if (warp == 1 && lane == 0) {
        // Every MMA issued has completed before the tensor memory is freed.
        umma_commit(drain);
        drain_phase(drain, 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
    }
}

}  // namespace dsa_proj_k

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
using dsa_detail::cuda_fail;
using dsa_detail::dev_alloc;
using dsa_detail::fail;

namespace {

constexpr uint32_t kProjMagic = 0x44535051u;  // "DSPQ"
constexpr size_t kSmemLimit = 227 * 1024;     // dynamic shared memory per CTA on sm_103
constexpr int kMaxStages = 8;

// Shared-memory bytes of the kernel's layout (see qkv_rope_kernel) for
// `stages` stages of `stage_bytes`, plus 1024 bytes of alignment slack.
size_t proj_smem(int stages, size_t stage_bytes)
{
    const size_t off_bar = (size_t)stages * stage_bytes;
    const size_t off_xch = (off_bar + 8 * (2 * (size_t)stages + dsa_proj_k::kExtraBars) + 32 + 15) & ~(size_t)15;
    return 1024 + off_xch + dsa_proj_k::kXchBytes;
}

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void **)&encode, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess) encode = nullptr;
    }
    return encode;
}

// Row-major bf16 matrix [rows, cols] seen by TMA in boxes of 64 columns x
// box_rows rows with 128-byte swizzling (the operand layout of the MMA
// descriptors).  Rows past the end read as zero.
int encode_operand(CUtensorMap *map, const void *base, int rows, int cols, int box_rows, bool stream_once)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
    if (!encode) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)dsa_proj_k::kBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        stream_once ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return DSA_OK;
}

// W [3 H D, hidden] seen by TMA as a 5-D tensor whose box is one 128-row
// tile of 64 columns with the two halves of each head interleaved in blocks
// of 8 rows: dimensions (column, row r < 8, half h < 2, block k < D/16,
// group of D rows), row = D group + (D/2) h + 8 k + r, box (64, 8, 2, D/16,
// 128/D).  The box lands in shared memory in the order r, h, k, group, so
// tile row (= MMA row = TMEM lane) 16 k + 8 h + r of a head holds feature
// (D/2) h + 8 k + r, and every feature's rotary partner is 8 lanes away.
int encode_w_interleaved(CUtensorMap *map, const void *W, int HD, int D, int hidden)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
    if (!encode) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t row = (cuuint64_t)hidden * 2;
    const cuuint64_t dims[5] = {(cuuint64_t)hidden, 8, 2, (cuuint64_t)(D / 16), (cuuint64_t)(3 * HD / D)};
    const cuuint64_t strides[4] = {row, row * (D / 2), row * 8, row * D};
    const cuuint32_t box[5] = {(cuuint32_t)dsa_proj_k::kBK, 8, 2, (cuuint32_t)(D / 16), (cuuint32_t)(dsa_proj_k::kBM / D)};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(W), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled (W) failed (%d)", (int)r);
    return DSA_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

struct dsa_proj_ctx {
    uint32_t magic;
    int B, H, D, hidden, HD, npad, tiles, kblocks, grid, stages, tmem_cols;
    size_t smem;
    float *part;
    int *counters;
    int *status;
    __nv_bfloat16 *staging;  // [B * HD]: q of dsa_decode_step_fused (k and v go to the decode state)
    uint32_t wait_limit;
    double inv_freq[64];
};

namespace {

bool valid(const dsa_proj_ctx *p) { return p != nullptr && p->magic == kProjMagic; }

void free_proj(dsa_proj_ctx *p)
{
    if (!p) return;
    cudaFree(p->part);
    cudaFree(p->counters);
    cudaFree(p->status);
    cudaFree(p->staging);
    p->magic = 0;
    delete p;
}

}  // namespace

namespace dsa_detail {

int proj_shape(const dsa_proj_ctx *p, int *batch, int *heads, int *head_dim)
{
    if (!valid(p)) return fail(DSA_ERR_STATE, "invalid projection context");
    *batch = p->B;
    *heads = p->H;
    *head_dim = p->D;
    return DSA_OK;
}

void proj_staging(const dsa_proj_ctx *p, void **q) { *q = p->staging; }

int proj_launch(dsa_proj_ctx *pr, const void *x, const void *W, int pos, void *q, void *k, void *v, cudaStream_t st,
                int kstride, int vstride, const float *kinv, const float *vinv)
{
    if (!valid(pr)) return fail(DSA_ERR_STATE, "invalid projection context");
    if (!x || !W || !q || !k || !v) return fail(DSA_ERR_ARG, "x, W, q, k and v must be non-NULL");
    if (!aligned16(x) || !aligned16(W) || !aligned16(q) || !aligned16(k) || !aligned16(v))
        return fail(DSA_ERR_ARG, "x, W, q, k and v must be 16-byte aligned");
    if (pos < 0) return fail(DSA_ERR_ARG, "pos must be >= 0 (got %d)", pos);
    CUtensorMap mapW, mapX;
    int rc = encode_w_interleaved(&mapW, W, pr->HD, pr->D, pr->hidden);
    if (rc == DSA_OK) rc = encode_operand(&mapX, x, pr->B, pr->hidden, pr->npad, false);
    if (rc != DSA_OK) return rc;

    dsa_proj_k::ProjParams p;
    p.q = static_cast<__nv_bfloat16 *>(q);
    p.k = static_cast<__nv_bfloat16 *>(k);
    p.v = static_cast<__nv_bfloat16 *>(v);
    p.kstride = kstride > 0 ? kstride : pr->D;
    p.vstride = vstride > 0 ? vstride : pr->D;
    p.kinv = kinv;
    p.vinv = vinv;
    p.H = pr->H;
    p.part = pr->part;
    p.counters = pr->counters;
    p.status = pr->status;
    p.B = pr->B;
    p.npad = pr->npad;
    p.HD = pr->HD;
    p.D = pr->D;
    p.tiles = pr->tiles;
    p.kblocks = pr->kblocks;
    p.stages = pr->stages;
    p.tmem_cols = pr->tmem_cols;
    p.pos = pos;
    p.wait_limit = pr->wait_limit;
    std::memcpy(p.inv_freq, pr->inv_freq, sizeof p.inv_freq);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pr->grid);
    cfg.blockDim = dim3(dsa_proj_k::kThreads);
    cfg.dynamicSmemBytes = pr->smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, dsa_proj_k::qkv_rope_kernel, mapW, mapX, p);
    if (e != cudaSuccess) return cuda_fail(e, "projection launch");
    return DSA_OK;
}

}  // namespace dsa_detail

extern "C" {

int dsa_proj_create(int batch, int heads, int head_dim, int hidden, dsa_proj *out)
{
    if (!out) return fail(DSA_ERR_ARG, "out is NULL");
    *out = nullptr;
    if (batch < 1 || batch > dsa_proj_k::kMaxBatch)
        return fail(DSA_ERR_ARG, "batch must be in [1, %d] (got %d)", dsa_proj_k::kMaxBatch, batch);
    if (heads < 1) return fail(DSA_ERR_ARG, "heads must be >= 1 (got %d)", heads);
    if (head_dim != 64 && head_dim != 128) return fail(DSA_ERR_ARG, "head_dim must be 64 or 128 (got %d)", head_dim);
    if ((long long)heads * head_dim % dsa_proj_k::kBM != 0)
        return fail(DSA_ERR_ARG, "heads * head_dim must be a multiple of 128 (got %d x %d)", heads, head_dim);
    if ((long long)3 * heads * head_dim > INT_MAX / 2) return fail(DSA_ERR_ARG, "heads * head_dim too large");
    if (hidden < dsa_proj_k::kBK || hidden % dsa_proj_k::kBK != 0)
        return fail(DSA_ERR_ARG, "hidden must be a positive multiple of 64 (got %d)", hidden);

    dsa_proj_ctx *p = new (std::nothrow) dsa_proj_ctx();
    if (!p) return fail(DSA_ERR_OOM, "host allocation failed");
    p->magic = kProjMagic;
    p->B = batch;
    p->H = heads;
    p->D = head_dim;
    p->hidden = hidden;
    p->HD = heads * head_dim;
    p->npad = (batch + 15) / 16 * 16;
    p->tiles = 3 * p->HD / dsa_proj_k::kBM;
    p->kblocks = hidden / dsa_proj_k::kBK;
    p->tmem_cols = p->npad <= 32 ? 32 : (p->npad <= 64 ? 64 : (p->npad <= 128 ? 128 : 256));
    p->wait_limit = 0xffffffffu;
    for (int j = 0; j < head_dim / 2; ++j) p->inv_freq[j] = std::pow(10000.0, -2.0 * j / head_dim);

    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        free_proj(p);
        return cuda_fail(e, "device query");
    }
    const size_t stage_bytes = (size_t)dsa_proj_k::kATile + (size_t)p->npad * dsa_proj_k::kBK * 2;
    p->stages = kMaxStages;
    while (p->stages > 2 && proj_smem(p->stages, stage_bytes) > kSmemLimit) --p->stages;
    p->smem = proj_smem(p->stages, stage_bytes);
    const long long units = (long long)p->tiles * p->kblocks;
    p->grid = (int)(units < sms ? units : sms);
    if (units * (p->grid + 1) > INT_MAX) {
        free_proj(p);
        return fail(DSA_ERR_ARG, "3 * heads * head_dim / 128 x hidden / 64 work units too many for this device");
    }
    e = cudaFuncSetAttribute(dsa_proj_k::qkv_rope_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p->smem);
    if (e != cudaSuccess) {
        free_proj(p);
        return cuda_fail(e, "projection kernel attribute (is this an sm_103 device?)");
    }

    const size_t n = (size_t)batch * p->HD;
    int rc = dev_alloc((void **)&p->part, sizeof(float) * (size_t)p->grid * p->npad * dsa_proj_k::kBM,
                       "projection partials");
    if (rc == DSA_OK) rc = dev_alloc((void **)&p->counters, sizeof(int) * (size_t)p->tiles, "projection counters");
    if (rc == DSA_OK) rc = dev_alloc((void **)&p->status, 16, "projection status");
    if (rc == DSA_OK) rc = dev_alloc((void **)&p->staging, sizeof(__nv_bfloat16) * n, "q staging");
    if (rc != DSA_OK) {
        free_proj(p);  // keeps the allocation's error message
        return rc;
    }
    if ((e = cudaMemset(p->counters, 0, sizeof(int) * (size_t)p->tiles)) != cudaSuccess ||
        (e = cudaMemset(p->status, 0, 16)) != cudaSuccess) {
        free_proj(p);
        return cuda_fail(e, "cudaMemset");
    }
    *out = p;
    return DSA_OK;
}

int dsa_proj_destroy(dsa_proj p)
{
    if (!p) return DSA_OK;
    if (!valid(p)) return fail(DSA_ERR_STATE, "invalid projection context");
    cudaDeviceSynchronize();
    free_proj(p);
    return DSA_OK;
}

int dsa_qkv_rope(dsa_proj p, const void *x, const void *W, int pos, void *q, void *k, void *v, void *stream)
{
    return dsa_detail::proj_launch(p, x, W, pos, q, k, v, (cudaStream_t)stream);
}

int dsa_proj_sync_status(dsa_proj p, void *stream)
{
    if (!valid(p)) return fail(DSA_ERR_STATE, "invalid projection context");
    cudaStream_t st = (cudaStream_t)stream;
    int word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, p->status, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "status copy");
    if (word == 0) return DSA_OK;
    // A launch that gave up may leave counters of shared tiles part-way.
    if ((e = cudaMemsetAsync(p->counters, 0, sizeof(int) * (size_t)p->tiles, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(p->status, 0, 16, st)) != cudaSuccess || (e = cudaStreamSynchronize(st)) != cudaSuccess)
        return cuda_fail(e, "status reset");
    return fail(DSA_ERR_TIMEOUT, "a bounded wait in the projection kernel gave up");
}

int dsa_proj_set_wait_limit(dsa_proj p, uint32_t limit)
{
    if (!valid(p)) return fail(DSA_ERR_STATE, "invalid projection context");
    p->wait_limit = limit;
    return DSA_OK;
}

}  // extern "C"
