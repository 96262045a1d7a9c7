// dsa_diag.cu -- attention diagnostics of dense decode attention over a
// trace ("Understanding and Exploiting Diagonal Attention Sparsity in
// Autoregressive Image Generation", section 3.4 "Attention Sparsity
// Analysis": Fig. 8 attention mass on prompt / local / middle tokens, Fig. 10
// vertical vs diagonal score-vector similarity).  C ABI in
// include/dsa_diag.h.
//
// Per chunk of heads, three kernels:
//   diag_logits_tc_kernel / diag_logits_kernel   logits z[i][c] = q_i .
//                        key_c / sqrt(d) for every decode query i and every key
//                        c it attends (prompt keys, then decode keys 0..i): for
//                        bf16 traces on the tcgen05 tensor cores (128 x 128
//                        tiles, TMA-staged, fp32 accumulators in tensor memory;
//                        bf16 products are exact), for fp32 traces 32 x 32 tiles
//                        of fp32 FMAs;
//   diag_softmax_kernel  per query: softmax over its keys, the prompt /
//                        local / middle weights, and the decode weights
//                        written back in place;
//   diag_similarity_kernel  per (query distance, query): cosine of the
//                        decode score vectors of queries i and i + d over the
//                        same keys (vertical) and over keys shifted by d
//                        (diagonal).
// Sums over heads and queries go to a few doubles per block (atomics).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <vector>

#include "../../include/dsa.h"
#include "../../include/dsa_diag.h"
#include "dsa_internal.h"
#include "dsa_ptx.cuh"
#include "dsa_tc.cuh"

namespace dsa_diag {

constexpr int kTile = 32;      // queries and keys per logits tile
constexpr int kThreads = 256;  // 32 queries x 8 key groups of 4
constexpr int kWarps = 8;      // per softmax / similarity block

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Logits of query tile [i0, i0 + 32) of head s: W[s][i][c] for every key
// column c < L_p + i + 1 (prompt keys first, then decode keys).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) diag_logits_kernel(const T *__restrict__ Q, const T *__restrict__ Kp,
                                                                const T *__restrict__ Kd, float *__restrict__ W,
                                                                int L_p, int L_dec, float scale)
{
    __shared__ float Qs[kTile][D + 1];
    __shared__ float Kt[D][kTile + 1];  // key tile, transposed
    const int s = blockIdx.y;
    const int i0 = blockIdx.x * kTile;
    const int tid = threadIdx.x;
    const int qi = tid / 8;             // query of the thread within the tile
    const int kk = (tid % 8) * 4;       // first of its four keys within a key tile
    const int ncol = L_p + L_dec;
    const T *Qh = Q + (size_t)s * L_dec * D;
    const T *Kph = Kp + (size_t)s * L_p * D;
    const T *Kdh = Kd + (size_t)s * L_dec * D;
    for (int e = tid; e < kTile * D; e += kThreads) {
        const int r = e / D, c = e % D;
        Qs[r][c] = (i0 + r < L_dec) ? to_f(Qh[(size_t)(i0 + r) * D + c]) : 0.f;
    }
    const int i_last = min(i0 + kTile, L_dec) - 1;
    const int cols = L_p + i_last + 1;  // key columns any query of the tile attends
    float *Wrow = W + ((size_t)s * L_dec + i0 + qi) * ncol;
    for (int c0 = 0; c0 < cols; c0 += kTile) {
        __syncthreads();
        for (int e = tid; e < kTile * D; e += kThreads) {
            const int r = e / D, c = e % D;
            const int col = c0 + r;
            float v = 0.f;
            if (col < cols) v = to_f(col < L_p ? Kph[(size_t)col * D + c] : Kdh[(size_t)(col - L_p) * D + c]);
            Kt[c][r] = v;
        }
        __syncthreads();
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
        for (int c = 0; c < D; ++c) {
            const float q = Qs[qi][c];
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[u] = fmaf(q, Kt[c][kk + u], acc[u]);
        }
        const int i = i0 + qi;
        if (i < L_dec) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int col = c0 + kk + u;
                if (col < L_p + i + 1) Wrow[col] = acc[u] * scale;
            }
        }
    }
}

// Tensor-core logits of bf16 traces: one CTA per (128-query tile, head),
// D[i][c] = sum_k Q[i][k] K[c][k] on tcgen05 (bf16 operands, fp32
// accumulator in tensor memory), 128 key columns at a time.  Q and key tiles
// are staged by TMA from 3-D tensor maps ([head, row, d], boxes of 64
// elements x 128 rows, 128-byte swizzle); rows outside a map read as zeros,
// so a key tile that straddles the prompt and the decoded keys is loaded
// from both maps at the same column offset (prompt rows c0.., decode rows
// c0 - L_p.., negative rows zero) and the two MMA chains accumulate into
// one result.  Thread 0 issues the copies and the MMAs; the four warps
// drain their 32 TMEM lanes (queries) 32 columns at a time and store them,
// turned through shared memory, as whole 128-byte row segments.  Every wait
// is time-capped; a CTA that gives up lets its copies and MMAs finish,
// frees its tensor memory and sets *err.
constexpr int kTcM = 128;        // queries per tile = TMEM lanes
constexpr int kTcN = 128;        // key columns per tile = TMEM columns
constexpr int kTcThreads = 128;  // warp w drains TMEM lanes 32 w .. 32 w + 31
constexpr uint32_t kBox = 128 * 128;  // bytes of one staged box: 128 rows of 64 bf16
constexpr uint64_t kTcWaitNs = 1000000000ull;

__device__ __forceinline__ uint64_t gtimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool wait_capped(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = gtimer_ns();
    while (!dsa::mbar_try_wait(bar, parity))
        if (gtimer_ns() - t0 > kTcWaitNs) return false;
    return true;
}

struct TcParams {
    float *W;      // [S, L_dec, L_p + L_dec] logits of the chunk
    int L_p, L_dec, ncol;
    float scale;   // 1 / sqrt(d)
    int *err;      // set when a wait gave up
};

template <int D>
constexpr size_t tc_smem_bytes()
{
    return 1024 + 3 * (size_t)(D / 64) * kBox + (size_t)4 * 32 * 33 * sizeof(float) + 64;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads) diag_logits_tc_kernel(const __grid_constant__ CUtensorMap mq,
                                                                     const __grid_constant__ CUtensorMap mkp,
                                                                     const __grid_constant__ CUtensorMap mkd,
                                                                     const TcParams p)
{
    using namespace dsa;
    constexpr int NB = D / 64;  // 128-byte boxes along the head dimension
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;  // swizzled tiles need 1024-byte alignment
    const uint32_t sq = sbase, skp = sq + NB * kBox, skd = skp + NB * kBox;
    float *xs = reinterpret_cast<float *>(smem_raw + (skd + NB * kBox - raw));  // [4 warps][32][33]
    unsigned char *tail = reinterpret_cast<unsigned char *>(xs + 4 * 32 * 33);
    uint64_t *bars = reinterpret_cast<uint64_t *>(tail);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tail + 16);
    int *flag = reinterpret_cast<int *>(tail + 24);
    const uint32_t load_bar = smem_u32(&bars[0]), mma_bar = smem_u32(&bars[1]);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s = blockIdx.y, i0 = blockIdx.x * kTcM;
    const int i_last = min(i0 + kTcM, p.L_dec) - 1;
    const int ntiles = (p.L_p + i_last + 1 + kTcN - 1) / kTcN;  // key columns any query of the tile attends
    if (threadIdx.x == 0) {
        mbar_init(load_bar, 1);
        mbar_init(mma_bar, 1);
        fence_barrier_init();
        *flag = 1;
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTcN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    uint32_t lph = 0, mph = 0;
    bool load_out = false, mma_out = false;  // thread 0: copies / MMAs issued and not yet waited for
    auto issue_loads = [&](int c0) {         // the tile's key boxes (and, for the first, the query boxes)
        const bool pre = c0 < p.L_p, dec = c0 + kTcN > p.L_p;
        const uint32_t boxes = (uint32_t)((pre ? NB : 0) + (dec ? NB : 0) + (c0 == 0 ? NB : 0));
        mbar_arrive_expect_tx(load_bar, boxes * kBox);
        for (int b = 0; b < NB; ++b) {
            if (c0 == 0) tma_load_3d(sq + b * kBox, &mq, 64 * b, i0, s, load_bar);
            if (pre) tma_load_3d(skp + b * kBox, &mkp, 64 * b, c0, s, load_bar);
            if (dec) tma_load_3d(skd + b * kBox, &mkd, 64 * b, c0 - p.L_p, s, load_bar);
        }
        load_out = true;
    };
    if (threadIdx.x == 0) issue_loads(0);
    for (int t = 0; t < ntiles; ++t) {
        const int c0 = t * kTcN;
        if (threadIdx.x == 0) {
            bool ok = wait_capped(load_bar, lph);
            if (ok) {
                load_out = false;
                lph ^= 1u;
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(kTcM, kTcN);
                uint32_t acc = 0;
                for (int part = 0; part < 2; ++part) {
                    if (part == 0 ? !(c0 < p.L_p) : !(c0 + kTcN > p.L_p)) continue;
                    const uint32_t sk = part == 0 ? skp : skd;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = (uint32_t)(k / 4) * kBox + (uint32_t)(k % 4) * 32u;
                        umma_bf16(tmem, sw128_kmajor_desc(sq + off), sw128_kmajor_desc(sk + off), idesc, acc);
                        acc = 1;
                    }
                }
                umma_commit(mma_bar);
                mma_out = true;
                ok = wait_capped(mma_bar, mph);  // MMAs done: key boxes free, accumulators ready
                if (ok) {
                    mma_out = false;
                    mph ^= 1u;
                    if (t + 1 < ntiles) issue_loads(c0 + kTcN);  // the next keys land while this tile drains
                }
            }
            if (!ok) *flag = 0;
        }
        __syncthreads();
        if (!*flag) break;
        tc_fence_after();
        // drain: lane l of warp w holds query i0 + 32 w + l; turned through
        // xs so that each row segment is stored by a whole warp
        float *xw = xs + warp * 32 * 33;
        const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
        for (int j0 = 0; j0 < kTcN; j0 += 32) {
            float y[32];
            tmem_ld32(trow + (uint32_t)j0, y);
#pragma unroll
            for (int j = 0; j < 32; ++j) xw[lane * 33 + j] = y[j] * p.scale;
            __syncwarp();
            const int c = c0 + j0 + lane;
            for (int r = 0; r < 32; ++r) {
                const int i = i0 + 32 * warp + r;
                if (i < p.L_dec && c < p.L_p + i + 1)
                    p.W[((size_t)s * p.L_dec + i) * p.ncol + c] = xw[r * 33 + lane];
            }
            __syncwarp();
        }
        tc_fence_before();
        __syncthreads();  // the accumulators are read: the next MMAs may overwrite them
    }
    if (threadIdx.x == 0 && !*flag) {  // let what was issued finish before the memory goes away
        if (mma_out) (void)wait_capped(mma_bar, mph);
        if (load_out) (void)wait_capped(load_bar, lph);
        atomicExch(p.err, 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTcN);
}

// One warp per query: softmax over its L_p + i + 1 logits; the prompt, local
// (the ceil(0.1 (i + 1)) most recent decoded keys) and middle weights; the
// decode weights written back over the logits.  Block sums of the three
// weights go to sums[0..2].
__global__ void __launch_bounds__(32 * kWarps) diag_softmax_kernel(float *__restrict__ W, int S, int L_p, int L_dec,
                                                                   float *__restrict__ step_mass,
                                                                   double *__restrict__ sums)
{
    __shared__ float part[kWarps][3];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kWarps + warp;  // s * L_dec + i
    const int ncol = L_p + L_dec;
    float mp = 0.f, ml = 0.f, mm = 0.f;
    if (row < (long long)S * L_dec) {
        const int i = (int)(row % L_dec);
        float *z = W + row * ncol;
        const int n = L_p + i + 1;
        float m = -INFINITY;
        for (int c = lane; c < n; c += 32) m = fmaxf(m, z[c]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int local_lo = L_p + i + 1 - (i + 1 + 9) / 10;  // first local key column
        float tot = 0.f;
        for (int c = lane; c < n; c += 32) {
            const float e = expf(z[c] - m);
            tot += e;
            if (c < L_p) mp += e;
            else if (c >= local_lo) ml += e;
            else mm += e;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            tot += __shfl_xor_sync(0xffffffffu, tot, o);
            mp += __shfl_xor_sync(0xffffffffu, mp, o);
            ml += __shfl_xor_sync(0xffffffffu, ml, o);
            mm += __shfl_xor_sync(0xffffffffu, mm, o);
        }
        const float inv = 1.f / tot;
        for (int c = L_p + lane; c < n; c += 32) z[c] = expf(z[c] - m) * inv;
        mp *= inv;
        ml *= inv;
        mm *= inv;
        if (lane == 0 && step_mass) {
            step_mass[row * 3 + 0] = mp;
            step_mass[row * 3 + 1] = ml;
            step_mass[row * 3 + 2] = mm;
        }
    }
    if (lane == 0) {
        part[warp][0] = mp;
        part[warp][1] = ml;
        part[warp][2] = mm;
    }
    __syncthreads();
    if (threadIdx.x < 3) {
        double a = 0.0;
        for (int w = 0; w < kWarps; ++w) a += part[w][threadIdx.x];
        atomicAdd(&sums[threadIdx.x], a);
    }
}

// One warp per (query distance k, query i) of head s: block y = s, block
// x covers kWarps queries of one distance.  Adds the vertical and diagonal
// cosines to sums[2k], sums[2k + 1].
__global__ void __launch_bounds__(32 * kWarps) diag_similarity_kernel(const float *__restrict__ W, int L_p, int L_dec,
                                                                      const int *__restrict__ dist, int n_dist,
                                                                      int blocks_per_dist, double *__restrict__ sums)
{
    __shared__ float part[kWarps][2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s = blockIdx.y;
    const int k = blockIdx.x / blocks_per_dist;
    const int i = (blockIdx.x % blocks_per_dist) * kWarps + warp;
    const int ncol = L_p + L_dec;
    float cv = 0.f, cd = 0.f;
    if (k < n_dist) {
        const int d = dist[k];
        if (i + d < L_dec) {
            const float *a = W + ((size_t)s * L_dec + i) * ncol + L_p;
            const float *b = W + ((size_t)s * L_dec + i + d) * ncol + L_p;
            float aa = 0.f, bb = 0.f, bs = 0.f, abv = 0.f, abd = 0.f;
            for (int j = lane; j <= i; j += 32) {
                const float x = a[j], y = b[j], z = b[j + d];
                aa = fmaf(x, x, aa);
                bb = fmaf(y, y, bb);
                bs = fmaf(z, z, bs);
                abv = fmaf(x, y, abv);
                abd = fmaf(x, z, abd);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                aa += __shfl_xor_sync(0xffffffffu, aa, o);
                bb += __shfl_xor_sync(0xffffffffu, bb, o);
                bs += __shfl_xor_sync(0xffffffffu, bs, o);
                abv += __shfl_xor_sync(0xffffffffu, abv, o);
                abd += __shfl_xor_sync(0xffffffffu, abd, o);
            }
            cv = abv * rsqrtf(aa * bb);
            cd = abd * rsqrtf(aa * bs);
        }
    }
    if (lane == 0) {
        part[warp][0] = cv;
        part[warp][1] = cd;
    }
    __syncthreads();
    if (threadIdx.x < 2 && k < n_dist) {
        double a = 0.0;
        for (int w = 0; w < kWarps; ++w) a += part[w][threadIdx.x];
        atomicAdd(&sums[2 * k + threadIdx.x], a);
    }
}

template <typename T, int D>
cudaError_t launch_logits(const void *Q, const void *Kp, const void *Kd, float *W, int S, int L_p, int L_dec,
                          cudaStream_t st)
{
    const dim3 grid((L_dec + kTile - 1) / kTile, S);
    diag_logits_kernel<T, D><<<grid, kThreads, 0, st>>>((const T *)Q, (const T *)Kp, (const T *)Kd, W, L_p, L_dec,
                                                       (float)(1.0 / std::sqrt((double)D)));
    return cudaGetLastError();
}

}  // namespace dsa_diag

namespace {

// [S, rows, D] bf16 seen by TMA in boxes of 64 elements x 128 rows x 1 head,
// 128-byte swizzled (the operand layout of the MMA descriptors); rows
// outside [0, rows) read as zeros.
int encode_rows3d(CUtensorMap *map, const void *base, int S, int rows, int D)
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void **)&encode, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !encode) {
            encode = nullptr;
            return dsa_detail::fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        }
    }
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)S};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)rows * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)dsa_diag::kTcM, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return dsa_detail::fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return DSA_OK;
}

// The tensor-core logits of S heads of bf16 traces into W.
template <int D>
int launch_logits_tc(const void *Q, const void *Kp, const void *Kd, float *W, int S, int L_p, int L_dec, int *err,
                     cudaStream_t st)
{
    using namespace dsa_diag;
    CUtensorMap mq, mkp, mkd;
    int rc = encode_rows3d(&mq, Q, S, L_dec, D);
    if (rc == DSA_OK) rc = encode_rows3d(&mkd, Kd, S, L_dec, D);
    if (rc == DSA_OK) rc = L_p > 0 ? encode_rows3d(&mkp, Kp, S, L_p, D) : (mkp = mkd, DSA_OK);  // unused without a prompt
    if (rc != DSA_OK) return rc;
    const size_t smem = tc_smem_bytes<D>();
    cudaError_t e = cudaFuncSetAttribute(diag_logits_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return dsa_detail::cuda_fail(e, "diagnostic logits kernel attribute");
    TcParams p;
    p.W = W;
    p.L_p = L_p;
    p.L_dec = L_dec;
    p.ncol = L_p + L_dec;
    p.scale = 1.0f / std::sqrt((float)D);
    p.err = err;
    const dim3 grid((unsigned)((L_dec + kTcM - 1) / kTcM), (unsigned)S);
    diag_logits_tc_kernel<D><<<grid, kTcThreads, smem, st>>>(mq, mkp, mkd, p);
    e = cudaGetLastError();
    return e == cudaSuccess ? DSA_OK : dsa_detail::cuda_fail(e, "diagnostic logits launch");
}

}  // namespace

extern "C" int dsa_diag_trace(int heads, int head_dim, int L_p, int L_dec, int dtype, const void *Q, const void *Kp,
                              const void *Kd, int n_dist, const int32_t *dist, float *step_mass, double *mass_mean,
                              double *vertical, double *diagonal, void *stream)
{
    using namespace dsa_diag;
    using dsa_detail::fail;
    if (heads < 1 || (head_dim != 64 && head_dim != 128) || L_p < 0 || L_dec < 1 || n_dist < 0)
        return fail(DSA_ERR_ARG, "dsa_diag_trace: need heads >= 1, head_dim 64 or 128, L_p >= 0, L_dec >= 1, n_dist >= 0");
    if (dtype != DSA_BF16 && dtype != DSA_F32) return fail(DSA_ERR_ARG, "dsa_diag_trace: dtype must be DSA_BF16 or DSA_F32");
    if (!Q || !Kd || (L_p > 0 && !Kp) || !mass_mean || (n_dist > 0 && (!dist || !vertical || !diagonal)))
        return fail(DSA_ERR_ARG, "dsa_diag_trace: NULL pointer");
    if (((uintptr_t)Q | (uintptr_t)Kd | (uintptr_t)(L_p > 0 ? Kp : Q) | (uintptr_t)step_mass) & 15u)
        return fail(DSA_ERR_ARG, "dsa_diag_trace: device pointers must be 16-byte aligned");
    for (int k = 0; k < n_dist; ++k)
        if (dist[k] < 1 || dist[k] >= L_dec)
            return fail(DSA_ERR_ARG, "dsa_diag_trace: distance %d outside [1, L_dec)", dist[k]);
    const size_t per_head = (size_t)L_dec * (size_t)(L_p + L_dec) * sizeof(float);
    const size_t budget = (size_t)1 << 30;
    if (per_head > ((size_t)4 << 30)) return fail(DSA_ERR_ARG, "dsa_diag_trace: L_dec x (L_p + L_dec) too large");
    const int chunk = (int)std::max<size_t>(1, std::min<size_t>((size_t)heads, budget / per_head));
    cudaStream_t st = (cudaStream_t)stream;

    float *W = nullptr;
    double *sums = nullptr;  // [3 + 2 n_dist]
    int *ddist = nullptr;
    int *derr = nullptr;     // set by the tensor-core logits kernel when a wait gave up
    int rc = dsa_detail::dev_alloc((void **)&W, per_head * chunk, "diagnostic weights");
    if (rc == DSA_OK) rc = dsa_detail::dev_alloc((void **)&derr, sizeof(int), "diagnostic status");
    if (rc == DSA_OK) rc = dsa_detail::dev_alloc((void **)&sums, sizeof(double) * (3 + 2 * (size_t)n_dist), "diagnostic sums");
    if (rc == DSA_OK) rc = dsa_detail::dev_alloc((void **)&ddist, sizeof(int) * (size_t)(n_dist > 0 ? n_dist : 1), "distances");
    cudaError_t e = cudaSuccess;
    if (rc == DSA_OK) {
        e = cudaMemsetAsync(sums, 0, sizeof(double) * (3 + 2 * (size_t)n_dist), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(derr, 0, sizeof(int), st);
        if (e == cudaSuccess && n_dist > 0)
            e = cudaMemcpyAsync(ddist, dist, sizeof(int) * n_dist, cudaMemcpyHostToDevice, st);
        const size_t eb = dtype == DSA_F32 ? 4 : 2;
        for (int s0 = 0; s0 < heads && e == cudaSuccess; s0 += chunk) {
            const int S = std::min(chunk, heads - s0);
            const char *q = (const char *)Q + (size_t)s0 * L_dec * head_dim * eb;
            const char *kp = L_p > 0 ? (const char *)Kp + (size_t)s0 * L_p * head_dim * eb : nullptr;
            const char *kd = (const char *)Kd + (size_t)s0 * L_dec * head_dim * eb;
            if (dtype == DSA_BF16) {  // tensor cores: bf16 products are exact, fp32 sums
                rc = head_dim == 64 ? launch_logits_tc<64>(q, kp, kd, W, S, L_p, L_dec, derr, st)
                                    : launch_logits_tc<128>(q, kp, kd, W, S, L_p, L_dec, derr, st);
                if (rc != DSA_OK) break;
            } else
                e = head_dim == 64 ? launch_logits<float, 64>(q, kp, kd, W, S, L_p, L_dec, st)
                                   : launch_logits<float, 128>(q, kp, kd, W, S, L_p, L_dec, st);
            if (e != cudaSuccess) break;
            const long long rows = (long long)S * L_dec;
            diag_softmax_kernel<<<(unsigned)((rows + kWarps - 1) / kWarps), 32 * kWarps, 0, st>>>(
                W, S, L_p, L_dec, step_mass ? step_mass + (size_t)s0 * L_dec * 3 : nullptr, sums);
            if ((e = cudaGetLastError()) != cudaSuccess) break;
            if (n_dist > 0) {
                const int bpd = (L_dec + kWarps - 1) / kWarps;
                diag_similarity_kernel<<<dim3((unsigned)(bpd * n_dist), S), 32 * kWarps, 0, st>>>(W, L_p, L_dec, ddist,
                                                                                                n_dist, bpd, sums + 3);
                if ((e = cudaGetLastError()) != cudaSuccess) break;
            }
        }
        std::vector<double> h(3 + 2 * (size_t)n_dist);
        int herr = 0;
        if (e == cudaSuccess && rc == DSA_OK)
            e = cudaMemcpyAsync(h.data(), sums, sizeof(double) * h.size(), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess && rc == DSA_OK) e = cudaMemcpyAsync(&herr, derr, sizeof(int), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e == cudaSuccess && rc == DSA_OK && herr)
            rc = dsa_detail::fail(DSA_ERR_TIMEOUT, "dsa_diag_trace: a bounded wait in the logits kernel gave up");
        if (e == cudaSuccess && rc == DSA_OK) {
            const double nq = (double)heads * L_dec;
            for (int c = 0; c < 3; ++c) mass_mean[c] = h[c] / nq;
            for (int k = 0; k < n_dist; ++k) {
                const double n = (double)heads * (L_dec - dist[k]);
                vertical[k] = h[3 + 2 * k] / n;
                diagonal[k] = h[3 + 2 * k + 1] / n;
            }
        }
    }
    if (rc == DSA_OK || W) {
        cudaStreamSynchronize(st);
        cudaFree(W);
        cudaFree(sums);
        cudaFree(ddist);
        cudaFree(derr);
    }
    if (rc != DSA_OK) return rc;
    if (e != cudaSuccess) return dsa_detail::cuda_fail(e, "dsa_diag_trace");
    return DSA_OK;
}
