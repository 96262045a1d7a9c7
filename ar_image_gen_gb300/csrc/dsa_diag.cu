// dsa_diag.cu -- attention diagnostics of dense decode attention over a
// trace ("Understanding and Exploiting Diagonal Attention Sparsity in
// Autoregressive Image Generation", section 3.4 "Attention Sparsity
// Analysis": Fig. 8 attention mass on prompt / local / middle tokens, Fig. 10
// vertical vs diagonal score-vector similarity).  C ABI in
// include/dsa_diag.h.
//
// Per chunk of heads, three kernels:
//   diag_logits_kernel   logits z[i][c] = q_i . key_c / sqrt(d) for every
//                        decode query i and every key c it attends (prompt
//                        keys, then decode keys 0..i), 32 x 32 tiles staged in
//                        shared memory (fp32 FMAs; bf16 products are exact);
//   diag_softmax_kernel  per query: softmax over its keys, the prompt /
//                        local / middle weights, and the decode weights
//                        written back in place;
//   diag_similarity_kernel  per (query distance, query): cosine of the
//                        decode score vectors of queries i and i + d over the
//                        same keys (vertical) and over keys shifted by d
//                        (diagonal).
// Sums over heads and queries go to a few doubles per block (atomics).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <vector>

#include "../../include/dsa.h"
#include "../../include/dsa_diag.h"
#include "dsa_internal.h"

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
    int rc = dsa_detail::dev_alloc((void **)&W, per_head * chunk, "diagnostic weights");
    if (rc == DSA_OK) rc = dsa_detail::dev_alloc((void **)&sums, sizeof(double) * (3 + 2 * (size_t)n_dist), "diagnostic sums");
    if (rc == DSA_OK) rc = dsa_detail::dev_alloc((void **)&ddist, sizeof(int) * (size_t)(n_dist > 0 ? n_dist : 1), "distances");
    cudaError_t e = cudaSuccess;
    if (rc == DSA_OK) {
        e = cudaMemsetAsync(sums, 0, sizeof(double) * (3 + 2 * (size_t)n_dist), st);
        if (e == cudaSuccess && n_dist > 0)
            e = cudaMemcpyAsync(ddist, dist, sizeof(int) * n_dist, cudaMemcpyHostToDevice, st);
        const size_t eb = dtype == DSA_F32 ? 4 : 2;
        for (int s0 = 0; s0 < heads && e == cudaSuccess; s0 += chunk) {
            const int S = std::min(chunk, heads - s0);
            const char *q = (const char *)Q + (size_t)s0 * L_dec * head_dim * eb;
            const char *kp = L_p > 0 ? (const char *)Kp + (size_t)s0 * L_p * head_dim * eb : nullptr;
            const char *kd = (const char *)Kd + (size_t)s0 * L_dec * head_dim * eb;
            if (dtype == DSA_BF16)
                e = head_dim == 64 ? launch_logits<__nv_bfloat16, 64>(q, kp, kd, W, S, L_p, L_dec, st)
                                   : launch_logits<__nv_bfloat16, 128>(q, kp, kd, W, S, L_p, L_dec, st);
            else
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
        if (e == cudaSuccess) e = cudaMemcpyAsync(h.data(), sums, sizeof(double) * h.size(), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e == cudaSuccess) {
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
    }
    if (rc != DSA_OK) return rc;
    if (e != cudaSuccess) return dsa_detail::cuda_fail(e, "dsa_diag_trace");
    return DSA_OK;
}
