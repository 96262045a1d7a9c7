// dsa_api.cu -- host side of the C ABI declared in include/dsa.h.
//
// Validation, device state (prompt prefix, decode ring, relative-offset skip
// mask, split partials), the per-step plan (phase, attended counts, split
// choice) and the kernel launches.  No CPU fallback: every step of the decode
// path runs in the kernels of dsa_decode.cuh.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "../../include/dsa.h"
#include "../../include/dsa_proj.h"
#include "dsa_decode.cuh"
#include "dsa_internal.h"

namespace {
thread_local std::string g_err;
std::atomic<int> g_fail_after{0};
}  // namespace

namespace dsa_detail {

int fail(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device allocation with the test hook of dsa_debug_fail_alloc_after().
int dev_alloc(void **p, size_t bytes, const char *what)
{
    *p = nullptr;
    int n = g_fail_after.load();
    if (n > 0) {
        if (n == 1) {
            g_fail_after.store(0);
            return fail(DSA_ERR_OOM, "allocation of %s (%zu bytes) failed (injected)", what, bytes);
        }
        g_fail_after.store(n - 1);
    }
    cudaError_t e = cudaMalloc(p, bytes ? bytes : 16);
    if (e != cudaSuccess) {
        *p = nullptr;
        cudaGetLastError();
        if (e == cudaErrorMemoryAllocation)
            return fail(DSA_ERR_OOM, "allocation of %s (%zu bytes) failed", what, bytes);
        return cuda_fail(e, what);
    }
    return DSA_OK;
}

}  // namespace dsa_detail

namespace {

using dsa_detail::cuda_fail;
using dsa_detail::dev_alloc;
using dsa_detail::fail;
using dsa_detail::forget_handle;
using dsa_detail::note_launch;

constexpr uint32_t kMagic = 0x44534131u;  // "DSA1"
constexpr uint32_t kDefaultWaitLimit = 0xffffffffu;

// Bytes of a stored K / V element and of a q / k_new / v_new / out element.
int elem_bytes(int dtype) { return dtype == DSA_F32 ? 4 : (dtype == DSA_FP8_E4M3 ? 1 : 2); }
int io_bytes(int dtype) { return dtype == DSA_F32 ? 4 : 2; }
bool valid_dtype(int dtype) { return dtype == DSA_BF16 || dtype == DSA_F32 || dtype == DSA_FP8_E4M3; }

// Stage rows and the rows-per-item limit of pipeline shape sh (a multiple of
// the stage rows, so that items end on stage boundaries).
int stage_bytes(int sh) { return sh == 0 ? dsa::Pipe<0>::STAGE_BYTES : dsa::Pipe<1>::STAGE_BYTES; }
int stage_rows(int dtype, int D, int sh) { return stage_bytes(sh) / (2 * D * elem_bytes(dtype)); }
int chunk_cap(int dtype, int D, int sh)
{
    const int rows = stage_rows(dtype, D, sh);
    const int cap = sh == 0 ? dsa::Pipe<0>::CHUNK_MAX : dsa::Pipe<1>::CHUNK_MAX;
    return cap / rows * rows;
}
constexpr int kWarpsPerCta = DSA_WARPS;

}  // namespace

struct dsa_ctx {
    uint32_t magic;
    int S, D, L_p, N_r, N_att, sink, dtype;
    int R, A, Lcap, MW;
    int t;
    int prefilled;
    int last_select;
    int device, sm_count;
    int ctas_per_sm[dsa::kPipelines];  // resident CTAs per SM of each launch pipeline (0: unavailable)
    int forced_split;
    int forced_pipe;  // 0: automatic, else launch pipeline + 1
    int xm_ok[dsa::kPipelines];  // 1: the CTA merge's shared memory keeps the pipeline's occupancy
    int merge_launch_only;       // 1: split streams always go through merge_kernel (test knob)
    int pstride;
    uint32_t wait_limit;
    void *prefix, *ring;
    uint32_t *mask;
    int32_t *last_sel;
    float *part_acc;
    float2 *part_ml, *part_min;
    int *status;
    float *scales;         // FP8 storage: [4, S] K scale, V scale, their fp32 inverses (else NULL)
    int *step_dev;         // graph mode: [0] the step t on the device, [1] CTAs finished (allocated on first use)
    uint16_t *glist;       // [S, LS] attended relative offsets of the steady state (NULL when nothing is skipped)
    int LS;
    int graph_mode;
    CUtensorMap ring_map;  // 2-D view of the ring: [S * R rows, 2 * D], one-row box
};

namespace {

bool valid(dsa_handle h) { return h != nullptr && h->magic == kMagic; }

int validate(int heads, int head_dim, int L_p, int N_r, int N_att, int sink, int dtype)
{
    if (heads < 1) return fail(DSA_ERR_ARG, "heads must be >= 1 (got %d)", heads);
    if (head_dim != 64 && head_dim != 128) return fail(DSA_ERR_ARG, "head_dim must be 64 or 128 (got %d)", head_dim);
    if (L_p < 0) return fail(DSA_ERR_ARG, "L_p must be >= 0 (got %d)", L_p);
    if (sink < 0) return fail(DSA_ERR_ARG, "sink must be >= 0 (got %d)", sink);
    if (N_att < 1 || N_att > N_r) return fail(DSA_ERR_ARG, "need 1 <= N_att <= N_r (got N_att=%d, N_r=%d)", N_att, N_r);
    if (sink > 0 && N_att <= sink) return fail(DSA_ERR_ARG, "need N_att > sink (got N_att=%d, sink=%d)", N_att, sink);
    if (N_r - sink > 65536) return fail(DSA_ERR_ARG, "N_r - sink must be <= 65536 (got %d)", N_r - sink);
    if (!valid_dtype(dtype))
        return fail(DSA_ERR_ARG, "dtype must be DSA_BF16, DSA_F32 or DSA_FP8_E4M3 (got %d)", dtype);
    if ((long long)L_p + sink > INT_MAX / 4) return fail(DSA_ERR_ARG, "L_p too large");
    if ((long long)heads * (N_r - sink) > INT_MAX) return fail(DSA_ERR_ARG, "heads * (N_r - sink) must fit in 31 bits");
    return DSA_OK;
}

struct Plan {
    int phase, tin, P, a, wlen, select, sinkmode, n, nsplit, chunk, nitems, grid;
    int pipe, shape, nbuf;  // launch pipeline: stage shape pipe & 1, 2 + (pipe >> 1) stages per warp
    long long rounds, stages;
    unsigned long long bytes;
};

long long resident_warps(const dsa_ctx *h, int pi) { return (long long)h->sm_count * h->ctas_per_sm[pi] * kWarpsPerCta; }

// Work items per stream under launch pipeline pi.  Splitting a stream costs a
// merge (inside the CTA, or partials and a merge launch; launch_cost weighs
// it); it pays when the streams alone leave most warps
// idle (each warp streams its rows through a short pipeline, so few warps
// cannot keep HBM busy).  Streams are split into about resident-warps /
// streams pieces (one round of items) once they fill at most half the warps,
// with at least two stages of rows per piece; streams longer than an item's
// row limit always split.
int auto_splits(const dsa_ctx *h, int n, int pi)
{
    const int sh = pi & 1;
    const int rows = stage_rows(h->dtype, h->D, sh);
    const int cap = chunk_cap(h->dtype, h->D, sh);
    const int need = (n + cap - 1) / cap;
    const long long warps = resident_warps(h, pi);
    const int want = 2LL * h->S <= warps ? (int)(warps / h->S) : 1;
    const int by_rows = n / (2 * rows) > 1 ? n / (2 * rows) : 1;
    const int ns = want < by_rows ? want : by_rows;
    return ns > need ? ns : need;
}

// Items, grid and stage count of launch pipeline pi for a step of n rows per
// stream, with the pieces per stream the split knob forces, else the fewest
// an item's row limit allows (fewest) or the automatic count above.
void shape_plan(const dsa_ctx *h, int pi, Plan &p, bool fewest = false)
{
    const int sh = pi & 1;
    const int rows = stage_rows(h->dtype, h->D, sh);
    const int cap = chunk_cap(h->dtype, h->D, sh);
    int ns = h->forced_split > 0 ? h->forced_split : (fewest ? 1 : auto_splits(h, p.n, pi));
    const int need = (p.n + cap - 1) / cap;
    if (ns < need) ns = need;
    if (ns > p.n) ns = p.n;
    int chunk = (p.n + ns - 1) / ns;
    chunk = (chunk + rows - 1) / rows * rows;
    if (chunk > cap) chunk = cap;
    p.pipe = pi;
    p.shape = sh;
    p.nbuf = 2 + (pi >> 1);
    p.chunk = chunk;
    p.nsplit = (p.n + chunk - 1) / chunk;
    p.nitems = p.nsplit * h->S;
    // Give every warp the same number of items: with k = ceil(items / resident
    // warps) rounds of items, use just enough warps for k items each, so no
    // warp runs a round that most others do not.
    const long long max_warps = resident_warps(h, pi);
    p.rounds = (p.nitems + max_warps - 1) / max_warps;
    const long long warps = (p.nitems + p.rounds - 1) / p.rounds;
    p.grid = (int)((warps + kWarpsPerCta - 1) / kWarpsPerCta);
    // A warp's run time is its rounds times the stages of one item, each
    // stage about one copy latency over the two stages in flight.
    const int item_rows = chunk < p.n ? chunk : p.n;
    p.stages = p.rounds * ((item_rows + rows - 1) / rows);
}

// Cost model of a launch, in microseconds: a launch is bound either by HBM
// bandwidth (its bytes at the rate its pipeline streams) or by the stages
// each warp waits on in sequence (rounds x stages per item, one loaded copy
// latency each); splitting streams adds the merge of the pieces.  The rates,
// stage latencies and the merge launch's cost are fitted per pipeline
// (least squares on the relative error) to launch times measured on GB300
// (152 SMs) for every pipeline, with the automatic and with the fewest
// pieces per stream, over 20 decode launches (13 sparse steady states and 7
// dense settings: 512 to 3072 streams of 93 to 8196 rows; all splits then
// merged by the merge launch), separately for 2-byte and for 1-byte rows:
// FP8 stages hold twice the rows of a bf16 stage and take longer, their
// warps being bound by their own widening arithmetic as much as by HBM.
// Over those launches the plans this model picks took 1.7 % (bf16) and
// 0.2 % (FP8) longer in total than the fastest measured plan of each.  fp32
// rows take the 2-byte fit (bandwidth bound at twice the bytes).
// Pieces of a stream merged inside the CTA (see cta_merge) cost far less
// than the merge launch: measured on the same launches, two pieces added
// about 0.5 us (bf16) and 0.1 us (FP8) over the unsplit cost model, against
// about 3 us through the merge launch.  Four bf16 pieces merged inside the
// CTA (its warps wait for the slowest of four) cost about what the merge
// launch does; four FP8 pieces, whose warps are bound by their own work,
// as little as two (the 512-stream lumina launches: 10.6 against 12.6 us
// in two pieces and 13.6 us in three through the merge launch).
struct CostFit {
    double gbs[dsa::kPipelines];       // streaming rate, GB/s
    double us_stage[dsa::kPipelines];  // one stage in sequence, us
    double split_us;                   // partials + merge launch of a split step, us
    double cta2_us, cta4_us;           // 2 or 4 pieces merged inside the CTA, us
};
constexpr CostFit kFit16 = {{6533, 6535, 6740, 6655}, {0.846, 0.999, 0.827, 0.433}, 2.32, 0.5, 2.32};
constexpr CostFit kFitFp8 = {{6286, 5864, 6736, 6219}, {1.644, 1.108, 1.420, 1.321}, 2.64, 0.1, 0.1};

bool cta_merge(const dsa_ctx *h, const Plan &pl);

double launch_cost(const dsa_ctx *h, const Plan &p)
{
    const CostFit &f = h->dtype == DSA_FP8_E4M3 ? kFitFp8 : kFit16;
    const double bw = (double)p.bytes / (f.gbs[p.pipe] * 1e3);
    const double lat = f.us_stage[p.pipe] * (double)p.stages;
    const double split = p.nsplit == 1       ? 0.0
                         : !cta_merge(h, p) ? f.split_us
                                            : (p.nsplit == 2 ? f.cta2_us : f.cta4_us);
    return (bw > lat ? bw : lat) + split;
}

// The plan of a step: every launch pipeline the device can hold (or the one
// the pipeline knob forces), each with the automatic and with the fewest
// pieces per stream (or the count the split knob forces), and the one the
// cost model above finishes first (the earlier candidate on a tie).  Three
// stages per warp win where their deeper pipelines take the streams in as
// few rounds as two stages do; shape 1's extra warps win where they save a
// round; unsplit items win where the split would leave the launch
// bandwidth bound anyway.
Plan make_plan(const dsa_ctx *h, int t)
{
    Plan p{};
    if (t < h->sink) {
        p.phase = 0;
        p.tin = -1;
        p.P = h->L_p + t;
        p.a = 1;
        p.wlen = 1;
        p.select = 0;
        p.sinkmode = 1;
    } else {
        const int tin = t - h->sink;
        p.tin = tin;
        p.P = h->L_p + h->sink;
        p.phase = tin < h->A - 1 ? 1 : (tin < h->R ? 2 : 3);
        p.a = tin + 1 < h->A ? tin + 1 : h->A;
        p.wlen = tin + 1 < h->R ? tin + 1 : h->R;
        p.select = (tin >= h->A - 1 && tin <= h->R - 2) ? 1 : 0;
        p.sinkmode = 0;
    }
    p.n = p.P + p.a;
    const unsigned long long De = (unsigned long long)h->D * elem_bytes(h->dtype);
    const unsigned long long Di = (unsigned long long)h->D * io_bytes(h->dtype);
    // K and V rows read (current token through k_new/v_new) + q, k_new, v_new
    // read + new entry written + out written.
    p.bytes = (unsigned long long)h->S * (2 * De * (unsigned long long)(p.n - 1) + 4 * Di + 2 * De);
    Plan best{};
    double best_cost = 0.0;
    bool have = false;
    for (int pi = 0; pi < dsa::kPipelines; ++pi) {
        if (h->forced_pipe > 0 ? pi != h->forced_pipe - 1 : h->ctas_per_sm[pi] < 1) continue;
        for (int fewest = 0; fewest < (h->forced_split > 0 ? 1 : 2); ++fewest) {
            Plan q = p;
            shape_plan(h, pi, q, fewest != 0);
            const double c = launch_cost(h, q);
            if (!have || c < best_cost) {
                best = q;
                best_cost = c;
                have = true;
            }
        }
    }
    return best;
}

// Pieces of a split stream merged inside the CTA (no merge launch): the
// pieces fill whole groups of the CTA's warps (nsplit 2 or 4), and the
// exchange area costs the pipeline no occupancy.
bool cta_merge(const dsa_ctx *h, const Plan &pl)
{
    return (pl.nsplit == 2 || pl.nsplit == 4) && kWarpsPerCta % pl.nsplit == 0 && h->xm_ok[pl.pipe] &&
           !h->merge_launch_only;
}

// The plan of a step as the C ABI reports it.
void fill_plan(const dsa_ctx *h, const Plan &p, dsa_step_plan *out)
{
    out->phase = p.phase;
    out->t_inner = p.tin;
    out->n_prefix = p.P;
    out->n_decode = p.a;
    out->select = p.select;
    out->nsplit = p.nsplit;
    out->chunk = p.chunk;
    out->grid = p.grid;
    out->pipeline = p.pipe + 1;
    out->algo_bytes = p.bytes;
    out->cta_merge = cta_merge(h, p) ? 1 : 0;
}

// A handle-shaped description of a state of these sizes (nothing allocated,
// no device queried): what the plan reads.
void describe(dsa_ctx &h, int heads, int head_dim, int L_p, int N_r, int N_att, int sink, int dtype)
{
    h.magic = kMagic;
    h.S = heads;
    h.D = head_dim;
    h.L_p = L_p;
    h.N_r = N_r;
    h.N_att = N_att;
    h.sink = sink;
    h.dtype = dtype;
    h.R = N_r - sink;
    h.A = N_att - sink;
    h.Lcap = L_p + sink;
    h.MW = (h.R + 31) / 32;
}

// The most work items per stream any step takes (steps from N_att - 1 on
// all attend the same row count), so that partials are sized once.
int max_splits(const dsa_ctx *h)
{
    int m = 1;
    for (int t = 0; t < h->N_att; ++t) {
        const int ns = make_plan(h, t).nsplit;
        m = ns > m ? ns : m;
    }
    return m;
}

int ensure_partials(dsa_ctx *h, int nsplit)
{
    if (nsplit <= h->pstride) return DSA_OK;
    float *acc = nullptr;
    float2 *ml = nullptr, *mn = nullptr;
    int rc = dev_alloc((void **)&acc, sizeof(float) * (size_t)h->S * nsplit * h->D, "split partials");
    if (rc == DSA_OK) rc = dev_alloc((void **)&ml, sizeof(float2) * (size_t)h->S * nsplit, "split partials");
    if (rc == DSA_OK) rc = dev_alloc((void **)&mn, sizeof(float2) * (size_t)h->S * nsplit, "split partials");
    if (rc != DSA_OK) {
        cudaFree(acc);
        cudaFree(ml);
        cudaFree(mn);
        return rc;
    }
    cudaFree(h->part_acc);
    cudaFree(h->part_ml);
    cudaFree(h->part_min);
    h->part_acc = acc;
    h->part_ml = ml;
    h->part_min = mn;
    h->pstride = nsplit;
    return DSA_OK;
}

void free_ctx(dsa_ctx *h)
{
    if (!h) return;
    cudaFree(h->prefix);
    cudaFree(h->ring);
    cudaFree(h->mask);
    cudaFree(h->last_sel);
    cudaFree(h->part_acc);
    cudaFree(h->part_ml);
    cudaFree(h->part_min);
    cudaFree(h->status);
    cudaFree(h->scales);
    cudaFree(h->step_dev);
    cudaFree(h->glist);
    h->magic = 0;
    forget_handle(h);
    delete h;
}

// Tensor map over the ring seen as a 2-D array of S * R rows of 2 * D
// elements (one K|V entry per row), box one row high and one entry wide:
// the form the TMA tile::gather4 load needs.
int encode_ring_map(dsa_ctx *h)
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void **)&encode, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !encode) {
            encode = nullptr;
            return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        }
    }
    const cuuint64_t dims[2] = {(cuuint64_t)(2 * h->D), (cuuint64_t)h->S * h->R};
    const cuuint64_t strides[1] = {(cuuint64_t)(2 * h->D * elem_bytes(h->dtype))};
    const cuuint32_t box[2] = {(cuuint32_t)(2 * h->D), 1};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType ty = h->dtype == DSA_F32        ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : h->dtype == DSA_FP8_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                              : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = encode(&h->ring_map, ty,
                        2, h->ring, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return DSA_OK;
}

// Resident CTAs per SM of the decode kernel with nbuf stages per warp,
// without (xm 0) or with (xm 1) the CTA merge's shared memory.
template <typename T, int D, int SH>
int occupancy(int nbuf, int xm)
{
    using C = dsa::KCfg<T, D, SH>;
    static int cached[2][dsa::kMaxNbuf + 1] = {{-1, -1, -1, -1}, {-1, -1, -1, -1}};
    static_assert(dsa::kMaxNbuf == 3, "one cache entry per stage count");
    if (cached[xm][nbuf] < 0) {
        // The attribute allows the largest layout, so every stage count launches.
        cudaError_t e = cudaFuncSetAttribute(dsa::decode_kernel<T, D, SH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::smem(dsa::kMaxNbuf) + C::xm_bytes());
        if (e != cudaSuccess) return -1;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dsa::decode_kernel<T, D, SH>, C::THREADS,
                                                          C::smem(nbuf) + (xm ? C::xm_bytes() : 0));
        if (e != cudaSuccess) return -1;
        cached[xm][nbuf] = n;
    }
    return cached[xm][nbuf];
}

template <int SH>
int occupancy_sh(int dtype, int D, int nbuf, int xm)
{
    if (dtype == DSA_BF16)
        return D == 64 ? occupancy<__nv_bfloat16, 64, SH>(nbuf, xm) : occupancy<__nv_bfloat16, 128, SH>(nbuf, xm);
    if (dtype == DSA_FP8_E4M3)
        return D == 64 ? occupancy<__nv_fp8_e4m3, 64, SH>(nbuf, xm) : occupancy<__nv_fp8_e4m3, 128, SH>(nbuf, xm);
    return D == 64 ? occupancy<float, 64, SH>(nbuf, xm) : occupancy<float, 128, SH>(nbuf, xm);
}

// Resident CTAs per SM of every launch pipeline (0: cannot launch); the
// first (shape 0, two stages per warp) must be launchable.  xm_ok (may be
// NULL): 1 where the CTA merge's shared memory leaves that number unchanged.
int query_occupancy(int dtype, int D, int *ctas, int *xm_ok = nullptr)
{
    for (int pi = 0; pi < dsa::kPipelines; ++pi) {
        const int nbuf = 2 + (pi >> 1);
        ctas[pi] = (pi & 1) ? occupancy_sh<1>(dtype, D, nbuf, 0) : occupancy_sh<0>(dtype, D, nbuf, 0);
        if (ctas[pi] < 1) {
            if (pi == 0) return cuda_fail(cudaGetLastError(), "kernel occupancy query (is this an sm_103 device?)");
            ctas[pi] = 0;
            cudaGetLastError();
        }
        if (xm_ok) {
            const int n = ctas[pi] < 1 ? 0 : (pi & 1) ? occupancy_sh<1>(dtype, D, nbuf, 1) : occupancy_sh<0>(dtype, D, nbuf, 1);
            if (n < 1) cudaGetLastError();
            xm_ok[pi] = (ctas[pi] >= 1 && n == ctas[pi]) ? 1 : 0;
        }
    }
    return DSA_OK;
}

// Launches the decode kernel as a programmatic dependent launch: its CTAs
// may start while the previous kernel in the stream finishes; the kernel
// itself waits for that kernel before it reads inputs or writes anything.
template <typename T, int D, int SH>
cudaError_t launch_decode(const dsa::DecodeParams &p, const CUtensorMap &map, int grid, cudaStream_t st)
{
    using C = dsa::KCfg<T, D, SH>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::smem(p.nbuf) + (p.cta_merge ? C::xm_bytes() : 0);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dsa::decode_kernel<T, D, SH>, p, map);
}

template <typename T, int D>
cudaError_t launch_merge(const dsa::DecodeParams &p, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.S + dsa::kMergeWarps - 1) / dsa::kMergeWarps);
    cfg.blockDim = dim3(32 * dsa::kMergeWarps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dsa::merge_kernel<T, D>, p);
}

template <int SH>
cudaError_t launch_decode_sh(int dtype, int D, const dsa::DecodeParams &p, const CUtensorMap &map, int grid,
                             cudaStream_t st)
{
    if (dtype == DSA_BF16)
        return D == 64 ? launch_decode<__nv_bfloat16, 64, SH>(p, map, grid, st)
                       : launch_decode<__nv_bfloat16, 128, SH>(p, map, grid, st);
    if (dtype == DSA_FP8_E4M3)
        return D == 64 ? launch_decode<__nv_fp8_e4m3, 64, SH>(p, map, grid, st)
                       : launch_decode<__nv_fp8_e4m3, 128, SH>(p, map, grid, st);
    return D == 64 ? launch_decode<float, 64, SH>(p, map, grid, st) : launch_decode<float, 128, SH>(p, map, grid, st);
}

// Decode launch plus, when streams are split and not merged inside the
// CTA, the merge launch.
cudaError_t launch_step(int dtype, int D, int shape, const dsa::DecodeParams &p, const CUtensorMap &map, int grid,
                        cudaStream_t st)
{
    cudaError_t e = shape == 0 ? launch_decode_sh<0>(dtype, D, p, map, grid, st)
                               : launch_decode_sh<1>(dtype, D, p, map, grid, st);
    if (e != cudaSuccess || p.nsplit == 1 || p.cta_merge) return e;
    if (dtype == DSA_BF16)
        return D == 64 ? launch_merge<__nv_bfloat16, 64>(p, st) : launch_merge<__nv_bfloat16, 128>(p, st);
    if (dtype == DSA_FP8_E4M3)
        return D == 64 ? launch_merge<__nv_fp8_e4m3, 64>(p, st) : launch_merge<__nv_fp8_e4m3, 128>(p, st);
    return D == 64 ? launch_merge<float, 64>(p, st) : launch_merge<float, 128>(p, st);
}

// The last handle (of any kind) this library launched a kernel for, per
// stream: a decode step may read its state before the grid dependency wait
// only when the kernel just before it in the stream was not one of this
// handle's own.
std::mutex g_last_mu;
struct LastLaunch {
    cudaStream_t stream;
    const void *handle;
};
LastLaunch g_last[16];
int g_last_next;

}  // namespace

bool dsa_detail::note_launch(cudaStream_t st, const void *h)
{
    std::lock_guard<std::mutex> lock(g_last_mu);
    for (auto &e : g_last)
        if (e.handle && e.stream == st) {
            const bool other = e.handle != h;
            e.handle = h;
            return other;
        }
    g_last[g_last_next] = {st, h};
    g_last_next = (g_last_next + 1) % 16;
    return false;  // unknown stream: be conservative
}

void dsa_detail::forget_handle(const void *h)
{
    std::lock_guard<std::mutex> lock(g_last_mu);
    for (auto &e : g_last)
        if (e.handle == h) e.handle = &g_last_mu;  // a value no handle has
}

namespace {

template <typename T, int D>
cudaError_t launch_prefill(const void *K, const void *V, void *prefix, const float *kinv, const float *vinv, int S,
                           int L_p, int Lcap, cudaStream_t st)
{
    using IO = typename dsa::Elem<T>::IO;
    const size_t total = (size_t)S * L_p * 2 * (D / dsa::Elem<T>::VEC);
    if (total == 0) return cudaSuccess;
    size_t blocks = (total + 255) / 256;
    if (blocks > 65535 * 8) blocks = 65535 * 8;
    dsa::prefill_kernel<T, D><<<(unsigned)blocks, 256, 0, st>>>((const IO *)K, (const IO *)V, (T *)prefix, kinv, vinv,
                                                                S, L_p, Lcap);
    return cudaGetLastError();
}

// FP8 storage: uploads K and V scales and their fp32 inverses ([4, S]).
int upload_scales(dsa_ctx *h, const float *k_scale, const float *v_scale)
{
    const size_t S = (size_t)h->S;
    float *host = new (std::nothrow) float[4 * S];
    if (!host) return fail(DSA_ERR_OOM, "host allocation failed");
    for (size_t i = 0; i < S; ++i) {
        host[i] = k_scale ? k_scale[i] : 1.0f;
        host[S + i] = v_scale ? v_scale[i] : 1.0f;
        host[2 * S + i] = 1.0f / host[i];
        host[3 * S + i] = 1.0f / host[S + i];
    }
    cudaError_t e = cudaMemcpy(h->scales, host, sizeof(float) * 4 * S, cudaMemcpyHostToDevice);
    delete[] host;
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, "scale upload");
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" {

const char *dsa_last_error(void) { return g_err.c_str(); }

int dsa_debug_fail_alloc_after(int n)
{
    g_fail_after.store(n > 0 ? n : 0);
    return DSA_OK;
}

size_t dsa_state_bytes(int heads, int head_dim, int L_p, int N_r, int sink, int dtype)
{
    if (heads < 1 || (head_dim != 64 && head_dim != 128) || L_p < 0 || sink < 0 || N_r <= sink || !valid_dtype(dtype))
        return 0;
    const size_t row = 2 * (size_t)head_dim * elem_bytes(dtype);
    const size_t R = (size_t)(N_r - sink);
    const size_t MW = (R + 31) / 32;
    return (size_t)heads * (((size_t)L_p + sink) * row + R * row + MW * 4);
}

int dsa_create_ex(int heads, int head_dim, int L_p, int N_r, int N_att, int sink, int dtype, dsa_handle *out)
{
    if (!out) return fail(DSA_ERR_ARG, "out is NULL");
    *out = nullptr;
    int rc = validate(heads, head_dim, L_p, N_r, N_att, sink, dtype);
    if (rc != DSA_OK) return rc;

    dsa_ctx *h = new (std::nothrow) dsa_ctx();
    if (!h) return fail(DSA_ERR_OOM, "host allocation failed");
    h->magic = kMagic;
    h->S = heads;
    h->D = head_dim;
    h->L_p = L_p;
    h->N_r = N_r;
    h->N_att = N_att;
    h->sink = sink;
    h->dtype = dtype;
    h->R = N_r - sink;
    h->A = N_att - sink;
    h->Lcap = L_p + sink;
    h->MW = (h->R + 31) / 32;
    h->wait_limit = kDefaultWaitLimit;

    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) {
        free_ctx(h);
        cudaGetLastError();
        return cuda_fail(e, "cudaGetDevice");
    }
    e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device);
    if (e != cudaSuccess) {
        free_ctx(h);
        return cuda_fail(e, "cudaDeviceGetAttribute");
    }
    rc = query_occupancy(dtype, head_dim, h->ctas_per_sm, h->xm_ok);
    if (rc != DSA_OK) {
        std::string msg = g_err;
        free_ctx(h);
        g_err = msg;
        return rc;
    }

    const size_t row = 2 * (size_t)head_dim * elem_bytes(dtype);
    const size_t S = (size_t)heads;
    rc = dev_alloc(&h->prefix, S * h->Lcap * row, "prompt prefix");
    if (rc == DSA_OK) rc = dev_alloc(&h->ring, S * h->R * row, "decode ring");
    if (rc == DSA_OK) rc = dev_alloc((void **)&h->mask, S * h->MW * 4, "skip mask");
    if (rc == DSA_OK) rc = dev_alloc((void **)&h->last_sel, S * 4, "last selection");
    if (rc == DSA_OK) rc = dev_alloc((void **)&h->status, 16, "status word");
    if (rc == DSA_OK && dtype == DSA_FP8_E4M3) rc = dev_alloc((void **)&h->scales, S * 4 * sizeof(float), "FP8 scales");
    if (rc == DSA_OK && dtype == DSA_FP8_E4M3) rc = upload_scales(h, nullptr, nullptr);
    // The steady state's attended offsets (A per stream): stored at the last
    // step before it, read afterwards.
    h->LS = (h->A + 1) & ~1;
    if (rc == DSA_OK && h->A < h->R) rc = dev_alloc((void **)&h->glist, S * h->LS * sizeof(uint16_t), "offset list");
    if (rc == DSA_OK) rc = ensure_partials(h, max_splits(h));
    if (rc == DSA_OK) rc = encode_ring_map(h);
    if (rc != DSA_OK) {
        std::string msg = g_err;
        free_ctx(h);
        g_err = msg;
        return rc;
    }
    if ((e = cudaMemset(h->mask, 0, S * h->MW * 4)) != cudaSuccess ||
        (e = cudaMemset(h->status, 0, 16)) != cudaSuccess ||
        (e = cudaMemset(h->last_sel, 0xff, S * 4)) != cudaSuccess) {
        free_ctx(h);
        return cuda_fail(e, "cudaMemset");
    }
    *out = h;
    return DSA_OK;
}

int dsa_create(int heads, int head_dim, int L_p, int N_r, int N_att, int sink, dsa_handle *out)
{
    return dsa_create_ex(heads, head_dim, L_p, N_r, N_att, sink, DSA_BF16, out);
}

int dsa_destroy(dsa_handle h)
{
    if (!h) return DSA_OK;
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    cudaDeviceSynchronize();
    free_ctx(h);
    return DSA_OK;
}

int dsa_prefill(dsa_handle h, const void *K, const void *V, void *stream)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    if (h->L_p > 0 && (!K || !V)) return fail(DSA_ERR_ARG, "K and V must be non-NULL when L_p > 0");
    if (h->L_p > 0 && (!aligned16(K) || !aligned16(V))) return fail(DSA_ERR_ARG, "K and V must be 16-byte aligned");
    cudaStream_t st = (cudaStream_t)stream;
    const size_t S = (size_t)h->S;
    cudaError_t e;
    if ((e = cudaMemsetAsync(h->mask, 0, S * h->MW * 4, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(h->status, 0, 16, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(h->last_sel, 0xff, S * 4, st)) != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync");
    const float *kinv = h->scales ? h->scales + 2 * S : nullptr;
    const float *vinv = h->scales ? h->scales + 3 * S : nullptr;
    if (h->dtype == DSA_BF16)
        e = h->D == 64 ? launch_prefill<__nv_bfloat16, 64>(K, V, h->prefix, kinv, vinv, h->S, h->L_p, h->Lcap, st)
                       : launch_prefill<__nv_bfloat16, 128>(K, V, h->prefix, kinv, vinv, h->S, h->L_p, h->Lcap, st);
    else if (h->dtype == DSA_FP8_E4M3)
        e = h->D == 64 ? launch_prefill<__nv_fp8_e4m3, 64>(K, V, h->prefix, kinv, vinv, h->S, h->L_p, h->Lcap, st)
                       : launch_prefill<__nv_fp8_e4m3, 128>(K, V, h->prefix, kinv, vinv, h->S, h->L_p, h->Lcap, st);
    else
        e = h->D == 64 ? launch_prefill<float, 64>(K, V, h->prefix, kinv, vinv, h->S, h->L_p, h->Lcap, st)
                       : launch_prefill<float, 128>(K, V, h->prefix, kinv, vinv, h->S, h->L_p, h->Lcap, st);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    note_launch(st, h);
    h->t = 0;
    h->prefilled = 1;
    h->last_select = 0;
    return DSA_OK;
}

int dsa_plan_step(dsa_handle h, int t, dsa_step_plan *out)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    if (!out || t < 0) return fail(DSA_ERR_ARG, "out must be non-NULL and t >= 0");
    fill_plan(h, make_plan(h, t), out);
    return DSA_OK;
}

int dsa_plan_query(int heads, int head_dim, int L_p, int N_r, int N_att, int sink, int dtype, int t, int sm_count,
                   const int *ctas_per_sm, const int *cta_merge_ok, dsa_step_plan *out)
{
    int rc = validate(heads, head_dim, L_p, N_r, N_att, sink, dtype);
    if (rc != DSA_OK) return rc;
    if (!out || !ctas_per_sm || t < 0 || sm_count < 1)
        return fail(DSA_ERR_ARG, "out and ctas_per_sm must be non-NULL, t >= 0 and sm_count >= 1");
    if (ctas_per_sm[0] < 1) return fail(DSA_ERR_ARG, "pipeline 1 must have at least one resident CTA per SM");
    dsa_ctx h{};
    describe(h, heads, head_dim, L_p, N_r, N_att, sink, dtype);
    h.sm_count = sm_count;
    for (int pi = 0; pi < dsa::kPipelines; ++pi) {
        h.ctas_per_sm[pi] = ctas_per_sm[pi] > 0 ? ctas_per_sm[pi] : 0;
        h.xm_ok[pi] = (cta_merge_ok && cta_merge_ok[pi] && h.ctas_per_sm[pi] > 0) ? 1 : 0;
    }
    fill_plan(&h, make_plan(&h, t), out);
    return DSA_OK;
}

}  // extern "C"

namespace {

// How a step lists the attended offsets.  From the last step before the
// steady state on (t' >= R - 1, no more selections) the relative-offset mask
// never changes, so neither do the attended offsets: that step lists them
// from the mask and stores them (1), later steps read the stored list (2),
// provided every item's slice fits the kernel's prefetch registers;
// otherwise, and before, the mask is scanned (0).
int list_mode(const dsa_ctx *h, const Plan &pl)
{
    if (!h->glist || pl.sinkmode || pl.tin < h->R - 1) return 0;
    if (pl.tin == h->R - 1) return 1;
    for (int c = 0; c < pl.nsplit; ++c) {
        const int lo = c * pl.chunk;
        const int hi = lo + pl.chunk < pl.n ? lo + pl.chunk : pl.n;
        const int klo = (lo > pl.P ? lo : pl.P) - pl.P;
        const int khi = (hi > pl.P ? hi : pl.P) - pl.P;
        if (khi - (klo & ~1) > dsa::kListSliceMax) return 0;
    }
    return 2;
}

// Host checks of a decode step that come before any launch.
int check_step(dsa_handle h, const void *q, const void *k_new, const void *v_new, void *out)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    if (!h->prefilled) return fail(DSA_ERR_STATE, "dsa_decode_step before dsa_prefill");
    if (!q || !k_new || !v_new || !out) return fail(DSA_ERR_ARG, "q, k_new, v_new and out must be non-NULL");
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out))
        return fail(DSA_ERR_ARG, "q, k_new, v_new and out must be 16-byte aligned");
    if (h->t == INT_MAX) return fail(DSA_ERR_STATE, "decode step counter exhausted");
    return DSA_OK;
}

// The decode launch(es) of one step.  after_proj: the kernel just before in
// the stream is the projection of this step, which touches none of the
// handle's state and lets its dependents start only after the kernel before
// it has completed, so the state may be read before the grid dependency wait.
int launch_decode_step(dsa_handle h, const void *q, const void *k_new, const void *v_new, void *out,
                       cudaStream_t st, bool after_proj, bool appended = false)
{
    const Plan pl = make_plan(h, h->t);
    if ((long long)pl.nsplit * h->S > INT_MAX) return fail(DSA_ERR_ARG, "grid too large");
    if (h->graph_mode && pl.phase != 3)
        return fail(DSA_ERR_STATE, "graph mode runs the steady state only (t - sink >= N_r - sink); step %d is in phase %d",
                    h->t, pl.phase);
    int rc = ensure_partials(h, pl.nsplit);
    if (rc != DSA_OK) return rc;

    dsa::DecodeParams p;
    p.q = q;
    p.knew = k_new;
    p.vnew = v_new;
    p.out = out;
    p.prefix = h->prefix;
    p.ring = h->ring;
    p.mask = h->mask;
    p.last_sel = h->last_sel;
    p.part_acc = h->part_acc;
    p.part_ml = h->part_ml;
    p.part_min = h->part_min;
    p.status = h->status;
    p.S = h->S;
    p.Lcap = h->Lcap;
    p.P = pl.P;
    p.sinkmode = pl.sinkmode;
    p.R = h->R;
    p.tin = pl.tin;
    p.tin_mod = pl.tin >= 0 ? pl.tin % h->R : 0;
    p.wlen = pl.wlen;
    p.a = pl.a;
    p.n = pl.n;
    p.nsplit = pl.nsplit;
    p.nbuf = pl.nbuf;
    p.chunk = pl.chunk;
    p.pstride = h->pstride;
    p.nitems = pl.nitems;
    p.noskip = (h->A == h->R) ? 1 : 0;
    p.select = pl.select;
    p.MW = h->MW;
    p.qscale = (float)(1.4426950408889634 / std::sqrt((double)h->D));
    p.kscale = h->scales ? h->scales : nullptr;
    p.vscale = h->scales ? h->scales + h->S : nullptr;
    p.kinv = h->scales ? h->scales + 2 * (size_t)h->S : nullptr;
    p.vinv = h->scales ? h->scales + 3 * (size_t)h->S : nullptr;
    p.wait_limit = h->wait_limit;
    p.step_dev = h->graph_mode ? h->step_dev : nullptr;
    p.sink = h->sink;

    p.glist = h->glist;
    p.LS = h->LS;
    p.list_mode = list_mode(h, pl);
    p.appended = appended ? 1 : 0;
    p.cta_merge = cta_merge(h, pl) ? 1 : 0;

    const bool other = note_launch(st, h);
    p.early = (other || after_proj) ? 1 : 0;
    cudaError_t e = launch_step(h->dtype, h->D, pl.shape, p, h->ring_map, pl.grid, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    h->last_select = pl.select;
    h->t += 1;
    return DSA_OK;
}

}  // namespace

extern "C" {

int dsa_decode_step(dsa_handle h, const void *q, const void *k_new, const void *v_new, void *out, void *stream)
{
    int rc = check_step(h, q, k_new, v_new, out);
    if (rc != DSA_OK) return rc;
    return launch_decode_step(h, q, k_new, v_new, out, (cudaStream_t)stream, false);
}

int dsa_decode_step_fused(dsa_handle h, dsa_proj pr, const void *x, const void *W, void *out, void *stream)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    int batch = 0, heads = 0, hd = 0;
    int rc = dsa_detail::proj_shape(pr, &batch, &heads, &hd);
    if (rc != DSA_OK) return rc;
    if (h->dtype != DSA_BF16 && h->dtype != DSA_FP8_E4M3)
        return fail(DSA_ERR_ARG, "dsa_decode_step_fused needs a DSA_BF16 or DSA_FP8_E4M3 handle");
    if ((long long)batch * heads != h->S || hd != h->D)
        return fail(DSA_ERR_ARG, "handle (%d streams of %d) and projection (%d x %d heads of %d) do not match", h->S,
                    h->D, batch, heads, hd);
    void *q = nullptr;  // k_new and v_new are written to the decode state (below)
    dsa_detail::proj_staging(pr, &q);
    rc = check_step(h, q, q, q, out);
    if (rc != DSA_OK) return rc;
    if (h->graph_mode)
        return fail(DSA_ERR_STATE, "dsa_decode_step_fused takes host-counted steps: switch graph mode off first");
    if ((long long)h->L_p + h->t > INT_MAX) return fail(DSA_ERR_STATE, "position out of range");
    cudaStream_t st = (cudaStream_t)stream;
    // The projection's epilogue writes k and v of the newest token straight
    // into the slot it takes at this step (ring slot t' mod R, or prefix row
    // L_p + t during the sink fill), K row then V row of each entry, in the
    // stored form (E4M3 codes with the stream's inverse scales for FP8
    // storage); the decode kernel reads them there and appends nothing.
    const size_t row = 2 * (size_t)h->D * elem_bytes(h->dtype);  // bytes of a K|V entry
    unsigned char *kdst;
    long long stride;  // bytes (= elements) between streams' entries, in stored elements
    if (h->t < h->sink) {
        kdst = static_cast<unsigned char *>(h->prefix) + (size_t)(h->L_p + h->t) * row;
        stride = (long long)h->Lcap * 2 * h->D;
    } else {
        kdst = static_cast<unsigned char *>(h->ring) + (size_t)((h->t - h->sink) % h->R) * row;
        stride = (long long)h->R * 2 * h->D;
    }
    if (stride > INT_MAX) return fail(DSA_ERR_ARG, "decode state rows too long for the fused step");
    unsigned char *vdst = kdst + (size_t)h->D * elem_bytes(h->dtype);
    const float *kinv = h->scales ? h->scales + 2 * (size_t)h->S : nullptr;
    const float *vinv = h->scales ? h->scales + 3 * (size_t)h->S : nullptr;
    rc = dsa_detail::proj_launch(pr, x, W, h->L_p + h->t, q, kdst, vdst, st, (int)stride, (int)stride, kinv, vinv);
    if (rc != DSA_OK) return rc;
    return launch_decode_step(h, q, kdst, vdst, out, st, true, true);
}

int dsa_get_step(dsa_handle h, int *t)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    if (!t) return fail(DSA_ERR_ARG, "t is NULL");
    *t = h->t;
    return DSA_OK;
}

int dsa_get_skip_mask(dsa_handle h, uint32_t *host_dst, void *stream)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    if (!host_dst) return fail(DSA_ERR_ARG, "host_dst is NULL");
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(host_dst, h->mask, (size_t)h->S * h->MW * 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, "skip mask copy");
}

int dsa_get_last_selection(dsa_handle h, int32_t *host_dst, void *stream)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    if (!host_dst) return fail(DSA_ERR_ARG, "host_dst is NULL");
    if (!h->last_select) {
        for (int i = 0; i < h->S; ++i) host_dst[i] = -1;
        return DSA_OK;
    }
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(host_dst, h->last_sel, (size_t)h->S * 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, "last selection copy");
}

int dsa_sync_status(dsa_handle h, void *stream)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    cudaStream_t st = (cudaStream_t)stream;
    int word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, h->status, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "status copy");
    if (word & dsa::ST_TIMEOUT) return fail(DSA_ERR_TIMEOUT, "a bounded wait in the decode kernel gave up");
    if (word & dsa::ST_CHECK) return fail(DSA_ERR_DEVICE_CHECK, "device consistency check failed (skip mask count)");
    return DSA_OK;
}

int dsa_set_splits(dsa_handle h, int nsplit)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    if (nsplit < 0) return fail(DSA_ERR_ARG, "nsplit must be >= 0");
    if (nsplit > 0) {
        int rc = ensure_partials(h, nsplit);
        if (rc != DSA_OK) return rc;
    }
    h->forced_split = nsplit;
    return DSA_OK;
}

int dsa_set_merge(dsa_handle h, int mode)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    if (mode != 0 && mode != 1) return fail(DSA_ERR_ARG, "merge mode must be 0 or 1 (got %d)", mode);
    h->merge_launch_only = mode;
    return DSA_OK;
}

int dsa_set_pipeline(dsa_handle h, int pipeline)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    if (pipeline < 0 || pipeline > dsa::kPipelines)
        return fail(DSA_ERR_ARG, "pipeline must be 0 .. %d (got %d)", dsa::kPipelines, pipeline);
    if (pipeline > 0 && h->ctas_per_sm[pipeline - 1] < 1)
        return fail(DSA_ERR_ARG, "pipeline %d cannot be launched on this device", pipeline);
    h->forced_pipe = pipeline;
    return DSA_OK;
}

int dsa_set_kv_scales(dsa_handle h, const float *k_scale, const float *v_scale)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    if (h->dtype != DSA_FP8_E4M3) return fail(DSA_ERR_ARG, "KV scales apply to DSA_FP8_E4M3 handles only");
    if (!k_scale || !v_scale) return fail(DSA_ERR_ARG, "k_scale and v_scale must be non-NULL");
    for (int i = 0; i < h->S; ++i)
        if (!(k_scale[i] > 0.0f) || !(v_scale[i] > 0.0f) || std::isinf(k_scale[i]) || std::isinf(v_scale[i]))
            return fail(DSA_ERR_ARG, "scales must be positive and finite (stream %d: %g, %g)", i, k_scale[i], v_scale[i]);
    // Kernels of earlier steps may still read the scales.
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    int rc = upload_scales(h, k_scale, v_scale);
    if (rc != DSA_OK) return rc;
    h->prefilled = 0;  // rows stored with the old scales are gone: dsa_prefill must follow
    return DSA_OK;
}

int dsa_set_graph_mode(dsa_handle h, int on)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    if (!on) {
        h->graph_mode = 0;
        return DSA_OK;
    }
    if (!h->step_dev) {
        int rc = dev_alloc((void **)&h->step_dev, 2 * sizeof(int), "device step counter");
        if (rc != DSA_OK) return rc;
    }
    // Earlier launches may still be in flight; the counter starts at the host's step.
    cudaError_t e = cudaDeviceSynchronize();
    const int init[2] = {h->t, 0};
    if (e == cudaSuccess) e = cudaMemcpy(h->step_dev, init, sizeof init, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "device step counter");
    h->graph_mode = 1;
    return DSA_OK;
}

int dsa_sync_step(dsa_handle h, void *stream)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    if (!h->graph_mode) return DSA_OK;
    int t = 0;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(&t, h->step_dev, sizeof t, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "device step copy");
    h->t = t;
    return DSA_OK;
}

int dsa_debug_copy_state(dsa_handle h, void *host_prefix, void *host_ring)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    const size_t row = 2 * (size_t)h->D * elem_bytes(h->dtype);
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess && host_prefix)
        e = cudaMemcpy(host_prefix, h->prefix, (size_t)h->S * h->Lcap * row, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && host_ring)
        e = cudaMemcpy(host_ring, h->ring, (size_t)h->S * h->R * row, cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, "state copy");
}

int dsa_debug_set_step(dsa_handle h, int t, void *stream)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    if (h->A != h->R) return fail(DSA_ERR_ARG, "dsa_debug_set_step needs N_att == N_r (no selection)");
    if (t < 0) return fail(DSA_ERR_ARG, "t must be >= 0 (got %d)", t);
    if (!h->prefilled || h->t != 0 || h->graph_mode)
        return fail(DSA_ERR_STATE, "dsa_debug_set_step needs a handle at step 0 after dsa_prefill, not in graph mode");
    cudaStream_t st = (cudaStream_t)stream;
    const size_t row = 2 * (size_t)h->D * elem_bytes(h->dtype);
    cudaError_t e = cudaMemsetAsync(h->ring, 0, (size_t)h->S * h->R * row, st);
    if (e == cudaSuccess && h->sink > 0)
        e = cudaMemset2DAsync(static_cast<unsigned char *>(h->prefix) + (size_t)h->L_p * row, (size_t)h->Lcap * row, 0,
                              (size_t)h->sink * row, (size_t)h->S, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    note_launch(st, h);
    h->t = t;
    return DSA_OK;
}

int dsa_set_wait_limit(dsa_handle h, uint32_t limit)
{
    if (!valid(h)) return fail(DSA_ERR_STATE, "invalid handle");
    h->wait_limit = limit;
    return DSA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free decode step.
//
// Some callers cannot allocate device memory when they decode: a serving
// engine that reserves all device memory up front for its own KV arena and
// forbids libraries from taking more, or code that must not call the
// allocator from its decode loop (allocation can synchronize the device).
// For them, dsa_decode_step_noalloc runs the same decode kernel on state
// buffers the caller owns; the only scratch it needs (the per-split partial
// results of split streams and a status word) lives in the
// file-scope array below, which every GPU that loads this library holds
// until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];
int g_noalloc_sms[kMaxDevices];

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Scratch layout for `heads` streams with `nsplit` partial slots each:
// status word, (m, l) and argmin partials, accumulator partials.
size_t noalloc_scratch_bytes(int heads, int nsplit, int D)
{
    const size_t slots = (size_t)heads * nsplit;
    return 256 + round256(slots * 8) * 2 + round256(slots * D * 4);
}

// Device address of the scratch array on the current device (looked up once
// per device) and the device's SM count.
int noalloc_setup(void **ptr, int *sms)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(DSA_ERR_CUDA, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return cuda_fail(e, "cudaGetSymbolAddress of the static scratch");
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        g_noalloc_sms[dev] = n;
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    *sms = g_noalloc_sms[dev];
    return DSA_OK;
}

}  // namespace

extern "C" int dsa_decode_step_noalloc(int heads, int head_dim, int L_p, int N_r, int N_att, int sink, int dtype,
                                       int t, void *prefix, void *ring, uint32_t *mask, int32_t *last_sel,
                                       const void *q, const void *k_new, const void *v_new, void *out, void *stream)
{
    int rc = validate(heads, head_dim, L_p, N_r, N_att, sink, dtype);
    if (rc != DSA_OK) return rc;
    if (dtype == DSA_FP8_E4M3)
        return fail(DSA_ERR_ARG, "dsa_decode_step_noalloc: FP8 storage needs per-stream scales; use the handle API");
    if (t < 0) return fail(DSA_ERR_ARG, "t must be >= 0 (got %d)", t);

    void *scratch = nullptr;
    int sms = 0;
    rc = noalloc_setup(&scratch, &sms);
    if (rc != DSA_OK) return rc;
    int occ[dsa::kPipelines];
    rc = query_occupancy(dtype, head_dim, occ);
    if (rc != DSA_OK) return rc;

    // A handle-shaped description of the caller's state; nothing is allocated.
    dsa_ctx h{};
    describe(h, heads, head_dim, L_p, N_r, N_att, sink, dtype);
    h.sm_count = sms;
    for (int pi = 0; pi < dsa::kPipelines; ++pi) h.ctas_per_sm[pi] = occ[pi];
    const Plan pl = make_plan(&h, t);
    // Split streams keep their partials in the static scratch; a step that
    // needs more than it holds is refused (before any pointer is used).
    if ((long long)pl.nsplit * heads > INT_MAX) return fail(DSA_ERR_ARG, "grid too large");
    const size_t need = pl.nsplit > 1 ? noalloc_scratch_bytes(heads, pl.nsplit, head_dim) : 256;
    if (need > kNoAllocScratchBytes)
        return fail(DSA_ERR_ARG,
                    "dsa_decode_step_noalloc: %d streams in %d work items each need %zu bytes of scratch, more than "
                    "the static %zu bytes; use the handle API (dsa_create / dsa_decode_step) for this size",
                    heads, pl.nsplit, need, kNoAllocScratchBytes);

    if (!ring || !mask || !last_sel || !q || !k_new || !v_new || !out || (L_p + sink > 0 && !prefix))
        return fail(DSA_ERR_ARG, "state and input/output pointers must be non-NULL");
    if (!aligned16(prefix) || !aligned16(ring) || !aligned16(q) || !aligned16(k_new) || !aligned16(v_new) ||
        !aligned16(out) || ((uintptr_t)mask & 3u) || ((uintptr_t)last_sel & 3u))
        return fail(DSA_ERR_ARG, "data pointers must be 16-byte aligned (mask and last_sel 4-byte aligned)");
    h.prefix = prefix;
    h.ring = ring;
    rc = encode_ring_map(&h);
    if (rc != DSA_OK) return rc;

    unsigned char *base = static_cast<unsigned char *>(scratch);
    const size_t slots = (size_t)heads * pl.nsplit;
    int *status = reinterpret_cast<int *>(base);
    float2 *part_ml = reinterpret_cast<float2 *>(base + 256);
    float2 *part_min = reinterpret_cast<float2 *>(reinterpret_cast<unsigned char *>(part_ml) + round256(slots * 8));
    float *part_acc = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(part_min) + round256(slots * 8));

    cudaStream_t st = (cudaStream_t)stream;
    // The status word must start at zero; the partials are fully written
    // before they are read.
    cudaError_t e = cudaMemsetAsync(scratch, 0, 256, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync of the static scratch");

    dsa::DecodeParams p;
    p.q = q;
    p.knew = k_new;
    p.vnew = v_new;
    p.out = out;
    p.prefix = prefix;
    p.ring = ring;
    p.mask = mask;
    p.last_sel = last_sel;
    p.part_acc = part_acc;
    p.part_ml = part_ml;
    p.part_min = part_min;
    p.status = status;
    p.S = heads;
    p.Lcap = h.Lcap;
    p.P = pl.P;
    p.sinkmode = pl.sinkmode;
    p.R = h.R;
    p.tin = pl.tin;
    p.tin_mod = pl.tin >= 0 ? pl.tin % h.R : 0;
    p.wlen = pl.wlen;
    p.a = pl.a;
    p.n = pl.n;
    p.nsplit = pl.nsplit;
    p.nbuf = pl.nbuf;
    p.chunk = pl.chunk;
    p.pstride = pl.nsplit;
    p.nitems = pl.nitems;
    p.noskip = (h.A == h.R) ? 1 : 0;
    p.select = pl.select;
    p.MW = h.MW;
    p.qscale = (float)(1.4426950408889634 / std::sqrt((double)head_dim));
    p.kscale = p.vscale = p.kinv = p.vinv = nullptr;
    p.wait_limit = kDefaultWaitLimit;
    p.step_dev = nullptr;
    p.sink = sink;
    p.early = 0;  // caller-owned state: the previous kernel may have written it
    p.glist = nullptr;  // no stored list: the offsets are listed from the mask every step
    p.LS = 0;
    p.list_mode = 0;
    p.appended = 0;
    p.cta_merge = 0;  // split partials in the static scratch, merged by merge_kernel
    e = launch_step(dtype, head_dim, pl.shape, p, h.ring_map, pl.grid, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return DSA_OK;
}

extern "C" int dsa_decode_step_noalloc_status(void *stream)
{
    void *scratch = nullptr;
    int sms = 0;
    int rc = noalloc_setup(&scratch, &sms);
    if (rc != DSA_OK) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    int word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, scratch, sizeof word, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "status copy from the static scratch");
    if (word & dsa::ST_TIMEOUT) return fail(DSA_ERR_TIMEOUT, "a bounded wait in the decode kernel gave up");
    if (word & dsa::ST_CHECK) return fail(DSA_ERR_DEVICE_CHECK, "device consistency check failed (skip mask count)");
    return DSA_OK;
}
