// C ABI of libr9q (declared in include/r9q.h): argument checks, planning and
// dispatch to the sm_103a kernels.  Host code only; every call is
// asynchronous on the caller's stream and allocates nothing.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "r9q.h"
#include "r9q_kernels.h"

namespace r9q {

// device error word: kernels record a bounded-wait timeout here
__device__ int g_dev_err = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kSmemLimit = 227 * 1024;

struct DeviceInfo {
    std::once_flag once;
    int status = R9Q_OK;
    int sms = 0;
    int* err = nullptr;
};
DeviceInfo g_dev[kMaxDevices];

int current_device(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return R9Q_ERR_DEVICE;
    if (dev < 0 || dev >= kMaxDevices) return R9Q_ERR_DEVICE;
    DeviceInfo& d = g_dev[dev];
    std::call_once(d.once, [&d, dev]() {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            d.status = R9Q_ERR_DEVICE;
            return;
        }
        if (major != 10 || minor != 3) {     // the library carries sm_103a code only
            d.status = R9Q_ERR_DEVICE;
            return;
        }
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dev_err) != cudaSuccess) {
            (void)cudaGetLastError();   // no pending error is left for the caller
            d.status = R9Q_ERR_LAUNCH;
            return;
        }
        d.err = static_cast<int*>(p);
        d.sms = sms;
    });
    *out = &d;
    return d.status;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Tensor map over an e4m3 weight matrix w[N][K]: boxes of 64 rows x 128 bytes,
// 128-byte swizzle (the layout the stream kernel's ldmatrix addressing expects).
int weight_tmap(const uint8_t* w, int64_t N, int64_t K, CUtensorMap* tm) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return R9Q_ERR_LAUNCH;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)K};
    cuuint32_t box[2] = {128, 64};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? R9Q_OK : R9Q_ERR_LAUNCH;
}

int tmap_2d(const void* base, CUtensorMapDataType dt, int esize, int64_t rows, int64_t cols, int box_cols,
            int box_rows, CUtensorMap* tm) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return R9Q_ERR_LAUNCH;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols * esize)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? R9Q_OK : R9Q_ERR_LAUNCH;
}

// R9Q_TC_SPLITK=0 keeps every tensor-core W8A8 call on persistent whole-K tiles
// (tests and benches only).
bool env_tc_splitk() {
    static int v = -1;
    if (v < 0) {
        const char* s = std::getenv("R9Q_TC_SPLITK");
        v = (s && std::atoi(s) == 0) ? 0 : 1;
    }
    return v != 0;
}

// Workspace of the tensor-core W8A8 path.  Counters first, in a fixed
// 64 KiB header (so that calls of any shape sharing one workspace find them
// where the previous call left them at zero): [ready m-tiles][done tiles]
// [exits] int32; then [aq M x K][as M x KB fp32][split-K partials tiles x S x
// 128 x 256 fp32] (aq/as only when the caller does not take them, partials
// only with split-K).  Shapes with more counters than the header holds keep
// them after the header and have them zeroed before every launch.
constexpr size_t kCounterHeader = 64 * 1024;
struct TcScratch {
    size_t ready, done, exits, counters_end;   // counters
    bool self_reset;                           // counters in the header, returned to zero by the kernel
    size_t aq, as, part, total;
};
TcScratch tc_scratch(int64_t M, int64_t N, int64_t K, bool need_aq, int splits) {
    TcScratch t;
    const size_t mtiles = (size_t)((M + 127) / 128), tiles = mtiles * (size_t)((N + 255) / 256);
    const size_t ncnt = mtiles + (splits > 1 ? tiles : 0) + 1;
    t.self_reset = ncnt * 4 <= kCounterHeader;
    size_t base = kCounterHeader;
    if (t.self_reset) {
        t.ready = 0;
    } else {
        t.ready = base;
        base = align256(base + ncnt * 4);
    }
    t.done = t.ready + mtiles * 4;
    t.exits = t.done + (splits > 1 ? tiles * 4 : 0);
    t.counters_end = t.exits + 4;
    t.aq = base;
    t.as = t.aq + (need_aq ? align256((size_t)(M * K)) : 0);
    t.part = t.as + (need_aq ? align256((size_t)M * (K / 128) * 4) : 0);
    t.total = t.part + (splits > 1 ? tiles * (size_t)splits * 128 * 256 * 4 : 0);
    return t;
}

// Split-K ranks the tensor-core path uses for (M, N, K) on the current device
// (R9Q_TC_SPLITK=0: always 1).  Without a device the SM count of a GB300 is
// assumed, which only matters for workspace queries made without a GPU.
int tc_splits_for(int64_t M, int64_t N, int64_t K) {
    int sms = 152;
    DeviceInfo* d = nullptr;
    if (current_device(&d) == R9Q_OK) sms = d->sms;
    return env_tc_splitk() ? tc_plan_splits(M, N, K, sms) : 1;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    if (!a || !b) return false;
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bn && y < x + an;
}

int check_mnk(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 128 || K < 128 || N % 128 || K % 128) return R9Q_ERR_DIM;
    if (M > (int64_t)64 * 65535 || N / 128 > 65535 || K > ((int64_t)1 << 30)) return R9Q_ERR_DIM;
    return R9Q_OK;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? R9Q_OK : R9Q_ERR_LAUNCH; }

std::atomic<int> g_pdl{0};

// Tuning override "S,G,stages" for tests and benches (R9Q_PLAN); 0 fields = planner's choice.
void env_plan(int* S, int* G, int* st) {
    static int v[3] = {-1, 0, 0};
    if (v[0] < 0) {
        v[0] = v[1] = v[2] = 0;
        if (const char* s = std::getenv("R9Q_PLAN")) std::sscanf(s, "%d,%d,%d", &v[0], &v[1], &v[2]);
    }
    *S = v[0];
    *G = v[1];
    *st = v[2];
}

// Smallest M of the tensor-core W8A8 path; R9Q_TC_MIN_M overrides it (tests and benches only).
int tc_min_m() {
    static int v = -1;
    if (v < 0) {
        const char* s = std::getenv("R9Q_TC_MIN_M");
        v = s ? std::atoi(s) : kTcMinM;
        if (v < 1) v = kTcMinM;
    }
    return v;
}

int env_splits() {
    static int v = -1;
    if (v < 0) {
        const char* s = std::getenv("R9Q_SPLITS");   // tuning override for tests and benches
        v = s ? std::atoi(s) : 0;
        if (v < 0) v = 0;
    }
    return v;
}

// Scratch of the expert MLP: [gu (unfused)] [h unless given] [hq, hs (unfused W8A8, unless given)]
size_t mlp_workspace(int64_t M, int64_t I, int flags, bool have_h, bool have_hq) {
    const bool unfused = flags & R9Q_MLP_UNFUSED;
    const bool wonly = flags & R9Q_MLP_WEIGHT_ONLY;
    size_t b = 0;
    if (unfused) b += align256((size_t)M * 2 * I * 2);
    if (!have_h) b += align256((size_t)M * I * 2);
    if (unfused && !wonly && !have_hq) b += align256((size_t)M * I) + align256((size_t)M * (I / 128) * 4);
    return b;
}

}  // namespace

// ------------------------------------------------------------ planning --

size_t stream_smem_bytes(int MT, int amode, int S, int kbs_max, int ntl_max, int stages) {
    const size_t kslice = (size_t)kbs_max * 128;
    const size_t npbuf = ntl_max > 1 ? 2 : 1;
    const size_t recv = npbuf * (size_t)S * stream_recv_rows(S) * MT * 4;
    const size_t scales = 4 * ((size_t)ntl_max * 2 * kbs_max + (size_t)MT * kbs_max);
    if (stream_uses_tc(MT, amode)) {
        // tcgen05 body, in order: weight ring, activation rows (later more
        // ring stages), B tile, barriers, receive buffers, scales; the first
        // three stay 1024-aligned
        const size_t act = (size_t)MT * ((amode == A_PREQ) ? kslice : 2 * kslice);
        const size_t bop = kslice * (size_t)stream_mma_n(MT);
        return 1024 + (size_t)stages * kStageBytes + act + bop + kBarBytes + recv + scales;
    }
    // mma.sync body, in order: weight ring, barriers, receive buffers, scales,
    // activation rows (padded so the B-fragment loads of the rows fall on
    // distinct banks)
    const size_t act_ld = (amode == A_QUANT) ? 2 * kslice + 16 : (amode == A_BF16) ? 2 * kslice + 32 : kslice + 16;
    size_t off = (size_t)stages * kStageBytes + kBarBytes + recv + scales;
    off = (off + 15) & ~static_cast<size_t>(15);
    return 1024 + off + (size_t)MT * act_ld;
}

bool plan_stream(int64_t M, int64_t N, int64_t K, int amode_launch, int sms, StreamPlan* plan) {
    // The split count fixes the fp32 summation order.  Fused (A_QUANT) and
    // unfused (A_PREQ) W8A8 calls must sum identically, so both are planned
    // with the fused A-load's shared-memory needs.
    const int amode = (amode_launch == A_PREQ) ? A_QUANT : amode_launch;
    const int MT = M <= 8 ? 8 : M <= 16 ? 16 : M <= 32 ? 32 : 64;
    const int ntiles = (int)(N / 128);
    const int mchunks = (int)((M + MT - 1) / MT);
    const int KB = (int)(K / 128);
    const int maxS = KB < kMaxSplits ? KB : kMaxSplits;
    const int per_sm_cap = stream_min_blocks(MT, amode);   // register-limited residency
    const int forced = env_splits();
    // Candidates: S | KB (S <= 8), G | ntiles, ring depth 4..2.  Keep every CTA
    // co-resident; among those take the most CTAs (up to two per SM), then
    // the deeper ring, then fewer splits.
    int bS = -1, bG = -1, bst = -1;
    long best_score = -1;
    for (int S = 1; S <= maxS; ++S) {
        if (KB % S) continue;
        if (forced && S != forced) continue;
        for (int G = 1; G <= ntiles; ++G) {
            if (ntiles % G) continue;
            const int ntl_max = ntiles / G;
            for (int st = kMaxStages; st >= 2; --st) {
                const size_t smem = stream_smem_bytes(MT, amode, S, KB / S, ntl_max, st);
                if (smem > kSmemLimit) continue;
                int per_sm = (int)((228 * 1024) / (smem + 1024));
                if (per_sm > per_sm_cap) per_sm = per_sm_cap;
                const int64_t ctas = (int64_t)S * G * mchunks;
                if (ctas > (int64_t)sms * per_sm) continue;
                const int64_t useful = ctas < 2 * (int64_t)sms ? ctas : 2 * (int64_t)sms;
                const long score = (long)useful * 64 + st * 8 - S;
                if (score > best_score) {
                    best_score = score;
                    bS = S;
                    bG = G;
                    bst = st;
                }
                break;   // deepest ring that fits for this (S, G)
            }
        }
    }
    if (bS < 0) {
        // not co-resident at any split: one tile per cluster, the smallest split that fits
        for (int S = 1; S <= maxS && bS < 0; ++S) {
            if (KB % S) continue;
            for (int st = kMaxStages; st >= 2; --st)
                if (stream_smem_bytes(MT, amode, S, KB / S, 1, st) <= kSmemLimit) {
                    bS = S;
                    bG = ntiles;
                    bst = st;
                    break;
                }
        }
    }
    {
        int fS, fG, fst;
        env_plan(&fS, &fG, &fst);
        if (fS > 0 && fS <= maxS && KB % fS == 0 && fG > 0 && ntiles % fG == 0 && fst >= 2 && fst <= kMaxStages &&
            stream_smem_bytes(MT, amode, fS, KB / fS, ntiles / fG, fst) <= kSmemLimit) {
            bS = fS;
            bG = fG;
            bst = fst;
        }
    }
    if (bS < 0) return false;
    plan->MT = MT;
    plan->splits = bS;
    plan->groups = bG;
    plan->ntiles = ntiles;
    plan->mchunks = mchunks;
    plan->stages = bst;
    plan->smem = stream_smem_bytes(MT, amode_launch, bS, KB / bS, (ntiles + bG - 1) / bG, bst);
    return true;
}

cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, size_t> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    size_t& cur = done[{dev, kernel}];
    if (cur >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
    if (e == cudaSuccess) cur = kSmemLimit;
    return e;
}

cudaError_t launch_stream(const StreamPlan& plan, int amode, int epi, const CUtensorMap& wmap,
                          const StreamParams& p, cudaStream_t st, bool pdl) {
    switch (amode) {
        case A_QUANT: return launch_stream_a_quant(plan, epi, wmap, p, st, pdl);
        case A_PREQ: return launch_stream_a_preq(plan, epi, wmap, p, st, pdl);
        case A_BF16: return launch_stream_a_bf16(plan, epi, wmap, p, st, pdl);
        default: return cudaErrorInvalidValue;
    }
}

namespace {

// One stream GEMM launch (plain bf16 store or SwiGLU epilogue).
int run_stream_gemm(int amode, int epi, const void* a, uint8_t* aq, float* as, const uint8_t* w,
                    const float* ws, void* y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                    const DeviceInfo* d, cudaStream_t st, bool pdl) {
    StreamPlan plan;
    if (!plan_stream(M, N, K, amode, d->sms, &plan)) return R9Q_ERR_DIM;
    CUtensorMap tm;
    int rc = weight_tmap(w, N, K, &tm);
    if (rc) return rc;
    StreamParams p;
    p.a = static_cast<const uint16_t*>(a);
    p.aq = aq;
    p.as = as;
    p.ws = ws;
    p.y = static_cast<uint16_t*>(y);
    p.M = (int)M;
    p.K = (int)K;
    p.KB = (int)(K / 128);
    p.ldy = (int)ldy;
    p.splits = plan.splits;
    p.groups = plan.groups;
    p.ntiles = plan.ntiles;
    p.stages = plan.stages;
    p.err = d->err;
    return to_status(launch_stream(plan, amode, epi, tm, p, st, pdl));
}

}  // namespace

int device_error_word(int** out) {
    DeviceInfo* d = nullptr;
    const int rc = current_device(&d);
    if (rc) return rc;
    *out = d->err;
    return R9Q_OK;
}

}  // namespace r9q

using namespace r9q;

extern "C" {

int r9q_version(void) { return R9Q_VERSION; }

int r9q_set_pdl(int enable) { return g_pdl.exchange(enable ? 1 : 0); }

const char* r9q_strerror(int code) {
    switch (code) {
        case R9Q_OK: return "ok";
        case R9Q_ERR_NULL: return "a required pointer is NULL";
        case R9Q_ERR_DIM: return "bad or unsupported dimensions (M >= 1; N, K multiples of 128)";
        case R9Q_ERR_ALIGN: return "pointer misaligned (data 16 bytes, scales 4 bytes)";
        case R9Q_ERR_WORKSPACE: return "workspace missing or too small";
        case R9Q_ERR_LAUNCH: return "CUDA launch or runtime error";
        case R9Q_ERR_TIMEOUT: return "a bounded device wait timed out";
        case R9Q_ERR_DEVICE: return "current device is not an sm_103 GPU";
        case R9Q_ERR_ARG: return "invalid argument";
        default: return "unknown error code";
    }
}

int r9q_last_device_error(void* stream) {
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int h = 0;
    if (cudaMemcpyAsync(&h, d->err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return R9Q_ERR_LAUNCH;
    if (cudaStreamSynchronize(st) != cudaSuccess) return R9Q_ERR_LAUNCH;
    if (h != 0) {
        if (cudaMemsetAsync(d->err, 0, sizeof(int), st) != cudaSuccess) return R9Q_ERR_LAUNCH;
        if (cudaStreamSynchronize(st) != cudaSuccess) return R9Q_ERR_LAUNCH;
    }
    return h;
}

int r9q_e4m3_from_f32(const float* x, int64_t n, uint8_t* q, void* stream) {
    if (n < 0) return R9Q_ERR_DIM;
    if (n == 0) return R9Q_OK;
    if (!x || !q) return R9Q_ERR_NULL;
    if (!aligned(x, 16) || !aligned(q, 16)) return R9Q_ERR_ALIGN;
    if (overlaps(x, 4 * (size_t)n, q, (size_t)n)) return R9Q_ERR_ARG;
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc) return rc;
    return to_status(launch_e4m3_from_f32(x, n, q, static_cast<cudaStream_t>(stream), d->sms));
}

int r9q_quant_group128(const void* x_bf16, int64_t M, int64_t K, uint8_t* xq, float* xs, void* stream) {
    if (!x_bf16 || !xq || !xs) return R9Q_ERR_NULL;
    if (M < 1 || K < 128 || K % 128) return R9Q_ERR_DIM;
    if (!aligned(x_bf16, 16) || !aligned(xq, 16) || !aligned(xs, 4)) return R9Q_ERR_ALIGN;
    if (overlaps(x_bf16, 2 * (size_t)(M * K), xq, (size_t)(M * K)) ||
        overlaps(x_bf16, 2 * (size_t)(M * K), xs, 4 * (size_t)(M * (K / 128))))
        return R9Q_ERR_ARG;
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc) return rc;
    return to_status(launch_quant_group128(static_cast<const uint16_t*>(x_bf16), M, K, xq, xs,
                                           static_cast<cudaStream_t>(stream), d->sms));
}

int r9q_swiglu_interleaved(const void* gu_bf16, int64_t M, int64_t I, void* h_bf16, void* stream) {
    if (!gu_bf16 || !h_bf16) return R9Q_ERR_NULL;
    if (M < 1 || I < 128 || I % 128 || M > INT_MAX / 2 || I > INT_MAX / 2) return R9Q_ERR_DIM;
    if (!aligned(gu_bf16, 16) || !aligned(h_bf16, 16)) return R9Q_ERR_ALIGN;
    if (overlaps(gu_bf16, 4 * (size_t)(M * I), h_bf16, 2 * (size_t)(M * I))) return R9Q_ERR_ARG;
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc) return rc;
    return to_status(launch_swiglu_interleaved(static_cast<const uint16_t*>(gu_bf16), M, I,
                                               static_cast<uint16_t*>(h_bf16), static_cast<cudaStream_t>(stream),
                                               d->sms));
}

int r9q_quant_weight_block128(const float* w, int64_t N, int64_t K, uint8_t* wq, float* ws, void* stream) {
    if (!w || !wq || !ws) return R9Q_ERR_NULL;
    if (N < 128 || K < 128 || N % 128 || K % 128 || N / 128 > 65535 || K / 128 > INT_MAX) return R9Q_ERR_DIM;
    if (!aligned(w, 16) || !aligned(wq, 16) || !aligned(ws, 4)) return R9Q_ERR_ALIGN;
    if (overlaps(w, 4 * (size_t)(N * K), wq, (size_t)(N * K))) return R9Q_ERR_ARG;
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc) return rc;
    return to_status(launch_quant_weight_block128(w, N, K, wq, ws, static_cast<cudaStream_t>(stream)));
}

int r9q_grouped_gemm_fp8(const void* a_bf16, const int64_t* offsets, int64_t E, const uint8_t* w, const float* ws,
                         void* y_bf16, int64_t N, int64_t K, int flags, void* stream) {
    if (flags & ~(R9Q_GROUPED_WEIGHT_ONLY | R9Q_GROUPED_SWIGLU)) return R9Q_ERR_ARG;
    if (!offsets) return R9Q_ERR_NULL;
    if (E < 1 || E > kMaxGroups) return R9Q_ERR_DIM;
    if (offsets[0] != 0) return R9Q_ERR_ARG;
    int64_t max_m = 0;
    int active = 0;
    for (int64_t g = 0; g < E; ++g) {
        const int64_t m = offsets[g + 1] - offsets[g];
        if (m < 0) return R9Q_ERR_ARG;
        if (m > max_m) max_m = m;
        active += m > 0;
    }
    const int64_t Mtot = offsets[E];
    if (Mtot > INT_MAX) return R9Q_ERR_DIM;
    if (Mtot == 0) return R9Q_OK;                          // no token routed anywhere
    if (!a_bf16 || !w || !ws || !y_bf16) return R9Q_ERR_NULL;
    const bool swiglu = flags & R9Q_GROUPED_SWIGLU;
    int rc = check_mnk(Mtot, N, K);
    if (rc) return rc;
    if (swiglu && N % 256) return R9Q_ERR_DIM;
    if (E * N > INT_MAX) return R9Q_ERR_DIM;
    if (!aligned(a_bf16, 16) || !aligned(w, 16) || !aligned(y_bf16, 16) || !aligned(ws, 4)) return R9Q_ERR_ALIGN;
    const int64_t ncols = swiglu ? N / 2 : N;
    const size_t ybytes = 2 * (size_t)(Mtot * ncols);
    if (overlaps(y_bf16, ybytes, a_bf16, 2 * (size_t)(Mtot * K)) || overlaps(y_bf16, ybytes, w, (size_t)(E * N * K)))
        return R9Q_ERR_ARG;
    DeviceInfo* d = nullptr;
    rc = current_device(&d);
    if (rc) return rc;
    const int amode = (flags & R9Q_GROUPED_WEIGHT_ONLY) ? A_BF16 : A_QUANT;
    // One expert's GEMM planned as if it had its share of the SMs.
    StreamPlan plan;
    const int share = d->sms / active > 0 ? d->sms / active : 1;
    if (!plan_stream(max_m, N, K, amode, share, &plan)) return R9Q_ERR_DIM;
    GroupTable gt;
    gt.zchunks = (int)((max_m + plan.MT - 1) / plan.MT);
    gt.wrows = (int)N;
    for (int64_t g = 0; g <= E; ++g) gt.off[g] = (int)offsets[g];
    if ((int64_t)E * gt.zchunks > 65535) return R9Q_ERR_DIM;
    CUtensorMap tm;
    rc = weight_tmap(w, E * N, K, &tm);
    if (rc) return rc;
    StreamParams p;
    p.a = static_cast<const uint16_t*>(a_bf16);
    p.aq = nullptr;
    p.as = nullptr;
    p.ws = ws;
    p.y = static_cast<uint16_t*>(y_bf16);
    p.M = (int)Mtot;
    p.K = (int)K;
    p.KB = (int)(K / 128);
    p.ldy = (int)ncols;
    p.splits = plan.splits;
    p.groups = plan.groups;
    p.ntiles = plan.ntiles;
    p.stages = plan.stages;
    p.err = d->err;
    return to_status(launch_stream_grouped(plan, amode, swiglu ? EPI_SWIGLU : EPI_STORE, tm, p, gt, (int)E,
                                           static_cast<cudaStream_t>(stream), g_pdl.load() != 0));
}

int r9q_workspace_bytes(int op, int64_t M, int64_t N, int64_t K, int64_t N2, int flags, size_t* bytes) {
    if (!bytes) return R9Q_ERR_NULL;
    switch (op) {
        case R9Q_OP_GEMM_W8A8:
        case R9Q_OP_GEMM_W8BF16: {
            int rc = check_mnk(M, N, K);
            if (rc) return rc;
            // decode widths: split-K is reduced in distributed shared memory (no
            // scratch); W8A8 above 64 rows quantises A once into scratch
            *bytes = (op == R9Q_OP_GEMM_W8A8 && M >= tc_min_m() && K / 128 <= tc_max_kb())
                         ? tc_scratch(M, N, K, true, tc_splits_for(M, N, K)).total
                         : 0;
            return R9Q_OK;
        }
        case R9Q_OP_GATE_UP_SWIGLU_DOWN: {
            if (flags & ~(R9Q_MLP_WEIGHT_ONLY | R9Q_MLP_UNFUSED)) return R9Q_ERR_ARG;
            int rc = check_mnk(M, 2 * N, K);
            if (!rc) rc = check_mnk(M, N2, N);
            if (rc) return rc;
            *bytes = mlp_workspace(M, N, flags, false, false);
            return R9Q_OK;
        }
        default: return R9Q_ERR_ARG;
    }
}

int r9q_gemm_fp8_block_qa(const void* a_bf16, uint8_t* aq, float* as, const uint8_t* w, const float* ws,
                          void* y_bf16, int64_t M, int64_t N, int64_t K, void* workspace,
                          size_t workspace_bytes, void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    if (!w || !ws || !y_bf16) return R9Q_ERR_NULL;
    if (!a_bf16 && (!aq || !as)) return R9Q_ERR_NULL;
    if (a_bf16 && ((aq == nullptr) != (as == nullptr))) return R9Q_ERR_ARG;
    int rc = check_mnk(M, N, K);
    if (rc) return rc;
    if (!aligned(a_bf16, 16) || !aligned(aq, 16) || !aligned(w, 16) || !aligned(y_bf16, 16) ||
        !aligned(as, 4) || !aligned(ws, 4))
        return R9Q_ERR_ALIGN;
    const size_t ybytes = 2 * (size_t)(M * N);
    if (overlaps(y_bf16, ybytes, a_bf16, 2 * (size_t)(M * K)) || overlaps(y_bf16, ybytes, aq, (size_t)(M * K)) ||
        overlaps(y_bf16, ybytes, w, (size_t)(N * K)) || overlaps(y_bf16, ybytes, as, 4 * (size_t)(M * (K / 128))))
        return R9Q_ERR_ARG;
    if (a_bf16 && aq && (overlaps(aq, (size_t)(M * K), a_bf16, 2 * (size_t)(M * K)) ||
                         overlaps(aq, (size_t)(M * K), w, (size_t)(N * K))))
        return R9Q_ERR_ARG;
    DeviceInfo* d = nullptr;
    rc = current_device(&d);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool tc_path = M >= tc_min_m() && K / 128 <= tc_max_kb();
    // a few tiles: split-K over the SMs (tc_plan_splits)
    const int splits = tc_path ? (env_tc_splitk() ? tc_plan_splits(M, N, K, d->sms) : 1) : 1;
    if (tc_path) {
        // tensor-core path: needs scratch for the ready counters, for the
        // quantised A unless the caller asked for aq/as as outputs, and for
        // the split-K partials
        const bool need_aq = a_bf16 && !aq;
        const TcScratch sc = tc_scratch(M, N, K, need_aq, splits);
        const size_t need = (a_bf16 || splits > 1) ? sc.total : 0;
        if (need > 0 && (!workspace || workspace_bytes < need)) return R9Q_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return R9Q_ERR_ALIGN;
        if (need > 0 && (overlaps(workspace, need, y_bf16, ybytes) || overlaps(workspace, need, a_bf16, 2 * (size_t)(M * K)) ||
                         overlaps(workspace, need, w, (size_t)(N * K))))
            return R9Q_ERR_ARG;
    }
    if (!tc_path)
        return run_stream_gemm(a_bf16 ? A_QUANT : A_PREQ, EPI_STORE, a_bf16, aq, as, w, ws, y_bf16, N, M, N, K, d, st,
                               g_pdl.load() != 0);

    const bool need_aq = a_bf16 && !aq;
    const TcScratch sc = tc_scratch(M, N, K, need_aq, splits);
    uint8_t* wsp = static_cast<uint8_t*>(workspace);
    uint8_t* aq_buf = need_aq ? wsp + sc.aq : aq;
    float* as_buf = need_aq ? reinterpret_cast<float*>(wsp + sc.as) : as;
    int* ready = a_bf16 ? reinterpret_cast<int*>(wsp + sc.ready) : nullptr;
    int* done = splits > 1 ? reinterpret_cast<int*>(wsp + sc.done) : nullptr;
    float* part = splits > 1 ? reinterpret_cast<float*>(wsp + sc.part) : nullptr;
    int* exits = (ready || done) && sc.self_reset ? reinterpret_cast<int*>(wsp + sc.exits) : nullptr;
    CUtensorMap amap, bmap, ymap;
    if ((rc = tmap_2d(aq_buf, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, M, K, 128, 128, &amap)) != 0) return rc;
    if ((rc = tmap_2d(w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, N, K, 128, 256, &bmap)) != 0) return rc;
    if ((rc = tmap_2d(y_bf16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, N, 64, 128, &ymap)) != 0) return rc;
    if ((ready || done) && !sc.self_reset &&
        cudaMemsetAsync(wsp + sc.ready, 0, sc.counters_end - sc.ready, st) != cudaSuccess)
        return R9Q_ERR_LAUNCH;
    return to_status(launch_tc_gemm(amap, bmap, ymap, static_cast<const uint16_t*>(a_bf16), aq_buf, as_buf, ws, ready,
                                    static_cast<uint16_t*>(y_bf16), splits, part, done, exits, (int)M, (int)N, (int)K,
                                    d->err, d->sms, st));
}

int r9q_gemm_fp8w_bf16a(const void* a_bf16, const uint8_t* w, const float* ws, void* y_bf16, int64_t M,
                        int64_t N, int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    if (!a_bf16 || !w || !ws || !y_bf16) return R9Q_ERR_NULL;
    int rc = check_mnk(M, N, K);
    if (rc) return rc;
    if (!aligned(a_bf16, 16) || !aligned(w, 16) || !aligned(y_bf16, 16) || !aligned(ws, 4)) return R9Q_ERR_ALIGN;
    const size_t ybytes = 2 * (size_t)(M * N);
    if (overlaps(y_bf16, ybytes, a_bf16, 2 * (size_t)(M * K)) || overlaps(y_bf16, ybytes, w, (size_t)(N * K)))
        return R9Q_ERR_ARG;
    DeviceInfo* d = nullptr;
    rc = current_device(&d);
    if (rc) return rc;
    return run_stream_gemm(A_BF16, EPI_STORE, a_bf16, nullptr, nullptr, w, ws, y_bf16, N, M, N, K, d,
                           static_cast<cudaStream_t>(stream), g_pdl.load() != 0);
}

int r9q_gate_up_swiglu_down(const void* x_bf16, const uint8_t* w_gu, const float* s_gu, const uint8_t* w_dn,
                            const float* s_dn, void* y_bf16, int64_t M, int64_t H, int64_t I, int64_t H_out,
                            void* h_bf16_out, uint8_t* hq_out, float* hs_out, int flags, void* workspace,
                            size_t workspace_bytes, void* stream) {
    if (!x_bf16 || !w_gu || !s_gu || !w_dn || !s_dn || !y_bf16) return R9Q_ERR_NULL;
    if (flags & ~(R9Q_MLP_WEIGHT_ONLY | R9Q_MLP_UNFUSED)) return R9Q_ERR_ARG;
    const bool wonly = flags & R9Q_MLP_WEIGHT_ONLY;
    const bool unfused = flags & R9Q_MLP_UNFUSED;
    if ((hq_out == nullptr) != (hs_out == nullptr)) return R9Q_ERR_ARG;
    if (wonly && hq_out) return R9Q_ERR_ARG;
    int rc = check_mnk(M, 2 * I, H);
    if (!rc) rc = check_mnk(M, H_out, I);
    if (rc) return rc;
    if (!aligned(x_bf16, 16) || !aligned(w_gu, 16) || !aligned(w_dn, 16) || !aligned(y_bf16, 16) ||
        !aligned(h_bf16_out, 16) || !aligned(hq_out, 16) || !aligned(s_gu, 4) || !aligned(s_dn, 4) ||
        !aligned(hs_out, 4) || !aligned(workspace, 256))
        return R9Q_ERR_ALIGN;
    const size_t need = mlp_workspace(M, I, flags, h_bf16_out != nullptr, hq_out != nullptr);
    if (need > 0 && (!workspace || workspace_bytes < need)) return R9Q_ERR_WORKSPACE;
    const size_t ybytes = 2 * (size_t)(M * H_out);
    if (overlaps(y_bf16, ybytes, x_bf16, 2 * (size_t)(M * H)) || overlaps(y_bf16, ybytes, h_bf16_out, 2 * (size_t)(M * I)) ||
        overlaps(y_bf16, ybytes, workspace, need))
        return R9Q_ERR_ARG;
    DeviceInfo* d = nullptr;
    rc = current_device(&d);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // carve the workspace
    uint8_t* wsp = static_cast<uint8_t*>(workspace);
    size_t off = 0;
    void* gu = nullptr;
    if (unfused) {
        gu = wsp + off;
        off += align256((size_t)M * 2 * I * 2);
    }
    void* h = h_bf16_out;
    if (!h) {
        h = wsp + off;
        off += align256((size_t)M * I * 2);
    }
    uint8_t* hq = hq_out;
    float* hs = hs_out;
    if (unfused && !wonly && !hq) {
        hq = wsp + off;
        off += align256((size_t)M * I);
        hs = reinterpret_cast<float*>(wsp + off);
        off += align256((size_t)M * (I / 128) * 4);
    }

    const int amode = wonly ? A_BF16 : A_QUANT;
    if (!unfused) {
        rc = run_stream_gemm(amode, EPI_SWIGLU, x_bf16, nullptr, nullptr, w_gu, s_gu, h, I, M, 2 * I, H, d, st,
                             g_pdl.load() != 0);
        if (rc) return rc;
        // the down GEMM streams its weights while the gate_up GEMM finishes (programmatic launch)
        return run_stream_gemm(amode, EPI_STORE, h, hq, hs, w_dn, s_dn, y_bf16, H_out, M, H_out, I, d, st, true);
    }
    rc = run_stream_gemm(amode, EPI_STORE, x_bf16, nullptr, nullptr, w_gu, s_gu, gu, 2 * I, M, 2 * I, H, d, st, false);
    if (rc) return rc;
    rc = to_status(launch_swiglu_interleaved(static_cast<const uint16_t*>(gu), M, I, static_cast<uint16_t*>(h), st, d->sms));
    if (rc) return rc;
    if (wonly)
        return run_stream_gemm(A_BF16, EPI_STORE, h, nullptr, nullptr, w_dn, s_dn, y_bf16, H_out, M, H_out, I, d, st, false);
    rc = to_status(launch_quant_group128(static_cast<const uint16_t*>(h), M, I, hq, hs, st, d->sms));
    if (rc) return rc;
    return run_stream_gemm(A_PREQ, EPI_STORE, nullptr, hq, hs, w_dn, s_dn, y_bf16, H_out, M, H_out, I, d, st, false);
}

}  // extern "C"
