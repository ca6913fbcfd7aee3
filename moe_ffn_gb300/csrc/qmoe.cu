// qmoe.cu — C-ABI entry points of libqmoe.so: argument validation, launch
// planning and programmatic-dependent launches of the sm_103a kernels.
// See include/qmoe.h for the contract of every function.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstddef>
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "../../include/qmoe.h"
#include "formats.cuh"
#include "ptx.cuh"
#include "stream.cuh"
#include "fused.cuh"
#include "batch.cuh"
#include "prefill.cuh"

namespace qmoe {

// ----------------------------------------------------------------- errors
static thread_local std::string g_last_error;

static qmoe_status fail(qmoe_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

static qmoe_status cuda_fail(cudaError_t e, const char* what) {
    return fail(QMOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// The device control block (ptx.cuh): error word, wait limit, fault
// injection.  One per device that loads the library.
__device__ DevCtl g_dev_ctl = {0u, -1, DEFAULT_WAIT_NS};

// ------------------------------------------------------------ formats
static int block_elems(int qt) {
    switch (qt) {
    case QT_F32: return 1;
    case QT_Q8_0: case QT_Q4_0: return 32;
    case QT_Q4_K: case QT_Q5_K: case QT_Q6_K: return 256;
    default: return 0;
    }
}
static int block_bytes(int qt) {
    switch (qt) {
    case QT_F32: return 4;
    case QT_Q8_0: return 34;
    case QT_Q4_0: return 18;
    case QT_Q4_K: return 144;
    case QT_Q5_K: return 176;
    case QT_Q6_K: return 210;
    default: return 0;
    }
}
static int64_t row_bytes_of(int qt, int64_t cols) {
    const int be = block_elems(qt);
    if (be <= 0 || cols <= 0 || cols % be) return -1;
    return cols / be * block_bytes(qt);
}
static const char* qname(int qt) {
    switch (qt) {
    case QT_F32: return "F32";
    case QT_Q8_0: return "Q8_0";
    case QT_Q4_0: return "Q4_0";
    case QT_Q4_K: return "Q4_K";
    case QT_Q5_K: return "Q5_K";
    case QT_Q6_K: return "Q6_K";
    default: return "unknown";
    }
}
static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int64_t MAX_K = 32768;
// Every workspace starts with the fused kernel's grid-barrier counters,
// which each call leaves at zero; the other regions follow.
constexpr size_t WS_SYNC_BYTES = 256;

// ------------------------------------------------------------ device info
struct DevInfo {
    bool init = false;
    bool supported = false;
    int sms = 0;
    int smem_optin = 0;
    int smem_pair = 0;  // dynamic shared memory per CTA that lets two CTAs share an SM
    DevCtl* err = nullptr;
    int cc_major = 0, cc_minor = 0;
};
static DevInfo g_dev[64];
static std::mutex g_dev_mu;

static qmoe_status device_info(DevInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(QMOE_ERR_UNSUPPORTED, "device ordinal %d >= 64", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo& d = g_dev[dev];
    if (!d.init) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
        d.cc_major = prop.major;
        d.cc_minor = prop.minor;
        d.sms = prop.multiProcessorCount;
        d.smem_optin = static_cast<int>(prop.sharedMemPerBlockOptin);
        d.smem_pair = static_cast<int>(prop.sharedMemPerMultiprocessor / 2 -
                                       prop.reservedSharedMemPerBlock);
        d.supported = (prop.major == 10 && prop.minor == 3);
        if (d.supported) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_dev_ctl);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device control)");
            d.err = static_cast<DevCtl*>(p);
        }
        d.init = true;
    }
    if (!d.supported)
        return fail(QMOE_ERR_UNSUPPORTED,
                    "device %d is compute capability %d.%d; this library is built for sm_103a "
                    "(GB300) only",
                    dev, d.cc_major, d.cc_minor);
    *out = &d;
    return QMOE_OK;
}

// ------------------------------------------------------------ launching
template <typename Kern, typename... Args>
static cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Plan chunking and pipeline depth for a streamed GEMV; false if it cannot
// fit in shared memory.
template <class Fmt, int MODE>
static bool plan(StreamParams& p, int smem_optin, int smem_pair, int grid, int* smem_bytes) {
    using G = ModeGeom<MODE>;
    p.stage_bytes = 0;
    p.nstages = 0;
    const int fixed0 = smem_layout(p).total;
    // A CTA with a single tile gains nothing from a ring: one stage then
    // holds the whole tile (whole rows, so few and large copies), planned
    // first within smem_pair bytes (half the SM's shared memory), else within
    // the opt-in maximum.  Otherwise the stage budget is at most 96 KB, and
    // two stages must fit beside the x table.
    const int64_t per_cta = (p.units + grid - 1) / grid;
    const bool one_tile = per_cta <= G::TU;
    if (one_tile) {
        const int rows = static_cast<int>(per_cta);
        for (const int cap : {smem_pair, smem_optin}) {
            if (cap - fixed0 > 0 && plan_chunks<Fmt, MODE>(p, cap - fixed0, rows) &&
                p.n_chunk == 1) {
                p.nstages = 1;
                *smem_bytes = smem_layout(p).total;
                if (*smem_bytes <= cap) return true;
            }
            p.nstages = 0;
        }
    }
    const int room = smem_optin - fixed0;
    const int budget = room / 2 < 96 * 1024 ? room / 2 : 96 * 1024;
    if (!plan_chunks<Fmt, MODE>(p, budget)) return false;
    const int fixed = smem_layout(p).total;
    int ns = (smem_optin - fixed) / p.stage_bytes;
    if (ns > MAX_STAGES) ns = MAX_STAGES;
    if (ns < 2) return false;
    p.nstages = ns;
    *smem_bytes = smem_layout(p).total;
    return true;
}

template <class Fmt, int MODE>
static qmoe_status run_stream(StreamParams p, const DevInfo& d, cudaStream_t st) {
    int smem = 0;
    const int64_t grid = p.units < d.sms ? p.units : d.sms;
    p.uq = p.units / grid;
    p.ur = static_cast<int>(p.units % grid);
    if (!plan<Fmt, MODE>(p, d.smem_optin, d.smem_pair, static_cast<int>(grid), &smem))
        return fail(QMOE_ERR_UNSUPPORTED,
                    "K = %d x %d groups of 256 does not fit the shared-memory pipeline",
                    p.n_kseg, p.nb_seg);
    // QMV whose rows fit one stage: the eight-warp kernel (two CTAs per SM
    // by registers)
    const bool tile8 = MODE == MODE_QMV && p.nstages == 1;
    auto kern = tile8 ? qmv_tile_kernel<Fmt> : stream_gemv_kernel<Fmt, MODE>;
    static int configured_smem[2][64] = {};  // per instantiation, kernel and device
    int dev = 0;
    cudaGetDevice(&dev);
    if (smem > configured_smem[tile8][dev & 63]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        // the whole unified L1 as shared memory: this launch's CTAs and the
        // next launch's can then share an SM where their registers allow
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        configured_smem[tile8][dev & 63] = smem;
    }
    p.err = d.err;
    cudaError_t e = launch_pdl(kern, dim3(static_cast<unsigned>(grid)),
                               dim3(tile8 ? NCW * 32 : NTHREADS), static_cast<size_t>(smem), st, p);
    if (e != cudaSuccess) return cuda_fail(e, "stream_gemv launch");
    return QMOE_OK;
}

template <int MODE>
static qmoe_status dispatch(int qt, const StreamParams& p, const DevInfo& d, cudaStream_t st) {
    switch (qt) {
    case QT_Q8_0: return run_stream<FmtQ80, MODE>(p, d, st);
    case QT_Q4_0: return run_stream<FmtQ40, MODE>(p, d, st);
    case QT_Q4_K: return run_stream<FmtQ4K, MODE>(p, d, st);
    case QT_Q5_K: return run_stream<FmtQ5K, MODE>(p, d, st);
    case QT_Q6_K: return run_stream<FmtQ6K, MODE>(p, d, st);
    default: return fail(QMOE_ERR_UNSUPPORTED, "qtype %d has no streamed GEMV", qt);
    }
}

// ------------------------------------------------------- fused FFN layer
// Plan both phases of the fused kernel with one stage size; false if the
// layer does not fit (then the caller runs the phases as separate kernels).
template <class FmtG, class FmtD>
static bool plan_fused(FusedParams& f, int smem_optin, int* smem_bytes) {
    f.gu.stage_bytes = f.dn.stage_bytes = 0;
    f.gu.nstages = f.dn.nstages = 0;
    const int room = smem_optin - fused_layout(f).total;
    const int budget = room / 2 < 96 * 1024 ? room / 2 : 96 * 1024;
    if (!plan_chunks<FmtG, MODE_GATEUP>(f.gu, budget)) return false;
    if (!plan_chunks<FmtD, MODE_DOWN>(f.dn, budget)) return false;
    const int sb = f.gu.stage_bytes > f.dn.stage_bytes ? f.gu.stage_bytes : f.dn.stage_bytes;
    int ns = room / sb;
    if (ns > MAX_STAGES) ns = MAX_STAGES;
    if (ns < 2) return false;
    f.gu.stage_bytes = f.dn.stage_bytes = sb;
    f.gu.nstages = f.dn.nstages = ns;
    *smem_bytes = fused_layout(f).total;
    return *smem_bytes <= smem_optin;
}

// Whether cooperative launches may also carry programmatic stream
// serialisation on this driver (probed on first use, per process).
static int g_coop_pdl = -1;

// 1: launched; 0: the layer does not fit the fused kernel (nothing
// launched); negative: a CUDA error (status in *err).
template <class FmtG, class FmtD>
static int run_fused(FusedParams f, const DevInfo& d, cudaStream_t st, qmoe_status* err) {
    int smem = 0;
    if (!plan_fused<FmtG, FmtD>(f, d.smem_optin, &smem)) return 0;
    auto kern = fused_ffn_kernel<FmtG, FmtD>;
    static int configured_smem[64] = {};  // per instantiation and device
    int dev = 0;
    cudaGetDevice(&dev);
    if (smem > configured_smem[dev & 63]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) {
            *err = cuda_fail(e, "cudaFuncSetAttribute (fused)");
            return -1;
        }
        configured_smem[dev & 63] = smem;
    }
    f.err = f.gu.err = f.dn.err = d.err;
    f.gu.uq = f.gu.units / d.sms;
    f.gu.ur = static_cast<int>(f.gu.units % d.sms);
    f.dn.uq = f.dn.units / d.sms;
    f.dn.ur = static_cast<int>(f.dn.units % d.sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(d.sms));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_coop_pdl == 0 ? 1 : 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, f);
    if (e != cudaSuccess && g_coop_pdl < 0) {
        // if the driver rejects the pair, run without programmatic serialisation
        (void)cudaGetLastError();
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, f);
        if (e == cudaSuccess) g_coop_pdl = 0;
    }
    if (e != cudaSuccess) {
        *err = cuda_fail(e, "fused FFN launch");
        return -1;
    }
    if (g_coop_pdl < 0) g_coop_pdl = 1;
    return 1;
}

template <class FmtG>
static int dispatch_fused_d(int dq, const FusedParams& f, const DevInfo& d, cudaStream_t st,
                            qmoe_status* err) {
    switch (dq) {
    case QT_Q8_0: return run_fused<FmtG, FmtQ80>(f, d, st, err);
    case QT_Q4_0: return run_fused<FmtG, FmtQ40>(f, d, st, err);
    case QT_Q4_K: return run_fused<FmtG, FmtQ4K>(f, d, st, err);
    case QT_Q5_K: return run_fused<FmtG, FmtQ5K>(f, d, st, err);
    case QT_Q6_K: return run_fused<FmtG, FmtQ6K>(f, d, st, err);
    default: return 0;
    }
}

// Execution mode (qmoe_set_exec_mode; diagnostics and tests): the default
// kernels, or the separate-kernel forms they replace.
static std::atomic<int> g_exec_mode{QMOE_EXEC_DEFAULT};

// Fused layer for these formats: 1 launched, 0 not applicable (the caller
// runs separate kernels), negative on a CUDA error.
static bool fused_enabled() { return g_exec_mode.load() != QMOE_EXEC_SEPARATE; }

// The batched decode kernel for 2..31 tokens.
static bool batch_enabled() { return g_exec_mode.load() == QMOE_EXEC_DEFAULT; }

static int dispatch_fused(int gq, int dq, const FusedParams& f, const DevInfo& d, cudaStream_t st,
                          qmoe_status* err) {
    if (!fused_enabled()) return 0;
    switch (gq) {
    case QT_Q8_0: return dispatch_fused_d<FmtQ80>(dq, f, d, st, err);
    case QT_Q4_0: return dispatch_fused_d<FmtQ40>(dq, f, d, st, err);
    case QT_Q4_K: return dispatch_fused_d<FmtQ4K>(dq, f, d, st, err);
    case QT_Q5_K: return dispatch_fused_d<FmtQ5K>(dq, f, d, st, err);
    case QT_Q6_K: return dispatch_fused_d<FmtQ6K>(dq, f, d, st, err);
    default: return 0;
    }
}

// ------------------------------------------------------------ f32 GEMV
// y[r] = R[r] . x for an f32 [rows][cols] matrix: one CTA of 128 threads
// per row.  The router GEMV of the MoE layer and qmv(F32).  Weights are
// loaded before the dependency wait.
constexpr int F32_THREADS = 128;
constexpr int F32_PREFETCH = 8;

__global__ void __launch_bounds__(F32_THREADS) f32_gemv_kernel(const float* __restrict__ R,
                                                               const float* __restrict__ x,
                                                               float* __restrict__ y,
                                                               int64_t cols) {
    const int64_t r = blockIdx.x;
    const int tid = threadIdx.x;
    const float4* r4 = reinterpret_cast<const float4*>(R + r * cols);
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const int64_t n4 = cols / 4;
    float4 w[F32_PREFETCH];
#pragma unroll
    for (int k = 0; k < F32_PREFETCH; ++k) {
        const int64_t i = tid + static_cast<int64_t>(k) * F32_THREADS;
        w[k] = i < n4 ? __ldg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_wait();
    pdl_trigger();
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < F32_PREFETCH; ++k) {
        const int64_t i = tid + static_cast<int64_t>(k) * F32_THREADS;
        if (i < n4) {
            const float4 xv = __ldcg(x4 + i);
            acc = fmaf(w[k].x, xv.x, acc);
            acc = fmaf(w[k].y, xv.y, acc);
            acc = fmaf(w[k].z, xv.z, acc);
            acc = fmaf(w[k].w, xv.w, acc);
        }
    }
    for (int64_t i = tid + static_cast<int64_t>(F32_PREFETCH) * F32_THREADS; i < n4;
         i += F32_THREADS) {
        const float4 wv = __ldg(r4 + i), xv = __ldcg(x4 + i);
        acc = fmaf(wv.x, xv.x, acc);
        acc = fmaf(wv.y, xv.y, acc);
        acc = fmaf(wv.z, xv.z, acc);
        acc = fmaf(wv.w, xv.w, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    __shared__ float red[F32_THREADS / 32];
    if ((tid & 31) == 0) red[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int k = 0; k < F32_THREADS / 32; ++k) s += red[k];
        y[r] = s;
    }
}

static qmoe_status run_f32_gemv(const float* R, const float* x, float* y, int64_t rows,
                                int64_t cols, cudaStream_t st) {
    cudaError_t e = launch_pdl(f32_gemv_kernel, dim3(static_cast<unsigned>(rows)),
                               dim3(F32_THREADS), 0, st, R, x, y, cols);
    if (e != cudaSuccess) return cuda_fail(e, "f32_gemv launch");
    return QMOE_OK;
}

// ffn_norm for T rows of n: out[t] = h[t] * w / sqrt(mean(h[t]^2) + eps), one
// CTA per row — the fused add+RMSNorm kernel of "ferrox-cuda 0.14.0 —
// src/gpu.rs" without the add (moe_layer norms the hidden state).  Used in
// front of the tensor-core and separate-kernel forms; the fused layer
// kernel norms its input itself.
constexpr int NORM_THREADS = 256;
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_kernel(const float* __restrict__ h,
                                                               const float* __restrict__ w, int n,
                                                               float eps, float* __restrict__ out) {
    __shared__ float red[NORM_THREADS / 32];
    const int64_t off = static_cast<int64_t>(blockIdx.x) * n;
    pdl_wait();
    pdl_trigger();
    const float inv = rms_inverse(h + off, n, eps, red, threadIdx.x, NORM_THREADS, 0);
    const float4* h4 = reinterpret_cast<const float4*>(h + off);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    float4* o4 = reinterpret_cast<float4*>(out + off);
    for (int i = threadIdx.x; i < n / 4; i += NORM_THREADS) {
        const float4 v = __ldcg(h4 + i), wv = __ldg(w4 + i);
        o4[i] = make_float4(v.x * (inv * wv.x), v.y * (inv * wv.y), v.z * (inv * wv.z),
                            v.w * (inv * wv.w));
    }
}

static qmoe_status run_rmsnorm(const float* h, const float* w, int64_t rows, int64_t n, float eps,
                               float* out, cudaStream_t st) {
    cudaError_t e = launch_pdl(rmsnorm_kernel, dim3(static_cast<unsigned>(rows)),
                               dim3(NORM_THREADS), 0, st, h, w, static_cast<int>(n), eps, out);
    if (e != cudaSuccess) return cuda_fail(e, "rmsnorm launch");
    return QMOE_OK;
}

}  // namespace qmoe

using namespace qmoe;

// ====================================================================== C ABI
extern "C" {

const char* qmoe_last_error(void) { return g_last_error.c_str(); }

int64_t qmoe_row_bytes(int qtype, int64_t cols) { return row_bytes_of(qtype, cols); }

qmoe_status qmv(int qtype, const void* W, int64_t rows, int64_t cols, const float* x, float* y,
                void* stream) {
    g_last_error.clear();
    if (qtype < QT_F32 || qtype > QT_Q6_K)
        return fail(QMOE_ERR_UNSUPPORTED, "qmv: unknown qtype %d", qtype);
    if (!W || !x || !y) return fail(QMOE_ERR_INVALID_ARGUMENT, "qmv: null pointer (W, x or y)");
    if (rows <= 0 || cols <= 0)
        return fail(QMOE_ERR_INVALID_ARGUMENT, "qmv: rows=%lld cols=%lld must be >= 1",
                    (long long)rows, (long long)cols);
    if (cols % block_elems(qtype))
        return fail(QMOE_ERR_INVALID_ARGUMENT,
                    "qmv: cols=%lld is not a whole number of %s blocks (%d elements)",
                    (long long)cols, qname(qtype), block_elems(qtype));
    if (qtype == QT_F32 && cols % 4 != 0)
        return fail(QMOE_ERR_UNSUPPORTED, "qmv: cols=%lld must be a multiple of 4 for F32",
                    (long long)cols);
    if (cols > MAX_K)
        return fail(QMOE_ERR_UNSUPPORTED, "qmv: cols=%lld exceeds %lld", (long long)cols,
                    (long long)MAX_K);
    if (rows > 0x7fffffffLL)
        return fail(QMOE_ERR_UNSUPPORTED, "qmv: rows=%lld exceeds 2^31-1", (long long)rows);
    if (!aligned(W, 16) || !aligned(x, 16) || !aligned(y, 4))
        return fail(QMOE_ERR_INVALID_ARGUMENT,
                    "qmv: W and x must be 16-byte aligned, y 4-byte aligned");
    DevInfo* d = nullptr;
    if (qmoe_status s = device_info(&d)) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (qtype == QT_F32)
        return run_f32_gemv(static_cast<const float*>(W), x, y, rows, cols, st);
    StreamParams p = {};
    p.units = rows;
    // Q8_0 / Q4_0 rows may end in a partial group of 32-element blocks
    p.nb_seg = static_cast<int>((cols + 255) / 256);
    p.tail = static_cast<int>((cols % 256) / 32);
    p.n_kseg = 1;
    p.W0 = static_cast<const uint8_t*>(W);
    p.rb0 = row_bytes_of(qtype, cols);
    p.x = x;
    p.out = y;
    return dispatch<MODE_QMV>(qtype, p, *d, st);
}

size_t ffn_swiglu_workspace_size(int64_t hidden, int64_t inter) {
    (void)hidden;
    if (inter <= 0) return 0;
    return WS_SYNC_BYTES + static_cast<size_t>(align_up(static_cast<int>(inter * 4), 256));
}

static qmoe_status check_ffn_qtypes(const char* fn, int gq, int uq, int dq) {
    for (int qt : {gq, uq, dq})
        if (qt < QT_F32 || qt > QT_Q6_K) return fail(QMOE_ERR_UNSUPPORTED, "%s: unknown qtype %d", fn, qt);
    if (gq == QT_F32 || uq == QT_F32 || dq == QT_F32)
        return fail(QMOE_ERR_UNSUPPORTED, "%s: F32 gate/up/down weights are not implemented", fn);
    if (gq != uq)
        return fail(QMOE_ERR_UNSUPPORTED,
                    "%s: gate (%s) and up (%s) must share a format (they are decoded by one "
                    "kernel)",
                    fn, qname(gq), qname(uq));
    return QMOE_OK;
}

// Checks shared by ffn_swiglu and ffn_swiglu_rmsnorm.  `x` is the FFN input
// (ffn_swiglu) or the norm weight (ffn_swiglu_rmsnorm); `need` the workspace.
static qmoe_status ffn_check(const char* fn, const void* gate, const void* up, const void* down,
                             int gate_qtype, int up_qtype, int down_qtype, int64_t hidden,
                             int64_t inter, const float* x, const float* residual, const void* ws,
                             size_t ws_bytes, size_t need, uintptr_t res_align) {
    if (!gate || !up || !down || !x || !residual || !ws)
        return fail(QMOE_ERR_INVALID_ARGUMENT, "%s: null pointer", fn);
    if (hidden <= 0 || inter <= 0)
        return fail(QMOE_ERR_INVALID_ARGUMENT, "%s: hidden=%lld inter=%lld must be >= 1", fn,
                    (long long)hidden, (long long)inter);
    if (qmoe_status s = check_ffn_qtypes(fn, gate_qtype, up_qtype, down_qtype)) return s;
    if (hidden % block_elems(gate_qtype) || inter % block_elems(down_qtype))
        return fail(QMOE_ERR_INVALID_ARGUMENT, "%s: hidden/inter not whole numbers of blocks", fn);
    if (hidden % 256 || inter % 256)
        return fail(QMOE_ERR_UNSUPPORTED, "%s: hidden and inter must be multiples of 256", fn);
    if (hidden > MAX_K || inter > MAX_K)
        return fail(QMOE_ERR_UNSUPPORTED, "%s: hidden/inter exceed %lld", fn, (long long)MAX_K);
    if (ws_bytes < need)
        return fail(QMOE_ERR_INVALID_ARGUMENT, "%s: workspace %zu < %zu bytes", fn, ws_bytes,
                    need);
    if (!aligned(gate, 16) || !aligned(up, 16) || !aligned(down, 16) || !aligned(x, 16) ||
        !aligned(residual, res_align) || !aligned(ws, 16))
        return fail(QMOE_ERR_INVALID_ARGUMENT,
                    "%s: weights, x/norm weight and ws must be 16-byte aligned, residual %d-byte",
                    fn, static_cast<int>(res_align));
    return QMOE_OK;
}

// The dense FFN layer.  With norm_w, the input is ffn_norm(residual) and x is
// unused; xn is workspace for the normed input of the two-kernel form.
static qmoe_status ffn_core(const void* gate, const void* up, const void* down, int gate_qtype,
                            int up_qtype, int down_qtype, int64_t hidden, int64_t inter,
                            const float* x, const float* norm_w, float eps, float* residual,
                            void* ws, float* xn, const DevInfo& d, cudaStream_t st) {
    float* a = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + WS_SYNC_BYTES);
    StreamParams pg = {};
    pg.units = inter;
    pg.nb_seg = static_cast<int>(hidden / 256);
    pg.n_kseg = 1;
    pg.W0 = static_cast<const uint8_t*>(gate);
    pg.rb0 = row_bytes_of(gate_qtype, hidden);
    pg.W1 = static_cast<const uint8_t*>(up);
    pg.rb1 = row_bytes_of(up_qtype, hidden);
    pg.x = norm_w ? residual : x;
    pg.out = a;

    StreamParams pd = {};
    pd.units = hidden;
    pd.nb_seg = static_cast<int>(inter / 256);
    pd.n_kseg = 1;
    pd.W0 = static_cast<const uint8_t*>(down);
    pd.rb0 = row_bytes_of(down_qtype, inter);
    pd.x = a;
    pd.out = residual;

    FusedParams f = {};
    f.gu = pg;
    f.dn = pd;
    f.sync = static_cast<unsigned long long*>(ws);
    f.norm_w = norm_w;
    f.eps = eps;
    qmoe_status ferr = QMOE_OK;
    const int fr = dispatch_fused(gate_qtype, down_qtype, f, d, st, &ferr);
    if (fr < 0) return ferr;
    if (fr > 0) return QMOE_OK;
    if (norm_w) {
        if (qmoe_status s = run_rmsnorm(residual, norm_w, 1, hidden, eps, xn, st)) return s;
        pg.x = xn;
    }
    if (qmoe_status s = dispatch<MODE_GATEUP>(gate_qtype, pg, d, st)) return s;
    return dispatch<MODE_DOWN>(down_qtype, pd, d, st);
}

qmoe_status ffn_swiglu(const void* gate, const void* up, const void* down, int gate_qtype,
                       int up_qtype, int down_qtype, int64_t hidden, int64_t inter,
                       const float* x, float* residual, void* ws, size_t ws_bytes, void* stream) {
    g_last_error.clear();
    if (qmoe_status s = ffn_check("ffn_swiglu", gate, up, down, gate_qtype, up_qtype, down_qtype,
                                  hidden, inter, x, residual, ws, ws_bytes,
                                  ffn_swiglu_workspace_size(hidden, inter), 4))
        return s;
    DevInfo* d = nullptr;
    if (qmoe_status s = device_info(&d)) return s;
    return ffn_core(gate, up, down, gate_qtype, up_qtype, down_qtype, hidden, inter, x, nullptr,
                    0.f, residual, ws, nullptr, *d, static_cast<cudaStream_t>(stream));
}

size_t ffn_swiglu_rmsnorm_workspace_size(int64_t hidden, int64_t inter) {
    if (hidden <= 0 || inter <= 0) return 0;
    return ffn_swiglu_workspace_size(hidden, inter) +
           static_cast<size_t>(align_up(static_cast<int>(hidden * 4), 256));
}

qmoe_status ffn_swiglu_rmsnorm(const void* gate, const void* up, const void* down,
                               int gate_qtype, int up_qtype, int down_qtype, int64_t hidden,
                               int64_t inter, const float* norm_w, float eps, float* residual,
                               void* ws, size_t ws_bytes, void* stream) {
    g_last_error.clear();
    if (qmoe_status s = ffn_check("ffn_swiglu_rmsnorm", gate, up, down, gate_qtype, up_qtype,
                                  down_qtype, hidden, inter, norm_w, residual, ws, ws_bytes,
                                  ffn_swiglu_rmsnorm_workspace_size(hidden, inter), 16))
        return s;
    if (!(eps >= 0.f) || !std::isfinite(eps))
        return fail(QMOE_ERR_INVALID_ARGUMENT, "ffn_swiglu_rmsnorm: eps=%g must be finite, >= 0",
                    static_cast<double>(eps));
    DevInfo* d = nullptr;
    if (qmoe_status s = device_info(&d)) return s;
    float* xn = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                         ffn_swiglu_workspace_size(hidden, inter));
    return ffn_core(gate, up, down, gate_qtype, up_qtype, down_qtype, hidden, inter, nullptr,
                    norm_w, eps, residual, ws, xn, *d, static_cast<cudaStream_t>(stream));
}

static size_t moe_logits_bytes(const qmoe_moe_shape* s) {
    return static_cast<size_t>(align_up(s->n_tokens * s->num_experts * 4, 256));
}

// Token count from which the grouped tensor-core path is used (for the
// formats it implements); below it tokens run the decode pipeline one by one.
constexpr int PF_MIN_TOKENS = 32;

static bool prefill_path(const qmoe_moe_shape* s) {
    return s->n_tokens >= PF_MIN_TOKENS && s->gate_qtype == QT_Q4_K && s->up_qtype == QT_Q4_K &&
           s->down_qtype == QT_Q6_K && s->expert_dim % 256 == 0 && s->hidden % 256 == 0 &&
           s->expert_dim <= pf::PF_DN_MAX_F;
}

// Prefill workspace carve-up (byte offsets from ws).
struct PfWs {
    size_t logits, tidx, tw, cnt, list, x16, xinv, a, total;
};
static PfWs pf_ws_layout(const qmoe_moe_shape* s) {
    const size_t T = s->n_tokens, E = s->num_experts, K = s->top_k, H = s->hidden,
                 F = s->expert_dim;
    auto al = [](size_t v) { return (v + 255) / 256 * 256; };
    PfWs w;
    size_t o = WS_SYNC_BYTES;
    w.logits = o; o += al(T * E * 4);
    w.tidx = o;   o += al(T * K * 4);
    w.tw = o;     o += al(T * K * 4);
    w.cnt = o;    o += al(E * 4);
    w.list = o;   o += al(E * T * 4);
    w.x16 = o;    o += al(T * H * 2);
    w.xinv = o;   o += al(T * 4);
    w.a = o;      o += al(T * K * F * 4);
    w.total = o;
    return w;
}

size_t moe_ffn_workspace_size(const qmoe_moe_shape* s) {
    if (!s || s->n_tokens <= 0 || s->num_experts <= 0 || s->top_k <= 0 || s->expert_dim <= 0 ||
        s->hidden <= 0)
        return 0;
    // activations of one token, or of the (token, expert) pairs of one
    // batched launch
    const int tb = s->n_tokens < TB_MAX ? s->n_tokens : TB_MAX;
    const size_t decode =
        WS_SYNC_BYTES + moe_logits_bytes(s) +
        static_cast<size_t>(align_up(tb * s->top_k * s->expert_dim * 4, 256));
    if (prefill_path(s)) {
        const size_t pf = pf_ws_layout(s).total;
        return pf > decode ? pf : decode;
    }
    return decode;
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no link
// against the driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// A [rows][row_bytes] byte matrix as a 2-D tensor map with boxes of
// box_bytes x box_rows.  row_bytes, box_bytes and the base must be multiples
// of 16 bytes.
static qmoe_status rows_map(CUtensorMap* m, const void* base, int64_t row_bytes, int64_t rows,
                            uint32_t box_bytes, uint32_t box_rows) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return fail(QMOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {box_bytes, box_rows};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                          strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QMOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return QMOE_OK;
}

// A [rows][cols] f32 matrix as a 2-D tensor map with boxes of box_cols x
// box_rows, 128-byte swizzled (box_cols * 4 == 128: the MMA's K-major
// operand layout).  cols * 4 and the base must be multiples of 16 bytes.
static qmoe_status f32_swizzled_map(CUtensorMap* m, const float* base, int64_t cols, int64_t rows,
                                    uint32_t box_cols, uint32_t box_rows) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return fail(QMOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                          const_cast<float*>(base), dims, strides, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QMOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return QMOE_OK;
}

static qmoe_status run_prefill(const float* router_W, const void* gate_stack,
                               const void* up_stack, const void* down_stack,
                               const qmoe_moe_shape& s, const float* x, float* residual,
                               int32_t* topk_idx, float* topk_w, void* ws, const DevInfo& d,
                               cudaStream_t st) {
    const PfWs L = pf_ws_layout(&s);
    uint8_t* w = static_cast<uint8_t*>(ws);
    float* logits = reinterpret_cast<float*>(w + L.logits);
    int32_t* tidx = reinterpret_cast<int32_t*>(w + L.tidx);
    float* tw = reinterpret_cast<float*>(w + L.tw);
    int32_t* cnt = reinterpret_cast<int32_t*>(w + L.cnt);
    int32_t* list = reinterpret_cast<int32_t*>(w + L.list);
    __half* x16 = reinterpret_cast<__half*>(w + L.x16);
    float* xinv = reinterpret_cast<float*>(w + L.xinv);
    float* a = reinterpret_cast<float*>(w + L.a);
    const int T = s.n_tokens, H = s.hidden, E = s.num_experts, K = s.top_k, F = s.expert_dim;

    static int configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configured[dev & 63]) {
        cudaError_t ce = cudaFuncSetAttribute(pf::pf_router_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              pf::RT_SMEM);
        if (ce == cudaSuccess)
            ce = cudaFuncSetAttribute(pf::pf_gateup_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, pf::GU_SMEM);
        if (ce == cudaSuccess)
            ce = cudaFuncSetAttribute(pf::pf_down_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, pf::DN_SMEM);
        if (ce != cudaSuccess) return cuda_fail(ce, "cudaFuncSetAttribute(prefill)");
        configured[dev & 63] = 1;
    }
    cudaError_t e = launch_pdl(pf::pf_router_kernel, dim3((T + 7) / 8, (E + 31) / 32), dim3(256),
                               static_cast<size_t>(pf::RT_SMEM), st, router_W, x, T, H, E, logits,
                               cnt);
    if (e != cudaSuccess) return cuda_fail(e, "pf_router launch");
    const int renorm = (s.route_flags & QMOE_ROUTE_NO_RENORM) ? 0 : 1;
    e = launch_pdl(pf::pf_topk_kernel, dim3((T + 7) / 8), dim3(256), 0, st,
                   static_cast<const float*>(logits), x, T, H, E, K, renorm, tidx, tw, topk_idx,
                   topk_w, cnt, list, x16, xinv, d.err);
    if (e != cudaSuccess) return cuda_fail(e, "pf_topk launch");

    pf::PfParams pg = {};
    pg.W0 = static_cast<const uint8_t*>(gate_stack);
    pg.W1 = static_cast<const uint8_t*>(up_stack);
    pg.rb = row_bytes_of(QT_Q4_K, H);
    pg.es = pg.rb * F;
    pg.H = H; pg.F = F; pg.E = E; pg.K = K; pg.T = T;
    pg.cnt = cnt; pg.list = list; pg.X16 = x16; pg.xinv = xinv; pg.tw = tw; pg.a = a;
    pg.residual = residual;
    pg.err = d.err;
    const int items_gu = E * (F / 128);
    CUtensorMap tm_gate, tm_up;
    if (qmoe_status r = rows_map(&tm_gate, gate_stack, pg.rb, static_cast<int64_t>(E) * F,
                                 pf::GU_RAW_ROW, 128))
        return r;
    if (qmoe_status r = rows_map(&tm_up, up_stack, pg.rb, static_cast<int64_t>(E) * F,
                                 pf::GU_RAW_ROW, 128))
        return r;
    e = launch_pdl(pf::pf_gateup_kernel, dim3(items_gu < d.sms ? items_gu : d.sms),
                   dim3(pf::PF_THREADS), static_cast<size_t>(pf::GU_SMEM), st, pg, tm_gate,
                   tm_up);
    if (e != cudaSuccess) return cuda_fail(e, "pf_gateup launch");
    pf::PfParams pd = pg;
    pd.W0 = static_cast<const uint8_t*>(down_stack);
    pd.W1 = nullptr;
    pd.rb = row_bytes_of(QT_Q6_K, F);
    pd.es = pd.rb * H;
    const int items_dn = E * (H / 128);
    // the activations, expert-major [T*K][F], as the down product's B tiles:
    // 32 columns (one 128-byte swizzle row) x PF_NP pairs per copy
    CUtensorMap tm_act;
    if (qmoe_status r = f32_swizzled_map(&tm_act, a, F, static_cast<int64_t>(T) * K, 32,
                                         pf::PF_NP))
        return r;
    e = launch_pdl(pf::pf_down_kernel, dim3(items_dn < d.sms ? items_dn : d.sms),
                   dim3(pf::PF_THREADS), static_cast<size_t>(pf::DN_SMEM), st, pd, tm_act);
    if (e != cudaSuccess) return cuda_fail(e, "pf_down launch");
    return QMOE_OK;
}

// Checks shared by moe_ffn and moe_ffn_rmsnorm.  `x` is the FFN input
// (moe_ffn) or the norm weight (moe_ffn_rmsnorm); `need` the workspace.
static qmoe_status moe_check(const char* fn, const float* router_W, const void* gate_stack,
                             const void* up_stack, const void* down_stack,
                             const qmoe_moe_shape* shape, const float* x, const float* residual,
                             const void* ws, size_t ws_bytes, size_t need, uintptr_t res_align) {
    if (!shape) return fail(QMOE_ERR_INVALID_ARGUMENT, "%s: null shape", fn);
    const qmoe_moe_shape s = *shape;
    if (!router_W || !gate_stack || !up_stack || !down_stack || !x || !residual || !ws)
        return fail(QMOE_ERR_INVALID_ARGUMENT, "%s: null pointer", fn);
    // check_moe_shape: every count positive, k <= E
    if (s.hidden <= 0 || s.expert_dim <= 0 || s.num_experts <= 0 || s.top_k <= 0 ||
        s.n_tokens <= 0)
        return fail(QMOE_ERR_INVALID_ARGUMENT,
                    "%s: incomplete MoE shape (hidden=%d expert_dim=%d num_experts=%d "
                    "top_k=%d n_tokens=%d)", fn,
                    s.hidden, s.expert_dim, s.num_experts, s.top_k, s.n_tokens);
    if (s.top_k > s.num_experts)
        return fail(QMOE_ERR_INVALID_ARGUMENT, "%s: top_k=%d > num_experts=%d", fn, s.top_k,
                    s.num_experts);
    if (s.route_flags & ~QMOE_ROUTE_NO_RENORM)
        return fail(QMOE_ERR_INVALID_ARGUMENT, "%s: unknown route_flags 0x%x", fn,
                    static_cast<unsigned>(s.route_flags));
    if (qmoe_status st = check_ffn_qtypes(fn, s.gate_qtype, s.up_qtype, s.down_qtype))
        return st;
    if (s.num_experts > MAX_EXPERTS || s.top_k > MAX_TOPK)
        return fail(QMOE_ERR_UNSUPPORTED,
                    "%s: on-device routing supports num_experts <= %d and top_k <= %d", fn,
                    MAX_EXPERTS, MAX_TOPK);
    if (s.hidden % block_elems(s.gate_qtype) || s.expert_dim % block_elems(s.down_qtype))
        return fail(QMOE_ERR_INVALID_ARGUMENT, "%s: hidden/expert_dim not whole blocks", fn);
    if (s.hidden % 256 || s.expert_dim % 256)
        return fail(QMOE_ERR_UNSUPPORTED, "%s: hidden and expert_dim must be multiples of 256", fn);
    if (s.hidden > MAX_K || static_cast<int64_t>(s.top_k) * s.expert_dim > MAX_K)
        return fail(QMOE_ERR_UNSUPPORTED, "%s: hidden or top_k*expert_dim exceeds %lld", fn,
                    (long long)MAX_K);
    if (ws_bytes < need)
        return fail(QMOE_ERR_INVALID_ARGUMENT, "%s: workspace %zu < %zu bytes", fn, ws_bytes,
                    need);
    if (!aligned(router_W, 16) || !aligned(gate_stack, 16) || !aligned(up_stack, 16) ||
        !aligned(down_stack, 16) || !aligned(x, 16) || !aligned(residual, res_align) ||
        !aligned(ws, 16))
        return fail(QMOE_ERR_INVALID_ARGUMENT,
                    "%s: router, stacks, x/norm weight and ws must be 16-byte aligned", fn);
    return QMOE_OK;
}

// One MoE layer for s.n_tokens tokens.  With norm_w the input of token t is
// ffn_norm(residual_t) and x is unused; xn is workspace for the normed
// inputs of the tensor-core and separate-kernel forms.
static qmoe_status moe_core(const float* router_W, const void* gate_stack, const void* up_stack,
                            const void* down_stack, const qmoe_moe_shape& s, const float* x,
                            const float* norm_w, float eps, float* residual, int32_t* topk_idx,
                            float* topk_w, void* ws, float* xn, const DevInfo& dv,
                            cudaStream_t st) {
    const DevInfo* d = &dv;
    if (prefill_path(&s) && norm_w) {
        if (qmoe_status r = run_rmsnorm(residual, norm_w, s.n_tokens, s.hidden, eps, xn, st))
            return r;
        x = xn;
    }
    if (prefill_path(&s))
        return run_prefill(router_W, gate_stack, up_stack, down_stack, s, x, residual, topk_idx,
                           topk_w, ws, *d, st);

    const int H = s.hidden, F = s.expert_dim, E = s.num_experts, K = s.top_k;
    const int renorm = (s.route_flags & QMOE_ROUTE_NO_RENORM) ? 0 : 1;
    float* logits = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + WS_SYNC_BYTES);
    float* a = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + WS_SYNC_BYTES +
                                        moe_logits_bytes(&s));
    const int64_t grb = row_bytes_of(s.gate_qtype, H), urb = row_bytes_of(s.up_qtype, H);
    const int64_t drb = row_bytes_of(s.down_qtype, F);

    // Several tokens: batched launches that read each routed expert once for
    // all the tokens routed to it, the tokens split evenly over the launches.
    if (s.n_tokens >= 2 && batch_enabled()) {
        const int tmax = batch_tokens_max(s.gate_qtype, s.down_qtype, H, F, K, d->smem_optin);
        if (tmax >= 2) {
            const int nl = (s.n_tokens + tmax - 1) / tmax;
            int t0 = 0;
            for (int l = 0; l < nl; ++l) {
                const int tn = (s.n_tokens - t0) / (nl - l);
                BatchParams b = {};
                b.gu.W0 = static_cast<const uint8_t*>(gate_stack);
                b.gu.rb0 = grb;
                b.gu.es0 = grb * F;
                b.gu.W1 = static_cast<const uint8_t*>(up_stack);
                b.gu.rb1 = urb;
                b.gu.es1 = urb * F;
                b.gu.F = F;
                b.gu.E = E;
                b.gu.topk = K;
                b.gu.moe = 1;
                b.gu.renorm = renorm;
                b.dn.W0 = static_cast<const uint8_t*>(down_stack);
                b.dn.rb0 = drb;
                b.dn.es0 = drb * H;
                b.dn.F = F;
                b.dn.E = E;
                b.dn.topk = K;
                b.dn.moe = 1;
                b.dn.renorm = renorm;
                b.router = router_W;
                b.x = (norm_w ? residual : x) + static_cast<int64_t>(t0) * H;
                b.residual = residual + static_cast<int64_t>(t0) * H;
                b.logits = logits + static_cast<int64_t>(t0) * E;
                b.act = a;
                b.sync = static_cast<unsigned long long*>(ws);
                b.T = tn;
                b.E = E;
                b.H = H;
                b.F = F;
                b.topk = K;
                b.topk_idx_out = topk_idx ? topk_idx + static_cast<int64_t>(t0) * K : nullptr;
                b.topk_w_out = topk_w ? topk_w + static_cast<int64_t>(t0) * K : nullptr;
                b.norm_w = norm_w;
                b.eps = eps;
                b.err = d->err;
                cudaError_t ce = cudaSuccess;
                const int r = run_batch(s.gate_qtype, s.down_qtype, b, d->sms, d->smem_optin,
                                        &g_coop_pdl, st, &ce);
                if (r < 0) return cuda_fail(ce, "batched MoE launch");
                if (r == 0)
                    return fail(QMOE_ERR_UNSUPPORTED, "batched MoE kernel refused %d tokens", tn);
                t0 += tn;
            }
            return QMOE_OK;
        }
    }

    for (int t = 0; t < s.n_tokens; ++t) {
        const float* xt = norm_w ? residual + static_cast<int64_t>(t) * H
                                 : x + static_cast<int64_t>(t) * H;
        float* rt = residual + static_cast<int64_t>(t) * H;
        float* lt = logits + static_cast<int64_t>(t) * E;

        StreamParams pg = {};
        pg.units = static_cast<int64_t>(K) * F;
        pg.nb_seg = H / 256;
        pg.n_kseg = 1;
        pg.W0 = static_cast<const uint8_t*>(gate_stack);
        pg.rb0 = grb;
        pg.es0 = grb * F;
        pg.W1 = static_cast<const uint8_t*>(up_stack);
        pg.rb1 = urb;
        pg.es1 = urb * F;
        pg.x = xt;
        pg.out = a;
        pg.logits = lt;
        pg.E = E;
        pg.topk = K;
        pg.F = F;
        pg.topk_idx_out = topk_idx ? topk_idx + static_cast<int64_t>(t) * K : nullptr;
        pg.topk_w_out = topk_w ? topk_w + static_cast<int64_t>(t) * K : nullptr;
        pg.moe = 1;
        pg.renorm = renorm;

        StreamParams pd = {};
        pd.units = H;
        pd.nb_seg = F / 256;
        pd.n_kseg = K;
        pd.W0 = static_cast<const uint8_t*>(down_stack);
        pd.rb0 = drb;
        pd.es0 = drb * H;
        pd.x = a;
        pd.out = rt;
        pd.logits = lt;
        pd.E = E;
        pd.topk = K;
        pd.F = F;
        pd.moe = 1;
        pd.renorm = renorm;

        FusedParams f = {};
        f.gu = pg;
        f.dn = pd;
        f.router = router_W;
        f.logits = lt;
        f.sync = static_cast<unsigned long long*>(ws);
        f.moe = 1;
        f.E = E;
        f.H = H;
        f.topk = K;
        f.topk_idx_out = pg.topk_idx_out;
        f.topk_w_out = pg.topk_w_out;
        f.norm_w = norm_w;
        f.eps = eps;
        qmoe_status ferr = QMOE_OK;
        const int fr = dispatch_fused(s.gate_qtype, s.down_qtype, f, *d, st, &ferr);
        if (fr < 0) return ferr;
        if (fr > 0) continue;
        // the layer does not fit the fused kernel: router, gate/up, down
        if (norm_w) {
            float* xnt = xn + static_cast<int64_t>(t) * H;
            if (qmoe_status r = run_rmsnorm(xt, norm_w, 1, H, eps, xnt, st)) return r;
            xt = xnt;
            pg.x = xt;
        }
        if (qmoe_status r = run_f32_gemv(router_W, xt, lt, E, H, st)) return r;
        if (qmoe_status r = dispatch<MODE_GATEUP>(s.gate_qtype, pg, *d, st)) return r;
        if (qmoe_status r = dispatch<MODE_DOWN>(s.down_qtype, pd, *d, st)) return r;
    }
    return QMOE_OK;
}

qmoe_status moe_ffn(const float* router_W, const void* gate_stack, const void* up_stack,
                    const void* down_stack, const qmoe_moe_shape* shape, const float* x,
                    float* residual, int32_t* topk_idx, float* topk_w, void* ws,
                    size_t ws_bytes, void* stream) {
    g_last_error.clear();
    if (qmoe_status r = moe_check("moe_ffn", router_W, gate_stack, up_stack, down_stack, shape, x,
                                  residual, ws, ws_bytes, moe_ffn_workspace_size(shape), 4))
        return r;
    DevInfo* d = nullptr;
    if (qmoe_status r = device_info(&d)) return r;
    return moe_core(router_W, gate_stack, up_stack, down_stack, *shape, x, nullptr, 0.f, residual,
                    topk_idx, topk_w, ws, nullptr, *d, static_cast<cudaStream_t>(stream));
}

size_t moe_ffn_rmsnorm_workspace_size(const qmoe_moe_shape* shape) {
    const size_t base = moe_ffn_workspace_size(shape);
    if (!base) return 0;
    return base + static_cast<size_t>(shape->n_tokens) * static_cast<size_t>(shape->hidden) * 4;
}

qmoe_status moe_ffn_rmsnorm(const float* router_W, const void* gate_stack, const void* up_stack,
                            const void* down_stack, const qmoe_moe_shape* shape,
                            const float* norm_w, float eps, float* residual, int32_t* topk_idx,
                            float* topk_w, void* ws, size_t ws_bytes, void* stream) {
    g_last_error.clear();
    if (qmoe_status r = moe_check("moe_ffn_rmsnorm", router_W, gate_stack, up_stack, down_stack,
                                  shape, norm_w, residual, ws, ws_bytes,
                                  moe_ffn_rmsnorm_workspace_size(shape), 16))
        return r;
    if (!(eps >= 0.f) || !std::isfinite(eps))
        return fail(QMOE_ERR_INVALID_ARGUMENT, "moe_ffn_rmsnorm: eps=%g must be finite, >= 0",
                    static_cast<double>(eps));
    DevInfo* d = nullptr;
    if (qmoe_status r = device_info(&d)) return r;
    float* xn = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + moe_ffn_workspace_size(shape));
    return moe_core(router_W, gate_stack, up_stack, down_stack, *shape, nullptr, norm_w, eps,
                    residual, topk_idx, topk_w, ws, xn, *d, static_cast<cudaStream_t>(stream));
}

// ----------------------------------------------------- allocation-free call
// Scratch for moe_ffn_noalloc: a file-scope device array, so the call needs
// no allocation at all.  Every GPU that loads the library holds it until the
// process exits.  Host code may not use the symbol's name as a device
// address: the address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and passed down.
static __device__ __align__(256) unsigned char g_noalloc_ws[QMOE_NOALLOC_SCRATCH_BYTES];
static void* g_noalloc_ptr[64];
static std::mutex g_noalloc_mu;

qmoe_status moe_ffn_noalloc(const float* router_W, const void* gate_stack, const void* up_stack,
                            const void* down_stack, const qmoe_moe_shape* shape, const float* x,
                            float* residual, int32_t* topk_idx, float* topk_w, void* stream) {
    g_last_error.clear();
    if (!shape) return fail(QMOE_ERR_INVALID_ARGUMENT, "moe_ffn_noalloc: null shape");
    const size_t need = moe_ffn_workspace_size(shape);
    if (need > QMOE_NOALLOC_SCRATCH_BYTES)
        return fail(QMOE_ERR_UNSUPPORTED,
                    "moe_ffn_noalloc: this shape needs %zu bytes of scratch; the built-in "
                    "scratch holds %zu (use moe_ffn with a workspace)",
                    need, static_cast<size_t>(QMOE_NOALLOC_SCRATCH_BYTES));
    // the device must be one this library runs on before its scratch is looked up
    DevInfo* d = nullptr;
    if (qmoe_status r = device_info(&d)) return r;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void* ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_noalloc_ws);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
            g_noalloc_ptr[dev] = ptr;
        }
        ws = g_noalloc_ptr[dev];
    }
    return moe_ffn(router_W, gate_stack, up_stack, down_stack, shape, x, residual, topk_idx,
                   topk_w, ws, QMOE_NOALLOC_SCRATCH_BYTES, stream);
}

qmoe_status qmoe_set_exec_mode(int mode) {
    g_last_error.clear();
    if (mode != QMOE_EXEC_DEFAULT && mode != QMOE_EXEC_SEPARATE && mode != QMOE_EXEC_UNBATCHED)
        return fail(QMOE_ERR_INVALID_ARGUMENT, "qmoe_set_exec_mode: unknown mode %d", mode);
    g_exec_mode.store(mode);
    return QMOE_OK;
}

qmoe_status qmoe_set_fault_injection(uint64_t wait_limit_ns, int skip_arrive_cta) {
    g_last_error.clear();
    DevInfo* d = nullptr;
    if (qmoe_status s = device_info(&d)) return s;
    if (skip_arrive_cta < -1)
        return fail(QMOE_ERR_INVALID_ARGUMENT,
                    "qmoe_set_fault_injection: skip_arrive_cta=%d must be >= -1", skip_arrive_cta);
    DevCtl c;
    c.code = 0u;
    c.skip_arrive_cta = skip_arrive_cta;
    c.wait_ns = wait_limit_ns ? static_cast<unsigned long long>(wait_limit_ns) : DEFAULT_WAIT_NS;
    // everything after the error word; the device is idle first, so no
    // kernel sees a half-written setting
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    e = cudaMemcpy(reinterpret_cast<uint8_t*>(d->err) + offsetof(DevCtl, skip_arrive_cta),
                   &c.skip_arrive_cta, sizeof(DevCtl) - offsetof(DevCtl, skip_arrive_cta),
                   cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "write device control");
    return QMOE_OK;
}

qmoe_status qmoe_device_status(void* stream) {
    g_last_error.clear();
    DevInfo* d = nullptr;
    if (qmoe_status s = device_info(&d)) return s;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned v = 0, zero = 0;
    e = cudaMemcpy(&v, &d->err->code, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    if (v) {
        e = cudaMemcpy(&d->err->code, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
        if (v == pf::DEV_PF_RANGE)
            return fail(QMOE_ERR_UNSUPPORTED,
                        "a decoded gate/up weight is outside f16 range (code %u); the "
                        "many-token path cannot represent it", v);
        if (v == DEV_X_RANGE)
            return fail(QMOE_ERR_UNSUPPORTED,
                        "an activation of magnitude 2^106 or more reached a quantized product "
                        "(code %u); its output is not valid", v);
        if (v == DEV_ROUTE_RANGE)
            return fail(QMOE_ERR_CUDA,
                        "internal error: the routing produced an expert index outside [0, E) "
                        "(code %u); it was clamped, and the layer's output is not valid", v);
        return fail(QMOE_ERR_TIMEOUT, "a bounded device wait expired (code %u: %s)", v,
                    v == DEV_TIMEOUT_FULL    ? "stage never filled"
                    : v == DEV_TIMEOUT_EMPTY ? "stage never released"
                    : v == DEV_TIMEOUT_GRID  ? "grid barrier: not every CTA arrived"
                                             : "tensor-core pipeline stalled");
    }
    return QMOE_OK;
}

}  // extern "C"
