// batch.cu — host side of the batched decode MoE kernel (batch.cuh):
// shared-memory planning, the largest token count per launch, and the
// cooperative launch for every pair of gate/up and down formats.  Built as
// its own translation unit beside qmoe.cu.
#include <cuda_runtime.h>

#include "batch.cuh"

namespace qmoe {

// One stage must hold a whole gate/up tile (32 rows); the down phase is
// chunked as the batch-1 kernel's.  Two stages and the x tables must fit.
template <class FmtG, class FmtD>
static bool plan_batch(BatchParams& b, int smem_optin, int* smem_bytes) {
    b.gu.stage_bytes = b.dn.stage_bytes = 0;
    b.gu.nstages = b.dn.nstages = 0;
    const int room = smem_optin - batch_layout(b).total;
    if (room <= 0) return false;
    const int budget = room / 2;
    if (!plan_chunks<FmtG, MODE_GATEUP>(b.gu, budget) || b.gu.n_chunk != 1) return false;
    if (!plan_chunks<FmtD, MODE_DOWN>(b.dn, budget)) return false;
    const int sb = b.gu.stage_bytes > b.dn.stage_bytes ? b.gu.stage_bytes : b.dn.stage_bytes;
    int ns = room / sb;
    if (ns > MAX_STAGES) ns = MAX_STAGES;
    if (ns < 2) return false;
    b.gu.stage_bytes = b.dn.stage_bytes = sb;
    b.gu.nstages = b.dn.nstages = ns;
    *smem_bytes = batch_layout(b).total;
    return *smem_bytes <= smem_optin;
}

static void batch_shape(BatchParams& b, int T, int H, int F, int K) {
    b.T = T;
    b.H = H;
    b.F = F;
    b.topk = K;
    b.gu.nb_seg = H / 256;
    b.gu.n_kseg = 1;
    b.dn.nb_seg = F / 256;
    b.dn.n_kseg = K;
}

template <class FmtG, class FmtD>
static int tokens_max(int H, int F, int K, int smem_optin) {
    for (int T = TB_MAX; T >= 2; --T) {
        BatchParams b = {};
        batch_shape(b, T, H, F, K);
        int smem = 0;
        if (plan_batch<FmtG, FmtD>(b, smem_optin, &smem)) return T;
    }
    return 0;
}

template <class FmtG, class FmtD>
static int launch(BatchParams b, int sms, int smem_optin, int* coop_pdl, cudaStream_t st,
                  cudaError_t* cerr) {
    int smem = 0;
    batch_shape(b, b.T, b.H, b.F, b.topk);
    if (!plan_batch<FmtG, FmtD>(b, smem_optin, &smem)) return 0;
    auto kern = moe_batch_kernel<FmtG, FmtD>;
    static int configured_smem[64] = {};  // per instantiation and device
    int dev = 0;
    cudaGetDevice(&dev);
    if (smem > configured_smem[dev & 63]) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) {
            *cerr = e;
            return -1;
        }
        configured_smem[dev & 63] = smem;
    }
    b.gu.err = b.dn.err = b.err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = *coop_pdl == 0 ? 1 : 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, b);
    if (e != cudaSuccess && *coop_pdl < 0) {
        (void)cudaGetLastError();
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, b);
        if (e == cudaSuccess) *coop_pdl = 0;
    }
    if (e != cudaSuccess) {
        *cerr = e;
        return -1;
    }
    if (*coop_pdl < 0) *coop_pdl = 1;
    return 1;
}

// Format dispatch: Op<FmtG, FmtD>::run(args...) for the qtype pair.
template <template <class, class> class Op, class FmtG, typename... A>
static int by_down(int dq, A... a) {
    switch (dq) {
    case QT_Q8_0: return Op<FmtG, FmtQ80>::run(a...);
    case QT_Q4_0: return Op<FmtG, FmtQ40>::run(a...);
    case QT_Q4_K: return Op<FmtG, FmtQ4K>::run(a...);
    case QT_Q5_K: return Op<FmtG, FmtQ5K>::run(a...);
    case QT_Q6_K: return Op<FmtG, FmtQ6K>::run(a...);
    default: return 0;
    }
}
template <template <class, class> class Op, typename... A>
static int by_formats(int gq, int dq, A... a) {
    switch (gq) {
    case QT_Q8_0: return by_down<Op, FmtQ80>(dq, a...);
    case QT_Q4_0: return by_down<Op, FmtQ40>(dq, a...);
    case QT_Q4_K: return by_down<Op, FmtQ4K>(dq, a...);
    case QT_Q5_K: return by_down<Op, FmtQ5K>(dq, a...);
    case QT_Q6_K: return by_down<Op, FmtQ6K>(dq, a...);
    default: return 0;
    }
}

template <class FmtG, class FmtD>
struct TokensMaxOp {
    static int run(int H, int F, int K, int smem_optin) {
        return tokens_max<FmtG, FmtD>(H, F, K, smem_optin);
    }
};
template <class FmtG, class FmtD>
struct LaunchOp {
    static int run(BatchParams b, int sms, int smem_optin, int* coop_pdl, cudaStream_t st,
                   cudaError_t* cerr) {
        return launch<FmtG, FmtD>(b, sms, smem_optin, coop_pdl, st, cerr);
    }
};

int batch_tokens_max(int gq, int dq, int H, int F, int K, int smem_optin) {
    if (H % 256 || F % 256 || H <= 0 || F <= 0 || K <= 0 || K > MAX_TOPK) return 0;
    return by_formats<TokensMaxOp>(gq, dq, H, F, K, smem_optin);
}

int run_batch(int gq, int dq, BatchParams b, int sms, int smem_optin, int* coop_pdl,
              cudaStream_t st, cudaError_t* cerr) {
    if (b.T < 2 || b.T > TB_MAX) return 0;
    return by_formats<LaunchOp>(gq, dq, b, sms, smem_optin, coop_pdl, st, cerr);
}

}  // namespace qmoe
