// fused.cuh — one persistent kernel for a whole FFN layer at batch 1: the
// dense SwiGLU FFN ("ferrox-cuda 0.14.0 — src/gpu.rs", launch_dense_ffn_swiglu)
// or the decode-time MoE FFN ("aprender-serve 0.70.2 —
// forward_qwen3_moe_resident.rs", moe_layer): router GEMV, routing, the
// routed experts' gate/up products with SwiGLU and the routing weight, and
// the down products added to the residual.
//
// Why one kernel: at batch 1 every phase is a few microseconds of streaming,
// and each kernel boundary costs about as much again (launch, dependency
// flush, pipeline ramp).  Here the producer warp streams the gate/up rows and
// then, without waiting, the down rows through the same ring, so the down
// weights arrive while the gate/up products are still being reduced.  Phases
// that need every CTA's results (the logits, the activations a) are
// separated by a grid barrier; the kernel is launched cooperatively, one CTA
// per SM, so all CTAs are resident.
//
// Phases (consumer warps; the producer only streams):
//   MoE:   logits[e] = R[e].x for this CTA's experts      -> grid barrier 1
//          route (softmax, top-k, renormalise) in every CTA -> producer starts
//          a[s*F + j] = w_s * silu(G_e_s[j].x) * (U_e_s[j].x) -> grid barrier 2
//          residual[i] += sum_s D_e_s[i] . a_s
//   dense: a = silu(G x) * (U x) -> grid barrier -> residual += D a
//
// Grid barriers count arrivals in the first bytes of the workspace, which
// the kernel validates and resets itself (sync_open / sync_close below), so
// the workspace may hold anything.
// Every wait is bounded (2 s unless a test shortened the limit); on expiry
// the kernel records an error code and returns.
#pragma once
#include "stream.cuh"

namespace qmoe {

enum : unsigned { DEV_TIMEOUT_GRID = 3 };

struct FusedParams {
    StreamParams gu, dn;      // the two streamed phases (same ring geometry)
    const float* router;      // MoE: [E][H] f32
    float* logits;            // MoE: [E] (workspace)
    unsigned long long* sync; // grid-barrier state (workspace, 24 bytes)
    int moe, E, H, topk;
    int32_t* topk_idx_out;    // nullable
    float* topk_w_out;        // nullable
    const float* norm_w;      // nullable: ffn_norm weight [H]; gu.x is then the hidden state
    float eps;
    DevCtl* err;
};

struct FusedLayout {
    int off_full, off_empty, off_tidx, off_tw, off_logit, off_red, off_rpart, off_part, off_xs,
        off_xq, off_stage, total;
};

__host__ __device__ inline FusedLayout fused_layout(const FusedParams& f) {
    FusedLayout L;
    int o = 0;
    L.off_full = o;  o += 8 * MAX_STAGES;
    L.off_empty = o; o += 8 * MAX_STAGES;
    L.off_tidx = o;  o += 4 * MAX_TOPK;
    L.off_tw = o;    o += 4 * MAX_TOPK;
    L.off_logit = o; o += 4 * MAX_EXPERTS;
    L.off_red = o;   o += 4 * NCW;
    L.off_rpart = o; o += 4 * (32768 / 512);
    L.off_part = o;  o += 4 * 2 * NCW * MAX_ROWS;
    const int ng_gu = f.gu.nb_seg * f.gu.n_kseg, ng_dn = f.dn.nb_seg * f.dn.n_kseg;
    const int ng = ng_gu > ng_dn ? ng_gu : ng_dn;  // the down x table reuses the gate/up region
    o = align_up(o, 16);
    L.off_xs = o;    o += XS_GROUP_BYTES * ng;
    o = align_up(o, 128);
    L.off_xq = o;    o += XQ_GROUP_BYTES * ng;
    o = align_up(o, 128);
    L.off_stage = o; o += f.gu.stage_bytes * f.gu.nstages;
    o += 16;  // tail slack (see smem_layout)
    L.total = o;
    return L;
}

// Grid-barrier state, the first 24 bytes of the workspace: arrivals,
// finished CTAs and a validity word.  A call that finds the validity word
// set trusts the counters (the previous call on this workspace left them
// at zero); otherwise CTA 0 zeroes them and sets it while the other CTAs
// wait.  The last CTA to finish zeroes the counters again; a call that
// gives up on a wait clears the validity word, so the next call starts
// clean whatever the workspace held.
constexpr unsigned long long SYNC_VALID = 0x51A7E5EEDC0FFEE5ull;
enum { SYNC_ARRIVE = 0, SYNC_EXIT = 1, SYNC_TAG = 2 };

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void sync_invalidate(unsigned long long* sync) {
    atomicExch(sync + SYNC_TAG, 0ull);
}

// By one thread per CTA, after the dependency wait.  False on a timeout.
__device__ __forceinline__ bool sync_open(unsigned long long* sync, DevCtl* err) {
    if (ld_acquire_u64(sync + SYNC_TAG) == SYNC_VALID) return true;
    if (blockIdx.x == 0) {
        sync[SYNC_ARRIVE] = 0;
        sync[SYNC_EXIT] = 0;
        st_release_u64(sync + SYNC_TAG, SYNC_VALID);
        return true;
    }
    const uint64_t t0 = global_ns();
    const unsigned long long lim = wait_limit(err);
    while (ld_acquire_u64(sync + SYNC_TAG) != SYNC_VALID) {
        if (global_ns() - t0 > lim) {
            record_error(err, DEV_TIMEOUT_GRID);
            return false;
        }
        __nanosleep(64);
    }
    return true;
}

// Whether this CTA arrives at the grid barriers (by one thread per CTA at the
// kernel's start): always, unless a fault-injection test named it.
__device__ __forceinline__ bool arrives(const DevCtl* err) {
    return __ldcg(&err->skip_arrive_cta) != static_cast<int>(blockIdx.x);
}

// Grid barrier number `n` (1, 2, ...) of this call, by one thread per CTA
// after a CTA barrier has ordered the CTA's writes.  The arrival is a
// release, the wait an acquire (no full fence: one would also wait for the
// producer's copies in flight).  False if the other CTAs did not arrive
// within the wait limit.  `arrive` is false only in a fault-injection test.
__device__ __forceinline__ bool grid_barrier(unsigned long long* sync, unsigned n, DevCtl* err,
                                             bool arrive = true) {
    if (arrive)
        asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(sync + SYNC_ARRIVE)
                     : "memory");
    const unsigned long long target = static_cast<unsigned long long>(n) * gridDim.x;
    const uint64_t t0 = global_ns();
    const unsigned long long lim = wait_limit(err);
    while (ld_acquire_u64(sync + SYNC_ARRIVE) < target) {
        if (global_ns() - t0 > lim) {
            record_error(err, DEV_TIMEOUT_GRID);
            sync_invalidate(sync);
            return false;
        }
        __nanosleep(32);
    }
    return true;
}

// By one thread per CTA after its last barrier: the last CTA out leaves the
// counters at zero for the next call.
__device__ __forceinline__ void sync_close(unsigned long long* sync) {
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], 1;"
                 : "=l"(old)
                 : "l"(sync + SYNC_EXIT)
                 : "memory");
    if (old == static_cast<unsigned long long>(gridDim.x) - 1) {
        sync[SYNC_ARRIVE] = 0;
        sync[SYNC_EXIT] = 0;
    }
}

template <class FmtG, class FmtD>
__global__ void __launch_bounds__(NTHREADS, 1) fused_ffn_kernel(const FusedParams f) {
    extern __shared__ __align__(128) uint8_t smem[];
    const FusedLayout L = fused_layout(f);
    Ring ring;
    ring.full = reinterpret_cast<uint64_t*>(smem + L.off_full);
    ring.empty = reinterpret_cast<uint64_t*>(smem + L.off_empty);
    ring.stages = smem + L.off_stage;
    ring.nstages = f.gu.nstages;
    ring.stage_bytes = f.gu.stage_bytes;
    int32_t* s_idx = reinterpret_cast<int32_t*>(smem + L.off_tidx);
    float* s_w = reinterpret_cast<float*>(smem + L.off_tw);
    uint32_t* s_key = reinterpret_cast<uint32_t*>(smem + L.off_logit);
    float* red = reinterpret_cast<float*>(smem + L.off_red);
    float* rpart = reinterpret_cast<float*>(smem + L.off_rpart);
    float* part = reinterpret_cast<float*>(smem + L.off_part);
    float* xs = reinterpret_cast<float*>(smem + L.off_xs);
    float* xq = reinterpret_cast<float*>(smem + L.off_xq);
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t cta = blockIdx.x, ncta = gridDim.x;
    int64_t gb, ge, db, de;
    unit_range(f.gu, static_cast<int>(cta), gb, ge);
    unit_range(f.dn, static_cast<int>(cta), db, de);
    constexpr int NC = NCW * 32;  // consumer threads

    if (tid == NC) {
        for (int s = 0; s < ring.nstages; ++s) {
            mbar_init(&ring.full[s], 1);
            mbar_init(&ring.empty[s], NCW);
        }
        fence_barrier_init();
        s_abort = 0;
    }
    __syncthreads();

    if (warp == NCW) {
        // ------------------------------------------------------ producer
        if (f.moe) {
            // this CTA's router rows are constant: pull them into L2 now
            if (lane == 0)
                for (int64_t e = cta; e < f.E; e += ncta)
                    bulk_prefetch_l2(f.router + e * f.H, static_cast<uint32_t>(f.H) * 4u);
            named_bar(2, NTHREADS);  // the consumers have routed this token
            if (s_abort) return;
        }
        int it = 0;
        if (produce_phase<FmtG, MODE_GATEUP>(f.gu, ring, s_idx, gb, ge, it, lane))
            produce_phase<FmtD, MODE_DOWN>(f.dn, ring, s_idx, db, de, it, lane);
        return;
    }

    // ---------------------------------------------------------- consumers
    pdl_wait();
    pdl_trigger();
    if (tid == 0 && !sync_open(f.sync, f.err)) s_abort = 1;
    const bool arrive = tid == 0 && arrives(f.err);
    // ffn_norm (optional): every CTA reads the whole hidden state anyway
    const float inv =
        f.norm_w ? rms_inverse(f.gu.x, f.gu.nb_seg * 256, f.eps, red, tid, NC, 1) : 1.f;
    // with H a multiple of 512 the x-table pass also forms this CTA's first logit
    const bool rmerge = f.moe && (f.H % 512) == 0 && cta < f.E;
    build_xprime<FmtG, 2>(f.gu.x, f.gu.nb_seg, f.gu.nb_seg * 16, xq, xs, tid, NC, f.err, f.norm_w,
                          inv, nullptr,
                          f.H / 16, rmerge ? f.router + cta * f.H : nullptr, rpart);
    if (f.moe) {
        if (rmerge) {
            named_bar(1, NC);
            if (tid == 0) {
                float sum = 0.f;
                for (int j = 0; j < f.H / 512; ++j) sum += rpart[j];
                f.logits[cta] = sum;
            }
        }
        // logits of this CTA's (other) experts: e = cta, cta + ncta, ...
        const float4* x4 = reinterpret_cast<const float4*>(f.gu.x);
        for (int64_t e = rmerge ? cta + ncta : cta; e < f.E; e += ncta) {
            const float4* r4 = reinterpret_cast<const float4*>(f.router + e * f.H);
            float acc = 0.f;
            const float4* n4 = reinterpret_cast<const float4*>(f.norm_w);
            for (int j = tid; j < f.H / 4; j += NC) {
                const float4 w = __ldg(r4 + j);
                float4 xv = __ldcg(x4 + j);
                if (n4) {
                    const float4 nv = __ldg(n4 + j);
                    xv.x *= inv * nv.x;
                    xv.y *= inv * nv.y;
                    xv.z *= inv * nv.z;
                    xv.w *= inv * nv.w;
                }
                acc = fmaf(w.x, xv.x, acc);
                acc = fmaf(w.y, xv.y, acc);
                acc = fmaf(w.z, xv.z, acc);
                acc = fmaf(w.w, xv.w, acc);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) red[warp] = acc;
            named_bar(1, NC);
            if (tid == 0) {
                float s = 0.f;
                for (int k = 0; k < NCW; ++k) s += red[k];
                f.logits[e] = s;
            }
            named_bar(1, NC);
        }
        named_bar(1, NC);
        if (tid == 0 && !s_abort && !grid_barrier(f.sync, 1, f.err, arrive)) s_abort = 1;
        named_bar(1, NC);
        if (s_abort) {
            if (tid == 0) sync_invalidate(f.sync);
            named_bar_arrive(2, NTHREADS);  // release the producer, which then returns
            return;
        }
        route_topk(f.logits, f.E, f.topk, s_key, s_idx, s_w, tid, NC, 1, f.gu.renorm, f.err);
        if (cta == 0 && tid < f.topk) {
            if (f.topk_idx_out) f.topk_idx_out[tid] = s_idx[tid];
            if (f.topk_w_out) f.topk_w_out[tid] = s_w[tid];
        }
        named_bar_arrive(2, NTHREADS);  // the producer may stream the routed experts
    } else {
        named_bar(1, NC);  // x table complete
        if (s_abort) {
            if (tid == 0) sync_invalidate(f.sync);
            return;
        }
    }

    int it = 0;
    bool good =
        consume_phase<FmtG, MODE_GATEUP>(f.gu, ring, s_idx, s_w, xq, xs, part, gb, ge, it, tid);
    // every CTA's activations a must be complete before any CTA reads them
    named_bar(1, NC);
    if (tid == 0 && good && !grid_barrier(f.sync, f.moe ? 2u : 1u, f.err, arrive)) s_abort = 1;
    named_bar(1, NC);
    if (!good || s_abort) {
        if (tid == 0) sync_invalidate(f.sync);
        return;
    }
    build_xprime<FmtD>(f.dn.x, f.dn.nb_seg * f.dn.n_kseg, f.dn.nb_seg * f.dn.n_kseg * 16, xq, xs,
                       tid, NC, f.err);
    named_bar(1, NC);
    good = consume_phase<FmtD, MODE_DOWN>(f.dn, ring, s_idx, s_w, xq, xs, part, db, de, it, tid);
    if (tid == 0) {
        if (good)
            sync_close(f.sync);
        else
            sync_invalidate(f.sync);
    }
}

}  // namespace qmoe
