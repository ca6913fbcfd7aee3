// stream.cuh — the streaming decode GEMV engine shared by qmv, ffn_swiglu and
// moe_ffn (decode).
//
// One CTA per SM (persistent over a contiguous range of output units).
// Warp 8 is the producer: it stages weight rows into a ring of shared-memory
// stages with 1-D bulk TMA copies (cp.async.bulk, completion counted on an
// mbarrier).  Warps 0..7 are consumers.  A tile holds 8*R row slots; lane
// (g = lane/4, q = lane%4) owns slots rr*8 + g (rr < R) and quarter q of each
// 256-element group its warp is given: warp v takes groups v, v+8, ... of
// the chunk.  A lane loads its 64 x' values of a group into registers once
// and applies them to its R rows.  Per-row partial sums are reduced by
// shuffles across the four quarters and through shared memory across warps,
// in a fixed order (deterministic).
//
// Weight operands are read-only constants: the producer starts streaming
// them before griddepcontrol.wait, so a launch overlaps the tail of the
// kernel before it.  x, outputs and routing data are touched only after the
// wait.
//
// Modes:
//   QMV     y[r] = W[r] . x                         (overwrite)           R = 4
//   GATEUP  a[j] = w_s * silu(G_e[jj].x) * (U_e[jj].x),  j = s*F + jj      R = 4
//           (slots rr = 0,1 gate rows, rr = 2,3 up rows of the same units;
//            dense: one slot, w = 1)
//   DOWN    residual[i] += sum_s D_e_s[i] . a_s      (k-segments = slots)  R = 2
#pragma once
#include "formats.cuh"
#include "ptx.cuh"

namespace qmoe {

constexpr int NCW = 8;                    // consumer warps
constexpr int NTHREADS = (NCW + 1) * 32;  // + producer warp
constexpr int MAX_STAGES = 4;
constexpr int MAX_EXPERTS = 256;
constexpr int MAX_TOPK = 16;
constexpr int MAX_ROWS = 32;              // row slots per tile (8 * R)

enum Mode : int { MODE_QMV = 0, MODE_GATEUP = 1, MODE_DOWN = 2 };

struct StreamParams {
    int64_t units;       // output units: rows (QMV, DOWN) or gate/up row pairs (GATEUP)
    int nb_seg;          // 256-element groups per k-segment
    int n_kseg;          // k-segments: 1, or top_k for the MoE down product
    int chunk_ks;        // whole k-segments per chunk (when n_sbc == 1)
    int chunk_sb;        // groups per k-segment per chunk
    int n_sbc;           // chunks per k-segment (1 => chunks hold whole k-segments)
    int n_chunk;         // chunks per tile
    int piece_stride;    // smem bytes per (row, k-segment) piece
    int slot_stride;     // smem bytes per row slot
    int stage_bytes;
    int nstages;
    const uint8_t* W0;   // QMV: W; GATEUP: gate; DOWN: down
    int64_t rb0, es0;    // row bytes, expert stride (bytes)
    const uint8_t* W1;   // GATEUP: up
    int64_t rb1, es1;
    const float* x;      // QMV/GATEUP: x[K]; DOWN: a[n_kseg * K]
    float* out;          // QMV: y; GATEUP: a; DOWN: residual
    // routing (MoE): logits of this token, E experts, top-k, rows per expert
    const float* logits;
    int E, topk, F;
    int32_t* topk_idx_out;  // nullable, written by CTA 0 of GATEUP
    float* topk_w_out;
    int moe;
    unsigned* err;
};

template <int MODE> struct ModeGeom {
    static constexpr int R = (MODE == MODE_DOWN) ? 2 : 4;  // row slots per lane
    static constexpr int ROWS = 8 * R;                     // row slots per tile
    static constexpr int TU = (MODE == MODE_GATEUP) ? ROWS / 2 : ROWS;  // units per tile
    static constexpr int WK = NCW;                         // warps along K
};

// Shared-memory carve-up (dynamic): [barriers][topk][part][xs16][xq][stages]
struct SmemLayout {
    int off_full, off_empty, off_tidx, off_tw, off_logit, off_part, off_xs, off_xq, off_stage,
        total;
};

__host__ __device__ inline int align_up(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline SmemLayout smem_layout(const StreamParams& p) {
    SmemLayout L;
    int o = 0;
    L.off_full = o;  o += 8 * MAX_STAGES;
    L.off_empty = o; o += 8 * MAX_STAGES;
    L.off_tidx = o;  o += 4 * MAX_TOPK;
    L.off_tw = o;    o += 4 * MAX_TOPK;
    L.off_logit = o; o += 4 * MAX_EXPERTS;
    L.off_part = o;  o += 4 * 2 * NCW * MAX_ROWS;
    o = align_up(o, 16);
    L.off_xs = o;    o += 4 * 16 * p.nb_seg * p.n_kseg;
    o = align_up(o, 128);
    L.off_xq = o;    o += 4 * 256 * p.nb_seg * p.n_kseg;
    o = align_up(o, 128);
    L.off_stage = o; o += p.stage_bytes * p.nstages;
    o += 16;  // tail slack: a Q6_K lane's word loads reach <= 2 bytes past a super-block
    L.total = o;
    return L;
}

// Routing: softmax over the E logits, the k largest (ties: lower index),
// renormalised over those k — the page's "softmax, top-k, renormalize" of
// "aprender-serve 0.70.2 — forward_qwen3_moe_resident.rs" (module doc,
// moe_layer).  The renormalised weight of a selected expert equals
// exp(l_s - l_max) / sum over the selected k of exp(l_t - l_max).
// All threads of the CTA must call it.
__device__ inline void route_topk_cta(const float* __restrict__ logits, int E, int k,
                                      float* s_logit, int32_t* s_idx, float* s_w) {
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int e = tid; e < E; e += nt) s_logit[e] = __ldcg(logits + e);
    __syncthreads();
    // two threads per expert: each counts the experts that beat it over half of E
    for (int base = 0; base < E; base += nt / 2) {
        const int e = base + tid / 2, half = tid & 1;
        int rank = 0;
        if (e < E) {
            const float v = s_logit[e];
            const int u0 = half ? E / 2 : 0, u1 = half ? E : E / 2;
            for (int u = u0; u < u1; ++u) {
                const float w = s_logit[u];
                rank += (w > v) || (w == v && u < e);
            }
        }
        rank += __shfl_xor_sync(0xffffffffu, rank, 1);
        if (e < E && half == 0 && rank < k) s_idx[rank] = e;
    }
    __syncthreads();
    if (tid == 0) {
        const float lmax = s_logit[s_idx[0]];
        float z = 0.f;
        for (int s = 0; s < k; ++s) {
            const float p = expf(s_logit[s_idx[s]] - lmax);
            s_w[s] = p;
            z += p;
        }
        const float inv = 1.0f / z;
        for (int s = 0; s < k; ++s) s_w[s] *= inv;
    }
    __syncthreads();
}

template <class Fmt>
__device__ inline void build_xprime(const float* __restrict__ x, int ngroups, float* xq,
                                    float* xs, int tid, int nthreads) {
    // x' in the per-quarter interleaved order; xs = sum of x per 16 elements.
    // Every x' float4 slot (group g, i4, quarter q) holds four consecutive,
    // 16-byte-aligned elements of x (the formats' element orders keep
    // i = 4*i4 .. 4*i4+3 contiguous), each scaled by its own power of two.
    // Loads are batched (UNR in flight per thread) before any use.
    constexpr int UNR = 8;
    const int n4 = ngroups * 64;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float4* xq4 = reinterpret_cast<float4*>(xq);
    for (int base = tid; base < n4; base += nthreads * UNR) {
        float4 v[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int f = base + u * nthreads;
            if (f < n4) {
                const int g = f >> 6, i4 = (f >> 2) & 15, q = f & 3;
                v[u] = __ldcg(x4 + ((g * 256 + Fmt::elem(q, 4 * i4)) >> 2));
            }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int f = base + u * nthreads;
            if (f < n4) {
                const int i4 = (f >> 2) & 15, q = f & 3, i = 4 * i4;
                float4 o;
                o.x = v[u].x * xprime_scale(Fmt::pos(q, i));
                o.y = v[u].y * xprime_scale(Fmt::pos(q, i + 1));
                o.z = v[u].z * xprime_scale(Fmt::pos(q, i + 2));
                o.w = v[u].w * xprime_scale(Fmt::pos(q, i + 3));
                xq4[f] = o;
            }
        }
    }
    const int n16 = ngroups * 16;
    for (int base = tid; base < n16; base += nthreads * 2) {
        float4 v[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int g16 = base + u * nthreads;
            if (g16 < n16) {
#pragma unroll
                for (int k = 0; k < 4; ++k) v[u][k] = __ldcg(x4 + g16 * 4 + k);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int g16 = base + u * nthreads;
            if (g16 < n16) {
                float s = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) s += (v[u][k].x + v[u][k].y) + (v[u][k].z + v[u][k].w);
                xs[g16] = s;
            }
        }
    }
}

// Address of the bytes of (row slot r, k-segment ks) for the tile starting
// at unit u0; nullptr if the row's unit is outside [.., uend).
template <int MODE>
__device__ __forceinline__ const uint8_t* row_addr(const StreamParams& p, const int32_t* s_idx,
                                                   int64_t u0, int64_t uend, int r, int ks) {
    const int g = r & 7, rr = r >> 3;
    if (MODE == MODE_GATEUP) {
        const bool up = rr >= 2;
        const int64_t u = u0 + (rr & 1) * 8 + g;
        if (u >= uend) return nullptr;
        const uint8_t* base = up ? p.W1 : p.W0;
        const int64_t rb = up ? p.rb1 : p.rb0, es = up ? p.es1 : p.es0;
        if (p.moe) {
            const int s = static_cast<int>(u / p.F);
            const int64_t jj = u - static_cast<int64_t>(s) * p.F;
            return base + static_cast<int64_t>(s_idx[s]) * es + jj * rb;
        }
        return base + u * rb;
    }
    const int64_t u = u0 + r;
    if (u >= uend) return nullptr;
    if (MODE == MODE_QMV) return p.W0 + u * p.rb0;
    // DOWN
    if (p.moe) return p.W0 + static_cast<int64_t>(s_idx[ks]) * p.es0 + u * p.rb0;
    return p.W0 + u * p.rb0;
}

struct ChunkDesc {
    int ks0, nks, b0, nbp;
};

__device__ __forceinline__ ChunkDesc chunk_desc(const StreamParams& p, int c) {
    ChunkDesc d;
    if (p.n_sbc == 1) {
        d.ks0 = c * p.chunk_ks;
        d.nks = min(p.chunk_ks, p.n_kseg - d.ks0);
        d.b0 = 0;
        d.nbp = p.nb_seg;
    } else {
        d.ks0 = c / p.n_sbc;
        d.nks = 1;
        d.b0 = (c % p.n_sbc) * p.chunk_sb;
        d.nbp = min(p.chunk_sb, p.nb_seg - d.b0);
    }
    return d;
}

template <class Fmt, int MODE>
__global__ void __launch_bounds__(NTHREADS, 1) stream_gemv_kernel(const StreamParams p) {
    using G = ModeGeom<MODE>;
    constexpr int R = G::R;
    extern __shared__ __align__(128) uint8_t smem[];
    const SmemLayout L = smem_layout(p);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.off_empty);
    int32_t* s_idx = reinterpret_cast<int32_t*>(smem + L.off_tidx);
    float* s_w = reinterpret_cast<float*>(smem + L.off_tw);
    float* s_logit = reinterpret_cast<float*>(smem + L.off_logit);
    float* part = reinterpret_cast<float*>(smem + L.off_part);
    float* xs = reinterpret_cast<float*>(smem + L.off_xs);
    float* xq = reinterpret_cast<float*>(smem + L.off_xq);
    uint8_t* stages = smem + L.off_stage;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t cta = blockIdx.x, ncta = gridDim.x;
    const int64_t ubeg = p.units * cta / ncta, uend = p.units * (cta + 1) / ncta;

    if (tid == 0) {
        for (int s = 0; s < p.nstages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCW);
        }
        fence_barrier_init();
    }
    // Routing decides which expert rows are streamed.  The down product's
    // logits come from the router kernel two launches back, complete before
    // this grid was allowed to start; the gate/up kernel reads them right
    // after its own dependency wait.
    if (p.moe && MODE == MODE_DOWN) {
        route_topk_cta(p.logits, p.E, p.topk, s_logit, s_idx, s_w);
    } else if (p.moe && MODE == MODE_GATEUP) {
        pdl_wait();
        pdl_trigger();
        route_topk_cta(p.logits, p.E, p.topk, s_logit, s_idx, s_w);
        if (blockIdx.x == 0 && tid < p.topk) {
            if (p.topk_idx_out) p.topk_idx_out[tid] = s_idx[tid];
            if (p.topk_w_out) p.topk_w_out[tid] = s_w[tid];
        }
    } else {
        __syncthreads();
    }

    const int ntiles = static_cast<int>((uend - ubeg + G::TU - 1) / G::TU);

    if (warp == NCW) {
        // ------------------------------------------------------ producer
        const uint64_t pol = policy_evict_first();
        int it = 0;
        for (int t = 0; t < ntiles; ++t) {
            const int64_t u0 = ubeg + static_cast<int64_t>(G::TU) * t;
            for (int c = 0; c < p.n_chunk; ++c, ++it) {
                const int s = it % p.nstages;
                const int round = it / p.nstages;
                if (round > 0 &&
                    !mbar_wait_bounded(&empty[s], (round - 1) & 1, p.err, DEV_TIMEOUT_EMPTY))
                    return;
                const ChunkDesc cd = chunk_desc(p, c);
                const int ncopy = G::ROWS * cd.nks;
                const uint32_t seg_bytes = static_cast<uint32_t>(cd.nbp * Fmt::SBB);
                uint32_t mine = 0;
                for (int k = lane; k < ncopy; k += 32) {
                    const int r = k / cd.nks, pk = k % cd.nks;
                    const uint8_t* a = row_addr<MODE>(p, s_idx, u0, uend, r, cd.ks0 + pk);
                    if (a) {
                        const uintptr_t src = reinterpret_cast<uintptr_t>(a) +
                                              static_cast<uintptr_t>(cd.b0) * Fmt::SBB;
                        const uintptr_t lo = src & ~uintptr_t(15);
                        mine += static_cast<uint32_t>(((src + seg_bytes + 15) & ~uintptr_t(15)) - lo);
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
                if (lane == 0) mbar_arrive_expect_tx(&full[s], mine);
                __syncwarp();
                uint8_t* st = stages + static_cast<size_t>(s) * p.stage_bytes;
                for (int k = lane; k < ncopy; k += 32) {
                    const int r = k / cd.nks, pk = k % cd.nks;
                    const uint8_t* a = row_addr<MODE>(p, s_idx, u0, uend, r, cd.ks0 + pk);
                    if (a) {
                        const uintptr_t src = reinterpret_cast<uintptr_t>(a) +
                                              static_cast<uintptr_t>(cd.b0) * Fmt::SBB;
                        const uintptr_t lo = src & ~uintptr_t(15);
                        const uint32_t n =
                            static_cast<uint32_t>(((src + seg_bytes + 15) & ~uintptr_t(15)) - lo);
                        bulk_g2s(st + r * p.slot_stride + pk * p.piece_stride,
                                 reinterpret_cast<const void*>(lo), n, &full[s], pol);
                    }
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    if (!(p.moe && MODE == MODE_GATEUP)) {  // the MoE gate/up grid waited above
        pdl_wait();
        pdl_trigger();
    }
    build_xprime<Fmt>(p.x, p.nb_seg * p.n_kseg, xq, xs, tid, NCW * 32);
    named_bar(1, NCW * 32);

    const int v = warp;
    const int g = lane >> 2, q = lane & 3;
    const float4* xq4 = reinterpret_cast<const float4*>(xq);
    int it = 0;
    bool ok = true;
    for (int t = 0; t < ntiles && ok; ++t) {
        const int64_t u0 = ubeg + static_cast<int64_t>(G::TU) * t;
        float acc[R];
        // low 32 bits of each row's address (k-segment 0): only the 16-byte
        // phase is needed to find the row inside its staged slot
        uint32_t rowlo[R];
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            acc[rr] = 0.f;
            const uint8_t* a = row_addr<MODE>(p, s_idx, u0, uend, rr * 8 + g, 0);
            rowlo[rr] = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(a));
            if (MODE == MODE_DOWN && p.moe && a)  // k-segment 0's expert offset removed
                rowlo[rr] -= static_cast<uint32_t>(s_idx[0]) * static_cast<uint32_t>(p.es0);
        }
        for (int c = 0; c < p.n_chunk; ++c, ++it) {
            const int s = it % p.nstages;
            const int round = it / p.nstages;
            if (!mbar_wait_bounded(&full[s], round & 1, p.err, DEV_TIMEOUT_FULL)) {
                ok = false;
                break;
            }
            const ChunkDesc cd = chunk_desc(p, c);
            const uint8_t* st = stages + static_cast<size_t>(s) * p.stage_bytes;
            const int ntot = cd.nks * cd.nbp;
            const uint32_t b0off = static_cast<uint32_t>(cd.b0) * Fmt::SBB;
            for (int tt = v; tt < ntot; tt += G::WK) {
                const int pk = tt / cd.nbp, bb = tt - pk * cd.nbp;
                const int ks = cd.ks0 + pk, b = cd.b0 + bb;
                const int gidx = ks * p.nb_seg + b;
                float x[64];
                load_xq(xq4 + gidx * 64, q, x);
                const float* xsg = xs + gidx * 16;
                const uint32_t ksoff =
                    (MODE == MODE_DOWN && p.moe)
                        ? static_cast<uint32_t>(s_idx[ks]) * static_cast<uint32_t>(p.es0)
                        : 0u;
                // rows outside the CTA's range read (in-bounds, stale) slot
                // bytes; their sums are never written out
                const uint8_t* sbp[R];
#pragma unroll
                for (int rr = 0; rr < R; ++rr) {
                    const int delta = static_cast<int>((rowlo[rr] + ksoff + b0off) & 15u);
                    sbp[rr] = st + (rr * 8 + g) * p.slot_stride + pk * p.piece_stride + delta +
                              bb * Fmt::SBB;
                }
                Fmt::template dotR<R>(sbp, q, x, xsg, acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (!ok) break;
        float* pt = part + (t & 1) * NCW * MAX_ROWS;
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            float a = acc[rr];
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            if (q == 0) pt[v * MAX_ROWS + rr * 8 + g] = a;
        }
        named_bar(1, NCW * 32);
        const int ct = tid;
        if (ct < G::TU && u0 + ct < uend) {
            const int64_t u = u0 + ct;
            if (MODE == MODE_GATEUP) {
                float gs = 0.f, us = 0.f;
                for (int k = 0; k < G::WK; ++k) {
                    gs += pt[k * MAX_ROWS + ct];
                    us += pt[k * MAX_ROWS + G::TU + ct];
                }
                const float w = p.moe ? s_w[static_cast<int>(u / p.F)] : 1.0f;
                p.out[u] = w * ((gs / (1.0f + expf(-gs))) * us);
            } else {
                float y = 0.f;
                for (int k = 0; k < G::WK; ++k) y += pt[k * MAX_ROWS + ct];
                if (MODE == MODE_QMV)
                    p.out[u] = y;
                else
                    p.out[u] += y;
            }
        }
    }
}

}  // namespace qmoe
