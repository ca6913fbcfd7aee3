// batch.cuh — the decode MoE FFN for a small batch of tokens (2..TB_MAX per
// launch) in one persistent kernel that stages each routed expert's gate/up
// rows once for all the tokens routed to it.
//
// The pages give the weight-read-once argument for batched input: the
// batched apply of "ferrox-core 0.16.0 — weight_matrix.rs" (apply_batch)
// streams a weight row once and dots it with every vector of the batch,
// where the per-token loop would stream the whole matrix again for each
// token.  The MoE op order of "aprender-serve 0.70.2 —
// forward_qwen3_moe_resident.rs" (moe_layer) is kept per token.
//
// Phases (one cooperative launch, one CTA per SM):
//   1. logits[t][e] = R[e] . x_t for this CTA's experts, all tokens
//                                                         -> grid barrier 1
//   2. every CTA routes every token (one warp per token: softmax, top-k,
//      renormalise) and groups the (token, slot) pairs by expert: the active
//      experts in ascending order, each with its pairs in token order
//   3. gate/up: units = (active expert, feature), tiles of 16 units inside
//      one expert, split over the CTAs by work (gu_range); each staged tile
//      is reduced once per pair of its expert:
//      a[t][s][f] = w_ts * silu(G_e[f] . x_t) * (U_e[f] . x_t) -> grid barrier 2
//   4. down: units = (token, output row), as the batch-1 kernel's down phase
//      per token: residual[t][i] += sum_s D_e_ts[i] . a[t][s] (the k routed
//      rows of a unit are its k-segments).  A unit's rows are reduced across
//      all eight consumer warps, and each residual element has one writer.
// The producer warp streams the gate/up tiles and then the down tiles of the
// CTA through one ring, as in the batch-1 fused kernel.
//
// x tables: phase 3 keeps one per token (T * H f32); phase 4 builds the
// table of one token's activations (k * F values) when the CTA's down units
// reach that token.  Gate/up tiles hold whole rows (one chunk per tile).
#pragma once
#include "fused.cuh"

namespace qmoe {

constexpr int TB_MAX = 16;                  // tokens per batched launch
constexpr int MAX_PAIRS = TB_MAX * MAX_TOPK;

struct BatchParams {
    StreamParams gu, dn;   // gate/up (MODE_GATEUP, expert-major) and down (MODE_DOWN, per token)
    const float* router;   // [E][H] f32
    const float* x;        // [T][H]: the FFN input, or the hidden state with norm_w
    float* residual;       // [T][H], in place
    float* logits;         // [T][E] (workspace)
    float* act;            // [T][k][F] (workspace): the activations of each (token, slot)
    unsigned long long* sync;
    int T, E, H, F, topk;
    int32_t* topk_idx_out;  // [T][k] or null
    float* topk_w_out;
    const float* norm_w;    // null, or the ffn_norm weight [H]
    float eps;
    DevCtl* err;
};

struct BatchLayout {
    int off_full, off_empty, off_ridx, off_rw, off_mask, off_slot, off_act, off_start, off_ptok,
        off_pw, off_porig, off_inv, off_red, off_rpart, off_part, off_xs, off_xq, off_stage,
        total;
};

// Groups of 256 the x region holds: every token's input (gate/up) or one
// token's k activation rows (down).
__host__ __device__ inline int batch_table_groups(const BatchParams& b) {
    const int gu = b.T * (b.H / 256), dn = b.topk * (b.F / 256);
    return gu > dn ? gu : dn;
}

__host__ __device__ inline BatchLayout batch_layout(const BatchParams& b) {
    BatchLayout L;
    int o = 0;
    L.off_full = o;  o += 8 * MAX_STAGES;
    L.off_empty = o; o += 8 * MAX_STAGES;
    L.off_ridx = o;  o += 4 * MAX_PAIRS;
    L.off_rw = o;    o += 4 * MAX_PAIRS;
    L.off_mask = o;  o += 4 * MAX_EXPERTS;
    L.off_slot = o;  o += 4 * MAX_EXPERTS;
    L.off_act = o;   o += 4 * MAX_EXPERTS;
    L.off_start = o; o += 4 * (MAX_EXPERTS + 4);
    L.off_ptok = o;  o += 4 * MAX_PAIRS;
    L.off_pw = o;    o += 4 * MAX_PAIRS;
    L.off_porig = o; o += 4 * MAX_PAIRS;
    L.off_inv = o;   o += 4 * TB_MAX;
    L.off_red = o;   o += 4 * NCW * TB_MAX;
    L.off_rpart = o; o += 4 * TB_MAX * (32768 / 512);
    L.off_part = o;  o += 4 * 2 * b.T * NCW * MAX_ROWS;
    const int ng = batch_table_groups(b);
    o = align_up(o, 16);
    L.off_xs = o;    o += XS_GROUP_BYTES * ng;
    o = align_up(o, 128);
    L.off_xq = o;    o += XQ_GROUP_BYTES * ng;
    o = align_up(o, 128);
    L.off_stage = o; o += b.gu.stage_bytes * b.gu.nstages;
    o += 16;  // tail slack (see smem_layout)
    L.total = o;
    return L;
}

// Routing of one token by one warp: softmax over the E logits, the k
// largest (ties: lower expert index), renormalised over those k — as
// route_topk, with the same ranking keys (route.cuh), the same non-finite
// rule and the same weights: w_s = exp(l_s - l_0) / sum over the k
// selected (over all E with renorm = 0).  Lane l holds experts
// [l*m, l*m + m), so among equal keys the lowest lane holds the lowest
// index; k rounds of a warp max pick the ranks in order.  A taken expert's
// key becomes 0, which no logit has.
__device__ __forceinline__ void route_warp(const float* __restrict__ lg, int E, int k, int lane,
                                           int renorm, int32_t* idx, float* w, DevCtl* err) {
    constexpr int M = MAX_EXPERTS / 32;
    const int m = (E + 31) >> 5;
    uint32_t key[M];
    float val[M];
#pragma unroll
    for (int j = 0; j < M; ++j) {
        const int e = lane * m + j;
        const bool valid = j < m && e < E;
        val[j] = valid ? __ldcg(lg + e) : 0.f;
        key[j] = valid ? route_key(val[j]) : 0u;
    }
    int my_e = 0;
    uint32_t my_key = 0u;
    for (int s = 0; s < k; ++s) {
        uint32_t bk = 0u;
        int bj = 0;
#pragma unroll
        for (int j = 0; j < M; ++j)
            if (key[j] > bk) {
                bk = key[j];
                bj = j;
            }
        const uint32_t mx = __reduce_max_sync(0xffffffffu, bk);
        const int wl = __ffs(__ballot_sync(0xffffffffu, bk == mx)) - 1;
        if (lane == wl) {
#pragma unroll
            for (int j = 0; j < M; ++j)
                if (j == bj) key[j] = 0u;
        }
        const int e = __shfl_sync(0xffffffffu, lane * m + bj, wl);
        if (lane == s) {
            my_e = e;
            my_key = mx;
        }
    }
    bool bad = false;
    if (lane < k) my_e = route_clamp(my_e, E, &bad);
    const float my_l = route_key_value(my_key);
    const float lmax = __shfl_sync(0xffffffffu, my_l, 0);
    const float pr = lane < k ? expf(my_l - lmax) : 0.f;
    float z = pr;
    if (!renorm) {
        z = 0.f;
#pragma unroll
        for (int j = 0; j < M; ++j)
            if (j < m && lane * m + j < E) z += expf(val[j] - lmax);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    float wv = pr / z;
    if (route_degenerate(lmax)) {
        my_e = lane;
        wv = __int_as_float(0x7FC00000);
    }
    if (lane < k) {
        idx[lane] = my_e;
        w[lane] = wv;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) record_error(err, DEV_ROUTE_RANGE);
}

// Pair lists shared by the consumer phases (shared memory).
struct PairLists {
    const int32_t* act_e;   // [n_act] expert of each active slot, ascending
    const int32_t* start;   // [n_act + 1] first pair of each slot
    const int32_t* tok;     // [pairs] token of each pair
    const float* w;         // [pairs] routing weight of each pair
    const int32_t* orig;    // [pairs] t * k + s: the pair's (token, rank) row of act
};

// Gate/up tiles of [ubeg, uend) (multiples of 16 units, one expert each).
// For every pair (t, s) of the tile's expert: act[t][s][f] = w * silu(g) * u.
template <class Fmt>
__device__ bool consume_batch_gateup(const StreamParams& p, const Ring& ring, const PairLists& pl,
                                     const float* xq, const float* xs, float* part, int T,
                                     float* act, int64_t ubeg, int64_t uend, int& it, int tid) {
    using G = ModeGeom<MODE_GATEUP>;
    constexpr int R = G::R;
    const int v = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q = lane & 3;
    const float4* xq4 = reinterpret_cast<const float4*>(xq);
    const int ntiles = static_cast<int>((uend - ubeg) / G::TU);
    const int nb = p.nb_seg;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
        const int64_t u0 = ubeg + static_cast<int64_t>(G::TU) * t;
        const int a = tile_slot<MODE_GATEUP>(p, u0);
        const int jj0 = static_cast<int>(u0 - static_cast<int64_t>(a) * p.F);
        const int pb = pl.start[a], pn = pl.start[a + 1] - pb;
        uint32_t rowlo[R];
        int rowoff[R];
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            const int r = rr * 8 + g;
            int h = r;
            if (p.runs) {
                const RunSlot rs = run_of<MODE_GATEUP>(p, u0, a, r);
                h = rs.head;
                rowoff[rr] = run_dst(p, rs.head, rs.idx) + (r - rs.head) * p.slot_stride;
            } else {
                rowoff[rr] = r * p.slot_stride;
            }
            rowlo[rr] = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(
                row_addr<MODE_GATEUP>(p, pl.act_e, u0, a, uend, h, 0)));
        }
        const int s = it % ring.nstages;
        const int round = it / ring.nstages;
        if (ok && !mbar_wait_bounded(&ring.full[s], round & 1, p.err, DEV_TIMEOUT_FULL)) ok = false;
        ok = __all_sync(0xffffffffu, ok);
        const uint8_t* st = ring.stages + static_cast<size_t>(s) * ring.stage_bytes;
        const uint8_t* sbp0[R];
#pragma unroll
        for (int rr = 0; rr < R; ++rr) sbp0[rr] = st + rowoff[rr] + (rowlo[rr] & 15u);
        float* pt = part + (t & 1) * T * NCW * MAX_ROWS;
        for (int j = 0; j < pn; ++j) {
            const int tok = pl.tok[pb + j];
            float acc[R];
#pragma unroll
            for (int rr = 0; rr < R; ++rr) acc[rr] = 0.f;
            if (ok) {
                for (int b = v; b < nb; b += G::WK) {
                    const int gidx = tok * nb + b;
                    const uint8_t* sbp[R];
#pragma unroll
                    for (int rr = 0; rr < R; ++rr) sbp[rr] = sbp0[rr] + b * Fmt::SBB;
                    const float* xsg = xs + gidx * XS_GROUP_FLOATS;
                    Fmt::template dotR<R>(sbp, q, xq4 + gidx * 64 + q, xsg, xsg + 16, 8, acc);
                }
            }
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                float sum = acc[rr];
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                if (q == 0) pt[(j * NCW + v) * MAX_ROWS + rr * 8 + g] = sum;
            }
        }
        ++it;
        __syncwarp();
        if (lane == 0) mbar_arrive(&ring.empty[s]);
        ok = named_bar_and(1, NCW * 32, ok);
        // lanes 0-7 of a 16-lane group: gate row of unit uu; 8-15: its up row
        const int k8 = tid & 7, uu = tid >> 4, up = (tid >> 3) & 1;
        for (int j = 0; j < pn; ++j) {
            float vs = pt[(j * NCW + k8) * MAX_ROWS + up * G::TU + uu];
            vs += __shfl_xor_sync(0xffffffffu, vs, 1);
            vs += __shfl_xor_sync(0xffffffffu, vs, 2);
            vs += __shfl_xor_sync(0xffffffffu, vs, 4);
            const float us = __shfl_down_sync(0xffffffffu, vs, 8);
            if (ok && up == 0 && k8 == 0)
                act[static_cast<int64_t>(pl.orig[pb + j]) * p.F + jj0 + uu] =
                    pl.w[pb + j] * ((vs / (1.0f + expf(-vs))) * us);
        }
    }
    return ok;
}

// Gate/up tiles are split over the CTAs by work, not by count: a tile is
// staged once and then reduced once per pair of its expert, so a tile of an
// expert with n pairs weighs GU_TILE_W + GU_PAIR_W * n.  Experts chosen by
// several tokens would otherwise make their CTAs the slowest of the grid.
constexpr int GU_TILE_W = 1, GU_PAIR_W = 2;

// Work before active expert a (tpe tiles per expert; start: first pair of
// each expert).
__device__ __forceinline__ int64_t gu_work_before(const int32_t* start, int a, int tpe) {
    return static_cast<int64_t>(tpe) * (GU_TILE_W * a + GU_PAIR_W * start[a]);
}

// The first tile whose work starts at or after `target`.
__device__ __forceinline__ int64_t gu_tile_at(int64_t target, const int32_t* start, int nact,
                                              int tpe) {
    int lo = 0, hi = nact;  // the largest a with work_before(a) <= target
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (gu_work_before(start, mid, tpe) <= target)
            lo = mid;
        else
            hi = mid - 1;
    }
    if (lo >= nact) return static_cast<int64_t>(nact) * tpe;
    const int64_t w = GU_TILE_W + GU_PAIR_W * (start[lo + 1] - start[lo]);
    return static_cast<int64_t>(lo) * tpe + (target - gu_work_before(start, lo, tpe) + w - 1) / w;
}

// Gate/up tiles [tb, te) of CTA `cta`.
__device__ __forceinline__ void gu_range(const int32_t* start, int nact, int tpe, int cta,
                                         int ncta, int64_t& tb, int64_t& te) {
    const int64_t total = gu_work_before(start, nact, tpe);
    tb = gu_tile_at(total * cta / ncta, start, nact, tpe);
    te = gu_tile_at(total * (cta + 1) / ncta, start, nact, tpe);
}

// Tiles [tb, te) of `ntiles`, split evenly over the grid.
__device__ __forceinline__ void tile_range(int64_t ntiles, int cta, int ncta, int64_t& tb,
                                           int64_t& te) {
    const int64_t q = ntiles / ncta, r = ntiles % ncta;
    tb = q * cta + (cta < r ? cta : r);
    te = tb + q + (cta < r ? 1 : 0);
}

template <class FmtG, class FmtD>
__global__ void __launch_bounds__(NTHREADS, 1) moe_batch_kernel(const BatchParams b) {
    extern __shared__ __align__(128) uint8_t smem[];
    const BatchLayout L = batch_layout(b);
    Ring ring;
    ring.full = reinterpret_cast<uint64_t*>(smem + L.off_full);
    ring.empty = reinterpret_cast<uint64_t*>(smem + L.off_empty);
    ring.stages = smem + L.off_stage;
    ring.nstages = b.gu.nstages;
    ring.stage_bytes = b.gu.stage_bytes;
    int32_t* s_ridx = reinterpret_cast<int32_t*>(smem + L.off_ridx);
    float* s_rw = reinterpret_cast<float*>(smem + L.off_rw);
    uint32_t* s_mask = reinterpret_cast<uint32_t*>(smem + L.off_mask);
    int32_t* s_slot = reinterpret_cast<int32_t*>(smem + L.off_slot);
    int32_t* s_act = reinterpret_cast<int32_t*>(smem + L.off_act);
    int32_t* s_start = reinterpret_cast<int32_t*>(smem + L.off_start);
    int32_t* s_ptok = reinterpret_cast<int32_t*>(smem + L.off_ptok);
    float* s_pw = reinterpret_cast<float*>(smem + L.off_pw);
    int32_t* s_porig = reinterpret_cast<int32_t*>(smem + L.off_porig);
    float* s_inv = reinterpret_cast<float*>(smem + L.off_inv);
    float* red = reinterpret_cast<float*>(smem + L.off_red);
    float* rpart = reinterpret_cast<float*>(smem + L.off_rpart);
    float* part = reinterpret_cast<float*>(smem + L.off_part);
    float* xs = reinterpret_cast<float*>(smem + L.off_xs);
    float* xq = reinterpret_cast<float*>(smem + L.off_xq);
    __shared__ int s_abort, s_nact;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x, ncta = gridDim.x;
    const int T = b.T, E = b.E, H = b.H, F = b.F, K = b.topk;
    constexpr int NC = NCW * 32;

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
        if (lane == 0)
            for (int e = cta; e < E; e += ncta)
                bulk_prefetch_l2(b.router + static_cast<int64_t>(e) * H,
                                 static_cast<uint32_t>(H) * 4u);
        named_bar(2, NTHREADS);  // the consumers have routed and grouped the tokens
        if (s_abort) return;
        int64_t tb, te;
        int it = 0;
        gu_range(s_start, s_nact, F / 16, cta, ncta, tb, te);
        if (!produce_phase<FmtG, MODE_GATEUP>(b.gu, ring, s_act, tb * 16, te * 16, it, lane))
            return;
        // down: this CTA's (token, row) units, one segment per token
        int64_t db, de;
        tile_range(static_cast<int64_t>(T) * H, cta, ncta, db, de);
        for (int64_t t = db / H; db < de; ++t) {
            const int64_t le = de < (t + 1) * H ? de : (t + 1) * H;
            if (!produce_phase<FmtD, MODE_DOWN>(b.dn, ring, s_ridx + t * K, db - t * H,
                                                le - t * H, it, lane))
                return;
            db = le;
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    pdl_wait();
    pdl_trigger();
    if (tid == 0 && !sync_open(b.sync, b.err)) s_abort = 1;
    const bool arrive = tid == 0 && arrives(b.err);
    const int H4 = H / 4;
    const float4* x4 = reinterpret_cast<const float4*>(b.x);
    if (b.norm_w) {
        // ffn_norm scale of each token: one warp per token
        for (int t = warp; t < T; t += NCW) {
            float ss = 0.f;
            for (int i = lane; i < H4; i += 32) {
                const float4 hv = __ldcg(x4 + static_cast<int64_t>(t) * H4 + i);
                ss = fmaf(hv.x, hv.x, ss);
                ss = fmaf(hv.y, hv.y, ss);
                ss = fmaf(hv.z, hv.z, ss);
                ss = fmaf(hv.w, hv.w, ss);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) s_inv[t] = 1.0f / sqrtf(ss / static_cast<float>(H) + b.eps);
        }
        named_bar(1, NC);
    }
    // x tables of every token for the gate/up phase; with H a multiple of
    // 512 the same pass forms the logits of this CTA's first expert
    const bool rmerge = (H % 512) == 0 && cta < E;
    build_xprime<FmtG, 2>(b.x, T * (H / 256), T * (H / 16), xq, xs, tid, NC, b.err, b.norm_w, 1.f,
                          b.norm_w ? s_inv : nullptr, H / 16,
                          rmerge ? b.router + static_cast<int64_t>(cta) * H : nullptr, rpart);
    if (rmerge) {
        named_bar(1, NC);
        if (tid < T) {
            float sum = 0.f;
            for (int j = 0; j < H / 512; ++j) sum += rpart[tid * (H / 512) + j];
            b.logits[static_cast<int64_t>(tid) * E + cta] = sum;
        }
    }
    // logits of this CTA's (other) experts for every token
    {
        const float4* n4 = reinterpret_cast<const float4*>(b.norm_w);
        for (int e = rmerge ? cta + ncta : cta; e < E; e += ncta) {
            const float4* r4 = reinterpret_cast<const float4*>(b.router + static_cast<int64_t>(e) * H);
            float acc[TB_MAX];
#pragma unroll
            for (int t = 0; t < TB_MAX; ++t) acc[t] = 0.f;
            for (int j = tid; j < H4; j += NC) {
                const float4 w = __ldg(r4 + j);
                const float4 nv = n4 ? __ldg(n4 + j) : make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
                for (int t = 0; t < TB_MAX; ++t) {
                    if (t < T) {
                        float4 xv = __ldcg(x4 + static_cast<int64_t>(t) * H4 + j);
                        if (n4) {
                            const float iv = s_inv[t];
                            xv.x *= iv * nv.x;
                            xv.y *= iv * nv.y;
                            xv.z *= iv * nv.z;
                            xv.w *= iv * nv.w;
                        }
                        acc[t] = fmaf(w.x, xv.x, acc[t]);
                        acc[t] = fmaf(w.y, xv.y, acc[t]);
                        acc[t] = fmaf(w.z, xv.z, acc[t]);
                        acc[t] = fmaf(w.w, xv.w, acc[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < TB_MAX; ++t) {
                if (t < T) {
                    float a = acc[t];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                    if (lane == 0) red[t * NCW + warp] = a;
                }
            }
            named_bar(1, NC);
            if (tid < T) {
                float sum = 0.f;
                for (int k = 0; k < NCW; ++k) sum += red[tid * NCW + k];
                b.logits[static_cast<int64_t>(tid) * E + e] = sum;
            }
            named_bar(1, NC);
        }
    }
    named_bar(1, NC);
    if (tid == 0 && !s_abort && !grid_barrier(b.sync, 1, b.err, arrive)) s_abort = 1;
    named_bar(1, NC);
    if (s_abort) {
        if (tid == 0) sync_invalidate(b.sync);
        named_bar_arrive(2, NTHREADS);  // release the producer, which then returns
        return;
    }
    // routing: one warp per token
    for (int t = warp; t < T; t += NCW)
        route_warp(b.logits + static_cast<int64_t>(t) * E, E, K, lane, b.gu.renorm,
                   s_ridx + t * K, s_rw + t * K, b.err);
    for (int e = tid; e < E; e += NC) s_mask[e] = 0u;
    named_bar(1, NC);
    if (cta == 0) {
        for (int p = tid; p < T * K; p += NC) {
            if (b.topk_idx_out) b.topk_idx_out[p] = s_ridx[p];
            if (b.topk_w_out) b.topk_w_out[p] = s_rw[p];
        }
    }
    for (int p = tid; p < T * K; p += NC) atomicOr(&s_mask[s_ridx[p]], 1u << (p / K));
    named_bar(1, NC);
    if (warp == 0) {
        // active experts in ascending order and their first pair: warp scan
        // over lanes holding 8 experts each
        int na = 0, np = 0;
        for (int j = 0; j < 8; ++j) {
            const int e = lane * 8 + j;
            if (e < E && s_mask[e]) {
                ++na;
                np += __popc(s_mask[e]);
            }
        }
        int ia = na, ip = np;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ya = __shfl_up_sync(0xffffffffu, ia, o);
            const int yp = __shfl_up_sync(0xffffffffu, ip, o);
            if (lane >= o) {
                ia += ya;
                ip += yp;
            }
        }
        int a = ia - na, pbase = ip - np;
        for (int j = 0; j < 8; ++j) {
            const int e = lane * 8 + j;
            if (e < E && s_mask[e]) {
                s_act[a] = e;
                s_slot[e] = a;
                s_start[a] = pbase;
                pbase += __popc(s_mask[e]);
                ++a;
            }
        }
        if (lane == 31) {
            s_start[ia] = ip;
            s_nact = ia;
        }
    }
    named_bar(1, NC);
    for (int p = tid; p < T * K; p += NC) {
        const int t = p / K, e = s_ridx[p];
        const int pos = s_start[s_slot[e]] + __popc(s_mask[e] & ((1u << t) - 1u));
        s_ptok[pos] = t;
        s_pw[pos] = s_rw[p];
        s_porig[pos] = p;
    }
    named_bar(1, NC);
    named_bar_arrive(2, NTHREADS);  // the producer may stream the active experts

    PairLists pl;
    pl.act_e = s_act;
    pl.start = s_start;
    pl.tok = s_ptok;
    pl.w = s_pw;
    pl.orig = s_porig;
    const int nact = s_nact;
    int it = 0;
    int64_t tb, te;
    gu_range(s_start, nact, F / 16, cta, ncta, tb, te);
    bool good = consume_batch_gateup<FmtG>(b.gu, ring, pl, xq, xs, part, T, b.act, tb * 16,
                                           te * 16, it, tid);
    // every CTA's activations must be complete before any CTA reads them
    named_bar(1, NC);
    if (tid == 0 && good && !grid_barrier(b.sync, 2u, b.err, arrive)) s_abort = 1;
    named_bar(1, NC);
    if (!good || s_abort) {
        if (tid == 0) sync_invalidate(b.sync);
        return;
    }
    // down, token by token: the x table of the token's k activation rows,
    // then its rows of this CTA through the batch-1 down consumer
    int64_t db, de;
    tile_range(static_cast<int64_t>(T) * H, cta, ncta, db, de);
    for (int64_t t = db / H; good && db < de; ++t) {
        const int64_t le = de < (t + 1) * H ? de : (t + 1) * H;
        build_xprime<FmtD, 1>(b.act + t * K * F, K * (F / 256), K * (F / 16), xq, xs, tid, NC,
                              b.err);
        named_bar(1, NC);
        StreamParams pd = b.dn;
        pd.out = b.residual + t * H;
        good = consume_phase<FmtD, MODE_DOWN>(pd, ring, s_ridx + t * K, s_rw + t * K, xq, xs,
                                              part, db - t * H, le - t * H, it, tid);
        db = le;
    }
    if (tid == 0) {
        if (good)
            sync_close(b.sync);
        else
            sync_invalidate(b.sync);
    }
}

// Host side (batch.cu).
// Largest token count per batched launch for these formats and sizes (0 if
// the batched kernel does not apply: tiles too large for shared memory).
int batch_tokens_max(int gq, int dq, int H, int F, int K, int smem_optin);
// Launch the batched kernel for b.T tokens.  Returns 1 when launched, 0 if
// it does not apply, -1 on a CUDA error (*cerr).  *coop_pdl: whether
// cooperative launches may carry programmatic serialisation (-1 unknown).
int run_batch(int gq, int dq, BatchParams b, int sms, int smem_optin, int* coop_pdl,
              cudaStream_t st, cudaError_t* cerr);

}  // namespace qmoe
