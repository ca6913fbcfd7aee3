// stream.cuh — the streaming decode GEMV engine shared by qmv, ffn_swiglu and
// moe_ffn (decode).
//
// One CTA per SM (persistent over a contiguous range of output units).
// Warp 8 is the producer: it stages weight rows into a ring of shared-memory
// stages with 1-D bulk TMA copies (cp.async.bulk, completion counted on an
// mbarrier).  Warps 0..7 are consumers.  A tile holds 8*R row slots; lane
// (g = lane/4, q = lane%4) owns slots rr*8 + g (rr < R) and quarter q of each
// 256-element group its warp is given: warp v takes groups v, v+8, ... of
// the chunk.  A lane reads its pre-scaled f32 activations of a group
// (formats.cuh) from shared memory word by word and applies each to its R
// rows.  Per-row partial sums are reduced by shuffles across the four
// quarters and through shared memory across warps, in a fixed order
// (deterministic).
//
// Weight operands are read-only constants: the producer starts streaming
// them before griddepcontrol.wait, so a launch overlaps the tail of the
// kernel before it.  x, outputs and routing data are touched only after the
// wait.
//
// The producer and consumer loops are device functions over a shared ring
// (produce_phase / consume_phase), so one kernel can run several phases
// back to back through the same stages (the fused FFN / MoE kernel).
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
#include "route.cuh"

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
    int64_t uq;          // units per CTA, rounded down (units / grid)
    int ur;              // CTAs that take one more unit (units % grid)
    int nb_seg;          // 256-element groups per k-segment (the last may be partial)
    int tail;            // Q8_0/Q4_0 only: 32-element blocks of a partial last group (0: none)
    int n_kseg;          // k-segments: 1, or top_k for the MoE down product
    int chunk_ks;        // whole k-segments per chunk (when n_sbc == 1)
    int chunk_sb;        // groups per k-segment per chunk
    int n_sbc;           // chunks per k-segment (1 => chunks hold whole k-segments)
    int n_chunk;         // chunks per tile
    int piece_stride;    // smem bytes per (row, k-segment) piece; runs: per k-segment
    int slot_stride;     // smem bytes per row slot; runs: the row bytes
    int runs;            // 1: chunks hold whole rows, copied as runs of consecutive rows
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
    int renorm;             // 1: weights renormalised over the k; 0: softmax over all E
    int32_t* topk_idx_out;  // nullable, written by CTA 0 of GATEUP
    float* topk_w_out;
    int moe;
    DevCtl* err;
};

template <int MODE> struct ModeGeom {
    static constexpr int R = (MODE == MODE_DOWN) ? 2 : 4;  // row slots per lane
    static constexpr int ROWS = 8 * R;                     // row slots per tile
    static constexpr int TU = (MODE == MODE_GATEUP) ? ROWS / 2 : ROWS;  // units per tile
    static constexpr int WK = NCW;                         // warps along K
};

// Bytes of one k-segment of a row: nb_seg groups, the last one short by the
// blocks a partial group lacks (Q8_0/Q4_0 rows of 32-element blocks).
template <class Fmt>
__host__ __device__ inline int seg_bytes(const StreamParams& p) {
    return p.nb_seg * Fmt::SBB - (p.tail ? (8 - p.tail) * (Fmt::SBB / 8) : 0);
}

// The x table of one 256-element group: the 64 pre-scaled activations x' of
// each quarter lane (float4 [16][4]), and beside it in the xs region 16 sums
// of x (one per 16 elements) then the 8 block de-scales 2^(21 + E_b).
constexpr int XQ_GROUP_BYTES = 1024;
constexpr int XS_GROUP_FLOATS = 24;
constexpr int XS_GROUP_BYTES = 4 * XS_GROUP_FLOATS;

// Shared-memory carve-up (dynamic): [barriers][topk][part][xs][xq][stages]
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
    L.off_xs = o;    o += XS_GROUP_BYTES * p.nb_seg * p.n_kseg;
    o = align_up(o, 128);
    L.off_xq = o;    o += XQ_GROUP_BYTES * p.nb_seg * p.n_kseg;
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
// exp(l_s - l_max) / sum over the selected k of exp(l_t - l_max); with
// renorm = 0 the sum runs over all E experts instead (the softmax
// probability itself).  Experts are ranked on the total order of
// route.cuh, so every one of the k slots is written whatever the logits
// hold; when the top logit is not finite the route is experts 0..k-1 with
// NaN weights (route.cuh).
// Threads [0, nthr) of the CTA call it together; they synchronise on named
// barrier `bar` (0: the whole CTA, nthr == blockDim.x).  k <= 32.
__device__ __forceinline__ void group_sync(int bar, int nthr) {
    if (bar == 0)
        __syncthreads();
    else
        named_bar(bar, nthr);
}

__device__ inline void route_topk(const float* __restrict__ logits, int E, int k, uint32_t* s_key,
                                  int32_t* s_idx, float* s_w, int tid, int nthr, int bar,
                                  int renorm, DevCtl* err) {
    for (int e = tid; e < E; e += nthr) s_key[e] = route_key(__ldcg(logits + e));
    if (tid < k) s_idx[tid] = -1;
    group_sync(bar, nthr);
    // two threads per expert: each counts the experts ranked before it over half of E
    for (int base = 0; base < E; base += nthr / 2) {
        const int e = base + tid / 2, half = tid & 1;
        int rank = 0;
        if (e < E) {
            const uint32_t v = s_key[e];
            const int u0 = half ? E / 2 : 0, u1 = half ? E : E / 2;
            int u = u0;
            if ((E & 7) == 0) {  // both halves are whole uint4s
                const uint4* k4 = reinterpret_cast<const uint4*>(s_key);
#pragma unroll 4
                for (; u < u1; u += 4) {
                    const uint4 w = k4[u >> 2];
                    rank += route_before(w.x, u, v, e);
                    rank += route_before(w.y, u + 1, v, e);
                    rank += route_before(w.z, u + 2, v, e);
                    rank += route_before(w.w, u + 3, v, e);
                }
            }
            for (; u < u1; ++u) rank += route_before(s_key[u], u, v, e);
        }
        rank += __shfl_xor_sync(0xffffffffu, rank, 1);
        if (e < E && half == 0 && rank < k) s_idx[rank] = e;
    }
    group_sync(bar, nthr);
    if (tid < 32) {
        bool bad = false;
        int e = tid < k ? route_clamp(s_idx[tid], E, &bad) : 0;
        const float l = tid < k ? route_key_value(s_key[e]) : 0.f;
        const float lmax = __shfl_sync(0xffffffffu, l, 0);
        const float pr = tid < k ? expf(l - lmax) : 0.f;
        float z = pr;
        if (!renorm) {
            z = 0.f;
            for (int u = tid; u < E; u += 32) z += expf(route_key_value(s_key[u]) - lmax);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        float w = pr / z;
        if (route_degenerate(lmax)) {
            e = tid;
            w = __int_as_float(0x7FC00000);
        }
        if (tid < k) {
            s_idx[tid] = e;
            s_w[tid] = w;
        }
        if (__any_sync(0xffffffffu, bad) && tid == 0) record_error(err, DEV_ROUTE_RANGE);
    }
    group_sync(bar, nthr);
}

// ffn_norm's scale 1 / sqrt(mean(h^2) + eps) over h[0..n), computed by
// threads [0, nthr) of the CTA (named barrier `bar`; red: NCW floats of
// shared scratch).  Every participating thread gets the value.
__device__ inline float rms_inverse(const float* __restrict__ h, int n, float eps, float* red,
                                    int tid, int nthr, int bar) {
    const float4* h4 = reinterpret_cast<const float4*>(h);
    float ss = 0.f;
    for (int i = tid; i < n / 4; i += nthr) {
        const float4 v = __ldcg(h4 + i);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    group_sync(bar, nthr);
    float tot = 0.f;
    for (int k = 0; k < nthr / 32; ++k) tot += red[k];
    group_sync(bar, nthr);  // red may be reused after this
    return 1.0f / sqrtf(tot / static_cast<float>(n) + eps);
}

template <class Fmt, int UNR = 4>
__device__ inline void build_xprime(const float* __restrict__ x, int ngroups, int n16_valid,
                                    float* xq, float* xs, int tid, int nthreads, DevCtl* err,
                                    const float* __restrict__ nw = nullptr, float inv = 1.f,
                                    const float* inv_tok = nullptr, int tok_n16 = 0,
                                    const float* __restrict__ rrow = nullptr,
                                    float* rpart = nullptr) {
    // The x table (see formats.cuh): x' = x * 2^(128 - E_b - pos) in the
    // lanes' register order, with E_b the exponent of the largest |x| of the
    // 32-element block (clamped to [1, 106]; 1 for a block holding a
    // non-finite value), the block's de-scale 2^(21 + E_b), and the f32 sum
    // of x per 16 elements.  Multiplying by a power of two is exact: x' holds
    // every bit of x.  A thread takes 16-element chunks of x: it loads the
    // chunk's four aligned float4s (all loads in flight before any use, so
    // the table costs one L2 round trip), takes the block maximum with its
    // neighbour (the chunk pair 2m, 2m+1 is block m), and scatters each
    // granule of four to its slot (the formats' element orders keep every
    // slot four consecutive elements), each element scaled for its field's
    // bit position.  A block whose largest |x| is 2^106 or more is outside
    // the range and is flagged (DEV_X_RANGE).
    // Only the first n16_valid chunks of x exist (a row whose last group is
    // partial); the table holds zeros past them.
    // With nw, the table is of the normed input x_j * inv * nw_j (ffn_norm).
    // With inv_tok, x holds several tokens of tok_n16 chunks each, token t
    // normed with inv_tok[t] (nw applies per token).  UNR chunks per thread
    // are in flight at once.
    // With rrow (one f32 router row), the same pass forms the router dot
    // product of every token: the row's chunk is loaded beside the token's,
    // and each warp's 32 chunks (one token: tok_n16 and nthreads multiples
    // of 32) leave one partial in rpart[t * tok_n16 / 32 + chunk / 32], to be
    // summed in that order.
    const int n16 = ngroups * 16;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const float4* r4 = reinterpret_cast<const float4*>(rrow);
    float4* xq4 = reinterpret_cast<float4*>(xq);
    bool range = false;
    // warps step together (the shuffles below need every lane of the warp,
    // also those whose chunks are past the end): nthreads is a multiple of 32
    for (int wbase = tid & ~31; wbase < n16; wbase += nthreads * UNR) {
        const int base = wbase + (tid & 31);
        float4 v[UNR][4];
        float4 rv[UNR][4];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            if (wbase + u * nthreads >= n16) break;  // warp-uniform: no lane of the warp has work
            const int c = base + u * nthreads;
            if (c < n16_valid) {
#pragma unroll
                for (int k = 0; k < 4; ++k) v[u][k] = __ldcg(x4 + 4 * c + k);
                int cw = c;
                float iv = inv;
                if (inv_tok || rrow) {
                    const int tk = c / tok_n16;
                    cw = c - tk * tok_n16;
                    if (inv_tok) iv = inv_tok[tk];
                }
                if (rrow) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) rv[u][k] = __ldg(r4 + 4 * cw + k);
                }
                if (nw) {
                    const float4* w4 = reinterpret_cast<const float4*>(nw);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float4 wv = __ldg(w4 + 4 * cw + k);
                        v[u][k].x *= iv * wv.x;
                        v[u][k].y *= iv * wv.y;
                        v[u][k].z *= iv * wv.z;
                        v[u][k].w *= iv * wv.w;
                    }
                }
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) v[u][k] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            if (wbase + u * nthreads >= n16) break;  // warp-uniform, as above
            const int c = base + u * nthreads;
            if (rrow && c - (c & 31) < n16) {  // whole warps: all lanes valid
                float d = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    d = fmaf(rv[u][k].x, v[u][k].x, d);
                    d = fmaf(rv[u][k].y, v[u][k].y, d);
                    d = fmaf(rv[u][k].z, v[u][k].z, d);
                    d = fmaf(rv[u][k].w, v[u][k].w, d);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                if ((c & 31) == 0) rpart[c >> 5] = d;
            }
            // block maximum over this chunk and its neighbour (lane ^ 1)
            float mx = 0.f;
            bool bad = false;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float a0 = fabsf(v[u][k].x), a1 = fabsf(v[u][k].y), a2 = fabsf(v[u][k].z),
                            a3 = fabsf(v[u][k].w);
                mx = fmaxf(mx, fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)));
                bad = bad || !(a0 <= 3.402823466e38f) || !(a1 <= 3.402823466e38f) ||
                      !(a2 <= 3.402823466e38f) || !(a3 <= 3.402823466e38f);
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            bad = __shfl_xor_sync(0xffffffffu, static_cast<int>(bad), 1) != 0 || bad;
            if (c < n16) {
                // mx < 2^E for E = its biased exponent - 126
                int E = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu) - 126;
                if (bad) E = XBLK_EMIN;
                if (E < XBLK_EMIN) E = XBLK_EMIN;
                if (E > XBLK_EMAX) {
                    E = XBLK_EMAX;
                    range = true;
                }
                float s = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) s += (v[u][k].x + v[u][k].y) + (v[u][k].z + v[u][k].w);
                const int g = c >> 4;
                xs[g * XS_GROUP_FLOATS + (c & 15)] = s;
                if ((c & 1) == 0) xs[g * XS_GROUP_FLOATS + 16 + ((c & 15) >> 1)] = pow2f(21 + E);
                // 2^(128 - E - pos) for the granule's four positions, which
                // are those of element index i % 8 (formats.cuh): {0, 8, 16,
                // 0} for i % 8 < 4, and {4, 12, 20, 0} above it where POS8
                const float base = pow2f(128 - E);
                const float m0 = base, m1 = base * 0x1p-8f, m2 = base * 0x1p-16f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int slot = Fmt::xslot(4 * (c & 15) + k);
                    const bool odd = Fmt::POS8 && ((slot >> 2) & 1);
                    float4 o;
                    o.x = v[u][k].x * (odd ? base * 0x1p-4f : m0);
                    o.y = v[u][k].y * (odd ? base * 0x1p-12f : m1);
                    o.z = v[u][k].z * (odd ? base * 0x1p-20f : m2);
                    o.w = v[u][k].w * base;
                    xq4[g * 64 + slot] = o;
                }
            }
        }
    }
    if (range) record_error(err, DEV_X_RANGE);
}

// Address of the bytes of (row slot r, k-segment ks) for the tile starting
// at unit u0; nullptr if the row's unit is outside [.., uend).  For the MoE
// gate/up product s0 = u0 / F, the routed slot of the tile's first unit
// (a tile spans fewer than F units, so it crosses at most one slot border).
template <int MODE>
__device__ __forceinline__ const uint8_t* row_addr(const StreamParams& p, const int32_t* s_idx,
                                                   int64_t u0, int s0, int64_t uend, int r,
                                                   int ks) {
    const int g = r & 7, rr = r >> 3;
    if (MODE == MODE_GATEUP) {
        const bool up = rr >= 2;
        const int64_t u = u0 + (rr & 1) * 8 + g;
        if (u >= uend) return nullptr;
        const uint8_t* base = up ? p.W1 : p.W0;
        const int64_t rb = up ? p.rb1 : p.rb0, es = up ? p.es1 : p.es0;
        if (p.moe) {
            int64_t jj = u - static_cast<int64_t>(s0) * p.F;
            int s = s0;
            if (jj >= p.F) {
                jj -= p.F;
                ++s;
            }
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

// The units [beg, end) of CTA `cta`: an even split, the first ur CTAs one
// unit larger (quotient and remainder come from the host).
__device__ __forceinline__ void unit_range(const StreamParams& p, int cta, int64_t& beg,
                                           int64_t& end) {
    beg = p.uq * cta + (cta < p.ur ? cta : p.ur);
    end = beg + p.uq + (cta < p.ur ? 1 : 0);
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

// Runs: when a chunk holds whole rows (k-segments), the rows of a tile that
// are consecutive in memory move as one bulk copy.  Row slot r belongs to
// the run that starts at slot head(r) (run index i: gate 0/1, up 2/3 for the
// gate/up product, whose units may cross one expert border; 0 otherwise).
// In a k-segment's region of the stage a run starts at
// run_dst = align16(head * row_bytes) + 32 * i, and its rows follow at the
// global row stride, offset by the head row's 16-byte phase.  A bulk copy
// costs a fixed time in the copy engine whatever its size, so fewer, larger
// copies are what lets small rows (MoE experts) stream at the HBM rate.
struct RunSlot {
    int head, idx;
};

template <int MODE>
__device__ __forceinline__ RunSlot run_of(const StreamParams& p, int64_t u0, int s0, int r) {
    RunSlot rs;
    if (MODE == MODE_GATEUP) {
        const int half = r >> 4, j = r & 15;
        int jb = 16;
        if (p.moe) {
            const int64_t b = static_cast<int64_t>(s0 + 1) * p.F - u0;
            jb = b < 16 ? static_cast<int>(b) : 16;
        }
        const int second = j >= jb ? 1 : 0;
        rs.head = half * 16 + (second ? jb : 0);
        rs.idx = half * 2 + second;
    } else {
        rs.head = 0;
        rs.idx = 0;
    }
    return rs;
}

__device__ __forceinline__ int run_dst(const StreamParams& p, int head, int idx) {
    return ((head * p.slot_stride + 15) & ~15) + 32 * idx;
}

// Prefetch `bytes` (a multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// The stage ring: nstages stages of stage_bytes, a full barrier (one
// arrival + transaction bytes) and an empty barrier (NCW consumer warps)
// per stage.  Producer and consumers number chunks with one running count
// `it` across phases, so phases of different geometry can follow each other
// through the same ring.
struct Ring {
    uint8_t* stages;
    uint64_t* full;
    uint64_t* empty;
    int nstages, stage_bytes;
};

template <int MODE>
__device__ __forceinline__ int tile_slot(const StreamParams& p, int64_t u0) {
    return (MODE == MODE_GATEUP && p.moe) ? static_cast<int>(static_cast<uint32_t>(u0) /
                                                             static_cast<uint32_t>(p.F))
                                          : 0;
}

// The bulk copies of one chunk: runs, one copy per run of consecutive rows
// and k-segment (gate/up tiles: 4 runs); otherwise one copy per row and
// k-segment.  chunk_copies counts them, chunk_copy gives copy k (source,
// bytes, stage offset; 0 bytes if the copy is empty).
template <int MODE>
__device__ __forceinline__ int chunk_copies(const StreamParams& p, const ChunkDesc& cd) {
    using G = ModeGeom<MODE>;
    constexpr int NR = (MODE == MODE_GATEUP) ? 4 : 1;
    return p.runs ? NR * cd.nks : G::ROWS * cd.nks;
}

template <class Fmt, int MODE>
__device__ __forceinline__ uint32_t chunk_copy(const StreamParams& p, const int32_t* s_idx,
                                               int64_t u0, int s0, int64_t uend,
                                               const ChunkDesc& cd, int k, uintptr_t& src,
                                               int& dst) {
    using G = ModeGeom<MODE>;
    if (p.runs) {
        constexpr int NR = (MODE == MODE_GATEUP) ? 4 : 1;
        const int pk = k / NR, ri = k % NR;
        const int nrow = static_cast<int>(uend - u0 < G::TU ? uend - u0 : G::TU);
        int h = 0, e = nrow;  // rows [h, e) of this run
        if (MODE == MODE_GATEUP) {
            int jb = 16;
            if (p.moe) {
                const int64_t b = static_cast<int64_t>(s0 + 1) * p.F - u0;
                jb = b < 16 ? static_cast<int>(b) : 16;
            }
            const int lo = (ri & 1) ? jb : 0, hi = (ri & 1) ? 16 : jb;
            h = (ri >> 1) * 16 + lo;
            e = (ri >> 1) * 16 + (hi < nrow ? hi : nrow);
        }
        if (e <= h) return 0u;
        const uintptr_t a = reinterpret_cast<uintptr_t>(
            row_addr<MODE>(p, s_idx, u0, s0, uend, h, cd.ks0 + pk));
        src = a & ~uintptr_t(15);
        dst = pk * p.piece_stride + run_dst(p, h, ri);
        return static_cast<uint32_t>(
            ((a + static_cast<uintptr_t>(e - h) * p.slot_stride + 15) & ~uintptr_t(15)) - src);
    }
    const int r = k / cd.nks, pk = k % cd.nks;
    const uint8_t* a = row_addr<MODE>(p, s_idx, u0, s0, uend, r, cd.ks0 + pk);
    if (!a) return 0u;
    const uintptr_t sa = reinterpret_cast<uintptr_t>(a) + static_cast<uintptr_t>(cd.b0) * Fmt::SBB;
    // never past the row's end (a partial last group is shorter)
    const int seg = seg_bytes<Fmt>(p), want = cd.nbp * Fmt::SBB, left = seg - cd.b0 * Fmt::SBB;
    const uintptr_t n = static_cast<uintptr_t>(want < left ? want : left);
    src = sa & ~uintptr_t(15);
    dst = r * p.slot_stride + pk * p.piece_stride;
    return static_cast<uint32_t>(((sa + n + 15) & ~uintptr_t(15)) - src);
}

// After a wait of the producer gave up: wait (bounded) until the copies of
// the last chunks it issued, numbers [it - nstages, it), have landed, so the
// CTA never exits with a bulk copy still writing its shared memory.
__device__ inline void ring_drain(const Ring& ring, int it, DevCtl* err) {
    for (int j = it - ring.nstages; j < it; ++j)
        if (j >= 0)
            mbar_wait_bounded(&ring.full[j % ring.nstages], (j / ring.nstages) & 1, err,
                              DEV_TIMEOUT_FULL);
}

// Producer warp: stream every chunk of the units [ubeg, uend) into the ring.
// False if a wait for a free stage timed out (the error word is set; the
// copies already issued have landed).
template <class Fmt, int MODE>
__device__ bool produce_phase(const StreamParams& p, const Ring& ring, const int32_t* s_idx,
                              int64_t ubeg, int64_t uend, int& it, int lane) {
    using G = ModeGeom<MODE>;
    const uint64_t pol = policy_evict_first();
    const int ntiles = static_cast<int>((uend - ubeg + G::TU - 1) / G::TU);
    for (int t = 0; t < ntiles; ++t) {
        const int64_t u0 = ubeg + static_cast<int64_t>(G::TU) * t;
        const int s0 = tile_slot<MODE>(p, u0);
        for (int c = 0; c < p.n_chunk; ++c, ++it) {
            const int s = it % ring.nstages;
            const int round = it / ring.nstages;
            if (round > 0 &&
                !mbar_wait_bounded(&ring.empty[s], (round - 1) & 1, p.err, DEV_TIMEOUT_EMPTY)) {
                ring_drain(ring, it, p.err);
                return false;
            }
            const ChunkDesc cd = chunk_desc(p, c);
            const int ncopy = chunk_copies<MODE>(p, cd);
            uint32_t mine = 0;
            for (int k = lane; k < ncopy; k += 32) {
                uintptr_t src = 0;
                int dst = 0;
                mine += chunk_copy<Fmt, MODE>(p, s_idx, u0, s0, uend, cd, k, src, dst);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
            if (lane == 0) mbar_arrive_expect_tx(&ring.full[s], mine);
            __syncwarp();
            uint8_t* st = ring.stages + static_cast<size_t>(s) * ring.stage_bytes;
            for (int k = lane; k < ncopy; k += 32) {
                uintptr_t src = 0;
                int dst = 0;
                const uint32_t n = chunk_copy<Fmt, MODE>(p, s_idx, u0, s0, uend, cd, k, src, dst);
                if (n)
                    bulk_g2s(st + dst, reinterpret_cast<const void*>(src), n, &ring.full[s], pol);
            }
        }
    }
    return true;
}

// Consumer warps 0..NCW-1: reduce every tile of [ubeg, uend) and write the
// outputs (QMV: y = W.x; GATEUP: a = w * silu(g) * u; DOWN: out += D.a).
// xq / xs must already hold the phase's x table.  False (in every consumer
// thread alike) if a stage wait timed out: a warp whose wait expired skips
// the rest of its waits and arithmetic but still takes part in every named
// barrier, so no warp is left waiting, and no output of a tile is written
// unless every warp's data for it arrived.
template <class Fmt, int MODE>
__device__ bool consume_phase(const StreamParams& p, const Ring& ring, const int32_t* s_idx,
                              const float* s_w, const float* xq, const float* xs, float* part,
                              int64_t ubeg, int64_t uend, int& it, int tid) {
    using G = ModeGeom<MODE>;
    constexpr int R = G::R;
    const int v = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q = lane & 3;
    const float4* xq4 = reinterpret_cast<const float4*>(xq);
    const int ntiles = static_cast<int>((uend - ubeg + G::TU - 1) / G::TU);
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
        const int64_t u0 = ubeg + static_cast<int64_t>(G::TU) * t;
        const int s0 = tile_slot<MODE>(p, u0);
        float acc[R];
        // low 32 bits of each row's address (k-segment 0): only the 16-byte
        // phase is needed to find the row inside its staged slot
        // and the row's offset in a k-segment region of the stage; for runs,
        // the phase is the run head's and the offset run_dst + rows * stride
        uint32_t rowlo[R];
        int rowoff[R];
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            acc[rr] = 0.f;
            // a QMV slot past the CTA's last row reads slot 0 (the stage may
            // hold only the CTA's rows); its sum is never written
            const int r = (MODE == MODE_QMV && u0 + rr * 8 + g >= uend) ? 0 : rr * 8 + g;
            int h = r;
            if (p.runs) {
                const RunSlot rs = run_of<MODE>(p, u0, s0, r);
                h = rs.head;
                rowoff[rr] = run_dst(p, rs.head, rs.idx) + (r - rs.head) * p.slot_stride;
            } else {
                rowoff[rr] = r * p.slot_stride;
            }
            const uint8_t* a = row_addr<MODE>(p, s_idx, u0, s0, uend, h, 0);
            rowlo[rr] = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(a));
            if (MODE == MODE_DOWN && p.moe && a)  // k-segment 0's expert offset removed
                rowlo[rr] -= static_cast<uint32_t>(s_idx[0]) * static_cast<uint32_t>(p.es0);
        }
        for (int c = 0; c < p.n_chunk; ++c, ++it) {
            const int s = it % ring.nstages;
            const int round = it / ring.nstages;
            if (ok && !mbar_wait_bounded(&ring.full[s], round & 1, p.err, DEV_TIMEOUT_FULL))
                ok = false;
            ok = __all_sync(0xffffffffu, ok);  // one decision per warp
            const ChunkDesc cd = chunk_desc(p, c);
            const uint8_t* st = ring.stages + static_cast<size_t>(s) * ring.stage_bytes;
            const int ntot = ok ? cd.nks * cd.nbp : 0;
            const uint32_t b0off = static_cast<uint32_t>(cd.b0) * Fmt::SBB;
            for (int tt = v; tt < ntot; tt += G::WK) {
                const int pk = tt / cd.nbp, bb = tt - pk * cd.nbp;
                const int ks = cd.ks0 + pk, b = cd.b0 + bb;
                const int gidx = ks * p.nb_seg + b;
                const float* xsg = xs + gidx * XS_GROUP_FLOATS;
                const int nblk = (p.tail && b == p.nb_seg - 1) ? p.tail : 8;
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
                    sbp[rr] = st + rowoff[rr] + pk * p.piece_stride + delta + bb * Fmt::SBB;
                }
                Fmt::template dotR<R>(sbp, q, xq4 + gidx * 64 + q, xsg, xsg + 16, nblk, acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ring.empty[s]);
        }
        float* pt = part + (t & 1) * NCW * MAX_ROWS;
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            float a = acc[rr];
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            if (q == 0) pt[v * MAX_ROWS + rr * 8 + g] = a;
        }
        ok = named_bar_and(1, NCW * 32, ok);
        // cross-warp sums as shuffle trees: eight consecutive lanes hold the
        // eight warps' partials of one row
        const int k8 = tid & 7;
        if (MODE == MODE_GATEUP) {
            // lanes 0-7 of a 16-lane group: gate row of unit uu; 8-15: its up row
            const int uu = tid >> 4, up = (tid >> 3) & 1;
            float vs = pt[k8 * MAX_ROWS + up * G::TU + uu];
            vs += __shfl_xor_sync(0xffffffffu, vs, 1);
            vs += __shfl_xor_sync(0xffffffffu, vs, 2);
            vs += __shfl_xor_sync(0xffffffffu, vs, 4);
            const float us = __shfl_down_sync(0xffffffffu, vs, 8);
            const int64_t u = u0 + uu;
            if (ok && up == 0 && k8 == 0 && u < uend) {
                float w = 1.0f;
                if (p.moe) {
                    const int sl = s0 + (u - static_cast<int64_t>(s0) * p.F >= p.F ? 1 : 0);
                    w = s_w[sl];
                }
                p.out[u] = w * ((vs / (1.0f + expf(-vs))) * us);
            }
        } else {
            const int r = tid >> 3;
            float vs = r < G::ROWS ? pt[k8 * MAX_ROWS + r] : 0.f;
            vs += __shfl_xor_sync(0xffffffffu, vs, 1);
            vs += __shfl_xor_sync(0xffffffffu, vs, 2);
            vs += __shfl_xor_sync(0xffffffffu, vs, 4);
            const int64_t u = u0 + r;
            if (ok && k8 == 0 && r < G::TU && u < uend) {
                if (MODE == MODE_QMV)
                    p.out[u] = vs;
                else
                    p.out[u] += vs;
            }
        }
    }
    return ok;
}

// Producer warp + eight consumer warps over a ring of stages: the phases of
// the fused and batched kernels, MoE and dense GATEUP/DOWN launches, and QMV
// when a CTA's rows span several stages (large GEMVs).  One CTA per SM.
// (QMV rows that fit one stage run qmv_tile_kernel below.)
template <class Fmt, int MODE>
__global__ void __launch_bounds__(NTHREADS, 1) stream_gemv_kernel(const StreamParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const SmemLayout L = smem_layout(p);
    Ring ring;
    ring.full = reinterpret_cast<uint64_t*>(smem + L.off_full);
    ring.empty = reinterpret_cast<uint64_t*>(smem + L.off_empty);
    ring.stages = smem + L.off_stage;
    ring.nstages = p.nstages;
    ring.stage_bytes = p.stage_bytes;
    int32_t* s_idx = reinterpret_cast<int32_t*>(smem + L.off_tidx);
    float* s_w = reinterpret_cast<float*>(smem + L.off_tw);
    uint32_t* s_key = reinterpret_cast<uint32_t*>(smem + L.off_logit);
    float* part = reinterpret_cast<float*>(smem + L.off_part);
    float* xs = reinterpret_cast<float*>(smem + L.off_xs);
    float* xq = reinterpret_cast<float*>(smem + L.off_xq);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int64_t ubeg, uend;
    unit_range(p, static_cast<int>(blockIdx.x), ubeg, uend);

    // The producer's lane 0 initialises the stage barriers.  Without routing
    // the producer starts streaming at once and only arrives on named
    // barrier 2; the consumers sync on it before their first stage wait.
    // With routing every thread takes part in route_topk, whose
    // __syncthreads also publishes the barriers.
    if (tid == NCW * 32) {
        for (int s = 0; s < p.nstages; ++s) {
            mbar_init(&ring.full[s], 1);
            mbar_init(&ring.empty[s], NCW);
        }
        fence_barrier_init();
    }
    // Routing decides which expert rows are streamed.  The logits come from
    // the router kernel, one launch back (gate/up) or two (down); the wait
    // covers both, since the launch in between waited for the router before
    // it could complete.
    if (p.moe) {
        pdl_wait();
        pdl_trigger();
        route_topk(p.logits, p.E, p.topk, s_key, s_idx, s_w, tid, NTHREADS, 0, p.renorm, p.err);
        if (MODE == MODE_GATEUP && blockIdx.x == 0 && tid < p.topk) {
            if (p.topk_idx_out) p.topk_idx_out[tid] = s_idx[tid];
            if (p.topk_w_out) p.topk_w_out[tid] = s_w[tid];
        }
    } else if (warp == NCW) {
        __syncwarp();
        named_bar_arrive(2, NTHREADS);
    }

    int it = 0;
    if (warp == NCW) {
        produce_phase<Fmt, MODE>(p, ring, s_idx, ubeg, uend, it, lane);
        return;
    }
    if (!p.moe) {  // the MoE grids waited above
        pdl_wait();
        pdl_trigger();
    }
    build_xprime<Fmt>(p.x, p.nb_seg * p.n_kseg,
                      p.tail ? (p.nb_seg - 1) * 16 + 2 * p.tail : p.nb_seg * p.n_kseg * 16, xq, xs,
                      tid, NCW * 32, p.err);
    named_bar(1, NCW * 32);
    if (!p.moe) named_bar(2, NTHREADS);  // the stage barriers are initialised
    consume_phase<Fmt, MODE>(p, ring, s_idx, s_w, xq, xs, part, ubeg, uend, it, tid);
}

// QMV with one tile per CTA (the plan's single stage holds all of the CTA's
// rows): eight consumer warps, the first of which issues the tile's copies
// before the dependency wait, so no warp is only a producer.  At 256
// threads and at most 128 registers (every format's decode fits without
// spilling), any two of these kernels fit one SM's register file, so the
// next launch's CTAs - the same GEMV or another format's - stream their
// weights beside this launch's wherever shared memory allows.  Measured on
// the mixed-format sweep: 33.2 -> 30.9 us per step; a Q8_0 instance given
// its own 149 registers blocks that pairing and costs 8 us per step.
template <class Fmt>
__global__ void __launch_bounds__(NCW * 32, 2) qmv_tile_kernel(const StreamParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const SmemLayout L = smem_layout(p);
    Ring ring;
    ring.full = reinterpret_cast<uint64_t*>(smem + L.off_full);
    ring.empty = reinterpret_cast<uint64_t*>(smem + L.off_empty);
    ring.stages = smem + L.off_stage;
    ring.nstages = 1;
    ring.stage_bytes = p.stage_bytes;
    int32_t* s_idx = reinterpret_cast<int32_t*>(smem + L.off_tidx);
    float* s_w = reinterpret_cast<float*>(smem + L.off_tw);
    float* part = reinterpret_cast<float*>(smem + L.off_part);
    float* xs = reinterpret_cast<float*>(smem + L.off_xs);
    float* xq = reinterpret_cast<float*>(smem + L.off_xq);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int64_t ubeg, uend;
    unit_range(p, static_cast<int>(blockIdx.x), ubeg, uend);
    if (tid == 0) {
        mbar_init(&ring.full[0], 1);
        mbar_init(&ring.empty[0], NCW);
        fence_barrier_init();
    }
    __syncthreads();
    if (warp == 0) {
        int itp = 0;
        produce_phase<Fmt, MODE_QMV>(p, ring, s_idx, ubeg, uend, itp, lane);
    }
    pdl_wait();
    pdl_trigger();
    build_xprime<Fmt>(p.x, p.nb_seg,
                      p.tail ? (p.nb_seg - 1) * 16 + 2 * p.tail : p.nb_seg * 16, xq, xs, tid,
                      NCW * 32, p.err);
    named_bar(1, NCW * 32);
    int it = 0;
    consume_phase<Fmt, MODE_QMV>(p, ring, s_idx, s_w, xq, xs, part, ubeg, uend, it, tid);
}

// ------------------------------------------------------------ host planning
// Chunk geometry of a streamed phase for a stage budget (bytes): how rows
// are cut into chunks, the slot strides and the bytes one stage needs.
// A stage holds `rows` row slots: all G::ROWS of a tile, or (QMV, when every
// CTA has a single tile) just the rows one CTA owns — its consumers then
// read slot 0 for the tile's unused slots.  False if not even one group per
// row fits.
template <class Fmt, int MODE>
inline bool plan_chunks(StreamParams& p, int budget, int rows = ModeGeom<MODE>::ROWS) {
    using G = ModeGeom<MODE>;
    if (MODE != MODE_QMV || rows > G::ROWS || rows < 1) rows = G::ROWS;
    if (budget < rows * (Fmt::SBB + 31)) return false;
    const int seg_full = seg_bytes<Fmt>(p);
    // a partial last group is read as a whole one: the bytes past the row
    // end are stale shared memory, masked off by the consumer
    const int tail_slack = p.tail ? Fmt::SBB : 0;
    // Whole k-segments fit: runs of consecutive rows, one bulk copy each.
    // A k-segment region holds the tile's rows at their global stride plus
    // slack for up to four run starts (32 bytes apart), a 16-byte phase and
    // the 14 bytes a Q6_K lane may read past its super-block.
    // Rows of 2 KB and more stream at the full rate as separate copies, so
    // formats whose loads would conflict at the global stride keep padded
    // per-row slots for them.
    const int run_piece = align_up(rows * seg_full, 16) + 144 + tail_slack;
    if (run_piece <= budget && (Fmt::RUNS_OK || seg_full < 2048)) {
        p.runs = 1;
        p.n_sbc = 1;
        p.chunk_ks = budget / run_piece < p.n_kseg ? budget / run_piece : p.n_kseg;
        p.chunk_sb = p.nb_seg;
        p.piece_stride = run_piece;
        p.slot_stride = seg_full;
        p.stage_bytes = p.chunk_ks * run_piece;
        p.n_chunk = (p.n_kseg + p.chunk_ks - 1) / p.chunk_ks;
        return true;
    }
    p.runs = 0;
    const int piece_full = align_up(seg_full + 15, 16);
    int nbp_max;
    if (rows * p.n_kseg * piece_full <= budget) {
        p.n_sbc = 1;
        p.chunk_ks = p.n_kseg;
        p.chunk_sb = p.nb_seg;
        nbp_max = p.nb_seg;
    } else if (rows * piece_full <= budget) {
        p.n_sbc = 1;
        p.chunk_ks = budget / (rows * piece_full);
        p.chunk_sb = p.nb_seg;
        nbp_max = p.nb_seg;
    } else {
        p.chunk_ks = 1;
        int csb = (budget / rows - 31) / Fmt::SBB;
        if (csb >= G::WK) csb -= csb % G::WK;
        if (csb < 1) csb = 1;
        p.chunk_sb = csb;
        p.n_sbc = (p.nb_seg + csb - 1) / csb;
        nbp_max = csb;
    }
    p.piece_stride = align_up(nbp_max * Fmt::SBB + 15, 16);
    p.slot_stride = p.chunk_ks * p.piece_stride;
    if (Fmt::SLOT_REM128 >= 0)
        p.slot_stride += (Fmt::SLOT_REM128 - p.slot_stride % 128 + 128) % 128;
    else if (p.slot_stride % 32 == 0)
        p.slot_stride += 16;  // alternate rows across bank halves
    p.stage_bytes = rows * p.slot_stride;
    p.n_chunk = (p.n_sbc == 1) ? (p.n_kseg + p.chunk_ks - 1) / p.chunk_ks : p.n_kseg * p.n_sbc;
    return true;
}

}  // namespace qmoe
