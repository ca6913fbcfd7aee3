// formats.cuh — per-format decode-and-dot of one lane's quarter of a
// 256-element group, for the GGUF block layouts given by the CUDA kernel
// sources on "ferrox-cuda 0.14.0 — src/gpu.rs" (Q8_0_MATVEC_KERNEL_SRC,
// Q4_0_MATVEC_KERNEL_SRC, Q4_K_MATVEC_KERNEL_SRC with ferrox_q4_k_scale_min,
// Q5_K_MATVEC_KERNEL_SRC, Q6_K_MATVEC_KERNEL_SRC).
//
// Arithmetic scheme (ours, not the pages'):
//   * The activations are held as 16-bit integers with one f32 scale per
//     32-element block: x_j ~ s_b * xi_j, s_b = max |x| over the block / 32767,
//     xi_j = round(x_j / s_b).  The rounding error of every x_j is at most
//     s_b / 2, 1/65534 of the block's largest |x|.
//   * The quants stay packed: masks and shifts leave four of them in the
//     bytes of a word, and dp2a (two 16-bit x times two bytes, summed into
//     32 bits) multiplies them with the x pairs.  A 32-bit integer sum per
//     (row, sub-block) is exact (|sum| < 2^26).
//   * Per sub-block the sum turns into f32 once and takes the block's scales:
//       sum (d*sc*q - dmin*m) x = d*sc*s_b*sum q xi - dmin*m*sum x
//     with the offsets and mins applied through sum x over each 16-element
//     group, computed once per call in f32 from the unrounded x.
//
// A lane owns quarter q (0..3) of a 256-element group ("super-block"; for
// Q8_0/Q4_0, 8 consecutive 32-element blocks).  It processes 64 elements;
// element i (0..63) of its quarter is elem(q,i) of the group, and 32-bit
// register k (0..31) of its x block holds elements elem(q,2k) (low half) and
// elem(q,2k+1) (high half).  The x table is stored in shared memory as
// uint4 [group][i/8][q] (registers 4p..4p+3 of quarter q in uint4 p), so the
// four quarter-lanes read 64 contiguous bytes; a lane loads its 32 registers
// once (load_xq) and applies them to several rows (dotR).
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace qmoe {

enum QType : int { QT_F32 = 0, QT_Q8_0 = 1, QT_Q4_0 = 2, QT_Q4_K = 3, QT_Q5_K = 4, QT_Q6_K = 5 };

__device__ __forceinline__ float f16_bits_to_f32(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// c + (x pair in xp) . (bytes 0, 1 of w)  /  (bytes 2, 3 of w)
__device__ __forceinline__ int dp_lo(uint32_t xp, uint32_t w, int c) {
    return __dp2a_lo(static_cast<int>(xp), static_cast<int>(w), c);
}
__device__ __forceinline__ int dp_hi(uint32_t xp, uint32_t w, int c) {
    return __dp2a_hi(static_cast<int>(xp), static_cast<int>(w), c);
}

// The 32 x registers of quarter q of one group.
__device__ __forceinline__ void load_xq(const uint4* xq_group, int q, uint32_t (&x)[32]) {
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const uint4 v = xq_group[p * 4 + q];
        x[4 * p] = v.x;
        x[4 * p + 1] = v.y;
        x[4 * p + 2] = v.z;
        x[4 * p + 3] = v.w;
    }
}

// Read 4 consecutive 32-bit words starting at a 2-byte-aligned shared-memory
// address: aligned loads plus a funnel shift by 0 or 16 bits.
__device__ __forceinline__ void load4_u16al(const uint8_t* p, uint32_t (&w)[4]) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* base = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = static_cast<uint32_t>(a & 3u) * 8u;
    uint32_t r[5];
#pragma unroll
    for (int k = 0; k < 5; ++k) r[k] = base[k];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = __funnelshift_r(r[k], r[k + 1], sh);
}

// Every format provides
//   elem(q, i)  — the lane element order (64 elements of quarter q);
//   xslot(e4)   — its inverse on 4-element granules: the slot 4*i4 + q whose
//                 elements elem(q, 4*i4 .. 4*i4+3) are elements 4*e4 .. 4*e4+3
//                 of the group (each slot is four consecutive elements);
//   dotR<R>(sb[R], q, x, xs16, sx, acc[R]) — for R rows whose super-blocks
//   start at sb[r] (shared memory), adds each row's dot over the lane's
//   quarter to acc[r]; x: the lane's 32 x registers, xs16: sum x per 16
//   elements of the group, sx: the group's eight 32-element x scales.
//   Words of all R rows are loaded first and the element loop runs over words
//   with the rows innermost, so a lane carries several independent dp2a
//   chains per row.

// ------------------------------------------------------------------ Q4_K
// 144-byte super-block: f16 d @0, f16 dmin @2, 12 bytes of 6-bit (sc, m)
// pairs @4, qs[128] @16.  Quarter q = group oi of the page kernel: qs bytes
// [32q, 32q+32); byte l's low nibble is element 64q+l (pair 2q), high nibble
// element 64q+32+l (pair 2q+1); value (d*sc)*q - dmin*m.
//
// Lane element order: word t (bytes 4t..4t+3), i = 8t + j: j<4 -> low
// nibble of byte j, j>=4 -> high nibble of byte j-4.  Masking a word with
// 0x0F0F0F0F (after a shift by 4 for the high nibbles) leaves four quants in
// its bytes, multiplied by x registers 4t, 4t+1 (low) and 4t+2, 4t+3 (high).
struct FmtQ4K {
    static constexpr int SBB = 144;
    // Rows may sit at their global stride in shared memory (runs): the
    // lanes' 128-bit loads of two rows conflict at most two ways.  Formats
    // read with 32-bit loads would conflict eight ways.
    static constexpr bool RUNS_OK = true;
    // Row slot stride wanted modulo 128 bytes (-1: any odd multiple of 16)
    static constexpr int SLOT_REM128 = -1;
    __host__ __device__ static int elem(int q, int i) {
        int t = i >> 3, j = i & 7;
        return j < 4 ? 64 * q + 4 * t + j : 64 * q + 32 + 4 * t + (j - 4);
    }
    __host__ __device__ static int xslot(int e4) {
        const int q = e4 >> 4, r4 = e4 & 15;
        const int i4 = r4 < 8 ? 2 * r4 : 2 * (r4 - 8) + 1;
        return 4 * i4 + q;
    }
    // 6-bit (sc, m) of pairs 2q and 2q+1 — the unpacking of
    // ferrox_q4_k_scale_min, four pairs per 32-bit word: pairs 0..3 are the
    // low 6 bits of bytes 0..3 (sc) and 4..7 (m); pairs 4..7 join the low /
    // high nibble of bytes 8..11 with the top two bits of bytes 0..3 / 4..7.
    // The lane's word is selected branch-free; a byte becomes a float by a
    // byte permute into the mantissa of 2^23 and one subtraction.
    __device__ __forceinline__ static void scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int q,
                                                     float& sca, float& ma, float& scb,
                                                     float& mb) {
        const bool hi = q >= 2;
        const uint32_t sc_w =
            ((hi ? s2 : s0) & 0x0F0F0F0Fu) | ((hi ? (s0 >> 2) : s0) & 0x30303030u);
        const uint32_t m_w =
            ((hi ? (s2 >> 4) : s1) & 0x0F0F0F0Fu) | ((hi ? (s1 >> 2) : s1) & 0x30303030u);
        const uint32_t ia = 0x7540u | (2u * (q & 1)), ib = ia + 1u;
        sca = __int_as_float(__byte_perm(sc_w, 0x4B000000u, ia)) - 8388608.f;
        scb = __int_as_float(__byte_perm(sc_w, 0x4B000000u, ib)) - 8388608.f;
        ma = __int_as_float(__byte_perm(m_w, 0x4B000000u, ia)) - 8388608.f;
        mb = __int_as_float(__byte_perm(m_w, 0x4B000000u, ib)) - 8388608.f;
    }
    template <int R>
    __device__ __forceinline__ static void dotR(const uint8_t* const (&sb)[R], int q,
                                                const uint32_t (&x)[32], const float* xs16,
                                                const float* sx, float (&acc)[R]) {
        uint32_t W[R][8];
        uint4 h[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            h[r] = *reinterpret_cast<const uint4*>(sb[r]);
            const uint4 wa = *reinterpret_cast<const uint4*>(sb[r] + 16 + 32 * q);
            const uint4 wb = *reinterpret_cast<const uint4*>(sb[r] + 16 + 32 * q + 16);
            W[r][0] = wa.x; W[r][1] = wa.y; W[r][2] = wa.z; W[r][3] = wa.w;
            W[r][4] = wb.x; W[r][5] = wb.y; W[r][6] = wb.z; W[r][7] = wb.w;
        }
        int ilo[R], ihi[R];
#pragma unroll
        for (int r = 0; r < R; ++r) ilo[r] = ihi[r] = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t lo = W[r][t] & 0x0F0F0F0Fu, hi = (W[r][t] >> 4) & 0x0F0F0F0Fu;
                ilo[r] = dp_lo(x[4 * t], lo, ilo[r]);
                ilo[r] = dp_hi(x[4 * t + 1], lo, ilo[r]);
                ihi[r] = dp_lo(x[4 * t + 2], hi, ihi[r]);
                ihi[r] = dp_hi(x[4 * t + 3], hi, ihi[r]);
            }
        }
        const float Xa = xs16[4 * q] + xs16[4 * q + 1];
        const float Xb = xs16[4 * q + 2] + xs16[4 * q + 3];
        const float sa = sx[2 * q], sbx = sx[2 * q + 1];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float sca, ma, scb, mb;
            scale_min(h[r].y, h[r].z, h[r].w, q, sca, ma, scb, mb);
            const float d = f16_bits_to_f32(h[r].x);
            const float dmin = f16_bits_to_f32(h[r].x >> 16);
            acc[r] += d * fmaf(sca * sa, static_cast<float>(ilo[r]),
                               scb * sbx * static_cast<float>(ihi[r])) -
                      dmin * fmaf(ma, Xa, mb * Xb);
        }
    }
};

// ------------------------------------------------------------------ Q5_K
// 176-byte super-block: d @0, dmin @2, scales @4, qh[32] @16, qs[128] @48.
// As Q4_K, plus 16 where bit 2q (low half) / 2q+1 (high half) of qh[l] is
// set: the qh bit is rotated into bit 4 of each byte and merged with the
// nibble.  Lane element order as Q4_K.
struct FmtQ5K {
    static constexpr int SBB = 176;
    static constexpr bool RUNS_OK = true;
    static constexpr int SLOT_REM128 = -1;
    __host__ __device__ static int elem(int q, int i) { return FmtQ4K::elem(q, i); }
    __host__ __device__ static int xslot(int e4) { return FmtQ4K::xslot(e4); }
    template <int R>
    __device__ __forceinline__ static void dotR(const uint8_t* const (&sb)[R], int q,
                                                const uint32_t (&x)[32], const float* xs16,
                                                const float* sx, float (&acc)[R]) {
        const uint32_t rlo = static_cast<uint32_t>(4 - 2 * q) & 31u;
        const uint32_t rhi = static_cast<uint32_t>(3 - 2 * q) & 31u;
        uint32_t W[R][8], H[R][8];
        uint4 h[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            h[r] = *reinterpret_cast<const uint4*>(sb[r]);
            const uint4 qa = *reinterpret_cast<const uint4*>(sb[r] + 48 + 32 * q);
            const uint4 qb = *reinterpret_cast<const uint4*>(sb[r] + 48 + 32 * q + 16);
            const uint4 ha = *reinterpret_cast<const uint4*>(sb[r] + 16);
            const uint4 hb = *reinterpret_cast<const uint4*>(sb[r] + 32);
            W[r][0] = qa.x; W[r][1] = qa.y; W[r][2] = qa.z; W[r][3] = qa.w;
            W[r][4] = qb.x; W[r][5] = qb.y; W[r][6] = qb.z; W[r][7] = qb.w;
            H[r][0] = ha.x; H[r][1] = ha.y; H[r][2] = ha.z; H[r][3] = ha.w;
            H[r][4] = hb.x; H[r][5] = hb.y; H[r][6] = hb.z; H[r][7] = hb.w;
        }
        int ilo[R], ihi[R];
#pragma unroll
        for (int r = 0; r < R; ++r) ilo[r] = ihi[r] = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t w = W[r][t], hw = H[r][t];
                const uint32_t lo =
                    (w & 0x0F0F0F0Fu) | (__funnelshift_l(hw, hw, rlo) & 0x10101010u);
                const uint32_t hi =
                    ((w >> 4) & 0x0F0F0F0Fu) | (__funnelshift_l(hw, hw, rhi) & 0x10101010u);
                ilo[r] = dp_lo(x[4 * t], lo, ilo[r]);
                ilo[r] = dp_hi(x[4 * t + 1], lo, ilo[r]);
                ihi[r] = dp_lo(x[4 * t + 2], hi, ihi[r]);
                ihi[r] = dp_hi(x[4 * t + 3], hi, ihi[r]);
            }
        }
        const float Xa = xs16[4 * q] + xs16[4 * q + 1];
        const float Xb = xs16[4 * q + 2] + xs16[4 * q + 3];
        const float sa = sx[2 * q], sbx = sx[2 * q + 1];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float sca, ma, scb, mb;
            FmtQ4K::scale_min(h[r].y, h[r].z, h[r].w, q, sca, ma, scb, mb);
            const float d = f16_bits_to_f32(h[r].x);
            const float dmin = f16_bits_to_f32(h[r].x >> 16);
            acc[r] += d * fmaf(sca * sa, static_cast<float>(ilo[r]),
                               scb * sbx * static_cast<float>(ihi[r])) -
                      dmin * fmaf(ma, Xa, mb * Xb);
        }
    }
};

// ------------------------------------------------------------------ Q6_K
// 210-byte super-block: ql[128] @0, qh[64] @128, int8 sc[16] @192, f16 d
// @208.  Quarter q: half h = q>>1, l in [16c, 16c+16) with c = q&1.  For
// each l four 6-bit values minus 32 (4 bits of ql[64h+l] / ql[64h+32+l],
// 2 bits of qh[32h+l]) land at elements 128h + l + {0,32,64,96}, scaled by
// sc[8h + c + {0,2,4,6}]; value (d*sc)*(q-32).  Super-blocks are only
// 2-byte aligned, so words are read with funnel shifts.
// Lane element order: i = 16u + 4t + j -> element 128h + 32t + 16c + 4u + j.
// The 6-bit values are merged into the bytes of four words v_t (bits 6..7
// zero), multiplied by x registers 8u + 2t and 8u + 2t + 1; sub-block t (16
// elements) lies in x block 4h + t.
struct FmtQ6K {
    static constexpr int SBB = 210;
    static constexpr bool RUNS_OK = true;
    // 32 mod 128: the aligned loads of two row groups in a quarter-warp
    // fall in disjoint 16-byte bank groups
    static constexpr int SLOT_REM128 = 32;
    __host__ __device__ static int elem(int q, int i) {
        int u = i >> 4, t = (i >> 2) & 3, j = i & 3;
        return 128 * (q >> 1) + 32 * t + 16 * (q & 1) + 4 * u + j;
    }
    __host__ __device__ static int xslot(int e4) {
        const int h = e4 >> 5, t = (e4 >> 3) & 3, c = (e4 >> 2) & 1, u = e4 & 3;
        return 4 * (4 * u + t) + 2 * h + c;
    }
    // Words [4k, 4k+4) of the 32-byte window (lo, hi), J words plus sh bits in.
    template <int J>
    __device__ __forceinline__ static void window4(const uint4& lo, const uint4& hi, uint32_t sh,
                                                   uint32_t (&w)[4]) {
        const uint32_t r[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = __funnelshift_r(r[J + k], r[J + k + 1], sh);
    }
    // Loads of R super-blocks that all sit at byte phase 4J + sh/8 of a
    // 16-byte granule: aligned 128-bit loads (conflict-free for the slot
    // strides the planner picks) and funnel shifts.  The tail window reads
    // up to 14 bytes past the super-block, inside the stage's slack.
    template <int J, int R>
    __device__ __forceinline__ static void load_phase(const uint8_t* const (&sb)[R], int h, int c,
                                                      uint32_t sh, uint32_t (&A)[R][4],
                                                      uint32_t (&B)[R][4], uint32_t (&H)[R][4],
                                                      uint32_t (&S)[R][2], uint32_t (&db)[R]) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint4* p = reinterpret_cast<const uint4*>(sb[r] - (4 * J + (sh >> 3)));
            const int oa = 4 * h + c, oh = 8 + 2 * h + c;
            window4<J>(p[oa], p[oa + 1], sh, A[r]);
            window4<J>(p[oa + 2], p[oa + 3], sh, B[r]);
            window4<J>(p[oh], p[oh + 1], sh, H[r]);
            const uint4 t1 = p[13];
            uint32_t T[4];
            window4<J>(p[12], t1, sh, T);  // sc[0..15]
            S[r][0] = h ? T[2] : T[0];
            S[r][1] = h ? T[3] : T[1];
            const uint32_t tw[4] = {t1.x, t1.y, t1.z, t1.w};
            db[r] = tw[J] >> sh;
        }
    }
    template <int R>
    __device__ __forceinline__ static void dotR(const uint8_t* const (&sb)[R], int q,
                                                const uint32_t (&x)[32], const float* xs16,
                                                const float* sx, float (&acc)[R]) {
        if constexpr (R == 4) {
            // four rows' words beside the x registers exceed the register
            // budget (168 with nine warps): two passes of two rows, same x
            const uint8_t* const s0[2] = {sb[0], sb[1]};
            const uint8_t* const s1[2] = {sb[2], sb[3]};
            float a0[2] = {acc[0], acc[1]}, a1[2] = {acc[2], acc[3]};
            dotR<2>(s0, q, x, xs16, sx, a0);
            dotR<2>(s1, q, x, xs16, sx, a1);
            acc[0] = a0[0];
            acc[1] = a0[1];
            acc[2] = a1[0];
            acc[3] = a1[1];
            return;
        }
        const int h = q >> 1, c = q & 1;
        uint32_t A[R][4], B[R][4], H[R][4], S[R][2], db[R];
        float sc[R][4], d[R];
        // fast path when every row of every lane has the same 16-byte phase
        const uint32_t ph = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(sb[0])) & 15u;
        bool same = ph == static_cast<uint32_t>(__shfl_sync(0xffffffffu, static_cast<int>(ph), 0));
#pragma unroll
        for (int r = 1; r < R; ++r)
            same = same && ((static_cast<uint32_t>(reinterpret_cast<uintptr_t>(sb[r])) & 15u) == ph);
        if (__all_sync(0xffffffffu, same)) {
            const uint32_t sh = (ph & 3u) * 8u;
            switch (ph >> 2) {
            case 0: load_phase<0, R>(sb, h, c, sh, A, B, H, S, db); break;
            case 1: load_phase<1, R>(sb, h, c, sh, A, B, H, S, db); break;
            case 2: load_phase<2, R>(sb, h, c, sh, A, B, H, S, db); break;
            default: load_phase<3, R>(sb, h, c, sh, A, B, H, S, db); break;
            }
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                load4_u16al(sb[r] + 64 * h + 16 * c, A[r]);
                load4_u16al(sb[r] + 64 * h + 32 + 16 * c, B[r]);
                load4_u16al(sb[r] + 128 + 32 * h + 16 * c, H[r]);
                uint32_t T[4];
                load4_u16al(sb[r] + 192, T);  // sc[0..15]
                S[r][0] = h ? T[2] : T[0];
                S[r][1] = h ? T[3] : T[1];
                const uintptr_t a = reinterpret_cast<uintptr_t>(sb[r] + 208);
                const uint32_t dw = *reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
                db[r] = dw >> ((a & 3u) * 8u);
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            d[r] = f16_bits_to_f32(db[r]);
            // scales sc[8h + c + 2t], t = 0..3: bytes of words 2h, 2h+1 of sc
            const uint32_t s_lo = S[r][0], s_hi = S[r][1];
            sc[r][0] = static_cast<float>(static_cast<int8_t>(s_lo >> (8 * c)));
            sc[r][1] = static_cast<float>(static_cast<int8_t>(s_lo >> (8 * c + 16)));
            sc[r][2] = static_cast<float>(static_cast<int8_t>(s_hi >> (8 * c)));
            sc[r][3] = static_cast<float>(static_cast<int8_t>(s_hi >> (8 * c + 16)));
        }
        int i0[R], i1[R], i2[R], i3[R];
#pragma unroll
        for (int r = 0; r < R; ++r) i0[r] = i1[r] = i2[r] = i3[r] = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t av = A[r][u], bv = B[r][u], hv = H[r][u];
                const uint32_t v0 = (av & 0x0F0F0F0Fu) | ((hv << 4) & 0x30303030u);
                const uint32_t v1 = (bv & 0x0F0F0F0Fu) | ((hv << 2) & 0x30303030u);
                const uint32_t v2 = ((av >> 4) & 0x0F0F0F0Fu) | (hv & 0x30303030u);
                const uint32_t v3 = ((bv >> 4) & 0x0F0F0F0Fu) | ((hv >> 2) & 0x30303030u);
                const uint32_t* xu = x + 8 * u;
                i0[r] = dp_hi(xu[1], v0, dp_lo(xu[0], v0, i0[r]));
                i1[r] = dp_hi(xu[3], v1, dp_lo(xu[2], v1, i1[r]));
                i2[r] = dp_hi(xu[5], v2, dp_lo(xu[4], v2, i2[r]));
                i3[r] = dp_hi(xu[7], v3, dp_lo(xu[6], v3, i3[r]));
            }
        }
        // 16-element groups of this lane: 8h + 2t + c; x blocks 4h + t
        const float* X = xs16 + 8 * h + c;
        const float* XS = sx + 4 * h;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float d32 = -32.f * d[r];
            float res = sc[r][0] * fmaf(d32, X[0], XS[0] * d[r] * static_cast<float>(i0[r]));
            res = fmaf(sc[r][1], fmaf(d32, X[2], XS[1] * d[r] * static_cast<float>(i1[r])), res);
            res = fmaf(sc[r][2], fmaf(d32, X[4], XS[2] * d[r] * static_cast<float>(i2[r])), res);
            res = fmaf(sc[r][3], fmaf(d32, X[6], XS[3] * d[r] * static_cast<float>(i3[r])), res);
            acc[r] += res;
        }
    }
};

// ------------------------------------------------------------------ Q8_0
// 34-byte blocks: f16 d, 32 int8; value d*q.  A group of 8 blocks is 272
// bytes; quarter q holds blocks 2q, 2q+1 at byte 68q (4-byte aligned when
// the group is).  The signed quants go to dp2a as they are stored.
// Lane element order: i = 32k + j -> element 64q + 32k + j; block k's words
// t = 0..7 meet x registers 16k + 2t, 16k + 2t + 1.
struct FmtQ80 {
    static constexpr int SBB = 272;
    static constexpr bool RUNS_OK = false;
    static constexpr int SLOT_REM128 = -1;
    __host__ __device__ static int elem(int q, int i) { return 64 * q + i; }
    __host__ __device__ static int xslot(int e4) { return 4 * (e4 & 15) + (e4 >> 4); }
    template <int R>
    __device__ __forceinline__ static void dotR(const uint8_t* const (&sb)[R], int q,
                                                const uint32_t (&x)[32], const float* xs16,
                                                const float* sx, float (&acc)[R]) {
        uint32_t U[R][17];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t* u = reinterpret_cast<const uint32_t*>(sb[r] + 68 * q);
#pragma unroll
            for (int k = 0; k < 17; ++k) U[r][k] = u[k];
        }
        int iA[R], iB[R];
#pragma unroll
        for (int r = 0; r < R; ++r) iA[r] = iB[r] = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                // block A's quants start 2 bytes into the quarter, block B's
                // 4-byte aligned at byte 36
                const uint32_t wa = __funnelshift_r(U[r][t], U[r][t + 1], 16);
                const uint32_t wb = U[r][9 + t];
                iA[r] = dp_hi(x[2 * t + 1], wa, dp_lo(x[2 * t], wa, iA[r]));
                iB[r] = dp_hi(x[17 + 2 * t], wb, dp_lo(x[16 + 2 * t], wb, iB[r]));
            }
        }
        const float sA = sx[2 * q], sB = sx[2 * q + 1];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float dA = f16_bits_to_f32(U[r][0]);
            const float dB = f16_bits_to_f32(U[r][8] >> 16);
            acc[r] += fmaf(dA * sA, static_cast<float>(iA[r]), dB * sB * static_cast<float>(iB[r]));
        }
    }
};

// ------------------------------------------------------------------ Q4_0
// 18-byte blocks: f16 d, 16 bytes; byte i's low nibble is element i, high
// nibble element i+16; value (nibble-8)*d.  A group of 8 blocks is 144
// bytes; quarter q holds blocks 2q, 2q+1 at byte 36q.
// Lane element order: i = 32k + 8t + j: j<4 -> element 32(2q+k) + 4t + j,
// j>=4 -> element 32(2q+k) + 16 + 4t + (j-4): word t of block k meets x
// registers 16k + 4t, +1 (low nibbles) and 16k + 4t + 2, +3 (high nibbles).
struct FmtQ40 {
    static constexpr int SBB = 144;
    static constexpr bool RUNS_OK = false;
    static constexpr int SLOT_REM128 = -1;
    __host__ __device__ static int elem(int q, int i) {
        int k = i >> 5, t = (i >> 3) & 3, j = i & 7;
        int base = 32 * (2 * q + k);
        return j < 4 ? base + 4 * t + j : base + 16 + 4 * t + (j - 4);
    }
    __host__ __device__ static int xslot(int e4) {
        const int blk = e4 >> 3, r = e4 & 7;  // blk = 2q + k
        const int i4 = 8 * (blk & 1) + 2 * (r & 3) + (r >= 4 ? 1 : 0);
        return 4 * i4 + (blk >> 1);
    }
    template <int R>
    __device__ __forceinline__ static void dotR(const uint8_t* const (&sb)[R], int q,
                                                const uint32_t (&x)[32], const float* xs16,
                                                const float* sx, float (&acc)[R]) {
        uint32_t U[R][9];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t* u = reinterpret_cast<const uint32_t*>(sb[r] + 36 * q);
#pragma unroll
            for (int k = 0; k < 9; ++k) U[r][k] = u[k];
        }
        int ia[R][2];
#pragma unroll
        for (int r = 0; r < R; ++r) ia[r][0] = ia[r][1] = 0;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int o = 16 * k + 4 * t;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t w = k == 0 ? __funnelshift_r(U[r][t], U[r][t + 1], 16)
                                              : U[r][5 + t];
                    const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
                    ia[r][k] = dp_hi(x[o + 1], lo, dp_lo(x[o], lo, ia[r][k]));
                    ia[r][k] = dp_hi(x[o + 3], hi, dp_lo(x[o + 2], hi, ia[r][k]));
                }
            }
        }
        const float XA = xs16[4 * q] + xs16[4 * q + 1];
        const float XB = xs16[4 * q + 2] + xs16[4 * q + 3];
        const float sA = sx[2 * q], sB = sx[2 * q + 1];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float dA = f16_bits_to_f32(U[r][0]);
            const float dB = f16_bits_to_f32(U[r][4] >> 16);
            acc[r] += dA * fmaf(sA, static_cast<float>(ia[r][0]), -8.f * XA) +
                      dB * fmaf(sB, static_cast<float>(ia[r][1]), -8.f * XB);
        }
    }
};

}  // namespace qmoe
