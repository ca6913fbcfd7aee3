// formats.cuh — per-format decode-and-dot of one lane's quarter of a
// 256-element group, for the GGUF block layouts given by the CUDA kernel
// sources on "ferrox-cuda 0.14.0 — src/gpu.rs" (Q8_0_MATVEC_KERNEL_SRC,
// Q4_0_MATVEC_KERNEL_SRC, Q4_K_MATVEC_KERNEL_SRC with ferrox_q4_k_scale_min,
// Q5_K_MATVEC_KERNEL_SRC, Q6_K_MATVEC_KERNEL_SRC).
//
// Arithmetic (f32, as the page kernels: every product is a decoded weight
// times an f32 activation, summed in f32):
//   * Every integer quant q in a field [pos, pos+w) of a 32-bit word with
//     pos + w <= 24 is, reinterpreted as an IEEE binary32 bit pattern,
//     exactly q * 2^(pos-149) (a subnormal, or a normal with exponent field
//     1: the mapping bits -> value is linear below 2^24).  One AND isolates
//     the field; one FFMA against the pre-scaled activation
//         x'_j = x_j * 2^(128 - E_b - pos_j)
//     adds q * x_j * 2^-(21 + E_b), exact before its one rounding, into an f32
//     accumulator.  No int->float conversion, and the activations keep all
//     24 bits of f32.  (fp32 denormals run at full rate; the library is built
//     with -ftz=false.)
//   * E_b is the exponent of the largest |x| of the activation's 32-element
//     block b (max |x| < 2^E_b), clamped to [1, 106]: x' never overflows, the
//     products stay normal unless |x_j| is 2^104 below its block's largest,
//     and the block's de-scale 2^(21 + E_b) is a float.  Blocks holding a
//     non-finite value take E_b = 1, so NaN and Inf reach the result.
//     Activations of magnitude 2^106 or more (about 8e31) are outside the
//     range: the x table flags them (DEV_X_RANGE).
//   * Per sub-block the sum takes the block's de-scale once, and offsets and
//     mins are pulled out of the inner loop:
//         sum (d*sc*q - dmin*m) x = d*sc*sum q x - dmin*m*sum x
//     with sum x over each 16-element group computed once per call.  Only the
//     order of rounding differs from the page kernels' per-element form.
//
// A lane owns quarter q (0..3) of a 256-element group ("super-block"; for
// Q8_0/Q4_0, 8 consecutive 32-element blocks).  It processes 64 elements;
// element i (0..63) of its quarter is elem(q,i) of the group, and its field
// sits at bit pos(q,i) once isolated.  x' is stored in shared memory as
// float4 [group][i/4][q], so the four quarter-lanes read 64 contiguous
// bytes; the element loop of dotR loads the x' of each word as it goes and
// applies them to several rows.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace qmoe {

enum QType : int { QT_F32 = 0, QT_Q8_0 = 1, QT_Q4_0 = 2, QT_Q4_K = 3, QT_Q5_K = 4, QT_Q6_K = 5 };

__device__ __forceinline__ float f16_bits_to_f32(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// Two isolated fields (their bits as floats, q * 2^(pos-149)) times their
// x' on the packed f32x2 FMA: acc.{x,y} += q{0,1} * x{0,1} * 2^-(21 + E_b).
__device__ __forceinline__ float2 qfma2(uint32_t m0, uint32_t m1, float x0, float x1,
                                        float2 acc) {
    return __ffma2_rn(make_float2(__uint_as_float(m0), __uint_as_float(m1)),
                      make_float2(x0, x1), acc);
}

// The x table's scales: 2^(128 - E - pos) for an activation of block
// exponent E whose field sits at bit pos, and the block's de-scale
// 2^(21 + E); E in [1, 106], pos in [0, 20], so both are normal floats.
__host__ __device__ __forceinline__ float pow2f(int e) {  // 2^e, -126 <= e <= 127
#ifdef __CUDA_ARCH__
    return __int_as_float((127 + e) << 23);
#else
    union { int i; float f; } u;
    u.i = (127 + e) << 23;
    return u.f;
#endif
}
constexpr int XBLK_EMIN = 1, XBLK_EMAX = 106;

// Bits [24, 24+n) of w isolated at bit 0, on the multiply pipe:
// (w << (8-n)) keeps them topmost, the high half of * 2^n keeps only them.
template <int N>
__device__ __forceinline__ uint32_t top_field(uint32_t w) {
    return __umulhi(w << (8 - N), 1u << N);
}

// A lane's x' values of one group: xg = (the group's float4 table) + q, so
// that its elements 4*i4 .. 4*i4+3 are xg[4 * i4].  Each format's element
// loop loads the four or eight x' it needs next from shared memory (a
// broadcast to the eight row lanes of each quarter) and applies them to all
// R rows, so no lane holds its 64 x' in registers.

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

// N consecutive 32-bit words from a 2-byte-aligned shared-memory address.
// Rows of whole 256-element groups are 4-byte aligned (plain loads); a
// Q8_0/Q4_0 row of an odd number of 32-element blocks is only 2-byte
// aligned, and its words are funnel-shifted out of aligned loads (one word
// more, inside the stage's slack).
template <int N>
__device__ __forceinline__ void load_words(const uint8_t* p, uint32_t (&w)[N]) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* u = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    if ((a & 2u) == 0) {
#pragma unroll
        for (int k = 0; k < N; ++k) w[k] = u[k];
    } else {
        uint32_t prev = u[0];
#pragma unroll
        for (int k = 0; k < N; ++k) {
            const uint32_t next = u[k + 1];
            w[k] = __funnelshift_r(prev, next, 16);
            prev = next;
        }
    }
}

// Every format provides
//   elem(q, i), pos(q, i)  — the lane element order and extraction offsets;
//   xslot(e4)   — the inverse of elem on 4-element granules: the slot
//                 4*i4 + q whose elements elem(q, 4*i4 .. 4*i4+3) are
//                 elements 4*e4 .. 4*e4+3 of the group;
//   dotR<R>(sb[R], q, xg, xs16, sx, nblk, acc[R]) — for R rows whose
//   super-blocks start at sb[r] (shared memory), adds each row's dot over the
//   lane's quarter to acc[r]; xg: the lane's x' (above), xs16: sum x per 16
//   elements of the group, sx: the de-scales 2^(21 + E_b) of its eight
//   32-element blocks; nblk: the group's valid 32-element blocks (8, or fewer
//   for the partial last group of a Q8_0/Q4_0 row; the other formats always
//   have 8).
//   Words of all R rows are loaded first and the element loop runs over
//   words with the rows innermost, so a lane carries several independent
//   FFMA chains.

// ------------------------------------------------------------------ Q4_K
// 144-byte super-block: f16 d @0, f16 dmin @2, 12 bytes of 6-bit (sc, m)
// pairs @4, qs[128] @16.  Quarter q = group oi of the page kernel: qs bytes
// [32q, 32q+32); byte l's low nibble is element 64q+l (pair 2q), high nibble
// element 64q+32+l (pair 2q+1); value (d*sc)*q - dmin*m.
//
// Lane element order: word t (bytes 4t..4t+3), i = 8t + j: j<4 -> low
// nibble of byte j, j>=4 -> high nibble of byte j-4.
// Extraction per word W: lo b0 &0xF (0), lo b1 &0xF00 (8), lo b2 &0xF0000
// (16), hi b0 &0xF0 (4), hi b1 &0xF000 (12), hi b2 &0xF00000 (20); byte 3's
// nibbles come from the multiply pipe (top_field, __umulhi): both at bit 0.
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
    // Inverse of elem on float4 granules: the x' slot (4*i4 + q) holding
    // elements 4*e4 .. 4*e4+3 of the group.
    __host__ __device__ static int xslot(int e4) {
        const int q = e4 >> 4, r4 = e4 & 15;
        const int i4 = r4 < 8 ? 2 * r4 : 2 * (r4 - 8) + 1;
        return 4 * i4 + q;
    }
    __host__ __device__ static int pos(int, int i) {
        // bit offsets {0, 8, 16, 0, 4, 12, 20, 0} by i % 8, one byte each
        return static_cast<int>((0x00140C0400100800ull >> (8 * (i & 7))) & 0xFFu);
    }
    // pos depends on i % 8 (not only i % 4): the x table's scales use it
    static constexpr bool POS8 = true;
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
                                                const float4* __restrict__ xg, const float* xs16,
                                                const float* sx, int nblk, float (&acc)[R]) {
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
        float2 alo[R], ahi[R];
#pragma unroll
        for (int r = 0; r < R; ++r) alo[r] = ahi[r] = make_float2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const float4 xa = xg[8 * t], xb = xg[8 * t + 4];  // elements 8t .. 8t+7
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t w = W[r][t];
                alo[r] = qfma2(w & 0xFu, w & 0xF00u, xa.x, xa.y, alo[r]);
                alo[r] = qfma2(w & 0xF0000u, top_field<4>(w), xa.z, xa.w, alo[r]);
                ahi[r] = qfma2(w & 0xF0u, w & 0xF000u, xb.x, xb.y, ahi[r]);
                ahi[r] = qfma2(w & 0xF00000u, __umulhi(w, 16u), xb.z, xb.w, ahi[r]);
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
            // (sum of the block's products) * de-scale = sum q x
            acc[r] += d * fmaf(sca, (alo[r].x + alo[r].y) * sa,
                               scb * ((ahi[r].x + ahi[r].y) * sbx)) -
                      dmin * fmaf(ma, Xa, mb * Xb);
        }
    }
};

// ------------------------------------------------------------------ Q5_K
// 176-byte super-block: d @0, dmin @2, scales @4, qh[32] @16, qs[128] @48.
// As Q4_K, plus 16 where bit 2q (low half) / 2q+1 (high half) of qh[l] is
// set.  The qh bit is rotated into bit 4 of each byte and merged with the
// nibble; bits 5..7 of every merged byte are zero, so byte 3's field is
// one shift.
// Lane element order as Q4_K; positions: byte k -> 8k for k<3, byte 3's
// field shifted down -> 0.
struct FmtQ5K {
    static constexpr int SBB = 176;
    static constexpr bool RUNS_OK = true;
    static constexpr int SLOT_REM128 = -1;
    __host__ __device__ static int elem(int q, int i) { return FmtQ4K::elem(q, i); }
    __host__ __device__ static int xslot(int e4) { return FmtQ4K::xslot(e4); }
    __host__ __device__ static int pos(int, int i) {
        // bit offsets {0, 8, 16, 0} by i % 4
        return static_cast<int>((0x00100800u >> (8 * (i & 3))) & 0xFFu);
    }
    static constexpr bool POS8 = false;
    template <int R>
    __device__ __forceinline__ static void dotR(const uint8_t* const (&sb)[R], int q,
                                                const float4* __restrict__ xg, const float* xs16,
                                                const float* sx, int nblk, float (&acc)[R]) {
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
        float2 alo[R], ahi[R];
#pragma unroll
        for (int r = 0; r < R; ++r) alo[r] = ahi[r] = make_float2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const float4 xa = xg[8 * t], xb = xg[8 * t + 4];  // elements 8t .. 8t+7
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t w = W[r][t], hw = H[r][t];
                const uint32_t lo =
                    (w & 0x0F0F0F0Fu) | (__funnelshift_l(hw, hw, rlo) & 0x10101010u);
                const uint32_t hi =
                    ((w >> 4) & 0x0F0F0F0Fu) | (__funnelshift_l(hw, hw, rhi) & 0x10101010u);
                alo[r] = qfma2(lo & 0x1Fu, lo & 0x1F00u, xa.x, xa.y, alo[r]);
                alo[r] = qfma2(lo & 0x1F0000u, lo >> 24, xa.z, xa.w, alo[r]);
                ahi[r] = qfma2(hi & 0x1Fu, hi & 0x1F00u, xb.x, xb.y, ahi[r]);
                ahi[r] = qfma2(hi & 0x1F0000u, hi >> 24, xb.z, xb.w, ahi[r]);
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
            acc[r] += d * fmaf(sca, (alo[r].x + alo[r].y) * sa,
                               scb * ((ahi[r].x + ahi[r].y) * sbx)) -
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
// Lane element order: i = 16u + 4t + j -> element 128h + 32t + 16c + 4u + j;
// positions (0, 8, 16, 0).  The 6-bit values are merged with bits 6..7 of
// every byte zero, so byte 3's field is one shift.
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
    __host__ __device__ static int pos(int, int i) {
        // bit offsets {0, 8, 16, 0} by i % 4
        return static_cast<int>((0x00100800u >> (8 * (i & 3))) & 0xFFu);
    }
    static constexpr bool POS8 = false;
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
                                                const float4* __restrict__ xg, const float* xs16,
                                                const float* sx, int nblk, float (&acc)[R]) {
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
        float2 a0[R], a1[R], a2[R], a3[R];
#pragma unroll
        for (int r = 0; r < R; ++r) a0[r] = a1[r] = a2[r] = a3[r] = make_float2(0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            // elements 16u .. 16u+15
            const float4 x0 = xg[16 * u], x1 = xg[16 * u + 4], x2 = xg[16 * u + 8],
                         x3 = xg[16 * u + 12];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t av = A[r][u], bv = B[r][u], hv = H[r][u];
                const uint32_t v0 = (av & 0x0F0F0F0Fu) | ((hv << 4) & 0x30303030u);
                const uint32_t v1 = (bv & 0x0F0F0F0Fu) | ((hv << 2) & 0x30303030u);
                const uint32_t v2 = ((av >> 4) & 0x0F0F0F0Fu) | (hv & 0x30303030u);
                const uint32_t v3 = ((bv >> 4) & 0x0F0F0F0Fu) | ((hv >> 2) & 0x30303030u);
                a0[r] = qfma2(v0 & 0x3Fu, v0 & 0x3F00u, x0.x, x0.y, a0[r]);
                a0[r] = qfma2(v0 & 0x3F0000u, v0 >> 24, x0.z, x0.w, a0[r]);
                a1[r] = qfma2(v1 & 0x3Fu, v1 & 0x3F00u, x1.x, x1.y, a1[r]);
                a1[r] = qfma2(v1 & 0x3F0000u, v1 >> 24, x1.z, x1.w, a1[r]);
                a2[r] = qfma2(v2 & 0x3Fu, v2 & 0x3F00u, x2.x, x2.y, a2[r]);
                a2[r] = qfma2(v2 & 0x3F0000u, v2 >> 24, x2.z, x2.w, a2[r]);
                a3[r] = qfma2(v3 & 0x3Fu, v3 & 0x3F00u, x3.x, x3.y, a3[r]);
                a3[r] = qfma2(v3 & 0x3F0000u, v3 >> 24, x3.z, x3.w, a3[r]);
            }
        }
        // 16-element groups of this lane: 8h + 2t + c; x blocks 4h + t
        const float* X = xs16 + 8 * h + c;
        const float* XS = sx + 4 * h;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float d32 = -32.f * d[r];
            float res = sc[r][0] * fmaf(d32, X[0], (a0[r].x + a0[r].y) * XS[0] * d[r]);
            res = fmaf(sc[r][1], fmaf(d32, X[2], (a1[r].x + a1[r].y) * XS[1] * d[r]), res);
            res = fmaf(sc[r][2], fmaf(d32, X[4], (a2[r].x + a2[r].y) * XS[2] * d[r]), res);
            res = fmaf(sc[r][3], fmaf(d32, X[6], (a3[r].x + a3[r].y) * XS[3] * d[r]), res);
            acc[r] += res;
        }
    }
};

// ------------------------------------------------------------------ Q8_0
// 34-byte blocks: f16 d, 32 int8; value d*q.  A group of 8 blocks is 272
// bytes; quarter q holds blocks 2q, 2q+1 at byte 68q (4-byte aligned when
// the group is; a row of an odd number of blocks is 2-byte aligned).  q+128 is extracted as an unsigned byte (XOR 0x80) and the
// 128*sum(x) offset removed per block.
// Lane element order: i = 32k + 4t + j -> element 64q + 32k + 4t + j;
// positions (0, 8, 16, 0).
struct FmtQ80 {
    static constexpr int SBB = 272;
    static constexpr bool RUNS_OK = false;
    static constexpr int SLOT_REM128 = -1;
    __host__ __device__ static int elem(int q, int i) { return 64 * q + i; }
    __host__ __device__ static int xslot(int e4) { return 4 * (e4 & 15) + (e4 >> 4); }
    __host__ __device__ static int pos(int, int i) {
        // bit offsets {0, 8, 16, 0} by i % 4
        return static_cast<int>((0x00100800u >> (8 * (i & 3))) & 0xFFu);
    }
    static constexpr bool POS8 = false;
    template <int R>
    __device__ __forceinline__ static void dotR(const uint8_t* const (&sb)[R], int q,
                                                const float4* __restrict__ xg, const float* xs16,
                                                const float* sx, int nblk, float (&acc)[R]) {
        uint32_t U[R][17];
#pragma unroll
        for (int r = 0; r < R; ++r) load_words<17>(sb[r] + 68 * q, U[r]);
        float2 aA[R], aB[R];
#pragma unroll
        for (int r = 0; r < R; ++r) aA[r] = aB[r] = make_float2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const float4 xa = xg[4 * t], xb = xg[32 + 4 * t];  // elements 4t.., 32+4t..
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t wa = __funnelshift_r(U[r][t], U[r][t + 1], 16);
                const uint32_t wb = U[r][9 + t];
                aA[r] = qfma2((wa ^ 0x80808080u) & 0xFFu, (wa ^ 0x80808080u) & 0xFF00u, xa.x,
                              xa.y, aA[r]);
                aA[r] = qfma2((wa ^ 0x80808080u) & 0xFF0000u, __umulhi(wa + 0x80000000u, 256u),
                              xa.z, xa.w, aA[r]);
                aB[r] = qfma2((wb ^ 0x80808080u) & 0xFFu, (wb ^ 0x80808080u) & 0xFF00u, xb.x,
                              xb.y, aB[r]);
                aB[r] = qfma2((wb ^ 0x80808080u) & 0xFF0000u, __umulhi(wb + 0x80000000u, 256u),
                              xb.z, xb.w, aB[r]);
            }
        }
        const float XA = xs16[4 * q] + xs16[4 * q + 1];
        const float XB = xs16[4 * q + 2] + xs16[4 * q + 3];
        const float sA = sx[2 * q], sB = sx[2 * q + 1];
        // blocks past a partial group's end hold stale bytes: selected away
        const bool okA = 2 * q < nblk, okB = 2 * q + 1 < nblk;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float dA = f16_bits_to_f32(U[r][0]);
            const float dB = f16_bits_to_f32(U[r][8] >> 16);
            const float vA = dA * fmaf(aA[r].x + aA[r].y, sA, -128.f * XA);
            const float vB = dB * fmaf(aB[r].x + aB[r].y, sB, -128.f * XB);
            acc[r] += (okA ? vA : 0.f) + (okB ? vB : 0.f);
        }
    }
};

// ------------------------------------------------------------------ Q4_0
// 18-byte blocks: f16 d, 16 bytes; byte i's low nibble is element i, high
// nibble element i+16; value (nibble-8)*d.  A group of 8 blocks is 144
// bytes; quarter q holds blocks 2q, 2q+1 at byte 36q.
// Lane element order: i = 32k + 8t + j: j<4 -> element 32(2q+k) + 4t + j,
// j>=4 -> element 32(2q+k) + 16 + 4t + (j-4); positions as Q4_K.
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
    __host__ __device__ static int pos(int q, int i) { return FmtQ4K::pos(q, i); }
    static constexpr bool POS8 = true;
    template <int R>
    __device__ __forceinline__ static void dotR(const uint8_t* const (&sb)[R], int q,
                                                const float4* __restrict__ xg, const float* xs16,
                                                const float* sx, int nblk, float (&acc)[R]) {
        uint32_t U[R][9];
#pragma unroll
        for (int r = 0; r < R; ++r) load_words<9>(sb[r] + 36 * q, U[r]);
        float2 a[R][2];
#pragma unroll
        for (int r = 0; r < R; ++r) a[r][0] = a[r][1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int o = 32 * k + 8 * t;  // elements o .. o+7
                const float4 xa = xg[o], xb = xg[o + 4];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t w = k == 0 ? __funnelshift_r(U[r][t], U[r][t + 1], 16)
                                              : U[r][5 + t];
                    a[r][k] = qfma2(w & 0xFu, w & 0xF00u, xa.x, xa.y, a[r][k]);
                    a[r][k] = qfma2(w & 0xF0000u, top_field<4>(w), xa.z, xa.w, a[r][k]);
                    a[r][k] = qfma2(w & 0xF0u, w & 0xF000u, xb.x, xb.y, a[r][k]);
                    a[r][k] = qfma2(w & 0xF00000u, __umulhi(w, 16u), xb.z, xb.w, a[r][k]);
                }
            }
        }
        const float XA = xs16[4 * q] + xs16[4 * q + 1];
        const float XB = xs16[4 * q + 2] + xs16[4 * q + 3];
        const float sA = sx[2 * q], sB = sx[2 * q + 1];
        // blocks past a partial group's end hold stale bytes: selected away
        const bool okA = 2 * q < nblk, okB = 2 * q + 1 < nblk;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float dA = f16_bits_to_f32(U[r][0]);
            const float dB = f16_bits_to_f32(U[r][4] >> 16);
            const float vA = dA * fmaf(a[r][0].x + a[r][0].y, sA, -8.f * XA);
            const float vB = dB * fmaf(a[r][1].x + a[r][1].y, sB, -8.f * XB);
            acc[r] += (okA ? vA : 0.f) + (okB ? vB : 0.f);
        }
    }
};

}  // namespace qmoe
