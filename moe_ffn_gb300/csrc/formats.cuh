// formats.cuh — per-format decode-and-dot of one lane's quarter of a
// 256-element group, for the GGUF block layouts given by the CUDA kernel
// sources on "ferrox-cuda 0.14.0 — src/gpu.rs" (Q8_0_MATVEC_KERNEL_SRC,
// Q4_0_MATVEC_KERNEL_SRC, Q4_K_MATVEC_KERNEL_SRC with ferrox_q4_k_scale_min,
// Q5_K_MATVEC_KERNEL_SRC, Q6_K_MATVEC_KERNEL_SRC).
//
// Arithmetic scheme (ours, not the pages'):
//   * Every integer quant q in a field [pos, pos+w) of a 32-bit word with
//     pos + w <= 24 is, reinterpreted as an IEEE binary32 bit pattern,
//     exactly q * 2^(pos-149) (a subnormal, or a normal with exponent field 1
//     — the mapping bits -> value is linear below 2^24).  One AND isolates
//     the field; one FFMA against x'_j = x_j * 2^(85-pos) adds q*x_j*2^-64
//     exactly-rounded into an f32 accumulator.  No int->float conversion.
//     (fp32 denormals are handled at full rate; the library is built with
//     -ftz=false.)
//   * Offsets and mins are pulled out of the inner loop:
//       sum (d*sc*q - dmin*m) x = d*sc*sum q x - dmin*m*sum x
//     with sum x over each 16-element group precomputed once per call.
//   * Accumulation is f32; only the order of rounding differs from the
//     page kernels' per-element form.
//
// A lane owns quarter q (0..3) of a 256-element group ("super-block"; for
// Q8_0/Q4_0, 8 consecutive 32-element blocks).  It processes 64 elements;
// element i (0..63) of its quarter is elem(q,i) of the group, and sits at
// bit offset pos(q,i) after extraction.  x' is stored in shared memory as
// float4 [group][i/4][q] so the four quarter-lanes read 64 contiguous bytes.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace qmoe {

enum QType : int { QT_F32 = 0, QT_Q8_0 = 1, QT_Q4_0 = 2, QT_Q4_K = 3, QT_Q5_K = 4, QT_Q6_K = 5 };

__device__ __forceinline__ float f16_bits_to_f32(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// q (integer bits) * x' (x * 2^(85-pos)) accumulated: acc += q*x*2^-64.
__device__ __forceinline__ float qfma(uint32_t masked_bits, float xs, float acc) {
    return fmaf(__uint_as_float(masked_bits), xs, acc);
}

// 2^(85 - pos) as a float, exact.
__host__ __device__ __forceinline__ float xprime_scale(int pos) {
#ifdef __CUDA_ARCH__
    return __int_as_float((127 + 85 - pos) << 23);
#else
    union { int i; float f; } u;
    u.i = (127 + 85 - pos) << 23;
    return u.f;
#endif
}

// 2^64, folded into d.
constexpr float TWO64 = 18446744073709551616.0f;

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

// ------------------------------------------------------------------ Q4_K
// 144-byte super-block: f16 d @0, f16 dmin @2, 12 bytes of 6-bit (sc, m)
// pairs @4, qs[128] @16.  Quarter q = group oi of the page kernel: qs bytes
// [32q, 32q+32); byte l's low nibble is element 64q+l (pair 2q), high nibble
// element 64q+32+l (pair 2q+1); value (d*sc)*q - dmin*m.
//
// Lane element order: word t (bytes 4t..4t+3), i = 8t + j: j<4 -> low
// nibble of byte j, j>=4 -> high nibble of byte j-4.
// Extraction per word W: lo b0 &0xF (0), lo b1 &0xF00 (8), lo b2 &0xF0000
// (16), hi b0 &0xF0 (4), hi b1 &0xF000 (12), hi b2 &0xF00000 (20); byte 3
// via W>>24: lo &0xF (0), hi &0xF0 (4).
struct FmtQ4K {
    static constexpr int SBB = 144;
    __host__ __device__ static int elem(int q, int i) {
        int t = i >> 3, j = i & 7;
        return j < 4 ? 64 * q + 4 * t + j : 64 * q + 32 + 4 * t + (j - 4);
    }
    __host__ __device__ static int pos(int, int i) {
        // bit offsets {0, 8, 16, 0, 4, 12, 20, 4} by i % 8, one byte each
        return static_cast<int>((0x04140C0400100800ull >> (8 * (i & 7))) & 0xFFu);
    }
    // 6-bit (sc, m) of pairs 2q and 2q+1 — the unpacking of
    // ferrox_q4_k_scale_min, written branch-free over the lane's q.
    __device__ __forceinline__ static void scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int q,
                                                     float& sca, float& ma, float& scb,
                                                     float& mb) {
        const bool hi = q >= 2;               // pairs j >= 4
        const int b = (2 * q) & 3;            // byte of pair 2q within its word
        const uint32_t lsc = hi ? s2 : s0;    // low nibble source for sc
        const uint32_t lm = hi ? s2 : s1;     // low nibble source for m
        const int lsc_sh = 8 * b, lm_sh = hi ? 8 * b + 4 : 8 * b;
        const int hsh = hi ? 8 * b + 6 : 8 * b + 4;
        // pair 2q (byte b) and 2q+1 (byte b+1)
        uint32_t sc0 = ((lsc >> lsc_sh) & 15u) | (((s0 >> hsh) & 3u) << 4);
        uint32_t m0 = ((lm >> lm_sh) & 15u) | (((s1 >> hsh) & 3u) << 4);
        uint32_t sc1 = ((lsc >> (lsc_sh + 8)) & 15u) | (((s0 >> (hsh + 8)) & 3u) << 4);
        uint32_t m1 = ((lm >> (lm_sh + 8)) & 15u) | (((s1 >> (hsh + 8)) & 3u) << 4);
        sca = static_cast<float>(sc0);
        ma = static_cast<float>(m0);
        scb = static_cast<float>(sc1);
        mb = static_cast<float>(m1);
    }
    __device__ __forceinline__ static float dot(const uint8_t* sb, int q, const float4* xq,
                                                const float* xs16) {
        const uint4 h = *reinterpret_cast<const uint4*>(sb);
        const float d = f16_bits_to_f32(h.x) * TWO64;
        const float dmin = f16_bits_to_f32(h.x >> 16);
        float sca, ma, scb, mb;
        scale_min(h.y, h.z, h.w, q, sca, ma, scb, mb);
        const uint4 wa = *reinterpret_cast<const uint4*>(sb + 16 + 32 * q);
        const uint4 wb = *reinterpret_cast<const uint4*>(sb + 16 + 32 * q + 16);
        const uint32_t W[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
        float alo = 0.f, ahi = 0.f, alo2 = 0.f, ahi2 = 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t w = W[t], v = w >> 24;
            const float4 xl = xq[(2 * t) * 4 + q];
            const float4 xh = xq[(2 * t + 1) * 4 + q];
            alo = qfma(w & 0xFu, xl.x, alo);
            alo2 = qfma(w & 0xF00u, xl.y, alo2);
            alo = qfma(w & 0xF0000u, xl.z, alo);
            alo2 = qfma(v & 0xFu, xl.w, alo2);
            ahi = qfma(w & 0xF0u, xh.x, ahi);
            ahi2 = qfma(w & 0xF000u, xh.y, ahi2);
            ahi = qfma(w & 0xF00000u, xh.z, ahi);
            ahi2 = qfma(v & 0xF0u, xh.w, ahi2);
        }
        alo += alo2;
        ahi += ahi2;
        const float Xa = xs16[4 * q] + xs16[4 * q + 1];
        const float Xb = xs16[4 * q + 2] + xs16[4 * q + 3];
        return d * fmaf(sca, alo, scb * ahi) - dmin * fmaf(ma, Xa, mb * Xb);
    }
};

// ------------------------------------------------------------------ Q5_K
// 176-byte super-block: d @0, dmin @2, scales @4, qh[32] @16, qs[128] @48.
// As Q4_K, plus 16 where bit 2q (low half) / 2q+1 (high half) of qh[l] is
// set.  The qh bit is rotated into bit 4 of each byte and merged with the
// nibble (bits 5..7 of the merge are don't-care: the 5-bit mask drops them).
// Lane element order as Q4_K; positions: byte k -> 8k for k<3, byte 3 via
// >>8 -> 16.
struct FmtQ5K {
    static constexpr int SBB = 176;
    __host__ __device__ static int elem(int q, int i) { return FmtQ4K::elem(q, i); }
    __host__ __device__ static int pos(int, int i) {
        // bit offsets {0, 8, 16, 16} by i % 4
        return static_cast<int>((0x10100800u >> (8 * (i & 3))) & 0xFFu);
    }
    __device__ __forceinline__ static float dot(const uint8_t* sb, int q, const float4* xq,
                                                const float* xs16) {
        const uint4 h = *reinterpret_cast<const uint4*>(sb);
        const float d = f16_bits_to_f32(h.x) * TWO64;
        const float dmin = f16_bits_to_f32(h.x >> 16);
        float sca, ma, scb, mb;
        FmtQ4K::scale_min(h.y, h.z, h.w, q, sca, ma, scb, mb);
        const uint4 qa = *reinterpret_cast<const uint4*>(sb + 48 + 32 * q);
        const uint4 qb = *reinterpret_cast<const uint4*>(sb + 48 + 32 * q + 16);
        const uint4 ha = *reinterpret_cast<const uint4*>(sb + 16);
        const uint4 hb = *reinterpret_cast<const uint4*>(sb + 32);
        const uint32_t W[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        const uint32_t H[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
        const uint32_t rlo = static_cast<uint32_t>(4 - 2 * q) & 31u;
        const uint32_t rhi = static_cast<uint32_t>(3 - 2 * q) & 31u;
        float alo = 0.f, ahi = 0.f, alo2 = 0.f, ahi2 = 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t w = W[t], hw = H[t];
            const uint32_t lo = (w & 0x0F0F0F0Fu) | (__funnelshift_l(hw, hw, rlo) & 0xF0F0F0F0u);
            const uint32_t hi =
                ((w >> 4) & 0x0F0F0F0Fu) | (__funnelshift_l(hw, hw, rhi) & 0xF0F0F0F0u);
            const float4 xl = xq[(2 * t) * 4 + q];
            const float4 xh = xq[(2 * t + 1) * 4 + q];
            alo = qfma(lo & 0x1Fu, xl.x, alo);
            alo2 = qfma(lo & 0x1F00u, xl.y, alo2);
            alo = qfma(lo & 0x1F0000u, xl.z, alo);
            alo2 = qfma((lo >> 8) & 0x1F0000u, xl.w, alo2);
            ahi = qfma(hi & 0x1Fu, xh.x, ahi);
            ahi2 = qfma(hi & 0x1F00u, xh.y, ahi2);
            ahi = qfma(hi & 0x1F0000u, xh.z, ahi);
            ahi2 = qfma((hi >> 8) & 0x1F0000u, xh.w, ahi2);
        }
        alo += alo2;
        ahi += ahi2;
        const float Xa = xs16[4 * q] + xs16[4 * q + 1];
        const float Xb = xs16[4 * q + 2] + xs16[4 * q + 3];
        return d * fmaf(sca, alo, scb * ahi) - dmin * fmaf(ma, Xa, mb * Xb);
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
// positions (0, 8, 16, 16).
struct FmtQ6K {
    static constexpr int SBB = 210;
    __host__ __device__ static int elem(int q, int i) {
        int u = i >> 4, t = (i >> 2) & 3, j = i & 3;
        return 128 * (q >> 1) + 32 * t + 16 * (q & 1) + 4 * u + j;
    }
    __host__ __device__ static int pos(int, int i) {
        // bit offsets {0, 8, 16, 16} by i % 4
        return static_cast<int>((0x10100800u >> (8 * (i & 3))) & 0xFFu);
    }
    __device__ __forceinline__ static float dot(const uint8_t* sb, int q, const float4* xq,
                                                const float* xs16) {
        const int h = q >> 1, c = q & 1;
        uint32_t A[4], B[4], H[4], S[4];
        load4_u16al(sb + 64 * h + 16 * c, A);
        load4_u16al(sb + 64 * h + 32 + 16 * c, B);
        load4_u16al(sb + 128 + 32 * h + 16 * c, H);
        load4_u16al(sb + 192, S);  // S[0..3] = sc[0..15]; S[4] would overrun: d read below
        const uintptr_t a = reinterpret_cast<uintptr_t>(sb + 208);
        const uint32_t dw = *reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
        const float d = f16_bits_to_f32(dw >> ((a & 3u) * 8u));
        const float d64 = d * TWO64, d32 = -32.f * d;
        // scales sc[8h + c + 2t], t = 0..3: bytes of S[2h], S[2h+1]
        const uint32_t s_lo = S[2 * h], s_hi = S[2 * h + 1];
        const float sc0 = static_cast<float>(static_cast<int8_t>(s_lo >> (8 * c)));
        const float sc1 = static_cast<float>(static_cast<int8_t>(s_lo >> (8 * c + 16)));
        const float sc2 = static_cast<float>(static_cast<int8_t>(s_hi >> (8 * c)));
        const float sc3 = static_cast<float>(static_cast<int8_t>(s_hi >> (8 * c + 16)));
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t av = A[u], bv = B[u], hv = H[u];
            const uint32_t v0 = (av & 0x0F0F0F0Fu) | ((hv << 4) & 0xF0F0F0F0u);
            const uint32_t v1 = (bv & 0x0F0F0F0Fu) | ((hv << 2) & 0xF0F0F0F0u);
            const uint32_t v2 = ((av >> 4) & 0x0F0F0F0Fu) | (hv & 0xF0F0F0F0u);
            const uint32_t v3 = ((bv >> 4) & 0x0F0F0F0Fu) | ((hv >> 2) & 0xF0F0F0F0u);
            const float4 x0 = xq[(4 * u + 0) * 4 + q];
            const float4 x1 = xq[(4 * u + 1) * 4 + q];
            const float4 x2 = xq[(4 * u + 2) * 4 + q];
            const float4 x3 = xq[(4 * u + 3) * 4 + q];
            a0 = qfma(v0 & 0x3Fu, x0.x, a0);
            a0 = qfma(v0 & 0x3F00u, x0.y, a0);
            a0 = qfma(v0 & 0x3F0000u, x0.z, a0);
            a0 = qfma((v0 >> 8) & 0x3F0000u, x0.w, a0);
            a1 = qfma(v1 & 0x3Fu, x1.x, a1);
            a1 = qfma(v1 & 0x3F00u, x1.y, a1);
            a1 = qfma(v1 & 0x3F0000u, x1.z, a1);
            a1 = qfma((v1 >> 8) & 0x3F0000u, x1.w, a1);
            a2 = qfma(v2 & 0x3Fu, x2.x, a2);
            a2 = qfma(v2 & 0x3F00u, x2.y, a2);
            a2 = qfma(v2 & 0x3F0000u, x2.z, a2);
            a2 = qfma((v2 >> 8) & 0x3F0000u, x2.w, a2);
            a3 = qfma(v3 & 0x3Fu, x3.x, a3);
            a3 = qfma(v3 & 0x3F00u, x3.y, a3);
            a3 = qfma(v3 & 0x3F0000u, x3.z, a3);
            a3 = qfma((v3 >> 8) & 0x3F0000u, x3.w, a3);
        }
        // 16-element groups of this lane: 8h + 2t + c
        const float* X = xs16 + 8 * h + c;
        float r = sc0 * fmaf(d32, X[0], a0 * d64);
        r = fmaf(sc1, fmaf(d32, X[2], a1 * d64), r);
        r = fmaf(sc2, fmaf(d32, X[4], a2 * d64), r);
        r = fmaf(sc3, fmaf(d32, X[6], a3 * d64), r);
        return r;
    }
};

// ------------------------------------------------------------------ Q8_0
// 34-byte blocks: f16 d, 32 int8; value d*q.  A group of 8 blocks is 272
// bytes; quarter q holds blocks 2q, 2q+1 at byte 68q (4-byte aligned when
// the group is).  q+128 is extracted as an unsigned byte (XOR 0x80) and the
// 128*sum(x) offset removed per block.
// Lane element order: i = 32k + 4t + j -> element 64q + 32k + 4t + j;
// positions (0, 8, 16, 0).
struct FmtQ80 {
    static constexpr int SBB = 272;
    __host__ __device__ static int elem(int q, int i) { return 64 * q + i; }
    __host__ __device__ static int pos(int, int i) {
        // bit offsets {0, 8, 16, 0} by i % 4
        return static_cast<int>((0x00100800u >> (8 * (i & 3))) & 0xFFu);
    }
    __device__ __forceinline__ static float dot(const uint8_t* sb, int q, const float4* xq,
                                                const float* xs16) {
        const uint32_t* u = reinterpret_cast<const uint32_t*>(sb + 68 * q);
        uint32_t U[17];
#pragma unroll
        for (int k = 0; k < 17; ++k) U[k] = u[k];
        const float dA = f16_bits_to_f32(U[0]);
        const float dB = f16_bits_to_f32(U[8] >> 16);
        float aA = 0.f, aB = 0.f, aA2 = 0.f, aB2 = 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t wa = __funnelshift_r(U[t], U[t + 1], 16) ^ 0x80808080u;
            const uint32_t wb = U[9 + t] ^ 0x80808080u;
            const float4 xa = xq[t * 4 + q];
            const float4 xb = xq[(8 + t) * 4 + q];
            aA = qfma(wa & 0xFFu, xa.x, aA);
            aA2 = qfma(wa & 0xFF00u, xa.y, aA2);
            aA = qfma(wa & 0xFF0000u, xa.z, aA);
            aA2 = qfma(wa >> 24, xa.w, aA2);
            aB = qfma(wb & 0xFFu, xb.x, aB);
            aB2 = qfma(wb & 0xFF00u, xb.y, aB2);
            aB = qfma(wb & 0xFF0000u, xb.z, aB);
            aB2 = qfma(wb >> 24, xb.w, aB2);
        }
        aA += aA2;
        aB += aB2;
        const float XA = xs16[4 * q] + xs16[4 * q + 1];
        const float XB = xs16[4 * q + 2] + xs16[4 * q + 3];
        return dA * fmaf(aA, TWO64, -128.f * XA) + dB * fmaf(aB, TWO64, -128.f * XB);
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
    __host__ __device__ static int elem(int q, int i) {
        int k = i >> 5, t = (i >> 3) & 3, j = i & 7;
        int base = 32 * (2 * q + k);
        return j < 4 ? base + 4 * t + j : base + 16 + 4 * t + (j - 4);
    }
    __host__ __device__ static int pos(int q, int i) { return FmtQ4K::pos(q, i); }
    __device__ __forceinline__ static float dot(const uint8_t* sb, int q, const float4* xq,
                                                const float* xs16) {
        const uint32_t* u = reinterpret_cast<const uint32_t*>(sb + 36 * q);
        uint32_t U[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) U[k] = u[k];
        const float dA = f16_bits_to_f32(U[0]);
        const float dB = f16_bits_to_f32(U[4] >> 16);
        float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const uint32_t w = k == 0 ? __funnelshift_r(U[t], U[t + 1], 16) : U[5 + t];
                const uint32_t v = w >> 24;
                const float4 xl = xq[(8 * k + 2 * t) * 4 + q];
                const float4 xh = xq[(8 * k + 2 * t + 1) * 4 + q];
                float a = acc[k][0], b = acc[k][1];
                a = qfma(w & 0xFu, xl.x, a);
                b = qfma(w & 0xF00u, xl.y, b);
                a = qfma(w & 0xF0000u, xl.z, a);
                b = qfma(v & 0xFu, xl.w, b);
                a = qfma(w & 0xF0u, xh.x, a);
                b = qfma(w & 0xF000u, xh.y, b);
                a = qfma(w & 0xF00000u, xh.z, a);
                b = qfma(v & 0xF0u, xh.w, b);
                acc[k][0] = a;
                acc[k][1] = b;
            }
        }
        const float aA = acc[0][0] + acc[0][1], aB = acc[1][0] + acc[1][1];
        const float XA = xs16[4 * q] + xs16[4 * q + 1];
        const float XB = xs16[4 * q + 2] + xs16[4 * q + 3];
        return dA * fmaf(aA, TWO64, -8.f * XA) + dB * fmaf(aB, TWO64, -8.f * XB);
    }
};

}  // namespace qmoe
