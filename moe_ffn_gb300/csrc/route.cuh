// route.cuh — the ranking rule and weights of the on-device routing, shared
// by every MoE path (the single-token fused kernel, the separate-kernel
// form, the batched decode kernel and the many-token top-k kernel) and
// compiled for the host as well, so the rule can be checked on a CPU.
//
// The step is "softmax, top-k, renormalize" of "aprender-serve 0.70.2 —
// forward_qwen3_moe_resident.rs" (module doc, moe_layer; last_routes keeps
// rank order): the k largest softmax probabilities of the E router logits,
// ties to the lower expert index, weights p_s / sum over the k selected (or
// the probabilities themselves without renormalisation).
//
// Ranking on a total order.  A float comparison is false both ways when
// either side is NaN, so ranks counted with it need not be a permutation:
// some of the k slots would never be written and an uninitialised expert
// index would then address the stacks.  Here every logit maps to a 32-bit
// key whose unsigned order is total:
//     NaN (any sign or payload)  >  +Inf  >  finite values  >  -Inf,
// with -0 ranking as +0 and equal keys broken by the lower expert index.
// (key, index) pairs are then strictly ordered, so the ranks of the E
// experts are a permutation of 0..E-1 and each of the k slots is written
// exactly once.  No key is 0, which the batched kernel uses to mark a taken
// expert.
//
// Non-finite logits.  The softmax probabilities are all NaN when a logit is
// NaN or +Inf, or when every logit is -Inf (exp(inf - inf), 0/0); the
// selection of "the k largest" is then undefined.  This library takes the
// reading under which the stable ranking of NaN probabilities keeps the
// experts in index order: the route is experts 0, 1, ..., k-1, each with a
// NaN weight, and the layer's output becomes NaN.  That case is exactly the
// one where the top-ranked logit is not finite.  A -Inf logit beside finite
// ones has probability 0 and ranks last.
#pragma once
#include <cstdint>
#include <cstring>

#if defined(__CUDACC__)
#define QMOE_HD __host__ __device__ __forceinline__
#else
#define QMOE_HD inline
#endif

namespace qmoe {

QMOE_HD uint32_t float_bits(float v) {
#if defined(__CUDA_ARCH__)
    return __float_as_uint(v);
#else
    uint32_t b;
    std::memcpy(&b, &v, 4);
    return b;
#endif
}

QMOE_HD float bits_float(uint32_t b) {
#if defined(__CUDA_ARCH__)
    return __uint_as_float(b);
#else
    float v;
    std::memcpy(&v, &b, 4);
    return v;
#endif
}

// The ranking key of a logit (larger key = ranked first).
QMOE_HD uint32_t route_key(float v) {
    uint32_t b = float_bits(v);
    if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0xFFFFFFFFu;  // NaN
    if ((b << 1) == 0u) b = 0u;                               // -0 ranks as +0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The logit a key stands for (NaN for the NaN key, +0 for a zero).
QMOE_HD float route_key_value(uint32_t k) {
    return bits_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Whether expert u (key ku) ranks before expert e (key ke).
QMOE_HD bool route_before(uint32_t ku, int u, uint32_t ke, int e) {
    return ku > ke || (ku == ke && u < e);
}

// The route is undefined (all probabilities NaN) when the top-ranked logit
// is not finite: see the header comment.
QMOE_HD bool route_degenerate(float top_logit) {
    return !(top_logit <= 3.402823466e38f && top_logit >= -3.402823466e38f);  // NaN, +-Inf
}

// An expert index clamped into [0, E).  The rule above writes every slot, so
// a clamp never fires; it keeps a broken invariant from forming an address
// outside the stacks, and reports it (*fired).
QMOE_HD int route_clamp(int e, int E, bool* fired) {
    if (e >= 0 && e < E) return e;
    *fired = true;
    return 0;
}

}  // namespace qmoe
