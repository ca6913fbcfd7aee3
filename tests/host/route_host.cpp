// Host build of the device routing rule (moe_ffn_gb300/csrc/route.cuh), for
// the CPU tests: the ranking keys, the rank count and the non-finite rule,
// composed as the kernels compose them (every expert's rank counted against
// all others; slot r takes the expert of rank r; weights from the
// top-ranked logit).  Test infrastructure: the library does not use it.
#include <cmath>
#include <cstdint>
#include <vector>

#include "../../moe_ffn_gb300/csrc/route.cuh"

extern "C" int route_host(const float* logits, int E, int k, int renorm, int32_t* idx, float* w,
                          int32_t* ranks) {
    using namespace qmoe;
    if (E <= 0 || k <= 0 || k > E) return -1;
    std::vector<uint32_t> key(E);
    for (int e = 0; e < E; ++e) key[e] = route_key(logits[e]);
    for (int s = 0; s < k; ++s) idx[s] = -1;
    for (int e = 0; e < E; ++e) {
        int rank = 0;
        for (int u = 0; u < E; ++u) rank += route_before(key[u], u, key[e], e) ? 1 : 0;
        ranks[e] = rank;
        if (rank < k) idx[rank] = e;
    }
    bool bad = false;
    for (int s = 0; s < k; ++s) idx[s] = route_clamp(idx[s], E, &bad);
    const float lmax = route_key_value(key[idx[0]]);
    float z = 0.f;
    if (renorm) {
        for (int s = 0; s < k; ++s) z += std::exp(route_key_value(key[idx[s]]) - lmax);
    } else {
        for (int e = 0; e < E; ++e) z += std::exp(route_key_value(key[e]) - lmax);
    }
    const bool degen = route_degenerate(lmax);
    for (int s = 0; s < k; ++s) {
        w[s] = std::exp(route_key_value(key[idx[s]]) - lmax) / z;
        if (degen) {
            idx[s] = s;
            w[s] = std::nanf("");
        }
    }
    return bad ? 1 : 0;
}

// The key itself, for direct checks of the order.
extern "C" uint32_t route_key_host(float v) { return qmoe::route_key(v); }
extern "C" float route_key_value_host(uint32_t k) { return qmoe::route_key_value(k); }
