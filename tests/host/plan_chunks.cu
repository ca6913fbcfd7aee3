// Host build of the streaming engine's chunk planner (plan_chunks in
// moe_ffn_gb300/csrc/stream.cuh) for the CPU tests: the geometry it returns
// for a format, a mode, a row shape and a stage budget.  Test
// infrastructure: the library does not use it.
#include <cstdint>

#include "../../moe_ffn_gb300/csrc/stream.cuh"

namespace {

// out: ok, runs, n_sbc, chunk_ks, chunk_sb, n_chunk, piece_stride,
//      slot_stride, stage_bytes, seg_bytes, sbb, rows (tile slots), wk
template <class F, int MODE>
int plan(int nb_seg, int n_kseg, int tail, int budget, int rows, int64_t* out) {
    using namespace qmoe;
    StreamParams p = {};
    p.nb_seg = nb_seg;
    p.n_kseg = n_kseg;
    p.tail = tail;
    const bool ok = rows > 0 ? plan_chunks<F, MODE>(p, budget, rows) : plan_chunks<F, MODE>(p, budget);
    int r = rows;
    if (MODE != MODE_QMV || r > ModeGeom<MODE>::ROWS || r < 1) r = ModeGeom<MODE>::ROWS;
    const int64_t v[13] = {ok ? 1 : 0, p.runs, p.n_sbc, p.chunk_ks, p.chunk_sb, p.n_chunk,
                           p.piece_stride, p.slot_stride, p.stage_bytes, seg_bytes<F>(p),
                           F::SBB, r, ModeGeom<MODE>::WK};
    for (int i = 0; i < 13; ++i) out[i] = v[i];
    return 0;
}

template <class F>
int by_mode(int mode, int nb_seg, int n_kseg, int tail, int budget, int rows, int64_t* out) {
    using namespace qmoe;
    switch (mode) {
    case MODE_QMV: return plan<F, MODE_QMV>(nb_seg, n_kseg, tail, budget, rows, out);
    case MODE_GATEUP: return plan<F, MODE_GATEUP>(nb_seg, n_kseg, tail, budget, rows, out);
    case MODE_DOWN: return plan<F, MODE_DOWN>(nb_seg, n_kseg, tail, budget, rows, out);
    default: return -1;
    }
}

}  // namespace

extern "C" int plan_chunks_host(int fmt, int mode, int nb_seg, int n_kseg, int tail, int budget,
                                int rows, int64_t* out) {
    using namespace qmoe;
    switch (fmt) {
    case QT_Q8_0: return by_mode<FmtQ80>(mode, nb_seg, n_kseg, tail, budget, rows, out);
    case QT_Q4_0: return by_mode<FmtQ40>(mode, nb_seg, n_kseg, tail, budget, rows, out);
    case QT_Q4_K: return by_mode<FmtQ4K>(mode, nb_seg, n_kseg, tail, budget, rows, out);
    case QT_Q5_K: return by_mode<FmtQ5K>(mode, nb_seg, n_kseg, tail, budget, rows, out);
    case QT_Q6_K: return by_mode<FmtQ6K>(mode, nb_seg, n_kseg, tail, budget, rows, out);
    default: return -1;
    }
}
