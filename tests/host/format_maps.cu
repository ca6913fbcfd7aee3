// Host build of the lane maps of the decoders (moe_ffn_gb300/csrc/formats.cuh)
// for the CPU tests: element order, x-table slots, field positions.  Test
// infrastructure: the library does not use it.
#include <cstdint>

#include "../../moe_ffn_gb300/csrc/formats.cuh"

template <class F>
static void maps(int* elem, int* xslot, int* pos, int* pos8) {
    for (int q = 0; q < 4; ++q)
        for (int i = 0; i < 64; ++i) {
            elem[q * 64 + i] = F::elem(q, i);
            pos[q * 64 + i] = F::pos(q, i);
        }
    for (int e4 = 0; e4 < 64; ++e4) xslot[e4] = F::xslot(e4);
    *pos8 = F::POS8 ? 1 : 0;
}

extern "C" int fmt_maps(int fmt, int* elem, int* xslot, int* pos, int* pos8) {
    using namespace qmoe;
    switch (fmt) {
    case QT_Q8_0: maps<FmtQ80>(elem, xslot, pos, pos8); return 0;
    case QT_Q4_0: maps<FmtQ40>(elem, xslot, pos, pos8); return 0;
    case QT_Q4_K: maps<FmtQ4K>(elem, xslot, pos, pos8); return 0;
    case QT_Q5_K: maps<FmtQ5K>(elem, xslot, pos, pos8); return 0;
    case QT_Q6_K: maps<FmtQ6K>(elem, xslot, pos, pos8); return 0;
    default: return -1;
    }
}
