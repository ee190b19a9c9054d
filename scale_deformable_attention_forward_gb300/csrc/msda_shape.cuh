// msda_shape.cuh -- how many lanes serve one (b, q, h) row, and how many
// 16-byte channel chunks each lane owns.
#pragma once

#include <cuda_bf16.h>

// Preferred lanes per row.  One load instruction of a group should cover a
// corner's whole channel row (L1 resolves about one distinct 128-byte line per
// clock, so splitting a line over several instructions costs lookups), and in
// the backward one atomic instruction should cover a whole accumulator line.
#ifndef MSDA_FWD_LANES
#define MSDA_FWD_LANES 8
#endif
#ifndef MSDA_BWD_LANES
#define MSDA_BWD_LANES 8
#endif

namespace msda {

// Elements per lane access: 4 channels per lane for both dtypes.  A group of
// 8 lanes then covers a 32-channel corner row with one load instruction (L1
// resolves about one distinct 128-byte line per clock whatever part of it an
// instruction reads, so 8-byte bfloat16 loads cost what 16-byte ones do), the
// forward sums the groups' partial outputs over few shuffles, and in the
// backward one red.global.add.v4.f32 per lane makes a group's atomics cover
// whole 128-byte lines of the binary32 accumulator.
template <typename T> struct VecWidth { static constexpr int value = 4; };
template <typename T> struct BwdVecWidth { static constexpr int value = 4; };

constexpr int pow2ceil(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

// (G, NCH) for `chunks` channel chunks per row and a preferred G: G starts at
// min(preferred, chunks rounded up to a power of two) and doubles until every
// lane owns at most 8 chunks; NCH is the per-lane count rounded up to a power
// of two.  Rows with more than 256 chunks are not supported.
struct Shape {
    int G, NCH;
};
constexpr Shape select_shape(int chunks, int preferred) {
    const int c = chunks < 1 ? 1 : chunks;
    int G = pow2ceil(c) < preferred ? pow2ceil(c) : preferred;
    while ((c + G - 1) / G > 8 && G < 32) G <<= 1;
    return Shape{G, pow2ceil((c + G - 1) / G)};
}
// Shapes that get kernels specialised for padding and backward outputs; the
// others (wide rows: C_h above 64 binary32 / 128 bfloat16 channels) get one
// kernel that reads both at run time.
constexpr bool specialised_shape(int G, int NCH) { return G <= 8 && NCH <= 2; }

constexpr bool reachable(int G, int NCH, int preferred) {
    for (int c = 1; c <= 256; ++c) {
        const Shape s = select_shape(c, preferred);
        if (s.G == G && s.NCH == NCH) return true;
    }
    return false;
}

}  // namespace msda
