// Tile scheduling shared by the persistent FFMA and TF32 kernels: the grouped
// tile raster, and the sequence of work items of one worker (data-parallel
// units, then its share of a stream-K span). A worker is a CTA, or a CTA pair
// working on the two halves of one tile (the TF32 pair kernel).
//
// Params (FfmaParams or Tf32Params) provide: tiles_m, tiles_n, units, splits,
// kblocks, sk_tiles, sk_grid. Units [0, units) are u = tile * splits + slice;
// tiles [units / splits, units / splits + sk_tiles) form the stream-K span of
// S = sk_tiles * kblocks k-blocks, of which worker g (< sk_grid = G) takes
// [g S / G, (g + 1) S / G). A tile inside one worker's range is finished by
// it; a tile shared by several workers gets one tile-packed partial from each,
// at slot 2g for the worker's first span tile and 2g + 1 for its last, which
// the stream-K reduction adds in worker (= k) order. The covering workers of
// span tile t are ((t kb + 1) G - 1) / S .. ((t + 1) kb G - 1) / S.
#pragma once

namespace sgemm_impl {

constexpr int kGroupM = 16;  // tile rows per raster group (L2 reuse of A and B)

// Tile index t -> (tile row, tile column): tiles run in groups of kGroupM tile
// rows, column by column, so concurrently running CTAs share B columns and A
// rows in L2.
__device__ __forceinline__ void decode_tile(int tiles_m, int tiles_n, int t, int &tm, int &tn)
{
    const int per_group = kGroupM * tiles_n;
    const int g = t / per_group;
    const int first_m = g * kGroupM;
    const int gsize = min(tiles_m - first_m, kGroupM);
    const int r = t - g * per_group;
    tm = first_m + r % gsize;
    tn = r / gsize;
}

// Where a work item's result goes: alpha/beta into C, a split-K slice (idx =
// slice), or a stream-K partial tile (idx = slot).
enum : int { kToC = 0, kToSplit = 1, kToPartial = 2 };

struct Work {
    int t, tm, tn, kb0, kb1, dest, idx;
};

// Item i of worker g's work (of G workers): first its units (u = g + i * G),
// then the pieces of its stream-K range, one per tile the range touches.
// Computed from i alone, so callers keep only i live across a mainloop, and
// every role of a CTA (copy issue, compute, epilogue) walks the same sequence.
// A worker is a CTA, or a CTA pair that shares its tiles. Returns false past
// the end.
template <class P>
__device__ __forceinline__ bool work_at_g(const P &p, int i, Work &w, int g, int G)
{
    const int n_units = g < p.units ? (p.units - g + G - 1) / G : 0;
    if (i < n_units) {
        const int u = g + i * G;
        const int ks = u % p.splits;
        w.t = u / p.splits;
        decode_tile(p.tiles_m, p.tiles_n, w.t, w.tm, w.tn);
        w.kb0 = static_cast<int>((static_cast<long long>(ks) * p.kblocks) / p.splits);
        w.kb1 = static_cast<int>((static_cast<long long>(ks + 1) * p.kblocks) / p.splits);
        w.dest = p.splits > 1 ? kToSplit : kToC;
        w.idx = ks;
        return true;
    }
    if (p.sk_tiles <= 0 || g >= p.sk_grid) return false;
    const long long S = static_cast<long long>(p.sk_tiles) * p.kblocks;
    const long long b0 = static_cast<long long>(g) * S / p.sk_grid;
    const long long b1 = static_cast<long long>(g + 1) * S / p.sk_grid;
    const int j = i - n_units;
    const long long rel = b0 / p.kblocks + j;
    const long long tile_start = rel * p.kblocks;
    const long long seg0 = j == 0 ? b0 : tile_start;
    if (seg0 >= b1) return false;
    const long long seg1 = b1 < tile_start + p.kblocks ? b1 : tile_start + p.kblocks;
    w.t = p.units / p.splits + static_cast<int>(rel);
    decode_tile(p.tiles_m, p.tiles_n, w.t, w.tm, w.tn);
    w.kb0 = static_cast<int>(seg0 - tile_start);
    w.kb1 = static_cast<int>(seg1 - tile_start);
    // a tile inside this CTA's range needs no partial
    w.dest = (w.kb0 == 0 && w.kb1 == p.kblocks) ? kToC : kToPartial;
    w.idx = 2 * g + (j == 0 ? 0 : 1);
    return true;
}

// Worker = this CTA.
template <class P>
__device__ __forceinline__ bool work_at(const P &p, int i, Work &w)
{
    return work_at_g(p, i, w, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x));
}

}  // namespace sgemm_impl
