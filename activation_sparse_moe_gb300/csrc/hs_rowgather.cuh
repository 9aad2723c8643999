// Row-gather plan of one (expert, token tile) for the prefill's down product
// (HS_PREFILL_ROW_GATHER).  "Skipping dead neurons..." section "What we do
// instead": per token tile, the rows live for any of its tokens are gathered
// into one dense product.
//
// The down product of a token tile multiplies H[tokens][neurons] by the
// expert's neuron-major down weights.  With the dead neurons scattered, whole
// 64-neuron tiles are seldom dead for every token of a tile, so instead the
// union-live neurons of the tile are packed into dense k-steps of 64 entries.
// Each group's live neurons (ascending) are padded to a multiple of 8 entries
// (the dequantiser's 8-row blocks never straddle two groups), and a k-step
// holds the entries of at most two groups: entries [0, 8 * split8) use the
// (scale, bias) slab of group gA, entries [8 * split8, 64) that of group gB.
// A padding entry (0xFFFF) reads any valid weight row against h = 0.
#pragma once
#include <cstdint>

#ifdef __CUDACC__
#define RG_HD __host__ __device__ inline
#else
#define RG_HD inline
#endif

namespace rowgather {

constexpr uint16_t kPad = 0xFFFFu;

RG_HD uint32_t ksd_pack(int gA, int gB, int split8) {
    return (uint32_t)gA | ((uint32_t)gB << 8) | ((uint32_t)split8 << 16);
}
RG_HD int ksd_gA(uint32_t d) { return (int)(d & 0xFFu); }
RG_HD int ksd_gB(uint32_t d) { return (int)((d >> 8) & 0xFFu); }
RG_HD int ksd_split8(uint32_t d) { return (int)((d >> 16) & 0xFFu); }

RG_HD int popc64(uint64_t v) {
#ifdef __CUDA_ARCH__
    return __popcll(v);
#else
    return __builtin_popcountll(v);
#endif
}

// Plans the k-steps of one tile from its union-live masks (mask[g] bit i =
// neuron 64 g + i is live for some token of the tile), NG <= 64 groups.
// Writes ksd[0 .. nks) and grp_ofs[g] (first entry of group g, -1 for a dead
// group).  Returns nks, or -1 when the packing would need more k-steps than
// NG (the caller then takes the identity plan: k-step j = group j).
RG_HD int plan_tile(const uint64_t* mask, int NG, uint32_t* ksd, int* grp_ofs) {
    int ks = 0, f = 0, gA = -1, gB = -1, split8 = 8;
    for (int g = 0; g < NG; ++g) {
        const int c = popc64(mask[g]);
        grp_ofs[g] = -1;
        if (c == 0) continue;
        const int p = (c + 7) & ~7;
        // a third group may not enter a k-step: close it (its tail is padding)
        if (f > 0 && gA != gB) {
            if (ks >= NG) return -1;
            ksd[ks++] = ksd_pack(gA, gB, split8);
            f = 0;
        }
        grp_ofs[g] = 64 * ks + f;
        int left = p;
        while (left > 0) {
            if (f == 0) {
                gA = gB = g;
                split8 = 8;
            } else if (g != gB) {
                gB = g;
                split8 = f / 8;
            }
            const int take = left < 64 - f ? left : 64 - f;
            f += take;
            left -= take;
            if (f == 64) {
                if (ks >= NG) return -1;
                ksd[ks++] = ksd_pack(gA, gB, split8);
                f = 0;
            }
        }
    }
    if (f > 0) {
        if (ks >= NG) return -1;
        ksd[ks++] = ksd_pack(gA, gB, split8);
    }
    return ks;
}

// The identity plan: k-step j is group j, every neuron an entry.
RG_HD int plan_identity(int NG, uint32_t* ksd, int* grp_ofs) {
    for (int g = 0; g < NG; ++g) {
        ksd[g] = ksd_pack(g, g, 8);
        grp_ofs[g] = 64 * g;
    }
    return NG;
}

// Stored position of entry i of a k-step: inside each block of 8 entries the
// order e0 e4 e1 e5 e2 e6 e3 e7 (the order in which the dequantiser yields
// nibble pairs; h is stored the same way).
RG_HD int stored_pos(int i) {
    const int i8 = i & 7;
    return (i & ~7) | (i8 < 4 ? 2 * i8 : 2 * (i8 - 4) + 1);
}

}  // namespace rowgather
