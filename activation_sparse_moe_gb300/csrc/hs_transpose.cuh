// Transpose of a 32 x 32 matrix of 4-bit elements held by one warp: lane l
// holds row l as 4 words (column c at bits 4(c % 8) of word c / 8); afterwards
// lane l holds column l in the same form.  Five exchange stages s = 16, 8, 4,
// 2, 1: an element whose row and column differ in bit s moves to lane l ^ s
// and column c ^ s (after all five, (l, c) -> (c, l)).  At each stage a lane
// packs the half it gives away into two words, swaps them with lane l ^ s and
// unpacks the two words it receives into the half it gave away.  The packing
// and unpacking are plain bit moves, shared by the device code and host-side
// checks.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define HS_HD __host__ __device__ __forceinline__
#else
#define HS_HD inline
#endif

namespace hs {

HS_HD uint32_t hs_byte_perm(uint32_t x, uint32_t y, uint32_t sel) {
#if defined(__CUDA_ARCH__)
    return __byte_perm(x, y, sel);
#else
    const uint64_t v = (uint64_t)x | ((uint64_t)y << 32);
    uint32_t r = 0;
    for (int i = 0; i < 4; ++i) r |= (uint32_t)((v >> (8 * ((sel >> (4 * i)) & 7))) & 0xffu) << (8 * i);
    return r;
#endif
}

// The two words lane `lane` gives away at stage s.
HS_HD void nib_tr_pack(const uint32_t (&a)[4], int lane, int s, uint32_t (&x)[2]) {
    const bool top = (lane & s) == 0;
    switch (s) {
        case 16: x[0] = top ? a[2] : a[0]; x[1] = top ? a[3] : a[1]; break;
        case 8: x[0] = top ? a[1] : a[0]; x[1] = top ? a[3] : a[2]; break;
        case 4:
            for (int i = 0; i < 2; ++i)
                x[i] = top ? (a[2 * i] >> 16) | (a[2 * i + 1] & 0xffff0000u) : (a[2 * i] & 0xffffu) | (a[2 * i + 1] << 16);
            break;
        case 2:
            for (int i = 0; i < 2; ++i) x[i] = hs_byte_perm(a[2 * i], a[2 * i + 1], top ? 0x7531u : 0x6420u);
            break;
        default:  // 1
            for (int i = 0; i < 2; ++i)
                x[i] = top ? ((a[2 * i] >> 4) & 0x0f0f0f0fu) | (a[2 * i + 1] & 0xf0f0f0f0u)
                           : (a[2 * i] & 0x0f0f0f0fu) | ((a[2 * i + 1] << 4) & 0xf0f0f0f0u);
            break;
    }
}

// Puts the two words received from lane `lane ^ s` into the half given away.
HS_HD void nib_tr_unpack(uint32_t (&a)[4], int lane, int s, const uint32_t (&y)[2]) {
    const bool top = (lane & s) == 0;
    switch (s) {
        case 16:
            if (top) { a[2] = y[0]; a[3] = y[1]; } else { a[0] = y[0]; a[1] = y[1]; }
            break;
        case 8:
            if (top) { a[1] = y[0]; a[3] = y[1]; } else { a[0] = y[0]; a[2] = y[1]; }
            break;
        case 4:
            for (int i = 0; i < 2; ++i) {
                if (top) {
                    a[2 * i] = (a[2 * i] & 0xffffu) | (y[i] << 16);
                    a[2 * i + 1] = (a[2 * i + 1] & 0xffffu) | (y[i] & 0xffff0000u);
                } else {
                    a[2 * i] = (a[2 * i] & 0xffff0000u) | (y[i] & 0xffffu);
                    a[2 * i + 1] = (a[2 * i + 1] & 0xffff0000u) | (y[i] >> 16);
                }
            }
            break;
        case 2:
            for (int i = 0; i < 2; ++i) {
                a[2 * i] = hs_byte_perm(a[2 * i], y[i], top ? 0x5240u : 0x3514u);
                a[2 * i + 1] = hs_byte_perm(a[2 * i + 1], y[i], top ? 0x7260u : 0x3716u);
            }
            break;
        default:  // 1
            for (int i = 0; i < 2; ++i) {
                if (top) {
                    a[2 * i] = (a[2 * i] & 0x0f0f0f0fu) | ((y[i] << 4) & 0xf0f0f0f0u);
                    a[2 * i + 1] = (a[2 * i + 1] & 0x0f0f0f0fu) | (y[i] & 0xf0f0f0f0u);
                } else {
                    a[2 * i] = (a[2 * i] & 0xf0f0f0f0u) | (y[i] & 0x0f0f0f0fu);
                    a[2 * i + 1] = (a[2 * i + 1] & 0xf0f0f0f0u) | ((y[i] >> 4) & 0x0f0f0f0fu);
                }
            }
            break;
    }
}

#if defined(__CUDACC__)
// Stages 4, 2 and 1 only: for data loaded so that the word-level stages (16
// and 8) are already done, i.e. lane l holds, as word k, word l / 8 of row
// 8k + l % 8.  The same bit moves as nib_tr_pack / nib_tr_unpack, with the
// lane's side of each exchange folded into per-lane byte selectors and shift
// counts (computed once), so each move is a single PRMT, SHF or LOP3.
struct NibTrLane {
    uint32_t p4, u4a, u4b, p2, u2a, u2b;  // byte selectors of stages 4 and 2
    uint32_t k1, sp0, sp1, su0, su1;      // stage 1: kept nibbles and shift counts
};

__device__ __forceinline__ NibTrLane nib_tr_lane() {
    const int lane = threadIdx.x & 31;
    NibTrLane c;
    const bool t4 = (lane & 4) == 0, t2 = (lane & 2) == 0, t1 = (lane & 1) == 0;
    c.p4 = t4 ? 0x7632u : 0x5410u;
    c.u4a = t4 ? 0x5410u : 0x3254u;
    c.u4b = t4 ? 0x7610u : 0x3276u;
    c.p2 = t2 ? 0x7531u : 0x6420u;
    c.u2a = t2 ? 0x5240u : 0x3514u;
    c.u2b = t2 ? 0x7260u : 0x3716u;
    c.k1 = t1 ? 0x0f0f0f0fu : 0xf0f0f0f0u;
    c.sp0 = t1 ? 4u : 0u;    // pack: first word >> sp0, second word << sp1
    c.sp1 = t1 ? 0u : 4u;
    c.su0 = t1 ? 4u : 0u;    // unpack: received << su0 into the first word, >> su1 into the second
    c.su1 = t1 ? 0u : 4u;
    return c;
}

__device__ __forceinline__ void nib_transpose32_in_words(uint32_t (&a)[4], const NibTrLane& c) {
    uint32_t x0, x1, y0, y1;
    // stage 4: 16-bit halves
    x0 = __byte_perm(a[0], a[1], c.p4);
    x1 = __byte_perm(a[2], a[3], c.p4);
    y0 = __shfl_xor_sync(0xffffffffu, x0, 4);
    y1 = __shfl_xor_sync(0xffffffffu, x1, 4);
    a[0] = __byte_perm(a[0], y0, c.u4a);
    a[1] = __byte_perm(a[1], y0, c.u4b);
    a[2] = __byte_perm(a[2], y1, c.u4a);
    a[3] = __byte_perm(a[3], y1, c.u4b);
    // stage 2: bytes
    x0 = __byte_perm(a[0], a[1], c.p2);
    x1 = __byte_perm(a[2], a[3], c.p2);
    y0 = __shfl_xor_sync(0xffffffffu, x0, 2);
    y1 = __shfl_xor_sync(0xffffffffu, x1, 2);
    a[0] = __byte_perm(a[0], y0, c.u2a);
    a[1] = __byte_perm(a[1], y0, c.u2b);
    a[2] = __byte_perm(a[2], y1, c.u2a);
    a[3] = __byte_perm(a[3], y1, c.u2b);
    // stage 1: nibbles
    x0 = ((a[0] >> c.sp0) & 0x0f0f0f0fu) | ((a[1] << c.sp1) & 0xf0f0f0f0u);
    x1 = ((a[2] >> c.sp0) & 0x0f0f0f0fu) | ((a[3] << c.sp1) & 0xf0f0f0f0u);
    y0 = __shfl_xor_sync(0xffffffffu, x0, 1);
    y1 = __shfl_xor_sync(0xffffffffu, x1, 1);
    a[0] = (a[0] & c.k1) | ((y0 << c.su0) & ~c.k1);
    a[1] = (a[1] & c.k1) | ((y0 >> c.su1) & ~c.k1);
    a[2] = (a[2] & c.k1) | ((y1 << c.su0) & ~c.k1);
    a[3] = (a[3] & c.k1) | ((y1 >> c.su1) & ~c.k1);
}

__device__ __forceinline__ void nib_transpose32(uint32_t (&a)[4]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 16; s; s >>= 1) {
        uint32_t x[2], y[2];
        nib_tr_pack(a, lane, s, x);
        y[0] = __shfl_xor_sync(0xffffffffu, x[0], s);
        y[1] = __shfl_xor_sync(0xffffffffu, x[1], s);
        nib_tr_unpack(a, lane, s, y);
    }
}
#endif

}  // namespace hs
