// Device code shared by the batch-1 and batch decode kernels: layer
// descriptors, the router, and the fixed-point DP4A up-projection pieces.
#pragma once

#include "hs_common.cuh"

namespace hs {

// Bytes per 64-wide group in the shared-memory fixed-point x table: 128 B of
// split bytes + 16 B pad (conflict-free 128-bit loads).
constexpr int kXfStride = 144;

struct ExpertPtrs {
    const uint8_t* up_codes;   // [neurons][hidden/2]
    const uint32_t* up_sb;     // [neurons][hidden/64] (scale, bias)
    const uint8_t* dn_codes;   // [neurons][hidden/2] neuron-major
    const uint32_t* dn_sb;     // [neurons/64][hidden] (scale, bias)
    const float* up_off;       // [neurons] or null
};

struct LayerParams {
    ExpertPtrs routed[kMaxRouted];
    ExpertPtrs shared;
    long long stride[5];  // when uniform: byte strides of the 5 fields between experts
    int uniform;          // routed[e] = routed[0] + e * stride (no table lookup)
    int n_routed;
    int routed_neurons;
    int shared_neurons;   // 0 if no shared expert
    int hidden;
    int top_k;
};

// Pointers of routed expert e: by arithmetic when the experts are stacked at
// uniform strides (no dependent load), else from the table.
__device__ __forceinline__ ExpertPtrs routed_ptrs(const LayerParams& P, int e) {
    if (P.uniform) {
        ExpertPtrs b = P.routed[0];
        b.up_codes += e * P.stride[0];
        b.up_sb = reinterpret_cast<const uint32_t*>(reinterpret_cast<const char*>(b.up_sb) + e * P.stride[1]);
        b.dn_codes += e * P.stride[2];
        b.dn_sb = reinterpret_cast<const uint32_t*>(reinterpret_cast<const char*>(b.dn_sb) + e * P.stride[3]);
        if (b.up_off) b.up_off = reinterpret_cast<const float*>(reinterpret_cast<const char*>(b.up_off) + e * P.stride[4]);
        return b;
    }
    return P.routed[e];
}

// ------------------------------------------------------------------ router
// Top-k of n <= 128 logits (ties -> lower index) and a softmax over the chosen
// k <= 8, by one warp in registers.  Each logit becomes an order-preserving
// 32-bit key (-0 taken as +0).  Lane l sorts its keys l, l+32, l+64, l+96
// (key descending, index ascending); then k rounds of a warp-wide maximum of
// the lanes' heads (redux.sync), the lowest index among the lanes that hold
// it (a second redux), and a pop by the winning lane.  Lane 0 writes idx[k]
// and w[k].

__device__ __forceinline__ uint32_t topk_key(float f) {
    const uint32_t b = __float_as_uint(f + 0.f);   // -0 -> +0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float topk_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

__device__ __forceinline__ void topk_cx(uint32_t (&k)[4], int (&id)[4], int a, int b) {
    // order positions a < b best-first (larger key; equal keys: lower index)
    const bool sw = k[b] > k[a] || (k[b] == k[a] && id[b] < id[a]);
    const uint32_t ka = k[a], kb = k[b];
    const int ia = id[a], ib = id[b];
    k[a] = sw ? kb : ka; k[b] = sw ? ka : kb;
    id[a] = sw ? ib : ia; id[b] = sw ? ia : ib;
}

__device__ inline void warp_topk_softmax(const float* __restrict__ logits, int n, int k, int* idx, float* w) {
    const int lane = threadIdx.x & 31;
    uint32_t key[4];
    int id[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = lane + 32 * i;
        const bool real = e < n;
        key[i] = real ? topk_key(logits[e]) : 0u;   // no finite logit has key 0
        id[i] = real ? e : 1024 + e;
    }
    topk_cx(key, id, 0, 1); topk_cx(key, id, 2, 3); topk_cx(key, id, 0, 2); topk_cx(key, id, 1, 3); topk_cx(key, id, 1, 2);
    uint32_t sk[kMaxTopK];
    int si[kMaxTopK];
#pragma unroll
    for (int r = 0; r < kMaxTopK; ++r) {
        sk[r] = 0u;
        si[r] = 0;
        if (r < k) {
            const uint32_t mx = __reduce_max_sync(0xffffffffu, key[0]);
            const uint32_t win = __reduce_min_sync(0xffffffffu, key[0] == mx ? (uint32_t)id[0] : 0xffffffffu);
            sk[r] = mx;
            si[r] = (int)win;
            if ((uint32_t)id[0] == win) {   // pop this lane's head
                key[0] = key[1]; key[1] = key[2]; key[2] = key[3]; key[3] = 0u;
                id[0] = id[1]; id[1] = id[2]; id[2] = id[3]; id[3] = 4096;
            }
        }
    }
    if (lane == 0) {
        const float v0 = topk_value(sk[0]);
        float ex[kMaxTopK];
        float den = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) ex[j] = (j < k) ? expf(topk_value(sk[j]) - v0) : 0.f;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) den += ex[j];
        const float inv = 1.f / den;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
            if (j < k) { idx[j] = si[j]; w[j] = ex[j] * inv; }
    }
}

// ------------------------------------------------------------- up phase
// Dot products of the CTA's 64 up rows with x on the integer pipes.
// Thread (gc, r0) owns scale group gc (64 codes, 32 bytes) of every row
// r = r0 + S*i.  Its 64 activations are held as a 16-bit fixed-point copy
// with one exponent for the group, X_k = round(x_k * 2^(15-E)) with
// max|x_k| < 2^E, split into a signed high byte and an unsigned low byte
// (X = 256*H + L).  A bf16 x with |x| >= 2^(E-8) is represented exactly (its
// 8 significant bits fit); smaller ones are off by at most 2^(E-16).  Per
// group and row:
//   sum_k q_k X_k = 256 * dp4a(q, H) + dp4a(q, L)    (exact in int32)
// with the codes split into even/odd nibble bytes by one mask each.
struct XFixed {
    int hE[8], hO[8];          // high bytes of X for even / odd codes of word j
    unsigned lE[8], lO[8];     // low bytes
    float inv;                 // 2^(E-15) / 16 (the group dot products carry a factor 16)
    float xsum;                // sum of the 64 x values (fp32)
};

// Cooperative conversion of x into the fixed-point table: 4 threads per
// group of 64, thread q covering x[16q..16q+15] (code words 2q, 2q+1).  The
// group maximum and sum combine the 4 partials by a fixed 2-level tree.
// Threads first..blockDim-1 (whole warps) take the work items round-robin.
// E comes from the exponent field of the maximum (max < 2^E); rounding to the
// integer grid uses the 1.5 * 2^23 magic constant (exact: |x * 2^(15-E)| < 2^15).
__device__ __forceinline__ void convert_x_fixed(const uint16_t* x_s, int G, uint8_t* xf_s, float* xs_s, int first) {
    const int nthr = blockDim.x - first;
    for (int i0 = threadIdx.x - first; i0 - (int)(threadIdx.x & 31) < 4 * G; i0 += nthr) {
        // whole warps iterate together (the shuffles need all lanes); idle lanes work on item 0
        const bool act = i0 < 4 * G;
        const int i = act ? i0 : 0;
        const int grp = i >> 2, q = i & 3;
        const uint4 r0 = reinterpret_cast<const uint4*>(x_s + 64 * grp + 16 * q)[0];
        const uint4 r1 = reinterpret_cast<const uint4*>(x_s + 64 * grp + 16 * q)[1];
        const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        float xv[16];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            xv[2 * m] = __uint_as_float(w[m] << 16);
            xv[2 * m + 1] = __uint_as_float(w[m] & 0xffff0000u);
        }
        float mx = 0.f, sa = 0.f, sb = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m += 2) {
            mx = fmaxf(mx, fmaxf(fabsf(xv[m]), fabsf(xv[m + 1])));
            sa += xv[m];
            sb += xv[m + 1];
        }
        float sm = sa + sb;
        // the 4 threads of a group are adjacent lanes: fixed xor tree
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        sm += __shfl_xor_sync(0xffffffffu, sm, 1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        sm += __shfl_xor_sync(0xffffffffu, sm, 2);
        int e = (int)((__float_as_uint(mx) >> 23) & 0xff) - 126;  // mx < 2^e (mx normal)
        e = max(e, -100);                                          // zero / subnormal maxima
        const float scale = __int_as_float((127 + 15 - e) << 23);  // 2^(15-e)
        // words 2q, 2q+1: byte b of word j <-> x[8j + 2b] (even) and x[8j + 2b + 1] (odd)
        uint32_t hE[2], hO[2], lE[2], lO[2];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            hE[jj] = hO[jj] = lE[jj] = lO[jj] = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int X0 = __float_as_int(fmaf(xv[8 * jj + 2 * b], scale, 12582912.f)) - 0x4B400000;
                const int X1 = __float_as_int(fmaf(xv[8 * jj + 2 * b + 1], scale, 12582912.f)) - 0x4B400000;
                hE[jj] |= (uint32_t)((X0 >> 8) & 0xff) << (8 * b);
                lE[jj] |= (uint32_t)(X0 & 0xff) << (8 * b);
                hO[jj] |= (uint32_t)((X1 >> 8) & 0xff) << (8 * b);
                lO[jj] |= (uint32_t)(X1 & 0xff) << (8 * b);
            }
        }
        if (act) {
            uint8_t* tb = xf_s + grp * kXfStride + 8 * q;
            *reinterpret_cast<uint2*>(tb) = make_uint2(hE[0], hE[1]);
            *reinterpret_cast<uint2*>(tb + 32) = make_uint2(hO[0], hO[1]);
            *reinterpret_cast<uint2*>(tb + 64) = make_uint2(lE[0], lE[1]);
            *reinterpret_cast<uint2*>(tb + 96) = make_uint2(lO[0], lO[1]);
            if (q == 0) {
                xs_s[2 * grp] = __int_as_float((127 + e - 19) << 23);   // 2^(E-15) / 16
                xs_s[2 * grp + 1] = sm;
            }
        }
    }
}

__device__ __forceinline__ void load_x_fixed(const uint8_t* xf_s, const float* xs_s, int gc, XFixed& xf) {
    const uint4* p = reinterpret_cast<const uint4*>(xf_s + gc * kXfStride);
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = p[i];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        xf.hE[4 * i] = (int)v[i].x; xf.hE[4 * i + 1] = (int)v[i].y; xf.hE[4 * i + 2] = (int)v[i].z; xf.hE[4 * i + 3] = (int)v[i].w;
        xf.hO[4 * i] = (int)v[2 + i].x; xf.hO[4 * i + 1] = (int)v[2 + i].y; xf.hO[4 * i + 2] = (int)v[2 + i].z; xf.hO[4 * i + 3] = (int)v[2 + i].w;
        xf.lE[4 * i] = v[4 + i].x; xf.lE[4 * i + 1] = v[4 + i].y; xf.lE[4 * i + 2] = v[4 + i].z; xf.lE[4 * i + 3] = v[4 + i].w;
        xf.lO[4 * i] = v[6 + i].x; xf.lO[4 * i + 1] = v[6 + i].y; xf.lO[4 * i + 2] = v[6 + i].z; xf.lO[4 * i + 3] = v[6 + i].w;
    }
    xf.inv = xs_s[2 * gc];
    xf.xsum = xs_s[2 * gc + 1];
}

// Where the up phase leaves the partial dot product of (row r, group gc): the
// 4 bytes at word (gc/4 + r)%8 of the group's 32-byte code block.  A warp's
// stores (consecutive gc, one row) and the row sums' loads (8 rows x 4
// threads, groups q + 4i) then hit 32 distinct banks (for rows of
// 1344 bytes; other widths stay correct, with some conflicts).
__device__ __forceinline__ float* part_slot(uint8_t* codes_buf, int rowb, int r, int gc) {
    return reinterpret_cast<float*>(codes_buf + r * rowb + 32 * gc + 4 * (((gc >> 2) + r) & 7));
}

// 16 * sum_k q_k X_k over one scale group: 32 code bytes in two 16-byte
// halves (codes 8j+i in nibble i of word j; half 1 holds words 4..7).  Even
// codes are masked in place (q), odd codes too (16 q): no shifts; the factor
// 16 is carried by the even sums instead.  |16 T| < 2^28: exact in int32.
__device__ __forceinline__ int group_dot_fixed16(const uint4 c0, const uint4 c1, const XFixed& xf) {
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    int hE = 0, hO = 0;
    unsigned lE = 0, lO = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t ev = w[j] & 0x0F0F0F0Fu;   // q of codes 8j, 8j+2, 8j+4, 8j+6
        const uint32_t od = w[j] & 0xF0F0F0F0u;   // 16 q of codes 8j+1, ..., 8j+7
        asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(hE) : "r"(ev), "r"(xf.hE[j]));
        asm("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(hO) : "r"(od), "r"(xf.hO[j]));
        lE = __dp4a(ev, xf.lE[j], lE);
        lO = __dp4a(od, xf.lO[j], lO);
    }
    // 16 T = 16 (256 hE + lE) + (256 hO + lO), hO and lO already carrying 16
    return (hE * 256 + (int)lE) * 16 + hO * 256 + (int)lO;
}

// Reads the two 16-byte halves of group gc of a row, in an order that makes
// the 8-lane phases of a warp's 128-bit shared loads hit distinct banks.
__device__ __forceinline__ void load_group_codes(const uint8_t* row, int gc, uint4& c0, uint4& c1) {
    const int f = (gc >> 2) & 1;
    const uint4 a = *reinterpret_cast<const uint4*>(row + 32 * gc + 16 * f);
    const uint4 b = *reinterpret_cast<const uint4*>(row + 32 * gc + 16 * (f ^ 1));
    c0 = f ? b : a;
    c1 = f ? a : b;
}

}  // namespace hs
