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
// it (a second redux), and a pop by the winning lane.  Every lane then forms
// the softmax, and lane j < k stores choice j (idx[j], w[j]) and returns it.
// The whole routine is straight-line code for every lane (the pop is a
// select; no block runs on one lane only): an earlier form in which lane 0
// alone stored all k choices gave -1 for the 8th index at k = 8 in kernels
// whose other lanes then read the choices back, though not elsewhere.

struct TopkPick {
    int idx;    // expert of this lane's choice (lanes >= k: -1)
    float w;    // its softmax weight (lanes >= k: 0)
};

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

__device__ inline TopkPick warp_topk_softmax(const float* __restrict__ logits, int n, int k, int* idx, float* w) {
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
        if (r < k) {   // k is the same for the whole warp
            const uint32_t mx = warp_max_u32(key[0]);
            const uint32_t win = warp_min_u32(key[0] == mx ? (uint32_t)id[0] : 0xffffffffu);
            sk[r] = mx;
            si[r] = (int)win;
            const bool pop = (uint32_t)id[0] == win;   // the winner drops its head
            key[0] = pop ? key[1] : key[0]; key[1] = pop ? key[2] : key[1]; key[2] = pop ? key[3] : key[2];
            key[3] = pop ? 0u : key[3];
            id[0] = pop ? id[1] : id[0]; id[1] = pop ? id[2] : id[1]; id[2] = pop ? id[3] : id[2];
            id[3] = pop ? 4096 : id[3];
        }
    }
    const float v0 = topk_value(sk[0]);
    float den = 0.f, mine = 0.f;
    int mine_i = -1;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        const float ex = j < k ? expf(topk_value(sk[j]) - v0) : 0.f;
        den += ex;
        if (j == lane) { mine = ex; mine_i = si[j]; }
    }
    TopkPick p{-1, 0.f};
    if (lane < k) {
        p.idx = mine_i;
        p.w = mine * (1.f / den);
        idx[lane] = p.idx;
        w[lane] = p.w;
    }
    return p;
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

// The fixed-point copy is built from quarters of a group: 16 bf16 values
// x[16q..16q+15] in 8 words (code words 2q, 2q+1).
// Maximum magnitude and sum of one quarter (even and odd elements in two
// ordered chains, then added).
__device__ __forceinline__ void x_quarter_stats(const uint32_t (&w)[8], float& mx, float& sm) {
    float sa = 0.f, sb = 0.f;
    mx = 0.f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const float x0 = __uint_as_float(w[m] << 16), x1 = __uint_as_float(w[m] & 0xffff0000u);
        mx = fmaxf(mx, fmaxf(fabsf(x0), fabsf(x1)));
        sa += x0;
        sb += x1;
    }
    sm = sa + sb;
}

// E from the exponent field of the group maximum (max < 2^E).
__device__ __forceinline__ int x_group_exp(float mx) {
    const int e = (int)((__float_as_uint(mx) >> 23) & 0xff) - 126;  // mx normal
    return max(e, -100);                                            // zero / subnormal maxima
}

// Words 2q, 2q+1 of the fixed-point copy: byte b of word j <-> x[8j + 2b]
// (even) and x[8j + 2b + 1] (odd).  Rounding to the integer grid uses the
// 1.5 * 2^23 magic constant (exact: |x * 2^(15-E)| < 2^15).
__device__ __forceinline__ void x_quarter_fixed(const uint32_t (&w)[8], int e, uint32_t (&hE)[2], uint32_t (&hO)[2],
                                                uint32_t (&lE)[2], uint32_t (&lO)[2]) {
    const float scale = __int_as_float((127 + 15 - e) << 23);  // 2^(15-e)
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        hE[jj] = hO[jj] = lE[jj] = lO[jj] = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t v = w[4 * jj + b];
            const int X0 = __float_as_int(fmaf(__uint_as_float(v << 16), scale, 12582912.f)) - 0x4B400000;
            const int X1 = __float_as_int(fmaf(__uint_as_float(v & 0xffff0000u), scale, 12582912.f)) - 0x4B400000;
            hE[jj] |= (uint32_t)((X0 >> 8) & 0xff) << (8 * b);
            lE[jj] |= (uint32_t)(X0 & 0xff) << (8 * b);
            hO[jj] |= (uint32_t)((X1 >> 8) & 0xff) << (8 * b);
            lO[jj] |= (uint32_t)(X1 & 0xff) << (8 * b);
        }
    }
}

// 2^(E-15) / 16: the factor that turns a group dot product into x units.
__device__ __forceinline__ float x_group_inv(int e) { return __int_as_float((127 + e - 19) << 23); }

// Cooperative conversion of x into the fixed-point table: 4 threads per
// group of 64, thread q covering quarter q.  The group maximum and sum
// combine the 4 partials by a fixed 2-level tree (lanes q^1, then q^2).
// Threads first..blockDim-1 (whole warps) take the work items round-robin.
// Table layout: kXfStride bytes per group (hE, hO, lE, lO: 32 bytes each,
// then padding), or with kPacked 128 bytes per group whose eight 16-byte
// chunks sit rotated by the group index (chunk c of group g at slot
// (c + g) % 8), so that lanes reading consecutive groups chunk by chunk hit
// distinct banks without any shuffling of registers (load_x_fixed_packed).
template <bool kPacked = false>
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
        float mx, sm;
        x_quarter_stats(w, mx, sm);
        // the 4 threads of a group are adjacent lanes: fixed xor tree
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        sm += __shfl_xor_sync(0xffffffffu, sm, 1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        sm += __shfl_xor_sync(0xffffffffu, sm, 2);
        const int e = x_group_exp(mx);
        uint32_t hE[2], hO[2], lE[2], lO[2];
        x_quarter_fixed(w, e, hE, hO, lE, lO);
        if (act) {
            // 8-byte piece at logical offset o = 32 * part + 8 * q of the group's table
            auto at = [&](int part) -> uint2* {
                const int o = 32 * part + 8 * q;
                if (!kPacked) return reinterpret_cast<uint2*>(xf_s + grp * kXfStride + o);
                return reinterpret_cast<uint2*>(xf_s + grp * 128 + 16 * (((o >> 4) + grp) & 7) + (o & 15));
            };
            *at(0) = make_uint2(hE[0], hE[1]);
            *at(1) = make_uint2(hO[0], hO[1]);
            *at(2) = make_uint2(lE[0], lE[1]);
            *at(3) = make_uint2(lO[0], lO[1]);
            if (q == 0) {
                xs_s[2 * grp] = x_group_inv(e);
                xs_s[2 * grp + 1] = sm;
            }
        }
    }
}

// The same fixed-point copy of group gc built by one thread from x in shared
// memory, in two steps (x_group_load reads the group's 64 values, then
// x_group_fixed converts them), combining the four quarter sums in the same
// tree order as convert_x_fixed: identical values, no table.
__device__ __forceinline__ void x_group_load(const uint16_t* x_s, int gc, uint32_t (&w)[4][8]) {
    const uint4* src = reinterpret_cast<const uint4*>(x_s + 64 * gc);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 r0 = src[2 * q], r1 = src[2 * q + 1];
        w[q][0] = r0.x; w[q][1] = r0.y; w[q][2] = r0.z; w[q][3] = r0.w;
        w[q][4] = r1.x; w[q][5] = r1.y; w[q][6] = r1.z; w[q][7] = r1.w;
    }
}

__device__ __forceinline__ void x_group_fixed(const uint32_t (&w)[4][8], XFixed& xf) {
    float mq[4], sq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) x_quarter_stats(w[q], mq[q], sq[q]);
    const int e = x_group_exp(fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])));
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t hE[2], hO[2], lE[2], lO[2];
        x_quarter_fixed(w[q], e, hE, hO, lE, lO);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            xf.hE[2 * q + jj] = (int)hE[jj];
            xf.hO[2 * q + jj] = (int)hO[jj];
            xf.lE[2 * q + jj] = lE[jj];
            xf.lO[2 * q + jj] = lO[jj];
        }
    }
    xf.inv = x_group_inv(e);
    xf.xsum = (sq[0] + sq[1]) + (sq[2] + sq[3]);
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

// Group gc of a packed table (convert_x_fixed<true>): step c reads slot
// (c + gc) % 8, which holds chunk c, into the registers of chunk c.
__device__ __forceinline__ void load_x_fixed_packed(const uint8_t* xf_s, const float* xs_s, int gc, XFixed& xf) {
    const uint4* p = reinterpret_cast<const uint4*>(xf_s + gc * 128);
    uint4 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = p[(c + gc) & 7];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        xf.hE[4 * i] = (int)v[i].x; xf.hE[4 * i + 1] = (int)v[i].y; xf.hE[4 * i + 2] = (int)v[i].z; xf.hE[4 * i + 3] = (int)v[i].w;
        xf.hO[4 * i] = (int)v[2 + i].x; xf.hO[4 * i + 1] = (int)v[2 + i].y; xf.hO[4 * i + 2] = (int)v[2 + i].z; xf.hO[4 * i + 3] = (int)v[2 + i].w;
        xf.lE[4 * i] = v[4 + i].x; xf.lE[4 * i + 1] = v[4 + i].y; xf.lE[4 * i + 2] = v[4 + i].z; xf.lE[4 * i + 3] = v[4 + i].w;
        xf.lO[4 * i] = v[6 + i].x; xf.lO[4 * i + 1] = v[6 + i].y; xf.lO[4 * i + 2] = v[6 + i].z; xf.lO[4 * i + 3] = v[6 + i].w;
    }
    const float2 sc = reinterpret_cast<const float2*>(xs_s)[gc];
    xf.inv = sc.x;
    xf.xsum = sc.y;
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
