// Activation-sparse decode of a ReLU^2 MoE layer on GB300 (sm_103a).
//
// Method: "Skipping dead neurons: a faster Nemotron 3.5 Lightning on Apple
// silicon" (sevren.ai, "Heimr Sparse Down").
//  * "Inside a MoE layer": a router picks 6 of 128 experts; a shared expert
//    runs for every token.
//  * "Two projections and a switch": up projection 2688 -> N, ReLU^2, down
//    projection N -> 2688, 4-bit weights.
//  * "Our way reads only the rows that fired": the down weights are stored one
//    row per neuron; only rows whose h_n > 0 are read; partial sums from
//    independent slices of neurons are added by a final small pass.
//  * "The whole decode step": one (scale, bias) slab per group of 64 neurons,
//    read only if a neuron of the group fired.
//
// GB300 design (ours, not the page's Metal split):
//  * One CTA per (expert slot, group of 64 neurons).  The CTA streams the
//    group's 64 up rows (86 KB of codes + 10.75 KB of scales) into shared
//    memory with bulk TMA copies issued at CTA start, computes z, ReLU^2 and
//    a 64-bit live mask (warp ballots), then bulk-copies only the live down
//    rows and, if any neuron fired, the group's slab, and writes one fp32
//    partial row of `hidden` outputs, already scaled by the router weight.
//  * A second kernel adds the partial rows in a fixed order (deterministic)
//    and rounds to bf16.  Both kernels use programmatic dependent launch, so
//    a kernel's launch overlaps the previous one; CTAs of the shared expert
//    start streaming their weights before waiting on the previous kernel.
//  * The up GEMV is CUDA-core work (HBM bound, no tensor cores): codes are
//    turned into bf16 (128 + q) with one LOP3 per two codes and multiplied
//    with the bf16 activations by mixed-precision FMA into fp32 (exact
//    products); the 128 * sum(x) term is removed per 32-code chunk.
#include "hs_common.cuh"

namespace hs {

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
    int n_routed;
    int routed_neurons;
    int shared_neurons;   // 0 if no shared expert
    int hidden;
    int top_k;
};

struct DecodeIO {
    const uint16_t* x;       // [hidden] bf16
    const float* logits;     // [n_routed]
    float* partial;          // [units][hidden]
    unsigned flags;
    int* dbg_topk_idx;
    float* dbg_topk_w;
    float* dbg_h;
    int* live_counts;        // [units] live rows per unit (workspace)
};

// Dynamic shared memory layout of one decode CTA.
struct SmemLayout {
    static constexpr int kBars = 6;  // 4 up chunks, 1 down, spare
    __host__ __device__ static int codes_bytes(int hidden) { return 64 * hidden / 2; }
    __host__ __device__ static int sb_bytes(int hidden) { return hidden * 4; }
    __host__ __device__ static int total(int hidden) {
        return codes_bytes(hidden) + sb_bytes(hidden) + 64 * 4 /*h*/ + 64 /*bars*/ + 128 /*misc*/;
    }
};

// ------------------------------------------------------------------ router
// Top-k of n logits (ties -> lower index) and softmax over the chosen k.
// Executed by one full warp; results in idx[k], w[k] (shared memory).
__device__ void warp_topk_softmax(const float* __restrict__ logits, int n, int k, int* idx, float* w) {
    const int lane = threadIdx.x & 31;
    float v[kMaxRouted / 32];
#pragma unroll
    for (int i = 0; i < kMaxRouted / 32; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < n) ? logits[e] : -INFINITY;
    }
    unsigned taken = 0;  // bit i: element lane+32i already chosen
    float sel[kMaxTopK];
    int seli[kMaxTopK];
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kMaxRouted / 32; ++i) {
            const int e = lane + 32 * i;
            if (e < n && !((taken >> i) & 1u)) {
                if (v[i] > bv || (v[i] == bv && e < bi)) { bv = v[i]; bi = e; }
            }
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        sel[j] = bv;
        seli[j] = bi;
    }
    if (lane == 0) {
        const float m = sel[0];
        float den = 0.f;
        float ex[kMaxTopK];
        for (int j = 0; j < k; ++j) { ex[j] = expf(sel[j] - m); den += ex[j]; }
        for (int j = 0; j < k; ++j) { idx[j] = seli[j]; w[j] = ex[j] / den; }
    }
    __syncwarp();
}

// ------------------------------------------------------------- up phase
// Dot products of the CTA's 64 up rows with x.  Thread (c, r0) owns the
// 32-code chunk c of every row r = r0 + S*i; its 32 activations stay in
// registers as bf16 pairs matched to the nibble order of the code words.
// Per-(row, chunk) partial dot products are written over the first 4 bytes of
// the chunk they were computed from (each chunk has exactly one reader).
__device__ __forceinline__ float chunk_dot(const uint4 cw, const uint32_t (&xp)[16]) {
    float a0 = 0.f, a1 = 0.f;
    const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            uint32_t q;
            const uint32_t ws = w[j] >> (4 * s);
            asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xea;" : "=r"(q) : "r"(ws));
            asm("{ .reg .b16 ql, qh, xl, xh;\n"
                "  mov.b32 {ql, qh}, %2;\n"
                "  mov.b32 {xl, xh}, %3;\n"
                "  fma.rn.f32.bf16 %0, ql, xl, %0;\n"
                "  fma.rn.f32.bf16 %1, qh, xh, %1;\n"
                "}"
                : "+f"(a0), "+f"(a1)
                : "r"(q), "r"(xp[4 * j + s]));
        }
    }
    return a0 + a1;  // = sum_k (128 + q_k) x_k
}

struct UpThread {
    int c;       // chunk index (32 codes)
    int r0;      // first row
    int S;       // row stride
    bool active;
};

__device__ __forceinline__ void load_x_chunk(const uint16_t* __restrict__ x, int c, uint32_t (&xp)[16],
                                             float& xsum) {
    const uint4* p = reinterpret_cast<const uint4*>(x + 32 * c);
    uint32_t xw[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(p + i);
        xw[4 * i] = v.x; xw[4 * i + 1] = v.y; xw[4 * i + 2] = v.z; xw[4 * i + 3] = v.w;
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t w0 = xw[4 * j], w1 = xw[4 * j + 1], w2 = xw[4 * j + 2], w3 = xw[4 * j + 3];
        xp[4 * j + 0] = __byte_perm(w0, w2, 0x5410);
        xp[4 * j + 1] = __byte_perm(w0, w2, 0x7632);
        xp[4 * j + 2] = __byte_perm(w1, w3, 0x5410);
        xp[4 * j + 3] = __byte_perm(w1, w3, 0x7632);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        s += __uint_as_float(xw[i] << 16);
        s += __uint_as_float(xw[i] & 0xffff0000u);
    }
    xsum = s;
}

// ------------------------------------------------------------ down phase
// Given h[64] and the live mask in shared memory, accumulate
//   partial_o = wgt * (sum_{n live} h_n * (s_o q_{n,o} + b_o))
// for the CTA's group, with the live rows at their row slot in codes_buf and
// the slab (s_o, b_o) in sb_buf.  Thread (c, r3) sums the live rows n with
// n % S == r3 in ascending order; the S sums are added in order r3 = 0..S-1.
__device__ void down_accumulate_and_store(const uint8_t* codes_buf, const uint32_t* sb_buf, float* red_buf,
                                          const float* h_s, uint64_t live, float Hsum, float wgt, int hidden,
                                          float* __restrict__ out_row) {
    const int C = hidden / 32;
    const int S = min(256 / C, 8);
    const int t = threadIdx.x;
    const int c = t % C, r3 = t / C;
    const int rowb = hidden / 2;
    float acc[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) acc[k] = 0.f;
    if (r3 < S) {
        uint64_t m = 0;
        for (int n = r3; n < 64; n += S) m |= 1ull << n;
        m &= live;
        while (m) {
            const int n = __ffsll((long long)m) - 1;
            m &= m - 1;
            const float hn = h_s[n];
            const uint4 cw = *reinterpret_cast<const uint4*>(codes_buf + n * rowb + 16 * c);
            const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float q = __uint_as_float(0x4B000000u | ((w[j] >> (4 * i)) & 15u)) - 8388608.f;
                    acc[8 * j + i] = fmaf(hn, q, acc[8 * j + i]);
                }
            }
        }
    }
    __syncthreads();  // all reads of codes_buf done: reuse it for the cross-subset sum
    if (r3 >= 1 && r3 < S) {
        float4* dst = reinterpret_cast<float4*>(red_buf + (size_t)(r3 - 1) * hidden + 32 * c);
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[k] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
    }
    __syncthreads();
    if (r3 == 0) {
        for (int s = 1; s < S; ++s) {
            const float4* src = reinterpret_cast<const float4*>(red_buf + (size_t)(s - 1) * hidden + 32 * c);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 v = src[k];
                acc[4 * k] += v.x; acc[4 * k + 1] += v.y; acc[4 * k + 2] += v.z; acc[4 * k + 3] += v.w;
            }
        }
        float4* dst = reinterpret_cast<float4*>(out_row + 32 * c);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float r[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int o = 32 * c + 4 * k + e;
                const float2 sb = half2_to_float2(sb_buf[o]);
                r[e] = wgt * fmaf(sb.x, acc[4 * k + e], sb.y * Hsum);
            }
            dst[k] = make_float4(r[0], r[1], r[2], r[3]);
        }
    }
}

__device__ __forceinline__ void store_zero_row(float* __restrict__ out_row, int hidden) {
    for (int i = threadIdx.x; i < hidden / 4; i += blockDim.x)
        reinterpret_cast<float4*>(out_row)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Live mask of h_s[0..63] (warp 0), the fixed-order sum of h, and the issue
// of the down copies: live rows to their row slots and, if any, the slab.
// Returns (through smem) the mask and sum.  Executed by warp 0.
__device__ __forceinline__ void warp0_mask_and_issue(const float* h_s, bool dense, const uint8_t* dn_codes_g,
                                                     const uint32_t* dn_slab, int hidden, uint8_t* codes_buf,
                                                     uint32_t* sb_buf, uint64_t* bar, uint64_t* mask_out,
                                                     float* hsum_out, uint64_t policy) {
    const int lane = threadIdx.x & 31;
    const float h0 = h_s[lane], h1 = h_s[lane + 32];
    const unsigned b0 = __ballot_sync(0xffffffffu, h0 > 0.f);
    const unsigned b1 = __ballot_sync(0xffffffffu, h1 > 0.f);
    uint64_t live = dense ? ~0ull : ((uint64_t)b1 << 32 | b0);
    float s = h0 + h1;
#pragma unroll
    for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    const int rowb = hidden / 2;
    if (live) {
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(__popcll(live) * rowb + hidden * 4));
        __syncwarp();
        if (lane == 0) bulk_g2s(sb_buf, dn_slab, hidden * 4, bar, policy);
        if ((live >> lane) & 1) bulk_g2s(codes_buf + lane * rowb, dn_codes_g + (size_t)lane * rowb, rowb, bar, policy);
        if ((live >> (lane + 32)) & 1)
            bulk_g2s(codes_buf + (lane + 32) * rowb, dn_codes_g + (size_t)(lane + 32) * rowb, rowb, bar, policy);
    }
    if (lane == 0) { *mask_out = live; *hsum_out = s; }
}

// --------------------------------------------------- fused layer kernel (B=1)
__global__ void __launch_bounds__(256, 2)
moe_decode_b1_kernel(const __grid_constant__ LayerParams P, const DecodeIO io) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int hidden = P.hidden;
    uint8_t* codes_buf = smem;
    uint32_t* sb_buf = reinterpret_cast<uint32_t*>(smem + SmemLayout::codes_bytes(hidden));
    float* h_s = reinterpret_cast<float*>(smem + SmemLayout::codes_bytes(hidden) + SmemLayout::sb_bytes(hidden));
    uint64_t* bars = reinterpret_cast<uint64_t*>(h_s + 64);
    int* topk_i = reinterpret_cast<int*>(bars + 8);
    float* topk_w = reinterpret_cast<float*>(topk_i + kMaxTopK);
    uint64_t* live_s = reinterpret_cast<uint64_t*>(topk_w + kMaxTopK);
    float* hsum_s = reinterpret_cast<float*>(live_s + 1);

    const int t = threadIdx.x;
    const int u = blockIdx.x;
    const int sg = P.shared_neurons / 64, rg = P.routed_neurons / 64;
    const bool is_shared = u < sg;
    const int slot = is_shared ? 0 : 1 + (u - sg) / rg;
    const int g = is_shared ? u : (u - sg) % rg;
    const int rowb = hidden / 2;
    const bool dense = (io.flags & HS_FORCE_DENSE) != 0;
    const uint64_t pol = policy_evict_first();

    if (t == 0) {
        for (int i = 0; i < SmemLayout::kBars; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const ExpertPtrs* ep = nullptr;
    auto issue_up = [&](const ExpertPtrs& e) {
        // 4 chunks of 16 rows; the up scales ride on the first chunk
        const uint8_t* src = e.up_codes + (size_t)g * 64 * rowb;
        const uint32_t chunk = 16 * rowb;
        mbar_arrive_expect_tx(&bars[0], chunk + hidden * 4);
        bulk_g2s(sb_buf, e.up_sb + (size_t)g * 64 * (hidden / 64), hidden * 4, &bars[0], pol);
        bulk_g2s(codes_buf, src, chunk, &bars[0], pol);
        for (int k = 1; k < 4; ++k) {
            mbar_arrive_expect_tx(&bars[k], chunk);
            bulk_g2s(codes_buf + k * chunk, src + (size_t)k * chunk, chunk, &bars[k], pol);
        }
    };

    if (is_shared) {
        ep = &P.shared;
        if (t == 0) issue_up(*ep);  // weights do not depend on the previous kernel
    }
    pdl_wait();
    pdl_trigger();
    if (!is_shared || (u == 0 && io.dbg_topk_idx)) {
        if (t < 32) warp_topk_softmax(io.logits, P.n_routed, P.top_k, topk_i, topk_w);
        __syncthreads();
        if (u == 0 && io.dbg_topk_idx && t < P.top_k) {
            io.dbg_topk_idx[t] = topk_i[t];
            io.dbg_topk_w[t] = topk_w[t];
        }
    }
    float wgt = 1.f;
    if (!is_shared) {
        const int e = topk_i[slot - 1];
        wgt = topk_w[slot - 1];
        ep = &P.routed[e];
        if (t == 0) issue_up(*ep);
    }

    // ---- up projection for 64 rows
    const int C = hidden / 32;
    const int S = 256 / C;
    const int c = t % C, r0 = t / C;
    const bool up_active = r0 < S;
    uint32_t xp[16];
    float xsum = 0.f;
    if (up_active) load_x_chunk(io.x, c, xp, xsum);
    bool ok = true;
    if (up_active) {
        int waited = -1;
        for (int r = r0; r < 64; r += S) {
            const int k = r >> 4;
            while (waited < k) { ++waited; ok &= mbar_wait(&bars[waited], 0); }
            if (!ok) break;
            const uint4 cw = *reinterpret_cast<const uint4*>(codes_buf + r * rowb + 16 * c);
            const float2 sb = half2_to_float2(sb_buf[r * (hidden / 64) + (c >> 1)]);
            const float acc = chunk_dot(cw, xp);
            const float part = fmaf(sb.x, acc, fmaf(-128.f, sb.x, sb.y) * xsum);
            *reinterpret_cast<float*>(codes_buf + r * rowb + 16 * c) = part;
        }
    } else {
        for (int k = 0; k < 4; ++k) ok &= mbar_wait(&bars[k], 0);
    }
    if (!__syncthreads_and(ok)) return;

    // ---- row sums: thread (r, q) adds chunks q, q+4, ... then a fixed 4-way tree
    {
        const int r = t >> 2, q = t & 3;
        float s = 0.f;
        for (int cc = q; cc < C; cc += 4) s += *reinterpret_cast<const float*>(codes_buf + r * rowb + 16 * cc);
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        if (q == 0) {
            const int n = g * 64 + r;
            const float off = ep->up_off ? ep->up_off[n] : 0.f;
            const float z = s + off;
            const float h = z > 0.f ? z * z : 0.f;
            h_s[r] = h;
            if (io.dbg_h) {
                const int base = is_shared ? 0 : P.shared_neurons + (slot - 1) * P.routed_neurons;
                io.dbg_h[base + n] = h;
            }
        }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- live mask, fixed-order sum of h, down copies
    if (t < 32)
        warp0_mask_and_issue(h_s, dense, ep->dn_codes + (size_t)g * 64 * rowb, ep->dn_sb + (size_t)g * hidden, hidden,
                             codes_buf, sb_buf, &bars[4], live_s, hsum_s, pol);
    __syncthreads();
    const uint64_t live = *live_s;
    float* out_row = io.partial + (size_t)u * hidden;
    if (t == 0) io.live_counts[u] = __popcll(live);
    if (!live) {
        store_zero_row(out_row, hidden);
        return;
    }
    if (!__syncthreads_and(mbar_wait(&bars[4], 0))) return;
    down_accumulate_and_store(codes_buf, sb_buf, reinterpret_cast<float*>(codes_buf), h_s, live, *hsum_s, wgt,
                              hidden, out_row);
}

// ------------------------------------------ single-expert sparse down (K1)
__global__ void __launch_bounds__(256, 2)
down_sparse_kernel(const float* __restrict__ h, const uint8_t* __restrict__ dn_codes,
                   const uint32_t* __restrict__ dn_sb, int hidden, unsigned flags, float* __restrict__ partial,
                   int* __restrict__ live_counts) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* codes_buf = smem;
    uint32_t* sb_buf = reinterpret_cast<uint32_t*>(smem + SmemLayout::codes_bytes(hidden));
    float* h_s = reinterpret_cast<float*>(smem + SmemLayout::codes_bytes(hidden) + SmemLayout::sb_bytes(hidden));
    uint64_t* bars = reinterpret_cast<uint64_t*>(h_s + 64);
    uint64_t* live_s = bars + 8;
    float* hsum_s = reinterpret_cast<float*>(live_s + 1);
    const int t = threadIdx.x, g = blockIdx.x;
    const int rowb = hidden / 2;
    if (t == 0) { mbar_init(&bars[0], 1); fence_mbar_init(); }
    pdl_wait();
    pdl_trigger();
    if (t < 64) h_s[t] = h[g * 64 + t];
    __syncthreads();
    if (t < 32)
        warp0_mask_and_issue(h_s, (flags & HS_FORCE_DENSE) != 0, dn_codes + (size_t)g * 64 * rowb,
                             dn_sb + (size_t)g * hidden, hidden, codes_buf, sb_buf, &bars[0], live_s, hsum_s,
                             policy_evict_first());
    __syncthreads();
    const uint64_t live = *live_s;
    float* out_row = partial + (size_t)g * hidden;
    if (t == 0) live_counts[g] = __popcll(live);
    if (!live) { store_zero_row(out_row, hidden); return; }
    if (!__syncthreads_and(mbar_wait(&bars[0], 0))) return;
    down_accumulate_and_store(codes_buf, sb_buf, reinterpret_cast<float*>(codes_buf), h_s, live, *hsum_s, 1.f,
                              hidden, out_row);
}

// ------------------------------------------------ fixed-order partial sum
// y[o] = sum_{u=0..U-1} partial[u][o] (u ascending within each of 32 strided
// subsets, then the 32 subset sums in order); bf16 round to nearest even.
// Also sums the per-unit live counts into *live_total (if non-null).
__global__ void __launch_bounds__(256)
reduce_partials_kernel(const float* __restrict__ partial, int U, int hidden, uint16_t* __restrict__ y_bf16,
                       float* __restrict__ y_f32, const int* __restrict__ live_counts, int* __restrict__ live_total) {
    __shared__ float4 red[32][8];
    pdl_wait();
    pdl_trigger();
    const int t = threadIdx.x;
    const int col = blockIdx.x * 8 + (t & 7);  // float4 column
    const int uc = t >> 3;
    const int ncol = hidden / 4;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col < ncol) {
        const float4* p = reinterpret_cast<const float4*>(partial) + col;
        for (int u = uc; u < U; u += 32) {
            const float4 v = __ldcg(p + (size_t)u * ncol);
            s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
        }
    }
    red[uc][t & 7] = s;
    __syncthreads();
    if (t < 8 && col < ncol) {
        float4 a = red[0][t];
        for (int i = 1; i < 32; ++i) {
            const float4 v = red[i][t];
            a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
        }
        if (y_f32) reinterpret_cast<float4*>(y_f32)[col] = a;
        const uint32_t lo = (uint32_t)f32_to_bf16_bits(a.x) | ((uint32_t)f32_to_bf16_bits(a.y) << 16);
        const uint32_t hi = (uint32_t)f32_to_bf16_bits(a.z) | ((uint32_t)f32_to_bf16_bits(a.w) << 16);
        reinterpret_cast<uint2*>(y_bf16)[col] = make_uint2(lo, hi);
    }
    if (live_total && blockIdx.x == 0 && t == 0) {
        int n = 0;
        for (int u = 0; u < U; ++u) n += live_counts[u];
        *live_total = n;
    }
}

}  // namespace hs

// ===================================================================== host
namespace {

bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool al4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int launch_err() { return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA; }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

int set_smem_attr(const void* fn, int bytes) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return HS_ERR_CUDA;
    return HS_OK;
}

int check_expert(const hs_expert& e, int hidden, int neurons_expected) {
    if (!e.up.codes || !e.up.sb || !e.down_nm.codes || !e.down_nm.sb) return HS_ERR_INVALID_ARG;
    if (e.neurons != neurons_expected) return HS_ERR_UNSUPPORTED_SHAPE;
    if (!al16(e.up.codes) || !al16(e.up.sb) || !al16(e.down_nm.codes) || !al16(e.down_nm.sb)) return HS_ERR_MISALIGNED;
    if (e.up_offset && !al4(e.up_offset)) return HS_ERR_MISALIGNED;
    (void)hidden;
    return HS_OK;
}

int check_layer(const hs_moe_layer* L) {
    if (!L || !L->routed) return HS_ERR_INVALID_ARG;
    if (L->n_routed < 1 || L->n_routed > hs::kMaxRouted) return HS_ERR_UNSUPPORTED_SHAPE;
    if (L->top_k < 1 || L->top_k > hs::kMaxTopK || L->top_k > L->n_routed) return HS_ERR_UNSUPPORTED_SHAPE;
    if (L->hidden < 64 || L->hidden > hs::kMaxHidden || L->hidden % 64) return HS_ERR_UNSUPPORTED_SHAPE;
    const int rn = L->routed[0].neurons;
    if (rn < 64 || rn % 64) return HS_ERR_UNSUPPORTED_SHAPE;
    for (int e = 0; e < L->n_routed; ++e) {
        const int st = check_expert(L->routed[e], L->hidden, rn);
        if (st != HS_OK) return st;
    }
    if (L->shared) {
        if (L->shared->neurons < 64 || L->shared->neurons % 64) return HS_ERR_UNSUPPORTED_SHAPE;
        const int st = check_expert(*L->shared, L->hidden, L->shared->neurons);
        if (st != HS_OK) return st;
    }
    return HS_OK;
}

int decode_units(const hs_moe_layer* L) {
    return (L->shared ? L->shared->neurons / 64 : 0) + L->top_k * (L->routed[0].neurons / 64);
}

}  // namespace

extern "C" const char* hs_status_string(int status) {
    switch (status) {
        case HS_OK: return "ok";
        case HS_ERR_INVALID_ARG: return "invalid argument";
        case HS_ERR_MISALIGNED: return "misaligned pointer (weights, activations, outputs need 16 bytes)";
        case HS_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case HS_ERR_WORKSPACE: return "workspace missing or too small";
        case HS_ERR_CUDA: return "CUDA error";
        case HS_ERR_TIMEOUT: return "a bounded device wait timed out";
        default: return "unknown status";
    }
}

extern "C" int hs_device_status(int* status) {
    if (!status) return HS_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return HS_ERR_CUDA;
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, hs::g_status, sizeof(v)) != cudaSuccess) return HS_ERR_CUDA;
    if (cudaMemcpyToSymbol(hs::g_status, &zero, sizeof(zero)) != cudaSuccess) return HS_ERR_CUDA;
    *status = v ? HS_ERR_TIMEOUT : HS_OK;
    return HS_OK;
}

// ----------------------------------------------------------- sparse down
extern "C" size_t hs_expert_down_sparse_workspace_size(int neurons, int out_dim) {
    if (neurons <= 0 || out_dim <= 0 || neurons % 64 || out_dim % 64) return 0;
    const size_t G = neurons / 64;
    return round_up(G * out_dim * sizeof(float), 256) + round_up(G * sizeof(int), 256);
}

extern "C" int hs_expert_down_sparse(const float* h, const hs_w4* down_nm, int neurons, int out_dim, uint16_t* y_bf16,
                                     float* y_f32, int* live_count, unsigned flags, void* ws, size_t ws_bytes,
                                     hs_stream_t stream) {
    if (!h || !down_nm || !down_nm->codes || !down_nm->sb || !y_bf16) return HS_ERR_INVALID_ARG;
    if (neurons <= 0 || out_dim <= 0) return HS_ERR_INVALID_ARG;
    if (neurons % 64 || out_dim % 64 || out_dim > hs::kMaxHidden) return HS_ERR_UNSUPPORTED_SHAPE;
    if (!al16(h) || !al16(down_nm->codes) || !al16(down_nm->sb) || !al16(y_bf16) || (y_f32 && !al16(y_f32)) ||
        (live_count && !al4(live_count)) || !al16(ws))
        return HS_ERR_MISALIGNED;
    const size_t need = hs_expert_down_sparse_workspace_size(neurons, out_dim);
    if (!ws || ws_bytes < need) return HS_ERR_WORKSPACE;
    const int G = neurons / 64;
    float* partial = static_cast<float*>(ws);
    int* counts = reinterpret_cast<int*>(static_cast<char*>(ws) + round_up((size_t)G * out_dim * sizeof(float), 256));
    const int smem = hs::SmemLayout::total(out_dim);
    if (set_smem_attr((const void*)hs::down_sparse_kernel, smem) != HS_OK) return HS_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_pdl(hs::down_sparse_kernel, dim3(G), dim3(256), smem, s, h, down_nm->codes,
                   static_cast<const uint32_t*>(down_nm->sb), out_dim, flags, partial, counts) != cudaSuccess)
        return HS_ERR_CUDA;
    if (launch_pdl(hs::reduce_partials_kernel, dim3((out_dim / 4 + 7) / 8), dim3(256), 0, s, (const float*)partial, G,
                   out_dim, y_bf16, y_f32, (const int*)counts, live_count) != cudaSuccess)
        return HS_ERR_CUDA;
    return launch_err();
}

// ---------------------------------------------------------- layer decode
extern "C" size_t hs_moe_layer_decode_workspace_size(const hs_moe_layer* L, int batch) {
    if (check_layer(L) != HS_OK || batch != 1) return 0;
    const size_t U = decode_units(L);
    return round_up(U * L->hidden * sizeof(float), 256) + round_up(U * sizeof(int), 256);
}

extern "C" int hs_moe_layer_decode(const hs_moe_layer* L, const uint16_t* x, const float* logits, int batch,
                                   uint16_t* y_bf16, float* y_f32, unsigned flags, const hs_decode_debug* dbg,
                                   void* ws, size_t ws_bytes, hs_stream_t stream) {
    int st = check_layer(L);
    if (st != HS_OK) return st;
    if (!x || !logits || !y_bf16) return HS_ERR_INVALID_ARG;
    if (batch < 1) return HS_ERR_INVALID_ARG;
    if (batch != 1) return HS_ERR_UNSUPPORTED_SHAPE;
    if (!al16(x) || !al4(logits) || !al16(y_bf16) || (y_f32 && !al16(y_f32)) || !al16(ws)) return HS_ERR_MISALIGNED;
    const size_t need = hs_moe_layer_decode_workspace_size(L, batch);
    if (!ws || ws_bytes < need) return HS_ERR_WORKSPACE;
    if (dbg && ((dbg->topk_idx == nullptr) != (dbg->topk_w == nullptr))) return HS_ERR_INVALID_ARG;

    hs::LayerParams P;
    memset(&P, 0, sizeof(P));
    auto fill = [](hs::ExpertPtrs& d, const hs_expert& e) {
        d.up_codes = e.up.codes;
        d.up_sb = static_cast<const uint32_t*>(e.up.sb);
        d.dn_codes = e.down_nm.codes;
        d.dn_sb = static_cast<const uint32_t*>(e.down_nm.sb);
        d.up_off = e.up_offset;
    };
    for (int e = 0; e < L->n_routed; ++e) fill(P.routed[e], L->routed[e]);
    if (L->shared) fill(P.shared, *L->shared);
    P.n_routed = L->n_routed;
    P.routed_neurons = L->routed[0].neurons;
    P.shared_neurons = L->shared ? L->shared->neurons : 0;
    P.hidden = L->hidden;
    P.top_k = L->top_k;

    const int U = decode_units(L);
    hs::DecodeIO io;
    io.x = x;
    io.logits = logits;
    io.partial = static_cast<float*>(ws);
    io.live_counts = reinterpret_cast<int*>(static_cast<char*>(ws) + round_up((size_t)U * L->hidden * sizeof(float), 256));
    io.flags = flags;
    io.dbg_topk_idx = dbg ? dbg->topk_idx : nullptr;
    io.dbg_topk_w = dbg ? dbg->topk_w : nullptr;
    io.dbg_h = dbg ? dbg->h : nullptr;
    int* live_out = dbg ? dbg->live_rows : nullptr;

    const int smem = hs::SmemLayout::total(L->hidden);
    if (set_smem_attr((const void*)hs::moe_decode_b1_kernel, smem) != HS_OK) return HS_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_pdl(hs::moe_decode_b1_kernel, dim3(U), dim3(256), smem, s, P, io) != cudaSuccess) return HS_ERR_CUDA;
    if (launch_pdl(hs::reduce_partials_kernel, dim3((L->hidden / 4 + 7) / 8), dim3(256), 0, s,
                   (const float*)io.partial, U, L->hidden, y_bf16, y_f32, (const int*)io.live_counts,
                   live_out) != cudaSuccess)
        return HS_ERR_CUDA;
    return launch_err();
}
