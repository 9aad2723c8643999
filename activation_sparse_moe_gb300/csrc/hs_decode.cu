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
//  * The up GEMV is integer-pipe work (HBM bound, no tensor cores): x is
//    converted once per CTA into a 16-bit fixed-point copy with one exponent
//    per 64-input scale group, split into a signed high and an unsigned low
//    byte; each 32-byte group of codes is split into even and odd nibbles by
//    two masks and dotted with the bytes by DP4A (exact int32 sums); the
//    group's scale and bias are applied to the integer sum in fp32
//    (group_dot_fixed16 in hs_kernels.cuh).
#include "hs_kernels.cuh"
#include "hs_host.h"

#include <cstring>
#include <mutex>

namespace hs {

struct DecodeIO {
    const uint16_t* x;       // [hidden] bf16
    const float* logits;     // [n_routed]
    float* partial;          // [units][hidden]
    unsigned flags;
    int* dbg_topk_idx;
    float* dbg_topk_w;
    float* dbg_h;
    int* live_counts;        // [units] live rows per unit (workspace)
    uint64_t* dbg_live;      // [units] live mask (h > 0) per unit, or null
    int units;
};

// Dynamic shared memory layout of one decode CTA (offsets in bytes).
struct SmemLayout {
    static constexpr int kBars = 6;  // 4 up chunks, 1 down, 1 activations
    __host__ __device__ static int codes_bytes(int hidden) { return 64 * hidden / 2; }
    // the up scales of 64 rows or the down slab (hidden pairs); with row scales
    // (row = true) at least the 64 rows' (scale, bias) rows of hidden/64 pairs
    // padded to 16 bytes
    __host__ __device__ static int row_sb_words(int hidden) { return ((hidden / 64) + 3) & ~3; }
    __host__ __device__ static int sb_bytes(int hidden, bool row = false) {
        return row && 64 * 4 * row_sb_words(hidden) > hidden * 4 ? 64 * 4 * row_sb_words(hidden) : hidden * 4;
    }
    __host__ __device__ static int misc_off(int hidden, bool row = false) {
        return codes_bytes(hidden) + sb_bytes(hidden, row);
    }
    // misc: h[64] f32, off[64] f32, topk_i[8] i32, topk_w[8] f32, bars[8] u64, live mask (u64, or
    //       8 bytes of per-warp row bits), 24 bytes (the slab claim flag i32 at +8),
    // then x[hidden] bf16 (staging), the fixed-point x table [G][144 B] and its
    // per-group (2^(E-15), sum x) pairs [G][2] f32.
    static constexpr int kH = 0, kOff = 256, kTopI = 512, kTopW = kTopI + 32, kBarsOff = kTopW + 32,
                         kLive = kBarsOff + 64, kHsum = kLive + 8, kX = kHsum + 24;
    __host__ __device__ static int x_off(int hidden, bool row = false) { return misc_off(hidden, row) + kX; }
    __host__ __device__ static int xf_off(int hidden, bool row = false) { return x_off(hidden, row) + 2 * hidden; }
    __host__ __device__ static int xs_off(int hidden, bool row = false) {
        return xf_off(hidden, row) + (hidden / 64) * hs::kXfStride;
    }
    __host__ __device__ static int total(int hidden, bool row = false) { return xs_off(hidden, row) + (hidden / 64) * 8; }
};

// Partial rows are stored column-block-major: the 32 outputs of block cb of
// unit u sit at partial[(cb * U + u) * 32 ...], so one reduce CTA reads the
// contiguous slice of its block for every unit with a single bulk copy.
struct PartialOut {
    float* base;  // [hidden/32][U][32]
    int U;
    int u;
    __device__ __forceinline__ float4* quad(int o4) const {  // outputs 4*o4 .. 4*o4+3
        return reinterpret_cast<float4*>(base + ((size_t)(o4 >> 3) * U + u) * 32) + (o4 & 7);
    }
};

// ------------------------------------------------------------ down phase
__device__ __forceinline__ void store_zero_row(const PartialOut out, int hidden) {
    for (int i = threadIdx.x; i < hidden / 4; i += blockDim.x) *out.quad(i) = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Down phase of the fused kernel: thread j < hidden/OPT owns outputs
// OPT*j .. OPT*j+OPT-1 (OPT = 12 when hidden is a multiple of 48, so that 224
// threads share the work at hidden 2688; else 16) and adds the live rows in
// ascending neuron order in one fp32 chain per output (a dead row would add
// h * q = +0 exactly, so the dense flag, which adds every row, gives
// identical bits), then
//   partial_o = wgt * (s_o * sum_n h_n q_{n,o} + b_o * sum_n h_n).
// Nibble i of a code word becomes a float by masking it in place under the
// exponent of 2^23 and subtracting 2^23 (exact: q * 16^i < 2^23); the row's h
// is pre-scaled by 16^-i to undo the position.
//
// kRow (HS_DOWN_ROW_SCALES): sb_buf holds each live row's own (scale, bias)
// per 64 outputs (row n at n * rsw words) instead of the group's slab, and
// each term is h_n * (s_{n,g(o)} q_{n,o} + b_{n,g(o)}), added to the chain as
// fma(h s 16^-i, q 16^i, acc + h b); partial_o = wgt * sum.
template <int OPT, bool kRow>
__device__ __forceinline__ void down_acc_and_store(const uint8_t* codes_buf, const uint32_t* sb_buf,
                                                   const float* h_s, uint64_t live, float Hsum, float wgt,
                                                   int rowb, int j, const PartialOut out, int rsw) {
    static_assert(OPT == 12 || OPT == 16, "12 or 16 outputs per thread");
    float acc[OPT];
#pragma unroll
    for (int e = 0; e < OPT; ++e) acc[e] = 0.f;
    // with row scales, this thread's outputs OPT*j .. OPT*j+OPT-1 lie in groups g0 and g0 + 1
    const int g0 = (OPT * j) >> 6;
    while (live) {
        const int n = __ffsll((long long)live) - 1;
        live &= live - 1;
        const float hn = h_s[n];
        float hs[5] = {hn, hn * 0.0625f, hn * 0.00390625f, hn * 0.000244140625f, hn * 1.52587890625e-05f};
        float hs1[5], hb0 = 0.f, hb1 = 0.f;
        if (kRow) {
            const uint32_t* sr = sb_buf + (size_t)n * rsw;
            const float2 p0 = half2_to_float2(sr[g0]);
            const float2 p1 = half2_to_float2(sr[min(g0 + 1, rsw - 1)]);
#pragma unroll
            for (int i = 0; i < 5; ++i) {
                hs1[i] = hs[i] * p1.x;
                hs[i] *= p0.x;
            }
            hb0 = hn * p0.y;
            hb1 = hn * p1.y;
        }
        const uint8_t* row = codes_buf + (size_t)n * rowb;
        uint32_t w[2];
        if (OPT == 16) {
            const uint2 cw = *reinterpret_cast<const uint2*>(row + 8 * j);
            w[0] = cw.x;
            w[1] = cw.y;
        } else if (j & 1) {  // bytes 6j .. 6j+5 start 2 bytes into a word
            const uint32_t lo = *reinterpret_cast<const uint16_t*>(row + 6 * j);
            const uint32_t hi = *reinterpret_cast<const uint32_t*>(row + 6 * j + 2);
            w[0] = lo | (hi << 16);
            w[1] = hi >> 16;
        } else {
            w[0] = *reinterpret_cast<const uint32_t*>(row + 6 * j);
            w[1] = *reinterpret_cast<const uint16_t*>(row + 6 * j + 4);
        }
#pragma unroll
        for (int jj = 0; jj < OPT / 8 + (OPT % 8 != 0); ++jj) {
            const uint32_t hi = w[jj] >> 12;  // nibbles 5, 6, 7 at positions 2, 3, 4
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (8 * jj + i >= OPT) break;
                const uint32_t src = i < 5 ? w[jj] : hi;
                const int pos = i < 5 ? i : i - 3;
                const float q = __uint_as_float((src & (15u << (4 * pos))) | 0x4B000000u) - 8388608.f;
                if (kRow) {
                    const bool second = OPT * j + 8 * jj + i >= 64 * (g0 + 1);
                    acc[8 * jj + i] = fmaf(second ? hs1[pos] : hs[pos], q, acc[8 * jj + i] + (second ? hb1 : hb0));
                } else {
                    acc[8 * jj + i] = fmaf(hs[pos], q, acc[8 * jj + i]);
                }
            }
        }
    }
    if (kRow) {
#pragma unroll
        for (int i = 0; i < OPT / 4; ++i)
            *out.quad((OPT / 4) * j + i) =
                make_float4(wgt * acc[4 * i], wgt * acc[4 * i + 1], wgt * acc[4 * i + 2], wgt * acc[4 * i + 3]);
        return;
    }
    const uint4* sbq = reinterpret_cast<const uint4*>(sb_buf) + (OPT / 4) * j;
#pragma unroll
    for (int i = 0; i < OPT / 4; ++i) {
        const uint4 v = sbq[i];
        const uint32_t sbw[4] = {v.x, v.y, v.z, v.w};
        float r[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 sb = half2_to_float2(sbw[e]);
            r[e] = wgt * fmaf(sb.x, acc[4 * i + e], sb.y * Hsum);
        }
        *out.quad((OPT / 4) * j + i) = make_float4(r[0], r[1], r[2], r[3]);
    }
}

// --------------------------------------------------- fused layer kernel (B=1)
// kRow: the experts' down projections carry per-row scales (HS_DOWN_ROW_SCALES).
template <bool kRow>
__global__ void __launch_bounds__(256, 2)
moe_decode_b1_kernel(const __grid_constant__ LayerParams P, const DecodeIO io) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int hidden = P.hidden;
    uint8_t* codes_buf = smem;
    uint32_t* sb_buf = reinterpret_cast<uint32_t*>(smem + SmemLayout::codes_bytes(hidden));
    uint8_t* misc = smem + SmemLayout::misc_off(hidden, kRow);
    float* h_s = reinterpret_cast<float*>(misc + SmemLayout::kH);
    float* off_s = reinterpret_cast<float*>(misc + SmemLayout::kOff);
    int* topk_i = reinterpret_cast<int*>(misc + SmemLayout::kTopI);
    float* topk_w = reinterpret_cast<float*>(misc + SmemLayout::kTopW);
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc + SmemLayout::kBarsOff);
    uint16_t* x_s = reinterpret_cast<uint16_t*>(smem + SmemLayout::x_off(hidden, kRow));

    const int t = threadIdx.x;
    const int u = blockIdx.x;
    const int sg = P.shared_neurons / 64, rg = P.routed_neurons / 64;
    const bool is_shared = u < sg;
    const int slot = is_shared ? 0 : 1 + (u - sg) / rg;
    const int g = is_shared ? u : (u - sg) % rg;
    const int rowb = hidden / 2;
    const int G = hidden / 64;  // scale groups per up row
    const bool dense = (io.flags & HS_FORCE_DENSE) != 0;
    const uint64_t pol = policy_evict_first();

    // set by the first live row of the group, whose thread then requests the slab
    int* slab_claim = reinterpret_cast<int*>(misc + SmemLayout::kHsum + 8);
    if (t == 0) {
        for (int i = 0; i < SmemLayout::kBars; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        *slab_claim = 0;
    }
    __syncthreads();

    auto issue_up = [&](const ExpertPtrs& e) {
        // 4 chunks of 16 rows; the up scales ride on the first chunk
        const uint8_t* src = e.up_codes + (size_t)g * 64 * rowb;
        const uint32_t chunk = 16 * rowb;
        mbar_arrive_expect_tx(&bars[0], chunk + hidden * 4);
        bulk_g2s(sb_buf, e.up_sb + (size_t)g * 64 * G, hidden * 4, &bars[0], pol);
        bulk_g2s(codes_buf, src, chunk, &bars[0], pol);
        for (int k = 1; k < 4; ++k) {
            mbar_arrive_expect_tx(&bars[k], chunk);
            bulk_g2s(codes_buf + k * chunk, src + (size_t)k * chunk, chunk, &bars[k], pol);
        }
    };

    ExpertPtrs ep;
    if (is_shared) {
        ep = P.shared;
        if (t == 0) issue_up(ep);  // weights do not depend on the previous kernel
    }
    // x and the logits into L2 ahead of the wait: nothing is read from them before it, and L2 holds
    // whatever the previous kernel writes there (when it produced them, they are in L2 already)
    if (t >= 32 && t < 64) {
        prefetch_l2_span(io.x, hidden * 2, t - 32);
        if (!is_shared) prefetch_l2_span(io.logits, P.n_routed * 4, t - 32);
    }
    pdl_wait();
    pdl_trigger();

    // activations and logits (may be produced by the previous kernel)
    if (t == 0) {
        mbar_arrive_expect_tx(&bars[5], hidden * 2);
        bulk_g2s(x_s, io.x, hidden * 2, &bars[5], policy_evict_last());
    }
    const bool dbg_topk = io.dbg_topk_idx || io.dbg_topk_w;
    const bool need_topk = !is_shared || (u == 0 && dbg_topk);
    // warp 0 routes (if this CTA needs it); the other warps convert x meanwhile
    const int S = 256 / G;
    const int gc = t % G, r0 = t / G;
    const bool up_active = r0 < S;
    uint8_t* xf_s = smem + SmemLayout::xf_off(hidden, kRow);
    float* xs_s = reinterpret_cast<float*>(smem + SmemLayout::xs_off(hidden, kRow));
    // routing first, with the rest of the CTA idle (a latency-bound chain);
    // the routed weight copies go out before x is converted, so the
    // conversion overlaps their latency
    if (need_topk) {
        if (t < 32) warp_topk_softmax(io.logits, P.n_routed, P.top_k, topk_i, topk_w);
        __syncthreads();
        if (u == 0 && dbg_topk && t < P.top_k) {
            if (io.dbg_topk_idx) io.dbg_topk_idx[t] = topk_i[t];
            if (io.dbg_topk_w) io.dbg_topk_w[t] = topk_w[t];
        }
    }
    float wgt = 1.f;
    if (!is_shared) {
        const int e = topk_i[slot - 1];
        wgt = topk_w[slot - 1];
        ep = routed_ptrs(P, e);
        if (t == 0) issue_up(ep);
    }
    float off_r = 0.f;
    if (t < 64 && ep.up_off) off_r = ep.up_off[g * 64 + t];
    // after a wait gave up (the error word is set): one thread waits, bounded
    // again, for every copy this CTA still has in flight before the CTA leaves
    auto drain_up = [&]() {
        if (t == 0) {
            for (int i = 0; i < 4; ++i) mbar_wait(&bars[i], 0);
            mbar_wait(&bars[5], 0);
        }
    };
    bool ok = mbar_wait(&bars[5], 0);
    if (ok) convert_x_fixed(x_s, G, xf_s, xs_s, 0);
    if (!__syncthreads_and(ok)) { drain_up(); return; }

    // ---- up projection for 64 rows
    XFixed xf;
    if (up_active) {
        load_x_fixed(xf_s, xs_s, gc, xf);
        int waited = -1;
        const uint8_t* base = codes_buf;
        int r = r0;
        for (; r + S < 64; r += 2 * S) {  // two rows at a time
            const int k = (r + S) >> 4;
            while (waited < k) { ++waited; ok &= mbar_wait(&bars[waited], 0); }
            if (!ok) break;
            uint4 a0, a1, b0, b1;
            load_group_codes(base + r * rowb, gc, a0, a1);
            load_group_codes(base + (r + S) * rowb, gc, b0, b1);
            const float2 sa = half2_to_float2(sb_buf[r * G + gc]);
            const float2 sbb = half2_to_float2(sb_buf[(r + S) * G + gc]);
            const int da = group_dot_fixed16(a0, a1, xf);
            const int db = group_dot_fixed16(b0, b1, xf);
            // part = s * sum_k q_k x_k + b * sum_k x_k
            *part_slot(codes_buf, rowb, r, gc) = fmaf(sa.x * xf.inv, (float)da, sa.y * xf.xsum);
            *part_slot(codes_buf, rowb, r + S, gc) = fmaf(sbb.x * xf.inv, (float)db, sbb.y * xf.xsum);
        }
        if (ok && r < 64) {
            const int k = r >> 4;
            while (waited < k) { ++waited; ok &= mbar_wait(&bars[waited], 0); }
            if (ok) {
                uint4 a0, a1;
                load_group_codes(base + r * rowb, gc, a0, a1);
                const float2 sa = half2_to_float2(sb_buf[r * G + gc]);
                const int da = group_dot_fixed16(a0, a1, xf);
                *part_slot(codes_buf, rowb, r, gc) = fmaf(sa.x * xf.inv, (float)da, sa.y * xf.xsum);
            }
        }
        while (ok && waited < 3) { ++waited; ok &= mbar_wait(&bars[waited], 0); }
    } else {
        for (int k = 0; k < 4; ++k) ok &= mbar_wait(&bars[k], 0);
    }
    if (t < 64) off_s[t] = off_r;
    fence_proxy_async_smem();  // the partial stores come before the down copies into the same rows
    if (!__syncthreads_and(ok)) { drain_up(); return; }

    // ---- row sums: thread (r, q) adds groups q, q+4, ... then a fixed 4-way
    // tree; the row's first thread then copies the row's down codes into the
    // row's slot if the neuron fired (the slot's partials are consumed)
    uint8_t* live8 = misc + SmemLayout::kLive;  // live bits of rows 8w .. 8w+7 per warp w
    bool lv = false;
    {
        const int r = t >> 2, q = t & 3;
        float s0 = 0.f, s1 = 0.f;
        int cc = q;
        for (; cc + 4 < G; cc += 8) {
            s0 += *part_slot(codes_buf, rowb, r, cc);
            s1 += *part_slot(codes_buf, rowb, r, cc + 4);
        }
        if (cc < G) s0 += *part_slot(codes_buf, rowb, r, cc);
        float s = s0 + s1;
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        if (q == 0) {
            const int n = g * 64 + r;
            const float z = s + off_s[r];
            const float h = z > 0.f ? z * z : 0.f;
            h_s[r] = h;
            if (io.dbg_h) {
                const int base = is_shared ? 0 : P.shared_neurons + (slot - 1) * P.routed_neurons;
                io.dbg_h[base + n] = h;
            }
            lv = dense || h > 0.f;
            if (lv) {
                const uint32_t rsb = kRow ? 4u * SmemLayout::row_sb_words(hidden) : 0u;
                mbar_expect_tx(&bars[4], (uint32_t)rowb + rsb);
                bulk_g2s(codes_buf + (size_t)r * rowb, ep.dn_codes + ((size_t)g * 64 + r) * rowb, rowb, &bars[4], pol);
                if (kRow)
                    bulk_g2s(reinterpret_cast<uint8_t*>(sb_buf) + (size_t)r * rsb,
                             reinterpret_cast<const uint8_t*>(ep.dn_sb) + ((size_t)g * 64 + r) * rsb, rsb, &bars[4], pol);
                // the group's slab, requested once, by the first live row's thread (the up scales it
                // replaces were read before the barrier above)
                if (!kRow && atomicExch(slab_claim, 1) == 0) {
                    mbar_expect_tx(&bars[4], (uint32_t)hidden * 4);
                    bulk_g2s(sb_buf, ep.dn_sb + (size_t)g * hidden, hidden * 4, &bars[4], pol);
                }
            }
        }
        const unsigned b = __ballot_sync(0xffffffffu, lv);  // bits at lanes 4i
        if ((t & 31) == 0) {
            unsigned m8 = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) m8 |= ((b >> (4 * i)) & 1u) << i;
            live8[t >> 5] = (uint8_t)m8;
        }
    }
    // the single arrival on the down barrier comes after every copy's expected
    // bytes (rows, and the slab if any neuron fired) were added
    const bool any = __syncthreads_or(lv) != 0;
    if (t == 0 && any) mbar_arrive(&bars[4]);
    const uint64_t live = *reinterpret_cast<const uint64_t*>(live8);
    const PartialOut out_row{io.partial, io.units, u};
    if (t == 0) io.live_counts[u] = __popcll(live);
    if (io.dbg_live && t < 32) {  // the live set itself (h > 0), whatever the dense flag reads
        const unsigned m0 = __ballot_sync(0xffffffffu, h_s[t] > 0.f), m1 = __ballot_sync(0xffffffffu, h_s[t + 32] > 0.f);
        if (t == 0) io.dbg_live[u] = (uint64_t)m1 << 32 | m0;
    }
    if (!any) {
        store_zero_row(out_row, hidden);
        return;
    }
    // fixed-order sum of the 64 h values (every warp computes the same value)
    float Hsum = h_s[t & 31] + h_s[(t & 31) + 32];
#pragma unroll
    for (int off = 16; off; off >>= 1) Hsum += __shfl_xor_sync(0xffffffffu, Hsum, off);
    const int nthr = hidden % 48 == 0 ? hidden / 12 : hidden / 16;
    if (t >= nthr) return;
    if (!mbar_wait(&bars[4], 0)) {
        if (t == 0) mbar_wait(&bars[4], 0);  // the rows' copies land before the CTA leaves
        return;
    }
    const int rsw = SmemLayout::row_sb_words(hidden);
    if (hidden % 48 == 0)
        down_acc_and_store<12, kRow>(codes_buf, sb_buf, h_s, live, Hsum, wgt, rowb, t, out_row, rsw);
    else
        down_acc_and_store<16, kRow>(codes_buf, sb_buf, h_s, live, Hsum, wgt, rowb, t, out_row, rsw);
}

// ------------------------------------------------ fixed-order partial sum
// y[o] = sum over the U partial rows, for the 32 outputs of block blockIdx.x:
// one bulk copy brings the block's [U][32] slice into shared memory; thread
// (lane, p) adds rows p, p+8, p+16, ... in ascending order, then the 8 sums
// are added in order p = 0..7; bf16 round to nearest even.  Block 0 also sums
// the per-unit live counts into *live_total (if non-null).
__global__ void __launch_bounds__(256)
reduce_partials_kernel(const float* __restrict__ partial, int U, int hidden, uint16_t* __restrict__ y_bf16,
                       float* __restrict__ y_f32, const int* __restrict__ live_counts, int* __restrict__ live_total,
                       int* __restrict__ live_groups) {
    extern __shared__ __align__(128) float slice[];  // [U][32]
    __shared__ float part[8][33];
    __shared__ __align__(8) uint64_t bar;
    const int t = threadIdx.x;
    const int cb = blockIdx.x;
    if (t == 0) { mbar_init(&bar, 1); fence_mbar_init(); }
    __syncthreads();
    pdl_trigger();  // the next kernel may start its weight prefetch now
    pdl_wait();
    if (t == 0) {
        mbar_arrive_expect_tx(&bar, (uint32_t)U * 128u);
        const float* src = partial + (size_t)cb * U * 32;
        // pieces of at most 32 KB, 16-byte aligned (rows are 128 B)
        for (int r0 = 0; r0 < U; r0 += 256) {
            const int rows = min(256, U - r0);
            bulk_g2s(slice + (size_t)r0 * 32, src + (size_t)r0 * 32, (uint32_t)rows * 128u, &bar, policy_evict_first());
        }
    }
    const bool ok = mbar_wait(&bar, 0);
    if (!__syncthreads_and(ok)) {
        if (t == 0) mbar_wait(&bar, 0);  // the slice's copies land before the CTA leaves
        return;
    }
    const int lane = t & 31, p = t >> 5;
    float a0 = 0.f, a1 = 0.f;
    int r = p;
    for (; r + 8 < U; r += 16) {
        a0 += slice[r * 32 + lane];
        a1 += slice[(r + 8) * 32 + lane];
    }
    if (r < U) a0 += slice[r * 32 + lane];
    part[p][lane] = a0 + a1;
    __syncthreads();
    if (t < 32) {
        float y = part[0][t];
#pragma unroll
        for (int i = 1; i < 8; ++i) y += part[i][t];
        const int o = cb * 32 + t;
        if (y_f32) y_f32[o] = y;
        y_bf16[o] = f32_to_bf16_bits(y);
    }
    if ((live_total || live_groups) && cb == 0 && t == 0) {
        int n = 0, ng = 0;
        for (int u = 0; u < U; ++u) { n += live_counts[u]; ng += live_counts[u] > 0; }
        if (live_total) *live_total = n;
        if (live_groups) *live_groups = ng;
    }
}

// Failure-path self-test: the same bounded wait as every kernel's (try_wait
// with a suspend hint, clock64 limit, error word), on a barrier that nothing
// completes, with a caller-chosen limit.
__global__ void selftest_wait_kernel(long long limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    const unsigned long long t0 = clock64();
    while (!mbar_test(&bar, 0)) {
        if ((long long)(clock64() - t0) > limit) {
            atomicOr(&g_status, 1u);
            return;
        }
        __nanosleep(1000);
    }
}

}  // namespace hs

// ===================================================================== host

using namespace hs_host;

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
    v |= hs_batch_take_status();
    v |= hs_prefill_take_status();
    *status = v ? HS_ERR_TIMEOUT : HS_OK;
    return HS_OK;
}

extern "C" int hs_selftest_bounded_wait(long long limit_cycles, hs_stream_t stream) {
    if (limit_cycles < 1 || limit_cycles > (1ll << 31)) return HS_ERR_INVALID_ARG;
    hs::selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_cycles);
    return launch_err();
}

// ---------------------------------------------------------- layer decode
extern "C" size_t hs_moe_layer_decode_workspace_size(const hs_moe_layer* L, int batch) {
    if (batch > 1) {
        // the larger of the two batch paths' needs (the flags choose between them per call)
        const size_t a = batch <= hs::kMaxBatchDecode ? hs_batch_decode_workspace_size(L, batch) : 0;
        const size_t b = batch >= kPrefillMinBatch && hs_prefill_layer_ok(L, batch) == HS_OK
                             ? hs_moe_prefill_workspace_size(L, batch) : 0;
        return std::max(a, b);
    }
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
    if (!al16(x) || !al4(logits) || !al16(y_bf16) || (y_f32 && !al16(y_f32)) || !al16(ws)) return HS_ERR_MISALIGNED;
    if (batch > 1) {
        if (flags & HS_DOWN_ROW_SCALES) return HS_ERR_INVALID_ARG;  // batch 1 only
        cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        if (batch >= kPrefillMinBatch && !(flags & HS_BATCH_EXPERT_UNION) && hs_prefill_layer_ok(L, batch) == HS_OK) {
            // many tokens per expert: the prefill's tensor-core products
            if (dbg && dbg->h) return HS_ERR_INVALID_ARG;  // the h dump covers batch 1 only
            const hs_prefill_debug pd{dbg ? dbg->topk_idx : nullptr, dbg ? dbg->topk_w : nullptr, nullptr, nullptr,
                                      dbg ? dbg->live_mask : nullptr, nullptr};
            const int st = hs_moe_prefill(L, x, logits, batch, y_bf16, y_f32,
                                          flags & (HS_FORCE_DENSE | HS_PREFILL_ROW_GATHER),
                                          dbg ? &pd : nullptr, ws, ws_bytes, stream);
            if (st != HS_OK || !dbg) return st;
            return hs_prefill_union_live(L, batch, ws, dbg->live_rows, dbg->live_groups, s);
        }
        if (batch > hs::kMaxBatchDecode) return HS_ERR_UNSUPPORTED_SHAPE;
        return hs_batch_decode(L, x, logits, batch, y_bf16, y_f32, flags, dbg, ws, ws_bytes, s);
    }
    const size_t need = hs_moe_layer_decode_workspace_size(L, batch);
    if (!ws || ws_bytes < need) return HS_ERR_WORKSPACE;

    hs::LayerParams P;
    fill_layer_params(L, P);

    const int U = decode_units(L);
    hs::DecodeIO io;
    io.x = x;
    io.logits = logits;
    io.partial = static_cast<float*>(ws);
    io.live_counts = reinterpret_cast<int*>(static_cast<char*>(ws) + round_up((size_t)U * L->hidden * sizeof(float), 256));
    io.units = U;
    io.flags = flags;
    io.dbg_topk_idx = dbg ? dbg->topk_idx : nullptr;
    io.dbg_topk_w = dbg ? dbg->topk_w : nullptr;
    io.dbg_h = dbg ? dbg->h : nullptr;
    io.dbg_live = dbg ? dbg->live_mask : nullptr;
    if (io.dbg_live && ((uintptr_t)io.dbg_live & 7u)) return HS_ERR_MISALIGNED;
    int* live_out = dbg ? dbg->live_rows : nullptr;

    const int smem = hs::SmemLayout::total(L->hidden, (flags & HS_DOWN_ROW_SCALES) != 0);
    void (*kern)(const hs::LayerParams, const hs::DecodeIO) =
        (flags & HS_DOWN_ROW_SCALES) ? hs::moe_decode_b1_kernel<true> : hs::moe_decode_b1_kernel<false>;
    if (set_smem_attr((const void*)kern, smem) != HS_OK) return HS_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_pdl(kern, dim3(U), dim3(256), smem, s, P, io) != cudaSuccess) return HS_ERR_CUDA;
    if (set_smem_attr((const void*)hs::reduce_partials_kernel, U * 128) != HS_OK) return HS_ERR_CUDA;
    if (launch_pdl(hs::reduce_partials_kernel, dim3(L->hidden / 32), dim3(256), (size_t)U * 128, s,
                   (const float*)io.partial, U, L->hidden, y_bf16, y_f32, (const int*)io.live_counts,
                   live_out, dbg ? dbg->live_groups : (int*)nullptr) != cudaSuccess)
        return HS_ERR_CUDA;
    return launch_err();
}
