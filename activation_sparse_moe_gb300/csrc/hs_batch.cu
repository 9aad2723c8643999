// Activation-sparse decode of a ReLU^2 MoE layer for a small batch of tokens
// (2..64), GB300 (sm_103a).
//
// "Skipping dead neurons..." (sevren.ai): each token routes to 6 of 128
// experts plus the shared expert ("Inside a MoE layer"); with the down
// weights stored by neuron, only neurons that fired are read ("Our way reads
// only the rows that fired").  With several tokens, the tokens are grouped by
// expert ("Sorted by expert") and every expert reads the union of its tokens'
// live rows once (the verify step of section "Speculative decoding." reads
// three rows' activations through the same weights this way).
//
// Kernels (one stream, programmatic dependent launch between them):
//  1. route:  top-k + softmax per token, counting sort of (token, slot) pairs
//             by expert (tokens ascending), work-unit tables, zeroed masks.
//  2. up:     persistent CTAs over units (expert, 32 neuron rows, <= 4 tokens):
//             bulk copies of the rows, DP4A fixed-point GEMV per token, ReLU^2,
//             h to global, union live bits OR-ed into a per-(expert, 32 rows)
//             mask word.
//  3. down:   persistent CTAs over units (expert, 128-output band): the union
//             live rows' band slices, dequantised once per row, times each
//             token's h; one partial row per (token, slot).
//  4. reduce: y[t] = shared + sum_j (partial of slot j) in slot order; bf16.
#include "hs_host.h"

namespace hs {

constexpr int kTC = 4;          // tokens per up unit
constexpr int kMaxBatch = 64;
constexpr int kBand = 128;      // outputs per down unit

struct BatchMeta {
    int n_pairs, n_touched, up_units, dn_units;
    int touched[kMaxRouted];        // routed experts with tokens, ascending
    int e_off[kMaxRouted + 1];      // grouped pair offsets per expert id
    int up_off[kMaxRouted + 2];     // up unit offsets per touched index (+ shared)
    int live_cnt[kMaxRouted + 1];   // union live rows per touched index (+ shared)
    int live_grp[kMaxRouted + 1];   // groups with a union live row, same indexing
};

struct BatchIO {
    const uint16_t* x;      // [B][H]
    const float* logits;    // [B][E]
    int batch;
    unsigned flags;
    BatchMeta* meta;
    int* topk_idx;          // [B][K]
    float* topk_w;          // [B][K]
    int* pair_tok;          // [B*K] grouped by expert
    float* pair_w;
    int* pair_slot;         // 1..K
    float* h_pair;          // [B*K][NR] by grouped pair index
    float* h_sh;            // [B][NS]
    uint32_t* mask_r;       // [E][NR/32]
    uint32_t* mask_s;       // [NS/32]
    float* partial;         // [B][K+1][H]
    uint16_t* y_bf16;
    float* y_f32;
    int* dbg_topk_idx;
    float* dbg_topk_w;
    int* live_total;
    int* live_groups;
};

// ------------------------------------------------------------------ route
__global__ void __launch_bounds__(256) batch_route_kernel(const __grid_constant__ LayerParams P, const BatchIO io) {
    __shared__ int s_idx[kMaxBatch * kMaxTopK];
    __shared__ float s_w[kMaxBatch * kMaxTopK];
    __shared__ int s_cnt[kMaxRouted];
    __shared__ int s_off[kMaxRouted + 1];
    pdl_wait();
    pdl_trigger();
    const int t = threadIdx.x, warp = t >> 5;
    const int B = io.batch, K = P.top_k, E = P.n_routed;
    for (int b = warp; b < B; b += 8) warp_topk_softmax(io.logits + (size_t)b * E, E, K, s_idx + b * K, s_w + b * K);
    if (t < kMaxRouted) s_cnt[t] = 0;
    __syncthreads();
    const int npair = B * K;
    for (int p = t; p < npair; p += blockDim.x) {
        atomicAdd(&s_cnt[s_idx[p]], 1);
        io.topk_idx[p] = s_idx[p];
        io.topk_w[p] = s_w[p];
        if (io.dbg_topk_idx) { io.dbg_topk_idx[p] = s_idx[p]; io.dbg_topk_w[p] = s_w[p]; }
    }
    __syncthreads();
    BatchMeta* m = io.meta;
    if (t == 0) {
        int acc = 0, nt = 0, units = 0;
        const int HGr = P.routed_neurons / 32;
        for (int e = 0; e < E; ++e) {
            s_off[e] = acc;
            m->e_off[e] = acc;
            acc += s_cnt[e];
            if (s_cnt[e]) {
                m->touched[nt] = e;
                m->up_off[nt] = units;
                units += ((s_cnt[e] + kTC - 1) / kTC) * HGr;
                ++nt;
            }
        }
        s_off[E] = acc;
        m->e_off[E] = acc;
        m->up_off[nt] = units;
        if (P.shared_neurons) units += ((B + kTC - 1) / kTC) * (P.shared_neurons / 32);
        m->up_off[nt + 1] = units;
        m->n_pairs = npair;
        m->n_touched = nt;
        m->up_units = units;
        m->dn_units = (nt + (P.shared_neurons ? 1 : 0)) * (P.hidden / kBand);
    }
    __syncthreads();
    // place pairs: tokens ascending within an expert (pair order is token-major)
    for (int p = t; p < npair; p += blockDim.x) {
        const int e = s_idx[p];
        int rank = 0;
        for (int q = 0; q < p; ++q) rank += (s_idx[q] == e);
        const int pos = s_off[e] + rank;
        io.pair_tok[pos] = p / K;
        io.pair_w[pos] = s_w[p];
        io.pair_slot[pos] = p % K + 1;
    }
    // clear the union masks
    const int wr = P.routed_neurons / 32;
    for (int i = t; i < E * wr; i += blockDim.x) io.mask_r[i] = 0u;
    for (int i = t; i < P.shared_neurons / 32; i += blockDim.x) io.mask_s[i] = 0u;
}

// ------------------------------------------------------------------ up
struct BatchUpSmem {
    __host__ __device__ static int codes(int H) { return 32 * (H / 2); }
    __host__ __device__ static int sb(int H) { return 32 * (H / 64) * 4; }
    __host__ __device__ static int xf(int H) { return kTC * (H / 64) * kXfStride; }
    __host__ __device__ static int xs(int H) { return kTC * (H / 64) * 8; }
    // parts row stride: 1 mod 32 words, so row-sum loads (lane = row) are conflict-free
    __host__ __device__ static int pstride(int H) { return ((H / 64 + 31) / 32) * 32 + 1; }
    // x staging (bf16) and the dot-product parts share one region
    __host__ __device__ static int stage(int H) {
        const int a = kTC * H * 2, b = kTC * 32 * pstride(H) * 4;
        return a > b ? a : b;
    }
    __host__ __device__ static int total(int H) { return codes(H) + sb(H) + xf(H) + xs(H) + stage(H) + 256 + 128; }
};

__device__ __forceinline__ int unit_owner(const int* off, int n, int u) {
    // largest i in [0, n) with off[i] <= u
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(256, 2) batch_up_kernel(const __grid_constant__ LayerParams P, const BatchIO io) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int H = P.hidden, G = H / 64, rowb = H / 2;
    uint8_t* codes = smem;
    uint32_t* sbuf = reinterpret_cast<uint32_t*>(smem + BatchUpSmem::codes(H));
    uint8_t* xf_s = smem + BatchUpSmem::codes(H) + BatchUpSmem::sb(H);
    float* xs_s = reinterpret_cast<float*>(xf_s + BatchUpSmem::xf(H));
    uint8_t* stage = reinterpret_cast<uint8_t*>(xs_s) + BatchUpSmem::xs(H);
    float* parts = reinterpret_cast<float*>(stage);                      // [kTC][32][pstride]
    uint16_t* xstage = reinterpret_cast<uint16_t*>(stage);               // [kTC][H]
    float* off_s = reinterpret_cast<float*>(stage + BatchUpSmem::stage(H));  // [32]
    int* tok_s = reinterpret_cast<int*>(off_s + 32);                     // [kTC] token ids
    int* hrow_s = tok_s + kTC;                                           // [kTC] h rows
    uint64_t* bars = reinterpret_cast<uint64_t*>(off_s + 64);            // 3 barriers
    const int t = threadIdx.x;
    const bool dense = (io.flags & HS_FORCE_DENSE) != 0;
    const uint64_t pol = policy_evict_first();
    if (t == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    const BatchMeta* m = io.meta;
    const int U = m->up_units, nt = m->n_touched;
    const int pstride = BatchUpSmem::pstride(H);
    uint32_t phase = 0;
    for (int u = blockIdx.x; u < U; u += gridDim.x, phase ^= 1u) {
        // ---- which expert, rows and tokens
        const int i = unit_owner(m->up_off, nt + 1, u);
        const bool shared = (i == nt);
        const int N = shared ? P.shared_neurons : P.routed_neurons;
        const int HG = N / 32;
        const int local = u - m->up_off[i];
        const int c = local / HG, hg = local % HG;
        ExpertPtrs ep;
        int T, pbase = 0, e = -1;
        if (shared) {
            ep = P.shared;
            T = min(kTC, io.batch - c * kTC);
        } else {
            e = m->touched[i];
            ep = routed_ptrs(P, e);
            pbase = m->e_off[e] + c * kTC;
            T = min(kTC, m->e_off[e + 1] - pbase);
        }
        if (t < T) {
            tok_s[t] = shared ? c * kTC + t : io.pair_tok[pbase + t];
            hrow_s[t] = shared ? c * kTC + t : pbase + t;
        }
        if (t < 32) off_s[t] = ep.up_off ? ep.up_off[32 * hg + t] : 0.f;
        fence_proxy_async_smem();
        __syncthreads();
        if (t == 0) {
            const uint8_t* src = ep.up_codes + (size_t)(32 * hg) * rowb;
            mbar_arrive_expect_tx(&bars[0], 16 * rowb + 32 * G * 4);
            bulk_g2s(sbuf, ep.up_sb + (size_t)(32 * hg) * G, 32 * G * 4, &bars[0], pol);
            bulk_g2s(codes, src, 16 * rowb, &bars[0], pol);
            mbar_arrive_expect_tx(&bars[1], 16 * rowb);
            bulk_g2s(codes + 16 * rowb, src + (size_t)16 * rowb, 16 * rowb, &bars[1], pol);
            mbar_arrive_expect_tx(&bars[2], T * H * 2);
            for (int k = 0; k < T; ++k)
                bulk_g2s(xstage + (size_t)k * H, io.x + (size_t)tok_s[k] * H, H * 2, &bars[2], policy_evict_last());
        }
        bool ok = __syncthreads_and(mbar_wait(&bars[2], phase));
        // ---- fixed-point x tables for the T tokens (4 threads per group)
        for (int k = 0; k < T && ok; ++k)
            convert_x_fixed(xstage + (size_t)k * H, G, xf_s + (size_t)k * G * kXfStride, xs_s + (size_t)k * G * 2, 0);
        if (!__syncthreads_and(ok)) return;  // x staging is free: parts may overwrite it
        // ---- dot products: thread (gc, tk) over the 32 rows
        const int gc = t % G, tk = t / G;
        if (tk < T) {
            XFixed xf;
            load_x_fixed(xf_s + (size_t)tk * G * kXfStride, xs_s + (size_t)tk * G * 2, gc, xf);
            float* pp = parts + (size_t)tk * 32 * pstride;
            int waited = -1;
            for (int r = 0; r < 32; ++r) {
                const int kb = r >> 4;
                while (waited < kb) { ++waited; ok &= mbar_wait(&bars[waited], phase); }
                if (!ok) break;
                uint4 a0, a1;
                load_group_codes(codes + r * rowb, gc, a0, a1);
                const float2 sb = half2_to_float2(sbuf[r * G + gc]);
                const int d = group_dot_fixed16(a0, a1, xf);
                pp[r * pstride + gc] = fmaf(sb.x * xf.inv, (float)d, sb.y * xf.xsum);
            }
            while (ok && waited < 1) { ++waited; ok &= mbar_wait(&bars[waited], phase); }
        } else {
            for (int k = 0; k < 2; ++k) ok &= mbar_wait(&bars[k], phase);
        }
        if (!__syncthreads_and(ok)) return;
        // ---- row sums, ReLU^2, h out, union live bits (warp w: token w/... rows)
        {
            const int lane = t & 31, w = t >> 5;
            uint32_t anyl = 0;
            for (int k = w; k < T; k += 8) {
                const float* pp = parts + (size_t)k * 32 * pstride + lane * pstride;
                float s0 = 0.f, s1 = 0.f;
                int g = 0;
                for (; g + 1 < G; g += 2) { s0 += pp[g]; s1 += pp[g + 1]; }
                if (g < G) s0 += pp[g];
                const float z = (s0 + s1) + off_s[lane];
                const float h = z > 0.f ? z * z : 0.f;
                const int n = 32 * hg + lane;
                if (shared) io.h_sh[(size_t)hrow_s[k] * N + n] = h;
                else io.h_pair[(size_t)hrow_s[k] * N + n] = h;
                anyl |= __ballot_sync(0xffffffffu, h > 0.f);
            }
            if (lane == 0 && (anyl || dense)) {
                uint32_t* mw = shared ? io.mask_s + hg : io.mask_r + (size_t)e * HG + hg;
                atomicOr(mw, dense ? 0xffffffffu : anyl);
            }
        }
        __syncthreads();  // parts, codes and tables are reused by the next unit
    }
}

// ------------------------------------------------------------------ down
// Unit (expert i, band of 128 outputs).  Thread (oq, tl): outputs
// 4*oq .. 4*oq+3 of the band, tokens tl, tl+8, ... of the expert.  Rows are
// taken in ascending order; each live row's weights are dequantised once
// (w = s*q + b, exact in fp32) and multiplied into every token's sum.
struct BatchDownSmem {
    static constexpr int kRows = 64;  // live rows staged per pass
    __host__ __device__ static int total() {
        return kRows * 64 /*codes*/ + kRows * kMaxBatch * 4 /*h*/ + kRows * 2 /*ids*/ + 3712 / 32 * 4 + 256;
    }
};

__global__ void __launch_bounds__(256) batch_down_kernel(const __grid_constant__ LayerParams P, const BatchIO io) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int R = BatchDownSmem::kRows;
    uint8_t* cs = smem;                                               // [R][64] band code bytes
    float* hs = reinterpret_cast<float*>(smem + R * 64);              // [R][kMaxBatch]
    uint16_t* ids = reinterpret_cast<uint16_t*>(hs + R * kMaxBatch);  // [R]
    int* wpre = reinterpret_cast<int*>(ids + R);                      // prefix of live counts per mask word
    int* misc = wpre + 3712 / 32 + 2;
    const int t = threadIdx.x;
    const int H = P.hidden, K = P.top_k;
    pdl_wait();
    pdl_trigger();
    const BatchMeta* m = io.meta;
    const int nt = m->n_touched, nb = H / kBand;
    const int U = m->dn_units;
    const int oq = t & 31, tl = t >> 5;
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        const int i = u / nb, band = u % nb;
        const bool shared = (i == nt);
        const int N = shared ? P.shared_neurons : P.routed_neurons;
        const int NW = N / 32;
        ExpertPtrs ep;
        int T, pbase = 0;
        const uint32_t* mask;
        if (shared) {
            ep = P.shared;
            T = io.batch;
            mask = io.mask_s;
        } else {
            const int e = m->touched[i];
            ep = routed_ptrs(P, e);
            pbase = m->e_off[e];
            T = m->e_off[e + 1] - pbase;
            mask = io.mask_r + (size_t)e * NW;
        }
        // prefix sums of live counts per mask word (thread 0, NW <= 116)
        if (t == 0) {
            int acc = 0, ng = 0;
            for (int w = 0; w < NW; ++w) {
                const uint32_t mw = __ldcg(mask + w);
                wpre[w] = acc;
                acc += __popc(mw);
                if ((w & 1) && (mw | __ldcg(mask + w - 1))) ++ng;  // words 2g, 2g+1 cover group g
            }
            wpre[NW] = acc;
            misc[0] = acc;
            if (band == 0) { io.meta->live_cnt[i] = acc; io.meta->live_grp[i] = ng; }
        }
        __syncthreads();
        const int nlive = misc[0];
        float acc[4][kMaxBatch / 8];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < kMaxBatch / 8; ++b) acc[a][b] = 0.f;
        int cur_g = -1;
        float2 sbv[4] = {};
        for (int base = 0; base < nlive; base += R) {
            const int nr = min(R, nlive - base);
            // live row ids of this pass: each thread expands one mask word
            for (int w = t; w < NW; w += blockDim.x) {
                uint32_t bits = __ldcg(mask + w);
                int pos = wpre[w];
                while (bits) {
                    const int b = __ffs(bits) - 1;
                    bits &= bits - 1;
                    if (pos >= base && pos < base + nr) ids[pos - base] = (uint16_t)(32 * w + b);
                    ++pos;
                }
            }
            __syncthreads();
            // band code bytes of the rows (64 B each) and h of every token
            for (int q = t; q < nr * 4; q += blockDim.x) {
                const int r = q >> 2, part = q & 3;
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(ep.dn_codes + (size_t)ids[r] * (H / 2) +
                                                                     band * (kBand / 2)) + part);
                reinterpret_cast<uint4*>(cs + r * 64)[part] = v;
            }
            for (int q = t; q < nr * T; q += blockDim.x) {
                const int r = q % nr, k = q / nr;
                const int n = ids[r];
                hs[r * kMaxBatch + k] = shared ? __ldcg(io.h_sh + (size_t)k * N + n)
                                               : __ldcg(io.h_pair + (size_t)(pbase + k) * N + n);
            }
            __syncthreads();
            for (int r = 0; r < nr; ++r) {
                const int n = ids[r];
                const int g = n >> 6;
                if (g != cur_g) {
                    cur_g = g;
                    const uint4 s4 = __ldg(reinterpret_cast<const uint4*>(ep.dn_sb + (size_t)g * H + band * kBand) + oq);
                    sbv[0] = half2_to_float2(s4.x); sbv[1] = half2_to_float2(s4.y);
                    sbv[2] = half2_to_float2(s4.z); sbv[3] = half2_to_float2(s4.w);
                }
                const uint32_t cw = reinterpret_cast<const uint16_t*>(cs + r * 64)[oq];  // 4 codes
                float wv[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) wv[a] = fmaf(sbv[a].x, (float)((cw >> (4 * a)) & 15u), sbv[a].y);
#pragma unroll
                for (int b = 0; b < kMaxBatch / 8; ++b) {
                    const int k = tl + 8 * b;
                    if (k < T) {
                        const float hv = hs[r * kMaxBatch + k];
#pragma unroll
                        for (int a = 0; a < 4; ++a) acc[a][b] = fmaf(hv, wv[a], acc[a][b]);
                    }
                }
            }
            __syncthreads();
        }
        // partial rows: (token, slot) of this expert, outputs of this band
#pragma unroll
        for (int b = 0; b < kMaxBatch / 8; ++b) {
            const int k = tl + 8 * b;
            if (k < T) {
                const int tok = shared ? k : io.pair_tok[pbase + k];
                const int slot = shared ? 0 : io.pair_slot[pbase + k];
                const float wgt = shared ? 1.f : io.pair_w[pbase + k];
                float* dst = io.partial + ((size_t)tok * (K + 1) + slot) * H + band * kBand + 4 * oq;
                *reinterpret_cast<float4*>(dst) =
                    make_float4(wgt * acc[0][b], wgt * acc[1][b], wgt * acc[2][b], wgt * acc[3][b]);
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ reduce
// y[t][o] = sum over slots 0..K of partial[t][slot][o], slots ascending
// (slot 0 = shared expert, skipped without one); bf16 RNE.
__global__ void __launch_bounds__(256) batch_reduce_kernel(const __grid_constant__ LayerParams P, const BatchIO io) {
    pdl_wait();
    pdl_trigger();
    const int H = P.hidden, K = P.top_k;
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;  // float4 index over [B][H/4]
    const int B = io.batch;
    if (idx < B * (H / 4)) {
        const int tok = idx / (H / 4), c4 = idx % (H / 4);
        const float4* p = reinterpret_cast<const float4*>(io.partial + (size_t)tok * (K + 1) * H) + c4;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = P.shared_neurons ? 0 : 1; s <= K; ++s) {
            const float4 v = __ldcg(p + (size_t)s * (H / 4));
            a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
        }
        if (io.y_f32) reinterpret_cast<float4*>(io.y_f32)[idx] = a;
        const uint32_t lo = (uint32_t)f32_to_bf16_bits(a.x) | ((uint32_t)f32_to_bf16_bits(a.y) << 16);
        const uint32_t hi = (uint32_t)f32_to_bf16_bits(a.z) | ((uint32_t)f32_to_bf16_bits(a.w) << 16);
        reinterpret_cast<uint2*>(io.y_bf16)[idx] = make_uint2(lo, hi);
    }
    if ((io.live_total || io.live_groups) && blockIdx.x == 0 && threadIdx.x == 0) {
        const BatchMeta* m = io.meta;
        int n = 0, ng = 0;
        for (int i = 0; i < m->n_touched + (P.shared_neurons ? 1 : 0); ++i) { n += m->live_cnt[i]; ng += m->live_grp[i]; }
        if (io.live_total) *io.live_total = n;
        if (io.live_groups) *io.live_groups = ng;
    }
}

}  // namespace hs

// ===================================================================== host
using namespace hs_host;

namespace {
struct BatchLayout {
    size_t meta, topk_idx, topk_w, pair_tok, pair_w, pair_slot, h_pair, h_sh, mask_r, mask_s, partial, total;
};

BatchLayout batch_layout(const hs_moe_layer* L, int B) {
    const int K = L->top_k, E = L->n_routed, NR = L->routed[0].neurons;
    const int NS = L->shared ? L->shared->neurons : 0, H = L->hidden;
    BatchLayout l{};
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o += round_up(bytes, 256); return at; };
    l.meta = take(sizeof(hs::BatchMeta));
    l.topk_idx = take((size_t)B * K * 4);
    l.topk_w = take((size_t)B * K * 4);
    l.pair_tok = take((size_t)B * K * 4);
    l.pair_w = take((size_t)B * K * 4);
    l.pair_slot = take((size_t)B * K * 4);
    l.h_pair = take((size_t)B * K * NR * 4);
    l.h_sh = take((size_t)B * (NS ? NS : 1) * 4);
    l.mask_r = take((size_t)E * (NR / 32) * 4);
    l.mask_s = take((size_t)(NS ? NS / 32 : 1) * 4);
    l.partial = take((size_t)B * (K + 1) * H * 4);
    l.total = o;
    return l;
}

int batch_shape_ok(const hs_moe_layer* L, int B) {
    if (B < 2 || B > hs::kMaxBatch) return HS_ERR_UNSUPPORTED_SHAPE;
    if (L->hidden % hs::kBand) return HS_ERR_UNSUPPORTED_SHAPE;
    if (L->shared && L->shared->neurons > 3712) return HS_ERR_UNSUPPORTED_SHAPE;
    if (L->routed[0].neurons > 3712) return HS_ERR_UNSUPPORTED_SHAPE;
    return HS_OK;
}
}  // namespace

unsigned hs_batch_take_status() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, hs::g_status, sizeof(v)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(hs::g_status, &zero, sizeof(zero));
    return v;
}

size_t hs_batch_decode_workspace_size(const hs_moe_layer* L, int batch) {
    if (check_layer(L) != HS_OK || batch_shape_ok(L, batch) != HS_OK) return 0;
    return batch_layout(L, batch).total;
}

int hs_batch_decode(const hs_moe_layer* L, const uint16_t* x, const float* logits, int batch, uint16_t* y_bf16,
                    float* y_f32, unsigned flags, const hs_decode_debug* dbg, void* ws, size_t ws_bytes,
                    cudaStream_t s) {
    int st = batch_shape_ok(L, batch);
    if (st != HS_OK) return st;
    if (dbg && dbg->h) return HS_ERR_INVALID_ARG;  // the h dump covers batch 1 only
    const BatchLayout l = batch_layout(L, batch);
    if (!ws || ws_bytes < l.total) return HS_ERR_WORKSPACE;
    char* w = static_cast<char*>(ws);
    hs::LayerParams P;
    fill_layer_params(L, P);
    hs::BatchIO io{};
    io.x = x;
    io.logits = logits;
    io.batch = batch;
    io.flags = flags;
    io.meta = reinterpret_cast<hs::BatchMeta*>(w + l.meta);
    io.topk_idx = reinterpret_cast<int*>(w + l.topk_idx);
    io.topk_w = reinterpret_cast<float*>(w + l.topk_w);
    io.pair_tok = reinterpret_cast<int*>(w + l.pair_tok);
    io.pair_w = reinterpret_cast<float*>(w + l.pair_w);
    io.pair_slot = reinterpret_cast<int*>(w + l.pair_slot);
    io.h_pair = reinterpret_cast<float*>(w + l.h_pair);
    io.h_sh = reinterpret_cast<float*>(w + l.h_sh);
    io.mask_r = reinterpret_cast<uint32_t*>(w + l.mask_r);
    io.mask_s = reinterpret_cast<uint32_t*>(w + l.mask_s);
    io.partial = reinterpret_cast<float*>(w + l.partial);
    io.y_bf16 = y_bf16;
    io.y_f32 = y_f32;
    io.dbg_topk_idx = dbg ? dbg->topk_idx : nullptr;
    io.dbg_topk_w = dbg ? dbg->topk_w : nullptr;
    io.live_total = dbg ? dbg->live_rows : nullptr;
    io.live_groups = dbg ? dbg->live_groups : nullptr;

    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return HS_ERR_CUDA;
    const int up_smem = hs::BatchUpSmem::total(L->hidden);
    const int dn_smem = hs::BatchDownSmem::total();
    if (set_smem_attr((const void*)hs::batch_up_kernel, up_smem) != HS_OK) return HS_ERR_CUDA;
    if (set_smem_attr((const void*)hs::batch_down_kernel, dn_smem) != HS_OK) return HS_ERR_CUDA;
    if (launch_pdl(hs::batch_route_kernel, dim3(1), dim3(256), 0, s, P, io) != cudaSuccess) return HS_ERR_CUDA;
    if (launch_pdl(hs::batch_up_kernel, dim3(2 * sms), dim3(256), up_smem, s, P, io) != cudaSuccess) return HS_ERR_CUDA;
    if (launch_pdl(hs::batch_down_kernel, dim3(2 * sms), dim3(256), dn_smem, s, P, io) != cudaSuccess)
        return HS_ERR_CUDA;
    const int nred = (batch * (L->hidden / 4) + 255) / 256;
    if (launch_pdl(hs::batch_reduce_kernel, dim3(nred), dim3(256), 0, s, P, io) != cudaSuccess) return HS_ERR_CUDA;
    return launch_err();
}
