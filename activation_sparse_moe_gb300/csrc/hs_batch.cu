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
// B <= 8 (batch_small_kernel + batch_fused_reduce_kernel, from 3 tokens
// after batch_small_plan_kernel): one CTA per (expert, 64-neuron group, up to
// 4 of the expert's tokens) unit, numbered before routing; the plan kernel
// routes the batch once and packs every token's fixed-point x table, and with
// 2 tokens every CTA routes the batch itself.  No meta block; programmatic
// dependent launch between the kernels.
//
// B <= 64 (batch_route_kernel, batch_fused_kernel, batch_fused_reduce_kernel):
// routing and planning first, then persistent CTAs take (expert, group, up to
// 4 tokens) units by an atomic ticket.
//
// HS_BATCH_EXPERT_UNION, every expert reading the union of all its tokens'
// live rows once (one stream; the meta block is zeroed first, then
// programmatic dependent launch between the kernels):
//  1. route:  one CTA per token: top-k + softmax (warp 0), per-expert pair
//             counts (integer atomics), and the token's fixed-point x table
//             for the integer-pipe GEMV (all threads).  The last CTA to finish
//  2. plans:  pair offsets, (token, slot) pairs grouped by expert in token
//             order, work-unit tables, zeroed union masks.
//  3. up:     four persistent CTAs per SM over units (expert, 32 neuron rows,
//             <= 2 tokens) handed out by an atomic ticket, shared expert first:
//             two chunked bulk copies per unit, DP4A fixed-point
//             GEMV per token, ReLU^2, h to global, union live bits OR-ed into
//             per-(expert, 32 rows) mask words.
//  4. down:   persistent CTAs over units (expert or shared-expert row chunk,
//             128-output band): the union live rows' band slices (and the
//             scale slabs of their groups) staged by asynchronous copies, two
//             passes in flight; each live row's weights dequantised once and
//             multiplied by every token's h; one partial row per (token, slot).
//  5. reduce: y[t] = sum of the token's partial rows in slot order; bf16.
#include "hs_host.h"

#include <algorithm>

namespace hs {

constexpr int kTC = 2;          // tokens per up unit
constexpr int kUpRows = 32;     // neuron rows per up unit (two 16-row chunks)
constexpr int kUpThreads = 128; // threads of an up CTA
constexpr int kUpCtasPerSm = 4;
constexpr int kFusedMaxBatch = 64;  // batches up to this size take the fused path (unless HS_BATCH_EXPERT_UNION)
constexpr int kFTok = 4;            // tokens per fused unit
constexpr int kMaxBatch = 64;
constexpr int kBand = 128;      // outputs per down unit
constexpr int kMaxShChunks = 8; // shared-expert row chunks in the down pass

// Row chunks of the shared expert's down product: the shared expert has every
// token of the batch and the widest union of live rows, so its work is split
// into ranges of rows (each a separate work item with its own partial rows).
__host__ __device__ inline int shared_chunks(int B) { return B > 0 ? kMaxShChunks : 0; }

struct BatchMeta {
    int cnt[kMaxRouted];            // pairs per expert (route kernel, atomics)
    int n_pairs, n_touched, up_units, dn_units, n_items;
    int up_shared;                  // shared-expert up units (numbered first)
    int up_next;                    // next up unit to hand out (atomic ticket)
    int fu_off[kMaxRouted + 1];     // fused-path unit offsets per touched index
    int fu_units, fu_shared, fu_next;
    int route_done;                 // route CTAs finished (the last one plans the batch)
    int touched[kMaxRouted];        // routed experts with tokens, ascending
    int e_off[kMaxRouted + 1];      // grouped pair offsets per expert id
    int up_off[kMaxRouted + 2];     // up unit offsets per touched index (+ shared)
    int live_cnt[kMaxRouted + 1];   // union live rows per touched index (+ shared)
    int live_grp[kMaxRouted + 1];   // groups with a union live row, same indexing
};

struct SmallPlan;

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
    uint8_t* xt;            // [B][G][kXfStride] fixed-point x tables ([B][G][128], packed, on the small-batch path)
    float* xsc;             // [B][G][2] (scale, sum) per group
    float* h_pair;          // [B*K][NR] by grouped pair index
    float* h_sh;            // [B][NS]
    uint32_t* mask_r;       // [E][NR/32]
    uint32_t* mask_s;       // [NS/32]
    float* partial;         // [B][S][H], S = shared chunks + K slots
    uint16_t* y_bf16;
    float* y_f32;
    int* dbg_topk_idx;
    float* dbg_topk_w;
    int* live_total;
    int* live_groups;
    uint64_t* dbg_live;     // [B][Ut] live mask (h > 0) per (token, slot group), or null
    SmallPlan* small_plan;  // small-batch path: the batch's routed entries
    uint64_t* unit_live;    // small-batch path: live mask per unit (else null)
    int* unit_key;          // small-batch path: the unit's expert (n_routed = shared, -1 = none)
    int n_units;
};

// ------------------------------------------------------------------ plan
// Inclusive sum over the threads of a CTA of at most 32 warps; `tmp` holds 32 ints.
__device__ __forceinline__ int block_incl_sum(int v, int* tmp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) tmp[warp] = v;
    __syncthreads();
    int before = 0;
    for (int i = 0; i < warp && i < nw; ++i) before += tmp[i];
    __syncthreads();
    return v + before;
}

// Run by the last route CTA to finish: pair offsets per expert, the touched
// experts, the unit tables of both paths, the pairs grouped by expert in
// token order, and cleared union masks.
__device__ __noinline__ void batch_plan(const LayerParams& P, const BatchIO& io) {
    __shared__ int s_idx[kMaxBatch * kMaxTopK];
    __shared__ int s_off[kMaxRouted + 1];
    __shared__ int tmp[32];
    __shared__ int tot[4];
    const int t = threadIdx.x;
    const int B = io.batch, K = P.top_k, E = P.n_routed;
    const int npair = B * K;
    BatchMeta* m = io.meta;
    for (int p = t; p < npair; p += blockDim.x) s_idx[p] = __ldcg(io.topk_idx + p);
    // offsets, touched experts and unit offsets: block scans over the experts (thread e)
    const int HGr = P.routed_neurons / kUpRows;
    const int c = t < E ? __ldcg(&m->cnt[t]) : 0;
    const int touched = c > 0 ? 1 : 0;
    const int units = ((c + kTC - 1) / kTC) * HGr;
    const int c_in = block_incl_sum(c, tmp);
    const int t_in = block_incl_sum(touched, tmp);
    const int u_in = block_incl_sum(units, tmp);
    const int funits = ((c + kFTok - 1) / kFTok) * (P.routed_neurons / 64);
    const int f_in = block_incl_sum(funits, tmp);
    if (t < E) {
        s_off[t] = c_in - c;
        m->e_off[t] = c_in - c;
        if (touched) {
            m->touched[t_in - 1] = t;
            m->up_off[t_in - 1] = u_in - units;
            m->fu_off[t_in - 1] = f_in - funits;
        }
    }
    if (t == E - 1) { tot[0] = c_in; tot[1] = t_in; tot[2] = u_in; tot[3] = f_in; }
    __syncthreads();
    if (t == 0) {
        const int nt = tot[1];
        int un = tot[2];
        s_off[E] = tot[0];
        m->e_off[E] = tot[0];
        m->up_off[nt] = un;
        const int su = P.shared_neurons ? ((B + kTC - 1) / kTC) * (P.shared_neurons / kUpRows) : 0;
        m->up_off[nt + 1] = un + su;
        m->n_pairs = npair;
        m->n_touched = nt;
        m->up_units = un + su;
        m->up_shared = su;
        m->n_items = nt + (P.shared_neurons ? shared_chunks(B) : 0);
        m->dn_units = m->n_items * (P.hidden / kBand);
        const int fsu = P.shared_neurons ? ((B + kFTok - 1) / kFTok) * (P.shared_neurons / 64) : 0;
        m->fu_off[nt] = tot[3];
        m->fu_shared = fsu;
        m->fu_units = tot[3] + fsu;
    }
    __syncthreads();
    // place pairs: tokens ascending within an expert (pair order is token-major)
    for (int p = t; p < npair; p += blockDim.x) {
        const int e = s_idx[p];
        int rank = 0;
        for (int q = 0; q < p; ++q) rank += (s_idx[q] == e);
        const int pos = s_off[e] + rank;
        io.pair_tok[pos] = p / K;
        io.pair_w[pos] = __ldcg(io.topk_w + p);
        io.pair_slot[pos] = p % K + 1;
    }
    // clear the union masks
    const int wr = P.routed_neurons / 32;
    for (int i = t; i < E * wr; i += blockDim.x) io.mask_r[i] = 0u;
    for (int i = t; i < P.shared_neurons / 32; i += blockDim.x) io.mask_s[i] = 0u;
}

// ------------------------------------------------------------------ route
__global__ void __launch_bounds__(256) batch_route_kernel(const __grid_constant__ LayerParams P, const BatchIO io) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x, t = threadIdx.x;
    const int K = P.top_k, E = P.n_routed, H = P.hidden, G = H / 64;
    if (t < 32) {
        const TopkPick pk = warp_topk_softmax(io.logits + (size_t)b * E, E, K, io.topk_idx + (size_t)b * K,
                                              io.topk_w + (size_t)b * K);
        if (t < K) {   // lane j holds choice j
            const int p = b * K + t;
            atomicAdd(&io.meta->cnt[pk.idx], 1);
            if (io.dbg_topk_idx) io.dbg_topk_idx[p] = pk.idx;
            if (io.dbg_topk_w) io.dbg_topk_w[p] = pk.w;
        }
    }
    // the token's fixed-point x table (read by every up unit that has this token)
    convert_x_fixed(io.x + (size_t)b * H, G, io.xt + (size_t)b * G * kXfStride, io.xsc + (size_t)b * G * 2, 0);
    // the last CTA to finish plans the batch (no CTA waits for another)
    __shared__ int last;
    __threadfence();   // this CTA's top-k, counts and x table before its increment
    __syncthreads();
    if (t == 0) last = atomicAdd(&io.meta->route_done, 1) == io.batch - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    batch_plan(P, io);
}

// ------------------------------------------------------------------ up
// Unit = (expert, kUpRows neurons, up to kTC of the expert's tokens).  Four
// small CTAs per SM, each working through units in turn: the unit's up rows
// are bulk-copied in 16-row chunks (scales with the first) so the dot
// products start on the first chunk while the rest is in flight, and the
// other CTAs of the SM compute while this one waits.
struct BatchUpSmem {
    __host__ __device__ static int codes(int H) { return kUpRows * (H / 2); }
    __host__ __device__ static int sb(int H) { return kUpRows * (H / 64) * 4; }
    __host__ __device__ static int total(int H);
};

struct UpUnitDesc {
    bool shared;
    int e, c, g, T, pbase, N, NG;
    ExpertPtrs ep;
};

// The unit tables of the meta block, copied into shared memory once per CTA.
struct MetaTables {
    int up_off[kMaxRouted + 2];
    int touched[kMaxRouted];
    int e_off[kMaxRouted + 1];
};

__host__ __device__ inline int BatchUpSmem::total(int H) {
    return codes(H) + sb(H) + 64 + (int)sizeof(MetaTables) + kUpRows * 4;
}

__device__ __forceinline__ void load_tables(const BatchMeta* m, int nt, int E, MetaTables* s) {
    for (int i = threadIdx.x; i < nt + 2; i += blockDim.x) s->up_off[i] = __ldcg(&m->up_off[i]);
    for (int i = threadIdx.x; i < nt; i += blockDim.x) s->touched[i] = __ldcg(&m->touched[i]);
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s->e_off[i] = __ldcg(&m->e_off[i]);
}

__device__ __forceinline__ int unit_owner(const int* off, int n, int u) {
    // largest i in [0, n) with off[i] <= u
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Units 0 .. su-1 are the shared expert's (the heaviest, handed out first),
// then the routed experts' in the order of the unit table.
__device__ __forceinline__ UpUnitDesc up_unit_desc(const LayerParams& P, const BatchIO& io, const MetaTables* tb, int nt,
                                                   int su, int u) {
    UpUnitDesc d;
    d.shared = u < su;
    const int i = d.shared ? nt : unit_owner(tb->up_off, nt, u - su);
    d.N = d.shared ? P.shared_neurons : P.routed_neurons;
    d.NG = d.N / kUpRows;
    const int local = d.shared ? u : u - su - tb->up_off[i];
    d.c = local / d.NG;
    d.g = local % d.NG;
    if (d.shared) {
        d.e = -1;
        d.ep = P.shared;
        d.pbase = d.c * kTC;
        d.T = min(kTC, io.batch - d.c * kTC);
    } else {
        d.e = tb->touched[i];
        d.ep = routed_ptrs(P, d.e);
        d.pbase = tb->e_off[d.e] + d.c * kTC;
        d.T = min(kTC, tb->e_off[d.e + 1] - d.pbase);
    }
    return d;
}

// This thread's role in a unit of T <= 2 tokens: token lane tk (the TL lanes
// of one scale group are adjacent in a warp), group gc, row lane rs of RS.
struct UpRole {
    int tk, gc, rs, RS, TL;
    bool active;  // owns (token, group) work
};
__device__ __forceinline__ UpRole up_role(int T, int G) {
    UpRole r;
    const int t = threadIdx.x;
    r.TL = T == 1 ? 1 : 2;
    r.RS = kUpThreads / (r.TL * G);
    r.tk = t % r.TL;
    r.gc = (t / r.TL) % G;
    r.rs = t / (r.TL * G);
    r.active = r.rs < r.RS && r.tk < T;
    return r;
}

// Where the dot product of (row r, group gc, token lane tk) is left: word
// (tk + gc/4 + r) % 8 of the group's own 32-byte code block, once every lane
// of the group has read the codes.
__device__ __forceinline__ float* up_part(uint8_t* codes, int rowb, int r, int gc, int tk) {
    return reinterpret_cast<float*>(codes + r * rowb + 32 * gc + 4 * ((tk + (gc >> 2) + r) & 7));
}

__global__ void __launch_bounds__(kUpThreads, kUpCtasPerSm) batch_up_kernel(const __grid_constant__ LayerParams P, const BatchIO io) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int H = P.hidden, G = H / 64, rowb = H / 2;
    uint8_t* codes = smem;
    uint32_t* sbs = reinterpret_cast<uint32_t*>(smem + BatchUpSmem::codes(H));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BatchUpSmem::codes(H) + BatchUpSmem::sb(H));
    MetaTables* tb = reinterpret_cast<MetaTables*>(bars + 8);
    float* offs_s = reinterpret_cast<float*>(tb + 1);  // [kUpRows] offsets of the unit's rows
    int* ticket_s = reinterpret_cast<int*>(bars + 4);   // the next unit of this CTA
    const int t = threadIdx.x, lane = t & 31;
    const bool dense = (io.flags & HS_FORCE_DENSE) != 0;
    if (t == 0) {
        for (int i = 0; i < kUpRows / 16; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    BatchMeta* m = io.meta;
    const int U = __ldcg(&m->up_units), nt = __ldcg(&m->n_touched), su = __ldcg(&m->up_shared);
    load_tables(m, nt, P.n_routed, tb);
    // units are handed out one at a time (heaviest first), so CTAs that drew
    // compute-heavy units take fewer of them
    if (t == 0) *ticket_s = atomicAdd(&m->up_next, 1);
    __syncthreads();
    const uint64_t pol = policy_evict_first();
    for (int it = 0;; ++it) {
        const int u = *ticket_s;
        if (u >= U) break;
        const UpUnitDesc d = up_unit_desc(P, io, tb, nt, su, u);
        const uint32_t par = it & 1;
        __syncthreads();  // every thread has read the ticket before the next one lands
        // the next ticket, fetched while this unit streams (read after the unit's last barrier)
        if (t == blockDim.x - 1) *ticket_s = atomicAdd(&m->up_next, 1);
        if (t == 0) {
            const uint8_t* src = d.ep.up_codes + (size_t)d.g * kUpRows * rowb;
            const uint32_t chunk = 16 * rowb;
            mbar_arrive_expect_tx(&bars[0], chunk + kUpRows * G * 4);
            bulk_g2s(sbs, d.ep.up_sb + (size_t)d.g * kUpRows * G, kUpRows * G * 4, &bars[0], pol);
            bulk_g2s(codes, src, chunk, &bars[0], pol);
            for (int k = 1; k < kUpRows / 16; ++k) {
                mbar_arrive_expect_tx(&bars[k], chunk);
                bulk_g2s(codes + k * chunk, src + (size_t)k * chunk, chunk, &bars[k], pol);
            }
        }
        const UpRole role = up_role(d.T, G);
        XFixed xf = {};
        if (role.active) {
            const int tok = d.shared ? d.pbase + role.tk : __ldcg(io.pair_tok + d.pbase + role.tk);
            load_x_fixed(io.xt + (size_t)tok * G * kXfStride, io.xsc + (size_t)tok * G * 2, role.gc, xf);
        }
        if (t < kUpRows) offs_s[t] = d.ep.up_off ? __ldg(d.ep.up_off + kUpRows * d.g + t) : 0.f;
        // ---- dot products: rows rs, rs + RS, ... two at a time, chunk by chunk.
        // Every thread runs the same number of steps (the warp synchronises
        // inside); threads without a row in a step only keep step.
        bool ok = true;
        int waited = -1;
        const int n_steps = (kUpRows + 2 * role.RS - 1) / (2 * role.RS);
        for (int i = 0; i < n_steps; ++i) {
            const int r = role.rs + 2 * role.RS * i, r2 = r + role.RS;
            const bool act = role.rs < role.RS && r < kUpRows;
            const bool two = act && r2 < kUpRows;
            if (act) {
                const int k = (two ? r2 : r) >> 4;
                while (ok && waited < k) { ++waited; ok = mbar_wait(&bars[waited], par); }
            }
            uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0, b0 = a0, b1 = a0;
            uint32_t sw0 = 0, sw1 = 0;
            if (act && ok) {
                load_group_codes(codes + r * rowb, role.gc, a0, a1);
                sw0 = sbs[r * G + role.gc];
                if (two) {
                    load_group_codes(codes + r2 * rowb, role.gc, b0, b1);
                    sw1 = sbs[r2 * G + role.gc];
                }
            }
            const int da = group_dot_fixed16(a0, a1, xf);
            const int db = group_dot_fixed16(b0, b1, xf);
            // the token lanes of a group have all read its codes before any part lands there
            __syncwarp();
            if (act && ok && role.active) {
                const float2 sa = half2_to_float2(sw0);
                *up_part(codes, rowb, r, role.gc, role.tk) = fmaf(sa.x * xf.inv, (float)da, sa.y * xf.xsum);
                if (two) {
                    const float2 sbv = half2_to_float2(sw1);
                    *up_part(codes, rowb, r2, role.gc, role.tk) = fmaf(sbv.x * xf.inv, (float)db, sbv.y * xf.xsum);
                }
            }
        }
        while (ok && waited < kUpRows / 16 - 1) { ++waited; ok = mbar_wait(&bars[waited], par); }
        if (!__syncthreads_and(ok)) {
            // a wait gave up (the error word is set): the unit's copies land before the CTA leaves
            if (t == 0)
                for (int i = 0; i < kUpRows / 16; ++i) mbar_wait(&bars[i], par);
            return;
        }
        // ---- row sums, ReLU^2, h out, union live bits: pass pt covers (row, token) pairs
        // (row t/4, token pt); four threads per pair add groups q, q+4, ... in two chains
        for (int pt = 0; pt < d.T; ++pt) {
            const int r = (t >> 2), q = t & 3, tk = pt;
            float s0 = 0.f, s1 = 0.f;
            int cc = q;
            for (; cc + 4 < G; cc += 8) {
                s0 += *up_part(codes, rowb, r, cc, tk);
                s1 += *up_part(codes, rowb, r, cc + 4, tk);
            }
            if (cc < G) s0 += *up_part(codes, rowb, r, cc, tk);
            float sum = s0 + s1;
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            const float z = sum + offs_s[r];
            const float h = z > 0.f ? z * z : 0.f;
            const int n = kUpRows * d.g + r;
            if (q == 0) {
                if (d.shared) io.h_sh[(size_t)(d.pbase + tk) * d.N + n] = h;
                else io.h_pair[(size_t)(d.pbase + tk) * d.N + n] = h;
            }
            if (io.dbg_live) {  // this token's own live bits (h > 0) for the warp's 8 rows
                const unsigned bt = __ballot_sync(0xffffffffu, q == 0 && h > 0.f);
                if (lane == 0 && bt) {
                    unsigned m8 = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) m8 |= ((bt >> (4 * i)) & 1u) << i;
                    const int r8 = kUpRows * d.g + 8 * (t >> 5);  // neuron of the warp's first row
                    const int Ut = P.shared_neurons / 64 + P.top_k * (P.routed_neurons / 64);
                    int tok, uidx;
                    if (d.shared) {
                        tok = d.pbase + tk;
                        uidx = r8 >> 6;
                    } else {
                        tok = __ldcg(io.pair_tok + d.pbase + tk);
                        uidx = P.shared_neurons / 64 + (__ldcg(io.pair_slot + d.pbase + tk) - 1) * (d.N / 64) + (r8 >> 6);
                    }
                    uint32_t* mw = reinterpret_cast<uint32_t*>(io.dbg_live + (size_t)tok * Ut + uidx) + ((r8 & 63) >> 5);
                    atomicOr(mw, m8 << (r8 & 31));
                }
            }
            const unsigned bl = __ballot_sync(0xffffffffu, q == 0 && (dense || h > 0.f));
            if (lane == 0 && bl) {
                unsigned m8 = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) m8 |= ((bl >> (4 * i)) & 1u) << i;
                // this warp's 8 rows: r = 8 (t / 32) .. + 7 of the unit
                const int r8 = kUpRows * d.g + 8 * (t >> 5);
                uint32_t* mw = d.shared ? io.mask_s + (r8 >> 5) : io.mask_r + (size_t)d.e * (d.N / 32) + (r8 >> 5);
                atomicOr(mw, m8 << (r8 & 31));
            }
        }
        fence_proxy_async_smem();  // the parts in the code buffer come before the next unit's copies
        __syncthreads();           // the code buffer, the parts and the offsets are reused by the next unit
    }
}

// ------------------------------------------------------------------ down
// Unit (item i, band of 128 outputs); an item is a touched routed expert or a
// row chunk of the shared expert.  The live rows come from the union mask
// (parallel prefix over the mask words); their band code bytes and their
// tokens' h are staged by cp.async, two passes of kRows rows in flight; the
// (scale, bias) slab slices of the live groups are staged once per unit.
// Thread (oq, warp): outputs 4*oq .. 4*oq+3 of the band.  With more than 8
// tokens, warp w takes tokens w, w+8, ... over all rows; with at most 8, warp
// w takes a fixed eighth of the rows (by mask word) for every token, streams
// its live rows through its own buffer, and the 8 warps' sums are added in a
// fixed order at the end.  Every split is by row index, never by position in
// the live list, so the sparse and the dense (all rows live) results are
// bit-identical: a dead row adds exact zeros.
struct BatchDownSmem {
    static constexpr int kRows = 64;                  // live rows per pass
    static constexpr int kMaxWords = 3712 / 32;       // mask words of the widest expert
    static constexpr int kMaxGroups = 3712 / 64;
    static constexpr int kCodes = kRows * 64;         // band bytes of the rows of a pass
    static constexpr int kH = kRows * kMaxBatch * 4;  // h of the rows of a pass
    static constexpr int kPass = kCodes + kH;
    static constexpr int kSlab = kMaxGroups * kBand * 4;
    static constexpr int kIds = 3712 * 2;
    static int total();
};
constexpr int kWarpRows = 16;                                  // rows per chunk of a warp's own pipeline
constexpr int kWarpBuf = 2 * (kWarpRows * 64 + kWarpRows * 8 * 4);  // two stages: codes + h of <= 8 tokens
static_assert(8 * kWarpBuf <= 2 * BatchDownSmem::kPass, "per-warp buffers fit in the pass buffers");

inline int BatchDownSmem::total() { return 2 * kPass + kSlab + kIds + (kMaxWords + 1) * 4 * 2 + (int)sizeof(MetaTables) + 64; }

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__global__ void __launch_bounds__(256) batch_down_kernel(const __grid_constant__ LayerParams P, const BatchIO io) {
    extern __shared__ __align__(128) uint8_t smem[];
    using S = BatchDownSmem;
    constexpr int R = S::kRows;
    uint8_t* pass_buf = smem;                                             // [2][kPass]
    uint32_t* slab = reinterpret_cast<uint32_t*>(smem + 2 * S::kPass);    // [group][128] (scale, bias)
    uint16_t* ids = reinterpret_cast<uint16_t*>(smem + 2 * S::kPass + S::kSlab);
    uint32_t* words = reinterpret_cast<uint32_t*>(ids + 3712);            // [kMaxWords + 1]
    int* wpre = reinterpret_cast<int*>(words + S::kMaxWords + 1);         // [kMaxWords + 1]
    MetaTables* tb = reinterpret_cast<MetaTables*>(wpre + S::kMaxWords + 1);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int H = P.hidden, B = io.batch;
    const int SC = P.shared_neurons ? shared_chunks(B) : 0;
    const int NSl = SC + P.top_k;
    pdl_wait();
    pdl_trigger();
    const BatchMeta* m = io.meta;
    const int nt = __ldcg(&m->n_touched), nb = H / kBand;
    const int U = __ldcg(&m->dn_units);
    const int oq = lane;
    load_tables(m, nt, P.n_routed, tb);
    __syncthreads();
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        const int i = u / nb, band = u % nb;
        const bool shared = (i >= nt);
        const int chunk = shared ? i - nt : 0;
        const int N = shared ? P.shared_neurons : P.routed_neurons;
        const int NW = N / 32;
        ExpertPtrs ep;
        int T, pbase = 0;
        const uint32_t* mask;
        if (shared) {
            ep = P.shared;
            T = B;
            mask = io.mask_s;
        } else {
            const int e = tb->touched[i];
            ep = routed_ptrs(P, e);
            pbase = tb->e_off[e];
            T = tb->e_off[e + 1] - pbase;
            mask = io.mask_r + (size_t)e * NW;
        }
        // ---- union live rows: mask words, prefix counts (warp 0), row ids
        if (t < NW) words[t] = __ldcg(mask + t);
        __syncthreads();
        if (warp == 0) {
            int c[4], s = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int w = 4 * lane + j;
                c[j] = w < NW ? __popc(words[w]) : 0;
                s += c[j];
            }
            int incl = s;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            int run = incl - s;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int w = 4 * lane + j;
                if (w < NW) wpre[w] = run;
                run += c[j];
            }
            if (lane == 31) wpre[NW] = incl;
        }
        __syncthreads();
        const int nlive = wpre[NW];
        // this item's live rows: a shared-expert chunk owns the rows of a fixed range of mask
        // words (by row index, so that the summation order does not depend on which rows are live)
        const int w_lo = shared ? NW * chunk / SC : 0, w_hi = shared ? NW * (chunk + 1) / SC : NW;
        const int lo = wpre[w_lo], hi = wpre[w_hi];
        if (t >= w_lo && t < w_hi) {
            uint32_t bits = words[t];
            int pos = wpre[t] - lo;
            while (bits) {
                const int bb = __ffs(bits) - 1;
                bits &= bits - 1;
                ids[pos++] = (uint16_t)(32 * t + bb);
            }
        }
        if (t == 0 && band == 0 && chunk == 0) {
            int ng = 0;
            for (int g = 0; g < NW / 2; ++g) ng += (words[2 * g] | words[2 * g + 1]) != 0u;
            io.meta->live_cnt[shared ? nt : i] = nlive;
            io.meta->live_grp[shared ? nt : i] = ng;
        }
        // slab slices of the groups holding a live row
        for (int q = t; q < (N / 64) * 32; q += blockDim.x) {
            const int g = q >> 5, part = q & 31;
            if (words[2 * g] | words[2 * g + 1])
                cp_async16(slab + g * kBand + 4 * part, ep.dn_sb + (size_t)g * H + band * kBand + 4 * part);
        }
        cp_async_commit();
        __syncthreads();
        const int nrows = hi - lo;
        float acc[4][kMaxBatch / 8];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < kMaxBatch / 8; ++b) acc[a][b] = 0.f;
        const bool rows_split = T <= 8;
        // dequantise row n's 4 weights of this thread's outputs (group scales from the slab)
        int cur_g = -1;
        float2 sbv[4] = {};
        auto weights = [&](int n, uint32_t cw, float (&wv)[4]) {
            const int g = n >> 6;
            if (g != cur_g) {
                cur_g = g;
                const uint4 s4 = *reinterpret_cast<const uint4*>(slab + g * kBand + 4 * oq);
                sbv[0] = half2_to_float2(s4.x); sbv[1] = half2_to_float2(s4.y);
                sbv[2] = half2_to_float2(s4.z); sbv[3] = half2_to_float2(s4.w);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                // the code as an exact float: (2^23 + q) - 2^23
                const float qf = __uint_as_float(0x4B000000u | ((cw >> (4 * a)) & 15u)) - 8388608.f;
                wv[a] = fmaf(sbv[a].x, qf, sbv[a].y);
            }
        };
        if (rows_split) {
            // ---- few tokens: warp w owns a fixed range of rows (mask words) and streams its own
            // live rows through a private double buffer of kWarpRows rows
            constexpr int WR = kWarpRows;
            uint8_t* wb = pass_buf + warp * kWarpBuf;
            const int ww_lo = w_lo + (w_hi - w_lo) * warp / 8, ww_hi = w_lo + (w_hi - w_lo) * (warp + 1) / 8;
            const int r_lo = wpre[ww_lo] - lo, r_hi = wpre[ww_hi] - lo;
            const int nchunk = (r_hi - r_lo + WR - 1) / WR;
            auto prefetch_w = [&](int c) {
                uint8_t* st = wb + (c & 1) * (kWarpBuf / 2);
                float* hbw = reinterpret_cast<float*>(st + WR * 64);
                const int r0 = r_lo + c * WR, nr = min(WR, r_hi - r0);
                for (int q = lane; q < nr * 4; q += 32) {
                    const int r = q >> 2, part = q & 3;
                    cp_async16(st + r * 64 + 16 * part,
                               ep.dn_codes + (size_t)ids[r0 + r] * (H / 2) + band * (kBand / 2) + 16 * part);
                }
                for (int q = lane; q < nr * T; q += 32) {
                    const int r = q % nr, k = q / nr;
                    const int n = ids[r0 + r];
                    cp_async4(hbw + r * 8 + k,
                              shared ? io.h_sh + (size_t)k * N + n : io.h_pair + (size_t)(pbase + k) * N + n);
                }
                cp_async_commit();
            };
            if (nchunk > 0) prefetch_w(0);
            // the slab copies (every thread's first group) are complete and visible to all warps
            if (nchunk > 0) cp_async_wait<1>(); else cp_async_wait<0>();
            __syncthreads();
            for (int c = 0; c < nchunk; ++c) {
                if (c + 1 < nchunk) {
                    prefetch_w(c + 1);
                    cp_async_wait<1>();
                } else {
                    cp_async_wait<0>();
                }
                __syncwarp();
                const uint8_t* st = wb + (c & 1) * (kWarpBuf / 2);
                const float* hbw = reinterpret_cast<const float*>(st + WR * 64);
                const int r0 = r_lo + c * WR, nr = min(WR, r_hi - r0);
                for (int r = 0; r < nr; ++r) {
                    float wv[4];
                    weights(ids[r0 + r], reinterpret_cast<const uint16_t*>(st + r * 64)[oq], wv);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        if (k < T) {
                            const float hv = hbw[r * 8 + k];
#pragma unroll
                            for (int a = 0; a < 4; ++a) acc[a][k] = fmaf(hv, wv[a], acc[a][k]);
                        }
                    }
                }
                __syncwarp();
            }
            __syncthreads();  // every warp is done with its buffer before the reduction reuses them
        } else {
            // ---- many tokens: CTA-wide passes of R rows, warp w takes tokens w, w + 8, ...
            const int npass = (nrows + R - 1) / R;
            auto prefetch = [&](int p) {
                uint8_t* pb = pass_buf + (p & 1) * S::kPass;
                float* hb = reinterpret_cast<float*>(pb + S::kCodes);
                const int r0 = p * R, nr = min(R, nrows - r0);
                for (int q = t; q < nr * 4; q += blockDim.x) {
                    const int r = q >> 2, part = q & 3;
                    cp_async16(pb + r * 64 + 16 * part,
                               ep.dn_codes + (size_t)ids[r0 + r] * (H / 2) + band * (kBand / 2) + 16 * part);
                }
                for (int q = t; q < nr * T; q += blockDim.x) {
                    const int r = q % nr, k = q / nr;
                    const int n = ids[r0 + r];
                    cp_async4(hb + r * kMaxBatch + k,
                              shared ? io.h_sh + (size_t)k * N + n : io.h_pair + (size_t)(pbase + k) * N + n);
                }
                cp_async_commit();
            };
            if (npass > 0) prefetch(0);
            for (int p = 0; p < npass; ++p) {
                if (p + 1 < npass) {
                    prefetch(p + 1);
                    cp_async_wait<1>();
                } else {
                    cp_async_wait<0>();
                }
                __syncthreads();
                const uint8_t* pb = pass_buf + (p & 1) * S::kPass;
                const float* hb = reinterpret_cast<const float*>(pb + S::kCodes);
                const int nr = min(R, nrows - p * R);
                for (int r = 0; r < nr; ++r) {
                    float wv[4];
                    weights(ids[p * R + r], reinterpret_cast<const uint16_t*>(pb + r * 64)[oq], wv);
#pragma unroll
                    for (int b = 0; b < kMaxBatch / 8; ++b) {
                        const int k = warp + 8 * b;
                        if (k < T) {
                            const float hv = hb[r * kMaxBatch + k];
#pragma unroll
                            for (int a = 0; a < 4; ++a) acc[a][b] = fmaf(hv, wv[a], acc[a][b]);
                        }
                    }
                }
                __syncthreads();
            }
            if (npass == 0) {
                cp_async_wait<0>();
                __syncthreads();
            }
        }
        // ---- partial rows: (token, slot) of this item, outputs of this band
        auto store = [&](int k, const float (&v)[4]) {
            const int tok = shared ? k : __ldcg(io.pair_tok + pbase + k);
            const int slot = shared ? chunk : SC + __ldcg(io.pair_slot + pbase + k) - 1;
            const float wgt = shared ? 1.f : __ldcg(io.pair_w + pbase + k);
            float* dst = io.partial + ((size_t)tok * NSl + slot) * H + band * kBand + 4 * oq;
            *reinterpret_cast<float4*>(dst) = make_float4(wgt * v[0], wgt * v[1], wgt * v[2], wgt * v[3]);
        };
        if (rows_split) {
            // fixed-order sum of the 8 warps' sums: red[warp][k][128] over the (now idle) pass buffers
            float* red = reinterpret_cast<float*>(pass_buf);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k < T)
                    *reinterpret_cast<float4*>(red + ((size_t)warp * 8 + k) * kBand + 4 * oq) =
                        make_float4(acc[0][k], acc[1][k], acc[2][k], acc[3][k]);
            __syncthreads();
            if (warp < T) {
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                for (int w = 0; w < 8; ++w) {
                    const float4 s4 = *reinterpret_cast<const float4*>(red + ((size_t)w * 8 + warp) * kBand + 4 * oq);
                    v[0] += s4.x; v[1] += s4.y; v[2] += s4.z; v[3] += s4.w;
                }
                store(warp, v);
            }
        } else {
#pragma unroll
            for (int b = 0; b < kMaxBatch / 8; ++b) {
                const int k = warp + 8 * b;
                if (k < T) {
                    const float v[4] = {acc[0][b], acc[1][b], acc[2][b], acc[3][b]};
                    store(k, v);
                }
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ fused (B <= 8)
// For a few tokens the whole expert product runs per unit (expert, 64-neuron
// group, up to kFTok of the expert's tokens), as in the batch-1 kernel: the
// group's 64 up rows stream in four chunked bulk copies, the DP4A GEMV runs
// per token, four threads per row add the row's partial sums for every
// token, and the first of them copies the row's down codes once if the row
// fired for ANY token (the union of the tokens' live rows, each read once);
// the group's slab follows if any row fired.  Thread j then owns OPT outputs
// of every token and adds the union rows in ascending order (one fp32 chain
// per (token, output); a row dead for one token adds h * q = +0 for it), and
// writes one partial row per (token, slot, group).  A second kernel adds each
// token's partial rows in a fixed order.
struct FusedTables {
    int fu_off[kMaxRouted + 1];
    int touched[kMaxRouted];
    int e_off[kMaxRouted + 1];
};
struct FusedSmem {
    // misc: h[kFTok][64] f32, off[64] f32, bars[8] u64, ticket, live bits u64, tables
    static constexpr int kHs = 0, kOffs = kFTok * 64 * 4, kBarsOff = kOffs + 256, kTicket = kBarsOff + 64,
                         kLive = kTicket + 8, kTables = kLive + 8;
    __host__ __device__ static int codes(int H) { return 64 * (H / 2); }
    __host__ __device__ static int sb(int H) { return H * 4; }  // up scales of 64 rows, then the down slab
    __host__ __device__ static int misc(int H) { return codes(H) + sb(H); }
    static constexpr int kTablesBytes = 1664;  // the ticketed kernel's FusedTables or the small kernel's tables
    __host__ __device__ static int total(int H) { return misc(H) + kTables + kTablesBytes; }
};
static_assert(sizeof(FusedTables) <= FusedSmem::kTablesBytes, "fused tables exceed their region");

// Partial row of (token b, row ri) in the fused layout [B][H/32][Ut][32].
struct FusedOut {
    float* base;
    int Ut, H;
    __device__ __forceinline__ float4* quad(int b, int ri, int o4) const {
        return reinterpret_cast<float4*>(base + (size_t)b * H * Ut + ((size_t)(o4 >> 3) * Ut + ri) * 32) + (o4 & 7);
    }
};

// NT: token slots compiled in (the unit's T <= NT), so that a unit of one or
// two tokens issues no multiply for the slots it does not have.
template <int OPT, int NT>
__device__ __forceinline__ void fused_down(const uint8_t* codes, const uint32_t* sb, const float* h_s, uint64_t live,
                                           const float (&Hsum)[kFTok], const float (&wgt)[kFTok],
                                           const int (&tok)[kFTok], const int (&ri)[kFTok], int T, int rowb, int j,
                                           const FusedOut& out) {
    float acc[NT][OPT];
#pragma unroll
    for (int k = 0; k < NT; ++k)
#pragma unroll
        for (int e = 0; e < OPT; ++e) acc[k][e] = 0.f;
    while (live) {
        const int n = __ffsll((long long)live) - 1;
        live &= live - 1;
        const uint8_t* row = codes + (size_t)n * rowb;
        uint32_t w[2];
        if (OPT == 16) {
            const uint2 cw = *reinterpret_cast<const uint2*>(row + 8 * j);
            w[0] = cw.x;
            w[1] = cw.y;
        } else if (j & 1) {
            const uint32_t lo = *reinterpret_cast<const uint16_t*>(row + 6 * j);
            const uint32_t hi = *reinterpret_cast<const uint32_t*>(row + 6 * j + 2);
            w[0] = lo | (hi << 16);
            w[1] = hi >> 16;
        } else {
            w[0] = *reinterpret_cast<const uint32_t*>(row + 6 * j);
            w[1] = *reinterpret_cast<const uint16_t*>(row + 6 * j + 4);
        }
        float hs[NT][5];
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            const float hn = k < T ? h_s[k * 64 + n] : 0.f;
            hs[k][0] = hn; hs[k][1] = hn * 0.0625f; hs[k][2] = hn * 0.00390625f;
            hs[k][3] = hn * 0.000244140625f; hs[k][4] = hn * 1.52587890625e-05f;
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
#pragma unroll
                for (int k = 0; k < NT; ++k)
                    if (k < T) acc[k][8 * jj + i] = fmaf(hs[k][pos], q, acc[k][8 * jj + i]);
            }
        }
    }
    const uint4* sbq = reinterpret_cast<const uint4*>(sb) + (OPT / 4) * j;
#pragma unroll
    for (int i = 0; i < OPT / 4; ++i) {
        const uint4 v = sbq[i];
        const uint32_t sbw[4] = {v.x, v.y, v.z, v.w};
        float2 sbf[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sbf[e] = half2_to_float2(sbw[e]);
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            if (k < T) {
                float r[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) r[e] = wgt[k] * fmaf(sbf[e].x, acc[k][4 * i + e], sbf[e].y * Hsum[k]);
                *out.quad(tok[k], ri[k], (OPT / 4) * j + i) = make_float4(r[0], r[1], r[2], r[3]);
            }
        }
    }
}

// Shared-memory buffers of a fused-unit CTA.
struct FusedBufs {
    uint8_t* codes;    // 64 up rows, then the parts, then the live rows' down codes
    uint32_t* sbs;     // the up scales of 64 rows, then the down slab
    float* h_s;        // [kFTok][64]
    float* offs_s;     // [64]
    uint64_t* bars;    // 4 up chunks, down
    uint8_t* live8;    // live bits of rows 8w .. 8w+7 per warp w
    uint8_t* tables;   // the kernel's own tables
};
__device__ __forceinline__ FusedBufs fused_bufs(uint8_t* smem, int H) {
    using S = FusedSmem;
    uint8_t* misc = smem + S::misc(H);
    return FusedBufs{smem, reinterpret_cast<uint32_t*>(smem + S::codes(H)), reinterpret_cast<float*>(misc + S::kHs),
                     reinterpret_cast<float*>(misc + S::kOffs), reinterpret_cast<uint64_t*>(misc + S::kBarsOff),
                     misc + S::kLive, misc + S::kTables};
}

// Per-token facts of a unit: the token, its partial row and its router weight.
struct UnitTokens {
    int tok[kFTok], ri[kFTok];
    float w[kFTok];
};

__device__ __forceinline__ int pick(const int (&a)[kFTok], int i) {
    int v = a[0];
#pragma unroll
    for (int k = 1; k < kFTok; ++k) v = i == k ? a[k] : v;
    return v;
}

// Thread 0: the bulk copies of chunks c0 .. c1-1 of group g's 64 up rows
// (16 rows each, chunk k on bars[k]; the group's up scales ride on chunk 0).
__device__ __forceinline__ void fused_issue_up(const FusedBufs& sm, const ExpertPtrs& ep, int g, int H, uint64_t pol,
                                               int c0 = 0, int c1 = 4) {
    const int rowb = H / 2, G = H / 64;
    const uint8_t* src = ep.up_codes + (size_t)g * 64 * rowb;
    const uint32_t chunk = 16 * rowb;
    if (c0 == 0) {
        mbar_arrive_expect_tx(&sm.bars[0], chunk + 64 * G * 4);
        bulk_g2s(sm.sbs, ep.up_sb + (size_t)g * 64 * G, 64 * G * 4, &sm.bars[0], pol);
        bulk_g2s(sm.codes, src, chunk, &sm.bars[0], pol);
        c0 = 1;
    }
    for (int k = c0; k < c1; ++k) {
        mbar_arrive_expect_tx(&sm.bars[k], chunk);
        bulk_g2s(sm.codes + k * chunk, src + (size_t)k * chunk, chunk, &sm.bars[k], pol);
    }
}

// A thread's part of a unit's up GEMV for T <= kFTok tokens: token lane tk
// (the TL lanes of one scale group are adjacent in a warp), group gc, row
// lane rs of RS.
// With pair (3 or 4 tokens) each lane takes two tokens, tk and tk + 2, at the
// same rows: the code masks are shared and every thread has rows to walk.
// Worth it where x comes ready-made (the ticketed kernel: 8.7% at 32 tokens);
// the small-batch kernel, which converts x per thread, keeps one token per lane.
struct FusedRole {
    int tk, tk2, gc, rs, RS;  // tk2: the lane's second token, or -1
    bool active;              // owns (token, group) work
};
__device__ __forceinline__ FusedRole fused_role(int T, int G, bool pair) {
    const int t = threadIdx.x;
    const int TL = T == 1 ? 1 : (T == 2 || pair ? 2 : 4);
    FusedRole r;
    r.RS = 256 / (TL * G);
    r.tk = t % TL;
    r.tk2 = pair && T >= 3 && r.tk + 2 < T ? r.tk + 2 : -1;
    r.gc = (t / TL) % G;
    r.rs = t / (TL * G);
    r.active = r.rs < r.RS && r.tk < T;
    return r;
}

// Off the unit's main path, out of line: thread 0 waits (bounded) for the
// phases of barriers bars[0 .. n); the debug output of each token's own live
// set (h > 0) of a unit (warp 0).
__device__ __noinline__ void drain_bars(uint64_t* bars, int n, uint32_t par) {
    for (int i = 0; i < n; ++i) mbar_wait(&bars[i], par);
}
__device__ __noinline__ void write_unit_live_masks(uint64_t* dbg_live, int Ut, const float* h_s, int T,
                                                   const UnitTokens ut) {
    const int t = threadIdx.x;
    for (int k = 0; k < T; ++k) {
        const unsigned m0 = __ballot_sync(0xffffffffu, h_s[k * 64 + t] > 0.f);
        const unsigned m1 = __ballot_sync(0xffffffffu, h_s[k * 64 + t + 32] > 0.f);
        if (t == 0) dbg_live[(size_t)pick(ut.tok, k) * Ut + pick(ut.ri, k)] = (uint64_t)m1 << 32 | m0;
    }
}

// One unit after its up copies were issued (phase `par` of bars[0..3]), with
// each active thread's x fixed-point copies in xf (token tk) and, with kPair,
// xf2 (token tk2): the DP4A GEMV per token, ReLU^2, the union-live rows' down
// codes and the slab, the down products into the tokens' partial rows.
// Returns 0, or, on every thread when a bounded wait gave up (the error word
// is set), where copies may still be landing: kFuUpInFlight (the up rows on
// bars[0..3], phase par), kFuDownInFlight (the down rows on bars[4], the phase
// before dn_par), kFuNoneInFlight.  The caller drains them (fused_drain), off
// this path.  `live` gets the unit's union live rows.
constexpr int kFuUpInFlight = 1, kFuDownInFlight = 2, kFuNoneInFlight = 3;
template <bool kPair>
__device__ __forceinline__ int fused_unit(const LayerParams& P, const BatchIO& io, const FusedBufs& sm,
                                           const ExpertPtrs& ep, int g, int T, const UnitTokens& ut, const XFixed& xf,
                                           const XFixed& xf2, uint32_t par, uint32_t& dn_par, uint64_t& live) {
    const int H = P.hidden, G = H / 64, rowb = H / 2;
    const int t = threadIdx.x, lane = t & 31;
    const bool dense = (io.flags & HS_FORCE_DENSE) != 0;
    const uint64_t pol = policy_evict_first();
    uint8_t* codes = sm.codes;
    const FusedRole role = fused_role(T, G, kPair);
    const int tk = role.tk, tk2 = role.tk2, gc = role.gc, rs = role.rs, RS = role.RS;
    const bool active = role.active;
    float off_r = 0.f;
    if (t < 64 && ep.up_off) off_r = __ldg(ep.up_off + 64 * g + t);
    // ---- dot products (every thread keeps the warp's step count)
    bool ok = true;
    int waited = -1;
    const int n_steps = (64 + 2 * RS - 1) / (2 * RS);
    for (int i = 0; i < n_steps; ++i) {
        const int r = rs + 2 * RS * i, r2 = r + RS;
        const bool act = rs < RS && r < 64;
        const bool two = act && r2 < 64;
        if (act) {
            const int k = (two ? r2 : r) >> 4;
            while (ok && waited < k) { ++waited; ok = mbar_wait(&sm.bars[waited], par); }
        }
        uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0, b0 = a0, b1 = a0;
        uint32_t sw0 = 0, sw1 = 0;
        if (act && ok) {
            load_group_codes(codes + r * rowb, gc, a0, a1);
            sw0 = sm.sbs[r * G + gc];
            if (two) {
                load_group_codes(codes + r2 * rowb, gc, b0, b1);
                sw1 = sm.sbs[r2 * G + gc];
            }
        }
        const int da = group_dot_fixed16(a0, a1, xf);
        const int db = group_dot_fixed16(b0, b1, xf);
        int da2 = 0, db2 = 0;
        if (kPair && tk2 >= 0) {
            da2 = group_dot_fixed16(a0, a1, xf2);
            db2 = group_dot_fixed16(b0, b1, xf2);
        }
        __syncwarp();  // the token lanes of a group have read its codes before parts land there
        if (act && ok && active) {
            const float2 sa = half2_to_float2(sw0);
            *up_part(codes, rowb, r, gc, tk) = fmaf(sa.x * xf.inv, (float)da, sa.y * xf.xsum);
            if (kPair && tk2 >= 0) *up_part(codes, rowb, r, gc, tk2) = fmaf(sa.x * xf2.inv, (float)da2, sa.y * xf2.xsum);
            if (two) {
                const float2 sbv = half2_to_float2(sw1);
                *up_part(codes, rowb, r2, gc, tk) = fmaf(sbv.x * xf.inv, (float)db, sbv.y * xf.xsum);
                if (kPair && tk2 >= 0)
                    *up_part(codes, rowb, r2, gc, tk2) = fmaf(sbv.x * xf2.inv, (float)db2, sbv.y * xf2.xsum);
            }
        }
    }
    while (ok && waited < 3) { ++waited; ok = mbar_wait(&sm.bars[waited], par); }
    if (t < 64) sm.offs_s[t] = off_r;
    fence_proxy_async_smem();  // the parts come before the down copies into the same rows
    if (!__syncthreads_and(ok)) return kFuUpInFlight;
    // ---- row sums for every token; the row's down codes are copied once if it fired for any
    bool lv = false;
    {
        const int r = t >> 2, q = t & 3;
        bool anyh = false;
        for (int k = 0; k < T; ++k) {
            float s0 = 0.f, s1 = 0.f;
            int cc = q;
            for (; cc + 4 < G; cc += 8) {
                s0 += *up_part(codes, rowb, r, cc, k);
                s1 += *up_part(codes, rowb, r, cc + 4, k);
            }
            if (cc < G) s0 += *up_part(codes, rowb, r, cc, k);
            float sum = s0 + s1;
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            const float z = sum + sm.offs_s[r];
            const float h = z > 0.f ? z * z : 0.f;
            if (q == 0) sm.h_s[k * 64 + r] = h;
            anyh |= h > 0.f;
        }
        if (q == 0) {
            lv = dense || anyh;
            if (lv) {
                mbar_expect_tx(&sm.bars[4], (uint32_t)rowb);
                bulk_g2s(codes + (size_t)r * rowb, ep.dn_codes + ((size_t)g * 64 + r) * rowb, rowb, &sm.bars[4], pol);
            }
        }
        const unsigned bl = __ballot_sync(0xffffffffu, lv);
        if (lane == 0) {
            unsigned m8 = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) m8 |= ((bl >> (4 * i)) & 1u) << i;
            sm.live8[t >> 5] = (uint8_t)m8;
        }
    }
    const bool any = __syncthreads_or(lv) != 0;
    if (t == 0 && any) {
        mbar_arrive_expect_tx(&sm.bars[4], (uint32_t)H * 4);
        bulk_g2s(sm.sbs, ep.dn_sb + (size_t)g * H, H * 4, &sm.bars[4], pol);
    }
    live = *reinterpret_cast<const uint64_t*>(sm.live8);
    // ---- per token: fixed-order sum of h
    float hsum[kFTok];
#pragma unroll
    for (int k = 0; k < kFTok; ++k) {
        hsum[k] = 0.f;
        if (k < T) {
            float hs = sm.h_s[k * 64 + lane] + sm.h_s[k * 64 + lane + 32];
#pragma unroll
            for (int off = 16; off; off >>= 1) hs += __shfl_xor_sync(0xffffffffu, hs, off);
            hsum[k] = hs;
        }
    }
    const int Ut = P.shared_neurons / 64 + P.top_k * (P.routed_neurons / 64);  // partial rows per token
    const FusedOut out{io.partial, Ut, H};
    const int nthr = H % 48 == 0 ? H / 12 : H / 16;
    if (t < nthr) {
        if (!any) {
            const int nq = H % 48 == 0 ? 3 : 4;
#pragma unroll
            for (int k = 0; k < kFTok; ++k)
                if (k < T)
                    for (int i = 0; i < nq; ++i)
                        *out.quad(ut.tok[k], ut.ri[k], nq * t + i) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            ok = mbar_wait(&sm.bars[4], dn_par);
            if (ok) {
                if (H % 48 == 0) {
                    if (T == 1) fused_down<12, 1>(codes, sm.sbs, sm.h_s, live, hsum, ut.w, ut.tok, ut.ri, T, rowb, t, out);
                    else if (T == 2) fused_down<12, 2>(codes, sm.sbs, sm.h_s, live, hsum, ut.w, ut.tok, ut.ri, T, rowb, t, out);
                    else fused_down<12, kFTok>(codes, sm.sbs, sm.h_s, live, hsum, ut.w, ut.tok, ut.ri, T, rowb, t, out);
                } else {
                    if (T == 1) fused_down<16, 1>(codes, sm.sbs, sm.h_s, live, hsum, ut.w, ut.tok, ut.ri, T, rowb, t, out);
                    else if (T == 2) fused_down<16, 2>(codes, sm.sbs, sm.h_s, live, hsum, ut.w, ut.tok, ut.ri, T, rowb, t, out);
                    else fused_down<16, kFTok>(codes, sm.sbs, sm.h_s, live, hsum, ut.w, ut.tok, ut.ri, T, rowb, t, out);
                }
            }
        }
    } else if (any) {
        ok = mbar_wait(&sm.bars[4], dn_par);  // every thread sees the phase before the buffers are reused
    }
    if (any) dn_par ^= 1u;
    fence_proxy_async_smem();
    if (!__syncthreads_and(ok)) return any ? kFuDownInFlight : kFuNoneInFlight;
    return 0;
}

// After fused_unit gave up with status st: thread 0 waits (bounded) for the
// copies still in flight, so that none lands after the CTA has left.
__device__ __noinline__ void fused_drain(const FusedBufs& sm, int st, uint32_t par, uint32_t dn_par) {
    if (st == kFuUpInFlight) drain_bars(sm.bars, 4, par);
    else if (st == kFuDownInFlight) drain_bars(&sm.bars[4], 1, dn_par ^ 1u);
}

// kLiveDbg: the instantiation that also writes each token's live masks (the
// debug output); the other carries no debug code.  This persistent loop sits
// at the register limit of two CTAs per SM: any code on its failure path
// (even a bounded wait for the unit's copies in flight) makes the compiler
// spill on the main path (13% slower at 32 tokens), so after a wait gave up
// (about a second, the error word set) its CTAs leave without that wait.
template <bool kLiveDbg>
__global__ void __launch_bounds__(256, 2) batch_fused_kernel(const __grid_constant__ LayerParams P, const BatchIO io) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int H = P.hidden;
    const FusedBufs sm = fused_bufs(smem, H);
    int* ticket_s = reinterpret_cast<int*>(smem + FusedSmem::misc(H) + FusedSmem::kTicket);
    FusedTables* tb = reinterpret_cast<FusedTables*>(sm.tables);
    const int t = threadIdx.x;
    if (t == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(&sm.bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    BatchMeta* m = io.meta;
    const int U = __ldcg(&m->fu_units), nt = __ldcg(&m->n_touched), su = __ldcg(&m->fu_shared);
    for (int i = t; i <= nt; i += blockDim.x) tb->fu_off[i] = __ldcg(&m->fu_off[i]);
    for (int i = t; i < nt; i += blockDim.x) tb->touched[i] = __ldcg(&m->touched[i]);
    for (int i = t; i <= P.n_routed; i += blockDim.x) tb->e_off[i] = __ldcg(&m->e_off[i]);
    if (t == 0) *ticket_s = atomicAdd(&m->fu_next, 1);
    __syncthreads();
    const int NGs = P.shared_neurons / 64, NGr = P.routed_neurons / 64, G = H / 64;
    const uint64_t pol = policy_evict_first();
    uint32_t dn_par = 0;
    for (int it = 0;; ++it) {
        const int u = *ticket_s;
        if (u >= U) break;
        // ---- the unit: expert, group g, tokens pbase .. pbase + T - 1 of the expert's list
        const bool shared = u < su;
        int g, T, pbase, e = -1;
        ExpertPtrs ep;
        if (shared) {
            const int c = u / NGs;
            g = u % NGs;
            pbase = c * kFTok;
            T = min(kFTok, io.batch - pbase);
            ep = P.shared;
        } else {
            const int i = unit_owner(tb->fu_off, nt, u - su);
            const int local = u - su - tb->fu_off[i];
            g = local % NGr;
            e = tb->touched[i];
            pbase = tb->e_off[e] + (local / NGr) * kFTok;
            T = min(kFTok, tb->e_off[e + 1] - pbase);
            ep = routed_ptrs(P, e);
        }
        __syncthreads();  // every thread has read the ticket
        if (t == blockDim.x - 1) *ticket_s = atomicAdd(&m->fu_next, 1);
        if (t == 0) fused_issue_up(sm, ep, g, H, pol);
        UnitTokens ut;
#pragma unroll
        for (int k = 0; k < kFTok; ++k) {
            ut.tok[k] = 0; ut.ri[k] = 0; ut.w[k] = 0.f;
            if (k < T) {
                if (shared) {
                    ut.tok[k] = pbase + k;
                    ut.ri[k] = g;
                    ut.w[k] = 1.f;
                } else {
                    ut.tok[k] = __ldcg(io.pair_tok + pbase + k);
                    ut.ri[k] = NGs + (__ldcg(io.pair_slot + pbase + k) - 1) * NGr + g;
                    ut.w[k] = __ldcg(io.pair_w + pbase + k);
                }
            }
        }
        // x from the route kernel's fixed-point tables (here, unlike the
        // small-batch kernel, staging x ahead of the weights measured slower:
        // it serialises each unit's copies behind an extra wait)
        const FusedRole role = fused_role(T, G, true);
        XFixed xf = {}, xf2 = {};
        if (role.active) {
            const int tok = pick(ut.tok, role.tk);
            load_x_fixed(io.xt + (size_t)tok * G * kXfStride, io.xsc + (size_t)tok * G * 2, role.gc, xf);
            if (role.tk2 >= 0) {
                const int tok2 = pick(ut.tok, role.tk2);
                load_x_fixed(io.xt + (size_t)tok2 * G * kXfStride, io.xsc + (size_t)tok2 * G * 2, role.gc, xf2);
            }
        }
        uint64_t live = 0;
        if (fused_unit<true>(P, io, sm, ep, g, T, ut, xf, xf2, it & 1, dn_par, live)) return;
        // the unit's h stays in shared memory until the next unit's row sums, past a barrier
        if (kLiveDbg && t < 32)  // each token's own live set (h > 0) for this group
            write_unit_live_masks(io.dbg_live, NGs + P.top_k * NGr, sm.h_s, T, ut);
        if (t < 2 && live) {  // the expert's union over all its tokens (for the live-row counts)
            const uint32_t bits = (uint32_t)(live >> (32 * t));
            uint32_t* mw = shared ? io.mask_s + 2 * g + t : io.mask_r + (size_t)e * (P.routed_neurons / 32) + 2 * g + t;
            if (bits) atomicOr(mw, bits);
        }
    }
}

// ------------------------------------------------------------------ small batch (B <= kSmallMaxBatch)
// With at most 8 tokens the units can be numbered before routing.  A unit
// holds at most kFTok of an expert's tokens: CTA u < NSu is the shared
// expert's group u % NGs with token group u / NGs (small_shared_tok(B)
// tokens each); CTA NSu + j * NGr + g is group g of the j-th (routed expert,
// token group) entry of the batch, experts ascending, each expert's tokens in
// order (an expert with c tokens has ceil(c / 4) entries), and exits if the
// batch has fewer entries.  From kSmallPlanMinBatch tokens the entries and
// the packed fixed-point x tables come from batch_small_plan_kernel; with
// fewer, each routed CTA routes the tokens itself (one warp per token) and
// converts its x group from the bf16 x.  The unit's x is bulk-copied into the
// space of the last 16-row weight chunk before its weights are requested (x
// read by every thread from L2 instead waited behind the weight stream), and
// that chunk is fetched once every thread holds its group.  The shared
// expert's CTAs issue their other weight copies before waiting for the
// previous kernel, as in the batch-1 kernel.  Each unit leaves its live mask
// and expert for the live-row counts (the union over an expert's units).
constexpr int kSmallMaxBatch = 8;

// One routed entry of the small-batch path: an expert and a group of up to
// kFTok of its tokens (ascending), with their top-k slots and router weights.
struct SmallEntry {
    int e, T;
    int tok[kFTok], slot[kFTok];
    float w[kFTok];
    int pad[2];
};
static_assert(sizeof(SmallEntry) == 64, "an entry is 16 words");
struct SmallPlan {
    int n_entries;
    int pad[15];
    SmallEntry ent[kSmallMaxBatch * kMaxTopK];
};
// The unit's per-group (scale, sum) words of its tokens' x tables, then its entry, in the tables region.
constexpr int kSmallXscBytes = kFTok * (kMaxHidden / 64) * 8;
static_assert(kSmallXscBytes + (int)sizeof(SmallEntry) <= FusedSmem::kTablesBytes, "small-batch tables exceed their region");

// Tokens per shared-expert unit of the small-batch kernel: kFTok, except 2
// for a batch of 3 (a 3-token unit leaves a quarter of its lanes idle: 34.5
// against 35.5 us per layer; 2-token units measured equal or slower at 4, 5
// and 8 tokens).
__host__ __device__ inline int small_shared_tok(int B) { return B == 3 ? 2 : kFTok; }
__host__ __device__ inline int small_shared_units(int NGs, int B) {
    return NGs * ((B + small_shared_tok(B) - 1) / small_shared_tok(B));
}

// The batch's routing, once: top-k and softmax of every token (warp per
// token), the routed entries (experts ascending, ceil(pairs / kFTok) entries
// each, an expert's tokens ascending in groups of kFTok), and every token's
// fixed-point x table in the packed layout, converted from a copy of the
// batch's x in shared memory (one bulk copy, in flight during the top-k).
// One CTA; dynamic shared memory 2 * B * H bytes.
__global__ void __launch_bounds__(256) batch_small_plan_kernel(const __grid_constant__ LayerParams P, const BatchIO io) {
    extern __shared__ __align__(128) uint16_t x_s[];  // [B][H]
    __shared__ int topi[kSmallMaxBatch][kMaxTopK];
    __shared__ float topw[kSmallMaxBatch][kMaxTopK];
    __shared__ int cnt[kMaxRouted];
    __shared__ int first[kMaxRouted + 1];
    __shared__ __align__(8) uint64_t xbar;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int B = io.batch, K = P.top_k, E = P.n_routed, H = P.hidden, G = H / 64;
    SmallPlan* pl = io.small_plan;
    if (t == 0) {
        mbar_init(&xbar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    if (t == 0) {
        mbar_arrive_expect_tx(&xbar, (uint32_t)(2 * B * H));
        bulk_g2s(x_s, io.x, (uint32_t)(2 * B * H), &xbar, policy_evict_last());
    }
    if (t < kMaxRouted) cnt[t] = 0;
    if (warp < B) {
        const TopkPick pk = warp_topk_softmax(io.logits + (size_t)warp * E, E, K, topi[warp], topw[warp]);
        if (lane < K) {
            if (io.dbg_topk_idx) io.dbg_topk_idx[warp * K + lane] = pk.idx;
            if (io.dbg_topk_w) io.dbg_topk_w[warp * K + lane] = pk.w;
        }
    }
    __syncthreads();
    if (t < B * K) atomicAdd(&cnt[topi[t / K][t % K]], 1);
    __syncthreads();
    if (warp == 0) {
        // first entry of each expert
        int n[kMaxRouted / 32], sum = 0;
#pragma unroll
        for (int i = 0; i < kMaxRouted / 32; ++i) {
            const int e = (kMaxRouted / 32) * lane + i;
            n[i] = e < E ? (cnt[e] + kFTok - 1) / kFTok : 0;
            sum += n[i];
        }
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        int run = incl - sum;
#pragma unroll
        for (int i = 0; i < kMaxRouted / 32; ++i) {
            const int e = (kMaxRouted / 32) * lane + i;
            if (e < E) first[e] = run;
            run += n[i];
        }
        if (lane == 31) pl->n_entries = incl;
    } else if (mbar_wait(&xbar, 0)) {
        for (int b = 0; b < B; ++b)
            convert_x_fixed<true>(x_s + (size_t)b * H, G, io.xt + (size_t)b * G * 128, io.xsc + (size_t)b * G * 2, 32);
    }
    if (warp == 0 && lane == 0) mbar_wait(&xbar, 0);  // the copy has landed before the CTA leaves
    __syncthreads();
    if (t < B * K) {
        // pair (token b, slot s): its rank among its expert's pairs in token order
        const int b = t / K, s = t % K, e = topi[b][s];
        int rank = 0;
        for (int q = 0; q < t; ++q) rank += topi[q / K][q % K] == e;
        SmallEntry* en = &pl->ent[first[e] + rank / kFTok];
        const int k = rank % kFTok;
        en->tok[k] = b;
        en->slot[k] = s;
        en->w[k] = topw[b][s];
        if (k == 0) {
            en->e = e;
            en->T = min(kFTok, cnt[e] - rank);
        }
    }
}

// The small-batch kernel's two ways to route a unit.  From kSmallPlanMinBatch
// tokens a one-CTA kernel routes the batch first (top-k, entries, packed x
// tables) and each routed unit reads its entry; below, every routed CTA
// routes the batch itself and converts its x group from the bf16 x (no
// kernel ahead of it on the dependency chain, which costs more than the
// redundant routing saves for 2 tokens: 29.9 against 28.4 us per layer).
constexpr int kSmallPlanMinBatch = 3;
static_assert(kSmallPlanMinBatch - 1 <= kFTok, "the in-kernel routing takes one entry per distinct expert");

// x_group_load with the group's eight 16-byte chunks read in an order rotated by the group
// index: the threads of a warp read different groups 128 bytes apart, so in the natural order
// every load of the warp falls on the same four banks.  The chunks are then rotated back into
// their natural registers (three select stages), so the values are exactly x_group_load's.
__device__ __forceinline__ void x_group_load_staggered(const uint16_t* x_s, int gc, uint32_t (&w)[4][8]) {
    const uint4* src = reinterpret_cast<const uint4*>(x_s + 64 * gc);
    const int r = gc & 7;
    uint4 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = src[(c + r) & 7];   // slot c holds chunk (c + r) % 8
#pragma unroll
    for (int st = 0; st < 3; ++st) {                       // rotate right by r: chunk k = slot (k - r) % 8
        const bool b = (r >> st) & 1;
        uint4 nv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) nv[i] = b ? v[(i - (1 << st) + 8) & 7] : v[i];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = nv[i];
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        w[q][0] = v[2 * q].x; w[q][1] = v[2 * q].y; w[q][2] = v[2 * q].z; w[q][3] = v[2 * q].w;
        w[q][4] = v[2 * q + 1].x; w[q][5] = v[2 * q + 1].y; w[q][6] = v[2 * q + 1].z; w[q][7] = v[2 * q + 1].w;
    }
}

// Tables of the in-kernel routing (fewer than kSmallPlanMinBatch tokens).
struct SmallRouteTables {
    int topi[kFTok][kMaxTopK];
    float topw[kFTok][kMaxTopK];
    int tok[kFTok], slot[kFTok];
    float w[kFTok];
    int T, e;
};
static_assert(sizeof(SmallRouteTables) <= FusedSmem::kTablesBytes, "small-batch tables exceed their region");

// One unit per CTA: the shared expert's (64-neuron group, group of up to
// small_shared_tok(B) tokens), then room for every (routed entry, group).  Shared units
// start their weight copies before the dependency wait; routed units past
// the batch's entries leave at once.  The unit's x (packed tables, or the
// bf16 x of the batch) is copied ahead of its weights into the space of the
// last weight chunk, which is fetched once every thread holds its x group.
template <bool kPlanned>
__global__ void __launch_bounds__(256, 2) batch_small_kernel(const __grid_constant__ LayerParams P, const BatchIO io) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int H = P.hidden, G = H / 64;
    const FusedBufs sm = fused_bufs(smem, H);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5, u = blockIdx.x;
    const int B = io.batch, K = P.top_k, E = P.n_routed;
    const int NGs = P.shared_neurons / 64, NGr = P.routed_neurons / 64;
    const int NSu = small_shared_units(NGs, B);
    const bool shared = u < NSu;
    uint64_t* xbar = &sm.bars[5];
    uint8_t* x_dst = sm.codes + 3 * 8 * H;  // chunk 3's space: 4 tokens' packed tables (or bf16 x) fit in it
    if (t == 0) {
        for (int i = 0; i < 6; ++i) mbar_init(&sm.bars[i], 1);
        fence_mbar_init();
        if (shared) fused_issue_up(sm, P.shared, u % NGs, H, policy_evict_first(), 0, 3);  // weights only
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    UnitTokens ut;
    ExpertPtrs ep;
    int g, T, key;
    if constexpr (!kPlanned) {
        // the batch's bf16 x, then the routing of every token by every routed CTA
        SmallRouteTables* st = reinterpret_cast<SmallRouteTables*>(sm.tables);
        if (t == 0) {
            mbar_arrive_expect_tx(xbar, (uint32_t)(2 * B * H));
            bulk_g2s(x_dst, io.x, (uint32_t)(2 * B * H), xbar, policy_evict_last());
        }
        const bool dbg_topk = io.dbg_topk_idx || io.dbg_topk_w;
        if (!shared || (u == 0 && dbg_topk)) {
            if (warp < B) warp_topk_softmax(io.logits + (size_t)warp * E, E, K, st->topi[warp], st->topw[warp]);
            __syncthreads();
            if (u == 0 && dbg_topk && t < B * K) {
                if (io.dbg_topk_idx) io.dbg_topk_idx[t] = st->topi[t / K][t % K];
                if (io.dbg_topk_w) io.dbg_topk_w[t] = st->topw[t / K][t % K];
            }
        }
        if (shared) {
            g = u % NGs;
            T = B;
            ep = P.shared;
            key = E;
#pragma unroll
            for (int k = 0; k < kFTok; ++k) { ut.tok[k] = k < T ? k : 0; ut.ri[k] = g; ut.w[k] = 1.f; }
        } else {
            const int j = (u - NSu) / NGr;
            g = (u - NSu) % NGr;
            if (warp == 0) {
                // one entry per distinct expert: the j-th member of the batch's expert set, its tokens ascending
                const int ei = lane < B * K ? st->topi[lane / K][lane % K] : -1;
                int e = -1, before = 0;
#pragma unroll
                for (int w = 0; w < kMaxRouted / 32; ++w) {
                    uint32_t m = warp_or_b32((ei >= 0 && (ei >> 5) == w) ? 1u << (ei & 31) : 0u);
                    const int c = __popc(m);
                    if (e < 0 && j < before + c) {
                        for (int i = 0; i < j - before; ++i) m &= m - 1;
                        e = 32 * w + __ffs(m) - 1;
                    }
                    before += c;
                }
                int slot = -1;
                if (e >= 0 && lane < B)
                    for (int s2 = 0; s2 < K; ++s2)
                        if (st->topi[lane][s2] == e) slot = s2;
                const unsigned has = __ballot_sync(0xffffffffu, slot >= 0);
                const int k = __popc(has & ((1u << lane) - 1u));
                if (slot >= 0) {
                    st->tok[k] = lane;
                    st->slot[k] = slot;
                    st->w[k] = st->topw[lane][slot];
                }
                if (lane == 0) {
                    st->e = e;
                    st->T = e >= 0 ? __popc(has) : 0;
                }
            }
            __syncthreads();
            T = st->T;
            if (T == 0) {
                if (t == 0) {
                    io.unit_live[u] = 0;
                    io.unit_key[u] = -1;
                    mbar_wait(xbar, 0);  // no copy may be in flight into an exiting CTA
                }
                return;
            }
            key = st->e;
            ep = routed_ptrs(P, key);
#pragma unroll
            for (int k = 0; k < kFTok; ++k) {
                ut.tok[k] = k < T ? st->tok[k] : 0;
                ut.ri[k] = k < T ? NGs + st->slot[k] * NGr + g : 0;
                ut.w[k] = k < T ? st->w[k] : 0.f;
            }
            if (t == 0) fused_issue_up(sm, ep, g, H, policy_evict_first(), 0, 3);
        }
    } else {
        float* xsc_s = reinterpret_cast<float*>(sm.tables);                   // [T][G][2]
        int* ent_s = reinterpret_cast<int*>(sm.tables + kSmallXscBytes);      // the unit's entry, then n_entries
        if (shared) {
            const int c = u / NGs, st = small_shared_tok(B);
            g = u % NGs;
            T = min(st, B - st * c);
            ep = P.shared;
            key = E;
#pragma unroll
            for (int k = 0; k < kFTok; ++k) { ut.tok[k] = st * c + (k < T ? k : 0); ut.ri[k] = g; ut.w[k] = 1.f; }
        } else {
            const int j = (u - NSu) / NGr;  // < B * K: the plan holds room for every pair
            g = (u - NSu) % NGr;
            const SmallPlan* pl = io.small_plan;
            if (t < 16) ent_s[t] = __ldcg(reinterpret_cast<const int*>(&pl->ent[j]) + t);
            if (t == 16) ent_s[16] = __ldcg(&pl->n_entries);
            __syncthreads();
            const SmallEntry* en = reinterpret_cast<const SmallEntry*>(ent_s);
            T = j < ent_s[16] ? en->T : 0;
            if (T == 0) {  // no copy was issued
                if (t == 0) {
                    io.unit_live[u] = 0;
                    io.unit_key[u] = -1;
                }
                return;
            }
            key = en->e;
            ep = routed_ptrs(P, key);
#pragma unroll
            for (int k = 0; k < kFTok; ++k) {
                ut.tok[k] = k < T ? en->tok[k] : 0;
                ut.ri[k] = k < T ? NGs + en->slot[k] * NGr + g : 0;
                ut.w[k] = k < T ? en->w[k] : 0.f;
            }
        }
        if (t == 0) {
            // the unit's x tables first (they gate the dot products), then its weights
            mbar_arrive_expect_tx(xbar, (uint32_t)(T * G * (128 + 8)));
            for (int k = 0; k < T; ++k) {
                const int b = ut.tok[k];
                bulk_g2s(x_dst + (size_t)k * G * 128, io.xt + (size_t)b * G * 128, (uint32_t)G * 128, xbar,
                         policy_evict_last());
                bulk_g2s(xsc_s + (size_t)k * G * 2, io.xsc + (size_t)b * G * 2, (uint32_t)G * 8, xbar,
                         policy_evict_last());
            }
            if (!shared) fused_issue_up(sm, ep, g, H, policy_evict_first(), 0, 3);
        }
    }
    const FusedRole role = fused_role(T, G, false);
    const bool xok = mbar_wait(xbar, 0);
    XFixed xf = {};
    if (role.active && xok) {
        if constexpr (kPlanned) {
            const float* xsc_s = reinterpret_cast<const float*>(sm.tables);
            load_x_fixed_packed(x_dst + (size_t)role.tk * G * 128, xsc_s + (size_t)role.tk * G * 2, role.gc, xf);
        } else {
            uint32_t xw[4][8];
            x_group_load_staggered(reinterpret_cast<const uint16_t*>(x_dst) + (size_t)pick(ut.tok, role.tk) * H,
                                   role.gc, xw);
            x_group_fixed(xw, xf);
        }
    }
    fence_proxy_async_smem();  // the reads of x come before the copy that overwrites them
    if (!__syncthreads_and(xok)) {
        // a wait gave up (the error word is set): the chunks already requested land before the CTA leaves
        if (t == 0)
            for (int i = 0; i < 3; ++i) mbar_wait(&sm.bars[i], 0);
        return;
    }
    if (t == 0) fused_issue_up(sm, ep, g, H, policy_evict_first(), 3, 4);
    uint32_t dn_par = 0;
    uint64_t live = 0;
    const int fst = fused_unit<false>(P, io, sm, ep, g, T, ut, xf, xf, 0, dn_par, live);
    if (fst) {
        if (t == 0) fused_drain(sm, fst, 0, dn_par);
        return;
    }
    if (io.dbg_live && t < 32)  // each token's own live set (h > 0) for this group
        write_unit_live_masks(io.dbg_live, P.shared_neurons / 64 + P.top_k * (P.routed_neurons / 64), sm.h_s, T, ut);
    if (t == 0) {
        io.unit_live[u] = live;
        io.unit_key[u] = key;
    }
}

// y[b][o] = the token's partial rows added in a fixed order (32 outputs per
// CTA, token b = blockIdx.y): one bulk copy of the [Ut][32] slice, thread
// (lane, p) adds rows p, p+8, ..., then the 8 sums in order; bf16 RNE.
__global__ void __launch_bounds__(256) batch_fused_reduce_kernel(const __grid_constant__ LayerParams P, const BatchIO io) {
    extern __shared__ __align__(128) float slice[];  // [Ut][32]
    __shared__ float part[8][33];
    __shared__ __align__(8) uint64_t bar;
    const int t = threadIdx.x, cb = blockIdx.x, b = blockIdx.y, H = P.hidden;
    const int Ut = P.shared_neurons / 64 + P.top_k * (P.routed_neurons / 64);
    if (t == 0) { mbar_init(&bar, 1); fence_mbar_init(); }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    if (t == 0) {
        mbar_arrive_expect_tx(&bar, (uint32_t)Ut * 128u);
        const float* src = io.partial + (size_t)b * H * Ut + (size_t)cb * Ut * 32;
        for (int r0 = 0; r0 < Ut; r0 += 256) {
            const int rows = min(256, Ut - r0);
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
    for (; r + 8 < Ut; r += 16) {
        a0 += slice[r * 32 + lane];
        a1 += slice[(r + 8) * 32 + lane];
    }
    if (r < Ut) a0 += slice[r * 32 + lane];
    part[p][lane] = a0 + a1;
    __syncthreads();
    if (t < 32) {
        float y = part[0][t];
#pragma unroll
        for (int i = 1; i < 8; ++i) y += part[i][t];
        const size_t o = (size_t)b * H + cb * 32 + t;
        if (io.y_f32) io.y_f32[o] = y;
        io.y_bf16[o] = f32_to_bf16_bits(y);
    }
    if ((io.live_total || io.live_groups) && cb == 0 && b == 0) {
        __syncthreads();  // part[] is reused below
        int n = 0, ng = 0;
        if (io.unit_live) {
            // small-batch path: thread q walks group q's units in order (an
            // expert's units are adjacent) and ORs the masks of each expert
            const int NGs = P.shared_neurons / 64, NGr = P.routed_neurons / 64;
            const int NSu = small_shared_units(NGs, io.batch);
            for (int q = t; q < NGs + NGr; q += blockDim.x) {
                const bool sh = q < NGs;
                const int first = sh ? q : NSu + (q - NGs), step = sh ? NGs : NGr;
                const int last = sh ? NSu : io.n_units;
                int key = -2;
                unsigned long long acc = 0;
                for (int v = first; v < last; v += step) {
                    const int kv = __ldcg(io.unit_key + v);
                    if (kv != key) {
                        n += __popcll(acc);
                        ng += acc != 0ull;
                        acc = 0;
                        key = kv;
                    }
                    if (kv >= 0) acc |= __ldcg(reinterpret_cast<const unsigned long long*>(io.unit_live) + v);
                }
                n += __popcll(acc);
                ng += acc != 0ull;
            }
        } else {
            // union live rows and groups per expert, from the union masks
            const BatchMeta* m = io.meta;
            const int nt = __ldcg(&m->n_touched), WR = P.routed_neurons / 32, WS = P.shared_neurons / 32;
            for (int q = t; q < nt * (WR / 2) + WS / 2; q += blockDim.x) {
                const uint32_t* mw = q < nt * (WR / 2)
                                         ? io.mask_r + (size_t)__ldcg(&m->touched[q / (WR / 2)]) * WR + 2 * (q % (WR / 2))
                                         : io.mask_s + 2 * (q - nt * (WR / 2));
                const uint32_t a = __ldcg(mw), c = __ldcg(mw + 1);
                n += __popc(a) + __popc(c);
                ng += (a | c) != 0u;
            }
        }
        n = (int)warp_add_u32((unsigned)n);
        ng = (int)warp_add_u32((unsigned)ng);
        if (lane == 0) { part[p][0] = __int_as_float(n); part[p][1] = __int_as_float(ng); }
        __syncthreads();
        if (t == 0) {
            int tn = 0, tg = 0;
            for (int i = 0; i < 8; ++i) { tn += __float_as_int(part[i][0]); tg += __float_as_int(part[i][1]); }
            if (io.live_total) *io.live_total = tn;
            if (io.live_groups) *io.live_groups = tg;
        }
    }
}

// ------------------------------------------------------------------ reduce
// y[t][o] = sum over the token's partial rows in slot order (shared-expert
// chunks first, then the routed slots 1..K); bf16 RNE.
__global__ void __launch_bounds__(256) batch_reduce_kernel(const __grid_constant__ LayerParams P, const BatchIO io) {
    pdl_wait();
    pdl_trigger();
    const int H = P.hidden, B = io.batch;
    const int NSl = (P.shared_neurons ? shared_chunks(B) : 0) + P.top_k;
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;  // float4 index over [B][H/4]
    if (idx < B * (H / 4)) {
        const int tok = idx / (H / 4), c4 = idx % (H / 4);
        const float4* p = reinterpret_cast<const float4*>(io.partial + (size_t)tok * NSl * H) + c4;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < NSl; ++s) {
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
    size_t meta, topk_idx, topk_w, pair_tok, pair_w, pair_slot, xt, xsc, h_pair, h_sh, mask_r, mask_s, small_plan,
        unit_live, unit_key, partial, total;
};

// Grid of the small-batch kernel: the shared expert's units, then room for
// B * K (routed expert, token group) entries.
int small_units(const hs_moe_layer* L, int B) {
    return hs::small_shared_units(L->shared ? L->shared->neurons / 64 : 0, B) +
           B * L->top_k * (L->routed[0].neurons / 64);
}

BatchLayout batch_layout(const hs_moe_layer* L, int B) {
    const int K = L->top_k, E = L->n_routed, NR = L->routed[0].neurons;
    const int NS = L->shared ? L->shared->neurons : 0, H = L->hidden, G = H / 64;
    const int SC = NS ? hs::shared_chunks(B) : 0;
    BatchLayout l{};
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o += round_up(bytes, 256); return at; };
    l.meta = take(sizeof(hs::BatchMeta));
    l.topk_idx = take((size_t)B * K * 4);
    l.topk_w = take((size_t)B * K * 4);
    l.pair_tok = take((size_t)B * K * 4);
    l.pair_w = take((size_t)B * K * 4);
    l.pair_slot = take((size_t)B * K * 4);
    l.xt = take((size_t)B * G * hs::kXfStride);
    l.xsc = take((size_t)B * G * 8);
    l.h_pair = take((size_t)B * K * NR * 4);
    l.h_sh = take((size_t)B * (NS ? NS : 1) * 4);
    l.mask_r = take((size_t)E * (NR / 32) * 4);
    l.mask_s = take((size_t)(NS ? NS / 32 : 1) * 4);
    const int Ut = (NS / 64) + K * (NR / 64);
    l.small_plan = take(sizeof(hs::SmallPlan));
    l.unit_live = take((size_t)small_units(L, B) * 8);
    l.unit_key = take((size_t)small_units(L, B) * 4);
    // the fused path's partial rows (per token, slot and group) or the banded path's (per token and slot)
    l.partial = take((size_t)B * std::max(Ut, SC + K) * H * 4);
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
    io.xt = reinterpret_cast<uint8_t*>(w + l.xt);
    io.xsc = reinterpret_cast<float*>(w + l.xsc);
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
    io.dbg_live = dbg ? dbg->live_mask : nullptr;
    if (io.dbg_live && ((uintptr_t)io.dbg_live & 7u)) return HS_ERR_MISALIGNED;

    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return HS_ERR_CUDA;
    const int up_smem = hs::BatchUpSmem::total(L->hidden);
    const int dn_smem = hs::BatchDownSmem::total();
    if (batch <= hs::kSmallMaxBatch && !(flags & HS_BATCH_EXPERT_UNION)) {
        // units are numbered before routing; from kSmallPlanMinBatch tokens one CTA routes the batch first
        const int f_smem = hs::FusedSmem::total(L->hidden);
        const int Ut = (L->shared ? L->shared->neurons / 64 : 0) + L->top_k * (L->routed[0].neurons / 64);
        io.unit_live = reinterpret_cast<uint64_t*>(w + l.unit_live);
        io.unit_key = reinterpret_cast<int*>(w + l.unit_key);
        io.n_units = small_units(L, batch);
        io.small_plan = reinterpret_cast<hs::SmallPlan*>(w + l.small_plan);
        const bool planned = batch >= hs::kSmallPlanMinBatch;
        const void* small = planned ? (const void*)hs::batch_small_kernel<true> : (const void*)hs::batch_small_kernel<false>;
        if (set_smem_attr(small, f_smem) != HS_OK) return HS_ERR_CUDA;
        if (set_smem_attr((const void*)hs::batch_fused_reduce_kernel, Ut * 128) != HS_OK) return HS_ERR_CUDA;
        const int plan_smem = 2 * batch * L->hidden;
        if (planned && (set_smem_attr((const void*)hs::batch_small_plan_kernel, plan_smem) != HS_OK ||
                        launch_pdl(hs::batch_small_plan_kernel, dim3(1), dim3(256), plan_smem, s, P, io) != cudaSuccess))
            return HS_ERR_CUDA;
        if ((planned ? launch_pdl(hs::batch_small_kernel<true>, dim3(io.n_units), dim3(256), f_smem, s, P, io)
                     : launch_pdl(hs::batch_small_kernel<false>, dim3(io.n_units), dim3(256), f_smem, s, P, io)) !=
            cudaSuccess)
            return HS_ERR_CUDA;
        if (launch_pdl(hs::batch_fused_reduce_kernel, dim3(L->hidden / 32, batch), dim3(256), (size_t)Ut * 128, s, P,
                       io) != cudaSuccess)
            return HS_ERR_CUDA;
        return launch_err();
    }
    if (cudaMemsetAsync(io.meta, 0, sizeof(hs::BatchMeta), s) != cudaSuccess) return HS_ERR_CUDA;
    // the first kernel follows the memset with ordinary stream ordering
    hs::batch_route_kernel<<<dim3(batch), dim3(256), 0, s>>>(P, io);
    if (cudaGetLastError() != cudaSuccess) return HS_ERR_CUDA;
    if (batch <= hs::kFusedMaxBatch && !(flags & HS_BATCH_EXPERT_UNION)) {
        const int f_smem = hs::FusedSmem::total(L->hidden);
        const int Ut = (L->shared ? L->shared->neurons / 64 : 0) + L->top_k * (L->routed[0].neurons / 64);
        if (set_smem_attr((const void*)hs::batch_fused_kernel<false>, f_smem) != HS_OK ||
            set_smem_attr((const void*)hs::batch_fused_kernel<true>, f_smem) != HS_OK)
            return HS_ERR_CUDA;
        if (set_smem_attr((const void*)hs::batch_fused_reduce_kernel, Ut * 128) != HS_OK) return HS_ERR_CUDA;
        if ((io.dbg_live ? launch_pdl(hs::batch_fused_kernel<true>, dim3(2 * sms), dim3(256), f_smem, s, P, io)
                         : launch_pdl(hs::batch_fused_kernel<false>, dim3(2 * sms), dim3(256), f_smem, s, P, io)) !=
            cudaSuccess)
            return HS_ERR_CUDA;
        if (launch_pdl(hs::batch_fused_reduce_kernel, dim3(L->hidden / 32, batch), dim3(256), (size_t)Ut * 128, s, P,
                       io) != cudaSuccess)
            return HS_ERR_CUDA;
        return launch_err();
    }
    if (set_smem_attr((const void*)hs::batch_up_kernel, up_smem) != HS_OK) return HS_ERR_CUDA;
    if (set_smem_attr((const void*)hs::batch_down_kernel, dn_smem) != HS_OK) return HS_ERR_CUDA;
    if (io.dbg_live) {  // debug only: the up kernel ORs each token's bits into zeroed words
        const int Ut = (L->shared ? L->shared->neurons / 64 : 0) + L->top_k * (L->routed[0].neurons / 64);
        if (cudaMemsetAsync(io.dbg_live, 0, (size_t)batch * Ut * sizeof(uint64_t), s) != cudaSuccess) return HS_ERR_CUDA;
    }
    if (launch_pdl(hs::batch_up_kernel, dim3(hs::kUpCtasPerSm * sms), dim3(hs::kUpThreads), up_smem, s, P, io) != cudaSuccess)
        return HS_ERR_CUDA;
    if (launch_pdl(hs::batch_down_kernel, dim3(2 * sms), dim3(256), dn_smem, s, P, io) != cudaSuccess)
        return HS_ERR_CUDA;
    const int nred = (batch * (L->hidden / 4) + 255) / 256;
    if (launch_pdl(hs::batch_reduce_kernel, dim3(nred), dim3(256), 0, s, P, io) != cudaSuccess) return HS_ERR_CUDA;
    return launch_err();
}
