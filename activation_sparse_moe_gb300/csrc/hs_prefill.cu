// Prefill of a ReLU^2 MoE layer with neuron-major 4-bit down weights, on the
// Blackwell tensor cores (tcgen05, accumulators in TMEM, operands staged by TMA).
//
// "Skipping dead neurons..." (sevren.ai), sections "The weights now face the
// wrong way.", "Sorted by expert", "Per token sparse, per prompt dense" and
// "What we do instead": a prompt's tokens are routed (top-6 of 128 plus the
// shared expert), grouped by expert, and each expert's tokens go through the
// up projection, ReLU^2 and the down projection as matrix products; the down
// product reads the neuron-major copy directly and skips neuron tiles that
// are dead for every token of a tile.
//
// GB300 design (ours):
//  * Tokens are gathered into expert order as fp16 (x is bf16; fp16 keeps the
//    products of 4-bit weights exact enough), with the K index permuted inside
//    each 64-block to the order in which the dequantiser emits nibble pairs
//    (the same permutation on both operands leaves the product unchanged).
//  * Up GEMM per (token tile <= 256, 128 neurons): D[neurons][tokens] in TMEM,
//    A = weights dequantised W4 -> fp16 by all threads into 128-byte-swizzled
//    K-major tiles, B = gathered tokens by TMA.  Epilogue: + offset, ReLU^2,
//    H (fp16, [token][neuron]) and a live flag per (token tile, 64 neurons).
//  * Down GEMM per (token tile, 128 outputs): D[outputs][tokens], A = the
//    neuron-major codes of one 64-neuron tile dequantised and transposed into
//    a K-major tile (the tile is one scale group), B = H by TMA; tiles whose
//    live flag is clear are skipped (no weight fetch, no product).
//  * One fp32 partial row per (token, slot), combined per token in slot order.
#include <cuda.h>

#include <type_traits>

#include "hs_host.h"
#include "hs_tc.cuh"
#include "hs_transpose.cuh"
#include "hs_rowgather.cuh"

namespace hs {

constexpr int kNt = 128;          // max tokens per tile (MMA N)
constexpr int kMaxTokens = 4096;
constexpr int kTokBlk = 8;       // tokens per CTA of the list/gather kernel
constexpr int kSuperBlk = 16;    // token blocks per superblock (pair counts are kept per superblock too)
constexpr int kMaxKTiles = 64;    // 64-neuron tiles per expert (neurons <= 4096): one 64-bit mask

struct PrefillMeta {
    int n_tiles;                  // token tiles (routed experts first, then shared)
    int up_units, dn_units;
    int skipped, total;           // down k-tiles skipped / considered
    unsigned long long union_rt;  // sum over tiles of tokens x union-live neurons
    unsigned long long exec_rt;   // sum over tiles of tokens x neurons the down product multiplies
    unsigned long long dense_rt;  // sum over tiles of tokens x all neurons
    int cnt[kMaxRouted];
    int off[kMaxRouted + 1];
    int tile_off[kMaxRouted + 2]; // first tile of each expert (index E = shared)
};

// Token tile: rows [row0, row0 + ntok) of the gathered arrays; expert e (E = shared).
struct TileInfo {
    int e, row0, ntok, pad;
};

struct PrefillIO {
    const uint16_t* x;        // [T][H] bf16
    const float* logits;      // [T][E]
    int T;
    unsigned flags;
    PrefillMeta* meta;
    int* blk_cnt;             // [ceil(T / kTokBlk)][E] pairs per (token block, expert), zeroed with meta
    int* sb_cnt;              // [ceil(T / (kTokBlk * kSuperBlk))][E] the same per superblock, zeroed with meta
    TileInfo* tiles;          // [max tiles]
    int* idx;                 // [T][K]
    float* w;                 // [T][K]
    int* pair_tok;            // [T*K] grouped by expert (routed)
    int* pos_of;              // [T*K] grouped position of (token, slot)
    float* pair_w;            // [T*K] router weight of each grouped pair
    uint16_t* xg;             // [T*K + T][H] fp16, K permuted per 64-block
    uint16_t* h_r;            // [T*K][NR] fp16
    uint16_t* h_s;            // [T][NS] fp16
    uint32_t* flag_r;         // [T*K/?] per (tile, k-tile): bit set = live
    float* partial;           // [T*K + T][H] fp32 (routed pairs, then shared tokens)
    uint16_t* y_bf16;
    float* y_f32;
    int* dbg_idx;
    float* dbg_w;
    int* dbg_tiles;           // [2] skipped, total
    long long* dbg_work;      // [3] union_rt, exec_rt, dense_rt
    uint64_t* dbg_live;       // [T][Ut] live mask (fp16 h > 0) per (token, slot group), or null
    uint64_t* dbg_tile_live;  // [tiles] 64-neuron tiles the down product multiplies, or null
    int max_tiles;
    // row gather (HS_PREFILL_ROW_GATHER)
    uint32_t* umask;          // [max tiles][kUWords]: bit i of word w = neuron 32w + i live for a token of the tile
    int* nks;                 // [max tiles] k-steps of the tile's plan
    uint32_t* ksd;            // [max tiles][kMaxKTiles] k-step descriptors (gA, gB, split8)
    uint16_t* glist;          // [max tiles][64 * kMaxKTiles] entries: neuron, or rowgather::kPad
    uint16_t* hc_r;           // [T*K][NR] fp16: h of each tile's entries, in k-step order
    uint16_t* hc_s;           // [T][NS] fp16
};
constexpr int kUWords = 2 * kMaxKTiles;

// Inside each 64-block the gathered x holds, for every group of 8 elements
// e0..e7 (one 32-bit word of codes), the order e0 e4 e1 e5 e2 e6 e3 e7: the
// order in which the dequantiser emits nibble pairs.  Both operands of the up
// product use it, so the product is unchanged.

// ------------------------------------------------------------ routing
// One warp per token: top-k + softmax, and the per-expert pair counts
// (integer atomics: the counts, hence everything after, do not depend on the
// order of the additions).  The meta block is zeroed before this kernel runs.
__global__ void __launch_bounds__(256) prefill_route_kernel(const __grid_constant__ LayerParams P, const PrefillIO io) {
    pdl_wait();
    pdl_trigger();
    const int tok = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (tok < io.T) {
        const int K = P.top_k;
        const TopkPick pk = warp_topk_softmax(io.logits + (size_t)tok * P.n_routed, P.n_routed, K,
                                              io.idx + (size_t)tok * K, io.w + (size_t)tok * K);
        if (lane < K) {   // lane j holds choice j
            const int e = pk.idx;
            atomicAdd(&io.meta->cnt[e], 1);
            atomicAdd(&io.blk_cnt[(tok / kTokBlk) * P.n_routed + e], 1);
            atomicAdd(&io.sb_cnt[(tok / (kTokBlk * kSuperBlk)) * P.n_routed + e], 1);
            if (io.dbg_idx) io.dbg_idx[(size_t)tok * K + lane] = e;
            if (io.dbg_w) io.dbg_w[(size_t)tok * K + lane] = pk.w;
        }
    }
}

// Inclusive sum over the 256 threads of a CTA (8 warps); `tmp` holds 8 ints.
__device__ __forceinline__ int block_inclusive_sum(int v, int* tmp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) tmp[warp] = v;
    __syncthreads();
    int before = 0;
    for (int i = 0; i < warp; ++i) before += tmp[i];
    __syncthreads();
    return v + before;
}

// One CTA: pair offsets, token tiles (an expert's pairs cut into tiles of up
// to kNt), work-unit counts, cleared live flags.
__global__ void __launch_bounds__(256) prefill_tiles_kernel(const __grid_constant__ LayerParams P, const PrefillIO io) {
    __shared__ int tmp[8];
    pdl_wait();
    pdl_trigger();
    PrefillMeta* m = io.meta;
    const int E = P.n_routed, e = threadIdx.x;
    const int c = e < E ? __ldcg(&m->cnt[e]) : 0;
    const int nt_e = (c + kNt - 1) / kNt;
    const int c_incl = block_inclusive_sum(c, tmp);
    const int t_incl = block_inclusive_sum(nt_e, tmp);
    const int off = c_incl - c, toff = t_incl - nt_e;
    if (e < E) {
        m->off[e] = off;
        m->tile_off[e] = toff;
        for (int i = 0; i < nt_e; ++i) io.tiles[toff + i] = TileInfo{e, off + kNt * i, min(kNt, c - kNt * i), 0};
    }
    __shared__ int tot_s[2];
    if (e == E - 1) { tot_s[0] = c_incl; tot_s[1] = t_incl; }
    __syncthreads();
    const int npairs = tot_s[0], nrt = tot_s[1];
    const int nst = P.shared_neurons ? (io.T + kNt - 1) / kNt : 0;
    for (int i = threadIdx.x; i < nst; i += blockDim.x)
        io.tiles[nrt + i] = TileInfo{E, kNt * i, min(kNt, io.T - kNt * i), 0};
    if (threadIdx.x == 0) {
        m->off[E] = npairs;
        m->tile_off[E] = nrt;
        m->tile_off[E + 1] = nrt + nst;
        m->n_tiles = nrt + nst;
        const int mr = (P.routed_neurons + 127) / 128, ms = (P.shared_neurons + 127) / 128;
        m->up_units = nrt * mr + nst * ms;
        m->dn_units = (nrt + nst) * (P.hidden / 128);  // 128-output bands of the down product
    }
    // live flags: one word per (tile, 32 k-tiles)
    const int words = io.max_tiles * ((max(P.routed_neurons, P.shared_neurons) / 64 + 31) / 32);
    for (int i = threadIdx.x; i < words; i += blockDim.x) io.flag_r[i] = 0u;
}

// CTA b handles tokens [16b, 16b + 16): each of its pairs (token, slot) gets
// its position in its expert's list, which keeps token order: the expert's
// offset, plus its pairs in earlier token blocks (counted by the route
// kernel), plus its pairs earlier in this block.  The CTA records positions
// and router weights, then gathers each of its tokens' x rows once and writes
// the row to the token's K routed positions and to its shared-expert row.
// Gathered rows are fp16; inside each group of 8 inputs (one word of codes)
// the order is e0 e4 e1 e5 e2 e6 e3 e7, the order in which the dequantiser
// emits nibble pairs (both operands of the up product use it).
constexpr int kListThreads = 256;

__device__ __forceinline__ uint4 bf16x8_to_fp16_perm(const uint4 v) {
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    __half hv[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        hv[2 * i] = __float2half_rn(__uint_as_float(wv[i] << 16));
        hv[2 * i + 1] = __float2half_rn(__uint_as_float(wv[i] & 0xffff0000u));
    }
    const __half2 p0 = __halves2half2(hv[0], hv[4]), p1 = __halves2half2(hv[1], hv[5]);
    const __half2 p2 = __halves2half2(hv[2], hv[6]), p3 = __halves2half2(hv[3], hv[7]);
    return make_uint4(*reinterpret_cast<const uint32_t*>(&p0), *reinterpret_cast<const uint32_t*>(&p1),
                      *reinterpret_cast<const uint32_t*>(&p2), *reinterpret_cast<const uint32_t*>(&p3));
}

__global__ void __launch_bounds__(kListThreads) prefill_list_kernel(const __grid_constant__ LayerParams P,
                                                                    const PrefillIO io) {
    __shared__ int base_e[kMaxRouted];
    __shared__ int e_of[kTokBlk * kMaxTopK];
    __shared__ int dst[kTokBlk][kMaxTopK + 1];  // destination rows of each token
    pdl_wait();
    pdl_trigger();
    const int E = P.n_routed, K = P.top_k, H = P.hidden, n = io.T * K;
    const int b = blockIdx.x, t0 = b * kTokBlk, nt = min(kTokBlk, io.T - t0), t = threadIdx.x;
    // expert offsets of this token block: the expert's offset, plus its pairs in the superblocks
    // before this block's (at most 31), plus those in the earlier blocks of this block's superblock
    // (at most kSuperBlk - 1); every load of a pass in flight together
    const int sb = b / kSuperBlk;
    for (int e = t; e < E; e += blockDim.x) {
        int c = __ldcg(&io.meta->off[e]);
        for (int s0 = 0; s0 < sb; s0 += 16) {
            int v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = s0 + i < sb ? __ldcg(&io.sb_cnt[(s0 + i) * E + e]) : 0;
#pragma unroll
            for (int i = 0; i < 16; ++i) c += v[i];
        }
        int w[kSuperBlk - 1];
#pragma unroll
        for (int i = 0; i < kSuperBlk - 1; ++i)
            w[i] = kSuperBlk * sb + i < b ? __ldcg(&io.blk_cnt[(kSuperBlk * sb + i) * E + e]) : 0;
#pragma unroll
        for (int i = 0; i < kSuperBlk - 1; ++i) c += w[i];
        base_e[e] = c;
    }
    for (int i = t; i < nt * K; i += blockDim.x) e_of[i] = __ldcg(io.idx + (size_t)t0 * K + i);
    __syncthreads();
    // positions: pairs of the block in token-major order, ranked within their expert
    for (int i = t; i < nt * K; i += blockDim.x) {
        const int e = e_of[i];
        int rank = 0;
        for (int j = 0; j < i; ++j) rank += (e_of[j] == e);
        const int p = t0 * K + i, pos = base_e[e] + rank;
        io.pair_tok[pos] = p / K;
        io.pair_w[pos] = __ldcg(io.w + p);
        io.pos_of[p] = pos;
        dst[i / K][i % K] = pos;
    }
    if (t < nt) dst[t][K] = P.shared_neurons ? n + t0 + t : -1;
    __syncthreads();
    // gather: each 16-byte piece of a token's row is loaded once and stored to every destination
    const int c8n = H / 8, nd = K + (P.shared_neurons ? 1 : 0);
    constexpr int kU = 4;
    for (int q0 = t; q0 < nt * c8n; q0 += kU * blockDim.x) {
        uint4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int q = q0 + u * blockDim.x;
            v[u] = q < nt * c8n ? __ldg(reinterpret_cast<const uint4*>(io.x + (size_t)(t0 + q / c8n) * H) + q % c8n)
                                : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int q = q0 + u * blockDim.x;
            if (q >= nt * c8n) break;
            const uint4 h = bf16x8_to_fp16_perm(v[u]);
            const int tk = q / c8n, c8 = q % c8n;
            for (int d = 0; d < nd; ++d)
                reinterpret_cast<uint4*>(io.xg + (size_t)dst[tk][d] * H)[c8] = h;
        }
    }
}

struct TMaps {
    CUtensorMap up_codes_r, up_codes_s;      // [rows][H/2] bytes, box 64 x 128, 64-byte swizzle
    CUtensorMap dn_codes_r, dn_codes_s;      // [rows][H/2] bytes, box 64 x 64, 64-byte swizzle
    CUtensorMap xg[8];                       // fp16 [rows][H], box 64 x 16(i+1), 128-byte swizzle
    CUtensorMap hr[8], hsh[8];               // fp16 h, box 64 x 16(i+1), 128-byte swizzle
    CUtensorMap hcr[8], hcs[8];              // fp16 h in entry order (row gather), same boxes
};

// ------------------------------------------------------------ GEMM kernels
// Both products run as persistent, warp-specialised kernels, one CTA per SM:
//   warps 0-3    epilogue: read the accumulator from TMEM (lanes 0-127)
//   warps 4-19   dequantise the 4-bit operand into fp16, in two groups of 8
//                warps that take alternate k-steps
//   warp 20      loads the 4-bit codes (and scales) by TMA: weight ring
//   warp 21      loads the 16-bit operand (x or h) by TMA: activation ring
//   warp 23      issues the tcgen05 MMAs (one thread); warp 22 idles
// Every ring slot has a "full" and an "empty" mbarrier; each role counts its
// own uses, so slot = q % depth and parity = (q / depth) & 1 (producers wait
// for the previous use of the slot to be released).  The accumulator is
// double-buffered in TMEM (two 128-column buffers), so the epilogue of one
// unit overlaps the main loop of the next.  Every wait is bounded; a role
// that gives up leaves its loop, and the others then give up in turn.
constexpr int kEpiWarps = 4;
constexpr int kDqGroup = 8;             // warps per dequantising group
constexpr int kDqWarps = 2 * kDqGroup;
constexpr int kWarpW = kEpiWarps + kDqWarps;   // 20
constexpr int kWarpX = kWarpW + 1;             // 21
constexpr int kWarpMma = kWarpX + 2;           // 23: sub-partition 3, which hosts the fewest other warps
constexpr int kGemmThreads = 32 * (kWarpMma + 1);
constexpr int kTileX = kNt * 128;       // up to 128 rows x 64 fp16
constexpr unsigned kProducerSleepNs = 64;
constexpr unsigned kEpilogueSleepNs = 256;

// Ring depths: weight codes (WD) and stages (SD).  A stage is one k-step's
// 16-bit operand (loaded by TMA) together with its dequantised tile: its
// "full" barrier completes when the TMA bytes have landed and every lane of
// the dequantising group's warps has arrived; one MMA commit releases both.
template <int WD, int SD, int DQ = kDqGroup>
struct GemmBars {
    uint64_t *wfull, *wempty, *sfull, *sempty, *sbfull, *sbempty, *tfull, *tempty;
    uint32_t* tmem_slot;
    static constexpr int kCount = 2 * WD + 2 * SD + 2 * 2 + 2 * 2;
    __device__ GemmBars(uint8_t* p) {
        uint64_t* b = reinterpret_cast<uint64_t*>(p);
        wfull = b; wempty = wfull + WD; sfull = wempty + WD; sempty = sfull + SD;
        sbfull = sempty + SD; sbempty = sbfull + 2; tfull = sbempty + 2; tempty = tfull + 2;
        tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
    }
    // wfull_count: arrivals that fill a weight slot (1: one TMA issuer; 32: a warp
    // whose lanes each count their own cp.async copies)
    __device__ void init(uint32_t wfull_count = 1) {
        for (int i = 0; i < WD; ++i) { mbar_init(&wfull[i], wfull_count); mbar_init(&wempty[i], DQ); }
        // every thread that wrote or read tensor memory arrives itself, after its
        // own wait and tcgen05 fence: the dequantising warps' 32 lanes on the
        // stage's full barrier (plus the TMA's arrival), the epilogue's on the
        // accumulator's empty barrier
        for (int i = 0; i < SD; ++i) { mbar_init(&sfull[i], 32 * DQ + 1); mbar_init(&sempty[i], 1); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sbfull[i], 1); mbar_init(&sbempty[i], kDqWarps);
            mbar_init(&tfull[i], 1); mbar_init(&tempty[i], 32 * kEpiWarps);
        }
        fence_mbar_init();
    }
};

// A parity wait is only sound when the barrier is at most one phase behind
// the phase waited for: two phases behind, the current (incomplete) phase has
// the parity of the one wanted and the test passes at once.  A role that
// takes every use of a slot has seen the slot's previous phase itself.  The
// dequantising groups take the k-steps round robin, so every ring they wait on
// either has a depth that is a multiple of the group count (each slot belongs
// to one group), or is waited on only after a wait that proves its previous
// phase complete (see the up kernel's weight ring).

// Producer-side wait for slot q of a ring of depth d to be free.
__device__ __forceinline__ bool wait_free(uint64_t* empty, int d, uint32_t q) {
    return mbar_wait(&empty[q % d], ((q / d) & 1u) ^ 1u);
}
__device__ __forceinline__ bool wait_full(uint64_t* full, int d, uint32_t q) {
    return mbar_wait(&full[q % d], (q / d) & 1u);
}
// The same with a sleep between polls (producers, epilogue).
__device__ __forceinline__ bool wait_free_sleep(uint64_t* empty, int d, uint32_t q, unsigned ns) {
    return mbar_wait_sleep(&empty[q % d], ((q / d) & 1u) ^ 1u, ns);
}
__device__ __forceinline__ bool wait_full_sleep(uint64_t* full, int d, uint32_t q, unsigned ns) {
    return mbar_wait_sleep(&full[q % d], (q / d) & 1u, ns);
}
// A producer on its way out: waits (bounded) for its last loads to land.
__device__ __forceinline__ void drain_loads(uint64_t* full, int d, uint32_t issued) {
    for (uint32_t q = issued > (uint32_t)d ? issued - d : 0; q < issued; ++q) wait_full(full, d, q);
}

// ---- up GEMM: unit = (token tile, 128-neuron block); D[neuron][token].  One k-step covers
// 128 inputs (two scale groups).  TMEM: columns 0-255 the two accumulators, 256-511 four
// dequantised A tiles (128 lanes x 64 columns = 128 rows x 128 fp16 each).
constexpr int kUpWD = 5, kUpSD = 4;
constexpr int kUpDqGroup = 4;   // warps per dequantising group (one per TMEM lane quadrant); 4 groups
using UpBars = GemmBars<kUpWD, kUpSD, kUpDqGroup>;
// Stage slot q % 4 belongs to group q % 4.  The weight slot q % 5 was last
// filled for k-step q - 5, which another group dequantised; a group therefore
// waits for its stage slot's release first: the MMA has then consumed k-step
// q - 4, hence q - 5, whose codes had landed, and the weight slot's barrier is
// at most one phase behind when the group waits on it.
static_assert(kUpSD == kDqWarps / kUpDqGroup && kUpWD >= kUpSD, "up rings: see the parity-wait invariant");
constexpr int kUpK = 128;                  // inputs per k-step

struct UpLayout {
    static constexpr int kXSlot = 2 * kTileX;           // two 64-input swizzled sub-tiles
    static constexpr int kX = 0;
    static constexpr int kW = kX + kUpSD * kXSlot;
    static constexpr int kWSlot = 128 * kUpK / 2;       // 128 rows x 128 codes
    static constexpr int kSB = kW + kUpWD * kWSlot;
    __host__ __device__ static int sb_words(int H) { return 128 * (H / 64); }
    __host__ __device__ static int bars(int H) { return kSB + 2 * 4 * sb_words(H); }
    __host__ __device__ static int total(int H) { return 1024 + bars(H) + 8 * UpBars::kCount + 64; }
};

struct UpUnit {
    int tile, row0, rows, ntok, nt16, cy, xrow, N, row_out;
    bool shared;
    ExpertPtrs ep;
};

__device__ __forceinline__ UpUnit up_unit(const LayerParams& P, const PrefillIO& io, int ntr, int mr, int ms, int u) {
    UpUnit d;
    int mb;
    if (u < ntr * mr) { d.tile = u / mr; mb = u % mr; }
    else { d.tile = ntr + (u - ntr * mr) / ms; mb = (u - ntr * mr) % ms; }
    const TileInfo ti = io.tiles[d.tile];
    d.shared = ti.e == P.n_routed;
    d.N = d.shared ? P.shared_neurons : P.routed_neurons;
    d.ep = d.shared ? P.shared : routed_ptrs(P, ti.e);
    d.row0 = 128 * mb;
    d.rows = min(128, d.N - d.row0);
    d.ntok = ti.ntok;
    d.nt16 = (ti.ntok + 15) & ~15;
    d.cy = d.shared ? d.row0 : ti.e * P.routed_neurons + d.row0;
    d.xrow = d.shared ? io.T * P.top_k + ti.row0 : ti.row0;
    d.row_out = ti.row0;
    return d;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
prefill_up_kernel(const __grid_constant__ LayerParams P, const PrefillIO io, const __grid_constant__ TMaps tm) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int H = P.hidden, G = H / 64, KS = H / kUpK;
    uint8_t* sX = smem + UpLayout::kX;
    uint8_t* sW = smem + UpLayout::kW;
    uint32_t* sSB = reinterpret_cast<uint32_t*>(smem + UpLayout::kSB);
    const int sbw = UpLayout::sb_words(H);
    UpBars br(smem + UpLayout::bars(H));
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    if (t == 0) br.init();
    if (warp == 0) tmem_alloc(br.tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *br.tmem_slot;
    const uint32_t tmem_a = tmem + 256;
    pdl_wait();
    pdl_trigger();
    const PrefillMeta* m = io.meta;
    const int E = P.n_routed, NR = P.routed_neurons, NS = P.shared_neurons;
    const int ntr = m->tile_off[E];
    const int mr = (NR + 127) / 128, ms = (NS + 127) / 128;
    const int U = m->up_units;
    const int words = (max(NR, NS) / 64 + 31) / 32;
    bool ok = true;

    if (warp == kWarpW) {
        // ---- weight codes and (scale, bias) of each unit's rows
        if (lane == 0) {
            const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
            uint32_t wq = 0, nsb = 0;
            // the next unit's descriptor is loaded one unit ahead (its loads overlap this unit's work)
            UpUnit dnext;
            if ((int)blockIdx.x < U) dnext = up_unit(P, io, ntr, mr, ms, blockIdx.x);
            for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
                const UpUnit d = dnext;
                if (u + (int)gridDim.x < U) dnext = up_unit(P, io, ntr, mr, ms, u + gridDim.x);
                const int b = nsb & 1;
                if (!(ok = wait_free_sleep(br.sbempty, 2, nsb, kProducerSleepNs))) break;
                mbar_arrive_expect_tx(&br.sbfull[b], (uint32_t)d.rows * G * 4);
                bulk_g2s(sSB + b * sbw, d.ep.up_sb + (size_t)d.row0 * G, (uint32_t)d.rows * G * 4, &br.sbfull[b],
                         d.shared ? pol_keep : pol_stream);
                ++nsb;
                const CUtensorMap* cmap = d.shared ? &tm.up_codes_s : &tm.up_codes_r;
                for (int k = 0; k < KS; ++k) {
                    if (!(ok = wait_free_sleep(br.wempty, kUpWD, wq, kProducerSleepNs))) break;
                    const int s = wq % kUpWD;
                    mbar_arrive_expect_tx(&br.wfull[s], UpLayout::kWSlot);
                    tma_load_2d_hint(sW + s * UpLayout::kWSlot, cmap, (kUpK / 2) * k, d.cy, &br.wfull[s],
                                     d.shared ? pol_keep : pol_stream);
                    ++wq;
                }
            }
            drain_loads(br.wfull, kUpWD, wq);
            drain_loads(br.sbfull, 2, nsb);
        }
        __syncwarp();
    } else if (warp == kWarpX) {
        // ---- gathered tokens (B operand): two 64-input sub-tiles per k-step
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            uint32_t xq = 0;
            // the next unit's descriptor is loaded one unit ahead (its loads overlap this unit's work)
            UpUnit dnext;
            if ((int)blockIdx.x < U) dnext = up_unit(P, io, ntr, mr, ms, blockIdx.x);
            for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
                const UpUnit d = dnext;
                if (u + (int)gridDim.x < U) dnext = up_unit(P, io, ntr, mr, ms, u + gridDim.x);
                // a box of exactly the tile's rows rounded up to 16 (the MMA's N)
                const CUtensorMap* xmap = &tm.xg[d.nt16 / 16 - 1];
                const uint32_t bytes = (uint32_t)d.nt16 * 128;
                for (int k = 0; k < KS; ++k) {
                    if (!(ok = wait_free_sleep(br.sempty, kUpSD, xq, kProducerSleepNs))) break;
                    const int x = xq % kUpSD;
                    uint8_t* dst = sX + x * UpLayout::kXSlot;
                    mbar_arrive_expect_tx(&br.sfull[x], 2 * bytes);
                    tma_load_2d_hint(dst, xmap, kUpK * k, d.xrow, &br.sfull[x], pol);
                    tma_load_2d_hint(dst + kTileX, xmap, kUpK * k + 64, d.xrow, &br.sfull[x], pol);
                    ++xq;
                }
            }
            drain_loads(br.sfull, kUpSD, xq);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ---- MMA issue: A (weights) from TMEM, B (tokens) from shared memory
        if (lane == 0) {
            uint32_t sq = 0, nu = 0;
            // the next unit's descriptor is loaded one unit ahead (its loads overlap this unit's work)
            UpUnit dnext;
            if ((int)blockIdx.x < U) dnext = up_unit(P, io, ntr, mr, ms, blockIdx.x);
            for (int u = blockIdx.x; u < U && ok; u += gridDim.x, ++nu) {
                const UpUnit d = dnext;
                if (u + (int)gridDim.x < U) dnext = up_unit(P, io, ntr, mr, ms, u + gridDim.x);
                const int acc = nu & 1;
                if (!(ok = wait_free(br.tempty, 2, nu))) break;
                tc_fence_after();
                const uint32_t idesc = umma_idesc_f16_f32(128, d.nt16);
                const uint32_t dt = tmem + (uint32_t)(acc * 128);
                for (int k = 0; k < KS; ++k) {
                    if (!(ok = wait_full(br.sfull, kUpSD, sq))) break;
                    tc_fence_after();
                    const int a = sq % kUpSD;
                    const uint64_t bd0 = umma_desc_sw128(smem_u32(sX + a * UpLayout::kXSlot));
                    const uint64_t bd1 = umma_desc_sw128(smem_u32(sX + a * UpLayout::kXSlot + kTileX));
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        umma_f16_tmem_a(dt, tmem_a + 64 * a + 8 * j, (j < 4 ? bd0 : bd1) + 2 * (j & 3), idesc,
                                        (k | j) != 0);
                    umma_commit(&br.sempty[a]);
                    ++sq;
                }
                if (ok) umma_commit(&br.tfull[acc]);
            }
            // every MMA issued has completed once the last commit has arrived
            if (sq) wait_full(br.sempty, kUpSD, sq - 1);
        }
        __syncwarp();
    } else if (warp >= kEpiWarps && warp < kWarpW) {
        // ---- dequantise into TMEM: group g = (warp - 4) / 4 takes the k-steps q with q % 4 == g.
        // Thread (row r) converts the 128 codes of scale groups 2k and 2k+1 (halves h = 0, 1) and
        // writes columns 32h..32h+31 of row r; each column holds two codes of one word in the
        // order (c0 c4) (c1 c5) (c2 c6) (c3 c7)
        const int g = (warp - kEpiWarps) / kUpDqGroup;
        const int r = 32 * (warp & 3) + lane;
        const uint32_t trow = tmem_a + ((uint32_t)(32 * (warp & 3)) << 16);
        uint32_t q = 0, nsb = 0;
        const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f), k1_16 = __floats2half2_rn(0.0625f, 0.0625f);
        // the next unit's descriptor is loaded one unit ahead (its loads overlap this unit's work)
        UpUnit dnext;
        if ((int)blockIdx.x < U) dnext = up_unit(P, io, ntr, mr, ms, blockIdx.x);
        for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
            const UpUnit d = dnext;
            if (u + (int)gridDim.x < U) dnext = up_unit(P, io, ntr, mr, ms, u + gridDim.x);
            const int b = nsb & 1;
            ok = __all_sync(0xffffffffu, wait_full(br.sbfull, 2, nsb));
            if (!ok) break;
            const uint32_t* sbr = sSB + b * sbw + r * G;
            for (int k = (g - (int)(q & 3u) + 4) & 3; k < KS; k += 4) {
                const uint32_t qk = q + k;
                // stage release first: it proves the weight slot's previous load complete
                ok = __all_sync(0xffffffffu, wait_free(br.sempty, kUpSD, qk) && wait_full(br.wfull, kUpWD, qk));
                if (!ok) break;
                tc_fence_after();
                const int s = qk % kUpWD;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                uint32_t o[32];
                if (r < d.rows) {
                    // the codes tile arrives with the 64-byte swizzle: 16-byte chunk c of row r sits at
                    // chunk c ^ ((r >> 1) & 3), so the 32 rows a warp reads cover all banks
                    const uint8_t* crow = sW + s * UpLayout::kWSlot + r * (kUpK / 2);
                    const int sw = (r >> 1) & 3;
                    const uint4 c0 = *reinterpret_cast<const uint4*>(crow + (((2 * h) ^ sw) << 4));
                    const uint4 c1 = *reinterpret_cast<const uint4*>(crow + (((2 * h + 1) ^ sw) << 4));
                    // (scale, bias) in fp16 as stored; scale / 16 is exact (or rounds as an fp32 division would)
                    const __half2 sbh = *reinterpret_cast<const __half2*>(&sbr[2 * k + h]);
                    const __half2 s1 = __low2half2(sbh), b2 = __high2half2(sbh);
                    const __half2 s16 = __hmul2(s1, k1_16);
                    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t lo = w[j], hi = w[j] >> 8;
                        // fp16 1024 + c (or 1024 + 16c): the code sits in the low mantissa bits
                        const uint32_t pr[4] = {(lo & 0x000F000Fu) | 0x64006400u, (lo & 0x00F000F0u) | 0x64006400u,
                                                (hi & 0x000F000Fu) | 0x64006400u, (hi & 0x00F000F0u) | 0x64006400u};
#pragma unroll
                        for (int p = 0; p < 4; ++p) {
                            const __half2 qv = __hsub2(*reinterpret_cast<const __half2*>(&pr[p]), k1024);
                            const __half2 v = __hfma2(qv, (p & 1) ? s16 : s1, b2);
                            o[4 * j + p] = *reinterpret_cast<const uint32_t*>(&v);
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                __syncwarp();
                tmem_st32(trow + 64 * (qk % kUpSD) + 32 * h, o);
                // tcgen05.st reads its source registers asynchronously: they hold
                // this half until the wait, before the next half is computed into them
                tmem_st_wait();
                }
                tc_fence_before();
                mbar_arrive(&br.sfull[qk % kUpSD]);   // each lane, after its own stores' wait and fence
                __syncwarp();
                if (lane == 0) mbar_arrive(&br.wempty[s]);
            }
            if (!ok) break;
            q += KS;
            __syncwarp();
            if (lane == 0) mbar_arrive(&br.sbempty[b]);
            ++nsb;
        }
    } else if (warp < kEpiWarps) {
        // ---- epilogue: + offset, ReLU^2, H (fp16) and the live flags of the block's 64-neuron tiles
        uint32_t nu = 0;
        // the next unit's descriptor is loaded one unit ahead (its loads overlap this unit's work)
        UpUnit dnext;
        if ((int)blockIdx.x < U) dnext = up_unit(P, io, ntr, mr, ms, blockIdx.x);
        for (int u = blockIdx.x; u < U && ok; u += gridDim.x, ++nu) {
            const UpUnit d = dnext;
            if (u + (int)gridDim.x < U) dnext = up_unit(P, io, ntr, mr, ms, u + gridDim.x);
            const int acc = nu & 1;
            const int r = 32 * warp + lane, n = d.row0 + r;
            const bool rowok = r < d.rows;
            const float off = (rowok && d.ep.up_off) ? __ldg(d.ep.up_off + n) : 0.f;
            // h is stored with each group of 8 neurons in the order n0 n4 n1 n5 n2 n6 n3 n7 (the order
            // in which the down product's dequantiser yields nibble pairs)
            const int n8 = n & 7, nst = (n & ~7) | (n8 < 4 ? 2 * n8 : 2 * (n8 - 4) + 1);
            uint16_t* hcol = (d.shared ? io.h_s : io.h_r) + (size_t)d.row_out * d.N + nst;
            ok = __all_sync(0xffffffffu, wait_full_sleep(br.tfull, 2, nu, kEpilogueSleepNs));
            if (!ok) break;
            tc_fence_after();
            uint32_t live = 0;
            for (int c0 = 0; c0 < d.nt16; c0 += 32) {
                float v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(acc * 128 + c0), v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int c = c0 + i;
                    const float z = v[i] + off;
                    const uint16_t hb = __half_as_ushort(__float2half_rn(z > 0.f ? z * z : 0.f));
                    if (rowok && c < d.ntok) {
                        hcol[(size_t)c * d.N] = hb;
                        live |= hb;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&br.tempty[acc]);   // each lane, after its own loads and fence
            const unsigned anylive = __ballot_sync(0xffffffffu, live != 0);
            const bool force = (io.flags & HS_FORCE_DENSE) != 0;
            if (lane == 0 && 32 * warp < d.rows && (anylive || force)) {
                const int kt = (d.row0 + 32 * warp) / 64;
                atomicOr(io.flag_r + (size_t)d.tile * words + kt / 32, 1u << (kt % 32));
            }
            if (lane == 0 && anylive)
                atomicAdd(&io.meta->union_rt, (unsigned long long)__popc(anylive) * (unsigned long long)d.ntok);
            if (io.umask && lane == 0 && 32 * warp < d.rows)
                io.umask[(size_t)d.tile * kUWords + (d.row0 + 32 * warp) / 32] = anylive;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---- down GEMM (operands swapped): unit = (token tile, band of 128 outputs); D^T[output][token]
// over the live 64-neuron tiles of the expert.  A = the band's weights, transposed and dequantised
// straight into TMEM: each warp loads 32 neuron rows x 32 outputs of codes (one 16-byte chunk per
// lane), transposes the 32 x 32 nibbles in registers (lane = output) and writes the fp16 weights
// (column c = the neurons at stored h positions 2c, 2c+1).  B = h of the tile's tokens (K-major,
// by TMA).  The up epilogue stores h with the neurons of each group of 8 in the order
// n0 n4 n1 n5 n2 n6 n3 n7, the order in which a code word yields nibble pairs, so no further
// shuffling is needed.  The epilogue lane owns one output and writes it for every token.
constexpr int kDnBand = 128;
constexpr int kDnWD = 8, kDnSD = 8;
constexpr int kDnDqGroup = 4;   // warps per dequantising group (one per TMEM lane quadrant); 4 groups
using DnBars = GemmBars<kDnWD, kDnSD, kDnDqGroup>;
// Both rings a multiple of the group count: slot q % 8 of either ring belongs
// to group q % 4, which has seen the slot's previous phase itself.  TMEM holds
// the two accumulators (256 columns) and the 8 A tiles of 32 columns.
static_assert(kDnWD % (kDqWarps / kDnDqGroup) == 0 && kDnSD % (kDqWarps / kDnDqGroup) == 0,
              "down rings: see the parity-wait invariant");
static_assert(256 + 32 * kDnSD <= 512, "down A tiles exceed the TMEM allocation");

struct DownLayout {
    static constexpr int kCodes = 64 * kDnBand / 2;     // 64 neurons x 64 bytes, 64-byte swizzle
    static constexpr int kWSlot = kCodes + kDnBand * 4;  // + the slab slice (scale, bias) of the band
    static constexpr int kX = 0;                         // h tiles: up to 128 rows x 128 B
    static constexpr int kW = kX + kDnSD * kTileX;
    static constexpr int kBarsOff = kW + kDnWD * kWSlot;
    static constexpr int kTotal = 1024 + kBarsOff + 8 * DnBars::kCount + 64;
};

// Row-gather weight slot: the k-step's 64 entry rows (64 bytes of codes each,
// at a stride of 80 bytes: the dequantiser's lane pattern then touches every
// bank once), the (scale, bias) slab slices of groups gA and gB, and the
// aligned 16 bytes of the tile's descriptor row that hold the k-step's
// descriptor (word kk % 4).
struct DownLayoutG {
    static constexpr int kRowStride = 80;
    static constexpr int kCodes = 64 * kRowStride;
    static constexpr int kSlab = kCodes;                       // two slices of kDnBand (scale, bias) pairs
    static constexpr int kDesc = kSlab + 2 * kDnBand * 4;
    static constexpr int kWSlot = (kDesc + 16 + 127) & ~127;
    static constexpr int kX = 0;
    static constexpr int kW = kX + kDnSD * kTileX;
    static constexpr int kBarsOff = kW + kDnWD * kWSlot;
    static constexpr int kTotal = 1024 + kBarsOff + 8 * DnBars::kCount + 64;
};

struct DownUnit {
    int tile, ob, ntok, nt16, cy0, NK, row0, nk;
    bool shared;
    ExpertPtrs ep;
    uint64_t live;   // tile mode: bit j = 64-neuron tile j is multiplied
};

template <bool kGather>
__device__ __forceinline__ DownUnit down_unit(const LayerParams& P, const PrefillIO& io, int nb, int words, bool dense,
                                              int u) {
    DownUnit d;
    d.tile = u / nb;
    d.ob = u % nb;
    const TileInfo ti = io.tiles[d.tile];
    d.shared = ti.e == P.n_routed;
    d.NK = (d.shared ? P.shared_neurons : P.routed_neurons) / 64;
    d.ep = d.shared ? P.shared : routed_ptrs(P, ti.e);
    d.ntok = ti.ntok;
    d.nt16 = (ti.ntok + 15) & ~15;
    d.cy0 = d.shared ? 0 : ti.e * P.routed_neurons;
    d.row0 = ti.row0;
    if (kGather) {
        d.live = 0;
        d.nk = __ldcg(io.nks + d.tile);
    } else {
        const uint32_t* f = io.flag_r + (size_t)d.tile * words;
        const uint64_t all = d.NK == 64 ? ~0ull : ((1ull << d.NK) - 1ull);
        d.live = dense ? all : ((uint64_t)__ldcg(f) | (words > 1 ? (uint64_t)__ldcg(f + 1) << 32 : 0ull)) & all;
        d.nk = __popcll(d.live);
    }
    return d;
}

// Iterates the live tiles of a unit in ascending order.
__device__ __forceinline__ int pop_live(uint64_t& m) {
    const int j = __ffsll((long long)m) - 1;
    m &= m - 1;
    return j;
}

// kGather: k-step kk of a unit multiplies the tile's entries 64 kk .. 64 kk + 63
// (rowgather plan) instead of its kk-th live 64-neuron tile.
template <bool kGather>
__global__ void __launch_bounds__(kGemmThreads, 1)
prefill_down_kernel(const __grid_constant__ LayerParams P, const PrefillIO io, const __grid_constant__ TMaps tm) {
    using Lay = typename std::conditional<kGather, DownLayoutG, DownLayout>::type;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int H = P.hidden;
    uint8_t* sX = smem + Lay::kX;
    uint8_t* sW = smem + Lay::kW;
    DnBars br(smem + Lay::kBarsOff);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    if (t == 0) br.init(kGather ? 32u : 1u);
    if (warp == 0) tmem_alloc(br.tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *br.tmem_slot;
    const uint32_t tmem_a = tmem + 256;   // kDnSD dequantised A tiles of 32 columns
    pdl_wait();
    pdl_trigger();
    PrefillMeta* m = io.meta;
    const int NR = P.routed_neurons, NS = P.shared_neurons, K = P.top_k;
    const int nb = H / kDnBand;
    const int U = m->dn_units;
    const int words = (max(NR, NS) / 64 + 31) / 32;
    const bool dense = (io.flags & HS_FORCE_DENSE) != 0;
    bool ok = true;

    if (warp == kWarpW && kGather) {
        // ---- each k-step's 64 entry rows and the slab slices of its groups gA and gB, by
        // 16-byte cp.async from every lane (row copies of 64 bytes are too small for the bulk
        // copy engine to keep up): 256 row chunks and 64 slab chunks, 10 per lane, plus the
        // k-step's descriptor (lane 0); each lane's copies arrive on the slot's barrier once
        // they have landed (32 arrivals)
        const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
        uint32_t wq = 0;
        DownUnit dnext;
        if ((int)blockIdx.x < U) dnext = down_unit<kGather>(P, io, nb, words, dense, blockIdx.x);
        for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
            const DownUnit d = dnext;
            if (u + (int)gridDim.x < U) dnext = down_unit<kGather>(P, io, nb, words, dense, u + gridDim.x);
            const uint64_t pol = d.shared ? pol_keep : pol_stream;
            const uint16_t* L = io.glist + (size_t)d.tile * 64 * kMaxKTiles;
            const uint32_t* D = io.ksd + (size_t)d.tile * kMaxKTiles;
            const uint8_t* codes = d.ep.dn_codes + (kDnBand / 2) * d.ob;
            const uint8_t* slab = reinterpret_cast<const uint8_t*>(d.ep.dn_sb + kDnBand * d.ob);
            // the entries (two per lane) and descriptor of k-step kk + 1 are loaded while kk is issued
            uint32_t e2 = d.nk > 0 ? __ldcg(reinterpret_cast<const uint32_t*>(L) + lane) : 0u;
            uint32_t desc = d.nk > 0 ? __ldcg(D) : 0u;
            for (int kk = 0; kk < d.nk; ++kk) {
                const uint32_t e2c = e2, descc = desc;
                if (kk + 1 < d.nk) {
                    e2 = __ldcg(reinterpret_cast<const uint32_t*>(L + 64 * (kk + 1)) + lane);
                    desc = __ldcg(D + kk + 1);
                }
                if (lane == 0) ok = wait_free_sleep(br.wempty, kDnWD, wq, kProducerSleepNs);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                const int s = wq % kDnWD;
                uint8_t* slot = sW + s * Lay::kWSlot;
                // chunk c = lane + 32 i: row c / 4 (entry lane / 4 + 8 i), 16-byte part c % 4
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = (lane >> 2) + 8 * i;
                    const uint32_t pair = __shfl_sync(0xffffffffu, e2c, row >> 1);
                    const uint32_t v = (pair >> (16 * (row & 1))) & 0xFFFFu;
                    const int n = v == rowgather::kPad ? 0 : (int)v;   // a padding entry reads row 0 against h = 0
                    cp_async16_hint(slot + row * DownLayoutG::kRowStride + 16 * (lane & 3),
                                    codes + (size_t)n * (H / 2) + 16 * (lane & 3), pol);
                }
                cp_async16_hint(slot + DownLayoutG::kSlab + 16 * lane,
                                slab + (size_t)rowgather::ksd_gA(descc) * H * 4 + 16 * lane, pol);
                cp_async16_hint(slot + DownLayoutG::kSlab + kDnBand * 4 + 16 * lane,
                                slab + (size_t)rowgather::ksd_gB(descc) * H * 4 + 16 * lane, pol);
                // the dequantisers read the descriptor from the slot, not from global memory
                if (lane == 0)
                    cp_async16_hint(slot + DownLayoutG::kDesc, D + (kk & ~3), pol_keep);
                cp_async_arrive_noinc(&br.wfull[s]);
                ++wq;
            }
            if (ok && d.ob == 0 && lane == 0) {
                atomicAdd(&m->total, d.NK);
                atomicAdd(&m->skipped, d.NK - d.nk);
                atomicAdd(&m->exec_rt, (unsigned long long)d.ntok * 64ull * (unsigned long long)d.nk);
                atomicAdd(&m->dense_rt, (unsigned long long)d.ntok * 64ull * (unsigned long long)d.NK);
            }
        }
        // every lane's copies have landed, and their arrivals are on the barriers, before the
        // CTA can leave
        cp_async_wait_all();
        __syncwarp();
        if (lane == 0) drain_loads(br.wfull, kDnWD, wq);
        __syncwarp();
    } else if (warp == kWarpW) {
        // ---- codes + (scale, bias) slab slice of each live 64-neuron tile, this band
        if (lane == 0) {
            const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
            uint32_t wq = 0;
            // the next unit's descriptor is loaded one unit ahead (its loads overlap this unit's work)
            DownUnit dnext;
            if ((int)blockIdx.x < U) dnext = down_unit<kGather>(P, io, nb, words, dense, blockIdx.x);
            for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
                const DownUnit d = dnext;
                if (u + (int)gridDim.x < U) dnext = down_unit<kGather>(P, io, nb, words, dense, u + gridDim.x);
                const CUtensorMap* cmap = d.shared ? &tm.dn_codes_s : &tm.dn_codes_r;
                const uint64_t pol = d.shared ? pol_keep : pol_stream;
                for (uint64_t lm = d.live; lm && ok;) {
                    const int j = pop_live(lm);
                    if (!(ok = wait_free_sleep(br.wempty, kDnWD, wq, kProducerSleepNs))) break;
                    const int s = wq % kDnWD;
                    uint8_t* slot = sW + s * Lay::kWSlot;
                    mbar_arrive_expect_tx(&br.wfull[s], (uint32_t)DownLayout::kWSlot);
                    tma_load_2d_hint(slot, cmap, (kDnBand / 2) * d.ob, d.cy0 + 64 * j, &br.wfull[s], pol);
                    bulk_g2s(slot + DownLayout::kCodes, d.ep.dn_sb + (size_t)j * H + kDnBand * d.ob, kDnBand * 4,
                             &br.wfull[s], pol);
                    ++wq;
                }
                if (ok && d.ob == 0) {
                    atomicAdd(&m->total, d.NK);
                    atomicAdd(&m->skipped, d.NK - d.nk);
                    atomicAdd(&m->exec_rt, (unsigned long long)d.ntok * 64ull * (unsigned long long)d.nk);
                    atomicAdd(&m->dense_rt, (unsigned long long)d.ntok * 64ull * (unsigned long long)d.NK);
                }
            }
            drain_loads(br.wfull, kDnWD, wq);
        }
        __syncwarp();
    } else if (warp == kWarpX) {
        // ---- h of the tile's tokens (B operand): a box of the tile's rows rounded up to 16
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            uint32_t xq = 0;
            // the next unit's descriptor is loaded one unit ahead (its loads overlap this unit's work)
            DownUnit dnext;
            if ((int)blockIdx.x < U) dnext = down_unit<kGather>(P, io, nb, words, dense, blockIdx.x);
            for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
                const DownUnit d = dnext;
                if (u + (int)gridDim.x < U) dnext = down_unit<kGather>(P, io, nb, words, dense, u + gridDim.x);
                const CUtensorMap* hmap = kGather ? (d.shared ? &tm.hcs[d.nt16 / 16 - 1] : &tm.hcr[d.nt16 / 16 - 1])
                                                  : (d.shared ? &tm.hsh[d.nt16 / 16 - 1] : &tm.hr[d.nt16 / 16 - 1]);
                uint64_t lm = d.live;
                for (int kk = 0; kk < d.nk && ok; ++kk) {
                    const int col = kGather ? 64 * kk : 64 * pop_live(lm);
                    if (!(ok = wait_free_sleep(br.sempty, kDnSD, xq, kProducerSleepNs))) break;
                    const int x = xq % kDnSD;
                    mbar_arrive_expect_tx(&br.sfull[x], (uint32_t)d.nt16 * 128u);
                    tma_load_2d_hint(sX + x * kTileX, hmap, col, d.row0, &br.sfull[x], pol);
                    ++xq;
                }
            }
            drain_loads(br.sfull, kDnSD, xq);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ---- MMA issue: A (weights) from TMEM, B (h) from shared memory
        if (lane == 0) {
            uint32_t sq = 0, nu = 0;
            // the next unit's descriptor is loaded one unit ahead (its loads overlap this unit's work)
            DownUnit dnext;
            if ((int)blockIdx.x < U) dnext = down_unit<kGather>(P, io, nb, words, dense, blockIdx.x);
            for (int u = blockIdx.x; u < U && ok; u += gridDim.x, ++nu) {
                const DownUnit d = dnext;
                if (u + (int)gridDim.x < U) dnext = down_unit<kGather>(P, io, nb, words, dense, u + gridDim.x);
                const int acc = nu & 1;
                if (!(ok = wait_free(br.tempty, 2, nu))) break;
                tc_fence_after();
                const uint32_t idesc = umma_idesc_f16_f32(128, d.nt16);
                const uint32_t dt = tmem + (uint32_t)(acc * 128);
                for (int kk = 0; kk < d.nk; ++kk) {
                    if (!(ok = wait_full(br.sfull, kDnSD, sq))) break;
                    tc_fence_after();
                    const int a = sq % kDnSD;
                    const uint64_t bd = umma_desc_sw128(smem_u32(sX + a * kTileX));
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        umma_f16_tmem_a(dt, tmem_a + 32 * a + 8 * j, bd + 2 * j, idesc, (kk | j) != 0);
                    umma_commit(&br.sempty[a]);
                    ++sq;
                }
                if (ok) umma_commit(&br.tfull[acc]);   // also when no tile was live
            }
            if (sq) wait_full(br.sempty, kDnSD, sq - 1);
        }
        __syncwarp();
    } else if (warp >= kEpiWarps && warp < kWarpW) {
        // ---- dequantise into TMEM: group g = (warp - 4) / 4 takes the k-steps q with q % 4 == g.
        // Warp quadrant qd = warp % 4: outputs 32qd .. 32qd+31 of the band (TMEM lanes), all 64
        // neurons (entries) of the k-step (32 columns of the A tile), in two halves of 32
        const int g = (warp - kEpiWarps) / kDnDqGroup, qd = warp & 3;
        const uint32_t trow = tmem_a + ((uint32_t)(32 * qd) << 16);
        // lane l takes word l/8 of the quadrant's 16-byte chunk in rows 32hh + 8k + l%8 (the
        // word-level steps of the transpose done by the loads).  Tile mode: 64-byte swizzle, chunk c
        // of row r at chunk c ^ ((r >> 1) & 3).  Gather mode: rows 80 bytes apart, unswizzled.
        int ldoff[2][4];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int r = 32 * hh + (lane & 7) + 8 * k;
                ldoff[hh][k] = kGather ? r * DownLayoutG::kRowStride + (qd << 4) + 4 * (lane >> 3)
                                       : r * (kDnBand / 2) + ((qd ^ ((r >> 1) & 3)) << 4) + 4 * (lane >> 3);
            }
        const NibTrLane trc = nib_tr_lane();
        const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f), k1_16 = __floats2half2_rn(0.0625f, 0.0625f);
        uint32_t q = 0;
        // the next unit's descriptor is loaded one unit ahead (its loads overlap this unit's work)
        DownUnit dnext;
        if ((int)blockIdx.x < U) dnext = down_unit<kGather>(P, io, nb, words, dense, blockIdx.x);
        for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
            const DownUnit d = dnext;
            if (u + (int)gridDim.x < U) dnext = down_unit<kGather>(P, io, nb, words, dense, u + gridDim.x);
            const int nk = d.nk;
            for (int kk = (g - (int)(q & 3u) + 4) & 3; kk < nk; kk += 4) {
                const uint32_t qk = q + kk;
                ok = __all_sync(0xffffffffu, wait_free(br.sempty, kDnSD, qk) && wait_full(br.wfull, kDnWD, qk));
                if (!ok) break;
                tc_fence_after();
                const int s = qk % kDnWD;
                const uint8_t* cs = sW + s * Lay::kWSlot;
                // (scale, bias) of groups A and B; 8-entry block kb takes A if kb < split8
                const uint32_t* sbw = reinterpret_cast<const uint32_t*>(cs + (kGather ? DownLayoutG::kSlab : DownLayout::kCodes));
                // (scale, bias) in fp16 as stored; scale / 16 is exact (or rounds as an fp32 division would)
                const __half2 sha = *reinterpret_cast<const __half2*>(&sbw[32 * qd + lane]);
                const __half2 shb = kGather ? *reinterpret_cast<const __half2*>(&sbw[kDnBand + 32 * qd + lane]) : sha;
                const int split8 =
                    kGather ? rowgather::ksd_split8(reinterpret_cast<const uint32_t*>(cs + DownLayoutG::kDesc)[kk & 3])
                            : 8;
                const __half2 s1a = __low2half2(sha), s1b = __low2half2(shb);
                const __half2 s16a = __hmul2(s1a, k1_16), s16b = __hmul2(s1b, k1_16);
                const __half2 b2a = __high2half2(sha), b2b = __high2half2(shb);
                uint32_t o[32];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t a[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) a[k] = *reinterpret_cast<const uint32_t*>(cs + ldoff[hh][k]);
                    nib_transpose32_in_words(a, trc);   // lane = output 32qd + lane, nibble j of word k = entry 32hh + 8k + j
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const bool useA = 4 * hh + k < split8;
                        const __half2 s1 = useA ? s1a : s1b, s16 = useA ? s16a : s16b, b2 = useA ? b2a : b2b;
                        const uint32_t lo = a[k], hi = a[k] >> 8;
                        // fp16 1024 + c (or 1024 + 16c): nibble pairs (0,4) (1,5) (2,6) (3,7)
                        const uint32_t pr[4] = {(lo & 0x000F000Fu) | 0x64006400u, (lo & 0x00F000F0u) | 0x64006400u,
                                                (hi & 0x000F000Fu) | 0x64006400u, (hi & 0x00F000F0u) | 0x64006400u};
#pragma unroll
                        for (int pp = 0; pp < 4; ++pp) {
                            const __half2 qv = __hsub2(*reinterpret_cast<const __half2*>(&pr[pp]), k1024);
                            const __half2 v = __hfma2(qv, (pp & 1) ? s16 : s1, b2);
                            o[16 * hh + 4 * k + pp] = *reinterpret_cast<const uint32_t*>(&v);
                        }
                    }
                }
                __syncwarp();
                tmem_st32(trow + 32 * (qk % kDnSD), o);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&br.sfull[qk % kDnSD]);   // each lane, after its own stores' wait and fence
                __syncwarp();
                if (lane == 0) mbar_arrive(&br.wempty[s]);
            }
            if (!ok) break;
            q += nk;
        }
    } else if (warp < kEpiWarps) {
        // ---- epilogue: lane = output of the band; router-weighted partial rows of the tile's tokens
        uint32_t nu = 0;
        // the next unit's descriptor is loaded one unit ahead (its loads overlap this unit's work)
        DownUnit dnext;
        if ((int)blockIdx.x < U) dnext = down_unit<kGather>(P, io, nb, words, dense, blockIdx.x);
        for (int u = blockIdx.x; u < U && ok; u += gridDim.x, ++nu) {
            const DownUnit d = dnext;
            if (u + (int)gridDim.x < U) dnext = down_unit<kGather>(P, io, nb, words, dense, u + gridDim.x);
            const int acc = nu & 1;
            const int col = kDnBand * d.ob + 32 * warp + lane;
            float* pbase = io.partial + (d.shared ? (size_t)io.T * K + d.row0 : (size_t)d.row0) * H + col;
            const float* wrow = io.pair_w + d.row0;
            ok = __all_sync(0xffffffffu, wait_full_sleep(br.tfull, 2, nu, kEpilogueSleepNs));
            if (!ok) break;
            tc_fence_after();
            for (int c0 = 0; c0 < d.nt16; c0 += 32) {
                float v[32];
                if (d.nk > 0) {
                    tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(acc * 128 + c0), v);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0.f;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int c = c0 + i;
                    if (c < d.ntok) {
                        const float wgt = d.shared ? 1.f : __ldg(wrow + c);
                        pbase[(size_t)c * H] = wgt * v[i];
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&br.tempty[acc]);   // each lane, after its own loads and fence
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// y[t] = shared partial + sum over slots j of the pair partials, in order; bf16 RNE.
__global__ void __launch_bounds__(256) prefill_combine_kernel(const __grid_constant__ LayerParams P, const PrefillIO io) {
    pdl_wait();
    pdl_trigger();
    const int H = P.hidden, K = P.top_k;
    const size_t n4 = (size_t)io.T * (H / 4);
    for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < n4; q += (size_t)gridDim.x * blockDim.x) {
        const int tok = (int)(q / (H / 4)), c4 = (int)(q % (H / 4));
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        int row[kMaxTopK];
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) row[j] = j < K ? __ldg(io.pos_of + tok * K + j) : 0;
        float4 v[kMaxTopK];
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
            v[j] = j < K ? __ldcs(reinterpret_cast<const float4*>(io.partial + (size_t)row[j] * H) + c4)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        if (P.shared_neurons) a = __ldcs(reinterpret_cast<const float4*>(io.partial + ((size_t)io.T * K + tok) * H) + c4);
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            if (j < K) { a.x += v[j].x; a.y += v[j].y; a.z += v[j].z; a.w += v[j].w; }
        }
        if (io.y_f32) reinterpret_cast<float4*>(io.y_f32)[q] = a;
        const uint32_t lo = (uint32_t)f32_to_bf16_bits(a.x) | ((uint32_t)f32_to_bf16_bits(a.y) << 16);
        const uint32_t hi = (uint32_t)f32_to_bf16_bits(a.z) | ((uint32_t)f32_to_bf16_bits(a.w) << 16);
        reinterpret_cast<uint2*>(io.y_bf16)[q] = make_uint2(lo, hi);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (io.dbg_tiles) {
            io.dbg_tiles[0] = io.meta->skipped;
            io.dbg_tiles[1] = io.meta->total;
        }
        if (io.dbg_work) {
            io.dbg_work[0] = (long long)io.meta->union_rt;
            io.dbg_work[1] = (long long)io.meta->exec_rt;
            io.dbg_work[2] = (long long)io.meta->dense_rt;
        }
    }
}

// Debug counts after a prefill: CTA e < E walks expert e's pair rows of h_r
// (rows off[e] .. off[e+1]), CTA E the shared expert's T rows of h_s; thread
// n ORs neuron n's h > 0 over the rows (fp16 bits; h >= 0).  h is stored
// permuted within blocks of 8 neurons only, so 64-neuron groups keep their
// members.  The totals are added into *live_rows and *live_groups.
__global__ void __launch_bounds__(256) prefill_union_live_kernel(const PrefillMeta* __restrict__ meta,
                                                                 const uint16_t* __restrict__ h_r,
                                                                 const uint16_t* __restrict__ h_s, int T, int E,
                                                                 int NR, int NS, int* live_rows, int* live_groups) {
    __shared__ int grp[kMaxKTiles];
    __shared__ int rows_cnt;
    const int e = blockIdx.x, t = threadIdx.x;
    const bool shared = e == E;
    const int N = shared ? NS : NR;
    const int r0 = shared ? 0 : meta->off[e], r1 = shared ? T : meta->off[e + 1];
    const uint16_t* h = shared ? h_s : h_r;
    for (int g = t; g < N / 64; g += blockDim.x) grp[g] = 0;
    if (t == 0) rows_cnt = 0;
    __syncthreads();
    int cnt = 0;
    for (int n = t; n < N; n += blockDim.x) {
        bool live = false;
        for (int r = r0; r < r1 && !live; ++r) live = (h[(size_t)r * N + n] & 0x7fffu) != 0u;
        if (live) {
            ++cnt;
            grp[n >> 6] = 1;
        }
    }
    atomicAdd(&rows_cnt, cnt);
    __syncthreads();
    if (t == 0) {
        int ng = 0;
        for (int g = 0; g < N / 64; ++g) ng += grp[g];
        if (live_rows) atomicAdd(live_rows, rows_cnt);
        if (live_groups) atomicAdd(live_groups, ng);
    }
}

// Debug outputs after a prefill (launched only when asked for).  CTA t: token
// t's live masks, one 64-bit word per (slot, 64-neuron group) in the decode
// layout (shared groups first, then slot j's groups), from the kernel's fp16
// h, which keeps each group of 8 neurons in the order n0 n4 n1 n5 n2 n6 n3 n7
// (stored position p holds neuron kPos8[p]).  CTA 0 also copies each token
// tile's multiplied 64-neuron tiles (the down product's own rule: the live
// flags of the up epilogue, or every tile with the dense flag).
__global__ void __launch_bounds__(256) prefill_live_debug_kernel(const __grid_constant__ LayerParams P,
                                                                 const PrefillIO io) {
    pdl_wait();
    pdl_trigger();
    const int tok = blockIdx.x, K = P.top_k;
    const int NGs = P.shared_neurons / 64, NGr = P.routed_neurons / 64, Ut = NGs + K * NGr;
    if (io.dbg_live) {
        for (int u = threadIdx.x; u < Ut; u += blockDim.x) {
            const uint16_t* row;
            int gi;
            if (u < NGs) {
                row = io.h_s + (size_t)tok * P.shared_neurons;
                gi = u;
            } else {
                const int j = (u - NGs) / NGr;
                gi = (u - NGs) % NGr;
                row = io.h_r + (size_t)__ldcg(io.pos_of + (size_t)tok * K + j) * P.routed_neurons;
            }
            const uint4* p = reinterpret_cast<const uint4*>(row + 64 * gi);
            uint64_t m = 0;
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const uint4 v = __ldcg(p + b);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    constexpr int kPos8[8] = {0, 4, 1, 5, 2, 6, 3, 7};
                    if (w[q] & 0x7fffu) m |= 1ull << (8 * b + kPos8[2 * q]);
                    if ((w[q] >> 16) & 0x7fffu) m |= 1ull << (8 * b + kPos8[2 * q + 1]);
                }
            }
            io.dbg_live[(size_t)tok * Ut + u] = m;
        }
    }
    if (io.dbg_tile_live && tok == 0) {
        const int n_tiles = __ldcg(&io.meta->n_tiles);
        const int words = (max(P.routed_neurons, P.shared_neurons) / 64 + 31) / 32;
        const bool dense = (io.flags & HS_FORCE_DENSE) != 0;
        for (int i = threadIdx.x; i < n_tiles; i += blockDim.x) {
            const TileInfo ti = io.tiles[i];
            const int NK = (ti.e == P.n_routed ? P.shared_neurons : P.routed_neurons) / 64;
            const uint64_t all = NK == 64 ? ~0ull : ((1ull << NK) - 1ull);
            const uint32_t* f = io.flag_r + (size_t)i * words;
            io.dbg_tile_live[i] =
                dense ? all : ((uint64_t)__ldcg(f) | (words > 1 ? (uint64_t)__ldcg(f + 1) << 32 : 0ull)) & all;
        }
    }
}

// ------------------------------------------------------------ row gather
// The page's prefill gathers, per token tile, the rows live for any of its
// tokens into a dense product ("What we do instead").  Here the up epilogue
// leaves each tile's union-live mask (one bit per neuron); this kernel plans
// the tile's down product and copies the tile's h into entry order, and the
// down product then copies the entries' weight rows.
//
// CTA (tile, part): every CTA of a tile plans it in shared memory
// (rowgather::plan_tile: each group's live neurons padded to 8 entries, at
// most two scale groups per 64-entry k-step; the identity plan if packing
// would take more k-steps than groups) and lists the entries; part 0 also
// publishes the plan (k-step count, descriptors, entry list) for the down
// product.  Then each CTA copies rows part * kGatherRows + ... of the tile's
// h into H_c: a pass reads kGatherRows rows whole (16-byte loads) into shared
// memory, and thread task (row, 8-entry block b) gathers the block's 8 values
// (zero at padding entries) into one 16-byte word at columns 8b .. 8b + 7, in
// the stored order of h.  H_c columns beyond the plan are never read.
constexpr int kGatherRows = 4;   // rows of h staged per pass
constexpr int kGatherParts = 8;  // CTAs per tile
__global__ void __launch_bounds__(256) prefill_gather_kernel(const __grid_constant__ LayerParams P, const PrefillIO io) {
    __shared__ __align__(16) uint16_t list_s[64 * kMaxKTiles];
    __shared__ __align__(16) uint16_t row_s[kGatherRows][64 * kMaxKTiles];
    __shared__ uint64_t msk[kMaxKTiles];
    __shared__ uint32_t ksd_s[kMaxKTiles];
    __shared__ int ofs[kMaxKTiles];
    __shared__ int nks_s, ident_s;
    pdl_wait();
    pdl_trigger();
    const int tile = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    if (tile >= __ldcg(&io.meta->n_tiles)) return;
    const TileInfo ti = io.tiles[tile];
    const bool shared = ti.e == P.n_routed;
    const int N = shared ? P.shared_neurons : P.routed_neurons, NG = N / 64;
    // ---- plan (thread 0), while warps 1-7 stage the first pass of rows of h
    const uint32_t* um = io.umask + (size_t)tile * kUWords;
    const uint16_t* H = shared ? io.h_s : io.h_r;
    uint16_t* Hc = shared ? io.hc_s : io.hc_r;
    const int c16 = N / 8;   // 16-byte chunks per row of h
    auto load_rows = [&](int r0, int nr, int first, int step) {
        for (int q = first; q < nr * c16; q += step) {
            const int rr = q / c16, c = q % c16;
            reinterpret_cast<uint4*>(row_s[rr])[c] =
                __ldcg(reinterpret_cast<const uint4*>(H + (size_t)(ti.row0 + r0 + rr) * N) + c);
        }
    };
    const int r_first = blockIdx.y * kGatherRows;
    if (warp == 0) {
        for (int g = lane; g < NG; g += 32)
            msk[g] = (uint64_t)__ldcg(um + 2 * g) | ((uint64_t)__ldcg(um + 2 * g + 1) << 32);
        __syncwarp();
        if (lane == 0) {
            int n = rowgather::plan_tile(msk, NG, ksd_s, ofs);
            ident_s = n < 0;
            if (n < 0) n = rowgather::plan_identity(NG, ksd_s, ofs);
            nks_s = n;
        }
    } else if (r_first < ti.ntok) {
        load_rows(r_first, min(kGatherRows, ti.ntok - r_first), t - 32, blockDim.x - 32);
    }
    __syncthreads();
    const int nks = nks_s, nb = 8 * nks;
    const bool ident = ident_s != 0;
    for (int e = t; e < 64 * nks; e += blockDim.x) list_s[e] = rowgather::kPad;
    __syncthreads();
    // warp per group: its live neurons, ascending, from the group's first entry
    for (int g = warp; g < NG; g += blockDim.x / 32) {
        if (ofs[g] < 0) continue;
        const uint64_t m = ident ? ~0ull : msk[g];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const bool live = (m >> (32 * half + lane)) & 1ull;
            const unsigned below = (unsigned)(m >> (32 * half)) & ((1u << lane) - 1u);
            const int rank = (half ? __popc((unsigned)m) : 0) + __popc(below);
            if (live) list_s[ofs[g] + rank] = (uint16_t)(64 * g + 32 * half + lane);
        }
    }
    __syncthreads();
    if (blockIdx.y == 0) {
        uint4* L = reinterpret_cast<uint4*>(io.glist + (size_t)tile * 64 * kMaxKTiles);
        for (int b = t; b < nb; b += blockDim.x) L[b] = reinterpret_cast<const uint4*>(list_s)[b];
        for (int k = t; k < nks; k += blockDim.x) io.ksd[(size_t)tile * kMaxKTiles + k] = ksd_s[k];
        if (t == 0) io.nks[tile] = nks;
    }
    // ---- H_c rows of this part (the first pass's rows are staged)
    for (int r0 = r_first; r0 < ti.ntok; r0 += gridDim.y * kGatherRows) {
        const int nr = min(kGatherRows, ti.ntok - r0);
        if (r0 != r_first) {
            __syncthreads();   // the previous pass has read its rows
            load_rows(r0, nr, t, blockDim.x);
            __syncthreads();
        }
        for (int q = t; q < nr * nb; q += blockDim.x) {
            const int rr = q / nb, b = q % nb;
            const uint4 ids = reinterpret_cast<const uint4*>(list_s)[b];
            const uint32_t w[4] = {ids.x, ids.y, ids.z, ids.w};
            uint16_t v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t n = (w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
                v[rowgather::stored_pos(i)] = n == rowgather::kPad ? (uint16_t)0 : row_s[rr][rowgather::stored_pos((int)n)];
            }
            uint4 o;
            o.x = (uint32_t)v[0] | ((uint32_t)v[1] << 16);
            o.y = (uint32_t)v[2] | ((uint32_t)v[3] << 16);
            o.z = (uint32_t)v[4] | ((uint32_t)v[5] << 16);
            o.w = (uint32_t)v[6] | ((uint32_t)v[7] << 16);
            *reinterpret_cast<uint4*>(Hc + (size_t)(ti.row0 + r0 + rr) * N + 8 * b) = o;
        }
    }
}

}  // namespace hs

// ===================================================================== host
using namespace hs_host;

unsigned hs_prefill_take_status() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, hs::g_status, sizeof(v)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(hs::g_status, &zero, sizeof(zero));
    return v;
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

bool make_map(EncodeTiledFn enc, CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
              uint64_t rows, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {pitch_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct PrefillLayout {
    size_t meta, blk_cnt, sb_cnt, tiles, idx, w, pair_tok, pos_of, pair_w, xg, h_r, h_s, flags, partial, umask, nks, ksd, glist,
        hc_r, hc_s, total;
    int max_tiles;
};

PrefillLayout prefill_layout(const hs_moe_layer* L, int T) {
    const int K = L->top_k, E = L->n_routed, NR = L->routed[0].neurons, H = L->hidden;
    const int NS = L->shared ? L->shared->neurons : 0;
    PrefillLayout l{};
    l.max_tiles = E + (T * K + hs::kNt - 1) / hs::kNt + (T + hs::kNt - 1) / hs::kNt + 1;
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o += round_up(bytes, 1024); return at; };
    const size_t rows = (size_t)T * K + (NS ? T : 0);
    l.meta = take(sizeof(hs::PrefillMeta));
    l.blk_cnt = take((size_t)((T + hs::kTokBlk - 1) / hs::kTokBlk) * E * 4);
    l.sb_cnt = take((size_t)((T + hs::kTokBlk * hs::kSuperBlk - 1) / (hs::kTokBlk * hs::kSuperBlk)) * E * 4);
    l.tiles = take((size_t)l.max_tiles * sizeof(hs::TileInfo));
    l.idx = take((size_t)T * K * 4);
    l.w = take((size_t)T * K * 4);
    l.pair_tok = take((size_t)T * K * 4);
    l.pos_of = take((size_t)T * K * 4);
    l.pair_w = take((size_t)T * K * 4);
    l.xg = take(rows * H * 2);
    l.h_r = take((size_t)T * K * NR * 2);
    l.h_s = take((size_t)(NS ? T : 1) * (NS ? NS : 64) * 2);
    l.flags = take((size_t)l.max_tiles * ((std::max(NR, NS) / 64 + 31) / 32) * 4);
    l.partial = take(rows * H * 4);
    // row gather
    l.umask = take((size_t)l.max_tiles * hs::kUWords * 4);
    l.nks = take((size_t)l.max_tiles * 4);
    l.ksd = take((size_t)l.max_tiles * hs::kMaxKTiles * 4);
    l.glist = take((size_t)l.max_tiles * 64 * hs::kMaxKTiles * 2);
    l.hc_r = take((size_t)T * K * NR * 2);
    l.hc_s = take((size_t)(NS ? T : 1) * (NS ? NS : 64) * 2);
    l.total = o;
    return l;
}

int prefill_shape_ok(const hs_moe_layer* L, int T) {
    if (T < 1 || T > hs::kMaxTokens) return HS_ERR_UNSUPPORTED_SHAPE;
    if (L->hidden % 128) return HS_ERR_UNSUPPORTED_SHAPE;
    if (L->routed[0].neurons % 64) return HS_ERR_UNSUPPORTED_SHAPE;
    if (L->shared && L->shared->neurons % 64) return HS_ERR_UNSUPPORTED_SHAPE;
    if (L->routed[0].neurons / 64 > hs::kMaxKTiles) return HS_ERR_UNSUPPORTED_SHAPE;
    if (L->shared && L->shared->neurons / 64 > hs::kMaxKTiles) return HS_ERR_UNSUPPORTED_SHAPE;
    // one tensor map spans the codes of all routed experts: they must be stacked back to back
    hs::LayerParams P;
    fill_layer_params(L, P);
    const long long rowbytes = (long long)L->routed[0].neurons * (L->hidden / 2);
    if (!P.uniform) return HS_ERR_UNSUPPORTED_SHAPE;
    if (L->n_routed > 1 && (P.stride[0] != rowbytes || P.stride[2] != rowbytes)) return HS_ERR_UNSUPPORTED_SHAPE;
    return HS_OK;
}
}  // namespace

int hs_prefill_layer_ok(const hs_moe_layer* L, int tokens) {
    const int st = check_layer(L);
    return st != HS_OK ? st : prefill_shape_ok(L, tokens);
}

int hs_prefill_union_live(const hs_moe_layer* L, int tokens, void* ws, int* live_rows, int* live_groups,
                          cudaStream_t s) {
    if (!live_rows && !live_groups) return HS_OK;
    const PrefillLayout l = prefill_layout(L, tokens);
    char* w = static_cast<char*>(ws);
    if (live_rows && cudaMemsetAsync(live_rows, 0, sizeof(int), s) != cudaSuccess) return HS_ERR_CUDA;
    if (live_groups && cudaMemsetAsync(live_groups, 0, sizeof(int), s) != cudaSuccess) return HS_ERR_CUDA;
    const int E = L->n_routed, NS = L->shared ? L->shared->neurons : 0;
    hs::prefill_union_live_kernel<<<E + (NS ? 1 : 0), 256, 0, s>>>(
        reinterpret_cast<const hs::PrefillMeta*>(w + l.meta), reinterpret_cast<const uint16_t*>(w + l.h_r),
        reinterpret_cast<const uint16_t*>(w + l.h_s), tokens, E, L->routed[0].neurons, NS, live_rows, live_groups);
    return launch_err();
}

extern "C" size_t hs_moe_prefill_workspace_size(const hs_moe_layer* L, int tokens) {
    if (check_layer(L) != HS_OK || prefill_shape_ok(L, tokens) != HS_OK) return 0;
    return prefill_layout(L, tokens).total;
}

extern "C" int hs_moe_prefill(const hs_moe_layer* L, const uint16_t* x, const float* logits, int tokens,
                              uint16_t* y_bf16, float* y_f32, unsigned flags, const hs_prefill_debug* dbg, void* ws,
                              size_t ws_bytes, hs_stream_t stream) {
    int st = check_layer(L);
    if (st != HS_OK) return st;
    if (!x || !logits || !y_bf16) return HS_ERR_INVALID_ARG;
    if (tokens < 1) return HS_ERR_INVALID_ARG;
    if (flags & HS_DOWN_ROW_SCALES) return HS_ERR_INVALID_ARG;  // group slabs only
    st = prefill_shape_ok(L, tokens);
    if (st != HS_OK) return st;
    if (!al16(x) || !al4(logits) || !al16(y_bf16) || (y_f32 && !al16(y_f32)) || !al16(ws)) return HS_ERR_MISALIGNED;
    const PrefillLayout l = prefill_layout(L, tokens);
    if (!ws || ws_bytes < l.total) return HS_ERR_WORKSPACE;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return HS_ERR_CUDA;

    char* w = static_cast<char*>(ws);
    hs::LayerParams P;
    fill_layer_params(L, P);
    const int T = tokens, K = L->top_k, E = L->n_routed, NR = L->routed[0].neurons, H = L->hidden;
    const int NS = L->shared ? L->shared->neurons : 0;
    hs::PrefillIO io{};
    io.x = x;
    io.logits = logits;
    io.T = T;
    io.flags = flags;
    io.meta = reinterpret_cast<hs::PrefillMeta*>(w + l.meta);
    io.blk_cnt = reinterpret_cast<int*>(w + l.blk_cnt);
    io.sb_cnt = reinterpret_cast<int*>(w + l.sb_cnt);
    io.tiles = reinterpret_cast<hs::TileInfo*>(w + l.tiles);
    io.idx = reinterpret_cast<int*>(w + l.idx);
    io.w = reinterpret_cast<float*>(w + l.w);
    io.pair_tok = reinterpret_cast<int*>(w + l.pair_tok);
    io.pos_of = reinterpret_cast<int*>(w + l.pos_of);
    io.pair_w = reinterpret_cast<float*>(w + l.pair_w);
    io.xg = reinterpret_cast<uint16_t*>(w + l.xg);
    io.h_r = reinterpret_cast<uint16_t*>(w + l.h_r);
    io.h_s = reinterpret_cast<uint16_t*>(w + l.h_s);
    io.flag_r = reinterpret_cast<uint32_t*>(w + l.flags);
    io.partial = reinterpret_cast<float*>(w + l.partial);
    io.y_bf16 = y_bf16;
    io.y_f32 = y_f32;
    io.dbg_idx = dbg ? dbg->topk_idx : nullptr;
    io.dbg_w = dbg ? dbg->topk_w : nullptr;
    io.dbg_tiles = dbg ? dbg->tiles : nullptr;
    io.dbg_work = dbg ? dbg->work : nullptr;
    io.dbg_live = dbg ? dbg->live_mask : nullptr;
    io.dbg_tile_live = dbg ? dbg->tile_live : nullptr;
    if (((uintptr_t)io.dbg_live & 7u) || ((uintptr_t)io.dbg_tile_live & 7u)) return HS_ERR_MISALIGNED;
    io.max_tiles = l.max_tiles;
    const bool gather = (flags & HS_PREFILL_ROW_GATHER) && !(flags & HS_FORCE_DENSE);
    if (gather) {
        io.umask = reinterpret_cast<uint32_t*>(w + l.umask);
        io.nks = reinterpret_cast<int*>(w + l.nks);
        io.ksd = reinterpret_cast<uint32_t*>(w + l.ksd);
        io.glist = reinterpret_cast<uint16_t*>(w + l.glist);
        io.hc_r = reinterpret_cast<uint16_t*>(w + l.hc_r);
        io.hc_s = reinterpret_cast<uint16_t*>(w + l.hc_s);
    }

    // tensor maps
    hs::TMaps tm;
    memset(&tm, 0, sizeof(tm));
    const uint64_t rows_x = (uint64_t)T * K + (NS ? T : 0);
    bool okm = true;
    okm &= make_map(enc, &tm.up_codes_r, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->routed[0].up.codes, H / 2, (uint64_t)E * NR,
                    H / 2, hs::kUpK / 2, 128, CU_TENSOR_MAP_SWIZZLE_64B);
    okm &= make_map(enc, &tm.dn_codes_r, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->routed[0].down_nm.codes, H / 2,
                    (uint64_t)E * NR, H / 2, hs::kDnBand / 2, 64, CU_TENSOR_MAP_SWIZZLE_64B);
    if (NS) {
        okm &= make_map(enc, &tm.up_codes_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->shared->up.codes, H / 2, NS, H / 2,
                        hs::kUpK / 2, 128, CU_TENSOR_MAP_SWIZZLE_64B);
        okm &= make_map(enc, &tm.dn_codes_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->shared->down_nm.codes, H / 2, NS, H / 2,
                        hs::kDnBand / 2, 64, CU_TENSOR_MAP_SWIZZLE_64B);
    }
    for (int b = 0; b < 8; ++b)
        okm &= make_map(enc, &tm.xg[b], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, io.xg, H, rows_x, (uint64_t)H * 2, 64,
                        16u * (b + 1), CU_TENSOR_MAP_SWIZZLE_128B);
    for (int b = 0; b < 8; ++b) {
        const uint32_t br = 16u * (b + 1);
        okm &= make_map(enc, &tm.hr[b], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, io.h_r, NR, (uint64_t)T * K, (uint64_t)NR * 2,
                        64, br, CU_TENSOR_MAP_SWIZZLE_128B);
        if (NS)
            okm &= make_map(enc, &tm.hsh[b], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, io.h_s, NS, T, (uint64_t)NS * 2, 64, br,
                            CU_TENSOR_MAP_SWIZZLE_128B);
        if (gather) {
            okm &= make_map(enc, &tm.hcr[b], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, io.hc_r, NR, (uint64_t)T * K,
                            (uint64_t)NR * 2, 64, br, CU_TENSOR_MAP_SWIZZLE_128B);
            if (NS)
                okm &= make_map(enc, &tm.hcs[b], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, io.hc_s, NS, T, (uint64_t)NS * 2, 64,
                                br, CU_TENSOR_MAP_SWIZZLE_128B);
        }
    }
    if (!okm) return HS_ERR_CUDA;

    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return HS_ERR_CUDA;
    const int up_smem = hs::UpLayout::total(H);
    const int dn_smem = gather ? hs::DownLayoutG::kTotal : hs::DownLayout::kTotal;
    const void* dn_kernel = gather ? (const void*)hs::prefill_down_kernel<true> : (const void*)hs::prefill_down_kernel<false>;
    if (set_smem_attr((const void*)hs::prefill_up_kernel, up_smem) != HS_OK) return HS_ERR_CUDA;
    if (set_smem_attr(dn_kernel, dn_smem) != HS_OK) return HS_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the meta block and the block and superblock counts are contiguous: one memset clears them
    if (cudaMemsetAsync(io.meta, 0, l.tiles - l.meta, s) != cudaSuccess) return HS_ERR_CUDA;
    // the first kernel follows the memset with ordinary stream ordering
    hs::prefill_route_kernel<<<dim3((T + 7) / 8), dim3(256), 0, s>>>(P, io);
    if (cudaGetLastError() != cudaSuccess) return HS_ERR_CUDA;
    if (launch_pdl(hs::prefill_tiles_kernel, dim3(1), dim3(256), 0, s, P, io) != cudaSuccess) return HS_ERR_CUDA;
    if (launch_pdl(hs::prefill_list_kernel, dim3((T + hs::kTokBlk - 1) / hs::kTokBlk), dim3(hs::kListThreads), 0, s, P,
                   io) != cudaSuccess)
        return HS_ERR_CUDA;
    if (launch_pdl(hs::prefill_up_kernel, dim3(sms), dim3(hs::kGemmThreads), up_smem, s, P, io, tm) != cudaSuccess)
        return HS_ERR_CUDA;
    if (gather) {
        if (launch_pdl(hs::prefill_gather_kernel, dim3(l.max_tiles, hs::kGatherParts), dim3(256), 0, s, P, io) !=
            cudaSuccess)
            return HS_ERR_CUDA;
        if (launch_pdl(hs::prefill_down_kernel<true>, dim3(sms), dim3(hs::kGemmThreads), dn_smem, s, P, io, tm) !=
            cudaSuccess)
            return HS_ERR_CUDA;
    } else if (launch_pdl(hs::prefill_down_kernel<false>, dim3(sms), dim3(hs::kGemmThreads), dn_smem, s, P, io, tm) !=
               cudaSuccess) {
        return HS_ERR_CUDA;
    }
    if (launch_pdl(hs::prefill_combine_kernel, dim3(4 * sms), dim3(256), 0, s, P, io) != cudaSuccess)
        return HS_ERR_CUDA;
    if ((io.dbg_live || io.dbg_tile_live) &&
        launch_pdl(hs::prefill_live_debug_kernel, dim3(T), dim3(256), 0, s, P, io) != cudaSuccess)
        return HS_ERR_CUDA;
    (void)NR;
    return launch_err();
}
