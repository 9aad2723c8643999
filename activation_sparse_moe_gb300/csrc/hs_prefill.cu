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

#include "hs_host.h"
#include "hs_tc.cuh"

namespace hs {

constexpr int kNt = 256;          // max tokens per tile (MMA N)
constexpr int kStages = 3;        // up / down pipeline depth
constexpr int kMaxTokens = 4096;
constexpr int kMaxKTiles = 1024;  // 64-neuron tiles per expert (neurons <= 65536)

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
    int max_tiles;
};

// Inside each 64-block the gathered x holds, for every group of 8 elements
// e0..e7 (one 32-bit word of codes), the order e0 e4 e1 e5 e2 e6 e3 e7: the
// order in which the dequantiser emits nibble pairs.  Both operands of the up
// product use it, so the product is unchanged.

// ------------------------------------------------------------ routing
__global__ void __launch_bounds__(256) prefill_route_kernel(const __grid_constant__ LayerParams P, const PrefillIO io) {
    pdl_wait();
    pdl_trigger();
    const int tok = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (tok < io.T) {
        const int K = P.top_k;
        warp_topk_softmax(io.logits + (size_t)tok * P.n_routed, P.n_routed, K, io.idx + (size_t)tok * K,
                          io.w + (size_t)tok * K);
        __syncwarp();
        if ((threadIdx.x & 31) < K && io.dbg_idx) {
            const int j = threadIdx.x & 31;
            io.dbg_idx[(size_t)tok * K + j] = io.idx[(size_t)tok * K + j];
            io.dbg_w[(size_t)tok * K + j] = io.w[(size_t)tok * K + j];
        }
    }
}

// CTA e counts the (token, slot) pairs routed to expert e.
__global__ void __launch_bounds__(256) prefill_count_kernel(const __grid_constant__ LayerParams P, const PrefillIO io) {
    __shared__ int part[8];
    pdl_wait();
    pdl_trigger();
    const int e = blockIdx.x, n = io.T * P.top_k;
    int c = 0;
    for (int p = threadIdx.x; p < n; p += blockDim.x) c += (io.idx[p] == e);
#pragma unroll
    for (int off = 16; off; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        int s = 0;
        for (int i = 0; i < 8; ++i) s += part[i];
        io.meta->cnt[e] = s;
    }
}

// One CTA: pair offsets, token tiles, work-unit counts, cleared flags.
__global__ void __launch_bounds__(256) prefill_tiles_kernel(const __grid_constant__ LayerParams P, const PrefillIO io) {
    pdl_wait();
    pdl_trigger();
    PrefillMeta* m = io.meta;
    const int E = P.n_routed;
    if (threadIdx.x == 0) {
        int acc = 0, nt = 0;
        for (int e = 0; e < E; ++e) {
            m->off[e] = acc;
            m->tile_off[e] = nt;
            const int c = m->cnt[e];
            for (int r = 0; r < c; r += kNt) {
                io.tiles[nt] = TileInfo{e, acc + r, min(kNt, c - r), 0};
                ++nt;
            }
            acc += c;
        }
        m->off[E] = acc;
        m->tile_off[E] = nt;
        if (P.shared_neurons) {
            for (int r = 0; r < io.T; r += kNt) {
                io.tiles[nt] = TileInfo{E, r, min(kNt, io.T - r), 0};
                ++nt;
            }
        }
        m->tile_off[E + 1] = nt;
        m->n_tiles = nt;
        const int mr = (P.routed_neurons + 127) / 128, ms = (P.shared_neurons + 127) / 128;
        m->up_units = (m->tile_off[E]) * mr + (nt - m->tile_off[E]) * ms;
        m->dn_units = nt * (P.hidden / 128);
        m->skipped = 0;
        m->total = 0;
        m->union_rt = 0;
        m->exec_rt = 0;
        m->dense_rt = 0;
    }
    // live flags: one word per (tile, 32 k-tiles); up to max_tiles * words
    const int words = io.max_tiles * ((max(P.routed_neurons, P.shared_neurons) / 64 + 31) / 32);
    for (int i = threadIdx.x; i < words; i += blockDim.x) io.flag_r[i] = 0u;
}

// CTA e lists its pairs in token order (ballot compaction over the token-major
// pair order) and records each pair's grouped position.
__global__ void __launch_bounds__(256) prefill_list_kernel(const __grid_constant__ LayerParams P, const PrefillIO io) {
    __shared__ int wsum[8];
    __shared__ int base_s;
    pdl_wait();
    pdl_trigger();
    const int e = blockIdx.x, K = P.top_k, n = io.T * K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) base_s = io.meta->off[e];
    __syncthreads();
    for (int p0 = 0; p0 < n; p0 += blockDim.x) {
        const int p = p0 + threadIdx.x;
        const bool hit = p < n && io.idx[p] == e;
        const unsigned b = __ballot_sync(0xffffffffu, hit);
        if (lane == 0) wsum[warp] = __popc(b);
        __syncthreads();
        int before = 0;
        for (int i = 0; i < warp; ++i) before += wsum[i];
        if (hit) {
            const int pos = base_s + before + __popc(b & ((1u << lane) - 1u));
            io.pair_tok[pos] = p / K;
            io.pair_w[pos] = io.w[p];
            io.pos_of[p] = pos;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int tot = 0;
            for (int i = 0; i < 8; ++i) tot += wsum[i];
            base_s += tot;
        }
        __syncthreads();
    }
}

// Gathered fp16 rows: row r < T*K is pair r (its token's x), row T*K + t is token t.
__global__ void __launch_bounds__(256) prefill_gather_kernel(const __grid_constant__ LayerParams P, const PrefillIO io) {
    pdl_wait();
    pdl_trigger();
    const int H = P.hidden, npairs = io.T * P.top_k;
    const int rows = npairs + (P.shared_neurons ? io.T : 0);
    const int per_row = H / 8;  // 8 elements per thread-chunk
    for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < (size_t)rows * per_row;
         q += (size_t)gridDim.x * blockDim.x) {
        const int r = (int)(q / per_row), c8 = (int)(q % per_row);
        const int tok = r < npairs ? io.pair_tok[r] : r - npairs;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(io.x + (size_t)tok * H) + c8);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        __half hv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            hv[2 * i] = __float2half_rn(__uint_as_float(wv[i] << 16));
            hv[2 * i + 1] = __float2half_rn(__uint_as_float(wv[i] & 0xffff0000u));
        }
        // elements 8*c8 .. 8*c8+7 are one code word: stored in the dequantiser's order
        const __half2 p0 = __halves2half2(hv[0], hv[4]), p1 = __halves2half2(hv[1], hv[5]);
        const __half2 p2 = __halves2half2(hv[2], hv[6]), p3 = __halves2half2(hv[3], hv[7]);
        *reinterpret_cast<uint4*>(io.xg + (size_t)r * H + 8 * c8) =
            make_uint4(*reinterpret_cast<const uint32_t*>(&p0), *reinterpret_cast<const uint32_t*>(&p1),
                       *reinterpret_cast<const uint32_t*>(&p2), *reinterpret_cast<const uint32_t*>(&p3));
    }
}

// ------------------------------------------------------------ shared memory
struct UpSmem {
    static constexpr int kA = 128 * 128;          // fp16 A tile 128 x 64
    static constexpr int kB = kNt * 128;          // fp16 B tile up to 256 x 64
    static constexpr int kC = 128 * 32;           // raw codes 128 rows x 32 B
    static constexpr int kStage = kA + kB + kC;   // multiple of 1024
    __host__ __device__ static int sb(int H) { return 128 * (H / 64) * 4; }
    __host__ __device__ static int total(int H) { return 1024 + kStages * kStage + sb(H) + 128 * 4 + 256; }
};

struct DownSmem {
    static constexpr int kA = 128 * 128;          // fp16 A tile 128 outputs x 64 neurons
    static constexpr int kB = kNt * 128;          // H tile up to 256 tokens x 64 neurons
    static constexpr int kC = 64 * 64;            // codes 64 neurons x 64 B (128 outputs)
    static constexpr int kSB = 128 * 4;           // slab slice
    static constexpr int kStage = kA + kB + kC + 1024;  // keep 1024 alignment
    __host__ __device__ static int total() { return 1024 + kStages * kStage + 64 + 4 * kMaxKTiles; }
};

struct TMaps {
    CUtensorMap up_codes_r, up_codes_s;      // [rows][H/2] bytes, box 32 x 128
    CUtensorMap dn_codes_r, dn_codes_s;      // [rows][H/2] bytes, box 64 x 64
    CUtensorMap xg[3];                       // fp16 [rows][H], box 64 x {64,128,256}, 128B swizzle
    CUtensorMap hr[3], hsh[3];               // fp16 H, box 64 x {64,128,256}
};

__device__ __forceinline__ int box_index(int ntok) { return ntok <= 64 ? 0 : (ntok <= 128 ? 1 : 2); }

// ------------------------------------------------------------ pipeline
// Stage ring shared by the two GEMM kernels.  Step q of the CTA (counted
// across its units) uses stage q % kStages; full[s] completes when the
// step's operands have landed, done[s] when the MMAs that read them have
// completed.  Thread 0 issues the loads; every thread dequantises; thread 0
// issues the MMAs.
struct Ring {
    uint64_t* full;
    uint64_t* done;
    uint32_t issued = 0;     // steps whose loads were issued (thread 0)
    uint32_t committed = 0;  // steps whose MMAs were committed (thread 0)
    // Thread 0: waits until the stage of step `issued` is free.  False on timeout.
    __device__ bool acquire() {
        const uint32_t q = issued;
        return q < kStages || mbar_wait(&done[q % kStages], ((q / kStages) - 1) & 1);
    }
    // Thread 0, on the way out: waits (bounded) for the loads still in flight
    // and for the last committed MMAs, so that no copy lands and no MMA reads
    // after the CTA leaves.
    __device__ void drain() {
        const uint32_t lo = issued > (uint32_t)kStages ? issued - kStages : 0;
        for (uint32_t q = lo; q < issued; ++q) mbar_wait(&full[q % kStages], (q / kStages) & 1);
        if (committed) mbar_wait(&done[(committed - 1) % kStages], ((committed - 1) / kStages) & 1);
    }
};

// ------------------------------------------------------------ up GEMM
__global__ void __launch_bounds__(256, 1)
prefill_up_kernel(const __grid_constant__ LayerParams P, const PrefillIO io, const __grid_constant__ TMaps tm) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int H = P.hidden, G = H / 64;
    uint8_t* stage0 = smem;
    uint32_t* sb_s = reinterpret_cast<uint32_t*>(smem + kStages * UpSmem::kStage);
    float* off_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(sb_s) + UpSmem::sb(H));
    uint64_t* bars = reinterpret_cast<uint64_t*>(off_s + 128);   // full[kStages], done[kStages], sb
    uint32_t* tmem_s = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 1);
    uint64_t* sbbar = bars + 2 * kStages;
    Ring ring;
    ring.full = bars;
    ring.done = bars + kStages;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    if (t == 0) {
        for (int i = 0; i < 2 * kStages + 1; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_s, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_s;
    pdl_wait();
    pdl_trigger();
    const PrefillMeta* m = io.meta;
    const int E = P.n_routed, NR = P.routed_neurons, NS = P.shared_neurons;
    const int ntr = m->tile_off[E];
    const int mr = (NR + 127) / 128, ms = (NS + 127) / 128;
    const int U = m->up_units;
    const int words = (max(NR, NS) / 64 + 31) / 32;
    uint32_t it = 0;  // steps consumed
    uint32_t sbphase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
        // ---- unit: token tile x 128-neuron block
        int tile, mb;
        if (u < ntr * mr) { tile = u / mr; mb = u % mr; }
        else { tile = ntr + (u - ntr * mr) / ms; mb = (u - ntr * mr) % ms; }
        const TileInfo ti = io.tiles[tile];
        const bool shared = ti.e == E;
        const int N = shared ? NS : NR;
        const ExpertPtrs ep = shared ? P.shared : routed_ptrs(P, ti.e);
        const int row0 = 128 * mb;
        const int rows = min(128, N - row0);
        const int nt16 = (ti.ntok + 15) & ~15;
        const int bi = box_index(ti.ntok);
        const uint32_t bbytes = (uint32_t)(64 << bi) * 128;
        const CUtensorMap* cmap = shared ? &tm.up_codes_s : &tm.up_codes_r;
        const CUtensorMap* xmap = &tm.xg[bi];
        const int cy = shared ? row0 : ti.e * NR + row0;
        const int xrow = shared ? io.T * P.top_k + ti.row0 : ti.row0;
        auto issue = [&](int k) -> bool {
            if (!ring.acquire()) return false;
            const int s = ring.issued % kStages;
            uint8_t* st = stage0 + s * UpSmem::kStage;
            mbar_arrive_expect_tx(&ring.full[s], (uint32_t)UpSmem::kC + bbytes);
            tma_load_2d(st + UpSmem::kA + UpSmem::kB, cmap, 32 * k, cy, &ring.full[s]);
            tma_load_2d(st + UpSmem::kA, xmap, 64 * k, xrow, &ring.full[s]);
            ++ring.issued;
            return true;
        };
        if (t == 0) {
            // scales and biases of the block's rows (the previous unit is done with them)
            mbar_arrive_expect_tx(sbbar, (uint32_t)rows * G * 4);
            bulk_g2s(sb_s, ep.up_sb + (size_t)row0 * G, (uint32_t)rows * G * 4, sbbar, policy_evict_first());
            for (int k = 0; k < kStages - 1 && k < G && ok; ++k) ok = issue(k);
        }
        if (t < 128) off_s[t] = (t < rows && ep.up_off) ? ep.up_off[row0 + t] : 0.f;
        ok = ok && mbar_wait(sbbar, sbphase);
        sbphase ^= 1u;
        ok = __syncthreads_and(ok);
        const uint32_t idesc = umma_idesc_f16_f32(128, nt16);
        for (int k = 0; k < G && ok; ++k) {
            const uint32_t q = it + k;
            const int s = q % kStages;
            uint8_t* st = stage0 + s * UpSmem::kStage;
            if (t == 0 && k + kStages - 1 < G) ok = issue(k + kStages - 1);
            ok = ok && mbar_wait(&ring.full[s], (q / kStages) & 1);
            if (ok) {
                // thread (row r, half hf): 32 codes -> chunks 4hf..4hf+3 of the swizzled fp16 row;
                // chunk c holds, for its 8 codes c0..c7, the order c0 c4 c1 c5 c2 c6 c3 c7
                const int r = t >> 1, hf = t & 1;
                uint8_t* A = st;
                if (r < rows) {
                    const uint4 cw = *reinterpret_cast<const uint4*>(st + UpSmem::kA + UpSmem::kB + r * 32 + 16 * hf);
                    const float2 sbv = half2_to_float2(sb_s[r * G + k]);
                    const __half2 s1 = __floats2half2_rn(sbv.x, sbv.x);
                    const __half2 s16 = __floats2half2_rn(sbv.x * 0.0625f, sbv.x * 0.0625f);
                    const __half2 b2 = __floats2half2_rn(sbv.y, sbv.y);
                    const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f);
                    const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t lo = w[j], hi = w[j] >> 8;
                        // fp16 1024 + c (or 1024 + 16c): the code in the low mantissa bits
                        const uint32_t pr[4] = {(lo & 0x000F000Fu) | 0x64006400u, (lo & 0x00F000F0u) | 0x64006400u,
                                                (hi & 0x000F000Fu) | 0x64006400u, (hi & 0x00F000F0u) | 0x64006400u};
                        uint32_t o[4];
#pragma unroll
                        for (int p = 0; p < 4; ++p) {
                            const __half2 qv = __hsub2(*reinterpret_cast<const __half2*>(&pr[p]), k1024);
                            const __half2 v = __hfma2(qv, (p & 1) ? s16 : s1, b2);
                            o[p] = *reinterpret_cast<const uint32_t*>(&v);
                        }
                        *reinterpret_cast<uint4*>(A + sw128_offset(r, 4 * hf + j)) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<uint4*>(A + sw128_offset(r, 4 * hf + j)) = make_uint4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            ok = __syncthreads_and(ok);
            if (t == 0 && ok) {
                tc_fence_after();
                const uint64_t ad = umma_desc_sw128(smem_u32(st));
                const uint64_t bd = umma_desc_sw128(smem_u32(st + UpSmem::kA));
#pragma unroll
                for (int j = 0; j < 4; ++j) umma_f16(tmem, ad + 2 * j, bd + 2 * j, idesc, (k | j) != 0);
                umma_commit(&ring.done[s]);
                ++ring.committed;
            }
        }
        if (ok) {
            const uint32_t ql = it + G - 1;
            ok = mbar_wait(&ring.done[ql % kStages], (ql / kStages) & 1);
        }
        ok = __syncthreads_and(ok);
        tc_fence_after();
        it += G;
        // ---- epilogue: + offset, ReLU^2, H (fp16) and the live flags of the block's 64-neuron tiles
        if (warp < 4 && ok) {
            const int r = 32 * warp + lane;
            const int n = row0 + r;
            const float off = off_s[r];
            uint16_t* hb = shared ? io.h_s : io.h_r;
            unsigned anylive = 0;
            for (int c0 = 0; c0 < nt16; c0 += 16) {
                float v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = c0 + i;
                    const float z = v[i] + off;
                    const __half hh = __float2half_rn(z > 0.f ? z * z : 0.f);
                    const bool in = c < ti.ntok && r < rows;
                    anylive |= __ballot_sync(0xffffffffu, in && __half2float(hh) > 0.f);
                    if (in) hb[(size_t)(ti.row0 + c) * N + n] = __half_as_ushort(hh);
                }
            }
            const bool force = (io.flags & HS_FORCE_DENSE) != 0;
            if (lane == 0 && 32 * warp < rows && (anylive || force)) {
                const int kt = n / 64;
                atomicOr(io.flag_r + (size_t)tile * words + kt / 32, 1u << (kt % 32));
            }
            if (lane == 0 && anylive)
                atomicAdd(&io.meta->union_rt, (unsigned long long)__popc(anylive) * (unsigned long long)ti.ntok);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (t == 0) ring.drain();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------ down GEMM
__global__ void __launch_bounds__(256, 1)
prefill_down_kernel(const __grid_constant__ LayerParams P, const PrefillIO io, const __grid_constant__ TMaps tm) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int H = P.hidden;
    uint8_t* stage0 = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * DownSmem::kStage);
    uint32_t* tmem_s = reinterpret_cast<uint32_t*>(bars + 2 * kStages);
    int* nk_s = reinterpret_cast<int*>(tmem_s + 2);
    int* klist = nk_s + 2;   // live k-tiles of the unit, ascending (<= kMaxKTiles)
    Ring ring;
    ring.full = bars;
    ring.done = bars + kStages;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    if (t == 0) {
        for (int i = 0; i < 2 * kStages; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_s, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_s;
    pdl_wait();
    pdl_trigger();
    PrefillMeta* m = io.meta;
    const int E = P.n_routed, NR = P.routed_neurons, NS = P.shared_neurons, K = P.top_k;
    const int nb = H / 128;
    const int U = m->dn_units;
    const int words = (max(NR, NS) / 64 + 31) / 32;
    const bool dense = (io.flags & HS_FORCE_DENSE) != 0;
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
        // ---- unit: token tile x 128-output band
        const int tile = u / nb, ob = u % nb;
        const TileInfo ti = io.tiles[tile];
        const bool shared = ti.e == E;
        const int N = shared ? NS : NR;
        const int NK = N / 64;
        const ExpertPtrs ep = shared ? P.shared : routed_ptrs(P, ti.e);
        const int nt16 = (ti.ntok + 15) & ~15;
        const int bi = box_index(ti.ntok);
        const uint32_t bbytes = (uint32_t)(64 << bi) * 128;
        const CUtensorMap* cmap = shared ? &tm.dn_codes_s : &tm.dn_codes_r;
        const CUtensorMap* hmap = shared ? &tm.hsh[bi] : &tm.hr[bi];
        const int cy0 = shared ? 0 : ti.e * NR;
        auto issue = [&](int kk) -> bool {
            if (!ring.acquire()) return false;
            const int s = ring.issued % kStages;
            uint8_t* st = stage0 + s * DownSmem::kStage;
            const int j = klist[kk];
            mbar_arrive_expect_tx(&ring.full[s], (uint32_t)(DownSmem::kC + DownSmem::kSB) + bbytes);
            tma_load_2d(st + DownSmem::kA + DownSmem::kB, cmap, 64 * ob, cy0 + 64 * j, &ring.full[s]);
            bulk_g2s(st + DownSmem::kA + DownSmem::kB + DownSmem::kC, ep.dn_sb + (size_t)j * H + 128 * ob,
                     DownSmem::kSB, &ring.full[s], policy_evict_first());
            tma_load_2d(st + DownSmem::kA, hmap, 64 * j, ti.row0, &ring.full[s]);
            ++ring.issued;
            return true;
        };
        if (t == 0) {
            int nk = 0;
            for (int j = 0; j < NK; ++j) {
                const uint32_t fw = __ldcg(io.flag_r + (size_t)tile * words + j / 32);
                if (dense || ((fw >> (j % 32)) & 1u)) klist[nk++] = j;
            }
            *nk_s = nk;
            if (ob == 0) {
                atomicAdd(&m->total, NK);
                atomicAdd(&m->skipped, NK - nk);
                atomicAdd(&m->exec_rt, (unsigned long long)ti.ntok * 64ull * (unsigned long long)nk);
                atomicAdd(&m->dense_rt, (unsigned long long)ti.ntok * (unsigned long long)N);
            }
            for (int kk = 0; kk < kStages - 1 && kk < nk && ok; ++kk) ok = issue(kk);
        }
        ok = __syncthreads_and(ok);
        const int nk = *nk_s;
        const uint32_t idesc = umma_idesc_f16_f32(128, nt16);
        for (int kk = 0; kk < nk && ok; ++kk) {
            const uint32_t q = it + kk;
            const int s = q % kStages;
            uint8_t* st = stage0 + s * DownSmem::kStage;
            if (t == 0 && kk + kStages - 1 < nk) ok = issue(kk + kStages - 1);
            ok = ok && mbar_wait(&ring.full[s], (q / kStages) & 1);
            if (ok) {
                // thread (output pair p, neuron quarter qn): neurons 16qn..16qn+15 of outputs 2p, 2p+1,
                // written as K-major fp16 rows (one output per row) of the swizzled tile
                const int p = t & 63, qn = t >> 6;
                const uint8_t* cs = st + DownSmem::kA + DownSmem::kB;
                const uint32_t* sbs = reinterpret_cast<const uint32_t*>(cs + DownSmem::kC);
                const float2 sb0 = half2_to_float2(sbs[2 * p]), sb1 = half2_to_float2(sbs[2 * p + 1]);
                uint32_t o0[8], o1[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t ba = cs[(16 * qn + 2 * i) * 64 + p];
                    const uint32_t bb = cs[(16 * qn + 2 * i + 1) * 64 + p];
                    const __half2 v0 = __floats2half2_rn(fmaf(sb0.x, (float)(ba & 15u), sb0.y),
                                                         fmaf(sb0.x, (float)(bb & 15u), sb0.y));
                    const __half2 v1 = __floats2half2_rn(fmaf(sb1.x, (float)(ba >> 4), sb1.y),
                                                         fmaf(sb1.x, (float)(bb >> 4), sb1.y));
                    o0[i] = *reinterpret_cast<const uint32_t*>(&v0);
                    o1[i] = *reinterpret_cast<const uint32_t*>(&v1);
                }
                uint8_t* A = st;
                *reinterpret_cast<uint4*>(A + sw128_offset(2 * p, 2 * qn)) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
                *reinterpret_cast<uint4*>(A + sw128_offset(2 * p, 2 * qn + 1)) = make_uint4(o0[4], o0[5], o0[6], o0[7]);
                *reinterpret_cast<uint4*>(A + sw128_offset(2 * p + 1, 2 * qn)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
                *reinterpret_cast<uint4*>(A + sw128_offset(2 * p + 1, 2 * qn + 1)) =
                    make_uint4(o1[4], o1[5], o1[6], o1[7]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            ok = __syncthreads_and(ok);
            if (t == 0 && ok) {
                tc_fence_after();
                const uint64_t ad = umma_desc_sw128(smem_u32(st));
                const uint64_t bd = umma_desc_sw128(smem_u32(st + DownSmem::kA));
#pragma unroll
                for (int j = 0; j < 4; ++j) umma_f16(tmem, ad + 2 * j, bd + 2 * j, idesc, (kk | j) != 0);
                umma_commit(&ring.done[s]);
                ++ring.committed;
            }
        }
        if (ok && nk > 0) {
            const uint32_t ql = it + nk - 1;
            ok = mbar_wait(&ring.done[ql % kStages], (ql / kStages) & 1);
        }
        ok = __syncthreads_and(ok);
        tc_fence_after();
        it += nk;
        // ---- epilogue: router-weighted partial rows of the tile's tokens for this band
        if (warp < 4 && ok) {
            const int o = 128 * ob + 32 * warp + lane;
            for (int c0 = 0; c0 < nt16; c0 += 16) {
                float v[16];
                if (nk > 0) {
                    tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = c0 + i;
                    if (c < ti.ntok) {
                        const int row = ti.row0 + c;  // grouped pair (routed) or token (shared)
                        const float wgt = shared ? 1.f : io.pair_w[row];
                        const size_t prow = shared ? (size_t)io.T * K + row : (size_t)row;
                        io.partial[prow * H + o] = wgt * v[i];
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (t == 0) ring.drain();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
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
        if (P.shared_neurons) a = __ldcg(reinterpret_cast<const float4*>(io.partial + ((size_t)io.T * K + tok) * H) + c4);
        for (int j = 0; j < K; ++j) {
            const int row = io.pos_of[tok * K + j];
            const float4 v = __ldcg(reinterpret_cast<const float4*>(io.partial + (size_t)row * H) + c4);
            a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
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
    size_t meta, tiles, idx, w, pair_tok, pos_of, pair_w, xg, h_r, h_s, flags, partial, total;
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
    io.max_tiles = l.max_tiles;

    // tensor maps
    hs::TMaps tm;
    memset(&tm, 0, sizeof(tm));
    const uint64_t rows_x = (uint64_t)T * K + (NS ? T : 0);
    bool okm = true;
    okm &= make_map(enc, &tm.up_codes_r, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->routed[0].up.codes, H / 2, (uint64_t)E * NR,
                    H / 2, 32, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    okm &= make_map(enc, &tm.dn_codes_r, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->routed[0].down_nm.codes, H / 2,
                    (uint64_t)E * NR, H / 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (NS) {
        okm &= make_map(enc, &tm.up_codes_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->shared->up.codes, H / 2, NS, H / 2, 32,
                        128, CU_TENSOR_MAP_SWIZZLE_NONE);
        okm &= make_map(enc, &tm.dn_codes_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, L->shared->down_nm.codes, H / 2, NS, H / 2,
                        64, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    for (int b = 0; b < 3; ++b) {
        const uint32_t br = 64u << b;
        okm &= make_map(enc, &tm.xg[b], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, io.xg, H, rows_x, (uint64_t)H * 2, 64, br,
                        CU_TENSOR_MAP_SWIZZLE_128B);
        okm &= make_map(enc, &tm.hr[b], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, io.h_r, NR, (uint64_t)T * K, (uint64_t)NR * 2,
                        64, br, CU_TENSOR_MAP_SWIZZLE_128B);
        if (NS)
            okm &= make_map(enc, &tm.hsh[b], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, io.h_s, NS, T, (uint64_t)NS * 2, 64, br,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (!okm) return HS_ERR_CUDA;

    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return HS_ERR_CUDA;
    const int up_smem = hs::UpSmem::total(H);
    const int dn_smem = hs::DownSmem::total();
    if (set_smem_attr((const void*)hs::prefill_up_kernel, up_smem) != HS_OK) return HS_ERR_CUDA;
    if (set_smem_attr((const void*)hs::prefill_down_kernel, dn_smem) != HS_OK) return HS_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_pdl(hs::prefill_route_kernel, dim3((T + 7) / 8), dim3(256), 0, s, P, io) != cudaSuccess) return HS_ERR_CUDA;
    if (launch_pdl(hs::prefill_count_kernel, dim3(E), dim3(256), 0, s, P, io) != cudaSuccess) return HS_ERR_CUDA;
    if (launch_pdl(hs::prefill_tiles_kernel, dim3(1), dim3(256), 0, s, P, io) != cudaSuccess) return HS_ERR_CUDA;
    if (launch_pdl(hs::prefill_list_kernel, dim3(E), dim3(256), 0, s, P, io) != cudaSuccess) return HS_ERR_CUDA;
    if (launch_pdl(hs::prefill_gather_kernel, dim3(4 * sms), dim3(256), 0, s, P, io) != cudaSuccess) return HS_ERR_CUDA;
    if (launch_pdl(hs::prefill_up_kernel, dim3(sms), dim3(256), up_smem, s, P, io, tm) != cudaSuccess)
        return HS_ERR_CUDA;
    if (launch_pdl(hs::prefill_down_kernel, dim3(sms), dim3(256), dn_smem, s, P, io, tm) != cudaSuccess)
        return HS_ERR_CUDA;
    if (launch_pdl(hs::prefill_combine_kernel, dim3(4 * sms), dim3(256), 0, s, P, io) != cudaSuccess)
        return HS_ERR_CUDA;
    (void)NR;
    return launch_err();
}
