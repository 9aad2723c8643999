// Single-expert activation-sparse down projection of one token, GB300 (sm_103a).
//
// Method: "Skipping dead neurons: a faster Nemotron 3.5 Lightning on Apple
// silicon" (sevren.ai, "Heimr Sparse Down").
//  * "Our way reads only the rows that fired": the down weights are stored one
//    row per neuron; only neurons with h_n > 0 are read; the work is split
//    into slices of neurons and bands of outputs so that every core is busy,
//    and a final small pass adds the slices' partial sums.
//  * "The whole decode step": the (scale, bias) slab of a group of 64 neurons
//    is read only if a neuron of the group fired.
//
// GB300 design (ours): CTA (b, c) = (band of 64 outputs, chunk of up to 32
// consecutive 64-neuron scale groups), 256 threads; thread (gi, j) owns
// group gi of the chunk and the 8 outputs of code word j of the band's 32
// bytes in every row.  The 8 threads of a group (adjacent lanes of one warp)
// each read 8 of its h values, and build the group's 64-bit live mask and
// fixed-order h sum by three shuffle steps (no CTA barrier: 4.48 against 5.00
// us per call with a staging pass and two barriers); each thread then loads
// word j of each live row of its group directly (up to 16 rows in flight; 8
// adjacent lanes read a row's 32-byte band slice, one sector) together with
// its 8 (scale, bias) pairs of the group's slab, so one round trip to memory
// follows the mask.  The groups'
// partial sums meet in shared memory and are added in group order.  An
// expert of at most 32 groups (2048 neurons) is one chunk: the CTA writes y
// directly, with no scratch and no second pass.  Wider experts use one CTA
// per chunk; each writes its chunk's partial band to the workspace and takes
// a ticket on its band's counter, and the last chunk of a band to arrive adds
// the chunks' partials in chunk order, rounds to bf16 and puts the counter
// back to zero: no CTA waits for another.  The summation order is fixed
// (rows ascending within a group, groups within a chunk, chunks in order),
// so results are deterministic and the dense flag gives identical bits.
#include <cuda.h>

#include "hs_common.cuh"
#include "hs_host.h"

#include <cstdlib>
#include <mutex>

namespace hs {

constexpr int kDsThreads = 256;
constexpr int kDsBand = 64;                 // outputs per band: 8 code words of 8 outputs
constexpr int kDsWords = kDsBand / 8;
constexpr int kDsChunk = kDsThreads / kDsWords;   // 32 groups per CTA
constexpr int kDsRowsInFlight = 16;         // live rows whose code words one thread loads before using them
constexpr int kDsMaxGroups = 1024;          // neurons <= 65536

// Accumulates one row n (h value hn) into acc[0..7] for the 8 outputs of code
// word w (output 8j+i in nibble i).  Nibble i becomes a float by masking it
// in place under the exponent of 2^23 and subtracting 2^23 (exact:
// q * 16^i < 2^23); h is pre-scaled by 16^-i to undo the position.  Rows are
// added in ascending n, one fp32 chain per output.
__device__ __forceinline__ void ds_accumulate_word(uint32_t w, float hn, float (&acc)[8]) {
    const float hs[5] = {hn, hn * 0.0625f, hn * 0.00390625f, hn * 0.000244140625f, hn * 1.52587890625e-05f};
    const uint32_t hi = w >> 12;  // nibbles 5, 6, 7 at positions 2, 3, 4
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t src = i < 5 ? w : hi;
        const int pos = i < 5 ? i : i - 3;
        const float q = __uint_as_float((src & (15u << (4 * pos))) | 0x4B000000u) - 8388608.f;
        acc[i] = fmaf(hs[pos], q, acc[i]);
    }
}

// Workspace of a call with more than one chunk per band: one ticket counter
// per band (zero between calls), the group live masks [G] (written by the
// CTAs of band 0) and the chunks' partial bands [nb][nc][64] fp32.
struct DsWork {
    float* partial;
    unsigned long long* gmask;
    unsigned* tickets;
};

// Exclusive prefix over the 256 threads of the CTA; `tmp` holds 8 ints.
__device__ __forceinline__ int ds_excl_scan(int v, int* tmp, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) tmp[warp] = incl;
    __syncthreads();
    int before = 0;
    total = 0;
#pragma unroll
    for (int i = 0; i < kDsThreads / 32; ++i) {
        before += i < warp ? tmp[i] : 0;
        total += tmp[i];
    }
    __syncthreads();
    return incl - v + before;
}

// Ascending indices of the rows read (group g's word in masks(g)), and their
// count, for G groups: thread t takes a run of consecutive groups.
template <typename MaskAt>
__device__ __forceinline__ void ds_write_live(int G, MaskAt masks, int* live_idx, int* live_count, int* tmp) {
    const int t = threadIdx.x;
    const int per = (G + kDsThreads - 1) / kDsThreads;
    const int g0 = min(G, t * per), g1 = min(G, g0 + per);
    int c = 0;
    for (int g = g0; g < g1; ++g) c += __popcll(masks(g));
    int total = 0;
    int o = ds_excl_scan(c, tmp, total);
    if (live_count && t == 0) *live_count = total;
    if (live_idx)
        for (int g = g0; g < g1; ++g) {
            uint64_t m = masks(g);
            while (m) {
                live_idx[o++] = 64 * g + __ffsll((long long)m) - 1;
                m &= m - 1;
            }
        }
}

__global__ void __launch_bounds__(kDsThreads)
down_sparse_kernel(const float* __restrict__ h, const uint8_t* __restrict__ dn_codes, const uint32_t* __restrict__ dn_sb,
                   int hidden, int G, unsigned flags, DsWork ws, uint16_t* __restrict__ y_bf16,
                   float* __restrict__ y_f32, int* __restrict__ live_idx, int* __restrict__ live_count) {
    __shared__ float h_s[kDsChunk * 64];
    __shared__ __align__(16) float red[kDsChunk][kDsBand + 4];   // padded rows: fewer bank conflicts
    __shared__ unsigned long long mask_s[kDsChunk];
    __shared__ int tmp[kDsThreads / 32];
    __shared__ int s_last;
    const int b = blockIdx.x, c = blockIdx.y, nc = gridDim.y;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int gbase = c * kDsChunk, ng = min(kDsChunk, G - gbase);
    const int rowb = hidden / 2;
    const bool dense = (flags & HS_FORCE_DENSE) != 0;
    // h of the chunk's groups into L2 ahead of the wait (nothing is read from it before it)
    if (warp == 1) prefetch_l2_span(h + (size_t)gbase * 64, ng * 64 * 4, lane);
    pdl_wait();
    pdl_trigger();
    // thread (gi, j): h values 8j .. 8j+7 of group gi (two 16-byte loads), into shared memory
    // for the accumulation; the group's live mask and fixed-order h sum by the 8 lanes of the
    // group (adjacent lanes of one warp), so no CTA barrier precedes the row loads
    const int gi = t / kDsWords, j = t % kDsWords;
    uint64_t gmask = 0;
    float hsum = 0.f;
    {
        float hv[8];
        if (gi < ng) {
            const float4* hp = reinterpret_cast<const float4*>(h + (size_t)(gbase + gi) * 64 + 8 * j);
            const float4 x0 = hp[0], x1 = hp[1];
            hv[0] = x0.x; hv[1] = x0.y; hv[2] = x0.z; hv[3] = x0.w;
            hv[4] = x1.x; hv[5] = x1.y; hv[6] = x1.z; hv[7] = x1.w;
            reinterpret_cast<float4*>(h_s + gi * 64 + 8 * j)[0] = x0;
            reinterpret_cast<float4*>(h_s + gi * 64 + 8 * j)[1] = x1;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) hv[i] = 0.f;
        }
        unsigned bits = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            bits |= (hv[i] > 0.f ? 1u : 0u) << i;
            hsum += hv[i];
        }
        gmask = (uint64_t)bits << (8 * j);
#pragma unroll
        for (int off = 1; off < kDsWords; off <<= 1) {
            gmask |= __shfl_xor_sync(0xffffffffu, gmask, off);
            hsum += __shfl_xor_sync(0xffffffffu, hsum, off);
        }
        if (gi < ng && j == 0) mask_s[gi] = gmask;  // for the live index list
    }
    __syncwarp();  // the group's h values were written by lanes of this warp
    // thread (gi, j): word j of the band in every live row of group gi
    if (gi < ng) {
        const int g = gbase + gi;
        const uint64_t live = dense ? ~0ull : gmask;
        float r[8];
        if (live) {
            const int o0 = b * kDsBand + 8 * j;  // first output of this thread
            const uint32_t* col = reinterpret_cast<const uint32_t*>(dn_codes + (size_t)g * 64 * rowb) + o0 / 8;
            const uint4* sbp = reinterpret_cast<const uint4*>(dn_sb + (size_t)g * hidden + o0);
            const uint4 sb0 = sbp[0], sb1 = sbp[1];
            const float* hg = h_s + gi * 64;
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.f;
            uint64_t m = live;
            while (m) {
                uint32_t wv[kDsRowsInFlight];
                int nv[kDsRowsInFlight];
#pragma unroll
                for (int i = 0; i < kDsRowsInFlight; ++i) {
                    nv[i] = -1;
                    wv[i] = 0u;
                    if (m) {
                        nv[i] = __ffsll((long long)m) - 1;
                        m &= m - 1;
                        wv[i] = col[(size_t)nv[i] * (rowb / 4)];
                    }
                }
#pragma unroll
                for (int i = 0; i < kDsRowsInFlight; ++i)
                    if (nv[i] >= 0) ds_accumulate_word(wv[i], hg[nv[i]], acc);
            }
            // partial_o = s_o * sum_n h_n q_{n,o} + b_o * sum_n h_n
            const uint32_t sbw[8] = {sb0.x, sb0.y, sb0.z, sb0.w, sb1.x, sb1.y, sb1.z, sb1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 sb = half2_to_float2(sbw[i]);
                r[i] = fmaf(sb.x, acc[i], sb.y * hsum);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) r[i] = 0.f;
        }
        reinterpret_cast<float4*>(&red[gi][8 * j])[0] = make_float4(r[0], r[1], r[2], r[3]);
        reinterpret_cast<float4*>(&red[gi][8 * j])[1] = make_float4(r[4], r[5], r[6], r[7]);
    }
    __syncthreads();
    // the chunk's groups added in order, one output per thread
    float yo = 0.f;
    if (t < kDsBand)
        for (int k = 0; k < ng; ++k) yo += red[k][t];
    const int o = b * kDsBand + t;
    if (nc == 1) {
        if (t < kDsBand) {
            if (y_f32) y_f32[o] = yo;
            y_bf16[o] = f32_to_bf16_bits(yo);
        }
        if (b == 0 && (live_idx || live_count))
            ds_write_live(ng, [&](int g) -> uint64_t { return dense ? ~0ull : mask_s[g]; }, live_idx, live_count, tmp);
        return;
    }
    // several chunks: publish this chunk's partial band, then take a ticket
    if (t < kDsBand) ws.partial[((size_t)b * nc + c) * kDsBand + t] = yo;
    if (b == 0 && t < ng) ws.gmask[gbase + t] = dense ? ~0ull : mask_s[t];
    __syncthreads();
    if (t == 0) {
        __threadfence();
        s_last = atomicAdd(&ws.tickets[b], 1u) == (unsigned)(nc - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (t < kDsBand) {
        float a = 0.f;
        for (int k = 0; k < nc; ++k) a += __ldcg(ws.partial + ((size_t)b * nc + k) * kDsBand + t);
        if (y_f32) y_f32[o] = a;
        y_bf16[o] = f32_to_bf16_bits(a);
    }
    if (b == 0 && (live_idx || live_count))
        ds_write_live(G, [&](int g) -> uint64_t { return __ldcg(&ws.gmask[g]); }, live_idx, live_count, tmp);
    if (t == 0) ws.tickets[b] = 0u;  // every chunk of the band has taken its ticket
}

}  // namespace hs

// ===================================================================== host
using namespace hs_host;

namespace {

struct DsLayout {
    size_t partial, gmask, tickets, total;
};

constexpr size_t ds_round(size_t v) { return (v + 255) / 256 * 256; }

// The ticket counters sit first, at the same offset for every shape, so that
// no call's partial sums overwrite another shape's counters: a workspace
// serves calls of any shapes it is large enough for without clearing.
constexpr size_t kDsTicketBytes = ds_round((size_t)(hs::kMaxHidden / hs::kDsBand) * sizeof(unsigned));

constexpr DsLayout ds_layout(int neurons, int out_dim) {
    return DsLayout{kDsTicketBytes + ds_round((size_t)(neurons / 64) * sizeof(unsigned long long)),
                    kDsTicketBytes, 0,
                    kDsTicketBytes + ds_round((size_t)(neurons / 64) * sizeof(unsigned long long)) +
                        ds_round((size_t)((neurons / 64 + hs::kDsChunk - 1) / hs::kDsChunk) * out_dim *
                                 sizeof(float))};
}

int ds_check(const float* h, const hs_w4* down_nm, int neurons, int out_dim, const uint16_t* y_bf16, const float* y_f32,
             const int* live_idx, const int* live_count, unsigned flags) {
    if (!h || !down_nm || !down_nm->codes || !down_nm->sb || !y_bf16) return HS_ERR_INVALID_ARG;
    if (flags & ~HS_FORCE_DENSE) return HS_ERR_INVALID_ARG;  // group slabs only; no batch flags
    if (neurons <= 0 || out_dim <= 0) return HS_ERR_INVALID_ARG;
    if (neurons % 64 || out_dim % 64 || out_dim > hs::kMaxHidden || neurons > 64 * hs::kDsMaxGroups)
        return HS_ERR_UNSUPPORTED_SHAPE;
    if (!al16(h) || !al16(down_nm->codes) || !al16(down_nm->sb) || !al16(y_bf16) || (y_f32 && !al16(y_f32)) ||
        (live_idx && !al4(live_idx)) || (live_count && !al4(live_count)))
        return HS_ERR_MISALIGNED;
    return HS_OK;
}

int ds_launch(const float* h, const hs_w4* down_nm, int neurons, int out_dim, uint16_t* y_bf16, float* y_f32,
              int* live_idx, int* live_count, unsigned flags, char* ws, hs_stream_t stream) {
    const int G = neurons / 64;
    const int nb = out_dim / hs::kDsBand, nc = (G + hs::kDsChunk - 1) / hs::kDsChunk;
    const DsLayout l = ds_layout(neurons, out_dim);
    hs::DsWork w{reinterpret_cast<float*>(ws + l.partial), reinterpret_cast<unsigned long long*>(ws + l.gmask),
                 reinterpret_cast<unsigned*>(ws + l.tickets)};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_pdl(hs::down_sparse_kernel, dim3(nb, nc), dim3(hs::kDsThreads), 0, s, h, down_nm->codes,
                   static_cast<const uint32_t*>(down_nm->sb), out_dim, G, flags, w, y_bf16, y_f32, live_idx,
                   live_count) != cudaSuccess)
        return HS_ERR_CUDA;
    return launch_err();
}

}  // namespace

extern "C" size_t hs_expert_down_sparse_workspace_size(int neurons, int out_dim) {
    if (neurons <= 0 || out_dim <= 0 || neurons % 64 || out_dim % 64 || neurons > 64 * hs::kDsMaxGroups ||
        out_dim > hs::kMaxHidden)
        return 0;
    return ds_layout(neurons, out_dim).total;
}

extern "C" int hs_expert_down_sparse(const float* h, const hs_w4* down_nm, int neurons, int out_dim, uint16_t* y_bf16,
                                     float* y_f32, int* live_idx, int* live_count, unsigned flags, void* ws,
                                     size_t ws_bytes, hs_stream_t stream) {
    const int st = ds_check(h, down_nm, neurons, out_dim, y_bf16, y_f32, live_idx, live_count, flags);
    if (st != HS_OK) return st;
    if (!al16(ws)) return HS_ERR_MISALIGNED;
    if (!ws || ws_bytes < ds_layout(neurons, out_dim).total) return HS_ERR_WORKSPACE;
    return ds_launch(h, down_nm, neurons, out_dim, y_bf16, y_f32, live_idx, live_count, flags, static_cast<char*>(ws),
                     stream);
}

// ============================================================================
// Allocation-free variant of hs_expert_down_sparse.
//
// Some callers cannot hand the library a workspace: code that runs where
// device allocation is not allowed or not available at call time (a plugin
// that only receives the tensors it must read and write from a host framework
// which owns every allocation, or a real-time path that must never enter the
// CUDA allocator).  For them the kernel's scratch (the chunks' partial bands,
// the group masks and the ticket counters that experts wider than one
// 32-group chunk need) lives in a fixed array compiled into the library; each
// GPU that loads the library keeps that array (about 0.4 MB) until the
// process exits.
//
// The host never dereferences the array's name or passes it to a kernel: in
// host code that name is only a stand-in.  Its device address is looked up
// with cudaGetSymbolAddress and cached per CUDA context, keyed by the
// context's unique id (a context created after a device reset has a new id,
// so the address is looked up again); a failed launch also drops the entry.
// ============================================================================
namespace {
constexpr int kNoAllocMaxNeurons = 64 * hs::kDsMaxGroups;   // the workspace entry point's limits
constexpr int kNoAllocMaxOut = hs::kMaxHidden;
constexpr size_t kNoAllocBytes = ds_layout(kNoAllocMaxNeurons, kNoAllocMaxOut).total;
}  // namespace

// Zero at load (static storage).  Every call puts the ticket counters in it
// back to zero, and writes each partial slice before reading it.
static __device__ __align__(256) unsigned char hs_noalloc_scratch[kNoAllocBytes];

namespace {
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct NoAllocCache {
    std::mutex mu;
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
    bool resolved = false;
    static constexpr int kSlots = 64;
    unsigned long long ctx_id[kSlots] = {};
    void* addr[kSlots] = {};
    int n = 0;
};

NoAllocCache& noalloc_cache() {
    static NoAllocCache c;
    return c;
}

// Unique id of the current context (0 if none can be had).
unsigned long long current_ctx_id(NoAllocCache& c) {
    if (!c.resolved) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess)
            c.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess)
            c.get_id = reinterpret_cast<CtxGetIdFn>(p);
        c.resolved = true;
    }
    if (!c.get_current || !c.get_id) return 0;
    CUcontext ctx = nullptr;
    if (c.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (c.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of hs_noalloc_scratch in the current context, or nullptr.
void* noalloc_scratch_address(unsigned long long* key_out) {
    NoAllocCache& c = noalloc_cache();
    std::lock_guard<std::mutex> lock(c.mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    unsigned long long id = current_ctx_id(c);
    if (id == 0) {
        // no context made current yet: the symbol lookup initialises the device's context
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, hs_noalloc_scratch) != cudaSuccess) return nullptr;
        id = current_ctx_id(c);
        if (id == 0) return nullptr;
    }
    *key_out = id;
    for (int i = 0; i < c.n; ++i)
        if (c.ctx_id[i] == id) return c.addr[i];
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, hs_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    const int slot = c.n < NoAllocCache::kSlots ? c.n++ : (int)(id % NoAllocCache::kSlots);
    c.ctx_id[slot] = id;
    c.addr[slot] = p;
    return p;
}

void noalloc_forget(unsigned long long id) {
    NoAllocCache& c = noalloc_cache();
    std::lock_guard<std::mutex> lock(c.mu);
    for (int i = 0; i < c.n; ++i)
        if (c.ctx_id[i] == id) c.ctx_id[i] = 0;
}
}  // namespace

extern "C" int hs_expert_down_sparse_noalloc(const float* h, const hs_w4* down_nm, int neurons, int out_dim,
                                             uint16_t* y_bf16, float* y_f32, int* live_idx, int* live_count,
                                             unsigned flags, hs_stream_t stream) {
    const int st = ds_check(h, down_nm, neurons, out_dim, y_bf16, y_f32, live_idx, live_count, flags);
    if (st != HS_OK) return st;
    // beyond the compiled-in scratch capacity
    if (neurons > kNoAllocMaxNeurons || out_dim > kNoAllocMaxOut) return HS_ERR_UNSUPPORTED_SHAPE;
    unsigned long long key = 0;
    char* scratch = static_cast<char*>(noalloc_scratch_address(&key));
    if (!scratch) return HS_ERR_CUDA;
    // the layout of a smaller shape fits inside the largest one's
    if (ds_layout(neurons, out_dim).total > kNoAllocBytes) return HS_ERR_UNSUPPORTED_SHAPE;
    const int r = ds_launch(h, down_nm, neurons, out_dim, y_bf16, y_f32, live_idx, live_count, flags, scratch, stream);
    if (r == HS_ERR_CUDA) noalloc_forget(key);
    return r;
}
